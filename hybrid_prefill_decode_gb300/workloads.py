"""Seeded synthetic hybrid batches (inputs only — no attention arithmetic lives here).

Both the CUDA path and the fp64 oracle are fed from these generators; this module computes
nothing of the method. A batch is one layer of one serving iteration: some prompt chunks
(prefill / extend) and some decoding sequences over one paged K/V pool
("Week 6: Beyond PyTorch: Custom Kernel과 vLLM", §"한 스텝에 여러 종류의 request 섞기" and
§"PagedAttention").

Recipe:
  * integer choices (lengths, prefix offsets) come from ``random.Random(seed)``;
  * physical blocks are a ``torch.randperm`` of the pool (seed-derived CPU generator), so a
    sequence's logical blocks are scattered;
  * Q, K, V are N(0, 1) fp32 draws from a seed-derived ``torch.Generator`` on the target
    device, rounded to bf16; draw order: q_prefill, q_decode, k_pool, v_pool;
  * the pool holds sum(ceil(kv_len/16)) blocks plus 5 % spare; spare blocks, the unused slots
    of every sequence's last block, and the block-table entries past each sequence's end (which
    point at a spare block) are poisoned with bf16 NaN, so any read outside the visible rows
    shows up as NaN in the output.
"""
from __future__ import annotations

import math
import random
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

HEAD_DIM = 128
BLOCK_SIZE = 16
BF16_NAN_BITS = 0x7FC0


@dataclass
class HybridBatch:
    """One hybrid batch. Tensors live on ``device``; host lists mirror the int32 tables."""
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    q_lens: List[int]               # prefill chunk lengths
    prefill_kv_lens: List[int]      # cached rows of each prefill sequence (chunk included)
    decode_kv_lens: List[int]       # cached rows of each decode sequence (new token included)
    scale: float
    q_prefill: torch.Tensor         # bf16 [Tp][Hq][D]
    q_decode: torch.Tensor          # bf16 [Nd][Hq][D]
    k_pool: torch.Tensor            # bf16 [NB][Hkv][16][D]
    v_pool: torch.Tensor            # bf16 [NB][Hkv][16][D]
    block_tables: torch.Tensor      # int32 [Np+Nd][max_blocks_per_seq]
    cu_seqlens_q: torch.Tensor      # int32 [Np+1]
    kv_lens: torch.Tensor           # int32 [Np+Nd]
    seed: int = 0
    name: str = ""
    meta: dict = field(default_factory=dict)
    causal: bool = True             # False: chunk tokens see every row of their sequence

    @property
    def num_prefill_seqs(self) -> int:
        return len(self.q_lens)

    @property
    def num_decode_seqs(self) -> int:
        return len(self.decode_kv_lens)

    @property
    def num_prefill_tokens(self) -> int:
        return int(sum(self.q_lens))

    @property
    def num_blocks(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def host_cu_seqlens(self) -> List[int]:
        cu = [0]
        for n in self.q_lens:
            cu.append(cu[-1] + n)
        return cu

    @property
    def host_kv_lens(self) -> List[int]:
        return list(self.prefill_kv_lens) + list(self.decode_kv_lens)

    def to(self, device) -> "HybridBatch":
        """A copy with every tensor moved to ``device``."""
        kw = dict(self.__dict__)
        for k, v in list(kw.items()):
            if isinstance(v, torch.Tensor):
                kw[k] = v.to(device)
        return HybridBatch(**kw)


def split_off_new_rows(batch: HybridBatch):
    """The inputs of an iteration whose new tokens' K/V are not yet in the pool: returns
    (k_new, v_new, k_pool, v_pool) where k_new / v_new (bf16 [T_p + Nd][Hkv][D]) hold the rows of
    the iteration's tokens — chunk token i of prefill sequence s at position
    kv_len - q_len + i, then each decode sequence's token at kv_len - 1 — and the returned pools
    are copies of the batch's with exactly those rows set to bf16 NaN (so a read before they are
    written shows up in the output)."""
    seq, pos = [], []
    for s, (q, L) in enumerate(zip(batch.q_lens, batch.prefill_kv_lens)):
        seq += [s] * q
        pos += list(range(L - q, L))
    for d, L in enumerate(batch.decode_kv_lens):
        seq.append(batch.num_prefill_seqs + d)
        pos.append(L - 1)
    dev = batch.k_pool.device
    seq_t = torch.tensor(seq, dtype=torch.long, device=dev)
    pos_t = torch.tensor(pos, dtype=torch.long, device=dev)
    phys = batch.block_tables.to(dev).long()[seq_t, pos_t // BLOCK_SIZE]
    off = pos_t % BLOCK_SIZE
    k_new = batch.k_pool[phys, :, off, :].contiguous()
    v_new = batch.v_pool[phys, :, off, :].contiguous()
    nan = torch.tensor(BF16_NAN_BITS, dtype=torch.int16).view(torch.bfloat16).item()
    k_pool, v_pool = batch.k_pool.clone(), batch.v_pool.clone()
    k_pool[phys, :, off, :] = nan
    v_pool[phys, :, off, :] = nan
    return k_new, v_new, k_pool, v_pool


def _blocks(n: int) -> int:
    return (n + BLOCK_SIZE - 1) // BLOCK_SIZE


def make_batch(num_q_heads: int, num_kv_heads: int, q_lens: Sequence[int],
               prefill_kv_lens: Sequence[int], decode_kv_lens: Sequence[int], seed: int,
               device="cpu", scale: Optional[float] = None, permute: bool = True,
               spare_frac: float = 0.05, poison: bool = True, std: float = 1.0,
               name: str = "", causal: bool = True, head_dim: int = HEAD_DIM) -> HybridBatch:
    """Build one seeded hybrid batch (see the module docstring for the recipe)."""
    q_lens = [int(x) for x in q_lens]
    prefill_kv_lens = [int(x) for x in prefill_kv_lens]
    decode_kv_lens = [int(x) for x in decode_kv_lens]
    assert len(q_lens) == len(prefill_kv_lens)
    D = int(head_dim)
    Hq, Hkv = int(num_q_heads), int(num_kv_heads)
    lens = prefill_kv_lens + decode_kv_lens
    nseq = len(lens)
    need = [_blocks(L) for L in lens]
    used = sum(need)
    spare = max(1, int(math.ceil(spare_frac * used))) if poison else 0
    nb = max(1, used + spare)
    maxb = max([1] + need)

    # physical block assignment: a random permutation of the pool, handed out in order
    g_cpu = torch.Generator().manual_seed(seed * 1_000_003 + 11)
    perm = torch.randperm(nb, generator=g_cpu) if permute else torch.arange(nb)
    spare_ids = perm[used:].tolist()
    tail_fill = spare_ids[0] if spare_ids else 0
    bt = torch.full((max(nseq, 1), maxb), tail_fill, dtype=torch.int32)
    pos = 0
    for s, n in enumerate(need):
        bt[s, :n] = perm[pos:pos + n].to(torch.int32)
        pos += n
    if nseq == 0:
        bt = bt[:0]

    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed * 1_000_003 + 29)

    def draw(*shape):
        x = torch.randn(*shape, generator=g, device=dev, dtype=torch.float32)
        if std != 1.0:
            x = x * std
        return x.to(torch.bfloat16)

    tp = sum(q_lens)
    q_prefill = draw(tp, Hq, D)
    q_decode = draw(len(decode_kv_lens), Hq, D)
    k_pool = draw(nb, Hkv, BLOCK_SIZE, D)
    v_pool = draw(nb, Hkv, BLOCK_SIZE, D)

    if poison:
        nan = torch.tensor(BF16_NAN_BITS, dtype=torch.int16).view(torch.bfloat16).item()
        if spare_ids:
            idx = torch.tensor(spare_ids, dtype=torch.long, device=dev)
            k_pool[idx] = nan
            v_pool[idx] = nan
        for s, L in enumerate(lens):
            r = L % BLOCK_SIZE
            if r:
                last = int(bt[s, need[s] - 1])
                k_pool[last, :, r:, :] = nan
                v_pool[last, :, r:, :] = nan

    cu = [0]
    for n in q_lens:
        cu.append(cu[-1] + n)
    return HybridBatch(
        num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=BLOCK_SIZE, q_lens=q_lens,
        prefill_kv_lens=prefill_kv_lens, decode_kv_lens=decode_kv_lens,
        scale=float(scale if scale is not None else 1.0 / math.sqrt(D)),
        q_prefill=q_prefill, q_decode=q_decode, k_pool=k_pool, v_pool=v_pool,
        block_tables=bt.to(dev), cu_seqlens_q=torch.tensor(cu, dtype=torch.int32, device=dev),
        kv_lens=torch.tensor(lens, dtype=torch.int32, device=dev), seed=seed, name=name,
        causal=causal)


# ----------------------------------------------------------------------------------------------
# The evaluation configurations: attention shapes of the models the POD-Attention digest
# evaluates (Yi-6B, Llama-2-7B, Llama-3-8B, 4K-32K context; "장문맥에서 커지는 이점").
# ----------------------------------------------------------------------------------------------

CONFIG_NAMES = {
    1: "tiny hybrid batch (Hq2/Hkv1, chunk 64 @ 64, 4 decodes)",
    2: "Llama-2-7B attention (32/32, chunk 512 @ 3584, 32 decodes ctx U[2048,4096])",
    3: "Llama-3-8B attention (32/8, chunk 1024 @ U[0,15360], 64 decodes ctx U[8192,16384])",
    4: "Yi-6B attention (32/4, chunk 2048 @ 28672, 16 decodes ctx U[16384,32768])",
}


def config_lengths(i: int):
    """(Hq, Hkv, q_lens, prefill_kv_lens, decode_kv_lens) of configuration i (seed = i)."""
    rng = random.Random(i)
    if i == 1:
        return 2, 1, [64], [128], [100, 150, 233, 300]
    if i == 2:
        return 32, 32, [512], [4096], [rng.randint(2048, 4096) for _ in range(32)]
    if i == 3:
        dec = [rng.randint(8192, 16384) for _ in range(64)]
        off = rng.randint(0, 15360)
        return 32, 8, [1024], [off + 1024], dec
    if i == 4:
        return 32, 4, [2048], [28672 + 2048], [rng.randint(16384, 32768) for _ in range(16)]
    raise ValueError(f"unknown configuration {i}")


def config(i: int, device="cpu", **kw) -> HybridBatch:
    """Configuration i (1..4) as a seeded batch on ``device``."""
    Hq, Hkv, ql, pkv, dkv = config_lengths(i)
    return make_batch(Hq, Hkv, ql, pkv, dkv, seed=i, device=device, name=CONFIG_NAMES[i], **kw)


# Small single-kind cases of the same shapes, used to profile one kernel path at a time (they fit
# a profiler's memory save/restore: at most ~1.6 GB of pool).
PROFILE_CASES = {
    "prefill4": ("Yi-6B prefill only (32/4, chunk 2048 @ 28672)", 4, 32, 4, [2048], [30720], 0),
    "prefill2": ("Llama-2-7B prefill only (32/32, chunk 512 @ 3584)", 2, 32, 32, [512], [4096], 0),
    "decode2": ("Llama-2-7B decodes only (32/32, 32 decodes ctx U[2048,4096])", 2, 32, 32, [],
                [], 32),
    "decode3": ("Llama-3-8B decodes only (32/8, 16 decodes ctx U[8192,16384])", 3, 32, 8, [], [],
                16),
}


def profile_case(name: str, device="cpu") -> HybridBatch:
    """A single-kind case: the prefill chunk or the first decodes of a configuration."""
    label, cfg, Hq, Hkv, ql, pkv, nd = PROFILE_CASES[name]
    _, _, _, _, dkv = config_lengths(cfg)
    return make_batch(Hq, Hkv, ql, pkv, dkv[:nd], seed=cfg, device=device, name=label)


# ----------------------------------------------------------------------------------------------
# Mixed-kind structural example: two decodes, one extend of 8 tokens after a cached prefix,
# one fresh prefill of 4 tokens — 14 new tokens in the step ("Week 6: Beyond PyTorch",
# §"한 스텝에 여러 종류의 request 섞기"). The prefix length of the extend is not printed; it
# is a parameter here.
# ----------------------------------------------------------------------------------------------

def mixed_kind_example(prefix_c: int = 24, ctx_a: int = 37, ctx_b: int = 5, seed: int = 0,
                       num_q_heads: int = 4, num_kv_heads: int = 2,
                       device="cpu") -> HybridBatch:
    """Requests A, B (decode, one token each), C (extend, 8 tokens after `prefix_c` cached
    rows) and D (prefill, 4 tokens, no cache)."""
    q_lens = [8, 4]                      # C, D
    prefill_kv = [prefix_c + 8, 4]       # C sees its prefix; D has none
    decode_kv = [ctx_a, ctx_b]           # A, B
    return make_batch(num_q_heads, num_kv_heads, q_lens, prefill_kv, decode_kv, seed=seed,
                      device=device, name="mixed-kind example (A,B decode; C extend; D prefill)")


# ----------------------------------------------------------------------------------------------
# Configuration 5: a seeded 200-iteration hybrid-batching trace on the Llama-3-8B shape.
# A chunked-prefill scheduler with a 2048-token budget takes every running decode first, then
# fills the rest of the budget with prompt chunks in FIFO order ("LLMSO - W4", §"Prefill-Decode
# 분리 스케줄링": decode first, then prefill up to the token budget).
# ----------------------------------------------------------------------------------------------

@dataclass
class TraceStep:
    q_lens: List[int]
    prefill_kv_lens: List[int]
    decode_kv_lens: List[int]
    prefill_rids: List[int] = field(default_factory=list)   # request of each prompt chunk
    decode_rids: List[int] = field(default_factory=list)    # request of each decode


@dataclass
class Trace:
    mix: str
    steps: List[TraceStep]
    max_rows: List[int]          # per request id: the most cached rows it ever reaches
    decode_targets: tuple = ()   # running decodes held in each quarter of the trace


def trace_decode_targets(num_sms: int, num_kv_heads: int = 8, waves: int = 4) -> tuple:
    """Running-decode counts whose (sequence, kv-head) units land just above 1, 2, 3, 4 times the
    SM count: k * num_sms // num_kv_heads + 1 sequences. For 148 SMs this gives 19, 38, 56, 75
    (152, 304, 448, 600 units); for 152 SMs 20, 39, 58, 77 (160, 312, 464, 616 units)."""
    return tuple(k * num_sms // num_kv_heads + 1 for k in range(1, waves + 1))


def trace(mix: str, seed: int = 5, iters: int = 200, budget: int = 2048,
          decode_targets=(19, 38, 56, 75)) -> Trace:
    """Iteration shapes of mix 'a' (decode-heavy) or 'b' (prefill-heavy).

    (a) prompts log-uniform in [4096, 32768], outputs geometric with mean 256;
    (b) prompts lognormal with mean 16384 (sigma 0.5 in log space), clipped to
        [4096, 32768], outputs geometric with mean 64.
    The number of running decodes is held at a target that changes every quarter of the trace
    (by default 19, 38, 56, 75 sequences -> 152, 304, 448, 600 decode (seq, kv-head) units for
    8 KV heads, just above multiples of 148; `trace_decode_targets` sizes them for another SM
    count). A finished decode is replaced by a request whose
    prompt is already cached (a warm request); prompt chunks come from a FIFO of new requests.
    Every request has an id; `max_rows[id]` sizes its blocks in a persistent pool.
    """
    assert mix in ("a", "b")
    rng = random.Random(seed * 31 + (1 if mix == "a" else 2))

    def prompt_len():
        if mix == "a":
            return int(math.exp(rng.uniform(math.log(4096), math.log(32768))))
        sigma = 0.5
        mu = math.log(16384) - sigma * sigma / 2
        return int(min(32768, max(4096, rng.lognormvariate(mu, sigma))))

    def out_len():
        mean = 256 if mix == "a" else 64
        n = 1
        while rng.random() > 1.0 / mean:
            n += 1
        return n

    max_rows: List[int] = []
    decodes = []    # [request id, context length, tokens left]
    fifo = []       # [request id, prompt length, rows already prefilled]
    steps = []
    for it in range(iters):
        target = decode_targets[(it * len(decode_targets)) // iters]
        decodes = [d for d in decodes if d[2] > 0]
        while len(decodes) < target:
            n, o = prompt_len(), out_len()
            decodes.append([len(max_rows), n, o])
            max_rows.append(n + o)
        while len(fifo) < 4:
            n = prompt_len()
            fifo.append([len(max_rows), n, 0])
            max_rows.append(n)
        dec_lens, dec_ids = [], []
        for d in decodes:
            d[1] += 1                     # the new token's K/V is appended before attention
            d[2] -= 1
            dec_lens.append(d[1])
            dec_ids.append(d[0])
        left = budget - len(dec_lens)
        ql, pkv, pids = [], [], []
        for r in fifo:
            if left <= 0:
                break
            c = min(left, r[1] - r[2])
            if c <= 0:
                continue
            ql.append(c)
            pkv.append(r[2] + c)
            pids.append(r[0])
            r[2] += c
            left -= c
        fifo = [r for r in fifo if r[2] < r[1]]
        steps.append(TraceStep(ql, pkv, dec_lens, pids, dec_ids))
    return Trace(mix, steps, max_rows, tuple(decode_targets))


class TracePool:
    """One persistent paged K/V pool holding every request of a trace (Llama-3-8B shape:
    32 query / 8 KV heads), and the per-iteration batches over it.

    Each request owns ceil(max_rows/16) physical blocks taken in order from a random permutation
    of the pool; K and V are seeded N(0,1) bf16 (generated once on `device`). An iteration's
    batch references the pool's tensors (no copy) and adds its own block tables, lengths and
    seeded queries."""

    def __init__(self, tr: Trace, seed: int = 5, device="cpu", num_q_heads: int = 32,
                 num_kv_heads: int = 8):
        self.trace = tr
        self.Hq, self.Hkv = num_q_heads, num_kv_heads
        self.seed = seed
        self.device = torch.device(device)
        need = [_blocks(n) for n in tr.max_rows]
        nb = sum(need)
        g_cpu = torch.Generator().manual_seed(seed * 1_000_003 + 101)
        perm = torch.randperm(nb, generator=g_cpu)
        self.blocks = []
        pos = 0
        for n in need:
            self.blocks.append(perm[pos:pos + n].to(torch.int32))
            pos += n
        self.max_blocks = max(need)
        g = torch.Generator(device=self.device).manual_seed(seed * 1_000_003 + 103)
        shape = (nb, num_kv_heads, BLOCK_SIZE, HEAD_DIM)
        self.k_pool = torch.randn(*shape, generator=g, device=self.device).to(torch.bfloat16)
        self.v_pool = torch.randn(*shape, generator=g, device=self.device).to(torch.bfloat16)

    def batch(self, i: int) -> HybridBatch:
        st = self.trace.steps[i]
        rids = st.prefill_rids + st.decode_rids
        lens = st.prefill_kv_lens + st.decode_kv_lens
        maxb = max([1] + [_blocks(L) for L in lens])
        bt = torch.zeros((max(1, len(rids)), maxb), dtype=torch.int32)
        for r, (rid, L) in enumerate(zip(rids, lens)):
            n = _blocks(L)
            bt[r, :n] = self.blocks[rid][:n]
        if not rids:
            bt = bt[:0]
        g = torch.Generator(device=self.device).manual_seed(self.seed * 7919 + i)
        tp = sum(st.q_lens)
        q_p = torch.randn(tp, self.Hq, HEAD_DIM, generator=g, device=self.device).to(torch.bfloat16)
        q_d = torch.randn(len(st.decode_kv_lens), self.Hq, HEAD_DIM, generator=g,
                          device=self.device).to(torch.bfloat16)
        cu = [0]
        for n in st.q_lens:
            cu.append(cu[-1] + n)
        return HybridBatch(
            num_q_heads=self.Hq, num_kv_heads=self.Hkv, head_dim=HEAD_DIM, block_size=BLOCK_SIZE,
            q_lens=list(st.q_lens), prefill_kv_lens=list(st.prefill_kv_lens),
            decode_kv_lens=list(st.decode_kv_lens), scale=1.0 / math.sqrt(HEAD_DIM),
            q_prefill=q_p, q_decode=q_d, k_pool=self.k_pool, v_pool=self.v_pool,
            block_tables=bt.to(self.device),
            cu_seqlens_q=torch.tensor(cu, dtype=torch.int32, device=self.device),
            kv_lens=torch.tensor(lens, dtype=torch.int32, device=self.device), seed=self.seed,
            name=f"trace {self.trace.mix} iteration {i}")


# ----------------------------------------------------------------------------------------------
# FP8 (e4m3) KV cache for the decode-only FP8 path: K with one scale per kv-head and channel,
# V with one scale per cached token and kv-head (quantised from a seeded bf16 batch).
# ----------------------------------------------------------------------------------------------

@dataclass
class Fp8DecodeBatch:
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    decode_kv_lens: List[int]
    scale: float
    q_decode: torch.Tensor          # bf16 [Nd][Hq][D]
    k8: torch.Tensor                # uint8 e4m3 [NB][Hkv][16][D]
    v8: torch.Tensor                # uint8 e4m3 [NB][Hkv][16][D]
    k_scale: torch.Tensor           # fp32 [Hkv][D]
    v_scale: torch.Tensor           # fp32 [NB][Hkv][16]
    block_tables: torch.Tensor      # int32 [Nd][max_blocks_per_seq]
    kv_lens: torch.Tensor           # int32 [Nd]
    seed: int = 0

    @property
    def num_decode_seqs(self) -> int:
        return len(self.decode_kv_lens)

    @property
    def num_blocks(self) -> int:
        return int(self.k8.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    def to(self, device) -> "Fp8DecodeBatch":
        kw = dict(self.__dict__)
        for k, v in list(kw.items()):
            if isinstance(v, torch.Tensor):
                kw[k] = v.to(device)
        return Fp8DecodeBatch(**kw)


def make_fp8_decode_batch(num_q_heads: int, num_kv_heads: int, decode_kv_lens: Sequence[int],
                          seed: int, device="cpu", pow2_scales: bool = False) -> Fp8DecodeBatch:
    """Quantise the pools of a seeded bf16 decode batch to e4m3: k_scale = max |K| over the
    finite cached rows of each (kv-head, channel) / 448, v_scale = max |V| over each row / 448
    (1 where that max is 0 or the row is poison), values rounded to nearest e4m3 by torch's
    float8 conversion. NaN-poisoned rows stay NaN. With pow2_scales every scale is rounded up to
    a power of two, so each dequantised value is exactly a bf16 value."""
    b = make_batch(num_q_heads, num_kv_heads, [], [], list(decode_kv_lens), seed=seed,
                   device=device)
    k = b.k_pool.float()
    v = b.v_pool.float()
    fk = torch.nan_to_num(k.abs(), nan=0.0)
    ks = fk.amax(dim=(0, 2)) / 448.0                          # [Hkv][D]
    vs = torch.nan_to_num(v.abs(), nan=0.0).amax(dim=3) / 448.0   # [NB][Hkv][16]
    ks = torch.where(ks > 0, ks, torch.ones_like(ks))
    vs = torch.where(vs > 0, vs, torch.ones_like(vs))
    if pow2_scales:
        ks = torch.exp2(torch.ceil(torch.log2(ks)))
        vs = torch.exp2(torch.ceil(torch.log2(vs)))
    k8 = (k / ks[None, :, None, :]).to(torch.float8_e4m3fn).view(torch.uint8)
    v8 = (v / vs[..., None]).to(torch.float8_e4m3fn).view(torch.uint8)
    return Fp8DecodeBatch(num_q_heads, num_kv_heads, b.head_dim, b.block_size,
                          list(decode_kv_lens), b.scale, b.q_decode, k8.contiguous(),
                          v8.contiguous(), ks.float().contiguous(), vs.float().contiguous(),
                          b.block_tables, b.kv_lens, seed=seed)


def fp8_append_case(num_q_heads: int, num_kv_heads: int, decode_kv_lens: Sequence[int],
                    seed: int, device="cpu"):
    """An FP8 decode batch whose newest row (position kv_len - 1) of every decode sequence and
    kv-head is missing from the cache (K and V bytes 0x7F = e4m3 NaN, V scale NaN), plus those
    rows in bf16 ([Nd][Hkv][D], the seeded batch's own values) to append. The K scales are those
    of the whole pool, new rows included, as a serving stack that fixed them earlier would have.
    Returns (batch, k_new, v_new)."""
    b = make_batch(num_q_heads, num_kv_heads, [], [], list(decode_kv_lens), seed=seed,
                   device=device)
    fb = make_fp8_decode_batch(num_q_heads, num_kv_heads, decode_kv_lens, seed=seed,
                               device=device)
    Nd, Hkv, D = len(decode_kv_lens), num_kv_heads, b.head_dim
    k_new = torch.empty((Nd, Hkv, D), dtype=torch.bfloat16, device=device)
    v_new = torch.empty_like(k_new)
    for d, L in enumerate(decode_kv_lens):
        pos = L - 1
        phys = int(b.block_tables[d, pos // 16])
        k_new[d] = b.k_pool[phys, :, pos % 16]
        v_new[d] = b.v_pool[phys, :, pos % 16]
        fb.k8[phys, :, pos % 16] = 0x7F
        fb.v8[phys, :, pos % 16] = 0x7F
        fb.v_scale[phys, :, pos % 16] = float("nan")
    return fb, k_new, v_new


def dequantised_batch(fb: Fp8DecodeBatch) -> HybridBatch:
    """The bf16 decode batch holding the dequantised cache e4m3(bits) * scale, rounded to bf16
    (exact when the scales are powers of two)."""
    k = fb.k8.view(torch.float8_e4m3fn).float() * fb.k_scale[None, :, None, :]
    v = fb.v8.view(torch.float8_e4m3fn).float() * fb.v_scale[..., None]
    dev = fb.q_decode.device
    return HybridBatch(
        num_q_heads=fb.num_q_heads, num_kv_heads=fb.num_kv_heads, head_dim=fb.head_dim,
        block_size=fb.block_size, q_lens=[], prefill_kv_lens=[],
        decode_kv_lens=list(fb.decode_kv_lens), scale=fb.scale,
        q_prefill=torch.zeros((0, fb.num_q_heads, fb.head_dim), dtype=torch.bfloat16, device=dev),
        q_decode=fb.q_decode, k_pool=k.to(torch.bfloat16), v_pool=v.to(torch.bfloat16),
        block_tables=fb.block_tables, cu_seqlens_q=torch.zeros((1,), dtype=torch.int32, device=dev),
        kv_lens=fb.kv_lens, seed=fb.seed)
