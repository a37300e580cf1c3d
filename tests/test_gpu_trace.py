"""GPU parity on the 200-iteration hybrid-batching trace (Llama-3-8B shape, persistent paged
pool): selected iterations of both mixes (every quarter's first and last, two inside) run
through the fused kernel exactly as the benchmark runs them; sampled outputs are checked against
the fp64 oracle row by row.

The oracle gets a compact CPU copy holding only the blocks of the sampled sequences (with the
block tables renumbered), so a check needs a few hundred MB instead of the whole pool.
"""
import random

import numpy as np
import pytest
import torch

import oracle
from hybrid_prefill_decode_gb300 import binding as B
from hybrid_prefill_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ATOL = 2e-2
RTOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _compact(batch, seqs):
    """A CPU HybridBatch with only sequences `seqs` (indices into the batch's rows, prefill
    rows first) and their blocks. Returns (batch, map from old prefill token -> new token)."""
    np_ = batch.num_prefill_seqs
    pre = [s for s in seqs if s < np_]
    dec = [s - np_ for s in seqs if s >= np_]
    lens = batch.host_kv_lens
    rows = pre + [np_ + d for d in dec]
    bt_old = batch.block_tables.cpu()
    blocks, new_rows = [], []
    nblk = 0
    for r in rows:
        n = (lens[r] + 15) // 16
        blocks.append(bt_old[r, :n].long())
        new_rows.append(list(range(nblk, nblk + n)))
        nblk += n
    ids = torch.cat(blocks)
    k = batch.k_pool[ids.to(batch.k_pool.device)].cpu()
    v = batch.v_pool[ids.to(batch.v_pool.device)].cpu()
    maxb = max(len(x) for x in new_rows)
    bt = torch.zeros((len(rows), maxb), dtype=torch.int32)
    for i, x in enumerate(new_rows):
        bt[i, :len(x)] = torch.tensor(x, dtype=torch.int32)
    cu_old = batch.host_cu_seqlens
    q_lens = [batch.q_lens[s] for s in pre]
    tok_map = {}
    qp = []
    pos = 0
    for s in pre:
        for t in range(cu_old[s], cu_old[s + 1]):
            tok_map[t] = pos
            pos += 1
        qp.append(batch.q_prefill[cu_old[s]:cu_old[s + 1]].cpu())
    cu = [0]
    for n in q_lens:
        cu.append(cu[-1] + n)
    qd = batch.q_decode[torch.tensor(dec, dtype=torch.long, device=batch.q_decode.device)].cpu() \
        if dec else batch.q_decode[:0].cpu()
    small = W.HybridBatch(
        num_q_heads=batch.num_q_heads, num_kv_heads=batch.num_kv_heads, head_dim=128,
        block_size=16, q_lens=q_lens, prefill_kv_lens=[lens[s] for s in pre],
        decode_kv_lens=[lens[np_ + d] for d in dec], scale=batch.scale,
        q_prefill=torch.cat(qp) if qp else batch.q_prefill[:0].cpu(), q_decode=qd,
        k_pool=k, v_pool=v, block_tables=bt, cu_seqlens_q=torch.tensor(cu, dtype=torch.int32),
        kv_lens=torch.tensor([lens[r] for r in rows], dtype=torch.int32))
    return small, tok_map, dec


@pytest.fixture(scope="module", params=["a", "b"])
def pool(request):
    # decode counts sized from this device's SM count, as the benchmark sizes them
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tr = W.trace(request.param, decode_targets=W.trace_decode_targets(sms))
    return W.TracePool(tr, device="cuda")


# the first and last iterations of each quarter (each holds a different decode count) and two
# inside them
@pytest.mark.parametrize("it", [0, 25, 49, 50, 77, 99, 100, 149, 150, 199])
def test_trace_iteration_sampled(pool, it):
    b = pool.batch(it)
    o_p, o_d = B.hybrid_attention(b, variant="fused")
    torch.cuda.synchronize()
    assert torch.isfinite(o_p.float()).all() and torch.isfinite(o_d.float()).all()
    rng = random.Random(it)
    np_ = b.num_prefill_seqs
    dec_pick = sorted(rng.sample(range(b.num_decode_seqs), min(6, b.num_decode_seqs)))
    seqs = list(range(np_)) + [np_ + d for d in dec_pick]
    small, tok_map, dec = _compact(b, seqs)
    Hq = b.num_q_heads
    cu = b.host_cu_seqlens
    prow = []
    for s in range(np_):
        q = b.q_lens[s]
        cand = {cu[s], cu[s] + q - 1} | set(range(cu[s], cu[s] + q, 97))
        cand |= {cu[s] + t for t in range(127, q, 128)} | {cu[s] + t for t in range(128, q, 128)}
        prow += sorted(cand)
    kinds = [0] * (len(prow) * Hq) + [1] * (len(dec) * Hq)
    idx = [tok_map[r] for r in prow for _ in range(Hq)] + [i for i in range(len(dec))
                                                           for _ in range(Hq)]
    heads = list(range(Hq)) * (len(prow) + len(dec))
    ref = oracle.rows(small, kinds, idx, heads)
    gp, gd = o_p.float().cpu(), o_d.float().cpu()
    got = torch.stack([gp[r, h] for r in prow for h in range(Hq)] +
                      [gd[d, h] for d in dec for h in range(Hq)]).numpy().astype(np.float64)
    err = np.abs(got - ref)
    assert (err <= ATOL + RTOL * np.abs(ref)).all(), float(err.max())
