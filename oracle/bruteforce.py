"""NumPy brute force of hybrid prefill+decode attention — TEST INFRASTRUCTURE ONLY.

An implementation independent of ``oracle.c``, for tiny cases: for each sequence it first
gathers the sequence's K and V rows into contiguous arrays through the block table
("Week 6: Beyond PyTorch: Custom Kernel과 vLLM", §"PagedAttention"), then forms the whole
[q_len x kv_len] score matrix, applies the causal mask with an explicit position comparison
unless the batch is non-causal (§"Non-Causal vs. Causal Attention"; chunk tokens sit after the
cached prefix,
§"한 스텝에 여러 종류의 request 섞기"), and takes a row softmax and a matrix product
(§"Attention에 적용하기"). Everything is float64.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def _gather(pool: np.ndarray, bt_row: np.ndarray, n: int, g: int) -> np.ndarray:
    """Rows 0..n-1 of kv-head g of one sequence, as a contiguous [n][D] array."""
    bs = pool.shape[2]
    rows = [pool[bt_row[j // bs], g, j % bs, :] for j in range(n)]
    return np.stack(rows, axis=0) if rows else np.zeros((0, pool.shape[3]))


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos: np.ndarray,
              scale: float, causal: bool = True) -> np.ndarray:
    """Attention of query rows q[t] at absolute positions q_pos[t] over keys 0..n-1, masked
    (causal: key j visible iff j <= p) or not (every key visible)."""
    n = k.shape[0]
    s = scale * (q @ k.T)                                   # [t][n]
    if causal:
        key_pos = np.arange(n)[None, :]
        s = np.where(key_pos <= q_pos[:, None], s, -np.inf)
    s = s - s.max(axis=1, keepdims=True)
    w = np.exp(s)
    w = w / w.sum(axis=1, keepdims=True)
    return w @ v


def hybrid_attention(batch):
    """(o_prefill [Tp][Hq][D], o_decode [Nd][Hq][D]) as float64, from a HybridBatch-like object
    whose tensors are bf16 torch tensors or uint16 numpy arrays of bf16 bits."""
    def f64(a):
        if isinstance(a, np.ndarray):
            return bf16_bits_to_f64(a)
        import torch
        return bf16_bits_to_f64(a.detach().cpu().contiguous().view(torch.int16).numpy()
                                .view(np.uint16))

    def i32(a):
        return np.asarray(a if isinstance(a, np.ndarray) else a.cpu().numpy(), dtype=np.int64)

    Hq, Hkv = int(batch.num_q_heads), int(batch.num_kv_heads)
    group = Hq // Hkv
    Np, Nd = int(batch.num_prefill_seqs), int(batch.num_decode_seqs)
    qp, qd = f64(batch.q_prefill), f64(batch.q_decode)
    kp, vp = f64(batch.k_pool), f64(batch.v_pool)
    bt, cu, kvl = i32(batch.block_tables), i32(batch.cu_seqlens_q), i32(batch.kv_lens)
    D = kp.shape[3]
    tp = int(cu[-1]) if Np > 0 else 0
    o_p = np.zeros((tp, Hq, D))
    o_d = np.zeros((Nd, Hq, D))
    for s in range(Np):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        L = int(kvl[s])
        pos = np.arange(L - (t1 - t0), L)            # absolute positions of the chunk tokens
        for h in range(Hq):
            g = h // group
            K, V = _gather(kp, bt[s], L, g), _gather(vp, bt[s], L, g)
            o_p[t0:t1, h, :] = attention(qp[t0:t1, h, :], K, V, pos, float(batch.scale),
                                         causal=getattr(batch, "causal", True))
    for d in range(Nd):
        s = Np + d
        L = int(kvl[s])
        for h in range(Hq):
            g = h // group
            K, V = _gather(kp, bt[s], L, g), _gather(vp, bt[s], L, g)
            o_d[d, h, :] = attention(qd[d:d + 1, h, :], K, V, np.array([L - 1]),
                                     float(batch.scale))[0]
    return o_p, o_d
