"""Algorithmic work of a hybrid batch and its roofline (host arithmetic, no GPU).

Roofline ("Week 6: Beyond PyTorch: Custom Kernel과 vLLM", §"보충: Roofline을 수식으로
정리하기"): T_math = FLOPs / peak FLOP/s, T_mem = bytes / peak bandwidth, T >= max of the two.
For one hybrid iteration the bound is

    T* = max((B_prefill + B_decode) / BW,  F_prefill / P_bf16)

with algorithmic work only (what the method must move or compute):

  * K/V bytes per cached row: 2 (K and V) x Hkv x d x 2 bytes (bf16) — the K/V-cache size rule
    of §"PagedAttention" for one layer;
  * B_prefill = sum over chunks (P + C) x row bytes   (each kv-head's rows read once)
              + 2 x C x Hq x d x 2                   (Q read, O written);
  * B_decode  = sum over decodes L x row bytes + 2 x Nd x Hq x d x 2;
  * F_prefill = 4 x d x Hq x (C x P + C (C + 1) / 2): QKᵀ and PV are 2 x d FLOPs each per visible
    (query, key) pair (§"행렬곱의 FLOPs 세는 법": a length-d dot product is 2d FLOPs), and
    causally masked pairs are not counted;
  * decode FLOPs (4 x d x Hq x L per sequence) run on the CUDA cores and are reported only;
    decode attention stays memory-bound whatever the batch (§"예외: attention은 배치로도 구제되지
    않는다").
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Sequence


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, dtype_bytes: int) -> int:
    """K/V-cache bytes one token occupies: 2 x layers x kv_heads x head_dim x dtype_bytes."""
    return 2 * layers * kv_heads * head_dim * dtype_bytes


@dataclass
class Work:
    prefill_flops: float
    prefill_bytes: float
    decode_bytes: float
    decode_flops: float

    @property
    def bytes(self) -> float:
        return self.prefill_bytes + self.decode_bytes

    def t_star(self, hbm_gbs: float, tflops: float) -> float:
        """Hybrid roofline lower bound in seconds."""
        return max(self.bytes / (hbm_gbs * 1e9), self.prefill_flops / (tflops * 1e12))

    def bound(self, hbm_gbs: float, tflops: float) -> str:
        return ("hbm" if self.bytes / (hbm_gbs * 1e9) >= self.prefill_flops / (tflops * 1e12)
                else "tensor")


def batch_work(num_q_heads: int, num_kv_heads: int, q_lens: Sequence[int],
               prefill_kv_lens: Sequence[int], decode_kv_lens: Sequence[int],
               head_dim: int = 128, causal: bool = True) -> Work:
    """Algorithmic FLOPs and bytes of one hybrid batch (see the module docstring); with
    causal=False every chunk token pairs with every row of its sequence."""
    d, Hq, Hkv = head_dim, num_q_heads, num_kv_heads
    row = kv_bytes_per_token(1, Hkv, d, 2)
    pf = pb = 0.0
    for C, L in zip(q_lens, prefill_kv_lens):
        P = L - C
        pairs = C * P + C * (C + 1) // 2 if causal else C * L
        pf += 4.0 * d * Hq * pairs
        pb += float(L) * row + 2.0 * C * Hq * d * 2
    db = sum(float(L) * row for L in decode_kv_lens) + 2.0 * len(decode_kv_lens) * Hq * d * 2
    df = sum(4.0 * d * Hq * L for L in decode_kv_lens)
    return Work(pf, pb, db, df)


def fp8_decode_bytes(num_q_heads: int, num_kv_heads: int, decode_kv_lens: Sequence[int],
                     head_dim: int = 128) -> float:
    """Algorithmic bytes of decode attention over an e4m3 cache: one byte per K and V value, a
    4-byte V scale per cached (row, kv-head), the [Hkv][d] fp32 K scales, and the bf16 queries
    read and outputs written."""
    d, Hq, Hkv = head_dim, num_q_heads, num_kv_heads
    rows = float(sum(decode_kv_lens)) * Hkv
    return rows * (2 * d + 4) + Hkv * d * 4 + 2.0 * len(decode_kv_lens) * Hq * d * 2
