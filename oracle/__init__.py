"""fp64 CPU oracle of hybrid prefill+decode attention — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import this package. The product (``hybrid_prefill_decode_gb300``) never
imports it, and this package imports nothing from the product.

Two independent implementations live here:

* ``oracle.c`` (compiled with gcc, OpenMP): gather through the block table, fp64 scores,
  3-pass safe softmax, weighted sum — "Week 6: Beyond PyTorch: Custom Kernel과 vLLM",
  §"Attention에 적용하기", §"Safe softmax (3-pass, 수치 안정성 확보)", §"PagedAttention",
  §"한 스텝에 여러 종류의 request 섞기"; split-KV partials and their exact merge —
  "LLMSO - W4 - Optimization & Frameworks", §"FlashDecoding — decode 단계의 병렬성 확보".
* ``bruteforce.py`` (NumPy): the full masked score matrix of each sequence, for tiny cases.

Inputs are the bf16 tensors of a batch (passed as uint16 bit patterns); results are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library next to it (plain gcc, -O2, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            L = ctypes.c_int64
            D = ctypes.c_double
            lib.oracle_num_threads.restype = I
            lib.oracle_attend_range.restype = I
            lib.oracle_attend_range.argtypes = [P, P, L, L, I, I, I, I, P, P, L, D, P, P, P, P]
            lib.oracle_merge.restype = None
            lib.oracle_merge.argtypes = [I, P, P, P, I, P]
            lib.oracle_attend_row.restype = I
            lib.oracle_attend_row.argtypes = [P, P, L, I, I, I, I, P, P, L, D, P, P]
            lib.oracle_rows.restype = I
            lib.oracle_rows.argtypes = [I, I, I, I, I, I, L, I, D, P, P, P, P, P, P, P,
                                        L, P, P, P, P, I]
            lib.oracle_hybrid_attention.restype = I
            lib.oracle_hybrid_attention.argtypes = [I, I, I, I, I, I, L, I, D, P, P, P, P,
                                                    P, P, P, P, P, I]
            lib.oracle_e4m3_to_double.restype = D
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_decode_fp8.restype = I
            lib.oracle_decode_fp8.argtypes = [I, I, I, I, I, L, I, D, P, P, P, P, P, P, P, P]
            lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
            lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
            lib.oracle_append_fp8.restype = I
            lib.oracle_append_fp8.argtypes = [I, I, I, I, L, I, P, P, P, P, P, P, P, P]
            lib.oracle_append_bf16.restype = I
            lib.oracle_append_bf16.argtypes = [I, I, I, I, I, L, I, P, P, P, P, P, P, P]
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the C oracle uses on this host."""
    return int(_load().oracle_num_threads())


def _u16(a) -> np.ndarray:
    """bf16 tensor (torch) or uint16 array -> contiguous uint16 numpy array of the bit patterns."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint16
        return np.ascontiguousarray(a)
    import torch  # the generators hand out torch tensors; only their bits are used here
    assert a.dtype == torch.bfloat16, a.dtype
    return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy()
                                .view(np.uint16))


def _i32(a) -> np.ndarray:
    if isinstance(a, np.ndarray):
        return np.ascontiguousarray(a, dtype=np.int32)
    return np.ascontiguousarray(a.detach().cpu().numpy(), dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class _Batch:
    """The arrays of a hybrid batch in the form the C oracle reads."""

    def __init__(self, b):
        self.Hq, self.Hkv = int(b.num_q_heads), int(b.num_kv_heads)
        self.D, self.BS = int(b.head_dim), int(b.block_size)
        self.Np, self.Nd = int(b.num_prefill_seqs), int(b.num_decode_seqs)
        self.scale = float(b.scale)
        self.q_prefill = _u16(b.q_prefill)
        self.q_decode = _u16(b.q_decode)
        self.k_pool = _u16(b.k_pool)
        self.v_pool = _u16(b.v_pool)
        self.block_tables = _i32(b.block_tables)
        self.cu = _i32(b.cu_seqlens_q)
        self.kv_lens = _i32(b.kv_lens)
        self.num_blocks = int(self.k_pool.shape[0])
        self.maxb = int(self.block_tables.shape[1]) if self.block_tables.ndim == 2 else 0
        self.tp = int(self.cu[-1]) if self.Np > 0 else 0
        self.causal = 1 if getattr(b, "causal", True) else 0

    def common(self):
        return (self.Hq, self.Hkv, self.D, self.BS, self.Np, self.Nd, self.num_blocks,
                self.maxb, self.scale, _ptr(self.q_prefill), _ptr(self.q_decode),
                _ptr(self.k_pool), _ptr(self.v_pool), _ptr(self.block_tables),
                _ptr(self.cu), _ptr(self.kv_lens))


def hybrid_attention(batch):
    """All outputs of a hybrid batch: (o_prefill [Tp][Hq][D], o_decode [Nd][Hq][D]), float64.

    ``batch`` is any object with the fields of ``hybrid_prefill_decode_gb300.workloads
    .HybridBatch`` (shapes, bf16 tensors, int32 tables)."""
    b = _Batch(batch)
    o_p = np.zeros((b.tp, b.Hq, b.D), dtype=np.float64)
    o_d = np.zeros((b.Nd, b.Hq, b.D), dtype=np.float64)
    rc = _load().oracle_hybrid_attention(*b.common(), _ptr(o_p), _ptr(o_d), b.causal)
    if rc != 0:
        raise ValueError(f"oracle_hybrid_attention failed with code {rc}")
    return o_p, o_d


def rows(batch, kinds, indices, heads) -> np.ndarray:
    """Selected output rows [n][D] (float64): kind 0 = prefill token index, 1 = decode seq."""
    b = _Batch(batch)
    kinds = np.ascontiguousarray(kinds, dtype=np.int32)
    indices = np.ascontiguousarray(indices, dtype=np.int64)
    heads = np.ascontiguousarray(heads, dtype=np.int32)
    n = int(kinds.shape[0])
    out = np.zeros((n, b.D), dtype=np.float64)
    rc = _load().oracle_rows(*b.common(), n, _ptr(kinds), _ptr(indices), _ptr(heads),
                             _ptr(out), b.causal)
    if rc != 0:
        raise ValueError(f"oracle_rows failed with code {rc}")
    return out


def attend_range(q_row, bt_row, j0, j1, kv_head, batch_like):
    """Split-KV partial state (m, l, o_unnormalised[D]) of one query over keys [j0, j1)."""
    lib = _load()
    q = _u16(q_row)
    bt = _i32(bt_row)
    kp, vp = _u16(batch_like.k_pool), _u16(batch_like.v_pool)
    D = int(q.shape[-1])
    o = np.zeros(D, dtype=np.float64)
    x = np.zeros(max(1, j1 - j0), dtype=np.float64)
    m = ctypes.c_double()
    l = ctypes.c_double()
    rc = lib.oracle_attend_range(_ptr(q), _ptr(bt), j0, j1, kv_head,
                                 int(batch_like.num_kv_heads), D, int(batch_like.block_size),
                                 _ptr(kp), _ptr(vp), int(kp.shape[0]),
                                 float(batch_like.scale), ctypes.byref(m), ctypes.byref(l),
                                 _ptr(o), _ptr(x))
    if rc != 0:
        raise ValueError(f"oracle_attend_range failed with code {rc}")
    return m.value, l.value, o


def merge(ms, ls, os_) -> np.ndarray:
    """Exact merge of split partials (m_i, l_i, o_i) into the normalised output row."""
    ms = np.ascontiguousarray(ms, dtype=np.float64)
    ls = np.ascontiguousarray(ls, dtype=np.float64)
    os_ = np.ascontiguousarray(os_, dtype=np.float64)
    n, D = os_.shape
    out = np.zeros(D, dtype=np.float64)
    _load().oracle_merge(n, _ptr(ms), _ptr(ls), _ptr(os_), D, _ptr(out))
    return out


def e4m3_to_double(bits: int) -> float:
    """The value of one e4m3 bit pattern (see oracle.c)."""
    return float(_load().oracle_e4m3_to_double(int(bits) & 0xFF))


def e4m3_from_float(x) -> int:
    """The e4m3 code of a float32 value (round to nearest even, saturating; see oracle.c)."""
    return int(_load().oracle_e4m3_from_float(float(x)))


def append_bf16(batch, k_new, v_new, k_pool=None, v_pool=None):
    """The bf16 pools after appending the iteration's new tokens (rows of k_new / v_new
    [T_p + Nd][Hkv][D]: the prefill chunks' tokens in order, then one per decode sequence) to
    ``batch`` (a ``HybridBatch``; its lengths and block tables say where each row goes). Starts
    from ``k_pool`` / ``v_pool`` when given, else from the batch's pools; returns new
    (k_pool, v_pool) numpy uint16 arrays; the inputs are not modified."""
    kp = np.array(_u16(batch.k_pool if k_pool is None else k_pool), copy=True)
    vp = np.array(_u16(batch.v_pool if v_pool is None else v_pool), copy=True)
    kn, vn = _u16(k_new), _u16(v_new)
    bt = _i32(batch.block_tables)
    cu = _i32(batch.cu_seqlens_q)
    kv = _i32(batch.kv_lens)
    rc = _load().oracle_append_bf16(int(batch.num_kv_heads), int(batch.head_dim),
                                    int(batch.block_size), int(batch.num_prefill_seqs),
                                    int(batch.num_decode_seqs), int(kp.shape[0]),
                                    int(bt.shape[1]) if bt.ndim == 2 else 0, _ptr(cu), _ptr(kv),
                                    _ptr(bt), _ptr(kn), _ptr(vn), _ptr(kp), _ptr(vp))
    if rc != 0:
        raise ValueError(f"oracle_append_bf16 failed with code {rc}")
    return kp, vp


def append_fp8(batch, k_new, v_new):
    """The FP8 cache of ``batch`` (an ``Fp8DecodeBatch``) after appending one token per decode
    sequence (rows of bf16 k_new / v_new [Nd][Hkv][D]) at position kv_len - 1: returns new
    (k8, v8, v_scale) numpy arrays; the inputs are not modified."""
    k8 = np.array(batch.k8.cpu().numpy(), dtype=np.uint8, copy=True)
    v8 = np.array(batch.v8.cpu().numpy(), dtype=np.uint8, copy=True)
    vs = np.array(batch.v_scale.cpu().numpy(), dtype=np.float32, copy=True)
    ks = np.ascontiguousarray(batch.k_scale.cpu().numpy(), dtype=np.float32)
    kn, vn = _u16(k_new), _u16(v_new)
    bt = _i32(batch.block_tables)
    kv = _i32(batch.kv_lens)
    Nd = int(kv.shape[0])
    rc = _load().oracle_append_fp8(int(batch.num_kv_heads), int(batch.head_dim),
                                   int(batch.block_size), Nd, int(k8.shape[0]),
                                   int(bt.shape[1]) if bt.ndim == 2 else 0, _ptr(kn), _ptr(vn),
                                   _ptr(ks), _ptr(bt), _ptr(kv), _ptr(k8), _ptr(v8), _ptr(vs))
    if rc != 0:
        raise ValueError(f"oracle_append_fp8 failed with code {rc}")
    return k8, v8, vs


def decode_fp8(batch):
    """Decode outputs [Nd][Hq][D] (float64) over an FP8 cache. ``batch`` has the fields of
    ``hybrid_prefill_decode_gb300.workloads.Fp8DecodeBatch`` (q_decode bf16, k8 / v8 uint8
    pools, k_scale [Hkv][D] and v_scale [NB][Hkv][16] float32, block tables and kv lengths of
    the decode sequences)."""
    q = _u16(batch.q_decode)
    k8 = np.ascontiguousarray(batch.k8.cpu().numpy(), dtype=np.uint8)
    v8 = np.ascontiguousarray(batch.v8.cpu().numpy(), dtype=np.uint8)
    ks = np.ascontiguousarray(batch.k_scale.cpu().numpy(), dtype=np.float32)
    vs = np.ascontiguousarray(batch.v_scale.cpu().numpy(), dtype=np.float32)
    bt = _i32(batch.block_tables)
    kv = _i32(batch.kv_lens)
    Nd, Hq, D = int(q.shape[0]), int(batch.num_q_heads), int(batch.head_dim)
    out = np.zeros((Nd, Hq, D), dtype=np.float64)
    rc = _load().oracle_decode_fp8(Hq, int(batch.num_kv_heads), D, int(batch.block_size), Nd,
                                   int(k8.shape[0]), int(bt.shape[1]) if bt.ndim == 2 else 0,
                                   float(batch.scale), _ptr(q), _ptr(k8), _ptr(v8), _ptr(ks),
                                   _ptr(vs), _ptr(bt), _ptr(kv), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_decode_fp8 failed with code {rc}")
    return out
