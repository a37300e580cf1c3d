"""Thin ctypes binding of the C ABI in ``include/pod_attn.h`` (argument marshalling only).

Every step of the computation runs in the CUDA kernels of ``libpod_attn.so``; this module only
converts Python/torch arguments to pointers and sizes. There is no fallback: if the library has
not been built, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libpod_attn.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "pod_attn.h")

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_WORKSPACE = -3
ERR_CUDA = -4
ERR_BAD_INDEX = -5
ERR_TIMEOUT = -6

VARIANTS = {"fused": 0, "serial": 1, "streams": 2}


class Problem(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_prefill_seqs", ctypes.c_int32), ("num_prefill_tokens", ctypes.c_int32),
                ("num_decode_seqs", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("scale", ctypes.c_float)]


class Options(ctypes.Structure):
    _fields_ = [("num_sms", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32),
                ("max_prefill_ctas", ctypes.c_int32), ("decode_splits", ctypes.c_int32),
                ("prefill_splits", ctypes.c_int32), ("instrument", ctypes.c_int32),
                ("variant", ctypes.c_int32), ("non_causal", ctypes.c_int32),
                ("kv_fp8", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("num_prefill_items", ctypes.c_int32), ("num_decode_items", ctypes.c_int32),
                ("num_units", ctypes.c_int32), ("num_sms", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32), ("max_prefill_ctas", ctypes.c_int32),
                ("grid_fused", ctypes.c_int32), ("grid_prefill", ctypes.c_int32),
                ("grid_decode", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("threads_per_cta", ctypes.c_int32), ("item_words", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_uint64), ("est_prefill_flops", ctypes.c_double),
                ("est_prefill_bytes", ctypes.c_double), ("est_decode_bytes", ctypes.c_double),
                ("est_decode_flops", ctypes.c_double)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class Bucket(ctypes.Structure):
    _fields_ = [("prefill_flops", ctypes.c_int64), ("read_bytes", ctypes.c_int64),
                ("prefill_ctas", ctypes.c_int32), ("decode_ctas", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("smem_per_cta", ctypes.c_int32),
                ("tmem_cols_per_cta", ctypes.c_int32), ("bucket_flops", ctypes.c_int32),
                ("bucket_bytes", ctypes.c_int32), ("bucket_ctas", ctypes.c_int32),
                ("intensity", ctypes.c_double)]


class ItemRecord(ctypes.Structure):
    _fields_ = [("smid", ctypes.c_int32), ("kind", ctypes.c_int32), ("item", ctypes.c_int32),
                ("cta", ctypes.c_int32), ("t_start", ctypes.c_uint64),
                ("t_end", ctypes.c_uint64)]


_lib = None


def declared_functions() -> list:
    """Names of the functions include/pod_attn.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pod_attn_[a-z_]+)\s*\(", text)))


def load():
    """Load libpod_attn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    lib.pod_attn_plan.restype = I32
    lib.pod_attn_plan.argtypes = [ctypes.POINTER(Problem), P, P, ctypes.POINTER(Options),
                                  ctypes.POINTER(P)]
    lib.pod_attn_workspace_bytes.restype = SZ
    lib.pod_attn_workspace_bytes.argtypes = [P]
    lib.pod_attn_upload.restype = I32
    lib.pod_attn_upload.argtypes = [P, P, SZ, P]
    lib.pod_attn_run.restype = I32
    lib.pod_attn_run.argtypes = [P, P, P, P, P, P, P, P, P, P, P, SZ, P, P]
    lib.pod_attn_run_decode_fp8.restype = I32
    lib.pod_attn_run_decode_fp8.argtypes = [P, P, P, P, P, P, P, P, P, P, SZ, P]
    lib.pod_attn_append_fp8.restype = I32
    lib.pod_attn_append_fp8.argtypes = [P, P, P, P, P, P, P, P, P, SZ, P]
    lib.pod_attn_plan_bucket.restype = I32
    lib.pod_attn_plan_bucket.argtypes = [P, ctypes.POINTER(Bucket)]
    lib.pod_attn_run_append.restype = I32
    lib.pod_attn_run_append.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P, P]
    lib.pod_attn_last_device_status.restype = I32
    lib.pod_attn_last_device_status.argtypes = [P, P, P]
    lib.pod_attn_get_plan_info.restype = I32
    lib.pod_attn_get_plan_info.argtypes = [P, ctypes.POINTER(PlanInfo)]
    lib.pod_attn_plan_items.restype = I32
    lib.pod_attn_plan_items.argtypes = [P, P, SZ, ctypes.POINTER(SZ)]
    lib.pod_attn_read_records.restype = I32
    lib.pod_attn_read_records.argtypes = [P, P, P, SZ, ctypes.POINTER(SZ), P]
    lib.pod_attn_plan_destroy.restype = None
    lib.pod_attn_plan_destroy.argtypes = [P]
    lib.pod_attn_status_string.restype = ctypes.c_char_p
    lib.pod_attn_status_string.argtypes = [I32]
    lib.pod_attn_selftest_timeout.restype = I32
    lib.pod_attn_selftest_timeout.argtypes = [P, I32, P]
    _lib = lib
    return lib


class PodAttnError(RuntimeError):
    def __init__(self, code, where):
        super().__init__(f"{where}: {load().pod_attn_status_string(code).decode()} ({code})")
        self.code = code


def _check(code, where):
    if code != OK:
        raise PodAttnError(code, where)


def _i32_array(values: Sequence[int]):
    arr = (ctypes.c_int32 * max(1, len(values)))(*values)
    return arr


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if t.numel() == 0:
        return None
    assert t.is_contiguous()
    return t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


class Plan:
    """A planned hybrid batch (host side). Mirrors pod_attn_plan / pod_attn_plan_destroy."""

    def __init__(self, num_q_heads: int, num_kv_heads: int, cu_seqlens: Sequence[int],
                 kv_lens: Sequence[int], num_decode_seqs: int, num_blocks: int,
                 max_blocks_per_seq: int, scale: float, variant: str = "fused",
                 num_sms: int = 0, ctas_per_sm: int = 0, max_prefill_ctas: int = 0,
                 decode_splits: int = 0, prefill_splits: int = 0, instrument: bool = False,
                 non_causal: bool = False, head_dim: int = 128, kv_fp8: bool = False):
        lib = load()
        np_ = len(cu_seqlens) - 1 if len(cu_seqlens) > 0 else 0
        self.problem = Problem(num_q_heads, num_kv_heads, head_dim, 16, np_,
                               int(cu_seqlens[-1]) if np_ > 0 else 0, num_decode_seqs,
                               num_blocks, max_blocks_per_seq, scale)
        self.options = Options(num_sms, ctas_per_sm, max_prefill_ctas, decode_splits,
                               prefill_splits, 1 if instrument else 0, VARIANTS[variant],
                               1 if non_causal else 0, 1 if kv_fp8 else 0)
        self.variant = variant
        cu = _i32_array(list(cu_seqlens) if np_ > 0 else [0])
        kv = _i32_array(list(kv_lens))
        handle = ctypes.c_void_p()
        code = lib.pod_attn_plan(ctypes.byref(self.problem), ctypes.cast(cu, ctypes.c_void_p),
                                 ctypes.cast(kv, ctypes.c_void_p), ctypes.byref(self.options),
                                 ctypes.byref(handle))
        _check(code, "pod_attn_plan")
        self.handle = handle

    @classmethod
    def for_batch(cls, batch, variant="fused", **kw) -> "Plan":
        kw.setdefault("non_causal", not getattr(batch, "causal", True))
        kw.setdefault("head_dim", int(batch.head_dim))
        return cls(batch.num_q_heads, batch.num_kv_heads, batch.host_cu_seqlens,
                   batch.host_kv_lens, batch.num_decode_seqs, batch.num_blocks,
                   batch.max_blocks_per_seq, batch.scale, variant=variant, **kw)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value and _lib is not None:
            _lib.pod_attn_plan_destroy(h)
            self.handle = None

    @property
    def workspace_bytes(self) -> int:
        return int(load().pod_attn_workspace_bytes(self.handle))

    def info(self) -> dict:
        inf = PlanInfo()
        _check(load().pod_attn_get_plan_info(self.handle, ctypes.byref(inf)), "plan_info")
        return inf.as_dict()

    def items(self):
        """(prefill items [n][8], decode items [n][8], units [n][4]) as lists of lists."""
        lib = load()
        count = ctypes.c_size_t()
        _check(lib.pod_attn_plan_items(self.handle, None, 0, ctypes.byref(count)), "items")
        buf = (ctypes.c_int32 * max(1, count.value))()
        _check(lib.pod_attn_plan_items(self.handle, ctypes.cast(buf, ctypes.c_void_p),
                                       count.value, ctypes.byref(count)), "items")
        inf = self.info()
        flat = list(buf)[:count.value]
        n_p, n_d = inf["num_prefill_items"] * 8, inf["num_decode_items"] * 8
        rows = lambda xs, w: [xs[i:i + w] for i in range(0, len(xs), w)]
        return rows(flat[:n_p], 8), rows(flat[n_p:n_p + n_d], 8), rows(flat[n_p + n_d:], 4)

    def alloc_workspace(self, device="cuda"):
        import torch
        n = max(256, self.workspace_bytes)
        return torch.empty(n, dtype=torch.uint8, device=device)

    def upload(self, workspace, stream=None):
        _check(load().pod_attn_upload(self.handle, workspace.data_ptr(), workspace.numel(),
                                      _stream_ptr(stream)), "pod_attn_upload")

    def run(self, q_prefill, q_decode, k_pool, v_pool, block_tables, cu_seqlens_q, kv_lens,
            o_prefill, o_decode, workspace, stream=None, stream2=None):
        code = load().pod_attn_run(
            self.handle, _ptr(q_prefill), _ptr(q_decode), _ptr(k_pool), _ptr(v_pool),
            _ptr(block_tables), _ptr(cu_seqlens_q), _ptr(kv_lens), _ptr(o_prefill),
            _ptr(o_decode), workspace.data_ptr(), workspace.numel(), _stream_ptr(stream),
            _stream_ptr(stream2) if stream2 is not None else None)
        _check(code, "pod_attn_run")

    def bucket(self) -> dict:
        """pod_attn_plan_bucket: the plan's resource features and buckets."""
        b = Bucket()
        _check(load().pod_attn_plan_bucket(self.handle, ctypes.byref(b)), "pod_attn_plan_bucket")
        return {name: getattr(b, name) for name, _ in Bucket._fields_}

    def run_append(self, q_prefill, q_decode, k_new, v_new, k_pool, v_pool, block_tables,
                   cu_seqlens_q, kv_lens, o_prefill, o_decode, workspace, stream=None,
                   stream2=None):
        """pod_attn_run_append: write the new tokens' K/V rows (`k_new`, `v_new`, bf16
        [T_p + Nd][Hkv][128]) into the pools, then run the attention."""
        code = load().pod_attn_run_append(
            self.handle, _ptr(q_prefill), _ptr(q_decode), _ptr(k_new), _ptr(v_new),
            _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(cu_seqlens_q), _ptr(kv_lens),
            _ptr(o_prefill), _ptr(o_decode), workspace.data_ptr(), workspace.numel(),
            _stream_ptr(stream), _stream_ptr(stream2) if stream2 is not None else None)
        _check(code, "pod_attn_run_append")

    def run_decode_fp8(self, q_decode, k_pool8, v_pool8, k_scale, v_scale, block_tables,
                       kv_lens, o_decode, workspace, stream=None):
        """pod_attn_run_decode_fp8: decode over an e4m3 cache with K / V scales."""
        code = load().pod_attn_run_decode_fp8(
            self.handle, _ptr(q_decode), _ptr(k_pool8), _ptr(v_pool8), _ptr(k_scale),
            _ptr(v_scale), _ptr(block_tables), _ptr(kv_lens), _ptr(o_decode),
            workspace.data_ptr(), workspace.numel(), _stream_ptr(stream))
        _check(code, "pod_attn_run_decode_fp8")

    def append_fp8(self, k_new, v_new, k_pool8, v_pool8, k_scale, v_scale, block_tables,
                   workspace, stream=None):
        """pod_attn_append_fp8: quantise one new token per decode into the e4m3 cache."""
        code = load().pod_attn_append_fp8(
            self.handle, _ptr(k_new), _ptr(v_new), _ptr(k_pool8), _ptr(v_pool8), _ptr(k_scale),
            _ptr(v_scale), _ptr(block_tables), workspace.data_ptr(), workspace.numel(),
            _stream_ptr(stream))
        _check(code, "pod_attn_append_fp8")

    def device_status(self, workspace, stream=None) -> int:
        return int(load().pod_attn_last_device_status(self.handle, workspace.data_ptr(),
                                                      _stream_ptr(stream)))

    def records(self, workspace, stream=None):
        lib = load()
        inf = self.info()
        n = inf["num_prefill_items"] + inf["num_decode_items"]
        buf = (ItemRecord * max(1, n))()
        count = ctypes.c_size_t()
        _check(lib.pod_attn_read_records(self.handle, workspace.data_ptr(),
                                         ctypes.cast(buf, ctypes.c_void_p), n,
                                         ctypes.byref(count), _stream_ptr(stream)), "records")
        return [dict(smid=r.smid, kind=r.kind, item=r.item, cta=r.cta, t_start=r.t_start,
                     t_end=r.t_end) for r in buf[:count.value]]


def run_batch(plan: Plan, batch, workspace, o_prefill=None, o_decode=None, stream=None,
              stream2=None):
    """Launch `plan` on the device tensors of `batch`; returns (o_prefill, o_decode)."""
    import torch
    if o_prefill is None:
        o_prefill = torch.empty_like(batch.q_prefill)
    if o_decode is None:
        o_decode = torch.empty_like(batch.q_decode)
    if plan.variant == "streams" and stream2 is None:
        stream2 = _side_stream(batch.q_decode.device)
    plan.run(batch.q_prefill, batch.q_decode, batch.k_pool, batch.v_pool, batch.block_tables,
             batch.cu_seqlens_q, batch.kv_lens, o_prefill, o_decode, workspace, stream=stream,
             stream2=stream2)
    return o_prefill, o_decode


_side = {}


def _side_stream(device):
    import torch
    key = str(device)
    if key not in _side:
        _side[key] = torch.cuda.Stream(device=device)
    return _side[key]


def hybrid_attention(batch, variant: str = "fused", check_status: bool = True, **plan_kw):
    """One-call helper: plan, allocate a workspace, upload, run; returns (o_prefill, o_decode).

    `batch` holds device tensors (see ``workloads.HybridBatch``)."""
    plan = Plan.for_batch(batch, variant=variant, **plan_kw)
    ws = plan.alloc_workspace(batch.k_pool.device)
    plan.upload(ws)
    out = run_batch(plan, batch, ws)
    if check_status:
        _check(plan.device_status(ws), "device status")
    return out


def selftest_timeout(workspace, timeout_us: int, stream=None) -> int:
    """Run the bounded-wait self-test kernel; returns the device status it leaves (expected
    ERR_TIMEOUT)."""
    lib = load()
    _check(lib.pod_attn_selftest_timeout(workspace.data_ptr(), int(timeout_us),
                                         _stream_ptr(stream)), "selftest_timeout")
    return int(lib.pod_attn_last_device_status(None, workspace.data_ptr(), _stream_ptr(stream)))


def decode_fp8(fb, workspace=None, stream=None, **plan_kw):
    """Run the FP8-cache decode on an ``workloads.Fp8DecodeBatch`` whose tensors are on the GPU;
    returns o_decode (bf16 [Nd][Hq][128])."""
    import torch
    plan = Plan(fb.num_q_heads, fb.num_kv_heads, [], list(fb.decode_kv_lens),
                fb.num_decode_seqs, fb.num_blocks, fb.max_blocks_per_seq, fb.scale, kv_fp8=True,
                **plan_kw)
    ws = workspace if workspace is not None else plan.alloc_workspace(fb.q_decode.device)
    plan.upload(ws, stream)
    out = torch.empty_like(fb.q_decode)
    plan.run_decode_fp8(fb.q_decode, fb.k8, fb.v8, fb.k_scale, fb.v_scale, fb.block_tables,
                        fb.kv_lens, out, ws, stream=stream)
    st = plan.device_status(ws, stream)
    if st != OK:
        raise PodAttnError(st, "pod_attn_run_decode_fp8 (device)")
    return out
