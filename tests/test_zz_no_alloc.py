"""The allocation-free entry point pod_attn_run_static against the workspace entry point.

pod_attn_run_static serves callers that cannot call cudaMalloc for a workspace (for example a
plugin inside a host program whose device memory belongs to that program's own allocator, or a
latency-critical loop that cannot afford cudaMalloc's implicit device synchronisation). It keeps
its scratch in one library-owned device array instead. This file is collected last so that a
run that stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from hybrid_prefill_decode_gb300 import binding as B
from hybrid_prefill_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ATOL = 2e-2
RTOL = 2e-2


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    lib = B.load()
    P = ctypes.c_void_p
    lib.pod_attn_run_static.restype = ctypes.c_int32
    lib.pod_attn_run_static.argtypes = [P] * 11
    return lib


def _p(t):
    return t.data_ptr() if t is not None and t.numel() > 0 else None


def _run_static(lib, plan, b, o_p, o_d):
    return lib.pod_attn_run_static(plan.handle, _p(b.q_prefill), _p(b.q_decode), _p(b.k_pool),
                                   _p(b.v_pool), _p(b.block_tables), _p(b.cu_seqlens_q),
                                   _p(b.kv_lens), _p(o_p), _p(o_d),
                                   torch.cuda.current_stream().cuda_stream or None)


def _close(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(a).all()
    assert (np.abs(a - b) <= ATOL + RTOL * np.abs(b)).all(), float(np.abs(a - b).max())


@pytest.mark.parametrize("case", ["tiny", "split_merges"])
def test_static_scratch_matches_workspace_entry_on_two_calls(lib, case):
    if case == "tiny":
        b = W.config(1, device="cuda")
        kw = {}
    else:   # forced splits: the merge counters and partial slots in the scratch are exercised
        b = W.make_batch(8, 2, [300, 40], [1000, 40], [1, 600, 2000, 31], seed=21,
                         device="cuda")
        kw = dict(decode_splits=3, prefill_splits=3)
    ref_p, ref_d = B.hybrid_attention(b, variant="fused", **kw)
    plan = B.Plan.for_batch(b, variant="fused", **kw)
    assert plan.workspace_bytes <= 32 * 1024 * 1024
    for _ in range(2):                         # the array keeps the previous call's contents
        o_p = torch.full_like(b.q_prefill, float("nan"))
        o_d = torch.full_like(b.q_decode, float("nan"))
        assert _run_static(lib, plan, b, o_p, o_d) == B.OK
        torch.cuda.synchronize()
        _close(o_p, ref_p)
        _close(o_d, ref_d)


def test_static_scratch_rejects_plans_beyond_its_size(lib):
    Hq, Hkv, ql, pkv, dkv = W.config_lengths(4)
    cu = [0, ql[0]]
    plan = B.Plan(Hq, Hkv, cu, pkv + dkv, len(dkv), 200000, 2048, 0.0883883, num_sms=152)
    assert plan.workspace_bytes > 32 * 1024 * 1024
    code = lib.pod_attn_run_static(plan.handle, None, None, None, None, None, None, None, None,
                                   None, None)
    assert code == B.ERR_WORKSPACE
    serial = B.Plan(4, 2, [0, 5], [9, 7], 1, 10, 4, 0.1, variant="serial", num_sms=148)
    assert lib.pod_attn_run_static(serial.handle, None, None, None, None, None, None, None,
                                   None, None, None) == B.ERR_INVALID_ARG
