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
    lib.pod_attn_last_device_status.restype = ctypes.c_int32
    lib.pod_attn_last_device_status.argtypes = [P, P, P]
    return lib


def _p(t):
    return t.data_ptr() if t is not None and t.numel() > 0 else None


def _run_static(lib, plan, b, o_p, o_d):
    return lib.pod_attn_run_static(plan.handle, _p(b.q_prefill), _p(b.q_decode), _p(b.k_pool),
                                   _p(b.v_pool), _p(b.block_tables), _p(b.cu_seqlens_q),
                                   _p(b.kv_lens), _p(o_p), _p(o_d),
                                   torch.cuda.current_stream().cuda_stream or None)


def _close(a, ref):
    """Element-wise |a - ref| <= ATOL + RTOL * |ref| against the fp64 oracle's output."""
    a = a.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(a).all()
    assert (np.abs(a - ref) <= ATOL + RTOL * np.abs(ref)).all(), float(np.abs(a - ref).max())


@pytest.mark.parametrize("case", ["tiny", "split_merges"])
def test_static_scratch_matches_workspace_entry_on_two_calls(lib, case):
    """Same plan, same inputs: the outputs equal the workspace entry point's bit for bit (the
    same items run the same arithmetic) and match the fp64 oracle, on two calls in a row (the
    array keeps the previous call's contents); the status word reads OK through the NULL
    workspace form of pod_attn_last_device_status."""
    import oracle
    if case == "tiny":
        cpu = W.config(1)
        kw = {}
    else:   # forced splits: the merge counters and partial slots in the scratch are exercised
        cpu = W.make_batch(8, 2, [300, 40], [1000, 40], [1, 600, 2000, 31], seed=21)
        kw = dict(decode_splits=3, prefill_splits=3)
    b = cpu.to("cuda")
    ref_p, ref_d = oracle.hybrid_attention(cpu)
    ws_p, ws_d = B.hybrid_attention(b, variant="fused", **kw)
    plan = B.Plan.for_batch(b, variant="fused", **kw)
    assert plan.workspace_bytes <= 32 * 1024 * 1024
    for _ in range(2):                         # the array keeps the previous call's contents
        o_p = torch.full_like(b.q_prefill, float("nan"))
        o_d = torch.full_like(b.q_decode, float("nan"))
        assert _run_static(lib, plan, b, o_p, o_d) == B.OK
        torch.cuda.synchronize()
        assert torch.equal(o_p.view(torch.int16), ws_p.view(torch.int16))
        assert torch.equal(o_d.view(torch.int16), ws_d.view(torch.int16))
        _close(o_p, ref_p)
        _close(o_d, ref_d)
        assert lib.pod_attn_last_device_status(plan.handle, None,
                                               torch.cuda.current_stream().cuda_stream
                                               or None) == B.OK


def test_static_scratch_reports_a_bad_block_index(lib):
    """A block-table entry outside the pool is reported through the array's status word, read
    with a NULL workspace, and the next clean call reads OK again."""
    b = W.make_batch(4, 2, [], [], [200, 90], seed=4, device="cuda")
    plan = B.Plan.for_batch(b, variant="fused")
    bad = b.block_tables.clone()
    bad[1, 2] = b.num_blocks + 7
    o_d = torch.empty_like(b.q_decode)
    stream = torch.cuda.current_stream().cuda_stream or None
    code = lib.pod_attn_run_static(plan.handle, None, _p(b.q_decode), _p(b.k_pool), _p(b.v_pool),
                                   _p(bad), None, _p(b.kv_lens), None, _p(o_d), stream)
    assert code == B.OK
    assert lib.pod_attn_last_device_status(plan.handle, None, stream) == B.ERR_BAD_INDEX
    assert _run_static(lib, plan, b, None, o_d) == B.OK
    assert lib.pod_attn_last_device_status(plan.handle, None, stream) == B.OK


def test_static_scratch_rejects_plans_it_cannot_run(lib):
    """Plans beyond the array's size (WORKSPACE), other variants and instrumented plans
    (INVALID_ARG), and plans for the e4m3 cache (UNSUPPORTED)."""
    Hq, Hkv, ql, pkv, dkv = W.config_lengths(4)
    cu = [0, ql[0]]
    plan = B.Plan(Hq, Hkv, cu, pkv + dkv, len(dkv), 200000, 2048, 0.0883883, num_sms=152)
    assert plan.workspace_bytes > 32 * 1024 * 1024
    none = [None] * 9
    assert lib.pod_attn_run_static(plan.handle, *none, None) == B.ERR_WORKSPACE
    serial = B.Plan(4, 2, [0, 5], [9, 7], 1, 10, 4, 0.1, variant="serial", num_sms=148)
    assert lib.pod_attn_run_static(serial.handle, *none, None) == B.ERR_INVALID_ARG
    inst = B.Plan(4, 2, [0, 5], [9, 7], 1, 10, 4, 0.1, instrument=True, num_sms=148)
    assert lib.pod_attn_run_static(inst.handle, *none, None) == B.ERR_INVALID_ARG
    fp8 = B.Plan(8, 2, [], [300, 17], 2, 40, 20, 0.1, kv_fp8=True, num_sms=148)
    assert lib.pod_attn_run_static(fp8.handle, *none, None) == B.ERR_UNSUPPORTED
