"""GPU checks of pod_attn_run_append (the KV append in front of the attention), through the
C ABI: the pools come in with the iteration's new rows missing (NaN), the call writes them and
attends. The pools afterwards must equal, bit for bit, the oracle's append of those rows
(oracle.append_bf16), and the outputs must equal, bit for bit, those of pod_attn_run on the
complete pools — itself checked against the fp64 oracle in test_gpu_parity.py (configuration 1
is checked against the oracle here too)."""
import numpy as np
import pytest
import torch

import oracle
from hybrid_prefill_decode_gb300 import binding as B
from hybrid_prefill_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu

VARIANTS = ("fused", "serial", "streams")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _bits(t):
    return t.contiguous().view(torch.int16)


def _run_both(batch, variant, **kw):
    plan = B.Plan.for_batch(batch, variant=variant, **kw)
    ws = plan.alloc_workspace()
    plan.upload(ws)
    ref_p, ref_d = B.run_batch(plan, batch, ws)                 # rows already in the pools
    assert plan.device_status(ws) == B.OK
    k_new, v_new, kp, vp = W.split_off_new_rows(batch)
    # the expected pools: the oracle's append of the new rows to the pools without them
    exp_k, exp_v = oracle.append_bf16(batch, k_new, v_new, kp, vp)
    o_p, o_d = torch.empty_like(batch.q_prefill), torch.empty_like(batch.q_decode)
    side = torch.cuda.Stream() if variant == "streams" else None
    plan.run_append(batch.q_prefill, batch.q_decode, k_new, v_new, kp, vp, batch.block_tables,
                    batch.cu_seqlens_q, batch.kv_lens, o_p, o_d, ws, stream2=side)
    assert plan.device_status(ws) == B.OK
    assert np.array_equal(oracle._u16(kp), exp_k) and np.array_equal(oracle._u16(vp), exp_v)
    assert torch.equal(_bits(o_p), _bits(ref_p)) and torch.equal(_bits(o_d), _bits(ref_d))
    return o_p, o_d


@pytest.mark.parametrize("variant", VARIANTS)
def test_append_tiny_matches_oracle(variant):
    b = W.config(1, device="cuda")
    o_p, o_d = _run_both(b, variant)
    ref_p, ref_d = oracle.hybrid_attention(b.to("cpu"))
    for got, ref in ((o_p, ref_p), (o_d, ref_d)):
        g = got.float().cpu().numpy().astype(np.float64)
        assert (np.abs(g - ref) <= 2e-2 + 2e-2 * np.abs(ref)).all()


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("case", ["mixed", "decode_only", "prefill_only", "ragged", "gqa"])
def test_append_edge_cases(variant, case):
    if case == "mixed":
        b = W.mixed_kind_example(device="cuda")
    elif case == "decode_only":
        b = W.make_batch(8, 8, [], [], [1, 15, 16, 17, 300], seed=21, device="cuda")
    elif case == "prefill_only":
        b = W.make_batch(8, 2, [1, 127, 129], [1, 200, 129], [], seed=22, device="cuda")
    elif case == "ragged":
        b = W.make_batch(4, 4, [33, 7], [100, 7], [49, 2, 64], seed=23, device="cuda")
    else:
        b = W.make_batch(32, 4, [300], [2000], [900, 1700, 31], seed=24, device="cuda")
    _run_both(b, variant)


@pytest.mark.parametrize("cfg", [2, 3])
def test_append_full_size_fused(cfg):
    _run_both(W.config(cfg, device="cuda"), "fused")


def test_append_forced_splits_and_few_ctas():
    b = W.make_batch(16, 4, [700], [3000], [2500] * 9, seed=25, device="cuda")
    _run_both(b, "fused", num_sms=3, prefill_splits=3, decode_splits=5)


def test_append_bad_block_index_is_reported():
    b = W.make_batch(4, 2, [20], [40], [17], seed=26, device="cuda")
    plan = B.Plan.for_batch(b)
    ws = plan.alloc_workspace()
    plan.upload(ws)
    k_new, v_new, kp, vp = W.split_off_new_rows(b)
    bt = b.block_tables.clone()
    bt[1, 1] = b.num_blocks + 7                      # the decode token's block: outside the pool
    o_p, o_d = torch.empty_like(b.q_prefill), torch.empty_like(b.q_decode)
    plan.run_append(b.q_prefill, b.q_decode, k_new, v_new, kp, vp, bt, b.cu_seqlens_q,
                    b.kv_lens, o_p, o_d, ws)
    assert plan.device_status(ws) == B.ERR_BAD_INDEX
