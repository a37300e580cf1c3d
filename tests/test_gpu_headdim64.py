"""GPU parity at head dim 64 (the library's second head dim) against the fp64 oracle, through
the C ABI: the same kernels instantiated for 64 dims, every variant, decode group sizes, ragged
prefill chunks, non-causal chunks, forced splits and the KV append."""
import pytest
import torch

from hybrid_prefill_decode_gb300 import binding as B
from hybrid_prefill_decode_gb300 import workloads as W
from test_gpu_parity import run_and_check

pytestmark = pytest.mark.gpu

VARIANTS = ("fused", "serial", "streams")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


CASES = {
    "tiny_mixed": dict(Hq=2, Hkv=1, q=[64], pkv=[128], dkv=[100, 150, 233, 300]),
    "decode_g1": dict(Hq=4, Hkv=4, q=[], pkv=[], dkv=[1, 15, 16, 17, 333]),
    "decode_g2": dict(Hq=8, Hkv=4, q=[], pkv=[], dkv=[1, 31, 700]),
    "decode_g4": dict(Hq=16, Hkv=4, q=[], pkv=[], dkv=[2, 47, 1000]),
    "decode_g8": dict(Hq=16, Hkv=2, q=[], pkv=[], dkv=[3, 190, 2047]),
    "prefill_ragged": dict(Hq=4, Hkv=4, q=[1, 127, 128, 129], pkv=[1, 200, 128, 300], dkv=[]),
    "gqa_mixed": dict(Hq=32, Hkv=8, q=[300, 17], pkv=[1500, 40], dkv=[900, 33, 2000]),
    "gqa8_mixed": dict(Hq=32, Hkv=4, q=[260], pkv=[2300], dkv=[17, 1200]),
}


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", sorted(CASES))
def test_head_dim_64(name, variant):
    c = CASES[name]
    b = W.make_batch(c["Hq"], c["Hkv"], c["q"], c["pkv"], c["dkv"], seed=sum(map(ord, name)),
                     head_dim=64)
    run_and_check(b, variant)


def test_head_dim_64_non_causal_and_forced_splits():
    b = W.make_batch(16, 4, [700], [3000], [2500] * 5, seed=71, head_dim=64, causal=False)
    run_and_check(b, "fused", num_sms=3, prefill_splits=3, decode_splits=4)


@pytest.mark.parametrize("variant", VARIANTS)
def test_head_dim_64_kv_append(variant):
    b = W.make_batch(8, 2, [33, 100], [60, 700], [49, 2, 1000], seed=72, head_dim=64,
                     device="cuda")
    plan = B.Plan.for_batch(b, variant=variant)
    ws = plan.alloc_workspace()
    plan.upload(ws)
    ref_p, ref_d = B.run_batch(plan, b, ws)
    k_new, v_new, kp, vp = W.split_off_new_rows(b)
    o_p, o_d = torch.empty_like(b.q_prefill), torch.empty_like(b.q_decode)
    side = torch.cuda.Stream() if variant == "streams" else None
    plan.run_append(b.q_prefill, b.q_decode, k_new, v_new, kp, vp, b.block_tables,
                    b.cu_seqlens_q, b.kv_lens, o_p, o_d, ws, stream2=side)
    assert plan.device_status(ws) == B.OK
    bits = lambda t: t.contiguous().view(torch.int16)
    assert torch.equal(bits(kp), bits(b.k_pool)) and torch.equal(bits(vp), bits(b.v_pool))
    assert torch.equal(bits(o_p), bits(ref_p)) and torch.equal(bits(o_d), bits(ref_d))
