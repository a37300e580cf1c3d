"""GPU parity of the decode over an FP8 (e4m3) KV cache against the fp64 oracle's reading.

Each cached K value is e4m3 x a per-(kv-head, channel) scale and each V value e4m3 x a
per-(row, kv-head) scale ("LLMSO - W4 - Optimization & Frameworks", §"2-4. 고급 KV 캐싱 기법":
K per channel, V per token). The kernel decodes e4m3 exactly (every e4m3 value is an
f16 value), folds the K scales into the query and the V scales into the P·V weights, and rounds
those to f16 for the tensor cores (11 significant bits, finer than bf16's 8): the tolerance
stays the library's |err| <= 2e-2 + 2e-2 |ref|.
"""
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


def assert_close(got, ref, what=""):
    g = got.float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    if bad.any():
        idx = np.argwhere(bad)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"max err {err.max():.4g}; first bad {idx[:5].tolist()}")


LENS = [1, 15, 16, 17, 300, 2047]


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (16, 4), (16, 2)])
def test_fp8_decode_group_sizes(hq, hkv):
    fb = W.make_fp8_decode_batch(hq, hkv, LENS, seed=31 + hq * 7 + hkv)
    ref = oracle.decode_fp8(fb)
    out = B.decode_fp8(fb.to("cuda"))
    torch.cuda.synchronize()
    assert_close(out, ref, f"fp8 G={hq // hkv}")


@pytest.mark.parametrize("splits", [1, 3, 64])
def test_fp8_decode_forced_splits(splits):
    fb = W.make_fp8_decode_batch(16, 2, [5, 190, 1000, 2047], seed=400 + splits)
    ref = oracle.decode_fp8(fb)
    out = B.decode_fp8(fb.to("cuda"), decode_splits=splits)
    torch.cuda.synchronize()
    assert_close(out, ref, f"fp8 splits={splits}")


def test_fp8_decode_few_sms_and_repeat_bitwise():
    fb = W.make_fp8_decode_batch(32, 8, [3000] * 5 + [17, 1], seed=12).to("cuda")
    a = B.decode_fp8(fb, num_sms=3)
    b = B.decode_fp8(fb, num_sms=3)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert_close(a, oracle.decode_fp8(fb.to("cpu")), "fp8 few SMs")


def test_fp8_pow2_scales_match_bf16_path():
    """With power-of-two scales the dequantised cache is exact in bf16, so the FP8 path and the
    bf16 library path compute from the same values: both within tolerance of the same oracle."""
    fb = W.make_fp8_decode_batch(32, 8, [40, 513, 2000], seed=8, pow2_scales=True)
    bb = W.dequantised_batch(fb)
    ref = oracle.hybrid_attention(bb)[1]
    np.testing.assert_allclose(oracle.decode_fp8(fb), ref, rtol=1e-12, atol=1e-12)
    out8 = B.decode_fp8(fb.to("cuda"))
    _, out16 = B.hybrid_attention(bb.to("cuda"))
    torch.cuda.synchronize()
    assert_close(out8, ref, "fp8 pow2")
    assert_close(out16, ref, "bf16 of the dequantised cache")


def test_fp8_bad_block_index_is_reported_not_faulted():
    fb = W.make_fp8_decode_batch(8, 2, [40, 300], seed=19)
    fb.block_tables[1, 3] = 1 << 28         # inside the visible range of decode 1
    dev = fb.to("cuda")
    with pytest.raises(B.PodAttnError) as e:
        B.decode_fp8(dev)
    assert e.value.code == B.ERR_BAD_INDEX
    # the context stays usable
    ok = W.make_fp8_decode_batch(8, 2, [1, 17, 300], seed=5)
    assert_close(B.decode_fp8(ok.to("cuda")), oracle.decode_fp8(ok), "fp8 after bad index")


@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_fp8_full_size_decodes_of_each_configuration(cfg):
    """The decodes the benchmark times (--kv-fp8 --config cfg), in its launch configuration
    (default plan, one launch), every output against the oracle."""
    Hq, Hkv, _, _, dkv = W.config_lengths(cfg)
    fb = W.make_fp8_decode_batch(Hq, Hkv, dkv, seed=cfg, device="cuda")
    out = B.decode_fp8(fb)
    torch.cuda.synchronize()
    assert_close(out, oracle.decode_fp8(fb.to("cpu")), f"fp8 config {cfg}")


def _append_plan(fb, **kw):
    return B.Plan(fb.num_q_heads, fb.num_kv_heads, [], list(fb.decode_kv_lens),
                  fb.num_decode_seqs, fb.num_blocks, fb.max_blocks_per_seq, fb.scale,
                  kv_fp8=True, **kw)


@pytest.mark.parametrize("hq,hkv,lens", [(8, 2, [1, 16, 17, 300]), (32, 8, [2047, 5, 64, 4096]),
                                         (4, 4, [1, 2, 3])])
def test_fp8_append_bit_exact_then_decode(hq, hkv, lens):
    fb, k_new, v_new = W.fp8_append_case(hq, hkv, lens, seed=hq + hkv + len(lens))
    want_k8, want_v8, want_vs = oracle.append_fp8(fb, k_new, v_new)
    dev = fb.to("cuda")
    plan = _append_plan(dev)
    ws = plan.alloc_workspace()
    plan.upload(ws)
    plan.append_fp8(k_new.to("cuda"), v_new.to("cuda"), dev.k8, dev.v8, dev.k_scale, dev.v_scale,
                    dev.block_tables, ws)
    assert plan.device_status(ws) == B.OK
    assert np.array_equal(dev.k8.cpu().numpy(), want_k8)
    assert np.array_equal(dev.v8.cpu().numpy(), want_v8)
    got_vs = dev.v_scale.cpu().numpy()
    assert np.array_equal(np.isnan(got_vs), np.isnan(want_vs))
    assert np.array_equal(got_vs[~np.isnan(got_vs)], want_vs[~np.isnan(want_vs)])
    # the decode over the appended cache, against the oracle on the oracle-appended cache
    ref_fb = fb.to("cpu")
    ref_fb.k8, ref_fb.v8 = torch.from_numpy(want_k8), torch.from_numpy(want_v8)
    ref_fb.v_scale = torch.from_numpy(want_vs)
    out = torch.empty_like(dev.q_decode)
    plan.run_decode_fp8(dev.q_decode, dev.k8, dev.v8, dev.k_scale, dev.v_scale,
                        dev.block_tables, dev.kv_lens, out, ws)
    assert plan.device_status(ws) == B.OK
    assert_close(out, oracle.decode_fp8(ref_fb), "fp8 decode after append")


def test_fp8_append_bad_block_index_is_reported():
    fb, k_new, v_new = W.fp8_append_case(8, 2, [40, 300], seed=7)
    fb.block_tables[1, 299 // 16] = -3          # the block of decode 1's new row
    dev = fb.to("cuda")
    before = dev.k8.clone()
    plan = _append_plan(dev)
    ws = plan.alloc_workspace()
    plan.upload(ws)
    plan.append_fp8(k_new.to("cuda"), v_new.to("cuda"), dev.k8, dev.v8, dev.k_scale, dev.v_scale,
                    dev.block_tables, ws)
    assert plan.device_status(ws) == B.ERR_BAD_INDEX
    # decode 0's row was written, decode 1's was not (and nothing else changed)
    changed = (dev.k8 != before).nonzero()
    assert changed.numel() > 0
    pos0 = 39
    phys0 = int(fb.block_tables[0, pos0 // 16])
    assert torch.all(changed[:, 0] == phys0) and torch.all(changed[:, 2] == pos0 % 16)


@pytest.mark.parametrize("seed", range(32))
def test_fp8_random_batches(seed):
    """Seeded random FP8 decode batches: group sizes 1-8 (3 included), ragged lengths, forced
    or automatic splits, small SM counts."""
    import random
    rng = random.Random(seed)
    Hkv = rng.choice([1, 2, 4])
    Hq = Hkv * rng.choice([1, 2, 3, 4, 8])
    lens = [rng.choice([1, rng.randint(2, 40), rng.randint(40, 3000)])
            for _ in range(rng.choice([1, 3, 12, 30]))]
    opts = {}
    if rng.random() < 0.3:
        opts["decode_splits"] = rng.choice([2, 7, 64])
    if rng.random() < 0.3:
        opts["num_sms"] = rng.choice([1, 5, 33])
    fb = W.make_fp8_decode_batch(Hq, Hkv, lens, seed=500 + seed)
    out = B.decode_fp8(fb.to("cuda"), **opts)
    torch.cuda.synchronize()
    assert_close(out, oracle.decode_fp8(fb), f"fp8 seed {seed}")
