"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, element by element.

Tolerance (bf16 inputs, fp32 accumulation, bf16 outputs): |gpu - oracle| <= 2e-2 + 2e-2 |oracle|
per element. Inputs come from the seeded generators; unused pool slots, spare blocks and
block-table tails are NaN-poisoned, so a read outside the visible rows fails the test.
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


def run_and_check(batch_cpu, variant="fused", **plan_kw):
    ref_p, ref_d = oracle.hybrid_attention(batch_cpu)
    dev = batch_cpu.to("cuda")
    o_p, o_d = B.hybrid_attention(dev, variant=variant, **plan_kw)
    torch.cuda.synchronize()
    assert_close(o_p, ref_p, f"{variant} prefill")
    assert_close(o_d, ref_d, f"{variant} decode")
    return o_p, o_d


@pytest.mark.parametrize("variant", ["fused", "serial", "streams"])
def test_tiny_hybrid_batch(variant):
    run_and_check(W.config(1), variant)


CASES = {
    # decode only, every supported group size, lengths around block boundaries
    "decode_g1": dict(Hq=4, Hkv=4, q=[], pkv=[], dkv=[1, 15, 16, 17, 100, 333]),
    "decode_g2": dict(Hq=8, Hkv=4, q=[], pkv=[], dkv=[1, 31, 32, 33, 700]),
    "decode_g3": dict(Hq=6, Hkv=2, q=[], pkv=[], dkv=[5, 64, 513]),
    "decode_g4": dict(Hq=16, Hkv=4, q=[], pkv=[], dkv=[2, 47, 1000]),
    "decode_g8": dict(Hq=16, Hkv=2, q=[], pkv=[], dkv=[3, 190, 2047]),
    # prefill only: ragged chunk tails, tile boundaries, prefixes of various sizes
    "prefill_fresh": dict(Hq=4, Hkv=2, q=[1, 127, 128, 129], pkv=[1, 127, 128, 129], dkv=[]),
    "prefill_extend": dict(Hq=4, Hkv=1, q=[300, 64, 5], pkv=[305, 1064, 70], dkv=[]),
    "prefill_g8": dict(Hq=8, Hkv=1, q=[200], pkv=[777], dkv=[]),
    # both kinds, several chunks, partial last blocks everywhere
    "mixed": dict(Hq=8, Hkv=2, q=[37, 256, 3], pkv=[37, 900, 51], dkv=[1, 17, 250, 4097]),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("variant", ["fused", "serial"])
def test_edge_cases(name, variant):
    c = CASES[name]
    b = W.make_batch(c["Hq"], c["Hkv"], c["q"], c["pkv"], c["dkv"], seed=sum(map(ord, name)))
    run_and_check(b, variant)


@pytest.mark.parametrize("opts", [
    dict(decode_splits=3, prefill_splits=3),           # exact split merge on both kinds
    dict(decode_splits=64, prefill_splits=8),          # many splits, some nearly empty rows
    dict(num_sms=3),                                   # few CTAs: long persistent loops
    dict(num_sms=2, ctas_per_sm=1, decode_splits=2),   # one CTA per SM
    dict(max_prefill_ctas=2),                          # prefill may fill both CTA slots
])
def test_planner_options(opts):
    b = W.make_batch(8, 2, [300, 40], [1000, 40], [1, 600, 2000, 31], seed=77)
    run_and_check(b, "fused", **opts)


def test_mixed_kind_worked_example():
    run_and_check(W.mixed_kind_example())


def test_variants_agree_bitwise_and_runs_repeat():
    b = W.make_batch(8, 2, [300, 40], [1000, 40], [1, 600, 2000, 31], seed=5).to("cuda")
    outs = {}
    for variant in ("fused", "serial", "streams"):
        plan = B.Plan.for_batch(b, variant=variant, decode_splits=4, prefill_splits=2)
        ws = plan.alloc_workspace()
        plan.upload(ws)
        runs = [tuple(t.clone() for t in B.run_batch(plan, b, ws)) for _ in range(3)]
        assert plan.device_status(ws) == B.OK
        for r in runs[1:]:                      # counters reset themselves between runs
            assert torch.equal(r[0], runs[0][0]) and torch.equal(r[1], runs[0][1])
        outs[variant] = runs[0]
    for v in ("serial", "streams"):             # same items, same arithmetic: same bits
        assert torch.equal(outs[v][0], outs["fused"][0])
        assert torch.equal(outs[v][1], outs["fused"][1])


def _sample_prefill_rows(q_lens):
    rows = set()
    cu = 0
    for q in q_lens:
        rows.update([cu, cu + q - 1])
        for t in range(128, q, 128):
            rows.update([cu + t - 1, cu + t])
        rows.update(range(cu, cu + q, 61))
        cu += q
    return sorted(rows)


@pytest.mark.parametrize("i", [2, 3, 4])
def test_full_size_configs_sampled(i):
    """Full-size configurations in the launch configuration the benchmark times (fused, default
    plan): every decode output and sampled prefill rows (chunk ends, every 128-row tile boundary,
    every 61st row), all heads, against the oracle row by row."""
    dev = W.config(i, device="cuda")
    o_p, o_d = B.hybrid_attention(dev, variant="fused")
    torch.cuda.synchronize()
    cpu = dev.to("cpu")
    Hq = dev.num_q_heads
    prow = _sample_prefill_rows(dev.q_lens)
    kinds = [0] * (len(prow) * Hq) + [1] * (dev.num_decode_seqs * Hq)
    idx = [r for r in prow for _ in range(Hq)] + [d for d in range(dev.num_decode_seqs)
                                                 for _ in range(Hq)]
    heads = list(range(Hq)) * (len(prow) + dev.num_decode_seqs)
    ref = oracle.rows(cpu, kinds, idx, heads)
    got_p = o_p.float().cpu()
    got_d = o_d.float().cpu()
    got = torch.stack([got_p[r, h] if k == 0 else got_d[r, h]
                       for k, r, h in zip(kinds, idx, heads)])
    assert_close(got.to(torch.bfloat16), ref, f"config {i}")
    # every output is finite (poisoned slots never leak)
    assert torch.isfinite(o_p.float()).all() and torch.isfinite(o_d.float()).all()


def test_bad_block_index_is_reported_not_faulted():
    b = W.make_batch(4, 2, [40], [100], [70], seed=9)
    b.block_tables[0, 2] = 1 << 28          # inside the visible range of the prefill sequence
    b.block_tables[1, 1] = -5               # inside the visible range of the decode sequence
    dev = b.to("cuda")
    plan = B.Plan.for_batch(dev)
    ws = plan.alloc_workspace()
    plan.upload(ws)
    B.run_batch(plan, dev, ws)
    assert plan.device_status(ws) == B.ERR_BAD_INDEX
    # the context stays usable
    run_and_check(W.config(1))


def test_bounded_wait_times_out_and_context_survives():
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    assert B.selftest_timeout(ws, 2000) == B.ERR_TIMEOUT
    run_and_check(W.config(1))


def test_instrumentation_records_every_item_and_mixes_kinds():
    dev = W.make_batch(32, 8, [1024], [4096], [3000] * 40, seed=3, device="cuda")
    plan = B.Plan.for_batch(dev, instrument=True)
    ws = plan.alloc_workspace()
    plan.upload(ws)
    B.run_batch(plan, dev, ws)
    recs = plan.records(ws)
    inf = plan.info()
    assert len(recs) == inf["num_prefill_items"] + inf["num_decode_items"]
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    for r in recs:
        assert 0 <= r["smid"] < nsm and r["t_end"] >= r["t_start"] > 0
    kinds_per_sm = {}
    for r in recs:
        kinds_per_sm.setdefault(r["smid"], set()).add(r["kind"])
    both = sum(1 for k in kinds_per_sm.values() if k == {0, 1})
    assert both >= len(kinds_per_sm) // 2, (both, len(kinds_per_sm))


@pytest.mark.parametrize("cap", [1, 5])
def test_prefill_cta_cap_keeps_prefill_on_the_first_ctas(cap):
    """max_prefill_ctas: every prefill item runs on a CTA below the cap (the kernel's own
    records), the other CTAs run decode work only, and the outputs match the oracle."""
    cpu = W.make_batch(32, 8, [700, 300], [2700, 300], [3000] * 24, seed=11)
    ref_p, ref_d = oracle.hybrid_attention(cpu)
    dev = cpu.to("cuda")
    plan = B.Plan.for_batch(dev, instrument=True, max_prefill_ctas=cap)
    assert plan.info()["max_prefill_ctas"] == cap
    ws = plan.alloc_workspace()
    plan.upload(ws)
    o_p, o_d = B.run_batch(plan, dev, ws)
    torch.cuda.synchronize()
    assert plan.device_status(ws) == B.OK
    recs = plan.records(ws)
    assert {r["cta"] for r in recs if r["kind"] == 0} <= set(range(cap))
    assert any(r["kind"] == 1 and r["cta"] >= cap for r in recs)
    assert_close(o_p, ref_p, f"cap {cap} prefill")
    assert_close(o_d, ref_d, f"cap {cap} decode")


def _ramp_batch(seed, q=(300, 40), pkv=(1300, 200), dkv=(900, 17), head_dim=128, causal=True):
    """A GQA batch whose scores grow along every sequence by ~10 (log2 units) per 128 keys: K row
    p is 0.6 p / 128 along the all-ones direction plus small noise, and every query is near that
    direction. Each 128-key step then moves the row max past the lazy-rescale threshold (2^8),
    so the prefill tile rescales O at every step (waiting for the previous P·V) and splits
    merge partials whose maxima differ by far more than the threshold."""
    b = W.make_batch(8, 2, list(q), list(pkv), list(dkv), seed=seed, head_dim=head_dim,
                     causal=causal)
    D, Hkv = b.head_dim, b.num_kv_heads
    g = torch.Generator().manual_seed(seed)
    bt = b.block_tables.long()
    for s, L in enumerate(b.host_kv_lens):
        pos = torch.arange(L)
        rows = (0.6 / D) * pos.float()[:, None, None].expand(L, Hkv, D) \
            + 0.05 * torch.randn(L, Hkv, D, generator=g)
        blk = bt[s, pos // 16]
        b.k_pool[blk, :, pos % 16, :] = rows.to(torch.bfloat16)
    b.q_prefill.copy_((1.0 + 0.1 * torch.randn(b.q_prefill.shape, generator=g)).to(torch.bfloat16))
    b.q_decode.copy_((1.0 + 0.1 * torch.randn(b.q_decode.shape, generator=g)).to(torch.bfloat16))
    return b


@pytest.mark.parametrize("variant,kw", [("fused", {}), ("fused", {"prefill_splits": 3}),
                                        ("serial", {}), ("fused", {"num_sms": 3})])
def test_growing_scores_rescale_every_step(variant, kw):
    run_and_check(_ramp_batch(41), variant, **kw)


@pytest.mark.parametrize("head_dim,causal", [(64, True), (128, False)])
def test_growing_scores_rescale_head_dim_64_and_non_causal(head_dim, causal):
    run_and_check(_ramp_batch(43, head_dim=head_dim, causal=causal), "fused")


@pytest.mark.parametrize("variant,kw", [("fused", {"num_sms": 1}), ("fused", {"num_sms": 2, "prefill_splits": 5}),
                                        ("serial", {"num_sms": 1, "prefill_splits": 3}),
                                        ("fused", {})])
def test_items_of_one_two_three_steps_through_few_ctas(variant, kw):
    """Prefill items of 1, 2 and 3 key steps (the ends of the ring's consumption order: K(0),
    K(1), then V(j), K(j + 2), then the last V's) and longer ones, split or not, many of them
    through one or two CTAs, so every ring stage and barrier carries its phases across items of
    different lengths."""
    b = W.make_batch(8, 2, [100, 60, 10, 1, 200, 129], [100, 200, 300, 257, 700, 1000],
                     [5, 130, 390], seed=47)
    run_and_check(b, variant, **kw)
