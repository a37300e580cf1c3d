"""Pins of the fp64 oracle to facts other than itself (no GPU).

Each test checks the oracle against something the pages or the mathematics fix: closed forms,
invariants, special cases, an independent NumPy brute force, and worked numbers printed on the
pages. Together they are chosen so that a plausible slip in the oracle (a dropped scale, a wrong
causal offset, a wrong head mapping, a transposed gather, a missing max subtraction, an inexact
merge) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import bruteforce
from hybrid_prefill_decode_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f64(t):
    return bruteforce.bf16_bits_to_f64(t.contiguous().view(torch.int16).numpy().view(np.uint16))


def _rows(batch, s, g, n, pool="v"):
    """Rows 0..n-1 of kv-head g of sequence s, read straight from the pool (test-side gather)."""
    p = _f64(batch.v_pool if pool == "v" else batch.k_pool)
    bt = batch.block_tables.numpy()
    return np.stack([p[bt[s, j // 16], g, j % 16] for j in range(n)])


def _small(seed=0, Hq=4, Hkv=2, q_lens=(5, 3), pkv=(9, 3), dkv=(1, 17, 33), **kw):
    return W.make_batch(Hq, Hkv, list(q_lens), list(pkv), list(dkv), seed=seed, **kw)


# 1. closed form: q = 0 (or scale = 0) -> every visible key has equal weight -> mean of V rows
@pytest.mark.parametrize("how", ["q_zero", "scale_zero"])
def test_uniform_scores_give_mean_of_visible_rows(how):
    b = _small(seed=1)
    if how == "q_zero":
        b.q_prefill.zero_()
        b.q_decode.zero_()
    else:
        b.scale = 0.0
    o_p, o_d = oracle.hybrid_attention(b)
    group = b.num_q_heads // b.num_kv_heads
    cu = b.host_cu_seqlens
    for s, (C, L) in enumerate(zip(b.q_lens, b.prefill_kv_lens)):
        for i in range(C):
            p = L - C + i
            for h in range(b.num_q_heads):
                ref = _rows(b, s, h // group, p + 1).mean(axis=0)
                np.testing.assert_allclose(o_p[cu[s] + i, h], ref, rtol=0, atol=1e-12)
    for d, L in enumerate(b.decode_kv_lens):
        for h in range(b.num_q_heads):
            ref = _rows(b, b.num_prefill_seqs + d, h // group, L).mean(axis=0)
            np.testing.assert_allclose(o_d[d, h], ref, rtol=0, atol=1e-12)


# 2. special case: a single visible key returns its V row exactly
def test_single_visible_key_returns_its_value_row():
    b = _small(seed=2, q_lens=(4,), pkv=(4,), dkv=(1, 1))
    o_p, o_d = oracle.hybrid_attention(b)
    group = b.num_q_heads // b.num_kv_heads
    for h in range(b.num_q_heads):
        # prefill row 0 of a chunk with no prefix sees key 0 only
        assert np.array_equal(o_p[0, h], _rows(b, 0, h // group, 1)[0])
        for d in range(2):
            assert np.array_equal(o_d[d, h], _rows(b, 1 + d, h // group, 1)[0])


# 3. invariant: causality — rows after position p do not influence the output at p
def test_causal_rows_unchanged_when_later_keys_perturbed():
    b = _small(seed=3, q_lens=(20,), pkv=(36,), dkv=())
    o_ref, _ = oracle.hybrid_attention(b)
    cut = 16 + 7                       # perturb every key/value row at positions > cut
    bt = b.block_tables
    for j in range(cut + 1, 36):
        blk = int(bt[0, j // 16])
        b.k_pool[blk, :, j % 16, :] = torch.randn(2, 128).to(torch.bfloat16) * 3
        b.v_pool[blk, :, j % 16, :] = torch.randn(2, 128).to(torch.bfloat16) * 3
    o_new, _ = oracle.hybrid_attention(b)
    P = 36 - 20
    for i in range(20):
        if P + i <= cut:
            assert np.array_equal(o_new[i], o_ref[i]), i
        else:
            assert not np.array_equal(o_new[i], o_ref[i]), i


# 4. invariant: split-KV partials merged by log-sum-exp equal the unsplit result
@pytest.mark.parametrize("nsplit", [2, 3, 5])
def test_split_merge_equals_unsplit(nsplit):
    b = _small(seed=4, q_lens=(1,), pkv=(1,), dkv=(203,))
    rng = np.random.default_rng(nsplit)
    L = 203
    cuts = np.sort(rng.choice(np.arange(1, L), size=nsplit - 1, replace=False))
    bounds = [0] + cuts.tolist() + [L]
    group = b.num_q_heads // b.num_kv_heads
    _, o_d = oracle.hybrid_attention(b)
    for h in range(b.num_q_heads):
        parts = [oracle.attend_range(b.q_decode[0, h], b.block_tables[1], j0, j1, h // group, b)
                 for j0, j1 in zip(bounds[:-1], bounds[1:])]
        merged = oracle.merge([p[0] for p in parts], [p[1] for p in parts],
                              np.stack([p[2] for p in parts]))
        np.testing.assert_allclose(merged, o_d[0, h], rtol=0, atol=1e-12)
    # an empty split carries no weight
    m, l, o = oracle.attend_range(b.q_decode[0, 0], b.block_tables[1], 50, 50, 0, b)
    assert m == -math.inf and l == 0.0 and not o.any()


# 5. invariant: paged and contiguous layouts give identical outputs
def test_paged_equals_contiguous():
    b = _small(seed=5, permute=False, poison=False)
    o1 = oracle.hybrid_attention(b)
    nb = b.k_pool.shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(99))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(nb)
    b.k_pool = b.k_pool[perm].clone()          # physical block i now holds old block perm[i]
    b.v_pool = b.v_pool[perm].clone()
    b.block_tables = inv[b.block_tables.long()].to(torch.int32)
    o2 = oracle.hybrid_attention(b)
    assert np.array_equal(o1[0], o2[0]) and np.array_equal(o1[1], o2[1])


# 6. independent implementation: NumPy full-matrix brute force on tiny and mixed cases
@pytest.mark.parametrize("case", [
    dict(q_lens=(4,), pkv=(4,), dkv=(4,)),                  # 4-token cases
    dict(q_lens=(4, 1), pkv=(4, 4), dkv=(4, 1, 2)),
    dict(q_lens=(5, 3), pkv=(9, 3), dkv=(1, 17, 33)),
    dict(q_lens=(17,), pkv=(50,), dkv=(16, 32, 48), Hq=8, Hkv=1),
])
def test_bruteforce_agrees(case):
    b = _small(seed=6, **case)
    o_p, o_d = oracle.hybrid_attention(b)
    r_p, r_d = bruteforce.hybrid_attention(b)
    np.testing.assert_allclose(o_p, r_p, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o_d, r_d, rtol=0, atol=1e-12)


# 7. decode is an extend of one token
def test_decode_equals_last_row_of_an_extend():
    L = 45
    b = _small(seed=7, q_lens=(6,), pkv=(L,), dkv=(L,), poison=False, permute=False)
    # make the decode sequence read the prefill sequence's blocks, and give it the chunk's last q
    b.block_tables[1] = b.block_tables[0]
    b.q_decode[0] = b.q_prefill[5]
    o_p, o_d = oracle.hybrid_attention(b)
    assert np.array_equal(o_p[5], o_d[0])


# 8. GQA equals MHA with every KV head repeated for its query group
def test_gqa_equals_mha_with_repeated_kv_heads():
    g = W.make_batch(8, 2, [7], [20], [9, 30], seed=8, poison=False)
    m = W.make_batch(8, 8, [7], [20], [9, 30], seed=8, poison=False)
    m.q_prefill, m.q_decode = g.q_prefill.clone(), g.q_decode.clone()
    m.block_tables = g.block_tables.clone()
    m.k_pool = g.k_pool.repeat_interleave(4, dim=1).clone()   # kv-head h of MHA = h // 4 of GQA
    m.v_pool = g.v_pool.repeat_interleave(4, dim=1).clone()
    a, b = oracle.hybrid_attention(g), oracle.hybrid_attention(m)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# 9. weights sum to one: constant V rows give that constant
def test_constant_value_rows_give_the_constant():
    b = _small(seed=9)
    c = torch.linspace(-2, 2, 128).to(torch.bfloat16)
    b.v_pool[:] = c
    o_p, o_d = oracle.hybrid_attention(b)
    cf = _f64(c)
    assert np.abs(o_p - cf).max() < 1e-13 and np.abs(o_d - cf).max() < 1e-13


# 10. two visible keys: the logistic closed form, including logits far beyond exp's range
@pytest.mark.parametrize("qscale", [1.0, 30.0, 300.0])
def test_two_keys_logistic_closed_form(qscale):
    b = _small(seed=10, q_lens=(2,), pkv=(2,), dkv=(2,), poison=False)
    b.q_prefill = (b.q_prefill.float() * qscale).to(torch.bfloat16)
    b.q_decode = (b.q_decode.float() * qscale).to(torch.bfloat16)
    o_p, o_d = oracle.hybrid_attention(b)
    assert np.isfinite(o_p).all() and np.isfinite(o_d).all()
    group = b.num_q_heads // b.num_kv_heads
    for which, seq, q, out in (("p", 0, b.q_prefill[1], o_p[1]), ("d", 1, b.q_decode[0], o_d[0])):
        for h in range(b.num_q_heads):
            k = _rows(b, seq, h // group, 2, pool="k")
            v = _rows(b, seq, h // group, 2)
            x = b.scale * (k @ _f64(q[h]))
            t = x[1] - x[0]
            w1 = 0.5 * (1.0 + math.tanh(t / 2))     # logistic(t), stable for any |t|
            ref = v[0] + w1 * (v[1] - v[0])
            np.testing.assert_allclose(out[h], ref, rtol=0, atol=1e-12 * max(1, np.abs(v).max()))


# 11. poisoned (NaN) slots outside the visible rows are never read
def test_poisoned_slots_are_not_read():
    b = _small(seed=11, q_lens=(13, 3), pkv=(29, 3), dkv=(1, 17, 33))
    o_p, o_d = oracle.hybrid_attention(b)
    assert np.isfinite(o_p).all() and np.isfinite(o_d).all()


# 12. sampled rows equal the corresponding rows of the full computation
def test_rows_api_matches_full():
    b = _small(seed=12)
    o_p, o_d = oracle.hybrid_attention(b)
    kinds = [0, 0, 1, 1, 0]
    idx = [0, 7, 2, 0, 5]
    heads = [3, 0, 1, 2, 2]
    r = oracle.rows(b, kinds, idx, heads)
    for t in range(5):
        ref = o_p[idx[t], heads[t]] if kinds[t] == 0 else o_d[idx[t], heads[t]]
        assert np.array_equal(r[t], ref)


def test_bad_block_index_is_an_error_not_a_read():
    b = _small(seed=13)
    b.block_tables[0, 0] = 10_000_000
    with pytest.raises(ValueError):
        oracle.hybrid_attention(b)


# worked numbers printed on the pages
def test_kv_cache_size_worked_examples():
    from hybrid_prefill_decode_gb300.roofline import kv_bytes_per_token
    cases = json.load(open(os.path.join(GOLDEN, "kv_cache_sizes.json")))["cases"]
    for c in cases:
        per_tok = kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"], c["dtype_bytes"])
        if "per_token_bytes_approx" in c:
            assert abs(per_tok / c["per_token_bytes_approx"] - 1) <= c["per_token_rel_tol"]
        total = per_tok * c["tokens"]
        assert abs(total / c["total_bytes_approx"] - 1) <= c["total_rel_tol"], (total, c)


def test_mixed_kind_worked_example_structure():
    ex = json.load(open(os.path.join(GOLDEN, "mixed_kind_example.json")))
    b = W.mixed_kind_example()
    new_tokens = b.num_prefill_tokens + b.num_decode_seqs
    assert new_tokens == ex["total_new_tokens"] == 14
    assert b.host_cu_seqlens == [0, 8, 12]
    # the extend (C) has a cached prefix, the prefill (D) has none; decodes add one token each
    assert b.prefill_kv_lens[0] > b.q_lens[0] and b.prefill_kv_lens[1] == b.q_lens[1]
    o_p, o_d = oracle.hybrid_attention(b)
    r_p, r_d = bruteforce.hybrid_attention(b)
    np.testing.assert_allclose(o_p, r_p, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o_d, r_d, rtol=0, atol=1e-12)


# ---- the non-causal reading ("Week 6: Beyond PyTorch", §"Non-Causal vs. Causal Attention":
# without the mask every token of the sequence is visible, including later tokens of the chunk)

def test_noncausal_uniform_scores_give_mean_of_all_rows():
    b = _small(seed=31, causal=False)
    b.q_prefill.zero_()
    o_p, _ = oracle.hybrid_attention(b)
    cu, group = b.host_cu_seqlens, b.num_q_heads // b.num_kv_heads
    for s in range(b.num_prefill_seqs):
        L = b.host_kv_lens[s]
        for h in range(b.num_q_heads):
            want = _rows(b, s, h // group, L).mean(axis=0)      # every row, whatever the token
            for t in range(cu[s], cu[s + 1]):
                assert np.abs(o_p[t, h] - want).max() <= 1e-12


def test_noncausal_later_rows_change_earlier_outputs():
    b = W.make_batch(2, 1, [6], [10], [], seed=32, causal=False)
    o1, _ = oracle.hybrid_attention(b)
    bt = b.block_tables
    b.v_pool[int(bt[0, 9 // 16]), 0, 9 % 16] += 1.0            # the chunk's last row
    o2, _ = oracle.hybrid_attention(b)
    assert np.abs(o2[0] - o1[0]).max() > 1e-3                # the chunk's first token sees it
    b.causal = True
    o3, _ = oracle.hybrid_attention(b)
    o4_first = o3[0].copy()
    b.v_pool[int(bt[0, 9 // 16]), 0, 9 % 16] -= 1.0
    o5, _ = oracle.hybrid_attention(b)
    assert np.array_equal(o4_first, o5[0])                   # causal: it does not


def test_noncausal_equal_queries_give_equal_rows():
    b = W.make_batch(4, 2, [7], [30], [], seed=33, causal=False)
    b.q_prefill[:] = b.q_prefill[0:1].clone()                # one query repeated on every token
    o_p, _ = oracle.hybrid_attention(b)
    for t in range(1, 7):
        assert np.array_equal(o_p[t], o_p[0])


def test_noncausal_chunk_row_equals_a_decode_over_the_sequence():
    b = W.make_batch(4, 2, [5], [21], [21], seed=34, causal=False)
    b.block_tables[1] = b.block_tables[0]                    # the decode reads the same rows
    for i in range(5):
        b.q_decode[0] = b.q_prefill[i]
        o_p, o_d = oracle.hybrid_attention(b)
        assert np.array_equal(o_d[0], o_p[i])


@pytest.mark.parametrize("case", range(3))
def test_bruteforce_agrees_noncausal(case):
    q_lens, pkv = [(4, 4), (4, 9), (1, 3, 4)][case], [(4, 4), (4, 20), (1, 7, 40)][case]
    b = W.make_batch(4, 2, list(q_lens), list(pkv), [3, 17], seed=40 + case, causal=False)
    o_p, o_d = oracle.hybrid_attention(b)
    r_p, r_d = bruteforce.hybrid_attention(b)
    assert np.abs(o_p - r_p).max() <= 1e-12 and np.abs(o_d - r_d).max() <= 1e-12


# ---- the FP8 (e4m3) cache of the decode path

def test_e4m3_decoding_matches_its_definition_and_torch():
    by_hand = {0x00: 0.0, 0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x7E: 448.0, 0xFE: -448.0,
               0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0xB8: -1.0}
    for bits, val in by_hand.items():
        assert oracle.e4m3_to_double(bits) == val, hex(bits)
    assert math.isnan(oracle.e4m3_to_double(0x7F)) and math.isnan(oracle.e4m3_to_double(0xFF))
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double()
    for bits in range(256):
        got, want = oracle.e4m3_to_double(bits), float(ref[bits])
        assert (math.isnan(got) and math.isnan(want)) or got == want, hex(bits)


def test_fp8_decode_equals_bf16_oracle_on_exact_dequantised_cache():
    fb = W.make_fp8_decode_batch(8, 2, [1, 17, 100, 333], seed=81, pow2_scales=True)
    deq = W.dequantised_batch(fb)
    # power-of-two scales: every dequantised value is exactly representable in bf16
    k_exact = fb.k8.view(torch.float8_e4m3fn).double() * fb.k_scale[None, :, None, :].double()
    assert torch.equal(deq.k_pool.double()[~torch.isnan(k_exact)], k_exact[~torch.isnan(k_exact)])
    _, ref = oracle.hybrid_attention(deq)
    got = oracle.decode_fp8(fb)
    assert np.abs(got - ref).max() <= 1e-12


def test_fp8_decode_scales_act_linearly():
    fb = W.make_fp8_decode_batch(4, 4, [40, 257], seed=82)
    base = oracle.decode_fp8(fb)
    fb.v_scale *= 2.0                                      # every V row doubles
    assert np.abs(oracle.decode_fp8(fb) - 2.0 * base).max() <= 1e-12 * max(1.0, np.abs(base).max())
    fb.v_scale /= 2.0
    fb.k_scale *= 2.0                                      # K doubles, q halves: same scores
    fb.q_decode = (fb.q_decode.double() * 0.5).to(torch.bfloat16)
    assert np.abs(oracle.decode_fp8(fb) - base).max() <= 1e-12


def test_fp8_decode_zero_query_gives_mean_of_dequantised_rows():
    fb = W.make_fp8_decode_batch(2, 1, [5, 70], seed=83)
    fb.q_decode.zero_()
    out = oracle.decode_fp8(fb)
    v = fb.v8.view(torch.float8_e4m3fn).double() * fb.v_scale[..., None].double()
    bt = fb.block_tables
    for d, L in enumerate(fb.decode_kv_lens):
        rows = torch.stack([v[int(bt[d, j // 16]), 0, j % 16] for j in range(L)])
        for h in range(2):
            assert np.abs(out[d, h] - rows.mean(dim=0).numpy()).max() <= 1e-12


# ---- the FP8 (e4m3) append: quantising the iteration's new rows into the cache

def test_e4m3_quantiser_round_trips_every_code_and_rounds_to_even():
    for code in list(range(0x00, 0x7F)) + list(range(0x80, 0xFF)):
        v = oracle.e4m3_to_double(code)
        assert oracle.e4m3_from_float(np.float32(v)) == code, hex(code)
    # midpoints between neighbours go to the even mantissa, both within a binade and across one
    for lo in (0x38, 0x39, 0x3E, 0x07, 0x00, 0x76):
        mid = (oracle.e4m3_to_double(lo) + oracle.e4m3_to_double(lo + 1)) / 2
        want = lo if lo % 2 == 0 else lo + 1
        assert oracle.e4m3_from_float(np.float32(mid)) == want, hex(lo)
        assert oracle.e4m3_from_float(np.float32(-mid)) == (want | 0x80), hex(lo)
    # saturation at 448, sign of zero kept, NaN
    assert oracle.e4m3_from_float(448.0) == 0x7E and oracle.e4m3_from_float(1e9) == 0x7E
    assert oracle.e4m3_from_float(-500.0) == 0xFE
    assert oracle.e4m3_from_float(-1e-30) == 0x80 and oracle.e4m3_from_float(0.0) == 0x00
    assert oracle.e4m3_from_float(float("nan")) == 0x7F


def test_e4m3_quantiser_matches_torch_in_range():
    g = torch.Generator().manual_seed(91)
    x = (torch.randn(20000, generator=g) * torch.exp2(torch.randint(-12, 8, (20000,),
                                                                     generator=g).float()))
    x = x.clamp(-440.0, 440.0)
    want = x.to(torch.float8_e4m3fn).view(torch.uint8)
    got = torch.tensor([oracle.e4m3_from_float(float(v)) for v in x], dtype=torch.uint8)
    assert torch.equal(got, want)


def test_fp8_append_rebuilds_the_quantised_rows():
    """The seeded cache was quantised by torch from the same bf16 rows with the same rules
    (binary32 division, V scale = row max / 448): appending those rows again must give back the
    very bytes and scales that were removed, and touch nothing else."""
    lens = [1, 16, 17, 300]
    fb, k_new, v_new = W.fp8_append_case(8, 2, lens, seed=93)
    full = W.make_fp8_decode_batch(8, 2, lens, seed=93)
    k8, v8, vs = oracle.append_fp8(fb, k_new, v_new)
    assert np.array_equal(k8, full.k8.numpy()) and np.array_equal(v8, full.v8.numpy())
    same = np.isnan(full.v_scale.numpy()) == np.isnan(vs)
    assert same.all() and np.array_equal(vs[~np.isnan(vs)], full.v_scale.numpy()[~np.isnan(vs)])
    # and the decode over the appended cache equals the decode over the original one
    fb.k8, fb.v8 = torch.from_numpy(k8), torch.from_numpy(v8)
    fb.v_scale = torch.from_numpy(vs)
    assert np.array_equal(oracle.decode_fp8(fb), oracle.decode_fp8(full))


def test_bf16_append_places_rows_at_their_hand_computed_slots():
    """A 5-token chunk at kv_len 20 (positions 15..19) through table [3, 1], then a decode at
    kv_len 33 (position 32) through table [0, 2, 4]: the rows land at (block 3, row 15),
    (block 1, rows 0..3) and (block 4, row 0), for each kv-head, and nothing else changes."""
    Hkv, D = 2, 4
    nb = 5
    zero = torch.zeros((nb, Hkv, 16, D), dtype=torch.bfloat16)
    b = W.HybridBatch(
        num_q_heads=2, num_kv_heads=Hkv, head_dim=D, block_size=16, q_lens=[5],
        prefill_kv_lens=[20], decode_kv_lens=[33], scale=0.5,
        q_prefill=torch.zeros((5, 2, D), dtype=torch.bfloat16),
        q_decode=torch.zeros((1, 2, D), dtype=torch.bfloat16), k_pool=zero, v_pool=zero,
        block_tables=torch.tensor([[3, 1, -1], [0, 2, 4]], dtype=torch.int32),
        cu_seqlens_q=torch.tensor([0, 5], dtype=torch.int32),
        kv_lens=torch.tensor([20, 33], dtype=torch.int32))
    # new token t, kv-head g, channel c holds t*10 + g + c/8 (exact in bf16); V is its negative
    vals = torch.tensor([[[t * 10 + g + c / 8 for c in range(D)] for g in range(Hkv)]
                         for t in range(6)], dtype=torch.float32).to(torch.bfloat16)
    kp, vp = oracle.append_bf16(b, vals, -vals)
    kf = torch.from_numpy(kp.view(np.int16)).view(torch.bfloat16).float()
    vf = torch.from_numpy(vp.view(np.int16)).view(torch.bfloat16).float()
    slots = [(3, 15), (1, 0), (1, 1), (1, 2), (1, 3), (4, 0)]   # token t -> (block, row)
    expect = torch.zeros((nb, Hkv, 16, D))
    for t, (blk, row) in enumerate(slots):
        expect[blk, :, row, :] = vals[t].float()
    assert torch.equal(kf, expect) and torch.equal(vf, -expect)


def test_bf16_append_rebuilds_the_removed_rows():
    """Remove an iteration's new rows from a seeded batch (NaN in their place) and append them
    again: the pools are the original ones bit for bit, so the attention over them is too."""
    full = W.make_batch(8, 2, [37, 16], [100, 16], [1, 17, 48], seed=13)
    k_new, v_new, kp0, vp0 = W.split_off_new_rows(full)
    kp, vp = oracle.append_bf16(full, k_new, v_new, kp0, vp0)
    assert np.array_equal(kp, oracle._u16(full.k_pool)) and np.array_equal(vp, oracle._u16(full.v_pool))


def test_bf16_append_skips_a_bad_table_entry():
    b = W.make_batch(4, 1, [], [], [20], seed=2)
    bad = b.block_tables.clone()
    bad[0, 1] = b.num_blocks + 3
    b.block_tables = bad
    rows = torch.ones((1, 1, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        oracle.append_bf16(b, rows, rows)
