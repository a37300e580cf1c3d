"""The seeded input generators: determinism, the shapes and length ranges of each configuration,
disjoint paged blocks, NaN poisoning outside the visible rows, and the trace scheduler's
token budget (decodes first, then prompt chunks; "LLMSO - W4", §"Prefill-Decode 분리 스케줄링")."""
import math

import torch

from hybrid_prefill_decode_gb300 import workloads as W


def _nan(t):
    return torch.isnan(t.float())


def test_generation_is_deterministic():
    a = W.make_batch(4, 2, [5, 9], [20, 9], [33, 1], seed=3)
    b = W.make_batch(4, 2, [5, 9], [20, 9], [33, 1], seed=3)
    c = W.make_batch(4, 2, [5, 9], [20, 9], [33, 1], seed=4)
    for k in ("q_prefill", "q_decode", "k_pool", "v_pool", "block_tables"):
        assert torch.equal(getattr(a, k).view(torch.int16) if getattr(a, k).dtype == torch.bfloat16
                           else getattr(a, k),
                           getattr(b, k).view(torch.int16) if getattr(b, k).dtype == torch.bfloat16
                           else getattr(b, k)), k
    assert not torch.equal(a.q_prefill.view(torch.int16), c.q_prefill.view(torch.int16))


def test_blocks_disjoint_and_poisoned_outside_visible_rows():
    b = W.make_batch(4, 2, [5, 40], [20, 40], [33, 1, 16], seed=7)
    lens = b.host_kv_lens
    seen = set()
    for s, L in enumerate(lens):
        n = (L + 15) // 16
        ids = b.block_tables[s, :n].tolist()
        assert not (set(ids) & seen)
        seen |= set(ids)
        # visible rows finite, the rest of the last block NaN
        for j in range(n * 16):
            row = b.k_pool[ids[j // 16], :, j % 16]
            assert bool(_nan(row).all()) == (j >= L)
        # table tail points at a poisoned spare block
        if b.block_tables.shape[1] > n:
            assert _nan(b.k_pool[int(b.block_tables[s, n])]).all()
    spare = set(range(b.num_blocks)) - seen
    assert spare and all(_nan(b.v_pool[i]).all() for i in spare)
    assert len(spare) >= math.ceil(0.05 * len(seen))


def test_configuration_shapes():
    for i, (hq, hkv) in {1: (2, 1), 2: (32, 32), 3: (32, 8), 4: (32, 4)}.items():
        Hq, Hkv, ql, pkv, dkv = W.config_lengths(i)
        assert (Hq, Hkv) == (hq, hkv)
    _, _, ql, pkv, dkv = W.config_lengths(1)
    assert ql == [64] and pkv == [128] and dkv == [100, 150, 233, 300]
    _, _, ql, pkv, dkv = W.config_lengths(2)
    assert ql == [512] and pkv == [4096] and len(dkv) == 32
    assert all(2048 <= x <= 4096 for x in dkv)
    _, _, ql, pkv, dkv = W.config_lengths(3)
    assert ql == [1024] and 1024 <= pkv[0] <= 15360 + 1024 and len(dkv) == 64
    assert all(8192 <= x <= 16384 for x in dkv)
    _, _, ql, pkv, dkv = W.config_lengths(4)
    assert ql == [2048] and pkv == [28672 + 2048] and len(dkv) == 16
    assert all(16384 <= x <= 32768 for x in dkv)


def test_inputs_are_standard_normal():
    b = W.make_batch(8, 2, [256], [256], [512] * 4, seed=1, poison=False)
    x = torch.cat([b.q_prefill.float().flatten(), b.k_pool.float().flatten()])
    assert abs(float(x.mean())) < 0.02 and abs(float(x.std()) - 1) < 0.02


def test_trace_budget_and_mix_properties():
    for mix, mean_out in (("a", 256), ("b", 64)):
        tr = W.trace(mix)
        assert len(tr.steps) == 200
        targets = (19, 38, 56, 75)
        for i, st in enumerate(tr.steps):
            nd = len(st.decode_kv_lens)
            assert nd == targets[(i * 4) // 200]           # decodes held at the target
            assert nd + sum(st.q_lens) == 2048             # budget filled: decodes first
            for q, L in zip(st.q_lens, st.prefill_kv_lens):
                assert 1 <= q <= L <= 32768
            assert all(4096 < L <= 32768 + 5000 for L in st.decode_kv_lens)
            assert len(st.prefill_rids) == len(st.q_lens)
            assert len(st.decode_rids) == nd and len(set(st.decode_rids)) == nd
        prompts = [n for n in tr.max_rows]
        assert all(4096 <= n for n in prompts)


def test_trace_pool_maps_requests_to_disjoint_blocks():
    tr = W.trace("a", iters=4, budget=300, decode_targets=(5,))
    tr.max_rows = [min(n, 200) for n in tr.max_rows]
    for st in tr.steps:
        st.decode_kv_lens = [min(x, 200) for x in st.decode_kv_lens]
        st.prefill_kv_lens = [min(x, 200) for x in st.prefill_kv_lens]
        st.q_lens = [min(q, L) for q, L in zip(st.q_lens, st.prefill_kv_lens)]
    pool = W.TracePool(tr, device="cpu", num_q_heads=4, num_kv_heads=2)
    all_ids = torch.cat(pool.blocks)
    assert all_ids.unique().numel() == all_ids.numel() == pool.k_pool.shape[0]
    b = pool.batch(2)
    for r, L in enumerate(b.host_kv_lens):
        n = (L + 15) // 16
        assert b.block_tables[r, :n].tolist() == pool.blocks[
            (tr.steps[2].prefill_rids + tr.steps[2].decode_rids)[r]][:n].tolist()


def test_split_off_new_rows_is_a_gather_of_the_iteration_tokens():
    b = W.make_batch(4, 2, [5, 9], [20, 9], [33, 1, 16], seed=11)
    k_new, v_new, kp, vp = W.split_off_new_rows(b)
    # positions written out by hand: chunk tokens follow the cached prefix, a decode token is
    # the sequence's last row
    want = [(0, p) for p in range(15, 20)] + [(1, p) for p in range(0, 9)] + \
        [(2, 32), (3, 0), (4, 15)]
    assert k_new.shape == (len(want), 2, 128)
    bt = b.block_tables
    holes = torch.zeros(b.k_pool.shape[:3], dtype=torch.bool)
    for i, (s, p) in enumerate(want):
        blk = int(bt[s, p // 16])
        for g in range(2):
            assert torch.equal(k_new[i, g].view(torch.int16), b.k_pool[blk, g, p % 16].view(torch.int16))
            assert torch.equal(v_new[i, g].view(torch.int16), b.v_pool[blk, g, p % 16].view(torch.int16))
        holes[blk, :, p % 16] = True
    # the returned pools differ from the batch's exactly at those rows, which are NaN there
    assert _nan(kp[holes]).all() and _nan(vp[holes]).all()
    assert torch.equal(kp[~holes].view(torch.int16), b.k_pool[~holes].view(torch.int16))
    assert torch.equal(vp[~holes].view(torch.int16), b.v_pool[~holes].view(torch.int16))
