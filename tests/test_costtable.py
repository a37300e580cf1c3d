"""The plan bucket of the C ABI (bit-exact against a plain restatement of its definition) and
the host logic of the validated-latency table (no GPU: plans are planned on the host only)."""
import json
import random

import pytest

from hybrid_prefill_decode_gb300 import binding as B
from hybrid_prefill_decode_gb300 import costtable as C


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _restated_bucket(Hq, Hkv, q_lens, pkv, dkv, causal=True):
    """prefill FLOPs = 4*128*Hq per visible (query, key) pair (all q*L pairs when non-causal);
    bytes = 512 per (row, kv-head) of every sequence plus 512 per (token, q-head); buckets = bit
    length of ceil(x / unit)."""
    flops = sum(4 * 128 * Hq * ((q * (L - q) + q * (q + 1) // 2) if causal else q * L)
                for q, L in zip(q_lens, pkv))
    by = sum(L * Hkv * 512 + q * Hq * 512 for q, L in zip(q_lens, pkv))
    by += sum(L * Hkv * 512 + Hq * 512 for L in dkv)

    def bucket(x, unit):
        return ((x + unit - 1) // unit).bit_length() if x > 0 else 0
    return flops, by, bucket(flops, 1 << 30), bucket(by, 1 << 20)


@pytest.mark.parametrize("seed", range(12))
def test_plan_bucket_matches_restatement(seed):
    rng = random.Random(seed)
    Hkv = rng.choice([1, 2, 4, 8])
    Hq = Hkv * rng.choice([1, 2, 4, 8])
    q_lens = [rng.randint(1, 3000) for _ in range(rng.randint(0, 3))]
    pkv = [q + rng.randint(0, 40000) for q in q_lens]
    dkv = [rng.randint(1, 40000) for _ in range(rng.randint(0, 80))]
    if not q_lens and not dkv:
        dkv = [5]
    causal = rng.random() < 0.7
    cu = [0]
    for q in q_lens:
        cu.append(cu[-1] + q)
    maxb = max(-(-x // 16) for x in pkv + dkv)
    p = B.Plan(Hq, Hkv, cu if q_lens else [], pkv + dkv, len(dkv), 10, maxb, 0.1, num_sms=152,
               non_causal=not causal)
    b = p.bucket()
    flops, by, bf, bb = _restated_bucket(Hq, Hkv, q_lens, pkv, dkv, causal)
    assert (b["prefill_flops"], b["read_bytes"], b["bucket_flops"], b["bucket_bytes"]) == \
        (flops, by, bf, bb)
    inf = p.info()
    assert b["prefill_ctas"] == inf["num_prefill_items"] and b["decode_ctas"] == inf["num_decode_items"]
    assert b["bucket_ctas"] == (b["prefill_ctas"] + b["decode_ctas"]).bit_length()
    assert b["grid"] == inf["grid_fused"] and b["smem_per_cta"] == inf["smem_bytes"]
    assert b["tmem_cols_per_cta"] == (512 if q_lens else 0)


def _table_with(entries):
    t = C.CostTable(32, 8, 152)
    for (q_lens, pkv, dkv), times in entries:
        t.add(t.plan_for(q_lens, pkv, dkv).bucket(), times)
    return t


def test_choose_chunk_takes_the_largest_validated_chunk_within_budget():
    dec = [16384] * 19
    t = _table_with([(([256], [4096 + 256], dec), [300.0] * 10),
                     (([1024], [4096 + 1024], dec), [350.0] * 9 + [420.0]),
                     (([4096], [4096 + 4096], dec), [900.0] * 10)])
    assert t.choose_chunk(4096, [256, 1024, 4096], dec, budget_us=500) == 1024
    assert t.choose_chunk(4096, [256, 1024, 4096], dec, budget_us=410) == 256   # p99 is 420
    assert t.choose_chunk(4096, [256, 1024, 4096], dec, budget_us=100) is None
    assert t.choose_chunk(4096, [4096], dec, budget_us=1000) == 4096
    # a bucket never measured is outside the validated range
    assert t.lookup(t.plan_for([64], [200000], [3] * 500)) is None


def test_buckets_keep_their_worst_figures_and_round_trip_json():
    dec = [2048] * 4
    t = _table_with([(([512], [512 + 1000], dec), [10.0, 11.0, 12.0]),
                     (([512], [512 + 1001], dec), [20.0, 30.0, 40.0])])  # same bucket
    assert len(t.entries) == 1
    e = next(iter(t.entries.values()))
    assert (e.p50_us, e.p99_us, e.samples, e.batches) == (30.0, 40.0, 6, 2)
    t2 = C.CostTable.from_json(t.to_json())
    assert t2.entries == t.entries and (t2.num_q_heads, t2.num_kv_heads, t2.num_sms) == (32, 8, 152)
    json.loads(t.to_json())
