"""GPU calibration of the validated-latency table through the C ABI on a small grid."""
import pytest

from hybrid_prefill_decode_gb300 import costtable as C
from hybrid_prefill_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_calibration_gives_lookups_for_the_measured_batches():
    t = C.calibrate(8, 2, chunks=[128, 1024], prefixes=[2048], decode_counts=[4], decode_ctx=4096,
                    iters=5, warmup=3)
    assert 1 <= len(t.entries) <= 2
    for e in t.entries.values():
        assert 0 < e.p50_us <= e.p99_us and e.samples == 5 * e.batches
    # a batch of a calibrated shape finds its bucket
    dl = [max(1, 2048 + (4096 * k) // 4) for k in range(4)]
    plan = t.plan_for([1024], [2048 + 1024], dl)
    assert t.lookup(plan) is not None
    c = t.choose_chunk(2048, [128, 1024], dl, budget_us=1e9)
    assert c == 1024
