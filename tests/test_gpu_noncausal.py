"""GPU parity of non-causal chunks (pod_attn_options.non_causal): every chunk token attends to
all rows of its sequence. Compared element by element with the fp64 oracle's non-causal reading
(pinned in test_oracle_pins.py), through the C ABI, for the three variants; same tolerance as
the causal path."""
import numpy as np
import pytest
import torch

import oracle
from hybrid_prefill_decode_gb300 import binding as B
from hybrid_prefill_decode_gb300 import workloads as W
from test_gpu_parity import assert_close, run_and_check

pytestmark = pytest.mark.gpu

VARIANTS = ("fused", "serial", "streams")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("variant", VARIANTS)
def test_tiny_hybrid_batch_non_causal(variant):
    b = W.config(1)
    b.causal = False
    run_and_check(b, variant)


CASES = {
    "fresh_ragged": dict(Hq=4, Hkv=4, q=[1, 127, 128, 129], pkv=[1, 127, 128, 129], dkv=[]),
    "after_prefix": dict(Hq=8, Hkv=2, q=[5, 130, 300], pkv=[21, 400, 1000], dkv=[33]),
    "gqa8_mixed": dict(Hq=32, Hkv=4, q=[260], pkv=[1300], dkv=[17, 900, 2000]),
    "mha_mixed": dict(Hq=8, Hkv=8, q=[64, 200], pkv=[64, 900], dkv=[1, 257]),
}


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", sorted(CASES))
def test_non_causal_edge_cases(name, variant):
    c = CASES[name]
    b = W.make_batch(c["Hq"], c["Hkv"], c["q"], c["pkv"], c["dkv"],
                     seed=sum(map(ord, name)), causal=False)
    run_and_check(b, variant)


def test_non_causal_forced_splits_and_few_ctas():
    b = W.make_batch(16, 4, [700], [3000], [2500] * 5, seed=61, causal=False)
    run_and_check(b, "fused", num_sms=3, prefill_splits=3, decode_splits=4)


def test_non_causal_differs_from_causal_only_where_later_rows_exist():
    """The last token of a chunk sees the same rows either way: identical output bits."""
    b = W.make_batch(8, 2, [100], [600], [], seed=62, device="cuda")
    o_c, _ = B.hybrid_attention(b)
    b.causal = False
    o_n, _ = B.hybrid_attention(b)
    assert torch.equal(o_c[-1].view(torch.int16), o_n[-1].view(torch.int16))
    assert not torch.equal(o_c[0].view(torch.int16), o_n[0].view(torch.int16))


def test_non_causal_full_size_sampled():
    """Configuration 3's shapes, non-causal, in the benchmark's launch configuration: sampled
    prefill rows of every head and every decode row against the oracle."""
    b = W.config(3, device="cuda")
    b.causal = False
    o_p, o_d = B.hybrid_attention(b)
    torch.cuda.synchronize()
    cpu = b.to("cpu")
    rows = sorted({0, 1, 127, 128, 500, b.num_prefill_tokens - 1})
    Hq = b.num_q_heads
    kinds = [0] * (len(rows) * Hq) + [1] * (8 * Hq)
    idx = [r for r in rows for _ in range(Hq)] + [d for d in range(8) for _ in range(Hq)]
    heads = list(range(Hq)) * (len(rows) + 8)
    ref = oracle.rows(cpu, kinds, idx, heads)
    got = torch.stack([o_p[r, h] for r in rows for h in range(Hq)] +
                      [o_d[d, h] for d in range(8) for h in range(Hq)])
    assert_close(got, ref, "non-causal config 3")
