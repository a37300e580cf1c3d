"""Seeded random batches across the library's whole input space, every output element against
the fp64 oracle (|err| <= 2e-2 + 2e-2 |ref|): group sizes 1-8, head dims 128 and 64, causal and
non-causal chunks, 0-3 chunks with ragged lengths and prefixes, 0-20 decodes, the three launch
variants, automatic or forced KV splits, small SM counts (long persistent loops)."""
import random

import numpy as np
import pytest
import torch

import oracle
from hybrid_prefill_decode_gb300 import binding as B
from hybrid_prefill_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _case(seed):
    rng = random.Random(seed)
    Hkv = rng.choice([1, 2, 4])
    G = rng.choice([1, 2, 3, 4, 8])
    head_dim = rng.choice([128, 128, 64])
    causal = rng.random() < 0.75
    np_ = rng.choice([0, 1, 1, 2, 3])
    nd = rng.choice([0, 1, 5, 20]) if np_ else rng.choice([1, 5, 20])
    q = [rng.choice([1, rng.randint(2, 130), rng.randint(130, 300)]) for _ in range(np_)]
    pkv = [x + rng.choice([0, rng.randint(1, 200), rng.randint(200, 2000)]) for x in q]
    dkv = [rng.choice([1, rng.randint(2, 40), rng.randint(40, 3000)]) for _ in range(nd)]
    opts = {}
    if rng.random() < 0.3:
        opts["decode_splits"] = rng.choice([2, 5, 64])
    if rng.random() < 0.3:
        opts["prefill_splits"] = rng.choice([2, 3, 8])
    if rng.random() < 0.25:
        opts["num_sms"] = rng.choice([1, 3, 17])
    variant = rng.choice(["fused", "fused", "serial", "streams"])
    return Hkv * G, Hkv, q, pkv, dkv, head_dim, causal, variant, opts


@pytest.mark.parametrize("seed", range(96))
def test_random_batch_against_oracle(seed):
    Hq, Hkv, q, pkv, dkv, hd, causal, variant, opts = _case(seed)
    b = W.make_batch(Hq, Hkv, q, pkv, dkv, seed=1000 + seed, causal=causal, head_dim=hd)
    ref_p, ref_d = oracle.hybrid_attention(b)
    o_p, o_d = B.hybrid_attention(b.to("cuda"), variant=variant, **opts)
    torch.cuda.synchronize()
    for got, ref, what in ((o_p, ref_p, "prefill"), (o_d, ref_d, "decode")):
        g = got.float().cpu().numpy().astype(np.float64)
        assert g.shape == ref.shape
        err = np.abs(g - ref)
        assert np.isfinite(g).all(), (seed, what)
        assert (err <= 2e-2 + 2e-2 * np.abs(ref)).all(), (seed, what, float(err.max()),
                                                          (Hq, Hkv, q, pkv, dkv, hd, causal,
                                                           variant, opts))
