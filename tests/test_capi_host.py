"""Host-side checks of the C ABI (no GPU): the library loads, exports every declared symbol,
validates its arguments, and its planner matches a plain Python restatement bit for bit."""
import ctypes
import math
import random

import pytest

from hybrid_prefill_decode_gb300 import binding as B
from hybrid_prefill_decode_gb300 import workloads as W


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return B.load()


def test_library_exports_every_declared_symbol(lib):
    names = B.declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(-6, 1):
        assert lib.pod_attn_status_string(code)


def _plan_code(Hq=4, Hkv=2, cu=(0, 5), kv=(9, 7), nd=1, nb=10, maxb=4, head_dim=128,
               block=16, scale=0.1, variant=0):
    lib = B.load()
    np_ = max(0, len(cu) - 1)
    prob = B.Problem(Hq, Hkv, head_dim, block, np_, cu[-1] if np_ else 0, nd, nb, maxb, scale)
    opt = B.Options(148, 0, 0, 0, 0, 0, variant)
    cua = (ctypes.c_int32 * max(1, len(cu)))(*cu)
    kva = (ctypes.c_int32 * max(1, len(kv)))(*kv)
    h = ctypes.c_void_p()
    code = lib.pod_attn_plan(ctypes.byref(prob), ctypes.cast(cua, ctypes.c_void_p),
                             ctypes.cast(kva, ctypes.c_void_p), ctypes.byref(opt),
                             ctypes.byref(h))
    if code == 0:
        lib.pod_attn_plan_destroy(h)
    return code


def test_plan_validation(lib):
    assert _plan_code() == B.OK
    assert _plan_code(head_dim=64) == B.OK                          # 128 and 64 supported
    assert _plan_code(head_dim=96) == B.ERR_UNSUPPORTED
    assert _plan_code(head_dim=256) == B.ERR_UNSUPPORTED
    assert _plan_code(block=32) == B.ERR_UNSUPPORTED
    assert _plan_code(Hq=18, Hkv=1) == B.ERR_UNSUPPORTED          # group 18 > 8
    assert _plan_code(Hq=6, Hkv=4) == B.ERR_INVALID_ARG           # Hq % Hkv != 0
    assert _plan_code(cu=(0, 5), kv=(4, 7)) == B.ERR_INVALID_ARG  # kv_len < q_len
    assert _plan_code(cu=(1, 5), kv=(9, 7)) == B.ERR_INVALID_ARG  # cu[0] != 0
    assert _plan_code(cu=(0, 5, 5), kv=(9, 9, 7)) == B.ERR_INVALID_ARG  # empty chunk
    assert _plan_code(kv=(9, 0)) == B.ERR_INVALID_ARG             # decode kv_len 0
    assert _plan_code(kv=(9, 65)) == B.ERR_INVALID_ARG            # beyond max_blocks_per_seq*16
    assert _plan_code(variant=7) == B.ERR_INVALID_ARG
    assert _plan_code(scale=0.0) == B.ERR_INVALID_ARG               # scale must be > 0
    assert _plan_code(scale=-0.1) == B.ERR_INVALID_ARG
    assert _plan_code(scale=float("inf")) == B.ERR_INVALID_ARG
    assert _plan_code(cu=(), kv=(), nd=0) == B.OK                  # empty batch is legal
    assert _plan_code(cu=(), kv=(3,), nd=1) == B.OK                # decode only
    assert _plan_code(cu=(0, 5), kv=(9,), nd=0) == B.OK            # prefill only
    assert lib.pod_attn_plan(None, None, None, None, None) == B.ERR_INVALID_ARG
    assert lib.pod_attn_workspace_bytes(None) == 0
    lib.pod_attn_plan_destroy(None)


def test_run_append_rejects_missing_rows(lib):
    p = B.Plan(4, 2, [0, 5], [9, 7], 1, 10, 4, 0.1, num_sms=148)
    for kn, vn in ((None, 16), (16, None), (None, None)):
        code = lib.pod_attn_run_append(p.handle, None, None, kn, vn, None, None, None, None,
                                       None, None, None, None, 0, None, None)
        assert code == B.ERR_INVALID_ARG


def test_run_rejects_bad_workspace(lib):
    p = B.Plan(4, 2, [0, 5], [9, 7], 1, 10, 4, 0.1, num_sms=148)
    code = lib.pod_attn_run(p.handle, None, None, None, None, None, None, None, None, None,
                            None, 0, None, None)
    assert code == B.ERR_INVALID_ARG
    code = lib.pod_attn_run(p.handle, None, None, None, None, None, None, None, None, None,
                            257, 1 << 20, None, None)
    assert code == B.ERR_WORKSPACE        # misaligned
    code = lib.pod_attn_upload(p.handle, 256, 16, None)
    assert code == B.ERR_WORKSPACE        # too small


# ---- the planner restated in plain Python (integer arithmetic, same rules) -----------------
def _cdiv(a, b):
    return -(-a // b)


def _wave_span(costs, slots):
    """Items taken longest first by `slots` groups, wave by wave: the sum over waves of the
    wave's longest item (costs sorted longest first)."""
    return sum(costs[w] for w in range(0, len(costs), slots))


def _rebalanced(nblk, c):
    ns = max(1, min(_cdiv(nblk, c), nblk))
    chunk = _cdiv(nblk, ns)
    return _cdiv(nblk, chunk), chunk


def _bucket(steps):
    """Cost buckets of the prefill order: exact below 16 steps, above that the bit length and
    the next three bits (so two costs share a bucket when they differ by under ~12 %)."""
    if steps < 16:
        return steps
    bl = steps.bit_length()
    return 16 + (bl - 5) * 8 + ((steps >> (bl - 4)) & 7)


def _list_span(costs, slots):
    """Items taken longest first, each by the slot that frees first: the last finish time."""
    free = [0] * slots
    for x in sorted(costs, reverse=True):
        i = min(range(slots), key=free.__getitem__)
        free[i] += x
    return max(free)


def restated_prefill_chunk(nts, num_sms):
    """Prefill: the chunk ceil(longest / k), k = 1..8, that minimises the makespan of the items
    (steps + 8 each) taken longest first by one slot per SM, each going to the slot that frees
    first; chunks under 4 steps are not tried (but k = 1 always is); ties keep the larger
    chunk."""
    longest = max(nts)
    best, best_c, prev = None, 0, None
    for k in range(1, 9):
        c = _cdiv(longest, k)
        if c == prev:
            continue
        if k > 1 and c < 4:
            break
        prev = c
        items = []
        for n in nts:
            ns, ch = _rebalanced(n, c)
            items += [min(n, (j + 1) * ch) - j * ch + 8 for j in range(ns)]
        t = _list_span(items, num_sms)
        if best is None or t < best:
            best, best_c = t, c
    return best_c


def restated_decode_only_chunk(nblks, num_sms, kv_fp8):
    """Decode-only plans: the chunk ceil(longest / k), k in the divisor list, that minimises the
    wave-by-wave makespan over (3 or 4) x SMs groups of items costing ceil(blocks / 4) + 2;
    chunks under 12 blocks are not tried (but k = 1 always is), the search stops past four
    waves of items, and ties keep the larger chunk."""
    groups = num_sms * (4 if kv_fp8 else 3)
    longest = max(nblks)
    best, best_c, prev = None, 0, None
    for k in (1, 2, 3, 4, 5, 6, 8, 10, 12, 16, 20, 24, 32, 40, 48, 64):
        c = _cdiv(longest, k)
        if c == prev or (k > 1 and c < 12):
            continue
        prev = c
        items = []
        for n in nblks:
            ns, ch = _rebalanced(n, c)
            items += [_cdiv(min(n, (j + 1) * ch) - j * ch, 4) + 2 for j in range(ns)]
        if k > 1 and len(items) > 4 * groups:
            break
        t = _wave_span(sorted(items, reverse=True), groups)
        if best is None or t < best:
            best, best_c = t, c
    return best_c


def restated_plan(Hq, Hkv, cu, kv, nd, num_sms, psplit=0, dsplit=0, causal=True, kv_fp8=False,
                  prefill_cap=0):
    """Items: prefill = (chunk, query tile of 128/hp tokens x hp heads, first head, split) over
    128-key steps of the tile (cost 57 each), with hp the largest power of two
    dividing the group size; decode = (sequence, kv-head, split) over 16-row blocks (cost 8
    each); two item slots per SM; split when an output costs more than a quarter of a slot's
    share."""
    np_ = len(cu) - 1 if cu else 0
    slots = num_sms * 2
    G = Hq // Hkv
    hp = max(x for x in (1, 2, 4, 8) if G % x == 0)
    tile = 128 // hp                                              # tokens of one prefill item
    pu, du, total = [], [], 0
    for s in range(np_):
        q, L = cu[s + 1] - cu[s], kv[s]
        P = L - q
        for t in range(_cdiv(q, tile)):
            kend = P + min(q, (t + 1) * tile) if causal else L    # non-causal: every row
            nt = _cdiv(kend, 128)
            for h in range(0, Hq, hp):
                pu.append((s, t, h, kend, nt))
                total += nt * 57
    for d in range(nd):
        L = kv[np_ + d]
        for g in range(Hkv):
            du.append((d, g, L, _cdiv(L, 16)))
            total += _cdiv(L, 16) * 8
    target = max(1, total // (slots * 4))
    prefill_ctas = min(prefill_cap, num_sms) if prefill_cap > 0 else num_sms
    chunk_p = restated_prefill_chunk([x[4] for x in pu], prefill_ctas) if pu and not psplit else 0
    units, lp, ld = [], [], []
    slots_used = [0, 0]

    def add_unit(ns, kind):
        u = len(units)
        units.append([ns, slots_used[kind], kind, 0])
        slots_used[kind] += ns
        return u

    for s, t, h, kend, nt in pu:
        if chunk_p:
            ns, chunk = _rebalanced(nt, chunk_p)
        else:
            ns = max(1, min(psplit, nt, 8))
            chunk = _cdiv(nt, ns)
            ns = _cdiv(nt, chunk)
        u = add_unit(ns, 0) if ns > 1 else -1
        for k in range(ns):
            t0, t1 = k * chunk, min(nt, (k + 1) * chunk)
            lp.append(((t1 - t0) * 57, [0, s, t, h, t0 * 128, min(kend, t1 * 128), u, k]))
    chunk_do = (restated_decode_only_chunk([x[3] for x in du], num_sms, kv_fp8)
                if not pu and du and not dsplit else 0)
    for d, g, L, nblk in du:
        if chunk_do:
            ns = _cdiv(nblk, chunk_do)
        elif dsplit:
            ns = min(dsplit, 64)
        else:
            ns = min(_cdiv(nblk * 8, target), max(1, nblk // 12), 64)
        ns = max(1, min(ns, nblk))
        chunk = _cdiv(nblk, ns)
        ns = _cdiv(nblk, chunk)
        u = add_unit(ns, 1) if ns > 1 else -1
        for k in range(ns):
            b0, b1 = k * chunk, min(nblk, (k + 1) * chunk)
            ld.append(((b1 - b0) * 8, [1, d, g, 0, b0 * 16, min(L, b1 * 16), u, k]))
    # prefill: cost in a coarse relative bucket (3 significant bits), then split index; decode:
    # cost; both stable (ties in enumeration order)
    lp.sort(key=lambda x: (-_bucket(x[0] // 57), x[1][7]))
    ld.sort(key=lambda x: -x[0])
    return ([w for _, w in lp], [w for _, w in ld], units, prefill_ctas,
            min(num_sms, len(lp) + len(ld)))


def _random_case(rng):
    Hkv = rng.choice([1, 2, 4, 8])
    Hq = Hkv * rng.choice([1, 2, 3, 4, 8])
    np_ = rng.randint(0, 3)
    nd = rng.randint(0, 40)
    q_lens = [rng.randint(1, 700) for _ in range(np_)]
    pkv = [q + rng.randint(0, 9000) for q in q_lens]
    dkv = [rng.randint(1, 20000) for _ in range(nd)]
    return Hq, Hkv, q_lens, pkv, dkv


@pytest.mark.parametrize("seed", range(12))
def test_planner_matches_python_restatement(lib, seed):
    rng = random.Random(seed)
    Hq, Hkv, q_lens, pkv, dkv = _random_case(rng)
    cu = [0]
    for q in q_lens:
        cu.append(cu[-1] + q)
    num_sms = rng.choice([148, 152, 7])
    psplit = rng.choice([0, 0, 3])
    dsplit = rng.choice([0, 0, 5, 100])
    pcap = rng.choice([0, 0, 1, 5, 500])
    maxb = _cdiv(max(pkv + dkv + [1]), 16)
    p = B.Plan(Hq, Hkv, cu if q_lens else [], pkv + dkv, len(dkv), 100, maxb, 0.1,
               num_sms=num_sms, prefill_splits=psplit, decode_splits=dsplit,
               max_prefill_ctas=pcap)
    got_p, got_d, got_u = p.items()
    exp_p, exp_d, exp_u, cap, grid = restated_plan(Hq, Hkv, cu if q_lens else [], pkv + dkv,
                                                   len(dkv), num_sms, psplit=psplit,
                                                   dsplit=dsplit, prefill_cap=pcap)
    assert got_p == exp_p
    assert got_d == exp_d
    assert got_u == exp_u
    inf = p.info()
    assert inf["max_prefill_ctas"] == cap and inf["grid_fused"] == grid


@pytest.mark.parametrize("seed", range(10))
def test_decode_only_planner_matches_restatement(lib, seed):
    """Decode-only batches take the wave-aware chunk rule (both caches, both SM counts)."""
    rng = random.Random(1000 + seed)
    Hkv = rng.choice([1, 2, 4, 8])
    Hq = Hkv * rng.choice([1, 2, 4, 8])
    nd = rng.randint(1, 80)
    lo = rng.choice([1, 500, 8000])
    dkv = [rng.randint(lo, lo + rng.choice([100, 5000, 30000])) for _ in range(nd)]
    num_sms = rng.choice([152, 148, 7])
    kv_fp8 = bool(seed % 2)
    maxb = _cdiv(max(dkv), 16)
    p = B.Plan(Hq, Hkv, [], dkv, nd, 100, maxb, 0.1, num_sms=num_sms, kv_fp8=kv_fp8)
    got_p, got_d, got_u = p.items()
    exp_p, exp_d, exp_u, _, grid = restated_plan(Hq, Hkv, [], dkv, nd, num_sms, kv_fp8=kv_fp8)
    assert got_p == [] and got_d == exp_d and got_u == exp_u
    assert p.info()["grid_fused"] == grid


def test_decode_only_rule_avoids_a_near_empty_last_wave():
    """16 long decodes x 4 kv-heads on 152 SMs: the W / (4 S) rule would cut about 1250 equal
    items (2.05 waves of 608 FP8 groups); the wave-aware rule keeps the modelled makespan of its
    choice no worse than any other candidate's, including the old rule's chunk."""
    dkv = [16384 + (16384 * k) // 16 for k in range(16)]
    nblks = [_cdiv(L, 16) for L in dkv for _ in range(4)]
    target = sum(n * 8 for n in nblks) // (304 * 4)

    def span(split):
        items = []
        for n in nblks:
            ns, ch = split(n)
            items += [_cdiv(min(n, (j + 1) * ch) - j * ch, 4) + 2 for j in range(ns)]
        return _wave_span(sorted(items, reverse=True), 608), len(items)

    def old(n):
        ns = max(1, min(_cdiv(n * 8, target), max(1, n // 12), 64, n))
        ch = _cdiv(n, ns)
        return _cdiv(n, ch), ch

    c = restated_decode_only_chunk(nblks, 152, True)
    new_span, _ = span(lambda n: _rebalanced(n, c))
    old_span, old_items = span(old)
    assert 608 * 2 < old_items < 608 * 2.1
    assert new_span < old_span


@pytest.mark.parametrize("seed", range(6))
def test_planner_matches_python_restatement_non_causal(lib, seed):
    rng = random.Random(100 + seed)
    Hq, Hkv, q_lens, pkv, dkv = _random_case(rng)
    cu = [0]
    for q in q_lens:
        cu.append(cu[-1] + q)
    maxb = _cdiv(max(pkv + dkv + [1]), 16)
    p = B.Plan(Hq, Hkv, cu if q_lens else [], pkv + dkv, len(dkv), 100, maxb, 0.1,
               num_sms=152, non_causal=True)
    got_p, got_d, got_u = p.items()
    exp_p, exp_d, exp_u, _, _ = restated_plan(Hq, Hkv, cu if q_lens else [], pkv + dkv,
                                              len(dkv), 152, causal=False)
    assert (got_p, got_d, got_u) == (exp_p, exp_d, exp_u)
    ends = {}                                         # every prefill tile reads all rows
    for it in got_p:
        ends[(it[1], it[2], it[3])] = max(ends.get((it[1], it[2], it[3]), 0), it[5])
    assert all(e == pkv[k[0]] for k, e in ends.items())


@pytest.mark.parametrize("i", [1, 2, 3, 4])
def test_planner_covers_every_key_once(lib, i):
    """Structural invariant: the items of each output tile exactly [0, visible end) in order."""
    Hq, Hkv, q_lens, pkv, dkv = W.config_lengths(i)
    cu = [0]
    for q in q_lens:
        cu.append(cu[-1] + q)
    p = B.Plan(Hq, Hkv, cu, pkv + dkv, len(dkv), 10, _cdiv(max(pkv + dkv), 16), 0.1,
               num_sms=152)
    hp = max(x for x in (1, 2, 4, 8) if (Hq // Hkv) % x == 0)   # heads per prefill tile
    tile = 128 // hp                                              # tokens per prefill item
    items_p, items_d, units = p.items()
    cover = {}
    for it in items_p + items_d:
        key = tuple(it[:4])
        cover.setdefault(key, []).append((it[7], it[4], it[5], it[6]))
    for key, parts in cover.items():
        parts.sort()
        assert parts[0][1] == 0
        for a, b in zip(parts, parts[1:]):
            assert a[2] == b[1]                      # contiguous key ranges
        if len(parts) > 1:
            u = parts[0][3]
            assert all(x[3] == u for x in parts) and units[u][0] == len(parts)
        kind, seq = key[0], key[1]
        if kind == 1:
            assert parts[-1][2] == dkv[seq]
        else:
            t = key[2]
            q = q_lens[seq]
            assert parts[-1][2] == pkv[seq] - q + min(q, (t + 1) * tile)
            assert key[3] % hp == 0
    # every (tile, block of hp heads) and (decode seq, kv-head) appears
    assert len([k for k in cover if k[0] == 0]) == sum(_cdiv(q, tile) for q in q_lens) * (Hq // hp)
    assert len([k for k in cover if k[0] == 1]) == len(dkv) * Hkv


def test_workspace_grows_with_instrumentation(lib):
    a = B.Plan(32, 8, [0, 1024], [9000] + [5000] * 10, 10, 4000, 600, 0.1, num_sms=148)
    b = B.Plan(32, 8, [0, 1024], [9000] + [5000] * 10, 10, 4000, 600, 0.1, num_sms=148,
               instrument=True)
    n = a.info()["num_prefill_items"] + a.info()["num_decode_items"]
    assert b.workspace_bytes - a.workspace_bytes >= n * ctypes.sizeof(B.ItemRecord)



def test_run_decode_fp8_validation(lib):
    big = 1 << 40
    # a plan with prefill work is not an FP8 decode plan
    p = B.Plan(4, 2, [0, 5], [9, 7], 1, 10, 4, 0.1, num_sms=148, kv_fp8=True)
    code = lib.pod_attn_run_decode_fp8(p.handle, *([None] * 8), 256, big, None)
    assert code == B.ERR_UNSUPPORTED
    # head dim 64 is not built for the FP8 cache
    p64 = B.Plan(4, 2, [], [7], 1, 10, 4, 0.1, num_sms=148, head_dim=64, kv_fp8=True)
    code = lib.pod_attn_run_decode_fp8(p64.handle, *([None] * 8), 256, big, None)
    assert code == B.ERR_UNSUPPORTED
    # a plan made for the bf16 cache is not an FP8 plan, and an FP8 plan runs nowhere else
    d16 = B.Plan(4, 2, [], [7, 40], 2, 10, 4, 0.1, num_sms=148)
    code = lib.pod_attn_run_decode_fp8(d16.handle, *([None] * 8), 256, big, None)
    assert code == B.ERR_UNSUPPORTED
    d = B.Plan(4, 2, [], [7, 40], 2, 10, 4, 0.1, num_sms=148, kv_fp8=True)
    code = lib.pod_attn_run(d.handle, *([None] * 9), 256, big, None, None)
    assert code == B.ERR_UNSUPPORTED
    code = lib.pod_attn_run_decode_fp8(d.handle, *([None] * 8), 256, big, None)
    assert code == B.ERR_INVALID_ARG                     # missing pointers
    ptrs = [4096 * (i + 1) for i in range(8)]
    ptrs[3] += 4                                         # misaligned V scales
    code = lib.pod_attn_run_decode_fp8(d.handle, *ptrs, 256, big, None)
    assert code == B.ERR_INVALID_ARG
    code = lib.pod_attn_run_decode_fp8(d.handle, *([None] * 8), 257, big, None)
    assert code == B.ERR_WORKSPACE


def test_append_fp8_validation(lib):
    big = 1 << 40
    p16 = B.Plan(4, 2, [], [7, 40], 2, 10, 4, 0.1, num_sms=148)          # bf16-cache plan
    assert lib.pod_attn_append_fp8(p16.handle, *([None] * 7), 256, big, None) == B.ERR_UNSUPPORTED
    pp = B.Plan(4, 2, [0, 5], [9, 7], 1, 10, 4, 0.1, num_sms=148, kv_fp8=True)  # has prefill
    assert lib.pod_attn_append_fp8(pp.handle, *([None] * 7), 256, big, None) == B.ERR_UNSUPPORTED
    d = B.Plan(4, 2, [], [7, 40], 2, 10, 4, 0.1, num_sms=148, kv_fp8=True)
    assert lib.pod_attn_append_fp8(d.handle, *([None] * 7), 256, big, None) == B.ERR_INVALID_ARG
    ptrs = [4096 * (i + 1) for i in range(7)]
    ptrs[1] += 8                                                           # misaligned v_new
    assert lib.pod_attn_append_fp8(d.handle, *ptrs, 256, big, None) == B.ERR_INVALID_ARG
    assert lib.pod_attn_append_fp8(d.handle, *([None] * 7), 257, big, None) == B.ERR_WORKSPACE
    empty = B.Plan(4, 2, [], [], 0, 1, 1, 0.1, num_sms=148, kv_fp8=True)  # nothing to append
    assert lib.pod_attn_append_fp8(empty.handle, *([None] * 7), 256, big, None) == B.OK


@pytest.mark.parametrize("i,items,max_steps", [(2, 128, 32), (3, 256, 63), (4, 1024, 120)])
def test_prefill_chunk_choice_on_configs(lib, i, items, max_steps):
    """The prefill chunk rule's choice on the full-size configurations at 152 SMs: configs 2
    and 3 keep their 128 and 256 tile outputs whole; config 4 cuts its 512 outputs of ~232
    steps into 2 splits (1024 items of at most 120 steps)."""
    Hq, Hkv, q_lens, pkv, dkv = W.config_lengths(i)
    cu = [0]
    for q in q_lens:
        cu.append(cu[-1] + q)
    nb = sum(_cdiv(x, 16) for x in pkv + dkv) + 8
    p = B.Plan(Hq, Hkv, cu, pkv + dkv, len(dkv), nb, _cdiv(max(pkv + dkv), 16), 0.1,
               num_sms=152)
    items_p, _, _ = p.items()
    steps = [_cdiv(it[5] - it[4], 128) for it in items_p]
    assert len(items_p) == items
    assert max(steps) == max_steps


def test_ctas_per_sm_option(lib):
    """One persistent CTA per SM is the only layout: 0 and 1 plan, larger values are
    unsupported, negative values invalid."""
    for v in (0, 1):
        p = B.Plan(8, 2, [0, 40], [40, 90], 1, 20, 8, 0.1, num_sms=4, ctas_per_sm=v)
        assert p.info()["ctas_per_sm"] == 1
    with pytest.raises(B.PodAttnError) as e:
        B.Plan(8, 2, [0, 40], [40, 90], 1, 20, 8, 0.1, num_sms=4, ctas_per_sm=2)
    assert e.value.code == B.ERR_UNSUPPORTED
    with pytest.raises(B.PodAttnError) as e:
        B.Plan(8, 2, [0, 40], [40, 90], 1, 20, 8, 0.1, num_sms=4, ctas_per_sm=-1)
    assert e.value.code == B.ERR_INVALID_ARG


def test_max_prefill_ctas_option(lib):
    """The prefill cap is reported, bounds the prefill-only grid and sizes the prefill splits
    for that many slots (a smaller cap makes the makespan model cut outputs differently); 0 or a
    value above the SM count means every CTA; negative values are invalid."""
    cu, kv = [0, 2048], [30720] + [20000] * 4
    base = B.Plan(32, 4, cu, kv, 4, 12000, 1920, 0.1, num_sms=152, variant="serial")
    assert base.info()["max_prefill_ctas"] == 152
    for cap in (1, 3, 40):
        p = B.Plan(32, 4, cu, kv, 4, 12000, 1920, 0.1, num_sms=152, variant="serial",
                   max_prefill_ctas=cap)
        inf = p.info()
        assert inf["max_prefill_ctas"] == cap
        assert inf["grid_prefill"] == min(cap, inf["num_prefill_items"])
        exp_p, _, _, exp_cap, _ = restated_plan(32, 4, cu, kv, 4, 152, prefill_cap=cap)
        assert p.items()[0] == exp_p and exp_cap == cap
    assert B.Plan(32, 4, cu, kv, 4, 12000, 1920, 0.1, num_sms=152,
                  max_prefill_ctas=500).info()["max_prefill_ctas"] == 152
    with pytest.raises(B.PodAttnError) as e:
        B.Plan(32, 4, cu, kv, 4, 12000, 1920, 0.1, num_sms=152, max_prefill_ctas=-2)
    assert e.value.code == B.ERR_INVALID_ARG
