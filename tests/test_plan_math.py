"""CPU: the decode work plan's arithmetic, as stated for the kernels (tile t of segment (b, h) at
weighted unit K t + A (Hkv b + h + 1); CTA c takes units [ceil(cU/C), ceil((c+1)U/C)); with a
partition size, ranges end on partition multiples; without, CTA c may instead take a share by its
dispatch wave c / WV: wave v of n weighs 64 + KS (n - 1 - 2 v), and CTA c starts at unit
ceil(W(c) U / W(C)), W the weight of the CTAs before it), re-enacted in integers on random batches
and compared with the library's own ranges (pa_debug_plan_ranges, host code, no GPU).
Checks the properties the kernels rely on: every tile has exactly one owner and cta_of agrees with
the range starts; no range is empty between two tiles of one segment, so a split segment's pieces
come from consecutive CTAs; and the counting merge: each CTA walks its range as pieces, and every
piece of a split segment names the same first CTA ca and piece count np, ca names no other split
segment (its counter is the segment's), the pieces come one from each CTA ca .. ca + np - 1 (so
the count reaches np exactly once), and a CTA's pieces use its partial slots as the kernel's slot
rule says (slot 0 only by the range's first piece, slot 1 only by its last).  The GPU parity tests
check the kernels themselves."""
import random


WAVE_WEIGHT = 64


def plan(lens_blocks, Hkv, C, PT, K=4, A=4, WV=1, KS=0):
    grid = C
    B = len(lens_blocks)
    pref = [0]
    for n in lens_blocks:
        pref.append(pref[-1] + n)
    T = Hkv * pref[B]
    upref = [0]
    for n in lens_blocks:
        upref.append(upref[-1] + ((n + PT - 1) // PT if PT else 0))
    U = Hkv * upref[B] if PT else K * T + A * Hkv * B
    units = U if PT else T
    ce = min(units, C)
    if PT and ce > 0:
        per = (units + ce - 1) // ce
        ce = (units + per - 1) // per
    C = ce
    nwv = (grid + WV - 1) // WV
    wave_w = lambda v: WAVE_WEIGHT + KS * (nwv - 1 - 2 * v)
    if PT or KS == 0 or nwv < 2 or wave_w(nwv - 1) <= 0 or U * wave_w(nwv - 1) < K * C * wave_w(0):
        KS = 0

    def weight_before(c):  # the weight of CTAs 0 .. c - 1
        return c if KS == 0 else sum(wave_w(x // WV) for x in range(c))

    WC = weight_before(C)

    def cta_of_unit(x):  # the largest c < C with ceil(W(c) U / WC) <= x
        y = x * WC // U
        c = 0
        while c + 1 < C and weight_before(c + 1) <= y:
            c += 1
        return c

    def find_seq(pre, x):
        lo, hi = 0, B - 1
        while lo < hi:
            mid = (lo + hi + 1) >> 1
            if Hkv * pre[mid] <= x:
                lo = mid
            else:
                hi = mid - 1
        return lo

    nbk = lambda b: pref[b + 1] - pref[b]
    seg_start = lambda b, h: Hkv * pref[b] + h * nbk(b)

    def first_tile_at_unit(x):
        lo, hi = 0, B - 1
        while lo < hi:
            mid = (lo + hi + 1) >> 1
            if Hkv * (K * pref[mid] + A * mid) <= x:
                lo = mid
            else:
                hi = mid - 1
        b = lo
        nb = nbk(b)
        local = x - Hkv * (K * pref[b] + A * b)
        span = K * nb + A
        if span == 0:
            return Hkv * pref[b]
        h, r = local // span, local % span
        j = 0 if r <= A else (r - A + K - 1) // K
        return Hkv * pref[b] + h * nb + j

    def tile_of_unit(u):
        if u >= U:
            return T
        b = find_seq(upref, u)
        local = u - Hkv * upref[b]
        ub = upref[b + 1] - upref[b]
        return seg_start(b, local // ub) + (local % ub) * PT

    def cta_start(c):
        if PT == 0:
            return T if c >= C else first_tile_at_unit((weight_before(c) * U + WC - 1) // WC)
        return tile_of_unit(c * U // C)

    def cta_of(t):
        b = find_seq(pref, t)
        local = t - Hkv * pref[b]
        nb = nbk(b)
        h, j = local // nb, local % nb
        if PT == 0:
            return cta_of_unit(K * t + A * (Hkv * b + h + 1))
        ub = upref[b + 1] - upref[b]
        u = Hkv * upref[b] + h * ub + j // PT
        return ((u + 1) * C - 1) // U

    return dict(B=B, C=C, T=T, pref=pref, nbk=nbk, seg_start=seg_start, find_seq=find_seq, cta_start=cta_start,
                cta_of=cta_of)


def _check(lens_blocks, Hkv, C, PT, WV=1, KS=0, lib=None):
    P = plan(lens_blocks, Hkv, C, PT, WV=WV, KS=KS)
    if P["T"] == 0:
        return
    starts = [P["cta_start"](c) for c in range(P["C"] + 1)]
    if lib is not None:  # the library's host build of the same arithmetic
        got, owners = lib.pa_debug_plan_ranges(lens_blocks, Hkv, PT, 4, C, WV, KS)
        assert list(got) == starts
        assert list(owners) == [P["cta_of"](t) for t in range(P["T"])]
    assert starts[0] == 0 and starts[-1] == P["T"]
    assert all(a <= b for a, b in zip(starts, starts[1:]))
    split = set()
    for b in range(P["B"]):
        nb = P["nbk"](b)
        for h in range(Hkv if nb else 0):
            s0 = P["seg_start"](b, h)
            owners = [P["cta_of"](t) for t in range(s0, s0 + nb)]
            for t, c in zip(range(s0, s0 + nb), owners):
                assert starts[c] <= t < starts[c + 1]
            ca, cb = owners[0], owners[-1]
            assert sorted(set(owners)) == list(range(ca, cb + 1))  # consecutive, none skipped
            if ca != cb:
                split.add((b, h, ca, cb - ca + 1))
    counters = {}
    for c in range(P["C"]):
        t, t_end = starts[c], starts[c + 1]
        slots = []
        while t < t_end:  # the kernel's piece walk
            b = P["find_seq"](P["pref"], t)
            nb = P["nbk"](b)
            local = t - Hkv * P["pref"][b]
            h, j0 = local // nb, local % nb
            j1 = min(nb, j0 + (t_end - t))
            if not (j0 == 0 and j1 == nb):
                s0 = P["seg_start"](b, h)
                ca = P["cta_of"](s0)
                np_ = P["cta_of"](s0 + nb - 1) - ca + 1
                slot = 0 if j0 > 0 else 1
                assert t == starts[c] if slot == 0 else t + (j1 - j0) == t_end
                slots.append(slot)
                counters.setdefault(ca, []).append((b, h, np_, c))
            t += j1 - j0
        assert len(slots) == len(set(slots))
    merged = set()
    for ca, pieces in counters.items():
        assert len({(b, h) for b, h, _, _ in pieces}) == 1  # one split segment per counter
        b, h, np_, _ = pieces[0]
        assert all(x[2] == np_ for x in pieces) and len(pieces) == np_ >= 2
        assert sorted(x[3] for x in pieces) == list(range(ca, ca + np_))
        merged.add((b, h, ca, np_))
    assert merged == split


def test_plan_properties_on_random_batches():
    import paged_kv_cache_280_gb300 as pa

    rng = random.Random(280)
    for i in range(1500):
        B = rng.randint(1, 10)
        Hkv = rng.choice([1, 2, 4, 8])
        lens = [rng.choice([0, 0, 1, 2, 3, 5, 9, 17, 40]) for _ in range(B)]
        _check(lens, Hkv, rng.randint(1, 64), rng.choice([0, 0, 0, 1, 2, 4]), lib=pa if i % 3 == 0 else None)


def test_wave_shares_on_random_batches():
    """CTA shares skewed by dispatch wave keep every property above and agree with the library."""
    import paged_kv_cache_280_gb300 as pa

    rng = random.Random(281)
    for _ in range(600):
        B = rng.randint(1, 12)
        Hkv = rng.choice([1, 2, 4, 8])
        lens = [rng.choice([0, 1, 2, 3, 5, 9, 17, 40, 90]) for _ in range(B)]
        WV = rng.randint(1, 12)
        _check(lens, Hkv, WV * rng.randint(1, 8), 0, WV=WV, KS=rng.choice([0, 1, 2, 4, 8]), lib=pa)


def test_wave_shares_follow_the_weights():
    """On a large uniform batch the first dispatch wave takes more tiles than the last, about in the
    ratio of their weights; partitioned launches keep equal shares."""
    import numpy as np
    import paged_kv_cache_280_gb300 as pa

    lens = [50] * 64
    starts, _ = pa.pa_debug_plan_ranges(lens, 8, 0, 4, 608, 152, 2, owners=False)
    tiles = np.diff(starts)
    first, last = tiles[:152].mean(), tiles[456:].mean()
    assert abs(first / last - 70 / 58) < 0.05
    even, _ = pa.pa_debug_plan_ranges(lens, 8, 0, 4, 608, 152, 0, owners=False)
    assert np.diff(even).max() - np.diff(even).min() <= 2
    part, _ = pa.pa_debug_plan_ranges(lens, 8, 5, 4, 608, 152, 2, owners=False)
    assert len(set(np.diff(part).tolist())) <= 2  # partitions: equal numbers of them


def test_weighted_balance_spreads_segment_cost():
    # a batch of one long sequence and many one-block ones: with a segment weight the CTAs that
    # take the many short segments get fewer tiles than those inside the long one
    lens = [64] + [1] * 32
    P = plan(lens, 1, 8, 0)
    starts = [P["cta_start"](c) for c in range(P["C"] + 1)]
    tiles = [b - a for a, b in zip(starts, starts[1:])]
    assert max(tiles[:3]) > min(tiles[-3:])
