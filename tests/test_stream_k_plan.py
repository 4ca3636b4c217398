"""The stream-K bookkeeping of the super-tile GEMM, restated on the CPU.

The kernel cuts U = tiles x stages units into G = min(U, gridDim.x) equal
contiguous ranges (CTA c < G owns [c U / G, (c + 1) U / G); the others idle), so
that every range is non-empty.  A tile cut between CTAs is summed by its
last contributor, which counts arrivals on a ticket and reads every
contributor's partial tile from one of two slots per CTA: the "first" slot (the
cut tile that CTA's range starts inside) or the "last" slot (the cut tile its
range ends inside).  The routed product keys the ticket by the tile's first CTA
instead of by the tile, so that its workspace does not depend on the tile count
the routing kernel finds on the device.  These tests check, over many shapes,
the facts the kernel relies on:

- every unit belongs to exactly one CTA, and the search for a unit's CTA finds it;
- a CTA range ends inside at most one cut tile that starts in it, so the
  first-CTA key is unique among cut tiles;
- the ticket target (c_hi - c_lo + 1) is the number of CTAs that hold part of
  the tile;
- a CTA needs at most one "first" and one "last" partial slot;
- the span rule that decides whether the routed product uses stream-K matches
  the dense plan's (10 x stream-K span < 9 x whole-tile span, a fix-up counted
  as two stages).
"""
import random


def sk_begin(U, G, c):
    """G is the effective CTA count min(U, gridDim.x)."""
    return U if c >= G else c * U // G


def sk_cta_of_unit(U, G, u):
    """The kernel's search: an estimate, then at most 4 steps each way."""
    c = u * G // U
    if c >= G:
        c = G - 1
    for _ in range(4):
        if c > 0 and sk_begin(U, G, c) > u:
            c -= 1
    for _ in range(4):
        if c + 1 < G and sk_begin(U, G, c + 1) <= u:
            c += 1
    return c


def segments(U, G, nst, c):
    """CTA c's segments (tile, s0, s1, first) in the order seg_next walks them."""
    start, end = sk_begin(U, G, c), sk_begin(U, G, c + 1)
    nxt, out = start, []
    while nxt < end:
        t = nxt // nst
        s0 = nxt - t * nst
        left = end - nxt
        s1 = nst if nst - s0 <= left else s0 + left
        out.append((t, s0, s1, nxt == start))
        nxt += s1 - s0
    return out


def check_plan(ntiles, nst, grid):
    U = ntiles * nst
    G = min(U, grid)  # the effective CTA count; CTAs G .. grid - 1 idle
    for c in range(grid):
        assert (sk_begin(U, G, c + 1) > sk_begin(U, G, c)) == (c < G), "an empty range below G"
    owner = [None] * U
    for c in range(grid):
        for u in range(sk_begin(U, G, c), sk_begin(U, G, c + 1)):
            assert owner[u] is None
            owner[u] = c
    assert all(o is not None for o in owner)
    for u in range(U):
        assert sk_cta_of_unit(U, G, u) == owner[u]
    # per tile: its contributors and the slot each one uses
    contributors = {}
    first_slot, last_slot = {}, {}
    for c in range(grid):
        segs = segments(U, G, nst, c)
        for t, s0, s1, first in segs:
            split = s0 > 0 or s1 < nst
            if not split:
                continue
            contributors.setdefault(t, []).append(c)
            slot = first_slot if first else last_slot
            assert c not in slot, "a CTA needs a second partial slot of one kind"
            slot[c] = t
    keys = {}
    for t, cs in contributors.items():
        c_lo = sk_cta_of_unit(U, G, t * nst)
        c_hi = sk_cta_of_unit(U, G, t * nst + nst - 1)
        assert cs == list(range(c_lo, c_hi + 1))
        assert c_hi - c_lo + 1 == len(cs) >= 2
        assert c_lo not in keys, f"tiles {keys.get(c_lo)} and {t} share the ticket key {c_lo}"
        keys[c_lo] = t
        # the fix-up reads contributor c's partial from its "first" slot exactly
        # when c's range starts at or after the tile's first unit
        for c in cs:
            use_first = sk_begin(U, G, c) >= t * nst
            assert (first_slot if use_first else last_slot).get(c) == t


def test_fewer_units_than_ctas():
    # one tile of two stages on four CTAs: cut over all four, CTAs 0 and 2 would own
    # nothing and the ticket would wait for three arrivals that never come; over
    # min(U, grid) = 2 CTAs both contribute
    check_plan(1, 2, 4)
    U, G = 2, 2
    assert [sk_begin(U, G, c) for c in range(5)] == [0, 1, 2, 2, 2]


def test_stream_k_plan_small_exhaustive():
    for G in range(2, 20):
        for ntiles in range(1, 40):
            for nst in (1, 2, 3, 5, 16):
                if ntiles * nst >= 2:
                    check_plan(ntiles, nst, G)


def test_stream_k_plan_random_large():
    rng = random.Random(11)
    for _ in range(300):
        G = rng.choice([148, 152, 160, 132])
        ntiles = rng.randint(1, 1200)
        nst = rng.choice([4, 6, 16, 40, 136])
        if ntiles * nst >= 2:
            check_plan(ntiles, nst, G)


def use_stream_k(ntiles, nst, G):
    """The routed product's device-side rule (and the dense plan's)."""
    U = ntiles * nst
    dp_span = -(-ntiles // G) * nst
    sk_span = -(-U // G) + 2
    return U >= 2 and 10 * sk_span < 9 * dp_span


def test_span_rule_on_the_moe_shapes():
    # ~320 gate tiles of 16 stages on 152 SMs: 3 whole tiles (48 stages) against
    # 34 + 2 -- stream-K; ~768 down tiles of 6 stages: 36 against 31 + 2 -- whole tiles
    assert use_stream_k(320, 16, 152)
    assert not use_stream_k(768, 6, 152)
    # the dense c1 plan: 80 tiles of 40 stages
    assert use_stream_k(80, 40, 152)
    # a whole number of waves gains nothing
    assert not use_stream_k(152, 16, 152)
