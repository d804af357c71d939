"""The split over K (stream-K) work schedule, checked on the host.

The kernel's WorkIter hands each cluster its stream-K run first (equal runs of
the first sk_tiles tiles' (tile, k-block) units), then whole tiles in waves;
the epilogue finds a split tile's contributors with unit_owner and indexes its
partial slots by tile (whole problem split) or by the first contributor's CTAs
(last waves split).  These formulas are restated here in Python and checked for
the invariants the kernel relies on: every unit is computed exactly once, a
split tile has at most two contributors when runs are at least a tile long
(three when at least half a tile), and no two split tiles share a slot.
"""


def schedule(T, C, kb, sk_tiles, c):
    items = []
    U = sk_tiles * kb
    u, u_end = U * c // C, U * (c + 1) // C
    while u < u_end:
        t = u // kb
        k0 = u - t * kb
        k1 = min(kb, k0 + (u_end - u))
        items.append((t, k0, k1))
        u += k1 - k0
    t = sk_tiles + c
    while t < T:
        items.append((t, 0, kb))
        t += C
    return items


def unit_owner(u, U, G):
    return ((u + 1) * G + U - 1) // U - 1


def check(T, C, kb, csize, sk_tiles, max_segs):
    done = {}
    slots = {}
    for c in range(C):
        for t, k0, k1 in schedule(T, C, kb, sk_tiles, c):
            for k in range(k0, k1):
                assert (t, k) not in done
                done[(t, k)] = c
            if (k0, k1) == (0, kb):
                continue
            U = sk_tiles * kb
            first = unit_owner(t * kb, U, C)
            nseg = unit_owner(t * kb + kb - 1, U, C) - first + 1
            seg = c - first
            assert 0 <= seg < nseg <= max_segs
            for r in range(csize):
                owner = t if sk_tiles == T else first * csize + r
                assert owner < (T if sk_tiles == T else C * csize)
                assert slots.setdefault((owner, seg), t) == t, "two split tiles share a slot"
    assert len(done) == T * kb


def test_last_waves_split_schedule():
    # the last partly filled wave and the one before it split: C..2C-1 tiles,
    # runs of at least one tile, then the same number of whole-tile waves per cluster
    for C, csize in ((76, 2), (152, 1), (74, 2), (10, 1), (3, 2)):
        for T in range(2 * C, 5 * C + 3, max(1, C // 5)):
            sk = T - (T // C - 1) * C
            assert C <= sk < 2 * C and (T - sk) % C == 0
            for kb in (2, 3, 8, 64, 172):
                check(T, C, kb, csize, sk, 2)


def test_few_tiles_split_schedule():
    # the whole problem split over G = min(units / ceil(kb / 2), grid) CTAs:
    # runs of at least half a tile
    for T in range(1, 77, 3):
        for kb in (2, 3, 16, 33, 64):
            for grid in (152, 9, 4):
                G = min(T * kb // ((kb + 1) // 2), grid)
                if G > T:
                    check(T, G, kb, 1, T, 3)
