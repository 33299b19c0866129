"""Properties of the decode attention's work split, on the CPU: the formulas
the kernels use (csrc/attn_core.cuh) restated here and checked over many
batch shapes and grid sizes.

Units are 16 cache positions of one (virtual) sequence, numbered in sequence
order; CTA c of C takes units [U c / C, U (c + 1) / C); a CTA's partial of a
sequence goes to slot 2c (the sequence starts at or before the CTA's range)
or 2c + 1 (it starts inside the range); a merge reads the slots of the CTAs
that hold units of the sequence. These must cover every unit once, give every
partial its own slot, and name exactly the CTAs that wrote partials."""
import random

UNIT = 16


def range_start(c, U, C):
    return U * c // C


def cta_of(u, U, C):
    return ((u + 1) * C + U - 1) // U - 1


def participants(ub, nu, U, C):
    return cta_of(ub + nu - 1, U, C) - cta_of(ub, U, C) + 1 if U >= C else nu


def participant(ub, cf, p, U, C):
    return cf + p if U >= C else cta_of(ub + p, U, C)


def shapes(n=3000, seed=0):
    g = random.Random(seed)
    for _ in range(n):
        B = g.randint(1, 12)
        C = g.choice([1, 2, 3, 7, 16, 76, 152])
        pos = [g.choice([-1, 0, 5, 15, 16, 130, 1000, 4095, 32767]) for _ in range(B)]  # -1: invalid start
        yield B, C, pos


def test_split_covers_every_unit_once_and_slots_are_unique():
    for B, C, pos in shapes():
        units = [0 if p < 0 else (p + 1 + UNIT - 1) // UNIT for p in pos]
        pre = [0]
        for n in units:
            pre.append(pre[-1] + n)
        U = pre[-1]
        owner = {}
        slots = {}
        for c in range(C):
            u0, u1 = range_start(c, U, C), range_start(c + 1, U, C)
            for u in range(u0, u1):
                assert u not in owner
                owner[u] = c
                assert cta_of(u, U, C) == c
            # segments: sequences met by this CTA's range
            for b in range(B):
                lo, hi = max(u0, pre[b]), min(u1, pre[b + 1])
                if lo >= hi or (lo == pre[b] and hi == pre[b + 1]):
                    continue                       # not met, or held whole: no partial
                slot = 2 * c + (0 if u0 >= pre[b] else 1)
                assert slot not in slots, (B, C, pos)
                slots[slot] = b
        assert sorted(owner) == list(range(U))
        # merges read exactly the CTAs that wrote a partial of each split sequence
        for b in range(B):
            if units[b] == 0:
                continue
            ub, nu = pre[b], units[b]
            cf = cta_of(ub, U, C)
            np_ = participants(ub, nu, U, C)
            got = [participant(ub, cf, p, U, C) for p in range(np_)]
            truth = sorted({owner[u] for u in range(ub, ub + nu)})
            assert got == truth, (B, C, pos, b)
            if np_ > 1:
                read = {2 * cc + (0 if range_start(cc, U, C) >= ub else 1) for cc in got}
                assert read == {s for s, bb in slots.items() if bb == b}


def test_32_bit_split_bound():
    """(U + 1)(C + 1) < 2^32 keeps U c and (u + 1) C + U - 1 below 2^32: the
    largest batch a GPU could hold (B x positions bounded by HBM) stays far
    inside it."""
    C = 152
    positions = 288e9 / 4096          # cache positions that fit in 288 GB (8 KV heads)
    U = int(positions // UNIT) + 1
    assert (U + 1) * (C + 1) < 2 ** 32
    assert U * C < 2 ** 32 and (U + 1) * C + U - 1 < 2 ** 32
