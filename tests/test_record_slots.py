"""The attention kernel's partial-state slots and the combine's enumeration of
them, restated on the host: blocks take chunk ranges [c W / N, (c + 1) W / N);
each block writes slots (c + u) * 4 + w for every unit u of its range but the
last, and slot (c + ub) * 4 for its last unit ub (its four warps merged); the
combine reads, for unit u over blocks c_first .. c_last, slot 0 of every block
before c_last and one slot (the unit ends with c_last's range) or four of
c_last, skipping blocks with empty ranges. Over random splits (including fewer
chunks than blocks, and units without chunks) the combine must read exactly the
slots written for that unit, so no slot read can hold another call's state.
The GPU parity tests check the kernels themselves."""
import random

import pytest


def cta_lo(c, W, N):
    return (c * W) // N


def cta_of(x, W, N):
    return ((x + 1) * N - 1) // W


def find_unit(prefix, U, x):
    lo, hi = 0, U - 1
    while lo < hi:
        mid = (lo + hi + 1) >> 1
        if prefix[mid] <= x:
            lo = mid
        else:
            hi = mid - 1
    return lo


def written_slots(prefix, U, W, N):
    out = {}
    for c in range(N):
        lo, hi = cta_lo(c, W, N), cta_lo(c + 1, W, N)
        if lo >= hi:
            continue
        ua, ub = find_unit(prefix, U, lo), find_unit(prefix, U, hi - 1)
        for u in range(ua, ub):
            for w in range(4):
                out[(c + u) * 4 + w] = u
        out[(c + ub) * 4] = ub
    return out


def combine_slots(prefix, u, W, N):
    s0, s1 = prefix[u], prefix[u + 1]
    cf, cl = cta_of(s0, W, N), cta_of(s1 - 1, W, N)
    nb1 = cl - cf
    R = nb1 + (1 if cta_lo(cl + 1, W, N) <= s1 else 4)
    slots = []
    for r in range(R):
        cc = cf + (r if r < nb1 else nb1)
        if W < N and cta_lo(cc, W, N) >= cta_lo(cc + 1, W, N):
            continue
        slots.append((cf + u) * 4 + (r * 4 if r < nb1 else nb1 * 4 + (r - nb1)))
    return slots


@pytest.mark.parametrize("seed", range(4))
def test_combine_reads_exactly_the_slots_written(seed):
    rng = random.Random(seed)
    for _ in range(2000):
        U, N = rng.randint(1, 12), rng.randint(1, 40)
        counts = [rng.choice([0, 0, 1, 2, 3, 5, 17, 60]) for _ in range(U)]
        prefix = [0]
        for n in counts:
            prefix.append(prefix[-1] + n)
        W = prefix[-1]
        if W == 0:
            continue
        written = written_slots(prefix, U, W, N)
        for u in range(U):
            if prefix[u] == prefix[u + 1]:
                continue
            got = combine_slots(prefix, u, W, N)
            assert len(got) == len(set(got))
            want = {s for s, owner in written.items() if owner == u
                    and any(max(cta_lo(c, W, N), prefix[u]) < min(cta_lo(c + 1, W, N), prefix[u + 1])
                            for c in [s // 4 - u])}
            assert set(got) == want, (U, N, counts, u)
