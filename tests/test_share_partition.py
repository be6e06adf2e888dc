"""The decode launch's split of the batch's 128-token tiles into per-CTA shares,
restated from the rule the kernel states and checked for the properties the
in-launch split-KV merge relies on.

Tiles are laid end to end, (sequence, KV head) pair after pair.  With fewer
than four pairs per CTA, CTA c owns [floor(c W / NC), floor((c+1) W / NC)).
Otherwise tile u of pair q starts at 8 u + 24 (q + 1) on a virtual line of
length V = 8 W + 24 B Hkv (every pair, empty ones included, preceded by a
charge of three tiles), CTA c's range is [floor(c V / NC), floor((c+1) V / NC))
and it owns the tiles whose start lies in it.  Required: the shares are
contiguous and cover [0, W) once; every CTA between a pair's first and last
owner holds some of its tiles (the merge counts contributors as
c_last - c_first + 1); with equal lengths and num_splits shares per pair
available, every pair is cut into exactly that many shares.  The set-up's
integer helpers (two 32-bit divisions for floor(n / d) with d < 2^11, a
single-precision estimate corrected exactly) are checked against exact
division.
"""
import random

import numpy as np

TILE, V_TILE, V_PAIR, PAIRS_PER_CTA = 128, 8, 24, 4


def div_small(n, d):
    hi, lo = n >> 20, n & 0xFFFFF
    qh = hi // d
    return (qh << 20) + ((((hi - qh * d) << 20) | lo) // d)


def div_est(n, d):
    q = max(int(np.float32(np.float32(n) / np.float32(d))), 0)
    while q > 0 and q * d > n:
        q -= 1
    while (q + 1) * d <= n:
        q += 1
    return q


def shares(lens, Hkv, num_ctas):
    nbs = [(L + TILE - 1) // TILE for L in lens]
    cum = [0]
    for n in nbs:
        cum.append(cum[-1] + n)
    B, W = len(lens), cum[-1] * Hkv
    NC = (W if W > 0 else 1) if W < num_ctas else num_ctas
    weighted = B * Hkv >= PAIRS_PER_CTA * num_ctas  # the host's choice of kernel (CTAs of the launch)
    nonempty = sum(1 for n in nbs if n > 0)
    vk = V_PAIR if weighted and nonempty * Hkv >= PAIRS_PER_CTA * NC else 0
    if W == 0:
        return nbs, cum, W, NC, [0] * (NC + 1)
    if vk == 0:
        return nbs, cum, W, NC, [div_small(c * W, NC) for c in range(NC)] + [W]

    def vpos(u, b, h):
        return V_TILE * u + vk * (b * Hkv + h + 1)

    def tile_at(vt):
        lo, hi = 0, B - 1
        while lo < hi:
            mid = (lo + hi + 1) >> 1
            if vpos(cum[mid] * Hkv, mid, 0) <= vt:
                lo = mid
            else:
                hi = mid - 1
        nb, u_b = nbs[lo], cum[lo] * Hkv
        base = vpos(u_b, lo, 0)
        if base >= vt:
            return u_b
        step = V_TILE * nb + vk
        h = min(div_est(vt - base, step), Hkv - 1)
        t = (vt - (base + h * step) + V_TILE - 1) // V_TILE
        return u_b + h * nb + (t if t < nb else nb)

    V = V_TILE * W + vk * B * Hkv
    return nbs, cum, W, NC, [tile_at(div_small(c * V, NC)) for c in range(NC)] + [W]


def check(lens, Hkv, num_ctas):
    nbs, cum, W, NC, st = shares(lens, Hkv, num_ctas)
    assert st[0] == 0 and st[-1] == W
    assert all(st[c] <= st[c + 1] for c in range(NC))
    starts = np.array(st[:-1])
    for b, nb in enumerate(nbs):
        for h in range(Hkv if nb else 0):
            f = cum[b] * Hkv + h * nb
            l = f + nb - 1
            cf = int(np.searchsorted(starts, f, side="right")) - 1  # the last share starting at or before f
            cl = int(np.searchsorted(starts, l, side="right")) - 1
            for c in range(cf, cl + 1):
                assert max(st[c], f) < min(st[c + 1], l + 1), (b, h, c)
    return NC, st


def test_integer_helpers_are_exact():
    rng = random.Random(3)
    for _ in range(20000):
        d = rng.randint(1, 2047)
        n = rng.randint(0, (1 << 52) - 1) if rng.random() < 0.5 else rng.randint(0, 1 << 40)
        assert div_small(n, d) == n // d
        d2 = rng.randint(1, 1 << 34)
        n2 = rng.randint(0, d2 * rng.randint(1, 1 << 16) - 1)
        assert div_est(n2, d2) == n2 // d2


def test_shares_cover_the_tiles_and_every_contributor_holds_tiles():
    rng = random.Random(1)
    for _ in range(300):
        B = rng.randint(1, 300)
        Hkv = rng.choice([1, 2, 4, 8])
        lens = [rng.choice([0, 1, 127, 128, 129, 1000, rng.randint(0, 20000), rng.randint(0, 200000)])
                for _ in range(B)]
        check(lens, Hkv, rng.choice([1, 7, 152, 184]))


def test_weighted_shares_engage_from_four_pairs_per_cta():
    lens = [6000] * 256
    NC, st = check(lens, 8, 152)
    nbs = -(-6000 // TILE)
    # pair boundaries attract share boundaries: more shares start on a pair's
    # first tile than the equal split gives
    eq = [c * (256 * 8 * nbs) // 152 for c in range(152)]
    on_pair = lambda s: sum(1 for x in s if x % nbs == 0)
    assert on_pair(st[:-1]) > on_pair(eq)


def test_equal_lengths_split_into_num_splits_shares():
    for B, Hkv, L, S in [(2, 8, 131072, 9), (16, 8, 8192, 1), (3, 2, 5000, 7), (4, 4, 1300, 3)]:
        nbs, cum, W, NC, st = shares([L] * B, Hkv, B * Hkv * S)
        starts = np.array(st[:-1])
        for b in range(B):
            for h in range(Hkv):
                f = cum[b] * Hkv + h * nbs[b]
                l = f + nbs[b] - 1
                n = int(np.searchsorted(starts, l, side="right")) - int(np.searchsorted(starts, f, side="right")) + 1
                assert n == S, (B, Hkv, L, S, b, h, n)
