"""The cluster splits' ranges: every range the size rules can produce holds work.

A CTA of a split whose range were empty would never receive the stage its MMA issuer waits
for, so the whole cluster would stop at that wait. The ranges are balanced,
[floor(r n / s), floor((r + 1) n / s)), and the rules take at least 8 tiles per range, so
every range is non-empty and together they cover the n tiles exactly, for every split count
up to 16. The earlier form, [r L, min(n, r L + L)) with L = ceil(n / s), leaves its last
ranges empty once s reaches 16 (130 query tiles over 16 CTAs: the last would start at 135);
those shapes now run.
"""
import random

from tests.split_rules import balanced_ranges, dkv_query_splits, dq_key_splits, fwd_key_splits


def _check(n, s):
    r = balanced_ranges(n, s)
    assert r[0][0] == 0 and r[-1][1] == n
    assert all(hi > lo for lo, hi in r)
    assert all(r[i][1] == r[i + 1][0] for i in range(s - 1))


def test_balanced_ranges_are_never_empty_for_the_split_counts_the_rules_take():
    for s in (2, 4, 8, 16):
        for n in range(8 * s, 4000):
            _check(n, s)


def test_sizes_the_rules_split_get_non_empty_ranges():
    rng = random.Random(7)
    seen = set()
    for _ in range(20000):
        bh = rng.randint(1, 80)
        n_q, n_k = rng.randint(1, 70000), rng.randint(1, 70000)
        d = rng.choice([8, 32, 40, 64, 72, 128])
        s = fwd_key_splits(bh, n_q, n_k, d)
        if s > 1:
            _check(-(-n_k // 128), s)
            seen.add(("fwd", s))
        s = dkv_query_splits(bh, n_q, n_k, d)
        if s > 1:
            _check(-(-n_q // 128), s)
            seen.add(("dkv", s))
    assert {("fwd", 16), ("dkv", 16), ("fwd", 2), ("dkv", 2)} <= seen


def test_the_ceiling_ranges_would_leave_a_cluster_rank_empty():
    n, s = 130, 16
    length = -(-n // s)
    assert (s - 1) * length >= n  # the last rank's start lies past the last tile
    _check(n, s)


def test_the_dq_passes_ceiling_ranges_are_never_empty():
    """The dQ pass's key ranges keep the ceiling form, [r L, min(n, r L + L)) with
    L = ceil(n / s); its rule takes at most 8 ranges of at least 8 key tiles, so
    (s - 1) L < n and the last range holds work (n >= 8 s > s (s - 1))."""
    for bh in (1, 2, 3, 7, 40):
        for n_q in (1, 128, 300, 1000, 4096):
            for n_kt in range(1, 700):
                s = dq_key_splits(bh, n_q, 128 * n_kt)
                if s > 1:
                    length = -(-n_kt // s)
                    assert 2 <= s <= 8 and (s - 1) * length < n_kt
