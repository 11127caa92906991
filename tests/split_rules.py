"""Mirrors of the library's size-driven kernel choices, for the tests.

The library decides from the sizes alone how a call is split: the forward's key ranges in a
cluster, the one-pass or two-pass backward, the dQ pass's key ranges, the dK/dV pass's query
ranges in a cluster. The tests use these mirrors to pick shapes that reach each choice and to
check the ranges themselves; they are written from the rules the library's comments state,
not shared with it.
"""


def kernel_head_dim(d):
    """The head size the kernels run at: 32, 64 or 128."""
    return 32 if d <= 32 else (64 if d <= 64 else 128)


def max_range_splits(d, n_tiles):
    """Largest cluster of the key- and query-range splits over n_tiles tiles: 16 where a CTA's
    share of a row, kernel head size / 16 columns, is still a group of 4 (64 and 128) and each
    range keeps at least 16 tiles, else 8."""
    return 16 if kernel_head_dim(d) >= 64 and n_tiles >= 256 else 8


def _power_of_two_up_to(cap):
    s = 1
    while 2 * s <= cap:
        s *= 2
    return s


def fwd_key_splits(bh, n_q, n_k, d):
    """Key ranges per query-tile pair of the forward: only while its CTAs (pairs x heads) fill
    at most half of 148 SMs; at most 148 CTAs and at least 8 key tiles per range."""
    ctas, n_kt = bh * -(-n_q // 256), -(-n_k // 128)
    if 2 * ctas > 148:
        return 1
    return _power_of_two_up_to(min(148 // ctas, n_kt // 8, max_range_splits(d, n_kt)))


def one_pass(bh, n_k, d):
    """Whether fa2_backward takes the one-pass kernel: head size up to 64 and more than 74 key
    tiles in all."""
    return d <= 64 and 2 * bh * -(-n_k // 128) > 148


def dkv_query_splits(bh, n_q, n_k, d):
    """Query ranges per key tile of the dK/dV pass: at least 16 query tiles per key tile, the
    dK/dV CTAs filling at most half of 148 SMs; at most 148 CTAs and at least 8 query tiles per
    range."""
    n_kt, n_qt = -(-n_k // 128), -(-n_q // 128)
    if 2 * bh * n_kt > 148 or n_qt < 16 * n_kt:
        return 1
    return _power_of_two_up_to(min(148 // (bh * n_kt), n_qt // 8, max_range_splits(d, n_qt)))


def dq_key_splits(bh, n_q, n_k):
    """Key ranges per query tile of the dQ pass (float32 partial sums in the workspace)."""
    n_qt, n_kt = -(-n_q // 128), -(-n_k // 128)
    s = min(-(-148 // (bh * n_qt)), n_kt // 8, 8)
    return 1 if s < 2 else s


def dkdv_tiles_per_cta(bh, n_q, n_k, sms):
    """Key tiles per dK/dV CTA of the kernel that runs both passes in one grid: enough for
    32 query tiles per CTA, at most 8, and fewer while the head's dK/dV CTAs would number
    fewer than the SMs."""
    n_qt, n_kt = -(-n_q // 128), -(-n_k // 128)
    m = min(8, max(1, -(-32 // n_qt)))
    while m > 1 and bh * -(-n_kt // m) < sms:
        m -= 1
    return m


def balanced_ranges(n, splits):
    """The tiles [lo, hi) of each of `splits` ranges over n tiles, as the cluster splits take
    them: range r = [floor(r n / splits), floor((r + 1) n / splits))."""
    return [(r * n // splits, (r + 1) * n // splits) for r in range(splits)]
