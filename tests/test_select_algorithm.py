"""Host model of the select kernel's ranking, checked against the oracle's
select_pools on the CPU.

The select kernel ranks a row by order-preserving uint32 keys with three radix
levels (bits 31..21, 20..10, 9..0), keeps a level's bin whole when its count is
exactly the number of keys still needed, breaks ties at the threshold key by
lower pool index, and pads a row to whole 256-pool columns with key 0 (the key
of NaN) instead of masking the padding out.  This file restates those rules in
numpy, so that the argument for the padding (it never changes the kept set)
is tested on every kind of row, including rows whose threshold is the NaN key.
No GPU needed."""
import numpy as np
import pytest

from oracle import kpool_oracle as O


def _keys(s: np.ndarray) -> np.ndarray:
    """The order-preserving key: -0 folded onto +0, NaN to 0, negatives bit-inverted."""
    s = np.asarray(s, np.float32) + np.float32(0.0)
    u = s.view(np.uint32).astype(np.uint64)
    k = np.where(u & 0x80000000, (~u) & 0xFFFFFFFF, u | 0x80000000)
    return np.where(np.isnan(s), 0, k).astype(np.uint64)


def _pick(hist: np.ndarray, remaining: int) -> tuple[int, int]:
    """Bin b (from the top) holding the remaining-th largest key, and remaining minus the keys above b."""
    above = 0
    for b in range(len(hist) - 1, -1, -1):
        if above < remaining <= above + int(hist[b]):
            return b, remaining - above
        above += int(hist[b])
    raise AssertionError("fewer keys than remaining")


def _kernel_select(scores: np.ndarray, topk: int, pad_to: int = 256) -> np.ndarray:
    n = len(scores)
    n_pad = -(-n // pad_to) * pad_to
    key = np.zeros(n_pad, np.uint64)
    key[:n] = _keys(scores)                         # the slots past the row keep key 0
    K, whole, rem = _threshold(key, topk)
    if whole:
        take = key >= K
    else:
        take = key > K
        eq = np.flatnonzero(key == K)
        take[eq[:rem]] = True                        # ties: the lowest pool indices
    kept = np.flatnonzero(take)
    kept = kept[kept < n]
    assert len(kept) == topk, (len(kept), topk)     # no slot past the row is ever kept
    return kept


def _chunked_compaction(key: np.ndarray, n: int, K: int, whole: bool, need_eq: int, topk: int,
                        chunk: int) -> np.ndarray:
    """The long-row compaction: chunks in pool order, each ranking its kept pools after the running
    count of kept pools and deciding its ties after the running count of ties; stops at topk."""
    out = np.full(topk, -1, np.int64)
    sel_base = eq_base = 0
    for c0 in range(0, len(key), chunk):
        if sel_base >= topk:
            break
        kc = key[c0:c0 + chunk]
        gt = kc >= K if whole else kc > K
        eq = np.zeros_like(gt) if whole else kc == K
        take = gt | eq
        eq_idx = np.flatnonzero(eq)
        take[eq_idx[eq_base + np.arange(len(eq_idx)) >= need_eq]] = False
        eq_base += len(eq_idx)
        kept = np.flatnonzero(take)
        rank = sel_base + np.arange(len(kept))
        ok = rank < topk
        out[rank[ok]] = c0 + kept[ok]
        sel_base += len(kept)
    assert np.all(out >= 0) and np.all(out < n)
    return out


def _threshold(key: np.ndarray, topk: int) -> tuple[int, bool, int]:
    """(K, whole, need_eq) of the three radix levels, as the kernel finds them: a level's bin is kept
    whole when its count is exactly the number of keys still needed."""
    levels = ((0x00000000, 21, 2048), (0xFFE00000, 10, 2048), (0xFFFFFC00, 0, 1024))
    prefix, rem = 0, topk
    for hi_mask, shift, nbins in levels:
        inbin = (key & hi_mask) == prefix
        hist = np.bincount(((key[inbin] >> shift) & (nbins - 1)).astype(np.int64), minlength=nbins)
        d, rem = _pick(hist, rem)
        prefix |= d << shift
        if int(hist[d]) == rem and shift > 0:
            return prefix, True, 0
    return prefix, False, rem


def _rows(kind: str, n: int, rng) -> np.ndarray:
    if kind == "normal":
        return rng.standard_normal(n).astype(np.float32)
    if kind == "few_values":
        return (rng.integers(-2, 3, n) * 0.25).astype(np.float32)
    if kind == "all_equal":
        return np.full(n, -1.5, np.float32)
    if kind == "signed_zeros":
        s = np.where(rng.random(n) < 0.5, np.float32(-0.0), np.float32(0.0)).astype(np.float32)
        s[rng.random(n) < 0.05] = 1.0
        return s
    if kind == "mostly_nan":                         # the threshold is the NaN key, next to the padding
        s = rng.standard_normal(n).astype(np.float32)
        s[rng.random(n) < 0.9] = np.nan
        s[rng.random(n) < 0.02] = np.inf
        s[rng.random(n) < 0.05] = -np.inf
        return s
    if kind == "tiny_and_huge":                      # denormals, extremes, one bin holding the threshold
        s = rng.choice(np.array([1e-45, -1e-45, 3e38, -3e38, 1.0, 2.0], np.float32), n)
        return s.astype(np.float32)
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["normal", "few_values", "all_equal", "signed_zeros", "mostly_nan",
                                  "tiny_and_huge"])
@pytest.mark.parametrize("n", [65, 300, 511, 1000, 2049, 8191])
def test_padded_radix_select_keeps_the_oracle_pools(kind, n):
    rng = np.random.default_rng([n, len(kind)])
    topk = 64
    for _ in range(3):
        s = _rows(kind, n, rng)
        np.testing.assert_array_equal(_kernel_select(s, topk), O.select_pools(s, topk))


def test_key_order_matches_the_oracle_order():
    """Larger score, larger key; -0 and +0 share a key; NaN has key 0, below -inf."""
    s = np.array([np.nan, -np.inf, -3e38, -1.0, -1e-45, -0.0, 0.0, 1e-45, 1.0, 3e38, np.inf], np.float32)
    k = _keys(s)
    assert k[0] == 0 and np.all(np.diff(k[1:].astype(np.int64)) >= 0)
    assert k[5] == k[6] and np.all(np.diff(np.delete(k[1:], 4).astype(np.int64)) > 0)


@pytest.mark.parametrize("kind", ["normal", "few_values", "all_equal", "mostly_nan", "tiny_and_huge"])
@pytest.mark.parametrize("chunk", [256, 1024, 8192])
def test_chunked_compaction_keeps_the_oracle_pools(kind, chunk):
    """Rows of several chunks (chunk sizes scaled down from the kernel's 8192 so that small rows span
    many): carrying the kept and tied counts from chunk to chunk keeps the oracle's pools."""
    rng = np.random.default_rng([chunk, len(kind), 7])
    topk = 64
    for n in (300, 2049, 9000):
        s = _rows(kind, n, rng)
        n_pad = -(-n // 256) * 256
        key = np.zeros(n_pad, np.uint64)
        key[:n] = _keys(s)
        K, whole, need_eq = _threshold(key, topk)
        got = _chunked_compaction(key, n, K, whole, need_eq, topk, chunk)
        np.testing.assert_array_equal(got, O.select_pools(s, topk))
