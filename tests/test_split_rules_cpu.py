"""The rules the split kernels rely on, checked on the CPU against the oracle.

The top-k of a row split over C slices (dsa_select, clustered rows): each slice first
offers its top kt = min(k, 2 ceil(k / C)) keys; the candidates are taken as they are
when every slice that left keys out has its kt-th key strictly below the candidates'
k-th key, and otherwise every slice offers its full top-k. Both ways must give the
row's exact top-k (oracle.topk_pools: score descending, lowest id first, -inf never).

The paged score's work split (dsa_score, up to 256 rows): the rows' visible 64-pool
stages, in (row, stage) order, are cut into G equal runs, a run starting at the row
found by a running sum over the rows, and the pools past each row's visible stages
are cut into G runs per row for the -inf fill; every pool is written exactly once.
"""
import numpy as np
import pytest

from oracle import dsa_oracle as O


def _slice_topk(s, base, k):
    """The slice's top-k as (score, id) pairs in id order, its k-th score (None when
    it offers nothing) and whether it left finite scores out."""
    fin = np.flatnonzero(np.isfinite(s))
    order = fin[np.lexsort((fin, -s[fin]))]
    take = np.sort(order[:k])
    kth = s[order[k - 1]] if len(order) >= k else (s[order[-1]] if len(order) else None)
    return [(s[i], base + i) for i in take], kth, len(order) > k


def _kth_of(cands, k):
    vals = sorted((v for v, _ in cands), reverse=True)
    return vals[k - 1] if len(vals) >= k else None


def _split_topk(row, k, C):
    P = len(row)
    chunk = -(-P // C)
    kt = min(k, 2 * (-(-k // C)))
    slices = [(row[c * chunk:(c + 1) * chunk], c * chunk) for c in range(C)]
    first = [_slice_topk(s, b, kt) for s, b in slices]
    cands = [p for part, _, _ in first for p in part]
    T = _kth_of(cands, k)
    exact = all(not cut or (T is not None and kth < T) for _, kth, cut in first)
    if kt < k and not exact:
        cands = [p for s, b in slices for p in _slice_topk(s, b, k)[0]]
    # the merge: the top-k of the candidates, ties to the earlier candidate (slot order)
    order = sorted(range(len(cands)), key=lambda j: (-cands[j][0], j))[:k]
    ids = np.sort(np.array([cands[j][1] for j in order], dtype=np.int64))
    out = np.full(k, -1, dtype=np.int64)
    out[:len(ids)] = ids
    return out, kt < k and not exact


def _rows(rng, kind, P):
    if kind == "normal":
        x = rng.standard_normal(P)
        x[rng.random(P) < 0.05] = -np.inf
        return x
    if kind == "ties":
        return rng.choice([-np.inf, -1.0, 0.0, 0.5, 1.0, 2.0], P)
    if kind == "ramp":
        return np.arange(P, dtype=np.float64)
    if kind == "prefix":  # a short row in a batch with a long maximum
        x = np.full(P, -np.inf)
        n = int(rng.integers(1, max(2, P // 4)))
        x[:n] = rng.standard_normal(n)
        return x
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["normal", "ties", "ramp", "prefix"])
def test_trimmed_split_topk_is_exact(kind):
    rng = np.random.default_rng(len(kind))
    second = 0
    for _ in range(60):
        C = int(rng.choice([2, 4, 8]))
        P = int(rng.integers(1, 700))
        k = int(rng.integers(1, 90))
        row = _rows(rng, kind, P)
        got, redo = _split_topk(row, k, C)
        second += redo
        np.testing.assert_array_equal(got, O.topk_pools(row, k))
    if kind in ("ramp", "prefix"):
        assert second > 0  # the second exchange is exercised


def test_balanced_score_split_writes_every_pool_once():
    rng = np.random.default_rng(7)
    for _ in range(200):
        rows = int(rng.integers(1, 257))
        P = int(rng.integers(1, 6000))
        spr = -(-P // 64)
        nvis = rng.integers(0, P + 1, rows)
        bad = rng.random(rows) < 0.1
        vs = np.where(bad, 0, np.minimum(spr, -(-nvis // 64)))
        G = max(1, min(rows * spr, 456))
        tot = int(vs.sum())
        hits = np.zeros((rows, spr * 64), dtype=np.int64)
        ends = np.cumsum(vs)
        for b in range(G):
            u0, u1 = b * tot // G, (b + 1) * tot // G
            if u0 == u1:
                continue
            r = int(np.searchsorted(ends, u0, side="right"))
            st = u0 - (int(ends[r]) - int(vs[r]))
            for _u in range(u0, u1):
                while st >= vs[r]:
                    r, st = r + 1, 0
                hits[r, st * 64:(st + 1) * 64] += 1
                st += 1
        for r in range(rows):
            t0 = int(vs[r]) * 64
            tail = P - t0
            if tail > 0:
                per = -(-tail // G)
                for b in range(G):
                    lo, hi = t0 + b * per, min(t0 + (b + 1) * per, P)
                    if lo < hi:
                        hits[r, lo:hi] += 1
        assert (hits[:, :P] == 1).all()
