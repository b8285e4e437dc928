"""CPU check of the decode kernel's work partition (no GPU).

The decode kernel deals a head's items over the cluster's G = ks * NG groups:
group g takes slot rows g, g + G, ... (when a token leaves the window) and
window tokens s_lo + g, s_lo + g + G, ...; it walks the ring entries of its
tokens by adding G mod w.  These are the kernel's index formulas, restated
here so that a sweep of positions, windows and cluster sizes can check that
every slot row and window token is served exactly once, that every ring entry
read is in bounds and holds the token meant, and that no window read touches
the entry the new token is written into.
"""
import itertools

import pytest


def partition(t, w, M, G):
    absorb = t - w >= 0
    s_lo = max(0, t - w + 1)
    nwin = max(0, t - s_lo)
    wr = w if w > 0 else 1
    rows, toks = [], []
    for g in range(G):
        ns = (M - g + G - 1) // G if absorb and g < M else 0
        nw = (nwin - g + G - 1) // G if g < nwin else 0
        rows += [g + G * r for r in range(ns)]
        ring, step = (s_lo + g) % wr, G % wr
        for r in range(nw):
            toks.append((s_lo + g + G * r, ring))
            ring += step
            if ring >= wr:
                ring -= wr
    return absorb, s_lo, nwin, rows, toks


@pytest.mark.parametrize("M,D", [(16, 64), (64, 64), (16, 128), (64, 128)])
def test_every_item_served_once_and_ring_reads_in_bounds(M, D):
    NG = 256 // (D // 8)  # groups per CTA
    for ks, w in itertools.product((1, 2, 4, 8), (0, 1, 3, 64, 100, 512)):
        G = ks * NG
        for t in list(range(0, 40)) + [w - 1, w, w + 1, 2 * w + 5, 4096, 65535]:
            if t < 0:
                continue
            absorb, s_lo, nwin, rows, toks = partition(t, w, M, G)
            assert sorted(rows) == (list(range(M)) if absorb else [])
            assert sorted(s for s, _ in toks) == list(range(s_lo, s_lo + nwin))
            assert nwin == (min(t, w - 1) if w > 0 else 0)
            for s, e in toks:
                assert 0 <= e < max(w, 1)
                assert e == s % w  # the entry holds token s
                assert e != t % w  # never the entry token t is written into
