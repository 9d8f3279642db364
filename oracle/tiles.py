"""Brute-force tile classification for the packed-varlen attention schedule.

TEST INFRASTRUCTURE ONLY (see the package docstring).

A query tile of sequence s covers local rows [q0, q1) with q0 = 128*qt and
q1 = min(q0 + 128, L); a key tile covers local keys [k0, k0 + 128).  The pair is

  skip    (0) if no (i, j) in the tile is visible,
  partial (1) if some are visible but not all of them, or the key tile runs
          past the end of the sequence (keys >= L must be masked),
  full    (2) if every query row of the tile sees every one of its 128 keys.

Visibility is decided element by element from the definition: key j is visible
from query i when j < L, j <= i if causal, and |i - j| <= window if
window >= 0 (kime-cuda 0.0.3 src/plan.rs, Op::Attention: window None is -1;
ffai-argus 0.7.3 src/text.rs, CausalSoftmax: row i sees keys 0..=i).

With per-sequence offsets pos (a chunk attending a KV cache, ffai-argus
TextTower::block with index_pos > 0) row i of sequence s sits at position
P = pos[s] + i and the keys are the cache rows j < pos[s] + L: j is visible
when j <= P if causal and |P - j| <= window if window >= 0; key tiles then
cover [0, pos[s] + L).  Nothing
here uses interval arithmetic on tile bounds: that is the scheduler's job, and
this module is what checks it.
"""
from __future__ import annotations

import numpy as np

BM = 128
BN = 128


def classify(cu, causal: bool, window: int, bm: int = BM, bn: int = BN, pos=None):
    """{(s, qt): int8 array over key tiles kt < ceil(Lk/bn) of codes 0/1/2},
    Lk = L (or pos[s] + L with offsets)."""
    cu = np.asarray(cu, np.int64)
    out = {}
    for s in range(len(cu) - 1):
        L = int(cu[s + 1] - cu[s])
        if L <= 0:
            continue
        off = 0 if pos is None else int(pos[s])
        Lk = off + L
        nk = -(-Lk // bn)
        j = np.arange(nk * bn)
        for qt in range(-(-L // bm)):
            q0, q1 = qt * bm, min(qt * bm + bm, L)
            i = off + np.arange(q0, q1)[:, None]
            vis = np.broadcast_to(j[None, :] < Lk, (q1 - q0, nk * bn)).copy()
            if causal:
                vis &= j[None, :] <= i
            if window >= 0:
                vis &= np.abs(i - j[None, :]) <= window
            v = vis.reshape(q1 - q0, nk, bn)
            anyv = v.any(axis=(0, 2))
            allv = v.all(axis=(0, 2))
            inside = (np.arange(nk) * bn + bn) <= Lk
            codes = np.where(anyv, np.where(allv & inside, 2, 1), 0).astype(np.int8)
            out[(s, qt)] = codes
    return out
