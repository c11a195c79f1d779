"""The oracle of the encoder's sequence compressor (TEST INFRASTRUCTURE ONLY, like the rest of
this package).

Source: the course's lesson "How CSA2 compresses, shares, and selects attention memory"
(section "two source positions -> learned pooling or projection -> one global latent
entry"): with a compression ratio above 1 the compressor pools consecutive token
representations with learned, channel-wise softmax gates; at ratio 1 there is no pooling.
"DeepSeek V4.1-Flash. Every layer, connected" gives the encoder's banks ratio 2 and the
decoder's ratio 1.

Readings (the pages print no formula):
* entry e of ratio m pools tokens m*e .. m*e + m - 1: for every channel c,
  entry[e, c] = sum_j softmax_j(gate[m*e + j, c]) * kv[m*e + j, c] (softmax over the m
  tokens, separately per channel); the gate logits and the values are per-token inputs
  (projections of the token representation, weights outside this path);
* an incomplete last group (T not a multiple of m) yields no entry;
* causality: an entry is visible to a query at position p only when all its tokens are,
  i.e. the first (p + 1) // m entries (the V4 page's causal rule for compressed entries:
  an entry holding a future token is forbidden to core attention).
"""
from __future__ import annotations

import numpy as np

__all__ = ["compress", "visible_entries"]


def compress(kv, gate, ratio: int) -> np.ndarray:
    """kv, gate [T, D] -> entries [T // ratio, D] (float64)."""
    kv = np.asarray(kv, np.float64)
    gate = np.asarray(gate, np.float64)
    T, D = kv.shape
    n = T // ratio
    kv = kv[: n * ratio].reshape(n, ratio, D)
    g = gate[: n * ratio].reshape(n, ratio, D)
    g = g - g.max(axis=1, keepdims=True)
    e = np.exp(g)
    w = e / e.sum(axis=1, keepdims=True)
    return (w * kv).sum(axis=1)


def visible_entries(pos, ratio: int):
    """Entries visible to a query at position pos: those whose every token is at or before it."""
    return (np.asarray(pos, np.int64) + 1) // ratio
