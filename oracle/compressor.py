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

The encoder bank's memory (encoder_memory), from "Every layer, connected" (the global and
index paths: global memory is created once and indexer keys are derived from the main KV) and
the V4 page (the compressed KV carries absolute positions; the cache is rotated before it is
stored):
* the compressor's output is float32 (the type it hands on);
* entry e's position is that of its last token, m*e + m - 1 (the position at which it
  becomes visible), and its latent cache row is the writer's bf16 record rotated there;
* its indexer key is W_IK times the entry (unrotated, in bf16), rounded once to bf16.
"""
from __future__ import annotations

import numpy as np

from .csa2 import bf16_to_f64
from .projections import linear
from .writer import write_records

__all__ = ["compress", "visible_entries", "bf16_round_f64", "encoder_memory"]


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


def bf16_round_f64(x) -> np.ndarray:
    """bf16 bit patterns of float64 values rounded once to bf16's 8 significant bits, to
    nearest with ties to even (no intermediate float32 rounding); normal range only."""
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)                          # x = m 2^e, 0.5 <= |m| < 1
    r = np.rint(m * 256.0) * np.exp2(e - 8.0)   # 8 significant bits, ties to even
    return (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def encoder_memory(kv, gate, ratio: int, w_ik, theta: float = 10000.0) -> dict:
    """One encoder bank's memory from its tokens' projections kv, gate [T, 512]: entries
    (float32), their positions, the latent cache rows (bf16 bits, rotated) and the indexer
    keys (bf16 bits) = W_IK [128, 512] times the unrotated bf16 entry."""
    entries = compress(kv, gate, ratio).astype(np.float32)
    pos = np.arange(entries.shape[0], dtype=np.int64) * ratio + ratio - 1
    lat, _ = write_records(entries, pos, theta, "bf16")
    plain, _ = write_records(entries, None, theta, "bf16")
    keys = bf16_round_f64(linear(bf16_to_f64(plain), w_ik))
    return {"entries": entries, "pos": pos, "lat": lat, "k_idx": keys}
