"""The oracle of the projections on either side of CSA2 attention: the low-rank query path
and the grouped low-rank output projection (TEST INFRASTRUCTURE ONLY, like the rest of this
package).

Sources: "DeepSeek V4.1-Flash. Every layer, connected", section "The query and output
paths" (the query and output projections are low-rank / grouped; the output's rotary
coordinates are rotated back before the grouped projection); "DeepSeek V4 Inside": the
Flash config (hidden 4096, 64 heads of 512, q_lora_rank 1024), the layer-0 attention
example (the heads' outputs are concatenated and go through a grouped W_O, 64 heads in
o_groups = 8), and the CSA example (RMSNorm on the query head before its partial RoPE).

Readings (the pages give no formula for either projection):
* query path: c = W_DQ x (hidden -> q_rank), c <- RMSNorm(c) * g_q, q = W_UQ c
  (q_rank -> heads x head_dim), then each head q_h <- RMSNorm(q_h) * g_head (one gain
  vector of head_dim entries shared by the heads).  The rotation of the head's last 64
  coordinates belongs to attention, which applies it to the query it receives.
* RMSNorm(v) = v / sqrt(mean(v^2) + eps) over the last axis; eps is not stated (1e-6 by
  default).
* grouped low-rank output projection: the heads split into G groups of consecutive heads;
  group g's outputs, concatenated (heads/G x head_dim values), go through its own
  W_OA[g] (-> o_rank), and the G results, concatenated, through W_OB (G x o_rank ->
  hidden).  o_rank is not stated; the callers use 1024, the query's stated rank.
* the output o is taken after attention's inverse rotation, as attention returns it.
"""
from __future__ import annotations

import numpy as np

__all__ = ["rms_norm", "query_proj", "out_proj", "linear"]


def rms_norm(v, gain=None, eps: float = 1e-6) -> np.ndarray:
    """v / sqrt(mean(v^2) + eps) over the last axis, times gain (None: 1), in float64."""
    v = np.asarray(v, np.float64)
    ms = np.mean(v * v, axis=-1, keepdims=True)
    y = v / np.sqrt(ms + eps)
    if gain is not None:
        y = y * np.asarray(gain, np.float64)
    return y


def query_proj(x, w_dq, g_q, w_uq, g_head, n_heads: int, eps: float = 1e-6) -> np.ndarray:
    """Queries [T, n_heads, head_dim] (float64) of hidden states x [T, hidden].

    w_dq [q_rank, hidden], g_q [q_rank] or None, w_uq [n_heads * head_dim, q_rank],
    g_head [head_dim] or None."""
    x = np.asarray(x, np.float64)
    c = x @ np.asarray(w_dq, np.float64).T          # down-projection to the query rank
    c = rms_norm(c, g_q, eps)
    q = c @ np.asarray(w_uq, np.float64).T          # up-projection to every head
    q = q.reshape(x.shape[0], n_heads, -1)
    return rms_norm(q, g_head, eps)                 # per head


def out_proj(o, w_oa, w_ob) -> np.ndarray:
    """Attention output o [T, heads, head_dim] -> [T, hidden] (float64).

    w_oa [G, o_rank, heads / G * head_dim], w_ob [hidden, G * o_rank]."""
    o = np.asarray(o, np.float64)
    w_oa = np.asarray(w_oa, np.float64)
    T, H, D = o.shape
    G, r, kg = w_oa.shape
    assert H % G == 0 and kg == H // G * D
    y = np.empty((T, G * r))
    for g in range(G):
        og = o[:, g * (H // G):(g + 1) * (H // G), :].reshape(T, kg)   # the group's heads, concatenated
        y[:, g * r:(g + 1) * r] = og @ w_oa[g].T
    return y @ np.asarray(w_ob, np.float64).T


def linear(x, w) -> np.ndarray:
    """x [T, in] times w [out, in] transposed, in float64."""
    return np.asarray(x, np.float64) @ np.asarray(w, np.float64).T
