"""Hybrid decode attention over the packed history plus the exact recent (ring) buffer.

[Guide] §五 (hooks) and §七 (limitations) say that the hybrid decode attends over the compressed
history together with an exact recent buffer (ring buffer, buffer_size=128). [Guide] §二 (the
TurboQuantProd estimator) says that keys give an unbiased inner-product estimate, E[estimate] =
<q, k>. Written out for one query head q and a packed token (n, idx, gamma, sign):

    q_rot = Pi q,  q_proj = S q_rot,
    <q, k>_est = n * ( <q_rot, c[idx]> + sqrt(pi/2)/d * gamma * <q_proj, 2 sign - 1> ).

The constant sqrt(pi/2)/d comes from E[sign(s.r) (s.x)] = sqrt(2/pi) <r, x> / ||r|| for s ~ N(0, I),
summed over the d rows of S. Ring tokens score exactly: <q, k_j>.

The output is one softmax over the concatenated [packed || ring] scores, times softmax_scale
(default 1/sqrt(d)). Values:
* packed tokens use Pi^T (level * s);
* ring tokens use the raw values.

Query head h reads KV head floor(h / G) (GQA).
"""

import numpy as np

from .quant import dequantize_values
from .rotation import rotation_matrix


def qjl_inner_product_estimate(q, keys, D, S, centroids):
    """<q, k_t>_est for one query vector q [d] against key records [T]."""
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[0]
    q_rot = rotation_matrix(D) @ q
    q_proj = np.asarray(S, dtype=np.float64) @ q_rot
    return estimated_scores(q_rot[None, :], q_proj[None, :], keys, centroids)[0]


def estimated_scores(q_rot, q_proj, keys, centroids):
    """Estimated <q_h, k_t> for rotated queries q_rot [G, d], projected queries q_proj [G, d] -> [G, T]."""
    d = q_rot.shape[1]
    kappa = np.sqrt(np.pi / 2.0) / d
    c = np.asarray(centroids, dtype=np.float64)[keys.idx]            # [T, d]
    pm = 2.0 * keys.sign.astype(np.float64) - 1.0                    # [T, d]
    mse = q_rot @ c.T                                                # [G, T]
    qjl = q_proj @ pm.T                                              # [G, T]
    n = keys.norm.astype(np.float64)[None, :]
    g = keys.gamma.astype(np.float64)[None, :]
    return n * (mse + kappa * g * qjl)


def decode_attention(q, keys, values, ring_k, ring_v, D, S, centroids, softmax_scale=None):
    """Attention of query heads q [G, d] (one KV head's group) over packed records + ring tokens.

    keys/values: records of the packed history (may be empty, T = 0); ring_k/ring_v: [R, d] exact
    recent tokens (values as fp64). Returns out [G, d] in fp64.
    """
    q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    G, d = q.shape
    scale = 1.0 / np.sqrt(d) if softmax_scale is None else float(softmax_scale)
    Pi = rotation_matrix(D)
    parts_s, parts_v = [], []
    if keys is not None and keys.idx.shape[0] > 0:
        q_rot = q @ Pi.T
        q_proj = q_rot @ np.asarray(S, dtype=np.float64).T
        parts_s.append(scale * estimated_scores(q_rot, q_proj, keys, centroids))
        parts_v.append(dequantize_values(values, D))
    ring_k = np.asarray(ring_k, dtype=np.float64).reshape(-1, d)
    ring_v = np.asarray(ring_v, dtype=np.float64).reshape(-1, d)
    if ring_k.shape[0] > 0:
        parts_s.append(scale * (q @ ring_k.T))
        parts_v.append(ring_v)
    if not parts_s:
        return np.zeros((G, d))
    s = np.concatenate(parts_s, axis=1)
    v = np.concatenate(parts_v, axis=0)
    s = s - np.max(s, axis=1, keepdims=True)
    p = np.exp(s)
    p /= np.sum(p, axis=1, keepdims=True)
    return p @ v


def prefill_attention(q, keys, values, ring_k, ring_v, L, D, S, centroids, softmax_scale=None):
    """Causal attention of a chunk's queries over one KV head's cache after the chunk's append.

    q [n_q, G, d]: the sequence's last n_q tokens, so query i sits at position p_i = L - n_q + i.
    keys / values: records of the P packed tokens (positions 0 .. P-1); ring_k / ring_v [L - P, d]: the
    exact tokens at positions P .. L-1. Query i attends to every position <= p_i with the decode
    estimator (packed tokens through their codes, ring tokens exactly). Written as one masked score
    matrix per head: s[i, t] over all L positions, -inf where t > p_i. Returns [n_q, G, d].
    """
    q = np.asarray(q, dtype=np.float64)
    n_q, G, d = q.shape
    scale = 1.0 / np.sqrt(d) if softmax_scale is None else float(softmax_scale)
    Pi = rotation_matrix(D)
    P = 0 if keys is None else keys.idx.shape[0]
    ring_k = np.asarray(ring_k, dtype=np.float64).reshape(-1, d)
    ring_v = np.asarray(ring_v, dtype=np.float64).reshape(-1, d)
    assert P + ring_k.shape[0] == L and n_q <= L
    vals = np.concatenate([dequantize_values(values, D) if P else np.zeros((0, d)), ring_v], axis=0)  # [L, d]
    pos = L - n_q + np.arange(n_q)
    out = np.zeros((n_q, G, d))
    for g in range(G):
        qg = q[:, g, :]                                             # [n_q, d]
        parts = []
        if P:
            q_rot = qg @ Pi.T
            parts.append(estimated_scores(q_rot, q_rot @ np.asarray(S, dtype=np.float64).T, keys, centroids))
        parts.append(qg @ ring_k.T)
        s = scale * np.concatenate(parts, axis=1)                   # [n_q, L]
        s = np.where(np.arange(L)[None, :] <= pos[:, None], s, -np.inf)
        s = s - np.max(s, axis=1, keepdims=True)
        p = np.exp(s)
        p /= np.sum(p, axis=1, keepdims=True)
        out[:, g, :] = p @ vals
    return out
