"""Chunk attention, float64 (test infrastructure only).

For each head and each query row i of the chunk:
    s_ij = scale * q_i . k_j           over every visible key j
    p_ij = exp(s_ij - max_j s_ij) / sum_j exp(s_ij - max_j s_ij)
    o_i  = sum_j p_ij v_j,             lse_i = max_j s_ij + ln sum_j exp(...)
No mask: the chunk's rows see every key of the window, earlier or later
([H3-page] "Interactive Coding Worlds with Real-time Streaming Diffusion
Render", section 3.1.2 and its "Prefix cache" paragraph). The visible set is assembled by the caller (see
``session.py``). The score matrix is built query block by query block only to
bound memory; each block is the plain definition above.
"""
import numpy as np


def _softmax_rows(s: np.ndarray):
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    z = e.sum(axis=-1, keepdims=True)
    return e / z, (m + np.log(z))[..., 0]


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, q_block: int = 1024):
    """q [Lq][H][d], k and v [Lk][H][d] (float64). Returns (o [Lq][H][d], lse [H][Lq])."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    Lq, H, d = q.shape
    o = np.empty((Lq, H, v.shape[2]), np.float64)
    lse = np.empty((H, Lq), np.float64)
    for h in range(H):
        kh = k[:, h, :]
        vh = v[:, h, :]
        for r0 in range(0, Lq, q_block):
            r1 = min(Lq, r0 + q_block)
            s = scale * (q[r0:r1, h, :] @ kh.T)
            p, l = _softmax_rows(s)
            o[r0:r1, h, :] = p @ vh
            lse[h, r0:r1] = l
    return o, lse


def attention_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, rows, heads):
    """The same definition for a sample of (row, head) pairs: returns
    (o [len(rows)][len(heads)][d], lse [len(heads)][len(rows)])."""
    rows = np.asarray(rows)
    heads = np.asarray(heads)
    qs = np.asarray(q, np.float64)[rows][:, heads, :]
    ks = np.asarray(k, np.float64)[:, heads, :]
    vs = np.asarray(v, np.float64)[:, heads, :]
    return attention(qs, ks, vs, scale)
