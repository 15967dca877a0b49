"""Helpers shared by the tests (no verification arithmetic of the product)."""
import numpy as np


def log_probs(p, dtype=np.float32):
    """Logits whose softmax is the probability vector p (zeros -> -inf)."""
    p = np.asarray(p, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.log(p).astype(dtype)


def within_sigma(freq, p, n, k=3.0):
    """True iff every |freq - p| is below k standard errors sqrt(p(1-p)/n)."""
    freq = np.asarray(freq, np.float64)
    p = np.asarray(p, np.float64)
    se = np.sqrt(np.maximum(p * (1 - p), 1e-300) / n)
    return bool(np.all(np.abs(freq - p) <= k * se)), np.abs(freq - p) / se


def midpoint_grid(n):
    """n uniforms at the midpoints (i + 0.5) / n, as float32."""
    return ((np.arange(n) + 0.5) / n).astype(np.float32)


def grid_chain_inputs(p_list, q_list, p_bonus, n, temperature=1.0):
    """Enumerate every draft tuple and every grid point of the uniforms.

    Positions j < K have target law p_list[j] and draft law q_list[j]; the
    bonus row has law p_bonus.  Logits are T * log(prob) so that softmax at
    temperature T returns the law.  Each row of the result is one point of
    (y_0..y_{K-1}, u_accept_0..u_accept_{K-1}, s) with u_sample = s at every
    position (only one u_sample entry is ever consumed).  Returns
    (inputs dict for oracle.verify_chain, weights [rows]).
    """
    K = len(p_list)
    V = len(p_bonus)
    g = midpoint_grid(n)
    ys = np.stack(np.meshgrid(*[np.arange(V)] * K, indexing="ij"), -1).reshape(-1, K)
    us = np.stack(np.meshgrid(*[g] * (K + 1), indexing="ij"), -1).reshape(-1, K + 1)
    rows_y = np.repeat(ys, len(us), axis=0)
    rows_u = np.tile(us, (len(ys), 1))
    B = len(rows_y)
    w_y = np.ones(len(ys))
    for j in range(K):
        w_y = w_y * np.asarray(q_list[j], np.float64)[ys[:, j]]
    weights = np.repeat(w_y, len(us)) / float(len(us))
    T = np.float32(temperature)
    tgt_row = np.stack([log_probs(p) * T for p in p_list] + [log_probs(p_bonus) * T])
    drf_row = np.stack([log_probs(q) * T for q in q_list])
    target = np.broadcast_to(tgt_row, (B, K + 1, V)).astype(np.float32)
    draft = np.broadcast_to(drf_row, (B, K, V)).astype(np.float32)
    inputs = dict(target=target, draft=draft, draft_tokens=rows_y.astype(np.int32),
                  temperature=np.full(B, T, np.float32),
                  u_accept=rows_u[:, :K].copy(),
                  u_sample=np.repeat(rows_u[:, K:K + 1], K + 1, axis=1))
    return inputs, weights


def softmax64(logits, T=1.0):
    x = np.asarray(logits, np.float64) / T
    m = np.max(x, axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / e.sum(axis=-1, keepdims=True)
