"""Speculative-decoding verification by rejection sampling (oracle; test
infrastructure).

Source: the "FlashSpec" practice page, §3.4 "验证器的具体实现" (how the
verifier decides to accept or reject).  For each sequence b, the draft
proposed tokens x_0 .. x_{gamma-1}; at position i the draft's distribution is
p_d[b, i, :] and the target model's is p_t[b, i, :].  Walking the positions
in order:

    accept x_i   with probability min(1, p_t[x_i] / p_d[x_i]);
    otherwise    sample one token from norm(max(0, p_t - p_d)) at that
                 position, append it, and stop.

Every accepted token is appended; the page's verifier draws nothing more when
all gamma tokens are accepted.  The page states the purpose: the tokens that
come out follow the target model's distribution exactly.

Readings where the page is silent:
  * The random numbers are inputs: u_accept[b, i] in [0, 1) for the test at
    position i, u_sample[b] in [0, 1) for the one resampling draw.  "With
    probability a" is u < a.
  * The test u < min(1, p_t / p_d) is evaluated as u * p_d < p_t in float64
    (exact for float32 inputs, and the same for p_d > 0); a draft token with
    p_d = 0 is accepted iff p_t > 0.
  * Sampling from norm(r) with one uniform u is the inverse CDF, on weights
    made exact so that the integer it decides does not depend on the order
    of a sum: r_v = min(1, max(0, p_t[v] - p_d[v])) with the difference
    rounded to float32, quantised to q_v = floor(r_v * 2^s) with
    s = 62 - bitlen(V) (so sum(q) < 2^63; weights below 2^-s, at most
    V * 2^-s of the mass, are dropped); u is quantised to
    u24 = floor(u * 2^24); the threshold is t = floor(u24 * Q / 2^24) with
    Q = sum(q), and the draw is the smallest y with q_0 + ... + q_y > t.
    All of it is integer arithmetic.
  * If Q = 0 the draw is taken from p_t itself by the same rule
    (convention: it arises only when p_t <= p_d everywhere).
  * A draft token outside [0, V) has probability 0 under both models, so it
    is never accepted (convention for invalid input).
  * A target row that is all zero leaves nothing to draw: the token is -1.
  * Output per sequence: the number of accepted draft tokens n_acc, and
    tokens[b, :] = x_0 .. x_{n_acc-1}, then the resampled token if
    n_acc < gamma, then -1.
"""

import math

import numpy as np


def quantised_weights(w, V):
    """q_v = floor(min(1, max(0, w_v)) * 2^(62 - bitlen(V))) as Python ints;
    w is float32 (the residual or the target row)."""
    s = 62 - int(V).bit_length()
    w = np.minimum(np.float32(1.0), np.maximum(np.float32(0.0), np.asarray(w, dtype=np.float32)))
    return [int(math.floor(float(x) * 2.0 ** s)) for x in w]


def inverse_cdf(q, u):
    """Smallest index y with q[0] + ... + q[y] > floor(u24 * Q / 2^24), where
    Q = sum(q) and u24 = floor(u * 2^24) (exact integer arithmetic); -1 if
    Q = 0."""
    Q = sum(q)
    if Q == 0:
        return -1
    u24 = int(math.floor(float(np.float32(u)) * 2.0 ** 24))
    t = (u24 * Q) >> 24
    acc = 0
    for y, x in enumerate(q):
        acc += x
        if acc > t:
            return y
    return -1


def verify_row(p_t, p_d, tokens, u_accept, u_sample):
    """One sequence: p_t, p_d [gamma, V]; tokens, u_accept [gamma]; u_sample scalar.
    Returns (n_acc, out [gamma] int64)."""
    p_t = np.asarray(p_t, dtype=np.float64)
    p_d = np.asarray(p_d, dtype=np.float64)
    gamma = len(tokens)
    out = np.full(gamma, -1, dtype=np.int64)
    V = p_t.shape[1]
    for i in range(gamma):
        x = int(tokens[i])
        # a token outside the vocabulary has no probability under either model
        pt, pd = (float(p_t[i, x]), float(p_d[i, x])) if 0 <= x < V else (0.0, 0.0)
        accept = (float(u_accept[i]) * pd < pt) if pd > 0.0 else (pt > 0.0)
        if accept:
            out[i] = x
            continue
        # the residual, with the difference rounded to float32
        r = np.asarray(p_t[i], dtype=np.float32) - np.asarray(p_d[i], dtype=np.float32)
        q = quantised_weights(r, V)
        if sum(q) == 0:
            q = quantised_weights(np.asarray(p_t[i], dtype=np.float32), V)
        out[i] = inverse_cdf(q, u_sample)
        return i, out
    return gamma, out


def verify(p_t, p_d, tokens, u_accept, u_sample):
    """All sequences: p_t, p_d [B, gamma, V]; tokens, u_accept [B, gamma];
    u_sample [B].  Returns (n_acc [B] int64, out [B, gamma] int64)."""
    B = len(tokens)
    n_acc = np.zeros(B, dtype=np.int64)
    out = np.zeros((B, len(tokens[0])), dtype=np.int64)
    for b in range(B):
        n_acc[b], out[b] = verify_row(p_t[b], p_d[b], tokens[b], u_accept[b], u_sample[b])
    return n_acc, out
