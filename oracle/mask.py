"""The sparse-tree BlockMask M, element by element (oracle; test infrastructure).

Source: SpecForge review, §三 "稀疏树注意力 / BlockMask 构造算法" and §四
"BlockMask 构造".  With q a query index in [0, Q_LEN) and kv an index into the
concatenation of the k+1 TTT KV blocks, kv in [0, (k+1)*Q_LEN):

    M_causal = (q >= kv) AND (kv < T)
    M_suffix = (kv >= Q_LEN) AND (kv mod Q_LEN < T) AND ((kv - q) mod Q_LEN == 0)
    M        = M_causal OR M_suffix

The page gives the name ``m_pad`` to two different predicates (kv < T in the
causal part, kv mod Q_LEN < T in the suffix part); each is read as written in
its own formula.  ``mod`` is the mathematical (non-negative) remainder, which
is what Python's ``%`` computes for a positive modulus.
"""

import numpy as np


def mask_element(q: int, kv: int, T: int, Q_LEN: int) -> bool:
    """M[q, kv] from the formula, for one pair of Python integers."""
    m_causal = q >= kv
    m_pad = kv < T
    causal = m_causal and m_pad
    m_suffix = kv >= Q_LEN
    m_pad_suffix = (kv % Q_LEN) < T
    m_diag = ((kv - q) % Q_LEN) == 0
    suffix = m_suffix and m_pad_suffix and m_diag
    return causal or suffix


def mask_matrix_loops(T: int, Q_LEN: int, k: int) -> np.ndarray:
    """Dense bool mask [Q_LEN, (k+1)*Q_LEN] built by literal Python loops.

    Slow (pure Python); meant for tiny sizes, where it is the most direct
    transcription of the formula.
    """
    kv_len = (k + 1) * Q_LEN
    out = np.zeros((Q_LEN, kv_len), dtype=bool)
    for q in range(Q_LEN):
        for kv in range(kv_len):
            out[q, kv] = mask_element(q, kv, T, Q_LEN)
    return out


def mask_matrix(T: int, Q_LEN: int, k: int, rows=None) -> np.ndarray:
    """The same predicate evaluated by NumPy broadcasting.

    ``rows`` optionally selects a subset of query indices (an int array); the
    result then has one row per selected query.
    """
    q = np.arange(Q_LEN, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    q = q[:, None]
    kv = np.arange((k + 1) * Q_LEN, dtype=np.int64)[None, :]
    m_causal = q >= kv
    m_pad = kv < T
    m_suffix = kv >= Q_LEN
    m_pad_suffix = np.mod(kv, Q_LEN) < T
    m_diag = np.mod(kv - q, Q_LEN) == 0
    return (m_causal & m_pad) | (m_suffix & m_pad_suffix & m_diag)


def causal_block_mask(T: int, Q_LEN: int, rows=None) -> np.ndarray:
    """The formula restricted to block 0 (kv in [0, Q_LEN)).

    Only M_causal can hold there, because M_suffix requires kv >= Q_LEN; the
    full predicate is still evaluated so nothing is assumed.
    """
    full = mask_matrix(T, Q_LEN, 0, rows)
    return full


def suffix_keys(T: int, Q_LEN: int, k: int, q: int):
    """Keys of blocks 1..k that the formula lets query q see.

    Within block j (kv = j*Q_LEN + c, 0 <= c < Q_LEN) the predicate reduces to
    c < T and (c - q) mod Q_LEN == 0, i.e. c == q, so query q < T sees exactly
    the key at position q of every later block and a query q >= T sees none.
    The return value is the list of (j, c) pairs; tests confirm it against the
    formula by brute force.
    """
    if q < T:
        return [(j, q) for j in range(1, k + 1)]
    return []
