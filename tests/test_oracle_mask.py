"""Pins of the oracle's BlockMask against the page's formula, a hand-derived
golden matrix and brute-force key counts (SpecForge review, §三 / §四 BlockMask)."""

import os

import numpy as np
import pytest

from oracle import mask as om
from oracle import attention as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_golden_mask():
    rows = []
    for line in open(os.path.join(GOLDEN, "mask_q4_t3_k2.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        rows.append([int(x) for x in line.split()])
    return np.array(rows, dtype=bool)


def test_golden_hand_mask():
    ref = _load_golden_mask()
    assert ref.shape == (4, 12)
    assert np.array_equal(om.mask_matrix_loops(3, 4, 2), ref)
    assert np.array_equal(om.mask_matrix(3, 4, 2), ref)
    assert ref.sum() == 15


CASES = [(T, Q, k) for Q in (1, 2, 5, 8, 13) for T in sorted({0, 1, Q // 2, Q - 1, Q}) if 0 <= T <= Q
         for k in (0, 1, 3)]


@pytest.mark.parametrize("T,Q,k", CASES)
def test_loops_equal_broadcast(T, Q, k):
    assert np.array_equal(om.mask_matrix_loops(T, Q, k), om.mask_matrix(T, Q, k))


@pytest.mark.parametrize("T,Q,k", CASES)
def test_bruteforce_key_sets(T, Q, k):
    """Each valid row q < T sees keys {0..q} of block 0 plus exactly key q of every
    later block; each padded row sees exactly {0..T-1}; nothing else."""
    M = om.mask_matrix_loops(T, Q, k)
    for q in range(Q):
        keys = set(np.nonzero(M[q])[0].tolist())
        if q < T:
            want = set(range(q + 1)) | {q + j * Q for j in range(1, k + 1)}
        else:
            want = set(range(T))
        assert keys == want, (q, sorted(keys), sorted(want))
        assert len(keys) == (q + 1 + k if q < T else T)


@pytest.mark.parametrize("T,Q,k", CASES)
def test_total_count_closed_form(T, Q, k):
    assert oa.unmasked_entries(T, Q, k) == T * (T + 1) // 2 + k * T + (Q - T) * T


@pytest.mark.parametrize("T,Q,k", CASES)
def test_suffix_keys_match_formula(T, Q, k):
    for q in range(Q):
        from_formula = [(kv // Q, kv % Q) for kv in range(Q, (k + 1) * Q)
                        if om.mask_element(q, kv, T, Q)]
        assert sorted(om.suffix_keys(T, Q, k, q)) == sorted(from_formula)


def test_causal_block_has_no_suffix_term():
    for T, Q in [(0, 4), (3, 7), (7, 7)]:
        B0 = om.causal_block_mask(T, Q)
        assert np.array_equal(B0, om.mask_matrix(T, Q, 3)[:, :Q])


def test_planted_mistakes_are_caught(monkeypatch):
    """A plausible slip in the formula (dropping m_pad, or a one-off diagonal) must
    break one of the pins above."""
    good = om.mask_matrix

    def no_pad(T, Q_LEN, k, rows=None):
        q = np.arange(Q_LEN)[:, None]
        kv = np.arange((k + 1) * Q_LEN)[None, :]
        return (q >= kv) | ((kv >= Q_LEN) & (np.mod(kv - q, Q_LEN) == 0))

    def shifted_diag(T, Q_LEN, k, rows=None):
        q = np.arange(Q_LEN)[:, None]
        kv = np.arange((k + 1) * Q_LEN)[None, :]
        return ((q >= kv) & (kv < T)) | ((kv >= Q_LEN) & (np.mod(kv, Q_LEN) < T)
                                         & (np.mod(kv - q - 1, Q_LEN) == 0))

    ref = _load_golden_mask()
    for bad in (no_pad, shifted_diag):
        assert not np.array_equal(bad(3, 4, 2), ref)
        assert bad(3, 4, 2).sum() != 15 or not np.array_equal(bad(3, 4, 2), good(3, 4, 2))
