"""Pins of the RoPE oracle (rotary position embedding of Q/K rows, and its
fusion with the zigzag row gather)."""
import numpy as np
import pytest

import oracle
from oracle import rope as OR
from tests._golden import load


@pytest.mark.parametrize("case", load("rope_hand.json")["cases"], ids=lambda c: c["name"])
def test_rope_hand_worked(case):
    x = np.asarray(case["x"], dtype=np.float64)[None, None, :]
    out = oracle.apply_rope(x, [case["pos"]], case["base"])
    np.testing.assert_allclose(out[0, 0], case["out"], atol=1e-14)


def _complex_rotation(x, positions, base):
    """The page's first formula, x e^{i m theta}, on complex numbers
    z_j = x_j + i x_{j+d/2}: an independent statement of the rotation."""
    d = x.shape[-1]
    h = d // 2
    theta = base ** (-2.0 * np.arange(h) / d)
    z = x[..., :h] + 1j * x[..., h:]
    z = z * np.exp(1j * np.asarray(positions, dtype=np.float64)[:, None, None] * theta)
    return np.concatenate([z.real, z.imag], axis=-1)


@pytest.mark.parametrize("d,base", [(2, 10000.0), (8, 10000.0), (64, 10000.0), (128, 500000.0)])
def test_rope_equals_complex_rotation(d, base):
    rng = np.random.default_rng(d)
    x = rng.standard_normal((9, 3, d))
    pos = rng.integers(0, 131072, size=9)
    np.testing.assert_allclose(oracle.apply_rope(x, pos, base), _complex_rotation(x, pos, base),
                               atol=1e-9, rtol=0)


def test_rope_scores_depend_on_relative_position_only():
    """Re<RoPE(q, m), RoPE(k, n)> is a function of m - n (the page's second formula)."""
    rng = np.random.default_rng(7)
    d = 64
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((1, 1, d))
    ref = None
    for shift in (0, 1, 17, 4096, 100000):
        m, n = 37 + shift, 5 + shift
        s = float(np.sum(oracle.apply_rope(q, [m]) * oracle.apply_rope(k, [n])))
        if ref is None:
            ref = s
        assert abs(s - ref) < 1e-9 * max(1.0, abs(ref))
    # and it does change with m - n
    s2 = float(np.sum(oracle.apply_rope(q, [38]) * oracle.apply_rope(k, [5])))
    assert abs(s2 - ref) > 1e-6


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((5, 2, 16))
    y = oracle.apply_rope(x, [0, 1, 2, 1000, 123456])
    nx = x[..., :8] ** 2 + x[..., 8:] ** 2
    ny = y[..., :8] ** 2 + y[..., 8:] ** 2
    np.testing.assert_allclose(ny, nx, rtol=1e-12)


def test_rope_gather_keeps_source_positions_and_zero_pads():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((6, 2, 8))
    pos = np.array([0, 1, 2, 0, 1, 2])              # two sequences of 3 tokens
    perm = np.array([2, -1, 0, 5, 3, -1, 4, 1])
    out = oracle.rope_gather(x, perm, pos)
    for i, p in enumerate(perm):
        if p < 0:
            assert np.all(out[i] == 0)
        else:
            np.testing.assert_array_equal(out[i], oracle.apply_rope(x[p:p + 1], [pos[p]])[0])


def test_rope_gather_under_zigzag_then_restore_is_plain_rope():
    rng = np.random.default_rng(10)
    lens = [13, 20]
    N = 2
    perm, restore, _ = oracle.zigzag_partition(lens, N)
    x = rng.standard_normal((sum(lens), 2, 16))
    pos = np.concatenate([np.arange(L) for L in lens])
    back = oracle.gather_rows(oracle.rope_gather(x, perm, pos), restore)
    np.testing.assert_allclose(back, oracle.apply_rope(x, pos), atol=0)


def test_planted_rotate_half_sign_is_caught(monkeypatch):
    monkeypatch.setattr(OR, "rotate_half",
                        lambda x: np.concatenate([x[..., x.shape[-1] // 2:], -x[..., :x.shape[-1] // 2]], axis=-1))
    rng = np.random.default_rng(11)
    x = rng.standard_normal((4, 1, 8))
    pos = [1, 2, 3, 4]
    assert not np.allclose(OR.apply_rope(x, pos), _complex_rotation(x, pos, 10000.0), atol=1e-6)


def test_planted_interleaved_pairing_is_caught(monkeypatch):
    # pairing (2j, 2j+1) instead of (j, j + d/2)
    def interleaved(x):
        y = np.empty_like(x)
        y[..., 0::2] = -x[..., 1::2]
        y[..., 1::2] = x[..., 0::2]
        return y
    monkeypatch.setattr(OR, "rotate_half", interleaved)
    rng = np.random.default_rng(12)
    x = rng.standard_normal((4, 1, 8))
    pos = [1, 2, 3, 4]
    assert not np.allclose(OR.apply_rope(x, pos), _complex_rotation(x, pos, 10000.0), atol=1e-6)


def test_planted_theta_exponent_is_caught(monkeypatch):
    monkeypatch.setattr(OR, "rope_theta", lambda d, base=10000.0: np.power(base, -np.arange(d // 2) / d))
    case = [c for c in load("rope_hand.json")["cases"] if c["name"] == "d8_third_frequency"][0]
    out = OR.apply_rope(np.asarray(case["x"])[None, None, :], [case["pos"]], case["base"])
    assert not np.allclose(out[0, 0], case["out"], atol=1e-6)
