"""Pins of the float64 attention oracle against things other than itself:
hand-worked golden values, closed forms, invariants, brute force on tiny
inputs and the ring == full-attention identity of the blockwise decomposition.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
from oracle import attention as OA
from tests._golden import load, arr

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand(rng, S, Hq, Hkv, d):
    return rng.standard_normal((S, Hq, d)), rng.standard_normal((S, Hkv, d)), rng.standard_normal((S, Hkv, d))


# ---------------------------------------------------------------- golden values

def _golden_cases():
    return load("attention_hand.json")["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_full_attention_hand_worked(case):
    O, LSE = oracle.full_attention(arr(case["q"]), arr(case["k"]), arr(case["v"]),
                                   case["causal"], case["scale"])
    np.testing.assert_allclose(O, arr(case["O"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE, arr(case["LSE"]), rtol=0, atol=1e-12)


@pytest.mark.parametrize("case", [c for c in _golden_cases() if len(c["q"]) % 2 == 0],
                         ids=lambda c: c["name"])
def test_ring_attention_hand_worked(case):
    S = len(case["q"])
    for N in [n for n in (1, 2, 4) if S % (2 * n) == 0]:
        O, LSE = oracle.ring_attention(arr(case["q"]), arr(case["k"]), arr(case["v"]),
                                       case["causal"], N, case["scale"])
        np.testing.assert_allclose(O, arr(case["O"]), rtol=0, atol=1e-12)
        np.testing.assert_allclose(LSE, arr(case["LSE"]), rtol=0, atol=1e-12)


def _golden_all_pass():
    for c in _golden_cases():
        O, LSE = oracle.full_attention(arr(c["q"]), arr(c["k"]), arr(c["v"]), c["causal"], c["scale"])
        if not (np.allclose(O, arr(c["O"]), atol=1e-9) and np.allclose(LSE, arr(c["LSE"]), atol=1e-9)):
            return False
    return True


# planted mistakes (in the oracle, on the CPU) must be caught by the golden pins
@pytest.mark.parametrize("mutation", ["gqa_mod", "mask_flipped", "mask_strict", "no_scale",
                                      "log2_lse"])
def test_planted_mistakes_are_caught(monkeypatch, mutation):
    if mutation == "gqa_mod":
        monkeypatch.setattr(OA, "_kv_head_of", lambda Hq, Hkv: np.arange(Hq) % Hkv)
    elif mutation == "mask_flipped":
        monkeypatch.setattr(OA, "_visible", lambda qp, kp: kp >= qp)
    elif mutation == "mask_strict":
        monkeypatch.setattr(OA, "_visible", lambda qp, kp: kp < qp)
    elif mutation == "no_scale":
        monkeypatch.setattr(OA, "_default_scale", lambda d, s: 1.0)
    elif mutation == "log2_lse":
        real = np.log
        monkeypatch.setattr(OA.np, "log", lambda x: real(x) / math.log(2))
    assert not _golden_all_pass()


def test_planted_operand_swap_is_caught():
    c = [c for c in _golden_cases() if c["name"] == "causal_three_tokens_direction_and_operand_order"][0]
    # scores q_j.k_i instead of q_i.k_j: feed k as queries and q as keys
    O, _ = oracle.full_attention(arr(c["k"]), arr(c["q"]), arr(c["v"]), True, 1.0)
    assert not np.allclose(O, arr(c["O"]), atol=1e-6)


# ---------------------------------------------------------------- brute force

def _brute(q, k, v, causal, scale):
    """Tiny-input brute force with math.exp and Python sums (no numpy algebra)."""
    S, Hq, d = q.shape
    Hkv = k.shape[1]
    grp = Hq // Hkv
    O = np.zeros(q.shape)
    L = np.zeros((S, Hq))
    for i in range(S):
        for h in range(Hq):
            g = h // grp
            js = [j for j in range(S) if (j <= i or not causal)]
            sc = [scale * sum(q[i, h, e] * k[j, g, e] for e in range(d)) for j in js]
            mx = max(sc)
            w = [math.exp(x - mx) for x in sc]
            tot = sum(w)
            for e in range(d):
                O[i, h, e] = sum(wj * v[j, g, e] for wj, j in zip(w, js)) / tot
            L[i, h] = mx + math.log(tot)
    return O, L


@pytest.mark.parametrize("causal", [False, True])
def test_full_attention_matches_brute_force(causal):
    rng = np.random.default_rng(7)
    q, k, v = _rand(rng, 6, 4, 2, 3)
    O, L = oracle.full_attention(q, k, v, causal)
    Ob, Lb = _brute(q, k, v, causal, 1 / math.sqrt(3))
    np.testing.assert_allclose(O, Ob, atol=1e-12)
    np.testing.assert_allclose(L, Lb, atol=1e-12)


# ---------------------------------------------------------------- special cases, invariants

def test_single_token_and_first_causal_row():
    rng = np.random.default_rng(1)
    q, k, v = _rand(rng, 5, 2, 2, 4)
    O, L = oracle.full_attention(q, k, v, True)
    np.testing.assert_allclose(O[0], v[0], atol=1e-15)
    np.testing.assert_allclose(L[0], 0.5 * np.einsum("hd,hd->h", q[0], k[0]), atol=1e-14)


def test_dominant_key():
    rng = np.random.default_rng(2)
    q, k, v = _rand(rng, 8, 1, 1, 4)
    k[5] = 60.0 * q[0]        # overwhelms every other score for query 0
    O, _ = oracle.full_attention(q[:1], k, v, False)
    np.testing.assert_allclose(O[0, 0], v[5, 0], atol=1e-9)


def test_key_order_invariance_non_causal():
    rng = np.random.default_rng(3)
    q, k, v = _rand(rng, 16, 2, 1, 8)
    p = rng.permutation(16)
    O1, L1 = oracle.full_attention(q, k, v, False)
    O2, L2 = oracle.full_attention(q, k[p], v[p], False)
    np.testing.assert_allclose(O1, O2, atol=1e-13)
    np.testing.assert_allclose(L1, L2, atol=1e-13)


def test_linearity_in_v():
    rng = np.random.default_rng(4)
    q, k, v1 = _rand(rng, 12, 2, 2, 4)
    v2 = rng.standard_normal(v1.shape)
    O1, _ = oracle.full_attention(q, k, v1, True)
    O2, _ = oracle.full_attention(q, k, v2, True)
    O3, _ = oracle.full_attention(q, k, 2.0 * v1 - 3.0 * v2, True)
    np.testing.assert_allclose(O3, 2.0 * O1 - 3.0 * O2, atol=1e-12)


def test_causal_rows_ignore_future_keys():
    rng = np.random.default_rng(5)
    q, k, v = _rand(rng, 10, 2, 1, 4)
    O1, L1 = oracle.full_attention(q, k, v, True)
    k2, v2 = k.copy(), v.copy()
    k2[6:] = rng.standard_normal(k2[6:].shape)
    v2[6:] = rng.standard_normal(v2[6:].shape)
    O2, L2 = oracle.full_attention(q, k2, v2, True)
    np.testing.assert_array_equal(O1[:6], O2[:6])
    np.testing.assert_array_equal(L1[:6], L2[:6])
    assert not np.allclose(O1[6:], O2[6:])


def test_lse_bounds_and_convex_hull():
    rng = np.random.default_rng(6)
    q, k, v = _rand(rng, 9, 1, 1, 3)
    O, L = oracle.full_attention(q, k, v, True)
    for i in range(9):
        s = (q[i, 0] @ k[: i + 1, 0].T) / math.sqrt(3)
        assert s.max() - 1e-12 <= L[i, 0] <= s.max() + math.log(i + 1) + 1e-12
        assert np.all(O[i, 0] >= v[: i + 1, 0].min(axis=0) - 1e-12)
        assert np.all(O[i, 0] <= v[: i + 1, 0].max(axis=0) + 1e-12)


def test_attention_rows_agrees_with_rows_of_full():
    rng = np.random.default_rng(8)
    q, k, v = _rand(rng, 20, 4, 2, 5)
    O, L = oracle.full_attention(q, k, v, True, row_block=7)
    rows = np.array([0, 3, 19, 7])
    Or, Lr = oracle.attention_rows(q[rows], rows, k, v, True)
    np.testing.assert_array_equal(Or, O[rows])
    np.testing.assert_array_equal(Lr, L[rows])


# ---------------------------------------------------------------- ring identity

@pytest.mark.parametrize("N", [1, 2, 4, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_ring_equals_full(N, causal):
    rng = np.random.default_rng(10 + N)
    S = 2 * N * 3
    q, k, v = _rand(rng, S, 4, 2, 8)
    O1, L1 = oracle.full_attention(q, k, v, causal)
    O2, L2 = oracle.ring_attention(q, k, v, causal, N)
    np.testing.assert_allclose(O2, O1, atol=1e-12)
    np.testing.assert_allclose(L2, L1, atol=1e-12)


def test_ring_rejects_unpadded_length():
    q = np.zeros((10, 1, 2))
    with pytest.raises(ValueError):
        oracle.ring_attention(q, q, q, True, 4)


@pytest.mark.parametrize("causal", [False, True])
def test_ring_partials_merge_in_any_order(causal):
    rng = np.random.default_rng(20)
    N = 3
    q, k, v = _rand(rng, 2 * N * 2, 2, 1, 4)
    O_full, L_full = oracle.full_attention(q, k, v, causal)
    parts, pos = oracle.ring_partials(q, k, v, causal, N)
    for r in range(N):
        for order in itertools.permutations(range(N)):
            Op = np.stack([parts[r][s][0] for s in order])
            Lp = np.stack([parts[r][s][1] for s in order])
            O, L = oracle.lse_merge(Op, Lp)
            np.testing.assert_allclose(O, O_full[pos[r]], atol=1e-12)
            np.testing.assert_allclose(L, L_full[pos[r]], atol=1e-12)


# ---------------------------------------------------------------- merge

@pytest.mark.parametrize("case", load("merge_hand.json")["cases"], ids=lambda c: c["name"])
def test_merge_hand_worked(case):
    O, L = oracle.lse_merge(arr(case["o"]), arr(case["lse"]))
    np.testing.assert_allclose(O, arr(case["O"]), atol=1e-12)
    np.testing.assert_allclose(L, arr(case["LSE"]), atol=1e-12)


def test_merge_single_partial_is_identity_and_order_free():
    rng = np.random.default_rng(30)
    o = rng.standard_normal((4, 3, 5, 6))
    lse = rng.standard_normal((4, 3, 5))
    O1, L1 = oracle.lse_merge(o[:1], lse[:1])
    np.testing.assert_allclose(O1, o[0], atol=1e-15)
    np.testing.assert_allclose(L1, lse[0], atol=1e-15)
    O, L = oracle.lse_merge(o, lse)
    for p in itertools.permutations(range(4)):
        O2, L2 = oracle.lse_merge(o[list(p)], lse[list(p)])
        np.testing.assert_allclose(O2, O, atol=1e-13)
        np.testing.assert_allclose(L2, L, atol=1e-13)


# ---------------------------------------------------------------- zigzag causal balance

@pytest.mark.parametrize("N,c", [(1, 4), (2, 3), (4, 5), (8, 2), (16, 4)])
def test_causal_pairs_equal_per_rank(N, c):
    counts = oracle.causal_pairs_per_rank(N, c)
    assert counts == [(2 * N - 1) * c * c + c * (c + 1)] * N


def _visible_pairs_per_step(N, c, r, t):
    s = (r - t) % N
    qp = np.concatenate([np.arange(ch * c, ch * c + c) for ch in oracle.rank_chunks(N, r)])
    kp = np.concatenate([np.arange(ch * c, ch * c + c) for ch in oracle.rank_chunks(N, s)])
    return int((kp[None, :] <= qp[:, None]).sum())


@pytest.mark.parametrize("N,c", [(2, 3), (4, 2), (8, 3)])
def test_ring_step_liveness(N, c):
    for r in range(N):
        assert _visible_pairs_per_step(N, c, r, 0) == c * c + c * (c + 1)
        for t in range(1, N):
            assert _visible_pairs_per_step(N, c, r, t) == 2 * c * c


@pytest.mark.parametrize("N,c,T", [(2, 8, 4), (4, 6, 2), (8, 4, 4), (3, 9, 3)])
def test_causal_tiles_closed_form(N, c, T):
    nt = c // T
    full = (2 * N - 1) * nt * nt + nt * (nt - 1)
    part = 2 * nt
    skip = 2 * nt * 2 * N * nt - full - part
    assert oracle.causal_tiles_per_rank(N, c, T) == [(full, part, skip)] * N


@pytest.mark.parametrize("N,c", [(2, 256), (3, 384), (1, 128)])
def test_causal_tiles_half_key_tiles_closed_form(N, c):
    """Query tiles of 128 and key tiles of 64 (tile-aligned chunks): a query tile i of
    chunk a sees 2*a*nt full key tiles before its chunk, 2*i full ones inside it, and
    two partial (diagonal) key tiles."""
    nt = c // 128
    res = oracle.causal_tiles_per_rank(N, c, 128, 64)
    for r in range(N):
        chunks = oracle.rank_chunks(N, r)
        full = sum(2 * a * nt + 2 * i for a in chunks for i in range(nt))
        part = 2 * 2 * nt
        skip = 2 * nt * 2 * N * 2 * nt - full - part
        assert res[r] == (full, part, skip)


def test_causal_tiles_ragged_totals():
    N, c, T = 2, 5, 2          # tiles of 2,2,1 per chunk
    res = oracle.causal_tiles_per_rank(N, c, T)
    nt = 3
    for full, part, skip in res:
        assert full + part + skip == 2 * nt * 2 * N * nt
    # every visible pair is covered by a full or partial tile exactly once
    assert sum(oracle.causal_pairs_per_rank(N, c)) == (2 * N * c) * (2 * N * c + 1) // 2


# ---------------------------------------------------------------- blocks and segmented prefill

@pytest.mark.parametrize("seg", [1, 7, 64, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_segmented_attention_equals_plain_rows(seg, causal):
    """A chunk of queries at positions 90..129 over keys 0..129, any segment length:
    merging the segment partials gives the plain attention of those rows."""
    rng = np.random.default_rng(40 + seg)
    q, k, v = _rand(rng, 130, 4, 2, 8)
    rows = np.arange(90, 130)
    O, L, Op, Lp = oracle.segmented_attention(q[rows], 90, k, v, causal, seg)
    Or, Lr = oracle.attention_rows(q[rows], rows, k, v, causal)
    np.testing.assert_allclose(O, Or, atol=1e-12)
    np.testing.assert_allclose(L, Lr, atol=1e-12)
    assert Op.shape[0] == -(-130 // seg)


def test_attention_block_rows_before_every_key_are_empty():
    rng = np.random.default_rng(41)
    q, k, v = _rand(rng, 12, 2, 1, 4)
    # queries at 0..5, keys at 3..14: rows 0..2 see nothing, row 3 sees key 3 only
    O, L = oracle.attention_block(q[:6], 0, k, v, 3, True)
    assert np.all(np.isneginf(L[:3])) and np.all(O[:3] == 0)
    np.testing.assert_allclose(O[3], v[0, [0, 0]], atol=1e-15)
    np.testing.assert_allclose(L[3], 0.5 * np.einsum("hd,hd->h", q[3], k[0, [0, 0]]), atol=1e-14)


# ---------------------------------------------------------------- one ring step of one rank

def _local(x, N, c, r, B):
    """Rank r's local rows of a [B*S, ...] natural-order array: per sequence chunk r, then 2N-1-r."""
    S = 2 * N * c
    idx = np.concatenate([b * S + np.concatenate([np.arange(ch * c, ch * c + c) for ch in oracle.rank_chunks(N, r)])
                          for b in range(B)])
    return x[idx], idx


@pytest.mark.parametrize("N,c,B", [(1, 3, 1), (2, 3, 1), (3, 2, 2), (4, 2, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_ring_steps_of_a_rank_equal_full_attention(N, c, B, causal):
    # steps t = 0..N-1 on the block of rank (r - t) mod N reach the rank's rows of full attention
    rng = np.random.default_rng(100 + N * 10 + c + B)
    S = 2 * N * c
    q, k, v = _rand(rng, B * S, 4, 2, 8)
    for r in range(N):
        ql, rows = _local(q, N, c, r, B)
        O = L = None
        for t in range(N):
            s = (r - t) % N
            kl, _ = _local(k, N, c, s, B)
            vl, _ = _local(v, N, c, s, B)
            O, L = oracle.ring_step(ql, kl, vl, N, r, s, causal, O, L, B=B)
        for b in range(B):
            Of, Lf = oracle.full_attention(q[b * S:(b + 1) * S], k[b * S:(b + 1) * S], v[b * S:(b + 1) * S], causal)
            sel = slice(b * 2 * c, (b + 1) * 2 * c)
            np.testing.assert_allclose(O[sel], Of[rows[sel] - b * S], atol=1e-12)
            np.testing.assert_allclose(L[sel], Lf[rows[sel] - b * S], atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_ring_steps_in_any_order(causal):
    rng = np.random.default_rng(120)
    N, c = 3, 2
    q, k, v = _rand(rng, 2 * N * c, 2, 1, 4)
    O_full, L_full = oracle.full_attention(q, k, v, causal)
    for r in range(N):
        ql, rows = _local(q, N, c, r, 1)
        for order in itertools.permutations(range(N)):
            O = L = None
            for s in order:
                O, L = oracle.ring_step(ql, _local(k, N, c, s, 1)[0], _local(v, N, c, s, 1)[0], N, r, s, causal, O, L)
            np.testing.assert_allclose(O, O_full[rows], atol=1e-12)
            np.testing.assert_allclose(L, L_full[rows], atol=1e-12)


def test_ring_step_first_row_sees_only_its_own_key():
    # N=2, c=1, S=4: rank 0 holds positions (0, 3), rank 1 holds (1, 2).  Under the causal mask the
    # query at position 0 sees no key of rank 1's block (LSE -inf, O 0) and only key 0 of its own.
    q = np.array([[[1.0]], [[2.0]], [[0.5]], [[1.5]]])
    k = np.array([[[0.3]], [[1.0]], [[-1.0]], [[2.0]]])
    v = np.array([[[10.0]], [[20.0]], [[30.0]], [[40.0]]])
    ql, _ = _local(q, 2, 1, 0, 1)
    O1, L1 = oracle.ring_step(ql, _local(k, 2, 1, 1, 1)[0], _local(v, 2, 1, 1, 1)[0], 2, 0, 1, True)
    assert L1[0, 0] == -np.inf and O1[0, 0, 0] == 0.0
    # row 1 (position 3) sees keys 1 and 2 of the held block: scores 1.5*1.0 and 1.5*(-1.0) at scale 1
    e1, e2 = np.exp(1.5), np.exp(-1.5)
    assert O1[1, 0, 0] == pytest.approx((20 * e1 + 30 * e2) / (e1 + e2), abs=1e-12)
    assert L1[1, 0] == pytest.approx(np.log(e1 + e2), abs=1e-12)
    O0, L0 = oracle.ring_step(ql, _local(k, 2, 1, 0, 1)[0], _local(v, 2, 1, 0, 1)[0], 2, 0, 0, True)
    assert O0[0, 0, 0] == pytest.approx(10.0) and L0[0, 0] == pytest.approx(1.0 * 0.3)


def test_planted_held_block_positions_are_caught(monkeypatch):
    # a step that took the held block's keys to sit at the rank's own positions must fail the identity
    import oracle.attention as A
    real = A._rows_over_keys
    monkeypatch.setattr(A, "_rows_over_keys",
                        lambda qr, qpos, kk, vv, kpos, causal, scale: real(qr, qpos, kk, vv, qpos, causal, scale))
    with pytest.raises(AssertionError):
        test_ring_steps_of_a_rank_equal_full_attention(2, 3, 1, True)
