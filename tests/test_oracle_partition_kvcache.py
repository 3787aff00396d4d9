"""Pins of the zigzag partition, slot-mapping, scatter and decode oracles."""
import numpy as np
import pytest

import oracle
from oracle import kvcache as OK
from tests._golden import load, arr

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- zigzag

@pytest.mark.parametrize("case", load("zigzag_hand.json")["cases"], ids=lambda c: c["name"])
def test_zigzag_hand_worked(case):
    perm, restore, padded = oracle.zigzag_partition(case["seq_lens"], case["n_ranks"])
    assert perm.tolist() == case["perm"]
    assert restore.tolist() == case["restore"]
    assert padded.tolist() == case["padded_lens"]


@pytest.mark.parametrize("N", [1, 2, 3, 8, 16])
def test_zigzag_bijection_and_round_trip(N):
    rng = np.random.default_rng(N)
    lens = rng.integers(0, 200, size=5)
    perm, restore, padded = oracle.zigzag_partition(lens, N)
    total = int(lens.sum())
    assert len(perm) == int(padded.sum())
    assert np.all(padded % (2 * N) == 0) and np.all(padded >= lens) and np.all(padded - lens < 2 * N)
    real = perm[perm >= 0]
    assert sorted(real.tolist()) == list(range(total))          # bijection onto the tokens
    assert np.array_equal(perm[restore], np.arange(total))      # perm o restore = id
    x = rng.standard_normal((total, 3))
    gathered = oracle.gather_rows(x, perm)
    assert np.array_equal(gathered[perm < 0], np.zeros(((perm < 0).sum(), 3)))
    assert np.array_equal(oracle.gather_rows(gathered, restore), x)


def test_zigzag_rank_regions_hold_head_and_tail():
    N, L = 4, 64
    perm, _, _ = oracle.zigzag_partition([L], N)
    c = L // (2 * N)
    for r in range(N):
        mine = perm[r * 2 * c:(r + 1) * 2 * c]
        assert mine.tolist() == list(range(r * c, r * c + c)) + \
            list(range((2 * N - 1 - r) * c, (2 * N - r) * c))


# ---------------------------------------------------------------- slot mapping

def test_slot_mapping_hand_worked_locations():
    g = load("slot_mapping_hand.json")
    for loc in g["locations"]:
        assert OK.cp_token_location(loc["x"], g["block_size"], g["interleave"], g["pcp"], g["dcp"]) \
            == (loc["vb"], loc["dev"], loc["off"])
    ex = g["slot_example"]
    slot = oracle.cp_slot_mapping(ex["query_start_loc"], ex["positions"], ex["block_table"],
                                  g["block_size"], g["interleave"], g["pcp"], g["dcp"])
    assert slot.tolist() == ex["slot"]


def test_slot_mapping_rejects_bad_interleave():
    for bad in load("slot_mapping_hand.json")["invalid"]:
        with pytest.raises(ValueError):
            oracle.cp_slot_mapping([0, 1], [0], [[0]], bad["block_size"], bad["interleave"],
                                   bad["pcp"], bad["dcp"])


@pytest.mark.parametrize("bs,I,pcp,dcp", [(128, 16, 2, 4), (16, 4, 1, 2), (8, 8, 3, 1), (12, 3, 2, 2)])
def test_slot_mapping_is_a_balanced_bijection(bs, I, pcp, dcp):
    W = pcp * dcp
    V = bs * W
    nvb = 3
    x = np.arange(nvb * V)
    bt = np.array([[7, 2, 11]])
    slot = oracle.cp_slot_mapping([0, len(x)], x, bt, bs, I, pcp, dcp)
    owners = (slot >= 0).sum(axis=0)
    assert np.all(owners == 1)                                   # exactly one device per token
    for w in range(W):
        s = slot[w][slot[w] >= 0]
        assert len(s) == nvb * bs                                # block_size tokens per full vblock
        assert len(np.unique(s)) == len(s)                       # no two tokens share a slot
        assert set((s // bs).tolist()) == {7, 2, 11}
    # interleave: runs of I consecutive tokens stay on one device, then move to the next
    dev = np.argmax(slot >= 0, axis=0)
    assert np.array_equal(dev, (x % V) // I % W)


# ---------------------------------------------------------------- decode

def _tiny_decode_case(seed=0, R=3, ctx=(1, 37, 300), bs=8, I=2, pcp=2, dcp=2, Hq=4, Hkv=2, d=8):
    rng = np.random.default_rng(seed)
    W = pcp * dcp
    V = bs * W
    nvb = [-(-L // V) for L in ctx]
    NB = sum(nvb) + 2
    ids = rng.permutation(NB)
    bt = np.full((R, max(nvb)), -1, dtype=np.int64)
    p = 0
    for r in range(R):
        bt[r, :nvb[r]] = ids[p:p + nvb[r]]
        p += nvb[r]
    qsl = np.concatenate([[0], np.cumsum(ctx)])
    pos = np.concatenate([np.arange(L) for L in ctx])
    T = int(qsl[-1])
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    q = rng.standard_normal((R, Hq, d))
    slot = oracle.cp_slot_mapping(qsl, pos, bt, bs, I, pcp, dcp)
    kc = np.full((W, NB, Hkv, bs, d), np.nan)
    vc = np.full((W, NB, Hkv, bs, d), np.nan)
    oracle.cp_kv_scatter(k, v, slot, kc, vc, bs)
    return dict(q=q, k=k, v=v, kc=kc, vc=vc, bt=bt, ctx=np.array(ctx), qsl=qsl, bs=bs, I=I,
                pcp=pcp, dcp=dcp)


@pytest.mark.parametrize("split_blocks", [1, 2, 5])
def test_decode_equals_plain_attention_over_tokens(split_blocks):
    c = _tiny_decode_case()
    O, L = oracle.cp_decode(c["q"], c["kc"], c["vc"], c["bt"], c["ctx"], c["bs"], c["I"],
                            c["pcp"], c["dcp"], split_blocks)
    for r in range(len(c["ctx"])):
        s0, s1 = c["qsl"][r], c["qsl"][r + 1]
        Or, Lr = oracle.decode_reference(c["q"][r], c["k"][s0:s1], c["v"][s0:s1])
        np.testing.assert_allclose(O[r], Or, atol=1e-12)
        np.testing.assert_allclose(L[r], Lr, atol=1e-12)


def test_decode_partials_cover_each_token_once():
    c = _tiny_decode_case(seed=1, ctx=(300,), R=1)
    Op, Lp, n_splits = oracle.cp_decode_partials(c["q"], c["kc"], c["vc"], c["bt"], c["ctx"],
                                                 c["bs"], c["I"], c["pcp"], c["dcp"], 1)
    # total weight across partials = total softmax mass over the request's keys
    _, L_ref = oracle.decode_reference(c["q"][0], c["k"], c["v"])
    mass = np.exp(Lp[:, 0, :])
    np.testing.assert_allclose(np.log(mass.sum(axis=0)), L_ref, atol=1e-12)


def test_planted_slot_formula_mistake_is_caught(monkeypatch):
    # reading the cache with a wrong inverse (device and offset order swapped) must fail the pin
    monkeypatch.setattr(OK, "_device_tokens",
                        lambda w, vb, bs, I, W: vb * bs * W + (np.arange(bs) % I) * W + w)
    c = _tiny_decode_case(seed=2)
    O, _ = oracle.cp_decode(c["q"], c["kc"], c["vc"], c["bt"], c["ctx"], c["bs"], c["I"],
                            c["pcp"], c["dcp"], 2)
    r = 2
    s0, s1 = c["qsl"][r], c["qsl"][r + 1]
    Or, _ = oracle.decode_reference(c["q"][r], c["k"][s0:s1], c["v"][s0:s1])
    assert not np.allclose(O[r], Or, atol=1e-6)


def test_kv_gather_inverts_the_scatter():
    """Scatter (driven by the per-device slot arrays) then gather (driven by the location
    formula directly) returns every token's K/V row: the two directions of the block-table
    formula agree."""
    c = _tiny_decode_case(seed=3)
    k, v = oracle.cp_kv_gather(c["kc"], c["vc"], c["bt"], c["qsl"],
                               np.concatenate([np.arange(L) for L in c["ctx"]]), c["bs"], c["I"], c["pcp"], c["dcp"])
    np.testing.assert_array_equal(k, c["k"])
    np.testing.assert_array_equal(v, c["v"])


def test_kv_gather_reorders_requests():
    """Rows come out in whatever order the positions ask for: request 2's tokens backwards."""
    c = _tiny_decode_case(seed=4)
    n2 = int(c["ctx"][2])
    k2, v2 = oracle.cp_kv_gather(c["kc"], c["vc"], c["bt"], [0, 0, 0, n2], np.arange(n2)[::-1], c["bs"], c["I"],
                                 c["pcp"], c["dcp"])
    s2 = int(c["qsl"][2])
    np.testing.assert_array_equal(k2, c["k"][s2:s2 + n2][::-1])
    np.testing.assert_array_equal(v2, c["v"][s2:s2 + n2][::-1])


# ---------------------------------------------------------------- cp_lse_ag_out_rs across devices

def test_cp_lse_ag_out_rs_hand_worked():
    # W=2 devices, R=1, Hq=2, d=1.  Head 0: LSEs 0 and ln 3 -> weights 1:3; head 1: ln 3 and 0 -> 3:1.
    o = [np.array([[[1.0], [2.0]]]), np.array([[[3.0], [8.0]]])]
    lse = [np.array([[0.0, np.log(3.0)]]), np.array([[np.log(3.0), 0.0]])]
    (O0, L0), (O1, L1) = oracle.cp_lse_ag_out_rs(o, lse)
    assert O0.shape == (1, 1, 1) and O1.shape == (1, 1, 1)
    assert O0[0, 0, 0] == pytest.approx((1 * 1.0 + 3 * 3.0) / 4, abs=1e-14)     # device 0 keeps head 0
    assert O1[0, 0, 0] == pytest.approx((3 * 2.0 + 1 * 8.0) / 4, abs=1e-14)     # device 1 keeps head 1
    assert L0[0, 0] == pytest.approx(np.log(4.0), abs=1e-14) and L1[0, 0] == pytest.approx(np.log(4.0), abs=1e-14)


@pytest.mark.parametrize("W", [1, 2, 4])
def test_cp_lse_ag_out_rs_equals_the_merge_over_devices(W):
    rng = np.random.default_rng(200 + W)
    R, Hq, d = 3, 8, 5
    o = [rng.standard_normal((R, Hq, d)) for _ in range(W)]
    lse = [rng.standard_normal((R, Hq)) * 3 for _ in range(W)]
    lse[0][1, 2] = -np.inf                       # a device with no key for one (request, head)
    if W > 1:
        for w in range(W):
            lse[w][2, 5] = -np.inf               # nobody has a key: O 0, LSE -inf
    O, L = oracle.lse_merge(np.stack(o), np.stack(lse))
    out = oracle.cp_lse_ag_out_rs(o, lse)
    np.testing.assert_allclose(np.concatenate([x[0] for x in out], axis=1), O, atol=1e-13)
    np.testing.assert_array_equal(np.concatenate([x[1] for x in out], axis=1), L)


def test_cp_lse_ag_out_rs_of_device_partials_is_plain_decode():
    # per device: merge of its split partials; across devices: the collective -> plain attention
    rng = np.random.default_rng(210)
    R, Hq, Hkv, d, bs, I_, pcp, dcp = 2, 4, 2, 8, 8, 4, 2, 1
    W = pcp * dcp
    lens = [37, 70]
    T = sum(lens)
    kt = rng.standard_normal((T, Hkv, d))
    vt = rng.standard_normal((T, Hkv, d))
    q = rng.standard_normal((R, Hq, d))
    vbs = bs * W
    nvb = [-(-L // vbs) for L in lens]
    bt = np.full((R, max(nvb)), -1)
    ids = rng.permutation(sum(nvb))
    bt[0, :nvb[0]], bt[1, :nvb[1]] = ids[:nvb[0]], ids[nvb[0]:]
    qsl = np.array([0, lens[0], T])
    pos = np.concatenate([np.arange(L) for L in lens])
    slot = oracle.cp_slot_mapping(qsl, pos, bt, bs, I_, pcp, dcp)
    kc = np.zeros((W, sum(nvb), Hkv, bs, d))
    vc = np.zeros_like(kc)
    oracle.cp_kv_scatter(kt, vt, slot, kc, vc, bs)
    Op, Lp, ns = oracle.cp_decode_partials(q, kc, vc, bt, np.array(lens), bs, I_, pcp, dcp, split_blocks=1)
    dev = [oracle.lse_merge(Op[w * ns:(w + 1) * ns], Lp[w * ns:(w + 1) * ns]) for w in range(W)]
    out = oracle.cp_lse_ag_out_rs([x[0] for x in dev], [x[1] for x in dev])
    O = np.concatenate([x[0] for x in out], axis=1)
    L = np.concatenate([x[1] for x in out], axis=1)
    for r in range(R):
        Or, Lr = oracle.decode_reference(q[r], kt[qsl[r]:qsl[r + 1]], vt[qsl[r]:qsl[r + 1]])
        np.testing.assert_allclose(O[r], Or, atol=1e-12)
        np.testing.assert_allclose(L[r], Lr, atol=1e-12)


def test_planted_head_share_is_caught(monkeypatch):
    # a device keeping another device's heads must fail the merge identity
    import oracle.kvcache as K
    real = K.cp_lse_ag_out_rs
    monkeypatch.setattr(oracle, "cp_lse_ag_out_rs", lambda o, l: real(o, l)[::-1])
    with pytest.raises(AssertionError):
        test_cp_lse_ag_out_rs_equals_the_merge_over_devices(2)
