"""GPU parity of the fused RoPE + row gather (C ABI) against the float64 oracle,
alone and as the prologue of zigzag ring attention."""
import numpy as np
import pytest
import torch

import oracle
from context_long_sequence_ring_gb300 import inputs as I
from tests._gpu import ra_lib, assert_parity, check_status

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]

DEV = torch.device("cuda")


@pytest.fixture(scope="module")
def ra():
    return ra_lib()


def _positions(lens):
    return np.concatenate([np.arange(L) for L in lens]).astype(np.int32)


def _assert_rope_close(out, ref, dtype, what=""):
    """bf16: within half a bf16 ulp of the float64 value plus the fp32 rotation error
    (the kernel rotates in fp32 and rounds once); nearly every element must equal the
    correctly rounded value.  fp32: the fp32 rotation error alone."""
    o = out.float().cpu().numpy().astype(np.float64)
    err = np.abs(o - ref)
    if dtype == torch.bfloat16:
        tol = 2.0 ** -8 * np.abs(ref) + 4e-6
        assert np.all(err <= tol), "%s: max excess %.3g" % (what, (err - tol).max())
        rounded = torch.from_numpy(ref).to(torch.bfloat16).float().numpy()
        assert np.mean(o == rounded) >= 0.999, what
    else:
        assert err.max() <= 5e-6 + 1e-6 * np.abs(ref).max(), "%s: max err %.3g" % (what, err.max())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("lens,N,H,d", [
    ([300], 2, 32, 128),           # the prefill's Q shape, ragged (padded to 304)
    ([517, 64, 3], 4, 8, 128),     # several requests, K shape
    ([129], 1, 3, 64),             # odd head count, d=64
    ([77], 2, 2, 256),             # d=256
    ([1], 1, 1, 16),               # one token, smallest bf16 head
    ([200], 2, 40, 128),           # five heads per thread (past the four held in flight)
    ([90, 31], 3, 9, 64),          # head groups that do not divide the heads
])
def test_rope_gather_zigzag_matches_oracle(ra, dtype, lens, N, H, d):
    if dtype == torch.float32 and d == 16:
        d = 8
    rows = sum(lens)
    x = I.synth_normal(11, I.TID_Q, (rows, H, d), dtype)
    pos = _positions(lens)
    perm, _ = ra.zigzag_partition(lens, N)
    out = ra.rope_gather(x.to(DEV), torch.from_numpy(pos).to(DEV), perm)
    check_status(ra)
    ref = oracle.rope_gather(x.double().numpy(), perm.cpu().numpy(), pos)
    _assert_rope_close(out, ref, dtype, "lens=%s H=%d d=%d" % (lens, H, d))
    pad = (perm < 0).cpu()
    assert torch.all(out.cpu()[pad] == 0)


def test_rope_in_place_and_large_positions(ra):
    """Identity gather done in place; positions up to 2^24 - 1 (angle error must not grow)."""
    rows, H, d = 1000, 4, 128
    x = I.synth_normal(12, I.TID_K, (rows, H, d), torch.bfloat16)
    rng = np.random.default_rng(12)
    pos = rng.integers(0, 1 << 24, size=rows).astype(np.int32)
    pos[:4] = [0, 1, (1 << 24) - 1, 131071]
    xd = x.to(DEV)
    ptr = xd.data_ptr()
    y = ra.rope_gather(xd, torch.from_numpy(pos).to(DEV), out=xd)
    check_status(ra)
    assert y.data_ptr() == ptr
    _assert_rope_close(y, oracle.apply_rope(x.double().numpy(), pos), torch.bfloat16, "in place")


def test_rope_base_parameter(ra):
    rows, H, d = 256, 2, 64
    x = I.synth_normal(13, I.TID_Q, (rows, H, d), torch.float32)
    pos = np.arange(rows, dtype=np.int32) * 37
    for base in (10000.0, 500000.0, 2.0):
        out = ra.rope_gather(x.to(DEV), torch.from_numpy(pos).to(DEV), base=base)
        _assert_rope_close(out, oracle.apply_rope(x.double().numpy(), pos, base), torch.float32, "base %g" % base)
    check_status(ra)


def test_rope_full_size_prefill_sampled(ra):
    """The 131072-token prefill's Q (Hq=32) and K (Hkv=8), d=128, gathered to 16 zigzag
    ranks with the rotation fused; rows sampled at chunk edges and at random."""
    S, N, d = 131072, 16, 128
    perm, _ = ra.zigzag_partition([S], N)
    pos = torch.arange(S, dtype=torch.int32, device=DEV)
    tab = I.normal_table(torch.bfloat16)
    rng = np.random.default_rng(14)
    c = S // (2 * N)
    g = sorted(set(rng.integers(0, S, size=200).tolist()) |
               {r * c + o for r in range(2 * N) for o in (0, c - 1)} | {S - 1})
    g = np.array(g)
    perm_h = perm.cpu().numpy()
    for tid, H in ((I.TID_Q, 32), (I.TID_K, 8)):
        x = ra.synth_fill(I.tensor_key(5, tid), tab, (S, H, d))
        out = ra.rope_gather(x, pos, perm)
        check_status(ra)
        src = perm_h[g]
        xr = I.synth_rows(5, tid, src, H * d, torch.bfloat16).reshape(len(g), H, d)
        ref = oracle.apply_rope(xr.double().numpy(), src)
        _assert_rope_close(out[torch.as_tensor(g, device=DEV)], ref, torch.bfloat16, "tid %d" % tid)
        del x, out


@pytest.mark.parametrize("B,S,Hq,Hkv,d,N", [(1, 512, 4, 2, 128, 2), (2, 384, 4, 4, 64, 3)])
def test_rope_prologue_then_zigzag_ring_attention(ra, B, S, Hq, Hkv, d, N):
    """Zigzag permute with the rotation fused (Q, K) or plain (V), ring attention in the
    gathered layout, restore: equals attention over RoPE(Q), RoPE(K) in the original order.
    The rotated Q and K are bf16 tensors on the GPU, so the oracle takes them rounded to
    bf16 too (the same precision decision on both sides)."""
    q, k, v = I.prefill_inputs(21, B, S, Hq, Hkv, d, torch.bfloat16)
    pos = _positions([S] * B)
    perm, restore = ra.zigzag_partition([S] * B, N)
    pos_d = torch.from_numpy(pos).to(DEV)
    qz = ra.rope_gather(q.to(DEV), pos_d, perm)
    kz = ra.rope_gather(k.to(DEV), pos_d, perm)
    vz = ra.gather_rows(v.to(DEV), perm)
    oz, lz = ra.ring_attn_fwd(qz, kz, vz, True, N, B=B, layout="zigzag")
    o, lse = ra.gather_rows(oz, restore), ra.gather_rows(lz, restore)
    check_status(ra)
    qr = torch.from_numpy(oracle.apply_rope(q.double().numpy(), pos)).to(torch.bfloat16).double().numpy()
    kr = torch.from_numpy(oracle.apply_rope(k.double().numpy(), pos)).to(torch.bfloat16).double().numpy()
    Os, Ls = [], []
    for b in range(B):
        sl = slice(b * S, (b + 1) * S)
        O, L = oracle.full_attention(qr[sl], kr[sl], v.double().numpy()[sl], True)
        Os.append(O)
        Ls.append(L)
    assert_parity(o, np.concatenate(Os), lse, np.concatenate(Ls), torch.bfloat16, "rope + ring")


def test_rope_bad_index_is_reported(ra):
    x = torch.zeros((8, 2, 16), dtype=torch.bfloat16, device=DEV)
    idx = torch.tensor([0, 1, 8, 2], dtype=torch.int32, device=DEV)     # 8 is out of range
    out = ra.rope_gather(x, torch.zeros(8, dtype=torch.int32, device=DEV), idx)
    st = ra.device_status()
    assert st == ra.RA_ERR_DEVICE_BOUNDS and "rope" in ra.last_error()
    assert torch.all(out[2] == 0)
    check_status(ra)
