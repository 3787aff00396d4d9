"""GPU parity of ring-order attention (C ABI) against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from context_long_sequence_ring_gb300 import inputs as I
from tests._gpu import ra_lib, assert_parity, check_status, TOL

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


@pytest.fixture(scope="module")
def ra():
    return ra_lib()


def _run(ra, seed, B, S, Hq, Hkv, d, N, causal, dtype, layout="natural", variant=0):
    q, k, v = I.prefill_inputs(seed, B, S, Hq, Hkv, d, dtype)
    dev = torch.device("cuda")
    if layout == "natural":
        o, lse = ra.ring_attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal, N, B=B, variant=variant)
    else:
        perm, restore = ra.zigzag_partition([S] * B, N)
        qz, kz, vz = (ra.gather_rows(x.to(dev), perm) for x in (q, k, v))
        oz, lz = ra.ring_attn_fwd(qz, kz, vz, causal, N, B=B, layout="zigzag", variant=variant)
        o, lse = ra.gather_rows(oz, restore), ra.gather_rows(lz, restore)
    check_status(ra)
    return q, k, v, o, lse


def _oracle_full(q, k, v, B, S, causal):
    Os, Ls = [], []
    for b in range(B):
        O, L = oracle.full_attention(q[b * S:(b + 1) * S], k[b * S:(b + 1) * S], v[b * S:(b + 1) * S], causal)
        Os.append(O)
        Ls.append(L)
    return np.concatenate(Os), np.concatenate(Ls)


# --------------------------------------------------------------------- tiny fp32 (exact path)

@pytest.mark.parametrize("layout", ["natural", "zigzag"])
def test_tiny_fp32_non_causal_four_ranks(ra, layout):
    """B=1, Hq=Hkv=2, S=256, d=64, fp32 N(0,1), non-causal, N=4 ranks of 64 tokens."""
    q, k, v, o, lse = _run(ra, 1, 1, 256, 2, 2, 64, 4, False, torch.float32, layout)
    O, L = oracle.full_attention(q, k, v, False)
    assert_parity(o, O, lse, L, torch.float32, "tiny fp32")


@pytest.mark.parametrize("S,N,causal,Hq,Hkv,d", [(96, 3, True, 4, 2, 128), (200, 2, True, 3, 1, 64),
                                                  (64, 1, False, 2, 2, 128)])
def test_fp32_ragged_and_gqa(ra, S, N, causal, Hq, Hkv, d):
    q, k, v, o, lse = _run(ra, 7, 2, S, Hq, Hkv, d, N, causal, torch.float32)
    O, L = _oracle_full(q, k, v, 2, S, causal)
    assert_parity(o, O, lse, L, torch.float32, "fp32 S=%d" % S)


# --------------------------------------------------------------------- bf16 tensor-core path

@pytest.mark.parametrize("S,N,B,Hq,Hkv,d,causal", [
    (512, 2, 1, 2, 2, 128, True),      # chunks of 128: tile-aligned
    (640, 2, 2, 4, 2, 128, True),      # chunks of 160: ragged last tile
    (1200, 3, 1, 4, 1, 128, True),     # chunks of 200, GQA group 4
    (640, 2, 1, 4, 2, 128, False),     # non-causal
    (768, 4, 1, 2, 1, 64, True),       # d = 64, chunks of 96 (single ragged tile)
    (2048, 4, 1, 2, 2, 64, False),
    (16, 8, 1, 2, 2, 128, True),       # chunks of 1 token
    (256, 1, 1, 4, 2, 128, True),      # one virtual rank: the ring is a single step
    (384, 1, 2, 2, 2, 128, False),
])
@pytest.mark.parametrize("variant", [1, 2, 3])
def test_bf16_parity_small(ra, S, N, B, Hq, Hkv, d, causal, variant):
    if variant == 2 and (Hq // Hkv) % 2:
        Hq = 2 * Hq                       # the two-head kernel needs an even GQA group
    q, k, v, o, lse = _run(ra, 3, B, S, Hq, Hkv, d, N, causal, torch.bfloat16, variant=variant)
    O, L = _oracle_full(q, k, v, B, S, causal)
    assert_parity(o, O, lse, L, torch.bfloat16, "bf16 v%d S=%d N=%d" % (variant, S, N))


@pytest.mark.parametrize("case", ["sharp_scale", "growing_keys"])
@pytest.mark.parametrize("variant", [1, 2, 3])
def test_bf16_rescale_paths(ra, case, variant):
    """Inputs that make the running max grow inside and across K/V tiles, so the lazy
    reference fails its check often: the two-pass fallback and the O rescale in tensor
    memory both run.  sharp_scale: softmax scale 0.5 (scores of std ~5.7); growing_keys:
    key rows scaled by 1 + 4 * position / S, so later tiles keep exceeding the reference."""
    B, S, Hq, Hkv, d, N = 1, 1536, 4, 2, 128, 3
    q, k, v = I.prefill_inputs(17, B, S, Hq, Hkv, d, torch.bfloat16)
    scale = None
    if case == "sharp_scale":
        scale = 0.5
    else:
        grow = 1.0 + 4.0 * torch.arange(S, dtype=torch.float32) / S
        k = (k.float() * grow[:, None, None]).to(torch.bfloat16)
    dev = torch.device("cuda")
    o, lse = ra.ring_attn_fwd(q.to(dev), k.to(dev), v.to(dev), True, N, B=B, scale=scale, variant=variant)
    check_status(ra)
    O, L = oracle.full_attention(q, k, v, True, scale=scale)
    assert_parity(o, O, lse, L, torch.bfloat16, "%s v%d" % (case, variant))


@pytest.mark.parametrize("other", [2, 3])
def test_bf16_variants_agree(ra, other):
    B, S, Hq, Hkv, d, N = 1, 2560, 8, 2, 128, 5
    _, _, _, o1, l1 = _run(ra, 6, B, S, Hq, Hkv, d, N, True, torch.bfloat16, variant=1)
    _, _, _, o2, l2 = _run(ra, 6, B, S, Hq, Hkv, d, N, True, torch.bfloat16, variant=other)
    assert (o1.float() - o2.float()).abs().max().item() <= 1.6e-2
    assert (l1 - l2).abs().max().item() <= 1e-4


def test_bf16_zigzag_layout_is_bitwise_natural(ra):
    B, S, Hq, Hkv, d, N = 2, 1280, 4, 2, 128, 4
    _, _, _, o1, l1 = _run(ra, 5, B, S, Hq, Hkv, d, N, True, torch.bfloat16, "natural")
    _, _, _, o2, l2 = _run(ra, 5, B, S, Hq, Hkv, d, N, True, torch.bfloat16, "zigzag")
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_bf16_causal_prefill_8k_full(ra):
    """B=1, Hq=Hkv=8, S=8192, d=128, causal, N=8 (16 chunks of 512), every output checked."""
    q, k, v, o, lse = _run(ra, 2, 1, 8192, 8, 8, 128, 8, True, torch.bfloat16)
    O, L = oracle.full_attention(q, k, v, True)
    assert_parity(o, O, lse, L, torch.bfloat16, "8k causal")


def _sample_rows(S, N, c, rng, n_random):
    rows = set()
    for ch in range(2 * N):
        for off in (0, 1, 127, 128, c - 1):
            if 0 <= off < c:
                rows.add(ch * c + off)
    rows |= set(rng.integers(0, S, size=n_random).tolist())
    return np.array(sorted(rows))


def _device_inputs(ra, seed, B, S, Hq, Hkv, d):
    tab = I.normal_table(torch.bfloat16)
    q = ra.synth_fill(I.tensor_key(seed, I.TID_Q), tab, (B * S, Hq, d))
    k = ra.synth_fill(I.tensor_key(seed, I.TID_K), tab, (B * S, Hkv, d))
    v = ra.synth_fill(I.tensor_key(seed, I.TID_V), tab, (B * S, Hkv, d))
    return q, k, v


def _check_sampled(o, lse, seed, b, S, Hq, Hkv, d, rows, causal=True):
    base = b * S
    qr = I.synth_rows(seed, I.TID_Q, base + rows, Hq * d, torch.bfloat16).reshape(len(rows), Hq, d)
    kk = I.synth_rows(seed, I.TID_K, base + np.arange(S), Hkv * d, torch.bfloat16).reshape(S, Hkv, d)
    vv = I.synth_rows(seed, I.TID_V, base + np.arange(S), Hkv * d, torch.bfloat16).reshape(S, Hkv, d)
    O, L = oracle.attention_rows(qr, rows, kk, vv, causal)
    idx = torch.as_tensor(base + rows, device=o.device)
    return assert_parity(o[idx], O, lse[idx], L, torch.bfloat16, "sampled rows seq %d" % b)


def test_device_generator_matches_host(ra):
    tab = I.normal_table(torch.bfloat16)
    key = I.tensor_key(9, I.TID_K)
    x = ra.synth_fill(key, tab, (1 << 20,))
    idx = np.arange(1 << 20)
    assert torch.equal(x.cpu(), I.synth_normal_at(9, I.TID_K, idx, torch.bfloat16))


def test_bf16_gqa_32k_zigzag_with_restore_round_trip(ra):
    """B=2, Hq=32, Hkv=8, S=32768, d=128, causal, N=8 zigzag ranks (16 chunks of 2048),
    tile 128; inputs permuted to the gathered layout, outputs restored; sampled rows."""
    B, S, Hq, Hkv, d, N, seed = 2, 32768, 32, 8, 128, 8, 3
    q, k, v = _device_inputs(ra, seed, B, S, Hq, Hkv, d)
    perm, restore = ra.zigzag_partition([S] * B, N)
    qz, kz, vz = (ra.gather_rows(x, perm) for x in (q, k, v))
    assert torch.equal(ra.gather_rows(qz, restore), q)          # restore o perm = identity, bit-exact
    oz, lz = ra.ring_attn_fwd(qz, kz, vz, True, N, B=B, layout="zigzag")
    o, lse = ra.gather_rows(oz, restore), ra.gather_rows(lz, restore)
    check_status(ra)
    rng = np.random.default_rng(33)
    c = S // (2 * N)
    for b in range(B):
        _check_sampled(o, lse, seed, b, S, Hq, Hkv, d, _sample_rows(S, N, c, rng, 32))


@pytest.mark.parametrize("Hq,Hkv,variant", [(24, 8, 0), (8, 8, 3)])
def test_bf16_odd_group_32k_adjacent_tiles(ra, Hq, Hkv, variant):
    """S=32768, N=8 zigzag ranks, GQA group 3 (automatic choice) and plain multi-head attention,
    on the adjacent-tile schedule with mirrored pairs (enough work to fill the GPU twice over);
    sampled rows against the oracle."""
    B, S, d, N, seed = 1, 32768, 128, 8, 8
    q, k, v = _device_inputs(ra, seed, B, S, Hq, Hkv, d)
    perm, restore = ra.zigzag_partition([S] * B, N)
    qz, kz, vz = (ra.gather_rows(x, perm) for x in (q, k, v))
    oz, lz = ra.ring_attn_fwd(qz, kz, vz, True, N, B=B, layout="zigzag", variant=variant)
    o, lse = ra.gather_rows(oz, restore), ra.gather_rows(lz, restore)
    check_status(ra)
    c = S // (2 * N)
    _check_sampled(o, lse, seed, 0, S, Hq, Hkv, d, _sample_rows(S, N, c, np.random.default_rng(81), 24))


@pytest.mark.parametrize("S,N,Hq,Hkv", [(3200, 8, 40, 8), (4800, 8, 40, 8), (4800, 8, 40, 40)])
def test_bf16_adjacent_tiles_mirrored_ragged(ra, S, N, Hq, Hkv):
    """Adjacent-tile schedule with mirrored pairs (enough CTAs for two waves) on ragged
    chunks: 200 rows (two tiles, the second short) and 300 rows (three tiles, so the last
    pair has an empty slot); sampled rows against the oracle."""
    B, d, seed = 1, 128, 9
    q, k, v = _device_inputs(ra, seed, B, S, Hq, Hkv, d)
    o, lse = ra.ring_attn_fwd(q, k, v, True, N, B=B, variant=3)
    check_status(ra)
    c = S // (2 * N)
    rows = _sample_rows(S, N, c, np.random.default_rng(91), 24)
    _check_sampled(o, lse, seed, 0, S, Hq, Hkv, d, rows)


@pytest.mark.parametrize("lens,N,Hq,Hkv,d,causal", [
    ([300, 0, 1, 1000, 77], 2, 4, 2, 128, True),     # padding in most requests, an empty and a 1-token one
    ([300, 0, 1, 1000, 77], 2, 3, 1, 128, False),    # non-causal: padding keys must be masked
    ([129, 257, 1], 3, 2, 1, 64, True),
    ([4096, 2048, 3000, 100], 4, 32, 8, 128, True),  # enough work for mirrored tile pairs
])
def test_varlen_ring_matches_per_request_attention(ra, lens, N, Hq, Hkv, d, causal):
    """Several requests of different lengths in one call on the head-tail gathered layout;
    after the restore every request equals its own full attention."""
    T = sum(lens)
    q = I.synth_normal(31, I.TID_Q, (T, Hq, d), torch.bfloat16)
    k = I.synth_normal(31, I.TID_K, (T, Hkv, d), torch.bfloat16)
    v = I.synth_normal(31, I.TID_V, (T, Hkv, d), torch.bfloat16)
    dev = torch.device("cuda")
    perm, restore = ra.zigzag_partition(lens, N)
    qz, kz, vz = (ra.gather_rows(x.to(dev), perm) for x in (q, k, v))
    oz, lz = ra.ring_attn_fwd_varlen(qz, kz, vz, lens, causal, N)
    o, lse = ra.gather_rows(oz, restore), ra.gather_rows(lz, restore)
    check_status(ra)
    Os, Ls = [], []
    start = 0
    for L in lens:
        if L:
            O, Lr = oracle.full_attention(q[start:start + L], k[start:start + L], v[start:start + L], causal)
            Os.append(O)
            Ls.append(Lr)
        start += L
    assert_parity(o, np.concatenate(Os), lse, np.concatenate(Ls), torch.bfloat16, "varlen %s" % lens)


def _long_context_rows(S, N, rng, n_random):
    """Rows checked at S=131072: the first and last row of query tiles 0, 1, nt/2-1, nt/2, nt-2 and
    nt-1 of every one of the 2N chunks (so both tiles of several mirrored pairs: tile j of chunk r
    runs with tile nt-1-j of chunk 2N-1-r), plus n_random seeded rows."""
    c = S // (2 * N)
    nt = -(-c // 128)
    rows = set()
    for ch in range(2 * N):
        for j in sorted({0, 1, nt // 2 - 1, nt // 2, nt - 2, nt - 1}):
            lo = ch * c + j * 128
            rows.update((lo, min(lo + 127, ch * c + c - 1)))
    rows.update(rng.integers(0, S, size=n_random).tolist())
    return np.array(sorted(rows))


def test_bf16_long_context_131k(ra):
    """B=1, Hq=32, Hkv=8, S=131072, d=128, causal, N=16 (32 chunks of 4096), in the launch
    configuration the benchmark times: head-tail partition, gather to the ranks' layout, ring
    attention on the zigzag layout, restore.  Checked on tile-boundary rows of all 32 chunks
    and 256 random rows."""
    B, S, Hq, Hkv, d, N, seed = 1, 131072, 32, 8, 128, 16, 5
    q, k, v = _device_inputs(ra, seed, B, S, Hq, Hkv, d)
    perm, restore = ra.zigzag_partition([S] * B, N)
    qz, kz, vz = (ra.gather_rows(x, perm) for x in (q, k, v))
    oz, lz = ra.ring_attn_fwd(qz, kz, vz, True, N, B=B, layout="zigzag")
    o, lse = ra.gather_rows(oz, restore), ra.gather_rows(lz, restore)
    check_status(ra)
    rows = _long_context_rows(S, N, np.random.default_rng(55), 256)
    kk = I.synth_rows(seed, I.TID_K, np.arange(S), Hkv * d, torch.bfloat16).reshape(S, Hkv, d).double().numpy()
    vv = I.synth_rows(seed, I.TID_V, np.arange(S), Hkv * d, torch.bfloat16).reshape(S, Hkv, d).double().numpy()
    c = S // (2 * N)
    O = np.zeros((len(rows), Hq, d))
    L = np.zeros((len(rows), Hq))
    for ch in range(2 * N):      # a causal row of chunk ch sees keys before (ch+1)*c only
        sel = np.nonzero((rows >= ch * c) & (rows < (ch + 1) * c))[0]
        if len(sel):
            qr = I.synth_rows(seed, I.TID_Q, rows[sel], Hq * d, torch.bfloat16).reshape(len(sel), Hq, d)
            O[sel], L[sel] = oracle.attention_rows(qr, rows[sel], kk[:(ch + 1) * c], vv[:(ch + 1) * c], True)
    idx = torch.as_tensor(rows, device=o.device)
    assert len(rows) >= 384 + 200
    assert_parity(o[idx], O, lse[idx], L, torch.bfloat16, "S=131072 sampled rows")


# --------------------------------------------------------------------- block partials and segmented prefill

@pytest.mark.parametrize("Tq,Tk,q0,k0,causal,Hq,Hkv,d", [
    (300, 500, 400, 0, True, 4, 2, 128),      # ragged tiles, queries after part of the keys
    (128, 256, 0, 100, True, 2, 2, 128),      # rows before every key: LSE -inf, O 0
    (77, 1000, 5000, 0, True, 8, 2, 64),      # every key visible
    (200, 333, 0, 0, False, 4, 1, 128),       # non-causal
    (256, 128, 0, 300, True, 2, 1, 128),      # no key visible to any row of the block
    (300, 500, 400, 0, True, 3, 1, 128),      # odd group, adjacent query tiles, last pair half empty
    (640, 300, 0, 200, True, 5, 5, 64),       # multi-head: early tile pairs see no key, later ones some
    (384, 256, 0, 0, False, 3, 3, 128),       # multi-head, non-causal
])
def test_block_partial_matches_oracle(ra, Tq, Tk, q0, k0, causal, Hq, Hkv, d):
    q = I.synth_normal(71, I.TID_Q, (Tq, Hq, d), torch.bfloat16)
    k = I.synth_normal(71, I.TID_K, (Tk, Hkv, d), torch.bfloat16)
    v = I.synth_normal(71, I.TID_V, (Tk, Hkv, d), torch.bfloat16)
    o, lse = ra.attn_block_fwd(q.cuda(), k.cuda(), v.cuda(), q0, k0, causal)
    check_status(ra)
    O, L = oracle.attention_block(q, q0, k, v, k0, causal)
    lg = lse.cpu().numpy()
    assert np.array_equal(np.isneginf(lg), np.isneginf(L))
    live = np.isfinite(L)
    e = np.abs(o.cpu().numpy().astype(np.float64) - O)
    assert e.max() <= 2e-2 and e.mean() <= 2e-3, (e.max(), e.mean())
    assert np.abs(lg[live] - L[live]).max(initial=0) <= 1e-3


@pytest.mark.parametrize("ctx,Tq,seg,Hq,Hkv", [(3000, 700, 1024, 4, 2), (513, 255, 128, 2, 1), (0, 600, 200, 4, 4),
                                               (3000, 700, 1024, 3, 1)])
def test_segmented_prefill_matches_full_attention(ra, ctx, Tq, seg, Hq, Hkv):
    """A chunk of Tq new tokens after ctx cached ones attends causally to all ctx+Tq keys, in
    segments of seg keys merged by LSE; equal to the plain attention rows."""
    d, T = 128, ctx + Tq
    q = I.synth_normal(72, I.TID_Q, (Tq, Hq, d), torch.bfloat16)
    k = I.synth_normal(72, I.TID_K, (T, Hkv, d), torch.bfloat16)
    v = I.synth_normal(72, I.TID_V, (T, Hkv, d), torch.bfloat16)
    o, lse = ra.segmented_prefill_fwd(q.cuda(), k.cuda(), v.cuda(), ctx, seg)
    check_status(ra)
    O, L = oracle.attention_rows(q, np.arange(ctx, T), k, v, True)
    assert_parity(o, O, lse, L, torch.bfloat16, "segmented prefill")


# --------------------------------------------------------------------- schedule

@pytest.mark.parametrize("S,N", [(512, 2), (640, 2), (8192, 8), (1200, 3), (16, 8), (2 * 16 * 300, 16)])
@pytest.mark.parametrize("kv_tile", [128, 64])
def test_schedule_counts_match_brute_force(ra, S, N, kv_tile):
    c = S // (2 * N)
    got = ra.ring_schedule_counts(S, N, True, kv_tile).cpu().tolist()
    check_status(ra)
    assert got == [list(x) for x in oracle.causal_tiles_per_rank(N, c, 128, kv_tile)]
    nt, ntk = -(-c // 128), -(-c // kv_tile)
    got_nc = ra.ring_schedule_counts(S, N, False, kv_tile).cpu().tolist()
    assert got_nc == [[2 * nt * 2 * N * ntk, 0, 0]] * N


# --------------------------------------------------------------------- failure detection

def test_bounded_wait_times_out_and_context_survives(ra):
    ra.selftest_wait_timeout(1 << 20)
    st = ra.device_status()
    assert st == ra.RA_ERR_TIMEOUT, (st, ra.last_error())
    assert ra.device_status() == 0          # cleared
    # the context is still usable
    q, k, v, o, lse = _run(ra, 1, 1, 256, 2, 2, 64, 4, False, torch.float32)
    O, L = oracle.full_attention(q, k, v, False)
    assert_parity(o, O, lse, L, torch.float32, "after timeout")


def test_invalid_arguments_raise(ra):
    q = torch.zeros((250, 2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ra.RingAttnError):
        ra.ring_attn_fwd(q, q, q, True, 4)
    assert TOL  # tolerance table is shared with the other GPU tests
