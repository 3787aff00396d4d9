"""CPU-side checks of the C ABI: the library loads, exports every function the
headers declare, and rejects invalid arguments on the host (no GPU needed:
validation happens before any CUDA call)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ra():
    from context_long_sequence_ring_gb300 import build, ringattn
    if not os.path.exists(build.LIB):
        build.build()
    return ringattn


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(ra_[a-z0-9_]+)\s*\(", src))
    return names


def test_headers_declare_the_boundary():
    names = _declared()
    for n in ["ra_zigzag_partition", "ra_gather_rows", "ra_ring_attn_fwd", "ra_lse_merge", "ra_cp_slot_mapping",
              "ra_cp_kv_scatter", "ra_cp_decode", "ra_cp_decode_workspace_size", "ra_device_status",
              "ra_last_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(ra):
    L = ctypes.CDLL(ra.LIB)
    missing = [n for n in sorted(_declared()) if not hasattr(L, n)]
    assert not missing, missing
    # and the binding knows every declared function
    known = set(ra.SIGNATURES) | set(ra.STRING_FUNCS)
    assert _declared() <= known, _declared() - known


def test_version_and_empty_error(ra):
    assert "sm_103a" in ra.version()
    assert ra.last_error() == ""


def _call(ra, name, *args):
    return getattr(ra.lib(), name)(*args)


def test_attention_argument_validation(ra):
    p = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    base = dict(B=1, Hq=4, Hkv=2, S=256, d=128, dt=1, causal=1, N=2, scale=0.0, layout=0)

    def run(**kw):
        a = dict(base, **kw)
        return _call(ra, "ra_ring_attn_fwd", p, p, p, p, p, a["B"], a["Hq"], a["Hkv"], a["S"], a["d"], a["dt"],
                     a["causal"], a["N"], a["scale"], a["layout"], None)

    assert run(Hq=3) == ra.RA_ERR_INVALID_ARG and "multiple of Hkv" in ra.last_error()
    assert run(S=250) == ra.RA_ERR_INVALID_ARG and "2*n_ranks" in ra.last_error()
    assert run(N=0) == ra.RA_ERR_INVALID_ARG
    assert run(d=96) == ra.RA_ERR_UNSUPPORTED
    assert run(layout=7) == ra.RA_ERR_INVALID_ARG
    assert run(dt=5) == ra.RA_ERR_INVALID_ARG
    assert _call(ra, "ra_ring_attn_fwd_ex", p, p, p, p, p, 1, 4, 2, 256, 128, 1, 1, 2, 0.0, 0, 4, None) == \
        ra.RA_ERR_INVALID_ARG and "variant" in ra.last_error()
    assert _call(ra, "ra_ring_attn_fwd_ex", p, p, p, p, p, 1, 6, 2, 256, 128, 1, 1, 2, 0.0, 0, 2, None) == \
        ra.RA_ERR_INVALID_ARG and "even" in ra.last_error()
    q = ctypes.c_void_p(24)  # misaligned
    assert _call(ra, "ra_ring_attn_fwd", q, p, p, p, p, 1, 4, 2, 256, 128, 1, 1, 2, 0.0, 0, None) == \
        ra.RA_ERR_INVALID_ARG


def test_slot_mapping_rejects_bad_interleave(ra):
    p = ctypes.c_void_p(16)
    st = _call(ra, "ra_cp_slot_mapping", p, p, p, 4, 1, 10, 100, 16, 2, 4, p, None)
    assert st == ra.RA_ERR_INVALID_ARG and "interleave" in ra.last_error()


def test_decode_validation_and_workspace(ra):
    n = ra.cp_decode_workspace_size(64, 32, 128, 129, 2, 4, 8)
    P = 8 * 17
    assert n >= P * 64 * 32 * 128 * 4 + P * 64 * 32 * 4
    p = ctypes.c_void_p(16)
    st = _call(ra, "ra_cp_decode", p, p, p, p, p, 2, 32, 8, 128, 100, 16, 2, 4, 4, 16, 0.0, 2, p, 1, p, p, 1 << 30,
               None)
    assert st == ra.RA_ERR_INVALID_ARG
    st = _call(ra, "ra_cp_decode", p, p, p, p, p, 2, 32, 8, 96, 128, 16, 2, 4, 4, 16, 0.0, 2, p, 1, p, p, 1 << 30,
               None)
    assert st == ra.RA_ERR_UNSUPPORTED
    st = _call(ra, "ra_cp_decode", p, p, p, p, p, 2, 32, 8, 128, 128, 16, 2, 4, 4, 16, 0.0, 2, p, 1, p, p, 16, None)
    assert st == ra.RA_ERR_INVALID_ARG and "workspace" in ra.last_error()


def test_zigzag_size_query_without_device(ra):
    lens = (ctypes.c_int64 * 2)(8, 5)
    G, T = ctypes.c_int64(0), ctypes.c_int64(0)
    assert _call(ra, "ra_zigzag_partition", lens, 2, 2, None, None, ctypes.byref(G), ctypes.byref(T), None) == 0
    assert (G.value, T.value) == (16, 13)
    bad = (ctypes.c_int64 * 1)(-1)
    assert _call(ra, "ra_zigzag_partition", bad, 1, 2, None, None, None, None, None) == ra.RA_ERR_INVALID_ARG


def test_merge_validation(ra):
    p = ctypes.c_void_p(16)
    assert _call(ra, "ra_lse_merge", p, p, 0, 4, 2, 8, p, 0, p, None) == ra.RA_ERR_INVALID_ARG
    assert _call(ra, "ra_lse_merge", p, p, 2, 4, 2, 6, p, 0, p, None) == ra.RA_ERR_UNSUPPORTED


def test_varlen_validation(ra):
    p = ctypes.c_void_p(1 << 20)

    def run(lens, n=None, dt=1, d=128, Hq=4, Hkv=2, N=2):
        arr = (ctypes.c_int64 * max(len(lens), 1))(*lens)
        return _call(ra, "ra_ring_attn_fwd_varlen", p, p, p, p, p, arr, len(lens) if n is None else n, Hq, Hkv, d, dt,
                     1, N, ctypes.c_float(0.0), None)

    assert run([8, 4], n=0) == ra.RA_ERR_INVALID_ARG
    assert run([8] * 257) == ra.RA_ERR_INVALID_ARG and "num_seqs" in ra.last_error()
    assert run([8, -1]) == ra.RA_ERR_INVALID_ARG and "negative" in ra.last_error()
    assert run([8], dt=0) == ra.RA_ERR_UNSUPPORTED
    assert run([8], d=96) == ra.RA_ERR_UNSUPPORTED
    assert run([8], Hq=3) == ra.RA_ERR_INVALID_ARG
    assert run([0, 0]) == ra.RA_OK                          # nothing to do, nothing launched


def test_rope_gather_validation(ra):
    p = ctypes.c_void_p(1 << 20)
    q = ctypes.c_void_p(1 << 24)

    def run(src=p, H=4, d=128, dt=1, idx=p, rows=8, pos=p, base=10000.0, dst=q, src_rows=8):
        return _call(ra, "ra_rope_gather", src, src_rows, H, d, dt, idx, rows, pos, ctypes.c_double(base), dst, None)

    assert run(d=120) == ra.RA_ERR_INVALID_ARG and "multiple of 16" in ra.last_error()
    assert run(d=264) == ra.RA_ERR_INVALID_ARG
    assert run(d=12, dt=0) == ra.RA_ERR_INVALID_ARG and "multiple of 8" in ra.last_error()
    assert run(base=1.0) == ra.RA_ERR_INVALID_ARG and "base" in ra.last_error()
    assert run(base=float("inf")) == ra.RA_ERR_INVALID_ARG
    assert run(dt=7) == ra.RA_ERR_INVALID_ARG
    assert run(pos=None) == ra.RA_ERR_INVALID_ARG and "NULL" in ra.last_error()
    assert run(dst=ctypes.c_void_p((1 << 20) + 1024)) == ra.RA_ERR_INVALID_ARG and "overlap" in ra.last_error()
    assert run(idx=None, rows=6) == ra.RA_ERR_INVALID_ARG
    assert run(src=ctypes.c_void_p((1 << 20) + 8)) == ra.RA_ERR_INVALID_ARG and "aligned" in ra.last_error()
    assert run(rows=0) == ra.RA_OK          # nothing to do, nothing launched


def test_product_path_has_no_oracle_or_fallback():
    pkg = os.path.join(ROOT, "context_long_sequence_ring_gb300")
    for f in glob.glob(os.path.join(pkg, "*.py")) + glob.glob(os.path.join(pkg, "csrc", "*")):
        src = open(f).read()
        assert "import oracle" not in src and "from oracle" not in src, f


def test_cross_device_entry_points_validate_on_the_host(ra):
    p = ctypes.c_void_p(16)   # never dereferenced: validation fails, or only sizes are returned, first
    # ring step: rank/src outside [0, N), o_in without lse_in, a bf16 output over the fp32 running one
    step = lambda **kw: _call(ra, "ra_ring_step_fwd", p, p, p, 1, kw.get("Hq", 4), 2, 128, kw.get("d", 128), 2,
                              kw.get("rank", 0), kw.get("src", 1), 1, 0.0, kw.get("o_in", None),
                              kw.get("lse_in", None), kw.get("o_out", p), kw.get("dt", 0), p, None)
    assert step(rank=2) == ra.RA_ERR_INVALID_ARG and "rank" in ra.last_error()
    assert step(src=-1) == ra.RA_ERR_INVALID_ARG
    assert step(Hq=3) == ra.RA_ERR_INVALID_ARG and "multiple of Hkv" in ra.last_error()
    assert step(o_in=p) == ra.RA_ERR_INVALID_ARG and "together" in ra.last_error()
    assert step(o_in=p, lse_in=p, o_out=p, dt=1) == ra.RA_ERR_INVALID_ARG and "in place" in ra.last_error()
    assert step(d=96) == ra.RA_ERR_UNSUPPORTED
    # decode partials: the device range must lie in [0, pcp*dcp); NULL outputs return the count only
    P = ctypes.c_int32(0)
    part = lambda dev0, n_dev, out=None: _call(ra, "ra_cp_decode_partials", p, p, p, p, p, 3, 32, 8, 128, 128, 16, 2,
                                               4, dev0, n_dev, 33, 64, 0.0, 8, out, out, ctypes.byref(P), None)
    assert part(6, 3) == ra.RA_ERR_INVALID_ARG and "devices" in ra.last_error()
    assert part(2, 3) == ra.RA_OK and P.value == 3 * 5        # 3 devices x ceil(33/8) splits
    # rescale and head split: heads must divide over the devices
    assert _call(ra, "ra_cp_lse_rescale", p, p, 3, 0, 4, 32, 128, p, p, None) == ra.RA_ERR_INVALID_ARG
    assert _call(ra, "ra_cp_lse_rescale", p, p, 4, 4, 4, 32, 128, p, p, None) == ra.RA_ERR_INVALID_ARG
    assert _call(ra, "ra_cp_lse_rescale", p, p, 4, 1, 0, 32, 128, p, p, None) == ra.RA_OK      # R = 0: nothing to do
    assert _call(ra, "ra_cp_head_split", p, p, 3, 4, 32, 128, p, p, None) == ra.RA_ERR_INVALID_ARG
    assert _call(ra, "ra_cp_head_split", p, p, 4, 4, 32, 6, p, p, None) == ra.RA_ERR_UNSUPPORTED
