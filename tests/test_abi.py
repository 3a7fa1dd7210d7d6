"""The C-ABI library loads, exports every symbol include/pa.h declares, and rejects
bad arguments before any CUDA call (no GPU needed)."""
import ctypes

import pytest

from paged_kv_cache_08_gb300 import _native


@pytest.fixture(scope="module")
def lib():
    return _native.load()


def test_exports_every_header_symbol(lib):
    names = _native.header_functions()
    assert "pa_decode" in names and "pa_cache_write" in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding declares a signature for each one
    assert set(names) <= set(_native._SIGNATURES), set(names) - set(_native._SIGNATURES)


def test_status_strings(lib):
    for code in _native.STATUS:
        s = lib.pa_status_string(code)
        assert s and s != b"unknown status"
    assert lib.pa_status_string(12345) == b"unknown status"


def _decode(lib, **kw):
    args = dict(out=16, q=16, kc=16, vc=16, bt=16, cl=16, scale=0.1, hkv=2, S=1, hq=12, d=128, b=16, nb=4,
                maxb=4, dtype=0, ws=None, wsb=0, stream=None)
    args.update(kw)
    return lib.pa_decode(args["out"], args["q"], args["kc"], args["vc"], args["bt"], args["cl"], args["scale"],
                         args["hkv"], args["S"], args["hq"], args["d"], args["b"], args["nb"], args["maxb"],
                         args["dtype"], args["ws"], args["wsb"], args["stream"])


def test_decode_rejects_before_launch(lib):
    E = {v: k for k, v in _native.STATUS.items()}
    assert _decode(lib, d=64) == E["PA_ERR_UNSUPPORTED"]          # head_dim other than 128
    assert _decode(lib, b=8) == E["PA_ERR_UNSUPPORTED"]           # block size outside 16..128
    assert _decode(lib, hq=7) == E["PA_ERR_INVALID_ARG"]          # Hq not a multiple of Hkv
    assert _decode(lib, dtype=5) == E["PA_ERR_INVALID_ARG"]
    assert _decode(lib, out=None) == E["PA_ERR_INVALID_ARG"]      # null output
    assert _decode(lib, q=24) == E["PA_ERR_INVALID_ARG"]          # misaligned q
    assert _decode(lib, hkv=1, hq=17) == E["PA_ERR_UNSUPPORTED"]  # G > 16: no kernel for that group
    assert _decode(lib, S=0) == 0                                 # empty batch: nothing to do
    # a long table needs a split workspace; none given
    assert _decode(lib, S=1, maxb=1024) == E["PA_ERR_WORKSPACE"]


def test_cache_write_rejects_before_launch(lib):
    E = {v: k for k, v in _native.STATUS.items()}
    f = lib.pa_cache_write
    assert f(16, 16, 16, 16, 16, 4, 2, 12, 16, 8, 0, None) == E["PA_ERR_INVALID_ARG"]   # D % 8
    assert f(16, 16, 16, 16, 16, 4, 2, 128, 16, 8, 3, None) == E["PA_ERR_INVALID_ARG"]  # dtype
    assert f(None, 16, 16, 16, 16, 4, 2, 128, 16, 8, 0, None) == E["PA_ERR_INVALID_ARG"]
    assert f(16, 16, 12, 16, 16, 4, 2, 128, 16, 8, 0, None) == E["PA_ERR_INVALID_ARG"]  # slots not 8-aligned
    assert f(None, None, None, None, None, 0, 2, 128, 16, 8, 0, None) == 0              # no tokens


def test_plan_and_workspace(lib):
    import paged_kv_cache_08_gb300 as pa
    # explicit split lengths must be multiples of max(block_size, 64)
    assert pa.plan_tokens_per_split(4, 12, 2, 128, 16, 128, tokens_per_split=128) == 128
    with pytest.raises(pa.PAError):
        pa.plan_tokens_per_split(4, 12, 2, 128, 128, 128, tokens_per_split=64)
    # one split per sequence -> no workspace
    tps = pa.plan_tokens_per_split(4096, 32, 32, 128, 32, 128)
    assert tps >= 128 * 32
    assert pa.decode_workspace_size(4096, 32, 32, 128, 32, 128) == 0
    # forced splits -> (S * Hq * splits) partial rows of 128 floats + (m, l)
    ws = pa.decode_workspace_size(2, 4, 2, 128, 16, 64, tokens_per_split=256, math="fma")
    assert ws == 2 * 4 * 4 * (128 * 4 + 8)
    # persistent kernel: 2 pieces per CTA of G rows, (m, l) per row, one counter per (seq, kv head)
    ws = pa.decode_workspace_size(3, 4, 2, 128, 16, 64, num_ctas=10)
    a256 = lambda n: (n + 255) // 256 * 256
    assert ws == a256(10 * 2 * 16 * 128 * 4) + a256(10 * 2 * 16 * 8) + a256(3 * 2 * 4)
    assert pa.kernel_kind(3, 4, 2) == 2 and pa.kernel_kind(3, 4, 2, math="fma") == 1
    assert pa.kernel_kind(2000, 4, 2) == 3           # too many sequences for the on-chip prefix sums
    with pytest.raises(pa.PAError):
        pa.kernel_kind(3, 17, 1)                     # G = 17: no kernel


def test_plan_sections_lie_inside_the_plan(lib):
    """pa_decode_plan_sections: the bounds and rates sections of a plan sit inside the bytes that
    pa_decode_plan_size asks for, and follow the grid the options name."""
    import ctypes
    import paged_kv_cache_08_gb300._native as nat
    for ctas_req, ctas_want in ((10, 10), (1, 1)):
        o = nat.DecodeOptions(0, 0, ctas_req, nat.PLAN_ADAPTIVE, None)
        size = lib.pa_decode_plan_size(4, 12, 2, 128, 16, 64, ctypes.byref(o))
        C, b, r = ctypes.c_int(0), ctypes.c_size_t(0), ctypes.c_size_t(0)
        assert lib.pa_decode_plan_sections(4, 12, 2, 128, 16, 64, ctypes.byref(o), ctypes.byref(C), ctypes.byref(b),
                                           ctypes.byref(r)) == 0
        assert C.value == ctas_want
        assert b.value % 4 == 0 and r.value % 16 == 0
        assert b.value + 4 * (2 * C.value + 1) <= r.value and r.value + 4 * C.value <= size
    o = nat.DecodeOptions(0, 0, -1, 0, None)
    assert lib.pa_decode_plan_sections(4, 12, 2, 128, 16, 64, ctypes.byref(o), ctypes.byref(C), ctypes.byref(b),
                                       ctypes.byref(r)) != 0
