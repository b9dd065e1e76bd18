"""The C ABI without a GPU: libfme.so loads, exports every function include/fme.h
declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

import fp8_moe_expert_gb300 as fme

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fme.h")


@pytest.fixture(scope="module")
def lib():
    fme.ensure_built()
    return fme.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^(?:fme_status|int64_t|const char \*)\s*(\w+)\(", text, flags=re.M)


def test_header_declares_the_five_calls():
    names = declared_functions()
    for call in ("quantize_nvfp4_pertoken", "quantize_nvfp4_pertensor", "swiglu_quantize_nvfp4", "quantize_mxfp8",
                 "grouped_gemm_fwd_nvfp4", "grouped_gemm_fwd_nvfp4_swiglu",
                 "grouped_gemm_fwd_mxfp8",
                 "grouped_gemm_dgrad_mxfp8", "grouped_gemm_wgrad_mxfp8", "moe_route", "permute_quantize_nvfp4",
                 "permute_quantize_mxfp8", "moe_combine", "swiglu_backward_quantize_mxfp8"):
        assert call in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in fme.SYMBOLS, f"binding does not declare {name}"


def test_helpers_closed_forms(lib):
    # padded rows: floor((rows + 127 G) / 128) * 128
    assert fme.sf_padded_rows(0, 1) == 0
    assert fme.sf_padded_rows(1, 1) == 128
    assert fme.sf_padded_rows(128, 1) == 128
    assert fme.sf_padded_rows(129, 1) == 256
    assert fme.sf_padded_rows(16384, 32) == 20352
    assert fme.sf_bytes(16384, 7168, 16, 32) == 20352 * 448
    assert fme.sf_bytes(100, 96, 32, 1) == 128 * 4          # 3 scales per row, rounded up to 4
    assert fme.colwise_ld(65536, 32) == ((65536 + 127 * 32) // 128) * 128
    assert lib.fme_version().startswith(b"fme")
    # route workspace: ceil(tokens * top_k / 1024) chunks x E counters, at least 16 bytes
    assert fme.route_workspace_bytes(32768, 8, 32) == 256 * 32 * 4
    assert fme.route_workspace_bytes(1, 1, 1) == 16
    assert fme.route_workspace_bytes(1025, 1, 3) == 24
    assert fme.route_workspace_bytes(1024, 1, 3) == 16
    assert fme.route_workspace_bytes(0, 8, 32) == 16
    assert fme.route_workspace_bytes(-1, 8, 32) == 0
    for code in range(9):
        assert lib.fme_error_string(code)


def _stream():
    return ctypes.c_void_p(0)


def test_host_argument_checks(lib):
    P = ctypes.c_void_p
    good = P(0x100000)      # never dereferenced: every call below fails before launching
    odd = P(0x100001)
    q = lib.quantize_nvfp4_pertoken
    assert q(good, -1, 256, None, 1, good, good, good, None, _stream()) == 1
    assert q(good, 10, 63, None, 1, good, good, good, None, _stream()) == 3
    assert q(good, 10, 8256, None, 1, good, good, good, None, _stream()) == 3
    assert q(good, 10, 256, None, 0, good, good, good, None, _stream()) == 1
    assert q(good, 10, 256, None, 2, good, good, good, None, _stream()) == 1
    assert q(None, 10, 256, None, 1, good, good, good, None, _stream()) == 1
    assert q(odd, 10, 256, None, 1, good, good, good, None, _stream()) == 2
    assert q(good, 0, 256, None, 1, None, None, None, None, _stream()) == 0     # nothing to do
    qt = lib.quantize_nvfp4_pertensor
    assert qt(good, 10, 96, None, 1, good, good, good, good, None, _stream()) == 3     # k % 64
    assert qt(good, 10, 256, None, 1, good, good, good, None, None, _stream()) == 1    # no amax word
    assert qt(good, 10, 256, None, 3, good, good, good, good, None, _stream()) == 1    # groups without offsets
    assert qt(good, 10, 256, None, 1, good, good, good, odd, None, _stream()) == 2
    sq = lib.swiglu_quantize_nvfp4
    assert sq(good, 10, 96, None, 1, good, good, good, None, None, _stream()) == 3      # inter % 64
    assert sq(good, 10, 8256, None, 1, good, good, good, None, None, _stream()) == 3
    assert sq(good, 10, 256, None, 2, good, good, good, None, None, _stream()) == 1     # groups without offsets
    assert sq(None, 10, 256, None, 1, good, good, good, None, None, _stream()) == 1
    assert sq(good, 10, 256, None, 1, good, good, good, odd, None, _stream()) == 2      # h misaligned
    assert sq(good, 0, 256, None, 1, None, None, None, None, None, _stream()) == 0
    m = lib.quantize_mxfp8
    assert m(good, 10, 256, 2, None, 1, good, good, None, None, _stream()) == 1
    assert m(good, 10, 256, 0, None, 1, good, good, good, None, _stream()) == 1  # row-wise takes no padded offsets
    assert m(good, 10, 48, 0, None, 1, good, good, None, None, _stream()) == 3
    assert m(good, 10, 96, 1, None, 1, good, good, good, None, _stream()) == 3   # column-wise needs cols % 128
    assert m(good, 10, 256, 1, None, 1, good, good, None, None, _stream()) == 1
    assert m(good, 10, 256, 1, None, 1, good, odd, good, None, _stream()) == 2
    sb = lib.swiglu_backward_quantize_mxfp8
    assert sb(good, good, 10, 192, None, 1, good, good, good, good, good, None, None, _stream()) == 3   # inter % 128
    assert sb(good, good, 10, 32896, None, 1, good, good, good, good, good, None, None, _stream()) == 3
    assert sb(good, good, 10, 256, None, 2, good, good, good, good, good, None, None, _stream()) == 1  # no offsets
    assert sb(good, None, 10, 256, None, 1, good, good, good, good, good, None, None, _stream()) == 1   # dh
    assert sb(good, good, 10, 256, None, 1, good, good, good, good, None, None, None, _stream()) == 1  # padded
    assert sb(good, good, 10, 256, None, 1, good, good, good, good, good, odd, None, _stream()) == 2   # d out
    assert m(good, 10, 256, 0x102, None, 1, good, good, None, None, _stream()) == 1   # ceil flag, bad axis
    assert m(good, 10, 96, 0x101, None, 1, good, good, good, None, _stream()) == 3   # ceil, column-wise cols % 128
    assert m(good, 10, 48, 0x100, None, 1, good, good, None, None, _stream()) == 3   # ceil, row-wise cols % 32
    f = lib.grouped_gemm_fwd_nvfp4
    assert f(good, good, good, good, good, good, good, 4, 100, 100, 256, good, None, _stream()) == 3
    assert f(good, good, good, good, good, good, good, 4, 100, 256, 100, good, None, _stream()) == 3
    assert f(good, good, good, good, good, good, None, 4, 100, 256, 256, good, None, _stream()) == 1
    assert f(good, good, good, good, good, good, good, 0, 100, 256, 256, good, None, _stream()) == 1
    assert f(good, good, good, good, good, good, good, 4, 100, 256, 256, odd, None, _stream()) == 2
    fm = lib.grouped_gemm_fwd_mxfp8
    assert fm(good, good, good, good, good, 4, 100, 100, 256, good, None, _stream()) == 3    # n % 256
    assert fm(good, good, good, good, good, 4, 100, 256, 96, good, None, _stream()) == 3     # k % 128
    assert fm(good, good, good, good, None, 4, 100, 256, 256, good, None, _stream()) == 1
    assert fm(good, good, good, good, good, 4, 100, 256, 256, odd, None, _stream()) == 2
    assert fm(good, good, good, good, good, 4, 0, 256, 256, None, None, _stream()) == 0     # no rows
    d = lib.grouped_gemm_dgrad_mxfp8
    assert d(good, good, good, good, 1024, good, 4, 100, 256, 512, good, None, _stream()) == 1  # ldb < E k
    assert d(good, good, good, good, 2048, good, 4, 100, 256, 96, good, None, _stream()) == 3
    w = lib.grouped_gemm_wgrad_mxfp8
    assert w(good, good, 128, good, good, 128, good, 4, 100, 256, good, None, _stream()) == 3
    assert w(good, good, 128, good, good, 128, good, 4, 128, 256, good, None, _stream()) == 3  # m % 256
    assert w(good, good, 128, good, good, 128, None, 4, 256, 256, good, None, _stream()) == 1
    r = lib.moe_route
    ws = 1 << 20
    assert r(good, 10, 8, 0, good, good, good, good, ws, None, _stream()) == 1       # no experts
    assert r(good, 10, 8, 1025, good, good, good, good, ws, None, _stream()) == 1    # too many
    assert r(good, 10, 65, 32, good, good, good, good, ws, None, _stream()) == 1     # top_k
    assert r(good, -1, 8, 32, good, good, good, good, ws, None, _stream()) == 1
    assert r(good, 1 << 29, 8, 32, good, good, good, good, ws, None, _stream()) == 3  # > 2^31 - 1 rows
    assert r(good, 10, 8, 32, good, good, good, good, 8, None, _stream()) == 1       # workspace too small
    assert r(None, 10, 8, 32, good, good, good, good, ws, None, _stream()) == 1
    assert r(good, 10, 8, 32, good, odd, good, good, ws, None, _stream()) == 2
    pn = lib.permute_quantize_nvfp4
    assert pn(good, 10, 96, good, 8, good, 32, good, good, good, None, _stream()) == 3    # k % 64
    assert pn(good, 10, 256, good, 0, good, 32, good, good, good, None, _stream()) == 1   # top_k
    assert pn(good, 10, 256, good, 8, None, 32, good, good, good, None, _stream()) == 1   # offsets
    assert pn(good, 10, 256, None, 8, good, 32, good, good, good, None, _stream()) == 1   # src_row
    assert pn(good, 10, 256, odd, 8, good, 32, good, good, good, None, _stream()) == 2
    assert pn(good, 0, 256, None, 8, good, 32, None, None, None, None, _stream()) == 0    # no rows
    pm = lib.permute_quantize_mxfp8
    assert pm(good, 10, 48, good, 8, good, 32, good, good, None, _stream()) == 3          # k % 32
    assert pm(good, 10, 256, good, 8, good, 0, good, good, None, _stream()) == 1
    assert pm(good, 10, 256, good, 8, good, 32, good, odd, None, _stream()) == 2
    assert pm(good, 0, 256, None, 8, good, 32, None, None, None, _stream()) == 0
    c = lib.moe_combine
    assert c(good, 80, good, good, 10, 8, 100, good, None, _stream()) == 3               # n % 8
    assert c(good, 80, good, good, 10, 0, 256, good, None, _stream()) == 1               # top_k
    assert c(good, 80, None, good, 10, 8, 256, good, None, _stream()) == 1
    assert c(good, 80, good, good, 10, 8, 256, odd, None, _stream()) == 2
    assert c(None, 0, None, None, 0, 8, 256, None, None, _stream()) == 0                  # no tokens
    wa = lib.grouped_gemm_wgrad_mxfp8_accumulate
    assert wa(good, good, 128, good, good, 128, good, 4, 128, 256, good, None, _stream()) == 3   # m % 256
    assert wa(good, good, 128, good, good, 128, good, 4, 256, 256, None, None, _stream()) == 1   # no buffer
    assert wa(good, good, 128, good, good, 128, good, 4, 256, 256, odd, None, _stream()) == 2
    assert lib.fme_read_device_status(None, _stream(), None) == 1


def test_binding_refuses_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(fme, "LIBRARY", str(tmp_path / "missing.so"))
    monkeypatch.setattr(fme, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        fme.lib()


def test_binding_status_constants_match_the_header():
    import re

    text = open(HEADER).read()
    for name, value in re.findall(r"#define FME_((?:OK|ERR_\w+|DEV_\w+))\s+(0x[0-9a-fA-F]+|\d+)", text):
        if name.startswith("DEV_") or name.startswith("ERR_") or name == "OK":
            assert getattr(fme, name) == int(value, 0), name
