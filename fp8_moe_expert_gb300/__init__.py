"""GB300-native low-precision MoE expert path: NVFP4 per-token forward, MXFP8 backward.

A thin ctypes binding over ``libfme.so`` (C ABI in ``include/fme.h``).  Every
step of the path runs in the library's CUDA kernels; this module only turns
torch tensors into pointers, allocates outputs with torch when the caller does
not pass them, and turns status codes into exceptions.  There is no fallback:
if the library is missing or the device is not a GB300, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(HERE, "libfme.so")

ROWWISE = 0
COLWISE = 1
MAX_GROUPS = 1024
MX_SCALE_CEIL = 0x100
DEV_TIMEOUT = 0x1
DEV_BAD_OFFSETS = 0x2
DEV_BAD_INDEX = 0x4
# status codes (fme_status) of include/fme.h
OK = 0
ERR_INVALID_ARGUMENT = 1
ERR_MISALIGNED = 2
ERR_UNSUPPORTED_SHAPE = 3
ERR_UNSUPPORTED_DEVICE = 4
ERR_CUDA = 5
ERR_DEVICE_TIMEOUT = 6
ERR_DEVICE_BAD_OFFSETS = 7
ERR_DEVICE_BAD_INDEX = 8

_lib = None
_lock = threading.Lock()


class FmeError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: status {status}"
        if _lib is not None:
            msg += f" ({_lib.fme_error_string(status).decode()})"
        if detail:
            msg += f": {detail}"
        super().__init__(msg)


def ensure_built() -> str:
    """Build libfme.so if it is missing or older than its sources."""
    from . import build as _build

    if _build.stale():
        _build.build()
    return LIBRARY


def lib() -> ctypes.CDLL:
    """The loaded CUDA library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIBRARY):
                raise RuntimeError(f"{LIBRARY} is missing: build it with "
                                   "`python -m fp8_moe_expert_gb300.build` (no CPU fallback exists)")
            _lib = _declare(ctypes.CDLL(LIBRARY))
    return _lib


SYMBOLS = {
    # name: (restype, argtypes)
    "quantize_nvfp4_pertoken": ("i32", ["p", "i64", "i64", "p", "i32", "p", "p", "p", "p", "p"]),
    "quantize_nvfp4_pertensor": ("i32", ["p", "i64", "i64", "p", "i32", "p", "p", "p", "p", "p", "p"]),
    "swiglu_quantize_nvfp4": ("i32", ["p", "i64", "i64", "p", "i32", "p", "p", "p", "p", "p", "p"]),
    "quantize_mxfp8": ("i32", ["p", "i64", "i64", "i32", "p", "i32", "p", "p", "p", "p", "p"]),
    "quantize_mxfp8_rowcol": ("i32", ["p", "i64", "i64", "p", "i32", "p", "p", "p", "p", "p", "p", "p"]),
    "swiglu_backward_quantize_mxfp8": ("i32", ["p", "p", "i64", "i64", "p", "i32", "p", "p", "p", "p", "p", "p",
                                               "p", "p"]),
    "grouped_gemm_fwd_nvfp4": ("i32", ["p", "p", "p", "p", "p", "p", "p", "i32", "i64", "i64", "i64", "p", "p",
                                       "p"]),
    "grouped_gemm_fwd_nvfp4_swiglu": ("i32", ["p", "p", "p", "p", "p", "p", "p", "i32", "i64", "i64", "i64", "p",
                                              "p", "p"]),
    "grouped_gemm_fwd_mxfp8": ("i32", ["p", "p", "p", "p", "p", "i32", "i64", "i64", "i64", "p", "p", "p"]),
    "grouped_gemm_dgrad_mxfp8": ("i32", ["p", "p", "p", "p", "i64", "p", "i32", "i64", "i64", "i64", "p", "p",
                                         "p"]),
    "grouped_gemm_wgrad_mxfp8": ("i32", ["p", "p", "i64", "p", "p", "i64", "p", "i32", "i64", "i64", "p", "p",
                                         "p"]),
    "moe_route": ("i32", ["p", "i64", "i32", "i32", "p", "p", "p", "p", "i64", "p", "p"]),
    "moe_route_noalloc": ("i32", ["p", "i64", "i32", "i32", "p", "p", "p", "p", "p"]),
    "permute_quantize_nvfp4": ("i32", ["p", "i64", "i64", "p", "i32", "p", "i32", "p", "p", "p", "p", "p"]),
    "permute_quantize_mxfp8": ("i32", ["p", "i64", "i64", "p", "i32", "p", "i32", "p", "p", "p", "p"]),
    "moe_combine": ("i32", ["p", "i64", "p", "p", "i64", "i32", "i64", "p", "p", "p"]),
    "grouped_gemm_wgrad_mxfp8_accumulate": ("i32", ["p", "p", "i64", "p", "p", "i64", "p", "i32", "i64", "i64", "p",
                                                    "p", "p"]),
    "fme_route_workspace_bytes": ("i64", ["i64", "i32", "i32"]),
    "fme_sf_padded_rows": ("i64", ["i64", "i32"]),
    "fme_sf_bytes": ("i64", ["i64", "i64", "i32", "i32"]),
    "fme_colwise_ld": ("i64", ["i64", "i32"]),
    "fme_read_device_status": ("i32", ["p", "p", "p"]),
    "fme_error_string": ("s", ["i32"]),
    "fme_last_cuda_error": ("s", []),
    "fme_version": ("s", []),
}

_CT = {"i32": ctypes.c_int32, "i64": ctypes.c_int64, "p": ctypes.c_void_p, "s": ctypes.c_char_p}


def _declare(handle):
    for name, (res, args) in SYMBOLS.items():
        fn = getattr(handle, name)
        fn.restype = _CT[res]
        fn.argtypes = [_CT[a] for a in args]
    return handle


# ------------------------------------------------------------------ helpers --
def sf_padded_rows(rows: int, num_groups: int = 1) -> int:
    return int(lib().fme_sf_padded_rows(rows, num_groups))


def sf_bytes(rows: int, cols: int, block: int, num_groups: int = 1) -> int:
    return int(lib().fme_sf_bytes(rows, cols, block, num_groups))


def colwise_ld(rows: int, num_groups: int = 1) -> int:
    return int(lib().fme_colwise_ld(rows, num_groups))


def route_workspace_bytes(tokens: int, top_k: int, num_experts: int) -> int:
    return int(lib().fme_route_workspace_bytes(tokens, top_k, num_experts))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, where: str):
    if status != 0:
        detail = lib().fme_last_cuda_error().decode() if status == 5 else ""
        raise FmeError(status, where, detail)


def _groups(offsets, num_groups):
    if offsets is None:
        return None, 1 if num_groups is None else num_groups
    n = offsets.numel() - 1 if num_groups is None else num_groups
    return offsets, n


def _empty(shape, dtype, device):
    import torch

    return torch.empty(shape, dtype=dtype, device=device)


# --------------------------------------------------------------- the five calls --
def quantize_nvfp4_pertoken(x, offsets=None, num_groups=None, *, codes=None, sf=None, row_scale=None,
                            status=None, stream=None):
    """NVFP4 per-token quantization of bf16 x [rows, k] -> (codes [rows, k/2] u8,
    sf (tiled E4M3 scales) u8, row_scale [rows] f32)."""
    import torch

    rows, k = x.shape
    offsets, g = _groups(offsets, num_groups)
    dev = x.device
    if codes is None:
        codes = _empty((rows, k // 2), torch.uint8, dev)
    if sf is None:
        sf = _empty((max(sf_bytes(rows, k, 16, g), 16),), torch.uint8, dev)
    if row_scale is None:
        row_scale = _empty((rows,), torch.float32, dev)
    st = lib().quantize_nvfp4_pertoken(_ptr(x), rows, k, _ptr(offsets), g, _ptr(codes), _ptr(sf), _ptr(row_scale),
                                       _ptr(status), _stream(stream))
    _check(st, "quantize_nvfp4_pertoken")
    return codes, sf, row_scale


def quantize_nvfp4_pertensor(x, offsets=None, num_groups=None, *, codes=None, sf=None, row_scale=None,
                             tensor_amax=None, status=None, stream=None):
    """Standard NVFP4 (one FP32 scale for the tensor) of bf16 x [rows, k] ->
    (codes, sf, row_scale (S in every row), tensor_amax [1])."""
    import torch

    rows, k = x.shape
    offsets, g = _groups(offsets, num_groups)
    dev = x.device
    if codes is None:
        codes = _empty((rows, k // 2), torch.uint8, dev)
    if sf is None:
        sf = _empty((max(sf_bytes(rows, k, 16, g), 16),), torch.uint8, dev)
    if row_scale is None:
        row_scale = _empty((max(rows, 1),), torch.float32, dev)
    if tensor_amax is None:
        tensor_amax = _empty((4,), torch.float32, dev)
    st = lib().quantize_nvfp4_pertensor(_ptr(x), rows, k, _ptr(offsets), g, _ptr(codes), _ptr(sf),
                                        _ptr(row_scale), _ptr(tensor_amax), _ptr(status), _stream(stream))
    _check(st, "quantize_nvfp4_pertensor")
    return codes, sf, row_scale[:rows], tensor_amax[:1]


def swiglu_quantize_nvfp4(gate_up, offsets=None, num_groups=None, *, codes=None, sf=None, row_scale=None, h=None,
                          want_h=True, status=None, stream=None):
    """h = silu(g) * u of gate_up [rows x 2*inter] (bf16), NVFP4-quantized per
    token -> (codes, sf, row_scale, h or None)."""
    import torch

    rows, two_inter = gate_up.shape
    inter = two_inter // 2
    offsets, g = _groups(offsets, num_groups)
    dev = gate_up.device
    if codes is None:
        codes = _empty((rows, inter // 2), torch.uint8, dev)
    if sf is None:
        sf = _empty((max(sf_bytes(rows, inter, 16, g), 16),), torch.uint8, dev)
    if row_scale is None:
        row_scale = _empty((rows,), torch.float32, dev)
    if h is None and want_h:
        h = _empty((rows, inter), torch.bfloat16, dev)
    st = lib().swiglu_quantize_nvfp4(_ptr(gate_up), rows, inter, _ptr(offsets), g, _ptr(codes), _ptr(sf),
                                     _ptr(row_scale), _ptr(h), _ptr(status), _stream(stream))
    _check(st, "swiglu_quantize_nvfp4")
    return codes, sf, row_scale, h


def quantize_mxfp8(x, axis=ROWWISE, offsets=None, num_groups=None, *, codes=None, sf=None, padded_offsets=None,
                   status=None, stream=None):
    """MXFP8 quantization of bf16 x [rows, cols].

    ROWWISE -> (codes [rows, cols] u8, sf tiled E8M0 u8).
    COLWISE -> (codes [cols, ld] u8, sf tiled u8, padded_offsets [G+1] i32, ld)."""
    import torch

    rows, cols = x.shape
    offsets, g = _groups(offsets, num_groups)
    dev = x.device
    if (axis & ~MX_SCALE_CEIL) == ROWWISE:
        if codes is None:
            codes = _empty((rows, cols), torch.uint8, dev)
        if sf is None:
            sf = _empty((max(sf_bytes(rows, cols, 32, g), 16),), torch.uint8, dev)
        st = lib().quantize_mxfp8(_ptr(x), rows, cols, axis, _ptr(offsets), g, _ptr(codes), _ptr(sf), None,
                                  _ptr(status), _stream(stream))
        _check(st, "quantize_mxfp8")
        return codes, sf
    ld = colwise_ld(rows, g)
    if codes is None:
        codes = _empty((cols, ld), torch.uint8, dev)
    if sf is None:
        sf = _empty((max(sf_bytes(cols, ld, 32, 1), 16),), torch.uint8, dev)
    if padded_offsets is None:
        padded_offsets = _empty((g + 1,), torch.int32, dev)
    st = lib().quantize_mxfp8(_ptr(x), rows, cols, axis, _ptr(offsets), g, _ptr(codes), _ptr(sf),
                              _ptr(padded_offsets), _ptr(status), _stream(stream))
    _check(st, "quantize_mxfp8")
    return codes, sf, padded_offsets, ld


def quantize_mxfp8_rowcol(x, offsets=None, num_groups=None, *, row_codes=None, row_sf=None, col_codes=None,
                          col_sf=None, padded_offsets=None, status=None, stream=None):
    """Row-wise and column-wise MXFP8 of bf16 x [rows, cols] in one pass ->
    ((row_codes, row_sf), (col_codes, col_sf, padded_offsets, ld))."""
    import torch

    rows, cols = x.shape
    offsets, g = _groups(offsets, num_groups)
    dev = x.device
    ld = colwise_ld(rows, g)
    if row_codes is None:
        row_codes = _empty((rows, cols), torch.uint8, dev)
    if row_sf is None:
        row_sf = _empty((max(sf_bytes(rows, cols, 32, g), 16),), torch.uint8, dev)
    if col_codes is None:
        col_codes = _empty((cols, ld), torch.uint8, dev)
    if col_sf is None:
        col_sf = _empty((max(sf_bytes(cols, ld, 32, 1), 16),), torch.uint8, dev)
    if padded_offsets is None:
        padded_offsets = _empty((g + 1,), torch.int32, dev)
    st = lib().quantize_mxfp8_rowcol(_ptr(x), rows, cols, _ptr(offsets), g, _ptr(row_codes), _ptr(row_sf),
                                     _ptr(col_codes), _ptr(col_sf), _ptr(padded_offsets), _ptr(status),
                                     _stream(stream))
    _check(st, "quantize_mxfp8_rowcol")
    return (row_codes, row_sf), (col_codes, col_sf, padded_offsets, ld)


def swiglu_backward_quantize_mxfp8(gate_up, dh, offsets=None, num_groups=None, *, row_codes=None, row_sf=None,
                                   col_codes=None, col_sf=None, padded_offsets=None, d_gate_up=None,
                                   want_d=False, status=None, stream=None):
    """d(gate/up) of h = silu(g) * u given dh, quantized to MXFP8 row-wise and
    column-wise -> (row_codes, row_sf, col_codes, col_sf, padded_offsets, ld,
    d_gate_up or None)."""
    import torch

    rows, two_inter = gate_up.shape
    inter = two_inter // 2
    offsets, g = _groups(offsets, num_groups)
    dev = gate_up.device
    ld = colwise_ld(rows, g)
    if row_codes is None:
        row_codes = _empty((rows, two_inter), torch.uint8, dev)
    if row_sf is None:
        row_sf = _empty((max(sf_bytes(rows, two_inter, 32, g), 16),), torch.uint8, dev)
    if col_codes is None:
        col_codes = _empty((two_inter, ld), torch.uint8, dev)
    if col_sf is None:
        col_sf = _empty((max(sf_bytes(two_inter, ld, 32, 1), 16),), torch.uint8, dev)
    if padded_offsets is None:
        padded_offsets = _empty((g + 1,), torch.int32, dev)
    if d_gate_up is None and want_d:
        d_gate_up = _empty((rows, two_inter), torch.bfloat16, dev)
    st = lib().swiglu_backward_quantize_mxfp8(_ptr(gate_up), _ptr(dh), rows, inter, _ptr(offsets), g,
                                              _ptr(row_codes), _ptr(row_sf), _ptr(col_codes), _ptr(col_sf),
                                              _ptr(padded_offsets), _ptr(d_gate_up), _ptr(status), _stream(stream))
    _check(st, "swiglu_backward_quantize_mxfp8")
    return row_codes, row_sf, col_codes, col_sf, padded_offsets, ld, d_gate_up


def grouped_gemm_fwd_nvfp4(a_codes, a_sf, a_scale, b_codes, b_sf, b_scale, offsets, n, k, *, y=None,
                           status=None, stream=None):
    import torch

    m = a_codes.shape[0]
    e = offsets.numel() - 1
    if y is None:
        y = _empty((m, n), torch.bfloat16, a_codes.device)
    st = lib().grouped_gemm_fwd_nvfp4(_ptr(a_codes), _ptr(a_sf), _ptr(a_scale), _ptr(b_codes), _ptr(b_sf),
                                      _ptr(b_scale), _ptr(offsets), e, m, n, k, _ptr(y), _ptr(status),
                                      _stream(stream))
    _check(st, "grouped_gemm_fwd_nvfp4")
    return y


def grouped_gemm_fwd_nvfp4_swiglu(a_codes, a_sf, a_scale, b_codes, b_sf, b_scale, offsets, n, k, *, h=None,
                                  status=None, stream=None):
    """The gate/up projection's NVFP4 forward with SwiGLU in the epilogue:
    h [m x n / 2] = silu(gate) * up (bf16), gate and up the first and last n / 2
    rows of each expert's weights."""
    import torch

    m = a_codes.shape[0]
    e = offsets.numel() - 1
    if h is None:
        h = _empty((m, n // 2), torch.bfloat16, a_codes.device)
    st = lib().grouped_gemm_fwd_nvfp4_swiglu(_ptr(a_codes), _ptr(a_sf), _ptr(a_scale), _ptr(b_codes), _ptr(b_sf),
                                             _ptr(b_scale), _ptr(offsets), e, m, n, k, _ptr(h), _ptr(status),
                                             _stream(stream))
    _check(st, "grouped_gemm_fwd_nvfp4_swiglu")
    return h


def grouped_gemm_fwd_mxfp8(a_codes, a_sf, b_codes, b_sf, offsets, n, k, *, y=None, status=None, stream=None):
    """MXFP8 forward: Y [m x n] bf16 from row-wise MXFP8 of X [m x k] and of the
    stacked weights [E*n x k]."""
    import torch

    m = a_codes.shape[0]
    e = offsets.numel() - 1
    if y is None:
        y = _empty((m, n), torch.bfloat16, a_codes.device)
    st = lib().grouped_gemm_fwd_mxfp8(_ptr(a_codes), _ptr(a_sf), _ptr(b_codes), _ptr(b_sf), _ptr(offsets), e, m, n, k,
                                      _ptr(y), _ptr(status), _stream(stream))
    _check(st, "grouped_gemm_fwd_mxfp8")
    return y


def grouped_gemm_dgrad_mxfp8(a_codes, a_sf, b_codes, b_sf, ldb, offsets, n, k, *, y=None, status=None,
                             stream=None):
    import torch

    m = a_codes.shape[0]
    e = offsets.numel() - 1
    if y is None:
        y = _empty((m, n), torch.bfloat16, a_codes.device)
    st = lib().grouped_gemm_dgrad_mxfp8(_ptr(a_codes), _ptr(a_sf), _ptr(b_codes), _ptr(b_sf), ldb, _ptr(offsets),
                                        e, m, n, k, _ptr(y), _ptr(status), _stream(stream))
    _check(st, "grouped_gemm_dgrad_mxfp8")
    return y


def grouped_gemm_wgrad_mxfp8(a_codes, a_sf, lda, b_codes, b_sf, ldb, padded_offsets, m, n, *, y=None,
                             status=None, stream=None):
    import torch

    e = padded_offsets.numel() - 1
    if y is None:
        y = _empty((e, m, n), torch.bfloat16, padded_offsets.device)
    st = lib().grouped_gemm_wgrad_mxfp8(_ptr(a_codes), _ptr(a_sf), lda, _ptr(b_codes), _ptr(b_sf), ldb,
                                        _ptr(padded_offsets), e, m, n, _ptr(y), _ptr(status), _stream(stream))
    _check(st, "grouped_gemm_wgrad_mxfp8")
    return y


# ------------------------------------------------------------------ routing --
def moe_route(topk_ids, num_experts, *, offsets=None, row_of=None, src_row=None, workspace=None, status=None,
              stream=None):
    """Group the assignments of topk_ids [tokens, top_k] (int32 expert ids) by
    expert, stably -> (offsets [E+1], row_of [tokens, top_k], src_row [tokens*top_k]),
    all int32."""
    import torch

    tokens, top_k = topk_ids.shape
    dev = topk_ids.device
    if offsets is None:
        offsets = _empty((num_experts + 1,), torch.int32, dev)
    if row_of is None:
        row_of = _empty((tokens, top_k), torch.int32, dev)
    if src_row is None:
        src_row = _empty((tokens * top_k,), torch.int32, dev)
    need = route_workspace_bytes(tokens, top_k, num_experts)
    if workspace is None:
        workspace = _empty((need,), torch.uint8, dev)
    st = lib().moe_route(_ptr(topk_ids), tokens, top_k, num_experts, _ptr(offsets), _ptr(row_of), _ptr(src_row),
                         _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status),
                         _stream(stream))
    _check(st, "moe_route")
    return offsets, row_of, src_row


def moe_route_noalloc(topk_ids, num_experts, offsets, row_of, src_row, *, status=None, stream=None):
    """moe_route into caller-owned outputs, with the library's static counters as
    the workspace: neither this call nor the library allocates memory."""
    import torch

    tokens, top_k = topk_ids.shape
    for name, t, n in (("topk_ids", topk_ids, tokens * top_k), ("offsets", offsets, num_experts + 1),
                       ("row_of", row_of, tokens * top_k), ("src_row", src_row, tokens * top_k)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous() or t.numel() != n:
            raise ValueError(f"moe_route_noalloc: {name} must be a contiguous int32 CUDA tensor of {n} elements")
        if t.device != topk_ids.device:
            raise ValueError(f"moe_route_noalloc: {name} is on {t.device}, topk_ids on {topk_ids.device}")
    st = lib().moe_route_noalloc(_ptr(topk_ids), tokens, top_k, num_experts, _ptr(offsets), _ptr(row_of),
                                 _ptr(src_row), _ptr(status), _stream(stream))
    _check(st, "moe_route_noalloc")
    return offsets, row_of, src_row


def permute_quantize_nvfp4(x, src_row, top_k, offsets, *, codes=None, sf=None, row_scale=None, status=None,
                           stream=None):
    """NVFP4 per-token quantization of the grouped rows x[src_row // top_k] ->
    (codes [tokens*top_k, k/2], sf, row_scale [tokens*top_k])."""
    import torch

    tokens, k = x.shape
    rows = tokens * top_k
    g = offsets.numel() - 1
    dev = x.device
    if codes is None:
        codes = _empty((rows, k // 2), torch.uint8, dev)
    if sf is None:
        sf = _empty((max(sf_bytes(rows, k, 16, g), 16),), torch.uint8, dev)
    if row_scale is None:
        row_scale = _empty((rows,), torch.float32, dev)
    st = lib().permute_quantize_nvfp4(_ptr(x), tokens, k, _ptr(src_row), top_k, _ptr(offsets), g, _ptr(codes),
                                      _ptr(sf), _ptr(row_scale), _ptr(status), _stream(stream))
    _check(st, "permute_quantize_nvfp4")
    return codes, sf, row_scale


def permute_quantize_mxfp8(x, src_row, top_k, offsets, *, codes=None, sf=None, status=None, stream=None):
    """MXFP8 row-wise quantization of the grouped rows x[src_row // top_k] ->
    (codes [tokens*top_k, k], sf)."""
    import torch

    tokens, k = x.shape
    rows = tokens * top_k
    g = offsets.numel() - 1
    dev = x.device
    if codes is None:
        codes = _empty((rows, k), torch.uint8, dev)
    if sf is None:
        sf = _empty((max(sf_bytes(rows, k, 32, g), 16),), torch.uint8, dev)
    st = lib().permute_quantize_mxfp8(_ptr(x), tokens, k, _ptr(src_row), top_k, _ptr(offsets), g, _ptr(codes),
                                      _ptr(sf), _ptr(status), _stream(stream))
    _check(st, "permute_quantize_mxfp8")
    return codes, sf


def moe_combine(y, row_of, weights, *, out=None, status=None, stream=None):
    """out[t] = bf16(sum_k weights[t, k] * y[row_of[t, k]]) (fp32, k in order) for
    grouped expert outputs y [rows_y, n] bf16 -> out [tokens, n] bf16."""
    import torch

    rows_y, n = y.shape
    tokens, top_k = row_of.shape
    if out is None:
        out = _empty((tokens, n), torch.bfloat16, y.device)
    st = lib().moe_combine(_ptr(y), rows_y, _ptr(row_of), _ptr(weights), tokens, top_k, n, _ptr(out), _ptr(status),
                           _stream(stream))
    _check(st, "moe_combine")
    return out


def grouped_gemm_wgrad_mxfp8_accumulate(a_codes, a_sf, lda, b_codes, b_sf, ldb, padded_offsets, m, n, dw_acc, *,
                                        status=None, stream=None):
    """dw_acc [E, m, n] (fp32) += dY_e^T H_e, the wgrad's fp32 result per expert."""
    e = padded_offsets.numel() - 1
    st = lib().grouped_gemm_wgrad_mxfp8_accumulate(_ptr(a_codes), _ptr(a_sf), lda, _ptr(b_codes), _ptr(b_sf), ldb,
                                                   _ptr(padded_offsets), e, m, n, _ptr(dw_acc), _ptr(status),
                                                   _stream(stream))
    _check(st, "grouped_gemm_wgrad_mxfp8_accumulate")
    return dw_acc


def read_device_status(status, stream=None) -> tuple[int, int]:
    """Synchronise the stream and read a device status word -> (status code, raw bits)."""
    raw = ctypes.c_int32(0)
    st = lib().fme_read_device_status(_ptr(status), _stream(stream), ctypes.byref(raw))
    return int(st), int(raw.value)
