"""Thin Python binding of the C ABI in include/mq.h (ctypes).

Argument marshalling only: buffers are torch CUDA tensors (PyTorch supplies
device memory and streams), every step runs in the library's kernels.  There
is no fallback: if the shared library is missing or the GPU is not sm_103a
the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libmq.so")

MQ_OK, MQ_ERR_INVALID_ARG, MQ_ERR_ALIGNMENT, MQ_ERR_UNSUPPORTED_DEVICE, MQ_ERR_CUDA, MQ_ERR_TIMEOUT, MQ_ERR_WORKSPACE = range(7)
MQ_F16, MQ_BF16, MQ_F32 = 0, 1, 2
WREC_BYTES, WREC_SCALES = 8448, 8192  # base record: 128x128 codes, then 128 fp16 scales
RREC_BYTES, RREC_SCALES = 4224, 4096  # residual record: 64x128 codes, then 64 fp16 scales

EXPORTS = (
    "mq_quantize_act", "mq_num_selected", "mq_select_workspace_bytes", "mq_select_blocks",
    "mq_pack_weights", "mq_gemm_workspace_bytes", "mq_gemm_workspace_init", "mq_w4a4_residual_gemm",
    "mq_w4a4_residual_gemm_noalloc", "mq_gemm_plan", "mq_linear_workspace_bytes", "mq_w4a4_residual_linear",
    "mq_debug_group_dots", "mq_check_device_error", "mq_set_wait_timeout_ns", "mq_debug_wait_timeout",
    "mq_status_string", "mq_last_error", "mq_version",
)


class MQError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: status {status}: {detail}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, i64, i32, dbl, sz, u64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                                     ctypes.c_size_t, ctypes.c_uint64)
        sig = {
            "mq_quantize_act": (i32, [P, i32, i64, i64, i64, P, P, P]),
            "mq_num_selected": (i64, [i64, i64, dbl]),
            "mq_select_workspace_bytes": (sz, [i64, i64]),
            "mq_select_blocks": (i32, [P, i64, i64, P, i32, i64, dbl, P, P, P, P, P, sz, P]),
            "mq_pack_weights": (i32, [P, i64, i64, P, P, i64, P, P, P]),
            "mq_gemm_workspace_bytes": (sz, [i64, i64, i64]),
            "mq_gemm_workspace_init": (i32, [P, sz, P]),
            "mq_w4a4_residual_gemm": (i32, [P, P, i64, P, i64, i64, P, P, i64, P, P, i32, P, sz, P]),
            "mq_w4a4_residual_gemm_noalloc": (i32, [P, P, i64, P, i64, i64, P, P, i64, P, P, i32, P]),
            "mq_debug_group_dots": (i32, [P, P, i64, P, i64, i64, P, P, i64, P, P, P, P, sz, P]),
            "mq_gemm_plan": (i32, [i64, i64, i64, P]),
            "mq_linear_workspace_bytes": (sz, [i64, i64, i32, P]),
            "mq_w4a4_residual_linear": (i32, [P, i32, i64, i64, i64, i32, P, i32, P, P, P, sz, P]),
            "mq_check_device_error": (i32, [P]),
            "mq_set_wait_timeout_ns": (None, [u64]),
            "mq_debug_wait_timeout": (i32, [P]),
            "mq_status_string": (ctypes.c_char_p, [i32]),
            "mq_last_error": (ctypes.c_char_p, []),
            "mq_version": (ctypes.c_char_p, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int, where: str):
    if status != MQ_OK:
        raise MQError(status, where, lib().mq_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(dt) -> int:
    if dt == torch.float16:
        return MQ_F16
    if dt == torch.bfloat16:
        return MQ_BF16
    if dt == torch.float32:
        return MQ_F32
    raise TypeError(f"unsupported dtype {dt}")


def padded_tokens(M: int) -> int:
    return (M + 7) // 8 * 8


# ---------------------------------------------------------------------------
# activation quantizer
# ---------------------------------------------------------------------------

def quantize_act(x: torch.Tensor, xq: torch.Tensor | None = None, xs: torch.Tensor | None = None, stream=None):
    """x [M, K] fp16/bf16 (row stride x.stride(0)) -> xq [K/128, Mp, 64] uint8, xs [K/128, Mp] fp16."""
    M, K = x.shape
    if x.stride(1) != 1:
        raise ValueError("x must have unit stride along K")
    if xq is None:
        xq = torch.empty((K // 128, padded_tokens(M), 64), dtype=torch.uint8, device=x.device)
    if xs is None:
        xs = torch.empty((K // 128, padded_tokens(M)), dtype=torch.float16, device=x.device)
    _check(lib().mq_quantize_act(_ptr(x), _dtype_code(x.dtype), M, K, x.stride(0), _ptr(xq), _ptr(xs),
                                 _stream(stream)), "mq_quantize_act")
    return xq, xs


# ---------------------------------------------------------------------------
# offline: selection and packing
# ---------------------------------------------------------------------------

def num_selected(N: int, K: int, budget: float) -> int:
    return int(lib().mq_num_selected(N, K, float(budget)))


def select_blocks(w: torch.Tensor, xcal: torch.Tensor, budget: float, want_h: bool = False,
                  want_delta: bool = False, stream=None):
    """w [N, K] fp16, xcal [C, K] fp16/bf16 -> (row_ptr, col_idx, h or None, delta or None)."""
    N, K = w.shape
    C = xcal.shape[0]
    dev = w.device
    ksel = num_selected(N, K, budget)
    row_ptr = torch.empty(N // 64 + 1, dtype=torch.int32, device=dev)
    col_idx = torch.empty(max(ksel, 1), dtype=torch.int32, device=dev)
    h = torch.empty(K, dtype=torch.float64, device=dev) if want_h else None
    delta = torch.empty((N // 64) * (K // 128), dtype=torch.float64, device=dev) if want_delta else None
    wsb = int(lib().mq_select_workspace_bytes(N, K))
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    _check(lib().mq_select_blocks(_ptr(w), N, K, _ptr(xcal), _dtype_code(xcal.dtype), C, float(budget),
                                  _ptr(row_ptr), _ptr(col_idx), _ptr(h), _ptr(delta), _ptr(ws), wsb,
                                  _stream(stream)), "mq_select_blocks")
    return row_ptr, col_idx[:ksel], h, delta


@dataclass
class PackedLinear:
    """A weight matrix in the GEMM's packed formats (see mq_pack_weights)."""
    N: int
    K: int
    nnzb: int
    wpk: torch.Tensor  # uint8 [(N/128)*(K/128), WREC_BYTES] base records
    row_ptr: torch.Tensor  # int32 [N/64 + 1]
    col_idx: torch.Tensor  # int32 [nnzb]
    rpk: torch.Tensor  # uint8 [nnzb, RREC_BYTES] residual records in CSR order

    def weight_bytes(self) -> int:
        """Bytes the GEMM must stream per call: base codes + scales + residual + CSR."""
        return (self.N * self.K // 2 + self.N * (self.K // 128) * 2 + self.nnzb * (4096 + 128 + 4)
                + 4 * (self.N // 64 + 1))

    def clone(self) -> "PackedLinear":
        return PackedLinear(self.N, self.K, self.nnzb, self.wpk.clone(), self.row_ptr.clone(), self.col_idx.clone(),
                            self.rpk.clone())


def pack_weights(w: torch.Tensor, row_ptr: torch.Tensor, col_idx: torch.Tensor, stream=None) -> PackedLinear:
    N, K = w.shape
    dev = w.device
    nnzb = int(col_idx.numel())
    wpk = torch.empty(((N // 128) * (K // 128), WREC_BYTES), dtype=torch.uint8, device=dev)
    rpk = torch.empty((max(nnzb, 1), RREC_BYTES), dtype=torch.uint8, device=dev)
    ci = col_idx if nnzb else torch.zeros(1, dtype=torch.int32, device=dev)
    _check(lib().mq_pack_weights(_ptr(w), N, K, _ptr(row_ptr), _ptr(ci), nnzb, _ptr(wpk), _ptr(rpk),
                                 _stream(stream)), "mq_pack_weights")
    return PackedLinear(N, K, nnzb, wpk, row_ptr, ci, rpk)


def prepare_linear(w: torch.Tensor, xcal: torch.Tensor, budget: float, stream=None) -> PackedLinear:
    row_ptr, col_idx, _, _ = select_blocks(w, xcal, budget, stream=stream)
    return pack_weights(w, row_ptr, col_idx, stream=stream)


# ---------------------------------------------------------------------------
# the fused GEMM
# ---------------------------------------------------------------------------

_ws_cache: dict = {}


def gemm_workspace(M: int, N: int, K: int, device) -> tuple[torch.Tensor | None, int]:
    """A zeroed workspace big enough for (M, N, K), cached per device and size."""
    nbytes = int(lib().mq_gemm_workspace_bytes(M, N, K))
    if nbytes == 0:
        return None, 0
    key = (torch.device(device).index, nbytes)
    ws = _ws_cache.get(key)
    if ws is None:
        ws = torch.zeros(nbytes + 256, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws, nbytes


def gemm(xq: torch.Tensor, xs: torch.Tensor, M: int, pl: PackedLinear, out: torch.Tensor | None = None,
         out_dtype=torch.bfloat16, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y [M, N] = Q(X) (Q(W) + R)^T with the fused kernel."""
    dev = xq.device
    if out is None:
        out = torch.empty((M, pl.N), dtype=out_dtype, device=dev)
    if ws is None:
        ws, wsb = gemm_workspace(M, pl.N, pl.K, dev)
    else:
        wsb = ws.numel()
    nz = pl.nnzb > 0
    _check(lib().mq_w4a4_residual_gemm(_ptr(xq), _ptr(xs), M, _ptr(pl.wpk), pl.N, pl.K, _ptr(pl.row_ptr),
                                       _ptr(pl.col_idx) if nz else None, pl.nnzb, _ptr(pl.rpk) if nz else None,
                                       _ptr(out), _dtype_code(out.dtype), _ptr(ws), wsb, _stream(stream)),
           "mq_w4a4_residual_gemm")
    return out


class Matrix(ctypes.Structure):
    """mq_matrix: one weight matrix of a fused (grouped) linear call."""
    _fields_ = [("wpk", ctypes.c_void_p), ("N", ctypes.c_int64), ("row_ptr", ctypes.c_void_p),
                ("col_idx", ctypes.c_void_p), ("nnzb", ctypes.c_int64), ("rpk", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("ldy", ctypes.c_int64)]


def linear_workspace(M: int, K: int, Ns, device) -> tuple[torch.Tensor, int]:
    """A zeroed workspace for mq_w4a4_residual_linear over matrices of N in Ns, cached per device and size."""
    arr = (ctypes.c_int64 * len(Ns))(*Ns)
    nbytes = int(lib().mq_linear_workspace_bytes(M, K, len(Ns), ctypes.cast(arr, ctypes.c_void_p)))
    if nbytes == 0:
        raise ValueError(f"no fused linear for M={M} K={K} N={list(Ns)}")
    key = (torch.device(device).index, nbytes)
    ws = _ws_cache.get(key)
    if ws is None:
        ws = torch.zeros(nbytes + 256, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws, nbytes


def fused_linear(x: torch.Tensor, pls, outs=None, out_dtype=torch.bfloat16, ws: torch.Tensor | None = None,
                 xq: torch.Tensor | None = None, xs: torch.Tensor | None = None, stream=None):
    """Y_i = Q(x) (Q(W_i) + R_i)^T for the packed matrices pls (1..4, sharing x), quantizer included.
    outs: optional list of [M, N_i] tensors (views with row stride >= N_i are allowed)."""
    M, K = x.shape
    if x.stride(1) != 1:
        raise ValueError("x must have unit stride along K")
    dev = x.device
    if outs is None:
        outs = [torch.empty((M, pl.N), dtype=out_dtype, device=dev) for pl in pls]
    mats = (Matrix * len(pls))()
    for i, (pl, y) in enumerate(zip(pls, outs)):
        nz = pl.nnzb > 0
        mats[i] = Matrix(pl.wpk.data_ptr(), pl.N, pl.row_ptr.data_ptr(), pl.col_idx.data_ptr() if nz else None, pl.nnzb,
                         pl.rpk.data_ptr() if nz else None, y.data_ptr(), y.stride(0))
    if ws is None:
        ws, wsb = linear_workspace(M, K, [pl.N for pl in pls], dev)
    else:
        wsb = ws.numel()
    _check(lib().mq_w4a4_residual_linear(_ptr(x), _dtype_code(x.dtype), M, K, x.stride(0), len(pls),
                                         ctypes.cast(mats, ctypes.c_void_p), _dtype_code(outs[0].dtype), _ptr(xq),
                                         _ptr(xs), _ptr(ws), wsb, _stream(stream)), "mq_w4a4_residual_linear")
    return outs


def gemm_plan(M: int, N: int, K: int) -> dict:
    """The kernel the GEMM entry points run for (M, N, K) on the current device."""
    info = (ctypes.c_int32 * 5)()
    _check(lib().mq_gemm_plan(M, N, K, ctypes.cast(info, ctypes.c_void_p)), "mq_gemm_plan")
    return {"decode": info[0] in (3, 4, 5),
            "variant": {0: "general", 3: "tensor-memory", 4: "warp-mma", 5: "column", 6: "image"}[info[0]],
            "tokens_per_tile": info[1], "cluster": info[2], "clusters": info[3], "stages": info[4]}


def debug_group_dots(xq, xs, M: int, pl: PackedLinear, stream=None):
    dev = xq.device
    G = pl.K // 128
    dw = torch.empty((M, pl.N, G), dtype=torch.int32, device=dev)
    dr = torch.empty((M, max(pl.nnzb, 1), 64), dtype=torch.int32, device=dev)
    ws, wsb = gemm_workspace(M, pl.N, pl.K, dev)
    nz = pl.nnzb > 0
    _check(lib().mq_debug_group_dots(_ptr(xq), _ptr(xs), M, _ptr(pl.wpk), pl.N, pl.K, _ptr(pl.row_ptr),
                                     _ptr(pl.col_idx) if nz else None, pl.nnzb, _ptr(pl.rpk) if nz else None,
                                     _ptr(dw), _ptr(dr) if nz else None, _ptr(ws), wsb, _stream(stream)),
           "mq_debug_group_dots")
    return dw, dr[:, : pl.nnzb]


def linear(x: torch.Tensor, pl: PackedLinear, out_dtype=torch.bfloat16, stream=None) -> torch.Tensor:
    """Quantize x and run the fused GEMM (two launches)."""
    xq, xs = quantize_act(x, stream=stream)
    return gemm(xq, xs, x.shape[0], pl, out_dtype=out_dtype, stream=stream)


def check_device_error(stream=None):
    _check(lib().mq_check_device_error(_stream(stream)), "device")


def set_wait_timeout_ns(ns: int):
    lib().mq_set_wait_timeout_ns(int(ns))


def debug_wait_timeout(stream=None):
    _check(lib().mq_debug_wait_timeout(_stream(stream)), "mq_debug_wait_timeout")


def version() -> str:
    return lib().mq_version().decode()
