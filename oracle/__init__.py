"""The oracle: a plain, slow, single-threaded CPU statement of the MosaicQuant
W4A4 + block-sparse 4-bit residual linear, in float64 / int64.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library (``dense_sparse_int4_gb300``) and never imports it.

The arithmetic lives in ``mq_oracle.c`` (compiled with gcc by ``build()``);
this module only marshals numpy arrays.  Citations refer to the page
"MosaicQuant: Inlier-Outlier Disaggregation for Unified 4-Bit LLM
Quantization" (technical summary), sections Metodologia 1 (W^ ~= Q(W^) + R),
Metodologia 2 (block budget, Hessian-guided Delta-score, top-K) and
Metodologia 3 (ZipperEngine: reduce-add of the dense and sparse products).

Every function here has a pin in ``tests/test_oracle_pins.py`` (values and
properties fixed by the definitions, brute force, closed forms, library
routines); see the header of that file for which pin covers which step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

GROUP = 128  # inputs per scale group / residual block column
BROWS = 64  # output rows per residual block
_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libmq_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle (plain gcc, no contraction of a*b+c)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-shared", "-fPIC",
             _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(_LIB_PATH)
        i64, dbl, i32 = ctypes.c_int64, ctypes.c_double, ctypes.c_int
        P = ctypes.c_void_p
        sigs = {
            "mqo_half_to_double_n": [P, i64, P],
            "mqo_bf16_to_double_n": [P, i64, P],
            "mqo_double_to_half_n": [P, i64, P],
            "mqo_double_to_bf16_n": [P, i64, P],
            "mqo_scale_from_amax_n": [P, i64, P],
            "mqo_quantize_group": [P, i32, P, P],
            "mqo_pack_nibbles": [P, i64, P],
            "mqo_unpack_nibbles": [P, i64, P],
            "mqo_quantize_act": [P, i32, i64, i64, P, P],
            "mqo_base_quant": [P, i64, i64, P, P, P],
            "mqo_hessian_diag": [P, i32, i64, i64, P],
            "mqo_delta_scores": [P, P, i64, i64, P],
            "mqo_num_selected": [i64, i64, dbl],
            "mqo_select_topk": [P, i64, i64, i64, P, P],
            "mqo_residual_quant": [P, i64, i64, P, P, P, P],
            "mqo_group_dots": [P, P, i64, i64, i64, P],
            "mqo_residual_dots": [P, P, P, i64, i64, i64, P],
            "mqo_linear_entries": [P, P, P, P, P, P, P, i64, i64, i64, P, P, i64, P, P],
        }
        for name, args in sigs.items():
            fn = getattr(_lib, name)
            fn.argtypes = args
            fn.restype = None
        _lib.mqo_num_selected.restype = i64
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# Formats
# --------------------------------------------------------------------------

def half_to_double(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, np.float64)
    _L().mqo_half_to_double_n(_p(b), b.size, _p(out))
    return out


def bf16_to_double(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, np.float64)
    _L().mqo_bf16_to_double_n(_p(b), b.size, _p(out))
    return out


def double_to_half(v) -> np.ndarray:
    a = _c(v, np.float64)
    out = np.empty(a.shape, np.uint16)
    _L().mqo_double_to_half_n(_p(a), a.size, _p(out))
    return out


def double_to_bf16(v) -> np.ndarray:
    a = _c(v, np.float64)
    out = np.empty(a.shape, np.uint16)
    _L().mqo_double_to_bf16_n(_p(a), a.size, _p(out))
    return out


def scale_from_amax(amax) -> np.ndarray:
    a = _c(amax, np.float64)
    out = np.empty(a.shape, np.uint16)
    _L().mqo_scale_from_amax_n(_p(a), a.size, _p(out))
    return out


def to_double(bits, is_bf16: bool) -> np.ndarray:
    return bf16_to_double(bits) if is_bf16 else half_to_double(bits)


# --------------------------------------------------------------------------
# Quantizer Qz and nibble packing  [Metodologia 1]
# --------------------------------------------------------------------------

def quantize_group(v) -> tuple[int, np.ndarray]:
    """Qz over one vector: (scale fp16 bits, int8 codes)."""
    a = _c(v, np.float64)
    q = np.empty(a.shape, np.int8)
    s = np.zeros(1, np.uint16)
    _L().mqo_quantize_group(_p(a), a.size, _p(s), _p(q))
    return int(s[0]), q


def pack_nibbles(q) -> np.ndarray:
    """[..., K] int8 codes -> [..., K/2] bytes (even index in the low nibble)."""
    a = _c(q, np.int8)
    out = np.empty(a.shape[:-1] + (a.shape[-1] // 2,), np.uint8)
    _L().mqo_pack_nibbles(_p(a), a.size, _p(out))
    return out


def unpack_nibbles(p) -> np.ndarray:
    a = _c(p, np.uint8)
    out = np.empty(a.shape[:-1] + (a.shape[-1] * 2,), np.int8)
    _L().mqo_unpack_nibbles(_p(a), out.size, _p(out))
    return out


def quantize_act(x_bits, is_bf16: bool) -> tuple[np.ndarray, np.ndarray]:
    """Per token, per 128-input group: codes [M, K] int8, scales [M, K/128] fp16 bits."""
    x = _c(x_bits, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.int8)
    s = np.empty((M, K // GROUP), np.uint16)
    _L().mqo_quantize_act(_p(x), int(is_bf16), M, K, _p(q), _p(s))
    return q, s


# --------------------------------------------------------------------------
# Offline: base, residual, Delta-score, top-K  [Metodologia 1, 2]
# --------------------------------------------------------------------------

def base_quant(w_bits) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Q(W^) and R = W^ - Q(W^): codes [N, K], scales [N, K/128], R [N, K] float64."""
    w = _c(w_bits, np.uint16)
    N, K = w.shape
    qw = np.empty((N, K), np.int8)
    sw = np.empty((N, K // GROUP), np.uint16)
    r = np.empty((N, K), np.float64)
    _L().mqo_base_quant(_p(w), N, K, _p(qw), _p(sw), _p(r))
    return qw, sw, r


def hessian_diag(xcal_bits, is_bf16: bool) -> np.ndarray:
    x = _c(xcal_bits, np.uint16)
    C, K = x.shape
    h = np.empty(K, np.float64)
    _L().mqo_hessian_diag(_p(x), int(is_bf16), C, K, _p(h))
    return h


def delta_scores(r, h) -> np.ndarray:
    """Delta_b for every block b = br*(K/128) + g."""
    r = _c(r, np.float64)
    h = _c(h, np.float64)
    N, K = r.shape
    d = np.empty((N // BROWS) * (K // GROUP), np.float64)
    _L().mqo_delta_scores(_p(r), _p(h), N, K, _p(d))
    return d


def num_selected(N: int, K: int, budget: float) -> int:
    return int(_L().mqo_num_selected(N, K, float(budget)))


def select_topk(delta, N: int, K: int, ksel: int) -> tuple[np.ndarray, np.ndarray]:
    d = _c(delta, np.float64)
    row_ptr = np.empty(N // BROWS + 1, np.int32)
    col_idx = np.empty(max(ksel, 1), np.int32)
    _L().mqo_select_topk(_p(d), N, K, ksel, _p(row_ptr), _p(col_idx))
    return row_ptr, col_idx[:ksel].copy()


def residual_quant(r, row_ptr, col_idx) -> tuple[np.ndarray, np.ndarray]:
    """Codes [nnzb, 64, 128] and scales [nnzb, 64] of the selected blocks, CSR order."""
    r = _c(r, np.float64)
    rp = _c(row_ptr, np.int32)
    ci = _c(col_idx, np.int32)
    N, K = r.shape
    nnzb = ci.size
    qr = np.zeros((max(nnzb, 1), BROWS, GROUP), np.int8)
    sr = np.zeros((max(nnzb, 1), BROWS), np.uint16)
    _L().mqo_residual_quant(_p(r), N, K, _p(rp), _p(ci if nnzb else np.zeros(1, np.int32)), _p(qr), _p(sr))
    return qr[:nnzb].copy(), sr[:nnzb].copy()


def csr_block_rows(row_ptr) -> np.ndarray:
    """Block row of every CSR entry."""
    rp = np.asarray(row_ptr, np.int64)
    return np.repeat(np.arange(rp.size - 1), np.diff(rp))


def sel_of(row_ptr, col_idx, N: int, K: int) -> np.ndarray:
    """Map block (br, g) -> CSR entry index or -1."""
    G = K // GROUP
    out = -np.ones((N // BROWS) * G, np.int64)
    brs = csr_block_rows(row_ptr)
    for i, (br, g) in enumerate(zip(brs, np.asarray(col_idx))):
        out[br * G + int(g)] = i
    return out


# --------------------------------------------------------------------------
# The linear  [Metodologia 3]
# --------------------------------------------------------------------------

def group_dots(qx, qw) -> np.ndarray:
    qx = _c(qx, np.int8)
    qw = _c(qw, np.int8)
    M, K = qx.shape
    N = qw.shape[0]
    d = np.empty((M, N, K // GROUP), np.int64)
    _L().mqo_group_dots(_p(qx), _p(qw), M, N, K, _p(d))
    return d


def residual_dots(qx, qr, col_idx) -> np.ndarray:
    qx = _c(qx, np.int8)
    qr = _c(qr, np.int8)
    ci = _c(col_idx, np.int32)
    M, K = qx.shape
    nnzb = ci.size
    d = np.empty((M, nnzb, BROWS), np.int64)
    if nnzb:
        _L().mqo_residual_dots(_p(qx), _p(qr), _p(ci), M, K, nnzb, _p(d))
    return d


@dataclass
class Prepared:
    """Offline products for one weight matrix (the oracle's own, logical layout)."""
    N: int
    K: int
    qw: np.ndarray  # [N, K] int8
    sw: np.ndarray  # [N, K/128] fp16 bits
    r: np.ndarray  # [N, K] float64 residual
    h: np.ndarray  # [K] diag-Hessian
    delta: np.ndarray  # [nb]
    ksel: int
    row_ptr: np.ndarray
    col_idx: np.ndarray
    qr: np.ndarray  # [nnzb, 64, 128]
    sr: np.ndarray  # [nnzb, 64]
    sel: np.ndarray  # [nb] block -> CSR entry or -1


def prepare(w_bits, xcal_bits, xcal_is_bf16: bool, budget: float) -> Prepared:
    """The offline chain: Q(W^), R, h, Delta, top-K, residual codes."""
    w = _c(w_bits, np.uint16)
    N, K = w.shape
    qw, sw, r = base_quant(w)
    h = hessian_diag(xcal_bits, xcal_is_bf16)
    d = delta_scores(r, h)
    ksel = num_selected(N, K, budget)
    rp, ci = select_topk(d, N, K, ksel)
    qr, sr = residual_quant(r, rp, ci)
    return Prepared(N, K, qw, sw, r, h, d, ksel, rp, ci, qr, sr, sel_of(rp, ci, N, K))


def linear_entries(qx, sx, prep: Prepared, ms, ns) -> tuple[np.ndarray, np.ndarray]:
    """y[m, n] (float64) and the absolute-term sum for the listed (m, n) pairs."""
    qx = _c(qx, np.int8)
    sx = _c(sx, np.uint16)
    ms = _c(ms, np.int64)
    ns = _c(ns, np.int64)
    M, K = qx.shape
    cnt = ms.size
    y = np.empty(cnt, np.float64)
    a = np.empty(cnt, np.float64)
    qr = prep.qr if prep.qr.size else np.zeros((1, BROWS, GROUP), np.int8)
    sr = prep.sr if prep.sr.size else np.zeros((1, BROWS), np.uint16)
    _L().mqo_linear_entries(_p(qx), _p(sx), _p(prep.qw), _p(prep.sw), _p(_c(qr, np.int8)),
                            _p(_c(sr, np.uint16)), _p(prep.sel), M, prep.N, K, _p(ms), _p(ns), cnt,
                            _p(y), _p(a))
    return y, a


def linear(qx, sx, prep: Prepared) -> tuple[np.ndarray, np.ndarray]:
    """Full output y [M, N] float64 and absolute-term sums."""
    M = qx.shape[0]
    mm, nn = np.meshgrid(np.arange(M), np.arange(prep.N), indexing="ij")
    y, a = linear_entries(qx, sx, prep, mm.ravel(), nn.ravel())
    return y.reshape(M, prep.N), a.reshape(M, prep.N)
