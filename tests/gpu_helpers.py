"""Helpers for the GPU parity tests: move synthetic inputs to the device, run
both paths, and map the library's tiled formats back to logical layouts so
they can be compared with the oracle element by element."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from dense_sparse_int4_gb300 import mq


def dev_half(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.float16)).to(device)


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def dev_act(bits: np.ndarray, is_bf16: bool, device="cuda") -> torch.Tensor:
    return dev_bf16(bits, device) if is_bf16 else dev_half(bits, device)


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _records(t: torch.Tensor, n: int, size: int) -> np.ndarray:
    return t.cpu().numpy().reshape(-1)[: n * size].reshape(n, size)


def logical_wq(wpk: torch.Tensor, N: int, K: int) -> np.ndarray:
    """base records [N/128][K/128] (codes [4][128][16] bytes, then scales) -> logical packed [N, K/2]."""
    T, G = N // 128, K // 128
    a = _records(wpk, T * G, mq.WREC_BYTES)[:, : mq.WREC_SCALES].reshape(T, G, 4, 128, 16)
    return a.transpose(0, 3, 1, 2, 4).reshape(N, K // 2)


def logical_wsc(wpk: torch.Tensor, N: int, K: int) -> np.ndarray:
    """base records -> scale bits [N, K/128]."""
    T, G = N // 128, K // 128
    a = _records(wpk, T * G, mq.WREC_BYTES)[:, mq.WREC_SCALES:].copy().view(np.uint16).reshape(T, G, 128)
    return a.transpose(0, 2, 1).reshape(N, G)


def logical_rq(rpk: torch.Tensor, nnzb: int) -> np.ndarray:
    """residual records (codes [4][64][16] bytes, then scales) -> codes [nnzb, 64, 128]."""
    if nnzb == 0:
        return np.zeros((0, 64, 128), np.int8)
    a = _records(rpk, nnzb, mq.RREC_BYTES)[:, : mq.RREC_SCALES].reshape(nnzb, 4, 64, 16)
    return O.unpack_nibbles(a.transpose(0, 2, 1, 3).reshape(nnzb, 64, 64))


def logical_rsc(rpk: torch.Tensor, nnzb: int) -> np.ndarray:
    """residual records -> scale bits [nnzb, 64]."""
    if nnzb == 0:
        return np.zeros((0, 64), np.uint16)
    return _records(rpk, nnzb, mq.RREC_BYTES)[:, mq.RREC_SCALES:].copy().view(np.uint16)


def logical_xq(xq: torch.Tensor, M: int) -> np.ndarray:
    """[K/128][Mp][64] bytes -> packed [M, K/2] (token-major)."""
    a = xq.cpu().numpy()
    G, Mp, _ = a.shape
    return a.transpose(1, 0, 2).reshape(Mp, G * 64)[:M].copy()


def xq_padding(xq: torch.Tensor, M: int) -> np.ndarray:
    return xq.cpu().numpy()[:, M:, :]


def logical_xs(xs: torch.Tensor, M: int) -> np.ndarray:
    """[K/128][Mp] -> [M, K/128]."""
    return host_u16(xs)[:, :M].T.copy()


def oracle_prep_for_csr(w_bits: np.ndarray, row_ptr: np.ndarray, col_idx: np.ndarray) -> O.Prepared:
    """Oracle offline products for a given block list (any CSR, not only top-K)."""
    N, K = w_bits.shape
    qw, sw, r = O.base_quant(w_bits)
    qr, sr = O.residual_quant(r, row_ptr, col_idx)
    nb = (N // 64) * (K // 128)
    return O.Prepared(N, K, qw, sw, r, np.zeros(K), np.zeros(nb), int(col_idx.size), row_ptr, col_idx, qr, sr,
                      O.sel_of(row_ptr, col_idx, N, K))


def packed_from_csr(w: torch.Tensor, row_ptr: np.ndarray, col_idx: np.ndarray) -> mq.PackedLinear:
    dev = w.device
    rp = torch.from_numpy(row_ptr.astype(np.int32)).to(dev)
    ci = torch.from_numpy(col_idx.astype(np.int32)).to(dev) if col_idx.size else torch.zeros(0, dtype=torch.int32, device=dev)
    return mq.pack_weights(w, rp, ci)


def check_close(y_gpu: np.ndarray, y: np.ndarray, a: np.ndarray, rel: float = 1e-5):
    """|y_gpu - y| <= rel * (sum of |terms|) element by element."""
    err = np.abs(y_gpu.astype(np.float64) - y)
    bound = rel * a
    bad = err > bound
    assert not bad.any(), f"{bad.sum()} of {bad.size} over tolerance; worst err {err[bad].max():.3e} bound {bound[bad].min():.3e}"
    return float((err / np.maximum(np.abs(y).max(), 1e-300)).max())


def bf16_ulp(bits: np.ndarray) -> np.ndarray:
    v = O.bf16_to_double(bits)
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def check_bf16(y_bits: np.ndarray, y: np.ndarray, a: np.ndarray, rel: float = 1e-5):
    """bf16 output within 1 ulp of bf16_RNE(y); where the fp32 epilogue's own
    bound exceeds that ulp (cancellation), within that bound plus half an ulp."""
    yb = O.double_to_bf16(y)
    gv = O.bf16_to_double(y_bits)
    rv = O.bf16_to_double(yb)
    ok = (np.abs(gv - rv) <= bf16_ulp(yb)) | (np.abs(gv - y) <= rel * a + bf16_ulp(y_bits) / 2)
    assert ok.all(), f"{(~ok).sum()} bf16 outputs off by more than 1 ulp"
    return float(np.mean(y_bits == yb))
