"""Seeded synthetic inputs for the W4A4 + sparse-residual linear.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic, so both the CUDA path and the oracle can take their
inputs from it.  Values follow the workloads the MosaicQuant summary
evaluates (LLaMA3 / Qwen3 linear layers, "Risultati Sperimentali"), on
random-init weights since no trained checkpoint is available:

* activations X: N(0, 1), a fixed set of outlier input channels scaled x50
  (0.1 % of K, at least 4; the channels are drawn from the seed);
* calibration rows Xcal (256 rows) drawn like X, same outlier channels;
* weights W^: N(0, 0.02);
* optional "concentrated" placement: in a seeded 2 % of the 64x128 blocks,
  every one of the 64 rows gets one entry set to +-1.0 (50 sigma).

All draws are float32 from numpy's PCG64, rounded to fp16 (or bf16) with
round-to-nearest-even, returned as uint16 bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# stream ids under one seed: independent PCG64 streams per input kind
_X, _XCAL, _W, _OUT, _INJ = 1, 2, 3, 4, 5


def _rng(seed: int, stream: int, sub: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), stream, int(sub)])))


def f32_to_f16_bits(a: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.float16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def to_bits(a: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(a) if dtype == "bf16" else f32_to_f16_bits(a)


def n_outliers(K: int, frac: float = 0.001, minimum: int = 4) -> int:
    return max(minimum, int(K * frac))


def outlier_channels(K: int, count: int, seed: int) -> np.ndarray:
    return np.sort(_rng(seed, _OUT, K).choice(K, size=count, replace=False))


def activations(M: int, K: int, seed: int, count: int, dtype: str = "f16", scale: float = 50.0,
                sub: int = 0) -> np.ndarray:
    x = _rng(seed, _X, sub).standard_normal((M, K), dtype=np.float32)
    x[:, outlier_channels(K, count, seed)] *= scale
    return to_bits(x, dtype)


def calibration(K: int, seed: int, count: int, C: int = 256, dtype: str = "f16",
                scale: float = 50.0) -> np.ndarray:
    x = _rng(seed, _XCAL).standard_normal((C, K), dtype=np.float32)
    x[:, outlier_channels(K, count, seed)] *= scale
    return to_bits(x, dtype)


def weights(N: int, K: int, seed: int, sigma: float = 0.02, sub: int = 0) -> np.ndarray:
    w = _rng(seed, _W, sub).standard_normal((N, K), dtype=np.float32) * np.float32(sigma)
    return f32_to_f16_bits(w)


def inject_concentrated(w_bits: np.ndarray, seed: int, frac: float = 0.02, value: float = 1.0) -> np.ndarray:
    """Copy of W^ where a seeded `frac` of 64x128 blocks get one +-value entry per row."""
    N, K = w_bits.shape
    nbr, G = N // 64, K // 128
    rng = _rng(seed, _INJ)
    blocks = rng.choice(nbr * G, size=max(1, int(round(frac * nbr * G))), replace=False)
    w = w_bits.copy()
    for b in blocks:
        br, g = divmod(int(b), G)
        cols = rng.integers(0, 128, size=64)
        signs = rng.choice(np.array([-1.0, 1.0], np.float32), size=64)
        vals = f32_to_f16_bits(signs * np.float32(value))
        w[br * 64 + np.arange(64), g * 128 + cols] = vals
    return w


def device_weights(N: int, K: int, seed: int, device, sigma: float = 0.02):
    """N(0, sigma) fp16 weights drawn on the device with torch's seeded Philox
    generator: for timing-only workloads too large to draw on the host."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return (torch.randn((N, K), generator=g, device=device, dtype=torch.float32) * sigma).to(torch.float16)


def inject_concentrated_device(w, seed: int, frac: float = 0.02, value: float = 1.0):
    """In place on a device [N, K] fp16 tensor: a seeded `frac` of the 64x128
    blocks get one +-value entry per row (the device counterpart of
    inject_concentrated, drawn with torch's seeded generator: for timing
    workloads too large to draw on the host)."""
    import torch
    N, K = w.shape
    nbr, G = N // 64, K // 128
    g = torch.Generator(device=w.device)
    g.manual_seed(int(seed) + 7919)
    nblk = max(1, int(round(frac * nbr * G)))
    blocks = torch.randperm(nbr * G, generator=g, device=w.device)[:nblk]
    br, gg = blocks // G, blocks % G
    rows = br[:, None] * 64 + torch.arange(64, device=w.device)[None, :]
    cols = gg[:, None] * 128 + torch.randint(0, 128, (nblk, 64), generator=g, device=w.device)
    signs = torch.randint(0, 2, (nblk, 64), generator=g, device=w.device).to(torch.float16) * 2 - 1
    w[rows.reshape(-1), cols.reshape(-1)] = (signs * value).reshape(-1)
    return w


# --------------------------------------------------------------------------
# The workloads
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Linear:
    name: str
    K: int  # input features
    N: int  # output features


LLAMA3_8B = (
    Linear("q", 4096, 4096), Linear("k", 4096, 1024), Linear("v", 4096, 1024),
    Linear("o", 4096, 4096), Linear("gate", 4096, 14336), Linear("up", 4096, 14336),
    Linear("down", 14336, 4096),
)
QWEN3_32B = (
    Linear("q", 5120, 8192), Linear("k", 5120, 1024), Linear("v", 5120, 1024),
    Linear("o", 8192, 5120), Linear("gate", 5120, 25600), Linear("up", 5120, 25600),
    Linear("down", 25600, 5120),
)


@dataclass(frozen=True)
class Workload:
    name: str
    linears: tuple
    Ms: tuple
    budgets: tuple
    x_dtype: str = "f16"
    outliers: int | None = None  # fixed outlier count, else 0.1 % of K
    seed: int = 0
    placements: tuple = ("uniform",)
    layers: int = 1
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "single-512": Workload("single-512", (Linear("single", 512, 512),), (4,), (0.10,), outliers=4),
    "llama3-8b-decode": Workload("llama3-8b-decode", LLAMA3_8B, (4, 8, 16, 32), (0.10,)),
    "prefill-2048x4096x14336": Workload("prefill-2048x4096x14336", (Linear("gate", 4096, 14336),),
                                        (2048,), (0.10, 0.0), x_dtype="bf16", outliers=8),
    "qwen3-32b": Workload("qwen3-32b", QWEN3_32B, (4, 32, 512), (0.0, 0.05, 0.10, 0.20),
                          placements=("concentrated", "uniform")),
    "llama3-8b-stack32": Workload("llama3-8b-stack32", LLAMA3_8B, (32,), (0.10,), layers=32),
}
