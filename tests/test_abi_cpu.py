"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol include/mq.h declares, sizes its workspaces, counts selected
blocks like the oracle, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

import oracle as O
from dense_sparse_int4_gb300 import build as B
from dense_sparse_int4_gb300 import mq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    B.build()
    return mq.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "mq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mq_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert len(names) >= 14
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(mq.EXPORTS)


def test_version_and_status_strings(L):
    assert "sm_103a" in mq.version()
    for s in range(7):
        assert L.mq_status_string(s)


def test_num_selected_matches_oracle(L, golden_dir):
    for line in open(os.path.join(golden_dir, "num_selected.txt")):
        if line.startswith("#") or not line.strip():
            continue
        N, K, b, want = line.split()
        assert L.mq_num_selected(int(N), int(K), float(b)) == int(want)
        assert O.num_selected(int(N), int(K), float(b)) == int(want)


def test_workspace_sizes(L):
    assert L.mq_select_workspace_bytes(4096, 4096) >= 2048 * 8 + 4096 * 8 + 2048
    # stream-K: two fp32 pieces of a 128 x TN tile per persistent CTA + one counter per tile
    ws32 = L.mq_gemm_workspace_bytes(32, 4096, 4096)
    assert ws32 >= 64 * 2 * 128 * 32 * 4 + 32 * 4  # at least 64 CTAs (4+ units of 2 groups each)
    assert L.mq_gemm_workspace_bytes(2048, 14336, 4096) >= 152 * 2 * 128 * 64 * 4  # 64-token tiles above 32 tokens
    # from 128 tokens: the image form's operand images (E4M3 weights, the densest residual, activations)
    assert L.mq_gemm_workspace_bytes(2048, 14336, 4096) >= 2 * 14336 * 4096 + 2048 * 4096
    assert L.mq_gemm_workspace_bytes(127, 14336, 4096) < 14336 * 4096
    # ... exactly: the counter prefix, 152 CTAs' two stream-K pieces of 128 x 128 fp32, the weight images
    # (16 KiB per tile and group), the densest residual's images (8 KiB per block), the activation images
    # (128 bytes per token and group, tokens padded to 128) and their fp32 scales
    M, N, K = 2048, 14336, 4096
    G, Mt = K // 128, (M + 127) // 128 * 128
    want = 16384 + 152 * 2 * 128 * 128 * 4 + (N // 128) * G * 16384 + (N // 64) * G * 8192 + G * Mt * 128 + G * Mt * 4
    assert L.mq_gemm_workspace_bytes(M, N, K) == want
    assert L.mq_gemm_workspace_bytes(4, 512, 512) > 0
    assert L.mq_gemm_workspace_bytes(4, 100, 4096) == 0  # invalid N


def test_argument_validation_before_device(L):
    P = ctypes.c_void_p
    bad = P(0)
    assert L.mq_quantize_act(bad, 0, 4, 512, 512, bad, bad, None) == mq.MQ_ERR_INVALID_ARG
    fake = P(4096)  # never dereferenced: validation fails first
    assert L.mq_quantize_act(fake, 0, 4, 500, 512, fake, fake, None) == mq.MQ_ERR_INVALID_ARG  # K % 128
    assert L.mq_quantize_act(P(4098), 0, 4, 512, 512, fake, fake, None) == mq.MQ_ERR_ALIGNMENT
    assert L.mq_quantize_act(fake, 7, 4, 512, 512, fake, fake, None) == mq.MQ_ERR_INVALID_ARG  # dtype
    # gemm (xq, xs, M, wpk, N, K, row_ptr, col_idx, nnzb, rpk, y, yt, ws, ws_bytes, stream):
    # N not a multiple of 128; misaligned xq; workspace too small
    args = [fake, fake, 4, fake, 192, 512, fake, fake, 0, None, fake, 1, None, 0, None]
    assert L.mq_w4a4_residual_gemm(*args) == mq.MQ_ERR_INVALID_ARG
    args[4] = 512
    args[0] = P(4097)
    assert L.mq_w4a4_residual_gemm(*args) == mq.MQ_ERR_ALIGNMENT
    args[0] = fake
    args[2] = 32
    args[5] = 4096
    args[4] = 4096
    assert L.mq_w4a4_residual_gemm(*args) == mq.MQ_ERR_WORKSPACE
    # residual count without residual records
    args = [fake, fake, 4, fake, 512, 512, fake, fake, 3, None, fake, 1, None, 0, None]
    assert L.mq_w4a4_residual_gemm(*args) == mq.MQ_ERR_INVALID_ARG
    # select: budget outside [0, 1]
    assert L.mq_select_blocks(fake, 512, 512, fake, 0, 256, 1.5, fake, fake, None, None, fake, 1 << 20,
                              None) == mq.MQ_ERR_INVALID_ARG
    assert b"budget" in L.mq_last_error()
