"""The byte accounting behind the roofline figure (host arithmetic, no GPU):
the algorithmic bytes a GEMM must move, against values worked out by hand from
the record layouts, and the packed buffers' sizes against those bytes."""
import pytest
import torch

from dense_sparse_int4_gb300 import mq

# (N, K, residual blocks at a 10 % budget, base bytes, residual bytes), worked by hand:
#   base     = N*K/2 codes + 2*N*K/128 fp16 scales
#   residual = nnzb * (4096 codes + 128 scale bytes + 4 column index) + 4*(N/64 + 1) row pointers
CASES = [
    (512, 512, 3, 135_168, 12_684 + 36),
    (4096, 4096, 204, 8_650_752, 862_512 + 260),
    (1024, 4096, 51, 2_162_688, 215_628 + 68),
    (14336, 4096, 716, 30_277_632, 3_027_248 + 900),
    (4096, 14336, 716, 30_277_632, 3_027_248 + 260),
]


def packed(N, K, nnzb):
    return mq.PackedLinear(N, K, nnzb,
                           torch.empty((N // 128) * (K // 128), mq.WREC_BYTES, dtype=torch.uint8),
                           torch.empty(N // 64 + 1, dtype=torch.int32), torch.empty(nnzb, dtype=torch.int32),
                           torch.empty(nnzb, mq.RREC_BYTES, dtype=torch.uint8))


@pytest.mark.parametrize("N,K,nnzb,base,res", CASES)
def test_weight_bytes_match_hand_values(N, K, nnzb, base, res):
    pl = packed(N, K, nnzb)
    assert pl.weight_bytes() == base + res
    # the packed buffers hold exactly those bytes
    stored = pl.wpk.numel() + pl.rpk.numel() + 4 * (pl.row_ptr.numel() + pl.col_idx.numel())
    assert stored == base + res


def test_nnzb_is_ten_percent_of_blocks():
    assert mq.num_selected(4096, 4096, 0.10) == 204
    assert mq.num_selected(1024, 4096, 0.10) == 51
    assert mq.num_selected(14336, 4096, 0.10) == 716
    assert mq.num_selected(512, 512, 0.10) == 3


def test_residual_adds_about_ten_percent_bytes():
    for N, K, nnzb, base, res in CASES[1:]:
        assert 0.09 < res / base < 0.11
