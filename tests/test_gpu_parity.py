"""GPU parity: the CUDA path (through the C ABI) against the oracle.

Integer stages (quantized activations, packed weights, block lists, group
dots) must match bit for bit; the fp32 epilogue within 1e-5 of the sum of
absolute terms; bf16 outputs within 1 ulp.  Small cases are compared whole;
the full-size workloads are compared on sampled outputs the oracle computes
one by one."""
import numpy as np
import pytest
import torch

import oracle as O
from dense_sparse_int4_gb300 import mq, synth
from tests.gpu_helpers import (check_bf16, check_close, dev_act, dev_half, host_u16, logical_rq, logical_rsc, logical_wq,
                               logical_wsc, logical_xq, logical_xs, oracle_prep_for_csr, packed_from_csr,
                               xq_padding)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    mq.check_device_error()


# ----------------------------------------------------------------------------
# activation quantizer
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("M,K,dtype", [(4, 512, "f16"), (37, 384, "f16"), (1, 128, "bf16"), (300, 1024, "bf16"),
                                       (2048, 4096, "bf16"), (32, 14336, "f16")])
def test_quantize_act_bit_exact(M, K, dtype):
    x = synth.activations(M, K, seed=M + K, count=synth.n_outliers(K), dtype=dtype)
    if M > 2:  # edge rows: all zeros, fp16-subnormal scale, huge values
        x[0] = 0
        sub = np.float32(2.0 ** -20)
        x[1] = synth.to_bits(np.full(K, sub, np.float32) * np.sign(np.random.default_rng(0).standard_normal(K)).astype(np.float32), dtype)
        if dtype == "bf16":
            x[2, ::7] = synth.to_bits(np.array([1e6], np.float32), "bf16")[0]
    xt = dev_act(x, dtype == "bf16")
    xq, xs = mq.quantize_act(xt)
    torch.cuda.synchronize()
    q, s = O.quantize_act(x, dtype == "bf16")
    assert np.array_equal(logical_xq(xq, M), O.pack_nibbles(q))
    assert np.array_equal(logical_xs(xs, M), s)
    assert not host_u16(xs)[:, M:].any() and not xq_padding(xq, M).any()  # padding tokens zeroed


def test_quantize_act_row_stride():
    M, K, ld = 5, 256, 384
    x = synth.activations(M, ld, seed=3, count=4)
    xt = dev_half(x)[:, :K]
    xq, xs = mq.quantize_act(xt)
    q, s = O.quantize_act(np.ascontiguousarray(x[:, :K]), False)
    assert np.array_equal(logical_xq(xq, M), O.pack_nibbles(q))
    assert np.array_equal(logical_xs(xs, M), s)


# ----------------------------------------------------------------------------
# offline: selection and packing
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("N,K,budget,conc", [(512, 512, 0.10, False), (512, 512, 0.0, False), (512, 512, 1.0, False),
                                             (1024, 4096, 0.10, True), (4096, 4096, 0.10, False),
                                             (1024, 5120, 0.20, True)])
def test_select_blocks_bit_exact(N, K, budget, conc):
    w = synth.weights(N, K, seed=N ^ K)
    if conc:
        w = synth.inject_concentrated(w, seed=1)
    xcal = synth.calibration(K, seed=N ^ K, count=synth.n_outliers(K))
    rp, ci, h, d = mq.select_blocks(dev_half(w), dev_half(xcal), budget, want_h=True, want_delta=True)
    p = O.prepare(w, xcal, False, budget)
    assert np.array_equal(h.cpu().numpy(), p.h)  # bitwise: fixed order, no FMA on either side
    assert np.array_equal(d.cpu().numpy(), p.delta)
    assert np.array_equal(rp.cpu().numpy(), p.row_ptr)
    assert np.array_equal(ci.cpu().numpy(), p.col_idx)


def test_select_blocks_bf16_calibration():
    N, K = 512, 1024
    w = synth.weights(N, K, seed=5)
    xcal = synth.calibration(K, seed=5, count=4, dtype="bf16")
    rp, ci, h, d = mq.select_blocks(dev_half(w), dev_act(xcal, True), 0.1, want_h=True, want_delta=True)
    p = O.prepare(w, xcal, True, 0.1)
    assert np.array_equal(h.cpu().numpy(), p.h) and np.array_equal(d.cpu().numpy(), p.delta)
    assert np.array_equal(ci.cpu().numpy(), p.col_idx)


@pytest.mark.parametrize("N,K,budget", [(512, 512, 0.10), (1024, 4096, 0.25), (256, 384, 1.0), (4096, 1024, 0.0)])
def test_pack_weights_bit_exact(N, K, budget):
    w = synth.inject_concentrated(synth.weights(N, K, seed=7), seed=7, frac=0.05)
    xcal = synth.calibration(K, seed=7, count=4)
    pl = mq.prepare_linear(dev_half(w), dev_half(xcal), budget)
    p = O.prepare(w, xcal, False, budget)
    assert np.array_equal(logical_wq(pl.wpk, N, K), O.pack_nibbles(p.qw))
    assert np.array_equal(logical_wsc(pl.wpk, N, K), p.sw)
    assert pl.nnzb == p.ksel
    assert np.array_equal(logical_rq(pl.rpk, pl.nnzb), p.qr)
    assert np.array_equal(logical_rsc(pl.rpk, pl.nnzb), p.sr)


# ----------------------------------------------------------------------------
# the fused GEMM
# ----------------------------------------------------------------------------

def _case(M, N, K, budget, seed, x_dtype="f16", conc=False):
    x = synth.activations(M, K, seed=seed, count=synth.n_outliers(K), dtype=x_dtype)
    w = synth.weights(N, K, seed=seed)
    if conc:
        w = synth.inject_concentrated(w, seed=seed)
    xcal = synth.calibration(K, seed=seed, count=synth.n_outliers(K), dtype=x_dtype)
    return x, w, xcal


@pytest.mark.parametrize("M,N,K,budget", [(4, 512, 512, 0.10), (17, 256, 512, 0.5), (33, 384, 768, 1.0),
                                          (64, 128, 256, 0.25), (100, 256, 1024, 0.3), (1, 128, 128, 1.0)])
def test_group_dots_bit_exact(M, N, K, budget):
    x, w, xcal = _case(M, N, K, budget, seed=11)
    pl = mq.prepare_linear(dev_half(w), dev_half(xcal), budget)
    xq, xs = mq.quantize_act(dev_half(x))
    dw, dr = mq.debug_group_dots(xq, xs, M, pl)
    mq.check_device_error()
    assert mq.gemm_plan(M, N, K)["decode"] == (M <= 32)  # which kernel these dots came from
    qx, sx = O.quantize_act(x, False)
    p = O.prepare(w, xcal, False, budget)
    assert np.array_equal(dw.cpu().numpy(), O.group_dots(qx, p.qw))
    if p.ksel:
        assert np.array_equal(dr.cpu().numpy(), O.residual_dots(qx, p.qr, p.col_idx))


@pytest.mark.parametrize("lin", synth.LLAMA3_8B + synth.QWEN3_32B, ids=lambda l: f"{l.name}-{l.K}x{l.N}")
def test_decode_kernel_covers_decode_shapes(lin):
    """Up to 32 tokens, every layer shape of the two model families runs on
    the decode kernel (a launch-resource failure would otherwise fall back to
    the general kernel silently); 33 tokens and more run on the general one."""
    for M in (1, 4, 8, 9, 16, 17, 32):
        plan = mq.gemm_plan(M, lin.N, lin.K)
        assert plan["decode"], (M, plan)
        assert plan["tokens_per_tile"] >= M and plan["clusters"] > 0 and plan["stages"] >= 2
    assert not mq.gemm_plan(33, lin.N, lin.K)["decode"]


@pytest.mark.parametrize("variant", ["col", "warp", "tc"])
@pytest.mark.parametrize("M,N,K,budget", [(9, 384, 1024, 0.3), (16, 512, 2048, 0.2), (24, 256, 768, 1.0),
                                          (3, 640, 384, 0.4)])
def test_decode_variants_match_oracle(variant, M, N, K, budget, monkeypatch):
    """Every form of the decode kernel (forced through MQ_DECODE_VARIANT):
    dots bit for bit, Y within the fp32 bound, on sizes any may serve (640
    rows: a ragged last tile-group of the column form)."""
    monkeypatch.setenv("MQ_DECODE_VARIANT", variant)
    plan = mq.gemm_plan(M, N, K)
    assert plan["variant"] == {"col": "column", "warp": "warp-mma", "tc": "tensor-memory"}[variant]
    x, w, xcal = _case(M, N, K, budget, seed=M + N)
    pl = mq.prepare_linear(dev_half(w), dev_half(xcal), budget)
    xq, xs = mq.quantize_act(dev_half(x))
    dw, dr = mq.debug_group_dots(xq, xs, M, pl)
    y32 = mq.gemm(xq, xs, M, pl, out_dtype=torch.float32)
    y16 = mq.gemm(xq, xs, M, pl, out_dtype=torch.bfloat16)
    mq.check_device_error()
    qx, sx = O.quantize_act(x, False)
    p = O.prepare(w, xcal, False, budget)
    assert np.array_equal(dw.cpu().numpy(), O.group_dots(qx, p.qw))
    if p.ksel:
        assert np.array_equal(dr.cpu().numpy(), O.residual_dots(qx, p.qr, p.col_idx))
    y, a = O.linear(qx, sx, p)
    check_close(y32.cpu().numpy(), y, a)
    check_bf16(host_u16(y16), y, a)


@pytest.mark.parametrize("M,variant", [(32, "col"), (16, "col"), (8, "col"), (4, "col"), (1, "col"),
                                       (32, "warp"), (32, "tc"), (16, "tc"), (8, "warp"), (8, "tc"), (4, "warp"),
                                       (1, "warp"), (1, "tc"), (33, None), (128, None), (33, "image"),
                                       (300, "image"), (300, "conv")])
def test_group_dots_extremes(M, variant, monkeypatch):
    """Adversarial codes: every product +49, every product -49, alternating
    cancellation; sums reach +-6272 per group, exactly.  Up to 32 tokens this
    runs the decode kernel, in its column and warp-MMA forms (mask-and-offset
    unpack to E4M3, fp32 MMA accumulators) and its tensor-memory form; above 32 tokens
    the general kernel (exact-integer E4M3 table), in its converter form and its
    image form (the default from 128 tokens)."""
    if variant in ("image", "conv"):
        monkeypatch.setenv("MQ_GENERAL_FORM", variant)
    elif variant:
        monkeypatch.setenv("MQ_DECODE_VARIANT", variant)
    N, K = 128, 256
    x = np.full((M, K), 7.0, np.float32)
    w = np.full((N, K), 7.0 * 0.01, np.float32)
    w[64:, :] *= -1.0
    if M > 1:  # the second half of the tokens cancel: odd products negative
        x[M // 2:, 1::2] *= -1.0
    xb, wb = synth.f32_to_f16_bits(x), synth.f32_to_f16_bits(w)
    xcal = synth.calibration(K, seed=1, count=4)
    pl = mq.prepare_linear(dev_half(wb), dev_half(xcal), 1.0)
    xq, xs = mq.quantize_act(dev_half(xb))
    dw, _ = mq.debug_group_dots(xq, xs, M, pl)
    qx, _ = O.quantize_act(xb, False)
    p = O.prepare(wb, xcal, False, 1.0)
    ref = O.group_dots(qx, p.qw)
    assert ref.max() == 6272 and ref.min() == -6272 and (ref == 0).any() == (M > 1)
    plan = mq.gemm_plan(M, N, K)
    assert plan["variant"] == {"col": "column", "warp": "warp-mma", "tc": "tensor-memory", "image": "image",
                               "conv": "general", None: "image" if M >= 128 else "general"}[variant]
    assert np.array_equal(dw.cpu().numpy(), ref)


@pytest.mark.parametrize("M,N,K,budget,x_dtype", [
    (4, 512, 512, 0.10, "f16"),      # the 512x512 single linear, top-3 of 32 blocks
    (1, 256, 512, 0.20, "f16"), (8, 1024, 2048, 0.10, "f16"), (16, 512, 1024, 0.0, "f16"),
    (17, 384, 640, 0.30, "bf16"), (32, 1024, 4096, 0.10, "f16"), (33, 256, 512, 1.0, "f16"),
    (64, 512, 1024, 0.10, "bf16"), (65, 256, 768, 0.10, "f16"), (128, 256, 512, 0.10, "f16"),
    (200, 384, 1280, 0.15, "bf16"),
])
def test_gemm_matches_oracle(M, N, K, budget, x_dtype):
    x, w, xcal = _case(M, N, K, budget, seed=M * 7 + N, x_dtype=x_dtype)
    isb = x_dtype == "bf16"
    pl = mq.prepare_linear(dev_half(w), dev_act(xcal, isb), budget)
    xq, xs = mq.quantize_act(dev_act(x, isb))
    y32 = mq.gemm(xq, xs, M, pl, out_dtype=torch.float32)
    y16 = mq.gemm(xq, xs, M, pl, out_dtype=torch.bfloat16)
    mq.check_device_error()
    qx, sx = O.quantize_act(x, isb)
    p = O.prepare(w, xcal, isb, budget)
    y, a = O.linear(qx, sx, p)
    check_close(y32.cpu().numpy(), y, a)
    check_bf16(host_u16(y16), y, a)
    # deterministic: a second call gives the same bits
    y32b = mq.gemm(xq, xs, M, pl, out_dtype=torch.float32)
    assert torch.equal(y32, y32b)


def test_gemm_concentrated_block_row():
    """Every residual block in one block row; no residual anywhere else."""
    M, N, K = 32, 512, 2048
    x, w, _ = _case(M, N, K, 0.0, seed=3)
    G = K // 128
    rp = np.zeros(N // 64 + 1, np.int32)
    rp[3:] = G  # block row 2 holds all G blocks
    ci = np.arange(G, dtype=np.int32)
    pl = packed_from_csr(dev_half(w), rp, ci)
    xq, xs = mq.quantize_act(dev_half(x))
    y32 = mq.gemm(xq, xs, M, pl, out_dtype=torch.float32)
    p = oracle_prep_for_csr(w, rp, ci)
    qx, sx = O.quantize_act(x, False)
    y, a = O.linear(qx, sx, p)
    check_close(y32.cpu().numpy(), y, a)


@pytest.mark.parametrize("M,form", [(20, None), (140, "image"), (140, "conv")])
def test_gemm_both_halves_and_empty_rows(M, form, monkeypatch):
    """Blocks in both 64-row halves of a tile at the same group, single halves,
    and tiles with no residual at all (decode kernel, and both forms of the
    general kernel)."""
    if form:
        monkeypatch.setenv("MQ_GENERAL_FORM", form)
    N, K = 512, 1024
    x, w, _ = _case(M, N, K, 0.0, seed=9)
    G = K // 128
    rows = {0: [0, 3, 7], 1: [3, 5], 2: [], 3: [1], 4: [], 5: [], 6: [0, 7], 7: [0, 1, 2, 3, 4, 5, 6, 7]}
    rp = np.zeros(N // 64 + 1, np.int32)
    ci = []
    for br in range(N // 64):
        ci += rows[br]
        rp[br + 1] = len(ci)
    ci = np.array(ci, np.int32)
    pl = packed_from_csr(dev_half(w), rp, ci)
    xq, xs = mq.quantize_act(dev_half(x))
    y32 = mq.gemm(xq, xs, M, pl, out_dtype=torch.float32)
    dw, dr = mq.debug_group_dots(xq, xs, M, pl)
    p = oracle_prep_for_csr(w, rp, ci)
    qx, sx = O.quantize_act(x, False)
    y, a = O.linear(qx, sx, p)
    check_close(y32.cpu().numpy(), y, a)
    assert np.array_equal(dr.cpu().numpy(), O.residual_dots(qx, p.qr, ci))
    assert np.array_equal(dw.cpu().numpy(), O.group_dots(qx, p.qw))
    if form:
        assert mq.gemm_plan(M, N, K)["variant"] == {"image": "image", "conv": "general"}[form]


@pytest.mark.parametrize("form", ["image", "conv"])
@pytest.mark.parametrize("M,N,K,budget,x_dtype", [(33, 256, 512, 1.0, "f16"), (130, 384, 1280, 0.2, "bf16"),
                                                  (300, 256, 640, 0.3, "f16"), (257, 1024, 2048, 0.1, "bf16"),
                                                  (512, 128, 128, 0.0, "f16"), (384, 640, 512, 0.5, "f16")])
def test_general_forms_match_oracle(form, M, N, K, budget, x_dtype, monkeypatch):
    """The general kernel's two forms, forced through MQ_GENERAL_FORM: the image
    form (a pre-pass writes every operand's shared-memory image; both MMA
    operands from shared memory) and the converter form.  Dots bit for bit, Y
    within the fp32 bound and bf16 within 1 ulp; ragged token tails, odd group
    counts, tiles cut across several CTAs (several rounds of pieces) and a
    single-group K; a second call gives the same bits."""
    monkeypatch.setenv("MQ_GENERAL_FORM", form)
    assert mq.gemm_plan(M, N, K)["variant"] == {"image": "image", "conv": "general"}[form]
    x, w, xcal = _case(M, N, K, budget, seed=M * 3 + N + K, x_dtype=x_dtype)
    isb = x_dtype == "bf16"
    pl = mq.prepare_linear(dev_half(w), dev_act(xcal, isb), budget)
    xq, xs = mq.quantize_act(dev_act(x, isb))
    dw, dr = mq.debug_group_dots(xq, xs, M, pl)
    y32 = mq.gemm(xq, xs, M, pl, out_dtype=torch.float32)
    y16 = mq.gemm(xq, xs, M, pl, out_dtype=torch.bfloat16)
    y32b = mq.gemm(xq, xs, M, pl, out_dtype=torch.float32)
    mq.check_device_error()
    qx, sx = O.quantize_act(x, isb)
    p = O.prepare(w, xcal, isb, budget)
    assert np.array_equal(dw.cpu().numpy(), O.group_dots(qx, p.qw))
    if p.ksel:
        assert np.array_equal(dr.cpu().numpy(), O.residual_dots(qx, p.qr, p.col_idx))
    y, a = O.linear(qx, sx, p)
    check_close(y32.cpu().numpy(), y, a)
    check_bf16(host_u16(y16), y, a)
    assert torch.equal(y32, y32b)


# ----------------------------------------------------------------------------
# the fused linear: quantizer + grouped GEMM in one call
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("M,K,Ns,budget,x_dtype", [
    (4, 512, [512], 0.10, "f16"),
    (1, 256, [256, 128], 0.20, "f16"),
    (9, 1024, [384, 128, 256], 0.30, "bf16"),
    (17, 2048, [512, 512], 0.50, "f16"),
    (32, 4096, [4096, 1024, 1024], 0.10, "f16"),  # q, k, v of the Llama-3-8B-shaped layer
    (40, 512, [256, 384], 0.10, "f16"),  # above 32 tokens: the quantizer, then the general kernel
    # from 128 tokens: the quantizer, then the image form
    (130, 640, [256, 384, 128], 0.20, "bf16"),
    (300, 1024, [512], 0.10, "f16"),
])
def test_fused_linear_matches_oracle(M, K, Ns, budget, x_dtype):
    """mq_w4a4_residual_linear: the quantized activations it reports are bit
    for bit mq_quantize_act's (the oracle's), and every matrix's Y, written as
    a column slice of one wider output, is within the fp32 bound."""
    isb = x_dtype == "bf16"
    x = synth.activations(M, K, seed=M + K, count=synth.n_outliers(K), dtype=x_dtype)
    pls, preps = [], []
    for i, N in enumerate(Ns):
        w = synth.weights(N, K, seed=100 + i)
        xcal = synth.calibration(K, seed=i, count=synth.n_outliers(K), dtype=x_dtype)
        pls.append(mq.prepare_linear(dev_half(w), dev_act(xcal, isb), budget))
        preps.append(O.prepare(w, xcal, isb, budget))
    Mp = mq.padded_tokens(M)
    xq = torch.full((K // 128, Mp, 64), 0xAB, dtype=torch.uint8, device="cuda")
    xs = torch.full((K // 128, Mp), float("nan"), dtype=torch.float16, device="cuda")
    wide = sum(Ns) + 8
    Y = torch.full((M, wide), float("nan"), dtype=torch.float32, device="cuda")
    offs = np.cumsum([0] + Ns)
    outs = [Y[:, offs[i]:offs[i + 1]] for i in range(len(Ns))]
    mq.fused_linear(dev_act(x, isb), pls, outs=outs, xq=xq, xs=xs)
    Yb = torch.full((M, wide), float("nan"), dtype=torch.bfloat16, device="cuda")
    mq.fused_linear(dev_act(x, isb), pls, outs=[Yb[:, offs[i]:offs[i + 1]] for i in range(len(Ns))])
    mq.check_device_error()
    qx, sx = O.quantize_act(x, isb)
    assert np.array_equal(logical_xq(xq, M), O.pack_nibbles(qx))
    assert np.array_equal(logical_xs(xs, M), sx)
    assert not host_u16(xs)[:, M:].any() and not xq_padding(xq, M).any()
    yh, ybh = Y.cpu().numpy(), host_u16(Yb)
    for i, p in enumerate(preps):
        y, a = O.linear(qx, sx, p)
        check_close(yh[:, offs[i]:offs[i + 1]], y, a)
        check_bf16(ybh[:, offs[i]:offs[i + 1]], y, a)
    assert np.isnan(yh[:, sum(Ns):]).all()  # columns past the last slice untouched
    assert mq.gemm_plan(M, sum(Ns), K)["decode"] == (M <= 32)


def _quantizer_corner_rows(M, K, dtype, seed):
    """Activation rows (as fp16 / bf16 bits) that hit the quantizer's corners,
    one kind per token: exact half-integer quotients v / s (round half to
    even) with amax = 7 s, the same moved one ulp of the input format either
    way, fp16-subnormal scales (codes clamp), all-zero groups, scales that
    saturate at 65504 (bf16 only), random rows."""
    rng = np.random.default_rng(seed)
    out = np.zeros((M, K), np.uint16)
    for m in range(M):
        kind = m % 6
        for g in range(K // 128):
            s = np.float32(2.0 ** int(rng.integers(-6, 4)) * (1 + int(rng.integers(0, 8)) / 8))
            if kind in (0, 1):
                row = ((rng.integers(-7, 7, 128) + 0.5) * s).astype(np.float32)  # exact in both formats
                bits = synth.to_bits(row, dtype)
                if kind == 1:  # one ulp up or down in magnitude: no longer a tie
                    bits = (bits.astype(np.int32) + rng.choice([-1, 1], 128)).astype(np.uint16)
                bits[int(rng.integers(0, 128))] = synth.to_bits(np.array([7 * s], np.float32), dtype)[0]
            elif kind == 2:
                bits = synth.to_bits((rng.standard_normal(128) * 2.0 ** -19).astype(np.float32), dtype)
            elif kind == 3:
                bits = np.zeros(128, np.uint16)
            elif kind == 4 and dtype == "bf16":
                bits = synth.to_bits((rng.standard_normal(128) * 1e6).astype(np.float32), dtype)
            else:
                bits = synth.to_bits((rng.standard_normal(128) * 3.0).astype(np.float32), dtype)
            out[m, 128 * g:128 * (g + 1)] = bits
    return out


@pytest.mark.parametrize("variant", ["col", "warp"])
@pytest.mark.parametrize("M,x_dtype,pad", [(32, "f16", 0), (32, "bf16", 0), (6, "f16", 0), (12, "bf16", 4)])
def test_fused_quantizer_corners(variant, M, x_dtype, pad, monkeypatch):
    """The quantizer inside the fused call (the column form's stage build and
    the image kernel, which round with a refined reciprocal rather than a
    division) against the oracle bit for bit on corner rows, and Y within the
    fp32 bound.  pad > 0 gives X a row stride that is not a multiple of 8
    elements: the column form then runs the stand-alone quantizer first."""
    monkeypatch.setenv("MQ_DECODE_VARIANT", variant)
    K, N = 512, 256
    isb = x_dtype == "bf16"
    x = _quantizer_corner_rows(M, K, x_dtype, seed=M + pad)
    xw = np.zeros((M, K + pad), np.uint16)
    xw[:, :K] = x
    xt = dev_act(xw, isb)[:, :K]
    w = synth.weights(N, K, seed=5)
    xcal = synth.calibration(K, seed=5, count=4, dtype=x_dtype)
    pl = mq.prepare_linear(dev_half(w), dev_act(xcal, isb), 0.25)
    Mp = mq.padded_tokens(M)
    xq = torch.full((K // 128, Mp, 64), 0xAB, dtype=torch.uint8, device="cuda")
    xs = torch.full((K // 128, Mp), float("nan"), dtype=torch.float16, device="cuda")
    y32 = mq.fused_linear(xt, [pl], out_dtype=torch.float32, xq=xq, xs=xs)[0]
    mq.check_device_error()
    assert mq.gemm_plan(M, N, K)["variant"] == {"col": "column", "warp": "warp-mma"}[variant]
    qx, sx = O.quantize_act(x, isb)
    assert np.array_equal(logical_xq(xq, M), O.pack_nibbles(qx))
    assert np.array_equal(logical_xs(xs, M), sx)
    assert not host_u16(xs)[:, M:].any() and not xq_padding(xq, M).any()
    y, a = O.linear(qx, sx, O.prepare(w, xcal, isb, 0.25))
    check_close(y32.cpu().numpy(), y, a)


@pytest.mark.parametrize("M,x_dtype,pad", [(160, "f16", 0), (160, "bf16", 4), (300, "f16", 4)])
def test_image_prepass_quantizer_corners(M, x_dtype, pad):
    """From 128 tokens the fused call quantizes X, then its image pre-pass turns
    the codes into the activation image: the xq / xs it reports against the
    oracle bit for bit on the corner rows (ties, ties moved one ulp, subnormal
    and saturating scales, zero groups; a row stride of K + pad), padding tokens
    zero, and Y within the fp32 bound (the activation image carries the same codes)."""
    K, N = 640, 256
    isb = x_dtype == "bf16"
    x = _quantizer_corner_rows(M, K, x_dtype, seed=M + 7 * pad)
    xw = np.zeros((M, K + pad), np.uint16)
    xw[:, :K] = x
    xt = dev_act(xw, isb)[:, :K]
    w = synth.weights(N, K, seed=9)
    xcal = synth.calibration(K, seed=9, count=4, dtype=x_dtype)
    pl = mq.prepare_linear(dev_half(w), dev_act(xcal, isb), 0.25)
    assert mq.gemm_plan(M, N, K)["variant"] == "image"
    Mp = mq.padded_tokens(M)
    xq = torch.full((K // 128, Mp, 64), 0xAB, dtype=torch.uint8, device="cuda")
    xs = torch.full((K // 128, Mp), float("nan"), dtype=torch.float16, device="cuda")
    y32 = mq.fused_linear(xt, [pl], out_dtype=torch.float32, xq=xq, xs=xs)[0]
    mq.check_device_error()
    qx, sx = O.quantize_act(x, isb)
    assert np.array_equal(logical_xq(xq, M), O.pack_nibbles(qx))
    assert np.array_equal(logical_xs(xs, M), sx)
    assert not host_u16(xs)[:, M:].any() and not xq_padding(xq, M).any()
    y, a = O.linear(qx, sx, O.prepare(w, xcal, isb, 0.25))
    check_close(y32.cpu().numpy(), y, a)


@pytest.mark.parametrize("M,K,x_dtype,pad", [(12, 512, "f16", 0), (12, 512, "bf16", 0), (37, 2304, "f16", 4),
                                             (300, 640, "bf16", 4)])
def test_quantize_act_corners(M, K, x_dtype, pad):
    """The stand-alone quantizer (a half-warp per token and group, rounding with
    a refined reciprocal instead of a division) against the oracle bit for bit
    on the corner rows: exact ties, ties moved one ulp, subnormal and saturating
    scales, zero groups; 18 groups (a block whose second half-warps have no
    group), padding tokens, and a row stride of K + 4 elements."""
    isb = x_dtype == "bf16"
    x = _quantizer_corner_rows(M, K, x_dtype, seed=3 * M + pad)
    xw = np.zeros((M, K + pad), np.uint16)
    xw[:, :K] = x
    xq, xs = mq.quantize_act(dev_act(xw, isb)[:, :K])
    mq.check_device_error()
    qx, sx = O.quantize_act(x, isb)
    assert np.array_equal(logical_xq(xq, M), O.pack_nibbles(qx))
    assert np.array_equal(logical_xs(xs, M), sx)
    assert not host_u16(xs)[:, M:].any() and not xq_padding(xq, M).any()


@pytest.mark.parametrize("M,N,K,budget", [(4, 4096, 4096, 0.10), (32, 4096, 4096, 0.10), (8, 1536, 4096, 0.3),
                                          (16, 640, 1024, 1.0), (3, 2048, 512, 0.2)])
def test_cluster_mode_matches_oracle(M, N, K, budget, monkeypatch):
    """Small launches give each weight tile a thread-block cluster whose CTAs send their
    stream-K pieces into the head CTA's shared memory: Y (fp32 and bf16) within the bound,
    the same bits twice in a row, and the stream-K form (clusters off) within the bound too."""
    x, w, xcal = _case(M, N, K, budget, seed=M + N + K)
    pl = mq.prepare_linear(dev_half(w), dev_half(xcal), budget)
    xq, xs = mq.quantize_act(dev_half(x))
    plan = mq.gemm_plan(M, N, K)
    assert plan["variant"] == "warp-mma" and plan["cluster"] >= 2, plan
    assert plan["clusters"] == plan["cluster"] * (N // 128)
    y32 = mq.gemm(xq, xs, M, pl, out_dtype=torch.float32)
    y32b = mq.gemm(xq, xs, M, pl, out_dtype=torch.float32)
    y16 = mq.gemm(xq, xs, M, pl, out_dtype=torch.bfloat16)
    mq.check_device_error()
    monkeypatch.setenv("MQ_DECODE_CLUSTER", "0")
    assert mq.gemm_plan(M, N, K)["cluster"] == 1
    y32s = mq.gemm(xq, xs, M, pl, out_dtype=torch.float32)
    mq.check_device_error()
    qx, sx = O.quantize_act(x, False)
    y, a = O.linear(qx, sx, O.prepare(w, xcal, False, budget))
    check_close(y32.cpu().numpy(), y, a)
    check_bf16(host_u16(y16), y, a)
    assert torch.equal(y32, y32b)
    check_close(y32s.cpu().numpy(), y, a)


@pytest.mark.parametrize("variant,M", [("col", 4), ("col", 32), ("warp", 4), ("tc", 32)])
def test_dense_residual_back_to_back(variant, M, monkeypatch):
    """Every block residual (budget 1): each stage fills the residual ring a
    full lap, and with ~4 stages per CTA the compute sets drift apart.  Twelve
    calls back to back on one stream and workspace (each launch overlapping
    the previous one's tail) must all equal the oracle: a set must never take
    a ring slot's older record for its own."""
    monkeypatch.setenv("MQ_DECODE_VARIANT", variant)
    N, K = 8192, 4096
    x = synth.activations(M, K, seed=91, count=synth.n_outliers(K))
    w = synth.weights(N, K, seed=92)
    xcal = synth.calibration(K, seed=93, count=synth.n_outliers(K))
    pl = mq.prepare_linear(dev_half(w), dev_half(xcal), 1.0)
    p = O.prepare(w, xcal, False, 1.0)
    assert pl.nnzb == p.ksel == (N // 64) * (K // 128)
    xt = dev_half(x)
    ys = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") for _ in range(12)]
    ws, _ = mq.linear_workspace(M, K, [N], "cuda")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for y in ys:
            mq.fused_linear(xt, [pl], outs=[y], ws=ws, stream=stream)
    stream.synchronize()
    mq.check_device_error()
    qx, sx = O.quantize_act(x, False)
    yo, a = O.linear(qx, sx, p)
    for y in ys:
        check_close(y.cpu().numpy(), yo, a)
    assert mq.gemm_plan(M, N, K)["variant"] == {"col": "column", "warp": "warp-mma", "tc": "tensor-memory"}[variant]


# ----------------------------------------------------------------------------
# full-size workloads, sampled outputs
# ----------------------------------------------------------------------------

def _sampled_parity(M, lin, budget, x_dtype, seed, conc=False, nsamp=384):
    N, K = lin.N, lin.K
    x, w, xcal = _case(M, N, K, budget, seed=seed, x_dtype=x_dtype, conc=conc)
    isb = x_dtype == "bf16"
    pl = mq.prepare_linear(dev_half(w), dev_act(xcal, isb), budget)
    xq, xs = mq.quantize_act(dev_act(x, isb))
    y16 = mq.gemm(xq, xs, M, pl, out_dtype=torch.bfloat16)
    y32 = mq.gemm(xq, xs, M, pl, out_dtype=torch.float32)
    mq.check_device_error()
    qx, sx = O.quantize_act(x, isb)
    assert np.array_equal(logical_xq(xq, M), O.pack_nibbles(qx))
    p = O.prepare(w, xcal, isb, budget)
    assert np.array_equal(pl.row_ptr.cpu().numpy(), p.row_ptr) and np.array_equal(pl.col_idx[: pl.nnzb].cpu().numpy(), p.col_idx)
    rng = np.random.default_rng(seed)
    ms = rng.integers(0, M, nsamp)
    ns = rng.integers(0, N, nsamp)
    # plus every row of one selected block row and the last tile's rows
    if p.ksel:
        br = int(O.csr_block_rows(p.row_ptr)[0])
        ns = np.concatenate([ns, np.arange(br * 64, br * 64 + 64), np.arange(N - 16, N)])
        ms = np.concatenate([ms, np.full(64, M - 1), np.zeros(16, np.int64)])
    y, a = O.linear_entries(qx, sx, p, ms, ns)
    check_close(y32.cpu().numpy()[ms, ns], y, a)
    check_bf16(host_u16(y16)[ms, ns], y, a)


@pytest.mark.parametrize("name,M,variant", [("gate", 8, "col"), ("gate", 32, "col"), ("down", 4, "col"),
                                            ("gate", 8, "warp"), ("gate", 16, "warp"), ("gate", 32, "tc"),
                                            ("down", 4, "warp")])
def test_full_size_whole_output(name, M, variant, monkeypatch):
    """One full-size Llama-3-8B linear through the fused call, every output
    (fp32 and bf16) against the oracle: the whole matrix, not a sample."""
    monkeypatch.setenv("MQ_DECODE_VARIANT", variant)
    lin = {l.name: l for l in synth.LLAMA3_8B}[name]
    x, w, xcal = _case(M, lin.N, lin.K, 0.10, seed=M * 13 + lin.N)
    pl = mq.prepare_linear(dev_half(w), dev_half(xcal), 0.10)
    xt = dev_half(x)
    y32 = mq.fused_linear(xt, [pl], out_dtype=torch.float32)[0]
    y16 = mq.fused_linear(xt, [pl])[0]
    mq.check_device_error()
    assert mq.gemm_plan(M, lin.N, lin.K)["variant"] == {"col": "column", "warp": "warp-mma", "tc": "tensor-memory"}[variant]
    qx, sx = O.quantize_act(x, False)
    y, a = O.linear(qx, sx, O.prepare(w, xcal, False, 0.10))
    check_close(y32.cpu().numpy(), y, a)
    check_bf16(host_u16(y16), y, a)


def test_prefill_row_slab_whole_rows():
    """M = 2048, K = 4096, N = 14336 (the general kernel): 48 whole output rows
    across a 128-token tile boundary, and the last token's row, against the oracle."""
    M, K, N, budget = 2048, 4096, 14336, 0.10
    x = synth.activations(M, K, seed=2, count=8, dtype="bf16")
    w = synth.weights(N, K, seed=77)
    xcal = synth.calibration(K, seed=2, count=8, dtype="bf16")
    pl = mq.prepare_linear(dev_half(w), dev_act(xcal, True), budget)
    y32 = mq.fused_linear(dev_act(x, True), [pl], out_dtype=torch.float32)[0]
    mq.check_device_error()
    assert not mq.gemm_plan(M, N, K)["decode"]
    rows = np.concatenate([np.arange(1000, 1048), [M - 1]])
    ms, ns = np.repeat(rows, N), np.tile(np.arange(N), rows.size)
    qx, sx = O.quantize_act(x[rows], True)
    # the oracle's activation quantization is per token: the slab's rows quantize alone
    y, a = O.linear_entries(qx, sx, O.prepare(w, xcal, True, budget), np.repeat(np.arange(rows.size), N), ns)
    check_close(y32.cpu().numpy()[ms, ns], y, a)


def _oracle_budgets(w, xcal, budgets):
    """O.prepare for several budgets of one matrix: the base products once, then per budget
    the selection and the residual codes (the oracle's own steps, in its order)."""
    N, K = w.shape
    qw, sw, r = O.base_quant(w)
    h = O.hessian_diag(xcal, False)
    d = O.delta_scores(r, h)
    out = {}
    for b in budgets:
        ksel = O.num_selected(N, K, b)
        rp, ci = O.select_topk(d, N, K, ksel)
        qr, sr = O.residual_quant(r, rp, ci)
        out[b] = O.Prepared(N, K, qw, sw, r, h, d, ksel, rp, ci, qr, sr, O.sel_of(rp, ci, N, K))
    return out


@pytest.mark.parametrize("placement", ["concentrated", "uniform"])
@pytest.mark.parametrize("lin", synth.QWEN3_32B, ids=lambda l: l.name)
def test_qwen3_sweep_sampled(lin, placement):
    """Qwen3-32B shapes: every linear x M in {4, 32, 512} x budgets {0, 5, 10, 20} %,
    errors injected into 2 % of the blocks or not: block lists bit for bit, and
    sampled outputs (plus a selected block row) against the oracle."""
    N, K = lin.N, lin.K
    seed = sum(map(ord, lin.name)) + (7 if placement == "concentrated" else 0)
    w = synth.weights(N, K, seed=seed)
    if placement == "concentrated":
        w = synth.inject_concentrated(w, seed=seed)
    xcal = synth.calibration(K, seed=seed, count=synth.n_outliers(K))
    budgets = (0.0, 0.05, 0.10, 0.20)
    preps = _oracle_budgets(w, xcal, budgets)
    wt, ct = dev_half(w), dev_half(xcal)
    rng = np.random.default_rng(seed)
    xs_host = {M: synth.activations(M, K, seed=seed + M, count=synth.n_outliers(K)) for M in (4, 32, 512)}
    qxs = {M: O.quantize_act(x, False) for M, x in xs_host.items()}
    xdev = {M: mq.quantize_act(dev_half(x)) for M, x in xs_host.items()}
    for b in budgets:
        p = preps[b]
        pl = mq.prepare_linear(wt, ct, b)
        assert np.array_equal(pl.row_ptr.cpu().numpy(), p.row_ptr)
        assert np.array_equal(pl.col_idx[: pl.nnzb].cpu().numpy(), p.col_idx)
        for M in (4, 32, 512):
            xq, xs = xdev[M]
            y32 = mq.gemm(xq, xs, M, pl, out_dtype=torch.float32)
            mq.check_device_error()
            ms, ns = rng.integers(0, M, 192), rng.integers(0, N, 192)
            if p.ksel:
                br = int(O.csr_block_rows(p.row_ptr)[rng.integers(0, p.ksel)])
                ns = np.concatenate([ns, np.arange(br * 64, br * 64 + 64)])
                ms = np.concatenate([ms, np.full(64, M - 1)])
            y, a = O.linear_entries(*qxs[M], p, ms, ns)
            check_close(y32.cpu().numpy()[ms, ns], y, a)
            del y32


@pytest.mark.parametrize("lin", synth.LLAMA3_8B, ids=lambda l: l.name)
@pytest.mark.parametrize("M", [4, 32])
def test_llama3_decode_linears_sampled(lin, M):
    _sampled_parity(M, lin, 0.10, "f16", seed=sum(map(ord, lin.name)) + M)


def test_prefill_2048_sampled():
    _sampled_parity(2048, synth.Linear("gate", 4096, 14336), 0.10, "bf16", seed=2)


@pytest.mark.parametrize("M,lin,budget", [(512, synth.QWEN3_32B[6], 0.20), (4, synth.QWEN3_32B[4], 0.05),
                                          (32, synth.QWEN3_32B[3], 0.10)], ids=["down-512", "gate-4", "o-32"])
def test_qwen3_sampled_concentrated(M, lin, budget):
    _sampled_parity(M, lin, budget, "f16", seed=5, conc=True, nsamp=256)


# ----------------------------------------------------------------------------
# failure detection: a bounded device wait that runs out
# ----------------------------------------------------------------------------

def test_bounded_wait_reports_timeout_and_context_survives():
    mq.set_wait_timeout_ns(2_000_000)  # 2 ms
    try:
        mq.debug_wait_timeout()
        with pytest.raises(mq.MQError) as ei:
            mq.check_device_error()
        assert ei.value.status == mq.MQ_ERR_TIMEOUT
    finally:
        mq.set_wait_timeout_ns(1_000_000_000)
    mq.check_device_error()  # cleared
    x, w, xcal = _case(4, 256, 512, 0.1, seed=1)
    pl = mq.prepare_linear(dev_half(w), dev_half(xcal), 0.1)
    y = mq.linear(dev_half(x), pl, out_dtype=torch.float32)
    mq.check_device_error()
    qx, sx = O.quantize_act(x, False)
    yo, a = O.linear(qx, sx, O.prepare(w, xcal, False, 0.1))
    check_close(y.cpu().numpy(), yo, a)
