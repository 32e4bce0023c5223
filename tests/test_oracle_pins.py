"""Pins of the oracle against what the definitions and mathematics fix.

Which pin covers which oracle step (each chosen so that a plausible mistake -
a dropped term, a wrong sign or index, a transposed operand - fails one):

  fp16 / bf16 decode       all 65536 bit patterns vs numpy float16 / torch bfloat16
  fp16 / bf16 RNE encode   random + constructed ties vs numpy float16 / torch bfloat16
  scale rule               every finite fp16 and bf16 amax: nearest fp16 to the
                           exact rational amax/7, ties to even, saturation
  Qz codes                 exact-rational nearest-integer property, ties even,
                           |v - s q| <= s/2, |q| <= 7; hand-worked cases
  nibble packing           all 15x15 code pairs round trip; hand-packed bytes
  activation quantizer     per-group consistency on a non-square [M, K]
  base + residual R        W == s*q + R exactly (rationals); |R| <= s/2
  Hessian diagonal         numpy mean of squares; hand value
  Delta-score              numpy einsum over blocks; closed form on constant R
  top-K + CSR              numpy lexsort; brute force over all subsets by true
                           output distortion with an orthogonal calibration set
  residual quant           |R - s_r q_r| <= |R| elementwise (so error can only shrink)
  group dots               closed forms (6272, 0); numpy int64 matmul per group
  linear                   budget 0 == plain W4A4 RTN (numpy float64 matmul);
                           hand-worked linear with and without the residual;
                           monotone diag-H error as the budget grows
"""
import itertools
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
from dense_sparse_int4_gb300 import synth


# ----------------------------------------------------------------------------
# helpers: exact rational properties (not a restatement of the oracle's code)
# ----------------------------------------------------------------------------

def _f16(bits):
    return Fraction(float(np.uint16(bits).view(np.float16)))


def _is_nearest_f16(sbits: int, target: Fraction) -> bool:
    """sbits is a nearest finite fp16 >= 0 to target, ties to an even mantissa."""
    s = _f16(sbits)
    d = abs(s - target)
    for nb in (sbits - 1, sbits + 1):
        if nb < 0 or nb > 0x7BFF:
            continue
        dn = abs(_f16(nb) - target)
        if dn < d:
            return False
        if dn == d and (sbits & 1):
            return False
    return True


def _nearest_int_even(f: Fraction) -> int:
    fl = f.numerator // f.denominator
    rem = f - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


# ----------------------------------------------------------------------------
# formats
# ----------------------------------------------------------------------------

def test_half_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = O.half_to_double(bits)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_bf16_decode_all_patterns():
    import torch
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = O.bf16_to_double(bits)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_half_encode_vs_numpy():
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.standard_normal(200000) * 10.0 ** rng.uniform(-9, 5, 200000),
        # constructed ties: midpoints between adjacent fp16 values
        ((np.arange(0, 0x7BFF, 7, dtype=np.uint16).view(np.float16).astype(np.float64)
          + np.arange(1, 0x7C00, 7, dtype=np.uint16).view(np.float16).astype(np.float64)) / 2),
        np.array([65504.0, 65519.99, 65520.0, 70000.0, 2.0 ** -25, 2.0 ** -26, 3 * 2.0 ** -26, 0.0, -0.0]),
    ])
    v = np.concatenate([v, -v])
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(O.double_to_half(v), ref)


def test_bf16_encode_vs_torch():
    import torch
    rng = np.random.default_rng(2)
    # float32-exact inputs so the library conversion rounds once
    v = (rng.standard_normal(200000) * 10.0 ** rng.uniform(-30, 30, 200000)).astype(np.float32)
    lo = np.arange(0x0000, 0x7F7F, 5, dtype=np.uint32)
    ties = ((lo << 16) | 0x8000).astype(np.uint32).view(np.float32)  # exact bf16 midpoints
    v = np.concatenate([v, ties, -v, -ties]).astype(np.float64)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.double_to_bf16(v), ref)


# ----------------------------------------------------------------------------
# scale rule and Qz
# ----------------------------------------------------------------------------

def test_scale_rule_every_fp16_amax():
    amax_bits = np.arange(0, 0x7C00, dtype=np.uint16)
    amax = amax_bits.view(np.float16).astype(np.float64)
    s = O.scale_from_amax(amax)
    for a_bits, sb in zip(amax_bits, s):
        t = _f16(a_bits) / 7
        assert _is_nearest_f16(int(sb), t), (hex(a_bits), hex(sb))


def test_scale_rule_every_bf16_amax():
    import torch
    amax_bits = np.arange(0, 0x7F80, dtype=np.uint32).astype(np.uint16)
    amax = torch.from_numpy(amax_bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    s = O.scale_from_amax(amax)
    big = Fraction(65520)
    for a, sb in zip(amax, s):
        t = Fraction(float(a)) / 7
        if t >= big:
            assert sb == 0x7BFF
        else:
            assert _is_nearest_f16(int(sb), t), (a, hex(sb))


def test_qz_codes_exact_property():
    rng = np.random.default_rng(3)
    for trial in range(300):
        scale = 10.0 ** rng.uniform(-7, 4)
        v = (rng.standard_normal(128) * scale).astype(np.float16)
        if trial % 3 == 0:  # plant exact ties k + 1/2 relative to the scale
            sb, _ = O.quantize_group(v.astype(np.float64))
            s = float(np.uint16(sb).view(np.float16))
            if s > 0:
                k = rng.integers(-6, 6, 16)
                cand = ((k + 0.5) * s).astype(np.float16)
                ok = (cand.astype(np.float64) == (k + 0.5) * s) & (np.abs(cand.astype(np.float64)) <= np.abs(v.astype(np.float64)).max())
                v[:16][ok] = cand[ok]
        vd = v.astype(np.float64)
        sb, q = O.quantize_group(vd)
        amax = Fraction(float(np.abs(vd).max()))
        assert _is_nearest_f16(sb, amax / 7) or (amax / 7 >= 65520 and sb == 0x7BFF)
        s = _f16(sb)
        assert np.all(np.abs(q) <= 7)
        for x, qq in zip(vd, q):
            if s == 0:
                assert qq == 0
                continue
            want = max(-7, min(7, _nearest_int_even(Fraction(float(x)) / s)))
            assert qq == want
            if abs(Fraction(float(x)) / s) <= 7:
                assert abs(Fraction(float(x)) - s * int(qq)) <= s / 2
        if s >= Fraction(1, 2 ** 14) and amax / 7 < 65504:
            # a normal scale is within 2^-11 of amax/7, so amax/s rounds to the end code
            assert np.abs(q).max() == 7


def test_residual_qz_exact_fraction():
    """The residual codes and scales (float64 inputs R = W^ - Q(W^)) against
    exact rationals: the scale is the fp16 nearest to amax/7 (ties to even),
    every code the integer nearest to r/s (ties to even), clamped to +-7.
    Real residual rows of a packed matrix, and rows with planted exact ties."""
    N, K = 128, 512
    w = synth.weights(N, K, seed=21)
    w = synth.inject_concentrated(w, seed=21, frac=0.25)
    xcal = synth.calibration(K, seed=21, count=4)
    p = O.prepare(w, xcal, False, 0.5)
    assert p.ksel > 0
    rng = np.random.default_rng(5)
    rows = []
    for e in range(p.ksel):  # the selected blocks' rows, as the residual quantizer saw them
        br = int(np.searchsorted(p.row_ptr, e, side="right") - 1)
        g = int(p.col_idx[e])
        for i in rng.choice(64, 4, replace=False):
            rows.append((p.r[br * 64 + i, g * 128:(g + 1) * 128].copy(), (e, int(i))))
    for trial in range(40):  # planted ties: k + 1/2 of the scale, exactly in float64
        v = rng.standard_normal(128) * 10.0 ** rng.uniform(-6, -2)
        sb, _ = O.quantize_group(v)
        sf = float(np.uint16(sb).view(np.float16))
        if sf > 0:
            k = rng.integers(-6, 6, 24)
            cand = (k + 0.5) * sf
            keep = np.abs(cand) <= np.abs(v).max()
            v[:24][keep] = cand[keep]
        rows.append((v, None))
    checked_ties = 0
    for vd, where in rows:
        sb, q = O.quantize_group(vd)
        t = max(abs(Fraction(float(x))) for x in vd) / 7  # amax / 7, exactly
        assert _is_nearest_f16(sb, t) or (t >= 65520 and sb == 0x7BFF)
        s = _f16(sb)
        for x, qq in zip(vd, q):
            if s == 0:
                assert qq == 0
                continue
            quo = Fraction(float(x)) / s
            want = max(-7, min(7, _nearest_int_even(quo)))
            assert qq == want, (x, float(s), int(qq), want)
            checked_ties += (quo - (quo.numerator // quo.denominator)) == Fraction(1, 2)
        if where is not None:  # the packed residual holds exactly these codes and this scale
            e, i = where
            assert np.array_equal(p.qr[e, i], q) and p.sr[e, i] == sb
    assert checked_ties > 50


def _read_cases(path):
    cases, cur = [], None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *rest = line.split()
        if key == "case":
            cur = {"name": rest[0], "dtype": rest[1]}
            cases.append(cur)
        else:
            cur[key] = rest
    return cases


def test_qz_hand_worked(golden_dir):
    for c in _read_cases(os.path.join(golden_dir, "qz_worked.txt")):
        v = np.zeros(128, np.float64)
        vals = np.array([float(t) for t in c["v"]])
        v[: vals.size] = vals
        bits = synth.to_bits(v.astype(np.float32), c["dtype"])
        vd = O.to_double(bits, c["dtype"] == "bf16")
        assert np.array_equal(vd[: vals.size], vals), c["name"]  # inputs are exact
        sb, q = O.quantize_group(vd)
        assert sb == int(c["s"][0], 16), (c["name"], hex(sb))
        assert q[: vals.size].tolist() == [int(t) for t in c["q"]], c["name"]
        assert not q[vals.size:].any()


def test_nibble_packing():
    codes = np.array(list(itertools.product(range(-7, 8), repeat=2)), np.int8).reshape(1, -1)
    packed = O.pack_nibbles(codes)
    assert np.array_equal(O.unpack_nibbles(packed), codes)
    # hand-packed: (lo, hi) -> byte
    for lo, hi, byte in [(0, 0, 0x00), (-1, 7, 0x7F), (1, -1, 0xF1), (-7, 3, 0x39), (7, -7, 0x97)]:
        assert O.pack_nibbles(np.array([[lo, hi]], np.int8))[0, 0] == byte


def test_quantize_act_groups_and_layout():
    M, K = 3, 384  # non-square, three groups
    x = synth.activations(M, K, seed=5, count=4)
    q, s = O.quantize_act(x, False)
    assert q.shape == (M, K) and s.shape == (M, K // 128)
    xd = O.half_to_double(x)
    for m in range(M):
        for g in range(K // 128):
            sb, qq = O.quantize_group(xd[m, g * 128:(g + 1) * 128])
            assert s[m, g] == sb and np.array_equal(q[m, g * 128:(g + 1) * 128], qq)
    # the outlier channels dominate their groups' scales: averaged over tokens,
    # groups that hold one have a scale far above the N(0,1) groups
    M = 32
    x = synth.activations(M, K, seed=5, count=4)
    _, s = O.quantize_act(x, False)
    ch = synth.outlier_channels(K, 4, 5)
    s_mean = O.half_to_double(s).mean(axis=0)
    for g in range(K // 128):
        has = np.any((ch >= g * 128) & (ch < (g + 1) * 128))
        assert (s_mean[g] > 2.0 if has else s_mean[g] < 1.0)


# ----------------------------------------------------------------------------
# base, residual, Hessian, Delta, top-K
# ----------------------------------------------------------------------------

def test_base_residual_exact():
    N, K = 64, 256
    w = synth.weights(N, K, seed=7)
    qw, sw, r = O.base_quant(w)
    wd = O.half_to_double(w)
    sd = O.half_to_double(sw)
    rng = np.random.default_rng(0)
    for _ in range(2000):
        n, k = rng.integers(0, N), rng.integers(0, K)
        s = Fraction(float(sd[n, k // 128]))
        assert Fraction(float(wd[n, k])) == s * int(qw[n, k]) + Fraction(float(r[n, k]))
        assert abs(Fraction(float(r[n, k]))) <= s / 2
    assert np.all(np.abs(qw) <= 7)


def test_hessian_diag():
    C, K = 256, 256
    x = synth.calibration(K, seed=3, count=4, C=C)
    h = O.hessian_diag(x, False)
    ref = np.mean(O.half_to_double(x) ** 2, axis=0)
    assert np.allclose(h, ref, rtol=1e-14, atol=0)
    # hand value: rows (1, 2) and (3, 4) -> h = ((1+9)/2, (4+16)/2)
    xx = np.array([[1.0, 2.0], [3.0, 4.0]], np.float16).view(np.uint16)
    assert O.hessian_diag(xx, False).tolist() == [5.0, 10.0]
    assert O.hessian_diag(synth.f32_to_bf16_bits(np.array([[1.0, 2.0], [3.0, 4.0]], np.float32)), True).tolist() == [5.0, 10.0]


def test_delta_scores_vs_einsum_and_closed_form():
    N, K = 192, 384
    rng = np.random.default_rng(11)
    r = rng.standard_normal((N, K)) * 1e-3
    h = rng.uniform(0.1, 5.0, K)
    d = O.delta_scores(r, h)
    ref = np.einsum("bnGk,Gk->bG", (r ** 2).reshape(N // 64, 64, K // 128, 128), h.reshape(K // 128, 128))
    assert np.allclose(d, ref.ravel(), rtol=1e-13, atol=0)
    # closed form: R = c in one block only, h = 1 -> Delta = 64*128*c^2 there, 0 elsewhere
    r = np.zeros((N, K))
    r[64:128, 256:384] = 2.0 ** -10
    d = O.delta_scores(r, np.ones(K))
    expect = np.zeros((N // 64) * (K // 128))
    expect[1 * 3 + 2] = 64 * 128 * 2.0 ** -20
    assert np.array_equal(d, expect)


def test_num_selected_table(golden_dir):
    for line in open(os.path.join(golden_dir, "num_selected.txt")):
        if line.startswith("#") or not line.strip():
            continue
        N, K, b, want = line.split()
        assert O.num_selected(int(N), int(K), float(b)) == int(want), line


def test_select_topk_vs_lexsort():
    N, K = 640, 1280
    rng = np.random.default_rng(5)
    nb = (N // 64) * (K // 128)
    delta = rng.uniform(0, 1, nb)
    delta[rng.integers(0, nb, 20)] = 0.5  # ties: lower block index first
    for ksel in (0, 1, 7, 50, nb):
        rp, ci = O.select_topk(delta, N, K, ksel)
        order = np.lexsort((np.arange(nb), -delta))[:ksel]
        chosen = np.zeros(nb, bool)
        chosen[order] = True
        G = K // 128
        want_rp = np.concatenate([[0], np.cumsum(chosen.reshape(N // 64, G).sum(1))])
        want_ci = np.concatenate([np.nonzero(chosen.reshape(N // 64, G)[br])[0] for br in range(N // 64)])
        assert np.array_equal(rp, want_rp) and np.array_equal(ci, want_ci)


def test_topk_equals_brute_force_distortion_orthogonal_calibration():
    """With an orthogonal calibration set (Xcal^T Xcal diagonal) the true output
    distortion ||Xcal (R - R_S)^T||^2 is C * sum of Delta over unselected blocks,
    so the Delta top-K set is exactly the brute-force minimiser."""
    N, K = 128, 512  # 2 block rows x 4 groups = 8 blocks
    w = synth.weights(N, K, seed=9)
    w = synth.inject_concentrated(w, seed=9, frac=0.25)
    rng = np.random.default_rng(9)
    d = rng.choice(np.array([0.25, 0.5, 1.0, 2.0, 4.0]), K)  # distinct channel scales
    xcal = np.diag(d).astype(np.float16).view(np.uint16)  # C = K rows, orthogonal columns
    _, _, r = O.base_quant(w)
    h = O.hessian_diag(xcal, False)
    delta = O.delta_scores(r, h)
    xc = O.half_to_double(xcal)
    G, nb = K // 128, 8

    def distortion(S):
        rs = r.copy()
        for b in S:
            br, g = divmod(b, G)
            rs[br * 64:(br + 1) * 64, g * 128:(g + 1) * 128] = 0.0
        return float(np.sum((xc @ rs.T) ** 2))

    for ksel in range(0, 4):
        best = min(itertools.combinations(range(nb), ksel), key=lambda S: (round(distortion(S), 30), S))
        rp, ci = O.select_topk(delta, N, K, ksel)
        got = sorted(int(br) * G + int(g) for br, g in zip(O.csr_block_rows(rp), ci))
        assert np.isclose(distortion(got), distortion(best), rtol=1e-12), (ksel, got, best)


def test_topk_near_brute_force_random_calibration():
    """Random calibration: Delta top-K is an approximation; report how close."""
    N, K = 128, 512
    w = synth.inject_concentrated(synth.weights(N, K, seed=4), seed=4, frac=0.25)
    xcal = synth.calibration(K, seed=4, count=4, C=256)
    _, _, r = O.base_quant(w)
    delta = O.delta_scores(r, O.hessian_diag(xcal, False))
    xc = O.half_to_double(xcal)
    G = K // 128

    def distortion(S):
        rs = r.copy()
        for b in S:
            br, g = divmod(b, G)
            rs[br * 64:(br + 1) * 64, g * 128:(g + 1) * 128] = 0.0
        return float(np.sum((xc @ rs.T) ** 2))

    for ksel in (1, 2, 3):
        best = min(distortion(S) for S in itertools.combinations(range(8), ksel))
        rp, ci = O.select_topk(delta, N, K, ksel)
        got = [int(br) * G + int(g) for br, g in zip(O.csr_block_rows(rp), ci)]
        assert distortion(got) <= best * 1.05


# ----------------------------------------------------------------------------
# residual quant, dots, linear
# ----------------------------------------------------------------------------

def test_residual_quant_never_grows_error():
    N, K = 256, 512
    w = synth.inject_concentrated(synth.weights(N, K, seed=12), seed=12, frac=0.1)
    xcal = synth.calibration(K, seed=12, count=4)
    p = O.prepare(w, xcal, False, 0.5)
    assert p.ksel == 8
    brs = O.csr_block_rows(p.row_ptr)
    for i, (br, g) in enumerate(zip(brs, p.col_idx)):
        R = p.r[br * 64:(br + 1) * 64, g * 128:(g + 1) * 128]
        s = O.half_to_double(p.sr[i])[:, None]
        err = R - s * p.qr[i]
        assert np.all(np.abs(err) <= np.abs(R))
        for rr in range(64):  # per-row scale follows the scale rule
            sb, q = O.quantize_group(R[rr])
            assert sb == p.sr[i, rr] and np.array_equal(q, p.qr[i, rr])


def test_group_dots_closed_forms_and_matmul():
    qx = np.full((2, 256), 7, np.int8)
    qw = np.full((3, 256), 7, np.int8)
    assert np.all(O.group_dots(qx, qw) == 6272)
    qw[:, 1::2] = -7
    assert np.all(O.group_dots(qx, qw) == 0)
    rng = np.random.default_rng(6)
    qx = rng.integers(-7, 8, (5, 384)).astype(np.int8)
    qw = rng.integers(-7, 8, (3, 384)).astype(np.int8)
    d = O.group_dots(qx, qw)
    for g in range(3):
        ref = qx[:, g * 128:(g + 1) * 128].astype(np.int64) @ qw[:, g * 128:(g + 1) * 128].astype(np.int64).T
        assert np.array_equal(d[:, :, g], ref)
    qr = rng.integers(-7, 8, (2, 64, 128)).astype(np.int8)
    ci = np.array([2, 0], np.int32)
    dr = O.residual_dots(qx, qr, ci)
    for i, g in enumerate(ci):
        assert np.array_equal(dr[:, i, :], qx[:, g * 128:(g + 1) * 128].astype(np.int64) @ qr[i].astype(np.int64).T)


def _cfg0(budget):
    x = synth.activations(4, 512, seed=0, count=4)
    w = synth.weights(512, 512, seed=0)
    xcal = synth.calibration(512, seed=0, count=4)
    qx, sx = O.quantize_act(x, False)
    return qx, sx, O.prepare(w, xcal, False, budget)


def test_budget_zero_is_plain_rtn():
    qx, sx, p = _cfg0(0.0)
    assert p.ksel == 0 and p.row_ptr.sum() == 0
    y, a = O.linear(qx, sx, p)
    G = 512 // 128
    xd = (qx.reshape(4, G, 128) * O.half_to_double(sx)[:, :, None]).reshape(4, 512)
    wd = (p.qw.reshape(512, G, 128) * O.half_to_double(p.sw)[:, :, None]).reshape(512, 512)
    ref = xd @ wd.T  # dequantize, then one float64 matmul
    assert np.all(np.abs(y - ref) <= 1e-12 * a)


def test_budget_ten_percent_cfg0_and_residual_term():
    qx, sx, p = _cfg0(0.10)
    assert p.ksel == 3  # top-3 of 32 blocks
    y, a = O.linear(qx, sx, p)
    y0, _ = O.linear(qx, sx, _cfg0(0.0)[2])
    G = 4
    xd = (qx.reshape(4, G, 128) * O.half_to_double(sx)[:, :, None]).reshape(4, 512)
    rhat = np.zeros((512, 512))
    for i, (br, g) in enumerate(zip(O.csr_block_rows(p.row_ptr), p.col_idx)):
        rhat[br * 64:(br + 1) * 64, g * 128:(g + 1) * 128] = O.half_to_double(p.sr[i])[:, None] * p.qr[i]
    assert np.all(np.abs((y - y0) - xd @ rhat.T) <= 1e-12 * a)
    # only rows of selected block rows move
    moved = np.any(y != y0, axis=0)
    sel_rows = np.zeros(512, bool)
    for br in O.csr_block_rows(p.row_ptr):
        sel_rows[br * 64:(br + 1) * 64] = True
    assert not np.any(moved & ~sel_rows)


def test_linear_hand_worked(golden_dir):
    kv = {}
    for line in open(os.path.join(golden_dir, "linear_worked.txt")):
        if line.startswith("#") or not line.strip():
            continue
        k, v = line.split(maxsplit=1)
        kv[k] = v.strip()
    M, N, K = int(kv["M"]), int(kv["N"]), int(kv["K"])
    x = np.full((M, K), float(kv["x"]), np.float16).view(np.uint16)
    w = np.full((N, K), float(kv["w"]), np.float16).view(np.uint16)
    xcal = np.full((int(kv["xcal_rows"]), K), float(kv["xcal"]), np.float16).view(np.uint16)
    qx, sx = O.quantize_act(x, False)
    assert np.all(sx == int(kv["sx"], 16))
    for budget, key in ((0.0, "y_budget0"), (1.0, "y_budget1")):
        p = O.prepare(w, xcal, False, budget)
        assert np.all(p.sw == int(kv["sw"], 16))
        assert np.all(p.r == float(kv["R"]))
        assert p.delta.tolist() == [float(kv["delta"])]
        if budget:
            assert np.all(p.sr == int(kv["sr"], 16)) and np.all(p.qr == int(kv["qr"]))
        assert np.all(O.group_dots(qx, p.qw) == int(kv["dw"]))
        y, _ = O.linear(qx, sx, p)
        assert np.all(y == float(Fraction(kv[key])))


def test_error_monotone_in_budget():
    """Diag-H weighted weight error sum_k h_k sum_n (R - Rhat)^2 never grows with the budget."""
    N, K = 256, 512
    w = synth.inject_concentrated(synth.weights(N, K, seed=21), seed=21, frac=0.1)
    xcal = synth.calibration(K, seed=21, count=4)
    prev = None
    G = K // 128
    for budget in np.linspace(0, 1, 11):
        p = O.prepare(w, xcal, False, budget)
        err = p.r.copy()
        for i, (br, g) in enumerate(zip(O.csr_block_rows(p.row_ptr), p.col_idx)):
            blk = (slice(br * 64, (br + 1) * 64), slice(g * 128, (g + 1) * 128))
            err[blk] = p.r[blk] - O.half_to_double(p.sr[i])[:, None] * p.qr[i]
        per_block = [float(np.sum(p.h[g * 128:(g + 1) * 128] * err[br * 64:(br + 1) * 64, g * 128:(g + 1) * 128] ** 2))
                     for br in range(N // 64) for g in range(G)]
        total = 0.0
        for e in per_block:  # fixed summation order across budgets
            total += e
        if prev is not None:
            assert total <= prev
        prev = total
