"""The arithmetic the decode kernel's unpacking rests on, checked on the host
from the E4M3 definition (no GPU):

* a byte 0x00..0x0F read as E4M3 is exactly b * 2^-9 (subnormals below 8, the
  lowest normal binade from 8 to 15);
* masking the nibbles u = q XOR 8 = q + 8 of a packed word into bytes, the even
  codes in one word and the odd ones in the other, and pairing them with the
  activation codes in the same even/odd order, gives 2^-9 * (sum q*x + 8 sum x)
  exactly, so subtracting 2^-9 * 8 * sum x recovers the integer dot;
* every partial sum of a 128-input group is a multiple of 2^-9 below 2^14 in
  magnitude, which fp32 holds exactly."""
import numpy as np
import pytest


def e4m3_value(byte: int) -> float:
    """OCP FP8 E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; S.1111.111 is NaN."""
    s, e, m = byte >> 7, (byte >> 3) & 0xF, byte & 7
    if e == 0xF and m == 7:
        return float("nan")
    mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


def e4m3_of_int(v: int) -> int:
    """The E4M3 byte of a small integer |v| <= 7 (exact)."""
    for b in range(256):
        if e4m3_value(b) == float(v) and not (v == 0 and b != 0):
            return b
    raise ValueError(v)


def pack_word(codes) -> int:
    """Eight signed 4-bit codes, element i in bits 4i .. 4i+3 (two's complement)."""
    w = 0
    for i, q in enumerate(codes):
        w |= (int(q) & 0xF) << (4 * i)
    return w


def bytes_of(word: int):
    return [(word >> (8 * i)) & 0xFF for i in range(4)]


def test_low_bytes_are_exact_multiples_of_2_pow_minus_9():
    for b in range(16):
        assert e4m3_value(b) == b * 2.0 ** -9
    # and nothing else in the positive range is on that grid with step 1
    assert e4m3_value(16) == 16 * 2.0 ** -9 and e4m3_value(17) == 18 * 2.0 ** -9


def unpack_weight_word(p: int):
    u = p ^ 0x88888888
    ev = u & 0x0F0F0F0F
    od = (u >> 4) & 0x0F0F0F0F
    return ev, od


def activation_word_even_odd(codes):
    """E4M3 bytes of the activation codes in the kernels' order: even codes, then odd."""
    lo = [e4m3_of_int(q) for q in codes[0::2]]
    hi = [e4m3_of_int(q) for q in codes[1::2]]
    return lo, hi


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_masked_unpack_gives_the_exact_dot(seed):
    rng = np.random.default_rng(seed)
    qw = rng.integers(-7, 8, size=128)
    qx = rng.integers(-7, 8, size=128)
    measured64 = 0.0
    measured32 = np.float32(0.0)
    for t in range(16):  # 16 words of 8 codes
        w = pack_word(qw[8 * t: 8 * t + 8])
        ev, od = unpack_weight_word(w)
        xe, xo = activation_word_even_odd(qx[8 * t: 8 * t + 8])
        for wb, xb in zip(bytes_of(ev) + bytes_of(od), xe + xo):
            prod = e4m3_value(wb) * e4m3_value(xb)
            measured64 += prod
            measured32 = np.float32(measured32 + np.float32(prod))
    c = 8 * int(qx.sum()) * 2.0 ** -9  # the offset term the kernels subtract
    exact = int(np.dot(qw, qx))
    assert measured64 - c == exact * 2.0 ** -9
    assert float(measured32) == measured64  # fp32 accumulation lost nothing
    assert float(np.float32(measured32) - np.float32(c)) * 512 == exact


def test_extreme_group_stays_exact_in_fp32():
    """All weights +7, all activations +7: the largest measured sum,
    (15 * 7 * 128) * 2^-9 = 26.25, and its correction."""
    qw = np.full(128, 7)
    qx = np.full(128, 7)
    acc = np.float32(0.0)
    for t in range(16):
        ev, od = unpack_weight_word(pack_word(qw[8 * t: 8 * t + 8]))
        xe, xo = activation_word_even_odd(qx[8 * t: 8 * t + 8])
        for wb, xb in zip(bytes_of(ev) + bytes_of(od), xe + xo):
            acc = np.float32(acc + np.float32(e4m3_value(wb) * e4m3_value(xb)))
    assert float(acc) == 15 * 7 * 128 * 2.0 ** -9
    c = np.float32(8 * 7 * 128 * 2.0 ** -9)
    assert float((acc - c) * np.float32(512)) == 6272
