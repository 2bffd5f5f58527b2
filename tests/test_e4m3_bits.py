"""The bit-level E4M3 steps the kernels use, restated in numpy and checked
against the oracle's definition over every finite fp16 value (the keys the
kernels round) and every code (the values they decode) — an exhaustive check
of the arithmetic that the GPU tests sample (Quest page §3, summary dtype).

Rounding, as the append and fused-step kernels do it, for a finite x in fp32:
magnitude a = |x|; below 2^-6 the step is 2^-9 and n = a * 2^9; otherwise,
with 2^e <= a < 2^(e+1) read from the exponent bits, n = a * 2^(3-e) lies in
[8, 16) and the code of the binade's first value is (e + 7) * 8; n is rounded
down for x >= 0 and up for x < 0 (toward -inf), a carry out of the mantissa
landing on the next binade's first code; codes above 0x7e saturate there (an
overflow only when the magnitude was rounded up); a zero code carries no sign.
Rounding toward +inf is minus the rounding of -x.

Decoding for the append's fold: the 7 magnitude bits moved down by one inside
an fp16 word (sign on top) read as the value times 2^-8."""

import numpy as np

from oracle import quest_oracle as qo


def _floor_codes(x):
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x)
    neg = x < 0
    sub = a < np.float32(2.0 ** -6)
    e = ((a.view(np.uint32) >> 23) & 0xFF).astype(np.int64) - 127
    scale = np.where(sub, 0, 130 - e).clip(0, 255).astype(np.uint32) << 23
    n = np.where(sub, a * np.float32(512.0), a * scale.view(np.float32))
    base = np.where(sub, 0, (e + 7) * 8 - 8)
    r = np.where(neg, np.ceil(n), np.floor(n)).astype(np.int64)
    c = base + r
    ovf = (c > 0x7E) & neg
    c = np.minimum(c, 0x7E)
    code = np.where(c == 0, 0, np.where(neg, 0x80 | c, c))
    return code.astype(np.uint8), ovf


def _ceil_codes(x):
    c, ovf = _floor_codes(-np.asarray(x, dtype=np.float32))
    return np.where(c == 0, 0, c ^ 0x80).astype(np.uint8), ovf


def _all_finite_fp16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    h = bits.view(np.float16)
    return h[np.isfinite(h)].astype(np.float32)


def test_floor_and_ceil_match_the_oracle_on_every_fp16_value():
    x = _all_finite_fp16()
    assert len(x) == 63488
    fc, fo = _floor_codes(x)
    cc, co = _ceil_codes(x)
    want_f, want_fo = qo.e4m3_round(x.astype(np.float64), -1)
    want_c, want_co = qo.e4m3_round(x.astype(np.float64), +1)
    assert np.array_equal(fc, want_f)
    assert np.array_equal(cc, want_c)
    assert np.array_equal(fo, want_fo) and np.array_equal(co, want_co)
    assert fo.any() and co.any()               # fp16 reaches beyond 448 both ways


def test_bit_placement_decode_matches_every_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint16)
    placed = codes << 8                          # the code in the high byte of a half
    h = ((placed >> 1) & 0x3F80) | (placed & 0x8000)
    got = h.astype(np.uint16).view(np.float16).astype(np.float64) * 256.0
    want = qo.e4m3_values()[codes]
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))
