"""The fp16 operand encoding of the integer-code GEMV modes (W4A4, W4A8), checked on the CPU.

The register-fragment GEMV multiplies INT4 weight codes by INT4 / INT8 activation codes on fp16
tensor-core MMAs and relies on three facts, restated here in numpy float16 (no GPU):

* a two's complement nibble placed at bits 0..3 of a half and XORed into 1032.0 (0x6408) reads
  1032 + code; at bits 4..7 XORed into 1152.0 (0x6480) it reads 1152 + 16 code; one fp16 subtract
  then leaves code or 16 code exactly;
* with the packed layout of the weights (word t holds channels 8t..8t+7, the even ones in nibbles
  0..3 and the odd ones in nibbles 4..7), the masks 0x000F000F and 0x00F000F0 on the word and on
  the word shifted right by 8 give the channel pairs (0, 1), 16 x (2, 3), (4, 5) and 16 x (6, 7);
* activation codes in [-128, 127] and their sixteenths are exact fp16 values, so every product
  (16 code_w) (code_a / 16) equals code_w code_a, and a 128-channel group sum (at most 131072 in
  magnitude) is exact in an fp32 accumulator.
"""
import numpy as np

import oracle

MAGIC_LO, MAGIC_HI = 0x6408, 0x6480  # fp16 bit patterns of 1032.0 and 1152.0


def as_half(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16)


def code_of(nibble):
    n = np.asarray(nibble, dtype=np.int32)
    return np.where(n >= 8, n - 16, n)


def test_magic_values():
    assert float(as_half(MAGIC_LO)) == 1032.0
    assert float(as_half(MAGIC_HI)) == 1152.0


def test_every_nibble_converts_exactly():
    n = np.arange(16, dtype=np.uint16)
    lo = as_half(n ^ MAGIC_LO) - np.float16(1032.0)          # fp16 subtract, as on the device
    hi = as_half((n << 4) ^ MAGIC_HI) - np.float16(1152.0)
    assert np.array_equal(lo.astype(np.int32), code_of(n))
    assert np.array_equal(hi.astype(np.int32), 16 * code_of(n))


def pair_f16(w, mask, magic):
    """Two fp16 values from one 32-bit word: (w & mask) ^ (magic, magic), minus the magic."""
    v = (w & np.uint32(mask)) ^ np.uint32(magic | (magic << 16))
    halves = np.stack([v & 0xFFFF, v >> 16], axis=-1).astype(np.uint16)
    return (as_half(halves) - as_half(np.uint16(magic))).astype(np.float64)


def test_packed_words_decode_to_channel_pairs():
    rng = np.random.default_rng(7)
    N, K = 16, 256
    codes = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    Wp = oracle.pack_codes(codes)
    assert np.array_equal(oracle.unpack_codes(Wp), codes)
    words = np.ascontiguousarray(Wp).view("<u4")              # [N, K / 8]
    c = codes.astype(np.float64).reshape(N, K // 8, 8)
    w8 = words >> np.uint32(8)
    assert np.array_equal(pair_f16(words, 0x000F000F, MAGIC_LO), c[..., 0:2])
    assert np.array_equal(pair_f16(words, 0x00F000F0, MAGIC_HI), 16 * c[..., 2:4])
    assert np.array_equal(pair_f16(w8, 0x000F000F, MAGIC_LO), c[..., 4:6])
    assert np.array_equal(pair_f16(w8, 0x00F000F0, MAGIC_HI), 16 * c[..., 6:8])


def test_activation_codes_and_sixteenths_are_exact_fp16():
    a = np.arange(-128, 128, dtype=np.float64)
    assert np.array_equal(a.astype(np.float16).astype(np.float64), a)
    assert np.array_equal((a / 16).astype(np.float16).astype(np.float64), a / 16)


def test_products_and_group_sums_are_exact():
    w = np.arange(-8, 8, dtype=np.float64)
    a = np.arange(-128, 128, dtype=np.float64)
    # (16 code_w) * (code_a / 16) in fp16 operands, product formed exactly (as the MMA does)
    prod = (16 * w[:, None]).astype(np.float16).astype(np.float64) * (a[None, :] / 16).astype(np.float16).astype(np.float64)
    assert np.array_equal(prod, w[:, None] * a[None, :])
    # the largest 128-term group sum of W4A8 stays below 2^24: fp32 adds it exactly in any order
    worst = 128 * 8 * 128
    assert worst < 2 ** 24
    terms = np.full(128, -8.0 * -128.0, dtype=np.float32)
    assert float(np.cumsum(terms, dtype=np.float32)[-1]) == float(worst)
