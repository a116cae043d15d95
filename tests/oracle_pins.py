"""Pins that tie the CPU oracle to facts fixed by the pages and by mathematics.

Each ``check_*`` function takes an oracle module (the real one, or a copy with a planted mistake)
and raises AssertionError when the oracle disagrees with a pinned fact.  The expected values come
from the pages' worked examples (tests/golden/), closed forms, hand-worked quantiser cases, brute
force on tiny inputs and mathematical bounds -- never from the oracle's own formulas retyped.
"""
from __future__ import annotations

import json
import os
from itertools import product

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "sd_tutorial_examples.json")


def golden():
    with open(GOLDEN, encoding="utf-8") as f:
        return json.load(f)


def bf16_bits(values):
    """Bit patterns of values that are exactly representable in bf16 (checked)."""
    v = np.asarray(values, dtype=np.float32)
    bits = (v.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    back = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    assert np.array_equal(back, v), "test value not exactly representable in bf16"
    return bits


# ---------------------------------------------------------------- bf16 rounding of fp64 results
#
# Every expected W4A4 / W4A8 output and every toy-model layer output is the fp64 result rounded to
# bf16 once (round to nearest, ties to even).  bf16 has 7 stored mantissa bits and fp32's exponent
# range: the spacing is 2^-7 on [1, 2), the largest finite value is (2 - 2^-7) * 2^127 (0x7F7F),
# the smallest subnormal 2^-133 (0x0001).  The expected bit patterns below are worked by hand from
# those facts.

def check_bf16_rounding(o):
    cases = [
        (1.0 + 2.0 ** -8, 0x3F80),                    # halfway between 1 and 1 + 2^-7: even mantissa 0
        (1.0 + 3 * 2.0 ** -8, 0x3F82),                # halfway between mantissas 1 and 2: up to 2
        (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),       # just above the tie (fp32 would round it to the tie)
        (1.0 + 2.0 ** -8 - 2.0 ** -40, 0x3F80),       # just below the tie
        (-(1.0 + 2.0 ** -8), 0xBF80),                 # the tie rule is symmetric in sign
        (-(1.0 + 3 * 2.0 ** -8), 0xBF82),
        ((2.0 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),     # the largest finite bf16 is kept
        ((2.0 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),     # halfway to 2^128: odd mantissa 0x7F rounds up to inf
        ((2.0 - 2.0 ** -8) * 2.0 ** 127 - 2.0 ** 100, 0x7F7F),  # just below that: the largest finite
        (-(2.0 - 2.0 ** -8) * 2.0 ** 127, 0xFF80),
        (2.0 ** -133, 0x0001),                        # smallest subnormal
        (2.0 ** -134, 0x0000),                        # halfway between 0 and 2^-133: to 0 (even)
        (3 * 2.0 ** -134, 0x0002),                    # halfway between 1 and 2 subnormal steps: to 2
        (2.0 ** -134 + 2.0 ** -160, 0x0001),          # just above the subnormal tie
        (-(2.0 ** -134), 0x8000),                     # a negative tie to zero keeps the sign
        (2.0 ** -126 - 2.0 ** -134, 0x0080),          # halfway between 127 and 128 steps: the smallest normal
        (1.5 * 2.0 ** -126 + 2.0 ** -134, 0x00C0),    # normal range at the bottom exponent: spacing 2^-133
        (-0.0, 0x8000), (0.0, 0x0000), (np.inf, 0x7F80), (-np.inf, 0xFF80),
        (3.0, 0x4040), (-2.0 ** 40, 0xD380), (1.0 / 3.0, 0x3EAB),  # 1/3 = 0x3EAAAAAB in fp32: up to 0x3EAB
    ]
    x = np.array([c[0] for c in cases], dtype=np.float64)
    want = np.array([c[1] for c in cases], dtype=np.uint16)
    got = np.asarray(o.f64_to_bf16_bits(x), dtype=np.uint16)
    for xi, w, g in zip(x, want, got):
        assert w == g, f"bf16({xi!r}) = {int(g):#06x}, expected {int(w):#06x}"
    vals = np.asarray(o.f64_to_bf16_value(x), dtype=np.float64)
    back = (want.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    assert np.array_equal(np.signbit(vals), np.signbit(back)) and np.array_equal(vals, back)

    # values that are fp32 numbers: the textbook integer rounding of the fp32 bit pattern (add
    # 0x7FFF plus the lowest kept bit, drop 16 bits) over random normal, subnormal and tie patterns
    rng = np.random.default_rng(5)
    u = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    u[:2000] &= np.uint32(0x807FFFFF)                 # subnormal fp32 inputs
    u[2000:4000] = (u[2000:4000] & np.uint32(0xFFFF0000)) | np.uint32(0x8000)  # exact ties
    f = u.view(np.float32)
    keep = np.isfinite(f) & (np.abs(f.astype(np.float64)) < (2.0 - 2.0 ** -8) * 2.0 ** 127)
    u, f = u[keep], f[keep]
    ref = ((u.astype(np.uint64) + 0x7FFF + ((u.astype(np.uint64) >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(np.asarray(o.f64_to_bf16_bits(f.astype(np.float64)), dtype=np.uint16), ref)


# ---------------------------------------------------------------- a1: weight quantiser / packer

def check_pack_layout(o):
    # little-endian word t holds k = 8t+0,2,4,6 in nibbles 0..3 and k = 8t+1,3,5,7 in nibbles
    # 4..7, two's complement: k0..k7 = 1,-2,7,-8,0,-1,3,4 give nibbles 1,7,0,3,E,8,F,4
    codes = np.array([[1, -2, 7, -8, 0, -1, 3, 4]], dtype=np.int8)
    assert o.pack_codes(codes).tolist() == [[0x71, 0x30, 0x8E, 0x4F]]
    word = int.from_bytes(bytes(o.pack_codes(codes)[0]), "little")
    assert [(word >> (4 * i)) & 0xF for i in range(8)] == [0x1, 0x7, 0x0, 0x3, 0xE, 0x8, 0xF, 0x4]
    # every byte value round-trips through unpack / pack
    allb = np.arange(256, dtype=np.uint8).reshape(1, 256)
    c = o.unpack_codes(allb)
    assert c.min() == -8 and c.max() == 7
    # byte 0x9F = 159 is byte 3 of word 39: nibble 6 (F = -1) is k = 312 + 5, nibble 7 (9 = -7) k = 312 + 7
    assert c[0, 317] == -1 and c[0, 319] == -7
    assert np.array_equal(o.pack_codes(c), allb)
    # one code at every position of a word lands in the nibble the layout names
    for k in range(8):
        one = np.zeros((1, 8), dtype=np.int8)
        one[0, k] = 5
        w = int.from_bytes(bytes(o.pack_codes(one)[0]), "little")
        slot = (0, 4, 1, 5, 2, 6, 3, 7)[k]
        assert w == 5 << (4 * slot)


def check_weight_grid_roundtrip(o):
    # W exactly on the grid code * s with s a power of two and +-7 present: codes and scales recovered
    rng = np.random.default_rng(11)
    N, K = 6, 512
    G = K // 128
    s = 2.0 ** rng.integers(-12, -2, size=(N, G))
    c = rng.integers(-7, 8, size=(N, K))
    for n in range(N):
        for g in range(G):
            c[n, g * 128] = 7 if (n + g) % 2 else -7
    c[0, 0:15] = np.arange(-7, 8)  # every producible code
    W = (c * np.repeat(s, 128, axis=1)).astype(np.float32)
    codes, S = o.quantize_weights(bf16_bits(W))
    assert S.dtype == np.float16
    assert np.array_equal(S.astype(np.float64), s)
    assert np.array_equal(codes.astype(np.int64), c)


def check_weight_hand_cases(o):
    def quant(group_values):
        row = np.zeros(128, dtype=np.float32)
        row[: len(group_values)] = group_values
        codes, S = o.quantize_weights(bf16_bits(row[None, :]))
        return codes[0, : len(group_values)].tolist(), float(S[0, 0])

    # amax 7 -> s = 1: ties go to even, 5 stays 5 (a divisor of 8 would give 6)
    codes, s = quant([7.0, 2.5, 3.5, -2.5, 5.0, 0.5, 1.5, -7.0, -0.5])
    assert s == 1.0
    assert codes == [7, 2, 4, -2, 5, 0, 2, -7, 0]
    # amax 1: fp16(1/7) = 0.142822265625; 0.5 / that = 3.5008... -> 4.  (The fp32 scale 1/7 would
    # give 0.5 / 0.14285715 = 3.4999998 -> 3: the scale must be rounded to fp16 first.)
    codes, s = quant([1.0, 0.5, -0.5])
    assert s == 0.142822265625
    assert codes == [7, 4, -4]
    # fp16-subnormal scale: amax = 7 * 2^-20 -> s = 2^-20 (subnormal in fp16, exact)
    t = 2.0 ** -20
    codes, s = quant([7 * t, 3 * t, -5 * t])
    assert s == t and codes == [7, 3, -5]
    # scale underflows to 0 in fp16 (2^-26 < half the smallest subnormal) -> all codes 0
    t = 2.0 ** -26
    codes, s = quant([7 * t, 3 * t])
    assert s == 0.0 and codes == [0, 0]
    # all-zero group
    codes, s = quant([0.0, 0.0])
    assert s == 0.0 and codes == [0, 0]


def check_pack_end_to_end(o):
    # pack_weights = quantise + nibble layout, on a hand case
    row = np.zeros((1, 128), dtype=np.float32)
    row[0, :4] = [7.0, -1.0, 2.0, -7.0]
    Wp, S = o.pack_weights(bf16_bits(row))
    assert Wp.shape == (1, 64) and S.shape == (1, 1)
    # codes 7, -1, 2, -7: word 0 nibbles (k0, k2, k4, k6, k1, k3, k5, k7) = 7, 2, 0, 0, F, 9, 0, 0
    assert Wp[0, :4].tolist() == [0x27, 0x00, 0x9F, 0x00] and float(S[0, 0]) == 1.0


# ---------------------------------------------------------------- a2: W4A16

def check_w4a16_onehot_and_grid(o):
    rng = np.random.default_rng(5)
    N, K = 40, 256
    s = 2.0 ** rng.integers(-8, -3, size=(N, K // 128))
    c = rng.integers(-7, 8, size=(N, K))
    c[:, 0] = 7
    c[:, 128] = -7
    W = (c * np.repeat(s, 128, axis=1)).astype(np.float32)
    Wp, S = o.pack_weights(bf16_bits(W))
    # one-hot activations select one input column of W (exactly)
    for k in [0, 1, 77, 128, 200, 255]:
        x = np.zeros((1, K), dtype=np.float32)
        x[0, k] = 1.0
        y = o.linear_w4a16(bf16_bits(x), Wp, S)
        assert y.shape == (1, N)
        assert np.array_equal(y[0], W[:, k].astype(np.float64))
    # on-grid weights: the W4A16 product equals the plain product with W
    x = rng.integers(-64, 64, size=(3, K)).astype(np.float32) / 16
    y = o.linear_w4a16(bf16_bits(x), Wp, S)
    ref = x.astype(np.float64) @ W.astype(np.float64).T
    assert np.allclose(y, ref, rtol=0, atol=1e-12)
    # a subset of output rows
    rows = np.array([3, 17, 39])
    assert np.allclose(o.linear_w4a16(bf16_bits(x), Wp, S, rows=rows), ref[:, rows], rtol=0, atol=1e-12)


def check_w4a16_error_bound(o):
    # |y - x W^T| <= sum_k |x_k| * s_{n,g(k)} / 2  (each weight moves at most half a step)
    rng = np.random.default_rng(6)
    N, K, M = 24, 384, 4
    Wf = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    Wb = bf16_bits((Wf.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32))
    Wv = (Wb.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    xf = rng.standard_normal((M, K)).astype(np.float32)
    xb = bf16_bits((xf.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32))
    xv = (xb.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    Wp, S = o.pack_weights(Wb)
    y = o.linear_w4a16(xb, Wp, S)
    exact = xv @ Wv.T
    s_full = np.repeat(S.astype(np.float64), 128, axis=1)        # [N, K]
    # the half-step bound uses the fp16-rounded scale; amax/fp16(amax/7) can exceed 7 by a rounding
    # margin, so allow the clamp's extra fraction of a step for the largest weights
    bound = np.abs(xv) @ (s_full * 0.5 * (1 + 2.0 ** -9)).T + 1e-12
    assert np.all(np.abs(y - exact) <= bound)
    # and the bound is not vacuous: the error is a small fraction of the output scale
    assert np.linalg.norm(y - exact) < 0.2 * np.linalg.norm(exact)


# ---------------------------------------------------------------- a3: activation quantiser

def check_act_quant_hand_cases(o):
    x = np.zeros((3, 128), dtype=np.float32)
    x[0, :8] = [7.0, 3.5, -3.5, 2.5, 0.0, -7.0, 0.5, 1.5]
    x[1, :3] = [1.0, 0.5, -0.5]           # fp32 scale 1/7: 0.5 / 0.14285715 = 3.4999998 -> 3
    qa, s_a = o.quantize_activations(bf16_bits(x))
    assert s_a.dtype == np.float32
    assert s_a[0] == 1.0
    assert qa[0, :8].tolist() == [7, 4, -4, 2, 0, -7, 0, 2]
    assert s_a[1] == np.float32(1.0) / np.float32(7.0)
    assert qa[1, :3].tolist() == [7, 3, -3]
    assert s_a[2] == 0.0 and not qa[2].any()       # all-zero token
    # an outlier channel takes the scale: codes +-7 there, everything below s/2 rounds to 0
    y = np.zeros((1, 256), dtype=np.float32)
    y[0, 10] = -140.0
    y[0, 20:30] = 9.0
    y[0, 30:40] = 11.0
    qa, s_a = o.quantize_activations(bf16_bits(y))
    assert s_a[0] == 20.0 and qa[0, 10] == -7
    assert not qa[0, 20:30].any() and (qa[0, 30:40] == 1).all()


# ---------------------------------------------------------------- a4: W4A4

def check_w4a4_bruteforce(o):
    rng = np.random.default_rng(7)
    M, N, K = 3, 5, 256
    x = rng.integers(-40, 41, size=(M, K)).astype(np.float32) / 4
    W = rng.integers(-7, 8, size=(N, K)).astype(np.float32) / 64
    W[:, 0] = 7 / 64
    W[:, 128] = -7 / 64
    Wp, S = o.pack_weights(bf16_bits(W))
    r = o.linear_w4a4(bf16_bits(x), Wp, S)
    qa, s_a = r["qa"], r["s_a"]
    wc = np.rint(W * 64).astype(np.int64)          # on-grid weights: codes are W * 64
    for m in range(M):
        for n in range(N):
            for g in range(2):
                total = 0
                for k in range(128 * g, 128 * g + 128):
                    total += int(qa[m, k]) * int(wc[n, k])
                assert r["acc"][m, n, g] == total
    assert r["acc"].dtype == np.int32
    # y equals the plain fp64 product of the dequantised activations and dequantised weights
    xa = qa.astype(np.float64) * s_a.astype(np.float64)[:, None]
    ref = xa @ o.dequantize_weights(Wp, S).T
    assert np.allclose(r["y"], ref, rtol=1e-12, atol=0)


def check_w4a4_extremes(o):
    # every pair of the 16 codes, including -8 which the packer never produces but kernels accept
    ca = np.repeat(np.arange(-8, 8), 16)             # [256]
    cw = np.tile(np.arange(-8, 8), 16)
    Wp = o.pack_codes(cw[None, :].astype(np.int8))
    acc = o.w4a4_group_sums(ca[None, :].astype(np.int8), Wp)
    # sum over all pairs of (a * w) for a, w in [-8, 7]: (sum a)(sum w) split per group of 128
    # group 0 holds a in [-8, -1], group 1 holds a in [0, 7]; each with the full w range (sum -8)
    assert acc.shape == (1, 1, 2)
    assert acc[0, 0, 0] == 288     # (sum_{a=-8..-1} a) * (sum_{w=-8..7} w) = (-36) * (-8)
    assert acc[0, 0, 1] == -224    # (sum_{a=0..7} a) * (sum_{w=-8..7} w) = 28 * (-8)
    # largest magnitude group: 128 products of (-8)(-8)
    big = o.w4a4_group_sums(np.full((1, 128), -8, np.int8), o.pack_codes(np.full((1, 128), -8, np.int8)))
    assert big[0, 0, 0] == 8192


def check_w4a4_constant_activation(o):
    # x constant c > 0: s_a = c / 7 and every code is 7, so y = c * sum_k w_k (on-grid weights)
    rng = np.random.default_rng(8)
    N, K = 7, 256
    W = rng.integers(-7, 8, size=(N, K)).astype(np.float32) / 32
    W[:, 0] = 7 / 32
    W[:, 128] = -7 / 32
    Wp, S = o.pack_weights(bf16_bits(W))
    x = np.full((2, K), 3.5, dtype=np.float32)
    r = o.linear_w4a4(bf16_bits(x), Wp, S)
    assert (r["qa"] == 7).all()
    assert np.allclose(r["y"][0], 3.5 * W.astype(np.float64).sum(axis=1), rtol=1e-6, atol=1e-9)


# ---------------------------------------------------------------- f3: W4A8

def check_w4a8_quantiser(o):
    # amax 127 gives s_a = 1: codes are the rounded values (ties to even), +-127 at +-amax
    x = np.zeros((3, 128), dtype=np.float32)
    x[0, :8] = [127.0, 2.5, 3.5, -2.5, -127.0, 0.5, 1.5, 100.0]
    x[1, :2] = [1.0, 0.5]            # s_a = 1/127 in fp32; 0.5 / s_a = 63.5 (fp32) -> 64 (even)
    qa, s_a = o.quantize_activations(bf16_bits(x), bits=8)
    assert s_a[0] == 1.0 and qa[0, :8].tolist() == [127, 2, 4, -2, -127, 0, 2, 100]
    assert s_a[1] == np.float32(1.0) / np.float32(127.0)
    q = np.float32(0.5) / s_a[1]
    assert q == np.float32(63.5) and qa[1, 0] == 127 and qa[1, 1] == 64
    assert s_a[2] == 0.0 and not qa[2].any()
    # the 4-bit quantiser is the same rule with divisor 7
    qa4, s4 = o.quantize_activations(bf16_bits(x), bits=4)
    assert s4[0] == np.float32(127.0) / np.float32(7.0) and qa4[0, 0] == 7


def check_w4a8_linear(o):
    rng = np.random.default_rng(9)
    M, N, K = 3, 6, 256
    x = rng.integers(-40, 41, size=(M, K)).astype(np.float32) / 4
    W = rng.integers(-7, 8, size=(N, K)).astype(np.float32) / 64
    W[:, 0] = 7 / 64
    W[:, 128] = -7 / 64
    Wp, S = o.pack_weights(bf16_bits(W))
    r = o.linear_w4a8(bf16_bits(x), Wp, S)
    qa, s_a = r["qa"], r["s_a"]
    assert int(np.abs(qa).max()) == 127
    wc = np.rint(W * 64).astype(np.int64)
    for m in range(M):
        for n in range(N):
            for g in range(2):
                sl = slice(128 * g, 128 * g + 128)
                assert r["acc"][m, n, g] == int(np.dot(qa[m, sl].astype(np.int64), wc[n, sl]))
    xa = qa.astype(np.float64) * s_a.astype(np.float64)[:, None]
    assert np.allclose(r["y"], xa @ o.dequantize_weights(Wp, S).T, rtol=1e-12, atol=0)
    # 8-bit activations track the 16-bit product far more closely than 4-bit ones
    xs = rng.standard_normal((4, 1024)).astype(np.float32)
    xs[:, ::97] *= 20
    W2 = (rng.standard_normal((64, 1024)) * 0.02).astype(np.float32)
    Wp2, S2 = o.pack_weights(o.f64_to_bf16_bits(W2))
    xb = o.f64_to_bf16_bits(xs)
    ref = o.linear_w4a16(xb, Wp2, S2)
    e8 = np.linalg.norm(o.linear_w4a8(xb, Wp2, S2)["y"] - ref) / np.linalg.norm(ref)
    e4 = np.linalg.norm(o.linear_w4a4(xb, Wp2, S2)["y"] - ref) / np.linalg.norm(ref)
    assert e8 < 0.25 * e4, (e8, e4)
    # largest group sum: 128 products of (-128)(-8)
    big = o.w4a4_group_sums(np.full((1, 128), -128, np.int8), o.pack_codes(np.full((1, 128), -8, np.int8)))
    assert big[0, 0, 0] == 131072


# ---------------------------------------------------------------- a5: softmax

def check_softmax(o):
    p = o.softmax(np.array([1.0, 0.0]))
    assert abs(p[0] - 1 / (1 + np.exp(-1.0))) < 1e-15
    assert np.allclose(o.softmax(np.zeros(7)), np.full(7, 1 / 7), rtol=0, atol=1e-15)
    p = o.softmax(np.array([-np.inf, 2.0, -np.inf, 2.0]))
    assert p.tolist() == [0.0, 0.5, 0.0, 0.5]
    p = o.softmax(np.array([1000.0, 0.0]))
    assert p[0] == 1.0 and 0 <= p[1] < 1e-300
    # rows are independent along the last axis
    q = o.softmax(np.array([[0.0, np.log(3.0)], [np.log(4.0), 0.0]]))
    assert np.allclose(q, [[0.25, 0.75], [0.8, 0.2]], rtol=0, atol=1e-15)


# ---------------------------------------------------------------- a6: greedy verify

def _onehot_logits(argmaxes, V):
    """bf16 bits [B, G1, V]: 0 everywhere, 1 at each given argmax."""
    a = np.asarray(argmaxes)
    L = np.zeros(a.shape + (V,), dtype=np.float32)
    for idx in np.ndindex(a.shape):
        L[idx + (a[idx],)] = 1.0
    return bf16_bits(L)


def check_greedy_tutorial_example(o):
    g = golden()["greedy_example"]
    d = np.array([g["draft_tokens"]])
    t = g["target_argmax_first4"] + [0]           # next-position argmax, unused here
    n, out, targ = o.verify_greedy(_onehot_logits([t], 8), d)
    assert n[0] == g["accepted"]
    emitted = [int(v) for v in out[0] if v >= 0]
    assert emitted == g["emitted"]
    assert out[0].tolist() == g["emitted"] + [-1, -1]
    # all four match: gamma + 1 tokens
    n, out, _ = o.verify_greedy(_onehot_logits([[1, 2, 3, 4, 6]], 8), d)
    assert n[0] == 4 and len([v for v in out[0] if v >= 0]) == g["max_tokens_if_all_match"]
    assert out[0].tolist() == [1, 2, 3, 4, 6]


def check_greedy_bruteforce(o):
    V = 3
    for gamma in (1, 2, 3):
        for targ in product(range(V), repeat=gamma + 1):
            L = _onehot_logits([list(targ)], V)
            for d in product(range(V), repeat=gamma):
                n, out, t = o.verify_greedy(L, np.array([d]))
                pre = os.path.commonprefix([list(d), list(targ[:gamma])])
                assert n[0] == len(pre)
                assert list(t[0]) == list(targ)
                assert out[0].tolist() == list(d[: len(pre)]) + [targ[len(pre)]] + [-1] * (gamma - len(pre))


def check_greedy_ties(o):
    L = np.zeros((1, 3, 6), dtype=np.float32)
    L[0, 0] = [0, 3, 1, 3, 3, 2]        # tie at 1, 3, 4 -> 1
    L[0, 1] = [-0.0, 0.0, -1, -2, 0.0, -0.0]  # +0 and -0 equal -> 0
    L[0, 2] = [-np.inf] * 5 + [-5.0]    # single finite value
    n, out, t = o.verify_greedy(bf16_bits(L), np.array([[1, 0]]))
    assert t[0].tolist() == [1, 0, 5]
    assert n[0] == 2 and out[0].tolist() == [1, 0, 5]


def _toy_logits(prefix, V, salt):
    """Deterministic pseudo-model: logits depend only on the prefix (and a salt)."""
    h = 1469598103934665603
    for tok in prefix:
        h = ((h ^ (int(tok) + 1)) * 1099511628211) & ((1 << 63) - 1)
    rng = np.random.default_rng([h, salt])
    l = rng.standard_normal(V).astype(np.float32)
    l[rng.integers(0, V)] += rng.uniform(1.0, 4.0)
    return l


def check_greedy_equivalence(o):
    # greedy speculative decoding emits exactly target-only greedy decoding
    V, gamma, L = 40, 3, 60
    def target(prefix):
        return _toy_logits(prefix, V, 0)
    def draft(prefix):
        return target(prefix) + 0.8 * _toy_logits(prefix, V, 1)
    def bits(l):
        return ((l.astype(np.float32).view(np.uint32) + np.uint32(0x8000)) >> np.uint32(16)).astype(np.uint16)
    def val(b):
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)

    ref = [7]
    while len(ref) < L + 1:
        v = val(bits(target(ref)))
        ref.append(int(np.flatnonzero(v == v.max())[0]))
    seq = [7]
    accepted = 0
    calls = 0
    while len(seq) < L + 1:
        d = []
        for _ in range(gamma):
            v = val(bits(draft(seq + d)))
            d.append(int(np.flatnonzero(v == v.max())[0]))
        rows = np.stack([bits(target(seq + d[:i])) for i in range(gamma + 1)])[None]
        n, out, _ = o.verify_greedy(rows, np.array([d]))
        seq += [int(v) for v in out[0] if v >= 0]
        accepted += int(n[0])
        calls += 1
    assert seq[: L + 1] == ref
    assert accepted > 0 and calls < L  # the draft is useful in this toy setup


# ---------------------------------------------------------------- f4: tree verification (greedy)

def check_tree_chain_is_greedy(o):
    # a chain (node j's parent is j - 1) is the ordinary greedy verification
    rng = np.random.default_rng(21)
    for trial in range(30):
        gamma, V = int(rng.integers(1, 6)), int(rng.integers(2, 6))
        targ = rng.integers(0, V, size=gamma + 1)
        L = _onehot_logits([list(targ)], V)
        d = np.where(rng.random(gamma) < 0.6, targ[:gamma], rng.integers(0, V, size=gamma))[None]
        n, out, _ = o.verify_greedy(L, d)
        tn, tout, nodes = o.verify_tree_greedy(L, d, np.arange(-1, gamma - 1)[None])
        assert tn.tolist() == n.tolist() and tout.tolist() == out.tolist()
        assert nodes[0, :n[0]].tolist() == list(range(n[0]))


def check_tree_bruteforce(o):
    # every tree over 4 nodes (each parent any earlier node or the prefix), tokens in {0, 1}: the
    # accepted path is the deepest node whose whole root path matches the target's argmax of each
    # parent row, taking the lowest-index node among equal-token siblings at every level
    V, T = 2, 4
    rng = np.random.default_rng(3)
    for parents in product(*[range(-1, j) for j in range(T)]):
        for toks in product(range(V), repeat=T):
            targ = rng.integers(0, V, size=T + 1)
            L = _onehot_logits([list(targ)], V)
            n, out, nodes = o.verify_tree_greedy(L, np.array([toks]), np.array([parents]))
            def ok(j):  # j is reached: its chain matches and it is the first matching sibling
                p = parents[j]
                row = 0 if p < 0 else p + 1
                if toks[j] != targ[row]:
                    return False
                if any(parents[k] == p and toks[k] == toks[j] for k in range(j)):
                    return False
                return p < 0 or ok(p)
            reached = [j for j in range(T) if ok(j)]
            depth = lambda j: 1 if parents[j] < 0 else 1 + depth(parents[j])
            last = max(reached, key=depth) if reached else None
            want = []
            j = last
            while j is not None and j >= 0:
                want.insert(0, j)
                j = parents[j] if parents[j] >= 0 else None
            assert nodes[0, :n[0]].tolist() == want, (parents, toks, targ)
            stop_row = 0 if last is None else last + 1
            assert out[0, n[0]] == targ[stop_row]


def check_tree_invalid_nodes(o):
    L = _onehot_logits([[1, 0, 1, 0]], 3)
    # node 0: token out of range; node 1: parent refers forward (to node 2, whose row wants token 0);
    # node 2: valid child of the prefix
    n, out, nodes = o.verify_tree_greedy(L, np.array([[5, 0, 1]]), np.array([[-1, 2, -1]]))
    assert n[0] == 1 and nodes[0].tolist() == [2, -1, -1] and out[0].tolist() == [1, 0, -1, -1]


# ---------------------------------------------------------------- a7, a8: sampling verify

def check_sampling_worked_example(o):
    g = golden()["three_token_example"]
    p = np.array(g["p_target"])
    q = np.array(g["q_draft"])
    x = g["draft_token"]
    P = np.stack([p, p])             # rows: draft position 0, bonus position
    Q = q[None, :]
    r = o.verify_sample_probs(P, Q, [x], [0.0], [0.5, 0.5])
    assert abs(r["a"][0] - g["accept_prob"]) < 1e-15
    assert abs(q[x] * r["a"][0] - g["p_proposed_and_accepted"]) < 1e-15
    # proposing B, which the target rates higher than the draft (0.5 > 0.4), is always accepted
    rb = o.verify_sample_probs(P, Q, [1], [0.999], [0.0, 0.0])
    assert rb["a"][0] == 1.0 and rb["n"] == 1
    # rejection (u >= a) always resamples B from the residual (0, 0.1, 0)
    for u_res in np.linspace(0.0, 0.999, 37):
        r = o.verify_sample_probs(P, Q, [x], [0.8], [u_res, 0.0])
        assert r["n"] == 0 and r["j"] == g["residual_choice"]
        assert np.allclose(r["residual"], g["residual_unnormalised"], atol=1e-15)
        assert r["out"].tolist() == [g["residual_choice"], -1]
    # the test is strict: u == a rejects, u just below accepts and then takes the bonus token
    # (binary fractions so that a = 0.375 / 0.5 = 0.75 exactly)
    P2 = np.array([[0.375, 0.375, 0.25], [0.25, 0.5, 0.25]])
    Q2 = np.array([[0.5, 0.25, 0.25]])
    r = o.verify_sample_probs(P2, Q2, [0], [0.75], [0.0, 0.0])
    assert r["a"][0] == 0.75 and r["n"] == 0
    r = o.verify_sample_probs(P2, Q2, [0], [np.nextafter(0.75, 0)], [0.0, 0.3])
    assert r["n"] == 1 and r["out"].tolist() == [0, 1]


def check_sampling_exact_marginal(o):
    # Integrating over the draft token x ~ q and both uniforms, out[0] is distributed as p_0.
    grid = (np.arange(4000) + 0.5) / 4000
    cases = [(np.array([0.3, 0.5, 0.2]), np.array([0.4, 0.4, 0.2]))]
    rng = np.random.default_rng(9)
    for _ in range(3):
        p = rng.dirichlet(np.ones(4))
        q = rng.dirichlet(np.ones(4))
        cases.append((p, q))
    for p, q in cases:
        V = p.size
        prob = np.zeros(V)
        P = np.stack([p, p])
        for x in range(V):
            acc_frac = np.mean([o.verify_sample_probs(P, q[None], [x], [u], [0.0, 0.0])["n"] == 1
                                for u in grid])
            bonus = np.zeros(V)
            for u in grid:
                bonus[o.verify_sample_probs(P, q[None], [x], [0.0], [0.0, u])["out"][1]] += 1 / grid.size
            # after acceptance the emitted token at position 0 is x itself
            prob[x] += q[x] * acc_frac
            res = np.zeros(V)
            for u in grid:
                res[o.verify_sample_probs(P, q[None], [x], [0.999999], [u, 0.0])["j"]] += 1 / grid.size
            prob += q[x] * (1 - acc_frac) * res
            assert abs(bonus.sum() - 1) < 1e-9
        assert np.allclose(prob, p, atol=2e-3), (prob, p)


def check_sampling_monte_carlo(o, trials=200_000):
    g = golden()["three_token_example"]
    p = np.array(g["p_target"])
    q = np.array(g["q_draft"])
    rng = np.random.default_rng(10)
    xs = rng.choice(3, size=trials, p=q)
    ua = rng.random(trials)
    ur = rng.random(trials)
    P = np.stack([p, p])
    counts = np.zeros(3)
    for i in range(trials):
        r = o.verify_sample_probs(P, q[None], [xs[i]], [ua[i]], [ur[i], 0.0])
        counts[r["out"][0]] += 1
    freq = counts / trials
    sigma = np.sqrt(p * (1 - p) / trials)
    assert np.all(np.abs(freq - np.array(g["final_distribution"])) < 5 * sigma), freq


def check_expected_tokens(o, trials=300_000):
    g = golden()["expected_tokens_example"]
    gamma, alpha = g["gamma"], g["alpha"]
    assert abs(o.expected_tokens(alpha, gamma) - g["E_T"]) < 1e-12
    assert o.expected_tokens(1.0, gamma) == gamma + 1
    # constant per-position acceptance alpha: q = (1, 0) proposes token 0, p = (alpha, 1 - alpha)
    P = np.tile([alpha, 1 - alpha], (gamma + 1, 1))
    Q = np.tile([1.0, 0.0], (gamma, 1))
    rng = np.random.default_rng(12)
    U = rng.random((trials, gamma))
    T = np.empty(trials)
    for i in range(trials):
        T[i] = o.verify_sample_probs(P, Q, [0] * gamma, U[i], [0.5] * (gamma + 1))["n"] + 1
    se = T.std() / np.sqrt(trials)
    assert abs(T.mean() - g["E_T"]) < 4 * se, (T.mean(), se)
    # alpha = 1: every draft accepted, gamma + 1 tokens every time
    P1 = np.tile([1.0, 0.0], (gamma + 1, 1))
    for i in range(200):
        assert o.verify_sample_probs(P1, Q, [0] * gamma, U[i], [0.5] * (gamma + 1))["n"] == gamma


def check_sampling_from_logits(o):
    # verify_sample on logits: the probabilities it reports are the softmax values at the tokens,
    # and a position where p == q is always accepted
    l = np.log(np.array([[[0.3, 0.5, 0.2], [0.1, 0.1, 0.8]]], dtype=np.float64))
    lq = np.log(np.array([[[0.4, 0.4, 0.2]]], dtype=np.float64))
    tb = ((l.astype(np.float32).view(np.uint32) + np.uint32(0x8000)) >> np.uint32(16)).astype(np.uint16)
    db = ((lq.astype(np.float32).view(np.uint32) + np.uint32(0x8000)) >> np.uint32(16)).astype(np.uint16)
    r = o.verify_sample(tb, db, np.array([[0]]), np.array([[0.9]], np.float32), np.array([[0.5, 0.5]], np.float32))
    assert abs(r["p_tok"][0, 0] - 0.3) < 2e-3 and abs(r["q_tok"][0, 0] - 0.4) < 2e-3
    assert abs(r["accept_prob"][0, 0] - 0.75) < 5e-3
    assert r["accept_len"][0] == 0 and r["out_tok"][0].tolist() == [1, -1]
    same = o.verify_sample(np.concatenate([db, db], axis=1), db, np.array([[2]]), np.array([[0.999]], np.float32),
                           np.array([[0.5, 0.1]], np.float32))
    assert same["accept_len"][0] == 1 and same["accept_prob"][0, 0] == 1.0


# ---------------------------------------------------------------- f1: decode loop

def _bits(l):
    return ((np.asarray(l, np.float32).view(np.uint32) + np.uint32(0x8000)) >> np.uint32(16)).astype(np.uint16)


def check_select_token(o):
    # greedy: lowest index among equal maxima; sampling: inverse CDF of softmax, strict '>'
    assert o.select_token(bf16_bits([1.0, 3.0, 3.0, -2.0])) == 1
    l = np.log(np.array([0.25, 0.5, 0.25]))     # bf16 rounding keeps the two 0.25 equal
    b = _bits(l)
    p = o.softmax(o.bf16_to_f32(b).astype(np.float64))
    assert abs(p[0] - p[2]) == 0.0
    for u, want in ((0.0, 0), (p[0] - 1e-9, 0), (p[0] + 1e-9, 1), (p[0] + p[1] + 1e-9, 2), (1 - 2 ** -24, 2)):
        assert o.select_token(b, u) == want, (u, want)
    assert o.select_token(bf16_bits([-np.inf, 5.0, -np.inf]), 0.999) == 1


def check_toy_forward_onehot(o):
    # one-hot weight rows quantise to code 7 with s = fp16(1/7): each layer maps x_v to x_v * 7 s
    # (verify mode), rounded to bf16; in draft mode x_v becomes s_a * qa_v * 7 s.
    D, V = 128, 128
    rng = np.random.default_rng(5)
    E = bf16_bits(o.bf16_to_f32(_bits(rng.standard_normal((6, D)))))
    W = np.zeros((V, D), dtype=np.float32)
    perm = rng.permutation(D)
    W[np.arange(V), perm] = 1.0
    Wp, S = o.pack_weights(bf16_bits(W))
    s = float(np.float16(1.0 / 7.0))
    tok = [3, 0, 5]
    x = o.bf16_to_f32(E[tok]).astype(np.float64)
    want = o.f64_to_bf16_bits(x[:, perm] * 7 * s)
    assert np.array_equal(o.toy_forward(E, [(Wp, S)], tok, False), want)
    qa, s_a = o.quantize_activations(E[tok])
    want4 = o.f64_to_bf16_bits(s_a.astype(np.float64)[:, None] * qa[:, perm].astype(np.float64) * 7 * s)
    assert np.array_equal(o.toy_forward(E, [(Wp, S)], tok, True), want4)
    # two layers apply in order: the second permutation acts on the first layer's output
    perm2 = rng.permutation(D)
    W2 = np.zeros((V, D), dtype=np.float32)
    W2[np.arange(V), perm2] = 1.0
    Wp2, S2 = o.pack_weights(bf16_bits(W2))
    y1 = o.bf16_to_f32(want).astype(np.float64)
    want2 = o.f64_to_bf16_bits(y1[:, perm2] * 7 * s)
    assert np.array_equal(o.toy_forward(E, [(Wp, S), (Wp2, S2)], tok, False), want2)


def check_decode_loop_greedy(o):
    # greedy speculative decoding emits exactly what target-only greedy decoding emits; a draft equal
    # to the target has every draft accepted (gamma + 1 tokens per iteration)
    V, gamma, n_iter = 40, 3, 12
    def target(seq):
        return _bits(_toy_logits(seq, V, 0))
    def draft(seq):
        return _bits(_toy_logits(seq, V, 0) + 0.8 * _toy_logits(seq, V, 1))
    gen, ns = o.speculative_decode(target, draft, [7], n_iter, gamma)
    assert len(gen) == sum(ns) + n_iter
    assert gen == o.target_only_decode(target, [7], len(gen))
    assert 0 < sum(ns) < gamma * n_iter
    gen2, ns2 = o.speculative_decode(target, target, [7], 4, gamma)
    assert ns2 == [gamma] * 4 and gen2 == o.target_only_decode(target, [7], 4 * (gamma + 1))


def check_decode_loop_sampling_marginal(o, trials=3000):
    # speculative sampling leaves the target's distribution of the next token unchanged: the first
    # generated token is distributed as softmax(target(prefix)), whatever the draft
    V, gamma = 3, 2
    lt = np.array([0.0, 1.0, -0.5], dtype=np.float32)
    ld = np.array([1.0, -1.0, 0.5], dtype=np.float32)
    def target(seq):
        return _bits(lt + 0.3 * (len(seq) % 2))
    def draft(seq):
        return _bits(ld)
    p = o.softmax(o.bf16_to_f32(target([0])).astype(np.float64))
    rng = np.random.default_rng(11)
    counts = np.zeros(V)
    for t in range(trials):
        u = rng.random((1, 3 * gamma + 1))
        gen, _ = o.speculative_decode(target, draft, [0], 1, gamma, u_draft=[u[0, :gamma]],
                                      u_acc=[u[0, gamma:2 * gamma]], u_res=[u[0, 2 * gamma:]])
        counts[gen[0]] += 1
    se = np.sqrt(p * (1 - p) / trials)
    assert np.all(np.abs(counts / trials - p) < 5 * se), (counts / trials, p)


# ---------------------------------------------------------------- f2: top-1 statistics

def check_top1_closed_forms(o):
    # one spike of height a over V-1 zeros: p1 = e^a / (e^a + V - 1); equal logits: p1 = 1/V at index 0;
    # a two-way tie [1, 1, 0]: the lower index, p1 = e / (2e + 1)
    V = 5
    tgt = np.zeros((1, 4, V), dtype=np.float32)
    drf = np.zeros((1, 3, V), dtype=np.float32)
    tgt[0, 0, 3] = 2.0
    drf[0, 0, 1] = 2.0                    # the draft's own top-1 is another token
    tgt[0, 2, [1, 4]] = 1.0
    drf[0, 2, [2, 3]] = -1.0              # draft top-1 = index 0 among three zeros: p1 = 1/(3 + 2/e)
    tgt[0, 3, :] = 9.0                    # row gamma is not a draft position
    tt, dt, tp, dp, _ = o.top1_stats(bf16_bits(tgt), bf16_bits(drf))
    e = np.e
    assert tt.tolist() == [[3, 0, 1]] and dt.tolist() == [[1, 0, 0]]
    assert abs(tp[0, 0] - e ** 2 / (e ** 2 + 4)) < 1e-12 and abs(dp[0, 0] - e ** 2 / (e ** 2 + 4)) < 1e-12
    assert abs(tp[0, 1] - 0.2) < 1e-12 and abs(dp[0, 1] - 0.2) < 1e-12
    assert abs(tp[0, 2] - e / (2 * e + 3)) < 1e-12
    assert abs(dp[0, 2] - 1.0 / (3 + 2 / e)) < 1e-12


def check_top1_tally(o):
    # positions: (agree, both high), (disagree, both low), (agree, one high one low),
    # (agree, both low), (disagree, both high)
    def row(top, big, V=4):
        r = np.zeros(V, dtype=np.float32)
        r[top] = big
        return r
    hi, lo = 8.0, 0.5                     # p1 = e^8/(e^8+3) > 0.9;  p1 = e^.5/(e^.5+3) < 0.5
    half = np.array([1.0, 1.0], dtype=np.float32)
    tgt = np.stack([row(0, hi), row(1, lo), row(2, hi), row(3, lo), row(0, hi)])
    drf = np.stack([row(0, hi), row(2, lo), row(2, lo), row(3, lo), row(1, hi)])
    tgt = np.concatenate([tgt, np.zeros((1, 4), np.float32)])[None]
    drf = drf[None]
    _, _, tp, dp, tally = o.top1_stats(bf16_bits(tgt), bf16_bits(drf), high=0.9)
    assert tally[:6].tolist() == [5, 3, 2, 1, 2, 1]
    assert abs(tally[6] - tp.sum()) < 1e-12 and abs(tally[7] - dp.sum()) < 1e-12
    assert abs(tally[6] - (3 * np.exp(8) / (np.exp(8) + 3) + 2 * np.exp(.5) / (np.exp(.5) + 3))) < 1e-12
    # threshold strictness: two equal logits give exactly 1/2, which is "at or below 0.5"
    t2 = np.stack([half, half])[None]
    _, _, tp2, dp2, tally2 = o.top1_stats(bf16_bits(t2), bf16_bits(half[None, None]), high=0.5)
    assert tp2[0, 0] == 0.5 and dp2[0, 0] == 0.5
    assert tally2[:6].tolist() == [1, 1, 0, 0, 1, 1]


ALL_FAST = [
    check_bf16_rounding, check_pack_layout, check_weight_grid_roundtrip, check_weight_hand_cases, check_pack_end_to_end,
    check_w4a16_onehot_and_grid, check_w4a16_error_bound, check_act_quant_hand_cases,
    check_w4a4_bruteforce, check_w4a4_extremes, check_w4a4_constant_activation, check_softmax,
    check_greedy_tutorial_example, check_greedy_bruteforce, check_greedy_ties,
    check_greedy_equivalence, check_sampling_worked_example, check_sampling_from_logits,
    check_top1_closed_forms, check_top1_tally, check_select_token, check_toy_forward_onehot,
    check_w4a8_quantiser, check_w4a8_linear, check_tree_chain_is_greedy, check_tree_bruteforce,
    check_tree_invalid_nodes,
    check_decode_loop_greedy, check_decode_loop_sampling_marginal,
]
