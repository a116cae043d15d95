"""GPU parity of the tensor-core W4A16 kernel (weights dequantised to fp16 on chip, TMEM accumulators
over the whole K range) against the CPU oracle, through the C ABI.

The kernel serves W4A16 from 65 tokens on (fewer run on the GEMV or the exact-code tensor-core
kernel).  The cases below take each of its instantiations (NM = 128 tokens per tile with J = 1 or 2
tiles per work item, NM = 256 with J = 1) and its schedule's cases: whole items, items cut between
CTAs, several token tiles; output rows are sampled where N is large (the first and last rows always
among them).  Tolerance: relative Frobenius error 5e-3 against the fp64 oracle, per token.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, bf16_dev, bf16_host_bits, bf16_host_f64, bf16_ulp_distance, lib, packed_dev, rel_fro
from quantized_speculative_decoding_qspec_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

W4A16_TOL = 5e-3


@pytest.fixture(scope="module")
def q():
    return lib()


def run_a16(q, X, Wp, S, M, N, K):
    ws = q.new_linear_workspace(M, N, K)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    q.qspec_linear_w4a16(bf16_dev(X), Wp, S, y, ws)
    q.qspec_check_status()
    return y, ws


def sampled_rows(N, seed, n=96):
    if N <= n:
        return np.arange(N)
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, N - 1], rng.choice(N, size=n, replace=False)]))


def check_rows(q, M, N, K, wid, X=None):
    W = syn.weights(N, K, wid, layer=K)
    if X is None:
        X = syn.activations(M, K, wid, step=M)
    Wp, S = packed_dev(q, W)
    rows = sampled_rows(N, N + K + M)
    Wp_ref, S_ref = oracle.pack_weights(W[rows])
    assert np.array_equal(Wp.cpu().numpy()[rows], Wp_ref)
    y, ws = run_a16(q, X, Wp, S, M, N, K)
    ref = oracle.linear_w4a16(X, Wp_ref, S_ref)
    got = bf16_host_f64(y)[:, rows]
    for m in range(M):
        err = rel_fro(got[m:m + 1], ref[m:m + 1])
        assert err <= W4A16_TOL, f"M={M} N={N} K={K} token {m}: rel err {err}"
    # a second call on the same workspace (tickets reset, partial sums rewritten) gives the same bits
    y2 = torch.empty_like(y)
    q.qspec_linear_w4a16(bf16_dev(X), Wp, S, y2, ws)
    q.qspec_check_status()
    assert torch.equal(y, y2)


# (M, N, K) -> the (NM, J) instantiation the plan takes for it on a 152-SM GB300
COVER = [
    (65, 136, 256),       # NM 128, J 1
    (65, 24576, 8192),    # NM 128, J 2
    (129, 136, 256),      # NM 256, J 1
]


@pytest.mark.parametrize("M,N,K", COVER)
def test_dq_every_instantiation(q, M, N, K):
    check_rows(q, M, N, K, wid=11)


@pytest.mark.parametrize("M,N,K", [(100, 264, 384), (100, 1000, 1152), (256, 520, 2048), (300, 264, 384),
                                   (513, 136, 1024), (65, 8, 128), (80, 4096, 4096), (200, 14336, 4096)])
def test_dq_ragged_shapes(q, M, N, K):
    # ragged token tiles (M not a multiple of NM, several token tiles above 256), ragged row tiles,
    # the smallest N and K, and a split of every item among several CTAs
    check_rows(q, M, N, K, wid=12)


def test_dq_token_magnitudes(q):
    # one power-of-two factor per token: tokens whose largest magnitude is far below or far above
    # the fp16 range (bf16 normals from 2^-120 to 2^120, a zero token, and a token whose values span
    # 2^-20 .. 2^20) are each computed to the same relative accuracy
    M, N, K = 80, 264, 512
    base = syn.activations(M, K, 13, step=1)
    Xf = syn.bf16_bits_to_f32(base).astype(np.float64)
    scale = np.ones((M, 1))
    scale[1], scale[2], scale[3], scale[4] = 2.0 ** -120, 2.0 ** 120, 2.0 ** -60, 2.0 ** 60
    Xf = Xf * scale
    Xf[5] = 0.0
    Xf[6] = Xf[6] * 2.0 ** np.linspace(-20, 20, K)
    X = syn.f32_to_bf16_bits(Xf.astype(np.float32))
    check_rows(q, M, N, K, wid=13, X=X)


def test_dq_rounds_each_weight_once(q):
    # weights that are exact multiples of a power-of-two scale and small integer activations: every
    # fp16 weight code * s is exact and so is every fp32 sum, so y is the oracle's exactly rounded
    # result bit for bit (any extra rounding or a lost term would show)
    M, N, K = 70, 264, 1024
    rng = np.random.default_rng(5)
    codes = rng.integers(-7, 8, size=(N, K)).astype(np.float64)
    codes[:, ::128] = 7.0  # every group's amax is 7 * s, so the packer picks s exactly
    W = syn.f32_to_bf16_bits((codes * 2.0 ** -4).astype(np.float32))
    X = syn.f32_to_bf16_bits(rng.integers(-4, 5, size=(M, K)).astype(np.float32))
    Wp, S = packed_dev(q, W)
    Wp_ref, S_ref = oracle.pack_weights(W)
    assert np.all(S_ref.astype(np.float64) == 2.0 ** -4)
    y, _ = run_a16(q, X, Wp, S, M, N, K)
    ref = oracle.linear_w4a16(X, Wp_ref, S_ref)
    assert np.array_equal(bf16_host_bits(y), oracle.f64_to_bf16_bits(ref))


@pytest.mark.parametrize("M,N,K", [(128, 264, 4096), (96, 1000, 2048)])
def test_dq_and_exact_code_kernel_share_a_workspace(q, M, N, K):
    # W4A16 (this kernel) and W4A4 (the exact-code tensor-core kernel) alternate on one workspace;
    # both split tiles between CTAs, and the tickets one leaves behind must be the zeros the other
    # starts from
    W = syn.weights(N, K, 14, layer=K)
    X = syn.activations(M, K, 14, step=M)
    Wp, S = packed_dev(q, W)
    Wp_ref, S_ref = oracle.pack_weights(W)
    ref16 = oracle.linear_w4a16(X, Wp_ref, S_ref)
    ref4 = oracle.linear_w4a4(X, Wp_ref, S_ref)
    ws = q.new_linear_workspace(M, N, K)
    x = bf16_dev(X)
    for _ in range(2):
        y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        q.qspec_linear_w4a16(x, Wp, S, y, ws)
        assert rel_fro(bf16_host_f64(y), ref16) <= W4A16_TOL
        y4 = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        q.qspec_linear_w4a4(x, Wp, S, y4, ws)
        assert bf16_ulp_distance(bf16_host_bits(y4), oracle.f64_to_bf16_bits(ref4["y"])).max() <= 1
        q.qspec_check_status()
