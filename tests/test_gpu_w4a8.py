"""GPU parity of the W4A8 configuration (f3) against the CPU oracle, through the C ABI.

Same bars as W4A4: int8 codes, fp32 scales and int32 group sums bit-exact; y within one bf16 ulp
of the fp64 oracle rounded to bf16.  The shapes cover the decode GEMV (M <= 16), the tensor-core
path on quantised codes (larger M, and long K whose activations do not fit the GEMV), tails.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, bf16_dev, bf16_host_bits, bf16_ulp_distance, lib, packed_dev
from quantized_speculative_decoding_qspec_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    return lib()


def w4a8_case(q, M, N, K, wid=5):
    W = syn.weights(N, K, wid, layer=K + 1)
    X = syn.activations(M, K, wid, step=M + 1)
    Wp, S = packed_dev(q, W)
    Wp_ref, S_ref = oracle.pack_weights(W)
    x = bf16_dev(X)
    ws = q.new_linear_workspace(M, N, K)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    xq = torch.empty(M, K, dtype=torch.int8, device=DEV)
    xs = torch.empty(M, dtype=torch.float32, device=DEV)
    acc = torch.empty(M, N, K // 128, dtype=torch.int32, device=DEV)
    q.qspec_linear_w4a8(x, Wp, S, y, ws, xq, xs, acc)
    r = oracle.linear_w4a8(X, Wp_ref, S_ref)
    assert np.array_equal(xs.cpu().numpy().view(np.uint32), r["s_a"].view(np.uint32))
    assert np.array_equal(xq.cpu().numpy(), r["qa"])
    assert np.array_equal(acc.cpu().numpy(), r["acc"])
    ulp = bf16_ulp_distance(bf16_host_bits(y), oracle.f64_to_bf16_bits(r["y"]))
    assert ulp.max() <= 1, f"W4A8 M={M} N={N} K={K}: max ulp {ulp.max()}"
    y2 = torch.empty_like(y)
    q.qspec_linear_w4a8(x, Wp, S, y2, ws)
    assert torch.equal(y, y2)
    # the 4-bit mode on the same weights is a different product (the modes are not aliased)
    y4 = torch.empty_like(y)
    q.qspec_linear_w4a4(x, Wp, S, y4, ws)
    assert not torch.equal(y, y4)
    q.qspec_check_status()


@pytest.mark.parametrize("M,N,K", [(1, 512, 256), (4, 264, 384), (8, 1000, 1152), (16, 136, 4096), (3, 24, 128),
                                   (17, 264, 384), (64, 512, 4096), (4, 64, 28672), (100, 136, 512),
                                   (8, 520, 8192), (1, 264, 28672), (16, 136, 14336), (4, 136, 28672), (32, 136, 4096)])
def test_w4a8_parity(q, M, N, K):
    w4a8_case(q, M, N, K)


@pytest.mark.parametrize("amax", [1.0, 127.0, 0.3, 3.0e38, 1.0e-36])
def test_w4a8_quantiser_dense_bf16(q, amax):
    # each token: its amax, then the largest bf16 magnitudes below it with alternating signs
    K, N = 16384, 16
    for M in (4, 20):  # the GEMV's in-kernel quantiser, and the separate quantiser kernel
        top = int(oracle.f64_to_bf16_bits(np.array([amax]))[0])
        X = np.zeros((M, K), dtype=np.uint16)
        for m in range(M):
            a_bits = top - m
            mags = np.maximum(np.arange(a_bits - 1, a_bits - K, -1), 0).astype(np.uint16)
            signs = np.where(np.arange(K - 1) % 2 == 0, 0, 0x8000).astype(np.uint16)
            X[m, 0] = a_bits
            X[m, 1:] = mags | signs
        W = syn.weights(N, K, 7)
        Wp, S = packed_dev(q, W)
        xq = torch.empty(M, K, dtype=torch.int8, device=DEV)
        xs = torch.empty(M, dtype=torch.float32, device=DEV)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        q.qspec_linear_w4a8(bf16_dev(X), Wp, S, y, q.new_linear_workspace(M, N, K), xq, xs)
        qa, s_a = oracle.quantize_activations(X, bits=8)
        assert np.array_equal(xs.cpu().numpy().view(np.uint32), s_a.view(np.uint32))
        assert np.array_equal(xq.cpu().numpy(), qa)
    q.qspec_check_status()
