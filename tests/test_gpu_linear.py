"""GPU parity of the packer (a1), W4A16 (a2), the activation quantiser (a3) and W4A4 (a4) against
the CPU oracle, through the C ABI.

Tolerances: packing, activation codes/scales and W4A4 int32 group sums are bit-exact.  W4A16 output
is within a relative Frobenius error of 5e-3 of the fp64 oracle; W4A4 output is within one bf16 ulp
of the oracle's exactly rounded result (only the fp32 order of the scale sums differs).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import (DEV, bf16_dev, bf16_host_bits, bf16_host_f64, bf16_ulp_distance, lib, packed_dev,
                      rel_fro)
from quantized_speculative_decoding_qspec_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

W4A16_TOL = 5e-3


@pytest.fixture(scope="module")
def q():
    return lib()


def check_pack(q, W):
    Wp, S = packed_dev(q, W)
    Wp_ref, S_ref = oracle.pack_weights(W)
    assert np.array_equal(Wp.cpu().numpy(), Wp_ref)
    assert np.array_equal(S.cpu().numpy().view(np.uint16), S_ref.view(np.uint16))
    return Wp, S, Wp_ref, S_ref


@pytest.mark.parametrize("N,K", [(512, 256), (8, 128), (24, 384), (1000, 1152), (136, 4096)])
def test_pack_bit_exact(q, N, K):
    check_pack(q, syn.weights(N, K, workload_id=7, layer=N + K))


def test_pack_edge_groups(q):
    # zero group, fp16-subnormal scale, scale underflow, exact ties, +-0, negative extremes
    N, K = 8, 256
    W = np.zeros((N, K), dtype=np.float32)
    W[1, :4] = [7.0, 2.5, 3.5, -2.5]
    W[2, :3] = [7 * 2.0 ** -20, 3 * 2.0 ** -20, -5 * 2.0 ** -20]
    W[3, :2] = [7 * 2.0 ** -26, 3 * 2.0 ** -26]
    W[4, :3] = [1.0, 0.5, -0.5]
    W[5, :] = -0.0
    W[6, 128:] = np.linspace(-3, 3, 128, dtype=np.float32)
    W[7, :] = -1e30
    check_pack(q, syn.f32_to_bf16_bits(W))


def linear_case(q, M, N, K, wid=3, a4=True, a16=True):
    W = syn.weights(N, K, wid, layer=K)
    X = syn.activations(M, K, wid, step=M)
    Wp, S, Wp_ref, S_ref = check_pack(q, W)
    x = bf16_dev(X)
    ws = q.new_linear_workspace(M, N, K)
    if a16:
        y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        q.qspec_linear_w4a16(x, Wp, S, y, ws)
        ref = oracle.linear_w4a16(X, Wp_ref, S_ref)
        err = rel_fro(bf16_host_f64(y), ref)
        assert err <= W4A16_TOL, f"W4A16 M={M} N={N} K={K}: rel err {err}"
    if a4:
        y4 = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        xq = torch.empty(M, K, dtype=torch.int8, device=DEV)
        xs = torch.empty(M, dtype=torch.float32, device=DEV)
        acc = torch.empty(M, N, K // 128, dtype=torch.int32, device=DEV)
        q.qspec_linear_w4a4(x, Wp, S, y4, ws, xq, xs, acc)
        r = oracle.linear_w4a4(X, Wp_ref, S_ref)
        assert np.array_equal(xs.cpu().numpy().view(np.uint32), r["s_a"].view(np.uint32))
        assert np.array_equal(xq.cpu().numpy(), r["qa"])
        assert np.array_equal(acc.cpu().numpy(), r["acc"])
        ulp = bf16_ulp_distance(bf16_host_bits(y4), oracle.f64_to_bf16_bits(r["y"]))
        assert ulp.max() <= 1, f"W4A4 M={M} N={N} K={K}: max ulp {ulp.max()}"
        # without the optional outputs the same y comes back
        y4b = torch.empty_like(y4)
        q.qspec_linear_w4a4(x, Wp, S, y4b, ws)
        assert torch.equal(y4, y4b)
        if a16:  # repeated calls on the same workspace give the same bits
            y2 = torch.empty_like(y)
            q.qspec_linear_w4a16(x, Wp, S, y2, ws)
            assert torch.equal(y, y2)
    q.qspec_check_status()


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 9, 15, 16, 17, 33, 64])
def test_linear_m_sweep(q, M):
    linear_case(q, M, 264, 384)


@pytest.mark.parametrize("M,N,K", [(4, 512, 256), (1, 8, 128), (3, 24, 1152), (16, 1000, 128),
                                   (1, 1024, 4096), (4, 4096, 4096), (16, 1024, 4096), (64, 512, 4096),
                                   (100, 136, 512), (256, 256, 1024), (8, 264, 8192), (12, 136, 2048),
                                   (32, 264, 4096), (24, 136, 1152), (20, 520, 28672)])
def test_linear_shapes(q, M, N, K):
    linear_case(q, M, N, K)


def test_linear_largest_k(q):
    linear_case(q, 4, 128, 14336)


@pytest.mark.parametrize("M,N,K", [(1, 64, 28672), (2, 136, 28672), (16, 256, 14336), (8, 200, 14336),
                                   (12, 520, 4096), (4, 520, 28672), (3, 24, 28672), (16, 264, 8192),
                                   (8, 136, 28672), (13, 40, 28672)])
def test_linear_staging_widths(q, M, N, K):
    # one- and two-token staging for long K, and the shapes whose staged activations do not fit
    # the GEMV's shared memory in one piece (K split into 2, 4 or 8 chunks across CTAs, partial
    # tiles summed by the last chunk; W4A4 with fewer than eight tokens reads all of x for amax)
    linear_case(q, M, N, K)


def test_linear_maximum_tokens(q):
    # the largest M the boundary accepts (4096 tokens), a ragged N tail, both modes
    linear_case(q, 4096, 40, 256)


def test_w4a4_extreme_codes(q):
    # -8 codes in the weights (not produced by the packer but accepted), +-7 activations everywhere
    N, K, M = 16, 256, 2
    codes = np.tile(np.arange(-8, 8, dtype=np.int8), (N, K // 16))
    Wp_ref = oracle.pack_codes(codes)
    S_ref = np.full((N, K // 128), 0.5, dtype=np.float16)
    X = syn.f32_to_bf16_bits(np.where(np.arange(K) % 2 == 0, 7.0, -7.0).astype(np.float32)[None].repeat(M, 0))
    Wp = torch.from_numpy(Wp_ref).to(DEV)
    S = torch.from_numpy(S_ref).to(DEV)
    x = bf16_dev(X)
    ws = q.new_linear_workspace(M, N, K)
    y4 = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    acc = torch.empty(M, N, K // 128, dtype=torch.int32, device=DEV)
    q.qspec_linear_w4a4(x, Wp, S, y4, ws, acc_out=acc)
    r = oracle.linear_w4a4(X, Wp_ref, S_ref)
    assert np.array_equal(acc.cpu().numpy(), r["acc"])
    y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    q.qspec_linear_w4a16(x, Wp, S, y, ws)
    assert rel_fro(bf16_host_f64(y), oracle.linear_w4a16(X, Wp_ref, S_ref)) <= W4A16_TOL


@pytest.mark.parametrize("amax", [1.0, 7.0, 0.3, 1.0e-3, 123.5, 3.0e5, 3.0e38, 1.0e-29, 2.0e-30, 1.0e-37])
def test_activation_quantiser_dense_bf16(q, amax):
    # Each token holds its amax and then the 16383 largest bf16 magnitudes below it, signs
    # alternating: every quotient x / s_a that can round differently lies in this range, and the
    # codes and scales must equal the oracle's bit for bit.
    K, M, N = 16384, 4, 16
    top = int(oracle.f64_to_bf16_bits(np.array([amax]))[0])
    X = np.zeros((M, K), dtype=np.uint16)
    for m in range(M):
        a_bits = top - m  # four neighbouring amax values
        mags = np.maximum(np.arange(a_bits - 1, a_bits - K, -1), 0).astype(np.uint16)
        signs = np.where(np.arange(K - 1) % 2 == 0, 0, 0x8000).astype(np.uint16)
        X[m, 0] = a_bits
        X[m, 1:] = mags | signs
    W = syn.weights(N, K, 7)
    Wp, S, Wp_ref, S_ref = check_pack(q, W)
    xq = torch.empty(M, K, dtype=torch.int8, device=DEV)
    xs = torch.empty(M, dtype=torch.float32, device=DEV)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    q.qspec_linear_w4a4(bf16_dev(X), Wp, S, y, q.new_linear_workspace(M, N, K), xq, xs)
    qa, s_a = oracle.quantize_activations(X)
    assert np.array_equal(xs.cpu().numpy().view(np.uint32), s_a.view(np.uint32))
    assert np.array_equal(xq.cpu().numpy(), qa)


def test_zero_activation_token(q):
    N, K, M = 64, 256, 3
    W = syn.weights(N, K, 5)
    X = syn.activations(M, K, 5)
    X[1] = 0  # an all-zero token: s_a = 0, codes 0, y = 0
    Wp, S, Wp_ref, S_ref = check_pack(q, W)
    y4 = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    xs = torch.empty(M, dtype=torch.float32, device=DEV)
    q.qspec_linear_w4a4(bf16_dev(X), Wp, S, y4, q.new_linear_workspace(M, N, K), xs_out=xs)
    assert xs[1].item() == 0.0 and torch.count_nonzero(y4[1]).item() == 0


# ---- full-size shapes of the bench workload (Llama-3-8B-shaped decode linears), sampled rows

LLAMA8B = {"qo": (4096, 4096), "kv": (1024, 4096), "gate_up": (14336, 4096), "down": (4096, 14336),
           "lm_head": (128256, 4096)}


@pytest.mark.parametrize("name", list(LLAMA8B))
def test_fullsize_sampled_rows(q, name):
    N, K = LLAMA8B[name]
    W = syn.weights(N, K, 1, layer=list(LLAMA8B).index(name))
    Wp, S = packed_dev(q, W)
    rows = np.sort(np.random.default_rng(N).choice(N, size=min(N, 192), replace=False))
    Wp_ref, S_ref = oracle.pack_weights(W[rows])
    assert np.array_equal(Wp.cpu().numpy()[rows], Wp_ref)
    assert np.array_equal(S.cpu().numpy()[rows].view(np.uint16), S_ref.view(np.uint16))
    for M, mode in ((4, "a16"), (1, "a4"), (64, "a16"), (16, "a4")):
        X = syn.activations(M, K, 1, step=M)
        x = bf16_dev(X)
        ws = q.new_linear_workspace(M, N, K)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        if mode == "a16":
            q.qspec_linear_w4a16(x, Wp, S, y, ws)
            ref = oracle.linear_w4a16(X, Wp_ref, S_ref)
            assert rel_fro(bf16_host_f64(y)[:, rows], ref) <= W4A16_TOL
        else:
            acc = torch.empty(M, N, K // 128, dtype=torch.int32, device=DEV)
            q.qspec_linear_w4a4(x, Wp, S, y, ws, acc_out=acc)
            r = oracle.linear_w4a4(X, Wp_ref, S_ref)
            assert np.array_equal(acc.cpu().numpy()[:, rows], r["acc"])
            ulp = bf16_ulp_distance(bf16_host_bits(y)[:, rows], oracle.f64_to_bf16_bits(r["y"]))
            assert ulp.max() <= 1
    q.qspec_check_status()


# ---- Llama-2-70B shapes above the decode sizes (the tensor-core kernel, stream-K over many SMs)

LLAMA70B_TC = {"gate_up": (28672, 8192, 2), "down": (8192, 28672, 3)}  # N, K, layer index of the sweep


@pytest.mark.parametrize("name", list(LLAMA70B_TC))
def test_fullsize_70b_tensor_core_sampled_rows(q, name):
    # the M = 4, 8, 16 (GEMV with K chunks: four or eight at 16 tokens) and 64, 128, 256 (tensor-core
    # kernels) cells of the Llama-2-70B sweep, both modes, on sampled output rows (the first and last
    # rows always among them); every token tile and K contributor of a sampled row takes part in its
    # value; W4A4 both through the checking path (exact group sums out) and the production one
    N, K, li = LLAMA70B_TC[name]
    W = syn.weights(N, K, 3, layer=li)
    Wp, S = packed_dev(q, W)
    rng = np.random.default_rng(N + K)
    rows = np.unique(np.concatenate([[0, N - 1], rng.choice(N, size=126, replace=False)]))
    Wp_ref, S_ref = oracle.pack_weights(W[rows])
    assert np.array_equal(Wp.cpu().numpy()[rows], Wp_ref)
    assert np.array_equal(S.cpu().numpy()[rows].view(np.uint16), S_ref.view(np.uint16))
    rows_dev = torch.from_numpy(rows).to(DEV)
    for M in (4, 8, 16, 64, 128, 256):
        X = syn.activations(M, K, 3, step=M)
        x = bf16_dev(X)
        ws = q.new_linear_workspace(M, N, K)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        q.qspec_linear_w4a16(x, Wp, S, y, ws)
        ref = oracle.linear_w4a16(X, Wp_ref, S_ref)
        err = rel_fro(bf16_host_f64(y[:, rows_dev]), ref)
        assert err <= W4A16_TOL, f"W4A16 {name} M={M}: rel err {err}"
        y4 = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        xs = torch.empty(M, dtype=torch.float32, device=DEV)
        acc = torch.empty(M, N, K // 128, dtype=torch.int32, device=DEV)
        q.qspec_linear_w4a4(x, Wp, S, y4, ws, xs_out=xs, acc_out=acc)
        r = oracle.linear_w4a4(X, Wp_ref, S_ref)
        assert np.array_equal(xs.cpu().numpy().view(np.uint32), r["s_a"].view(np.uint32))
        assert np.array_equal(acc[:, rows_dev].cpu().numpy(), r["acc"]), f"W4A4 {name} M={M}: group sums"
        ulp = bf16_ulp_distance(bf16_host_bits(y4[:, rows_dev]), oracle.f64_to_bf16_bits(r["y"]))
        assert ulp.max() <= 1, f"W4A4 {name} M={M}: max ulp {ulp.max()}"
        del acc
        q.qspec_linear_w4a4(x, Wp, S, y4, ws)
        ulp = bf16_ulp_distance(bf16_host_bits(y4[:, rows_dev]), oracle.f64_to_bf16_bits(r["y"]))
        assert ulp.max() <= 1, f"W4A4 {name} M={M} (no sums out): max ulp {ulp.max()}"
        q.qspec_check_status()


def test_workspace_of_another_shape_is_refused(q):
    # A workspace records the (M, N, K) of the calls that use its regions.  W4A4 at M = 8 writes the
    # quantised codes there; W4A16 at M = 64 (tensor-core kernel: tickets, partial sums) on the same
    # workspace must then touch nothing and report QSPEC_ERR_WORKSPACE, leaving y as it was.
    N, K = 264, 1024
    W = syn.weights(N, K, 4)
    Wp, S, Wp_ref, S_ref = check_pack(q, W)
    Xa, Xb, X1 = syn.activations(8, K, 4, step=1), syn.activations(64, K, 4, step=2), syn.activations(1, K, 4, step=3)
    n = max(q.qspec_linear_workspace_size(8, N, K), q.qspec_linear_workspace_size(64, N, K))
    ws = torch.zeros(n, dtype=torch.uint8, device=DEV)
    ya = torch.empty(8, N, dtype=torch.bfloat16, device=DEV)
    q.qspec_linear_w4a4(bf16_dev(Xa), Wp, S, ya, ws)
    q.qspec_check_status()
    yb = torch.full((64, N), 3.0, dtype=torch.bfloat16, device=DEV)
    q.qspec_linear_w4a16(bf16_dev(Xb), Wp, S, yb, ws)
    with pytest.raises(q.QSpecError) as e:
        q.qspec_check_status()
    assert q.STATUS[e.value.code] == "QSPEC_ERR_WORKSPACE"
    assert bool((yb.float() == 3.0).all())
    q.qspec_check_status()  # the error was reported once and cleared
    # a zero-fill hands the workspace to the other shape: now M = 64 works and M = 8 is refused
    ws.zero_()
    q.qspec_linear_w4a16(bf16_dev(Xb), Wp, S, yb, ws)
    q.qspec_check_status()
    assert rel_fro(bf16_host_f64(yb), oracle.linear_w4a16(Xb, Wp_ref, S_ref)) <= W4A16_TOL
    q.qspec_linear_w4a4(bf16_dev(Xa), Wp, S, ya, ws)
    with pytest.raises(q.QSpecError) as e:
        q.qspec_check_status()
    assert q.STATUS[e.value.code] == "QSPEC_ERR_WORKSPACE"
    # calls that use no region of the workspace (one token, quantised inside the GEMV) run on it
    y1 = torch.empty(1, N, dtype=torch.bfloat16, device=DEV)
    q.qspec_linear_w4a4(bf16_dev(X1), Wp, S, y1, ws)
    q.qspec_check_status()
    r = oracle.linear_w4a4(X1, Wp_ref, S_ref)
    assert bf16_ulp_distance(bf16_host_bits(y1), oracle.f64_to_bf16_bits(r["y"])).max() <= 1


# ---- seeded random shapes across the three kernels (the GEMV up to 32 tokens, the exact-code
# tcgen05 kernel above it, the dequantising one for W4A16 from 65 tokens) and the K-chunk planner

def _random_shapes(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        M = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 11, 16, 23, 32, 40, 64, 65, 100, 128, 200, 256]))
        N = int(rng.integers(1, 400)) * 8
        K = int(rng.integers(1, 120)) * 128
        out.append((M, N, K))
    return out


@pytest.mark.parametrize("M,N,K", _random_shapes(24, 2024))
def test_linear_random_shapes(q, M, N, K):
    W = syn.weights(N, K, 5, layer=N % 97)
    X = syn.activations(M, K, 5, step=M + K)
    Wp, S = packed_dev(q, W)
    rng = np.random.default_rng(M * 7 + N + K)
    rows = np.unique(np.concatenate([[0, N - 1], rng.choice(N, size=min(N, 48), replace=False)]))
    Wp_ref, S_ref = oracle.pack_weights(W[rows])
    rows_dev = torch.from_numpy(rows).to(DEV)
    x = bf16_dev(X)
    ws = q.new_linear_workspace(M, N, K)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    q.qspec_linear_w4a16(x, Wp, S, y, ws)
    err = rel_fro(bf16_host_f64(y[:, rows_dev]), oracle.linear_w4a16(X, Wp_ref, S_ref))
    assert err <= W4A16_TOL, f"W4A16 M={M} N={N} K={K}: rel err {err}"
    r = oracle.linear_w4a4(X, Wp_ref, S_ref)
    for f in (q.qspec_linear_w4a4, q.qspec_linear_w4a8):
        if f is q.qspec_linear_w4a8:
            r = oracle.linear_w4a8(X, Wp_ref, S_ref)
        yq = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        f(x, Wp, S, yq, ws)
        ulp = bf16_ulp_distance(bf16_host_bits(yq[:, rows_dev]), oracle.f64_to_bf16_bits(r["y"]))
        assert ulp.max() <= 1, f"{f.__name__} M={M} N={N} K={K}: max ulp {ulp.max()}"
    q.qspec_check_status()
