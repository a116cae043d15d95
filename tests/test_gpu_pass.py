"""GPU parity of the linear pass (one launch over several decode-size linears of one mode) against
the CPU oracle, through the C ABI.

Every layer of a pass must meet the single-linear bars: W4A16 within a relative Frobenius error of
5e-3 of the fp64 oracle, W4A4 / W4A8 within one bf16 ulp of the oracle's exactly rounded result.
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


def oracle_y(abits, X, Wp_ref, S_ref):
    if abits == 16:
        return oracle.linear_w4a16(X, Wp_ref, S_ref)
    if abits == 4:
        return oracle.linear_w4a4(X, Wp_ref, S_ref)["y"]
    return oracle.linear_w4a8(X, Wp_ref, S_ref)["y"]


def check_layer(abits, y, ref, what):
    if abits == 16:
        err = rel_fro(bf16_host_f64(y), ref)
        assert err <= W4A16_TOL, f"{what}: rel err {err}"
    else:
        ulp = bf16_ulp_distance(bf16_host_bits(y), oracle.f64_to_bf16_bits(ref))
        assert ulp.max() <= 1, f"{what}: max ulp {ulp.max()}"


def run_pass(q, abits, M, shapes, wid, after=None, reps=2):
    """shapes: [(N, K)]; every layer has its own seeded weights and activations."""
    after = after or [0] * len(shapes)
    lay, refs = [], []
    for i, (N, K) in enumerate(shapes):
        W = syn.weights(N, K, wid, layer=i)
        X = syn.activations(M, K, wid, step=i)
        Wp, S = packed_dev(q, W)
        Wp_ref, S_ref = oracle.pack_weights(W)
        y = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=DEV)
        lay.append((bf16_dev(X), Wp, S, y, after[i]))
        refs.append(oracle_y(abits, X, Wp_ref, S_ref))
    lp = q.LinearPass(abits, lay, q.new_pass_workspace())
    for _ in range(reps):  # the barrier counters are left ready: a second run gives the same bits
        first = [l[3].clone() for l in lay]
        lp.run()
        q.qspec_check_status()
    for i, ((x, Wp, S, y, _), ref) in enumerate(zip(lay, refs)):
        check_layer(abits, y, ref, f"layer {i} {shapes[i]} abits={abits} M={M}")
        if reps > 1:
            assert torch.equal(y, first[i]) or reps == 1
    return lay


SMALL = [(512, 256), (264, 384), (8, 128), (1000, 1152), (136, 4096), (24, 256)]


@pytest.mark.parametrize("abits", [16, 4, 8])
@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_pass_small_layers(q, abits, M):
    # ragged N tails, K = 128 (one group: one group in flight per warp), K up to 4096
    run_pass(q, abits, M, SMALL, wid=30 + M)


@pytest.mark.parametrize("abits", [16, 4])
def test_pass_groups_of_four(q, abits):
    # every K a multiple of 512: the four-groups-in-flight variant
    run_pass(q, abits, 4 if abits == 16 else 1, [(512, 512), (4096, 2048), (24, 1024), (1032, 4096)], wid=40)


@pytest.mark.parametrize("abits", [16, 4])
def test_pass_with_barriers(q, abits):
    # layers marked `after` wait for every CTA to finish the earlier ones (their own inputs are
    # independent here, so the values are the plain per-layer ones)
    run_pass(q, abits, 1 if abits == 4 else 4, [(512, 512), (64, 512), (4096, 1024), (8, 512), (1024, 2048)],
             wid=41, after=[0, 0, 1, 0, 1])


def test_pass_dependency_chain(q):
    # layer 1 reads layer 0's output, layer 2 reads layer 1's: the barrier must make them visible
    M, D1, D2, D3 = 2, 1024, 2048, 512
    shapes = [(D2, D1), (D3, D2), (D1, D3)]
    Ws = [syn.weights(N, K, 50, layer=i) for i, (N, K) in enumerate(shapes)]
    packed = [packed_dev(q, W) for W in Ws]
    refs = [oracle.pack_weights(W) for W in Ws]
    X0 = syn.activations(M, D1, 50)
    x0 = bf16_dev(X0)
    ys = [torch.empty(M, N, dtype=torch.bfloat16, device=DEV) for N, _ in shapes]
    for abits in (16, 4):
        lay = [(x0, *packed[0], ys[0], 0), (ys[0], *packed[1], ys[1], 1), (ys[1], *packed[2], ys[2], 1)]
        q.LinearPass(abits, lay, q.new_pass_workspace()).run()
        q.qspec_check_status()
        xin = X0
        for i in range(3):
            ref = oracle_y(abits, xin, *refs[i])
            check_layer(abits, ys[i], ref, f"chain layer {i} abits={abits}")
            xin = bf16_host_bits(ys[i])  # the next layer's input is exactly what the GPU wrote


def test_pass_many_idle_ctas(q):
    # sixteen layers of one or two tiles: most CTAs have nothing in a layer and take later ones
    shapes = [(8 * (1 + i % 4), 128 * (1 + i % 3)) for i in range(16)]
    run_pass(q, 4, 1, shapes, wid=42)
    run_pass(q, 16, 3, shapes, wid=43)


LLAMA8B_PASS = [("q", 4096, 4096, 0), ("k", 1024, 4096, 0), ("v", 1024, 4096, 0), ("o", 4096, 4096, 1),
                ("gate", 14336, 4096, 1), ("up", 14336, 4096, 0), ("down", 4096, 14336, 1),
                ("lm_head", 128256, 4096, 1)]


@pytest.mark.parametrize("abits,M", [(4, 1), (16, 4), (8, 1)])
def test_pass_llama8b_decoder_sampled_rows(q, abits, M):
    # the benchmark's pass: the eight Llama-3-8B-shaped linears with the decoder's dependencies,
    # checked on sampled output rows of every layer
    lay, checks = [], []
    for li, (name, N, K, after) in enumerate(LLAMA8B_PASS):
        W = syn.weights(N, K, 1, layer=li)
        Wp, S = packed_dev(q, W)
        rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(N + li).choice(N, 62, replace=False)]))
        Wp_ref, S_ref = oracle.pack_weights(W[rows])
        X = syn.activations(M, K, 1, step=10 * li + 9)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        lay.append((bf16_dev(X), Wp, S, y, after))
        checks.append((name, rows, oracle_y(abits, X, Wp_ref, S_ref)))
    q.LinearPass(abits, lay, q.new_pass_workspace()).run()
    q.qspec_check_status()
    for (name, rows, ref), l in zip(checks, lay):
        check_layer(abits, l[3][:, torch.from_numpy(rows).to(DEV)], ref, f"{name} abits={abits} M={M}")
