"""GPU parity of qspec_linear_group (several linears that read the same activations, one launch)
against the CPU oracle, through the C ABI.

Each part must match what the single-linear definitions give for it: W4A16 within a relative
Frobenius error of 5e-3 of the fp64 oracle, W4A4 and W4A8 within one bf16 ulp of the oracle's exactly
rounded result.  Cases: every mode at 1-4 tokens, parts whose row counts end inside a 16-row tile,
four parts, long K (split into chunks across CTAs), the Llama-3-8B q/k/v and gate/up groups on sampled
rows, repeated calls on one workspace, and the shapes the grouped launch refuses.
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


def reference(abits, X, Wp_ref, S_ref):
    if abits == 16:
        return oracle.linear_w4a16(X, Wp_ref, S_ref)
    return (oracle.linear_w4a4 if abits == 4 else oracle.linear_w4a8)(X, Wp_ref, S_ref)["y"]


def check_part(abits, y, ref, rows=None, what=""):
    got = y if rows is None else y[:, rows]
    if abits == 16:
        err = rel_fro(bf16_host_f64(got), ref)
        assert err <= W4A16_TOL, f"{what}: rel err {err}"
    else:
        ulp = bf16_ulp_distance(bf16_host_bits(got), oracle.f64_to_bf16_bits(ref))
        assert ulp.max() <= 1, f"{what}: max ulp {ulp.max()}"


def run_group(q, abits, M, K, Ns, wid, sample=None):
    X = syn.activations(M, K, wid, step=M)
    x = bf16_dev(X)
    packs, ys, Ws = [], [], []
    for i, N in enumerate(Ns):
        W = syn.weights(N, K, wid, layer=i)
        Wp, S = packed_dev(q, W)
        packs.append((Wp, S))
        Ws.append(W)
        ys.append(torch.full((M, N), 7.0, dtype=torch.bfloat16, device=DEV))
    ws = q.new_linear_group_workspace(M, Ns, K)
    q.qspec_linear_group(abits, x, [(Wp, S, y) for (Wp, S), y in zip(packs, ys)], ws)
    q.qspec_check_status()
    for i, (N, W, y) in enumerate(zip(Ns, Ws, ys)):
        rows = None
        if sample and N > sample:
            rng = np.random.default_rng(N + K + i)
            rows = np.unique(np.concatenate([[0, N - 1], rng.choice(N, size=sample, replace=False)]))
        Wp_ref, S_ref = oracle.pack_weights(W if rows is None else W[rows])
        check_part(abits, ys[i], reference(abits, X, Wp_ref, S_ref),
                   None if rows is None else torch.from_numpy(rows).to(DEV), f"abits {abits} M {M} part {i}")
    return x, packs, ys, ws


@pytest.mark.parametrize("abits", [16, 4, 8])
@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_group_modes_and_tokens(q, abits, M):
    run_group(q, abits, M, 384, [264, 136, 40], wid=21)


@pytest.mark.parametrize("abits", [16, 4])
def test_group_four_ragged_parts(q, abits):
    # row counts 8 past a 16-row tile boundary: each part starts on a tile of its own
    run_group(q, abits, 3, 1152, [8, 24, 520, 1000], wid=22)


@pytest.mark.parametrize("abits", [16, 4])
@pytest.mark.parametrize("M", [1, 4])
def test_group_long_k_chunked(q, abits, M):
    # K = 14336 (the down projection's width) is split into chunks across CTAs; the partial tiles of
    # every part are summed by the chunk that finishes last
    run_group(q, abits, M, 14336, [264, 520], wid=23)


@pytest.mark.parametrize("abits,M", [(4, 1), (16, 4), (8, 1)])
def test_group_llama8b_qkv_and_gate_up(q, abits, M):
    run_group(q, abits, M, 4096, [4096, 1024, 1024], wid=24, sample=96)
    run_group(q, abits, M, 4096, [14336, 14336], wid=25, sample=96)


def test_group_repeats_bit_for_bit(q):
    x, packs, ys, ws = run_group(q, 4, 1, 14336, [264, 520], wid=26)
    again = [torch.empty_like(y) for y in ys]
    q.qspec_linear_group(4, x, [(Wp, S, y) for (Wp, S), y in zip(packs, again)], ws)
    q.qspec_check_status()
    for y, y2 in zip(ys, again):
        assert torch.equal(y, y2)


def test_group_refuses_unserved_shapes(q):
    K = 256
    W = syn.weights(64, K, 27)
    Wp, S = packed_dev(q, W)
    x = bf16_dev(syn.activations(5, K, 27))
    y = torch.empty(5, 64, dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)
    with pytest.raises(q.QSpecError) as e:
        q.qspec_linear_group(16, x, [(Wp, S, y)], ws)  # five tokens: above QSPEC_GROUP_MAX_M
    assert q.STATUS[e.value.code] == "QSPEC_ERR_UNSUPPORTED_SHAPE"
