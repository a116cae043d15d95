"""GPU parity of the top-1 statistics (f2) against the CPU oracle, through the C ABI.

Top-1 tokens of both modes are bit-exact; top-1 probabilities within 1e-5 absolute of the fp64
oracle; the tally's counts are exact except for positions whose probability lies within 1e-5 of the
threshold (there the fp32 and fp64 sides may classify differently), its sums within 1e-5 per
position.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, bf16_dev, lib
from quantized_speculative_decoding_qspec_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

PROB_TOL = 1e-5


@pytest.fixture(scope="module")
def q():
    return lib()


def run_top1(q, tgt_bits, drf_bits, high=0.8, reps=2, ws=None):
    B, G1, V = tgt_bits.shape
    gamma = G1 - 1
    if ws is None:
        ws = q.new_verify_workspace(B, gamma, V)
    tt = torch.empty(B, gamma, dtype=torch.int32, device=DEV)
    dt = torch.empty(B, gamma, dtype=torch.int32, device=DEV)
    tp = torch.empty(B, gamma, dtype=torch.float32, device=DEV)
    dp = torch.empty(B, gamma, dtype=torch.float32, device=DEV)
    tally = torch.zeros(8, dtype=torch.float64, device=DEV)
    tgt, drf = bf16_dev(tgt_bits), bf16_dev(drf_bits)
    for _ in range(reps):  # the tally accumulates; the workspace is reusable without re-zeroing
        q.qspec_verify_top1(tgt, drf, tt, dt, ws, tgt_p1=tp, draft_p1=dp, high=high, tally=tally)
        q.qspec_check_status(ws)
    return (tt.cpu().numpy(), dt.cpu().numpy(), tp.cpu().numpy(), dp.cpu().numpy(),
            tally.cpu().numpy() / reps)


def check_top1(q, tgt_bits, drf_bits, high=0.8):
    got = run_top1(q, tgt_bits, drf_bits, high)
    ref = oracle.top1_stats(tgt_bits, drf_bits, high)
    assert np.array_equal(got[0], ref[0])
    assert np.array_equal(got[1], ref[1])
    for g, r in ((got[2], ref[2]), (got[3], ref[3])):
        assert np.abs(g.astype(np.float64) - r).max() <= PROB_TOL
    near = int(np.sum((np.abs(ref[2] - high) < PROB_TOL) | (np.abs(ref[3] - high) < PROB_TOL)))
    assert got[4][0] == ref[4][0] and got[4][1] == ref[4][1]
    assert np.abs(got[4][2:6] - ref[4][2:6]).max() <= near
    n = ref[4][0]
    assert np.abs(got[4][6:] - ref[4][6:]).max() <= PROB_TOL * n
    return ref


@pytest.mark.parametrize("B,gamma,V,sigma", [(1, 3, 128256, 0.5), (16, 3, 128256, 1.0), (2, 16, 4096, 0.5),
                                             (3, 3, 1001, 0.5), (5, 2, 2, 1.0), (4, 7, 152064, 2.0),
                                             (64, 3, 32000, 0.5)])
def test_top1_parity(q, B, gamma, V, sigma):
    inp = syn.verify_inputs(B, gamma, V, sigma, workload_id=300 + B * 5 + gamma, sampling=True)
    check_top1(q, inp["tgt"], inp["drf"])


def test_top1_both_regions_present(q):
    # a mix of confident and flat rows, so that both threshold regions and disagreements occur
    B, gamma, V = 8, 4, 20000
    inp = syn.verify_inputs(B, gamma, V, 2.0, workload_id=17, sampling=True)
    t = syn.bf16_bits_to_f32(inp["tgt"]).copy()
    d = syn.bf16_bits_to_f32(inp["drf"]).copy()
    t[::2, :, 11] += 30.0
    d[::2, :, 11] += 30.0
    ref = check_top1(q, syn.f32_to_bf16_bits(t), syn.f32_to_bf16_bits(d))
    assert ref[4][2] > 0 and ref[4][4] > 0


def test_top1_ties_and_inf(q):
    B, gamma, V = 2, 2, 3000
    rng = np.random.default_rng(3)
    t = rng.standard_normal((B, gamma + 1, V)).astype(np.float32)
    d = rng.standard_normal((B, gamma, V)).astype(np.float32)
    t[0, 0, [5, 2999, 1500]] = 50.0      # tie across chunks -> 5, p1 = 1/3 up to the rest
    d[0, 0, :] = 0.0                     # uniform -> index 0, p1 = 1/V
    t[0, 1, :] = -np.inf
    t[0, 1, 2500] = -1.0                 # single finite value -> p1 = 1
    d[1, 1, :] = -np.inf
    d[1, 1, [7, 9]] = 2.0                # two finite, equal -> 7, p1 = 1/2
    check_top1(q, syn.f32_to_bf16_bits(t), syn.f32_to_bf16_bits(d), high=0.5)


def test_top1_shares_workspace_with_greedy(q):
    # the per-sequence tickets are shared with the verify calls: interleaving leaves both correct
    B, gamma, V = 4, 3, 50000
    inp = syn.verify_inputs(B, gamma, V, 0.5, workload_id=23, sampling=True)
    ws = q.new_verify_workspace(B, gamma, V)
    n = torch.empty(B, dtype=torch.int32, device=DEV)
    out = torch.empty(B, gamma + 1, dtype=torch.int32, device=DEV)
    tgt, dd = bf16_dev(inp["tgt"]), torch.from_numpy(inp["d"].astype(np.int32)).to(DEV)
    rn, rout, _ = oracle.verify_greedy(inp["tgt"], inp["d"])
    ref = oracle.top1_stats(inp["tgt"], inp["drf"])
    for _ in range(2):
        q.qspec_verify_greedy(tgt, dd, n, out, ws)
        got = run_top1(q, inp["tgt"], inp["drf"], reps=1, ws=ws)
        assert np.array_equal(n.cpu().numpy(), rn) and np.array_equal(out.cpu().numpy(), rout)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
