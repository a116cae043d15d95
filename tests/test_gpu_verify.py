"""GPU parity of the verify step (a5-a8) against the CPU oracle, through the C ABI.

Greedy: accept lengths, emitted tokens and target argmaxes are bit-exact.
Sampling: exposed probabilities (a_i, p_i(d_i), q_i(d_i)) within 1e-5 absolute of the fp64 oracle;
accept/reject decisions identical except where |u - a| < 1e-6; the resampled token identical
except where the oracle's CDF step bounding it lies within 1e-6 * R of u * R.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, bf16_dev, f32_dev, i32_dev, lib
from quantized_speculative_decoding_qspec_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

PROB_TOL = 1e-5
DECISION_EPS = 1e-6


@pytest.fixture(scope="module")
def q():
    return lib()


def run_greedy(q, tgt_bits, d):
    B, G1, V = tgt_bits.shape
    ws = q.new_verify_workspace(B, G1 - 1, V)
    n = torch.empty(B, dtype=torch.int32, device=DEV)
    out = torch.empty(B, G1, dtype=torch.int32, device=DEV)
    t = torch.empty(B, G1, dtype=torch.int32, device=DEV)
    tgt = bf16_dev(tgt_bits)
    dd = i32_dev(d)
    for _ in range(2):  # the workspace is reusable without re-zeroing
        q.qspec_verify_greedy(tgt, dd, n, out, ws, tgt_argmax=t)
        q.qspec_check_status(ws)
    return n.cpu().numpy(), out.cpu().numpy(), t.cpu().numpy()


def check_greedy(q, tgt_bits, d):
    n, out, t = run_greedy(q, tgt_bits, d)
    rn, rout, rt = oracle.verify_greedy(tgt_bits, d)
    assert np.array_equal(t, rt)
    assert np.array_equal(n, rn)
    assert np.array_equal(out, rout)
    return rn


@pytest.mark.parametrize("B,gamma,V,sigma", [(1, 3, 1024, 0.5), (1, 3, 128256, 0.5), (16, 3, 128256, 0.5), (4, 1, 32000, 1.0),
                                             (3, 16, 4096, 0.25), (2, 7, 152064, 0.5), (5, 3, 1001, 0.5),
                                             (7, 2, 2, 1.0), (1, 5, 9, 0.5)])
def test_greedy_parity(q, B, gamma, V, sigma):
    inp = syn.verify_inputs(B, gamma, V, sigma, workload_id=B * 31 + gamma)
    check_greedy(q, inp["tgt"], inp["d"])


def test_greedy_all_accept_and_first_reject(q):
    B, gamma, V = 6, 4, 5000
    inp = syn.verify_inputs(B, gamma, V, 0.5, workload_id=2)
    rt = oracle.verify_greedy(inp["tgt"], inp["d"])[2]
    d = rt[:, :gamma].copy()
    d[1, 0] = (d[1, 0] + 1) % V          # reject at 0
    d[2, 2] = (d[2, 2] + 1) % V          # reject at 2
    n = check_greedy(q, inp["tgt"], d)
    assert n[0] == gamma and n[1] == 0 and n[2] == 2


def test_greedy_ties_zeros_and_inf(q):
    B, gamma, V = 2, 2, 3000
    L = np.random.default_rng(0).standard_normal((B, gamma + 1, V)).astype(np.float32)
    L[0, 0, [5, 2999, 1500]] = 50.0                  # tie across chunks -> 5
    L[0, 1, :] = -0.0
    L[0, 1, [7, 2048]] = 0.0                         # all zeros of both signs -> 0
    L[0, 2, :] = -np.inf
    L[0, 2, 2500] = -1.0                             # single finite value
    L[1, :, :] = -np.inf                             # all -inf -> index 0
    check_greedy(q, syn.f32_to_bf16_bits(L), np.array([[5, 0], [0, 1]]))


def test_greedy_invalid_token_reports(q):
    B, gamma, V = 1, 3, 1024
    inp = syn.verify_inputs(B, gamma, V, 0.5)
    d = inp["d"].copy()
    d[0, 1] = V + 5
    ws = q.new_verify_workspace(B, gamma, V)
    n = torch.empty(B, dtype=torch.int32, device=DEV)
    out = torch.empty(B, gamma + 1, dtype=torch.int32, device=DEV)
    q.qspec_verify_greedy(bf16_dev(inp["tgt"]), i32_dev(d), n, out, ws)
    with pytest.raises(q.QSpecError) as e:
        q.qspec_check_status(ws)
    assert e.value.code == 1
    assert n.item() <= 1
    q.qspec_check_status(ws)  # the error word was cleared


# ----------------------------------------------------------------------------- sampling


def run_sample(q, inp, reps=2):
    tgt, drf, d, ua, ur = inp["tgt"], inp["drf"], inp["d"], inp["u_acc"], inp["u_res"]
    B, G1, V = tgt.shape
    gamma = G1 - 1
    ws = q.new_verify_workspace(B, gamma, V)
    n = torch.empty(B, dtype=torch.int32, device=DEV)
    out = torch.empty(B, G1, dtype=torch.int32, device=DEV)
    a = torch.empty(B, gamma, dtype=torch.float32, device=DEV)
    p = torch.empty(B, gamma, dtype=torch.float32, device=DEV)
    qq = torch.empty(B, gamma, dtype=torch.float32, device=DEV)
    args = (bf16_dev(tgt), bf16_dev(drf), i32_dev(d), f32_dev(ua), f32_dev(ur))
    for _ in range(reps):
        q.qspec_verify_sample(*args, n, out, ws, accept_prob=a, p_tok=p, q_tok=qq)
        q.qspec_check_status(ws)
    return {"accept_len": n.cpu().numpy(), "out_tok": out.cpu().numpy(), "accept_prob": a.cpu().numpy(),
            "p_tok": p.cpu().numpy(), "q_tok": qq.cpu().numpy()}


def compare_sample(got, ref, u_acc):
    """Assert parity under the decision tolerances; returns the number of sequences compared exactly."""
    for k in ("accept_prob", "p_tok", "q_tok"):
        err = np.abs(got[k].astype(np.float64) - ref[k]).max()
        assert err <= PROB_TOL, f"{k}: {err}"
    B = got["accept_len"].shape[0]
    exact = 0
    for b in range(B):
        gn, rn = int(got["accept_len"][b]), int(ref["accept_len"][b])
        if gn != rn:
            i = min(gn, rn)  # first position where the decisions differ
            assert ref["acc_margin"][b, i] < DECISION_EPS, f"seq {b}: n {gn} vs {rn}"
            continue
        if not np.array_equal(got["out_tok"][b], ref["out_tok"][b]):
            assert np.array_equal(got["out_tok"][b, :gn], ref["out_tok"][b, :rn])
            assert ref["res_margin"][b] < DECISION_EPS, f"seq {b}: resampled {got['out_tok'][b]} vs {ref['out_tok'][b]}"
            continue
        exact += 1
    return exact


SAMPLE_CASES = [(1, 3, 1024, 0.5), (1, 3, 128256, 0.5), (8, 3, 32000, 0.5), (8, 1, 128256, 1.0), (4, 7, 152064, 0.25),
                (8, 5, 32000, 1.0), (2, 16, 4096, 0.5), (3, 3, 1001, 0.5), (5, 2, 2, 1.0), (64, 3, 32000, 0.5)]


@pytest.mark.parametrize("B,gamma,V,sigma", SAMPLE_CASES)
def test_sample_parity(q, B, gamma, V, sigma):
    inp = syn.verify_inputs(B, gamma, V, sigma, workload_id=100 + B * 7 + gamma, sampling=True)
    got = run_sample(q, inp)
    ref = oracle.verify_sample(inp["tgt"], inp["drf"], inp["d"], inp["u_acc"], inp["u_res"])
    exact = compare_sample(got, ref, inp["u_acc"])
    assert exact >= B - max(1, B // 16)


def test_sample_bonus_and_certain_reject(q):
    # u_acc = 0 accepts everything whose a > 0 (bonus token path); u_acc -> 1 rejects unless a == 1
    B, gamma, V = 6, 3, 20000
    inp = syn.verify_inputs(B, gamma, V, 0.5, workload_id=9, sampling=True)
    inp["u_acc"][:3] = 0.0
    inp["u_acc"][3:] = np.float32(1 - 2.0 ** -24)
    got = run_sample(q, inp)
    ref = oracle.verify_sample(inp["tgt"], inp["drf"], inp["d"], inp["u_acc"], inp["u_res"])
    compare_sample(got, ref, inp["u_acc"])
    assert (got["accept_len"][:3] == gamma).all()


def test_sample_residual_falls_back_to_p(q):
    # identical target and draft rows: the residual has no mass; the draw uses p
    B, gamma, V = 2, 2, 3000
    inp = syn.verify_inputs(B, gamma, V, 0.5, workload_id=11, sampling=True)
    inp["drf"] = inp["tgt"][:, :gamma].copy()
    inp["u_acc"][:] = np.float32(1 - 2.0 ** -24)   # a == 1 everywhere, still accepted (u < 1)
    got = run_sample(q, inp)
    ref = oracle.verify_sample(inp["tgt"], inp["drf"], inp["d"], inp["u_acc"], inp["u_res"])
    compare_sample(got, ref, inp["u_acc"])


def test_expected_tokens_on_gpu(q):
    # constant acceptance alpha: draft logits (0, -inf) propose token 0 with q = 1; target logits
    # (ln alpha, ln(1 - alpha)) give p(0) = alpha.  Mean tokens per call -> (1 - a^(g+1)) / (1 - a).
    gamma, alpha, B, V = 4, 0.8, 40000, 2
    tgt = np.tile(np.array([math.log(alpha), math.log(1 - alpha)], np.float32), (B, gamma + 1, 1))
    drf = np.tile(np.array([0.0, -np.inf], np.float32), (B, gamma, 1))
    tb, db = syn.f32_to_bf16_bits(tgt), syn.f32_to_bf16_bits(drf)
    tq = syn.bf16_bits_to_f32(tb[0, 0]).astype(np.float64)
    alpha_eff = float(oracle.softmax(tq)[0])
    inp = {"tgt": tb, "drf": db, "d": np.zeros((B, gamma), np.int32),
           "u_acc": syn.uniforms((B, gamma), 5, syn.STREAM_U_ACCEPT),
           "u_res": syn.uniforms((B, gamma + 1), 5, syn.STREAM_U_RESAMPLE)}
    got = run_sample(q, inp, reps=1)
    T = got["accept_len"].astype(np.float64) + 1
    se = T.std() / math.sqrt(B)
    assert abs(T.mean() - oracle.expected_tokens(alpha_eff, gamma)) < 4 * se
    assert np.abs(got["accept_prob"] - alpha_eff).max() < PROB_TOL


def test_sample_long_vocab_two_scan_tiles(q):
    # V = 300000: 147 chunks of 2048, 1176 warp segments, so the last CTA's scan of the segment sums
    # runs over two tiles of 1024; u_res near 0, mid, near 1 put the crossing in either tile
    B, gamma, V = 4, 2, 300000
    inp = syn.verify_inputs(B, gamma, V, 0.5, workload_id=12, sampling=True)
    for b, u in enumerate((0.3, 0.95, 0.999, 0.01)):
        inp["u_res"][b, :] = np.float32(u)
    got = run_sample(q, inp)
    ref = oracle.verify_sample(inp["tgt"], inp["drf"], inp["d"], inp["u_acc"], inp["u_res"])
    exact = compare_sample(got, ref, inp["u_acc"])
    assert exact >= B - 1


def test_sample_parity_largest_sweep_cell(q):
    # the largest cell of the sampling sweep: 64 sequences, gamma = 7, V = 152064 (1920 CTAs in pass 1,
    # two vocabulary chunks per row)
    B, gamma, V, sigma = 64, 7, 152064, 0.5
    inp = syn.verify_inputs(B, gamma, V, sigma, workload_id=104, sampling=True)
    got = run_sample(q, inp, reps=1)
    ref = oracle.verify_sample(inp["tgt"], inp["drf"], inp["d"], inp["u_acc"], inp["u_res"])
    exact = compare_sample(got, ref, inp["u_acc"])
    assert exact >= B - max(1, B // 16)
