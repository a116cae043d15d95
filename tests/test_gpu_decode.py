"""GPU parity of the decode-loop building blocks (f1) and of the loop itself, through the C ABI.

Gather: bit-exact.  Token selection: greedy bit-exact; sampling identical except where the oracle's
fp64 CDF lies within 1e-6 of u at the chosen boundary.  The toy model's layers: each linear against
the oracle on the GPU's own input to that layer (the a2 / a4 bars).  The loop: every iteration's
draft tokens, accept length and emitted tokens equal the oracle's decisions on the logits the GPU
produced; greedy speculative decoding emits exactly what target-only decoding emits.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, bf16_dev, bf16_host_bits, bf16_ulp_distance, f32_dev, i32_dev, lib
from quantized_speculative_decoding_qspec_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

DECISION_EPS = 1e-6


@pytest.fixture(scope="module")
def q():
    return lib()


@pytest.fixture(scope="module")
def dec(q):
    from quantized_speculative_decoding_qspec_gb300 import decode
    return decode


def cdf_margin(row_bits, u, j):
    p = oracle.softmax(oracle.bf16_to_f32(row_bits).astype(np.float64))
    c = np.cumsum(p)
    lo = c[j - 1] if j > 0 else 0.0
    return min(abs(c[j] - u), abs(u - lo))


# ---------------------------------------------------------------- gather

@pytest.mark.parametrize("n_src,row_elems,n", [(1000, 4096, 7), (50, 512, 64), (9, 1, 33), (6, 4, 5)])
def test_gather_rows(q, n_src, row_elems, n):
    rng = np.random.default_rng(n_src + n)
    src = rng.integers(-2 ** 31, 2 ** 31 - 1, size=(n_src, row_elems), dtype=np.int64).astype(np.int32)
    idx = rng.integers(0, n_src, size=n).astype(np.int32)
    s, i = i32_dev(src), i32_dev(idx)
    dst = torch.empty(n, row_elems, dtype=torch.int32, device=DEV)
    q.qspec_gather_rows(s, i, dst)
    q.qspec_check_status()
    assert np.array_equal(dst.cpu().numpy(), src[idx])


def test_gather_rows_out_of_range_reports(q):
    src = i32_dev(np.arange(8 * 256, dtype=np.int32).reshape(8, 256))
    dst = torch.full((3, 256), 7, dtype=torch.int32, device=DEV)
    q.qspec_gather_rows(src, i32_dev(np.array([1, 8, -1], np.int32)), dst)
    with pytest.raises(q.QSpecError) as e:
        q.qspec_check_status()
    assert e.value.code == 1  # QSPEC_ERR_INVALID_ARG
    got = dst.cpu().numpy()
    assert np.array_equal(got[0], np.arange(256, 512)) and not got[1:].any()
    q.qspec_check_status()  # cleared


# ---------------------------------------------------------------- token selection

@pytest.mark.parametrize("R,V", [(4, 128256), (3, 1001), (5, 2), (2, 152064), (16, 32000)])
def test_select_greedy(q, R, V):
    L = syn.target_logits_f32(R, V, workload_id=R * 13 + V % 97)
    L[0, [V // 3, V - 1]] = L[0].max() + 1.0         # a tie: the lower index
    bits = syn.f32_to_bf16_bits(L)
    tok = torch.empty(R, dtype=torch.int32, device=DEV)
    q.qspec_select_tokens(bf16_dev(bits), tok)
    q.qspec_check_status()
    want = [oracle.select_token(bits[r]) for r in range(R)]
    assert tok.cpu().numpy().tolist() == want


@pytest.mark.parametrize("R,V,flat", [(64, 128256, False), (64, 1001, False), (32, 32000, True), (16, 2, True),
                                      (8, 152064, True)])
def test_select_sampling(q, R, V, flat):
    L = syn.target_logits_f32(R, V, workload_id=7 + R + V % 89)
    if flat:
        L *= np.float32(0.05)                          # probability spread over the whole vocabulary
    bits = syn.f32_to_bf16_bits(L)
    u = syn.uniforms((R,), workload_id=R + V % 89, stream=syn.STREAM_U_DRAFT)
    u[0] = 0.0
    u[1] = np.float32(1 - 2.0 ** -24)
    tok = torch.empty(R, dtype=torch.int32, device=DEV)
    q.qspec_select_tokens(bf16_dev(bits), tok, u=f32_dev(u))
    q.qspec_check_status()
    got = tok.cpu().numpy()
    exact = 0
    for r in range(R):
        want = oracle.select_token(bits[r], u[r])
        if got[r] == want:
            exact += 1
        else:
            assert cdf_margin(bits[r], float(u[r]), want) < DECISION_EPS, (r, got[r], want)
    assert exact >= R - max(1, R // 16)


def test_select_degenerate_rows(q):
    # a row of only -inf gives token 0 (the documented choice: the distribution is undefined); a
    # single finite value is chosen by both rules whatever the uniform
    V = 4096
    L = np.full((3, V), -np.inf, dtype=np.float32)
    L[1, 1234] = -3.0
    L[2, V - 1] = 7.0
    bits = syn.f32_to_bf16_bits(L)
    tok = torch.empty(3, dtype=torch.int32, device=DEV)
    q.qspec_select_tokens(bf16_dev(bits), tok)
    assert tok.cpu().numpy().tolist() == [0, 1234, V - 1]
    q.qspec_select_tokens(bf16_dev(bits), tok, u=f32_dev(np.array([0.5, 0.999, 0.0], np.float32)))
    q.qspec_check_status()
    assert tok.cpu().numpy().tolist() == [0, 1234, V - 1]


# ---------------------------------------------------------------- the toy model and the loop

def small_model(dec, V=1000, workload_id=3):
    return dec.ToyModel(D=256, F=512, V=V, workload_id=workload_id, device=DEV)


def host_layers(model):
    return [(Wp.cpu().numpy(), S.cpu().numpy()) for Wp, S in model.layers]


@pytest.mark.parametrize("draft_mode", [False, True])
def test_toy_model_layers(q, dec, draft_mode):
    model = small_model(dec)
    tok = i32_dev(np.array([5, 999, 0, 417, 5], np.int32))
    logits = torch.empty(5, model.V, dtype=torch.bfloat16, device=DEV)
    model.forward(tok, logits, draft_mode)
    q.qspec_check_status()
    b = model._buffers(5)
    E = bf16_host_bits(model.E)
    x = bf16_host_bits(b["x"])
    assert np.array_equal(x, E[[5, 999, 0, 417, 5]])
    ins = [x, bf16_host_bits(b["h"][0]), bf16_host_bits(b["h"][1])]
    outs = ins[1:] + [bf16_host_bits(logits)]
    for (Wp, S), xin, y in zip(host_layers(model), ins, outs):
        got = oracle.bf16_to_f32(y).astype(np.float64)
        if draft_mode:
            ref = oracle.linear_w4a4(xin, Wp, S)["y"]
            assert bf16_ulp_distance(y, oracle.f64_to_bf16_bits(ref)).max() <= 1
        else:
            ref = oracle.linear_w4a16(xin, Wp, S)
            assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 5e-3


def check_iterations(res, gamma, sampling, workload_id):
    recs = res["records"]
    B = recs[0]["n"].shape[0]
    for it, r in enumerate(recs):
        d, n, out = r["d"], r["n"], r["out"]
        dl = bf16_host_bits(r["dl"])
        tl = bf16_host_bits(r["tl"])
        if it > 0:
            prev = recs[it - 1]
            want_in = prev["out"][np.arange(B), prev["n"]]
            assert np.array_equal(r["tokens_in"], want_in)
        if not sampling:
            for b in range(B):
                assert d[b].tolist() == [oracle.select_token(dl[b, i]) for i in range(gamma)]
            rn, rout, _ = oracle.verify_greedy(tl, d)
            assert np.array_equal(n, rn) and np.array_equal(out, rout)
        else:
            ud = syn.uniforms((gamma, B), workload_id, syn.STREAM_U_DRAFT, it)
            ua = syn.uniforms((B, gamma), workload_id, syn.STREAM_U_ACCEPT, it)
            ur = syn.uniforms((B, gamma + 1), workload_id, syn.STREAM_U_RESAMPLE, it)
            for b in range(B):
                for i in range(gamma):
                    want = oracle.select_token(dl[b, i], ud[i, b])
                    if d[b, i] != want:
                        assert cdf_margin(dl[b, i], float(ud[i, b]), want) < DECISION_EPS
            ref = oracle.verify_sample(tl, dl, d, ua, ur)
            for b in range(B):
                if n[b] != ref["accept_len"][b]:
                    i = min(n[b], ref["accept_len"][b])
                    assert ref["acc_margin"][b, i] < DECISION_EPS
                elif not np.array_equal(out[b], ref["out_tok"][b]):
                    assert ref["res_margin"][b] < DECISION_EPS
    gen = res["generated"]
    for b in range(B):
        want = [int(t) for r in recs for t in r["out"][b, :r["n"][b] + 1]]
        assert gen[b] == want


def check_target_logits(model, rec, tol=1e-2):
    """The verify pass's logits against the oracle's toy model on the same input tokens (three chained
    W4A16 layers, each output rounded to bf16: relative Frobenius error within 1e-2)."""
    tokens = np.concatenate([rec["tokens_in"][:, None], rec["d"]], axis=1).reshape(-1)
    E = bf16_host_bits(model.E)
    ref = oracle.bf16_to_f32(oracle.toy_forward(E, host_layers(model), tokens, False)).astype(np.float64)
    got = oracle.bf16_to_f32(bf16_host_bits(rec["tl"])).astype(np.float64).reshape(ref.shape)
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= tol


# (9, 3): the verify pass runs at M = 36, on the tensor-core linear; V = 16384 gives the last layer
# more output tiles than the first two, so layers sharing one workspace would corrupt its tickets.
# (5, 3): M = 20, the GEMV's 32 token slots.
@pytest.mark.parametrize("B,gamma,use_graphs,V", [(1, 3, True, 1000), (3, 2, True, 1000), (2, 4, False, 1000),
                                                  (9, 3, True, 16384), (5, 3, True, 16384)])
def test_decode_loop_greedy(q, dec, B, gamma, use_graphs, V):
    model = small_model(dec, V=V)
    sd = dec.SpecDecoder(model, B, gamma, use_graphs=use_graphs)
    first = np.arange(B, dtype=np.int32) * 37 + 1
    res = sd.run(first, n_iter=6, record=True)
    check_iterations(res, gamma, False, 0)
    check_target_logits(model, res["records"][0])
    check_target_logits(model, res["records"][-1])
    # output equivalence: greedy speculative decoding emits exactly what the target alone emits
    n_tok = min(len(g) for g in res["generated"])
    base = sd.run_target_only(first, n_tok, padded=True)
    for b in range(B):
        assert res["generated"][b][:n_tok] == base["generated"][b]
    # top-1 tally: positions counted once per draft position, agreement as the oracle counts it
    t = res["tally"]
    assert t[0] == 6 * B * gamma
    agree = 0
    for r in res["records"]:
        tt, dd, _, _, _ = oracle.top1_stats(bf16_host_bits(r["tl"]), bf16_host_bits(r["dl"]))
        agree += int(np.sum(tt == dd))
    assert t[1] == agree


@pytest.mark.parametrize("B,gamma", [(1, 3), (4, 3)])
def test_decode_loop_sampling(q, dec, B, gamma):
    model = small_model(dec, workload_id=4)
    sd = dec.SpecDecoder(model, B, gamma, sampling=True)
    res = sd.run(np.arange(B, dtype=np.int32) + 10, n_iter=5, workload_id=9, record=True)
    check_iterations(res, gamma, True, 9)


def test_decode_summary(q, dec):
    model = small_model(dec)
    sd = dec.SpecDecoder(model, 1, 3)
    spec = sd.run([1], n_iter=5)
    base = sd.run_target_only([1], 8)
    s = dec.summarize(spec, base, 3)
    assert 1.0 <= s["accepted_tokens_per_iteration"] <= 4.0
    assert 0.0 <= s["acceptance_rate"] <= 1.0
    assert s["t_verify_ms"] > 0 and s["t_draft_ms_per_token"] > 0 and s["speedup_model"] > 0
    assert s["top1"]["positions"] == 15
