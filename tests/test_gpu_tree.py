"""GPU parity of greedy tree verification (f4) against the CPU oracle, through the C ABI.

Accept lengths, emitted tokens and accepted node ids are bit-exact.  Trees are seeded: each node's
parent is the prefix or an earlier node, and its token is, with probability 0.7, the target's most
likely token after its parent (so long paths are accepted), otherwise a random token.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, bf16_dev, i32_dev, lib
from quantized_speculative_decoding_qspec_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    return lib()


def make_tree(B, T, V, seed, chain=False):
    tgt = syn.f32_to_bf16_bits(syn.target_logits_f32(B * (T + 1), V, workload_id=seed).reshape(B, T + 1, V))
    f = syn.bf16_bits_to_f32(tgt)
    rng = np.random.default_rng(seed)
    tok = np.zeros((B, T), np.int32)
    par = np.zeros((B, T), np.int32)
    for b in range(B):
        for j in range(T):
            p = j - 1 if chain else int(rng.integers(-1, j)) if j > 0 else -1
            par[b, j] = p
            best = int(syn.first_max_index(f[b, p + 1]))
            tok[b, j] = best if rng.random() < 0.7 else int(rng.integers(0, V))
    return tgt, tok, par


def run_tree(q, tgt, tok, par, reps=2):
    B, R, V = tgt.shape
    T = R - 1
    ws = q.new_tree_workspace(B, T, V)
    n = torch.empty(B, dtype=torch.int32, device=DEV)
    out = torch.empty(B, R, dtype=torch.int32, device=DEV)
    nodes = torch.empty(B, T, dtype=torch.int32, device=DEV)
    args = (bf16_dev(tgt), i32_dev(tok), i32_dev(par))
    for _ in range(reps):  # the workspace is reusable without re-zeroing
        q.qspec_verify_tree_greedy(*args, n, out, ws, accept_nodes=nodes)
        q.qspec_check_status(ws)
    return n.cpu().numpy(), out.cpu().numpy(), nodes.cpu().numpy()


@pytest.mark.parametrize("B,T,V", [(4, 1, 1001), (4, 7, 32000), (3, 15, 128256), (2, 63, 4096), (2, 64, 32000),
                                   (8, 5, 2)])
def test_tree_parity(q, B, T, V):
    tgt, tok, par = make_tree(B, T, V, seed=B * 100 + T)
    got = run_tree(q, tgt, tok, par)
    ref = oracle.verify_tree_greedy(tgt, tok, par)
    for g, r in zip(got, ref):
        assert np.array_equal(g, r)


def test_tree_chain_equals_greedy(q):
    B, T, V = 4, 6, 32000
    tgt, tok, par = make_tree(B, T, V, seed=7, chain=True)
    n, out, nodes = run_tree(q, tgt, tok, par)
    ws = q.new_verify_workspace(B, T, V)
    gn = torch.empty(B, dtype=torch.int32, device=DEV)
    gout = torch.empty(B, T + 1, dtype=torch.int32, device=DEV)
    q.qspec_verify_greedy(bf16_dev(tgt), i32_dev(tok), gn, gout, ws)
    q.qspec_check_status(ws)
    assert np.array_equal(n, gn.cpu().numpy()) and np.array_equal(out, gout.cpu().numpy())


def test_tree_invalid_nodes_report(q):
    B, T, V = 1, 3, 3000
    tgt, tok, par = make_tree(B, T, V, seed=9)
    tok[0, 0] = V + 5          # token out of range
    par[0, 1] = 2              # parent after the node
    ws = q.new_tree_workspace(B, T, V)
    n = torch.empty(B, dtype=torch.int32, device=DEV)
    out = torch.empty(B, T + 1, dtype=torch.int32, device=DEV)
    q.qspec_verify_tree_greedy(bf16_dev(tgt), i32_dev(tok), i32_dev(par), n, out, ws)
    with pytest.raises(q.QSpecError):
        q.qspec_check_status(ws)
    rn, rout, _ = oracle.verify_tree_greedy(tgt, tok, par)
    assert np.array_equal(n.cpu().numpy(), rn) and np.array_equal(out.cpu().numpy(), rout)
