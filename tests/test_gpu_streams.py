"""Independent calls on two CUDA streams at once (separate workspaces) give the same results as one
at a time: the library keeps no per-call state outside the caller's workspaces."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, bf16_dev, bf16_host_bits, bf16_ulp_distance, i32_dev, lib, packed_dev
from quantized_speculative_decoding_qspec_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    return lib()


def test_two_streams(q):
    N, K, V, B, gamma = 1000, 1152, 20000, 3, 3
    W = syn.weights(N, K, 41)
    Wp, S = packed_dev(q, W)
    Wp_ref, S_ref = oracle.pack_weights(W)
    jobs = []
    for k, (M, mode) in enumerate(((1, "a4"), (20, "a16"))):
        X = syn.activations(M, K, 41, step=k)
        inp = syn.verify_inputs(B, gamma, V, 0.5, workload_id=50 + k)
        jobs.append({"M": M, "mode": mode, "X": X, "x": bf16_dev(X), "inp": inp,
                     "tgt": bf16_dev(inp["tgt"]), "d": i32_dev(inp["d"]),
                     "y": torch.empty(M, N, dtype=torch.bfloat16, device=DEV),
                     "lws": q.new_linear_workspace(M, N, K), "vws": q.new_verify_workspace(B, gamma, V),
                     "n": torch.empty(B, dtype=torch.int32, device=DEV),
                     "out": torch.empty(B, gamma + 1, dtype=torch.int32, device=DEV),
                     "stream": torch.cuda.Stream()})
    torch.cuda.synchronize()
    for _ in range(20):  # interleave the two streams' launches
        for j in jobs:
            fn = q.qspec_linear_w4a4 if j["mode"] == "a4" else q.qspec_linear_w4a16
            fn(j["x"], Wp, S, j["y"], j["lws"], stream=j["stream"])
            q.qspec_verify_greedy(j["tgt"], j["d"], j["n"], j["out"], j["vws"], stream=j["stream"])
    for j in jobs:
        q.qspec_check_status(j["vws"], stream=j["stream"])
        rn, rout, _ = oracle.verify_greedy(j["inp"]["tgt"], j["inp"]["d"])
        assert np.array_equal(j["n"].cpu().numpy(), rn) and np.array_equal(j["out"].cpu().numpy(), rout)
        if j["mode"] == "a4":
            r = oracle.linear_w4a4(j["X"], Wp_ref, S_ref)
            assert bf16_ulp_distance(bf16_host_bits(j["y"]), oracle.f64_to_bf16_bits(r["y"])).max() <= 1
        else:
            ref = oracle.linear_w4a16(j["X"], Wp_ref, S_ref)
            got = oracle.bf16_to_f32(bf16_host_bits(j["y"])).astype(np.float64)
            assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 5e-3
