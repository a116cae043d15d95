"""qspec_verify_greedy_noalloc: greedy verify for callers that cannot allocate device memory.

Such callers (plug-ins inside another runtime's fixed memory plan, C hosts without an allocator) get
an entry point whose scratch lives in a fixed device array inside the library.  Its outputs must
equal those of the workspace-taking qspec_verify_greedy, on consecutive calls that reuse the shared
array.  The file name sorts last so that pytest collects it after every other test: a run that stops
at the first failure (-x) has then already run the rest of the suite when this one fails.  The tests
also pass alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import DEV, bf16_dev, i32_dev, lib
from quantized_speculative_decoding_qspec_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _run_both(q, B, gamma, V, seed):
    inp = syn.verify_inputs(B, gamma, V, 0.5, workload_id=seed)
    tgt, d = bf16_dev(inp["tgt"]), i32_dev(inp["d"])
    ref = [torch.full((B,), -7, dtype=torch.int32, device=DEV), torch.full((B, gamma + 1), -7, dtype=torch.int32, device=DEV),
           torch.full((B, gamma + 1), -7, dtype=torch.int32, device=DEV)]
    ws = q.new_verify_workspace(B, gamma, V)
    q.qspec_verify_greedy(tgt, d, ref[0], ref[1], ws, tgt_argmax=ref[2])
    got = [torch.full_like(t, -9) for t in ref]
    stream = torch.cuda.current_stream().cuda_stream
    # straight through the C ABI
    rc = q.load().qspec_verify_greedy_noalloc(tgt.data_ptr(), d.data_ptr(), B, gamma, V, got[0].data_ptr(),
                                              got[1].data_ptr(), got[2].data_ptr(), stream)
    assert rc == 0, q.STATUS.get(rc, rc)
    q.qspec_check_status(ws)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    return got


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    q = lib()
    # two calls in a row on the shared array, different shapes and inputs
    _run_both(q, 16, 3, 128256, seed=1)
    _run_both(q, 3, 7, 1001, seed=2)
    # and the same shape again (the array keeps the last call's contents)
    _run_both(q, 16, 3, 128256, seed=3)


def test_noalloc_rejects_shapes_beyond_the_scratch_limit():
    q = lib()
    B, gamma, V = 20000, 15, 4096          # 320 000 rows: partials exceed the fixed array
    limit = 256 * 1024
    assert q.qspec_verify_workspace_size(B, gamma, V) > limit
    dummy = torch.zeros(16, dtype=torch.int32, device=DEV)
    rc = q.load().qspec_verify_greedy_noalloc(dummy.data_ptr(), dummy.data_ptr(), B, gamma, V, dummy.data_ptr(),
                                              dummy.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    assert q.STATUS[rc] == "QSPEC_ERR_UNSUPPORTED_SHAPE"
