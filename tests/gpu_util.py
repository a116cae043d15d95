"""Helpers for GPU parity tests: move seeded numpy inputs to the device and back."""
import numpy as np
import torch

DEV = "cuda"


def lib():
    import __graft_entry__ as g
    g.build()
    from quantized_speculative_decoding_qspec_gb300 import qspec as q
    q.load()
    return q


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def i32_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(DEV)


def f32_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DEV)


def bf16_host_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_host_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def packed_dev(q, W_bits):
    """Pack on the GPU: returns (Wp, S) device tensors."""
    N, K = W_bits.shape
    Wp = torch.empty(N, K // 2, dtype=torch.uint8, device=DEV)
    S = torch.empty(N, K // 128, dtype=torch.float16, device=DEV)
    q.qspec_pack_weights(bf16_dev(W_bits), Wp, S)
    return Wp, S


def rel_fro(got, ref):
    den = np.linalg.norm(ref)
    return np.linalg.norm(got - ref) / (den if den > 0 else 1.0)


def bf16_ulp_distance(a_bits, b_bits):
    """|difference| in units in the last place between bf16 bit patterns (monotone integer map)."""
    def key(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + b)
    return np.abs(key(a_bits) - key(b_bits))
