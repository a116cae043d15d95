"""Seeded synthetic inputs for the QSpec hot path.

This module only draws random inputs.  It contains none of the method's arithmetic (no
quantisation, no softmax, no verification), so the CPU oracle and the CUDA path can both be fed
from it without sharing any of the computation they are compared on.

Every stream comes from ``numpy.random.default_rng([workload_id, stream_id])``.  Floating inputs are
drawn in fp32 and rounded to bfloat16 (round to nearest, ties to even); bfloat16 tensors are
returned as their uint16 bit patterns so that no library's bf16 conversion is involved.

Distributions (the workloads of the QSpec top-1 agreement article, "QSpec実行時の2つの量子化による推論の
一致率を調べる", §実験条件 -- Llama-3-8B decoding with draft length 3 -- replaced by seeded stand-ins):

* weights: N(0, 0.02), one [N, K] matrix per linear layer;
* activations: N(0, 1) per token, with round(0.01*K) outlier channels (the same channels for every
  token) scaled by 20;
* target logits: N(0, 1) plus a U(4, 12) spike on one uniformly chosen token per row;
* draft logits: target logits plus N(0, sigma) on every element;
* uniforms: ``integers(0, 2**24) * 2**-24``, exact fp32 values in [0, 1);
* the decode loop's toy model: an N(0, 1) token embedding table and N(0, 0.02) weights per linear.
"""
from __future__ import annotations

import numpy as np

# Stream ids: one independent stream per kind of input.
STREAM_WEIGHTS = 1
STREAM_ACTIVATIONS = 2
STREAM_OUTLIERS = 3
STREAM_LOGITS = 4
STREAM_SPIKE_INDEX = 5
STREAM_SPIKE_HEIGHT = 6
STREAM_DRAFT_NOISE = 7
STREAM_DRAFT_SAMPLE = 8
STREAM_U_ACCEPT = 9
STREAM_U_RESAMPLE = 10
STREAM_EMBEDDINGS = 11
STREAM_U_DRAFT = 12


def rng(workload_id: int, stream_id: int, sub: int = 0) -> np.random.Generator:
    """The generator for one (workload, stream[, sub-stream]) triple."""
    return np.random.default_rng([int(workload_id), int(stream_id), int(sub)])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bfloat16 (nearest, ties to even); returns uint16 bit patterns.

    NaN maps to the canonical quiet NaN 0x7FC0; +-inf and overflow map to +-inf.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    step = 1 << 24
    for i in range(0, flat.size, step):  # bounded temporaries for large tensors
        f = flat[i:i + step]
        u = f.view(np.uint32)
        nan = np.isnan(f)
        # finite inputs: u + 0x7FFF + lsb stays below 2**32, so uint32 arithmetic is exact
        r = ((np.where(nan, np.uint32(0), u) + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
             >> np.uint32(16)).astype(np.uint16)
        if nan.any():
            r = np.where(nan, np.uint16(0x7FC0), r)
        out[i:i + step] = r
    return out.reshape(x.shape)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to fp32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def weights(N: int, K: int, workload_id: int = 0, layer: int = 0, std: float = 0.02) -> np.ndarray:
    """bf16 bits of an [N, K] weight matrix (out x in, K contiguous), N(0, std)."""
    g = rng(workload_id, STREAM_WEIGHTS, layer)
    w = g.standard_normal((N, K), dtype=np.float32)
    w *= np.float32(std)
    return f32_to_bf16_bits(w)


def embeddings(V: int, D: int, workload_id: int = 0, std: float = 1.0) -> np.ndarray:
    """bf16 bits of a [V, D] token embedding table, N(0, std)."""
    g = rng(workload_id, STREAM_EMBEDDINGS)
    e = g.standard_normal((V, D), dtype=np.float32)
    if std != 1.0:
        e *= np.float32(std)
    return f32_to_bf16_bits(e)


def outlier_channels(K: int, workload_id: int = 0, frac: float = 0.01) -> np.ndarray:
    """Sorted indices of the round(frac*K) outlier input channels."""
    n_out = int(round(frac * K))
    g = rng(workload_id, STREAM_OUTLIERS)
    return np.sort(g.choice(K, size=n_out, replace=False)) if n_out > 0 else np.zeros(0, np.int64)


def activations(M: int, K: int, workload_id: int = 0, step: int = 0, scale: float = 20.0) -> np.ndarray:
    """bf16 bits of [M, K] activations: N(0, 1) with the outlier channels scaled by ``scale``."""
    g = rng(workload_id, STREAM_ACTIVATIONS, step)
    x = g.standard_normal((M, K), dtype=np.float32)
    ch = outlier_channels(K, workload_id)
    x[:, ch] *= np.float32(scale)
    return f32_to_bf16_bits(x)


def target_logits_f32(R: int, V: int, workload_id: int = 0, step: int = 0,
                      spike_lo: float = 4.0, spike_hi: float = 12.0) -> np.ndarray:
    """fp32 target logits [R, V]: N(0, 1) plus a U(spike_lo, spike_hi) spike on one token per row."""
    l = rng(workload_id, STREAM_LOGITS, step).standard_normal((R, V), dtype=np.float32)
    idx = rng(workload_id, STREAM_SPIKE_INDEX, step).integers(0, V, size=R)
    h = rng(workload_id, STREAM_SPIKE_HEIGHT, step).uniform(spike_lo, spike_hi, size=R).astype(np.float32)
    l[np.arange(R), idx] += h
    return l


def draft_logits_f32(target_f32: np.ndarray, sigma: float, workload_id: int = 0, step: int = 0) -> np.ndarray:
    """Draft logits: target plus N(0, sigma) noise on every element (fp32)."""
    noise = rng(workload_id, STREAM_DRAFT_NOISE, step).standard_normal(target_f32.shape, dtype=np.float32)
    return target_f32 + np.float32(sigma) * noise


def first_max_index(values: np.ndarray) -> np.ndarray:
    """Index of the largest value along the last axis (the lowest index among equal maxima).

    Used to stand in for a greedy draft model's token choice.
    """
    v = np.asarray(values)
    mx = v.max(axis=-1, keepdims=True)
    return np.argmax(v == mx, axis=-1).astype(np.int32)


def gumbel_sample(logits_f32: np.ndarray, workload_id: int = 0, step: int = 0) -> np.ndarray:
    """A sample from softmax(logits) per row, drawn with the Gumbel-max construction.

    Stands in for a sampling draft model; it never forms the softmax itself.
    """
    u = rng(workload_id, STREAM_DRAFT_SAMPLE, step).random(logits_f32.shape)
    u = np.clip(u, 1e-300, 1.0)
    gumbel = -np.log(-np.log(u))
    return first_max_index(logits_f32.astype(np.float64) + gumbel)


def uniforms(shape, workload_id: int = 0, stream: int = STREAM_U_ACCEPT, step: int = 0) -> np.ndarray:
    """Exact fp32 uniforms in [0, 1): integers(0, 2**24) * 2**-24."""
    k = rng(workload_id, stream, step).integers(0, 1 << 24, size=shape)
    return (k.astype(np.float64) * 2.0 ** -24).astype(np.float32)


def verify_inputs(B: int, gamma: int, V: int, sigma: float, workload_id: int = 0, step: int = 0,
                  sampling: bool = False):
    """One batch of verify inputs.

    Returns a dict with bf16 bits ``tgt`` [B, gamma+1, V] and ``drf`` [B, gamma, V], int32 draft
    tokens ``d`` [B, gamma] (the draft argmax, or a draft sample when ``sampling``), and exact fp32
    uniforms ``u_acc`` [B, gamma] and ``u_res`` [B, gamma+1].
    """
    t = target_logits_f32(B * (gamma + 1), V, workload_id, step).reshape(B, gamma + 1, V)
    t_bits = f32_to_bf16_bits(t)
    t_q = bf16_bits_to_f32(t_bits)
    d = draft_logits_f32(t_q[:, :gamma, :], sigma, workload_id, step)
    d_bits = f32_to_bf16_bits(d)
    d_q = bf16_bits_to_f32(d_bits)
    if sampling:
        toks = gumbel_sample(d_q.reshape(B * gamma, V), workload_id, step).reshape(B, gamma)
    else:
        toks = first_max_index(d_q).reshape(B, gamma)
    return {
        "tgt": t_bits,
        "drf": d_bits,
        "d": np.ascontiguousarray(toks, dtype=np.int32),
        "u_acc": uniforms((B, gamma), workload_id, STREAM_U_ACCEPT, step),
        "u_res": uniforms((B, gamma + 1), workload_id, STREAM_U_RESAMPLE, step),
    }
