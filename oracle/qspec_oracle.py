"""Plain CPU oracle for the QSpec hot path.  TEST INFRASTRUCTURE, NOT PRODUCT CODE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import this module.  The library under ``quantized_speculative_decoding_qspec_gb300``
never imports it and shares no code with it; the two only see the same seeded inputs.

Everything is written for a reader checking it against the method by eye: numpy with fp64 wherever
a real number is meant, fp32 only where the quantiser definition fixes fp32 arithmetic, no blocking,
no fusion, Python loops where the method is a sequential rule.

Sources (web pages; cited by title and section):

* [QSpec-article]  "QSpec実行時の2つの量子化による推論の一致率を調べる" (qiita.com/joule), sections
  "W4A4 と W4A16 量子化" (W4A16: 4-bit weights converted while multiplying 16-bit activations;
  W4A4: weights and activations both 4-bit) and "QSpec の W4A4 モードと W4A16 モード" (one shared
  4-bit weight set serves both modes).
* [SD+Q summary]  the summary of a study of speculative decoding with quantisation (aibr.jp),
  section "中核となる技術的要素" (names W4A16 and W4A8 configurations).
* [SD-tutorial]  "Speculative Decodingとは？LLM生成を速くする方法" (kasblo.com), sections
  "greedy decodingでは一致するprefixを採用する" (greedy rule), "samplingでもtargetの確率分布を保つ"
  (eq. a(x) = min(1, p(x)/q(x)) and the residual eq. p'(x)), "3 tokenの数値例" (worked example) and
  "1回のtarget検証で何token進むか" (E[T] closed form).

Readings where the pages are silent (each is listed in the design notes of the repository):

* Weight quantiser: symmetric, per group of 128 input channels along K, divisor 7, scale rounded to
  fp16 before the codes are formed, codes = clamp(rint(w / s), -8, 7) with ties to even, s == 0
  gives all-zero codes.  Packed layout (the pages fix no bit order): each 32-bit little-endian
  word t of a row holds k = 8t..8t+7 as two's complement nibbles, the even channels k = 8t+0,2,4,6
  in nibbles 0..3 (bits 0..15) and the odd channels k = 8t+1,3,5,7 in nibbles 4..7 (bits 16..31).
* Activation quantiser: one fp32 scale per token over all of K, s_a = amax / 7 (not rounded to
  fp16), codes = clamp(rint(x / s_a), -8, 7); s_a == 0 gives all-zero codes.
* Greedy argmax compares bf16 logit values; ties (and +0 / -0) go to the lowest index.
* Sampling: temperature 1, one acceptance uniform per draft position, one resampling uniform per
  position indexed by the first rejected position n (or gamma for the bonus token), inverse CDF in
  index order with a strict ">" test, a = 1 when q(x) == 0, residual falls back to p when its sum
  is 0.
"""
from __future__ import annotations

import numpy as np

GROUP = 128  # input channels per weight-scale group

# ----------------------------------------------------------------------------------------------
# bfloat16 / fp16 helpers (written here, independent of any other module)
# ----------------------------------------------------------------------------------------------


def bf16_to_f32(bits) -> np.ndarray:
    """bfloat16 bit patterns -> fp32 values (exact: a bf16 is the top half of an fp32)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f64_to_bf16_value(x) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 value (ties to even), returned as fp64.

    Done directly in fp64 (no intermediate fp32 rounding): the bf16 spacing at |x| is
    2**(e - 7) with e = floor(log2 |x|), or 2**-133 below the normal range; x / spacing is rounded
    to an integer with ties to even.  Overflow beyond the largest bf16 gives +-inf.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    fin = np.isfinite(x) & (x != 0)
    xf = x[fin]
    _, e2 = np.frexp(np.abs(xf))  # |x| = m * 2**e2, m in [0.5, 1)  ->  floor(log2|x|) = e2 - 1
    e = np.maximum(e2 - 1, -126)
    spacing = np.ldexp(1.0, e - 7)
    r = np.rint(xf / spacing) * spacing
    bf16_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(np.abs(r) > bf16_max, np.copysign(np.inf, r), r)
    out[fin] = r
    return out


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round fp64 -> bfloat16 (ties to even) and return the uint16 bit patterns."""
    v = f64_to_bf16_value(x).astype(np.float32)  # exact: the value is already a bf16
    return (v.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ----------------------------------------------------------------------------------------------
# a1: weight quantiser and packer        [QSpec-article] "W4A4 と W4A16 量子化", shared weights
# ----------------------------------------------------------------------------------------------


def quantize_weights(W_bits):
    """Symmetric per-group INT4 weight quantisation.

    W_bits: uint16 bf16 bits [N, K], K % 128 == 0.
    Returns (codes int8 [N, K] in [-8, 7], S float16 [N, K/128]).
    Per group of 128 consecutive k of one row n:
        amax = max |w|;  s = fp16(amax / 7)  (fp32 IEEE division, then round to fp16);
        code = clamp(rint(w / fp32(s)), -8, 7)  (fp32 IEEE division, ties to even); s == 0 -> 0.
    """
    W = bf16_to_f32(W_bits)
    N, K = W.shape
    assert K % GROUP == 0, "K must be a multiple of 128"
    G = K // GROUP
    Wg = W.reshape(N, G, GROUP)
    amax = np.max(np.abs(Wg), axis=2)                      # fp32, exact
    s32 = amax / np.float32(7.0)                           # fp32 IEEE division
    S = s32.astype(np.float16)                             # round to nearest even fp16
    s = S.astype(np.float32)[:, :, None]                   # exact widening
    codes = np.zeros((N, G, GROUP), dtype=np.int8)
    nz = np.broadcast_to(s != 0, Wg.shape)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = Wg / s                                         # fp32 IEEE division
    q = np.clip(np.rint(q), -8, 7)
    codes[nz] = q[nz].astype(np.int8)
    return codes.reshape(N, K), S


# Nibble slot i (bits 4i..4i+3 of a little-endian 32-bit word) holds channel 8t + WORD_ORDER[i].
WORD_ORDER = (0, 2, 4, 6, 1, 3, 5, 7)


def pack_codes(codes) -> np.ndarray:
    """int8 codes [N, K] -> uint8 [N, K/2]; word t holds k = 8t + WORD_ORDER[i] in nibble i."""
    c = np.asarray(codes, dtype=np.int8).astype(np.int16) & 0xF
    N, K = c.shape
    blocks = c.reshape(N, K // 8, 8)
    nib = blocks[:, :, list(WORD_ORDER)]                 # nibbles 0..7 of each word
    byte = nib[:, :, 0::2] | (nib[:, :, 1::2] << 4)      # byte b = nibble 2b | nibble 2b+1 << 4
    return byte.reshape(N, K // 2).astype(np.uint8)


def unpack_codes(Wp) -> np.ndarray:
    """uint8 [N, K/2] -> int8 codes [N, K] (inverse of pack_codes)."""
    b = np.asarray(Wp, dtype=np.uint8).astype(np.int16)
    N, H = b.shape
    byte = b.reshape(N, H // 4, 4)
    nib = np.empty((N, H // 4, 8), dtype=np.int16)
    nib[:, :, 0::2] = byte & 0xF
    nib[:, :, 1::2] = (byte >> 4) & 0xF
    out = np.empty_like(nib)
    out[:, :, list(WORD_ORDER)] = nib
    out = np.where(out >= 8, out - 16, out)
    return out.reshape(N, 2 * H).astype(np.int8)


def pack_weights(W_bits):
    """a1 end to end: bf16 W [N, K] -> (Wp uint8 [N, K/2], S float16 [N, K/128])."""
    codes, S = quantize_weights(W_bits)
    return pack_codes(codes), S


def dequantize_weights(Wp, S, rows=None) -> np.ndarray:
    """Dequantised weights code * s in fp64 [N, K] (optionally only the given rows)."""
    Wp = np.asarray(Wp)
    S = np.asarray(S, dtype=np.float16)
    if rows is not None:
        Wp = Wp[rows]
        S = S[rows]
    codes = unpack_codes(Wp).astype(np.float64)
    scale = np.repeat(S.astype(np.float64), GROUP, axis=1)
    return codes * scale


# ----------------------------------------------------------------------------------------------
# a2: W4A16 linear (verify mode)          [QSpec-article] "W4A16: 重みのみを 4-bit に量子化"
# ----------------------------------------------------------------------------------------------


def linear_w4a16(x_bits, Wp, S, rows=None) -> np.ndarray:
    """y[m, n] = sum_k x[m, k] * code[n, k] * s[n, k // 128], in fp64.

    x_bits: bf16 bits [M, K]; returns fp64 [M, N] (or [M, len(rows)] for a subset of outputs).
    """
    x = bf16_to_f32(x_bits).astype(np.float64)
    Wd = dequantize_weights(Wp, S, rows)
    return x @ Wd.T


# ----------------------------------------------------------------------------------------------
# a3: per-token activation quantiser      [QSpec-article] "W4A4 : 重みと活性値の両方を 4-bit に量子化"
# ----------------------------------------------------------------------------------------------


def quantize_activations(x_bits, bits=4):
    """Per-token symmetric activation quantisation to `bits`-bit codes (4: W4A4, 8: W4A8).

    Returns (qa int8 [M, K], s_a float32 [M]), with qmax = 2**(bits-1) - 1 (7 or 127):
        amax = max_k |x[m, k]|;  s_a = amax / qmax (fp32 IEEE division, kept in fp32);
        qa = clamp(rint(x / s_a), -qmax - 1, qmax) (fp32 IEEE division, ties to even); s_a == 0 -> 0.
    """
    qmax = 2 ** (bits - 1) - 1
    x = bf16_to_f32(x_bits)
    amax = np.max(np.abs(x), axis=1)
    s_a = (amax / np.float32(qmax)).astype(np.float32)
    qa = np.zeros(x.shape, dtype=np.int8)
    for m in range(x.shape[0]):
        if s_a[m] != 0:
            qa[m] = np.clip(np.rint(x[m] / s_a[m]), -qmax - 1, qmax).astype(np.int8)
    return qa, s_a


# ----------------------------------------------------------------------------------------------
# a4: W4A4 linear (draft mode)            [QSpec-article] "W4A4 : 重みと活性値の両方を 4-bit に量子化"
# ----------------------------------------------------------------------------------------------


def w4a4_group_sums(qa, Wp, rows=None) -> np.ndarray:
    """acc[m, n, g] = sum_{k in group g} qa[m, k] * code[n, k]  (exact integers, int32)."""
    qa = np.asarray(qa, dtype=np.int64)
    Wp = np.asarray(Wp)
    if rows is not None:
        Wp = Wp[rows]
    codes = unpack_codes(Wp).astype(np.int64)
    M, K = qa.shape
    N = codes.shape[0]
    G = K // GROUP
    acc = np.einsum("mgk,ngk->mng", qa.reshape(M, G, GROUP), codes.reshape(N, G, GROUP))
    return acc.astype(np.int32)


def linear_w4a4(x_bits, Wp, S, rows=None, bits=4):
    """Draft-mode linear (bits=8: the W4A8 configuration on the same weights).

    Returns dict(qa, s_a, acc int32 [M, N, G], y fp64 [M, N]) with
        y[m, n] = s_a[m] * sum_g s[n, g] * acc[m, n, g]   (fp64).
    """
    qa, s_a = quantize_activations(x_bits, bits)
    acc = w4a4_group_sums(qa, Wp, rows)
    S = np.asarray(S, dtype=np.float16)
    if rows is not None:
        S = S[rows]
    Sg = S.astype(np.float64)                                        # [N, G]
    y = s_a.astype(np.float64)[:, None] * np.einsum("mng,ng->mn", acc.astype(np.float64), Sg)
    return {"qa": qa, "s_a": s_a, "acc": acc, "y": y}


# ----------------------------------------------------------------------------------------------
# f3: W4A8       [SD+Q summary] "中核となる技術的要素" names W4A8 beside W4A16; the quantiser is the
#                W4A4 one at 8 bits (the summary gives none)
# ----------------------------------------------------------------------------------------------


def linear_w4a8(x_bits, Wp, S, rows=None):
    """W4A8 linear: per-token 8-bit activation codes (s_a = amax / 127), 4-bit shared weights."""
    return linear_w4a4(x_bits, Wp, S, rows, bits=8)


# ----------------------------------------------------------------------------------------------
# a5: softmax over the vocabulary          [SD-tutorial] p and q are the model distributions
# ----------------------------------------------------------------------------------------------


def softmax(logits) -> np.ndarray:
    """p_j = exp(l_j - max l) / sum_i exp(l_i - max l) along the last axis, fp64; -inf -> 0."""
    l = np.asarray(logits, dtype=np.float64)
    m = np.max(l, axis=-1, keepdims=True)
    e = np.exp(l - m)
    return e / np.sum(e, axis=-1, keepdims=True)


# ----------------------------------------------------------------------------------------------
# a6: greedy verify        [SD-tutorial] "greedy decodingでは一致するprefixを採用する"
# ----------------------------------------------------------------------------------------------


def first_argmax(values) -> int:
    """The lowest index j with values[j] == max(values)  (+0 and -0 compare equal)."""
    v = np.asarray(values)
    hits = np.flatnonzero(v == np.max(v))
    if hits.size == 0:
        raise ValueError("no maximum (NaN input)")
    return int(hits[0])


def verify_greedy(tgt_bits, draft_tok):
    """Greedy verification of gamma draft tokens per sequence.

    tgt_bits: bf16 bits [B, gamma+1, V] (target logits at the gamma draft positions and the next
    one); draft_tok int [B, gamma].
    Per sequence: t_i = argmax of target row i; accept draft tokens left to right while d_i == t_i;
    at the first mismatch n emit t_n and drop the rest; when all gamma match, n = gamma and the
    target's token t_gamma for the next position is emitted as well.
    Returns (accept_len int32 [B], out_tok int32 [B, gamma+1] with unused slots -1,
    tgt_argmax int32 [B, gamma+1]).
    """
    L = bf16_to_f32(tgt_bits)
    B, G1, V = L.shape
    gamma = G1 - 1
    d = np.asarray(draft_tok)
    t = np.zeros((B, G1), dtype=np.int32)
    n = np.zeros(B, dtype=np.int32)
    out = np.full((B, G1), -1, dtype=np.int32)
    for b in range(B):
        for i in range(G1):
            t[b, i] = first_argmax(L[b, i])
        k = 0
        while k < gamma and int(d[b, k]) == int(t[b, k]):
            k += 1
        n[b] = k
        out[b, :k] = d[b, :k]
        out[b, k] = t[b, k]
    return n, out, t


# ----------------------------------------------------------------------------------------------
# f4: tree verification (greedy)   [SD+Q summary] "先行研究との差別化ポイント", "中核となる技術的要素"
#     name tree-style verification without an algorithm; this is the greedy rule on a tree
# ----------------------------------------------------------------------------------------------


def verify_tree_greedy(tgt_bits, tree_tok, tree_parent):
    """Greedy verification of a candidate tree per sequence.

    tgt_bits: bf16 bits [B, T+1, V] (row 0: the token after the committed prefix; row j+1: the token
    after node j); tree_tok, tree_parent int [B, T] (parent -1 is the prefix, otherwise an earlier
    node).  From the prefix, repeatedly accept the lowest-index child whose token equals the target's
    most likely token at the current row; stop when no child matches and emit the target's token.
    Nodes with a token outside [0, V) or a parent outside [-1, j-1] never match.
    Returns (accept_len int32 [B], out_tok int32 [B, T+1] (-1 fill), accept_nodes int32 [B, T] (-1 fill)).
    """
    L = bf16_to_f32(tgt_bits)
    B, R, V = L.shape
    T = R - 1
    tok = np.asarray(tree_tok)
    par = np.asarray(tree_parent)
    n = np.zeros(B, dtype=np.int32)
    out = np.full((B, R), -1, dtype=np.int32)
    nodes = np.full((B, T), -1, dtype=np.int32)
    for b in range(B):
        t = [first_argmax(L[b, r]) for r in range(R)]
        valid = [0 <= int(tok[b, j]) < V and -1 <= int(par[b, j]) < j for j in range(T)]
        cur, row, path = -1, 0, []
        while True:
            children = [j for j in range(T) if valid[j] and int(par[b, j]) == cur and int(tok[b, j]) == t[row]]
            if not children:
                break
            cur = min(children)
            path.append(cur)
            row = cur + 1
        n[b] = len(path)
        out[b, :len(path)] = [int(tok[b, j]) for j in path]
        out[b, len(path)] = t[row]
        nodes[b, :len(path)] = path
    return n, out, nodes


# ----------------------------------------------------------------------------------------------
# a7, a8: sampling verify  [SD-tutorial] "samplingでもtargetの確率分布を保つ", eq. a(x), eq. p'(x)
# ----------------------------------------------------------------------------------------------


def inverse_cdf(r, u) -> int:
    """Smallest j with sum_{i<=j} r_i > u * sum(r)   (index order, strict '>').

    If rounding leaves no such j (u * R at the very top), the last j with r_j > 0 is taken.
    """
    r = np.asarray(r, dtype=np.float64)
    R = np.sum(r)
    c = np.cumsum(r)
    hit = np.nonzero(c > u * R)[0]
    if hit.size:
        return int(hit[0])
    return int(np.nonzero(r > 0)[0][-1])


def verify_sample_probs(p_rows, q_rows, draft_tok, u_acc, u_res):
    """Sampling verification of one sequence, in probability space.

    p_rows [gamma+1, V]: target distributions; q_rows [gamma, V]: draft distributions;
    draft_tok [gamma]; u_acc [gamma], u_res [gamma+1]: uniforms in [0, 1).
    Position i accepts x = d_i iff u_acc[i] < a_i with a_i = min(1, p_i(x) / q_i(x)) (a_i = 1 when
    q_i(x) == 0).  At the first rejection n the replacement token is drawn from the residual
    max(0, p_n - q_n) / sum(...) (p_n itself when that sum is 0) with u_res[n]; when all gamma are
    accepted, n = gamma and the bonus token is drawn from p_gamma with u_res[gamma].
    Returns dict(n, out [gamma+1] (-1 padded), a [gamma], p_tok [gamma], q_tok [gamma], j, R,
    residual) where a / p_tok / q_tok are evaluated at every draft position.
    """
    p_rows = np.asarray(p_rows, dtype=np.float64)
    q_rows = np.asarray(q_rows, dtype=np.float64)
    gamma = q_rows.shape[0]
    d = np.asarray(draft_tok)
    a = np.zeros(gamma)
    p_tok = np.zeros(gamma)
    q_tok = np.zeros(gamma)
    for i in range(gamma):
        x = int(d[i])
        p_tok[i] = p_rows[i, x]
        q_tok[i] = q_rows[i, x]
        a[i] = 1.0 if q_tok[i] == 0 else min(1.0, p_tok[i] / q_tok[i])
    n = gamma
    for i in range(gamma):
        if not (float(u_acc[i]) < a[i]):
            n = i
            break
    if n < gamma:
        r = np.maximum(0.0, p_rows[n] - q_rows[n])
        if np.sum(r) == 0:
            r = p_rows[n]
    else:
        r = p_rows[gamma]
    j = inverse_cdf(r, float(u_res[n]))
    out = np.full(gamma + 1, -1, dtype=np.int64)
    out[:n] = d[:n]
    out[n] = j
    return {"n": n, "out": out, "a": a, "p_tok": p_tok, "q_tok": q_tok, "j": j,
            "R": float(np.sum(r)), "residual": r}


def verify_sample(tgt_bits, drf_bits, draft_tok, u_acc, u_res):
    """Sampling verification from bf16 logits (temperature 1).

    tgt_bits [B, gamma+1, V], drf_bits [B, gamma, V] bf16 bits; draft_tok [B, gamma];
    u_acc [B, gamma], u_res [B, gamma+1].  p and q are fp64 softmaxes of the bf16 logits.
    Returns dict of arrays: accept_len [B], out_tok [B, gamma+1], accept_prob / p_tok / q_tok
    [B, gamma], plus per-sequence diagnostics used to apply decision tolerances:
    ``acc_margin`` [B, gamma] = |u_acc - a| and ``res_margin`` [B] = distance of u_res * R from the
    nearest CDF step that bounds the chosen index, divided by R.
    """
    T = bf16_to_f32(tgt_bits).astype(np.float64)
    D = bf16_to_f32(drf_bits).astype(np.float64)
    B, G1, V = T.shape
    gamma = G1 - 1
    res = {
        "accept_len": np.zeros(B, dtype=np.int32),
        "out_tok": np.full((B, G1), -1, dtype=np.int32),
        "accept_prob": np.zeros((B, gamma)),
        "p_tok": np.zeros((B, gamma)),
        "q_tok": np.zeros((B, gamma)),
        "acc_margin": np.zeros((B, gamma)),
        "res_margin": np.zeros(B),
    }
    for b in range(B):
        P = softmax(T[b])
        Q = softmax(D[b])
        r = verify_sample_probs(P, Q, draft_tok[b], u_acc[b], u_res[b])
        res["accept_len"][b] = r["n"]
        res["out_tok"][b] = r["out"]
        res["accept_prob"][b] = r["a"]
        res["p_tok"][b] = r["p_tok"]
        res["q_tok"][b] = r["q_tok"]
        res["acc_margin"][b] = np.abs(np.asarray(u_acc[b], dtype=np.float64) - r["a"])
        c = np.cumsum(r["residual"])
        target = float(u_res[b][r["n"]]) * r["R"]
        j = r["j"]
        lo = c[j - 1] if j > 0 else 0.0
        res["res_margin"][b] = min(abs(c[j] - target), abs(target - lo)) / r["R"] if r["R"] > 0 else 0.0
    return res


# ----------------------------------------------------------------------------------------------
# f1: the decode loop     [SD-tutorial] "draft modelとtarget modelの処理フロー"
# ----------------------------------------------------------------------------------------------


def select_token(logits_bits, u=None) -> int:
    """A model's next token from its bf16 logits row: the most likely token when decoding greedily
    (u is None), else the inverse-CDF draw from softmax(logits) with uniform u."""
    l = bf16_to_f32(logits_bits).astype(np.float64)
    if u is None:
        return first_argmax(l)
    return inverse_cdf(softmax(l), float(u))


def toy_forward(E_bits, layers, tok, draft_mode):
    """Logits of a stack of linears on the shared packed weights, for one input token per row.

    x = E[tok] (bf16 embedding rows); then for each (Wp, S) in order, x = bf16(linear(x)) with the
    draft-mode (W4A4) or verify-mode (W4A16) linear; the last layer's output are the bf16 logits.
    Returns bf16 bits [len(tok), N_last].
    """
    x = np.asarray(E_bits)[np.asarray(tok, dtype=np.int64)]
    for Wp, S in layers:
        y = linear_w4a4(x, Wp, S)["y"] if draft_mode else linear_w4a16(x, Wp, S)
        x = f64_to_bf16_bits(y)
    return x


def speculative_decode(target, draft, prefix, n_iter, gamma, u_draft=None, u_acc=None, u_res=None):
    """The classic draft-then-verify loop for one sequence, n_iter iterations.

    target(seq) / draft(seq) return the bf16 logits row of the token that follows seq.  Each
    iteration: the draft model extends its own copy of the sequence one token at a time, gamma times
    (select_token with u_draft[it][i], greedy when u_draft is None); the target scores the gamma
    draft positions and the one after them; verify_greedy (u_acc is None) or verify_sample decides
    how many drafts stand and which token follows them; those n + 1 tokens are appended.
    Returns (generated tokens, accept lengths n per iteration).
    """
    seq = [int(t) for t in prefix]
    start = len(seq)
    ns = []
    for it in range(n_iter):
        d, dl = [], []
        for i in range(gamma):
            l = draft(seq + d)
            dl.append(l)
            d.append(select_token(l, None if u_draft is None else u_draft[it][i]))
        tl = np.stack([target(seq + d[:i]) for i in range(gamma + 1)])[None]
        dt = np.array([d], dtype=np.int32)
        if u_acc is None:
            n, out, _ = verify_greedy(tl, dt)
            n, out = int(n[0]), out[0]
        else:
            r = verify_sample(tl, np.stack(dl)[None], dt, np.asarray(u_acc[it])[None], np.asarray(u_res[it])[None])
            n, out = int(r["accept_len"][0]), r["out_tok"][0]
        seq += [int(t) for t in out[:n + 1]]
        ns.append(n)
    return seq[start:], ns


def target_only_decode(target, prefix, n_new, u=None):
    """Plain decoding with the target alone: one target call per token (greedy when u is None)."""
    seq = [int(t) for t in prefix]
    for k in range(n_new):
        seq.append(select_token(target(seq), None if u is None else u[k]))
    return seq[len(prefix):]


# ----------------------------------------------------------------------------------------------
# f2: top-1 statistics   [QSpec-article] sections "実験：W4A4 と W4A16 の Top-1 一致率を調べる", "結果"
# ----------------------------------------------------------------------------------------------

TOP1_TALLY = ("positions", "agree", "both_high", "agree_both_high", "both_low", "agree_both_low",
              "sum_p1_target", "sum_p1_draft")


def top1_stats(tgt_bits, drf_bits, high=0.8):
    """Per draft position: each mode's most likely token and the probability that mode gives it.

    tgt_bits: bf16 bits [B, gamma+1, V] (verify mode, only rows 0..gamma-1 are draft positions);
    drf_bits: bf16 bits [B, gamma, V] (draft mode).  The article records, at every draft position,
    the top-1 token of W4A4 and of W4A16 and each one's own top-1 probability (they may be different
    tokens); it reports the agreement rate, the mean top-1 probability per mode, and the agreement
    inside "both above the threshold" (p > high in both modes) and "both at or below it".
    Returns (tgt_top1 int32 [B, gamma], draft_top1 int32 [B, gamma], tgt_p1 fp64, draft_p1 fp64,
    tally fp64 [8] in the order of TOP1_TALLY).
    """
    Lt = bf16_to_f32(tgt_bits)
    Ld = bf16_to_f32(drf_bits)
    B, gamma, V = Ld.shape
    t_tok = np.zeros((B, gamma), dtype=np.int32)
    d_tok = np.zeros((B, gamma), dtype=np.int32)
    t_p = np.zeros((B, gamma))
    d_p = np.zeros((B, gamma))
    tally = np.zeros(len(TOP1_TALLY))
    for b in range(B):
        for i in range(gamma):
            t_tok[b, i] = first_argmax(Lt[b, i])
            d_tok[b, i] = first_argmax(Ld[b, i])
            t_p[b, i] = softmax(Lt[b, i])[t_tok[b, i]]
            d_p[b, i] = softmax(Ld[b, i])[d_tok[b, i]]
            agree = t_tok[b, i] == d_tok[b, i]
            tally[0] += 1
            tally[1] += agree
            if t_p[b, i] > high and d_p[b, i] > high:
                tally[2] += 1
                tally[3] += agree
            if t_p[b, i] <= high and d_p[b, i] <= high:
                tally[4] += 1
                tally[5] += agree
            tally[6] += t_p[b, i]
            tally[7] += d_p[b, i]
    return t_tok, d_tok, t_p, d_p, tally


# ----------------------------------------------------------------------------------------------
# Expected tokens per target call    [SD-tutorial] "1回のtarget検証で何token進むか"
# ----------------------------------------------------------------------------------------------


def expected_tokens(alpha: float, gamma: int) -> float:
    """E[T] = 1 + alpha + ... + alpha**gamma = (1 - alpha**(gamma+1)) / (1 - alpha); gamma+1 at 1."""
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)
