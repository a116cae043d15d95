"""Thin ctypes binding of libqspec.so: same names as the C ABI in include/qspec.h.

Every function only marshals arguments (torch tensors -> device pointers and sizes, the current
CUDA stream) and raises ``QSpecError`` on a non-OK status.  All computation happens in the CUDA
library; there is no fallback of any kind -- if the library is missing, loading fails loudly.
The sizes passed to the library come from the leading input's shape; every other tensor must hold
at least the elements the call reads or writes (ValueError otherwise, before any launch), since
the C ABI sees plain pointers and cannot check them itself.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqspec.so")

STATUS = {
    0: "QSPEC_OK",
    1: "QSPEC_ERR_INVALID_ARG",
    2: "QSPEC_ERR_UNSUPPORTED_SHAPE",
    3: "QSPEC_ERR_MISALIGNED",
    4: "QSPEC_ERR_WORKSPACE",
    5: "QSPEC_ERR_CUDA",
    6: "QSPEC_ERR_TIMEOUT",
}

# exported symbol -> (restype, argtypes)
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
SIGNATURES = {
    "qspec_pack_weights": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P]),
    "qspec_linear_workspace_size": (ctypes.c_size_t, [_I64, _I64, _I64]),
    "qspec_linear_w4a16": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _I64, _P, _P, ctypes.c_size_t, _P]),
    "qspec_linear_w4a4": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _I64, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "qspec_linear_w4a8": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _I64, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "qspec_verify_workspace_size": (ctypes.c_size_t, [_I32, _I32, _I32]),
    "qspec_verify_greedy": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "qspec_verify_sample": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P,
                                           ctypes.c_size_t, _P]),
    "qspec_verify_top1": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _P, _P, _P, _P, ctypes.c_float, _P, _P,
                                         ctypes.c_size_t, _P]),
    "qspec_verify_greedy_noalloc": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _P, _P, _P, _P]),
    "qspec_verify_tree_workspace_size": (ctypes.c_size_t, [_I32, _I32, _I32]),
    "qspec_verify_tree_greedy": (ctypes.c_int, [_P, _P, _P, _I32, _I32, _I32, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "qspec_gather_rows": (ctypes.c_int, [_P, _I64, _I64, _P, _I64, _P, _P]),
    "qspec_select_tokens": (ctypes.c_int, [_P, _I32, _I32, _P, _P, _P]),
    "qspec_linear_group_workspace_size": (ctypes.c_size_t, [_I64, _P, _I32, _I64]),
    "qspec_linear_group": (ctypes.c_int, [_I32, _P, _I64, _I64, _P, _I32, _P, ctypes.c_size_t, _P]),
    "qspec_linear_pass_workspace_size": (ctypes.c_size_t, []),
    "qspec_linear_pass": (ctypes.c_int, [_I32, _I64, _P, _I32, _P, ctypes.c_size_t, _P]),
    "qspec_check_status": (ctypes.c_int, [_P, _P]),
    "qspec_copy": (ctypes.c_int, [_P, _P, ctypes.c_size_t, _P]),
    "qspec_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}


class QSpecError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libqspec.so (built by build.py / __graft_entry__.build()) and declare its signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libqspec.so not found at {p}: build it first (python -m "
                           "quantized_speculative_decoding_qspec_gb300.build)")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("tensor must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(fn: str, code: int):
    if code != 0:
        raise QSpecError(fn, code)


def _dt(t, dtype, name):
    if t is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _need(t, n, name):
    """The library writes or reads n elements of t: refuse a smaller tensor before any launch."""
    if t is not None and t.numel() < n:
        raise ValueError(f"{name} holds {t.numel()} elements, the call needs {n}")


def qspec_pack_weights(W, Wp, S, stream=None):
    """W bf16 [N, K] -> Wp uint8 [N, K/2], S fp16 [N, K/128] (outputs written in place)."""
    _dt(W, torch.bfloat16, "W"); _dt(Wp, torch.uint8, "Wp"); _dt(S, torch.float16, "S")
    N, K = W.shape
    _need(Wp, N * (K // 2), "Wp"); _need(S, N * (K // 128), "S")
    _check("qspec_pack_weights", load().qspec_pack_weights(_ptr(W), N, K, _ptr(Wp), _ptr(S), _stream(stream)))


def qspec_linear_workspace_size(M, N, K):
    """Workspace bytes for an [M, K] x [N, K] product on the current device."""
    return int(load().qspec_linear_workspace_size(M, N, K))


def new_linear_workspace(M, N, K, device="cuda"):
    """A zero-filled linear workspace (zero once; calls of this (M, N, K) keep it ready, other shapes
    need their own)."""
    n = qspec_linear_workspace_size(M, N, K)
    if n == 0:
        raise ValueError("invalid linear shape")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _need_linear(M, N, K, Wp, S, y, xq_out=None, xs_out=None, acc_out=None):
    _need(Wp, N * (K // 2), "Wp"); _need(S, N * (K // 128), "S"); _need(y, M * N, "y")
    _need(xq_out, M * K, "xq_out"); _need(xs_out, M, "xs_out"); _need(acc_out, M * N * (K // 128), "acc_out")


def qspec_linear_w4a16(x, Wp, S, y, ws, stream=None):
    """y bf16 [M, N] = x bf16 [M, K] . dequant(Wp, S)^T."""
    _dt(x, torch.bfloat16, "x"); _dt(Wp, torch.uint8, "Wp"); _dt(S, torch.float16, "S"); _dt(y, torch.bfloat16, "y")
    _dt(ws, torch.uint8, "ws")
    M, K = x.shape
    N = Wp.shape[0]
    _need_linear(M, N, K, Wp, S, y)
    _check("qspec_linear_w4a16",
           load().qspec_linear_w4a16(_ptr(x), _ptr(Wp), _ptr(S), M, N, K, _ptr(y), _ptr(ws), ws.numel(),
                                     _stream(stream)))


def qspec_linear_w4a4(x, Wp, S, y, ws, xq_out=None, xs_out=None, acc_out=None, stream=None):
    """Draft-mode linear with the per-token INT4 activation quantiser fused."""
    _dt(x, torch.bfloat16, "x"); _dt(Wp, torch.uint8, "Wp"); _dt(S, torch.float16, "S"); _dt(y, torch.bfloat16, "y")
    _dt(xq_out, torch.int8, "xq_out"); _dt(xs_out, torch.float32, "xs_out"); _dt(acc_out, torch.int32, "acc_out")
    _dt(ws, torch.uint8, "ws")
    M, K = x.shape
    N = Wp.shape[0]
    _need_linear(M, N, K, Wp, S, y, xq_out, xs_out, acc_out)
    _check("qspec_linear_w4a4",
           load().qspec_linear_w4a4(_ptr(x), _ptr(Wp), _ptr(S), M, N, K, _ptr(y), _ptr(xq_out), _ptr(xs_out),
                                    _ptr(acc_out), _ptr(ws), ws.numel(), _stream(stream)))


def qspec_linear_w4a8(x, Wp, S, y, ws, xq_out=None, xs_out=None, acc_out=None, stream=None):
    """The W4A8 configuration: qspec_linear_w4a4 with per-token INT8 activation codes."""
    _dt(x, torch.bfloat16, "x"); _dt(Wp, torch.uint8, "Wp"); _dt(S, torch.float16, "S"); _dt(y, torch.bfloat16, "y")
    _dt(xq_out, torch.int8, "xq_out"); _dt(xs_out, torch.float32, "xs_out"); _dt(acc_out, torch.int32, "acc_out")
    _dt(ws, torch.uint8, "ws")
    M, K = x.shape
    N = Wp.shape[0]
    _need_linear(M, N, K, Wp, S, y, xq_out, xs_out, acc_out)
    _check("qspec_linear_w4a8",
           load().qspec_linear_w4a8(_ptr(x), _ptr(Wp), _ptr(S), M, N, K, _ptr(y), _ptr(xq_out), _ptr(xs_out),
                                    _ptr(acc_out), _ptr(ws), ws.numel(), _stream(stream)))


class LinearPart(ctypes.Structure):
    """One part of qspec_linear_group (the C struct qspec_linear_part)."""
    _fields_ = [("Wp", ctypes.c_void_p), ("S", ctypes.c_void_p), ("y", ctypes.c_void_p), ("N", ctypes.c_int64)]


class LinearGroup:
    """Several linears that read the same activations, in one launch (qspec_linear_group).

    x: bf16 [M, K]; parts: list of (Wp, S, y) -- Wp uint8 [N, K/2], S fp16 [N, K/128], y bf16 [M, N].
    abits: 16 (W4A16), 4 (W4A4) or 8 (W4A8).  The tensors must stay alive while the group is used.
    """

    def __init__(self, abits, x, parts, ws):
        _dt(x, torch.bfloat16, "x"); _dt(ws, torch.uint8, "ws")
        if not parts:
            raise ValueError("a group needs at least one part")
        self.M, self.K = x.shape
        self.abits, self.x, self.ws = int(abits), x, ws
        self.arr = (LinearPart * len(parts))()
        self._keep = [x]
        for i, (Wp, S, y) in enumerate(parts):
            _dt(Wp, torch.uint8, "Wp"); _dt(S, torch.float16, "S"); _dt(y, torch.bfloat16, "y")
            N = Wp.shape[0]
            _need_linear(self.M, N, self.K, Wp, S, y)
            self.arr[i] = LinearPart(_ptr(Wp), _ptr(S), _ptr(y), N)
            self._keep += [Wp, S, y]

    def run(self, stream=None):
        _check("qspec_linear_group", load().qspec_linear_group(self.abits, _ptr(self.x), self.M, self.K, self.arr,
                                                               len(self.arr), _ptr(self.ws), self.ws.numel(),
                                                               _stream(stream)))


def qspec_linear_group_workspace_size(M, Ns, K):
    """Bytes of the workspace for a group of parts with N in Ns (0 if the arguments are invalid)."""
    arr = (LinearPart * len(Ns))()
    for i, N in enumerate(Ns):
        arr[i] = LinearPart(16, 16, 16, int(N))  # (only N is read; non-null, aligned placeholders)
    return int(load().qspec_linear_group_workspace_size(M, arr, len(Ns), K))


def new_linear_group_workspace(M, Ns, K, device="cuda"):
    """A zero-filled workspace for qspec_linear_group over parts with N in Ns."""
    n = qspec_linear_group_workspace_size(M, Ns, K)
    if n == 0:
        raise ValueError("invalid group shape")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def qspec_linear_group(abits, x, parts, ws, stream=None):
    """One launch over (Wp, S, y) parts that read the same x (see LinearGroup)."""
    LinearGroup(abits, x, parts, ws).run(stream)


class PassLayer(ctypes.Structure):
    """One layer of qspec_linear_pass (the C struct qspec_pass_layer)."""
    _fields_ = [("x", ctypes.c_void_p), ("Wp", ctypes.c_void_p), ("S", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("after", ctypes.c_int32), ("reserved", ctypes.c_int32)]


def qspec_linear_pass_workspace_size():
    return int(load().qspec_linear_pass_workspace_size())


def new_pass_workspace(device="cuda"):
    """A zero-filled linear-pass workspace (zero once; passes keep it ready)."""
    return torch.zeros(qspec_linear_pass_workspace_size(), dtype=torch.uint8, device=device)


class LinearPass:
    """A pass of decode-size linears in one mode, described once and launched with run().

    layers: list of (x, Wp, S, y, after) -- x bf16 [M, K] (the same M for all), Wp uint8 [N, K/2],
    S fp16 [N, K/128], y bf16 [M, N], after: the layer reads outputs of earlier layers of the pass.
    abits: 16 (W4A16), 4 (W4A4) or 8 (W4A8).  The tensors must stay alive while the pass is used.
    """

    def __init__(self, abits, layers, ws):
        _dt(ws, torch.uint8, "ws")
        if not layers:
            raise ValueError("a pass needs at least one layer")
        self.M = layers[0][0].shape[0]
        self.abits = int(abits)
        self.ws = ws
        self.arr = (PassLayer * len(layers))()
        self._keep = []
        for i, (x, Wp, S, y, after) in enumerate(layers):
            _dt(x, torch.bfloat16, "x"); _dt(Wp, torch.uint8, "Wp"); _dt(S, torch.float16, "S")
            _dt(y, torch.bfloat16, "y")
            M, K = x.shape
            if M != self.M:
                raise ValueError("every layer of a pass has the same number of tokens")
            N = Wp.shape[0]
            _need_linear(M, N, K, Wp, S, y)
            self.arr[i] = PassLayer(_ptr(x), _ptr(Wp), _ptr(S), _ptr(y), N, K, 1 if after else 0, 0)
            self._keep += [x, Wp, S, y]

    def run(self, stream=None):
        _check("qspec_linear_pass", load().qspec_linear_pass(self.abits, self.M, self.arr, len(self.arr),
                                                             _ptr(self.ws), self.ws.numel(), _stream(stream)))


def qspec_linear_pass(abits, layers, ws, stream=None):
    """One launch over a list of (x, Wp, S, y, after) linears in one mode (see LinearPass)."""
    LinearPass(abits, layers, ws).run(stream)


def qspec_verify_workspace_size(B, gamma, V):
    return int(load().qspec_verify_workspace_size(B, gamma, V))


def _need_greedy(B, G1, draft_tok, accept_len, out_tok, tgt_argmax):
    _need(draft_tok, B * (G1 - 1), "draft_tok"); _need(accept_len, B, "accept_len")
    _need(out_tok, B * G1, "out_tok"); _need(tgt_argmax, B * G1, "tgt_argmax")


def qspec_verify_greedy(tgt_logits, draft_tok, accept_len, out_tok, ws, tgt_argmax=None, stream=None):
    """Greedy verify: tgt_logits bf16 [B, gamma+1, V], draft_tok int32 [B, gamma]."""
    _dt(tgt_logits, torch.bfloat16, "tgt_logits"); _dt(draft_tok, torch.int32, "draft_tok")
    _dt(accept_len, torch.int32, "accept_len"); _dt(out_tok, torch.int32, "out_tok")
    _dt(tgt_argmax, torch.int32, "tgt_argmax"); _dt(ws, torch.uint8, "ws")
    B, G1, V = tgt_logits.shape
    _need_greedy(B, G1, draft_tok, accept_len, out_tok, tgt_argmax)
    _check("qspec_verify_greedy",
           load().qspec_verify_greedy(_ptr(tgt_logits), _ptr(draft_tok), B, G1 - 1, V, _ptr(accept_len),
                                      _ptr(out_tok), _ptr(tgt_argmax), _ptr(ws), ws.numel(), _stream(stream)))


def qspec_verify_greedy_noalloc(tgt_logits, draft_tok, accept_len, out_tok, tgt_argmax=None, stream=None):
    """Greedy verify without a workspace (scratch inside the library; for callers that cannot allocate)."""
    _dt(tgt_logits, torch.bfloat16, "tgt_logits"); _dt(draft_tok, torch.int32, "draft_tok")
    _dt(accept_len, torch.int32, "accept_len"); _dt(out_tok, torch.int32, "out_tok")
    _dt(tgt_argmax, torch.int32, "tgt_argmax")
    B, G1, V = tgt_logits.shape
    _need_greedy(B, G1, draft_tok, accept_len, out_tok, tgt_argmax)
    _check("qspec_verify_greedy_noalloc",
           load().qspec_verify_greedy_noalloc(_ptr(tgt_logits), _ptr(draft_tok), B, G1 - 1, V, _ptr(accept_len),
                                              _ptr(out_tok), _ptr(tgt_argmax), _stream(stream)))


def qspec_verify_sample(tgt_logits, draft_logits, draft_tok, u_accept, u_resample, accept_len, out_tok, ws,
                        accept_prob=None, p_tok=None, q_tok=None, stream=None):
    """Sampling verify (min(1, p/q) test, residual / bonus resampling from the given uniforms)."""
    _dt(tgt_logits, torch.bfloat16, "tgt_logits"); _dt(draft_logits, torch.bfloat16, "draft_logits")
    _dt(draft_tok, torch.int32, "draft_tok"); _dt(u_accept, torch.float32, "u_accept")
    _dt(u_resample, torch.float32, "u_resample"); _dt(accept_len, torch.int32, "accept_len")
    _dt(out_tok, torch.int32, "out_tok"); _dt(ws, torch.uint8, "ws")
    for name, t in (("accept_prob", accept_prob), ("p_tok", p_tok), ("q_tok", q_tok)):
        _dt(t, torch.float32, name)
    B, G1, V = tgt_logits.shape
    g = G1 - 1
    _need(draft_logits, B * g * V, "draft_logits"); _need(draft_tok, B * g, "draft_tok")
    _need(u_accept, B * g, "u_accept"); _need(u_resample, B * G1, "u_resample")
    _need(accept_len, B, "accept_len"); _need(out_tok, B * G1, "out_tok")
    _need(accept_prob, B * g, "accept_prob"); _need(p_tok, B * g, "p_tok"); _need(q_tok, B * g, "q_tok")
    _check("qspec_verify_sample",
           load().qspec_verify_sample(_ptr(tgt_logits), _ptr(draft_logits), _ptr(draft_tok), _ptr(u_accept),
                                      _ptr(u_resample), B, G1 - 1, V, _ptr(accept_len), _ptr(out_tok),
                                      _ptr(accept_prob), _ptr(p_tok), _ptr(q_tok), _ptr(ws), ws.numel(),
                                      _stream(stream)))


def qspec_verify_top1(tgt_logits, draft_logits, tgt_top1, draft_top1, ws, tgt_p1=None, draft_p1=None,
                      high=0.8, tally=None, stream=None):
    """Each mode's top-1 token and top-1 probability at every draft position; optional running tally
    (fp64 [8], accumulated: positions, agree, both>high, agree there, both<=high, agree there, sums of p1)."""
    _dt(tgt_logits, torch.bfloat16, "tgt_logits"); _dt(draft_logits, torch.bfloat16, "draft_logits")
    _dt(tgt_top1, torch.int32, "tgt_top1"); _dt(draft_top1, torch.int32, "draft_top1")
    _dt(tgt_p1, torch.float32, "tgt_p1"); _dt(draft_p1, torch.float32, "draft_p1")
    _dt(tally, torch.float64, "tally"); _dt(ws, torch.uint8, "ws")
    if tally is not None and tally.numel() < 8:
        raise ValueError("tally needs 8 fp64 entries")
    B, G1, V = tgt_logits.shape
    g = G1 - 1
    _need(draft_logits, B * g * V, "draft_logits")
    _need(tgt_top1, B * g, "tgt_top1"); _need(draft_top1, B * g, "draft_top1")
    _need(tgt_p1, B * g, "tgt_p1"); _need(draft_p1, B * g, "draft_p1")
    _check("qspec_verify_top1",
           load().qspec_verify_top1(_ptr(tgt_logits), _ptr(draft_logits), B, G1 - 1, V, _ptr(tgt_top1),
                                    _ptr(draft_top1), _ptr(tgt_p1), _ptr(draft_p1), float(high), _ptr(tally),
                                    _ptr(ws), ws.numel(), _stream(stream)))


def qspec_gather_rows(src, idx, dst, stream=None):
    """dst[m] = src[idx[m]] over the leading dimension (rows of src.numel() / src.shape[0] elements)."""
    _dt(idx, torch.int32, "idx")
    if src.dtype != dst.dtype:
        raise TypeError("src and dst must have the same dtype")
    n_src, n = src.shape[0], idx.numel()
    row_bytes = src[0].numel() * src.element_size()
    if dst.shape[0] != n or dst[0].numel() * dst.element_size() != row_bytes:
        raise ValueError("dst must be [len(idx), row of src]")
    _check("qspec_gather_rows", load().qspec_gather_rows(_ptr(src), n_src, row_bytes, _ptr(idx), n, _ptr(dst),
                                                         _stream(stream)))


def qspec_select_tokens(logits, tok, u=None, stream=None):
    """Next token per row of bf16 logits [R, V]: argmax when u is None, else an inverse-CDF draw with u [R]."""
    _dt(logits, torch.bfloat16, "logits"); _dt(tok, torch.int32, "tok"); _dt(u, torch.float32, "u")
    R, V = logits.shape
    _need(tok, R, "tok"); _need(u, R, "u")
    _check("qspec_select_tokens", load().qspec_select_tokens(_ptr(logits), R, V, _ptr(u), _ptr(tok), _stream(stream)))


def qspec_verify_tree_workspace_size(B, T, V):
    return int(load().qspec_verify_tree_workspace_size(B, T, V))


def new_tree_workspace(B, T, V, device="cuda"):
    """A zero-filled tree-verify workspace (zero once; calls keep it ready)."""
    n = qspec_verify_tree_workspace_size(B, T, V)
    if n == 0:
        raise ValueError("invalid tree shape")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def qspec_verify_tree_greedy(tgt_logits, tree_tok, tree_parent, accept_len, out_tok, ws, accept_nodes=None,
                             stream=None):
    """Greedy verify of a candidate tree: tgt_logits bf16 [B, T+1, V], tree_tok / tree_parent int32 [B, T]."""
    _dt(tgt_logits, torch.bfloat16, "tgt_logits"); _dt(tree_tok, torch.int32, "tree_tok")
    _dt(tree_parent, torch.int32, "tree_parent"); _dt(accept_len, torch.int32, "accept_len")
    _dt(out_tok, torch.int32, "out_tok"); _dt(accept_nodes, torch.int32, "accept_nodes"); _dt(ws, torch.uint8, "ws")
    B, R, V = tgt_logits.shape
    T = R - 1
    _need(tree_tok, B * T, "tree_tok"); _need(tree_parent, B * T, "tree_parent")
    _need(accept_len, B, "accept_len"); _need(out_tok, B * R, "out_tok"); _need(accept_nodes, B * T, "accept_nodes")
    _check("qspec_verify_tree_greedy",
           load().qspec_verify_tree_greedy(_ptr(tgt_logits), _ptr(tree_tok), _ptr(tree_parent), B, R - 1, V,
                                           _ptr(accept_len), _ptr(out_tok), _ptr(accept_nodes), _ptr(ws),
                                           ws.numel(), _stream(stream)))


def _ptr_any(t, name):
    """Pointer of a contiguous device tensor or pinned host tensor (qspec_copy's operands)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{name} must live on the GPU or in pinned host memory")
    return t.data_ptr()


def qspec_copy(dst, src, stream=None):
    """Copy src into dst (same number of bytes, device or pinned host tensors) with one kernel."""
    nb = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nb:
        raise ValueError(f"dst holds {dst.numel() * dst.element_size()} bytes, src {nb}")
    _check("qspec_copy", load().qspec_copy(_ptr_any(dst, "dst"), _ptr_any(src, "src"), nb, _stream(stream)))


def qspec_check_status(ws=None, stream=None):
    """Synchronise the stream and raise on device-side errors (timeouts, invalid draft tokens)."""
    _check("qspec_check_status", load().qspec_check_status(_ptr(ws), _stream(stream)))


def qspec_status_string(code: int) -> str:
    return load().qspec_status_string(int(code)).decode()


def new_verify_workspace(B, gamma, V, device="cuda"):
    """A zero-filled verify workspace of the required size (zero once; calls keep it ready)."""
    n = qspec_verify_workspace_size(B, gamma, V)
    if n == 0:
        raise ValueError("invalid verify shape")
    return torch.zeros(n, dtype=torch.uint8, device=device)
