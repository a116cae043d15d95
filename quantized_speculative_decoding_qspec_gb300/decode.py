"""Speculative decode loop on one set of shared 4-bit weights.

QSpec article "QSpec実行時の2つの量子化による推論の一致率を調べる", sections "QSpec の W4A4 モードと
W4A16 モード" and "測定スクリプト": one packed 4-bit weight set serves both modes; the W4A4 mode
drafts tokens one at a time and the W4A16 mode checks them together, and the measurement records
both modes' top-1 token and probability at every draft position.
Tutorial "Speculative Decodingとは？LLM生成を速くする方法", sections "draft modelとtarget modelの処理
フロー" (the loop), "3.36 token進んでも3.36倍速いとは限らない" (speedup ~ E[T] t_target /
(gamma t_draft + t_verify + t_overhead)) and "導入前に測る項目" (acceptance rate, accepted tokens per
iteration, draft and verification latency, output equivalence).

The model is a toy stand-in for a decoder (no trained weights exist here): an embedding table and a
stack of linears, [F x D], [D x F], [V x D], on seeded synthetic weights.  Its next-token logits
depend on the last token only, so no KV cache and no rollback are needed.

Every step on the device is a library kernel (embedding gather, the two linear modes, token
selection, verify, top-1 statistics).  The host only orders the calls, reads the accept lengths once
per iteration and writes the next input tokens.  The device work of an iteration is captured once
into CUDA graphs (draft phase, verify phase) and replayed.
"""
from __future__ import annotations

import time

import numpy as np
import torch

from . import qspec as q
from . import synthetic as syn


def _bf16_dev(bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


class ToyModel:
    """Embedding [V, D] (bf16) and linears [F, D], [D, F], [V, D] packed once (group 128, fp16 scales)."""

    def __init__(self, D: int, F: int, V: int, workload_id: int = 0, device: str = "cuda", weight_std: float = 0.02):
        self.D, self.F, self.V = D, F, V
        self.device = device
        self.shapes = [(F, D), (D, F), (V, D)]
        self.E = _bf16_dev(syn.embeddings(V, D, workload_id), device)
        self.layers = []
        for i, (N, K) in enumerate(self.shapes):
            W = _bf16_dev(syn.weights(N, K, workload_id, layer=100 + i, std=weight_std), device)
            Wp = torch.empty(N, K // 2, dtype=torch.uint8, device=device)
            S = torch.empty(N, K // 128, dtype=torch.float16, device=device)
            q.qspec_pack_weights(W, Wp, S)
            del W
            self.layers.append((Wp, S))
        q.qspec_check_status()
        self._bufs = {}

    def weight_bytes(self) -> int:
        return sum(Wp.numel() + 2 * S.numel() for Wp, S in self.layers)

    def _buffers(self, M: int):
        b = self._bufs.get(M)
        if b is None:
            # one workspace per layer: a linear workspace stays ready only for calls of its own shape
            b = {"x": torch.empty(M, self.D, dtype=torch.bfloat16, device=self.device),
                 "h": [torch.empty(M, N, dtype=torch.bfloat16, device=self.device) for N, _ in self.shapes[:-1]],
                 "ws": [q.new_linear_workspace(M, N, K, device=self.device) for N, K in self.shapes]}
            self._bufs[M] = b
        return b

    def forward(self, tok: torch.Tensor, logits: torch.Tensor, draft_mode: bool):
        """logits [M, V] bf16 <- model(tok [M] int32); draft_mode selects W4A4, else W4A16."""
        M = tok.numel()
        b = self._buffers(M)
        q.qspec_gather_rows(self.E, tok, b["x"])
        x = b["x"]
        lin = q.qspec_linear_w4a4 if draft_mode else q.qspec_linear_w4a16
        for i, (Wp, S) in enumerate(self.layers):
            y = logits if i == len(self.layers) - 1 else b["h"][i]
            lin(x, Wp, S, y, b["ws"][i])
            x = y
        return logits


class SpecDecoder:
    """B sequences decoded together: gamma W4A4 draft steps, one W4A16 pass over the gamma + 1
    positions, then the verify kernel (greedy, or sampling with caller-drawn uniforms)."""

    def __init__(self, model: ToyModel, B: int, gamma: int, sampling: bool = False, top1_stats: bool = True,
                 high: float = 0.8, use_graphs: bool = True):
        dev = model.device
        self.model, self.B, self.gamma, self.sampling = model, B, gamma, sampling
        self.top1_stats, self.high = top1_stats, high
        G1, V = gamma + 1, model.V
        i32 = dict(dtype=torch.int32, device=dev)
        # token ids position-major: tp[0] = last committed token, tp[1 + i] = draft token i
        self.tp = torch.zeros(G1, B, **i32)
        self.tv = torch.zeros(B, G1, **i32)          # target inputs, sequence-major
        self.d = torch.zeros(B, gamma, **i32)
        bb, ii = np.meshgrid(np.arange(B), np.arange(G1), indexing="ij")
        self.idx_tv = torch.from_numpy((ii * B + bb).reshape(-1).astype(np.int32)).to(dev)
        self.idx_d = torch.from_numpy(((ii[:, 1:]) * B + bb[:, 1:]).reshape(-1).astype(np.int32)).to(dev)
        self.idx_dl = torch.from_numpy(((ii[:, :-1]) * B + bb[:, :-1]).reshape(-1).astype(np.int32)).to(dev)
        self.dl = torch.empty(gamma, B, V, dtype=torch.bfloat16, device=dev)    # draft logits per step
        self.dlv = self.dl.view(B, gamma, V) if B == 1 else torch.empty(B, gamma, V, dtype=torch.bfloat16, device=dev)
        self.tl = torch.empty(B, G1, V, dtype=torch.bfloat16, device=dev)
        self.n = torch.zeros(B, **i32)
        self.out = torch.zeros(B, G1, **i32)
        self.ws = q.new_verify_workspace(B, gamma, V, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        self.u_draft = torch.zeros(gamma, B, **f32)
        self.u_acc = torch.zeros(B, gamma, **f32)
        self.u_res = torch.zeros(B, G1, **f32)
        self.t1 = torch.zeros(B, gamma, **i32)
        self.d1 = torch.zeros(B, gamma, **i32)
        self.tp1 = torch.zeros(B, gamma, **f32)
        self.dp1 = torch.zeros(B, gamma, **f32)
        self.tally = torch.zeros(8, dtype=torch.float64, device=dev)
        # target-only decoding, the baseline: at M = B (one token per sequence and step, for timing)
        # and padded to the verify pass's M = B (gamma + 1), whose logits come from the same kernel
        # configuration as the verify pass (for the output-equivalence check)
        self.tgt = {}
        for padded, M in ((False, B), (True, B * G1)):
            self.tgt[padded] = {"tok": torch.zeros(M, **i32), "logits": torch.empty(M, V, dtype=torch.bfloat16, device=dev),
                                "sel": torch.zeros(M, **i32), "u": torch.zeros(M, **f32)}
        # host staging (pinned)
        self.h_n = torch.zeros(B, dtype=torch.int32).pin_memory()
        self.h_out = torch.zeros(B, G1, dtype=torch.int32).pin_memory()
        self.h_last = torch.zeros(B, dtype=torch.int32).pin_memory()
        self.h_u = torch.zeros(gamma * B + B * gamma + B * G1, dtype=torch.float32).pin_memory()
        self.use_graphs = use_graphs
        self.graphs = None

    # ---- device phases (every call a library kernel)
    def _draft_phase(self):
        for i in range(self.gamma):
            self.model.forward(self.tp[i], self.dl[i], draft_mode=True)
            q.qspec_select_tokens(self.dl[i], self.tp[i + 1], u=self.u_draft[i] if self.sampling else None)

    def _verify_phase(self):
        V = self.model.V
        q.qspec_gather_rows(self.tp.view(-1, 1), self.idx_tv, self.tv.view(-1, 1))
        q.qspec_gather_rows(self.tp.view(-1, 1), self.idx_d, self.d.view(-1, 1))
        self.model.forward(self.tv.view(-1), self.tl.view(-1, V), draft_mode=False)
        if self.B > 1 and (self.sampling or self.top1_stats):
            q.qspec_gather_rows(self.dl.view(-1, V), self.idx_dl, self.dlv.view(-1, V))
        if self.sampling:
            q.qspec_verify_sample(self.tl, self.dlv, self.d, self.u_acc, self.u_res, self.n, self.out, self.ws)
        else:
            q.qspec_verify_greedy(self.tl, self.d, self.n, self.out, self.ws)
        if self.top1_stats:
            q.qspec_verify_top1(self.tl, self.dlv, self.t1, self.d1, self.ws, tgt_p1=self.tp1, draft_p1=self.dp1,
                                high=self.high, tally=self.tally)

    def _target_phase(self, padded):
        t = self.tgt[padded]
        self.model.forward(t["tok"], t["logits"], draft_mode=False)
        q.qspec_select_tokens(t["logits"], t["sel"], u=t["u"] if self.sampling else None)

    def _phases(self):
        return (self._draft_phase, self._verify_phase, lambda: self._target_phase(False),
                lambda: self._target_phase(True))

    def _capture(self):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):  # warm up (workspaces, lazy module loading) before capture
            for fn in self._phases():
                fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.tally.zero_()
        graphs = []
        for fn in self._phases():
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            graphs.append(g)
        self.graphs = graphs

    def _run(self, k):
        if self.use_graphs:
            if self.graphs is None:
                self._capture()
            self.graphs[k].replay()
        else:
            self._phases()[k]()

    # ---- host loop
    def run(self, first_tokens, n_iter: int, workload_id: int = 0, record: bool = False):
        """Decode n_iter iterations from first_tokens [B].  Returns a dict with the generated tokens
        per sequence, accept lengths [n_iter, B], per-phase device times (ms) and, when record is
        set, per-iteration copies of the draft tokens, logits and verify outputs."""
        B, gamma, G1 = self.B, self.gamma, self.gamma + 1
        if self.use_graphs and self.graphs is None:
            self._capture()
        self.tally.zero_()
        last = np.array(first_tokens, dtype=np.int32).reshape(B)  # a copy: updated in place below
        gen = [[] for _ in range(B)]
        ns = np.zeros((n_iter, B), dtype=np.int32)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        t_draft, t_verify = [], []
        rec = []
        stream = torch.cuda.current_stream()
        t0 = time.perf_counter()
        for it in range(n_iter):
            self.h_last.numpy()[:] = last
            self.tp[0].copy_(self.h_last, non_blocking=True)
            if self.sampling:
                ud = syn.uniforms((gamma, B), workload_id, syn.STREAM_U_DRAFT, it)
                ua = syn.uniforms((B, gamma), workload_id, syn.STREAM_U_ACCEPT, it)
                ur = syn.uniforms((B, G1), workload_id, syn.STREAM_U_RESAMPLE, it)
                h = self.h_u.numpy()
                h[:gamma * B] = ud.reshape(-1)
                h[gamma * B:2 * gamma * B] = ua.reshape(-1)
                h[2 * gamma * B:] = ur.reshape(-1)
                self.u_draft.view(-1).copy_(self.h_u[:gamma * B], non_blocking=True)
                self.u_acc.view(-1).copy_(self.h_u[gamma * B:2 * gamma * B], non_blocking=True)
                self.u_res.view(-1).copy_(self.h_u[2 * gamma * B:], non_blocking=True)
            ev[0].record(stream)
            self._run(0)
            ev[1].record(stream)
            self._run(1)
            ev[2].record(stream)
            self.h_n.copy_(self.n, non_blocking=True)
            self.h_out.copy_(self.out, non_blocking=True)
            stream.synchronize()
            t_draft.append(ev[0].elapsed_time(ev[1]))
            t_verify.append(ev[1].elapsed_time(ev[2]))
            n = self.h_n.numpy().copy()
            out = self.h_out.numpy().copy()
            ns[it] = n
            for b in range(B):
                gen[b].extend(int(t) for t in out[b, :n[b] + 1])
                last[b] = out[b, n[b]]
            if record:
                rec.append({"tokens_in": self.tp[0].cpu().numpy(), "d": self.d.cpu().numpy(),
                            "dl": self.dlv.cpu().clone(), "tl": self.tl.cpu().clone(),
                            "n": n, "out": out})
        wall = time.perf_counter() - t0
        q.qspec_check_status(self.ws)
        res = {"generated": gen, "accept_len": ns, "t_draft_ms": np.array(t_draft), "t_verify_ms": np.array(t_verify),
               "wall_s": wall, "records": rec}
        if self.top1_stats:
            res["tally"] = self.tally.cpu().numpy()
        return res

    def run_target_only(self, first_tokens, n_tokens: int, workload_id: int = 0, padded: bool = False):
        """Plain decoding with the W4A16 model alone, one target pass per token (the baseline).
        padded: run each step at the verify pass's M (sequence b's token in rows b(gamma+1) ..
        b(gamma+1)+gamma), so that its logits are bit-identical to the verify pass's."""
        B = self.B
        G1 = self.gamma + 1 if padded else 1
        t = self.tgt[padded]
        if self.use_graphs and self.graphs is None:
            self._capture()
        last = np.array(first_tokens, dtype=np.int32).reshape(B)  # a copy: updated in place below
        gen = [[] for _ in range(B)]
        h_tt = torch.zeros(B * G1, dtype=torch.int32).pin_memory()
        h_sel = torch.zeros(B * G1, dtype=torch.int32).pin_memory()
        h_u = torch.zeros(B * G1, dtype=torch.float32).pin_memory()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        t_target = []
        stream = torch.cuda.current_stream()
        t0 = time.perf_counter()
        for k in range(n_tokens):
            h_tt.numpy()[:] = np.repeat(last, G1)
            t["tok"].copy_(h_tt, non_blocking=True)
            if self.sampling:
                u = syn.uniforms((B,), workload_id, syn.STREAM_U_DRAFT, 10_000_000 + k)
                h_u.numpy()[:] = np.repeat(u, G1)
                t["u"].copy_(h_u, non_blocking=True)
            ev[0].record(stream)
            self._run(3 if padded else 2)
            ev[1].record(stream)
            h_sel.copy_(t["sel"], non_blocking=True)
            stream.synchronize()
            t_target.append(ev[0].elapsed_time(ev[1]))
            sel = h_sel.numpy()
            for b in range(B):
                last[b] = sel[b * G1]
                gen[b].append(int(last[b]))
        wall = time.perf_counter() - t0
        q.qspec_check_status()
        return {"generated": gen, "t_target_ms": np.array(t_target), "wall_s": wall}


def summarize(spec: dict, target: dict, gamma: int) -> dict:
    """The tutorial's measures: acceptance rate, accepted tokens per iteration (E[T]), draft and
    verification latency, the speedup estimate E[T] t_target / (gamma t_draft + t_verify + t_overhead)
    and the measured tokens-per-second ratio against target-only decoding."""
    n = spec["accept_len"]
    iters, B = n.shape
    ET = float(np.mean(n + 1))
    t_draft_tok = float(np.median(spec["t_draft_ms"])) / gamma
    t_verify = float(np.median(spec["t_verify_ms"]))
    t_target = float(np.median(target["t_target_ms"]))
    iter_wall_ms = 1e3 * spec["wall_s"] / iters
    t_overhead = max(0.0, iter_wall_ms - (gamma * t_draft_tok + t_verify))
    spec_tok_s = B * ET * iters / spec["wall_s"]
    n_target_tok = len(target["generated"][0])
    target_tok_s = B * n_target_tok / target["wall_s"]
    out = {
        "acceptance_rate": float(np.mean(n) / gamma),
        "accepted_tokens_per_iteration": ET,
        "t_draft_ms_per_token": t_draft_tok,
        "t_verify_ms": t_verify,
        "t_target_ms": t_target,
        "t_overhead_ms": t_overhead,
        "speedup_model": ET * t_target / (gamma * t_draft_tok + t_verify + t_overhead),
        "speedup_model_device_only": ET * t_target / (gamma * t_draft_tok + t_verify),
        "spec_tokens_per_s": spec_tok_s,
        "target_only_tokens_per_s": target_tok_s,
        "speedup_measured": spec_tok_s / target_tok_s,
    }
    if "tally" in spec:
        t = spec["tally"]
        out["top1"] = {
            "positions": int(t[0]),
            "agreement": float(t[1] / t[0]) if t[0] else None,
            "mean_p1_verify_mode": float(t[6] / t[0]) if t[0] else None,
            "mean_p1_draft_mode": float(t[7] / t[0]) if t[0] else None,
            "both_high_share": float(t[2] / t[0]) if t[0] else None,
            "agreement_both_high": float(t[3] / t[2]) if t[2] else None,
            "agreement_both_low": float(t[5] / t[4]) if t[4] else None,
        }
    return out
