"""Benchmark of the QSpec hot path on one GB300 (or N independent replicas under torchrun).

A step is one QSpec decode iteration over Llama-3-8B-shaped decode linears (q, k, v, o, gate, up,
down, lm_head; weights [N, K] packed to INT4 once, before timing), for one sequence with draft
length 3:
  * draft:  3 x W4A4 linears at M = 1 token over all 8 layers (fused activation quantiser);
  * verify: 1 x W4A16 linears at M = 4 tokens over all 8 layers, on the same packed weights;
  * verify kernels over bf16 logits [1, 4, 128256]: greedy verify and sampling verify.
Inputs are seeded synthetic stand-ins (weights N(0, 0.02); activations N(0, 1) with 1% outlier
channels x20; spiked target logits and noisy draft logits).  The packed weights (1.5 GB read per
step) are far larger than L2, so no flush is needed between steps.

value = algorithmic bytes of the step (packed weights + scales + activations + outputs of every
linear, plus the logits every verify kernel must read) / device time per step, in GB/s.

``--impl reference`` times the CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A16/W4A4 GEMM HBM GB/s & TOPS vs roofline; verify positions/sec"
GAMMA = 3
VOCAB = 128256
LAYERS = [  # name, N (out), K (in)
    ("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
    ("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336), ("lm_head", VOCAB, 4096),
]
# The linears of a decoder layer that read the same activations go out as one grouped launch
# (qspec_linear_group): q, k and v read the normed hidden state, gate and up the post-attention one.
GROUPS = [("qkv", ("q", "k", "v")), ("o", ("o",)), ("gate_up", ("gate", "up")), ("down", ("down",)),
          ("lm_head", ("lm_head",))]
LEADER = {m: members[0] for _, members in GROUPS for m in members}
SHAPE = {name: (N, K) for name, N, K in LAYERS}
WORKLOAD = ("Llama-3-8B-shaped decode linears q,k,v,o,gate,up,down,lm_head ([N,K] packed INT4, group 128, "
            "fp16 scales; q,k,v and gate,up read one input each and go out as grouped launches); one QSpec "
            "iteration for 1 sequence, gamma=3: 3 W4A4 draft passes at M=1 + 1 W4A16 verify pass at M=4, then "
            "greedy and sampling verify over bf16 logits [1,4,128256]")


def linear_bytes(M, N, K):
    """Algorithmic bytes of one linear: packed weights, fp16 scales, bf16 x and y."""
    return N * K // 2 + N * (K // 128) * 2 + M * K * 2 + M * N * 2


def verify_bytes(B, gamma, V, sampling):
    """Logits bytes a verify call must read (all rows once; pass 2 re-reads one row pair)."""
    if not sampling:
        return B * (gamma + 1) * V * 2
    return B * (2 * gamma + 1) * V * 2 + B * 2 * V * 2


def group_bytes(M, members):
    """Algorithmic bytes of one grouped launch: every part's weights, scales and y; x once."""
    K = SHAPE[members[0]][1]
    return sum(linear_bytes(M, SHAPE[m][0], K) for m in members) - (len(members) - 1) * M * K * 2


def step_bytes():
    lin16 = sum(group_bytes(GAMMA + 1, members) for _, members in GROUPS)
    lin4 = sum(group_bytes(1, members) for _, members in GROUPS)
    ver = verify_bytes(1, GAMMA, VOCAB, False) + verify_bytes(1, GAMMA, VOCAB, True)
    return {"w4a4": GAMMA * lin4, "w4a16": lin16, "verify": ver, "total": GAMMA * lin4 + lin16 + ver}


def step_flops():
    return {"w4a4": GAMMA * sum(2 * 1 * N * K for _, N, K in LAYERS),
            "w4a16": sum(2 * (GAMMA + 1) * N * K for _, N, K in LAYERS)}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# CUDA sources each kernel family's launches are built from (a change to any of them invalidates the
# recorded DRAM traffic)
KERNEL_SOURCES = {
    "linear_w4a4": ["gemv.cu", "gemv_impl.cuh", "gemv_a4.cu", "linear.cu", "common.cuh"],
    "linear_w4a16": ["gemv.cu", "gemv_impl.cuh", "gemv_a16.cu", "linear.cu", "common.cuh"],
    "verify_greedy": ["verify.cu", "common.cuh"],
    "verify_sample": ["verify.cu", "common.cuh"],
}


def kernel_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        ent = d[kernel]
    except Exception:
        return None
    if ent.get("source_sha256") != source_hash(KERNEL_SOURCES[kernel]):
        return None
    return ent.get("dram_bytes_per_launch")


def source_hash(files):
    """sha256 over the named files of the library's csrc directory (name + contents, in order)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_speculative_decoding_qspec_gb300", "csrc")
    for name in files:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()


# ---------------------------------------------------------------------------------------------- CPU oracle


def oracle_sample_step(data, frac):
    """One oracle pass over a row sample (fraction ``frac`` of every layer's output rows) plus the
    full verify; returns the algorithmic bytes that sample stands for."""
    import oracle
    nbytes = 0
    for name, N, K in LAYERS:
        rows = max(1, int(round(frac * N)))
        Wp, S = data["packed"][name]
        Wp, S = Wp[:rows], S[:rows]
        lead = LEADER[name]
        shared_x = lead != name  # a group's input is counted once, with its first member
        for d in range(GAMMA):
            oracle.linear_w4a4(data["x1"][lead][d], Wp, S)
            nbytes += linear_bytes(1, rows, K) - (K * 2 if shared_x else 0)
        oracle.linear_w4a16(data["x4"][lead], Wp, S)
        nbytes += linear_bytes(GAMMA + 1, rows, K) - ((GAMMA + 1) * K * 2 if shared_x else 0)
    v = data["verify"]
    oracle.verify_greedy(v["tgt"], v["d_greedy"])
    oracle.verify_sample(v["tgt"], v["drf"], v["d_sample"], v["u_acc"], v["u_res"])
    nbytes += verify_bytes(1, GAMMA, VOCAB, False) + verify_bytes(1, GAMMA, VOCAB, True)
    return nbytes


def oracle_inputs(frac):
    """Seeded inputs for the oracle sample: only the sampled weight rows are generated and packed."""
    import numpy as np
    import oracle
    from quantized_speculative_decoding_qspec_gb300 import synthetic as syn
    data = {"packed": {}, "x1": {}, "x4": {}}
    for li, (name, N, K) in enumerate(LAYERS):
        rows = max(1, int(round(frac * N)))
        g = syn.rng(1, syn.STREAM_WEIGHTS, li)
        w = g.standard_normal((rows, K), dtype=np.float32) * np.float32(0.02)  # same rows as the GPU's
        data["packed"][name] = oracle.pack_weights(syn.f32_to_bf16_bits(w))
        if LEADER[name] == name:
            data["x1"][name] = [syn.activations(1, K, 1, step=10 * li + d) for d in range(GAMMA)]
            data["x4"][name] = syn.activations(GAMMA + 1, K, 1, step=10 * li + 9)
    data["verify"] = verify_data()
    return data


def verify_data():
    from quantized_speculative_decoding_qspec_gb300 import synthetic as syn
    g = syn.verify_inputs(1, GAMMA, VOCAB, 0.5, workload_id=1)
    s = syn.verify_inputs(1, GAMMA, VOCAB, 0.5, workload_id=1, sampling=True)
    return {"tgt": g["tgt"], "drf": g["drf"], "d_greedy": g["d"], "d_sample": s["d"], "u_acc": s["u_acc"],
            "u_res": s["u_res"]}


def time_oracle(budget_s, frac=None):
    """Oracle throughput on a bounded sample; calibrates the row fraction to the time budget."""
    if frac is None:
        probe = 1.0 / 4096
        data = oracle_inputs(probe)
        t0 = time.perf_counter()
        oracle_sample_step(data, probe)
        dt = time.perf_counter() - t0
        frac = min(1.0, max(probe, probe * budget_s / max(dt, 1e-3)))
    data = oracle_inputs(frac)
    t0 = time.perf_counter()
    nbytes = oracle_sample_step(data, frac)
    dt = time.perf_counter() - t0
    return nbytes, dt, frac


def _oracle_worker(frac, q_ready, ev_go, q_out):
    """One process of the all-cores oracle timing (started with spawn, BLAS pinned to one thread by
    the inherited environment): build the sample, wait for the start signal, time one pass."""
    data = oracle_inputs(frac)
    q_ready.put(1)
    ev_go.wait()
    t0 = time.time()
    nbytes = oracle_sample_step(data, frac)
    q_out.put((t0, time.time(), nbytes))


def time_oracle_all_cores(frac, procs):
    """The oracle on every host core: `procs` single-threaded processes run the same row sample at
    once; bytes of all of them / wall time from the first start to the last finish."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q_ready, q_out, ev_go = ctx.Queue(), ctx.Queue(), ctx.Event()
    ps = [ctx.Process(target=_oracle_worker, args=(frac, q_ready, ev_go, q_out)) for _ in range(procs)]
    import queue

    def get(qq, deadline):  # a result, or an error as soon as a worker has died
        while True:
            try:
                return qq.get(timeout=1.0)
            except queue.Empty:
                if time.time() > deadline or any(p_.exitcode not in (None, 0) for p_ in ps):
                    for p_ in ps:
                        if p_.is_alive():
                            p_.terminate()
                    raise RuntimeError("all-cores oracle timing: a worker failed")

    for p_ in ps:
        p_.start()
    deadline = time.time() + 900
    for _ in ps:
        get(q_ready, deadline)
    ev_go.set()
    res = [get(q_out, deadline) for _ in ps]
    for p_ in ps:
        p_.join()
    return sum(r[2] for r in res), max(r[1] for r in res) - min(r[0] for r in res)


def threads_used():
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var) == "1":
            return 1
    return os.cpu_count()


# ---------------------------------------------------------------------------------------------- replicas


def reduce_max(value, device="cpu"):
    """Max of a float over all ranks (identity without an initialised process group)."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, bytes_per_step, steps, elapsed_max):
    """Whole-job GB/s of ``world`` independent replicas timed by the slowest rank."""
    return world * bytes_per_step * steps / elapsed_max / 1e9


# ---------------------------------------------------------------------------------------------- GPU arm


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region.  Entering waits (at most a few
    seconds) for the first sample, so a timed region shorter than the sampling interval still has
    the reading taken just before it; every sample up to the exit counts."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def _read(self):
        for line in self.proc.stdout:
            if line.strip():
                self.lines.append(line)

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
            time.sleep(0.01)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)  # one more sampling interval, so the region's end is covered too
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except Exception:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def gpu_arm(args, rank, world):
    import numpy as np
    import torch

    import __graft_entry__ as g
    g.build()
    from quantized_speculative_decoding_qspec_gb300 import qspec as q
    from quantized_speculative_decoding_qspec_gb300 import synthetic as syn

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    # ---- weights: generate, pack on the GPU (timed separately: step a1 is offline), drop bf16
    packed, pack_times, pack_bytes = {}, [], 0
    for li, (name, N, K) in enumerate(LAYERS):
        W = bf(syn.weights(N, K, 1, layer=li))
        Wp = torch.empty(N, K // 2, dtype=torch.uint8, device=dev)
        S = torch.empty(N, K // 128, dtype=torch.float16, device=dev)
        q.qspec_pack_weights(W, Wp, S)  # warm
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        q.qspec_pack_weights(W, Wp, S)
        e1.record()
        torch.cuda.synchronize()
        pack_times.append(e0.elapsed_time(e1) * 1e-3)
        pack_bytes += N * K * 2 + N * K // 2 + N * (K // 128) * 2
        packed[name] = (Wp, S)
        del W
    torch.cuda.empty_cache()

    # ---- per-step inputs (resident in HBM) and outputs
    # the step's activations are views of one device buffer, so that the end-to-end run moves them
    # with one host-to-device copy per step
    xbuf = torch.empty(sum((2 * GAMMA + 1) * K for n, _, K in LAYERS if LEADER[n] == n), dtype=torch.bfloat16,
                       device=dev)
    x1, x4, off = {}, {}, 0
    for li, (n, N, K) in enumerate(LAYERS):
        if LEADER[n] != n:  # the group's later members read the first member's input
            continue
        x1[n] = []
        for d in range(GAMMA):
            x1[n].append(xbuf[off:off + K].view(1, K))
            x1[n][d].copy_(bf(syn.activations(1, K, 1, step=10 * li + d)))
            off += K
        x4[n] = xbuf[off:off + (GAMMA + 1) * K].view(GAMMA + 1, K)
        x4[n].copy_(bf(syn.activations(GAMMA + 1, K, 1, step=10 * li + 9)))
        off += (GAMMA + 1) * K
    for n, _, _ in LAYERS:
        x1[n], x4[n] = x1[LEADER[n]], x4[LEADER[n]]
    y1 = {n: torch.empty(1, N, dtype=torch.bfloat16, device=dev) for n, N, K in LAYERS}
    y4 = {n: torch.empty(GAMMA + 1, N, dtype=torch.bfloat16, device=dev) for n, N, K in LAYERS}
    # one grouped call per (group, draft position) and per group for the verify pass, built once
    gws = {gn: {M: q.new_linear_group_workspace(M, [SHAPE[m][0] for m in members], SHAPE[members[0]][1], device=dev)
                for M in (1, GAMMA + 1)} for gn, members in GROUPS}
    calls4 = [{gn: q.LinearGroup(4, x1[members[0]][d], [(packed[m][0], packed[m][1], y1[m]) for m in members],
                                 gws[gn][1]) for gn, members in GROUPS} for d in range(GAMMA)]
    calls16 = {gn: q.LinearGroup(16, x4[members[0]], [(packed[m][0], packed[m][1], y4[m]) for m in members],
                                 gws[gn][GAMMA + 1]) for gn, members in GROUPS}
    # the verify inputs are views of one device buffer (each at a 256-byte offset) and the four
    # verify results views of one 64-byte buffer (16-byte offsets), so that the end-to-end run moves
    # each side with one copy per step
    vd = verify_data()
    vsrc = [("tgt", vd["tgt"].view(np.int16), torch.bfloat16), ("drf", vd["drf"].view(np.int16), torch.bfloat16),
            ("dg", vd["d_greedy"], torch.int32), ("ds", vd["d_sample"], torch.int32),
            ("ua", vd["u_acc"], torch.float32), ("ur", vd["u_res"], torch.float32)]
    voff, off = {}, 0
    for k, a, _ in vsrc:
        voff[k] = off
        off += (a.nbytes + 255) // 256 * 256
    vbuf = torch.empty(off, dtype=torch.uint8, device=dev)
    vin = {}
    for k, a, dt in vsrc:
        view = vbuf[voff[k]:voff[k] + a.nbytes].view(dt).view(a.shape)
        view.copy_(torch.from_numpy(np.ascontiguousarray(a)).view(dt))
        vin[k] = view
    tgt, drf, dg, ds, ua, ur = (vin[k] for k in ("tgt", "drf", "dg", "ds", "ua", "ur"))
    ws_g = q.new_verify_workspace(1, GAMMA, VOCAB, device=dev)
    ws_s = q.new_verify_workspace(1, GAMMA, VOCAB, device=dev)
    res = torch.zeros(16, dtype=torch.int32, device=dev)
    n_g, o_g = res[0:1], res[4:4 + GAMMA + 1].view(1, GAMMA + 1)
    n_s, o_s = res[8:9], res[12:12 + GAMMA + 1].view(1, GAMMA + 1)

    vstream = torch.cuda.Stream(device=dev)

    def step(timers=None, per_kernel=False, before_verify=None):
        """One step.  With timers: external events around each kernel family (per_kernel=False; the
        launches of a family stay back to back) or around every kernel (per_kernel=True).
        before_verify: called between the linears and the verify calls (the end-to-end run joins
        its copy stream there)."""
        def event():
            e = torch.cuda.Event(enable_timing=True, external=True)
            e.record()
            return e

        def timed(kind, fn):
            if timers is None or not per_kernel:
                fn()
                return
            a = event()
            fn()
            timers.append((kind, a, event()))

        def family(fam, body):
            if timers is None or per_kernel:
                body()
                return
            a = event()
            body()
            timers.append(((fam, "*"), a, event()))

        def draft():
            for d in range(GAMMA):
                for gn, _ in GROUPS:
                    timed(("w4a4", gn), calls4[d][gn].run)

        def verify_pass():
            for gn, _ in GROUPS:
                timed(("w4a16", gn), calls16[gn].run)

        family("w4a4", draft)
        family("w4a16", verify_pass)
        if before_verify is not None:
            before_verify()
        if timers is None:
            # the two verify calls read the same logits and nothing of each other's: greedy goes on a
            # second stream beside sampling (their short latency-bound chains overlap) and joins
            # before the step ends.  The instrumented steps keep them in order, one family at a time.
            main = torch.cuda.current_stream()
            vstream.wait_stream(main)
            with torch.cuda.stream(vstream):
                q.qspec_verify_greedy(tgt, dg, n_g, o_g, ws_g)
            q.qspec_verify_sample(tgt, drf, ds, ua, ur, n_s, o_s, ws_s)
            main.wait_stream(vstream)
            return
        family("greedy", lambda: timed(("greedy", ""), lambda: q.qspec_verify_greedy(tgt, dg, n_g, o_g, ws_g)))
        family("sample", lambda: timed(("sample", ""),
                                       lambda: q.qspec_verify_sample(tgt, drf, ds, ua, ur, n_s, o_s, ws_s)))

    launches_per_step = GAMMA * len(GROUPS) + len(GROUPS) + 1 + 2

    for _ in range(max(args.warmup, 3)):
        step()
    q.qspec_check_status(ws_g)
    q.qspec_check_status(ws_s)

    # ---- CUDA graphs: one plain graph for the timed loop, and a pool of instrumented graphs whose
    # external events time the kernel families (the roofline figures) and, in a few of them, every
    # kernel (the per-layer breakdown).  The instrumented graphs replay in a region of their own
    # after the timed one, so the headline number never includes their events.
    # (--eager: the same launches issued directly, for profilers that do not follow stream capture)
    n_inst = max(2, args.timed_graphs)
    n_kern = min(4, n_inst // 2)
    inst = []
    if args.eager:
        replay = step
        for i in range(n_inst):
            timers = []
            inst.append((lambda t=timers, pk=i < n_kern: step(t, pk), timers))
    else:
        side = torch.cuda.Stream(device=dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            step()
        replay = graph.replay
        for i in range(n_inst):
            gi = torch.cuda.CUDAGraph()
            timers = []
            with torch.cuda.graph(gi, stream=side):
                step(timers, i < n_kern)
            inst.append((gi.replay, timers))
    for _ in range(3):
        replay()
    torch.cuda.synchronize()

    dist = world > 1
    if dist:
        import torch.distributed as tdist
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        if dist:
            tdist.barrier()
        torch.cuda.synchronize()
        start.record()
        for _ in range(args.steps):
            replay()
        stop.record()
        torch.cuda.synchronize()
        if dist:
            tdist.barrier()
    elapsed = reduce_max(start.elapsed_time(stop) * 1e-3, dev)
    q.qspec_check_status(ws_g)
    q.qspec_check_status(ws_s)
    # the instrumented steps, back to back after the timed region
    for run_inst, _ in inst:
        run_inst()
    torch.cuda.synchronize()
    q.qspec_check_status(ws_g)
    q.qspec_check_status(ws_s)

    # ---- per-kernel durations from the instrumented steps
    per_kind = {}
    for _, timers in inst:
        for kind, a, b in timers:
            per_kind.setdefault(kind, []).append(a.elapsed_time(b) * 1e-3)

    sb = step_bytes()
    sf = step_flops()
    ms_per_step = elapsed / args.steps * 1e3
    value = replica_throughput(world, sb["total"], args.steps, elapsed)

    def family_time(fam):
        v = per_kind[(fam, "*")]
        return sum(v) / len(v)

    fam_bytes = {"w4a4": sb["w4a4"], "w4a16": sb["w4a16"],
                 "greedy": verify_bytes(1, GAMMA, VOCAB, False), "sample": verify_bytes(1, GAMMA, VOCAB, True)}
    fam_time = {f: family_time(f) for f in fam_bytes}
    fam_launches = {"w4a4": GAMMA * len(GROUPS), "w4a16": len(GROUPS), "greedy": 1, "sample": 2}
    dominant = max(fam_time, key=fam_time.get)
    hbm_peak, peak_kind = peaks()
    achieved = fam_bytes[dominant] / fam_time[dominant] / 1e9
    kernel_names = {"w4a4": "linear_w4a4", "w4a16": "linear_w4a16", "greedy": "verify_greedy",
                    "sample": "verify_sample"}
    layers = {}
    for (fam, name), v in sorted(per_kind.items()):
        if fam in ("w4a4", "w4a16") and name != "*":
            members = dict(GROUPS)[name]
            M = 1 if fam == "w4a4" else GAMMA + 1
            t = sum(v) / len(v)
            flops = sum(2 * M * SHAPE[m][0] * SHAPE[m][1] for m in members)
            layers[f"{fam}:{name}"] = {"us": round(t * 1e6, 2),
                                       "GB_s": round(group_bytes(M, members) / t / 1e9, 1),
                                       "TOPS": round(flops / t / 1e12, 3)}
    ver_t = {f: fam_time[f] for f in ("greedy", "sample")}

    # ---- one decoder layer: its grouped launches (q+k+v, o, gate+up, down) back to back in one CUDA
    # graph per mode, rotating through weight copies of at least 3x L2 (113 MB of packed weights per layer)
    dec_groups = [(gn, members) for gn, members in GROUPS if gn != "lm_head"]
    dec_names = [m for _, members in dec_groups for m in members]
    dec_bytes = {4: sum(group_bytes(1, members) for _, members in dec_groups),
                 16: sum(group_bytes(GAMMA + 1, members) for _, members in dec_groups)}
    R_dec = copies_for(dec_bytes[4])
    dec_sets = [{n: packed[n] for n in dec_names}]
    dec_sets += [{n: (packed[n][0].clone(), packed[n][1].clone()) for n in dec_names} for _ in range(R_dec - 1)]
    decoder_layer = {}
    for abits, M in ((4, 1), (16, GAMMA + 1)):
        xin = {n: (x1[n][0] if abits == 4 else x4[n]) for n in dec_names}
        yout = {n: (y1[n] if abits == 4 else y4[n]) for n in dec_names}
        calls = []
        for i in range(R_dec):
            gl = []
            for gn, members in dec_groups:
                K = SHAPE[members[0]][1]
                ws = q.new_linear_group_workspace(M, [SHAPE[m][0] for m in members], K, device=dev)
                gl.append(q.LinearGroup(abits, xin[members[0]], [(*dec_sets[i][m], yout[m]) for m in members], ws))
            calls.append(gl)

        def layer_call(i, calls=calls):
            for c in calls[i]:
                c.run()

        t_dec = _rotating_time([(lambda i=i: layer_call(i)) for i in range(R_dec)])
        decoder_layer[f"w4a{abits}_M{M}"] = {"us": round(t_dec * 1e6, 2),
                                              "GB_s": round(dec_bytes[abits] / t_dec / 1e9, 1),
                                              "hbm_frac": round(dec_bytes[abits] / t_dec / 1e9 / peaks()[0], 4)}
        del calls
    q.qspec_check_status()
    del dec_sets

    # ---- end to end through the public API with host buffers: H2D of the step's inputs from pinned
    # memory, the calls, D2H of the verify results.  The activations go over in one copy ahead of
    # the linears; the verify inputs are copied on a second stream while the linears run and joined
    # before the verify calls (the previous step's work is finished before that stream starts).
    host_x = xbuf.cpu().pin_memory()
    host_v = vbuf.cpu().pin_memory()
    host_res = torch.empty_like(res, device="cpu").pin_memory()
    h2d = host_x.numel() * host_x.element_size() + host_v.numel() * host_v.element_size()
    d2h = host_res.numel() * host_res.element_size()
    copy_stream = torch.cuda.Stream()

    def e2e_step():
        # the library's copy kernel (qspec_copy) moves each side: a copy-engine transfer of these few
        # hundred KB is mostly fixed latency that the first linear would wait out (measured: the
        # activations' cudaMemcpyAsync added 16 us a step, the results' 6.5 us)
        main = torch.cuda.current_stream()
        copy_stream.wait_stream(main)
        with torch.cuda.stream(copy_stream):
            q.qspec_copy(vbuf, host_v)
        q.qspec_copy(xbuf, host_x)
        step(before_verify=lambda: main.wait_stream(copy_stream))
        q.qspec_copy(host_res, res)

    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(e2e_steps):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    e2e_t_eager = e0.elapsed_time(e1) * 1e-3 / e2e_steps

    # the same end-to-end step captured once into a CUDA graph through the same public calls (the
    # H2D copies from the pinned buffers, the library calls, the D2H copies) and replayed per step
    # -- how a serving loop drives it (the decode loop does the same)
    if args.eager:
        e2e_t = e2e_t_eager
        e2e_how = "eager"
    else:
        s_cap = torch.cuda.Stream()
        s_cap.wait_stream(torch.cuda.current_stream())
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s_cap):
            e2e_step()
            torch.cuda.current_stream().synchronize()
            with torch.cuda.graph(g_e2e):
                e2e_step()
        torch.cuda.current_stream().wait_stream(s_cap)
        for _ in range(3):
            g_e2e.replay()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(e2e_steps):
            g_e2e.replay()
        e1.record()
        torch.cuda.synchronize()
        e2e_t = e0.elapsed_time(e1) * 1e-3 / e2e_steps
        e2e_how = "graph"
    e2e_val = world * sb["total"] / e2e_t / 1e9

    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int4 weights x bf16 / int4 activations, fp32 accumulate; fp32 softmax",
        "data": "synthetic (seeded; random-init weights of the named shapes)",
        "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (1.5 GB of packed weights streamed per step)",
                   "timing": ("direct launches" if args.eager else "CUDA graph replays") +
                             " of whole steps, CUDA events on the launching stream"},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"kernel": kernel_names[dominant], "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": hbm_peak, "peak_source": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4),
                     "traffic": kernel_traffic(kernel_names[dominant]),
                     "algorithmic_bytes_per_launch": fam_bytes[dominant] // fam_launches[dominant],
                     "algorithmic_bytes_per_step": fam_bytes[dominant],
                     "timing": f"CUDA events around the kernel family in {n_inst - n_kern} instrumented steps "
                               "replayed back to back after the timed region"},
        "breakdown": {
            "step_bytes": sb,
            "family_us_per_step": {k: round(v * 1e6, 2) for k, v in fam_time.items()},
            "w4a4_TOPS": round(sf["w4a4"] / fam_time["w4a4"] / 1e12, 3),
            "w4a16_TOPS": round(sf["w4a16"] / fam_time["w4a16"] / 1e12, 3),
            "verify_positions_per_s": {k: round((GAMMA + 1) / v, 1) for k, v in ver_t.items()},
            "verify_GB_s": {k: round(fam_bytes[k] / v / 1e9, 1) for k, v in ver_t.items()},
            "layers": layers,
            "layers_timing": f"CUDA events around every kernel in {n_kern} instrumented steps after the timed "
                             "region (separating the launches adds gaps: per-layer times are upper bounds)",
            "pack_GB_s": round(pack_bytes / sum(pack_times) / 1e9, 1),
            "decoder_layer": decoder_layer,
            "decoder_layer_timing": ("the grouped launches q+k+v, o, gate+up, down back to back in one CUDA graph, "
                                     "rotating through "
                                     f"{R_dec} weight copies (at least 3x L2); W4A4 at M=1, W4A16 at M={GAMMA + 1}"),
        },
        "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "ms_per_step": round(e2e_t * 1e3, 4),
                "how": ("the step's public-API calls with pinned-host H2D of that step's inputs (activations in "
                        "one copy ahead of the linears, verify inputs in one copy on a second stream overlapping "
                        "them) and one D2H of the four verify results, each copy by the library's copy kernel "
                        "(qspec_copy, reading or writing the pinned host buffers over the host link), " +
                        ("captured once into a CUDA graph and replayed per step, inside the CUDA-event region"
                         if e2e_how == "graph" else "eager calls per step inside the CUDA-event region")),
                "eager_value": round(world * sb["total"] / e2e_t_eager / 1e9, 2),
                "eager_ms_per_step": round(e2e_t_eager * 1e3, 4)},
    }
    clk = clk.summary()
    if clk:
        result["clocks"] = clk
    return result


def profile_case(spec, reps):
    """Run one kernel of the step repeatedly (for profilers): LAYER:MODE:M, e.g. lm_head:a4:1, a group
    of the step as one grouped launch (qkv:a4:1, gate_up:a16:4), or verify:greedy / verify:sample on
    the step's logits."""
    import numpy as np
    import torch

    import __graft_entry__ as g
    g.build()
    from quantized_speculative_decoding_qspec_gb300 import qspec as q
    from quantized_speculative_decoding_qspec_gb300 import synthetic as syn
    dev = torch.device("cuda", 0)

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    parts = spec.split(":")
    if parts[0] == "verify":
        if len(parts) == 5:  # verify:MODE:B:GAMMA:V -- a sweep cell
            Bc, gc, Vc = int(parts[2]), int(parts[3]), int(parts[4])
            vi = syn.verify_inputs(Bc, gc, Vc, 0.5, workload_id=4, sampling=parts[1] != "greedy")
            vd = {"tgt": vi["tgt"], "drf": vi.get("drf", vi["tgt"][:, :gc]), "d_greedy": vi["d"], "d_sample": vi["d"],
                  "u_acc": vi.get("u_acc", np.zeros((Bc, gc), np.float32)),
                  "u_res": vi.get("u_res", np.zeros((Bc, gc + 1), np.float32))}
        else:
            Bc, gc, Vc = 1, GAMMA, VOCAB
            vd = verify_data()
        tgt, drf = bf(vd["tgt"]), bf(np.ascontiguousarray(vd["drf"]))
        d = torch.from_numpy(vd["d_greedy" if parts[1] == "greedy" else "d_sample"]).to(dev)
        ua, ur = torch.from_numpy(vd["u_acc"]).to(dev), torch.from_numpy(vd["u_res"]).to(dev)
        ws = q.new_verify_workspace(Bc, gc, Vc, device=dev)
        n = torch.empty(Bc, dtype=torch.int32, device=dev)
        o = torch.empty(Bc, gc + 1, dtype=torch.int32, device=dev)
        fn = ((lambda: q.qspec_verify_greedy(tgt, d, n, o, ws)) if parts[1] == "greedy"
              else (lambda: q.qspec_verify_sample(tgt, drf, d, ua, ur, n, o, ws)))
        nbytes = verify_bytes(Bc, gc, Vc, parts[1] != "greedy")
    else:
        # a layer (one linear) or a group of the step (one grouped launch, e.g. qkv:a4:1), or a
        # Llama-2-70B layer of the linear sweep (70b_gate_up:a16:16)
        name, mode, M = parts[0], parts[1], int(parts[2])
        if name.startswith("70b_"):
            li = [l[0] for l in LLAMA70B].index(name[4:])
            _, N, K = LLAMA70B[li]
            W = bf(syn.weights(N, K, 3, layer=li))
            Wp = torch.empty(N, K // 2, dtype=torch.uint8, device=dev)
            S = torch.empty(N, K // 128, dtype=torch.float16, device=dev)
            q.qspec_pack_weights(W, Wp, S)
            del W
            x = bf(syn.activations(M, K, 3, step=M))
            y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            ws = q.new_linear_workspace(M, N, K, device=dev)
            f = {"a4": q.qspec_linear_w4a4, "a8": q.qspec_linear_w4a8, "a16": q.qspec_linear_w4a16}[mode]
            fn = lambda: f(x, Wp, S, y, ws)
            nbytes = linear_bytes(M, N, K)
        else:
            groups = dict(GROUPS)
            grouped = name in groups and M <= 4  # the grouped launch serves up to 4 tokens
            members = groups[name] if grouped else (name,)
            K = SHAPE[members[0]][1]
            lead = [l[0] for l in LAYERS].index(members[0])
            x = bf(syn.activations(M, K, 1, step=10 * lead))
            mats = []
            for m in members:
                li = [l[0] for l in LAYERS].index(m)
                N = SHAPE[m][0]
                W = bf(syn.weights(N, K, 1, layer=li))
                Wp = torch.empty(N, K // 2, dtype=torch.uint8, device=dev)
                S = torch.empty(N, K // 128, dtype=torch.float16, device=dev)
                q.qspec_pack_weights(W, Wp, S)
                del W
                mats.append((Wp, S, torch.empty(M, N, dtype=torch.bfloat16, device=dev)))
            abits = {"a4": 4, "a8": 8, "a16": 16}[mode]
            if grouped:
                ws = q.new_linear_group_workspace(M, [SHAPE[m][0] for m in members], K, device=dev)
                fn = q.LinearGroup(abits, x, mats, ws).run
                nbytes = group_bytes(M, members)
            else:
                Wp, S, y = mats[0]
                ws = q.new_linear_workspace(M, SHAPE[name][0], K, device=dev)
                f = {4: q.qspec_linear_w4a4, 8: q.qspec_linear_w4a8, 16: q.qspec_linear_w4a16}[abits]
                fn = lambda: f(x, Wp, S, y, ws)
                nbytes = linear_bytes(M, SHAPE[name][0], K)
    for _ in range(reps):
        fn()
    torch.cuda.synchronize()
    q.qspec_check_status()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) * 1e-3 / reps
    print(json.dumps({"case": spec, "us_per_launch": round(t * 1e6, 2), "GB_s": round(nbytes / t / 1e9, 1),
                      "note": "eager back-to-back launches; inputs resident"}))


def l2_bytes():
    import torch
    try:
        return int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    except Exception:
        return 129 * 2 ** 20


def copies_for(nbytes, cap=512):
    """Input copies whose total is at least 3x L2, so that a rotation through them reads HBM (at
    most `cap` copies: the tiniest cells, latency-bound anyway, then rotate through less; each sweep
    line reports the bytes its rotation covers)."""
    return max(1, min(cap, -(-3 * l2_bytes() // max(1, nbytes))))


def _rotating_time(calls, iters=5):
    """Seconds per call, from CUDA-graph replays of the given calls (one per input copy, rotated so
    that every call reads inputs no earlier call of the replay touched)."""
    import torch
    for c in calls:
        c()
    torch.cuda.synchronize()
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for c in calls:
            c()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e-3 / (len(calls) * iters)


LLAMA70B = [("qo", 8192, 8192), ("kv", 1024, 8192), ("gate_up", 28672, 8192), ("down", 8192, 28672),
            ("lm_head", 32000, 8192)]


def _graph_time(fn, reps=10, iters=5):
    """Seconds per call of fn, from CUDA-graph replays of `reps` back-to-back calls."""
    import torch
    fn()
    torch.cuda.synchronize()
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e-3 / (reps * iters)


def sweep_linear():
    """Llama-2-70B-shaped linears, M swept 1..256 in both modes (the HBM-bound to tensor-bound
    crossover): one JSON line per (layer, mode, M) with GB/s and TOPS."""
    import numpy as np
    import torch

    import __graft_entry__ as g
    g.build()
    from quantized_speculative_decoding_qspec_gb300 import qspec as q
    from quantized_speculative_decoding_qspec_gb300 import synthetic as syn
    dev = torch.device("cuda", 0)
    hbm, _ = peaks()
    for li, (name, N, K) in enumerate(LLAMA70B):
        W = torch.from_numpy(syn.weights(N, K, 3, layer=li).view(np.int16)).to(dev).view(torch.bfloat16)
        Wp = torch.empty(N, K // 2, dtype=torch.uint8, device=dev)
        S = torch.empty(N, K // 128, dtype=torch.float16, device=dev)
        q.qspec_pack_weights(W, Wp, S)
        del W
        # rotate through weight copies of at least 3x L2 (the smaller layers would stay in L2)
        R = copies_for(linear_bytes(1, N, K))
        sets = [(Wp, S)] + [(Wp.clone(), S.clone()) for _ in range(R - 1)]
        for M in (1, 2, 4, 8, 16, 32, 64, 128, 256):
            x = torch.from_numpy(syn.activations(M, K, 3, step=M).view(np.int16)).to(dev).view(torch.bfloat16)
            y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            wss = [q.new_linear_workspace(M, N, K, device=dev) for _ in range(R)]
            for mode in ("a16", "a4", "a8") if M in (1, 4, 16, 64) else ("a16", "a4"):
                f = {"a16": q.qspec_linear_w4a16, "a4": q.qspec_linear_w4a4, "a8": q.qspec_linear_w4a8}[mode]
                t = _rotating_time([(lambda i=i: f(x, sets[i][0], sets[i][1], y, wss[i])) for i in range(R)])
                b = linear_bytes(M, N, K)
                print(json.dumps({"sweep": "llama70b_linear", "layer": name, "N": N, "K": K, "M": M, "mode": mode,
                                  "us": round(t * 1e6, 2), "GB_s": round(b / t / 1e9, 1),
                                  "hbm_frac": round(b / t / 1e9 / hbm, 3), "weight_copies": R,
                                  "rotation_bytes": R * b, "l2_bytes": l2_bytes(),
                                  "TOPS": round(2 * M * N * K / t / 1e12, 2)}), flush=True)
            del wss
        q.qspec_check_status()
        del sets


def sweep_batched():
    """Batched verify (16 sequences x gamma = 3): W4A16 at M = 64 and W4A4 at M = 16 on the
    Llama-3-8B shapes, and greedy verify over [64, 128256] bf16 logits with per-sequence accept
    lengths.  Every cell rotates through input copies of at least 3x L2 (HBM, not L2, figures).
    One JSON line per item."""
    import numpy as np
    import torch

    import __graft_entry__ as g
    g.build()
    from quantized_speculative_decoding_qspec_gb300 import qspec as q
    from quantized_speculative_decoding_qspec_gb300 import synthetic as syn
    dev = torch.device("cuda", 0)
    hbm, _ = peaks()
    for li, (name, N, K) in enumerate(LAYERS):
        W = torch.from_numpy(syn.weights(N, K, 2, layer=li).view(np.int16)).to(dev).view(torch.bfloat16)
        Wp = torch.empty(N, K // 2, dtype=torch.uint8, device=dev)
        S = torch.empty(N, K // 128, dtype=torch.float16, device=dev)
        q.qspec_pack_weights(W, Wp, S)
        del W
        R = copies_for(linear_bytes(64, N, K))
        sets = [(Wp, S)] + [(Wp.clone(), S.clone()) for _ in range(R - 1)]
        for M, mode in ((64, "a16"), (16, "a4")):
            x = torch.from_numpy(syn.activations(M, K, 2, step=M).view(np.int16)).to(dev).view(torch.bfloat16)
            ys = [torch.empty(M, N, dtype=torch.bfloat16, device=dev) for _ in range(R)]
            ws = [q.new_linear_workspace(M, N, K, device=dev) for _ in range(R)]
            f = q.qspec_linear_w4a16 if mode == "a16" else q.qspec_linear_w4a4
            t = _rotating_time([(lambda i=i: f(x, sets[i][0], sets[i][1], ys[i], ws[i])) for i in range(R)])
            b = linear_bytes(M, N, K)
            print(json.dumps({"sweep": "batched_linear", "layer": name, "N": N, "K": K, "M": M, "mode": mode,
                              "us": round(t * 1e6, 2), "GB_s": round(b / t / 1e9, 1),
                              "hbm_frac": round(b / t / 1e9 / hbm, 3), "weight_copies": R,
                              "rotation_bytes": R * b, "l2_bytes": l2_bytes(),
                              "TOPS": round(2 * M * N * K / t / 1e12, 2)}), flush=True)
            del ys, ws
        q.qspec_check_status()
        del Wp, S, sets
    B, gamma = 16, GAMMA
    inp = syn.verify_inputs(B, gamma, VOCAB, 0.5, workload_id=2, sampling=False)
    gt = torch.from_numpy(np.ascontiguousarray(inp["tgt"]).view(np.int16)).to(dev).view(torch.bfloat16)
    gd = torch.from_numpy(inp["d"]).to(dev)
    b = verify_bytes(B, gamma, VOCAB, False)
    R = copies_for(b)
    gts = [gt] + [gt.clone() for _ in range(R - 1)]
    gws = [q.new_verify_workspace(B, gamma, VOCAB, device=dev) for _ in range(R)]
    gn = torch.empty(B, dtype=torch.int32, device=dev)
    go = torch.empty(B, gamma + 1, dtype=torch.int32, device=dev)
    t = _rotating_time([(lambda i=i: q.qspec_verify_greedy(gts[i], gd, gn, go, gws[i])) for i in range(R)])
    for w in gws:
        q.qspec_check_status(w)
    print(json.dumps({"sweep": "batched_greedy_verify", "B": B, "gamma": gamma, "V": VOCAB,
                      "us": round(t * 1e6, 2), "GB_s": round(b / t / 1e9, 1), "hbm_frac": round(b / t / 1e9 / hbm, 3),
                      "logits_copies": R, "rotation_bytes": R * b, "l2_bytes": l2_bytes(),
                      "accept_len": gn.cpu().tolist()}), flush=True)


def sweep_sampling(quick=False):
    """Sampling-verify sweep: gamma x batch x vocab x draft noise.  Per cell: time, logits GB/s,
    positions/s, mean emitted tokens per sequence and call, and E[T] = (1 - a^(g+1)) / (1 - a)
    at the measured mean acceptance probability a (the tutorial's constant-acceptance model)."""
    import numpy as np
    import torch

    import __graft_entry__ as g
    g.build()
    from quantized_speculative_decoding_qspec_gb300 import qspec as q
    from quantized_speculative_decoding_qspec_gb300 import synthetic as syn
    dev = torch.device("cuda", 0)
    hbm, _ = peaks()
    gammas, batches = ((1, 3, 5, 7), (1, 8, 32, 64)) if not quick else ((3,), (8,))
    vocabs, sigmas = ((32000, 128256, 152064), (0.25, 0.5, 1.0)) if not quick else ((32000,), (0.5,))

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    for gamma in gammas:
        for B in batches:
            for V in vocabs:
                # greedy verify on the same shapes (it does not depend on the draft noise)
                ginp = syn.verify_inputs(B, gamma, V, 0.5, workload_id=4, sampling=False)
                # every cell rotates through logits copies of at least 3x L2 (HBM, not L2, figures)
                bg = verify_bytes(B, gamma, V, False)
                R = copies_for(bg)
                gt = bf(ginp["tgt"])
                gts = [gt] + [gt.clone() for _ in range(R - 1)]
                gd = torch.from_numpy(ginp["d"]).to(dev)
                gws = [q.new_verify_workspace(B, gamma, V, device=dev) for _ in range(R)]
                gn = torch.empty(B, dtype=torch.int32, device=dev)
                go = torch.empty(B, gamma + 1, dtype=torch.int32, device=dev)
                tg = _rotating_time([(lambda i=i: q.qspec_verify_greedy(gts[i], gd, gn, go, gws[i]))
                                     for i in range(R)], iters=3)
                for w in gws:
                    q.qspec_check_status(w)
                print(json.dumps({"sweep": "greedy_verify", "gamma": gamma, "B": B, "V": V,
                                  "us": round(tg * 1e6, 2), "GB_s": round(bg / tg / 1e9, 1),
                                  "hbm_frac": round(bg / tg / 1e9 / hbm, 3), "logits_copies": R,
                                  "rotation_bytes": R * bg,
                                  "positions_per_s": round(B * (gamma + 1) / tg, 1),
                                  "tokens_per_call": round(float(gn.float().mean().item()) + 1, 3)}), flush=True)
                del gt, gts, gd, gws
                for sigma in sigmas:
                    inp = syn.verify_inputs(B, gamma, V, sigma, workload_id=4, sampling=True)
                    b = verify_bytes(B, gamma, V, True)
                    R = copies_for(B * (2 * gamma + 1) * V * 2)
                    tgt, drf = bf(inp["tgt"]), bf(inp["drf"])
                    sets = [(tgt, drf)] + [(tgt.clone(), drf.clone()) for _ in range(R - 1)]
                    d = torch.from_numpy(inp["d"]).to(dev)
                    ua, ur = torch.from_numpy(inp["u_acc"]).to(dev), torch.from_numpy(inp["u_res"]).to(dev)
                    wss = [q.new_verify_workspace(B, gamma, V, device=dev) for _ in range(R)]
                    n = torch.empty(B, dtype=torch.int32, device=dev)
                    o = torch.empty(B, gamma + 1, dtype=torch.int32, device=dev)
                    a = torch.empty(B, gamma, dtype=torch.float32, device=dev)
                    t = _rotating_time([(lambda i=i: q.qspec_verify_sample(sets[i][0], sets[i][1], d, ua, ur, n, o,
                                                                           wss[i], accept_prob=a))
                                        for i in range(R)], iters=3)
                    for w in wss:
                        q.qspec_check_status(w)
                    alpha = float(a.mean().item())
                    et = (gamma + 1.0) if alpha >= 1.0 else (1 - alpha ** (gamma + 1)) / (1 - alpha)
                    del sets, wss
                    print(json.dumps({"sweep": "sampling_verify", "gamma": gamma, "B": B, "V": V, "sigma": sigma,
                                      "us": round(t * 1e6, 2), "GB_s": round(b / t / 1e9, 1),
                                      "hbm_frac": round(b / t / 1e9 / hbm, 3), "logits_copies": R,
                                      "rotation_bytes": R * b,
                                      "positions_per_s": round(B * (gamma + 1) / t, 1),
                                      "tokens_per_call": round(float(n.float().mean().item()) + 1, 3),
                                      "mean_accept_prob": round(alpha, 4), "E_T_at_mean_alpha": round(et, 3)}),
                          flush=True)


def decode_report(args):
    """The decode loop on a one-block toy model with Llama-3-8B widths (D 4096, F 14336, V 128256):
    gamma W4A4 draft passes, one W4A16 pass over gamma + 1 positions, verify, and top-1 statistics of
    both modes; then target-only decoding for the speedup comparison.  One JSON line."""
    import torch
    import numpy as np
    from quantized_speculative_decoding_qspec_gb300 import decode
    from quantized_speculative_decoding_qspec_gb300 import qspec as q
    D, F, V = 4096, 14336, 128256
    t0 = time.perf_counter()
    model = decode.ToyModel(D, F, V, workload_id=21, device="cuda")
    t_init = time.perf_counter() - t0
    out = {"metric": "speculative decode loop on a toy model (tutorial measures)", "config": {
        "workload": f"toy decoder: embedding [{V},{D}] bf16, packed linears [{F},{D}], [{D},{F}], [{V},{D}]; "
                    f"B={args.decode_batch}, gamma={args.decode_gamma}, "
                    f"{'sampling' if args.decode_sampling else 'greedy'}",
        "weight_bytes_packed": model.weight_bytes(), "iterations": args.decode_iters}}
    sd = decode.SpecDecoder(model, args.decode_batch, args.decode_gamma, sampling=args.decode_sampling)
    first = np.arange(args.decode_batch, dtype=np.int32) * 1013 + 17
    sd.run(first, 4, workload_id=22)                       # warm-up (graph capture)
    spec = sd.run(first, args.decode_iters, workload_id=22)
    n_tok = int(np.mean([len(g) for g in spec["generated"]]))
    sd.run_target_only(first, 4, workload_id=22)
    base = sd.run_target_only(first, n_tok, workload_id=22)
    summ = decode.summarize(spec, base, args.decode_gamma)
    if not args.decode_sampling:
        m = min(len(g) for g in spec["generated"])
        same_m = sd.run_target_only(first, m, workload_id=22, padded=True)
        summ["output_equivalence_greedy"] = all(spec["generated"][b][:m] == same_m["generated"][b]
                                                for b in range(args.decode_batch))
    out.update({k: (round(v, 4) if isinstance(v, float) else v) for k, v in summ.items()})
    out["init_s"] = round(t_init, 1)
    q.qspec_check_status()
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--decode", action="store_true",
                    help="run the speculative decode loop on a toy model and print its measures")
    ap.add_argument("--decode-batch", type=int, default=1)
    ap.add_argument("--decode-gamma", type=int, default=3)
    ap.add_argument("--decode-iters", type=int, default=64)
    ap.add_argument("--decode-sampling", action="store_true")
    ap.add_argument("--sweep", choices=["linear", "batched", "sampling", "sampling-quick"], default=None,
                    help="measurement sweeps instead of the step benchmark")
    ap.add_argument("--profile-case", default=None,
                    help="run only one kernel of the step, e.g. lm_head:a4:1 or verify:greedy (for ncu)")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--timed-graphs", type=int, default=64,
                    help="instrumented step graphs replayed after the timed loop (roofline and per-layer timing)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-all-cores", action="store_true", help="skip the all-cores oracle timing")
    ap.add_argument("--eager", action="store_true",
                    help="issue the step's launches directly instead of replaying CUDA graphs (for ncu)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.profile_case:
        profile_case(args.profile_case, args.reps)
        return
    if args.decode:
        decode_report(args)
        return
    if args.sweep == "linear":
        sweep_linear()
        return
    if args.sweep == "batched":
        sweep_batched()
        return
    if args.sweep in ("sampling", "sampling-quick"):
        sweep_sampling(quick=args.sweep == "sampling-quick")
        return

    if args.impl == "reference":
        if rank != 0:
            return
        budget = 120.0  # whole reference run
        per_step = budget / (args.steps + args.warmup)
        nbytes, dt, frac = time_oracle(per_step)
        data = oracle_inputs(frac)
        for _ in range(args.warmup):
            oracle_sample_step(data, frac)
        t0 = time.perf_counter()
        total = 0
        for _ in range(args.steps):
            total += oracle_sample_step(data, frac)
        el = time.perf_counter() - t0
        v = total / el / 1e9
        sample = f"oracle on {frac:.6f} of every layer's output rows (all 8 layers, 3 W4A4 + 1 W4A16 passes) plus full greedy and sampling verify per step"
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64 (oracle)", "data": "synthetic (seeded)",
            "config": {"workload": WORKLOAD},
            "cpu_baseline": {"value": round(v, 6), "unit": "GB/s", "cores": threads_used(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }))
        return

    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group(backend="nccl")
    result = gpu_arm(args, rank, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nbytes, dt, frac = time_oracle(args.cpu_budget)
        result["cpu_baseline"] = {
            "value": round(nbytes / dt / 1e9, 6), "unit": "GB/s", "cores": threads_used(), "kind": "oracle",
            "sample": f"one oracle pass over {frac:.5f} of every layer's output rows (3 W4A4 + 1 W4A16 passes) "
                      f"plus full greedy and sampling verify; {dt:.1f} s; GB/s of the same algorithmic bytes"}
        if not args.no_all_cores:
            procs = os.cpu_count() or 1
            nb_all, dt_all = time_oracle_all_cores(frac, procs)
            result["cpu_baseline"]["all_cores"] = {
                "value": round(nb_all / dt_all / 1e9, 6), "unit": "GB/s", "cores": procs,
                "sample": f"{procs} single-threaded oracle processes, each the same sample as above at once; "
                          f"{dt_all:.1f} s wall"}
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


if __name__ == "__main__":
    # the oracle baseline is timed single-threaded: pin BLAS pools before numpy loads
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ.setdefault(_v, "1")
    main()
