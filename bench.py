"""Benchmark of the GB300 LoongTrain 2D-Attention ring step.

One step = one pass of the 2D-attention hot path over one batch of synthetic
input (default ``--layout rank-major``): the Ulysses head-context repack of Q,
K, V and dO from the natural layout into every emulated rank's (S/cp, H/hp)
layout, the fused ring-attention forward (online softmax merged over the
double-ring schedule) and backward (row statistics, dQ/dK/dV) reading and
writing that layout, and the repack of O, dQ, dK, dV back.  ``--layout
natural`` runs the ring kernels on the natural layout with no repack.
Metric: algorithmic causal TFLOP/s of forward + backward, 7 * B * S^2 * Hq * d
per step (forward 2 GEMMs over the causal half, backward 2.5x the forward).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--layout rank-major|natural] [--mode fused|stepwise]
                    [--impl reference] [--no-e2e] [--no-cpu-baseline]

Under torchrun each rank runs the whole workload on its own GPU as an
independent replica (weak scaling); value = all ranks' FLOPs / max rank time.
``--impl reference`` times the float64 CPU oracle on the host cores on a
bounded sample of the same workload (rank 0 only).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "llama3-8b-s128k"
METRIC = "causal ring-attention fwd+bwd TFLOP/s and % of GB300 BF16 dense peak"
SLOWDOWN_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--mode", default="fused", choices=["fused", "stepwise", "stepwise-copy", "stepwise-copy-ab"],
                   help="stepwise-copy: one launch per ring step, K/V delivered by device-to-device copies "
                        "on a side stream (rank-major layout); -ab: blocks A and B on two streams (two rings)")
    p.add_argument("--layout", default="rank-major", choices=["rank-major", "natural"],
                   help="rank-major: the step repacks in and out around the ring kernels (2D attention)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--e2e-overlap", action=argparse.BooleanOptionalAction, default=True,
                   help="end-to-end leg: copies overlapped with the kernels (default) or each call synchronised")
    p.add_argument("--per-rank", action=argparse.BooleanOptionalAction, default=True,
                   help="after the timed steps, time each emulated ring rank's forward on its own")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--seqlen", type=int, default=0,
                   help="override S (a smaller case of the same shape, e.g. for profiler captures)")
    p.add_argument("--fwd-only", action="store_true", help="time the forward pass alone")
    p.add_argument("--non-causal", action="store_true",
                   help="every query sees every key (FLOPs counted over all S^2 pairs)")
    p.add_argument("--configs", action=argparse.BooleanOptionalAction, default=None,
                   help="after the headline workload, time the other full-size configurations "
                        "(1 warm-up + 2 steps each); default: on for the default workload at N=1")
    return p.parse_args(argv)


# The other configurations timed after the headline one (--configs), and the
# GB300 dense bf16 tensor-core rate from NVIDIA's datasheet (no sparsity),
# reported beside the measured peaks.
OTHER_CONFIGS = ("llama3-8b-s32k-fwd", "llama3-70b-s256k", "headgroup-s1m-peaky")
DATASHEET_BF16_TFLOPS = 2250.0


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d["bf16_tflops_sustained"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ------------------------------------------------------------------ ncu traffic
KERNEL_SOURCES = ("attn_fwd.cu", "attn_bwd.cu", "ptx.cuh", "ring.cuh")


def kernel_source_hash():
    """SHA-256 of the kernel sources' code: `//` comments, trailing blanks and
    empty lines are dropped, so a comment-only edit keeps the recorded counters."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "head_context_attention_gb300", "csrc", f)) as fh:
            for line in fh:
                code = re.sub(r"//.*$", "", line).rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()


def recorded_traffic(kernel, workload, layout="rank-major"):
    """DRAM bytes per launch of `kernel` on `workload` in `layout` from the
    committed ncu record, or None when absent or taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != kernel_source_hash():
        return None
    ent = rec.get("kernels", {}).get(kernel, {}).get(workload, {}).get(layout)
    return None if ent is None else int(ent["dram_bytes_per_launch"])


# ------------------------------------------------------------------ merge
def time_lse_merge(w, o, lse, stream, dev, reps=5):
    """The n-way log-sum-exp merge on its own (outside the timed step, which
    merges inside the attention kernels): n = 2 fp32 partials of every
    (token, q-head) row of the workload, fp32 output; inputs exceed L2."""
    import torch

    from head_context_attention_gb300 import ops
    rows = w.batch * w.seqlen * w.hq
    o_parts = torch.empty((2, rows, w.head_dim), dtype=torch.float32, device=dev)
    o_parts[0].copy_(o.reshape(rows, w.head_dim))
    o_parts[1].copy_(o.reshape(rows, w.head_dim).flip(0))
    lse_parts = torch.stack([lse.reshape(rows), lse.reshape(rows).flip(0) - 1.0])
    o_out = torch.empty((rows, w.head_dim), dtype=torch.float32, device=dev)
    lse_out = torch.empty(rows, dtype=torch.float32, device=dev)
    for _ in range(2):
        ops.loong_lse_merge(o_parts, lse_parts, o_out, lse_out, stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        a.record(stream)
        ops.loong_lse_merge(o_parts, lse_parts, o_out, lse_out, stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    nbytes = rows * (2 * (4 * w.head_dim + 4) + 4 * w.head_dim + 4)
    del o_parts, lse_parts, o_out, lse_out
    return {"ms": round(ms, 3), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "bytes": nbytes, "parts": 2,
            "rows": rows}


# ------------------------------------------------------------------ exchange copies
def time_exchange_alone(w, path, stream, dev, reps=3):
    """The device-to-device copies of one STEPWISE_COPY pass on their own: for
    ring steps 1..cp-1, every rank's incoming K and V chunk into a receive
    buffer, the same transfers the library issues on its side stream."""
    import torch

    from head_context_attention_gb300 import ops

    sched = ops.loong_ring_schedule(w.ring_inner, w.ring_outer)
    k, v = path.kt["k"], path.kt["v"]
    rk, rv = torch.empty_like(k), torch.empty_like(v)

    def copies():
        for t in range(1, w.cp):
            for b in range(w.batch):
                for c in range(w.cp):
                    j = sched[t][c]
                    rk[b * w.cp + c].copy_(k[b * w.cp + j], non_blocking=True)
                    rv[b * w.cp + c].copy_(v[b * w.cp + j], non_blocking=True)

    copies()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        a.record(stream)
        copies()
        b.record(stream)
    torch.cuda.synchronize(dev)
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    nbytes = (w.cp - 1) * 2 * k.numel() * k.element_size()
    return {"bytes_per_pass": nbytes, "copy_ms_alone": round(ms, 3), "gbs": round(2 * nbytes / (ms * 1e-3) / 1e9, 1),
            "note": "copies of one pass timed alone; in the step they run on a side stream beside the kernels"}


# ------------------------------------------------------------------ per-rank work
def rank_pairs(w, placement, c):
    """Causal (query, key) pairs of ring rank c's query rows, per head: the
    work the rank's share of the ring pass holds (query i sees keys 0..i)."""
    nb = 2 * w.cp if placement == 1 else w.cp
    L = w.seqlen // nb
    blocks = (c, 2 * w.cp - 1 - c) if placement == 1 else (c,)
    # rows of block j are j*L .. j*L + L - 1; row i sees i + 1 keys
    return sum(L * (j * L) + L * (L + 1) // 2 for j in blocks)


def time_per_rank(w, x, stream, dev, reps=3):
    """Forward time of every emulated ring rank's query rows on its own
    (loong_attn_fwd_ranks), FUSED, natural layout, for the paired-block and the
    contiguous placement of the same workload, beside each rank's share of the
    causal work."""
    import torch

    from head_context_attention_gb300 import ops

    res = {}
    o = torch.empty_like(x["q"])
    lse = torch.empty((w.batch, w.hq, w.seqlen), dtype=torch.float32, device=dev)
    for name, pl in (("zigzag", ops.PLACEMENT_ZIGZAG), ("contiguous", ops.PLACEMENT_CONTIGUOUS)):
        wp = w.with_(placement=pl)
        desc = ops.make_desc(wp, ops.MODE_FUSED)
        if ops.loong_attn_check(desc) != ops.LOONG_OK:
            continue
        ws = ops.workspace(desc, 0, dev)
        ms = []
        for c in range(w.cp):
            ops.loong_attn_fwd_ranks(desc, c, c + 1, x["q"], x["k"], x["v"], o, lse, ws, stream)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            for a, b in ev:
                a.record(stream)
                ops.loong_attn_fwd_ranks(desc, c, c + 1, x["q"], x["k"], x["v"], o, lse, ws, stream)
                b.record(stream)
            torch.cuda.synchronize(dev)
            ms.append(statistics.median(a.elapsed_time(b) for a, b in ev))
        work = [rank_pairs(w, pl, c) for c in range(w.cp)]
        tot_ms, tot_w = sum(ms), sum(work)
        res[name] = {"ms": [round(m, 3) for m in ms],
                     "time_share": [round(m / tot_ms, 4) for m in ms],
                     "work_share": [round(u / tot_w, 4) for u in work],
                     "max_over_mean_time": round(max(ms) * len(ms) / tot_ms, 3),
                     "max_over_mean_work": round(max(work) * len(work) / tot_w, 3)}
    return res


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ distributed
def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        pg = dist
    if n_gpus != world and world > 1:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE {world}")
    return rank, local, world, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, value, device):
    """Max of a float over ranks (identity for one rank)."""
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ oracle timing
def oracle_inputs(w, x=None):
    """Head 0 (and its kv head 0) of the workload's seeded inputs as float64
    numpy arrays [S, 1, d]; drawn on the GPU when one is present."""
    import torch

    from head_context_attention_gb300 import inputs

    if x is None:
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        x = inputs.make_inputs(w, device=dev, with_do=True)
    return {n: t[0, :, :1].to("cpu", torch.float64).numpy() for n, t in x.items()}


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_sample(w, seconds, arrays):
    """Time the float64 oracle on a bounded sample of workload ``w``.

    Sample: query rows of head 0 spread over the sequence; for each row the
    oracle's forward (softmax over keys 0..i) and backward (dQ row) at the
    workload's full S.  FLOPs per row i follow the metric's accounting,
    3.5 * 4 * (i + 1) * d.  Rows are added until ``seconds`` have elapsed.
    """
    import numpy as np

    from oracle import attention

    q, k, v, do = arrays["q"], arrays["k"], arrays["v"], arrays["do"]
    rng = np.random.default_rng(0)
    rows_done, flops, t0 = 0, 0.0, time.perf_counter()
    chunk = 8
    while time.perf_counter() - t0 < seconds:
        rows = np.sort(rng.integers(0, w.seqlen, size=chunk))
        attention.attention_rows(q, k, v, rows, [0])
        attention.attention_backward_rows(q, k, v, do, rows, [0])
        flops += float(np.sum(3.5 * 4.0 * (rows + 1) * w.head_dim))
        rows_done += chunk
    el = time.perf_counter() - t0
    rate = flops / el
    return {"value": rate / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "extrapolated_full_step_s": round(w.flops / rate, 1),
            "sample": f"{rows_done} query rows of head 0 at S={w.seqlen} (forward row + dQ row, float64), "
                      f"{el:.1f} s"}


# ------------------------------------------------------------------ other configurations
def time_config(w, dev, stream, peaks, steps=2, warmup=1):
    """One configuration at full size, the headline's step (rank-major repack in,
    FUSED ring forward (+ backward), repack out): step and kernel rates.  A
    workload with the Q/K/V repack in its definition also gets that repack
    timed alone (one launch, Q, K, V) against 75 % of the measured HBM rate."""
    import torch

    from head_context_attention_gb300 import inputs, ops

    path = TwoDPath(w, ops.MODE_FUSED, "rank-major", dev, stream)
    x = inputs.make_inputs(w, device=dev, with_do=w.backward)

    def step():
        path.pack_in(x)
        path.fwd(x)
        path.bwd(x)
        path.unpack_out()

    for _ in range(warmup):
        step()
    mk = lambda: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(steps)]
    ev_f, ev_b, ev_p, ev_u = mk(), mk(), mk(), mk()
    for a, b in ev_f + ev_b:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        ev_p[i][0].record(stream)
        path.pack_in(x)
        ev_p[i][1].record(stream)
        ops.loong_set_timing_events(*ev_f[i])
        path.fwd(x)
        if w.backward:
            ops.loong_set_timing_events(*ev_b[i])
            path.bwd(x)
        ops.loong_set_timing_events(None, None)
        ev_u[i][0].record(stream)
        path.unpack_out()
        ev_u[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if ops.loong_get_device_status(stream) != ops.LOONG_OK:
        raise SystemExit(f"device status after {w.name}")
    ms = t0.elapsed_time(t1) / steps
    peak = peaks["bf16_tflops_sustained"]
    f_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_f)
    rec = {"seqlen": w.seqlen, "hq": w.hq, "hkv": w.hkv, "hp": w.hp, "cp": w.cp,
           "ring": f"{w.ring_inner}x{w.ring_outer}", "pass": "fwd+bwd" if w.backward else "fwd",
           "peaky_keys": w.peaky_keys, "steps": steps, "warmup": warmup, "ms_per_step": round(ms, 3),
           "tflops": round(w.flops / (ms * 1e-3) / 1e12, 2)}
    fwd_tf = w.fwd_flops / (f_ms * 1e-3) / 1e12
    rec["ring_fwd_kernel"] = {"ms": round(f_ms, 3), "tflops": round(fwd_tf, 2), "frac_of_peak": round(fwd_tf / peak, 4)}
    if w.backward:
        b_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_b)
        bwd_tf = 2.5 * w.fwd_flops / (b_ms * 1e-3) / 1e12
        rec["ring_bwd_kernel"] = {"ms": round(b_ms, 3), "tflops": round(bwd_tf, 2),
                                  "frac_of_peak": round(bwd_tf / peak, 4)}
    in_bytes, out_bytes = path.repack_bytes()
    for key, evs, nbytes in (("headctx_pack_in", ev_p, in_bytes), ("headctx_pack_out", ev_u, out_bytes)):
        p_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        gbs = nbytes / (p_ms * 1e-3) / 1e9
        rec[key] = {"ms": round(p_ms, 3), "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
                    "bytes": nbytes}
    if w.repack:
        names = TwoDPath.FWD_IN
        nbytes = sum(2 * x[n].numel() * x[n].element_size() for n in names)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(5)]
        for a, b in ev:
            a.record(stream)
            path._pack([x[n] for n in names], [path.kt[n] for n in names], names, 0)
            b.record(stream)
        torch.cuda.synchronize(dev)
        q_ms = statistics.median(a.elapsed_time(b) for a, b in ev)
        gbs = nbytes / (q_ms * 1e-3) / 1e9
        rec["qkv_repack"] = {"ms": round(q_ms, 3), "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
                             "bytes": nbytes, "target_ms_at_75pct_hbm": round(nbytes / (0.75 * peaks["hbm_gbs"] * 1e9) * 1e3, 3)}
    del path, x
    torch.cuda.empty_cache()
    return rec


def run_other_configs(names, dev, stream, peaks, local):
    """Every configuration in `names`, one after the other, under one clock sampler."""
    from head_context_attention_gb300 import inputs

    out = {}
    with ClockSampler(local) as clk:
        for n in names:
            out[n] = time_config(inputs.WORKLOADS[n], dev, stream, peaks)
    out["clocks"] = clk.summary()
    return out


# ------------------------------------------------------------------ GPU arm
class TwoDPath:
    """One fwd+bwd pass of 2D attention through the library's C entry points.

    rank-major: Q, K, V, dO arrive in the natural [B, S, H, d] layout; the
    Ulysses repack (loong_headctx_pack, paired- or contiguous-block gather)
    moves them into the per-rank layout [B*cp, hp, S/cp, H/hp, d]; the ring
    forward and backward read and write that layout (LAYOUT_RANK_MAJOR); O, dQ,
    dK, dV are packed back to the natural layout.  natural: the ring kernels on
    the natural layout directly, no repack."""

    def __init__(self, w, mode, layout, dev, stream):
        import torch

        from head_context_attention_gb300 import ops

        self.ops, self.w, self.stream = ops, w, stream
        self.rank_major = layout == "rank-major"
        self.desc = ops.make_desc(w, mode, layout=ops.LAYOUT_RANK_MAJOR if self.rank_major else ops.LAYOUT_NATURAL)
        st = ops.loong_attn_check(self.desc)
        if st != ops.LOONG_OK:
            raise SystemExit(f"workload {w.name} rejected: {st}")
        self.ws0, self.ws1 = ops.workspace(self.desc, 0, dev), ops.workspace(self.desc, 1, dev)
        self.gather = 1 if w.placement == ops.PLACEMENT_ZIGZAG else 2
        self.s_local = w.seqlen // (w.cp * w.hp)
        B, S, d = w.batch, w.seqlen, w.head_dim
        bf = dict(dtype=torch.bfloat16, device=dev)
        nat = {"q": w.hq, "o": w.hq, "do": w.hq, "dq": w.hq, "k": w.hkv, "v": w.hkv, "dk": w.hkv, "dv": w.hkv}
        self.heads = nat
        # natural-layout outputs, and the tensors the ring kernels use
        self.out = {n: torch.empty((B, S, nat[n], d), **bf) for n in ("o", "dq", "dk", "dv")}
        self.lse = torch.empty((B, w.hq, S), dtype=torch.float32, device=dev)
        if self.rank_major:
            self.kt = {n: torch.empty((B * w.cp, w.hp, S // w.cp, h // w.hp, d), **bf) for n, h in nat.items()}
        self.do_bwd = w.backward
        # the forward's rounding residual of O, kept on the device for the
        # backward's D (in the layout the ring kernels use)
        self.o_res = (torch.empty_like(self.kt["o"] if self.rank_major else self.out["o"])
                      if self.do_bwd else None)

    def launches(self):
        """Kernels of one step: forward = max |V| + V to fp16 + ring kernel(s)
        (+ LSE fill and O conversion, STEPWISE); backward = row statistics +
        ring kernel(s) + dQ conversion (+ dK, dV conversions, STEPWISE)."""
        ops, w = self.ops, self.w
        fused = self.desc.mode == ops.MODE_FUSED
        n = (3 if fused else w.cp + 4) + (((3 if fused else w.cp + 4)) if self.do_bwd else 0)
        if self.rank_major:
            n += 2   # one repack launch in, one out
        return n

    FWD_IN, BWD_IN, FWD_OUT, BWD_OUT = ("q", "k", "v"), ("do",), ("o",), ("dq", "dk", "dv")

    def pack_in(self, x, names=None):
        """Repack the named inputs (default: every input of the pass) into the per-rank layout."""
        if not self.rank_major:
            return
        if names is None:
            names = self.FWD_IN + (self.BWD_IN if self.do_bwd else ())
        self._pack([x[n] for n in names], [self.kt[n] for n in names], names, 0)

    def _pack(self, srcs, dsts, names, direction):
        """One launch repacks every named tensor (the pass's one all-to-all per direction)."""
        w = self.w
        self.ops.loong_headctx_pack_n(srcs, dsts, w.batch, w.cp, w.hp, self.s_local, [self.heads[n] for n in names],
                                      w.head_dim, direction, self.gather, self.stream)

    def fwd(self, x):
        t = self.kt if self.rank_major else x
        o = self.kt["o"] if self.rank_major else self.out["o"]
        self.ops.loong_attn_fwd(self.desc, t["q"], t["k"], t["v"], o, self.lse, self.o_res, self.ws0, self.stream)

    def bwd(self, x):
        if not self.do_bwd:
            return
        t = self.kt if self.rank_major else x
        g = self.kt if self.rank_major else self.out
        o = self.kt["o"] if self.rank_major else self.out["o"]
        self.ops.loong_attn_bwd(self.desc, t["q"], t["k"], t["v"], o, self.o_res, self.lse, t["do"], g["dq"],
                                g["dk"], g["dv"], self.ws1, self.stream)

    def unpack_out(self, names=None):
        """Repack the named outputs (default: every output of the pass) back to the natural layout."""
        if not self.rank_major:
            return
        if names is None:
            names = self.FWD_OUT + (self.BWD_OUT if self.do_bwd else ())
        self._pack([self.kt[n] for n in names], [self.out[n] for n in names], names, 1)

    def repack_bytes(self):
        """Algorithmic bytes of the repacks of one step (read + write), in and out."""
        w = self.w
        if not self.rank_major:
            return 0, 0
        row = 2 * w.batch * w.seqlen * w.head_dim * 2
        h_in = 2 * w.hq + 2 * w.hkv if self.do_bwd else w.hq + 2 * w.hkv
        h_out = 2 * w.hq + 2 * w.hkv if self.do_bwd else w.hq
        return row * h_in, row * h_out


def run_gpu(args, w, rank, local, world, pg):
    import torch

    from head_context_attention_gb300 import inputs, ops

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    mode = {"fused": ops.MODE_FUSED, "stepwise": ops.MODE_STEPWISE, "stepwise-copy": ops.MODE_STEPWISE_COPY,
            "stepwise-copy-ab": ops.MODE_STEPWISE_COPY_AB}[args.mode]
    stream = torch.cuda.current_stream(dev)
    path = TwoDPath(w, mode, args.layout, dev, stream)
    x = inputs.make_inputs(w, device=dev, with_do=True)
    do_bwd = w.backward
    # pinned host buffers of the end-to-end leg, taken before any timed work
    e2e_bufs = None if args.no_e2e else pinned_buffers(w, path, x)

    def step():
        path.pack_in(x)
        path.fwd(x)
        path.bwd(x)
        path.unpack_out()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = ops.loong_get_device_status(stream)
    if st != ops.LOONG_OK:
        raise SystemExit(f"device status {st} after warm-up")
    # The end-to-end leg runs before the clock-sampled region: host copies made
    # after an nvidia-smi sampling loop has run measured 6-8x slower.
    e2e = None if args.no_e2e else run_e2e(args, w, path, dev, stream, world, pg, x, e2e_bufs)
    if e2e is not None:
        e2e["check"] = e2e_outputs_match(path, e2e_bufs[1], step, dev)

    # Timed region: K steps; per-kernel events for the forward and backward kernels.
    mk = lambda: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
    ev_f, ev_b, ev_p, ev_u = mk(), mk(), mk(), mk()
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # torch creates events lazily and tracks recording itself: record each once
    # here so the handle exists (the library re-records it around its kernels).
    for a, b in ev_f + ev_b:
        a.record(stream)
        b.record(stream)
    barrier(pg)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_start.record(stream)
        for i in range(args.steps):
            ev_p[i][0].record(stream)
            path.pack_in(x)
            ev_p[i][1].record(stream)
            ops.loong_set_timing_events(*ev_f[i])
            path.fwd(x)
            if do_bwd:
                ops.loong_set_timing_events(*ev_b[i])
                path.bwd(x)
            ops.loong_set_timing_events(None, None)
            ev_u[i][0].record(stream)
            path.unpack_out()
            ev_u[i][1].record(stream)
        t_stop.record(stream)
        torch.cuda.synchronize(dev)
    barrier(pg)
    st = ops.loong_get_device_status(stream)
    if st != ops.LOONG_OK:
        raise SystemExit(f"device status {st} in the timed region")
    ms_total = t_start.elapsed_time(t_stop)
    ms_total = max_over_ranks(pg, ms_total, dev)
    merge_rec = time_lse_merge(w, path.out["o"], path.lse, stream, dev)
    per_rank = time_per_rank(w, x, stream, dev) if args.per_rank else None
    exchange = time_exchange_alone(w, path, stream, dev) if mode in (ops.MODE_STEPWISE_COPY,
                                                                      ops.MODE_STEPWISE_COPY_AB) else None
    ms_step = ms_total / args.steps
    f_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_f)
    b_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_b) if do_bwd else 0.0
    p_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_p)
    u_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_u)
    peaks = measured_peaks()
    flops_step = w.flops
    tflops = flops_step * world / (ms_step * 1e-3) / 1e12

    bwd_flops = w.fwd_flops * 2.5
    bwd_tf = bwd_flops / (b_ms * 1e-3) / 1e12 if do_bwd else 0.0
    fwd_tf = w.fwd_flops / (f_ms * 1e-3) / 1e12
    in_bytes, out_bytes = path.repack_bytes()
    dominant = "bwd" if b_ms >= f_ms else "fwd"
    dom_tf = bwd_tf if dominant == "bwd" else fwd_tf
    peak = peaks["bf16_tflops_sustained"]
    clocks = clk.summary()

    kernels = {
        "ring_fwd_kernel": {"ms": round(f_ms, 3), "tflops": round(fwd_tf, 2), "frac_of_peak": round(fwd_tf / peak, 4)},
        "ring_bwd_kernel": {"ms": round(b_ms, 3), "tflops": round(bwd_tf, 2), "frac_of_peak": round(bwd_tf / peak, 4)},
    }
    if path.rank_major:
        for key, ms, nbytes, what in (("headctx_pack_in", p_ms, in_bytes, "Q, K, V, dO natural -> rank-major"),
                                      ("headctx_pack_out", u_ms, out_bytes, "O, dQ, dK, dV rank-major -> natural")):
            gbs = nbytes / (ms * 1e-3) / 1e9
            kernels[key] = {"ms": round(ms, 3), "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
                            "bytes": nbytes, "tensors": what}
    kernels["lse_merge"] = dict(merge_rec, frac_of_hbm=round(merge_rec["gbs"] / peaks["hbm_gbs"], 4))
    result = {
        "metric": METRIC, "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, Llama-3-shaped attention layer)",
        "config": {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "hq": w.hq, "hkv": w.hkv,
                   "head_dim": w.head_dim, "hp": w.hp, "cp": w.cp, "ring_inner": w.ring_inner,
                   "ring_outer": w.ring_outer, "placement": "zigzag" if w.placement == 1 else "contiguous",
                   "mode": args.mode, "layout": args.layout, "causal": w.causal,
                   "step": ("repack Q,K,V,dO -> ring fwd + bwd on the rank-major layout -> repack O,dQ,dK,dV"
                            if path.rank_major else "ring fwd + bwd on the natural layout"),
                   "parallelism": f"replicas x{world} (each rank: all hp x cp ranks emulated)",
                   "l2": f"inputs exceed L2 (Q {w.batch * w.seqlen * w.hq * w.head_dim * 2 / 2**20:.0f} MiB vs 126 MiB "
                         "of L2); no flush",
                   "flops_per_step": flops_step},
        "pct_of_peak": round(100.0 * tflops / world / peak, 2),
        "pct_of_datasheet_peak": round(100.0 * tflops / world / DATASHEET_BF16_TFLOPS, 2),
        "roofline": {"bound": "tensor", "kernel": f"ring_{dominant}_kernel", "achieved": round(dom_tf, 2),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(dom_tf / peak, 4),
                     "peak_kind": f"bf16 sustained, of {peaks['source']}",
                     "frac_of_burst": round(dom_tf / peaks["bf16_tflops"], 4),
                     "frac_of_datasheet": round(dom_tf / DATASHEET_BF16_TFLOPS, 4),
                     # the record holds FUSED launches (one launch per pass)
                     "traffic": (recorded_traffic(f"ring_{dominant}_kernel", w.name, args.layout)
                                 if mode == ops.MODE_FUSED and w.causal else None),
                     "traffic_unit": "DRAM bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)"},
        "kernels": kernels,
        "clocks": clocks,
        "gpu_launches": path.launches() * args.steps,
    }
    if per_rank is not None:
        result["per_rank_fwd"] = per_rank
    if exchange is not None:
        result["exchange"] = exchange
    rejected = [r for r in clocks.get("reasons", []) if r in SLOWDOWN_REASONS]
    if rejected:
        result["clocks"]["rejected"] = rejected

    if not do_bwd:
        del result["kernels"]["ring_bwd_kernel"]
        result["config"]["pass"] = "forward only"
    if e2e is not None:
        result["e2e"] = e2e
    return result, x


def pinned_buffers(w, path, x):
    """Pinned host copies of the inputs and pinned host buffers for the outputs,
    from the library's host allocator (loong_host_alloc: registered memory on
    transparent huge pages, which keeps the copies at full speed when the
    device's translations of host pages have gone cold)."""
    from head_context_attention_gb300 import ops

    names = path.FWD_IN + (path.BWD_IN if w.backward else ())
    host_in = {n: ops.host_empty(x[n].shape, x[n].dtype) for n in names}
    for n in names:
        host_in[n].copy_(x[n])
    outs = dict(path.out, lse=path.lse)
    if not w.backward:
        outs = {"o": path.out["o"], "lse": path.lse}
    host_out = {n: ops.host_empty(t.shape, t.dtype) for n, t in outs.items()}
    return host_in, host_out


def huge_page_share(tensors):
    """Share of the bytes of the mappings that hold `tensors` (host buffers from
    loong_host_alloc, one mapping each) backed by transparent huge pages, from
    /proc/self/smaps; None where that file cannot be read."""
    try:
        lines = open("/proc/self/smaps").read().splitlines()
    except OSError:
        return None
    vmas, cur = {}, None
    for line in lines:
        head = line.split(" ", 1)[0]
        if "-" in head and ":" not in head:
            lo, hi = head.split("-")
            cur = int(lo, 16)
            vmas[cur] = [int(hi, 16) - cur, 0]
        elif line.startswith("AnonHugePages:") and cur is not None:
            vmas[cur][1] = int(line.split()[1]) * 1024
    size = huge = 0
    for t in tensors:
        s, h = vmas.get(t.data_ptr(), (0, 0))
        size, huge = size + s, huge + h
    return round(huge / size, 4) if size else None


def e2e_outputs_match(path, host_out, step, dev):
    """The last end-to-end step's results, read back to the host, against a
    device-only pass over the same inputs: O, LSE, dK, dV bit for bit (their
    kernels are deterministic), dQ (summed by unordered reductions) within
    2^-7 of its largest magnitude.  A copy that raced its kernels fails."""
    import torch

    step()
    torch.cuda.synchronize(dev)
    ok = True
    for n, h in host_out.items():
        d = (path.lse if n == "lse" else path.out[n]).cpu()
        if n == "dq":
            ok &= bool((h.float() - d.float()).abs().max() <= 2.0 ** -7 * d.float().abs().max())
        else:
            ok &= torch.equal(h, d)
    return ok


def run_e2e(args, w, path, dev, stream, world, pg, x, bufs):
    """Same metric through the C ABI with host buffers: each step is one
    loong_attn_2d_host call, natural-layout Q, K, V, dO in pinned host memory
    to O, LSE, dQ, dK, dV in pinned host memory.  The library's two copy
    streams carry the copies; consecutive calls alternate the two device input
    slots, so a step's inputs arrive and the previous step's results leave
    while the kernels run.  Every copy of every step lies inside the timed
    region, which ends when the last step's results are in host memory.
    ``--no-e2e-overlap`` synchronises after every call instead (copies and
    kernels in series)."""
    import torch

    from head_context_attention_gb300 import ops

    host_in, host_out = bufs
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    overlap = args.e2e_overlap
    desc = path.desc
    ws = torch.empty(ops.loong_attn_2d_host_workspace_size(desc, 1 if w.backward else 0), dtype=torch.uint8,
                     device=dev)
    grads = (host_out["dq"], host_out["dk"], host_out["dv"]) if w.backward else (None, None, None)

    def call(slot, done):
        ops.loong_attn_2d_host(desc, slot, host_in["q"], host_in["k"], host_in["v"], host_in.get("do"),
                               host_out["o"], host_out["lse"], *grads, ws, stream, done)

    def run(nsteps):
        dones = [torch.cuda.Event() for _ in range(nsteps)]
        for e in dones:
            e.record(stream)   # torch creates the event on its first record; the library records it again
        torch.cuda.synchronize(dev)
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(nsteps):
            call(i % 2, dones[i] if overlap else None)
            if not overlap:
                stream.synchronize()
        if overlap:
            stream.wait_event(dones[-1])
        stop.record(stream)
        torch.cuda.synchronize(dev)
        return start.elapsed_time(stop)

    # the copy speed of the moment: one plain H2D of the inputs and one D2H of the outputs
    a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    dev_in = {n: torch.empty_like(t, device=dev) for n, t in host_in.items()}
    dev_out = {n: torch.empty_like(t, device=dev) for n, t in host_out.items()}
    a.record(stream)
    for n in dev_in:
        dev_in[n].copy_(host_in[n], non_blocking=True)
    b.record(stream)
    for n in dev_out:
        host_out[n].copy_(dev_out[n], non_blocking=True)
    c.record(stream)
    torch.cuda.synchronize(dev)
    copy_ms = {"h2d": round(a.elapsed_time(b), 3), "d2h": round(b.elapsed_time(c), 3)}
    del dev_in, dev_out

    run(max(1, args.warmup))
    barrier(pg)
    ms = max_over_ranks(pg, run(args.steps), dev) / args.steps
    if ops.loong_get_device_status(stream) != ops.LOONG_OK:
        raise SystemExit("device status after the end-to-end leg")
    return {"value": round(w.flops * world / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 3), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "api": "loong_attn_2d_host (C ABI, host buffers from loong_host_alloc)",
            "copies": ("library copy streams overlapped with the kernels, two input slots" if overlap
                       else "in series: each call synchronised before the next"),
            "copy_alone_ms": copy_ms,
            "host_huge_page_share": {"in": huge_page_share(host_in.values()),
                                     "out": huge_page_share(host_out.values())}}


def main(argv=None):
    args = parse_args(argv)
    from head_context_attention_gb300 import inputs

    if args.workload not in inputs.WORKLOADS:
        raise SystemExit(f"unknown workload {args.workload}; one of {sorted(inputs.WORKLOADS)}")
    w = inputs.WORKLOADS[args.workload]
    if args.seqlen:
        w = w.with_(seqlen=args.seqlen, name=f"{w.name}@S={args.seqlen}")
    w = w.with_(backward=w.backward and not args.fwd_only)   # a forward-only workload stays forward only
    if args.non_causal:
        w = w.with_(causal=False, name=f"{w.name}@non-causal")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        per_step = max(2.0, args.cpu_seconds / max(1, args.steps + args.warmup))
        arrays = oracle_inputs(w)
        for _ in range(args.warmup):
            cpu_sample(w, per_step, arrays)
        vals, t0 = [], time.perf_counter()
        last = None
        for _ in range(args.steps):
            last = cpu_sample(w, per_step, arrays)
            vals.append(last["value"])
        el = time.perf_counter() - t0
        v = statistics.mean(vals)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * el / args.steps, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded N(0,1) bf16 widened to float64)",
                "config": {"workload": w.name, "seqlen": w.seqlen, "hq": w.hq, "hkv": w.hkv,
                           "head_dim": w.head_dim, "hp": w.hp, "cp": w.cp},
                "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": last["cores"], "kind": "oracle",
                                 "sample": last["sample"]},
                "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    rank, local, world, pg = dist_setup(args.gpus)
    result, x = run_gpu(args, w, rank, local, world, pg)
    arrays = oracle_inputs(w, x) if rank == 0 and not args.no_cpu_baseline else None
    del x
    configs = args.configs if args.configs is not None else (args.workload == DEFAULT_WORKLOAD and world == 1
                                                             and not args.seqlen and not args.fwd_only
                                                             and not args.non_causal)
    if configs:
        import torch
        torch.cuda.empty_cache()
        dev = torch.device("cuda", local)
        result["configs"] = run_other_configs([n for n in OTHER_CONFIGS if n != w.name], dev,
                                              torch.cuda.current_stream(dev), measured_peaks(), local)
    if arrays is not None:
        result["cpu_baseline"] = cpu_sample(w, args.cpu_seconds, arrays)
    if rank == 0:
        print(json.dumps(result))
    if pg is not None:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
