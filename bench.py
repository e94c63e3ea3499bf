"""Benchmark: optimizer-step time per megabatch on one GB300 (or N replicas).

One step = one Dion step (dion_step_batched, one call per shape group) over the
whole megabatch of the workload.  The Newton-Schulz comparison path
(muon_ns_batched over the same megabatch, per-head on attention QKV) is timed
the same way and reported under "muon".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gb300|reference]

Prints one JSON line (rank 0).  Inputs are synthetic (workloads/), resident in
HBM.  Workloads whose X, G and M total less than three times the L2 size get
an L2 flush (a 258 MB write) before every timed step, outside that step's
event pair; larger ones need none.  Timing: CUDA
events on the launching stream, a barrier plus torch.cuda.synchronize() on both
sides, max over ranks.  Per-kernel device times come from libdion's event
recording around every launch inside the timed region.  "e2e" repeats the
Dion step through the same public call with the gradients copied in from
pinned host memory and the weights copied back every step, each shape group
stepped as eight calls on eighths of its batch, each on its own stream, so
that copies in both directions overlap the steps.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "optimizer-step ms per megabatch; % of HBM (Dion) / bf16 tensor (NS) roofline"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------- clock sampling

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [ln.strip().split(",") for ln in self.file.read().splitlines() if ln.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
                for k, name in enumerate(names):
                    if r[5 + k].strip().lower().startswith("active"):
                        reasons.add(name)
            except Exception:
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------ DRAM traffic from ncu

def csrc_digest():
    """sha256 over libdion's sources: a DRAM-traffic figure captured with other
    sources no longer describes the kernel and is not reported."""
    import glob
    import hashlib
    h = hashlib.sha256()
    src = os.path.join(ROOT, "orthonormal_optimizer_step_gb300", "csrc")
    for f in sorted(glob.glob(os.path.join(src, "*"))):
        h.update(os.path.basename(f).encode())
        h.update(open(f, "rb").read())
    return h.hexdigest()


def profiled_traffic(workload, kernel):
    """DRAM bytes (read + write) per launch of `kernel` on `workload`, from the
    committed summary profiles/dram_traffic_<workload>.txt (lines
    "launch <i> <kernel> read_bytes <r> write_bytes <w>" and
    "csrc_sha256 <hex>"), or (None, why)."""
    path = os.path.join(ROOT, "profiles", f"dram_traffic_{workload}.txt")
    if not os.path.exists(path):
        return None, "no capture for this workload"
    digest, vals = None, []
    for ln in open(path):
        f = ln.split()
        if len(f) >= 2 and f[0] == "csrc_sha256":
            digest = f[1]
        if len(f) >= 7 and f[0] == "launch" and f[2] == kernel:
            vals.append(float(f[4]) + float(f[6]))
    if not vals:
        return None, f"no launches of {kernel} in {os.path.basename(path)}"
    if digest != csrc_digest():
        return None, "kernel sources changed since the capture"
    return sum(vals) / len(vals), f"profiles/{os.path.basename(path)} ({len(vals)} launches)"


# ----------------------------------------------------------- workload setup

def build_state(w, device, seed0):
    import workloads as wl
    state = []
    for gi, g in enumerate(w.groups):
        r = g.rank(w.fraction)
        X, M, Q = wl.make_state(g, r, w.dtype, device, seed0 + gi, w.x_std)
        G = wl.make_grad(g, w.g_std, w.dtype, device, seed0 + gi, step=0)
        state.append({"g": g, "r": r, "X": X, "M": M, "Q": Q, "G": G})
    return state


def dion_bytes_flops(g, r, dtype_bytes):
    """Algorithmic traffic and flops of one Dion step on one shape group:
    B read twice (M fp32 + G), M written once, X read and written, plus the
    m x r and n x r panels; flops 8 m n r (B Q, B^T P, P R^T, P Q^T) plus
    CholeskyQR2 (4 m r^2 + 2 m r^2 per pass)."""
    mn = g.batch * g.m * g.n
    by = mn * (2 * (4 + dtype_bytes) + 4 + 2 * dtype_bytes) + g.batch * 12 * (g.m + g.n) * r
    fl = 8.0 * mn * r + g.batch * 12.0 * g.m * r * r
    return by, fl


def ns_flops(g, steps):
    hd = g.head_dim if g.head_dim else g.n
    heads = g.n // hd
    s, l = min(g.m, hd), max(g.m, hd)
    return g.batch * heads * steps * (4.0 * s * s * l + 2.0 * s ** 3)


# Algorithmic cost of one step's launches of a kernel, summed over the shape
# groups: ("hbm", bytes) for the streaming passes, ("alu", fp32 flops) for the
# r x r factorization, ("tensor", flops) for the QR products.
def kernel_cost(name, w, state):
    eb = 2 if str(w.dtype).endswith("bfloat16") else 4
    tot, bound = 0.0, "hbm"
    for st in state:
        g, r = st["g"], st["r"]
        rp = -(-r // 64) * 64
        mn = g.batch * g.m * g.n
        # which B the products read: wide ranks (rp > 256) form bf16 B and B^T
        # once (dion_formb); narrow bf16 ranks with n % 8 == 0 store bf16 B from
        # the B Q pass; otherwise both passes form B from M and G
        wide = eb == 2 and rp > 256
        b16 = eb == 2 and not wide and g.n % 8 == 0
        if name.startswith("dion_formb"):
            tot += mn * (4 + eb + 2)
        elif name.startswith("dion_bq"):
            tot += mn * (2 if wide else (4 + eb + (2 if b16 else 0))) + g.batch * (g.n * r * 2 + g.m * rp * 4)
        elif name.startswith("dion_btp"):
            tot += mn * (2 if (wide or b16) else (4 + eb)) + g.batch * (g.m * rp * 2 + g.n * rp * (6 if (wide or b16) else 4))
        elif name.startswith("dion_update"):
            tot += mn * (4 + eb + eb + 4 + eb) + g.batch * (g.m * rp * 2 + 2 * g.n * rp * 2)
        elif name in ("chol_inv_pass1", "chol_inv_pass2"):
            # Cholesky r^3/3 + triangular inverse r^3/3; the second pass is
            # counted as a full factorization (its launches return at once for
            # matrices whose Gram passed the near-identity test)
            bound = "alu"
            if r <= 248:
                tot += g.batch * (2.0 / 3.0) * r ** 3
        elif name == "qr_gram_tc" or name == "qr_apply_tc":
            # six bf16 cross-term products per launch; both CholeskyQR passes
            # form a Gram, and both apply through this GEMM up to rank 248
            # (above it the first pass applies inside the blocked factorization)
            bound = "tensor"
            per_step = 2 if (name == "qr_gram_tc" or r <= 248) else 1
            tot += per_step * g.batch * 6 * 2.0 * g.m * r * r
        elif name == "qr_gram_sum":
            tot += g.batch * (6 * 4 + 4) * r * r            # six fp32 partials in, one out
        elif name.startswith("chol_blk_"):
            # blocked factorization (r > 248, blocks of 128), first CholeskyQR pass;
            # the second pass is gated off for near-identity Grams
            bound = "alu" if name == "chol_blk_diag" else "tensor"
            for j0 in range(0, r if r > 248 else 0, 128):
                wb = min(128, r - j0)
                rest = r - j0 - wb
                if name == "chol_blk_diag":
                    tot += g.batch * (2.0 / 3.0) * wb ** 3
                elif name == "chol_blk_panel":
                    tot += g.batch * 6 * 2.0 * rest * wb * wb
                elif name == "chol_blk_trail":
                    tot += g.batch * 6 * 2.0 * rest * (rest + 1) / 2 * wb
                elif name == "chol_blk_solve":
                    tot += g.batch * 6 * 2.0 * g.m * wb * j0
                elif name == "chol_blk_apply":
                    tot += g.batch * 6 * 2.0 * g.m * wb * wb
                else:
                    return None, 0.0
        else:
            return None, 0.0
    return bound, tot


# Tensor-core flops of one step's launches of a streaming kernel: B Q and
# B^T P are 2 m n r each, the update's two products 4 m n r.  At wide ranks
# these, not the bytes, can set the kernel's floor.
def kernel_flops(name, w, state):
    tot = 0.0
    for st in state:
        g, r = st["g"], st["r"]
        mn = g.batch * g.m * g.n
        if name.startswith("dion_bq") or name.startswith("dion_btp"):
            tot += 2.0 * mn * r
        elif name.startswith("dion_update"):
            tot += 4.0 * mn * r
    return tot


# The floor of a kernel that both streams bytes and runs tensor products is
# the larger of the two times; returns (bound, cost) for that floor.
def mixed_bound(bound, cost, flops, hbm_gbs, bf16_tflops):
    if bound == "hbm" and flops / (bf16_tflops * 1e12) > cost / (hbm_gbs * 1e9):
        return "tensor", flops
    return bound, cost


def alu_peak_tflops(sm_mhz=2070.0, sms=152):
    """fp32 FMA peak: SMs x 128 lanes x 2 flops x clock."""
    return sms * 128 * 2 * sm_mhz * 1e6 / 1e12


# ----------------------------------------------------------------- arms

def max_over_ranks(ms, world, device):
    """The slowest rank's time: every rank contributes its own timed region
    and all ranks receive the maximum (a no-op for one rank)."""
    if world <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


L2_BYTES = 129 * 1000 ** 2     # GB300 L2


def input_footprint(w):
    """Bytes of X, G and M a step streams (bf16 or f32 X and G, f32 M)."""
    eb = 2 if str(w.dtype).endswith("bfloat16") else 4
    return sum(g.batch * g.m * g.n * (2 * eb + 4) for g in w.groups)


def needs_l2_flush(w):
    """Workloads whose inputs are not several times the L2 size get an L2
    flush before every timed step, outside the step's own event pair."""
    return input_footprint(w) < 3 * L2_BYTES


def job_value(ms_per_step, world):
    """Whole-job time per megabatch: each of the world replicas steps its own
    megabatch in ms_per_step (the max over ranks), so the job advances world
    megabatches in that time."""
    return ms_per_step / max(1, world)


def run_gb300(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import orthonormal_optimizer_step_gb300 as od
    import workloads as wl

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = select_groups(wl.WORKLOADS[args.workload](), args.group, args.fraction)
    pk = peaks()
    state = build_state(w, dev, 1000 + 17 * rank)
    for st in state:
        st["ws"] = od.new_workspace(od.dion_workspace_size(st["g"].batch, st["g"].m, st["g"].n, st["r"],
                                                           od.DION_BF16 if st["X"].dtype == torch.bfloat16
                                                           else od.DION_F32), dev)

    # Shape groups are independent: each runs on its own stream, forked from
    # and joined back to the timing stream every step.
    main = torch.cuda.current_stream()
    streams = [torch.cuda.Stream() for _ in state] if args.group_streams else [main for _ in state]
    fork = [torch.cuda.Event() for _ in state]
    join = [torch.cuda.Event() for _ in state]

    def grouped(fn):
        for i, st in enumerate(state):
            if streams[i] is not main:
                fork[i].record(main)
                streams[i].wait_event(fork[i])
            with torch.cuda.stream(streams[i]):
                fn(st, streams[i])
            if streams[i] is not main:
                join[i].record(streams[i])
        for i in range(len(state)):
            if streams[i] is not main:
                main.wait_event(join[i])

    def dion_one(st, s):
        od.dion_step_batched(st["X"], st["G"], st["M"], st["Q"], mu=w.mu, lr=w.lr, weight_decay=w.wd,
                             workspace=st["ws"], stream=s)

    def dion_step():
        grouped(dion_one)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # Small workloads: a 2 x L2 buffer is written before every timed step, and
    # each step is timed by its own event pair, so that no step starts with
    # its inputs in L2 and the flush itself is not timed.
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if needs_l2_flush(w) else None

    def timed(fn, steps, prof=None):
        barrier()
        if prof is not None:
            prof.__enter__()
        if flush_buf is None:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(steps):
                fn()
            e1.record()
        else:
            pairs = []
            for _ in range(steps):
                flush_buf.fill_(1.0)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                pairs.append((e0, e1))
        if prof is not None:
            prof.__exit__(None, None, None)
        barrier()
        ms = e0.elapsed_time(e1) if flush_buf is None else sum(a.elapsed_time(b) for a, b in pairs)
        return max_over_ranks(ms, world, dev)

    clocks = Clocks(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[0])
                    if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local_rank)

    if args.skip_dion:   # Newton-Schulz only (profiling captures of its GEMM chain)
        clocks.start()
        ms_step = ms_seq = None
        kernels, gpu_launches, roofline, by, fl = {}, 0, None, 0, 0.0
    else:
        # --- Dion (headline): groups on their own streams, no per-kernel events
        for _ in range(args.warmup):
            dion_step()
        clocks.start()
        ms = timed(dion_step, args.steps)
        ms_step = ms / args.steps
        # --- the same steps again, one group after another on one stream, with an
        # event pair around every libdion kernel: per-kernel device times for the
        # roofline (kernels of different groups do not share the GPU here)
        saved_streams = list(streams)
        streams[:] = [main for _ in state]
        prof = od.profile(max_launches=2048 * args.steps * len(state) + 64)
        ms_seq = timed(dion_step, args.steps, prof) / args.steps
        torch.cuda.synchronize()
        streams[:] = saved_streams
        kernels = prof.read()
        gpu_launches = sum(v[0] for v in kernels.values())   # the headline region launches the same kernels
        by, fl = 0, 0.0
        eb = 2 if w.dtype == torch.bfloat16 else 4
        for st in state:
            b, f = dion_bytes_flops(st["g"], st["r"], eb)
            by += b
            fl += f
        # dominant kernel by device time
        dom = max(kernels.items(), key=lambda kv: kv[1][1]) if kernels else (None, (0, 0.0))
        dom_name, (dom_launches, dom_ms) = dom
        bound, cost_step = kernel_cost(dom_name or "", w, state)
        bound_bytes = bound == "hbm"
        bound, cost_step = mixed_bound(bound, cost_step, kernel_flops(dom_name or "", w, state), pk["hbm_gbs"],
                                       pk["bf16_tflops"])
        per_launch_ms = dom_ms / max(dom_launches, 1)
        achieved, peak, unit = None, None, None
        if bound and dom_ms > 0:
            rate = cost_step * args.steps / (dom_ms * 1e-3)
            if bound == "hbm":
                achieved, peak, unit = rate / 1e9, pk["hbm_gbs"], "GB/s"
            elif bound == "tensor":
                achieved, peak, unit = rate / 1e12, pk["bf16_tflops"], "TFLOP/s"
            else:
                achieved, peak, unit = rate / 1e12, alu_peak_tflops(), "TFLOP/s"
        # every streaming kernel's own fraction, for context
        per_kernel, per_kernel_t = {}, {}
        for k, (nl, kms) in kernels.items():
            kb, kc = kernel_cost(k, w, state)
            if kb == "hbm" and kms > 0:
                per_kernel[k] = round(kc * args.steps / (kms * 1e-3) / 1e9 / pk["hbm_gbs"], 4)
                kf = kernel_flops(k, w, state)
                if mixed_bound(kb, kc, kf, pk["hbm_gbs"], pk["bf16_tflops"])[0] == "tensor":
                    per_kernel_t[k] = round(kf * args.steps / (kms * 1e-3) / 1e12 / pk["bf16_tflops"], 4)
        traffic, traffic_src = profiled_traffic(w.name, dom_name) if dom_name else (None, "no kernel")
        roofline = {"bound": bound or "hbm", "kernel": dom_name, "achieved": achieved, "peak": peak, "unit": unit,
                    "frac": (achieved / peak) if achieved and peak else None, "traffic": traffic,
                    "traffic_unit": "bytes per launch (dram read + write, ncu)", "traffic_source": traffic_src,
                    "algorithmic_bytes_per_launch": kernel_cost(dom_name, w, state)[1] / max(dom_launches / args.steps, 1)
                    if bound_bytes else None,
                    "peak_source": pk["source"] if bound != "alu" else "derived: 152 SMs x 128 FMA x 2 x 2070 MHz",
                    "launches": dom_launches, "ms_per_launch": per_launch_ms,
                    "hbm_frac_by_kernel": per_kernel,
                    # streaming kernels whose tensor products outweigh their
                    # bytes (wide ranks): fraction of the bf16 peak instead
                    "tensor_frac_by_kernel": per_kernel_t,
                    "step_hbm_floor_ms": by / (pk["hbm_gbs"] * 1e9) * 1e3,
                    "step_tensor_floor_ms": fl / (pk["bf16_tflops"] * 1e12) * 1e3,
                    "step_frac_of_floor": max(by / (pk["hbm_gbs"] * 1e9), fl / (pk["bf16_tflops"] * 1e12)) * 1e3
                    / ms_step}

    # --- Muon / Newton-Schulz comparison path ---
    muon = None
    if not args.skip_muon:
        for st in state:
            g = st["g"]
            st["Mn"] = torch.zeros((g.batch, g.m, g.n), dtype=torch.float32, device=dev)
            st["wsn"] = od.new_workspace(od.muon_workspace_size(g.batch, g.m, g.n, g.head_dim,
                                                                od.DION_BF16 if w.dtype == torch.bfloat16
                                                                else od.DION_F32), dev)

        def muon_one(st, s):
            od.muon_ns_batched(st["G"], X=st["X"], M=st["Mn"], head_dim=st["g"].head_dim, steps=w.ns_steps,
                               mu=w.mu, lr=w.lr, weight_decay=w.wd, workspace=st["wsn"], stream=s)

        def muon_step():
            grouped(muon_one)
        msteps = max(1, args.steps // 2)
        for _ in range(max(1, args.warmup)):
            muon_step()
        mms_streams = timed(muon_step, msteps) / msteps
        saved_streams = list(streams)
        streams[:] = [main for _ in state]
        # Each Newton-Schulz GEMM fills the GPU by itself, so at large shapes the
        # groups run faster one after another (concurrent GEMMs on huge matrices
        # evict each other's tiles from L2); both launch orders are timed and the
        # faster one is reported, with which it was.
        mms_seq = timed(muon_step, msteps) / msteps
        mprof = od.profile(max_launches=64 * msteps * len(state) * (w.ns_steps + 2) + 64)
        timed(muon_step, msteps, mprof)
        streams[:] = saved_streams
        mms = min(mms_streams, mms_seq)
        mk = mprof.read()
        nfl = sum(ns_flops(st["g"], w.ns_steps) for st in state)
        gemm_ms = sum(v[1] for k, v in mk.items() if k.startswith("ns_") and ("gram" in k or "poly" in k
                                                                              or "axpy" in k))
        ach = nfl / (gemm_ms / msteps * 1e-3) / 1e12 if gemm_ms > 0 else None
        # the GEMM chain runs back to back for the whole timed region: past about
        # a second of it the GPU sits at its power cap, so the sustained peak applies
        sustained = mms * msteps >= 1000.0
        npk = pk["bf16_tflops_sustained"] if sustained else pk["bf16_tflops"]
        muon = {"ms_per_step": mms, "group_streams": bool(mms_streams <= mms_seq),
                "ms_per_step_streams": mms_streams, "ms_per_step_one_stream": mms_seq,
                "tflops_step": nfl / (mms * 1e-3) / 1e12,
                "roofline": {"bound": "tensor", "kernel": "ns gemm chain", "achieved": ach,
                             "peak": npk, "unit": "TFLOP/s",
                             "frac": ach / npk if ach else None, "traffic": None,
                             "peak_source": pk["source"] + (" sustained" if sustained else " burst")},
                "kernels": {k: {"launches": v[0], "ms": v[1]} for k, v in mk.items()}}
    clk = clocks.stop()

    # --- end to end through the public API with host buffers ---
    e2e = None
    if not args.skip_e2e:
        hostG = [st["G"].cpu().pin_memory() for st in state]
        hostX = [torch.empty_like(st["X"], device="cpu").pin_memory() for st in state]
        h2d = sum(t.numel() * t.element_size() for t in hostG)
        d2h = sum(t.numel() * t.element_size() for t in hostX)

        # Each shape group is stepped as --e2e-parts calls (eight by default) on
        # their own streams (the matrices are independent), so that one part's
        # step and weight copy-out overlap the next part's gradient copy-in.
        nsplit = max(1, args.e2e_parts)
        parts = []
        for st, hg, hx in zip(state, hostG, hostX):
            B = st["g"].batch
            for h in range(nsplit):
                lo, hi = h * B // nsplit, (h + 1) * B // nsplit
                if hi <= lo:
                    continue
                dt_code = od.DION_BF16 if st["X"].dtype == torch.bfloat16 else od.DION_F32
                parts.append({"sl": slice(lo, hi), "st": st, "hG": hg, "hX": hx,
                              "ws": od.new_workspace(od.dion_workspace_size(hi - lo, st["g"].m, st["g"].n, st["r"],
                                                                            dt_code), dev)})
        pstreams = [torch.cuda.Stream() for _ in parts]

        def e2e_step():
            cur = torch.cuda.current_stream()
            for p, s in zip(parts, pstreams):
                s.wait_stream(cur)
                st, sl = p["st"], p["sl"]
                with torch.cuda.stream(s):
                    st["G"][sl].copy_(p["hG"][sl], non_blocking=True)
                    od.dion_step_batched(st["X"][sl], st["G"][sl], st["M"][sl], st["Q"][sl], mu=w.mu, lr=w.lr,
                                         weight_decay=w.wd, workspace=p["ws"], stream=s)
                    p["hX"][sl].copy_(st["X"][sl], non_blocking=True)
            for s in pstreams:
                cur.wait_stream(s)
        for _ in range(2):
            e2e_step()
        esteps = max(1, args.steps // 2)
        ems = timed(e2e_step, esteps) / esteps
        e2e = {"value": job_value(ems, world), "unit": "ms", "ms_per_step": ems, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "calls_per_group": nsplit}

    # --- CPU baseline: the oracle on a bounded sample ---
    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu:
        cpu = cpu_baseline(w, budget_s=args.cpu_budget)

    if rank == 0:
        line = {"metric": METRIC, "value": job_value(ms_step, world) if ms_step is not None else None, "unit": "ms", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
                "data": "synthetic (seeded Gaussian, workloads/)",
                "config": {"workload": w.name, "groups": [[g.batch, g.m, g.n, g.rank(w.fraction)]
                                                          for g in w.groups],
                           "rank_fraction": w.fraction, "params": w.params,
                           "l2": (f"L2 flushed before every timed step ({2 * L2_BYTES // 10**6} MB written, "
                                  f"outside the step's events); X, G, M {input_footprint(w) // 10**6} MB"
                                  if needs_l2_flush(w) else
                                  f"inputs larger than L2 (no flush): X, G, M {input_footprint(w) // 10**6} MB"),
                           "parallelism": f"replicas x{world}",
                           "group_streams": len(state) if args.group_streams else 1},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": gpu_launches,
                "clocks": clk, "kernels": {k: {"launches": v[0], "ms": v[1]} for k, v in kernels.items()},
                "muon": muon, "step_bytes": by, "step_flops": fl, "ms_per_step_one_stream": ms_seq,
                "kernels_note": "per-kernel times from a one-stream pass of the same steps"}
        print(json.dumps(line), flush=True)


def _oracle_inputs(w, g, rng):
    import numpy as np
    r = g.rank(w.fraction)
    X = 0.02 * rng.standard_normal((g.m, g.n))
    G = w.g_std * rng.standard_normal((g.m, g.n))
    M = w.g_std * rng.standard_normal((g.m, g.n))
    Q = rng.standard_normal((g.n, r))
    Q /= np.linalg.norm(Q, axis=0)
    return X, G, M, Q


def oracle_megabatch_ms(w, budget_s, seed=5):
    """Times the oracle's dense-library form (numpy products and LAPACK QR in
    float64, as it stands) on the host cores for one Dion step of the
    workload.  One matrix per shape group is timed first; when the whole
    megabatch fits in budget_s by that estimate, it is then timed in full,
    else the per-group times are scaled by the batch counts (extrapolated).
    Returns (ms per megabatch, ms actually timed, sample description,
    extrapolated)."""
    import numpy as np
    import oracle.dense as dense
    rng = np.random.default_rng(seed)
    per = []
    for g in w.groups:
        ins = _oracle_inputs(w, g, rng)
        t0 = time.perf_counter()
        dense.dion_step(*ins, w.mu, w.lr, w.wd)
        per.append((time.perf_counter() - t0) * 1e3)
    one = sum(per)
    est = sum(g.batch * t for g, t in zip(w.groups, per))
    if est <= budget_s * 1e3:
        t0 = time.perf_counter()
        for g in w.groups:
            for _ in range(g.batch):
                dense.dion_step(*_oracle_inputs(w, g, rng), w.mu, w.lr, w.wd)
        full = (time.perf_counter() - t0) * 1e3
        return full, full + one, "the whole megabatch (" + ", ".join(
            f"{g.batch}x{g.m}x{g.n} r={g.rank(w.fraction)}" for g in w.groups) + "), one Dion step", False
    return est, one, "one matrix per shape group (" + ", ".join(
        f"1x{g.m}x{g.n} r={g.rank(w.fraction)}" for g in w.groups) + "), one Dion step each; the megabatch " \
        "value is extrapolated by the batch counts (" + ", ".join(str(g.batch) for g in w.groups) + ")", True


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def cpu_baseline(w, budget_s=30.0, seed=5):
    """The oracle on the host cores, on a bounded sample of the workload."""
    ms, timed_ms, sample, extrap = oracle_megabatch_ms(w, budget_s, seed)
    return {"value": ms, "unit": "ms", "cores": host_cores(), "kind": "oracle",
            "form": "dense-library form (numpy/LAPACK, float64)", "sample": sample, "extrapolated": extrap,
            "timed_ms": timed_ms}


def select_groups(w, groups, fraction=None):
    """The workload restricted to the shape groups listed (all if None), at
    another rank fraction if one is given."""
    import dataclasses
    if fraction is not None:
        w = dataclasses.replace(w, name=f"{w.name}@r{fraction:g}", fraction=float(fraction))
    if not groups:
        return w
    return dataclasses.replace(w, name=w.name + "[" + ",".join(str(g) for g in groups) + "]",
                               groups=tuple(w.groups[g] for g in groups))


def run_reference(args, rank, world):
    """The reference arm: the oracle itself, on the host cores.  Each step is
    one bounded sample of the workload (the whole megabatch when it fits the
    per-step budget, else one matrix per shape group, extrapolated by the batch
    counts)."""
    if rank != 0:
        return
    import workloads as wl
    w = select_groups(wl.WORKLOADS[args.workload](), args.group, args.fraction)
    for _ in range(args.warmup):
        oracle_megabatch_ms(w, args.cpu_budget)
    vals, timed = [], []
    sample, extrap = "", False
    for k in range(args.steps):
        v, t, sample, extrap = oracle_megabatch_ms(w, args.cpu_budget, seed=5 + k)
        vals.append(v)
        timed.append(t)
    ms = statistics.mean(vals)
    cb = {"value": ms, "unit": "ms", "cores": host_cores(), "kind": "oracle",
          "form": "dense-library form (numpy/LAPACK, float64)", "sample": sample, "extrapolated": extrap,
          "timed_ms_per_step": statistics.mean(timed)}
    line = {"impl": "reference", "metric": METRIC, "value": ms, "unit": "ms", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded Gaussian)",
            "config": {"workload": w.name}, "cpu_baseline": cb, "extrapolated": extrap,
            "timed_ms_per_step": statistics.mean(timed),
            "e2e": {"value": ms, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="llama3-8b-megabatch",
                    help="workload name (workloads.WORKLOADS); default: the Llama-3-8B megabatch, the largest "
                         "single-GPU workload")
    ap.add_argument("--group", type=int, action="append", default=None,
                    help="run only this shape group of the workload (repeatable; for profiling captures)")
    ap.add_argument("--fraction", type=float, default=None,
                    help="override the workload's Dion rank fraction (for profiling captures)")
    ap.add_argument("--skip-dion", action="store_true",
                    help="time only the Newton-Schulz path (no Dion line; for profiling captures)")
    ap.add_argument("--skip-muon", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--e2e-parts", type=int, default=8,
                    help="calls per shape group in the end-to-end run (each on its own stream); on the "
                         "Llama-3-8B megabatch 2, 4, 8 and 16 parts took 104.7, 93.4, 88.8 and 110.4 ms")
    ap.add_argument("--cpu-budget", type=float, default=30.0,
                    help="seconds of oracle time for the CPU baseline (and per reference-arm step)")
    ap.add_argument("--one-stream", dest="group_streams", action="store_false",
                    help="run the shape groups one after another on one stream")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "gb300" else args.warmup

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch.distributed as dist
        import torch
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_gb300(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
