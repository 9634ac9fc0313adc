"""Benchmark of the sharded-weight decode path on GB300.

One step = one pass of the hot path over the shared-expert layer (gate_up
[24576, 7168] + down [7168, 12288], FP8 e4m3 with 128x128 float32 block scales,
stored as N = 16 chunks): gather the chunks into a slot, then the two decode
linears at M = 32 on zero-copy views of the slot. `value` is the algorithmic
HBM traffic of the step (gather 2S + weight read S + activations) divided by
the step time. The JSON line also carries per-M results, the fused (no-slot)
variant, the 92-layer lookahead stack with its exposed gather time, the
roofline of the dominant kernel, the end-to-end number through the C ABI with
host buffers, and the CPU oracle timed on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import datetime
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "gather+FP8 GEMM weight GB/s vs HBM peak; exposed gather µs/layer"
HEADLINE_M = 32
L2_FLUSH_BYTES = 512 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--stack-layers", type=int, default=92, help="layers of the lookahead stack (0 skips it)")
    ap.add_argument("--prefill-layers", type=int, default=8, help="layers of the prefill run (0 skips it)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the KDA-layer and tiny-layer decode sections")
    ap.add_argument("--no-bf16", action="store_true", help="skip the 16-bit (bf16, f16) weight sections")
    ap.add_argument("--no-prefetch", action="store_true", help="skip the draft-model prefetch section")
    ap.add_argument("--clock-soak-s", type=float, default=0.5,
                    help="untimed run of the same step for clock samples when the timed region is too short")
    ap.add_argument("--only", choices=["gather", "decode", "layer", "fused", "step", "noalloc", "prefill", "bf16layer"],
                    default=None,
                    help="profiling driver: build the shared-expert layer and run one kernel --reps times")
    ap.add_argument("--m", type=int, default=HEADLINE_M)
    ap.add_argument("--entry", type=int, default=0, help="0 = gate_up, 1 = down")
    ap.add_argument("--reps", type=int, default=4)
    ap.add_argument("--prefill-kernel", choices=["auto", "single", "pair"], default="auto",
                    help="prefill GEMM: one CTA per tile, a CTA pair per tile, or the library's choice")
    ap.add_argument("--decode-kernel", choices=["auto", "mma", "tcgen05"], default="auto",
                    help="which kernel serves decode linears from views")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# process group (one rank per GPU; replicas: no collective on the data path)
# ---------------------------------------------------------------------------
class Dist:
    def __init__(self):
        import torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if torch.cuda.is_available():
            torch.cuda.set_device(self.local)
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            kw = {"device_id": torch.device("cuda", self.local)} if backend == "nccl" else {}
            dist.init_process_group(backend, **kw)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 50 ms, each sample with its
    own timestamp, so a summary can keep only the samples inside a window."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)  # let the sampler start before the caller's window opens
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self, t_from=None, t_to=None):
        """Median SM clock, max clock and active throttle reasons of the samples
        taken between host times t_from and t_to (seconds since the epoch)."""
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                clk, cmax = float(p[2]), float(p[3])
            except ValueError:
                continue
            if (t_from is not None and ts < t_from) or (t_to is not None and ts > t_to):
                continue
            sm.append(clk)
            smax = cmax
            for n, v in zip(names, p[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def fp8_peak():
    """Dense FP8 peak: the measured bf16 cuBLAS peak times the nominal fp8/bf16
    ratio (4.5 / 2.25 = 2); (burst, sustained, source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return 2 * float(d["bf16_tflops"]), 2 * float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), \
            "measured bf16 x 2"
    return 2 * 1900.0, 2 * 1700.0, "fallback bf16 x 2"


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------
def layer_bytes(entries, m):
    """Algorithmic HBM bytes of the decode linears of one layer at batch m."""
    wb = sc = act = 0
    for (_, rows, cols) in entries:
        wb += rows * cols
        sc += 4 * (-(-rows // 128)) * (-(-cols // 128))
        act += 2 * m * cols + 2 * m * rows
    return wb, sc, act


def src_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "sharded_weight_storage_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key, sha):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on
    the current source of the kernel; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_key)
    if not d or d.get("source_sha") != sha:
        return None
    return d.get("dram_bytes_per_launch")


def set_decode_kernel(S, name):
    S.set_option(S.OPT_DECODE_KERNEL, {"auto": S.DECODE_AUTO, "mma": S.DECODE_MMA, "tcgen05": S.DECODE_TCGEN05}[name])


def set_prefill_kernel(S, name):
    S.set_option(S.OPT_PREFILL_KERNEL, {"auto": S.PREFILL_AUTO, "single": S.PREFILL_SINGLE, "pair": S.PREFILL_PAIR}[name])


def decode_kernel_info(name):
    """(dominant kernel name, its sources, launches per decode group) of a
    slot-path decode launch: the library's default is the tcgen05 kernel, which
    runs as three kernels (activation split, GEMM, split-K settle)."""
    if name == "mma":
        return "decode_kernel", ("decode_gemm.cu", "decode_common.cuh", "ptx.cuh"), 1
    return "decode_tc_kernel", ("decode_tc.cu", "decode_common.cuh", "ptx.cuh"), 3


class Timer:
    """CUDA events on one stream; pairs are resolved after a synchronize."""

    def __init__(self, stream):
        self.stream = stream
        self.pairs = {}

    def ev(self):
        import torch
        e = torch.cuda.Event(enable_timing=True)
        e.record(self.stream)
        return e

    def add(self, key, a, b):
        self.pairs.setdefault(key, []).append((a, b))

    def ms(self, key):
        return [a.elapsed_time(b) for a, b in self.pairs.get(key, [])]


KERNEL_TIMING_STEPS = 50  # at least this many event-bracketed steps give the per-kernel durations


def run_ours(args, dist):
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import sharded_weight_storage_gb300 as S
    import workloads as WL
    from sharded_weight_storage_gb300.storage import ShardedStack

    dev = torch.device("cuda", dist.local)
    set_decode_kernel(S, args.decode_kernel)
    set_prefill_kernel(S, args.prefill_kernel)
    w = WL.SHARED_EXPERT
    n = w.n_shards
    ents = [(0, e.rows, e.cols) for e in w.entries]
    t_gen = time.time()
    lw = WL.layer_weights(w, 0)
    st = ShardedStack([(0, S.E4M3, r, c) for (_, r, c) in ents], n, max_m=64, device=str(dev))
    st.load_layer(0, {j: torch.from_numpy(lw.codes[j]) for j in range(len(ents))},
                  {j: torch.from_numpy(lw.scales[j]) for j in range(len(ents))})
    ctx = st.make_ctx()
    del lw
    gen_s = time.time() - t_gen
    total, chunk, _ = st.layout[0]
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream
    scratch = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sink = torch.empty(1024, dtype=torch.float32, device=dev)

    def flush():
        # Reads 512 MB (> L2) so the timed kernel starts with no useful lines
        # and no dirty ones to write back.
        torch.amax(scratch.view(1024, -1), dim=1, out=sink)

    ms_all = sorted(set(w.m_values) | {HEADLINE_M})
    xs = {m: [WL.draw_x(w.key, j, m, c).to(dev) for j, (_, r, c) in enumerate(ents)] for m in ms_all}
    ys = {m: [torch.empty((m, r), dtype=torch.bfloat16, device=dev) for (_, r, c) in ents] for m in ms_all}

    def step(m, tm=None, slot=0):
        prev = tm.ev() if tm else None
        ctx.gather_to_slot(0, slot, sp)
        if tm:
            e = tm.ev()
            tm.add("gather", prev, e)
            prev = e
        ctx.layer_linears(0, slot, [x.data_ptr() for x in xs[m]], [y.data_ptr() for y in ys[m]], m, sp)
        if tm:
            tm.add("linears", prev, tm.ev())

    results = {"per_m": {}}
    torch.cuda.synchronize()

    # ---- headline: K steps at M = 32, inputs larger than L2 ----------------
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step(HEADLINE_M)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    tm = Timer(stream)
    with ClockSampler(dist.local) as clk:
        with torch.cuda.stream(stream):
            h0 = time.time()
            t0 = tm.ev()
            # No events inside: a timing event between one step's settle
            # kernel and the next step's gather keeps the gather from starting
            # under the settle, so per-kernel events would slow the steps.
            for i in range(args.steps):
                step(HEADLINE_M)
            t1 = tm.ev()
            torch.cuda.synchronize()
            h1 = time.time()
            clocks = clk.summary(h0, h1)
            clocks["window"] = "timed region"
            if clocks["samples"] < 3 and args.clock_soak_s > 0:
                # The timed region is shorter than a few sampling intervals: keep
                # the same step running, untimed, for 0.5 s and report those samples.
                h2 = time.time()
                while time.time() - h2 < args.clock_soak_s:
                    for _ in range(50):
                        step(HEADLINE_M)
                    torch.cuda.synchronize()
                clocks = clk.summary(h2, time.time())
                clocks["window"] = (f"{args.clock_soak_s} s of the same step right after the timed region "
                                    "(timed region too short to sample)")
    dist.barrier()
    torch.cuda.synchronize()
    window_ms = t0.elapsed_time(t1)
    window_ms = dist.max(window_ms)
    wb, scb, actb = layer_bytes(ents, HEADLINE_M)
    step_bytes = 2 * total + wb + scb + actb
    # Per-kernel durations behind `roofline`: the same step, right after the
    # timed region (clocks and caches as they were there), repeated at least
    # KERNEL_TIMING_STEPS times with events around each of its two launches.
    kt = Timer(stream)
    n_kt = max(KERNEL_TIMING_STEPS, args.steps)
    with torch.cuda.stream(stream):
        for _ in range(3):
            step(HEADLINE_M)
        for _ in range(n_kt):
            step(HEADLINE_M, kt)
    torch.cuda.synchronize()
    per_kernel = {k: statistics.mean(kt.ms(k)) for k in ("gather", "linears")}
    # The same step on the chunk-map source: the linears read the chunks
    # directly, no gather and no slot (back to back, no events inside).
    with torch.cuda.stream(stream):
        fused = lambda: ctx.layer_linears(0, S.SRC_FUSED, [x.data_ptr() for x in xs[HEADLINE_M]],
                                          [y.data_ptr() for y in ys[HEADLINE_M]], HEADLINE_M, sp)
        for _ in range(args.warmup):
            fused()
        f0 = tm.ev()
        for _ in range(args.steps):
            fused()
        f1 = tm.ev()
    torch.cuda.synchronize()
    results["fused_step_ms"] = dist.max(f0.elapsed_time(f1)) / args.steps
    per_kernel_median = {k: statistics.median(kt.ms(k)) for k in ("gather", "linears")}
    results["headline"] = dict(window_ms=window_ms, step_bytes=step_bytes, per_kernel_ms=per_kernel,
                               per_kernel_median_ms=per_kernel_median, kernel_timing_steps=n_kt)

    # ---- per-M breakdown: step, slot linears, fused linears, gather alone --
    def timed(fn, reps, do_flush=True):
        out = []
        for _ in range(reps):
            if do_flush:
                flush()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            out.append((a, b))
        torch.cuda.synchronize()
        return statistics.median([a.elapsed_time(b) for a, b in out])

    reps = max(10, args.steps)
    with torch.cuda.stream(stream):
        for _ in range(3):
            ctx.gather_to_slot(0, 0, sp)
        g_ms = timed(lambda: ctx.gather_to_slot(0, 0, sp), reps)
        results["gather_alone"] = {"us": g_ms * 1e3, "GBps": 2 * total / g_ms / 1e6}
        # the same gather by the copy engines (N cudaMemcpyAsync, no SMs)
        S.set_option(S.OPT_GATHER_ENGINE, S.GATHER_COPY_ENGINE)
        for _ in range(3):
            ctx.gather_to_slot(0, 0, sp)
        ce_ms = timed(lambda: ctx.gather_to_slot(0, 0, sp), reps)
        # the shared-SM gather kernel (one 48 KB CTA per SM) on its own
        S.set_option(S.OPT_GATHER_ENGINE, S.GATHER_TMA_SHARED_SM)
        for _ in range(3):
            ctx.gather_to_slot(0, 0, sp)
        sh_ms = timed(lambda: ctx.gather_to_slot(0, 0, sp), reps)
        S.set_option(S.OPT_GATHER_ENGINE, S.GATHER_TMA)
        results["gather_copy_engine"] = {"us": ce_ms * 1e3, "GBps": 2 * total / ce_ms / 1e6}
        results["gather_shared_sm_alone"] = {"us": sh_ms * 1e3, "GBps": 2 * total / sh_ms / 1e6}
        # shared-expert chain: gate_up -> SiLU(gate) * up -> down at each m
        f = ents[0][1] // 2
        chain = {}
        for m in w.m_values:
            gu = torch.empty((m, ents[0][1]), dtype=torch.bfloat16, device=dev)
            act = torch.empty((m, f), dtype=torch.bfloat16, device=dev)
            yd = torch.empty((m, ents[1][1]), dtype=torch.bfloat16, device=dev)

            def run_chain(src, m=m, gu=gu, act=act, yd=yd):
                ctx.linear(0, src, xs[m][0].data_ptr(), m, gu.data_ptr(), sp)
                S.silu_mul(gu.data_ptr(), m, f, act.data_ptr(), sp)
                ctx.linear(1, src, act.data_ptr(), m, yd.data_ptr(), sp)

            for _ in range(3):
                run_chain(S.SRC_SLOT0)
                run_chain(S.SRC_FUSED)
            c_ms = timed(lambda: run_chain(S.SRC_SLOT0), reps)
            cf_ms = timed(lambda: run_chain(S.SRC_FUSED), reps)
            a_ms = timed(lambda: S.silu_mul(gu.data_ptr(), m, f, act.data_ptr(), sp), reps)
            chain[m] = {"slot_us": c_ms * 1e3, "fused_us": cf_ms * 1e3, "silu_mul_us": a_ms * 1e3,
                        "silu_mul_GBps": 8 * m * f / a_ms / 1e6, "weight_GBps_slot": total / c_ms / 1e6}
        results["shared_expert_chain"] = chain
        for m in w.m_values:
            wb, scb, actb = layer_bytes(ents, m)
            lin_bytes = wb + scb + actb

            def lins(src):
                ctx.layer_linears(0, src, [x.data_ptr() for x in xs[m]], [y.data_ptr() for y in ys[m]], m, sp)

            for _ in range(3):
                lins(S.SRC_SLOT0)
                lins(S.SRC_FUSED)
            slot_ms = timed(lambda: lins(S.SRC_SLOT0), reps)
            fused_ms = timed(lambda: lins(S.SRC_FUSED), reps)
            step_ms = timed(lambda: step(m), reps, do_flush=False)
            per_entry = {}
            for j, (_, r, c) in enumerate(ents):
                e_ms = timed(lambda j=j: ctx.linear(j, S.SRC_SLOT0, xs[m][j].data_ptr(), m, ys[m][j].data_ptr(), sp),
                             reps)
                eb = layer_bytes([ents[j]], m)
                per_entry[w.entries[j].name] = {"us": e_ms * 1e3, "GBps": sum(eb) / e_ms / 1e6}
            results["per_m"][m] = {
                "step_us": step_ms * 1e3, "step_GBps": (2 * total + lin_bytes) / step_ms / 1e6,
                "weight_GBps_step": total / step_ms / 1e6,
                "slot_linears_us": slot_ms * 1e3, "slot_linears_GBps": lin_bytes / slot_ms / 1e6,
                "fused_linears_us": fused_ms * 1e3, "fused_linears_GBps": lin_bytes / fused_ms / 1e6,
                "per_entry_slot": per_entry,
            }
        # the decode linear that allocates nothing (fixed scratch in the
        # library, warp-level mma.sync kernel) on gate_up from slot 0, beside
        # sws_linear of the same entry (default tcgen05 kernel)
        off0, _, _ = st.entry_info[0]
        rows0, cols0 = ents[0][1], ents[0][2]
        noalloc = {}
        for m in w.m_values:
            def na(m=m):
                S.linear_noalloc(st.slots[0].data_ptr() + off0, st.scales[0].data_ptr(), rows0, cols0,
                                 xs[m][0].data_ptr(), m, ys[m][0].data_ptr(), sp)
            na()
            assert S.noalloc_status() == 0
            na_ms = timed(na, reps)
            nb = sum(layer_bytes([ents[0]], m))
            noalloc[m] = {"us": na_ms * 1e3, "GBps": nb / na_ms / 1e6,
                          "sws_linear_GBps": results["per_m"][m]["per_entry_slot"]["gate_up"]["GBps"]}
        results["noalloc_gate_up"] = noalloc
    torch.cuda.synchronize()

    # ---- end to end through the C ABI with host buffers (M = 32) -----------
    m = HEADLINE_M
    hx = [x.cpu().pin_memory() for x in xs[m]]
    hy = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in ys[m]]

    # A serving loop's order: the step's activations come in from pinned host
    # memory and its outputs go back on a copy stream, beside the gather on the
    # compute stream; events keep every buffer's readers and writers in order
    # (x is overwritten only after the previous step's linears read it, y only
    # after its previous copy out finished).
    cs = torch.cuda.Stream(device=dev)
    lin_done = torch.cuda.Event()
    y_free = torch.cuda.Event()
    x_ready = torch.cuda.Event()
    lin_done.record(stream)
    y_free.record(stream)

    def e2e_step():
        cs.wait_event(lin_done)
        with torch.cuda.stream(cs):
            for j in range(len(ents)):
                xs[m][j].copy_(hx[j], non_blocking=True)
        x_ready.record(cs)
        ctx.gather_to_slot(0, 0, sp)
        stream.wait_event(x_ready)
        stream.wait_event(y_free)
        ctx.layer_linears(0, 0, [x.data_ptr() for x in xs[m]], [y.data_ptr() for y in ys[m]], m, sp)
        lin_done.record(stream)
        cs.wait_event(lin_done)
        with torch.cuda.stream(cs):
            for j in range(len(ents)):
                hy[j].copy_(ys[m][j], non_blocking=True)
        y_free.record(cs)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            e2e_step()
        stream.wait_event(y_free)  # the last step's outputs are back on the host
        b.record(stream)
        torch.cuda.synchronize()
    e2e_ms = dist.max(a.elapsed_time(b)) / args.steps
    h2d = sum(x.numel() * 2 for x in hx)
    d2h = sum(y.numel() * 2 for y in hy)
    results["e2e"] = {"step_ms": e2e_ms, "h2d": h2d, "d2h": d2h}
    results["gen_s"] = gen_s
    results["total"] = total
    results["chunk"] = chunk
    results["clocks"] = clocks
    del st, ctx, scratch
    torch.cuda.empty_cache()
    return results


def run_stack(args, dist, n_layers):
    """Lookahead over a stack of shared-expert layers (92 by default): per-layer
    time, exposed gather time and resident memory."""
    import torch

    import sharded_weight_storage_gb300 as S
    import workloads as WL
    from sharded_weight_storage_gb300.storage import ShardedStack

    dev = torch.device("cuda", dist.local)
    w = WL.STACK92
    n = w.n_shards
    ne = len(w.entries)
    ents = [(l, e.rows, e.cols) for l in range(n_layers) for e in w.entries]
    t_gen = time.time()
    bases = [WL.base_layer(w, b) for b in range(min(w.n_base, n_layers))]
    base_dev = [[torch.from_numpy(c).to(dev) for c in b.codes] for b in bases]
    base_sc = [[torch.from_numpy(s).to(dev) for s in b.scales] for b in bases]
    del bases
    st = ShardedStack([(l, S.E4M3, r, c) for (l, r, c) in ents], n, max_m=64, device=str(dev))
    for l in range(n_layers):
        b = l % len(base_dev)
        codes, scales = {}, {}
        for j, e in enumerate(w.entries):
            signs = torch.from_numpy(WL.draw_row_signs(w.key, l, j, e.rows)).to(dev)
            codes[l * ne + j] = WL.apply_row_signs(base_dev[b][j], signs)
            scales[l * ne + j] = base_sc[b][j]
        st.load_layer(l, codes, scales)
    del base_dev
    ctx = st.make_ctx()
    gen_s = time.time() - t_gen
    m = HEADLINE_M
    xs = [WL.draw_x(w.key, j, m, e.cols).to(dev) for j, e in enumerate(w.entries)]
    ys = [torch.empty((m, e.rows), dtype=torch.bfloat16, device=dev) for e in w.entries]
    io = [([x.data_ptr() for x in xs], [y.data_ptr() for y in ys], m) for _ in range(n_layers)]
    # The gather kernel and the linears share the SMs: the compute stream gets
    # the higher priority, so the block scheduler places the linears' CTAs
    # first when both are waiting for SMs (the equal-priority case is also
    # timed below).
    main = torch.cuda.Stream(device=dev, priority=-5)
    side = torch.cuda.Stream(device=dev, priority=0)

    def steps(k, flags):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(main)
        for _ in range(k):
            ctx.run_layers(0, n_layers - 1, io, flags, main.cuda_stream, side.cuda_stream)
        b.record(main)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / k

    def graph_steps(k, flags):
        # The whole stack recorded once into a CUDA graph, then replayed: the
        # host issues one launch per step instead of ~4 per layer.
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=main):
            ctx.run_layers(0, n_layers - 1, io, flags, main.cuda_stream, side.cuda_stream)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(main):
            for _ in range(2):
                g.replay()
            a.record(main)
            for _ in range(k):
                g.replay()
            b.record(main)
        torch.cuda.synchronize()
        del g
        return a.elapsed_time(b) / k

    def lib_graph_steps(k, flags):
        # The library's own capture (sws_graph_capture), instantiated with
        # per-node priorities, so the linears keep their launch priority.
        g = ctx.graph_capture(0, n_layers - 1, io, flags, main.cuda_stream, side.cuda_stream)
        try:
            for _ in range(2):
                g.launch(main.cuda_stream)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(main)
            for _ in range(k):
                g.launch(main.cuda_stream)
            b.record(main)
            torch.cuda.synchronize()
        finally:
            g.close()
        return a.elapsed_time(b) / k

    k = max(3, args.steps // 2)
    steps(max(2, args.warmup // 2), 0)
    slot_ms = dist.max(steps(k, 0))
    main_hi = main
    main = torch.cuda.Stream(device=dev, priority=0)
    steps(1, 0)
    slot_equal_prio_ms = dist.max(steps(k, 0))
    main = main_hi
    steps(1, S.RUN_FUSED)
    fused_ms = dist.max(steps(k, S.RUN_FUSED))

    def prefilled_steps(k):
        # The same linears with their weights already in a slot (layer 0's,
        # gathered once, read n_layers times): the baseline of the second
        # reading of the exposed gather (lookahead step minus this).
        ctx.gather_to_slot(0, 0, main.cuda_stream)
        ents0 = st.layer_entries(0)
        xs0 = [xs[j] for j in range(len(ents0))]
        ys0 = [ys[j] for j in range(len(ents0))]
        run = lambda: ctx.layer_linears(0, S.SRC_SLOT0, [x.data_ptr() for x in xs0], [y.data_ptr() for y in ys0], m,
                                        main.cuda_stream)
        for _ in range(n_layers):
            run()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(main)
        for _ in range(k):
            for _ in range(n_layers):
                run()
        b.record(main)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / k

    prefilled_ms = dist.max(prefilled_steps(k))
    graph_ms = dist.max(graph_steps(k, 0))
    graph_fused_ms = dist.max(graph_steps(k, S.RUN_FUSED))
    lib_graph_ms = dist.max(lib_graph_steps(k, 0))
    lib_graph_fused_ms = dist.max(lib_graph_steps(k, S.RUN_FUSED))
    # the lookahead with the gather on the copy engines (no SMs taken from the linears)
    S.set_option(S.OPT_GATHER_ENGINE, S.GATHER_COPY_ENGINE)
    steps(1, 0)
    ce_ms = dist.max(steps(k, 0))
    ce_exposed = []
    for _ in range(3):
        ctx.run_layers(0, n_layers - 1, io, S.RUN_TIMING, main.cuda_stream, side.cuda_stream)
        ce_exposed.append(ctx.run_timing(n_layers)[0])
    torch.cuda.synchronize()
    # the lookahead with the shared-SM gather: one 48 KB gather CTA per SM fits
    # beside the linears' GEMM CTA, so gather(l+1) and the linears of l run on
    # the same SMs at once (eager, graph replay, and the stamp-based exposure)
    S.set_option(S.OPT_GATHER_ENGINE, S.GATHER_TMA_SHARED_SM)
    steps(1, 0)
    sh_ms = dist.max(steps(k, 0))
    sh_graph_ms = dist.max(graph_steps(k, 0))
    sh_lib_graph_ms = dist.max(lib_graph_steps(k, 0))
    sh_exposed = []
    for _ in range(3):
        ctx.run_layers(0, n_layers - 1, io, S.RUN_TIMING, main.cuda_stream, side.cuda_stream)
        sh_exposed.append(ctx.run_timing(n_layers)[0])
    torch.cuda.synchronize()
    sh_ex = [statistics.median(v[l] for v in sh_exposed) for l in range(n_layers)]
    S.set_option(S.OPT_GATHER_ENGINE, S.GATHER_TMA)
    ce_ex = [statistics.median(v[l] for v in ce_exposed) for l in range(n_layers)]
    exposed, layer_ms = [], []
    for _ in range(3):
        ctx.run_layers(0, n_layers - 1, io, S.RUN_TIMING, main.cuda_stream, side.cuda_stream)
        e, lm = ctx.run_timing(n_layers)
        exposed.append(e)
        layer_ms.append(lm)
    torch.cuda.synchronize()
    ex = [statistics.median(v[l] for v in exposed) for l in range(n_layers)]
    lm = [statistics.median(v[l] for v in layer_ms) for l in range(n_layers)]
    total = st.layout[0][0]
    resident = st.resident_chunk_bytes() + 2 * st.plan.slot_bytes
    r_bytes = sum(t for (t, _, _) in st.layout)
    out = {
        "workload": f"{n_layers}-layer stack of shared-expert layers, N={n}, M={m}",
        "layers": n_layers, "gen_s": round(gen_s, 1),
        "step_ms": slot_ms, "per_layer_us": slot_ms * 1e3 / n_layers,
        "equal_stream_priority_per_layer_us": slot_equal_prio_ms * 1e3 / n_layers,
        "fused_step_ms": fused_ms, "fused_per_layer_us": fused_ms * 1e3 / n_layers,
        "graph_step_ms": graph_ms, "graph_per_layer_us": graph_ms * 1e3 / n_layers,
        "library_graph_per_layer_us": lib_graph_ms * 1e3 / n_layers,
        "library_graph_fused_per_layer_us": lib_graph_fused_ms * 1e3 / n_layers,
        "copy_engine_gather_step_ms": ce_ms, "copy_engine_gather_per_layer_us": ce_ms * 1e3 / n_layers,
        "copy_engine_exposed_gather_us_per_layer": 1e3 * statistics.mean(ce_ex[1:]) if n_layers > 1 else 1e3 * ce_ex[0],
        "graph_fused_step_ms": graph_fused_ms, "graph_fused_per_layer_us": graph_fused_ms * 1e3 / n_layers,
        "shared_sm_gather_per_layer_us": sh_ms * 1e3 / n_layers,
        "shared_sm_gather_graph_per_layer_us": sh_graph_ms * 1e3 / n_layers,
        "shared_sm_gather_library_graph_per_layer_us": sh_lib_graph_ms * 1e3 / n_layers,
        "shared_sm_gather_exposed_us_per_layer": 1e3 * statistics.mean(sh_ex[1:]) if n_layers > 1 else 1e3 * sh_ex[0],
        "shared_sm_gather_exposed_vs_resident_us_per_layer": (sh_ms - fused_ms) * 1e3 / n_layers,
        "shared_sm_gather_step_GBps": n_layers * (3 * total + sum(layer_bytes(ents[:ne], m)[1:])) / sh_ms / 1e6,
        "exposed_gather_us_per_layer": 1e3 * statistics.mean(ex[1:]) if n_layers > 1 else 1e3 * ex[0],
        "exposed_gather_first_layer_us": 1e3 * ex[0],
        "exposed_frac_of_step": sum(ex) / sum(lm + ex) if sum(lm + ex) > 0 else 0.0,
        "exposed_vs_resident_us_per_layer": (slot_ms - fused_ms) * 1e3 / n_layers,
        "prefilled_slot_per_layer_us": prefilled_ms * 1e3 / n_layers,
        "exposed_vs_prefilled_slot_us_per_layer": (slot_ms - prefilled_ms) * 1e3 / n_layers,
        "layer_linears_us": 1e3 * statistics.mean(lm),
        "step_GBps": n_layers * (3 * total + sum(layer_bytes(ents[:ne], m)[1:])) / slot_ms / 1e6,
        "fused_weight_GBps": n_layers * total / fused_ms / 1e6,
        "resident_bytes_gpu": resident,
        "resident_formula_all_ranks": r_bytes + 2 * st.plan.slot_bytes,
        "resident_formula_per_rank": r_bytes // n + 2 * st.plan.slot_bytes,
        "launches_per_step": n_layers * (1 + decode_kernel_info(args.decode_kernel)[2]),
        "gather_ctas": 2 * torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count,
    }
    del st, ctx, io
    torch.cuda.empty_cache()
    return out


def run_decode_config(args, dist, w, relayout: bool):
    """Decode linears of one layer of workload w at each of its m values: the
    gather, slot linears, chunk-map (fused) linears and gather + linears (µs,
    GB/s), and optionally the one-time relayout from row shards."""
    import torch

    import sharded_weight_storage_gb300 as S
    import sharded_weight_storage_gb300._lib as L
    import workloads as WL
    from sharded_weight_storage_gb300.storage import ShardedStack

    dev = torch.device("cuda", dist.local)
    ents = [(0, e.rows, e.cols) for e in w.entries]
    lw = WL.layer_weights(WL.scaled_workload(w, n_layers=1), 0)
    st = ShardedStack([(0, S.E4M3, r, c) for (_, r, c) in ents], w.n_shards, max_m=64, device=str(dev))
    codes = {j: torch.from_numpy(lw.codes[j]).to(dev) for j in range(len(ents))}
    st.load_layer(0, codes, {j: torch.from_numpy(lw.scales[j]) for j in range(len(ents))})
    ctx = st.make_ctx()
    total = st.layout[0][0]
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream
    scratch = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sink = torch.empty(1024, dtype=torch.float32, device=dev)

    def timed(fn, reps=20, flush=True):
        out = []
        for _ in range(reps):
            if flush:
                torch.amax(scratch.view(1024, -1), dim=1, out=sink)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            out.append((a, b))
        torch.cuda.synchronize()
        return statistics.median([a.elapsed_time(b) for a, b in out])

    out = {"workload": f"{w.name}: {len(ents)} linears, |T| = {total} B, N = {w.n_shards}", "per_m": {}}
    with torch.cuda.stream(stream):
        if relayout:
            n = w.n_shards
            parts = [codes[j][r * (ents[j][1] // n):(r + 1) * (ents[j][1] // n)].contiguous()
                     for j in range(len(ents)) for r in range(n)]
            chunk_ptrs = [c.data_ptr() for c in st.chunks[0]]
            rl = lambda: L.relayout(st.plan, 0, [q.data_ptr() for q in parts], chunk_ptrs, sp)
            rl()
            r_ms = timed(rl, reps=10)
            out["relayout"] = {"us": r_ms * 1e3, "GBps": 2 * total / r_ms / 1e6}
            del parts
        ctx.gather_to_slot(0, 0, sp)
        g_ms = timed(lambda: ctx.gather_to_slot(0, 0, sp))
        out["gather"] = {"us": g_ms * 1e3, "GBps": 2 * total / g_ms / 1e6}
        for m in w.m_values:
            xs = [WL.draw_x(w.key, j, m, c).to(dev) for j, (_, r, c) in enumerate(ents)]
            ys = [torch.empty((m, r), dtype=torch.bfloat16, device=dev) for (_, r, c) in ents]
            lins = lambda src: ctx.layer_linears(0, src, [x.data_ptr() for x in xs], [y.data_ptr() for y in ys],
                                                 m, sp)
            for _ in range(3):
                lins(S.SRC_SLOT0)
                lins(S.SRC_FUSED)
            lb = sum(layer_bytes(ents, m))
            slot_ms = timed(lambda: lins(S.SRC_SLOT0))
            fused_ms = timed(lambda: lins(S.SRC_FUSED))
            step_ms = timed(lambda: (ctx.gather_to_slot(0, 0, sp), lins(S.SRC_SLOT0)))
            out["per_m"][m] = {
                "slot_linears_us": slot_ms * 1e3, "slot_linears_GBps": lb / slot_ms / 1e6,
                "fused_linears_us": fused_ms * 1e3, "fused_linears_GBps": lb / fused_ms / 1e6,
                "gather_plus_linears_us": step_ms * 1e3, "gather_plus_linears_GBps": (2 * total + lb) / step_ms / 1e6,
            }
    assert ctx.status() == 0
    del st, ctx
    torch.cuda.empty_cache()
    return out


def run_16bit(args, dist, f16=False):
    """16-bit weights (the unquantised variants, bf16 or f16): the
    shared-expert layer's two linears in that format (|T| = 528 MB, N = 16):
    gather, decode linears (slot and chunk-map) at each m, weight GB/s against
    the HBM peak; and the prefill GEMM on one KDA-like [12288, 7168] linear at
    m = 8192 against the 16-bit tensor peak (f16 and bf16 share it; for f16
    the time includes the rounding of x to f16). Weights are drawn on the
    device (seeded)."""
    import torch

    import sharded_weight_storage_gb300 as S
    import sharded_weight_storage_gb300._lib as L
    import workloads as WL
    from sharded_weight_storage_gb300.storage import ShardedStack

    dev = torch.device("cuda", dist.local)
    gen = torch.Generator(device=dev)
    gen.manual_seed(20260 + f16)
    wdt, sdt, name = (torch.float16, S.F16, "f16") if f16 else (torch.bfloat16, S.BF16, "bf16")

    def weight(rows, cols):
        w = torch.randn((rows, cols), generator=gen, device=dev, dtype=torch.float32).mul_(0.02)
        return w.to(wdt).view(torch.uint8)

    w = WL.SHARED_EXPERT
    ents = [(0, e.rows, e.cols) for e in w.entries]
    st = ShardedStack([(0, sdt, r, c) for (_, r, c) in ents], w.n_shards, max_m=64, device=str(dev))
    st.load_layer(0, {j: weight(r, c) for j, (_, r, c) in enumerate(ents)}, {})
    ctx = st.make_ctx()
    total = st.layout[0][0]
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream
    scratch = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sink = torch.empty(1024, dtype=torch.float32, device=dev)
    hbm, _ = peaks()

    def timed(fn, reps=20, flush=True):
        out = []
        for _ in range(reps):
            if flush:
                torch.amax(scratch.view(1024, -1), dim=1, out=sink)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            out.append((a, b))
        torch.cuda.synchronize()
        return statistics.median([a.elapsed_time(b) for a, b in out])

    out = {"workload": f"shared_expert_layer with {name} weights: |T| = {total} B, N = {w.n_shards}",
           "kernel": f"decode_tc_kernel (tcgen05 kind::f16, {name} operands)", "per_m": {}}
    with torch.cuda.stream(stream):
        ctx.gather_to_slot(0, 0, sp)
        g_ms = timed(lambda: ctx.gather_to_slot(0, 0, sp))
        out["gather"] = {"us": g_ms * 1e3, "GBps": 2 * total / g_ms / 1e6}
        for m in (1, 8, 32, 64):
            xs = [WL.draw_x(w.key, j, m, c).to(dev) for j, (_, r, c) in enumerate(ents)]
            ys = [torch.empty((m, r), dtype=torch.bfloat16, device=dev) for (_, r, c) in ents]
            lins = lambda src: ctx.layer_linears(0, src, [x.data_ptr() for x in xs], [y.data_ptr() for y in ys],
                                                 m, sp)
            for _ in range(3):
                lins(S.SRC_SLOT0)
                lins(S.SRC_FUSED)
            wb = sum(2 * r * c for (_, r, c) in ents)
            lb = wb + sum(2 * m * (r + c) for (_, r, c) in ents)
            slot_ms = timed(lambda: lins(S.SRC_SLOT0))
            fused_ms = timed(lambda: lins(S.SRC_FUSED))
            out["per_m"][m] = {
                "slot_linears_us": slot_ms * 1e3, "slot_linears_GBps": lb / slot_ms / 1e6,
                "slot_frac_of_hbm": lb / slot_ms / 1e6 / hbm,
                "fused_linears_us": fused_ms * 1e3, "fused_linears_GBps": lb / fused_ms / 1e6,
            }
    assert ctx.status() == 0
    del st, ctx
    torch.cuda.empty_cache()
    # prefill
    rows, cols, m = 12288, 7168, 8192
    st = ShardedStack([(0, sdt, rows, cols)], 8, max_m=m, device=str(dev))
    st.load_layer(0, {0: weight(rows, cols)}, {})
    ctx = st.make_ctx()
    bf16_burst = fp8_peak()[0] / 2
    with torch.cuda.stream(stream):
        ctx.gather_to_slot(0, 0, sp)
        x = torch.randn((m, cols), generator=gen, device=dev).to(torch.bfloat16)
        y = torch.empty((m, rows), dtype=torch.bfloat16, device=dev)
        call = lambda: ctx.linear(0, S.SRC_SLOT0, x.data_ptr(), m, y.data_ptr(), sp)
        call()
        t = timed(call, reps=5)
    fl = 2.0 * m * rows * cols
    kern = "to_f16_kernel + prefill_16_kernel<true>" if f16 else "prefill_16_kernel<false>"
    out["prefill"] = {"linear": f"[{rows}, {cols}] {name} at m = {m}", "kernel": f"{kern} (tcgen05 kind::f16)",
                      "us": t * 1e3, "TFLOPS": fl / t / 1e9, "frac_of_bf16_peak": fl / t / 1e9 / bf16_burst,
                      "bf16_peak_tflops": bf16_burst}
    assert ctx.status() == 0
    del st, ctx, x, y
    torch.cuda.empty_cache()
    return out


def run_prefetch(args, dist, n_target=16, reps=10):
    """Draft-model layer-0 prefetch: a target stack of n_target shared-expert
    layers runs its lookahead, then (after an optional host-side window that
    stands for the work between the two models) a one-layer draft context runs
    its first layer. The exposed part of the draft's first gather (time its
    compute stream waits for the layer) is measured for: a cold start (gather
    inline), a prefetch on a dedicated stream issued before the target, and a
    prefetch on the target's side stream issued after the target's layers."""
    import torch

    import sharded_weight_storage_gb300 as S
    import workloads as WL
    from sharded_weight_storage_gb300.storage import ShardedStack

    dev = torch.device("cuda", dist.local)
    w = WL.SHARED_EXPERT
    base = WL.base_layer(w, 0)
    codes = [torch.from_numpy(c).to(dev) for c in base.codes]
    scales = [torch.from_numpy(s_).to(dev) for s_ in base.scales]
    ne = len(w.entries)
    tst = ShardedStack([(l, S.E4M3, e.rows, e.cols) for l in range(n_target) for e in w.entries], w.n_shards,
                       max_m=64, device=str(dev))
    for l in range(n_target):
        tst.load_layer(l, {l * ne + j: codes[j] for j in range(ne)}, {l * ne + j: scales[j] for j in range(ne)})
    dst = ShardedStack([(0, S.E4M3, e.rows, e.cols) for e in w.entries], w.n_shards, max_m=64, device=str(dev))
    dst.load_layer(0, {j: codes[j] for j in range(ne)}, {j: scales[j] for j in range(ne)})
    tctx, dctx = tst.make_ctx(), dst.make_ctx()
    m = HEADLINE_M
    xs = [WL.draw_x(w.key, j, m, e.cols).to(dev) for j, e in enumerate(w.entries)]
    ys = [torch.empty((m, e.rows), dtype=torch.bfloat16, device=dev) for e in w.entries]
    tio = [([x.data_ptr() for x in xs], [y.data_ptr() for y in ys], m) for _ in range(n_target)]
    dio = [([x.data_ptr() for x in xs], [y.data_ptr() for y in ys], m)]
    main, side, dside, pre = (torch.cuda.Stream(device=dev) for _ in range(4))

    def step(variant, window_s):
        if variant == "dedicated":
            dctx.prefetch_layer(0, 0, pre.cuda_stream)
        tctx.run_layers(0, n_target - 1, tio, 0, main.cuda_stream, side.cuda_stream)
        if variant == "shared_side":
            dctx.prefetch_layer(0, 0, side.cuda_stream)
        if window_s > 0:
            time.sleep(window_s)
        flags = S.RUN_TIMING | (0 if variant == "cold" else S.RUN_FIRST_PREFETCHED)
        dctx.run_layers(0, 0, dio, flags, main.cuda_stream, dside.cuda_stream)
        exposed, _ = dctx.run_timing(1)
        return exposed[0]

    out = {"workload": f"target: {n_target} shared-expert layers (N=16, M={m}); draft: one shared-expert layer",
           "gather_bytes": dst.layout[0][0], "exposed_draft_gather_us": {}}
    for window_ms in (0.0, 4.0):
        res = {}
        for variant in ("cold", "dedicated", "shared_side"):
            step(variant, window_ms / 1e3)
            vals = [step(variant, window_ms / 1e3) for _ in range(reps)]
            res[variant] = 1e3 * statistics.median(vals)
        out["exposed_draft_gather_us"][f"host_window_{window_ms:g}ms"] = res
    torch.cuda.synchronize()
    del tst, dst, tctx, dctx, codes, scales
    torch.cuda.empty_cache()
    return out


def run_prefill(args, dist, n_layers):
    """Prefill on the KDA-layer weights (N = 8): per-linear tcgen05 GEMM
    throughput at M = 2048 and 8192, whole-layer time, and lookahead over
    n_layers layers with the gather overlapped."""
    import torch

    import sharded_weight_storage_gb300 as S
    import workloads as WL
    from sharded_weight_storage_gb300.storage import ShardedStack

    dev = torch.device("cuda", dist.local)
    w = WL.PREFILL
    n = w.n_shards
    ne = len(w.entries)
    ents = [(l, e.rows, e.cols) for l in range(n_layers) for e in w.entries]
    base = WL.base_layer(w, 0)
    base_dev = [torch.from_numpy(c).to(dev) for c in base.codes]
    base_sc = [torch.from_numpy(s).to(dev) for s in base.scales]
    del base
    mmax = max(w.m_values)
    st = ShardedStack([(l, S.E4M3, r, c) for (l, r, c) in ents], n, max_m=mmax, device=str(dev))
    for l in range(n_layers):
        codes, scales = {}, {}
        for j, e in enumerate(w.entries):
            signs = torch.from_numpy(WL.draw_row_signs(w.key, l, j, e.rows)).to(dev)
            codes[l * ne + j] = WL.apply_row_signs(base_dev[j], signs)
            scales[l * ne + j] = base_sc[j]
        st.load_layer(l, codes, scales)
    del base_dev
    ctx = st.make_ctx()
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream
    burst, sustained, src = fp8_peak()
    out = {"workload": f"KDA-like layer x{n_layers}, N={n}, FP8 e4m3 weights and quantised activations",
           "fp8_peak_tflops": burst, "fp8_peak_source": src, "per_m": {}}

    def timed(fn, reps=5):
        ts = []
        for _ in range(reps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    with torch.cuda.stream(stream):
        ctx.gather_to_slot(0, 0, sp)
        for m in w.m_values:
            ctx.gather_to_slot(0, 0, sp)  # the lookahead run below retags both slots
            xs = [WL.draw_x(w.key, j, m, e.cols).to(dev) for j, e in enumerate(w.entries)]
            ys = [torch.empty((m, e.rows), dtype=torch.bfloat16, device=dev) for e in w.entries]
            per = {}
            flops_layer = 0
            for j, e in enumerate(w.entries):
                call = lambda j=j: ctx.linear(j, 0, xs[j].data_ptr(), m, ys[j].data_ptr(), sp)
                call()
                t = timed(call)
                fl = 2.0 * m * e.rows * e.cols
                flops_layer += fl
                per[e.name] = {"us": t * 1e3, "TFLOPS": fl / t / 1e9, "frac_of_fp8_peak": fl / t / 1e9 / burst}
                for kname in ("single", "pair"):  # each GEMM kernel forced, quantiser included
                    set_prefill_kernel(S, kname)
                    call()
                    tk = timed(call)
                    per[e.name][kname + "_us"] = tk * 1e3
                    per[e.name][kname + "_frac_of_fp8_peak"] = fl / tk / 1e9 / burst
                set_prefill_kernel(S, args.prefill_kernel)
            # quantiser alone for the widest activation
            xq = torch.empty((m, 8192), dtype=torch.uint8, device=dev)
            ex = torch.empty((m, 64), dtype=torch.float32, device=dev)
            xw = WL.draw_x(w.key, 99, m, 8192).to(dev)
            q_ms = timed(lambda: S.quantize_x(xw.data_ptr(), m, 8192, xq.data_ptr(), ex.data_ptr(), sp))
            lay = lambda: ctx.layer_linears(0, 0, [x.data_ptr() for x in xs], [y.data_ptr() for y in ys], m, sp)
            lay()
            t_layer = timed(lay)
            io = [([x.data_ptr() for x in xs], [y.data_ptr() for y in ys], m) for _ in range(n_layers)]
            side = torch.cuda.Stream(device=dev)
            ctx.run_layers(0, n_layers - 1, io, 0, sp, side.cuda_stream)
            t_run = timed(lambda: ctx.run_layers(0, n_layers - 1, io, 0, sp, side.cuda_stream), reps=3)
            ctx.run_layers(0, n_layers - 1, io, S.RUN_TIMING, sp, side.cuda_stream)
            exposed, layer_ms = ctx.run_timing(n_layers)
            out["per_m"][m] = {
                "linears": per, "layer_us": t_layer * 1e3, "layer_TFLOPS": flops_layer / t_layer / 1e9,
                "layer_frac_of_fp8_peak": flops_layer / t_layer / 1e9 / burst,
                "quantize_8192_cols_us": q_ms * 1e3,
                "lookahead_step_ms": t_run, "lookahead_TFLOPS": n_layers * flops_layer / t_run / 1e9,
                "exposed_gather_us_per_layer": 1e3 * statistics.mean(exposed[1:]) if n_layers > 1 else 1e3 * exposed[0],
                "exposed_frac_of_step": sum(exposed) / t_run,
            }
            del xs, ys, xq, ex, xw
    torch.cuda.synchronize()
    del st, ctx
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline only; never on the GPU path)
# ---------------------------------------------------------------------------
def oracle_step_setup(rows_frac):
    import oracle as O
    import workloads as WL
    w = WL.SHARED_EXPERT
    lw = WL.layer_weights(w, 0)
    ents = [(0, e.rows, e.cols, 1) for e in w.entries]
    plan = O.plan_layout(ents, w.n_shards)
    t = O.pack(plan, 0, {j: lw.codes[j] for j in range(len(ents))})
    chunks = O.split_chunks(plan, 0, t)
    xs = [WL.bf16_to_f64(WL.bf16_bits(WL.draw_x(w.key, j, HEADLINE_M, e.cols))) for j, e in enumerate(w.entries)]
    sel = [max(1, int(e.rows * rows_frac)) for e in w.entries]
    byts = 2 * t.size
    for j, e in enumerate(w.entries):
        byts += sel[j] * e.cols + 4 * (-(-sel[j] // 128)) * (-(-e.cols // 128)) + 2 * HEADLINE_M * (e.cols + sel[j])
    return plan, chunks, xs, lw, sel, byts


def oracle_step(plan, chunks, xs, lw, sel):
    import oracle as O
    t = O.gather(chunks)
    for j in range(len(xs)):
        v = O.view(plan, 0, t, j)[:sel[j]]
        O.linear(xs[j], v, lw.scales[j][: -(-sel[j] // 128)])


def cpu_baseline(rows_frac=0.25, reps=3):
    setup = oracle_step_setup(rows_frac)
    plan, chunks, xs, lw, sel, byts = setup
    ts = []
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle_step(plan, chunks, xs, lw, sel)
        ts.append(time.perf_counter() - t0)
    t = statistics.median(ts)
    return {"value": byts / t / 1e9, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"shared-expert layer at M={HEADLINE_M}: full gather of the 16 chunks (np.concatenate) + "
                      f"float64 linears on the first {rows_frac:.0%} of each weight's rows; median of {reps}; "
                      "elementwise NumPy on one core, BLAS matmul on all cores",
            "s_per_step": t}


def run_reference(args, dist):
    if dist.rank != 0:
        return None
    rows_frac = 1.0 / 16
    plan, chunks, xs, lw, sel, byts = oracle_step_setup(rows_frac)
    for _ in range(args.warmup):
        oracle_step(plan, chunks, xs, lw, sel)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(plan, chunks, xs, lw, sel)
    dt = (time.perf_counter() - t0) / args.steps
    v = byts / dt / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(1),
        "cpu_baseline": {"value": v, "unit": "GB/s", "kind": "oracle", "cores": os.cpu_count(),
                         "sample": f"per step: full gather of the 16 chunks + float64 linears on the first "
                                   f"{rows_frac:.2%} of each weight's rows at M={HEADLINE_M}; elementwise NumPy "
                                   "on one core, BLAS matmul on all cores"},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def config_block(world):
    return {"workload": "shared_expert_layer: gate_up [24576,7168] + down [7168,12288] FP8 e4m3, 128x128 fp32 "
                        "block scales, one flat T of 264,241,152 B in N=16 chunks; step = gather to slot + "
                        f"2 decode linears at M={HEADLINE_M}",
            "N_chunks": 16, "M": HEADLINE_M,
            "l2": "inputs larger than L2 (264 MB chunks + 264 MB slot per step); kernel-only timings flush L2 "
                  "by reading 512 MB before each launch",
            "kernel_events": f"none inside the timed region; the roofline's per-kernel durations are the mean "
                             f"of >= {KERNEL_TIMING_STEPS} further steps with events around each launch",
            "parallelism": f"replicas x{world} (no collective)"}


def run_only(args, dist):
    """Launches one kernel of the shared-expert layer --reps times (for ncu)."""
    import ctypes as C

    import torch

    import __graft_entry__
    __graft_entry__.build()
    import sharded_weight_storage_gb300 as S
    import workloads as WL
    from sharded_weight_storage_gb300.storage import ShardedStack

    set_decode_kernel(S, args.decode_kernel)
    set_prefill_kernel(S, args.prefill_kernel)
    if args.only == "bf16layer":  # the shared-expert layer's linears with bf16 weights at m = --m
        w = WL.SHARED_EXPERT
        ents = [(0, e.rows, e.cols) for e in w.entries]
        gen = torch.Generator(device="cuda")
        gen.manual_seed(20260)
        st = ShardedStack([(0, S.BF16, r, c) for (_, r, c) in ents], w.n_shards, max_m=64)
        st.load_layer(0, {j: torch.randn((r, c), generator=gen, device="cuda").mul_(0.02).to(torch.bfloat16)
                          .view(torch.uint8) for j, (_, r, c) in enumerate(ents)}, {})
        ctx = st.make_ctx()
        ctx.gather_to_slot(0, 0, 0)
        m = args.m
        xs = [WL.draw_x(w.key, j, m, c).cuda() for j, (_, r, c) in enumerate(ents)]
        ys = [torch.empty((m, r), dtype=torch.bfloat16, device="cuda") for (_, r, c) in ents]
        for _ in range(args.reps):
            ctx.layer_linears(0, S.SRC_SLOT0, [x.data_ptr() for x in xs], [y.data_ptr() for y in ys], m, 0)
        torch.cuda.synchronize()
        assert ctx.status() == 0
        print(f"only=bf16layer m={m} reps={args.reps}: ok")
        return
    if args.only == "prefill":  # one KDA-layer linear (entry --entry) at m = --m tokens
        w = WL.PREFILL
        ents = [(0, e.rows, e.cols) for e in w.entries]
        lw = WL.layer_weights(WL.scaled_workload(w, n_layers=1), 0)
        st = ShardedStack([(0, S.E4M3, r, c) for (_, r, c) in ents], w.n_shards, max_m=args.m)
        st.load_layer(0, {j: torch.from_numpy(lw.codes[j]) for j in range(len(ents))},
                      {j: torch.from_numpy(lw.scales[j]) for j in range(len(ents))})
        ctx = st.make_ctx()
        ctx.gather_to_slot(0, 0, 0)
        j, m = args.entry, args.m
        x = WL.draw_x(w.key, j, m, ents[j][2]).cuda()
        y = torch.empty((m, ents[j][1]), dtype=torch.bfloat16, device="cuda")
        for _ in range(args.reps):
            ctx.linear(j, S.SRC_SLOT0, x.data_ptr(), m, y.data_ptr(), 0)
        torch.cuda.synchronize()
        assert ctx.status() == 0
        print(f"only=prefill m={m} entry={j} reps={args.reps}: ok")
        return
    w = WL.SHARED_EXPERT
    ents = [(0, e.rows, e.cols) for e in w.entries]
    lw = WL.layer_weights(w, 0)
    st = ShardedStack([(0, S.E4M3, r, c) for (_, r, c) in ents], w.n_shards, max_m=64)
    st.load_layer(0, {j: torch.from_numpy(lw.codes[j]) for j in range(len(ents))},
                  {j: torch.from_numpy(lw.scales[j]) for j in range(len(ents))})
    ctx = st.make_ctx()
    ctx.gather_to_slot(0, 0, 0)
    j, m = args.entry, args.m
    x = WL.draw_x(w.key, j, m, ents[j][2]).cuda()
    y = torch.empty((m, ents[j][1]), dtype=torch.bfloat16, device="cuda")
    xl = [WL.draw_x(w.key, jj, m, ents[jj][2]).cuda() for jj in range(len(ents))]
    yl = [torch.empty((m, ents[jj][1]), dtype=torch.bfloat16, device="cuda") for jj in range(len(ents))]
    off = st.entry_info[j][0]
    for _ in range(args.reps):
        if args.only == "gather":
            ctx.gather_to_slot(0, 0, 0)
        elif args.only == "decode":
            ctx.linear(j, S.SRC_SLOT0, x.data_ptr(), m, y.data_ptr(), 0)
        elif args.only == "layer":
            ctx.layer_linears(0, S.SRC_SLOT0, [xx.data_ptr() for xx in xl], [yy.data_ptr() for yy in yl], m, 0)
        elif args.only == "fused":
            ctx.linear(j, S.SRC_FUSED, x.data_ptr(), m, y.data_ptr(), 0)
        elif args.only == "noalloc":
            rc = S.lib().sws_linear_noalloc(C.c_void_p(st.slots[0].data_ptr() + off),
                                            C.c_void_p(st.scales[j].data_ptr()), ents[j][1], ents[j][2],
                                            C.c_void_p(x.data_ptr()), m, C.c_void_p(y.data_ptr()), None)
            assert rc == 0, f"sws_linear_noalloc: {S.last_error()}"
        else:
            ctx.gather_to_slot(0, 0, 0)
            for jj in range(len(ents)):
                xx = WL.draw_x(w.key, jj, m, ents[jj][2]).cuda()
                yy = torch.empty((m, ents[jj][1]), dtype=torch.bfloat16, device="cuda")
                ctx.linear(jj, S.SRC_SLOT0, xx.data_ptr(), m, yy.data_ptr(), 0)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    if args.only == "noalloc":
        assert S.noalloc_status() == 0
    print(f"only={args.only} m={m} entry={j} reps={args.reps}: ok")


def main():
    args = parse()
    dist = Dist()
    if args.only:
        run_only(args, dist)
        return
    if args.impl == "reference":
        line = run_reference(args, dist)
        if line is not None:
            print(json.dumps(line), flush=True)
        dist.close()
        return
    r = run_ours(args, dist)
    stack = run_stack(args, dist, args.stack_layers) if args.stack_layers > 0 else None
    configs = None
    if not args.no_configs:
        import workloads as WL
        configs = {"attn_kda_layer": run_decode_config(args, dist, WL.ATTN_KDA, relayout=True),
                   "tiny_flat_layer": run_decode_config(args, dist, WL.TINY, relayout=True)}
    prefill = run_prefill(args, dist, args.prefill_layers) if args.prefill_layers > 0 else None
    bf16 = run_16bit(args, dist) if not args.no_bf16 else None
    f16 = run_16bit(args, dist, f16=True) if not args.no_bf16 else None
    prefetch = run_prefetch(args, dist) if not args.no_prefetch else None
    if dist.rank != 0:
        dist.close()
        return
    hbm, peak_kind = peaks()
    h = r["headline"]
    ms_step = h["window_ms"] / args.steps
    value = dist.world * h["step_bytes"] / ms_step / 1e6
    pk = h["per_kernel_ms"]
    total = r["total"]
    ents = [(0, 24576, 7168), (0, 7168, 12288)]
    kbytes = {"gather": 2 * total, "linears": sum(layer_bytes(ents, HEADLINE_M))}
    dk_name, dk_src, dk_launches = decode_kernel_info(args.decode_kernel)
    knames = {"gather": ("gather_kernel", src_sha("gather.cu", "ptx.cuh")),
              "linears": (dk_name, src_sha(*dk_src))}
    dom = max(pk, key=lambda k: pk[k])
    achieved = kbytes[dom] / pk[dom] / 1e6
    traffic = ncu_traffic(f"{knames[dom][0]}:{dom}", knames[dom][1])
    pkm = h["per_kernel_median_ms"]
    kernels = {k: {"kernel": knames[k][0], "us": pk[k] * 1e3, "median_us": pkm[k] * 1e3,
                   "GBps": kbytes[k] / pk[k] / 1e6, "frac_of_hbm": kbytes[k] / pk[k] / 1e6 / hbm,
                   "share_of_step": pk[k] / sum(pk.values()), "launches_timed": h["kernel_timing_steps"],
                   "algorithmic_bytes_per_launch": kbytes[k],
                   "traffic": ncu_traffic(f"{knames[k][0]}:{k}", knames[k][1])}
               for k in pk}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8_e4m3 weights (u8 gather); bf16 activations split exactly into two e4m3 terms; e4m3 tensor-core MMA, fp32 accumulate",
        "data": "synthetic (seeded: N(0,0.02) weights, log-uniform 128x128 scales, N(0,1) bf16 activations)",
        "config": config_block(dist.world),
        "roofline": {"bound": "hbm", "kernel": knames[dom][0], "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "peak_source": f"{peak_kind} hbm_gbs", "traffic": traffic,
                     "algorithmic_bytes_per_launch": kbytes[dom], "launches_timed": h["kernel_timing_steps"],
                     "kernels": {k: {"kernel": v["kernel"], "achieved": v["GBps"], "frac": v["frac_of_hbm"]}
                                 for k, v in kernels.items()}},
        "e2e": {"value": dist.world * h["step_bytes"] / r["e2e"]["step_ms"] / 1e6, "unit": "GB/s",
                "h2d_bytes_per_step": r["e2e"]["h2d"], "d2h_bytes_per_step": r["e2e"]["d2h"],
                "ms_per_step": r["e2e"]["step_ms"]},
        "gpu_launches": (1 + dk_launches) * args.steps,
        "clocks": r["clocks"],
        "exposed_gather_us_per_layer": stack["exposed_gather_us_per_layer"] if stack else None,
        "kernels": kernels,
        "gather_alone": r["gather_alone"],
        "gather_shared_sm_alone": r["gather_shared_sm_alone"],
        "gather_copy_engine": r["gather_copy_engine"],
        "shared_expert_chain": r["shared_expert_chain"],
        "per_m": r["per_m"],
        "lookahead_stack": stack,
        "decode_configs": configs,
        "prefill": prefill,
        "bf16_weights": bf16,
        "f16_weights": f16,
        "draft_prefetch": prefetch,
        "noalloc_gate_up": r["noalloc_gate_up"],
        "weight_GBps_step": total / ms_step / 1e6,
        # the chunk-map step: the same linears reading the chunks (no gather, no slot)
        "fused_step": {"ms_per_step": r["fused_step_ms"],
                       "GBps": dist.world * (h["step_bytes"] - 2 * total) / r["fused_step_ms"] / 1e6,
                       "weight_GBps": dist.world * total / r["fused_step_ms"] / 1e6,
                       "frac_of_hbm": (h["step_bytes"] - 2 * total) / r["fused_step_ms"] / 1e6 / hbm},
    }
    if dist.world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
