"""Benchmark of the ragged batched speculative-verify step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 2|3|4|5] [--points B:gamma,...] [--sweep]

One step = one verify pass of the whole hot path (embedding, QKV + RoPE + KV
append, paged attention, O, SwiGLU FFN, LM head + softmax statistics,
acceptance + sampling, realignment) over one batch of synthetic inputs that
stay resident in HBM.  Every step draws fresh uniforms, so emitted tokens
follow the acceptance statistics.

Default (workload 4): the metric's own curve, verified tokens/s and step time
against the verify rows B * (gamma + 1), on the crossover sweep's shapes (a
9B-class layer, hidden 4096, 32/8 heads of 128, FFN 12288, vocab 151936,
bf16, KV context 2048 in 16-token pages, per-draft acceptance 0.8).  K timed
steps run at each point of the curve; the line's headline `value` is the
point B = 128, gamma = 3 (512 verify rows: past the memory-to-compute
crossover, and the draft length the pages find throughput-optimal at 128
sequences), and every point is listed in `curve` with its roofline fraction.
Weights (1.63 GB) and, from 8 sequences on, the KV cache exceed L2 (129 MB),
so no L2 flush is needed between steps.

Metric: verified (emitted) tokens per second, sum over sequences of
(accepted + 1) per step / step time; ms per step beside it.  Multi-GPU: one
independent replica per GPU (the step does not shard: every sequence needs
all weights), value = all ranks' tokens / slowest rank's time.  Without an
outer torchrun, --gpus N > 1 launches the N replicas itself.

``--impl reference`` times the CPU oracle (float64 numpy, the plain
restatement of the method, BLAS pinned to one thread) on a bounded sample of
the same workload on the host.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified tokens/s & verify-step us vs B*(gamma+1); % of HBM/tensor roofline"
UNIT = "tokens/s"

# the curve of the default run: (B, gamma) at verify rows 8, 128, 256, 320, 512, 1152
CURVE_POINTS = ((1, 7), (32, 3), (64, 3), (64, 4), (128, 3), (128, 8))
HEADLINE = (128, 3)
# environment that pins the oracle's BLAS to one thread
ONE_THREAD = {"OPENBLAS_NUM_THREADS": "1", "OMP_NUM_THREADS": "1", "MKL_NUM_THREADS": "1",
              "BLIS_NUM_THREADS": "1", "VECLIB_MAXIMUM_THREADS": "1"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=4, choices=[2, 3, 4, 5],
                    help="4: the verify-row curve on the sweep's shapes (default); 2: batch of one; "
                         "3: eight agents; 5: the continuous-batching swarm")
    ap.add_argument("--points", default=None,
                    help="workload 4: the curve's points as B:gamma pairs (default "
                         + ",".join(f"{b}:{g}" for b, g in CURVE_POINTS) + "); the headline is 128:3 when listed, "
                         "else the last point")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the timed steps one by one instead of replaying them as one captured CUDA graph")
    ap.add_argument("--quick", action="store_true",
                    help="profiling run: no clock pre-roll, no e2e or CPU legs (its numbers are not bench values)")
    ap.add_argument("--sweep", action="store_true",
                    help="the whole crossover sweep: B in {1,4,16,32,64,128} x gamma in {0,1,2,3,4,7,8}, ctx 2048; "
                         "one JSON line per point, then a summary line")
    ap.add_argument("--sweep-points", default=None,
                    help="subset of the sweep as B:gamma pairs, e.g. 1:7,32:7,128:8")
    ap.add_argument("--gemm-path", type=int, default=0, choices=[0, 1, 2],
                    help="GEMM kernel: 0 auto by row count, 1 mma.sync, 2 tcgen05")
    ap.add_argument("--timeline", action="store_true",
                    help="kernel timeline of one step (builds and loads libsdv_trace.so): per kernel the entry, "
                         "the end of its wait for the kernel ahead and the exit, and the first and last block "
                         "at each point inside the sampling kernel, medians over --steps steps; "
                         "a markdown table, not a bench line")
    ap.add_argument("--timeline-shapes", default=None,
                    help="timeline of the ctx-2048 sweep shapes instead of --workload, as B:gamma pairs")
    ap.add_argument("--cpu-oracle-child", default=None, help=argparse.SUPPRESS)
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def parse_points(text):
    return [tuple(int(v) for v in pt.split(":")) for pt in text.split(",")]


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

LAYER_DESC = "9B-class layer bf16 (hidden 4096, 32/8 heads x 128, FFN 12288), vocab 151936"


def workload_desc(wid, points=None, headline=None):
    import workloads as wl
    if wid == 2:
        return dict(workload=f"batch-of-one: B=1, gamma=7, {LAYER_DESC}, ctx 2048, acceptance 0.8",
                    B=1, gamma=[7], ctx=[2048], rows=8, l2="inputs larger than L2 (weights 1.63 GB)")
    if wid == 4:
        B, g = headline
        return dict(workload=f"verify-row curve on the roofline crossover sweep's shapes: {LAYER_DESC}, "
                             f"ctx 2048, acceptance 0.8; headline point B={B}, gamma={g} "
                             f"({B * (g + 1)} verify rows), curve points (B, gamma) {list(points)}",
                    B=B, gamma=g, ctx=2048, rows=B * (g + 1), points=[list(p) for p in points],
                    l2="inputs larger than L2 (weights 1.63 GB, KV 1.07 GB at the headline)")
    lens, gam, _ = wl.workload3_shape()
    return dict(workload=f"eight-agent ragged: B=8, gamma_b in {{1,2,3}} (sum<=16), ctx U{{512..8192}}, "
                         f"acceptance {{0.97,0.8,0.14}}, {LAYER_DESC}",
                B=8, gamma=[int(x) for x in gam], ctx=[int(x) for x in lens], rows=int((gam + 1).sum()),
                l2="inputs larger than L2 (weights 1.63 GB)")


def host_batch(wid, B=None, gamma=None, lazy=False):
    import workloads as wl
    if wid == 2:
        return wl.workload2(extra_pages=8)
    if wid == 3:
        return wl.workload3(extra_pages=16)
    return wl.workload4(B, gamma, kv_fill="lazy" if lazy else "normal", extra_pages=4 * B + 8)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------

def phase_work(batch):
    """Algorithmic (flops, bytes) of each phase of one step on the 9B-class layer.

    Flops count the contraction once (2 per multiply-add), whatever the
    kernel's operand split; attention counts QK^T and PV over each row's
    visible positions.  Bytes count what the phase must move at least once:
    weights, KV read and written, activations in and out, draft
    probabilities read by the rule.
    """
    H, F, V, D, nq, nkv = 4096, 12288, 151936, 128, 32, 8
    R, B, G = int(batch.R), int(batch.B), int(batch.G)
    nqkv = (nq + 2 * nkv) * D
    vis = sum(int(L) * (int(g) + 1) + (int(g) + 1) * (int(g) + 2) // 2
              for L, g in zip(batch.seq_lens, batch.draft_lens))
    kv_read = int(sum(batch.seq_lens)) * nkv * 2 * D * 2
    kv_write = R * nkv * 2 * D * 2
    return {
        "prologue": (0, R * H * 2 + R * H * 4),
        "qkv": (2 * R * nqkv * H, nqkv * H * 2 + kv_write + R * nq * D * 4),
        "attention": (4 * vis * nq * D, kv_read + kv_write + 2 * R * nq * D * 4),
        "o_proj": (2 * R * H * nq * D, H * nq * D * 2 + 2 * R * H * 4),
        "ffn": (2 * R * 3 * F * H, 3 * F * H * 2 + 2 * R * H * 4),
        "lm_head": (2 * R * V * H, V * H * 2 + R * H * 2 + ((V + 127) // 128) * R * 8),
        "accept": (0, G * 4 + B * V * 4),
        "realign": (0, 0),
    }


# DRAM traffic of one LM-head launch (dram__bytes_read.sum + dram__bytes_write.sum) from ncu
# captures of this bench's own command, keyed by the launch's row count and recorded with a hash of
# the GEMM sources they were taken on; once those sources change the numbers no longer describe the
# kernel and the bench reports null.
LM_HEAD_TRAFFIC = {"sources_sha": "9958fa8877ecfd9d", "bytes": {512: 1250407168 + 300421376}}
GEMM_SOURCES = ("gemm.cu", "gemm_tc.cu", "gemm_common.cuh", "common.cuh", "tcgen05.cuh")


def gemm_sources_sha():
    import hashlib
    d = os.path.join(ROOT, "speculative_decoding_verify_ragged_gb300", "csrc")
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def lm_head_traffic(rows):
    if gemm_sources_sha() != LM_HEAD_TRAFFIC["sources_sha"]:
        return None
    return LM_HEAD_TRAFFIC["bytes"].get(int(rows))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1932.1)), "measured"
    return 6800.0, 1900.0, "fallback"


def box_copy_gbps():
    """This box's device-to-device copy bandwidth (torch copy of 1 Gi bf16, best of 5):
    context for comparing runs on different boxes; the roofline uses the peaks file."""
    import torch
    a = torch.empty(1 << 30, dtype=torch.bfloat16, device="cuda")
    b = torch.empty_like(a)
    best = None
    for _ in range(6):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        b.copy_(a)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None else min(best, ms)
    del a, b
    return 2 * (1 << 30) * 2 / (best / 1e3) / 1e9


# ---------------------------------------------------------------------------
# our arm: K timed steps of one batch resident on the device
# ---------------------------------------------------------------------------

def lm_head_work(R, V=151936, H=4096):
    """(flops, bytes) one LM-head launch must do/move: the contraction once,
    the weights once, the normed rows and the per-(vocab tile, row) softmax
    statistics it produces."""
    return 2 * R * V * H, V * H * 2 + R * H * 2 + ((V + 127) // 128) * R * 8


def kernel_roofline(R, avg_us, hbm, tflops, peak_kind, traffic):
    """The LM-head launch against the roofline that binds it at R rows."""
    flops, nbytes = lm_head_work(R)
    t = avg_us * 1e-6
    tensor = flops / (tflops * 1e12) > nbytes / (hbm * 1e9)
    if tensor:
        achieved, peak, unit = flops / t / 1e12, tflops, "TFLOP/s"
    else:
        achieved, peak, unit = nbytes / t / 1e9, hbm, "GB/s"
    return {"bound": "tensor" if tensor else "hbm", "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": traffic, "kernel": "LM-head GEMM (EPI_LMHEAD)",
            "peak_kind": peak_kind, "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": nbytes,
            "avg_launch_us": avg_us}


def step_roofline(batch, ms, hbm, tflops):
    work = phase_work(batch)
    flops = sum(f for f, _ in work.values())
    nbytes = sum(b for _, b in work.values())
    t_hbm, t_tc = nbytes / (hbm * 1e9), flops / (tflops * 1e12)
    return {"bound": "tensor" if t_tc > t_hbm else "hbm", "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
            "roofline_us": max(t_hbm, t_tc) * 1e6, "t_hbm_us": t_hbm * 1e6, "t_tensor_us": t_tc * 1e6,
            "achieved_GBps": nbytes / (ms / 1e3) / 1e9, "achieved_TFLOPs": flops / (ms / 1e3) / 1e12,
            "frac": max(t_hbm, t_tc) / (ms / 1e3)}


class Bench:
    """The device-side state shared by the points of a run: the weights on the
    device and one verify context per draft-length cap."""

    def __init__(self, seed, max_rows, max_slots, gemm_path=0, fmt="bf16"):
        import torch
        import workloads as wl
        from workloads import device as wd
        W = wl.make_weights(wl.NINE_B, seed, fmt=fmt)
        self.Wd = wd.weights_to_device(W)
        del W
        self.max_rows, self.max_slots, self.gemm_path, self.fmt = max_rows, max_slots, gemm_path, fmt
        self.engines = {}
        self.stream = torch.cuda.current_stream()

    def engine(self, gamma_max):
        import torch
        import workloads as wl
        from workloads import device as wd
        from speculative_decoding_verify_ragged_gb300 import VerifyEngine
        if gamma_max not in self.engines:
            self.engines.clear()
            torch.cuda.empty_cache()
            e = VerifyEngine(wd.config(wl.NINE_B, gamma_max, self.fmt), self.Wd, max_rows=self.max_rows,
                             max_slots=self.max_slots)
            e.set_gemm_path(self.gemm_path)
            self.engines[gamma_max] = e
        return self.engines[gamma_max]

    def inputs(self, eng, batch, wid, kv_key=None):
        """The batch on the device with q rebuilt around the target's own p (the
        input recipe: each draft accepted with its sequence's alpha), from an
        untimed prepass of the step."""
        import torch
        import workloads as wl
        from workloads import device as wd
        bd = wd.batch_to_device(batch)
        if kv_key is not None:
            wd.normal_bf16_device_(bd["kv_pool"], kv_key)
        if batch.G == 0:
            return bd
        res = wd.alloc_result(batch.B, batch.R, wl.NINE_B["vocab"], batch.gamma_max, batch.page_table.shape[1],
                              probs=True)
        eng.verify_step(bd, res)
        assert eng.read_status(res["status"]) == 0
        gam = batch.draft_lens
        if (gam == gam[0]).all():
            alphas = torch.as_tensor(batch.alphas, dtype=torch.float64)
            wd.retarget_draft_probs_device(bd["draft_probs"], res["probs"], bd["tokens"], int(gam[0]), alphas)
            batch.draft_probs = bd["draft_probs"].cpu().numpy()
        else:
            wl.retarget_draft_probs(batch, res["probs"].cpu().numpy(), wid)
            bd["draft_probs"].copy_(torch.from_numpy(batch.draft_probs.reshape(batch.G, -1)))
        del res
        # the prepass realigned the page tables: put the step's inputs back
        bd["page_table"].copy_(torch.from_numpy(batch.page_table))
        bd["num_pages"].copy_(torch.from_numpy(batch.num_pages))
        bd["free_pages"].copy_(torch.from_numpy(batch.free_pages))
        bd["num_free_in"].fill_(batch.num_free)
        torch.cuda.synchronize()
        return bd

    def time_steps(self, eng, batch, bd, args, u_key, world, clocks_for=None):
        """W untimed steps, then K steps back to back between two events on the
        launching stream (barrier + synchronize on both sides), with the
        LM-head launch of each step bracketed by its own event pair; then a few
        steps with every phase boundary recorded (serialised, informational)."""
        import torch
        import workloads as wl
        from workloads import device as wd
        from speculative_decoding_verify_ragged_gb300 import PHASES, kernel_launches
        stream = self.stream
        nsteps = args.warmup + args.steps
        g = wl.rng(*u_key)
        U = torch.from_numpy(np.stack([wl.uniform24(g, batch.R) for _ in range(nsteps)])).cuda()
        res = wd.alloc_result(batch.B, batch.R, wl.NINE_B["vocab"], batch.gamma_max, batch.page_table.shape[1])
        # one emitted-offsets row per step, so the token count is read after the timed region
        EO = torch.zeros((nsteps, batch.B + 1), dtype=torch.int32, device="cuda")

        def step(i, s=None):
            bd["uniforms"] = U[i]
            res["emitted_offsets"] = EO[i]
            eng.verify_step(bd, res, stream if s is None else s)

        for i in range(args.warmup):
            step(i)
        assert eng.read_status(res["status"]) == 0
        torch.cuda.synchronize()
        K_LM = PHASES.index("lm_head")
        lm_pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for _ in range(args.steps)]
        for a_, b_ in lm_pairs:
            a_.record(stream)
            b_.record(stream)
        torch.cuda.synchronize()
        clocks = None
        if clocks_for is not None and not args.quick:
            clocks = ClockSampler(clocks_for)
            # pre-roll: the same step back to back for ~1 s so the clock samples see the GPU under load
            t_end = time.perf_counter() + 1.0
            while time.perf_counter() < t_end:
                step(args.warmup - 1)
                torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        launches0 = kernel_launches()

        def timed_steps(s):
            for j, i in enumerate(range(args.warmup, nsteps)):
                evs = [None] * (len(PHASES) + 1)
                evs[K_LM], evs[K_LM + 1] = lm_pairs[j]
                eng.set_phase_events(evs)
                step(i, s)
            eng.set_phase_events(None)

        # the K timed steps captured once as a CUDA graph (programmatic dependent
        # launches and the LM-head event pairs included) and launched once, so a
        # stall of the launching host thread cannot leave the GPU idle inside the
        # timed region; the steps do the same work as launched one by one
        graph = None
        if not args.no_graph:
            try:
                g = torch.cuda.CUDAGraph()
                cap = torch.cuda.Stream()
                cap.wait_stream(stream)
                with torch.cuda.graph(g, stream=cap):
                    timed_steps(cap)
                stream.wait_stream(cap)
                graph = g
            except Exception as e:  # a driver without capture of these launches: one by one
                print(f"bench.py: graph capture failed ({e}); timing launches one by one", file=sys.stderr)
                eng.set_phase_events(None)
                torch.cuda.synchronize()
                graph = None
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            timed_steps(stream)
        t1.record(stream)
        torch.cuda.synchronize()
        launches = kernel_launches() - launches0
        if world > 1:
            torch.distributed.barrier()
        clk = clocks.stop() if clocks else None
        eng.set_phase_events(None)
        assert eng.read_status(res["status"]) == 0
        lm_ms = [a_.elapsed_time(b_) for a_, b_ in lm_pairs]
        # phase breakdown, every boundary recorded (serialised), outside the timed region
        nph = min(10, args.steps)
        evsets = [[torch.cuda.Event(enable_timing=True) for _ in range(len(PHASES) + 1)] for _ in range(nph)]
        for j in range(nph):
            eng.set_phase_events(evsets[j])
            step(args.warmup + j)
        torch.cuda.synchronize()
        eng.set_phase_events(None)
        assert eng.read_status(res["status"]) == 0
        phase_us = {p: statistics.mean(es[k].elapsed_time(es[k + 1]) for es in evsets) * 1e3
                    for k, p in enumerate(PHASES)}
        tokens = int(EO[args.warmup:, batch.B].sum().item())
        return dict(elapsed_ms=t0.elapsed_time(t1), tokens=tokens, lm_us=statistics.mean(lm_ms) * 1e3,
                    phase_us=phase_us, launches=int(launches), clocks=clk, U=U)


def point_summary(batch, ms, tokens_per_s, lm_us, phase_us, hbm, tflops, peak_kind, traffic=None):
    """One curve point: step time, tokens/s, the step's and the LM head's
    roofline fractions, and each phase's fractions (serialised timings)."""
    work = phase_work(batch)
    phases = {}
    for p, us in phase_us.items():
        f, b = work[p]
        t = us * 1e-6
        phases[p] = {"us": us, "hbm_frac": b / t / 1e9 / hbm if t > 0 else None,
                     "tensor_frac": f / t / 1e12 / tflops if t > 0 else None}
    gemm = ("qkv", "o_proj", "ffn", "lm_head")
    g_t = sum(phase_us[p] for p in gemm) * 1e-6
    g_f = sum(work[p][0] for p in gemm)
    g_b = sum(work[p][1] for p in gemm)
    lay = ("qkv", "o_proj", "ffn")
    l_t = sum(phase_us[p] for p in lay) * 1e-6
    l_f = sum(work[p][0] for p in lay)
    B, gam = int(batch.B), [int(x) for x in batch.draft_lens]
    return {"B": B, "gamma": gam[0] if len(set(gam)) == 1 else gam, "rows": int(batch.R), "ms_per_step": ms,
            "tokens_per_s": tokens_per_s, "rows_per_s": batch.R / (ms / 1e3),
            "step_roofline": step_roofline(batch, ms, hbm, tflops),
            "lm_head": kernel_roofline(int(batch.R), lm_us, hbm, tflops, peak_kind, traffic),
            "gemm_hbm_frac": g_b / g_t / 1e9 / hbm, "gemm_tensor_frac": g_f / g_t / 1e12 / tflops,
            "layer_gemm_tensor_frac": l_f / l_t / 1e12 / tflops,
            "phases_serialised": phases}


def init_dist():
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


def finish_dist(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def run_curve(args):
    """Workload 4: K timed steps at each point of the verify-row curve; the
    line's value, e2e and roofline are the headline point's."""
    import torch
    import workloads as wl
    rank, world, local = init_dist()
    points = parse_points(args.points) if args.points else list(CURVE_POINTS)
    headline = HEADLINE if HEADLINE in points else points[-1]
    bench = Bench(4, max(B * (g + 1) for B, g in points), max(B for B, _ in points), args.gemm_path)
    hbm, tflops, peak_kind = measured_peaks()
    curve, head = [], None
    for B, g in points:
        eng = bench.engine(max(1, g))
        batch = host_batch(4, B, g, lazy=True)
        bd = bench.inputs(eng, batch, 4, kv_key=wl._key(4, wl.S_KV, 1000 * B + g))
        is_head = (B, g) == headline
        t = bench.time_steps(eng, batch, bd, args, (4, wl.S_U, 1000 + 16 * B + g + rank), world,
                             clocks_for=local if is_head else None)
        elapsed, tokens, _ = reduce_over_ranks(t["elapsed_ms"], t["tokens"], None, "cuda")
        ms = elapsed / args.steps
        pt = point_summary(batch, ms, tokens / (elapsed / 1e3), t["lm_us"], t["phase_us"], hbm, tflops, peak_kind,
                           lm_head_traffic(batch.R))
        curve.append(pt)
        if is_head:
            e2e = run_e2e(eng, batch, bd, t["U"], args, bench.stream, t["tokens"]) if not args.quick else None
            head = (batch, pt, t, e2e)
        del bd
        torch.cuda.empty_cache()
    batch, pt, t, e2e = head
    elapsed, tokens, e2e_ms = reduce_over_ranks(t["elapsed_ms"], t["tokens"],
                                                e2e["ms_per_step"] if e2e else None, "cuda")
    if e2e is not None:
        e2e["ms_per_step"] = e2e_ms
        e2e["value"] = tokens / (e2e_ms * args.steps / 1e3)
    # the measured crossover: the first row count whose GEMMs run closer to the
    # tensor peak than to the HBM peak; the modelled one from the weights' bytes and flops
    cross = next((p["rows"] for p in sorted(curve, key=lambda x: x["rows"])
                  if p["gemm_tensor_frac"] >= p["gemm_hbm_frac"]), None)
    w_bytes = 2 * (48 * 128 * 4096 + 4096 * 4096 + 3 * 12288 * 4096 + 151936 * 4096)
    model = (w_bytes / (hbm * 1e9)) / (w_bytes / (tflops * 1e12))
    line = {
        "metric": METRIC, "value": tokens / (elapsed / 1e3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**workload_desc(4, points, headline), "parallelism": f"replicas{world}"},
        "e2e": e2e, "gpu_launches": t["launches"], "clocks": t["clocks"],
        "roofline": pt["lm_head"], "step_roofline": pt["step_roofline"],
        "curve": curve,
        "crossover": {"measured_rows": cross, "model_rows": model,
                      "rule": "first curve point whose GEMMs reach a larger fraction of the tensor peak than of "
                              "the HBM peak"},
        "peaks": {"hbm_GBps": hbm, "bf16_TFLOPs": tflops, "kind": peak_kind},
        "box_copy_GBps": box_copy_gbps() if not args.quick else None,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.quick:
        line["cpu_baseline"] = cpu_baseline(headline)
    finish_dist(world)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_ours(args):
    """Workloads 2 and 3: one batch, K timed steps."""
    import workloads as wl
    rank, world, local = init_dist()
    batch = host_batch(args.workload)
    bench = Bench(args.workload, max(64, batch.R), max(16, batch.B), args.gemm_path)
    eng = bench.engine(int(batch.gamma_max))
    bd = bench.inputs(eng, batch, args.workload)
    t = bench.time_steps(eng, batch, bd, args, (args.workload, wl.S_U, 1000 + rank), world, clocks_for=local)
    tokens_rank = t["tokens"]
    e2e = run_e2e(eng, batch, bd, t["U"], args, bench.stream, tokens_rank) if not args.quick else None
    elapsed_ms, tokens, e2e_ms = reduce_over_ranks(t["elapsed_ms"], tokens_rank,
                                                   e2e["ms_per_step"] if e2e else None, "cuda")
    if e2e is not None:
        e2e["ms_per_step"] = e2e_ms
        e2e["value"] = tokens / (e2e_ms * args.steps / 1e3)
    hbm, tflops, peak_kind = measured_peaks()
    ms = elapsed_ms / args.steps
    pt = point_summary(batch, ms, tokens / (elapsed_ms / 1e3), t["lm_us"], t["phase_us"], hbm, tflops, peak_kind,
                       lm_head_traffic(batch.R))
    line = {
        "metric": METRIC, "value": tokens / (elapsed_ms / 1e3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**workload_desc(args.workload), "parallelism": f"replicas{world}",
                   "verify_rows_per_step": batch.R},
        "e2e": e2e, "gpu_launches": t["launches"], "clocks": t["clocks"],
        "roofline": pt["lm_head"], "step_roofline": pt["step_roofline"],
        "phases_us_serialised": t["phase_us"],
        "emitted_tokens_per_step": tokens / (args.steps * world),
        "box_copy_GBps": box_copy_gbps() if not args.quick else None,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.quick:
        line["cpu_baseline"] = cpu_baseline((1, 7) if args.workload == 2 else None)
    finish_dist(world)
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the whole roofline crossover sweep (9B-class layer, ctx 2048, uniform gamma)
# ---------------------------------------------------------------------------

SWEEP_B = (1, 4, 16, 32, 64, 128)
SWEEP_GAMMA = (0, 1, 2, 3, 4, 7, 8)


def run_sweep(args):
    import torch
    import workloads as wl
    init_dist()
    points = parse_points(args.sweep_points) if args.sweep_points else \
        [(B, g) for B in SWEEP_B for g in SWEEP_GAMMA]
    bench = Bench(4, max(B * (g + 1) for B, g in points), max(B for B, _ in points), args.gemm_path)
    hbm, tflops, peak_kind = measured_peaks()
    results = []
    for B, g in points:
        eng = bench.engine(max(1, g))
        batch = host_batch(4, B, g, lazy=True)
        bd = bench.inputs(eng, batch, 4, kv_key=wl._key(4, wl.S_KV, 1000 * B + g))
        t = bench.time_steps(eng, batch, bd, args, (4, wl.S_U, 1000 + 16 * B + g), 1)
        ms = t["elapsed_ms"] / args.steps
        pt = point_summary(batch, ms, t["tokens"] / (t["elapsed_ms"] / 1e3), t["lm_us"], t["phase_us"], hbm,
                           tflops, peak_kind)
        pt.update(sweep="crossover", gemm_path=args.gemm_path)
        results.append(pt)
        print(json.dumps(pt), flush=True)
        del bd
        torch.cuda.empty_cache()
    cross = next((p["rows"] for p in sorted(results, key=lambda x: x["rows"])
                  if p["gemm_tensor_frac"] >= p["gemm_hbm_frac"]), None)
    w_bytes = 2 * (48 * 128 * 4096 + 4096 * 4096 + 3 * 12288 * 4096 + 151936 * 4096)
    model = (w_bytes / (hbm * 1e9)) / (w_bytes / (tflops * 1e12))
    # the pages' step model fitted to these steps (ms): B*, best gamma per B, break-even
    from speculative_decoding_verify_ragged_gb300 import roofline as rf
    fitted = rf.fit_regimes([(pt["B"], pt["gamma"] + 1, pt["ms_per_step"]) for pt in results]) \
        if len(results) >= 3 else None
    print(json.dumps({"sweep": "crossover-summary", "points": len(results), "measured_crossover_rows": cross,
                      "model_crossover_rows": model, "peaks": {"hbm_GBps": hbm, "bf16_TFLOPs": tflops,
                                                               "kind": peak_kind},
                      "step_model_ms": rf.report(fitted) if fitted else None,
                      "gemm_path": args.gemm_path}, default=str), flush=True)


# ---------------------------------------------------------------------------
# the agent swarm: continuous batching with the budget rule (int4 layer)
# ---------------------------------------------------------------------------

SWARM = dict(slots=128, budget=512, gamma_max=3, ctx=(1024, 16384), outs=(40, 900), requests=4096)


def swarm_desc():
    s = SWARM
    return dict(workload=f"agent swarm: {s['slots']} slots refilled every step from a queue (continuous batching), "
                         f"gamma = clamp((512 - B) / B, 0, 3), ctx U{{1024..16384}}, outputs log-uniform 40..900, "
                         f"acceptance {{0.97, 0.8, 0.14}} per sequence, 9B-class layer int4 g32 + bf16 LM head, "
                         f"vocab 151936",
                slots=s["slots"], budget_rows=s["budget"], gamma_max=s["gamma_max"],
                l2="inputs larger than L2 (KV ~4.5 GB per step)")


class SwarmDrafter:
    """Stand-in for the drafters: tokens uniform over the vocabulary, q built around
    the target's own p (a prepass of the forward on a copy of the slot state) so each
    draft is accepted with its sequence's alpha, uniforms on the 24-bit grid."""

    def __init__(self, eng, run, alphas, V, max_rows):
        import torch
        self.eng, self.run, self.V = eng, run, V
        self.alphas = torch.as_tensor(alphas, dtype=torch.float64)
        self.probs = torch.empty((max_rows, V), dtype=torch.float32, device="cuda")
        self.pstatus = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.n = 0

    def __call__(self, st, batch):
        import torch
        import workloads as wl
        from workloads import device as wd
        k = self.n
        self.n += 1
        R, G, B, gam = st["rows"], st["drafts"], st["live"], st["gamma"]
        g = wl.rng(5, wl.S_TOKENS, k)
        batch["tokens"] = torch.from_numpy(g.integers(0, self.V, size=R).astype(np.int32)).cuda()
        batch["uniforms"] = torch.from_numpy(wl.uniform24(wl.rng(5, wl.S_U, k), R)).cuda()
        q = wd.draft_probs_device(G, self.V, wl._key(5, wl.S_Q, k))
        batch["draft_probs"] = q
        if G == 0:
            return
        # prepass on a copy of the state realignment moves (page rows, counts, free stack)
        pt, npg = batch["page_table"].clone(), batch["num_pages"].clone()
        fp, nf = self.run.free_pages.clone(), self.run.num_free.clone()
        self.pstatus.zero_()
        self.eng.verify_step(batch, dict(probs=self.probs[:R], status=self.pstatus))
        batch["page_table"].copy_(pt)
        batch["num_pages"].copy_(npg)
        self.run.free_pages.copy_(fp)
        self.run.num_free.copy_(nf)
        ids = torch.tensor(st["ids"], dtype=torch.long)
        wd.retarget_draft_probs_device(q, self.probs[:R], batch["tokens"], gam, self.alphas[ids])


def swarm_step_bytes(seq_lens, R, B, G, V=151936):
    """Algorithmic bytes of one swarm step: int4 layer weights (codes + fp16 group
    scales) and the bf16 LM head once, every sequence's KV read, the new rows' KV
    written, q at the draft tokens plus each sequence's final q row, activations."""
    H, F, D, nq, nkv = 4096, 12288, 128, 32, 8
    layer = ((nq + 2 * nkv) * D * H + H * nq * D + 3 * F * H)
    w = layer // 2 + layer // 32 * 2 + V * H * 2
    kv = int(sum(seq_lens)) * nkv * 2 * D * 2 + R * nkv * 2 * D * 2
    return w + kv + G * 4 + B * V * 4 + R * H * 2


def run_swarm(args):
    import torch
    import workloads as wl
    from workloads import device as wd
    from speculative_decoding_verify_ragged_gb300 import PHASES, VerifyEngine, kernel_launches
    from speculative_decoding_verify_ragged_gb300.serve import SwarmRunner

    torch.cuda.set_device(0)
    S = SWARM
    slots, budget, gmax, page, V = S["slots"], S["budget"], S["gamma_max"], 16, wl.NINE_B["vocab"]
    W = wl.make_weights(wl.NINE_B, 5, fmt="int4")
    Wd = wd.weights_to_device(W)
    del W
    eng = VerifyEngine(wd.config(wl.NINE_B, gmax, fmt="int4"), Wd, max_rows=budget, max_slots=slots)
    max_pages = (S["ctx"][1] + S["outs"][1] + 2 * gmax + 1 + page - 1) // page + 1
    pool_pages = slots * max_pages
    pool = torch.empty((pool_pages, 8, 2, page, 128), dtype=torch.bfloat16, device="cuda")
    wd.normal_bf16_device_(pool, wl._key(5, wl.S_KV, 0))
    perm = torch.from_numpy(wl.rng(5, wl.S_SEQ, 3).permutation(pool_pages).astype(np.int32))
    run = SwarmRunner(eng, pool, pool_pages, slots, budget, max_pages, free_order=perm)
    lens, limits, alphas = wl.swarm_requests(S["requests"], ctx=S["ctx"], outs=S["outs"])
    for i in range(len(lens)):
        run.submit(i, int(lens[i]), int(limits[i]))
    drafter = SwarmDrafter(eng, run, alphas, V, budget)
    stream = torch.cuda.current_stream()

    def one(timed):
        m = run.sched.slots()
        st, batch = run.plan()
        ctx_now = m["seq_lens"] + st["admit_ctx"]
        drafter(st, batch)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(stream)
        run.verify(st, batch, stream)
        e1.record(stream)
        run.complete(st)
        wall = time.perf_counter() - t0
        return st, ctx_now, e0, e1, wall

    for _ in range(args.warmup):
        one(False)
    clocks = ClockSampler(0)
    n0 = kernel_launches()
    e_before = run.sched.stats()["emitted"]
    recs = [one(True) for _ in range(args.steps)]
    launches = kernel_launches() - n0
    clk = clocks.stop()
    torch.cuda.synchronize()
    emitted = run.sched.stats()["emitted"] - e_before
    ms = [r[2].elapsed_time(r[3]) for r in recs]
    total_ms = sum(ms)
    hbm, tflops, peak_kind = measured_peaks()
    step_bytes = [swarm_step_bytes(r[1], r[0]["rows"], r[0]["live"], r[0]["drafts"]) for r in recs]
    achieved = sum(step_bytes) / (total_ms / 1e3) / 1e9
    # phases of a few more steps, every boundary recorded (serialised), for the dominant kernel
    nph = 5
    evsets = [[torch.cuda.Event(enable_timing=True) for _ in range(len(PHASES) + 1)] for _ in range(nph)]
    ph_ctx = []
    for j in range(nph):
        eng.set_phase_events(evsets[j])
        st, ctx_now, *_ = one(False)
        ph_ctx.append((st, ctx_now))
    eng.set_phase_events(None)
    torch.cuda.synchronize()
    ph_us = {p: statistics.mean(es[k].elapsed_time(es[k + 1]) for es in evsets) * 1e3 for k, p in enumerate(PHASES)}
    kv_bytes = statistics.mean(int(sum(c)) * 4096 + st["rows"] * 4096 for st, c in ph_ctx)
    attn_gbs = kv_bytes / (ph_us["attention"] * 1e-6) / 1e9
    live = [r[0]["live"] for r in recs]
    line = {"metric": METRIC, "value": emitted / (total_ms / 1e3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {**swarm_desc(), "parallelism": "replicas1",
                       "mean_live": statistics.mean(live), "mean_rows": statistics.mean(r[0]["rows"] for r in recs),
                       "mean_ctx": statistics.mean(statistics.mean(r[1]) for r in recs)},
            "gpu_launches": int(launches), "clocks": clk,
            "roofline": {"bound": "hbm", "achieved": attn_gbs, "peak": hbm, "unit": "GB/s", "frac": attn_gbs / hbm,
                         "traffic": None, "kernel": "paged attention (phase, serialised events)",
                         "peak_kind": peak_kind, "algorithmic_bytes_per_launch": kv_bytes,
                         "avg_launch_us": ph_us["attention"]},
            "step_roofline": {"bound": "hbm", "achieved_GBps": achieved, "frac": achieved / hbm,
                              "algorithmic_bytes": statistics.mean(step_bytes)},
            "phases_us_serialised": ph_us,
            "loop_wall_ms_per_step": statistics.mean(r[4] for r in recs) * 1e3,
            "emitted_tokens_per_step": emitted / args.steps,
            "finished_sequences": run.sched.stats()["finished"]}
    print(json.dumps(line), flush=True)


def reduce_over_ranks(elapsed_ms: float, tokens: int, e2e_ms_per_step, device):
    """Whole-job numbers over the replicas: the slowest rank's times and every
    rank's emitted tokens.  One process: the inputs unchanged."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return elapsed_ms, tokens, e2e_ms_per_step
    t = torch.tensor([elapsed_ms, -1.0 if e2e_ms_per_step is None else e2e_ms_per_step], dtype=torch.float64,
                     device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    k = torch.tensor([tokens], dtype=torch.int64, device=device)
    dist.all_reduce(k)
    return float(t[0].item()), int(k[0].item()), (None if e2e_ms_per_step is None else float(t[1].item()))


def run_e2e(eng, batch, bd, U, args, stream, tokens):
    """The same step through the public API with host inputs: every step copies
    its inputs from pinned host memory and reads its results back.  The copies
    run on a second stream into two sets of device inputs used in turn, so step
    i + 1's inputs cross while step i computes (as a serving loop would); every
    copy of the timed steps lies between the two timing events."""
    import torch
    import workloads as wl
    from workloads import device as wd

    def pin(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if dtype is not None:
            t = t.view(dtype)
        return t.pin_memory()

    host_in = {
        "seq_lens": pin(batch.seq_lens.astype(np.int32)), "draft_lens": pin(batch.draft_lens.astype(np.int32)),
        "tokens": pin(batch.tokens.astype(np.int32)),
        "draft_probs": pin(batch.draft_probs.astype(np.float32).reshape(batch.G, -1)),
        "page_table": pin(batch.page_table.astype(np.int32)), "num_pages": pin(batch.num_pages.astype(np.int32)),
        "num_free_in": pin(np.array([batch.num_free], np.int32)),
    }
    Uh = U.cpu().pin_memory()
    devs = []
    for _ in range(2):
        dev = dict(bd)
        for k, v in host_in.items():
            dev[k] = torch.empty_like(v, device="cuda")
        dev["num_free_out"] = dev["num_free_in"]
        dev["uniforms"] = torch.empty(batch.R, dtype=torch.float32, device="cuda")
        devs.append(dev)
    res = wd.alloc_result(batch.B, batch.R, wl.NINE_B["vocab"], batch.gamma_max, batch.page_table.shape[1],
                          next_view=False)
    outs = ("accepted", "final_tokens", "emitted_tokens", "emitted_offsets", "new_seq_lens")
    host_out = {k: torch.empty_like(res[k], device="cpu").pin_memory() for k in outs}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values()) + batch.R * 4
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    copy_stream = torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in range(2)]
    used = [torch.cuda.Event() for _ in range(2)]
    in_use = [False, False]

    def upload(i):
        slot = i & 1
        with torch.cuda.stream(copy_stream):
            if in_use[slot]:
                copy_stream.wait_event(used[slot])  # the step two back has read this set
            for k, v in host_in.items():
                devs[slot][k].copy_(v, non_blocking=True)
            devs[slot]["uniforms"].copy_(Uh[i], non_blocking=True)
            copied[slot].record(copy_stream)

    def compute(i):
        slot = i & 1
        stream.wait_event(copied[slot])
        eng.verify_step(devs[slot], res, stream)
        used[slot].record(stream)
        in_use[slot] = True
        for k in outs:
            host_out[k].copy_(res[k], non_blocking=True)

    def run(first, n):
        upload(first)
        for i in range(first, first + n):
            if i + 1 < first + n:
                upload(i + 1)
            compute(i)

    run(0, args.warmup)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    copy_stream.wait_event(t0)
    run(args.warmup, args.steps)
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    # the e2e steps use the same uniforms as the device-resident loop, so they
    # emit the same tokens
    return {"value": tokens / (ms / 1e3), "unit": UNIT, "ms_per_step": ms / args.steps,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "overlap": "each step's inputs copied on a second stream while the previous step computes"}


# ---------------------------------------------------------------------------
# the oracle on the host: the CPU baseline and the reference arm
# ---------------------------------------------------------------------------
# A bounded sample of the workload: ONE sequence of the point's shape (its
# gamma + 1 rows, context 2048, its own pages of bf16 N(0,1) KV) through the
# whole step, q rebuilt around the oracle's own p.  The oracle runs with its
# BLAS pinned to one thread (the environment below is set before numpy loads,
# in a child process), warmed once before timing.

def oracle_sample(gamma, ctx=2048):
    import workloads as wl
    from oracle import verify_step as o
    W = wl.make_weights(wl.NINE_B, 4)
    batch = wl.make_batch(wl.NINE_B, 4, seq_lens=[ctx], draft_lens=[gamma], gamma_max=max(1, gamma),
                          alphas=[0.8])
    if batch.G:
        fw = o.forward(batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens, batch.draft_lens,
                       batch.tokens)
        wl.retarget_draft_probs(batch, fw["probs"].astype(np.float32), 4)
    return W, batch


def oracle_steps(W, batch, n_min, seconds_min, seconds_max, key):
    """Time oracle steps (fresh uniforms each) until both n_min steps and
    seconds_min have passed (stopping at seconds_max)."""
    import workloads as wl
    from oracle import verify_step as o
    g = wl.rng(4, wl.S_U, key)
    times, tokens = [], []
    while len(times) < n_min or (sum(times) < seconds_min and sum(times) < seconds_max):
        batch.uniforms = wl.uniform24(g, batch.R)
        t = time.perf_counter()
        out = o.verify_step(batch, W)
        times.append(time.perf_counter() - t)
        tokens.append(int(out["emitted_offsets"][-1]))
    return times, tokens


def cpu_oracle_child(spec):
    """In the child process: warm the oracle once, then time it."""
    gamma, ctx, n_min, s_min, s_max = (int(x) for x in spec.split(":"))
    W, batch = oracle_sample(gamma, ctx)
    oracle_steps(W, batch, 1, 0, 0, 3000)
    times, tokens = oracle_steps(W, batch, n_min, s_min, s_max, 3001)
    print(json.dumps({"times": times, "tokens": tokens, "rows": batch.R}), flush=True)


def run_oracle_child(gamma, ctx, n_min, s_min, s_max):
    env = dict(os.environ, **ONE_THREAD)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-oracle-child",
                        f"{gamma}:{ctx}:{n_min}:{s_min}:{s_max}"], env=env, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"oracle child failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(shape):
    """The oracle as it stands, one thread, on one sequence of the point's shape
    (about 10 to 30 s of CPU work)."""
    gamma, ctx = (shape[1], 2048) if shape is not None else (2, 4352)
    d = run_oracle_child(gamma, ctx, 1, 10, 30)
    total = sum(d["times"])
    return {"value": sum(d["tokens"]) / total, "unit": UNIT, "cores": os.cpu_count(), "threads": 1, "kind": "oracle",
            "sample": f"{len(d['times'])} oracle steps of one sequence of the workload's shape ({d['rows']} rows, "
                      f"gamma {gamma}, ctx {ctx}), BLAS on one thread, warmed once, {total:.1f} s"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    if args.workload == 4:
        points = parse_points(args.points) if args.points else list(CURVE_POINTS)
        headline = HEADLINE if HEADLINE in points else points[-1]
        gamma, ctx, desc = headline[1], 2048, workload_desc(4, points, headline)
    elif args.workload == 2:
        gamma, ctx, desc = 7, 2048, workload_desc(2)
    else:
        gamma, ctx, desc = 2, 4352, workload_desc(3)
    # the oracle as it stands: each step one verify pass over one sequence of the
    # workload's shape (a bounded sample), W untimed steps then K timed ones
    d = run_oracle_child(gamma, ctx, args.warmup + args.steps, 0, 0)
    times = d["times"][args.warmup:]
    total = sum(times)
    value = sum(d["tokens"][args.warmup:]) / total
    sample = (f"each step: one oracle verify pass over one sequence of the workload's shape ({d['rows']} rows, "
              f"gamma {gamma}, ctx {ctx}), BLAS on one thread")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total / len(times) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {**desc, "parallelism": "host"},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "threads": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# kernel timeline (libsdv_trace.so): where a live step's time goes, with the
# kernels overlapping as in the bench (programmatic dependent launch)
# ---------------------------------------------------------------------------

TIMELINE_ROWS = ["prologue", "QKV GEMM", "attention", "attention merge", "O GEMM", "gate/up GEMM", "down GEMM",
                 "final RMSNorm", "LM-head GEMM", "acceptance", "sampling", "realignment", "probabilities",
                 "admission", "planes", "other GEMM"]
# points inside the sampling kernel (stochastic verification from logits):
# first block to reach each, last block to reach it
SAMPLE_PHASES = {25: "status read", 26: "row statistics merged", 27: "draft tests done",
                 28: "chunk sums stored", 29: "slot's last block starts", 30: "draw's chunk found"}
TIMELINE_ORDER = [0, 1, 17, 2, 3, 4, 20, 5, 21, 6, 22, 7, 8, 24, 9, 10, 25, 26, 27, 28, 29, 30, 11]


def timeline_name(k):
    if k in SAMPLE_PHASES:
        return "- sampling: " + SAMPLE_PHASES[k]
    return TIMELINE_ROWS[k] if k < 16 else TIMELINE_ROWS[k - 16] + " fixup"


def timeline_of(eng, step, steps):
    """Medians over `steps` traced steps of (entry, wait done, exit) per
    kernel, in us from the prologue's entry, and the untraced step time."""
    import torch
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for i in range(steps):
        step(i)
    e1.record(s)
    torch.cuda.synchronize()
    live_us = e0.elapsed_time(e1) / steps * 1e3
    table = torch.zeros((32, 3), dtype=torch.int64, device="cuda")
    eng.set_trace(table)
    rows = []
    try:
        for i in range(steps):
            table[:, 0:2] = 2 ** 62
            table[:, 2] = 0
            step(i)
            torch.cuda.synchronize()
            rows.append(table.cpu().numpy().astype(np.float64))
    finally:
        eng.set_trace(None)
    return live_us, timeline_rows(np.stack(rows))


def timeline_rows(a):
    """(row, entry, wait done, exit) per stamped row of the trace tables `a`
    [steps, 32, 3] (global-timer ns): medians over the steps, in us from the
    prologue's entry, in TIMELINE_ORDER; a row some step left unstamped is
    left out, and a kernel none of whose blocks passed its wait in some step
    (a fixup with no cut tile: every block leaves before it) has wait None."""
    t0 = a[:, 0, 0]
    out = []
    for k in TIMELINE_ORDER:
        if not (a[:, k, 2] > 0).all():
            continue
        rel = lambda col: float(np.median(a[:, k, col] - t0)) / 1e3  # noqa: E731
        waited = (a[:, k, 1] < 2 ** 62).all()
        out.append((k, rel(0), rel(1) if waited else None, rel(2)))
    return out


def print_timeline(title, live_us, out):
    print(f"\n### {title}: step {live_us:.1f} us (untraced, back to back)\n")
    print("| kernel | entry (us) | wait done | exit | busy (exit - max(wait done, previous exit)) |")
    print("|---|---|---|---|---|")
    prev = 0.0
    prev_point = 0.0
    for k, ent, wt, ex in out:
        if k in SAMPLE_PHASES:
            # a point: first block, -, last block, time since the previous point's last block
            print(f"| {timeline_name(k)} | {ent:.1f} | - | {ex:.1f} | {ex - prev_point:.1f} |")
            prev_point = ex
            continue
        if wt is None:
            # no block waited for the kernel ahead: it added nothing after it
            print(f"| {timeline_name(k)} | {ent:.1f} | - | {ex:.1f} | {max(0.0, ex - prev):.1f} |")
            prev = max(prev, ex)
            continue
        print(f"| {timeline_name(k)} | {ent:.1f} | {wt:.1f} | {ex:.1f} | {ex - max(wt, prev):.1f} |")
        prev = ex
        prev_point = wt
    print(flush=True)


def run_timeline(args):
    import torch
    import workloads as wl
    from workloads import device as wd
    from speculative_decoding_verify_ragged_gb300 import VerifyEngine, _abi, build
    build.build(trace=True)
    torch.cuda.set_device(0)
    W = wl.make_weights(wl.NINE_B, 2)
    Wd = wd.weights_to_device(W)
    if args.timeline_shapes:
        cases = [(int(x.split(":")[0]), int(x.split(":")[1])) for x in args.timeline_shapes.split(",")]
    else:
        cases = [None]
    for case in cases:
        if case is None:
            batch = wl.workload2(extra_pages=8) if args.workload == 2 else wl.workload3(extra_pages=16)
            wid, title = args.workload, workload_desc(args.workload)["workload"]
        else:
            batch = wl.workload4(case[0], case[1], kv_fill="lazy", extra_pages=4 * case[0] + 8)
            wid, title = 4, f"B = {case[0]}, gamma = {case[1]}, ctx 2048 (R = {batch.R})"
        gmax = int(batch.gamma_max)
        eng = VerifyEngine(wd.config(wl.NINE_B, gmax), Wd, max_rows=max(64, batch.R), max_slots=max(16, batch.B),
                           lib_path=_abi.TRACE_LIB_PATH)
        eng.set_gemm_path(args.gemm_path)
        bd = wd.batch_to_device(batch)
        res = wd.alloc_result(batch.B, batch.R, wl.NINE_B["vocab"], gmax, batch.page_table.shape[1], probs=True)
        eng.verify_step(bd, res)
        assert eng.read_status(res["status"]) == 0
        wl.retarget_draft_probs(batch, res["probs"].cpu().numpy(), wid)
        bd = wd.batch_to_device(batch)
        res = wd.alloc_result(batch.B, batch.R, wl.NINE_B["vocab"], gmax, batch.page_table.shape[1])
        g = wl.rng(wid, wl.S_U, 1000)
        U = torch.from_numpy(np.stack([wl.uniform24(g, batch.R) for _ in range(args.steps)])).cuda()

        def step(i):
            bd["uniforms"] = U[i]
            eng.verify_step(bd, res)

        for i in range(args.warmup):
            step(i % args.steps)
        torch.cuda.synchronize()
        assert eng.read_status(res["status"]) == 0
        live_us, out = timeline_of(eng, step, args.steps)
        assert eng.read_status(res["status"]) == 0
        print_timeline(title, live_us, out)
        del eng
        torch.cuda.empty_cache()


def main():
    args = parse()
    if args.cpu_oracle_child:
        cpu_oracle_child(args.cpu_oracle_child)
        return
    if args.warmup < 3:
        args.warmup = 3
    rank, world, _ = dist_env()
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # no outer launcher: start the N replicas here, one process per GPU
        port = 29400 + (os.getpid() % 1000)
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
        sys.exit(subprocess.run(cmd).returncode)
    if world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
        sys.exit(2)
    if args.impl == "reference":
        run_reference(args)
    elif args.timeline:
        run_timeline(args)
    elif args.sweep:
        run_sweep(args)
    elif args.workload == 5:
        run_swarm(args)
    elif args.workload == 4:
        run_curve(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
