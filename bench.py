#!/usr/bin/env python3
"""Benchmark of the chunked KDA forward on one node.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one chunked KDA forward over one batch of synthetic input: by
default the pages' representative fixed training shape B=1, H=32, T=8192,
K=V=128, bf16 q/k/v, fp32 g/beta, random fp32 initial state, final state
returned.  Inputs are seeded and drawn on the CPU (``kda_inputs``), then held
in HBM.  The timed region is bracketed by a barrier and a device synchronise;
each step's kernel time is taken with CUDA events on the launching stream,
and a 256 MiB buffer (twice the 129 MB L2) is written between steps, outside
the events, so no step starts with its inputs in L2.

One JSON line is printed by rank 0.  ``value`` is whole-job tokens/s (B*T
tokens per forward, summed over ranks; every rank runs its own replica of the
workload, so scaling is weak).  ``e2e`` is the same metric through the public
call with host buffers: pinned host->device copies of the inputs and the
device->host read of o and the final state inside the timed region.
``roofline`` relates the dominant kernel's algorithmic bytes per launch to
the measured HBM copy bandwidth; ``cpu_baseline`` is the fp64 oracle timed on
this machine's host cores on a bounded sample.

``--impl reference`` times the oracle itself (the slow reference program) on
the host cores, one bounded sample of the workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import kda_inputs as ki  # noqa: E402

METRIC = "KDA forward tokens/s (ms/fwd) at H=32 T=8192 K=V=128 bf16; % of roofline"
# The kernels one forward launches, per implementation (the roofline covers
# the whole forward: for the split path that is its two kernels together).
KERNEL_NAMES = {"simt": "fwd_simt_kernel", "tc": "fwd_tc_kernel",
                "split": "fwd_prep_kernel + fwd_rec_kernel"}
HEADLINE = "fixed_bf16_h32_t8192"
PACKED = "packed_bf16_h32_t8192_25seg"
PROLOGUE = "packed_bf16_h32_t8192_25seg_conv"   # the packed shape behind the conv prologue
LONG_FEW_HEADS = "fixed_bf16_h8_t32768"          # long context, few heads: the scan's case
L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# The pages' fastest forward on this shape (TPU v7x, tokamax #19, run 2:
# 1.870 ms for B*T = 8192 tokens); context for vs_baseline, not the target.
PAGES_TPU_FIXED_MS = 1.870
PAGES_TPU_PACKED_MS = 2.891
CHUNK = 64


# ----------------------------------------------------------------------------
# algorithmic work (bytes and FLOPs a perfect kernel must move / do)
# ----------------------------------------------------------------------------
def algorithmic_bytes(w) -> int:
    e = 2 if w.dtype == "bf16" else 4
    per_th = 2 * w.K * e + w.V * e + w.K * 4 + 4 + w.V * e   # q k v g beta o
    n = w.token_heads * per_th
    if w.segments is not None:
        n += w.B * w.T * 4
    state = w.B * w.H * w.K * w.V * 4
    if w.init_state_std is not None:
        n += state
    if w.output_final_state:
        n += state
    return n


def flops_per_chunk_head(K, V, C=CHUNK) -> float:
    """Masked-triangle FLOPs of one full chunk for one head: the intra-chunk
    products (KK^T, QK^T over K; T*beta*[V|K] over V and K), the inter-chunk
    products (w S, Q S, K^T U) and the triangular solve."""
    tri = C * (C + 1) / 2
    return 2 * tri * (3 * K + 2 * V) + 6 * C * K * V + C ** 3 / 3


def algorithmic_flops(w) -> float:
    return w.token_heads * flops_per_chunk_head(w.K, w.V) / CHUNK


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_digest(impl_name: str) -> str:
    """Digest of the source(s) of a path's kernels (the tensor-core backward
    also runs the split forward's prep and recurrence)."""
    fnames = {"tc": ("kda_fwd_tc.cu",), "simt": ("kda_fwd_simt.cu",),
              "split": ("kda_fwd_split.cu",), "conv": ("kda_conv.cu",), "bwd": ("kda_bwd.cu",),
              "bwd_tc": ("kda_bwd_tc.cu", "kda_fwd_split.cu")}[impl_name]
    h = hashlib.sha256()
    for fname in fnames:
        with open(os.path.join(ROOT, "gated_delta_rule_21_gb300", "csrc", fname), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(impl_name: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(impl_name, {}).get(workload)
    if not e or e.get("source_sha") != kernel_source_digest(impl_name):
        return None
    return e.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------
# distributed plumbing (one process per GPU; weak scaling, no collective on
# the data path -- only the barrier and the max-over-ranks of the timings)
# ----------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.rank = int(os.environ.get("RANK", "0"))
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            if torch.cuda.is_available():
                self.pg.barrier(device_ids=[self.local_rank])
            else:
                self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        dev = f"cuda:{self.local_rank}" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def head_partition(h_total: int, world: int, rank: int):
    """Heads [h0, h1) that rank ``rank`` of ``world`` owns in a problem of
    ``h_total`` heads: equal contiguous blocks.  Heads are independent in the
    recurrence, so a rank computes its block with no data exchange."""
    if world < 1 or not 0 <= rank < world or h_total % world:
        raise ValueError(f"cannot split {h_total} heads over {world} ranks")
    per = h_total // world
    return rank * per, (rank + 1) * per


def head_block_seed(seed: int, h0: int, heads_per_rank: int) -> int:
    """Seed of the input block of heads [h0, h0 + heads_per_rank): the inputs
    of the multi-rank problem are drawn block by block, so every rank makes
    only its own block and the blocks differ."""
    return seed + h0 // heads_per_rank


def whole_job_value(world: int, tokens_per_rank: int, ms_max: float) -> float:
    """Whole-job throughput in tokens/s of an H-head layer (H the heads one
    rank owns): the problem has world x H heads, every rank runs the forward
    of its H heads over all tokens, and the job takes as long as its slowest
    rank; equivalently the sum over ranks of each rank's tokens/s."""
    return world * tokens_per_rank / (ms_max * 1e-3)


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.windows = []
        try:
            p = torch.cuda.get_device_properties(device_index)
            self.bus = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        except Exception:  # older torch without the PCI fields
            self.bus = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="kda_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) < 10:
                        continue
                    rows.append(parts)
            os.unlink(self.path)
        except OSError:
            pass
        return self.summarise(rows)

    def summarise(self, rows):
        import datetime as _dt
        mine = [r for r in rows if self.bus and r[1].lower() == self.bus]
        if not mine:
            mine = rows
        def ts(r):
            try:
                return _dt.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                return None
        inside = [r for r in mine if ts(r) is not None and any(a <= ts(r) <= b for a, b in self.windows)]
        window = "timed regions of every leg"
        if not inside:
            inside, window = mine, "timed+warmup (timed region shorter than the sampling period)"
        if not inside:
            return {"samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in inside if num(r[2]) is not None]
        mx = [num(r[3]) for r in inside if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "window": window,
                "power_w_max": max((num(r[4]) or 0.0) for r in inside)}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def device_inputs(x, dev):
    return {n: (x[n].to(dev) if isinstance(x.get(n), torch.Tensor) else None)
            for n in ("q", "k", "v", "g", "beta", "initial_state", "segment_ids")}


def time_steps(fn, steps, warmup, stream, flush, dist, clocks=None):
    for _ in range(warmup):
        flush.zero_()
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    t1 = time.time()
    if clocks is not None:
        clocks.mark(t0, t1)
    return [a.elapsed_time(b) for a, b in evs], t1 - t0


def run_ours(args, dist):
    import gated_delta_rule_21_gb300 as kda
    from gated_delta_rule_21_gb300 import build as kbuild
    kbuild.build()
    dev = torch.device(f"cuda:{dist.local_rank}")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clocks = ClockSampler(dist.local_rank)
    hbm_peak, tc_peak, peak_src = measured_peaks()

    def rank_seed(w):
        h0, _ = head_partition(w.H * dist.world, dist.world, dist.rank)
        return head_block_seed(args.seed, h0, w.H)

    def measure(wname, with_e2e, clocks_=None):
        w = ki.WORKLOADS[wname]
        x = ki.make_inputs(w, seed=rank_seed(w))
        d = device_inputs(x, dev)
        has_seg = d["segment_ids"] is not None
        o = torch.empty(w.B, w.T, w.H, w.V, dtype=d["q"].dtype, device=dev)
        fs = torch.empty(w.B, w.H, w.K, w.V, dtype=torch.float32, device=dev)
        # packed inputs: the split path's items are sized for the workload's
        # runs per row (the pages' bound on segments per row)
        max_runs = len(w.segments) if w.segments is not None else None
        ws = kda.alloc_workspace(w.B, w.T, w.H, w.K, w.V, d["q"].dtype, has_seg, dev,
                                 impl=args.kda_impl, max_runs_per_row=max_runs)

        def step():
            kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                          initial_state=d["initial_state"], segment_ids=d["segment_ids"],
                          output_final_state=True, out=o, final_state_out=fs,
                          workspace=ws, impl=args.kda_impl, v_tile=args.v_tile, stream=stream)

        times, wall = time_steps(step, args.steps, args.warmup, stream, flush, dist, clocks_)
        status = kda.read_device_status(ws)
        if status:
            raise RuntimeError(f"device status bits {status:#x} after the timed steps")
        ms = statistics.mean(times)
        ms_max = dist.max(ms)
        tokens = w.B * w.T
        res = dict(workload=w, ms=ms, ms_max=ms_max, ms_median=statistics.median(times),
                   ms_min=min(times), wall=wall, tokens=tokens, has_seg=has_seg)
        if with_e2e:
            res["e2e"] = measure_e2e(kda, x, d, o, fs, ws, step_args=(w, has_seg))
        return res

    def measure_e2e(kda, x, d, o, fs, ws, step_args):
        w, has_seg = step_args
        names = [n for n in ("q", "k", "v", "g", "beta", "initial_state", "segment_ids")
                 if d[n] is not None]
        host = {n: x[n].contiguous().pin_memory() for n in names}
        o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        fs_h = torch.empty(fs.shape, dtype=fs.dtype).pin_memory()
        h2d = sum(host[n].numel() * host[n].element_size() for n in names)
        d2h = o_h.numel() * o_h.element_size() + fs_h.numel() * fs_h.element_size()

        if args.kda_impl == "auto" and args.v_tile == 0:
            # the library's host-buffer call: copies in, forward, copies out,
            # pipelined over token ranges
            dbuf = torch.zeros(kda.host_buffer_size(w.B, w.T, w.H, w.K, w.V, d["q"].dtype,
                                                    has_seg),
                               dtype=torch.uint8, device=d["q"].device)

            def e2e_step():
                kda.chunk_fwd_host(host["q"], host["k"], host["v"], host["g"], host["beta"],
                                   scale=x["scale"], initial_state=host.get("initial_state"),
                                   segment_ids=host.get("segment_ids"), output_final_state=True,
                                   out=o_h, final_state_out=fs_h, device_buffer=dbuf,
                                   stream=stream)
        else:
            def e2e_step():
                for n in names:
                    d[n].copy_(host[n], non_blocking=True)
                kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                              initial_state=d["initial_state"], segment_ids=d["segment_ids"],
                              output_final_state=True, out=o, final_state_out=fs,
                              workspace=ws, impl=args.kda_impl, v_tile=args.v_tile,
                              stream=stream)
                o_h.copy_(o, non_blocking=True)
                fs_h.copy_(fs, non_blocking=True)

        times, _ = time_steps(e2e_step, args.steps, args.warmup, stream, flush, dist)
        ms = dist.max(statistics.mean(times))
        return {"value": dist.world * w.B * w.T / (ms * 1e-3), "unit": "tokens/s",
                "ms_per_step": ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    def roofline(res):
        w = res["workload"]
        nbytes = algorithmic_bytes(w)
        flops = algorithmic_flops(w)
        t = res["ms"] * 1e-3
        gbs = nbytes / t / 1e9
        impl_name = kernel_impl(w)
        traffic = profiled_traffic(impl_name, w.name)
        return {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(gbs / hbm_peak, 4), "traffic": traffic,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst)"
                if peak_src == "measured" else "fallback 6.8 TB/s",
                "kernel": KERNEL_NAMES[impl_name], "algorithmic_bytes": nbytes,
                "algorithmic_flops": flops,
                "tensor_frac": round(flops / t / 1e12 / tc_peak, 4),
                "roofline_ms": round(max(nbytes / (hbm_peak * 1e9), flops / (tc_peak * 1e12)) * 1e3, 4)}

    def measure_prologue(wname):
        """The short-conv prologue (conv + SiLU + L2 on q, k) alone and followed
        by the forward, on the packed shape with pre-conv inputs."""
        w = ki.WORKLOADS[wname]
        x = ki.make_inputs(w, seed=rank_seed(w))
        d = device_inputs(x, dev)
        cw = x["conv_w"].to(dev)
        o = torch.empty(w.B, w.T, w.H, w.V, dtype=d["q"].dtype, device=dev)
        fs = torch.empty(w.B, w.H, w.K, w.V, dtype=torch.float32, device=dev)
        ws = kda.alloc_workspace(w.B, w.T, w.H, w.K, w.V, d["q"].dtype, True, dev,
                                 impl=args.kda_impl, max_runs_per_row=len(w.segments))

        def conv():
            return kda.short_conv_silu(d["q"], d["k"], d["v"], cw, segment_ids=d["segment_ids"],
                                       l2norm_qk=True, stream=stream)

        def full():
            q, k_, v = conv()
            kda.chunk_fwd(q, k_, v, d["g"], d["beta"], scale=x["scale"],
                          initial_state=d["initial_state"], segment_ids=d["segment_ids"],
                          output_final_state=True, out=o, final_state_out=fs, workspace=ws,
                          impl=args.kda_impl, v_tile=args.v_tile, stream=stream)

        t_conv, _ = time_steps(conv, args.steps, args.warmup, stream, flush, dist, clocks)
        t_full, _ = time_steps(full, args.steps, args.warmup, stream, flush, dist, clocks)
        conv_ms = dist.max(statistics.mean(t_conv))
        full_ms = dist.max(statistics.mean(t_full))
        esz = d["q"].element_size()
        # reads x_q, x_k, x_v, the weights and the ids; writes q, k, v
        conv_bytes = (2 * w.B * w.T * w.H * (2 * w.K + w.V) * esz
                      + 4 * 4 * w.H * (2 * w.K + w.V) + 4 * w.B * w.T)
        gbs = conv_bytes / (conv_ms * 1e-3) / 1e9
        return {"workload": w.name, "conv_ms": conv_ms,
                "conv_roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak,
                                  "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                                  "traffic": profiled_traffic("conv", w.name),
                                  "algorithmic_bytes": conv_bytes, "kernel": "short_conv_kernel"},
                "ms_per_step": full_ms, "unit": "tokens/s",
                "value": whole_job_value(dist.world, w.B * w.T, full_ms),
                # the conv leg, then conv + the packed forward
                "gpu_launches": args.steps * (2 + packed_launches(w))}

    def measure_backward(wname):
        """The backward (kda_chunk_bwd) on the same workload: the gradients
        of sum(d_o * o) + sum(d_final * final_state) for seeded upstream
        gradients, workspace allocated once."""
        w = ki.WORKLOADS[wname]
        x = ki.make_inputs(w, seed=rank_seed(w))
        u = ki.make_upstream_grads(w, seed=rank_seed(w))
        d = device_inputs(x, dev)
        d_o, d_f = u["d_o"].to(dev), u["d_final"].to(dev)
        has_seg = d["segment_ids"] is not None
        # AUTO: the tensor-core backward where it applies (bf16, K = V = 128,
        # no segment ids), else the CUDA-core one
        tc = kda.bwd_workspace_size(w.B, w.T, w.H, w.K, w.V, d["q"].dtype, has_seg,
                                    impl="tc") > 0
        ws = torch.zeros(kda.bwd_workspace_size(w.B, w.T, w.H, w.K, w.V, d["q"].dtype, has_seg),
                         dtype=torch.uint8, device=dev)

        def step():
            kda.chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d_o, scale=x["scale"],
                          initial_state=d["initial_state"], segment_ids=d["segment_ids"],
                          d_final=d_f, workspace=ws, stream=stream)

        steps = args.steps if tc else min(args.steps, 20)
        times, _ = time_steps(step, steps, args.warmup, stream, flush, dist, clocks)
        ms = dist.max(statistics.mean(times))
        th = w.token_heads
        esz = d["q"].element_size()
        # reads q k v d_o (input dtype), g, beta; writes dq dk dg dv (fp32), dbeta;
        # initial state and d_final read, d_initial written
        nbytes = (th * (2 * w.K * esz + 2 * w.V * esz + 4 * w.K + 4)
                  + th * (3 * 4 * w.K + 4 * w.V + 4) + 3 * w.B * w.H * w.K * w.V * 4)
        gbs = nbytes / (ms * 1e-3) / 1e9
        res = {"workload": w.name, "ms_per_step": ms, "unit": "tokens/s",
               "value": whole_job_value(dist.world, w.B * w.T, ms), "steps": steps,
               "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak,
                            "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                            "traffic": profiled_traffic("bwd_tc" if tc else "bwd", w.name),
                            "algorithmic_bytes": nbytes,
                            "kernel": ("fwd_prep_kernel + fwd_rec_kernel (save) + "
                                       "bwd_chain_kernel + bwd_grad_kernel") if tc
                            else "bwd_simt_kernel + bwd_reduce_kernel"},
               "impl": "tc" if tc else "simt",
               # tensor cores: prep, recurrence (save), chain, gradients (with
               # segment ids also the run builder and the padding zero-fill);
               # CUDA cores: (runs +) the backward kernel + the reduction
               "gpu_launches": steps * ((6 if has_seg else 4) if tc else (3 if has_seg else 2))}
        if tc:
            # a training step without repeated work: the forward that saves
            # (kda_chunk_fwd_save), then the backward on its saves
            # (kda_chunk_bwd_from_saved); each timed alone and as the pair
            tws = torch.zeros(kda.fwd_save_workspace_size(w.B, w.T, w.H, w.K, w.V, d["q"].dtype,
                                                          has_seg),
                              dtype=torch.uint8, device=dev)

            def fwd_save():
                kda.chunk_fwd_save(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                                   initial_state=d["initial_state"],
                                   segment_ids=d["segment_ids"], workspace=tws, stream=stream)

            def bwd_saved():
                kda.chunk_bwd_from_saved(d["q"], d["k"], d["v"], d["g"], d["beta"], d_o, tws,
                                         scale=x["scale"], initial_state=d["initial_state"],
                                         segment_ids=d["segment_ids"], d_final=d_f,
                                         stream=stream)

            def pair():
                fwd_save()
                bwd_saved()

            t_f, _ = time_steps(fwd_save, steps, args.warmup, stream, flush, dist, clocks)
            t_b, _ = time_steps(bwd_saved, steps, args.warmup, stream, flush, dist, clocks)
            t_p, _ = time_steps(pair, steps, args.warmup, stream, flush, dist, clocks)
            ms_p = dist.max(statistics.mean(t_p))
            res["training_step"] = {
                "fwd_save_ms": dist.max(statistics.mean(t_f)),
                "bwd_from_saved_ms": dist.max(statistics.mean(t_b)),
                "ms_per_step": ms_p, "unit": "tokens/s",
                "value": whole_job_value(dist.world, w.B * w.T, ms_p),
                "note": "forward (o, final state, saves) + backward from the saves; "
                        "against the separate forward and backward calls",
                # fwd_save: prep + recurrence; bwd_from_saved: chain + gradients,
                # each alone and as the pair (with segment ids also the run
                # builder in both and the padding zero-fill in the backward)
                "gpu_launches": steps * (14 if has_seg else 8)}
            res["gpu_launches"] += res["training_step"]["gpu_launches"]
        if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline_backward(w, args.seed, budget_s=args.cpu_seconds / 2)
        return res

    def measure_scan(wname):
        """The forward as a chunk-parallel state scan (kda_chunk_fwd_scan,
        automatic segment count) beside the split path, on one workload."""
        w = ki.WORKLOADS[wname]
        x = ki.make_inputs(w, seed=rank_seed(w))
        d = device_inputs(x, dev)
        o = torch.empty(w.B, w.T, w.H, w.V, dtype=d["q"].dtype, device=dev)
        fs = torch.empty(w.B, w.H, w.K, w.V, dtype=torch.float32, device=dev)
        ws_scan = torch.zeros(kda.scan_workspace_size(w.B, w.T, w.H, w.K, w.V, d["q"].dtype),
                              dtype=torch.uint8, device=dev)
        ws_split = kda.alloc_workspace(w.B, w.T, w.H, w.K, w.V, d["q"].dtype, False, dev,
                                       impl="split")

        def scan():
            kda.chunk_fwd_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                               initial_state=d["initial_state"], output_final_state=True,
                               out=o, final_state_out=fs, workspace=ws_scan, stream=stream)

        def split():
            kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                          initial_state=d["initial_state"], output_final_state=True, out=o,
                          final_state_out=fs, workspace=ws_split, impl="split", stream=stream)

        steps = min(args.steps, 50)
        t_scan, _ = time_steps(scan, steps, args.warmup, stream, flush, dist, clocks)
        if kda.read_device_status(ws_scan):
            raise RuntimeError("device status bits after the scan steps")
        t_split, _ = time_steps(split, steps, args.warmup, stream, flush, dist, clocks)
        ms_scan = dist.max(statistics.mean(t_scan))
        ms_split = dist.max(statistics.mean(t_split))
        tokens = w.B * w.T
        return {"workload": w.name, "ms_per_step": ms_scan, "unit": "tokens/s",
                "value": whole_job_value(dist.world, tokens, ms_scan),
                "split_ms_per_step": ms_split,
                "split_value": whole_job_value(dist.world, tokens, ms_split),
                "segments": kda_scan_segments(w),
                # prep, map pass, combine, finish pass (+ split: prep, rec)
                "gpu_launches": steps * (4 + 2)}

    def kda_scan_segments(w):
        return kda.scan_segments(w.B, w.T, w.H, w.K, w.V)

    def packed_launches(w):
        """Kernels one packed forward launches: segment runs (with the chunk
        coordinates), prep, recurrence (+ the fused kernel AUTO enqueues
        gated on an overflow of the split items); 2 on the one-kernel paths."""
        if kernel_impl(w) == "split":
            return 4 if args.kda_impl == "auto" else 3
        return 2

    def kernel_impl(w):
        import gated_delta_rule_21_gb300 as kda
        dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        has_seg = w.segments is not None
        if args.kda_impl in ("simt", "tc", "split"):
            return args.kda_impl
        if kda.impl_available("split", w.B, w.T, w.H, w.K, w.V, dt):
            return "split"
        return "tc" if kda.impl_available("tc", w.B, w.T, w.H, w.K, w.V, dt) else "simt"

    clocks.start()
    head = measure(args.workload, with_e2e=not args.no_e2e, clocks_=clocks)
    packed = (measure(PACKED, with_e2e=False, clocks_=clocks)
              if args.workload == HEADLINE and not args.no_packed else None)
    prologue = (measure_prologue(PROLOGUE)
                if args.workload == HEADLINE and not args.no_prologue else None)
    scan = ([measure_scan(n) for n in (HEADLINE, LONG_FEW_HEADS)]
            if args.workload == HEADLINE and not args.no_scan else None)
    backward = (measure_backward(args.workload)
                if not args.no_backward and kda.bwd_workspace_size(
                    1, 64, 1, ki.WORKLOADS[args.workload].K, ki.WORKLOADS[args.workload].V) > 0
                else None)
    clk = clocks.stop()

    w = head["workload"]
    value = whole_job_value(dist.world, head["tokens"], head["ms_max"])
    impl_used = kernel_impl(w)
    launches_per_step = (2 if impl_used == "split" else 1) + (1 if head["has_seg"] else 0)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_max"],
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (value / (w.B * w.T / (PAGES_TPU_FIXED_MS * 1e-3))
                        if args.workload == HEADLINE else None),
        "vs_baseline_ref": "pages' TPU v7x tokamax #19 fixed forward, 1.870 ms (other hardware; context)",
        "dtype": "bf16" if impl_used in ("tc", "split") else "f32",
        "data": "synthetic (seeded; shapes and distributions of the pages' workloads)",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "K": w.K, "V": w.V,
                   "qkv_dtype": w.dtype, "chunk": CHUNK, "initial_state": w.init_state_std is not None,
                   "output_final_state": True, "impl": impl_used,
                   "l2": "flushed: 256 MiB write between timed steps",
                   "parallelism": (f"heads sharded: {w.H * dist.world} heads, {w.H} per rank "
                                   f"on {dist.world} ranks, no data exchange"
                                   if dist.world > 1 else "one GPU"),
                   "ms_median": head["ms_median"], "ms_min": head["ms_min"]},
        "roofline": roofline(head),
        "e2e": head.get("e2e"),
        "clocks": clk,
        "gpu_launches": launches_per_step * args.steps,
    }
    if packed is not None:
        pw = packed["workload"]
        line["packed"] = {"workload": pw.name, "ms_per_step": packed["ms_max"],
                          "value": whole_job_value(dist.world, packed["tokens"], packed["ms_max"]),
                          "unit": "tokens/s", "roofline": roofline(packed),
                          "vs_pages_tpu": (packed["tokens"] / (packed["ms_max"] * 1e-3))
                          / (pw.B * pw.T / (PAGES_TPU_PACKED_MS * 1e-3)),
                          # run builder (+ the chunk table for the split path), then
                          "gpu_launches": packed_launches(pw) * args.steps}
        line["gpu_launches"] += line["packed"]["gpu_launches"]
    if prologue is not None:
        line["prologue"] = prologue
        line["gpu_launches"] += prologue["gpu_launches"]
    if scan is not None:
        line["scan"] = scan
        line["gpu_launches"] += sum(x["gpu_launches"] for x in scan)
    if backward is not None:
        line["backward"] = backward
        line["gpu_launches"] += backward["gpu_launches"]
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.seed, budget_s=args.cpu_seconds)
    return line


# ----------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ----------------------------------------------------------------------------
def oracle_sample(w, seed, heads):
    """The first ``heads`` heads of the workload, as the oracle's fp64 input."""
    import oracle
    x = ki.make_inputs(w, seed=seed)
    sl = slice(0, heads)
    arrs = [oracle._f64(x[n][:, :, sl]) for n in ("q", "k", "v", "g", "beta")]
    s0 = x["initial_state"]
    s0 = None if s0 is None else oracle._f64(s0[:, sl])
    seg = x["segment_ids"]
    return arrs, s0, seg, x["scale"]


def cpu_baseline(w, seed, budget_s=10.0):
    import oracle
    cores = oracle.default_threads()
    heads = min(w.H, cores)
    arrs, s0, seg, scale = oracle_sample(w, seed, heads)
    runs, t_total = 0, 0.0
    while t_total < budget_s and runs < 100:
        t = time.perf_counter()
        oracle.kda_forward(*arrs, scale, initial_state=s0, segment_ids=seg, threads=cores)
        t_total += time.perf_counter() - t
        runs += 1
    per_run = t_total / runs
    tokens_equiv = w.B * w.T * heads / w.H
    # and on one thread, the whole B1 H8 T1024 fixed workload
    w1 = ki.WORKLOADS["fixed_bf16_h8_t1024"]
    a1, s1, seg1, scale1 = oracle_sample(w1, seed, w1.H)
    t = time.perf_counter()
    oracle.kda_forward(*a1, scale1, initial_state=s1, segment_ids=seg1, threads=1)
    t1 = time.perf_counter() - t
    return {"value": tokens_equiv / per_run, "unit": "tokens/s", "cores": min(cores, w.B * heads),
            "host_cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{heads} of {w.H} heads x {w.B * w.T} tokens (fp64 token recurrence), "
                      f"{runs} runs, {t_total:.1f} s; tokens/s scaled by heads/H",
            "one_thread": {"workload": w1.name, "ms": round(t1 * 1e3, 1),
                           "value": w1.B * w1.T / t1, "unit": "tokens/s", "threads": 1}}


def cpu_baseline_backward(w, seed, budget_s=5.0):
    """The fp64 backward oracle on a head sample of the workload."""
    import oracle
    cores = oracle.default_threads()
    heads = min(w.H, cores)
    arrs, s0, seg, scale = oracle_sample(w, seed, heads)
    u = ki.make_upstream_grads(w, seed=seed)
    d_o = oracle._f64(u["d_o"][:, :, :heads])
    d_f = oracle._f64(u["d_final"][:, :heads])
    runs, t_total = 0, 0.0
    while t_total < budget_s and runs < 100:
        t = time.perf_counter()
        oracle.kda_backward(*arrs, scale, initial_state=s0, segment_ids=seg, d_o=d_o,
                            d_final=d_f, threads=cores)
        t_total += time.perf_counter() - t
        runs += 1
    per_run = t_total / runs
    return {"value": w.B * w.T * heads / w.H / per_run, "unit": "tokens/s",
            "cores": min(cores, w.B * heads), "kind": "oracle",
            "sample": f"{heads} of {w.H} heads x {w.B * w.T} tokens (fp64 reverse-mode token "
                      f"recurrence), {runs} runs, {t_total:.1f} s; tokens/s scaled by heads/H"}


def run_reference(args, dist):
    """The oracle as the reference program, on the host cores."""
    import oracle
    w = ki.WORKLOADS[args.workload]
    cores = oracle.default_threads()
    heads = min(w.H, cores)
    arrs, s0, seg, scale = oracle_sample(w, args.seed, heads)
    fn = lambda: oracle.kda_forward(*arrs, scale, initial_state=s0, segment_ids=seg,  # noqa: E731
                                    threads=cores)
    for _ in range(args.warmup):
        fn()
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        fn()
        times.append(time.perf_counter() - t)
    ms = statistics.mean(times) * 1e3
    tokens_equiv = w.B * w.T * heads / w.H
    value = tokens_equiv / (ms * 1e-3)
    sample = (f"{heads} of {w.H} heads x {w.B * w.T} tokens per step (fp64 token "
              f"recurrence); tokens/s scaled by heads/H")
    return {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "K": w.K, "V": w.V},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": min(cores, w.B * heads),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(ki.WORKLOADS))
    ap.add_argument("--kda-impl", default="auto", choices=["auto", "simt", "tc"])
    ap.add_argument("--v-tile", type=int, default=0)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer e2e leg")
    ap.add_argument("--no-packed", action="store_true", help="skip the packed N=25 leg")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward leg")
    ap.add_argument("--no-scan", action="store_true",
                    help="skip the chunk-parallel scan leg (headline and long-context shapes)")
    ap.add_argument("--no-prologue", action="store_true",
                    help="skip the conv prologue leg (packed N=25 shape)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return 0
        dist = Dist.__new__(Dist)
        dist.rank, dist.world, dist.local_rank, dist.pg = 0, int(os.environ.get("WORLD_SIZE", "1")), 0, None
        print(json.dumps(run_reference(args, dist)))
        return 0

    dist = Dist()
    try:
        line = run_ours(args, dist)
        if dist.rank == 0:
            print(json.dumps(line))
    finally:
        dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
