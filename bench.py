#!/usr/bin/env python
"""Benchmark: MLA decode over a paged latent cache, DeepSeek-V3 shapes.

One step = one pass of the whole decode path over one batch: append this step's
new token of every sequence into the paged cache, then decode attention for
all sequences (split schedule, attention kernel, split combine, W_UV
up-projection). The workload: B=32, q_len=1, H=128, kv_lora_rank=512,
qk_rope_head_dim=64, v_head_dim=128, per-sequence lengths ~ U[1024, 8192],
block size 64 with a permuted block table, bf16. The new token written each
step is the sequence's last position, so the cache (and the work) is identical
every step.

Prints one JSON line (rank 0). ``--impl reference`` times the CPU oracle on the
host cores instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode KV-tokens/s, TFLOP/s and HBM GB/s as fraction of GB300 roofline"
UNIT = "KV-tokens/s"
L2_FLUSH_BYTES = 512 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--configs", action="store_true",
                    help="time the other workloads only (one JSON line each) instead of the bench step")
    ap.add_argument("--no-configs", action="store_true", help="leave the per-workload record out of the bench line")
    ap.add_argument("--only", default="", help="with --configs: comma-separated workload keys (e.g. C3,C4)")
    ap.add_argument("--reps", type=int, default=0, help="with --configs: timed calls per workload (0: defaults)")
    return ap.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(values, world, device=None):
    """Each timing's maximum over the ranks: the slowest rank sets the job's time."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_throughput(tokens_per_rank, world, step_ms):
    """Whole-job KV-tokens/s: every rank decodes its own copy of the workload (weak
    scaling), all within the slowest rank's step time."""
    return tokens_per_rank * world / (step_ms * 1e-3)


# ------------------------------------------------------------------ accounting

def workload_config(w):
    return {
        "workload": (f"DeepSeek-V3-shaped MLA decode: B={w.B} q_len=1 H={w.H} kv_lora_rank={w.r} "
                     f"qk_rope_head_dim={w.d_rope} v_head_dim={w.d_v} L~U[1024,8192] (sum {w.total_tokens}) "
                     f"block_size={w.block_size} permuted block table, bf16"),
        "global_batch": w.B,
        "seq_len_sum": w.total_tokens,
        "seq_len_mean": round(w.total_tokens / w.B, 1),
        "cache_bytes": w.total_tokens * w.D * 2,
        "l2": "flushed between timed steps (512 MiB write)",
    }


def algorithmic(w):
    """Algorithmic bytes and flops of one decode step and of its attention kernel."""
    tok = w.total_tokens
    H, r, D, dv, B = w.H, w.r, w.D, w.d_v, w.B
    kernel_bytes = tok * D * 2 + B * H * D * 2                 # cache read once + absorbed query
    step_bytes = (kernel_bytes + H * r * dv * 2                # W_UV
                  + B * H * dv * 2 + B * H * 4                 # out + lse
                  + B * D * 2 * 2)                             # appended token: read + write
    kernel_flops = 2 * tok * H * (D + r)                       # QK^T + PV
    step_flops = kernel_flops + 2 * B * H * r * dv             # + W_UV up-projection
    return kernel_bytes, step_bytes, kernel_flops, step_flops


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            flat = {}

            def walk(x, pre=""):
                if isinstance(x, dict):
                    for k, v in x.items():
                        walk(v, f"{pre}{k}.")
                elif isinstance(x, (int, float)):
                    flat[pre[:-1]] = float(x)
            walk(d)

            def pick(*names):
                for k, v in flat.items():
                    if k.split(".")[-1] in names:
                        return v
                return None
            hbm = pick("hbm_gbs", "hbm_GBs", "copy_gbs")
            tf = pick("bf16_tflops", "bf16_tflops_burst")
            tfs = pick("bf16_tflops_sustained")
            if hbm and tf:
                return {"hbm_gbs": hbm, "bf16_tflops": tf, "bf16_tflops_sustained": tfs or tf,
                        "source": "measured"}
        except Exception:
            pass
    return dict(FALLBACK_PEAKS, source="fallback")


# the files that define the bf16 tensor-core decode kernel (its DRAM counters are
# recorded against their hash; host-side changes elsewhere do not invalidate them)
KERNEL_SOURCES = ("mla_wide.cu", "mla_ptx.cuh", "mla_internal.cuh")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_latent_kv_08_gb300", "csrc")
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash()
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        kv = dict(x.split("=", 1) for x in line.split())
        if kv.get("kernel") == kernel and kv.get("source_sha") == src:
            return float(kv["bytes_per_launch_full_workload"])
    return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling, timestamped, so that the samples
    of each measured window (the timed steps, the other legs) can be summarised."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0, interval_ms=20):
        self.samples = []          # (host time, fields)
        self.proc = None
        self.dev = device_index
        self.interval_ms = interval_ms

    def start(self):
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", str(self.interval_ms)]
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            first = vis.split(",")[0].strip() if vis else str(self.dev)
            if first:
                cmd += ["-i", first]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.perf_counter(), parts))

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()

    def summary(self, t0=None, t1=None, slack=0.06):
        """Median SM clock, max clock, power and the throttle reasons seen between t0
        and t1 (host perf_counter seconds; widened by `slack` on both sides so that a
        short window still holds the samples taken while it ran)."""
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, pw, reasons = [], [], [], set()
        for ts, p in self.samples:
            if t0 is not None and (ts < t0 - slack or ts > t1 + slack):
                continue
            try:
                sm.append(float(p[0]))
                mx.append(float(p[1]))
                pw.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(pw) if pw else None}


def cpu_model():
    """The host CPU's model name (lscpu, then /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


# ------------------------------------------------------------------ oracle arm

def oracle_throughput(w, budget_s, max_tokens_per_call=None):
    """Time the CPU oracle over sequences of the workload until ``budget_s`` of
    work is done. Returns (tokens/s, tokens, seconds, description)."""
    from oracle import attention
    done_tok, t_total, calls = 0, 0.0, 0
    b = 0
    while t_total < budget_s or calls == 0:
        L = w.latent[b].shape[0] if max_tokens_per_call is None else min(max_tokens_per_call, w.latent[b].shape[0])
        t0 = time.perf_counter()
        attention.absorbed(w.q[b], w.latent[b][:L], w.rope[b][:L], w.W_UV, w.scale)
        t_total += time.perf_counter() - t0
        done_tok += L
        calls += 1
        b = (b + 1) % w.B
    return done_tok / t_total, done_tok, t_total, calls


def cpu_threads():
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(k, "").isdigit():
            return int(os.environ[k])
    return os.cpu_count() or 1


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import workloads
    w = workloads.dsv3(args.seed)
    # size each step so the whole run stays within about two minutes
    rate, _, _, _ = oracle_throughput(w, 2.0, max_tokens_per_call=2048)
    per_step = int(max(64, min(8192, rate * 120.0 / max(1, args.steps + args.warmup))))
    from oracle import attention
    for k in range(args.warmup):
        b = k % w.B
        n = min(per_step, w.latent[b].shape[0])
        attention.absorbed(w.q[b], w.latent[b][:n], w.rope[b][:n], w.W_UV, w.scale)
    tok, t = 0, 0.0
    for k in range(args.steps):
        b = k % w.B
        n = min(per_step, w.latent[b].shape[0])
        t0 = time.perf_counter()
        attention.absorbed(w.q[b], w.latent[b][:n], w.rope[b][:n], w.W_UV, w.scale)
        t += time.perf_counter() - t0
        tok += n
    value = tok / t
    sample = (f"each step: absorbed attention of one sequence's first <= {per_step} cached tokens, "
              f"all {w.H} heads, fp64 numpy (cycling over the {w.B} sequences)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm

def run_gb300(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    from mla_latent_kv_08_gb300 import build as _build
    if rank == 0:
        _build.build()
    if world > 1:
        dist.barrier()
    import mla_latent_kv_08_gb300 as mla
    import workloads

    dev = torch.device("cuda", local)
    w = workloads.dsv3(args.seed)
    shape = mla.Shape(num_heads=w.H, kv_lora_rank=w.r, rope_dim=w.d_rope, v_head_dim=w.d_v,
                      block_size=w.block_size, num_blocks=w.num_blocks, kind=mla.MLA_KV_BF16)
    bf = torch.bfloat16

    def t(x, dtype=None):
        tt = torch.from_numpy(np.ascontiguousarray(x))
        return (tt.to(dtype) if dtype is not None else tt).to(dev)

    cache = mla.Cache.allocate(shape, dev)
    bt = t(w.block_table)
    seq_lens = t(w.seq_lens.astype(np.int32))
    # fill the cache (untimed) through the library's append
    cu_all = t(np.concatenate([[0], np.cumsum(w.seq_lens)]).astype(np.int32))
    mla.mla_latent_append(cache, bt, t(np.zeros(w.B, np.int32)), cu_all,
                          t(np.concatenate(w.latent), bf), t(np.concatenate(w.rope), bf))
    # per-step inputs: the last token of each sequence (rewritten every step) and q
    new_c = t(np.stack([x[-1] for x in w.latent]), bf)
    new_r = t(np.stack([x[-1] for x in w.rope]), bf)
    start = t((w.seq_lens - 1).astype(np.int32))
    cu1 = t(np.arange(w.B + 1, dtype=np.int32))
    q = t(w.q, bf)
    W_UV = t(w.W_UV, bf)
    out = torch.empty((w.B, 1, w.H, w.d_v), dtype=bf, device=dev)
    lse = torch.empty((w.B, 1, w.H), dtype=torch.float32, device=dev)
    ws = mla.alloc_workspace(shape, w.B, 1, dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # one step: this step's new token of every sequence appended, then the decode, in
    # one call (mla_append_decode: the copy rides on the planner's launch)
    def step(qq=q, cc=new_c, rr=new_r):
        mla.mla_append_decode(cache, bt, start, cu1, cc, rr, seq_lens, qq, W_UV, w.scale, out, lse, ws,
                              stream=stream)

    # clocks are sampled from the warm-up on, through every leg; each leg's window is
    # summarised on its own
    sampler = ClockSampler(local)
    sampler.start()
    windows = {}
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    code, flags = mla.mla_get_status(ws)
    if code != mla.MLA_OK:
        raise RuntimeError(f"device status {code} flags {flags}")

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_a = time.perf_counter()
    mla.mla_profile_enable(2)          # launch counting only in this loop (no events)
    for k in range(K):
        flush.zero_()
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    windows["timed_steps"] = (t_a, time.perf_counter())
    if world > 1:
        dist.barrier()
    _, _, n_kernels = mla.mla_profile_read()
    step_ms = sum(a.elapsed_time(b) for a, b in ev) / K
    # the same steps, untimed, for about 0.4 s: the clock record of this load when the
    # timed region is shorter than a few sampling periods
    t_a = time.perf_counter()
    while time.perf_counter() - t_a < 0.4:
        for _ in range(50):
            flush.zero_()
            step()
        torch.cuda.synchronize(dev)
    windows["soak"] = (t_a, time.perf_counter())
    # the attention kernel's own duration, in separate steps: the library's event pair
    # around it would otherwise sit between the kernels of the timed steps
    t_a = time.perf_counter()
    mla.mla_profile_enable(1)
    for k in range(max(20, K // 4)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    att_ms, att_n, _ = mla.mla_profile_read()
    mla.mla_profile_enable(False)
    att_avg_ms = att_ms / max(att_n, 1)
    windows["roofline"] = (t_a, time.perf_counter())

    e2e = None
    if not args.no_e2e:
        # The step's inputs (query, new latents, new rope keys) sit in one pinned host
        # buffer and one device buffer, and its results (out, lse) in one device buffer
        # read back into one pinned buffer: one copy each way per step, as a caller
        # would lay them out. Tensors are views at 256-byte-aligned offsets.
        def packed(parts, device, pin):
            offs, n = [], 0
            for t in parts:
                offs.append(n)
                n += (t.numel() * t.element_size() + 255) // 256 * 256
            raw = torch.empty(n, dtype=torch.uint8, device=device)
            if pin:
                raw = raw.pin_memory()
            views = [raw[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, parts)]
            return raw, views
        q_host = torch.from_numpy(np.ascontiguousarray(w.q)).to(bf)
        hin, (hq, hc, hr) = packed([q_host, new_c, new_r], "cpu", True)
        hq.copy_(q_host)
        hc.copy_(new_c.cpu())
        hr.copy_(new_r.cpu())
        din, (q_d, c_d, r_d) = packed([q, new_c, new_r], dev, False)
        dres, (out_d, lse_d) = packed([out, lse], dev, False)
        hres = torch.empty(dres.shape, dtype=torch.uint8).pin_memory()

        def e2e_step(st):
            din.copy_(hin, non_blocking=True)
            mla.mla_append_decode(cache, bt, start, cu1, c_d, r_d, seq_lens, q_d, W_UV, w.scale, out_d, lse_d, ws,
                                  stream=st)
            hres.copy_(dres, non_blocking=True)

        # The whole step (copies from and to pinned host memory, append, decode) is
        # captured once as a CUDA graph and replayed: its copies read and write the
        # host buffers at every replay, and the host issues one launch per step, so
        # the timed region holds the device work and the transfers, not the Python
        # overhead of seven calls. If capture fails, the step runs eagerly.
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        graph = None
        with torch.cuda.stream(side):
            for _ in range(max(3, args.warmup // 4)):
                e2e_step(side)
        side.synchronize()
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                e2e_step(side)
            torch.cuda.synchronize(dev)
        except Exception as exc:   # noqa: BLE001 - fall back to eager launches
            print(f"e2e: graph capture failed ({exc}); timing eager launches", file=sys.stderr)
            graph = None
            torch.cuda.synchronize(dev)

        def e2e_run():
            if graph is not None:
                graph.replay()
            else:
                with torch.cuda.stream(stream):
                    e2e_step(stream)

        for _ in range(3):
            e2e_run()
        torch.cuda.synchronize(dev)
        ke = max(20, K)
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(ke)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t_a = time.perf_counter()
        for k in range(ke):
            flush.zero_()
            ev2[k][0].record(stream)
            e2e_run()
            ev2[k][1].record(stream)
        torch.cuda.synchronize(dev)
        windows["e2e"] = (t_a, time.perf_counter())
        e2e_ms = sum(a.elapsed_time(b) for a, b in ev2) / ke
        code, flags = mla.mla_get_status(ws)
        if code != mla.MLA_OK:
            raise RuntimeError(f"device status {code} flags {flags} after the end-to-end steps")
        h2d = hin.numel()
        d2h = hres.numel()
        e2e = {"ms": e2e_ms, "h2d": h2d, "d2h": d2h,
               "mode": "CUDA graph replay" if graph is not None else "eager launches"}
        # Overlapped variant: the inputs of step k + 1 are uploaded (on a second stream)
        # while step k computes, into the other of two device buffers; step k's
        # result is read back as before. One graph per buffer parity; the timed region
        # starts with the upload of step 0's inputs, so every step's copies are in it.
        if graph is not None:
            try:
                bufs = [packed([q, new_c, new_r], dev, False) for _ in range(2)]
                cstream = torch.cuda.Stream(dev)

                def upload(buf, st):
                    with torch.cuda.stream(st):
                        buf[0].copy_(hin, non_blocking=True)

                def overlapped_step(par):
                    cur, nxt = bufs[par], bufs[1 - par]
                    cstream.wait_stream(side)           # fork the copy branch off the step
                    upload(nxt, cstream)
                    qv, cv, rv = cur[1]
                    mla.mla_append_decode(cache, bt, start, cu1, cv, rv, seq_lens, qv, W_UV, w.scale, out_d, lse_d,
                                          ws, stream=side)
                    hres.copy_(dres, non_blocking=True)
                    side.wait_stream(cstream)           # join: the next inputs have landed

                graphs = []
                for par in range(2):
                    side.wait_stream(stream)
                    with torch.cuda.stream(side):
                        overlapped_step(par)
                    side.synchronize()
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=side):
                        overlapped_step(par)
                    torch.cuda.synchronize(dev)
                    graphs.append(g)
                upload(bufs[0], stream)
                for k in range(4):
                    graphs[k & 1].replay()
                torch.cuda.synchronize(dev)
                ev3 = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
                torch.cuda.synchronize(dev)
                ev3[0].record(stream)
                upload(bufs[0], stream)
                for k in range(ke):
                    graphs[k & 1].replay()
                ev3[1].record(stream)
                torch.cuda.synchronize(dev)
                e2e["overlapped_ms"] = ev3[0].elapsed_time(ev3[1]) / ke
                e2e["overlapped_note"] = ("inputs of step k+1 uploaded on a second stream during step k, two "
                                          "device buffers; L2 not flushed between these steps")
                code, flags = mla.mla_get_status(ws)
                if code != mla.MLA_OK:
                    raise RuntimeError(f"device status {code} flags {flags} after the overlapped steps")
            except RuntimeError:
                raise
            except Exception as exc:   # noqa: BLE001 - the serial number stands alone
                print(f"e2e: overlapped variant not measured ({exc})", file=sys.stderr)

    if world > 1:
        step_ms, att_avg_ms, e2e_max = max_over_ranks([step_ms, att_avg_ms, e2e["ms"] if e2e else 0.0], world, dev)
        if e2e:
            e2e["ms"] = e2e_max

    if rank != 0:
        sampler.stop()
        if world > 1:
            dist.destroy_process_group()
        return 0

    kb, sb, kf, sf = algorithmic(w)
    peaks = load_peaks()
    tokens = w.total_tokens * world
    value = job_throughput(w.total_tokens, world, step_ms)
    achieved = kb / (att_avg_ms * 1e-3) / 1e9
    kernel_name = {mla.MLA_IMPL_SIMT: "decode_simt_kernel", mla.MLA_IMPL_TCGEN05: "decode_wide_kernel"}[
        mla.mla_resolve_impl(shape, 1)]
    configs = None
    if not args.no_configs:
        t_a = time.perf_counter()
        configs = measure_configs(mla, dev, peaks, flush)
        windows["configs"] = (t_a, time.perf_counter())
    sampler.stop()
    clocks = sampler.summary(*windows["timed_steps"])
    clock_legs = {k: sampler.summary(*v) for k, v in windows.items() if k != "timed_steps"}
    cpu = None
    if not args.no_cpu_baseline:
        rate, tok, secs, calls = oracle_throughput(w, 12.0)
        cpu = {"value": rate, "unit": UNIT, "cores": cpu_threads(), "cpu_model": cpu_model(), "kind": "oracle",
               "sample": f"{calls} whole sequences of this workload ({tok} cached tokens, all heads), "
                         f"fp64 numpy, {secs:.1f} s"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded numpy PCG64)",
        "config": dict(workload_config(w), parallelism=f"replica x{world} (independent sequences)"),
        "tflops": sf / (step_ms * 1e-3) / 1e12 * world,
        "gbs": sb / (step_ms * 1e-3) / 1e9 * world,
        # whole step against min(HBM bound, tensor bound): roofline time / measured time
        "step_roofline_frac": max(sb / (peaks["hbm_gbs"] * 1e9),
                                  sf / (peaks["bf16_tflops_sustained"] * 1e12)) / (step_ms * 1e-3),
        "arithmetic_intensity": sf / sb,
        "roofline": {"kernel": kernel_name, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": recorded_traffic(kernel_name),
                     "algorithmic_bytes": kb, "launch_ms": att_avg_ms,
                     "peak_source": peaks["source"],
                     "tensor_tflops": kf / (att_avg_ms * 1e-3) / 1e12},
        "gpu_launches": int(n_kernels),
        "clocks": clocks,
        "clocks_legs": clock_legs,
        "cpu_baseline": cpu,
    }
    if e2e:
        line["e2e"] = {"value": tokens / (e2e["ms"] * 1e-3), "unit": UNIT, "h2d_bytes_per_step": e2e["h2d"],
                       "d2h_bytes_per_step": e2e["d2h"], "ms_per_step": e2e["ms"], "launch": e2e["mode"]}
        if "overlapped_ms" in e2e:
            line["e2e"]["overlapped"] = {"value": tokens / (e2e["overlapped_ms"] * 1e-3),
                                         "ms_per_step": e2e["overlapped_ms"], "note": e2e["overlapped_note"]}
    if configs is not None:
        line["configs"] = configs
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def measure_configs(mla, dev, peaks, flush, only=(), reps=0):
    """The other workloads of the parity suite, each timed as whole calls (plan,
    attention kernel, combine; INT2: and the query rotation) and its attention kernel
    alone in separate calls (the library's event pair around it), L2 flushed before
    every call. Each entry: algorithmic bytes (cache read once + the query) and flops
    (QK^T + PV) of the attention kernel, their ratio, the bound it implies against the
    measured peaks (burst figures: every kernel here is timed alone) and the
    fraction reached. The rotated-INT2 workloads are calibrated with the library's
    own calibration; their up-projection is folded (MLA_FLAG_WUV_FOLDED)."""
    import numpy as np
    import torch
    import workloads
    bf = torch.bfloat16
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    res = {}

    def t(x, dtype=None):
        tt = torch.from_numpy(np.ascontiguousarray(x))
        return (tt.to(dtype) if dtype is not None else tt).to(dev)

    def timed(fn, n):
        """Device time of fn: captured once as a CUDA graph, replayed n times right
        after an L2 flush, so that the host's launch latency is not in the number."""
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            fn()
        side.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            fn()
        torch.cuda.synchronize(dev)
        tot = 0.0
        for _ in range(n):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize(dev)
            tot += e0.elapsed_time(e1)
        return tot / n

    def run(key, desc, w, kind, q_len, R=None, T=None, n=20, fold=False, append=False, q_rotated=False):
        if only and key not in only:
            return
        if reps:
            n = reps
        shape = mla.Shape(num_heads=w.H, kv_lora_rank=w.r, rope_dim=w.d_rope, v_head_dim=w.d_v,
                          block_size=w.block_size, num_blocks=w.num_blocks, kind=kind,
                          flags=(mla.MLA_FLAG_WUV_FOLDED if fold else 0) | (mla.MLA_FLAG_Q_ROTATED if q_rotated else 0))
        cache = mla.Cache.allocate(shape, dev)
        cu = t(np.concatenate([[0], np.cumsum(w.seq_lens)]).astype(np.int32))
        Rd = None if R is None else t(R.astype(np.float32))
        Td = None if T is None else t(T.astype(np.float32))
        bt, sl = t(w.block_table), t(w.seq_lens.astype(np.int32))
        mla.mla_latent_append(cache, bt, t(np.zeros(w.B, np.int32)), cu, t(np.concatenate(w.latent), bf),
                              t(np.concatenate(w.rope), bf), R=Rd, clip=Td)
        entry = {"workload": desc}
        if append:
            # the workload's 1024 appended tokens (32 per sequence) rotated and quantised
            nc, nr = t(np.concatenate(w.new_latent), bf), t(np.concatenate(w.new_rope), bf)
            cun = t(np.arange(0, 32 * w.B + 1, 32, dtype=np.int32))
            sp = t(w.start_pos.astype(np.int32))
            app_ms = timed(lambda: mla.mla_latent_append(cache, bt, sp, cun, nc, nr, R=Rd, clip=Td), n)
            entry_note = "device time of one call, captured as a CUDA graph and replayed after an L2 flush"
            D = w.r + w.d_rope
            qd = D if kind == mla.MLA_KV_INT2_JOINT else w.r
            abytes = (int(nc.numel()) + int(nr.numel())) * 2 + int(nc.shape[0]) * cache.bytes_per_token() + qd * qd * 4
            entry["append"] = {"tokens": int(nc.shape[0]), "us": app_ms * 1e3, "timing": entry_note,
                               "algorithmic_bytes": abytes, "GBs": abytes / (app_ms * 1e-3) / 1e9}
        q, W = t(w.q, bf), t(w.W_UV, bf)
        if fold:                    # once per layer: W'_UV = R^T . W_UV
            Wf = torch.empty_like(W)
            mla.mla_fold_rotation(shape, Rd, W, Wf)
            W = Wf
        Rcall = Rd
        if q_rotated:
            # the caller's query projection carries R (folded once, like W_UV): its
            # latent dims arrive as bf16(q_lat . R), and R is not passed at all
            qf = t(w.q)
            qf[..., :w.r] = qf[..., :w.r] @ Rd
            q = qf.to(bf)
            Rcall = None
        out = torch.empty((w.B, q_len, w.H, w.d_v), dtype=bf, device=dev)
        lse = torch.empty((w.B, q_len, w.H), dtype=torch.float32, device=dev)
        ws = mla.alloc_workspace(shape, w.B, q_len, dev)
        call = mla.mla_decode if q_len == 1 else mla.mla_verify
        go = lambda: call(cache, bt, sl, q, W, w.scale, out, lse, ws, R=Rcall)   # noqa: E731
        for _ in range(3):
            go()
        torch.cuda.synchronize(dev)
        call_ms = timed(go, n)
        mla.mla_profile_enable(1)
        for _ in range(n):
            flush.zero_()
            go()
        torch.cuda.synchronize(dev)
        ms, na, _ = mla.mla_profile_read()
        mla.mla_profile_enable(0)
        code, flags = mla.mla_get_status(ws)
        tok = int(w.seq_lens.sum())
        D = w.r + w.d_rope
        kb = tok * cache.bytes_per_token() + w.B * q_len * w.H * D * 2
        kf = 2 * tok * q_len * w.H * (D + w.r)
        att = ms / max(na, 1)
        ai = kf / kb
        bound = "tensor" if ai > ridge else "hbm"
        gbs, tfs = kb / (att * 1e-3) / 1e9, kf / (att * 1e-3) / 1e12
        entry.update({
            "tokens": tok, "q_len": q_len, "impl": "tcgen05" if mla.mla_resolve_impl(shape, q_len) == 2 else "simt",
            "call_us": call_ms * 1e3, "call_timing": "device time of one call (CUDA graph replay after an L2 flush)",
            "attention_us": att * 1e3, "KV_tokens_per_s": tok / (call_ms * 1e-3),
            "algorithmic_bytes": kb, "algorithmic_flops": kf, "arithmetic_intensity": ai, "bound": bound,
            "attention_GBs": gbs, "attention_TFLOPs": tfs,
            "frac": (gbs / peaks["hbm_gbs"]) if bound == "hbm" else (tfs / peaks["bf16_tflops"]),
            "frac_of": "measured HBM GB/s" if bound == "hbm" else "measured bf16 TFLOP/s (burst)",
            "status": [int(code), int(flags)]})
        res[key] = entry
        del cache, ws
        torch.cuda.empty_cache()

    want = lambda *keys: not only or any(k in only for k in keys)   # noqa: E731
    if want("C2"):
        w = workloads.long_context(2)
        run("C2", "long context: B=2, L=32768/131072, H=64, bf16", w, mla.MLA_KV_BF16, 1)
    if want("C3"):
        w = workloads.verify(3)
        run("C3", "speculative verify: B=16, q_len=8, L~U[4096,32768], H=128, bf16", w, mla.MLA_KV_BF16, 8, n=5)
    if want("C5"):
        w = workloads.verify(5, B=1, q_len=512, len_range=(8192, 8192))
        run("C5", "chunked prefill: one 512-token chunk at L=8192, H=128, bf16", w, mla.MLA_KV_BF16, 512, n=3)
    if not want("C4", "C4q", "C6", "C7"):
        return res
    # rotated INT2: the workload's 65536 calibration latents through the library's own calibration
    w = workloads.int2_rotated(4)
    X = torch.from_numpy(np.asarray(w.calib)).to(dev)
    R32, clip, _, _ = mla.calibrate_rotation(X)
    run("C4", "rotated INT2 (DeepSeek-V3 shapes, 320 B/token), calibrated by the library, W_UV folded",
        w, mla.MLA_KV_INT2_ROT, 1, R=R32, T=clip, fold=True, append=True)
    run("C4q", "rotated INT2 as C4, R folded into both W_UV and the query's projection (query given rotated)",
        w, mla.MLA_KV_INT2_ROT, 1, R=R32, T=clip, fold=True, q_rotated=True)
    # the two rope/nope variants: the rope key's thresholds from calibration rope keys
    # of the cache's rope law (N(0,1) rounded to bf16)
    rng = np.random.Generator(np.random.PCG64(11))
    KRcal = workloads.bf16_round(rng.standard_normal((X.shape[0], w.d_rope)).astype(np.float32)).astype(np.float64)
    clip_r = mla.calib_thresholds(np.abs(KRcal), 32, 99.0)
    run("C6", "rotated INT2 with the rope key as two more INT2 groups (216 B/token), W_UV folded",
        w, mla.MLA_KV_INT2_ROT_QR, 1, R=R32, T=np.concatenate([clip, clip_r]), fold=True, append=True)
    Xj = torch.cat([X, torch.from_numpy(KRcal).to(dev)], dim=1).contiguous()
    del X
    Rj32, clip_j, _, _ = mla.calibrate_rotation(Xj)
    del Xj
    run("C7", "joint INT2: [c ; k_R] rotated by one 576-dim basis (216 B/token), generic kernel",
        w, mla.MLA_KV_INT2_JOINT, 1, R=Rj32, T=clip_j, n=3, append=True)
    return res


def run_configs(args):
    """--configs: the other workloads only, one JSON line each."""
    import torch
    from mla_latent_kv_08_gb300 import build as _build
    _build.build()
    import mla_latent_kv_08_gb300 as mla
    dev = torch.device("cuda", 0)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    only = tuple(k.strip() for k in args.only.split(",") if k.strip())
    for key, entry in measure_configs(mla, dev, load_peaks(), flush, only, args.reps).items():
        print(json.dumps(dict(config=key, **entry)), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.configs:
        return run_configs(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
