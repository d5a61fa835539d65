"""Benchmark of the packed BitLinear hot path on GB300.

Headline workload (one step = the BitNet-2B-shaped MLP for one token):
    h = max(0, W_g x)^2 * (W_u x)   (fused gate/up, i2_s 2560 -> 6912 twice,
                                     bf16 in, bf16 out; one launch)
    y = W_d h                       (i2_s 6912 -> 2560, bf16 in/out)
so the down projection consumes the fused kernel's output, as in the model.
The three matrices are held in 24 rotating copies (320 MB, more than twice
the 129 MB L2), so every step streams its weights from HBM.  Steps are
captured in CUDA graphs (with programmatic dependent launch between the
kernels) and replayed; the timed region is exactly --steps steps, bracketed by
a barrier and a device synchronize, timed with CUDA events on the launching
stream.

metric: packed-weight GB/s = (packed i2_s bytes of the three matrices,
scales included) * steps / time.  The roofline object times the dominant
kernel (the fused gate/up launch) in its own graph of back-to-back launches.  Secondary lines report the other
workloads (i2_s fp32 2560x2560, TQ2_0 5120x13824, W1A8 LM head at M=1/4/8,
i2_s int8 prefill at M=512 in TOPS).

--impl reference times the CPU oracle (oracle/) on this machine's cores on
a bounded sample of the same workload and prints the same JSON line.
"""
import argparse
import contextlib
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gemm_bl_gemv_gb300 import synth  # noqa: E402

METRIC = "M=1 packed-weight GB/s (% of HBM peak); M=512 int8 TOPS (% of peak)"
UNIT = "GB/s"
WL = synth.WORKLOADS["i2s_mlp_bitnet2b"]
MATS = ("gate", "up", "down")
COPIES = 24
FALLBACK_HBM = 6800.0
FALLBACK_BF16 = 1900.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), \
            "measured"
    return FALLBACK_HBM, FALLBACK_BF16, 1700.0, "fallback"


def packed_bytes(N, K):
    return N * (K // 4) + 4


def mlp_bytes():
    return sum(packed_bytes(*WL.extra[m]) for m in MATS)


DTYPE = "bf16 io; s16 fixed point x ternary codes -> s32"
ARITH = ("bf16 x and h and y; per 128-element group x is carried as 16-bit fixed point (two byte digits) and "
         "dotted with the 2-bit codes by dp4a into exact int32 sums; fp32 epilogue")


def headline_config(world):
    """The workload both arms time (the same dict in both JSON lines)."""
    return {"workload": WL.name, "model": "BitNet-2B-shaped MLP (random ternary weights)",
            "global_batch": 1, "seq_len": 1, "parallelism": "replicas" if world > 1 else "single",
            "M": 1, "shapes_NxK": [list(WL.extra[m]) for m in MATS], "x": "bf16", "y": "bf16",
            "step": "h = relu(W_gate x)^2 * (W_up x) [one fused launch]; y = W_down h",
            "l2": "GPU arm: inputs larger than L2 (%d rotating weight copies, %d MB); CPU reference arm: one copy"
                  % (COPIES, COPIES * mlp_bytes() >> 20)}


def gate_up_algorithmic_bytes():
    """Per fused gate/up launch: both packed tensors (scales included) + x (bf16) + h (bf16)."""
    N, K = WL.extra["gate"]
    return 2 * packed_bytes(N, K) + 2 * K + 2 * N


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: no collective on the data path)
# ---------------------------------------------------------------------------

class Dist:
    """One process per GPU (replicas: no data-path collective).  NCCL carries
    the barrier and the max over ranks on GPUs; gloo does on a CPU-only host."""

    def __init__(self, n_gpus):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        self.cuda = False
        if self.world > 1:
            import torch
            import torch.distributed as dist
            self.cuda = torch.cuda.is_available()
            if self.cuda:
                torch.cuda.set_device(self.local)
            dist.init_process_group("nccl" if self.cuda else "gloo")
            self.pg = dist

    def barrier(self):
        if self.pg:
            import torch
            self.pg.barrier()
            if self.cuda:
                torch.cuda.synchronize()

    def max(self, v):
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device="cuda" if self.cuda else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------

def upload_i2s(B, torch, wl_index, tensor, N, K, p_zero, scale, copies):
    """Pack one seeded ternary matrix on the GPU and replicate the packed bytes."""
    w = synth.weight_matrix(wl_index, tensor, N, K, "ternary", p_zero)
    packed = B.bl_pack_i2s(torch.from_numpy(w).cuda(), scale)
    return [packed] + [packed.clone() for _ in range(copies - 1)]


@contextlib.contextmanager
def nvtx(torch, name):
    """An NVTX range for profilers (ncu --nvtx); nothing when NVTX is unavailable."""
    try:
        torch.cuda.nvtx.range_push(name)
        pushed = True
    except Exception:  # noqa: BLE001
        pushed = False
    try:
        yield
    finally:
        if pushed:
            torch.cuda.nvtx.range_pop()


def graph_size(steps, cap):
    """The largest divisor of `steps` that is at most `cap`: a graph of that
    many steps, replayed, times exactly `steps` steps."""
    for g in range(min(cap, steps), 0, -1):
        if steps % g == 0:
            return g
    return 1


def warm_steps(warmup, graph_steps):
    """Warm-up in whole graph replays: at least `warmup` steps (and at least 3), at least one replay."""
    return max(1, -(-max(3, warmup) // graph_steps)) * graph_steps


def time_graph(torch, dist, body, steps, warmup, graph_steps, stream):
    """Capture `graph_steps` steps in a graph, replay: warm-up (whole replays
    covering at least `warmup` steps), then exactly `steps` timed steps."""
    assert steps % graph_steps == 0
    warmup = warm_steps(warmup, graph_steps)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for i in range(2):  # eager warm-up (kernel attributes, lazy loading)
            body(i)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(graph_steps):
                body(i)
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        for _ in range(warmup // graph_steps):
            g.replay()
        torch.cuda.synchronize()
        dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps // graph_steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gemm_bl_gemv_gb300", "csrc")
    for f in ("gemv_i2s_slot.cu", "bl_device.cuh"):  # the kernel's device code
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """dram bytes per launch of the dominant kernel from the committed ncu summary, or None
    when the kernel source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "gemv_i2s_mlp_bitnet2b.md")
    if not os.path.exists(p):
        return None
    vals = {}
    for line in open(p):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_hash") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def bench_ours(args, dist):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from gemm_bl_gemv_gb300 import binding as B

    torch.cuda.set_device(dist.local)
    hbm, bf16_burst, bf16_sust, peak_src = peaks()
    stream = torch.cuda.Stream()
    B.set_overlap(True)

    # ---- headline: BitNet-2B MLP, M=1, bf16 -----------------------------------------
    with torch.cuda.stream(stream):
        mats = {}
        for m in MATS:
            N, K = WL.extra[m]
            mats[m] = upload_i2s(B, torch, WL.index, "w_" + m, N, K, WL.p_zero,
                                 synth.tensor_scale(WL.index, "scale_" + m), COPIES)
        x_bits = synth.activations(WL.index, 1, 2560, "bf16")[0]
        x = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
        yg = torch.empty(6912, dtype=torch.bfloat16, device="cuda")   # h, the down projection's input
        ydn = torch.empty(2560, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()

    def mlp_step(i):
        c = i % COPIES
        B.bl_gemv_i2s_gate_up(mats["gate"][c], mats["up"][c], x, 6912, 2560, h=yg)
        B.bl_gemv_i2s(mats["down"][c], yg, 2560, 6912, y=ydn)

    gs = graph_size(args.steps, args.graph_steps)
    with ClockSampler(torch.cuda.current_device()) as clk, nvtx(torch, "mlp_step_timed"):
        ms = time_graph(torch, dist, mlp_step, args.steps, args.warmup, gs, stream)
    ms = dist.max(ms)
    step_bytes = mlp_bytes()
    value = step_bytes * args.steps * dist.world / (ms * 1e-3) / 1e9
    launches = 2 * args.steps

    # the dominant kernel alone: back-to-back fused gate/up launches (same copies, same PDL setting)
    def gate_up_only(i):
        c = i % COPIES
        B.bl_gemv_i2s_gate_up(mats["gate"][c], mats["up"][c], x, 6912, 2560, h=yg)

    gu_steps = args.roofline_launches
    gu_gs = graph_size(gu_steps, 1000)
    with nvtx(torch, "gate_up_alone"):
        gu_ms = dist.max(time_graph(torch, dist, gate_up_only, gu_steps, 2 * gu_gs, gu_gs, stream))
    avg_launch_s = gu_ms * 1e-3 / gu_steps
    achieved = gate_up_algorithmic_bytes() / avg_launch_s / 1e9

    # ---- e2e: host buffers, copies inside the timed region, public API per step -------
    e2e_steps = min(args.steps, args.e2e_steps)
    hx = torch.from_numpy(x_bits.view(np.int16).copy()).pin_memory()
    hyd = torch.empty(2560, dtype=torch.int16).pin_memory()
    dx = torch.empty(2560, dtype=torch.int16, device="cuda")

    # Per step, through the C ABI (include/bl.h) with arguments marshalled once:
    # pinned host x -> device, fused gate/up, down, device y -> pinned host.
    L, rt = B.lib(), B.cudart()
    vp = ctypes.c_void_p
    st = vp(stream.cuda_stream)
    dxp, hxp, hyp, ygp, ydp = vp(dx.data_ptr()), vp(hx.data_ptr()), vp(hyd.data_ptr()), vp(yg.data_ptr()), vp(ydn.data_ptr())
    gu_args = [(vp(mats["gate"][c].data_ptr()), vp(mats["up"][c].data_ptr()), dxp, B.BL_BF16, ygp, B.BL_BF16, 6912, 2560, st)
               for c in range(COPIES)]
    dn_args = [(vp(mats["down"][c].data_ptr()), ygp, B.BL_BF16, ydp, B.BL_BF16, 2560, 6912, st) for c in range(COPIES)]
    h2d_n, d2h_n = ctypes.c_size_t(2 * 2560), ctypes.c_size_t(2 * 2560)

    def e2e_step(i):
        c = i % COPIES
        return (rt.cudaMemcpyAsync(dxp, hxp, h2d_n, B.CUDA_MEMCPY_H2D, st) | L.bl_gemv_i2s_gate_up(*gu_args[c]) |
                L.bl_gemv_i2s(*dn_args[c]) | rt.cudaMemcpyAsync(hyp, ydp, d2h_n, B.CUDA_MEMCPY_D2H, st))

    with torch.cuda.stream(stream):
        bad = 0
        for i in range(min(200, e2e_steps)):
            bad |= e2e_step(i)
        torch.cuda.synchronize()
        dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(e2e_steps):
            bad |= e2e_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
        if bad:
            raise RuntimeError("e2e: a C ABI call or copy failed: %s" % B.lib().bl_last_error().decode())
    e2e_ms = dist.max(e0.elapsed_time(e1))
    e2e_value = step_bytes * e2e_steps * dist.world / (e2e_ms * 1e-3) / 1e9
    h2d = 2 * 2560
    d2h = 2 * 2560
    B.set_overlap(True)

    extra = {}
    if not args.no_extra:
        with nvtx(torch, "secondary"):
            extra = bench_secondary(args, B, torch, stream, dist, hbm, bf16_burst)
        try:  # a reported extra: it never stops the headline line
            extra["cold_single_launch_mlp"] = cold_launches(
                torch, stream, {"mlp_step": mlp_step, "gate_up": gate_up_only,
                                "down": lambda i: B.bl_gemv_i2s(mats["down"][i % COPIES], yg, 2560, 6912, y=ydn)})
        except Exception as e:  # noqa: BLE001
            extra["cold_single_launch_mlp"] = {"error": repr(e)[:200]}
        try:
            extra["act_quant_bf16"] = act_quant_times(torch, B, stream, hbm)
        except Exception as e:  # noqa: BLE001
            extra["act_quant_bf16"] = {"error": repr(e)[:200]}
        try:
            extra["e2e_graph_replay"] = e2e_graph_replay(torch, stream, e2e_step, step_bytes)
        except Exception as e:  # noqa: BLE001
            extra["e2e_graph_replay"] = {"error": repr(e)[:200]}
        try:
            extra["e2e_pipelined"] = e2e_pipelined(torch, B, mats, x_bits, step_bytes)
        except Exception as e:  # noqa: BLE001
            extra["e2e_pipelined"] = {"error": repr(e)[:200]}
    del mats
    torch.cuda.empty_cache()

    cpu = None
    if dist.rank == 0 and dist.world == 1 and args.cpu_seconds > 0:
        cpu = cpu_baseline(args.cpu_seconds)

    if dist.rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": DTYPE, "arith": ARITH, "data": "synthetic",
            "config": headline_config(dist.world),
            "launch": "CUDA graph of %d steps replayed %d times, programmatic dependent launch; warm-up %d steps "
                      "(whole replays)" % (gs, args.steps // gs, warm_steps(args.warmup, gs)),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(achieved / hbm, 4), "traffic": profiled_traffic(),
                         "kernel": "gemv_i2s_slot_kernel<D=2, bf16 x, bf16 y, gate+up>",
                         "algorithmic_bytes_per_launch": gate_up_algorithmic_bytes(),
                         "avg_launch_us": round(avg_launch_s * 1e6, 3), "launches_timed": gu_steps,
                         "peak_source": peak_src + " copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"},
            "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps, "api": "C ABI (bl_gemv_i2s_gate_up, bl_gemv_i2s) per step with cudaMemcpyAsync from/to pinned host memory, eager"},
            "gpu_launches": launches,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
            "secondary": extra,
        }
        print(json.dumps(line))


def e2e_graph_replay(torch, stream, step, step_bytes, steps=2000, graph_steps=100):
    """The e2e step (pinned host x in, both products, y back to pinned host)
    through the same C-ABI calls, captured once in a CUDA graph of
    `graph_steps` steps and replayed: what a serving loop built on graphs pays
    per step.  Reported beside the eager e2e figure, not in its place."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        bad = 0
        with torch.cuda.graph(g, stream=stream):
            for i in range(graph_steps):
                bad |= step(i)
        if bad:
            raise RuntimeError("a C ABI call or copy failed during capture")
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps // graph_steps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    n = (steps // graph_steps) * graph_steps
    return {"value": round(step_bytes * n / (ms * 1e-3) / 1e9, 2), "unit": UNIT,
            "us_per_step": round(ms * 1e3 / n, 3),
            "how": "C ABI calls and both copies captured in a CUDA graph of %d steps, %d steps replayed" % (graph_steps, n)}


def e2e_pipelined(torch, B, mats, x_bits, step_bytes, steps=2000, graph_steps=100):
    """The e2e step with its copies overlapped with the neighbouring steps'
    products, as a serving loop runs it: step i's x goes host -> device on one
    copy stream while step i - 1 computes, and step i's y goes back on another
    while step i + 1 computes.  x and y are double-buffered on the device and
    in pinned host memory, and every step still copies its own input in and
    its own result out.  The same C-ABI calls, captured once in a CUDA graph
    (three streams joined by events) and replayed.  Reported beside the eager
    e2e figure, not in its place."""
    L, rt = B.lib(), B.cudart()
    vp = ctypes.c_void_p
    sc, sh, sd = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    hx = [torch.from_numpy(x_bits.view(np.int16).copy()).pin_memory() for _ in range(2)]
    hy = [torch.empty(2560, dtype=torch.int16).pin_memory() for _ in range(2)]
    dx = [torch.empty(2560, dtype=torch.int16, device="cuda") for _ in range(2)]
    dy = [torch.empty(2560, dtype=torch.int16, device="cuda") for _ in range(2)]
    h = torch.empty(6912, dtype=torch.int16, device="cuda")
    ev_x = [torch.cuda.Event() for _ in range(2)]  # x[b] is on the device
    ev_y = [torch.cuda.Event() for _ in range(2)]  # y[b] is computed, so x[b] is consumed
    ev_d = [torch.cuda.Event() for _ in range(2)]  # y[b] is back in host memory, so dy[b] is free
    n = ctypes.c_size_t(2 * 2560)
    gate = [vp(t.data_ptr()) for t in mats["gate"]]
    up = [vp(t.data_ptr()) for t in mats["up"]]
    down = [vp(t.data_ptr()) for t in mats["down"]]
    c_sc, c_sh, c_sd = vp(sc.cuda_stream), vp(sh.cuda_stream), vp(sd.cuda_stream)

    def step(i):
        b, c = i % 2, i % COPIES
        bad = 0
        if i >= 2:
            sh.wait_event(ev_y[b])
        bad |= rt.cudaMemcpyAsync(vp(dx[b].data_ptr()), vp(hx[b].data_ptr()), n, B.CUDA_MEMCPY_H2D, c_sh)
        ev_x[b].record(sh)
        sc.wait_event(ev_x[b])
        if i >= 2:
            sc.wait_event(ev_d[b])
        bad |= L.bl_gemv_i2s_gate_up(gate[c], up[c], vp(dx[b].data_ptr()), B.BL_BF16, vp(h.data_ptr()), B.BL_BF16,
                                     6912, 2560, c_sc)
        bad |= L.bl_gemv_i2s(down[c], vp(h.data_ptr()), B.BL_BF16, vp(dy[b].data_ptr()), B.BL_BF16, 2560, 6912, c_sc)
        ev_y[b].record(sc)
        sd.wait_event(ev_y[b])
        bad |= rt.cudaMemcpyAsync(vp(hy[b].data_ptr()), vp(dy[b].data_ptr()), n, B.CUDA_MEMCPY_D2H, c_sd)
        ev_d[b].record(sd)
        return bad

    g = torch.cuda.CUDAGraph()
    fork, jh, jd = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
    torch.cuda.synchronize()
    bad = 0
    with torch.cuda.graph(g, stream=sc):
        fork.record(sc)  # the copy streams join the capture
        sh.wait_event(fork)
        sd.wait_event(fork)
        for i in range(graph_steps):
            bad |= step(i)
        jh.record(sh)  # and rejoin it
        jd.record(sd)
        sc.wait_event(jh)
        sc.wait_event(jd)
    if bad:
        raise RuntimeError("a C ABI call or copy failed during capture")
    with torch.cuda.stream(sc):
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(sc)
        for _ in range(steps // graph_steps):
            g.replay()
        e1.record(sc)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    reps = steps // graph_steps
    total = reps * graph_steps
    ok = bool(torch.equal(hy[0], hy[1]))  # the same x every step: both host results must agree
    return {"value": round(step_bytes * total / (ms * 1e-3) / 1e9, 2), "unit": UNIT,
            "us_per_step": round(ms * 1e3 / total, 3), "h2d_bytes_per_step": 2 * 2560, "d2h_bytes_per_step": 2 * 2560,
            "results_agree": ok,
            "how": "per step: x host->device on a copy stream, fused gate/up and down, y device->host on another copy "
                   "stream; x and y double-buffered, copies of step i overlapping the products of steps i -/+ 1; "
                   "C ABI calls captured in a CUDA graph of %d steps, %d steps replayed" % (graph_steps, total)}


def cold_launches(torch, stream, calls, reps=50):
    """Median time of one call with L2 flushed before it (a buffer of twice the L2
    size is written between calls), for each named call; microseconds."""
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    l2 = int(getattr(props, "L2_cache_size", 0) or (129 << 20))
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device="cuda")
    out = {}
    with torch.cuda.stream(stream):
        for name, fn in calls.items():
            ts = []
            for i in range(reps + 3):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn(i)
                e1.record(stream)
                e1.synchronize()
                if i >= 3:
                    ts.append(e0.elapsed_time(e1) * 1e3)
            out[name + "_us"] = round(float(np.median(ts)), 3)
    torch.cuda.synchronize()
    del flush
    out["how"] = "median of %d single calls, each after writing %d MB (2x L2)" % (reps, 2 * l2 >> 20)
    return out


def act_quant_times(torch, B, stream, hbm, shapes=((512, 2560), (8, 5120)), reps=200):
    """The per-token act-quant launch alone (bf16 x), eager back-to-back
    launches timed with events: microseconds and GB/s of x read plus q and s
    written."""
    L = B.lib()
    out = {}
    vp = ctypes.c_void_p
    for M, K in shapes:
        xb = synth.activations(WL.index, M, K, "bf16")
        x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
        q = torch.empty((M, K), dtype=torch.int8, device="cuda")
        sc = torch.empty(M, dtype=torch.float32, device="cuda")
        args = (vp(x.data_ptr()), B.BL_BF16, M, K, vp(q.data_ptr()), vp(sc.data_ptr()), vp(stream.cuda_stream))
        with torch.cuda.stream(stream):
            bad = 0
            for _ in range(10):
                bad |= L.bl_quantize_act_absmax_int8(*args)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                bad |= L.bl_quantize_act_absmax_int8(*args)
            e1.record(stream)
            torch.cuda.synchronize()
        if bad:
            raise RuntimeError("bl_quantize_act_absmax_int8: " + L.bl_last_error().decode())
        us = e0.elapsed_time(e1) * 1e3 / reps
        gbs = (2 * M * K + M * K + 4 * M) / (us * 1e-6) / 1e9
        out["M%d_K%d" % (M, K)] = {"us_per_launch": round(us, 3), "GBps": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4)}
    return out


def bench_secondary(args, B, torch, stream, dist, hbm, bf16_peak):
    """Other workloads: single-workload GB/s (or TOPS) with rotating copies, graphs + PDL."""
    out = {}
    gs = 100
    steps = max(gs, (args.secondary_steps // gs) * gs)

    def run(body):
        return dist.max(time_graph(torch, dist, body, steps, gs, gs, stream)) / steps  # ms per step

    with torch.cuda.stream(stream):
        # i2_s GEMV 2560x2560 fp32
        wl = synth.WORKLOADS["i2s_gemv_2560"]
        cps = 160
        ws = upload_i2s(B, torch, wl.index, "w", wl.N, wl.K, wl.p_zero, synth.tensor_scale(wl.index), cps)
        x = torch.from_numpy(synth.activations(wl.index, 1, wl.K, "f32")[0]).cuda()
        y = torch.empty(wl.N, dtype=torch.float32, device="cuda")
        t = run(lambda i: B.bl_gemv_i2s(ws[i % cps], x, wl.N, wl.K, y=y))
        gbs = packed_bytes(wl.N, wl.K) / (t * 1e-3) / 1e9
        out[wl.name] = {"value": round(gbs, 1), "unit": "GB/s", "frac_hbm": round(gbs / hbm, 4), "us_per_launch": t * 1e3}
        del ws

        # TQ2_0 GEMV 5120 -> 13824, bf16 x, fp32 y
        wl = synth.WORKLOADS["tq2_0_gemv_5120x13824"]
        cps = 16
        w = synth.weight_matrix(wl.index, "w", wl.N, wl.K, "ternary", wl.p_zero)
        d = synth.block_scale_matrix(wl.index, wl.N, wl.K // 256)
        p0 = B.bl_pack_tq2_0(torch.from_numpy(w).cuda(), torch.from_numpy(d.view(np.int16)).cuda())
        ws = [p0] + [p0.clone() for _ in range(cps - 1)]
        x = torch.from_numpy(synth.activations(wl.index, 1, wl.K, "bf16")[0].view(np.int16)).cuda().view(torch.bfloat16)
        y = torch.empty(wl.N, dtype=torch.float32, device="cuda")
        t = run(lambda i: B.bl_gemv_tq2_0(ws[i % cps], x, wl.N, wl.K, y=y))
        nbytes = wl.N * (wl.K // 256) * 66
        gbs = nbytes / (t * 1e-3) / 1e9
        out[wl.name] = {"value": round(gbs, 1), "unit": "GB/s", "frac_hbm": round(gbs / hbm, 4), "us_per_launch": t * 1e3}
        # the same TQ2_0 weights against 512 int8 tokens (tensor cores: TOPS)
        Mq = 512
        xb = synth.activations(wl.index, Mq, wl.K, "bf16")
        q, s = B.bl_quantize_act_absmax_int8(torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16))
        y = torch.empty((Mq, wl.N), dtype=torch.float32, device="cuda")
        t = run(lambda i: B.bl_gemm_tq2_0_int8(q, s, ws[i % cps], wl.N, y=y))
        tops = 2.0 * Mq * wl.N * wl.K / (t * 1e-3) / 1e12
        out["tq2_0_int8_5120x13824_M512"] = {"value": round(tops, 1), "unit": "TOPS (int8 ops)",
                                             "frac_bf16_dense_peak": round(tops / bf16_peak, 4), "us_per_launch": t * 1e3}
        del ws, p0, y

        # W1A8 LM head, M = 1, 4, 8
        wl = synth.WORKLOADS["w1a8_lmhead_248320"]
        N, K, G = wl.N, wl.K, wl.group
        wq = torch.empty((N, K // 32), dtype=torch.int32, device="cuda")
        for b in range((N + synth.ROW_BLOCK - 1) // synth.ROW_BLOCK):
            blk = synth.weight_block(wl.index, "w", N, K, b, "signs")
            B.bl_pack_w1(torch.from_numpy(blk).cuda(), out=wq[b * synth.ROW_BLOCK:b * synth.ROW_BLOCK + blk.shape[0]])
        wsc = torch.from_numpy(synth.block_scale_matrix(wl.index, N, K // G, tensor="group_scale").view(np.int16)).cuda()
        wqs, wss = [wq, wq.clone()], [wsc, wsc.clone()]
        wbytes = N * K // 8 + N * (K // G) * 2
        for M in (1, 4, 8):
            xb = synth.activations(wl.index, M, K, "bf16")
            xg = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
            q, s = B.bl_quantize_act_absmax_int8(xg)
            y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            t = run(lambda i: B.bl_gemm_w1a8(q, s, wqs[i % 2], wss[i % 2].view(torch.float16), group=G, y=y))
            gbs = wbytes / (t * 1e-3) / 1e9
            # from unquantized bf16 x: quantization fused into the product vs the two launches
            t_f = run(lambda i: B.bl_gemm_w1a8_act(xg, wqs[i % 2], wss[i % 2].view(torch.float16), group=G, y=y))

            def two_calls(i):
                B.bl_quantize_act_absmax_int8(xg, q, s)
                B.bl_gemm_w1a8(q, s, wqs[i % 2], wss[i % 2].view(torch.float16), group=G, y=y)
            t_2 = run(two_calls)
            out["%s_M%d" % (wl.name, M)] = {"value": round(gbs, 1), "unit": "GB/s", "frac_hbm": round(gbs / hbm, 4),
                                            "us_per_launch": t * 1e3,
                                            "int_ops_per_s": 2.0 * M * N * K / (t * 1e-3),
                                            "us_from_bf16_x_fused_quant": t_f * 1e3,
                                            "us_from_bf16_x_two_launches": t_2 * 1e3}
        # larger batches of the same LM head run on the tensor cores (TOPS)
        for M in (128, 512):
            xb = synth.activations(wl.index, M, K, "bf16")
            q, s = B.bl_quantize_act_absmax_int8(torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16))
            y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            n_l = 40
            t = dist.max(time_graph(torch, dist, lambda i: B.bl_gemm_w1a8(q, s, wqs[i % 2], wss[i % 2].view(torch.float16),
                                                                         group=G, y=y), n_l, 4, 4, stream)) / n_l
            tops = 2.0 * M * N * K / (t * 1e-3) / 1e12
            out["%s_M%d" % (wl.name, M)] = {"value": round(tops, 1), "unit": "TOPS (int8 ops)",
                                            "frac_bf16_dense_peak": round(tops / bf16_peak, 4), "us_per_launch": t * 1e3}
            del y
        del wqs, wss, wq, wsc

        # i2_s int8 prefill M = 512 (tensor-bound: TOPS)
        wl = synth.WORKLOADS["i2s_prefill_512"]
        cps = 24
        ws = upload_i2s(B, torch, wl.index, "w", wl.N, wl.K, wl.p_zero, synth.tensor_scale(wl.index), cps)
        xb = synth.activations(wl.index, wl.M, wl.K, "bf16")
        q, s = B.bl_quantize_act_absmax_int8(torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16))
        y = torch.empty((wl.M, wl.N), dtype=torch.float32, device="cuda")
        t = run(lambda i: B.bl_gemm_i2s_int8(q, s, ws[i % cps], wl.N, y=y))
        tops = 2.0 * wl.M * wl.N * wl.K / (t * 1e-3) / 1e12
        # from bf16 x: the quantization fused into the product's launch, against act-quant + product
        xg = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
        wsp = B.gemm_i2s_int8_act_workspace(wl.M, wl.K)
        try:  # a reported extra (a cooperative launch inside a graph): it never stops the headline line
            t_f = run(lambda i: B.bl_gemm_i2s_int8_act(xg, ws[i % cps], wl.N, workspace=wsp, y=y, fuse=True))
        except Exception as e:  # noqa: BLE001
            t_f = float("nan")
            out["i2s_prefill_512_fused_error"] = repr(e)[:200]
        t_2 = run(lambda i: B.bl_gemm_i2s_int8_act(xg, ws[i % cps], wl.N, workspace=wsp, y=y))
        out[wl.name] = {"value": round(tops, 2), "unit": "TOPS (int8 ops)", "frac_bf16_dense_peak": round(tops / bf16_peak, 4),
                        "us_per_launch": t * 1e3, "us_from_bf16_x_one_launch": t_f * 1e3,
                        "us_from_bf16_x_two_launches": t_2 * 1e3}
        del ws, wsp
        if not args.no_cublas:
            out.update(bench_cublas(args, torch, stream, dist, run))
    torch.cuda.synchronize()
    return out


def bench_cublas(args, torch, stream, dist, run):
    """cuBLAS bf16 (called through torch.matmul) on dense bf16 weights of the same shapes, rotated past L2:
    the comparison column the binary-gemm card reports its speedups against."""
    out = {}
    gen = torch.Generator(device="cuda").manual_seed(1)

    def dense(N, K, copies):
        return [torch.randn(N, K, device="cuda", dtype=torch.bfloat16, generator=gen) for _ in range(copies)]

    # MLP step, M = 1: gate, up, relu^2 * up, down (3 copies x 106 MB)
    cps = 3
    Wg, Wu, Wd = dense(6912, 2560, cps), dense(6912, 2560, cps), dense(2560, 6912, cps)
    x = torch.randn(1, 2560, device="cuda", dtype=torch.bfloat16, generator=gen)

    def mlp(i):
        c = i % cps
        g = torch.matmul(x, Wg[c].t())
        u = torch.matmul(x, Wu[c].t())
        h = torch.relu(g) ** 2 * u
        torch.matmul(h, Wd[c].t())

    t = run(mlp)
    out["cublas_bf16_mlp_bitnet2b"] = {"us_per_step": t * 1e3, "unit": "us",
                                       "bf16_weight_GBps": round(3 * 6912 * 2560 * 2 / (t * 1e-3) / 1e9, 1)}
    del Wg, Wu, Wd
    # LM head, M = 1, 4, 8 (2 copies x 2.5 GB)
    W = dense(248320, 5120, 2)
    for M in (1, 4, 8):
        xm = torch.randn(M, 5120, device="cuda", dtype=torch.bfloat16, generator=gen)
        t = run(lambda i: torch.matmul(xm, W[i % 2].t()))
        out["cublas_bf16_lmhead_248320_M%d" % M] = {"us_per_launch": t * 1e3, "unit": "us",
                                                    "bf16_weight_GBps": round(248320 * 5120 * 2 / (t * 1e-3) / 1e9, 1)}
    del W
    # prefill M = 512 (bf16 GEMM, TFLOP/s)
    W = dense(6912, 2560, 8)
    xm = torch.randn(512, 2560, device="cuda", dtype=torch.bfloat16, generator=gen)
    t = run(lambda i: torch.matmul(xm, W[i % 8].t()))
    out["cublas_bf16_prefill_512"] = {"us_per_launch": t * 1e3, "unit": "us",
                                      "tflops": round(2.0 * 512 * 6912 * 2560 / (t * 1e-3) / 1e12, 1)}
    del W, xm
    # the TQ2_0 shape, M = 512
    W = dense(13824, 5120, 4)
    xm = torch.randn(512, 5120, device="cuda", dtype=torch.bfloat16, generator=gen)
    t = run(lambda i: torch.matmul(xm, W[i % 4].t()))
    out["cublas_bf16_5120x13824_M512"] = {"us_per_launch": t * 1e3, "unit": "us",
                                          "tflops": round(2.0 * 512 * 13824 * 5120 / (t * 1e-3) / 1e12, 1)}
    del W, xm
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------

class OracleMLP:
    """The oracle computing the MLP step (fused gate/up, then down) on
    `rows_frac` of each matrix's rows; the down projection reads the full h of
    one oracle step computed at construction."""

    def __init__(self, rows_frac=1.0):
        from oracle import oracle as O
        self.O = O
        self.cores = len(os.sched_getaffinity(0))
        O.set_threads(self.cores)
        self.mats = {}
        for m in MATS:
            N, K = WL.extra[m]
            w = synth.weight_matrix(WL.index, "w_" + m, N, K, "ternary", WL.p_zero)
            nr = max(1, int(round(N * rows_frac)))
            rows = np.linspace(0, N - 1, nr).astype(np.int64)
            self.mats[m] = (O.pack_i2s(w, synth.tensor_scale(WL.index, "scale_" + m)), N, K, rows)
        xb = synth.activations(WL.index, 1, 2560, "bf16")[0]
        self.x = O.bf16_to_f64(xb)
        pg, N, K, _ = self.mats["gate"]
        self.h, _ = O.gemv_i2s_gate_up(pg, self.mats["up"][0], self.x, N, K)
        self.bytes_per_step = sum(len(r) * (K // 4) for (_, _, K, r) in self.mats.values())

    def step(self):
        pg, N, K, rows = self.mats["gate"]
        self.O.gemv_i2s_gate_up(pg, self.mats["up"][0], self.x, N, K, rows=rows)
        pd, Nd, Kd, rows_d = self.mats["down"]
        self.O.gemv_i2s(pd, self.h, Nd, Kd, rows=rows_d)


def cpu_baseline(seconds):
    o = OracleMLP(1.0)
    o.step()
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < seconds:
        o.step()
        n += 1
    dt = time.perf_counter() - t0
    out = {"value": round(o.bytes_per_step * n / dt / 1e9, 4), "unit": UNIT, "cores": o.cores if o.O.has_openmp() else 1,
           "kind": "oracle",
           "sample": "%d full MLP steps (fused gate/up then down, all rows, one token) in %.1f s" % (n, dt)}
    # the same oracle on one host thread, for a quarter of the time
    o.O.set_threads(1)
    try:
        t0 = time.perf_counter()
        n1 = 0
        while n1 == 0 or time.perf_counter() - t0 < seconds / 4:
            o.step()
            n1 += 1
        dt1 = time.perf_counter() - t0
    finally:
        o.O.set_threads(o.cores)
    out["one_thread"] = {"value": round(o.bytes_per_step * n1 / dt1 / 1e9, 4), "unit": UNIT, "cores": 1,
                         "sample": "%d full MLP steps in %.1f s" % (n1, dt1)}
    return out


def bench_reference(args, dist):
    if dist.rank != 0:
        return
    probe = OracleMLP(1.0)
    probe.step()
    t0 = time.perf_counter()
    probe.step()
    t_full = time.perf_counter() - t0
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    frac = min(1.0, max(1e-4, budget / max(t_full, 1e-9)))
    o = OracleMLP(frac)
    for _ in range(args.warmup):
        o.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        o.step()
    dt = time.perf_counter() - t0
    value = o.bytes_per_step * args.steps / dt / 1e9
    cores = o.cores if o.O.has_openmp() else 1
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (oracle)", "arith": "fp64 accumulation of the decoded ternary weights times x",
        "data": "synthetic", "impl": "reference",
        "config": headline_config(dist.world),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "each step: the MLP on %.4f of each matrix's rows" % frac},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200000)
    ap.add_argument("--warmup", type=int, default=4000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--graph-steps", type=int, default=1000, help="most steps captured in one graph")
    ap.add_argument("--roofline-launches", type=int, default=20000,
                    help="back-to-back launches of the dominant kernel timed for the roofline object")
    ap.add_argument("--e2e-steps", type=int, default=20000)
    ap.add_argument("--secondary-steps", type=int, default=2000)
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cublas", action="store_true", help="skip the cuBLAS comparison column (5 GB of dense weights)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    args = ap.parse_args()
    dist = Dist(args.gpus)
    try:
        if args.impl == "reference":
            bench_reference(args, dist)
        else:
            bench_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
