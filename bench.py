"""Benchmark of the attention core: one step = forward + backward of one packed batch.

Default workload: the packed batch of 12 + 925 + 4253 + 8349 tokens (13539),
48 heads, head_dim 128, bf16 q/k/v ~ N(0, 1), dO ~ N(0, 1) (synthetic, seeded).
The metric is attention forward+backward TFLOP/s on that batch, counting
4 H d sum_s L_s^2 forward and 2.5x that backward (algorithmic flops of the
per-sample attention; the masked cross-sample blocks are not counted).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same batch on its own GPU (replicas;
the path has no data-path collective) and the value is the sum over ranks.
``--impl reference`` times the FP64 CPU oracle on the host cores instead,
on a bounded sample of the same workload (one 925-token sample per step).
"""

from __future__ import annotations

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

import numpy as np  # noqa: E402
import torch  # noqa: E402

from invariant_dit_attention_gb300 import workloads as W  # noqa: E402

METRIC = "attention fwd/bwd TFLOP/s at 8349 packed tokens, % of GB300 BF16 peak"
WORKLOAD = "packed_13539"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
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
            out = {}
            for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                cands = [v for k, v in flat.items() if k.split(".")[-1] == key]
                if cands:
                    out[key] = cands[0]
            if "hbm_gbs" in out and "bf16_tflops" in out:
                out.setdefault("bf16_tflops_sustained", out["bf16_tflops"])
                out["source"] = "measured"
                return out
        except Exception:
            pass
    return dict(FALLBACK_PEAKS, source="fallback")


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region: sampling starts
    (20 ms interval) before the region, and only the samples taken between
    mark_start() and mark_end() (host clock) are summarised."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t_end = time.time() + 5.0  # let the sampler start before the timed region
            while not self.lines and time.time() < t_end:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = getattr(self, "t0", None), getattr(self, "t1", None)
        inside = [ln for t, ln in self.lines if t0 is not None and t1 is not None and t0 <= t <= t1]
        for ln in inside:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def projection_rate(S, D, stream, pk):
    """QKV (D -> 3D) and output (D -> D) projections of S tokens with h3attn_linear
    (synthetic bf16 activations and weights, FP32 bias), CUDA-event timed."""
    from invariant_dit_attention_gb300.h3attn import linear
    g = torch.Generator(device="cuda").manual_seed(7)
    x = torch.randn(S, D, device="cuda", generator=g).to(torch.bfloat16)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = {}
    for name, n in (("qkv", 3 * D), ("out", D)):
        w = (torch.randn(n, D, device="cuda", generator=g) / D ** 0.5).to(torch.bfloat16)
        b = torch.randn(n, device="cuda", generator=g)
        y = torch.empty(S, n, dtype=torch.bfloat16, device="cuda")
        for _ in range(3):
            linear(x, w, b, out=y, error_flags=flags)
        reps = 5
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            linear(x, w, b, out=y, error_flags=flags)
        e1.record(stream)
        torch.cuda.synchronize()
        if int(flags.item()) != 0:
            raise RuntimeError("h3attn_linear reported a device error")
        ms = e0.elapsed_time(e1) / reps
        tf = 2.0 * S * D * n / (ms * 1e-3) / 1e12
        res[name] = {"shape": [S, D, n], "ms": round(ms, 4), "tflops": round(tf, 1),
                     "frac": round(tf / pk["bf16_tflops"], 4)}
        if name == "qkv":
            res[name]["traffic"] = measured_traffic("linear_qkv")
        del w, b, y
    return res


def qkv_rate(H, S, d, stream, reps=5):
    """QKV projection (D = H * 128 -> 3D) plus the attention forward of the same
    tokens: fused (h3attn_qkv_forward: the q/k norm and RoPE in the projection's
    epilogue) against the separate calls (h3attn_linear, then h3attn_forward on
    its q, k, v), CUDA-event timed."""
    from invariant_dit_attention_gb300.h3attn import H3Attn, linear
    D = H * 128
    g = torch.Generator(device="cuda").manual_seed(11)
    x = torch.randn(S, D, device="cuda", generator=g).to(torch.bfloat16)
    w = (torch.randn(3 * D, D, device="cuda", generator=g) / D ** 0.5).to(torch.bfloat16)
    b = 0.1 * torch.randn(3 * D, device="cuda", generator=g)
    h = H3Attn(H, S, 8, store_ds=False)  # forward only
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    qkv = [torch.empty(S, H, 128, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    out = torch.empty_like(qkv[0])
    lse = torch.empty(H, S, device="cuda")

    def fused():
        h.qkv_forward(x, w, b, d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"], q=qkv[0], k=qkv[1],
                      v=qkv[2], out=out, lse=lse)

    def separate():
        for i in range(3):  # one projection per q, k, v slice of W, straight into its tensor
            linear(x, w[i * D:(i + 1) * D], b[i * D:(i + 1) * D], out=qkv[i].view(S, D), error_flags=flags)
        h.forward(qkv[0], qkv[1], qkv[2], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"], out=out,
                  lse=lse)

    res = {}
    for name, fn in (("fused_ms", fused), ("separate_ms", separate)):
        for _ in range(2):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        res[name] = round(e0.elapsed_time(e1) / reps, 4)
    h.check()
    h.close()
    if int(flags.item()) != 0:
        raise RuntimeError("h3attn_linear reported a device error")
    res["shape"] = [S, D, 3 * D]
    res["separate_includes"] = "three projections (the q, k, v slices of W), forward (prologue + attention)"
    return res


def canonical_rate(H, S, d, grads, step_flops, packed_ms, stream, steps=10):
    """The same forward + backward step with the canonical key order (sums over a
    sample's tokens in an order fixed by the tokens, not by their packing),
    CUDA-event timed outside the headline's timed region."""
    from invariant_dit_attention_gb300.h3attn import H3Attn
    h = H3Attn(H, S, 8, key_order="canonical")

    def step():
        out, lse = h.forward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
        h.backward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"],
                   out, lse, d["dout"], grads=grads)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    h.check()
    h.set_stage_timing(True)
    h.stage_times()  # reset
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    st = h.stage_times()
    h.check()
    h.close()
    ms = e0.elapsed_time(e1) / steps
    return {"ms_per_step": round(ms, 4), "tflops": round(step_flops / (ms * 1e-3) / 1e12, 2),
            "overhead_vs_packed": round(ms / packed_ms - 1.0, 4),
            "order_ms": round(st["order"][0] / steps, 4), "permute_ms": round(st["permute"][0] / steps, 4),
            "steps": steps}


def measured_traffic(kernel_key):
    """DRAM bytes (read + write) of one launch from the committed ncu summary, or
    None if the kernel's source changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        k = json.load(open(path))["kernels"][kernel_key]
        src = os.path.join(ROOT, k["source"])
        if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != k["sha256_16"]:
            return None
        return int(k["dram_read_bytes"]) + int(k["dram_write_bytes"])
    except Exception:
        return None


def traffic_note(kernel_key):
    """How the committed traffic figure was taken, when it was scaled from a smaller capture."""
    try:
        k = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))["kernels"][kernel_key]
        return k["workload"] if "scaled" in k.get("workload", "") else None
    except Exception:
        return None


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def barrier_max(x: float, ws: int) -> float:
    """The largest of the ranks' values (the slowest rank's time sets the job's)."""
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, steps: int, ws: int, ms_max: float) -> float:
    """Whole-job rate: every rank runs the same steps on its own replica of the
    workload (weak scaling), so the job's work is ws times one rank's, done in
    the slowest rank's time."""
    return flops_per_step * steps * ws / (ms_max * 1e-3) / 1e12


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def bwd_flops(fwd):
    return 2.5 * fwd


def run_ours(args):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    from invariant_dit_attention_gb300 import build
    build.build()
    from invariant_dit_attention_gb300.h3attn import H3Attn, to_device

    wname = args.profile_workload if args.profile and args.profile_workload else WORKLOAD
    w, inp = W.make_workload(wname)
    inp = W.make_inputs(w.samples, w.num_heads, w.seed, w.std, w.outlier_frac, w.outlier_scale, with_grad=True)
    S, H = inp.total_tokens, inp.num_heads
    fwd_flops = w.fwd_flops()
    step_flops = fwd_flops + bwd_flops(fwd_flops)
    h = H3Attn(H, S, 8)
    d = to_device(inp)
    stream = torch.cuda.current_stream()

    def step():
        out, lse = h.forward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
        g = h.backward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"],
                       out, lse, d["dout"], grads=grads)
        return out, g

    grads = {"dq": torch.empty_like(d["q"]), "dk": torch.empty_like(d["k"]), "dv": torch.empty_like(d["v"]),
             "dq_norm_w": torch.empty(128, device="cuda"), "dk_norm_w": torch.empty(128, device="cuda"),
             "dq_norm_w_per_sample": torch.empty(inp.num_samples, 128, device="cuda"),
             "dk_norm_w_per_sample": torch.empty(inp.num_samples, 128, device="cuda")}
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    h.check()
    if args.profile:
        # fixed launch sequence for a profiler: the steps only, no timing extras
        for _ in range(args.steps):
            step()
        torch.cuda.synchronize()
        h.check()
        # then one QKV and one output projection of the same tokens (h3attn_linear)
        from invariant_dit_attention_gb300.h3attn import linear
        D = H * 128
        x = torch.randn(S, D, device="cuda").to(torch.bfloat16)
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")
        for n in (3 * D, D):
            w = (torch.randn(n, D, device="cuda") / D ** 0.5).to(torch.bfloat16)
            linear(x, w, torch.randn(n, device="cuda"), error_flags=flags)
        # and one fused QKV projection + forward (h3attn_qkv_forward) of the same tokens
        w = (torch.randn(3 * D, D, device="cuda") / D ** 0.5).to(torch.bfloat16)
        h.qkv_forward(x, w, 0.1 * torch.randn(3 * D, device="cuda"), d["q_norm_w"], d["k_norm_w"], d["pos"],
                      d["seg_offsets"])
        torch.cuda.synchronize()
        h.check()
        if rank == 0:
            print(json.dumps({"profile_run": wname, "steps": args.steps, "warmup": args.warmup,
                              "then": "projections qkv, out; fused qkv forward"}))
        return

    # ---- device-resident timed region: two events around the steps, nothing inside
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(ws)
        torch.cuda.synchronize()
        clk.mark_start()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
        barrier(ws)
    ms = e0.elapsed_time(e1)
    h.check()
    ms_max = barrier_max(ms, ws)
    value = whole_job_tflops(step_flops, args.steps, ws, ms_max)

    # ---- per-stage times: the same steps once more, every launch bracketed by events
    h.set_stage_timing(True)
    h.stage_times()  # reset
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    stages = h.stage_times()
    h.set_stage_timing(False)
    h.check()

    # ---- forward-only rates: whole batch and every sample alone (same kernels)
    # forward's share: the attention kernel, its norm/RoPE prologue (the backward reuses the
    # rotated rows, so every prologue launch is a forward's) and one of the two plans
    fwd_ms = stages["fwd"][0] + stages["prologue"][0] + 0.5 * stages["plan"][0]
    per_sample = {}
    for s in range(inp.num_samples):
        alone = to_device(W.slice_sample(inp, s))
        L = inp.meta["lengths"][s]
        for _ in range(3):
            h.forward(alone["q"], alone["k"], alone["v"], alone["q_norm_w"], alone["k_norm_w"], alone["pos"],
                      alone["seg_offsets"])
        reps = 10 if L > 1000 else 50
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h.set_stage_timing(True)
        h.stage_times()  # reset
        a0.record(stream)
        for _ in range(reps):
            h.forward(alone["q"], alone["k"], alone["v"], alone["q_norm_w"], alone["k_norm_w"], alone["pos"],
                      alone["seg_offsets"])
        a1.record(stream)
        torch.cuda.synchronize()
        st_alone = h.stage_times()
        h.set_stage_timing(False)
        t = a0.elapsed_time(a1) / reps
        tk = st_alone["fwd"][0] / max(st_alone["fwd"][1], 1)
        flops = 4.0 * H * 128 * L * L
        # fwd_*: the whole call (plan, norm/RoPE prologue, attention); fwd_kernel_*: the attention kernel
        per_sample[str(L)] = {"fwd_ms": round(t, 4), "fwd_tflops": round(flops / (t * 1e-3) / 1e12, 2),
                              "fwd_kernel_ms": round(tk, 4),
                              "fwd_kernel_tflops": round(flops / (tk * 1e-3) / 1e12, 2)}
        del alone

    # ---- end to end: host (pinned) inputs -> device -> fwd + bwd -> host results.
    # Pipelined as a training loop would run it: step n+1's inputs go up on one
    # copy stream and step n-1's results come back on another while step n's
    # kernels run; device buffers are double-buffered, so every step still
    # copies all of its inputs up and all of its results back.
    host_in = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in
               {"q": inp.q, "k": inp.k, "v": inp.v, "q_norm_w": inp.q_norm_w, "k_norm_w": inp.k_norm_w,
                "dout": inp.dout, "seg_offsets": inp.seg_offsets}.items()}
    host_pos = [inp.pos[a].contiguous().pin_memory() for a in range(3)]
    host_out = {"out": torch.empty_like(inp.q).pin_memory(), "dq": torch.empty_like(inp.q).pin_memory(),
                "dk": torch.empty_like(inp.k).pin_memory(), "dv": torch.empty_like(inp.v).pin_memory(),
                "dq_norm_w": torch.empty(128).pin_memory(), "dk_norm_w": torch.empty(128).pin_memory()}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values()) + sum(
        t.numel() * t.element_size() for t in host_pos)
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    dbuf = [d, {k: ([torch.empty_like(t) for t in v] if k == "pos" else torch.empty_like(v)) for k, v in d.items()}]
    gbuf = [grads, {k: torch.empty_like(v) for k, v in grads.items()}]
    obuf = [(torch.empty_like(d["q"]), torch.empty(H, S, device="cuda")) for _ in range(2)]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in", "in_bwd", "fwd", "done", "read")}

    def e2e_step(n):
        b = n % 2
        db, gb, (ob, lb) = dbuf[b], gbuf[b], obuf[b]
        up.wait_event(ev["done"][b])  # step n-2's kernels have finished with these inputs
        with torch.cuda.stream(up):
            # the forward's inputs first, then dO, which only the backward reads
            for k in host_in:
                if k != "dout":
                    db[k].copy_(host_in[k], non_blocking=True)
            for a in range(3):
                db["pos"][a].copy_(host_pos[a], non_blocking=True)
            ev["in"][b].record(up)
            db["dout"].copy_(host_in["dout"], non_blocking=True)
            ev["in_bwd"][b].record(up)
        stream.wait_event(ev["in"][b])
        stream.wait_event(ev["read"][b])  # step n-2's results have been read back
        out, lse = h.forward(db["q"], db["k"], db["v"], db["q_norm_w"], db["k_norm_w"], db["pos"],
                             db["seg_offsets"], out=ob, lse=lb)
        ev["fwd"][b].record(stream)
        stream.wait_event(ev["in_bwd"][b])
        h.backward(db["q"], db["k"], db["v"], db["q_norm_w"], db["k_norm_w"], db["pos"], db["seg_offsets"],
                   out, lse, db["dout"], grads=gb)
        ev["done"][b].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(ev["fwd"][b])  # out comes down while the backward runs
            host_out["out"].copy_(out, non_blocking=True)
            down.wait_event(ev["done"][b])
            for k in ("dq", "dk", "dv", "dq_norm_w", "dk_norm_w"):
                host_out[k].copy_(gb[k], non_blocking=True)
            ev["read"][b].record(down)

    for n in range(3):
        e2e_step(n)
    torch.cuda.synchronize()
    barrier(ws)
    e0.record(stream)
    up.wait_stream(stream)
    for n in range(args.steps):
        e2e_step(n)
    stream.wait_stream(down)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = barrier_max(e0.elapsed_time(e1), ws)
    e2e_value = whole_job_tflops(step_flops, args.steps, ws, e2e_ms)
    h.check()

    # ---- roofline of the dominant kernel (stage timing over the timed region)
    pk = peaks()
    L2 = [L * L for L in inp.meta["lengths"]]
    unit = 2.0 * H * 128 * float(sum(L2))  # one S-shaped GEMM over the batch
    algo = {"fwd": 2 * unit, "bwd_dkdv": 4 * unit, "bwd_dq": 1 * unit}
    kern = max(("fwd", "bwd_dkdv", "bwd_dq"), key=lambda k: stages[k][0])
    kms = stages[kern][0] / max(stages[kern][1], 1)
    ach = algo[kern] / (kms * 1e-3) / 1e12
    roof = {"kernel": kern, "bound": "tensor", "achieved": round(ach, 2), "peak": pk["bf16_tflops"],
            "unit": "TFLOP/s", "frac": round(ach / pk["bf16_tflops"], 4), "traffic": measured_traffic(kern),
            "peak_source": f"{pk['source']} bf16 burst", "traffic_note": traffic_note(kern),
            "frac_of_sustained": round(ach / pk["bf16_tflops_sustained"], 4)}
    fwd_ms_launch = stages["fwd"][0] / max(stages["fwd"][1], 1)
    fwd_ach = algo["fwd"] / (fwd_ms_launch * 1e-3) / 1e12
    fwd_roof = {"kernel": "fwd", "bound": "tensor", "achieved": round(fwd_ach, 2), "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(fwd_ach / pk["bf16_tflops"], 4), "traffic": measured_traffic("fwd")}
    pro_ms = stages["prologue"][0] / max(stages["prologue"][1], 1)
    pro_bytes = 8.0 * S * H * 128  # q, k read (bf16) + q^, k^ written (bf16)
    prologue = {"bound": "hbm", "achieved": round(pro_bytes / (pro_ms * 1e-3) / 1e9, 1), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(pro_bytes / (pro_ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                "traffic": measured_traffic("prologue"), "ms": round(pro_ms, 4)}
    launches_per_step = 3 + 8  # forward: plan, prologue, attention; backward: plan, delta, dK/dV, rotary
    #                             table, dQ (with the row backward beside its products: dS is stored), dw per
    #                             (sample, head), dw per sample, dw total (the backward reuses the forward's
    #                             q^/k^, so it runs no prologue)

    # ---- the projections either side of the path (h3attn_linear), same tokens, D = H * 128
    projection = projection_rate(S, H * 128, stream, pk)

    # ---- the QKV projection with the norm/RoPE fused in, then the forward
    qkv = qkv_rate(H, S, d, stream)

    # ---- the canonical key order (packing-permutation-invariant sums), same step
    canonical = canonical_rate(H, S, d, grads, step_flops, ms_max / args.steps, stream)

    # ---- CPU baseline: the oracle as it stands, bounded sample, rank 0 only
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(H)

    result = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "samples": inp.meta["lengths"], "heads": H, "head_dim": 128,
                   "total_tokens": S, "step": "forward + backward (attention core, norm/RoPE prologue, "
                   "norm-weight gradients)", "flops_per_step": step_flops,
                   "l2": "inputs larger than L2 (q, k, v, dO 166 MB each)", "parallelism": f"replicas x{ws}",
                   "qk_hat": "rotated q/k rows computed once per step by the forward, reused by the backward",
                   "stage_times": "a second pass of the same steps with every launch bracketed by CUDA events "
                                  "(the headline region has two events only)"},
        "fwd_tflops_batch": round(fwd_flops / (fwd_ms / args.steps * 1e-3) / 1e12, 2) if fwd_ms else None,
        "fwd_per_sample": per_sample,
        "stages_ms_per_step": {k: round(v[0] / args.steps, 4) for k, v in stages.items()},
        "roofline": roof, "fwd_roofline": fwd_roof, "prologue_roofline": prologue, "projection": projection,
        "canonical_order": canonical,
        "qkv_forward": qkv,
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / args.steps, 4),
                "pipelining": "inputs up and results down on two copy streams beside the kernels, "
                              "double-buffered device tensors; dO goes up after the forward's inputs and "
                              "out comes down while the backward runs"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(result))
    h.close()
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def cpu_baseline(H):
    """The FP64 oracle on the host cores: forward + backward of one 4253-token
    sample of the workload with a third of its heads (about 10-20 s of CPU work)."""
    import oracle
    w = W.WORKLOADS[WORKLOAD]
    H = max(1, H // 3)
    inp = W.make_inputs([W.S4253], H, seed=w.seed + 1, with_grad=True)
    L = inp.total_tokens
    flops = 3.5 * 4.0 * H * 128 * L * L
    t0 = time.perf_counter()
    oracle.forward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets)
    oracle.backward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets, inp.dout)
    t = time.perf_counter() - t0
    return {"value": round(flops / t / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": round(t, 2),
            "sample": f"oracle forward + backward of one {L}-token sample of the workload layout, H={H}, FP64"}


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import oracle
    w = W.WORKLOADS[WORKLOAD]
    H = w.num_heads
    inp = W.make_inputs([W.S925], H, seed=w.seed + 1, with_grad=True)
    L = inp.total_tokens
    flops = 3.5 * 4.0 * H * 128 * L * L

    def step():
        oracle.forward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets)
        oracle.backward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets, inp.dout)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    t = time.perf_counter() - t0
    value = flops * args.steps / t / 1e12
    cores = oracle.num_threads()
    sample = f"one {L}-token sample of the {WORKLOAD} workload per step (forward + backward, H={H}, FP64)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "samples": [L], "heads": H, "head_dim": 128},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="run warm-up + steps only (a fixed launch sequence for ncu); prints no bench line")
    ap.add_argument("--profile-workload", default=None, choices=sorted(W.WORKLOADS),
                    help="with --profile: a smaller workload than the bench's, for multi-pass ncu captures")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours" and not args.profile:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
