"""Benchmark of the fused mixed-precision Any-Precision MoE layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pw|reference]
                    [--workload NAME] [--tokens T] [--offload] [--sweep PATH]

One step = one pass of the hot path over one batch: top-k routing and the
fused expert layer (gather, gate_up at each block's committed bitwidth,
SiLU*mul, down, top-k weighted combine).  On the decode path both run in one
launch (pw_moe_route_apl_ffn); on the prefill path routing is its own launch
(pw_moe_route_topk) before the fused layer (pw_moe_apl_ffn), so that the
timed kernel is the fused layer alone.
Weights are resident in HBM (bit-planes + LUTs, packed once before timing).
The default workload is the Mixtral-8x7B-shaped decode layer (H 4096, I 14336,
8 experts, top-2, 32 tokens, per-block bitwidths uniform on 3..8).

Prints ONE JSON line on rank 0.  Under torchrun every rank runs an independent
replica of the workload on its own GPU (the path has no exchange step);
``value`` is the tokens of all ranks over the slowest rank's time.

``--impl reference`` times the CPU oracle (numpy, float64) on the host cores
on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import signal
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from any_precision_bit_pw_gb300 import synth  # noqa: E402

METRIC = "MoE APL layer tokens/s; achieved HBM GB/s vs ~8 TB/s peak per bitwidth"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = synth.MIXTRAL_8X7B_DECODE.name


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _tensor_peak():
    """Dense fp16 tensor peak in TFLOP/s: the measured bf16 cuBLAS figure
    (fp16 and bf16 share the nominal rate), sustained (the kernel is timed
    inside a long loop)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), "measured sustained bf16 cuBLAS (fp16 same nominal rate)"
    except Exception:
        return 1700.0, "fallback sustained"


def source_digest(paths) -> str:
    """sha256 of the code in `paths` with comments and blank space removed (a
    comment edit does not change the kernel the record was taken on)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for path in paths:
        with open(path) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("\n".join(line.strip() for line in text.splitlines() if line.strip()).encode())
    return h.hexdigest()


def measured_traffic(kernel: str, workload: str, tokens: int):
    """DRAM bytes per launch of `kernel` on `workload` at `tokens` from the
    committed ncu record (profiles/traffic.json), or None when there is no
    record or the kernel's code changed since it was taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            recs = json.load(f)[kernel]
        for rec in recs:
            if rec["workload"] != workload or int(rec["tokens"]) != tokens:
                continue
            paths = [os.path.join(ROOT, "any_precision_bit_pw_gb300", "csrc", n) for n in rec["source_files"]]
            return float(rec["dram_bytes_per_launch"]) if source_digest(paths) == rec["source_sha256"] else None
        return None
    except (OSError, KeyError, ValueError, TypeError):
        return None


def get_workload(name: str, tokens=None, bits=None):
    """A named workload, with its token count replaced when `tokens` is given
    and every block committed at `bits` when that is given."""
    wl = synth.WORKLOADS[name]
    if tokens:
        wl = wl.with_(tokens=tokens)
    if bits:
        wl = wl.with_(bits_mode="fixed", fixed_bits=bits)
    return wl


def ffn_kernel(tokens: int, top_k: int, experts: int) -> str:
    """The fused-layer kernel pw_moe_apl_ffn picks for this size (token-tile
    width from the average tokens per expert, as in the library)."""
    A = tokens * top_k
    return "apl_ffn_t16_kernel" if A < 12 * experts else ("apl_ffn_t64_kernel" if A < 96 * experts
                                                           else "apl_ffn_t128_kernel")


def prefill_path(tokens: int, top_k: int, experts: int) -> bool:
    """The library's path choice between the decode and prefill layouts."""
    return tokens * top_k >= 48 * experts


def kernel_routes(tokens: int, top_k: int, experts: int) -> bool:
    """Whether a routed call routes inside the fused launch (one warp: at most
    32 tokens, 8 experts and 4 slots per token, on the decode path); other
    batches get a routing launch of their own first."""
    return not prefill_path(tokens, top_k, experts) and tokens <= 32 and experts <= 8 and top_k <= 4


KERNEL_TILE = {"apl_ffn_t16_kernel": 16, "apl_ffn_t64_kernel": 64, "apl_ffn_t128_kernel": 128}


def kernel_label(name: str) -> str:
    return f"{name} (pw_moe_apl_ffn, {KERNEL_TILE[name]}-token tiles)"


def layer_call(pw, stack, call, layer, x, logits, mass, ev, stream, routed: bool) -> None:
    """One layer call of a timed step; `ev` (start, stop) brackets the fused
    kernel's launch."""
    r, sh = call.route, stack
    opts = None
    if sh.shared:
        opts = pw.pw_ffn_options()
        opts.shared_experts = sh.shared
    if routed:
        ev[0].record(stream)
        pw.pw_moe_route_apl_ffn(stack.desc, layer, x, logits, sh.I, sh.routed, sh.k, r.ids, r.w, r.offsets, r.perm,
                                r.inv_perm, mass, call.ws, call.y, call.status, options=opts)
        ev[1].record(stream)
    else:
        pw.pw_moe_route_topk_shared(logits, sh.k, sh.shared, r.ids, r.w, r.offsets, r.perm, r.inv_perm, mass)
        ev[0].record(stream)
        pw.pw_moe_apl_ffn(stack.desc, layer, x, sh.I, sh.E, sh.k + sh.shared, r.ids, r.w, r.offsets, r.perm,
                          r.inv_perm, call.ws, call.y, call.status)
        ev[1].record(stream)


def algorithmic_flops(wl, offsets):
    """2 * A * (2I*H + H*I): the gate_up and down contractions of every assignment."""
    sh = wl.shape
    A = int(offsets[-1])
    return 2.0 * A * (2 * sh.intermediate * sh.hidden + sh.hidden * sh.intermediate)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.send_signal(signal.SIGTERM)
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest replica's time: every rank contributes its own timed-region
    milliseconds and all get the maximum (the job finishes with its slowest
    replica)."""
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job tokens/s: the tokens of all replicas over the slowest one's time."""
    return tokens_per_step * steps * world / (max_ms * 1e-3)


def algorithmic_bytes(wl, bits, offsets):
    """Bytes one fused-layer launch must move: the committed planes and LUT_q
    of every block of every active expert, x, y and the h write + read."""
    sh = wl.shape
    H, I, E, k = sh.hidden, sh.intermediate, sh.total_experts, sh.top_k + sh.shared   # all experts, slots
    T = int(offsets[-1]) // k
    planes = luts = 0
    for e in range(E):
        if offsets[e + 1] > offsets[e]:
            for u, (N, K) in ((0, (2 * I, H)), (1, (H, I))):
                q = bits[2 * e + u]
                planes += q * N * K // 8
                luts += N * (1 << q) * 2
    other = 2 * T * H + 2 * T * H + 2 * 2 * T * k * I
    return planes + luts + other, planes, luts


def gpu_arm(args, rank, world, local_rank):
    from any_precision_bit_pw_gb300 import pw
    from any_precision_bit_pw_gb300.layer import APLMoEStack, MoECall, load_layer

    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    pw.lib()
    wl = get_workload(args.workload, args.tokens, args.bits)
    sh = wl.shape
    li = synth.layer_inputs(wl, device=dev)
    stack = APLMoEStack(sh.hidden, sh.intermediate, sh.experts, sh.top_k, 1, wl.parent_bits, wl.seed_bits, dev,
                        shared=sh.shared)
    load_layer(stack, 0, li)
    stack.sync()
    del li.idx
    n_batches = 4
    xs = [synth.activations(wl, 0, s, dev) for s in range(n_batches)]
    lgs = [synth.router_logits(wl, 0, s, dev) for s in range(n_batches)]
    call = MoECall(stack, wl.tokens)
    stream = torch.cuda.current_stream()
    kname = ffn_kernel(wl.tokens, sh.top_k + sh.shared, sh.total_experts)
    routed = kernel_routes(wl.tokens, sh.top_k + sh.shared, sh.total_experts)

    # routing of each batch (for the algorithmic byte count)
    bytes_per_batch = []
    offsets_per_batch = []
    for s in range(n_batches):
        call(0, xs[s], lgs[s])
        torch.cuda.synchronize()
        off = call.route.offsets.cpu().numpy()
        offsets_per_batch.append(off)
        bytes_per_batch.append(algorithmic_bytes(wl, li.bits, off))
    assert int(call.status.item()) == 0, "device status after warm-up calls"

    for i in range(args.warmup):
        call(0, xs[i % n_batches], lgs[i % n_batches])
    torch.cuda.synchronize()

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    smi_index = vis.split(",")[local_rank] if vis and len(vis.split(",")) > local_rank else str(local_rank)
    with ClockSampler(smi_index) as clk:
        start.record(stream)
        for i in range(K):
            s = i % n_batches
            layer_call(pw, stack, call, 0, xs[s], lgs[s], call.mass[0], ev[i], stream, routed)
        stop.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = start.elapsed_time(stop)
    ffn_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    status = int(call.status.item())

    # end-to-end through the C ABI with pinned host buffers
    T, H, E = wl.tokens, sh.hidden, sh.experts
    hx = [x.cpu().pin_memory() for x in xs]
    hl = [l.cpu().pin_memory() for l in lgs]
    hy = torch.empty((T, H), dtype=torch.float16).pin_memory()
    dx = torch.empty_like(xs[0])
    dl = torch.empty_like(lgs[0])
    K2 = max(1, min(K, 200))
    for i in range(3):
        dx.copy_(hx[i % n_batches], non_blocking=True)
        dl.copy_(hl[i % n_batches], non_blocking=True)
        y = call(0, dx, dl)
        hy.copy_(y, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(K2):
        dx.copy_(hx[i % n_batches], non_blocking=True)
        dl.copy_(hl[i % n_batches], non_blocking=True)
        y = call(0, dx, dl)
        hy.copy_(y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / K2

    total_ms = max_over_ranks(total_ms, world, dev)

    mean_bytes = float(np.mean([b[0] for b in bytes_per_batch]))
    mean_planes = float(np.mean([b[1] for b in bytes_per_batch]))
    ffn_avg_ms = float(np.mean(ffn_ms))
    achieved = mean_bytes / (ffn_avg_ms * 1e-3) / 1e9
    peak, peak_kind = _peaks()
    prefill = prefill_path(wl.tokens, sh.top_k + sh.shared, sh.total_experts)
    hbm_roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": measured_traffic(kname, wl.name, wl.tokens),
                "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
                "kernel": kernel_label(kname),
                "algorithmic_bytes_per_launch": mean_bytes, "plane_bytes_per_launch": mean_planes,
                "launch_ms": ffn_avg_ms, "peak_kind": f"{peak_kind} HBM copy (MEASURED_PEAKS.json hbm_gbs)"}
    roofline = hbm_roof
    if prefill:
        flops = float(np.mean([algorithmic_flops(wl, o) for o in offsets_per_batch]))
        tpk, tkind = _tensor_peak()
        ach_t = flops / (ffn_avg_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": ach_t, "peak": tpk, "unit": "TFLOP/s", "frac": ach_t / tpk,
                    "traffic": measured_traffic(kname, wl.name, wl.tokens),
                    "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
                    "kernel": kernel_label(kname),
                    "algorithmic_flops_per_launch": flops, "launch_ms": ffn_avg_ms, "peak_kind": tkind}
    clocks = clk.summary()
    value = job_throughput(wl.tokens, K, world, total_ms)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic (seeded; bit-plane indices uniform, LUTs sorted N(0,0.02), x N(0,1))",
        "config": line_config(wl, li.bits, world),
        "roofline": roofline,
        "roofline_hbm": hbm_roof if prefill else None,
        "e2e": {"value": wl.tokens / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": T * H * 2 + T * E * 4, "d2h_bytes_per_step": T * H * 2},
        "gpu_launches": (1 if routed else 2) * K,
        "clocks": clocks,
        "status": status,
    }
    return line


def stack_arm(args, rank, world, local_rank):
    """The 32-layer decode stack: every step runs routing + the fused layer
    for each of the L layers on fresh seeded inputs -- all layers in one
    launch (pw_moe_route_apl_ffn_layers), or with --per-layer one launch per
    layer; every 8 steps the step boundary reads the accumulated routing
    mass, lowers blocks to the byte target and releases their pages (all
    inside the timed region)."""
    from any_precision_bit_pw_gb300 import pw
    from any_precision_bit_pw_gb300.stack import StackRun

    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    pw.lib()
    wl = get_workload(args.workload, args.tokens, args.bits)
    sh = wl.shape
    T, H, E, L = wl.tokens, sh.hidden, sh.experts, wl.layers
    batched = not args.per_layer
    run = StackRun(wl, dev, commit_every=synth.STACK_COMMIT_EVERY,
                   n_commits=synth.STACK_STEPS // synth.STACK_COMMIT_EVERY - 1, offload=args.offload,
                   batched=batched)
    f8 = run.schedule.f8
    K = args.steps
    n_in = min(K, 16)
    xs = [[synth.activations(wl, l, s, dev) for l in range(L)] for s in range(n_in)]
    lgs = [[synth.router_logits(wl, l, s, dev) for l in range(L)] for s in range(n_in)]
    if batched:
        xs_b = [torch.stack(xs[s]).contiguous() for s in range(n_in)]
        lgs_b = [torch.stack(lgs[s]).contiguous() for s in range(n_in)]
    call, stack = run.call, run.stack
    stream = torch.cuda.current_stream()
    routed = kernel_routes(T, sh.top_k, E)

    # warm-up: the layer calls without step boundaries (no commits, no mass)
    for i in range(args.warmup):
        if batched:
            run.layers_call(0, xs_b[i % n_in], lgs_b[i % n_in])
        else:
            for l in range(L):
                call(l, xs[i % n_in][l], lgs[i % n_in][l], accumulate_mass=False)
    torch.cuda.synchronize()
    call.mass.zero_()

    n_ev = 1 if batched else L
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_ev)]
          for _ in range(K)]
    bits_at = []            # committed bits of every block during each step
    resident = []
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    released_total = 0
    commits = 0
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    smi_index = vis.split(",")[local_rank] if vis and len(vis.split(",")) > local_rank else str(local_rank)
    r = call.route
    with ClockSampler(smi_index) as clk:
        start.record(stream)
        for i in range(K):
            bits_at.append([stack.committed_bits(b) for b in range(stack.n_blocks)])
            resident.append(stack.resident_bytes())
            s = i % n_in
            if batched:
                ev[i][0][0].record(stream)
                run.layers_call(0, xs_b[s], lgs_b[s], mass=call.mass)
                ev[i][0][1].record(stream)
            else:
                for l in range(L):
                    layer_call(pw, stack, call, l, xs[s][l], lgs[s][l], call.mass[l], ev[i][l], stream, routed)
            run.step_no += 1
            plan, released = run.boundary()
            released_total += released
            commits += bool(plan)
        if args.offload:
            stream.wait_stream(run.copy_stream)   # copies that did not overlap count against the steps
        stop.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = start.elapsed_time(stop)
    ffn_ms = np.array([[ev[i][l][0].elapsed_time(ev[i][l][1]) for l in range(n_ev)] for i in range(K)])
    status = run.status()

    # algorithmic bytes of each launch: replay the routing (deterministic) untimed
    nbytes = np.zeros((K, L))
    for i in range(K):
        for l in range(L):
            pw.pw_moe_route_topk(lgs[i % n_in][l], sh.top_k, r.ids, r.w, r.offsets, r.perm, r.inv_perm, None)
            off = r.offsets.cpu().numpy()
            bl = bits_at[i][2 * E * l: 2 * E * (l + 1)]
            nbytes[i, l] = algorithmic_bytes(wl, bl, off)[0]

    # end to end: per step, every layer's x and logits from pinned host
    # memory and every layer's y back to it
    K2 = max(1, min(K, 8))
    hx = [[xs[s][l].cpu().pin_memory() for l in range(L)] for s in range(min(n_in, 2))]
    hl = [[lgs[s][l].cpu().pin_memory() for l in range(L)] for s in range(min(n_in, 2))]
    hy = torch.empty((L, T, H), dtype=torch.float16).pin_memory()
    dx, dl = torch.empty_like(xs[0][0]), torch.empty_like(lgs[0][0])
    if batched:
        hx = [torch.stack(h).pin_memory() for h in hx]
        hl = [torch.stack(h).pin_memory() for h in hl]
        dx, dl = torch.empty_like(xs_b[0]), torch.empty_like(lgs_b[0])
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(K2):
        s = i % len(hx)
        if batched:
            dx.copy_(hx[s], non_blocking=True)
            dl.copy_(hl[s], non_blocking=True)
            hy.copy_(run.layers_call(0, dx, dl), non_blocking=True)
            continue
        for l in range(L):
            dx.copy_(hx[s][l], non_blocking=True)
            dl.copy_(hl[s][l], non_blocking=True)
            hy[l].copy_(call(l, dx, dl, accumulate_mass=False), non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / K2

    total_ms = max_over_ranks(total_ms, world, dev)
    peak, peak_kind = _peaks()
    achieved = float(nbytes.sum() / (ffn_ms.sum() * 1e-3) / 1e9)
    per_launch = nbytes.sum(axis=1) if batched else nbytes.reshape(-1)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": None, "kernel": kernel_label(ffn_kernel(T, sh.top_k, E)),
                "launch": (("all layers of a step in one launch" if routed else
                            "a routing launch, then all layers of a step in one launch") if batched
                           else "one launch per layer"),
                "algorithmic_bytes_per_launch": float(per_launch.mean()), "launch_ms": float(ffn_ms.mean()),
                "layer_ms": float(ffn_ms.sum() / (K * L)),
                "peak_kind": f"{peak_kind} HBM copy (MEASURED_PEAKS.json hbm_gbs)"}
    value = job_throughput(T, K, world, total_ms)
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic (seeded; bit-plane indices uniform, LUTs sorted N(0,0.02), x N(0,1), "
                                "router logits N(0,1) + per-expert N(0,1) bias)",
        "config": {"workload": wl.name, "layers": L, "hidden": H, "intermediate": sh.intermediate, "experts": E,
                   "top_k": sh.top_k, "tokens": T, "parent_bits": wl.parent_bits, "seed_bits": wl.seed_bits,
                   "commit_every": synth.STACK_COMMIT_EVERY, "commits_in_timed_region": commits,
                   "released_bytes": released_total, "resident_bytes_first_last": [resident[0], resident[-1]],
                   "offload": ({"d2h_bytes": run.offloaded_bytes, "pinned_arena_bytes": int(run.arena.numel()),
                                "copy_stream": "separate; the stop event waits for it"} if args.offload else None),
                   "f8_bytes": f8, "parallelism": f"replicas x{world}",
                   "l2": "no flush: the planes read per step (%.1f GB) exceed the 129 MB L2" % (nbytes.sum() / K / 1e9)},
        "roofline": roofline,
        "e2e": {"value": T / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": L * (T * H * 2 + T * E * 4), "d2h_bytes_per_step": L * T * H * 2,
                "steps": K2, "bits": "those of the schedule's last commit (after the timed steps), without "
                                    "step boundaries: fewer plane bytes per step than the timed steps' mean"},
        "gpu_launches": (1 if routed else 2) * (1 if batched else L) * K,
        "clocks": clk.summary(),
        "status": status,
    }


def sweep(args, dev, out_path):
    """Uniform-bitwidth sweep (b x T) of the fused layer: tokens/s, GB/s and
    fraction of the HBM roofline per point.  Writes JSON to ``out_path``."""
    from any_precision_bit_pw_gb300 import pw
    from any_precision_bit_pw_gb300.layer import APLMoEStack, MoECall, load_layer
    base = synth.MIXTRAL_8X7B_SWEEP
    sh = base.shape
    peak, _ = _peaks()
    li8 = synth.layer_inputs(base.with_(fixed_bits=8), device=dev)
    results = []
    for b in synth.SWEEP_BITS:
        wl = base.with_(fixed_bits=b)
        li8.bits = synth.committed_bits(wl)
        stack = APLMoEStack(sh.hidden, sh.intermediate, sh.experts, sh.top_k, 1, wl.parent_bits, wl.seed_bits, dev)
        load_layer(stack, 0, li8)
        stack.sync()
        for T in synth.SWEEP_TOKENS:
            call = MoECall(stack, T)
            x = synth.activations(wl, 0, 0, dev, tokens=T)
            lg = synth.router_logits(wl, 0, 0, dev, tokens=T)
            for _ in range(5):
                call(0, x, lg)
            torch.cuda.synchronize()
            off = call.route.offsets.cpu().numpy()
            nbytes, planes, _ = algorithmic_bytes(wl.with_(tokens=T), li8.bits, off)

            def timed(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(reps):
                    pw.pw_moe_apl_ffn(stack.desc, 0, x, sh.intermediate, sh.experts, sh.top_k, call.route.ids,
                                      call.route.w, call.route.offsets, call.route.perm, call.route.inv_perm,
                                      call.ws, call.y, call.status)
                e1.record()
                torch.cuda.synchronize()
                return e0.elapsed_time(e1) / reps
            # enough launches for about half a second, with the clocks sampled meanwhile
            reps = max(50, int(500.0 / max(timed(10), 1e-3)))
            with ClockSampler(args.smi_index) as clk:
                ms = timed(reps)
            gbs = nbytes / (ms * 1e-3) / 1e9
            results.append({"bits": b, "tokens": T, "kernel": ffn_kernel(T, sh.top_k, sh.experts),
                            "path": "prefill" if prefill_path(T, sh.top_k, sh.experts) else "decode",
                            "ffn_ms": ms, "launches": reps, "tokens_per_s": T / (ms * 1e-3),
                            "algorithmic_bytes": nbytes, "plane_bytes": planes,
                            "algorithmic_GBps": gbs, "plane_GBps": planes / (ms * 1e-3) / 1e9,
                            "frac_of_measured_hbm": gbs / peak, "clocks": clk.summary(),
                            "status": int(call.status.item())})
            print(json.dumps(results[-1]), file=sys.stderr)
        del stack
        torch.cuda.empty_cache()
    with open(out_path, "w") as f:
        json.dump(results, f, indent=1)


# ---------------------------------------------------------------------------
# the reference arm / CPU baseline: the oracle on the host cores
# ---------------------------------------------------------------------------
REF_BUDGET_S = 210.0    # the reference arm's warm-up + timed steps end within about this


def line_config(wl, bits, world: int) -> dict:
    """The ``config`` object of a single-layer bench line (both arms)."""
    sh = wl.shape
    return {"workload": wl.name, "hidden": sh.hidden, "intermediate": sh.intermediate, "experts": sh.experts,
            "shared_experts": sh.shared, "top_k": sh.top_k, "tokens": wl.tokens, "parent_bits": wl.parent_bits,
            "seed_bits": wl.seed_bits, "committed_bits": list(bits), "parallelism": f"replicas x{world}",
            "l2": "no flush: each step streams the committed planes of the active experts, "
                  "hundreds of MB, above the 129 MB L2"}


def oracle_workers(workload: str, tokens=None, bits=None):
    """The oracle's layer on the host cores: one process per active expert,
    each holding its expert's gate_up and down blocks as packed bit-planes at
    the committed bitwidths (seeded CPU draws of the workload's
    distributions)."""
    from oracle import apl, parallel
    wl = get_workload(workload, tokens, bits)
    sh = wl.shape
    x = synth.activations(wl).numpy()
    r = apl.route_topk_shared(synth.router_logits(wl).numpy(), sh.top_k, sh.shared)
    active = sorted({int(e) for e in r["ids"].ravel()})
    files = parallel.ExpertFiles()
    for e in active:
        for u in (0, 1):
            q = synth.committed_bits(wl)[2 * e + u]
            files.add(e, u, synth.parent_indices(wl, 0, e, u).numpy(), synth.lut(wl, 0, e, u, q).numpy(), q)
    ew = parallel.ExpertWorkers(files, x, r["ids"], r["w"], sh.intermediate, wl.parent_bits)
    return wl, files, ew


def _sample_text(wl, ew, frac: float) -> str:
    part = "the whole layer" if frac >= 1.0 else f"the first {frac:.4f} of every block's rows of the layer"
    per = "; one layer of the {} per step".format(wl.layers) if wl.layers > 1 else ""
    return (f"{part}: {len(ew.experts)} active experts' gate_up ({2 * wl.shape.intermediate}x{wl.shape.hidden}) "
            f"and down ({wl.shape.hidden}x{wl.shape.intermediate}) read from packed bit-planes, one process per "
            f"expert on {ew.cores} host cores ({ew.threads_per_worker} BLAS threads each){per}")


def oracle_baseline(workload: str, tokens=None, passes: int = 1, bits=None) -> dict:
    """CPU baseline: wall time of whole-layer oracle passes (one by default:
    a pass of the 8x7B layer is about 20 s of CPU work); tokens/s of the job
    step (a stack step is its layers one after another, so its time is the
    layer's times the layer count)."""
    wl, files, ew = oracle_workers(workload, tokens, bits)
    try:
        times = [ew.step(1.0) for _ in range(passes)]
    finally:
        ew.close()
        files.close()
    layer_s = float(np.median(times))
    return {"value": wl.tokens / (layer_s * wl.layers), "layer_s": layer_s, "pass_s": times, "cores": ew.cores,
            "sample": _sample_text(wl, ew, 1.0) + (f"; median of {passes} passes" if passes > 1 else "; one pass")}


def oracle_reference_steps(workload: str, steps: int, warmup: int, tokens=None, bits=None) -> dict:
    """The reference arm's steps: each step is a timed oracle pass over the
    layer (every active expert at once, as in oracle_baseline), or, when K + W
    whole-layer passes would not end within REF_BUDGET_S, over the same first
    fraction of every block's rows.  A step processes that fraction of the
    job step (one layer of a stack step), so the line's tokens/s is
    T * fraction / step time."""
    wl, files, ew = oracle_workers(workload, tokens, bits)
    try:
        t_full = ew.step(1.0)
        n = max(1, steps) + max(0, warmup)
        frac = 1.0 if n * t_full <= REF_BUDGET_S else max(REF_BUDGET_S / (n * t_full), 1e-4)
        for _ in range(max(0, warmup)):
            ew.step(frac)
        times = [ew.step(frac) for _ in range(max(1, steps))]
    finally:
        ew.close()
        files.close()
    return {"step_s": times, "frac": frac / wl.layers, "cores": ew.cores, "sample": _sample_text(wl, ew, frac)}


def _child_cmd(workload: str, tokens=None, bits=None) -> list:
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-baseline-child", "--workload", workload]
    if tokens:
        cmd += ["--tokens", str(tokens)]
    if bits:
        cmd += ["--bits", str(bits)]
    return cmd


def _child_env() -> dict:
    return dict(os.environ, CUDA_VISIBLE_DEVICES="")


def cpu_baseline(workload: str, tokens=None, bits=None) -> dict:
    """The oracle's whole layer on the host cores, in a child process started
    before this process touches the GPU."""
    r = subprocess.run(_child_cmd(workload, tokens, bits), env=_child_env(), capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        return {"value": None, "unit": UNIT, "cores": None, "kind": "oracle", "sample": "failed: " + r.stderr[-300:]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": d["value"], "unit": UNIT, "cores": d["cores"], "kind": "oracle", "sample": d["sample"],
            "layer_s": d["layer_s"]}


def reference_arm(args, rank, world):
    if rank != 0:
        return None
    wl = get_workload(args.workload, args.tokens, args.bits)
    cmd = _child_cmd(args.workload, args.tokens, args.bits) + ["--steps", str(max(1, args.steps)), "--warmup",
                                                    str(max(0, args.warmup)), "--reference-child"]
    r = subprocess.run(cmd, env=_child_env(), capture_output=True, text=True, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError("oracle child failed: " + r.stderr[-500:])
    d = json.loads(r.stdout.strip().splitlines()[-1])
    times = d["step_s"]
    step_s = float(np.mean(times))
    value = wl.tokens * d["frac"] / step_s
    cfg = line_config(wl, synth.committed_bits(wl), world) if wl.layers == 1 else \
        {"workload": wl.name, "layers": wl.layers, "hidden": wl.shape.hidden,
         "intermediate": wl.shape.intermediate, "experts": wl.shape.experts, "top_k": wl.shape.top_k,
         "tokens": wl.tokens, "parent_bits": wl.parent_bits, "seed_bits": wl.seed_bits,
         "parallelism": f"replicas x{world}"}
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": len(times),
            "warmup": args.warmup, "ms_per_step": 1e3 * step_s, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded CPU draws of the same distributions)",
            "impl": "reference", "config": cfg,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": d["cores"], "kind": "oracle",
                             "sample": d["sample"], "fraction_of_job_step": d["frac"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pw", choices=["pw", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--tokens", type=int, default=None, help="replace the workload's token count")
    ap.add_argument("--bits", type=int, default=None,
                    help="commit every block at this bitwidth (from the seed to the parent bitwidth)")
    ap.add_argument("--offload", action="store_true",
                    help="stack workload: lowering copies the released pages to pinned host memory first (§3.3)")
    ap.add_argument("--sweep", default=None, help="also run the uniform-bitwidth sweep, JSON to this path")
    ap.add_argument("--per-layer", action="store_true",
                    help="stack workload: one launch per layer instead of all layers of a step in one launch")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-baseline-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--reference-child", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "pw":
        args.warmup = 3

    if args.cpu_baseline_child and args.reference_child:
        print(json.dumps(oracle_reference_steps(args.workload, args.steps, args.warmup, tokens=args.tokens,
                                                bits=args.bits)))
        return
    if args.cpu_baseline_child:
        print(json.dumps(oracle_baseline(args.workload, tokens=args.tokens, bits=args.bits)))
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        line = reference_arm(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    if not torch.cuda.is_available():
        sys.exit("bench.py: the pw arm runs the CUDA library and needs a GPU (--impl reference times the CPU oracle)")
    # the CPU baseline runs in a child process started before this process touches the GPU
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload, args.tokens, args.bits)
    if world > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    arm = stack_arm if synth.WORKLOADS[args.workload].layers > 1 else gpu_arm
    line = arm(args, rank, world, local_rank)
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if args.sweep and rank == 0:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        args.smi_index = vis.split(",")[local_rank] if vis and len(vis.split(",")) > local_rank else str(local_rank)
        sweep(args, torch.device(f"cuda:{local_rank}"), args.sweep)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
