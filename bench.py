"""Benchmark of the routed-expert MoE layer on GB300.

One step = one pass of the whole hot path over one synthetic batch:
shared-expert forward (BF16, dense), routed forward (route, gather/quantise,
W13 + SwiGLU, W2, combine, accumulated onto the shared output) and, for the
training workloads, the routed and shared backward (dh3 bundles, W2 DGRAD +
SwiGLU backward, W2 WGRAD, W13 DGRAD, W13 WGRAD, dX reduction).  The step is
captured once in a CUDA graph and replayed.

Metric: useful TFLOP/s of the routed expert GEMMs (6 R D F forward, 12 R D F
backward, R = active routes; padding, the shared expert and the router are
not counted, as on the Dist-MoE explainer's "Performance Metrics" panel),
plus tokens/s and the fraction of the dense tensor peak.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
       python bench.py --impl reference ...   (the fp64 oracle on host cores)
Under torchrun each rank runs an independent replica (weak scaling) and the
slowest rank's time is reported.
"""

import argparse
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

METRIC = "useful TFLOP/s and tokens/s per GB300 (fraction of FP8/BF16 tensor peak)"
DEFAULT_WORKLOAD = "e384_mxfp8_zipf_train"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fused", action="store_true")    # MXFP8 inference: the routed forward as one launch
    ap.add_argument("--mn-major", action="store_true")  # MXFP8 training: no transposed weight codes; the
                                                        # input-gradient GEMMs read the forward codes MN-major
    ap.add_argument("--replay", action="store_true")   # training: the routed layer saves only its input and
                                                       # its backward replays the forward (activation slots)
    ap.add_argument("--tied", action="store_true")     # layer stacks: one weight set shared by the layers
    ap.add_argument("--slot-gb", type=float, default=0.0)   # layer stacks: one activation slot of this size
                                                            # holds every layer's saved state (0: full states)
    ap.add_argument("--cpu-sample-experts", type=int, default=3)        # reference arm: experts per step
    ap.add_argument("--cpu-sample-seconds", type=float, default=12.0)   # cpu_baseline: oracle work to time
    ap.add_argument("--cpu-sample-max-experts", type=int, default=384)
    ap.add_argument("--cpu-sample-max-gb", type=float, default=2.0)      # host copy of the sampled BF16 weights
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock and throttle-reason samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            ids = [v.strip() for v in vis.split(",") if v.strip()]
            if self.index < len(ids):
                self.index = ids[self.index]
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------- algorithmic bytes

def stage_bytes(w, rows_padded, routes, precision, train, experts_used=None, dw_bytes=2):
    """Unique bytes each stage must move (read once + written once), per launch.

    rows_padded = sum of expert row counts padded to 32; routes = active
    routes; experts_used = experts with at least one route (the GEMMs read
    only their weights; the weight gradients write dW of every expert).
    MXFP8 operands cost 1 + 1/32 bytes per element (E4M3 + E8M0), NVFP4
    operands 9/16 (E2M1 + one E4M3 scale per 16; inference only: its W13
    stage also writes the FP32 h2 and its quantisation reads it back).
    dw_bytes = bytes moved per weight-gradient element: 2 (BF16 written),
    4 (FP32 written), 8 (FP32 read and written back when accumulating)."""
    T, D, F, E = w.T, w.D, w.F, w.E
    Eu = w.E if experts_used is None else experts_used
    q = {"mxfp8": 1 + 1 / 32, "nvfp4": 9 / 16}.get(precision, 2.0)
    Rp, R = rows_padded, routes
    h2_f32 = Rp * F * 8 if precision == "nvfp4" else 0
    fwd = {
        "route": T * w.K * 8 + (Rp + 2 * T * w.K) * 4,
        "gather_x": T * D * 2 + Rp * D * q * (2 if train else 1),
        "gemm_w13_swiglu": Eu * 2 * F * D * q + Rp * D * q + Rp * F * q + h2_f32
                           + (Rp * 2 * F * 2 + Rp * F * q if train else 0),
        "gemm_w2": Eu * D * F * q + Rp * F * q + Rp * D * 2,
        "combine": R * D * 2 + T * D * 2 * 2,
    }
    bwd = {
        "gather_dh3": T * D * 2 + 2 * Rp * D * q,
        "gemm_w2_dgrad_swiglu_bwd": Eu * D * F * q + Rp * D * q + Rp * 2 * F * 2 + 2 * Rp * 2 * F * q,
        "gemm_w2_wgrad": D * Rp * q + F * Rp * q + E * D * F * dw_bytes,
        "gemm_w13_dgrad": Eu * 2 * F * D * q + Rp * 2 * F * q + Rp * D * 2,
        "gemm_w13_wgrad": 2 * F * Rp * q + D * Rp * q + E * 2 * F * D * dw_bytes,
        "reduce_dx": R * D * 2 + T * D * 2 * 2,
    }
    return fwd, bwd


# useful FLOPs of each grouped GEMM per active route, in units of D * F
GEMM_FLOPS = {"gemm_w13_swiglu": 4.0, "gemm_w2": 2.0, "gemm_w2_dgrad_swiglu_bwd": 2.0, "gemm_w2_wgrad": 2.0,
              "gemm_w13_dgrad": 4.0, "gemm_w13_wgrad": 4.0}


def gemm_tensor(stage_ms, routes, w, peak_t):
    """The grouped GEMMs alone: their useful FLOPs over their own stage
    times against the tensor peak, in total and per GEMM (the step's
    tensor_frac also carries the HBM-bound routing, gather and combine)."""
    ms = {k: v for k, v in stage_ms.items() if k in GEMM_FLOPS and v > 0}
    if not ms:
        return None
    per = {k: round(GEMM_FLOPS[k] * routes * w.D * w.F / (v * 1e-3) / 1e12 / peak_t, 4) for k, v in ms.items()}
    total = sum(GEMM_FLOPS[k] * routes * w.D * w.F for k in ms)
    t = sum(ms.values())
    return {"ms": round(t, 4), "tflops": round(total / (t * 1e-3) / 1e12, 1),
            "tensor_frac": round(total / (t * 1e-3) / 1e12 / peak_t, 4), "per_gemm_tensor_frac": per}


def roofline(kernel, ms, nbytes, routes, w, pk, peak_t, traffic):
    """The dominant kernel against the roof that bounds it: its useful FLOPs
    per algorithmic byte above the ridge (tensor peak / copy bandwidth) put
    it under the tensor roof (TFLOP/s of the dtype's peak), else under HBM."""
    base = {"kernel": kernel, "traffic": traffic, "algorithmic_bytes": int(nbytes), "avg_launch_ms": round(ms, 4),
            "peak_source": pk["source"]}
    flops = GEMM_FLOPS.get(kernel, 0.0) * routes * w.D * w.F
    ridge = peak_t * 1e12 / (pk["hbm_gbs"] * 1e9)
    if flops > 0 and flops / nbytes > ridge:
        achieved = flops / (ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak_t, 1), "unit": "TFLOP/s",
                "frac": round(achieved / peak_t, 4), "flop_per_byte": round(flops / nbytes, 1),
                "ridge_flop_per_byte": round(ridge, 1), **base}
    achieved = nbytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / pk["hbm_gbs"], 4), **base}


def gemm_source_digest():
    """SHA-256 prefix of the GEMM kernels' sources (gemm.cu, gemm_core.cuh,
    common.cuh): a traffic record holds only for the code it was taken on."""
    h = hashlib.sha256()
    for name in ("gemm.cu", "gemm_core.cuh", "common.cuh"):
        h.update(open(os.path.join(ROOT, "mixture_experts_routed_route_gb300", "csrc", name), "rb").read())
    return h.hexdigest()[:16]


def traffic_record(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if its kernel
    source is unchanged since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    digest = gemm_source_digest()
    for line in open(path):
        line = line.strip()
        if not line.startswith("{"):
            continue
        rec = json.loads(line)
        if rec.get("stage") == kernel and rec.get("workload") == workload and rec.get("gemm_src") == digest:
            return rec.get("dram_bytes_per_launch_full")
    return None


# ------------------------------------------------------------ our arm (GPU)

class Step:
    """Inputs, weights, contexts and the captured CUDA graph of one step."""

    def __init__(self, w, device, replay=False, fused=False, mn_major=False):
        import torch
        from mixture_experts_routed_route_gb300 import synth
        from mixture_experts_routed_route_gb300.layer import MoELayer, PreparedWeight

        self.w = w
        self.dev = device
        self.train = w.train
        T, D, F, E, K = w.T, w.D, w.F, w.E, w.K
        ids, scores = synth.make_routing(w)
        self.ids_np, self.scores_np = ids, scores
        self.x = synth.make_tokens(w, device)
        self.dy = synth.make_grad_out(w, device)
        self.ids = torch.from_numpy(ids).to(device)
        self.scores = torch.from_numpy(scores).to(device)
        w13, w2 = synth.make_weights(w, device)
        self.sample_experts = None
        mn = bool(mn_major and self.train and w.precision == "mxfp8")
        self.mn_major = mn
        self.W13 = PreparedWeight(w13, w.precision, with_transpose=self.train, mn_major=mn)
        self.W2 = PreparedWeight(w2, w.precision, with_transpose=self.train, mn_major=mn)
        self.w13_bf16, self.w2_bf16 = w13, w2   # kept only until the oracle sample is taken
        self.replay = bool(replay and self.train)
        self.fused = bool(fused and not self.train and w.precision == "mxfp8")
        self.layer = MoELayer(T, D, F, E, K, w.precision, training=self.train, device=device, replay=self.replay)
        self.saved = self.layer.new_saved(input_only=self.replay) if self.train else None
        self.shared = None
        if w.shared_F:
            sw13, sw2 = synth.make_shared_weights(w, device)
            self.sW13 = PreparedWeight(sw13, "bf16", with_transpose=self.train)
            self.sW2 = PreparedWeight(sw2, "bf16", with_transpose=self.train)
            self.shared = MoELayer(T, D, w.shared_F, 1, 1, "bf16", training=self.train, device=device)
            self.s_ids = torch.zeros((T, 1), dtype=torch.int32, device=device)
            self.s_scores = torch.ones((T, 1), dtype=torch.float32, device=device)
            self.s_saved = self.shared.new_saved() if self.train else None
        self.out = torch.empty((T, D), dtype=torch.bfloat16, device=device)
        if self.train:
            self.dx = torch.empty((T, D), dtype=torch.bfloat16, device=device)
            self.dW13 = torch.empty((E, 2 * F, D), dtype=torch.bfloat16, device=device)
            self.dW2 = torch.empty((E, D, F), dtype=torch.bfloat16, device=device)
            if self.shared:
                self.sdW13 = torch.empty((1, 2 * w.shared_F, D), dtype=torch.bfloat16, device=device)
                self.sdW2 = torch.empty((1, D, w.shared_F), dtype=torch.bfloat16, device=device)
        self.graph = None

    def layers(self):
        return [l for l in (self.layer, self.shared) if l is not None]

    def io_set(self):
        """The step's per-step inputs and outputs (the ones a host feeds and reads)."""
        return {"x": self.x, "ids": self.ids, "scores": self.scores, "dy": self.dy if self.train else None,
                "out": self.out, "dx": self.dx if self.train else None}

    def enqueue(self, io=None):
        """The step, through the public C ABI (enqueue only, no host sync), on
        the step's own buffers or on another set of the same shapes."""
        io = io or self.io_set()
        x, out, dx = io["x"], io["out"], io["dx"]
        acc = False
        if self.shared:
            self.shared.forward(x, self.s_ids, self.s_scores, self.sW13, self.sW2, out=out, saved=self.s_saved)
            acc = True
        self.layer.forward(x, io["ids"], io["scores"], self.W13, self.W2, out=out, saved=self.saved,
                           accumulate=acc, save_input_only=self.replay, fused=self.fused)
        if self.train:
            acc = False
            if self.shared:
                self.shared.backward(self.s_saved, io["dy"], self.sW13, self.sW2, dx=dx, dW13=self.sdW13,
                                     dW2=self.sdW2)
                acc = True
            self.layer.backward(self.saved, io["dy"], self.W13, self.W2, dx=dx, dW13=self.dW13, dW2=self.dW2,
                                accumulate_dx=acc, replay=self.replay)

    def capture(self):
        """Two graphs of the same step: the timed one, and one that also
        records the library's per-stage events (kept out of the timed one)."""
        import torch
        from mixture_experts_routed_route_gb300 import abi
        before = sum(abi.moe_ctx_launch_count(l.ctx) for l in self.layers())
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.enqueue()
        self.launches_per_step = sum(abi.moe_ctx_launch_count(l.ctx) for l in self.layers()) - before
        for l in self.layers():
            abi.moe_ctx_enable_stage_timing(l.ctx, True)
        self.stage_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.stage_graph):
            self.enqueue()
        for l in self.layers():
            abi.moe_ctx_enable_stage_timing(l.ctx, False)

    def rows_used(self):
        from mixture_experts_routed_route_gb300 import abi
        import torch
        if self.train:
            hdr = self.layer.saved_field(self.saved, abi.MOE_SAVED_HEADER, torch.int32, (16,),
                                         input_only=self.replay).cpu().numpy()
        else:
            hdr = self.layer.read_buffer(abi.MOE_BUF_ROUTING, np.int32, (16,))
        return int(hdr[2]), int(hdr[3])


class StackStep:
    """A stack of `w.layers` training layers on one context: every layer's
    forward in order, then the backwards in reverse, captured as one CUDA
    graph.  Each layer has its own routing (Zipf with a per-layer exponent),
    tokens and output gradient.

    Independent weights (the default): each layer has its own MXFP8 weight
    set, prepared without transposed codes (the input-gradient GEMMs read the
    forward codes MN-major), and each backward writes its layer's BF16 weight
    gradients into one pair of buffers that the next backward overwrites (a
    framework consumes each layer's gradient as it is produced).  Tied
    weights: one weight set shared by the layers, whose weight gradients
    accumulate in one FP32 buffer (the first backward writes it).  With
    `slot_bytes`, the saved states share one activation slot and the planner
    decides which layers keep only their input."""

    def __init__(self, w, device, slot_bytes=0, tied=False):
        import torch
        from mixture_experts_routed_route_gb300 import synth
        from mixture_experts_routed_route_gb300.layer import ActivationSlot, MoELayer, PreparedWeight

        self.w, self.dev, self.train = w, device, True
        T, D, F, E, K, L = w.T, w.D, w.F, w.E, w.K, w.layers
        self.tied = tied
        self.W13, self.W2 = [], []
        for l in range(1 if tied else L):
            w13, w2 = synth.make_weights(w, device, layer=l)
            mn = not tied and w.precision == "mxfp8"
            self.W13.append(PreparedWeight(w13, w.precision, with_transpose=True, mn_major=mn))
            self.W2.append(PreparedWeight(w2, w.precision, with_transpose=True, mn_major=mn))
            del w13, w2
            torch.cuda.empty_cache()
        self.layer = MoELayer(T, D, F, E, K, w.precision, training=True, device=device, replay=slot_bytes > 0)
        self.ids_np, self.io = [], []
        for l in range(L):
            ids, scores = synth.make_routing(w, layer=l, zipf_s=synth.layer_zipf_s(w, l))
            self.ids_np.append(ids)
            self.io.append({"ids": torch.from_numpy(ids).to(device), "scores": torch.from_numpy(scores).to(device),
                            "x": synth.make_tokens(w, device, layer=l), "dy": synth.make_grad_out(w, device, layer=l),
                            "out": torch.empty((T, D), dtype=torch.bfloat16, device=device),
                            "dx": torch.empty((T, D), dtype=torch.bfloat16, device=device)})
        dt = torch.float32 if tied else torch.bfloat16
        self.dW13 = torch.empty((E, 2 * F, D), dtype=dt, device=device)
        self.dW2 = torch.empty((E, D, F), dtype=dt, device=device)
        self.slot = None
        if slot_bytes > 0:
            # the decisions depend only on the sizes, so they are taken once
            # here and hold for every replay of the captured graph
            self.slot = ActivationSlot(slot_bytes, max_layers=L, device=device)
            self.states = [self.slot.push(self.layer, L - 1 - l) for l in range(L)]
        else:
            self.states = [(self.layer.new_saved(), False) for _ in range(L)]
        self.graph = None

    def layers(self):
        return [self.layer]

    def weights(self, l):
        return (self.W13[0], self.W2[0]) if self.tied else (self.W13[l], self.W2[l])

    def enqueue(self):
        for l, io in enumerate(self.io):
            saved, input_only = self.states[l]
            W13, W2 = self.weights(l)
            self.layer.forward(io["x"], io["ids"], io["scores"], W13, W2, out=io["out"], saved=saved,
                               save_input_only=input_only)
        for n, l in enumerate(reversed(range(len(self.io)))):
            saved, input_only = self.states[l]
            W13, W2 = self.weights(l)
            self.layer.backward(saved, self.io[l]["dy"], W13, W2, dx=self.io[l]["dx"], dW13=self.dW13, dW2=self.dW2,
                                dw_fp32=self.tied, dw_accumulate=self.tied and n > 0, replay=input_only)

    capture = Step.capture

    def rows_used(self):
        """(padded rows, active routes) of every layer."""
        import torch
        from mixture_experts_routed_route_gb300 import abi
        out = []
        for saved, input_only in self.states:
            hdr = self.layer.saved_field(saved, abi.MOE_SAVED_HEADER, torch.int32, (16,),
                                         input_only=input_only).cpu().numpy()
            out.append((int(hdr[2]), int(hdr[3])))
        return out


def cpu_sample(w, ids, scores, x_cpu, dy_cpu, w13_sub, w2_sub, experts):
    """Time the oracle on a bounded sample (the routes of a few experts)."""
    from oracle import sample as osample
    f64 = lambda t: t.to("cpu").double().numpy()
    xs, dys = f64(x_cpu), (f64(dy_cpu) if w.train else None)
    a13, a2 = f64(w13_sub), f64(w2_sub)
    t0 = time.perf_counter()
    osample.run(xs, ids, scores, a13, a2, experts, w.precision, dY=dys)
    dt = time.perf_counter() - t0
    sub_ids = osample.restrict_routes(ids, experts)
    flops = osample.useful_flops(sub_ids, w.D, w.F, w.train)
    return dt, flops, int(np.sum(sub_ids >= 0))


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count()


def pick_sample_experts(w, ids, n):
    """The first n routed experts of a fixed seeded order (prefixes nest)."""
    rng = np.random.default_rng(12345)
    present = sorted(set(int(e) for e in np.asarray(ids).reshape(-1) if e >= 0))
    order = [present[i] for i in rng.permutation(len(present))]
    return order[:n]


def timed_cpu_sample(w, ids, scores, x, dy, w13s, w2s, experts, target_s):
    """The oracle timed on a sample of about target_s seconds: the experts of
    `experts` (a seeded order) are run one oracle call each, in that order,
    until the calls' total time reaches target_s.  No cost prediction: an
    expert's cost is mostly fixed (its weight preparation and full weight
    gradient), so route counts say little about it.  Returns the totals of
    time, useful FLOPs and routes, and the number of experts run."""
    tot_t, tot_f, tot_r, n = 0.0, 0.0, 0, 0
    while n < len(experts) and (n == 0 or tot_t < target_s):
        dt, fl, r = cpu_sample(w, ids, scores, x, dy, w13s[n:n + 1], w2s[n:n + 1], experts[n:n + 1])
        tot_t, tot_f, tot_r, n = tot_t + dt, tot_f + fl, tot_r + r, n + 1
    return tot_t, tot_f, tot_r, n


def run_ours(args, rank, world):
    import torch
    from mixture_experts_routed_route_gb300 import abi, synth

    w = synth.WORKLOADS[args.workload]
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk = peaks()
    st = Step(w, dev, replay=args.replay, fused=args.fused, mn_major=args.mn_major)

    # eager warm-up (configures kernels), then correctness guard: no device error
    st.enqueue()
    torch.cuda.synchronize(dev)
    for l in st.layers():
        bits = l.error_bits()
        if bits:
            raise RuntimeError(f"device error bits {bits:#x} in warm-up")
    rows_padded, routes = st.rows_used()

    # oracle sample weights (host copies) before the BF16 masters are dropped
    sample = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        per_expert = 3 * w.F * w.D * 2          # W13 + W2 of one expert, BF16
        cap = max(1, min(args.cpu_sample_max_experts, int(args.cpu_sample_max_gb * 1e9) // per_expert))
        experts = pick_sample_experts(w, st.ids_np, cap)
        sample = (experts, st.w13_bf16[experts].cpu(), st.w2_bf16[experts].cpu(), st.x.cpu(), st.dy.cpu())
    st.w13_bf16 = st.w2_bf16 = None
    torch.cuda.empty_cache()

    st.capture()
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        st.graph.replay()
    torch.cuda.synchronize(dev)

    # ---------------- timed region: K graph replays
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        st.graph.replay()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / args.steps
    if world > 1:
        tt = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        ms = float(tt.item())

    # ---------------- per-stage durations (CUDA events inside the graph)
    fwd_t = {n: [] for n in abi.FWD_STAGE_NAMES}
    bwd_t = {n: [] for n in abi.BWD_STAGE_NAMES}
    shared_t = []   # the shared expert's own time per step: its forward (+ backward) stages
    for _ in range(max(3, min(args.steps, 10))):
        st.stage_graph.replay()
        torch.cuda.synchronize(dev)
        for n, v in zip(abi.FWD_STAGE_NAMES, abi.moe_ctx_stage_times(st.layer.ctx, 0)):
            fwd_t[n].append(v)
        if st.train:
            for n, v in zip(abi.BWD_STAGE_NAMES, abi.moe_ctx_stage_times(st.layer.ctx, 1)):
                bwd_t[n].append(v)
        if st.shared:
            t_sh = sum(abi.moe_ctx_stage_times(st.shared.ctx, 0))
            if st.train:
                t_sh += sum(abi.moe_ctx_stage_times(st.shared.ctx, 1))
            shared_t.append(t_sh)
    stage_ms = {k: statistics.mean(v) for k, v in list(fwd_t.items()) + list(bwd_t.items()) if v}
    ids = np.asarray(st.ids_np)
    used = int(np.unique(ids[(ids >= 0) & (ids < w.E)]).size)
    fb, bb = stage_bytes(w, rows_padded, routes, w.precision, st.train, experts_used=used)
    sbytes = {**fb, **(bb if st.train else {})}
    if st.fused:
        # one launch: its time (the forward's first stage event to its last)
        # against the bytes of every forward stage
        stage_ms = {"fused_forward": sum(statistics.mean(fwd_t[n]) for n in abi.FWD_STAGE_NAMES)}
        sbytes = {"fused_forward": sum(fb.values())}
    dom = max(stage_ms, key=lambda k: stage_ms[k])
    fp8_peak = pk["bf16_tflops"] * 2.0
    # NVFP4 operands reach the tensor cores as FP16 (kind::f16): the 16-bit peak
    peak_t = fp8_peak if w.precision == "mxfp8" else pk["bf16_tflops"]
    roof = roofline(dom, stage_ms[dom], sbytes[dom], routes, w, pk, peak_t, traffic_record(dom, w.name))
    stages = {k: {"ms": round(v, 4), "GB/s": round(sbytes[k] / (v * 1e-3) / 1e9, 1) if v > 0 else None}
              for k, v in stage_ms.items()}

    # ---------------- metric
    flops = 6.0 * routes * w.D * w.F * (3.0 if st.train else 1.0)
    tflops = flops / (ms * 1e-3) / 1e12 * world
    shared_flops = (6.0 * w.T * w.D * w.shared_F * (3.0 if st.train else 1.0)) if w.shared_F else 0.0

    # ---------------- end to end through the ABI with host buffers
    # Every step uploads its inputs from pinned host memory and downloads its
    # outputs.  Two device buffer sets and two copy streams pipeline the
    # steps: step i+1's upload and step i-1's download run on the copy
    # engines while step i's kernels run.  The timed region spans the first
    # upload to the last download.
    e2e = None
    if not args.no_e2e:
        io0 = st.io_set()
        ios = [io0, {k: (torch.empty_like(v) if v is not None else None) for k, v in io0.items()}]
        h_in = {k: io0[k].cpu().pin_memory() for k in ("x", "ids", "scores", "dy") if io0[k] is not None}
        h_out = [{k: torch.empty(io0[k].shape, dtype=io0[k].dtype).pin_memory() for k in ("out", "dx")
                  if io0[k] is not None} for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in h_in.values())
        d2h = sum(t.numel() * t.element_size() for t in h_out[0].values())
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        uploaded = [torch.cuda.Event() for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        downloaded = [torch.cuda.Event() for _ in range(2)]

        def e2e_steps(n):
            for i in range(n):
                j = i % 2
                io = ios[j]
                with torch.cuda.stream(up):
                    if i >= 2:
                        up.wait_event(computed[j])        # step i-2 has read this set's inputs
                    for k, t in h_in.items():
                        io[k].copy_(t, non_blocking=True)
                    uploaded[j].record(up)
                stream.wait_event(uploaded[j])
                if i >= 2:
                    stream.wait_event(downloaded[j])      # step i-2's outputs have left this set
                st.enqueue(io)
                computed[j].record(stream)
                with torch.cuda.stream(down):
                    down.wait_event(computed[j])
                    for k, t in h_out[j].items():
                        t.copy_(io[k], non_blocking=True)
                    downloaded[j].record(down)
            for j in range(min(n, 2)):
                stream.wait_event(downloaded[j])

        e2e_steps(2)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        n_e2e = max(3, args.steps // 2)
        e0.record(stream)
        up.wait_event(e0)
        e2e_steps(n_e2e)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ems = e0.elapsed_time(e1) / n_e2e
        if world > 1:
            tt = torch.tensor([ems], device=dev)
            torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
            ems = float(tt.item())
        e2e = {"value": round(flops / (ems * 1e-3) / 1e12 * world, 3), "unit": "TFLOP/s",
               "ms_per_step": round(ems, 4), "tokens_per_s": round(w.T * world / (ems * 1e-3), 1),
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "pipelined": "2 buffer sets; uploads and downloads overlap the neighbouring steps' kernels"}

    # ---------------- oracle baseline on host cores (rank 0, N = 1)
    cpu = None
    if sample is not None:
        experts, s13, s2, xc, dyc = sample
        dt, sflops, sroutes, n = timed_cpu_sample(w, st.ids_np, st.scores_np, xc, dyc, s13, s2, experts,
                                                  args.cpu_sample_seconds)
        cpu = {"value": round(sflops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": blas_threads(),
               "host_cores": os.cpu_count(), "kind": "oracle",
               "sample": f"fp64 numpy oracle, {'forward+backward' if w.train else 'forward'} of the {sroutes} "
                         f"routes of {n} of {w.E} experts, one oracle call per expert (all {w.T} tokens), {dt:.1f} s"}

    line = {
        "metric": METRIC, "value": round(tflops, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.precision, "data": "synthetic",
        "tokens_per_s": round(w.T * world / (ms * 1e-3), 1),
        "tensor_frac": round(tflops / world / peak_t, 4),
        "tensor_peak_tflops": round(peak_t, 1),
        "gemms": None if st.fused else gemm_tensor(stage_ms, routes, w, peak_t),
        "config": {"workload": w.name, "T": w.T, "D": w.D, "F": w.F, "E": w.E, "K": w.K,
                   "routing": w.routing, "inactive_frac": w.inactive_frac, "shared_F": w.shared_F,
                   "train": w.train, "active_routes": routes, "padded_rows": rows_padded,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (expert weights stream from HBM every step)",
                   "graph": "one CUDA graph per step, replayed",
                   **({"forward": "single launch (MOE_FUSED_LAUNCH)"} if st.fused else {}),
                   **({"weights": "MXFP8 without transposed codes (input-gradient GEMMs read them MN-major)"}
                      if st.mn_major else {}),
                   **({"saved_state": ("input only: the backward replays the gather, W13 and W2 GEMMs "
                                       "(their FLOPs not counted as useful)") if st.replay else "full"}
                      if st.train else {})},
        "roofline": roof, "stages": stages,
        # the BF16 shared expert over its own stage time (not counted in `value`)
        "shared_expert": ({"ms": round(statistics.mean(shared_t), 4),
                           "tflops": round(shared_flops / (statistics.mean(shared_t) * 1e-3) / 1e12, 3),
                           "bf16_frac": round(shared_flops / (statistics.mean(shared_t) * 1e-3) / 1e12
                                              / pk["bf16_tflops"], 4)} if shared_t else None),
        "clocks": clk, "gpu_launches": int(st.launches_per_step * args.steps),
        "e2e": e2e, "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_stack(args, rank, world):
    """A layer stack (the ten-layer MXFP8 graph): every layer's forward, then
    the backwards in reverse, replayed as one CUDA graph; one JSON line."""
    import torch
    from mixture_experts_routed_route_gb300 import abi, synth

    w = synth.WORKLOADS[args.workload]
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk = peaks()
    st = StackStep(w, dev, slot_bytes=int(args.slot_gb * 1e9), tied=args.tied)
    st.enqueue()
    torch.cuda.synchronize(dev)
    bits = st.layer.error_bits()
    if bits:
        raise RuntimeError(f"device error bits {bits:#x} in warm-up")
    rows = st.rows_used()
    torch.cuda.empty_cache()
    st.capture()
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        st.graph.replay()
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        st.graph.replay()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / args.steps
    if world > 1:
        tt = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        ms = float(tt.item())
    if st.layer.error_bits():
        raise RuntimeError("device error bits set in the timed replays")

    # stage events keep the last call's records: the last layer's forward
    # and the first layer's backward (the last in reverse order, accumulating
    # into the FP32 weight gradients)
    fwd_t = {n: [] for n in abi.FWD_STAGE_NAMES}
    bwd_t = {n: [] for n in abi.BWD_STAGE_NAMES}
    for _ in range(3):
        st.stage_graph.replay()
        torch.cuda.synchronize(dev)
        for n, v in zip(abi.FWD_STAGE_NAMES, abi.moe_ctx_stage_times(st.layer.ctx, 0)):
            fwd_t[n].append(v)
        for n, v in zip(abi.BWD_STAGE_NAMES, abi.moe_ctx_stage_times(st.layer.ctx, 1)):
            bwd_t[n].append(v)
    stage_ms = {k: statistics.mean(v) for k, v in list(fwd_t.items()) + list(bwd_t.items())}

    def used(l):
        ids = np.asarray(st.ids_np[l])
        return int(np.unique(ids[(ids >= 0) & (ids < w.E)]).size)

    fb, _ = stage_bytes(w, rows[-1][0], rows[-1][1], w.precision, True, experts_used=used(len(rows) - 1))
    _, bb = stage_bytes(w, rows[0][0], rows[0][1], w.precision, True, experts_used=used(0),
                        dw_bytes=8 if st.tied else 2)
    sbytes = {**fb, **bb}
    dom = max(stage_ms, key=lambda k: stage_ms[k])
    achieved = sbytes[dom] / (stage_ms[dom] * 1e-3) / 1e9
    roof = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": None,
            "algorithmic_bytes": int(sbytes[dom]), "avg_launch_ms": round(stage_ms[dom], 4),
            "peak_source": pk["source"]}
    stages = {k: {"ms": round(v, 4), "GB/s": round(sbytes[k] / (v * 1e-3) / 1e9, 1) if v > 0 else None}
              for k, v in stage_ms.items()}
    routes = sum(r for _, r in rows)
    flops = 6.0 * routes * w.D * w.F * 3.0
    tflops = flops / (ms * 1e-3) / 1e12 * world
    peak_t = pk["bf16_tflops"] * 2.0
    replayed = [l for l, (_, input_only) in enumerate(st.states) if input_only]
    line = {
        "metric": METRIC, "value": round(tflops, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.precision, "data": "synthetic",
        "tokens_per_s": round(w.T * w.layers * world / (ms * 1e-3), 1),
        "tensor_frac": round(tflops / world / peak_t, 4), "tensor_peak_tflops": round(peak_t, 1),
        "config": {"workload": w.name, "layers": w.layers, "T": w.T, "D": w.D, "F": w.F, "E": w.E, "K": w.K,
                   "routing": "Zipf, exponent per layer in [0.8, 1.5]", "active_routes": routes,
                   "padded_rows": [r for r, _ in rows], "train": True,
                   "weights": ("one MXFP8 weight set shared by the layers (tied); dW13/dW2 FP32, accumulated "
                               "over the layers" if st.tied else
                               "an independent MXFP8 weight set per layer (input-gradient GEMMs read the forward "
                               "codes MN-major); each layer's dW13/dW2 BF16, written into one reused pair of "
                               "buffers"),
                   "saved_state": ("full, one buffer per layer" if st.slot is None else
                                   f"one {args.slot_gb:g} GB activation slot; layers {replayed} keep only their "
                                   f"input and replay (their replay FLOPs not counted as useful)"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2", "graph": "the whole stack in one CUDA graph, replayed"},
        "roofline": roof, "stages": stages,
        "stage_note": "stage times of the last layer's forward and the first layer's backward",
        "clocks": clk, "gpu_launches": int(st.launches_per_step * args.steps),
        "e2e": None, "cpu_baseline": None,
    }
    if st.slot is not None:
        for saved, _ in reversed(st.states):
            st.slot.pop(saved)
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------ reference arm (CPU)

def run_reference(args, rank, world):
    """The fp64 oracle timed on the host cores, on bounded samples of the
    same workload (each step = the oracle on the routes of a few experts)."""
    if rank != 0:
        return
    import torch
    from mixture_experts_routed_route_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    ids, scores = synth.make_routing(w)
    x = synth.make_tokens(w, "cpu")
    dy = synth.make_grad_out(w, "cpu")
    experts = pick_sample_experts(w, ids, args.cpu_sample_experts)
    w13s, w2s = synth.make_weights(w, "cpu", experts=experts)
    # at most 3 warm-up and 5 timed samples (a few seconds each), so the arm
    # ends within about a minute whatever --steps / --warmup ask; the line
    # reports the counts it ran
    warm = max(0, min(args.warmup, 3))
    for _ in range(warm):
        cpu_sample(w, ids, scores, x, dy, w13s, w2s, experts)
    times, fl = [], 0.0
    steps = max(1, min(args.steps, 5))
    for _ in range(steps):
        dt, fl, sroutes = cpu_sample(w, ids, scores, x, dy, w13s, w2s, experts)
        times.append(dt)
    dt = statistics.median(times)
    val = fl / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": round(dt * 1e3, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "D": w.D, "F": w.F, "E": w.E, "K": w.K, "train": w.train},
        "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "cores": blas_threads(),
                         "host_cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"fp64 numpy oracle, routes of {len(experts)} of {w.E} experts per step "
                                   f"({sroutes} routes, all {w.T} tokens)"},
        "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group(backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            from mixture_experts_routed_route_gb300 import synth
            (run_stack if synth.WORKLOADS[args.workload].layers > 1 else run_ours)(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
