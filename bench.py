#!/usr/bin/env python3
"""Throughput of the activation-sparse FFN decode step on GB300.

One step = one decode token through every layer of the workload's stack:
per layer the predictor (hidden + scores/threshold/ballot), the gather of
active up/gate rows with the fused activation, the down projection with the
residual add, then one momentum (TAM) update for all layers (and, for the
adaptive-lambda workload, one balancer step). Inputs are seeded synthetic
layers and token sequences resident in HBM before timing starts; every step
touches more distinct weight bytes than L2 holds.

Output: one JSON line (rank 0). Multi-GPU runs are independent replicas
(launch with torchrun); value = all ranks' tokens / max elapsed.

  python bench.py [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "llama2_70b_reglu_d8192_f28672_bf16_8l"
METRIC = "sparse-FFN decode tokens/s at B=1; active-byte HBM GB/s as % of GB300 peak"
FALLBACK_HBM_GBS = 6800.0
KERNELS = ("pred_hidden", "pred_scores", "ffn", "ffn_reduce")
KERNELS_BATCH = ("hidden_gemm", "scores_gemm", "upgate_gemm", "down_gemm")
KERNELS_BATCH_CC = ("cc_hidden", "cc_scores", "cc_ffn", "cc_reduce")
BF16_PEAK_KEY = "bf16_tflops"


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--layers", type=int, default=0, help="override the number of layers (0 = the workload's)")
    p.add_argument("--batch", type=int, default=1, help="tokens per decode step (independent streams)")
    p.add_argument("--tokens", type=int, default=128, help="distinct tokens cycled through (one graph each)")
    p.add_argument("--no-graph", action="store_true", help="launch eagerly instead of replaying CUDA graphs")
    p.add_argument("--profile-steps", type=int, default=64)
    p.add_argument("--e2e-steps", type=int, default=300)
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--lookahead", type=int, default=0, metavar="SMS",
                   help="B = 1: predict layer l+1 from layer l's input on a second stream while layer l's FFN "
                        "runs; SMS = SMs given to the predictor (0 = off, the exact method)")
    p.add_argument("--l2-resident-mb", type=float, default=0.0, metavar="MB",
                   help="B = 1: L2 share (all layers) for the rows of hot neuron groups, which a second momentum "
                        "state sized to that share picks each token; 0 = off")
    p.add_argument("--zero-skip", action="store_true",
                   help="B = 1: read the downT rows of predicted-active neurons with h != 0 only (actual-activation "
                        "zero-skip); the byte counts then count the rows read")
    p.add_argument("--no-prefetch-next", action="store_true",
                   help="do not let each layer prefetch the next layer's predictor weights into L2")
    p.add_argument("--normalize", action="store_true",
                   help="harness stand-in for the rest of a transformer block: each layer is fed x_l / rms(x_l) "
                        "(torch ops between the layers, outside the library) and the residual stream is "
                        "x_{l+1} = x_l + y_l; needed to run a deep gated stack without overflow")
    p.add_argument("--e2e-eager-steps", type=int, default=100,
                   help="steps of the end-to-end run without CUDA graphs (per-layer C ABI calls)")
    p.add_argument("--cpu1-seconds", type=float, default=15.0,
                   help="seconds of the single-thread oracle baseline (0 = skip)")
    p.add_argument("--ref-budget-s", type=float, default=240.0,
                   help="reference arm: seconds its warm-up and timed steps may take; beyond it fewer steps are "
                        "timed and the line says so")
    p.add_argument("--batch-path", choices=("auto", "tensor", "cuda_cores"), default="auto",
                   help="B > 1: the tensor-core products, or the CUDA-core arm (2 <= B <= 4)")
    p.add_argument("--stack", action="store_true",
                   help="B = 1: run each token through the whole stack in one persistent kernel "
                        "(sffn_stack_decode) instead of four kernels per layer; the momentum step follows it")
    p.add_argument("--no-topic-shift", action="store_true",
                   help="workloads with a topic shift: keep one topic (by default the second half of the cycled "
                        "tokens runs with every layer's group ranks redrawn)")
    p.add_argument("--cpu-worker", default=None, help=argparse.SUPPRESS)
    args = p.parse_args()
    if args.profile_steps < 1:
        p.error("--profile-steps must be at least 1: the roofline line comes from the traced pass")
    return args


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def replica_job_rate(elapsed_ms: float, units_per_rank: float, world: int, device="cpu"):
    """Replicas only (no collective on the data path): every rank processes its
    own units; the job's elapsed time is the slowest rank's (max over ranks)
    and its rate counts the units of all ranks. Returns (elapsed_ms, rate)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    return elapsed_ms, world * units_per_rank / (elapsed_ms / 1e3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# DRAM counters of one kernel on one workload, taken by ncu on a named
# capture and stored beside its summary in profiles/ (one file per workload);
# valid only while the kernel's sources hash to the value recorded with them.
TRAFFIC_FILES = {"ffn": "profiles/k_ffn_dram_traffic_{workload}.json"}


def sources_sha256(paths) -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(kernel: str, units_per_launch: float, prefetch: bool, workload: str):
    """DRAM bytes (read + write) per launch of `kernel` at `units_per_launch`
    active neurons, scaled from the stored capture by units processed (the
    kernel's traffic grows with the active rows it streams), plus the
    next-layer W1 prefetch when the L2 hint is on; or None. Bytes per neuron
    depend on the row length and storage, so a capture only serves the
    workload it was taken on."""
    rel = TRAFFIC_FILES.get(kernel)
    if rel is None:
        return None
    rel = rel.format(workload=workload)
    if not os.path.exists(os.path.join(ROOT, rel)):
        return None
    with open(os.path.join(ROOT, rel)) as fh:
        d = json.load(fh)
    if d.get("bench_workload") != workload:
        return None   # captured on another layer shape or row format
    if sources_sha256(d["sources"]) != d["sources_sha256"]:
        return None   # the kernel changed since the counters were taken
    l0 = d["launches"][0]
    fixed = d.get("l2_prefetch_bytes_per_launch", 0) if prefetch else 0
    per_unit = (l0["dram_read"] + l0["dram_write"] - d.get("l2_prefetch_bytes_per_launch", 0)) / l0["active_neurons"]
    return per_unit * units_per_launch + fixed


def measured_tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)[BF16_PEAK_KEY]), "measured"
    except Exception:
        return 1900.0, "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) while the timed region runs."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "200"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 11:
                    rows.append(parts)
        os.unlink(self.path)
        busy = [r for r in rows if _num(r[5]) is not None and _num(r[5]) >= 50] or rows
        sm = [_num(r[2]) for r in busy if _num(r[2]) is not None]
        smax = [_num(r[3]) for r in rows if _num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i in range(4) if r[7 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(busy),
                "power_w_max": max((_num(r[4]) or 0) for r in busy) if busy else None}


def _num(s):
    try:
        return float(s)
    except Exception:
        return None


# ----------------------------------------------------------------------------- bytes

def batch_layer_cost(spec, ucount: int, B: int, with_b2: bool) -> dict:
    """Algorithmic bytes of one layer and batch step (predictor weights once,
    every union row once, x and y of every token) and the tensor-core work
    executed per product (128-row tiles, N padded to 16/32, two MMAs per
    product for the hi/lo parts of the activations)."""
    d, f, h, wb = spec.d, spec.f, spec.h, spec.wbytes
    nmat_up = 2 if spec.gated else 1
    npad = 16 if B <= 16 else 32
    tiles = lambda m: -(-m // 128) * 128
    k = {
        "hidden_gemm": h * d * wb,
        "scores_gemm": f * h * wb + (f * 4 if with_b2 else 0),
        "upgate_gemm": ucount * nmat_up * d * wb,
        "down_gemm": ucount * d * wb,
    }
    flops = {
        "hidden_gemm": 2 * 2 * tiles(h) * npad * d,
        "scores_gemm": 2 * 2 * tiles(f) * npad * h,
        "upgate_gemm": 2 * 2 * nmat_up * tiles(ucount) * npad * d,
        "down_gemm": 2 * 2 * d * npad * (-(-ucount // 64) * 64),
    }
    metric = h * d * wb + f * h * wb + (f * 4 if with_b2 else 0) + ucount * spec.n_mats * d * wb + 2 * B * d * 4
    # the CUDA-core arm (B <= 4): the same weight bytes, one kernel each for
    # the hidden layer, the scores, the union FFN (all its rows) and the reduction
    kcc = {"cc_hidden": h * d * wb + B * d * 4, "cc_scores": f * h * wb + (f * 4 if with_b2 else 0),
           "cc_ffn": ucount * spec.n_mats * d * wb + B * d * 4, "cc_reduce": 3 * B * d * 4}
    return {"kernels": k | kcc, "flops": flops, "metric": metric}


def layer_bytes(spec, count: int, with_b2: bool, kept: int | None = None) -> dict:
    """Algorithmic bytes of one layer-token, per kernel: the weight rows the
    method must read plus the small vectors each kernel must move. kept: with
    zero-skip, the downT rows read (neurons with h != 0); None reads all."""
    d, f, h, wb = spec.d, spec.f, spec.h, spec.wbytes
    # bytes of one FFN row (plus its scale for 8-bit and 4-bit rows)
    one = int(d * spec.fbytes) + (4 if spec.ffn_quant else 0)
    rows = count * spec.n_mats * one if kept is None else count * (spec.n_mats - 1) * one + kept * one
    k = {
        "pred_hidden": h * d * wb + d * 4 + h * 4,
        "pred_scores": f * h * wb + h * 4 + f // 8 + (f * 4 if with_b2 else 0),
        # active up/gate/down rows + x + mask words (the per-block partials stay in L2)
        "ffn": rows + d * 4 + f // 8,
        # x read, y and x + y written (partials read from L2 are not HBM traffic)
        "ffn_reduce": 3 * d * 4,
    }
    # the metric: predictor weights + the FFN rows read + x + y
    metric = h * d * wb + f * h * wb + (f * 4 if with_b2 else 0) + rows + 2 * d * 4
    return {"kernels": k, "metric": metric}


L2_BYTES = 126e6   # GB300 L2 (a little below the marketed 129 MB once reserved lines are counted)


def stack_bytes(spec, n_layers: int) -> tuple[float, float]:
    """(weights held by the stack, bytes a token is expected to read): per
    layer the predictor plus every FFN row, and the predictor plus the rows
    of p_mean * f active neurons."""
    d, f, h, wb = spec.d, spec.f, spec.h, spec.wbytes
    pred = h * d * wb + f * h * wb + (f * 4 if spec.bias_mode else 0)
    row = int(d * spec.fbytes) + (4 if spec.ffn_quant else 0)
    held = n_layers * (pred + f * spec.n_mats * row)
    read = n_layers * (pred + spec.p_mean * f * spec.n_mats * row)
    return held, read


def topic_shift_note(spec, args, distinct: int) -> str | None:
    """The workload's topic shift, placed inside the cycled token set: tokens
    [P/2, P) of every P-token cycle run with every layer's group ranks redrawn
    (a second W2 per layer), so the shift and the shift back are both timed."""
    if not spec.topic_shift_at or args.no_topic_shift or args.batch > 1 or args.lookahead or args.l2_resident_mb:
        return None
    return (f"group ranks of every layer redrawn (new W2) for tokens {distinct // 2}..{distinct - 1} of each "
            f"{distinct}-token cycle, and back at the cycle's start")


def bench_config(spec, batch: int, n_layers: int, distinct: int, normalize: bool, zero_skip: bool, world: int,
                 replicas_note: str | None, topic: str | None = None) -> dict:
    """The workload part of the line's config: identical for both arms."""
    held, read = stack_bytes(spec, n_layers)
    if read > L2_BYTES:
        l2 = (f"inputs larger than L2: the stack holds {held / 1e9:.2f} GB of weights and a token reads about "
              f"{read / 1e6:.0f} MB of distinct weights (predictors and active rows of every layer)")
    else:
        l2 = (f"L2-resident correctness workload: a token reads about {read / 1e6:.1f} MB of weights, less than "
              f"L2 holds")
    cfg = {
        "workload": spec.name, "d": spec.d, "f": spec.f, "h": spec.h, "layers": n_layers, "batch": batch,
        "group_size": spec.group_size, "act": spec.act, "weights": spec.wdtype,
        "ffn_rows": "q4" if spec.ffn_q4 else "q8" if spec.ffn_q8 else spec.wdtype, "thres": spec.thres,
        "tam": {"lambda": spec.tam_lambda, "eps": spec.tam_eps, "capacity": spec.capacity,
                "adaptive_lambda": bool(spec.anb)},
        "distinct_tokens": distinct,
        "normalize": ("each layer is fed x_l / rms(x_l), a harness stand-in for the rest of the block (torch ops "
                      "outside the library); residual x_{l+1} = x_l + y_l") if normalize else None,
        "zero_skip": zero_skip,
        "topic_shift": topic,
        "l2": l2,
        "parallelism": "replicas" if world > 1 else "single",
    }
    if replicas_note:
        cfg["replicas"] = replicas_note
    return cfg


def stack_layers(spec, args) -> tuple[object, str | None]:
    """The stack the step runs: the workload's layers, or --layers, and a
    single-layer workload rotated over 4 replicas (so L2 never holds a step's
    rows). Returns (spec with that layer count, note or None)."""
    from activation_sparse_ffn_gb300 import workload as W
    if args.layers:
        return W.spec_replace(spec, layers=args.layers), None
    if spec.layers == 1:
        return (W.spec_replace(spec, layers=4),
                "single-layer workload rotated over 4 independent layer replicas")
    return spec, None


def rms_normalize(x):
    """x / rms(x) over the last axis (no learned scale, no epsilon): the
    harness stand-in for the normalisation a transformer block applies before
    its FFN. PyTorch's fused rms_norm: half the cost of the same expression
    spelled out in elementwise ops."""
    import torch.nn.functional as F
    return F.rms_norm(x, (x.shape[-1],), eps=0.0)


def percentiles_ms(durs: list[float]) -> dict:
    import numpy as np
    a = np.asarray(durs, dtype=np.float64)
    return {"p10": round(float(np.percentile(a, 10)), 5), "p50": round(float(np.percentile(a, 50)), 5),
            "p90": round(float(np.percentile(a, 90)), 5), "min": round(float(a.min()), 5),
            "max": round(float(a.max()), 5), "n": int(a.size)}


# ----------------------------------------------------------------------------- our arm

def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    import __graft_entry__
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        if rank == 0:
            __graft_entry__.build()
        dist.barrier()
    else:
        torch.cuda.set_device(local)
        __graft_entry__.build()
    from activation_sparse_ffn_gb300 import sffn
    from activation_sparse_ffn_gb300 import workload as W

    spec, replicas_note = stack_layers(W.WORKLOADS[args.workload], args)
    Bt = max(1, args.batch)
    normalize = bool(args.normalize)
    if normalize and (args.lookahead or args.l2_resident_mb):
        raise SystemExit("--normalize runs the exact method without look-ahead or L2 residency")
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    nL = spec.layers
    want_cpu = (not args.no_cpu_baseline) and rank == 0 and world == 1

    P = max(1, min(args.tokens, spec.tokens))
    topic = topic_shift_note(spec, args, P)
    # ---- layers (generated on the device, packed, originals freed); with a
    # topic shift, a second set whose W2 places the redrawn group ranks
    layers, layers_t1, host0 = [], [], None
    with torch.cuda.stream(stream):
        for l in range(nL):
            w = W.make_layer(spec, seed=args.seed, layer=l, device=dev)
            layers.append(sffn.Layer.from_weights(w, spec.group_size, spec.act, max_batch=Bt, stream=stream))
            if topic:
                w1 = dict(w)
                w1["W2"] = W.make_w2_topic(spec, args.seed, l, 1, w["W1"], w["perm"])
                layers_t1.append(sffn.Layer.from_weights(w1, spec.group_size, spec.act, max_batch=Bt,
                                                         stream=stream))
                del w1
            if l == 0 and want_cpu:
                host0 = {k: (W.stored_numpy(v) if torch.is_tensor(v) and v.dtype != torch.int32 else v)
                         for k, v in w.items()}
                host0["perm"] = w["perm"].cpu().numpy()
                host0["b2f"] = None if w["b2"] is None else w["b2"].double().cpu().numpy()
            del w
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    with_b2 = spec.bias_mode
    cc_arm = False
    if Bt > 1:
        for L in layers + layers_t1:
            L.set_batch_path(args.batch_path)
        cc_arm = sffn.sffn_layer_batch_arm(layers[0].handle, Bt) == "cuda_cores"
    # L2 hint: each layer's FFN kernel warms the next layer's predictor weights
    # (the last layer warms layer 0 for the next token)
    prefetch_next = Bt == 1 and not args.no_prefetch_next
    # actual-activation zero-skip: each layer reports the downT rows it read
    zero_skip = bool(args.zero_skip)
    if zero_skip and Bt != 1:
        raise SystemExit("--zero-skip applies to B = 1")
    rows_read = torch.zeros(nL, dtype=torch.int32, device=dev) if zero_skip else None
    if zero_skip:
        for l in range(nL):
            layers[l].set_zero_skip(True, rows_read[l:l + 1])
    if prefetch_next:
        for Ls in (layers, layers_t1):
            for l in range(len(Ls)):
                Ls[l].set_next(Ls[(l + 1) % nL])
    # one-layer-ahead prediction: the predictor and the FFN run on disjoint SMs
    lookahead = args.lookahead if Bt == 1 else 0
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    if lookahead:
        if not 0 < lookahead < n_sms:
            raise SystemExit(f"--lookahead must lie in 1..{n_sms - 1}")
        for L in layers:
            L.set_grid(n_sms - lookahead, lookahead)

    # ---- whole-stack kernel: one launch per token (per topic, one stack)
    use_stack = bool(args.stack)
    if use_stack and (Bt != 1 or normalize or lookahead or zero_skip or args.l2_resident_mb):
        raise SystemExit("--stack runs B = 1 without --normalize, --lookahead, --zero-skip or --l2-resident-mb")
    if use_stack:
        stacks = [sffn.Stack(layers)] + ([sffn.Stack(layers_t1)] if topic else [])
        stacks = stacks + stacks[:1] if len(stacks) == 1 else stacks
        smasks = [stacks[0].masks(device=dev) for _ in range(2)]
        sws = stacks[0].workspace(device=dev)
        sxs = torch.empty(nL, spec.d, device=dev)

    # ---- buffers
    sets = (layers, layers_t1 if topic else layers)

    def topic_of(t):
        return 1 if topic and (t % P) >= P // 2 else 0
    X = W.spec_tokens(spec, P, seed=args.seed, batch=Bt, device=dev).contiguous()  # [P,B,d]
    gw = (spec.n_groups + 31) // 32
    # group masks of all layers, double-buffered by token parity: the momentum
    # update of token t-1 runs while token t's layers write the other buffer
    gmask_buf = torch.zeros(2, nL, gw, dtype=torch.int32, device=dev)
    gmask_all = gmask_buf[0]
    masks = [layers[l].masks(Bt, device=dev) for l in range(nL)]
    side = torch.cuda.Stream(device=dev)
    ev_fork, ev_join = torch.cuda.Event(), torch.cuda.Event()

    def set_tam_mask(l, ptr):
        # the momentum update reads the token's group mask (B = 1) or the batch union's
        if Bt == 1:
            masks[l].c.gmask = ptr
        else:
            masks[l].c.ugmask = ptr
    ws = layers[0].workspace(Bt, device=dev)
    xa = torch.empty(Bt, spec.d, device=dev)
    xb = torch.empty(Bt, spec.d, device=dev)
    ybuf = torch.empty(Bt, spec.d, device=dev)
    tam = sffn.Tam(nL, spec.n_groups, spec.tam_lambda)
    K = spec.capacity
    outs = sffn.TamOutputs(nL, spec.n_groups, K, device=dev)
    # optional L2 residency of hot groups: a momentum state whose capacity is
    # the number of groups per layer that fit the requested L2 share
    l2_groups = 0
    if Bt == 1 and args.l2_resident_mb > 0:
        group_bytes = spec.group_size * spec.n_mats * (int(spec.d * spec.fbytes) + (4 if spec.ffn_quant else 0))
        l2_groups = max(1, min(spec.n_groups, int(args.l2_resident_mb * 1e6 / (nL * group_bytes))))
        tam_l2 = sffn.Tam(nL, spec.n_groups, spec.tam_lambda)
        outs_l2 = sffn.TamOutputs(nL, spec.n_groups, l2_groups, device=dev)
        for l in range(nL):
            layers[l].set_l2_resident(outs_l2.resident[l])
    stalls = torch.from_numpy(W.make_stall_bits(P, nL, seed=args.seed)).to(dev) if spec.anb else None
    # B = 1: hidden, scores, fused FFN, reduction. B > 1: split of x, hidden
    # product + finisher, scores product + finisher, mask views, up/gate
    # product + activation, down product + finisher.
    # CUDA-core arm (2 <= B <= 4): hidden, scores, views, union FFN, reduction.
    launches_per_step = nL * (4 if Bt == 1 else 5 if cc_arm else 10) + 1 + (1 if spec.anb else 0) + (1 if l2_groups else 0)
    if use_stack:
        launches_per_step = 1 + 1 + (1 if spec.anb else 0)
    if lookahead:
        launches_per_step += nL   # sffn_predict adds the mask-views kernel
        pstream = torch.cuda.Stream(device=dev)
        ws_pred = layers[0].workspace(1, device=dev)
        ev_x = [torch.cuda.Event() for _ in range(nL)]
        ev_p = [torch.cuda.Event() for _ in range(nL)]

    def layers_pass(x, saved=None, tp=0):
        """One token through every layer on `stream`; returns the last x_out.
        Exact method: sffn_decode_step per layer. Look-ahead: layer 0 is
        predicted from its own input, layer l + 1 from x_l on `pstream` while
        layer l's FFN runs (sffn_forward). `saved` collects each layer's input."""
        outb = (xa, xb)
        Ls = sets[tp]
        if normalize:
            resid = x
            for l in range(nL):
                xn = rms_normalize(resid)
                if saved is not None:
                    saved.append(xn.clone())
                sffn.sffn_decode_step(Ls[l].handle, xn, Bt, spec.thres, masks[l], ybuf, None, ws, stream)
                resid = resid + ybuf
            return resid
        if lookahead:
            sffn.sffn_predict(layers[0].handle, x, 1, spec.thres, masks[0], ws_pred, stream)
        for l in range(nL):
            xo = outb[l % 2]
            if saved is not None:
                saved.append(x.clone())
            if not lookahead:
                sffn.sffn_decode_step(Ls[l].handle, x, Bt, spec.thres, masks[l], ybuf, xo, ws, stream)
            else:
                if l + 1 < nL:
                    ev_x[l].record(stream)
                    pstream.wait_event(ev_x[l])
                    sffn.sffn_predict(layers[l + 1].handle, x, 1, spec.thres, masks[l + 1], ws_pred, pstream)
                    ev_p[l].record(pstream)
                sffn.sffn_forward(layers[l].handle, x, 1, masks[l], ybuf, xo, ws, stream)
                if l + 1 < nL:
                    stream.wait_event(ev_p[l])
            x = xo
        return x

    def stack_step(t, xin=None):
        """Token t through the whole stack in one launch, then its momentum
        step (and lambda step) on the same stream: the stack kernel holds
        every SM, so a concurrent branch would only delay it."""
        par = t % 2
        x = (X[t % P] if xin is None else xin)[0]
        sffn.sffn_stack_decode(stacks[topic_of(t)].handle, x, sxs, None, spec.thres, smasks[par], sws, stream)
        sffn.tam_update(tam.handle, 0, nL, smasks[par].gmask, gw, -1.0, spec.tam_eps, K, outs, stream)
        if spec.anb:
            sffn.tam_adapt(tam.handle, 0, nL, stalls[t % P], spec.anb_alpha, spec.anb_lo, spec.anb_hi, stream)
        return sxs[nL - 1:nL]

    def step(t, xin=None, saved=None):
        """Token t through every layer; in parallel, on a side stream, the
        momentum update (and lambda step) of token t-1, whose group masks sit in
        the other parity buffer. One momentum update per step."""
        if use_stack:
            return stack_step(t, xin)
        par = t % 2
        ev_fork.record(stream)
        side.wait_event(ev_fork)
        sffn.tam_update(tam.handle, 0, nL, gmask_buf[1 - par], gw, -1.0, spec.tam_eps, K, outs, side)
        if l2_groups:
            sffn.tam_update(tam_l2.handle, 0, nL, gmask_buf[1 - par], gw, -1.0, spec.tam_eps, l2_groups, outs_l2, side)
        if spec.anb:
            sffn.tam_adapt(tam.handle, 0, nL, stalls[(t - 1) % P], spec.anb_alpha, spec.anb_lo, spec.anb_hi, side)
        ev_join.record(side)
        x = X[t % P] if xin is None else xin
        for l in range(nL):
            set_tam_mask(l, gmask_buf[par, l].data_ptr())
        x = layers_pass(x, saved, topic_of(t))
        stream.wait_event(ev_join)
        return x

    # ---- census: active counts per (token, layer); deterministic given the token
    counts = np.zeros((P, nL), dtype=np.int64)       # active (B = 1) or union (B > 1) neurons
    tok_counts = np.zeros((P, nL), dtype=np.int64)   # sum over tokens of their own active neurons
    kept = np.zeros((P, nL), dtype=np.int64)         # zero-skip: downT rows read
    la_hits = la_exact = la_extra = 0   # look-ahead vs exact masks along the same trajectory
    ex_masks = layers[0].masks(1, device=dev) if lookahead else None

    def bits(t_):
        return int(np.unpackbits(t_.cpu().numpy().view(np.uint8)).sum())
    with torch.cuda.stream(stream):
        for t in range(P):
            saved = [] if lookahead else None
            xl = step(t, saved=saved)
            if lookahead:
                for l in range(1, nL):
                    sffn.sffn_predict(layers[l].handle, saved[l], 1, spec.thres, ex_masks, ws_pred, stream)
                    la, ex = masks[l].nmask[0], ex_masks.nmask[0]
                    la_hits += bits(la & ex)
                    la_exact += bits(ex)
                    la_extra += bits(la & ~ex)
            if not bool(torch.isfinite(xl).all()):
                raise SystemExit(f"{spec.name}: the residual stream overflowed within {nL} layers (a gated FFN grows "
                                 "with the square of its input and this stack has no block normalisation); "
                                 "use --layers to shorten it")
            if use_stack:
                counts[t] = smasks[t % 2].count.cpu().numpy()
                tok_counts[t] = counts[t]
            elif Bt == 1:
                counts[t] = torch.stack([m.count[0] for m in masks]).cpu().numpy()
                tok_counts[t] = counts[t]
                if zero_skip:
                    kept[t] = rows_read.cpu().numpy()
            else:
                counts[t] = torch.stack([m.ucount[0] for m in masks]).cpu().numpy()
                tok_counts[t] = torch.stack([m.count.sum() for m in masks]).cpu().numpy()
    for L in layers + layers_t1:
        L.check_error(stream)

    def cost(t_, l_):
        c = int(counts[t_, l_])
        if Bt > 1:
            return batch_layer_cost(spec, c, Bt, with_b2)
        return layer_bytes(spec, c, with_b2, int(kept[t_, l_]) if zero_skip else None)

    metric_bytes = np.array([[cost(t, l)["metric"] for l in range(nL)] for t in range(P)]).sum(axis=1)

    # ---- graphs: one per distinct token
    graphs = None
    if not args.no_graph:
        graphs = []
        with torch.cuda.stream(stream):
            for t in range(P):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    step(t)
                graphs.append(g)
        torch.cuda.synchronize()

    def run(t):
        if graphs is not None:
            graphs[t % P].replay()
        else:
            step(t)

    # ---- warm-up, then the timed region
    with torch.cuda.stream(stream):
        for t in range(args.warmup):
            run(t)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    # one event after every step (graph launches are serialised anyway, so the
    # events cost nothing measurable): the total and the per-step percentiles
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_start = args.warmup
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for i in range(args.steps):
            run(t_start + i)
            evs[i + 1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    step_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]
    elapsed_ms, value = replica_job_rate(evs[0].elapsed_time(evs[-1]), Bt * args.steps, world, dev)
    for L in layers + layers_t1:
        L.check_error(stream)
    if use_stack:
        for st_ in stacks:
            st_.check_error(stream)
    sffn.tam_check_error(tam.handle, stream)
    toks = [(t_start + i) % P for i in range(args.steps)]
    timed_bytes = float(sum(metric_bytes[t] for t in toks))
    sec = elapsed_ms / 1e3
    ms_per_step = elapsed_ms / args.steps
    step_gbs = timed_bytes / sec / 1e9

    # ---- traced pass: per-kernel durations (events around each kernel)
    R = min(args.profile_steps, P)
    KN = KERNELS if Bt == 1 else KERNELS_BATCH_CC if cc_arm else KERNELS_BATCH
    if use_stack:
        KN = ("decode_stack",)
    ev = {k: [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nL)]
              for _ in range(R)] for k in KN}
    tam_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(R)]
    with torch.cuda.stream(stream):
        for r in range(R):
            if use_stack:
                ev["decode_stack"][r][0][0].record(stream)
                sffn.sffn_stack_decode(stacks[0].handle, X[r % P][0], sxs, None, spec.thres, smasks[0], sws, stream)
                ev["decode_stack"][r][0][1].record(stream)
                tam_ev[r][0].record(stream)
                sffn.tam_update(tam.handle, 0, nL, smasks[0].gmask, gw, -1.0, spec.tam_eps, K, outs, stream)
                tam_ev[r][1].record(stream)
                continue
            for l in range(nL):
                sffn.sffn_layer_set_trace(layers[l].handle, [ev[k][r][l][0] for k in KN],
                                          [ev[k][r][l][1] for k in KN])
                set_tam_mask(l, gmask_all[l].data_ptr())
            layers_pass(X[r % P])
            tam_ev[r][0].record(stream)
            sffn.tam_update(tam.handle, 0, nL, gmask_all, gw, -1.0, spec.tam_eps, K, outs, stream)
            tam_ev[r][1].record(stream)
    torch.cuda.synchronize()
    for L in layers:
        sffn.sffn_layer_set_trace(L.handle)
    per_kernel = {}
    for k in KN:
        if k == "decode_stack":
            # one launch per token: its algorithmic bytes are the whole token's
            durs = [ev[k][r][0][0].elapsed_time(ev[k][r][0][1]) for r in range(R)]
            kb = [sum(cost(r % P, l)["metric"] for l in range(nL)) for r in range(R)]
            per_kernel[k] = {"us": 1e3 * sum(durs) / len(durs), "bytes": sum(kb) / len(kb),
                             "gbs": sum(kb) / (sum(durs) / 1e3) / 1e9}
            continue
        durs = [ev[k][r][l][0].elapsed_time(ev[k][r][l][1]) for r in range(R) for l in range(nL)]
        kb = [cost(r % P, l)["kernels"][k] for r in range(R) for l in range(nL)]
        per_kernel[k] = {"us": 1e3 * sum(durs) / len(durs), "bytes": sum(kb) / len(kb),
                         "gbs": sum(kb) / (sum(durs) / 1e3) / 1e9}
        if Bt > 1 and not cc_arm:
            kf = [cost(r % P, l)["flops"][k] for r in range(R) for l in range(nL)]
            per_kernel[k]["tflops"] = sum(kf) / (sum(durs) / 1e3) / 1e12
    tam_us = 1e3 * sum(a.elapsed_time(b) for a, b in tam_ev) / R
    dom = max(KN, key=lambda k: per_kernel[k]["us"])

    # ---- dense run of the same layer: every FFN row, no predictor. (1) our
    # kernels on an all-active caller mask (sffn_forward); (2) the library
    # reference: the same FFN as cuBLAS GEMVs on the packed weights (torch
    # matmul with 16-bit x, fp32 accumulation inside cuBLAS), for context.
    nd = 20
    for L in layers:   # the dense run reads every row
        if zero_skip:
            L.set_zero_skip(False)
    dense_masks = [layers[l].masks(Bt, device=dev) for l in range(nL)]
    for m in dense_masks:
        m.nmask.fill_(-1)
    with torch.cuda.stream(stream):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for i in range(3):
            sffn.sffn_forward(layers[0].handle, X[i % P], Bt, dense_masks[0], ybuf, None, ws, stream)
        e0.record(stream)
        for i in range(nd):
            sffn.sffn_forward(layers[i % nL].handle, X[i % P], Bt, dense_masks[i % nL], ybuf, None, ws, stream)
        e1.record(stream)
    torch.cuda.synchronize()
    dense_us = 1e3 * e0.elapsed_time(e1) / nd
    dense_lib_us = None
    if spec.wdtype != "f32" and not spec.ffn_quant:
        tdt = torch.bfloat16 if spec.wdtype == "bf16" else torch.float16
        views = []
        for L in layers:
            pv = L.packed()
            mk = lambda ptr: sffn.view_device(ptr, (spec.f, spec.d), tdt)
            views.append((mk(pv.up), mk(pv.gate) if spec.gated else None, mk(pv.downT)))

        def dense_lib(l, xv):
            up, gate, downT = views[l]
            xt = xv.to(tdt).t()                      # [d][B]
            u = torch.matmul(up, xt)                 # [f][B]
            if spec.act == "relu":
                hh = torch.relu(u)
            elif spec.act == "relu2":
                hh = torch.square(torch.relu(u))
            else:
                g = torch.matmul(gate, xt)
                hh = (torch.relu(g) if spec.act == "reglu" else torch.nn.functional.silu(g)) * u
            return torch.matmul(hh.t(), downT)       # [B][d]

        with torch.cuda.stream(stream):
            for i in range(3):
                dense_lib(0, X[i % P])
            e0.record(stream)
            for i in range(nd):
                dense_lib(i % nL, X[i % P])
            e1.record(stream)
        torch.cuda.synchronize()
        dense_lib_us = 1e3 * e0.elapsed_time(e1) / nd
        del views
    if zero_skip:
        for l in range(nL):
            layers[l].set_zero_skip(True, rows_read[l:l + 1])

    # ---- end to end through the public API with host buffers
    Xh = X.cpu().pin_memory()
    xin = torch.empty(Bt, spec.d, device=dev)
    yh = torch.empty(Bt, spec.d).pin_memory()
    g_e2e = None
    if graphs is not None:
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g_e2e, stream=stream):
                xfin = step(0, xin=xin)
    def e2e_run(n, graph):
        """n tokens: pinned host x -> device, the step, y -> pinned host, one
        synchronisation per token. Returns (seconds, per-token ms)."""
        per = []
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for i in range(n):
                ti = time.perf_counter()
                t = (t_start + i) % P
                xin.copy_(Xh[t], non_blocking=True)
                if graph is not None:
                    graph.replay()
                    out = xfin
                else:
                    out = step(t, xin=xin)
                yh.copy_(out, non_blocking=True)
                stream.synchronize()
                per.append(1e3 * (time.perf_counter() - ti))
        return time.perf_counter() - t0, per

    E = min(args.e2e_steps, args.steps)
    e2e_sec, e2e_per = e2e_run(E, g_e2e)
    e2e_value = world * Bt * E / e2e_sec
    # the same without graphs: every layer's C ABI call issued from Python per token
    Ee = min(args.e2e_eager_steps, args.steps)
    e2e_eager = None
    if Ee > 0:
        e2e_run(min(3, Ee), None)
        eager_sec, eager_per = e2e_run(Ee, None)
        e2e_eager = {"value": round(world * Bt * Ee / eager_sec, 2), "unit": "tokens/s", "steps": Ee,
                     "ms_per_step": percentiles_ms(eager_per),
                     "note": "no CUDA graph: each token issues every layer's sffn_decode_step (and the momentum "
                             "calls) through ctypes, host x in, host y out, one sync per token"}

    # ---- harness cost (the --normalize stand-in alone, same count per step)
    harness_us = 0.0
    if normalize:
        # captured like the step (one graph of a token's worth of harness ops)
        hg = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            hx = X[0].clone()
            with torch.cuda.graph(hg, stream=stream):
                hy = hx
                for i in range(nL):
                    hy = rms_normalize(hy) + ybuf
            hg.replay()
            e0.record(stream)
            for i in range(nd):
                hg.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        harness_us = 1e3 * e0.elapsed_time(e1) / (nd * nL)

    # ---- CPU baselines: the oracle on layer 0, as it stands (all host
    # cores through BLAS, and one thread in a separate process)
    cpu = cpu1 = None
    if want_cpu and host0 is not None:
        Xs = X[:, 0].double().cpu().numpy()
        cpu = cpu_baseline(spec, host0, Xs, args.cpu_seconds)
        cpu["sample"] += "; one token at a time (a batch costs its tokens' sum)" if Bt > 1 else ""
        if args.cpu1_seconds > 0:
            cpu1 = cpu_baseline_single_thread(spec, host0, Xs, args.cpu1_seconds)

    peak, peak_kind = measured_peaks()
    pk = per_kernel[dom]
    dom_traffic = None
    if Bt == 1 and not zero_skip:  # the stored counters are of the kernel without zero-skip
        t = measured_traffic(dom, float(counts.mean()), prefetch_next, spec.name)
        dom_traffic = round(t) if t is not None else None
    active_frac = float(tok_counts.mean() / Bt / spec.f)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": bench_config(spec, Bt, nL, P, normalize, zero_skip, world, replicas_note, topic),
        "run": {"kernels": "one whole-stack kernel per token (sffn_stack_decode)" if use_stack
                           else "four kernels per layer (sffn_decode_step)" if Bt == 1
                           else "batched CUDA-core arm (sffn_decode_step, 2 <= B <= 4)" if cc_arm
                           else "batched tensor-core path (sffn_decode_step, B > 1)",
                "graphs": graphs is not None, "l2_prefetch_next": prefetch_next and not use_stack,
                "l2_resident": ({"mb": args.l2_resident_mb, "groups_per_layer": l2_groups} if l2_groups else None),
                "timed_bytes_per_step_gb": round(timed_bytes / args.steps / 1e9, 4),
                "l2_between_steps": "not flushed: every step reads more distinct weights than L2 holds"
                                    if stack_bytes(spec, nL)[1] > L2_BYTES else "not flushed (L2-resident workload)"},
        "ms_per_step_pct": percentiles_ms(step_ms),
        "us_per_layer": round(1e3 * ms_per_step / nL, 3),
        "active_frac": round(active_frac, 5),
        "algorithmic_gbs": round(step_gbs, 1),
        "algorithmic_hbm_frac": round(step_gbs / peak, 4),
        "dense_us_per_layer": round(dense_us, 3),
        "dense_speedup": round(dense_us / (1e3 * ms_per_step / nL), 3),
        "dense_cublas_us_per_layer": round(dense_lib_us, 3) if dense_lib_us is not None else None,
        "dense_note": "all FFN rows, no predictor: our kernels on an all-active mask; cuBLAS GEMVs as reference",
        "kernels_us": {k: round(v["us"], 3) for k, v in per_kernel.items()} | {"tam_all_layers": round(tam_us, 3)},
        "kernels_gbs": {k: round(v["gbs"], 1) for k, v in per_kernel.items()},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(pk["gbs"], 1), "peak": peak,
                     "unit": "GB/s", "frac": round(pk["gbs"] / peak, 4), "traffic": dom_traffic,
                     "peak_kind": peak_kind},
        "e2e": {"value": round(e2e_value, 2), "unit": "tokens/s", "h2d_bytes_per_step": Bt * spec.d * 4,
                "d2h_bytes_per_step": Bt * spec.d * 4, "steps": E, "sync_per_step": True,
                "ms_per_step": percentiles_ms(e2e_per),
                "note": "one CUDA graph per token (all layers and the momentum step) through the library's C ABI"},
        "e2e_eager": e2e_eager,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    if cpu1 is not None:
        line["cpu_baseline_single_thread"] = cpu1
    if normalize:
        line["harness_us_per_layer"] = round(harness_us, 3)
    line["census"] = {"distinct_tokens": P, "active_count_token0_by_layer": [int(c) for c in counts[0]]}
    if zero_skip:
        line["zero_skip"] = {"down_rows_read_frac": round(float(kept.sum() / max(1, counts.sum())), 5),
                             "note": "bytes count the downT rows read (neurons with h != 0), all up/gate rows"}
    if lookahead:
        line["config"]["mode"] = "one-layer-ahead prediction (layer l+1 predicted from layer l's input)"
        line["run"]["sm_split"] = {"predictor": lookahead, "ffn": n_sms - lookahead}
        line["lookahead"] = {"recall": round(la_hits / max(1, la_exact), 4),
                             "extra_over_exact": round(la_extra / max(1, la_exact), 4),
                             "note": "layers 1.. of every census token; layer 0 is predicted from its own input"}
    if Bt > 1:
        line["union_frac"] = round(float(counts.mean() / spec.f), 5)
    if Bt > 1 and not cc_arm:
        tpk, _ = measured_tensor_peak()
        line["kernels_tflops"] = {k: round(v["tflops"], 2) for k, v in per_kernel.items()}
        line["tensor"] = {"kernel": dom, "achieved_tflops": round(pk["tflops"], 2), "peak": tpk,
                          "frac": round(pk["tflops"] / tpk, 5), "note": "executed MMA work incl. padding and hi/lo"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def oracle_ffn(O, spec, host, x, active, perm):
    """The oracle's sparse FFN on the stored rows (8-bit or 4-bit codes and scales, or wdtype rows)."""
    if spec.ffn_quant:
        fn = O.ffn_sparse_q4 if spec.ffn_q4 else O.ffn_sparse_q8
        return fn(x, host["up_q"], host["up_s"], host.get("gate_q"), host.get("gate_s"), host["down_q"],
                  host["down_s"], spec.act, active, perm)
    return O.ffn_sparse_stored(x, host["up"], host.get("gate"), host["down"], spec.wdtype, spec.act, active, perm)


def cpu_baseline(spec, host, Xs, seconds):
    """The oracle as it stands on layer 0 of the stack, token after token,
    for about ``seconds``; tokens/s of the whole stack = 1 / (layers x time
    per layer-token)."""
    import numpy as np
    from oracle import sffn_oracle as O

    W1 = O.widen(host["W1"], spec.wdtype)
    W2 = O.widen(host["W2"], spec.wdtype)
    perm = host["perm"]
    times = []
    t_end = time.perf_counter() + seconds
    t = 0
    while (time.perf_counter() < t_end or len(times) < 2) and len(times) < 10000:
        x = Xs[t % Xs.shape[0]]
        t0 = time.perf_counter()
        s = O.predictor_scores(W2, O.predictor_hidden(W1, x), host.get("b2f"))[perm]
        a = O.active_from_scores(s, spec.thres)
        O.mask_views(a, spec.group_size)
        oracle_ffn(O, spec, host, x, a, perm)
        times.append(time.perf_counter() - t0)
        t += 1
    per_layer = sum(times) / len(times)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(1.0 / (spec.layers * per_layer), 4), "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"layer 0 of {spec.layers}, {len(times)} tokens, {per_layer * 1e3:.1f} ms per layer-token "
                      f"(numpy fp64, BLAS threads = available cores), stack time = {spec.layers} x layer time"}


def cpu_baseline_single_thread(spec, host, Xs, seconds):
    """cpu_baseline with one thread: the layer's stored arrays go to a
    temporary directory and a fresh interpreter, started with every BLAS
    thread count at 1, times the oracle on them (a child process: the
    thread count of numpy's BLAS is fixed when it loads)."""
    import numpy as np
    with tempfile.TemporaryDirectory(prefix="sffn_cpu1_") as tmp:
        meta = {"workload": spec.name, "layers": spec.layers, "seconds": seconds, "arrays": []}
        for k, v in host.items():
            if isinstance(v, np.ndarray):
                np.save(os.path.join(tmp, k + ".npy"), v)
                meta["arrays"].append(k)
        np.save(os.path.join(tmp, "_X.npy"), Xs)
        with open(os.path.join(tmp, "meta.json"), "w") as fh:
            json.dump(meta, fh)
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
                   BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", tmp], capture_output=True,
                           text=True, env=env, timeout=600 + 4 * seconds)
        lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
        if r.returncode != 0 or not lines:
            return {"unavailable": f"single-thread worker failed (rc {r.returncode}): {r.stderr[-300:]}"}
        return json.loads(lines[-1])


def cpu_worker(tmp: str) -> None:
    """Child process of cpu_baseline_single_thread."""
    import numpy as np
    from activation_sparse_ffn_gb300 import workload as W
    with open(os.path.join(tmp, "meta.json")) as fh:
        meta = json.load(fh)
    host = {k: np.load(os.path.join(tmp, k + ".npy")) for k in meta["arrays"]}
    for k in ("b2f", "gate", "gate_q", "gate_s"):
        host.setdefault(k, None)
    spec = W.spec_replace(W.WORKLOADS[meta["workload"]], layers=meta["layers"])
    r = cpu_baseline(spec, host, np.load(os.path.join(tmp, "_X.npy")), meta["seconds"])
    r["cores"] = 1
    r["sample"] = r["sample"].replace("BLAS threads = available cores", "one thread: BLAS and OpenMP threads = 1")
    print(json.dumps(r), flush=True)


# ----------------------------------------------------------------------------- reference arm (the oracle)

def host_layer(W, O, spec, seed, layer, dev, topic=0):
    """Stored host copies of one layer, in the form the oracle reads (topic 1:
    the W2 of the redrawn group ranks)."""
    import torch
    w = W.make_layer(spec, seed=seed, layer=layer, device=dev)
    if topic:
        w["W2"] = W.make_w2_topic(spec, seed, layer, topic, w["W1"], w["perm"])
    host = {k: (W.stored_numpy(v) if torch.is_tensor(v) and v.dtype != torch.int32 else v) for k, v in w.items()}
    host["perm"] = w["perm"].cpu().numpy()
    host["b2f"] = None if w["b2"] is None else w["b2"].double().cpu().numpy()
    host["W1w"] = O.widen(host["W1"], spec.wdtype)
    host["W2w"] = O.widen(host["W2"], spec.wdtype)
    del w
    return host


def oracle_layer(O, spec, host, x):
    """One layer of the decode step in the oracle: predictor, threshold,
    mask views, sparse FFN. Returns y."""
    perm = host["perm"]
    s = O.predictor_scores(host["W2w"], O.predictor_hidden(host["W1w"], x), host["b2f"])[perm]
    a = O.active_from_scores(s, spec.thres)
    O.mask_views(a, spec.group_size)
    y, _ = oracle_ffn(O, spec, host, x, a, perm)
    return y


def run_reference(args, world, rank, local):
    """The reference arm: the oracle as it stands on the host cores, on the
    same workload, stack and token sequence as our arm. One step = one decode
    token (every token of the batch) through every layer of the stack, the
    residual x_{l+1} = x_l + y_l (or the --normalize stand-in), as our arm's
    step. Warm-up steps are all run; the timed steps are all run unless they
    would exceed --ref-budget-s, in which case the line times fewer and says so."""
    if rank != 0:
        return
    import numpy as np
    import torch

    from activation_sparse_ffn_gb300 import workload as W
    from oracle import sffn_oracle as O

    spec, replicas_note = stack_layers(W.WORKLOADS[args.workload], args)
    Bt = max(1, args.batch)
    nL = spec.layers
    P = max(1, min(args.tokens, spec.tokens))
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    topic = topic_shift_note(spec, args, P)
    hosts = [host_layer(W, O, spec, args.seed, l, dev) for l in range(nL)]
    hosts1 = [host_layer(W, O, spec, args.seed, l, dev, topic=1) for l in range(nL)] if topic else hosts
    X = W.spec_tokens(spec, P, seed=args.seed, batch=Bt).double().numpy()     # [P, B, d]

    def rms(v):
        return v / np.sqrt(np.mean(v * v))

    def one(t):
        hs = hosts1 if topic and (t % P) >= P // 2 else hosts
        for b in range(Bt):
            x = X[t % P, b]
            for l in range(nL):
                xin = rms(x) if args.normalize else x
                x = x + oracle_layer(O, spec, hs[l], xin)

    t_begin = time.perf_counter()
    warm = []
    for t in range(args.warmup):
        t0 = time.perf_counter()
        one(t)
        warm.append(time.perf_counter() - t0)
    est = (warm[-1] if warm else None)
    K = max(1, args.steps)
    if est is None:
        t0 = time.perf_counter()
        one(0)
        est = time.perf_counter() - t0
    left = args.ref_budget_s - (time.perf_counter() - t_begin)
    K_run = max(1, min(K, int(left / est)))
    per = []
    for i in range(K_run):
        t0 = time.perf_counter()
        one(args.warmup + i)
        per.append(time.perf_counter() - t0)
    sec = sum(per)
    value = Bt * K_run / sec
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = (f"each step = {Bt} token(s) through all {nL} layers of the stack (oracle: numpy fp64, BLAS threads "
              f"= available cores); {K_run} timed steps" + (f" of {K} requested (time budget "
                                                           f"{args.ref_budget_s:.0f} s)" if K_run < K else ""))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": world,
        "steps": K_run, "warmup": args.warmup, "ms_per_step": round(1e3 * sec / K_run, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(spec, Bt, nL, P, bool(args.normalize), bool(args.zero_skip), world, replicas_note,
                               topic),
        "ms_per_step_pct": percentiles_ms([1e3 * v for v in per]),
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    if K_run < K:
        line["steps_requested"] = K
    print(json.dumps(line), flush=True)


def launch_replicas(n: int) -> int:
    """`bench.py --gpus N` run directly (no WORLD_SIZE): start N replica
    processes of this command under torch.distributed.run on 127.0.0.1 and
    return its exit status."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(n),
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    args = parse_args()
    if args.cpu_worker:
        cpu_worker(args.cpu_worker)
        return
    world, rank, local = dist_env()
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        raise SystemExit(launch_replicas(args.gpus))
    if args.gpus != world:
        raise SystemExit(f"--gpus {args.gpus} but the launcher started {world} rank(s)")
    if args.impl == "reference":
        run_reference(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
