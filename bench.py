#!/usr/bin/env python
"""CSA forward throughput on one GB300 (tokens/s) with its roofline fraction.

Workload (default): the mixed 32k THD pack -- 32768 tokens in 64 lognormal
sequences (median 400, lengths 1..4000, including one of length 1 and one of
length 3) -- run through two attention layers back to back: a cmp_ratio-4
CSA layer (lightning indexer 64x128, top-512) and a cmp_ratio-128
compressor-only (HCA) layer. Both: 64 query heads, shared 512-wide bf16 KV,
window 128, per-head sinks. Inputs are synthetic (seeded N(0,1)).

One step = the whole path for both layers: compressed cu_seqlens, window
rows, indexer + top-k (CSA layer), sparse MLA with sinks. Inputs are resident
in HBM when the timed region starts; L2 is flushed between steps (a 256 MB
write, then a 256 MB read that evicts the write's dirty lines), outside the
per-step CUDA events. ``value`` is tokens / device time.
The timed steps record events only before each step and after each layer (the
kernels of a layer are launched back to back, each allowed to start while the
one before it finishes); per-kernel times come from separate steps after the
timed region, with an event after every launch.

Extra objects on the JSON line:
* roofline  -- the dominant kernel's algorithmic bytes (gathered KV rows,
               1 KB each) per launch / its CUDA-event time, against the
               measured HBM copy bandwidth;
* cpu_baseline -- the fp64 CPU oracle on a bounded token sample (rank 0, N=1);
* e2e       -- the same metric through the public Python API with pinned
               host buffers: H2D of every input and D2H of every output
               inside the timed region;
* clocks    -- nvidia-smi samples taken during the timed region.

``--impl reference`` times the oracle itself as the step (a bounded token
sample per step) on the host cores. ``--bwd`` adds a JSON line: the sparse
MLA backward of every layer, timed per launch from the forward's out and
lse, with its FLOPs against the bf16 tensor peak. ``--kl`` adds one more: the
indexer KL-loss gradient of the indexer layer, on its own top-k rows with
the attention backward's distribution as target, against the fp32 ALU peak.
``--cmp`` adds the THD compressor core (grouping, overlap, slot pooling) for
each layer's ratio, against the measured HBM bandwidth.
"""

from __future__ import annotations

import argparse
import hashlib
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

import numpy as np  # noqa: E402
import torch  # noqa: E402

from csa_inputs import packs  # noqa: E402

METRIC = "CSA fwd tokens/s (indexer+topk+sparse MLA) on 1 GB300; % of HBM/tensor roofline"
UNIT = "tokens/s"
FLUSH_BYTES = 256 << 20
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------------- setup
def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=60)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="mixed32k", choices=list(packs.CONFIGS))
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--bwd", action="store_true",
                   help="also time the sparse MLA backward of every layer and print its own "
                        "JSON line after the forward's (off by default: one line per run)")
    p.add_argument("--bwd-steps", type=int, default=5)
    p.add_argument("--cmp", action="store_true",
                   help="also time the THD compressor core for each layer's ratio "
                        "(one more JSON line)")
    p.add_argument("--cmp-only", action="store_true",
                   help="time only the THD compressor core (its own inputs; the forward "
                        "layers' tensors are not allocated) and print its line alone")
    p.add_argument("--kl", action="store_true",
                   help="also time the indexer KL-loss gradient of each indexer layer "
                        "(one more JSON line)")
    return p.parse_args()


def dist_setup(backend):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(step_ms, tokens_per_step, world, device):
    """Whole-job throughput: every rank ran the same number of steps on its own
    pack (replicas, weak scaling); time is the slowest rank's summed step time."""
    total_ms = max_over_ranks(float(sum(step_ms)), world, device)
    steps = len(step_ms)
    return {"value": world * tokens_per_step * steps / (total_ms / 1e3),
            "ms_per_step": total_ms / steps, "total_ms": total_ms}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


def layer_accounting(spec, layer):
    """Algorithmic units of one layer: keys per token, gathered KV bytes,
    MLA and indexer FLOPs (per launch of each kernel)."""
    W = spec.win_left + 1
    keys = 0
    nvis_sum = 0
    cmp_keys = 0
    for L in spec.lengths:
        pos = np.arange(L, dtype=np.int64)
        win = np.minimum(W, pos + 1)
        nvis = (pos + 1) // layer.cmp_ratio
        cmp = np.minimum(layer.topk, nvis) if layer.indexer else nvis
        keys += int(win.sum() + cmp.sum())
        nvis_sum += int(nvis.sum())
        cmp_keys += int(cmp.sum())
    D, H = spec.dim, spec.heads
    acc = {
        "keys": keys,
        "cmp_keys": cmp_keys,
        "kv_bytes": keys * D * 2,
        "mla_flops": 4 * D * H * keys,
        "idx_flops": (2 * layer.index_heads * layer.index_dim * nvis_sum) if layer.indexer else 0,
        "q_out_bytes": spec.total_tokens * H * D * 2 * 2,
    }
    return acc


# --------------------------------------------------------------------------- workload
class Layer:
    def __init__(self, spec, layer, tens, device):
        import sparse_attention_csa_gb300 as csa
        self.spec, self.layer = spec, layer
        T = spec.total_tokens
        cu = np.concatenate([[0], np.cumsum(spec.lengths)]).astype(np.int32)
        self.cu = torch.from_numpy(cu).to(device)
        cuc = csa.csa_compress_cu_seqlens(self.cu, layer.cmp_ratio)
        self.Tc = int(cuc[-1].item())  # the product's own compressed row count
        self.host = {k: v for k, v in tens.items()}
        self.host["cmp_kv"] = self.host["cmp_kv"][: self.Tc].contiguous()
        if layer.indexer:
            self.host["k_idx"] = self.host["k_idx"][: self.Tc].contiguous()
        self.dev = {k: v.to(device) for k, v in self.host.items()}
        self.host["cu"] = torch.from_numpy(cu)
        self.dev["cu"] = self.cu
        H, D, W = spec.heads, spec.dim, spec.win_left + 1
        self.out = torch.empty((T, H, D), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((T, H), dtype=torch.float32, device=device)
        self.cuc = torch.empty_like(self.cu)
        self.win = torch.empty((T, W), dtype=torch.int32, device=device)
        self.idx = (torch.empty((T, layer.topk), dtype=torch.int32, device=device)
                    if layer.indexer else None)
        self.ws = None
        if layer.indexer:
            need = csa.csa_indexer_topk_workspace_size(T, self.Tc, layer.index_heads,
                                                       layer.index_dim, layer.topk)
            self.ws = torch.empty(need, dtype=torch.uint8, device=device) if need else None
        self.acc = layer_accounting(spec, layer)
        self.side = torch.cuda.Stream(device=device)
        self.win_done = torch.cuda.Event()

    def launches(self, stream, events=None, names=None, per_kernel=True):
        """Run the layer; optionally record an event after each launch
        (per_kernel) or only after the layer's last one."""
        import sparse_attention_csa_gb300 as csa
        d, L, spec = self.dev, self.layer, self.spec
        n = 0

        def mark(name, last=False):
            if events is not None and (per_kernel or last):
                e = torch.cuda.Event(enable_timing=True)
                e.record(stream)
                events.append(e)
                names.append(name)

        csa.csa_compress_cu_seqlens(d["cu"], L.cmp_ratio, out=self.cuc, stream=stream)
        n += 1
        mark(f"compress_cu_seqlens/r{L.cmp_ratio}")
        if per_kernel:
            csa.csa_window_idx(d["cu"], spec.total_tokens, spec.win_left, 0, out=self.win,
                               stream=stream)
            mark(f"window_idx/r{L.cmp_ratio}")
        else:
            # the window rows depend on nothing else of the layer: on a side
            # stream, beside the indexer, joined before the layer ends
            fork = torch.cuda.Event()
            fork.record(stream)
            self.side.wait_event(fork)
            csa.csa_window_idx(d["cu"], spec.total_tokens, spec.win_left, 0, out=self.win,
                               stream=self.side)
            self.win_done.record(self.side)
        n += 1
        idx = None
        if L.indexer:
            idx, _ = csa.csa_indexer_topk(d["q_idx"], d["k_idx"], d["w"], d["cu"], self.cuc,
                                          L.cmp_ratio, L.topk, workspace=self.ws, out=self.idx,
                                          stream=stream)
            n += 1
            mark(f"indexer_topk/r{L.cmp_ratio}")
        csa.csa_sparse_mla_fwd(d["q"], d["ori_kv"], d["cmp_kv"], idx, d["cu"], d["cu"], self.cuc,
                               d["sinks"], spec.scale, L.cmp_ratio, spec.win_left, 0, True,
                               out=self.out, lse=self.lse, stream=stream)
        n += 1
        if not per_kernel:
            stream.wait_event(self.win_done)
        mark(f"sparse_mla_fwd/r{L.cmp_ratio}" if per_kernel else f"layer/r{L.cmp_ratio}", last=True)
        return n


class L2Flush:
    """Between timed steps: write a buffer larger than L2, then read another
    one, so that the next step starts with L2 holding none of its inputs and
    no dirty lines (the write's lines are written back while the read evicts
    them, not while the timed kernels run). Both run outside the step events."""

    def __init__(self, device):
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.max()


def build_layers(spec, device):
    return [Layer(spec, layer, tens, device)
            for layer, tens in zip(spec.layers, packs.draw_pack(spec))]


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")

        sm = [num(r[1]) for r in rows]
        mx = [num(r[2]) for r in rows]
        pw = [num(r[3]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        pmax = max(p for p in pw if not math.isnan(p)) if any(not math.isnan(p) for p in pw) else 0
        loaded = [s for s, p in zip(sm, pw) if not math.isnan(s) and p >= 0.3 * pmax] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx),
                "reasons": reasons, "samples": len(rows), "power_w_max": pmax}


# --------------------------------------------------------------------------- oracle arms
def oracle_inputs(layers):
    """fp64 copies of the tensors the oracle reads whole (rows of q, q_idx, w
    are converted per sampled token inside the calls)."""
    out = []
    for L in layers:
        h = L.host
        d = {"cu": h["cu"].numpy(), "ori_kv": h["ori_kv"].double().numpy(),
             "cmp_kv": h["cmp_kv"].double().numpy(), "sinks": h["sinks"].double().numpy()}
        if L.layer.indexer:
            d["k_idx"] = h["k_idx"].double().numpy()
        out.append(d)
    return out


def oracle_step(layers, prepared, tokens, stages=None):
    """The whole path for the listed tokens through the fp64 oracle; adds each
    stage's seconds to ``stages`` (A1 compressed cu_seqlens, A2 window rows,
    A3+A4 indexer and top-k, A6 sparse attention) when given."""
    import oracle
    tk = torch.from_numpy(tokens).long()

    def timed(name, fn):
        t0 = time.perf_counter()
        r = fn()
        if stages is not None:
            stages[name] = stages.get(name, 0.0) + time.perf_counter() - t0
        return r

    for L, d in zip(layers, prepared):
        spec, layer, h = L.spec, L.layer, L.host
        cuc = timed("A1", lambda: oracle.compress_cu_seqlens(d["cu"], layer.cmp_ratio))
        timed("A2", lambda: oracle.window_idx(d["cu"], spec.total_tokens, spec.win_left, tokens))
        idx = None
        if layer.indexer:
            idx = timed("A3+A4", lambda: oracle.indexer_topk(
                h["q_idx"][tk], d["k_idx"], h["w"][tk], spec.total_tokens, d["cu"], cuc,
                layer.cmp_ratio, layer.topk, tokens=tokens)[0])
        timed("A6", lambda: oracle.sparse_mla_fwd(
            h["q"][tk], d["ori_kv"], d["cmp_kv"], idx, d["cu"], cuc, spec.total_tokens,
            d["sinks"], spec.scale, layer.cmp_ratio, spec.win_left, tokens=tokens))


def token_sample(T, n, offset):
    stride = max(1, T // n)
    return ((np.arange(n, dtype=np.int64) * stride + offset) % T).astype(np.int32)


def cpu_model():
    """The host CPU's model name (lscpu), else what the platform reports."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(layers, seconds):
    """The fp64 oracle on evenly spaced tokens of the pack: all host threads for
    about ``seconds``, then one thread for a quarter of that; per-stage times
    from the all-thread run."""
    import oracle
    prepared = oracle_inputs(layers)
    T = layers[0].spec.total_tokens

    def run(budget, stages=None):
        done, batch, off = 0, 64, 0
        t0 = time.perf_counter()
        while True:
            oracle_step(layers, prepared, token_sample(T, batch, off), stages)
            done += batch
            off += 1
            el = time.perf_counter() - t0
            if el >= budget or done >= T:
                return done, el

    threads = oracle.num_threads()
    stages = {}
    done, el = run(seconds, stages)
    oracle.set_num_threads(1)
    try:
        done1, el1 = run(seconds / 4)
    finally:
        oracle.set_num_threads(threads)
    return {"value": done / el, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{done} tokens of the {layers[0].spec.name} pack (evenly spaced), "
                      f"all layers, fp64 C oracle, {el:.1f} s on {threads} threads",
            "nproc": os.cpu_count(), "cpu_model": cpu_model(),
            "single_thread": {"value": done1 / el1, "unit": UNIT, "tokens": done1,
                              "seconds": round(el1, 2)},
            "stage_ms_per_1k_tokens": {k: 1e6 * v / done for k, v in stages.items()}}


# --------------------------------------------------------------------------- arms
def traffic_record(kernel_name, config, layer):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source, for the same workload and layer; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel_name)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("config") != config or rec.get("layer") != layer:
        return None
    src = os.path.join(ROOT, "sparse_attention_csa_gb300", "csrc", rec["source"])
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    return rec["dram_bytes_per_launch"] if sha == rec["source_sha"] else None


def run_ours(args, world, rank, local):
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    spec = packs.pack_spec(args.config)
    layers = build_layers(spec, device)
    stream = torch.cuda.current_stream()
    flush = L2Flush(device)
    T = spec.total_tokens

    import sparse_attention_csa_gb300 as csa

    def step(events=None, names=None, per_kernel=True):
        return sum(L.launches(stream, events, names, per_kernel) for L in layers)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    st, word = csa.csa_device_error()
    if st != 0:
        raise RuntimeError(f"device error after warm-up: {word:#x}")

    clocks = ClockSampler(torch.cuda.current_device())
    step_ms, kern_ms, names = [], {}, None
    launches = 0
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    wall0 = time.perf_counter()
    # Timed steps: events before the step and after each layer only, so that the
    # launches of a layer follow each other with nothing in between (each
    # kernel may then start while the one before it finishes).
    recs = []
    for _ in range(args.steps):
        flush()
        ev = [torch.cuda.Event(enable_timing=True)]
        ev[0].record(stream)
        nm = []
        launches += step(ev, nm, per_kernel=False)
        recs.append((ev, nm))
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(world)
    clk = clocks.stop()
    layer_ms = {}
    for ev, nm in recs:
        step_ms.append(ev[0].elapsed_time(ev[-1]))
        for i, n in enumerate(nm):
            layer_ms.setdefault(n, []).append(ev[i].elapsed_time(ev[i + 1]))
    st, word = csa.csa_device_error()
    if st != 0:
        raise RuntimeError(f"device error in the timed region: {word:#x}")
    # Per-kernel breakdown (dominant kernel, kernels_ms): separate steps with an
    # event after every launch, after the timed region.
    for _ in range(max(3, min(args.steps, 10))):
        flush()
        ev = [torch.cuda.Event(enable_timing=True)]
        ev[0].record(stream)
        nm = []
        step(ev, nm)
        torch.cuda.synchronize()
        for i, n in enumerate(nm):
            kern_ms.setdefault(n, []).append(ev[i].elapsed_time(ev[i + 1]))

    agg = aggregate(step_ms, T, world, device)
    value, ms_per_step = agg["value"], agg["ms_per_step"]

    # roofline of the dominant kernel
    peaks, peak_kind = load_peaks()
    avg = {n: statistics.mean(v) for n, v in kern_ms.items()}
    dom = max(avg, key=avg.get)
    r = int(dom.split("/r")[1])
    lay = next(L for L in layers if L.layer.cmp_ratio == r)
    t_s = avg[dom] / 1e3
    if dom.startswith("sparse_mla_fwd"):
        achieved = lay.acc["kv_bytes"] / t_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"]}
        tflops = lay.acc["mla_flops"] / t_s / 1e12
        extra = {"tensor_tflops": tflops,
                 "tensor_frac_of_measured": tflops / peaks["bf16_tflops_sustained"],
                 "q_out_gbs": lay.acc["q_out_bytes"] / t_s / 1e9}
    else:
        achieved = lay.acc["idx_flops"] / t_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops_sustained"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops_sustained"]}
        extra = {}
    roof["traffic"] = traffic_record(dom.split("/")[0], spec.name, dom.split("/")[1])
    roof.update({"kernel": dom, "kernel_ms": avg[dom], "peak_source": peak_kind, **extra})
    # path-level roofline as the method defines it: max(gathered bytes/BW, flops/peak)
    bytes_all = sum(L.acc["kv_bytes"] for L in layers)
    flops_all = sum(L.acc["mla_flops"] + L.acc["idx_flops"] for L in layers)
    t_roof = max(bytes_all / (peaks["hbm_gbs"] * 1e9), flops_all / (peaks["bf16_tflops"] * 1e12))
    roof["path_roofline_ms"] = t_roof * 1e3
    roof["path_frac"] = t_roof * 1e3 / ms_per_step
    per_layer = {}
    for L in layers:
        r = L.layer.cmp_ratio
        lt = statistics.mean(layer_ms[f"layer/r{r}"])
        tl = max(L.acc["kv_bytes"] / (peaks["hbm_gbs"] * 1e9),
                 (L.acc["mla_flops"] + L.acc["idx_flops"]) / (peaks["bf16_tflops"] * 1e12))
        per_layer[f"r{r}"] = {"ms": lt, "roofline_ms": tl * 1e3, "frac": tl * 1e3 / lt}
    roof["layers"] = per_layer

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{spec.name}: {T} tokens, {len(spec.lengths)} sequences, "
                               + " + ".join(
                                   (f"CSA r={l.cmp_ratio} top{l.topk} idx {l.index_heads}x"
                                    f"{l.index_dim}") if l.indexer else f"HCA r={l.cmp_ratio}"
                                   for l in spec.layers)
                               + f", H={spec.heads}, D={spec.dim}, window {spec.win_left + 1}",
                   "tokens_per_step": T, "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed between steps (256 MB write, then a 256 MB read that "
                         "evicts its dirty lines; outside the step events)",
                   "timing": "events at step and layer boundaries; per-kernel times from "
                             "separate steps with an event after every launch",
                   "indexer_values": "not requested: tokens whose visible blocks fit in top-k "
                                     "keep them all unscored",
                   "wall_ms_incl_flush": wall * 1e3 / args.steps},
        "roofline": roof,
        "kernels_ms": avg,
        "gpu_launches": launches,
    }
    if clk:
        result["clocks"] = clk

    if not args.no_e2e:
        result["e2e"] = run_e2e(args, layers, stream, flush, world, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(layers, args.cpu_seconds)
    if args.bwd and rank == 0:
        result["_bwd"] = run_bwd(args, layers, stream, flush, peaks, peak_kind)
    if args.kl and rank == 0:
        result["_kl"] = run_kl(args, layers, stream, flush, peaks, peak_kind)
    if args.cmp and rank == 0:
        result["_cmp"] = run_cmp(args, layers, stream, flush, peaks, peak_kind)
    return result


class CmpLayer:
    """A layer's compressed-row offsets alone, for the compressor-only run."""

    def __init__(self, spec, layer, device):
        import sparse_attention_csa_gb300 as csa
        self.spec, self.layer = spec, layer
        cu = np.concatenate([[0], np.cumsum(spec.lengths)]).astype(np.int32)
        self.cu = torch.from_numpy(cu).to(device)
        self.cuc = csa.csa_compress_cu_seqlens(self.cu, layer.cmp_ratio)
        self.Tc = int(self.cuc[-1].item())


def run_cmp_only(args):
    device = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(device)
    spec = packs.pack_spec(args.config)
    layers = [CmpLayer(spec, layer, device) for layer in spec.layers]
    flush = L2Flush(device)
    peaks, peak_kind = load_peaks()
    return run_cmp(args, layers, torch.cuda.current_stream(), flush, peaks, peak_kind)


def run_cmp(args, layers, stream, flush, peaks, peak_src):
    """The THD compressor core for each layer's ratio on this pack (head_dim
    512, overlap, position embedding), from seeded N(0,1) projections drawn
    on the device, timed per launch with CUDA events between L2 flushes.
    Algorithmic bytes: every half row the overlap transform uses, read once
    from both projections (512 fp32 each), the position embedding and the
    fp32 output."""
    import sparse_attention_csa_gb300 as csa
    spec = layers[0].spec
    T, hd = spec.total_tokens, 512
    dev = layers[0].cu.device
    gen = torch.Generator(device=dev).manual_seed(9)
    kv = torch.randn((T, 2 * hd), generator=gen, device=dev)
    score = torch.randn((T, 2 * hd), generator=gen, device=dev)
    per, nbytes = {}, 0
    for L in layers:
        r = L.layer.cmp_ratio
        ape = torch.randn((r, 2 * hd), generator=gen, device=dev)
        out = torch.empty((L.Tc, hd), dtype=torch.float32, device=dev)

        def call():
            return csa.csa_compress_thd(kv, score, ape, L.cu, L.cuc, L.Tc, r, hd, True, out=out,
                                        stream=stream)

        csa.csa_compress_cu_seqlens(L.cu, r, out=L.cuc, stream=stream)
        for _ in range(3):
            flush()
            call()
        ms = []
        for _ in range(max(args.bwd_steps, 5)):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        per[f"compress_thd/r{r}"] = statistics.median(ms)
        # every group reads the second halves of its own r rows and, unless it
        # is its sequence's first, the first halves of the previous group's
        # rows, in both projections; plus the position embedding and the output
        cuc = L.cuc.cpu().numpy()
        firsts = int(np.count_nonzero(cuc[1:] > cuc[:-1]))
        halves = L.Tc * r + (L.Tc - firsts) * r
        nbytes += halves * 2 * hd * 4 + r * 2 * hd * 4 + L.Tc * hd * 4
    st, word = csa.csa_device_error()
    if st != 0:
        raise RuntimeError(f"device error in the compressor: {word:#x}")
    total = sum(per.values())
    achieved = nbytes / (total * 1e-3) / 1e9
    return {
        "metric": "THD compressor core tokens/s (grouping, overlap, slot softmax pooling) on 1 GB300",
        "value": T * len(layers) / (total * 1e-3), "unit": UNIT, "n_gpus": 1,
        "steps": max(args.bwd_steps, 5), "warmup": 3, "ms_per_step": total,
        "higher_is_better": True, "dtype": "f32", "data": "synthetic", "part": "compressor",
        "config": {"workload": f"{spec.name}, one compressor per layer ratio, head_dim 512, "
                               "overlap, projections given",
                   "l2": "flushed between launches (256 MB write, then 256 MB read)"},
        "kernels_ms": per,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "peak_source": peak_src, "bytes": nbytes},
    }


def run_kl(args, layers, stream, flush, peaks, peak_src):
    """The indexer KL-loss gradient of each indexer layer, on that layer's own
    top-k rows with the attention backward's head-averaged distribution over
    them (cmp_softmax_l1_norm) as the target, timed per launch with CUDA
    events between L2 flushes. Algorithmic FLOPs per (token, listed row):
    2 Hi Di each for the score, d_q and d_k -> 6 Hi Di; the contractions run
    on the tensor cores (bf16 operands, fp32 accumulation), so the roofline is
    the bf16 tensor peak."""
    import sparse_attention_csa_gb300 as csa
    gen = torch.Generator().manual_seed(8)
    per, flops, entries = {}, 0, 0
    for L in layers:
        if not L.layer.indexer:
            continue
        spec, r = L.spec, L.layer.cmp_ratio
        T = spec.total_tokens
        dout = torch.randn(tuple(L.out.shape), generator=gen).to(torch.bfloat16).to(L.out.device)
        L.launches(stream)
        bwd = csa.csa_sparse_mla_bwd(L.dev["q"], dout, L.out, L.lse, L.dev["ori_kv"],
                                     L.dev["cmp_kv"], L.idx, L.dev["cu"], L.dev["cu"], L.cuc,
                                     L.dev["sinks"], spec.scale, r, spec.win_left, stream=stream)
        l1 = bwd["cmp_l1"]
        del bwd, dout

        def call():
            return csa.csa_indexer_kl_loss_grad(L.dev["q_idx"], L.dev["k_idx"], L.dev["w"], L.idx,
                                                l1, L.dev["cu"], L.cuc, r, 1.0 / T,
                                                stream=stream)

        for _ in range(2):
            flush()
            call()
        ms = []
        for _ in range(args.bwd_steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        per[f"indexer_kl_grad/r{r}"] = statistics.median(ms)
        hi, di = L.layer.index_heads, L.layer.index_dim
        flops += 6 * hi * di * L.acc["cmp_keys"]
        entries += L.acc["cmp_keys"]
    st, word = csa.csa_device_error()
    if st != 0:
        raise RuntimeError(f"device error in the KL gradient: {word:#x}")
    total = sum(per.values())
    spec = layers[0].spec
    achieved = flops / (total * 1e-3) / 1e12
    return {
        "metric": "indexer KL-loss gradient tokens/s (loss, d_q, d_k, d_w) on 1 GB300",
        "value": spec.total_tokens / (total * 1e-3), "unit": UNIT, "n_gpus": 1,
        "steps": args.bwd_steps, "warmup": 2, "ms_per_step": total, "higher_is_better": True,
        "dtype": "bf16 (tcgen05, fp32 accumulate; G as a bf16 hi + lo pair)", "data": "synthetic",
        "part": "indexer KL",
        "config": {"workload": f"{spec.name}, indexer layers, own top-k rows, attention "
                               "distribution as target", "list_entries": entries,
                   "l2": "flushed between launches (256 MB write, then 256 MB read)"},
        "kernels_ms": per,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                     "peak_source": peak_src, "flops": flops},
    }


def run_bwd(args, layers, stream, flush, peaks, peak_src):
    """The sparse MLA backward of each layer (from that layer's forward out and
    lse, seeded N(0,1) dout), timed per launch with CUDA events between L2
    flushes. Algorithmic FLOPs per (key, head): 2D each for the recomputed
    scores, dout . k, d_q and the row gradient's two terms -> 10 D."""
    import sparse_attention_csa_gb300 as csa
    gen = torch.Generator().manual_seed(7)
    per, flops = {}, 0
    for L in layers:
        spec, r = L.spec, L.layer.cmp_ratio
        dout = torch.randn(tuple(L.out.shape), generator=gen).to(torch.bfloat16).to(L.out.device)
        L.launches(stream)  # this layer's out, lse and top-k rows
        idx = L.idx if L.layer.indexer else None

        def call():
            return csa.csa_sparse_mla_bwd(L.dev["q"], dout, L.out, L.lse, L.dev["ori_kv"],
                                          L.dev["cmp_kv"], idx, L.dev["cu"], L.dev["cu"], L.cuc,
                                          L.dev["sinks"], spec.scale, r, spec.win_left,
                                          stream=stream)

        for _ in range(2):
            flush()
            call()
        ms = []
        for _ in range(args.bwd_steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        per[f"sparse_mla_bwd/r{r}"] = statistics.median(ms)
        flops += 10 * spec.dim * spec.heads * L.acc["keys"]
    st, word = csa.csa_device_error()
    if st != 0:
        raise RuntimeError(f"device error in the backward: {word:#x}")
    total = sum(per.values())
    spec = layers[0].spec
    achieved = flops / (total * 1e-3) / 1e12
    return {
        "metric": "sparse MLA backward tokens/s (d_q, d_kv, d_sinks, distributions) on 1 GB300",
        "value": spec.total_tokens / (total * 1e-3), "unit": UNIT, "n_gpus": 1,
        "steps": args.bwd_steps, "warmup": 2, "ms_per_step": total, "higher_is_better": True,
        "dtype": "bf16 (tcgen05, fp32 accumulate)", "data": "synthetic", "part": "backward",
        "config": {"workload": f"{spec.name}, every layer, forward out/lse as inputs",
                   "l2": "flushed between launches (256 MB write, then 256 MB read)"},
        "kernels_ms": per,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                     "peak_source": peak_src, "flops": flops},
    }


def run_e2e(args, layers, stream, flush, world, device):
    """Same metric through the public API, host buffers in the timed region."""
    pinned_in, pinned_out = [], []
    h2d = d2h = 0
    for L in layers:
        ins = {}
        for k, v in L.host.items():
            p = torch.empty_like(v).pin_memory()
            p.copy_(v)
            ins[k] = p
            h2d += p.numel() * p.element_size()
        pinned_in.append(ins)
        outs = {"out": torch.empty(L.out.shape, dtype=L.out.dtype).pin_memory(),
                "lse": torch.empty(L.lse.shape, dtype=L.lse.dtype).pin_memory()}
        d2h += sum(t.numel() * t.element_size() for t in outs.values())
        pinned_out.append(outs)

    # Three streams: inputs copied in on one, the layers on the compute stream,
    # outputs copied out on a third. Layer 2's inputs load while layer 1 runs,
    # each layer's outputs leave as soon as it is done, and copies in and out
    # overlap (the link is full duplex). A step starts and ends on the compute
    # stream; its events bracket every copy and kernel of the step.
    s_in, s_out = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)

    def step(start, end):
        n = 0
        s_in.wait_event(start)
        loaded = []
        for L, ins in zip(layers, pinned_in):
            with torch.cuda.stream(s_in):
                for k, p in ins.items():
                    L.dev[k].copy_(p, non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_in)
            loaded.append(e)
        for L, outs, e in zip(layers, pinned_out, loaded):
            stream.wait_event(e)
            n += L.launches(stream)
            done = torch.cuda.Event()
            done.record(stream)
            s_out.wait_event(done)
            with torch.cuda.stream(s_out):
                outs["out"].copy_(L.out, non_blocking=True)
                outs["lse"].copy_(L.lse, non_blocking=True)
        fin = torch.cuda.Event()
        fin.record(s_out)
        stream.wait_event(fin)
        end.record(stream)
        return n

    for _ in range(max(1, args.warmup)):
        a, b = torch.cuda.Event(), torch.cuda.Event()
        a.record(stream)
        step(a, b)
    torch.cuda.synchronize()
    times = []
    barrier(world)
    for _ in range(args.steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step(a, b)
        times.append((a, b))
    torch.cuda.synchronize()
    barrier(world)
    ms = sum(a.elapsed_time(b) for a, b in times)
    ms = max_over_ranks(ms, world, device)
    T = layers[0].spec.total_tokens
    return {"value": world * T * args.steps / (ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms / args.steps}


def run_reference(args, world, rank):
    """The oracle as the step, on the host cores; rank 0 only."""
    if rank != 0:
        return None
    import oracle
    spec = packs.pack_spec(args.config)
    layers = [type("L", (), {})() for _ in spec.layers]
    tens_all = packs.draw_pack(spec)
    cu = np.concatenate([[0], np.cumsum(spec.lengths)]).astype(np.int32)
    for L, layer, tens in zip(layers, spec.layers, tens_all):
        L.spec, L.layer = spec, layer
        tc = int(oracle.compress_cu_seqlens(cu, layer.cmp_ratio)[-1])
        h = dict(tens)
        h["cmp_kv"] = h["cmp_kv"][:tc].contiguous()
        if layer.indexer:
            h["k_idx"] = h["k_idx"][:tc].contiguous()
        h["cu"] = torch.from_numpy(cu)
        L.host = h
    prepared = oracle_inputs(layers)
    T = spec.total_tokens
    per_step = 512
    for i in range(args.warmup):
        oracle_step(layers, prepared, token_sample(T, per_step, 7 + i))
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(layers, prepared, token_sample(T, per_step, 101 + i))
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = per_step * args.steps / total
    sample = (f"{per_step} evenly spaced tokens of the {spec.name} pack per step, all layers, "
              f"fp64 C oracle")
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": spec.name, "tokens_per_step": per_step},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    if args.impl == "reference":
        # no process group: rank 0 alone runs the oracle, the other ranks exit
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        res = run_reference(args, world, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if args.cmp_only:
        print(json.dumps(run_cmp_only(args)), flush=True)
        return
    world, rank, local = dist_setup("nccl")
    res = run_ours(args, world, rank, local)
    bwd = res.pop("_bwd", None)
    kl = res.pop("_kl", None)
    cmp_line = res.pop("_cmp", None)
    if rank == 0:
        print(json.dumps(res), flush=True)
        for extra in (bwd, kl, cmp_line):
            if extra is not None:
                print(json.dumps(extra), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
