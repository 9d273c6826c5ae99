"""Benchmark of the HYPIC state-algebra hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  plan + segment build of one Qwen3.5-35B-A3B-shaped GDN layer
    (64 segments x 1024 tokens, 16 key / 32 value heads, d = 128, bf16,
     one batched launch, fp32 pairs into the cache pool), then
  compose of a warm RAG prompt
    (30 GDN layers x 32 value heads, d = 128, 100 cached segments with
     lognormal lengths, 8 seam tokens per segment, ~12.6 GB of fp32 pairs
     resident in HBM).
`value` is the build throughput in tokens/s (tokens of the layer per second of
build time); the compose's GB/s against the HBM roofline is reported beside
it.  Inputs are seeded and synthetic and larger than L2, so no flush is
needed between timed steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs the same per-GPU work (weak scaling); times
are the max over ranks.  `--impl reference` times the fp64 CPU oracle on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "(T_C,S) build tokens/s (tensor %peak); compose GB/s vs HBM peak, GDN H=32 d=128"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ---------------------------------------------------------------- algorithmic work
C = 64


def build_flops(lengths, h_v, d_k=128, d_v=128, g=2, chunk=C):
    """Algorithmic FLOPs of the chunkwise build: per chunk of c tokens and
    value head, Gram 2c^2 d_k / g + W,U solves 2c^2 (d_k + d_v) + K^T Y
    2c d_k (d_k + d_v) + W X (skipped on the first chunk) 2c d_k (d_k + d_v).
    The chunk length is the kernel's (64 for the scalar gates, 32 for the
    per-channel gate)."""
    tot = 0.0
    for L in lengths:
        n_full, tail = divmod(int(L), chunk)
        chunks = [chunk] * n_full + ([tail] if tail else [])
        for j, c in enumerate(chunks):
            f = 2 * c * c * d_k / g + 2 * c * c * (d_k + d_v) + 2 * c * d_k * (d_k + d_v)
            if j > 0:
                f += 2 * c * d_k * (d_k + d_v)
            tot += f
    return tot * h_v


def build_bytes(n_tokens, n_pairs, h_k, h_v, d_k=128, d_v=128, in_bytes=2):
    """Inputs read once per key-head group (k) / value head (v, g, beta),
    fp32 pairs written once."""
    return (n_tokens * h_k * d_k * in_bytes + n_tokens * h_v * d_v * in_bytes + n_tokens * h_v * 8
            + n_pairs * h_v * (d_k * d_k + d_k * d_v) * 4)


def compose_bytes(n_layers, n_seg, w, h_k, h_v, d_k=128, d_v=128, in_bytes=2, with_init=False, gate_floats=1):
    """gate_floats: fp32 gate values per (token, value head): 1 (scalar),
    d_k (per-channel) or 0 (DeltaNet)."""
    pairs = n_layers * n_seg * h_v * (d_k * d_k + d_k * d_v) * 4
    seam_in = n_layers * n_seg * w * (2 * h_k * d_k * in_bytes + h_v * d_v * in_bytes + (1 + gate_floats) * h_v * 4)
    seam_out = n_layers * n_seg * w * h_v * d_v * 4
    states = n_layers * h_v * d_k * d_v * 4 * (2 if with_init else 1)
    slots = n_layers * n_seg * 4
    return pairs + seam_in + seam_out + states + slots


def compose_flops(n_layers, n_seg, w, h_v, d_k=128, d_v=128):
    ts = 2.0 * d_k * d_k * d_v
    seam = w * (6.0 * d_k * d_v)
    return n_layers * n_seg * h_v * (ts + seam)


# ---------------------------------------------------------------- ncu traffic
E2E_CHUNKS = 4  # groups of the end-to-end calls (copies overlap the kernels; 4 to 16 measured within 2%)

KERNEL_SOURCES = {
    "build": ("build_tc.cu", "tc.cuh", "common.cuh", "internal.h"),
    "compose": ("compose_tc.cu", "tc.cuh", "common.cuh", "internal.h"),
    "compose_channel": ("compose_tc.cu", "tc.cuh", "common.cuh", "internal.h"),
    "channel": ("build_channel.cu", "tc.cuh", "common.cuh", "internal.h"),
    "merge": ("merge.cu", "tc.cuh", "common.cuh", "internal.h"),
    "rerotate": ("rerotate.cu", "tc.cuh", "common.cuh", "internal.h"),
    "forward": ("forward_tc.cu", "tc.cuh", "common.cuh", "internal.h"),
    "fast": ("build_fast.cu", "tc.cuh", "common.cuh", "internal.h"),
}
PROFILE_FILES = {"build": "segment_build_tc__gdn_16x1024.md", "compose": "compose_seam_mma__gdn_4x32x100.md",
                 "compose_channel": "compose_seam_mma__channel_4x32x100.md",
                 "channel": "segment_build_channel__16x1024.md", "merge": "pair_merge_tc__4x32x50.md",
                 "rerotate": "pair_rerotate__4x100x32.md", "forward": "forward_tc__gdn_16x1024.md",
                 "fast": "build_fast__retnet_8x16x8192.md"}


def source_hash(kind):
    """sha256 over the kernel's source files: a captured traffic figure is
    only reported while the kernel is unchanged."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "hybrid_linear_attention_chunkwise_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def captured_traffic(kind, units_full):
    """DRAM bytes per full launch from the committed ncu summary of a small
    case (scaled by the units processed), or None when the summary is missing
    or was taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", PROFILE_FILES[kind])
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and line.split(":", 1)[0].strip() in ("source_sha256", "dram_bytes_per_unit"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip().split()[0]
    if vals.get("source_sha256") != source_hash(kind) or "dram_bytes_per_unit" not in vals:
        return None
    return float(vals["dram_bytes_per_unit"]) * units_full


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle samples every 50 ms; `region()` marks the
    timed region, and the summary uses the samples taken inside it (or the
    nearest ones when the region is shorter than the sampling period)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []  # (time, line)
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            deadline = time.time() + 3.0
            while not self.lines and time.time() < deadline:
                time.sleep(0.01)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def start(self):
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()
        time.sleep(0.06)  # one more sample after the region

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        lines = self.lines
        if self.t0 is not None and self.t1 is not None and lines:
            inside = [x for x in lines if self.t0 <= x[0] <= self.t1]
            if not inside:
                mid = 0.5 * (self.t0 + self.t1)
                inside = sorted(lines, key=lambda x: abs(x[0] - mid))[:2]
            lines = inside
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, ln in lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workloads
def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def setup_build(dev, seed=0):
    import synth_inputs as si
    W = si.workload(3, seed=seed, device=dev)
    return W


def setup_compose(dev, hy, seed=0, n_layers=30, variant="gdn"):
    """Cache pool of the warm RAG prompt: pairs of 30 GDN layers (or another
    dense-transition variant) built on the GPU from seeded token inputs
    (untimed set-up), plus the seam tokens."""
    import torch
    import synth_inputs as si
    W = si.workload(4, seed=seed, device=dev, n_layers=1, variant=variant)
    n_seg = W.n_seg
    n_slots = n_layers * n_seg
    T_pool = torch.empty((n_slots, W.h_v, W.d_k, W.d_k), device=dev)
    S_pool = torch.empty((n_slots, W.h_v, W.d_k, W.d_v), device=dev)
    seams = []
    for l in range(n_layers):
        lay = W.layers[0] if l == 0 else si.make_layer(seed=seed, cfg=4, layer=l, n_tokens=W.n_tokens, h_k=W.h_k,
                                                        h_v=W.h_v, d_k=W.d_k, d_v=W.d_v, variant=variant,
                                                        dtype=torch.bfloat16, device=dev)
        slots = np.arange(n_seg, dtype=np.int32) + l * n_seg
        hy.segment_build(lay.k, lay.v, lay.g, lay.beta, W.seg_offsets, variant=variant, seam_w=W.seam_w,
                         T_pool=T_pool, S_pool=S_pool, slot_of_seg=slots)
        W.layers = [lay]
        seams.append(si.seam_gather(W, lay))
        del lay
    torch.cuda.synchronize()
    sa = {k: (torch.stack([s[k] for s in seams]).contiguous() if seams[0][k] is not None else None)
          for k in ("k", "v", "q", "g", "beta")}
    slot = torch.arange(n_slots, dtype=torch.int32, device=dev).reshape(n_layers, n_seg)
    S_out = torch.empty((n_layers, W.h_v, W.d_k, W.d_v), device=dev)
    seam_out = torch.empty((n_layers, n_seg, W.seam_w, W.h_v, W.d_v), device=dev)
    return dict(W=W, n_layers=n_layers, T_pool=T_pool, S_pool=S_pool, sa=sa, slot=slot, S_out=S_out,
                seam_out=seam_out)


# ---------------------------------------------------------------- CPU oracle leg
def _time_ms(fn, reps=5, warm=2):
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def merge_row(dev, hy, peaks, comp):
    """The pair merge on the warm-prompt pool: every layer's segments 2i+1
    and 2i merged (1500 merges x 32 heads), into a fresh output pool.  Bytes
    per (merge, head): four 64 KiB inputs read, two written."""
    import torch
    W = comp["W"]
    n_l, n_seg = comp["n_layers"], W.n_seg
    pairs = [(l * n_seg + 2 * i + 1, l * n_seg + 2 * i) for l in range(n_l) for i in range(n_seg // 2)]
    later = torch.tensor([a for a, _ in pairs], dtype=torch.int32, device=dev)
    earlier = torch.tensor([b for _, b in pairs], dtype=torch.int32, device=dev)
    out = torch.arange(len(pairs), dtype=torch.int32, device=dev)
    To = torch.empty((len(pairs), W.h_v, W.d_k, W.d_k), device=dev)
    So = torch.empty((len(pairs), W.h_v, W.d_k, W.d_v), device=dev)
    ms = _time_ms(lambda: hy.pair_merge(later, earlier, out, comp["T_pool"], comp["S_pool"], To, So,
                                        variant="gdn"))
    units = len(pairs) * W.h_v
    nbytes = units * (4 + 2) * W.d_k * W.d_v * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    del To, So
    torch.cuda.empty_cache()
    return {"ms": ms, "merges_per_s": units / (ms * 1e-3), "algorithmic_bytes": nbytes,
            "hbm": {"achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s", "frac": gbs / peaks["hbm"]},
            "kernel": "tensor-core pair merge (split tf32)"}


def rerotate_row(dev, hy, peaks, comp):
    """State re-rotation of the whole warm-prompt pool in place (every layer's
    100 segments moved by a random shift, RoPE pairs (i, i + 64), all 128
    channels): each pool byte read once and written once, 4 x 64 KiB per
    (slot, head)."""
    import torch
    W = comp["W"]
    n = comp["n_layers"] * W.n_seg
    slots = torch.arange(n, dtype=torch.int32, device=dev)
    gen = torch.Generator(device="cpu").manual_seed(5)
    deltas = torch.randint(-100000, 100000, (n,), generator=gen, dtype=torch.int64).to(dev)
    ms = _time_ms(lambda: hy.pair_rerotate(slots, slots, deltas, comp["T_pool"], comp["S_pool"], comp["T_pool"],
                                           comp["S_pool"], variant="gdn", rot_dim=W.d_k, layout="half"))
    nbytes = n * W.h_v * 4 * W.d_k * W.d_v * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"ms": ms, "algorithmic_bytes": nbytes,
            "hbm": {"achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s", "frac": gbs / peaks["hbm"]},
            "kernel": "pair re-rotation (fp32, in place)"}


def compose_variant_rows(dev, hy, peaks, n_layers=8):
    """The compose of the other dense-transition variants on the warm-prompt
    shape (8 layers x 32 heads x 100 segments, w = 8): DeltaNet (tensor-core
    seam) and the per-channel gate (tensor-core seam with per-channel
    operand tiles); the kernel named is the one the path query reports."""
    import torch
    rows = {}
    for var, gate in (("deltanet", 0), ("channel", 128)):
        comp = setup_compose(dev, hy, n_layers=n_layers, variant=var)
        W, sa = comp["W"], comp["sa"]
        args = (comp["slot"], comp["T_pool"], comp["S_pool"], sa["k"], sa["v"], sa["q"], sa["g"], sa["beta"])
        ms = _time_ms(lambda: hy.compose(*args, variant=var, S_out=comp["S_out"], seam_out=comp["seam_out"]))
        path = hy.compose_path(*args, variant=var, S_out=comp["S_out"], seam_out=comp["seam_out"])
        nbytes = compose_bytes(n_layers, W.n_seg, W.seam_w, W.h_k, W.h_v, W.d_k, W.d_v, gate_floats=gate)
        gbs = nbytes / (ms * 1e-3) / 1e9
        rows[f"compose: {var}, {n_layers} layers x {W.h_v} heads x {W.n_seg} segments, w={W.seam_w}"] = {
            "ms": ms, "algorithmic_bytes": nbytes,
            "hbm": {"achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s", "frac": gbs / peaks["hbm"]},
            "kernel": path}
        del comp, sa
        torch.cuda.empty_cache()
    return rows


def forward_flops(lengths, h_v, d_k=128, d_v=128, g=2, chunk=C):
    """Algorithmic FLOPs of the prefill forward's per-token outputs on top of
    the build's: per chunk of c tokens and value head, Q S_0 2 c d_k d_v, the
    causal (Q K^T) part c (c + 1) d_k / g (its Gram shared by the g value
    heads of a key head) and its product with Delta c (c + 1) d_v."""
    tot = 0.0
    for L in lengths:
        n_full, tail = divmod(int(L), chunk)
        for c in [chunk] * n_full + ([tail] if tail else []):
            tot += 2 * c * d_k * d_v + c * (c + 1) * d_k / g + c * (c + 1) * d_v
    return tot * h_v


def forward_row(dev, hy, peaks):
    """hypic_segment_forward on the config-3 GDN layer (64 x 1024 tokens,
    16 key / 32 value heads, d = 128, bf16): the pairs and the output of
    every body token from the zero-initial body state.  On the tensor-core
    path the build records every chunk's start state and Delta and a second
    kernel forms the outputs chunk by chunk; the row reports the whole
    call's algorithmic FLOPs (build plus outputs) against the bf16 tensor
    peak, and names the output kernel that ran."""
    import torch
    import synth_inputs as si
    W = si.workload(3, seed=0, device=dev)
    L = W.layers[0]
    T = torch.empty((W.n_seg, W.h_v, W.d_k, W.d_k), device=dev)
    S = torch.empty((W.n_seg, W.h_v, W.d_k, W.d_v), device=dev)
    o = torch.empty((W.n_tokens, W.h_v, W.d_v), device=dev)
    ws = [None]

    def run():
        ws[0] = hy.segment_forward(L.k, L.v, L.q, L.g, L.beta, W.seg_offsets, variant="gdn", seam_w=0, T_pool=T,
                                   S_pool=S, o_out=o, workspace=ws[0])
    ms = _time_ms(run, reps=5, warm=2)
    path = hy.forward_path(L.k, L.v, L.q, L.g, L.beta, W.seg_offsets, variant="gdn", seam_w=0, T_pool=T, S_pool=S,
                           o_out=o)
    bodies = np.diff(W.seg_offsets) - W.seam_w
    fl = build_flops(bodies, W.h_v) + forward_flops(bodies, W.h_v)
    tf = fl / (ms * 1e-3) / 1e12
    del T, S, o, ws
    torch.cuda.empty_cache()
    return {"ms": ms, "tokens_per_s": W.n_tokens / (ms * 1e-3), "algorithmic_flops": fl,
            "tensor": {"achieved": tf, "peak": peaks["bf16"], "unit": "TFLOP/s", "frac": tf / peaks["bf16"],
                       "peak_source": peaks["src"] + " bf16 dense (burst)"},
            "kernel": "outputs: " + path}


def measure_rows(dev, hy, peaks):
    """The build rows outside the timed step, each against its own roofline:
    the RetNet-style scalar-decay fast path (8 heads, d = 128, 16 x 512
    tokens, bf16) and the cold uneven mix (256 segments of 256..8192
    tokens, 16 key / 32 value heads, d = 128, w = 8, bf16) for GDN,
    DeltaNet and the per-channel gate.  Which kernel ran is named."""
    import torch
    import synth_inputs as si
    rows = {}

    def one(name, W, round_robin=False):
        L = W.layers[0]
        T = torch.empty(hy.pool_T_shape(W.variant, W.n_seg, W.h_v, W.d_k), device=dev)
        S = torch.empty((W.n_seg, W.h_v, W.d_k, W.d_v), device=dev)
        # the workspace once, as the timed step does (a small build is
        # otherwise timed partly on the host's per-call allocation)
        ws = hy.segment_build(L.k, L.v, L.g, L.beta, W.seg_offsets, variant=W.variant, seam_w=W.seam_w,
                              T_pool=T, S_pool=S)
        ms = _time_ms(lambda: hy.segment_build(L.k, L.v, L.g, L.beta, W.seg_offsets, variant=W.variant,
                                               seam_w=W.seam_w, T_pool=T, S_pool=S, workspace=ws))
        if round_robin:
            # the same kernel and items, handed to the SMs round-robin in
            # segment order instead of longest-first (pages §2.3: LPT against
            # round-robin balancing of uneven segments)
            ms_rr = _time_ms(lambda: hy.segment_build(L.k, L.v, L.g, L.beta, W.seg_offsets, variant=W.variant,
                                                      seam_w=W.seam_w, T_pool=T, S_pool=S, workspace=ws,
                                                      flags=hy.FLAG_ROUND_ROBIN))
        bodies = np.maximum(np.diff(W.seg_offsets) - W.seam_w, 0)
        in_b = 2 if W.dtype == torch.bfloat16 else 4
        nbytes = (W.n_tokens * (W.h_k * W.d_k + W.h_v * W.d_v) * in_b + S.numel() * 4 + T.numel() * 4
                  + (L.g.numel() * 4 if L.g is not None and L.g.dim() > 1 else 0)
                  + (L.beta.numel() * 4 if L.beta is not None else 0))
        gbs = nbytes / (ms * 1e-3) / 1e9
        r = {"ms": ms, "tokens_per_s": W.n_tokens / (ms * 1e-3), "algorithmic_bytes": nbytes,
             "hbm": {"achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s", "frac": gbs / peaks["hbm"]}}
        if W.variant in ("gdn", "deltanet", "channel"):
            # the 64-token chunk formula for every variant (the per-channel
            # kernel's own chunk length does not change the algorithmic work)
            fl = build_flops(bodies, W.h_v, g=1 if W.variant == "channel" else 2)
            tf = fl / (ms * 1e-3) / 1e12
            r["tensor"] = {"achieved": tf, "peak": peaks["bf16"], "unit": "TFLOP/s", "frac": tf / peaks["bf16"]}
        r["kernel"] = hy.build_path(L.k, L.v, L.g, L.beta, W.seg_offsets, variant=W.variant, seam_w=W.seam_w,
                                    T_pool=T, S_pool=S)
        if round_robin:
            r["lpt_vs_round_robin"] = {"lpt_ms": ms, "round_robin_ms": ms_rr, "speedup": ms_rr / ms}
        rows[name] = r
        del L, T, S, ws

    one("build: RetNet scalar decay, 8 heads, 16 x 512 tokens", si.workload(2, seed=0, device=dev))
    rows["forward: GDN layer 64 x 1024 tokens, pairs + body outputs"] = forward_row(dev, hy, peaks)
    for var in ("gdn", "deltanet", "channel"):
        W = si.workload(5, seed=0, device=dev, variant=var)
        one(f"build: uneven 256-segment mix ({W.n_tokens} tokens), {var}", W, round_robin=var == "gdn")
        del W
        torch.cuda.empty_cache()
    return rows


def segment_parallel_rows(dev, hy, comp, compose_ms_one, ws, rank):
    """N > 1: the pages' segment parallelism (nav.aitube.vip §2.3) across the
    ranks, each timed as the max over ranks of CUDA-event times after two
    warm-up runs:
      cold build: the uneven 256-segment GDN prompt, segments LPT-scattered
        over the ranks, each rank's pairs sent to rank 0's pool while its
        next group builds; against rank 0 building all of it alone;
      compose: the warm-prompt chains split into one span per rank (span
        pairs all-gathered, scanned, spans composed), against one GPU's
        compose of the whole chains (the timed step's compose)."""
    import torch
    import torch.distributed as dist
    import synth_inputs as si
    from hybrid_linear_attention_chunkwise_gb300 import segment_parallel as sp

    def timed(fn, reps=3):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        t = torch.tensor([a.elapsed_time(b) / reps], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    W = si.workload(5, seed=0, device=dev, variant="gdn")
    L = W.layers[0]
    T = S = None
    if rank == 0:
        T = torch.empty((W.n_seg, W.h_v, W.d_k, W.d_k), device=dev)
        S = torch.empty_like(T)
    scatter_ms = timed(lambda: sp.cold_build_scatter(L.k, L.v, L.g, L.beta, W.seg_offsets, variant="gdn",
                                                     seam_w=W.seam_w, T_pool=T, S_pool=S, n_groups=4))
    one_ms = None
    if rank == 0:
        for _ in range(2):
            hy.segment_build(L.k, L.v, L.g, L.beta, W.seg_offsets, variant="gdn", seam_w=W.seam_w, T_pool=T,
                             S_pool=S)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(3):
            hy.segment_build(L.k, L.v, L.g, L.beta, W.seg_offsets, variant="gdn", seam_w=W.seam_w, T_pool=T,
                             S_pool=S)
        b.record()
        torch.cuda.synchronize()
        one_ms = a.elapsed_time(b) / 3
    dist.barrier()
    del W, L, T, S
    torch.cuda.empty_cache()
    sa = comp["sa"]
    seam = {k: sa[k] for k in ("k", "v", "q", "g", "beta")}
    S_out = torch.empty_like(comp["S_out"])
    shard_ms = timed(lambda: sp.compose_sharded(comp["slot"], comp["T_pool"], comp["S_pool"], seam, variant="gdn",
                                                S_out=S_out, seam_out=comp["seam_out"]))
    out = {"cold_build_scatter": {"ms": scatter_ms, "one_gpu_ms": one_ms, "ranks": ws,
                                  "speedup": (one_ms / scatter_ms) if one_ms else None,
                                  "what": "uneven 256-segment GDN prompt, LPT scatter, pairs to rank 0 by NCCL p2p"},
           "compose_sharded": {"ms": shard_ms, "one_gpu_ms": compose_ms_one, "ranks": ws,
                               "speedup": compose_ms_one / shard_ms,
                               "what": "warm-prompt chains, one span per rank, span pairs all-gathered"}}
    return out


def run_profile_case(kind):
    """One small case of one kernel for an ncu capture: two warm-up launches,
    then the launch to capture.  Inputs are larger than L2 and a few GB at
    most.  build: GDN, 16 segments x 1024 tokens, h_k = 16, h_v = 32 (512
    (segment, head) pairs); channel: the same shape with per-channel gates;
    compose: 4 GDN layers x 32 heads x 100 segments, w = 8 (12800 pairs,
    1.7 GB pool); compose_channel: the same with per-channel gates; merge: that pool's adjacent segment pairs merged (4 x 50
    merges x 32 heads); rerotate: that pool re-rotated in place (400 slots x
    32 heads); forward: the build case's forward (its output kernel); fast:
    the RetNet fast path, 8 heads x 16 segments x 8192 tokens (128 items,
    0.5 GB of keys and values)."""
    import torch
    import hybrid_linear_attention_chunkwise_gb300 as hy
    import synth_inputs as si
    dev = torch.device("cuda", 0)
    hy.load()
    if kind in ("build", "channel"):
        var = "gdn" if kind == "build" else "channel"
        W = si.workload(3, seed=0, device=dev, n_seg=16, variant=var)
        L = W.layers[0]
        T = torch.empty((W.n_seg, W.h_v, W.d_k, W.d_k), device=dev)
        S = torch.empty((W.n_seg, W.h_v, W.d_k, W.d_v), device=dev)
        ws = hy.alloc_workspace(hy.build_workspace_bytes(W.n_seg, W.h_k, W.h_v, W.d_k, W.d_v), dev)
        run = lambda: hy.segment_build(L.k, L.v, L.g, L.beta, W.seg_offsets, variant=var, seam_w=W.seam_w,
                                       T_pool=T, S_pool=S, workspace=ws)
        units = W.n_seg * W.h_v
    elif kind == "fast":
        W = si.workload(2, seed=0, device=dev, seg_len=8192)
        L = W.layers[0]
        T = torch.empty(hy.pool_T_shape(W.variant, W.n_seg, W.h_v, W.d_k), device=dev)
        S = torch.empty((W.n_seg, W.h_v, W.d_k, W.d_v), device=dev)
        ws = hy.alloc_workspace(hy.build_workspace_bytes(W.n_seg, W.h_k, W.h_v, W.d_k, W.d_v), dev)
        run = lambda: hy.segment_build(L.k, L.v, L.g, L.beta, W.seg_offsets, variant=W.variant, seam_w=W.seam_w,
                                       T_pool=T, S_pool=S, workspace=ws)
        units = W.n_seg * W.h_v
    elif kind == "merge":
        comp = setup_compose(dev, hy, n_layers=4)
        W, n_seg = comp["W"], comp["W"].n_seg
        pairs = [(l * n_seg + 2 * i + 1, l * n_seg + 2 * i) for l in range(4) for i in range(n_seg // 2)]
        later = torch.tensor([a for a, _ in pairs], dtype=torch.int32, device=dev)
        earlier = torch.tensor([b for _, b in pairs], dtype=torch.int32, device=dev)
        outs = torch.arange(len(pairs), dtype=torch.int32, device=dev)
        To = torch.empty((len(pairs), W.h_v, W.d_k, W.d_k), device=dev)
        So = torch.empty_like(To)
        run = lambda: hy.pair_merge(later, earlier, outs, comp["T_pool"], comp["S_pool"], To, So, variant="gdn")
        units = len(pairs) * W.h_v
    elif kind == "rerotate":
        comp = setup_compose(dev, hy, n_layers=4)
        W = comp["W"]
        n = comp["n_layers"] * W.n_seg
        slots = torch.arange(n, dtype=torch.int32, device=dev)
        deltas = torch.arange(n, dtype=torch.int64, device=dev) * 997 - 50000
        run = lambda: hy.pair_rerotate(slots, slots, deltas, comp["T_pool"], comp["S_pool"], comp["T_pool"],
                                       comp["S_pool"], variant="gdn", rot_dim=W.d_k, layout="half")
        units = n * W.h_v
    elif kind == "forward":
        W = si.workload(3, seed=0, device=dev, n_seg=16)
        L = W.layers[0]
        T = torch.empty((W.n_seg, W.h_v, W.d_k, W.d_k), device=dev)
        S = torch.empty((W.n_seg, W.h_v, W.d_k, W.d_v), device=dev)
        o = torch.empty((W.n_tokens, W.h_v, W.d_v), device=dev)
        run = lambda: hy.segment_forward(L.k, L.v, L.q, L.g, L.beta, W.seg_offsets, variant="gdn", seam_w=0,
                                         T_pool=T, S_pool=S, o_out=o)
        units = W.n_tokens * W.h_v
    else:
        var = "channel" if kind == "compose_channel" else "gdn"
        comp = setup_compose(dev, hy, n_layers=4, variant=var)
        sa = comp["sa"]
        run = lambda: hy.compose(comp["slot"], comp["T_pool"], comp["S_pool"], sa["k"], sa["v"], sa["q"], sa["g"],
                                 sa["beta"], variant=var, S_out=comp["S_out"], seam_out=comp["seam_out"])
        units = comp["n_layers"] * comp["W"].n_seg * comp["W"].h_v
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    print(json.dumps({"profile": kind, "units_per_launch": units, "source_sha256": source_hash(kind)}), flush=True)
    return 0


def oracle_build_sample(W, n_seg_sample, threads):
    import oracle
    L = W.layers[0]
    off = W.seg_offsets
    end = int(off[n_seg_sample])
    sub = np.asarray(off[:n_seg_sample + 1])
    k, v, g, b = (x[:end].cpu() for x in (L.k, L.v, L.g, L.beta))
    t0 = time.perf_counter()
    oracle.build_pairs("gdn", sub, W.seam_w, W.h_k, W.h_v, W.d_k, W.d_v, k, v, g, b, n_threads=threads)
    return time.perf_counter() - t0, end


def cpu_baseline(W3, threads, budget_s=15.0):
    """Oracle build throughput on a bounded sample of the same layer: the
    first few segments, all 32 value heads."""
    n = 1
    dt, tok = oracle_build_sample(W3, n, threads)
    if dt < budget_s / 4:
        n = max(1, min(W3.n_seg, int(budget_s / 2 / max(dt, 1e-3))))
        dt, tok = oracle_build_sample(W3, n, threads)
    return {"value": tok / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"fp64 token-by-token build of the first {n} of 64 segments (x1024 tokens, all 32 value "
                      f"heads) of the GDN layer; {dt:.1f} s"}


def arm_config(ws):
    """The workload both arms report (the reference arm times a bounded
    sample of it, described in its cpu_baseline)."""
    return {"workload": "build: GDN layer 64x1024 tokens, h_k=16 h_v=32 d=128 bf16 (one launch); "
                        "compose: 30 GDN layers x 32 heads, 100 lognormal segments, w=8, "
                        "12.6 GB fp32 pairs in HBM",
            "global_batch": 65536 * ws, "seq_len": 1024, "parallelism": f"dp{ws}",
            "l2": "inputs larger than L2 (no flush)"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    import torch  # noqa: F401  (inputs are drawn with torch's CPU generator)
    W3 = setup_build("cpu")
    threads = os.cpu_count() or 1
    n_seg = 1
    for _ in range(args.warmup):
        oracle_build_sample(W3, n_seg, threads)
    times = []
    for _ in range(args.steps):
        dt, tok = oracle_build_sample(W3, n_seg, threads)
        times.append(dt)
    tot = sum(times)
    value = args.steps * tok / tot
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": arm_config(1),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": "fp64 token-by-token build of 1 of the layer's 64 segments "
                                       "(1024 tokens, all 32 value heads) per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU leg
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rows", action="store_true", help="skip the per-row measurements after the step")
    ap.add_argument("--profile", choices=["build", "compose", "compose_channel", "channel", "merge", "rerotate", "forward",
                                          "fast"],
                    default=None,
                    help="run one small case of one kernel (for an ncu capture) and exit")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        return run_profile_case(args.profile)

    import torch
    import torch.distributed as dist
    import hybrid_linear_attention_chunkwise_gb300 as hy

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)
    hy.load()
    peaks = _peaks()

    # ---- set-up (untimed): inputs resident in HBM
    # weak scaling: each rank runs its own shard of independent units (seeded
    # by rank); no data-path exchange between ranks
    W3 = setup_build(dev, seed=rank)
    L3 = W3.layers[0]
    T3 = torch.empty((W3.n_seg, W3.h_v, W3.d_k, W3.d_k), device=dev)
    S3 = torch.empty((W3.n_seg, W3.h_v, W3.d_k, W3.d_v), device=dev)
    ws3 = hy.alloc_workspace(hy.build_workspace_bytes(W3.n_seg, W3.h_k, W3.h_v, W3.d_k, W3.d_v), dev)
    comp = setup_compose(dev, hy, seed=rank)
    W4 = comp["W"]
    stream = torch.cuda.current_stream()

    def do_build():
        hy.segment_build(L3.k, L3.v, L3.g, L3.beta, W3.seg_offsets, variant="gdn", seam_w=W3.seam_w,
                         T_pool=T3, S_pool=S3, workspace=ws3)

    def do_compose():
        sa = comp["sa"]
        hy.compose(comp["slot"], comp["T_pool"], comp["S_pool"], sa["k"], sa["v"], sa["q"], sa["g"], sa["beta"],
                   variant="gdn", S_out=comp["S_out"], seam_out=comp["seam_out"])

    for _ in range(args.warmup):
        do_build()
        do_compose()
    torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        clk.start()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            do_build()
            ev[i][1].record(stream)
            do_compose()
            ev[i][2].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        clk.stop()
        if ws > 1:
            dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    b_ms = float(np.mean([a.elapsed_time(b) for a, b, _ in ev]))
    c_ms = float(np.mean([b.elapsed_time(c) for _, b, c in ev]))
    if ws > 1:
        t = torch.tensor([total_ms, b_ms, c_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms, b_ms, c_ms = (float(x) for x in t.tolist())

    lens3 = np.diff(W3.seg_offsets) - W3.seam_w
    bflops = build_flops(lens3, W3.h_v)
    bbytes = build_bytes(W3.n_tokens, W3.n_seg, W3.h_k, W3.h_v)
    cbytes = compose_bytes(comp["n_layers"], W4.n_seg, W4.seam_w, W4.h_k, W4.h_v)
    cflops = compose_flops(comp["n_layers"], W4.n_seg, W4.seam_w, W4.h_v)
    tokens_per_s = ws * W3.n_tokens / (b_ms * 1e-3)
    b_tflops = bflops / (b_ms * 1e-3) / 1e12
    c_gbs = cbytes / (c_ms * 1e-3) / 1e9
    roof_build = {"bound": "tensor", "achieved": b_tflops, "peak": peaks["bf16"], "unit": "TFLOP/s",
                  "frac": b_tflops / peaks["bf16"], "traffic": captured_traffic("build", W3.n_seg * W3.h_v),
                  "kernel": "segment build", "algorithmic": bbytes,
                  "peak_source": peaks["src"] + " bf16 dense (burst)"}
    roof_comp = {"bound": "hbm", "achieved": c_gbs, "peak": peaks["hbm"], "unit": "GB/s",
                 "frac": c_gbs / peaks["hbm"],
                 "traffic": captured_traffic("compose", comp["n_layers"] * W4.n_seg * W4.h_v),
                 "kernel": "compose", "algorithmic": cbytes, "peak_source": peaks["src"] + " HBM copy"}
    dominant = roof_comp if c_ms >= b_ms else roof_build

    # ---- end to end through the public API with host buffers
    e2e = None
    if rank == 0 or ws > 1:
        pin = {n: getattr(L3, n).cpu().pin_memory() for n in ("k", "v", "g", "beta")}
        dk = {n: torch.empty_like(getattr(L3, n)) for n in ("k", "v", "g", "beta")}
        hT = torch.empty(T3.shape, dtype=torch.float32).pin_memory()
        hS = torch.empty(S3.shape, dtype=torch.float32).pin_memory()
        # the compose leg: seam tokens from host memory, states and seam
        # outputs back to host memory, the pool resident on the device
        sa4 = comp["sa"]
        keys = ("k", "v", "q", "g", "beta")
        pin4 = {n: sa4[n].cpu().pin_memory() for n in keys}
        st4 = {n: torch.empty_like(sa4[n]) for n in keys}
        hS4 = torch.empty(comp["S_out"].shape, dtype=torch.float32).pin_memory()
        ho4 = torch.empty(comp["seam_out"].shape, dtype=torch.float32).pin_memory()
        h2d = (sum(x.numel() * x.element_size() for x in pin.values())
               + sum(x.numel() * x.element_size() for x in pin4.values()))
        d2h = hT.numel() * 4 + hS.numel() * 4 + hS4.numel() * 4 + ho4.numel() * 4

        side = torch.cuda.Stream()

        def e2e_step():
            # two C-ABI calls, on two streams (the cold prompt's build and the
            # warm prompt's compose are independent): host inputs in, host
            # pairs out, the copies of one group of segments overlapping the
            # build of the next; and host seam tokens in, host states and
            # seam outputs out, the copies of one group of layers overlapping
            # the next's compose.  The step ends when both have.
            side.wait_stream(stream)
            hy.compose_host(*(pin4[n] for n in keys), comp["slot"], comp["T_pool"], comp["S_pool"], variant="gdn",
                            seam_k=st4["k"], seam_v=st4["v"], seam_q=st4["q"], seam_g=st4["g"], seam_beta=st4["beta"],
                            S_out=comp["S_out"], S_out_host=hS4, seam_out=comp["seam_out"], seam_out_host=ho4,
                            n_chunks=E2E_CHUNKS, stream=side)
            hy.segment_build_host(pin["k"], pin["v"], pin["g"], pin["beta"], W3.seg_offsets, variant="gdn",
                                  seam_w=W3.seam_w, k=dk["k"], v=dk["v"], g=dk["g"], beta=dk["beta"],
                                  T_pool=T3, S_pool=S3, T_host=hT, S_host=hS, n_chunks=E2E_CHUNKS,
                                  workspace=ws3, stream=stream)
            stream.wait_stream(side)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = e0.elapsed_time(e1) / args.steps
        e2e = {"value": ws * W3.n_tokens / (e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "what": "the whole step from host buffers, two C-ABI calls on two streams: "
                       "hypic_segment_build_host (H2D of the layer's "
                       f"k/v/g/beta from pinned memory, build, D2H of all pairs, {E2E_CHUNKS} overlapped groups of "
                       "segments) and hypic_compose_host (H2D of the warm prompt's seam tokens, compose against "
                       "the resident pool, D2H of the final states and seam outputs, overlapped groups of "
                       "layers); the host link moves about 210 GB/s one way and 300 GB/s both ways on this "
                       "GB300, so the step's copies alone take about 6.6 ms"}

    # the other build rows, each against its own roofline (after the timed
    # region; not part of the step)
    rows = None
    if rank == 0 and not args.no_rows:
        rows = {f"merge: {comp['n_layers']} layers x {W4.h_v} heads x {W4.n_seg // 2} adjacent segment pairs":
                merge_row(dev, hy, peaks, comp)}
        rows[f"re-rotation: {comp['n_layers']} layers x {W4.n_seg} segments x {W4.h_v} heads, in place"] = \
            rerotate_row(dev, hy, peaks, comp)
        rows.update(compose_variant_rows(dev, hy, peaks))
        rows.update(measure_rows(dev, hy, peaks))

    # segment parallelism across the ranks (N > 1 only; every rank takes part)
    seg_par = None
    if ws > 1 and not args.no_rows:
        seg_par = segment_parallel_rows(dev, hy, comp, c_ms, ws, rank)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(W3, os.cpu_count() or 1)

    if rank == 0:
        line = {
            "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": arm_config(ws),
            "build_ms": b_ms, "build_tflops": b_tflops,
            "compose_ms": c_ms, "compose_gbs": c_gbs, "compose_tflops": cflops / (c_ms * 1e-3) / 1e12,
            "roofline": dominant, "roofline_build": roof_build, "roofline_compose": roof_comp,
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": 2 * args.steps,
            "clocks": clk.summary(),
            "rows": rows,
            "segment_parallel": seg_par,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
