"""Seeded synthetic inputs for the segment build and the compose.

This module draws random numbers and lays them out; it holds none of the
method's arithmetic.  It is the one module that both the fp64 oracle (through
the tests) and the CUDA path (through the binding, the tests and the bench)
read their inputs from.

Shapes and distributions follow the five workloads of the HYPIC state algebra:

  1  tiny gated delta rule: 1 head, d=16, 4 segments x 64 tokens, seam w=8,
     fp32 values (the fp64 check case)
  2  RetNet-style scalar decay: 8 heads, gamma_h = 1 - 2^(-5-h), d=128,
     16 segments x 512 tokens, bf16 k/v/q
  3  gated delta (GDN) layer shaped like a Qwen3.5-35B-A3B linear layer:
     16 key heads shared by 32 value heads, d=128, 64 segments x 1024 tokens,
     no seam, bf16
  4  warm RAG prompt: 30 GDN layers with the shapes of 3, 100 segments with
     lognormal lengths (median 1000, sigma 0.3, clipped to 512..4096), w=8
  5  cold uneven build: 256 segments with lengths from {256,1024,4096,8192}
     (p = 0.4/0.3/0.2/0.1), 32 value heads, 16 key heads, d=128, bf16, w=8,
     variants gdn / deltanet / channel (per-channel gate)

Draws: k ~ N(0,1) then L2-normalised (in fp64); v, q ~ N(0,1);
beta = sigmoid(N(0,1)); gates are stored as log-gates g = log(alpha):
workload 1 g = -u, u ~ U(0.001, 0.1); workloads 3-5 g ~ U(-0.1, -0.001);
per-channel g = -softplus(N(0,1)).  Every tensor is rounded once to its
storage dtype (fp32 or bf16, round-to-nearest-even); the oracle reads the
rounded values upcast to fp64.

Seeds: numpy SeedSequence([seed, config_id, layer, tensor_id]) drives every
stream; torch generators are seeded from it, so the same call gives the same
tensors on the CPU and, for a given torch build, on a GPU.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

# tensor ids inside one (config, layer) stream
_TID = {"k": 0, "v": 1, "q": 2, "g": 3, "beta": 4, "len": 5, "sinit": 6, "misc": 7}

VARIANTS = ("gdn", "deltanet", "channel", "scalar", "ungated", "diag")


def _seed(seed: int, cfg: int, layer: int, tid: str) -> int:
    ss = np.random.SeedSequence([seed, cfg, layer, _TID[tid]])
    return int(ss.generate_state(1, dtype=np.uint64)[0] & ((1 << 63) - 1))


def _gen(seed, cfg, layer, tid, device):
    g = torch.Generator(device=device)
    g.manual_seed(_seed(seed, cfg, layer, tid))
    return g


@dataclass
class Layer:
    """One linear-attention layer's token inputs over the whole prompt.

    k [N, h_k, d_k], v [N, h_v, d_v], q [N, h_k, d_k] in `dtype`;
    g: gdn [N, h_v] fp32, channel/diag [N, h_v, d_k] fp32, scalar [h_v] fp32,
    None for deltanet/ungated; beta [N, h_v] fp32 for the delta variants, else None.
    """
    k: torch.Tensor
    v: torch.Tensor
    q: torch.Tensor
    g: torch.Tensor | None
    beta: torch.Tensor | None


@dataclass
class Workload:
    cfg: int
    variant: str
    h_k: int
    h_v: int
    d_k: int
    d_v: int
    seam_w: int
    dtype: torch.dtype            # storage dtype of k, v, q
    seg_offsets: np.ndarray       # int64 [n_seg+1]
    layers: list = field(default_factory=list)

    @property
    def n_seg(self):
        return len(self.seg_offsets) - 1

    @property
    def n_tokens(self):
        return int(self.seg_offsets[-1])


def _normal(shape, gen, device, dtype=torch.float64):
    return torch.randn(shape, generator=gen, device=device, dtype=dtype)


def _uniform(shape, lo, hi, gen, device, dtype=torch.float64):
    u = torch.rand(shape, generator=gen, device=device, dtype=dtype)
    return lo + (hi - lo) * u


def make_layer(*, seed, cfg, layer, n_tokens, h_k, h_v, d_k, d_v, variant,
               dtype, gate="u_small", device="cpu", decay_h=None):
    """Draw one layer's inputs.  `gate` picks the log-gate law:
    'neg_u' (g = -U(0.001, 0.1)), 'u_small' (g ~ U(-0.1, -0.001)),
    'softplus' (g = -softplus(N(0,1)), per channel)."""
    dev = torch.device(device)
    big = n_tokens * max(h_k * d_k, h_v * d_v) > (1 << 27)
    fdt = torch.float32 if big else torch.float64
    kk = _normal((n_tokens, h_k, d_k), _gen(seed, cfg, layer, "k", dev), dev, torch.float64 if not big else torch.float32)
    kk = kk.to(torch.float64) if not big else kk
    kk = kk / kk.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    k = kk.to(dtype)
    del kk
    v = _normal((n_tokens, h_v, d_v), _gen(seed, cfg, layer, "v", dev), dev, fdt).to(dtype)
    q = _normal((n_tokens, h_k, d_k), _gen(seed, cfg, layer, "q", dev), dev, fdt).to(dtype)
    gg = _gen(seed, cfg, layer, "g", dev)
    if variant in ("gdn",):
        if gate == "neg_u":
            g = -_uniform((n_tokens, h_v), 0.001, 0.1, gg, dev, fdt)
        else:
            g = _uniform((n_tokens, h_v), -0.1, -0.001, gg, dev, fdt)
        g = g.to(torch.float32)
    elif variant in ("channel", "diag"):
        x = _normal((n_tokens, h_v, d_k), gg, dev, torch.float32)
        g = (-torch.nn.functional.softplus(x)).to(torch.float32)
    elif variant == "scalar":
        assert decay_h is not None
        g = torch.tensor([math.log(x) for x in decay_h], dtype=torch.float64).to(torch.float32).to(dev)
    else:
        g = None
    if variant in ("gdn", "deltanet", "channel"):
        b = _normal((n_tokens, h_v), _gen(seed, cfg, layer, "beta", dev), dev, fdt)
        beta = torch.sigmoid(b).to(torch.float32)
    else:
        beta = None
    return Layer(k=k, v=v, q=q, g=g, beta=beta)


def offsets_from_lengths(lengths) -> np.ndarray:
    off = np.zeros(len(lengths) + 1, dtype=np.int64)
    off[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return off


def lognormal_lengths(n, seed, cfg, median=1000.0, sigma=0.3, lo=512, hi=4096):
    rng = np.random.default_rng(np.random.SeedSequence([seed, cfg, 0, _TID["len"]]))
    x = np.exp(np.log(median) + sigma * rng.standard_normal(n))
    return np.clip(np.rint(x), lo, hi).astype(np.int64)


def mix_lengths(n, seed, cfg, choices=(256, 1024, 4096, 8192), p=(0.4, 0.3, 0.2, 0.1)):
    rng = np.random.default_rng(np.random.SeedSequence([seed, cfg, 0, _TID["len"]]))
    return rng.choice(np.asarray(choices, dtype=np.int64), size=n, p=np.asarray(p))


def retnet_gammas(h):
    return [1.0 - 2.0 ** (-5 - i) for i in range(h)]


def workload(cfg: int, *, seed: int = 0, device="cpu", variant=None, n_layers=None,
             n_seg=None, seg_len=None, lengths=None, h_k=None, h_v=None, d=None,
             seam_w=None, dtype=None) -> Workload:
    """Build config `cfg` (1..5).  Keyword overrides give scaled-down cases
    with the same structure (used for CPU-sized parity runs)."""
    if cfg == 1:
        P = dict(variant="gdn", h_k=1, h_v=1, d=16, n_seg=4, seg_len=64, w=8,
                 dtype=torch.float32, gate="neg_u", n_layers=1)
    elif cfg == 2:
        P = dict(variant="scalar", h_k=8, h_v=8, d=128, n_seg=16, seg_len=512, w=8,
                 dtype=torch.bfloat16, gate=None, n_layers=1)
    elif cfg == 3:
        P = dict(variant="gdn", h_k=16, h_v=32, d=128, n_seg=64, seg_len=1024, w=0,
                 dtype=torch.bfloat16, gate="u_small", n_layers=1)
    elif cfg == 4:
        P = dict(variant="gdn", h_k=16, h_v=32, d=128, n_seg=100, seg_len=None, w=8,
                 dtype=torch.bfloat16, gate="u_small", n_layers=30)
    elif cfg == 5:
        P = dict(variant="gdn", h_k=16, h_v=32, d=128, n_seg=256, seg_len=None, w=8,
                 dtype=torch.bfloat16, gate="u_small", n_layers=1)
    else:
        raise ValueError(cfg)
    if variant is not None:
        P["variant"] = variant
    if P["variant"] == "channel":
        P["gate"] = "softplus"
    for key, val in (("n_layers", n_layers), ("n_seg", n_seg), ("seg_len", seg_len),
                     ("h_k", h_k), ("h_v", h_v), ("d", d), ("w", seam_w), ("dtype", dtype)):
        if val is not None:
            P[key] = val
    if lengths is not None:
        lens = np.asarray(lengths, dtype=np.int64)
    elif P["seg_len"] is not None:
        lens = np.full(P["n_seg"], P["seg_len"], dtype=np.int64)
    elif cfg == 4:
        lens = lognormal_lengths(P["n_seg"], seed, cfg)
    else:
        lens = mix_lengths(P["n_seg"], seed, cfg)
    off = offsets_from_lengths(lens)
    W = Workload(cfg=cfg, variant=P["variant"], h_k=P["h_k"], h_v=P["h_v"], d_k=P["d"],
                 d_v=P["d"], seam_w=P["w"], dtype=P["dtype"], seg_offsets=off)
    decay = retnet_gammas(P["h_v"]) if P["variant"] == "scalar" else None
    for layer in range(P["n_layers"]):
        W.layers.append(make_layer(seed=seed, cfg=cfg, layer=layer, n_tokens=int(off[-1]),
                                   h_k=P["h_k"], h_v=P["h_v"], d_k=P["d"], d_v=P["d"],
                                   variant=P["variant"], dtype=P["dtype"], gate=P["gate"],
                                   device=device, decay_h=decay))
    return W


def random_state(shape, *, seed, cfg, layer=0, device="cpu", scale=1.0):
    """A random fp32 prefix state S_0 (for composition checks)."""
    g = _gen(seed, cfg, layer, "sinit", torch.device(device))
    return (scale * torch.randn(shape, generator=g, device=device, dtype=torch.float64)).to(torch.float32)


def seam_gather(W: Workload, layer: Layer, w: int | None = None):
    """Gather the first w tokens of every segment into [n_seg, w, ...] arrays.
    Segments shorter than w are padded with identity tokens (k=v=q=0, g=0,
    beta=0), whose outputs carry no meaning."""
    w = W.seam_w if w is None else w
    off = W.seg_offsets
    n_seg = len(off) - 1
    dev = layer.k.device
    idx = torch.zeros((n_seg, w), dtype=torch.long)
    valid = torch.zeros((n_seg, w), dtype=torch.bool)
    for i in range(n_seg):
        L = int(off[i + 1] - off[i])
        for t in range(min(w, L)):
            idx[i, t] = int(off[i]) + t
            valid[i, t] = True
    idx = idx.to(dev)
    valid = valid.to(dev)

    def take(x):
        if x is None:
            return None
        if x.dim() == 1:             # per-head constant (scalar decay)
            return x
        y = x[idx.reshape(-1)].reshape((n_seg, w) + tuple(x.shape[1:])).clone()
        m = valid.reshape((n_seg, w) + (1,) * (x.dim() - 1))
        return torch.where(m, y, torch.zeros((), dtype=y.dtype, device=dev))

    return dict(k=take(layer.k), v=take(layer.v), q=take(layer.q), g=take(layer.g),
                beta=take(layer.beta), valid=valid)
