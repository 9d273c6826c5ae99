"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
binding, run the fp64 oracle on the same seeded inputs (or on sampled
segments / heads of them), and compare with the per-head relative Frobenius
rule of tolerance.py."""
from __future__ import annotations

import numpy as np
import torch

import hybrid_linear_attention_chunkwise_gb300 as hy
import oracle
import synth_inputs as si
from tolerance import TOL_BF16, TOL_F32, per_head_rel_err

DENSE = ("gdn", "deltanet", "channel")


def tol_for(dtype):
    return TOL_BF16 if dtype == torch.bfloat16 else TOL_F32


def new_pools(variant, n_slots, h_v, d_k, d_v, device="cuda", fill=float("nan")):
    T = torch.full(hy.pool_T_shape(variant, n_slots, h_v, d_k), fill, device=device)
    S = torch.full((n_slots, h_v, d_k, d_v), fill, device=device)
    return T, S


def gpu_build(W, layer=0, slots=None, n_slots=None, status=None, flags=0, stream=None, T_pool=None,
              S_pool=None, variant=None):
    L = W.layers[layer]
    variant = variant or W.variant
    n_slots = n_slots or (W.n_seg if slots is None else int(max(slots)) + 1)
    if T_pool is None:
        T_pool, S_pool = new_pools(variant, n_slots, W.h_v, W.d_k, W.d_v, L.k.device)
    hy.segment_build(L.k, L.v, L.g, L.beta, W.seg_offsets, variant=variant, seam_w=W.seam_w,
                     T_pool=T_pool, S_pool=S_pool, slot_of_seg=slots, status=status, flags=flags,
                     stream=stream)
    return T_pool, S_pool


def dense_T(variant, T, d_k):
    """Expand scalar / diagonal pool transitions to dense matrices (fp64)."""
    T = T.detach().cpu().double().numpy() if hasattr(T, "detach") else np.asarray(T, np.float64)
    if variant in DENSE:
        return T
    if variant == "diag":
        return np.einsum("...i,ij->...ij", T, np.eye(d_k))
    return T[..., None, None] * np.eye(d_k)


def _cpu(x):
    return None if x is None else x.detach().cpu()


def sub_layer(W, layer, segs, heads=None):
    """Token inputs of the listed segments (concatenated) and, optionally,
    of one key-head group: returns (k, v, g, beta, q, offsets, h_k, h_v)."""
    L = W.layers[layer]
    off = W.seg_offsets
    idx = np.concatenate([np.arange(off[i], off[i + 1]) for i in segs]) if len(segs) else np.zeros(0, np.int64)
    lens = [int(off[i + 1] - off[i]) for i in segs]
    sub_off = si.offsets_from_lengths(lens)
    t = torch.as_tensor(idx, dtype=torch.long, device=L.k.device)
    k, v, q = L.k[t], L.v[t], L.q[t]
    g = L.g
    if g is not None and g.dim() > 1:
        g = g[t]
    beta = L.beta[t] if L.beta is not None else None
    h_k, h_v = W.h_k, W.h_v
    if heads is not None:
        kh, vh = heads
        k, q = k[:, kh], q[:, kh]
        v = v[:, vh]
        if g is not None:
            g = g[vh] if g.dim() == 1 else g[:, vh]
        if beta is not None:
            beta = beta[:, vh]
        h_k, h_v = len(kh), len(vh)
    return [_cpu(x) for x in (k, v, g, beta, q)] + [sub_off, h_k, h_v]


def oracle_pairs(W, layer=0, segs=None, heads=None, variant=None):
    segs = list(range(W.n_seg)) if segs is None else list(segs)
    k, v, g, beta, q, off, h_k, h_v = sub_layer(W, layer, segs, heads)
    return oracle.build_pairs(variant or W.variant, off, W.seam_w, h_k, h_v, W.d_k, W.d_v, k, v, g, beta)


def compare_pairs(W, T_pool, S_pool, T_ref, S_ref, segs, slots=None, heads=None, variant=None):
    """Max per-head relative error of T and S for the listed segments."""
    variant = variant or W.variant
    slots = np.arange(W.n_seg) if slots is None else np.asarray(slots)
    sl = torch.as_tensor(slots[list(segs)], dtype=torch.long, device=T_pool.device)
    Tg = T_pool[sl]
    Sg = S_pool[sl]
    if heads is not None:
        hv = torch.as_tensor(heads[1], dtype=torch.long, device=T_pool.device)
        Tg, Sg = Tg[:, hv], Sg[:, hv]
    eT = per_head_rel_err(dense_T(variant, Tg, W.d_k), T_ref)
    eS = per_head_rel_err(Sg, S_ref)
    return float(eT.max()), float(eS.max())


def seam_arrays(W, layers=None):
    """Stack the seam tokens of the given layers: dict of [L, n_seg, w, ...]."""
    layers = range(len(W.layers)) if layers is None else layers
    parts = [si.seam_gather(W, W.layers[l]) for l in layers]
    out = {}
    for key in ("k", "v", "q", "g", "beta"):
        if parts[0][key] is None:
            out[key] = None
        elif parts[0][key].dim() == 1:          # scalar decay: per layer per head
            out[key] = torch.stack([p[key] for p in parts]).contiguous()
        else:
            out[key] = torch.stack([p[key] for p in parts]).contiguous()
    return out
