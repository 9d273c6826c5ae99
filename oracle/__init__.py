"""fp64 CPU oracle for the HYPIC linear-attention state algebra.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may import this package; the product library never
does, and this package imports nothing from it.

What it computes (per the HYPIC news pages, nav.aitube.vip §2.1/§2.2 and the
xix.ai linear-layer and seam paragraphs):
  build    -- per segment and value head, T_C = product of the body's token
              transitions and S(C|0) = the body's final state from zero;
  compose  -- in prompt order: seam tokens one at a time (emit o_t = S_t^T q_t),
              then S <- T_C S + S(C|0);
  full     -- the plain recurrence over a whole prompt (the full recompute);
  merge    -- (T2,S2) o (T1,S1) = (T2 T1, T2 S1 + S2);
  rerotate -- the state re-rotation patch for RoPE-shifted reuse
              (R T_C R^T, R S(C|0)), numpy fp64 (reading of the pages' one
              sentence on it: rotary angles position x base^(-2i/rot_dim));
  naive    -- the straw man: sum of zero-initial states.
The arithmetic is the C file ``hypic_oracle.c`` (fp64, token by token);
``dense_twin`` restates the definition with explicit dense matrices for tiny
cases and is one of the oracle's pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hypic_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "libhypic_oracle.so")
_lock = threading.Lock()
_default = None

VARIANT_CODE = {"gdn": 0, "deltanet": 1, "channel": 2, "scalar": 3, "ungated": 4, "diag": 5}


def compile_oracle(src: str, out: str) -> str:
    """gcc -O2 -fopenmp: compile an oracle C source into a shared object."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the C oracle into oracle/_build/ (if stale)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        compile_oracle(_SRC, _SO)
    return _SO


def _f64(x):
    """Upcast to a contiguous fp64 numpy array (None passes through)."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu").to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


class OracleLib:
    """ctypes view of one compiled oracle shared object."""

    def __init__(self, so_path: str):
        lib = ctypes.CDLL(so_path)
        P, I, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        lib.oracle_build.argtypes = [I, I, P, I, I, I, I, I, P, P, P, P, P, P, I]
        lib.oracle_compose.argtypes = [I, I, I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, I]
        lib.oracle_full.argtypes = [I, L, I, I, I, I, P, P, P, P, P, P, P, L, P, P, I]
        lib.oracle_merge.argtypes = [I, I, I, P, P, P, P, P, P]
        for f in (lib.oracle_build, lib.oracle_compose, lib.oracle_full, lib.oracle_merge):
            f.restype = I
        self.lib = lib

    def build_pairs(self, variant, seg_offsets, seam_w, h_k, h_v, d_k, d_v, k, v, g=None, beta=None,
                    n_threads=0):
        """Returns (T [n_seg,h_v,d_k,d_k], S [n_seg,h_v,d_k,d_v]) in fp64."""
        off = np.ascontiguousarray(np.asarray(seg_offsets, dtype=np.int64))
        n_seg = len(off) - 1
        k, v, g, beta = _f64(k), _f64(v), _f64(g), _f64(beta)
        T = np.empty((n_seg, h_v, d_k, d_k))
        S = np.empty((n_seg, h_v, d_k, d_v))
        self.lib.oracle_build(VARIANT_CODE[variant], n_seg, _p(off), int(seam_w), h_k, h_v, d_k, d_v,
                              _p(k), _p(v), _p(g), _p(beta), _p(T), _p(S), _threads(n_threads))
        return T, S

    def compose(self, variant, T_pairs, S_pairs, seam_k, seam_v, seam_q, seam_g, seam_beta, h_k, h_v,
                S_init=None, n_threads=0):
        """Pairs in prompt order: T_pairs [L,n_seg,h_v,d_k,d_k] (dense),
        S_pairs [L,n_seg,h_v,d_k,d_v]; seam arrays [L,n_seg,w,heads,...]
        (scalar-decay gate: [h_v]).  Returns (S_out [L,h_v,d_k,d_v],
        seam_out [L,n_seg,w,h_v,d_v])."""
        T_pairs, S_pairs = _f64(T_pairs), _f64(S_pairs)
        n_layers, n_seg, _, d_k, _ = T_pairs.shape
        d_v = S_pairs.shape[-1]
        sk, sv, sq, sg, sb = _f64(seam_k), _f64(seam_v), _f64(seam_q), _f64(seam_g), _f64(seam_beta)
        w = sk.shape[2]
        S_init = _f64(S_init)
        S_out = np.empty((n_layers, h_v, d_k, d_v))
        seam_out = np.empty((n_layers, n_seg, w, h_v, d_v))
        self.lib.oracle_compose(VARIANT_CODE[variant], n_layers, n_seg, w, h_k, h_v, d_k, d_v,
                                _p(T_pairs), _p(S_pairs), _p(sk), _p(sv), _p(sq), _p(sg), _p(sb),
                                _p(S_init), _p(S_out), _p(seam_out), _threads(n_threads))
        return S_out, seam_out

    def full(self, variant, k, v, q, g, beta, h_k, h_v, S_init=None, out_pos=(), n_threads=0):
        """Plain recurrence over one layer's tokens.  Returns (S_final
        [h_v,d_k,d_v], outs [len(out_pos),h_v,d_v]) with o_t = S_t^T q_t after
        token t."""
        k, v, q, g, beta, S_init = _f64(k), _f64(v), _f64(q), _f64(g), _f64(beta), _f64(S_init)
        N, _, d_k = k.shape
        d_v = v.shape[-1]
        pos = np.ascontiguousarray(np.asarray(out_pos, dtype=np.int64))
        assert np.all(np.diff(pos) >= 0)
        S = np.empty((h_v, d_k, d_v))
        outs = np.empty((len(pos), h_v, d_v))
        self.lib.oracle_full(VARIANT_CODE[variant], N, h_k, h_v, d_k, d_v, _p(k), _p(v), _p(q), _p(g),
                             _p(beta), _p(S_init), _p(pos) if len(pos) else None, len(pos), _p(S),
                             _p(outs), _threads(n_threads))
        return S, outs

    def merge(self, T2, S2, T1, S1):
        """(T2,S2) o (T1,S1) = (T2 T1, T2 S1 + S2) over leading batch axes."""
        T2, S2, T1, S1 = (_f64(x) for x in (T2, S2, T1, S1))
        d_k, d_v = T2.shape[-1], S2.shape[-1]
        n = int(np.prod(T2.shape[:-2]))
        To = np.empty(T2.shape)
        So = np.empty(S2.shape)
        self.lib.oracle_merge(n, d_k, d_v, _p(T2), _p(S2), _p(T1), _p(S1), _p(To), _p(So))
        return To, So


def default() -> OracleLib:
    global _default
    with _lock:
        if _default is None:
            _default = OracleLib(build())
    return _default


def build_pairs(*a, **kw):
    return default().build_pairs(*a, **kw)


def compose(*a, **kw):
    return default().compose(*a, **kw)


def full(*a, **kw):
    return default().full(*a, **kw)


def merge(*a, **kw):
    return default().merge(*a, **kw)


def rerotation_matrix(d_k, delta, rot_dim, layout="interleaved", base=10000.0):
    """R(delta) for the state re-rotation patch (HYPIC news pages §2.1, last
    paragraph: variants with RoPE re-rotate the cached state; the pages give
    no formula).  Reading used here: rotary position embedding rotates key
    channel pairs by the angle (position x theta_i), theta_i =
    base^(-2i / rot_dim), i < rot_dim / 2; moving a segment by delta positions
    therefore multiplies every key by the block-diagonal R(delta) below.
    Pairs are (2i, 2i + 1) ("interleaved") or (i, i + rot_dim / 2) ("half");
    channels >= rot_dim are not rotated.  Each pair block is
    [[cos phi, -sin phi], [sin phi, cos phi]], phi = delta theta_i."""
    R = np.eye(d_k)
    h = rot_dim // 2
    for i in range(h):
        phi = float(delta) * base ** (-2.0 * i / rot_dim)
        c, s = np.cos(phi), np.sin(phi)
        a, b = (2 * i, 2 * i + 1) if layout == "interleaved" else (i, i + h)
        R[a, a], R[a, b], R[b, a], R[b, b] = c, -s, s, c
    return R


def rerotate(variant, T, S, deltas, rot_dim, layout="interleaved", base=10000.0):
    """State re-rotation of cached pairs moved by deltas[m] positions: with
    keys k' = R k every token transition of a scalar-gated variant becomes
    R T_t R^T and every write R U_t, so the pair becomes
    (R T_C R^T, R S(C|0)).  T: dense [n, h_v, d_k, d_k] (gdn, deltanet) or
    scalar [n, h_v] (scalar, ungated; unchanged); S: [n, h_v, d_k, d_v]."""
    T, S = _f64(T), _f64(S)
    d_k = S.shape[-2]
    To, So = T.copy(), np.empty_like(S)
    for m, dl in enumerate(np.asarray(deltas).reshape(-1)):
        R = rerotation_matrix(d_k, dl, rot_dim, layout, base)
        So[m] = R @ S[m]
        if variant in ("gdn", "deltanet"):
            To[m] = R @ T[m] @ R.T
        elif variant not in ("scalar", "ungated"):
            raise ValueError(f"re-rotation is exact only for scalar gates, not {variant}")
    return To, So


def naive_sum(S_pairs):
    """The straw man the pages reject: sum of zero-initial final states over
    the segment axis (axis -4 of [.., n_seg, h_v, d_k, d_v])."""
    return _f64(S_pairs).sum(axis=-4)
