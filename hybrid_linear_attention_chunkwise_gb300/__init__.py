"""Python binding of libhypic: the linear-attention state algebra behind
HYPIC's position-independent caching, on GB300 (sm_103a).

Argument marshalling only -- every step of the path runs in the CUDA kernels
of ``libhypic.so`` behind the C ABI of ``include/hypic.h``.  PyTorch supplies
device memory and streams.  There is no CPU fallback: if the library is not
built, every call raises.

Entry points (same names as the C ABI):
  segment_build(...)   -> cache (T_C, S(C|0)) of every (segment, value head)
  compose(...)         -> running state + seam outputs from cached pairs
  plan_lpt(...)        -> longest-processing-time-first packing (host)
  build_workspace_bytes(...), alloc_workspace(...)
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libhypic.so")
_lock = threading.Lock()
_lib = None

GDN, DELTANET, CHANNEL_DELTA, SCALAR_DECAY, UNGATED, DIAG_GATE = range(6)
VARIANT = {"gdn": GDN, "deltanet": DELTANET, "channel": CHANNEL_DELTA, "scalar": SCALAR_DECAY,
           "ungated": UNGATED, "diag": DIAG_GATE}
IN_BF16, IN_F32 = 0, 1
FLAG_CHECK_FINITE = 1
FLAG_ROUND_ROBIN = 2            # build: static round-robin schedule (measurement)
FLAG_REQUIRE_TENSOR_CORES = 4   # refuse calls that would run an fp32 CUDA-core kernel
FLAG_TRANSITION_ONLY = 8        # compose: the product of the transitions alone
SLOT_SKIP = -1                  # build: leave this segment out
PATHS = ("none", "tc_chunkwise", "tc_channel", "tc_fast", "f32_token", "tc_compose", "f32_compose", "tc_merge",
         "f32_merge", "tc_forward")
STATUS_TIMEOUT, STATUS_NONFINITE, STATUS_BAD_SLOT = 1, 2, 4
OK = 0

P = ctypes.c_void_p


class BuildDesc(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_int32), ("n_seg", ctypes.c_int32),
                ("h_k", ctypes.c_int32), ("h_v", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("seam_w", ctypes.c_int32), ("variant", ctypes.c_int32),
                ("in_dtype", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("k", P), ("v", P), ("g", P), ("beta", P),
                ("seg_offsets", P), ("slot_of_seg", P), ("n_slots", ctypes.c_int64),
                ("T_pool", P), ("S_pool", P), ("workspace", P), ("workspace_bytes", ctypes.c_size_t),
                ("status", P)]


class ComposeDesc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_seg", ctypes.c_int32),
                ("h_k", ctypes.c_int32), ("h_v", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("seam_w", ctypes.c_int32), ("variant", ctypes.c_int32),
                ("in_dtype", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("slot", P), ("n_slots", ctypes.c_int64), ("T_pool", P), ("S_pool", P),
                ("seam_k", P), ("seam_v", P), ("seam_q", P), ("seam_g", P), ("seam_beta", P),
                ("S_init", P), ("S_out", P), ("seam_out", P),
                ("workspace", P), ("workspace_bytes", ctypes.c_size_t), ("status", P),
                ("seg_stride", ctypes.c_int32)]


class HostComposeDesc(ctypes.Structure):
    _fields_ = [("compose", ComposeDesc), ("host_seam_k", P), ("host_seam_v", P), ("host_seam_q", P),
                ("host_seam_g", P), ("host_seam_beta", P), ("host_S_init", P), ("host_S_out", P),
                ("host_seam_out", P), ("n_chunks", ctypes.c_int32)]


class SpanScanDesc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_spans", ctypes.c_int32), ("h_v", ctypes.c_int32),
                ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("T_span", P), ("S_span", P), ("S_init", P), ("S_start", P),
                ("workspace", P), ("workspace_bytes", ctypes.c_size_t), ("status", P)]


class MergeDesc(ctypes.Structure):
    _fields_ = [("n_merge", ctypes.c_int32), ("h_v", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("variant", ctypes.c_int32),
                ("later", P), ("earlier", P), ("out", P),
                ("n_slots_a", ctypes.c_int64), ("n_slots_b", ctypes.c_int64), ("n_slots_out", ctypes.c_int64),
                ("T_a", P), ("S_a", P), ("T_b", P), ("S_b", P), ("T_out", P), ("S_out", P), ("status", P)]


class ForwardDesc(ctypes.Structure):
    _fields_ = [("build", BuildDesc), ("q", P), ("o_out", P)]


class HostBuildDesc(ctypes.Structure):
    _fields_ = [("build", BuildDesc), ("host_k", P), ("host_v", P), ("host_g", P), ("host_beta", P),
                ("host_T", P), ("host_S", P), ("n_chunks", ctypes.c_int32)]


class RerotateDesc(ctypes.Structure):
    _fields_ = [("n_items", ctypes.c_int32), ("h_v", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("variant", ctypes.c_int32), ("rot_dim", ctypes.c_int32),
                ("layout", ctypes.c_int32), ("base", ctypes.c_double),
                ("slot_in", P), ("slot_out", P), ("delta", P),
                ("n_slots_in", ctypes.c_int64), ("n_slots_out", ctypes.c_int64),
                ("T_in", P), ("S_in", P), ("T_out", P), ("S_out", P), ("status", P)]


ROPE_LAYOUT = {"interleaved": 0, "half": 1}

SYMBOLS = ("hypic_segment_build", "hypic_segment_build_noalloc", "hypic_build_workspace_bytes", "hypic_compose",
           "hypic_compose_workspace_bytes", "hypic_pair_merge", "hypic_pair_rerotate", "hypic_segment_forward",
           "hypic_segment_build_host", "hypic_compose_host",
           "hypic_build_path", "hypic_forward_path", "hypic_compose_path", "hypic_merge_path",
           "hypic_span_scan", "hypic_span_scan_workspace_bytes", "hypic_compose_spans", "hypic_forward_workspace_bytes",
           "hypic_compose_spans_workspace_bytes",
           "hypic_plan_lpt",
           "hypic_status_from_word", "hypic_status_string", "hypic_version")


class HypicError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load libhypic.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"libhypic.so is not built ({_LIB_PATH}); run __graft_entry__.build()")
            lib = ctypes.CDLL(_LIB_PATH)
            lib.hypic_segment_build.argtypes = [ctypes.POINTER(BuildDesc), P]
            lib.hypic_segment_build.restype = ctypes.c_int
            lib.hypic_segment_build_noalloc.argtypes = [ctypes.POINTER(BuildDesc), P]
            lib.hypic_segment_build_noalloc.restype = ctypes.c_int
            lib.hypic_build_workspace_bytes.argtypes = [ctypes.POINTER(BuildDesc)]
            lib.hypic_build_workspace_bytes.restype = ctypes.c_size_t
            lib.hypic_compose.argtypes = [ctypes.POINTER(ComposeDesc), P]
            lib.hypic_compose.restype = ctypes.c_int
            lib.hypic_compose_workspace_bytes.argtypes = [ctypes.POINTER(ComposeDesc)]
            lib.hypic_compose_workspace_bytes.restype = ctypes.c_size_t
            lib.hypic_pair_merge.argtypes = [ctypes.POINTER(MergeDesc), P]
            lib.hypic_pair_merge.restype = ctypes.c_int
            lib.hypic_segment_forward.argtypes = [ctypes.POINTER(ForwardDesc), P]
            lib.hypic_segment_forward.restype = ctypes.c_int
            lib.hypic_segment_build_host.argtypes = [ctypes.POINTER(HostBuildDesc), P]
            lib.hypic_segment_build_host.restype = ctypes.c_int
            lib.hypic_pair_rerotate.argtypes = [ctypes.POINTER(RerotateDesc), P]
            lib.hypic_pair_rerotate.restype = ctypes.c_int
            for name, desc in (("hypic_build_path", BuildDesc), ("hypic_forward_path", ForwardDesc),
                               ("hypic_compose_path", ComposeDesc), ("hypic_merge_path", MergeDesc)):
                getattr(lib, name).argtypes = [ctypes.POINTER(desc)]
                getattr(lib, name).restype = ctypes.c_int
            lib.hypic_compose_host.argtypes = [ctypes.POINTER(HostComposeDesc), P]
            lib.hypic_compose_host.restype = ctypes.c_int
            lib.hypic_forward_workspace_bytes.argtypes = [ctypes.POINTER(ForwardDesc)]
            lib.hypic_forward_workspace_bytes.restype = ctypes.c_size_t
            lib.hypic_span_scan.argtypes = [ctypes.POINTER(SpanScanDesc), P]
            lib.hypic_span_scan.restype = ctypes.c_int
            lib.hypic_span_scan_workspace_bytes.argtypes = [ctypes.POINTER(SpanScanDesc)]
            lib.hypic_span_scan_workspace_bytes.restype = ctypes.c_size_t
            lib.hypic_compose_spans.argtypes = [ctypes.POINTER(ComposeDesc), ctypes.c_int32, P, P]
            lib.hypic_compose_spans.restype = ctypes.c_int
            lib.hypic_compose_spans_workspace_bytes.argtypes = [ctypes.POINTER(ComposeDesc), ctypes.c_int32]
            lib.hypic_compose_spans_workspace_bytes.restype = ctypes.c_size_t
            lib.hypic_plan_lpt.argtypes = [P, ctypes.c_int32, ctypes.c_int32, P, P, P]
            lib.hypic_plan_lpt.restype = ctypes.c_int
            lib.hypic_status_from_word.argtypes = [ctypes.c_uint32]
            lib.hypic_status_from_word.restype = ctypes.c_int
            lib.hypic_status_string.argtypes = [ctypes.c_int]
            lib.hypic_status_string.restype = ctypes.c_char_p
            lib.hypic_version.restype = ctypes.c_int
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load().hypic_status_string(int(code)).decode()


def status_from_word(word: int) -> int:
    return load().hypic_status_from_word(int(word) & 0xFFFFFFFF)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _in_dtype(t):
    if t.dtype == torch.bfloat16:
        return IN_BF16
    if t.dtype == torch.float32:
        return IN_F32
    raise ValueError(f"unsupported input dtype {t.dtype}")


def pool_T_shape(variant: str, n_slots: int, h_v: int, d_k: int):
    v = VARIANT[variant]
    if v in (GDN, DELTANET, CHANNEL_DELTA):
        return (n_slots, h_v, d_k, d_k)
    if v == DIAG_GATE:
        return (n_slots, h_v, d_k)
    return (n_slots, h_v)


def _check(t, name, dtype=None, ndim=None):
    if t is None:
        return
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")


def _build_desc(k, v, g, beta, seg_offsets, variant, seam_w, T_pool, S_pool, slot_of_seg, workspace,
                status, flags):
    _check(k, "k", ndim=3)
    _check(v, "v", dtype=k.dtype, ndim=3)
    _check(g, "g", dtype=torch.float32)
    _check(beta, "beta", dtype=torch.float32)
    _check(T_pool, "T_pool", dtype=torch.float32)
    _check(S_pool, "S_pool", dtype=torch.float32, ndim=4)
    off = np.ascontiguousarray(np.asarray(seg_offsets, dtype=np.int64))
    slots = None if slot_of_seg is None else np.ascontiguousarray(np.asarray(slot_of_seg, dtype=np.int32))
    d = BuildDesc()
    d.n_tokens, d.h_k, d.d_k = k.shape[0], k.shape[1], k.shape[2]
    d.h_v, d.d_v = v.shape[1], v.shape[2]
    d.n_seg = len(off) - 1
    d.seam_w = int(seam_w)
    d.variant = VARIANT[variant]
    d.in_dtype = _in_dtype(k)
    d.flags = int(flags)
    d.k, d.v, d.g, d.beta = _ptr(k), _ptr(v), _ptr(g), _ptr(beta)
    d.seg_offsets = off.ctypes.data_as(P)
    d.slot_of_seg = None if slots is None else slots.ctypes.data_as(P)
    d.n_slots = S_pool.shape[0]
    d.T_pool, d.S_pool = _ptr(T_pool), _ptr(S_pool)
    d.workspace = _ptr(workspace)
    d.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    d.status = _ptr(status)
    return d, (off, slots)


def build_workspace_bytes(n_seg: int, h_k: int, h_v: int, d_k: int, d_v: int, variant: str = "gdn",
                          dtype=torch.bfloat16, seam_w: int = 0) -> int:
    d = BuildDesc()
    d.n_seg, d.h_k, d.h_v, d.d_k, d.d_v = n_seg, h_k, h_v, d_k, d_v
    d.variant = VARIANT[variant]
    d.in_dtype = IN_BF16 if dtype == torch.bfloat16 else IN_F32
    d.seam_w = seam_w
    return int(load().hypic_build_workspace_bytes(ctypes.byref(d)))


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A 256-byte aligned device buffer of at least `nbytes` bytes."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def segment_build(k, v, g, beta, seg_offsets, *, variant: str, seam_w: int, T_pool, S_pool,
                  slot_of_seg=None, workspace=None, status=None, flags: int = 0, stream=None):
    """hypic_segment_build on torch tensors.  k [N,h_k,d_k], v [N,h_v,d_v]
    (bf16 or fp32), g / beta fp32 as in hypic.h, seg_offsets host int64
    [n_seg+1].  Writes T_pool / S_pool slots in place."""
    lib = load()
    d, keep = _build_desc(k, v, g, beta, seg_offsets, variant, seam_w, T_pool, S_pool, slot_of_seg,
                          workspace, status, flags)
    if workspace is None:
        nb = int(lib.hypic_build_workspace_bytes(ctypes.byref(d)))
        workspace = alloc_workspace(nb, k.device)
        d.workspace = _ptr(workspace)
        d.workspace_bytes = workspace.numel()
    rc = lib.hypic_segment_build(ctypes.byref(d), _stream(stream))
    del keep
    if rc != OK:
        raise HypicError(rc, "hypic_segment_build")
    return workspace


def segment_forward(k, v, q, g, beta, seg_offsets, *, variant: str, seam_w: int, T_pool, S_pool, o_out,
                    slot_of_seg=None, workspace=None, status=None, flags: int = 0, stream=None):
    """hypic_segment_forward on torch tensors: segment_build's pairs plus
    o_out [N, h_v, d_v] fp32, the output of every body token from the
    zero-initial body state (seam-token rows are not written).  q [N, h_k,
    d_k] in k's dtype.  The workspace (allocated here when None) is
    hypic_forward_workspace_bytes: about 96 KiB per 64-token chunk and value
    head on the tensor-core path."""
    lib = load()
    _check(q, "q", dtype=k.dtype, ndim=3)
    _check(o_out, "o_out", dtype=torch.float32, ndim=3)
    d = ForwardDesc()
    b, keep = _build_desc(k, v, g, beta, seg_offsets, variant, seam_w, T_pool, S_pool, slot_of_seg,
                          workspace, status, flags)
    d.build = b
    d.q, d.o_out = _ptr(q), _ptr(o_out)
    if workspace is None:
        nb = int(lib.hypic_forward_workspace_bytes(ctypes.byref(d)))
        workspace = alloc_workspace(nb, k.device)
        d.build.workspace = _ptr(workspace)
        d.build.workspace_bytes = workspace.numel()
    rc = lib.hypic_segment_forward(ctypes.byref(d), _stream(stream))
    del keep
    if rc != OK:
        raise HypicError(rc, "hypic_segment_forward")
    return workspace


def _host_ptr(t, like, name):
    """Address of a host tensor shaped and typed like its device twin."""
    if t is None:
        if like is not None:
            raise ValueError(f"{name}: host array missing")
        return None
    if t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: contiguous host tensor expected")
    if like is None or t.dtype != like.dtype or t.shape != like.shape:
        raise ValueError(f"{name}: must match its device buffer in shape and dtype")
    return ctypes.c_void_p(t.data_ptr())


def segment_build_host(k_host, v_host, g_host, beta_host, seg_offsets, *, variant: str, seam_w: int, k, v, g, beta,
                       T_pool, S_pool, T_host, S_host, n_chunks: int = 8, slot_of_seg=None, workspace=None,
                       status=None, flags: int = 0, stream=None):
    """hypic_segment_build_host on torch tensors: the build from host inputs
    (k_host, v_host, g_host, beta_host, page-locked for overlap) to host
    pools (T_host, S_host), with k, v, g, beta, T_pool, S_pool the device
    buffers of the same shapes used as staging.  Segments go in n_chunks
    groups whose input copies, builds and output copies overlap.  The host
    pools are complete once `stream` is synchronised."""
    lib = load()
    b, keep = _build_desc(k, v, g, beta, seg_offsets, variant, seam_w, T_pool, S_pool, slot_of_seg,
                          workspace, status, flags)
    if workspace is None:
        nb = int(lib.hypic_build_workspace_bytes(ctypes.byref(b)))
        workspace = alloc_workspace(nb, k.device)
        b.workspace = _ptr(workspace)
        b.workspace_bytes = workspace.numel()
    d = HostBuildDesc()
    d.build = b
    d.host_k, d.host_v = _host_ptr(k_host, k, "k_host"), _host_ptr(v_host, v, "v_host")
    d.host_g, d.host_beta = _host_ptr(g_host, g, "g_host"), _host_ptr(beta_host, beta, "beta_host")
    d.host_T, d.host_S = _host_ptr(T_host, T_pool, "T_host"), _host_ptr(S_host, S_pool, "S_host")
    d.n_chunks = int(n_chunks)
    rc = lib.hypic_segment_build_host(ctypes.byref(d), _stream(stream))
    del keep
    if rc != OK:
        raise HypicError(rc, "hypic_segment_build_host")
    return workspace


NOALLOC_MAX_PAIRS = 32766  # HYPIC_NOALLOC_MAX_PAIRS


def segment_build_noalloc(k, v, g, beta, seg_offsets, *, variant: str, seam_w: int, T_pool, S_pool,
                          slot_of_seg=None, status=None, flags: int = 0, stream=None):
    """hypic_segment_build_noalloc on torch tensors: the same build with its
    plan in the library's fixed device scratch (no workspace, no allocation).
    At most NOALLOC_MAX_PAIRS (segment, value head) pairs; calls that overlap
    on the GPU race on the shared scratch."""
    lib = load()
    d, keep = _build_desc(k, v, g, beta, seg_offsets, variant, seam_w, T_pool, S_pool, slot_of_seg,
                          None, status, flags)
    rc = lib.hypic_segment_build_noalloc(ctypes.byref(d), _stream(stream))
    del keep
    if rc != OK:
        raise HypicError(rc, "hypic_segment_build_noalloc")


def _compose_desc(slot, T_pool, S_pool, seam_k, seam_v, seam_q, seam_g, seam_beta, variant, S_out, seam_out,
                  S_init, h_k, status, flags, span=None):
    _check(slot, "slot", dtype=torch.int32, ndim=2)
    _check(S_out, "S_out", dtype=torch.float32, ndim=4)
    for name, t in (("seam_k", seam_k), ("seam_v", seam_v), ("seam_q", seam_q)):
        _check(t, name, ndim=5)
    d = ComposeDesc()
    d.n_layers, d.n_seg = slot.shape
    _, d.h_v, d.d_k, d.d_v = S_out.shape
    w = 0 if seam_k is None else seam_k.shape[2]
    d.seam_w = w
    d.h_k = seam_k.shape[3] if seam_k is not None else (h_k if h_k is not None else d.h_v)
    d.variant = VARIANT[variant]
    d.in_dtype = _in_dtype(seam_k) if seam_k is not None else IN_BF16
    d.flags = int(flags)
    at = lambda t: _ptr(t)  # whole arrays
    if span is not None:
        # segments [a, b) of the per-layer arrays, composed in place: the
        # pointers advance by a segments, the layer stride stays n_seg
        a, b = int(span[0]), int(span[1])
        if not 0 <= a <= b <= d.n_seg:
            raise ValueError(f"span {span} outside 0..{d.n_seg}")
        d.seg_stride, d.n_seg = d.n_seg, b - a

        def at(t):
            if t is None or t.dim() < 2 or t.shape[1] == 0 or a == t.shape[1]:
                return _ptr(t)
            return ctypes.c_void_p(t[:, a].data_ptr())
    d.slot = at(slot)
    d.n_slots = T_pool.shape[0]
    d.T_pool, d.S_pool = _ptr(T_pool), _ptr(S_pool)
    d.seam_k, d.seam_v, d.seam_q = at(seam_k), at(seam_v), at(seam_q)
    d.seam_g = _ptr(seam_g) if (seam_g is not None and seam_g.dim() == 2) else at(seam_g)  # scalar decay: per layer
    d.seam_beta = at(seam_beta)
    d.S_init, d.S_out, d.seam_out = _ptr(S_init), _ptr(S_out), at(seam_out)
    d.status = _ptr(status)
    return d


def compose(slot, T_pool, S_pool, seam_k, seam_v, seam_q, seam_g, seam_beta, *, variant: str,
            S_out, seam_out=None, S_init=None, h_k=None, d_k=None, d_v=None, status=None,
            flags: int = 0, stream=None, span=None):
    """hypic_compose on torch tensors.  slot int32 [L, n_seg] (device);
    seam arrays [L, n_seg, w, heads, d]; S_out [L, h_v, d_k, d_v].
    span=(a, b) composes segments a .. b-1 of those arrays only, in place
    (seam outputs of the other segments untouched).  With
    flags=FLAG_TRANSITION_ONLY, S_pool may be None and S_init None stands
    for the identity."""
    lib = load()
    d = _compose_desc(slot, T_pool, S_pool, seam_k, seam_v, seam_q, seam_g, seam_beta, variant, S_out, seam_out,
                      S_init, h_k, status, flags, span)
    nb = int(lib.hypic_compose_workspace_bytes(ctypes.byref(d)))
    ws = alloc_workspace(nb, S_out.device) if nb else None
    d.workspace = _ptr(ws)
    d.workspace_bytes = 0 if ws is None else ws.numel()
    rc = lib.hypic_compose(ctypes.byref(d), _stream(stream))
    if rc != OK:
        raise HypicError(rc, "hypic_compose")


def compose_host(seam_k_host, seam_v_host, seam_q_host, seam_g_host, seam_beta_host, slot, T_pool, S_pool, *,
                 variant: str, seam_k, seam_v, seam_q, seam_g, seam_beta, S_out, S_out_host, seam_out=None,
                 seam_out_host=None, S_init=None, S_init_host=None, n_chunks: int = 8, h_k=None, status=None,
                 flags: int = 0, stream=None):
    """hypic_compose_host on torch tensors: compose() from host seam tokens
    (page-locked for overlap) to host states and seam outputs, with the
    device seam arrays, S_init, S_out and seam_out used as staging; the
    layers go in n_chunks groups whose copies overlap the compose.  The host
    arrays are complete once `stream` is synchronised."""
    lib = load()
    d = HostComposeDesc()
    d.compose = _compose_desc(slot, T_pool, S_pool, seam_k, seam_v, seam_q, seam_g, seam_beta, variant, S_out,
                              seam_out, S_init, h_k, status, flags)
    d.host_seam_k = _host_ptr(seam_k_host, seam_k, "seam_k_host")
    d.host_seam_v = _host_ptr(seam_v_host, seam_v, "seam_v_host")
    d.host_seam_q = _host_ptr(seam_q_host, seam_q, "seam_q_host")
    d.host_seam_g = _host_ptr(seam_g_host, seam_g, "seam_g_host")
    d.host_seam_beta = _host_ptr(seam_beta_host, seam_beta, "seam_beta_host")
    d.host_S_init = _host_ptr(S_init_host, S_init, "S_init_host") if S_init_host is not None else None
    d.host_S_out = _host_ptr(S_out_host, S_out, "S_out_host")
    d.host_seam_out = _host_ptr(seam_out_host, seam_out, "seam_out_host")
    d.n_chunks = int(n_chunks)
    rc = lib.hypic_compose_host(ctypes.byref(d), _stream(stream))
    if rc != OK:
        raise HypicError(rc, "hypic_compose_host")


def compose_path(slot, T_pool, S_pool, seam_k, seam_v, seam_q, seam_g, seam_beta, *, variant: str, S_out,
                 seam_out=None, S_init=None, h_k=None, flags: int = 0) -> str:
    """hypic_compose_path: the kernel compose() runs for these arguments."""
    d = _compose_desc(slot, T_pool, S_pool, seam_k, seam_v, seam_q, seam_g, seam_beta, variant, S_out, seam_out,
                      S_init, h_k, None, flags)
    return _path_name(load().hypic_compose_path(ctypes.byref(d)), "hypic_compose_path")


def _path_name(rc, where):
    if rc < 0:
        raise HypicError(-rc, where)
    return PATHS[rc]


def build_path(k, v, g, beta, seg_offsets, *, variant: str, seam_w: int, T_pool, S_pool, slot_of_seg=None,
               flags: int = 0) -> str:
    """hypic_build_path: the kernel segment_build() runs for these arguments."""
    d, keep = _build_desc(k, v, g, beta, seg_offsets, variant, seam_w, T_pool, S_pool, slot_of_seg, None, None,
                          flags)
    rc = load().hypic_build_path(ctypes.byref(d))
    del keep
    return _path_name(rc, "hypic_build_path")


def forward_path(k, v, q, g, beta, seg_offsets, *, variant: str, seam_w: int, T_pool, S_pool, o_out,
                 flags: int = 0) -> str:
    """hypic_forward_path: the kernel of segment_forward()'s per-token outputs."""
    d = ForwardDesc()
    b, keep = _build_desc(k, v, g, beta, seg_offsets, variant, seam_w, T_pool, S_pool, None, None, None, flags)
    d.build = b
    d.q, d.o_out = _ptr(q), _ptr(o_out)
    rc = load().hypic_forward_path(ctypes.byref(d))
    del keep
    return _path_name(rc, "hypic_forward_path")


def _merge_desc(later, earlier, out, T_a, S_a, T_out, S_out, variant, T_b, S_b, status):
    if T_b is None:
        T_b, S_b = T_a, S_a
    for name, t in (("later", later), ("earlier", earlier), ("out", out)):
        _check(t, name, dtype=torch.int32, ndim=1)
    for name, t in (("S_a", S_a), ("S_b", S_b), ("S_out", S_out)):
        _check(t, name, dtype=torch.float32, ndim=4)
    d = MergeDesc()
    d.n_merge = later.shape[0]
    _, d.h_v, d.d_k, d.d_v = S_a.shape
    d.variant = VARIANT[variant]
    d.later, d.earlier, d.out = _ptr(later), _ptr(earlier), _ptr(out)
    d.n_slots_a, d.n_slots_b, d.n_slots_out = S_a.shape[0], S_b.shape[0], S_out.shape[0]
    d.T_a, d.S_a, d.T_b, d.S_b = _ptr(T_a), _ptr(S_a), _ptr(T_b), _ptr(S_b)
    d.T_out, d.S_out = _ptr(T_out), _ptr(S_out)
    d.status = _ptr(status)
    return d


def pair_merge(later, earlier, out, T_a, S_a, T_out, S_out, *, variant: str, T_b=None, S_b=None, status=None,
               stream=None):
    """hypic_pair_merge on torch tensors: for every merge m and head h,
    T_out[out[m], h] = T_a[later[m], h] T_b[earlier[m], h] and
    S_out[out[m], h] = T_a[later[m], h] S_b[earlier[m], h] + S_a[later[m], h].
    later / earlier / out int32 [n_merge] (device); pools as written by
    segment_build (T layout per variant, S [slots, h_v, d_k, d_v]); the pool
    of the earlier pairs defaults to that of the later ones."""
    d = _merge_desc(later, earlier, out, T_a, S_a, T_out, S_out, variant, T_b, S_b, status)
    rc = load().hypic_pair_merge(ctypes.byref(d), _stream(stream))
    if rc != OK:
        raise HypicError(rc, "hypic_pair_merge")


def merge_path(later, earlier, out, T_a, S_a, T_out, S_out, *, variant: str, T_b=None, S_b=None) -> str:
    """hypic_merge_path: the kernel pair_merge() runs for these arguments."""
    d = _merge_desc(later, earlier, out, T_a, S_a, T_out, S_out, variant, T_b, S_b, None)
    return _path_name(load().hypic_merge_path(ctypes.byref(d)), "hypic_merge_path")


def pair_rerotate(slot_in, slot_out, delta, T_in, S_in, T_out, S_out, *, variant: str, rot_dim: int,
                  layout: str = "interleaved", base: float = 10000.0, status=None, stream=None):
    """hypic_pair_rerotate on torch tensors: the pair in slot_in[m] of a
    segment moved by delta[m] positions, re-rotated into slot_out[m]:
    T_out = R T_in R^T, S_out = R S_in with R = R(delta[m]) the rotary
    rotation of the key channels (pairs per `layout`, the first rot_dim
    channels, theta_i = base^(-2i / rot_dim)).  slot_in / slot_out int32
    [n_items], delta int64 [n_items] (device); the output pool may be the
    input pool (in place)."""
    lib = load()
    for name, t in (("slot_in", slot_in), ("slot_out", slot_out)):
        _check(t, name, dtype=torch.int32, ndim=1)
    _check(delta, "delta", dtype=torch.int64, ndim=1)
    for name, t in (("S_in", S_in), ("S_out", S_out)):
        _check(t, name, dtype=torch.float32, ndim=4)
    d = RerotateDesc()
    d.n_items = slot_in.shape[0]
    _, d.h_v, d.d_k, d.d_v = S_in.shape
    d.variant = VARIANT[variant]
    d.rot_dim = int(rot_dim)
    d.layout = ROPE_LAYOUT[layout]
    d.base = float(base)
    d.slot_in, d.slot_out, d.delta = _ptr(slot_in), _ptr(slot_out), _ptr(delta)
    d.n_slots_in, d.n_slots_out = S_in.shape[0], S_out.shape[0]
    d.T_in, d.S_in, d.T_out, d.S_out = _ptr(T_in), _ptr(S_in), _ptr(T_out), _ptr(S_out)
    d.status = _ptr(status)
    rc = lib.hypic_pair_rerotate(ctypes.byref(d), _stream(stream))
    if rc != OK:
        raise HypicError(rc, "hypic_pair_rerotate")


def span_scan(T_span, S_span, S_start, *, S_init=None, status=None, stream=None):
    """hypic_span_scan on torch tensors: the start state of every span,
    S_start[0] = S_init (or 0), S_start[s] = T_span[s-1] S_start[s-1] +
    S_span[s-1].  T_span [n_spans, L, h_v, d_k, d_k], S_span / S_start
    [n_spans, L, h_v, d_k, d_v], S_init [L, h_v, d_k, d_v] (device, fp32)."""
    lib = load()
    _check(S_start, "S_start", dtype=torch.float32, ndim=5)
    d = SpanScanDesc()
    d.n_spans, d.n_layers, d.h_v, d.d_k, d.d_v = S_start.shape
    for name, t in (("T_span", T_span), ("S_span", S_span)):
        _check(t, name, dtype=torch.float32, ndim=5)
    d.T_span, d.S_span, d.S_init, d.S_start = _ptr(T_span), _ptr(S_span), _ptr(S_init), _ptr(S_start)
    ws = alloc_workspace(int(lib.hypic_span_scan_workspace_bytes(ctypes.byref(d))), S_start.device)
    d.workspace, d.workspace_bytes = _ptr(ws), ws.numel()
    d.status = _ptr(status)
    rc = lib.hypic_span_scan(ctypes.byref(d), _stream(stream))
    if rc != OK:
        raise HypicError(rc, "hypic_span_scan")


def span_bounds(n_seg: int, n_spans: int):
    """Segment boundaries of n_spans consecutive spans of about equal segment
    counts (every segment costs its seam window plus one pair)."""
    n_spans = max(1, min(int(n_spans), max(int(n_seg), 1)))
    return np.linspace(0, n_seg, n_spans + 1).round().astype(np.int32)


def compose_spans(slot, T_pool, S_pool, seam_k, seam_v, seam_q, seam_g, seam_beta, *, variant: str, S_out,
                  seam_out=None, S_init=None, n_spans: int = 2, bounds=None, h_k=None, status=None, flags: int = 0,
                  stream=None):
    """hypic_compose_spans on torch tensors: compose() computed by segment
    parallelism (nav.aitube.vip §2.3) with the chains split into n_spans
    consecutive spans of segments (or at `bounds`): the span pairs, their
    exclusive scan, then every span from its start state.  Same arguments
    and results as compose()."""
    lib = load()
    d = _compose_desc(slot, T_pool, S_pool, seam_k, seam_v, seam_q, seam_g, seam_beta, variant, S_out, seam_out,
                      S_init, h_k, status, flags)
    b = span_bounds(d.n_seg, n_spans) if bounds is None else np.ascontiguousarray(np.asarray(bounds, np.int32))
    ns = len(b) - 1
    ws = alloc_workspace(int(lib.hypic_compose_spans_workspace_bytes(ctypes.byref(d), ns)), S_out.device)
    d.workspace, d.workspace_bytes = _ptr(ws), ws.numel()
    rc = lib.hypic_compose_spans(ctypes.byref(d), ns, b.ctypes.data_as(P), _stream(stream))
    if rc != OK:
        raise HypicError(rc, "hypic_compose_spans")


def plan_lpt(costs, n_workers: int):
    """Host LPT packing: returns (order, worker_of_item, makespan)."""
    lib = load()
    c = np.ascontiguousarray(np.asarray(costs, dtype=np.int64))
    n = len(c)
    order = np.zeros(n, dtype=np.int32)
    worker = np.zeros(n, dtype=np.int32)
    mk = ctypes.c_int64(0)
    rc = lib.hypic_plan_lpt(c.ctypes.data_as(P), n, int(n_workers), order.ctypes.data_as(P),
                            worker.ctypes.data_as(P), ctypes.byref(mk))
    if rc != OK:
        raise HypicError(rc, "hypic_plan_lpt")
    return order, worker, int(mk.value)


def shard_lpt(costs, world_size: int):
    """Multi-GPU partition of independent units (cold segments to build, or
    (layer, head) chains to compose) over ranks by the same LPT rule the
    pages use to balance segments over scatter workers (nav.aitube.vip
    §2.3).  Returns one sorted index array per rank; every unit lands on
    exactly one rank and the units need no exchange while they run."""
    _, worker, _ = plan_lpt(costs, world_size)
    return [np.sort(np.nonzero(worker == r)[0]) for r in range(int(world_size))]
