"""Host-side checks that need no GPU: the C ABI library loads and exports
every entry point that include/hypic.h declares, the LPT planner is the
greedy longest-first rule (checked against brute force and Graham's bound),
and invalid descriptors are rejected before anything is launched."""
import ctypes
import itertools
import os
import re

import numpy as np
import pytest
import torch

import hybrid_linear_attention_chunkwise_gb300 as hy

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__ as g
    g.build()


def _declared():
    src = open(os.path.join(ROOT, "include", "hypic.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hypic_[a-z_0-9]+)\s*\(", src)))


def test_library_exports_every_declared_entry_point():
    lib = hy.load()
    names = _declared()
    assert "hypic_segment_build" in names and "hypic_compose" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in hypic.h but not exported"
    assert set(hy.SYMBOLS) <= set(names)


def test_status_strings_and_word_decoding():
    assert hy.status_string(0) == "ok"
    for c in range(1, 8):
        assert hy.status_string(c) != "unknown status"
    assert hy.status_from_word(0) == 0
    assert hy.status_from_word(hy.STATUS_TIMEOUT) == 5
    assert hy.status_from_word(hy.STATUS_BAD_SLOT) == 7
    assert hy.status_from_word(hy.STATUS_NONFINITE) == 6


def _lpt_reference(costs, m):
    order = sorted(range(len(costs)), key=lambda i: (-costs[i], i))
    loads = [0] * m
    for i in order:
        w = min(range(m), key=lambda j: (loads[j], j))
        loads[w] += costs[i]
    return order, max(loads) if costs else 0


def _optimum(costs, m):
    best = None
    for assign in itertools.product(range(m), repeat=len(costs)):
        loads = [0] * m
        for c, w in zip(costs, assign):
            loads[w] += c
        mk = max(loads)
        best = mk if best is None else min(best, mk)
    return best


def test_lpt_matches_rule_and_graham_bound():
    rng = np.random.default_rng(3)
    for trial in range(60):
        n = int(rng.integers(1, 9))
        m = int(rng.integers(1, 4))
        costs = [int(x) for x in rng.integers(1, 20, n)]
        if trial % 5 == 0:
            costs = [7] * n  # all ties: index order
        order, worker, mk = hy.plan_lpt(costs, m)
        ref_order, ref_mk = _lpt_reference(costs, m)
        assert list(order) == ref_order
        assert mk == ref_mk
        loads = np.zeros(m, dtype=np.int64)
        for i, w in enumerate(worker):
            loads[w] += costs[i]
        assert loads.max() == mk
        opt = _optimum(costs, m)
        assert mk <= (4.0 / 3.0 - 1.0 / (3 * m)) * opt + 1e-9


def test_lpt_beats_round_robin_on_uneven_mix():
    # segments of 256..8192 tokens as in the cold uneven build
    rng = np.random.default_rng(0)
    costs = rng.choice([256, 1024, 4096, 8192], size=256, p=[0.4, 0.3, 0.2, 0.1])
    _, _, mk = hy.plan_lpt(costs, 8)
    rr = max(costs[w::8].sum() for w in range(8))
    assert mk <= rr
    assert mk <= costs.sum() / 8 + costs.max()


def _fake_build_desc(**over):
    d = hy.BuildDesc()
    d.n_tokens, d.n_seg, d.h_k, d.h_v, d.d_k, d.d_v, d.seam_w = 8, 2, 1, 2, 16, 16, 0
    d.variant, d.in_dtype = hy.GDN, hy.IN_F32
    fake = ctypes.c_void_p(1 << 20)
    d.k = d.v = d.g = d.beta = d.T_pool = d.S_pool = fake
    d.n_slots = 2
    d.workspace = ctypes.c_void_p(1 << 24)
    d.workspace_bytes = 1 << 20
    for k, v in over.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("case,offs,expect", [
    ("non-monotone offsets", [0, 6, 4, 8], 1),
    ("offsets not ending at n_tokens", [0, 3, 7], 1),
    ("offsets not starting at 0", [1, 3, 8], 1),
])
def test_build_rejects_bad_offsets(case, offs, expect):
    off = np.asarray(offs, dtype=np.int64)
    d = _fake_build_desc(n_seg=len(offs) - 1, seg_offsets=off.ctypes.data_as(ctypes.c_void_p), n_slots=8)
    assert hy.load().hypic_segment_build(ctypes.byref(d), None) == expect, case


def test_build_rejects_bad_descriptors():
    lib = hy.load()
    off = np.asarray([0, 3, 8], dtype=np.int64)
    po = off.ctypes.data_as(ctypes.c_void_p)
    cases = [
        (dict(h_v=3, h_k=2), 1),                          # h_v not a multiple of h_k
        (dict(d_k=129), 2),                               # head size > 128
        (dict(d_k=0), 1),
        (dict(variant=9), 1),
        (dict(k=None), 1),
        (dict(beta=None), 1),                              # delta variant needs beta
        (dict(g=None), 1),                                 # GDN needs log-gates
        (dict(k=ctypes.c_void_p((1 << 20) + 2)), 1),       # misaligned fp32 input
        (dict(workspace_bytes=16), 3),
        (dict(workspace=None), 3),
        (dict(n_slots=1), 1),                              # slot 1 out of range
        (dict(seam_w=-1), 1),
    ]
    for over, want in cases:
        d = _fake_build_desc(seg_offsets=po, **over)
        assert lib.hypic_segment_build(ctypes.byref(d), None) == want, over
    dup = np.asarray([1, 1], dtype=np.int32)
    d = _fake_build_desc(seg_offsets=po, slot_of_seg=dup.ctypes.data_as(ctypes.c_void_p))
    assert lib.hypic_segment_build(ctypes.byref(d), None) == 1


def test_forward_rejects_bad_descriptors():
    lib = hy.load()
    off = np.asarray([0, 3, 8], dtype=np.int64)
    po = off.ctypes.data_as(ctypes.c_void_p)
    fake = ctypes.c_void_p(1 << 20)
    for over, want in [(dict(q=None), 1), (dict(o_out=None), 1), (dict(o_out=ctypes.c_void_p((1 << 20) + 2)), 1),
                       (dict(build=dict(d_k=129)), 2), (dict(build=dict(k=None)), 1),
                       (dict(build=dict(workspace=None)), 3)]:
        d = hy.ForwardDesc()
        d.build = _fake_build_desc(seg_offsets=po, **over.get("build", {}))
        d.q = over.get("q", fake)
        d.o_out = over.get("o_out", fake)
        assert lib.hypic_segment_forward(ctypes.byref(d), None) == want, over


def test_build_host_rejects_bad_descriptors():
    """hypic_segment_build_host checks everything before the first CUDA call:
    the build's own checks, the chunk count, the host arrays (present exactly
    where their device twins are), then the workspace."""
    lib = hy.load()
    off = np.asarray([0, 3, 8], dtype=np.int64)
    po = off.ctypes.data_as(ctypes.c_void_p)
    host = ctypes.c_void_p(1 << 21)
    for over, want in [(dict(n_chunks=0), 1), (dict(host_T=None), 1), (dict(host_S=None), 1),
                       (dict(host_k=None), 1), (dict(host_v=None), 1), (dict(host_g=None), 1),
                       (dict(host_beta=None), 1), (dict(build=dict(beta=None)), 1),
                       (dict(build=dict(d_k=129)), 2), (dict(build=dict(workspace=None)), 3),
                       (dict(build=dict(workspace_bytes=16)), 3)]:
        d = hy.HostBuildDesc()
        d.build = _fake_build_desc(seg_offsets=po, **over.get("build", {}))
        for name in ("host_k", "host_v", "host_g", "host_beta", "host_T", "host_S"):
            setattr(d, name, over.get(name, host))
        d.n_chunks = over.get("n_chunks", 4)
        assert lib.hypic_segment_build_host(ctypes.byref(d), None) == want, over
    d = hy.HostBuildDesc()  # a gate-free variant given a host gate array
    d.build = _fake_build_desc(seg_offsets=po, variant=hy.UNGATED, g=None, beta=None)
    d.host_k = d.host_v = d.host_T = d.host_S = d.host_g = host
    d.n_chunks = 2
    assert lib.hypic_segment_build_host(ctypes.byref(d), None) == 1


def test_compose_rejects_bad_descriptors():
    lib = hy.load()
    fake = ctypes.c_void_p(1 << 20)

    def desc(**over):
        d = hy.ComposeDesc()
        d.n_layers, d.n_seg, d.h_k, d.h_v, d.d_k, d.d_v, d.seam_w = 1, 2, 1, 1, 16, 16, 2
        d.variant, d.in_dtype = hy.GDN, hy.IN_F32
        d.slot = d.T_pool = d.S_pool = d.seam_k = d.seam_v = d.seam_q = d.seam_g = d.seam_beta = fake
        d.S_out = d.seam_out = fake
        d.n_slots = 2
        for k, v in over.items():
            setattr(d, k, v)
        return d
    for over, want in [(dict(S_out=None), 1), (dict(seam_beta=None), 1), (dict(seam_g=None), 1),
                       (dict(d_v=200), 2), (dict(slot=None), 1), (dict(seam_out=None), 1),
                       (dict(seam_k=ctypes.c_void_p((1 << 20) + 1)), 1)]:
        assert lib.hypic_compose(ctypes.byref(desc(**over)), None) == want, over


def test_merge_rejects_bad_descriptors():
    lib = hy.load()
    fake = ctypes.c_void_p(1 << 20)

    def desc(**over):
        d = hy.MergeDesc()
        d.n_merge, d.h_v, d.d_k, d.d_v, d.variant = 2, 4, 128, 128, hy.GDN
        d.later = d.earlier = d.out = d.T_a = d.S_a = d.T_b = d.S_b = d.T_out = d.S_out = fake
        d.n_slots_a, d.n_slots_b, d.n_slots_out = 4, 4, 2
        for k, v in over.items():
            setattr(d, k, v)
        return d
    for over, want in [(dict(n_merge=-1), 1), (dict(later=None), 1), (dict(out=None), 1),
                       (dict(T_out=None), 1), (dict(S_a=None), 1), (dict(T_b=None), 1), (dict(d_k=200), 2), (dict(variant=9), 1),
                       (dict(h_v=0), 1), (dict(n_slots_a=-1), 1), (dict(n_slots_b=-1), 1),
                       (dict(earlier=ctypes.c_void_p((1 << 20) + 2)), 1),
                       (dict(S_out=ctypes.c_void_p((1 << 20) + 1)), 1)]:
        assert lib.hypic_pair_merge(ctypes.byref(desc(**over)), None) == want, over
    # nothing to do: accepted without touching any pointer
    assert lib.hypic_pair_merge(ctypes.byref(desc(n_merge=0, later=None, T_a=None)), None) == 0


def test_rerotate_rejects_bad_descriptors():
    lib = hy.load()
    fake = ctypes.c_void_p(1 << 20)

    def desc(**over):
        d = hy.RerotateDesc()
        d.n_items, d.h_v, d.d_k, d.d_v, d.variant = 2, 4, 128, 128, hy.GDN
        d.rot_dim, d.layout, d.base = 128, 0, 10000.0
        d.slot_in = d.slot_out = d.delta = d.T_in = d.S_in = d.T_out = d.S_out = fake
        d.n_slots_in, d.n_slots_out = 4, 4
        for k, v in over.items():
            setattr(d, k, v)
        return d
    for over, want in [(dict(n_items=-1), 1), (dict(slot_in=None), 1), (dict(delta=None), 1),
                       (dict(T_out=None), 1), (dict(S_in=None), 1), (dict(variant=9), 1), (dict(h_v=0), 1),
                       (dict(rot_dim=0), 1), (dict(rot_dim=7), 1), (dict(rot_dim=130), 1), (dict(layout=2), 1),
                       (dict(layout=1, rot_dim=12), 1), (dict(base=0.0), 1), (dict(base=float("nan")), 1),
                       (dict(n_slots_in=-1), 1), (dict(d_k=200, rot_dim=128), 2), (dict(d_v=126), 2),
                       (dict(variant=hy.VARIANT["channel"]), 2), (dict(variant=hy.VARIANT["diag"]), 2),
                       (dict(delta=ctypes.c_void_p((1 << 20) + 4)), 1),
                       (dict(S_out=ctypes.c_void_p((1 << 20) + 4)), 1)]:
        assert lib.hypic_pair_rerotate(ctypes.byref(desc(**over)), None) == want, over
    assert lib.hypic_pair_rerotate(ctypes.byref(desc(n_items=0, slot_in=None, T_in=None)), None) == 0


def test_binding_refuses_host_tensors():
    with pytest.raises(ValueError):
        hy._ptr(torch.zeros(4))


# ---- which kernel a call runs, and refusing the CUDA-core fallbacks

def test_build_path_query_follows_dtype_shape_and_alignment():
    """hypic_build_path names the kernel the build dispatch picks: the
    tensor-core kernels for bf16 128-wide heads with 16-byte aligned inputs,
    the fp32 token recurrence otherwise (and for a call with no tokens)."""
    lib = hy.load()
    off = np.asarray([0, 3, 8], dtype=np.int64)
    po = off.ctypes.data_as(ctypes.c_void_p)
    tc = dict(in_dtype=hy.IN_BF16, d_k=128, d_v=128)
    cases = [
        (dict(variant=hy.GDN, **tc), "tc_chunkwise"),
        (dict(variant=hy.DELTANET, **tc), "tc_chunkwise"),
        (dict(variant=hy.CHANNEL_DELTA, **tc), "tc_channel"),
        (dict(variant=hy.SCALAR_DECAY, **tc), "tc_fast"),
        (dict(variant=hy.UNGATED, **tc), "tc_fast"),
        (dict(variant=hy.DIAG_GATE, **tc), "tc_fast"),
        (dict(variant=hy.GDN, k=ctypes.c_void_p((1 << 20) + 2), **tc), "f32_token"),   # k not 16-byte aligned
        (dict(variant=hy.GDN, v=ctypes.c_void_p((1 << 20) + 8), **tc), "f32_token"),
        (dict(variant=hy.GDN, in_dtype=hy.IN_F32, d_k=128, d_v=128), "f32_token"),
        (dict(variant=hy.GDN, in_dtype=hy.IN_BF16, d_k=64, d_v=128), "f32_token"),
        (dict(variant=hy.GDN, n_tokens=0, seg_offsets=np.zeros(3, np.int64).ctypes.data_as(ctypes.c_void_p),
              **tc), "f32_token"),
        (dict(variant=hy.GDN, n_seg=0, **tc), "none"),
    ]
    for over, want in cases:
        over.setdefault("seg_offsets", po)
        if over.get("n_seg") == 0:
            over["seg_offsets"] = np.zeros(1, np.int64).ctypes.data_as(ctypes.c_void_p)
            over["n_tokens"] = 0
        d = _fake_build_desc(**over)
        assert hy.PATHS[lib.hypic_build_path(ctypes.byref(d))] == want, over
    assert lib.hypic_build_path(ctypes.byref(_fake_build_desc(seg_offsets=po, d_k=129))) == -2
    assert lib.hypic_build_path(ctypes.byref(_fake_build_desc(seg_offsets=po, h_v=3, h_k=2))) == -1


def test_compose_and_merge_path_queries():
    lib = hy.load()
    fake = ctypes.c_void_p(1 << 20)

    def cdesc(**over):
        d = hy.ComposeDesc()
        d.n_layers, d.n_seg, d.h_k, d.h_v, d.d_k, d.d_v, d.seam_w = 1, 2, 2, 4, 128, 128, 8
        d.variant, d.in_dtype = hy.GDN, hy.IN_BF16
        d.slot = d.T_pool = d.S_pool = d.seam_k = d.seam_v = d.seam_q = d.seam_g = d.seam_beta = fake
        d.S_out = d.seam_out = fake
        d.n_slots = 2
        for k, v in over.items():
            setattr(d, k, v)
        return d
    assert hy.PATHS[lib.hypic_compose_path(ctypes.byref(cdesc()))] == "tc_compose"
    assert hy.PATHS[lib.hypic_compose_path(ctypes.byref(cdesc(variant=hy.CHANNEL_DELTA)))] == "tc_compose"
    for over in (dict(h_v=2, h_k=2), dict(in_dtype=hy.IN_F32), dict(d_k=64),
                 dict(seam_k=ctypes.c_void_p((1 << 20) + 8)), dict(variant=hy.SCALAR_DECAY, seam_beta=None)):
        assert hy.PATHS[lib.hypic_compose_path(ctypes.byref(cdesc(**over)))] == "f32_compose", over
    assert hy.PATHS[lib.hypic_compose_path(ctypes.byref(cdesc(n_layers=0)))] == "none"
    assert lib.hypic_compose_path(ctypes.byref(cdesc(S_out=None))) == -1

    def mdesc(**over):
        d = hy.MergeDesc()
        d.n_merge, d.h_v, d.d_k, d.d_v, d.variant = 2, 4, 128, 128, hy.GDN
        d.later = d.earlier = d.out = d.T_a = d.S_a = d.T_b = d.S_b = d.T_out = d.S_out = fake
        d.n_slots_a, d.n_slots_b, d.n_slots_out = 4, 4, 2
        for k, v in over.items():
            setattr(d, k, v)
        return d
    assert hy.PATHS[lib.hypic_merge_path(ctypes.byref(mdesc()))] == "tc_merge"
    assert hy.PATHS[lib.hypic_merge_path(ctypes.byref(mdesc(d_k=64)))] == "f32_merge"
    assert hy.PATHS[lib.hypic_merge_path(ctypes.byref(mdesc(variant=hy.SCALAR_DECAY)))] == "f32_merge"
    assert hy.PATHS[lib.hypic_merge_path(ctypes.byref(mdesc(T_a=ctypes.c_void_p((1 << 20) + 4))))] == "f32_merge"
    assert hy.PATHS[lib.hypic_merge_path(ctypes.byref(mdesc(n_merge=0)))] == "none"


def test_require_tensor_cores_refuses_fallbacks_before_any_cuda_call():
    """With HYPIC_FLAG_REQUIRE_TENSOR_CORES a call that would fall back to an
    fp32 CUDA-core kernel returns HYPIC_ERR_UNSUPPORTED and launches nothing
    (so these fake pointers are never touched, with or without a GPU)."""
    lib = hy.load()
    off = np.asarray([0, 3, 8], dtype=np.int64)
    po = off.ctypes.data_as(ctypes.c_void_p)
    req = hy.FLAG_REQUIRE_TENSOR_CORES
    for over in (dict(in_dtype=hy.IN_BF16, d_k=128, d_v=128, k=ctypes.c_void_p((1 << 20) + 2)),
                 dict(in_dtype=hy.IN_F32, d_k=128, d_v=128), dict(in_dtype=hy.IN_BF16, d_k=32, d_v=32)):
        d = _fake_build_desc(seg_offsets=po, flags=req, **over)
        assert lib.hypic_segment_build(ctypes.byref(d), None) == 2, over
        assert lib.hypic_segment_build_noalloc(ctypes.byref(d), None) == 2, over
    # a q off the 16-byte grid sends the forward's outputs to the CUDA
    # cores: refused under the flag
    d = hy.ForwardDesc()
    d.build = _fake_build_desc(seg_offsets=po, flags=req, in_dtype=hy.IN_BF16, d_k=128, d_v=128)
    d.q = ctypes.c_void_p((1 << 20) + 2)
    d.o_out = ctypes.c_void_p(1 << 20)
    assert hy.PATHS[lib.hypic_forward_path(ctypes.byref(d))] == "f32_token"
    assert lib.hypic_segment_forward(ctypes.byref(d), None) == 2
    d.q = ctypes.c_void_p(1 << 20)
    assert hy.PATHS[lib.hypic_forward_path(ctypes.byref(d))] == "tc_forward"
    fake = ctypes.c_void_p(1 << 20)
    c = hy.ComposeDesc()
    c.n_layers, c.n_seg, c.h_k, c.h_v, c.d_k, c.d_v, c.seam_w = 1, 2, 2, 2, 128, 128, 8
    c.variant, c.in_dtype, c.flags = hy.GDN, hy.IN_BF16, req
    c.slot = c.T_pool = c.S_pool = c.seam_k = c.seam_v = c.seam_q = c.seam_g = c.seam_beta = fake
    c.S_out = c.seam_out = fake
    c.n_slots = 2
    assert lib.hypic_compose(ctypes.byref(c), None) == 2  # h_v = 2: not a multiple of 4
    # unknown flag bits are refused
    d = _fake_build_desc(seg_offsets=po, flags=64)
    assert lib.hypic_segment_build(ctypes.byref(d), None) == 1
    c.flags = hy.FLAG_ROUND_ROBIN   # a build-only flag
    assert lib.hypic_compose(ctypes.byref(c), None) == 1


def test_build_workspace_is_one_item_per_pair():
    """64-byte plan header plus 32 bytes per (segment, value head), rounded
    up to 256 bytes; the allocation-free entry point's limit fills its 1 MiB
    array exactly."""
    for n_seg, h_v in ((1, 1), (64, 32), (7, 3)):
        nb = hy.build_workspace_bytes(n_seg, 1, h_v, 128, 128)
        assert nb == (64 + 32 * n_seg * h_v + 255) // 256 * 256
    assert 64 + 32 * hy.NOALLOC_MAX_PAIRS == 1 << 20


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake device pointers: only where no GPU can be reached")
def test_noalloc_and_workspace_build_agree_on_a_no_token_call():
    """A GDN descriptor with no tokens and no log-gate array is valid for
    hypic_segment_build (the gates are never read); the allocation-free entry
    point runs the same checks, so it must not refuse it either.  Without a
    GPU both get as far as their first CUDA call and fail there alike."""
    lib = hy.load()
    off = np.zeros(3, np.int64)
    d = _fake_build_desc(n_tokens=0, seg_offsets=off.ctypes.data_as(ctypes.c_void_p), g=None, beta=None, k=None,
                         v=None)
    a = lib.hypic_segment_build(ctypes.byref(d), None)
    b = lib.hypic_segment_build_noalloc(ctypes.byref(d), None)
    assert a == b == 4, (a, b)  # HYPIC_ERR_CUDA: validation passed on both


def test_span_entry_points_reject_bad_descriptors():
    """Transition-only compose, compose over spans and the span scan check
    their arguments before any CUDA call."""
    lib = hy.load()
    fake = ctypes.c_void_p(1 << 20)

    def cdesc(**over):
        d = hy.ComposeDesc()
        d.n_layers, d.n_seg, d.h_k, d.h_v, d.d_k, d.d_v, d.seam_w = 1, 4, 1, 1, 16, 16, 2
        d.variant, d.in_dtype = hy.GDN, hy.IN_F32
        d.slot = d.T_pool = d.S_pool = d.seam_k = d.seam_v = d.seam_q = d.seam_g = d.seam_beta = fake
        d.S_out = d.seam_out = fake
        d.n_slots = 4
        for k, v in over.items():
            setattr(d, k, v)
        return d
    T = hy.FLAG_TRANSITION_ONLY
    for over, want in [(dict(flags=T, d_v=8), 1),             # the state of a transition is d_k x d_k
                       (dict(seg_stride=3), 1),                # a stride below n_seg
                       (dict(flags=16), 1)]:                   # unknown flag
        assert lib.hypic_compose(ctypes.byref(cdesc(**over)), None) == want, over
    bnd = lambda *b: np.asarray(b, dtype=np.int32)
    for b, want in [(bnd(0, 2, 3), 1), (bnd(1, 2, 4), 1), (bnd(0, 3, 2, 4), 1)]:
        d = cdesc()
        d.workspace, d.workspace_bytes = ctypes.c_void_p(1 << 24), 1 << 30
        assert lib.hypic_compose_spans(ctypes.byref(d), len(b) - 1, b.ctypes.data_as(ctypes.c_void_p), None) == want
    d = cdesc(flags=T)
    b = bnd(0, 2, 4)
    assert lib.hypic_compose_spans(ctypes.byref(d), 2, b.ctypes.data_as(ctypes.c_void_p), None) == 1
    d = cdesc()
    d.workspace, d.workspace_bytes = ctypes.c_void_p(1 << 24), 16
    assert lib.hypic_compose_spans(ctypes.byref(d), 2, b.ctypes.data_as(ctypes.c_void_p), None) == 3
    s = hy.SpanScanDesc()
    s.n_layers, s.n_spans, s.h_v, s.d_k, s.d_v = 2, 3, 4, 128, 128
    s.T_span = s.S_span = s.S_start = fake
    assert lib.hypic_span_scan(ctypes.byref(s), None) == 3          # no workspace
    s.workspace, s.workspace_bytes = ctypes.c_void_p(1 << 24), 1 << 20
    s.S_start = None
    assert lib.hypic_span_scan(ctypes.byref(s), None) == 1
    s.S_start, s.d_k = fake, 200
    assert lib.hypic_span_scan(ctypes.byref(s), None) == 2
    assert lib.hypic_span_scan_workspace_bytes(ctypes.byref(s)) == 256


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake device pointers: only where no GPU can be reached")
def test_build_accepts_skipped_segments_and_rejects_duplicates():
    """HYPIC_SLOT_SKIP leaves a segment out; the other slots must stay
    distinct and in range (checked before any CUDA call)."""
    lib = hy.load()
    off = np.asarray([0, 3, 8], dtype=np.int64)
    po = off.ctypes.data_as(ctypes.c_void_p)
    for slots, want_invalid in (([-1, 1], False), ([-1, -1], False), ([1, 1], True), ([-2, 0], True), ([0, 2], True)):
        sl = np.asarray(slots, dtype=np.int32)
        d = _fake_build_desc(seg_offsets=po, slot_of_seg=sl.ctypes.data_as(ctypes.c_void_p))
        rc = lib.hypic_segment_build(ctypes.byref(d), None)
        assert (rc == 1) == want_invalid, (slots, rc)


def test_compose_host_rejects_bad_descriptors():
    """hypic_compose_host checks the compose descriptor, the chunk count and
    the host arrays (present exactly where their device twins are) before
    its first CUDA call."""
    lib = hy.load()
    fake = ctypes.c_void_p(1 << 20)
    host = ctypes.c_void_p(1 << 21)

    def desc(**over):
        d = hy.HostComposeDesc()
        c = d.compose
        c.n_layers, c.n_seg, c.h_k, c.h_v, c.d_k, c.d_v, c.seam_w = 2, 3, 1, 1, 16, 16, 2
        c.variant, c.in_dtype = hy.GDN, hy.IN_F32
        c.slot = c.T_pool = c.S_pool = c.seam_k = c.seam_v = c.seam_q = c.seam_g = c.seam_beta = fake
        c.S_out = c.seam_out = fake
        c.n_slots = 6
        for n in ("host_seam_k", "host_seam_v", "host_seam_q", "host_seam_g", "host_seam_beta", "host_S_out",
                  "host_seam_out"):
            setattr(d, n, host)
        d.n_chunks = 2
        for k, v in over.items():
            if k.startswith("c_"):
                setattr(d.compose, k[2:], v)
            else:
                setattr(d, k, v)
        return d
    for over, want in [(dict(n_chunks=0), 1), (dict(host_S_out=None), 1), (dict(host_seam_q=None), 1),
                       (dict(host_seam_out=None), 1), (dict(host_seam_g=None), 1), (dict(host_seam_beta=None), 1),
                       (dict(host_S_init=host), 1),            # a host S_init needs its device staging
                       (dict(c_S_out=None), 1), (dict(c_d_v=200), 2),
                       (dict(c_flags=hy.FLAG_TRANSITION_ONLY), 1)]:
        assert lib.hypic_compose_host(ctypes.byref(desc(**over)), None) == want, over
