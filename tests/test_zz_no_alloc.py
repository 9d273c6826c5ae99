"""hypic_segment_build_noalloc: the build with its work plan in the library's
fixed device scratch, for callers that cannot allocate device memory.  Two
calls in a row through the C ABI, on different inputs, must each equal the
workspace entry point's result bit for bit (the second call only can if the
first left no stale plan or ticket behind); at exactly the pair limit the
plan (64-byte header, 32 bytes per (segment, value head)) fills the 1 MiB
scratch to its last byte; a larger problem is refused before any CUDA call;
a call that the workspace entry point accepts is accepted too.

Collected last on purpose (file name), so it also runs after every other
test in the same process."""
import ctypes

import numpy as np
import pytest
import torch

import hybrid_linear_attention_chunkwise_gb300 as hy
import synth_inputs as si
from gpu_common import new_pools

DEV = "cuda"


@pytest.fixture(scope="module")
def _lib():
    import __graft_entry__ as g
    g.build()
    return hy.load()


@pytest.fixture(scope="module")
def _built(_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _both(W, slots, n_slots):
    """(workspace entry point, no-allocation entry point) pools for layer 0."""
    L = W.layers[0]
    out = []
    for fn in (hy.segment_build, hy.segment_build_noalloc):
        T, S = new_pools(W.variant, n_slots, W.h_v, W.d_k, W.d_v, DEV)
        fn(L.k, L.v, L.g, L.beta, W.seg_offsets, variant=W.variant, seam_w=W.seam_w, T_pool=T, S_pool=S,
           slot_of_seg=slots)
        out.append((T, S))
    return out


CASES = [
    # tensor-core chunkwise path
    dict(cfg=5, variant="gdn", lengths=[1, 64, 65, 300, 129, 8, 9, 700], h_k=2, h_v=4, seam_w=8),
    dict(cfg=5, variant="deltanet", lengths=[200, 63, 1000, 16], h_k=1, h_v=2, seam_w=8),
    # fp32 token path
    dict(cfg=1, variant="channel", lengths=[50, 3, 90, 17, 64], h_k=1, h_v=2, seam_w=4, d=32),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", range(len(CASES)))
def test_noalloc_two_calls_match_workspace_build(_built, case):
    c = dict(CASES[case])
    runs = []
    for seed in (11, 12):                       # two different problems, one after the other
        W = si.workload(c["cfg"], seed=seed, device=DEV, variant=c["variant"], lengths=c["lengths"],
                        h_k=c["h_k"], h_v=c["h_v"], seam_w=c["seam_w"], d=c.get("d"))
        n = W.n_seg
        slots = np.random.default_rng(seed).permutation(n + 3)[:n].astype(np.int32)
        runs.append((W, slots, n + 3))
    # workspace entry point first, then both no-allocation calls back to back
    # on one stream with no host synchronisation between them
    ref = []
    for W, slots, n_slots in runs:
        T, S = new_pools(W.variant, n_slots, W.h_v, W.d_k, W.d_v, DEV)
        L = W.layers[0]
        hy.segment_build(L.k, L.v, L.g, L.beta, W.seg_offsets, variant=W.variant, seam_w=W.seam_w,
                         T_pool=T, S_pool=S, slot_of_seg=slots)
        ref.append((T, S))
    got = []
    for W, slots, n_slots in runs:
        T, S = new_pools(W.variant, n_slots, W.h_v, W.d_k, W.d_v, DEV)
        L = W.layers[0]
        hy.segment_build_noalloc(L.k, L.v, L.g, L.beta, W.seg_offsets, variant=W.variant, seam_w=W.seam_w,
                                 T_pool=T, S_pool=S, slot_of_seg=slots)
        got.append((T, S))
    torch.cuda.synchronize()
    for (W, slots, _), (Tr, Sr), (Tg, Sg) in zip(runs, ref, got):
        s = torch.as_tensor(slots, dtype=torch.long, device=DEV)
        assert torch.isfinite(Tr[s]).all() and torch.isfinite(Sr[s]).all()
        assert torch.equal(Tg[s], Tr[s]) and torch.equal(Sg[s], Sr[s])


@pytest.mark.gpu
def test_noalloc_at_the_pair_limit(_built):
    """n_seg * h_v == HYPIC_NOALLOC_MAX_PAIRS on the tensor-core path: the
    plan fills the whole fixed scratch; every slot must match the workspace
    build.  Short segments (0..70 body tokens) keep it quick."""
    assert 64 + 32 * hy.NOALLOC_MAX_PAIRS == 1 << 20
    n = hy.NOALLOC_MAX_PAIRS
    lens = np.random.default_rng(5).integers(1, 79, size=n).tolist()
    W = si.workload(5, seed=3, device=DEV, variant="gdn", lengths=lens, h_k=1, h_v=1, seam_w=8)
    (Tr, Sr), (Tg, Sg) = _both(W, None, n)
    torch.cuda.synchronize()
    assert torch.isfinite(Tr).all() and torch.isfinite(Sr).all()
    assert torch.equal(Tg, Tr) and torch.equal(Sg, Sr)


@pytest.mark.parametrize("n_seg,h_v", [(hy.NOALLOC_MAX_PAIRS + 1, 1), (16384, 2)])
def test_noalloc_refuses_problems_beyond_the_limit(_lib, n_seg, h_v):
    """Refused with HYPIC_ERR_WORKSPACE before any CUDA call (runs without a
    GPU too: no device pointer is read)."""
    lib = _lib
    d = hy.BuildDesc()
    off = np.zeros(n_seg + 1, np.int64)
    d.n_tokens, d.n_seg, d.h_k, d.h_v, d.d_k, d.d_v = 0, n_seg, 1, h_v, 128, 128
    d.variant, d.in_dtype = 0, hy.IN_BF16
    d.seg_offsets = off.ctypes.data_as(ctypes.c_void_p)
    d.n_slots = n_seg
    rc = lib.hypic_segment_build_noalloc(ctypes.byref(d), None)
    assert rc == 3, hy.status_string(rc)      # HYPIC_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_accepts_a_no_token_call_like_the_workspace_build(_built):
    """GDN with no tokens and no log-gate array (never read): both entry
    points accept it and write (I, 0) into every segment's slot."""
    k = torch.zeros((0, 1, 128), dtype=torch.bfloat16, device=DEV)
    v = torch.zeros((0, 2, 128), dtype=torch.bfloat16, device=DEV)
    off = np.zeros(4, np.int64)
    eye = torch.eye(128, device=DEV)
    for fn in (hy.segment_build, hy.segment_build_noalloc):
        T, S = new_pools("gdn", 3, 2, 128, 128, DEV)
        fn(k, v, None, None, off, variant="gdn", seam_w=8, T_pool=T, S_pool=S)
        torch.cuda.synchronize()
        assert torch.equal(T, eye.expand_as(T)) and torch.equal(S, torch.zeros_like(S))
