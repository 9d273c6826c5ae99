"""GPU tests of the host-buffer build (hypic_segment_build_host): inputs in
page-locked host memory, pairs back in host memory, with the copies of one
group of segments overlapping the build of the next.  The pools must equal
the device build's bit for bit (every (segment, value head) item computes
the same thing whichever launch runs it), for every variant, bf16 and fp32
inputs, chunk counts from one to more than the segments, permuted slots in
a larger pool (slots no segment owns stay untouched), on a side stream; and
at the 64 x 1024-token GDN layer size."""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_common import gpu_build, new_pools
import hybrid_linear_attention_chunkwise_gb300 as hy

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__ as g
    g.build()


def _pinned(t):
    return None if t is None else t.detach().cpu().contiguous().pin_memory()


def _host_build(W, slots, n_slots, n_chunks, stream=None):
    L = W.layers[0]
    hk, hv, hg, hb = (_pinned(getattr(L, n)) for n in ("k", "v", "g", "beta"))
    # device staging that does not hold the inputs yet
    dk = torch.zeros_like(L.k)
    dv = torch.zeros_like(L.v)
    dg = None if L.g is None else torch.zeros_like(L.g)
    db = None if L.beta is None else torch.zeros_like(L.beta)
    T, S = new_pools(W.variant, n_slots, W.h_v, W.d_k, W.d_v, DEV)
    hT = torch.full(T.shape, 7.0).pin_memory()
    hS = torch.full(S.shape, 7.0).pin_memory()
    hy.segment_build_host(hk, hv, hg, hb, W.seg_offsets, variant=W.variant, seam_w=W.seam_w, k=dk, v=dv, g=dg,
                          beta=db, T_pool=T, S_pool=S, T_host=hT, S_host=hS, n_chunks=n_chunks, slot_of_seg=slots,
                          stream=stream)
    (stream or torch.cuda.current_stream()).synchronize()
    return hT, hS


VARIANTS = [("gdn", 5), ("deltanet", 5), ("channel", 5), ("scalar", 2), ("ungated", 5), ("diag", 5)]


@pytest.mark.parametrize("variant,cfg", VARIANTS)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("n_chunks", [1, 3, 100])
def test_host_build_equals_device_build(variant, cfg, dtype, n_chunks):
    lens = [40, 130, 12, 64, 300, 5, 0, 77]
    W = si.workload(cfg, device=DEV, variant=variant, lengths=lens, h_k=2, h_v=4, d=128, seam_w=8, dtype=dtype)
    n_slots = 12
    slots = np.asarray([9, 2, 5, 3, 4, 11, 0, 6], dtype=np.int32)  # runs 3-4 and single slots
    hT, hS = _host_build(W, slots, n_slots, n_chunks)
    T, S = gpu_build(W, slots=slots, n_slots=n_slots)
    torch.cuda.synchronize()
    T, S = T.cpu(), S.cpu()
    for i, sl in enumerate(slots):
        assert torch.equal(hT[sl], T[sl]) and torch.equal(hS[sl], S[sl]), (i, sl)
    free = sorted(set(range(n_slots)) - set(slots.tolist()))
    assert torch.all(hT[free] == 7.0) and torch.all(hS[free] == 7.0)


def test_host_build_on_a_side_stream_with_default_slots():
    W = si.workload(5, device=DEV, variant="gdn", lengths=[200, 3, 90, 513], h_k=2, h_v=4, d=64, seam_w=4)
    s = torch.cuda.Stream()
    hT, hS = _host_build(W, None, W.n_seg, 2, stream=s)
    T, S = gpu_build(W)
    torch.cuda.synchronize()
    assert torch.equal(hT, T.cpu()) and torch.equal(hS, S.cpu())


def test_host_build_gdn_layer():
    """The 64 x 1024-token GDN layer (16 key / 32 value heads, d = 128, bf16)
    in eight groups: every pair equals the device build's."""
    W = si.workload(3, seed=0, device=DEV)
    hT, hS = _host_build(W, None, W.n_seg, 8)
    T, S = gpu_build(W)
    torch.cuda.synchronize()
    assert torch.equal(hT, T.cpu()) and torch.equal(hS, S.cpu())


@pytest.mark.parametrize("variant", ["gdn", "channel", "scalar", "diag"])
def test_build_with_no_tokens(variant):
    """Segments that are all empty: every pair is (I, 0), or the empty gate
    product 1 for the scalar and diagonal transitions, by the device build
    and by the host-buffer build (no input is read)."""
    h_k, h_v, d = 2, 4, 128
    k = torch.empty(0, h_k, d, dtype=torch.bfloat16, device=DEV)
    v = torch.empty(0, h_v, d, dtype=torch.bfloat16, device=DEV)
    g = {"gdn": torch.empty(0, h_v, device=DEV), "channel": torch.empty(0, h_v, d, device=DEV),
         "scalar": -torch.rand(h_v, device=DEV), "diag": torch.empty(0, h_v, d, device=DEV)}[variant]
    beta = torch.empty(0, h_v, device=DEV) if variant in ("gdn", "channel") else None
    off = np.zeros(4, dtype=np.int64)
    T, S = new_pools(variant, 3, h_v, d, d, DEV)
    hy.segment_build(k, v, g, beta, off, variant=variant, seam_w=2, T_pool=T, S_pool=S)
    torch.cuda.synchronize()
    if variant in ("gdn", "channel"):
        want_T = torch.eye(d).expand(3, h_v, d, d)
    else:
        want_T = torch.ones(T.shape)
    assert torch.equal(T.cpu(), want_T) and torch.equal(S.cpu(), torch.zeros(S.shape))
    T2, S2 = new_pools(variant, 3, h_v, d, d, DEV)
    hT, hS = torch.full(T2.shape, 7.0).pin_memory(), torch.full(S2.shape, 7.0).pin_memory()
    hy.segment_build_host(k.cpu(), v.cpu(), g.cpu(), None if beta is None else beta.cpu(), off, variant=variant,
                          seam_w=2, k=k, v=v, g=g, beta=beta, T_pool=T2, S_pool=S2, T_host=hT, S_host=hS,
                          n_chunks=3)
    torch.cuda.synchronize()
    assert torch.equal(hT, want_T) and torch.equal(hS, torch.zeros(S.shape))


def test_host_build_and_host_compose_on_two_streams():
    """A host-buffer build and a host-buffer compose enqueued on two streams
    (each caller stream gets its own copy streams, so they overlap) give the
    device calls' results bit for bit; repeated, the pipes are reused."""
    lens = [40, 130, 12, 64, 300, 5, 77, 200]
    W = si.workload(5, device=DEV, variant="gdn", lengths=lens, h_k=2, h_v=4, seam_w=8, n_layers=3)
    L = W.layers[0]
    hk, hv, hg, hb = (_pinned(getattr(L, n)) for n in ("k", "v", "g", "beta"))
    T_ref, S_ref = gpu_build(W)
    # a compose over the three layers' pools
    from gpu_common import seam_arrays
    pools = [gpu_build(W, layer=l) for l in range(3)]
    T_pool = torch.cat([p[0] for p in pools])
    S_pool = torch.cat([p[1] for p in pools])
    sa = seam_arrays(W, range(3))
    keys = ("k", "v", "q", "g", "beta")
    slot = torch.arange(3 * W.n_seg, dtype=torch.int32, device=DEV).reshape(3, W.n_seg)
    So_ref = torch.empty((3, W.h_v, 128, 128), device=DEV)
    oo_ref = torch.empty((3, W.n_seg, W.seam_w, W.h_v, 128), device=DEV)
    hy.compose(slot, T_pool, S_pool, *(sa[k] for k in keys), variant="gdn", S_out=So_ref, seam_out=oo_ref, h_k=W.h_k)
    torch.cuda.synchronize()
    host4 = {k: _pinned(sa[k]) for k in keys}
    sA, sB = torch.cuda.Stream(), torch.cuda.Stream()
    for rep in range(2):
        T, S = new_pools("gdn", W.n_seg, W.h_v, 128, 128, DEV)
        hT = torch.full(T.shape, 7.0).pin_memory()
        hS = torch.full(S.shape, 7.0).pin_memory()
        st = {k: torch.zeros_like(sa[k]) for k in keys}
        So = torch.empty_like(So_ref)
        oo = torch.empty_like(oo_ref)
        hSo = torch.full(So.shape, float("nan")).pin_memory()
        hoo = torch.full(oo.shape, float("nan")).pin_memory()
        stage = [torch.zeros_like(x) for x in (L.k, L.v, L.g, L.beta)]
        sA.wait_stream(torch.cuda.current_stream())  # the buffers above are filled on the current stream
        sB.wait_stream(torch.cuda.current_stream())
        hy.segment_build_host(hk, hv, hg, hb, W.seg_offsets, variant="gdn", seam_w=W.seam_w, k=stage[0], v=stage[1],
                              g=stage[2], beta=stage[3], T_pool=T, S_pool=S, T_host=hT, S_host=hS, n_chunks=3,
                              stream=sA)
        hy.compose_host(*(host4[k] for k in keys), slot, T_pool, S_pool, variant="gdn", seam_k=st["k"],
                        seam_v=st["v"], seam_q=st["q"], seam_g=st["g"], seam_beta=st["beta"], S_out=So,
                        S_out_host=hSo, seam_out=oo, seam_out_host=hoo, n_chunks=3, h_k=W.h_k, stream=sB)
        sA.synchronize()
        sB.synchronize()
        assert torch.equal(hT, T_ref.cpu()) and torch.equal(hS, S_ref.cpu()), rep
        assert torch.equal(hSo, So_ref.cpu()) and torch.equal(hoo, oo_ref.cpu()), rep
