"""GPU tests of the host-buffer compose (hypic_compose_host): seam tokens and
initial states in page-locked host memory, the cached pairs on the device,
final states and seam outputs back in host memory, with the copies of one
group of layers overlapping the compose of the next.  The results must equal
the device compose's bit for bit (every (layer, value head) chain computes
the same thing whichever launch runs it): the tensor-core and fp32 kernels,
chunk counts from one to more than the layers, with and without host initial
states, on a side stream."""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_common import gpu_build, seam_arrays
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


def _prompt(variant, n_layers, w=8, h_k=2, h_v=4):
    cfg = 2 if variant == "scalar" else 5
    W = si.workload(cfg, device=DEV, variant=variant, lengths=[60, 200, 33, 128, 90], h_k=h_k, h_v=h_v, seam_w=w,
                    n_layers=n_layers)
    pools = [gpu_build(W, layer=l) for l in range(n_layers)]
    T_pool = torch.cat([p[0] for p in pools])
    S_pool = torch.cat([p[1] for p in pools])
    sa = seam_arrays(W, range(n_layers))
    slot = torch.arange(n_layers * W.n_seg, dtype=torch.int32, device=DEV).reshape(n_layers, W.n_seg)
    return W, T_pool, S_pool, sa, slot


@pytest.mark.parametrize("variant", ["gdn", "channel", "scalar"])
@pytest.mark.parametrize("n_chunks,with_init,L,h_v", [(1, False, 5, 4), (3, True, 5, 4), (9, True, 12, 32),
                                                     (2, False, 12, 32)])
def test_compose_host_equals_device_compose(variant, n_chunks, with_init, L, h_v):
    """12 layers x 32 heads (384 chains) take two waves on the device, so the
    call runs two groups of layers; 5 x 4 chains run as one."""
    W, T_pool, S_pool, sa, slot = _prompt(variant, L, h_k=h_v // 2, h_v=h_v)
    S_init = si.random_state((L, W.h_v, 128, 128), seed=4, cfg=5, device=DEV) if with_init else None
    keys = ("k", "v", "q", "g", "beta")
    # the device compose
    S_ref = torch.empty((L, W.h_v, 128, 128), device=DEV)
    o_ref = torch.empty((L, W.n_seg, W.seam_w, W.h_v, 128), device=DEV)
    hy.compose(slot, T_pool, S_pool, *(sa[k] for k in keys), variant=variant, S_out=S_ref, seam_out=o_ref,
               S_init=S_init, h_k=W.h_k)
    # the host-buffer compose: device staging starts zeroed
    host = {k: _pinned(sa[k]) for k in keys}
    stage = {k: (None if sa[k] is None else torch.zeros_like(sa[k])) for k in keys}
    S_init_dev = torch.zeros_like(S_init) if with_init else None
    S_out = torch.empty_like(S_ref)
    o_out = torch.empty_like(o_ref)
    S_host = torch.full(S_ref.shape, float("nan")).pin_memory()
    o_host = torch.full(o_ref.shape, float("nan")).pin_memory()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        hy.compose_host(*(host[k] for k in keys), slot, T_pool, S_pool, variant=variant,
                        seam_k=stage["k"], seam_v=stage["v"], seam_q=stage["q"], seam_g=stage["g"],
                        seam_beta=stage["beta"], S_out=S_out, S_out_host=S_host, seam_out=o_out,
                        seam_out_host=o_host, S_init=S_init_dev, S_init_host=_pinned(S_init), n_chunks=n_chunks,
                        h_k=W.h_k, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(S_host, S_ref.cpu())
    assert torch.equal(o_host, o_ref.cpu())


def test_compose_host_rejects_a_missing_host_array():
    W, T_pool, S_pool, sa, slot = _prompt("gdn", 1)
    keys = ("k", "v", "q", "g", "beta")
    host = {k: _pinned(sa[k]) for k in keys}
    host["q"] = None
    S_out = torch.empty((1, W.h_v, 128, 128), device=DEV)
    with pytest.raises(ValueError):
        hy.compose_host(*(host[k] for k in keys), slot, T_pool, S_pool, variant="gdn", seam_k=sa["k"],
                        seam_v=sa["v"], seam_q=sa["q"], seam_g=sa["g"], seam_beta=sa["beta"], S_out=S_out,
                        S_out_host=torch.empty(S_out.shape), h_k=W.h_k)
