"""GPU tests of the dispatch that callers can see: the path queries name the
kernel that actually runs (a sliced, misaligned input falls back to an fp32
CUDA-core kernel with the same results within its bar), the
require-tensor-cores flag refuses that fallback, and the round-robin
schedule (kept to measure what the LPT schedule gains, nav.aitube.vip §2.3)
gives the same pools bit for bit as the LPT one."""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_common import compare_pairs, new_pools, oracle_pairs, seam_arrays
from tolerance import TOL_BF16
import hybrid_linear_attention_chunkwise_gb300 as hy

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__ as g
    g.build()


@pytest.mark.parametrize("variant,cfg", [("gdn", 5), ("channel", 5), ("scalar", 2), ("deltanet", 5)])
def test_round_robin_schedule_gives_identical_pools(variant, cfg):
    lens = [300, 20, 1000, 64, 5, 700, 129, 250, 2048, 33]
    W = si.workload(cfg, device=DEV, variant=variant, lengths=lens, h_k=2, h_v=4, seam_w=8)
    L = W.layers[0]
    out = []
    for flags in (0, hy.FLAG_ROUND_ROBIN):
        T, S = new_pools(variant, W.n_seg, W.h_v, W.d_k, W.d_v, DEV)
        hy.segment_build(L.k, L.v, L.g, L.beta, W.seg_offsets, variant=variant, seam_w=W.seam_w, T_pool=T,
                         S_pool=S, flags=flags)
        out.append((T, S))
    torch.cuda.synchronize()
    (T0, S0), (T1, S1) = out
    assert torch.isfinite(S0).all() and torch.equal(T0, T1) and torch.equal(S0, S1)


def test_misaligned_input_path_is_reported_and_refusable():
    """k sliced one element off its 16-byte grid: the build cannot describe it
    as a TMA tensor, so it runs the fp32 token kernel.  The path query says
    so, the results still meet the bf16 bar, and the require-tensor-cores
    flag refuses the call without launching."""
    lens = [100, 300, 64]
    W = si.workload(5, device=DEV, variant="gdn", lengths=lens, h_k=2, h_v=4, seam_w=8)
    L = W.layers[0]
    T, S = new_pools("gdn", W.n_seg, W.h_v, 128, 128, DEV)
    kw = dict(variant="gdn", seam_w=W.seam_w, T_pool=T, S_pool=S)
    assert hy.build_path(L.k, L.v, L.g, L.beta, W.seg_offsets, **kw) == "tc_chunkwise"
    flat = torch.empty(L.k.numel() + 1, dtype=L.k.dtype, device=DEV)
    k_off = flat[1:].view(L.k.shape)          # same values, 2 bytes off the 16-byte grid
    k_off.copy_(L.k)
    assert hy.build_path(k_off, L.v, L.g, L.beta, W.seg_offsets, **kw) == "f32_token"
    with pytest.raises(hy.HypicError) as e:
        hy.segment_build(k_off, L.v, L.g, L.beta, W.seg_offsets, flags=hy.FLAG_REQUIRE_TENSOR_CORES, **kw)
    assert e.value.code == 2
    torch.cuda.synchronize()
    assert torch.isnan(S).all(), "a refused call launches nothing"
    hy.segment_build(k_off, L.v, L.g, L.beta, W.seg_offsets, **kw)
    torch.cuda.synchronize()
    eT, eS = compare_pairs(W, T, S, *oracle_pairs(W), range(W.n_seg))
    assert eT <= TOL_BF16 and eS <= TOL_BF16, (eT, eS)


def test_compose_path_with_two_value_heads_is_the_fp32_kernel():
    """h_v = 2 is not a multiple of 4: the compose runs the fp32 kernel; the
    query says so and the flag refuses it."""
    W = si.workload(5, device=DEV, variant="deltanet", lengths=[60, 90], h_k=1, h_v=2, seam_w=8)
    L = W.layers[0]
    T, S = new_pools("deltanet", W.n_seg, W.h_v, 128, 128, DEV)
    hy.segment_build(L.k, L.v, L.g, L.beta, W.seg_offsets, variant="deltanet", seam_w=8, T_pool=T, S_pool=S)
    sa = seam_arrays(W)
    slot = torch.arange(W.n_seg, dtype=torch.int32, device=DEV)[None]
    S_out = torch.empty((1, W.h_v, 128, 128), device=DEV)
    seam_out = torch.empty((1, W.n_seg, 8, W.h_v, 128), device=DEV)
    args = (slot, T, S, sa["k"], sa["v"], sa["q"], sa["g"], sa["beta"])
    assert hy.compose_path(*args, variant="deltanet", S_out=S_out, seam_out=seam_out) == "f32_compose"
    with pytest.raises(hy.HypicError):
        hy.compose(*args, variant="deltanet", S_out=S_out, seam_out=seam_out, flags=hy.FLAG_REQUIRE_TENSOR_CORES)
