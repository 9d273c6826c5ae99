"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs, element by element, with the per-head relative
Frobenius bound: 5e-3 for bf16 inputs, 1e-5 for fp32 inputs."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from gpu_common import (DENSE, compare_pairs, dense_T, gpu_build, new_pools, oracle_pairs,
                        seam_arrays, tol_for)
from tolerance import TOL_BF16, TOL_F32, per_head_rel_err
import hybrid_linear_attention_chunkwise_gb300 as hy

pytestmark = pytest.mark.gpu

ALL = ("gdn", "deltanet", "channel", "scalar", "ungated", "diag")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__ as g
    g.build()
    torch.cuda.set_device(0)


DEV = "cuda"


def _compose_vs_full(W, T_pool, S_pool, tol, S_init=None, layers=(0,)):
    """Compose the pool in prompt order with the seam tokens and compare the
    final state and seam outputs with the fp64 full recurrence of each
    layer's whole prompt."""
    n_l = len(layers)
    sa = seam_arrays(W, layers)
    slot = torch.arange(W.n_seg, dtype=torch.int32, device=DEV)[None].repeat(n_l, 1)
    for j, l in enumerate(layers):
        slot[j] += l * W.n_seg
    S_out = torch.empty((n_l, W.h_v, W.d_k, W.d_v), device=DEV)
    seam_out = torch.empty((n_l, W.n_seg, W.seam_w, W.h_v, W.d_v), device=DEV) if W.seam_w else None
    g = sa["g"]
    hy.compose(slot, T_pool, S_pool, sa["k"], sa["v"], sa["q"], g, sa["beta"], variant=W.variant,
               S_out=S_out, seam_out=seam_out, S_init=S_init)
    torch.cuda.synchronize()
    worst = 0.0
    valid = si.seam_gather(W, W.layers[layers[0]])["valid"].cpu().numpy()
    for j, l in enumerate(layers):
        L = W.layers[l]
        pos = [int(W.seg_offsets[i]) + t for i in range(W.n_seg) for t in range(W.seam_w) if valid[i, t]]
        cpu = [None if x is None else x.cpu() for x in (L.k, L.v, L.q, L.g, L.beta)]
        S0 = None if S_init is None else S_init[j].cpu()
        Sf, outs = oracle.full(W.variant, *cpu, W.h_k, W.h_v, S_init=S0, out_pos=pos)
        worst = max(worst, float(per_head_rel_err(S_out[j], Sf).max()))
        if W.seam_w:
            so = seam_out[j].cpu().numpy()[valid]          # [n_valid, h_v, d_v]
            e = per_head_rel_err(np.transpose(so, (1, 0, 2)), np.transpose(outs, (1, 0, 2)))
            worst = max(worst, float(e.max()))
    assert worst <= tol, worst
    return worst


def test_config1_tiny_gdn_fp32():
    """1 head, d=16, 4 x 64 tokens, w=8, fp32: pairs vs oracle and composed
    state + seam outputs vs the full token-by-token recurrence."""
    W = si.workload(1, device=DEV)
    T_pool, S_pool = gpu_build(W)
    T, S = oracle_pairs(W)
    eT, eS = compare_pairs(W, T_pool, S_pool, T, S, range(W.n_seg))
    assert eT <= TOL_F32 and eS <= TOL_F32, (eT, eS)
    _compose_vs_full(W, T_pool, S_pool, TOL_F32)
    S0 = si.random_state((1, W.h_v, W.d_k, W.d_v), seed=0, cfg=1, device=DEV)
    _compose_vs_full(W, T_pool, S_pool, TOL_F32, S_init=S0)


@pytest.mark.parametrize("variant", ALL)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("d,w", [(32, 8), (128, 0), (128, 8)])
def test_variants_fuzzed_lengths(variant, dtype, d, w):
    """Ragged lengths (empty, shorter than / equal to the seam, one chunk,
    several chunks with a tail), grouped heads, every variant."""
    lens = [0, 1, 5, 8, 9, 64, 65, 130, 300]
    W = si.workload(5, device=DEV, variant=variant, lengths=lens, h_k=2, h_v=4, d=d, seam_w=w,
                    dtype=dtype)
    slots = np.random.default_rng(1).permutation(len(lens)).astype(np.int32)
    T_pool, S_pool = gpu_build(W, slots=slots, n_slots=len(lens) + 3)
    T, S = oracle_pairs(W)
    eT, eS = compare_pairs(W, T_pool, S_pool, T, S, range(W.n_seg), slots=slots)
    tol = tol_for(dtype)
    assert eT <= tol and eS <= tol, (eT, eS)
    # untouched slots stay as they were
    unused = sorted(set(range(len(lens) + 3)) - set(slots.tolist()))
    assert torch.isnan(S_pool[unused]).all()


@pytest.mark.parametrize("variant", ALL)
def test_compose_all_variants(variant):
    lens = [12, 40, 9, 70, 33]
    for dtype in (torch.float32, torch.bfloat16):
        W = si.workload(5, device=DEV, variant=variant, lengths=lens, h_k=2, h_v=4, d=32, seam_w=8,
                        dtype=dtype, n_layers=2)
        pools = [gpu_build(W, layer=l) for l in range(2)]
        T_pool = torch.cat([p[0] for p in pools])
        S_pool = torch.cat([p[1] for p in pools])
        S0 = si.random_state((2, W.h_v, W.d_k, W.d_v), seed=0, cfg=5, device=DEV)
        _compose_vs_full(W, T_pool, S_pool, tol_for(dtype), S_init=S0, layers=(0, 1))


def test_config2_retnet_fast_path_and_naive_sum():
    """RetNet decay, 8 heads, d=128, 16 x 512 bf16: scalar T_C = gamma^L and
    S(C|0); the naive sum of zero-initial states misses the decay."""
    W = si.workload(2, device=DEV)
    W0 = si.workload(2, device=DEV, seam_w=0)
    T_pool, S_pool = gpu_build(W0)
    T, S = oracle_pairs(W0)
    eT, eS = compare_pairs(W0, T_pool, S_pool, T, S, range(W0.n_seg))
    assert eT <= TOL_BF16 and eS <= TOL_BF16, (eT, eS)
    L = W0.layers[0]
    cpu = [None if x is None else x.cpu() for x in (L.k, L.v, L.q, L.g, L.beta)]
    Sf, _ = oracle.full("scalar", *cpu, W0.h_k, W0.h_v)
    naive = S_pool.sum(0)
    err = per_head_rel_err(naive, Sf)
    assert err.min() >= 0.10, err
    # with seams: compose reproduces the full recurrence
    Tw, Sw = gpu_build(W)
    _compose_vs_full(W, Tw, Sw, TOL_BF16)


def test_config3_gdn_layer_sampled():
    """Qwen3.5-35B-A3B-shaped GDN layer: 64 x 1024 tokens, 16 key / 32 value
    heads, d=128, one batched launch; the oracle checks 3 sampled segments,
    all 32 heads."""
    W = si.workload(3, device=DEV)
    T_pool, S_pool = gpu_build(W)
    assert not torch.isnan(S_pool).any() and not torch.isnan(T_pool).any()
    segs = [0, 37, 63]
    T, S = oracle_pairs(W, segs=segs)
    eT, eS = compare_pairs(W, T_pool, S_pool, T, S, segs)
    assert eT <= TOL_BF16 and eS <= TOL_BF16, (eT, eS)


@pytest.mark.parametrize("variant", ["gdn", "deltanet", "channel"])
def test_config5_cold_uneven_sampled(variant):
    """256 segments of 256..8192 tokens, 32 value heads: one launch; the
    oracle checks the longest segment and two others on one key-head group."""
    W = si.workload(5, device=DEV, variant=variant)
    T_pool, S_pool = gpu_build(W)
    assert not torch.isnan(S_pool).any()
    lens = np.diff(W.seg_offsets)
    segs = [int(np.argmax(lens)), 1, 100]
    heads = ([5], [10, 11])
    T, S = oracle_pairs(W, segs=segs, heads=heads)
    eT, eS = compare_pairs(W, T_pool, S_pool, T, S, segs, heads=heads)
    assert eT <= TOL_BF16 and eS <= TOL_BF16, (eT, eS)


def test_config4_compose_sampled_chains():
    """Warm RAG prompt: 30 GDN layers x 32 heads, 100 lognormal segments,
    w=8.  Pairs are built on the GPU from seeded inputs; sampled (layer, head)
    chains are composed by the oracle from the same fp32 pairs."""
    W = si.workload(4, device=DEV, n_layers=1)
    n_layers = 30
    n_slots = n_layers * W.n_seg
    T_pool, S_pool = new_pools("gdn", n_slots, W.h_v, W.d_k, W.d_v, DEV, fill=0.0)
    seams = []
    layer0 = W.layers[0]
    for l in range(n_layers):
        lay = layer0 if l == 0 else si.make_layer(seed=0, cfg=4, layer=l, n_tokens=W.n_tokens, h_k=W.h_k,
                                                        h_v=W.h_v, d_k=W.d_k, d_v=W.d_v, variant="gdn",
                                                        dtype=torch.bfloat16, device=DEV)
        W.layers = [lay]
        slots = np.arange(W.n_seg, dtype=np.int32) + l * W.n_seg
        gpu_build(W, slots=slots, T_pool=T_pool, S_pool=S_pool)
        seams.append(si.seam_gather(W, lay))
    sa = {k: torch.stack([s[k] for s in seams]).contiguous() for k in ("k", "v", "q", "g", "beta")}
    slot = torch.arange(n_slots, dtype=torch.int32, device=DEV).reshape(n_layers, W.n_seg)
    S_out = torch.empty((n_layers, W.h_v, W.d_k, W.d_v), device=DEV)
    seam_out = torch.empty((n_layers, W.n_seg, W.seam_w, W.h_v, W.d_v), device=DEV)
    hy.compose(slot, T_pool, S_pool, sa["k"], sa["v"], sa["q"], sa["g"], sa["beta"], variant="gdn",
               S_out=S_out, seam_out=seam_out)
    torch.cuda.synchronize()
    for (l, h) in [(0, 0), (17, 31), (29, 6)]:
        kh = h * W.h_k // W.h_v
        rows = slice(l * W.n_seg, (l + 1) * W.n_seg)
        Tp = T_pool[rows, h:h + 1][None]
        Sp = S_pool[rows, h:h + 1][None]
        sk = sa["k"][l:l + 1, :, :, kh:kh + 1]
        sq = sa["q"][l:l + 1, :, :, kh:kh + 1]
        sv = sa["v"][l:l + 1, :, :, h:h + 1]
        sg = sa["g"][l:l + 1, :, :, h:h + 1]
        sb = sa["beta"][l:l + 1, :, :, h:h + 1]
        So, seam = oracle.compose("gdn", Tp.cpu(), Sp.cpu(), sk.cpu(), sv.cpu(), sq.cpu(), sg.cpu(), sb.cpu(), 1, 1)
        e1 = per_head_rel_err(S_out[l, h:h + 1], So[0]).max()
        e2 = per_head_rel_err(seam_out[l, :, :, h].reshape(1, -1, W.d_v), seam[0, :, :, 0].reshape(1, -1, W.d_v)).max()
        assert e1 <= TOL_BF16 and e2 <= TOL_BF16, (l, h, e1, e2)


def test_deltanet_compose_nontrivial_T():
    """With alpha = 1 the cached T_C is far from zero, so T_C S matters."""
    W = si.workload(4, device=DEV, variant="deltanet", n_layers=2, n_seg=12, h_k=2, h_v=4)
    pools = [gpu_build(W, layer=l) for l in range(2)]
    T_pool = torch.cat([p[0] for p in pools])
    S_pool = torch.cat([p[1] for p in pools])
    assert float(T_pool.abs().max()) > 1e-3
    S0 = si.random_state((2, W.h_v, W.d_k, W.d_v), seed=0, cfg=4, device=DEV)
    _compose_vs_full(W, T_pool, S_pool, TOL_BF16, S_init=S0, layers=(0, 1))


def test_build_deterministic_and_order_free():
    W = si.workload(5, device=DEV, variant="gdn", lengths=[300, 64, 1000, 129], h_k=2, h_v=4, seam_w=8)
    a = [x.clone() for x in gpu_build(W)]
    b = gpu_build(W)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    slots = np.array([3, 1, 0, 2], dtype=np.int32)
    c = gpu_build(W, slots=slots)
    assert torch.equal(c[1][torch.as_tensor(slots, dtype=torch.long)], a[1])


def test_empty_and_degenerate():
    W = si.workload(5, device=DEV, variant="gdn", lengths=[0, 0, 3], h_k=1, h_v=1, d=16, seam_w=8)
    T_pool, S_pool = gpu_build(W)
    eye = torch.eye(16, device=DEV)
    for i in range(3):
        assert torch.equal(T_pool[i, 0], eye) and torch.equal(S_pool[i, 0], torch.zeros_like(eye))
    W0 = si.workload(5, device=DEV, variant="gdn", lengths=[], h_k=1, h_v=1, d=16, seam_w=0)
    T_pool, S_pool = new_pools("gdn", 1, 1, 16, 16, DEV)
    hy.segment_build(W0.layers[0].k, W0.layers[0].v, W0.layers[0].g, W0.layers[0].beta, W0.seg_offsets,
                     variant="gdn", seam_w=0, T_pool=T_pool, S_pool=S_pool)
    torch.cuda.synchronize()
    assert torch.isnan(S_pool).all()


def test_status_word_bad_slot_and_nonfinite():
    W = si.workload(5, device=DEV, variant="gdn", lengths=[20, 30], h_k=1, h_v=2, d=32, seam_w=4)
    T_pool, S_pool = gpu_build(W)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sa = seam_arrays(W)
    slot = torch.tensor([[0, 7]], dtype=torch.int32, device=DEV)
    S_out = torch.empty((1, W.h_v, W.d_k, W.d_v), device=DEV)
    seam_out = torch.empty((1, W.n_seg, W.seam_w, W.h_v, W.d_v), device=DEV)
    hy.compose(slot, T_pool, S_pool, sa["k"], sa["v"], sa["q"], sa["g"], sa["beta"], variant="gdn",
               S_out=S_out, seam_out=seam_out, status=status)
    torch.cuda.synchronize()
    assert hy.status_from_word(int(status.item())) == 7
    # a NaN planted in the host-made inputs (token 10: inside the first
    # segment's body, past its 4 seam tokens) is reported, not trapped
    W.layers[0].v[10, 1, 5] = float("nan")
    status.zero_()
    gpu_build(W, status=status, flags=hy.FLAG_CHECK_FINITE)
    torch.cuda.synchronize()
    assert hy.status_from_word(int(status.item())) == 6
