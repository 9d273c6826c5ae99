"""GPU parity on the full warm-prompt workload: 30 GDN layers x 32 value heads
(16 key heads), d = 128, 100 segments with lognormal lengths (median 1000,
sigma 0.3, clipped to 512..4096; about 105k tokens), seam window w = 8, bf16
tokens, fp32 pairs.

The pairs of all 30 layers are built on the GPU into one 12.6 GB pool and
composed in one launch, as the bench times them.  For sampled (layer, value
head) chains the test then checks, against the fp64 oracle:
  - every GPU-built pair of the chain (100 segments) against the oracle's
    token-by-token build of the same segment bodies (nav.aitube.vip §2.1:
    T_C is the product of the body's token transitions, S(C|0) its state
    from zero);
  - end to end, GPU build then GPU compose against the plain recurrence over
    the whole ~105k-token prompt: the final state and every seam token's
    output (§2.1: the composed state equals the full recompute; §2.2: the
    seam tokens advance the running state and emit their outputs).
Per-head relative Frobenius error 5e-3 (bf16 inputs, fp32 state).  A
DeltaNet prompt (alpha = 1, so T_C carries the whole history) runs the same
checks on two layers."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from tolerance import TOL_BF16, per_head_rel_err
import hybrid_linear_attention_chunkwise_gb300 as hy

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__ as g
    g.build()


def _layer(W, l, variant, seed=0):
    return si.make_layer(seed=seed, cfg=4, layer=l, n_tokens=W.n_tokens, h_k=W.h_k, h_v=W.h_v, d_k=W.d_k,
                         d_v=W.d_v, variant=variant, dtype=torch.bfloat16, device=DEV)


def _prompt(n_layers, variant):
    """Pools of every layer, built on the GPU, and the composed chains."""
    W = si.workload(4, seed=0, device=DEV, n_layers=1, variant=variant)
    n_seg = W.n_seg
    T_pool = torch.empty((n_layers * n_seg, W.h_v, 128, 128), device=DEV)
    S_pool = torch.empty_like(T_pool)
    seams = []
    for l in range(n_layers):
        lay = _layer(W, l, variant)
        hy.segment_build(lay.k, lay.v, lay.g, lay.beta, W.seg_offsets, variant=variant, seam_w=W.seam_w,
                         T_pool=T_pool, S_pool=S_pool, slot_of_seg=np.arange(n_seg, dtype=np.int32) + l * n_seg)
        seams.append(si.seam_gather(W, lay))
        del lay
    sa = {k: (torch.stack([s[k] for s in seams]).contiguous() if seams[0][k] is not None else None)
          for k in ("k", "v", "q", "g", "beta")}
    del seams
    slot = torch.arange(n_layers * n_seg, dtype=torch.int32, device=DEV).reshape(n_layers, n_seg)
    S_out = torch.empty((n_layers, W.h_v, 128, 128), device=DEV)
    seam_out = torch.empty((n_layers, n_seg, W.seam_w, W.h_v, 128), device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert hy.compose_path(slot, T_pool, S_pool, sa["k"], sa["v"], sa["q"], sa["g"], sa["beta"], variant=variant,
                           S_out=S_out, seam_out=seam_out) == "tc_compose"
    hy.compose(slot, T_pool, S_pool, sa["k"], sa["v"], sa["q"], sa["g"], sa["beta"], variant=variant, S_out=S_out,
               seam_out=seam_out, status=status, flags=hy.FLAG_CHECK_FINITE)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return W, T_pool, S_pool, S_out, seam_out


def _check_chain(W, variant, l, h, T_pool, S_pool, S_out, seam_out):
    n_seg, w = W.n_seg, W.seam_w
    kh = h * W.h_k // W.h_v
    lay = _layer(W, l, variant)
    cpu = lambda x, hh: None if x is None else x[:, hh:hh + 1].cpu()
    k, q, v = cpu(lay.k, kh), cpu(lay.q, kh), cpu(lay.v, h)
    g, beta = cpu(lay.g, h), cpu(lay.beta, h)
    del lay
    # the pairs of the chain
    To, So = oracle.build_pairs(variant, W.seg_offsets, w, 1, 1, 128, 128, k, v, g, beta)
    sl = slice(l * n_seg, (l + 1) * n_seg)
    eT = per_head_rel_err(T_pool[sl, h:h + 1].cpu(), To).max()
    eS = per_head_rel_err(S_pool[sl, h:h + 1].cpu(), So).max()
    assert eT <= TOL_BF16 and eS <= TOL_BF16, (l, h, eT, eS)
    # end to end against the plain recurrence over the whole prompt
    pos = [int(W.seg_offsets[i]) + t for i in range(n_seg) for t in range(w)]
    Sf, outs = oracle.full(variant, k, v, q, g, beta, 1, 1, out_pos=pos)
    eF = per_head_rel_err(S_out[l, h:h + 1].cpu(), Sf).max()
    got = seam_out[l, :, :, h].reshape(1, n_seg * w, 128).cpu()
    eO = per_head_rel_err(got, np.transpose(outs, (1, 0, 2))).max()
    assert eF <= TOL_BF16 and eO <= TOL_BF16, (l, h, eF, eO)
    return eT, eS, eF, eO


def test_warm_prompt_gdn_30_layers_sampled_chains_vs_oracle():
    W, T_pool, S_pool, S_out, seam_out = _prompt(30, "gdn")
    assert 95_000 <= W.n_tokens <= 115_000 and W.n_seg == 100
    for l, h in ((3, 0), (17, 13), (29, 31)):
        _check_chain(W, "gdn", l, h, T_pool, S_pool, S_out, seam_out)


def test_warm_prompt_deltanet_sampled_chains_vs_oracle():
    W, T_pool, S_pool, S_out, seam_out = _prompt(2, "deltanet")
    for l, h in ((0, 6), (1, 27)):
        _check_chain(W, "deltanet", l, h, T_pool, S_pool, S_out, seam_out)
