"""GPU tests of the prefill forward (hypic_segment_forward): the pairs as
for the build, and the output o_t = S_t^T q_t of every body token from the
zero-initial body state, against the fp64 oracle's plain recurrence run on
each body alone (every variant, bf16 and fp32 inputs, narrow and 128-wide
heads, with and without a seam window; bf16 heads of width 20 have rows off the
16-byte grid, so their inputs are staged by plain loads instead of
asynchronous copies); seam-token rows stay untouched; a sampled check on the
64 x 1024-token GDN layer."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from gpu_common import compare_pairs, new_pools, oracle_pairs, tol_for
from tolerance import per_head_rel_err
import hybrid_linear_attention_chunkwise_gb300 as hy

pytestmark = pytest.mark.gpu
DEV = "cuda"
ALL = ("gdn", "deltanet", "channel", "scalar", "ungated", "diag")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__ as g
    g.build()


def _forward(W):
    L = W.layers[0]
    T, S = new_pools(W.variant, W.n_seg, W.h_v, W.d_k, W.d_v, DEV)
    o = torch.full((W.n_tokens, W.h_v, W.d_v), float("nan"), device=DEV)
    hy.segment_forward(L.k, L.v, L.q, L.g, L.beta, W.seg_offsets, variant=W.variant, seam_w=W.seam_w,
                       T_pool=T, S_pool=S, o_out=o)
    torch.cuda.synchronize()
    return T, S, o


def _body_outputs_ref(W, seg, heads=None):
    """oracle.full over segment seg's body alone, from a zero state."""
    L = W.layers[0]
    off = W.seg_offsets
    s0, e = min(int(off[seg]) + W.seam_w, int(off[seg + 1])), int(off[seg + 1])
    if e <= s0:
        return s0, e, None
    cpu = lambda x: None if x is None else x.detach().cpu()
    g = cpu(L.g)
    gb = g if (g is None or g.dim() == 1) else g[s0:e]
    beta = None if L.beta is None else cpu(L.beta)[s0:e]
    _, outs = oracle.full(W.variant, cpu(L.k)[s0:e], cpu(L.v)[s0:e], cpu(L.q)[s0:e], gb, beta, W.h_k, W.h_v,
                          out_pos=np.arange(e - s0))
    return s0, e, outs


@pytest.mark.parametrize("variant", ALL)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("d,w", [(32, 8), (128, 0), (128, 8), (20, 4)])
def test_forward_outputs_vs_oracle(variant, dtype, d, w):
    lens = [40, 130, 12, 64, 300, 5]
    W = si.workload(2 if variant == "scalar" else 5, device=DEV, variant=variant, lengths=lens, h_k=2, h_v=4,
                    d=d, seam_w=w, dtype=dtype)
    T, S, o = _forward(W)
    tol = tol_for(dtype)
    eT, eS = compare_pairs(W, T, S, *oracle_pairs(W), range(W.n_seg))
    assert eT <= tol and eS <= tol, (eT, eS)
    oc = o.cpu().double().numpy()
    for i in range(W.n_seg):
        s0, e, ref = _body_outputs_ref(W, i)
        assert np.isnan(oc[int(W.seg_offsets[i]):s0]).all(), "seam rows must stay untouched"
        if ref is None:
            continue
        err = per_head_rel_err(np.transpose(oc[s0:e], (1, 0, 2)), np.transpose(ref, (1, 0, 2))).max()
        assert err <= tol, (i, err)


def test_forward_gdn_layer_sampled():
    """The 64 x 1024-token GDN layer (16 key / 32 value heads, d = 128,
    bf16): every pair and output written, three segments checked against the
    oracle on every head."""
    W = si.workload(3, seed=0, device=DEV)
    T, S, o = _forward(W)
    assert torch.isfinite(o).all()
    oc = o.cpu().double().numpy()
    for i in (0, 31, 63):
        s0, e, ref = _body_outputs_ref(W, i)
        err = per_head_rel_err(np.transpose(oc[s0:e], (1, 0, 2)), np.transpose(ref, (1, 0, 2))).max()
        assert err <= tol_for(torch.bfloat16), (i, err)
    eT, eS = compare_pairs(W, T, S, *oracle_pairs(W, segs=[5]), [5])
    assert eT <= tol_for(torch.bfloat16) and eS <= tol_for(torch.bfloat16)


@pytest.mark.parametrize("variant", ["gdn", "gdn_f32", "deltanet", "scalar"])
@pytest.mark.parametrize("gate", ["steep", "underflow"])
def test_forward_steep_gates_token_by_token(variant, gate):
    """Scalar gates keep the state as A * X with the scale folded into X
    before A drops below 2^-64.  Log-gates around -20 per token fold at
    nearly every token; a gate of -200 underflows e^g to 0 in fp32 and must
    clear the state.  Every body token's output is checked on its own,
    relative to the larger of its own norm and the head's RMS output norm, so
    a slip at one token (e.g. just after a fold) fails.  DeltaNet has no gate
    and must be unaffected.  bf16 GDN runs the tensor-core outputs, fp32 GDN
    and the scalar decay the fp32 token recurrence whose state folds the
    scale."""
    lens = [70, 200, 33, 129]
    dtype = torch.float32 if variant == "gdn_f32" else torch.bfloat16
    variant = "gdn" if variant == "gdn_f32" else variant
    W = si.workload(2 if variant == "scalar" else 5, device=DEV, variant=variant, lengths=lens, h_k=2, h_v=4,
                    seam_w=4, dtype=dtype)
    L = W.layers[0]
    gen = torch.Generator(device="cpu").manual_seed(7)
    if variant == "gdn":
        g = -15.0 - 10.0 * torch.rand(L.g.shape, generator=gen)
        if gate == "underflow":
            g[50:60] = -200.0   # inside the first body, and a run of them
            g[300:301] = -200.0
        L.g.copy_(g.to(L.g.device))
    elif variant == "scalar":
        L.g.fill_(-200.0 if gate == "underflow" else -20.0)
    T, S, o = _forward(W)
    oc = o.cpu().double().numpy()
    tol = tol_for(dtype)
    for i in range(W.n_seg):
        s0, e, ref = _body_outputs_ref(W, i)
        if ref is None:
            continue
        got = oc[s0:e]                                   # [tokens, h_v, d_v]
        dn = np.linalg.norm(got - ref, axis=-1)           # [tokens, h_v]
        rn = np.linalg.norm(ref, axis=-1)
        rms = np.sqrt((rn ** 2).mean(axis=0, keepdims=True))
        worst = (dn / np.maximum(rn, rms)).max()
        assert np.isfinite(got).all() and worst <= tol, (i, worst)
    eT, eS = compare_pairs(W, T, S, *oracle_pairs(W), range(W.n_seg))
    assert eT <= tol and eS <= tol, (eT, eS)


def test_forward_path_query_names_the_tensor_core_outputs():
    """bf16 GDN / DeltaNet with 128-wide heads take the tensor-core output
    kernel (chunk records of the build); fp32 inputs, narrower heads and the
    other variants the fp32 token recurrence."""
    lens = [70, 130]
    for variant, d, dtype, want in (("gdn", 128, torch.bfloat16, "tc_forward"),
                                    ("deltanet", 128, torch.bfloat16, "tc_forward"),
                                    ("gdn", 128, torch.float32, "f32_token"),
                                    ("gdn", 32, torch.bfloat16, "f32_token"),
                                    ("channel", 128, torch.bfloat16, "f32_token")):
        W = si.workload(5, device=DEV, variant=variant, lengths=lens, h_k=2, h_v=4, d=d, seam_w=8, dtype=dtype)
        L = W.layers[0]
        T, S = new_pools(variant, W.n_seg, W.h_v, W.d_k, W.d_v, DEV)
        o = torch.empty((W.n_tokens, W.h_v, W.d_v), device=DEV)
        got = hy.forward_path(L.k, L.v, L.q, L.g, L.beta, W.seg_offsets, variant=variant, seam_w=8, T_pool=T,
                              S_pool=S, o_out=o)
        assert got == want, (variant, d, dtype, got)


@pytest.mark.parametrize("variant", ["gdn", "deltanet"])
def test_forward_tc_long_bodies_every_token(variant):
    """Bodies of 1 .. 1100 tokens (chunk tails of every length class, one
    body of a single token) on the tensor-core output path: every output
    token against the oracle recurrence, the pairs against the oracle's."""
    lens = [9, 72, 1100, 200, 65, 127, 64, 8]
    W = si.workload(5, device=DEV, variant=variant, lengths=lens, h_k=2, h_v=4, seam_w=8)
    T, S, o = _forward(W)
    oc = o.cpu().double().numpy()
    tol = tol_for(torch.bfloat16)
    for i in range(W.n_seg):
        s0, e, ref = _body_outputs_ref(W, i)
        assert np.isnan(oc[int(W.seg_offsets[i]):s0]).all()
        if ref is None:
            continue
        err = per_head_rel_err(np.transpose(oc[s0:e], (1, 0, 2)), np.transpose(ref, (1, 0, 2))).max()
        assert err <= tol, (i, err)
    eT, eS = compare_pairs(W, T, S, *oracle_pairs(W), range(W.n_seg))
    assert eT <= tol and eS <= tol, (eT, eS)
