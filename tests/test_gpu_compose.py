"""GPU tests of the tensor-core compose path (dense transitions, bf16 seam
tokens, d = 128): parity with the fp64 oracle composing the same fp32 pairs,
seam widths that need one or two seam buffers per segment, out-of-range
slots, and the bounded-wait timeout."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from gpu_common import dense_T, gpu_build, seam_arrays
from tolerance import TOL_BF16, per_head_rel_err
import hybrid_linear_attention_chunkwise_gb300 as hy

pytestmark = pytest.mark.gpu
DEV = "cuda"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__ as g
    g.build()


def _run(W, n_layers, S_init=None, status=None, slot=None):
    pools = [gpu_build(W, layer=l) for l in range(n_layers)]
    T_pool = torch.cat([p[0] for p in pools])
    S_pool = torch.cat([p[1] for p in pools])
    sa = seam_arrays(W, range(n_layers))
    if slot is None:
        slot = torch.arange(n_layers * W.n_seg, dtype=torch.int32, device=DEV).reshape(n_layers, W.n_seg)
    S_out = torch.empty((n_layers, W.h_v, 128, 128), device=DEV)
    seam_out = torch.zeros((n_layers, W.n_seg, W.seam_w, W.h_v, 128), device=DEV) if W.seam_w else None
    hy.compose(slot, T_pool, S_pool, sa["k"], sa["v"], sa["q"], sa["g"], sa["beta"], variant=W.variant,
               S_out=S_out, seam_out=seam_out, S_init=S_init, status=status)
    torch.cuda.synchronize()
    return T_pool, S_pool, sa, slot, S_out, seam_out


def _oracle_compose(W, T_pool, S_pool, sa, slot, S_init, n_layers):
    sl = slot.long().cpu()
    Tp = dense_T(W.variant, T_pool, 128)[sl.numpy()]   # [L, n_seg, h_v, 128, 128]
    Sp = S_pool.cpu()[sl]
    outs = []
    for l in range(n_layers):
        g = sa["g"][l:l + 1].cpu() if sa["g"] is not None else None
        b = sa["beta"][l:l + 1].cpu() if sa["beta"] is not None else None
        S0 = None if S_init is None else S_init[l:l + 1].cpu()
        outs.append(oracle.compose(W.variant, Tp[l:l + 1], Sp[l:l + 1], sa["k"][l:l + 1].cpu(),
                                   sa["v"][l:l + 1].cpu(), sa["q"][l:l + 1].cpu(), g, b, W.h_k, W.h_v,
                                   S_init=S0))
    return np.concatenate([o[0] for o in outs]), np.concatenate([o[1] for o in outs])


@pytest.mark.parametrize("variant", ["gdn", "deltanet", "channel"])
@pytest.mark.parametrize("w", [0, 3, 8, 11])
def test_compose_tc_parity(variant, w):
    lens = [40, 130, 12, 64, 300, 25]
    W = si.workload(5, device=DEV, variant=variant, lengths=lens, h_k=2, h_v=4, seam_w=w, n_layers=2)
    S_init = si.random_state((2, W.h_v, 128, 128), seed=0, cfg=5, device=DEV)
    T_pool, S_pool, sa, slot, S_out, seam_out = _run(W, 2, S_init=S_init)
    So, seam = _oracle_compose(W, T_pool, S_pool, sa, slot, S_init, 2)
    assert per_head_rel_err(S_out, So).max() <= TOL_BF16
    if w:
        e = per_head_rel_err(seam_out.permute(0, 3, 1, 2, 4).reshape(2, W.h_v, -1),
                             np.transpose(seam, (0, 3, 1, 2, 4)).reshape(2, W.h_v, -1), inner=1)
        assert e.max() <= TOL_BF16, e.max()


@pytest.mark.parametrize("variant", ["deltanet", "channel"])
def test_compose_tc_bad_slot_reported_and_skipped(variant):
    W = si.workload(5, device=DEV, variant=variant, lengths=[30, 40, 50, 60], h_k=1, h_v=4, seam_w=8)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    slot = torch.tensor([[0, 99, 2, 3]], dtype=torch.int32, device=DEV)
    T_pool, S_pool, sa, _, S_out, seam_out = _run(W, 1, status=status, slot=slot)
    assert hy.status_from_word(int(status.item())) == 7   # HYPIC_ERR_BAD_SLOT
    # the chain skipped the bad pair: same as composing with (I, 0) there
    T2 = T_pool.clone()
    S2 = S_pool.clone()
    T2[1] = torch.eye(128, device=DEV)
    S2[1] = 0
    ok_slot = torch.tensor([[0, 1, 2, 3]], dtype=torch.int32, device=DEV)
    ref = torch.empty_like(S_out)
    hy.compose(ok_slot, T2, S2, sa["k"], sa["v"], sa["q"], sa["g"], sa["beta"], variant=variant, S_out=ref,
               seam_out=torch.empty_like(seam_out))
    torch.cuda.synchronize()
    assert per_head_rel_err(S_out, ref).max() <= TOL_BF16


_TIMEOUT_CHILD = r"""
import sys, torch
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + '/tests')
import synth_inputs as si
import hybrid_linear_attention_chunkwise_gb300 as hy
from gpu_common import dense_T, gpu_build, seam_arrays
W = si.workload(5, device='cuda', variant='gdn', lengths=[40, 70, 33], h_k=1, h_v=4, seam_w=8)
T, S = gpu_build(W)
torch.cuda.synchronize()
sa = seam_arrays(W)
status = torch.zeros(1, dtype=torch.int32, device='cuda')
slot = torch.arange(3, dtype=torch.int32, device='cuda')[None]
out = torch.empty((1, 4, 128, 128), device='cuda')
so = torch.empty((1, 3, 8, 4, 128), device='cuda')
hy.compose(slot, T, S, sa['k'], sa['v'], sa['q'], sa['g'], sa['beta'], variant='gdn', S_out=out, seam_out=so,
           status=status)
torch.cuda.synchronize()
code = hy.status_from_word(int(status.item()))
x = torch.ones(4, device='cuda').sum().item()   # the context is still usable
print('STATUS', code, 'CTX', x)
"""


def test_compose_tc_bounded_wait_reports_timeout():
    """The debug stall makes every CTA wait on an mbarrier that nothing ever
    signals, with a short poll limit: the wait runs out, the kernel reports
    HYPIC_ERR_TIMEOUT through the status word, drains its copies and returns;
    nothing spins and the context stays usable."""
    env = dict(os.environ, HYPIC_DEBUG_WAIT_LIMIT="2000", HYPIC_DEBUG_STALL="1")
    r = subprocess.run([sys.executable, "-c", _TIMEOUT_CHILD, ROOT], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("STATUS")][-1]
    assert line.split()[1] == "5" and line.split()[3] == "4.0", line


@pytest.mark.parametrize("variant", ["deltanet", "gdn"])
def test_compose_tc_long_chain(variant):
    """100 lognormal segments (the warm-prompt length law), w = 8, random
    S_init.  With alpha = 1 (DeltaNet) T_C stays of order one, so the
    tensor-core rounding of T_C and of the state enters all 100 products of
    the chain; the error must stay within the bf16 bar at the far end."""
    W = si.workload(4, device=DEV, variant=variant, n_layers=1, h_k=1, h_v=4)
    S_init = si.random_state((1, W.h_v, 128, 128), seed=1, cfg=4, device=DEV)
    T_pool, S_pool, sa, slot, S_out, seam_out = _run(W, 1, S_init=S_init)
    So, seam = _oracle_compose(W, T_pool, S_pool, sa, slot, S_init, 1)
    e1 = per_head_rel_err(S_out, So).max()
    e2 = per_head_rel_err(seam_out.permute(0, 3, 1, 2, 4).reshape(1, W.h_v, -1),
                          np.transpose(seam, (0, 3, 1, 2, 4)).reshape(1, W.h_v, -1), inner=1).max()
    print(f"{variant} 100-segment chain: state {e1:.2e}, seam outputs {e2:.2e}")
    assert e1 <= TOL_BF16 and e2 <= TOL_BF16, (e1, e2)


def _chains(variant, w, n_layers=2, lens=(40, 130, 12, 64, 300, 25, 90)):
    cfg = 2 if variant == "scalar" else 5
    W = si.workload(cfg, device=DEV, variant=variant, lengths=list(lens), h_k=2, h_v=4, seam_w=w, n_layers=n_layers)
    pools = [gpu_build(W, layer=l) for l in range(n_layers)]
    T_pool = torch.cat([p[0] for p in pools])
    S_pool = torch.cat([p[1] for p in pools])
    sa = seam_arrays(W, range(n_layers))
    slot = torch.arange(n_layers * W.n_seg, dtype=torch.int32, device=DEV).reshape(n_layers, W.n_seg)
    return W, T_pool, S_pool, sa, slot


@pytest.mark.parametrize("variant", ["gdn", "deltanet", "channel", "scalar", "diag"])
@pytest.mark.parametrize("w,bounds", [(8, [0, 4, 7]), (8, [0, 2, 5, 7]), (3, [0, 1, 2, 3, 5, 7]), (0, [0, 2, 4, 6, 7]),
                                      (8, [0, 3, 3, 7]), (8, [0, 7])])
def test_compose_spans_vs_oracle(variant, w, bounds):
    """Segment parallelism through the C ABI (hypic_compose_spans): each
    span's pair from two composes of its own segments (S from zero, T by
    the transition-only compose from the identity), the span start states by
    the exclusive scan, each span composed from its start state.  Equals the
    oracle composition (final state and every seam output) to the bf16 bar,
    like the one-pass compose; an empty span and a single span included."""
    W, T_pool, S_pool, sa, slot = _chains(variant, w)
    S_init = si.random_state((2, W.h_v, 128, 128), seed=1, cfg=5, device=DEV)
    S_out = torch.empty((2, W.h_v, 128, 128), device=DEV)
    seam_out = torch.zeros((2, W.n_seg, w, W.h_v, 128), device=DEV) if w else None
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    hy.compose_spans(slot, T_pool, S_pool, sa["k"], sa["v"], sa["q"], sa["g"], sa["beta"], variant=variant,
                     S_out=S_out, seam_out=seam_out, S_init=S_init, bounds=bounds, h_k=W.h_k, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, hy.status_from_word(int(status.item()))
    So, seam = _oracle_compose(W, T_pool, S_pool, sa, slot, S_init, 2)
    assert per_head_rel_err(S_out, So).max() <= TOL_BF16
    if w:
        e = per_head_rel_err(seam_out.permute(0, 3, 1, 2, 4).reshape(2, W.h_v, -1),
                             np.transpose(seam, (0, 3, 1, 2, 4)).reshape(2, W.h_v, -1), inner=1)
        assert e.max() <= TOL_BF16, e.max()


@pytest.mark.parametrize("variant", ["gdn", "deltanet", "channel", "scalar", "diag"])
def test_transition_only_compose_is_the_product_of_transitions(variant):
    """HYPIC_FLAG_TRANSITION_ONLY from the identity gives the transition of
    the whole chain: the oracle composition of the same pairs and seam tokens
    with every write (v, S(C|0)) set to zero, from S_init = I."""
    W, T_pool, S_pool, sa, slot = _chains(variant, 8)
    T_out = torch.empty((2, W.h_v, 128, 128), device=DEV)
    hy.compose(slot, T_pool, None, sa["k"], sa["v"], sa["q"], sa["g"], sa["beta"], variant=variant, S_out=T_out,
               seam_out=None, flags=hy.FLAG_TRANSITION_ONLY, h_k=W.h_k)
    torch.cuda.synchronize()
    eye = torch.eye(128).expand(2, W.h_v, 128, 128).contiguous()
    zero_v = {**sa, "v": torch.zeros_like(sa["v"])}
    So, _ = _oracle_compose(W, T_pool, torch.zeros_like(S_pool), zero_v, slot, eye, 2)
    assert per_head_rel_err(T_out, So).max() <= TOL_BF16


def test_span_scan_vs_oracle_merges():
    """hypic_span_scan: S_start[s] = T_{s-1} S_start[s-1] + S_{s-1}, against
    the oracle merge of the same fp32 pairs, 5 spans x 3 layers x 4 heads."""
    gen = torch.Generator(device="cpu").manual_seed(9)
    n_sp, L, H = 5, 3, 4
    T = (torch.randn(n_sp, L, H, 128, 128, generator=gen, dtype=torch.float64) / np.sqrt(128)).float()
    S = torch.randn(n_sp, L, H, 128, 128, generator=gen, dtype=torch.float64).float()
    S0 = torch.randn(L, H, 128, 128, generator=gen, dtype=torch.float64).float()
    out = torch.empty((n_sp, L, H, 128, 128), device=DEV)
    hy.span_scan(T.to(DEV), S.to(DEV), out, S_init=S0.to(DEV))
    torch.cuda.synchronize()
    ref = [S0.numpy().astype(np.float64)]
    for s in range(1, n_sp):
        _, nxt = oracle.merge(T[s - 1].numpy(), S[s - 1].numpy(), T[s - 1].numpy(), ref[-1])
        ref.append(nxt)
    for s in range(n_sp):
        assert per_head_rel_err(out[s].cpu(), ref[s]).max() <= TOL_BF16, s


def test_compose_channel_steep_gates():
    """Per-channel gates: a few channels decay below e^-80 over a seam group
    (those groups take the exact-state path), the rest stay mild (fused with
    the pair); both against the oracle composing the same fp32 pairs."""
    lens = [40, 130, 64, 300, 25, 90]
    W = si.workload(5, device=DEV, variant="channel", lengths=lens, h_k=2, h_v=4, seam_w=8)
    pools = [gpu_build(W)]
    T_pool, S_pool = pools[0]
    sa = seam_arrays(W, [0])
    g = sa["g"].clone()
    g[0, 1::2, :, :, 5::17] *= 40.0  # odd segments: a few channels decay steeply
    S_init = si.random_state((1, W.h_v, 128, 128), seed=2, cfg=5, device=DEV)
    slot = torch.arange(W.n_seg, dtype=torch.int32, device=DEV).reshape(1, W.n_seg)
    S_out = torch.empty((1, W.h_v, 128, 128), device=DEV)
    seam_out = torch.zeros((1, W.n_seg, W.seam_w, W.h_v, 128), device=DEV)
    hy.compose(slot, T_pool, S_pool, sa["k"], sa["v"], sa["q"], g, sa["beta"], variant="channel", S_out=S_out,
               seam_out=seam_out, S_init=S_init)
    torch.cuda.synchronize()
    So, seam = oracle.compose("channel", T_pool.cpu()[None], S_pool.cpu()[None], sa["k"].cpu(), sa["v"].cpu(),
                              sa["q"].cpu(), g.cpu(), sa["beta"].cpu(), W.h_k, W.h_v, S_init=S_init.cpu())
    assert per_head_rel_err(S_out, So).max() <= TOL_BF16
    e = per_head_rel_err(seam_out.permute(0, 3, 1, 2, 4).reshape(1, W.h_v, -1),
                         np.transpose(seam, (0, 3, 1, 2, 4)).reshape(1, W.h_v, -1), inner=1)
    assert e.max() <= TOL_BF16, e.max()


@pytest.mark.parametrize("variant", ["gdn", "channel", "scalar"])
def test_compose_of_no_segment_passes_the_state_through(variant):
    """A chain with no segment (an empty span of a longer prompt) returns
    S_init unchanged, writes no seam output and reports nothing, seam window
    or not."""
    W, T_pool, S_pool, sa, slot = _chains(variant, 8)
    S_init = si.random_state((2, W.h_v, 128, 128), seed=3, cfg=5, device=DEV)
    S_out = torch.empty_like(S_init)
    seam_out = torch.full((2, W.n_seg, 8, W.h_v, 128), 7.0, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    hy.compose(slot, T_pool, S_pool, sa["k"], sa["v"], sa["q"], sa["g"], sa["beta"], variant=variant, S_out=S_out,
               seam_out=seam_out, S_init=S_init, h_k=W.h_k, status=status, span=(3, 3))
    torch.cuda.synchronize()
    assert int(status.item()) == 0, hy.status_from_word(int(status.item()))
    assert torch.equal(S_out, S_init) and torch.all(seam_out == 7.0)


def test_compose_widest_heads_on_the_tensor_cores():
    """128 value heads (the widest the tensor-core compose takes) against the
    oracle; 132 heads run the fp32 kernel, as the path query says."""
    for h_v, want in ((128, "tc_compose"), (132, "f32_compose")):
        W = si.workload(5, device=DEV, variant="gdn", lengths=[40, 90, 30], h_k=h_v // 4, h_v=h_v, seam_w=8,
                        n_layers=1)
        S_init = si.random_state((1, W.h_v, 128, 128), seed=2, cfg=5, device=DEV)
        pools = [gpu_build(W, layer=0)]
        T_pool, S_pool = pools[0]
        sa = seam_arrays(W, range(1))
        slot = torch.arange(W.n_seg, dtype=torch.int32, device=DEV).reshape(1, W.n_seg)
        args = (slot, T_pool, S_pool, sa["k"], sa["v"], sa["q"], sa["g"], sa["beta"])
        S_out = torch.empty((1, W.h_v, 128, 128), device=DEV)
        seam_out = torch.zeros((1, W.n_seg, 8, W.h_v, 128), device=DEV)
        assert hy.compose_path(*args, variant="gdn", S_out=S_out, seam_out=seam_out, S_init=S_init) == want
        hy.compose(*args, variant="gdn", S_out=S_out, seam_out=seam_out, S_init=S_init)
        torch.cuda.synchronize()
        So, seam = _oracle_compose(W, T_pool, S_pool, sa, slot, S_init, 1)
        assert per_head_rel_err(S_out, So).max() <= TOL_BF16, h_v
        e = per_head_rel_err(seam_out.permute(0, 3, 1, 2, 4).reshape(1, W.h_v, -1),
                             np.transpose(seam, (0, 3, 1, 2, 4)).reshape(1, W.h_v, -1), inner=1)
        assert e.max() <= TOL_BF16, (h_v, e.max())
