"""GPU tests of the tensor-core chunkwise builds (GDN / DeltaNet and the
per-channel gated delta rule, bf16, d = 128): many items of every chunk count
(exercising the hand-off between the two warp groups across item
boundaries), gate laws that stress each kernel's exponent handling, bitwise
determinism, and the bounded-wait timeout."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_common import compare_pairs, gpu_build, oracle_pairs
from tolerance import TOL_BF16

pytestmark = pytest.mark.gpu
DEV = "cuda"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__ as g
    g.build()


@pytest.mark.parametrize("variant", ["gdn", "deltanet"])
def test_build_tc_many_lengths(variant):
    lens = [1, 2, 63, 64, 65, 127, 128, 129, 200, 257, 511, 1000, 8, 9, 16, 300]
    W = si.workload(5, device=DEV, variant=variant, lengths=lens, h_k=2, h_v=4, seam_w=8)
    T_pool, S_pool = gpu_build(W)
    T, S = oracle_pairs(W)
    eT, eS = compare_pairs(W, T_pool, S_pool, T, S, range(W.n_seg))
    assert eT <= TOL_BF16 and eS <= TOL_BF16, (eT, eS)


@pytest.mark.parametrize("variant", ["gdn", "channel"])
def test_build_tc_bitwise_deterministic(variant):
    W = si.workload(3, device=DEV, n_seg=6, seg_len=700, variant=variant)
    a = [x.clone() for x in gpu_build(W)]
    b = gpu_build(W)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_build_channel_many_lengths():
    """Per-channel gates: lengths around the 32-token chunk and the 16-token
    Gram sub-block, grouped heads, slots out of order."""
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 100, 257, 1000, 8, 9]
    W = si.workload(5, device=DEV, variant="channel", lengths=lens, h_k=2, h_v=4, seam_w=8)
    slots = np.random.default_rng(5).permutation(len(lens)).astype(np.int32)
    T_pool, S_pool = gpu_build(W, slots=slots, n_slots=len(lens))
    T, S = oracle_pairs(W)
    eT, eS = compare_pairs(W, T_pool, S_pool, T, S, range(W.n_seg), slots=slots)
    assert eT <= TOL_BF16 and eS <= TOL_BF16, (eT, eS)


def _regate(W, fn):
    """Replace the per-channel log-gates of layer 0 by fn(x), x ~ N(0, 1)
    (seeded)."""
    L = W.layers[0]
    gen = torch.Generator(device="cpu").manual_seed(1234)
    x = torch.randn(L.g.shape, generator=gen, dtype=torch.float64)
    L.g = fn(x).to(torch.float32).to(L.g.device)


def test_build_channel_weak_gates_long():
    """Log-gates near zero (-softplus(x - 6), about -0.003): the transition
    product keeps thousands of tokens alive, so rounding errors accumulate
    over the whole 8192-token body."""
    W = si.workload(5, device=DEV, variant="channel", lengths=[8192, 1500], h_k=1, h_v=2, seam_w=8)
    _regate(W, lambda x: -torch.nn.functional.softplus(x - 6.0))
    T_pool, S_pool = gpu_build(W)
    T, S = oracle_pairs(W)
    eT, eS = compare_pairs(W, T_pool, S_pool, T, S, range(W.n_seg))
    assert eT <= TOL_BF16 and eS <= TOL_BF16, (eT, eS)


def test_build_channel_steep_gates_direct_gram():
    """Log-gates 40x steeper in some token ranges: the log-decay moves by
    more than 80 inside a 16-token sub-block there, so those chunks form the
    Gram term by term; the others take the factored form.  Steep runs at the
    start of a segment's last chunks leave the rest of that chunk (whose
    Gram entries shape the final state) on ordinary gates."""
    W = si.workload(5, device=DEV, variant="channel", lengths=[300, 64, 40], h_k=1, h_v=2, seam_w=0)
    n = W.n_tokens
    scale = torch.ones(n, 1, 1, dtype=torch.float64)
    scale[40:100] = 40.0     # chunks 1-3 of segment 0
    scale[256:262] = 40.0    # head of segment 0's last full chunk
    scale[310:330] = 40.0    # inside segment 1
    scale[364:370] = 40.0    # head of segment 2's first chunk
    _regate(W, lambda x: -scale * torch.nn.functional.softplus(x))
    T_pool, S_pool = gpu_build(W)
    T, S = oracle_pairs(W)
    eT, eS = compare_pairs(W, T_pool, S_pool, T, S, range(W.n_seg))
    assert eT <= TOL_BF16 and eS <= TOL_BF16, (eT, eS)


_TIMEOUT_CHILD = r"""
import sys, torch
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + '/tests')
import synth_inputs as si
import hybrid_linear_attention_chunkwise_gb300 as hy
from gpu_common import gpu_build
W = si.workload(5, device='cuda', variant=sys.argv[2], lengths=[100, 300], h_k=1, h_v=2, seam_w=0)
status = torch.zeros(1, dtype=torch.int32, device='cuda')
gpu_build(W, status=status)
torch.cuda.synchronize()
code = hy.status_from_word(int(status.item()))
x = torch.ones(4, device='cuda').sum().item()   # the context is still usable
print('STATUS', code, 'CTX', x)
"""


@pytest.mark.parametrize("variant", ["gdn", "channel"])
def test_build_tc_bounded_wait_reports_timeout(variant):
    """Every CTA first waits on an mbarrier that nothing signals, with a short
    poll limit: the wait runs out, HYPIC_ERR_TIMEOUT comes back through the
    status word, the kernel returns and the context stays usable."""
    env = dict(os.environ, HYPIC_DEBUG_WAIT_LIMIT="2000", HYPIC_DEBUG_STALL="1")
    r = subprocess.run([sys.executable, "-c", _TIMEOUT_CHILD, ROOT, variant], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("STATUS")][-1]
    assert line.split()[1] == "5" and line.split()[3] == "4.0", line


@pytest.mark.parametrize("variant", ["scalar", "ungated", "diag"])
def test_fast_path_long_segments(variant):
    """The tensor-core fast path (no erase) over long bodies: the weighted
    sum over thousands of tokens (RetNet decays close to one keep old tokens
    alive) stays within the bf16 bar."""
    W = si.workload(5, device=DEV, variant=variant, lengths=[4100, 2049, 77], h_k=2, h_v=2, seam_w=8)
    if variant == "scalar":
        W = si.workload(2, device=DEV, lengths=[4100, 2049, 77], h_k=2, h_v=2, seam_w=8)
    T_pool, S_pool = gpu_build(W)
    T, S = oracle_pairs(W)
    eT, eS = compare_pairs(W, T_pool, S_pool, T, S, range(W.n_seg))
    assert eT <= TOL_BF16 and eS <= TOL_BF16, (eT, eS)
