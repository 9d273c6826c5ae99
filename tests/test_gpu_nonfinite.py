"""GPU tests: a non-finite value in a cached pair survives compose and the
pair merge, and the finite check reports it.

The composition rule (nav.aitube.vip §2.1: S(C1.C2) = T(C2) S(C1) + S(C2))
is exact, so a corrupted cached pair must give a corrupted state, never a
clean-looking one.  The NaN planted here is the all-ones pattern
0x7FFFFFFF that fp32 arithmetic on the GPU produces; rounding it to a
tensor-core operand by adding half a unit would carry into the sign bit and
give -0.0.  The planted values go in on the host side of the test (a write
into the pool tensors); no kernel is made to fault.

The oracle composes / merges the same corrupted fp32 pairs in fp64; the
non-finite elements of the GPU result must be exactly those of the oracle
where the corruption stays confined to one state column (a value planted in
S), and must cover them where it spreads (a value planted in T)."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from gpu_common import gpu_build, seam_arrays
from tolerance import TOL_BF16
import hybrid_linear_attention_chunkwise_gb300 as hy

pytestmark = pytest.mark.gpu
DEV = "cuda"
NAN_ALL_ONES = 0x7FFFFFFF
INF_BITS = 0x7F800000


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__ as g
    g.build()


def _plant(pool, index, bits):
    pool.view(torch.int32)[index] = bits if bits < 2 ** 31 else bits - 2 ** 32


def _finite_close(x, ref, mask):
    """Elements finite in both: within the bf16 bar relative to the finite
    part of the reference."""
    x = np.where(mask, 0.0, x)
    ref = np.where(mask, 0.0, ref)
    den = np.linalg.norm(ref)
    return np.linalg.norm(x - ref) <= TOL_BF16 * max(den, 1e-30)


def _compose_chain(variant, where, bits):
    """10-segment chain, 4 value heads (the tensor-core compose), with one
    value planted in the pair of segment 4: `where` = "S" or "T"."""
    lens = [60, 90, 40, 130, 75, 50, 110, 64, 33, 80]
    W = si.workload(5, device=DEV, variant=variant, lengths=lens, h_k=2, h_v=4, seam_w=8)
    T_pool, S_pool = gpu_build(W)
    h, i, j = 2, 17, 45
    if where == "S":
        _plant(S_pool, (4, h, i, j), bits)
    else:
        _plant(T_pool, (4, h, i, j), bits)
    sa = seam_arrays(W)
    slot = torch.arange(W.n_seg, dtype=torch.int32, device=DEV).reshape(1, W.n_seg)
    S_out = torch.empty((1, W.h_v, 128, 128), device=DEV)
    seam_out = torch.zeros((1, W.n_seg, W.seam_w, W.h_v, 128), device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    hy.compose(slot, T_pool, S_pool, sa["k"], sa["v"], sa["q"], sa["g"], sa["beta"], variant=variant,
               S_out=S_out, seam_out=seam_out, status=status, flags=hy.FLAG_CHECK_FINITE)
    torch.cuda.synchronize()
    g = sa["g"].cpu() if sa["g"] is not None else None
    b = sa["beta"].cpu() if sa["beta"] is not None else None
    So, seam = oracle.compose(variant, T_pool.cpu()[None], S_pool.cpu()[None], sa["k"].cpu(), sa["v"].cpu(),
                              sa["q"].cpu(), g, b, W.h_k, W.h_v)
    return status, S_out.cpu().double().numpy(), seam_out.cpu().double().numpy(), So, seam, h, j


@pytest.mark.parametrize("variant", ["gdn", "deltanet", "channel"])
@pytest.mark.parametrize("bits", [NAN_ALL_ONES, INF_BITS], ids=["nan", "inf"])
def test_compose_nonfinite_state_column_survives(variant, bits):
    status, S, seam, So, seam_ref, h, j = _compose_chain(variant, "S", bits)
    assert hy.status_from_word(int(status.item())) == 6  # HYPIC_ERR_NONFINITE
    bad_ref, bad = ~np.isfinite(So), ~np.isfinite(S)
    assert bad_ref.any()
    # the corrupted state column of head h, and nothing else
    assert np.array_equal(bad, bad_ref), (np.argwhere(bad != bad_ref)[:5])
    assert bad[0, h, :, j].all() and not np.delete(bad[0, h], j, axis=1).any()
    assert _finite_close(S, So, bad_ref)
    sbad_ref, sbad = ~np.isfinite(seam_ref), ~np.isfinite(seam)
    assert np.array_equal(sbad, sbad_ref)
    assert _finite_close(seam, seam_ref, sbad_ref)


@pytest.mark.parametrize("variant", ["gdn", "deltanet"])
@pytest.mark.parametrize("bits", [NAN_ALL_ONES, INF_BITS], ids=["nan", "inf"])
def test_compose_nonfinite_transition_spreads(variant, bits):
    status, S, seam, So, seam_ref, h, j = _compose_chain(variant, "T", bits)
    assert hy.status_from_word(int(status.item())) == 6  # HYPIC_ERR_NONFINITE
    bad_ref, bad = ~np.isfinite(So), ~np.isfinite(S)
    assert bad_ref[0, h].all()
    assert np.all(bad[bad_ref])
    assert not bad[0, np.arange(4) != h].any()


def test_compose_nonfinite_reported_on_a_middle_segment_only():
    """A NaN that only lives through part of the chain still reports: the
    pair of segment 4 has a NaN in S while every later pair is finite, and
    the check runs after every segment."""
    status, *_ = _compose_chain("deltanet", "S", NAN_ALL_ONES)
    assert int(status.item()) & hy.STATUS_NONFINITE


def _pairs(n, h_v, seed):
    gen = torch.Generator(device="cpu").manual_seed(seed)
    T = torch.randn(n, h_v, 128, 128, generator=gen, dtype=torch.float64) / np.sqrt(128)
    S = torch.randn(n, h_v, 128, 128, generator=gen, dtype=torch.float64)
    return T.to(torch.float32).to(DEV), S.to(torch.float32).to(DEV)


@pytest.mark.parametrize("operand,bits", [("T_b", NAN_ALL_ONES), ("S_b", NAN_ALL_ONES), ("S_b", INF_BITS),
                                          ("T_a", NAN_ALL_ONES), ("T_a", INF_BITS), ("S_a", NAN_ALL_ONES)])
def test_merge_nonfinite_operand_survives(operand, bits):
    """One non-finite element in one operand of one merge: the output is
    non-finite wherever the fp64 oracle merge of the same pairs is, and the
    other merges of the call are untouched."""
    T, S = _pairs(4, 4, seed=21)
    h, r, c = 1, 70, 33
    later, earlier = 1, 0  # merge 0: (T1, S1) o (T0, S0); merge 1: (T3, S3) o (T2, S2)
    target = {"T_b": (T, earlier), "S_b": (S, earlier), "T_a": (T, later), "S_a": (S, later)}[operand]
    _plant(target[0], (target[1], h, r, c), bits)
    To = torch.empty((2, 4, 128, 128), device=DEV)
    So = torch.empty_like(To)
    i32 = lambda x: torch.as_tensor(np.asarray(x, np.int32), device=DEV)
    hy.pair_merge(i32([1, 3]), i32([0, 2]), i32([0, 1]), T, S, To, So, variant="deltanet")
    torch.cuda.synchronize()
    Tc, Sc = T.cpu().numpy(), S.cpu().numpy()
    Tr, Sr = oracle.merge(Tc[[1, 3]], Sc[[1, 3]], Tc[[0, 2]], Sc[[0, 2]])
    Tg, Sg = To.cpu().double().numpy(), So.cpu().double().numpy()
    for got, ref in ((Tg, Tr), (Sg, Sr)):
        bad_ref, bad = ~np.isfinite(ref), ~np.isfinite(got)
        assert np.all(bad[bad_ref])
        assert not bad[1].any() and not bad[0, np.arange(4) != h].any()
    assert (~np.isfinite(Tr)).any() or (~np.isfinite(Sr)).any()
