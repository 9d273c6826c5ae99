"""GPU tests of the pair merge (T2, S2) o (T1, S1) = (T2 T1, T2 S1 + S2):
against the fp64 oracle merge of the same fp32 pairs (per-head relative
Frobenius error 1e-5: the tensor-core path splits its tf32 operands), against
the build of the joined span, for every transition form, through a tree of
merges, and with bad slots."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from gpu_common import DENSE, dense_T, gpu_build, new_pools
from tolerance import TOL_BF16, per_head_rel_err
import hybrid_linear_attention_chunkwise_gb300 as hy

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_MERGE = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__ as g
    g.build()


def _i32(x):
    return torch.as_tensor(np.asarray(x, dtype=np.int32), device=DEV)


def _random_pairs(n, h_v, d, seed, contraction=True):
    """Random fp32 pairs: T with spectral scale about 1 (a product of
    contractions), S ~ N(0, 1)."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    T = torch.randn(n, h_v, d, d, generator=gen, dtype=torch.float64) / np.sqrt(d)
    if not contraction:
        T = T + torch.eye(d, dtype=torch.float64)
    S = torch.randn(n, h_v, d, d, generator=gen, dtype=torch.float64)
    return T.to(torch.float32).to(DEV), S.to(torch.float32).to(DEV)


@pytest.mark.parametrize("d", [128, 32])
def test_merge_random_pairs_vs_oracle(d):
    """Tensor-core path (d = 128) and the fp32 CUDA-core path (d = 32)."""
    T, S = _random_pairs(10, 4, d, seed=11 + d)
    later, earlier, out = [1, 3, 5, 9, 0], [0, 2, 4, 8, 7], [0, 1, 2, 3, 4]
    To = torch.full((5, 4, d, d), float("nan"), device=DEV)
    So = torch.full((5, 4, d, d), float("nan"), device=DEV)
    hy.pair_merge(_i32(later), _i32(earlier), _i32(out), T, S, To, So, variant="deltanet")
    torch.cuda.synchronize()
    Tc, Sc = T.cpu().numpy(), S.cpu().numpy()
    Tr, Sr = oracle.merge(Tc[later], Sc[later], Tc[earlier], Sc[earlier])
    eT = per_head_rel_err(To.cpu(), Tr).max()
    eS = per_head_rel_err(So.cpu(), Sr).max()
    assert eT <= TOL_MERGE and eS <= TOL_MERGE, (eT, eS)


@pytest.mark.parametrize("variant", DENSE)
def test_merge_equals_build_of_joined_span(variant):
    """Pairs of two adjacent bodies merge into the pair of the joined body
    (no seam), to the bf16 bar against the oracle's pair of the joined body."""
    lens = [300, 200, 129, 64]
    W = si.workload(5, device=DEV, variant=variant, lengths=lens, h_k=2, h_v=4, seam_w=0)
    T_pool, S_pool = gpu_build(W)
    To, So = new_pools(variant, 2, W.h_v, W.d_k, W.d_v, DEV)
    hy.pair_merge(_i32([1, 3]), _i32([0, 2]), _i32([0, 1]), T_pool, S_pool, To, So, variant=variant)
    torch.cuda.synchronize()
    off = W.seg_offsets
    joined = np.array([0, off[2], off[4]], dtype=np.int64)
    L = W.layers[0]
    cpu = [None if x is None else x.cpu() for x in (L.k, L.v, L.g, L.beta)]
    Tj, Sj = oracle.build_pairs(variant, joined, 0, W.h_k, W.h_v, W.d_k, W.d_v, *cpu)
    eT = per_head_rel_err(To.cpu(), Tj).max()
    eS = per_head_rel_err(So.cpu(), Sj).max()
    assert eT <= TOL_BF16 and eS <= TOL_BF16, (eT, eS)
    # and, on the same GPU pairs, the oracle merge to the fp32 bar
    Tc, Sc = T_pool.cpu().numpy(), S_pool.cpu().numpy()
    Tr, Sr = oracle.merge(Tc[[1, 3]], Sc[[1, 3]], Tc[[0, 2]], Sc[[0, 2]])
    assert per_head_rel_err(To.cpu(), Tr).max() <= TOL_MERGE
    assert per_head_rel_err(So.cpu(), Sr).max() <= TOL_MERGE


@pytest.mark.parametrize("variant", ["scalar", "ungated", "diag"])
def test_merge_scalar_and_diagonal(variant):
    lens = [100, 77, 64, 300]
    if variant == "scalar":
        W = si.workload(2, device=DEV, lengths=lens, h_k=2, h_v=2, seam_w=0)
    else:
        W = si.workload(5, device=DEV, variant=variant, lengths=lens, h_k=2, h_v=2, seam_w=0)
    T_pool, S_pool = gpu_build(W)
    To, So = new_pools(variant, 2, W.h_v, W.d_k, W.d_v, DEV)
    hy.pair_merge(_i32([1, 3]), _i32([0, 2]), _i32([1, 0]), T_pool, S_pool, To, So, variant=variant)
    torch.cuda.synchronize()
    Td = dense_T(variant, T_pool, W.d_k)
    Sc = S_pool.cpu().numpy()
    Tr, Sr = oracle.merge(Td[[3, 1]], Sc[[3, 1]], Td[[2, 0]], Sc[[2, 0]])
    eT = per_head_rel_err(dense_T(variant, To, W.d_k), Tr).max()
    eS = per_head_rel_err(So.cpu(), Sr).max()
    assert eT <= TOL_MERGE and eS <= TOL_MERGE, (eT, eS)


def test_merge_tree_equals_sequential_composition():
    """Eight DeltaNet pairs merged as a balanced tree (three levels, each level
    one call into a fresh pool) equal the left-to-right oracle merge chain."""
    T, S = _random_pairs(8, 4, 128, seed=5, contraction=False)
    T = T / 1.5
    cur_T, cur_S = T, S
    n = 8
    while n > 1:
        To = torch.empty((n // 2, 4, 128, 128), device=DEV)
        So = torch.empty_like(To)
        hy.pair_merge(_i32(list(range(1, n, 2))), _i32(list(range(0, n, 2))), _i32(list(range(n // 2))),
                      cur_T, cur_S, To, So, variant="deltanet")
        cur_T, cur_S, n = To, So, n // 2
    torch.cuda.synchronize()
    Tc, Sc = T.cpu().numpy().astype(np.float64), S.cpu().numpy().astype(np.float64)
    accT, accS = Tc[0], Sc[0]
    for i in range(1, 8):
        accT, accS = oracle.merge(Tc[i], Sc[i], accT, accS)
    eT = per_head_rel_err(cur_T[0].cpu(), accT).max()
    eS = per_head_rel_err(cur_S[0].cpu(), accS).max()
    assert eT <= 5 * TOL_MERGE and eS <= 5 * TOL_MERGE, (eT, eS)


def test_merge_bad_slot_is_skipped_and_reported():
    T, S = _random_pairs(4, 2, 128, seed=3)
    To = torch.full((3, 2, 128, 128), 7.0, device=DEV)
    So = torch.full_like(To, 7.0)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    hy.pair_merge(_i32([1, 9, 3]), _i32([0, 0, 2]), _i32([0, 1, 2]), T, S, To, So, variant="gdn", status=status)
    torch.cuda.synchronize()
    assert hy.status_from_word(int(status.item())) == 7  # HYPIC_ERR_BAD_SLOT
    assert torch.all(To[1] == 7.0) and torch.all(So[1] == 7.0)
    Tc, Sc = T.cpu().numpy(), S.cpu().numpy()
    Tr, Sr = oracle.merge(Tc[[1, 3]], Sc[[1, 3]], Tc[[0, 2]], Sc[[0, 2]])
    assert per_head_rel_err(To[[0, 2]].cpu(), Tr).max() <= TOL_MERGE
