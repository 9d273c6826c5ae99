"""GPU tests of the state re-rotation of cached pairs (RoPE-shifted reuse):
against the fp64 oracle on the same fp32 pairs (both channel pairings, full
and partial rotary dim, shifts up to 10^6 positions, scalar T passed
through), in place against out of place, bad slots, and the rotated-key
identity end to end: a GPU build from rotated fp32 keys equals the GPU
re-rotation of the GPU pair of the original keys."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from gpu_common import gpu_build, new_pools
from tolerance import TOL_F32, per_head_rel_err
import hybrid_linear_attention_chunkwise_gb300 as hy

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_ROT = 1e-6  # fp32 inputs and outputs, two fp32 products per element


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__ as g
    g.build()


def _i32(x):
    return torch.as_tensor(np.asarray(x, dtype=np.int32), device=DEV)


def _i64(x):
    return torch.as_tensor(np.asarray(x, dtype=np.int64), device=DEV)


def _pools(variant, n, h_v, d_k, d_v, seed):
    gen = torch.Generator(device="cpu").manual_seed(seed)
    S = torch.randn(n, h_v, d_k, d_v, generator=gen, dtype=torch.float64).to(torch.float32)
    if variant in ("gdn", "deltanet"):
        T = (torch.randn(n, h_v, d_k, d_k, generator=gen, dtype=torch.float64) / np.sqrt(d_k)).to(torch.float32)
    else:
        T = torch.rand(n, h_v, generator=gen, dtype=torch.float64).to(torch.float32)
    return T.to(DEV), S.to(DEV)


CASES = [("gdn", "interleaved", 128, 128, 128), ("gdn", "half", 128, 128, 128), ("deltanet", "half", 64, 128, 128),
         ("deltanet", "interleaved", 32, 128, 128), ("gdn", "interleaved", 48, 64, 96), ("scalar", "half", 128, 128, 128),
         ("ungated", "interleaved", 16, 32, 16)]


@pytest.mark.parametrize("variant,layout,rot,d_k,d_v", CASES)
def test_rerotate_vs_oracle(variant, layout, rot, d_k, d_v):
    h_v = 6  # not a multiple of the eight heads a CTA takes
    T, S = _pools(variant, 5, h_v, d_k, d_v, seed=rot + d_k)
    deltas = [0, 1, -37, 1000003, -999983]
    slot_in, slot_out = [4, 0, 2, 1, 3], [0, 1, 2, 3, 4]
    To, So = new_pools(variant, 5, h_v, d_k, d_v, DEV)
    hy.pair_rerotate(_i32(slot_in), _i32(slot_out), _i64(deltas), T, S, To, So, variant=variant, rot_dim=rot,
                     layout=layout, base=10000.0)
    torch.cuda.synchronize()
    Tr, Sr = oracle.rerotate(variant, T.cpu().numpy()[slot_in], S.cpu().numpy()[slot_in], deltas, rot, layout,
                             10000.0)
    eS = per_head_rel_err(So.cpu(), Sr).max()
    if variant in ("gdn", "deltanet"):
        eT = per_head_rel_err(To.cpu(), Tr).max()
    else:
        eT = float(np.abs(To.cpu().numpy() - Tr).max())  # copied bit for bit
        assert eT == 0.0
    assert eT <= TOL_ROT and eS <= TOL_ROT, (eT, eS)


def test_rerotate_in_place_equals_out_of_place():
    T, S = _pools("gdn", 4, 8, 128, 128, seed=9)
    deltas = _i64([5, -5, 123456, 7])
    slots = _i32([0, 1, 2, 3])
    To, So = new_pools("gdn", 4, 8, 128, 128, DEV)
    hy.pair_rerotate(slots, slots, deltas, T, S, To, So, variant="gdn", rot_dim=128, layout="half")
    T2, S2 = T.clone(), S.clone()
    hy.pair_rerotate(slots, slots, deltas, T2, S2, T2, S2, variant="gdn", rot_dim=128, layout="half")
    torch.cuda.synchronize()
    assert torch.equal(T2, To) and torch.equal(S2, So)


def test_rerotate_bad_slot_is_skipped_and_reported():
    T, S = _pools("deltanet", 3, 4, 128, 128, seed=1)
    To = torch.full_like(T, 7.0)
    So = torch.full_like(S, 7.0)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    hy.pair_rerotate(_i32([0, 5, 2]), _i32([0, 1, 2]), _i64([3, 3, 3]), T, S, To, So, variant="deltanet",
                     rot_dim=128, status=status)
    torch.cuda.synchronize()
    assert hy.status_from_word(int(status.item())) == 7  # HYPIC_ERR_BAD_SLOT
    assert torch.all(To[1] == 7.0) and torch.all(So[1] == 7.0)
    Tr, Sr = oracle.rerotate("deltanet", T.cpu().numpy()[[0, 2]], S.cpu().numpy()[[0, 2]], [3, 3], 128)
    assert per_head_rel_err(So[[0, 2]].cpu(), Sr).max() <= TOL_ROT


@pytest.mark.parametrize("variant", ["gdn", "deltanet", "scalar"])
def test_rotated_key_build_equals_rerotated_pair(variant):
    """End to end on the GPU: segments whose keys are rotated by R(delta_i)
    build (fp32 inputs) into the re-rotated pairs of the original keys."""
    lens = [70, 129, 33, 200]
    W = si.workload(2 if variant == "scalar" else 5, device=DEV, variant=variant, lengths=lens, h_k=2, h_v=4,
                    seam_w=0, dtype=torch.float32)
    T0, S0 = gpu_build(W)
    deltas = [11, -400, 0, 54321]
    L = W.layers[0]
    k = L.k.detach().cpu().double().numpy()
    off = W.seg_offsets
    for i, dl in enumerate(deltas):
        R = oracle.rerotation_matrix(W.d_k, dl, 64, "half")
        k[off[i]:off[i + 1]] = np.einsum("ab,thb->tha", R, k[off[i]:off[i + 1]])
    L.k = torch.as_tensor(k, dtype=torch.float32, device=DEV)
    T1, S1 = gpu_build(W)
    slots = _i32(range(len(lens)))
    To, So = new_pools(variant, len(lens), W.h_v, W.d_k, W.d_v, DEV)
    hy.pair_rerotate(slots, slots, _i64(deltas), T0, S0, To, So, variant=variant, rot_dim=64, layout="half")
    torch.cuda.synchronize()
    assert per_head_rel_err(So.cpu(), S1.cpu().double().numpy()).max() <= TOL_F32
    if variant != "scalar":
        assert per_head_rel_err(To.cpu(), T1.cpu().double().numpy()).max() <= TOL_F32
