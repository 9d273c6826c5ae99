"""Multi-rank runs of the package's segment-parallel orchestration on CPU
(gloo, world sizes 2 and 3): hybrid_linear_attention_chunkwise_gb300.
segment_parallel drives the ranks exactly as on GPUs, with the fp64 oracle
standing in for each rank's GPU at the kernel boundary only (build, compose,
span scan).  The cold build is LPT-scattered and its pairs sent to the
combine rank point to point; the compose is split by segments with the span
pairs all-gathered.  Both must equal the single-process oracle."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import hybrid_linear_attention_chunkwise_gb300 as hy
import oracle
import synth_inputs as si


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleKernels:
    """The kernel boundary of segment_parallel, served by the fp64 oracle on
    the CPU with the library's semantics (skipped slots, spans of the
    per-layer arrays, transition-only compose from the identity, the span
    scan).  Buffers are fp64 so that results compare at 1e-9."""

    def empty(self, shape, dtype=torch.float32):
        return torch.empty(shape, dtype=torch.float64)

    def build(self, k, v, g, beta, seg_offsets, *, variant, seam_w, T_pool, S_pool, slot_of_seg):
        T, S = oracle.build_pairs(variant, seg_offsets, seam_w, k.shape[1], v.shape[1], k.shape[2], v.shape[2], k, v,
                                  g, beta)
        for i, sl in enumerate(slot_of_seg):
            if sl != hy.SLOT_SKIP:
                T_pool[sl] = torch.from_numpy(np.asarray(T[i]))
                S_pool[sl] = torch.from_numpy(np.asarray(S[i]))

    def compose(self, slot, T_pool, S_pool, seam, *, variant, S_out, seam_out=None, S_init=None, flags=0, span=None,
                h_k=None):
        L, n_seg = slot.shape
        a, b = span if span is not None else (0, n_seg)
        trans = bool(flags & hy.FLAG_TRANSITION_ONLY)
        sl = slot[:, a:b].long()
        Tp = T_pool[sl]
        Sp = torch.zeros(Tp.shape[:-1] + (S_out.shape[-1],), dtype=torch.float64) if trans else S_pool[sl]
        cut = lambda x: None if x is None else x[:, a:b]
        v = cut(seam["v"])
        if trans:
            v = torch.zeros_like(v)
        if S_init is None:
            S_init = (torch.eye(S_out.shape[-2], dtype=torch.float64).expand(S_out.shape).contiguous() if trans
                      else torch.zeros(S_out.shape, dtype=torch.float64))
        So, outs = oracle.compose(variant, Tp, Sp, cut(seam["k"]), v, cut(seam["q"]), cut(seam["g"]),
                                  cut(seam["beta"]), seam["k"].shape[3], S_out.shape[1], S_init=S_init)
        S_out.copy_(torch.from_numpy(So))
        if seam_out is not None and not trans:
            seam_out[:, a:b] = torch.from_numpy(outs).to(seam_out.dtype)

    def span_scan(self, T_span, S_span, S_start, *, S_init=None):
        S_start[0] = 0 if S_init is None else S_init
        for s in range(1, S_start.shape[0]):
            _, nxt = oracle.merge(T_span[s - 1], S_span[s - 1], T_span[s - 1], S_start[s - 1])
            S_start[s] = torch.from_numpy(nxt)


def _layer_inputs(lens, variant, w, n_layers=1, seed=2):
    return si.workload(5, seed=seed, device="cpu", variant=variant, lengths=lens, h_k=1, h_v=2, d=16, seam_w=w,
                       dtype=torch.float32, n_layers=n_layers)


def _scatter_main(rank, world, port, lens, out_dir):
    from hybrid_linear_attention_chunkwise_gb300 import segment_parallel as sp
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        W = _layer_inputs(lens, "gdn", 8)
        L = W.layers[0]
        kern = OracleKernels()
        T_pool = S_pool = None
        if rank == 0:
            T_pool = kern.empty((W.n_seg, 2, 16, 16))
            S_pool = kern.empty((W.n_seg, 2, 16, 16))
        slots = sp.cold_build_scatter(L.k, L.v, L.g, L.beta, W.seg_offsets, variant="gdn", seam_w=8, T_pool=T_pool,
                                      S_pool=S_pool, combine_rank=0, n_groups=2, kernels=kern)
        if rank == 0:
            np.save(os.path.join(out_dir, "slots.npy"), slots)
            np.save(os.path.join(out_dir, "T.npy"), T_pool.numpy())
            np.save(os.path.join(out_dir, "S.npy"), S_pool.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_cold_build_scatter_equals_single_process(tmp_path, world):
    """segment_parallel.cold_build_scatter: LPT shards over the ranks, each
    rank builds its share in groups and sends the group's pairs to rank 0,
    whose pool then holds every segment's pair exactly once."""
    lens = [130, 64, 200, 9, 77, 300, 40, 151, 500, 33]
    mp.start_processes(_scatter_main, args=(world, _free_port(), lens, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    slots = np.load(tmp_path / "slots.npy")
    assert sorted(slots.tolist()) == list(range(len(lens)))
    W = _layer_inputs(lens, "gdn", 8)
    L = W.layers[0]
    T, S = oracle.build_pairs("gdn", W.seg_offsets, 8, 1, 2, 16, 16, L.k, L.v, L.g, L.beta)
    assert np.array_equal(np.load(tmp_path / "T.npy")[slots], np.asarray(T))
    assert np.array_equal(np.load(tmp_path / "S.npy")[slots], np.asarray(S))
    # the plan: LPT shards, rank-major slots
    from hybrid_linear_attention_chunkwise_gb300 import segment_parallel as sp
    shards, groups, sl = sp.build_plan(W.seg_offsets, 8, world, 2)
    assert np.array_equal(sl, slots)
    bodies = np.maximum(np.diff(W.seg_offsets) - 8, 0)
    assert [int(bodies[s].sum()) for s in shards] == [int(bodies[s].sum()) for s in hy.shard_lpt(bodies, world)]


def _compose_main(rank, world, port, lens, w, variant, out_dir):
    from hybrid_linear_attention_chunkwise_gb300 import segment_parallel as sp
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        W = _layer_inputs(lens, variant, w, n_layers=2, seed=3)
        T_pool, S_pool, seam, slot = _chain_pools(W, variant)
        S_init = si.random_state((2, 2, 16, 16), seed=0, cfg=5).double()
        S_out = torch.empty((2, 2, 16, 16), dtype=torch.float64)
        seam_out = torch.zeros((2, W.n_seg, w, 2, 16), dtype=torch.float64)
        a, b = sp.compose_sharded(slot, T_pool, S_pool, seam, variant=variant, S_out=S_out, seam_out=seam_out,
                                  S_init=S_init, kernels=OracleKernels())
        got = [None] * world
        dist.all_gather_object(got, (a, b, S_out.numpy(), seam_out[:, a:b].numpy()))
        if rank == 0:
            np.save(os.path.join(out_dir, "S_final.npy"), got[-1][2])
            np.save(os.path.join(out_dir, "outs.npy"), np.concatenate([g[3] for g in got], axis=1))
            np.save(os.path.join(out_dir, "spans.npy"), np.array([[g[0], g[1]] for g in got]))
    finally:
        dist.destroy_process_group()


def _chain_pools(W, variant):
    """fp64 pairs of both layers in one pool (slot l * n_seg + i) and the
    stacked seam tokens."""
    Ts, Ss, seams = [], [], []
    for lay in W.layers:
        T, S = oracle.build_pairs(variant, W.seg_offsets, W.seam_w, 1, 2, 16, 16, lay.k, lay.v, lay.g, lay.beta)
        Ts.append(torch.from_numpy(np.asarray(T)))
        Ss.append(torch.from_numpy(np.asarray(S)))
        seams.append(si.seam_gather(W, lay))
    seam = {k: (torch.stack([s[k] for s in seams]) if seams[0][k] is not None else None)
            for k in ("k", "v", "q", "g", "beta")}
    slot = torch.arange(2 * W.n_seg, dtype=torch.int32).reshape(2, W.n_seg)
    return torch.cat(Ts), torch.cat(Ss), seam, slot


@pytest.mark.parametrize("world,variant,w", [(2, "deltanet", 4), (3, "gdn", 8), (2, "channel", 3)])
def test_compose_sharded_equals_single_chain(tmp_path, world, variant, w):
    """segment_parallel.compose_sharded: one span per rank, span pairs from
    two composes (S from zero, T transition-only), all-gathered, scanned;
    each rank composes its span from its start state.  The last rank's state
    and the seam outputs of every span equal the single oracle compose."""
    lens = [130, 64, 200, 9, 77, 300, 40]
    mp.start_processes(_compose_main, args=(world, _free_port(), lens, w, variant, str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    W = _layer_inputs(lens, variant, w, n_layers=2, seed=3)
    T_pool, S_pool, seam, slot = _chain_pools(W, variant)
    S0 = si.random_state((2, 2, 16, 16), seed=0, cfg=5).double()
    Sf, outs = oracle.compose(variant, T_pool[slot.long()], S_pool[slot.long()], seam["k"], seam["v"], seam["q"],
                              seam["g"], seam["beta"], 1, 2, S_init=S0)
    spans = np.load(tmp_path / "spans.npy")
    assert spans[0][0] == 0 and spans[-1][1] == len(lens) and all(spans[i][1] == spans[i + 1][0]
                                                                  for i in range(world - 1))
    got_S = np.load(tmp_path / "S_final.npy")
    assert np.abs(got_S - Sf).max() <= 1e-9 * max(1.0, np.abs(Sf).max())
    got_o = np.load(tmp_path / "outs.npy")
    assert np.abs(got_o - outs).max() <= 1e-9 * max(1.0, np.abs(outs).max())


def test_lpt_shards_are_a_partition():
    costs = np.array([700, 10, 300, 300, 90, 4000, 8, 1000, 1000, 50])
    for world in (1, 2, 3, 8):
        sh = hy.shard_lpt(costs, world)
        allidx = np.concatenate(sh)
        assert sorted(allidx.tolist()) == list(range(len(costs)))
        loads = [int(costs[s].sum()) for s in sh]
        opt_lb = max(costs.max(), costs.sum() / world)
        assert max(loads) <= (4 / 3 - 1 / (3 * world)) * opt_lb + 1e-9 or max(loads) == costs.max()


