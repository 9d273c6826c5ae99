"""World-size-2 runs of the multi-GPU host path on CPU (gloo): cold segments
are sharded over ranks by LPT with no data-path exchange, each rank builds
its shard (here with the fp64 oracle standing in for a rank's GPU), and the
union equals the single-process build; timings reduce by max over ranks."""
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


def _rank_main(rank, world, port, lens, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        W = si.workload(5, seed=2, device="cpu", variant="gdn", lengths=lens, h_k=1, h_v=2, d=16,
                        seam_w=8, dtype=torch.float32)
        costs = np.diff(W.seg_offsets) - W.seam_w
        shards = hy.shard_lpt(np.maximum(costs, 0), world)
        mine = shards[rank]
        # build this rank's segments only (the oracle stands in for the GPU)
        L = W.layers[0]
        sub_lens = [int(lens[i]) for i in mine]
        idx = np.concatenate([np.arange(W.seg_offsets[i], W.seg_offsets[i + 1]) for i in mine])
        T, S = oracle.build_pairs("gdn", si.offsets_from_lengths(sub_lens), W.seam_w, 1, 2, 16, 16,
                                  L.k[idx], L.v[idx], L.g[idx], L.beta[idx])
        # gather every rank's shard and pairs on rank 0
        got = [None] * world
        dist.all_gather_object(got, (mine.tolist(), np.asarray(T), np.asarray(S)))
        # max over ranks of a per-rank time, as the bench reports it
        t = torch.tensor([float(rank + 1)])
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        if rank == 0:
            np.save(os.path.join(out_dir, "tmax.npy"), t.numpy())
            T_all = np.zeros((len(lens), 2, 16, 16))
            S_all = np.zeros((len(lens), 2, 16, 16))
            seen = []
            for segs, Tr, Sr in got:
                for j, i in enumerate(segs):
                    T_all[i], S_all[i] = Tr[j], Sr[j]
                    seen.append(i)
            np.save(os.path.join(out_dir, "seen.npy"), np.array(seen))
            np.save(os.path.join(out_dir, "T.npy"), T_all)
            np.save(os.path.join(out_dir, "S.npy"), S_all)
    finally:
        dist.destroy_process_group()


def test_lpt_shards_are_a_partition():
    costs = np.array([700, 10, 300, 300, 90, 4000, 8, 1000, 1000, 50])
    for world in (1, 2, 3, 8):
        sh = hy.shard_lpt(costs, world)
        allidx = np.concatenate(sh)
        assert sorted(allidx.tolist()) == list(range(len(costs)))
        loads = [int(costs[s].sum()) for s in sh]
        opt_lb = max(costs.max(), costs.sum() / world)
        assert max(loads) <= (4 / 3 - 1 / (3 * world)) * opt_lb + 1e-9 or max(loads) == costs.max()


def test_two_rank_sharded_build_equals_single_process(tmp_path):
    lens = [130, 64, 200, 9, 77, 300, 40, 151]
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, lens, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    seen = np.load(tmp_path / "seen.npy")
    assert sorted(seen.tolist()) == list(range(len(lens)))
    assert float(np.load(tmp_path / "tmax.npy")[0]) == 2.0
    W = si.workload(5, seed=2, device="cpu", variant="gdn", lengths=lens, h_k=1, h_v=2, d=16, seam_w=8,
                    dtype=torch.float32)
    L = W.layers[0]
    T, S = oracle.build_pairs("gdn", W.seg_offsets, W.seam_w, 1, 2, 16, 16, L.k, L.v, L.g, L.beta)
    assert np.array_equal(np.load(tmp_path / "T.npy"), np.asarray(T))
    assert np.array_equal(np.load(tmp_path / "S.npy"), np.asarray(S))


def _span_rank_main(rank, world, port, lens, w, out_dir):
    """Segment parallelism on one chain, one span per rank: each rank forms
    its span's pair from its segments' seam-window and cached pairs, the
    span pairs are exchanged by all-gather (the one collective), each rank
    takes its start state from the exclusive scan and composes its span
    (the fp64 oracle stands in for each rank's GPU)."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        W = si.workload(5, seed=3, device="cpu", variant="deltanet", lengths=lens, h_k=1, h_v=2, d=16,
                        seam_w=w, dtype=torch.float32)
        L = W.layers[0]
        sa = si.seam_gather(W, L)
        n_seg = W.n_seg
        bounds = np.linspace(0, n_seg, world + 1).round().astype(int)
        a, b = int(bounds[rank]), int(bounds[rank + 1])
        # cached pairs of my segments' bodies
        idx = np.concatenate([np.arange(W.seg_offsets[i], W.seg_offsets[i + 1]) for i in range(a, b)])
        Tb, Sb = oracle.build_pairs("deltanet", si.offsets_from_lengths([lens[i] for i in range(a, b)]), w,
                                    1, 2, 16, 16, L.k[idx], L.v[idx], None, L.beta[idx])
        # pairs of my segments' seam windows (each window a body of w tokens)
        n = b - a
        Tw, Sw = oracle.build_pairs("deltanet", np.arange(0, n * w + 1, w), 0, 1, 2, 16, 16,
                                    sa["k"][a:b].reshape(n * w, 1, 16), sa["v"][a:b].reshape(n * w, 2, 16), None,
                                    sa["beta"][a:b].reshape(n * w, 2))
        # my span's pair: seam, body, seam, body, ... merged in prompt order
        accT, accS = np.asarray(Tw[0]), np.asarray(Sw[0])
        for j in range(n):
            if j > 0:
                accT, accS = oracle.merge(Tw[j], Sw[j], accT, accS)
            accT, accS = oracle.merge(Tb[j], Sb[j], accT, accS)
        # exclusive scan over the ranks' span pairs
        mine = torch.from_numpy(np.stack([accT, accS]))
        allp = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(allp, mine)
        S0 = si.random_state((1, 2, 16, 16), seed=0, cfg=5).double().numpy()[0]
        state = S0
        for r in range(rank):
            Tr, Sr = allp[r][0].numpy(), allp[r][1].numpy()
            state = np.einsum("hij,hjk->hik", Tr, state) + Sr
        Sf, outs = oracle.compose("deltanet", Tb[None], Sb[None], sa["k"][None, a:b], sa["v"][None, a:b],
                                  sa["q"][None, a:b], None, sa["beta"][None, a:b], 1, 2, S_init=state[None])
        got = [None] * world
        dist.all_gather_object(got, (np.asarray(Sf), np.asarray(outs)))
        if rank == 0:
            np.save(os.path.join(out_dir, "S_final.npy"), got[-1][0])
            np.save(os.path.join(out_dir, "outs.npy"), np.concatenate([g[1] for g in got], axis=1))
    finally:
        dist.destroy_process_group()


def test_two_rank_span_parallel_compose_equals_single_chain(tmp_path):
    lens = [130, 64, 200, 9, 77, 300, 40]
    w = 4
    port = _free_port()
    mp.start_processes(_span_rank_main, args=(2, port, lens, w, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    W = si.workload(5, seed=3, device="cpu", variant="deltanet", lengths=lens, h_k=1, h_v=2, d=16, seam_w=w,
                    dtype=torch.float32)
    L = W.layers[0]
    sa = si.seam_gather(W, L)
    T, S = oracle.build_pairs("deltanet", W.seg_offsets, w, 1, 2, 16, 16, L.k, L.v, None, L.beta)
    S0 = si.random_state((1, 2, 16, 16), seed=0, cfg=5).double().numpy()
    Sf, outs = oracle.compose("deltanet", np.asarray(T)[None], np.asarray(S)[None], sa["k"][None], sa["v"][None],
                              sa["q"][None], None, sa["beta"][None], 1, 2, S_init=S0)
    got_S = np.load(tmp_path / "S_final.npy")
    got_o = np.load(tmp_path / "outs.npy")
    assert np.abs(got_S - np.asarray(Sf)).max() <= 1e-9 * max(1.0, np.abs(Sf).max())
    valid = sa["valid"].numpy()
    assert np.abs(got_o[0][valid] - np.asarray(outs)[0][valid]).max() <= 1e-9 * max(1.0, np.abs(outs).max())
