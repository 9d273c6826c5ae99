"""Segment parallelism over several GPUs (nav.aitube.vip §2.3): the cold
build scattered over workers, and one compose chain split by segments.

One process per GPU, ranks of a torch.distributed group.  Everything that
computes runs behind the kernel boundary `kernels` (by default the library's
C ABI through this package's binding); this module only decides who does
what and moves pairs between ranks:

cold_build_scatter
    The segments of a cold prompt are packed over the ranks longest body
    first (LPT; the pages balance uneven segments over scatter workers the
    same way).  Every rank holds the prompt's tokens and builds its own share
    (the other segments are skipped, HYPIC_SLOT_SKIP), in groups; each
    group's pairs travel to the combine rank by point-to-point sends while
    the next group builds.  Under NCCL the receives land straight in the
    combine rank's pool in its own HBM.  The combine rank's pool is laid out
    rank-major (every rank's share is one run of consecutive slots), so each
    transfer is one contiguous message.

compose_sharded
    The segments of every (layer, head) chain are split into one span per
    rank.  Each rank forms its span's pair with two composes of its own
    segments (S from a zero state, T by the transition-only compose from the
    identity), the pairs are all-gathered (one (T, S) per layer, head and
    span: the only exchange), every rank scans them for its start state and
    composes its span from there, writing its own seam outputs.  The last
    rank's final state is the chain's.

Both keep to the pages' data flow: per-segment work is independent and only
pairs move.  No collective or transfer touches a peer's memory directly.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

from . import FLAG_TRANSITION_ONLY, SLOT_SKIP, compose, pool_T_shape, segment_build, shard_lpt, span_scan


class LibraryKernels:
    """The kernel boundary: the library's entry points on this rank's GPU."""

    def __init__(self, device=None):
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)

    def empty(self, shape, dtype=torch.float32):
        return torch.empty(shape, dtype=dtype, device=self.device)

    def build(self, k, v, g, beta, seg_offsets, *, variant, seam_w, T_pool, S_pool, slot_of_seg):
        segment_build(k, v, g, beta, seg_offsets, variant=variant, seam_w=seam_w, T_pool=T_pool, S_pool=S_pool,
                      slot_of_seg=slot_of_seg)

    def compose(self, slot, T_pool, S_pool, seam, *, variant, S_out, seam_out=None, S_init=None, flags=0, span=None,
                h_k=None):
        compose(slot, T_pool, S_pool, seam["k"], seam["v"], seam["q"], seam["g"], seam["beta"], variant=variant,
                S_out=S_out, seam_out=seam_out, S_init=S_init, flags=flags, span=span, h_k=h_k)

    def span_scan(self, T_span, S_span, S_start, *, S_init=None):
        span_scan(T_span, S_span, S_start, S_init=S_init)


def _group_info(group):
    return dist.get_rank(group), dist.get_world_size(group)


def build_plan(seg_offsets, seam_w: int, world: int, n_groups: int):
    """The scatter plan every rank derives alike: shards[r] (segments of rank
    r, longest body first), groups[r] (consecutive runs of shards[r]) and
    slot_of_seg (combine-pool slot of every segment: rank-major, in shard
    order)."""
    off = np.asarray(seg_offsets, dtype=np.int64)
    bodies = np.maximum(np.diff(off) - int(seam_w), 0)
    shards = [s[np.argsort(-bodies[s], kind="stable")] for s in shard_lpt(bodies, world)]
    slot_of_seg = np.full(len(bodies), -1, dtype=np.int32)
    base = 0
    groups = []
    for r in range(world):
        sh = shards[r]
        slot_of_seg[sh] = base + np.arange(len(sh), dtype=np.int32)
        base += len(sh)
        ng = max(1, min(int(n_groups), len(sh)))
        groups.append([g for g in np.array_split(np.arange(len(sh)), ng) if len(g)])
    return shards, groups, slot_of_seg


def cold_build_scatter(k, v, g, beta, seg_offsets, *, variant: str, seam_w: int, T_pool=None, S_pool=None,
                       group=None, combine_rank: int = 0, n_groups: int = 4, kernels=None):
    """Build every segment's pair once, spread over the ranks of `group`, and
    collect the pairs in the combine rank's pool.  Every rank passes the
    whole prompt (k, v, g, beta, seg_offsets as for segment_build); the
    combine rank passes its pool (T_pool, S_pool with at least n_seg slots).
    Returns slot_of_seg, the combine-pool slot of every segment (the same on
    every rank).  Collective: every rank of `group` must call it."""
    kernels = kernels or LibraryKernels()
    rank, world = _group_info(group)
    n_seg = len(seg_offsets) - 1
    h_v, d_k, d_v = v.shape[1], k.shape[2], v.shape[2]
    shards, groups, slot_of_seg = build_plan(seg_offsets, seam_w, world, n_groups)
    starts = np.concatenate([[0], np.cumsum([len(s) for s in shards])])
    peer = lambda r: dist.get_global_rank(group, r) if group is not None else r
    pending = []
    if rank == combine_rank:
        # receives first (posted before the local builds), each into the run
        # of slots of one group of one rank
        for r in range(world):
            if r == rank:
                continue
            for gi in groups[r]:
                a, b = starts[r] + gi[0], starts[r] + gi[-1] + 1
                pending.append(dist.irecv(T_pool[a:b], src=peer(r), group=group))
                pending.append(dist.irecv(S_pool[a:b], src=peer(r), group=group))
        for gi in groups[rank]:
            sl = np.full(n_seg, SLOT_SKIP, dtype=np.int32)
            sl[shards[rank][gi]] = slot_of_seg[shards[rank][gi]]
            kernels.build(k, v, g, beta, seg_offsets, variant=variant, seam_w=seam_w, T_pool=T_pool, S_pool=S_pool,
                          slot_of_seg=sl)
    else:
        # two staging pools, alternating by group: group j + 1 builds while
        # group j's pairs are on the wire; a pool is reused once its sends
        # of two groups ago are complete
        cap = max((len(gi) for gi in groups[rank]), default=0)
        stage = [(kernels.empty(pool_T_shape(variant, cap, h_v, d_k)), kernels.empty((cap, h_v, d_k, d_v)))
                 for _ in range(2)] if cap else []
        sends = [[], []]
        for j, gi in enumerate(groups[rank]):
            Tb, Sb = stage[j & 1]
            for w_ in sends[j & 1]:
                w_.wait()
            sl = np.full(n_seg, SLOT_SKIP, dtype=np.int32)
            sl[shards[rank][gi]] = np.arange(len(gi), dtype=np.int32)
            kernels.build(k, v, g, beta, seg_offsets, variant=variant, seam_w=seam_w, T_pool=Tb, S_pool=Sb,
                          slot_of_seg=sl)
            sends[j & 1] = [dist.isend(Tb[:len(gi)], dst=peer(combine_rank), group=group),
                            dist.isend(Sb[:len(gi)], dst=peer(combine_rank), group=group)]
        pending = sends[0] + sends[1]
    for w_ in pending:
        w_.wait()
    return slot_of_seg


def compose_sharded(slot, T_pool, S_pool, seam, *, variant: str, S_out, seam_out=None, S_init=None, group=None,
                    bounds=None, h_k=None, kernels=None):
    """compose() of every (layer, head) chain with the segments split into
    one span per rank of `group` (bounds: [world + 1] segment boundaries,
    default about equal counts).  Rank r needs the pairs (slot -> T_pool,
    S_pool) and seam tokens of its own span only; seam arrays are the whole
    prompt's [L, n_seg, w, ...] (rows of other spans are not read) and
    seam_out rows of rank r's span are written.  S_out [L, h_v, d_k, d_v]
    receives the chain's final state on the last rank (on the others: the
    state after their own span).  Returns this rank's (a, b) span.
    Collective: every rank of `group` must call it."""
    kernels = kernels or LibraryKernels()
    rank, world = _group_info(group)
    L, n_seg = slot.shape
    _, h_v, d_k, d_v = S_out.shape
    b = (np.linspace(0, n_seg, world + 1).round().astype(np.int32) if bounds is None
         else np.asarray(bounds, dtype=np.int32))
    assert len(b) == world + 1 and b[0] == 0 and b[-1] == n_seg
    span = (int(b[rank]), int(b[rank + 1]))
    # 1. this span's pair: S from zero, T from the identity
    T_loc = kernels.empty((L, h_v, d_k, d_k))
    S_loc = kernels.empty((L, h_v, d_k, d_v))
    kernels.compose(slot, T_pool, S_pool, seam, variant=variant, S_out=S_loc, seam_out=seam_out, span=span, h_k=h_k)
    kernels.compose(slot, T_pool, None, seam, variant=variant, S_out=T_loc, flags=FLAG_TRANSITION_ONLY, span=span,
                    h_k=h_k)
    # 2. every span's pair on every rank (the one exchange)
    T_all = kernels.empty((world, L, h_v, d_k, d_k))
    S_all = kernels.empty((world, L, h_v, d_k, d_v))
    dist.all_gather(list(T_all.unbind(0)), T_loc, group=group)
    dist.all_gather(list(S_all.unbind(0)), S_loc, group=group)
    # 3. the start state of every span, 4. this span from its own
    S_start = kernels.empty((world, L, h_v, d_k, d_v))
    kernels.span_scan(T_all, S_all, S_start, S_init=S_init)
    kernels.compose(slot, T_pool, S_pool, seam, variant=variant, S_out=S_out, seam_out=seam_out,
                    S_init=S_start[rank].contiguous(), span=span, h_k=h_k)
    return span
