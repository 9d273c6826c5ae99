"""Pins for the fp64 oracle: checks against what the HYPIC pages and plain
mathematics fix, none of which re-types the oracle's own arithmetic.

Each pin takes an ``OracleLib`` (so the same pins can be run against a copy of
the oracle with a planted mistake) and raises AssertionError on failure.

  dense_product     T_C and S(C|0) equal the explicit product of dense token
                    matrices (the pages' definition of T_C), every variant
  outputs           o_t = S_t^T q_t and the final state of `full` equal a
                    dense-matrix recurrence, every variant, with GQA
  composition       compose (seams + T_C S + S(C|0)) equals the full
                    recurrence from any prefix state (the pages' rule
                    S(C1·C2) = T(C2)·S(C1) + S(C2)), on the tiny GDN workload
  split_merge       splitting a segment at any token and merging the two
                    pairs reproduces the pair (associativity of the rule)
  ungated_sum       T = I reduces the state to the plain sum of k v^T, and
                    the naive sum is then exact (pages: valid for plain
                    linear attention)
  retnet_closed     T_C = gamma^L I and S = sum gamma^(L-t) k v^T
  householder       single token: spectrum {1 - b|k|^2, 1, ..., 1};
                    b = 2 with |k| = 1 gives an orthogonal T_C
  contraction       ||T_C||_2 <= 1 for unit k, b in (0,1], gates <= 1
  cross_variant     channel gate a*1 == gdn; gdn with g=0 == deltanet;
                    constant diagonal == scalar decay; zero diagonal == ungated
  prefix_free       a segment's pair does not depend on the tokens before it
  naive_wrong       (slow) with decay the naive sum is off by >= 10% of the
                    state norm on every head of the RetNet workload
  rerotation_keys   re-rotating a pair by R(delta) equals building the pair
                    from keys rotated by R(delta) (GDN, DeltaNet, RetNet,
                    ungated; both channel pairings, partial rotary dim)
  rerotation_group  R(0) = I, R orthogonal, re-rotation by d1 then d2 equals
                    re-rotation by d1 + d2, norms and spectra preserved
"""
from __future__ import annotations

import numpy as np

from oracle import dense_twin

TIGHT = 1e-12


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    n = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (n if n > 0 else 1.0))


def tiny_inputs(variant, N, h_k, h_v, d_k, d_v, seed, beta_hi=1.0):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((N, h_k, d_k))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((N, h_v, d_v))
    q = rng.standard_normal((N, h_k, d_k))
    g = None
    beta = None
    if variant == "gdn":
        g = -rng.uniform(0.001, 0.3, (N, h_v))
    elif variant in ("channel", "diag"):
        g = -np.log1p(np.exp(rng.standard_normal((N, h_v, d_k))))
    elif variant == "scalar":
        g = np.log(1.0 - 2.0 ** (-1.0 - np.arange(h_v)))
    if variant in ("gdn", "deltanet", "channel"):
        beta = rng.uniform(0.05, beta_hi, (N, h_v))
    return k, v, q, g, beta


ALL = ("gdn", "deltanet", "channel", "scalar", "ungated", "diag")


def dense_product(orc):
    lens = [5, 1, 9, 0, 3]
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    h_k, h_v, d_k, d_v = 2, 4, 5, 3
    for vi, var in enumerate(ALL):
        k, v, q, g, beta = tiny_inputs(var, int(off[-1]), h_k, h_v, d_k, d_v, 100 + vi, beta_hi=1.8)
        for w in (0, 2):
            T, S = orc.build_pairs(var, off, w, h_k, h_v, d_k, d_v, k, v, g, beta)
            for i in range(len(lens)):
                for h in range(h_v):
                    s = min(int(off[i]) + w, int(off[i + 1]))
                    Td, Sd = dense_twin.pair(var, k, v, g, beta, s, int(off[i + 1]), h, h_k, h_v)
                    assert _rel(T[i, h], Td) < TIGHT, (var, w, i, h, "T")
                    assert np.linalg.norm(S[i, h] - Sd) <= TIGHT * max(1.0, np.linalg.norm(Sd)), (var, w, i, h, "S")


def outputs(orc):
    h_k, h_v, d_k, d_v, N = 2, 4, 4, 6, 11
    rng = np.random.default_rng(7)
    for vi, var in enumerate(ALL):
        k, v, q, g, beta = tiny_inputs(var, N, h_k, h_v, d_k, d_v, 200 + vi, beta_hi=1.5)
        S0 = rng.standard_normal((h_v, d_k, d_v))
        S, outs = orc.full(var, k, v, q, g, beta, h_k, h_v, S_init=S0, out_pos=np.arange(N))
        for h in range(h_v):
            od, Sd = dense_twin.outputs(var, k, v, q, g, beta, h, h_k, h_v, S0=S0[h])
            assert _rel(outs[:, h], od) < TIGHT, (var, h, "outs")
            assert _rel(S[h], Sd) < TIGHT, (var, h, "S")


def _gather_seams(off, w, arrs):
    n_seg = len(off) - 1
    out = []
    for a in arrs:
        if a is None or a.ndim == 1:
            out.append(a)
            continue
        idx = np.array([[int(off[i]) + t for t in range(w)] for i in range(n_seg)])
        out.append(a[idx][None])          # [1, n_seg, w, ...]
    return out


def composition(orc, k=None, v=None, q=None, g=None, beta=None, off=None, variant="gdn",
                h_k=1, h_v=1, w=8, seed=0):
    """Default: the tiny GDN workload (1 head, d=16, 4 x 64 tokens, w=8)."""
    if k is None:
        import synth_inputs as si
        W = si.workload(1, seed=seed)
        L = W.layers[0]
        k, v, q, g, beta = (None if x is None else x.double().numpy() for x in (L.k, L.v, L.q, L.g, L.beta))
        off, variant, h_k, h_v, w = W.seg_offsets, W.variant, W.h_k, W.h_v, W.seam_w
    d_k, d_v = k.shape[-1], v.shape[-1]
    T, S = orc.build_pairs(variant, off, w, h_k, h_v, d_k, d_v, k, v, g, beta)
    sk, sv, sq, sg, sb = _gather_seams(off, w, (k, v, q, g, beta))
    pos = np.array([int(off[i]) + t for i in range(len(off) - 1) for t in range(w)], dtype=np.int64)
    rng = np.random.default_rng(seed + 1)
    for S0 in (None, rng.standard_normal((h_v, d_k, d_v))):
        So, seam = orc.compose(variant, T[None], S[None], sk, sv, sq, sg, sb, h_k, h_v,
                               S_init=None if S0 is None else S0[None])
        Sf, outs = orc.full(variant, k, v, q, g, beta, h_k, h_v, S_init=S0, out_pos=pos)
        assert _rel(So[0], Sf) < TIGHT, "final state"
        if w:
            assert _rel(seam[0].reshape(-1, h_v, d_v), outs) < TIGHT, "seam outputs"


def composition_all(orc):
    lens = [7, 12, 3, 9]
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    for vi, var in enumerate(ALL):
        k, v, q, g, beta = tiny_inputs(var, int(off[-1]), 2, 4, 5, 3, 300 + vi)
        composition(orc, k, v, q, g, beta, off, var, 2, 4, w=3, seed=vi)


def split_merge(orc):
    N = 12
    h_k, h_v, d_k, d_v = 1, 2, 4, 3
    for vi, var in enumerate(ALL):
        k, v, q, g, beta = tiny_inputs(var, N, h_k, h_v, d_k, d_v, 400 + vi)
        Tw, Sw = orc.build_pairs(var, [0, N], 0, h_k, h_v, d_k, d_v, k, v, g, beta)
        for m in range(0, N + 1):
            T, S = orc.build_pairs(var, [0, m, N], 0, h_k, h_v, d_k, d_v, k, v, g, beta)
            To, So = orc.merge(T[1], S[1], T[0], S[0])
            assert _rel(To, Tw[0]) < TIGHT and _rel(So, Sw[0]) < TIGHT, (var, m)
    rng = np.random.default_rng(5)
    P = [(rng.standard_normal((3, 4, 4)), rng.standard_normal((3, 4, 2))) for _ in range(3)]
    ab = orc.merge(*P[0], *P[1])
    left = orc.merge(*ab, *P[2])
    bc = orc.merge(*P[1], *P[2])
    right = orc.merge(*P[0], *bc)
    assert _rel(left[0], right[0]) < TIGHT and _rel(left[1], right[1]) < TIGHT


def ungated_sum(orc):
    lens = [6, 10, 4]
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    h_k, h_v, d_k, d_v = 2, 4, 5, 3
    k, v, q, g, beta = tiny_inputs("ungated", int(off[-1]), h_k, h_v, d_k, d_v, 11)
    T, S = orc.build_pairs("ungated", off, 0, h_k, h_v, d_k, d_v, k, v)
    kmap = (np.arange(h_v) * h_k) // h_v
    for i in range(len(lens)):
        sl = slice(int(off[i]), int(off[i + 1]))
        ref = np.einsum("thd,the->hde", k[sl][:, kmap], v[sl])
        assert np.abs(T[i] - np.eye(d_k)).max() == 0.0
        assert _rel(S[i], ref) < TIGHT
    Sf, _ = orc.full("ungated", k, v, q, None, None, h_k, h_v)
    assert _rel(S.sum(0), Sf) < TIGHT


def retnet_closed(orc):
    lens = [9, 4]
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    h_k, h_v, d_k, d_v = 3, 3, 4, 5
    k, v, q, g, beta = tiny_inputs("scalar", int(off[-1]), h_k, h_v, d_k, d_v, 12)
    T, S = orc.build_pairs("scalar", off, 0, h_k, h_v, d_k, d_v, k, v, g)
    gam = np.exp(g)
    for i in range(len(lens)):
        L = lens[i]
        for h in range(h_v):
            assert _rel(T[i, h], gam[h] ** L * np.eye(d_k)) < TIGHT
            ref = sum(gam[h] ** (L - 1 - t) * np.outer(k[off[i] + t, h], v[off[i] + t, h]) for t in range(L))
            assert _rel(S[i, h], ref) < TIGHT


def householder(orc):
    d = 6
    rng = np.random.default_rng(13)
    kk = rng.standard_normal((1, 1, d))
    kk /= np.linalg.norm(kk)
    v = rng.standard_normal((1, 1, 2))
    for b in (0.3, 0.7, 1.0):
        T, _ = orc.build_pairs("deltanet", [0, 1], 0, 1, 1, d, 2, kk, v, None, np.array([[b]]))
        ev = np.sort(np.linalg.eigvalsh(0.5 * (T[0, 0] + T[0, 0].T)))
        want = np.sort(np.array([1.0 - b] + [1.0] * (d - 1)))
        assert np.abs(ev - want).max() < TIGHT
    N = 25
    k = rng.standard_normal((N, 1, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((N, 1, 2))
    T, _ = orc.build_pairs("deltanet", [0, N], 0, 1, 1, d, 2, k, v, None, np.full((N, 1), 2.0))
    assert np.abs(T[0, 0].T @ T[0, 0] - np.eye(d)).max() < 1e-11


def contraction(orc):
    N = 40
    for vi, var in enumerate(("gdn", "deltanet", "channel")):
        k, v, q, g, beta = tiny_inputs(var, N, 1, 2, 6, 3, 500 + vi, beta_hi=1.0)
        T, _ = orc.build_pairs(var, [0, 13, N], 0, 1, 2, 6, 3, k, v, g, beta)
        for Tm in T.reshape(-1, 6, 6):
            assert np.linalg.norm(Tm, 2) <= 1.0 + 1e-12


def cross_variant(orc):
    N, h_k, h_v, d_k, d_v = 14, 2, 4, 5, 3
    off = [0, 6, N]
    k, v, q, g, beta = tiny_inputs("gdn", N, h_k, h_v, d_k, d_v, 21)
    Tg, Sg = orc.build_pairs("gdn", off, 0, h_k, h_v, d_k, d_v, k, v, g, beta)
    gc = np.repeat(g[:, :, None], d_k, axis=2)
    Tc, Sc = orc.build_pairs("channel", off, 0, h_k, h_v, d_k, d_v, k, v, gc, beta)
    assert _rel(Tc, Tg) < TIGHT and _rel(Sc, Sg) < TIGHT
    T0, S0 = orc.build_pairs("gdn", off, 0, h_k, h_v, d_k, d_v, k, v, np.zeros_like(g), beta)
    Td, Sd = orc.build_pairs("deltanet", off, 0, h_k, h_v, d_k, d_v, k, v, None, beta)
    assert _rel(T0, Td) < TIGHT and _rel(S0, Sd) < TIGHT
    gh = np.log(np.array([0.9, 0.8, 0.95, 0.5]))
    gd = np.broadcast_to(gh[None, :, None], (N, h_v, d_k)).copy()
    Ta, Sa = orc.build_pairs("diag", off, 0, h_k, h_v, d_k, d_v, k, v, gd)
    Ts, Ss = orc.build_pairs("scalar", off, 0, h_k, h_v, d_k, d_v, k, v, gh)
    assert _rel(Ta, Ts) < TIGHT and _rel(Sa, Ss) < TIGHT
    Tz, Sz = orc.build_pairs("diag", off, 0, h_k, h_v, d_k, d_v, k, v, np.zeros((N, h_v, d_k)))
    Tu, Su = orc.build_pairs("ungated", off, 0, h_k, h_v, d_k, d_v, k, v)
    assert _rel(Tz, Tu) < TIGHT and _rel(Sz, Su) < TIGHT


def prefix_free(orc):
    h_k, h_v, d_k, d_v = 1, 2, 4, 3
    for vi, var in enumerate(ALL):
        k, v, q, g, beta = tiny_inputs(var, 20, h_k, h_v, d_k, d_v, 600 + vi)
        k2, v2, q2, g2, beta2 = tiny_inputs(var, 20, h_k, h_v, d_k, d_v, 700 + vi)
        # prompt A = [first 8 tokens of draw 1, segment C]; prompt B = [5 tokens of draw 2, C]
        def cat(a, b, na, nb=12):
            if a is None or a.ndim == 1:
                return a
            return np.concatenate([b[:na], a[8:8 + nb]])
        A = [cat(x, x, 8) for x in (k, v, g, beta)]
        B = [cat(x, y, 5) for x, y in zip((k, v, g, beta), (k2, v2, g2, beta2))]
        Ta, Sa = orc.build_pairs(var, [0, 8, 20], 0, h_k, h_v, d_k, d_v, *A)
        Tb, Sb = orc.build_pairs(var, [0, 5, 17], 0, h_k, h_v, d_k, d_v, *B)
        assert np.array_equal(Ta[1], Tb[1]) and np.array_equal(Sa[1], Sb[1]), var


def naive_wrong(orc, min_err=0.10):
    """RetNet workload (8 heads, gamma_h = 1 - 2^(-5-h), d=128, 16 x 512): the
    naive sum of zero-initial states misses the decay of earlier segments."""
    import synth_inputs as si
    W = si.workload(2, seed=0)
    L = W.layers[0]
    T, S = orc.build_pairs("scalar", W.seg_offsets, 0, W.h_k, W.h_v, W.d_k, W.d_v, L.k, L.v, L.g)
    Sf, _ = orc.full("scalar", L.k, L.v, L.q, L.g, None, W.h_k, W.h_v)
    naive = S.sum(0)
    errs = [_rel(naive[h], Sf[h]) for h in range(W.h_v)]
    assert min(errs) >= min_err, errs
    return errs


def rerotation_keys(orc, rerotate=None):
    """The pair of a segment whose keys are all multiplied by R(delta) is the
    re-rotated pair: every token transition becomes R T_t R^T and every write
    R U_t.  Checked against the oracle's token-by-token build, one delta per
    segment (negative, zero, large), with the rotary dim below d_k."""
    import oracle
    rerotate = rerotate or oracle.rerotate
    lens = [5, 7, 1, 7]
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    deltas = [3, -7, 0, 12345]
    h_k, h_v, d_k, d_v = 2, 4, 6, 3
    for vi, var in enumerate(("gdn", "deltanet", "scalar", "ungated")):
        k, v, q, g, beta = tiny_inputs(var, int(off[-1]), h_k, h_v, d_k, d_v, 300 + vi)
        T, S = orc.build_pairs(var, off, 0, h_k, h_v, d_k, d_v, k, v, g, beta)
        for layout, rot in (("interleaved", 6), ("interleaved", 4), ("half", 4), ("half", 6)):
            kr = k.copy()
            for i, dl in enumerate(deltas):
                R = oracle.rerotation_matrix(d_k, dl, rot, layout, base=50.0)
                kr[off[i]:off[i + 1]] = np.einsum("ab,thb->tha", R, k[off[i]:off[i + 1]])
            T2, S2 = orc.build_pairs(var, off, 0, h_k, h_v, d_k, d_v, kr, v, g, beta)
            To, So = rerotate(var, T, S, deltas, rot, layout, base=50.0)
            assert _rel(To, T2) < TIGHT, (var, layout, rot, "T")
            assert _rel(So, S2) < TIGHT, (var, layout, rot, "S")


def rerotation_group(orc, rerotate=None):
    import oracle
    rerotate = rerotate or oracle.rerotate
    rng = np.random.default_rng(11)
    d_k, d_v = 8, 5
    T = rng.standard_normal((3, 2, d_k, d_k))
    S = rng.standard_normal((3, 2, d_k, d_v))
    for layout in ("interleaved", "half"):
        R = oracle.rerotation_matrix(d_k, 777, d_k, layout)
        assert np.abs(R @ R.T - np.eye(d_k)).max() < TIGHT
        assert np.abs(oracle.rerotation_matrix(d_k, 0, d_k, layout) - np.eye(d_k)).max() == 0.0
        d1, d2 = np.array([5, -40, 900]), np.array([-3, 41, 77])
        Ta, Sa = rerotate("gdn", *rerotate("gdn", T, S, d1, d_k, layout), d2, d_k, layout)
        Tb, Sb = rerotate("gdn", T, S, d1 + d2, d_k, layout)
        assert _rel(Ta, Tb) < 1e-11 and _rel(Sa, Sb) < 1e-11, layout
        To, So = rerotate("gdn", T, S, d1, d_k, layout)
        assert abs(np.linalg.norm(So) - np.linalg.norm(S)) < TIGHT * np.linalg.norm(S)
        ev0 = np.sort_complex(np.linalg.eigvals(T[1, 0]))
        ev1 = np.sort_complex(np.linalg.eigvals(To[1, 0]))
        assert np.abs(ev0 - ev1).max() < 1e-9, layout


FAST_PINS = (dense_product, outputs, composition, composition_all, split_merge, ungated_sum,
             retnet_closed, householder, contraction, cross_variant, prefix_free, rerotation_keys,
             rerotation_group)
