"""Chunkwise (WY / UT-transform) form of the segment build, in torch on the
CPU.  Test and design tool only: in fp64 it checks that the chunk algebra the
tensor-core kernel implements reaches the token-by-token definition; with
operand rounding switched on it predicts the kernel's error for a choice of
MMA operand precision.

Derivation (scalar or per-channel gate, delta variants).  Inside a chunk of C
tokens let lam_t = sum_{j<=t} g_j (a scalar or a d_k vector) and
Gam_t = exp(lam_t).  With delta_t = b_t (v_t - S_{t-1}^T Diag(a_t) k_t) the
token step reads S_t = Diag(a_t) S_{t-1} + k_t delta_t^T, which unrolls to
    S_t = Gam_t S_0 + sum_{i<=t} (Gam_t / Gam_i) k_i delta_i^T.
Substituting back gives the unit lower-triangular system
    (I + diag(b) M) Delta = diag(b) V - diag(b) (K*Gam) S_0,
    M_ti = sum_c k_t[c] k_i[c] exp(lam_t[c] - lam_i[c])   (i < t),
so with A = (I + diag(b) M)^{-1}, W = A diag(b) (K*Gam), U = A diag(b) V:
    Delta = U - W S_0,   S_C = Gam_C S_0 + Khat^T (U - W S_0),
    Khat_i = k_i * exp(lam_C - lam_i).
On the augmented block X = [T | S] (d_k x (d_k + d_v)) one chunk is
    Y = W X - [0 | U],   X <- Gam_C (row scale) X - Khat^T Y,
starting from X = [I | 0].  The variants without an erase (scalar decay,
ungated, diagonal gate) have A = I, b = 1, and need no chain: T_C = Gam_L,
S = Khat^T V over the whole body.
"""
from __future__ import annotations

import torch

C = 64


def rnd_bf16(x):
    return x.to(torch.bfloat16).to(x.dtype)


def rnd_tf32(x):
    """Keep the top 10 mantissa bits (what an fp32 operand of a tf32 MMA
    contributes, truncating)."""
    y = x.to(torch.float32).contiguous()
    i = y.view(torch.int32) & ~((1 << 13) - 1)
    return i.view(torch.float32).to(x.dtype)


def ident(x):
    return x


def split2(r):
    """hi + lo operand split: the product with both halves through `r`."""
    def f(x):
        hi = r(x)
        return hi, r(x - hi)
    return f


def _mm(a, b, ra, rb, split_a=False, split_b=False):
    """a @ b with the operands rounded by ra / rb; split_* adds the residual
    term of that operand (a 2-term split of one side)."""
    ah = ra(a)
    bh = rb(b)
    out = ah @ bh
    if split_a:
        out = out + ra(a - ah) @ bh
    if split_b:
        out = out + ah @ rb(b - bh)
    return out


def build_chunked(variant, k, v, g, beta, start, end, h, h_k, h_v, *, chunk=C,
                  op=ident, split_x=False, split_y=False, split_w=False, dtype=torch.float64):
    """(T_C, S(C|0)) of value head h over tokens [start, end) via the chunk
    algebra.  k [N,h_k,d_k], v [N,h_v,d_v], g / beta as in the oracle.
    `op` rounds MMA operands (ident = exact)."""
    kh = (h * h_k) // h_v
    K = torch.as_tensor(k[start:end, kh]).to(dtype)
    V = torch.as_tensor(v[start:end, h]).to(dtype)
    n, d_k = K.shape
    d_v = V.shape[1]
    vec = variant in ("channel", "diag")
    has_beta = variant in ("gdn", "deltanet", "channel")
    if variant == "gdn":
        gg = torch.as_tensor(g[start:end, h]).to(dtype)
    elif variant in ("channel", "diag"):
        gg = torch.as_tensor(g[start:end, h]).to(dtype)
    elif variant == "scalar":
        gg = torch.full((n,), float(g[h]), dtype=dtype)
    else:
        gg = torch.zeros(n, dtype=dtype)
    bb = torch.as_tensor(beta[start:end, h]).to(dtype) if has_beta else torch.ones(n, dtype=dtype)
    X = torch.zeros(d_k, d_k + d_v, dtype=dtype)
    X[:, :d_k] = torch.eye(d_k, dtype=dtype)
    for c0 in range(0, n, chunk):
        c1 = min(n, c0 + chunk)
        Kc, Vc, gc, bc = K[c0:c1], V[c0:c1], gg[c0:c1], bb[c0:c1]
        lam = torch.cumsum(gc, 0)                     # [m] or [m, d_k]
        lamC = lam[-1]
        if has_beta:
            if vec:
                # M_ti = sum_c k_t k_i exp(lam_t - lam_i), i < t
                E = torch.exp(lam[:, None, :] - lam[None, :, :])
                M = torch.tril(torch.einsum("tc,ic,tic->ti", Kc, Kc, E), -1)
            else:
                M = torch.tril(torch.exp(lam[:, None] - lam[None, :]), -1) * (op(Kc) @ op(Kc).T)
            Lm = torch.eye(len(bc), dtype=dtype) + bc[:, None] * M
            A = torch.linalg.solve_triangular(Lm, torch.eye(len(bc), dtype=dtype), upper=False)
            KG = Kc * (torch.exp(lam) if vec else torch.exp(lam)[:, None])
            W = _mm(A, bc[:, None] * KG, op, op, split_b=split_w, split_a=split_w)
            U = _mm(A, bc[:, None] * Vc, op, op)
        else:
            W = None
            U = Vc
        Gc = torch.exp(lamC)
        decay = torch.exp(lamC[None, :] - lam) if vec else torch.exp(lamC - lam)[:, None]
        if W is None:
            Khat = Kc * decay
            X = (Gc[:, None] if vec else Gc) * X
            X[:, d_k:] = X[:, d_k:] + _mm(Khat.T, Vc, op, op)
            continue
        Y = _mm(W, X, op, op, split_b=split_x)
        Y[:, d_k:] = Y[:, d_k:] - U
        if vec:
            Khat = Kc * decay
            corr = _mm(Khat.T, Y, op, op, split_b=split_y)
        else:
            # scalar gate: move exp(lam_C - lam_i) onto Y's rows, K stays exact
            corr = _mm(Kc.T, decay * Y, op, op, split_b=split_y)
        X = (Gc[:, None] if vec else Gc) * X - corr
    return X[:, :d_k], X[:, d_k:]


def gram_subblocks(Kc, lam, sb=16):
    """The decayed Gram of a chunk with a per-channel gate, strictly lower
    part, M_ti = sum_c k_t[c] k_i[c] exp(lam_t[c] - lam_i[c]) (i < t), formed
    the way the tensor-core kernel forms it: token rows in sub-blocks of
    `sb`, each with the reference ref = lam just before the sub-block, as
    the product of Q_t = k_t exp(lam_t - ref) and R_i = k_i exp(ref - lam_i).
    Every exponent is bounded by the log-gate range of one sub-block."""
    m = Kc.shape[0]
    M = torch.zeros(m, m, dtype=Kc.dtype)
    for b0 in range(0, m, sb):
        b1 = min(m, b0 + sb)
        ref = lam[b0 - 1] if b0 > 0 else torch.zeros_like(lam[0])
        Q = Kc[b0:b1] * torch.exp(lam[b0:b1] - ref)
        R = Kc[:b1] * torch.exp(ref - lam[:b1])
        M[b0:b1, :b1] = Q @ R.T
    return torch.tril(M, -1)


def block_inverse(N, b=16):
    """A = (I + N)^{-1} for a strictly lower N, by the block schedule of the
    tensor-core build's preparation group (blocks of `b`, four of them for a
    64-token chunk, two for a 32-token one):
      1. the diagonal blocks by forward substitution;
      2. A_10 = -A_11 N_10 A_00 and A_32 = -A_33 N_32 A_22;
      3. with the leading half done, P_aj = sum_{k=j}^{1} N_ak A_kj for
         a in {2, 3}, j in {0, 1}, then A_ij = -sum_{a=2}^{i} A_ia P_aj.
    Blocks above the block diagonal are never read (they start as NaN here,
    so a read of one shows in the result)."""
    m = N.shape[0]
    nb = m // b
    assert nb * b == m and nb in (2, 4)
    A = torch.full((m, m), float("nan"), dtype=N.dtype)
    blk = lambda X, i, j: X[b * i:b * (i + 1), b * j:b * (j + 1)]
    for d in range(nb):  # stage 1: column by column, row by row
        Nd = blk(N, d, d)
        Ad = torch.zeros(b, b, dtype=N.dtype)
        for col in range(b):
            Ad[col, col] = 1.0
            for r in range(col + 1, b):
                Ad[r, col] = -(Nd[r, :r] * Ad[:r, col]).sum()
        blk(A, d, d)[:] = Ad
    for h in range(nb // 2):  # stage 2
        i, j = 2 * h + 1, 2 * h
        blk(A, i, j)[:] = -blk(A, i, i) @ (blk(N, i, j) @ blk(A, j, j))
    if nb == 4:  # stage 3
        P = {(a, j): sum(blk(N, a, k) @ blk(A, k, j) for k in range(j, 2)) for a in (2, 3) for j in (0, 1)}
        for i in (2, 3):
            for j in (0, 1):
                blk(A, i, j)[:] = -sum(blk(A, i, a) @ P[(a, j)] for a in range(2, i + 1))
    return torch.tril(A)
