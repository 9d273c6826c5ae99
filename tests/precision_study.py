"""Operand-precision study for the tensor-core chunkwise build (GDN and
DeltaNet, d = 128, 64-token chunks), on the CPU.

The chunk algebra of the build (see tests/chunkform.py for its derivation,
pinned there against the token oracle in fp64) is emulated in fp64 with every
MMA operand rounded as a given kernel design rounds it, and fp32 results
where the kernel keeps fp32 (accumulators, the inverse, the state).  The
error of the emulated pair against the fp64 token oracle (oracle/) predicts
the kernel's error for that design, so an operand precision can be chosen
before a kernel is written.  Nothing here is used by the library.

Operands, one rounding each (rn = tf32 rounded to nearest by the threads,
trunc = tf32 as the tensor core reads a raw fp32 value, bf16, split = hi + lo
bf16 pair, exact to about 2^-17):
  F     the factor tiles A diag(b G) and A diag(b) of the W and U products
        (K and V are exact bf16 inputs)
  X     the state block [T | S] as the A operand of chain 1 (Y = W X - U)
  W     W as the B operand of chain 1
  Yt    Ytilde = -Y diag(exp(lam_C - lam)) as the A operand of chain 2
        (X <- G_C X + Ytilde^T K)

    python tests/precision_study.py [--tokens 8192] [--heads 4]

prints the worst per-head relative Frobenius error of T_C and S(C|0) for
each design, on config-5-shaped inputs (bf16 k, v; beta = sigmoid(N(0,1));
GDN log-gates U(-0.1, -0.001)) of one body of the given length.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

C = 64


def rn_tf32(x):
    y = x.to(torch.float32).contiguous()
    i = y.view(torch.int32).to(torch.int64)
    i = ((i + 0x1000) & ~0x1FFF) & 0xFFFFFFFF
    i = torch.where(i >= 2 ** 31, i - 2 ** 32, i).to(torch.int32)
    return i.view(torch.float32).to(torch.float64)


def trunc_tf32(x):
    y = x.to(torch.float32).contiguous()
    return (y.view(torch.int32) & ~0x1FFF).view(torch.float32).to(torch.float64)


def bf16(x):
    return x.to(torch.bfloat16).to(torch.float64)


def f32(x):
    return x.to(torch.float32).to(torch.float64)


ROUND = {"rn": rn_tf32, "trunc": trunc_tf32, "bf16": bf16, "f32": f32}


def operand(x, how):
    """The operand as the MMA sees it: one rounded copy, or hi + lo."""
    if how == "split":
        hi = bf16(x)
        return [hi, bf16(x - hi)]
    return [ROUND[how](x)]


def mm(a_parts, b_parts):
    """Product of split operands without the lo * lo term (fp64 sum of the
    fp32-exact partial products; the fp32 accumulation is applied by the
    caller)."""
    out = 0
    for i, a in enumerate(a_parts):
        for j, b in enumerate(b_parts):
            if i + j <= 1:
                out = out + a @ b
    return out


def build_emulated(K, V, g, beta, design):
    """(T_C, S(C|0)) of one body (K [L, d], V [L, d] fp64 holding bf16
    values; g, beta [L]) through the chunk algebra with the design's operand
    roundings."""
    L, d = K.shape
    X = torch.zeros(d, 2 * d, dtype=torch.float64)
    X[:, :d] = torch.eye(d, dtype=torch.float64)
    for c0 in range(0, L, C):
        Kc, Vc, gc, bc = K[c0:c0 + C], V[c0:c0 + C], g[c0:c0 + C], beta[c0:c0 + C]
        m = len(bc)
        lam = torch.cumsum(gc, 0)
        M = f32(torch.tril(torch.exp(lam[:, None] - lam[None, :]), -1) * (Kc @ Kc.T) * bc[:, None])
        A = f32(torch.linalg.solve_triangular(torch.eye(m, dtype=torch.float64) + M,
                                              torch.eye(m, dtype=torch.float64), upper=False))
        G = torch.exp(lam)
        W = f32(mm(operand(A * (bc * G)[None, :], design["F"]), [Kc]))
        U = f32(mm(operand(A * bc[None, :], design["F"]), [Vc]))
        Y = mm(operand(W, design["W"]), operand(X, design["X"]))
        Y[:, d:] = Y[:, d:] - U
        Y = f32(Y)
        Yt = -Y * torch.exp(lam[-1] - lam)[:, None]
        X = f32(f32(torch.exp(lam[-1]) * X) + mm([Kc.T], operand(Yt, design["Yt"])))
    return X[:, :d], X[:, d:]


DESIGNS = {
    # the kernel as built: split factors, tf32 (rounded) chain 1, split chain 2
    "built: F split, X rn, W rn, Yt split": dict(F="split", X="rn", W="rn", Yt="split"),
    "X trunc (A straight from the accumulator)": dict(F="split", X="trunc", W="rn", Yt="split"),
    "X trunc, W trunc": dict(F="split", X="trunc", W="trunc", Yt="split"),
    "F bf16": dict(F="bf16", X="rn", W="rn", Yt="split"),
    "Yt bf16": dict(F="split", X="rn", W="rn", Yt="bf16"),
    "X bf16, W bf16 (chain 1 in bf16)": dict(F="split", X="bf16", W="bf16", Yt="split"),
    "X split, W bf16": dict(F="split", X="split", W="bf16", Yt="split"),
    "X split, W split": dict(F="split", X="split", W="split", Yt="split"),
    "all bf16": dict(F="bf16", X="bf16", W="bf16", Yt="bf16"),
}


def rel(a, b):
    n = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / n) if n > 1e-30 else float(np.linalg.norm(a))


def study(tokens=8192, heads=4, variants=("gdn", "deltanet"), designs=None, seed=0):
    import oracle
    import synth_inputs as si
    designs = designs or list(DESIGNS)
    rows = []
    for variant in variants:
        W = si.workload(5, seed=seed, variant=variant, lengths=[tokens], h_k=max(1, heads // 2), h_v=heads,
                        seam_w=0)
        lay = W.layers[0]
        k, v, g, b = (None if x is None else x.double() for x in (lay.k, lay.v, lay.g, lay.beta))
        T, S = oracle.build_pairs(variant, W.seg_offsets, 0, W.h_k, W.h_v, 128, 128, k, v, g, b)
        for name in designs:
            eT = eS = 0.0
            for h in range(heads):
                kh = h * W.h_k // W.h_v
                gh = g[:, h] if g is not None else torch.zeros(tokens, dtype=torch.float64)
                Tc, Sc = build_emulated(k[:, kh], v[:, h], gh, b[:, h], DESIGNS[name])
                eT = max(eT, rel(Tc.numpy(), T[0, h]))
                eS = max(eS, rel(Sc.numpy(), S[0, h]))
            rows.append((variant, tokens, name, eT, eS))
    return rows


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--tokens", type=int, default=8192)
    ap.add_argument("--heads", type=int, default=4)
    ap.add_argument("--designs", nargs="*", default=None)
    a = ap.parse_args()
    torch.set_num_threads(os.cpu_count() or 1)
    print(f"| variant | tokens | design | worst T_C error | worst S(C|0) error |")
    print("|---|---|---|---|---|")
    for variant, tokens, name, eT, eS in study(a.tokens, a.heads, designs=a.designs):
        print(f"| {variant} | {tokens} | {name} | {eT:.2e} | {eS:.2e} |", flush=True)


if __name__ == "__main__":
    main()
