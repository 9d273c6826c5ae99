"""Dense-matrix restatement of the per-token transitions, for tiny cases.

TEST INFRASTRUCTURE ONLY (a pin for the C oracle).  Where the C oracle
applies T_t through rank-1 updates, this module forms every T_t and U_t as an
explicit matrix, straight from its definition, and multiplies them in token
order: T_C = T_L ... T_1 and S(C|0) = sum_t (T_L ... T_{t+1}) U_t, which is
"the product of every token transition matrix in the segment" of the HYPIC
news pages (nav.aitube.vip §2.1; xix.ai paragraph on linear layers).
"""
from __future__ import annotations

import numpy as np


def token_matrices(variant, k, v, g, beta, t, h, h_k, h_v):
    """(T_t, U_t) of value head h at token t as dense fp64 matrices."""
    kh = (h * h_k) // h_v
    kv = np.asarray(k[t, kh], dtype=np.float64)
    vv = np.asarray(v[t, h], dtype=np.float64)
    d_k = kv.shape[0]
    I = np.eye(d_k)
    E = None
    if variant in ("gdn", "deltanet", "channel"):
        b = float(beta[t, h])
        E = I - b * np.outer(kv, kv)
        U = b * np.outer(kv, vv)
    else:
        U = np.outer(kv, vv)
    if variant == "gdn":
        T = np.exp(float(g[t, h])) * E
    elif variant == "deltanet":
        T = E
    elif variant == "channel":
        T = E @ np.diag(np.exp(np.asarray(g[t, h], dtype=np.float64)))
    elif variant == "scalar":
        T = np.exp(float(g[h])) * I
    elif variant == "ungated":
        T = I.copy()
    elif variant == "diag":
        T = np.diag(np.exp(np.asarray(g[t, h], dtype=np.float64)))
    else:
        raise ValueError(variant)
    return T, U


def pair(variant, k, v, g, beta, start, end, h, h_k, h_v):
    """Dense (T_C, S(C|0)) over tokens [start, end) for value head h."""
    d_k = k.shape[-1]
    d_v = v.shape[-1]
    Ts, Us = [], []
    for t in range(start, end):
        T, U = token_matrices(variant, k, v, g, beta, t, h, h_k, h_v)
        Ts.append(T)
        Us.append(U)
    T_C = np.eye(d_k)
    for T in Ts:                      # T_C = T_L ... T_1: each new token on the left
        T_C = T @ T_C
    S = np.zeros((d_k, d_v))
    for i, U in enumerate(Us):        # S(C|0) = sum_t (T_L ... T_{t+1}) U_t
        P = np.eye(d_k)
        for T in Ts[i + 1:]:
            P = T @ P
        S = S + P @ U
    return T_C, S


def outputs(variant, k, v, q, g, beta, h, h_k, h_v, S0=None):
    """Every o_t = S_t^T q_t of value head h over all tokens, and the final
    state, with S_t = T_t S_{t-1} + U_t formed from dense matrices."""
    N, _, d_k = k.shape
    d_v = v.shape[-1]
    S = np.zeros((d_k, d_v)) if S0 is None else np.array(S0, dtype=np.float64)
    kh = (h * h_k) // h_v
    outs = []
    for t in range(N):
        T, U = token_matrices(variant, k, v, g, beta, t, h, h_k, h_v)
        S = T @ S + U
        outs.append(S.T @ np.asarray(q[t, kh], dtype=np.float64))
    return np.array(outs), S
