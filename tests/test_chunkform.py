"""The chunk algebra used by the tensor-core build reaches the token-by-token
definition (fp64, several chunks with a ragged tail, every variant)."""
import numpy as np
import pytest

import oracle
import oracle_pins as pins
from chunkform import build_chunked


@pytest.mark.parametrize("variant", pins.ALL)
@pytest.mark.parametrize("chunk", [4, 7, 64])
def test_chunk_form_equals_token_form(variant, chunk):
    N, h_k, h_v, d_k, d_v = 37, 2, 4, 6, 5
    k, v, q, g, beta = pins.tiny_inputs(variant, N, h_k, h_v, d_k, d_v, 900)
    off = [0, 3, 30, N]
    T, S = oracle.build_pairs(variant, off, 0, h_k, h_v, d_k, d_v, k, v, g, beta)
    for i in range(3):
        for h in range(h_v):
            Tc, Sc = build_chunked(variant, k, v, g, beta, off[i], off[i + 1], h, h_k, h_v, chunk=chunk)
            assert np.abs(Tc.numpy() - T[i, h]).max() < 1e-12
            assert np.abs(Sc.numpy() - S[i, h]).max() < 1e-12 * max(1.0, np.abs(S[i, h]).max())


@pytest.mark.parametrize("m,sb", [(32, 16), (29, 16), (64, 16)])
def test_subblock_gram_equals_direct(m, sb):
    """The per-channel decayed Gram as the kernel forms it (sub-block
    references) equals the direct definition."""
    import torch
    from chunkform import gram_subblocks
    gen = torch.Generator().manual_seed(7)
    K = torch.randn(m, 8, generator=gen, dtype=torch.float64)
    g = -torch.nn.functional.softplus(torch.randn(m, 8, generator=gen, dtype=torch.float64))
    lam = torch.cumsum(g, 0)
    E = torch.exp(lam[:, None, :] - lam[None, :, :])
    direct = torch.tril(torch.einsum("tc,ic,tic->ti", K, K, E), -1)
    got = gram_subblocks(K, lam, sb)
    assert torch.allclose(got, direct, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("m", [32, 64])
def test_block_inverse_schedule(m):
    """The preparation group's block schedule for A = (I + N)^{-1} (the
    diagonal blocks, then A_10 and A_32, then the P blocks and the lower-left
    quarter) equals the inverse, and reads no block above the diagonal."""
    import torch
    from chunkform import block_inverse
    gen = torch.Generator().manual_seed(11)
    K = torch.nn.functional.normalize(torch.randn(m, 128, generator=gen, dtype=torch.float64), dim=1)
    beta = torch.sigmoid(torch.randn(m, generator=gen, dtype=torch.float64))
    lam = torch.cumsum(-torch.rand(m, generator=gen, dtype=torch.float64) * 0.1, 0)
    N = torch.tril(beta[:, None] * torch.exp(lam[:, None] - lam[None, :]) * (K @ K.T), -1)
    A = block_inverse(N)
    assert not torch.isnan(A).any()
    eye = torch.eye(m, dtype=torch.float64)
    assert torch.allclose(A, torch.linalg.inv(eye + N), rtol=1e-12, atol=1e-12)
    assert torch.allclose((eye + N) @ A, eye, atol=1e-12)
