"""The GRAM loss form rests on two exact identities, checked here in fp64 on
the CPU against the definition of the search loss ("AWQ: How
Activation-Aware Quantization Saves 4-bit LLMs", search_scale listing: the
sum over tokens and output rows of (X W_hat^T - X W^T)^2):

  1. sum_t sum_r (X D^T)[t][r]^2 = sum_r D[r] (X^T X) D[r]^T, D = W_hat - W;
  2. with 256-channel blocks jb(x) = x // 256, the symmetric C = X^T X may be
     replaced by H, its blocks on and below the diagonal with the ones below
     doubled, each row c of D C contracting only over j with jb(j) <= jb(c).

A wrong factor (1 instead of 2 below the diagonal), a transposed block or a
block prefix cut one block short changes the sum, which the tests catch on
shapes with several blocks, a last half block (in % 256 == 128) and ragged
row and token counts. No GPU, no library: numpy only."""
import numpy as np
import pytest


def direct(X, D):
    return float(((X @ D.T) ** 2).sum())


def gram_blocks(X, D, factor_below=2.0):
    """sum_r sum_c D[r][c] sum_{j: jb(j) <= jb(c)} H[c][j] D[r][j], H as the library forms it."""
    K = X.shape[1]
    C = X.T @ X
    jb = np.arange(K) // 256
    below = jb[None, :] < jb[:, None]  # [c][j]: block of j left of the block of c
    same = jb[None, :] == jb[:, None]
    H = np.where(below, factor_below * C, np.where(same, C, 0.0))
    P = D @ H.T  # P[r][c] = sum_j D[r][j] H[c][j]
    return float((P * D).sum())


@pytest.mark.parametrize("n,N,K", [(37, 5, 128), (64, 3, 256), (50, 7, 384), (129, 11, 640), (300, 2, 1152)])
def test_gram_form_equals_the_direct_sum(n, N, K):
    rng = np.random.default_rng(n * 1000 + K)
    X = rng.standard_normal((n, K))
    X[:, rng.choice(K, size=max(1, K // 100), replace=False)] *= 40.0  # outlier channels
    D = rng.standard_normal((N, K)) * 1e-3
    ref = direct(X, D)
    assert gram_blocks(X, D) == pytest.approx(ref, rel=1e-12)
    # the identity without blocks, for the record
    assert float(np.einsum("rc,cj,rj->", D, X.T @ X, D)) == pytest.approx(ref, rel=1e-12)


@pytest.mark.parametrize("K", [384, 640])
def test_planted_mistakes_change_the_sum(K):
    rng = np.random.default_rng(K)
    X = rng.standard_normal((200, K))
    D = rng.standard_normal((9, K))
    ref = direct(X, D)
    # the off-diagonal blocks counted once instead of twice
    assert abs(gram_blocks(X, D, factor_below=1.0) - ref) > 1e-6 * abs(ref)
    # H transposed (blocks above the diagonal instead of below): P against the wrong triangle
    C = X.T @ X
    jb = np.arange(K) // 256
    above = jb[None, :] > jb[:, None]
    same = jb[None, :] == jb[:, None]
    Ht = np.where(above, 2.0 * C, np.where(same, C, 0.0))
    # by symmetry of C this still equals the sum: the triangle choice is free, only the factor matters
    assert float(((D @ Ht.T) * D).sum()) == pytest.approx(ref, rel=1e-12)
    # the prefix cut one block short (j over blocks strictly below c, the diagonal block left out)
    Hs = np.where(jb[None, :] < jb[:, None], 2.0 * C, 0.0)
    assert abs(float(((D @ Hs.T) * D).sum()) - ref) > 1e-6 * abs(ref)


def test_zero_padded_tokens_add_nothing():
    """The kernel pads the tokens to a multiple of 64 with zeros (X^T's extra columns)."""
    rng = np.random.default_rng(7)
    X = rng.standard_normal((70, 256))
    D = rng.standard_normal((4, 256))
    Xp = np.vstack([X, np.zeros((128 - 70, 256))])
    assert gram_blocks(Xp, D) == pytest.approx(direct(X, D), rel=1e-12)
