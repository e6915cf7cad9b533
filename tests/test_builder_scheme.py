"""The tensor-core builder's reformulation of randomized subspace iteration,
checked on the CPU against the oracle (HMT Algorithm 4.4 with Householder QR).

The kernel never forms the n x l iterates: with M = delta^T delta it uses
Y^T Y = X^T M X for the implicit CholeskyQR of Y = delta X, delta^T Q =
M X R_Y^-1 for the next iterate, B^T = delta^T Q for the small SVD, and U =
delta (X R_Y^-1 Ub_r diag(sigma_r)).  The spans, and so U W^T, equal the
oracle's in exact arithmetic.  This test replays that sequence in NumPy --
M accumulated from the hi/lo bf16 split of the delta (RNE; hi.hi + hi.lo +
lo.hi, as the tensor-core Gram forms it), fp32 elsewhere,
Cholesky with dependent-column dropping -- and requires U W^T within 1e-3 of
the oracle's (the GPU tolerance is 2e-2 for bf16), on the longctx shape
(geometric spectrum, bf16 caches) and the noise-free planted tiny delta.
The model is test code: it shares nothing with the CUDA library.
"""
import numpy as np
import pytest

import oracle as O


def _bf16(x):
    """Round float32 values to bfloat16 (round to nearest, ties to even)."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return b.astype(np.uint32).view(np.float32)


def _chol_drop(G):
    l = G.shape[0]
    R = np.zeros_like(G)
    keep = np.zeros(l, bool)
    for j in range(l):
        piv = G[j, j] - np.dot(R[:j, j], R[:j, j])
        keep[j] = G[j, j] > 0 and piv > 1e-6 * G[j, j]
        if keep[j]:
            R[j, j] = np.sqrt(piv)
            R[j, j + 1:] = (G[j, j + 1:] - R[:j, j] @ R[:j, j + 1:]) / R[j, j]
    return R, keep


def _rinv(R, keep):
    l = R.shape[0]
    Ri = np.zeros_like(R)
    for i in range(l):
        x = np.zeros(l, R.dtype)
        for j in range(l):
            v = (1.0 if i == j else 0.0) - x[:j] @ R[:j, j]
            x[j] = v / R[j, j] if keep[j] else 0.0
        Ri[i] = x
    return Ri


def _orth(X, G):
    R, keep = _chol_drop(G)
    return X @ _rinv(R, keep).astype(X.dtype)


def _feature_side_state(E1, E0, r, omega, q):
    D = np.asarray(E1, np.float32) - np.asarray(E0, np.float32)
    hi = _bf16(D)
    lo = _bf16(D - hi)
    # the bf16 kernel's three products (the lo.lo term is left out)
    M = (hi.T.astype(np.float64) @ hi + hi.T.astype(np.float64) @ lo
         + lo.T.astype(np.float64) @ hi).astype(np.float32)
    X = np.asarray(omega, np.float32)
    for _ in range(q):
        G = X.T @ (M @ X)                               # Y^T Y
        R1, k1 = _chol_drop(G)
        Z = (M @ X) @ _rinv(R1, k1)                      # delta^T Q
        X = _orth(Z, Z.T @ Z)
    MX = M @ X
    G = X.T @ MX
    R1, k1 = _chol_drop(G)
    Ri1 = _rinv(R1, k1)
    R2, k2 = _chol_drop(Ri1.T @ G @ Ri1)                 # CholeskyQR2, second pass
    RiY = Ri1 @ _rinv(R2, k2)
    Bt = MX @ RiY                                        # B^T = delta^T Q
    lam, Ub = np.linalg.eigh(Bt.T @ Bt)
    order = np.argsort(-lam)
    lam, Ub = np.maximum(lam[order], 0.0), Ub[:, order]
    s = np.sqrt(lam[:r])
    W = (Bt @ Ub[:, :r]) / np.where(s > 1e-6 * s[0], s, np.inf)
    U = D @ ((X @ RiY @ Ub[:, :r]) * s)
    return U, W


def _haar(rng, n, m):
    q, rr = np.linalg.qr(rng.standard_normal((n, m)))
    return q * np.sign(np.diag(rr))


@pytest.mark.parametrize("case", ["longctx-bf16", "tiny-noise-free"])
def test_feature_side_iteration_matches_hmt(case):
    rng = np.random.default_rng(7)
    if case == "longctx-bf16":
        T, d, r, p, q = 512, 128, 32, 8, 2
        spec, noise = 21.6 * 0.85 ** np.arange(d), 0.02
    else:
        T, d, r, p, q = 256, 64, 8, 8, 2
        spec, noise = np.array([2.0, 1.0, 0.5, 0.25]), 0.0
    m = min(len(spec), d)
    for _ in range(2):
        ref = rng.standard_normal((T, d))
        D = (_haar(rng, T, m) * spec[:m]) @ _haar(rng, d, m).T + noise * rng.standard_normal((T, d))
        if case == "longctx-bf16":
            E0 = _bf16(ref).astype(np.float64)
            E1 = _bf16(E0 + D).astype(np.float64)
        else:
            E0 = np.float32(ref).astype(np.float64)
            E1 = np.float32(E0 + D).astype(np.float64)
        om = rng.standard_normal((d, r + p))
        Uo, Wo, _, _ = O.build_unit(E1, E0, r, om, q)
        U, W = _feature_side_state(E1, E0, r, om, q)
        assert O.relative_error(U @ W.T, Uo @ Wo.T) <= 1e-3
