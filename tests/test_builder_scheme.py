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
The final l x l eigenproblem runs either through a library eigensolver or
through the bf16 builder's own method (one-sided Jacobi on the Cholesky
factor with tracked norms, float32): ~1e-5 and ~1e-4 of the oracle's U W^T
on the longctx shape.
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


def _jacobi_eig(G, sweeps=20):
    """The eigen stage as the bf16 builder runs it, in float32: G = R^T R by
    the Cholesky with dependent-column dropping, then one-sided (Hestenes)
    Jacobi on the rows of R with round-robin pairs; the squared row norms are
    recomputed at each sweep's start and updated by every rotation, and a
    pair rotates while |y_p . y_q| > max(1e-7 sqrt(a_pp a_qq), 2e-7 max a).
    Eigenvalues are the squared norms, eigenvectors the normalised rows,
    sorted by descending eigenvalue (ties to the lower index)."""
    f32 = np.float32
    R, _ = _chol_drop(np.asarray(G, np.float32))
    Y = np.asarray(R, np.float32).copy()              # row p = y_p
    l = Y.shape[0]
    n = (l + 1) & ~1
    for _ in range(sweeps):
        nrm = np.array([f32(np.dot(Y[p], Y[p])) for p in range(l)], np.float32)
        abs_tol = f32(2e-7) * nrm.max()
        rotated = False
        for rnd in range(n - 1):
            for k in range(n // 2):
                if k == 0:
                    pa, pb = n - 1, rnd
                else:
                    pa, pb = (rnd + k) % (n - 1), (rnd - k + n - 1) % (n - 1)
                pa, pb = min(pa, pb), max(pa, pb)
                if pb >= l:
                    continue
                u, v = Y[pa].copy(), Y[pb].copy()
                app, aqq = nrm[pa], nrm[pb]
                apq = f32(np.dot(u, v))
                if abs(apq) > max(f32(1e-7) * np.sqrt(app * aqq), abs_tol):
                    th = (aqq - app) / (f32(2) * apq)
                    t = np.copysign(f32(1), th) / (abs(th) + np.sqrt(th * th + f32(1)))
                    c = f32(1) / np.sqrt(t * t + f32(1))
                    sn = t * c
                    Y[pa] = c * u - sn * v
                    Y[pb] = sn * u + c * v
                    nrm[pa] = app - t * apq
                    nrm[pb] = aqq + t * apq
                    rotated = True
        if not rotated:
            break
    lam = np.array([np.dot(Y[p].astype(np.float64), Y[p]) for p in range(l)])
    order = sorted(range(l), key=lambda p: (-lam[p], p))
    Ub = np.stack([Y[p] / np.sqrt(lam[p]) if lam[p] > 0 else np.zeros(l, np.float32)
                   for p in order], axis=1)
    return lam[order], Ub


def _feature_side_state(E1, E0, r, omega, q, eig="eigh"):
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
    if eig == "jacobi":
        lam, Ub = _jacobi_eig(Bt.T @ Bt)
    else:
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


@pytest.mark.parametrize("eig", ["eigh", "jacobi"])
@pytest.mark.parametrize("case", ["longctx-bf16", "tiny-noise-free"])
def test_feature_side_iteration_matches_hmt(case, eig):
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
        U, W = _feature_side_state(E1, E0, r, om, q, eig)
        assert O.relative_error(U @ W.T, Uo @ Wo.T) <= 1e-3


def _chol_inv_inplace(A):
    """The l x l stage of the bf16 builder on one float32 array, in its step
    order: right-looking Cholesky in place (pivot row scaled by -1/pivot,
    a pivot at or below 1e-6 of its column's original diagonal drops the
    column), then the in-place back substitution whose step i first updates
    the columns k > i from column i of R and then turns column i into column
    i of the inverse.  Returns (R, R^-1, keep)."""
    f32 = np.float32
    A = np.array(A, np.float32)
    l = A.shape[0]
    gd = np.diag(A).copy()
    A = np.triu(A)
    keep = np.zeros(l, bool)
    dinv = np.zeros(l, np.float32)
    for j in range(l):
        piv = A[j, j]
        ok = gd[j] > 0 and piv > f32(1e-6) * gd[j]
        inv2 = f32(1) / piv if ok else f32(0)
        keep[j] = ok
        dinv[j] = f32(1) / np.sqrt(piv) if ok else f32(0)
        prow = -A[j, j + 1:] * inv2
        for k in range(j + 1, l):
            A[j + 1:k + 1, k] = prow[:k - j] * A[j, k] + A[j + 1:k + 1, k]
    A = A * dinv[:, None]
    R = A.copy()
    diag = np.diag(R).copy()
    for i in range(l - 1, -1, -1):
        inv = f32(1) / diag[i] if keep[i] else f32(0)
        col = A[:i, i].copy()
        for k in range(i + 1, l):
            xi = A[i, k] * inv
            A[:i, k] = -col * xi + A[:i, k]
        A[:i, i] = -col * inv
        A[i, i] = f32(1) if keep[i] else f32(0)
    scale = np.where(keep, f32(1) / np.where(keep, diag, f32(1)), f32(0)).astype(np.float32)
    return R, np.triu(A) * scale[:, None], keep


@pytest.mark.parametrize("l", [8, 21, 40, 64])
def test_inplace_cholesky_and_inverse(l):
    """G = R^T R on the kept columns, R^-1 R = I there, dropped indices give
    zero rows and columns of R^-1, and both factors are upper triangular --
    on Grams of graded columns with one exactly dependent column."""
    rng = np.random.default_rng(l)
    X = rng.standard_normal((200, l)) * np.geomspace(1.0, 1e-2, l)
    X[:, l // 2] = X[:, l // 2 - 1]                      # a dependent column
    G = (X.T @ X).astype(np.float32)
    R, Ri, keep = _chol_inv_inplace(G)
    assert keep.sum() == l - 1 and not keep[l // 2]
    kept = np.flatnonzero(keep)
    Rk = R[np.ix_(kept, kept)].astype(np.float64)
    assert np.abs(Rk.T @ Rk - G[np.ix_(kept, kept)]).max() <= 1e-5 * np.abs(G).max()
    assert np.abs(Ri[np.ix_(kept, kept)].astype(np.float64) @ Rk - np.eye(len(kept))).max() <= 1e-3
    assert np.all(Ri[~keep, :] == 0) and np.all(Ri[:, ~keep] == 0)
    assert np.all(np.tril(R, -1) == 0) and np.all(np.tril(Ri, -1) == 0)
