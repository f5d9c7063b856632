"""The unrolled adjoint of the delta-rule writes, restated in numpy, against
the oracle's write-by-write adjoint (oracle/armt_backward.py).

The backward kernels (csrc/backward.cuh) do not undo the M writes of a cell
one state at a time: every write is a rank-one update, so each product of a
state with a feature is expanded into the entry state (or the final state's
adjoint) plus earlier (or later) rank-one terms, with G = Phi Phi^T.  That
turns the reverse walk into a per-row recurrence over the rows of the state
plus M x M scalar work (section 二 of the summary page of "Diagonal Batching
Unlocks Parallelism in Recurrent Memory Transformers for Long Contexts"
defines the writes).  This test checks the expansion itself -- the formulas
the kernels evaluate, in the kernels' order -- against the sequential adjoint
of the oracle in fp64, including the zero-state case where the normaliser's
clip sits exactly at its upper end.
"""
import numpy as np
import pytest

from oracle import armt_backward as G
from oracle import armt_oracle as O

pytestmark = pytest.mark.oracle


def _unrolled(h_mem, wk, wv, wb, A0, z0, nu, eps, Abar, zbar):
    M = h_mem.shape[0]
    keys, vals = h_mem @ wk.T, h_mem @ wv.T
    beta = 1/(1+np.exp(-(h_mem @ wb)))
    Phi = O.dpfp(keys, nu)
    Gm = Phi @ Phi.T
    z0phi = Phi @ z0
    gam = np.zeros(M); D = np.zeros(M); Q = np.zeros(M); gu = np.zeros(M); zphi = np.zeros(M)
    for i in range(M):
        zp = z0phi[i] + sum(gam[j]*Gm[j,i] for j in range(i))
        Q[i] = Gm[i,i] + eps; gu[i] = 1 - zp/Q[i]; gam[i] = min(max(gu[i],0),1); D[i] = zp+eps; zphi[i]=zp
    d = A0.shape[0]
    C = np.zeros((M,d)); Vb = np.zeros((M,d)); CB = np.zeros((M,d)); Wv = np.zeros((M,d))
    a = A0.copy()
    for i in range(M):
        Vb[i] = (a @ Phi[i]) / D[i]
        C[i] = beta[i]*(vals[i]-Vb[i])
        a = a + np.outer(C[i], Phi[i])
    ab = Abar.copy()
    for i in reversed(range(M)):
        CB[i] = ab @ Phi[i]
        Wv[i] = -beta[i]*CB[i]/D[i]
        ab = ab + np.outer(Wv[i], Phi[i])
    Ain_bar = ab
    X = Wv @ C.T
    bbar = np.sum(CB*(vals-Vb), axis=1)
    e = np.sum(Wv*Vb, axis=1)
    zfp = Phi @ zbar
    zeta = np.zeros(M); dg = np.zeros(M)
    for i in reversed(range(M)):
        gb = zfp[i] + sum(zeta[j]*Gm[j,i] for j in range(i+1, M))
        gub = gb if 0 <= gu[i] <= 1 else 0.0
        zeta[i] = -e[i] - gub/Q[i]
        dg[i] = 2*gub*zphi[i]/Q[i]**2
    Coef = np.zeros((M,M))
    for i in range(M):
        for j in range(M):
            Coef[i,j] = (X[j,i] + gam[i]*zeta[j]) if j > i else ((X[i,j] + zeta[i]*gam[j]) if j < i else dg[i])
    PhiBar = C @ Abar + Wv @ A0 + Coef @ Phi + np.outer(gam, zbar) + np.outer(zeta, z0)
    kbar = G.dpfp_backward(keys, PhiBar, nu)
    vbar = beta[:,None]*CB
    logit_bar = bbar*beta*(1-beta)
    hbar = kbar @ wk + vbar @ wv + np.outer(logit_bar, wb)
    zin_bar = zbar + zeta @ Phi
    return hbar, kbar.T @ h_mem, vbar.T @ h_mem, logit_bar @ h_mem, Ain_bar, zin_bar


@pytest.mark.parametrize("trial", range(5))
def test_unrolled_write_adjoint_equals_sequential(trial):
    rng = np.random.default_rng(trial)
    M, d, k, nu = 8, 24, 6, 3
    P = 2 * k * nu
    h = rng.standard_normal((M, d))
    wk = rng.standard_normal((k, d)) * 0.3
    wv = rng.standard_normal((d, d)) * 0.3
    wb = rng.standard_normal(d) * 0.3
    A0 = rng.standard_normal((d, P)) * 0.1 if trial else np.zeros((d, P))
    z0 = np.abs(rng.standard_normal(P)) * 0.1 if trial else np.zeros(P)
    Abar, zbar = rng.standard_normal((d, P)), rng.standard_normal(P)
    ref = G.assoc_write_backward(h, wk, wv, wb, A0, z0, nu, 1e-6, Abar, zbar)
    got = _unrolled(h, wk, wv, wb, A0, z0, nu, 1e-6, Abar, zbar)
    for name, a, b in zip(("h", "wk", "wv", "wbeta", "A0", "z0"), got, ref):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12 * np.max(np.abs(b)), err_msg=name)
