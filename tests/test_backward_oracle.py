"""The fp64 gradient reference (oracle/armt_backward.py) against what fixes it
independently of itself: the numpy oracle's forward (values, and central
finite differences for directional derivatives), the schedule equivalence of
the summary page (section 二: the diagonal order computes exactly the
sequential recurrence), causality of the segment recurrence, and embedding
rows that no token uses."""
import dataclasses

import numpy as np
import pytest

from oracle import armt_backward as G
from oracle import armt_oracle as O
from recurrent_memory_transformer_gb300 import inputs as I

pytestmark = pytest.mark.oracle

torch = pytest.importorskip("torch")


def _setup(n_tok_short=0, seed=71, n_seg=3, over=None):
    cfg = dataclasses.replace(I.TINY, **(over or {}))
    W = I.make_weights(cfg, seed=seed, norm_jitter=0.1)
    tok = I.make_tokens(cfg, n_seg, seed=seed)
    tok = tok[:tok.shape[0] - n_tok_short]
    rng = np.random.default_rng(seed + 1)
    L, d, P = cfg.n_layers, cfg.d_model, cfg.phi_dim
    cot = {"hidden": rng.standard_normal((tok.shape[0], d)),
           "A": rng.standard_normal((L, d, P)), "z": rng.standard_normal((L, P))}
    return cfg, W, tok, n_seg, cot, rng


def test_restated_forward_matches_oracle():
    for short in (0, 5):
        cfg, W, tok, n, cot, rng = _setup(short)
        A0 = 0.01 * np.abs(rng.standard_normal((cfg.n_layers, cfg.d_model, cfg.phi_dim)))
        z0 = 0.01 * np.abs(rng.standard_normal((cfg.n_layers, cfg.phi_dim)))
        ho, Ao, zo = O.forward(cfg, W, tok, n, A0=A0, z0=z0)
        Wt = {k: G._t(W[k]) for k in G.WEIGHT_KEYS}
        ht, At, zt = G.forward(cfg, Wt, tok, n, "seq", G._t(A0), G._t(z0))
        for a, b in ((ht, ho), (At, Ao), (zt, zo)):
            b = np.asarray(b)
            np.testing.assert_allclose(a.numpy(), b, rtol=1e-10, atol=1e-12 * np.abs(b).max())


@pytest.mark.parametrize("key", ["embed", "mem", "wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down",
                                 "a_wq", "a_wk", "a_wv", "a_wbeta", "norm1", "norm2", "norm_f", "A0", "z0"])
def test_directional_derivative_matches_central_differences(key):
    # d/de loss(x + e V) from the gradient vs (loss(x + e V) - loss(x - e V)) / 2e
    # computed with the numpy oracle's forward (an implementation the gradient
    # code does not use); a nonzero initial state exercises the state path
    cfg, W, tok, n, cot, rng = _setup(3, seed=72)
    A0 = 0.01 * np.abs(rng.standard_normal((cfg.n_layers, cfg.d_model, cfg.phi_dim)))
    z0 = 0.05 * np.abs(rng.standard_normal((cfg.n_layers, cfg.phi_dim)))
    _, grads = G.gradients(cfg, W, tok, n, cot, "seq", A0, z0)
    base = {"A0": A0, "z0": z0}
    x0 = np.asarray(base[key] if key in base else W[key], np.float64)
    V = rng.standard_normal(x0.shape)
    if key == "z0":
        V = np.abs(V)          # keep the normaliser non-negative on both sides
    # small steps: the DPFP features have relu kinks, and a step that carries a
    # query or key component across zero measures the average slope of two
    # pieces (1e-5 does so for the query projection here; 1e-7 agrees to 2e-10)
    eps = 1e-7 * max(1.0, float(np.abs(x0).max())) / max(1.0, float(np.abs(V).max()))

    def loss_at(x):
        Wk, A, z = dict(W), A0, z0
        if key == "A0":
            A = x
        elif key == "z0":
            z = x
        else:
            Wk[key] = x
        return G.loss_value(O.forward(cfg, Wk, tok, n, A0=A, z0=z), cot)

    fd = (loss_at(x0 + eps * V) - loss_at(x0 - eps * V)) / (2 * eps)
    an = float(np.sum(grads[key] * V))
    assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (key, fd, an)


def test_diagonal_and_sequential_orders_give_the_same_gradients():
    cfg, W, tok, n, cot, rng = _setup(0, seed=73, n_seg=4, over={"n_layers": 3})
    ls, gs = G.gradients(cfg, W, tok, n, cot, "seq")
    ld, gd = G.gradients(cfg, W, tok, n, cot, "diag")
    assert abs(ls - ld) <= 1e-12 * max(1.0, abs(ls))
    for k in G.WEIGHT_KEYS:
        np.testing.assert_allclose(gd[k], gs[k], rtol=1e-11, atol=1e-13 * max(1.0, np.abs(gs[k]).max()))


def test_gradients_respect_causality_and_unused_embedding_rows():
    cfg, W, tok, n, cot, rng = _setup(0, seed=74, n_seg=3)
    S = cfg.seg_len
    # only segment 0's outputs in the loss: tokens of later segments cannot matter
    cot0 = {"hidden": cot["hidden"].copy(), "A": np.zeros_like(cot["A"]), "z": np.zeros_like(cot["z"])}
    cot0["hidden"][S:] = 0.0
    _, g = G.gradients(cfg, W, tok, n, cot0, "diag")
    later = np.setdiff1d(np.unique(tok[S:]), np.unique(tok[:S]))
    assert later.size > 0
    assert np.all(g["embed"][later] == 0.0)
    # with every output in the loss, rows of ids that appear nowhere get no gradient
    _, g = G.gradients(cfg, W, tok, n, cot, "diag")
    unused = np.setdiff1d(np.arange(cfg.vocab), np.unique(tok))
    assert unused.size > 0 and np.all(g["embed"][unused] == 0.0)
    assert np.abs(g["embed"][np.unique(tok)]).max() > 0.0


@pytest.mark.parametrize("short,over", [(0, {"n_layers": 3}), (5, {})])
def test_backward_by_reverse_diagonals_equals_whole_graph_gradient(short, over):
    # the schedule a diagonal-batched backward pass follows -- reverse
    # anti-diagonals, per-cell vector-Jacobian products passing adjoints to
    # (l-1, s) and (l, s-1) -- gives the gradient of the whole graph
    cfg, W, tok, n, cot, rng = _setup(short, seed=75, n_seg=4, over=over)
    A0 = 0.01 * np.abs(rng.standard_normal((cfg.n_layers, cfg.d_model, cfg.phi_dim)))
    z0 = 0.05 * np.abs(rng.standard_normal((cfg.n_layers, cfg.phi_dim)))
    _, whole = G.gradients(cfg, W, tok, n, cot, "diag", A0, z0)
    diag = G.backward_by_diagonals(cfg, W, tok, n, cot, A0, z0)
    assert set(diag) == set(whole)
    for k in whole:
        np.testing.assert_allclose(diag[k], whole[k], rtol=1e-10,
                                   atol=1e-12 * max(1.0, float(np.abs(whole[k]).max())), err_msg=k)


def _t64(a):
    return torch.tensor(np.asarray(a, np.float64), dtype=torch.float64, requires_grad=True)


def test_explicit_adjoints_of_dpfp_and_the_read_match_autograd():
    rng = np.random.default_rng(76)
    R, d, k, nu, eps = 7, 24, 8, 3, 1e-6
    P = 2 * k * nu
    x = rng.standard_normal((R, d))
    wq = 0.3 * rng.standard_normal((k, d))
    A = 0.2 * rng.standard_normal((d, P))
    z = np.abs(rng.standard_normal(P))
    y_bar = rng.standard_normal((R, d))
    q = x @ wq.T
    phi_bar = rng.standard_normal((R, P))
    qt = _t64(q)
    (G.dpfp(qt, nu) * torch.tensor(phi_bar)).sum().backward()
    np.testing.assert_allclose(G.dpfp_backward(q, phi_bar, nu), qt.grad.numpy(), rtol=1e-12, atol=1e-12)
    xt, wt, At, zt = _t64(x), _t64(wq), _t64(A), _t64(z)
    (G.assoc_read(xt, wt, At, zt, nu, eps) * torch.tensor(y_bar)).sum().backward()
    got = G.assoc_read_backward(x, wq, A, z, nu, eps, y_bar)
    for g, t in zip(got, (xt, wt, At, zt)):
        np.testing.assert_allclose(g, t.grad.numpy(), rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("z_scale", [0.0, 0.05, 5.0])   # zero state (gamma = 1), interior, clipped (gamma = 0)
def test_explicit_adjoint_of_the_in_order_writes_matches_autograd(z_scale):
    rng = np.random.default_rng(77)
    M, d, k, nu, eps = 5, 16, 8, 3, 1e-6
    P = 2 * k * nu
    h = rng.standard_normal((M, d))
    wk, wv = 0.4 * rng.standard_normal((k, d)), 0.3 * rng.standard_normal((d, d))
    wb = 0.3 * rng.standard_normal(d)
    A0 = 0.1 * rng.standard_normal((d, P))
    z0 = z_scale * np.abs(rng.standard_normal(P))
    A_bar, z_bar = rng.standard_normal((d, P)), rng.standard_normal(P)
    ht, wkt, wvt, wbt, At, zt = (_t64(a) for a in (h, wk, wv, wb, A0, z0))
    keys, values = ht @ wkt.T, ht @ wvt.T
    beta = torch.sigmoid(ht @ wbt)
    Aw, zw = At, zt
    for i in range(M):
        Aw, zw = G.delta_rule_write(Aw, zw, keys[i], values[i], beta[i], nu, eps)
    ((Aw * torch.tensor(A_bar)).sum() + (zw * torch.tensor(z_bar)).sum()).backward()
    got = G.assoc_write_backward(h, wk, wv, wb, A0, z0, nu, eps, A_bar, z_bar)
    for g, t in zip(got, (ht, wkt, wvt, wbt, At, zt)):
        np.testing.assert_allclose(g, t.grad.numpy(), rtol=1e-9, atol=1e-9 * max(1.0, float(np.abs(g).max())))
    # the forward the adjoint walks back is the oracle's own
    A1, z1 = O.assoc_write(h, wk, wv, wb, A0, z0, nu, eps)
    np.testing.assert_allclose(A1, Aw.detach().numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("short,over", [(0, {"n_layers": 3}), (5, {}),
                                        (0, {"n_q_heads": 4, "n_kv_heads": 2, "head_dim": 16})])
def test_explicit_backward_equals_whole_graph_gradient(short, over):
    # the whole backward pass written out with explicit adjoints (RMSNorm,
    # RoPE, causal GQA attention, SwiGLU, read, in-order writes), cell by cell
    # in reverse diagonal order
    cfg, W, tok, n, cot, rng = _setup(short, seed=78, n_seg=3, over=over)
    A0 = 0.01 * np.abs(rng.standard_normal((cfg.n_layers, cfg.d_model, cfg.phi_dim)))
    z0 = 0.05 * np.abs(rng.standard_normal((cfg.n_layers, cfg.phi_dim)))
    _, whole = G.gradients(cfg, W, tok, n, cot, "diag", A0, z0)
    expl = G.backward_explicit(cfg, W, tok, n, cot, A0, z0)
    assert set(expl) == set(whole)
    for k in whole:
        np.testing.assert_allclose(expl[k], whole[k], rtol=1e-9,
                                   atol=1e-11 * max(1.0, float(np.abs(whole[k]).max())), err_msg=k)
