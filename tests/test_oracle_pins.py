"""Pins for the fp64 oracle against facts fixed by the pages and by mathematics.

Every check here compares the oracle with something other than itself: a
closed form, a brute-force loop written differently, a special case that
reduces to an independently written plain transformer, or an invariant the
method must satisfy (the diagonal order reaching the sequential result
exactly: summary page of "Diagonal Batching Unlocks Parallelism in Recurrent
Memory Transformers for Long Contexts", sections 二 and 五).
"""
import dataclasses
import math

import numpy as np
import pytest

from oracle import armt_oracle as O
from recurrent_memory_transformer_gb300 import inputs as I
from tests import plain_bf16_cell
from tests.plain_llama import plain_layer, plain_stack

pytestmark = pytest.mark.oracle


# ---------------------------------------------------------------- DPFP ----

def _dpfp_loops(x, nu):
    k = len(x)
    r = [max(v, 0.0) for v in x] + [max(-v, 0.0) for v in x]
    n = 2 * k
    out = []
    for j in range(1, nu + 1):
        for i in range(n):
            out.append(r[i] * r[(i - j) % n])
    return np.array(out)


def test_dpfp_shape_and_sign():
    rng = np.random.default_rng(0)
    for k, nu in ((16, 3), (64, 3), (5, 2)):
        x = rng.standard_normal((7, k))
        phi = O.dpfp(x, nu)
        assert phi.shape == (7, 2 * k * nu)
        assert (phi >= 0).all()
    assert O.dpfp(np.zeros(16), 3).shape == (96,)
    assert O.dpfp(np.zeros(64), 3).shape == (384,)


def test_dpfp_brute_force():
    rng = np.random.default_rng(1)
    for _ in range(5):
        x = rng.standard_normal(6)
        np.testing.assert_array_equal(O.dpfp(x, 3), _dpfp_loops(list(x), 3))


def test_dpfp_closed_form_adjacent_pair():
    # x = [a, b, 0, ...]: r has a at 0 and b at 1, so only block j=1 at index 1
    # holds r_1 * r_0 = a*b; this fixes the roll direction.
    a, b, k = 1.5, 0.25, 8
    x = np.zeros(k); x[0], x[1] = a, b
    phi = O.dpfp(x, 3)
    expect = np.zeros(2 * k * 3); expect[1] = a * b
    np.testing.assert_array_equal(phi, expect)


def test_dpfp_closed_form_wraparound():
    # x_{k-1} = a > 0 puts a at r_{k-1}; x_0 = -b puts b at r_k: adjacent in r,
    # so block 1 holds a*b at index k.  x = [c] * ... at both ends of r wraps:
    # r_{2k-1} = relu(-x_{k-1}) and r_0 = relu(x_0) meet at index 0 of block 1.
    k, a, b = 4, 2.0, 3.0
    x = np.zeros(k); x[k - 1], x[0] = a, -b
    phi = O.dpfp(x, 2)
    expect = np.zeros(2 * k * 2); expect[k] = a * b
    np.testing.assert_array_equal(phi, expect)
    x = np.zeros(k); x[k - 1], x[0] = -a, b
    phi = O.dpfp(x, 2)
    expect = np.zeros(2 * k * 2); expect[0] = a * b
    np.testing.assert_array_equal(phi, expect)


# ---------------------------------------------------------- row blocks ----

def test_rmsnorm_closed_form():
    c, eps, d = 0.3, 1e-5, 10
    g = np.arange(1, d + 1, dtype=float)
    out = O.rmsnorm(np.full(d, c), g, eps)
    np.testing.assert_allclose(out, c / math.sqrt(c * c + eps) * g, rtol=1e-15)


def test_silu_sigmoid_closed_forms():
    from scipy.special import expit
    x = np.linspace(-8, 8, 101)
    np.testing.assert_allclose(O.sigmoid(x), expit(x), rtol=1e-14)
    np.testing.assert_allclose(O.silu(x), x * expit(x), rtol=1e-13, atol=1e-300)


def test_rope_identity_norm_relative():
    rng = np.random.default_rng(2)
    T, H, hd = 9, 3, 8
    x = rng.standard_normal((T, H, hd))
    y = O.rope_rotate_half(x, 10000.0)
    np.testing.assert_array_equal(y[0], x[0])                       # position 0
    half = hd // 2
    pn = lambda a: a[..., :half] ** 2 + a[..., half:] ** 2
    np.testing.assert_allclose(pn(y), pn(x), rtol=1e-12)            # pairwise norms
    # <R_t q, R_u k> depends only on t - u
    q = rng.standard_normal(hd); kk = rng.standard_normal(hd)
    Q = O.rope_rotate_half(np.tile(q, (T, 1, 1)), 10000.0)[:, 0]
    K = O.rope_rotate_half(np.tile(kk, (T, 1, 1)), 10000.0)[:, 0]
    for t, u in ((5, 3), (7, 5), (2, 0)):
        np.testing.assert_allclose(Q[t] @ K[u], Q[8] @ K[6], rtol=1e-10)
    # explicit angle for pair 1 at position 3
    th = 3 * 10000.0 ** (-2.0 / hd)
    np.testing.assert_allclose(y[3, 0, 1], x[3, 0, 1] * math.cos(th) - x[3, 0, 1 + half] * math.sin(th))


def test_attention_special_cases():
    rng = np.random.default_rng(3)
    T, Hq, Hkv, hd = 6, 4, 2, 4
    q = rng.standard_normal((T, Hq, hd)); k = rng.standard_normal((T, Hkv, hd))
    v = rng.standard_normal((T, Hkv, hd))
    out = O.causal_gqa_attention(q, k, v).reshape(T, Hq, hd)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h], v[0, h // 2], rtol=1e-14)   # row 0 sees only 0
    out0 = O.causal_gqa_attention(q, np.zeros_like(k), v).reshape(T, Hq, hd)
    for t in range(T):                                                    # equal scores: mean
        np.testing.assert_allclose(out0[t, 3], v[:t + 1, 1].mean(axis=0), rtol=1e-12)


# -------------------------------------------------------- delta rule ----

def test_single_write_then_read_returns_value():
    rng = np.random.default_rng(4)
    k, d, nu, eps = 16, 12, 3, 1e-6
    P = 2 * k * nu
    key = rng.standard_normal(k); val = rng.standard_normal(d)
    for beta in (1.0, 0.37):
        A, z = O.delta_rule_update(np.zeros((d, P)), np.zeros(P), key[None], val[None],
                                   np.array([beta]), nu, eps)
        phi = _dpfp_loops(list(key), nu)
        ff = phi @ phi
        np.testing.assert_allclose(z, phi, rtol=1e-15)                    # gamma = 1 at z = 0
        got = O.assoc_lookup(A, z, phi[None], eps)[0]
        np.testing.assert_allclose(got, beta * val * ff / (ff + eps), rtol=1e-12)
        assert np.max(np.abs(got - beta * val)) <= abs(beta) * np.max(np.abs(val)) * eps / ff * 1.01


def test_disjoint_keys_recall_exactly():
    # Keys whose DPFP features have disjoint supports do not interfere.
    k, d, nu, eps = 8, 5, 1, 1e-6
    k1 = np.zeros(k); k1[0], k1[1] = 1.0, 2.0
    k2 = np.zeros(k); k2[4], k2[5] = 0.5, 1.5
    rng = np.random.default_rng(5)
    vals = rng.standard_normal((2, d))
    A, z = O.delta_rule_update(np.zeros((d, 2 * k * nu)), np.zeros(2 * k * nu), np.stack([k1, k2]),
                               vals, np.ones(2), nu, eps)
    for key, v in ((k1, vals[0]), (k2, vals[1])):
        phi = _dpfp_loops(list(key), nu)
        ff = phi @ phi
        np.testing.assert_allclose(O.assoc_lookup(A, z, phi[None], eps)[0], v * ff / (ff + eps), rtol=1e-12)


def test_rewrite_same_pair_is_nearly_idempotent():
    rng = np.random.default_rng(6)
    k, d, nu, eps = 16, 9, 3, 1e-6
    P = 2 * k * nu
    key = rng.standard_normal(k); val = rng.standard_normal(d)
    A1, z1 = O.delta_rule_update(np.zeros((d, P)), np.zeros(P), key[None], val[None], np.ones(1), nu, eps)
    A2, z2 = O.delta_rule_update(A1, z1, key[None], val[None], np.ones(1), nu, eps)
    phi = _dpfp_loops(list(key), nu)
    ff = phi @ phi
    # second write only adds the eps-sized residue (v - vbar) ~ v * eps / ff
    assert np.max(np.abs(A2 - A1)) <= np.max(np.abs(val)) * eps / ff * np.max(phi) * 2
    assert np.max(np.abs(z2 - z1)) <= eps / ff * np.max(phi) * 2


def test_assoc_read_empty_memory_is_exact_zero():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((5, 6)); wq = rng.standard_normal((4, 6))
    np.testing.assert_array_equal(O.assoc_read(x, wq, np.zeros((6, 24)), np.zeros(24), 3, 1e-6), x)


# -------------------------------------------------------- whole model ----

def _tiny(**over):
    return dataclasses.replace(I.TINY, **over)


@pytest.mark.parametrize("over,n_seg", [({}, 4), ({"n_q_heads": 4, "n_kv_heads": 2, "head_dim": 16}, 3),
                                         ({"n_layers": 3}, 5), ({"n_layers": 4}, 2)])
def test_diag_order_equals_seq_order_bitwise(over, n_seg):
    cfg = _tiny(**over)
    W = I.make_weights(cfg, seed=11, norm_jitter=0.1)
    tok = I.make_tokens(cfg, n_seg, seed=11)
    a = O.forward(cfg, W, tok, n_seg, order="seq")
    b = O.forward(cfg, W, tok, n_seg, order="diag")
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_schedule_covers_grid_in_dependency_order():
    for L, n in ((1, 1), (2, 4), (16, 8), (5, 3)):
        steps = O.schedule(L, n, "diag")
        assert len(steps) == L + n - 1
        seen = {}
        for i, step in enumerate(steps):
            assert 1 <= len(step) <= min(L, n)
            for (l, s) in step:
                assert (l, s) not in seen
                seen[(l, s)] = i
        assert len(seen) == L * n
        for (l, s), i in seen.items():
            if l > 0:
                assert seen[(l - 1, s)] < i
            if s > 0:
                assert seen[(l, s - 1)] < i


@pytest.mark.parametrize("over,short", [({}, 0), ({"n_q_heads": 4, "n_kv_heads": 2, "head_dim": 16}, 0),
                                        ({}, 7)])
def test_one_segment_empty_memory_equals_plain_transformer(over, short):
    cfg = _tiny(**over)
    W = I.make_weights(cfg, seed=12, norm_jitter=0.1)
    tok = I.make_tokens(cfg, 1, seed=12)
    tok = tok[:tok.shape[0] - short]             # short > 0: a partial segment
    out, _, _ = O.forward(cfg, W, tok, 1)
    S = cfg.seg_len - short
    X = np.concatenate([W["embed"][tok], W["mem"]]).astype(np.float64)
    ref = plain_stack(X, W, cfg)
    np.testing.assert_allclose(out, ref[:S], rtol=1e-10, atol=1e-12)
    # causality: memory rows come after the segment, so the segment rows are
    # also the plain transformer over the S segment tokens alone
    ref_s = plain_stack(X[:S], W, cfg)
    np.testing.assert_allclose(out, ref_s, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("short", [0, 5])
def test_two_segments_one_layer_hand_expansion(short):
    # short > 0: the second segment is `short` tokens shorter (a partial last
    # segment: its memory rows follow its S - short tokens)
    cfg = _tiny(n_layers=1)
    W = I.make_weights(cfg, seed=13, norm_jitter=0.1)
    tok = I.make_tokens(cfg, 2, seed=13)
    tok = tok[:tok.shape[0] - short]
    out, A, z = O.forward(cfg, W, tok, 2)
    S, k, nu, eps = cfg.seg_len, cfg.key_dim, cfg.dpfp_nu, cfg.assoc_eps
    S1 = S - short
    W64 = {kk: np.asarray(v, np.float64) for kk, v in W.items()}
    gf = W64["norm_f"]

    def write(Hm, A, z):
        # memory rows written one after another, each against the state the
        # previous one left, with the entries written out
        A = A.copy(); z = z.copy()
        for i in range(Hm.shape[0]):
            key = W64["a_wk"][0] @ Hm[i]; val = W64["a_wv"][0] @ Hm[i]
            beta = 1.0 / (1.0 + math.exp(-(W64["a_wbeta"][0] @ Hm[i])))
            phi = _dpfp_loops(list(key), nu)
            zp = float(z @ phi)
            ff = float(phi @ phi)
            for r in range(A.shape[0]):
                vbar_r = float(A[r] @ phi) / (zp + eps)
                A[r] = A[r] + beta * (val[r] - vbar_r) * phi
            z = z + min(max(1.0 - zp / (ff + eps), 0.0), 1.0) * phi
        return A, z

    P = cfg.phi_dim
    X0 = np.concatenate([W64["embed"][tok[:S]], W64["mem"]])
    H0 = plain_layer(X0, W64, 0, cfg)
    A1, z1 = write(H0[S:], np.zeros((cfg.d_model, P)), np.zeros(P))
    X1 = np.concatenate([W64["embed"][tok[S:]], W64["mem"]])
    for t in range(X1.shape[0]):
        phi = _dpfp_loops(list(W64["a_wq"][0] @ X1[t]), nu)
        X1[t] = X1[t] + (A1 @ phi) / (float(z1 @ phi) + eps)
    assert X1.shape[0] == S1 + cfg.n_mem
    H1 = plain_layer(X1, W64, 0, cfg)
    A2, z2 = write(H1[S1:], A1, z1)
    ms = lambda r: r / math.sqrt(float(np.mean(r * r)) + cfg.norm_eps) * gf
    ref = np.stack([ms(r) for r in np.concatenate([H0[:S], H1[:S1]])])
    assert out.shape == (S + S1, cfg.d_model)
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(A[0], A2, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(z[0], z2, rtol=1e-9, atol=1e-11)


def test_resume_from_carried_state():
    cfg = I.TINY
    W = I.make_weights(cfg, seed=14)
    tok = I.make_tokens(cfg, 4, seed=14)
    full = O.forward(cfg, W, tok, 4)
    S = cfg.seg_len
    h1, A1, z1 = O.forward(cfg, W, tok[:2 * S], 2)
    h2, A2, z2 = O.forward(cfg, W, tok[2 * S:], 2, A0=A1, z0=z1)
    np.testing.assert_array_equal(np.concatenate([h1, h2]), full[0])
    np.testing.assert_array_equal(A2, full[1])
    np.testing.assert_array_equal(z2, full[2])


def test_memory_tokens_written_in_order():
    # a state written from rows (h0, h1) differs from one written from (h1, h0)
    # once the keys interact: the writes are sequential, not a sum
    rng = np.random.default_rng(8)
    d, k, nu, eps = 6, 4, 2, 1e-6
    H = rng.standard_normal((2, d)); wk = rng.standard_normal((k, d)); wv = rng.standard_normal((d, d))
    H[1] = H[0] + 0.3 * H[1]                     # nearby keys: overlapping features
    wb = rng.standard_normal(d)
    P = 2 * k * nu
    assert _dpfp_loops(list(wk @ H[0]), nu) @ _dpfp_loops(list(wk @ H[1]), nu) > 0.1
    A1, z1 = O.assoc_write(H, wk, wv, wb, np.zeros((d, P)), np.zeros(P), nu, eps)
    A2, z2 = O.assoc_write(H[::-1], wk, wv, wb, np.zeros((d, P)), np.zeros(P), nu, eps)
    assert np.max(np.abs(A1 - A2)) > 1e-6
    # and the first write into an empty memory is exact recall, whatever follows
    A0, z0 = O.assoc_write(H[:1], wk, wv, wb, np.zeros((d, P)), np.zeros(P), nu, eps)
    phi = _dpfp_loops(list(wk @ H[0]), nu)
    beta = 1.0 / (1.0 + math.exp(-(wb @ H[0])))
    ff = phi @ phi
    np.testing.assert_allclose(O.assoc_lookup(A0, z0, phi[None], eps)[0], beta * (wv @ H[0]) * ff / (ff + eps),
                               rtol=1e-12)


def test_state_stays_bounded_on_a_mid_size_model():
    # 12 segments of a 2-layer d=256 model with the benchmark's weight scale:
    # the memory state and residual stream stay O(1)
    cfg = dataclasses.replace(I.ARMT_1B, n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=2,
                              head_dim=64, ffn_dim=512, vocab=500, seg_len=64, dtype="f32")
    W = I.make_weights(cfg, seed=3)
    tok = I.make_tokens(cfg, 12, seed=3)
    out, A, z = O.forward(cfg, W, tok, 12)
    assert np.isfinite(out).all()
    assert np.abs(A).max() < 1.0 and np.abs(z).max() < 10.0


def test_normaliser_stays_nonnegative_and_denominators_positive():
    # with the correction clipped to [0, 1], z is a non-negative combination of
    # non-negative features: z >= 0 and z^T phi + eps >= eps for any query
    rng = np.random.default_rng(10)
    k, d, nu, eps = 8, 5, 3, 1e-6
    P = 2 * k * nu
    A, z = np.zeros((d, P)), np.zeros(P)
    for _ in range(200):
        keys = rng.standard_normal((1, k)) * rng.uniform(0.1, 5.0)
        A, z = O.delta_rule_update(A, z, keys, rng.standard_normal((1, d)), rng.uniform(0, 1, 1), nu, eps)
        assert (z >= 0).all()
    # an over-full normaliser (z^T phi > phi^T phi) is not pushed negative
    key = rng.standard_normal((1, k))
    phi = _dpfp_loops(list(key[0]), nu)
    z_big = 10.0 * phi
    _, z2 = O.delta_rule_update(np.zeros((d, P)), z_big, key, np.ones((1, d)), np.ones(1), nu, eps)
    np.testing.assert_array_equal(z2, z_big)      # gamma clipped to 0


def test_tiny_workload_is_well_conditioned():
    cfg, n, W, tok = I.make_workload("tiny")
    out, A, z = O.forward(cfg, W, tok, n)
    assert np.isfinite(out).all() and np.isfinite(A).all() and np.isfinite(z).all()
    # the memory was actually written and read: later segments differ from a
    # run whose memory is reset at every segment
    S = cfg.seg_len
    alone = np.concatenate([O.forward(cfg, W, tok[s * S:(s + 1) * S], 1)[0] for s in range(n)])
    np.testing.assert_array_equal(out[:S], alone[:S])
    assert np.max(np.abs(out[S:] - alone[S:])) > 1e-3


# ------------------------------------------------- bf16 precision model ----

def test_round_bf16_matches_torch_and_ties_to_even():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(10000) * 10.0 ** rng.integers(-6, 6, 10000),
                        [0.0, -0.0, 1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8)]])
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(O.round_bf16(x), want)
    # exact ties: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1.0)
    assert O.round_bf16(np.array([1.0 + 2.0 ** -8]))[0] == 1.0
    assert O.round_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6
    # fp16 (the attention operands' type): against torch, ties to even, range
    y = x[np.abs(x) < 6e4]
    want16 = torch.from_numpy(y.astype(np.float32)).to(torch.float16).double().numpy()
    np.testing.assert_array_equal(O.round_f16(y), want16)
    assert O.round_f16(np.array([1.0 + 2.0 ** -11]))[0] == 1.0
    assert O.round_f16(np.array([1.0 + 3 * 2.0 ** -11]))[0] == 1.0 + 2.0 ** -9
    assert O.round_f16(np.array([65504.0]))[0] == 65504.0


def test_bf16_precision_model_is_close_to_fp64_and_rounds():
    cfg = dataclasses.replace(I.TINY, dtype="bf16")
    W = I.make_weights(cfg, seed=15)
    tok = I.make_tokens(cfg, 3, seed=15)
    exact = O.forward(cfg, W, tok, 3)
    model = O.forward(cfg, W, tok, 3, operands="bf16")
    diff = np.abs(model[0] - exact[0]).max()
    assert 1e-5 < diff < 0.2        # rounding is applied, and only perturbs
    # diagonal order still equals sequential order under the precision model
    model_d = O.forward(cfg, W, tok, 3, order="diag", operands="bf16")
    for a, b in zip(model, model_d):
        np.testing.assert_array_equal(a, b)


def test_bf16_precision_model_matches_an_independent_emulation():
    """The precision model rounds to bf16 at exactly its listed operand points.

    tests/plain_bf16_cell.py re-implements two-layer ARMT cells with loops and
    torch's bfloat16 conversion, rounding at the named points and nowhere
    else.  The oracle's model must agree with it to fp64 rounding noise, and
    leaving out any single rounding point of the emulation must move the
    result by far more than that -- so a missing, misplaced or extra rounding
    point in the model fails here.  Weights are N(0, 0.1) so that at this tiny
    size the memory read carries enough weight for its points to show."""
    cfg = dataclasses.replace(I.TINY, n_layers=2, dtype="bf16")
    W = I.make_weights(cfg, seed=16, std=0.1, norm_jitter=0.1)
    tok = I.make_tokens(cfg, 2, seed=16)
    model = O.forward(cfg, W, tok, 2, operands="bf16")
    rel = lambda a, b: float(np.abs(a - b).max() / np.abs(b).max())
    emu = plain_bf16_cell.forward(cfg, W, tok, 2)
    for a, b in zip(emu, model):
        assert rel(a, b) <= 1e-12
    for point in plain_bf16_cell.ALL_POINTS:
        part = plain_bf16_cell.forward(cfg, W, tok, 2, points=set(plain_bf16_cell.ALL_POINTS) - {point})
        assert max(rel(a, b) for a, b in zip(part, model)) >= 1e-4, point
    exact = O.forward(cfg, W, tok, 2)
    assert min(rel(a, b) for a, b in zip(exact, model)) >= 1e-4
    # the split precision mode's model: same agreement; every point still
    # matters (its ~2^-17 rounding moves the result far beyond fp64 noise),
    # and the split model sits far closer to fp64 than the bf16 one
    split = O.forward(cfg, W, tok, 2, operands="bf16x2")
    emu_split = plain_bf16_cell.forward(cfg, W, tok, 2, split=True)
    for a, b in zip(emu_split, split):
        assert rel(a, b) <= 1e-12
    for point in plain_bf16_cell.ALL_POINTS:
        part = plain_bf16_cell.forward(cfg, W, tok, 2, points=set(plain_bf16_cell.ALL_POINTS) - {point},
                                       split=True)
        assert max(rel(a, b) for a, b in zip(part, split)) >= 1e-8, point
    for a, b, c in zip(split, model, exact):
        assert rel(a, c) <= 0.3 * rel(b, c)


def test_lm_head_logits_closed_forms():
    # with an identity head (V = d) the logits are the hidden rows themselves;
    # with a permutation head they are those rows permuted -- a transposed or
    # swapped operand fails one of the two
    rng = np.random.default_rng(5)
    h = rng.standard_normal((3, 6))
    np.testing.assert_array_equal(O.lm_head_logits(h, np.eye(6)), h)
    perm = np.array([2, 0, 5, 1, 4, 3])
    head = np.eye(6)[perm]                       # row v picks coordinate perm[v]
    np.testing.assert_array_equal(O.lm_head_logits(h, head), h[:, perm])
    # a tied head and a hidden row equal to embedding row j: logit j is ||e_j||^2
    E = rng.standard_normal((10, 6))
    lg = O.lm_head_logits(E[[7]], E)
    assert lg.shape == (1, 10)
    assert abs(lg[0, 7] - float(E[7] @ E[7])) < 1e-12


def test_relative_logits_error_closed_forms():
    ref = np.random.default_rng(6).standard_normal((4, 9))
    assert O.relative_logits_error(ref, ref) == 0.0
    assert abs(O.relative_logits_error(1.01 * ref, ref) - 0.01) < 1e-12
    assert abs(O.relative_logits_error(np.zeros_like(ref), ref) - 1.0) < 1e-15


def test_linear_map_matches_printed_two_layer_example():
    # A worked example printed on a page of the same bundle (two chained linear
    # layers on small integers, tests/golden/two_linear_layers_small_integers.txt):
    # the oracle's linear map (rows times the transpose of an (out, in) matrix,
    # the form of every projection and of the LM head) reproduces it exactly.
    from tests.golden.load import read_matrices
    g = read_matrices("two_linear_layers_small_integers.txt")
    inter = O.lm_head_logits(g["x"], g["weights_A"].T)        # (out, in) = transpose of (in, out)
    np.testing.assert_array_equal(inter, g["intermediate"])
    out = O.lm_head_logits(inter, g["weights_B"].T)
    np.testing.assert_array_equal(out, g["output"])
    # a transposed operand would give a different (or ill-shaped) product
    assert not np.array_equal(O.lm_head_logits(g["x"].T, g["weights_A"].T), g["intermediate"])
