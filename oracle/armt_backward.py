"""fp64 gradients of the ARMT forward pass: the reference for a backward pass.

TEST INFRASTRUCTURE ONLY, like ``armt_oracle``: only the tests may import
this module; the library and its binding never do, and it imports nothing
from them.

The summary page of "Diagonal Batching Unlocks Parallelism in Recurrent
Memory Transformers for Long Contexts" (section 四) reports that diagonal
batching was also carried over to the backward pass so that training and
inference share one schedule.  The backward of the recurrence is the adjoint
of the forward that ``armt_oracle.forward`` defines: every cell (l, s) passes
gradients back to its input rows (cell (l-1, s)) and to the state it read
(cell (l, s-1)), and each layer's weights collect the gradients of all of its
cells.  Here that forward is restated term by term on torch float64 CPU
tensors -- the same definitions, in the same order: associative read, LLaMA
block, delta-rule writes of the memory rows one after another, final RMSNorm
of the segment rows -- and differentiated with torch's reverse-mode autograd,
used as a library primitive.  Nothing is fused or reordered; a short last
segment and an initial state are handled as in the oracle.

The loss is the inner product of the outputs with fixed cotangents:
    loss = <hidden, R_h> + <A_final, R_A> + <z_final, R_z>,
so its gradient is the vector-Jacobian product a backward kernel computes.
Pinned in tests/test_backward_oracle.py: the restated forward agrees with
``armt_oracle.forward``; directional derivatives agree with central finite
differences of ``armt_oracle.forward`` for every weight group and the initial
state; the diagonal and sequential cell orders give the same gradients;
gradients respect causality (later segments do not influence earlier
outputs) and vanish for embedding rows no token uses.

``backward_by_diagonals`` computes the same gradients in the order a
diagonal-batched backward pass would: anti-diagonals in reverse, each cell's
vector-Jacobian product handing adjoints to the cell below it (same segment)
and to the cell before it (same layer); pinned against the whole-graph
gradient.  ``backward_explicit`` does the same with every adjoint written out
in numpy (``rmsnorm_backward``, ``rope_backward``, ``attention_backward``,
``dpfp_backward``, ``assoc_read_backward``, ``assoc_write_backward``,
``cell_backward``): the per-op reference for backward kernels.
"""
from typing import Dict, Optional, Tuple

import numpy as np
import torch

from . import armt_oracle as O

F64 = torch.float64
WEIGHT_KEYS = ("embed", "mem", "wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "a_wq", "a_wk",
               "a_wv", "a_wbeta", "norm1", "norm2", "norm_f")


def _t(a, grad=False):
    t = torch.as_tensor(np.asarray(a, dtype=np.float64), dtype=F64).clone()
    return t.requires_grad_(grad)


def rmsnorm(x, gain, eps):
    return x / torch.sqrt((x * x).mean(dim=-1, keepdim=True) + eps) * gain


def dpfp(x, nu):
    r = torch.cat([torch.relu(x), torch.relu(-x)], dim=-1)
    return torch.cat([r * torch.roll(r, j, dims=-1) for j in range(1, nu + 1)], dim=-1)


def rope_rotate_half(x, base):
    T, _, hd = x.shape
    half = hd // 2
    inv_freq = base ** (-(2.0 * torch.arange(half, dtype=F64)) / hd)
    ang = torch.arange(T, dtype=F64)[:, None] * inv_freq[None, :]
    cos, sin = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1)


def causal_gqa_attention(q, k, v):
    T, Hq, hd = q.shape
    Hkv = k.shape[1]
    mask = torch.triu(torch.ones((T, T), dtype=torch.bool), diagonal=1)
    heads = []
    for h in range(Hq):
        g = (h * Hkv) // Hq
        s = (q[:, h, :] @ k[:, g, :].T) / np.sqrt(hd)
        p = torch.softmax(s.masked_fill(mask, float("-inf")), dim=-1)
        heads.append(p @ v[:, g, :])
    return torch.stack(heads, dim=1).reshape(T, Hq * hd)


def assoc_read(x, wq_a, A, z, nu, eps):
    phi = dpfp(x @ wq_a.T, nu)
    return x + (phi @ A.T) / (phi @ z + eps)[:, None]


def delta_rule_write(A, z, key, value, beta, nu, eps):
    """One write (key [k], value [d], beta scalar) against the current state."""
    phi = dpfp(key, nu)
    zphi = phi @ z
    vbar = (A @ phi) / (zphi + eps)
    gamma = torch.clamp(1.0 - zphi / (phi @ phi + eps), 0.0, 1.0)
    return A + torch.outer(beta * (value - vbar), phi), z + gamma * phi


def llama_block(x, cfg, W, l):
    T = x.shape[0]
    Hq, Hkv, hd = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    n = rmsnorm(x, W["norm1"][l], cfg.norm_eps)
    q = rope_rotate_half((n @ W["wq"][l].T).reshape(T, Hq, hd), cfg.rope_base)
    k = rope_rotate_half((n @ W["wk"][l].T).reshape(T, Hkv, hd), cfg.rope_base)
    v = (n @ W["wv"][l].T).reshape(T, Hkv, hd)
    y = x + causal_gqa_attention(q, k, v) @ W["wo"][l].T
    n2 = rmsnorm(y, W["norm2"][l], cfg.norm_eps)
    u = torch.nn.functional.silu(n2 @ W["w_gate"][l].T) * (n2 @ W["w_up"][l].T)
    return y + u @ W["w_down"][l].T


def cell_forward(x, cfg, W, l, A, z):
    nu, eps = cfg.dpfp_nu, cfg.assoc_eps
    x = assoc_read(x, W["a_wq"][l], A, z, nu, eps)
    h = llama_block(x, cfg, W, l)
    m0 = h.shape[0] - cfg.n_mem
    hm = h[m0:]
    keys, values = hm @ W["a_wk"][l].T, hm @ W["a_wv"][l].T
    beta = torch.sigmoid(hm @ W["a_wbeta"][l])
    for i in range(hm.shape[0]):
        A, z = delta_rule_write(A, z, keys[i], values[i], beta[i], nu, eps)
    return h, A, z


def forward(cfg, W, tokens, n_segments, order="seq", A0=None, z0=None):
    """The oracle's forward on torch tensors; W: dict of float64 tensors
    (leaves that may require grad), A0 [L, d, P] / z0 [L, P] tensors or None.
    Returns (hidden [N, d], A [L, d, P], z [L, P])."""
    L, d, P, S = cfg.n_layers, cfg.d_model, cfg.phi_dim, cfg.seg_len
    tokens = np.asarray(tokens)
    N = tokens.shape[0]
    assert (n_segments - 1) * S < N <= n_segments * S
    A = [A0[l] if A0 is not None else torch.zeros((d, P), dtype=F64) for l in range(L)]
    z = [z0[l] if z0 is not None else torch.zeros((P,), dtype=F64) for l in range(L)]
    acts, rows = {}, [None] * n_segments
    for step in O.schedule(L, n_segments, order):
        for (l, s) in step:
            if l == 0:
                ids = torch.as_tensor(tokens[s * S:(s + 1) * S], dtype=torch.long)
                x = torch.cat([W["embed"][ids], W["mem"]], dim=0)
            else:
                x = acts.pop((l - 1, s))
            h, A[l], z[l] = cell_forward(x, cfg, W, l, A[l], z[l])
            if l == L - 1:
                seg = h.shape[0] - cfg.n_mem
                rows[s] = rmsnorm(h[:seg], W["norm_f"], cfg.norm_eps)
            else:
                acts[(l, s)] = h
    return torch.cat(rows, dim=0), torch.stack(A), torch.stack(z)


def loss_value(out: Tuple, cot: Dict[str, np.ndarray]) -> float:
    """<hidden, R_h> + <A, R_A> + <z, R_z> for numpy outputs (fp64)."""
    h, A, z = (np.asarray(o, np.float64) for o in out)
    return float(np.sum(h * cot["hidden"]) + np.sum(A * cot["A"]) + np.sum(z * cot["z"]))


def gradients(cfg, W: Dict[str, np.ndarray], tokens, n_segments, cot: Dict[str, np.ndarray],
              order="seq", A0: Optional[np.ndarray] = None, z0: Optional[np.ndarray] = None):
    """Gradient of the loss above with respect to every weight (and to the
    initial state A0, z0 when given).  Returns (loss, {name: fp64 array})."""
    Wt = {k: _t(W[k], grad=True) for k in WEIGHT_KEYS}
    A0t = _t(A0, grad=True) if A0 is not None else None
    z0t = _t(z0, grad=True) if z0 is not None else None
    h, A, z = forward(cfg, Wt, tokens, n_segments, order, A0t, z0t)
    loss = (h * _t(cot["hidden"])).sum() + (A * _t(cot["A"])).sum() + (z * _t(cot["z"])).sum()
    leaves = [Wt[k] for k in WEIGHT_KEYS] + [t for t in (A0t, z0t) if t is not None]
    grads = torch.autograd.grad(loss, leaves, allow_unused=True)
    names = list(WEIGHT_KEYS) + [n for n, t in (("A0", A0t), ("z0", z0t)) if t is not None]
    out = {}
    for n, g, leaf in zip(names, grads, leaves):
        out[n] = (g if g is not None else torch.zeros_like(leaf)).detach().numpy()
    return float(loss.detach()), out


def backward_by_diagonals(cfg, W: Dict[str, np.ndarray], tokens, n_segments, cot: Dict[str, np.ndarray],
                          A0: Optional[np.ndarray] = None, z0: Optional[np.ndarray] = None):
    """The same gradients, computed the way a diagonal-batched backward pass
    runs: anti-diagonals in reverse order (i = L + n - 2 down to 0), every
    cell (l, s) of a diagonal taking the adjoints of its outputs -- its rows
    from cell (l+1, s) (or the final RMSNorm when l = L-1) and its written
    state from cell (l, s+1) (or the final-state cotangent) -- and returning
    the adjoints of its input rows (to cell (l-1, s), or to the embeddings)
    and of the state it read (to cell (l, s-1), or to A0/z0), plus its share
    of layer l's weight gradients.  The cell's vector-Jacobian product is
    taken on a recomputed forward of that one cell (the forward keeps only
    cell inputs and states).  Returns {name: fp64 array} like ``gradients``."""
    L, d, P, S, M = cfg.n_layers, cfg.d_model, cfg.phi_dim, cfg.seg_len, cfg.n_mem
    tokens = np.asarray(tokens)
    n = n_segments
    Wt = {k: _t(W[k]) for k in WEIGHT_KEYS}
    # forward, keeping what each cell read: its input rows and the state before it
    x_in, state_in = {}, {}
    A = [_t(A0[l]) if A0 is not None else torch.zeros((d, P), dtype=F64) for l in range(L)]
    z = [_t(z0[l]) if z0 is not None else torch.zeros((P,), dtype=F64) for l in range(L)]
    acts = {}
    with torch.no_grad():
        for step in O.schedule(L, n, "diag"):
            for (l, s) in step:
                if l == 0:
                    ids = torch.as_tensor(tokens[s * S:(s + 1) * S], dtype=torch.long)
                    x = torch.cat([Wt["embed"][ids], Wt["mem"]], dim=0)
                else:
                    x = acts.pop((l - 1, s))
                x_in[(l, s)], state_in[(l, s)] = x, (A[l], z[l])
                h, A[l], z[l] = cell_forward(x, cfg, Wt, l, A[l], z[l])
                if l < L - 1:
                    acts[(l, s)] = h
    grads = {k: torch.zeros_like(Wt[k]) for k in WEIGHT_KEYS}
    gA0, gz0 = torch.zeros((L, d, P), dtype=F64), torch.zeros((L, P), dtype=F64)
    h_bar = {}                                             # adjoint of each cell's output rows
    st_bar = {l: (_t(cot["A"][l]), _t(cot["z"][l])) for l in range(L)}  # adjoint of the state a cell wrote
    R_h = _t(cot["hidden"])
    for i in reversed(range(L + n - 1)):
        for l in range(L):
            s = i - l
            if not 0 <= s < n:
                continue
            x = x_in[(l, s)].clone().requires_grad_(True)
            Ain = state_in[(l, s)][0].clone().requires_grad_(True)
            zin = state_in[(l, s)][1].clone().requires_grad_(True)
            Wl = {k: (Wt[k].clone().requires_grad_(True) if k != "embed" else Wt[k]) for k in WEIGHT_KEYS}
            h, A_out, z_out = cell_forward(x, cfg, Wl, l, Ain, zin)
            Abar, zbar = st_bar[l]
            terms = (A_out * Abar).sum() + (z_out * zbar).sum()
            if l == L - 1:
                seg = h.shape[0] - M
                lo_row = s * S
                terms = terms + (rmsnorm(h[:seg], Wl["norm_f"], cfg.norm_eps) * R_h[lo_row:lo_row + seg]).sum()
            else:
                terms = terms + (h * h_bar.pop((l, s))).sum()
            leaves = [x, Ain, zin] + [Wl[k] for k in WEIGHT_KEYS if k != "embed"]
            g = torch.autograd.grad(terms, leaves, allow_unused=True)
            gx, gA, gz = g[0], g[1], g[2]
            for k, gk in zip([k for k in WEIGHT_KEYS if k != "embed"], g[3:]):
                if gk is not None:
                    grads[k] += gk
            st_bar[l] = (gA, gz)                            # to cell (l, s - 1)
            if l > 0:
                h_bar[(l - 1, s)] = gx                      # to cell (l - 1, s)
            else:
                seg = x.shape[0] - M                        # the embedding rows and the memory rows
                ids = torch.as_tensor(tokens[s * S:s * S + seg], dtype=torch.long)
                grads["embed"].index_add_(0, ids, gx[:seg])
                grads["mem"] += gx[seg:]
    for l in range(L):
        gA0[l], gz0[l] = st_bar[l]
    out = {k: v.numpy() for k, v in grads.items()}
    if A0 is not None:
        out["A0"] = gA0.numpy()
    if z0 is not None:
        out["z0"] = gz0.numpy()
    return out


# --------------------------------------------------------------------------
# Explicit adjoints of the associative block (numpy fp64), the per-op
# reference for backward kernels: each function takes the forward inputs and
# the adjoints of the outputs and returns the adjoints of the inputs, derived
# step by step from the forward definitions in armt_oracle.
# --------------------------------------------------------------------------

def dpfp_backward(x, phi_bar, nu):
    """Adjoint of phi = DPFP_nu(x) for x [..., k]: with r = [relu(x), relu(-x)]
    and phi_{(j-1) 2k + c} = r_c r_{(c-j) mod 2k}, each product sends
    phi_bar * (other factor) to both factors; relu passes where its input > 0."""
    x = np.asarray(x, np.float64)
    k = x.shape[-1]
    k2 = 2 * k
    r = np.concatenate([np.maximum(x, 0.0), np.maximum(-x, 0.0)], axis=-1)
    r_bar = np.zeros_like(r)
    for j in range(1, nu + 1):
        blk = phi_bar[..., (j - 1) * k2:j * k2]
        rolled = np.roll(r, j, axis=-1)                  # rolled_c = r_{(c-j) mod 2k}
        r_bar += blk * rolled
        r_bar += np.roll(blk * r, -j, axis=-1)           # to r_{(c-j)}: index c' = c - j
    return r_bar[..., :k] * (x > 0) - r_bar[..., k:] * (x < 0)


def assoc_read_backward(x, wq_a, A, z, nu, eps, y_bar):
    """Adjoint of y = x + A phi / (z^T phi + eps), phi = DPFP(W_Q x), rows x [R, d].
    Returns (x_bar, wq_bar, A_bar, z_bar)."""
    x = np.asarray(x, np.float64)
    q = x @ wq_a.T
    phi = O.dpfp(q, nu)
    D = phi @ z + eps                                    # [R]
    r = (phi @ A.T) / D[:, None]                         # [R, d] the read
    coef = np.sum(y_bar * r, axis=-1) / D                # (y_bar . r) / D per row
    A_bar = (y_bar / D[:, None]).T @ phi                 # sum_rows y_bar phi^T / D
    z_bar = -(coef[:, None] * phi).sum(axis=0)
    phi_bar = (y_bar @ A) / D[:, None] - coef[:, None] * z[None, :]
    q_bar = dpfp_backward(q, phi_bar, nu)
    return y_bar + q_bar @ wq_a, q_bar.T @ x, A_bar, z_bar


def assoc_write_backward(h_mem, wk_a, wv_a, wb_a, A0, z0, nu, eps, A_bar, z_bar):
    """Adjoint of the in-order delta-rule writes of the memory rows h_mem [M, d]
    from state (A0, z0) (armt_oracle.assoc_write), given the adjoints of the
    final state.  The writes are undone in reverse order, carrying the state's
    adjoint back through each one.  Returns (h_bar, wk_bar, wv_bar, wb_bar,
    A0_bar, z0_bar)."""
    h_mem = np.asarray(h_mem, np.float64)
    M = h_mem.shape[0]
    keys, values = h_mem @ wk_a.T, h_mem @ wv_a.T
    beta = 1.0 / (1.0 + np.exp(-(h_mem @ wb_a)))
    states = [(np.asarray(A0, np.float64), np.asarray(z0, np.float64))]
    for i in range(M):                                   # forward, keeping the state before each write
        states.append(O.delta_rule_update(states[-1][0], states[-1][1], keys[i:i + 1], values[i:i + 1],
                                          beta[i:i + 1], nu, eps))
    A_bar, z_bar = np.array(A_bar, np.float64), np.array(z_bar, np.float64)
    k_bar, v_bar, b_bar = np.zeros_like(keys), np.zeros_like(values), np.zeros(M)
    for i in reversed(range(M)):
        A, z = states[i]
        phi = O.dpfp(keys[i], nu)
        zphi = phi @ z
        D = zphi + eps
        vbar = (A @ phi) / D
        Q = phi @ phi + eps
        gu = 1.0 - zphi / Q
        gamma = min(max(gu, 0.0), 1.0)
        c = beta[i] * (values[i] - vbar)
        # A' = A + c phi^T,  z' = z + gamma phi
        c_bar = A_bar @ phi
        phi_bar = A_bar.T @ c + gamma * z_bar
        gamma_bar = z_bar @ phi
        # c = beta (v - vbar)
        b_bar[i] = c_bar @ (values[i] - vbar)
        v_bar[i] = beta[i] * c_bar
        vbar_bar = -beta[i] * c_bar
        # vbar = A phi / D
        A_prev_bar = A_bar + np.outer(vbar_bar / D, phi)
        phi_bar += A.T @ vbar_bar / D
        zphi_bar = -(vbar_bar @ vbar) / D
        # gamma = clip(1 - zphi / Q, 0, 1), Q = phi^T phi + eps
        gu_bar = gamma_bar if 0.0 <= gu <= 1.0 else 0.0
        zphi_bar += -gu_bar / Q
        phi_bar += 2.0 * (gu_bar * zphi / (Q * Q)) * phi
        # zphi = z^T phi
        z_prev_bar = z_bar + zphi_bar * phi
        phi_bar += zphi_bar * z
        k_bar[i] = dpfp_backward(keys[i], phi_bar, nu)
        A_bar, z_bar = A_prev_bar, z_prev_bar
    logit_bar = b_bar * beta * (1.0 - beta)
    h_bar = k_bar @ wk_a + v_bar @ wv_a + np.outer(logit_bar, wb_a)
    return h_bar, k_bar.T @ h_mem, v_bar.T @ h_mem, logit_bar @ h_mem, A_bar, z_bar


def rmsnorm_backward(x, gain, eps, y_bar):
    """Adjoint of y = x s gain, s = 1 / sqrt(mean(x^2) + eps), rows x [R, d].
    Returns (x_bar, gain_bar)."""
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    s = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    g_bar = np.sum(y_bar * x * s, axis=0)
    t = y_bar * gain                                     # adjoint of x s
    x_bar = s * t - (s ** 3) * np.sum(t * x, axis=-1, keepdims=True) * x / d
    return x_bar, g_bar


def rope_backward(y_bar, base):
    """Adjoint of the rotate-half rotation (a rotation per pair: its transpose)."""
    T, _, hd = y_bar.shape
    half = hd // 2
    inv_freq = base ** (-(2.0 * np.arange(half, dtype=np.float64)) / hd)
    ang = np.arange(T, dtype=np.float64)[:, None] * inv_freq[None, :]
    cos, sin = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    y1, y2 = y_bar[..., :half], y_bar[..., half:]
    return np.concatenate([y1 * cos + y2 * sin, -y1 * sin + y2 * cos], axis=-1)


def attention_backward(q, k, v, o_bar):
    """Adjoint of causal GQA attention (armt_oracle.causal_gqa_attention):
    q [T, Hq, hd], k/v [T, Hkv, hd], o_bar [T, Hq*hd].  Per query head:
    v_bar += P^T O_bar, P_bar = O_bar v^T, S_bar = P (P_bar - rowsum(P_bar P)),
    q_bar = S_bar k / sqrt(hd), k_bar += S_bar^T q / sqrt(hd)."""
    T, Hq, hd = q.shape
    Hkv = k.shape[1]
    o_bar = o_bar.reshape(T, Hq, hd)
    q_bar, k_bar, v_bar = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    mask = np.triu(np.ones((T, T), dtype=bool), k=1)
    for h in range(Hq):
        g = (h * Hkv) // Hq
        s = np.where(mask, -np.inf, (q[:, h, :] @ k[:, g, :].T) / np.sqrt(hd))
        p = np.exp(s - s.max(axis=-1, keepdims=True))
        p /= p.sum(axis=-1, keepdims=True)
        v_bar[:, g, :] += p.T @ o_bar[:, h, :]
        p_bar = o_bar[:, h, :] @ v[:, g, :].T
        s_bar = p * (p_bar - np.sum(p_bar * p, axis=-1, keepdims=True))
        q_bar[:, h, :] = s_bar @ k[:, g, :] / np.sqrt(hd)
        k_bar[:, g, :] += s_bar.T @ q[:, h, :] / np.sqrt(hd)
    return q_bar, k_bar, v_bar


def cell_backward(x, cfg, W, l, A, z, h_bar, A_bar, z_bar):
    """Explicit adjoint of armt_oracle.cell_forward (read, LLaMA block, writes)
    for one cell: inputs x [T, d] and state (A, z), adjoints of the output rows
    h_bar [T, d] and of the written state (A_bar, z_bar).  Returns (x_bar,
    A_in_bar, z_in_bar, {weight name: layer-l gradient})."""
    W = {kk: np.asarray(v, np.float64) for kk, v in W.items()}
    nu, eps, ne = cfg.dpfp_nu, cfg.assoc_eps, cfg.norm_eps
    T = x.shape[0]
    Hq, Hkv, hd = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    g = {}
    # forward, keeping the intermediates
    x1 = O.assoc_read(x, W["a_wq"][l], A, z, nu, eps)
    n1 = O.rmsnorm(x1, W["norm1"][l], ne)
    q0 = (n1 @ W["wq"][l].T).reshape(T, Hq, hd)
    k0 = (n1 @ W["wk"][l].T).reshape(T, Hkv, hd)
    v = (n1 @ W["wv"][l].T).reshape(T, Hkv, hd)
    q, k = O.rope_rotate_half(q0, cfg.rope_base), O.rope_rotate_half(k0, cfg.rope_base)
    att = O.causal_gqa_attention(q, k, v)
    y = x1 + att @ W["wo"][l].T
    n2 = O.rmsnorm(y, W["norm2"][l], ne)
    a, b = n2 @ W["w_gate"][l].T, n2 @ W["w_up"][l].T
    sa = 1.0 / (1.0 + np.exp(-a))
    u = a * sa * b
    h = y + u @ W["w_down"][l].T
    m0 = T - cfg.n_mem
    # the writes (from the state the read used)
    hw_bar, g["a_wk"], g["a_wv"], g["a_wbeta"], A_in_bar, z_in_bar = assoc_write_backward(
        h[m0:], W["a_wk"][l], W["a_wv"][l], W["a_wbeta"][l], A, z, nu, eps, A_bar, z_bar)
    h_bar = np.array(h_bar, np.float64)
    h_bar[m0:] += hw_bar
    # h = y + u Wd^T
    y_bar = h_bar.copy()
    u_bar = h_bar @ W["w_down"][l]
    g["w_down"] = h_bar.T @ u
    # u = silu(a) b
    a_bar = u_bar * b * sa * (1.0 + a * (1.0 - sa))
    b_bar = u_bar * a * sa
    g["w_gate"], g["w_up"] = a_bar.T @ n2, b_bar.T @ n2
    n2_bar = a_bar @ W["w_gate"][l] + b_bar @ W["w_up"][l]
    dy, g["norm2"] = rmsnorm_backward(y, W["norm2"][l], ne, n2_bar)
    y_bar += dy
    # y = x1 + att Wo^T
    x1_bar = y_bar.copy()
    att_bar = y_bar @ W["wo"][l]
    g["wo"] = y_bar.T @ att
    q_bar, k_bar, v_bar = attention_backward(q, k, v, att_bar)
    q0_bar, k0_bar = rope_backward(q_bar, cfg.rope_base), rope_backward(k_bar, cfg.rope_base)
    q0_bar, k0_bar, v_bar = q0_bar.reshape(T, -1), k0_bar.reshape(T, -1), v_bar.reshape(T, -1)
    g["wq"], g["wk"], g["wv"] = q0_bar.T @ n1, k0_bar.T @ n1, v_bar.T @ n1
    n1_bar = q0_bar @ W["wq"][l] + k0_bar @ W["wk"][l] + v_bar @ W["wv"][l]
    dx1, g["norm1"] = rmsnorm_backward(x1, W["norm1"][l], ne, n1_bar)
    x1_bar += dx1
    # the read
    x_bar, g["a_wq"], Ar_bar, zr_bar = assoc_read_backward(x, W["a_wq"][l], A, z, nu, eps, x1_bar)
    return x_bar, A_in_bar + Ar_bar, z_in_bar + zr_bar, g


def backward_explicit(cfg, W: Dict[str, np.ndarray], tokens, n_segments, cot: Dict[str, np.ndarray],
                      A0: Optional[np.ndarray] = None, z0: Optional[np.ndarray] = None):
    """backward_by_diagonals with the explicit numpy adjoints above in place
    of autograd: the complete backward pass written out, cell by cell, in
    reverse diagonal order.  Returns {name: fp64 array}."""
    L, d, P, S, M = cfg.n_layers, cfg.d_model, cfg.phi_dim, cfg.seg_len, cfg.n_mem
    W64 = O.widen_weights(W)
    tokens = np.asarray(tokens)
    n = n_segments
    x_in, state_in, acts = {}, {}, {}
    A = [np.asarray(A0[l], np.float64).copy() if A0 is not None else np.zeros((d, P)) for l in range(L)]
    z = [np.asarray(z0[l], np.float64).copy() if z0 is not None else np.zeros(P) for l in range(L)]
    h_last = {}
    for step in O.schedule(L, n, "diag"):
        for (l, s) in step:
            x = O.layer0_input(cfg, W64, tokens, s) if l == 0 else acts.pop((l - 1, s))
            x_in[(l, s)], state_in[(l, s)] = x, (A[l], z[l])
            h, A[l], z[l] = O.cell_forward(x, cfg, W64, l, A[l], z[l])
            if l < L - 1:
                acts[(l, s)] = h
            else:
                h_last[s] = h
    grads = {kk: np.zeros_like(W64[kk]) for kk in WEIGHT_KEYS}
    st_bar = {l: (np.asarray(cot["A"][l], np.float64), np.asarray(cot["z"][l], np.float64)) for l in range(L)}
    h_bar = {}
    for i in reversed(range(L + n - 1)):
        for l in range(L):
            s = i - l
            if not 0 <= s < n:
                continue
            x = x_in[(l, s)]
            if l == L - 1:
                h = h_last[s]
                seg = h.shape[0] - M
                hb = np.zeros_like(h)
                hb[:seg], gf = rmsnorm_backward(h[:seg], W64["norm_f"], cfg.norm_eps,
                                                np.asarray(cot["hidden"][s * S:s * S + seg], np.float64))
                grads["norm_f"] += gf
            else:
                hb = h_bar.pop((l, s))
            A_, z_ = state_in[(l, s)]
            x_bar, Ab, zb, g = cell_backward(x, cfg, W64, l, A_, z_, hb, *st_bar[l])
            st_bar[l] = (Ab, zb)
            for kk, v in g.items():
                grads[kk][l] += v
            if l > 0:
                h_bar[(l - 1, s)] = x_bar
            else:
                seg = x.shape[0] - M
                np.add.at(grads["embed"], tokens[s * S:s * S + seg], x_bar[:seg])
                grads["mem"] += x_bar[seg:]
    out = dict(grads)
    if A0 is not None:
        out["A0"] = np.stack([st_bar[l][0] for l in range(L)])
    if z0 is not None:
        out["z0"] = np.stack([st_bar[l][1] for l in range(L)])
    return out
