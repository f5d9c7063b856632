"""fp64 CPU oracle for the ARMT forward pass under both cell schedules.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The library and its Python binding never do, and this module imports
nothing from them: it takes plain numpy arrays (weights from the seeded input
generator, widened here to float64) and shares no code with the CUDA path.

What it computes, with the passage each part follows.  "The summary page"
below is the summary of "Diagonal Batching Unlocks Parallelism in Recurrent
Memory Transformers for Long Contexts" (Sivtsov, Rodkin, Kuzmin, Kuratov,
Oseledets, arXiv:2506.05229):

* The recurrence (summary page, section 二): the input is cut into segments;
  every layer l keeps its own memory state (an associative matrix A_l, plus
  the normaliser vector z_l that the delta-rule form carries), updated by an
  associative block from that layer's output on the previous segment.  So
  cell (layer l, segment s) needs only cell (l-1, s) (its input rows) and
  cell (l, s-1) (the state A_l, z_l).
* The schedule (section 二, last paragraphs; section 五): every cell with
  l + s = i can run in iteration i, one anti-diagonal at a time, giving
  n_layers + n_segments - 1 grouped steps instead of n_layers * n_segments;
  the reordering keeps the exact recurrence.  ``forward(order="diag")``
  walks the grid in that order, ``order="seq"`` segment by segment; the
  per-cell arithmetic is the same function, so fp64 results are identical.
* The associative block (section 二: quasi-linear attention with a delta rule,
  equations not printed on the page).  Reading used here, the standard ARMT
  delta rule with DPFP features:
    read:  x <- x + A phi(W_Q x) / (z^T phi(W_Q x) + eps)       (every row)
    write: for the memory rows h_i, i = 0..M-1 in order, one at a time:
           k = W_K h_i, v = W_V h_i, beta = sigmoid(w_b^T h_i), p = phi(k),
           vbar = A p / (z^T p + eps),
           gamma = clip(1 - z^T p / (p^T p + eps), 0, 1),
           A <- A + beta (v - vbar) p^T,  z <- z + gamma p
           (a delta rule: each write corrects against the state the previous
           write left; applying all M writes against the pre-segment state
           instead makes the state diverge on random-init models).  Clipping
           gamma to [0, 1] keeps z a non-negative combination of the
           non-negative features, so every denominator z^T phi + eps stays
           >= eps; unclipped, z turns negative and the state diverges within
           ~60 segments of the 1B-shaped model.
  DPFP_nu(x): r = [relu(x), relu(-x)], phi = concat_{j=1..nu} r * roll(r, j),
  roll(r, j)_i = r_{(i - j) mod 2k}.
* The LLaMA block run inside each cell (section 三: Llama-3-family models,
  attention run unchanged): pre-RMSNorm, rotate-half RoPE at positions
  0..T_c-1 within the cell, causal grouped-query attention, SwiGLU MLP, no
  biases.  Memory tokens are appended after the S segment tokens of every
  segment (the write-memory position of the RMT form in section 二).
* Output: the last layer's segment rows after the final RMSNorm, and the
  final A_l, z_l of every layer.
* LM head and error measure (section 四: the drift of diagonal batching from
  the sequential recurrence, read through the logits): logits = hidden
  head^T, compared as a relative Frobenius norm.

Everything is float64 with no intermediate rounding; bf16 models arrive as
float32 arrays holding bf16 values and are widened exactly.  numpy matmul is
used as a library primitive; nothing is blocked, fused or reordered beyond
the definitions above.

Optional precision model (``operands="bf16"``): the same arithmetic in fp64,
except that every tensor-core operand of the bf16 kernel path is rounded to
its 16-bit type first.  Operands of the weight products are rounded to bf16
(the weights' type): the layer input for the associative query, the features
and the state copy of the associative read, both RMSNorm outputs, the
attention output, the SwiGLU output, and the memory rows fed to the write
projections.  The attention's own operands -- q and k after RoPE, v, and the
probabilities (before normalisation by the row sum) -- are activations only,
and the kernel path gives them fp16 (same width, three more mantissa bits),
so the model rounds them to fp16.  ``operands="bf16x2"`` models the split
precision mode of the same path: the operands of the weight products and of
the associative read (features and state copy) are carried as a bf16 high
part plus the bf16 rounding of the residual (about 16 significant bits);
the attention operands stay fp16.  These are models of
design choices, not of the method; the default (``operands=None``) is the
method itself.
"""
from __future__ import annotations

from typing import Dict, Tuple

import numpy as np

F64 = np.float64


def _f64(a):
    return np.asarray(a, dtype=F64)


def _identity(a):
    return a


def round_bf16(a):
    """Nearest bf16 value (ties to even), via float32, returned as float64.

    Values are first rounded to float32; the fp32 -> bf16 step keeps the top
    16 bits after adding 0x7FFF plus the lowest kept bit (round half to even).
    """
    b = np.ascontiguousarray(np.asarray(a, dtype=np.float32)).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32).astype(F64)


def round_f16(a):
    """Nearest IEEE half-precision value (ties to even), via float32, as float64."""
    return np.asarray(a, dtype=np.float32).astype(np.float16).astype(F64)


class OperandRounding:
    """Where the precision model rounds: ``mm`` for operands of the weight
    products, ``att`` for the attention's q, k, v and probabilities, ``read``
    for the associative read's features and state copy (default: ``mm``)."""

    def __init__(self, mm, att, read=None):
        self.mm, self.att = mm, att
        self.read = mm if read is None else read


def round_split(a):
    """bf16 high part plus the bf16 rounding of what it drops (via float32)."""
    a32 = np.asarray(a, dtype=np.float32).astype(F64)
    hi = round_bf16(a32)
    return hi + round_bf16(a32 - hi)


EXACT = OperandRounding(_identity, _identity)
ROUNDING = {None: EXACT, "bf16": OperandRounding(round_bf16, round_f16),
            "bf16x2": OperandRounding(round_split, round_f16)}


# --------------------------------------------------------------------------
# Elementwise / row building blocks
# --------------------------------------------------------------------------

def rmsnorm(x, gain, eps):
    """x / sqrt(mean(x^2) + eps) * gain over the last axis (LLaMA RMSNorm)."""
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * _f64(gain)


def silu(x):
    return x / (1.0 + np.exp(-x))


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def dpfp(x, nu):
    """Deterministic parameter-free projection of order nu, on the last axis.

    r = [relu(x), relu(-x)] (length 2k); block j (j = 1..nu) is r * roll(r, j)
    with roll(r, j)_i = r_{(i-j) mod 2k} (numpy's np.roll convention).
    Output length 2 k nu, every entry >= 0.
    """
    x = _f64(x)
    r = np.concatenate([np.maximum(x, 0.0), np.maximum(-x, 0.0)], axis=-1)
    return np.concatenate([r * np.roll(r, j, axis=-1) for j in range(1, nu + 1)], axis=-1)


def rope_rotate_half(x, base):
    """Rotate-half rotary embedding on x [T, H, hd], position of row t = t.

    Pairs (i, i + hd/2) are rotated by angle t * base^(-2i/hd).
    """
    x = _f64(x)
    T, _, hd = x.shape
    half = hd // 2
    inv_freq = base ** (-(2.0 * np.arange(half, dtype=F64)) / hd)
    ang = np.arange(T, dtype=F64)[:, None] * inv_freq[None, :]        # [T, half]
    cos, sin = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def causal_gqa_attention(q, k, v, rnd=_identity):
    """softmax(q k^T / sqrt(hd) + causal mask) v per query head.

    q [T, Hq, hd], k/v [T, Hkv, hd]; query head h reads kv head h*Hkv//Hq.
    Returns [T, Hq*hd].  ``rnd`` (precision model only) is applied to the
    unnormalised probabilities before they multiply v.
    """
    T, Hq, hd = q.shape
    Hkv = k.shape[1]
    out = np.empty((T, Hq, hd), dtype=F64)
    mask = np.triu(np.ones((T, T), dtype=bool), k=1)
    for h in range(Hq):
        g = (h * Hkv) // Hq
        s = (q[:, h, :] @ k[:, g, :].T) / np.sqrt(hd)
        s = np.where(mask, -np.inf, s)
        s = s - s.max(axis=-1, keepdims=True)
        p = np.exp(s)
        out[:, h, :] = (rnd(p) @ v[:, g, :]) / p.sum(axis=-1, keepdims=True)
    return out.reshape(T, Hq * hd)


# --------------------------------------------------------------------------
# Associative memory (delta rule)
# --------------------------------------------------------------------------

def assoc_lookup(A, z, phi, eps, rnd=EXACT):
    """A phi / (z^T phi + eps) for each row of phi [R, P]; A [d, P], z [P]."""
    num = rnd.read(phi) @ rnd.read(A).T
    den = phi @ z + eps
    return num / den[:, None]


def assoc_read(x, wq_a, A, z, nu, eps, rnd=EXACT):
    """Memory read added to the residual stream: x + lookup(phi(W_Q x))."""
    phi = dpfp(rnd.mm(x) @ wq_a.T, nu)
    return x + assoc_lookup(A, z, phi, eps, rnd)


def delta_rule_update(A, z, keys, values, beta, nu, eps) -> Tuple[np.ndarray, np.ndarray]:
    """Delta-rule write of (keys [R,k], values [R,d], beta [R]) into (A, z).

    All R terms use the state from before the call (R = 1 for one write).
    """
    phi = dpfp(keys, nu)                                   # [R, P]
    zphi = phi @ z                                         # [R]
    vbar = (phi @ A.T) / (zphi + eps)[:, None]             # [R, d]
    gamma = np.clip(1.0 - zphi / (np.sum(phi * phi, axis=-1) + eps), 0.0, 1.0)
    dA = (beta[:, None] * (values - vbar)).T @ phi         # [d, P]
    dz = gamma @ phi                                       # [P]
    return A + dA, z + dz


def assoc_write(h_mem, wk_a, wv_a, wb_a, A, z, nu, eps, rnd=EXACT):
    """Write from the memory-token rows h_mem [M, d] of one layer's output.

    The rows are written one after another in row order; write i sees the
    state that write i-1 produced.
    """
    h_mem = rnd.mm(h_mem)
    keys = h_mem @ wk_a.T
    values = h_mem @ wv_a.T
    beta = sigmoid(h_mem @ wb_a)
    for i in range(h_mem.shape[0]):
        A, z = delta_rule_update(A, z, keys[i:i + 1], values[i:i + 1], beta[i:i + 1], nu, eps)
    return A, z


# --------------------------------------------------------------------------
# One cell and the whole grid
# --------------------------------------------------------------------------

def llama_block(x, cfg, W, l, rnd=EXACT):
    """Pre-norm LLaMA decoder layer on the rows of one cell (x [T_c, d])."""
    T = x.shape[0]
    Hq, Hkv, hd = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    n = rnd.mm(rmsnorm(x, W["norm1"][l], cfg.norm_eps))
    q = (n @ W["wq"][l].T).reshape(T, Hq, hd)
    k = (n @ W["wk"][l].T).reshape(T, Hkv, hd)
    v = rnd.att((n @ W["wv"][l].T).reshape(T, Hkv, hd))
    q = rnd.att(rope_rotate_half(q, cfg.rope_base))
    k = rnd.att(rope_rotate_half(k, cfg.rope_base))
    y = x + rnd.mm(causal_gqa_attention(q, k, v, rnd.att)) @ W["wo"][l].T
    n2 = rnd.mm(rmsnorm(y, W["norm2"][l], cfg.norm_eps))
    u = rnd.mm(silu(n2 @ W["w_gate"][l].T) * (n2 @ W["w_up"][l].T))
    return y + u @ W["w_down"][l].T


def cell_forward(x, cfg, W, l, A, z, rnd=EXACT):
    """Cell (l, s): read, LLaMA block, write.  Returns (h, A', z')."""
    nu, eps = cfg.dpfp_nu, cfg.assoc_eps
    x = assoc_read(x, W["a_wq"][l], A, z, nu, eps, rnd)
    h = llama_block(x, cfg, W, l, rnd)
    m0 = h.shape[0] - cfg.n_mem               # the memory rows close the cell
    A2, z2 = assoc_write(h[m0:], W["a_wk"][l], W["a_wv"][l], W["a_wbeta"][l], A, z, nu, eps, rnd)
    return h, A2, z2


def layer0_input(cfg, W, tokens, s):
    """[E[tokens of segment s]; memory embeddings] -> [T_c, d] (fewer rows for a short last segment)."""
    S = cfg.seg_len
    return np.concatenate([W["embed"][tokens[s * S:(s + 1) * S]], W["mem"]], axis=0)


def widen_weights(W: Dict[str, np.ndarray]) -> Dict[str, np.ndarray]:
    return {k: _f64(v) for k, v in W.items()}


def schedule(n_layers: int, n_segments: int, order: str):
    """The cell visiting order: list of steps, each a list of (l, s)."""
    if order == "seq":
        return [[(l, s)] for s in range(n_segments) for l in range(n_layers)]
    if order == "diag":
        steps = []
        for i in range(n_layers + n_segments - 1):
            steps.append([(l, i - l) for l in range(n_layers) if 0 <= i - l < n_segments])
        return steps
    raise ValueError(order)


def forward(cfg, W, tokens, n_segments, order="seq", A0=None, z0=None, W64=None, operands=None):
    """ARMT forward over n_segments segments.

    ``tokens`` holds N ids with (n_segments - 1) * S < N <= n_segments * S.
    The last segment may be short: it takes the remaining S' = N - (n - 1) S
    tokens, followed as usual by the M memory tokens (S' + M rows, positions
    0..S'+M-1).  The pages do not discuss a partial segment; this is the
    plainest reading (the segment is just shorter).
    Returns (hidden [N, d], A [L, d, P], z [L, P]) in float64.  ``A0``/``z0``
    give an initial memory state (zeros when None).  ``operands="bf16"``
    selects the bf16 operand-rounding precision model (module docstring).
    """
    rnd = ROUNDING[operands]
    L, d, P, S = cfg.n_layers, cfg.d_model, cfg.phi_dim, cfg.seg_len
    W = W64 if W64 is not None else widen_weights(W)
    tokens = np.asarray(tokens)
    N = tokens.shape[0]
    assert (n_segments - 1) * S < N <= n_segments * S
    A = [(_f64(A0[l]).copy() if A0 is not None else np.zeros((d, P), F64)) for l in range(L)]
    z = [(_f64(z0[l]).copy() if z0 is not None else np.zeros((P,), F64)) for l in range(L)]
    # outputs of each layer per segment; in a real run only the live wavefront
    # is kept, here a dict keyed by (l, s) is plain and small enough.
    acts = {}
    out = np.zeros((N, d), F64)
    for step in schedule(L, n_segments, order):
        for (l, s) in step:
            x = layer0_input(cfg, W, tokens, s) if l == 0 else acts.pop((l - 1, s))
            h, A[l], z[l] = cell_forward(x, cfg, W, l, A[l], z[l], rnd)
            if l == L - 1:
                seg = h.shape[0] - cfg.n_mem
                out[s * S:s * S + seg] = rmsnorm(h[:seg], W["norm_f"], cfg.norm_eps)
            else:
                acts[(l, s)] = h
    return out, np.stack(A), np.stack(z)



# --------------------------------------------------------------------------
# LM head and the relative-logits error (summary page, section 四)
# --------------------------------------------------------------------------
def lm_head_logits(hidden, head):
    """Logits of hidden rows against a head matrix [V, d]: logits = hidden head^T.

    The summary page (section 四) measures how far diagonal batching drifts
    from the sequential recurrence through the logits of the final hidden
    states; with a tied head the matrix is the token embedding.
    """
    return _f64(hidden) @ _f64(head).T


def relative_logits_error(logits, ref):
    """||logits - ref||_F / ||ref||_F, in fp64 (the section 四 error measure, as a relative norm)."""
    logits, ref = _f64(logits), _f64(ref)
    return float(np.linalg.norm(logits - ref) / np.linalg.norm(ref))
