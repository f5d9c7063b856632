"""An independently written 16-bit-operand emulation of ARMT cells, for pinning
the oracle's precision model (``armt_oracle.forward(operands="bf16")``).

Used only by tests.  It shares nothing with oracle/armt_oracle.py: every
step is written out per row and per head with Python loops, DPFP by index
arithmetic, rotary embedding as multiplication by unit complex numbers,
softmax with an explicit maximum, and the rounding to bf16 goes through
torch's own float32 -> bfloat16 conversion (round to nearest even) instead
of the oracle's bit manipulation (torch's float16 conversion for the
attention operands).  Slow by design; tiny inputs only.

The precision model rounds a value to its operand type at the points where
the bf16 kernel path feeds a tensor-core operand, and nowhere else -- bf16
for the operands of weight products, fp16 for the attention's own operands
(marked *):
  "xq"    the layer input, before the associative query projection;
  "phi"   the read features in the numerator A phi (the denominator
          z^T phi + eps keeps the unrounded features);
  "A"     the state copy in that numerator;
  "n1"    the first RMSNorm output (input of the q, k, v projections);
  "qk"    q and k after the rotary embedding (*);
  "v"     v (*);
  "P"     the attention probabilities exp(s - max) before they multiply v
          (the row sum stays unrounded) (*);
  "att"   the attention output (input of the output projection);
  "n2"    the second RMSNorm output (input of the gate / up projections);
  "u"     the SwiGLU output (input of the down projection);
  "hmem"  the memory-token rows of the cell's output, before the write's
          key / value / strength projections.
Everything else -- the residual stream, norm statistics, softmax maxima and
sums, the memory state and the write arithmetic -- is exact (fp64).

With ``split=True`` it emulates the split precision mode instead: the
operands of the weight products and of the read ("xq", "phi", "A", "n1",
"att", "n2", "u", "hmem") are carried as a bf16 high part plus the bf16
rounding of the residual; the attention operands stay fp16.
"""
import math

import numpy as np

ALL_POINTS = ("xq", "phi", "A", "n1", "qk", "v", "P", "att", "n2", "u", "hmem")
HALF_POINTS = ("qk", "v", "P")   # rounded to fp16; the rest to bf16


def _to_16bit(a, half):
    import torch
    t = torch.from_numpy(np.asarray(a, np.float64).astype(np.float32))
    return t.to(torch.float16 if half else torch.bfloat16).to(torch.float64).numpy()


def _to_split(a):
    import torch
    t = torch.from_numpy(np.asarray(a, np.float64).astype(np.float32))
    hi = t.to(torch.bfloat16).to(torch.float32)
    lo = (t - hi).to(torch.bfloat16).to(torch.float32)
    return hi.to(torch.float64).numpy() + lo.to(torch.float64).numpy()


class _Round:
    def __init__(self, points, split=False):
        self.points = set(points)
        self.split = split

    def __call__(self, name, a):
        if name not in self.points:
            return np.asarray(a, np.float64)
        if self.split and name not in HALF_POINTS:
            return _to_split(a)
        return _to_16bit(a, name in HALF_POINTS)


def _dpfp(x, nu):
    k = len(x)
    r = [max(float(v), 0.0) for v in x] + [max(-float(v), 0.0) for v in x]
    n = 2 * k
    return np.array([r[i] * r[(i - j) % n] for j in range(1, nu + 1) for i in range(n)])


def _rms(v, g, eps):
    s = sum(float(a) * float(a) for a in v)
    inv = 1.0 / math.sqrt(s / len(v) + eps)
    return np.array([float(a) * inv * float(b) for a, b in zip(v, g)])


def _rotate(vec, t, base):
    hd = len(vec)
    half = hd // 2
    out = np.empty(hd)
    for i in range(half):
        ang = t * base ** (-2.0 * i / hd)
        c = complex(vec[i], vec[i + half]) * complex(math.cos(ang), math.sin(ang))
        out[i], out[i + half] = c.real, c.imag
    return out


def cell(X, W, l, A, z, cfg, rnd):
    """One cell: read, decoder layer, in-order delta-rule writes.  X [T, d]."""
    T, d = X.shape
    Hq, Hkv, hd = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    nu, eps = cfg.dpfp_nu, cfg.assoc_eps
    w = {k: np.asarray(v[l] if k not in ("embed", "mem", "norm_f") else v, np.float64) for k, v in W.items()}
    # associative read, row by row
    A_num = rnd("A", A)
    Xr = np.empty_like(X)
    for t in range(T):
        phi = _dpfp(w["a_wq"] @ rnd("xq", X[t]), nu)
        den = float(z @ phi) + eps
        Xr[t] = X[t] + (A_num @ rnd("phi", phi)) / den
    # attention sub-layer
    Q = np.zeros((T, Hq, hd)); K = np.zeros((T, Hkv, hd)); V = np.zeros((T, Hkv, hd))
    for t in range(T):
        n = rnd("n1", _rms(Xr[t], w["norm1"], cfg.norm_eps))
        for h in range(Hq):
            Q[t, h] = rnd("qk", _rotate(w["wq"][h * hd:(h + 1) * hd] @ n, t, cfg.rope_base))
        for h in range(Hkv):
            K[t, h] = rnd("qk", _rotate(w["wk"][h * hd:(h + 1) * hd] @ n, t, cfg.rope_base))
            V[t, h] = rnd("v", w["wv"][h * hd:(h + 1) * hd] @ n)
    Y = Xr.copy()
    for t in range(T):
        att = np.zeros(Hq * hd)
        for h in range(Hq):
            g = h * Hkv // Hq
            s = [float(Q[t, h] @ K[u, g]) / math.sqrt(hd) for u in range(t + 1)]
            mx = max(s)
            p = [math.exp(a - mx) for a in s]
            pr = rnd("P", np.array(p))
            o = sum(pr[u] * V[u, g] for u in range(t + 1)) / sum(p)
            att[h * hd:(h + 1) * hd] = o
        Y[t] = Y[t] + w["wo"] @ rnd("att", att)
    # MLP sub-layer
    H = Y.copy()
    for t in range(T):
        n2 = rnd("n2", _rms(Y[t], w["norm2"], cfg.norm_eps))
        gate = w["w_gate"] @ n2
        up = w["w_up"] @ n2
        u = rnd("u", np.array([a / (1.0 + math.exp(-a)) * b for a, b in zip(gate, up)]))
        H[t] = H[t] + w["w_down"] @ u
    # writes from the memory-token rows, one after another
    A = A.copy(); z = z.copy()
    for t in range(T - cfg.n_mem, T):
        hm = rnd("hmem", H[t])
        key = w["a_wk"] @ hm
        val = w["a_wv"] @ hm
        beta = 1.0 / (1.0 + math.exp(-float(w["a_wbeta"] @ hm)))
        phi = _dpfp(key, nu)
        zp = float(z @ phi)
        ff = float(phi @ phi)
        vbar = (A @ phi) / (zp + eps)
        A = A + beta * np.outer(val - vbar, phi)
        z = z + min(max(1.0 - zp / (ff + eps), 0.0), 1.0) * phi
    return H, A, z


def forward(cfg, W, tokens, n_segments, points=ALL_POINTS, split=False):
    """Segment by segment, layer by layer; returns (hidden, A [L,d,P], z [L,P])."""
    rnd = _Round(points, split)
    L, d, P, S = cfg.n_layers, cfg.d_model, cfg.phi_dim, cfg.seg_len
    emb, mem, gf = (np.asarray(W[k], np.float64) for k in ("embed", "mem", "norm_f"))
    A = [np.zeros((d, P)) for _ in range(L)]
    z = [np.zeros(P) for _ in range(L)]
    out = []
    for s in range(n_segments):
        seg = tokens[s * S:(s + 1) * S]
        X = np.concatenate([emb[seg], mem])
        for l in range(L):
            X, A[l], z[l] = cell(X, W, l, A[l], z[l], cfg, rnd)
        out.extend(_rms(X[t], gf, cfg.norm_eps) for t in range(len(seg)))
    return np.array(out), np.stack(A), np.stack(z)
