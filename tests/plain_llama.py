"""An independently written plain causal LLaMA stack, for pinning the oracle.

Used only by tests.  It shares nothing with oracle/armt_oracle.py: attention is
a per-position loop with an explicit running softmax, RoPE is written as
multiplication by unit complex numbers (x_i + j x_{i+hd/2}) e^{j t theta_i},
RMSNorm and SwiGLU are spelled out per row.  Slow by design; tiny inputs only.

With the associative memory empty (A = 0, z = 0) the memory read of an ARMT
cell adds exactly zero, so one ARMT segment must equal this plain stack run on
the segment rows followed by the memory-token rows (section 二 of the summary
page of "Diagonal Batching Unlocks Parallelism in Recurrent Memory
Transformers for Long Contexts": a recurrent memory transformer is a standard
transformer plus memory tokens carrying state between segments).
"""
import math

import numpy as np


def _rms_row(v, g, eps):
    s = 0.0
    for a in v:
        s += float(a) * float(a)
    scale = 1.0 / math.sqrt(s / len(v) + eps)
    return np.array([float(a) * scale * float(b) for a, b in zip(v, g)])


def _rope_complex(vec, t, base):
    hd = len(vec)
    half = hd // 2
    out = np.empty(hd)
    for i in range(half):
        theta = t * base ** (-2.0 * i / hd)
        c = complex(vec[i], vec[i + half]) * complex(math.cos(theta), math.sin(theta))
        out[i] = c.real
        out[i + half] = c.imag
    return out


def plain_layer(X, W, l, cfg):
    """One pre-norm decoder layer over rows X [T, d] (positions 0..T-1)."""
    T, d = X.shape
    Hq, Hkv, hd = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    wq = np.asarray(W["wq"][l], np.float64)
    wk = np.asarray(W["wk"][l], np.float64)
    wv = np.asarray(W["wv"][l], np.float64)
    wo = np.asarray(W["wo"][l], np.float64)
    g1 = np.asarray(W["norm1"][l], np.float64)
    g2 = np.asarray(W["norm2"][l], np.float64)
    Q = np.zeros((T, Hq, hd)); K = np.zeros((T, Hkv, hd)); V = np.zeros((T, Hkv, hd))
    for t in range(T):
        nrow = _rms_row(X[t], g1, cfg.norm_eps)
        for h in range(Hq):
            Q[t, h] = _rope_complex(wq[h * hd:(h + 1) * hd] @ nrow, t, cfg.rope_base)
        for h in range(Hkv):
            K[t, h] = _rope_complex(wk[h * hd:(h + 1) * hd] @ nrow, t, cfg.rope_base)
            V[t, h] = wv[h * hd:(h + 1) * hd] @ nrow
    group = Hq // Hkv
    Y = np.array(X, dtype=np.float64, copy=True)
    for t in range(T):
        att = np.zeros(Hq * hd)
        for h in range(Hq):
            kvh = h // group
            # running (online) softmax over positions 0..t
            m, den, acc = -math.inf, 0.0, np.zeros(hd)
            for u in range(t + 1):
                sc = float(Q[t, h] @ K[u, kvh]) / math.sqrt(hd)
                if sc > m:
                    r = math.exp(m - sc) if m > -math.inf else 0.0
                    den *= r
                    acc *= r
                    m = sc
                w = math.exp(sc - m)
                den += w
                acc += w * V[u, kvh]
            att[h * hd:(h + 1) * hd] = acc / den
        Y[t] += wo @ att
    wg = np.asarray(W["w_gate"][l], np.float64)
    wu = np.asarray(W["w_up"][l], np.float64)
    wd = np.asarray(W["w_down"][l], np.float64)
    H = Y.copy()
    for t in range(T):
        nrow = _rms_row(Y[t], g2, cfg.norm_eps)
        gate = wg @ nrow
        up = wu @ nrow
        act = np.array([gv / (1.0 + math.exp(-gv)) * uv for gv, uv in zip(gate, up)])
        H[t] += wd @ act
    return H


def plain_stack(X, W, cfg):
    """All layers then the final RMSNorm on every row."""
    for l in range(cfg.n_layers):
        X = plain_layer(X, W, l, cfg)
    gf = np.asarray(W["norm_f"], np.float64)
    return np.stack([_rms_row(row, gf, cfg.norm_eps) for row in X])
