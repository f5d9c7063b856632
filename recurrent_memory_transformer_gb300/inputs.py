"""Seeded synthetic inputs: model shapes, random-init weights and token ids.

This module is the one piece shared by the CUDA path's tests/benchmarks and the
fp64 oracle.  It holds no arithmetic of the method itself: it only names the
model shapes and draws random numbers in a fixed, documented order.

Workloads follow the summary page of "Diagonal Batching Unlocks Parallelism in
Recurrent Memory Transformers for Long Contexts" (section 三: Llama-3-family
models at 160M/1B/3B/8B; section 四: random input sequences).  No dataset and
no trained checkpoint is involved: weights are N(0, 0.02) (every projection
matrix, the token embedding and the memory-token embeddings), RMSNorm gains
are 1 unless ``norm_jitter`` asks for 1 + jitter * N(0, 1) (tests use that so
a misapplied gain cannot hide), token ids are uniform in [0, vocab).

Draw order (numpy PCG64 ``default_rng(seed)``, float32 standard normals):
  embed [V, d], mem [M, d],
  wq [L, Hq*hd, d], wk [L, Hkv*hd, d], wv [L, Hkv*hd, d], wo [L, d, Hq*hd],
  w_gate [L, F, d], w_up [L, F, d], w_down [L, d, F],
  a_wq [L, k, d], a_wk [L, k, d], a_wv [L, d, d], a_wbeta [L, d],
  then (only when norm_jitter > 0) norm1 [L, d], norm2 [L, d], norm_f [d].
Token ids [n_segments * S] (int32, uniform in [0, V)) come from a second
PCG64 stream, ``default_rng([seed, 1])``, so they can be drawn alone.
For bf16 models every floating tensor is rounded to the nearest bf16 value
(ties to even) and kept as float32 holding exactly that value, so the GPU and
the oracle see the same numbers.
"""
from __future__ import annotations

import dataclasses
from typing import Dict

import numpy as np

WEIGHT_KEYS = (
    "embed", "mem",
    "wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down",
    "a_wq", "a_wk", "a_wv", "a_wbeta",
    "norm1", "norm2", "norm_f",
)


@dataclasses.dataclass(frozen=True)
class ArmtConfig:
    """Shape of one ARMT model (LLaMA block + per-layer associative memory)."""
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    seg_len: int          # S: segment tokens per cell
    n_mem: int            # M: memory tokens appended to each segment
    key_dim: int          # k: associative key dim (DPFP input)
    dpfp_nu: int          # nu: DPFP order; feature dim P = 2 * k * nu
    norm_eps: float = 1e-5
    rope_base: float = 10000.0
    assoc_eps: float = 1e-6
    dtype: str = "f32"    # "f32" or "bf16"
    precision: str = "bf16"  # bf16 models: "bf16" or "bf16x2" (split activations)

    @property
    def rows(self) -> int:
        """T_c = S + M rows per cell."""
        return self.seg_len + self.n_mem

    @property
    def phi_dim(self) -> int:
        return 2 * self.key_dim * self.dpfp_nu

    def n_params_layer(self) -> int:
        d, hd = self.d_model, self.head_dim
        return (d * (self.n_q_heads + 2 * self.n_kv_heads) * hd + self.n_q_heads * hd * d
                + 3 * d * self.ffn_dim)


# The five workloads: tiny fp32 parity model, ARMT-1B at 8 segments (parity +
# throughput), ARMT-1B at 128 segments (131,072 tokens, the headline), 3B, 8B.
TINY = ArmtConfig(n_layers=2, d_model=64, n_q_heads=2, n_kv_heads=2, head_dim=32, ffn_dim=128,
                  vocab=256, seg_len=16, n_mem=4, key_dim=16, dpfp_nu=3, norm_eps=1e-5,
                  rope_base=10000.0, dtype="f32")
ARMT_1B = ArmtConfig(n_layers=16, d_model=2048, n_q_heads=32, n_kv_heads=8, head_dim=64,
                     ffn_dim=8192, vocab=128256, seg_len=1024, n_mem=16, key_dim=64, dpfp_nu=3,
                     norm_eps=1e-5, rope_base=500000.0, dtype="bf16")
ARMT_3B = ArmtConfig(n_layers=28, d_model=3072, n_q_heads=24, n_kv_heads=8, head_dim=128,
                     ffn_dim=8192, vocab=128256, seg_len=1024, n_mem=16, key_dim=64, dpfp_nu=3,
                     norm_eps=1e-5, rope_base=500000.0, dtype="bf16")
ARMT_8B = ArmtConfig(n_layers=32, d_model=4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
                     ffn_dim=14336, vocab=128256, seg_len=1024, n_mem=16, key_dim=64, dpfp_nu=3,
                     norm_eps=1e-5, rope_base=500000.0, dtype="bf16")

WORKLOADS = {
    "tiny": (TINY, 4, 0),              # (config, n_segments, seed)
    "armt-1b-8k": (ARMT_1B, 8, 1),
    "armt-1b-131k": (ARMT_1B, 128, 1),
    "armt-3b-32k": (ARMT_3B, 32, 2),
    "armt-3b-131k": (ARMT_3B, 128, 2),
    # 8B at 131,072 tokens with segment lengths 512 / 1024 / 2048 (the
    # segment-size sweep of section 三), 16 memory tokens each
    "armt-8b-131k-s512": (dataclasses.replace(ARMT_8B, seg_len=512), 256, 3),
    "armt-8b-131k": (ARMT_8B, 128, 3),
    "armt-8b-131k-s2048": (dataclasses.replace(ARMT_8B, seg_len=2048), 64, 3),
}

# Workloads whose weights are drawn on the GPU (make_weights_device): the 3B
# and 8B shapes need no oracle parity, and a host draw of 6-15 GB of normals
# would dominate a benchmark run.
DEVICE_WEIGHT_WORKLOADS = ("armt-3b-32k", "armt-3b-131k", "armt-8b-131k-s512", "armt-8b-131k",
                           "armt-8b-131k-s2048")


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 value (ties to even), kept as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    rounded = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return rounded.view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values that are already bf16-representable."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def make_weights(cfg: ArmtConfig, seed: int, std: float = 0.02,
                 norm_jitter: float = 0.0) -> Dict[str, np.ndarray]:
    """Random-init weights in the draw order given in the module docstring.

    Returns float32 arrays (bf16-representable when ``cfg.dtype == "bf16"``),
    stacked over layers, each linear map stored (out, in).
    """
    rng = np.random.default_rng(seed)
    L, d, hd, F = cfg.n_layers, cfg.d_model, cfg.head_dim, cfg.ffn_dim

    def normal(*shape):
        a = rng.standard_normal(size=shape, dtype=np.float32)
        a *= np.float32(std)
        return a

    w = {}
    w["embed"] = normal(cfg.vocab, d)
    w["mem"] = normal(cfg.n_mem, d)
    w["wq"] = normal(L, cfg.n_q_heads * hd, d)
    w["wk"] = normal(L, cfg.n_kv_heads * hd, d)
    w["wv"] = normal(L, cfg.n_kv_heads * hd, d)
    w["wo"] = normal(L, d, cfg.n_q_heads * hd)
    w["w_gate"] = normal(L, F, d)
    w["w_up"] = normal(L, F, d)
    w["w_down"] = normal(L, d, F)
    w["a_wq"] = normal(L, cfg.key_dim, d)
    w["a_wk"] = normal(L, cfg.key_dim, d)
    w["a_wv"] = normal(L, d, d)
    w["a_wbeta"] = normal(L, d)
    if norm_jitter > 0:
        for key, shape in (("norm1", (L, d)), ("norm2", (L, d)), ("norm_f", (d,))):
            g = rng.standard_normal(size=shape, dtype=np.float32)
            w[key] = np.float32(1.0) + np.float32(norm_jitter) * g
    else:
        w["norm1"] = np.ones((L, d), np.float32)
        w["norm2"] = np.ones((L, d), np.float32)
        w["norm_f"] = np.ones((d,), np.float32)
    if cfg.dtype == "bf16":
        for key in WEIGHT_KEYS:
            w[key] = round_to_bf16(w[key])
    return w


def weight_shapes(cfg: ArmtConfig) -> Dict[str, tuple]:
    """Shape of every weight array, in draw order (linear maps stored (out, in))."""
    L, d, hd, F = cfg.n_layers, cfg.d_model, cfg.head_dim, cfg.ffn_dim
    return {"embed": (cfg.vocab, d), "mem": (cfg.n_mem, d),
            "wq": (L, cfg.n_q_heads * hd, d), "wk": (L, cfg.n_kv_heads * hd, d),
            "wv": (L, cfg.n_kv_heads * hd, d), "wo": (L, d, cfg.n_q_heads * hd),
            "w_gate": (L, F, d), "w_up": (L, F, d), "w_down": (L, d, F),
            "a_wq": (L, cfg.key_dim, d), "a_wk": (L, cfg.key_dim, d), "a_wv": (L, d, d),
            "a_wbeta": (L, d), "norm1": (L, d), "norm2": (L, d), "norm_f": (d,)}


def make_weights_device(cfg: ArmtConfig, seed: int, std: float = 0.02, device="cuda"):
    """Random-init weights drawn on the GPU, for shapes too large to draw on the host.

    Same keys, shapes and key order as ``make_weights`` (norm gains 1), but the
    normals come from a torch CUDA generator seeded with ``seed``, so the
    values differ from the host draw.  Returns torch tensors on ``device`` in
    the model's element type (bf16 or fp32).
    """
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    L, d, hd, F = cfg.n_layers, cfg.d_model, cfg.head_dim, cfg.ffn_dim

    def normal(*shape):
        a = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        a.mul_(std)
        return a.to(dt)

    shapes = weight_shapes(cfg)
    w = {k: normal(*shapes[k]) for k in shapes if not k.startswith("norm")}
    w["norm1"] = torch.ones((L, d), device=device, dtype=dt)
    w["norm2"] = torch.ones((L, d), device=device, dtype=dt)
    w["norm_f"] = torch.ones((d,), device=device, dtype=dt)
    return w


def make_tokens(cfg: ArmtConfig, n_segments: int, seed: int, stream: int = 1) -> np.ndarray:
    """Token ids, int32 uniform in [0, vocab), n_segments * S of them.

    Drawn from their own PCG64 stream (``seed`` spawned with ``stream``) so
    that generating tokens does not require generating the weights first.
    """
    rng = np.random.default_rng([seed, stream])
    return rng.integers(0, cfg.vocab, size=n_segments * cfg.seg_len, dtype=np.int64).astype(np.int32)


def make_workload(name: str, norm_jitter: float = 0.0):
    """(cfg, n_segments, weights, tokens) for one named workload."""
    cfg, n_seg, seed = WORKLOADS[name]
    return cfg, n_seg, make_weights(cfg, seed, norm_jitter=norm_jitter), make_tokens(cfg, n_seg, seed)
