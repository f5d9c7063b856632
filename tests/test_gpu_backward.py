"""GPU: the backward pass (armt_backward) against the fp64 gradient reference.

Section 四 of the summary page of "Diagonal Batching Unlocks Parallelism in
Recurrent Memory Transformers for Long Contexts" carries diagonal batching
over to the backward pass.  The library runs the adjoint over the reverse
anti-diagonals in fp32; oracle/armt_backward.py's backward_explicit (pinned
against finite differences of the numpy oracle's forward) gives the exact
gradients.  Every gradient tensor -- all weights, the initial state -- is held
to the fp32 bound of the forward tests: max-abs error <= 1e-4 of the
tensor's largest exact entry, cosine >= 1 - 1e-9.
"""
import dataclasses

import numpy as np
import pytest

from oracle import armt_backward as G
from recurrent_memory_transformer_gb300 import inputs as I

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from recurrent_memory_transformer_gb300 import armt as B  # noqa: E402
from recurrent_memory_transformer_gb300 import build as build_mod  # noqa: E402

from tests.test_gpu_parity import record  # noqa: E402

ERR_ARG = 1
REL, COS = 1e-4, 1e-9


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_mod.build()
    B.load_library()


def _cot(cfg, n_tok, seed, parts=("hidden", "A", "z")):
    rng = np.random.default_rng(seed)
    L, d, P = cfg.n_layers, cfg.d_model, cfg.phi_dim
    full = {"hidden": rng.standard_normal((n_tok, d)), "A": rng.standard_normal((L, d, P)),
            "z": rng.standard_normal((L, P))}
    return {k: (v if k in parts else np.zeros_like(v)) for k, v in full.items()}, parts


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _compare(name, got, ref):
    out = {}
    for k, r in ref.items():
        g = got[k].detach().cpu().numpy().astype(np.float64).reshape(r.shape)
        err = float(np.max(np.abs(g - r))) if r.size else 0.0
        scale = float(np.max(np.abs(r))) if r.size else 0.0
        nr, ng = np.linalg.norm(r), np.linalg.norm(g)
        cos = float(np.sum(g * r) / (nr * ng)) if nr > 0 and ng > 0 else (1.0 if nr == ng else 0.0)
        out[k] = {"max_abs": err, "scale": scale, "cos": cos}
    record(f"backward_{name}", **out)
    for k, st in out.items():
        assert np.isfinite(st["max_abs"]), (name, k)
        assert st["max_abs"] <= REL * st["scale"] + 1e-30, (name, k, st)
        if st["scale"] > 0:
            assert st["cos"] >= 1.0 - COS, (name, k, st)
    return out


CASES = [
    # name, config overrides, segments, tokens short of full, initial state, cotangents
    ("tiny", {}, 3, 0, False, ("hidden", "A", "z")),
    ("tiny_short_last_state", {}, 3, 5, True, ("hidden", "A", "z")),
    ("tiny_gqa", {"n_q_heads": 4, "n_kv_heads": 2, "head_dim": 32, "d_model": 128}, 2, 0, False,
     ("hidden", "A", "z")),
    ("tiny_hd64_L3_n5", {"n_layers": 3, "n_q_heads": 2, "n_kv_heads": 1, "head_dim": 64, "d_model": 128}, 5, 0,
     True, ("hidden", "A", "z")),
    ("tiny_one_segment", {}, 1, 0, False, ("hidden", "A", "z")),
    ("tiny_hidden_only", {}, 3, 0, False, ("hidden",)),
    ("tiny_state_only", {"n_layers": 3}, 4, 3, True, ("A", "z")),
    ("tiny_mem8_P192", {"n_mem": 8, "key_dim": 32}, 3, 0, True, ("hidden", "A", "z")),
    ("tiny_hd128", {"n_q_heads": 2, "n_kv_heads": 1, "head_dim": 128, "d_model": 256, "ffn_dim": 256}, 2, 3,
     False, ("hidden", "A", "z")),
    # several 64-wide tiles with ragged edges in every GEMM dimension, 3 attention tiles
    ("mid_tiles", {"n_layers": 3, "d_model": 128, "n_q_heads": 4, "n_kv_heads": 2, "head_dim": 32,
                   "ffn_dim": 256, "seg_len": 64, "n_mem": 16, "key_dim": 32}, 4, 7, True, ("hidden", "A", "z")),
]


@pytest.mark.parametrize("name,over,n_seg,short,with_state,parts", CASES)
def test_backward_matches_fp64_gradients(name, over, n_seg, short, with_state, parts):
    cfg = dataclasses.replace(I.TINY, **over)
    W = I.make_weights(cfg, seed=101, norm_jitter=0.1)
    tok = I.make_tokens(cfg, n_seg, seed=101)
    tok = tok[:tok.shape[0] - short]
    L, d, P = cfg.n_layers, cfg.d_model, cfg.phi_dim
    rng = np.random.default_rng(102)
    A0 = 0.01 * np.abs(rng.standard_normal((L, d, P))) if with_state else None
    z0 = 0.05 * np.abs(rng.standard_normal((L, P))) if with_state else None
    cot, parts = _cot(cfg, tok.shape[0], 103, parts)
    ref = G.backward_explicit(cfg, W, tok, n_seg, cot, A0, z0)
    m = B.Model(cfg, W)
    t = torch.from_numpy(tok).cuda()
    grads, (h, A, z) = m.backward(t, cot_hidden=_dev(cot["hidden"]) if "hidden" in parts else None,
                                  cot_A=_dev(cot["A"]) if "A" in parts else None,
                                  cot_z=_dev(cot["z"]) if "z" in parts else None,
                                  mem_A0=None if A0 is None else _dev(A0), mem_z0=None if z0 is None else _dev(z0),
                                  state_grads=with_state)
    torch.cuda.synchronize()
    m.armt_sync_status()
    # the forward it ran is the library's forward
    hf, Af, zf = m.forward_batch(t.view(1, -1), mem_A=None if A0 is None else _dev(A0).view(L, 1, d, P),
                                 mem_z=None if z0 is None else _dev(z0).view(L, 1, P))
    torch.cuda.synchronize()
    assert torch.equal(h, hf[0]) and torch.equal(A, Af[:, 0]) and torch.equal(z, zf[:, 0])
    got = dict(grads)
    if with_state:
        got["A0"], got["z0"] = grads["mem_A"], grads["mem_z"]
    ref = {k: v for k, v in ref.items()}
    _compare(name, got, ref)
    # bitwise reproducible
    grads2, _ = m.backward(t, cot_hidden=_dev(cot["hidden"]) if "hidden" in parts else None,
                           cot_A=_dev(cot["A"]) if "A" in parts else None,
                           cot_z=_dev(cot["z"]) if "z" in parts else None,
                           mem_A0=None if A0 is None else _dev(A0), mem_z0=None if z0 is None else _dev(z0),
                           state_grads=with_state)
    torch.cuda.synchronize()
    for k in grads:
        assert torch.equal(grads[k], grads2[k]), k
    launches, flops, ws = m.armt_backward_stats()
    assert launches > 0 and flops > 0 and ws > 0
    m.close()


BF16_SMALL = dataclasses.replace(I.ARMT_1B, n_layers=2, d_model=512, n_q_heads=4, n_kv_heads=4, head_dim=64,
                                 ffn_dim=1024, vocab=512, seg_len=128)


@pytest.mark.parametrize("precision", ["bf16", "bf16x2"])
def test_backward_of_bf16_models(precision):
    """bf16 models: the forward runs in the model's precision on the tensor
    cores and keeps fp32 cell inputs and states; the adjoint runs in fp32
    against fp32 copies of the bf16 weights.  The gradients are those of the
    exact model evaluated at the bf16 forward's cell inputs, so they sit
    within the forward's rounding of the fp64 gradients: cosine >= 0.999
    (the bound the forward's outputs are held to) on every gradient tensor
    in both precision modes, and in split precision also a relative L2
    error <= 5e-3 (its forward is accurate to ~1e-3).  Measured: bf16
    1 - cos <= 2.8e-4, relative L2 <= 2.4 %; split 1 - cos < 5e-7, relative
    L2 <= 6e-4."""
    cfg = dataclasses.replace(BF16_SMALL, precision=precision)
    W = I.make_weights(cfg, seed=131, norm_jitter=0.1)
    n_seg = 3
    tok = I.make_tokens(cfg, n_seg, seed=131)[:-9]
    cot, _ = _cot(cfg, tok.shape[0], 132)
    ref = G.backward_explicit(cfg, W, tok, n_seg, cot)
    m = B.Model(cfg, B.device_weight_tensors(cfg, W))
    t = torch.from_numpy(tok).cuda()
    grads, (h, A, z) = m.backward(t, cot_hidden=_dev(cot["hidden"]), cot_A=_dev(cot["A"]), cot_z=_dev(cot["z"]))
    torch.cuda.synchronize()
    m.armt_sync_status()
    hf, Af, zf = m.forward_batch(t.view(1, -1))
    torch.cuda.synchronize()
    assert torch.equal(h, hf[0]) and torch.equal(A, Af[:, 0]) and torch.equal(z, zf[:, 0])
    m.close()
    out = {}
    for k, r in ref.items():
        g = grads[k].cpu().numpy().astype(np.float64).reshape(r.shape)
        nr, ng = np.linalg.norm(r), np.linalg.norm(g)
        out[k] = {"cos": float(np.sum(g * r) / (nr * ng)) if nr > 0 and ng > 0 else 1.0,
                  "rel_l2": float(np.linalg.norm(g - r) / nr) if nr > 0 else 0.0}
    record(f"backward_bf16_model_{precision}", **out)
    for k, st in out.items():
        assert np.isfinite(st["rel_l2"]) and st["cos"] >= 0.999, (k, st)
        if precision == "bf16x2":
            assert st["rel_l2"] <= 5e-3, (k, st)


def test_backward_rejects_half_given_state():
    cfg = I.TINY
    m = B.Model(cfg, I.make_weights(cfg, seed=94))
    t = torch.from_numpy(I.make_tokens(cfg, 2, seed=94)).cuda()
    A0 = torch.zeros((cfg.n_layers, cfg.d_model, cfg.phi_dim), device="cuda")
    with pytest.raises(B.ArmtError) as e:
        m.backward(t, mem_A0=A0)
    assert e.value.status == ERR_ARG
    m.close()


def test_backward_allocation_cap_then_recovers(monkeypatch):
    """The backward's workspace is allocated on the first call: under a cap
    that leaves no room for it the call fails with ARMT_ERR_OOM and writes
    nothing; with the cap lifted the next call is correct."""
    cfg = I.TINY
    W = I.make_weights(cfg, seed=121, norm_jitter=0.1)
    tok = I.make_tokens(cfg, 3, seed=121)
    cot, _ = _cot(cfg, tok.shape[0], 122)
    m = B.Model(cfg, W)
    t = torch.from_numpy(tok).cuda()
    monkeypatch.setenv("ARMT_ALLOC_CAP_BYTES", "1")
    with pytest.raises(B.ArmtError) as e:
        m.backward(t, cot_hidden=_dev(cot["hidden"]))
    assert e.value.status == 4  # ARMT_ERR_OOM
    monkeypatch.delenv("ARMT_ALLOC_CAP_BYTES")
    grads, _ = m.backward(t, cot_hidden=_dev(cot["hidden"]), cot_A=_dev(cot["A"]), cot_z=_dev(cot["z"]))
    torch.cuda.synchronize()
    m.armt_sync_status()
    m.close()
    _compare("after_oom", grads, G.backward_explicit(cfg, W, tok, 3, cot))
