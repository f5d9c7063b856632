"""GPU: the persistent wavefront schedule (ARMT_SCHEDULE_WAVEFRONT, fp32 models).

One cooperative launch runs the whole forward; each stage of each cell starts
once the device-side counters of the stages it reads from are complete
(section 二 of the summary page of "Diagonal Batching Unlocks Parallelism in
Recurrent Memory Transformers for Long Contexts": cell (l, s) needs only
(l-1, s) and (l, s-1)).  It runs the same block code on the same data as the
diagonal and sequential schedules, so the three agree bitwise; against the
fp64 oracle it meets the fp32 bounds.  A dependency that never completes (the
ARMT_TEST_STALL_AFTER hook) makes the waiting tasks give up with
ARMT_ERR_TIMEOUT, and the next call is correct.
"""
import dataclasses
import time

import numpy as np
import pytest

from oracle import armt_oracle as O
from recurrent_memory_transformer_gb300 import inputs as I

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from recurrent_memory_transformer_gb300 import armt as B  # noqa: E402
from recurrent_memory_transformer_gb300 import build as build_mod  # noqa: E402

from tests.test_gpu_parity import assert_fp32_close, record, stats  # noqa: E402

ERR_UNSUPPORTED, ERR_TIMEOUT = 3, 6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_mod.build()
    B.load_library()


def _run(m, tok, schedule):
    t = torch.from_numpy(np.ascontiguousarray(tok)).cuda().view(1, -1)
    h, A, z = m.forward_batch(t, schedule=schedule)
    torch.cuda.synchronize()
    m.armt_sync_status()
    return h[0], A[:, 0], z[:, 0]


CASES = [
    ("tiny", {}, 64),
    ("tiny_gqa", {"n_q_heads": 4, "n_kv_heads": 2, "head_dim": 32, "d_model": 128}, 48),
    ("tiny_L3_n5", {"n_layers": 3}, 80),
    ("tiny_one_segment", {}, 16),
    ("tiny_hd64", {"n_q_heads": 2, "n_kv_heads": 1, "head_dim": 64, "d_model": 128}, 48),
    ("tiny_short_last", {"n_layers": 3}, 64 - 5),
    ("tiny_L4_n12", {"n_layers": 4}, 16 * 12),
    ("tiny_hd128", {"n_q_heads": 2, "n_kv_heads": 1, "head_dim": 128, "d_model": 256, "ffn_dim": 256}, 40),
]


@pytest.mark.parametrize("name,over,n_tok", CASES)
def test_wavefront_equals_diagonal_and_matches_oracle(name, over, n_tok):
    cfg = dataclasses.replace(I.TINY, **over)
    W = I.make_weights(cfg, seed=91, norm_jitter=0.1)
    tok = np.random.default_rng(91).integers(0, cfg.vocab, size=n_tok).astype(np.int32)
    m = B.Model(cfg, W)
    hw, Aw, zw = _run(m, tok, B.SCHEDULE_WAVEFRONT)
    hd, Ad, zd = _run(m, tok, B.SCHEDULE_DIAGONAL)
    hs, As, zs = _run(m, tok, B.SCHEDULE_SEQUENTIAL)
    hw2, Aw2, zw2 = _run(m, tok, B.SCHEDULE_WAVEFRONT)   # twice: deterministic
    m.close()
    assert torch.equal(hw, hd) and torch.equal(Aw, Ad) and torch.equal(zw, zd), name
    assert torch.equal(hw, hs) and torch.equal(Aw, As) and torch.equal(zw, zs), name
    assert torch.equal(hw, hw2) and torch.equal(Aw, Aw2) and torch.equal(zw, zw2), name
    n_seg = -(-n_tok // cfg.seg_len)
    ho, Ao, zo = O.forward(cfg, W, tok, n_seg)
    sh, sa, sz = stats(hw.cpu().numpy(), ho), stats(Aw.cpu().numpy(), Ao), stats(zw.cpu().numpy(), zo)
    record(f"wavefront_{name}", hidden=sh, A=sa, z=sz)
    assert_fp32_close(sh, sa, sz)


def test_wavefront_resume_and_host_entry_point():
    cfg = I.TINY
    W = I.make_weights(cfg, seed=92, norm_jitter=0.1)
    tok = I.make_tokens(cfg, 6, seed=92)
    m = B.Model(cfg, W)
    h, A, z = _run(m, tok, B.SCHEDULE_WAVEFRONT)
    S = cfg.seg_len
    ta = torch.from_numpy(tok[:2 * S]).cuda().view(1, -1)
    tb = torch.from_numpy(tok[2 * S:]).cuda().view(1, -1)
    ha, Aa, za = m.forward_batch(ta, schedule=B.SCHEDULE_WAVEFRONT)
    hb, Ab, zb = m.forward_batch(tb, schedule=B.SCHEDULE_WAVEFRONT, mem_A=Aa, mem_z=za)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([ha[0], hb[0]]), h) and torch.equal(Ab[:, 0], A) and torch.equal(zb[:, 0], z)
    hh = np.empty((6 * S, cfg.d_model), np.float32)
    Ah = np.empty(m.a_elems, np.float32)
    zh = np.empty(m.z_elems, np.float32)
    m.armt_forward_host(tok, 6, hh, Ah, zh, schedule=B.SCHEDULE_WAVEFRONT)
    assert np.array_equal(hh, h.cpu().numpy())
    assert np.array_equal(Ah, A.cpu().numpy().ravel()) and np.array_equal(zh, z.cpu().numpy().ravel())
    assert m.armt_launch_count(6, B.SCHEDULE_WAVEFRONT) == 1
    m.close()


def test_wavefront_dependency_timeout_then_recovers(monkeypatch):
    cfg = dataclasses.replace(I.TINY, n_layers=3)
    W = I.make_weights(cfg, seed=93)
    tok = I.make_tokens(cfg, 4, seed=93)
    m = B.Model(cfg, W)
    h0, A0, z0 = _run(m, tok, B.SCHEDULE_WAVEFRONT)
    # completions from task 200 on are never counted: the tasks that depend on
    # them wait until the (shortened) limit runs out
    monkeypatch.setenv("ARMT_TEST_STALL_AFTER", "200")
    monkeypatch.setenv("ARMT_WAIT_LIMIT_MS", "50")
    t = torch.from_numpy(tok).cuda().view(1, -1)
    m.forward_batch(t, schedule=B.SCHEDULE_WAVEFRONT)
    with pytest.raises(B.ArmtError) as e:
        m.armt_sync_status()
    assert e.value.status == ERR_TIMEOUT
    monkeypatch.delenv("ARMT_TEST_STALL_AFTER")
    monkeypatch.delenv("ARMT_WAIT_LIMIT_MS")
    h1, A1, z1 = _run(m, tok, B.SCHEDULE_WAVEFRONT)
    assert torch.equal(h1, h0) and torch.equal(A1, A0) and torch.equal(z1, z0)
    m.close()


def test_wavefront_rejects_bf16_models_and_batches():
    cfg = dataclasses.replace(I.ARMT_1B, n_layers=1, vocab=4096)
    W = I.make_weights(cfg, seed=94)
    m = B.Model(cfg, B.device_weight_tensors(cfg, W))
    t = torch.from_numpy(I.make_tokens(cfg, 1, seed=94)).cuda().view(1, -1)
    with pytest.raises(B.ArmtError) as e:
        m.forward_batch(t, schedule=B.SCHEDULE_WAVEFRONT)
    assert e.value.status == ERR_UNSUPPORTED
    m.close()
    cfg = I.TINY
    m = B.Model(cfg, I.make_weights(cfg, seed=94))
    t2 = torch.from_numpy(np.stack([I.make_tokens(cfg, 2, seed=94)] * 2)).cuda()
    with pytest.raises(B.ArmtError) as e:
        m.forward_batch(t2, schedule=B.SCHEDULE_WAVEFRONT)
    assert e.value.status == ERR_UNSUPPORTED
    m.close()


def test_wavefront_time_against_per_diagonal_launches():
    """A mid-size fp32 model (4 layers, d 256) over 8 and 64 segments: the
    wavefront's one launch against the diagonal schedule's ~13 launches per
    step, bitwise equal; the times are recorded."""
    cfg = dataclasses.replace(I.ARMT_1B, n_layers=4, d_model=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                              ffn_dim=512, vocab=1000, seg_len=64, dtype="f32")
    W = I.make_weights(cfg, seed=95)
    m = B.Model(cfg, W)
    res = {}
    for n_seg in (8, 64):
        tok = I.make_tokens(cfg, n_seg, seed=95)
        out = {}
        for name, sch in (("diagonal", B.SCHEDULE_DIAGONAL), ("wavefront", B.SCHEDULE_WAVEFRONT)):
            out[name] = _run(m, tok, sch)
            t0 = time.perf_counter()
            for _ in range(3):
                _run(m, tok, sch)
            res[f"{name}_{n_seg}_ms"] = (time.perf_counter() - t0) / 3 * 1000.0
        for a, b in zip(out["diagonal"], out["wavefront"]):
            assert torch.equal(a, b), n_seg
    record("wavefront_timing_fp32_d256_L4", **res)
    m.close()


def test_tracing_changes_no_result():
    """armt_set_tracing only wraps steps in NVTX ranges: every schedule and
    the backward give bitwise the same results with it on."""
    cfg = dataclasses.replace(I.TINY, n_layers=3)
    W = I.make_weights(cfg, seed=96, norm_jitter=0.1)
    tok = I.make_tokens(cfg, 4, seed=96)
    t = torch.from_numpy(tok).cuda()
    m = B.Model(cfg, W)
    outs = {}
    for tracing in (False, True):
        m.armt_set_tracing(tracing)
        res = [_run(m, tok, sch) for sch in (B.SCHEDULE_DIAGONAL, B.SCHEDULE_SEQUENTIAL, B.SCHEDULE_WAVEFRONT)]
        g, _ = m.backward(t, cot_hidden=torch.ones((tok.shape[0], cfg.d_model), device="cuda"))
        torch.cuda.synchronize()
        outs[tracing] = (res, g)
    m.close()
    for a, b in zip(outs[False][0], outs[True][0]):
        for x, y in zip(a, b):
            assert torch.equal(x, y)
    for k in outs[False][1]:
        assert torch.equal(outs[False][1][k], outs[True][1][k]), k
