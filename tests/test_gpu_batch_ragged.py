"""GPU: a short last segment and the batched forward (armt_forward_batch).

  - short last segment: n_tokens not a multiple of S; the last segment holds
    the remaining tokens followed by the memory tokens.  Against the fp64
    oracle (fp32 model: the bounds of test_gpu_parity.assert_fp32_close; bf16:
    the derived bounds of test_gpu_parity), diagonal == sequential bitwise, and everything before
    the last segment bitwise equal to the run without it;
  - batch: each sequence of a batched call is bitwise equal to the same
    sequence run alone (batch 1), in both schedules; resuming a batch from
    its state reproduces the one-call result bitwise.
"""
import dataclasses

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

from tests.test_gpu_parity import _derived_bounds_hold, assert_fp32_close, record, stats  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_mod.build()
    B.load_library()


def _tokens(cfg, n_tok, seed, batch=1):
    rng = np.random.default_rng(seed)
    return rng.integers(0, cfg.vocab, size=(batch, n_tok)).astype(np.int32)


def _equal(a, b):
    return bool(torch.equal(a, b))


@pytest.mark.parametrize("n_tok", [64 - 1, 64 - 5, 48 + 1, 7, 16])
def test_tiny_fp32_short_last_segment_matches_oracle(n_tok):
    cfg = I.TINY
    W = I.make_weights(cfg, seed=61, norm_jitter=0.1)
    tok = _tokens(cfg, n_tok, 61)
    m = B.Model(cfg, W)
    t = torch.from_numpy(tok).cuda()
    hd, Ad, zd = m.forward_batch(t)
    hs, As, zs = m.forward_batch(t, schedule=B.SCHEDULE_SEQUENTIAL)
    torch.cuda.synchronize()
    m.armt_sync_status()
    assert _equal(hd, hs) and _equal(Ad, As) and _equal(zd, zs)
    n_seg = -(-n_tok // cfg.seg_len)
    ho, Ao, zo = O.forward(cfg, W, tok[0], n_seg)
    sh = stats(hd[0].cpu().numpy(), ho)
    sa = stats(Ad[:, 0].cpu().numpy(), Ao)
    sz = stats(zd[:, 0].cpu().numpy(), zo)
    record(f"tiny_short_{n_tok}", hidden=sh, A=sa, z=sz)
    assert hd.shape == (1, n_tok, cfg.d_model)
    assert_fp32_close(sh, sa, sz)
    # the full segments before the short one do not depend on it
    full = (n_seg - 1) * cfg.seg_len
    if full > 0:
        hp, Ap, zp = m.forward(t[0, :full].contiguous(), n_seg - 1)
        torch.cuda.synchronize()
        assert _equal(hp, hd[0, :full])
    m.close()


def test_forward_batch_of_one_equals_forward():
    cfg = I.TINY
    W = I.make_weights(cfg, seed=62)
    tok = I.make_tokens(cfg, 4, seed=62)
    m = B.Model(cfg, W)
    t = torch.from_numpy(tok).cuda()
    h, A, z = m.forward(t, 4)
    hb, Ab, zb = m.forward_batch(t.view(1, -1))
    torch.cuda.synchronize()
    assert _equal(h, hb[0]) and _equal(A, Ab[:, 0]) and _equal(z, zb[:, 0])
    m.close()


@pytest.mark.parametrize("batch,n_tok", [(3, 64), (2, 41), (4, 16)])
def test_tiny_fp32_batch_equals_each_sequence_alone(batch, n_tok):
    cfg = dataclasses.replace(I.TINY, n_layers=3)
    W = I.make_weights(cfg, seed=63, norm_jitter=0.1)
    tok = _tokens(cfg, n_tok, 63, batch)
    m = B.Model(cfg, W)
    t = torch.from_numpy(tok).cuda()
    outs = {}
    for sched in (B.SCHEDULE_DIAGONAL, B.SCHEDULE_SEQUENTIAL):
        outs[sched] = m.forward_batch(t, schedule=sched)
    torch.cuda.synchronize()
    hd, Ad, zd = outs[B.SCHEDULE_DIAGONAL]
    hs, As, zs = outs[B.SCHEDULE_SEQUENTIAL]
    assert _equal(hd, hs) and _equal(Ad, As) and _equal(zd, zs)
    n_seg = -(-n_tok // cfg.seg_len)
    for b in range(batch):
        h1, A1, z1 = m.forward_batch(t[b:b + 1].contiguous())
        torch.cuda.synchronize()
        assert _equal(h1[0], hd[b]) and _equal(A1[:, 0], Ad[:, b]) and _equal(z1[:, 0], zd[:, b]), b
        ho, Ao, zo = O.forward(cfg, W, tok[b], n_seg)
        assert_fp32_close(stats(hd[b].cpu().numpy(), ho), stats(Ad[:, b].cpu().numpy(), Ao),
                          stats(zd[:, b].cpu().numpy(), zo))
    m.armt_sync_status()
    m.close()


def test_tiny_batch_resume_from_state():
    cfg = I.TINY
    W = I.make_weights(cfg, seed=64, norm_jitter=0.1)
    tok = _tokens(cfg, 64 - 3, 64, 3)
    m = B.Model(cfg, W)
    t = torch.from_numpy(tok).cuda()
    h, A, z = m.forward_batch(t)
    S = cfg.seg_len
    ha, Aa, za = m.forward_batch(t[:, :2 * S].contiguous())
    hb, Ab, zb = m.forward_batch(t[:, 2 * S:].contiguous(), mem_A=Aa, mem_z=za)
    torch.cuda.synchronize()
    assert _equal(torch.cat([ha, hb], dim=1), h) and _equal(Ab, A) and _equal(zb, z)
    m.close()


def test_armt1b_shape_batch_with_short_last_segment():
    """ARMT-1B cell shape at reduced depth: a batch of 2 sequences of
    1024 + 300 tokens (the second segment is short), in the bf16 model.
    Each sequence matches the oracle under the derived bf16 bounds and equals
    its batch-1 run bitwise; diagonal == sequential bitwise."""
    cfg = dataclasses.replace(I.ARMT_1B, n_layers=2, vocab=4096)
    W = I.make_weights(cfg, 65, norm_jitter=0.1)
    n_tok = cfg.seg_len + 300
    tok = _tokens(cfg, n_tok, 65, 2)
    m = B.Model(cfg, B.device_weight_tensors(cfg, W))
    t = torch.from_numpy(tok).cuda()
    hd, Ad, zd = m.forward_batch(t)
    hs, As, zs = m.forward_batch(t, schedule=B.SCHEDULE_SEQUENTIAL)
    torch.cuda.synchronize()
    bitwise = _equal(hd, hs) and _equal(Ad, As) and _equal(zd, zs)
    alone = []
    for b in range(2):
        h1, A1, z1 = m.forward_batch(t[b:b + 1].contiguous())
        torch.cuda.synchronize()
        alone.append(_equal(h1[0], hd[b]) and _equal(A1[:, 0], Ad[:, b]) and _equal(z1[:, 0], zd[:, b]))
    m.armt_sync_status()
    gpu = [(hd[b].cpu().numpy(), Ad[:, b].cpu().numpy(), zd[:, b].cpu().numpy()) for b in range(2)]
    m.close()
    res = {"bitwise_diag_seq": bitwise, "batch_equals_alone": alone}
    ok_all = True
    for b in range(2):
        exact = O.forward(cfg, W, tok[b], 2)
        model = O.forward(cfg, W, tok[b], 2, operands="bf16")
        ok, g, ms = _derived_bounds_hold(gpu[b], exact, model, cfg.seg_len, 2)
        res[f"seq{b}"] = dict(gpu_vs_fp64=g, model_vs_fp64=ms)
        ok_all &= ok
    record("armt1b_shape_batch2_short", **res)
    assert bitwise and all(alone)
    assert ok_all, res


def test_armt1b_shape_batch8_pair_tiles_equal_each_sequence_alone():
    """A batch of 8 cells per layer (8 x 1040 rows) runs the weight GEMMs on
    CTA-pair tiles, a single sequence on single-CTA tiles: every sequence of
    the batch must still equal its batch-1 run bitwise (same per-element
    reduction order), in both schedules."""
    cfg = dataclasses.replace(I.ARMT_1B, n_layers=2, vocab=4096)
    W = I.make_weights(cfg, 66, norm_jitter=0.1)
    n_tok = cfg.seg_len + 100
    tok = _tokens(cfg, n_tok, 66, 8)
    m = B.Model(cfg, B.device_weight_tensors(cfg, W))
    t = torch.from_numpy(tok).cuda()
    hd, Ad, zd = m.forward_batch(t)
    hs, As, zs = m.forward_batch(t, schedule=B.SCHEDULE_SEQUENTIAL)
    torch.cuda.synchronize()
    assert _equal(hd, hs) and _equal(Ad, As) and _equal(zd, zs)
    for b in (0, 5, 7):
        h1, A1, z1 = m.forward_batch(t[b:b + 1].contiguous())
        torch.cuda.synchronize()
        assert _equal(h1[0], hd[b]) and _equal(A1[:, 0], Ad[:, b]) and _equal(z1[:, 0], zd[:, b]), b
    m.armt_sync_status()
    assert torch.isfinite(hd).all()
    m.close()
