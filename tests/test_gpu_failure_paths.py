"""Failure paths on the GPU, without faulting it.

Failures are made on the host side or with the library's test hooks, never by
a bad address, a trap or an endless wait:
  * ARMT_ALLOC_CAP_BYTES caps what a model may allocate: armt_create and the
    first batched call (which grows a second workspace) then return
    ARMT_ERR_OOM, and the model keeps working once the cap is lifted;
  * ARMT_TEST_STALL_AFTER makes the tensor-core kernels' copy producers stop
    after that many stage loads -- a stuck producer -- so the consumers'
    bounded waits (ARMT_WAIT_LIMIT_MS, shortened here) run out.  The kernels
    record the timeout, let the copies and MMAs they issued finish, free their
    tensor memory and return; the status call reports ARMT_ERR_TIMEOUT, and
    the next call without the hook gives the correct result.
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

ERR_OOM, ERR_TIMEOUT = 4, 6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_mod.build()
    B.load_library()


def _stall(monkeypatch, after):
    monkeypatch.setenv("ARMT_TEST_STALL_AFTER", str(after))
    monkeypatch.setenv("ARMT_WAIT_LIMIT_MS", "50")


def _unstall(monkeypatch):
    monkeypatch.delenv("ARMT_TEST_STALL_AFTER", raising=False)
    monkeypatch.delenv("ARMT_WAIT_LIMIT_MS", raising=False)


# ------------------------------------------------------------- allocation --

def test_allocation_cap_gives_oom_and_the_model_stays_usable(monkeypatch):
    cfg = I.TINY
    W = I.make_weights(cfg, seed=61, norm_jitter=0.1)
    monkeypatch.setenv("ARMT_ALLOC_CAP_BYTES", "4096")
    with pytest.raises(B.ArmtError) as e:
        B.Model(cfg, W)
    assert e.value.status == ERR_OOM
    monkeypatch.delenv("ARMT_ALLOC_CAP_BYTES")
    m = B.Model(cfg, W)
    tok = I.make_tokens(cfg, 3, seed=61)
    tok2 = np.stack([tok, np.roll(tok, 5)]).astype(np.int32)
    # the batched workspace is a separate pool: a 1-byte cap fails its first allocation
    monkeypatch.setenv("ARMT_ALLOC_CAP_BYTES", "1")
    with pytest.raises(B.ArmtError) as e:
        m.forward_batch(torch.from_numpy(tok2).cuda())
    assert e.value.status == ERR_OOM
    # batch 1 needs nothing new and still runs under the cap
    h1, A1, z1 = m.forward(torch.from_numpy(tok).cuda(), 3)
    monkeypatch.delenv("ARMT_ALLOC_CAP_BYTES")
    hb, Ab, zb = m.forward_batch(torch.from_numpy(tok2).cuda())
    torch.cuda.synchronize()
    m.armt_sync_status()
    assert torch.equal(hb[0], h1) and torch.equal(Ab[:, 0], A1) and torch.equal(zb[:, 0], z1)
    ho, Ao, zo = O.forward(cfg, W, tok2[1], 3)
    assert np.abs(hb[1].cpu().numpy() - ho).max() <= 1e-4
    m.close()


# ------------------------------------------------------------ timeouts --

# (G, M, N, K): a single-CTA tile shape and one that runs on CTA pairs
@pytest.mark.parametrize("G,M,N,K", [(2, 300, 768, 2048), (1, 2304, 1024, 1024)])
def test_grouped_gemm_stalled_producer_reports_timeout_then_recovers(monkeypatch, G, M, N, K):
    g = torch.Generator(device="cpu").manual_seed(M + N)
    A = torch.randn(G, M, K, generator=g).to(torch.bfloat16).cuda()
    Bm = torch.randn(G, N, K, generator=g).to(torch.bfloat16).cuda()
    C = torch.zeros(G, M, N, device="cuda")
    B.armt_block_sync_status()                      # nothing recorded before
    _stall(monkeypatch, 3)
    B.armt_grouped_gemm_bf16(A, Bm, C)
    with pytest.raises(B.ArmtError) as e:
        B.armt_block_sync_status()
    assert e.value.status == ERR_TIMEOUT
    B.armt_block_sync_status()                      # reported once, then clear
    _unstall(monkeypatch)
    C.fill_(float("nan"))
    B.armt_grouped_gemm_bf16(A, Bm, C)
    B.armt_block_sync_status()
    ref = torch.einsum("gmk,gnk->gmn", A.double().cpu(), Bm.double().cpu())
    err = (C.double().cpu() - ref).abs().max().item()
    assert err <= 1e-5 * K * 4, err


def _attention_inputs(G, T, Hq, Hkv, hd, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    qkv = torch.randn(G, T, (Hq + 2 * Hkv) * hd, generator=g).to(torch.bfloat16).cuda()
    qk = qkv[:, :, :(Hq + Hkv) * hd].contiguous()
    vt = qkv[:, :, (Hq + Hkv) * hd:].reshape(G, T, Hkv, hd).permute(0, 2, 3, 1).contiguous()
    return qkv, qk, vt


def test_segment_attention_stalled_producer_reports_timeout_then_recovers(monkeypatch):
    G, T, Hq, Hkv, hd = 2, 1040, 8, 2, 64
    qkv, qk, vt = _attention_inputs(G, T, Hq, Hkv, hd, seed=71)
    ref = torch.empty(G, T, Hq * hd, dtype=torch.bfloat16, device="cuda")
    B.armt_segment_attention_bf16(qk, vt, ref, Hq, Hkv)
    B.armt_block_sync_status()
    out = torch.zeros_like(ref)
    _stall(monkeypatch, 2)
    B.armt_segment_attention_bf16(qk, vt, out, Hq, Hkv)
    with pytest.raises(B.ArmtError) as e:
        B.armt_block_sync_status()
    assert e.value.status == ERR_TIMEOUT
    _unstall(monkeypatch)
    out.fill_(float("nan"))
    B.armt_segment_attention_bf16(qk, vt, out, Hq, Hkv)
    B.armt_block_sync_status()
    assert torch.equal(out, ref)


def test_model_forward_stalled_reports_timeout_then_recovers(monkeypatch):
    # one ARMT-1B-shaped layer, two segments: every tensor-core kernel of the
    # forward runs; once the first one times out the rest give up early
    cfg = dataclasses.replace(I.ARMT_1B, n_layers=1, vocab=4096)
    W = I.make_weights(cfg, seed=62)
    tok = torch.from_numpy(I.make_tokens(cfg, 2, seed=62)).cuda()
    m = B.Model(cfg, B.device_weight_tensors(cfg, W))
    h0, A0, z0 = m.forward(tok, 2)
    m.armt_sync_status()
    _stall(monkeypatch, 1)
    m.forward(tok, 2)
    with pytest.raises(B.ArmtError) as e:
        m.armt_sync_status()
    assert e.value.status == ERR_TIMEOUT
    _unstall(monkeypatch)
    h1, A1, z1 = m.forward(tok, 2)
    m.armt_sync_status()
    assert torch.equal(h1, h0) and torch.equal(A1, A0) and torch.equal(z1, z0)
    m.close()
