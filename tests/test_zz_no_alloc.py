"""The no-allocation attention entry point against the allocating one.

armt_segment_attention_bf16_noalloc serves callers that cannot allocate
device memory (an arena-owned or capped serving process, or a path that must
not trigger cudaMalloc's device-wide synchronisation).  It keeps its scratch
in a fixed file-scope device array.  It runs the same attention kernel on
the same operands as armt_segment_attention_bf16, so the two agree bitwise.
This file is named so that pytest collects it last; it passes on its own in
a fresh process and after the other tests.
"""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from recurrent_memory_transformer_gb300 import armt as B  # noqa: E402
from recurrent_memory_transformer_gb300 import build as build_mod  # noqa: E402

TOL = 2e-2  # the attention tests' bound against fp32 (bf16 probabilities and outputs)
ERR_TIMEOUT = 6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_mod.build()
    B.load_library()


def _inputs(G, T, Hq, Hkv, hd, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    qkv = torch.randn(G, T, (Hq + 2 * Hkv) * hd, generator=g).to(torch.bfloat16).cuda()
    qk = qkv[:, :, :(Hq + Hkv) * hd].contiguous()
    v = qkv[:, :, (Hq + Hkv) * hd:].reshape(G, T, Hkv, hd)
    vt = v.permute(0, 2, 3, 1).contiguous()
    return qkv, qk, vt


def _torch_fp32_attention(qkv, Hq, Hkv, hd):
    """Plain PyTorch fp32 causal GQA from the fused rows: [G, T, Hq*hd]."""
    G, T, _ = qkv.shape
    x = qkv.float()
    q = x[:, :, :Hq * hd].reshape(G, T, Hq, hd).transpose(1, 2)
    k = x[:, :, Hq * hd:(Hq + Hkv) * hd].reshape(G, T, Hkv, hd).transpose(1, 2)
    v = x[:, :, (Hq + Hkv) * hd:].reshape(G, T, Hkv, hd).transpose(1, 2)
    k = k.repeat_interleave(Hq // Hkv, dim=1)
    v = v.repeat_interleave(Hq // Hkv, dim=1)
    s = q @ k.transpose(-1, -2) / math.sqrt(hd)
    mask = torch.triu(torch.ones(T, T, dtype=torch.bool, device=qkv.device), diagonal=1)
    p = torch.softmax(s.masked_fill(mask, float("-inf")), dim=-1)
    return (p @ v).transpose(1, 2).reshape(G, T, Hq * hd)


@pytest.mark.parametrize("shapes", [[(3, 1040, 8, 2, 64), (2, 264, 4, 4, 128)]])
def test_noalloc_attention_matches_allocating_entry_point_on_two_calls(shapes):
    for call, (G, T, Hq, Hkv, hd) in enumerate(shapes):
        qkv, qk, vt = _inputs(G, T, Hq, Hkv, hd, seed=100 + call)
        ref = torch.empty(G, T, Hq * hd, dtype=torch.bfloat16, device="cuda")
        got = torch.full((G, T, Hq * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
        B.armt_segment_attention_bf16(qk, vt, ref, Hq, Hkv)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        B.armt_segment_attention_bf16_noalloc(qkv, got, Hq, Hkv, hd)
        B.armt_noalloc_sync_status()
        if call > 0:  # after set-up on this device, a call takes no device memory
            assert torch.cuda.mem_get_info()[0] == free_before
        assert torch.equal(got, ref), call


@pytest.mark.parametrize("G,T,Hq,Hkv,hd", [(1, 1037, 8, 2, 64), (2, 13, 2, 1, 128)])
def test_noalloc_attention_ragged_length_matches_fp32(G, T, Hq, Hkv, hd):
    # T not a multiple of 8: the values are padded to round_up(T, 8) with
    # zero columns inside the scratch (the allocating entry point rejects
    # such T); the padding rows never reach a real row, and the caller's
    # buffer is written only up to its G * T rows
    qkv, _, _ = _inputs(G, T, Hq, Hkv, hd, seed=T + hd)
    sentinel = 7.0
    buf = torch.full((G * T + 8, Hq * hd), sentinel, dtype=torch.bfloat16, device="cuda")
    B.armt_segment_attention_bf16_noalloc(qkv, buf, Hq, Hkv, hd)
    B.armt_noalloc_sync_status()
    got = buf[:G * T].reshape(G, T, Hq * hd).float()
    ref = _torch_fp32_attention(qkv, Hq, Hkv, hd)
    assert torch.isfinite(got).all()
    err = (got - ref).abs().max().item()
    assert err <= TOL, err
    assert torch.equal(buf[G * T:], torch.full_like(buf[G * T:], sentinel))


def test_noalloc_stalled_producer_reports_timeout_then_recovers(monkeypatch):
    G, T, Hq, Hkv, hd = 2, 520, 8, 2, 64
    qkv, qk, vt = _inputs(G, T, Hq, Hkv, hd, seed=300)
    ref = torch.empty(G, T, Hq * hd, dtype=torch.bfloat16, device="cuda")
    B.armt_segment_attention_bf16(qk, vt, ref, Hq, Hkv)
    B.armt_block_sync_status()
    out = torch.zeros_like(ref)
    monkeypatch.setenv("ARMT_TEST_STALL_AFTER", "2")
    monkeypatch.setenv("ARMT_WAIT_LIMIT_MS", "50")
    B.armt_segment_attention_bf16_noalloc(qkv, out, Hq, Hkv, hd)
    with pytest.raises(B.ArmtError) as e:
        B.armt_noalloc_sync_status()
    assert e.value.status == ERR_TIMEOUT
    B.armt_noalloc_sync_status()                    # reported once, then clear
    monkeypatch.delenv("ARMT_TEST_STALL_AFTER")
    monkeypatch.delenv("ARMT_WAIT_LIMIT_MS")
    for _ in range(2):
        out.fill_(float("nan"))
        B.armt_segment_attention_bf16_noalloc(qkv, out, Hq, Hkv, hd)
        B.armt_noalloc_sync_status()
        assert torch.equal(out, ref)


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 64 cells * 8 kv heads * 128 dims * 1024 rows * 2 bytes = 128 MiB > 32 MiB
    qkv = torch.zeros(1, 8, 16, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1, 8, 16, dtype=torch.bfloat16, device="cuda")
    lib = B.load_library()
    st = lib.armt_segment_attention_bf16_noalloc(qkv.data_ptr(), out.data_ptr(), 64, 1024, 8, 8, 128,
                                                 None)
    assert st == 2  # ARMT_ERR_SHAPE, nothing enqueued
    assert b"exceeds the fixed scratch" in lib.armt_last_error()
