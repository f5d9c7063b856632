"""The no-allocation attention entry point against the allocating one.

armt_segment_attention_bf16_noalloc serves callers that cannot allocate
device memory (an arena-owned or capped serving process, or a path that must
not trigger cudaMalloc's device-wide synchronisation).  It keeps its scratch
in a fixed file-scope device array.  This file is named so that pytest
collects it last; it passes on its own in a fresh process and after the
other tests.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from recurrent_memory_transformer_gb300 import armt as B  # noqa: E402
from recurrent_memory_transformer_gb300 import build as build_mod  # noqa: E402

TOL = 2e-2  # the attention tests' bound (bf16 probabilities and outputs)


def _inputs(G, T, Hq, Hkv, hd, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    qkv = torch.randn(G, T, (Hq + 2 * Hkv) * hd, generator=g).to(torch.bfloat16).cuda()
    qk = qkv[:, :, :(Hq + Hkv) * hd].contiguous()
    v = qkv[:, :, (Hq + Hkv) * hd:].reshape(G, T, Hkv, hd)
    vt = v.permute(0, 2, 3, 1).contiguous()
    return qkv, qk, vt


@pytest.mark.parametrize("shapes", [[(3, 1040, 8, 2, 64), (2, 264, 4, 4, 128)]])
def test_noalloc_attention_matches_allocating_entry_point_on_two_calls(shapes):
    build_mod.build()
    B.load_library()
    for call, (G, T, Hq, Hkv, hd) in enumerate(shapes):
        qkv, qk, vt = _inputs(G, T, Hq, Hkv, hd, seed=100 + call)
        ref = torch.empty(G, T, Hq * hd, dtype=torch.bfloat16, device="cuda")
        got = torch.full((G, T, Hq * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
        B.armt_segment_attention_bf16(qk, vt, ref, Hq, Hkv)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        B.armt_segment_attention_bf16_noalloc(qkv, got, Hq, Hkv, hd)
        torch.cuda.synchronize()
        if call > 0:  # after set-up on this device, a call takes no device memory
            assert torch.cuda.mem_get_info()[0] == free_before
        diff = (got.float() - ref.float()).abs().max().item()
        assert np.isfinite(got.float().cpu().numpy()).all()
        assert diff <= TOL, (call, diff)


def test_noalloc_rejects_problems_beyond_its_scratch():
    build_mod.build()
    B.load_library()
    # 64 cells * 8 kv heads * 128 dims * 1024 rows * 2 bytes = 128 MiB > 32 MiB
    qkv = torch.zeros(1, 8, 16, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1, 8, 16, dtype=torch.bfloat16, device="cuda")
    lib = B.load_library()
    st = lib.armt_segment_attention_bf16_noalloc(qkv.data_ptr(), out.data_ptr(), 64, 1024, 8, 8, 128,
                                                 None)
    assert st == 2  # ARMT_ERR_SHAPE, nothing enqueued
    assert b"exceeds the fixed scratch" in lib.armt_last_error()
