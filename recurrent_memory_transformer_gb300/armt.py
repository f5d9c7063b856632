"""ctypes binding of libarmt.so (include/armt.h), same entry-point names.

Argument marshalling only: every step of the forward pass runs in the
library's CUDA kernels.  PyTorch is used for device memory and streams.  If
the library has not been built, importing the binding raises; there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import numpy as np

from . import inputs as _inputs

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libarmt.so")

ARMT_OK = 0
STATUS_NAMES = {0: "ARMT_OK", 1: "ARMT_ERR_ARG", 2: "ARMT_ERR_SHAPE", 3: "ARMT_ERR_UNSUPPORTED",
                4: "ARMT_ERR_OOM", 5: "ARMT_ERR_CUDA", 6: "ARMT_ERR_TIMEOUT", 7: "ARMT_ERR_NO_DEVICE"}
ARMT_F32, ARMT_BF16 = 0, 1
PRECISION_BF16, PRECISION_BF16X2 = 0, 1
SCHEDULE_DIAGONAL, SCHEDULE_SEQUENTIAL, SCHEDULE_WAVEFRONT = 0, 1, 2
KERNEL_CLASSES = ("gemm_qkv", "gemm_o", "gemm_gateup", "gemm_down", "attention", "assoc_read",
                  "assoc_write", "norm", "other")

EXPORTED = ("armt_create", "armt_destroy", "armt_forward", "armt_forward_sequential",
            "armt_forward_batch", "armt_forward_host", "armt_grouped_gemm_bf16", "armt_segment_attention_bf16",
            "armt_segment_attention_bf16_noalloc", "armt_forward_full_attention", "armt_state_sizes",
            "armt_memory_bytes", "armt_lm_head", "armt_launch_count",
            "armt_set_profiling", "armt_set_profiling_mask", "armt_kernel_times", "armt_sync_status", "armt_status_string",
            "armt_last_error", "armt_block_sync_status", "armt_noalloc_sync_status", "armt_backward",
            "armt_backward_stats", "armt_set_tracing")


class ArmtError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {detail}")


class armt_config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("ffn_dim", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("seg_len", ctypes.c_int32),
                ("n_mem", ctypes.c_int32), ("key_dim", ctypes.c_int32),
                ("dpfp_nu", ctypes.c_int32), ("norm_eps", ctypes.c_float),
                ("assoc_eps", ctypes.c_float), ("rope_base", ctypes.c_double),
                ("dtype", ctypes.c_int32), ("precision", ctypes.c_int32)]


_WKEYS = ("embed", "mem", "wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "a_wq", "a_wk",
          "a_wv", "a_wbeta", "norm1", "norm2", "norm_f")


class armt_weights(ctypes.Structure):
    _fields_ = [(k, ctypes.c_void_p) for k in _WKEYS] + [("on_device", ctypes.c_int32)]


GRAD_KEYS = _WKEYS + ("mem_A", "mem_z")


class armt_grads(ctypes.Structure):
    _fields_ = [(k, ctypes.c_void_p) for k in GRAD_KEYS]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libarmt.so; raises FileNotFoundError when it was not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise FileNotFoundError(f"{path} not built: run python -m recurrent_memory_transformer_gb300.build")
    lib = ctypes.CDLL(path)
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    S = ctypes.c_int
    lib.armt_create.argtypes = [ctypes.POINTER(armt_config), ctypes.POINTER(armt_weights), P,
                                ctypes.POINTER(P)]
    lib.armt_destroy.argtypes = [P]
    for fn in (lib.armt_forward, lib.armt_forward_sequential):
        fn.argtypes = [P, P, I64, P, P, P, I32, P]
    lib.armt_forward_batch.argtypes = [P, P, I32, I64, P, P, P, I32, I32, P]
    lib.armt_forward_host.argtypes = [P, P, I64, P, P, P, I32, I32, P]
    lib.armt_forward_full_attention.argtypes = [P, P, I64, P, P]
    lib.armt_grouped_gemm_bf16.argtypes = [P, P, P, I32, I32, I32, I32, P]
    lib.armt_segment_attention_bf16.argtypes = [P, P, P, I32, I32, I32, I32, I32, P]
    lib.armt_segment_attention_bf16_noalloc.argtypes = [P, P, I32, I32, I32, I32, I32, P]
    lib.armt_state_sizes.argtypes = [P, ctypes.POINTER(I64), ctypes.POINTER(I64)]
    lib.armt_lm_head.argtypes = [P, P, I64, P, P, P]
    lib.armt_memory_bytes.argtypes = [P, ctypes.POINTER(I64), ctypes.POINTER(I64), ctypes.POINTER(I64)]
    lib.armt_launch_count.argtypes = [P, I64, I32, ctypes.POINTER(I64)]
    lib.armt_set_profiling.argtypes = [P, I32]
    lib.armt_set_tracing.argtypes = [P, I32]
    lib.armt_set_profiling_mask.argtypes = [P, ctypes.c_uint32]
    lib.armt_kernel_times.argtypes = [P, ctypes.POINTER(I64), ctypes.POINTER(ctypes.c_double), I32]
    lib.armt_sync_status.argtypes = [P, P]
    lib.armt_block_sync_status.argtypes = [P]
    lib.armt_noalloc_sync_status.argtypes = [P]
    lib.armt_backward.argtypes = [P, P, I64, P, P, P, P, P, P, P, P, ctypes.POINTER(armt_grads), P]
    lib.armt_backward_stats.argtypes = [P, ctypes.POINTER(I64), ctypes.POINTER(I64), ctypes.POINTER(ctypes.c_double)]
    for name in EXPORTED:
        getattr(lib, name).restype = S
    lib.armt_status_string.restype = ctypes.c_char_p
    lib.armt_status_string.argtypes = [S]
    lib.armt_last_error.restype = ctypes.c_char_p
    lib.armt_last_error.argtypes = []
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != ARMT_OK:
        detail = _lib.armt_last_error().decode(errors="replace")
        raise ArmtError(status, where, detail)


def make_config(cfg: "_inputs.ArmtConfig") -> armt_config:
    return armt_config(cfg.n_layers, cfg.d_model, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                       cfg.ffn_dim, cfg.vocab, cfg.seg_len, cfg.n_mem, cfg.key_dim, cfg.dpfp_nu,
                       cfg.norm_eps, cfg.assoc_eps, cfg.rope_base,
                       ARMT_BF16 if cfg.dtype == "bf16" else ARMT_F32,
                       PRECISION_BF16X2 if cfg.precision == "bf16x2" else PRECISION_BF16)


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _ptr(t) -> int:
    return t.data_ptr()


def host_weight_arrays(cfg, weights: Dict[str, np.ndarray]) -> Dict[str, np.ndarray]:
    """Contiguous host arrays in the model's element type (fp32, or bf16 bits as uint16)."""
    out = {}
    for k in _WKEYS:
        a = np.ascontiguousarray(weights[k], dtype=np.float32)
        out[k] = _inputs.bf16_bits(a) if cfg.dtype == "bf16" else a
    return out


def device_weight_tensors(cfg, weights: Dict[str, np.ndarray], device="cuda"):
    """Device tensors in the model's element type (exact: inputs are bf16-representable)."""
    import torch
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    return {k: torch.from_numpy(np.ascontiguousarray(weights[k], dtype=np.float32)).to(device).to(dt)
            for k in _WKEYS}


class Model:
    """Owns one armt_model; wraps the forward entry points."""

    def __init__(self, cfg, weights, stream=None):
        """`weights`: dict of numpy arrays (host path) or torch tensors on the device."""
        lib = load_library()
        self.cfg = cfg
        self._c = make_config(cfg)
        w = armt_weights()
        keep = []
        first = weights["embed"]
        on_device = hasattr(first, "is_cuda") and first.is_cuda
        if on_device:
            for k in _WKEYS:
                t = weights[k].contiguous()
                keep.append(t)
                setattr(w, k, t.data_ptr())
        else:
            arrs = host_weight_arrays(cfg, weights)
            for k in _WKEYS:
                keep.append(arrs[k])
                setattr(w, k, arrs[k].ctypes.data)
        w.on_device = 1 if on_device else 0
        h = ctypes.c_void_p()
        _check(lib.armt_create(ctypes.byref(self._c), ctypes.byref(w), _stream_ptr(stream),
                               ctypes.byref(h)), "armt_create")
        self._h = h
        a, z = ctypes.c_int64(), ctypes.c_int64()
        _check(lib.armt_state_sizes(h, ctypes.byref(a), ctypes.byref(z)), "armt_state_sizes")
        self.a_elems, self.z_elems = a.value, z.value

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _check(_lib.armt_destroy(self._h), "armt_destroy")
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def armt_forward(self, tokens, n_segments, hidden_out, mem_A, mem_z, mem_in_valid=0,
                     stream=None, schedule=SCHEDULE_DIAGONAL):
        fn = _lib.armt_forward if schedule == SCHEDULE_DIAGONAL else _lib.armt_forward_sequential
        _check(fn(self._h, _ptr(tokens), int(n_segments), _ptr(hidden_out), _ptr(mem_A),
                  _ptr(mem_z), int(mem_in_valid), _stream_ptr(stream)),
               "armt_forward" if schedule == SCHEDULE_DIAGONAL else "armt_forward_sequential")

    def armt_forward_sequential(self, tokens, n_segments, hidden_out, mem_A, mem_z, mem_in_valid=0,
                                stream=None):
        self.armt_forward(tokens, n_segments, hidden_out, mem_A, mem_z, mem_in_valid, stream,
                          SCHEDULE_SEQUENTIAL)

    def armt_forward_batch(self, tokens, hidden_out, mem_A, mem_z, mem_in_valid=0,
                           schedule=SCHEDULE_DIAGONAL, stream=None):
        """tokens int32 [B, N] (device), hidden fp32 [B, N, d], state [L, B, d, P] and [L, B, P]."""
        B_, N = tokens.shape
        _check(_lib.armt_forward_batch(self._h, _ptr(tokens), int(B_), int(N), _ptr(hidden_out),
                                       _ptr(mem_A), _ptr(mem_z), int(mem_in_valid), int(schedule),
                                       _stream_ptr(stream)), "armt_forward_batch")

    def forward_batch(self, tokens, schedule=SCHEDULE_DIAGONAL, mem_A=None, mem_z=None, stream=None):
        """Allocates outputs with torch; tokens int32 [B, N] on the device (N any
        positive count: a short last segment is allowed).  Returns (hidden
        [B, N, d], A [L, B, d, P], z [L, B, P])."""
        import torch
        dev = tokens.device
        B_, N = tokens.shape
        L, d, P = self.cfg.n_layers, self.cfg.d_model, self.cfg.phi_dim
        hidden = torch.empty((B_, N, d), dtype=torch.float32, device=dev)
        valid = mem_A is not None
        A = mem_A.clone() if valid else torch.empty((L, B_, d, P), dtype=torch.float32, device=dev)
        z = mem_z.clone() if valid else torch.empty((L, B_, P), dtype=torch.float32, device=dev)
        self.armt_forward_batch(tokens, hidden, A, z, 1 if valid else 0, schedule, stream)
        return hidden, A.view(L, B_, d, P), z.view(L, B_, P)

    def armt_forward_host(self, tokens: np.ndarray, n_segments, hidden_out: np.ndarray,
                          mem_A: np.ndarray, mem_z: np.ndarray, mem_in_valid=0,
                          schedule=SCHEDULE_DIAGONAL, stream=None):
        """Host-buffer forward (numpy arrays or pinned CPU tensors); synchronous."""
        def hp(x):
            return x.data_ptr() if hasattr(x, "data_ptr") else x.ctypes.data
        _check(_lib.armt_forward_host(self._h, hp(tokens), int(n_segments), hp(hidden_out),
                                      hp(mem_A), hp(mem_z), int(mem_in_valid), int(schedule),
                                      _stream_ptr(stream)), "armt_forward_host")

    def forward(self, tokens, n_segments, schedule=SCHEDULE_DIAGONAL, mem_A=None, mem_z=None,
                stream=None):
        """Allocates outputs with torch and runs one forward; returns (hidden, A, z)."""
        import torch
        dev = tokens.device
        hidden = torch.empty((n_segments * self.cfg.seg_len, self.cfg.d_model), dtype=torch.float32,
                             device=dev)
        valid = mem_A is not None
        A = mem_A.clone() if valid else torch.empty(self.a_elems, dtype=torch.float32, device=dev)
        z = mem_z.clone() if valid else torch.empty(self.z_elems, dtype=torch.float32, device=dev)
        self.armt_forward(tokens, n_segments, hidden, A, z, 1 if valid else 0, stream, schedule)
        L, d, P = self.cfg.n_layers, self.cfg.d_model, self.cfg.phi_dim
        return hidden, A.view(L, d, P), z.view(L, P)

    def armt_backward(self, tokens, grads, mem_A0=None, mem_z0=None, cot_hidden=None, cot_A=None,
                      cot_z=None, hidden_out=None, mem_A_out=None, mem_z_out=None, stream=None):
        """Device tensors (None where the header allows NULL); grads: dict of
        fp32 device tensors keyed like the weights (+ optional mem_A, mem_z)."""
        g = armt_grads()
        for k in GRAD_KEYS:
            t = grads.get(k)
            setattr(g, k, None if t is None else _ptr(t))

        def opt(t):
            return None if t is None else _ptr(t)
        _check(_lib.armt_backward(self._h, _ptr(tokens), int(tokens.numel()), opt(mem_A0), opt(mem_z0),
                                  opt(cot_hidden), opt(cot_A), opt(cot_z), opt(hidden_out), opt(mem_A_out),
                                  opt(mem_z_out), ctypes.byref(g), _stream_ptr(stream)), "armt_backward")

    def armt_backward_stats(self):
        """(kernel launches, algorithmic FLOPs) of the last backward, and its workspace bytes."""
        a, b, f = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_double()
        _check(_lib.armt_backward_stats(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(f)),
               "armt_backward_stats")
        return a.value, f.value, b.value

    def backward(self, tokens, cot_hidden=None, cot_A=None, cot_z=None, mem_A0=None, mem_z0=None,
                 state_grads=False, stream=None):
        """Allocates the gradients with torch; returns (grads dict, (hidden, A, z))."""
        import torch
        c, dev = self.cfg, tokens.device
        L, d, P = c.n_layers, c.d_model, c.phi_dim
        shapes = _inputs.weight_shapes(c)
        grads = {k: torch.empty(shapes[k], dtype=torch.float32, device=dev) for k in _WKEYS}
        if state_grads:
            grads["mem_A"] = torch.empty((L, d, P), dtype=torch.float32, device=dev)
            grads["mem_z"] = torch.empty((L, P), dtype=torch.float32, device=dev)
        hidden = torch.empty((tokens.numel(), d), dtype=torch.float32, device=dev)
        A = torch.empty((L, d, P), dtype=torch.float32, device=dev)
        z = torch.empty((L, P), dtype=torch.float32, device=dev)
        self.armt_backward(tokens, grads, mem_A0, mem_z0, cot_hidden, cot_A, cot_z, hidden, A, z, stream)
        return grads, (hidden, A, z)

    def armt_set_tracing(self, enable=True):
        """NVTX ranges around every step (forward diagonals or cells, backward diagonals)."""
        _check(_lib.armt_set_tracing(self._h, 1 if enable else 0), "armt_set_tracing")

    def armt_forward_full_attention(self, tokens, hidden_out, stream=None):
        """Plain causal LLaMA over all tokens (no memory), same weights."""
        _check(_lib.armt_forward_full_attention(self._h, _ptr(tokens), int(tokens.numel()),
                                                _ptr(hidden_out), _stream_ptr(stream)),
               "armt_forward_full_attention")

    def armt_lm_head(self, hidden, logits, w_head=None, stream=None):
        """logits fp32 [rows, vocab] = hidden fp32 [rows, d] @ head^T (head: w_head or the tied embedding)."""
        _check(_lib.armt_lm_head(self._h, _ptr(hidden), int(hidden.shape[0]),
                                 None if w_head is None else _ptr(w_head), _ptr(logits),
                                 _stream_ptr(stream)), "armt_lm_head")

    def armt_memory_bytes(self):
        """(weights, workspace, full_workspace): device bytes the library holds for this model."""
        w, ws, fw = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(_lib.armt_memory_bytes(self._h, ctypes.byref(w), ctypes.byref(ws), ctypes.byref(fw)),
               "armt_memory_bytes")
        return w.value, ws.value, fw.value

    def armt_launch_count(self, n_segments, schedule=SCHEDULE_DIAGONAL) -> int:
        n = ctypes.c_int64()
        _check(_lib.armt_launch_count(self._h, int(n_segments), int(schedule), ctypes.byref(n)),
               "armt_launch_count")
        return n.value

    def armt_set_profiling(self, enable: bool):
        _check(_lib.armt_set_profiling(self._h, 1 if enable else 0), "armt_set_profiling")

    def armt_set_profiling_mask(self, classes):
        """Time only the launches of the named kernel classes (KERNEL_CLASSES); [] turns it off."""
        mask = 0
        for c in classes:
            mask |= 1 << KERNEL_CLASSES.index(c)
        _check(_lib.armt_set_profiling_mask(self._h, mask), "armt_set_profiling_mask")

    def armt_kernel_times(self):
        n = len(KERNEL_CLASSES)
        launches = (ctypes.c_int64 * n)()
        ms = (ctypes.c_double * n)()
        _check(_lib.armt_kernel_times(self._h, launches, ms, n), "armt_kernel_times")
        return {KERNEL_CLASSES[i]: (launches[i], ms[i]) for i in range(n)}

    def armt_sync_status(self, stream=None):
        _check(_lib.armt_sync_status(self._h, _stream_ptr(stream)), "armt_sync_status")


def armt_grouped_gemm_bf16(A, B, C, stream=None):
    """C[g] = A[g] @ B[g]^T: A bf16 [G,M,K], B bf16 [G,N,K], C fp32 [G,M,N] (torch, cuda)."""
    lib = load_library()
    G, M, K = A.shape
    N = B.shape[1]
    _check(lib.armt_grouped_gemm_bf16(_ptr(A), _ptr(B), _ptr(C), G, M, N, K, _stream_ptr(stream)),
           "armt_grouped_gemm_bf16")


def armt_segment_attention_bf16(qk, vt, out, Hq, Hkv, stream=None):
    """Causal GQA per cell: qk bf16 [G,T,(Hq+Hkv)*hd], vt bf16 [G,Hkv,hd,T], out bf16 [G,T,Hq*hd]."""
    lib = load_library()
    G, T, _ = qk.shape
    hd = vt.shape[2]
    _check(lib.armt_segment_attention_bf16(_ptr(qk), _ptr(vt), _ptr(out), G, T, Hq, Hkv, hd,
                                           _stream_ptr(stream)), "armt_segment_attention_bf16")


def armt_segment_attention_bf16_noalloc(qkv, out, Hq, Hkv, hd, stream=None):
    """Same attention from the fused row layout qkv bf16 [G,T,(Hq+2Hkv)*hd]; allocates nothing."""
    lib = load_library()
    G, T, _ = qkv.shape
    _check(lib.armt_segment_attention_bf16_noalloc(_ptr(qkv), _ptr(out), G, T, Hq, Hkv, hd,
                                                   _stream_ptr(stream)),
           "armt_segment_attention_bf16_noalloc")


def armt_block_sync_status(stream=None):
    """Raises ArmtError(ARMT_ERR_TIMEOUT) if a building block's bounded wait gave up on this device."""
    lib = load_library()
    _check(lib.armt_block_sync_status(_stream_ptr(stream)), "armt_block_sync_status")


def armt_noalloc_sync_status(stream=None):
    """Raises ArmtError(ARMT_ERR_TIMEOUT) if the no-allocation attention's bounded wait gave up."""
    lib = load_library()
    _check(lib.armt_noalloc_sync_status(_stream_ptr(stream)), "armt_noalloc_sync_status")
