"""Thin ctypes binding of libgdn.so: one Python function per C entry point, same names.

Argument marshalling only -- dtype/shape/device checks, output allocation when not supplied,
and the current torch stream.  Every step of the computation runs in the library's CUDA kernels;
there is no fallback of any kind: if ``libgdn.so`` is missing or cannot be loaded, every call
raises.

The verification hooks of ``include/gdn_debug.h`` live only in the test build of the library,
``libgdn_test.so``: the ``gdn_debug_*`` functions call into it, and inside
``with using_test_library():`` every other function does too (the tests use this to run the
same calls under the chunk designs the hooks select).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .synth import QWEN_GDN, Geometry

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn.so")
TEST_LIB_PATH = os.path.join(_HERE, "libgdn_test.so")

GDN_OK = 0
_lock = threading.Lock()
_lib = None
_test_lib = None
_override = None  # the test library while inside using_test_library()


class GdnError(RuntimeError):
    def __init__(self, status: int, name: str, message: str):
        super().__init__(f"{name}: {message}")
        self.status = status
        self.name = name


class _Geo(ctypes.Structure):
    _fields_ = [("num_k_heads", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
                ("head_k_dim", ctypes.c_int32), ("head_v_dim", ctypes.c_int32),
                ("conv_width", ctypes.c_int32)]


def _configure(lib, debug: bool):
    P, I, F, S = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    G = ctypes.POINTER(_Geo)
    sig = {
        "gdn_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "gdn_last_error_message": ([], ctypes.c_char_p),
        "gdn_version": ([], ctypes.c_char_p),
        "gdn_conv1d_prefill": ([G, P, P, P, I, I, P, P, P, P], ctypes.c_int),
        "gdn_chunk_prefill_workspace_size": ([G, I, I], S),
        "gdn_chunk_prefill_min_workspace_size": ([G, I, I], S),
        "gdn_chunk_prefill": ([G, P, P, P, P, I, I, F, F, P, P, P, P, F, P, P, S, P], ctypes.c_int),
        "gdn_chunk_prefill_noalloc": ([G, P, P, P, P, I, I, F, F, P, P, P, P, F, P, P], ctypes.c_int),
        "gdn_prefill": ([G, P, P, P, I, I, P, P, P, P, P, F, F, P, P, P, P, F, P, P, S, P], ctypes.c_int),
        "gdn_gated_rmsnorm": ([G, P, P, P, F, P, I, P], ctypes.c_int),
        "gdn_decode_step": ([G, P, P, P, P, P, P, P, P, F, F, F, P, I, P], ctypes.c_int),
        "gdn_decode_step_fp16_state": ([G, P, P, P, P, P, P, P, P, F, F, F, P, I, P], ctypes.c_int),
        "gdn_gates": ([G, P, P, P, P, P, P, I, P], ctypes.c_int),
        "gdn_chunk_prefill_fused_gates": ([G, P, P, P, P, P, P, I, I, F, F, P, P, P, P, F, P, P, S, P], ctypes.c_int),
        "gdn_decode_step_fused_gates": ([G, P, P, P, P, P, P, P, P, P, P, F, F, F, P, I, P], ctypes.c_int),
        "gdn_kda_decode_step": ([G, P, P, P, P, F, P, P, P, P, F, F, F, P, I, P], ctypes.c_int),
        "gdn_kda_recurrence": ([G, P, P, F, P, P, I, I, F, F, P, P, P, P, F, P, P], ctypes.c_int),
        "gdn_kda_chunk_prefill_workspace_size": ([G, I, I], S),
        "gdn_kda_chunk_prefill": ([G, P, P, F, P, P, I, I, F, F, P, P, P, P, F, P, P, S, P], ctypes.c_int),
        "gdn_kda_prefill": ([G, P, P, P, I, I, P, P, P, P, F, P, F, F, P, P, P, P, F, P, P, S, P], ctypes.c_int),
        "gdn_verify_stash_size": ([G, I, I], S),
        "gdn_verify": ([G, P, P, P, P, P, P, P, P, F, F, F, P, I, I, P, S, P], ctypes.c_int),
        "gdn_verify_commit": ([G, P, P, S, P, P, I, I, P], ctypes.c_int),
        "gdn_verify_fp16_state": ([G, P, P, P, P, P, P, P, P, F, F, F, P, I, I, P, S, P], ctypes.c_int),
        "gdn_verify_commit_fp16_state": ([G, P, P, S, P, P, I, I, P], ctypes.c_int),
        "gdn_check_device_errors": ([P], ctypes.c_int),
    }
    if debug:
        sig.update({
            "gdn_debug_set_chunk_mode": ([ctypes.c_int], ctypes.c_int),
            "gdn_debug_get_chunk_mode": ([], ctypes.c_int),
            "gdn_debug_mma_probe": ([P, P, ctypes.c_int, P, P, P], ctypes.c_int),
            "gdn_debug_mma_probe_ex": ([P, P, ctypes.c_int, ctypes.c_int, P, P, P], ctypes.c_int),
            "gdn_debug_set_dropped_copy": ([ctypes.c_uint], ctypes.c_int),
        })
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


def load_library():
    """Load libgdn.so (built by ``linear_attention_ssm_gb300.build``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m linear_attention_ssm_gb300.build` (needs nvcc)")
        _lib = _configure(ctypes.CDLL(LIB_PATH), debug=False)
        return _lib


def load_test_library():
    """Load libgdn_test.so, the build with the verification hooks of gdn_debug.h; raises if it is
    missing."""
    global _test_lib
    with _lock:
        if _test_lib is not None:
            return _test_lib
        if not os.path.exists(TEST_LIB_PATH):
            raise RuntimeError(f"{TEST_LIB_PATH} is missing: build it with "
                               "`python -m linear_attention_ssm_gb300.build` (needs nvcc)")
        _test_lib = _configure(ctypes.CDLL(TEST_LIB_PATH), debug=True)
        return _test_lib


class using_test_library:
    """Context manager: every binding call inside goes to libgdn_test.so (not thread-safe: for
    tests)."""

    def __enter__(self):
        global _override
        self._prev = _override
        _override = load_test_library()
        return _override

    def __exit__(self, *exc):
        global _override
        _override = self._prev
        return False


def _L():
    return _override if _override is not None else load_library()


def _check(status: int):
    if status != GDN_OK:
        lib = _L()
        name = lib.gdn_status_string(status).decode()
        msg = lib.gdn_last_error_message().decode()
        raise GdnError(status, name, msg)


def _geo(geo: Geometry):
    return ctypes.byref(_Geo(geo.num_k_heads, geo.num_v_heads, geo.head_k_dim, geo.head_v_dim,
                             geo.conv_width))


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t, dtype, name, shape=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def gdn_version() -> str:
    return _L().gdn_version().decode()


def gdn_status_string(status: int) -> str:
    return _L().gdn_status_string(int(status)).decode()


def gdn_last_error_message() -> str:
    """The library's message for the last error returned on this thread ("" if none)."""
    return _L().gdn_last_error_message().decode()


def gdn_conv1d_prefill(x, conv_w, cu_seqlens, conv_state_in=None, conv_state_out=None, y=None,
                       geometry: Geometry = QWEN_GDN, stream=None):
    """Causal depthwise conv1d + SiLU over packed sequences; returns y [T, C] bf16."""
    lib = _L()
    C, W = geometry.conv_dim, geometry.conv_width
    _dev(x, torch.bfloat16, "x")
    T = x.shape[0]
    N = cu_seqlens.numel() - 1
    _dev(x, torch.bfloat16, "x", (T, C))
    _dev(conv_w, torch.bfloat16, "conv_w", (C, W))
    _dev(cu_seqlens, torch.int32, "cu_seqlens", (N + 1,))
    _dev(conv_state_in, torch.bfloat16, "conv_state_in", (N, C, W - 1))
    _dev(conv_state_out, torch.bfloat16, "conv_state_out", (N, C, W - 1))
    if y is None:
        y = torch.empty((T, C), dtype=torch.bfloat16, device=x.device)
    _dev(y, torch.bfloat16, "y", (T, C))
    _check(lib.gdn_conv1d_prefill(_geo(geometry), _p(x), _p(conv_w), _p(cu_seqlens), N, T,
                                  _p(conv_state_in), _p(conv_state_out), _p(y), _stream(stream)))
    return y


def gdn_chunk_prefill_workspace_size(num_seqs: int, total_tokens: int,
                                     geometry: Geometry = QWEN_GDN) -> int:
    return int(_L().gdn_chunk_prefill_workspace_size(_geo(geometry), num_seqs, total_tokens))


def gdn_chunk_prefill_min_workspace_size(num_seqs: int, total_tokens: int,
                                         geometry: Geometry = QWEN_GDN) -> int:
    return int(_L().gdn_chunk_prefill_min_workspace_size(_geo(geometry), num_seqs, total_tokens))


def gdn_chunk_prefill(qkv, g, beta, cu_seqlens, q_scale, l2_eps=1e-6, state_in=None, state_out=None,
                      z=None, norm_w=None, rms_eps=1e-6, out=None, workspace=None,
                      geometry: Geometry = QWEN_GDN, stream=None):
    """Chunk-wise gated delta rule (optionally fused with the gated RMSNorm when z is given).

    Returns out [T, Hv, Dv] bf16 (o itself when z is None).  state_out, when given, receives the
    final fp32 states [N, Hv, Dv, Dk]; it may be state_in itself.
    """
    lib = _L()
    C, hv, dv, dk = geometry.conv_dim, geometry.num_v_heads, geometry.head_v_dim, geometry.head_k_dim
    N = cu_seqlens.numel() - 1
    T = qkv.shape[0]
    _dev(qkv, torch.bfloat16, "qkv", (T, C))
    _dev(g, torch.float32, "g", (T, hv))
    _dev(beta, torch.float32, "beta", (T, hv))
    _dev(cu_seqlens, torch.int32, "cu_seqlens", (N + 1,))
    _dev(state_in, torch.float32, "state_in", (N, hv, dv, dk))
    _dev(state_out, torch.float32, "state_out", (N, hv, dv, dk))
    _dev(z, torch.bfloat16, "z", (T, hv, dv))
    _dev(norm_w, torch.bfloat16, "norm_w", (dv,))
    if out is None:
        out = torch.empty((T, hv, dv), dtype=torch.bfloat16, device=qkv.device)
    _dev(out, torch.bfloat16, "out", (T, hv, dv))
    need = lib.gdn_chunk_prefill_workspace_size(_geo(geometry), N, T)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=qkv.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.gdn_chunk_prefill(_geo(geometry), _p(qkv), _p(g), _p(beta), _p(cu_seqlens), N, T,
                                 float(q_scale), float(l2_eps), _p(state_in), _p(state_out), _p(z),
                                 _p(norm_w), float(rms_eps), _p(out), _p(workspace), wbytes,
                                 _stream(stream)))
    return out


def gdn_chunk_prefill_noalloc(qkv, g, beta, cu_seqlens, q_scale, l2_eps=1e-6, state_in=None, state_out=None,
                              z=None, norm_w=None, rms_eps=1e-6, out=None, geometry: Geometry = QWEN_GDN,
                              stream=None):
    """gdn_chunk_prefill without a caller workspace: the schedule goes to a fixed scratch inside the
    library (at most GDN_NOALLOC_MAX_SEQS sequences per call; calls that overlap on the GPU race on
    it).  Same arguments and result as gdn_chunk_prefill otherwise."""
    lib = _L()
    C, hv, dv, dk = geometry.conv_dim, geometry.num_v_heads, geometry.head_v_dim, geometry.head_k_dim
    N = cu_seqlens.numel() - 1
    T = qkv.shape[0]
    _dev(qkv, torch.bfloat16, "qkv", (T, C))
    _dev(g, torch.float32, "g", (T, hv))
    _dev(beta, torch.float32, "beta", (T, hv))
    _dev(cu_seqlens, torch.int32, "cu_seqlens", (N + 1,))
    _dev(state_in, torch.float32, "state_in", (N, hv, dv, dk))
    _dev(state_out, torch.float32, "state_out", (N, hv, dv, dk))
    _dev(z, torch.bfloat16, "z", (T, hv, dv))
    _dev(norm_w, torch.bfloat16, "norm_w", (dv,))
    if out is None:
        out = torch.empty((T, hv, dv), dtype=torch.bfloat16, device=qkv.device)
    _dev(out, torch.bfloat16, "out", (T, hv, dv))
    _check(lib.gdn_chunk_prefill_noalloc(_geo(geometry), _p(qkv), _p(g), _p(beta), _p(cu_seqlens), N, T,
                                         float(q_scale), float(l2_eps), _p(state_in), _p(state_out), _p(z),
                                         _p(norm_w), float(rms_eps), _p(out), _stream(stream)))
    return out


def gdn_gated_rmsnorm(o, z, norm_w, eps=1e-6, out=None, geometry: Geometry = QWEN_GDN, stream=None):
    lib = _L()
    hv, dv = geometry.num_v_heads, geometry.head_v_dim
    T = o.shape[0]
    _dev(o, torch.bfloat16, "o", (T, hv, dv))
    _dev(z, torch.bfloat16, "z", (T, hv, dv))
    _dev(norm_w, torch.bfloat16, "norm_w", (dv,))
    if out is None:
        out = torch.empty_like(o)
    _dev(out, torch.bfloat16, "out", (T, hv, dv))
    _check(lib.gdn_gated_rmsnorm(_geo(geometry), _p(o), _p(z), _p(norm_w), float(eps), _p(out), T,
                                 _stream(stream)))
    return out


def gdn_decode_step(x, conv_w, conv_state, g, beta, state, z, norm_w, q_scale, l2_eps=1e-6,
                    rms_eps=1e-6, out=None, geometry: Geometry = QWEN_GDN, stream=None):
    """One fused decode step; conv_state and state are updated in place.  Returns out.

    ``state`` is fp32 (gdn_decode_step) or fp16 (gdn_decode_step_fp16_state: the state is half
    precision in memory, widened on load and rounded once on store).
    """
    lib = _L()
    fp16_state = state.dtype == torch.float16
    C, W = geometry.conv_dim, geometry.conv_width
    hv, dv, dk = geometry.num_v_heads, geometry.head_v_dim, geometry.head_k_dim
    B = x.shape[0]
    _dev(x, torch.bfloat16, "x", (B, C))
    _dev(conv_w, torch.bfloat16, "conv_w", (C, W))
    _dev(conv_state, torch.bfloat16, "conv_state", (B, C, W - 1))
    _dev(g, torch.float32, "g", (B, hv))
    _dev(beta, torch.float32, "beta", (B, hv))
    _dev(state, torch.float16 if fp16_state else torch.float32, "state", (B, hv, dv, dk))
    _dev(z, torch.bfloat16, "z", (B, hv, dv))
    _dev(norm_w, torch.bfloat16, "norm_w", (dv,))
    if out is None:
        out = torch.empty((B, hv, dv), dtype=torch.bfloat16, device=x.device)
    _dev(out, torch.bfloat16, "out", (B, hv, dv))
    fn = lib.gdn_decode_step_fp16_state if fp16_state else lib.gdn_decode_step
    _check(fn(_geo(geometry), _p(x), _p(conv_w), _p(conv_state), _p(g), _p(beta), _p(state), _p(z),
              _p(norm_w), float(q_scale), float(l2_eps), float(rms_eps), _p(out), B, _stream(stream)))
    return out


def gdn_kda_decode_step(x, conv_w, conv_state, g, beta, state, z, norm_w, q_scale, g_min=float("-inf"),
                        l2_eps=1e-6, rms_eps=1e-6, out=None, geometry: Geometry = QWEN_GDN, stream=None):
    """One KDA decode step (decay per key channel, g [B, Hv, Dk] fp32, clamped below at g_min);
    conv_state and state are updated in place.  Returns out."""
    lib = _L()
    C, W = geometry.conv_dim, geometry.conv_width
    hv, dv, dk = geometry.num_v_heads, geometry.head_v_dim, geometry.head_k_dim
    B = x.shape[0]
    _dev(x, torch.bfloat16, "x", (B, C))
    _dev(conv_w, torch.bfloat16, "conv_w", (C, W))
    _dev(conv_state, torch.bfloat16, "conv_state", (B, C, W - 1))
    _dev(g, torch.float32, "g", (B, hv, dk))
    _dev(beta, torch.float32, "beta", (B, hv))
    _dev(state, torch.float32, "state", (B, hv, dv, dk))
    _dev(z, torch.bfloat16, "z", (B, hv, dv))
    _dev(norm_w, torch.bfloat16, "norm_w", (dv,))
    if out is None:
        out = torch.empty((B, hv, dv), dtype=torch.bfloat16, device=x.device)
    _dev(out, torch.bfloat16, "out", (B, hv, dv))
    _check(lib.gdn_kda_decode_step(_geo(geometry), _p(x), _p(conv_w), _p(conv_state), _p(g), float(g_min), _p(beta),
                                   _p(state), _p(z), _p(norm_w), float(q_scale), float(l2_eps), float(rms_eps),
                                   _p(out), B, _stream(stream)))
    return out


def gdn_kda_recurrence(qkv, g, beta, cu_seqlens, q_scale, g_min=float("-inf"), l2_eps=1e-6, state_in=None,
                       state_out=None, z=None, norm_w=None, rms_eps=1e-6, out=None,
                       geometry: Geometry = QWEN_GDN, stream=None):
    """The KDA recurrence over packed sequences, token by token (g [T, Hv, Dk] fp32 per-channel log
    decay, clamped below at g_min), optionally fused with the gated RMSNorm when z is given.

    Returns out [T, Hv, Dv] bf16 (o itself when z is None).  state_out, when given, receives the
    final fp32 states [N, Hv, Dv, Dk]; it may be state_in itself.
    """
    lib = _L()
    C, hv, dv, dk = geometry.conv_dim, geometry.num_v_heads, geometry.head_v_dim, geometry.head_k_dim
    N = cu_seqlens.numel() - 1
    T = qkv.shape[0]
    _dev(qkv, torch.bfloat16, "qkv", (T, C))
    _dev(g, torch.float32, "g", (T, hv, dk))
    _dev(beta, torch.float32, "beta", (T, hv))
    _dev(cu_seqlens, torch.int32, "cu_seqlens", (N + 1,))
    _dev(state_in, torch.float32, "state_in", (N, hv, dv, dk))
    _dev(state_out, torch.float32, "state_out", (N, hv, dv, dk))
    _dev(z, torch.bfloat16, "z", (T, hv, dv))
    _dev(norm_w, torch.bfloat16, "norm_w", (dv,))
    if out is None:
        out = torch.empty((T, hv, dv), dtype=torch.bfloat16, device=qkv.device)
    _dev(out, torch.bfloat16, "out", (T, hv, dv))
    _check(lib.gdn_kda_recurrence(_geo(geometry), _p(qkv), _p(g), float(g_min), _p(beta), _p(cu_seqlens), N, T,
                                  float(q_scale), float(l2_eps), _p(state_in), _p(state_out), _p(z), _p(norm_w),
                                  float(rms_eps), _p(out), _stream(stream)))
    return out


def gdn_kda_chunk_prefill_workspace_size(num_seqs: int, total_tokens: int,
                                         geometry: Geometry = QWEN_GDN) -> int:
    return int(_L().gdn_kda_chunk_prefill_workspace_size(_geo(geometry), num_seqs, total_tokens))


def gdn_kda_chunk_prefill(qkv, g, beta, cu_seqlens, q_scale, g_min=float("-inf"), l2_eps=1e-6, state_in=None,
                          state_out=None, z=None, norm_w=None, rms_eps=1e-6, out=None, workspace=None,
                          geometry: Geometry = QWEN_GDN, stream=None):
    """gdn_kda_recurrence in its chunk-wise form (64-token chunks on the tensor cores): same
    arguments and result, plus a workspace of gdn_kda_chunk_prefill_workspace_size() bytes
    (allocated here when None).  After the clamp g must be finite."""
    lib = _L()
    C, hv, dv, dk = geometry.conv_dim, geometry.num_v_heads, geometry.head_v_dim, geometry.head_k_dim
    N = cu_seqlens.numel() - 1
    T = qkv.shape[0]
    _dev(qkv, torch.bfloat16, "qkv", (T, C))
    _dev(g, torch.float32, "g", (T, hv, dk))
    _dev(beta, torch.float32, "beta", (T, hv))
    _dev(cu_seqlens, torch.int32, "cu_seqlens", (N + 1,))
    _dev(state_in, torch.float32, "state_in", (N, hv, dv, dk))
    _dev(state_out, torch.float32, "state_out", (N, hv, dv, dk))
    _dev(z, torch.bfloat16, "z", (T, hv, dv))
    _dev(norm_w, torch.bfloat16, "norm_w", (dv,))
    if out is None:
        out = torch.empty((T, hv, dv), dtype=torch.bfloat16, device=qkv.device)
    _dev(out, torch.bfloat16, "out", (T, hv, dv))
    need = lib.gdn_kda_chunk_prefill_workspace_size(_geo(geometry), N, T)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=qkv.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.gdn_kda_chunk_prefill(_geo(geometry), _p(qkv), _p(g), float(g_min), _p(beta), _p(cu_seqlens), N, T,
                                     float(q_scale), float(l2_eps), _p(state_in), _p(state_out), _p(z), _p(norm_w),
                                     float(rms_eps), _p(out), _p(workspace), wbytes, _stream(stream)))
    return out


def gdn_decode_step_fp16_state(x, conv_w, conv_state, g, beta, state, z, norm_w, q_scale, l2_eps=1e-6,
                               rms_eps=1e-6, out=None, geometry: Geometry = QWEN_GDN, stream=None):
    """gdn_decode_step on an fp16 (binary16) recurrent state [B, Hv, Dv, Dk], updated in place."""
    if state.dtype != torch.float16:
        raise TypeError(f"state must be torch.float16, got {state.dtype}")
    return gdn_decode_step(x, conv_w, conv_state, g, beta, state, z, norm_w, q_scale, l2_eps, rms_eps, out,
                           geometry, stream)


def gdn_gates(a, b, A_log, dt_bias, g=None, beta=None, geometry: Geometry = QWEN_GDN, stream=None):
    """g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b) for every row and V head.

    a, b: [rows, Hv] bf16; A_log, dt_bias: [Hv] fp32.  Returns (g, beta), [rows, Hv] fp32.
    """
    lib = _L()
    hv = geometry.num_v_heads
    rows = a.shape[0]
    _dev(a, torch.bfloat16, "a", (rows, hv))
    _dev(b, torch.bfloat16, "b", (rows, hv))
    _dev(A_log, torch.float32, "A_log", (hv,))
    _dev(dt_bias, torch.float32, "dt_bias", (hv,))
    if g is None:
        g = torch.empty((rows, hv), dtype=torch.float32, device=a.device)
    if beta is None:
        beta = torch.empty((rows, hv), dtype=torch.float32, device=a.device)
    _dev(g, torch.float32, "g", (rows, hv))
    _dev(beta, torch.float32, "beta", (rows, hv))
    _check(lib.gdn_gates(_geo(geometry), _p(a), _p(b), _p(A_log), _p(dt_bias), _p(g), _p(beta), rows,
                         _stream(stream)))
    return g, beta


def gdn_chunk_prefill_fused_gates(qkv, a, b, A_log, dt_bias, cu_seqlens, q_scale, l2_eps=1e-6, state_in=None,
                                  state_out=None, z=None, norm_w=None, rms_eps=1e-6, out=None, workspace=None,
                                  geometry: Geometry = QWEN_GDN, stream=None):
    """gdn_chunk_prefill with the gates derived in the kernel from a, b ([T, Hv] bf16) and A_log,
    dt_bias ([Hv] fp32).  Returns out [T, Hv, Dv] bf16."""
    lib = _L()
    C, hv, dv, dk = geometry.conv_dim, geometry.num_v_heads, geometry.head_v_dim, geometry.head_k_dim
    N = cu_seqlens.numel() - 1
    T = qkv.shape[0]
    _dev(qkv, torch.bfloat16, "qkv", (T, C))
    _dev(a, torch.bfloat16, "a", (T, hv))
    _dev(b, torch.bfloat16, "b", (T, hv))
    _dev(A_log, torch.float32, "A_log", (hv,))
    _dev(dt_bias, torch.float32, "dt_bias", (hv,))
    _dev(cu_seqlens, torch.int32, "cu_seqlens", (N + 1,))
    _dev(state_in, torch.float32, "state_in", (N, hv, dv, dk))
    _dev(state_out, torch.float32, "state_out", (N, hv, dv, dk))
    _dev(z, torch.bfloat16, "z", (T, hv, dv))
    _dev(norm_w, torch.bfloat16, "norm_w", (dv,))
    if out is None:
        out = torch.empty((T, hv, dv), dtype=torch.bfloat16, device=qkv.device)
    _dev(out, torch.bfloat16, "out", (T, hv, dv))
    need = lib.gdn_chunk_prefill_workspace_size(_geo(geometry), N, T)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=qkv.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.gdn_chunk_prefill_fused_gates(_geo(geometry), _p(qkv), _p(a), _p(b), _p(A_log), _p(dt_bias),
                                             _p(cu_seqlens), N, T, float(q_scale), float(l2_eps), _p(state_in),
                                             _p(state_out), _p(z), _p(norm_w), float(rms_eps), _p(out),
                                             _p(workspace), wbytes, _stream(stream)))
    return out


def gdn_decode_step_fused_gates(x, conv_w, conv_state, a, b, A_log, dt_bias, state, z, norm_w, q_scale, l2_eps=1e-6,
                                rms_eps=1e-6, out=None, geometry: Geometry = QWEN_GDN, stream=None):
    """gdn_decode_step (fp32 state) with the gates derived in the kernel from a, b ([B, Hv] bf16) and
    A_log, dt_bias ([Hv] fp32); conv_state and state are updated in place.  Returns out."""
    lib = _L()
    C, W = geometry.conv_dim, geometry.conv_width
    hv, dv, dk = geometry.num_v_heads, geometry.head_v_dim, geometry.head_k_dim
    B = x.shape[0]
    _dev(x, torch.bfloat16, "x", (B, C))
    _dev(conv_w, torch.bfloat16, "conv_w", (C, W))
    _dev(conv_state, torch.bfloat16, "conv_state", (B, C, W - 1))
    _dev(a, torch.bfloat16, "a", (B, hv))
    _dev(b, torch.bfloat16, "b", (B, hv))
    _dev(A_log, torch.float32, "A_log", (hv,))
    _dev(dt_bias, torch.float32, "dt_bias", (hv,))
    _dev(state, torch.float32, "state", (B, hv, dv, dk))
    _dev(z, torch.bfloat16, "z", (B, hv, dv))
    _dev(norm_w, torch.bfloat16, "norm_w", (dv,))
    if out is None:
        out = torch.empty((B, hv, dv), dtype=torch.bfloat16, device=x.device)
    _dev(out, torch.bfloat16, "out", (B, hv, dv))
    _check(lib.gdn_decode_step_fused_gates(_geo(geometry), _p(x), _p(conv_w), _p(conv_state), _p(a), _p(b),
                                           _p(A_log), _p(dt_bias), _p(state), _p(z), _p(norm_w), float(q_scale),
                                           float(l2_eps), float(rms_eps), _p(out), B, _stream(stream)))
    return out


def gdn_verify_stash_size(batch: int, rows: int, geometry: Geometry = QWEN_GDN) -> int:
    return int(_L().gdn_verify_stash_size(_geo(geometry), int(batch), int(rows)))


def gdn_verify(x, conv_w, conv_state, g, beta, state, z, norm_w, q_scale, l2_eps=1e-6, rms_eps=1e-6,
               out=None, stash=None, geometry: Geometry = QWEN_GDN, stream=None):
    """Multi-token verify: rows = x.shape[1] tokens per sequence, states read only.

    ``state`` is fp32 (gdn_verify) or fp16 (gdn_verify_fp16_state).  Returns (out [B, K, Hv, Dv]
    bf16, stash uint8) -- pass the stash to gdn_verify_commit.
    """
    lib = _L()
    fp16_state = state.dtype == torch.float16
    C, W = geometry.conv_dim, geometry.conv_width
    hv, dv, dk = geometry.num_v_heads, geometry.head_v_dim, geometry.head_k_dim
    B, K = x.shape[0], x.shape[1]
    _dev(x, torch.bfloat16, "x", (B, K, C))
    _dev(conv_w, torch.bfloat16, "conv_w", (C, W))
    _dev(conv_state, torch.bfloat16, "conv_state", (B, C, W - 1))
    _dev(g, torch.float32, "g", (B, K, hv))
    _dev(beta, torch.float32, "beta", (B, K, hv))
    _dev(state, torch.float16 if fp16_state else torch.float32, "state", (B, hv, dv, dk))
    _dev(z, torch.bfloat16, "z", (B, K, hv, dv))
    _dev(norm_w, torch.bfloat16, "norm_w", (dv,))
    if out is None:
        out = torch.empty((B, K, hv, dv), dtype=torch.bfloat16, device=x.device)
    _dev(out, torch.bfloat16, "out", (B, K, hv, dv))
    need = gdn_verify_stash_size(B, K, geometry)
    if stash is None:
        stash = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _dev(stash, torch.uint8, "stash")
    fn = lib.gdn_verify_fp16_state if fp16_state else lib.gdn_verify
    _check(fn(_geo(geometry), _p(x), _p(conv_w), _p(conv_state), _p(g), _p(beta), _p(state), _p(z), _p(norm_w),
              float(q_scale), float(l2_eps), float(rms_eps), _p(out), B, K, _p(stash), stash.numel(),
              _stream(stream)))
    return out, stash


def gdn_verify_commit(committed_rows, stash, conv_state, state, rows: int, geometry: Geometry = QWEN_GDN,
                      stream=None):
    """Commit committed_rows[b] (device int32, 0..rows) rows of a verify into conv_state and state
    (fp32, or fp16: gdn_verify_commit_fp16_state)."""
    lib = _L()
    fp16_state = state.dtype == torch.float16
    C, W = geometry.conv_dim, geometry.conv_width
    hv, dv, dk = geometry.num_v_heads, geometry.head_v_dim, geometry.head_k_dim
    B = committed_rows.shape[0]
    _dev(committed_rows, torch.int32, "committed_rows", (B,))
    _dev(stash, torch.uint8, "stash")
    _dev(conv_state, torch.bfloat16, "conv_state", (B, C, W - 1))
    _dev(state, torch.float16 if fp16_state else torch.float32, "state", (B, hv, dv, dk))
    fn = lib.gdn_verify_commit_fp16_state if fp16_state else lib.gdn_verify_commit
    _check(fn(_geo(geometry), _p(committed_rows), _p(stash), stash.numel(), _p(conv_state), _p(state), B, int(rows),
              _stream(stream)))


def gdn_verify_fp16_state(x, conv_w, conv_state, g, beta, state, z, norm_w, q_scale, l2_eps=1e-6, rms_eps=1e-6,
                          out=None, stash=None, geometry: Geometry = QWEN_GDN, stream=None):
    """gdn_verify on a binary16 recurrent state [B, Hv, Dv, Dk] (read only)."""
    if state.dtype != torch.float16:
        raise TypeError(f"state must be torch.float16, got {state.dtype}")
    return gdn_verify(x, conv_w, conv_state, g, beta, state, z, norm_w, q_scale, l2_eps, rms_eps, out, stash,
                      geometry, stream)


def gdn_verify_commit_fp16_state(committed_rows, stash, conv_state, state, rows: int,
                                 geometry: Geometry = QWEN_GDN, stream=None):
    """gdn_verify_commit into a binary16 recurrent state (rounded once per committed element)."""
    if state.dtype != torch.float16:
        raise TypeError(f"state must be torch.float16, got {state.dtype}")
    return gdn_verify_commit(committed_rows, stash, conv_state, state, rows, geometry, stream)


def gdn_check_device_errors(stream=None):
    """Synchronise the stream and raise GdnError if a kernel flagged a device-side fault."""
    _check(_L().gdn_check_device_errors(_stream(stream)))


def _check_test(status: int):
    if status != GDN_OK:
        lib = load_test_library()
        raise GdnError(status, lib.gdn_status_string(status).decode(), lib.gdn_last_error_message().decode())


def gdn_debug_set_chunk_mode(mode: int):
    """Chunk design of later libgdn_test.so calls (0 default, 1 fused emulated, 2 fused)."""
    _check_test(load_test_library().gdn_debug_set_chunk_mode(int(mode)))


def gdn_debug_get_chunk_mode() -> int:
    return int(load_test_library().gdn_debug_get_chunk_mode())


def gdn_debug_set_dropped_copy(which: int):
    """libgdn_test.so only: bit 0 drops the binary16 decode step's state copy, bit 1 the chunk
    state kernel's first vector-block copy, so that the bounded wait on it runs out (0: off)."""
    _check_test(load_test_library().gdn_debug_set_dropped_copy(int(which)))


def gdn_debug_mma_probe(A, B, stream=None):
    """D = A @ B.T on one tcgen05 tile (A [128, 64], B [64 or 128, 64] bf16 CUDA tensors);
    libgdn_test.so."""
    lib = load_test_library()
    _dev(A, torch.bfloat16, "A", (128, 64))
    n = B.shape[0]
    _dev(B, torch.bfloat16, "B", (n, 64))
    D = torch.full((128, n), float("nan"), dtype=torch.float32, device=A.device)
    status = torch.zeros(1, dtype=torch.int32, device=A.device)
    _check_test(lib.gdn_debug_mma_probe(_p(A), _p(B), n, _p(D), _p(status), _stream(stream)))
    return D, status


def gdn_debug_mma_probe_ex(A, B, flags, stream=None):
    """As gdn_debug_mma_probe with flags: bit 0 A from tensor memory, bit 1 B MN-major."""
    lib = load_test_library()
    _dev(A, torch.bfloat16, "A", (128, 64))
    n = B.shape[0]
    _dev(B, torch.bfloat16, "B", (n, 64))
    D = torch.full((128, n), float("nan"), dtype=torch.float32, device=A.device)
    status = torch.zeros(1, dtype=torch.int32, device=A.device)
    _check_test(lib.gdn_debug_mma_probe_ex(_p(A), _p(B), n, int(flags), _p(D), _p(status), _stream(stream)))
    return D, status


def gdn_prefill(x, conv_w, cu_seqlens, g, beta, z, norm_w, q_scale, l2_eps=1e-6, rms_eps=1e-6,
                state_in=None, state_out=None, conv_state_in=None, conv_state_out=None,
                qkv_buf=None, out=None, workspace=None, geometry: Geometry = QWEN_GDN, stream=None):
    """The whole prefill sublayer in one call (gdn_prefill): the conv1d+SiLU stage into qkv_buf,
    then the chunk-wise gated delta rule with the gated RMSNorm fused (z, norm_w given) or not.
    Returns out [T, Hv, Dv] bf16."""
    lib = _L()
    C, W = geometry.conv_dim, geometry.conv_width
    hv, dv, dk = geometry.num_v_heads, geometry.head_v_dim, geometry.head_k_dim
    N = cu_seqlens.numel() - 1
    T = x.shape[0]
    _dev(x, torch.bfloat16, "x", (T, C))
    _dev(conv_w, torch.bfloat16, "conv_w", (C, W))
    _dev(cu_seqlens, torch.int32, "cu_seqlens", (N + 1,))
    _dev(conv_state_in, torch.bfloat16, "conv_state_in", (N, C, W - 1))
    _dev(conv_state_out, torch.bfloat16, "conv_state_out", (N, C, W - 1))
    _dev(g, torch.float32, "g", (T, hv))
    _dev(beta, torch.float32, "beta", (T, hv))
    _dev(state_in, torch.float32, "state_in", (N, hv, dv, dk))
    _dev(state_out, torch.float32, "state_out", (N, hv, dv, dk))
    _dev(z, torch.bfloat16, "z", (T, hv, dv))
    _dev(norm_w, torch.bfloat16, "norm_w", (dv,))
    if qkv_buf is None:
        qkv_buf = torch.empty((T, C), dtype=torch.bfloat16, device=x.device)
    _dev(qkv_buf, torch.bfloat16, "qkv_buf", (T, C))
    if out is None:
        out = torch.empty((T, hv, dv), dtype=torch.bfloat16, device=x.device)
    _dev(out, torch.bfloat16, "out", (T, hv, dv))
    need = lib.gdn_chunk_prefill_workspace_size(_geo(geometry), N, T)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.gdn_prefill(_geo(geometry), _p(x), _p(conv_w), _p(cu_seqlens), N, T, _p(conv_state_in),
                           _p(conv_state_out), _p(qkv_buf), _p(g), _p(beta), float(q_scale), float(l2_eps),
                           _p(state_in), _p(state_out), _p(z), _p(norm_w), float(rms_eps), _p(out), _p(workspace),
                           wbytes, _stream(stream)))
    return out


def gdn_kda_prefill(x, conv_w, cu_seqlens, g, beta, z, norm_w, q_scale, g_min=float("-inf"), l2_eps=1e-6,
                    rms_eps=1e-6, state_in=None, state_out=None, conv_state_in=None, conv_state_out=None,
                    qkv_buf=None, out=None, workspace=None, chunked=True, geometry: Geometry = QWEN_GDN,
                    stream=None):
    """The KDA prefill: conv1d, then the KDA recurrence with the gated RMSNorm fused -- in its
    chunk-wise form as one call (gdn_kda_prefill of the C ABI; `workspace` or one allocated here),
    or, with chunked=False, gdn_conv1d_prefill then the token-by-token gdn_kda_recurrence.  The
    conv output goes to `qkv_buf` (allocated when None).  Returns out [T, Hv, Dv] bf16."""
    if not chunked:
        qkv = gdn_conv1d_prefill(x, conv_w, cu_seqlens, conv_state_in, conv_state_out, qkv_buf,
                                 geometry=geometry, stream=stream)
        return gdn_kda_recurrence(qkv, g, beta, cu_seqlens, q_scale, g_min, l2_eps, state_in, state_out, z,
                                  norm_w, rms_eps, out, geometry=geometry, stream=stream)
    lib = _L()
    C, hv, dv, dk, W = (geometry.conv_dim, geometry.num_v_heads, geometry.head_v_dim, geometry.head_k_dim,
                        geometry.conv_width)
    N = cu_seqlens.numel() - 1
    T = x.shape[0]
    _dev(x, torch.bfloat16, "x", (T, C))
    _dev(conv_w, torch.bfloat16, "conv_w", (C, W))
    _dev(cu_seqlens, torch.int32, "cu_seqlens", (N + 1,))
    _dev(conv_state_in, torch.bfloat16, "conv_state_in", (N, C, W - 1))
    _dev(conv_state_out, torch.bfloat16, "conv_state_out", (N, C, W - 1))
    _dev(g, torch.float32, "g", (T, hv, dk))
    _dev(beta, torch.float32, "beta", (T, hv))
    _dev(state_in, torch.float32, "state_in", (N, hv, dv, dk))
    _dev(state_out, torch.float32, "state_out", (N, hv, dv, dk))
    _dev(z, torch.bfloat16, "z", (T, hv, dv))
    _dev(norm_w, torch.bfloat16, "norm_w", (dv,))
    if qkv_buf is None:
        qkv_buf = torch.empty((T, C), dtype=torch.bfloat16, device=x.device)
    _dev(qkv_buf, torch.bfloat16, "qkv_buf", (T, C))
    if out is None:
        out = torch.empty((T, hv, dv), dtype=torch.bfloat16, device=x.device)
    _dev(out, torch.bfloat16, "out", (T, hv, dv))
    need = lib.gdn_kda_chunk_prefill_workspace_size(_geo(geometry), N, T)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.gdn_kda_prefill(_geo(geometry), _p(x), _p(conv_w), _p(cu_seqlens), N, T, _p(conv_state_in),
                               _p(conv_state_out), _p(qkv_buf), _p(g), float(g_min), _p(beta), float(q_scale),
                               float(l2_eps), _p(state_in), _p(state_out), _p(z), _p(norm_w), float(rms_eps),
                               _p(out), _p(workspace), wbytes, _stream(stream)))
    return out
