"""Test-infrastructure oracle of the Gated DeltaNet sublayer (plain sequential fp64 C on the CPU).

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg import this
package.  It shares no code with the CUDA library in ``linear_attention_ssm_gb300``; both sides
only share the seeded input generators, which hold none of the method's arithmetic.

Every function takes CPU tensors (bf16 as ``torch.bfloat16``, fp32 as ``torch.float32``) and
returns float64 tensors.  The C source, ``gdn_oracle.c``, states what each step computes and the
page/section it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# mutation bits (negative controls planted in the oracle, never in the CUDA path)
MUT_SILU_GATE = 0x001
MUT_NO_CONV = 0x002
MUT_DROP_CARRY = 0x004
MUT_TRANSPOSE = 0x008
MUT_TILED_HEADS = 0x010
MUT_CONV_SHIFT = 0x020
MUT_DECAY_SIGN = 0x040
MUT_NO_BETA = 0x080
MUT_NO_QNORM = 0x100


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into liboracle.so beside it (gcc, -O2, no target-specific flags)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_round_bf16.argtypes = [D]
            lib.oracle_round_bf16.restype = ctypes.c_uint16
            lib.oracle_num_threads.restype = I
            lib.oracle_conv1d_prefill.argtypes = [I, I, I, P, P, P, I, P, P, P, P, I]
            lib.oracle_conv1d_prefill.restype = I
            lib.oracle_gdn_recurrence.argtypes = [
                I, I, I, I, I, P, P, P, P, I, D, D, P, P, P, P, I, I, I]
            lib.oracle_gdn_recurrence.restype = I
            lib.oracle_gated_rmsnorm.argtypes = [ctypes.c_long, I, P, P, P, D, P, I]
            lib.oracle_gated_rmsnorm.restype = I
            lib.oracle_decode_step.argtypes = [
                I, I, I, I, I, I, P, P, P, P, P, P, P, P, D, D, D, P, P, I, I]
            lib.oracle_decode_step.restype = I
            lib.oracle_round_f16.argtypes = [D]
            lib.oracle_round_f16.restype = ctypes.c_uint16
            lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_double.restype = D
            lib.oracle_decode_step_h16.argtypes = [
                I, I, I, I, I, I, P, P, P, P, P, P, P, P, D, D, D, P, P, I, I]
            lib.oracle_decode_step_h16.restype = I
            lib.oracle_gates.argtypes = [ctypes.c_long, I, P, P, P, P, P, P]
            lib.oracle_gates.restype = I
            lib.oracle_kda_decode_step.argtypes = [
                I, I, I, I, I, I, P, P, P, P, D, P, P, P, P, D, D, D, P, P, I]
            lib.oracle_kda_decode_step.restype = I
            lib.oracle_kda_recurrence.argtypes = [
                I, I, I, I, I, P, P, D, P, P, I, D, D, P, P, P, P, I, I, I]
            lib.oracle_kda_recurrence.restype = I
            _lib = lib
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _bf16_bits(t: torch.Tensor) -> torch.Tensor:
    assert t.dtype == torch.bfloat16, t.dtype
    return t.detach().cpu().contiguous().view(torch.int16)


def _f32(t):
    return None if t is None else t.detach().cpu().to(torch.float32).contiguous()


def _f64(t):
    return None if t is None else t.detach().cpu().to(torch.float64).contiguous()


def _i32(t):
    return torch.as_tensor(t, dtype=torch.int32).cpu().contiguous()


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def round_bf16(x: torch.Tensor) -> torch.Tensor:
    """Round float64 values to bf16 with ties to even, directly from the exact value."""
    lib = _load()
    flat = x.detach().cpu().to(torch.float64).reshape(-1).tolist()
    bits = np.array([lib.oracle_round_bf16(v) for v in flat], dtype=np.uint16)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).reshape(x.shape)


def round_f16(x: torch.Tensor) -> torch.Tensor:
    """Round float64 values to IEEE binary16 with ties to even; returns a torch.float16 tensor."""
    lib = _load()
    flat = x.detach().cpu().to(torch.float64).reshape(-1).tolist()
    bits = np.array([lib.oracle_round_f16(v) for v in flat], dtype=np.uint16)
    return torch.from_numpy(bits.view(np.int16)).view(torch.float16).reshape(x.shape)


def f16_to_double(h: torch.Tensor) -> torch.Tensor:
    """Widen binary16 values (torch.float16) to float64 by decoding their bit patterns."""
    lib = _load()
    assert h.dtype == torch.float16, h.dtype
    bits = h.detach().cpu().contiguous().view(torch.int16).reshape(-1).numpy().view(np.uint16)
    vals = [lib.oracle_f16_to_double(int(b)) for b in bits]
    return torch.tensor(vals, dtype=torch.float64).reshape(h.shape)


def gates(a, b, A_log, dt_bias):
    """g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b) per (token, V head); float64.

    Parity unpinned against the pages (they give no formula); the published Gated DeltaNet /
    Mamba-2 gate is the reading taken.  a, b: bf16 [T, Hv]; A_log, dt_bias: fp32 [Hv].
    """
    lib = _load()
    T, hv = a.shape
    ab, bb = _bf16_bits(a), _bf16_bits(b)
    al, db = _f32(A_log), _f32(dt_bias)
    g = torch.empty((T, hv), dtype=torch.float64)
    beta = torch.empty((T, hv), dtype=torch.float64)
    lib.oracle_gates(T, hv, _ptr(ab), _ptr(bb), _ptr(al), _ptr(db), _ptr(g), _ptr(beta))
    return g, beta


def conv1d_prefill(x, conv_w, cu_seqlens, conv_state_in=None, mutation: int = 0):
    """Causal depthwise conv1d + SiLU, rounded once to bf16.

    Returns (y bf16 [T,C], y_exact float64 [T,C], conv_state_out bf16 [N,C,W-1]).
    """
    lib = _load()
    T, C = x.shape
    W = conv_w.shape[1]
    cu = _i32(cu_seqlens)
    N = cu.numel() - 1
    xb, wb = _bf16_bits(x), _bf16_bits(conv_w)
    sin = _bf16_bits(conv_state_in) if conv_state_in is not None else None
    y = torch.empty((T, C), dtype=torch.int16)
    y_exact = torch.empty((T, C), dtype=torch.float64)
    sout = torch.empty((N, C, W - 1), dtype=torch.int16)
    rc = lib.oracle_conv1d_prefill(C, W, T, _ptr(xb), _ptr(wb), _ptr(cu), N, _ptr(sin), _ptr(y),
                                   _ptr(y_exact), _ptr(sout), int(mutation))
    if rc != 0:
        raise ValueError(f"oracle_conv1d_prefill failed ({rc})")
    return y.view(torch.bfloat16), y_exact, sout.view(torch.bfloat16)


def gdn_recurrence(qkv, g, beta, cu_seqlens, num_k_heads, num_v_heads, head_k_dim, head_v_dim,
                   q_scale, l2_eps=1e-6, state_in=None, heads=None, nthreads: int = 0,
                   mutation: int = 0):
    """The gated delta rule, token by token, one chain per (sequence, V head).

    qkv: bf16 [T, 2*Hk*Dk + Hv*Dv]; g, beta: [T, Hv]; state_in: [N, Hv, Dv, Dk] or None.
    Returns (o float64 [T, Hv, Dv], state_out float64 [N, Hv, Dv, Dk]).  With ``heads`` only
    those V heads are computed (the others are NaN).
    """
    lib = _load()
    T = qkv.shape[0]
    cu = _i32(cu_seqlens)
    N = cu.numel() - 1
    hk, hv, dk, dv = num_k_heads, num_v_heads, head_k_dim, head_v_dim
    assert qkv.shape[1] == 2 * hk * dk + hv * dv
    q = _bf16_bits(qkv)
    gg, bb = _f32(g), _f32(beta)
    sin = _f64(state_in)
    o = torch.full((T, hv, dv), float("nan"), dtype=torch.float64)
    sout = torch.full((N, hv, dv, dk), float("nan"), dtype=torch.float64)
    hl = _i32(heads) if heads is not None else None
    rc = lib.oracle_gdn_recurrence(hk, hv, dk, dv, T, _ptr(q), _ptr(gg), _ptr(bb), _ptr(cu), N,
                                   float(q_scale), float(l2_eps), _ptr(sin), _ptr(o), _ptr(sout),
                                   _ptr(hl), 0 if hl is None else hl.numel(), int(nthreads),
                                   int(mutation))
    if rc != 0:
        raise ValueError(f"oracle_gdn_recurrence failed ({rc})")
    return o, sout


def gated_rmsnorm(o, z, norm_w, eps=1e-6, mutation: int = 0):
    """out = o * (mean(o^2) + eps)^-1/2 * w * sigmoid(z) over the last dim; float64 result."""
    lib = _load()
    dv = o.shape[-1]
    oo = _f64(o).reshape(-1, dv)
    zz = _bf16_bits(z).reshape(-1, dv)
    ww = _bf16_bits(norm_w)
    out = torch.empty_like(oo)
    lib.oracle_gated_rmsnorm(oo.shape[0], dv, _ptr(oo), _ptr(zz), _ptr(ww), float(eps), _ptr(out),
                             int(mutation))
    return out.reshape(o.shape)


def decode_step(x, conv_w, conv_state, g, beta, state, z, norm_w, num_k_heads, num_v_heads,
                head_k_dim, head_v_dim, q_scale, l2_eps=1e-6, rms_eps=1e-6, nthreads: int = 0,
                mutation: int = 0):
    """One decode token per sequence.

    conv_state (bf16 [B,C,W-1]) and state (float64 [B,Hv,Dv,Dk]) are returned updated (new
    tensors; the arguments are not modified).  Returns (out float64 [B,Hv,Dv],
    o_raw float64 [B,Hv,Dv], conv_state', state').
    """
    lib = _load()
    B, C = x.shape
    W = conv_w.shape[1]
    hk, hv, dk, dv = num_k_heads, num_v_heads, head_k_dim, head_v_dim
    cs = _bf16_bits(conv_state).clone()
    st = _f64(state).clone()
    out = torch.empty((B, hv, dv), dtype=torch.float64)
    o_raw = torch.empty((B, hv, dv), dtype=torch.float64)
    # the converted inputs are held in locals: a temporary copy would be freed before the call
    xb, wb, gg, bb, zb, nb = (_bf16_bits(x), _bf16_bits(conv_w), _f32(g), _f32(beta), _bf16_bits(z),
                              _bf16_bits(norm_w))
    rc = lib.oracle_decode_step(hk, hv, dk, dv, W, B, _ptr(xb), _ptr(wb),
                                _ptr(cs), _ptr(gg), _ptr(bb), _ptr(st),
                                _ptr(zb), _ptr(nb), float(q_scale),
                                float(l2_eps), float(rms_eps), _ptr(out), _ptr(o_raw),
                                int(nthreads), int(mutation))
    if rc != 0:
        raise ValueError(f"oracle_decode_step failed ({rc})")
    return out, o_raw, cs.view(torch.bfloat16), st


def decode_step_h16(x, conv_w, conv_state, g, beta, state, z, norm_w, num_k_heads, num_v_heads,
                    head_k_dim, head_v_dim, q_scale, l2_eps=1e-6, rms_eps=1e-6, nthreads: int = 0,
                    mutation: int = 0):
    """decode_step with the recurrent state stored as binary16 (torch.float16 [B,Hv,Dv,Dk]).

    The state is widened exactly, the step runs in float64, the output comes from the new state
    before rounding and the new state is rounded once to binary16.  Returns (out, o_raw,
    conv_state', state' float16); the arguments are not modified.
    """
    lib = _load()
    assert state.dtype == torch.float16, state.dtype
    B, C = x.shape
    W = conv_w.shape[1]
    hk, hv, dk, dv = num_k_heads, num_v_heads, head_k_dim, head_v_dim
    cs = _bf16_bits(conv_state).clone()
    st = state.detach().cpu().contiguous().view(torch.int16).clone()
    out = torch.empty((B, hv, dv), dtype=torch.float64)
    o_raw = torch.empty((B, hv, dv), dtype=torch.float64)
    xb, wb, gg, bb, zb, nb = (_bf16_bits(x), _bf16_bits(conv_w), _f32(g), _f32(beta), _bf16_bits(z),
                              _bf16_bits(norm_w))
    rc = lib.oracle_decode_step_h16(hk, hv, dk, dv, W, B, _ptr(xb), _ptr(wb),
                                    _ptr(cs), _ptr(gg), _ptr(bb), _ptr(st),
                                    _ptr(zb), _ptr(nb), float(q_scale),
                                    float(l2_eps), float(rms_eps), _ptr(out), _ptr(o_raw),
                                    int(nthreads), int(mutation))
    if rc != 0:
        raise ValueError(f"oracle_decode_step_h16 failed ({rc})")
    return out, o_raw, cs.view(torch.bfloat16), st.view(torch.float16)


def kda_decode_step(x, conv_w, conv_state, g, beta, state, z, norm_w, num_k_heads, num_v_heads,
                    head_k_dim, head_v_dim, q_scale, g_min=float("-inf"), l2_eps=1e-6, rms_eps=1e-6,
                    mutation: int = 0):
    """One KDA decode token per sequence: the delta rule with a per-channel decay
    exp(max(g, g_min)), g [B, Hv, Dk] fp32.  Returns (out, o_raw, conv_state', state') like
    decode_step (new tensors; the arguments are not modified)."""
    lib = _load()
    B, C = x.shape
    W = conv_w.shape[1]
    hk, hv, dk, dv = num_k_heads, num_v_heads, head_k_dim, head_v_dim
    cs = _bf16_bits(conv_state).clone()
    st = _f64(state).clone()
    xb, wb, gg, bb, zb, nb = (_bf16_bits(x), _bf16_bits(conv_w), _f32(g), _f32(beta), _bf16_bits(z),
                              _bf16_bits(norm_w))
    out = torch.empty((B, hv, dv), dtype=torch.float64)
    o_raw = torch.empty((B, hv, dv), dtype=torch.float64)
    rc = lib.oracle_kda_decode_step(hk, hv, dk, dv, W, B, _ptr(xb), _ptr(wb), _ptr(cs), _ptr(gg),
                                    float(g_min), _ptr(bb), _ptr(st), _ptr(zb), _ptr(nb), float(q_scale),
                                    float(l2_eps), float(rms_eps), _ptr(out), _ptr(o_raw), int(mutation))
    if rc != 0:
        raise ValueError(f"oracle_kda_decode_step failed ({rc})")
    return out, o_raw, cs.view(torch.bfloat16), st


def verify(x, conv_w, conv_state, g, beta, state, z, norm_w, committed_rows, num_k_heads, num_v_heads,
           head_k_dim, head_v_dim, q_scale, l2_eps=1e-6, rms_eps=1e-6, nthreads: int = 0,
           mutation: int = 0):
    """A multi-token verify transaction: K rows per sequence, then commit of a prefix.

    x [B,K,C], g/beta [B,K,Hv], z [B,K,Hv,Dv]; committed_rows: B integers in [0, K].  The rows of
    every sequence are decoded in order from (conv_state, state), exactly as K one-token decode
    steps; the outputs of all K rows are returned, and each sequence's states become those after
    its first committed_rows[b] rows (0: the prior states, an abort).  Qwen3.8 kernel
    architecture and TDD ledger, "Transaction and width vocabulary" (commit publishes only the
    selected state; abort restores the prior state).  Returns (out float64 [B,K,Hv,Dv],
    conv_state' bf16, state' float64); the arguments are not modified.
    """
    B, K = x.shape[0], x.shape[1]
    m = [int(c) for c in committed_rows]
    if len(m) != B or any(c < 0 or c > K for c in m):
        raise ValueError("committed_rows must hold B values in [0, K]")
    a = dict(num_k_heads=num_k_heads, num_v_heads=num_v_heads, head_k_dim=head_k_dim,
             head_v_dim=head_v_dim, q_scale=q_scale, l2_eps=l2_eps, rms_eps=rms_eps,
             nthreads=nthreads, mutation=mutation)
    cs, st = conv_state, _f64(state)
    cs_out, st_out = conv_state.clone(), st.clone()
    outs = []
    for i in range(K):
        out, _, cs, st = decode_step(x[:, i], conv_w, cs, g[:, i], beta[:, i], st, z[:, i], norm_w, **a)
        outs.append(out)
        for b in range(B):
            if m[b] == i + 1:
                cs_out[b], st_out[b] = cs[b], st[b]
    return torch.stack(outs, 1), cs_out, st_out


def verify_h16(x, conv_w, conv_state, g, beta, state, z, norm_w, committed_rows, num_k_heads, num_v_heads,
               head_k_dim, head_v_dim, q_scale, l2_eps=1e-6, rms_eps=1e-6, nthreads: int = 0,
               mutation: int = 0):
    """verify with the recurrent state stored as binary16 (torch.float16 [B,Hv,Dv,Dk]).

    The state is widened exactly, the transaction runs in float64 (no state is stored between the
    rows, so none is rounded there), and each committed state is rounded once to binary16; a
    sequence with committed_rows 0 keeps its state's bits.  Returns (out float64, conv_state',
    state' float16).
    """
    assert state.dtype == torch.float16, state.dtype
    out, cs, st = verify(x, conv_w, conv_state, g, beta, f16_to_double(state), z, norm_w, committed_rows,
                         num_k_heads, num_v_heads, head_k_dim, head_v_dim, q_scale, l2_eps, rms_eps,
                         nthreads, mutation)
    st16 = state.detach().cpu().clone()
    for b, m in enumerate(committed_rows):
        if int(m) > 0:
            st16[b] = round_f16(st[b])
    return out, cs, st16


def prefill(x, conv_w, cu_seqlens, g, beta, z, norm_w, num_k_heads, num_v_heads, head_k_dim,
            head_v_dim, q_scale, l2_eps=1e-6, rms_eps=1e-6, state_in=None, conv_state_in=None,
            heads=None, nthreads: int = 0, mutation: int = 0):
    """The whole prefill sublayer: conv1d+SiLU -> recurrence -> gated RMSNorm.

    Returns a dict with y (bf16 conv output), o (float64), out (float64 gated output),
    state (float64 final states) and conv_state (bf16).
    """
    y, _, cs = conv1d_prefill(x, conv_w, cu_seqlens, conv_state_in, mutation=mutation)
    o, st = gdn_recurrence(y, g, beta, cu_seqlens, num_k_heads, num_v_heads, head_k_dim,
                           head_v_dim, q_scale, l2_eps, state_in, heads=heads, nthreads=nthreads,
                           mutation=mutation)
    out = gated_rmsnorm(o, z, norm_w, rms_eps, mutation=mutation)
    return {"y": y, "o": o, "out": out, "state": st, "conv_state": cs}


def kda_recurrence(qkv, g, beta, cu_seqlens, num_k_heads, num_v_heads, head_k_dim, head_v_dim,
                   q_scale, g_min=float("-inf"), l2_eps=1e-6, state_in=None, heads=None,
                   nthreads: int = 0, mutation: int = 0):
    """The KDA recurrence, token by token: gdn_recurrence with g [T, Hv, Dk] fp32, a log decay
    per key channel applied as exp(max(g, g_min)) to the state's key columns.  GLM-5.3-Flash
    kernel TDD ledger, slices I2 and I4.  Returns (o float64 [T, Hv, Dv], state_out float64
    [N, Hv, Dv, Dk])."""
    lib = _load()
    T = qkv.shape[0]
    cu = _i32(cu_seqlens)
    N = cu.numel() - 1
    hk, hv, dk, dv = num_k_heads, num_v_heads, head_k_dim, head_v_dim
    assert qkv.shape[1] == 2 * hk * dk + hv * dv
    assert tuple(g.shape) == (T, hv, dk), g.shape
    q = _bf16_bits(qkv)
    gg, bb = _f32(g), _f32(beta)
    sin = _f64(state_in)
    o = torch.full((T, hv, dv), float("nan"), dtype=torch.float64)
    sout = torch.full((N, hv, dv, dk), float("nan"), dtype=torch.float64)
    hl = _i32(heads) if heads is not None else None
    rc = lib.oracle_kda_recurrence(hk, hv, dk, dv, T, _ptr(q), _ptr(gg), float(g_min), _ptr(bb),
                                   _ptr(cu), N, float(q_scale), float(l2_eps), _ptr(sin), _ptr(o),
                                   _ptr(sout), _ptr(hl), 0 if hl is None else hl.numel(),
                                   int(nthreads), int(mutation))
    if rc != 0:
        raise ValueError(f"oracle_kda_recurrence failed ({rc})")
    return o, sout


def kda_prefill(x, conv_w, cu_seqlens, g, beta, z, norm_w, num_k_heads, num_v_heads, head_k_dim,
                head_v_dim, q_scale, g_min=float("-inf"), l2_eps=1e-6, rms_eps=1e-6, state_in=None,
                conv_state_in=None, heads=None, nthreads: int = 0, mutation: int = 0):
    """The KDA prefill: conv1d+SiLU -> KDA recurrence -> gated RMSNorm (the output gate of the
    GDN sublayer).  Returns the same dict as prefill."""
    y, _, cs = conv1d_prefill(x, conv_w, cu_seqlens, conv_state_in, mutation=mutation)
    o, st = kda_recurrence(y, g, beta, cu_seqlens, num_k_heads, num_v_heads, head_k_dim,
                           head_v_dim, q_scale, g_min, l2_eps, state_in, heads=heads,
                           nthreads=nthreads, mutation=mutation)
    out = gated_rmsnorm(o, z, norm_w, rms_eps, mutation=mutation)
    return {"y": y, "o": o, "out": out, "state": st, "conv_state": cs}
