"""The allocation-free chunk prefill entry point, called through the C ABI.

Some callers cannot call cudaMalloc when they run the prefill (a host that gives all device
memory to its own pool up front, or a loop that must not synchronise the device), so
gdn_chunk_prefill_noalloc keeps its scratch in a fixed array inside the library instead of a
caller workspace.  This test checks that two calls in a row give the same results as
gdn_chunk_prefill with a workspace, within the tolerances the other parity tests use, and that
a call too large for the fixed scratch is refused.  It lives in its own file, collected last.
"""
import ctypes

import pytest
import torch

import oracle
from linear_attention_ssm_gb300.synth import QWEN_GDN, Geometry, cu_seqlens_of, prefill_inputs
from tests.gpu_common import DEV, assert_out_close, assert_state_close, lib

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc_call(clib, geo, qkv, g, beta, cu, N, T, q_scale, state_in, state_out, z, norm_w, out):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return clib.gdn_chunk_prefill_noalloc(geo, _p(qkv), _p(g), _p(beta), _p(cu), N, T, q_scale, 1e-6,
                                          _p(state_in), _p(state_out), _p(z), _p(norm_w), 1e-6, _p(out), stream)


def test_noalloc_entry_point_matches_workspace_entry_point_twice():
    g = lib()
    from linear_attention_ssm_gb300 import binding
    clib = binding.load_library()
    geo = binding._geo(QWEN_GDN)
    for lengths, seed in (([100, 1, 64, 200], 41), ([65, 130, 7], 42)):   # two calls in a row
        inp = prefill_inputs(lengths, seed=seed)
        N, T = len(lengths), sum(lengths)
        cu = inp["cu_seqlens"].to(DEV)
        qkv = g.gdn_conv1d_prefill(inp["x"].to(DEV), inp["conv_w"].to(DEV), cu)
        gg, bb, z, nw = inp["g"].to(DEV), inp["beta"].to(DEV), inp["z"].to(DEV), inp["norm_w"].to(DEV)
        s0 = inp["state0"].to(DEV)
        st_ref = torch.empty_like(s0)
        out_ref = g.gdn_chunk_prefill(qkv, gg, bb, cu, inp["q_scale"], 1e-6, s0, st_ref, z, nw, 1e-6)
        st = torch.full_like(s0, float("nan"))
        out = torch.full((T, 48, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
        rc = _noalloc_call(clib, geo, qkv, gg, bb, cu, N, T, inp["q_scale"], s0, st, z, nw, out)
        assert rc == 0, clib.gdn_last_error_message().decode()
        g.gdn_check_device_errors()
        assert_out_close(out, out_ref.double())
        assert_state_close(st, st_ref.double())
        # and against the oracle itself, on the conv output both calls read
        ref = oracle.gdn_recurrence(qkv.cpu(), inp["g"], inp["beta"], inp["cu_seqlens"], 16, 48, 128, 128,
                                    inp["q_scale"], 1e-6, inp["state0"])
        assert_out_close(out, oracle.gated_rmsnorm(ref[0], inp["z"], inp["norm_w"], 1e-6))
        assert_state_close(st, ref[1])


def test_noalloc_at_the_scratch_limit():
    """16,384 sequences (the most the fixed scratch holds; beyond the longest-first sort, so the
    schedule keeps the given order), nearly all empty, on a small head geometry (1 K head, 2 V
    heads: 128 KB of state per sequence): the few real ones match the workspace entry point and
    the oracle, and the empty ones pass their states through."""
    g = lib()
    from linear_attention_ssm_gb300 import binding
    clib = binding.load_library()
    gq = Geometry(num_k_heads=1, num_v_heads=2)
    geo = binding._geo(gq)
    n = 16384
    real = {0: 70, 5000: 1, 9999: 130, 16383: 64}
    lengths = [real.get(i, 0) for i in range(n)]
    inp = prefill_inputs([real[k] for k in sorted(real)], seed=43, geo=gq)
    T = sum(lengths)
    cu = cu_seqlens_of(lengths).to(DEV)
    gen = torch.Generator(device=DEV).manual_seed(44)
    s0 = 0.1 * torch.randn((n, 2, 128, 128), generator=gen, device=DEV)
    for j, i in enumerate(sorted(real)):
        s0[i] = inp["state0"][j].to(DEV)
    qkv = g.gdn_conv1d_prefill(inp["x"].to(DEV), inp["conv_w"].to(DEV), inp["cu_seqlens"].to(DEV), geometry=gq)
    gg, bb, z, nw = inp["g"].to(DEV), inp["beta"].to(DEV), inp["z"].to(DEV), inp["norm_w"].to(DEV)
    st_ref = torch.empty_like(s0)
    out_ref = g.gdn_chunk_prefill(qkv, gg, bb, cu, inp["q_scale"], 1e-6, s0, st_ref, z, nw, 1e-6, geometry=gq)
    st = torch.full_like(s0, float("nan"))
    out = torch.full((T, 2, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    rc = _noalloc_call(clib, geo, qkv, gg, bb, cu, n, T, inp["q_scale"], s0, st, z, nw, out)
    assert rc == 0, clib.gdn_last_error_message().decode()
    g.gdn_check_device_errors()
    assert_out_close(out, out_ref.double())
    empty = torch.tensor([L == 0 for L in lengths], device=DEV)
    assert torch.equal(st[empty], s0[empty])
    ref = oracle.gdn_recurrence(qkv.cpu(), inp["g"], inp["beta"], inp["cu_seqlens"], 1, 2, 128, 128,
                                inp["q_scale"], 1e-6, inp["state0"])
    assert_out_close(out, oracle.gated_rmsnorm(ref[0], inp["z"], inp["norm_w"], 1e-6))
    for j, i in enumerate(sorted(real)):
        assert_state_close(st[i], ref[1][j], f"state of sequence {i}")
        assert_state_close(st[i], st_ref[i].double(), f"state of sequence {i} against the workspace call")


def test_noalloc_refuses_more_sequences_than_its_scratch_holds():
    g = lib()
    from linear_attention_ssm_gb300 import binding
    clib = binding.load_library()
    geo = binding._geo(QWEN_GDN)
    n = 16384 + 1
    cu = cu_seqlens_of([0] * n).to(DEV)
    buf = torch.zeros(64, dtype=torch.float32, device=DEV)
    rc = _noalloc_call(clib, geo, buf, buf, buf, cu, n, 0, 0.088, None, None, None, None, buf)
    assert rc == 1
    assert "scratch" in clib.gdn_last_error_message().decode()
    g.gdn_check_device_errors()
