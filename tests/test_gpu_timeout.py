"""The timeout path of the bounded in-kernel waits, exercised without a GPU fault.

The test build of the library (libgdn_test.so) can drop one copy while still arming the mbarrier
that waits for it (gdn_debug_set_dropped_copy): the wait then runs out after a short limit, the
kernel raises the timeout bit of the device error word and returns with nothing in flight, and
gdn_check_device_errors reports GDN_ERR_TIMEOUT.  The next call, with the hook off, must be clean
and match the oracle.  Covered: the binary16-state decode step (its staged state slice) and the
split chunk prefill's state kernel (an item's first vector-block copy; tensor memory released on
the way out)."""
import pytest
import torch

import oracle
from linear_attention_ssm_gb300.synth import decode_inputs, prefill_inputs
from tests.gpu_common import DEV, assert_out_close, assert_state_close, lib, state_rel_l2, STATE_TOL_F16

pytestmark = pytest.mark.gpu
GDN_ERR_TIMEOUT = 5
A = dict(num_k_heads=16, num_v_heads=48, head_k_dim=128, head_v_dim=128)


def _expect_timeout(g):
    with pytest.raises(g.GdnError) as ei:
        g.gdn_check_device_errors()
    assert ei.value.status == GDN_ERR_TIMEOUT, ei.value


def test_decode_state_copy_dropped_times_out_then_recovers():
    g = lib()
    d = decode_inputs(4, 1, seed=400)
    h0 = d["state0"].to(torch.float16)
    args = lambda cs, sh: (d["x"][0].to(DEV), d["conv_w"].to(DEV), cs, d["g"][0].to(DEV), d["beta"][0].to(DEV), sh,
                           d["z"][0].to(DEV), d["norm_w"].to(DEV), d["q_scale"])
    with g.using_test_library():
        g.gdn_check_device_errors()  # starts clean
        g.gdn_debug_set_dropped_copy(1)
        try:
            g.gdn_decode_step_fp16_state(*args(d["conv_state0"].to(DEV), h0.to(DEV)))
            _expect_timeout(g)
        finally:
            g.gdn_debug_set_dropped_copy(0)
        sh, cs = h0.to(DEV), d["conv_state0"].to(DEV)
        out = g.gdn_decode_step_fp16_state(*args(cs, sh))
        g.gdn_check_device_errors()
    ref, _, _, ref_h = oracle.decode_step_h16(d["x"][0], d["conv_w"], d["conv_state0"], d["g"][0], d["beta"][0], h0,
                                              d["z"][0], d["norm_w"], q_scale=d["q_scale"], **A)
    assert_out_close(out, ref)
    assert state_rel_l2(sh.double(), ref_h.double()) <= STATE_TOL_F16


def test_chunk_state_kernel_copy_dropped_times_out_then_recovers():
    g = lib()
    inp = prefill_inputs([130, 64, 7], seed=401)
    ref = oracle.prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"], inp["g"], inp["beta"], inp["z"], inp["norm_w"],
                         16, 48, 128, 128, inp["q_scale"], state_in=inp["state0"])
    dv = {k: v.to(DEV) for k, v in inp.items() if torch.is_tensor(v)}
    y = ref["y"].to(DEV)

    def call():
        st = torch.empty_like(dv["state0"])
        out = g.gdn_chunk_prefill(y, dv["g"], dv["beta"], dv["cu_seqlens"], inp["q_scale"], 1e-6, dv["state0"], st,
                                  dv["z"], dv["norm_w"], 1e-6)
        return out, st
    with g.using_test_library():
        g.gdn_check_device_errors()
        g.gdn_debug_set_dropped_copy(2)
        try:
            call()
            _expect_timeout(g)
        finally:
            g.gdn_debug_set_dropped_copy(0)
        out, st = call()
        g.gdn_check_device_errors()
    assert_out_close(out, ref["out"])
    assert_state_close(st, ref["state"])
