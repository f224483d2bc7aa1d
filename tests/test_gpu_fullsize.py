"""Parity at the full benchmark sizes, in the launch configuration bench.py times: the prefill
sublayer (conv1d kernel, then the chunk kernel with the fused gate) on 4 x 4096 tokens and on
the varlen pack {1, 17, 63, 64, 65, 1000, 8191, 22334}, and 64 consecutive decode steps of 256
sequences.  The oracle computes a sample of V heads (prefill) or of sequences (decode); every
other element is checked for finiteness."""
import pytest
import torch

import oracle
from linear_attention_ssm_gb300.synth import (BATCHED_LENGTHS, VARLEN_LENGTHS, DECODE_BATCH, DECODE_STEPS,
                                              decode_inputs, prefill_inputs)
from tests.gpu_common import DEV, STATE_TOL_F16, assert_out_close, assert_state_close, lib

pytestmark = pytest.mark.gpu
SAMPLE_HEADS = [0, 1, 2, 25, 47]   # a whole K-head group plus heads of two other groups
A = dict(num_k_heads=16, num_v_heads=48, head_k_dim=128, head_v_dim=128)


def _prefill_case(lengths, seed):
    g = lib()
    inp = prefill_inputs(lengths, seed=seed)
    st = inp["state0"].to(DEV).clone()
    out = g.gdn_prefill(inp["x"].to(DEV), inp["conv_w"].to(DEV), inp["cu_seqlens"].to(DEV), inp["g"].to(DEV),
                        inp["beta"].to(DEV), inp["z"].to(DEV), inp["norm_w"].to(DEV), inp["q_scale"],
                        state_in=st, state_out=st)
    g.gdn_check_device_errors()
    out, st = out.cpu(), st.cpu()
    assert torch.isfinite(out.float()).all() and torch.isfinite(st).all()
    ref = oracle.prefill(inp["x"], inp["conv_w"], inp["cu_seqlens"], inp["g"], inp["beta"], inp["z"],
                         inp["norm_w"], q_scale=inp["q_scale"], state_in=inp["state0"], heads=SAMPLE_HEADS, **A)
    for h in SAMPLE_HEADS:
        assert_out_close(out[:, h], ref["out"][:, h], f"out, head {h}")
        for n in range(len(lengths)):
            assert_state_close(st[n, h], ref["state"][n, h], f"state, sequence {n}, head {h}")


def test_batched_prefill_4x4096():
    _prefill_case(BATCHED_LENGTHS, seed=2)


def test_varlen_prefill_31735_tokens():
    """The varlen workload's eight lengths sum to 31,735 tokens (the workload text says 32,735;
    the listed lengths decide)."""
    assert sum(VARLEN_LENGTHS) == 31735
    _prefill_case(VARLEN_LENGTHS, seed=3)


def test_decode_256_sequences_64_steps():
    g = lib()
    d = decode_inputs(DECODE_BATCH, DECODE_STEPS, seed=4)
    sample = [0, 77, 255]
    cs = d["conv_state0"].to(DEV).clone()
    st = d["state0"].to(DEV).clone()
    x, gg, bb, z = d["x"].to(DEV), d["g"].to(DEV), d["beta"].to(DEV), d["z"].to(DEV)
    w, nw = d["conv_w"].to(DEV), d["norm_w"].to(DEV)
    outs = torch.empty((DECODE_STEPS, DECODE_BATCH, 48, 128), dtype=torch.bfloat16, device=DEV)
    for s in range(DECODE_STEPS):
        g.gdn_decode_step(x[s], w, cs, gg[s], bb[s], st, z[s], nw, d["q_scale"], out=outs[s])
    g.gdn_check_device_errors()
    outs, st = outs.cpu(), st.cpu()
    assert torch.isfinite(outs.float()).all() and torch.isfinite(st).all()
    cs_ref = d["conv_state0"][sample]
    st_ref = d["state0"][sample].double()
    for s in range(DECODE_STEPS):
        ref, _, cs_ref, st_ref = oracle.decode_step(d["x"][s][sample], d["conv_w"], cs_ref, d["g"][s][sample],
                                                    d["beta"][s][sample], st_ref, d["z"][s][sample], d["norm_w"],
                                                    q_scale=d["q_scale"], **A)
        assert_out_close(outs[s][sample], ref, f"out of step {s}")
    assert_state_close(st[sample], st_ref, "state after 64 steps")
    assert torch.equal(cs.cpu()[sample].view(torch.int16), cs_ref.view(torch.int16))


def test_decode_256_sequences_64_steps_fp16_state():
    """The decode workload with the state stored as binary16, sampled sequences against the
    oracle's binary16 chain."""
    g = lib()
    d = decode_inputs(DECODE_BATCH, DECODE_STEPS, seed=4)
    sample = [0, 131, 255]
    cs = d["conv_state0"].to(DEV).clone()
    st = d["state0"].to(torch.float16).to(DEV)
    x, gg, bb, z = d["x"].to(DEV), d["g"].to(DEV), d["beta"].to(DEV), d["z"].to(DEV)
    w, nw = d["conv_w"].to(DEV), d["norm_w"].to(DEV)
    outs = torch.empty((DECODE_STEPS, DECODE_BATCH, 48, 128), dtype=torch.bfloat16, device=DEV)
    for s in range(DECODE_STEPS):
        g.gdn_decode_step_fp16_state(x[s], w, cs, gg[s], bb[s], st, z[s], nw, d["q_scale"], out=outs[s])
    g.gdn_check_device_errors()
    outs, st = outs.cpu(), st.cpu()
    assert torch.isfinite(outs.float()).all() and torch.isfinite(st.float()).all()
    cs_ref = d["conv_state0"][sample]
    st_ref = d["state0"][sample].to(torch.float16)
    for s in range(DECODE_STEPS):
        ref, _, cs_ref, st_ref = oracle.decode_step_h16(d["x"][s][sample], d["conv_w"], cs_ref, d["g"][s][sample],
                                                        d["beta"][s][sample], st_ref, d["z"][s][sample],
                                                        d["norm_w"], q_scale=d["q_scale"], **A)
        assert_out_close(outs[s][sample], ref, f"out of step {s}")
    assert_state_close(st[sample].double(), st_ref.double(), "state after 64 steps", tol=STATE_TOL_F16)
    assert torch.equal(cs.cpu()[sample].view(torch.int16), cs_ref.view(torch.int16))
