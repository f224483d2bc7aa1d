"""GPU parity of the multi-token verify and its commit against the oracle's verify transaction:
every row's output, the committed states for prefixes 0..K, untouched states after the verify,
stash rows past the committed prefix never read (poisoned), bad verdicts refused, and the
equivalence with K one-token decode steps."""
import pytest
import torch

import oracle
from linear_attention_ssm_gb300.synth import DECODE_BATCH, decode_inputs
from tests.gpu_common import DEV, STATE_TOL_F16, assert_out_close, assert_state_close, lib

pytestmark = pytest.mark.gpu
A = dict(num_k_heads=16, num_v_heads=48, head_k_dim=128, head_v_dim=128)
RECORD = 53440  # stash bytes per (sequence, row) at the 16 / 48 / 128 geometry


def _inputs(B, K, seed):
    d = decode_inputs(B, K, seed=seed)
    for k in ("x", "g", "beta", "z"):
        d[k] = d[k].transpose(0, 1).contiguous()  # [K, B, ...] -> [B, K, ...]
    return d


def _dev(d):
    return {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in d.items()}


def _verify(g, dd, cs, st):
    return g.gdn_verify(dd["x"], dd["conv_w"], cs, dd["g"], dd["beta"], st, dd["z"], dd["norm_w"], dd["q_scale"])


@pytest.mark.parametrize("B,K,committed", [(5, 6, [0, 1, 3, 6, 2]), (3, 17, [17, 9, 4]), (4, 1, [1, 0, 1, 1])],
                         ids=["k6", "k17", "k1"])
def test_verify_and_commit_match_oracle(B, K, committed):
    g = lib()
    d = _inputs(B, K, seed=50 + K)
    dd = _dev(d)
    cs, st = dd["conv_state0"].clone(), dd["state0"].clone()
    out, stash = _verify(g, dd, cs, st)
    g.gdn_check_device_errors()
    assert torch.equal(cs, dd["conv_state0"]) and torch.equal(st, dd["state0"])  # the verify reads only
    g.gdn_verify_commit(torch.tensor(committed, dtype=torch.int32, device=DEV), stash, cs, st, K)
    g.gdn_check_device_errors()
    ref, cs_ref, st_ref = oracle.verify(d["x"], d["conv_w"], d["conv_state0"], d["g"], d["beta"], d["state0"],
                                        d["z"], d["norm_w"], committed, q_scale=d["q_scale"], **A)
    out = out.cpu()
    for r in range(K):
        assert_out_close(out[:, r], ref[:, r], f"out of row {r}")
    for b in range(B):
        assert_state_close(st[b], st_ref[b], f"state of sequence {b} after committing {committed[b]} rows")
    assert torch.equal(cs.cpu().view(torch.int16), cs_ref.view(torch.int16))
    for b in range(B):
        if committed[b] == 0:
            assert torch.equal(st[b], dd["state0"][b])


def test_commit_never_reads_rows_past_the_prefix():
    """Stash records of rejected rows are poisoned (all bits set: NaN keys, deltas and gates); the
    commit gives the same bits as from the clean stash."""
    g = lib()
    B, K = 4, 8
    committed = [2, 8, 0, 5]
    d = _inputs(B, K, seed=60)
    dd = _dev(d)
    _, stash = _verify(g, dd, dd["conv_state0"], dd["state0"])
    poisoned = stash.clone()
    rec = stash.numel() // (B * K)
    assert rec == RECORD
    for b, m in enumerate(committed):
        poisoned[(b * K + m) * rec:(b + 1) * K * rec] = 0xFF
    cm = torch.tensor(committed, dtype=torch.int32, device=DEV)
    cs1, st1 = dd["conv_state0"].clone(), dd["state0"].clone()
    cs2, st2 = dd["conv_state0"].clone(), dd["state0"].clone()
    g.gdn_verify_commit(cm, stash, cs1, st1, K)
    g.gdn_verify_commit(cm, poisoned, cs2, st2, K)
    g.gdn_check_device_errors()
    assert torch.equal(st1, st2) and torch.equal(cs1, cs2)
    assert torch.isfinite(st2).all()


def test_verify_then_full_commit_equals_decode_steps():
    """K one-token decode steps and a K-row verify committed in full agree to fp32 rounding: the
    same conv arithmetic (the same bf16 conv outputs) and the same recurrence, the verify's in
    the WY form (another order of the same sums)."""
    g = lib()
    B, K = 3, 5
    d = _inputs(B, K, seed=61)
    dd = _dev(d)
    cs, st = dd["conv_state0"].clone(), dd["state0"].clone()
    outs = []
    for r in range(K):
        outs.append(g.gdn_decode_step(dd["x"][:, r].contiguous(), dd["conv_w"], cs, dd["g"][:, r].contiguous(),
                                      dd["beta"][:, r].contiguous(), st, dd["z"][:, r].contiguous(), dd["norm_w"],
                                      dd["q_scale"]))
    cs_v, st_v = dd["conv_state0"].clone(), dd["state0"].clone()
    out_v, stash = _verify(g, dd, cs_v, st_v)
    g.gdn_verify_commit(torch.full((B,), K, dtype=torch.int32, device=DEV), stash, cs_v, st_v, K)
    g.gdn_check_device_errors()
    dec = torch.stack(outs, 1)
    assert torch.equal(cs_v, cs)
    for b in range(B):
        assert_state_close(st_v[b], st[b].double(), f"state of sequence {b}", tol=1e-5)
        for r in range(K):
            assert_out_close(out_v[b, r], dec[b, r].double(), f"out of sequence {b}, row {r}")


def test_commit_refuses_a_verdict_out_of_range():
    g = lib()
    B, K = 2, 4
    d = _inputs(B, K, seed=62)
    dd = _dev(d)
    _, stash = _verify(g, dd, dd["conv_state0"], dd["state0"])
    g.gdn_check_device_errors()
    cs, st = dd["conv_state0"].clone(), dd["state0"].clone()
    g.gdn_verify_commit(torch.tensor([K + 1, -1], dtype=torch.int32, device=DEV), stash, cs, st, K)
    with pytest.raises(g.GdnError):
        g.gdn_check_device_errors()
    assert torch.equal(cs, dd["conv_state0"]) and torch.equal(st, dd["state0"])


def test_verify_256_sequences_8_rows_sampled():
    """The verify workload: 256 sequences x 8 rows, a seeded random verdict per sequence in 0..8;
    three sequences checked against the oracle (outputs of every row, committed states)."""
    g = lib()
    B, K = DECODE_BATCH, 8
    d = _inputs(B, K, seed=63)
    gen = torch.Generator().manual_seed(63)
    committed = torch.randint(0, K + 1, (B,), generator=gen, dtype=torch.int32)
    dd = _dev(d)
    cs, st = dd["conv_state0"].clone(), dd["state0"].clone()
    out, stash = _verify(g, dd, cs, st)
    g.gdn_verify_commit(committed.to(DEV), stash, cs, st, K)
    g.gdn_check_device_errors()
    out, cs, st = out.cpu(), cs.cpu(), st.cpu()
    assert torch.isfinite(out.float()).all() and torch.isfinite(st).all()
    sample = [0, 100, 255]
    ref, cs_ref, st_ref = oracle.verify(d["x"][sample], d["conv_w"], d["conv_state0"][sample], d["g"][sample],
                                        d["beta"][sample], d["state0"][sample], d["z"][sample], d["norm_w"],
                                        [int(committed[b]) for b in sample], q_scale=d["q_scale"], **A)
    for r in range(K):
        assert_out_close(out[sample, r], ref[:, r], f"out of row {r}")
    for i, b in enumerate(sample):
        assert_state_close(st[b], st_ref[i], f"state of sequence {b}")
    assert torch.equal(cs[sample].view(torch.int16), cs_ref.view(torch.int16))


# ------------------------------------------------------------------ binary16 state

def test_fp16_state_verify_and_commit_match_oracle():
    g = lib()
    B, K = 4, 6
    committed = [0, 2, 6, 5]
    d = _inputs(B, K, seed=64)
    dd = _dev(d)
    h0 = d["state0"].to(torch.float16)
    st = h0.to(DEV)
    cs = dd["conv_state0"].clone()
    out, stash = _verify(g, dd, cs, st)
    g.gdn_check_device_errors()
    assert torch.equal(st.cpu().view(torch.int16), h0.view(torch.int16))  # the verify reads only
    g.gdn_verify_commit(torch.tensor(committed, dtype=torch.int32, device=DEV), stash, cs, st, K)
    g.gdn_check_device_errors()
    ref, cs_ref, st_ref = oracle.verify_h16(d["x"], d["conv_w"], d["conv_state0"], d["g"], d["beta"], h0, d["z"],
                                            d["norm_w"], committed, q_scale=d["q_scale"], **A)
    out, st = out.cpu(), st.cpu()
    for r in range(K):
        assert_out_close(out[:, r], ref[:, r], f"out of row {r}")
    assert torch.equal(st[0].view(torch.int16), h0[0].view(torch.int16))  # aborted: the bits stand
    for b in range(1, B):
        # the same values rounded once on both sides: at most one rounding apart, rarely, where the
        # fp32 error of the terms (2^-20 of the state's scale bounds it) stays below the quantum
        want = st_ref[b].double()
        diff = (st[b].double() - want).abs()
        _, ex = torch.frexp(want.abs())
        quantum = torch.exp2(torch.clamp(ex - 11, min=-24).double())
        bound = quantum + 2.0 ** -20 * want.abs().max()
        bad = diff > bound
        worst = int(torch.argmax(diff - bound))
        assert not bad.any(), (f"sequence {b}: {int(bad.sum())} elements beyond one rounding; worst diff "
                               f"{diff.flatten()[worst]:.3g} at value {want.flatten()[worst]:.4g} (quantum "
                               f"{quantum.flatten()[worst]:.3g}); max diff {diff.max():.3g}, max |S| {want.abs().max():.3g}; "
                               f"{int((diff > 0).sum())} of {diff.numel()} differ")
        assert (diff > 0).double().mean().item() < 1e-2
    assert torch.equal(cs.cpu().view(torch.int16), cs_ref.view(torch.int16))


def test_fp16_state_verify_matches_decode_steps():
    """A committed fp16-state verify against K fp16-state decode steps: they round the state at
    different points (once, against after every row), so they agree within the binary16 chain
    tolerance."""
    g = lib()
    B, K = 3, 5
    d = _inputs(B, K, seed=65)
    dd = _dev(d)
    h0 = d["state0"].to(torch.float16).to(DEV)
    cs, st = dd["conv_state0"].clone(), h0.clone()
    outs = []
    for r in range(K):
        outs.append(g.gdn_decode_step_fp16_state(dd["x"][:, r].contiguous(), dd["conv_w"], cs,
                                                 dd["g"][:, r].contiguous(), dd["beta"][:, r].contiguous(), st,
                                                 dd["z"][:, r].contiguous(), dd["norm_w"], dd["q_scale"]))
    cs_v, st_v = dd["conv_state0"].clone(), h0.clone()
    out_v, stash = _verify(g, dd, cs_v, st_v)
    g.gdn_verify_commit(torch.full((B,), K, dtype=torch.int32, device=DEV), stash, cs_v, st_v, K)
    g.gdn_check_device_errors()
    dec = torch.stack(outs, 1)
    assert torch.equal(cs_v, cs)
    for b in range(B):
        assert_state_close(st_v[b].double(), st[b].double(), f"state of sequence {b}", tol=STATE_TOL_F16)
        for r in range(K):
            assert_out_close(out_v[b, r], dec[b, r].double(), f"out of sequence {b}, row {r}")


@pytest.mark.parametrize("hk,hv", [(4, 4), (2, 8)], ids=["ratio1", "ratio4"])
def test_verify_other_head_ratios(hk, hv):
    """V heads per K head 1 and 4 (the CTA owns 1 or 4 V heads' channels and state slices)."""
    from linear_attention_ssm_gb300.synth import Geometry
    g = lib()
    geo = Geometry(num_k_heads=hk, num_v_heads=hv)
    B, K = 3, 7
    committed = [7, 0, 3]
    d = decode_inputs(B, K, seed=66, geo=geo)
    for k in ("x", "g", "beta", "z"):
        d[k] = d[k].transpose(0, 1).contiguous()
    dd = _dev(d)
    cs, st = dd["conv_state0"].clone(), dd["state0"].clone()
    out, stash = g.gdn_verify(dd["x"], dd["conv_w"], cs, dd["g"], dd["beta"], st, dd["z"], dd["norm_w"],
                              dd["q_scale"], geometry=geo)
    g.gdn_verify_commit(torch.tensor(committed, dtype=torch.int32, device=DEV), stash, cs, st, K, geometry=geo)
    g.gdn_check_device_errors()
    a = dict(num_k_heads=hk, num_v_heads=hv, head_k_dim=128, head_v_dim=128)
    ref, cs_ref, st_ref = oracle.verify(d["x"], d["conv_w"], d["conv_state0"], d["g"], d["beta"], d["state0"],
                                        d["z"], d["norm_w"], committed, q_scale=d["q_scale"], **a)
    out = out.cpu()
    for r in range(K):
        assert_out_close(out[:, r], ref[:, r], f"out of row {r}")
    for b in range(B):
        assert_state_close(st[b], st_ref[b], f"state of sequence {b}")
    assert torch.equal(cs.cpu().view(torch.int16), cs_ref.view(torch.int16))


def test_fp16_state_verify_17_rows():
    """The longest verify (17 rows, the 48-column row bucket) with a binary16 state."""
    g = lib()
    B, K = 2, 17
    committed = [17, 11]
    d = _inputs(B, K, seed=67)
    dd = _dev(d)
    h0 = d["state0"].to(torch.float16)
    st, cs = h0.to(DEV), dd["conv_state0"].clone()
    out, stash = _verify(g, dd, cs, st)
    g.gdn_verify_commit(torch.tensor(committed, dtype=torch.int32, device=DEV), stash, cs, st, K)
    g.gdn_check_device_errors()
    ref, cs_ref, st_ref = oracle.verify_h16(d["x"], d["conv_w"], d["conv_state0"], d["g"], d["beta"], h0, d["z"],
                                            d["norm_w"], committed, q_scale=d["q_scale"], **A)
    out = out.cpu()
    for r in range(K):
        assert_out_close(out[:, r], ref[:, r], f"out of row {r}")
    for b in range(B):
        assert_state_close(st[b].cpu().double(), st_ref[b].double(), f"state of sequence {b}", tol=STATE_TOL_F16)
    assert torch.equal(cs.cpu().view(torch.int16), cs_ref.view(torch.int16))
