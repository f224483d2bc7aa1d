"""Shared helpers of the GPU parity tests: tolerances, guard (canary) buffers, comparisons."""
from __future__ import annotations

import pytest
import torch

# Tolerances of the GDN sublayer's GPU path against the fp64 oracle:
#   output:      max |got - want| <= 2e-2 * max |want|       (bf16 output)
#   final state: ||got - want||_2 <= 1e-4 * ||want||_2         (fp32 state)
#   conv output: within one bf16 ulp of the oracle's rounding of the exact value
OUT_TOL = 2e-2
STATE_TOL = 1e-4
NEG_CONTROL_RATIO = 10.0  # a planted fault must exceed the output bound by this factor
# A binary16-stored state chain against the oracle's binary16 chain.  The two round the same
# exact values, but the GPU computes them in fp32: wherever that puts a value on the other side
# of a rounding midpoint the stored states differ by one quantum, and the next steps turn such
# differences into further whole-quantum differences, so after a few steps the chains differ by
# a fraction of a quantum RMS.  One quantum is 2^-11..2^-10 of the value: bound 2^-10 rel. L2.
STATE_TOL_F16 = 2.0 ** -10

DEV = "cuda"


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def lib():
    need_gpu()
    import linear_attention_ssm_gb300 as g
    g.load_library()
    return g


@pytest.fixture(params=[0, 1, 2], ids=["split", "emulated", "fused"], name="mode")
def chunk_mode(request):
    """Runs a chunk-prefill test once per chunk design: the product library's split path (prep +
    state kernels), and in the test build (libgdn_test.so) the fused kernel with its MMAs emulated
    on the CUDA cores and the fused kernel on the tensor cores."""
    g = lib()
    if request.param == 0:  # the product library's own design
        yield 0
        return
    with g.using_test_library():  # the other designs exist only in the test build
        g.gdn_debug_set_chunk_mode(request.param)
        try:
            yield request.param
        finally:
            g.gdn_debug_set_chunk_mode(0)


def to_dev(t):
    return None if t is None else t.to(DEV).contiguous()


def out_error_ratio(got, want):
    """max |got - want| / (OUT_TOL * max |want|): <= 1 passes."""
    got = got.detach().double().cpu()
    want = want.detach().double().cpu()
    bound = OUT_TOL * want.abs().max().item()
    err = (got - want).abs().max().item()
    return err / bound if bound > 0 else (0.0 if err == 0 else float("inf"))


def assert_out_close(got, want, what="out"):
    r = out_error_ratio(got, want)
    assert torch.isfinite(got.detach().float()).all(), f"{what}: non-finite values"
    assert r <= 1.0, f"{what}: max error is {r:.3g}x the bound ({OUT_TOL} * absmax)"
    return r


def state_rel_l2(got, want):
    got = got.detach().double().cpu()
    want = want.detach().double().cpu()
    return ((got - want).norm() / want.norm().clamp_min(1e-300)).item()


def assert_state_close(got, want, what="state", tol=STATE_TOL):
    assert torch.isfinite(got.detach().float()).all(), f"{what}: non-finite values"
    r = state_rel_l2(got, want)
    assert r <= tol, f"{what}: relative L2 error {r:.3g} > {tol}"
    return r


def assert_bf16_within_one_ulp(got, want, abs_floor=0.0, what="conv"):
    """Every element within one bf16 ulp of the oracle's correctly rounded value, except where
    the value is so close to zero that the kernel's fp32 accumulation error (abs_floor, a scalar
    or a per-element tensor) exceeds one ulp; returns the fraction of bit-exact elements."""
    a = got.detach().cpu().view(torch.int16).int()
    b = want.detach().cpu().view(torch.int16).int()
    # same sign => adjacent patterns differ by one; +0/-0 treated as equal
    diff = (a - b).abs()
    zero_pair = ((a & 0x7FFF) == 0) & ((b & 0x7FFF) == 0)
    diff = torch.where(zero_pair, torch.zeros_like(diff), diff)
    absdiff = (got.detach().cpu().double() - want.double()).abs()
    bad = (diff > 1) & (absdiff > abs_floor)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements differ by more than one bf16 ulp and their floor"
    return float((diff == 0).float().mean())


def conv_accumulation_floor(x, w, cu_seqlens, conv_state=None):
    """Per-element absolute error allowance of the conv kernel near zero: 10 * 2^-24 * sum_i
    |w_i x_(t-3+i)| over the element's four taps (the history from conv_state, else zeros).

    The kernel sums four exact bf16 x bf16 products in fp32 (error at most 4 * 2^-24 times that
    magnitude sum); SiLU's slope is at most 1.1, so the pre-rounding output is off by at most
    E = 4.4 * 2^-24 * sum|w x|. Two correctly placed roundings differ by more than one bf16 ulp
    only when the values they round are more than one ulp apart, and then the rounded results are
    at most |error| + one ulp < 2E apart; 10 * 2^-24 covers 2E with room for the fp32 SiLU's own
    relative error, which is negligible at the magnitudes where this happens."""
    xa = x.detach().cpu().double().abs()
    wa = w.detach().cpu().double().abs()
    C, W = wa.shape
    H = W - 1
    cu = [int(v) for v in (cu_seqlens.tolist() if torch.is_tensor(cu_seqlens) else cu_seqlens)]
    mag = torch.zeros_like(xa)
    for n in range(len(cu) - 1):
        s, e = cu[n], cu[n + 1]
        if e == s:
            continue
        hist = (conv_state[n].detach().cpu().double().abs().t() if conv_state is not None
                else torch.zeros(H, C, dtype=torch.float64))
        pad = torch.cat([hist, xa[s:e]])
        for i in range(W):
            mag[s:e] += wa[:, i] * pad[i:i + e - s]
    return 10.0 * 2.0 ** -24 * mag


class Guarded:
    """A device tensor with poisoned guard regions on both sides, to catch out-of-range writes."""

    GUARD = 64  # elements on each side (keeps 16-byte alignment for 2- and 4-byte types)

    def __init__(self, shape, dtype, fill=None):
        n = 1
        for s in shape:
            n *= s
        self.n = n
        self.buf = torch.empty(n + 2 * self.GUARD, dtype=dtype, device=DEV)
        self.buf.view(torch.uint8).fill_(0x7F)
        self.t = self.buf[self.GUARD:self.GUARD + n].view(shape)
        if fill is not None:
            self.t.copy_(fill)
        self.pattern = self.buf[:self.GUARD].clone()

    def check(self, what="buffer"):
        assert torch.equal(self.buf[:self.GUARD].view(torch.uint8), self.pattern.view(torch.uint8)), \
            f"{what}: write below the buffer"
        assert torch.equal(self.buf[self.GUARD + self.n:].view(torch.uint8), self.pattern.view(torch.uint8)), \
            f"{what}: write above the buffer"
