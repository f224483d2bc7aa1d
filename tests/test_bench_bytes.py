"""The benchmark's algorithmic byte counts (the numerators of its roofline fractions) against the
sizes of the tensors each call reads and writes once, taken from the seeded input generators at
the workloads' geometries: a wrong constant in bench.py would move every reported fraction."""
import torch

import bench
from linear_attention_ssm_gb300.synth import KDA_GEO, QWEN_GDN, decode_inputs, kda_prefill_inputs, prefill_inputs


def _nbytes(*ts):
    return sum(t.numel() * t.element_size() for t in ts)


def _out(T, geo):  # the bf16 output rows [T, Hv, Dv]
    return T * geo.num_v_heads * geo.head_v_dim * 2


def test_chunk_prefill_bytes_are_its_tensors():
    lengths = [5, 0, 9]
    d = prefill_inputs(lengths, seed=1)
    T, N = sum(lengths), len(lengths)
    qkv = d["x"]  # the conv output has the input's shape and type
    want = _nbytes(qkv, d["g"], d["beta"], d["z"]) + _out(T, QWEN_GDN) + 2 * _nbytes(d["state0"])
    assert bench.CHUNK_BYTES_PER_TOKEN * T + bench.STATE_BYTES_PER_SEQ * N == want


def test_fused_prefill_pass_bytes_are_its_tensors():
    lengths = [7, 3]
    d = prefill_inputs(lengths, seed=2, random_conv_state=True)
    T, N = sum(lengths), len(lengths)
    want = (_nbytes(d["x"], d["g"], d["beta"], d["z"], d["conv_w"], d["norm_w"]) + _out(T, QWEN_GDN)
            + 2 * _nbytes(d["state0"], d["conv_state0"]))
    assert bench.step_bytes(T, N) == want


def test_conv_bytes_are_its_tensors():
    lengths = [4, 11]
    d = prefill_inputs(lengths, seed=3, random_conv_state=True)
    T, N = sum(lengths), len(lengths)
    want = 2 * _nbytes(d["x"]) + 2 * _nbytes(d["conv_state0"]) + _nbytes(d["conv_w"])
    assert T * 10240 * 2 * 2 + N * 10240 * 3 * 2 * 2 + 10240 * 4 * 2 == want


def test_decode_bytes_are_its_tensors():
    B = 5
    d = decode_inputs(B, 1, seed=4)
    want = (_nbytes(d["x"][0], d["g"][0], d["beta"][0], d["z"][0]) + B * QWEN_GDN.num_v_heads * 128 * 2
            + 2 * _nbytes(d["state0"], d["conv_state0"]))
    assert bench.DECODE_BYTES_PER_SEQ * B == want


def test_kda_prefill_bytes_are_its_tensors():
    lengths = [6, 10]
    d = kda_prefill_inputs(lengths, seed=5, geo=KDA_GEO)
    T, N = sum(lengths), len(lengths)
    assert KDA_GEO.num_k_heads == KDA_GEO.num_v_heads  # q, k and v each one 256-byte row per V head
    want = _nbytes(d["x"], d["g"], d["beta"], d["z"]) + _out(T, KDA_GEO) + 2 * _nbytes(d["state0"])
    assert bench.kda_prefill_bytes(T, N, KDA_GEO.num_v_heads) == want
    assert torch.equal(torch.tensor(d["g"].shape), torch.tensor([T, KDA_GEO.num_v_heads, KDA_GEO.head_k_dim]))
