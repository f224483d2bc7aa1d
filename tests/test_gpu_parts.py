"""GPU tests of the chunk prefill's intra-sequence parallelism: a sequence much longer than its
share of the GPU is cut into parts that run at once.  Each part after the first starts from
S_p = S_(p-1) Phi_(p-1) + L_(p-1), with L the previous part's end state from a zero start and Phi
its transition, both computed beside the previous segment.  The recurrence is the Gated DeltaNet
sublayer's (pegainfer PR #1152, Summary and Code review); outputs and final states are compared
with the fp64 oracle on every head.  The plan the library chose is read back from the caller's
workspace, so the tests know the split really happened."""
import pytest
import torch

from linear_attention_ssm_gb300.synth import Geometry, prefill_inputs
from tests.gpu_common import DEV, assert_out_close, assert_state_close, lib
from tests.test_gpu_chunk import run_oracle

pytestmark = pytest.mark.gpu
GEO = Geometry(num_k_heads=2, num_v_heads=6)
# 55 chunks, 2, 57, 0 and 22 chunks: the share of one CTA slot is 8 chunks here, a sequence splits
# when a segment of it holds more than 16, into ceil(m / 8) parts: 3 for the first and the third
LENGTHS = [3500, 100, 3600, 0, 1351]
PARTS = [3, 1, 3, 1, 1]


def _pad(b):
    return -(-b // 256) * 256


def _parts_read_back(ws, n):
    """The per-sequence part counts the library wrote into the workspace (after the counters,
    the order, the chunk offsets and four per-segment prefixes)."""
    off = 256 + _pad(4 * n) + _pad(4 * (n + 1)) + _pad(16 * (n + 1))
    return ws[off:off + 4 * n].view(torch.int32).cpu().tolist()


def _dev(inp):
    return {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in inp.items()}


def _run(g, d, y, state_in, state_out, ws, out=None, stream=None):
    return g.gdn_chunk_prefill(y, d["g"], d["beta"], d["cu_seqlens"], d["q_scale"], 1e-6, state_in, state_out,
                               d["z"], d["norm_w"], 1e-6, out, workspace=ws, geometry=GEO, stream=stream)


def _check(out, st, ref, what):
    assert_out_close(out, ref["out"], f"{what}: out")
    for n in range(len(LENGTHS)):
        for h in range(GEO.num_v_heads):
            assert_state_close(st[n, h], ref["state"][n, h], f"{what}: state of sequence {n}, head {h}")


@pytest.mark.parametrize("in_place", [False, True], ids=["out_of_place", "in_place"])
def test_split_sequences_match_the_oracle(in_place):
    g = lib()
    inp = prefill_inputs(LENGTHS, seed=510, geo=GEO)
    ref = run_oracle(inp, geo=GEO)
    y = ref["y"].to(DEV)
    N, T = len(LENGTHS), sum(LENGTHS)
    ws = torch.zeros(g.gdn_chunk_prefill_workspace_size(N, T, geometry=GEO), dtype=torch.uint8, device=DEV)
    s0 = inp["state0"].to(DEV)
    st = s0.clone() if in_place else torch.full_like(s0, float("nan"))
    out = _run(g, _dev(inp), y, st if in_place else s0, st, ws)
    g.gdn_check_device_errors()
    assert _parts_read_back(ws, N) == PARTS
    _check(out, st, ref, "split")


def test_split_inside_a_captured_graph():
    """Under stream capture the call runs as one segment on the capturing stream (the auxiliary
    launch before the main one); replays give the oracle's results."""
    g = lib()
    inp = prefill_inputs(LENGTHS, seed=511, geo=GEO)
    ref = run_oracle(inp, geo=GEO)
    y = ref["y"].to(DEV)
    N, T = len(LENGTHS), sum(LENGTHS)
    ws = torch.zeros(g.gdn_chunk_prefill_workspace_size(N, T, geometry=GEO), dtype=torch.uint8, device=DEV)
    d = _dev(inp)  # every input on the device before the capture
    s0 = d["state0"]
    st = torch.empty_like(s0)
    out = torch.empty((T, GEO.num_v_heads, 128), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            _run(g, d, y, s0, st, ws, out=out, stream=s)
    for _ in range(2):
        st.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        g.gdn_check_device_errors()
        _check(out, st, ref, "graph replay")
    # one segment: 55 and 57 chunks against a share of 8 -> four parts each, 22 -> three
    parts = _parts_read_back(ws, N)
    assert parts == [4, 1, 4, 1, 3], parts
