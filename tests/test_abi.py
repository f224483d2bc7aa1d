"""The C ABI without a GPU: the library loads, exports every declared symbol, and rejects bad
arguments on the host before any launch (no compute call is made here)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

from linear_attention_ssm_gb300 import binding  # noqa: E402
from linear_attention_ssm_gb300.synth import QWEN_GDN, Geometry  # noqa: E402


def declared_symbols(headers=None):
    names = set()
    for fn in os.listdir(INCLUDE):
        if fn.endswith(".h") and (headers is None or fn in headers):
            text = open(os.path.join(INCLUDE, fn)).read()
            names |= set(re.findall(r"GDN_API\s+[\w\s\*]+?\b(gdn_\w+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.LIB_PATH) or not os.path.exists(binding.TEST_LIB_PATH):
        from linear_attention_ssm_gb300 import build
        build.build()
    return binding.load_library()


@pytest.fixture(scope="module")
def test_lib(lib):
    return binding.load_test_library()


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("gdn_conv1d_prefill", "gdn_chunk_prefill", "gdn_gated_rmsnorm", "gdn_decode_step",
                     "gdn_chunk_prefill_workspace_size", "gdn_check_device_errors", "gdn_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib, test_lib):
    """libgdn.so exports every entry point of gdn.h and none of the verification hooks of
    gdn_debug.h; the test build, libgdn_test.so, exports both."""
    product = declared_symbols({"gdn.h"})
    hooks = declared_symbols({"gdn_debug.h"})
    assert hooks and set(product) | set(hooks) == set(declared_symbols())
    missing = [n for n in product if not hasattr(lib, n)]
    assert not missing, missing
    leaked = [n for n in hooks if hasattr(lib, n)]
    assert not leaked, f"the product library exports test hooks: {leaked}"
    missing = [n for n in product + hooks if not hasattr(test_lib, n)]
    assert not missing, missing


def test_test_hooks_validate_their_arguments(test_lib):
    assert test_lib.gdn_debug_set_chunk_mode(3) == 1
    assert test_lib.gdn_debug_get_chunk_mode() == 0
    assert test_lib.gdn_debug_set_dropped_copy(4) == 1


def test_chunk_size_constant_matches_pages():
    text = open(os.path.join(INCLUDE, "gdn.h")).read()
    assert re.search(r"#define\s+GDN_CHUNK_SIZE\s+64\b", text)


def test_status_strings(lib):
    for code in range(8):
        assert lib.gdn_status_string(code).decode().startswith("GDN_")


FAKE = ctypes.c_void_p(0x10000)      # 16-byte aligned, never dereferenced: every call below fails
ODD = ctypes.c_void_p(0x10002)       # validation before any launch


def _geo(**kw):
    g = dict(num_k_heads=16, num_v_heads=48, head_k_dim=128, head_v_dim=128, conv_width=4)
    g.update(kw)
    return ctypes.byref(binding._Geo(g["num_k_heads"], g["num_v_heads"], g["head_k_dim"],
                                     g["head_v_dim"], g["conv_width"]))


def _chunk(lib, geo=None, qkv=FAKE, g=FAKE, beta=FAKE, cu=FAKE, N=1, T=16, state_in=None, state_out=None,
           z=None, norm_w=None, out=FAKE, l2=1e-6, ws=None, wsb=0):
    return lib.gdn_chunk_prefill(geo or _geo(), qkv, g, beta, cu, N, T, 0.088, l2, state_in, state_out, z,
                                 norm_w, 1e-6, out, ws, wsb, None)


def test_chunk_prefill_rejects_bad_arguments(lib):
    E = binding
    assert _chunk(lib, geo=_geo(head_k_dim=64)) == 2           # unsupported geometry
    assert _chunk(lib, geo=_geo(num_v_heads=40)) == 2          # Hv not a multiple of Hk
    assert _chunk(lib, geo=_geo(conv_width=3)) == 2
    assert _chunk(lib, cu=None) == 1                            # null cu_seqlens
    assert _chunk(lib, qkv=None) == 1
    assert _chunk(lib, qkv=ODD) == 3                            # misaligned
    assert _chunk(lib, out=ODD) == 3
    assert _chunk(lib, N=-1) == 1
    assert _chunk(lib, N=0, T=5) == 1                           # tokens without a sequence
    assert _chunk(lib, z=FAKE, norm_w=None) == 1                # gate without its weight
    assert _chunk(lib, l2=-1.0) == 1
    assert "l2" in lib.gdn_last_error_message().decode() or "eps" in lib.gdn_last_error_message().decode()
    assert lib.gdn_chunk_prefill(None, FAKE, FAKE, FAKE, FAKE, 1, 16, 1.0, 1e-6, None, None, None, None, 1e-6,
                                 FAKE, None, 0, None) == 1
    assert E.GDN_OK == 0


def test_conv_rejects_bad_arguments(lib):
    geo = _geo()
    assert lib.gdn_conv1d_prefill(geo, FAKE, FAKE, None, 1, 8, None, None, FAKE, None) == 1
    assert lib.gdn_conv1d_prefill(geo, ODD, FAKE, FAKE, 1, 8, None, None, FAKE, None) == 3
    assert lib.gdn_conv1d_prefill(geo, FAKE, FAKE, FAKE, 1, 8, None, None, FAKE, None) == 1  # y overlaps x
    assert lib.gdn_conv1d_prefill(_geo(conv_width=2), FAKE, FAKE, FAKE, 1, 8, None, None, FAKE, None) == 2
    # nothing to do is not an error
    assert lib.gdn_conv1d_prefill(geo, None, None, None, 0, 0, None, None, None, None) == 0


def test_decode_and_norm_reject_bad_arguments(lib):
    geo = _geo()
    args = [geo, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.088, 1e-6, 1e-6, FAKE]
    assert lib.gdn_decode_step(*args, -1, None) == 1
    assert lib.gdn_decode_step(*args, 70000, None) == 1
    assert lib.gdn_decode_step(*args, 0, None) == 0
    bad = list(args)
    bad[6] = ODD   # state
    assert lib.gdn_decode_step(*bad, 4, None) == 3
    assert lib.gdn_decode_step(_geo(num_k_heads=1, num_v_heads=48), *args[1:], 4, None) == 2
    assert lib.gdn_gated_rmsnorm(geo, FAKE, None, FAKE, 1e-6, FAKE, 4, None) == 1
    assert lib.gdn_gated_rmsnorm(geo, FAKE, FAKE, FAKE, 1e-6, ODD, 4, None) == 3
    assert lib.gdn_gated_rmsnorm(geo, None, None, None, 1e-6, None, 0, None) == 0


def test_workspace_is_required_and_aligned(lib):
    need = lib.gdn_chunk_prefill_min_workspace_size(_geo(), 8, 32735)
    assert need == 512                                   # counter block + 8 sequence slots, 256-rounded
    assert lib.gdn_chunk_prefill_min_workspace_size(_geo(), 0, 0) == 0
    assert lib.gdn_chunk_prefill_workspace_size(_geo(), 0, 0) == 0
    assert _chunk(lib, N=8, T=32735) == 7                                    # missing workspace
    assert _chunk(lib, N=8, T=32735, ws=FAKE, wsb=need - 1) == 7             # too small
    assert _chunk(lib, N=8, T=32735, ws=ctypes.c_void_p(0x10010), wsb=need) == 3  # not 256-byte aligned


def test_fast_path_workspace_size():
    """Header blocks plus one 25,856-byte record per (chunk, V head), with the chunk count bounded
    by sum_n ceil(L_n / 64) <= (T + 63 N) / 64."""
    lib = binding.load_library()
    rec = 2 * 8192 + 8192 + 5 * 64 * 4
    for n, t in ((1, 16), (4, 4 * 4096), (8, 32735), (3, 0)):
        chunks = (t + 63 * n) // 64
        pad = lambda b: -(-b // 256) * 256
        # counters, order, chunk offsets, four per-segment chunk prefixes; parts per sequence, slot
        # bases, work items (one per sequence plus up to 2 x 32 for parts), 32 x 192 completion flags
        head = (256 + pad(4 * n) + pad(4 * (n + 1)) + pad(4 * 4 * (n + 1)) + 2 * pad(4 * n) + pad(8 * (n + 64)) +
                pad(4 * 32 * 192))
        # from 4,096 tokens on: 32 state slots of 48 heads x 128 x 128 fp32 for the parts of long sequences
        slots = 32 * 48 * 128 * 128 * 4 if t >= 4096 else 0
        assert lib.gdn_chunk_prefill_workspace_size(_geo(), n, t) == head + chunks * 48 * rec + slots
    # the bound covers the worst case: every sequence one token past a chunk boundary
    lengths = [65] * 7
    assert sum(-(-L // 64) for L in lengths) <= (sum(lengths) + 63 * 7) // 64


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(4, QWEN_GDN.conv_dim, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        binding.gdn_conv1d_prefill(x, x, torch.zeros(2, dtype=torch.int32))


def test_verify_stash_size_and_argument_checks(lib):
    """One 53,440-byte record per (sequence, row): raw inputs 20,480 + keys 16 x 128 x 4 + deltas
    48 x 128 x 4 + g 48 x 4.  Rows outside [1, 17] and a short stash are refused before any
    launch; batch 0 is a no-op."""
    geo = _geo()
    assert lib.gdn_verify_stash_size(geo, 256, 8) == 256 * 8 * 53440
    assert lib.gdn_verify_stash_size(geo, 3, 17) == 3 * 17 * 53440
    assert lib.gdn_verify_stash_size(geo, 1, 0) == 0 and lib.gdn_verify_stash_size(geo, 1, 18) == 0
    args = [geo, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.088, 1e-6, 1e-6, FAKE]
    big = 1 << 40
    assert lib.gdn_verify(*args, 4, 0, FAKE, big, None) == 1        # rows 0
    assert lib.gdn_verify(*args, 4, 18, FAKE, big, None) == 1       # rows 18
    assert lib.gdn_verify(*args, -1, 8, FAKE, big, None) == 1       # negative batch
    assert lib.gdn_verify(*args, 4, 8, FAKE, 4 * 8 * 53440 - 1, None) == 7  # stash too small
    assert lib.gdn_verify(*args, 4, 8, None, big, None) == 1        # no stash
    assert lib.gdn_verify(*args, 0, 8, None, 0, None) == 0          # nothing to do
    # 12 V heads per K head: 17 rows no longer fit the kernel's shared memory
    assert lib.gdn_verify(_geo(num_k_heads=4, num_v_heads=48), *args[1:], 4, 17, FAKE, big, None) == 2
    assert lib.gdn_verify_commit(geo, FAKE, FAKE, big, FAKE, FAKE, 4, 18, None) == 1
    assert lib.gdn_verify_commit(geo, None, FAKE, big, FAKE, FAKE, 4, 8, None) == 1
    assert lib.gdn_verify_commit(geo, ctypes.c_void_p(0x10002), FAKE, big, FAKE, FAKE, 4, 8, None) == 3
    assert lib.gdn_verify_commit(geo, None, None, 0, None, None, 0, 8, None) == 0
    # a stash sized for fewer rows (or sequences) than the commit names is refused
    assert lib.gdn_verify_commit(geo, FAKE, FAKE, 4 * 8 * 53440 - 1, FAKE, FAKE, 4, 8, None) == 7
    assert lib.gdn_verify_commit(geo, FAKE, FAKE, 4 * 6 * 53440, FAKE, FAKE, 4, 8, None) == 7
    assert lib.gdn_verify_fp16_state(*args, 4, 18, FAKE, big, None) == 1
    assert lib.gdn_verify_fp16_state(*args, 4, 8, FAKE, 4 * 8 * 53440 - 1, None) == 7
    assert lib.gdn_verify_commit_fp16_state(geo, FAKE, FAKE, big, FAKE, ODD, 4, 8, None) == 3
    assert lib.gdn_verify_commit_fp16_state(geo, FAKE, FAKE, 3 * 8 * 53440, FAKE, FAKE, 4, 8, None) == 7


def test_fused_gate_entry_points_reject_bad_arguments(lib):
    geo = _geo()
    P = ctypes.c_void_p
    # prefill: (geo, qkv, a, b, A_log, dt_bias, cu, N, T, q_scale, l2_eps, s_in, s_out, z, w, rms_eps, out, ws, wsb, stream)
    args = lambda a, b, al, db: (geo, FAKE, a, b, al, db, FAKE, 2, 8, 0.088, 1e-6, None, None, None, None, 1e-6, FAKE,
                                 FAKE, 1 << 20, None)
    assert lib.gdn_chunk_prefill_fused_gates(*args(None, FAKE, FAKE, FAKE)) == 1      # a missing
    assert lib.gdn_chunk_prefill_fused_gates(*args(FAKE, None, FAKE, FAKE)) == 1      # b missing
    assert lib.gdn_chunk_prefill_fused_gates(*args(FAKE, FAKE, None, FAKE)) == 1      # A_log missing
    assert lib.gdn_chunk_prefill_fused_gates(*args(P(0x10001), FAKE, FAKE, FAKE)) == 3  # a odd
    assert lib.gdn_chunk_prefill_fused_gates(*args(FAKE, FAKE, FAKE, ODD)) == 3       # dt_bias not 4-aligned
    # decode: (geo, x, w, cs, a, b, A_log, dt_bias, state, z, nw, q_scale, l2, rms, out, batch, stream)
    dargs = lambda a, al: (geo, FAKE, FAKE, FAKE, a, FAKE, al, FAKE, FAKE, FAKE, FAKE, 0.088, 1e-6, 1e-6, FAKE, 4, None)
    assert lib.gdn_decode_step_fused_gates(*dargs(None, FAKE)) == 1
    assert lib.gdn_decode_step_fused_gates(*dargs(FAKE, ODD)) == 3
    assert lib.gdn_decode_step_fused_gates(geo, None, None, None, None, None, None, None, None, None, None, 0.088,
                                           1e-6, 1e-6, None, 0, None) == 0    # batch 0: nothing to do


def test_one_call_prefill_checks_both_stages_before_launching(lib):
    """gdn_prefill refuses a bad argument of either stage with the stage's own status, before any
    CUDA call (here, with no GPU, any CUDA call would end in GDN_ERR_CUDA instead)."""
    geo = _geo()
    X, QKV = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x4000000)  # apart by more than T * C * 2 bytes
    # (geo, x, conv_w, cu, N, T, cs_in, cs_out, qkv, g, beta, q_scale, l2, s_in, s_out, z, nw, rms, out, ws, wsb, stream)
    def call(x=X, w=FAKE, cs_out=None, qkv=QKV, g=FAKE, ws=FAKE, wsb=1 << 30, n=2, t=8):
        return lib.gdn_prefill(geo, x, w, FAKE, n, t, None, cs_out, qkv, g, FAKE, 0.088, 1e-6, None, None, None,
                               None, 1e-6, FAKE, ws, wsb, None)
    assert call(w=None) == 1                        # conv weights missing
    assert call(qkv=None) == 1                      # conv output buffer missing
    assert call(qkv=X) == 1                         # conv output overlaps its input
    assert call(cs_out=ODD) == 3                    # conv state misaligned
    assert call(g=None) == 1                        # the chunk stage's gates missing
    assert call(ws=None) == 7                       # the chunk stage's workspace missing
    assert call(n=0, t=0) == 0                      # nothing to do
    assert call(n=-1) == 1


def test_gates_reject_bad_arguments(lib):
    geo = _geo()
    assert lib.gdn_gates(geo, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, -1, None) == 1
    assert lib.gdn_gates(geo, None, None, None, None, None, None, 0, None) == 0
    assert lib.gdn_gates(geo, FAKE, FAKE, None, FAKE, FAKE, FAKE, 4, None) == 1
    assert lib.gdn_gates(geo, FAKE, FAKE, ctypes.c_void_p(0x10001), FAKE, FAKE, FAKE, 4, None) == 3
    assert lib.gdn_gates(geo, ODD, FAKE, FAKE, FAKE, FAKE, FAKE, 4, None) == 3


def test_kda_decode_rejects_bad_arguments(lib):
    geo = _geo(num_k_heads=64, num_v_heads=64)
    tail = [FAKE, FAKE, FAKE, 0.088, 1e-6, 1e-6, FAKE]  # state, z, norm_w, q_scale, eps, eps, out
    assert lib.gdn_kda_decode_step(geo, FAKE, FAKE, FAKE, FAKE, -1.0, FAKE, *tail, -1, None) == 1
    assert lib.gdn_kda_decode_step(geo, FAKE, FAKE, FAKE, FAKE, float("nan"), FAKE, *tail, 4, None) == 1
    assert lib.gdn_kda_decode_step(geo, FAKE, FAKE, FAKE, ODD, -1.0, FAKE, *tail, 4, None) == 3
    assert lib.gdn_kda_decode_step(geo, None, None, None, None, -1.0, None, None, None, None, 0.088, 1e-6,
                                   1e-6, None, 0, None) == 0


def test_kda_recurrence_rejects_bad_arguments(lib):
    geo = _geo(num_k_heads=64, num_v_heads=64)

    def call(qkv=FAKE, g=FAKE, g_min=-1.0, beta=FAKE, cu=FAKE, N=2, T=8, state_in=None, state_out=None, z=None,
             norm_w=None, out=FAKE, l2=1e-6):
        return lib.gdn_kda_recurrence(geo, qkv, g, g_min, beta, cu, N, T, 0.088, l2, state_in, state_out, z,
                                      norm_w, 1e-6, out, None)

    assert call(N=-1) == 1
    assert call(N=0, T=4) == 1
    assert call(N=70000) == 1                      # the grid's sequence dimension
    assert call(cu=None) == 1
    assert call(g=None) == 1
    assert call(beta=None) == 1
    assert call(g_min=float("nan")) == 1
    assert call(l2=-1.0) == 1
    assert call(z=FAKE, norm_w=None) == 1
    assert call(g=ODD) == 3
    assert call(qkv=ODD) == 3
    assert call(state_in=ODD) == 3
    assert call(state_in=FAKE, state_out=ctypes.c_void_p(0x10000 + 4096)) == 1   # partial overlap
    assert lib.gdn_kda_recurrence(_geo(head_k_dim=64), FAKE, FAKE, -1.0, FAKE, FAKE, 1, 4, 0.088, 1e-6, None,
                                  None, None, None, 1e-6, FAKE, None) == 2
    assert call(N=0, T=0, qkv=None, g=None, beta=None, cu=None, out=None) == 0


def test_kda_chunk_prefill_rejects_bad_arguments(lib):
    geo = _geo(num_k_heads=64, num_v_heads=64)
    need = lib.gdn_kda_chunk_prefill_workspace_size(geo, 2, 8)

    def call(qkv=FAKE, g=FAKE, g_min=-1.0, beta=FAKE, cu=FAKE, N=2, T=8, state_in=None, state_out=None, z=None,
             norm_w=None, out=FAKE, l2=1e-6, ws=ctypes.c_void_p(0x100000), wsb=need):
        return lib.gdn_kda_chunk_prefill(geo, qkv, g, g_min, beta, cu, N, T, 0.088, l2, state_in, state_out, z,
                                         norm_w, 1e-6, out, ws, wsb, None)

    assert call(N=-1) == 1
    assert call(N=0, T=4) == 1
    assert call(cu=None) == 1
    assert call(g=None) == 1
    assert call(beta=None) == 1
    assert call(g_min=float("nan")) == 1
    assert call(l2=-1.0) == 1
    assert call(z=FAKE, norm_w=None) == 1
    assert call(g=ODD) == 3
    assert call(qkv=ODD) == 3
    assert call(state_in=ODD) == 3
    assert call(state_in=FAKE, state_out=ctypes.c_void_p(0x10000 + 4096)) == 1   # partial overlap
    assert call(ws=None) == 7                                                     # missing workspace
    assert call(wsb=need - 1) == 7                                                # too small
    assert call(ws=ctypes.c_void_p(0x100010)) == 3                                # not 256-byte aligned
    assert lib.gdn_kda_chunk_prefill(_geo(head_k_dim=64), FAKE, FAKE, -1.0, FAKE, FAKE, 1, 4, 0.088, 1e-6, None,
                                     None, None, None, 1e-6, FAKE, FAKE, need, None) == 2
    assert call(N=0, T=0, qkv=None, g=None, beta=None, cu=None, out=None, ws=None, wsb=0) == 0


def test_kda_one_call_prefill_checks_both_stages_before_launching(lib):
    """gdn_kda_prefill refuses a bad argument of either stage before it launches anything."""
    geo = _geo(num_k_heads=64, num_v_heads=64)
    need = lib.gdn_kda_chunk_prefill_workspace_size(geo, 2, 8)
    WS = ctypes.c_void_p(0x100000)
    C = (2 * 64 + 64) * 128

    def call(x=FAKE, conv_w=FAKE, cs_in=None, cs_out=None, qkv=ctypes.c_void_p(0x10000 + 8 * C * 2), g=FAKE,
             g_min=-1.0, ws=WS, wsb=need, N=2, T=8):
        return lib.gdn_kda_prefill(geo, x, conv_w, FAKE, N, T, cs_in, cs_out, qkv, g, g_min, FAKE, 0.088, 1e-6, None,
                                   None, None, None, 1e-6, FAKE, ws, wsb, None)

    assert call(conv_w=None) == 1                        # the conv stage's own arguments
    assert call(x=None) == 1
    assert call(cs_in=ODD) == 3
    assert call(qkv=ctypes.c_void_p(0x10000 + 64)) == 1  # qkv overlaps x
    assert call(g=None) == 1                             # the chunk stage's
    assert call(g_min=float("nan")) == 1
    assert call(ws=None) == 7
    assert call(N=0, T=0, x=None, conv_w=None, qkv=None, g=None, ws=None, wsb=0) == 0


def test_kda_chunk_workspace_size():
    """Counters, order and chunk offsets, then one 108,032-byte record per (chunk, V head): K~ hi
    and Q~ (64 + 64 token rows x 128 bf16), K~ lo (64 x 128), Kd hi / lo (2 x 64 x 128), T hi / lo
    and P (3 x 64 x 64 bf16), and 384 floats of per-token and per-channel factors."""
    lib = binding.load_library()
    rec = 128 * 128 * 2 + 64 * 128 * 2 + 2 * 64 * 128 * 2 + 3 * 64 * 64 * 2 + 384 * 4
    assert rec == 108032
    pad = lambda b: -(-b // 256) * 256
    for n, t in ((1, 16), (4, 4 * 4096), (8, 32735), (3, 0)):
        chunks = (t + 63 * n) // 64
        want = 256 + pad(4 * n) + pad(4 * (n + 1)) + chunks * 64 * rec
        assert lib.gdn_kda_chunk_prefill_workspace_size(_geo(num_k_heads=64, num_v_heads=64), n, t) == want
    assert lib.gdn_kda_chunk_prefill_workspace_size(_geo(num_k_heads=64, num_v_heads=64), 0, 0) == 0


def test_header_is_a_plain_c_abi(lib, tmp_path):
    """A C11 program built against include/*.h alone (gcc -Wall -Wextra -Werror) links against
    libgdn.so and gets the documented status from every entry point it calls."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "c_abi_check")
    libdir = os.path.dirname(binding.LIB_PATH)
    src = os.path.join(ROOT, "tests", "c_abi_check.c")
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE, src, "-o", exe,
                    "-L", libdir, "-lgdn", f"-Wl,-rpath,{libdir}", "-lm"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stderr


def test_python_binding_has_every_c_entry_point_by_name():
    """The binding is the C ABI under the same names: every declared entry point has a Python
    function of that name (exported by the package too)."""
    import linear_attention_ssm_gb300 as pkg
    missing = [n for n in declared_symbols() if not callable(getattr(binding, n, None))]
    assert not missing, missing
    not_exported = [n for n in declared_symbols() if not hasattr(pkg, n)]
    assert not not_exported, not_exported


def test_binding_helpers_without_a_gpu(lib):
    import torch
    assert binding.gdn_status_string(3) == "GDN_ERR_MISALIGNED"
    assert isinstance(binding.gdn_last_error_message(), str)
    f32 = torch.zeros(1, 48, 128, 128)
    with pytest.raises(TypeError):   # the fp16 entry points refuse an fp32 state before anything else
        binding.gdn_verify_fp16_state(None, None, None, None, None, f32, None, None, 0.088)
    with pytest.raises(TypeError):
        binding.gdn_verify_commit_fp16_state(None, None, None, f32, 4)
    with pytest.raises(TypeError):   # host tensors are refused
        binding.gdn_chunk_prefill_noalloc(torch.zeros(4, 10240, dtype=torch.bfloat16), torch.zeros(4, 48),
                                          torch.zeros(4, 48), torch.tensor([0, 4], dtype=torch.int32), 0.088)
