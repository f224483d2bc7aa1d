"""One tcgen05 tile through the library's debug probe: checks the shared-memory swizzle layout,
the matrix and instruction descriptors and the tensor-memory read-back that the chunk prefill
builds on, against torch's matmul of the same bf16 operands."""
import pytest
import torch

from tests.gpu_common import lib, DEV

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n", [64, 128])
def test_mma_probe_matches_matmul(n):
    g = lib()
    gen = torch.Generator().manual_seed(n)
    A = torch.randn(128, 64, generator=gen).to(torch.bfloat16)
    B = torch.randn(n, 64, generator=gen).to(torch.bfloat16)
    D, status = g.gdn_debug_mma_probe(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "the MMA completion wait ran out"
    ref = A.double() @ B.double().T
    err = (D.cpu().double() - ref).abs().max().item()
    assert err < 1e-3 * ref.abs().max().item(), err


def test_mma_probe_structured_operands():
    """Identity-like operands make any row/column permutation visible."""
    g = lib()
    A = torch.zeros(128, 64)
    for r in range(128):
        A[r, r % 64] = 1.0 + (r // 64)        # rows 64..127 scaled by 2: exact in bf16
    B = torch.arange(64 * 64, dtype=torch.float32).reshape(64, 64) % 251 - 125
    D, status = g.gdn_debug_mma_probe(A.to(torch.bfloat16).to(DEV), B.to(torch.bfloat16).to(DEV))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = A.to(torch.bfloat16).double() @ B.to(torch.bfloat16).double().T
    assert torch.equal(D.cpu().double(), ref)


@pytest.mark.parametrize("flags", [1, 2, 3], ids=["a_tmem", "b_mn", "a_tmem_b_mn"])
@pytest.mark.parametrize("n", [64, 128])
def test_mma_probe_operand_placements(n, flags):
    """A from tensor memory and B MN-major, as the split chunk prefill's state kernel uses them:
    structured operands (a permutation of rows, columns or K would show) and random ones."""
    g = lib()
    A = torch.zeros(128, 64)
    for r in range(128):
        A[r, (5 * r) % 64] = 1.0 + (r // 64)
    B = torch.arange(n * 64, dtype=torch.float32).reshape(n, 64) % 251 - 125
    D, status = g.gdn_debug_mma_probe_ex(A.to(torch.bfloat16).to(DEV), B.to(torch.bfloat16).to(DEV), flags)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = A.to(torch.bfloat16).double() @ B.to(torch.bfloat16).double().T
    assert torch.equal(D.cpu().double(), ref)
    gen = torch.Generator().manual_seed(100 + n + flags)
    A = torch.randn(128, 64, generator=gen).to(torch.bfloat16)
    B = torch.randn(n, 64, generator=gen).to(torch.bfloat16)
    D, status = g.gdn_debug_mma_probe_ex(A.to(DEV), B.to(DEV), flags)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = A.double() @ B.double().T
    assert (D.cpu().double() - ref).abs().max().item() < 1e-3 * ref.abs().max().item()
