"""The tensor-core building block (tcgen05.mma from shared memory into TMEM)
against a host GEMM of the same bf16 operands."""
import numpy as np
import pytest

from gated_deltanet_linear_12_gb300 import synthetic as syn
from tests.helpers import to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def G():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_linear_12_gb300 import gdn
    gdn.load()
    return gdn


def _gemm(G, A, B):
    D = torch.full((128, B.shape[0]), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.gdn_selftest_tc_gemm(to_dev(A), to_dev(B), D, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "tensor-core completion wait timed out"
    return D.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("N,K", [(16, 16), (64, 128), (128, 64), (256, 128)])
def test_tc_gemm_matches_host(G, N, K):
    rng = np.random.default_rng(N * 1000 + K)
    A = syn.f32_to_bf16_bits(rng.standard_normal((128, K)).astype(np.float32))
    B = syn.f32_to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32))
    ref = syn.bf16_bits_to_f32(A).astype(np.float64) @ syn.bf16_bits_to_f32(B).astype(np.float64).T
    got = _gemm(G, A, B)
    scale = np.abs(syn.bf16_bits_to_f32(A)).astype(np.float64) @ np.abs(syn.bf16_bits_to_f32(B)).astype(np.float64).T
    assert np.all(np.abs(got - ref) <= 1e-5 * scale + 1e-30)


def test_bounded_wait_gives_up_and_reports(G):
    """Failure detection without a fault: the block waits on a barrier nothing
    arrives on; the wait must give up, report, release TMEM and return, and the
    context must stay usable (the next GEMM is exact)."""
    rng = np.random.default_rng(7)
    A = syn.f32_to_bf16_bits(rng.standard_normal((128, 32)).astype(np.float32))
    B = syn.f32_to_bf16_bits(rng.standard_normal((16, 32)).astype(np.float32))
    D = torch.full((128, 16), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.gdn_selftest_tc_gemm(to_dev(A), to_dev(B), D, starve_wait=True, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    assert torch.isnan(D).all(), "a block that gave up must not write results"
    ref = syn.bf16_bits_to_f32(A).astype(np.float64) @ syn.bf16_bits_to_f32(B).astype(np.float64).T
    got = _gemm(G, A, B)
    assert np.allclose(got, ref, rtol=1e-5, atol=1e-5)


def _gemm_tf32(G, A, B):
    D = torch.full((128, B.shape[0]), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.gdn_selftest_tc_gemm_tf32(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), D, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "tensor-core completion wait timed out"
    return D.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("N,K", [(16, 128), (64, 32)])
def test_tc_gemm_tf32_within_tf32_rounding(G, N, K):
    """kind::tf32 with f32 operands: each product carries at most the tf32
    rounding of both operands (10 explicit mantissa bits)."""
    rng = np.random.default_rng(N * 100 + K)
    A = rng.standard_normal((128, K)).astype(np.float32)
    B = rng.standard_normal((N, K)).astype(np.float32)
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    scale = np.abs(A).astype(np.float64) @ np.abs(B).astype(np.float64).T
    got = _gemm_tf32(G, A, B)
    assert np.all(np.abs(got - ref) <= 2.0 ** -9 * scale + 1e-30)


def test_tc_gemm_tf32_operand_conversion():
    """Records how an f32 operand becomes tf32: A = 1 + 0.75 * 2^-10 against a
    unit vector gives 1 (low bits dropped) or 1 + 2^-10 (rounded to nearest)."""
    pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_linear_12_gb300 import gdn
    A = np.full((128, 8), 1.0 + 0.75 * 2.0 ** -10, np.float32)
    B = np.zeros((16, 8), np.float32)
    B[:, 0] = 1.0
    got = _gemm_tf32(gdn, A, B)
    assert np.all((got == 1.0) | (got == 1.0 + 2.0 ** -10)), np.unique(got)
    print("tf32 operand conversion:", "truncation" if got[0, 0] == 1.0 else "round to nearest")
