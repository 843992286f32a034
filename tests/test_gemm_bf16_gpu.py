"""GPU parity of gemm_bf16 (tcgen05 kind::f16 with bf16 operands) against the
CPU oracle, through the C-ABI binding."""

import numpy as np
import pytest
import torch

import implicit_gemm_conv_tcgen05_gb300 as igc
import oracle
import synth
from gpu_helpers import assert_fp16_bound, check_device_ok

pytestmark = pytest.mark.gpu


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _run(A_bits, Bt_bits):
    M, N = A_bits.shape[0], Bt_bits.shape[0]
    C16 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    C32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    igc.gemm_bf16(_dev_bf16(A_bits), _dev_bf16(Bt_bits), C16, C32)
    check_device_ok()
    torch.cuda.synchronize()
    return C16.view(torch.int16).cpu().numpy().view(np.uint16), C32.cpu().numpy()


def _assert_rne(c16_bits, c32, what):
    want = oracle.f32_to_bf16_bits_array(c32)
    bad = np.count_nonzero(c16_bits != want)
    assert bad == 0, f"{what}: {bad} bf16 outputs are not the RNE rounding of the fp32 copy"


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (200, 300, 72), (129, 257, 8), (333, 520, 1000)])
def test_bf16_parity(M, N, K):
    A = synth.normal_bf16_bits(M + 7, 1, (M, K))
    Bt = synth.normal_bf16_bits(N + 7, 2, (N, K))
    c16, c32 = _run(A, Bt)
    ref, sabs = oracle.gemm_bf16(A, Bt)
    assert_fp16_bound(c32, ref, sabs, f"bf16 {M}x{N}x{K}")
    _assert_rne(c16, c32, f"bf16 {M}x{N}x{K}")


def test_bf16_small_integers_bit_exact():
    rng = np.random.default_rng(2)
    A = rng.integers(-2, 3, size=(384, 512)).astype(np.float32)
    Bt = rng.integers(-2, 3, size=(256, 512)).astype(np.float32)
    bits = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    c16, c32 = _run(bits(A), bits(Bt))
    assert np.array_equal(c32.astype(np.float64), A.astype(np.float64) @ Bt.T.astype(np.float64))


def test_bf16_4096_cubed_sampled_rows():
    A = synth.normal_bf16_bits(31, 1, (4096, 4096))
    Bt = synth.normal_bf16_bits(31, 2, (4096, 4096))
    c16, c32 = _run(A, Bt)
    _assert_rne(c16, c32, "bf16 4096^3")
    rows = np.array([0, 255, 256, 2049, 4095])
    ref, sabs = oracle.gemm_bf16(A[rows], Bt)
    assert_fp16_bound(c32[rows], ref, sabs, "bf16 4096^3 rows")
