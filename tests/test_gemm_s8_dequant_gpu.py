"""GPU parity of gemm_s8_zp_dequant (int8 GEMM with the dequantise + bias half
of the four-term fusion fused into the epilogue): fp32 outputs bit-exact
against the CPU oracle."""

import numpy as np
import pytest
import torch

import implicit_gemm_conv_tcgen05_gb300 as igc
import oracle
import synth
from gpu_helpers import check_device_ok, dev, host

pytestmark = pytest.mark.gpu


def _case(M, N, K, a_signed, b_signed, with_row, with_col, with_bias, seed):
    rng = np.random.default_rng(seed)
    A = (rng.integers(-128, 128, size=(M, K)).astype(np.int8) if a_signed
         else rng.integers(0, 256, size=(M, K)).astype(np.uint8))
    Bt = (rng.integers(-128, 128, size=(N, K)).astype(np.int8) if b_signed
          else rng.integers(0, 256, size=(N, K)).astype(np.uint8))
    zA_row = rng.integers(0, 200, size=M).astype(np.int32)
    zB = int(rng.integers(-10, 130))
    s_row = synth.uniform_f32(seed, 5, (M,), 1e-3, 1e-1) if with_row else None
    s_col = synth.uniform_f32(seed, 6, (N,), 1e-3, 1e-1) if with_col else None
    bias = synth.uniform_f32(seed, 7, (N,), -5.0, 5.0) if with_bias else None
    return A, Bt, zA_row, zB, s_row, s_col, bias


@pytest.mark.parametrize("M,N,K,signs,steps", [
    (256, 256, 256, (0, 1), (1, 1, 1)),
    (130, 300, 272, (0, 0), (1, 1, 1)),
    (300, 129, 1040, (1, 1), (0, 1, 1)),
    (64, 512, 48, (1, 0), (1, 0, 0)),
    (1024, 1024, 1024, (0, 1), (0, 0, 0)),
])
def test_dequant_output_bit_exact(M, N, K, signs, steps):
    A, Bt, zA_row, zB, s_row, s_col, bias = _case(M, N, K, *signs, *steps, seed=M + N + K)
    Y = igc.gemm_s8_zp_dequant(dev(A), dev(Bt), zA_row=dev(zA_row), zB=zB,
                               scale_row=None if s_row is None else dev(s_row),
                               scale_col=None if s_col is None else dev(s_col),
                               bias=None if bias is None else dev(bias))
    check_device_ok()
    C32, _, _, _ = oracle.gemm_s8_zp(A, Bt, a_signed=signs[0], b_signed=signs[1],
                                     zA_row=zA_row, zB=zB, want_c8=False)
    want = oracle.dequant_matrix(C32, s_row, s_col, bias)
    got = host(Y)
    bad = np.count_nonzero(got.view(np.uint32) != want.view(np.uint32))
    assert bad == 0, f"{bad} of {got.size} dequantised outputs differ"


def test_dequant_rejects_k_zero():
    A = torch.empty((8, 0), dtype=torch.uint8, device="cuda")
    Bt = torch.empty((16, 0), dtype=torch.uint8, device="cuda")
    with pytest.raises(igc.IGCError) as e:
        igc.gemm_s8_zp_dequant(A, Bt)
    assert e.value.status == igc.IGC_ERR_UNSUPPORTED
