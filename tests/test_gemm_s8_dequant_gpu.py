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


def test_dequant_per_column_zero_points_and_strided_output():
    """Per-column zB with a Y view whose rows are longer than N (row stride 200 > N)."""
    M, N, K = 192, 136, 320
    A, Bt, zA_row, _, s_row, s_col, bias = _case(M, N, K, 0, 1, True, True, True, seed=9)
    zB_col = np.random.default_rng(9).integers(-128, 128, size=N).astype(np.int32)
    Ybig = torch.full((M, 200), -7.0, dtype=torch.float32, device="cuda")
    Y = Ybig[:, 8:8 + N]
    igc.gemm_s8_zp_dequant(dev(A), dev(Bt), zA_row=dev(zA_row), zB_col=dev(zB_col),
                           scale_row=dev(s_row), scale_col=dev(s_col), bias=dev(bias), Y=Y)
    check_device_ok()
    C32, _, _, _ = oracle.gemm_s8_zp(A, Bt, a_signed=0, b_signed=1, zA_row=zA_row,
                                     zB_col=zB_col, want_c8=False)
    want = oracle.dequant_matrix(C32, s_row, s_col, bias)
    got = host(Ybig)
    assert np.array_equal(got[:, 8:8 + N].view(np.uint32), want.view(np.uint32))
    assert np.all(got[:, :8] == -7.0) and np.all(got[:, 8 + N:] == -7.0)


def test_dequant_8192_cubed_sampled_rows():
    """The benchmark's dequantised 8192^3 problem: the whole output on the GPU,
    sampled rows (every 256-row tile edge class) against the oracle."""
    w5 = synth.workload(5)
    srow = synth.uniform_f32(42, 1, (8192,), 1e-3, 1e-2)
    bias = synth.uniform_f32(42, 2, (8192,), -1.0, 1.0)
    Y = igc.gemm_s8_zp_dequant(dev(w5["A"]), dev(w5["Bt"]), zA_row=dev(w5["zA_row"]),
                               scale_row=dev(srow), scale_col=dev(w5["scale_col"]),
                               bias=dev(bias))
    check_device_ok()
    rows = np.array([0, 127, 128, 255, 4096, 8191])
    C32, _, _, _ = oracle.gemm_s8_zp(w5["A"][rows], w5["Bt"], a_signed=0, b_signed=1,
                                     zA_row=w5["zA_row"][rows], want_c8=False)
    want = oracle.dequant_matrix(C32, srow[rows], w5["scale_col"], bias)
    got = host(Y)[rows]
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
