"""GPU parity of gemm_s8_zp on the warp-level path (igc_set_int8_path(1):
mma.sync m16n8k32 on the raw uint8 / int8 operands) against the CPU oracle,
bit for bit, and against the tcgen05 path: both must give identical int32 and
int8 outputs.  Shapes leave ragged 128-blocks and K tails that are not multiples
of the 32-deep MMA step."""

import numpy as np
import pytest
import torch

import implicit_gemm_conv_tcgen05_gb300 as igc
import oracle
import synth
from gpu_helpers import check_device_ok, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture
def imma():
    old = igc.igc_set_int8_path(igc.INT8_PATH_MMA_SYNC)
    yield
    igc.igc_set_int8_path(old)


def _run(A, Bt, lda=None, **kw):
    M, K = A.shape
    N = Bt.shape[0]
    if lda is not None:  # operands inside wider rows (row stride a multiple of 16)
        Aw = np.zeros((M, lda), dtype=A.dtype)
        Aw[:, :K] = A
        Bw = np.zeros((N, lda), dtype=Bt.dtype)
        Bw[:, :K] = Bt
        dA, dB = dev(Aw)[:, :K], dev(Bw)[:, :K]
    else:
        dA, dB = dev(A), dev(Bt)
    C32 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    C8 = torch.empty((M, N), dtype=torch.int8, device="cuda")
    args = {k: (dev(v) if isinstance(v, np.ndarray) else v) for k, v in kw.items()}
    igc.gemm_s8_zp(dA, dB, C32=C32, C8=C8, **args)
    check_device_ok()
    return host(C32), host(C8)


@pytest.mark.parametrize("a_signed,b_signed", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K,lda", [(64, 64, 32, None), (333, 610, 1104, None),
                                       (130, 200, 1000, 1008), (257, 129, 48, None)])
def test_imma_matches_oracle(imma, a_signed, b_signed, M, N, K, lda):
    rng = np.random.default_rng(M * 3 + N + K + 10 * a_signed + b_signed)
    A = (rng.integers(-128, 128, size=(M, K)).astype(np.int8) if a_signed
         else rng.integers(0, 256, size=(M, K)).astype(np.uint8))
    Bt = (rng.integers(-128, 128, size=(N, K)).astype(np.int8) if b_signed
          else rng.integers(0, 256, size=(N, K)).astype(np.uint8))
    zA_row = rng.integers(-128 if a_signed else 0, 128 if a_signed else 256, size=M).astype(np.int32)
    zB_col = rng.integers(-128 if b_signed else 0, 128 if b_signed else 256, size=N).astype(np.int32)
    scale_col = synth.uniform_f32(M + N, 5, (N,), 1e-6, 1e-3)
    c32, c8 = _run(A, Bt, lda=lda, zA_row=zA_row, zB_col=zB_col, scale_col=scale_col)
    o32, o8, _, _ = oracle.gemm_s8_zp(A, Bt, a_signed=a_signed, b_signed=b_signed, zA_row=zA_row,
                                      zB_col=zB_col, scale_col=scale_col)
    assert np.array_equal(c32, o32)
    assert np.array_equal(c8, o8)


def test_imma_config2_equals_tcgen05_and_oracle():
    w2 = synth.workload(2)
    A, Bt = w2["A"], w2["Bt"]
    kw = dict(zA=128, zB=121, scale=w2["scale"])
    old = igc.igc_set_int8_path(igc.INT8_PATH_MMA_SYNC)
    try:
        i32, i8 = _run(A, Bt, **kw)
    finally:
        igc.igc_set_int8_path(old)
    t32, t8 = _run(A, Bt, **kw)
    assert np.array_equal(i32, t32) and np.array_equal(i8, t8)
    o32, o8, _, _ = oracle.gemm_s8_zp(A, Bt, a_signed=0, b_signed=0, **kw)
    assert np.array_equal(i32, o32) and np.array_equal(i8, o8)


def test_imma_per_tensor_scale_and_zero_points(imma):
    rng = np.random.default_rng(7)
    M, N, K = 200, 300, 512
    A = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    Bt = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
    c32, c8 = _run(A, Bt, zA=100, zB=-3, scale=2.0 ** -12)
    o32, o8, _, _ = oracle.gemm_s8_zp(A, Bt, a_signed=0, b_signed=1, zA=100, zB=-3,
                                      scale=2.0 ** -12)
    assert np.array_equal(c32, o32) and np.array_equal(c8, o8)
