"""GPU parity of gemm_f16 (tcgen05 kind::f16, TMEM fp32 accumulators) against
the CPU oracle, through the C-ABI binding."""

import numpy as np
import pytest
import torch

import implicit_gemm_conv_tcgen05_gb300 as igc
import oracle
import synth
from gpu_helpers import (assert_f16_is_rne_of_f32, assert_fp16_bound, check_device_ok, dev,
                         host)

pytestmark = pytest.mark.gpu


def _run(A, Bt, out_dtype=torch.float32, with_check=False):
    M, N = A.shape[0], Bt.shape[0]
    C = torch.empty((M, N), dtype=out_dtype, device="cuda")
    C32 = torch.empty((M, N), dtype=torch.float32, device="cuda") if with_check else None
    igc.gemm_f16(dev(A), dev(Bt), C, C32)
    check_device_ok()
    return host(C), (host(C32) if with_check else None)


def test_config1_256_cubed_fp32_out():
    w = synth.workload(1)
    C, _ = _run(w["A"], w["Bt"])
    ref, sabs = oracle.gemm_f16(w["A"], w["Bt"])
    assert_fp16_bound(C, ref, sabs, "256^3")


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 300, 72), (1, 1, 8), (129, 257, 8),
                                   (333, 520, 1000), (640, 512, 192), (77, 1031, 136)])
def test_ragged_shapes_fp16_out_with_check(M, N, K):
    A = synth.uniform_f16(100 + M, 1, (M, K))
    Bt = synth.uniform_f16(100 + N, 2, (N, K))
    C16, C32 = _run(A, Bt, torch.float16, with_check=True)
    ref, sabs = oracle.gemm_f16(A, Bt)
    assert_fp16_bound(C32, ref, sabs, f"{M}x{N}x{K} fp32 copy")
    assert_fp16_bound(C16, ref, sabs, f"{M}x{N}x{K} fp16")
    assert_f16_is_rne_of_f32(C16, C32, f"{M}x{N}x{K}")


def test_small_integers_bit_exact():
    # every partial sum is an integer below 2^14: fp32 and fp16 results are exact
    rng = np.random.default_rng(1)
    M, N, K = 384, 512, 1024
    A = rng.integers(-2, 3, size=(M, K)).astype(np.float16)
    Bt = rng.integers(-2, 3, size=(N, K)).astype(np.float16)
    C16, C32 = _run(A, Bt, torch.float16, with_check=True)
    ref, _ = oracle.gemm_f16(A, Bt)
    assert np.array_equal(C32.astype(np.float64), ref)
    assert np.array_equal(C16.astype(np.float64), ref)


def test_identity_and_permutation():
    n = 256
    B = synth.uniform_f16(5, 2, (n, n))
    eye = np.eye(n, dtype=np.float16)
    C, _ = _run(eye, B)
    assert np.array_equal(C, B.astype(np.float32).T)
    perm = np.random.default_rng(2).permutation(n)
    P = eye[perm]
    C, _ = _run(B, P)          # C[i,j] = sum_k B[i,k] P[j,k] = B[i, perm[j]]
    assert np.array_equal(C, B.astype(np.float32)[:, perm])


def test_strided_views():
    M, N, K = 192, 320, 128
    Abig = torch.from_numpy(synth.uniform_f16(9, 1, (M, K + 64))).cuda()
    Bbig = torch.from_numpy(synth.uniform_f16(9, 2, (N, K + 16))).cuda()
    A, Bt = Abig[:, :K], Bbig[:, 8:8 + K]
    Cbig = torch.zeros((M, N + 8), dtype=torch.float32, device="cuda")
    C = Cbig[:, :N]
    igc.gemm_f16(A, Bt, C)
    check_device_ok()
    ref, sabs = oracle.gemm_f16(A.cpu().numpy(), Bt.cpu().numpy())
    assert_fp16_bound(host(C), ref, sabs, "strided")
    assert torch.all(Cbig[:, N:] == 0)   # nothing written outside C


def test_k_zero_writes_zeros_and_empty_is_noop():
    A = torch.empty((64, 0), dtype=torch.float16, device="cuda")
    Bt = torch.empty((48, 0), dtype=torch.float16, device="cuda")
    C = torch.full((64, 48), 7.0, dtype=torch.float32, device="cuda")
    igc.gemm_f16(A, Bt, C)
    assert torch.all(C == 0)
    A0 = torch.empty((0, 16), dtype=torch.float16, device="cuda")
    Bt0 = torch.empty((8, 16), dtype=torch.float16, device="cuda")
    igc.gemm_f16(A0, Bt0, torch.empty((0, 8), dtype=torch.float32, device="cuda"))


def test_misaligned_operand_rejected():
    buf = torch.zeros(64 * 72 + 8, dtype=torch.float16, device="cuda")
    A = buf[1:1 + 64 * 64].view(64, 64)           # 2-byte offset: not 16-byte aligned
    Bt = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(igc.IGCError) as e:
        igc.gemm_f16(A, Bt)
    assert e.value.status == igc.IGC_ERR_MISALIGNED


def test_config3_4096_cubed_sampled_rows():
    w = synth.workload(3)
    M = w["M"]
    C16, C32 = _run(w["A"], w["Bt"], torch.float16, with_check=True)
    assert_f16_is_rne_of_f32(C16, C32, "4096^3")
    rows = np.array([0, 1, 127, 128, 1000, 2047, 2048, 3333, 4094, 4095])
    ref, sabs = oracle.gemm_f16(w["A"][rows], w["Bt"])
    assert_fp16_bound(C32[rows], ref, sabs, "4096^3 rows")
    assert_fp16_bound(C16[rows], ref, sabs, "4096^3 fp16 rows")
    # a column sample too (every m-tile)
    cols = np.array([0, 255, 256, 4095])
    ref_c, sabs_c = oracle.gemm_f16(w["A"], w["Bt"][cols])
    assert_fp16_bound(C32[:, cols], ref_c, sabs_c, "4096^3 cols")


def test_repeated_calls_are_deterministic():
    A = synth.normal_f16(3, 1, (512, 768))
    Bt = synth.normal_f16(3, 2, (640, 768))
    C1, _ = _run(A, Bt)
    C2, _ = _run(A, Bt)
    assert np.array_equal(C1, C2)


@pytest.mark.parametrize("M,N,K", [(2560, 2048, 128), (2304, 2304, 64)])
def test_whole_tiles_and_split_last_round_full_output(M, N, K):
    """80 and 81 tiles of 256 x 256: more than one round of the persistent
    schedule, with a short last round that runs as column halves.  Every
    output is compared."""
    A = synth.uniform_f16(M + 1, 1, (M, K))
    Bt = synth.uniform_f16(N + 2, 2, (N, K))
    C16, C32 = _run(A, Bt, torch.float16, with_check=True)
    ref, sabs = oracle.gemm_f16(A, Bt)
    assert_fp16_bound(C32, ref, sabs, f"{M}x{N}x{K} fp32")
    assert_f16_is_rne_of_f32(C16, C32, f"{M}x{N}x{K}")
