"""GPU parity with each output tile width forced (igc_set_tile_width): 128, 224
and 256 columns for the fp16 / bf16 GEMM and the fp16 convolution (224-wide
tiles store 128 + 96 columns per row-quadrant and 112 per half-width unit, with
direct stores for columns past the last whole TMA box), 128 and 256 for the
integer paths.  Shapes are ragged and include schedules with whole tiles and a
split last round."""

import numpy as np
import pytest
import torch

import implicit_gemm_conv_tcgen05_gb300 as igc
import oracle
import synth
from gpu_helpers import (assert_f16_is_rne_of_f32, assert_fp16_bound, check_device_ok, dev,
                         host)

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[128, 224, 256])
def width(request):
    old = igc.igc_set_tile_width(request.param)
    yield request.param
    igc.igc_set_tile_width(old)


@pytest.mark.parametrize("M,N,K", [(300, 470, 136), (513, 1000, 64), (64, 2000, 1032),
                                   (2560, 2048, 64)])
def test_gemm_f16_every_width(width, M, N, K):
    A = synth.uniform_f16(M + 7, 1, (M, K))
    Bt = synth.uniform_f16(N + 7, 2, (N, K))
    C = torch.empty((M, N), dtype=torch.float16, device="cuda")
    C32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    igc.gemm_f16(dev(A), dev(Bt), C, C32)
    check_device_ok()
    ref, sabs = oracle.gemm_f16(A, Bt)
    c16, c32 = host(C), host(C32)
    assert_fp16_bound(c32, ref, sabs, f"width {width} fp32")
    assert_f16_is_rne_of_f32(c16, c32, f"width {width}")


def test_gemm_f16_fp32_output_in_strided_view(width):
    M, N, K = 270, 700, 96
    A = synth.normal_f16(71, 1, (M, K))
    Bt = synth.normal_f16(71, 2, (N, K))
    Cbig = torch.full((M, N + 20), 3.0, dtype=torch.float32, device="cuda")
    C = Cbig[:, 4:4 + N]
    igc.gemm_f16(dev(A), dev(Bt), C)
    check_device_ok()
    ref, sabs = oracle.gemm_f16(A, Bt)
    got = host(Cbig)
    assert_fp16_bound(got[:, 4:4 + N], ref, sabs, f"width {width}")
    assert np.all(got[:, :4] == 3.0) and np.all(got[:, 4 + N:] == 3.0)


def test_gemm_bf16_every_width(width):
    M, N, K = 384, 900, 200
    Ab = synth.normal_bf16_bits(72, 1, (M, K))
    Bb = synth.normal_bf16_bits(72, 2, (N, K))
    A = torch.from_numpy(Ab.view(np.int16)).cuda().view(torch.bfloat16)
    Bt = torch.from_numpy(Bb.view(np.int16)).cuda().view(torch.bfloat16)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    C32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    igc.gemm_bf16(A, Bt, C, C32)
    check_device_ok()
    ref, sabs = oracle.gemm_bf16(Ab, Bb)
    c32 = host(C32)
    assert_fp16_bound(c32, ref, sabs, f"bf16 width {width}")
    want = oracle.f32_to_bf16_bits_array(c32)
    got = C.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_conv_every_width(width):
    x = synth.normal_f16(73, 6, (3, 10, 11, 64))
    w = synth.normal_f16(73, 7, (200, 3, 3, 64), std=1.0 / 24)
    y = torch.empty((3, 10, 11, 200), dtype=torch.float16, device="cuda")
    y32 = torch.empty((3, 10, 11, 200), dtype=torch.float32, device="cuda")
    igc.conv2d_nhwc_f16_implicit(dev(x), dev(w), y, y32, pad=(1, 1))
    check_device_ok()
    ref, sabs = oracle.conv2d_nhwc_f16(x, w, pad=(1, 1))
    assert_fp16_bound(host(y32), ref, sabs, f"conv width {width}")
    assert_f16_is_rne_of_f32(host(y), host(y32), f"conv width {width}")


def test_int8_gemm_every_width(width):
    """224 is not built for the integer path: forcing it leaves the choice automatic."""
    rng = np.random.default_rng(width)
    M, N, K = 333, 610, 1104
    A = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    Bt = rng.integers(-128, 128, size=(N, K)).astype(np.int8)
    zA_row = rng.integers(0, 256, size=M).astype(np.int32)
    scale_col = synth.uniform_f32(74, 5, (N,), 1e-5, 1e-4)
    C32 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    C8 = torch.empty((M, N), dtype=torch.int8, device="cuda")
    igc.gemm_s8_zp(dev(A), dev(Bt), zA_row=dev(zA_row), zB=3, C32=C32, C8=C8,
                   scale_col=dev(scale_col))
    check_device_ok()
    o32, o8, _, _ = oracle.gemm_s8_zp(A, Bt, a_signed=0, b_signed=1, zA_row=zA_row, zB=3,
                                      scale_col=scale_col)
    assert np.array_equal(host(C32), o32)
    assert np.array_equal(host(C8), o8)
