"""GPU parity of conv2d_nhwc_s8_zp (int8 implicit-GEMM convolution, zero-point
padding, exact integer tensor-core path, fused requantisation): bit-exact."""

import numpy as np
import pytest
import torch

import implicit_gemm_conv_tcgen05_gb300 as igc
import oracle
from gpu_helpers import check_device_ok, dev, host

pytestmark = pytest.mark.gpu


def _data(N, H, W, C, K, R, S, x_signed, w_signed, seed):
    rng = np.random.default_rng(seed)
    x = (rng.integers(-128, 128, size=(N, H, W, C)).astype(np.int8) if x_signed
         else rng.integers(0, 256, size=(N, H, W, C)).astype(np.uint8))
    w = (rng.integers(-128, 128, size=(K, R, S, C)).astype(np.int8) if w_signed
         else rng.integers(0, 256, size=(K, R, S, C)).astype(np.uint8))
    return x, w, rng


@pytest.mark.parametrize("N,H,W,C,K,R,S,pad,stride,signs", [
    (2, 14, 14, 256, 512, 3, 3, (1, 1), (1, 1), (0, 1)),   # the page's layer, small batch
    (3, 7, 9, 16, 64, 3, 3, (1, 1), (1, 1), (0, 0)),
    (2, 9, 8, 24, 40, 3, 3, (1, 1), (2, 2), (1, 1)),       # stride 2
    (1, 10, 12, 72, 200, 5, 3, (2, 1), (1, 2), (1, 0)),    # rectangular window, mixed strides
    (2, 8, 8, 32, 64, 1, 1, (0, 0), (1, 1), (0, 1)),       # 1x1
    (4, 6, 6, 128, 96, 3, 3, (0, 0), (1, 1), (0, 1)),      # no padding
    (2, 6, 7, 64, 48, 3, 3, (1, 1), (1, 1), (1, 1)),       # int8 input, 4 chunks per pixel
    (1, 5, 5, 512, 32, 3, 3, (1, 1), (1, 1), (1, 0)),      # int8 input, 32 chunks per pixel
    (2, 9, 10, 16, 40, 7, 7, (3, 3), (1, 2), (0, 1)),      # 7x7: window sums by their own pass
])
def test_conv_s8_parity(N, H, W, C, K, R, S, pad, stride, signs):
    x, w, rng = _data(N, H, W, C, K, R, S, *signs, seed=N * 100 + C + K)
    zX = int(rng.integers(-128, 128)) if signs[0] else int(rng.integers(0, 256))
    zW_k = rng.integers(-20, 20, size=K).astype(np.int32)
    scale_k = rng.uniform(1e-5, 1e-3, size=K).astype(np.float32)
    P = (H + 2 * pad[0] - R) // stride[0] + 1
    Q = (W + 2 * pad[1] - S) // stride[1] + 1
    y32 = torch.empty((N, P, Q, K), dtype=torch.int32, device="cuda")
    y8 = torch.empty((N, P, Q, K), dtype=torch.int8, device="cuda")
    igc.conv2d_nhwc_s8_zp(dev(x), dev(w), zX, zW_k=dev(zW_k), y32=y32, y8=y8,
                          scale_k=dev(scale_k), pad=pad, stride=stride)
    check_device_ok()
    o32, o8, ovf = oracle.conv2d_nhwc_s8_zp(x, w, x_signed=signs[0], w_signed=signs[1], zX=zX,
                                            zW_k=zW_k, pad=pad, stride=stride, scale_k=scale_k)
    assert not ovf
    g32, g8 = host(y32), host(y8)
    assert np.count_nonzero(g32 != o32) == 0, "y32 differs"
    assert np.count_nonzero(g8 != o8) == 0, "y8 differs"


def test_conv_s8_constant_zero_point_input_is_zero_at_the_borders():
    x = np.full((2, 14, 14, 64), 77, np.uint8)
    w = np.random.default_rng(1).integers(-128, 128, size=(128, 3, 3, 64)).astype(np.int8)
    y32 = torch.full((2, 14, 14, 128), 5, dtype=torch.int32, device="cuda")
    igc.conv2d_nhwc_s8_zp(dev(x), dev(w), 77, zW=3, y32=y32)
    check_device_ok()
    assert not host(y32).any()
