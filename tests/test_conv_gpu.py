"""GPU parity of conv2d_nhwc_f16_implicit (TMA im2col implicit GEMM on tcgen05)
against the CPU oracle's direct convolution."""

import numpy as np
import pytest
import torch

import implicit_gemm_conv_tcgen05_gb300 as igc
import oracle
import synth
from gpu_helpers import (assert_f16_is_rne_of_f32, assert_fp16_bound, check_device_ok, dev,
                         host)

pytestmark = pytest.mark.gpu


def _gpu(x, w, pad, stride=(1, 1)):
    N, H, W, C = x.shape
    K, R, S, _ = w.shape
    P = (H + 2 * pad[0] - R) // stride[0] + 1
    Q = (W + 2 * pad[1] - S) // stride[1] + 1
    y = torch.empty((N, P, Q, K), dtype=torch.float16, device="cuda")
    y32 = torch.empty((N, P, Q, K), dtype=torch.float32, device="cuda")
    igc.conv2d_nhwc_f16_implicit(dev(x), dev(w), y, y32, pad=pad, stride=stride)
    check_device_ok()
    return host(y), host(y32)


@pytest.mark.parametrize("N,H,W,C,K,R,S,pad", [
    (2, 5, 5, 8, 16, 3, 3, (1, 1)),
    (3, 7, 9, 16, 64, 3, 3, (1, 1)),
    (2, 14, 14, 64, 256, 3, 3, (1, 1)),
    (1, 14, 14, 72, 200, 3, 3, (1, 1)),      # C not a multiple of 64, K not of 256
    (4, 6, 6, 128, 96, 3, 3, (0, 0)),        # no padding: P = Q = 4
    (2, 8, 8, 32, 64, 1, 1, (0, 0)),         # 1x1
    (2, 9, 7, 16, 48, 5, 5, (2, 2)),         # 5x5
    (1, 10, 12, 24, 40, 3, 5, (1, 2)),       # rectangular window, per-axis padding
    (1, 9, 11, 16, 32, 5, 3, (2, 1)),        # the transposed case
    (2, 7, 7, 8, 24, 1, 3, (0, 1)),          # 1x3 window
    (1, 6, 9, 16, 16, 3, 3, (0, 2)),         # padding only along W
    (5, 14, 14, 256, 512, 3, 3, (1, 1)),     # the page's layer, small batch (M tail: 980 pixels)
])
def test_conv_parity(N, H, W, C, K, R, S, pad):
    x = synth.normal_f16(N * 1000 + C, 6, (N, H, W, C))
    w = synth.normal_f16(K * 1000 + R, 7, (K, R, S, C), std=1.0 / np.sqrt(R * S * C))
    y, y32 = _gpu(x, w, pad)
    ref, sabs = oracle.conv2d_nhwc_f16(x, w, pad=pad)
    assert_fp16_bound(y32, ref, sabs, "fp32 copy")
    assert_fp16_bound(y, ref, sabs, "fp16")
    assert_f16_is_rne_of_f32(y, y32, "conv")


def test_delta_kernels_exact():
    x = synth.normal_f16(3, 6, (2, 14, 14, 256))
    w = np.zeros((256, 3, 3, 256), np.float16)
    w[np.arange(256), 1, 1, np.arange(256)] = 1.0
    y, _ = _gpu(x, w, (1, 1))
    assert np.array_equal(y, x)
    w = np.zeros((64, 3, 3, 64), np.float16)
    w[np.arange(64), 0, 0, np.arange(64)] = 1.0
    x = synth.normal_f16(4, 6, (3, 9, 11, 64))
    y, _ = _gpu(x, w, (1, 1))
    want = np.zeros_like(x)
    want[:, 1:, 1:, :] = x[:, :-1, :-1, :]
    assert np.array_equal(y, want)


def test_small_integers_bit_exact():
    rng = np.random.default_rng(5)
    x = rng.integers(-2, 3, size=(3, 14, 14, 128)).astype(np.float16)
    w = rng.integers(-2, 3, size=(256, 3, 3, 128)).astype(np.float16)
    y, y32 = _gpu(x, w, (1, 1))
    ref, _ = oracle.conv2d_nhwc_f16(x, w)
    assert np.array_equal(y32.astype(np.float64), ref)
    assert np.array_equal(y.astype(np.float64), ref)


def test_config4_full_size_sampled_images():
    wl = synth.workload(4)
    x, w = wl["x"], wl["w"]
    y, y32 = _gpu(x, w, (1, 1))
    assert_f16_is_rne_of_f32(y, y32, "conv full")
    imgs = np.array([0, 1, 100, 254, 255])
    ref, sabs = oracle.conv2d_nhwc_f16(x[imgs], w)
    assert_fp16_bound(y32[imgs], ref, sabs, "config 4 fp32")
    assert_fp16_bound(y[imgs], ref, sabs, "config 4 fp16")


def test_unsupported_stride_reports_status():
    x = torch.zeros((1, 8, 8, 16), dtype=torch.float16, device="cuda")
    w = torch.zeros((16, 3, 3, 16), dtype=torch.float16, device="cuda")
    with pytest.raises(igc.IGCError) as e:
        igc.conv2d_nhwc_f16_implicit(x, w, pad=(1, 1), stride=(9, 9))
    assert e.value.status == igc.IGC_ERR_UNSUPPORTED


@pytest.mark.parametrize("N,H,W,C,K,R,S,pad,stride", [
    (2, 14, 14, 64, 128, 3, 3, (1, 1), (2, 2)),
    (2, 9, 11, 16, 48, 3, 3, (1, 0), (2, 1)),
    (1, 15, 15, 32, 64, 5, 5, (2, 2), (3, 3)),
    (3, 28, 28, 128, 96, 3, 3, (1, 1), (2, 2)),      # the strided layer's shape, small batch
    (2, 12, 12, 256, 64, 1, 1, (0, 0), (2, 2)),      # 1x1 stride 2, two channel blocks
    (1, 15, 18, 128, 48, 5, 5, (2, 2), (2, 3)),      # stride 3 along W
    (1, 16, 16, 128, 32, 3, 3, (1, 1), (1, 4)),      # stride 4 along W only
    (2, 10, 12, 128, 40, 3, 2, (0, 0), (2, 2)),      # no padding, even window
    (1, 11, 14, 128, 24, 3, 7, (1, 3), (2, 2)),      # wide window with padding 3
])
def test_conv_strided_parity(N, H, W, C, K, R, S, pad, stride):
    x = synth.normal_f16(N * 77 + C, 6, (N, H, W, C))
    w = synth.normal_f16(K * 77 + R, 7, (K, R, S, C), std=1.0 / np.sqrt(R * S * C))
    y, y32 = _gpu(x, w, pad, stride)
    ref, sabs = oracle.conv2d_nhwc_f16(x, w, pad=pad, stride=stride)
    assert_fp16_bound(y32, ref, sabs, f"stride {stride}")
    assert_f16_is_rne_of_f32(y, y32, "strided conv")
