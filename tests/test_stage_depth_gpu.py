"""GPU parity of the fp16 / bf16 GEMMs with each pipeline stage depth forced
(igc_set_stage_depth: 64-deep stages, twice as many, or the default 128) and
each tile width, and at shapes whose automatic choice takes 64-deep stages (at
most two rounds of tiles filling at least a quarter of the CTA pairs, K >=
2048).  K values leave a partial last stage."""

import numpy as np
import pytest
import torch

import implicit_gemm_conv_tcgen05_gb300 as igc
import oracle
import synth
from gpu_helpers import (assert_f16_is_rne_of_f32, assert_fp16_bound, check_device_ok, dev,
                         host)

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[64, 128])
def depth(request):
    old = igc.igc_set_stage_depth(request.param)
    yield request.param
    igc.igc_set_stage_depth(old)


@pytest.mark.parametrize("width", [128, 224, 256])
@pytest.mark.parametrize("M,N,K", [(300, 470, 136), (513, 1000, 2056), (64, 2000, 1032),
                                   (2560, 2048, 72)])
def test_gemm_f16_every_depth(depth, width, M, N, K):
    old = igc.igc_set_tile_width(width)
    try:
        A = synth.normal_f16(M + 11, 1, (M, K))
        Bt = synth.normal_f16(N + 11, 2, (N, K))
        C = torch.empty((M, N), dtype=torch.float16, device="cuda")
        C32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
        igc.gemm_f16(dev(A), dev(Bt), C, C32)
        check_device_ok()
    finally:
        igc.igc_set_tile_width(old)
    ref, sabs = oracle.gemm_f16(A, Bt)
    c32 = host(C32)
    assert_fp16_bound(c32, ref, sabs, f"depth {depth} width {width}")
    assert_f16_is_rne_of_f32(host(C), c32, f"depth {depth} width {width}")


def test_gemm_bf16_every_depth(depth):
    M, N, K = 384, 900, 2100 - 2100 % 8
    Ab = synth.normal_bf16_bits(75, 1, (M, K))
    Bb = synth.normal_bf16_bits(75, 2, (N, K))
    A = torch.from_numpy(Ab.view(np.int16)).cuda().view(torch.bfloat16)
    Bt = torch.from_numpy(Bb.view(np.int16)).cuda().view(torch.bfloat16)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    C32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    igc.gemm_bf16(A, Bt, C, C32)
    check_device_ok()
    ref, sabs = oracle.gemm_bf16(Ab, Bb)
    c32 = host(C32)
    assert_fp16_bound(c32, ref, sabs, f"bf16 depth {depth}")
    want = oracle.f32_to_bf16_bits_array(c32)
    got = C.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("M,N,K", [(768, 2048, 2048), (700, 3000, 4096 + 64)])
def test_gemm_f16_automatic_deep_stages(M, N, K):
    """Few tiles over a long k: the automatic choice is 64-deep stages; the small
    integers make every sum exact, so the result must equal the oracle's bit for bit."""
    assert igc.igc_set_stage_depth(0) == 0
    rng = np.random.default_rng(M + K)
    A = rng.integers(-2, 3, size=(M, K)).astype(np.float16)
    Bt = rng.integers(-2, 3, size=(N, K)).astype(np.float16)
    C32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    igc.gemm_f16(dev(A), dev(Bt), C32)
    check_device_ok()
    ref, _ = oracle.gemm_f16(A, Bt)
    assert np.array_equal(host(C32), ref.astype(np.float32))


@pytest.mark.parametrize("N,H,W,C,K,R,S,pad,stride", [
    (3, 10, 11, 64, 200, 3, 3, (1, 1), (1, 1)),
    (2, 9, 9, 72, 96, 3, 3, (1, 1), (1, 1)),     # C not a multiple of 64: zero-filled channels
    (2, 12, 13, 136, 64, 5, 3, (2, 1), (2, 1)),
    (4, 14, 14, 256, 512, 3, 3, (1, 1), (1, 1)),
])
def test_conv_f16_every_depth(depth, N, H, W, C, K, R, S, pad, stride):
    x = synth.normal_f16(N * 31 + C, 6, (N, H, W, C))
    w = synth.normal_f16(K * 31 + R, 7, (K, R, S, C), std=1.0 / np.sqrt(R * S * C))
    P = (H + 2 * pad[0] - R) // stride[0] + 1
    Q = (W + 2 * pad[1] - S) // stride[1] + 1
    y = torch.empty((N, P, Q, K), dtype=torch.float16, device="cuda")
    y32 = torch.empty((N, P, Q, K), dtype=torch.float32, device="cuda")
    igc.conv2d_nhwc_f16_implicit(dev(x), dev(w), y, y32, pad=pad, stride=stride)
    check_device_ok()
    ref, sabs = oracle.conv2d_nhwc_f16(x, w, pad=pad, stride=stride)
    assert_fp16_bound(host(y32), ref, sabs, f"conv depth {depth}")
    assert_f16_is_rne_of_f32(host(y), host(y32), f"conv depth {depth}")
