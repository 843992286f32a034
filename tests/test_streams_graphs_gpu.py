"""The library's calls inside CUDA graphs and on several streams, checked against
the oracle: every kernel is launched with programmatic stream serialization and
waits for its predecessor inside the kernel, so chains of dependent calls
(pre-pass -> GEMM, a call reading the previous call's output) must keep their
order in a graph and on a plain stream alike."""

import numpy as np
import pytest
import torch

import implicit_gemm_conv_tcgen05_gb300 as igc
import oracle
import synth
from gpu_helpers import assert_fp16_bound, check_device_ok, dev, host

pytestmark = pytest.mark.gpu


def _capture(fn, n=1):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()                                   # first call outside the capture (set-up)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for _ in range(n):
                fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    return g


def test_graph_replay_of_int8_gemm_with_new_inputs():
    """gemm_s8_zp (pre-pass + GEMM) captured once; the replay after the inputs
    change must give the oracle's result for the new inputs, bit for bit."""
    M, N, K = 384, 640, 1024
    rng = np.random.default_rng(5)
    A = torch.from_numpy(rng.integers(0, 256, size=(M, K)).astype(np.uint8)).cuda()
    Bt = torch.from_numpy(rng.integers(-128, 128, size=(N, K)).astype(np.int8)).cuda()
    C32 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    C8 = torch.empty((M, N), dtype=torch.int8, device="cuda")
    ws = torch.empty(igc.gemm_s8_zp_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    scale = float(np.float32(2.0 ** -14))
    g = _capture(lambda: igc.gemm_s8_zp(A, Bt, zA=17, zB=-3, C32=C32, C8=C8, scale=scale,
                                        workspace=ws))
    A2 = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    B2 = rng.integers(-128, 128, size=(N, K)).astype(np.int8)
    A.copy_(torch.from_numpy(A2))
    Bt.copy_(torch.from_numpy(B2))
    g.replay()
    check_device_ok()
    o32, o8, _, _ = oracle.gemm_s8_zp(A2, B2, a_signed=0, b_signed=1, zA=17, zB=-3, scale=scale)
    assert np.array_equal(host(C32), o32)
    assert np.array_equal(host(C8), o8)


def test_graph_of_dependent_calls():
    """A graph holding C = A B and then D = C E (the second call reads the first
    call's output) matches the oracle chain."""
    M, K, N, P = 256, 512, 384, 320
    A = synth.uniform_f16(61, 1, (M, K))
    Bt = synth.uniform_f16(61, 2, (N, K))
    Et = synth.uniform_f16(61, 3, (P, N))
    dA, dB, dE = dev(A), dev(Bt), dev(Et)
    C = torch.empty((M, N), dtype=torch.float16, device="cuda")
    D = torch.empty((M, P), dtype=torch.float32, device="cuda")

    def chain():
        igc.gemm_f16(dA, dB, C)
        igc.gemm_f16(C, dE, D)

    C.zero_()
    D.zero_()
    g = _capture(chain)
    D.zero_()
    C.zero_()
    g.replay()
    check_device_ok()
    C_host = host(C)
    ref1, sabs1 = oracle.gemm_f16(A, Bt)
    assert_fp16_bound(C_host.astype(np.float32), ref1, sabs1, "first call")
    ref2, sabs2 = oracle.gemm_f16(C_host, Et)   # the second call consumed the fp16 C
    assert_fp16_bound(host(D), ref2, sabs2, "second call")


def test_back_to_back_calls_on_one_stream_keep_their_order():
    """Many dependent launches queued without synchronisation: each GEMM reads the
    previous one's output (C_{t+1} = C_t * I shifted), so any overlap of a
    kernel with its predecessor's writes would show."""
    n = 256
    P = np.roll(np.eye(n, dtype=np.float16), 1, axis=0)   # a cyclic permutation
    X0 = synth.uniform_f16(62, 1, (n, n))
    bufs = [dev(X0), torch.empty((n, n), dtype=torch.float16, device="cuda")]
    dP = dev(P)
    steps = 40
    for t in range(steps):
        igc.gemm_f16(bufs[t % 2], dP, bufs[(t + 1) % 2])  # C[i,j] = X[i, perm(j)]
    check_device_ok()
    got = host(bufs[steps % 2])
    want = X0.copy()
    perm = np.argmax(P, axis=1)                             # P[j, perm[j]] = 1
    for _ in range(steps):
        want = want[:, perm]
    assert np.array_equal(got, want)


def test_calls_on_two_streams():
    """Independent calls issued on two streams with a cross-stream dependency
    (the second stream's conv reads what the first stream's conv wrote)."""
    x = synth.normal_f16(63, 6, (2, 8, 8, 64))
    w1 = synth.normal_f16(63, 7, (64, 3, 3, 64), std=1.0 / 24)
    w2 = synth.normal_f16(63, 8, (32, 1, 1, 64), std=1.0 / 8)
    dx, dw1, dw2 = dev(x), dev(w1), dev(w2)
    y1 = torch.empty((2, 8, 8, 64), dtype=torch.float16, device="cuda")
    y2 = torch.empty((2, 8, 8, 32), dtype=torch.float32, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s1):
        igc.conv2d_nhwc_f16_implicit(dx, dw1, y1, pad=(1, 1))
    s2.wait_stream(s1)
    with torch.cuda.stream(s2):
        igc.conv2d_nhwc_f16_implicit(y1, dw2, None, y2, pad=(0, 0))
    torch.cuda.current_stream().wait_stream(s2)
    check_device_ok()
    y1h = host(y1)
    ref1, sabs1 = oracle.conv2d_nhwc_f16(x, w1, pad=(1, 1))
    assert_fp16_bound(y1h.astype(np.float32), ref1, sabs1, "first conv")
    ref2, sabs2 = oracle.conv2d_nhwc_f16(y1h, w2, pad=(0, 0))
    assert_fp16_bound(host(y2), ref2, sabs2, "second conv")
