"""Seeded randomized parity sweep: many shapes and parameter combinations per
operation, each compared with the oracle (int8 bit-exact, floating point within
the per-element bound).  Shapes are drawn so that tile widths, the split last
round, ragged edges, strides, zero-point kinds and signedness vary together."""

import numpy as np
import pytest
import torch

import implicit_gemm_conv_tcgen05_gb300 as igc
import oracle
import synth
from gpu_helpers import (assert_f16_is_rne_of_f32, assert_fp16_bound, check_device_ok, dev,
                         host)

pytestmark = pytest.mark.gpu

_RNG = np.random.default_rng(20261202)
_GEMM_F16 = [(int(_RNG.integers(1, 700)), int(_RNG.integers(1, 1300)), 8 * int(_RNG.integers(1, 160)))
             for _ in range(16)]
_GEMM_S8 = [(int(_RNG.integers(1, 600)), int(_RNG.integers(1, 900)), 16 * int(_RNG.integers(1, 100)),
             int(_RNG.integers(0, 2)), int(_RNG.integers(0, 2)), int(_RNG.integers(0, 4)))
            for _ in range(16)]
_CONV = []
while len(_CONV) < 12:
    R, S = int(_RNG.integers(1, 6)), int(_RNG.integers(1, 6))
    ph, pw = int(_RNG.integers(0, R)), int(_RNG.integers(0, S))
    sh, sw = int(_RNG.integers(1, 4)), int(_RNG.integers(1, 4))
    H, W = int(_RNG.integers(R, 16)), int(_RNG.integers(S, 16))
    C = 8 * int(_RNG.integers(1, 24))
    K = 8 * int(_RNG.integers(1, 40))
    N = int(_RNG.integers(1, 4))
    _CONV.append((N, H, W, C, K, R, S, (ph, pw), (sh, sw)))


@pytest.mark.parametrize("M,N,K", _GEMM_F16)
def test_random_gemm_f16(M, N, K):
    A = synth.normal_f16(M * 31 + K, 1, (M, K))
    Bt = synth.normal_f16(N * 37 + K, 2, (N, K))
    C = torch.empty((M, N), dtype=torch.float16, device="cuda")
    C32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    igc.gemm_f16(dev(A), dev(Bt), C, C32)
    check_device_ok()
    ref, sabs = oracle.gemm_f16(A, Bt)
    c32 = host(C32)
    assert_fp16_bound(c32, ref, sabs, f"{M}x{N}x{K}")
    assert_f16_is_rne_of_f32(host(C), c32, f"{M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,a_signed,b_signed,zkind", _GEMM_S8)
def test_random_gemm_s8(M, N, K, a_signed, b_signed, zkind):
    """zkind: 0 per-tensor zero points and scale, 1 per-row zA, 2 per-column zB and
    scale, 3 both vectors."""
    rng = np.random.default_rng(M * 1000 + N * 7 + K)
    A = (rng.integers(-128, 128, size=(M, K)).astype(np.int8) if a_signed
         else rng.integers(0, 256, size=(M, K)).astype(np.uint8))
    Bt = (rng.integers(-128, 128, size=(N, K)).astype(np.int8) if b_signed
          else rng.integers(0, 256, size=(N, K)).astype(np.uint8))
    lo_a, hi_a = (-128, 128) if a_signed else (0, 256)
    lo_b, hi_b = (-128, 128) if b_signed else (0, 256)
    kw = dict(zA=int(rng.integers(lo_a, hi_a)), zB=int(rng.integers(lo_b, hi_b)),
              scale=float(np.float32(2.0 ** -int(rng.integers(8, 16)))))
    if zkind in (1, 3):
        kw["zA_row"] = rng.integers(lo_a, hi_a, size=M).astype(np.int32)
    if zkind in (2, 3):
        kw["zB_col"] = rng.integers(lo_b, hi_b, size=N).astype(np.int32)
        kw["scale_col"] = synth.uniform_f32(M + N, 5, (N,), 1e-6, 1e-3)
    C32 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    C8 = torch.empty((M, N), dtype=torch.int8, device="cuda")
    igc.gemm_s8_zp(dev(A), dev(Bt), zA=kw["zA"], zB=kw["zB"], scale=kw["scale"],
                   zA_row=dev(kw["zA_row"]) if "zA_row" in kw else None,
                   zB_col=dev(kw["zB_col"]) if "zB_col" in kw else None,
                   scale_col=dev(kw["scale_col"]) if "scale_col" in kw else None,
                   C32=C32, C8=C8)
    check_device_ok()
    o32, o8, _, _ = oracle.gemm_s8_zp(A, Bt, a_signed=a_signed, b_signed=b_signed, **kw)
    assert np.array_equal(host(C32), o32)
    assert np.array_equal(host(C8), o8)


@pytest.mark.parametrize("N,H,W,C,K,R,S,pad,stride", _CONV)
def test_random_conv_f16_and_s8(N, H, W, C, K, R, S, pad, stride):
    x = synth.normal_f16(N * 100 + C, 6, (N, H, W, C))
    w = synth.normal_f16(K * 100 + R * 10 + S, 7, (K, R, S, C), std=1.0 / np.sqrt(R * S * C))
    P = (H + 2 * pad[0] - R) // stride[0] + 1
    Q = (W + 2 * pad[1] - S) // stride[1] + 1
    y = torch.empty((N, P, Q, K), dtype=torch.float16, device="cuda")
    y32 = torch.empty((N, P, Q, K), dtype=torch.float32, device="cuda")
    igc.conv2d_nhwc_f16_implicit(dev(x), dev(w), y, y32, pad=pad, stride=stride)
    check_device_ok()
    ref, sabs = oracle.conv2d_nhwc_f16(x, w, pad=pad, stride=stride)
    assert_fp16_bound(host(y32), ref, sabs, "conv f16")
    assert_f16_is_rne_of_f32(host(y), host(y32), "conv f16")

    rng = np.random.default_rng(N * 7 + C + K)
    x8 = rng.integers(0, 256, size=(N, H, W, C)).astype(np.uint8)
    w8 = rng.integers(-128, 128, size=(K, R, S, C)).astype(np.int8)
    zX = int(rng.integers(0, 256))
    zW_k = rng.integers(-30, 30, size=K).astype(np.int32)
    scale_k = rng.uniform(1e-5, 1e-3, size=K).astype(np.float32)
    g32 = torch.empty((N, P, Q, K), dtype=torch.int32, device="cuda")
    g8 = torch.empty((N, P, Q, K), dtype=torch.int8, device="cuda")
    igc.conv2d_nhwc_s8_zp(dev(x8), dev(w8), zX, zW_k=dev(zW_k), y32=g32, y8=g8,
                          scale_k=dev(scale_k), pad=pad, stride=stride)
    check_device_ok()
    o32, o8, _ = oracle.conv2d_nhwc_s8_zp(x8, w8, x_signed=0, w_signed=1, zX=zX, zW_k=zW_k,
                                          pad=pad, stride=stride, scale_k=scale_k)
    assert np.array_equal(host(g32), o32)
    assert np.array_equal(host(g8), o8)


def test_random_sweep_exact_small_integers():
    """A seeded sweep of 150 more cases drawn across operations and forced schedule
    choices (tile width, stage depth, the int8 tensor path): fp16 GEMMs and
    convolutions on small-integer operands, whose sums are exact in fp32, compared
    with the oracle bit for bit; int8 GEMMs bit for bit."""
    rng = np.random.default_rng(20261203)
    done = 0
    while done < 150:
        kind = int(rng.integers(0, 3))
        if kind == 0:
            M, N, K = int(rng.integers(1, 3000)), int(rng.integers(1, 3000)), 8 * int(rng.integers(1, 700))
            if M * N * K > 3e9:
                continue
            A = rng.integers(-2, 3, size=(M, K)).astype(np.float16)
            Bt = rng.integers(-2, 3, size=(N, K)).astype(np.float16)
            w, d = int(rng.choice([0, 0, 0, 128, 224, 256])), int(rng.choice([0, 0, 64, 128]))
            old_w, old_d = igc.igc_set_tile_width(w), igc.igc_set_stage_depth(d)
            try:
                C = torch.empty((M, N), dtype=torch.float32, device="cuda")
                igc.gemm_f16(dev(A), dev(Bt), C)
                check_device_ok()
            finally:
                igc.igc_set_tile_width(old_w)
                igc.igc_set_stage_depth(old_d)
            ref, _ = oracle.gemm_f16(A, Bt)
            assert np.array_equal(host(C), ref.astype(np.float32)), ("f16", M, N, K, w, d)
        elif kind == 1:
            M, N, K = int(rng.integers(1, 2500)), int(rng.integers(1, 2500)), 16 * int(rng.integers(1, 300))
            if M * N * K > 3e9:
                continue
            A = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
            Bt = rng.integers(-128, 128, size=(N, K)).astype(np.int8)
            zA = rng.integers(0, 256, size=M).astype(np.int32)
            zB = int(rng.integers(-128, 128))
            sc = rng.uniform(1e-6, 1e-3, size=N).astype(np.float32)
            w, path = int(rng.choice([0, 0, 128, 256])), int(rng.choice([0, 0, 2, 1]))
            old_w, old_p = igc.igc_set_tile_width(w), igc.igc_set_int8_path(path)
            try:
                C32 = torch.empty((M, N), dtype=torch.int32, device="cuda")
                C8 = torch.empty((M, N), dtype=torch.int8, device="cuda")
                igc.gemm_s8_zp(dev(A), dev(Bt), zA_row=dev(zA), zB=zB, C32=C32, C8=C8,
                               scale_col=dev(sc))
                check_device_ok()
            finally:
                igc.igc_set_tile_width(old_w)
                igc.igc_set_int8_path(old_p)
            o32, o8, _, _ = oracle.gemm_s8_zp(A, Bt, a_signed=0, b_signed=1, zA_row=zA, zB=zB,
                                              scale_col=sc)
            assert np.array_equal(host(C32), o32) and np.array_equal(host(C8), o8), \
                ("s8", M, N, K, w, path)
        else:
            n, H, W = int(rng.integers(1, 5)), int(rng.integers(3, 20)), int(rng.integers(3, 20))
            C, K = 8 * int(rng.integers(1, 40)), 8 * int(rng.integers(1, 64))
            R, S = int(rng.integers(1, 6)), int(rng.integers(1, 6))
            if R > H or S > W:
                continue
            pad = (int(rng.integers(0, R)), int(rng.integers(0, S)))
            stride = (int(rng.integers(1, 3)), int(rng.integers(1, 3)))
            x = rng.integers(-2, 3, size=(n, H, W, C)).astype(np.float16)
            wt = rng.integers(-1, 2, size=(K, R, S, C)).astype(np.float16)
            d, w = int(rng.choice([0, 0, 64])), int(rng.choice([0, 0, 128, 224, 256]))
            old_d, old_w = igc.igc_set_stage_depth(d), igc.igc_set_tile_width(w)
            P = (H + 2 * pad[0] - R) // stride[0] + 1
            Q = (W + 2 * pad[1] - S) // stride[1] + 1
            try:
                y = torch.empty((n, P, Q, K), dtype=torch.float16, device="cuda")
                y32 = torch.empty((n, P, Q, K), dtype=torch.float32, device="cuda")
                igc.conv2d_nhwc_f16_implicit(dev(x), dev(wt), y, y32, pad=pad, stride=stride)
                check_device_ok()
            finally:
                igc.igc_set_stage_depth(old_d)
                igc.igc_set_tile_width(old_w)
            ref, _ = oracle.conv2d_nhwc_f16(x, wt, pad=pad, stride=stride)
            assert np.array_equal(host(y32), ref.astype(np.float32)), \
                ("conv", n, H, W, C, K, R, S, pad, stride, d, w)
        done += 1


def _forced(width=None, depth=None, int8_path=None):
    """Sets the calling thread's schedule hooks; returns a function that restores them."""
    old = []
    if width is not None:
        old.append((igc.igc_set_tile_width, igc.igc_set_tile_width(width)))
    if depth is not None:
        old.append((igc.igc_set_stage_depth, igc.igc_set_stage_depth(depth)))
    if int8_path is not None:
        old.append((igc.igc_set_int8_path, igc.igc_set_int8_path(int8_path)))

    def restore():
        for setter, value in old:
            setter(value)
    return restore


def _stress_gemm_float(rng):
    M, N, K = int(rng.integers(1, 5000)), int(rng.integers(1, 5000)), 8 * int(rng.integers(1, 900))
    if M * N * K > 4e9:
        return None
    A = rng.integers(-2, 3, size=(M, K)).astype(np.float16)
    Bt = rng.integers(-2, 3, size=(N, K)).astype(np.float16)
    width, depth = int(rng.choice([0, 0, 128, 224, 256])), int(rng.choice([0, 0, 64, 128]))
    bf16 = bool(rng.integers(0, 2))
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    restore = _forced(width, depth)
    try:
        if bf16:
            igc.gemm_bf16(dev(A).to(torch.bfloat16), dev(Bt).to(torch.bfloat16), C)
        else:
            igc.gemm_f16(dev(A), dev(Bt), C)
        check_device_ok()
    finally:
        restore()
    ref, _ = oracle.gemm_f16(A, Bt)   # small integers: the same exact sums in either type
    assert np.array_equal(host(C), ref.astype(np.float32)), ("float", bf16, M, N, K, width, depth)
    return "bf16" if bf16 else "f16"


def _stress_gemm_s8(rng):
    M, N, K = int(rng.integers(1, 4500)), int(rng.integers(1, 4500)), 16 * int(rng.integers(1, 400))
    if M * N * K > 4e9:
        return None
    a_s, b_s = int(rng.integers(0, 2)), int(rng.integers(0, 2))
    A = (rng.integers(-128, 128, size=(M, K)).astype(np.int8) if a_s
         else rng.integers(0, 256, size=(M, K)).astype(np.uint8))
    Bt = (rng.integers(-128, 128, size=(N, K)).astype(np.int8) if b_s
          else rng.integers(0, 256, size=(N, K)).astype(np.uint8))
    zA = rng.integers(-200, 256, size=M).astype(np.int32)
    zB = rng.integers(-200, 256, size=N).astype(np.int32)
    sc = rng.uniform(1e-7, 1e-4, size=N).astype(np.float32)
    width, path = int(rng.choice([0, 0, 128, 256])), int(rng.choice([0, 0, 1, 2, 3]))
    C32 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    C8 = torch.empty((M, N), dtype=torch.int8, device="cuda")
    restore = _forced(width, int8_path=path)
    try:
        igc.gemm_s8_zp(dev(A), dev(Bt), zA_row=dev(zA), zB_col=dev(zB), C32=C32, C8=C8,
                       scale_col=dev(sc))
        check_device_ok()
    finally:
        restore()
    o32, o8, _, _ = oracle.gemm_s8_zp(A, Bt, a_signed=a_s, b_signed=b_s, zA_row=zA, zB_col=zB,
                                      scale_col=sc)
    assert np.array_equal(host(C32), o32) and np.array_equal(host(C8), o8), \
        ("s8", M, N, K, a_s, b_s, width, path)
    return f"s8 path {path}"


def _conv_shape(rng, max_n, max_hw, max_k):
    n = int(rng.integers(1, max_n))
    H, W = int(rng.integers(3, max_hw)), int(rng.integers(3, max_hw))
    C, K = 8 * int(rng.integers(1, 40)), 8 * int(rng.integers(1, max_k))
    R, S = int(rng.integers(1, 8)), int(rng.integers(1, 8))
    if R > H or S > W:
        return None
    pad = (int(rng.integers(0, R)), int(rng.integers(0, S)))
    stride = (int(rng.integers(1, 4)), int(rng.integers(1, 4)))
    P = (H + 2 * pad[0] - R) // stride[0] + 1
    Q = (W + 2 * pad[1] - S) // stride[1] + 1
    return n, H, W, C, K, R, S, pad, stride, P, Q


def _stress_conv_f16(rng):
    shape = _conv_shape(rng, 5, 24, 64)
    if shape is None:
        return None
    n, H, W, C, K, R, S, pad, stride, P, Q = shape
    x = rng.integers(-2, 3, size=(n, H, W, C)).astype(np.float16)
    wt = rng.integers(-1, 2, size=(K, R, S, C)).astype(np.float16)
    depth, width = int(rng.choice([0, 0, 64])), int(rng.choice([0, 0, 128, 224, 256]))
    y32 = torch.empty((n, P, Q, K), dtype=torch.float32, device="cuda")
    restore = _forced(width, depth)
    try:
        igc.conv2d_nhwc_f16_implicit(dev(x), dev(wt), None, y32, pad=pad, stride=stride)
        check_device_ok()
    finally:
        restore()
    ref, _ = oracle.conv2d_nhwc_f16(x, wt, pad=pad, stride=stride)
    assert np.array_equal(host(y32), ref.astype(np.float32)), ("conv", shape, depth, width)
    return "conv f16"


def _stress_conv_s8(rng):
    shape = _conv_shape(rng, 4, 20, 48)
    if shape is None:
        return None
    n, H, W, C, K, R, S, pad, stride, P, Q = shape
    xs, ws = int(rng.integers(0, 2)), int(rng.integers(0, 2))
    x8 = (rng.integers(-128, 128, size=(n, H, W, C)).astype(np.int8) if xs
          else rng.integers(0, 256, size=(n, H, W, C)).astype(np.uint8))
    w8 = (rng.integers(-128, 128, size=(K, R, S, C)).astype(np.int8) if ws
          else rng.integers(0, 256, size=(K, R, S, C)).astype(np.uint8))
    zX = int(rng.integers(-128, 128)) if xs else int(rng.integers(0, 256))
    zW_k = rng.integers(-60, 60, size=K).astype(np.int32)
    scale_k = rng.uniform(1e-6, 1e-3, size=K).astype(np.float32)
    g32 = torch.empty((n, P, Q, K), dtype=torch.int32, device="cuda")
    g8 = torch.empty((n, P, Q, K), dtype=torch.int8, device="cuda")
    width = int(rng.choice([0, 0, 128, 256]))
    restore = _forced(width)
    try:
        igc.conv2d_nhwc_s8_zp(dev(x8), dev(w8), zX, zW_k=dev(zW_k), y32=g32, y8=g8,
                              scale_k=dev(scale_k), pad=pad, stride=stride)
        check_device_ok()
    finally:
        restore()
    o32, o8, _ = oracle.conv2d_nhwc_s8_zp(x8, w8, x_signed=xs, w_signed=ws, zX=zX, zW_k=zW_k,
                                          pad=pad, stride=stride, scale_k=scale_k)
    assert np.array_equal(host(g32), o32) and np.array_equal(host(g8), o8), \
        ("conv s8", shape, xs, ws, width)
    return "conv s8"


def test_random_stress_all_paths():
    """400 more seeded cases across every operation, path and forced schedule: fp16 and
    bf16 GEMMs and fp16 convolutions on small-integer operands (exact in fp32, so
    compared bit for bit), int8 GEMMs on all four paths with per-row and per-column
    zero points and per-column scales, and int8 convolutions in all signedness
    combinations with per-channel weight zero points, windows up to 7 x 7 and strides
    up to 3, compared bit for bit with the oracle."""
    rng = np.random.default_rng(20261204)
    kinds = (_stress_gemm_float, _stress_gemm_s8, _stress_conv_f16, _stress_conv_s8)
    seen = {}
    while sum(seen.values()) < 400:
        key = kinds[int(rng.integers(0, len(kinds)))](rng)
        if key is not None:
            seen[key] = seen.get(key, 0) + 1
    assert len(seen) == 8, seen     # every kind and every int8 path came up
