"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test here would fail for a plausible mistake in the oracle: a dropped
term, a sign or index error, a transposed operand, a wrong rounding rule.
The references are closed forms, exact integer arithmetic, hand-computed
tables (tests/golden/), numpy's IEEE conversions, float64 library routines
on tiny shapes, and the shapes / index constant the convolution page prints.
"""

import os
import struct

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import GOLDEN, read_kv

RNG = np.random.default_rng(12345)


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def test_f16_decode_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def _f32_samples():
    raw = RNG.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    # values around the fp16 range, including subnormal and overflow boundaries
    exps = RNG.integers(-30, 18, size=200_000)
    mant = RNG.random(200_000) + 1.0
    sgn = np.where(RNG.random(200_000) < 0.5, -1.0, 1.0)
    near = (sgn * mant * np.exp2(exps)).astype(np.float32)
    edge = np.array([0.0, -0.0, 65504.0, 65519.996, 65520.0, 65536.0, 1e30, -1e30,
                     2.0**-24, 2.0**-25, 3 * 2.0**-26, 2.0**-25 * 1.0000001, 2.0**-14,
                     2.0**-14 - 2.0**-25, 1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11, np.inf, -np.inf,
                     1e-45, -1e-45], dtype=np.float32)
    return np.concatenate([raw, near, edge])


def test_f32_to_f16_rne_matches_ieee_conversion():
    x = _f32_samples()
    got = oracle.f32_to_f16_array(x).view(np.uint16)
    with np.errstate(over="ignore", invalid="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all(np.isnan(got[nan].view(np.float16)))


def test_i32_to_f32_rne_matches_ieee_conversion():
    v = np.concatenate([
        RNG.integers(-2**31, 2**31, size=100_000, dtype=np.int64),
        np.array([0, 1, -1, 2**24 - 1, 2**24, 2**24 + 1, 2**24 + 2, 2**24 + 3, -(2**24 + 1),
                  2**25 + 2, 2**25 + 6, 2**31 - 1, -2**31, -2**31 + 1, 2**30 + 64, 2**30 + 192]),
    ]).astype(np.int32)
    want = v.astype(np.float32)
    got = np.array([oracle.i32_to_f32(int(a)) for a in v], dtype=np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_requant_hand_table():
    path = os.path.join(GOLDEN, "requant_cases.txt")
    n = 0
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            c32, sbits, expected = line.split()[:3]
            scale = struct.unpack("<f", struct.pack("<I", int(sbits, 16)))[0]
            assert oracle.requant(int(c32), scale) == int(expected), line
            n += 1
    assert n >= 20


# ---------------------------------------------------------------------------
# fp16 GEMM
# ---------------------------------------------------------------------------

def test_gemm_identity_left_and_right():
    n = 96
    B = synth.uniform_f16(7, 2, (n, n))
    eye = np.eye(n, dtype=np.float16)
    ref, _ = oracle.gemm_f16(eye, B)                 # C[i,j] = Bt[j,i]
    assert np.array_equal(ref, B.astype(np.float64).T)
    ref, _ = oracle.gemm_f16(B, eye)                 # C[i,j] = A[i,j]
    assert np.array_equal(ref, B.astype(np.float64))


def test_gemm_permutation():
    M, K, N = 40, 40, 24
    perm = RNG.permutation(K)
    Pm = np.zeros((M, K), np.float16)
    Pm[np.arange(M), perm] = 1.0
    Bt = synth.normal_f16(3, 2, (N, K))
    ref, sabs = oracle.gemm_f16(Pm, Bt)
    # row i of C is column perm[i] of Bt, i.e. Bt[:, perm[i]]
    assert np.array_equal(ref, Bt.astype(np.float64)[:, perm].T)
    assert np.array_equal(sabs, np.abs(Bt.astype(np.float64))[:, perm].T)


def test_gemm_small_integers_exact():
    M, N, K = 37, 53, 515
    A = RNG.integers(-2, 3, size=(M, K))
    Bt = RNG.integers(-2, 3, size=(N, K))
    ref, sabs = oracle.gemm_f16(A.astype(np.float16), Bt.astype(np.float16))
    assert np.array_equal(ref, (A @ Bt.T).astype(np.float64))
    assert np.array_equal(sabs, (np.abs(A) @ np.abs(Bt).T).astype(np.float64))


def test_gemm_random_vs_float64_matmul():
    M, N, K = 33, 65, 130
    A = synth.uniform_f16(11, 1, (M, K))
    Bt = synth.uniform_f16(11, 2, (N, K))
    ref, _ = oracle.gemm_f16(A, Bt)
    want = (torch.from_numpy(A.astype(np.float64)) @ torch.from_numpy(Bt.astype(np.float64)).T).numpy()
    assert np.allclose(ref, want, rtol=0, atol=1e-12)


def test_gemm_rectangular_not_transposed():
    # distinguishes A @ Bt.T from A @ Bt or A.T @ ...: shapes would not even agree
    A = np.arange(6, dtype=np.float16).reshape(2, 3)
    Bt = np.array([[1, 0, 0], [0, 0, 1], [1, 1, 1], [0, 2, 0]], dtype=np.float16)
    ref, _ = oracle.gemm_f16(A, Bt)
    assert ref.tolist() == [[0, 2, 3, 2], [3, 5, 12, 8]]


# ---------------------------------------------------------------------------
# int8 GEMM with zero points
# ---------------------------------------------------------------------------

def _expanded(A, Bt, zA, zB):
    """sum A_q B_q - zB rowsum(A_q) - zA colsum(B_q) + K zA zB, in int64."""
    K = A.shape[1]
    A = A.astype(np.int64)
    Bt = Bt.astype(np.int64)
    zA = np.asarray(zA, np.int64).reshape(-1, 1)
    zB = np.asarray(zB, np.int64).reshape(1, -1)
    return A @ Bt.T - zB * A.sum(1, keepdims=True) - zA * Bt.sum(1)[None, :] + K * zA * zB


@pytest.mark.parametrize("a_signed,b_signed", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_zero_point_expansion_identity(a_signed, b_signed):
    M, N, K = 29, 41, 333
    lo_a, hi_a = (-128, 127) if a_signed else (0, 255)
    lo_b, hi_b = (-128, 127) if b_signed else (0, 255)
    A = RNG.integers(lo_a, hi_a + 1, size=(M, K)).astype(np.int8 if a_signed else np.uint8)
    Bt = RNG.integers(lo_b, hi_b + 1, size=(N, K)).astype(np.int8 if b_signed else np.uint8)
    zA_row = RNG.integers(-20, 200, size=M).astype(np.int32)
    zB_col = RNG.integers(-20, 200, size=N).astype(np.int32)
    C32, _, C64, ovf = oracle.gemm_s8_zp(A, Bt, a_signed=a_signed, b_signed=b_signed,
                                         zA_row=zA_row, zB_col=zB_col, want_c8=False, want_c64=True)
    assert not ovf
    assert np.array_equal(C64, _expanded(A, Bt, zA_row, zB_col))
    assert np.array_equal(C32.astype(np.int64), C64)
    # per-tensor zero points
    C32, _, C64, _ = oracle.gemm_s8_zp(A, Bt, a_signed=a_signed, b_signed=b_signed,
                                       zA=77, zB=-5, want_c8=False, want_c64=True)
    assert np.array_equal(C64, _expanded(A, Bt, np.full(M, 77), np.full(N, -5)))


def test_zero_points_zero_is_plain_integer_gemm():
    A = RNG.integers(0, 256, size=(19, 70)).astype(np.uint8)
    Bt = RNG.integers(-128, 128, size=(23, 70)).astype(np.int8)
    C32, _, _, _ = oracle.gemm_s8_zp(A, Bt, a_signed=0, b_signed=1, want_c8=False)
    assert np.array_equal(C32, (A.astype(np.int64) @ Bt.astype(np.int64).T).astype(np.int32))


def test_signedness_matters():
    # byte 0xFF is 255 unsigned and -1 signed
    A = np.full((1, 4), 0xFF, np.uint8)
    Bt = np.full((1, 4), 1, np.uint8)
    assert oracle.gemm_s8_zp(A, Bt, a_signed=0, b_signed=0, want_c8=False)[0][0, 0] == 1020
    assert oracle.gemm_s8_zp(A, Bt, a_signed=1, b_signed=0, want_c8=False)[0][0, 0] == -4


def test_int32_overflow_flag_and_wrap():
    K = 40000                                     # 255 * 255 * 40000 > 2^31
    A = np.full((1, K), 255, np.uint8)
    Bt = np.full((1, K), 255, np.uint8)
    C32, _, C64, ovf = oracle.gemm_s8_zp(A, Bt, a_signed=0, b_signed=0, want_c8=False, want_c64=True)
    assert ovf
    assert C64[0, 0] == 255 * 255 * K
    assert C32[0, 0] == np.int64(C64[0, 0]).astype(np.int32)  # two's complement wrap


def test_requant_in_gemm_uses_per_column_scale():
    A = np.array([[1, 2, 3, 4]], np.uint8)
    Bt = np.array([[1, 1, 1, 1], [2, 2, 2, 2]], np.uint8)       # C32 = 10, 20
    _, C8, _, _ = oracle.gemm_s8_zp(A, Bt, a_signed=0, b_signed=0,
                                    scale_col=np.array([0.25, 0.125], np.float32))
    assert C8.tolist() == [[2, 2]]                              # 2.5 -> 2, 2.5 -> 2
    _, C8, _, _ = oracle.gemm_s8_zp(A, Bt, a_signed=0, b_signed=0, scale=0.35)
    assert C8.tolist() == [[4, 7]]                              # 3.5 -> 4, 7.0 -> 7


# ---------------------------------------------------------------------------
# convolution
# ---------------------------------------------------------------------------

def test_conv_page_shapes():
    g = read_kv(os.path.join(GOLDEN, "conv_page_shapes.txt"))
    n, h, w, c, k, r = (g["batch"], g["height"], g["width"], g["in_channels"],
                        g["out_channels"], g["kernel"])
    P = oracle.conv_out_dim(h, r, g["pad"], g["stride"])
    Q = oracle.conv_out_dim(w, r, g["pad"], g["stride"])
    assert n * h * w * c == g["A_elements"]
    assert r * r * c * k == g["W_elements"]
    assert n * P * Q * k == g["Conv_elements"]
    # blocked layout strides printed by the page follow from the shape
    b = g["block"]
    assert g["A_stride_w"] == (c // b) * b * b
    assert g["A_stride_h"] == w * g["A_stride_w"]


def test_conv_tap_offset_matches_page_index_constant():
    """The page reads Apad tap (kh, kw) of output (p, q) at flattened offset
    kh*stride_h + kw*stride_w - 61440 relative to pixel (p, q): the input pixel
    is (p + kh - 1, q + kw - 1).  Check the oracle uses the same convention by
    a single-impulse experiment for every tap."""
    g = read_kv(os.path.join(GOLDEN, "conv_page_shapes.txt"))
    off = -g["A_index_offset"]
    pad_h, rem = divmod(off, g["A_stride_h"])
    pad_w, rem = divmod(rem, g["A_stride_w"])
    assert (pad_h, pad_w, rem) == (g["pad"], g["pad"], 0)
    H = W = 6
    C = K = 8
    for kh in range(3):
        for kw in range(3):
            x = np.zeros((1, H, W, C), np.float16)
            x[0, 3, 2, 5] = 1.0
            wt = np.zeros((K, 3, 3, C), np.float16)
            wt[4, kh, kw, 5] = 1.0
            ref, _ = oracle.conv2d_nhwc_f16(x, wt, pad=(pad_h, pad_w))
            nz = np.argwhere(ref != 0)
            # input pixel (3, 2) = (p + kh - pad_h, q + kw - pad_w)
            assert nz.tolist() == [[0, 3 - kh + pad_h, 2 - kw + pad_w, 4]]


def test_conv_delta_center_is_identity():
    x = synth.normal_f16(5, 6, (2, 7, 9, 16))
    w = np.zeros((16, 3, 3, 16), np.float16)
    w[np.arange(16), 1, 1, np.arange(16)] = 1.0
    ref, _ = oracle.conv2d_nhwc_f16(x, w)
    assert np.array_equal(ref, x.astype(np.float64))


def test_conv_delta_corner_is_shifted_copy():
    x = synth.normal_f16(5, 6, (2, 7, 9, 8))
    w = np.zeros((8, 3, 3, 8), np.float16)
    w[np.arange(8), 0, 0, np.arange(8)] = 1.0
    ref, _ = oracle.conv2d_nhwc_f16(x, w)
    want = np.zeros_like(ref)
    want[:, 1:, 1:, :] = x.astype(np.float64)[:, :-1, :-1, :]
    assert np.array_equal(ref, want)


def test_conv_delta_full_size_channels():
    # the page's channel count and spatial size, small batch
    x = synth.normal_f16(9, 6, (1, 14, 14, 256))
    w = np.zeros((256, 3, 3, 256), np.float16)
    w[np.arange(256), 1, 1, np.arange(256)] = 1.0
    ref, _ = oracle.conv2d_nhwc_f16(x, w)
    assert np.array_equal(ref, x.astype(np.float64))


def test_conv_1x1_equals_gemm():
    x = synth.normal_f16(4, 6, (3, 5, 6, 24))
    w = synth.normal_f16(4, 7, (40, 1, 1, 24))
    ref, sabs = oracle.conv2d_nhwc_f16(x, w, pad=(0, 0))
    g_ref, g_sabs = oracle.gemm_f16(x.reshape(-1, 24), w.reshape(40, 24))
    assert np.array_equal(ref.reshape(-1, 40), g_ref)
    assert np.array_equal(sabs.reshape(-1, 40), g_sabs)


def _im2col_conv(x, w, pad, stride):
    """Test-only brute force: explicit zero-padded im2col matrix times weights."""
    N, H, W, C = x.shape
    K, R, S, _ = w.shape
    xp = np.zeros((N, H + 2 * pad[0], W + 2 * pad[1], C), np.float64)
    xp[:, pad[0]:pad[0] + H, pad[1]:pad[1] + W, :] = x
    P = (H + 2 * pad[0] - R) // stride[0] + 1
    Q = (W + 2 * pad[1] - S) // stride[1] + 1
    cols = np.zeros((N, P, Q, R, S, C))
    for p in range(P):
        for q in range(Q):
            cols[:, p, q] = xp[:, p * stride[0]:p * stride[0] + R, q * stride[1]:q * stride[1] + S, :]
    return cols.reshape(N * P * Q, R * S * C) @ w.astype(np.float64).reshape(K, -1).T, (N, P, Q, K)


@pytest.mark.parametrize("pad,stride", [((0, 0), (1, 1)), ((1, 1), (1, 1)), ((2, 2), (1, 1)),
                                        ((1, 1), (2, 2)), ((0, 2), (2, 1)), ((2, 1), (1, 2))])
def test_conv_brute_force_im2col(pad, stride):
    x = RNG.integers(-3, 4, size=(2, 5, 5, 8)).astype(np.float16)
    w = RNG.integers(-3, 4, size=(16, 3, 3, 8)).astype(np.float16)
    ref, _ = oracle.conv2d_nhwc_f16(x, w, pad=pad, stride=stride)
    want, shape = _im2col_conv(x.astype(np.float64), w, pad, stride)
    assert ref.shape == shape
    assert np.array_equal(ref.reshape(-1, 16), want)


@pytest.mark.parametrize("pad,stride", [((1, 1), (1, 1)), ((0, 1), (2, 1))])
def test_conv_vs_float64_library_conv2d(pad, stride):
    x = synth.normal_f16(21, 6, (2, 9, 8, 16))
    w = synth.normal_f16(21, 7, (12, 3, 3, 16), std=0.25)
    ref, _ = oracle.conv2d_nhwc_f16(x, w, pad=pad, stride=stride)
    xt = torch.from_numpy(x.astype(np.float64)).permute(0, 3, 1, 2)
    wt = torch.from_numpy(w.astype(np.float64)).permute(0, 3, 1, 2)
    want = torch.nn.functional.conv2d(xt, wt, padding=pad, stride=stride).permute(0, 2, 3, 1).numpy()
    assert np.allclose(ref, want, rtol=0, atol=1e-12)


def test_conv_sabs_is_abs_conv():
    x = synth.normal_f16(2, 6, (1, 6, 6, 8))
    w = synth.normal_f16(2, 7, (4, 3, 3, 8))
    _, sabs = oracle.conv2d_nhwc_f16(x, w)
    ref_abs, _ = oracle.conv2d_nhwc_f16(np.abs(x), np.abs(w))
    assert np.array_equal(sabs, ref_abs)


# ---------------------------------------------------------------------------
# the generators the parity tests draw from
# ---------------------------------------------------------------------------

def test_generators_are_counter_based_and_in_range():
    a = synth.uniform_int(1, 1, (1000,), 0, 255, np.uint8)
    b = synth.uniform_int(1, 1, (2000,), 0, 255, np.uint8)
    assert np.array_equal(a, b[:1000])
    assert a.min() == 0 and a.max() == 255
    s = synth.uniform_int(2, 2, (100000,), -127, 127, np.int8)
    assert s.min() == -127 and s.max() == 127
    z = synth.uniform_int(3, 3, (5000,), 100, 156, np.int32)
    assert z.min() == 100 and z.max() == 156
    n = synth.normal_f16(4, 4, (200000,)).astype(np.float64)
    assert abs(n.mean()) < 0.01 and abs(n.std() - 1) < 0.01
    u = synth.uniform_f16(4, 5, (100000,)).astype(np.float64)
    assert u.min() >= -1 and u.max() <= 1 and abs(u.mean()) < 0.01
    sc = synth.uniform_f32(4, 6, (10000,), 1e-4, 1e-3)
    assert sc.dtype == np.float32 and sc.min() >= np.float32(1e-4) and sc.max() <= np.float32(1e-3)


# ---------------------------------------------------------------------------
# bf16 (the f16 -> bf16 swap of the GEMM)
# ---------------------------------------------------------------------------

def _bits_to_bf16_tensor(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)


def test_bf16_decode_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = _bits_to_bf16_tensor(bits).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_f32_to_bf16_rne_matches_library_conversion():
    x = _f32_samples()
    got = oracle.f32_to_bf16_bits_array(x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all(np.isnan(_bits_to_bf16_tensor(got[nan]).to(torch.float32).numpy()))


def test_gemm_bf16_exact_cases_and_float64_matmul():
    rng = np.random.default_rng(3)
    M, N, K = 37, 45, 300
    A = rng.integers(-3, 4, size=(M, K))
    Bt = rng.integers(-3, 4, size=(N, K))
    to_bits = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    ref, sabs = oracle.gemm_bf16(to_bits(A), to_bits(Bt))
    assert np.array_equal(ref, (A @ Bt.T).astype(np.float64))
    assert np.array_equal(sabs, (np.abs(A) @ np.abs(Bt).T).astype(np.float64))
    eye = np.eye(64)
    B = synth.normal_bf16_bits(4, 2, (64, 64))
    ref, _ = oracle.gemm_bf16(to_bits(eye), B)
    assert np.array_equal(ref, _bits_to_bf16_tensor(B).to(torch.float64).numpy().T)
    A2 = synth.normal_bf16_bits(5, 1, (19, 70))
    B2 = synth.normal_bf16_bits(5, 2, (23, 70))
    ref, _ = oracle.gemm_bf16(A2, B2)
    want = (_bits_to_bf16_tensor(A2).double() @ _bits_to_bf16_tensor(B2).double().T).numpy()
    assert np.allclose(ref, want, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# dequantised float output (four-term fusion)
# ---------------------------------------------------------------------------

def _f32_from_bits(h):
    return struct.unpack("<f", struct.pack("<I", int(h, 16)))[0]


def test_dequant_hand_table():
    n = 0
    with open(os.path.join(GOLDEN, "dequant_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            c32, sr, sc, b, want = line.split()[:5]
            args = [None if v == "-" else _f32_from_bits(v) for v in (sr, sc, b)]
            got = oracle.dequant(int(c32), *args)
            assert struct.pack("<f", got) == struct.pack("<I", int(want, 16)), line
            n += 1
    assert n >= 7


def test_dequant_closed_forms():
    rng = np.random.default_rng(8)
    C32 = rng.integers(-2**23, 2**23, size=(7, 11)).astype(np.int32)
    # no steps: exactly the int32 values (all below 2^24)
    assert np.array_equal(oracle.dequant_matrix(C32), C32.astype(np.float32))
    # power-of-two scales: exact scaling; small-integer bias: exact shift
    s_row = np.exp2(rng.integers(-8, 3, size=7)).astype(np.float32)
    s_col = np.exp2(rng.integers(-8, 3, size=11)).astype(np.float32)
    bias = rng.integers(-100, 100, size=11).astype(np.float32)
    want = (C32.astype(np.float64) * s_row[:, None] * s_col[None, :]) + bias[None, :]
    got = oracle.dequant_matrix(C32, s_row, s_col, bias)
    exact = np.abs(want) < 2**24
    assert np.array_equal(got[exact].astype(np.float64), want[exact])


# ---------------------------------------------------------------------------
# int8 convolution with zero points (padding value = zX)
# ---------------------------------------------------------------------------

def test_conv_s8_constant_zero_point_input_gives_zero_everywhere():
    # with zero padding the border outputs would be (0 - zX)(w - zW) != 0
    x = np.full((2, 6, 7, 8), 37, np.uint8)
    w = RNG.integers(-128, 128, size=(5, 3, 3, 8)).astype(np.int8)
    y32, _, _ = oracle.conv2d_nhwc_s8_zp(x, w, x_signed=0, w_signed=1, zX=37, zW=3, pad=(1, 1),
                                         want_y8=False)
    assert not y32.any()


def test_conv_s8_1x1_equals_int8_gemm():
    x = RNG.integers(0, 256, size=(3, 5, 4, 24)).astype(np.uint8)
    w = RNG.integers(-128, 128, size=(16, 1, 1, 24)).astype(np.int8)
    zW_k = RNG.integers(-5, 5, size=16).astype(np.int32)
    y32, _, _ = oracle.conv2d_nhwc_s8_zp(x, w, x_signed=0, w_signed=1, zX=121, zW_k=zW_k,
                                         pad=(0, 0), want_y8=False)
    g32, _, _, _ = oracle.gemm_s8_zp(x.reshape(-1, 24), w.reshape(16, 24), a_signed=0, b_signed=1,
                                     zA=121, zB_col=zW_k, want_c8=False)
    assert np.array_equal(y32.reshape(-1, 16), g32)


@pytest.mark.parametrize("pad,stride", [((1, 1), (1, 1)), ((0, 2), (2, 1)), ((2, 1), (2, 2))])
def test_conv_s8_brute_force_im2col_with_zero_point_padding(pad, stride):
    x = RNG.integers(0, 256, size=(2, 6, 5, 8)).astype(np.uint8)
    w = RNG.integers(0, 256, size=(12, 3, 3, 8)).astype(np.uint8)
    zX, zW = 90, 140
    y32, _, _ = oracle.conv2d_nhwc_s8_zp(x, w, x_signed=0, w_signed=0, zX=zX, zW=zW, pad=pad,
                                         stride=stride, want_y8=False)
    N, H, W, C = x.shape
    xp = np.full((N, H + 2 * pad[0], W + 2 * pad[1], C), zX, np.int64)
    xp[:, pad[0]:pad[0] + H, pad[1]:pad[1] + W, :] = x
    P = (H + 2 * pad[0] - 3) // stride[0] + 1
    Q = (W + 2 * pad[1] - 3) // stride[1] + 1
    cols = np.stack([xp[:, p * stride[0]:p * stride[0] + 3, q * stride[1]:q * stride[1] + 3, :]
                     for p in range(P) for q in range(Q)], axis=1).reshape(N * P * Q, -1)
    want = (cols - zX) @ (w.astype(np.int64).reshape(12, -1) - zW).T
    assert np.array_equal(y32.reshape(-1, 12).astype(np.int64), want)


def test_conv_s8_vs_float64_library_conv_on_shifted_values():
    x = RNG.integers(-128, 128, size=(2, 7, 9, 16)).astype(np.int8)
    w = RNG.integers(-128, 128, size=(8, 3, 3, 16)).astype(np.int8)
    zX, zW = -3, 5
    y32, _, _ = oracle.conv2d_nhwc_s8_zp(x, w, x_signed=1, w_signed=1, zX=zX, zW=zW, pad=(1, 1),
                                         want_y8=False)
    xt = torch.from_numpy(x.astype(np.float64) - zX).permute(0, 3, 1, 2)
    wt = torch.from_numpy(w.astype(np.float64) - zW).permute(0, 3, 1, 2)
    want = torch.nn.functional.conv2d(xt, wt, padding=1).permute(0, 2, 3, 1).numpy()
    assert np.array_equal(y32.astype(np.float64), want)


def test_conv_s8_delta_kernel_and_requant():
    x = RNG.integers(0, 256, size=(1, 5, 6, 8)).astype(np.uint8)
    zW = 7
    w = np.full((8, 3, 3, 8), zW, np.int8)
    w[np.arange(8), 1, 1, np.arange(8)] += 1                 # w - zW = delta at the centre tap
    y32, y8, _ = oracle.conv2d_nhwc_s8_zp(x, w, x_signed=0, w_signed=1, zX=100, zW=zW,
                                          pad=(1, 1), scale=0.5)
    assert np.array_equal(y32, x.astype(np.int32) - 100)
    assert np.array_equal(y8, np.array([[oracle.requant(int(v), 0.5) for v in row]
                                        for row in y32.reshape(-1, 8)], np.int8).reshape(y8.shape))


# ---------------------------------------------------------------------------
# the acceptance test of every fp16 / bf16 parity check
# ---------------------------------------------------------------------------
# oracle.fp16_accept decides "|gpu - exact| <= rel * sum_k |a_ik b_kj|" per element
# (the stated tolerance of the floating-point GEMM and convolution, applied to the
# GEMM definition of the GEMM page, §4.1).  Hand-built cases: an error exactly at
# the bound is accepted and the next representable value beyond it is not, on
# either side of the exact value and in float32 and float64; NaN / inf results
# are rejected wherever they sit; an element whose |a b| sum is 0 must be exactly
# 0; a custom rel is honoured; one bad element among good ones rejects the lot.

def test_fp16_accept_error_at_the_bound_is_accepted_and_just_beyond_is_not():
    sabs = np.array([500.0, 1000.0, 250.0])          # bounds 1.0, 2.0, 0.5 (exact)
    # ref +- bound and its neighbours lie within a factor of two of ref, so every
    # error below is computed exactly in float64 (Sterbenz)
    ref = np.array([3.0, -7.0, 2.0])
    bound = 2e-3 * sabs
    assert bound.tolist() == [1.0, 2.0, 0.5]
    for dt in (np.float32, np.float64):
        for sign in (1.0, -1.0):
            at = (ref + sign * bound).astype(dt)
            assert np.array_equal(at.astype(np.float64), ref + sign * bound)  # representable
            ok, worst = oracle.fp16_accept(at, ref, sabs)
            assert ok and worst == 1.0
            for i in range(3):
                beyond = at.copy()
                beyond[i] = np.nextafter(at[i], dt(sign * np.inf))
                ok, worst = oracle.fp16_accept(beyond, ref, sabs)
                assert not ok and worst > 1.0, (dt, sign, i)


def test_fp16_accept_rejects_nan_and_inf_results():
    ref = np.zeros(4)
    sabs = np.full(4, 1e30)                       # a bound no finite error reaches
    for bad in (np.nan, np.inf, -np.inf):
        for i in range(4):
            g = np.zeros(4, np.float32)
            g[i] = bad
            ok, _ = oracle.fp16_accept(g, ref, sabs)
            assert not ok, (bad, i)
    ok, _ = oracle.fp16_accept(np.zeros(4, np.float16), ref, sabs)
    assert ok


def test_fp16_accept_zero_abs_sum_demands_exact_zero():
    ref = np.array([0.0, 0.0])
    sabs = np.array([0.0, 5.0])
    ok, worst = oracle.fp16_accept(np.array([0.0, 0.01], np.float32), ref, sabs)
    assert ok and worst <= 1.0
    for tiny in (np.float32(1e-45), np.float32(-1e-45), np.float16(6e-8)):
        g = np.array([tiny, 0.0]).astype(np.float32)
        ok, worst = oracle.fp16_accept(g, ref, sabs)
        assert not ok and worst == np.inf


def test_fp16_accept_honours_rel():
    ref = np.array([1.0])
    sabs = np.array([1000.0])
    g = np.array([1.0 + 5.0])                     # 2.5 x the default bound of 2.0
    assert not oracle.fp16_accept(g, ref, sabs)[0]
    ok, worst = oracle.fp16_accept(g, ref, sabs, rel=5e-3)   # bound 5.0: at it
    assert ok and worst == 1.0
    assert not oracle.fp16_accept(g, ref, sabs, rel=4e-3)[0]


def test_fp16_accept_one_bad_element_rejects_the_array():
    rng = np.random.default_rng(7)
    sabs = rng.uniform(1.0, 100.0, (64, 64))
    ref = rng.normal(size=(64, 64))
    g = ref + 0.5 * 2e-3 * sabs * rng.uniform(-1.0, 1.0, (64, 64))
    ok, worst = oracle.fp16_accept(g, ref, sabs)
    assert ok and worst <= 0.5
    g[17, 41] = ref[17, 41] + 1.5 * 2e-3 * sabs[17, 41]
    ok, worst = oracle.fp16_accept(g, ref, sabs)
    assert not ok and abs(worst - 1.5) < 1e-9
