"""Parity where byte offsets pass 2^31: operands, workspaces and outputs larger
than 2 GiB, so that every address in the kernels, the int8 pre-passes and the
tensor maps has to be computed in 64 bits.  Inputs are drawn on the device from
seeded generators; the rows (or images) around the first one that starts at or
beyond 2^31 bytes, and the last one, go to the CPU oracle.  Sizes stay within the
limits the header states (each size below 2^31, a convolution's N*H*W*C and
N*P*Q*K below 2^31 elements)."""

import numpy as np
import pytest
import torch

import implicit_gemm_conv_tcgen05_gb300 as igc
import oracle
from gpu_helpers import assert_f16_is_rne_of_f32, assert_fp16_bound, check_device_ok, host

pytestmark = pytest.mark.gpu

TWO_GIB = 2 ** 31


@pytest.fixture(autouse=True)
def _release_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _gen(seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return g


def _crossing(unit_bytes, count):
    """Indices of the units (rows, images) around the first one that starts at or
    beyond 2^31 bytes, plus the first and the last."""
    r = TWO_GIB // unit_bytes
    assert 0 < r < count - 2, "the buffer does not pass 2^31 bytes"
    return np.unique(np.array([0, r - 1, r, r + 1, count - 1]))


def _on_device(idx):
    return torch.as_tensor(idx, device="cuda")


def _assert_equal(got, want, what):
    bad = np.count_nonzero(got != want)
    assert bad == 0, f"{what}: {bad} of {want.size} outputs differ"


def test_gemm_f16_operand_beyond_2_gib():
    M, N, K = 278528, 256, 4096                       # A: 2.28 GB
    g = _gen(101)
    A = torch.empty((M, K), dtype=torch.float16, device="cuda").uniform_(-1, 1, generator=g)
    Bt = torch.empty((N, K), dtype=torch.float16, device="cuda").uniform_(-1, 1, generator=g)
    C16 = torch.empty((M, N), dtype=torch.float16, device="cuda")
    C32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    igc.gemm_f16(A, Bt, C16, C32)
    check_device_ok()
    rows = _crossing(K * 2, M)
    ref, sabs = oracle.gemm_f16(host(A[_on_device(rows)]), host(Bt))
    c32 = host(C32[_on_device(rows)])
    assert_fp16_bound(c32, ref, sabs, "A beyond 2 GiB, fp32 copy")
    assert_f16_is_rne_of_f32(host(C16[_on_device(rows)]), c32, "A beyond 2 GiB")


def test_gemm_bf16_operand_and_output_beyond_2_gib():
    M, N, K = 278528, 2048, 4096                      # A: 2.28 GB; bf16 C: 1.14 GB, fp32: 2.28 GB
    g = _gen(109)
    A = torch.empty((M, K), dtype=torch.bfloat16, device="cuda").uniform_(-1, 1, generator=g)
    Bt = torch.empty((N, K), dtype=torch.bfloat16, device="cuda").uniform_(-1, 1, generator=g)
    C16 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    C32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    igc.gemm_bf16(A, Bt, C16, C32)
    check_device_ok()
    rows = np.unique(np.concatenate([_crossing(K * 2, M), _crossing(N * 4, M)]))
    r = _on_device(rows)
    a_bits = host(A[r].view(torch.int16)).view(np.uint16)
    b_bits = host(Bt.view(torch.int16)).view(np.uint16)
    ref, sabs = oracle.gemm_bf16(a_bits, b_bits)
    c32 = host(C32[r])
    assert_fp16_bound(c32, ref, sabs, "bf16 beyond 2 GiB, fp32 copy")
    want = oracle.f32_to_bf16_bits_array(c32)
    got = host(C16[r].view(torch.int16)).view(np.uint16)
    assert np.array_equal(got, want), "bf16 outputs are not the RNE rounding of the fp32 copy"


@pytest.mark.parametrize("pad", [0, 1])   # row stride N: TMA stores; N + 1: direct stores
def test_gemm_f16_output_beyond_2_gib(pad):
    M, N, K = 24576, 24576, 64                        # C: 2.42 GB of fp32
    g = _gen(102 + pad)
    A = torch.empty((M, K), dtype=torch.float16, device="cuda").uniform_(-1, 1, generator=g)
    Bt = torch.empty((N, K), dtype=torch.float16, device="cuda").uniform_(-1, 1, generator=g)
    buf = torch.empty((M, N + pad), dtype=torch.float32, device="cuda")
    if pad:
        buf[:, N:] = 7.0
    C = buf[:, :N]
    igc.gemm_f16(A, Bt, C)
    check_device_ok()
    rows = _crossing((N + pad) * 4, M)
    ref, sabs = oracle.gemm_f16(host(A[_on_device(rows)]), host(Bt))
    assert_fp16_bound(host(C[_on_device(rows)]), ref, sabs,
                      f"C beyond 2 GiB (row stride N + {pad})")
    cols = np.array([0, 1, 12345, N - 1])
    ref_c, sabs_c = oracle.gemm_f16(host(A), host(Bt[_on_device(cols)]))
    assert_fp16_bound(host(C[:, _on_device(cols)]), ref_c, sabs_c, "C beyond 2 GiB, columns")
    if pad:
        assert torch.all(buf[:, N:] == 7.0)          # nothing written past a row


def test_gemm_s8_zp_operand_and_workspace_beyond_2_gib():
    # A: 2.28 GB of uint8; the pre-pass's fp16 copy of it in the workspace: 4.56 GB
    M, N, K = 557056, 256, 4096
    g = _gen(104)
    A = torch.randint(0, 256, (M, K), dtype=torch.uint8, device="cuda", generator=g)
    Bt = torch.randint(-127, 128, (N, K), dtype=torch.int8, device="cuda", generator=g)
    zA_row = torch.randint(100, 157, (M,), dtype=torch.int32, device="cuda", generator=g)
    scale_col = torch.empty(N, dtype=torch.float32, device="cuda").uniform_(1e-4, 1e-3,
                                                                            generator=g)
    C32 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    C8 = torch.empty((M, N), dtype=torch.int8, device="cuda")
    igc.gemm_s8_zp(A, Bt, zA_row=zA_row, C32=C32, C8=C8, scale_col=scale_col)
    check_device_ok()
    rows = _crossing(K, M)
    r = _on_device(rows)
    o32, o8, _, ovf = oracle.gemm_s8_zp(host(A[r]), host(Bt), a_signed=0, b_signed=1,
                                        zA_row=host(zA_row[r]), scale_col=host(scale_col))
    assert not ovf
    _assert_equal(host(C32[_on_device(rows)]), o32, "C32 rows")
    _assert_equal(host(C8[_on_device(rows)]), o8, "C8 rows")


def test_gemm_s8_zp_int32_output_beyond_2_gib():
    M, N, K = 24576, 24576, 64                        # C32: 2.42 GB
    g = _gen(105)
    A = torch.randint(-128, 128, (M, K), dtype=torch.int8, device="cuda", generator=g)
    Bt = torch.randint(0, 256, (N, K), dtype=torch.uint8, device="cuda", generator=g)
    C32 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    C8 = torch.empty((M, N), dtype=torch.int8, device="cuda")
    igc.gemm_s8_zp(A, Bt, zA=-3, zB=131, C32=C32, C8=C8, scale=1.0 / 16384)
    check_device_ok()
    rows = _crossing(N * 4, M)
    r = _on_device(rows)
    o32, o8, _, ovf = oracle.gemm_s8_zp(host(A[r]), host(Bt), a_signed=1, b_signed=0,
                                        zA=-3, zB=131, scale=1.0 / 16384)
    assert not ovf
    _assert_equal(host(C32[_on_device(rows)]), o32, "C32 rows")
    _assert_equal(host(C8[_on_device(rows)]), o8, "C8 rows")


def test_conv_f16_input_beyond_2_gib():
    N, H, W, C, K = 1408, 28, 28, 1024, 64            # x: 2.26 GB
    g = _gen(106)
    x = torch.randn((N, H, W, C), dtype=torch.float16, device="cuda", generator=g)
    w = (torch.randn((K, 3, 3, C), dtype=torch.float16, device="cuda", generator=g) *
         (1.0 / 96.0)).half()
    y = torch.empty((N, H, W, K), dtype=torch.float16, device="cuda")
    y32 = torch.empty((N, H, W, K), dtype=torch.float32, device="cuda")
    igc.conv2d_nhwc_f16_implicit(x, w, y, y32, pad=(1, 1))
    check_device_ok()
    imgs = _crossing(H * W * C * 2, N)[-3:]           # the crossing image, its successor, the last
    ref, sabs = oracle.conv2d_nhwc_f16(host(x[_on_device(imgs)]), host(w))
    y32s = host(y32[_on_device(imgs)])
    assert_fp16_bound(y32s, ref, sabs, "x beyond 2 GiB, fp32 copy")
    assert_f16_is_rne_of_f32(host(y[_on_device(imgs)]), y32s, "x beyond 2 GiB")


def test_conv_f16_output_beyond_2_gib():
    N, H, W, C, K = 2816, 28, 28, 64, 512             # y: 2.26 GB
    g = _gen(107)
    x = torch.randn((N, H, W, C), dtype=torch.float16, device="cuda", generator=g)
    w = (torch.randn((K, 3, 3, C), dtype=torch.float16, device="cuda", generator=g) *
         (1.0 / 24.0)).half()
    y = torch.empty((N, H, W, K), dtype=torch.float16, device="cuda")
    igc.conv2d_nhwc_f16_implicit(x, w, y, pad=(1, 1))
    check_device_ok()
    imgs = _crossing(H * W * K * 2, N)[-3:]
    ref, sabs = oracle.conv2d_nhwc_f16(host(x[_on_device(imgs)]), host(w))
    assert_fp16_bound(host(y[_on_device(imgs)]), ref, sabs, "y beyond 2 GiB")


def test_conv_s8_zp_padded_copy_beyond_2_gib():
    # x: 1.13 GB of uint8; its padded fp16 copy in the workspace: 2.6 GB
    N, H, W, C, K = 1408, 28, 28, 1024, 64
    g = _gen(108)
    x = torch.randint(0, 256, (N, H, W, C), dtype=torch.uint8, device="cuda", generator=g)
    w = torch.randint(-127, 128, (K, 3, 3, C), dtype=torch.int8, device="cuda", generator=g)
    scale_k = torch.empty(K, dtype=torch.float32, device="cuda").uniform_(1e-5, 1e-4,
                                                                          generator=g)
    y32 = torch.empty((N, H, W, K), dtype=torch.int32, device="cuda")
    y8 = torch.empty((N, H, W, K), dtype=torch.int8, device="cuda")
    igc.conv2d_nhwc_s8_zp(x, w, zX=121, y32=y32, y8=y8, scale_k=scale_k, pad=(1, 1))
    check_device_ok()
    imgs = _crossing((H + 2) * (W + 2) * C * 2, N)[-3:]
    o32, o8, ovf = oracle.conv2d_nhwc_s8_zp(host(x[_on_device(imgs)]), host(w), x_signed=0,
                                            w_signed=1, zX=121, scale_k=host(scale_k),
                                            pad=(1, 1))
    assert not ovf
    _assert_equal(host(y32[_on_device(imgs)]), o32, "y32 images")
    _assert_equal(host(y8[_on_device(imgs)]), o8, "y8 images")
