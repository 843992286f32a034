"""GPU parity of gemm_s8_zp (exact integer GEMM on the fp16 tensor pipe, fused
zero-point correction and requantisation) against the CPU oracle: every int32
and int8 output must match bit for bit."""

import numpy as np
import pytest
import torch

import implicit_gemm_conv_tcgen05_gb300 as igc
import oracle
import synth
from gpu_helpers import check_device_ok, dev, host

pytestmark = pytest.mark.gpu


def _gpu(A, Bt, zA=0, zA_row=None, zB=0, zB_col=None, scale=0.0, scale_col=None,
         want32=True, want8=True):
    M, N = A.shape[0], Bt.shape[0]
    C32 = torch.empty((M, N), dtype=torch.int32, device="cuda") if want32 else None
    C8 = torch.empty((M, N), dtype=torch.int8, device="cuda") if want8 else None
    igc.gemm_s8_zp(dev(A), dev(Bt), zA=zA, zA_row=None if zA_row is None else dev(zA_row),
                   zB=zB, zB_col=None if zB_col is None else dev(zB_col), C32=C32, C8=C8,
                   scale=scale, scale_col=None if scale_col is None else dev(scale_col))
    check_device_ok()
    return (host(C32) if want32 else None), (host(C8) if want8 else None)


def _oracle(A, Bt, **kw):
    a_signed = 1 if A.dtype == np.int8 else 0
    b_signed = 1 if Bt.dtype == np.int8 else 0
    C32, C8, _, ovf = oracle.gemm_s8_zp(A, Bt, a_signed=a_signed, b_signed=b_signed, **kw)
    return C32, C8, ovf


def _assert_equal(got, want, what):
    bad = np.count_nonzero(got != want)
    assert bad == 0, f"{what}: {bad} of {want.size} outputs differ"


def test_config2_1024_cubed_per_tensor_bit_exact():
    w = synth.workload(2)
    kw = dict(zA=w["zA"], zB=w["zB"], scale=w["scale"])
    g32, g8 = _gpu(w["A"], w["Bt"], **kw)
    o32, o8, ovf = _oracle(w["A"], w["Bt"], **kw)
    assert not ovf
    _assert_equal(g32, o32, "C32")
    _assert_equal(g8, o8, "C8")
    # ties (C32 = 2048 mod 4096 with scale 2^-12) occur in this workload and are covered
    assert np.count_nonzero((o32 & 4095) == 2048) > 0


def test_config5_8192_cubed_sampled_rows_bit_exact():
    w = synth.workload(5)
    kw = dict(zA_row=w["zA_row"], scale_col=w["scale_col"])
    g32, g8 = _gpu(w["A"], w["Bt"], **kw)
    rows = np.array([0, 1, 127, 128, 255, 4095, 4096, 5000, 8190, 8191])
    o32, o8, ovf = _oracle(w["A"][rows], w["Bt"], zA_row=w["zA_row"][rows],
                           scale_col=w["scale_col"])
    assert not ovf
    _assert_equal(g32[rows], o32, "C32 rows")
    _assert_equal(g8[rows], o8, "C8 rows")
    cols = np.array([0, 255, 256, 8191])
    o32c, o8c, _ = _oracle(w["A"], w["Bt"][cols], zA_row=w["zA_row"],
                           scale_col=w["scale_col"][cols])
    _assert_equal(g32[:, cols], o32c, "C32 cols")
    _assert_equal(g8[:, cols], o8c, "C8 cols")


@pytest.mark.parametrize("a_val,b_val,a_signed,b_signed", [
    (255, 255, 0, 0), (0, 255, 0, 0), (255, 0, 0, 0), (-128, -128, 1, 1), (127, -128, 1, 1),
    (255, -128, 0, 1), (0, 127, 0, 1)])
@pytest.mark.parametrize("K", [256, 512, 1024, 4096 + 256])
def test_extreme_magnitudes_exact(a_val, b_val, a_signed, b_signed, K):
    """Constant operands at the ends of their ranges: every fp32 chunk sum sits
    at its largest magnitude (2^24 for a full 1024-k chunk of (-128)(-128)
    products), testing the exactness of the chunking."""
    M, N = 128, 256
    A = np.full((M, K), a_val, np.int8 if a_signed else np.uint8)
    Bt = np.full((N, K), b_val, np.int8 if b_signed else np.uint8)
    g32, _ = _gpu(A, Bt, want8=False)
    o32, _, _ = _oracle(A, Bt, want_c8=False)
    _assert_equal(g32, o32, "C32")


def test_alternating_signs_and_random_extremes():
    rng = np.random.default_rng(7)
    M, N, K = 256, 512, 2048
    A = rng.choice(np.array([0, 255], np.uint8), size=(M, K))
    Bt = rng.choice(np.array([-128, 127], np.int8), size=(N, K))
    zA_row = rng.integers(0, 256, size=M).astype(np.int32)
    zB_col = rng.integers(-128, 128, size=N).astype(np.int32)
    scale_col = synth.uniform_f32(3, 5, (N,), 1e-6, 1e-4)
    kw = dict(zA_row=zA_row, zB_col=zB_col, scale_col=scale_col)
    g32, g8 = _gpu(A, Bt, **kw)
    o32, o8, _ = _oracle(A, Bt, **kw)
    _assert_equal(g32, o32, "C32")
    _assert_equal(g8, o8, "C8")


@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (130, 257, 48), (129, 300, 272), (300, 129, 1040),
                                   (64, 1000, 16)])
@pytest.mark.parametrize("signs", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_ragged_shapes_all_signedness(M, N, K, signs):
    a_signed, b_signed = signs
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    A = (rng.integers(-128, 128, size=(M, K)).astype(np.int8) if a_signed
         else rng.integers(0, 256, size=(M, K)).astype(np.uint8))
    Bt = (rng.integers(-128, 128, size=(N, K)).astype(np.int8) if b_signed
          else rng.integers(0, 256, size=(N, K)).astype(np.uint8))
    kw = dict(zA=int(rng.integers(-50, 200)), zB=int(rng.integers(-50, 200)),
              scale=float(np.float32(2.0 ** -13)))
    g32, g8 = _gpu(A, Bt, **kw)
    o32, o8, _ = _oracle(A, Bt, **kw)
    _assert_equal(g32, o32, "C32")
    _assert_equal(g8, o8, "C8")


def test_unaligned_k_uses_scalar_prepass():
    # K % 16 != 0 but row strides still 16-byte multiples (views of wider rows)
    rng = np.random.default_rng(11)
    M, N, K = 100, 200, 40
    Abig = torch.from_numpy(rng.integers(0, 256, size=(M, 48)).astype(np.uint8)).cuda()
    Bbig = torch.from_numpy(rng.integers(0, 256, size=(N, 48)).astype(np.uint8)).cuda()
    A, Bt = Abig[:, :K], Bbig[:, :K]
    C32 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    igc.gemm_s8_zp(A, Bt, zA=3, zB=250, C32=C32)
    check_device_ok()
    o32, _, _ = _oracle(A.cpu().numpy(), Bt.cpu().numpy(), zA=3, zB=250, want_c8=False)
    _assert_equal(host(C32), o32, "C32")


def test_only_c8_output_and_k_zero():
    w = synth.gemm_s8_inputs(256, 256, 256, 5, "per_tensor")
    _, g8 = _gpu(w["A"], w["Bt"], zA=w["zA"], zB=w["zB"], scale=w["scale"], want32=False)
    _, o8, _ = _oracle(w["A"], w["Bt"], zA=w["zA"], zB=w["zB"], scale=w["scale"])
    _assert_equal(g8, o8, "C8")
    A = torch.empty((16, 0), dtype=torch.uint8, device="cuda")
    Bt = torch.empty((32, 0), dtype=torch.uint8, device="cuda")
    C32 = torch.full((16, 32), 5, dtype=torch.int32, device="cuda")
    C8 = torch.full((16, 32), 5, dtype=torch.int8, device="cuda")
    igc.gemm_s8_zp(A, Bt, zA=1, zB=2, C32=C32, C8=C8, scale=1.0)
    assert torch.all(C32 == 0) and torch.all(C8 == 0)


def test_workspace_too_small_rejected():
    A = torch.zeros((64, 64), dtype=torch.uint8, device="cuda")
    Bt = torch.zeros((64, 64), dtype=torch.uint8, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(igc.IGCError) as e:
        igc.gemm_s8_zp(A, Bt, C32=torch.empty((64, 64), dtype=torch.int32, device="cuda"),
                       workspace=ws)
    assert e.value.status == igc.IGC_ERR_WORKSPACE


def test_whole_tiles_and_split_last_round_bit_exact():
    """80 tiles of 256 x 256 (more than one round of the persistent schedule, a
    short last round of column halves), per-row zA and per-column zB, every
    output compared."""
    rng = np.random.default_rng(80)
    M, N, K = 2560, 2048, 320
    A = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    Bt = rng.integers(-128, 128, size=(N, K)).astype(np.int8)
    kw = dict(zA_row=rng.integers(0, 256, size=M).astype(np.int32),
              zB_col=rng.integers(-128, 128, size=N).astype(np.int32),
              scale_col=synth.uniform_f32(80, 5, (N,), 1e-5, 1e-4))
    g32, g8 = _gpu(A, Bt, **kw)
    o32, o8, _ = _oracle(A, Bt, **kw)
    _assert_equal(g32, o32, "C32")
    _assert_equal(g8, o8, "C8")


def test_requant_with_non_finite_scales():
    """Per-column scales holding +inf, -inf, NaN, 0 and the largest finite value:
    the product is clamped (infinities to the ends), a NaN product gives 0."""
    rng = np.random.default_rng(12)
    M, N, K = 128, 256, 64
    A = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    Bt = rng.integers(-128, 128, size=(N, K)).astype(np.int8)
    special = np.array([np.inf, -np.inf, np.nan, 0.0, np.finfo(np.float32).max, 1e-30],
                       dtype=np.float32)
    scale_col = np.resize(special, N).astype(np.float32)
    kw = dict(zA=100, zB=-5, scale_col=scale_col)
    g32, g8 = _gpu(A, Bt, **kw)
    o32, o8, _ = _oracle(A, Bt, **kw)
    _assert_equal(g32, o32, "C32")
    _assert_equal(g8, o8, "C8")


def test_outputs_at_unaligned_addresses_use_direct_stores():
    """C32 and C8 views that start 4 / 1 bytes past an aligned address: the kernel
    cannot use TMA stores for them and must write exactly the view."""
    rng = np.random.default_rng(13)
    M, N, K = 200, 300, 96
    A = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    Bt = rng.integers(0, 256, size=(N, K)).astype(np.uint8)
    C32big = torch.full((M, N + 4), 9, dtype=torch.int32, device="cuda")
    C8big = torch.full((M, N + 32), 9, dtype=torch.int8, device="cuda")
    C32 = C32big[:, 1:1 + N]
    C8 = C8big[:, 1:1 + N]
    igc.gemm_s8_zp(dev(A), dev(Bt), zA=7, zB=200, C32=C32, C8=C8,
                   scale=float(np.float32(2.0 ** -10)))
    check_device_ok()
    o32, o8, _ = _oracle(A, Bt, zA=7, zB=200, scale=float(np.float32(2.0 ** -10)))
    g32, g8 = host(C32big), host(C8big)
    _assert_equal(g32[:, 1:1 + N], o32, "C32")
    _assert_equal(g8[:, 1:1 + N], o8, "C8")
    assert np.all(g32[:, 0] == 9) and np.all(g32[:, 1 + N:] == 9)
    assert np.all(g8[:, 0] == 9) and np.all(g8[:, 1 + N:] == 9)


def test_running_sum_near_2_pow_24_with_unit_products_in_one_mma():
    """A 1024-k chunk whose running sum reaches 2^24 - 16384 before its last 16-k
    MMA, which mixes (-128)(-128) products with +-1 and +-128 products (so the
    chunk ends at 2^24 - 16384 +- 1, an odd integer at the top exponent); the
    next chunk does the same with 127 x (-128) products and its unit products in
    the middle.  Every C32 must be exact (uint8 A with zA = 128 gives the shifted
    operand A - 128; int8 B with zB = 0 is used as is)."""
    M, N, K = 256, 256, 2048
    a = np.full((M, K), -128, np.int64)       # the shifted A values a' = A - 128
    b = np.full((N, K), -128, np.int64)       # B values (int8, zB = 0)
    a[:, 1024:] = 127
    i = np.arange(M)
    j = np.arange(N)
    sign = np.where((i // 16) % 2 == 0, 1, -1)
    # chunk 0: the last MMA (k 1008..1023) holds one unit entry per row and column
    a[i, 1008 + i % 16] = sign
    b[j, 1008 + j % 16] = 1
    # chunk 1: unit entries in an MMA in the middle of the chunk (k 1536..1551)
    a[i, 1536 + (i * 7) % 16] = -sign
    b[j, 1536 + (j * 7) % 16] = -1
    A = (a + 128).astype(np.uint8)
    Bt = b.astype(np.int8)
    want = a @ b.T                            # exact int64
    assert np.abs(want).max() < 2 ** 31
    kw = dict(zA=128, zB=0, scale=2.0 ** -20)
    g32, g8 = _gpu(A, Bt, **kw)
    o32, o8, ovf = _oracle(A, Bt, **kw)
    assert not ovf
    _assert_equal(o32, want, "oracle C32 vs int64 matmul")
    _assert_equal(g32, want, "C32")
    _assert_equal(g8, o8, "C8")
    # the chunk-0 partial sums of the diagonal blocks are 2^24 - 16384 +- 1
    part = a[:, :1024] @ b[:, :1024].T
    diag = (i[:, None] % 16) == (j[None, :] % 16)
    assert set(np.unique(part[diag])) == {2 ** 24 - 16384 - 1, 2 ** 24 - 16384 + 1}
