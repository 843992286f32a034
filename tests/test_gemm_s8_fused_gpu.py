"""GPU parity of the fused int8 path (IGC_INT8_PATH_FUSED: the operands
converted to fp16 inside the GEMM kernel, row / column sums taken in the same
pass) against the CPU oracle,
bit for bit, where it differs from the pre-pass form: K that is no multiple of
the 64-k stage (the converters treat bytes past K as the value 0), K below 16,
both tile widths and the split last round, all four signedness combinations,
and equality of the three int8 tensor paths on one problem."""

import numpy as np
import pytest
import torch

import implicit_gemm_conv_tcgen05_gb300 as igc
import oracle
from gpu_helpers import check_device_ok, host

pytestmark = pytest.mark.gpu


def _operands(rng, M, N, K, a_signed, b_signed, pad=16):
    """A (M,K) and Bt (N,K) as views of buffers whose rows are padded to a multiple
    of `pad` bytes (the TMA row-stride rule) and filled with other values past K."""
    ld = (K + pad - 1) // pad * pad + pad
    lo_a, hi_a = (-128, 128) if a_signed else (0, 256)
    lo_b, hi_b = (-128, 128) if b_signed else (0, 256)
    Abuf = rng.integers(lo_a, hi_a, (M, ld)).astype(np.int8 if a_signed else np.uint8)
    Bbuf = rng.integers(lo_b, hi_b, (N, ld)).astype(np.int8 if b_signed else np.uint8)
    return Abuf, Bbuf, ld


def _run(Abuf, Bbuf, K, path=igc.INT8_PATH_FUSED, width=0, **kw):
    M, N = Abuf.shape[0], Bbuf.shape[0]
    A = torch.from_numpy(Abuf).cuda()[:, :K]
    Bt = torch.from_numpy(Bbuf).cuda()[:, :K]
    C32 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    C8 = torch.empty((M, N), dtype=torch.int8, device="cuda")
    dkw = {k: (torch.from_numpy(np.ascontiguousarray(v)).cuda() if isinstance(v, np.ndarray) else v)
           for k, v in kw.items()}
    old_p, old_w = igc.igc_set_int8_path(path), igc.igc_set_tile_width(width)
    try:
        igc.gemm_s8_zp(A, Bt, C32=C32, C8=C8, **dkw)
    finally:
        igc.igc_set_int8_path(old_p)
        igc.igc_set_tile_width(old_w)
    check_device_ok()
    return host(C32), host(C8)


def _oracle(Abuf, Bbuf, K, a_signed, b_signed, **kw):
    o32, o8, _, ovf = oracle.gemm_s8_zp(Abuf[:, :K], Bbuf[:, :K], a_signed=a_signed,
                                        b_signed=b_signed, **kw)
    assert not ovf
    return o32, o8


@pytest.mark.parametrize("K", [1, 7, 15, 16, 17, 63, 64, 65, 100, 1023, 1024, 1025, 2100])
@pytest.mark.parametrize("signs", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_fused_ragged_k_bit_exact(K, signs):
    a_signed, b_signed = signs
    rng = np.random.default_rng(1000 * K + 10 * a_signed + b_signed)
    M, N = 300, 200
    Abuf, Bbuf, _ = _operands(rng, M, N, K, a_signed, b_signed)
    kw = dict(zA=int(rng.integers(-5, 200)), zB=int(rng.integers(-5, 200)), scale=2.0 ** -9)
    g32, g8 = _run(Abuf, Bbuf, K, **kw)
    o32, o8 = _oracle(Abuf, Bbuf, K, a_signed, b_signed, **kw)
    assert np.array_equal(g32, o32), f"C32: {np.count_nonzero(g32 != o32)} differ"
    assert np.array_equal(g8, o8), f"C8: {np.count_nonzero(g8 != o8)} differ"


@pytest.mark.parametrize("width", [128, 256])
@pytest.mark.parametrize("shape", [(2560, 2048, 1088), (520, 2304, 320), (256, 80, 4096)])
def test_fused_each_width_and_split_last_round(width, shape):
    """Shapes whose schedule has whole tiles and a last round of column halves
    (2560 x 2048 at width 256: 80 tiles over 76 pairs), ragged M and N, and a
    skinny problem over several exact 1024-k chunks; per-row and per-column zero
    points and scales."""
    M, N, K = shape
    rng = np.random.default_rng(M + N + K + width)
    Abuf, Bbuf, _ = _operands(rng, M, N, K, 0, 1)
    kw = dict(zA_row=rng.integers(100, 157, M).astype(np.int32),
              zB_col=rng.integers(-20, 21, N).astype(np.int32),
              scale_col=rng.uniform(1e-4, 1e-3, N).astype(np.float32))
    g32, g8 = _run(Abuf, Bbuf, K, width=width, **kw)
    o32, o8 = _oracle(Abuf, Bbuf, K, 0, 1, **kw)
    assert np.array_equal(g32, o32), f"C32: {np.count_nonzero(g32 != o32)} differ"
    assert np.array_equal(g8, o8), f"C8: {np.count_nonzero(g8 != o8)} differ"


def test_three_int8_paths_agree_bit_for_bit():
    rng = np.random.default_rng(77)
    M, N, K = 1000, 1100, 1300
    Abuf, Bbuf, _ = _operands(rng, M, N, K, 1, 0)
    kw = dict(zA=3, zB_col=rng.integers(0, 256, N).astype(np.int32), scale=1.0 / 3000.0)
    outs = [_run(Abuf, Bbuf, K, path=p, **kw) for p in
            (igc.INT8_PATH_FUSED, igc.INT8_PATH_TCGEN05, igc.INT8_PATH_MMA_SYNC)]
    o32, o8 = _oracle(Abuf, Bbuf, K, 1, 0, **kw)
    for g32, g8 in outs:
        assert np.array_equal(g32, o32) and np.array_equal(g8, o8)


@pytest.mark.parametrize("M,N,K,signs,width", [
    (256, 256, 256, (0, 1), 0),
    (300, 520, 1100, (1, 0), 0),
    (2560, 2048, 320, (0, 0), 256),
    (130, 200, 96, (1, 1), 128),
])
def test_fused_dequantised_output_bit_exact(M, N, K, signs, width):
    """gemm_s8_zp_dequant on the fused path: Y = ((fp32(C32) s_row) s_col) + bias,
    bit for bit against the oracle's dequantisation of its own C32."""
    import synth
    a_signed, b_signed = signs
    rng = np.random.default_rng(7 * M + N + K)
    Abuf, Bbuf, _ = _operands(rng, M, N, K, a_signed, b_signed)
    zA_row = rng.integers(0, 200, size=M).astype(np.int32)
    zB = int(rng.integers(-10, 130))
    s_row = synth.uniform_f32(M + K, 5, (M,), 1e-3, 1e-1)
    s_col = synth.uniform_f32(N + K, 6, (N,), 1e-3, 1e-1)
    bias = synth.uniform_f32(M + N, 7, (N,), -5.0, 5.0)
    A = torch.from_numpy(Abuf).cuda()[:, :K]
    Bt = torch.from_numpy(Bbuf).cuda()[:, :K]
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    old_p, old_w = igc.igc_set_int8_path(igc.INT8_PATH_FUSED), igc.igc_set_tile_width(width)
    try:
        Y = igc.gemm_s8_zp_dequant(A, Bt, zA_row=d(zA_row), zB=zB, scale_row=d(s_row),
                                   scale_col=d(s_col), bias=d(bias))
    finally:
        igc.igc_set_int8_path(old_p)
        igc.igc_set_tile_width(old_w)
    check_device_ok()
    C32, _, _, _ = oracle.gemm_s8_zp(Abuf[:, :K], Bbuf[:, :K], a_signed=a_signed,
                                     b_signed=b_signed, zA_row=zA_row, zB=zB, want_c8=False)
    want = oracle.dequant_matrix(C32, s_row, s_col, bias)
    got = host(Y)
    bad = np.count_nonzero(got.view(np.uint32) != want.view(np.uint32))
    assert bad == 0, f"{bad} of {got.size} dequantised outputs differ"


def test_fused_path_in_a_cuda_graph_with_new_inputs():
    """The fused kernel captured in a CUDA graph and replayed after the inputs
    changed in place gives the new inputs' results."""
    rng = np.random.default_rng(91)
    M, N, K = 512, 640, 768
    A = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    Bt = torch.empty((N, K), dtype=torch.int8, device="cuda")
    C32 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    C8 = torch.empty((M, N), dtype=torch.int8, device="cuda")
    kw = dict(zA=100, zB=3, scale=2.0 ** -11)
    old = igc.igc_set_int8_path(igc.INT8_PATH_FUSED)
    try:
        igc.gemm_s8_zp(A.zero_(), Bt.zero_(), C32=C32, C8=C8, **kw)  # set-up outside capture
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                igc.gemm_s8_zp(A, Bt, C32=C32, C8=C8, **kw)
        torch.cuda.current_stream().wait_stream(side)
        for trial in range(2):
            Ah = rng.integers(0, 256, (M, K)).astype(np.uint8)
            Bh = rng.integers(-128, 128, (N, K)).astype(np.int8)
            A.copy_(torch.from_numpy(Ah))
            Bt.copy_(torch.from_numpy(Bh))
            g.replay()
            check_device_ok()
            o32, o8 = _oracle(Ah, Bh, K, 0, 1, **kw)
            assert np.array_equal(host(C32), o32), f"C32 differs on replay {trial}"
            assert np.array_equal(host(C8), o8), f"C8 differs on replay {trial}"
    finally:
        igc.igc_set_int8_path(old)
