"""GPU parity of the converting int8 path (IGC_INT8_PATH_CONVERT: the GEMM
kernel's spare warps convert each 128-row block of the operands, 1024 k at a
time, into the workspace while the tensor cores work; the copies of a block wait
for its flag) against the CPU oracle, bit for bit: K over partial and whole
chunks, ragged blocks, all four signedness combinations, both tile widths, the
split last round and schedules of several rounds (several bands of jobs), the
dequantised output, repeated calls on one workspace, CUDA-graph replay, the
fallback of ineligible calls, and the full-size problem the benchmark times."""

import numpy as np
import pytest
import torch

import implicit_gemm_conv_tcgen05_gb300 as igc
import oracle
from gpu_helpers import check_device_ok, host

pytestmark = pytest.mark.gpu


def _operands(rng, M, N, K, a_signed, b_signed, pad=16):
    """A (M,K) and Bt (N,K) as views of buffers whose rows are padded to a multiple
    of `pad` bytes and filled with other values past K."""
    ld = (K + pad - 1) // pad * pad + pad
    lo_a, hi_a = (-128, 128) if a_signed else (0, 256)
    lo_b, hi_b = (-128, 128) if b_signed else (0, 256)
    Abuf = rng.integers(lo_a, hi_a, (M, ld)).astype(np.int8 if a_signed else np.uint8)
    Bbuf = rng.integers(lo_b, hi_b, (N, ld)).astype(np.int8 if b_signed else np.uint8)
    return Abuf, Bbuf


def _dev(kw):
    return {k: (torch.from_numpy(np.ascontiguousarray(v)).cuda() if isinstance(v, np.ndarray) else v)
            for k, v in kw.items()}


def _run(Abuf, Bbuf, K, path=igc.INT8_PATH_CONVERT, width=0, workspace=None, **kw):
    M, N = Abuf.shape[0], Bbuf.shape[0]
    A = torch.from_numpy(Abuf).cuda()[:, :K]
    Bt = torch.from_numpy(Bbuf).cuda()[:, :K]
    C32 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    C8 = torch.empty((M, N), dtype=torch.int8, device="cuda")
    old_p, old_w = igc.igc_set_int8_path(path), igc.igc_set_tile_width(width)
    try:
        igc.gemm_s8_zp(A, Bt, C32=C32, C8=C8, workspace=workspace, **_dev(kw))
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


def _same(g32, g8, o32, o8):
    assert np.array_equal(g32, o32), f"C32: {np.count_nonzero(g32 != o32)} differ"
    assert np.array_equal(g8, o8), f"C8: {np.count_nonzero(g8 != o8)} differ"


@pytest.mark.parametrize("K", [16, 32, 1008, 1024, 1040, 2064, 3072])
@pytest.mark.parametrize("signs", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_convert_chunks_and_signs_bit_exact(K, signs):
    """K within one chunk, exactly one, and one or two chunks plus a partial
    last one; M = 300 and N = 200 leave partial 128-row blocks of both operands."""
    a_signed, b_signed = signs
    rng = np.random.default_rng(1000 * K + 10 * a_signed + b_signed)
    M, N = 300, 200
    Abuf, Bbuf = _operands(rng, M, N, K, a_signed, b_signed)
    kw = dict(zA=int(rng.integers(-5, 200)), zB=int(rng.integers(-5, 200)), scale=2.0 ** -9)
    _same(*_run(Abuf, Bbuf, K, **kw), *_oracle(Abuf, Bbuf, K, a_signed, b_signed, **kw))


@pytest.mark.parametrize("width", [128, 256])
@pytest.mark.parametrize("shape", [(2560, 2048, 1088), (520, 2304, 320), (256, 80, 4096),
                                   (3000, 1500, 1024)])
def test_convert_widths_rounds_and_split_last_round(width, shape):
    """Schedules of one to three rounds (2560 x 2048 at width 128: 160 tiles over
    76 pairs, three bands of jobs) with whole tiles and a last round of column
    halves, ragged M and N, a skinny problem over four chunks; per-row and
    per-column zero points and scales."""
    M, N, K = shape
    rng = np.random.default_rng(M + N + K + width)
    Abuf, Bbuf = _operands(rng, M, N, K, 0, 1)
    kw = dict(zA_row=rng.integers(100, 157, M).astype(np.int32),
              zB_col=rng.integers(-20, 21, N).astype(np.int32),
              scale_col=rng.uniform(1e-4, 1e-3, N).astype(np.float32))
    _same(*_run(Abuf, Bbuf, K, width=width, **kw), *_oracle(Abuf, Bbuf, K, 0, 1, **kw))


def test_convert_many_bands_equals_default_and_sampled_oracle():
    """4096 x 4096 x 2048 at width 256: 256 tiles, four rounds, so blocks are
    converted in four bands while earlier rounds run.  The whole output equals
    the pre-pass path's (itself oracle-checked) bit for bit, and 64 sampled rows
    equal the oracle's."""
    rng = np.random.default_rng(4096)
    M, N, K = 4096, 4096, 2048
    Abuf, Bbuf = _operands(rng, M, N, K, 0, 0)
    kw = dict(zA=128, zB=121, scale=2.0 ** -16)
    g32, g8 = _run(Abuf, Bbuf, K, width=256, **kw)
    d32, d8 = _run(Abuf, Bbuf, K, path=igc.INT8_PATH_TCGEN05, width=256, **kw)
    _same(g32, g8, d32, d8)
    rows = np.sort(rng.choice(M, 64, replace=False))
    o32, o8 = _oracle(np.ascontiguousarray(Abuf[rows]), Bbuf, K, 0, 0, **kw)
    _same(g32[rows], g8[rows], o32, o8)


def test_four_int8_paths_agree_bit_for_bit():
    rng = np.random.default_rng(77)
    M, N, K = 1000, 1100, 1312
    Abuf, Bbuf = _operands(rng, M, N, K, 1, 0)
    kw = dict(zA=3, zB_col=rng.integers(0, 256, N).astype(np.int32), scale=1.0 / 3000.0)
    outs = [_run(Abuf, Bbuf, K, path=p, **kw) for p in
            (igc.INT8_PATH_CONVERT, igc.INT8_PATH_FUSED, igc.INT8_PATH_TCGEN05,
             igc.INT8_PATH_MMA_SYNC)]
    o32, o8 = _oracle(Abuf, Bbuf, K, 1, 0, **kw)
    for g32, g8 in outs:
        _same(g32, g8, o32, o8)


@pytest.mark.parametrize("K", [100, 1000])
def test_convert_ineligible_call_takes_the_default(K):
    """K that is no multiple of 16: the call takes the pre-pass form and is exact."""
    rng = np.random.default_rng(K)
    Abuf, Bbuf = _operands(rng, 200, 300, K, 1, 1)
    kw = dict(zA=-3, zB=4, scale=2.0 ** -10)
    _same(*_run(Abuf, Bbuf, K, **kw), *_oracle(Abuf, Bbuf, K, 1, 1, **kw))


@pytest.mark.parametrize("M,N,K,signs,width", [
    (256, 256, 256, (0, 1), 0),
    (300, 520, 1104, (1, 0), 0),
    (2560, 2048, 320, (0, 0), 256),
    (130, 200, 96, (1, 1), 128),
])
def test_convert_dequantised_output_bit_exact(M, N, K, signs, width):
    """gemm_s8_zp_dequant on the converting path: Y = ((fp32(C32) s_row) s_col)
    + bias, bit for bit against the oracle's dequantisation of its own C32."""
    import synth
    a_signed, b_signed = signs
    rng = np.random.default_rng(7 * M + N + K)
    Abuf, Bbuf = _operands(rng, M, N, K, a_signed, b_signed)
    zA_row = rng.integers(0, 200, size=M).astype(np.int32)
    zB = int(rng.integers(-10, 130))
    s_row = synth.uniform_f32(M + K, 5, (M,), 1e-3, 1e-1)
    s_col = synth.uniform_f32(N + K, 6, (N,), 1e-3, 1e-1)
    bias = synth.uniform_f32(M + N, 7, (N,), -5.0, 5.0)
    A = torch.from_numpy(Abuf).cuda()[:, :K]
    Bt = torch.from_numpy(Bbuf).cuda()[:, :K]
    d = _dev(dict(zA_row=zA_row, scale_row=s_row, scale_col=s_col, bias=bias))
    old_p, old_w = igc.igc_set_int8_path(igc.INT8_PATH_CONVERT), igc.igc_set_tile_width(width)
    try:
        Y = igc.gemm_s8_zp_dequant(A, Bt, zB=zB, **d)
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


def test_convert_repeated_calls_on_one_workspace():
    """Back-to-back calls with different operands on one workspace: each call
    starts from cleared flags and converts its own operands."""
    rng = np.random.default_rng(5)
    M, N, K = 700, 900, 2080
    ws = torch.empty(igc.gemm_s8_zp_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    kw = dict(zA=7, zB=250, scale=2.0 ** -12)
    for trial in range(3):
        Abuf, Bbuf = _operands(rng, M, N, K, trial % 2, 0)
        _same(*_run(Abuf, Bbuf, K, workspace=ws, **kw),
              *_oracle(Abuf, Bbuf, K, trial % 2, 0, **kw))


def test_convert_path_in_a_cuda_graph_with_new_inputs():
    """The flag clearing and the converting kernel captured in a CUDA graph and
    replayed after the inputs changed in place give the new inputs' results."""
    rng = np.random.default_rng(91)
    M, N, K = 512, 640, 1536
    A = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    Bt = torch.empty((N, K), dtype=torch.int8, device="cuda")
    C32 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    C8 = torch.empty((M, N), dtype=torch.int8, device="cuda")
    ws = torch.empty(igc.gemm_s8_zp_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    kw = dict(zA=100, zB=3, scale=2.0 ** -11)
    old = igc.igc_set_int8_path(igc.INT8_PATH_CONVERT)
    try:
        igc.gemm_s8_zp(A.zero_(), Bt.zero_(), C32=C32, C8=C8, workspace=ws, **kw)
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                igc.gemm_s8_zp(A, Bt, C32=C32, C8=C8, workspace=ws, **kw)
        torch.cuda.current_stream().wait_stream(side)
        for _ in range(2):
            Ah = rng.integers(0, 256, (M, K)).astype(np.uint8)
            Bh = rng.integers(-128, 128, (N, K)).astype(np.int8)
            A.copy_(torch.from_numpy(Ah))
            Bt.copy_(torch.from_numpy(Bh))
            g.replay()
            torch.cuda.synchronize()
            check_device_ok()
            o32, o8, _, _ = oracle.gemm_s8_zp(Ah, Bh, a_signed=0, b_signed=1, **kw)
            _same(host(C32), host(C8), o32, o8)
    finally:
        igc.igc_set_int8_path(old)


def test_convert_full_size_8192_c8_sampled():
    """The benchmark's int8 problem (8192^3, uint8 A with per-row zA, int8 B,
    per-column scales, C8 alone) on the converting path: sampled rows and
    columns against the oracle, bit for bit."""
    import synth
    w = synth.workload(5)
    A = torch.from_numpy(w["A"]).cuda()
    Bt = torch.from_numpy(w["Bt"]).cuda()
    C8 = torch.empty((8192, 8192), dtype=torch.int8, device="cuda")
    d = _dev(dict(zA_row=w["zA_row"], scale_col=w["scale_col"]))
    old = igc.igc_set_int8_path(igc.INT8_PATH_CONVERT)
    try:
        igc.gemm_s8_zp(A, Bt, C8=C8, **d)
    finally:
        igc.igc_set_int8_path(old)
    check_device_ok()
    g8 = host(C8)
    del A, Bt, C8
    torch.cuda.empty_cache()
    rows = np.array([0, 1, 127, 128, 255, 4095, 4096, 5000, 8190, 8191])
    _, o8, _, ovf = oracle.gemm_s8_zp(w["A"][rows], w["Bt"], a_signed=0, b_signed=1,
                                      zA_row=w["zA_row"][rows], scale_col=w["scale_col"])
    assert not ovf
    assert np.array_equal(g8[rows], o8), "rows differ"
    cols = np.array([0, 255, 256, 8191])
    _, o8c, _, _ = oracle.gemm_s8_zp(w["A"], w["Bt"][cols], a_signed=0, b_signed=1,
                                     zA_row=w["zA_row"], scale_col=w["scale_col"][cols])
    assert np.array_equal(g8[:, cols], o8c), "columns differ"
