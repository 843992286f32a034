"""GPU parity of exactly the calls the benchmark times, at full size.

bench.Step builds the benchmark's device buffers from its seeded workloads and
run() makes the step's calls with the output variants the timed region uses:
the fp16 GEMM 4096^3 with the fp16 C alone (no fp32 copy), the 3x3 convolution
over 256 images with the fp16 y alone, and the int8 GEMM 8192^3 through
gemm_s8_zp_prepare + gemm_s8_zp_run with the requantised C8 alone.  These take
their own epilogue branches and TMA store maps, so they are checked here as
they run in the benchmark: sampled rows, columns and images against the CPU
oracle (fp16 within the stated per-element bound, int8 bit for bit), after an
L2 flush and a warm-up step like the benchmark's.
"""

import numpy as np
import pytest
import torch

import bench
import oracle
from gpu_helpers import assert_fp16_bound, check_device_ok, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def step_outputs():
    w3, w4, w5 = bench.make_inputs()
    step = bench.Step(w3, w4, w5, torch.device("cuda", 0))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(2):              # the benchmark's warm-up, then the checked step
        flush.zero_()
        step.run()
    check_device_ok()
    out = {"C3": host(step.C3), "y": host(step.y), "C8": host(step.C8)}
    del step
    torch.cuda.empty_cache()
    return (w3, w4, w5), out


def test_step_fp16_gemm_4096_fp16_c_only(step_outputs):
    (w3, _, _), out = step_outputs
    C = out["C3"]
    assert C.dtype == np.float16 and C.shape == (4096, 4096)
    rows = np.array([0, 1, 255, 256, 2047, 2048, 3071, 4094, 4095])
    ref, sabs = oracle.gemm_f16(w3["A"][rows], w3["Bt"])
    assert_fp16_bound(C[rows], ref, sabs, "fp16 GEMM rows")
    cols = np.array([0, 127, 128, 255, 256, 1000, 3967, 4095])
    ref, sabs = oracle.gemm_f16(w3["A"], w3["Bt"][cols])
    assert_fp16_bound(C[:, cols], ref, sabs, "fp16 GEMM columns")


def test_step_conv_256_images_y_only(step_outputs):
    (_, w4, _), out = step_outputs
    y = out["y"]
    assert y.dtype == np.float16 and y.shape == (256, 14, 14, 512)
    for n in (0, 1, 127, 255):
        ref, sabs = oracle.conv2d_nhwc_f16(w4["x"][n:n + 1], w4["w"], pad=(1, 1))
        assert_fp16_bound(y[n:n + 1], ref, sabs, f"conv image {n}")


def test_step_int8_gemm_8192_c8_only(step_outputs):
    (_, _, w5), out = step_outputs
    C8 = out["C8"]
    assert C8.dtype == np.int8 and C8.shape == (8192, 8192)
    rows = np.array([0, 1, 255, 256, 4095, 4096, 8191])
    _, o8, _, ovf = oracle.gemm_s8_zp(w5["A"][rows], w5["Bt"], a_signed=0, b_signed=1,
                                      zA_row=w5["zA_row"][rows], scale_col=w5["scale_col"])
    assert not ovf
    assert np.array_equal(C8[rows], o8), "int8 GEMM rows differ"
    cols = np.array([0, 1, 127, 128, 255, 256, 8190, 8191])
    _, o8, _, _ = oracle.gemm_s8_zp(w5["A"], w5["Bt"][cols], a_signed=0, b_signed=1,
                                    zA_row=w5["zA_row"], scale_col=w5["scale_col"][cols])
    assert np.array_equal(C8[:, cols], o8), "int8 GEMM columns differ"
