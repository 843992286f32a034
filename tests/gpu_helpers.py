"""Shared helpers of the GPU parity tests (inputs come from synth, expected
values from the CPU oracle; the GPU results come through the C-ABI binding)."""

import numpy as np
import torch

import oracle

REL_TOL = 2e-3  # per element: |gpu - exact| <= 2e-3 * sum_k |a_ik * b_kj|


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    return t.cpu().numpy()


def assert_fp16_bound(gpu: np.ndarray, ref: np.ndarray, sabs: np.ndarray, what: str):
    ok, worst = oracle.fp16_accept(gpu, ref, sabs, REL_TOL)
    assert ok, f"{what}: error bound exceeded, worst |err|/(2e-3*sabs) = {worst:.3g}"


def assert_f16_is_rne_of_f32(c16: np.ndarray, c32: np.ndarray, what: str):
    want = oracle.f32_to_f16_array(c32).view(np.uint16)
    got = np.ascontiguousarray(c16).view(np.uint16)
    bad = np.count_nonzero(got != want)
    assert bad == 0, f"{what}: {bad} fp16 outputs are not the RNE rounding of the fp32 copy"


def check_device_ok():
    import implicit_gemm_conv_tcgen05_gb300 as igc
    rc = igc.igc_check_device_status()
    assert rc == igc.IGC_OK, f"device status {igc.status_string(rc)} ({igc.igc_last_device_status():#x})"
