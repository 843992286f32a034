"""The failure path without a GPU fault: a kernel whose wait can never complete
gives up after a short limit, records IGC_ERR_DEVICE_TIMEOUT, and the context
stays usable."""

import numpy as np
import pytest
import torch

import implicit_gemm_conv_tcgen05_gb300 as igc
import oracle
import synth
from gpu_helpers import assert_fp16_bound, dev, host

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    assert igc.igc_check_device_status() == igc.IGC_OK
    old = igc.igc_set_wait_limit_ns(50_000_000)  # 50 ms
    try:
        assert igc.igc_debug_wait_timeout_probe() == igc.IGC_OK
        assert igc.igc_check_device_status() == igc.IGC_ERR_DEVICE_TIMEOUT
        word = igc.igc_last_device_status()
        assert word >> 56 == 1 and (word >> 32) & 0xFFFFFF == 0xABCD
        assert igc.igc_check_device_status() == igc.IGC_OK   # cleared by the read
    finally:
        igc.igc_set_wait_limit_ns(old)
    # the context still works
    A = synth.uniform_f16(1, 1, (128, 64))
    Bt = synth.uniform_f16(1, 2, (256, 64))
    C = igc.gemm_f16(dev(A), dev(Bt))
    assert igc.igc_check_device_status() == igc.IGC_OK
    ref, sabs = oracle.gemm_f16(A, Bt)
    assert_fp16_bound(host(C), ref, sabs, "after timeout")
