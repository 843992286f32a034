"""gemm_s8_zp_noalloc: the int8 zero-point GEMM for callers that cannot
allocate device memory (it runs on the library's own fixed scratch array
instead of a caller-provided workspace).

The entry point is called through the C ABI directly and its int32 and int8
outputs are compared with those of gemm_s8_zp (which takes a workspace) and
with the CPU oracle on two calls in a row with different problems, bit for
bit (the int8 path is exact).  A further test checks the property callers
rely on: once the first call on the device has loaded the library's int8
module (which reserves the fixed array), a call takes no device memory.
This file is collected last on purpose: it must pass on its own in a fresh
process and after every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import implicit_gemm_conv_tcgen05_gb300 as igc
import oracle

pytestmark = pytest.mark.gpu


def _call_noalloc(A, Bt, zA, zA_row, zB, zB_col, C32, C8, scale, scale_col):
    L = igc.lib()
    M, K = A.shape
    N = Bt.shape[0]
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.gemm_s8_zp_noalloc(M, N, K, p(A), int(A.dtype == torch.int8), A.stride(0),
                                p(Bt), int(Bt.dtype == torch.int8), Bt.stride(0),
                                zA, p(zA_row), zB, p(zB_col), p(C32), N, p(C8), N,
                                ctypes.c_float(scale), p(scale_col), stream)


def _case(seed, M, N, K, a_signed, b_signed, per_row):
    g = torch.Generator().manual_seed(seed)
    if a_signed:
        A = torch.randint(-128, 128, (M, K), generator=g, dtype=torch.int8)
    else:
        A = torch.randint(0, 256, (M, K), generator=g, dtype=torch.uint8)
    if b_signed:
        Bt = torch.randint(-128, 128, (N, K), generator=g, dtype=torch.int8)
    else:
        Bt = torch.randint(0, 256, (N, K), generator=g, dtype=torch.uint8)
    kw = dict(zA=int(torch.randint(0, 200, (1,), generator=g)), zA_row=None,
              zB=int(torch.randint(0, 200, (1,), generator=g)), zB_col=None,
              scale=2.0 ** -12, scale_col=None)
    if per_row:
        kw["zA_row"] = torch.randint(100, 157, (M,), generator=g, dtype=torch.int32).cuda()
        kw["zB_col"] = torch.randint(-20, 20, (N,), generator=g, dtype=torch.int32).cuda()
        kw["scale_col"] = (torch.rand(N, generator=g) * 9e-4 + 1e-4).float().cuda()
    return A.cuda(), Bt.cuda(), kw


@pytest.mark.parametrize("first,second", [
    ((1, 1024, 1024, 1024, 0, 0, False), (2, 768, 1280, 528, 0, 1, True)),
])
def test_noalloc_matches_workspace_entry_point_on_two_calls(first, second):
    for case in (first, second):
        A, Bt, kw = _case(*case)
        M, N = A.shape[0], Bt.shape[0]
        want32 = torch.empty((M, N), dtype=torch.int32, device="cuda")
        want8 = torch.empty((M, N), dtype=torch.int8, device="cuda")
        igc.gemm_s8_zp(A, Bt, C32=want32, C8=want8, **kw)
        got32 = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
        got8 = torch.full((M, N), -7, dtype=torch.int8, device="cuda")
        rc = _call_noalloc(A, Bt, kw["zA"], kw["zA_row"], kw["zB"], kw["zB_col"], got32, got8,
                           kw["scale"], kw["scale_col"])
        assert rc == igc.IGC_OK, igc.status_string(rc)
        assert igc.igc_check_device_status() == igc.IGC_OK
        torch.cuda.synchronize()
        assert torch.equal(got32, want32), f"C32 differs for case {case}"
        assert torch.equal(got8, want8), f"C8 differs for case {case}"
        o32, o8, _, _ = oracle.gemm_s8_zp(
            A.cpu().numpy(), Bt.cpu().numpy(), a_signed=int(A.dtype == torch.int8),
            b_signed=int(Bt.dtype == torch.int8), zA=kw["zA"],
            zA_row=None if kw["zA_row"] is None else kw["zA_row"].cpu().numpy(),
            zB=kw["zB"], zB_col=None if kw["zB_col"] is None else kw["zB_col"].cpu().numpy(),
            scale=kw["scale"],
            scale_col=None if kw["scale_col"] is None else kw["scale_col"].cpu().numpy())
        assert np.array_equal(got32.cpu().numpy(), o32), f"C32 differs from the oracle, {case}"
        assert np.array_equal(got8.cpu().numpy(), o8), f"C8 differs from the oracle, {case}"


def test_noalloc_takes_no_device_memory_after_its_first_call():
    """A warm-up call loads the module (reserving the fixed array); a second call
    on another shape then leaves the device's free memory and torch's allocator
    exactly as they were."""
    A, Bt, kw = _case(3, 512, 640, 1024, 0, 1, True)
    C32 = torch.empty((512, 640), dtype=torch.int32, device="cuda")
    C8 = torch.empty((512, 640), dtype=torch.int8, device="cuda")
    assert _call_noalloc(A, Bt, kw["zA"], kw["zA_row"], kw["zB"], kw["zB_col"], C32, C8,
                         kw["scale"], kw["scale_col"]) == igc.IGC_OK
    A2, Bt2, kw2 = _case(4, 1536, 768, 2048, 1, 0, False)
    D32 = torch.empty((1536, 768), dtype=torch.int32, device="cuda")
    D8 = torch.empty((1536, 768), dtype=torch.int8, device="cuda")
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    reserved0 = torch.cuda.memory_reserved()
    for _ in range(2):
        assert _call_noalloc(A2, Bt2, kw2["zA"], kw2["zA_row"], kw2["zB"], kw2["zB_col"], D32,
                             D8, kw2["scale"], kw2["scale_col"]) == igc.IGC_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.memory_reserved() == reserved0
    assert igc.igc_check_device_status() == igc.IGC_OK


def test_noalloc_rejects_problems_beyond_its_scratch():
    M = N = K = 4096                      # needs 64 MiB of scratch, more than the fixed array
    assert igc.gemm_s8_zp_workspace_size(M, N, K) > igc.IGC_NOALLOC_SCRATCH_BYTES
    A = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    Bt = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    C32 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    rc = _call_noalloc(A, Bt, 0, None, 0, None, C32, None, 1.0, None)
    assert rc == igc.IGC_ERR_WORKSPACE
    # a bad argument is reported as such whatever the size
    assert _call_noalloc(A, Bt, 0, None, 0, None, None, None, 1.0, None) == \
        igc.IGC_ERR_INVALID_ARG
