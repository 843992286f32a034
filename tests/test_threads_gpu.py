"""Calls made from several host threads at once, each thread on its own stream, with
its own schedule hooks: the library's host state (per-thread tensor-map cache and
hooks, per-device set-up done once) must keep every call's result the same as the
same call made alone.  Each thread's results are compared bit for bit with the
results of the identical calls made beforehand on one thread (the kernels are
deterministic for a given schedule), and those with the oracle."""

import threading

import numpy as np
import pytest
import torch

import implicit_gemm_conv_tcgen05_gb300 as igc
import oracle
from gpu_helpers import check_device_ok

pytestmark = pytest.mark.gpu

THREADS, CALLS = 4, 12


def _case(t, i):
    """Call i of thread t: an operation, its inputs and forced schedule (as a closure
    that writes fresh outputs on the current stream) and its oracle result, chosen
    so that threads mix operations and hooks."""
    rng = np.random.default_rng(1000 * t + i)
    kind = (t + i) % 3
    if kind == 0:
        M, N = int(rng.integers(64, 1500)), int(rng.integers(64, 1500))
        K = 8 * int(rng.integers(8, 200))
        A = torch.from_numpy(rng.integers(-2, 3, size=(M, K)).astype(np.float16)).cuda()
        Bt = torch.from_numpy(rng.integers(-2, 3, size=(N, K)).astype(np.float16)).cuda()
        width = int(rng.choice([0, 128, 224, 256]))

        def run():
            C = torch.empty((M, N), dtype=torch.float32, device="cuda")
            old = igc.igc_set_tile_width(width)
            try:
                igc.gemm_f16(A, Bt, C)
            finally:
                igc.igc_set_tile_width(old)
            return [C]

        def ref():
            return [oracle.gemm_f16(A.cpu().numpy(), Bt.cpu().numpy())[0].astype(np.float32)]
        return run, ref
    if kind == 1:
        M, N = int(rng.integers(64, 1500)), int(rng.integers(64, 1500))
        K = 16 * int(rng.integers(4, 100))
        A = torch.from_numpy(rng.integers(0, 256, size=(M, K)).astype(np.uint8)).cuda()
        Bt = torch.from_numpy(rng.integers(-128, 128, size=(N, K)).astype(np.int8)).cuda()
        zA = torch.from_numpy(rng.integers(0, 256, size=M).astype(np.int32)).cuda()
        sc = torch.from_numpy(rng.uniform(1e-6, 1e-4, size=N).astype(np.float32)).cuda()
        # (not the converting path: its CTAs wait on each other's conversion jobs, so it
        # needs all of them resident, which concurrent launches on other streams do
        # not leave it)
        path = int(rng.choice([0, 0, 1, 2]))

        def run():
            C32 = torch.empty((M, N), dtype=torch.int32, device="cuda")
            C8 = torch.empty((M, N), dtype=torch.int8, device="cuda")
            ws = torch.empty(igc.gemm_s8_zp_workspace_size(M, N, K), dtype=torch.uint8,
                             device="cuda")
            old = igc.igc_set_int8_path(path)
            try:
                igc.gemm_s8_zp(A, Bt, zA_row=zA, zB=5, C32=C32, C8=C8, scale_col=sc,
                               workspace=ws)
            finally:
                igc.igc_set_int8_path(old)
            return [C32, C8]

        def ref():
            o32, o8, _, _ = oracle.gemm_s8_zp(A.cpu().numpy(), Bt.cpu().numpy(), a_signed=0,
                                              b_signed=1, zA_row=zA.cpu().numpy(), zB=5,
                                              scale_col=sc.cpu().numpy())
            return [o32, o8]
        return run, ref
    n, H = int(rng.integers(1, 4)), int(rng.integers(5, 16))
    C, K = 8 * int(rng.integers(1, 32)), 8 * int(rng.integers(1, 40))
    x = torch.from_numpy(rng.integers(-2, 3, size=(n, H, H, C)).astype(np.float16)).cuda()
    w = torch.from_numpy(rng.integers(-1, 2, size=(K, 3, 3, C)).astype(np.float16)).cuda()
    stride = int(rng.integers(1, 3))
    P = (H + 2 - 3) // stride + 1

    def run():
        y32 = torch.empty((n, P, P, K), dtype=torch.float32, device="cuda")
        igc.conv2d_nhwc_f16_implicit(x, w, None, y32, pad=(1, 1), stride=(stride, stride))
        return [y32]

    def ref():
        r, _ = oracle.conv2d_nhwc_f16(x.cpu().numpy(), w.cpu().numpy(), pad=(1, 1),
                                      stride=(stride, stride))
        return [r.astype(np.float32)]
    return run, ref


def test_calls_from_several_threads_and_streams():
    cases = [[_case(t, i) for i in range(CALLS)] for t in range(THREADS)]
    # the same calls on one thread, one after the other
    alone = [[[o.cpu().numpy() for o in run()] for run, _ in row] for row in cases]
    torch.cuda.synchronize()
    check_device_ok()
    for row, outs in zip(cases, alone):
        for (_, ref), got in zip(row, outs):
            for g, want in zip(got, ref()):
                assert np.array_equal(g, want)
    results = [[None] * CALLS for _ in range(THREADS)]
    errors = []
    start = threading.Barrier(THREADS)

    def worker(t):
        try:
            # allocations and calls on the thread's own stream, so that no buffer is
            # reused while a call on another stream may still use it
            stream = torch.cuda.Stream()
            start.wait()
            with torch.cuda.stream(stream):
                outs = [run() for run, _ in cases[t]]
            stream.synchronize()
            results[t] = [[o.cpu().numpy() for o in out] for out in outs]
        except Exception as e:  # reported below, on the test's thread
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(THREADS)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    check_device_ok()
    for t in range(THREADS):
        for i in range(CALLS):
            for g, want in zip(results[t][i], alone[t][i]):
                assert np.array_equal(g, want), (t, i)
