"""Host-side checks of the C-ABI library that need no GPU: it builds, loads,
exports every function include/igc.h declares, and rejects bad arguments on
the host before touching a device."""

import ctypes
import os
import re

import pytest

import implicit_gemm_conv_tcgen05_gb300 as igc


def test_library_loads_and_exports_every_declared_symbol():
    L = igc.lib()
    names = igc.declared_functions(igc.HEADER) + igc.declared_functions(igc.DEBUG_HEADER)
    expected = {"gemm_f16", "gemm_bf16", "gemm_s8_zp", "gemm_s8_zp_workspace_size", "gemm_s8_zp_prepare",
                "gemm_s8_zp_run", "gemm_s8_zp_dequant", "gemm_s8_zp_noalloc",
                "conv2d_nhwc_s8_zp", "conv2d_nhwc_s8_zp_workspace_size", "conv2d_nhwc_f16_implicit",
                "igc_status_string", "igc_check_device_status", "igc_last_device_status",
                "igc_set_wait_limit_ns", "igc_set_tile_width", "igc_set_stage_depth",
                "igc_set_int8_path", "igc_plan_gemm",
                "igc_debug_wait_timeout_probe",
                "igc_version"}
    assert expected <= set(names)
    for n in names:
        assert hasattr(L, n), n
        assert ctypes.cast(getattr(L, n), ctypes.c_void_p).value


def test_status_strings_and_version():
    for code in range(7):
        s = igc.status_string(code)
        assert s and s != "unknown status"
    assert igc.status_string(99) == "unknown status"
    assert re.fullmatch(r"\d+\.\d+\.\d+", igc.igc_version())


def test_workspace_size_arithmetic():
    # A' (M x Kp fp16) + B' (N x Kp fp16) + row sums + column sums, then the
    # converting kernel's flags (one per 128-row block and 1024-k chunk, one per
    # block) and its job counter, each 256-aligned
    def up(v):
        return (v + 255) // 256 * 256
    for M, N, K in [(1024, 1024, 1024), (8192, 8192, 8192), (3, 5, 7), (1, 1, 1),
                    (300, 200, 2064)]:
        Kp = (K + 7) // 8 * 8
        chunks = (K + 1023) // 1024
        blocks = (M + 127) // 128 + (N + 127) // 128
        want = (up(M * Kp * 2) + up(N * Kp * 2) + up(4 * M) + up(4 * N) +
                up(4 * (blocks * chunks + blocks + 1)))
        assert igc.gemm_s8_zp_workspace_size(M, N, K) == want
    assert igc.gemm_s8_zp_workspace_size(-1, 2, 3) == 0


def test_wait_limit_setter_roundtrip():
    old = igc.igc_set_wait_limit_ns(5_000_000)
    assert igc.igc_set_wait_limit_ns(10) == 5_000_000      # returns the previous value
    assert igc.igc_set_wait_limit_ns(old) == 1000          # raised to the 1 us floor
    assert igc.igc_set_wait_limit_ns(old) == old


def test_host_validation_before_any_device_call():
    L = igc.lib()
    dummy = ctypes.c_void_p(4096)
    # negative sizes, bad output type, no outputs: rejected on the host
    assert L.gemm_f16(-1, 4, 4, dummy, 4, dummy, 4, dummy, 4, 0, None, 0, None) == igc.IGC_ERR_INVALID_ARG
    assert L.gemm_f16(4, 4, 4, dummy, 4, dummy, 4, dummy, 4, 7, None, 0, None) == igc.IGC_ERR_INVALID_ARG
    assert L.gemm_f16(4, 4, 4, dummy, 4, dummy, 4, None, 0, 0, None, 0, None) == igc.IGC_ERR_INVALID_ARG
    assert L.gemm_f16(4, 4, 4, dummy, 4, dummy, 4, dummy, 3, 0, None, 0, None) == igc.IGC_ERR_INVALID_ARG
    # empty problems are a no-op, even with null operands and outputs (empty tensors)
    assert L.gemm_f16(0, 8, 16, None, 16, None, 16, None, 8, 0, None, 0, None) == igc.IGC_OK
    assert L.gemm_f16(8, 0, 16, None, 16, None, 16, None, 0, 1, None, 0, None) == igc.IGC_OK
    assert L.gemm_s8_zp(0, 8, 16, None, 0, 16, None, 0, 16, 0, None, 0, None,
                        None, 8, None, 8, 1.0, None, None, 0, None) == igc.IGC_OK
    assert L.conv2d_nhwc_f16_implicit(0, 4, 4, 8, 8, 3, 3, 1, 1, 1, 1, None, None, None, None,
                                      None) == igc.IGC_OK
    assert L.gemm_f16(0, 4, 4, None, 4, None, 4, dummy, 4, 0, None, 0, None) == igc.IGC_OK
    assert L.gemm_f16(4, 0, 4, None, 4, None, 4, dummy, 4, 0, None, 0, None) == igc.IGC_OK
    assert L.gemm_s8_zp(-3, 4, 4, dummy, 0, 16, dummy, 0, 16, 0, None, 0, None,
                        dummy, 4, None, 0, 1.0, None, None, 0, None) == igc.IGC_ERR_INVALID_ARG
    assert L.gemm_s8_zp(4, 4, 4, dummy, 0, 16, dummy, 0, 16, 0, None, 0, None,
                        None, 0, None, 0, 1.0, None, None, 0, None) == igc.IGC_ERR_INVALID_ARG
    assert L.gemm_s8_zp(0, 4, 4, None, 0, 16, None, 0, 16, 0, None, 0, None,
                        dummy, 4, None, 0, 1.0, None, None, 0, None) == igc.IGC_OK
    conv = L.conv2d_nhwc_f16_implicit
    assert conv(1, 14, 14, 256, 512, 3, 3, -1, 1, 1, 1, dummy, dummy, dummy, None, None) == igc.IGC_ERR_INVALID_ARG
    assert conv(1, 2, 2, 8, 8, 5, 5, 0, 0, 1, 1, dummy, dummy, dummy, None, None) == igc.IGC_ERR_INVALID_ARG
    assert conv(1, 14, 14, 256, 512, 3, 3, 1, 1, 1, 1, dummy, dummy, None, None, None) == igc.IGC_ERR_INVALID_ARG
    assert conv(0, 14, 14, 256, 512, 3, 3, 1, 1, 1, 1, None, None, dummy, None, None) == igc.IGC_OK
    # stride and channel-count limits are reported as unsupported before any device call
    assert conv(1, 14, 14, 256, 512, 3, 3, 1, 1, 9, 9, dummy, dummy, dummy, None, None) == igc.IGC_ERR_UNSUPPORTED
    # int8 convolution: the padding value must be a value of the input type
    c8 = L.conv2d_nhwc_s8_zp
    assert c8(1, 8, 8, 16, 16, 3, 3, 1, 1, 1, 1, dummy, 0, 300, dummy, 1, 0, None, dummy, None,
              1.0, None, dummy, 1 << 30, None) == igc.IGC_ERR_INVALID_ARG
    assert L.conv2d_nhwc_s8_zp_workspace_size(1, 8, 8, 12, 16, 3, 3, 1, 1, 1, 1) == 0
    assert conv(1, 14, 14, 12, 512, 3, 3, 1, 1, 1, 1, dummy, dummy, dummy, None, None) == igc.IGC_ERR_UNSUPPORTED


def test_header_declares_c_linkage_and_statuses():
    with open(igc.HEADER) as f:
        text = f.read()
    assert 'extern "C"' in text
    for name, code in [("IGC_OK", 0), ("IGC_ERR_INVALID_ARG", 1), ("IGC_ERR_MISALIGNED", 2),
                       ("IGC_ERR_UNSUPPORTED", 3), ("IGC_ERR_CUDA", 4), ("IGC_ERR_DEVICE_TIMEOUT", 5),
                       ("IGC_ERR_WORKSPACE", 6), ("IGC_F32", 0), ("IGC_F16", 1), ("IGC_BF16", 2)]:
        assert re.search(rf"#define {name} {code}\b", text)
        assert getattr(igc, name) == code


def test_tile_width_setter_roundtrip():
    assert igc.igc_set_tile_width(224) == 0
    assert igc.igc_set_tile_width(96) == -1          # not a built width: unchanged
    assert igc.igc_set_tile_width(128) == 224
    assert igc.igc_set_tile_width(0) == 128


def test_int8_path_setter_roundtrip():
    assert igc.igc_set_int8_path(igc.INT8_PATH_MMA_SYNC) == igc.INT8_PATH_TCGEN05
    assert igc.igc_set_int8_path(4) == -1            # no such path: unchanged
    assert igc.igc_set_int8_path(igc.INT8_PATH_FUSED) == igc.INT8_PATH_MMA_SYNC
    assert igc.igc_set_int8_path(igc.INT8_PATH_CONVERT) == igc.INT8_PATH_FUSED
    assert igc.igc_set_int8_path(igc.INT8_PATH_TCGEN05) == igc.INT8_PATH_CONVERT


def test_stage_depth_setter_roundtrip():
    assert igc.igc_set_stage_depth(64) == 0
    assert igc.igc_set_stage_depth(96) == -1         # not a built depth: unchanged
    assert igc.igc_set_stage_depth(128) == 64
    assert igc.igc_set_stage_depth(0) == 128


def test_header_is_c99_and_links_from_c(tmp_path):
    """A C99 program includes include/igc.h, links libigc.so and calls the host-only
    entry points (no GPU): the boundary is a plain C ABI."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    lib = igc.lib()._name
    src = tmp_path / "use_igc.c"
    src.write_text(
        '#include <string.h>\n#include "igc.h"\n#include "igc_debug.h"\n'
        "int main(void) {\n"
        "  int32_t out[8];\n"
        "  if (igc_plan_gemm(IGC_PLAN_GEMM_F16, 4096, 4096, 4096, 76, out) != IGC_OK) return 1;\n"
        "  if (out[0] != 256 || out[4] != 228 || out[5] != 284) return 2;\n"
        "  if (gemm_s8_zp_workspace_size(-1, 1, 1) != 0) return 3;\n"
        "  if (strlen(igc_status_string(IGC_ERR_MISALIGNED)) == 0) return 4;\n"
        "  if (igc_set_tile_width(96) != -1) return 5;\n"
        "  return 0;\n}\n")
    exe = tmp_path / "use_igc"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", inc, str(src), lib, "-o", str(exe),
                    f"-Wl,-rpath,{os.path.dirname(lib)}"], check=True)
    assert subprocess.run([str(exe)]).returncode == 0


def test_headers_declare_exactly_the_boundary_and_the_debug_hooks():
    """include/igc.h holds the operations of the path and their documented
    companions only; the schedule-forcing test hooks live in include/igc_debug.h."""
    product = {"gemm_f16", "gemm_bf16", "gemm_s8_zp", "gemm_s8_zp_workspace_size",
               "gemm_s8_zp_prepare", "gemm_s8_zp_run", "gemm_s8_zp_dequant",
               "gemm_s8_zp_noalloc", "conv2d_nhwc_f16_implicit", "conv2d_nhwc_s8_zp",
               "conv2d_nhwc_s8_zp_workspace_size", "igc_status_string",
               "igc_check_device_status", "igc_last_device_status", "igc_set_wait_limit_ns",
               "igc_plan_gemm", "igc_version"}
    debug = {"igc_set_tile_width", "igc_set_stage_depth", "igc_set_int8_path",
             "igc_debug_wait_timeout_probe"}
    assert set(igc.declared_functions(igc.HEADER)) == product
    assert set(igc.declared_functions(igc.DEBUG_HEADER)) == debug
    L = igc.lib()
    for n in product | debug:
        assert ctypes.cast(getattr(L, n), ctypes.c_void_p).value, n


def test_schedule_hooks_are_thread_local():
    """A hook set on one thread is invisible to calls made on another thread."""
    import threading
    seen = {}

    def other():
        # a fresh thread starts at the defaults and its settings stay its own
        seen["width"] = igc.igc_set_tile_width(128)
        seen["depth"] = igc.igc_set_stage_depth(64)
        seen["path"] = igc.igc_set_int8_path(igc.INT8_PATH_MMA_SYNC)
        seen["plan"] = igc.igc_plan_gemm(igc.PLAN_GEMM_F16, 4096, 4096, 4096, clusters=76)

    assert igc.igc_set_tile_width(224) == 0
    assert igc.igc_set_stage_depth(128) == 0
    assert igc.igc_set_int8_path(igc.INT8_PATH_TCGEN05) == 0
    try:
        th = threading.Thread(target=other)
        th.start()
        th.join()
        assert seen["width"] == 0 and seen["depth"] == 0 and seen["path"] == 0
        assert seen["plan"]["tile_width"] == 128 and seen["plan"]["stage_k"] == 64
        # this thread's settings were not touched by the other thread
        plan = igc.igc_plan_gemm(igc.PLAN_GEMM_F16, 4096, 4096, 4096, clusters=76)
        assert plan["tile_width"] == 224 and plan["stage_k"] == 128
        assert igc.igc_set_tile_width(0) == 224
        assert igc.igc_set_stage_depth(0) == 128
    finally:
        igc.igc_set_tile_width(0)
        igc.igc_set_stage_depth(0)
        igc.igc_set_int8_path(igc.INT8_PATH_TCGEN05)


def test_binding_checks_outputs_and_vectors_before_the_device():
    """Short or mistyped outputs and vectors raise on the host: the C entry points
    take raw pointers and cannot see a buffer's length."""
    import torch
    A = torch.zeros((64, 32), dtype=torch.uint8)
    Bt = torch.zeros((48, 32), dtype=torch.int8)
    ws = torch.zeros(igc.gemm_s8_zp_workspace_size(64, 48, 32), dtype=torch.uint8)
    C8 = torch.zeros((64, 48), dtype=torch.int8)
    short8 = torch.zeros((63, 48), dtype=torch.int8)
    short32 = torch.zeros((64, 47), dtype=torch.int32)
    with pytest.raises(ValueError, match="C8 has shape"):
        igc.gemm_s8_zp_run(64, 48, 32, 0, 1, ws, C8=short8, scale=1.0)
    with pytest.raises(ValueError, match="C32 has shape"):
        igc.gemm_s8_zp_run(64, 48, 32, 0, 1, ws, C32=short32)
    with pytest.raises(TypeError, match="C8 has dtype"):
        igc.gemm_s8_zp_run(64, 48, 32, 0, 1, ws, C8=C8.view(torch.uint8), scale=1.0)
    with pytest.raises(ValueError, match="scale_col must be"):
        igc.gemm_s8_zp_run(64, 48, 32, 0, 1, ws, C8=C8, scale_col=torch.ones(47))
    with pytest.raises(ValueError, match="zA_row must be"):
        igc.gemm_s8_zp_run(64, 48, 32, 0, 1, ws, C8=C8, scale=1.0,
                           zA_row=torch.zeros(64, dtype=torch.int64))
    with pytest.raises(ValueError, match="zB_col must be"):
        igc.gemm_s8_zp_run(64, 48, 32, 0, 1, ws, C8=C8, scale=1.0,
                           zB_col=torch.zeros(49, dtype=torch.int32))
    # the same checks on the no-allocation entry point and the combined call
    for fn in (igc.gemm_s8_zp_noalloc, igc.gemm_s8_zp):
        with pytest.raises(ValueError, match="C8 has shape"):
            fn(A, Bt, C8=short8, scale=1.0)
        with pytest.raises(ValueError, match="scale_col must be"):
            fn(A, Bt, C8=C8, scale_col=torch.ones(50))
    # right shapes and dtypes, host memory: rejected as not being CUDA tensors
    with pytest.raises(ValueError, match="CUDA"):
        igc.gemm_s8_zp_run(64, 48, 32, 0, 1, ws, C8=C8, scale=1.0)
    with pytest.raises(ValueError, match="Y has shape"):
        igc.gemm_s8_zp_dequant(A, Bt, Y=torch.zeros((64, 47), dtype=torch.float32))


def test_binding_fails_loudly_without_the_library(tmp_path):
    """With no libigc.so (and none that can be built) every entry point raises:
    there is no CPU fallback that could return a value instead."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    missing = os.path.join(str(tmp_path), "missing", "libigc.so")
    code = (
        "import implicit_gemm_conv_tcgen05_gb300.build as b\n"
        f"b.build = lambda *a, **k: {missing!r}\n"
        "import implicit_gemm_conv_tcgen05_gb300 as igc\n"
        "calls = [lambda: igc.igc_version(), lambda: igc.gemm_s8_zp_workspace_size(8, 8, 8),\n"
        "         lambda: igc.igc_plan_gemm(igc.PLAN_GEMM_F16, 256, 256, 256, 76)]\n"
        "for c in calls:\n"
        "    try:\n"
        "        c()\n"
        "    except ImportError:\n"
        "        continue\n"
        "    raise SystemExit('a call returned without the library')\n"
        "print('all raised')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "all raised" in r.stdout
