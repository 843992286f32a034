// Host-side helpers shared by the entry points of libigc.so (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "igc.h"
#include "igc_debug.h"

namespace igc {

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  size_t smem_optin = 0;
};

// Current device's properties (cached per device).  Returns IGC_OK,
// IGC_ERR_CUDA, or IGC_ERR_UNSUPPORTED when the device is not sm_103.
int current_device(DeviceInfo* out);

// Device address of the status word of the current device.
unsigned long long* status_word();

// Wait limit for kernels launched now.
unsigned long long wait_limit_ns();
// The calling thread's schedule overrides (test hooks of igc_debug.h).
int tile_width_override();   // 0, or the tile width set by igc_set_tile_width
int stage_depth_override();  // 0, or the stage depth set by igc_set_stage_depth
int int8_path_override();    // 0 (tcgen05) or 1 (mma.sync), set by igc_set_int8_path

// gemm_s8_zp on the warp-level (mma.sync) tensor path; arguments checked by the caller
int imma_gemm_s8_zp(int M, int N, int K, const void* A, int a_signed, long long lda,
                    const void* Bt, int b_signed, long long ldb, int32_t zA,
                    const int32_t* zA_row, int32_t zB, const int32_t* zB_col, int32_t* C32,
                    long long ldc32, int8_t* C8, long long ldc8, float scale,
                    const float* scale_col, int32_t* rA, int32_t* cB, cudaStream_t stream);

// cuTensorMapEncodeTiled / cuTensorMapEncodeIm2col through the runtime's
// driver entry point (the library does not link libcuda directly).
int encode_tiled_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    uint64_t inner, uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner,
                    uint32_t box_rows);

// The same with a chosen swizzle (encode_tiled_2d: 128-byte).
int encode_tiled_2d_swizzle(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                            uint64_t inner, uint64_t rows, uint64_t row_stride_bytes,
                            uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle);

int encode_im2col_nhwc(CUtensorMap* map, const void* base, int N, int H, int W, int C,
                       int lower_h, int lower_w, int upper_h, int upper_w, uint32_t channels,
                       uint32_t pixels, int stride_h, int stride_w);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launches a non-cluster kernel with programmatic stream serialization: it may
// start while the previous kernel in the stream runs and waits for it in the
// kernel (griddepcontrol.wait) before touching memory.
template <typename... Params, typename... Args>
int launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
               Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...) != cudaSuccess) {
    (void)cudaGetLastError();
    return IGC_ERR_CUDA;
  }
  return IGC_OK;
}

}  // namespace igc
