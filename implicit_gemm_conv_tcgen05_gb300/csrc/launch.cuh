// Shared launch code for the tcgen05 GEMM kernel template.
#pragma once

#include <mutex>

#include "gemm_tc.cuh"
#include "igc_host.h"

namespace igc {

template <Mode kMode>
int launch_tc_gemm(const DeviceInfo& dev, const CUtensorMap& tmA, const CUtensorMap& tmB,
                   KParams p, cudaStream_t stream) {
  static std::once_flag attr_once[64];
  static int attr_rc[64];
  const int d = dev.device;
  std::call_once(attr_once[d], [&] {
    attr_rc[d] = cudaFuncSetAttribute(igc_tc_gemm_kernel<kMode>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kSmemBytes)) == cudaSuccess
                     ? IGC_OK
                     : IGC_ERR_CUDA;
  });
  if (attr_rc[d] != IGC_OK) return attr_rc[d];
  if (dev.smem_optin < kSmemBytes) return IGC_ERR_UNSUPPORTED;

  p.tiles_m = static_cast<int>((static_cast<long long>(p.M) + BM - 1) / BM);
  p.tiles_n = static_cast<int>((static_cast<long long>(p.N) + BN - 1) / BN);
  const long long tiles = static_cast<long long>(p.tiles_m) * p.tiles_n;
  if (tiles > 0x7fffffffLL) return IGC_ERR_UNSUPPORTED;
  p.num_tiles = static_cast<int>(tiles);
  p.group_m = p.tiles_m < 16 ? p.tiles_m : 16;
  p.wait_limit_ns = wait_limit_ns();
  p.status = status_word();
  const int grid = p.num_tiles < dev.sm_count ? p.num_tiles : dev.sm_count;
  igc_tc_gemm_kernel<kMode><<<grid, kThreads, kSmemBytes, stream>>>(tmA, tmB, p);
  return cudaGetLastError() == cudaSuccess ? IGC_OK : IGC_ERR_CUDA;
}

// Zero an M x N row-major output (K == 0 case: an empty sum is 0).
inline int zero_rows(void* ptr, long long ld, long long rows, long long cols, size_t esize,
                     cudaStream_t stream) {
  if (!ptr) return IGC_OK;
  return cudaMemset2DAsync(ptr, static_cast<size_t>(ld) * esize, 0,
                           static_cast<size_t>(cols) * esize, static_cast<size_t>(rows),
                           stream) == cudaSuccess
             ? IGC_OK
             : IGC_ERR_CUDA;
}

inline bool vec_store_ok(const void* p, long long ld, size_t esize) {
  return p == nullptr || (aligned16(p) && (static_cast<unsigned long long>(ld) * esize) % 16 == 0);
}

}  // namespace igc
