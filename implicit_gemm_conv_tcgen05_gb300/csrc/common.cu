// Host plumbing shared by every entry point: device checks, the device status
// word, tensor-map encoding through the driver entry point, status strings and
// the wait-timeout diagnostic.
#include <atomic>
#include <cstdio>
#include <mutex>

#include "igc_host.h"
#include "sm100_ptx.cuh"

namespace igc {

namespace {

constexpr int kMaxDevices = 64;

// One status word per device (each device that loads the module gets its own copy).
__device__ unsigned long long g_status_word;

std::atomic<unsigned long long> g_wait_limit{2000000000ull};
// Schedule overrides of the test hooks (igc_debug.h): per thread, so that a
// thread that forces a schedule never changes another thread's calls.
thread_local int t_tile_width = 0;   // 0: chosen per problem
thread_local int t_stage_depth = 0;  // 0: chosen per problem
thread_local int t_int8_path = 0;    // IGC_INT8_PATH_*
std::atomic<unsigned long long> g_last_status{0};

struct DeviceSlot {
  std::once_flag once;
  DeviceInfo info;
  int rc = IGC_ERR_CUDA;
  unsigned long long* status = nullptr;
};
DeviceSlot g_slots[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
using EncodeIm2colFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const int*,
                                    const int*, cuuint32_t, cuuint32_t, const cuuint32_t*,
                                    CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode_tiled = nullptr;
EncodeIm2colFn g_encode_im2col = nullptr;

void load_encoders() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode_tiled = reinterpret_cast<EncodeTiledFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode_im2col = reinterpret_cast<EncodeIm2colFn>(fn);
  });
}

// Waits on an mbarrier that nothing completes; gives up after the limit.
__global__ void wait_timeout_probe_kernel(unsigned long long limit_ns,
                                          unsigned long long* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, limit_ns, &abort_flag, status, 0xABCDu);
}

}  // namespace

int current_device(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IGC_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return IGC_ERR_UNSUPPORTED;
  DeviceSlot& s = g_slots[dev];
  std::call_once(s.once, [&] {
    DeviceInfo d;
    d.device = dev;
    int v = 0;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
      s.rc = IGC_ERR_CUDA;
      return;
    }
    d.smem_optin = static_cast<size_t>(v);
    s.info = d;
    if (d.cc_major != 10 || d.cc_minor != 3) {
      s.rc = IGC_ERR_UNSUPPORTED;
      return;
    }
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) {
      s.rc = IGC_ERR_CUDA;
      return;
    }
    s.status = static_cast<unsigned long long*>(addr);
    s.rc = IGC_OK;
  });
  if (out) *out = s.info;
  return s.rc;
}

unsigned long long* status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  return g_slots[dev].status;
}

unsigned long long wait_limit_ns() { return g_wait_limit.load(); }

int tile_width_override() { return t_tile_width; }

int stage_depth_override() { return t_stage_depth; }

int int8_path_override() { return t_int8_path; }

int encode_tiled_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    uint64_t inner, uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner,
                    uint32_t box_rows) {
  return encode_tiled_2d_swizzle(map, dtype, base, inner, rows, row_stride_bytes, box_inner,
                                 box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

namespace {

// Tensor maps are pure functions of their arguments (address, extents, stride,
// box, swizzle), so the ones a thread encoded recently are kept and reused:
// repeated calls on the same buffers skip the driver's encode.  Direct-mapped,
// per thread (no locking); a slot holds the full key it was encoded from.
struct TiledKey {
  uint64_t base, inner, rows, stride;
  uint32_t box_inner, box_rows, dtype, swizzle;
  bool operator==(const TiledKey& o) const {
    return base == o.base && inner == o.inner && rows == o.rows && stride == o.stride &&
           box_inner == o.box_inner && box_rows == o.box_rows && dtype == o.dtype &&
           swizzle == o.swizzle;
  }
};

struct TiledSlot {
  TiledKey key;
  CUtensorMap map;
  bool valid = false;
};

constexpr int kMapCacheSlots = 64;
thread_local TiledSlot t_map_cache[kMapCacheSlots];

int map_cache_index(const TiledKey& k) {
  uint64_t h = k.base * 0x9E3779B97F4A7C15ull;
  h ^= (k.inner + 0x632BE59BD9B4E019ull) * 0xC2B2AE3D27D4EB4Full;
  h ^= (k.rows + (k.stride << 20)) * 0x165667B19E3779F9ull;
  h ^= (static_cast<uint64_t>(k.box_inner) << 32 | k.box_rows) * 0x27D4EB2F165667C5ull;
  h ^= (static_cast<uint64_t>(k.dtype) << 8 | k.swizzle) * 0x94D049BB133111EBull;
  h ^= h >> 29;
  return static_cast<int>(h % kMapCacheSlots);
}

}  // namespace

int encode_tiled_2d_swizzle(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                            uint64_t inner, uint64_t rows, uint64_t row_stride_bytes,
                            uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  const TiledKey key{reinterpret_cast<uint64_t>(base), inner, rows, row_stride_bytes,
                     box_inner, box_rows, static_cast<uint32_t>(dtype),
                     static_cast<uint32_t>(swizzle)};
  TiledSlot& slot = t_map_cache[map_cache_index(key)];
  if (slot.valid && slot.key == key) {
    *map = slot.map;
    return IGC_OK;
  }
  load_encoders();
  if (!g_encode_tiled) return IGC_ERR_CUDA;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode_tiled(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return IGC_ERR_CUDA;
  slot.key = key;
  slot.map = *map;
  slot.valid = true;
  return IGC_OK;
}

int encode_im2col_nhwc(CUtensorMap* map, const void* base, int N, int H, int W, int C,
                       int lower_h, int lower_w, int upper_h, int upper_w, uint32_t channels,
                       uint32_t pixels, int stride_h, int stride_w) {
  load_encoders();
  if (!g_encode_im2col) return IGC_ERR_CUDA;
  const uint64_t es = 2;  // fp16
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(W),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(N)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(C) * es, static_cast<cuuint64_t>(W) * C * es,
                           static_cast<cuuint64_t>(H) * W * C * es};
  // bounding-box corners follow the tensor's dimension order: W (inner) first, then H
  int lower[2] = {lower_w, lower_h};
  int upper[2] = {upper_w, upper_h};
  cuuint32_t estr[4] = {1, static_cast<cuuint32_t>(stride_w), static_cast<cuuint32_t>(stride_h),
                        1};
  CUresult r = g_encode_im2col(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(base),
                               dims, strides, lower, upper, channels, pixels, estr,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? IGC_OK : IGC_ERR_CUDA;
}

}  // namespace igc

extern "C" {

const char* igc_status_string(int status) {
  switch (status) {
    case IGC_OK: return "ok";
    case IGC_ERR_INVALID_ARG: return "invalid argument";
    case IGC_ERR_MISALIGNED: return "operand pointer or row stride not 16-byte aligned";
    case IGC_ERR_UNSUPPORTED: return "unsupported shape, parameter or device";
    case IGC_ERR_CUDA: return "CUDA runtime or driver call failed";
    case IGC_ERR_DEVICE_TIMEOUT: return "a kernel pipeline wait timed out";
    case IGC_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int igc_check_device_status(igc_stream_t stream) {
  igc::DeviceInfo d;
  int rc = igc::current_device(&d);
  if (rc != IGC_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return IGC_ERR_CUDA;
  unsigned long long v = 0;
  if (cudaMemcpyFromSymbol(&v, igc::g_status_word, sizeof(v)) != cudaSuccess) return IGC_ERR_CUDA;
  igc::g_last_status.store(v);
  if (v != 0) {
    const unsigned long long zero = 0;
    if (cudaMemcpyToSymbol(igc::g_status_word, &zero, sizeof(zero)) != cudaSuccess)
      return IGC_ERR_CUDA;
    return IGC_ERR_DEVICE_TIMEOUT;
  }
  return IGC_OK;
}

uint64_t igc_last_device_status(void) { return igc::g_last_status.load(); }

int igc_set_tile_width(int bn) {
  if (bn != 0 && bn != 128 && bn != 224 && bn != 256) return -1;
  const int old = igc::t_tile_width;
  igc::t_tile_width = bn;
  return old;
}

int igc_set_stage_depth(int k) {
  if (k != 0 && k != 64 && k != 128) return -1;
  const int old = igc::t_stage_depth;
  igc::t_stage_depth = k;
  return old;
}

int igc_set_int8_path(int path) {
  if (path != IGC_INT8_PATH_TCGEN05 && path != IGC_INT8_PATH_MMA_SYNC &&
      path != IGC_INT8_PATH_FUSED && path != IGC_INT8_PATH_CONVERT)
    return -1;
  const int old = igc::t_int8_path;
  igc::t_int8_path = path;
  return old;
}

uint64_t igc_set_wait_limit_ns(uint64_t limit_ns) {
  if (limit_ns < 1000) limit_ns = 1000;
  return igc::g_wait_limit.exchange(limit_ns);
}

int igc_debug_wait_timeout_probe(igc_stream_t stream) {
  igc::DeviceInfo d;
  int rc = igc::current_device(&d);
  if (rc != IGC_OK) return rc;
  igc::wait_timeout_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      igc::wait_limit_ns(), igc::status_word());
  return cudaGetLastError() == cudaSuccess ? IGC_OK : IGC_ERR_CUDA;
}

const char* igc_version(void) { return "0.1.0"; }

}  // extern "C"
