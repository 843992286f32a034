// Shared launch code for the tcgen05 GEMM kernel template: cluster launch of
// CTA pairs, grid sized to the pairs that fit at once, tile width chosen per
// problem to balance the last wave.
#pragma once

#include <mutex>

#include "gemm_tc.cuh"
#include "igc_host.h"

namespace igc {

inline bool vec_store_ok(const void* p, long long ld, size_t esize) {
  return p == nullptr || (aligned16(p) && (static_cast<unsigned long long>(ld) * esize) % 16 == 0);
}

template <Mode kMode, int BN, int ATOMS>
struct KernelSlot {
  std::once_flag once[64];
  int rc[64];
  int max_clusters[64];
};

template <Mode kMode, int BN, int ATOMS>
KernelSlot<kMode, BN, ATOMS>& kernel_slot() {
  static KernelSlot<kMode, BN, ATOMS> s;
  return s;
}

// Sets the kernel's shared-memory attribute and finds how many CTA pairs fit
// on the device at once (cached per device).
template <Mode kMode, int BN, int ATOMS = kAtoms>
int kernel_setup(const DeviceInfo& dev, int* max_clusters) {
  using Cfg = TileCfg<BN, ATOMS>;
  auto& s = kernel_slot<kMode, BN, ATOMS>();
  const int d = dev.device;
  std::call_once(s.once[d], [&] {
    s.rc[d] = IGC_ERR_CUDA;
    s.max_clusters[d] = 0;
    if (dev.smem_optin < Cfg::kSmemBytes) {
      s.rc[d] = IGC_ERR_UNSUPPORTED;
      return;
    }
    auto kern = igc_tc_gemm_kernel<kMode, BN, ATOMS>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Cfg::kSmemBytes)) != cudaSuccess)
      return;
    // the kernel's register split assumes at least kMinLaunchRegs per thread at launch
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return;
    if (fa.numRegs < kMinLaunchRegs) {
      s.rc[d] = IGC_ERR_UNSUPPORTED;
      return;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (dev.sm_count / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      n = dev.sm_count / 2;  // one CTA per SM, pairs
    }
    s.max_clusters[d] = n;
    s.rc[d] = n > 0 ? IGC_OK : IGC_ERR_UNSUPPORTED;
  });
  *max_clusters = s.max_clusters[d];
  return s.rc[d];
}

// Tensor maps of the outputs written by bulk tensor stores from the epilogue's
// staging buffers; bit i of mask enables map i (the others are never read).
struct OutMaps {
  CUtensorMap map[3] = {};
  int mask = 0;
};

// Enables output slot `slot` (an M x N row-major matrix, row stride ld elements
// of esize bytes) for bulk tensor stores when its base and row stride are
// 16-byte aligned; boxes are 32 rows x 128 bytes, 128-byte swizzled.  Otherwise
// the slot stays on direct stores.
inline void add_out_map(OutMaps& o, int slot, CUtensorMapDataType dtype, const void* ptr,
                        long long ld, long long M, long long N, size_t esize) {
  if (ptr == nullptr || !vec_store_ok(ptr, ld, esize)) return;
  if (encode_tiled_2d(&o.map[slot], dtype, ptr, static_cast<uint64_t>(N),
                      static_cast<uint64_t>(M), static_cast<uint64_t>(ld) * esize,
                      static_cast<uint32_t>(128 / esize), 32) == IGC_OK)
    o.mask |= 1 << slot;
}

// First unit index of the column-half tail: when the last round of the schedule
// would be at most half full, its tiles run as column halves (the round holds
// twice the units at half the length); otherwise there is no tail.
inline int tail_start_of(int num_tiles, int clusters) {
  const int rem = num_tiles % clusters;
  return (rem > 0 && 2 * rem <= clusters) ? num_tiles - rem : num_tiles;
}

template <Mode kMode, int BN, int ATOMS = kAtoms>
int launch_tc_gemm(const DeviceInfo& dev, const CUtensorMap& tmA, const CUtensorMap& tmB,
                   const CUtensorMap& tmBh, const OutMaps& om, KParams p, cudaStream_t stream) {
  int max_clusters = 0;
  int rc = kernel_setup<kMode, BN, ATOMS>(dev, &max_clusters);
  if (rc != IGC_OK) return rc;
  p.tiles_m = static_cast<int>((static_cast<long long>(p.M) + BM - 1) / BM);
  p.tiles_n = static_cast<int>((static_cast<long long>(p.N) + BN - 1) / BN);
  const long long tiles = static_cast<long long>(p.tiles_m) * p.tiles_n;
  if (tiles > 0x7fff0000LL) return IGC_ERR_UNSUPPORTED;  // units (tiles + tail halves) fit an int
  p.num_tiles = static_cast<int>(tiles);
  p.group_m = p.tiles_m < 8 ? p.tiles_m : 8;  // m-tiles walked together (measured best of 2-16)
  p.tail_start = tail_start_of(p.num_tiles, max_clusters);
  p.num_units = p.num_tiles + (p.num_tiles - p.tail_start);
  p.wait_limit_ns = wait_limit_ns();
  p.status = status_word();
  p.tma_out = om.mask;
  const int clusters = p.num_units < max_clusters ? p.num_units : max_clusters;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = TileCfg<BN, ATOMS>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, igc_tc_gemm_kernel<kMode, BN, ATOMS>, tmA, tmB, tmBh, om.map[0],
                         om.map[1], om.map[2], p) != cudaSuccess) {
    (void)cudaGetLastError();
    return IGC_ERR_CUDA;
  }
  return IGC_OK;
}

// Tile width for an M x N output: the candidate with the smallest estimated
// time, (rounds of the schedule over the CTA pairs, a last round of column
// halves counting one half) x (tile width / relative efficiency of that width);
// ties go to the wider tile.
inline int pick_bn(long long M, long long N, int clusters, const int* cands, const double* eff,
                   int n_cands) {
  const long long tm = (M + BM - 1) / BM;
  int best = cands[0];
  double best_cost = 1e300;
  for (int i = 0; i < n_cands; ++i) {
    const long long tiles = tm * ((N + cands[i] - 1) / cands[i]);
    const long long rem = tiles % clusters;
    const double rounds = static_cast<double>(tiles / clusters) +
                          (rem == 0 ? 0.0 : (2 * rem <= clusters ? 0.5 : 1.0));
    const double cost = rounds * cands[i] / eff[i];
    if (cost < best_cost * 0.999) {
      best_cost = cost;
      best = cands[i];
    }
  }
  return best;
}

// Tile widths each operation is built for, with their relative mainloop
// efficiency (wider tiles move fewer operand bytes per flop).  224 lets skinny
// problems fill the CTA pairs (e.g. 8192 columns = 37 tiles of 224 instead of
// 32 of 256); the integer modes drain in 64-column steps and use 256 and 128.
constexpr int kBnCands[] = {256, 224, 128};
// measured on fp16 M x 8192 x 8192 with many rounds: BN 224 runs 0.987x and
// BN 128 0.87-0.92x the rate of BN 256
constexpr double kBnEff[] = {1.0, 0.97, 0.87};
constexpr int kBnCandsInt[] = {256, 128};
constexpr double kBnEffInt[] = {1.0, 0.87};
// shortest k for which a floating-point GEMM of at most two rounds takes 64-deep stages
constexpr int kDeepMinK = 2048;
// GEMMs whose operands take at most this many bytes (half of the 129 MB L2) prefetch
// the panels of each CTA pair's first two work units, larger ones of the first only
constexpr double kPrefetchTwoUnitsBytes = 64.0 * 1024 * 1024;

// The automatic stage depth of a floating-point GEMM: 64-deep stages when its
// schedule is at most two rounds, but at least a quarter of the CTA pairs, over a
// long k: each unit then streams its operands mostly from DRAM (measured on GB300:
// +4 to +8 % at 512-1024 x 8192 x 8192, 2048 x 2048 x 8192 and 1024 x 4096 x
// 16384; -2 to -4 % at 2048 x 8192 x 8192 and 4096^3; -12 % at 512 x 512 x 2048,
// four tiles).
inline bool auto_deep_stages(long long M, long long N, long long K, int bn, int clusters) {
  const long long tiles = ((M + BM - 1) / BM) * ((N + bn - 1) / bn);
  return tiles <= 2LL * clusters && 4 * tiles >= clusters && K >= kDeepMinK;
}

// Leading work units per CTA pair whose panels the prefetch warps bring into L2.
inline int prefetch_units_of(double operand_bytes) {
  return operand_bytes <= kPrefetchTwoUnitsBytes ? 2 : 1;
}

// Tile width after an igc_set_tile_width override (integer modes have no 224).
inline int apply_width_override(int bn, bool int_mode) {
  const int forced = tile_width_override();
  if (forced == 256 || forced == 128 || (forced == 224 && !int_mode)) return forced;
  return bn;
}

// Picks the tile width for this problem, encodes B's tensor maps with boxes of
// BN/2 rows (each CTA of the pair loads half of the B tile) and BN/4 rows (half
// of a column-half unit's B) and launches.
template <Mode kMode>
int launch_auto_bn(const DeviceInfo& dev, const CUtensorMap& tmA, const void* b_base,
                   uint64_t b_inner, uint64_t b_rows, uint64_t b_row_bytes, const OutMaps& om,
                   KParams p, cudaStream_t stream) {
  constexpr CUtensorMapDataType kBType = kMode == Mode::GemmBF16
                                             ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  int clusters = 0;
  int rc = kernel_setup<kMode, kBnCands[0]>(dev, &clusters);
  if (rc != IGC_OK) return rc;
  int bn = mode_is_int(kMode) ? pick_bn(p.M, p.N, clusters, kBnCandsInt, kBnEffInt, 2)
                              : pick_bn(p.M, p.N, clusters, kBnCands, kBnEff, 3);
  bn = apply_width_override(bn, mode_is_int(kMode));
  bool deep = false;
  if constexpr (!mode_is_int(kMode)) {
    if constexpr (!mode_is_conv(kMode)) deep = auto_deep_stages(p.M, p.N, p.K, bn, clusters);
    const int fd = stage_depth_override();
    if (fd == 64) deep = true;
    if (fd == 128) deep = false;
    if (deep) {
      if constexpr (mode_is_conv(kMode)) {  // channel blocks of BK per filter tap
        const int taps = p.num_kb / p.conv_cblocks;
        p.conv_cblocks = (p.conv_C + BK - 1) / BK;
        p.num_kb = taps * p.conv_cblocks;
      } else {
        p.num_kb = (p.K + BK - 1) / BK;
      }
      p.chunk_kb = p.num_kb;
    }
  }
  if constexpr (!mode_is_conv(kMode)) {
    // L2 prefetch of the first rounds' panels (the entry set pf_a / pf_lda)
    if (p.pf_a != nullptr && p.K <= (1 << 29)) {
      p.pf_b = static_cast<const char*>(b_base);
      p.pf_ldb = static_cast<long long>(b_row_bytes);
      p.pf_kbytes = p.K * 2;
      p.pf_units = prefetch_units_of(static_cast<double>(p.M) * static_cast<double>(p.pf_lda) +
                                     static_cast<double>(p.N) * static_cast<double>(p.pf_ldb));
    }
  }
  CUtensorMap tmB, tmBh;  // boxes of BN/2 rows (whole tiles) and BN/4 rows (column halves)
  rc = encode_tiled_2d(&tmB, kBType, b_base, b_inner, b_rows,
                       b_row_bytes, BK, static_cast<uint32_t>(bn / 2));
  if (rc != IGC_OK) return rc;
  rc = encode_tiled_2d(&tmBh, kBType, b_base, b_inner, b_rows,
                       b_row_bytes, BK, static_cast<uint32_t>(bn / 4));
  if (rc != IGC_OK) return rc;
  if constexpr (!mode_is_int(kMode)) {
    if (deep) {
      switch (bn) {
        case 256: return launch_tc_gemm<kMode, 256, 1>(dev, tmA, tmB, tmBh, om, p, stream);
        case 224: return launch_tc_gemm<kMode, 224, 1>(dev, tmA, tmB, tmBh, om, p, stream);
        case 128: return launch_tc_gemm<kMode, 128, 1>(dev, tmA, tmB, tmBh, om, p, stream);
        default: return IGC_ERR_UNSUPPORTED;
      }
    }
  }
  if constexpr (!mode_is_int(kMode))
    if (bn == 224) return launch_tc_gemm<kMode, 224>(dev, tmA, tmB, tmBh, om, p, stream);
  switch (bn) {
    case 256: return launch_tc_gemm<kMode, 256>(dev, tmA, tmB, tmBh, om, p, stream);
    case 128: return launch_tc_gemm<kMode, 128>(dev, tmA, tmB, tmBh, om, p, stream);
    default: return IGC_ERR_UNSUPPORTED;
  }
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

}  // namespace igc
