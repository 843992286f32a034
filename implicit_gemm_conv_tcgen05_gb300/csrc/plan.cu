// igc_plan_gemm: the schedule a GEMM call would run with (tile width, stage depth,
// tiles, column-half tail, grid, prefetched units), computed on the host by the
// same decision functions the launches use.
#include "launch.cuh"

using namespace igc;

extern "C" int igc_plan_gemm(int op, int64_t M, int64_t N, int64_t K, int clusters,
                             int32_t* out) {
  if (out == nullptr || M <= 0 || N <= 0 || K <= 0) return IGC_ERR_INVALID_ARG;
  if (op != IGC_PLAN_GEMM_F16 && op != IGC_PLAN_GEMM_BF16 && op != IGC_PLAN_GEMM_S8)
    return IGC_ERR_INVALID_ARG;
  if (M > 0x7fffffff || N > 0x7fffffff || K > 0x7fffffff) return IGC_ERR_UNSUPPORTED;
  if (clusters <= 0) {  // the current device's CTA pairs
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc != IGC_OK) return rc;
    rc = kernel_setup<Mode::GemmF16, kBnCands[0]>(dev, &clusters);
    if (rc != IGC_OK) return rc;
  }
  const bool int_mode = op == IGC_PLAN_GEMM_S8;
  int bn = int_mode ? pick_bn(M, N, clusters, kBnCandsInt, kBnEffInt, 2)
                    : pick_bn(M, N, clusters, kBnCands, kBnEff, 3);
  bn = apply_width_override(bn, int_mode);
  bool deep = false;
  if (!int_mode) {
    deep = auto_deep_stages(M, N, K, bn, clusters);
    const int fd = stage_depth_override();
    if (fd == 64) deep = true;
    if (fd == 128) deep = false;
  }
  const long long tiles_m = (M + BM - 1) / BM;
  const long long tiles_n = (N + bn - 1) / bn;
  const long long tiles = tiles_m * tiles_n;
  if (tiles > 0x7fff0000LL) return IGC_ERR_UNSUPPORTED;
  const int tail_start = tail_start_of(static_cast<int>(tiles), clusters);
  const int num_units = static_cast<int>(tiles) + (static_cast<int>(tiles) - tail_start);
  // fp16 operand rows: the int8 path's pre-pass widens K to a multiple of 8
  const double row_bytes = 2.0 * static_cast<double>(int_mode ? (K + 7) / 8 * 8 : K);
  out[0] = bn;
  out[1] = deep ? BK : KS;
  out[2] = static_cast<int32_t>(tiles_m);
  out[3] = static_cast<int32_t>(tiles_n);
  out[4] = tail_start;
  out[5] = num_units;
  out[6] = 2 * (num_units < clusters ? num_units : clusters);
  out[7] = K <= (1 << 29) ? prefetch_units_of((static_cast<double>(M) + static_cast<double>(N)) *
                                              row_bytes)
                          : 0;
  return IGC_OK;
}
