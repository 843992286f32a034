// gemm_s8_zp: INT8 GEMM with input zero points and requantisation (page
// "TVM在CUDA GPU上跑GEMM的全套张量化实现", §2.3: C = (A_q - zp_A)(B_q - zp_B)
// accumulated in int32, dequantise / requantise fused into the GEMM).
//
// sm_103a has no integer tcgen05 MMA kind, so the contraction runs exactly on
// the fp16 tensor pipe:
//  1. pre-pass (HBM-bound, one read of A_q and B_q): A' = A_q - oA and
//     B' = B_q - oB with oX = 128 for uint8, 0 for int8, so every value lies in
//     [-128, 127] and is exact in fp16; written as fp16 into the workspace
//     together with the sums rA'[i] = sum_k A'[i,k] and cB'[j] = sum_k B'[j,k].
//  2. tcgen05 kind::f16 GEMM over A', B' in chunks of 1024 k: each chunk's
//     partial sums are integers of magnitude <= 1024 * 128 * 128 = 2^24, so the
//     fp32 accumulator holds them exactly; the epilogue drains every chunk
//     (exact float-to-int conversion) into an int32 running sum
//     S'[i,j] = sum_k A'[i,k] B'[j,k].
//  3. fused epilogue, in int32 two's complement (mod 2^32):
//        C32 = S' - zB'_j rA'_i - zA'_i cB'_j + K zA'_i zB'_j,
//     with zA'_i = zA_i - oA and zB'_j = zB_j - oB -- the zero-point expansion of
//     sum_k (A'[i,k] - zA'_i)(B'[j,k] - zB'_j) = sum_k (A_q - zA_i)(B_q - zB_j),
//     then C8 = clamp(rne(fp32(C32) * scale_j), -128, 127).
#include <atomic>
#include <mutex>

#include "gemm_i8.cuh"
#include "int8_prepass.cuh"
#include "launch.cuh"

using namespace igc;
using namespace igc::prepass;

namespace {

constexpr size_t kWsAlign = 256;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline long long k_padded(long long K) { return (K + 7) / 8 * 8; }  // 16-byte fp16 rows

// The fp16 operands and their row sums (written by the pre-pass, or by the
// converting kernel, which accumulates the sums chunk by chunk), then the
// converting kernel's flags (one per 128-row block and 1024-k chunk, one per
// block) and job counter.  The converting kernel's sums, flags and counter are
// zeroed before each of its launches (one memset from ra_off to the end).
struct WsLayout {
  size_t a_off, b_off, ra_off, cb_off, flags_off, flags_bytes, total;
};

WsLayout ws_layout(long long M, long long N, long long K) {
  const long long Kp = k_padded(K);
  const long long chunks = (K + kCvChunk - 1) / kCvChunk;
  const long long blocks =
      (M + kCvBlockRows - 1) / kCvBlockRows + (N + kCvBlockRows - 1) / kCvBlockRows;
  WsLayout l;
  l.a_off = 0;
  l.b_off = l.a_off + align_up(static_cast<size_t>(M) * Kp * 2, kWsAlign);
  l.ra_off = l.b_off + align_up(static_cast<size_t>(N) * Kp * 2, kWsAlign);
  l.cb_off = l.ra_off + align_up(static_cast<size_t>(M) * 4, kWsAlign);
  l.flags_off = l.cb_off + align_up(static_cast<size_t>(N) * 4, kWsAlign);
  l.flags_bytes = static_cast<size_t>(blocks * chunks + blocks + 1) * 4;
  l.total = l.flags_off + align_up(l.flags_bytes, kWsAlign);
  return l;
}

}  // namespace

extern "C" size_t gemm_s8_zp_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0) return 0;
  return ws_layout(M, N, K).total;
}

namespace {

// Checks shared by the three entry points; returns IGC_OK or a status.
int check_common(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0) return IGC_ERR_INVALID_ARG;
  if (M > 0x7fffffff || N > 0x7fffffff || K > 0x7fffffff) return IGC_ERR_UNSUPPORTED;
  return IGC_OK;
}

int check_workspace(const void* workspace, size_t bytes, const WsLayout& l) {
  if (workspace == nullptr || bytes < l.total ||
      (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) != 0)
    return IGC_ERR_WORKSPACE;
  return IGC_OK;
}

}  // namespace

extern "C" int gemm_s8_zp_prepare(int64_t M, int64_t N, int64_t K, const void* A, int a_signed,
                                  int64_t lda, const void* Bt, int b_signed, int64_t ldb,
                                  void* workspace, size_t workspace_bytes, igc_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int rc = check_common(M, N, K);
  if (rc != IGC_OK) return rc;
  if (A == nullptr && Bt == nullptr) return IGC_ERR_INVALID_ARG;
  if (M == 0 || N == 0 || K == 0) return IGC_OK;  // nothing to prepare
  if ((A != nullptr && lda < K) || (Bt != nullptr && ldb < K)) return IGC_ERR_INVALID_ARG;
  if ((A != nullptr && (!aligned16(A) || lda % 16 != 0)) ||
      (Bt != nullptr && (!aligned16(Bt) || ldb % 16 != 0)))
    return IGC_ERR_MISALIGNED;
  const WsLayout l = ws_layout(M, N, K);
  rc = check_workspace(workspace, workspace_bytes, l);
  if (rc != IGC_OK) return rc;
  DeviceInfo dev;
  rc = current_device(&dev);
  if (rc != IGC_OK) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const long long Kp = k_padded(K);
  PrepassOperand ops[2];
  int n_ops = 0;
  if (A != nullptr)
    ops[n_ops++] = prepass_operand(A, lda, M, K, Kp, a_signed ? 1 : 0,
                                   reinterpret_cast<__half*>(ws + l.a_off),
                                   reinterpret_cast<int32_t*>(ws + l.ra_off));
  if (Bt != nullptr)
    ops[n_ops++] = prepass_operand(Bt, ldb, N, K, Kp, b_signed ? 1 : 0,
                                   reinterpret_cast<__half*>(ws + l.b_off),
                                   reinterpret_cast<int32_t*>(ws + l.cb_off));
  return launch_prepass(ops, n_ops, K, Kp, stream);
}

namespace {

struct DequantOut {
  float* y = nullptr;
  long long ldy = 0;
  const float* dq_row = nullptr;
  const float* dq_col = nullptr;
  const float* bias = nullptr;
};

// The GEMM kernel over the workspace's fp16 operands.  With A_raw set (the
// converting path: K a multiple of 16, both operands 16-byte aligned with row
// strides lda, ldb that are multiples of 16) the kernel converts A_raw / Bt_raw
// itself; otherwise the pre-pass has written the operands and their sums.
int run_int_gemm(int64_t M, int64_t N, int64_t K, int a_signed, int b_signed, int32_t zA,
                 const int32_t* zA_row, int32_t zB, const int32_t* zB_col, int32_t* C32,
                 int64_t ldc32, int8_t* C8, int64_t ldc8, float scale, const float* scale_col,
                 const DequantOut& dq, const void* workspace, size_t workspace_bytes,
                 cudaStream_t stream, const void* A_raw = nullptr, int64_t lda = 0,
                 const void* Bt_raw = nullptr, int64_t ldb = 0) {
  int rc = check_common(M, N, K);
  if (rc != IGC_OK) return rc;
  if (M == 0 || N == 0) return IGC_OK;  // empty output: nothing is read or written
  if (C32 == nullptr && C8 == nullptr && dq.y == nullptr) return IGC_ERR_INVALID_ARG;
  if (C32 != nullptr && ldc32 < N) return IGC_ERR_INVALID_ARG;
  if (C8 != nullptr && ldc8 < N) return IGC_ERR_INVALID_ARG;
  if (dq.y != nullptr && dq.ldy < N) return IGC_ERR_INVALID_ARG;
  DeviceInfo dev;
  rc = current_device(&dev);
  if (rc != IGC_OK) return rc;
  if (K == 0) {
    if (dq.y != nullptr) return IGC_ERR_UNSUPPORTED;  // a dequantised output needs K >= 1
    // empty sum: C32 = 0 and C8 = requant(0) = 0; nothing is read
    rc = zero_rows(C32, ldc32, M, N, 4, stream);
    if (rc == IGC_OK) rc = zero_rows(C8, ldc8, M, N, 1, stream);
    return rc;
  }
  const WsLayout l = ws_layout(M, N, K);
  rc = check_workspace(workspace, workspace_bytes, l);
  if (rc != IGC_OK) return rc;

  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  const long long Kp = k_padded(K);
  CUtensorMap tmA;
  rc = encode_tiled_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, ws + l.a_off, Kp, M, Kp * 2, BK,
                       BM_CTA);
  if (rc != IGC_OK) return rc;

  KParams p{};
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.num_kb = static_cast<int>((Kp + KS - 1) / KS);
  p.chunk_kb = kIntChunkKb;
  if (A_raw == nullptr) {
    p.pf_a = reinterpret_cast<const char*>(ws + l.a_off);
    p.pf_lda = Kp * 2;
    p.rsumA = reinterpret_cast<const int32_t*>(ws + l.ra_off);
    p.csumB = reinterpret_cast<const int32_t*>(ws + l.cb_off);
  } else {
    uint8_t* wsm = const_cast<uint8_t*>(ws);
    if (cudaMemsetAsync(wsm + l.ra_off, 0, l.flags_off + l.flags_bytes - l.ra_off, stream) !=
        cudaSuccess) {
      (void)cudaGetLastError();
      return IGC_ERR_CUDA;
    }
    const long long chunks = (K + kCvChunk - 1) / kCvChunk;
    p.cv_a = static_cast<const uint8_t*>(A_raw);
    p.cv_b = static_cast<const uint8_t*>(Bt_raw);
    p.cv_lda = lda;
    p.cv_ldb = ldb;
    p.cv_flip_a = a_signed ? 0x80808080u : 0u;
    p.cv_flip_b = b_signed ? 0x80808080u : 0u;
    p.cv_da = reinterpret_cast<__half*>(wsm + l.a_off);
    p.cv_db = reinterpret_cast<__half*>(wsm + l.b_off);
    p.cv_sa = reinterpret_cast<int32_t*>(wsm + l.ra_off);
    p.cv_sb = reinterpret_cast<int32_t*>(wsm + l.cb_off);
    p.cv_flags = reinterpret_cast<int*>(wsm + l.flags_off);
    p.cv_blocks_a = static_cast<int>((M + kCvBlockRows - 1) / kCvBlockRows);
    p.cv_blocks_b = static_cast<int>((N + kCvBlockRows - 1) / kCvBlockRows);
    p.cv_chunks = static_cast<int>(chunks);
    const long long blocks = p.cv_blocks_a + p.cv_blocks_b;
    p.cv_done = p.cv_flags + blocks * chunks;
    p.cv_queue = p.cv_done + blocks;
    p.cv_Kp = static_cast<int>(Kp);
  }
  p.c32 = C32;
  p.ldc32 = ldc32;
  p.c8 = C8;
  p.ldc8 = ldc8;
  p.zA = zA;
  p.zA_row = zA_row;
  p.zB = zB;
  p.zB_col = zB_col;
  p.oA = a_signed ? 0 : 128;
  p.oB = b_signed ? 0 : 128;
  p.scale = scale;
  p.scale_col = scale_col;
  p.yf = dq.y;
  p.ldyf = dq.ldy;
  p.dq_row = dq.dq_row;
  p.dq_col = dq.dq_col;
  p.bias = dq.bias;
  p.vec_ok = vec_store_ok(C32, ldc32, 4) && vec_store_ok(C8, ldc8, 1) &&
             vec_store_ok(dq.y, dq.ldy, 4);
  OutMaps om;
  add_out_map(om, 0, CU_TENSOR_MAP_DATA_TYPE_INT32, C32, ldc32, M, N, 4);
  add_out_map(om, 1, CU_TENSOR_MAP_DATA_TYPE_UINT8, C8, ldc8, M, N, 1);
  add_out_map(om, 2, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dq.y, dq.ldy, M, N, 4);
  if (A_raw != nullptr)
    return launch_auto_bn<Mode::GemmIntCv>(dev, tmA, ws + l.b_off, Kp, N, Kp * 2, om, p, stream);
  return launch_auto_bn<Mode::GemmInt>(dev, tmA, ws + l.b_off, Kp, N, Kp * 2, om, p, stream);
}

// ---------------------------------------------------------------------------
// The fused path: int8 operands converted inside the GEMM kernel (gemm_i8.cuh)
// ---------------------------------------------------------------------------
template <int BN, bool kDequant>
struct I8Slot {
  std::once_flag once[64];
  int rc[64];
  int max_clusters[64];
};

template <int BN, bool kDequant>
I8Slot<BN, kDequant>& i8_slot() {
  static I8Slot<BN, kDequant> s;
  return s;
}

// Shared-memory attribute and the CTA pairs that fit at once (cached per device).
template <int BN, bool kDequant>
int i8_setup(const DeviceInfo& dev, int* max_clusters) {
  using Cfg = I8Cfg<BN>;
  auto& s = i8_slot<BN, kDequant>();
  const int d = dev.device;
  std::call_once(s.once[d], [&] {
    s.rc[d] = IGC_ERR_CUDA;
    s.max_clusters[d] = 0;
    if (dev.smem_optin < Cfg::kSmemBytes) {
      s.rc[d] = IGC_ERR_UNSUPPORTED;
      return;
    }
    auto kern = igc_i8_gemm_kernel<BN, kDequant>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Cfg::kSmemBytes)) != cudaSuccess)
      return;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return;
    if (fa.numRegs < kI8LaunchRegs) {  // the register split assumes 128 per thread at launch
      s.rc[d] = IGC_ERR_UNSUPPORTED;
      return;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (dev.sm_count / 2), 1, 1);
    cfg.blockDim = dim3(kI8Threads, 1, 1);
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
      n = dev.sm_count / 2;
    }
    s.max_clusters[d] = n;
    s.rc[d] = IGC_OK;
  });
  *max_clusters = s.max_clusters[d];
  return s.rc[d];
}

template <int BN, bool kDequant>
int launch_i8(const DeviceInfo& dev, const CUtensorMap& tmA, const void* Bt, int64_t N,
              int64_t K, int64_t ldb, const OutMaps& om, KParams p, uint32_t flipA,
              uint32_t flipB, int clusters_avail, cudaStream_t stream) {
  CUtensorMap tmB, tmBh;
  int rc = encode_tiled_2d_swizzle(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, Bt,
                                   static_cast<uint64_t>(K), static_cast<uint64_t>(N),
                                   static_cast<uint64_t>(ldb), kI8KS, BN / 2,
                                   CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc != IGC_OK) return rc;
  rc = encode_tiled_2d_swizzle(&tmBh, CU_TENSOR_MAP_DATA_TYPE_UINT8, Bt,
                               static_cast<uint64_t>(K), static_cast<uint64_t>(N),
                               static_cast<uint64_t>(ldb), kI8KS, BN / 4,
                               CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc != IGC_OK) return rc;
  int max_clusters = 0;
  rc = i8_setup<BN, kDequant>(dev, &max_clusters);
  if (rc != IGC_OK) return rc;
  (void)clusters_avail;
  p.tiles_m = static_cast<int>((static_cast<long long>(p.M) + BM - 1) / BM);
  p.tiles_n = static_cast<int>((static_cast<long long>(p.N) + BN - 1) / BN);
  const long long tiles = static_cast<long long>(p.tiles_m) * p.tiles_n;
  if (tiles > 0x7fff0000LL) return IGC_ERR_UNSUPPORTED;
  p.num_tiles = static_cast<int>(tiles);
  p.group_m = p.tiles_m < 8 ? p.tiles_m : 8;
  p.tail_start = tail_start_of(p.num_tiles, max_clusters);
  p.num_units = p.num_tiles + (p.num_tiles - p.tail_start);
  p.wait_limit_ns = wait_limit_ns();
  p.status = status_word();
  p.tma_out = om.mask;
  const int clusters = p.num_units < max_clusters ? p.num_units : max_clusters;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(kI8Threads, 1, 1);
  cfg.dynamicSmemBytes = I8Cfg<BN>::kSmemBytes;
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
  if (cudaLaunchKernelEx(&cfg, igc_i8_gemm_kernel<BN, kDequant>, tmA, tmB, tmBh, om.map[0], om.map[1],
                         om.map[2], p, flipA, flipB) != cudaSuccess) {
    (void)cudaGetLastError();
    return IGC_ERR_CUDA;
  }
  return IGC_OK;
}

// gemm_s8_zp / gemm_s8_zp_dequant on the fused path: arguments as for
// run_int_gemm plus the raw operands (K >= 1, checked by the caller's rules).
int run_int_gemm_fused(int64_t M, int64_t N, int64_t K, const void* A, int a_signed, int64_t lda,
                       const void* Bt, int b_signed, int64_t ldb, int32_t zA,
                       const int32_t* zA_row, int32_t zB, const int32_t* zB_col, int32_t* C32,
                       int64_t ldc32, int8_t* C8, int64_t ldc8, float scale,
                       const float* scale_col, const DequantOut& dq, cudaStream_t stream) {
  if (A == nullptr || Bt == nullptr || lda < K || ldb < K) return IGC_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(Bt) || lda % 16 != 0 || ldb % 16 != 0)
    return IGC_ERR_MISALIGNED;
  DeviceInfo dev;
  int rc = current_device(&dev);
  if (rc != IGC_OK) return rc;
  CUtensorMap tmA;
  rc = encode_tiled_2d_swizzle(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, static_cast<uint64_t>(K),
                               static_cast<uint64_t>(M), static_cast<uint64_t>(lda), kI8KS,
                               BM_CTA, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc != IGC_OK) return rc;
  KParams p{};
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.num_kb = static_cast<int>((K + kI8KS - 1) / kI8KS);
  p.chunk_kb = kI8ChunkKb;
  p.c32 = C32;
  p.ldc32 = ldc32;
  p.c8 = C8;
  p.ldc8 = ldc8;
  p.zA = zA;
  p.zA_row = zA_row;
  p.zB = zB;
  p.zB_col = zB_col;
  p.oA = a_signed ? 0 : 128;
  p.oB = b_signed ? 0 : 128;
  p.scale = scale;
  p.scale_col = scale_col;
  p.yf = dq.y;
  p.ldyf = dq.ldy;
  p.dq_row = dq.dq_row;
  p.dq_col = dq.dq_col;
  p.bias = dq.bias;
  p.vec_ok = vec_store_ok(C32, ldc32, 4) && vec_store_ok(C8, ldc8, 1) &&
             vec_store_ok(dq.y, dq.ldy, 4);
  OutMaps om;
  add_out_map(om, 0, CU_TENSOR_MAP_DATA_TYPE_INT32, C32, ldc32, M, N, 4);
  add_out_map(om, 1, CU_TENSOR_MAP_DATA_TYPE_UINT8, C8, ldc8, M, N, 1);
  add_out_map(om, 2, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dq.y, dq.ldy, M, N, 4);
  // uint8 keeps its byte (u = value + 128 - 128 offset), int8 flips the top bit
  const uint32_t flipA = a_signed ? 0x80808080u : 0u;
  const uint32_t flipB = b_signed ? 0x80808080u : 0u;
  int clusters = 0;
  rc = i8_setup<256, false>(dev, &clusters);
  if (rc != IGC_OK) return rc;
  int bn = pick_bn(M, N, clusters, kBnCandsInt, kBnEffInt, 2);
  bn = apply_width_override(bn, true);
  const bool dq_out = dq.y != nullptr;
  if (bn == 128)
    return dq_out ? launch_i8<128, true>(dev, tmA, Bt, N, K, ldb, om, p, flipA, flipB, clusters,
                                         stream)
                  : launch_i8<128, false>(dev, tmA, Bt, N, K, ldb, om, p, flipA, flipB, clusters,
                                          stream);
  return dq_out ? launch_i8<256, true>(dev, tmA, Bt, N, K, ldb, om, p, flipA, flipB, clusters,
                                       stream)
                : launch_i8<256, false>(dev, tmA, Bt, N, K, ldb, om, p, flipA, flipB, clusters,
                                        stream);
}

// The converting path's conditions (IGC_INT8_PATH_CONVERT): 16-byte rows and
// strides, K a multiple of 16 (so the fp16 rows need no padding).
bool convert_ok(int64_t K, const void* A, int64_t lda, const void* Bt, int64_t ldb) {
  return K > 0 && K % 16 == 0 && A != nullptr && Bt != nullptr && lda >= K && ldb >= K &&
         aligned16(A) && aligned16(Bt) && lda % 16 == 0 && ldb % 16 == 0;
}

}  // namespace

extern "C" int gemm_s8_zp_run(int64_t M, int64_t N, int64_t K, int a_signed, int b_signed,
                              int32_t zA, const int32_t* zA_row, int32_t zB,
                              const int32_t* zB_col, int32_t* C32, int64_t ldc32, int8_t* C8,
                              int64_t ldc8, float scale, const float* scale_col,
                              const void* workspace, size_t workspace_bytes,
                              igc_stream_t stream) {
  return run_int_gemm(M, N, K, a_signed, b_signed, zA, zA_row, zB, zB_col, C32, ldc32, C8, ldc8,
                      scale, scale_col, DequantOut(), workspace, workspace_bytes,
                      reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int gemm_s8_zp_dequant(int64_t M, int64_t N, int64_t K, const void* A, int a_signed,
                                  int64_t lda, const void* Bt, int b_signed, int64_t ldb,
                                  int32_t zA, const int32_t* zA_row, int32_t zB,
                                  const int32_t* zB_col, const float* scale_row,
                                  const float* scale_col, const float* bias, float* Y,
                                  int64_t ldy, void* workspace, size_t workspace_bytes,
                                  igc_stream_t stream) {
  int rc = check_common(M, N, K);
  if (rc != IGC_OK) return rc;
  if (M == 0 || N == 0) return IGC_OK;  // empty output: nothing is read or written
  if (Y == nullptr || ldy < N) return IGC_ERR_INVALID_ARG;
  if (K == 0) return IGC_ERR_UNSUPPORTED;
  if (A == nullptr || Bt == nullptr) return IGC_ERR_INVALID_ARG;
  DequantOut dq;
  dq.y = Y;
  dq.ldy = ldy;
  dq.dq_row = scale_row;
  dq.dq_col = scale_col;
  dq.bias = bias;
  if (int8_path_override() == IGC_INT8_PATH_FUSED)
    return run_int_gemm_fused(M, N, K, A, a_signed, lda, Bt, b_signed, ldb, zA, zA_row, zB,
                              zB_col, nullptr, 0, nullptr, 0, 0.0f, nullptr, dq,
                              reinterpret_cast<cudaStream_t>(stream));
  if (int8_path_override() == IGC_INT8_PATH_CONVERT && convert_ok(K, A, lda, Bt, ldb))
    return run_int_gemm(M, N, K, a_signed, b_signed, zA, zA_row, zB, zB_col, nullptr, 0, nullptr,
                        0, 0.0f, nullptr, dq, workspace, workspace_bytes,
                        reinterpret_cast<cudaStream_t>(stream), A, lda, Bt, ldb);
  rc = gemm_s8_zp_prepare(M, N, K, A, a_signed, lda, Bt, b_signed, ldb, workspace,
                          workspace_bytes, stream);
  if (rc != IGC_OK) return rc;
  return run_int_gemm(M, N, K, a_signed, b_signed, zA, zA_row, zB, zB_col, nullptr, 0, nullptr,
                      0, 0.0f, nullptr, dq, workspace, workspace_bytes,
                      reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int gemm_s8_zp(int64_t M, int64_t N, int64_t K, const void* A, int a_signed,
                          int64_t lda, const void* Bt, int b_signed, int64_t ldb, int32_t zA,
                          const int32_t* zA_row, int32_t zB, const int32_t* zB_col, int32_t* C32,
                          int64_t ldc32, int8_t* C8, int64_t ldc8, float scale,
                          const float* scale_col, void* workspace, size_t workspace_bytes,
                          igc_stream_t stream) {
  int rc = check_common(M, N, K);
  if (rc != IGC_OK) return rc;
  if (M == 0 || N == 0) return IGC_OK;  // empty output: nothing is read or written
  if (C32 == nullptr && C8 == nullptr) return IGC_ERR_INVALID_ARG;
  if ((C32 != nullptr && ldc32 < N) || (C8 != nullptr && ldc8 < N)) return IGC_ERR_INVALID_ARG;
  if (K > 0 && int8_path_override() == IGC_INT8_PATH_MMA_SYNC) {
    if (A == nullptr || Bt == nullptr || lda < K || ldb < K) return IGC_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(Bt) || lda % 16 != 0 || ldb % 16 != 0)
      return IGC_ERR_MISALIGNED;
    const WsLayout l = ws_layout(M, N, K);
    rc = check_workspace(workspace, workspace_bytes, l);
    if (rc != IGC_OK) return rc;
    DeviceInfo dev;
    rc = current_device(&dev);
    if (rc != IGC_OK) return rc;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    return imma_gemm_s8_zp(static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), A,
                           a_signed, lda, Bt, b_signed, ldb, zA, zA_row, zB, zB_col, C32, ldc32,
                           C8, ldc8, scale, scale_col, reinterpret_cast<int32_t*>(ws + l.ra_off),
                           reinterpret_cast<int32_t*>(ws + l.cb_off),
                           reinterpret_cast<cudaStream_t>(stream));
  }
  if (K > 0 && int8_path_override() == IGC_INT8_PATH_FUSED)
    return run_int_gemm_fused(M, N, K, A, a_signed, lda, Bt, b_signed, ldb, zA, zA_row, zB,
                              zB_col, C32, ldc32, C8, ldc8, scale, scale_col, DequantOut(),
                              reinterpret_cast<cudaStream_t>(stream));
  if (int8_path_override() == IGC_INT8_PATH_CONVERT && convert_ok(K, A, lda, Bt, ldb))
    return run_int_gemm(M, N, K, a_signed, b_signed, zA, zA_row, zB, zB_col, C32, ldc32, C8,
                        ldc8, scale, scale_col, DequantOut(), workspace, workspace_bytes,
                        reinterpret_cast<cudaStream_t>(stream), A, lda, Bt, ldb);
  if (K > 0) {
    if (A == nullptr || Bt == nullptr) return IGC_ERR_INVALID_ARG;
    rc = gemm_s8_zp_prepare(M, N, K, A, a_signed, lda, Bt, b_signed, ldb, workspace,
                            workspace_bytes, stream);
    if (rc != IGC_OK) return rc;
  }
  return gemm_s8_zp_run(M, N, K, a_signed, b_signed, zA, zA_row, zB, zB_col, C32, ldc32, C8,
                        ldc8, scale, scale_col, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------------------
// gemm_s8_zp_noalloc: the same operation for callers that cannot allocate
// device memory.  Its scratch is a fixed array in the library's device image
// (every GPU that loads the library holds it until the process exits); the
// caller still passes inputs and outputs.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(IGC_NOALLOC_SCRATCH_BYTES);

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch per device, cached once a lookup succeeded
// (a failed lookup is not cached: the next call tries again).
std::atomic<void*> g_noalloc_ptr[64];
std::mutex g_noalloc_mutex;

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// the device current (cudaGetSymbolAddress) and cached.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IGC_ERR_CUDA;
  if (dev < 0 || dev >= 64) return IGC_ERR_UNSUPPORTED;
  void* p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return IGC_ERR_CUDA;
      }
      g_noalloc_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return IGC_OK;
}

}  // namespace

extern "C" int gemm_s8_zp_noalloc(int64_t M, int64_t N, int64_t K, const void* A, int a_signed,
                                  int64_t lda, const void* Bt, int b_signed, int64_t ldb,
                                  int32_t zA, const int32_t* zA_row, int32_t zB,
                                  const int32_t* zB_col, int32_t* C32, int64_t ldc32, int8_t* C8,
                                  int64_t ldc8, float scale, const float* scale_col,
                                  igc_stream_t stream) {
  // the argument checks of gemm_s8_zp come first, so that a bad argument is
  // reported as such whatever the problem's size
  int rc0 = check_common(M, N, K);
  if (rc0 != IGC_OK) return rc0;
  if (M == 0 || N == 0) return IGC_OK;  // empty output: nothing is read or written
  if (C32 == nullptr && C8 == nullptr) return IGC_ERR_INVALID_ARG;
  if ((C32 != nullptr && ldc32 < N) || (C8 != nullptr && ldc8 < N)) return IGC_ERR_INVALID_ARG;
  if (K == 0)  // an empty sum needs no scratch: C32 = 0, C8 = 0
    return gemm_s8_zp(M, N, K, A, a_signed, lda, Bt, b_signed, ldb, zA, zA_row, zB, zB_col, C32,
                      ldc32, C8, ldc8, scale, scale_col, nullptr, 0, stream);
  if (A == nullptr || Bt == nullptr || lda < K || ldb < K) return IGC_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(Bt) || lda % 16 != 0 || ldb % 16 != 0)
    return IGC_ERR_MISALIGNED;
  if (gemm_s8_zp_workspace_size(M, N, K) > kNoAllocScratchBytes) return IGC_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = noalloc_scratch(&scratch);
  if (rc != IGC_OK) return rc;
  return gemm_s8_zp(M, N, K, A, a_signed, lda, Bt, b_signed, ldb, zA, zA_row, zB, zB_col, C32,
                    ldc32, C8, ldc8, scale, scale_col, scratch, kNoAllocScratchBytes, stream);
}
