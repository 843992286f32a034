// conv2d_nhwc_f16_implicit: 2-D convolution as an implicit GEMM on tcgen05
// (page "如何使用 TensorCores 优化卷积", section "准备和算法": zero-padded input
// Apad, reduction over input channels and the R x S window, fp32 accumulation).
//
// GEMM view: M = N*P*Q output pixels, N_gemm = K filters, K_gemm = R*S*C.
// Row m of A (pixel (n, p, q)) at column (r, s, c) is
//   x[n, p*stride_h + r - pad_h, q*stride_w + s - pad_w, c]  (0 outside the image).
// A is never materialised: each 128-pixel x 64-channel tile is gathered by
// TMA in im2col mode (the tensor map's bounding box encodes the padding, the
// per-load offsets (s, r) select the filter tap; out-of-image pixels, the
// channels beyond C and the pixels past the last image are zero-filled).
// The KRSC weights already form the K-major N_gemm x K_gemm matrix B.
#include "launch.cuh"

using namespace igc;

extern "C" int conv2d_nhwc_f16_implicit(int N, int H, int W, int C, int K, int R, int S,
                                        int pad_h, int pad_w, int stride_h, int stride_w,
                                        const void* x, const void* w, void* y,
                                        float* y_f32_check, igc_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (N < 0 || H <= 0 || W <= 0 || C <= 0 || K <= 0 || R <= 0 || S <= 0) return IGC_ERR_INVALID_ARG;
  if (pad_h < 0 || pad_w < 0 || stride_h <= 0 || stride_w <= 0) return IGC_ERR_INVALID_ARG;
  if (H + 2 * pad_h < R || W + 2 * pad_w < S) return IGC_ERR_INVALID_ARG;
  if (N == 0) return IGC_OK;  // empty batch: nothing is read or written
  if (y == nullptr && y_f32_check == nullptr) return IGC_ERR_INVALID_ARG;
  if (x == nullptr || w == nullptr) return IGC_ERR_INVALID_ARG;

  const long long P = (H + 2LL * pad_h - R) / stride_h + 1;
  const long long Q = (W + 2LL * pad_w - S) / stride_w + 1;
  const long long M = static_cast<long long>(N) * P * Q;
  if (stride_h > 8 || stride_w > 8) return IGC_ERR_UNSUPPORTED;  // TMA traversal stride <= 8
  if (C % 8 != 0) return IGC_ERR_UNSUPPORTED;
  // im2col bounding-box corners of a rank-4 tensor map are limited to [-128, 127]
  const int lower_h = -pad_h, lower_w = -pad_w;
  const int upper_h = pad_h - (R - 1), upper_w = pad_w - (S - 1);
  if (lower_h < -128 || lower_w < -128 || upper_h < -128 || upper_w < -128 || upper_h > 127 ||
      upper_w > 127)
    return IGC_ERR_UNSUPPORTED;
  if (static_cast<long long>(N) * H * W * C >= 0x7fffffffLL || M * K >= 0x7fffffffLL ||
      static_cast<long long>(R) * S * C >= 0x7fffffffLL)
    return IGC_ERR_UNSUPPORTED;

  DeviceInfo dev;
  int rc = current_device(&dev);
  if (rc != IGC_OK) return rc;
  if (!aligned16(x) || !aligned16(w)) return IGC_ERR_MISALIGNED;

  const int Kg = R * S * C;
  CUtensorMap tmA;
  rc = encode_im2col_nhwc(&tmA, x, N, H, W, C, lower_h, lower_w, upper_h, upper_w, BK, BM_CTA,
                          stride_h, stride_w);
  if (rc != IGC_OK) return rc;

  KParams p{};
  p.M = static_cast<int>(M);
  p.N = K;
  p.K = Kg;
  p.conv_cblocks = (C + KS - 1) / KS;
  p.num_kb = R * S * p.conv_cblocks;
  p.chunk_kb = p.num_kb;
  p.conv_P = static_cast<int>(P);
  p.conv_Q = static_cast<int>(Q);
  p.conv_S = S;
  p.conv_C = C;
  p.pad_h = pad_h;
  p.pad_w = pad_w;
  p.stride_h = stride_h;
  p.stride_w = stride_w;
  p.out = y;
  p.ldo = K;
  p.out_type = kOutF16;
  p.out_f32 = y_f32_check;
  p.ldo32 = K;
  p.vec_ok = vec_store_ok(y, K, 2) && vec_store_ok(y_f32_check, K, 4);
  OutMaps om;
  add_out_map(om, 0, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, y, K, M, K, 2);
  add_out_map(om, 1, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, y_f32_check, K, M, K, 4);
  return launch_auto_bn<Mode::ConvF16>(dev, tmA, w, Kg, K, static_cast<uint64_t>(Kg) * 2, om, p,
                                       stream);
}
