// conv2d_nhwc_s8_zp: INT8 convolution as an implicit GEMM with input zero
// points and requantisation -- the pages pair the im2col lowering with the
// INT8 path (page "TVM在CUDA GPU上跑GEMM的全套张量化实现", §2.2 / §2.3: im2col turns
// the convolution into a regular GEMM; C = (A_q - zp_A)(B_q - zp_B)), with the
// padded input of page "如何使用 TensorCores 优化卷积", section "准备和算法".
//
// With asymmetric quantisation the real zero of the input is its zero point,
// so padding is zX, not 0: a padded tap contributes (zX - zX)(w - zW) = 0.
//
//  1. pad_shift_pixels: writes x' = x_q - oX (oX = 128 for uint8, 0 for int8)
//     as fp16 into a padded NHWC tensor (H + 2 pad_h) x (W + 2 pad_w) whose
//     border holds zX - oX, and the channel sum of every padded pixel.
//  2. the weights go through the int8 GEMM pre-pass (w' = w_q - oW as fp16,
//     with the sum of every output channel's R*S*C weights).
//  3. window_sums: for every output pixel, the sum of x' over its R x S window
//     (the row sums of the implicit im2col matrix).
//  4. the tcgen05 kernel: TMA im2col over the padded x' (no further padding),
//     exact fp32 chunks drained to int32, then the zero-point expansion
//        y32 = S' - zW'_k rX'_m - zX' cW'_k + (R S C) zX' zW'_k
//     (zX' = zX - oX, zW' = zW - oW) and the requantisation of gemm_s8_zp.
#include <mutex>

#include "int8_prepass.cuh"
#include "launch.cuh"

using namespace igc;
using namespace igc::prepass;

namespace igc {
namespace conv_s8 {

constexpr size_t kWsAlign = 256;
constexpr int kEpilogueWindowMax = 25;  // filter windows up to 5 x 5 are summed in the epilogue
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct ConvShape {
  long long N, H, W, C, K, R, S, ph, pw, sh, sw, Hp, Wp, P, Q, M, Kg, Kgp;
};

struct ConvWs {
  size_t xp_off, w_off, px_off, rx_off, cw_off, total;
};

ConvShape conv_shape(int N, int H, int W, int C, int K, int R, int S, int ph, int pw, int sh,
                     int sw) {
  ConvShape c;
  c.N = N; c.H = H; c.W = W; c.C = C; c.K = K; c.R = R; c.S = S;
  c.ph = ph; c.pw = pw; c.sh = sh; c.sw = sw;
  c.Hp = H + 2LL * ph;
  c.Wp = W + 2LL * pw;
  c.P = (c.Hp - R) / sh + 1;
  c.Q = (c.Wp - S) / sw + 1;
  c.M = c.N * c.P * c.Q;
  c.Kg = static_cast<long long>(R) * S * C;
  c.Kgp = (c.Kg + 7) / 8 * 8;
  return c;
}

ConvWs conv_ws_layout(const ConvShape& c) {
  ConvWs l;
  l.xp_off = 0;
  l.w_off = l.xp_off + align_up(static_cast<size_t>(c.N * c.Hp * c.Wp * c.C) * 2, kWsAlign);
  l.px_off = l.w_off + align_up(static_cast<size_t>(c.K * c.Kgp) * 2, kWsAlign);
  l.rx_off = l.px_off + align_up(static_cast<size_t>(c.N * c.Hp * c.Wp) * 4, kWsAlign);
  l.cw_off = l.rx_off + align_up(static_cast<size_t>(c.M) * 4, kWsAlign);
  l.total = l.cw_off + align_up(static_cast<size_t>(c.K) * 4, kWsAlign);
  return l;
}

// One warp per padded pixel (n, hp, wp): x' = x_q - oX inside the image, zX - oX
// in the border; px = sum over the pixel's C channels of x'.
static __global__ void __launch_bounds__(256) pad_shift_pixels_kernel(
    const uint8_t* __restrict__ x, int is_signed, int offset, int border, int N, int H, int W,
    int C, int ph, int pw, int Hp, int Wp, int vec, __half* __restrict__ xp,
    int32_t* __restrict__ px) {
  grid_dependency_wait();
  grid_dependents_launch();
  const long long pixel = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = static_cast<int>(threadIdx.x % 32);
  const long long npix = static_cast<long long>(N) * Hp * Wp;
  if (pixel >= npix) return;
  const int n = static_cast<int>(pixel / (static_cast<long long>(Hp) * Wp));
  const int rem = static_cast<int>(pixel - static_cast<long long>(n) * Hp * Wp);
  const int h = rem / Wp - ph;
  const int w = rem % Wp - pw;
  const bool inside = h >= 0 && h < H && w >= 0 && w < W;
  const uint8_t* src = x + ((static_cast<size_t>(n) * H + (inside ? h : 0)) * W + (inside ? w : 0)) * C;
  __half* dst = xp + static_cast<size_t>(pixel) * C;
  int32_t acc = 0;
  if (!inside) {
    const __half hb = __int2half_rn(border);
    for (int c = lane; c < C; c += 32) {
      dst[c] = hb;
      acc += border;
    }
  } else if (vec) {  // C % 16 == 0 and 16-byte aligned pixels
    for (int c = lane * 16; c < C; c += 32 * 16) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src + c));
      const uint32_t words[4] = {raw.x, raw.y, raw.z, raw.w};
      uint32_t out[8];
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        int v[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          v[b] = shifted_byte((words[wi] >> (8 * b)) & 0xFFu, is_signed, offset);
          acc += v[b];
        }
        __half2 h0 = __halves2half2(__int2half_rn(v[0]), __int2half_rn(v[1]));
        __half2 h1 = __halves2half2(__int2half_rn(v[2]), __int2half_rn(v[3]));
        out[2 * wi] = *reinterpret_cast<uint32_t*>(&h0);
        out[2 * wi + 1] = *reinterpret_cast<uint32_t*>(&h1);
      }
      reinterpret_cast<uint4*>(dst + c)[0] = make_uint4(out[0], out[1], out[2], out[3]);
      reinterpret_cast<uint4*>(dst + c)[1] = make_uint4(out[4], out[5], out[6], out[7]);
    }
  } else {
    for (int c = lane; c < C; c += 32) {
      const int v = shifted_byte(src[c], is_signed, offset);
      dst[c] = __int2half_rn(v);
      acc += v;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) px[pixel] = acc;
}

// One thread per 16 channels of a padded pixel, for C = 16 G with G a power of
// two <= 32, so the G threads of a pixel are an aligned group of lanes of one
// warp: x' = x_q - oX inside the image (exact fp16 by the pre-pass's byte
// widening), zX - oX in the border; lane 0 of the group writes the pixel's
// channel sum.  Threads past the end still take part in the shuffles.  The
// first w_blocks blocks widen the weights instead (one row of wop per warp), so
// that both operands' pre-passes are one launch.
static __global__ void __launch_bounds__(256) pad_shift_chunks_kernel(
    const uint8_t* __restrict__ x, uint32_t flip, int border, int N, int H, int W, int C, int ph,
    int pw, int Hp, int Wp, int log2g, __half* __restrict__ xp, int32_t* __restrict__ px,
    unsigned w_blocks, const PrepassOperand wop, int wK, int wKp) {
  grid_dependency_wait();
  grid_dependents_launch();
  if (blockIdx.x < w_blocks) {
    const int row = static_cast<int>(blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32);
    if (row < wop.rows) widen_row(wop, row, wK, wKp, static_cast<int>(threadIdx.x % 32));
    return;
  }
  const long long t = static_cast<long long>(blockIdx.x - w_blocks) * blockDim.x + threadIdx.x;
  const long long npix = static_cast<long long>(N) * Hp * Wp;
  const bool valid = t < (npix << log2g);
  const long long pixel = t >> log2g;
  const int g = static_cast<int>(t & ((1 << log2g) - 1));
  int32_t part = 0;
  if (valid) {
    const int n = static_cast<int>(pixel / (static_cast<long long>(Hp) * Wp));
    const int rem = static_cast<int>(pixel - static_cast<long long>(n) * Hp * Wp);
    const int h = rem / Wp - ph;
    const int w = rem % Wp - pw;
    uint4* dst = reinterpret_cast<uint4*>(xp + static_cast<size_t>(pixel) * C + g * 16);
    if (h >= 0 && h < H && w >= 0 && w < W) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(
          x + ((static_cast<size_t>(n) * H + h) * W + w) * C + g * 16));
      uint32_t out[8];
      uint32_t usum = 0;
      widen4(raw.x, flip, out[0], out[1], usum);
      widen4(raw.y, flip, out[2], out[3], usum);
      widen4(raw.z, flip, out[4], out[5], usum);
      widen4(raw.w, flip, out[6], out[7], usum);
      dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
      dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
      part = static_cast<int32_t>(usum - 128u * 16u);
    } else {
      const uint32_t hb = static_cast<uint32_t>(__half_as_ushort(__int2half_rn(border)));
      const uint32_t bb = hb | (hb << 16);
      dst[0] = make_uint4(bb, bb, bb, bb);
      dst[1] = make_uint4(bb, bb, bb, bb);
      part = 16 * border;
    }
  }
  for (int off = (1 << log2g) >> 1; off > 0; off >>= 1)
    part += __shfl_xor_sync(0xffffffffu, part, off);
  if (valid && g == 0) px[pixel] = part;
}

// One thread per output pixel m = (n, p, q): rX'[m] = sum over the R x S window
// (in padded coordinates, origin (p sh, q sw)) of the pixel sums.
static __global__ void __launch_bounds__(256) window_sums_kernel(const int32_t* __restrict__ px, int N,
                                                          int Hp, int Wp, int P, int Q, int R,
                                                          int S, int sh, int sw,
                                                          int32_t* __restrict__ rx) {
  grid_dependency_wait();
  grid_dependents_launch();
  const long long m = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long M = static_cast<long long>(N) * P * Q;
  if (m >= M) return;
  const int n = static_cast<int>(m / (static_cast<long long>(P) * Q));
  const int rem = static_cast<int>(m - static_cast<long long>(n) * P * Q);
  const int p = rem / Q;
  const int q = rem % Q;
  const int32_t* base = px + (static_cast<size_t>(n) * Hp + static_cast<size_t>(p) * sh) * Wp +
                        static_cast<size_t>(q) * sw;
  int32_t acc = 0;
  for (int r = 0; r < R; ++r)
    for (int s = 0; s < S; ++s) acc += __ldg(base + static_cast<size_t>(r) * Wp + s);
  rx[m] = acc;
}

int check_conv(int N, int H, int W, int C, int K, int R, int S, int ph, int pw, int sh, int sw) {
  if (N < 0 || H <= 0 || W <= 0 || C <= 0 || K <= 0 || R <= 0 || S <= 0) return IGC_ERR_INVALID_ARG;
  if (ph < 0 || pw < 0 || sh <= 0 || sw <= 0) return IGC_ERR_INVALID_ARG;
  if (H + 2 * ph < R || W + 2 * pw < S) return IGC_ERR_INVALID_ARG;
  if (sh > 8 || sw > 8 || R > 32 || S > 32 || C % 8 != 0) return IGC_ERR_UNSUPPORTED;
  const ConvShape c = conv_shape(N, H, W, C, K, R, S, ph, pw, sh, sw);
  if (c.N * c.Hp * c.Wp * c.C >= 0x7fffffffLL || c.M * c.K >= 0x7fffffffLL ||
      c.Kg >= (1LL << 24) || c.Hp > 65535 || c.Wp > 65535)
    return IGC_ERR_UNSUPPORTED;
  return IGC_OK;
}

}  // namespace conv_s8
}  // namespace igc

using namespace igc::conv_s8;

extern "C" size_t conv2d_nhwc_s8_zp_workspace_size(int N, int H, int W, int C, int K, int R,
                                                   int S, int pad_h, int pad_w, int stride_h,
                                                   int stride_w) {
  if (check_conv(N, H, W, C, K, R, S, pad_h, pad_w, stride_h, stride_w) != IGC_OK) return 0;
  return conv_ws_layout(conv_shape(N, H, W, C, K, R, S, pad_h, pad_w, stride_h, stride_w)).total;
}

extern "C" int conv2d_nhwc_s8_zp(int N, int H, int W, int C, int K, int R, int S, int pad_h,
                                 int pad_w, int stride_h, int stride_w, const void* x,
                                 int x_signed, int32_t zX, const void* w, int w_signed,
                                 int32_t zW, const int32_t* zW_k, int32_t* y32, int8_t* y8,
                                 float scale, const float* scale_k, void* workspace,
                                 size_t workspace_bytes, igc_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int rc = check_conv(N, H, W, C, K, R, S, pad_h, pad_w, stride_h, stride_w);
  if (rc != IGC_OK) return rc;
  if (N == 0) return IGC_OK;  // empty batch: nothing is read or written
  if (y32 == nullptr && y8 == nullptr) return IGC_ERR_INVALID_ARG;
  if (x == nullptr || w == nullptr) return IGC_ERR_INVALID_ARG;
  // the padding value must be a value of the input type (it enters the exact fp16 operand)
  if (x_signed ? (zX < -128 || zX > 127) : (zX < 0 || zX > 255)) return IGC_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w)) return IGC_ERR_MISALIGNED;
  const ConvShape c = conv_shape(N, H, W, C, K, R, S, pad_h, pad_w, stride_h, stride_w);
  const ConvWs l = conv_ws_layout(c);
  if (workspace == nullptr || workspace_bytes < l.total ||
      (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) != 0)
    return IGC_ERR_WORKSPACE;
  DeviceInfo dev;
  rc = current_device(&dev);
  if (rc != IGC_OK) return rc;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __half* xp = reinterpret_cast<__half*>(ws + l.xp_off);
  __half* wp = reinterpret_cast<__half*>(ws + l.w_off);
  int32_t* px = reinterpret_cast<int32_t*>(ws + l.px_off);
  int32_t* rx = reinterpret_cast<int32_t*>(ws + l.rx_off);
  int32_t* cw = reinterpret_cast<int32_t*>(ws + l.cw_off);
  const int oX = x_signed ? 0 : 128;
  const int oW = w_signed ? 0 : 128;

  // 1. padded, shifted input and its pixel sums (with the chunked pass, the
  //    weights of step 2 go through the same launch)
  const PrepassOperand wop = prepass_operand(w, c.Kg, K, c.Kg, c.Kgp, w_signed ? 1 : 0, wp, cw);
  bool weights_done = false;
  {
    const long long npix = c.N * c.Hp * c.Wp;
    const int vec = (C % 16 == 0) && aligned16(x);
    const int groups = C / 16;
    if (vec && groups <= 32 && (groups & (groups - 1)) == 0) {
      int log2g = 0;
      while ((1 << log2g) < groups) ++log2g;
      const long long threads = npix << log2g;
      const long long pix_blocks = (threads + 255) / 256;
      const long long w_blocks = (static_cast<long long>(K) + 7) / 8;  // 8 weight rows per block
      if (pix_blocks + w_blocks >= (1LL << 31)) return IGC_ERR_UNSUPPORTED;
      rc = launch_pdl(pad_shift_chunks_kernel, dim3(static_cast<unsigned>(pix_blocks + w_blocks)),
                      dim3(256), 0, stream, static_cast<const uint8_t*>(x),
                      x_signed ? 0x80808080u : 0u, zX - oX, N, H, W, C, pad_h, pad_w,
                      static_cast<int>(c.Hp), static_cast<int>(c.Wp), log2g, xp, px,
                      static_cast<unsigned>(w_blocks), wop, static_cast<int>(c.Kg),
                      static_cast<int>(c.Kgp));
      weights_done = true;
    } else {
      rc = launch_pdl(pad_shift_pixels_kernel, dim3(static_cast<unsigned>((npix + 7) / 8)),
                      dim3(256), 0, stream, static_cast<const uint8_t*>(x), x_signed ? 1 : 0, oX,
                      zX - oX, N, H, W, C, pad_h, pad_w, static_cast<int>(c.Hp),
                      static_cast<int>(c.Wp), vec, xp, px);
    }
    if (rc != IGC_OK) return rc;
  }
  // 2. weights: K rows of R*S*C values
  if (!weights_done) {
    rc = launch_prepass(&wop, 1, c.Kg, c.Kgp, stream);
    if (rc != IGC_OK) return rc;
  }
  // 3. window sums of the im2col rows: for small windows the GEMM's epilogue
  //    sums the pixel sums itself (R*S loads per output row, from L2)
  const bool sums_in_epilogue = R * S <= kEpilogueWindowMax;
  if (!sums_in_epilogue) {
    rc = launch_pdl(window_sums_kernel, dim3(static_cast<unsigned>((c.M + 255) / 256)),
                    dim3(256), 0, stream, static_cast<const int32_t*>(px), N,
                    static_cast<int>(c.Hp), static_cast<int>(c.Wp), static_cast<int>(c.P),
                    static_cast<int>(c.Q), R, S, stride_h, stride_w, rx);
    if (rc != IGC_OK) return rc;
  }

  // 4. the implicit GEMM over the padded tensor (no padding left for TMA)
  CUtensorMap tmA;
  rc = encode_im2col_nhwc(&tmA, xp, N, static_cast<int>(c.Hp), static_cast<int>(c.Wp), C, 0, 0,
                          -(R - 1), -(S - 1), BK, BM_CTA, stride_h, stride_w);
  if (rc != IGC_OK) return rc;

  KParams p{};
  p.M = static_cast<int>(c.M);
  p.N = K;
  p.K = static_cast<int>(c.Kg);
  p.conv_cblocks = (C + KS - 1) / KS;
  p.num_kb = R * S * p.conv_cblocks;
  p.chunk_kb = kIntChunkKb;
  p.conv_P = static_cast<int>(c.P);
  p.conv_Q = static_cast<int>(c.Q);
  p.conv_S = S;
  p.conv_C = C;
  p.pad_h = 0;
  p.pad_w = 0;
  p.stride_h = stride_h;
  p.stride_w = stride_w;
  p.c32 = y32;
  p.ldc32 = K;
  p.c8 = y8;
  p.ldc8 = K;
  p.rsumA = rx;
  if (sums_in_epilogue) {
    p.px = px;
    p.conv_R = R;
    p.conv_Hp = static_cast<int>(c.Hp);
    p.conv_Wp = static_cast<int>(c.Wp);
  }
  p.csumB = cw;
  p.zA = zX;
  p.zA_row = nullptr;
  p.zB = zW;
  p.zB_col = zW_k;
  p.oA = oX;
  p.oB = oW;
  p.scale = scale;
  p.scale_col = scale_k;
  p.vec_ok = vec_store_ok(y32, K, 4) && vec_store_ok(y8, K, 1);
  OutMaps om;
  add_out_map(om, 0, CU_TENSOR_MAP_DATA_TYPE_INT32, y32, K, c.M, K, 4);
  add_out_map(om, 1, CU_TENSOR_MAP_DATA_TYPE_UINT8, y8, K, c.M, K, 1);
  return launch_auto_bn<Mode::ConvInt>(dev, tmA, wp, c.Kgp, K, static_cast<uint64_t>(c.Kgp) * 2,
                                       om, p, stream);
}
