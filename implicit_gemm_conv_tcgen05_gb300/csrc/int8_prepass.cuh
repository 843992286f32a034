// Operand pre-pass of the exact-integer tensor-core path (shared by the int8
// GEMM and the int8 convolution): int8 / uint8 values shifted to [-128, 127]
// (uint8 minus 128, int8 unchanged) are written as fp16 -- exact -- with the
// row sums of the shifted values.
#pragma once

#include <cuda_fp16.h>

#include "igc_host.h"
#include "int8_widen.cuh"
#include "sm100_ptx.cuh"

namespace igc {
namespace prepass {

// One operand of the pre-pass: `rows` rows of K bytes (row stride ld), uint8
// (offset 128) or int8 (offset 0).
struct PrepassOperand {
  const uint8_t* src;
  long long ld;
  int rows;
  int is_signed;
  int offset;
  int vec;  // K % 16 == 0, 16-byte aligned rows: vector loads and stores
  __half* dst;
  int32_t* sums;
};

struct PrepassParams {
  PrepassOperand op[2];  // rows of op[0] first, then those of op[1]
  int K, Kp;
};

constexpr int kPrepassUnroll = 8;  // 8-byte loads in flight per thread

static __device__ __forceinline__ int shifted_byte(uint32_t byte, int is_signed, int offset) {
  return (is_signed ? static_cast<int>(static_cast<int8_t>(byte)) : static_cast<int>(byte)) -
         offset;
}

// One warp per row: dst[row, k] = fp16(src[row, k] - offset) for k < K, 0 for
// K <= k < Kp; sums[row] = sum_k (src[row, k] - offset).  Every lane of the
// warp must call it (the row sum is reduced by shuffles).
static __device__ __forceinline__ void widen_row(const PrepassOperand& o, int row, int K, int Kp,
                                                 int lane) {
  const uint8_t* s = o.src + static_cast<size_t>(row) * o.ld;
  __half* d = o.dst + static_cast<size_t>(row) * Kp;
  int32_t acc = 0;
  if (o.vec) {
    // offset 128 (uint8) keeps the byte, offset 0 (int8) flips its top bit
    const uint32_t flip = o.offset == 128 ? 0u : 0x80808080u;
    uint32_t usum = 0;  // sum of the u bytes; the shifted sum is usum - 128 K
    // lane l reads 8 bytes at k = 8 l + 256 i and writes their 16 output bytes, so
    // each warp-wide store covers 512 contiguous bytes
    for (int k0 = lane * 8; k0 < K; k0 += 32 * 8 * kPrepassUnroll) {
      uint2 raw[kPrepassUnroll];
#pragma unroll
      for (int u = 0; u < kPrepassUnroll; ++u) {
        const int k = k0 + u * 32 * 8;
        raw[u] = k < K ? __ldg(reinterpret_cast<const uint2*>(s + k)) : make_uint2(0, 0);
      }
#pragma unroll
      for (int u = 0; u < kPrepassUnroll; ++u) {
        const int k = k0 + u * 32 * 8;
        if (k >= K) break;
        uint32_t out[4];
        widen4(raw[u].x, flip, out[0], out[1], usum);
        widen4(raw[u].y, flip, out[2], out[3], usum);
        *reinterpret_cast<uint4*>(d + k) = make_uint4(out[0], out[1], out[2], out[3]);
      }
    }
    // the lane read 8 bytes at k = 8 lane + 256 i for every such k < K
    const uint32_t nbytes =
        K > lane * 8 ? 8u * static_cast<uint32_t>((K - lane * 8 + 255) / 256) : 0u;
    acc = static_cast<int32_t>(usum - 128u * nbytes);
  } else {
    for (int k = lane; k < Kp; k += 32) {
      int v = 0;
      if (k < K) v = shifted_byte(s[k], o.is_signed, o.offset);
      acc += v;
      d[k] = __int2half_rn(v);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) o.sums[row] = acc;
}

// Both operands of a GEMM go through one launch: rows of op[0], then of op[1].
static __global__ void __launch_bounds__(256) shift_widen_rowsum_kernel(const PrepassParams pp) {
  grid_dependency_wait();
  grid_dependents_launch();
  int row = blockIdx.x * (blockDim.x / 32) + static_cast<int>(threadIdx.x / 32);
  const int lane = static_cast<int>(threadIdx.x % 32);
  // select the operand field by field (a dynamic index into the parameter
  // struct would copy it to local memory)
  const bool second = row >= pp.op[0].rows;
  PrepassOperand o;
  o.src = second ? pp.op[1].src : pp.op[0].src;
  o.ld = second ? pp.op[1].ld : pp.op[0].ld;
  o.rows = second ? pp.op[1].rows : pp.op[0].rows;
  o.is_signed = second ? pp.op[1].is_signed : pp.op[0].is_signed;
  o.offset = second ? pp.op[1].offset : pp.op[0].offset;
  o.vec = second ? pp.op[1].vec : pp.op[0].vec;
  o.dst = second ? pp.op[1].dst : pp.op[0].dst;
  o.sums = second ? pp.op[1].sums : pp.op[0].sums;
  if (second) row -= pp.op[0].rows;
  if (row >= o.rows) return;
  widen_row(o, row, pp.K, pp.Kp, lane);
}

inline PrepassOperand prepass_operand(const void* src, long long ld, long long rows, long long K,
                               long long Kp, int is_signed, __half* dst, int32_t* sums) {
  PrepassOperand o;
  o.src = static_cast<const uint8_t*>(src);
  o.ld = ld;
  o.rows = static_cast<int>(rows);
  o.is_signed = is_signed;
  o.offset = is_signed ? 0 : 128;
  o.vec = (K % 16 == 0) && aligned16(src) && (ld % 16 == 0) && (Kp == K);
  o.dst = dst;
  o.sums = sums;
  return o;
}

inline int launch_prepass(const PrepassOperand* ops, int n_ops, long long K, long long Kp,
                   cudaStream_t stream) {
  PrepassParams pp{};
  pp.op[0] = ops[0];
  if (n_ops > 1) pp.op[1] = ops[1];
  pp.K = static_cast<int>(K);
  pp.Kp = static_cast<int>(Kp);
  const long long rows = static_cast<long long>(pp.op[0].rows) + (n_ops > 1 ? pp.op[1].rows : 0);
  const long long blocks = (rows + 7) / 8;
  return launch_pdl(shift_widen_rowsum_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                    stream, pp);
}

}  // namespace prepass
}  // namespace igc
