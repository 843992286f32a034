// Persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
// One kernel template serves the three operations of the library:
//   GemmF16 : C[i,j] = sum_k A[i,k] * Bt[j,k], fp16 operands, fp32 accumulate
//             (page "TVM在CUDA GPU上跑GEMM的全套张量化实现", §4.1: the GEMM compute
//             definition; §2.1: the tensor-core "row.col" operand forms, i.e. both
//             operands contiguous along k).
//   ConvF16 : the same contraction where row i of A is the im2col row of output
//             pixel (n, p, q) -- fetched by TMA in im2col mode, never materialised
//             (page "如何使用 TensorCores 优化卷积", section "准备和算法": Apad and the
//             reduction over ic, kh, kw).
//   GemmInt : exact integer GEMM of int8 operands that were shifted to [-128, 127]
//             and widened to fp16 by the pre-pass (every such value, and every
//             product, is exact in fp16/fp32), with the zero-point correction and
//             requantisation fused into the epilogue (page "TVM在CUDA GPU上跑GEMM
//             的全套张量化实现", §2.3).
//
// Tile 128 x 256 x 64, fp32 accumulators in tensor memory.  Warp roles:
//   warp 0      TMA producer (one lane): global -> 4-stage shared-memory ring,
//               128-byte swizzle, completion on `full[s]` mbarriers.
//   warp 1      MMA issuer (one lane): tcgen05.mma kind::f16 128x256x16, 4 per
//               k-block; tcgen05.commit frees ring stages (`empty[s]`) and hands
//               finished accumulators to the epilogue (`tfull[a]`).  Also owns the
//               tensor-memory allocation (512 columns = two accumulators, so the
//               epilogue of one tile overlaps the main loop of the next).
//   warps 2..9  epilogue: tcgen05.ld of their lane quadrant / column half, fused
//               output math, predicated global stores.
//
// GemmInt keeps each accumulation chunk (chunk_kb k-blocks = 256 k) below
// 2^22 in magnitude, so fp32 holds it exactly; the epilogue drains every chunk
// into an int32 running sum with the round-to-integer trick x + 1.5*2^23.
#pragma once

#include <cuda_fp16.h>

#include "sm100_ptx.cuh"

namespace igc {

enum class Mode : int { GemmF16 = 0, ConvF16 = 1, GemmInt = 2 };

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;  // 64 fp16 = one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;  // 320
constexpr uint32_t kTmemCols = 2 * BN;         // two 128 x 256 fp32 accumulators
constexpr uint32_t kStageABytes = BM * BK * 2;
constexpr uint32_t kStageBBytes = BN * BK * 2;
constexpr uint32_t kBarrierBytes = 256;
constexpr size_t kSmemBytes = 1024 /*alignment slack*/ +
                              kStages * (kStageABytes + kStageBBytes) + kBarrierBytes;
constexpr int kIntChunkKb = 4;  // 256 k per exact fp32 chunk

// wait sites, reported in the device status word
enum : uint32_t {
  kSiteProducerEmpty = 1,
  kSiteMmaTmemEmpty = 2,
  kSiteMmaFull = 3,
  kSiteEpiFull = 4,
  kSiteDrain = 5,
};

struct KParams {
  // GEMM view of the problem
  int M, N, K;
  int num_kb;
  int tiles_m, tiles_n, num_tiles;
  int group_m;   // tile raster: this many m-blocks are walked together
  int chunk_kb;  // k-blocks per accumulation chunk (>= num_kb except GemmInt)
  // convolution geometry (ConvF16)
  int conv_P, conv_Q, conv_cblocks, conv_S, conv_C;
  int pad_h, pad_w, stride_h, stride_w;
  // floating outputs (GemmF16 / ConvF16)
  void* out;
  long long ldo;
  int out_f16;  // 1: out is fp16 (RNE), 0: out is fp32
  float* out_f32;
  long long ldo32;
  int vec_ok;  // outputs allow 16-byte vector stores
  // integer outputs (GemmInt)
  int32_t* c32;
  long long ldc32;
  int8_t* c8;
  long long ldc8;
  const int32_t* rsumA;  // sum_k A'[i,k] of the shifted operand
  const int32_t* csumB;  // sum_k B'[j,k]
  int32_t zA;
  const int32_t* zA_row;
  int32_t zB;
  const int32_t* zB_col;
  int32_t oA, oB;  // shift applied by the pre-pass: A' = A_q - oA, B' = B_q - oB
  float scale;
  const float* scale_col;
  // control
  unsigned long long wait_limit_ns;
  unsigned long long* status;
};

__device__ __forceinline__ void tile_coords(const KParams& p, int t, int& mb, int& nb) {
  const int per_group = p.group_m * p.tiles_n;
  const int g = t / per_group;
  const int first_m = g * p.group_m;
  const int gm = min(p.tiles_m - first_m, p.group_m);
  const int r = t - g * per_group;
  mb = first_m + r % gm;
  nb = r / gm;
}

// ---------------------------------------------------------------------------
// epilogue helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_half2(uint32_t lo_bits, uint32_t hi_bits) {
  __half2 h = __floats2half2_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
  return *reinterpret_cast<uint32_t*>(&h);
}

// Row m of the tile, columns n0 .. n0+127, values v (fp32 bit patterns).
__device__ __forceinline__ void store_row_float(const KParams& p, int m, int n0,
                                                const uint32_t (&v)[128]) {
  if (m >= p.M) return;
  const bool full = p.vec_ok && (n0 + 128 <= p.N);
  if (p.out != nullptr) {
    if (p.out_f16) {
      __half* row = reinterpret_cast<__half*>(p.out) + static_cast<size_t>(m) * p.ldo + n0;
      if (full) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          uint4 q;
          q.x = pack_half2(v[8 * j + 0], v[8 * j + 1]);
          q.y = pack_half2(v[8 * j + 2], v[8 * j + 3]);
          q.z = pack_half2(v[8 * j + 4], v[8 * j + 5]);
          q.w = pack_half2(v[8 * j + 6], v[8 * j + 7]);
          reinterpret_cast<uint4*>(row)[j] = q;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (n0 + i < p.N) row[i] = __float2half_rn(__uint_as_float(v[i]));
      }
    } else {
      float* row = reinterpret_cast<float*>(p.out) + static_cast<size_t>(m) * p.ldo + n0;
      if (full) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          reinterpret_cast<uint4*>(row)[j] =
              make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (n0 + i < p.N) row[i] = __uint_as_float(v[i]);
      }
    }
  }
  if (p.out_f32 != nullptr) {
    float* row = p.out_f32 + static_cast<size_t>(m) * p.ldo32 + n0;
    if (full) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        reinterpret_cast<uint4*>(row)[j] =
            make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 128; ++i)
        if (n0 + i < p.N) row[i] = __uint_as_float(v[i]);
    }
  }
}

__device__ __forceinline__ int8_t requant_i8(int32_t c, float s) {
  // fp32(c) rounded to nearest even, one fp32 multiply, round half to even, clamp.
  const float f = __fmul_rn(__int2float_rn(c), s);
  int q = __float2int_rn(f);  // NaN -> 0, +-inf saturate
  q = max(-128, min(127, q));
  return static_cast<int8_t>(q);
}

// sum[] holds, per column, n_chunks * 0x4B400000 + sum_k A'B' (mod 2^32).
__device__ __forceinline__ void store_row_int(const KParams& p, int m, int n0,
                                              const uint32_t (&sum)[128], int n_chunks) {
  if (m >= p.M) return;
  const uint32_t bias = static_cast<uint32_t>(n_chunks) * 0x4B400000u;
  const uint32_t rA = static_cast<uint32_t>(p.rsumA[m]);
  const uint32_t zAp = static_cast<uint32_t>((p.zA_row ? __ldg(p.zA_row + m) : p.zA) - p.oA);
  const uint32_t Ku = static_cast<uint32_t>(p.K);
  const bool full = p.vec_ok && (n0 + 128 <= p.N);
  int32_t* row32 = p.c32 ? p.c32 + static_cast<size_t>(m) * p.ldc32 + n0 : nullptr;
  int8_t* row8 = p.c8 ? p.c8 + static_cast<size_t>(m) * p.ldc8 + n0 : nullptr;
#pragma unroll
  for (int j = 0; j < 8; ++j) {  // 16 columns per step
    int32_t c[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int col = j * 16 + i;
      const int n = n0 + col;
      const int nn = n < p.N ? n : p.N - 1;  // keep the side loads in bounds on the tail
      const uint32_t zBp = static_cast<uint32_t>((p.zB_col ? __ldg(p.zB_col + nn) : p.zB) - p.oB);
      const uint32_t cB = static_cast<uint32_t>(__ldg(p.csumB + nn));
      const uint32_t v = sum[col] - bias - zBp * rA - zAp * cB + Ku * zAp * zBp;
      c[i] = static_cast<int32_t>(v);
    }
    if (row32) {
      if (full) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          reinterpret_cast<int4*>(row32 + j * 16)[i] =
              make_int4(c[4 * i], c[4 * i + 1], c[4 * i + 2], c[4 * i + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (n0 + j * 16 + i < p.N) row32[j * 16 + i] = c[i];
      }
    }
    if (row8) {
      int8_t q[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int n = n0 + j * 16 + i;
        const int nn = n < p.N ? n : p.N - 1;
        const float s = p.scale_col ? __ldg(p.scale_col + nn) : p.scale;
        q[i] = requant_i8(c[i], s);
      }
      if (full) {
        uint4 w;
        w.x = (uint32_t)(uint8_t)q[0] | ((uint32_t)(uint8_t)q[1] << 8) |
              ((uint32_t)(uint8_t)q[2] << 16) | ((uint32_t)(uint8_t)q[3] << 24);
        w.y = (uint32_t)(uint8_t)q[4] | ((uint32_t)(uint8_t)q[5] << 8) |
              ((uint32_t)(uint8_t)q[6] << 16) | ((uint32_t)(uint8_t)q[7] << 24);
        w.z = (uint32_t)(uint8_t)q[8] | ((uint32_t)(uint8_t)q[9] << 8) |
              ((uint32_t)(uint8_t)q[10] << 16) | ((uint32_t)(uint8_t)q[11] << 24);
        w.w = (uint32_t)(uint8_t)q[12] | ((uint32_t)(uint8_t)q[13] << 8) |
              ((uint32_t)(uint8_t)q[14] << 16) | ((uint32_t)(uint8_t)q[15] << 24);
        reinterpret_cast<uint4*>(row8)[j] = w;
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (n0 + j * 16 + i < p.N) row8[j * 16 + i] = q[i];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <Mode kMode>
__global__ void __launch_bounds__(kThreads, 1)
    igc_tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB, const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);

  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kStageABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kStages * kStageBBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 32, 0);
  const int lane = static_cast<int>(lane_id());

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiWarps);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint64_t lim = p.wait_limit_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
        int mb, nb;
        tile_coords(p, t, mb, nb);
        int cn = 0, ch = 0, cw = 0;
        if constexpr (kMode == Mode::ConvF16) {
          const int m0 = mb * BM;
          const int PQ = p.conv_P * p.conv_Q;
          cn = m0 / PQ;
          const int rem = m0 - cn * PQ;
          const int pp = rem / p.conv_Q;
          const int qq = rem - pp * p.conv_Q;
          ch = pp * p.stride_h - p.pad_h;
          cw = qq * p.stride_w - p.pad_w;
        }
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, lim, abort_flag, p.status, kSiteProducerEmpty))
            goto producer_done;
          uint8_t* a_dst = sA + stage * kStageABytes;
          uint8_t* b_dst = sB + stage * kStageBBytes;
          mbar_arrive_expect_tx(&full[stage], kStageABytes + kStageBBytes);
          if constexpr (kMode == Mode::ConvF16) {
            const int tap = kb / p.conv_cblocks;
            const int c0 = (kb - tap * p.conv_cblocks) * BK;
            const int r = tap / p.conv_S;
            const int s = tap - r * p.conv_S;
            tma_load_im2col_4d(a_dst, &tmA, &full[stage], c0, cw, ch, cn,
                               static_cast<uint16_t>(s), static_cast<uint16_t>(r));
            tma_load_2d(b_dst, &tmB, &full[stage], tap * p.conv_C + c0, nb * BN);
          } else {
            tma_load_2d(a_dst, &tmA, &full[stage], kb * BK, mb * BM);
            tma_load_2d(b_dst, &tmB, &full[stage], kb * BK, nb * BN);
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    producer_done:
      // Make sure no copy into this CTA's shared memory is still in flight
      // before the CTA can exit (only matters when a wait gave up).
      if (*abort_flag) {
        int s = stage;
        uint32_t ph = phase;
        for (long long i = 0; i < issued && i < kStages; ++i) {
          if (--s < 0) {
            s = kStages - 1;
            ph ^= 1u;
          }
          int dummy = 0;
          mbar_wait(&full[s], ph, lim, &dummy, nullptr, kSiteDrain);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_f16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
        for (int kb = 0; kb < p.num_kb; ++kb) {
          const int kin = kb % p.chunk_kb;
          if (kin == 0) {
            if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, lim, abort_flag, p.status,
                           kSiteMmaTmemEmpty))
              goto mma_done_label;
            tc_fence_after();
          }
          if (!mbar_wait(&full[stage], phase, lim, abort_flag, p.status, kSiteMmaFull))
            goto mma_done_label;
          tc_fence_after();
          {
            const uint32_t a_base = smem_u32(sA + stage * kStageABytes);
            const uint32_t b_base = smem_u32(sB + stage * kStageBBytes);
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              const uint64_t ad = make_sw128_kmajor_desc(a_base + k * 32);
              const uint64_t bd = make_sw128_kmajor_desc(b_base + k * 32);
              umma_f16_ss(d_tmem, ad, bd, idesc, (kin > 0 || k > 0) ? 1u : 0u);
            }
          }
          umma_commit(&empty[stage]);
          if (kin == p.chunk_kb - 1 || kb == p.num_kb - 1) {
            umma_commit(&tfull[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    mma_done_label:
      // every MMA issued by this thread has finished once mma_done completes
      umma_commit(mma_done);
      {
        int dummy = 0;
        mbar_wait(mma_done, 0, lim, &dummy, p.status, kSiteDrain);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int quad = warp & 3;  // tcgen05.ld: warp w may access lanes 32*(w%4) .. +31
    const int half = ew >> 2;   // which 128-column half of the tile
    const int row_in_tile = quad * 32 + lane;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                               static_cast<uint32_t>(half * 128);
    const int n_chunks = (p.num_kb + p.chunk_kb - 1) / p.chunk_kb;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(p, t, mb, nb);
      const int m = mb * BM + row_in_tile;
      const int n0 = nb * BN + half * 128;
      if constexpr (kMode != Mode::GemmInt) {
        // every lane waits (acquire); the warp then agrees before the .aligned loads
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&tfull[acc], acc_phase, lim, abort_flag, p.status, kSiteEpiFull)))
          goto epi_done;
        tc_fence_after();
        uint32_t v[128];
        {
          const uint32_t a = lane_base + static_cast<uint32_t>(acc * BN);
          uint32_t r0[32], r1[32], r2[32], r3[32];
          tmem_ld_32x32b_x32(a + 0, r0);
          tmem_ld_32x32b_x32(a + 32, r1);
          tmem_ld_32x32b_x32(a + 64, r2);
          tmem_ld_32x32b_x32(a + 96, r3);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v[i] = r0[i];
            v[32 + i] = r1[i];
            v[64 + i] = r2[i];
            v[96 + i] = r3[i];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
        store_row_float(p, m, n0, v);
      } else {
        uint32_t sum[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) sum[i] = 0u;
        for (int c = 0; c < n_chunks; ++c) {
          if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, lim, abort_flag,
                                                  p.status, kSiteEpiFull)))
            goto epi_done;
          tc_fence_after();
          const uint32_t a = lane_base + static_cast<uint32_t>(acc * BN);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(a + j * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              sum[j * 32 + i] += __float_as_uint(__fadd_rn(__uint_as_float(r[i]), 12582912.0f));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[acc]);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
        store_row_int(p, m, n0, sum, n_chunks);
      }
    }
  epi_done:;
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace igc
