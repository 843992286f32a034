// INT8 GEMM with input zero points on the tcgen05 fp16 pipe, the operands
// converted inside the kernel (page "TVM在CUDA GPU上跑GEMM的全套张量化实现", §2.3:
// C = (A_q - zp_A)(B_q - zp_B) in one fused pass; the page's four-term fusion
// reads the quantised operands once and writes the output once).
//
// sm_103a has no integer tcgen05 MMA kind, so the int8 values are shifted to
// [-128, 127] (uint8 minus 128, int8 as is) and widened to fp16 -- exact -- and
// multiplied on the kind::f16 pipe in exact 1024-k fp32 chunks (as in the
// GemmInt mode of gemm_tc.cuh).  Here the widening happens on chip, so the
// quantised operands are read from HBM once and nothing else is written:
//
//   TMA (int8 tiles, 64 k per stage) -> int8 ring in shared memory
//     -> converter warpgroup: 16-byte loads, shift + widen to fp16 (byte
//        permutes against the fp16 pattern of 1024 and one packed subtraction),
//        16-byte stores into the 128-byte-swizzled K-major layout the UMMA
//        descriptors read; row sums of the shifted operands in the same pass
//     -> fp16 ring -> tcgen05.mma.cta_group::2.kind::f16 -> TMEM
//     -> epilogue: exact chunk drains into int32, zero-point correction with
//        the sums the converters left in shared memory, requantisation.
//
// Roles in each CTA of the pair (512 threads, four warpgroups):
//   warp 0      TMA producer of this CTA's int8 A rows and B rows (its own
//               barriers: each CTA converts what it loads).
//   warp 1      tensor-memory owner; in the leader CTA the MMA issuer.
//   warps 2-3   idle (their warpgroup gives registers away).
//   warps 4-7   converters.  Per 64-k stage, thread t converts items
//               (row 32 i + t / 4, 16-byte piece t % 4) of the A and B tiles, so
//               that every 8 lanes read 128 contiguous bytes and write eight
//               distinct bank groups of the swizzled rows.
//   warps 8-15  epilogue, as in gemm_tc.cuh's integer modes.
// Barriers: i8full / i8empty (producer <-> own converters), f16full (both
// CTAs' converters -> leader's MMA: each converter thread fences its stores to
// the async proxy, then lane 0 arrives; each CTA's tensor core reads only what
// its own converters wrote), f16empty (MMA commit, multicast), tfull / tempty
// (accumulators), sfull / sempty (the per-unit sums in shared memory,
// double-buffered, read by both CTAs' epilogues through the cluster window:
// release / acquire at cluster scope, once per unit).  The per-stage hand-off
// uses CTA-scope arrivals: with cluster-scope release / acquire on it the
// kernel ran 1.9 ms instead of 1.07 ms at 8192^3 (each cluster-scope release
// stalls the arriving warp on a memory barrier).
//
// Measured on GB300 at 8192^3 (u8 x s8, per-row zA, C8 out): 1074 us, against
// 592 us for the pre-pass + GEMM path (IGC_INT8_PATH_TCGEN05).  With the
// conversion taken out (barrier protocol and int8 TMA only) the kernel takes
// 500 us, less than the pre-pass path's GEMM (532 us), since int8 tiles move
// half the bytes.  Two costs then hold it near twice the MMA time each: the
// shared-memory stores of the fp16 stages beside the tensor cores' and TMA's
// traffic (stores alone: 902 us), and the conversion arithmetic on four
// converter warps per SM (every tile converts its own A and B panels, 4.3 GB of
// int8 for 128 MB of distinct operand bytes, about 1.8 instructions per byte).
// The BN = 256 instantiations spill a few words (ptxas: 24-36 bytes) at this
// register split; the epilogue needs its 208 and the converters their 64.
#pragma once

#include "gemm_tc.cuh"
#include "int8_prepass.cuh"

namespace igc {

constexpr int kI8Threads = 512;
constexpr int kI8ConvThreads = 128;
// Register split over the four warpgroups (setmaxnreg): control 32, converters
// 64, epilogue 208 each; 32 * 128 + 64 * 128 + 208 * 256 = 65536 registers, the
// launch's 512 threads x 128.
constexpr int kI8RegsCtl = 32;
constexpr int kI8RegsCvt = 64;
constexpr int kI8RegsEpi = 208;
constexpr int kI8LaunchRegs = 128;
static_assert(kI8RegsCtl * 128 + kI8RegsCvt * 128 + kI8RegsEpi * 256 <=
                  kI8Threads * kI8LaunchRegs,
              "register split");
// setmaxnreg.dec may only lower a warpgroup's count and setmaxnreg.inc only
// raise it: the control and converter warpgroups give registers away (dec from
// the launch's 128), the epilogue warpgroups take them (inc).
static_assert(kI8RegsCtl <= kI8LaunchRegs && kI8RegsCvt <= kI8LaunchRegs &&
                  kI8RegsEpi >= kI8LaunchRegs,
              "register split direction");
constexpr int kI8KS = 64;                   // k per stage
constexpr int kI8ChunkKb = 1024 / kI8KS;    // stages per exact fp32 chunk

template <int BN>
struct I8Cfg {
  static_assert(BN == 256 || BN == 128, "BN");
  static constexpr int kBRows = BN / 2;                         // B rows per CTA, whole unit
  static constexpr uint32_t kF16A = BM_CTA * kI8KS * 2;          // 16 KB
  static constexpr uint32_t kF16B = kBRows * kI8KS * 2;
  static constexpr uint32_t kF16Stage = kF16A + kF16B;
  static constexpr uint32_t kI8A = BM_CTA * kI8KS;               // 8 KB
  static constexpr uint32_t kI8B = kBRows * kI8KS;
  static constexpr uint32_t kI8Stage = kI8A + kI8B;
  static constexpr int kF16Stages = BN == 256 ? 3 : 4;
  static constexpr uint32_t kSumsBytes = 2u * (BM_CTA + kBRows) * 4u;
  static constexpr uint32_t kBarBytes = 512;
  static constexpr size_t kFixed = 1024 + kF16Stages * kF16Stage + kStagingBytes + kSumsBytes +
                                   kBarBytes;
  static constexpr int kI8StagesFit = static_cast<int>((kSmemBudget - kFixed) / kI8Stage);
  static constexpr int kI8Stages = kI8StagesFit > 8 ? 8 : kI8StagesFit;
  static_assert(kI8Stages >= 3, "int8 ring");
  static constexpr size_t kSmemBytes = kFixed + kI8Stages * kI8Stage;
  static_assert(kSmemBytes <= kSmemBudget, "shared memory");
  static constexpr uint32_t kTmemCols = 2 * BN <= 256 ? 256 : 512;
  static constexpr uint32_t kAccStride = kTmemCols / 2;
  static constexpr int kEpiCols = BN / 2;
};

enum : uint32_t {
  kSiteCvtFull = 7,
  kSiteCvtEmpty = 8,
  kSiteSumsEmpty = 9,
  kSiteSumsFull = 10,
};

// Converts one 16-byte item of int8 values (k0 .. k0+15 of a row) into the
// fp16 row at `dst_row` (128-byte swizzled, 16-byte chunks 2 c and 2 c + 1),
// adding the sum of the u bytes (value + 128) to usum.  Bytes at k >= K
// convert as the value 0 (u = 128).
__device__ __forceinline__ void cvt_item(uint4 raw, uint32_t flip, uint8_t* dst_row, int r, int c,
                                         int valid, uint32_t& usum) {
  uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  if (valid < 16) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int nv = valid - 4 * j;
      const uint32_t keep = nv >= 4 ? 0xFFFFFFFFu : (nv <= 0 ? 0u : (1u << (8 * nv)) - 1u);
      w[j] = (w[j] & keep) | ((0x80808080u ^ flip) & ~keep);
    }
  }
  uint32_t o[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) prepass::widen4(w[j], flip, o[2 * j], o[2 * j + 1], usum);
  const int x = r & 7;
  *reinterpret_cast<uint4*>(dst_row + (((2 * c) ^ x) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
  *reinterpret_cast<uint4*>(dst_row + (((2 * c + 1) ^ x) << 4)) =
      make_uint4(o[4], o[5], o[6], o[7]);
}

// One converter thread's share of a 64-k stage: its four A items (rows r0 + 32 i)
// and NBI B items, two in flight at a time (the converters run on a small
// register budget).
template <int NBI>
__device__ __forceinline__ void convert_stage(const uint8_t* srcA, const uint8_t* srcB,
                                              uint8_t* dstA, uint8_t* dstB, int r0, int c,
                                              int valid, uint32_t flipA, uint32_t flipB,
                                              uint32_t (&usA)[4], uint32_t (&usB)[4]) {
#pragma unroll
  for (int i = 0; i < 4; i += 2) {
    const int ra0 = r0 + 32 * i, ra1 = ra0 + 32;
    const uint4 x0 = *reinterpret_cast<const uint4*>(srcA + ra0 * kI8KS + c * 16);
    const uint4 x1 = *reinterpret_cast<const uint4*>(srcA + ra1 * kI8KS + c * 16);
    cvt_item(x0, flipA, dstA + ra0 * 128, ra0, c, valid, usA[i]);
    cvt_item(x1, flipA, dstA + ra1 * 128, ra1, c, valid, usA[i + 1]);
  }
#pragma unroll
  for (int i = 0; i < NBI; i += 2) {
    const int rb0 = r0 + 32 * i;
    const uint4 x0 = *reinterpret_cast<const uint4*>(srcB + rb0 * kI8KS + c * 16);
    if (i + 1 < NBI) {
      const int rb1 = rb0 + 32;
      const uint4 x1 = *reinterpret_cast<const uint4*>(srcB + rb1 * kI8KS + c * 16);
      cvt_item(x0, flipB, dstB + rb0 * 128, rb0, c, valid, usB[i]);
      cvt_item(x1, flipB, dstB + rb1 * 128, rb1, c, valid, usB[i + 1]);
    } else {
      cvt_item(x0, flipB, dstB + rb0 * 128, rb0, c, valid, usB[i]);
    }
  }
}

template <int BN, bool kDequant>
__global__ void __launch_bounds__(kI8Threads, 1)
    igc_i8_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmBh,
                       const __grid_constant__ CUtensorMap tmO0,
                       const __grid_constant__ CUtensorMap tmO1,
                       const __grid_constant__ CUtensorMap tmO2, const KParams p,
                       const uint32_t flipA, const uint32_t flipB) {
  using Cfg = I8Cfg<BN>;
  constexpr int kF16Stages = Cfg::kF16Stages;
  constexpr int kI8Stages = Cfg::kI8Stages;
  constexpr int NC = Cfg::kEpiCols;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);

  uint8_t* sF16 = smem;                                    // kF16Stages x (A 16 KB, B)
  uint8_t* staging = sF16 + kF16Stages * Cfg::kF16Stage;   // 1024-byte aligned
  uint8_t* sI8 = staging + kStagingBytes;                  // kI8Stages x (A 8 KB, B)
  int32_t* sums = reinterpret_cast<int32_t*>(sI8 + kI8Stages * Cfg::kI8Stage);
  // sums[b * (128 + kBRows) + i]: rA' of row i (i < 128), then cB' of this CTA's B rows
  uint64_t* bars = reinterpret_cast<uint64_t*>(sums + 2 * (BM_CTA + Cfg::kBRows));
  uint64_t* i8full = bars;
  uint64_t* i8empty = i8full + kI8Stages;
  uint64_t* f16full = i8empty + kI8Stages;    // leader: both CTAs' converters
  uint64_t* f16empty = f16full + kF16Stages;  // each CTA: MMA done with the stage
  uint64_t* tfull = f16empty + kF16Stages;
  uint64_t* tempty = tfull + 2;
  uint64_t* sfull = tempty + 2;               // each CTA: both CTAs' sums of a unit written
  uint64_t* sempty = sfull + 2;               // each CTA: both CTAs' epilogues read them
  uint64_t* mma_done = sempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 32, 0);
  const int lane = static_cast<int>(lane_id());
  const uint32_t rank = cluster_ctarank();  // 0 = leader
  const uint32_t peer = rank ^ 1u;
  const int cluster = static_cast<int>(blockIdx.x) >> 1;
  const int num_clusters = static_cast<int>(gridDim.x) >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kI8Stages; ++s) {
      mbar_init(&i8full[s], 1);
      mbar_init(&i8empty[s], kI8ConvThreads / 32);
    }
    for (int s = 0; s < kF16Stages; ++s) {
      mbar_init(&f16full[s], 2 * kI8ConvThreads / 32);
      mbar_init(&f16empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * kEpiWarps);
      mbar_init(&sfull[a], 2 * kI8ConvThreads / 32);
      mbar_init(&sempty[a], 2 * kEpiWarps);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmBh);
  }
  if (warp == 1) {
    tmem_alloc_2cta(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish_2cta();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after();
  grid_dependency_wait();  // programmatic dependent launch, as in gemm_tc.cuh
  grid_dependents_launch();
  const uint32_t tmem_base = *tmem_slot;
  const uint64_t lim = p.wait_limit_ns;
  const uint32_t peer_base = ld_shared_cluster_u32(mapa_shared(smem_u32(tmem_slot), peer));
  const bool pair_ok = peer_base == tmem_base;
  if (!pair_ok && threadIdx.x == 0) report_status(p.status, kStatusBadLaunch, kSiteTmemMismatch);
  const uint32_t f16full_lead = mapa_shared(smem_u32(f16full), 0);
  const uint32_t tempty_lead = mapa_shared(smem_u32(tempty), 0);
  const int nkb = p.num_kb;

  if (warp < 4) {
    warpgroup_regs_dec<kI8RegsCtl>();
    if (pair_ok && warp == 0) {
      // ---------------------------------------------------------- TMA producer (int8)
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      for (int u = cluster; u < p.num_units; u += num_clusters) {
        const Unit w = unit_coords(p, u);
        const int m_cta = w.mb * BM + static_cast<int>(rank) * BM_CTA;
        const int n_cta = w.half ? w.nb * BN + w.j * (BN / 2) + static_cast<int>(rank) * (BN / 4)
                                 : w.nb * BN + static_cast<int>(rank) * Cfg::kBRows;
        const CUtensorMap* mapB = w.half ? &tmBh : &tmB;
        const uint32_t tx = Cfg::kI8A + (w.half ? Cfg::kI8B / 2 : Cfg::kI8B);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(&i8empty[stage], phase ^ 1u, lim, abort_flag,
                                                  p.status, kSiteProducerEmpty)))
            goto producer_done;
          if (lane == 0) {
            uint8_t* dst = sI8 + stage * Cfg::kI8Stage;
            mbar_arrive_expect_tx(&i8full[stage], tx);
            tma_load_2d(dst, &tmA, &i8full[stage], kb * kI8KS, m_cta);
            tma_load_2d(dst + Cfg::kI8A, mapB, &i8full[stage], kb * kI8KS, n_cta);
          }
          __syncwarp();
          ++issued;
          if (++stage == kI8Stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    producer_done:
      if (lane == 0 && *abort_flag && issued > 0)
        drain_fills(i8full, kI8Stages, stage, phase, issued, lim);
    } else if (pair_ok && warp == 1 && rank == 0) {
      // ---------------------------------------------------------- MMA issuer (leader)
      constexpr uint32_t idesc_full = make_idesc_kind_f16(BM, BN, 0u);
      constexpr uint32_t idesc_half = make_idesc_kind_f16(BM, BN / 2, 0u);
      const uint64_t adesc0 = make_sw128_kmajor_desc(smem_u32(sF16));
      const uint64_t bdesc0 = make_sw128_kmajor_desc(smem_u32(sF16 + Cfg::kF16A));
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int u = cluster; u < p.num_units; u += num_clusters) {
        const uint32_t idesc = u >= p.tail_start ? idesc_half : idesc_full;
        int kin = 0;
        for (int kb = 0; kb < nkb; ++kb) {
          if (kin == 0) {
            if (!__all_sync(0xffffffffu, mbar_wait(&tempty[acc], acc_phase ^ 1u, lim,
                                                    abort_flag, p.status, kSiteMmaTmemEmpty)))
              goto mma_done_label;
            tc_fence_after();
          }
          if (!__all_sync(0xffffffffu, mbar_wait(&f16full[stage], phase, lim, abort_flag,
                                                        p.status, kSiteMmaFull)))
            goto mma_done_label;
          tc_fence_after();
          const bool chunk_end = (kin == kI8ChunkKb - 1) || (kb == nkb - 1);
          if (lane == 0) {
            const uint32_t off = (static_cast<uint32_t>(stage) * Cfg::kF16Stage) >> 4;
            mma_stage<1, 0>(tmem_base + static_cast<uint32_t>(acc) * Cfg::kAccStride,
                            adesc0 + off, bdesc0 + off, idesc, kin > 0);
            umma_commit_2cta_multicast(&f16empty[stage], 0x3);
            if (chunk_end) umma_commit_2cta_multicast(&tfull[acc], 0x3);
          }
          __syncwarp();
          if (chunk_end) {
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
          }
          if (++kin == kI8ChunkKb) kin = 0;
          if (++stage == kF16Stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    mma_done_label:
      if (lane == 0) {
        umma_commit_2cta(mma_done);
        int dummy = 0;
        mbar_wait(mma_done, 0, lim, &dummy, p.status, kSiteDrain);
      }
      __syncwarp();
    }
  } else if (warp < 8) {
    warpgroup_regs_dec<kI8RegsCvt>();
    if (pair_ok) {
      // ---------------------------------------------------------- converters
      const int t = static_cast<int>(threadIdx.x) - 128;  // 0 .. 127
      const int c = t & 3;                                // 16-byte piece of a 64-byte row
      const int r0 = t >> 2;                              // rows r0 + 32 i
      int s8 = 0, s16 = 0, ub = 0;
      uint32_t ph8 = 0, ph16 = 0, sph = 0;
      const uint32_t sfull_own = mapa_shared(smem_u32(sfull), rank);
      const uint32_t sfull_peer = mapa_shared(smem_u32(sfull), peer);
      for (int u = cluster; u < p.num_units; u += num_clusters) {
        const bool half_unit = u >= p.tail_start;
        const int nbi = (half_unit ? BN / 4 : BN / 2) / 32;  // B items per thread
        uint32_t usA[4] = {0u, 0u, 0u, 0u};
        uint32_t usB[4] = {0u, 0u, 0u, 0u};
        for (int kb = 0; kb < nkb; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(&i8full[s8], ph8, lim, abort_flag, p.status,
                                                  kSiteCvtFull)))
            goto cvt_done;
          if (!__all_sync(0xffffffffu, mbar_wait(&f16empty[s16], ph16 ^ 1u, lim, abort_flag,
                                                  p.status, kSiteCvtEmpty)))
            goto cvt_done;
          {
            const uint8_t* srcA = sI8 + s8 * Cfg::kI8Stage;
            const uint8_t* srcB = srcA + Cfg::kI8A;
            uint8_t* dstA = sF16 + s16 * Cfg::kF16Stage;
            uint8_t* dstB = dstA + Cfg::kF16A;
            const int valid = p.K - (kb * kI8KS + c * 16);  // bytes of this piece below K
            if (nbi == 4)
              convert_stage<4>(srcA, srcB, dstA, dstB, r0, c, valid, flipA, flipB, usA, usB);
            else if (nbi == 2)
              convert_stage<2>(srcA, srcB, dstA, dstB, r0, c, valid, flipA, flipB, usA, usB);
            else
              convert_stage<1>(srcA, srcB, dstA, dstB, r0, c, valid, flipA, flipB, usA, usB);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive_local(&i8empty[s8]);
            mbar_arrive_remote(f16full_lead + static_cast<uint32_t>(s16) * 8u);
          }
          if (++s8 == kI8Stages) {
            s8 = 0;
            ph8 ^= 1u;
          }
          if (++s16 == kF16Stages) {
            s16 = 0;
            ph16 ^= 1u;
          }
        }
        // row sums of this unit: the four lanes of a row hold its four pieces
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          usA[i] += __shfl_xor_sync(0xffffffffu, usA[i], 1);
          usA[i] += __shfl_xor_sync(0xffffffffu, usA[i], 2);
          usB[i] += __shfl_xor_sync(0xffffffffu, usB[i], 1);
          usB[i] += __shfl_xor_sync(0xffffffffu, usB[i], 2);
        }
        if (!__all_sync(0xffffffffu, mbar_wait<true>(&sempty[ub], sph ^ 1u, lim, abort_flag,
                                                      p.status, kSiteSumsEmpty)))
          goto cvt_done;
        if (c == 0) {
          // shifted sums: sum of u - 128 per byte over the nkb * 64 bytes converted
          const uint32_t bias = 128u * static_cast<uint32_t>(nkb) * static_cast<uint32_t>(kI8KS);
          int32_t* sb = sums + ub * (BM_CTA + Cfg::kBRows);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            sb[r0 + 32 * i] = static_cast<int32_t>(usA[i] - bias);
            if (i < nbi) sb[BM_CTA + r0 + 32 * i] = static_cast<int32_t>(usB[i] - bias);
          }
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_cluster(sfull_own + static_cast<uint32_t>(ub) * 8u);
          mbar_arrive_cluster(sfull_peer + static_cast<uint32_t>(ub) * 8u);
        }
        ub ^= 1;
        if (ub == 0) sph ^= 1u;
      }
    cvt_done:;
    }
  } else {
    warpgroup_regs_inc<kI8RegsEpi>();
    if (pair_ok) {
      // ---------------------------------------------------------- epilogue
      const int ew = warp - 8;
      const int quad = warp & 3;
      const int half = ew >> 2;
      const int row_in_cta = quad * 32 + lane;
      const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                 static_cast<uint32_t>(half * NC);
      const int n_chunks = (nkb + kI8ChunkKb - 1) / kI8ChunkKb;
      const uint32_t sums_own = smem_u32(sums);
      const uint32_t sempty_own = mapa_shared(smem_u32(sempty), rank);
      const uint32_t sempty_peer = mapa_shared(smem_u32(sempty), peer);
      Stager st;
      st.buf = staging + ew * kStagingWarpBytes;
      st.lane = lane;
      st.M = p.M;
      st.N = p.N;
      int acc = 0, ub = 0;
      uint32_t acc_phase = 0, sph = 0;
      for (int u = cluster; u < p.num_units; u += num_clusters) {
        const Unit w = unit_coords(p, u);
        const int m = w.mb * BM + static_cast<int>(rank) * BM_CTA + row_in_cta;
        const bool active = !w.half || half == 0;
        const int n0 = w.half ? w.nb * BN + w.j * NC : w.nb * BN + half * NC;
        st.row0 = m - lane;
        uint32_t sum[NC];
#pragma unroll
        for (int i = 0; i < NC; ++i) sum[i] = 0u;
        for (int ch = 0; ch < n_chunks; ++ch) {
          if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, lim, abort_flag,
                                                  p.status, kSiteEpiFull)))
            goto epi_done;
          tc_fence_after();
          if (active)
            tmem_drain_x32<NC>(lane_base + static_cast<uint32_t>(acc) * Cfg::kAccStride, sum, ch == 0);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(tempty_lead + static_cast<uint32_t>(acc) * 8u);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
        // the unit's sums: rA' of this row (own CTA), cB' of this warp's columns
        // (whole unit: CTA `half` holds them; column half: CTA col / (BN / 4))
        if (!__all_sync(0xffffffffu, mbar_wait<true>(&sfull[ub], sph, lim, abort_flag, p.status,
                                                      kSiteSumsFull)))
          goto epi_done;
        {
          const uint32_t base = sums_own + static_cast<uint32_t>(ub * (BM_CTA + Cfg::kBRows)) * 4u;
          uint32_t rs;
          asm volatile("ld.shared.u32 %0, [%1];"
                       : "=r"(rs)
                       : "r"(base + static_cast<uint32_t>(row_in_cta) * 4u)
                       : "memory");
          ColVecs<NC> V;
          load_col_vec(p.zB_col, n0, p.N, lane, V.zB);
          load_col_vec(p.scale_col, n0, p.N, lane, V.sc);
          if constexpr (kDequant) {
            load_col_vec(p.dq_col, n0, p.N, lane, V.dq);
            load_col_vec(p.bias, n0, p.N, lane, V.bi);
          } else {
#pragma unroll
            for (int b = 0; b < ColVecs<NC>::kB; ++b) V.dq[b] = V.bi[b] = 0u;
          }
#pragma unroll
          for (int b = 0; b < ColVecs<NC>::kB; ++b) {
            const int col = 32 * b + lane;
            const uint32_t cta = w.half ? static_cast<uint32_t>(col / (BN / 4))
                                        : static_cast<uint32_t>(half);
            const int idx = w.half ? col % (BN / 4) : col;
            V.cB[b] = ld_shared_cluster_u32(
                mapa_shared(base + static_cast<uint32_t>(BM_CTA + idx) * 4u, cta));
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive_cluster(sempty_own + static_cast<uint32_t>(ub) * 8u);
            mbar_arrive_cluster(sempty_peer + static_cast<uint32_t>(ub) * 8u);
          }
          ub ^= 1;
          if (ub == 0) sph ^= 1u;
          if (active)
            store_row_int_v<NC, kDequant>(p, tmO0, tmO1, tmO2, st, m, n0, sum,
                                          int_row_from(p, m, rs), V);
        }
      }
    epi_done:
      if (lane == 0) bulk_wait_group0();
      __syncwarp();
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_2cta(tmem_base, Cfg::kTmemCols);
  }
}

}  // namespace igc
