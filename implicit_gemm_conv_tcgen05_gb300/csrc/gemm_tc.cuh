// Persistent, warp-specialised tcgen05 GEMM for sm_103a, 2-CTA (cta_group::2) tiles.
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
//             requantisation (or dequantisation + bias) fused into the epilogue
//             (page "TVM在CUDA GPU上跑GEMM的全套张量化实现", §2.3).
//   GemmBF16: GemmF16 with bf16 operands (the same kind::f16 pipe, §3.3's
//             "f16 -> bf16" swap).
//   ConvInt : ConvF16's gather with GemmInt's arithmetic (int8 convolution over
//             a zero-point-padded, shifted input).
//
// A cluster of two CTAs (on two SMs) computes one 256 x BN output tile with
// tcgen05.mma.cta_group::2 (M = 256): CTA r holds rows [128 r, 128 r + 128) of
// the A tile and rows [BN/2 r, BN/2 (r+1)) of the B tile in its own shared
// memory, and receives its 128 x BN accumulator in its own tensor memory.
// Warp roles in each CTA (384 threads, three warpgroups):
//   warp 0      TMA producer: its CTA's halves of A and B into a ring of
//               128-deep stages (two 128-byte swizzle atoms per operand; 64-deep
//               stages, twice as many, for GEMMs of one or two rounds); both
//               CTAs' copies complete on the leader CTA's `full[s]` barrier.
//   warp 1      tensor-memory owner; in the leader CTA also the MMA issuer: 8 x
//               tcgen05.mma per stage (4 when 64-deep), tcgen05.commit multicast
//               to both CTAs frees
//               ring stages (`empty[s]`) and hands finished accumulators to both
//               epilogues (`tfull[a]`).  Warps 0 and 1 run their loops converged;
//               lane 0 issues.
//   warps 2-3   GEMMs: L2 prefetch of the first rounds' operand panels, paced by
//               the producer (convolutions: idle); their warpgroup gives registers
//               to the epilogue.
//   warps 4-11  epilogue: tcgen05.ld of their lane quadrant / column half, fused
//               output math, outputs staged in 128-byte-swizzled shared memory and
//               written by TMA bulk tensor stores (direct stores for outputs TMA
//               cannot address); they release an accumulator on the leader's
//               `tempty[a]` (16 arrivals).
// Two accumulators (2 x BN of the 512 TMEM columns) let the epilogue of one
// tile overlap the main loop of the next.  The persistent schedule walks tiles
// in groups of 8 m-tiles; when its last round would fill at most half of the
// CTA pairs, that round's tiles run as two BN/2-wide column halves (at BN = 256
// on a four-stage ring laid over the three main stages, tail_slot).
//
// The integer modes accumulate in chunks that fp32 holds exactly: products of
// the shifted operands are integers of magnitude <= 2^14, so every partial sum
// of a 1024-k chunk is an integer of magnitude <= 2^24.  Each chunk is drained
// into the int32 running sums by a float-to-int conversion toward zero, exact
// for integral values; a chunk's MMAs (about 5 us) let the main loop run ahead
// while the epilogue finishes the previous unit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "int8_widen.cuh"
#include "sm100_ptx.cuh"

namespace igc {

// GemmIntCv: the integer GEMM that converts its own operands (KParams::cv_*), a
// separate instantiation so that the default integer GEMM carries none of its code.
enum class Mode : int {
  GemmF16 = 0,
  ConvF16 = 1,
  GemmInt = 2,
  GemmBF16 = 3,
  ConvInt = 4,
  GemmIntCv = 5
};

// A operand gathered by TMA im2col (a convolution) / integer epilogue
__host__ __device__ constexpr bool mode_is_conv(Mode m) { return m == Mode::ConvF16 || m == Mode::ConvInt; }
__host__ __device__ constexpr bool mode_is_int(Mode m) {
  return m == Mode::GemmInt || m == Mode::ConvInt || m == Mode::GemmIntCv;
}

// element type of the floating output
enum : int { kOutF32 = 0, kOutF16 = 1, kOutBF16 = 2 };

constexpr int BM = 256;        // rows per cluster tile (128 per CTA)
constexpr int BM_CTA = 128;
constexpr int BK = 64;         // 64 fp16 = one 128-byte swizzle row (one TMA box, one atom)
constexpr int kAtoms = 2;      // swizzle atoms along k per pipeline stage (default)
constexpr int KS = BK * kAtoms;  // k depth of one default pipeline stage (8 MMAs of k = 16)
constexpr int kEpiWarps = 8;
// Three warpgroups: warps 0-3 (TMA producer, MMA issuer / TMEM owner, two prefetch)
// and two epilogue warpgroups (warps 4-11).  After set-up the first warpgroup
// gives registers to the epilogue ones (setmaxnreg): kRegsLow + 2 kRegsHigh
// warpgroup shares = 72 * 128 + 216 * 256 = 64512 registers, exactly the
// launch's 384 threads x kMinLaunchRegs (checked on the host before launch).
constexpr int kThreads = 128 + 32 * kEpiWarps;  // 384
constexpr int kRegsLow = 72;
constexpr int kRegsHigh = 216;
constexpr int kMinLaunchRegs = 168;
static_assert(kRegsLow * 128 + kRegsHigh * 256 <= kThreads * kMinLaunchRegs, "register split");
// setmaxnreg.dec only lowers and setmaxnreg.inc only raises a warpgroup's count
static_assert(kRegsLow <= kMinLaunchRegs && kRegsHigh >= kMinLaunchRegs, "register split direction");
constexpr uint32_t kAtomABytes = BM_CTA * BK * 2;   // 16 KB
// barriers and small shared state (512 bytes), then the band table of an integer
// GEMM converting its own operands (kCvBandTab int2 entries)
constexpr uint32_t kBarrierBytes = 1536;
// Each epilogue warp stages 32 rows x 128 bytes of output in shared memory (128-byte
// swizzle, the layout of a TMA box) and writes them with one bulk tensor store.
constexpr uint32_t kStagingWarpBytes = 32 * 128;
constexpr uint32_t kStagingBytes = kEpiWarps * kStagingWarpBytes;
constexpr size_t kSmemBudget = 227 * 1024;
constexpr int kIntChunkKb = 1024 / KS;  // stages per exact fp32 accumulation chunk (1024 k)

// ATOMS: swizzle atoms along k per pipeline stage.  The default, 2 (128-deep
// stages, 8 MMAs each), has the least per-stage overhead; 1 (64-deep stages,
// about twice as many) keeps more of the ring in flight, which pays for shapes
// that run one or two rounds and stream their operands from DRAM.
template <int BN, int ATOMS = kAtoms>
struct TileCfg {
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(ATOMS == 1 || ATOMS == 2, "ATOMS");
  static constexpr int kKS = BK * ATOMS;                        // k depth of a stage
  static constexpr uint32_t kStageABytes = kAtomABytes * ATOMS;
  static constexpr int kBNHalf = BN / 2;                        // B rows per CTA
  static constexpr uint32_t kAtomBBytes = kBNHalf * BK * 2;
  static constexpr uint32_t kStageBBytes = kAtomBBytes * ATOMS;
  static constexpr uint32_t kStageBytes = kStageABytes + kStageBBytes;
  static constexpr int kStages =
      static_cast<int>((kSmemBudget - 1024 - kBarrierBytes - kStagingBytes) / kStageBytes) > 8
          ? 8
          : static_cast<int>((kSmemBudget - 1024 - kBarrierBytes - kStagingBytes) / kStageBytes);
  static constexpr size_t kSmemBytes =
      1024 + kStages * kStageBytes + kStagingBytes + kBarrierBytes;
  static constexpr uint32_t kTmemCols = 2 * BN <= 256 ? 256 : 512;  // power of two >= 2*BN
  // column of accumulator 1 (a multiple of 32, so every tcgen05.ld starts aligned)
  static constexpr uint32_t kAccStride = kTmemCols / 2;
  static constexpr int kEpiCols = BN / 2;  // columns per epilogue warp
  // Column-half units take A 32 KB + B 16 KB per stage and use them up in half the
  // MMA time of a whole tile's stage, so with three stages the copies in flight
  // cover half the time.  At BN = 256 the last round therefore switches to a ring
  // of four such 48 KB stages laid over the memory of the three 64 KB ones
  // (tail_slot); slot i is filled only once the main stages whose memory it
  // reuses have been released.
  static constexpr bool kTailRing = BN == 256 && kStages == 3;
  static constexpr int kTailStages = 4;
  static_assert(!kTailRing || (kStageABytes == 32768 && kStageBBytes == 32768), "tail ring");
};

// wait sites, reported in the device status word
enum : uint32_t {
  kSiteProducerEmpty = 1,
  kSiteMmaTmemEmpty = 2,
  kSiteMmaFull = 3,
  kSiteEpiFull = 4,
  kSiteDrain = 5,
  kSiteTmemMismatch = 6,
  kSiteCvFlag = 7,
};

// Tail-ring slot `i` (BN = 256) after the switch from the main ring, whose stages
// lie at A: 32K s and B: 96K + 32K s and whose oldest stage (the first the MMAs
// release) is m0; m1, m2 follow in release order.  Byte offsets of the slot's A
// (32 KB) and B (16 KB) parts:
//   slot 0: A(m0), B(m0) low half     slot 1: A(m1), B(m0) high half
//   slot 2: B(m1), B(m2) low half     slot 3: A(m2), B(m2) high half
// Slot i's first fill therefore needs main stages m0..m_min(i,2) released, in order.
__host__ __device__ constexpr void tail_slot(int i, int m0, uint32_t& a_off, uint32_t& b_off) {
  constexpr uint32_t kS = 32768u, kB0 = 3u * 32768u, kHalfB = 16384u;
  const uint32_t m1 = m0 == 2 ? 0u : static_cast<uint32_t>(m0) + 1u;
  const uint32_t m2 = m1 == 2u ? 0u : m1 + 1u;
  const uint32_t s0 = static_cast<uint32_t>(m0);
  if (i == 0) {
    a_off = s0 * kS;
    b_off = kB0 + s0 * kS;
  } else if (i == 1) {
    a_off = m1 * kS;
    b_off = kB0 + s0 * kS + kHalfB;
  } else if (i == 2) {
    a_off = kB0 + m1 * kS;
    b_off = kB0 + m2 * kS;
  } else {
    a_off = m2 * kS;
    b_off = kB0 + m2 * kS + kHalfB;
  }
}

// Compile-time check of the tail-ring map for every oldest main stage m0: the four
// slots' A (32 KB) and B (16 KB) parts are 1024-byte aligned, disjoint, cover the
// three main stages' 192 KB exactly, and slot i overlaps only main stages released
// no later than m_min(i,2), the ones its first fill waits for.
constexpr bool tail_ring_map_ok() {
  constexpr uint32_t kS = 32768u, kB0 = 3u * 32768u;
  for (int m0 = 0; m0 < 3; ++m0) {
    uint32_t lo[8] = {}, hi[8] = {};
    uint32_t total = 0;
    for (int i = 0; i < 4; ++i) {
      uint32_t a = 0, b = 0;
      tail_slot(i, m0, a, b);
      lo[2 * i] = a;
      hi[2 * i] = a + kS;
      lo[2 * i + 1] = b;
      hi[2 * i + 1] = b + kS / 2;
      total += kS + kS / 2;
      for (int part = 0; part < 2; ++part) {
        const uint32_t l = lo[2 * i + part], h = hi[2 * i + part];
        if (l % 1024u != 0 || h > 6u * kS) return false;
        // main stages this part overlaps must be among m0 .. m_min(i,2)
        for (int ms = 0; ms < 3; ++ms) {
          const uint32_t la = ms * kS, ha = la + kS, lb = kB0 + ms * kS, hb = lb + kS;
          const bool overlaps = (l < ha && la < h) || (l < hb && lb < h);
          const int order = (ms - m0 + 3) % 3;  // release order of main stage ms
          if (overlaps && order > (i < 2 ? i : 2)) return false;
        }
      }
    }
    for (int x = 0; x < 8; ++x)
      for (int y = x + 1; y < 8; ++y)
        if (lo[x] < hi[y] && lo[y] < hi[x]) return false;
    if (total != 6u * kS) return false;
  }
  return true;
}
static_assert(tail_ring_map_ok(), "tail ring map");

// Leader CTA, after an abort: waits (briefly) for the last fills of a ring whose
// next fill would be `stage` in `phase`, so that no copy is still landing when the
// CTA exits.
__device__ __forceinline__ void drain_fills(uint64_t* full_arr, int n, int stage, uint32_t phase,
                                            long long issued, uint64_t lim) {
  int s = stage;
  uint32_t ph = phase;
  for (long long i = 0; i < issued && i < n; ++i) {
    if (--s < 0) {
      s = n - 1;
      ph ^= 1u;
    }
    int dummy = 0;
    mbar_wait(&full_arr[s], ph, lim / 64 + 1000, &dummy, nullptr, kSiteDrain);
  }
}

struct KParams {
  int M, N, K;
  int num_kb;
  int tiles_m, tiles_n, num_tiles;
  int group_m;
  // persistent schedule: tiles before tail_start are whole work units; every
  // tile from tail_start on is split into two column halves (num_units in all)
  int tail_start, num_units;
  int chunk_kb;  // k-blocks per accumulation chunk (an accumulator hand-off after each)
  int conv_P, conv_Q, conv_cblocks, conv_S, conv_C;
  int pad_h, pad_w, stride_h, stride_w;
  // integer convolution: when px is set, the row sums of the implicit im2col
  // matrix are the sums of px (per padded pixel, conv_Hp x conv_Wp per image)
  // over each output pixel's conv_R x conv_S window, taken in the epilogue
  const int32_t* px;
  int conv_R, conv_Hp, conv_Wp;
  void* out;
  long long ldo;
  int out_type;  // kOutF32 / kOutF16 / kOutBF16
  float* out_f32;
  long long ldo32;
  int vec_ok;
  int32_t* c32;
  long long ldc32;
  int8_t* c8;
  long long ldc8;
  const int32_t* rsumA;
  const int32_t* csumB;
  int32_t zA;
  const int32_t* zA_row;
  int32_t zB;
  const int32_t* zB_col;
  int32_t oA, oB;
  float scale;
  const float* scale_col;
  // bit i set: output i is written by TMA stores through tensor map tmO<i>
  // (float modes: 0 = out, 1 = out_f32; integer modes: 0 = c32, 1 = c8, 2 = yf)
  int tma_out;
  // dequantised float output of the int8 path: y = ((fp32(C32) * dq_row_i) * dq_col_j) + bias_j
  float* yf;
  long long ldyf;
  const float* dq_row;
  const float* dq_col;
  const float* bias;
  unsigned long long wait_limit_ns;
  unsigned long long* status;
  // GEMMs: the operands' rows (row strides in bytes, k extent in bytes) for the L2
  // prefetch of the first pf_units work units of each CTA pair (0: none)
  const char* pf_a;
  const char* pf_b;
  long long pf_lda, pf_ldb;
  int pf_kbytes;
  int pf_units;
  // Integer GEMM that converts its own operands (cv_flags != nullptr; see cv_step):
  // the raw uint8 / int8 operands A and Bt, their conversion into the fp16 operands
  // that the copies read (row stride cv_Kp), the sums of their rows (accumulated
  // chunk by chunk), one flag per 128-row block and 1024-k chunk and one per block
  // (each counting the finished jobs; A's blocks first) and the job counter of the
  // queue, all zero at launch.  rsumA / csumB are unused then.
  const uint8_t* cv_a;
  const uint8_t* cv_b;
  long long cv_lda, cv_ldb;
  uint32_t cv_flip_a, cv_flip_b;  // 0 for uint8, 0x80808080 for int8
  __half* cv_da;
  __half* cv_db;
  int32_t* cv_sa;
  int32_t* cv_sb;
  int* cv_flags;
  int* cv_done;
  int* cv_queue;
  int cv_blocks_a, cv_blocks_b, cv_chunks, cv_Kp;
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

// Work unit u: a whole BM x BN tile, or (u past tail_start) one BM x BN/2 column
// half j of a tile.  The halves fill the schedule's last round with twice as
// many units of half the length.
struct Unit {
  int mb, nb;
  int j;      // column half (0 for a whole tile)
  bool half;  // the unit covers BN/2 columns starting at nb*BN + j*BN/2
};

__device__ __forceinline__ Unit unit_coords(const KParams& p, int u) {
  Unit w;
  int t = u;
  w.j = 0;
  w.half = false;
  if (u >= p.tail_start) {
    const int v = u - p.tail_start;
    t = p.tail_start + (v >> 1);
    w.j = v & 1;
    w.half = true;
  }
  tile_coords(p, t, w.mb, w.nb);
  return w;
}

// First B row (output column) this CTA loads for unit w: each CTA holds half of
// the unit's B rows at the start of its stage buffer; a half unit's BN/4 rows
// come through tmBh, whose box is BN/4 rows.
template <int BN>
__device__ __forceinline__ int b_row0(const Unit& w, uint32_t rank) {
  return w.half ? w.nb * BN + w.j * (BN / 2) + static_cast<int>(rank) * (BN / 4)
                : w.nb * BN + static_cast<int>(rank) * (BN / 2);
}

// The CTA's first unit u, worked out by one thread during the set-up (integer
// divisions, first parameter reads) instead of in front of the producer's first
// copies, and left in first_unit[0..3] (shared memory).
__device__ __forceinline__ void store_first_unit(const KParams& p, int u, int* first_unit) {
  const Unit w = unit_coords(p, u);
  first_unit[0] = w.mb;
  first_unit[1] = w.nb;
  first_unit[2] = w.j;
  first_unit[3] = w.half ? 1 : 0;
}

__device__ __forceinline__ Unit load_first_unit(const int* first_unit) {
  Unit w;
  w.mb = first_unit[0];
  w.nb = first_unit[1];
  w.j = first_unit[2];
  w.half = first_unit[3] != 0;
  return w;
}

// L2 prefetch (TMA boxes) of the first n_stages pipeline stages of the CTA's
// first unit (store_first_unit), by one thread during the set-up, so that the
// first copies after it find their tiles in L2 instead of DRAM.  A prefetch
// makes nothing visible to the kernel, so it may run before the grid dependency
// wait: L2 stays coherent with the previous kernel's writes.  Not inlined: it
// runs once, and kept out of the kernel body its values stay out of the
// producer's register budget.
template <int BN, int ATOMS>
__device__ __noinline__ void prefetch_first_stages(const KParams& p, const CUtensorMap* tmA,
                                                   const CUtensorMap* tmB,
                                                   const CUtensorMap* tmBh,
                                                   const int* first_unit, uint32_t rank,
                                                   int n_stages) {
  const Unit w = load_first_unit(first_unit);
  const int m_cta = w.mb * BM + static_cast<int>(rank) * BM_CTA;
  const int n_cta = b_row0<BN>(w, rank);
  const CUtensorMap* mapB = w.half ? tmBh : tmB;
  const int atoms = (p.num_kb < n_stages ? p.num_kb : n_stages) * ATOMS;
  for (int j = 0; j < atoms; ++j) {
    tma_prefetch_2d(tmA, j * BK, m_cta);
    tma_prefetch_2d(mapB, j * BK, n_cta);
  }
}

// ---------------------------------------------------------------------------
// Integer GEMM converting its own operands (Mode::GemmIntCv, p.cv_flags set)
//
// The raw uint8 / int8 operands are shifted and widened to fp16 once, in jobs of
// 8 rows x one 1024-k chunk done by the CTAs' spare warps: warps 2-3 throughout,
// the epilogue warps while they wait for an accumulator (between polls of its
// barrier, one job at a time; see epi_int_unit).  A job writes the fp16 values
// where the copies read them and adds each row's chunk sum to the row's sum, then
// adds one to the flag of its 128-row block and chunk; the producer waits for a
// block's flag before copying that block's chunk.  Jobs come in bands: band b
// holds the blocks that the schedule's tiles b*C .. (b+1)*C - 1 (C CTA pairs: one
// round of the persistent schedule) use first, chunk after chunk, so the first
// round's blocks are ready first, and every block is converted once.  The first
// band is shared out statically over the converting warps; the later bands come
// from one queue, at most one round ahead of the taking CTA's producer.  No job
// waits on anything, so the flags always complete.
// ---------------------------------------------------------------------------
constexpr int kCvRows = 8;                                   // rows of one job
constexpr int kCvBlockRows = 128;                            // rows under one flag
constexpr int kCvJobsPerFlag = kCvBlockRows / kCvRows;       // 16
constexpr int kCvChunk = 1024;                               // k under one flag
constexpr int kCvBandTab = 128;  // bands whose first blocks are tabulated in shared memory
static_assert(kIntChunkKb * KS == kCvChunk, "a flag's chunk is one accumulation chunk");

// m-tiles / n-tiles of the raster (tile_coords) whose first tile comes before
// tile U: a group's m-tiles appear in its first gm tiles, the n-tiles in the
// first group, one every gm tiles.
__device__ __forceinline__ int cv_mtiles_before(const KParams& p, int U) {
  const int per_group = p.group_m * p.tiles_n;
  const int full = U / per_group;
  const int first_m = full * p.group_m;
  if (first_m >= p.tiles_m) return p.tiles_m;
  const int gm = min(p.tiles_m - first_m, p.group_m);
  return first_m + min(U - full * per_group, gm);
}

__device__ __forceinline__ int cv_ntiles_before(const KParams& p, int U) {
  const int gm0 = min(p.tiles_m, p.group_m);
  return min((U + gm0 - 1) / gm0, p.tiles_n);
}

// Bands of the schedule: one per round of C CTA pairs.
__device__ __forceinline__ int cv_num_bands(const KParams& p, int C) {
  return (p.num_tiles + C - 1) / C;
}

// Blocks that band b and the bands before it hold: A [0, a), B [0, b) of the
// returned pair, from the first tile of band b on.
template <int BN>
__device__ __forceinline__ int2 cv_blocks_before(const KParams& p, int band, int C) {
  constexpr int kBnb = BN / kCvBlockRows;  // B blocks per n-tile
  const long long t = static_cast<long long>(band) * C;
  const int u = static_cast<int>(t < p.num_tiles ? t : p.num_tiles);
  return make_int2(min(2 * cv_mtiles_before(p, u), p.cv_blocks_a),
                   min(kBnb * cv_ntiles_before(p, u), p.cv_blocks_b));
}

// One job: rows r0 .. r0+7 of operand A (opB false) or Bt, chunk c.  Lane l takes
// the 16 bytes at 16 l and at 512 + 16 l of each row's chunk; kRowsInFlight rows'
// loads are in flight at a time (fewer for the warps with fewer registers).  Each
// row's chunk sum of the shifted values is added to its row sum.  Every lane must
// call it (the sums are reduced by shuffles).
template <int kRowsInFlight>
__device__ __forceinline__ void cv_job(const KParams& p, bool opB, int r0, int c, int lane) {
  const uint8_t* src = opB ? p.cv_b : p.cv_a;
  const long long ld = opB ? p.cv_ldb : p.cv_lda;
  const uint32_t flip = opB ? p.cv_flip_b : p.cv_flip_a;
  __half* dst = opB ? p.cv_db : p.cv_da;
  int32_t* sums = opB ? p.cv_sb : p.cv_sa;
  const int rows = opB ? p.N : p.M;
  const int k0 = c * kCvChunk;
  const int kb = min(kCvChunk, p.K - k0);  // bytes of this chunk (a multiple of 16)
#pragma unroll 1
  for (int i0 = 0; i0 < kCvRows; i0 += kRowsInFlight) {
    uint4 raw[kRowsInFlight][2];
#pragma unroll
    for (int i = 0; i < kRowsInFlight; ++i) {
      const int row = r0 + i0 + i;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int k = j * 512 + lane * 16;
        raw[i][j] = (row < rows && k < kb)
                        ? __ldcs(reinterpret_cast<const uint4*>(
                              src + static_cast<long long>(row) * ld + k0 + k))
                        : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int i = 0; i < kRowsInFlight; ++i) {
      const int row = r0 + i0 + i;
      uint32_t usum = 0;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int k = j * 512 + lane * 16;
        if (row < rows && k < kb) {
          uint32_t o[8];
          prepass::widen4(raw[i][j].x, flip, o[0], o[1], usum);
          prepass::widen4(raw[i][j].y, flip, o[2], o[3], usum);
          prepass::widen4(raw[i][j].z, flip, o[4], o[5], usum);
          prepass::widen4(raw[i][j].w, flip, o[6], o[7], usum);
          uint4* d =
              reinterpret_cast<uint4*>(dst + static_cast<long long>(row) * p.cv_Kp + k0 + k);
          __stcs(d, make_uint4(o[0], o[1], o[2], o[3]));
          __stcs(d + 1, make_uint4(o[4], o[5], o[6], o[7]));
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) usum += __shfl_xor_sync(0xffffffffu, usum, off);
      // the shifted sum: each byte read contributed u = value + 128
      if (lane == 0 && row < rows)
        atomicAdd(sums + row, static_cast<int32_t>(usum - 128u * static_cast<uint32_t>(kb)));
    }
  }
}

// The band that job s belongs to: the last band whose first job is at or before
// s (s below the total), found by bisection over the bands' first jobs.
// (tab: the blocks before bands 0 .. nb, worked out once per CTA, when nb < kCvBandTab)
template <int BN>
__device__ __forceinline__ int2 cv_blocks_before_t(const KParams& p, const int2* tab, int band,
                                                   int nb, int C) {
  return nb < kCvBandTab ? tab[band] : cv_blocks_before<BN>(p, band, C);
}

template <int BN>
__device__ __forceinline__ int cv_band_of(const KParams& p, const int2* tab, int s, int nb, int C,
                                          int jobs_per_block) {
  int lo = 0, hi = nb - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const int2 bb = cv_blocks_before_t<BN>(p, tab, mid, nb, C);
    if ((bb.x + bb.y) * jobs_per_block <= s)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

enum : int { kCvNone = 0, kCvDid = 1, kCvLater = 2 };

// Does job s (the s-th of all bands, in band order, chunk-major within a band)
// and publishes it: every lane orders its stores before the copy engine's later
// reads, and lane 0 adds one to the job's chunk flag and block count (release).
// Every lane must call it.
template <int BN, int kRowsInFlight>
__device__ __forceinline__ void cv_do_job(const KParams& p, const int2* tab, int s, int nb, int C,
                                          int lane) {
  const int jobs_per_block = p.cv_chunks * kCvJobsPerFlag;
  const int band = cv_band_of<BN>(p, tab, s, nb, C, jobs_per_block);
  const int2 b0 = cv_blocks_before_t<BN>(p, tab, band, nb, C);
  const int2 b1 = cv_blocks_before_t<BN>(p, tab, band + 1, nb, C);
  const int na = b1.x - b0.x;
  const int per_chunk = (na + (b1.y - b0.y)) * kCvJobsPerFlag;
  const int r = s - (b0.x + b0.y) * jobs_per_block;
  const int c = r / per_chunk;
  const int rem = r - c * per_chunk;
  const int blk = rem / kCvJobsPerFlag;
  const int jr = rem - blk * kCvJobsPerFlag;
  const bool opB = blk >= na;
  const int block = opB ? b0.y + (blk - na) : b0.x + blk;
  cv_job<kRowsInFlight>(p, opB, block * kCvBlockRows + jr * kCvRows, c, lane);
  fence_proxy_async_global();
  __syncwarp();
  if (lane == 0) {
    const int gb = opB ? p.cv_blocks_a + block : block;
    red_release_gpu_add(p.cv_flags + gb * p.cv_chunks + c, 1);
    red_release_gpu_add(p.cv_done + gb, 1);
  }
}

// Jobs of the first band (the first round's blocks), which are needed at once:
// shared out statically, job j to converting warp j mod W (W = 10 per CTA, the
// epilogue warps' numbers first and spread over the CTAs), so the start takes no
// turns on a shared counter.
__device__ __forceinline__ int cv_first_band_jobs(const int2* tab) {
  return (tab[1].x + tab[1].y);  // blocks of band 0 (tab[0] is zero)
}

__device__ __forceinline__ int cv_static_worker(int warp) {
  // epilogue warps 4..11 -> 0..7, warps 2-3 -> 8-9, times the CTAs
  const int local = warp >= 4 ? warp - 4 : warp + 6;
  return local * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
}

// Takes the next job from the queue of the later bands and does it (kCvDid), unless
// no job is left (kCvNone) or the next job belongs to a band past max_band
// (kCvLater: blocks the schedule needs more than a round ahead of this CTA's
// producer are left for later, so that converted blocks do not crowd the working
// set out of L2 and the conversion traffic spreads over the run).  Every lane must
// call it.
template <int BN, int kRowsInFlight>
__device__ __forceinline__ int cv_step(const KParams& p, const int2* tab, int C, int max_band,
                                       int lane) {
  const int nb = cv_num_bands(p, C);
  const int jobs_per_block = p.cv_chunks * kCvJobsPerFlag;
  const int total = (p.cv_blocks_a + p.cv_blocks_b) * jobs_per_block;
  const int first = cv_first_band_jobs(tab) * jobs_per_block;
  int s = 0;
  if (lane == 0) {
    const int next = first + ld_relaxed_gpu(p.cv_queue);
    if (next >= total)
      s = -1;
    else if (max_band < nb - 1 && cv_band_of<BN>(p, tab, next, nb, C, jobs_per_block) > max_band)
      s = -2;
    else
      s = first + atomicAdd(p.cv_queue, 1);
  }
  s = __shfl_sync(0xffffffffu, s, 0);
  if (s == -2) return kCvLater;
  if (s < 0 || s >= total) return kCvNone;
  cv_do_job<BN, kRowsInFlight>(p, tab, s, nb, C, lane);
  return kCvDid;
}

// The next of this warp's first-band jobs (advancing *next by W); false when its
// share is done.  Every lane must call it.
template <int BN, int kRowsInFlight>
__device__ __forceinline__ bool cv_static_step(const KParams& p, const int2* tab, int C, int& next,
                                               int lane) {
  const int jobs_per_block = p.cv_chunks * kCvJobsPerFlag;
  if (next >= cv_first_band_jobs(tab) * jobs_per_block) return false;
  cv_do_job<BN, kRowsInFlight>(p, tab, next, cv_num_bands(p, C), C, lane);
  next += 10 * static_cast<int>(gridDim.x);
  return true;
}

// The band a CTA's converters may reach: one round past the unit its producer
// is copying (its main ring publishes the stages issued in *progress).
__device__ __forceinline__ int cv_max_band(const KParams& p, const volatile int* progress) {
  return *progress / p.num_kb + 1;
}

// The producer's wait (lane 0) until the conversion of flag `flag` is complete,
// after which its copies are ordered after the converters' stores.  Every lane
// must call it; false if the wait gave up (bounded like every other wait).
__device__ __forceinline__ bool cv_wait(const KParams& p, int flag, uint64_t limit_ns,
                                        volatile int* abort, int lane) {
  int ok = 1;
  if (lane == 0) {
    const int* f = p.cv_flags + flag;
    if (ld_acquire_gpu(f) < kCvJobsPerFlag) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(f) < kCvJobsPerFlag) {
        if (*abort) {
          ok = 0;
          break;
        }
        if (globaltimer_ns() - t0 > limit_ns) {
          *abort = 1;
          report_status(p.status, kStatusTimeout, kSiteCvFlag);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    fence_proxy_async_global();
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// The producer's waits before the first copy of chunk c of a unit: the CTA's A
// block (rows m_cta ..) and B block (rows n_cta ..), where they lie inside the
// operands (rows outside are zero-filled by the copy, nothing to wait for).
__device__ __forceinline__ bool cv_wait_chunk(const KParams& p, int m_cta, int n_cta, int c,
                                              uint64_t limit_ns, volatile int* abort, int lane) {
  if (m_cta < p.M &&
      !cv_wait(p, (m_cta / kCvBlockRows) * p.cv_chunks + c, limit_ns, abort, lane))
    return false;
  if (n_cta < p.N &&
      !cv_wait(p, (p.cv_blocks_a + n_cta / kCvBlockRows) * p.cv_chunks + c, limit_ns, abort, lane))
    return false;
  return true;
}

// True when every job of the CTA's A and B blocks for this unit is done (the
// blocks' job counts, read relaxed, made an acquire by a fence): then the unit's
// copies need no per-chunk waits.  One round trip at the unit's start instead of
// two acquire loads before every chunk.  Every lane must call it.
__device__ __forceinline__ bool cv_unit_ready(const KParams& p, int m_cta, int n_cta, int lane) {
  int ready = 0;
  if (lane == 0) {
    const int full = p.cv_chunks * kCvJobsPerFlag;
    const int a = m_cta < p.M ? ld_relaxed_gpu(p.cv_done + m_cta / kCvBlockRows) : full;
    const int b =
        n_cta < p.N ? ld_relaxed_gpu(p.cv_done + p.cv_blocks_a + n_cta / kCvBlockRows) : full;
    if (a >= full && b >= full) {
      fence_acq_rel_gpu();
      fence_proxy_async_global();
      ready = 1;
    }
  }
  return __shfl_sync(0xffffffffu, ready, 0) != 0;
}

// Sum over k of the shifted row `row` of A (opB false) or Bt, read after
// cv_acquire_sums (so not through the read-only cache).
__device__ __forceinline__ uint32_t cv_sum(const KParams& p, bool opB, int row) {
  return static_cast<uint32_t>(__ldcg((opB ? p.cv_sb : p.cv_sa) + row));
}

// Before the epilogue of a unit reads its row and column sums: the job counts of
// the blocks that hold them, read relaxed (all at once) and made an acquire by one
// fence.  Every job of those blocks is complete by then (the unit's copies waited
// for them), each having added its sums before its release.
template <int NB>
__device__ __forceinline__ void cv_acquire_sums(const KParams& p, int m, int n0, int lane) {
  int seen = ld_relaxed_gpu(p.cv_done + (m < p.M ? m : p.M - 1) / kCvBlockRows);
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const int n = n0 + 32 * b + lane;
    seen += ld_relaxed_gpu(p.cv_done + p.cv_blocks_a + (n < p.N ? n : p.N - 1) / kCvBlockRows);
  }
  asm volatile("" ::"r"(seen));
  fence_acq_rel_gpu();
}

// ---------------------------------------------------------------------------
// L2 prefetch of k bytes [k0, k0 + kb) of `nrows` operand rows from row0 (rows
// past rows_total and bytes past kbytes skipped), by the 64 threads t = 0..63
// of warps 2-3, one 128-byte line each.
__device__ __forceinline__ void prefetch_rows(const char* base, long long ld, int row0, int nrows,
                                              int rows_total, int k0, int kb, int kbytes, int t) {
  const int lines = kb / 128;
  for (int i = t; i < nrows * lines; i += 64) {
    const int r = i / lines;
    const int kc = k0 + (i - r * lines) * 128;
    const int row = row0 + r;
    if (row < rows_total && kc < kbytes)
      prefetch_l2(base + static_cast<long long>(row) * ld + kc);
  }
}

// Warps 2-3 of a GEMM: L2 prefetch of the A and B rows of this CTA's first
// p.pf_units work units (whole tiles), kPrefetchAhead stages ahead of the
// producer's copies, which it publishes in *progress (stages issued).  The first
// rounds of a schedule take all their panels from DRAM in lockstep, and three
// ring stages do not cover DRAM latency; lines requested this far ahead are in
// L2 when the copies ask for them.  A panel is prefetched only by the unit that
// first uses it in its round (the one with the same m-tile one group column back,
// or the previous tile with the same n-tile, is in the round already otherwise),
// so each line is requested about once.  The waits are bounded and give up
// silently: a prefetch is only a hint.
template <int BN, int kStageKBytes>
__device__ __forceinline__ void prefetch_first_units(const KParams& p, int cluster, int num_clusters,
                                                     uint32_t rank, int t,
                                                     const volatile int* progress,
                                                     const volatile int* abort) {
  constexpr int kPrefetchAhead = 6;
  const uint64_t t0 = globaltimer_ns();
  for (int i = 0; i < p.pf_units; ++i) {
    const int u = cluster + i * num_clusters;
    if (u >= p.tail_start) return;  // whole tiles only
    int mb, nb;
    tile_coords(p, u, mb, nb);
    const int per_group = p.group_m * p.tiles_n;
    const int g = u / per_group;
    const int gstart = g * per_group;
    const int gm = min(p.tiles_m - g * p.group_m, p.group_m);
    const int lo = max(u - cluster, gstart);  // first unit of this round within the group
    const bool first_a = u - gm < lo;
    const bool first_b = u - 1 < max(lo, gstart + nb * gm);
    if (!first_a && !first_b) continue;
    for (int kb = 0; kb < p.num_kb; ++kb) {
      const int need = i * p.num_kb + kb - kPrefetchAhead;  // producer stages issued first
      while (*progress < need) {
        if (*abort || globaltimer_ns() - t0 > 20000000ull) return;
        __nanosleep(200);
      }
      if (first_a)
        prefetch_rows(p.pf_a, p.pf_lda, mb * BM + static_cast<int>(rank) * BM_CTA, BM_CTA, p.M,
                      kb * kStageKBytes, kStageKBytes, p.pf_kbytes, t);
      if (first_b)
        prefetch_rows(p.pf_b, p.pf_ldb, nb * BN + static_cast<int>(rank) * (BN / 2), BN / 2, p.N,
                      kb * kStageKBytes, kStageKBytes, p.pf_kbytes, t);
    }
  }
}

// Where a pipeline stage lies along k: for a GEMM, k0 is the k of its first
// atom in A and B; for a convolution, k0 is the channel offset within filter
// tap (r, s) and bcol the matching column of the K x (R*S*C) weights.  The
// producer advances it stage by stage (advance), with no division in its loop.
struct StagePos {
  int k0, r, s, bcol;
};

template <Mode kMode, int ATOMS>
__device__ __forceinline__ void advance(StagePos& q, const KParams& p, int tap_end) {
  constexpr int kKS = BK * ATOMS;
  q.k0 += kKS;
  q.bcol += kKS;
  if constexpr (mode_is_conv(kMode)) {
    if (q.k0 == tap_end) {  // next filter tap: channel block 0, columns from tap * C
      q.k0 = 0;
      q.bcol += p.conv_C - tap_end;
      if (++q.s == p.conv_S) {
        q.s = 0;
        ++q.r;
      }
    }
  }
}

// One pipeline stage's TMA copies into a_dst / b_dst: ATOMS swizzle atoms of A
// (kAtomABytes apart) and of B (kBAtom apart), all completing on barrier `bar`
// of the leader CTA.  A convolution's A rows are gathered by TMA im2col.
template <Mode kMode, int ATOMS, uint32_t kBAtom>
__device__ __forceinline__ void load_stage(const CUtensorMap* tmA, const CUtensorMap* mapB,
                                           uint8_t* a_dst, uint8_t* b_dst, uint32_t bar,
                                           const StagePos& q, int m_cta, int n_cta, int cn, int ch,
                                           int cw) {
  if constexpr (mode_is_conv(kMode)) {
#pragma unroll
    for (int j = 0; j < ATOMS; ++j) {
      tma_load_im2col_4d_2cta(a_dst + j * kAtomABytes, tmA, bar, q.k0 + j * BK, cw, ch, cn,
                              static_cast<uint16_t>(q.s), static_cast<uint16_t>(q.r));
      tma_load_2d_2cta(b_dst + j * kBAtom, mapB, bar, q.bcol + j * BK, n_cta);
    }
  } else {
#pragma unroll
    for (int j = 0; j < ATOMS; ++j) {
      tma_load_2d_2cta(a_dst + j * kAtomABytes, tmA, bar, q.k0 + j * BK, m_cta);
      tma_load_2d_2cta(b_dst + j * kBAtom, mapB, bar, q.bcol + j * BK, n_cta);
    }
  }
}

// One pipeline stage's MMAs (ATOMS atoms x BK/16 steps of k = 16) into the
// accumulator at d_tmem; a_st / b_st are the stage's first descriptors, B atoms
// lie kBAtom apart.  The first MMA of a chunk overwrites the accumulator.
template <int ATOMS, uint32_t kBAtom>
__device__ __forceinline__ void mma_stage(uint32_t d_tmem, uint64_t a_st, uint64_t b_st,
                                          uint32_t idesc, bool accumulate) {
#pragma unroll
  for (int j = 0; j < ATOMS; ++j) {
#pragma unroll
    for (int k = 0; k < BK / 16; ++k) {
      const uint64_t ad = a_st + ((j * kAtomABytes + k * 32) >> 4);
      const uint64_t bd = b_st + ((j * kBAtom + k * 32) >> 4);
      umma_f16_ss_2cta(d_tmem, ad, bd, idesc, (accumulate || j > 0 || k > 0) ? 1u : 0u);
    }
  }
}

// ---------------------------------------------------------------------------
// epilogue helpers (one thread = one output row, NC consecutive columns)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_half2(uint32_t lo_bits, uint32_t hi_bits) {
  __half2 h = __floats2half2_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf162(uint32_t lo_bits, uint32_t hi_bits) {
  __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
  return *reinterpret_cast<uint32_t*>(&h);
}

template <bool kBf16>
__device__ __forceinline__ uint32_t pack2(uint32_t lo_bits, uint32_t hi_bits) {
  if constexpr (kBf16)
    return pack_bf162(lo_bits, hi_bits);
  else
    return pack_half2(lo_bits, hi_bits);
}

// Direct stores of columns c0 .. c1-1 of row m (a row per thread; c0 and c1
// multiples of 8, constants after inlining where the tile width allows).
// vec: 16-byte stores allowed for groups that lie inside the matrix.
template <int NC, bool kBf16>
__device__ __forceinline__ void store_cols_16bit(void* out, long long ldo, int N, int m, int n0,
                                                 bool vec, int c0, int c1,
                                                 const uint32_t (&v)[NC]) {
  static_assert(NC % 8 == 0, "16-byte groups");
  uint16_t* row = reinterpret_cast<uint16_t*>(out) + static_cast<size_t>(m) * ldo + n0;
#pragma unroll
  for (int j = 0; j < NC / 8; ++j) {
    if (8 * j < c0 || 8 * j >= c1) continue;
    if (vec && n0 + 8 * j + 8 <= N) {
      uint4 q;
      q.x = pack2<kBf16>(v[8 * j + 0], v[8 * j + 1]);
      q.y = pack2<kBf16>(v[8 * j + 2], v[8 * j + 3]);
      q.z = pack2<kBf16>(v[8 * j + 4], v[8 * j + 5]);
      q.w = pack2<kBf16>(v[8 * j + 6], v[8 * j + 7]);
      reinterpret_cast<uint4*>(row)[j] = q;
    } else {
#pragma unroll
      for (int i = 8 * j; i < 8 * j + 8; ++i)
        if (n0 + i < N) row[i] = static_cast<uint16_t>(pack2<kBf16>(v[i], 0u) & 0xFFFFu);
    }
  }
}

template <int NC>
__device__ __forceinline__ void store_cols_f32(float* out, long long ldo, int N, int m, int n0,
                                               bool vec, int c0, int c1, const uint32_t (&v)[NC]) {
  static_assert(NC % 4 == 0, "16-byte groups");
  float* row = out + static_cast<size_t>(m) * ldo + n0;
#pragma unroll
  for (int j = 0; j < NC / 4; ++j) {
    if (4 * j < c0 || 4 * j >= c1) continue;
    if (vec && n0 + 4 * j + 4 <= N) {
      reinterpret_cast<uint4*>(row)[j] =
          make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    } else {
#pragma unroll
      for (int i = 4 * j; i < 4 * j + 4; ++i)
        if (n0 + i < N) row[i] = __uint_as_float(v[i]);
    }
  }
}

// One epilogue warp's staging buffer: lane l owns row l (128 bytes) of a 32-row
// TMA box; 16-byte chunk k of the row sits at chunk k ^ (l % 8) (128-byte swizzle).
struct Stager {
  uint8_t* buf;  // 4 KB, 1024-byte aligned
  int lane;
  int row0;      // output row of lane 0
  int M, N;      // output extent (a box wholly outside it is not issued)

  // the previous store from this buffer must have read it before it is rewritten
  __device__ __forceinline__ void begin() const {
    if (lane == 0) bulk_wait_group_read0();
    __syncwarp();
  }
  __device__ __forceinline__ void put(int k, uint4 v) const {
    *reinterpret_cast<uint4*>(buf + lane * 128 + ((k ^ (lane & 7)) << 4)) = v;
  }
  __device__ __forceinline__ void issue(const CUtensorMap* map, int col0) const {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && row0 < M && col0 < N) {
      tma_store_2d(map, buf, col0, row0);
      bulk_commit_group();
    }
  }
};

// 32-bit values (fp32 / int32 bit patterns), boxes of 32 columns: the boxes that
// lie wholly inside the first nvalid columns.
template <int NC>
__device__ __forceinline__ void stage_store_u32(const Stager& st, const CUtensorMap* map, int n0,
                                                const uint32_t (&v)[NC], int nvalid = NC) {
#pragma unroll
  for (int b = 0; b < NC / 32; ++b) {
    if (32 * b + 32 > nvalid) continue;
    st.begin();
#pragma unroll
    for (int k = 0; k < 8; ++k)
      st.put(k, make_uint4(v[b * 32 + 4 * k], v[b * 32 + 4 * k + 1], v[b * 32 + 4 * k + 2],
                           v[b * 32 + 4 * k + 3]));
    st.issue(map, n0 + b * 32);
  }
}

// fp32 values rounded to fp16 / bf16, boxes of 64 columns: the boxes that lie
// wholly inside the first nvalid columns.
template <int NC, bool kBf16>
__device__ __forceinline__ void stage_store_16bit(const Stager& st, const CUtensorMap* map, int n0,
                                                  const uint32_t (&v)[NC], int nvalid = NC) {
#pragma unroll
  for (int b = 0; b < NC / 64; ++b) {
    if (64 * b + 64 > nvalid) continue;
    st.begin();
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = b * 64 + 8 * k;
      st.put(k, make_uint4(pack2<kBf16>(v[c], v[c + 1]), pack2<kBf16>(v[c + 2], v[c + 3]),
                           pack2<kBf16>(v[c + 4], v[c + 5]), pack2<kBf16>(v[c + 6], v[c + 7])));
    }
    st.issue(map, n0 + b * 64);
  }
}

// Row m of the tile, columns n0 .. n0+nvalid-1 (nvalid <= NC; the warp holds NC
// columns), values v (fp32 bit patterns).  Every lane of the warp must call it
// (the TMA path is warp-collective); rows past M are clipped by the store.
// Columns past the last whole TMA box inside nvalid are stored directly.
template <int NC>
__device__ __forceinline__ void store_row_float(const KParams& p, const CUtensorMap& tmO0,
                                                const CUtensorMap& tmO1, const Stager& st, int m,
                                                int n0, const uint32_t (&v)[NC],
                                                int nvalid = NC) {
  const int boxed16 = nvalid / 64 * 64;  // columns stored by whole 16-bit boxes
  const int boxed32 = nvalid / 32 * 32;  // columns stored by whole 32-bit boxes
  const bool in_row = m < p.M;
  if (p.out != nullptr) {
    const bool tma = p.tma_out & 1;
    if (p.out_type == kOutF16) {
      if (tma) stage_store_16bit<NC, false>(st, &tmO0, n0, v, nvalid);
      if (in_row)
        store_cols_16bit<NC, false>(p.out, p.ldo, p.N, m, n0, p.vec_ok, tma ? boxed16 : 0, nvalid, v);
    } else if (p.out_type == kOutBF16) {
      if (tma) stage_store_16bit<NC, true>(st, &tmO0, n0, v, nvalid);
      if (in_row)
        store_cols_16bit<NC, true>(p.out, p.ldo, p.N, m, n0, p.vec_ok, tma ? boxed16 : 0, nvalid, v);
    } else {
      if (tma) stage_store_u32<NC>(st, &tmO0, n0, v, nvalid);
      if (in_row)
        store_cols_f32<NC>(reinterpret_cast<float*>(p.out), p.ldo, p.N, m, n0, p.vec_ok,
                           tma ? boxed32 : 0, nvalid, v);
    }
  }
  if (p.out_f32 != nullptr) {
    const bool tma = p.tma_out & 2;
    if (tma) stage_store_u32<NC>(st, &tmO1, n0, v, nvalid);
    if (in_row)
      store_cols_f32<NC>(p.out_f32, p.ldo32, p.N, m, n0, p.vec_ok, tma ? boxed32 : 0, nvalid, v);
  }
}

// Requantisation of one int32 result: fp32(c) rounded to nearest even, one fp32
// multiply, then one conversion to int8 that rounds to nearest even and
// saturates to [-128, 127] (a NaN product converts to 0).  Returns the byte.
__device__ __forceinline__ uint32_t requant_byte(int32_t c, float s) {
  const float f = __fmul_rn(__int2float_rn(c), s);
  int32_t q;
  asm("cvt.rni.sat.s8.f32 %0, %1;" : "=r"(q) : "f"(f));
  return static_cast<uint32_t>(q) & 0xFFu;
}

constexpr int kG = 16;  // columns per step of the integer epilogue

// The per-column vectors of one warp's NC columns, spread over its lanes: lane l
// holds column n0 + 32 b + l in element b.  They are read with one coalesced
// load per 32 columns, all issued together, and a column's value is broadcast
// to the warp by a shuffle where it is used.  Columns past N read column N-1
// (their outputs are never stored); absent vectors read as 0.
template <int NC>
struct ColVecs {
  static constexpr int kB = (NC + 31) / 32;
  uint32_t cB[kB], zB[kB], sc[kB], dq[kB], bi[kB];
};

template <int NB>
__device__ __forceinline__ void load_col_vec(const void* base, int n0, int N, int lane,
                                             uint32_t (&v)[NB]) {
  const uint32_t* b32 = static_cast<const uint32_t*>(base);
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const int n = n0 + 32 * b + lane;
    v[b] = b32 ? __ldg(b32 + (n < N ? n : N - 1)) : 0u;
  }
}

template <int NC, bool kCv = false>
__device__ __forceinline__ void load_col_vecs(const KParams& p, int n0, int lane,
                                              ColVecs<NC>& V) {
  if constexpr (kCv) {
#pragma unroll
    for (int b = 0; b < ColVecs<NC>::kB; ++b) {
      const int n = n0 + 32 * b + lane;
      V.cB[b] = cv_sum(p, true, n < p.N ? n : p.N - 1);
    }
  } else {
    load_col_vec(p.csumB, n0, p.N, lane, V.cB);
  }
  load_col_vec(p.zB_col, n0, p.N, lane, V.zB);
  load_col_vec(p.scale_col, n0, p.N, lane, V.sc);
  load_col_vec(p.dq_col, n0, p.N, lane, V.dq);
  load_col_vec(p.bias, n0, p.N, lane, V.bi);
}

// Column c (0 .. NC-1, a constant after unrolling) of a lane-spread vector.
template <int NB>
__device__ __forceinline__ uint32_t col_val(const uint32_t (&v)[NB], int c) {
  return __shfl_sync(0xffffffffu, v[c >> 5], c & 31);
}

// Per-row terms of the zero-point expansion, evaluated as
//   C32 = S' - zB'_j (rA'_i - K zA'_i) - zA'_i cB'_j          (int32, mod 2^32)
// which equals S' - zB'_j rA'_i - zA'_i cB'_j + K zA'_i zB'_j.
struct IntRow {
  uint32_t zAp;        // zA'_i
  uint32_t u;          // rA'_i - K zA'_i
  uint32_t t_uniform;  // zB' u when zB is per tensor
  float sA;            // dequantisation row scale
};

// The row terms from rs = rA'_i, the row sum of the shifted A operand.
__device__ __forceinline__ IntRow int_row_from(const KParams& p, int m, uint32_t rs) {
  const int mm = m < p.M ? m : p.M - 1;  // rows past M are computed (and clipped) like row M-1
  IntRow r;
  r.zAp = static_cast<uint32_t>((p.zA_row ? __ldg(p.zA_row + mm) : p.zA) - p.oA);
  r.u = rs - static_cast<uint32_t>(p.K) * r.zAp;
  r.t_uniform = static_cast<uint32_t>(p.zB - p.oB) * r.u;
  r.sA = p.dq_row ? __ldg(p.dq_row + mm) : 1.0f;
  return r;
}

template <bool kCv = false>
__device__ __forceinline__ IntRow int_row(const KParams& p, int m) {
  const int mm = m < p.M ? m : p.M - 1;  // rows past M are computed (and clipped) like row M-1
  uint32_t rs;
  if (p.px != nullptr) {
    const int PQ = p.conv_P * p.conv_Q;
    const int n = mm / PQ;
    const int rem = mm - n * PQ;
    const int pp = rem / p.conv_Q;
    const int qq = rem - pp * p.conv_Q;
    const int32_t* base = p.px + (static_cast<size_t>(n) * p.conv_Hp + static_cast<size_t>(pp) *
                                  p.stride_h) * p.conv_Wp + static_cast<size_t>(qq) * p.stride_w;
    rs = 0;
    for (int r = 0; r < p.conv_R; ++r)
      for (int s = 0; s < p.conv_S; ++s)
        rs += static_cast<uint32_t>(__ldg(base + static_cast<size_t>(r) * p.conv_Wp + s));
  } else if constexpr (kCv) {
    rs = cv_sum(p, false, mm);
  } else {
    rs = static_cast<uint32_t>(__ldg(p.rsumA + mm));
  }
  return int_row_from(p, m, rs);
}

// C32 of the kG columns of group j (tile columns j kG ...).
template <int NC>
__device__ __forceinline__ void int_group(const KParams& p, const IntRow& r, const ColVecs<NC>& V,
                                          const uint32_t (&sum)[NC], int j, int32_t (&c)[kG]) {
  if (p.zB_col) {
#pragma unroll
    for (int i = 0; i < kG; ++i)
      c[i] = static_cast<int32_t>(sum[j * kG + i] -
                                  (col_val(V.zB, j * kG + i) - static_cast<uint32_t>(p.oB)) * r.u -
                                  r.zAp * col_val(V.cB, j * kG + i));
  } else {
#pragma unroll
    for (int i = 0; i < kG; ++i)
      c[i] = static_cast<int32_t>(sum[j * kG + i] - r.t_uniform -
                                  r.zAp * col_val(V.cB, j * kG + i));
  }
}

// The four requantised bytes of columns 4i .. 4i+3 of c, packed little-endian.
template <int NC>
__device__ __forceinline__ void int8_group(const KParams& p, const ColVecs<NC>& V, int j,
                                           const int32_t (&c)[kG], uint32_t (&w)[kG / 4]) {
  float sc[kG];
#pragma unroll
  for (int i = 0; i < kG; ++i)
    sc[i] = p.scale_col ? __uint_as_float(col_val(V.sc, j * kG + i)) : p.scale;
#pragma unroll
  for (int i = 0; i < kG / 4; ++i)
    w[i] = requant_byte(c[4 * i], sc[4 * i]) | (requant_byte(c[4 * i + 1], sc[4 * i + 1]) << 8) |
           (requant_byte(c[4 * i + 2], sc[4 * i + 2]) << 16) |
           (requant_byte(c[4 * i + 3], sc[4 * i + 3]) << 24);
}

// Dequantised fp32 values of c: one RNE fp32 operation per step, in this order, no FMA.
template <int NC>
__device__ __forceinline__ void float_group(const KParams& p, const IntRow& r,
                                            const ColVecs<NC>& V, int j, const int32_t (&c)[kG],
                                            uint32_t (&y)[kG]) {
#pragma unroll
  for (int i = 0; i < kG; ++i) {
    float t = __int2float_rn(c[i]);
    if (p.dq_row) t = __fmul_rn(t, r.sA);
    if (p.dq_col) t = __fmul_rn(t, __uint_as_float(col_val(V.dq, j * kG + i)));
    if (p.bias) t = __fadd_rn(t, __uint_as_float(col_val(V.bi, j * kG + i)));
    y[i] = __float_as_uint(t);
  }
}

// sum[] holds, per column, sum_k A'B' (mod 2^32).  Writes
// the requested integer-mode outputs of row m, columns n0 .. n0+NC-1.  Every lane
// of the warp must call it and run every group: the column values are broadcast
// by shuffles and the TMA paths are warp-collective; only the direct stores are
// predicated on the row.
// The row terms r and the column vectors V come ready-made: the pre-pass
// kernels' epilogue reads them from global memory (epi_int_unit), the kernel
// that converts its operands itself takes the sums from shared memory.
// kDequant false: the caller guarantees p.yf == nullptr (no dequantised output),
// which drops that output's code and registers.
template <int NC, bool kDequant = true>
__device__ __forceinline__ void store_row_int_v(const KParams& p, const CUtensorMap& tmO0,
                                                const CUtensorMap& tmO1, const CUtensorMap& tmO2,
                                                const Stager& st, int m, int n0,
                                                const uint32_t (&sum)[NC], const IntRow& r,
                                                const ColVecs<NC>& V) {
  const bool in_row = m < p.M;
  const bool full = p.vec_ok && (n0 + NC <= p.N);
  // int8 (requantised)
  if (p.c8) {
    if constexpr (NC >= 128) {
      if (p.tma_out & 2) {
#pragma unroll
        for (int b = 0; b < NC / 128; ++b) {
          st.begin();
#pragma unroll
          for (int g = 0; g < 128 / kG; ++g) {
            int32_t c[kG];
            uint32_t w[kG / 4];
            int_group<NC>(p, r, V, sum, b * (128 / kG) + g, c);
            int8_group<NC>(p, V, b * (128 / kG) + g, c, w);
            st.put(g, make_uint4(w[0], w[1], w[2], w[3]));
          }
          st.issue(&tmO1, n0 + b * 128);
        }
      }
    }
    if (!(NC >= 128 && (p.tma_out & 2))) {
      // every lane computes (the column values are shuffled across the warp);
      // rows past M store nothing
      int8_t* row8 = p.c8 + static_cast<size_t>(in_row ? m : 0) * p.ldc8 + n0;
#pragma unroll
      for (int j = 0; j < NC / kG; ++j) {
        int32_t c[kG];
        uint32_t w[kG / 4];
        int_group<NC>(p, r, V, sum, j, c);
        int8_group<NC>(p, V, j, c, w);
        if (!in_row) continue;
        if (full) {
          reinterpret_cast<uint4*>(row8)[j] = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
#pragma unroll
          for (int i = 0; i < kG; ++i)
            if (n0 + j * kG + i < p.N)
              row8[j * kG + i] = static_cast<int8_t>((w[i / 4] >> (8 * (i % 4))) & 0xFFu);
        }
      }
    }
  }
  // int32 and dequantised fp32: 32-bit values, boxes of 32 columns (two groups);
  // one copy of the loop body for both outputs keeps the register count down
#pragma unroll 1
  for (int o = 0; o < (kDequant ? 2 : 1); ++o) {
    void* outp = o == 0 ? static_cast<void*>(p.c32) : static_cast<void*>(p.yf);
    if (outp == nullptr) continue;
    const bool tma = (p.tma_out >> (o == 0 ? 0 : 2)) & 1;
    const CUtensorMap* map = o == 0 ? &tmO0 : &tmO2;
    const long long ld = o == 0 ? p.ldc32 : p.ldyf;
    uint32_t* row = reinterpret_cast<uint32_t*>(outp) + static_cast<size_t>(in_row ? m : 0) * ld + n0;
#pragma unroll
    for (int b = 0; b < NC / 32; ++b) {
      if (tma) st.begin();
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const int j = 2 * b + g;
        int32_t c[kG];
        uint32_t y[kG];
        int_group<NC>(p, r, V, sum, j, c);
        if (!kDequant || o == 0) {
#pragma unroll
          for (int i = 0; i < kG; ++i) y[i] = static_cast<uint32_t>(c[i]);
        } else {
          float_group<NC>(p, r, V, j, c, y);
        }
        if (tma) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            st.put(g * 4 + i, make_uint4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]));
        } else if (in_row) {
          if (full) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              reinterpret_cast<uint4*>(row + j * kG)[i] =
                  make_uint4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < kG; ++i)
              if (n0 + j * kG + i < p.N) row[j * kG + i] = y[i];
          }
        }
      }
      if (tma) st.issue(map, n0 + b * 32);
    }
  }
}

// Loads NC consecutive TMEM columns (this warp's 32 lanes) into v: 32 columns
// per tcgen05.ld, then 16 for a remainder.  The caller waits (tmem_ld_wait).
template <int NC>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, uint32_t (&v)[NC]) {
#pragma unroll
  for (int j = 0; j < NC / 32; ++j) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(taddr + j * 32, r);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[j * 32 + i] = r[i];
  }
  if constexpr (NC % 32 != 0) {
    uint32_t r[16];
    tmem_ld_32x32b_x16(taddr + (NC / 32) * 32, r);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[(NC / 32) * 32 + i] = r[i];
  }
}

// Drains NC fp32 TMEM columns holding the exact integer sums of one chunk into
// the int32 running sums (set by the first chunk, added after it), two
// 32-column loads per wait.  Conversion toward zero is exact for integral values.
template <int NC>
__device__ __forceinline__ void tmem_drain(uint32_t taddr, uint32_t (&sum)[NC], bool first) {
  static_assert(NC % 64 == 0, "drain in steps of 64 columns");
#pragma unroll
  for (int j = 0; j < NC / 64; ++j) {
    uint32_t r0[32], r1[32];
    tmem_ld_32x32b_x32(taddr + j * 64, r0);
    tmem_ld_32x32b_x32(taddr + j * 64 + 32, r1);
    tmem_ld_wait();
    if (first) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        sum[j * 64 + i] = static_cast<uint32_t>(__float2int_rz(__uint_as_float(r0[i])));
        sum[j * 64 + 32 + i] = static_cast<uint32_t>(__float2int_rz(__uint_as_float(r1[i])));
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        sum[j * 64 + i] += static_cast<uint32_t>(__float2int_rz(__uint_as_float(r0[i])));
        sum[j * 64 + 32 + i] += static_cast<uint32_t>(__float2int_rz(__uint_as_float(r1[i])));
      }
    }
  }
}

// tmem_drain with one 32-column load per wait (half the registers in flight),
// for epilogues that run with a smaller register budget.
template <int NC>
__device__ __forceinline__ void tmem_drain_x32(uint32_t taddr, uint32_t (&sum)[NC], bool first) {
  static_assert(NC % 32 == 0, "drain in steps of 32 columns");
#pragma unroll
  for (int j = 0; j < NC / 32; ++j) {
    uint32_t r0[32];
    tmem_ld_32x32b_x32(taddr + j * 32, r0);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint32_t v = static_cast<uint32_t>(__float2int_rz(__uint_as_float(r0[i])));
      sum[j * 32 + i] = first ? v : sum[j * 32 + i] + v;
    }
  }
}

// One warp's float epilogue for a unit: NCX accumulator columns from TMEM
// address taddr, the accumulator released (arrival on the leader's `tempty`)
// as soon as they are in registers, then row m's outputs at columns
// n0 .. n0+nvalid-1.
// Inactive warps (the idle half of a half unit) only take part in the release.
template <int NCX>
__device__ __forceinline__ void epi_float_cols(const KParams& p, const CUtensorMap& tmO0,
                                               const CUtensorMap& tmO1, const Stager& st,
                                               uint32_t taddr, int m, int n0, int nvalid,
                                               bool active, uint32_t release_bar, int lane) {
  uint32_t v[NCX];
  if (active) {
    tmem_load_cols<NCX>(taddr, v);
    tmem_ld_wait();
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive_remote(release_bar);
  if (active) store_row_float<NCX>(p, tmO0, tmO1, st, m, n0, v, nvalid);
}

// One warp's integer epilogue for a unit: NCX columns of this warp's lanes at
// TMEM address cols (accumulator 0; accumulator a lies a * acc_stride further),
// drained chunk by chunk into int32 running sums, each accumulator released
// (arrival on the leader's tempty) once drained, then row m's outputs at columns
// n0 .. n0+NCX-1.  kEarly: the row terms and column vectors are read before the
// first accumulator wait, where their latency hides behind the MMAs; the widest
// warps (NCX = 128) read them after the drain, when the registers are free.
// An inactive warp (the idle half of a half unit) only takes part in the
// releases.  An integer GEMM converting its own operands: between polls of the
// accumulator barrier the warp does conversion jobs: its share of the first band
// (cv_next: its next one), then jobs of the later bands while cv_left (as many as
// fit before the warp's first accumulator, cv_first and chunk 0; one per chunk
// after that; cv_left turns false once their queue is empty).  Returns false if a
// wait gave up.
template <int BN, int NCX, bool kEarly, bool kCv>
__device__ __forceinline__ bool epi_int_unit(const KParams& p, const CUtensorMap& tmO0,
                                             const CUtensorMap& tmO1, const CUtensorMap& tmO2,
                                             const Stager& st, uint32_t cols, uint32_t acc_stride,
                                             int m, int n0, int n_chunks, bool active,
                                             bool& cv_left, int& cv_next, bool cv_first,
                                             const int2* cv_tab, int C,
                                             const volatile int* progress, uint64_t* tfull,
                                             uint32_t tempty_lead, int& acc, uint32_t& acc_phase,
                                             uint64_t lim, volatile int* abort_flag, int lane) {
  uint32_t sum[NCX];
  IntRow r;
  ColVecs<NCX> V;
  // (a kernel converting its own operands has its sums only once the MMAs could run)
  constexpr bool early = kEarly && !kCv;
  if constexpr (early) {
    r = int_row<kCv>(p, m);
    load_col_vecs<NCX, kCv>(p, n0, lane, V);
  }
  for (int c = 0; c < n_chunks; ++c) {
    if constexpr (kCv) {
      // The warp's share of the first band comes first, whenever it waits; then, from
      // the queue of the later bands, as many jobs as fit before its first
      // accumulator and one every other chunk after that, none in a unit's last two
      // chunks: a job taken right after a drain ends before the accumulator after
      // next is needed, and the unit's outputs are written without conversion
      // traffic of the warp's own in flight, so the drains (and the MMAs that wait
      // for them) are not held up.
      const uint32_t bar = smem_u32(&tfull[acc]);
      int budget = (cv_first && c == 0) ? 0x7fffffff : ((c & 1) && c < n_chunks - 2 ? 1 : 0);
      while (__shfl_sync(0xffffffffu, lane == 0 ? (mbar_test_wait(bar, acc_phase) ? 1 : 0) : 0,
                         0) == 0) {
        if (cv_static_step<BN, 4>(p, cv_tab, C, cv_next, lane)) continue;
        if (!cv_left || budget <= 0) break;
        const int r = cv_step<BN, 4>(p, cv_tab, C, cv_max_band(p, progress), lane);
        if (r == kCvNone) cv_left = false;
        if (r != kCvDid) break;
        --budget;
      }
    }
    if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, lim, abort_flag, p.status,
                                            kSiteEpiFull)))
      return false;
    tc_fence_after();
    const uint32_t taddr = cols + static_cast<uint32_t>(acc) * acc_stride;
    if (active) {
      if constexpr (NCX % 64 == 0)
        tmem_drain<NCX>(taddr, sum, c == 0);
      else
        tmem_drain_x32<NCX>(taddr, sum, c == 0);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive_remote(tempty_lead + static_cast<uint32_t>(acc) * 8u);
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
  }
  if constexpr (!early) {
    if constexpr (kCv) cv_acquire_sums<ColVecs<NCX>::kB>(p, m, n0, lane);
    r = int_row<kCv>(p, m);
    load_col_vecs<NCX, kCv>(p, n0, lane, V);
  }
  if (active) store_row_int_v<NCX>(p, tmO0, tmO1, tmO2, st, m, n0, sum, r, V);
  return true;
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <Mode kMode, int BN, int ATOMS>
__global__ void __launch_bounds__(kThreads, 1)
    igc_tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmBh,
                       const __grid_constant__ CUtensorMap tmO0,
                       const __grid_constant__ CUtensorMap tmO1,
                       const __grid_constant__ CUtensorMap tmO2, const KParams p) {
  using Cfg = TileCfg<BN, ATOMS>;
  // the integer modes (exact 1024-k chunks of kIntChunkKb stages) use the default depth
  static_assert(ATOMS == kAtoms || !mode_is_int(kMode), "ATOMS");
  constexpr int kStages = Cfg::kStages;
  constexpr uint32_t kStageABytes = Cfg::kStageABytes;
  constexpr int NC = Cfg::kEpiCols;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);

  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kStageABytes;
  uint8_t* staging = sB + kStages * Cfg::kStageBBytes;  // 1024-byte aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + kStagingBytes);
  uint64_t* full = bars;                 // leader: both CTAs' copies of stage s landed
  uint64_t* empty = bars + kStages;      // each CTA: stage s may be overwritten
  uint64_t* tfull = bars + 2 * kStages;  // each CTA: accumulator a is ready
  uint64_t* tempty = tfull + 2;          // leader: both epilogues released accumulator a
  uint64_t* mma_done = tempty + 2;
  uint64_t* full_t = mma_done + 1;                // tail ring (Cfg::kTailRing)
  uint64_t* empty_t = full_t + Cfg::kTailStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(empty_t + Cfg::kTailStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* progress = abort_flag + 1;  // producer: stages issued (prefetch, converters)
  int* first_unit = const_cast<int*>(progress) + 1;  // the first unit's Unit fields
  int2* cv_tab = reinterpret_cast<int2*>(reinterpret_cast<uint8_t*>(bars) + 512);

  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 32, 0);
  const int lane = static_cast<int>(lane_id());
  const uint32_t rank = cluster_ctarank();  // 0 = leader
  const int cluster = static_cast<int>(blockIdx.x) >> 1;
  const int num_clusters = static_cast<int>(gridDim.x) >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * kEpiWarps);
    }
    mbar_init(mma_done, 1);
    if constexpr (Cfg::kTailRing) {
      for (int s = 0; s < Cfg::kTailStages; ++s) {
        mbar_init(&full_t[s], 1);
        mbar_init(&empty_t[s], 1);
      }
    }
    *abort_flag = 0;
    *progress = 0;
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
  if (warp == 3 && lane == 0) store_first_unit(p, cluster, first_unit);
  if constexpr (kMode == Mode::GemmIntCv) {
    // the conversion jobs' band table: the blocks before each band
    if (p.cv_flags != nullptr && warp == 2) {
      const int nb = cv_num_bands(p, num_clusters);
      for (int b = lane; b <= nb && b < kCvBandTab; b += 32)
        cv_tab[b] = cv_blocks_before<BN>(p, b, num_clusters);
    }
  }
  tc_fence_before();
  // barriers of both CTAs initialised, TMEM allocated in both, first unit known
  cluster_arrive();
  // Between its arrival and the barrier's completion warp 3 prefetches a floating
  // GEMM's first stages into L2 (an integer GEMM's operands are written by its
  // pre-pass, the kernel before it in the stream).  The copy engine may hold the
  // thread until the tensor maps are fetched, which then delays only this warp.
  if constexpr (kMode == Mode::GemmF16 || kMode == Mode::GemmBF16)
    if (warp == 3 && lane == 0)
      prefetch_first_stages<BN, ATOMS>(p, &tmA, &tmB, &tmBh, first_unit, rank, kStages);
  cluster_wait();
  tc_fence_after();
  // Set-up above reads and writes no global memory (an L2 prefetch makes nothing
  // visible); from here on the previous kernel in the stream must have finished
  // (programmatic dependent launch).
  grid_dependency_wait();
  grid_dependents_launch();
  const uint32_t tmem_base = *tmem_slot;
  const uint64_t lim = p.wait_limit_ns;
  // The pair's MMAs write both CTAs' tensor memory at the leader's address: both
  // allocations must agree, else the pair does no work at all.
  const uint32_t peer_base = ld_shared_cluster_u32(mapa_shared(smem_u32(tmem_slot), rank ^ 1u));
  const bool pair_ok = peer_base == tmem_base;
  if (!pair_ok && threadIdx.x == 0) report_status(p.status, kStatusBadLaunch, kSiteTmemMismatch);
  // the leader's barriers, as cluster addresses usable from either CTA
  const uint32_t full_lead = mapa_shared(smem_u32(full), 0);
  const uint32_t full_t_lead = mapa_shared(smem_u32(full_t), 0);
  const uint32_t tempty_lead = mapa_shared(smem_u32(tempty), 0);

  if (warp < 4) {
    warpgroup_regs_dec<kRegsLow>();
    if (pair_ok && warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop (converged); lane 0 issues the copies.
    int stage = 0;
    uint32_t phase = 0;
    long long issued = 0;
    // tail ring: the main ring's next stage and phase at the switch (sw_stage >= 0
    // once switched) and the fills issued on the main ring before it
    int sw_stage = -1;
    uint32_t sw_phase = 0;
    long long issued_main = 0;
    // a convolution's stages walk the channel blocks of each filter tap in turn
    const int tap_end = p.conv_cblocks * Cfg::kKS;
    for (int u = cluster; u < p.num_units; u += num_clusters) {
      const Unit w = u == cluster ? load_first_unit(first_unit) : unit_coords(p, u);
      const int mb = w.mb;
      const int m_cta = mb * BM + static_cast<int>(rank) * BM_CTA;
      const int n_cta = b_row0<BN>(w, rank);
      const CUtensorMap* mapB = w.half ? &tmBh : &tmB;
      const uint32_t stage_tx =
          2u * (kStageABytes + (w.half ? Cfg::kStageBBytes / 2 : Cfg::kStageBBytes));
      int cn = 0, ch = 0, cw = 0;
      if constexpr (mode_is_conv(kMode)) {
        const int PQ = p.conv_P * p.conv_Q;
        cn = m_cta / PQ;
        const int rem = m_cta - cn * PQ;
        const int pp = rem / p.conv_Q;
        const int qq = rem - pp * p.conv_Q;
        ch = pp * p.stride_h - p.pad_h;
        cw = qq * p.stride_w - p.pad_w;
      }
      StagePos q{0, 0, 0, 0};
      // integer GEMM converting its operands: the unit's blocks all done (checked
      // before the first free slot is waited for, while the ring is still full)
      bool cv_ready = false;
      if constexpr (kMode == Mode::GemmIntCv)
        if (p.cv_flags != nullptr) cv_ready = cv_unit_ready(p, m_cta, n_cta, lane);
      if (!Cfg::kTailRing || !w.half) {
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(&empty[stage], phase ^ 1u, lim, abort_flag,
                                                  p.status, kSiteProducerEmpty)))
            goto producer_done;
          if constexpr (kMode == Mode::GemmIntCv) {
            if (p.cv_flags != nullptr && !cv_ready && kb % p.chunk_kb == 0 &&
                !cv_wait_chunk(p, m_cta, n_cta, kb / p.chunk_kb, lim, abort_flag, lane))
              goto producer_done;
          }
          if (lane == 0) {
            if (rank == 0) mbar_arrive_expect_tx(&full[stage], stage_tx);
            load_stage<kMode, ATOMS, Cfg::kAtomBBytes>(
                &tmA, mapB, sA + stage * kStageABytes, sB + stage * Cfg::kStageBBytes,
                full_lead + static_cast<uint32_t>(stage) * 8u, q, m_cta, n_cta, cn, ch, cw);
          }
          __syncwarp();
          advance<kMode, ATOMS>(q, p, tap_end);
          ++issued;
          if (lane == 0) *progress = static_cast<int>(issued);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      } else if constexpr (Cfg::kTailRing) {
        if (sw_stage < 0) {
          sw_stage = stage;
          sw_phase = phase;
          issued_main = issued;
          stage = 0;
          phase = 0;
          issued = 0;
        }
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(&empty_t[stage], phase ^ 1u, lim, abort_flag,
                                                  p.status, kSiteProducerEmpty)))
            goto producer_done;
          if (issued < kStages) {
            // first fill of tail slot `issued`: main stage m_issued (released after
            // m_0 .. m_issued-1, which earlier fills waited for) must be free
            const int ms = (sw_stage + static_cast<int>(issued)) % kStages;
            const uint32_t par = ms < sw_stage ? sw_phase : (sw_phase ^ 1u);
            if (!__all_sync(0xffffffffu, mbar_wait(&empty[ms], par, lim, abort_flag, p.status,
                                                    kSiteProducerEmpty)))
              goto producer_done;
          }
          if constexpr (kMode == Mode::GemmIntCv) {
            if (p.cv_flags != nullptr && !cv_ready && kb % p.chunk_kb == 0 &&
                !cv_wait_chunk(p, m_cta, n_cta, kb / p.chunk_kb, lim, abort_flag, lane))
              goto producer_done;
          }
          if (lane == 0) {
            uint32_t a_off, b_off;
            tail_slot(stage, sw_stage, a_off, b_off);
            if (rank == 0) mbar_arrive_expect_tx(&full_t[stage], stage_tx);
            load_stage<kMode, ATOMS, Cfg::kAtomBBytes / 2>(
                &tmA, mapB, smem + a_off, smem + b_off,
                full_t_lead + static_cast<uint32_t>(stage) * 8u, q, m_cta, n_cta, cn, ch, cw);
          }
          __syncwarp();
          advance<kMode, ATOMS>(q, p, tap_end);
          ++issued;
          if (++stage == Cfg::kTailStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  producer_done:
    if (lane == 0 && *abort_flag && (issued > 0 || issued_main > 0)) {
      // The copies signal the leader's barriers; give this CTA's own in-flight
      // copies time to land before the CTA may exit (a copy takes microseconds).
      if (rank == 0) {
        if (sw_stage >= 0) {
          drain_fills(full_t, Cfg::kTailStages, stage, phase, issued, lim);
          drain_fills(full, kStages, sw_stage, sw_phase, issued_main, lim);
        } else {
          drain_fills(full, kStages, stage, phase, issued, lim);
        }
      } else {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
    } else if (pair_ok && warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    // The whole warp runs the loop (converged); lane 0 issues MMAs and commits.
    if (rank == 0) {
      constexpr uint32_t idesc_full =
          make_idesc_kind_f16(BM, BN, kMode == Mode::GemmBF16 ? 1u : 0u);
      constexpr uint32_t idesc_half =
          make_idesc_kind_f16(BM, BN / 2, kMode == Mode::GemmBF16 ? 1u : 0u);
      // descriptors of stage 0, atom 0, k 0; the start-address field (bits 0-13,
      // in 16-byte units) is advanced by adding offsets >> 4 (no carry: < 256 KB)
      const uint64_t adesc0 = make_sw128_kmajor_desc(smem_u32(sA));
      const uint64_t bdesc0 = make_sw128_kmajor_desc(smem_u32(sB));
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int sw_stage = -1;  // main-ring stage at the switch to the tail ring
      for (int u = cluster; u < p.num_units; u += num_clusters) {
        const bool half_unit = u >= p.tail_start;
        const uint32_t idesc = half_unit ? idesc_half : idesc_full;
        int kin = 0;
        if (!Cfg::kTailRing || !half_unit) {
          for (int kb = 0; kb < p.num_kb; ++kb) {
            if (kin == 0) {
              if (!__all_sync(0xffffffffu, mbar_wait(&tempty[acc], acc_phase ^ 1u, lim,
                                                      abort_flag, p.status, kSiteMmaTmemEmpty)))
                goto mma_done_label;
              tc_fence_after();
            }
            if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase, lim, abort_flag, p.status,
                                                    kSiteMmaFull)))
              goto mma_done_label;
            tc_fence_after();
            const bool chunk_end = (kin == p.chunk_kb - 1) || (kb == p.num_kb - 1);
            if (lane == 0) {
              mma_stage<ATOMS, Cfg::kAtomBBytes>(
                  tmem_base + static_cast<uint32_t>(acc) * Cfg::kAccStride,
                  adesc0 + ((static_cast<uint32_t>(stage) * kStageABytes) >> 4),
                  bdesc0 + ((static_cast<uint32_t>(stage) * Cfg::kStageBBytes) >> 4), idesc,
                  kin > 0);
              umma_commit_2cta_multicast(&empty[stage], 0x3);
              if (chunk_end) umma_commit_2cta_multicast(&tfull[acc], 0x3);
            }
            __syncwarp();
            if (chunk_end) {
              acc ^= 1;
              if (acc == 0) acc_phase ^= 1u;
            }
            if (++kin == p.chunk_kb) kin = 0;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        } else if constexpr (Cfg::kTailRing) {
          if (sw_stage < 0) {
            sw_stage = stage;
            stage = 0;
            phase = 0;
          }
          for (int kb = 0; kb < p.num_kb; ++kb) {
            if (kin == 0) {
              if (!__all_sync(0xffffffffu, mbar_wait(&tempty[acc], acc_phase ^ 1u, lim,
                                                      abort_flag, p.status, kSiteMmaTmemEmpty)))
                goto mma_done_label;
              tc_fence_after();
            }
            if (!__all_sync(0xffffffffu, mbar_wait(&full_t[stage], phase, lim, abort_flag,
                                                    p.status, kSiteMmaFull)))
              goto mma_done_label;
            tc_fence_after();
            const bool chunk_end = (kin == p.chunk_kb - 1) || (kb == p.num_kb - 1);
            if (lane == 0) {
              // the rings share their base, sA, whose descriptor is adesc0
              uint32_t a_off, b_off;
              tail_slot(stage, sw_stage, a_off, b_off);
              mma_stage<ATOMS, Cfg::kAtomBBytes / 2>(
                  tmem_base + static_cast<uint32_t>(acc) * Cfg::kAccStride, adesc0 + (a_off >> 4),
                  adesc0 + (b_off >> 4), idesc, kin > 0);
              umma_commit_2cta_multicast(&empty_t[stage], 0x3);
              if (chunk_end) umma_commit_2cta_multicast(&tfull[acc], 0x3);
            }
            __syncwarp();
            if (chunk_end) {
              acc ^= 1;
              if (acc == 0) acc_phase ^= 1u;
            }
            if (++kin == p.chunk_kb) kin = 0;
            if (++stage == Cfg::kTailStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
    mma_done_label:
      if (lane == 0) {
        // every MMA issued by this thread has finished once mma_done completes
        umma_commit_2cta(mma_done);
        int dummy = 0;
        mbar_wait(mma_done, 0, lim, &dummy, p.status, kSiteDrain);
      }
      __syncwarp();
    }
    } else if (pair_ok && (p.pf_units > 0 || p.cv_flags != nullptr)) {
    // ------------------------------------------------------------ L2 prefetch (warps 2-3)
    // or, in an integer GEMM converting its own operands, operand conversion
      if constexpr (kMode == Mode::GemmIntCv) {
        if (p.cv_flags != nullptr) {
          // until the queue is empty; a job that may not be taken yet is waited
          // for (bounded: a producer that stopped lets this warp stop too)
          int next = cv_static_worker(warp);
          while (cv_static_step<BN, 2>(p, cv_tab, num_clusters, next, lane)) {
          }
          uint64_t t_later = 0;
          for (;;) {
            const int r = cv_step<BN, 2>(p, cv_tab, num_clusters, cv_max_band(p, progress), lane);
            if (r == kCvNone || *abort_flag) break;
            if (r == kCvDid) {
              t_later = 0;
            } else {
              const uint64_t now = globaltimer_ns();
              if (t_later == 0) t_later = now;
              if (now - t_later > lim) break;
              __nanosleep(1000);
            }
          }
        }
      }
      if constexpr (!mode_is_conv(kMode))
        if (p.pf_units > 0)
          prefetch_first_units<BN, Cfg::kKS * 2>(p, cluster, num_clusters, rank,
                                                 (warp - 2) * 32 + lane, progress, abort_flag);
    }
  } else {
    warpgroup_regs_inc<kRegsHigh>();
    if (pair_ok) {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 4;
    const int quad = warp & 3;  // tcgen05.ld: warp w may access lanes 32*(w%4) .. +31
    const int half = ew >> 2;   // which column half of the tile
    const int row_in_cta = quad * 32 + lane;
    // TMEM address of this warp's lanes, accumulator 0, column 0
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    const int n_chunks = (p.num_kb + p.chunk_kb - 1) / p.chunk_kb;
    Stager st;
    st.buf = staging + ew * kStagingWarpBytes;
    st.lane = lane;
    st.M = p.M;
    st.N = p.N;
    // An integer GEMM converting its own operands: the epilogue warps convert while
    // they wait for an accumulator (epi_int_unit) until no job is left.
    bool cv_left = false;
    int cv_next = cv_static_worker(warp);  // this warp's next first-band job
    if constexpr (kMode == Mode::GemmIntCv) cv_left = p.cv_flags != nullptr;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = cluster; u < p.num_units; u += num_clusters) {
      const Unit w = unit_coords(p, u);
      const int m = w.mb * BM + static_cast<int>(rank) * BM_CTA + row_in_cta;
      // A whole tile's warps take NC columns each (warpgroup `half` the tile's
      // column half); a half unit's BN/2 columns are split the same way, NC/2
      // per warp, except at BN = 224 and in the integer modes' BN = 256, where the
      // half-0 warps take all of them and the others only take part in the
      // accumulator hand-offs.
      const bool active = !w.half || half == 0;
      const int n0 = w.half ? w.nb * BN + w.j * NC : w.nb * BN + half * NC;
      const int n0h = w.nb * BN + w.j * NC + half * (NC / 2);  // split half unit
      st.row0 = m - lane;
      if constexpr (!mode_is_int(kMode)) {
        if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, lim, abort_flag,
                                                        p.status, kSiteEpiFull)))
          goto epi_done;
        tc_fence_after();
        const uint32_t rel = tempty_lead + static_cast<uint32_t>(acc) * 8u;
        const uint32_t acc_cols = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                  static_cast<uint32_t>(acc) * Cfg::kAccStride;
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
        if constexpr (BN == 224) {
          // every warp loads 128 columns from a 32-aligned column (0 or 128) and
          // stores the ones its unit owns: 128 + 96 for a whole tile, 112 (from
          // column 0, half-0 warps) for a half unit
          const int col = w.half ? 0 : half * 128;
          const int nvalid = w.half ? BN / 2 : (half == 0 ? 128 : BN - 128);
          epi_float_cols<128>(p, tmO0, tmO1, st, acc_cols + static_cast<uint32_t>(col), m,
                              w.half ? n0 : w.nb * BN + col, nvalid, active, rel, lane);
        } else if (w.half) {
          epi_float_cols<NC / 2>(p, tmO0, tmO1, st,
                                 acc_cols + static_cast<uint32_t>(half * (NC / 2)), m, n0h,
                                 NC / 2, true, rel, lane);
        } else {
          epi_float_cols<NC>(p, tmO0, tmO1, st, acc_cols + static_cast<uint32_t>(half * NC), m,
                             n0, NC, true, rel, lane);
        }
      } else {
        // (two inlined copies of the widest epilogue would not fit the registers:
        // at NC = 128 a half unit keeps the half-0 warps alone)
        bool ok;
        const bool cv_first = u == cluster;
        if constexpr (NC <= 64) {
          ok = w.half
                   ? epi_int_unit<BN, NC / 2, true, kMode == Mode::GemmIntCv>(
                         p, tmO0, tmO1, tmO2, st,
                         lane_base + static_cast<uint32_t>(half * (NC / 2)), Cfg::kAccStride, m,
                         n0h, n_chunks, true, cv_left, cv_next, cv_first, cv_tab, num_clusters, progress,
                         tfull, tempty_lead, acc, acc_phase, lim, abort_flag, lane)
                   : epi_int_unit<BN, NC, true, kMode == Mode::GemmIntCv>(
                         p, tmO0, tmO1, tmO2, st, lane_base + static_cast<uint32_t>(half * NC),
                         Cfg::kAccStride, m, n0, n_chunks, true, cv_left, cv_next, cv_first, cv_tab,
                         num_clusters, progress, tfull, tempty_lead, acc, acc_phase, lim,
                         abort_flag, lane);
        } else {
          ok = epi_int_unit<BN, NC, false, kMode == Mode::GemmIntCv>(
              p, tmO0, tmO1, tmO2, st, lane_base + static_cast<uint32_t>(half * NC),
              Cfg::kAccStride, m, n0, n_chunks, active, cv_left, cv_next, cv_first, cv_tab, num_clusters,
              progress, tfull, tempty_lead, acc, acc_phase, lim, abort_flag, lane);
        }
        if (!ok) goto epi_done;
      }
    }
    // whatever is left of this warp's first-band share (other CTAs' copies may
    // wait for it even when this CTA's own units are done)
    if constexpr (kMode == Mode::GemmIntCv)
      if (p.cv_flags != nullptr)
        while (cv_static_step<BN, 4>(p, cv_tab, num_clusters, cv_next, lane)) {
        }
  epi_done:
    // every staged store of this warp has completed before the CTA may exit
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
    }
  }

  // ---------------------------------------------------------------- teardown
  // No CTA of the pair may exit (or free tensor memory) while its peer can still
  // touch its shared memory or barriers.
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_2cta(tmem_base, Cfg::kTmemCols);
  }
}

}  // namespace igc
