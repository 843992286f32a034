// The warp-level (IMMA) path of gemm_s8_zp, chosen by igc_set_int8_path(1): the
// exact integer GEMM S[i,j] = sum_k A_q[i,k] B_q[j,k] on the raw uint8 / int8
// operands with mma.sync m16n8k32 (int32 accumulators in registers), then the
// zero-point correction and requantisation of page "TVM在CUDA GPU上跑GEMM的全套
// 张量化实现", §2.3 in int32 two's complement:
//    C32 = S - zB_j rA_i - zA_i cB_j + K zA_i zB_j,   rA_i = sum_k A_q[i,k],
//    cB_j = sum_k B_q[j,k];   C8 = clamp(rne(fp32(C32) * scale_j), -128, 127).
// It is the legacy tensor path (sm_103a runs warp-level integer MMA far below its
// tcgen05 fp16 rate); the tcgen05 path of gemm_s8.cu computes the same results.
#include "igc_host.h"

namespace igc {
namespace imma {

constexpr int kBM = 128;  // block tile rows (A) and columns (B rows)
constexpr int kBN = 128;
constexpr int kBK = 32;   // k of one mma.sync.m16n8k32
constexpr int kPad = 16;  // shared row stride 48 bytes: fragment loads hit 32 distinct banks
constexpr int kThreadsImma = 256;  // 8 warps, 2 (m) x 4 (n), each 64 x 32 outputs

struct Params {
  int M, N, K;
  const uint8_t* A;
  long long lda;
  const uint8_t* B;
  long long ldb;
  const int32_t* rA;
  const int32_t* cB;
  int32_t zA;
  const int32_t* zA_row;
  int32_t zB;
  const int32_t* zB_col;
  int32_t* c32;
  long long ldc32;
  int8_t* c8;
  long long ldc8;
  float scale;
  const float* scale_col;
};

// Raw sums of the rows of a rows x K byte matrix (row stride ld): one warp per row.
template <bool kSigned>
__global__ void row_sums_kernel(const uint8_t* X, long long ld, int rows, int K, int32_t* sums) {
  const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = static_cast<int>(threadIdx.x & 31u);
  if (w >= rows) return;
  const uint8_t* r = X + w * ld;
  int32_t s = 0;
  for (int k = lane; k < K; k += 32)
    s += kSigned ? static_cast<int32_t>(static_cast<int8_t>(r[k])) : static_cast<int32_t>(r[k]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) sums[w] = s;
}

// 16 bytes of row `row` from k0, zero past K (whole vectors where they fit).
__device__ __forceinline__ uint4 load_k16(const uint8_t* row, int k0, int K) {
  if (k0 + 16 <= K) return *reinterpret_cast<const uint4*>(row + k0);
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  for (int b = 0; b < 16 && k0 + b < K; ++b)
    w[b >> 2] |= static_cast<uint32_t>(row[k0 + b]) << (8 * (b & 3));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <bool kAS, bool kBS>
__device__ __forceinline__ void mma_s8(int32_t (&d)[4], const uint32_t (&a)[4],
                                       const uint32_t (&b)[2]) {
  if constexpr (kAS && kBS)
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  else if constexpr (kAS && !kBS)
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.u8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  else if constexpr (!kAS && kBS)
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.u8.u8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// One 128 x 128 output block per CTA.  Per k step of 32 every thread stages 16
// bytes of A and of B (row = thread / 2), then each warp runs 4 x 4 mma.sync on
// its 64 x 32 sub-block.  Fragment layout of m16n8k32 (groupID g = lane / 4,
// t = lane % 4): A regs {row g, k 4t..4t+3}, {row g+8, same k}, {row g, k+16},
// {row g+8, k+16}; B regs {k 4t..4t+3, col g}, {k+16, col g}; D regs {row g,
// cols 2t, 2t+1}, {row g+8, cols 2t, 2t+1}.
template <bool kAS, bool kBS>
__global__ void __launch_bounds__(kThreadsImma) imma_gemm_kernel(const Params p) {
  __shared__ __align__(16) uint8_t sA[kBM][kBK + kPad];
  __shared__ __align__(16) uint8_t sB[kBN][kBK + kPad];
  const int m0 = static_cast<int>(blockIdx.y) * kBM;
  const int n0 = static_cast<int>(blockIdx.x) * kBN;
  const int tid = static_cast<int>(threadIdx.x);
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = warp >> 2, wn = warp & 3;
  const int g = lane >> 2, t = lane & 3;
  const int lrow = tid >> 1, lpart = (tid & 1) * 16;  // staging: row, 16-byte half
  int32_t acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[i][j][c] = 0;

  for (int k0 = 0; k0 < p.K; k0 += kBK) {
    const int am = m0 + lrow, bn = n0 + lrow;
    *reinterpret_cast<uint4*>(&sA[lrow][lpart]) =
        am < p.M ? load_k16(p.A + am * p.lda, k0 + lpart, p.K) : make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(&sB[lrow][lpart]) =
        bn < p.N ? load_k16(p.B + bn * p.ldb, k0 + lpart, p.K) : make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    uint32_t b[4][2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = wn * 32 + j * 8 + g;
      b[j][0] = *reinterpret_cast<const uint32_t*>(&sB[c][4 * t]);
      b[j][1] = *reinterpret_cast<const uint32_t*>(&sB[c][4 * t + 16]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = wm * 64 + i * 16 + g;
      const uint32_t a[4] = {*reinterpret_cast<const uint32_t*>(&sA[r][4 * t]),
                             *reinterpret_cast<const uint32_t*>(&sA[r + 8][4 * t]),
                             *reinterpret_cast<const uint32_t*>(&sA[r][4 * t + 16]),
                             *reinterpret_cast<const uint32_t*>(&sA[r + 8][4 * t + 16])};
#pragma unroll
      for (int j = 0; j < 4; ++j) mma_s8<kAS, kBS>(acc[i][j], a, b[j]);
    }
    __syncthreads();
  }

  // zero-point correction (mod 2^32) and requantisation
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = m0 + wm * 64 + i * 16 + g + 8 * h;
      if (row >= p.M) continue;
      const uint32_t za = static_cast<uint32_t>(p.zA_row ? p.zA_row[row] : p.zA);
      const uint32_t ra = static_cast<uint32_t>(p.rA[row]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int col = n0 + wn * 32 + j * 8 + 2 * t + e;
          if (col >= p.N) continue;
          const uint32_t zb = static_cast<uint32_t>(p.zB_col ? p.zB_col[col] : p.zB);
          const uint32_t cb = static_cast<uint32_t>(p.cB[col]);
          const uint32_t c = static_cast<uint32_t>(acc[i][j][2 * h + e]) - zb * ra - za * cb +
                             static_cast<uint32_t>(p.K) * za * zb;
          const int32_t c32 = static_cast<int32_t>(c);
          if (p.c32) p.c32[static_cast<long long>(row) * p.ldc32 + col] = c32;
          if (p.c8) {
            const float s = p.scale_col ? p.scale_col[col] : p.scale;
            const float f = __fmul_rn(__int2float_rn(c32), s);
            int32_t q;
            asm("cvt.rni.sat.s8.f32 %0, %1;" : "=r"(q) : "f"(f));
            p.c8[static_cast<long long>(row) * p.ldc8 + col] = static_cast<int8_t>(q);
          }
        }
      }
    }
  }
}

template <bool kAS, bool kBS>
int launch_gemm(const Params& p, cudaStream_t stream) {
  const dim3 grid((p.N + kBN - 1) / kBN, (p.M + kBM - 1) / kBM);
  imma_gemm_kernel<kAS, kBS><<<grid, kThreadsImma, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? IGC_OK : IGC_ERR_CUDA;
}

}  // namespace imma

// Called by gemm_s8_zp when the IMMA path is selected, after its argument and
// workspace checks (K >= 1, M, N >= 1, operands 16-byte aligned with row strides
// multiples of 16); rA / cB are int32[M] / int32[N] scratch in the workspace.
int imma_gemm_s8_zp(int M, int N, int K, const void* A, int a_signed, long long lda,
                    const void* Bt, int b_signed, long long ldb, int32_t zA,
                    const int32_t* zA_row, int32_t zB, const int32_t* zB_col, int32_t* C32,
                    long long ldc32, int8_t* C8, long long ldc8, float scale,
                    const float* scale_col, int32_t* rA, int32_t* cB, cudaStream_t stream) {
  if (M > 65535 * imma::kBM) return IGC_ERR_UNSUPPORTED;  // grid.y
  const auto* a = static_cast<const uint8_t*>(A);
  const auto* b = static_cast<const uint8_t*>(Bt);
  constexpr int kSumThreads = 256;  // 8 rows per block
  const unsigned ga = static_cast<unsigned>((static_cast<long long>(M) * 32 + kSumThreads - 1) /
                                            kSumThreads);
  const unsigned gb = static_cast<unsigned>((static_cast<long long>(N) * 32 + kSumThreads - 1) /
                                            kSumThreads);
  if (a_signed)
    imma::row_sums_kernel<true><<<ga, kSumThreads, 0, stream>>>(a, lda, M, K, rA);
  else
    imma::row_sums_kernel<false><<<ga, kSumThreads, 0, stream>>>(a, lda, M, K, rA);
  if (b_signed)
    imma::row_sums_kernel<true><<<gb, kSumThreads, 0, stream>>>(b, ldb, N, K, cB);
  else
    imma::row_sums_kernel<false><<<gb, kSumThreads, 0, stream>>>(b, ldb, N, K, cB);
  if (cudaGetLastError() != cudaSuccess) return IGC_ERR_CUDA;
  imma::Params p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.A = a;
  p.lda = lda;
  p.B = b;
  p.ldb = ldb;
  p.rA = rA;
  p.cB = cB;
  p.zA = zA;
  p.zA_row = zA_row;
  p.zB = zB;
  p.zB_col = zB_col;
  p.c32 = C32;
  p.ldc32 = ldc32;
  p.c8 = C8;
  p.ldc8 = ldc8;
  p.scale = scale;
  p.scale_col = scale_col;
  if (a_signed && b_signed) return imma::launch_gemm<true, true>(p, stream);
  if (a_signed) return imma::launch_gemm<true, false>(p, stream);
  if (b_signed) return imma::launch_gemm<false, true>(p, stream);
  return imma::launch_gemm<false, false>(p, stream);
}

}  // namespace igc
