// gemm_bf16: C = A * B with bf16 operands and fp32 accumulation on tcgen05 --
// the "f16 -> bf16" swap of the tensor intrinsic (page "TVM在CUDA GPU上跑GEMM的
// 全套张量化实现", §3.3), on the same kind::f16 pipe as gemm_f16 (§4.1 compute
// definition, §2.1 row.col operand forms).
#include "launch.cuh"

using namespace igc;

extern "C" int gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                         const void* Bt, int64_t ldb, void* C, int64_t ldc, int c_dtype,
                         float* C_f32_check, int64_t ldc32, igc_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (M < 0 || N < 0 || K < 0) return IGC_ERR_INVALID_ARG;
  if (c_dtype != IGC_F32 && c_dtype != IGC_BF16) return IGC_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return IGC_OK;  // empty output: nothing is read or written
  if (C == nullptr && C_f32_check == nullptr) return IGC_ERR_INVALID_ARG;
  if (C != nullptr && ldc < N) return IGC_ERR_INVALID_ARG;
  if (C_f32_check != nullptr && ldc32 < N) return IGC_ERR_INVALID_ARG;
  if (M > 0x7fffffff || N > 0x7fffffff || K > 0x7fffffff) return IGC_ERR_UNSUPPORTED;

  DeviceInfo dev;
  int rc = current_device(&dev);
  if (rc != IGC_OK) return rc;

  const size_t esize = c_dtype == IGC_BF16 ? 2 : 4;
  if (K == 0) {  // empty sum: C = 0 (A and Bt are not read and may be NULL)
    rc = zero_rows(C, ldc, M, N, esize, stream);
    if (rc == IGC_OK) rc = zero_rows(C_f32_check, ldc32, M, N, 4, stream);
    return rc;
  }
  if (A == nullptr || Bt == nullptr || lda < K || ldb < K) return IGC_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(Bt) || (lda % 8) != 0 || (ldb % 8) != 0)
    return IGC_ERR_MISALIGNED;

  CUtensorMap tmA;
  rc = encode_tiled_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, K, M, lda * 2, BK, BM_CTA);
  if (rc != IGC_OK) return rc;

  KParams p{};
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.num_kb = static_cast<int>((K + KS - 1) / KS);
  p.chunk_kb = p.num_kb;
  p.pf_a = static_cast<const char*>(A);
  p.pf_lda = lda * 2;
  p.out = C;
  p.ldo = ldc;
  p.out_type = c_dtype == IGC_BF16 ? kOutBF16 : kOutF32;
  p.out_f32 = C_f32_check;
  p.ldo32 = ldc32;
  p.vec_ok = vec_store_ok(C, ldc, esize) && vec_store_ok(C_f32_check, ldc32, 4);
  OutMaps om;
  add_out_map(om, 0, c_dtype == IGC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
              C, ldc, M, N, esize);
  add_out_map(om, 1, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C_f32_check, ldc32, M, N, 4);
  return launch_auto_bn<Mode::GemmBF16>(dev, tmA, Bt, K, N, ldb * 2, om, p, stream);
}
