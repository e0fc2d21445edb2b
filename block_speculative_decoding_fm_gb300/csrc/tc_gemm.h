// tc_gemm.h -- argument block of the tcgen05 prefill GEMM (k_gemm.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace fm {

enum TcEpi : int32_t {
  TC_EPI_FC = 0,  // C' = c * colw[n] (f16) and per-row partial sum of c^2 per 256-column block
  TC_EPI_KV = 1,  // row scale 1/rms, k_norm + RoPE on K heads, f16 stores into the head-major caches
};

struct TcGemmArgs {
  CUtensorMap tma_a;  // A [M][K] f16, box 64 x 128
  CUtensorMap tma_b;  // B [N][K] f16, box 64 x 256
  int32_t M, N, K;
  int32_t epi;
  // tile order: groups of group_m consecutive 128-row blocks; inside a group
  // the row block runs fastest, so the CTAs in flight share B tiles while the
  // group's A panel stays in L2 (1: the column block runs fastest)
  int32_t group_m;
  int32_t *err;       // set to 1 when a bounded wait gives up
  // FC
  const __nv_bfloat16 *colw;
  __half *out16;
  int32_t ldo;
  float *row_st;      // [M][st_ld]
  int32_t st_ld;
  // KV
  const float *in_st; // [M][in_st_n] partial sums of squares of the fc output
  int32_t in_st_n;
  float eps, inv_n;
  int32_t seg_cols;   // columns per K or V segment (= D)
  int32_t hd, max_ctx, start;
  const float2 *rope;
  float qk_eps;
  const __nv_bfloat16 *kn_w;  // [layers][hd]
  __half *cache;              // [layers][2][n_heads][max_ctx][hd] of one sequence
  size_t plane;               // elements of one [n_heads][max_ctx][hd] plane
};

bool make_tma_f16(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows);
size_t tc_gemm_smem_bytes();
cudaError_t launch_tc_gemm(const TcGemmArgs &a, int n_sm, cudaStream_t s);
cudaError_t launch_f32_to_f16(const float *in, __half *out, size_t n, int n_sm, cudaStream_t s);
cudaError_t launch_bf16_to_f16(const __nv_bfloat16 *in, __half *out, size_t n, cudaStream_t s);

}  // namespace fm
