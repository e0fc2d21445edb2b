// tc_gemm.h -- argument block of the tcgen05 GEMM (k_gemm.cu): the dense
// context prefill and the products of a batched draft (many sequences' slot
// rows sharing each weight read).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace fm {

enum TcEpi : int32_t {
  TC_EPI_FC = 0,      // c = acc (+ bias); C' = c * colw[n] (f16) and per-row partial sum of c^2 per 256 columns
  TC_EPI_KV = 1,      // row scale 1/rms, k_norm + RoPE on K heads, f16 stores into the head-major caches
  TC_EPI_F16 = 2,     // out16 = f16(act(acc + bias)), act = identity or exact GELU (out16 null: none);
                      // optionally out32 = acc + bias
  TC_EPI_GATED = 3,   // out32[row][n] = gate[n] * (acc + bias[n])   (a gated residual branch; treduce: +=)
  TC_EPI_SEGS = 4,    // out32: per-head RMSNorm + interleaved-pair RoPE on segments 0 / 1, plain elsewhere
  TC_EPI_ARGMAX = 5,  // per row, the best (value, lowest index) over the tile's columns < n_valid
};

struct TcGemmArgs {
  CUtensorMap tma_a;  // A [M][K] f16, box 64 x 128
  CUtensorMap tma_b;  // B [N][K] f16, box 64 x 256
  // tensor stores (tstore = 1; SEGS / GATED / F16 with a single output, when each CTA has one tile):
  // the epilogue writes its columns into shared memory in the 128-byte-swizzle layout and tensor
  // copies store them through this map of the output ([M][cols], f32 box 32 x 128 or f16 box
  // 64 x 128; rows past M are clipped).  With several tiles per CTA the plain stores run instead.
  CUtensorMap tma_o;
  int32_t tstore;
  // GATED with tstore: the tensor copies add the tile into out32 (the residual stream X += branch, one
  // addend per element) instead of storing it; without the staged path the epilogue adds in place
  int32_t treduce;
  int32_t M, N, K;
  int32_t epi;
  // tile order: groups of group_m consecutive 128-row blocks; inside a group
  // the row block runs fastest, so the CTAs in flight share B tiles while the
  // group's A panel stays in L2 (1: the column block runs fastest)
  int32_t group_m;
  int32_t *err;       // set to 1 when a bounded wait gives up
  int32_t a_row0;     // A rows start at this row of the map (rows past the map's extent read as zero)
  // split-K: each output tile is computed by a cluster of ksplit CTAs (1, 2 or
  // 4), one K slice each; the partial tiles are summed through distributed
  // shared memory in slice order (deterministic), slice s finishing its piece
  // of the columns (an FC output then has ksplit row-statistics entries per
  // 256 columns: st_ld = N / 256 * ksplit)
  int32_t ksplit;
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
  int32_t seg_cols;   // columns per K or V segment (= D); SEGS: columns per segment
  int32_t hd, max_ctx, start;
  const float2 *rope;
  float qk_eps;
  const __nv_bfloat16 *kn_w;  // [layers][hd]
  __half *cache;              // [layers][2][n_heads][max_ctx][hd] of one sequence
  size_t plane;               // elements of one [n_heads][max_ctx][hd] plane
  // per-row targets (KV, SEGS): position of row r = row_pos[r] (null: start + r);
  // KV: cache of row r = cache + row_seq[r] * seq_stride (null: cache)
  const int32_t *row_pos;
  const int32_t *row_seq;
  size_t seq_stride;
  // F16 / GATED / FC
  const __nv_bfloat16 *bias;  // [N] or null
  int32_t gelu;
  const float *gate;          // GATED: [N]
  // SEGS, GATED (and F16's optional f32 copy)
  float *out32;
  int32_t ldo32;
  const __nv_bfloat16 *nw0, *nw1;  // per-head norm weights [hd] of segments 0 and 1 (null: plain)
  // ARGMAX
  float2 *amax;               // [M][amax_ld]: (best value, index bits) per row and column block
  int32_t amax_ld;
  int32_t n_valid;            // columns < n_valid take part
};

bool make_tma_f16(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows);
// the output map of a tensor-store epilogue: [rows][cols] f32 (box 32 x 128) or f16 (box 64 x 128)
bool make_tma_out(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols, bool f32);
size_t tc_gemm_smem_bytes();
// column blocks of 256 (N must be a multiple of 256), row blocks of 128
inline int tc_gemm_tiles(int M, int N) { return ((M + 127) / 128) * (N / 256); }
cudaError_t launch_tc_gemm(const TcGemmArgs &a, int n_sm, cudaStream_t s);
cudaError_t launch_f32_to_f16(const float *in, __half *out, size_t n, int n_sm, cudaStream_t s);
cudaError_t launch_bf16_to_f16(const __nv_bfloat16 *in, __half *out, size_t n, cudaStream_t s);

}  // namespace fm
