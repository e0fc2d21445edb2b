// k_lmhead.cu -- lm_head over the tied token table fused with the per-row
// argmax: tok[t] = argmax_v sum_k Y[t][k] E[v][k]   (ties -> lowest v).
//
// The pages run the 16 slots through the target's token-table matvec and a
// separate argmaxRows pass (flashmap_drafter.js ``draft``; the table is Q8_0 in
// the GGUF block format the MTP loader on ternary_bonsai_2_mtp.js repacks into
// an int8 plane and a scale plane).  Here one persistent kernel streams the
// table once: each CTA keeps Y (split into hi + lo 16-bit halves) resident in
// shared memory, walks 128-row vocab tiles through a cp.async ring, runs the
// products on the tensor cores (Q8_0: int8 -> f16 exactly, per-32 block
// partial sums scaled by the block's f16 scale; bf16: directly), and keeps a
// running (value, index) best per row in registers.  The logits never reach
// memory; pass two is the last CTA reducing the per-CTA bests.
#include "dev_common.cuh"
#include "fm_internal.h"

namespace fm {

namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 64;
constexpr int kQ8Stage = kTile * kChunk + 2 * kTile * 2;  // int8 tile + 2 blocks of scales
constexpr int kBfStage = kTile * kChunk * 2;
constexpr int kQ8Stages = 6;
constexpr int kBfStages = 3;

__device__ __forceinline__ uint32_t wslot_bf(int r, int u) { return r * 128 + ((u ^ ((r & 1) << 2)) << 4); }
// int8 tile row r: 64 bytes = 4 pieces of 16; swap pieces 0/1 with 2/3 on rows with bit 1 set
__device__ __forceinline__ uint32_t q8slot(int r, int piece) { return r * 64 + ((piece ^ (((r >> 1) & 1) << 1)) << 4); }

template <bool Q8>
__device__ __forceinline__ void issue(const LmArgs &a, uint32_t buf, int tile, int kc) {
  if (Q8) {
    // 128 rows x 4 pieces of int8, then 2 blocks x 128 scales (32 pieces)
    for (int i = threadIdx.x; i < kTile * 4 + 32; i += kThreads) {
      if (i < kTile * 4) {
        const int r = i >> 2, p = i & 3;
        const int8_t *src = a.q8 + (size_t)(tile * kTile + r) * a.H + kc * kChunk + p * 16;
        cp_async16(buf + q8slot(r, p), src, 16u);
      } else {
        const int j = i - kTile * 4;  // 0..31: block j / 16, piece j % 16
        const int b = j >> 4, p = j & 15;
        const __half *src = a.q8s + ((size_t)tile * (a.H >> 5) + kc * 2 + b) * kTile + p * 8;
        cp_async16(buf + kTile * kChunk + b * 256 + p * 16, src, 16u);
      }
    }
  } else {
    for (int i = threadIdx.x; i < kTile * 8; i += kThreads) {
      const int r = i >> 3, u = i & 7;
      const int v = tile * kTile + r;
      const bool ok = v < a.V;
      const __nv_bfloat16 *src = a.wb + (size_t)(ok ? v : 0) * a.H + kc * kChunk + u * 8;
      cp_async16(buf + wslot_bf(r, u), src, ok ? 16u : 0u);
    }
  }
}

}  // namespace

template <bool Q8>
__global__ void __launch_bounds__(kThreads, 1) lmhead_kernel(const __grid_constant__ LmArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int S = Q8 ? kQ8Stages : kBfStages;
  constexpr int SB = Q8 ? kQ8Stage : kBfStage;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int H = a.H;
  const int lda = H + 32;  // 16-bit elements per A row (64-byte pad)
  const uint32_t ring = smem_u32(smem);
  const uint32_t ahi = ring + S * SB, alo = ahi + 16 * lda * 2;

  const int n_tiles = (a.V + kTile - 1) / kTile;
  const int kcs = H / kChunk;
  const int my_tiles = blockIdx.x < n_tiles ? (n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int total = my_tiles * kcs;

  // the table does not depend on earlier kernels
#pragma unroll
  for (int c = 0; c < S - 1; ++c) {
    if (c < total) issue<Q8>(a, ring + c * SB, blockIdx.x + (c / kcs) * gridDim.x, c % kcs);
    cp_async_commit();
  }
  pdl_trigger();
  pdl_wait();
  const int T = a.T_const > 0 ? a.T_const : a.sp->T;

  // Y -> 16-bit hi / lo, rows >= T zero
  for (int i = threadIdx.x; i < 16 * (H >> 2); i += kThreads) {
    const int t = i / (H >> 2), k = (i - t * (H >> 2)) * 4;
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < T) y = __ldcg(reinterpret_cast<const float4 *>(a.Y + (size_t)t * a.ldy + k));
    const float v[4] = {y.x, y.y, y.z, y.w};
    uint32_t hw[2], lw[2];
    if (Q8) {
      __half h[4], l[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) split_f16(v[e], h[e], l[e]);
      hw[0] = pack_f16(h[0], h[1]); hw[1] = pack_f16(h[2], h[3]);
      lw[0] = pack_f16(l[0], l[1]); lw[1] = pack_f16(l[2], l[3]);
    } else {
      __nv_bfloat16 h[4], l[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) split_bf16(v[e], h[e], l[e]);
      hw[0] = pack_bf16(h[0], h[1]); hw[1] = pack_bf16(h[2], h[3]);
      lw[0] = pack_bf16(l[0], l[1]); lw[1] = pack_bf16(l[2], l[3]);
    }
    const uint32_t off = (uint32_t)(t * lda + k) * 2;
    asm volatile("st.shared.v2.u32 [%0], {%1,%2};\n" ::"r"(ahi + off), "r"(hw[0]), "r"(hw[1]));
    asm volatile("st.shared.v2.u32 [%0], {%1,%2};\n" ::"r"(alo + off), "r"(lw[0]), "r"(lw[1]));
  }

  float acc[2][4];
  float bv[2] = {-INFINITY, -INFINITY};  // running best for rows g and g + 8
  int bi[2] = {0x7fffffff, 0x7fffffff};
#pragma unroll
  for (int j = 0; j < 2; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

  for (int c = 0; c < total; ++c) {
    const int tile = blockIdx.x + (c / kcs) * gridDim.x;
    const int kc = c % kcs;
    if (c + S - 1 < total) {
      const int cn = c + S - 1;
      issue<Q8>(a, ring + (cn % S) * SB, blockIdx.x + (cn / kcs) * gridDim.x, cn % kcs);
    }
    cp_async_commit();
    cp_async_wait<S - 1>();
    __syncthreads();
    const uint32_t buf = ring + (c % S) * SB;
    if (Q8) {
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const uint32_t ar0 = (uint32_t)(g * lda + kc * kChunk + 32 * b + 8 * q) * 2;
        const uint32_t ar1 = ar0 + 8 * lda * 2;
        const uint4 h0 = lds128(ahi + ar0), h1 = lds128(ahi + ar1);
        const uint4 l0 = lds128(alo + ar0), l1 = lds128(alo + ar1);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int r = 16 * w + 8 * j + g;
          const int u = 4 * b + q;  // 8-byte unit inside the row
          const uint2 raw = lds64(buf + q8slot(r, u >> 1) + (u & 1) * 8);
          uint32_t wq[4];
          i8x4_to_f16x4(raw.x, wq[0], wq[1]);
          i8x4_to_f16x4(raw.y, wq[2], wq[3]);
          float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            mma_f16(p, word(h0, 2 * jj), word(h1, 2 * jj), word(h0, 2 * jj + 1), word(h1, 2 * jj + 1),
                    wq[2 * jj], wq[2 * jj + 1]);
            mma_f16(p, word(l0, 2 * jj), word(l1, 2 * jj), word(l0, 2 * jj + 1), word(l1, 2 * jj + 1),
                    wq[2 * jj], wq[2 * jj + 1]);
          }
          const uint32_t sw = lds32(buf + kTile * kChunk + b * 256 + (16 * w + 8 * j + 2 * q) * 2);
          const __half2 d2 = *reinterpret_cast<const __half2 *>(&sw);
          const float d0 = __low2float(d2), d1 = __high2float(d2);
          acc[j][0] += d0 * p[0];
          acc[j][1] += d1 * p[1];
          acc[j][2] += d0 * p[2];
          acc[j][3] += d1 * p[3];
        }
      }
    } else {
      uint4 blo[2], bhi[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = 16 * w + 8 * j + g;
        blo[j] = lds128(buf + wslot_bf(r, q));
        bhi[j] = lds128(buf + wslot_bf(r, 4 + q));
      }
      const uint32_t r0 = (uint32_t)(g * lda + kc * kChunk + 8 * q) * 2, r1 = r0 + 8 * lda * 2;
      const uint4 h0 = lds128(ahi + r0), h1 = lds128(ahi + r1), h2 = lds128(ahi + r0 + 64), h3 = lds128(ahi + r1 + 64);
      const uint4 l0 = lds128(alo + r0), l1 = lds128(alo + r1), l2 = lds128(alo + r0 + 64), l3 = lds128(alo + r1 + 64);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          mma_bf16(acc[j], word(h0, jj), word(h1, jj), word(h2, jj), word(h3, jj), word(blo[j], jj), word(bhi[j], jj));
          mma_bf16(acc[j], word(l0, jj), word(l1, jj), word(l2, jj), word(l3, jj), word(blo[j], jj), word(bhi[j], jj));
        }
    }
    if (kc == kcs - 1) {
      // tile finished: fold into the running best, optionally store the logits
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int v = tile * kTile + 16 * w + 8 * j + 2 * q + (e & 1);
          const int row = g + 8 * (e >> 1);
          if (v < a.V && row < T) {
            if (a.logits) a.logits[(size_t)row * a.V + v] = acc[j][e];
            if (better(acc[j][e], v, bv[e >> 1], bi[e >> 1])) {
              bv[e >> 1] = acc[j][e];
              bi[e >> 1] = v;
            }
          }
          acc[j][e] = 0.f;
        }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  // per-CTA best: across the 4 lanes of a row, then across the 8 warps
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv[h], o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi[h], o);
      if (better(ov, oi, bv[h], bi[h])) { bv[h] = ov; bi[h] = oi; }
    }
  __shared__ float s_v[8][16];
  __shared__ int s_i[8][16];
  __shared__ int s_last;
  if (q == 0) {
    s_v[w][g] = bv[0]; s_i[w][g] = bi[0];
    s_v[w][g + 8] = bv[1]; s_i[w][g + 8] = bi[1];
  }
  __syncthreads();
  if (threadIdx.x < 16) {
    const int t = threadIdx.x;
    float v = s_v[0][t];
    int i = s_i[0][t];
    for (int ww = 1; ww < 8; ++ww)
      if (better(s_v[ww][t], s_i[ww][t], v, i)) { v = s_v[ww][t]; i = s_i[ww][t]; }
    __stcg(a.part + blockIdx.x * kMaxT + t, make_float2(v, __int_as_float(i)));
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atomicAdd(a.ticket, 1);
    s_last = old == (int)gridDim.x - 1;
    if (s_last) atomicExch(a.ticket, 0);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x < T) {
    const int t = threadIdx.x;
    float v = -INFINITY;
    int i = 0x7fffffff;
    for (int b = 0; b < (int)gridDim.x; ++b) {
      const float2 p = __ldcg(a.part + b * kMaxT + t);
      const int pi = __float_as_int(p.y);
      if (better(p.x, pi, v, i)) { v = p.x; i = pi; }
    }
    int32_t *out = a.tokens ? a.tokens : a.sp->tokens;
    out[t] = i == 0x7fffffff ? -1 : i;
  }
}

int lmhead_grid(const LmArgs &a, int n_sm) {
  const int n_tiles = (a.V + kTile - 1) / kTile;
  return n_tiles < n_sm ? n_tiles : n_sm;
}

cudaError_t launch_lmhead(const LmArgs &a, int grid, cudaStream_t st, bool pdl) {
  const bool q8 = a.q8 != nullptr;
  const size_t smem = (size_t)(q8 ? kQ8Stages * kQ8Stage : kBfStages * kBfStage) + 2 * 16 * (size_t)(a.H + 32) * 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e;
  if (q8) {
    e = cudaFuncSetAttribute(lmhead_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, lmhead_kernel<true>, a);
  }
  e = cudaFuncSetAttribute(lmhead_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, lmhead_kernel<false>, a);
}

}  // namespace fm
