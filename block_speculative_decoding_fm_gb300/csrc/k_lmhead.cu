// k_lmhead.cu -- lm_head over the tied token table fused with the per-row
// argmax: tok[t] = argmax_v sum_k Y[t][k] E[v][k]   (ties -> lowest v).
//
// The pages run the 16 slots through the target's token-table matvec and a
// separate argmaxRows pass (flashmap_drafter.js ``draft``; the table is Q8_0 in
// the GGUF block format the MTP loader on ternary_bonsai_2_mtp.js repacks into
// an int8 plane and a scale plane).  Here one persistent kernel streams the
// table once: each CTA keeps Y (split into hi + lo 16-bit halves) resident in
// shared memory, a producer warp streams 128-row x 64-column table chunks with
// 1-D bulk TMA copies into an mbarrier ring, consumer warps run the
// products on the tensor cores (Q8_0: int8 -> f16 exactly, per-32 block
// partial sums scaled by the block's f16 scale; bf16: directly), and keeps a
// running (value, index) best per row in registers.  The logits never reach
// memory; pass two is the last CTA reducing the per-CTA bests.
#include "dev_common.cuh"
#include "fm_internal.h"

namespace fm {

namespace {

constexpr int kThreads = 256;        // consumer warps 0..7
constexpr int kAll = kThreads + 32;  // + the producer warp
constexpr int kChunk = 64;
constexpr int kBfStage = kTile * kChunk * 2;

__host__ __device__ constexpr int lm_stage_bytes(bool q8) { return q8 ? kQ8Chunk : kBfStage; }

}  // namespace

template <bool Q8>
__global__ void __launch_bounds__(kAll, 1) lmhead_kernel(const __grid_constant__ LmArgs a, const int S) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int SB = lm_stage_bytes(Q8);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int H = a.H;
  const int lda = H + 32;  // 16-bit elements per A row (64-byte pad)
  const uint32_t ring = smem_u32(smem);
  const uint32_t ahi = ring + S * SB, alo = ahi + 16 * lda * 2;
  const uint32_t bars = alo + 16 * lda * 2;
  auto full = [&](int i) { return bars + 8 * i; };
  auto empty = [&](int i) { return bars + 8 * (S + i); };

  const int n_tiles = (a.V + kTile - 1) / kTile;
  const int kcs = H / kChunk;
  const int my_tiles = blockIdx.x < n_tiles ? (n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int total = my_tiles * kcs;
  const uint8_t *table = Q8 ? a.q8 : a.wb;
  auto src_of = [&](int c) {
    const int tile = blockIdx.x + (c / kcs) * gridDim.x;
    return table + ((size_t)tile * kcs + (c % kcs)) * SB;
  };

  if (threadIdx.x == kThreads) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), kThreads / 32);
    }
    mbar_fence_init();
    // the table does not depend on earlier kernels
    for (int c = 0; c < S && c < total; ++c) {
      mbar_expect_tx(full(c), SB);
      bulk_g2s(ring + c * SB, src_of(c), SB, full(c));
    }
  }
  pdl_trigger();
  __syncthreads();
  pdl_wait();
  const int T = a.T_const > 0 ? a.T_const : a.sp->T;

  float bv[2] = {-INFINITY, -INFINITY};  // running best for rows g and g + 8
  int bi[2] = {0x7fffffff, 0x7fffffff};
  if (w == kThreads / 32) {
    if (lane == 0) {
      for (int c = S; c < total; ++c) {
        const int st = c % S;
        if (!mbar_wait_bounded(empty(st), (c / S - 1) & 1, a.err)) break;
        mbar_expect_tx(full(st), SB);
        bulk_g2s(ring + st * SB, src_of(c), SB, full(st));
      }
    }
  } else {
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
    named_sync(1, kThreads);

    float acc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    // per-thread shared-memory offsets that do not change from chunk to chunk
    uint32_t woff[2][2], soff[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int r = 16 * w + 8 * j + g;
      if (Q8) {
        woff[j][0] = q8_slot(r, 8 * q);        // block 0: columns 8q .. 8q+7
        woff[j][1] = q8_slot(r, 32 + 8 * q);   // block 1
      } else {
        woff[j][0] = r * 128 + ((q ^ ((r & 1) << 2)) << 4);
        woff[j][1] = r * 128 + (((4 + q) ^ ((r & 1) << 2)) << 4);
      }
      soff[j] = kTile * kChunk + (16 * w + 8 * j + 2 * q) * 2;
    }
    bool ok = true;
    int tile = blockIdx.x, kc = 0;
    for (int c = 0; c < total; ++c) {
      const int st = c % S;
      if (ok && !mbar_wait_bounded(full(st), (c / S) & 1, a.err)) ok = false;
      const uint32_t buf = ring + st * SB;
      if (ok) {
        if (Q8) {
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            const uint32_t ar0 = (uint32_t)(g * lda + kc * kChunk + 32 * b + 8 * q) * 2;
            const uint32_t ar1 = ar0 + 8 * lda * 2;
            const uint4 h0 = lds128(ahi + ar0), h1 = lds128(ahi + ar1);
            const uint4 l0 = lds128(alo + ar0), l1 = lds128(alo + ar1);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const uint2 raw = lds64(buf + woff[j][b]);
              uint32_t wq[4];
              i8x4_to_f16x4(raw.x, wq[0], wq[1]);
              i8x4_to_f16x4(raw.y, wq[2], wq[3]);
              // four independent products (k16 step x hi / lo), summed after
              float p[4][4];
#pragma unroll
              for (int u = 0; u < 4; ++u) p[u][0] = p[u][1] = p[u][2] = p[u][3] = 0.f;
              mma_f16(p[0], word(h0, 0), word(h1, 0), word(h0, 1), word(h1, 1), wq[0], wq[1]);
              mma_f16(p[1], word(h0, 2), word(h1, 2), word(h0, 3), word(h1, 3), wq[2], wq[3]);
              mma_f16(p[2], word(l0, 0), word(l1, 0), word(l0, 1), word(l1, 1), wq[0], wq[1]);
              mma_f16(p[3], word(l0, 2), word(l1, 2), word(l0, 3), word(l1, 3), wq[2], wq[3]);
              const uint32_t sw = lds32(buf + soff[j] + b * 256);
              const __half2 d2 = *reinterpret_cast<const __half2 *>(&sw);
              const float d0 = __low2float(d2), d1 = __high2float(d2);
              acc[j][0] += d0 * ((p[0][0] + p[1][0]) + (p[2][0] + p[3][0]));
              acc[j][1] += d1 * ((p[0][1] + p[1][1]) + (p[2][1] + p[3][1]));
              acc[j][2] += d0 * ((p[0][2] + p[1][2]) + (p[2][2] + p[3][2]));
              acc[j][3] += d1 * ((p[0][3] + p[1][3]) + (p[2][3] + p[3][3]));
            }
          }
        } else {
          uint4 blo[2], bhi[2];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            blo[j] = lds128(buf + woff[j][0]);
            bhi[j] = lds128(buf + woff[j][1]);
          }
          const uint32_t r0 = (uint32_t)(g * lda + kc * kChunk + 8 * q) * 2, r1 = r0 + 8 * lda * 2;
          const uint4 h0 = lds128(ahi + r0), h1 = lds128(ahi + r1), h2 = lds128(ahi + r0 + 64),
                      h3 = lds128(ahi + r1 + 64);
          const uint4 l0 = lds128(alo + r0), l1 = lds128(alo + r1), l2 = lds128(alo + r0 + 64),
                      l3 = lds128(alo + r1 + 64);
          float p[2][4][4];
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int u = 0; u < 4; ++u) p[j][u][0] = p[j][u][1] = p[j][u][2] = p[j][u][3] = 0.f;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int ch = (jj & 1) * 2;
              mma_bf16(p[j][ch], word(h0, jj), word(h1, jj), word(h2, jj), word(h3, jj), word(blo[j], jj),
                       word(bhi[j], jj));
              mma_bf16(p[j][ch + 1], word(l0, jj), word(l1, jj), word(l2, jj), word(l3, jj), word(blo[j], jj),
                       word(bhi[j], jj));
            }
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[j][e] += (p[j][0][e] + p[j][2][e]) + (p[j][1][e] + p[j][3][e]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(st));
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
        kc = 0;
        tile += gridDim.x;
      } else {
        ++kc;
      }
    }
    // per-warp best: across the 4 lanes of a row
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv[h], o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi[h], o);
        if (better(ov, oi, bv[h], bi[h])) { bv[h] = ov; bi[h] = oi; }
      }
  }
  __shared__ float s_v[8][16];
  __shared__ int s_i[8][16];
  __shared__ int s_last;
  if (w < kThreads / 32 && q == 0) {
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
  const size_t a_bytes = 2 * 16 * (size_t)(a.H + 32) * 2;
  const size_t budget = 227 * 1024 - a_bytes - 1024;
  const size_t sb = lm_stage_bytes(q8);
  int S = (int)(budget / (sb + 16));
  if (S > 16) S = 16;
  if (S < 2) return cudaErrorInvalidValue;
  const size_t smem = (size_t)S * sb + a_bytes + 16 * S;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kAll, 1, 1);
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
    return cudaLaunchKernelEx(&cfg, lmhead_kernel<true>, a, S);
  }
  e = cudaFuncSetAttribute(lmhead_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, lmhead_kernel<false>, a, S);
}

}  // namespace fm
