// k_gemm.cu -- dense products on the 5th-generation tensor cores:
// D[m][n] = sum_k A[m][k] B[n][k] with A the activation rows (f16) and B a
// weight matrix (f16 copy of the bf16 weights, or of the token table), both
// K-major.  Two callers: the context-injection prefill (thousands of feature
// rows) and the batched draft, where the slot rows of many sequences share
// each weight read.
//
// The page runs these products as a 16 x 16 tiled WGSL GEMM (flashmap_drafter.js,
// ``gemmBf16`` via ``runGemm`` for more than 17 rows).  Here it is a persistent,
// warp-specialised sm_103a kernel:
//   warp 0      one thread issues TMA (cp.async.bulk.tensor) loads of 128 x 64
//               A tiles and 256 x 64 B tiles (128-byte swizzle) into a 4-stage
//               shared-memory ring guarded by mbarriers;
//   warp 1      allocates 512 TMEM columns (two 128 x 256 f32 accumulators) and
//               runs the issue loop warp-wide, an elected lane issuing
//               tcgen05.mma (kind::f16, M 128, N 256, K 16);
//               tcgen05.commit frees ring stages and publishes accumulators;
//   warps 2..9  read an accumulator with tcgen05.ld (two threads per row, one
//               half of the columns each) while the next tile accumulates into
//               the other buffer, and run the fused epilogue:
//                 FC:     C' = (c + bias) * norm_w[n] -> f16 and per-row partial
//                         sum of squares (the RMSNorm that follows fc);
//                 KV:     row scale 1/rms(c), per-head RMSNorm (k_norm) and
//                         interleaved-pair RoPE on K heads, f16 stores into the
//                         head-major caches of every layer at the row's
//                         sequence and position;
//                 F16:    bias (+ exact GELU) -> f16, the next product's operand;
//                 GATED:  gate * (c + bias), a gated residual branch, f32 out;
//                 SEGS:   per-head RMSNorm + RoPE of q / k heads, f32 out;
//                 ARGMAX: per row, the largest logit of the tile (lowest index
//                         on ties), for the lm_head.
// Split-K: a tile's K blocks can be dealt to a cluster of 2 or 4 CTAs; each
// stores its partial tile into its own shared memory, and after a cluster
// barrier each sums its piece of the columns over every slice (distributed
// shared memory, slice order) and runs the epilogue on that piece.
// Every mbarrier wait is bounded by a clock budget; on expiry the kernel sets
// an error flag, drains, frees its TMEM and returns.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "dev_common.cuh"
#include "fm_internal.h"
#include "tc_gemm.h"

namespace fm {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, ST = 4;
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE = A_BYTES + B_BYTES;
// Epilogue warps: 4 (one per TMEM lane quarter) or 8 (two per quarter, each
// row's columns in two halves) -- the launch picks 8 when every CTA has a
// single tile, whose epilogue is then not hidden behind a next tile's MMAs.
__device__ __forceinline__ int n_epi() { return (int)blockDim.x - 64; }   // epilogue threads
__device__ __forceinline__ int n_halves() { return ((int)blockDim.x - 64) >> 7; }
constexpr long long kWaitBudget = 4000000000LL;  // clock cycles (~2 s) before a wait gives up

// bounded wait; honor_err = false keeps waiting (by time only) after another role gave up
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t *err, bool honor_err = true) {
  if (honor_err) return mbar_wait_bounded(bar, parity, err);
  if (mbar_try(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try(bar, parity)) {
    if (clock64() - t0 > kWaitBudget) {
      atomicExch(err, 1);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// K-major operand, 128-byte swizzle: rows of 128 bytes, 8-row atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;            // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: next 8-row atom
  d |= (uint64_t)1 << 46;            // descriptor version for sm_100 family
  d |= (uint64_t)2 << 61;            // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: D f32, A/B f16, both K-major, M 128, N 256
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

#define FM_TLD32(taddr, v)                                                                                          \
  asm volatile(                                                                                                     \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19," \
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"                                                  \
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),           \
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),       \
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),     \
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])      \
      : "r"(taddr))

__device__ __forceinline__ void tld32(uint32_t taddr, float (&f)[32]) {
  uint32_t v[32];
  FM_TLD32(taddr, v);
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
}


__device__ __forceinline__ void store_h8(__half *dst, const float *v) {
  uint4 pk;
  __half2 h0 = __floats2half2_rn(v[0], v[1]), h1 = __floats2half2_rn(v[2], v[3]);
  __half2 h2 = __floats2half2_rn(v[4], v[5]), h3 = __floats2half2_rn(v[6], v[7]);
  pk.x = *reinterpret_cast<uint32_t *>(&h0);
  pk.y = *reinterpret_cast<uint32_t *>(&h1);
  pk.z = *reinterpret_cast<uint32_t *>(&h2);
  pk.w = *reinterpret_cast<uint32_t *>(&h3);
  *reinterpret_cast<uint4 *>(dst) = pk;
}

__device__ __forceinline__ void store_f32x32(float *dst, const float *v) {
#pragma unroll
  for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4 *>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
}
__device__ __forceinline__ void store_f16x32(__half *dst, const float *v) {
#pragma unroll
  for (int j = 0; j < 32; j += 8) store_h8(dst + j, v + j);
}

// Tensor-store staging: the epilogue's columns [c_lo, c_hi) as boxes of 128 rows x 128 bytes (32 f32 or
// 64 f16 columns, 16 KB each, one after another), each row's 16-byte units XOR-swizzled by (row & 7): the
// layout a 128-byte-swizzle tensor copy reads (box bases 1024-byte aligned).
constexpr int kBoxBytes = BM * 128;
__device__ __forceinline__ void stage_f32x32(uint8_t *stage, int rel, int rl, const float *v) {
  uint8_t *row = stage + (size_t)(rel >> 5) * kBoxBytes + rl * 128;
  const int sw = rl & 7;
#pragma unroll
  for (int u = 0; u < 8; ++u)
    *reinterpret_cast<float4 *>(row + ((u ^ sw) << 4)) = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
}
__device__ __forceinline__ void stage_f16x32(uint8_t *stage, int rel, int rl, const float *v) {
  uint8_t *row = stage + (size_t)(rel >> 6) * kBoxBytes + rl * 128;
  const int sw = rl & 7, u0 = (rel & 63) >> 3;   // these 32 columns are units u0 .. u0 + 3 of the row
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float *w = v + 8 * j;
    __half2 h0 = __floats2half2_rn(w[0], w[1]), h1 = __floats2half2_rn(w[2], w[3]);
    __half2 h2 = __floats2half2_rn(w[4], w[5]), h3 = __floats2half2_rn(w[6], w[7]);
    uint4 pk;
    pk.x = *reinterpret_cast<uint32_t *>(&h0);
    pk.y = *reinterpret_cast<uint32_t *>(&h1);
    pk.z = *reinterpret_cast<uint32_t *>(&h2);
    pk.w = *reinterpret_cast<uint32_t *>(&h3);
    *reinterpret_cast<uint4 *>(row + (((u0 + j) ^ sw) << 4)) = pk;
  }
}
__device__ __forceinline__ void tma_add_2d(const CUtensorMap *map, uint32_t src, int x, int y) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];\n" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];\n" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}

// Per-column operands of a tile (gate, bias, norm weight), staged once per tile
// in shared memory by the epilogue threads (one round trip for all of them),
// and the per-row values the two threads of a row exchange.
struct EpCols {
  float gate[BN], bias[BN], w[BN];
  float xs[2][BM];
  int xi[2][BM];
};

__device__ void stage_cols(const TcGemmArgs &a, EpCols *ep, int n0, int i) {
  named_sync(1, n_epi());   // the previous tile's epilogue has finished reading
  for (int k = i; k < BN; k += n_epi()) {
    const int n = n0 + k;
    float w = 1.f;
    if (a.epi == TC_EPI_FC) {
      w = __bfloat162float(a.colw[n]);
    } else if (a.epi == TC_EPI_SEGS) {
      const int seg = n / a.seg_cols;
      const __nv_bfloat16 *nw = seg == 0 ? a.nw0 : seg == 1 ? a.nw1 : nullptr;
      w = nw ? __bfloat162float(nw[n % a.hd]) : 1.f;
    } else if (a.epi == TC_EPI_KV) {
      w = __bfloat162float(a.kn_w[(size_t)((n / a.seg_cols) >> 1) * a.hd + n % a.hd]);
    }
    ep->gate[k] = a.gate ? a.gate[n] : 1.f;
    ep->bias[k] = a.bias ? __bfloat162float(a.bias[n]) : 0.f;
    ep->w[k] = w;
  }
  named_sync(1, n_epi());
}

// The two epilogue threads of a row (halves 0 and 1) add a per-row value, half 0's first.
__device__ __forceinline__ float pair_sum(EpCols *ep, int rl, int h, float v) {
  if (n_halves() == 1) return v;
  ep->xs[h][rl] = v;
  named_sync(1, n_epi());
  const float s = ep->xs[0][rl] + ep->xs[1][rl];
  named_sync(1, n_epi());
  return s;
}

// Each epilogue gets columns [c_lo, c_hi) of the tile (all of it, or the piece a
// K slice owns after the cluster reduction); the two threads of a row take one
// half each (h).

__device__ void epilogue_fc(const TcGemmArgs &a, EpCols *ep, uint32_t taddr, int rl, int h, int row, int n0,
                            int st_col, int c_lo, int c_hi) {
  float ss = 0.f;
  const bool live = row < a.M;
  const int w = (c_hi - c_lo) / n_halves();
  for (int c0 = c_lo + h * w; c0 < c_lo + (h + 1) * w; c0 += 32) {
    float v[32];
    tld32(taddr + c0, v);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      v[j] += ep->bias[c0 + j];
      ss += v[j] * v[j];
      v[j] *= ep->w[c0 + j];
    }
    if (live) store_f16x32(a.out16 + (size_t)row * a.ldo + n0 + c0, v);
  }
  ss = pair_sum(ep, rl, h, ss);
  if (live && h == 0) a.row_st[(size_t)row * a.st_ld + st_col] = ss;
}

// rotate the interleaved pairs of 32 channels; r: their 16 (cos, sin) pairs as 8 float4
__device__ __forceinline__ void rope32(float *v, const float4 (&r)[8]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 cs = r[q];
    const float a0 = v[4 * q], a1 = v[4 * q + 1], b0 = v[4 * q + 2], b1 = v[4 * q + 3];
    v[4 * q] = a0 * cs.x - a1 * cs.y;
    v[4 * q + 1] = a1 * cs.x + a0 * cs.y;
    v[4 * q + 2] = b0 * cs.z - b1 * cs.w;
    v[4 * q + 3] = b1 * cs.z + b0 * cs.w;
  }
}

// Per-head RMSNorm (weight by channel, from the staged columns; row scale rs
// first) and RoPE at position p of this thread's half of [c_lo, c_hi), then
// `emit(col, v)` for each 32-column chunk.  A half narrower than a head (a
// one-head piece) shares the head's sum of squares with the other half.  The
// RoPE pairs of the next chunk are requested while the current one is done.
template <typename Emit>
__device__ __forceinline__ void norm_rope_half(const TcGemmArgs &a, EpCols *ep, uint32_t taddr, int rl, int h,
                                               float rs, bool norm, int p, int c_lo, int c_hi, Emit &&emit) {
  const int hd = a.hd;
  const float4 *rrow = reinterpret_cast<const float4 *>(a.rope + (size_t)p * (hd >> 1));
  const int w = (c_hi - c_lo) / n_halves(), lo = c_lo + h * w, hi = lo + w;
  const bool shared_head = w < hd;   // then [c_lo, c_hi) is one head
  for (int h0 = shared_head ? c_lo : lo; h0 < (shared_head ? c_lo + 1 : hi); h0 += hd) {
    const int b0 = shared_head ? lo : h0, b1 = shared_head ? hi : h0 + hd;   // this thread's columns of the head
    float r2 = 1.f;
    if (norm) {
      float ss = 0.f;
      for (int c0 = b0; c0 < b1; c0 += 32) {
        float v[32];
        tld32(taddr + c0, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) ss += (v[j] * rs) * (v[j] * rs);
      }
      if (shared_head) ss = pair_sum(ep, rl, h, ss);
      r2 = rsqrtf(ss / (float)hd + a.qk_eps);
    }
    // chunks in pairs (this thread's columns of a head are a multiple of 64): pair members use
    // the register buffers ra / rb, the next chunk's pairs requested one chunk ahead
    float4 ra[8], rb[8];
    if (norm) {
#pragma unroll
      for (int q = 0; q < 8; ++q) ra[q] = __ldg(rrow + ((b0 - h0) >> 2) + q);
    }
    for (int c0 = b0; c0 < b1; c0 += 64) {
      if (norm) {
#pragma unroll
        for (int q = 0; q < 8; ++q) rb[q] = __ldg(rrow + ((c0 + 32 - h0) >> 2) + q);
      }
      {
        float v[32];
        tld32(taddr + c0, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= rs;
        if (norm) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = v[j] * r2 * ep->w[c0 + j];
          rope32(v, ra);
        }
        emit(c0, v);
      }
      if (norm && c0 + 64 < b1) {
#pragma unroll
        for (int q = 0; q < 8; ++q) ra[q] = __ldg(rrow + ((c0 + 64 - h0) >> 2) + q);
      }
      {
        float v[32];
        tld32(taddr + c0 + 32, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= rs;
        if (norm) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = v[j] * r2 * ep->w[c0 + 32 + j];
          rope32(v, rb);
        }
        emit(c0 + 32, v);
      }
    }
  }
}

__device__ void epilogue_kv(const TcGemmArgs &a, EpCols *ep, uint32_t taddr, int rl, int h, int row, int n0, int c_lo,
                            int c_hi) {
  const bool live = row < a.M;
  const int seg = n0 / a.seg_cols;
  const int layer = seg >> 1, kind = seg & 1;
  const int hd = a.hd;
  float rs = 1.f;
  if (live) {
    float s = 0.f;
    for (int i = 0; i < a.in_st_n; ++i) s += __ldcg(a.in_st + (size_t)row * a.in_st_n + i);
    rs = rsqrtf(s * a.inv_n + a.eps);
  }
  const int p = a.row_pos ? (live ? a.row_pos[row] : 0) : a.start + row;
  __half *cache = a.cache + (a.row_seq && live ? (size_t)a.row_seq[row] * a.seq_stride : 0) +
                  (size_t)(layer * 2 + kind) * a.plane + (size_t)p * hd;
  const int head0 = (n0 % a.seg_cols) / hd;
  norm_rope_half(a, ep, taddr, rl, h, rs, kind == 0, p, c_lo, c_hi, [&](int c0, const float *v) {
    if (live) store_f16x32(cache + (size_t)(head0 + c0 / hd) * a.max_ctx * hd + c0 % hd, v);
  });
}

// q / k / v rows: segment s = n / seg_cols; segments 0 and 1 take a per-head
// RMSNorm with their weight (when given) and RoPE at the row's position
__device__ void epilogue_segs(const TcGemmArgs &a, EpCols *ep, uint32_t taddr, int rl, int h, int row, int n0,
                              int c_lo, int c_hi, uint8_t *stage) {
  const bool live = row < a.M;
  const int seg = n0 / a.seg_cols;
  const bool norm = (seg == 0 && a.nw0) || (seg == 1 && a.nw1);
  const int p = live ? (a.row_pos ? a.row_pos[row] : a.start + row) : 0;
  float *out = a.out32 + (size_t)(live ? row : 0) * a.ldo32 + n0;
  norm_rope_half(a, ep, taddr, rl, h, 1.f, norm, p, c_lo, c_hi, [&](int c0, const float *v) {
    if (!live) return;
    if (stage)
      stage_f32x32(stage, c0 - c_lo, rl, v);
    else
      store_f32x32(out + c0, v);
  });
}

// F16: bias (+ exact GELU) -> f16; GATED: gate * (acc + bias) -> f32, the residual branch
// (treduce: added into out32, the residual stream, by the tensor reduce-add copies or in place)
__device__ void epilogue_f16(const TcGemmArgs &a, EpCols *ep, uint32_t taddr, int rl, int h, int row, int n0,
                             int c_lo, int c_hi, uint8_t *stage) {
  const bool live = row < a.M;
  const bool gated = a.epi == TC_EPI_GATED;
  const int w = (c_hi - c_lo) / n_halves();
  for (int c0 = c_lo + h * w; c0 < c_lo + (h + 1) * w; c0 += 32) {
    float v[32];
    tld32(taddr + c0, v);
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] += ep->bias[c0 + j];
    if (gated) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= ep->gate[c0 + j];
    }
    if (!live) continue;
    if (a.out32) {
      float *dst = a.out32 + (size_t)row * a.ldo32 + n0 + c0;
      if (stage) {   // a staged epilogue has this single output
        stage_f32x32(stage, c0 - c_lo, rl, v);
      } else {
        if (a.treduce) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] += __ldcg(dst + j);
        }
        store_f32x32(dst, v);
      }
    }
    if (!a.out16) continue;
    if (a.gelu) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = gelu_erf(v[j]);
    }
    if (stage)
      stage_f16x32(stage, c0 - c_lo, rl, v);
    else
      store_f16x32(a.out16 + (size_t)row * a.ldo + n0 + c0, v);
  }
}

__device__ void epilogue_argmax(const TcGemmArgs &a, EpCols *ep, uint32_t taddr, int rl, int h, int row, int n0,
                                int nb) {
  float best = -INFINITY;
  int bi = 0x7fffffff;
  const int hw = BN / n_halves();
  for (int c0 = h * hw; c0 < (h + 1) * hw; c0 += 32) {
    float v[32];
    tld32(taddr + c0, v);
#pragma unroll
    for (int j = 0; j < 32; ++j)   // ascending columns, strict '>': the lowest index wins a tie
      if (n0 + c0 + j < a.n_valid && v[j] > best) {
        best = v[j];
        bi = n0 + c0 + j;
      }
  }
  if (n_halves() == 1) {
    if (row < a.M) a.amax[(size_t)row * a.amax_ld + nb] = make_float2(best, __int_as_float(bi));
    return;
  }
  ep->xs[h][rl] = best;
  ep->xi[h][rl] = bi;
  named_sync(1, n_epi());
  if (h == 0 && row < a.M) {
    // the upper half's columns come later: it wins only with a strictly larger value
    const float b1 = ep->xs[1][rl];
    if (b1 > best) {
      best = b1;
      bi = ep->xi[1][rl];
    }
    a.amax[(size_t)row * a.amax_ld + nb] = make_float2(best, __int_as_float(bi));
  }
  named_sync(1, n_epi());
}

// Split-K partial tile in shared memory (the operand ring, idle once the MMAs
// are done): 8 chunk blocks of 128 rows x 32 f32, the 16-byte units of a row
// XOR-swizzled by (row & 7) so that a warp's accesses spread over the banks.
// Half h of the epilogue threads stores its share of the chunks.
__device__ __forceinline__ void store_partial(uint32_t taddr, int rl, int h, float *part) {
  const int sw = rl & 7, per = (BN / 32) / n_halves();
  for (int c = per * h; c < per * (h + 1); ++c) {
    float v[32];
    tld32(taddr + 32 * c, v);
    float *dst = part + ((size_t)c * BM + rl) * 32;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      *reinterpret_cast<float4 *>(dst + 4 * (u ^ sw)) = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
  }
}

// This half's columns of [c_lo, c_hi) summed over the cluster's K slices in
// slice order (deterministic), into TMEM.  Warp q reads its 32 rows of each
// slice's chunk block (4 KB, contiguous) with 512-byte instructions from the
// slices' shared memory (distributed shared memory serves contiguous reads far
// better than 32 rows' scattered 16-byte pieces), sums, and turns the sums back
// into one row per lane through its own block.
__device__ void reduce_piece(uint32_t taddr, int rl, int h, float *part, int ks, int c_lo, int c_hi) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int q = rl >> 5, l = rl & 31, sw = rl & 7;
  const int w = (c_hi - c_lo) / n_halves();
  for (int c = (c_lo + h * w) / 32; c < (c_lo + (h + 1) * w) / 32; ++c) {
    float4 acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    float *mine = part + ((size_t)c * BM + 32 * q) * 32;
    for (int s = 0; s < ks; ++s) {
      const float *src = cluster.map_shared_rank(mine, s);
      float4 t[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) t[i] = *reinterpret_cast<const float4 *>(src + (i * 32 + l) * 4);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        acc[i].x += t[i].x;
        acc[i].y += t[i].y;
        acc[i].z += t[i].z;
        acc[i].w += t[i].w;
      }
    }
    // this block is this CTA's own piece: no peer reads it
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i) *reinterpret_cast<float4 *>(mine + (i * 32 + l) * 4) = acc[i];
    __syncwarp();
    float v[32];
    const float *row = mine + (size_t)l * 32;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float4 t = *reinterpret_cast<const float4 *>(row + 4 * (u ^ sw));
      v[4 * u] = t.x;
      v[4 * u + 1] = t.y;
      v[4 * u + 2] = t.z;
      v[4 * u + 3] = t.w;
    }
    tmem_st32(taddr + 32 * c, v);
  }
}

// Column pieces a split tile's epilogue is dealt in: whole heads for the
// per-head norms, the whole tile for the argmax, else 256 / ks columns.
__device__ __forceinline__ int epilogue_pieces(const TcGemmArgs &a, int ks) {
  if (a.epi == TC_EPI_ARGMAX) return 1;
  if (a.epi == TC_EPI_KV || a.epi == TC_EPI_SEGS) return ks < BN / a.hd ? ks : BN / a.hd;
  return ks;
}

// staged: the tile's columns are already in shared memory (the CTA's first tile, staged
// before griddepcontrol.wait).  stage: the tensor-store staging area (null: plain stores);
// its boxes go out through a.tma_o once every epilogue thread has written its rows.
__device__ __forceinline__ void run_epilogue(const TcGemmArgs &a, EpCols *ep, uint32_t taddr, int rl, int h, int row,
                                             int nb, int st_col, int c_lo, int c_hi, bool staged, uint8_t *stage) {
  const int n0 = nb * BN;
  if (a.epi != TC_EPI_ARGMAX && !staged) stage_cols(a, ep, n0, (int)threadIdx.x - 64);
  if ((a.epi != TC_EPI_SEGS && a.epi != TC_EPI_F16 && a.epi != TC_EPI_GATED) || (a.out16 && a.out32)) stage = nullptr;
  switch (a.epi) {
    case TC_EPI_FC: epilogue_fc(a, ep, taddr, rl, h, row, n0, st_col, c_lo, c_hi); break;
    case TC_EPI_KV: epilogue_kv(a, ep, taddr, rl, h, row, n0, c_lo, c_hi); break;
    case TC_EPI_F16:
    case TC_EPI_GATED: epilogue_f16(a, ep, taddr, rl, h, row, n0, c_lo, c_hi, stage); break;
    case TC_EPI_SEGS: epilogue_segs(a, ep, taddr, rl, h, row, n0, c_lo, c_hi, stage); break;
    default: epilogue_argmax(a, ep, taddr, rl, h, row, n0, nb); break;
  }
  if (!stage) return;
  fence_proxy_async();            // the rows written above are visible to the tensor copies
  named_sync(1, n_epi());
  if (threadIdx.x == 64) {
    const int cols = a.out16 ? 64 : 32;   // per box
    for (int i = 0; i < (c_hi - c_lo) / cols; ++i) {
      const uint32_t src = smem_u32(stage + (size_t)i * kBoxBytes);
      if (a.treduce)
        tma_add_2d(&a.tma_o, src, n0 + c_lo + i * cols, row - rl);
      else
        tma_store_2d(&a.tma_o, src, n0 + c_lo + i * cols, row - rl);
    }
    asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
    asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");   // written before the CTA ends
  }
}

// tile -> (row block, column block) in the grouped order of TcGemmArgs::group_m
__device__ __forceinline__ void tile_coords(int tile, int n_mb, int n_nb, int gm_full, int &mb, int &nb) {
  const int per_group = gm_full * n_nb;
  const int g = tile / per_group, local = tile - g * per_group;
  const int gm = min(gm_full, n_mb - g * gm_full);
  mb = g * gm_full + local % gm;
  nb = local / gm;
}

}  // namespace

// NT: threads per CTA (192: 4 epilogue warps, 320: 8), the register budget follows
template <int NT>
__global__ void __launch_bounds__(NT, 1) fm_prefill_gemm_kernel(const __grid_constant__ TcGemmArgs a) {
  __builtin_assume(blockDim.x == NT);   // the epilogue's split into halves is known at compile time
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - smem_u32(smem_raw));
  const uint32_t bars = base + ST * STAGE;
  auto full = [&](int s) { return bars + 8 * s; };
  auto empty = [&](int s) { return bars + 8 * (ST + s); };
  auto tfull = [&](int b) { return bars + 8 * (2 * ST + b); };
  auto tempty = [&](int b) { return bars + 8 * (2 * ST + 2 + b); };
  const uint32_t tslot = bars + 8 * (2 * ST + 4);
  EpCols *ep = reinterpret_cast<EpCols *>(gbase + ST * STAGE + 256);   // the epilogue's staged columns
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull(b), 1);
      mbar_init(tempty(b), n_epi());
    }
    mbar_fence_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(tslot) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = lds32(tslot);

  pdl_trigger();

  const int n_nb = a.N / BN;
  const int n_mb = (a.M + BM - 1) / BM;
  const int n_tiles = n_mb * n_nb;
  const int gm = a.group_m > 0 ? a.group_m : 1;
  const int nk = a.K / BK;
  const int ks = a.ksplit > 1 ? a.ksplit : 1;
  const int n_units = n_tiles * ks;   // unit u: tile u / ks, K slice u % ks (slices of a tile adjacent)
  // Nothing an earlier kernel writes is read before griddepcontrol.wait: the producer requests its first
  // weight tiles first, the epilogue warps stage the first tile's per-column operands (weights) first.
  if (warp >= 2 && a.epi != TC_EPI_ARGMAX && (int)blockIdx.x < n_units) {
    int mb0, nb0;
    tile_coords(blockIdx.x / ks, n_mb, n_nb, gm, mb0, nb0);
    stage_cols(a, ep, nb0 * BN, (int)threadIdx.x - 64);
  }
  if (warp != 0) pdl_wait();
  auto kslice = [&](int slice, int &kb0, int &kb1) {
    kb0 = slice * nk / ks;
    kb1 = (slice + 1) * nk / ks;
  };

  if (warp == 0) {
    if (lane == 0) {
      // B (weights, or the token table) is never written by an earlier kernel: the first
      // unit's first stages request their B tiles before griddepcontrol.wait, their A
      // tiles (activations) after it
      int pre = 0;
      if ((int)blockIdx.x < n_units) {
        int mb, nb, kb0, kb1;
        tile_coords(blockIdx.x / ks, n_mb, n_nb, gm, mb, nb);
        kslice(blockIdx.x % ks, kb0, kb1);
        pre = kb1 - kb0 < ST ? kb1 - kb0 : ST;
        for (int j = 0; j < pre; ++j) {
          mbar_expect_tx(full(j), STAGE);
          tma_load_2d(base + j * STAGE + A_BYTES, &a.tma_b, (kb0 + j) * BK, nb * BN, full(j));
        }
      }
      pdl_wait();
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        int mb, nb, kb0, kb1;
        tile_coords(u / ks, n_mb, n_nb, gm, mb, nb);
        kslice(u % ks, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % ST;
          const uint32_t sa = base + s * STAGE, sb = sa + A_BYTES;
          if ((int)it < pre) {   // stage set up before the wait: only its A tile is missing
            tma_load_2d(sa, &a.tma_a, kb * BK, a.a_row0 + mb * BM, full(s));
            continue;
          }
          if (!mbar_wait(empty(s), ((it / ST) & 1) ^ 1, a.err)) { ok = false; break; }
          mbar_expect_tx(full(s), STAGE);
          tma_load_2d(sa, &a.tma_a, kb * BK, a.a_row0 + mb * BM, full(s));
          tma_load_2d(sb, &a.tma_b, kb * BK, nb * BN, full(s));
        }
      }
      // drain: the last stages issued must have landed before the CTA leaves
      for (uint32_t j = it > ST ? it - ST : 0; j < it; ++j) mbar_wait(full(j % ST), (j / ST) & 1, a.err, false);
    }
  } else if (warp == 1) {
    // the whole warp runs the issue loop (warp-uniform state); one elected lane
    // issues each MMA and commit, and every wait's verdict is made warp-uniform
    uint32_t it = 0, tc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++tc) {
      const int b = tc & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(tempty(b), ((tc >> 1) & 1) ^ 1, a.err))) break;
      tc_fence_after();
      const uint32_t d = tmem + b * BN;
      int kb0, kb1;
      kslice(u % ks, kb0, kb1);
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const int s = it % ST;
        if (!__all_sync(0xffffffffu, mbar_wait(full(s), (it / ST) & 1, a.err))) { ok = false; break; }
        tc_fence_after();
        const uint32_t sa = base + s * STAGE, sb = sa + A_BYTES;
        const uint64_t ad = sdesc(sa), bd = sdesc(sb);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          umma_ss_elect(d, ad + 2 * kk, bd + 2 * kk, kIdesc, (kb > kb0 || kk) ? 1u : 0u);
        umma_commit_elect(empty(s));
      }
      if (ok) umma_commit_elect(tfull(b));
    }
  } else {
    const int quad = warp & 3;  // TMEM lanes 32 * quad .. + 31 belong to this warp
    const int rl = quad * 32 + lane;
    const int half = (warp - 2) >> 2;   // the two warps of a lane quarter split the columns
    uint32_t tc = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++tc) {
      const int b = tc & 1;
      if (!mbar_wait(tfull(b), (tc >> 1) & 1, a.err)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + b * BN + ((uint32_t)(quad * 32) << 16);
      if (ks > 1) {
        // this slice's partial tile goes to the cluster reduction below
        store_partial(taddr, rl, half, reinterpret_cast<float *>(gbase));
        continue;
      }
      int mb, nb;
      tile_coords(u, n_mb, n_nb, gm, mb, nb);
      // one tile per CTA: the operand ring is idle once its MMAs are done and stages the tensor stores
      uint8_t *stage = a.tstore && (int)gridDim.x >= n_units ? gbase : nullptr;
      run_epilogue(a, ep, taddr, rl, half, mb * BM + rl, nb, nb, 0, BN, tc == 0, stage);
      tc_fence_before();
      mbar_arrive(tempty(b));
    }
  }
  if (ks > 1) {
    // Split-K over a cluster of the tile's ks slices (one unit per CTA): every
    // slice's partial is in its shared memory; slice s sums its piece of the
    // columns over all slices (slice order) and runs the epilogue there.
    __syncwarp();
    cluster_arrive_release();
    cluster_wait_acquire();
    const int u = blockIdx.x, slice = u % ks;
    if (warp >= 2 && u < n_units) {
      const int quad = warp & 3, rl = quad * 32 + lane, half = (warp - 2) >> 2;
      int mb, nb;
      tile_coords(u / ks, n_mb, n_nb, gm, mb, nb);
      const int pieces = epilogue_pieces(a, ks);
      if (slice < pieces) {
        const int w = BN / pieces, c_lo = slice * w;
        const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16);
        tc_fence_after();
        reduce_piece(taddr, rl, half, reinterpret_cast<float *>(gbase), ks, c_lo, c_lo + w);
        // the tensor-store staging sits behind the partial tile (8 blocks of 128 x 32 f32) that peers read
        uint8_t *stage = a.tstore ? gbase + (size_t)(BN / 32) * BM * 32 * 4 : nullptr;
        run_epilogue(a, ep, taddr, rl, half, mb * BM + rl, nb, nb * pieces + slice, c_lo, c_lo + w, true, stage);
      }
    }
    // no CTA leaves (or frees its shared memory) while a peer may still read its partial
    cluster_arrive_relaxed();
    cluster_wait_acquire();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem) : "memory");
  }
}

__global__ void f32_to_f16_kernel(const float4 *__restrict__ in, uint2 *__restrict__ out, size_t n4) {
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  pdl_trigger();
  pdl_wait();
  for (; i < n4; i += stride) {
    const float4 v = __ldcs(in + i);
    __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t *>(&a);
    o.y = *reinterpret_cast<uint32_t *>(&b);
    out[i] = o;
  }
}

__global__ void bf16_to_f16_kernel(const __nv_bfloat16 *__restrict__ in, __half *__restrict__ out, size_t n) {
  const size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (i < n) out[i] = __float2half_rn(__bfloat162float(in[i]));
}

// ------------------------------------------------------------------ host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool make_tma_f16(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tma_out(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols, bool f32) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint64_t es = f32 ? 4 : 2;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * es};
  cuuint32_t box[2] = {(cuuint32_t)(128 / es), (cuuint32_t)BM};
  cuuint32_t el[2] = {1, 1};
  CUresult r = fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                  const_cast<void *>(ptr), dims, strides, box, el, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

size_t tc_gemm_smem_bytes() { return (size_t)ST * STAGE + 1024 + 256 + sizeof(EpCols); }

cudaError_t launch_tc_gemm(const TcGemmArgs &a, int n_sm, cudaStream_t s) {
  if (a.N % BN != 0 || a.K % BK != 0 || a.M < 1) return cudaErrorInvalidValue;
  const int ks = a.ksplit > 1 ? a.ksplit : 1;
  const int n_units = ((a.M + BM - 1) / BM) * (a.N / BN) * ks;
  // K slices: a power of two up to 4 (a cluster of them per tile, 256 / ks columns each in the epilogue),
  // one unit per CTA
  if (ks > 1 && (ks > 4 || (ks & (ks - 1)) || ks > a.K / BK || n_units > n_sm)) return cudaErrorInvalidValue;
  const int grid = ks > 1 ? n_units : (n_units < n_sm ? n_units : n_sm);
  const size_t smem = tc_gemm_smem_bytes();
  // two epilogue threads per row when each CTA has one tile (its epilogue is not overlapped)
  const bool wide_epi = grid >= n_units;
  auto kern = wide_epi ? fm_prefill_gemm_kernel<64 + 256> : fm_prefill_gemm_kernel<64 + 128>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(wide_epi ? 64 + 256 : 64 + 128, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int na = 1;
  if (ks > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = ks;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t launch_f32_to_f16(const float *in, __half *out, size_t n, int n_sm, cudaStream_t s) {
  const size_t n4 = n / 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_sm * 4, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, f32_to_f16_kernel, reinterpret_cast<const float4 *>(in),
                            reinterpret_cast<uint2 *>(out), n4);
}

cudaError_t launch_bf16_to_f16(const __nv_bfloat16 *in, __half *out, size_t n, cudaStream_t s) {
  bf16_to_f16_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(in, out, n);
  return cudaGetLastError();
}

}  // namespace fm
