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
//   warps 2..5  read an accumulator with tcgen05.ld (one row per thread) while
//               the next tile accumulates into the other buffer, and run the
//               fused epilogue:
//                 FC:     C' = (c + bias) * norm_w[n] -> f16 and per-row partial
//                         sum of squares (the RMSNorm that follows fc);
//                 KV:     row scale 1/rms(c), per-head RMSNorm (k_norm) and
//                         interleaved-pair RoPE on K heads, f16 stores into the
//                         head-major caches of every layer at the row's
//                         sequence and position;
//                 F16:    bias (+ exact GELU) -> f16, the next product's operand;
//                 RESID:  X += gate * (c + bias), the gated residual;
//                 SEGS:   per-head RMSNorm + RoPE of q / k heads, f32 out;
//                 ARGMAX: per row, the largest logit of the tile (lowest index
//                         on ties), for the lm_head.
// Split-K: a tile's K blocks can be dealt to several CTAs; each stores its
// partial tile to a workspace and the last to finish (atomic ticket) sums the
// partials in slice order into its TMEM accumulator and runs the epilogue.
// Every mbarrier wait is bounded by a clock budget; on expiry the kernel sets
// an error flag, drains, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "dev_common.cuh"
#include "fm_internal.h"
#include "tc_gemm.h"

namespace fm {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, ST = 4;
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE = A_BYTES + B_BYTES;
constexpr int kThreads = 192;
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

// 32 bf16 values (64-byte aligned), fetched raw (16 registers) and widened when used
struct Bf16x32 {
  uint4 u[4];
};
__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16 *__restrict__ p, Bf16x32 &r) {
#pragma unroll
  for (int q = 0; q < 4; ++q) r.u[q] = __ldg(reinterpret_cast<const uint4 *>(p) + q);
}
__device__ __forceinline__ float bf16_at(const Bf16x32 &r, int j) {   // j: a compile-time index
  const uint4 &u = r.u[j >> 3];
  const uint32_t w = (j & 7) < 2 ? u.x : (j & 7) < 4 ? u.y : (j & 7) < 6 ? u.z : u.w;
  return __uint_as_float((j & 1) ? (w & 0xffff0000u) : (w << 16));
}

// RoPE of 32 interleaved channels: (cos, sin) pairs in 8 float4
__device__ __forceinline__ void load_rope16(const float2 *__restrict__ p, float4 (&r)[8]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) r[q] = __ldg(reinterpret_cast<const float4 *>(p) + q);
}
__device__ __forceinline__ void apply_rope16(float *v, const float4 (&r)[8]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float c0 = r[q].x, s0 = r[q].y, c1 = r[q].z, s1 = r[q].w;
    const float a0 = v[4 * q], a1 = v[4 * q + 1], b0 = v[4 * q + 2], b1 = v[4 * q + 3];
    v[4 * q] = a0 * c0 - a1 * s0;
    v[4 * q + 1] = a1 * c0 + a0 * s0;
    v[4 * q + 2] = b0 * c1 - b1 * s1;
    v[4 * q + 3] = b1 * c1 + b0 * s1;
  }
}

__device__ __forceinline__ void store_f4(float *dst, const float *v) {
#pragma unroll
  for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4 *>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
}

// The epilogues below read their per-column operands (norm weights, bias,
// RoPE rows, the residual) before the chunk's accumulator values, so the
// global loads are in flight while tcgen05.ld runs.

__device__ void epilogue_fc(const TcGemmArgs &a, uint32_t taddr, int row, int n0, int nb) {
  float ss = 0.f;
  const bool live = row < a.M;
  for (int c0 = 0; c0 < BN; c0 += 32) {
    Bf16x32 w, b;
    load_bf16x32(a.colw + n0 + c0, w);
    if (a.bias) load_bf16x32(a.bias + n0 + c0, b);
    float v[32];
    tld32(taddr + c0, v);
    if (!live) continue;
    if (a.bias) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] += bf16_at(b, j);
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      ss += v[j] * v[j];
      v[j] *= bf16_at(w, j);
    }
    __half *dst = a.out16 + (size_t)row * a.ldo + n0 + c0;
#pragma unroll
    for (int j = 0; j < 32; j += 8) store_h8(dst + j, v + j);
  }
  if (live) a.row_st[(size_t)row * a.st_ld + nb] = ss;
}

__device__ void epilogue_kv(const TcGemmArgs &a, uint32_t taddr, int row, int n0) {
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
  __half *cache = a.cache + (a.row_seq && live ? (size_t)a.row_seq[row] * a.seq_stride : 0);
  const float2 *rrow = a.rope + (size_t)p * (hd >> 1);
  for (int h0 = 0; h0 < BN; h0 += hd) {
    const int head = ((n0 % a.seg_cols) + h0) / hd;
    float r2 = 1.f;
    if (kind == 0) {
      float ss = 0.f;
      for (int c0 = 0; c0 < hd; c0 += 32) {
        float v[32];
        tld32(taddr + h0 + c0, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) ss += (v[j] * rs) * (v[j] * rs);
      }
      r2 = rsqrtf(ss / (float)hd + a.qk_eps);
    }
    __half *dst = cache + (size_t)(layer * 2 + kind) * a.plane + ((size_t)head * a.max_ctx + p) * hd;
    const __nv_bfloat16 *kw = a.kn_w + (size_t)layer * hd;
    for (int c0 = 0; c0 < hd; c0 += 32) {
      Bf16x32 w;
      float4 rp[8];
      if (kind == 0) {
        load_bf16x32(kw + c0, w);
        load_rope16(rrow + (c0 >> 1), rp);
      }
      float v[32];
      tld32(taddr + h0 + c0, v);
      if (!live) continue;
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= rs;
      if (kind == 0) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = v[j] * r2 * bf16_at(w, j);
        apply_rope16(v, rp);
      }
#pragma unroll
      for (int j = 0; j < 32; j += 8) store_h8(dst + c0 + j, v + j);
    }
  }
}

__device__ void epilogue_f16(const TcGemmArgs &a, uint32_t taddr, int row, int n0) {
  const bool live = row < a.M;
  for (int c0 = 0; c0 < BN; c0 += 32) {
    Bf16x32 bias;
    if (a.bias) load_bf16x32(a.bias + n0 + c0, bias);
    float v[32];
    tld32(taddr + c0, v);
    if (!live) continue;
    if (a.bias) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] += bf16_at(bias, j);
    }
    if (a.out32) store_f4(a.out32 + (size_t)row * a.ldo32 + n0 + c0, v);
    if (!a.out16) continue;
    if (a.gelu) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = gelu_erf(v[j]);
    }
    __half *dst = a.out16 + (size_t)row * a.ldo + n0 + c0;
#pragma unroll
    for (int j = 0; j < 32; j += 8) store_h8(dst + j, v + j);
  }
}

// X += gate * (acc + bias).  With one tile per CTA this epilogue's latency is
// exposed: the next chunk's residual values (L2) are requested before the
// current chunk is finished; gate and bias are shared by every row (L1).
__device__ void epilogue_resid(const TcGemmArgs &a, uint32_t taddr, int row, int n0) {
  const bool live = row < a.M;
  float *__restrict__ x = a.X + (size_t)(live ? row : 0) * a.ldx + n0;
  const float4 *__restrict__ g4 = reinterpret_cast<const float4 *>(a.gate + n0);
  const uint2 *__restrict__ b4 = a.bias ? reinterpret_cast<const uint2 *>(a.bias + n0) : nullptr;
  float4 xv[2][8];
  auto fetch = [&](int c0, int b) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      xv[b][q] = live ? __ldcg(reinterpret_cast<const float4 *>(x + c0) + q) : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  fetch(0, 0);
#pragma unroll
  for (int c = 0; c < BN / 32; ++c) {
    const int c0 = 32 * c, b = c & 1;
    if (c + 1 < BN / 32) fetch(c0 + 32, b ^ 1);
    float v[32];
    tld32(taddr + c0, v);
    if (!live) continue;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 gg = __ldg(g4 + 8 * c + q);
      float bb[4] = {0.f, 0.f, 0.f, 0.f};
      if (b4) {
        const uint2 u = __ldg(b4 + 8 * c + q);
        bb[0] = __uint_as_float(u.x << 16);
        bb[1] = __uint_as_float(u.x & 0xffff0000u);
        bb[2] = __uint_as_float(u.y << 16);
        bb[3] = __uint_as_float(u.y & 0xffff0000u);
      }
      float4 o = xv[b][q];
      o.x += gg.x * (v[4 * q] + bb[0]);
      o.y += gg.y * (v[4 * q + 1] + bb[1]);
      o.z += gg.z * (v[4 * q + 2] + bb[2]);
      o.w += gg.w * (v[4 * q + 3] + bb[3]);
      __stcg(reinterpret_cast<float4 *>(x + c0) + q, o);
    }
  }
}

// q / k / v rows: segment s = n / seg_cols; segments 0 and 1 take a per-head
// RMSNorm with their weight (when given) and RoPE at the row's position
__device__ void epilogue_segs(const TcGemmArgs &a, uint32_t taddr, int row, int n0) {
  const bool live = row < a.M;
  const int seg = n0 / a.seg_cols;
  const __nv_bfloat16 *nw = seg == 0 ? a.nw0 : seg == 1 ? a.nw1 : nullptr;
  const int hd = a.hd;
  const int p = live ? (a.row_pos ? a.row_pos[row] : a.start + row) : 0;
  const float2 *rrow = a.rope + (size_t)p * (hd >> 1);
  float *__restrict__ out = a.out32 + (size_t)(live ? row : 0) * a.ldo32 + n0;
  for (int h0 = 0; h0 < BN; h0 += hd) {
    float r2 = 1.f;
    if (nw) {
      float ss = 0.f;
      for (int c0 = 0; c0 < hd; c0 += 32) {
        float v[32];
        tld32(taddr + h0 + c0, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) ss += v[j] * v[j];
      }
      r2 = rsqrtf(ss / (float)hd + a.qk_eps);
    }
    for (int c0 = 0; c0 < hd; c0 += 32) {
      Bf16x32 w;
      float4 rp[8];
      if (nw) {
        load_bf16x32(nw + c0, w);
        load_rope16(rrow + (c0 >> 1), rp);
      }
      float v[32];
      tld32(taddr + h0 + c0, v);
      if (!live) continue;
      if (nw) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = v[j] * r2 * bf16_at(w, j);
        apply_rope16(v, rp);
      }
      store_f4(out + h0 + c0, v);
    }
  }
}

__device__ void epilogue_argmax(const TcGemmArgs &a, uint32_t taddr, int row, int n0, int nb) {
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int c0 = 0; c0 < BN; c0 += 32) {
    float v[32];
    tld32(taddr + c0, v);
#pragma unroll
    for (int j = 0; j < 32; ++j)   // ascending columns, strict '>': the lowest index wins a tie
      if (n0 + c0 + j < a.n_valid && v[j] > best) {
        best = v[j];
        bi = n0 + c0 + j;
      }
  }
  if (row < a.M) a.amax[(size_t)row * a.amax_ld + nb] = make_float2(best, __int_as_float(bi));
}

// Split-K partial tiles in the workspace: per (tile, slice) 8 chunk blocks of
// 128 rows x 32 f32 (16 KB each), the 16-byte units of a row XOR-swizzled by
// (row & 7) so that a warp's reads of one unit column spread over the banks.
__device__ __forceinline__ size_t ws_block(int tile, int ks, int slice, int c) {
  return ((((size_t)tile * ks + slice) * 8 + c) * BM) * 32;
}

// Split-K: store this slice's partial tile; the last slice of the tile to get
// here sums every slice's partial (in slice order, its own from TMEM) back into
// the accumulator.  The other slices' blocks come through the bulk-copy engine
// into the operand ring, which is idle by then (a split GEMM gives each CTA
// one unit), two chunks in flight.  Returns whether this CTA runs the tile's
// epilogue.  All 128 epilogue threads call it together.
__device__ bool splitk_gather(const TcGemmArgs &a, uint32_t taddr, int rl, int tile, int slice, int *s_last,
                              uint32_t stage, const uint8_t *stage_ptr, uint32_t gbar) {
  const int ks = a.ksplit;
  const int sw = rl & 7;
  for (int c = 0; c < BN / 32; ++c) {
    float v[32];
    tld32(taddr + 32 * c, v);
    float *dst = a.ws + ws_block(tile, ks, slice, c) + (size_t)rl * 32;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      *reinterpret_cast<float4 *>(dst + 4 * (u ^ sw)) = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
  }
  named_sync(1, 128);
  if (threadIdx.x == 64) {
    __threadfence();
    const int old = atomicAdd(a.tile_tickets + tile, 1);
    const int last = old == ks - 1;
    if (last) atomicExch(a.tile_tickets + tile, 0);
    *s_last = last;
  }
  named_sync(1, 128);
  if (!*s_last) return false;
  __threadfence();
  constexpr uint32_t kBlk = BM * 32 * 4;
  const uint32_t buf = (uint32_t)(ks - 1) * kBlk;
  auto issue = [&](int c) {
    const uint32_t bar = gbar + 8 * (c & 1);
    mbar_expect_tx(bar, buf);
    int k = 0;
    for (int s = 0; s < ks; ++s)
      if (s != slice) bulk_g2s(stage + (c & 1) * buf + (k++) * kBlk, a.ws + ws_block(tile, ks, s, c), kBlk, bar);
  };
  if (threadIdx.x == 64) {
    // the blocks were written through the generic proxy by other CTAs
    asm volatile("fence.proxy.async.global;\n" ::: "memory");
    issue(0);
    issue(1);
  }
  for (int c = 0; c < BN / 32; ++c) {
    const int b = c & 1;
    mbar_wait_bounded(gbar + 8 * b, (c >> 1) & 1, a.err);
    float v[32], acc[32];
    tld32(taddr + 32 * c, v);
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = 0.f;
    int k = 0;
    for (int s = 0; s < ks; ++s) {
      if (s == slice) {
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] += v[j];
      } else {
        const float *blk = reinterpret_cast<const float *>(stage_ptr + b * buf + (k++) * kBlk) + (size_t)rl * 32;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 q = *reinterpret_cast<const float4 *>(blk + 4 * (u ^ sw));
          acc[4 * u] += q.x;
          acc[4 * u + 1] += q.y;
          acc[4 * u + 2] += q.z;
          acc[4 * u + 3] += q.w;
        }
      }
    }
    tmem_st32(taddr + 32 * c, acc);
    named_sync(1, 128);   // buffer b has been read by the group
    if (threadIdx.x == 64 && c + 2 < BN / 32) issue(c + 2);
  }
  return true;
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

__global__ void __launch_bounds__(kThreads, 1) fm_prefill_gemm_kernel(const __grid_constant__ TcGemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint8_t *gbase = smem_raw + (base - smem_u32(smem_raw));
  const uint32_t bars = base + ST * STAGE;
  auto full = [&](int s) { return bars + 8 * s; };
  auto empty = [&](int s) { return bars + 8 * (ST + s); };
  auto tfull = [&](int b) { return bars + 8 * (2 * ST + b); };
  auto tempty = [&](int b) { return bars + 8 * (2 * ST + 2 + b); };
  const uint32_t tslot = bars + 8 * (2 * ST + 4);
  const uint32_t gbar = bars + 8 * (2 * ST + 5);   // two: split-K gather buffers
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull(b), 1);
      mbar_init(tempty(b), 128);
      mbar_init(gbar + 8 * b, 1);
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
  pdl_wait();

  const int n_nb = a.N / BN;
  const int n_mb = (a.M + BM - 1) / BM;
  const int n_tiles = n_mb * n_nb;
  const int gm = a.group_m > 0 ? a.group_m : 1;
  const int nk = a.K / BK;
  const int ks = a.ksplit > 1 ? a.ksplit : 1;
  const int n_units = n_tiles * ks;   // unit u: tile u / ks, K slice u % ks (slices of a tile adjacent)
  auto kslice = [&](int slice, int &kb0, int &kb1) {
    kb0 = slice * nk / ks;
    kb1 = (slice + 1) * nk / ks;
  };

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        int mb, nb, kb0, kb1;
        tile_coords(u / ks, n_mb, n_nb, gm, mb, nb);
        kslice(u % ks, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % ST;
          if (!mbar_wait(empty(s), ((it / ST) & 1) ^ 1, a.err)) { ok = false; break; }
          const uint32_t sa = base + s * STAGE, sb = sa + A_BYTES;
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
    __shared__ int s_last;
    uint32_t tc = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++tc) {
      const int b = tc & 1;
      const bool ok = mbar_wait(tfull(b), (tc >> 1) & 1, a.err);
      // with K slices the group meets at named barriers: its verdict must be one
      if (ks > 1 ? bar_any(1, 128, !ok) : !ok) break;
      tc_fence_after();
      const int tile = u / ks;
      int mb, nb;
      tile_coords(tile, n_mb, n_nb, gm, mb, nb);
      const uint32_t taddr = tmem + b * BN + ((uint32_t)(quad * 32) << 16);
      const int row = mb * BM + rl;
      if (ks == 1 || splitk_gather(a, taddr, rl, tile, u % ks, &s_last, base, gbase, gbar)) {
        switch (a.epi) {
          case TC_EPI_FC: epilogue_fc(a, taddr, row, nb * BN, nb); break;
          case TC_EPI_KV: epilogue_kv(a, taddr, row, nb * BN); break;
          case TC_EPI_F16: epilogue_f16(a, taddr, row, nb * BN); break;
          case TC_EPI_RESID: epilogue_resid(a, taddr, row, nb * BN); break;
          case TC_EPI_SEGS: epilogue_segs(a, taddr, row, nb * BN); break;
          default: epilogue_argmax(a, taddr, row, nb * BN, nb); break;
        }
      }
      tc_fence_before();
      mbar_arrive(tempty(b));
    }
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

size_t tc_gemm_smem_bytes() { return (size_t)ST * STAGE + 1024 + 256; }

cudaError_t launch_tc_gemm(const TcGemmArgs &a, int n_sm, cudaStream_t s) {
  if (a.N % BN != 0 || a.K % BK != 0 || a.M < 1) return cudaErrorInvalidValue;
  const int ks = a.ksplit > 1 ? a.ksplit : 1;
  if (ks > a.K / BK || (ks > 1 && (!a.ws || !a.tile_tickets))) return cudaErrorInvalidValue;
  const int n_units = ((a.M + BM - 1) / BM) * (a.N / BN) * ks;
  // a split GEMM gives each CTA one unit (the gather stages its partials in the idle operand
  // ring: two chunks of ks - 1 blocks of 16 KB must fit)
  if (ks > 1 && (n_units > n_sm || 2 * (ks - 1) * BM * 32 * 4 > ST * STAGE)) return cudaErrorInvalidValue;
  const int grid = n_units < n_sm ? n_units : n_sm;
  const size_t smem = tc_gemm_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(fm_prefill_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fm_prefill_gemm_kernel, a);
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
