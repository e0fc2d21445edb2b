// linear_parts.cuh -- the device pieces of the skinny weight-streaming linear
// layer shared by the one-launch-per-product kernel (k_gemv.cu) and the
// persistent draft-step kernel (k_step.cu): warp roles, row statistics of
// normalised inputs, staging of the activations as the tensor cores' B operand
// (RMSNorm / adaLN LayerNorm-modulate / table-row prologues, bf16 hi + lo
// split), the fused epilogues, and the block self-attention of one head.
#pragma once

#include "dev_common.cuh"
#include "fm_internal.h"

namespace fm {
namespace {

constexpr int kWorkers = 256;          // warps 2..9: stage activations, read TMEM, epilogue
constexpr int kAll = 64 + kWorkers;    // warp 0 streams weights, warp 1 owns TMEM and issues MMAs
constexpr int kThreads = kWorkers;     // threads that share the epilogue loops
constexpr int kWorkerBase = 64;        // first worker thread
__device__ __forceinline__ int wtid() { return (int)threadIdx.x - kWorkerBase; }
constexpr int kChunk = 64;                       // k per pipeline stage
constexpr int kStageBytes = kTile * kChunk * 2;  // 16 KB of bf16 weights
constexpr int kCsStride = kTile + 8;             // f32 partial tile row stride
static_assert(kWorkers == 8 * kMaxT, "row statistics: eight worker threads per row");

// (mean, M2) of one row over one 128-column tile, two-pass inside a warp: lane l
// holds columns 4l .. 4l + 3 (live lanes only; n = the tile's live columns).
__device__ __forceinline__ float2 tile_moments(const float (&v)[4], bool live, float n) {
  float s = live ? (v[0] + v[1]) + (v[2] + v[3]) : 0.f;
  s = warp_sum(s);
  const float mean = s / n;
  float q = 0.f;
  if (live) {
#pragma unroll
    for (int e = 0; e < 4; ++e) q += (v[e] - mean) * (v[e] - mean);
  }
  q = warp_sum(q);
  return make_float2(mean, q);
}

// Row statistics of the input rows from the producer's per-tile partials, in
// f32, by all worker threads.  For A_RMS / A_LNMOD a partial is the tile's
// (mean, M2 = sum of squared deviations from that mean) over its columns (see
// tile_moments); the tiles are combined with the pairwise update of Chan,
// Golub and LeVeque ("Updating formulae and a pairwise algorithm for computing
// sample variances", 1979): for parts A, B of counts nA, nB,
//   n = nA + nB, d = mean_B - mean_A, mean = mean_A + d nB / n,
//   M2 = M2_A + M2_B + d^2 nA nB / n,
// so the variance never comes from a difference of two large sums (a row with
// |mean| >> std keeps its precision), matching the two-pass LayerNorm of the
// pages (flashmap_drafter.js, ``lnMod``).  A_RMS needs only the sum of squares,
// sum_i (M2_i + n_i mean_i^2).  A_RMS2 partials are raw (sum v^2, sum (v w)^2).
// (FP64 runs at a small fraction of the f32 rate on this GPU: this arithmetic in
// double cost about a microsecond on the critical path of every normalised GEMV.)
__device__ __forceinline__ void chan_merge(float &n, float &mean, float &m2, float nb, float meanb, float m2b) {
  const float tot = n + nb;
  if (tot <= 0.f) return;
  const float d = meanb - mean;
  const float f = nb / tot;
  mean = mean + d * f;
  m2 = m2 + m2b + d * d * n * f;
  n = tot;
}

__device__ void load_row_stats(const GemvArgs &a, int T, float *mu, float *rs, int tid) {
  // eight threads per row (kMaxT rows): thread j takes tiles j, j + 8, ..., all
  // its loads in flight at once; the row's eight partial results meet by shuffles
  const int t = tid >> 3, j = tid & 7;
  const bool active =
      t < T && (a.amode == A_RMS || a.amode == A_LNMOD || a.amode == A_RMS2);
  const bool raw = a.amode == A_RMS2;
  float cnt = 0.f, s1 = 0.f, s2 = 0.f;   // moments: (count, mean, M2); raw: (-, sum, sum)
  if (active) {
    const bool second = a.split > 0 && t >= a.split;
    const int ts = a.st_bcast ? 0 : (second ? t - a.split : t);
    const float2 *stp = second ? a.st2 : a.st;
    const int n = a.st_tiles;
    float2 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = j + 8 * u;
      v[u] = i < n ? __ldcg(stp + i * kMaxT + ts) : make_float2(0.f, 0.f);
    }
    auto take = [&](int i, float2 w) {
      if (raw) {
        s1 += w.x; s2 += w.y;
      } else {
        const float ni = (float)min(kTile, a.K - i * kTile);
        chan_merge(cnt, s1, s2, ni, w.x, w.y);
      }
    };
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (j + 8 * u < n) take(j + 8 * u, v[u]);
    for (int i = j + 32; i < n; i += 8) take(i, __ldcg(stp + i * kMaxT + ts));
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    const float c2 = __shfl_xor_sync(0xffffffffu, cnt, o);
    const float a2 = __shfl_xor_sync(0xffffffffu, s1, o);
    const float b2 = __shfl_xor_sync(0xffffffffu, s2, o);
    if (raw) {
      s1 += a2; s2 += b2;
    } else if ((tid & o) == 0) {
      chan_merge(cnt, s1, s2, c2, a2, b2);   // lower partner first: the same order on both lanes
    } else {
      float c = c2, m = a2, q = b2;
      chan_merge(c, m, q, cnt, s1, s2);
      cnt = c; s1 = m; s2 = q;
    }
  }
  if (j == 0 && t < kMaxT) {
    float m = 0.f, r = 1.f;
    if (active) {
      if (a.amode == A_RMS) {
        // sum of squares = M2 + n mean^2 over the whole row
        r = rsqrtf((s2 + cnt * s1 * s1) * a.inv_n + a.eps);
      } else if (a.amode == A_RMS2) {
        const float r1 = rsqrtf(s1 * a.inv_n + a.eps);
        const float r2 = rsqrtf(r1 * r1 * s2 * a.inv_n + a.eps);
        m = r1;   // A_RMS2 keeps r1 in the mean slot
        r = r2;
      } else {
        m = s1;
        r = rsqrtf(fmaxf(s2 * a.inv_n, 0.f) + a.eps);   // population variance M2 / n
      }
    }
    mu[t] = m;
    rs[t] = r;
  }
}


// Staging of activation columns k0 .. k0 + kp as the MMA's B operand: rows
// 0 .. 16MT-1 hold the bf16 hi parts, rows 16MT .. 32MT-1 the lo parts, one
// 64-column chunk after another (each chunk 32MT rows x 128 bytes, 128-byte
// swizzle).  Two phases, so that a piece's global loads (activations and norm
// weights) are in flight while the row statistics are formed: stage_load
// issues them into registers, stage_store transforms and stores.
template <int MT>
struct StageRegs {
  static constexpr int rows = 16 * MT;
  static constexpr int tpr = kWorkers / rows;   // threads per activation row (16 or 8)
  static constexpr int kMaxKp = MT == 1 ? 256 : 128;   // piece width (17..32 rows: 128, see the launcher)
  static constexpr int kMaxQ = kMaxKp / 4 / tpr;       // quads per thread for a full piece
  float4 xv[kMaxQ];
  // per-column operands of the transform, loaded with the activations:
  // A_RMS: p0.xy = 4 bf16 norm weights; A_RMS2: p0.xy, p0.zw = both weight quads;
  // A_LNMOD: p0 = scale, p1 = shift
  float4 p0[kMaxQ], p1[kMaxQ];
};

template <int MT>
__device__ __forceinline__ void stage_load(const GemvArgs &a, int T, int m0, int k0, int kp, StageRegs<MT> &g) {
  using R = StageRegs<MT>;
  const int tid = wtid();
  const int t = tid / R::tpr, q0 = tid % R::tpr;   // constant divisors
  const int nq = (kp >> 2) / R::tpr;               // kp is a multiple of 64
  const float *X = a.x_from_sp ? a.sp->feats : a.X;
  const bool second = a.split > 0 && t >= a.split;
  const bool load = t < T && a.amode != A_ROW_Q8 && a.amode != A_ROW_BF16;
  const float *xr = second ? a.X2 + (size_t)(t - a.split) * a.ldx : X + (size_t)t * a.ldx;
  const __nv_bfloat16 *wv = (a.amode == A_RMS && second) ? a.nw_alt : a.nw;
  const __nv_bfloat16 *nw2 = a.nw2;
  if (a.amode == A_RMS2 && a.nw_rows > 0) nw2 += (size_t)(m0 / a.nw_rows) * a.K;
  const bool wload = t < T && (a.amode == A_RMS || a.amode == A_RMS2);
  const bool mload = t < T && a.amode == A_LNMOD;
#pragma unroll
  for (int j = 0; j < R::kMaxQ; ++j) {
    g.xv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    g.p0[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    g.p1[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int k = k0 + 4 * (q0 + R::tpr * j);
    if (j < nq && load) g.xv[j] = __ldcg(reinterpret_cast<const float4 *>(xr + k));
    if (j < nq && wload) {
      const uint2 w = *reinterpret_cast<const uint2 *>(wv + k);
      uint2 w2 = make_uint2(0u, 0u);
      if (a.amode == A_RMS2) w2 = *reinterpret_cast<const uint2 *>(nw2 + k);
      g.p0[j] = make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w2.x), __uint_as_float(w2.y));
    }
    if (j < nq && mload) {
      g.p0[j] = *reinterpret_cast<const float4 *>(a.sc + k);
      g.p1[j] = *reinterpret_cast<const float4 *>(a.sh + k);
    }
  }
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int MT>
__device__ __forceinline__ void stage_store(const GemvArgs &a, const float *stat_mu, const float *stat_rs, uint32_t dst, int T, int k0, int kp,
                                            const StageRegs<MT> &g) {
  using R = StageRegs<MT>;
  const int tid = wtid();
  const int t = tid / R::tpr, q0 = tid % R::tpr;
  const int nq = (kp >> 2) / R::tpr;
  float mu = 0.f, rs = 1.f;
  if (t < T) { mu = stat_mu[t]; rs = stat_rs[t]; }
#pragma unroll
  for (int j = 0; j < R::kMaxQ; ++j) {
    if (j >= nq) break;
    const int kq = 4 * (q0 + R::tpr * j);   // column inside the piece
    const int k = k0 + kq;
    float v[4] = {g.xv[j].x, g.xv[j].y, g.xv[j].z, g.xv[j].w};
    if (t < T) {
      if (a.amode == A_ROW_Q8 || a.amode == A_ROW_BF16) {
        v[0] = v[1] = v[2] = v[3] = 0.f;
        if (t == 0) {
          const int r = a.sp->anchor;
          const size_t chunk = (size_t)(r >> 7) * (a.K / 64) + (k >> 6);
          const int rr = r & 127, kk = k & 63;
          if (a.amode == A_ROW_Q8) {
            const uint8_t *base = a.tq8 + chunk * kQ8Chunk;
            const uchar4 qv = *reinterpret_cast<const uchar4 *>(base + q8_slot(rr, kk));   // q + 128
            const float d = __half2float(
                *reinterpret_cast<const __half *>(base + kTile * 64 + (kk >> 5) * 256 + rr * 2));
            v[0] = d * (float)((int)qv.x - 128); v[1] = d * (float)((int)qv.y - 128);
            v[2] = d * (float)((int)qv.z - 128); v[3] = d * (float)((int)qv.w - 128);
          } else {
            const uint8_t *base = a.tb + chunk * 16384;
            const uint2 u = *reinterpret_cast<const uint2 *>(base + w_slot(rr, kk));
            v[0] = bf_lo(u.x); v[1] = bf_hi(u.x); v[2] = bf_lo(u.y); v[3] = bf_hi(u.y);
          }
        }
      } else if (a.amode == A_RMS) {
        const uint32_t w01 = __float_as_uint(g.p0[j].x), w23 = __float_as_uint(g.p0[j].y);
        const float w[4] = {bf_lo(w01), bf_hi(w01), bf_lo(w23), bf_hi(w23)};
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = v[e] * rs * w[e];
      } else if (a.amode == A_RMS2) {
        const uint32_t w01 = __float_as_uint(g.p0[j].x), w23 = __float_as_uint(g.p0[j].y);
        const uint32_t u01 = __float_as_uint(g.p0[j].z), u23 = __float_as_uint(g.p0[j].w);
        const float w[4] = {bf_lo(w01), bf_hi(w01), bf_lo(w23), bf_hi(w23)};
        const float w2[4] = {bf_lo(u01), bf_hi(u01), bf_lo(u23), bf_hi(u23)};
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = (v[e] * mu * w[e]) * rs * w2[e];
      } else if (a.amode == A_LNMOD) {
        const float4 sc = g.p0[j];
        const float4 sh = g.p1[j];
        v[0] = (v[0] - mu) * rs * (1.f + sc.x) + sh.x;
        v[1] = (v[1] - mu) * rs * (1.f + sc.y) + sh.y;
        v[2] = (v[2] - mu) * rs * (1.f + sc.z) + sh.z;
        v[3] = (v[3] - mu) * rs * (1.f + sc.w) + sh.w;
      }
    }
    uint32_t h01, l01, h23, l23;
    split2_bf16(v[0], v[1], h01, l01);
    split2_bf16(v[2], v[3], h23, l23);
    const uint32_t cbase = dst + (uint32_t)(kq >> 6) * (32 * MT * 128);
    const int kk = kq & 63;
    asm volatile("st.shared.v2.u32 [%0], {%1,%2};\n" ::"r"(cbase + sw128(t, kk)), "r"(h01), "r"(h23));
    asm volatile("st.shared.v2.u32 [%0], {%1,%2};\n" ::"r"(cbase + sw128(R::rows + t, kk)), "r"(l01), "r"(l23));
  }
}

__device__ __forceinline__ int row_pos(const GemvArgs &a, int t) {
  if (a.pos_src == 3) return t < a.split ? a.sp->start + t : a.sp->pos + (t - a.split);
  const int base = a.pos_src == 0 ? a.sp->pos : a.pos_src == 1 ? a.sp->start : a.sp->L;
  return base + a.pos_add + t;
}

// Epilogue for one (token t, 128-row tile): lane holds rows 4 * lane .. + 3.
// The global operands of an epilogue unit (bias, residual row, gate), loaded
// ahead of time so their L2 latency overlaps the cluster barrier.
struct EpiIn {
  float4 r, g;
  float b[4];
  uint2 nw;          // E_SEGS: the four per-head norm weights of this lane's rows (bf16)
  float2 cs0, cs1;   // E_SEGS: the rotation (cos, sin) of the two pairs, at the row's position
};
__device__ __forceinline__ void epilogue_load(const GemvArgs &a, int t, int m0, EpiIn &in) {
  const int mrow = m0 + 4 * (threadIdx.x & 31);
  const bool live = mrow < a.M;
  in.r = make_float4(0.f, 0.f, 0.f, 0.f);
  in.g = make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll
  for (int e = 0; e < 4; ++e) in.b[e] = 0.f;
  in.nw = make_uint2(0u, 0u);
  in.cs0 = in.cs1 = make_float2(1.f, 0.f);
  if (!live) return;
  if (a.emode == E_SEGS) {
    const int seg = m0 / a.seg_rows;
    const SegDesc &sd = a.segs[seg];
    const int d0 = (mrow - seg * a.seg_rows) % a.hd;
    if (sd.norm_w) {
      in.nw = *reinterpret_cast<const uint2 *>(sd.norm_w + d0);
      if (sd.rope) {
        const int p = row_pos(a, t);
        in.cs0 = a.rope[(size_t)p * (a.hd >> 1) + (d0 >> 1)];
        in.cs1 = a.rope[(size_t)p * (a.hd >> 1) + (d0 >> 1) + 1];
      }
    }
  }
  if (a.bias) {
    const uint2 u = *reinterpret_cast<const uint2 *>(a.bias + mrow);
    const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162 *>(&u.x);
    const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162 *>(&u.y);
    in.b[0] = __low2float(p0); in.b[1] = __high2float(p0); in.b[2] = __low2float(p1); in.b[3] = __high2float(p1);
  }
  if (a.emode == E_RESID) {
    in.r = __ldcg(reinterpret_cast<const float4 *>(a.R + (size_t)t * a.ldr + mrow));
    if (a.gate) in.g = *reinterpret_cast<const float4 *>(a.gate + mrow);
  }
}

__device__ void epilogue_unit(const GemvArgs &a, int t, int m0, float (&v)[4], int tile, const EpiIn &in) {
  const int lane = threadIdx.x & 31;
  const int mrow = m0 + 4 * lane;
  const bool live = mrow < a.M;  // M is a multiple of 4
#pragma unroll
  for (int e = 0; e < 4; ++e) v[e] += in.b[e];
  switch (a.emode) {
    case E_STORE:
    case E_GELU:
    case E_RESID: {
      if (a.emode == E_GELU) {
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = gelu_erf(v[e]);
      } else if (a.emode == E_RESID && live) {
        v[0] = in.r.x + in.g.x * v[0];
        v[1] = in.r.y + in.g.y * v[1];
        v[2] = in.r.z + in.g.z * v[2];
        v[3] = in.r.w + in.g.w * v[3];
      }
      if (live)
        __stcg(reinterpret_cast<float4 *>(a.Y + (size_t)t * a.ldy + mrow), make_float4(v[0], v[1], v[2], v[3]));
      if (a.Y2 && live)
        __stcg(reinterpret_cast<float4 *>(a.Y2 + (size_t)t * a.ldy2 + mrow), make_float4(v[0], v[1], v[2], v[3]));
      if (a.ylm && live) {
        // the same rows split into the lm_head's resident operand (hi row, lo row 8 further)
        uint32_t hw[2], lw[2];
        if (a.ylm_f16) {
          split2_f16(v[0], v[1], hw[0], lw[0]);
          split2_f16(v[2], v[3], hw[1], lw[1]);
        } else {
          split2_bf16(v[0], v[1], hw[0], lw[0]);
          split2_bf16(v[2], v[3], hw[1], lw[1]);
        }
        uint8_t *cb = a.ylm + (size_t)(mrow >> 6) * kLmYChunk;
        const int r = lm_yrow(t);
        *reinterpret_cast<uint2 *>(cb + sw128(r, mrow & 63)) = make_uint2(hw[0], hw[1]);
        *reinterpret_cast<uint2 *>(cb + sw128(r + 8, mrow & 63)) = make_uint2(lw[0], lw[1]);
      }
      if (a.out_st) {
        float2 st;
        if (a.st_w) {
          // raw (sum v^2, sum (v w)^2) for the two chained RMSNorms of A_RMS2
          float s1 = 0.f, s2 = 0.f;
          if (live) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float vw = v[e] * __bfloat162float(a.st_w[mrow + e]);
              s1 += v[e] * v[e];
              s2 += vw * vw;
            }
          }
          st = make_float2(warp_sum(s1), warp_sum(s2));
        } else {
          st = tile_moments(v, live, (float)min(kTile, a.M - m0));
        }
        if (lane == 0) a.out_st[tile * kMaxT + t] = st;
      }
      break;
    }
    case E_GEGLU: {
      // rows 0..63 of the tile are gate rows f0 .. f0+63, rows 64..127 the up rows
      const float other0 = __shfl_xor_sync(0xffffffffu, v[0], 16);
      const float other1 = __shfl_xor_sync(0xffffffffu, v[1], 16);
      const float other2 = __shfl_xor_sync(0xffffffffu, v[2], 16);
      const float other3 = __shfl_xor_sync(0xffffffffu, v[3], 16);
      if (lane < 16) {
        const int f = (m0 >> 1) + 4 * lane;
        float4 o;
        o.x = gelu_tanh(v[0]) * other0;
        o.y = gelu_tanh(v[1]) * other1;
        o.z = gelu_tanh(v[2]) * other2;
        o.w = gelu_tanh(v[3]) * other3;
        __stcg(reinterpret_cast<float4 *>(a.Y + (size_t)t * a.ldy + f), o);
      }
      break;
    }
    case E_SEGS: {
      const int seg = m0 / a.seg_rows;
      const SegDesc &sd = a.segs[seg];
      const int mseg = mrow - seg * a.seg_rows;   // row inside the segment
      const int hd = a.hd;
      const int lanes_per_head = hd >> 2;
      if (sd.norm_w) {
        float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
        ss = group_sum(ss, lanes_per_head);
        const float r = rsqrtf(ss / (float)hd + a.qk_eps);
        const float w[4] = {__uint_as_float(in.nw.x << 16), __uint_as_float(in.nw.x & 0xffff0000u),
                            __uint_as_float(in.nw.y << 16), __uint_as_float(in.nw.y & 0xffff0000u)};
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = v[e] * r * w[e];
        if (sd.rope) {
          const float2 cs0 = in.cs0, cs1 = in.cs1;
          const float x0 = v[0], x1 = v[1], x2 = v[2], x3 = v[3];
          v[0] = x0 * cs0.x - x1 * cs0.y;
          v[1] = x1 * cs0.x + x0 * cs0.y;
          v[2] = x2 * cs1.x - x3 * cs1.y;
          v[3] = x3 * cs1.x + x2 * cs1.y;
        }
      }
      if (sd.kind == SEG_F32) {
        __stcg(reinterpret_cast<float4 *>(a.Y + (size_t)t * a.ldy + sd.y_col + mseg),
               make_float4(v[0], v[1], v[2], v[3]));
      } else {
        const int p = row_pos(a, t);
        const int head = mseg / hd, d0 = mseg % hd;
        __half2 lo = __floats2half2_rn(v[0], v[1]);
        __half2 hi = __floats2half2_rn(v[2], v[3]);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t *>(&lo);
        pk.y = *reinterpret_cast<uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(sd.cache + ((size_t)head * a.max_ctx + p) * hd + d0) = pk;
      }
      break;
    }
  }
}

// Attention of the block over itself for one head (rows t < T, unmasked):
// O = softmax(q k^T * scale) v from the q/k/v segments in Y.
__device__ void self_attention_head(const GemvArgs &a, int head, int T, float *sm) {
  const int hd = a.hd, D = a.self_D;
  const int ks = hd + 4;  // padded row stride (floats) in shared memory, keeps float4 alignment
  float *qq = sm, *kk = sm + kMaxT * ks, *vv = sm + 2 * kMaxT * ks;
  const int q4 = hd / 4;
  const bool consumer = wtid() >= 0;  // the weight and MMA warps only join the barriers
  for (int i = wtid(); consumer && i < T * q4; i += kThreads) {
    const int t = i / q4, d = 4 * (i - t * q4);
    const float *row = a.Y + (size_t)t * a.ldy + head * hd + d;
    const float4 q = __ldcg(reinterpret_cast<const float4 *>(row));
    const float4 k = __ldcg(reinterpret_cast<const float4 *>(row + D));
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(row + 2 * D));
    *reinterpret_cast<float4 *>(qq + t * ks + d) = q;
    *reinterpret_cast<float4 *>(kk + t * ks + d) = k;
    *reinterpret_cast<float4 *>(vv + t * ks + d) = v;
  }
  __syncthreads();
  // one warp per query row.  Scores: lane j < T forms q_t . k_j over the head's dims
  // (no cross-lane sums); softmax over the lanes; output: lane l owns dims 4l .. 4l+3
  // and gathers p_j from lane j.
  const int lane = threadIdx.x & 31, w = wtid() >> 5;
  const bool on = lane < q4;
  for (int t = w; consumer && t < T; t += kThreads / 32) {
    const float *qrow = qq + t * ks;
    const float *krow = kk + (lane < T ? lane : 0) * ks;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    for (int d = 0; d < hd; d += 4) {
      const float4 q = *reinterpret_cast<const float4 *>(qrow + d);
      const float4 k = *reinterpret_cast<const float4 *>(krow + d);
      s0 += q.x * k.x; s1 += q.y * k.y; s2 += q.z * k.z; s3 += q.w * k.w;
    }
    const float sc = lane < T ? ((s0 + s1) + (s2 + s3)) * a.attn_scale : -INFINITY;
    float mx = sc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float p = lane < T ? __expf(sc - mx) : 0.f;
    const float den = warp_sum(p);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < T; ++j) {
      const float pj = __shfl_sync(0xffffffffu, p, j);
      if (on) {
        const float4 v = *reinterpret_cast<const float4 *>(vv + j * ks + 4 * lane);
        o.x += pj * v.x; o.y += pj * v.y; o.z += pj * v.z; o.w += pj * v.w;
      }
    }
    if (on) {
      const float inv = 1.f / den;
      *reinterpret_cast<float4 *>(a.attn_out + (size_t)t * D + head * hd + 4 * lane) =
          make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
    }
  }
  __syncthreads();
}

}  // namespace
}  // namespace fm
