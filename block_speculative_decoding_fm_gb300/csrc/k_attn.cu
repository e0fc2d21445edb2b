// k_attn.cu -- cross-attention of the draft block over the context cache.
//
// Computes, per head h and block row t < T <= 16,
//   O[t] = softmax_j(q_t . k_j / sqrt(hd)) v_j   over cache rows j < L, no mask,
// as the pages do with one workgroup per (head, row) and all scores in shared
// memory (flashmap_drafter.js ``attn``, L <= 4096).  Here the keys are split
// across CTAs (flash-decoding): each (head, split) CTA streams its share of the
// head-major f16 cache through shared memory with cp.async, computes scores
// and P.V on the tensor cores (f16 m16n8k16, queries and probabilities split
// into f16 hi + lo), keeps an online softmax (running max / sum, rescaled as
// the MTP head's attention kernel does on ternary_bonsai_2_mtp.js), and the
// last CTA of a head merges the splits in a fixed order.  Any L is handled.
#include "dev_common.cuh"
#include "fm_internal.h"

namespace fm {

namespace {

constexpr int kThreads = 128;  // 4 warps, 16 keys each per 64-key stage
constexpr int kKeys = 64;

__device__ __forceinline__ uint32_t kslot(int r, int u, int hd) {  // K tile: XOR bit 2 of the unit by row parity
  return r * hd * 2 + ((u ^ ((r & 1) << 2)) << 4);
}
__device__ __forceinline__ uint32_t vslot(int r, int u, int hd) {  // V tile: XOR the unit by row % 8
  return r * hd * 2 + ((u ^ (r & 7)) << 4);
}

template <int HD>
__device__ __forceinline__ void issue_kv(const AttnArgs &a, int head, uint32_t kbuf, uint32_t vbuf, int k0,
                                         int kend) {
  constexpr int U = HD / 8;  // 16-byte units per row
  const __half *kb = a.Kc + (size_t)head * a.max_ctx * HD;
  const __half *vb = a.Vc + (size_t)head * a.max_ctx * HD;
  for (int i = threadIdx.x; i < kKeys * U; i += kThreads) {
    const int r = i / U, u = i - r * U;
    const int key = k0 + r;
    const bool ok = key < kend;
    const size_t off = (size_t)(ok ? key : 0) * HD + u * 8;
    cp_async16(kbuf + kslot(r, u, HD), kb + off, ok ? 16u : 0u);
    cp_async16(vbuf + vslot(r, u, HD), vb + off, ok ? 16u : 0u);
  }
}

}  // namespace

template <int HD>
__global__ void __launch_bounds__(kThreads) attn_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int NT = HD / 8;        // n8 tiles of the output
  constexpr int QS = HD + 32;       // f16 row stride of the query tile (64-byte pad)
  const int head = blockIdx.x, split = blockIdx.y;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t tile_bytes = kKeys * HD * 2;
  const uint32_t kb0 = sbase, vb0 = sbase + tile_bytes, kb1 = sbase + 2 * tile_bytes, vb1 = sbase + 3 * tile_bytes;
  const uint32_t qhi = sbase + 4 * tile_bytes, qlo = qhi + 16 * QS * 2;
  float *merge = reinterpret_cast<float *>(smem);  // reused after the key loop

  pdl_trigger();
  pdl_wait();
  const int T = a.T_const > 0 ? a.T_const : a.sp->T;
  const int L = (a.L_src == 0 ? a.sp->L : a.sp->pos + 1) + a.L_add;
  int per = (L + a.splits - 1) / a.splits;
  per = (per + 15) & ~15;
  const int kbeg = min(L, split * per), kend = min(L, kbeg + per);
  const int nst = (kend - kbeg + kKeys - 1) / kKeys;

  if (nst > 0) issue_kv<HD>(a, head, kb0, vb0, kbeg, kend);
  cp_async_commit();

  // queries -> f16 hi / lo (rows >= T are zero)
  for (int i = threadIdx.x; i < 16 * HD; i += kThreads) {
    const int t = i / HD, d = i - t * HD;
    float x = t < T ? __ldcg(a.Q + (size_t)t * a.ldq + head * HD + d) : 0.f;
    __half h, l;
    split_f16(x, h, l);
    reinterpret_cast<__half *>(smem + (qhi - sbase))[t * QS + d] = h;
    reinterpret_cast<__half *>(smem + (qlo - sbase))[t * QS + d] = l;
  }

  float o[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};

  for (int st = 0; st < nst; ++st) {
    const uint32_t kb = (st & 1) ? kb1 : kb0, vb = (st & 1) ? vb1 : vb0;
    if (st + 1 < nst) issue_kv<HD>(a, head, (st & 1) ? kb0 : kb1, (st & 1) ? vb0 : vb1, kbeg + (st + 1) * kKeys, kend);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    // scores for keys 16w .. 16w+15 of this stage
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int c = 0; c < HD / 64; ++c) {
      uint4 blo[2], bhi[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = 16 * w + 8 * j + g;
        blo[j] = lds128(kb + kslot(r, 8 * c + q, HD));
        bhi[j] = lds128(kb + kslot(r, 8 * c + 4 + q, HD));
      }
      const uint32_t r0 = (uint32_t)(g * QS + 64 * c + 8 * q) * 2, r1 = r0 + 8 * QS * 2;
      const uint4 h0 = lds128(qhi + r0), h1 = lds128(qhi + r1), h2 = lds128(qhi + r0 + 64), h3 = lds128(qhi + r1 + 64);
      const uint4 l0 = lds128(qlo + r0), l1 = lds128(qlo + r1), l2 = lds128(qlo + r0 + 64), l3 = lds128(qlo + r1 + 64);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          mma_f16(s[j], word(h0, jj), word(h1, jj), word(h2, jj), word(h3, jj), word(blo[j], jj), word(bhi[j], jj));
          mma_f16(s[j], word(l0, jj), word(l1, jj), word(l2, jj), word(l3, jj), word(blo[j], jj), word(bhi[j], jj));
        }
    }
    // mask, scale into the log2 domain, online softmax (rows g and g + 8)
    const int key0 = kbeg + st * kKeys + 16 * w;
    float rmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = key0 + 8 * j + 2 * q + (e & 1);
        s[j][e] = key < kend ? s[j][e] * a.scale_log2 : -INFINITY;
        rmax[e >> 1] = fmaxf(rmax[e >> 1], s[j][e]);
      }
    float alpha[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      rmax[h] = fmaxf(rmax[h], __shfl_xor_sync(0xffffffffu, rmax[h], 1));
      rmax[h] = fmaxf(rmax[h], __shfl_xor_sync(0xffffffffu, rmax[h], 2));
      const float mn = fmaxf(m_r[h], rmax[h]);
      alpha[h] = mn == -INFINITY ? 1.f : exp2f(m_r[h] - mn);
      m_r[h] = mn;
    }
    float rsum[2] = {0.f, 0.f};
    uint32_t ph[4], pl[4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float mm = m_r[e >> 1];
        p[e] = mm == -INFINITY ? 0.f : exp2f(s[j][e] - mm);
        rsum[e >> 1] += p[e];
      }
      __half h[4], l[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) split_f16(p[e], h[e], l[e]);
      ph[2 * j] = pack_f16(h[0], h[1]);      // row g
      ph[2 * j + 1] = pack_f16(h[2], h[3]);  // row g + 8
      pl[2 * j] = pack_f16(l[0], l[1]);
      pl[2 * j + 1] = pack_f16(l[2], l[3]);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      rsum[h] += __shfl_xor_sync(0xffffffffu, rsum[h], 1);
      rsum[h] += __shfl_xor_sync(0xffffffffu, rsum[h], 2);
      l_r[h] = l_r[h] * alpha[h] + rsum[h];
    }
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      o[i][0] *= alpha[0]; o[i][1] *= alpha[0];
      o[i][2] *= alpha[1]; o[i][3] *= alpha[1];
    }
    // O += P V: A = P (16 rows x 16 keys), B = V (16 keys x 8 dims) via ldmatrix.trans
    const int mi = lane >> 3, ri = lane & 7;
    const int vrow = 16 * w + (mi & 1) * 8 + ri;
#pragma unroll
    for (int i = 0; i < NT; i += 2) {
      const int u = i + (mi >> 1);  // 16-byte unit = 8 dims
      uint32_t b0, b1, b2, b3;
      ldsm_x4_trans(vb + vslot(vrow, u, HD), b0, b1, b2, b3);
      mma_f16(o[i], ph[0], ph[1], ph[2], ph[3], b0, b1);
      mma_f16(o[i], pl[0], pl[1], pl[2], pl[3], b0, b1);
      mma_f16(o[i + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
      mma_f16(o[i + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  __syncthreads();

  // merge the 4 warps: merge[w][16 rows][HD] and (m, l) per warp and row
  float *mo = merge;                       // [4][16][HD]
  float *mml = merge + 4 * 16 * HD;        // [4][16][2]
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const int d = 8 * i + 2 * q;
    mo[(w * 16 + g) * HD + d] = o[i][0];
    mo[(w * 16 + g) * HD + d + 1] = o[i][1];
    mo[(w * 16 + g + 8) * HD + d] = o[i][2];
    mo[(w * 16 + g + 8) * HD + d + 1] = o[i][3];
  }
  if (q == 0) {
    mml[(w * 16 + g) * 2] = m_r[0];
    mml[(w * 16 + g) * 2 + 1] = l_r[0];
    mml[(w * 16 + g + 8) * 2] = m_r[1];
    mml[(w * 16 + g + 8) * 2 + 1] = l_r[1];
  }
  __syncthreads();
  float *po = a.part_o + ((size_t)(head * a.splits + split) * kMaxT) * HD;
  float2 *pml = a.part_ml + (size_t)(head * a.splits + split) * kMaxT;
  for (int i = threadIdx.x; i < T * (HD / 4); i += kThreads) {
    const int t = i / (HD / 4), d = 4 * (i - t * (HD / 4));
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < 4; ++ww) M = fmaxf(M, mml[(ww * 16 + t) * 2]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lsum = 0.f;
#pragma unroll
    for (int ww = 0; ww < 4; ++ww) {
      const float mw = mml[(ww * 16 + t) * 2];
      const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
      const float *src = mo + (ww * 16 + t) * HD + d;
      acc.x += f * src[0];
      acc.y += f * src[1];
      acc.z += f * src[2];
      acc.w += f * src[3];
      lsum += f * mml[(ww * 16 + t) * 2 + 1];
    }
    __stcg(reinterpret_cast<float4 *>(po + t * HD + d), acc);
    if (d == 0) __stcg(pml + t, make_float2(M, lsum));
  }

  // the last split of this head combines all splits in order
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atomicAdd(a.tickets + head, 1);
    s_last = old == a.splits - 1;
    if (s_last) atomicExch(a.tickets + head, 0);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float *pob = a.part_o + (size_t)head * a.splits * kMaxT * HD;
  const float2 *pmb = a.part_ml + (size_t)head * a.splits * kMaxT;
  // (max, sum) of every split and row -> shared memory, then per-row weights
  float *fm_ = merge;                      // [splits][16] weight of split sp for row t
  float *fl_ = merge + a.splits * 16;      // [splits][16] partial sums
  for (int i = threadIdx.x; i < a.splits * T; i += kThreads) {
    const int sp = i / T, t = i - sp * T;
    const float2 ml = __ldcg(pmb + sp * kMaxT + t);
    fm_[sp * 16 + t] = ml.x;
    fl_[sp * 16 + t] = ml.y;
  }
  __syncthreads();
  if (threadIdx.x < T) {
    const int t = threadIdx.x;
    float M = -INFINITY;
    for (int sp = 0; sp < a.splits; ++sp) M = fmaxf(M, fm_[sp * 16 + t]);
    float lsum = 0.f;
    for (int sp = 0; sp < a.splits; ++sp) {
      const float mw = fm_[sp * 16 + t];
      const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
      fm_[sp * 16 + t] = f;
      lsum += f * fl_[sp * 16 + t];
    }
    const float inv = 1.f / lsum;
    for (int sp = 0; sp < a.splits; ++sp) fm_[sp * 16 + t] *= inv;
  }
  __syncthreads();
  // out[t][4 d4 .. 4 d4 + 3] = sum over splits of weight * partial O (independent vector loads)
  for (int i = threadIdx.x; i < T * (HD / 4); i += kThreads) {
    const int t = i / (HD / 4), d4 = i - t * (HD / 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int sp = 0; sp < a.splits; ++sp) {
      const float f = fm_[sp * 16 + t];
      const float4 v = __ldcg(reinterpret_cast<const float4 *>(pob + ((size_t)sp * kMaxT + t) * HD) + d4);
      acc.x += f * v.x;
      acc.y += f * v.y;
      acc.z += f * v.z;
      acc.w += f * v.w;
    }
    *reinterpret_cast<float4 *>(a.out + (size_t)t * a.ldo + head * HD + 4 * d4) = acc;
  }
}

cudaError_t launch_attn(const AttnArgs &a, cudaStream_t st, bool pdl) {
  const int HD = a.hd;
  const size_t tile = (size_t)kKeys * HD * 2;
  size_t smem = 4 * tile + 2 * 16 * (HD + 32) * 2;
  const size_t merge = (size_t)4 * 16 * HD * 4 + 4 * 16 * 2 * 4;
  if (merge > smem) smem = merge;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_heads, a.splits, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e;
  if (HD == 128) {
    e = cudaFuncSetAttribute(attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, attn_kernel<128>, a);
  }
  e = cudaFuncSetAttribute(attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, attn_kernel<64>, a);
}

}  // namespace fm
