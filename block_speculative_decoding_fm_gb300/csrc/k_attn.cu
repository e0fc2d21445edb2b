// k_attn.cu -- cross-attention of the draft block over the context cache.
//
// Computes, per head h and block row t < T <= 16,
//   O[t] = softmax_j(q_t . k_j / sqrt(hd)) v_j   over cache rows j < L, no mask,
// as the pages do with one workgroup per (head, row) and all scores in shared
// memory (flashmap_drafter.js ``attn``, L <= 4096).  Here the keys are split
// across the CTAs of one thread-block cluster per head (flash-decoding): each
// CTA streams its share of the head-major f16 cache through shared memory with
// cp.async (rows that no kernel of the current call writes are requested before
// griddepcontrol.wait), computes scores and P.V on the tensor cores (f16
// m16n8k16, queries and probabilities split into f16 hi + lo), keeps an online
// softmax (running max / sum, rescaled as the MTP head attention kernel on
// ternary_bonsai_2_mtp.js does), and the cluster merges its partial results
// through distributed shared memory in a fixed order.  Any L is handled.
#include <cooperative_groups.h>

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

// stage rows [rlo, rhi) of the 64-key tile starting at k0 (rows past kend are zero-filled)
template <int HD>
__device__ __forceinline__ void issue_kv(const AttnArgs &a, int head, uint32_t kbuf, uint32_t vbuf, int k0,
                                         int kend, int rlo = 0, int rhi = kKeys) {
  constexpr int U = HD / 8;  // 16-byte units per row
  const __half *kb = a.Kc + (size_t)head * a.max_ctx * HD;
  const __half *vb = a.Vc + (size_t)head * a.max_ctx * HD;
  for (int i = threadIdx.x + rlo * U; i < rhi * U; i += kThreads) {
    const int r = i / U, u = i - r * U;
    const int key = k0 + r;
    const bool ok = key < kend;
    const size_t off = (size_t)(ok ? key : 0) * HD + u * 8;
    cp_async16(kbuf + kslot(r, u, HD), kb + off, ok ? 16u : 0u);
    cp_async16(vbuf + vslot(r, u, HD), vb + off, ok ? 16u : 0u);
  }
}

}  // namespace

template <int HD, int NS>
__global__ void __launch_bounds__(kThreads) fm_attn_decode_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int NT = HD / 8;        // n8 tiles of the output
  constexpr int QS = HD + 32;       // f16 row stride of the query tile (64-byte pad)
  const int head = blockIdx.x, split = blockIdx.y;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t tile_bytes = kKeys * HD * 2;
  auto kbuf = [&](int i) { return sbase + 2 * i * tile_bytes; };  // NS stages of (K tile, V tile)
  auto vbuf = [&](int i) { return sbase + (2 * i + 1) * tile_bytes; };
  const uint32_t kb0 = kbuf(0), vb0 = vbuf(0);
  const uint32_t qhi = sbase + 2 * NS * tile_bytes, qlo = qhi + 16 * QS * 2;
  float *merge = reinterpret_cast<float *>(smem);  // reused after the key loop

  pdl_trigger();
  // the per-call values were uploaded before the chain started
  const int L = (a.L_src == 0 ? a.sp->L : a.sp->pos + 1) + a.L_add;
  int per = (L + a.splits - 1) / a.splits;
  per = (per + 15) & ~15;
  const int kbeg = min(L, split * per), kend = min(L, kbeg + per);
  const int nst = (kend - kbeg + kKeys - 1) / kKeys;
  // rows below `stable` are not written by this call's kernels: the first NS - 1
  // stages' stable rows are requested before griddepcontrol.wait, the rest after it
  const int stable = a.sp->stable;
  int pre[NS];
#pragma unroll
  for (int st = 0; st < NS - 1; ++st) {
    pre[st] = st < nst ? max(0, min(kKeys, stable - (kbeg + st * kKeys))) : 0;
    if (pre[st] > 0) issue_kv<HD>(a, head, kbuf(st), vbuf(st), kbeg + st * kKeys, kend, 0, pre[st]);
  }
  pdl_wait();
  const int T = a.T_const > 0 ? a.T_const : a.sp->T;
#pragma unroll
  for (int st = 0; st < NS - 1; ++st) {
    if (st < nst && pre[st] < kKeys) issue_kv<HD>(a, head, kbuf(st), vbuf(st), kbeg + st * kKeys, kend, pre[st], kKeys);
    cp_async_commit();   // one group per stage, as the main loop expects
  }

  // queries -> f16 hi / lo (rows >= T are zero): every load in flight before the first is used
  {
    constexpr int Q4 = 16 * HD / 4 / kThreads;   // float4 per thread
    float4 xq[Q4];
#pragma unroll
    for (int j = 0; j < Q4; ++j) {
      const int i = threadIdx.x + j * kThreads;
      const int t = i / (HD / 4), d = 4 * (i - t * (HD / 4));
      xq[j] = t < T ? __ldcg(reinterpret_cast<const float4 *>(a.Q + (size_t)t * a.ldq + head * HD + d))
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < Q4; ++j) {
      const int i = threadIdx.x + j * kThreads;
      const int t = i / (HD / 4), d = 4 * (i - t * (HD / 4));
      uint2 hv, lv;
      split2_f16(xq[j].x, xq[j].y, hv.x, lv.x);
      split2_f16(xq[j].z, xq[j].w, hv.y, lv.y);
      *reinterpret_cast<uint2 *>(smem + (qhi - sbase) + (size_t)(t * QS + d) * 2) = hv;
      *reinterpret_cast<uint2 *>(smem + (qlo - sbase) + (size_t)(t * QS + d) * 2) = lv;
    }
  }

  float o[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};

  for (int st = 0; st < nst; ++st) {
    const uint32_t kb = kbuf(st % NS), vb = vbuf(st % NS);
    const int nx = st + NS - 1;
    if (nx < nst) issue_kv<HD>(a, head, kbuf(nx % NS), vbuf(nx % NS), kbeg + nx * kKeys, kend);
    cp_async_commit();
    cp_async_wait<NS - 1>();
    __syncthreads();

    // scores for keys 16w .. 16w+15 of this stage (four independent chains per n-tile)
    float sp[2][4][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int u = 0; u < 4; ++u) sp[j][u][0] = sp[j][u][1] = sp[j][u][2] = sp[j][u][3] = 0.f;
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
          const int ch = (jj & 1) * 2;
          mma_f16(sp[j][ch], word(h0, jj), word(h1, jj), word(h2, jj), word(h3, jj), word(blo[j], jj), word(bhi[j], jj));
          mma_f16(sp[j][ch + 1], word(l0, jj), word(l1, jj), word(l2, jj), word(l3, jj), word(blo[j], jj),
                  word(bhi[j], jj));
        }
    }
    float s[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[j][e] = (sp[j][0][e] + sp[j][2][e]) + (sp[j][1][e] + sp[j][3][e]);
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
      split2_f16(p[0], p[1], ph[2 * j], pl[2 * j]);          // row g
      split2_f16(p[2], p[3], ph[2 * j + 1], pl[2 * j + 1]);  // row g + 8
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
  // this CTA's partial (unnormalised O, running max in the log2 domain, sum) per row
  float *co = mml + 4 * 16 * 2;            // [16][HD]
  float *cml = co + 16 * HD;               // [16][2]
  for (int i = threadIdx.x; i < 16 * (HD / 4); i += kThreads) {
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
    *reinterpret_cast<float4 *>(co + t * HD + d) = acc;
    if (d == 0) {
      cml[t * 2] = M;
      cml[t * 2 + 1] = lsum;
    }
  }
  // merge the splits of this head through distributed shared memory: rank r
  // finishes rows t = r, r + splits, ... reading every CTA's partial in rank order
  cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
  cluster.sync();
  const int rank = (int)cluster.block_rank();
  const int ns = a.splits;
  constexpr int PL = HD / 32;  // values per lane
  constexpr int kBatch = 8;   // up to this many ranks: every remote load in flight before any is used
  for (int t = rank + ns * w; t < T; t += ns * (kThreads / 32)) {
    float M = -INFINITY;
    float lsum = 0.f;
    float acc[PL];
#pragma unroll
    for (int e = 0; e < PL; ++e) acc[e] = 0.f;
    if (ns <= kBatch) {
      float mr[kBatch], lr[kBatch], ov[kBatch][PL];
#pragma unroll
      for (int r = 0; r < kBatch; ++r) {
        mr[r] = -INFINITY;
        lr[r] = 0.f;
#pragma unroll
        for (int e = 0; e < PL; ++e) ov[r][e] = 0.f;
        if (r < ns) {
          const float *rml = cluster.map_shared_rank(cml, r);
          const float *ro = cluster.map_shared_rank(co, r) + t * HD + PL * lane;
          mr[r] = rml[t * 2];
          lr[r] = rml[t * 2 + 1];
#pragma unroll
          for (int e = 0; e < PL; ++e) ov[r][e] = ro[e];
        }
      }
#pragma unroll
      for (int r = 0; r < kBatch; ++r) M = fmaxf(M, mr[r]);
#pragma unroll
      for (int r = 0; r < kBatch; ++r) {   // rank order
        const float f = mr[r] == -INFINITY ? 0.f : exp2f(mr[r] - M);
        lsum += f * lr[r];
#pragma unroll
        for (int e = 0; e < PL; ++e) acc[e] += f * ov[r][e];
      }
    } else {
      for (int r = 0; r < ns; ++r) M = fmaxf(M, cluster.map_shared_rank(cml, r)[t * 2]);
      for (int r = 0; r < ns; ++r) {
        const float *rml = cluster.map_shared_rank(cml, r);
        const float mr = rml[t * 2];
        const float f = mr == -INFINITY ? 0.f : exp2f(mr - M);
        lsum += f * rml[t * 2 + 1];
        const float *ro = cluster.map_shared_rank(co, r) + t * HD + PL * lane;
#pragma unroll
        for (int e = 0; e < PL; ++e) acc[e] += f * ro[e];
      }
    }
    const float inv = 1.f / lsum;
    float *dst = a.out + (size_t)t * a.ldo + head * HD + PL * lane;
#pragma unroll
    for (int e = 0; e < PL; ++e) dst[e] = acc[e] * inv;
  }
  // no CTA leaves while a peer may still read its partials (the reads above are consumed)
  cluster_arrive_relaxed();
  cluster_wait_acquire();
}

cudaError_t launch_attn(const AttnArgs &a, int L_now, cudaStream_t st, bool pdl) {
  const int HD = a.hd;
  const size_t tile = (size_t)kKeys * HD * 2;
  // deeper ring when each CTA streams several key tiles (NS - 1 of them are requested
  // before griddepcontrol.wait); three stages (~106 KB) still start beside a GEMV CTA
  const int per_cta = (L_now + a.splits - 1) / a.splits;
  const int NS = per_cta > 4 * kKeys ? 4 : per_cta > kKeys ? 3 : 2;
  size_t smem = 2 * NS * tile + 2 * 16 * (HD + 32) * 2;
  const size_t merge = (size_t)4 * 16 * HD * 4 + 4 * 16 * 2 * 4 + (size_t)16 * HD * 4 + 16 * 2 * 4;
  if (merge > smem) smem = merge;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_heads, a.splits, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = a.splits;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  auto go = [&](auto kern) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (a.splits > 8) {   // clusters of up to 16 CTAs are an opt-in on this GPU
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    return cudaLaunchKernelEx(&cfg, kern, a);
  };
  if (HD == 128) return NS == 4 ? go(fm_attn_decode_kernel<128, 4>) : NS == 3 ? go(fm_attn_decode_kernel<128, 3>) : go(fm_attn_decode_kernel<128, 2>);
  return NS == 4 ? go(fm_attn_decode_kernel<64, 4>) : NS == 3 ? go(fm_attn_decode_kernel<64, 3>) : go(fm_attn_decode_kernel<64, 2>);
}

}  // namespace fm
