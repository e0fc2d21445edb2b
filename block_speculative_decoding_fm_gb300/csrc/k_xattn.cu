// k_xattn.cu -- attention of the draft block over a head-major f16 cache on the
// 5th-generation tensor cores (head dim 128).
//
// Computes, per head h and block row t < T <= 16,
//   O[t] = softmax_j(q_t . k_j / sqrt(hd)) v_j   over cache rows j < L, no mask,
// (flashmap_drafter.js ``attn`` / ``attnF16``; module-dflash.ts ``#layer``
// attends the same way over [context ++ block]).  The keys are split into
// ranges, one CTA per (head, range); a range is walked in 128-key tiles:
//   warp 0      one thread loads each tile's K and V with 2-D tensor copies
//               (128 keys x 64 dims per box, 128-byte swizzle) into two
//               mbarrier rings (three stages for multi-tile ranges), K one
//               tile ahead of V; tiles whose rows no kernel of the current call
//               writes are requested before griddepcontrol.wait;
//   warp 1      issues tcgen05.mma: S^T = K Q^T (M = 128 keys, N = 32: the 16
//               queries' f16 hi rows then lo rows, K = 128 dims) into a TMEM
//               slot, and O^T += V^T P^T (M = 128 dims, A = the V tile read
//               MN-major, N = 32: the probabilities' hi and lo rows, K = 128
//               keys) into the TMEM accumulator;
//   warps 2-5   one thread per key: read its scores from TMEM, form
//               p = exp2(s - m) against a per-query reference m shared by the
//               CTA, accumulate the row sums, and write p as f16 hi + lo into
//               the shared-memory B operand of the next P.V.  The reference is
//               the first tile's maximum; it moves (and the accumulator is
//               rescaled in TMEM) only when a score exceeds it by more than
//               2^8, so the online softmax costs no per-tile reduction (the
//               rescale-when-needed scheme of FlashAttention-4).
// Each CTA stores its unnormalised O, m and row sums; the last CTA of a head
// (atomic ticket) merges the ranges in order (deterministic) and writes O / l.
// A batched draft runs every sequence of the call in one launch (grid z), each
// over its own cache and context length, writing f16 rows for the next product.
// Every mbarrier wait is bounded; on expiry the kernel raises the error word,
// drains its copies and MMAs, frees its TMEM and returns.
#include <cooperative_groups.h>
#include <cuda.h>

#include "dev_common.cuh"
#include "fm_internal.h"
#include "tc_gemm.h"

namespace fm {

namespace {

constexpr int HD = 128;
constexpr int kTileKeys = 128;
constexpr int kBox = kTileKeys * 128;              // one 64-dim box of a tile: 16 KB
constexpr int kKV = 2 * kBox;                      // a K or V tile: 32 KB
constexpr int kQB = 32 * 128;                      // one 64-column chunk of a 32-row B operand: 4 KB
constexpr int kThreads = 192;
constexpr float kRescale = 8.f;                    // log2 of the growth a reference tolerates

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// MN-major operand with 128-byte swizzle: 64-element rows along M, 8-row atoms
// along K 1024 bytes apart (sbo), the next 64 elements of M lbo bytes further
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// byte offset of element (row, col) of a 32-row B operand, 64-column chunks 4 KB apart
__device__ __forceinline__ uint32_t b_slot(int row, int col) { return (uint32_t)(col >> 6) * kQB + sw128(row, col & 63); }

// Merge of the ranges' partials for this thread's items (item = query n, dims 4c .. 4c + 3;
// the thread takes items i, i + 128, ...): O = sum_r w[r][n] O_r in range order, PT items a
// thread and 16 / PT ranges per batch, so that 16 loads are in flight at a time.
template <int PT>
__device__ __forceinline__ void merge_ranges(const float *ho, const float *sw, int ns, int items, int i, float *out,
                                             __half *out16, int ldo, int head) {
  constexpr int RB = 16 / PT;
  float4 acc[PT];
#pragma unroll
  for (int q = 0; q < PT; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int r0 = 0; r0 < ns; r0 += RB) {
    float4 v[PT][RB];
#pragma unroll
    for (int q = 0; q < PT; ++q)
#pragma unroll
      for (int rr = 0; rr < RB; ++rr) {
        const int itm = i + 128 * q, r = r0 + rr;
        v[q][rr] = r < ns && itm < items
                       ? __ldcg(reinterpret_cast<const float4 *>(ho + ((size_t)r * 16 + itm / 32) * HD + 4 * (itm % 32)))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
    for (int q = 0; q < PT; ++q)
#pragma unroll
      for (int rr = 0; rr < RB; ++rr) {
        const int itm = i + 128 * q, r = r0 + rr;
        const float f = r < ns && itm < items ? sw[r * 16 + itm / 32] : 0.f;
        acc[q].x += f * v[q][rr].x;
        acc[q].y += f * v[q][rr].y;
        acc[q].z += f * v[q][rr].z;
        acc[q].w += f * v[q][rr].w;
      }
  }
#pragma unroll
  for (int q = 0; q < PT; ++q) {
    const int itm = i + 128 * q;
    if (itm >= items) continue;
    const size_t o = (size_t)(itm / 32) * ldo + head * HD + 4 * (itm % 32);
    if (out16) {
      const __half2 h01 = __floats2half2_rn(acc[q].x, acc[q].y), h23 = __floats2half2_rn(acc[q].z, acc[q].w);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t *>(&h01);
      pk.y = *reinterpret_cast<const uint32_t *>(&h23);
      *reinterpret_cast<uint2 *>(out16 + o) = pk;
    } else {
      *reinterpret_cast<float4 *>(out + o) = acc[q];
    }
  }
}

}  // namespace

// kNS: ring stages for K and for V.  kCluster: the ranges of a head form one thread-block
// cluster and merge through distributed shared memory (launched so when every range is one
// tile: the CTA is then small enough to start beside a linear-layer CTA under programmatic
// dependent launch); otherwise the last range of a head to finish merges them (ticket).
template <int kNS, bool kCluster>
__global__ void __launch_bounds__(kThreads, 1) fm_xattn_kernel(const __grid_constant__ XAttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - smem_u32(smem_raw));
  const uint32_t kring = base, vring = base + kNS * kKV;
  const uint32_t qbuf = vring + kNS * kKV;           // [2 chunks][32 rows][128 B]
  const uint32_t pbuf = qbuf + 2 * kQB;              // [2 buffers][2 chunks][32 rows][128 B]
  float *red = reinterpret_cast<float *>(gbase + (pbuf - base) + 4 * kQB);   // [4 warps][16]
  const uint32_t bars = smem_u32(red + 4 * 16);
  auto kfull = [&](int s) { return bars + 8 * s; };
  auto kempty = [&](int s) { return bars + 8 * (kNS + s); };
  auto vfull = [&](int s) { return bars + 8 * (2 * kNS + s); };
  auto vempty = [&](int s) { return bars + 8 * (3 * kNS + s); };
  const uint32_t b2 = bars + 8 * (4 * kNS);
  auto sfull = [&](int b) { return b2 + 8 * b; };
  auto sfree = [&](int b) { return b2 + 8 * (2 + b); };
  auto pfull = [&](int b) { return b2 + 8 * (4 + b); };
  auto pfree = [&](int b) { return b2 + 8 * (6 + b); };
  const uint32_t qfull = b2 + 64, odone = b2 + 72, tslot = b2 + 80;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.x, split = blockIdx.y, ns = gridDim.y;
  const bool batch = a.bz_call != nullptr;
  const int z = blockIdx.z;

  // the per-call values were uploaded before the chain started
  const int L = batch ? a.bz_L[z] : (a.L_src == 0 ? a.sp->L : a.sp->pos + 1) + a.L_add;
  // this launch slot's query / output rows, partials and ticket
  const int qrow0 = batch ? a.bz_call[z] * a.T_const : 0;
  const size_t zslot = batch ? (size_t)z * a.n_heads + head : (size_t)head;
  // whole 128-key tiles dealt out evenly: range r takes tiles [tb, tb + ntiles)
  const int ntot = (L + kTileKeys - 1) / kTileKeys;
  const int tq = ntot / ns, trem = ntot - tq * ns;
  const int tb = split * tq + min(split, trem);
  const int ntiles = tq + (split < trem ? 1 : 0);
  const int kbeg = min(L, tb * kTileKeys), kend = min(L, (tb + ntiles) * kTileKeys);
  // tensor-map rows of this range's first key (K) and the V plane's offset from it
  const int kv_base = batch ? ((a.bz_seq[z] * a.n_layers + a.layer) * 2) * a.n_heads * a.max_ctx : 0;
  const int row0 = kv_base + head * a.max_ctx + kbeg;
  const int voff = batch ? a.n_heads * a.max_ctx : 0;

  pdl_trigger();
  if (threadIdx.x == 0) {
    // the tensor maps' descriptors are fetched while the barriers are set up
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&a.tm_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&a.tm_v)) : "memory");
    for (int s = 0; s < kNS; ++s) {
      mbar_init(kfull(s), 1);
      mbar_init(kempty(s), 1);
      mbar_init(vfull(s), 1);
      mbar_init(vempty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sfull(b), 1);
      mbar_init(sfree(b), 128);
      mbar_init(pfull(b), 128);
      mbar_init(pfree(b), 1);
    }
    mbar_init(qfull, 128);
    mbar_init(odone, 1);
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc<128>(tslot);   // S slots at columns 0 and 32, O at 64
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = lds32(tslot);

  if (warp == 0) {
    if (lane == 0) {
      // tiles below `stable` (rows no kernel of this call writes) go before griddepcontrol.wait
      const int stable = batch ? 0 : a.sp->stable;
      // K runs one tile ahead of V (the MMA warp issues QK(t + 1) before P.V(t)); each ring
      // slot is refilled as soon as the MMAs that read it have completed
      auto load_k = [&](int t) -> bool {
        const int s = t % kNS;
        if (!mbar_wait_bounded(kempty(s), ((t / kNS) & 1) ^ 1, a.err)) return false;
        mbar_expect_tx(kfull(s), kKV);
        tma_2d(kring + s * kKV, &a.tm_k, 0, row0 + t * kTileKeys, kfull(s));
        tma_2d(kring + s * kKV + kBox, &a.tm_k, 64, row0 + t * kTileKeys, kfull(s));
        return true;
      };
      auto load_v = [&](int t) -> bool {
        const int s = t % kNS;
        if (!mbar_wait_bounded(vempty(s), ((t / kNS) & 1) ^ 1, a.err)) return false;
        mbar_expect_tx(vfull(s), kKV);
        tma_2d(vring + s * kKV, &a.tm_v, 0, row0 + voff + t * kTileKeys, vfull(s));
        tma_2d(vring + s * kKV + kBox, &a.tm_v, 64, row0 + voff + t * kTileKeys, vfull(s));
        return true;
      };
      int nk = 0, nv = 0;
      // tiles below `stable` (rows no kernel of this call writes) go before griddepcontrol.wait
      while (nk < ntiles && nk < kNS && kbeg + (nk + 1) * kTileKeys <= stable) {
        load_k(nk);
        ++nk;
      }
      while (nv < nk) {
        load_v(nv);
        ++nv;
      }
      pdl_wait();
      while (nv < ntiles) {
        if (nk < ntiles && nk <= nv + 1) {
          if (!load_k(nk)) break;
          ++nk;
        } else {
          if (!load_v(nv)) break;
          ++nv;
        }
      }
      // the CTA leaves only after its copies have landed
      for (int t = nk > kNS ? nk - kNS : 0; t < nk; ++t) mbar_wait_drain(kfull(t % kNS), (t / kNS) & 1);
      for (int t = nv > kNS ? nv - kNS : 0; t < nv; ++t) mbar_wait_drain(vfull(t % kNS), (t / kNS) & 1);
    } else {
      pdl_wait();
    }
  } else if (warp == 1) {
    pdl_wait();
    // whole-warp issue loop; an elected lane issues each MMA and commit
    constexpr uint32_t IQK = umma_idesc(128, 32, false);
    constexpr uint32_t IPV = umma_idesc(128, 32, false) | (1u << 15);   // A (V^T) MN-major
    const uint32_t o_tm = tmem + 64;
    bool ok = mbar_wait_warp(qfull, 0, a.err);
    auto qk = [&](int t) -> bool {
      const int s = t % kNS, b = t & 1;
      if (!mbar_wait_warp(kfull(s), (t / kNS) & 1, a.err)) return false;
      if (!mbar_wait_warp(sfree(b), ((t >> 1) & 1) ^ 1, a.err)) return false;
      tc_fence_after();
      const uint32_t kt = kring + s * kKV;
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint64_t ad = umma_desc_sw128(kt + (kk >> 2) * kBox) + 2 * (kk & 3);
        const uint64_t bd = umma_desc_sw128(qbuf + (kk >> 2) * kQB) + 2 * (kk & 3);
        umma_ss_elect(tmem + 32 * b, ad, bd, IQK, kk > 0 ? 1u : 0u);
      }
      umma_commit_elect(kempty(s));
      umma_commit_elect(sfull(b));
      return true;
    };
    if (ok && ntiles > 0) ok = qk(0);
    for (int t = 0; ok && t < ntiles; ++t) {
      if (t + 1 < ntiles && !qk(t + 1)) break;
      const int s = t % kNS, b = t & 1;
      if (!mbar_wait_warp(pfull(b), (t >> 1) & 1, a.err)) break;
      if (!mbar_wait_warp(vfull(s), (t / kNS) & 1, a.err)) break;
      tc_fence_after();
      const uint32_t vt = vring + s * kKV;
#pragma unroll
      for (int kk = 0; kk < kTileKeys / 16; ++kk) {
        const uint64_t ad = desc_mn_sw128(vt + kk * 2048, kBox, 1024);
        const uint64_t bd = umma_desc_sw128(pbuf + b * 2 * kQB + (kk >> 2) * kQB) + 2 * (kk & 3);
        umma_ss_elect(o_tm, ad, bd, IPV, (t | kk) ? 1u : 0u);
      }
      umma_commit_elect(vempty(s));
      umma_commit_elect(pfree(b));
    }
    umma_commit_elect(odone);   // every MMA issued above has completed when this arrives
  } else {
    // ---- one thread per key of a tile (TMEM lane quarter = warp % 4) ----
    const int quad = warp & 3;
    const int j = quad * 32 + lane;                 // key within the tile, and dim in the epilogue
    const int i = threadIdx.x - 64;                 // 0 .. 127 within this group
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    pdl_wait();
    const int T = a.T_const > 0 ? a.T_const : a.sp->T;
    // queries, pre-scaled into the log2 domain, as f16 hi (rows 0..15) and lo (rows 16..31)
    {
      const int n = i >> 3, d0 = (i & 7) * 16;
      float x[16];
      if (n < T) {
        const float4 *src = reinterpret_cast<const float4 *>(a.Q + (size_t)(qrow0 + n) * a.ldq + head * HD + d0);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float4 v = __ldcg(src + u);
          x[4 * u] = v.x * a.scale_log2;
          x[4 * u + 1] = v.y * a.scale_log2;
          x[4 * u + 2] = v.z * a.scale_log2;
          x[4 * u + 3] = v.w * a.scale_log2;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] = 0.f;
      }
#pragma unroll
      for (int h8 = 0; h8 < 2; ++h8) {
        uint4 hv, lv;
        split2_f16(x[8 * h8 + 0], x[8 * h8 + 1], hv.x, lv.x);
        split2_f16(x[8 * h8 + 2], x[8 * h8 + 3], hv.y, lv.y);
        split2_f16(x[8 * h8 + 4], x[8 * h8 + 5], hv.z, lv.z);
        split2_f16(x[8 * h8 + 6], x[8 * h8 + 7], hv.w, lv.w);
        const int d = d0 + 8 * h8;
        *reinterpret_cast<uint4 *>(gbase + (qbuf - base) + b_slot(n, d)) = hv;
        *reinterpret_cast<uint4 *>(gbase + (qbuf - base) + b_slot(16 + n, d)) = lv;
      }
    }
    fence_proxy_async();
    mbar_arrive(qfull);

    float m_ref[16], l_part[16];
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      m_ref[n] = -INFINITY;
      l_part[n] = 0.f;
    }
    // this thread's P column in the B operand: key j, rows n (hi) and 16 + n (lo)
    uint32_t pofs[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) pofs[r] = b_slot(r, j);
    for (int t = 0; t < ntiles; ++t) {
      const int b = t & 1;
      // scores: never break out of the loop (the named barriers below must stay matched);
      // after a failed wait the values are garbage and the error word is raised
      mbar_wait_bounded(sfull(b), (t >> 1) & 1, a.err);
      tc_fence_after();
      float c[32];
      tmem_ld32(tmem + lane_off + 32 * b, c);
      tc_fence_before();
      mbar_arrive(sfree(b));
      const bool live = kbeg + t * kTileKeys + j < kend;
      float s[16];
#pragma unroll
      for (int n = 0; n < 16; ++n) s[n] = live ? c[n] + c[16 + n] : -INFINITY;
      bool grow = false;
#pragma unroll
      for (int n = 0; n < 16; ++n) grow |= s[n] > m_ref[n] + kRescale;
      if (bar_any(1, 128, grow)) {
        // a new reference: the CTA's maximum so far, per query (first tile, or a rare jump)
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          const float w = warp_max(s[n]);
          if (lane == n) red[quad * 16 + n] = w;
        }
        named_sync(1, 128);
        float alpha[16];
        bool any_scale = false;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          const float tm = fmaxf(fmaxf(red[n], red[16 + n]), fmaxf(red[32 + n], red[48 + n]));
          const float mn = fmaxf(m_ref[n], tm);
          alpha[n] = m_ref[n] == -INFINITY ? 1.f : exp2f(m_ref[n] - mn);
          any_scale |= m_ref[n] != -INFINITY && mn != m_ref[n];
          m_ref[n] = mn;
        }
        named_sync(1, 128);   // red is read by every thread before it is written again
        if (any_scale && t > 0) {
          // rescale the accumulator once every P.V issued so far has completed
          mbar_wait_bounded(pfree((t - 1) & 1), ((t - 1) >> 1) & 1, a.err);
          tc_fence_after();
          float o[32];
          tmem_ld32(tmem + lane_off + 64, o);
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            o[n] *= alpha[n];
            o[16 + n] *= alpha[n];
          }
          tmem_st32(tmem + lane_off + 64, o);
        }
#pragma unroll
        for (int n = 0; n < 16; ++n) l_part[n] *= alpha[n];
      }
      // the P buffer b was last read by the P.V of tile t - 2
      mbar_wait_bounded(pfree(b), ((t >> 1) & 1) ^ 1, a.err);
      uint8_t *pb = gbase + (pbuf - base) + b * 2 * kQB;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        const float p = s[n] == -INFINITY ? 0.f : exp2f(s[n] - m_ref[n]);
        l_part[n] += p;
        const __half ph = __float2half_rn(p);
        const __half pl = __float2half_rn(p - __half2float(ph));
        *reinterpret_cast<__half *>(pb + pofs[n & 7] + (n >> 3) * 1024) = ph;
        *reinterpret_cast<__half *>(pb + pofs[n & 7] + (2 + (n >> 3)) * 1024) = pl;
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(pfull(b));
    }
    // row sums over the CTA's keys
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      const float w = warp_sum(l_part[n]);
      if (lane == n) red[quad * 16 + n] = w;
    }
    mbar_wait_drain(odone, 0);
    tc_fence_after();
    float o[32];
    tmem_ld32(tmem + lane_off + 64, o);
    named_sync(1, 128);
    // this range's partial: unnormalised O (dim j), the reference m and the row sum l
    if constexpr (kCluster) {
      // into this CTA's shared memory: the K ring is free (every tile has been consumed)
      float *co = reinterpret_cast<float *>(gbase);
      float2 *cml = reinterpret_cast<float2 *>(gbase + 16 * HD * sizeof(float));
#pragma unroll
      for (int n = 0; n < 16; ++n) co[n * HD + j] = ntiles ? o[n] + o[16 + n] : 0.f;
#pragma unroll
      for (int n = 0; n < 16; ++n)
        if (i == n) {
          const float l = red[n] + red[16 + n] + red[32 + n] + red[48 + n];
          cml[n] = make_float2(ntiles ? m_ref[n] : -INFINITY, ntiles ? l : 0.f);
        }
    } else if (ns == 1) {
      // one range per head: the output directly, O / l (thread j: dim j of every query row)
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        if (n < T) {
          const float l = red[n] + red[16 + n] + red[32 + n] + red[48 + n];
          const float val = (o[n] + o[16 + n]) / l;
          const size_t off = (size_t)(qrow0 + n) * a.ldo + head * HD + j;
          if (a.out16)
            a.out16[off] = __float2half_rn(val);
          else
            a.out[off] = val;
        }
      }
    } else {
      float *po = a.part_o + (zslot * ns + split) * 16 * HD;
      float2 *pml = a.part_ml + (zslot * ns + split) * 16;
#pragma unroll
      for (int n = 0; n < 16; ++n)
        if (n < T) po[n * HD + j] = ntiles ? o[n] + o[16 + n] : 0.f;
#pragma unroll
      for (int n = 0; n < 16; ++n)
        if (i == n) {
          const float l = red[n] + red[16 + n] + red[32 + n] + red[48 + n];
          pml[n] = make_float2(ntiles ? m_ref[n] : -INFINITY, ntiles ? l : 0.f);
        }
      // publish: the group's stores are ordered before thread 0's fence and ticket
      named_sync(1, 128);
      __shared__ int last;
      if (i == 0) {
        __threadfence();
        const int old = atomicAdd(a.tickets + zslot, 1);
        const bool is_last = old == ns - 1;
        if (is_last) atomicExch(a.tickets + zslot, 0);
        last = is_last && !*reinterpret_cast<volatile int32_t *>(a.err);   // one verdict for the group
        if (last) __threadfence();
      }
      named_sync(1, 128);
      if (last) {
        // merge the ranges in order: O[t] = sum_r w_r O_r, w_r = 2^(m_r - M) / sum_r' 2^(m_r' - M) l_r'.
        // The K ring is free: it holds the (m, l) pairs and the weights.
        const float *ho = a.part_o + zslot * ns * 16 * HD;
        const float2 *hml = a.part_ml + zslot * ns * 16;
        float2 *sml = reinterpret_cast<float2 *>(gbase);
        float *sw = reinterpret_cast<float *>(gbase + kMaxXSplits * 16 * sizeof(float2));
        for (int idx = i; idx < ns * 16; idx += 128) sml[idx] = __ldcg(hml + idx);
        named_sync(1, 128);
        if (i < 16) {
          float M = -INFINITY;
          for (int r = 0; r < ns; ++r) M = fmaxf(M, sml[r * 16 + i].x);
          float lsum = 0.f;
          for (int r = 0; r < ns; ++r) {
            const float2 ml = sml[r * 16 + i];
            const float f = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
            sw[r * 16 + i] = f;
            lsum += f * ml.y;
          }
          const float inv = 1.f / lsum;
          for (int r = 0; r < ns; ++r) sw[r * 16 + i] *= inv;
        }
        named_sync(1, 128);
        // items (query n, 4 dims): T * 32 of them over the group's 128 threads
        const int items = T * (HD / 4);
        float *out = a.out16 ? nullptr : a.out + (size_t)qrow0 * a.ldo;
        __half *out16 = a.out16 ? a.out16 + (size_t)qrow0 * a.ldo : nullptr;
        switch ((items + 127) / 128) {
          case 1: merge_ranges<1>(ho, sw, ns, items, i, out, out16, a.ldo, head); break;
          case 2: merge_ranges<2>(ho, sw, ns, items, i, out, out16, a.ldo, head); break;
          case 3: merge_ranges<3>(ho, sw, ns, items, i, out, out16, a.ldo, head); break;
          default: merge_ranges<4>(ho, sw, ns, items, i, out, out16, a.ldo, head); break;
        }
      }
    }
  }
  if constexpr (kCluster) {
    // rank r finishes rows r, r + ns, ... from every rank's partial, in rank order
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    cluster_arrive_release();
    cluster_wait_acquire();
    if (warp >= 2) {
      const int j = (warp & 3) * 32 + lane;
      const int T = a.T_const > 0 ? a.T_const : a.sp->T;
      const int rank = (int)cluster.block_rank();
      float *co = reinterpret_cast<float *>(gbase);
      float2 *cml = reinterpret_cast<float2 *>(gbase + 16 * HD * sizeof(float));
      for (int n = rank; n < T; n += ns) {
        float mr[16], lr[16], ov[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          mr[r] = -INFINITY;
          lr[r] = 0.f;
          ov[r] = 0.f;
          if (r < ns) {
            const float2 ml = cluster.map_shared_rank(cml, r)[n];
            mr[r] = ml.x;
            lr[r] = ml.y;
            ov[r] = cluster.map_shared_rank(co, r)[n * HD + j];
          }
        }
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < 16; ++r) M = fmaxf(M, mr[r]);
        float acc = 0.f, lsum = 0.f;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const float f = mr[r] == -INFINITY ? 0.f : exp2f(mr[r] - M);
          lsum += f * lr[r];
          acc += f * ov[r];
        }
        a.out[(size_t)n * a.ldo + head * HD + j] = acc / lsum;
      }
    }
    // no CTA leaves while a peer may still read its partial
    cluster_arrive_relaxed();
    cluster_wait_acquire();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_free<128>(tmem);
  }
}

size_t xattn_smem_bytes(int stages) { return 1024 + 2 * (size_t)stages * kKV + 2 * kQB + 4 * kQB + 4 * 16 * 4 + 256; }

cudaError_t launch_xattn(const XAttnArgs &a, int stages, bool cluster, cudaStream_t st, bool pdl) {
  if (a.splits < 1 || a.splits > kMaxXSplits || (stages != 1 && stages != 3) || (cluster && a.splits > 16))
    return cudaErrorInvalidValue;
  // several sequences per launch: ticket merge only, one query row block per sequence
  const int nz = a.bz_call ? a.n_z : 1;
  if (a.bz_call && (cluster || nz < 1 || !a.bz_seq || !a.bz_L || a.T_const < 1 || a.T_const > 16))
    return cudaErrorInvalidValue;
  const size_t smem = xattn_smem_bytes(stages);
  auto kern = cluster ? (stages == 1 ? fm_xattn_kernel<1, true> : fm_xattn_kernel<3, true>)
                      : (stages == 1 ? fm_xattn_kernel<1, false> : fm_xattn_kernel<3, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (cluster && a.splits > 8) {   // clusters of up to 16 CTAs are an opt-in
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_heads, a.splits, nz);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (cluster) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = a.splits;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// Clusters of `cluster` ranges that can run at once (one-stage ring, cluster merge); 0 on error.
int xattn_max_active_clusters(int cluster, int n_heads) {
  auto kern = fm_xattn_kernel<1, true>;
  const size_t smem = xattn_smem_bytes(1);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
      (cluster > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_heads, cluster, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = cluster;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

bool make_cache_map(CUtensorMap *map, const __half *plane, int n_heads, int max_ctx) {
  return make_tma_f16(map, plane, (uint64_t)n_heads * max_ctx, HD, kTileKeys);
}

}  // namespace fm
