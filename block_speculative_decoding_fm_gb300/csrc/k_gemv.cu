// k_gemv.cu -- the skinny weight-streaming GEMV of the drafter:
//   Y[t][m] = sum_k A[t][k] W[m][k],  t < T <= 32,  W bf16 [M][K] row-major.
//
// The pages run this product as gemvT17 / gemmBf16 in WGSL (flashmap_drafter.js,
// ``gemvT``: one weight read, token sums in registers).  On sm_103a:
//   * weights are stored pre-tiled (128 rows x 64 k, 16 KB, already in the
//     swizzled shared-memory order); a producer warp streams a CTA's tiles with
//     1-D bulk TMA copies into an mbarrier ring, issuing the first stages before
//     griddepcontrol.wait so a kernel's weights are in flight while its
//     predecessor is still finishing; consumer warps never block on each other
//     inside the main loop;
//   * the activations are transformed on the way in (RMSNorm, adaLN LayerNorm
//     modulate, a table row) and split into bf16 hi + lo, so the bf16 tensor
//     cores see f32-accurate operands: A*W = hi*W + lo*W, f32 accumulate;
//   * the contraction runs on the 5th-generation tensor cores: the MMA warp
//     runs the issue loop warp-wide and an elected lane issues tcgen05.mma
//     (M = 128 weight rows, N = the hi rows then the lo rows of the
//     activations, K = 16) from shared-memory operands in the 128-byte swizzle
//     layout into a TMEM accumulator; worker warps read it back with
//     tcgen05.ld;
//   * split-K across a thread-block cluster; the partial tiles are summed
//     through distributed shared memory in a fixed order (deterministic);
//   * fused epilogues: bias, exact GELU, gated residual + row statistics for
//     the next norm, per-head RMSNorm + interleaved-pair RoPE, f16 cache store,
//     gated GELU(tanh) FFN, and the block self-attention tail.
#include <cooperative_groups.h>

#include "linear_parts.cuh"

namespace cg = cooperative_groups;

namespace fm {

namespace {

struct Smem {
  uint32_t bbuf0, bbuf_stride;  // staged activation pieces (128-byte swizzle), double buffered
  float *cs_ptr;
  float *stat_mu, *stat_rs;     // [kMaxT]
};

}  // namespace

template <int MT>
__global__ void __launch_bounds__(kAll, 2) fm_linear_kernel(const __grid_constant__ GemvArgs a, const int S, const int U) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  constexpr int NR = 32 * MT;                 // B rows: hi rows then lo rows
  constexpr int BCH = NR * 128;               // bytes of one 64-column B chunk
  constexpr uint32_t IDESC = umma_idesc(128, NR, true);
  const int tile = blockIdx.x;
  const int m0 = tile * kTile;
  const int split = blockIdx.y;
  const int k_begin = split * a.Kc;
  const int nchunks = a.Kc / kChunk;
  const int cpp = a.Kp / kChunk;              // chunks per staged piece
  const int npieces = (nchunks + cpp - 1) / cpp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - smem_u32(smem_raw));
  const uint32_t ring = base;
  // a ring stage holds U consecutive chunks moved by one bulk copy (the copy engine
  // takes a roughly fixed time per copy, so larger copies stream faster)
  const int UB = U * kStageBytes;
  const int units = nchunks / U;
  Smem s;
  s.bbuf0 = ring + S * UB;
  s.bbuf_stride = cpp * BCH;
  s.cs_ptr = reinterpret_cast<float *>(gbase + S * UB + 2 * cpp * BCH);
  s.stat_mu = s.cs_ptr + 16 * MT * kCsStride;
  s.stat_rs = s.stat_mu + kMaxT;
  const uint32_t bars = smem_u32(s.stat_rs + kMaxT);
  auto full = [&](int i) { return bars + 8 * i; };
  auto empty = [&](int i) { return bars + 8 * (S + i); };
  const uint32_t bfull0 = bars + 8 * (2 * S), bempty0 = bfull0 + 16, accfull = bfull0 + 32;
  const uint32_t tslot = accfull + 8;
  const uint8_t *wsrc = a.Wt + ((size_t)tile * (a.K / kChunk) + k_begin / kChunk) * kStageBytes;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bfull0 + 8 * i, 1);
      mbar_init(bempty0 + 8 * i, 1);
    }
    mbar_init(accfull, 1);
    mbar_fence_init();
    // weights do not depend on earlier kernels: start streaming them now
    for (int j = 0; j < S && j < units; ++j) {
      mbar_expect_tx(full(j), UB);
      bulk_g2s(ring + j * UB, wsrc + (size_t)j * UB, UB, full(j));
    }
  }
  if (warp == 1) tmem_alloc<NR>(tslot);
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = lds32(tslot);
  pdl_wait();
  const int T = a.T_const > 0 ? a.T_const : a.sp->T;

  if (warp == 0) {
    // weights: refill a stage once the MMAs that read it have completed
    if (lane == 0) {
      int st = 0;
      uint32_t par = 0;
      for (int j = S; j < units; ++j) {
        if (!mbar_wait_bounded(empty(st), par, a.err)) break;
        mbar_expect_tx(full(st), UB);
        bulk_g2s(ring + st * UB, wsrc + (size_t)j * UB, UB, full(st));
        if (++st == S) { st = 0; par ^= 1; }
      }
    }
  } else if (warp == 1) {
    // the whole warp runs the issue loop (warp-uniform counters and descriptors);
    // one elected lane issues each MMA and commit.  Counters, not divisions.
    int st = 0, uo = 0, pc = 0, pb = 0;
    uint32_t fpar = 0, ppar = 0;
    for (int c = 0; c < nchunks; ++c) {
      if (pc == 0 && !mbar_wait_warp(bfull0 + 8 * pb, ppar, a.err)) break;
      if (uo == 0 && !mbar_wait_warp(full(st), fpar, a.err)) break;
      tc_fence_after();
      const uint64_t ad = umma_desc_sw128(ring + st * UB + uo * kStageBytes);
      const uint64_t bd = umma_desc_sw128(s.bbuf0 + pb * s.bbuf_stride + pc * BCH);
#pragma unroll
      for (int kk = 0; kk < kChunk / 16; ++kk) umma_ss_elect(tmem, ad + 2 * kk, bd + 2 * kk, IDESC, (c | kk) ? 1u : 0u);
      if (uo == U - 1) umma_commit_elect(empty(st));
      if (pc == cpp - 1 || c == nchunks - 1) umma_commit_elect(bempty0 + 8 * pb);
      if (++uo == U) { uo = 0; if (++st == S) { st = 0; fpar ^= 1; } }
      if (++pc == cpp) { pc = 0; pb ^= 1; if (pb == 0) ppar ^= 1; }
    }
    umma_commit_elect(accfull);
  } else {
    // workers: stage the activation pieces, then read the accumulator
    for (int p = 0; p < npieces; ++p) {
      const int pb = p & 1;
      if (p >= 2) mbar_wait_bounded(bempty0 + 8 * pb, ((p - 2) >> 1) & 1, a.err);
      const int kp = min(a.Kp, a.Kc - p * a.Kp);
      StageRegs<MT> g;
      stage_load<MT>(a, T, m0, k_begin + p * a.Kp, kp, g);
      if (p == 0) {
        // the row statistics while the first piece's loads are in flight
        load_row_stats(a, T, s.stat_mu, s.stat_rs, wtid());
        named_sync(1, kWorkers);
      }
      stage_store<MT>(a, s.stat_mu, s.stat_rs, s.bbuf0 + pb * s.bbuf_stride, T, k_begin + p * a.Kp, kp, g);
      fence_proxy_async();
      named_sync(1, kWorkers);
      if (wtid() == 0) mbar_arrive(bfull0 + 8 * pb);
    }
    mbar_wait_bounded(accfull, 0, a.err);
    tc_fence_after();
  }
  if (warp >= 2 && warp < 6) {
    // TMEM lane = weight row; columns: hi rows then lo rows of the activations
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16);
    if (MT == 1) {
      float v[32];
      tmem_ld32(taddr, v);   // columns 0..15 hi, 16..31 lo
#pragma unroll
      for (int t = 0; t < 16; ++t) s.cs_ptr[t * kCsStride + row] = v[t] + v[16 + t];
    } else {
      float hi[32], lo[32];
      tmem_ld32(taddr, hi);        // columns 0..31 hi
      tmem_ld32(taddr + 32, lo);   // columns 32..63 lo
#pragma unroll
      for (int t = 0; t < 32; ++t) s.cs_ptr[t * kCsStride + row] = hi[t] + lo[t];
    }
    tc_fence_before();
  }
  __syncthreads();

  cg::cluster_group cluster = cg::this_cluster();
  const int ks = a.ksplit;
  const int rank = ks > 1 ? (int)cluster.block_rank() : 0;
  // the partial tiles are published; the first unit's epilogue operands load meanwhile
  if (ks > 1) cluster_arrive_release();
  const int ew = warp - 2;
  const int t0 = rank + ks * ew;             // this warp's first (token, tile) unit
  constexpr int kMaxUnits = kMaxT / (kWorkers / 32);
  EpiIn pre;
  if (warp >= 2 && t0 < T) epilogue_load(a, t0, m0, pre);
  if (ks > 1) cluster_wait_acquire();

  // sum the partial tiles of this warp's units in rank order (deterministic)
  float vs[kMaxUnits][4];
  int nu = 0;
  if (warp >= 2) {
    for (int t = t0; t < T; t += ks * (kWorkers / 32), ++nu) {
      float4 part[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {  // all partial rows requested before any is summed (ks <= 8)
        part[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < ks) {
          const float *src = ks > 1 ? cluster.map_shared_rank(s.cs_ptr, r) : s.cs_ptr;
          part[r] = *reinterpret_cast<const float4 *>(src + t * kCsStride + 4 * lane);
        }
      }
      float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        v[0] += part[r].x; v[1] += part[r].y; v[2] += part[r].z; v[3] += part[r].w;
      }
#pragma unroll
      for (int u = 0; u < kMaxUnits; ++u)
        if (u == nu) { vs[u][0] = v[0]; vs[u][1] = v[1]; vs[u][2] = v[2]; vs[u][3] = v[3]; }
    }
  }
  // done reading the peers' tiles (the values are summed): they may leave once everyone has arrived
  if (ks > 1) cluster_arrive_relaxed();
  if (warp >= 2) {
    // the next unit's operands load while this unit's epilogue runs
    EpiIn cur = pre;
#pragma unroll
    for (int u = 0; u < kMaxUnits; ++u) {
      if (u >= nu) break;
      const int t = t0 + u * ks * (kWorkers / 32);
      EpiIn nxt;
      if (u + 1 < nu) epilogue_load(a, t + ks * (kWorkers / 32), m0, nxt);
      float v[4] = {vs[u][0], vs[u][1], vs[u][2], vs[u][3]};
      epilogue_unit(a, t, m0, v, tile, cur);
      cur = nxt;
    }
  }

  // self-attention tail: the last CTA to finish a head's q, k and v computes it
  if (a.self_D > 0) {
    __shared__ int s_last[4];
    const int D = a.self_D;
    const int mseg = m0 % D;
    const int heads_in_tile = kTile / a.hd;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int i = 0; i < heads_in_tile; ++i) {
        const int h = mseg / a.hd + i;
        const int old = atomicAdd(a.tickets + h, 1);
        const bool last = old == 3 * ks - 1;
        if (last) atomicExch(a.tickets + h, 0);
        s_last[i] = last ? h : -1;
      }
    }
    __syncthreads();
    for (int i = 0; i < heads_in_tile; ++i) {
      if (s_last[i] >= 0) {
        __threadfence();
        self_attention_head(a, s_last[i], T, reinterpret_cast<float *>(gbase));
      }
    }
  }
  // no CTA leaves (or reuses its tile buffer) before every peer has read it
  if (ks > 1) cluster_wait_acquire();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_free<NR>(tmem);
  }
}

// ring chunks (16 KB each), and chunks per bulk copy
static int gemv_stages(const GemvArgs &a, int mt) {
  const int nchunks = a.Kc / kChunk;
  const int most = mt == 1 ? 4 : 3;   // 17..32 rows: a shorter ring keeps two CTAs per SM
  return nchunks < most ? nchunks : most;
}
static int gemv_unit(const GemvArgs &a, int mt) {
  return (a.Kc / kChunk) % 2 == 0 && gemv_stages(a, mt) % 2 == 0 ? 2 : 1;
}

size_t gemv_smem_bytes(const GemvArgs &a, int mt) {
  const int S = gemv_stages(a, mt);
  const int cpp = a.Kp / kChunk;
  size_t bytes = 1024 + (size_t)S * kStageBytes + 2 * (size_t)cpp * (32 * mt * 128) +
                 (size_t)(16 * mt) * kCsStride * 4 + 2 * kMaxT * 4 + 16 * S + 64;
  const size_t attn = 1024 + (size_t)3 * kMaxT * (a.hd + 4) * 4;
  return bytes > attn ? bytes : attn;
}

cudaError_t launch_gemv(const GemvArgs &a, int n_tiles, cudaStream_t st, bool pdl) {
  const int mt = (a.T_const > 0 && a.T_const <= 16) ? 1 : 2;
  if (a.Kp > (mt == 1 ? 256 : 128) || a.Kp % kChunk != 0) return cudaErrorInvalidValue;   // the staging registers hold one piece
  const size_t smem = gemv_smem_bytes(a, mt);
  const int U = gemv_unit(a, mt);
  const int S = gemv_stages(a, mt) / U;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_tiles, a.ksplit, 1);
  cfg.blockDim = dim3(kAll, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (a.ksplit > 1) {   // (without K slices each CTA is its own cluster, and two may share an SM)
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = a.ksplit;
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
  cudaError_t e;
  if (mt == 1) {
    e = cudaFuncSetAttribute(fm_linear_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, fm_linear_kernel<1>, a, S, U);
  }
  e = cudaFuncSetAttribute(fm_linear_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, fm_linear_kernel<2>, a, S, U);
}

}  // namespace fm
