// k_step.cu -- the whole 16-slot draft block in one persistent launch.
//
// The pages run the draft as a list of dispatches, one GEMM / attention / norm
// kernel after another, each reading its weights once (flashmap_drafter.js,
// ``draft``).  With a launch per product every SM idles while each small
// product's chain of row statistics -> staging -> MMA -> reduction ->
// epilogue runs, and on this GPU a dependent round trip through L2 costs well
// over a microsecond, so latency, not HBM, bounded the step.  Here clusters of
// 8 CTAs (one CTA per SM) run the whole program of phases -- per layer the
// q/k/v, o (with the block self-attention as its prologue), cross-q (with the
// cross-attention as its tail), cross-o, fc1 and fc2 products -- and the head:
//   * warp 0 streams the CTA's share of every phase's weights, in program
//     order, with 32 KB bulk copies into a shared-memory ring; weights do not
//     depend on activations, so the stream runs ahead across phase boundaries;
//   * warp 1 issues tcgen05.mma (M = 128 weight rows, N = 16 hi + 16 lo
//     activation rows, K = 16) into one TMEM accumulator per owned tile;
//   * the 128-row tiles of a phase are dealt to clusters; every rank of a
//     cluster owns the same K slice of each of its cluster's tiles, so warps
//     2..9 stage that slice of the activations (RMSNorm / adaLN
//     LayerNorm-modulate prologues, bf16 hi + lo split) once per phase;
//   * the partial tiles meet through distributed shared memory: a worker-only
//     cluster barrier (remote mbarrier arrivals, release / acquire at cluster
//     scope) publishes them, and rank r adds rows r and r + 8 of every tile in
//     rank order (deterministic) and runs the fused epilogue (bias, GELU, gated
//     residual + row moments, per-head RMSNorm + RoPE, the lm_head operand);
//   * the block self-attention of a head is the prologue of the o product:
//     each rank attends the heads its K slice covers;
//   * the cross-attention is the tail of the cross-q product: each cluster
//     owns its heads' q tiles, splits the keys over its 8 CTAs (f16 mma.sync
//     on swizzled cp.async stages, online softmax, warps merged in shared
//     memory) and merges the ranks through distributed shared memory;
//   * phases are separated by a grid-wide barrier (an arrival counter and a
//     generation word); every wait is bounded: one that exceeds its budget
//     raises the error word and the kernel winds down (its copies in flight
//     land and its MMAs complete before it frees TMEM and exits).
#include <cooperative_groups.h>

#include "linear_parts.cuh"

namespace fm {

namespace {

namespace cg = cooperative_groups;

constexpr int kRing = 4;                          // ring stages
constexpr int kUnit = 2 * kStageBytes;            // 32 KB: two 16 KB chunks per bulk copy
constexpr int kPieceCols = 256;                   // activation columns per staged B piece
constexpr int kCpp = kPieceCols / kChunk;         // chunks per piece
constexpr int kBch = 32 * 128;                    // bytes of one 64-column B chunk (32 rows)
constexpr int kPieceBytes = kCpp * kBch;          // 16 KB
constexpr int kRows = 16;                         // block rows a phase carries
constexpr int kPartTile = kRows * kTile * 4;      // one partial tile, f32 [16][128]
constexpr int kNAcc = kStepMaxTiles;              // one TMEM accumulator (32 columns) per owned tile
constexpr int kTmemCols = 256;
constexpr uint32_t kIdesc = umma_idesc(128, 32, true);
constexpr int kKeys = 64;                         // keys per attention stage

// shared-memory layout (offsets from the 1024-aligned base)
constexpr int kOffRing = 0;
constexpr int kOffB = kOffRing + kRing * kUnit;                  // 2 B pieces (or a key stage)
constexpr int kOffPart = kOffB + 2 * kPieceBytes;                // partial tiles / q, k, v / key stage
constexpr int kPartArea = 52 * 1024;
constexpr int kOffQ = kOffPart + kPartArea;                      // f16 hi / lo query tiles [16][hd]
constexpr int kOffMisc = kOffQ + 8 * 1024;
constexpr int kOffStats = kOffMisc;                              // mu, rs [kMaxT]
constexpr int kOffFlags = kOffStats + 2 * kMaxT * 4;
constexpr int kOffBars = kOffFlags + 64;
constexpr int kNBars = 2 * kRing + 2 + 2 + kNAcc + 1 + 2;
constexpr int kOffTslot = kOffBars + 8 * kNBars;
constexpr int kSmemUsed = kOffTslot + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;
static_assert(kSmemBytes <= 232448, "shared memory beyond the per-CTA limit");
static_assert(kStepMaxTiles * kPartTile <= kPartArea, "partial tiles beyond their area");

struct Bars {
  uint32_t base;
  __device__ uint32_t full(int i) const { return base + 8 * i; }
  __device__ uint32_t empty(int i) const { return base + 8 * (kRing + i); }
  __device__ uint32_t bfull(int i) const { return base + 8 * (2 * kRing + i); }
  __device__ uint32_t bempty(int i) const { return base + 8 * (2 * kRing + 2 + i); }
  __device__ uint32_t accfull(int i) const { return base + 8 * (2 * kRing + 4 + i); }
  __device__ uint32_t drain() const { return base + 8 * (2 * kRing + 4 + kNAcc); }
  // two cluster barriers used alternately: a rank arrives on a barrier again only
  // after every rank has finished its arrivals of the sync before (it passed the
  // sync in between), so no arrival can land in a phase that is still open
  __device__ uint32_t cluster(int i) const { return base + 8 * (2 * kRing + 5 + kNAcc + i); }
};

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
  return t;
}
__device__ __forceinline__ void stamp(const StepArgs &a, int p, int slot) {
  if (a.trace) a.trace[((size_t)p * gridDim.x + blockIdx.x) * kStepTraceSlots + slot] = gtimer();
}

// ---- grid barrier ------------------------------------------------------------
// A monotonic 64-bit arrival counter: after each phase every CTA adds one with
// release semantics (no returned value, no separate fence); the phase is
// complete everywhere when the counter has grown by G past the phase's base.
// Every launch adds exactly n_phases * G, so at a launch's start the counter,
// rounded down to a multiple of G, is the launch's base (no CTA of this
// launch can have completed a phase before this CTA arrives).
__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];\n" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void grid_arrive(unsigned long long *ctr) {
  asm volatile("red.release.gpu.global.add.u64 [%0], 1;\n" ::"l"(ctr) : "memory");
}
// Wait until the counter reaches target; bounded.
__device__ __forceinline__ bool grid_wait(const unsigned long long *ctr, unsigned long long target, int32_t *err) {
  if (ld_acquire64(ctr) >= target) return true;
  const long long t0 = clock64();
  long long next = t0 + 4096;
  while (ld_acquire64(ctr) < target) {
    const long long t = clock64();
    if (t > next) {
      if (*reinterpret_cast<volatile int32_t *>(err)) return false;
      if (t - t0 > kWaitBudgetCycles) {
        atomicExch(err, 1);
        return false;
      }
      next = t + 4096;
    }
  }
  return true;
}

// the L2 prefetch of a byte range (no shared memory, no completion to wait for)
__device__ __forceinline__ void l2_prefetch(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}

// ---- cluster barrier among the worker warps ---------------------------------------
// The producer and MMA warps run ahead on their own, so the hardware cluster
// barrier (which counts every thread) cannot be used inside the phase loop.
// Instead one worker thread per CTA arrives, with release semantics at cluster
// scope, on an mbarrier of every CTA of the cluster (the CTA's named barrier
// before it orders all its workers' writes), and waits for its own barrier's 8
// arrivals with acquire semantics.
__device__ __forceinline__ bool cl_sync(const Bars &bars, uint32_t &n, int tid, int32_t *err, volatile int *flag) {
  const uint32_t bar = bars.cluster(n & 1), parity = (n >> 1) & 1;
  ++n;
  named_sync(1, kWorkers);
  if (tid < kStepCS) {
    // eight lanes of one warp arrive on the eight ranks' barriers at once; a release
    // after the named barrier covers every worker's earlier writes
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(remote) : "r"(bar), "r"(tid));
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n" ::"r"(remote) : "memory");
  }
  if (tid == 0) {
    bool ok = true;
    const long long t0 = clock64();
    long long next = t0 + 4096;
    for (;;) {
      uint32_t done;
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
          " selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(done)
          : "r"(bar), "r"(parity)
          : "memory");
      if (done) break;
      const long long t = clock64();
      if (t > next) {
        if (t - t0 > kWaitBudgetCycles || *reinterpret_cast<volatile int32_t *>(err)) {
          atomicExch(err, 1);
          ok = false;
          break;
        }
        next = t + 4096;
      }
    }
    *flag = ok ? 1 : 0;
  }
  named_sync(1, kWorkers);
  return *flag != 0;
}

// ---- a phase's work of this CTA -------------------------------------------------------
// The tiles of cluster c in a phase (tile i -> cluster (i + rot) % n_clusters):
// c0, c0 + ncl, c0 + 2 ncl, ... (computed, not stored: local arrays cost an L2
// round trip here, where shared memory leaves little L1).
struct Own {
  int c0, n;    // first tile and number of tiles of this cluster
  int ncl;
  int kc0, kc1; // this rank's chunk range in every tile
  __device__ __forceinline__ int tile(int ti) const { return c0 + ti * ncl; }
};
__device__ __forceinline__ void phase_own(const StepPhase &P, int c, int r, int ncl, Own &o) {
  o.ncl = ncl;
  o.c0 = ((c - P.rot) % ncl + ncl) % ncl;
  o.n = o.c0 < P.ntiles ? (P.ntiles - o.c0 + ncl - 1) / ncl : 0;
  if (o.n > kStepMaxTiles) o.n = kStepMaxTiles;   // the host checked the schedule
  o.kc0 = step_klo(r, P.cpt);
  o.kc1 = step_klo(r + 1, P.cpt);
}

// ---- attention helpers --------------------------------------------------------------
__device__ __forceinline__ void mma_f16_k8(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(b0));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// byte offset of 16-byte unit u of row r in a tile of (hd * 2)-byte rows, the
// units permuted by r % 8 so that eight rows reading one unit hit eight bank groups
__device__ __forceinline__ uint32_t kv_slot(int r, int u, int hd) {
  return (uint32_t)(r * hd * 2 + ((u ^ (r & 7)) << 4));
}
// request rows [rlo, rhi) of the 64-key stage starting at key k0 (rows at or past
// kend read as zero) into K / V tiles; 256 worker threads
__device__ __forceinline__ void kv_issue(const StepAttn &A, int head, int k0, int kend, uint32_t kb, uint32_t vb,
                                         int rlo, int rhi, int tid) {
  const int hd = A.hd;
  const int U = hd / 8;
  const __half *kh = A.Kc + (size_t)head * A.max_ctx * hd;
  const __half *vh = A.Vc + (size_t)head * A.max_ctx * hd;
  for (int i = tid + rlo * U; i < rhi * U; i += kWorkers) {
    const int rr = i / U, u = i - rr * U;
    const int key = k0 + rr;
    const bool ok = key < kend;
    const size_t off = (size_t)(ok ? key : 0) * hd + u * 8;
    cp_async16(kb + kv_slot(rr, u, hd), kh + off, ok ? 16u : 0u);
    cp_async16(vb + kv_slot(rr, u, hd), vh + off, ok ? 16u : 0u);
  }
}
// keys of rank r of a head: [kbeg, kend)
__device__ __forceinline__ void rank_keys(int L, int r, int &kbeg, int &kend) {
  int per = (L + kStepCS - 1) / kStepCS;
  per = (per + 15) & ~15;
  kbeg = min(L, r * per);
  kend = min(L, kbeg + per);
}

// The cross-attention tail of a cross-q phase for the cluster's heads (its own
// function: its registers are not held across the rest of the phase loop).
__device__ __noinline__ bool cross_tail(const StepArgs &a, const StepPhase &P, const Own &o, int r, int T, int tid,
                                        const Bars &bars, uint32_t &clpar, volatile int *flags, uint8_t *gbase,
                                        uint32_t base, int kbeg, int kend, int pre) {
  cg::cluster_group cluster = cg::this_cluster();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, w = warp - 2;
  float *partf = reinterpret_cast<float *>(gbase + kOffPart);
  const uint32_t bbuf = base + kOffB, part = base + kOffPart, qbuf = base + kOffQ;
  const uint32_t stageA = part + 16 * 1024, stageB = bbuf;
  const uint32_t tileb = (uint32_t)kKeys * P.at.hd * 2;
  (void)stageB;
  const StepAttn &A = P.at;
  const int hd = A.hd;
  // every rank's q rows are stored (global) and every rank is done reading the partials
  if (!cl_sync(bars, clpar, tid, a.err, flags + 2)) return false;
  const int heads_per_tile = kTile / hd;
  bool ok = true;
  for (int hi = 0; hi < o.n * heads_per_tile && ok; ++hi) {
    const int head = o.tile(hi / heads_per_tile) * heads_per_tile + hi % heads_per_tile;
    if (head >= A.n_heads) continue;
    if (hi > 0) {
      // the previous head's partial slot is read by the peers before it is reused
      if (!cl_sync(bars, clpar, tid, a.err, flags + 2)) { ok = false; break; }
      pre = 0;
      cp_async_commit();
    }
    const int nst = (kend - kbeg + kKeys - 1) / kKeys;
    // the rest of the first key stage, and the second (buffer B: the MMAs are done)
    if (nst > 0 && pre < kKeys) kv_issue(A, head, kbeg, kend, stageA, stageA + tileb, pre, kKeys, tid);
    cp_async_commit();
    if (nst > 1) kv_issue(A, head, kbeg + kKeys, kend, stageB, stageB + tileb, 0, kKeys, tid);
    cp_async_commit();
    // queries -> f16 hi / lo tiles [16][hd], units permuted by row
    const uint32_t qhi = qbuf, qlo = qbuf + kRows * hd * 2;
    const int q4 = hd / 4;
    {
      float4 xq[2];   // 16 rows x hd / 4 quads over 256 threads: two each, both in flight
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int i = tid + x * kWorkers;
        const int t = i / q4, d = 4 * (i - t * q4);
        xq[x] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < kRows * q4 && t < T)
          xq[x] = __ldcg(reinterpret_cast<const float4 *>(A.Q + (size_t)t * A.ldq + head * hd + d));
      }
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int i = tid + x * kWorkers;
        if (i >= kRows * q4) continue;
        const int t = i / q4, d = 4 * (i - t * q4);
        uint32_t h01, l01, h23, l23;
        split2_f16(xq[x].x, xq[x].y, h01, l01);
        split2_f16(xq[x].z, xq[x].w, h23, l23);
        const uint32_t off = kv_slot(t, d >> 3, hd) + (d & 7) * 2;
        asm volatile("st.shared.v2.u32 [%0], {%1,%2};\n" ::"r"(qhi + off), "r"(h01), "r"(h23));
        asm volatile("st.shared.v2.u32 [%0], {%1,%2};\n" ::"r"(qlo + off), "r"(l01), "r"(l23));
      }
    }
    // per warp: keys 8w .. 8w + 7 of each stage; thread rows g and g + 8
    const int gq = lane >> 2, qq = lane & 3;
    const int NT = hd / 8;
    float oacc[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
    const int mi = lane >> 3, ri = lane & 7;
    for (int st = 0; st < nst; ++st) {
      cp_async_wait<1>();
      named_sync(1, kWorkers);
      const uint32_t kbuf = (st & 1) ? stageB : stageA, vbuf = kbuf + tileb;
      const int key = 8 * w + ri;
      float s4[4] = {0.f, 0.f, 0.f, 0.f}, s4b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int ks = 0; ks < hd / 16; ks += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbuf + kv_slot(key, 2 * ks + mi, hd), b0, b1, b2, b3);
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int kq = ks + h2;
          const int arow = ri + 8 * (mi & 1), aunit = 2 * kq + (mi >> 1);
          uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
          ldsm_x4(qhi + kv_slot(arow, aunit, hd), a0, a1, a2, a3);
          ldsm_x4(qlo + kv_slot(arow, aunit, hd), c0, c1, c2, c3);
          const uint32_t bb0 = h2 ? b2 : b0, bb1 = h2 ? b3 : b1;
          mma_f16(s4, a0, a1, a2, a3, bb0, bb1);
          mma_f16(s4b, c0, c1, c2, c3, bb0, bb1);
        }
      }
      // scores in the log2 domain, masked past kend; rows g (s[0], s[1]) and g + 8 (s[2], s[3])
      const int kabs = kbeg + st * kKeys + 8 * w + 2 * qq;
      float s[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) s[e] = kabs + (e & 1) < kend ? (s4[e] + s4b[e]) * A.scale_log2 : -INFINITY;
      float alpha[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        float mx = fmaxf(s[2 * h2], s[2 * h2 + 1]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mn = fmaxf(m_r[h2], mx);
        alpha[h2] = mn == -INFINITY ? 1.f : exp2f(m_r[h2] - mn);
        m_r[h2] = mn;
      }
      float prb[4];
      float rsum[2] = {0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float mm = m_r[e >> 1];
        prb[e] = mm == -INFINITY ? 0.f : exp2f(s[e] - mm);
        rsum[e >> 1] += prb[e];
      }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        rsum[h2] += __shfl_xor_sync(0xffffffffu, rsum[h2], 1);
        rsum[h2] += __shfl_xor_sync(0xffffffffu, rsum[h2], 2);
        l_r[h2] = l_r[h2] * alpha[h2] + rsum[h2];
      }
      uint32_t ph0, pl0, ph1, pl1;
      split2_f16(prb[0], prb[1], ph0, pl0);
      split2_f16(prb[2], prb[3], ph1, pl1);
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        if (nt < NT) {
          oacc[nt][0] *= alpha[0]; oacc[nt][1] *= alpha[0];
          oacc[nt][2] *= alpha[1]; oacc[nt][3] *= alpha[1];
        }
      }
#pragma unroll
      for (int nt = 0; nt < 16; nt += 4) {
        if (nt < NT) {
          uint32_t v0, v1, v2, v3;
          ldsm_x4_t(vbuf + kv_slot(key, nt + mi, hd), v0, v1, v2, v3);
          mma_f16_k8(oacc[nt], ph0, ph1, v0);
          mma_f16_k8(oacc[nt], pl0, pl1, v0);
          mma_f16_k8(oacc[nt + 1], ph0, ph1, v1);
          mma_f16_k8(oacc[nt + 1], pl0, pl1, v1);
          mma_f16_k8(oacc[nt + 2], ph0, ph1, v2);
          mma_f16_k8(oacc[nt + 2], pl0, pl1, v2);
          mma_f16_k8(oacc[nt + 3], ph0, ph1, v3);
          mma_f16_k8(oacc[nt + 3], pl0, pl1, v3);
        }
      }
      named_sync(1, kWorkers);   // every warp is done with this stage's buffers
      if (st + 2 < nst)
        kv_issue(A, head, kbeg + (st + 2) * kKeys, kend, kbuf, vbuf, 0, kKeys, tid);
      cp_async_commit();
    }
    cp_async_wait<0>();
    named_sync(1, kWorkers);
    // merge the eight warps in three halving rounds (scratch: the B buffers, 32 KB,
    // then the (max, sum) pairs past the first key stage)
    float *mo = reinterpret_cast<float *>(gbase + kOffB);                 // [4][16][hd]
    float *mml = reinterpret_cast<float *>(gbase + kOffPart + 16 * 1024 + 2 * tileb);
    for (int half = 4; half >= 1; half >>= 1) {
      if (w >= half && w < 2 * half) {
        const int ww = w - half;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
          if (nt < NT) {
            const int d = 8 * nt + 2 * qq;
            *reinterpret_cast<float2 *>(mo + (ww * 16 + gq) * hd + d) = make_float2(oacc[nt][0], oacc[nt][1]);
            *reinterpret_cast<float2 *>(mo + (ww * 16 + gq + 8) * hd + d) = make_float2(oacc[nt][2], oacc[nt][3]);
          }
        }
        if (qq == 0) {
          mml[(ww * 16 + gq) * 2] = m_r[0];
          mml[(ww * 16 + gq) * 2 + 1] = l_r[0];
          mml[(ww * 16 + gq + 8) * 2] = m_r[1];
          mml[(ww * 16 + gq + 8) * 2 + 1] = l_r[1];
        }
      }
      named_sync(1, kWorkers);
      if (w < half) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int row = gq + 8 * h2;
          const float m2 = mml[(w * 16 + row) * 2], l2 = mml[(w * 16 + row) * 2 + 1];
          const float M = fmaxf(m_r[h2], m2);
          const float f1 = m_r[h2] == -INFINITY ? 0.f : exp2f(m_r[h2] - M);
          const float f2 = m2 == -INFINITY ? 0.f : exp2f(m2 - M);
          l_r[h2] = l_r[h2] * f1 + l2 * f2;
          m_r[h2] = M;
#pragma unroll
          for (int nt = 0; nt < 16; ++nt) {
            if (nt < NT) {
              const float2 xo = *reinterpret_cast<const float2 *>(mo + (w * 16 + row) * hd + 8 * nt + 2 * qq);
              oacc[nt][2 * h2] = oacc[nt][2 * h2] * f1 + xo.x * f2;
              oacc[nt][2 * h2 + 1] = oacc[nt][2 * h2 + 1] * f1 + xo.y * f2;
            }
          }
        }
      }
      named_sync(1, kWorkers);
    }
    // this rank's partial (unnormalised rows, max, sum) into its partial slot
    float *po = partf;                   // [16][hd], then [16][2]
    float *pml = partf + kRows * hd;
    if (w == 0) {
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        if (nt < NT) {
          const int d = 8 * nt + 2 * qq;
          *reinterpret_cast<float2 *>(po + gq * hd + d) = make_float2(oacc[nt][0], oacc[nt][1]);
          *reinterpret_cast<float2 *>(po + (gq + 8) * hd + d) = make_float2(oacc[nt][2], oacc[nt][3]);
        }
      }
      if (qq == 0) {
        pml[2 * gq] = m_r[0];
        pml[2 * gq + 1] = l_r[0];
        pml[2 * (gq + 8)] = m_r[1];
        pml[2 * (gq + 8) + 1] = l_r[1];
      }
    }
    if (!cl_sync(bars, clpar, tid, a.err, flags + 2)) { ok = false; break; }
    // rank r merges rows r and r + 8 over the cluster's ranks, in rank order
    if (w < 2) {
      const int t = r + kStepCS * w;
      if (t < T) {
        float mq[kStepCS], lq[kStepCS];
        float M = -INFINITY;
#pragma unroll
        for (int q = 0; q < kStepCS; ++q) {
          const float *rm = cluster.map_shared_rank(pml, q);
          mq[q] = rm[2 * t];
          lq[q] = rm[2 * t + 1];
          M = fmaxf(M, mq[q]);
        }
        float den = 0.f;
        float f[kStepCS];
#pragma unroll
        for (int q = 0; q < kStepCS; ++q) {
          f[q] = mq[q] == -INFINITY ? 0.f : exp2f(mq[q] - M);
          den += f[q] * lq[q];
        }
        const float inv = 1.f / den;
        for (int d = 4 * lane; d < hd; d += 128) {
          float4 accv = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int q = 0; q < kStepCS; ++q) {
            const float4 xo = *reinterpret_cast<const float4 *>(cluster.map_shared_rank(po, q) + t * hd + d);
            accv.x += f[q] * xo.x; accv.y += f[q] * xo.y; accv.z += f[q] * xo.z; accv.w += f[q] * xo.w;
          }
          *reinterpret_cast<float4 *>(A.out + (size_t)t * A.ldo + head * hd + d) =
              make_float4(accv.x * inv, accv.y * inv, accv.z * inv, accv.w * inv);
        }
      }
    }
  }
  return ok;
}

}  // namespace

__global__ void __launch_bounds__(kAll, 1) fm_draft_step_kernel(const __grid_constant__ StepArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - smem_u32(smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const int c = blockIdx.x / kStepCS;
  cg::cluster_group cluster = cg::this_cluster();
  const int r = (int)cluster.block_rank();
  const int ncl = a.n_clusters;
  const int T = a.T;
  const uint32_t ring = base + kOffRing, bbuf = base + kOffB, part = base + kOffPart, qbuf = base + kOffQ;
  float *partf = reinterpret_cast<float *>(gbase + kOffPart);
  float *stats = reinterpret_cast<float *>(gbase + kOffStats);
  volatile int *flags = reinterpret_cast<volatile int *>(gbase + kOffFlags);
  const Bars bars{base + kOffBars};
  const uint32_t tslot = base + kOffTslot;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNBars - 2; ++i) mbar_init(bars.base + 8 * i, 1);
    mbar_init(bars.cluster(0), kStepCS);
    mbar_init(bars.cluster(1), kStepCS);
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc<kTmemCols>(tslot);
  tc_fence_before();
  // every CTA's barriers are initialised before any peer arrives on them
  cluster.sync();
  tc_fence_after();
  const uint32_t tmem = lds32(tslot);

  if (warp == 0) {
    // ---------------------------------------------------------------- weight stream
    if (lane == 0) {
      int u = 0;
      bool ok = true;
      for (int p = 0; p < a.n_phases && ok; ++p) {
        const StepPhase &P = a.ph[p];
        Own o;
        phase_own(P, c, r, ncl, o);
        // this CTA's weight slices (and cross-attention key rows) two phases ahead into L2:
        // HBM idles while a phase waits on its chain, so the next big phases stream from L2
        for (int pp = (p == 0 ? 0 : p + 2); pp <= p + 2 && pp < a.n_phases; ++pp) {
          const StepPhase &Q = a.ph[pp];
          Own oq;
          phase_own(Q, c, r, ncl, oq);
          if (oq.kc1 > oq.kc0)
            for (int ti = 0; ti < oq.n; ++ti)
              l2_prefetch(Q.g.Wt + ((size_t)oq.tile(ti) * Q.cpt + oq.kc0) * kStageBytes,
                          (uint32_t)(oq.kc1 - oq.kc0) * kStageBytes);
          if (Q.tail == ST_CROSS_ATTN && oq.n > 0) {
            const StepAttn &A = Q.at;
            const int L = (A.L_src == 0 ? a.sp->L : a.sp->pos + 1) + A.L_add;
            int kb0, ke0;
            rank_keys(L, r, kb0, ke0);
            const int top = min(ke0, a.sp->stable);   // rows later phases do not write
            if (top > kb0)
              for (int hi = 0; hi < oq.n * (kTile / A.hd); ++hi) {
                const int head = oq.tile(hi / (kTile / A.hd)) * (kTile / A.hd) + hi % (kTile / A.hd);
                if (head >= A.n_heads) continue;
                const size_t off = ((size_t)head * A.max_ctx + kb0) * A.hd;
                l2_prefetch(A.Kc + off, (uint32_t)(top - kb0) * A.hd * 2);
                l2_prefetch(A.Vc + off, (uint32_t)(top - kb0) * A.hd * 2);
              }
          }
        }
        for (int ti = 0; ti < o.n && ok; ++ti) {
          const uint8_t *src = P.g.Wt + ((size_t)o.tile(ti) * P.cpt + o.kc0) * kStageBytes;
          for (int kc = o.kc0; kc < o.kc1; kc += 2) {
            const int st = u % kRing, rd = u / kRing;
            if (rd >= 1 && !mbar_wait_bounded(bars.empty(st), (rd - 1) & 1, a.err)) { ok = false; break; }
            const int nch = min(2, o.kc1 - kc);
            mbar_expect_tx(bars.full(st), nch * kStageBytes);
            bulk_g2s(ring + st * kUnit, src + (size_t)(kc - o.kc0) * kStageBytes, nch * kStageBytes, bars.full(st));
            ++u;
          }
        }
        stamp(a, p, 3);
      }
      // wind down: every copy this CTA issued (the last kRing units) has landed before the CTA may exit
      for (int v = u > kRing ? u - kRing : 0; v < u; ++v) mbar_wait_drain(bars.full(v % kRing), (v / kRing) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issue
    int u = 0, pc = 0;   // units consumed, B pieces consumed (counter shared with the workers)
    bool ok = true;
    for (int p = 0; p < a.n_phases && ok; ++p) {
      const StepPhase &P = a.ph[p];
      Own o;
      phase_own(P, c, r, ncl, o);
      const int nch = o.kc1 - o.kc0;
      if (o.n == 0 || nch == 0) continue;
      const int npc = (nch + kCpp - 1) / kCpp;
      const bool resident = npc <= 2;
      const int pc0 = pc;
      for (int ti = 0; ti < o.n && ok; ++ti) {
        const uint32_t d = tmem + ti * 32;
        for (int j = 0; j < nch && ok; j += 2) {
          const int st = u % kRing, rd = u / kRing;
          if (!mbar_wait_warp(bars.full(st), rd & 1, a.err)) { ok = false; break; }
          tc_fence_after();
          const int nu = min(2, nch - j);
          for (int x = 0; x < nu; ++x) {
            const int jj = j + x;
            const int q = resident ? pc0 + jj / kCpp : pc0 + ti * npc + jj / kCpp;
            const int pb = q & 1;
            if (jj % kCpp == 0 && (!resident || ti == 0)) {
              if (!mbar_wait_warp(bars.bfull(pb), (q >> 1) & 1, a.err)) { ok = false; break; }
              tc_fence_after();
            }
            const uint64_t ad = umma_desc_sw128(ring + st * kUnit + x * kStageBytes);
            const uint64_t bd = umma_desc_sw128(bbuf + pb * kPieceBytes + (jj % kCpp) * kBch);
#pragma unroll
            for (int kk = 0; kk < kChunk / 16; ++kk)
              umma_ss_elect(d, ad + 2 * kk, bd + 2 * kk, kIdesc, (jj | kk) ? 1u : 0u);
            if ((jj % kCpp == kCpp - 1 || jj == nch - 1) && (!resident || ti == o.n - 1))
              umma_commit_elect(bars.bempty(pb));
          }
          if (!ok) break;
          umma_commit_elect(bars.empty(st));
          ++u;
        }
        if (ok) umma_commit_elect(bars.accfull(ti));
      }
      pc = pc0 + (resident ? npc : npc * o.n);
      if (lane == 0) stamp(a, p, 4);
    }
    // wind down: every MMA issued has completed before TMEM is freed
    umma_commit_elect(bars.drain());
    mbar_wait_drain(bars.drain(), 0);
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- workers
    const int tid = wtid();
    const int w = warp - 2;
    pdl_wait();
    unsigned long long *ctr = reinterpret_cast<unsigned long long *>(a.bar);
    const unsigned long long base0 = ld_acquire64(ctr) / (unsigned long long)G * (unsigned long long)G;
    uint32_t clpar = 0;
    int pc = 0;
    uint32_t acc_par = 0;   // bit ti: parity of accumulator ti's next completion
    for (int p = 0; p < a.n_phases; ++p) {
      const StepPhase &P = a.ph[p];
      const GemvArgs &g = P.g;
      Own o;
      phase_own(P, c, r, ncl, o);
      const int nch = o.kc1 - o.kc0;
      // cross-attention tail: this rank's first key stage of its cluster's first
      // head (rows below `stable` are not written by this call) is requested early
      int kbeg = 0, kend = 0, pre = 0;
      const uint32_t stageA = part + 16 * 1024, stageB = bbuf;
      const uint32_t tileb = (uint32_t)kKeys * P.at.hd * 2;
      if (P.tail == ST_CROSS_ATTN && o.n > 0) {
        const int L = (P.at.L_src == 0 ? a.sp->L : a.sp->pos + 1) + P.at.L_add;
        rank_keys(L, r, kbeg, kend);
        const int stable = a.sp->stable;
        pre = kend > kbeg ? max(0, min(kKeys, stable - kbeg)) : 0;
        const int head0 = o.tile(0) * kTile / P.at.hd;
        if (pre > 0) kv_issue(P.at, head0, kbeg, kend, stageA, stageA + tileb, 0, pre, tid);
        cp_async_commit();
      }
      if (p > 0) {
        if (tid == 0) flags[1] = grid_wait(ctr, base0 + (unsigned long long)p * G, a.err) ? 1 : 0;
        named_sync(1, kWorkers);
        if (!flags[1]) break;
      }
      if (tid == 0) stamp(a, p, 0);
      if (o.n > 0 && nch > 0) {
        const int npc = (nch + kCpp - 1) / kCpp;
        const bool resident = npc <= 2;
        const int kb = o.kc0 * kChunk, ncol = nch * kChunk;
        float *mu = stats, *rs = stats + kMaxT;
        // -------------------------------------------- prologue: the block self-attention of this rank's heads
        const float *osm = nullptr;     // activations from shared memory (f32 [16][ncol]) instead of global
        if (P.prologue == SP_SELF_ATTN) {
          const StepAttn &A = P.at;
          const int hd = A.hd, D = A.D;
          const int h0 = kb / hd, h1 = (kb + ncol - 1) / hd;
          const int nh = h1 - h0 + 1;
          // q, k, v rows of the heads into the partial area: [head][q|k|v][16][hd + 4]
          const int ks = hd + 4;
          float *qkv = partf;
          const int q4 = hd / 4;
          // every load in flight before any is stored (one round trip, not one per element)
          const int total = nh * 3 * kRows * q4;
          for (int i0 = tid; i0 < total; i0 += kWorkers * 6) {
            float4 v[6];
#pragma unroll
            for (int x = 0; x < 6; ++x) {
              const int i = i0 + x * kWorkers;
              v[x] = make_float4(0.f, 0.f, 0.f, 0.f);
              if (i < total) {
                const int d4 = i % q4, rest = i / q4;
                const int t = rest % kRows, m = (rest / kRows) % 3, hh = rest / (3 * kRows);
                if (t < T)
                  v[x] = __ldcg(
                      reinterpret_cast<const float4 *>(A.qkv + (size_t)t * 3 * D + m * D + (h0 + hh) * hd + 4 * d4));
              }
            }
#pragma unroll
            for (int x = 0; x < 6; ++x) {
              const int i = i0 + x * kWorkers;
              if (i < total) {
                const int d4 = i % q4, rest = i / q4;
                const int t = rest % kRows, m = (rest / kRows) % 3, hh = rest / (3 * kRows);
                *reinterpret_cast<float4 *>(qkv + ((hh * 3 + m) * kRows + t) * ks + 4 * d4) = v[x];
              }
            }
          }
          named_sync(1, kWorkers);
          if (tid == 0) stamp(a, p, 7);
          // one warp per (head, query row); lane j < T holds the score of key j
          float *ob = reinterpret_cast<float *>(gbase + kOffB + kPieceBytes);   // f32 [16][ncol]
          for (int u = w; u < nh * T; u += 8) {
            const int hh = u / T, t = u - hh * T;
            const float *qr = qkv + ((hh * 3 + 0) * kRows + t) * ks;
            const float *kr = qkv + ((hh * 3 + 1) * kRows + (lane < T ? lane : 0)) * ks;
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
            for (int d = 0; d < hd; d += 4) {
              const float4 qv = *reinterpret_cast<const float4 *>(qr + d);
              const float4 kv = *reinterpret_cast<const float4 *>(kr + d);
              s0 += qv.x * kv.x; s1 += qv.y * kv.y; s2 += qv.z * kv.z; s3 += qv.w * kv.w;
            }
            const float sc = lane < T ? ((s0 + s1) + (s2 + s3)) * A.scale : -INFINITY;
            const float mx = warp_max(sc);
            const float pr = lane < T ? __expf(sc - mx) : 0.f;
            const float inv = 1.f / warp_sum(pr);
            // output: lane l owns dims 4l .. 4l + 3 of the head
            const float *vb = qkv + ((hh * 3 + 2) * kRows) * ks;
            const bool on = 4 * lane < hd;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j = 0; j < T; ++j) {
              const float pj = __shfl_sync(0xffffffffu, pr, j);
              if (on) {
                const float4 v = *reinterpret_cast<const float4 *>(vb + j * ks + 4 * lane);
                acc.x += pj * v.x; acc.y += pj * v.y; acc.z += pj * v.z; acc.w += pj * v.w;
              }
            }
            const int col = (h0 + hh) * hd + 4 * lane - kb;
            if (on && col >= 0 && col < ncol)
              *reinterpret_cast<float4 *>(ob + t * ncol + col) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
          }
          named_sync(1, kWorkers);
          osm = ob;
        }
        // -------------------------------------------- stage this rank's K slice of the activations
        const int passes = resident ? 1 : o.n;
        bool stats_done = false;
        for (int ps = 0; ps < passes; ++ps) {
          const int m0 = o.tile(resident ? 0 : ps) * kTile;
          for (int x = 0; x < ncol; x += kPieceCols) {
            const int pb = pc & 1;
            // (a wait that gives up raises the error word; the workers still take every
            // named barrier together, so a failure winds the CTA down instead of hanging it)
            if (pc >= 2) mbar_wait_bounded(bars.bempty(pb), ((pc >> 1) - 1) & 1, a.err);
            const int kp = min(kPieceCols, ncol - x);
            StageRegs<1> rg;
            if (osm) {
              using R = StageRegs<1>;
              const int t = tid / R::tpr, q0 = tid % R::tpr;
              const int nq = (kp >> 2) / R::tpr;
#pragma unroll
              for (int j = 0; j < R::kMaxQ; ++j) {
                rg.xv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                rg.p0[j] = rg.p1[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (j < nq && t < T)
                  rg.xv[j] = *reinterpret_cast<const float4 *>(osm + t * ncol + x + 4 * (q0 + R::tpr * j));
              }
            } else {
              stage_load<1>(g, T, m0, kb + x, kp, rg);
            }
            if (!stats_done) {
              // the row statistics while the first piece's loads are in flight
              load_row_stats(g, T, mu, rs, tid);
              named_sync(1, kWorkers);
              stats_done = true;
            }
            stage_store<1>(g, mu, rs, bbuf + pb * kPieceBytes, T, kb + x, kp, rg);
            fence_proxy_async();
            named_sync(1, kWorkers);
            if (tid == 0) mbar_arrive(bars.bfull(pb));
            ++pc;
          }
        }
        if (tid == 0) stamp(a, p, 1);
        // -------------------------------------------- accumulators -> partial tiles in shared memory
        for (int ti = w >> 2; ti < o.n; ti += 2) {
          mbar_wait_bounded(bars.accfull(ti), (acc_par >> ti) & 1, a.err);
          tc_fence_after();
          const int quad = warp & 3;
          float v[32];
          tmem_ld32(tmem + ti * 32 + ((uint32_t)(quad * 32) << 16), v);   // columns 0..15 hi, 16..31 lo
          tc_fence_before();
          float *pt = partf + ti * (kPartTile / 4);
          const int row = quad * 32 + lane;
#pragma unroll
          for (int t = 0; t < kRows; ++t) pt[t * kTile + row] = v[t] + v[16 + t];
        }
        acc_par ^= (1u << o.n) - 1u;
      } else if (o.n > 0) {
        // a rank without chunks in this phase (a short K) contributes zero tiles
        for (int i = tid; i < o.n * kPartTile / 16; i += kWorkers)
          reinterpret_cast<float4 *>(partf)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      // the epilogue operands of this rank's units (bias, residual, gate, norm
      // weights, rotations) load while the partials are published
      const int nrows = T > kStepCS ? 2 : 1;
      EpiIn epre;   // the first unit of this warp (most phases give a warp at most one)
      if (o.n > 0 && w < o.n * nrows) {
        const int ti = w / nrows, t = r + kStepCS * (w - ti * nrows);
        if (t < T) epilogue_load(g, t, o.tile(ti) * kTile, epre);
      }
      // -------------------------------------------------- publish the partials to the cluster
      if (!cl_sync(bars, clpar, tid, a.err, flags + 2)) break;
      if (tid == 0) stamp(a, p, 5);
      // -------------------------------------------------- rank r finishes rows r, r + 8 of every tile
      if (o.n > 0) {
        for (int uu = w; uu < o.n * nrows; uu += 8) {
          const int ti = uu / nrows, t = r + kStepCS * (uu - ti * nrows);
          if (t >= T) continue;
          const int tile = o.tile(ti);
          const int m0 = tile * kTile;
          EpiIn in;
          if (uu == w)
            in = epre;
          else
            epilogue_load(g, t, m0, in);
          float4 pv[kStepCS];
#pragma unroll
          for (int q = 0; q < kStepCS; ++q) {
            const float *src = cluster.map_shared_rank(partf, q) + ti * (kPartTile / 4) + t * kTile + 4 * lane;
            pv[q] = *reinterpret_cast<const float4 *>(src);
          }
          float vv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int q = 0; q < kStepCS; ++q) {   // rank order
            vv[0] += pv[q].x; vv[1] += pv[q].y; vv[2] += pv[q].z; vv[3] += pv[q].w;
          }
          epilogue_unit(g, t, m0, vv, tile, in);
        }
      }
      if (tid == 0) stamp(a, p, 6);
      // -------------------------------------------------- tail: cross-attention of the cluster's heads
      if (P.tail == ST_CROSS_ATTN && o.n > 0) {
        if (!cross_tail(a, P, o, r, T, tid, bars, clpar, flags, gbase, base, kbeg, kend, pre)) break;
      } else if (P.tail == ST_CROSS_ATTN) {
        cp_async_wait<0>();
      }
      // this phase is done here
      named_sync(1, kWorkers);
      if (tid == 0) {
        stamp(a, p, 2);
        grid_arrive(ctr);
      }
    }
    cp_async_wait<0>();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_free<kTmemCols>(tmem);
  }
  // no CTA leaves while a peer may still read its shared memory
  cluster.sync();
}

size_t step_smem_bytes() { return (size_t)kSmemBytes; }

// attrs: bit 0 = cooperative launch (every CTA is guaranteed co-resident), bit 1 =
// programmatic stream serialisation (the CTAs may start while the previous
// kernel drains; they call griddepcontrol.wait before reading its results)
cudaError_t launch_step(const StepArgs &a, int clusters, cudaStream_t st, int attrs) {
  cudaError_t e = cudaFuncSetAttribute(fm_draft_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(clusters * kStepCS, 1, 1);
  cfg.blockDim = dim3(kAll, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[3];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = kStepCS;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (attrs & 1) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  }
  if (attrs & 2) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, fm_draft_step_kernel, a);
}

int step_max_clusters() {
  if (cudaFuncSetAttribute(fm_draft_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kStepCS * 64, 1, 1);
  cfg.blockDim = dim3(kAll, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kStepCS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fm_draft_step_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace fm
