// k_step.cu -- the whole 16-slot draft block in one persistent launch.
//
// The pages run the draft as a list of dispatches, one GEMM / attention / norm
// kernel after another, each reading its weights once (flashmap_drafter.js,
// ``draft``).  A launch per product leaves every SM idle between products while
// the chain of row statistics -> staging -> MMA -> reduction -> epilogue of
// each small product runs; on sm_103a that latency, not HBM, bounded the step.
// Here one CTA per SM runs the whole program of phases (the q/k/v, o, cross-q,
// cross-attention, o, fc1, fc2 products of every layer and the head):
//   * warp 0 streams this CTA's share of every phase's weights, in program
//     order, with 32 KB bulk copies into a shared-memory ring; weights do not
//     depend on activations, so the stream runs ahead across phase boundaries,
//     limited only by the ring;
//   * warp 1 issues tcgen05.mma (M = 128 weight rows, N = 16 hi + 16 lo
//     activation rows, K = 16) into one of four TMEM accumulators per segment;
//   * warps 2..9 wait for the phase's grid barrier, stage the activations
//     (RMSNorm / adaLN LayerNorm-modulate prologues, bf16 hi + lo split) as the
//     MMA's B operand, read the accumulators, and publish partial tiles;
//   * a linear phase's chunks are dealt to CTAs in equal contiguous ranges
//     (stream-K), so every SM streams the same number of bytes; the last CTA to
//     finish a tile (a ticket) adds the tile's partials in CTA order
//     (deterministic) and runs the fused epilogue (bias, GELU, gated residual,
//     per-head RMSNorm + RoPE, row statistics, the head's lm_head operand);
//   * the block self-attention of a head runs after the last of its q, k and v
//     tiles is finished (a head ticket);
//   * cross-attention is a phase of its own: every head's keys are split over
//     CTAs (flash-decoding), f16 mma.sync on swizzled cp.async stages, an
//     online softmax per warp, a merge of the warps in shared memory and of the
//     CTAs by the last one to finish (a head ticket);
//   * phases are separated by a grid-wide barrier (an arrival counter and a
//     generation word); every wait is bounded: a wait that exceeds its budget
//     raises the error word and the kernel winds down (waits for its own copies
//     in flight and its MMAs, frees its TMEM) instead of hanging.
// The grid is one CTA per SM (the shared-memory footprint admits no second),
// launched cooperatively so that all CTAs are resident together.
#include <cooperative_groups.h>

#include "linear_parts.cuh"

namespace fm {

namespace {

constexpr int kRing = 4;                          // ring stages
constexpr int kUnit = 2 * kStageBytes;            // 32 KB: two 16 KB chunks per bulk copy
constexpr int kPieceCols = 256;                   // activation columns per staged B piece
constexpr int kCpp = kPieceCols / kChunk;         // chunks per piece
constexpr int kBch = 32 * 128;                    // bytes of one 64-column B chunk (32 rows)
constexpr int kPieceBytes = kCpp * kBch;          // 16 KB
constexpr int kScratch = 64 * 1024;
constexpr int kNAcc = 4;                          // TMEM accumulators of 32 columns
constexpr int kTmemCols = 128;
constexpr uint32_t kIdesc = umma_idesc(128, 32, true);
constexpr int kKeys = 64;                         // keys per attention stage

// shared-memory layout (offsets from the 1024-aligned base)
constexpr int kOffRing = 0;
constexpr int kOffPiece = kOffRing + kRing * kUnit;
constexpr int kOffScratch = kOffPiece + 2 * kPieceBytes;
constexpr int kOffMisc = kOffScratch + kScratch;
// misc: stats [2 jobs][2][kMaxT] f32, flags, barriers, TMEM slot
constexpr int kOffStats = kOffMisc;
constexpr int kOffFlags = kOffStats + 2 * 2 * kMaxT * 4;
constexpr int kOffBars = kOffFlags + 64;
constexpr int kNBars = 2 * kRing + 2 + 2 + 2 * kNAcc + 1;
constexpr int kOffTslot = kOffBars + 8 * kNBars;
constexpr int kSmemUsed = kOffTslot + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;
static_assert(kSmemBytes <= 232448, "shared memory beyond the per-CTA limit");

struct Bars {
  uint32_t base;
  __device__ uint32_t full(int i) const { return base + 8 * i; }
  __device__ uint32_t empty(int i) const { return base + 8 * (kRing + i); }
  __device__ uint32_t bfull(int i) const { return base + 8 * (2 * kRing + i); }
  __device__ uint32_t bempty(int i) const { return base + 8 * (2 * kRing + 2 + i); }
  __device__ uint32_t accfull(int i) const { return base + 8 * (2 * kRing + 4 + i); }
  __device__ uint32_t accempty(int i) const { return base + 8 * (2 * kRing + 4 + kNAcc + i); }
  __device__ uint32_t drain() const { return base + 8 * (2 * kRing + 4 + 2 * kNAcc); }
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
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// All of this CTA's earlier writes are made visible, then the CTA counts itself
// in; the last of G resets the counter and advances the generation.
__device__ __forceinline__ void grid_arrive(uint32_t *bar, int G) {
  __threadfence();
  const uint32_t old = atomicAdd(bar, 1u);
  if (old == (uint32_t)(G - 1)) {
    atomicExch(bar, 0u);
    __threadfence();
    atomicAdd(bar + 32, 1u);
  }
}
// Wait until the generation has advanced `k` times past g0; bounded.
__device__ __forceinline__ bool grid_wait(const uint32_t *bar, uint32_t g0, uint32_t k, int32_t *err) {
  if (ld_acquire(bar + 32) - g0 >= k) return true;
  const long long t0 = clock64();
  long long next = t0 + 4096;
  while (ld_acquire(bar + 32) - g0 < k) {
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

// ---- schedule walkers ------------------------------------------------------------
// A CTA's segments in a linear phase: maximal runs of its chunks inside one tile.
struct Seg {
  int job, tile, gt;   // job, tile in the job, tile in the phase
  int c0, c1;          // chunks [c0, c1) in the phase's sequence
  int k0;              // first chunk column inside the tile (kc)
};
__device__ __forceinline__ int phase_segments(const StepPhase &P, int lo, int hi, Seg (&s)[kStepMaxSeg]) {
  int n = 0;
  int c = lo;
  while (c < hi && n < kStepMaxSeg) {
    const int j = step_job(P, c);
    const StepJob &J = P.jobs[j];
    const int lc = c - J.chunk0;
    const int tile = lc / J.cpt;
    const int end = min(hi, J.chunk0 + (tile + 1) * J.cpt);
    s[n].job = j;
    s[n].tile = tile;
    s[n].gt = J.tile0 + tile;
    s[n].c0 = c;
    s[n].c1 = end;
    s[n].k0 = lc - tile * J.cpt;
    ++n;
    c = end;
  }
  return n;
}

// ---- block self-attention of one head by a group of 4 warps ------------------------
// O = softmax(q k^T * scale) v over the T rows of the block (no mask), from the
// q / k / v rows the head's epilogues stored; one warp per query row.
__device__ void group_self_attention(const GemvArgs &a, int head, int T, float *sm, int bar_id, int gtid) {
  const int hd = a.hd, D = a.self_D;
  const int ks = hd + 4;
  // three [16][hd + 4] f32 tiles: 25 KB at hd 128, inside the group's 32 KB half of the scratch
  float *qq = sm, *kk = sm + 16 * ks, *vv = sm + 2 * 16 * ks;
  const int q4 = hd / 4;
  for (int i = gtid; i < T * q4; i += 128) {
    const int t = i / q4, d = 4 * (i - t * q4);
    const float *row = a.Y + (size_t)t * a.ldy + head * hd + d;
    *reinterpret_cast<float4 *>(qq + t * ks + d) = __ldcg(reinterpret_cast<const float4 *>(row));
    *reinterpret_cast<float4 *>(kk + t * ks + d) = __ldcg(reinterpret_cast<const float4 *>(row + D));
    *reinterpret_cast<float4 *>(vv + t * ks + d) = __ldcg(reinterpret_cast<const float4 *>(row + 2 * D));
  }
  named_sync(bar_id, 128);
  const int lane = threadIdx.x & 31, w = gtid >> 5;
  const bool on = lane < q4;
  for (int t = w; t < T; t += 4) {
    const float *qrow = qq + t * ks;
    const float *krow = kk + (lane < T ? lane : 0) * ks;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    for (int d = 0; d < hd; d += 4) {
      const float4 q = *reinterpret_cast<const float4 *>(qrow + d);
      const float4 k = *reinterpret_cast<const float4 *>(krow + d);
      s0 += q.x * k.x; s1 += q.y * k.y; s2 += q.z * k.z; s3 += q.w * k.w;
    }
    const float sc = lane < T ? ((s0 + s1) + (s2 + s3)) * a.attn_scale : -INFINITY;
    const float mx = warp_max(sc);
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
  named_sync(bar_id, 128);
}

// ---- cross-attention helpers --------------------------------------------------------
// m16n8k8 f16 MMA, f32 accumulate
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
// byte offset of 16-byte unit u of row r in a stage tile of 256-byte rows (hd 128)
// or 128-byte rows (hd 64): units permuted by r % 8, so eight rows reading the
// same unit hit eight distinct bank groups
__device__ __forceinline__ uint32_t kv_slot(int r, int u, int hd) {
  return (uint32_t)(r * hd * 2 + ((u ^ (r & 7)) << 4));
}
// key range of one attention item
struct AttnItem {
  int head, split, kbeg, kend, nst, L;
};
__device__ __forceinline__ AttnItem attn_item(const StepAttn &A, const StepParams *sp, int b) {
  AttnItem it;
  it.head = b / A.nsp;
  it.split = b - it.head * A.nsp;
  it.L = (A.L_src == 0 ? sp->L : sp->pos + 1) + A.L_add;
  int per = (it.L + A.nsp - 1) / A.nsp;
  per = (per + 15) & ~15;
  it.kbeg = min(it.L, it.split * per);
  it.kend = min(it.L, it.kbeg + per);
  it.nst = (it.kend - it.kbeg + kKeys - 1) / kKeys;
  return it;
}
// request rows [rlo, rhi) of key stage st (64 keys) into K / V buffers (rows past
// kend read as zero); 256 worker threads
__device__ __forceinline__ void attn_issue(const StepAttn &A, const AttnItem &it, int st, uint32_t kb, uint32_t vb,
                                           int rlo, int rhi, int tid) {
  const int hd = A.hd;
  const int U = hd / 8;
  const __half *kh = A.Kc + (size_t)it.head * A.max_ctx * hd;
  const __half *vh = A.Vc + (size_t)it.head * A.max_ctx * hd;
  const int k0 = it.kbeg + st * kKeys;
  for (int i = tid + rlo * U; i < rhi * U; i += kWorkers) {
    const int r = i / U, u = i - r * U;
    const int key = k0 + r;
    const bool ok = key < it.kend;
    const size_t off = (size_t)(ok ? key : 0) * hd + u * 8;
    cp_async16(kb + kv_slot(r, u, hd), kh + off, ok ? 16u : 0u);
    cp_async16(vb + kv_slot(r, u, hd), vh + off, ok ? 16u : 0u);
  }
}

}  // namespace

__global__ void __launch_bounds__(kAll, 1) fm_draft_step_kernel(const __grid_constant__ StepArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - smem_u32(smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const int T = a.T;
  const uint32_t ring = base + kOffRing, piece0 = base + kOffPiece, scratch = base + kOffScratch;
  float *stats = reinterpret_cast<float *>(gbase + kOffStats);      // [2][2][kMaxT]: mu, rs per job
  volatile int *flags = reinterpret_cast<volatile int *>(gbase + kOffFlags);
  const Bars bars{base + kOffBars};
  const uint32_t tslot = base + kOffTslot;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNBars; ++i) mbar_init(bars.base + 8 * i, 1);
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc<kTmemCols>(tslot);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = lds32(tslot);

  if (warp == 0) {
    // ---------------------------------------------------------------- weight stream
    if (lane == 0) {
      int u = 0;                 // units issued
      int last_round[kRing];
      for (int i = 0; i < kRing; ++i) last_round[i] = -1;
      bool waited = false;       // griddepcontrol.wait done (the first kRing units go before it)
      bool ok = true;
      for (int p = 0; p < a.n_phases && ok; ++p) {
        const StepPhase &P = a.ph[p];
        if (P.kind != PH_LINEAR) continue;
        const int lo = step_lo(b, P.nchunks, G), hi = step_lo(b + 1, P.nchunks, G);
        for (int j = 0; j < P.njobs && ok; ++j) {
          const StepJob &J = P.jobs[j];
          const int c0 = max(lo, J.chunk0), c1 = min(hi, J.chunk0 + J.nchunks);
          for (int c = c0; c < c1; c += 2) {
            const int st = u % kRing, r = u / kRing;
            if (r >= 1) {
              if (!waited) { pdl_wait(); waited = true; }
              if (!mbar_wait_bounded(bars.empty(st), (r - 1) & 1, a.err)) { ok = false; break; }
            }
            const int nch = min(2, c1 - c);
            mbar_expect_tx(bars.full(st), nch * kStageBytes);
            bulk_g2s(ring + st * kUnit, J.g.Wt + (size_t)(c - J.chunk0) * kStageBytes, nch * kStageBytes,
                     bars.full(st));
            last_round[st] = r;
            ++u;
          }
        }
        stamp(a, p, 3);
      }
      if (!waited) pdl_wait();
      // wind down: every copy this CTA issued has landed before the CTA may exit
      for (int st = 0; st < kRing; ++st)
        if (last_round[st] >= 0) mbar_wait_drain(bars.full(st), last_round[st] & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issue
    pdl_wait();
    int u = 0, sc = 0, pc = 0;   // units, segments, B pieces consumed
    bool ok = true;
    for (int p = 0; p < a.n_phases && ok; ++p) {
      const StepPhase &P = a.ph[p];
      if (P.kind != PH_LINEAR) continue;
      const int lo = step_lo(b, P.nchunks, G), hi = step_lo(b + 1, P.nchunks, G);
      Seg segs[kStepMaxSeg];
      const int ns = phase_segments(P, lo, hi, segs);
      int si = -1, i_in_seg = 0, acc = 0;
      for (int j = 0; j < P.njobs && ok; ++j) {
        const StepJob &J = P.jobs[j];
        const int c0 = max(lo, J.chunk0), c1 = min(hi, J.chunk0 + J.nchunks);
        for (int c = c0; c < c1 && ok; c += 2) {
          const int st = u % kRing, r = u / kRing;
          if (!mbar_wait_warp(bars.full(st), r & 1, a.err)) { ok = false; break; }
          tc_fence_after();
          const int nch = min(2, c1 - c);
          for (int x = 0; x < nch; ++x) {
            const int cc = c + x;
            if (si < 0 || cc >= segs[si].c1) {
              // a new segment: the previous one's accumulator is complete
              if (si >= 0) { umma_commit_elect(bars.accfull(acc)); ++sc; }
              ++si;
              if (si >= ns) { ok = false; break; }   // cannot happen: the host checked the schedule
              acc = sc % kNAcc;
              if (sc >= kNAcc && !mbar_wait_warp(bars.accempty(acc), ((sc / kNAcc) - 1) & 1, a.err)) { ok = false; break; }
              tc_fence_after();
              i_in_seg = 0;
            }
            const int pb = pc & 1;
            if (i_in_seg % kCpp == 0) {
              if (!mbar_wait_warp(bars.bfull(pb), (pc >> 1) & 1, a.err)) { ok = false; break; }
              tc_fence_after();
            }
            const uint64_t ad = umma_desc_sw128(ring + st * kUnit + x * kStageBytes);
            const uint64_t bd = umma_desc_sw128(piece0 + pb * kPieceBytes + (i_in_seg % kCpp) * kBch);
            const uint32_t d = tmem + acc * 32;
#pragma unroll
            for (int kk = 0; kk < kChunk / 16; ++kk)
              umma_ss_elect(d, ad + 2 * kk, bd + 2 * kk, kIdesc, (i_in_seg | kk) ? 1u : 0u);
            if (i_in_seg % kCpp == kCpp - 1 || cc + 1 == segs[si].c1) {
              umma_commit_elect(bars.bempty(pb));
              ++pc;
            }
            ++i_in_seg;
          }
          if (!ok) break;
          umma_commit_elect(bars.empty(st));
          ++u;
        }
      }
      if (ok && si >= 0) { umma_commit_elect(bars.accfull(acc)); ++sc; }
      if (lane == 0) stamp(a, p, 4);
    }
    // wind down: every MMA issued has completed before TMEM is freed
    umma_commit_elect(bars.drain());
    mbar_wait_drain(bars.drain(), 0);
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- workers
    const int tid = wtid();
    const int grp = (warp - 2) >> 2;            // two groups of four warps
    const int gtid = tid & 127;
    pdl_wait();
    uint32_t g0 = 0;
    if (tid == 0) flags[0] = (int)ld_acquire(a.bar + 32);
    named_sync(1, kWorkers);
    g0 = (uint32_t)flags[0];
    int pc = 0, sc = 0;                          // B pieces staged, segments read
    bool ok = true;
    for (int p = 0; p < a.n_phases && ok; ++p) {
      const StepPhase &P = a.ph[p];
      // an earlier request of a later attention phase's stable key rows
      if (P.prefetch >= 0) {
        const StepAttn &A = a.ph[P.prefetch].at;
        if (b < A.n_heads * A.nsp) {
          const AttnItem it = attn_item(A, a.sp, b);
          const int stable = a.sp->stable;
          for (int st = 0; st < 2; ++st) {
            const int pre = st < it.nst ? max(0, min(kKeys, stable - (it.kbeg + st * kKeys))) : 0;
            if (pre > 0)
              attn_issue(A, it, st, scratch + st * 2 * kKeys * A.hd * 2, scratch + (st * 2 + 1) * kKeys * A.hd * 2, 0,
                         pre, tid);
            cp_async_commit();
          }
        }
      }
      // the previous phase is complete everywhere
      if (p > 0) {
        if (tid == 0) flags[1] = grid_wait(a.bar, g0, (uint32_t)p, a.err) ? 1 : 0;
        named_sync(1, kWorkers);
        if (!flags[1]) { ok = false; break; }
      }
      if (tid == 0) stamp(a, p, 0);
      if (P.kind == PH_LINEAR) {
        const int lo = step_lo(b, P.nchunks, G), hi = step_lo(b + 1, P.nchunks, G);
        Seg segs[kStepMaxSeg];
        const int ns = phase_segments(P, lo, hi, segs);
        // stage every piece of every segment (the MMA warp consumes them in order)
        int last_job = -1;
        for (int s = 0; s < ns; ++s) {
          const GemvArgs &g = P.jobs[segs[s].job].g;
          const int kb = segs[s].k0 * kChunk;                     // first column of the segment
          const int ncol = (segs[s].c1 - segs[s].c0) * kChunk;
          const int m0 = segs[s].tile * kTile;
          float *mu = stats + segs[s].job * 2 * kMaxT, *rs = mu + kMaxT;
          for (int x = 0; x < ncol; x += kPieceCols) {
            const int pb = pc & 1;
            // (a wait that gives up raises the error word; the workers still take every
            // named barrier together, so a failure winds the CTA down instead of hanging it)
            if (pc >= 2) mbar_wait_bounded(bars.bempty(pb), ((pc >> 1) - 1) & 1, a.err);
            const int kp = min(kPieceCols, ncol - x);
            StageRegs<1> rg;
            stage_load<1>(g, T, m0, kb + x, kp, rg);
            if (segs[s].job != last_job) {
              // this job's row statistics while the first piece's loads are in flight
              load_row_stats(g, T, mu, rs, tid);
              named_sync(1, kWorkers);
              last_job = segs[s].job;
              if (tid == 0) stamp(a, p, 5);
            }
            stage_store<1>(g, mu, rs, piece0 + pb * kPieceBytes, T, kb + x, kp, rg);
            fence_proxy_async();
            named_sync(1, kWorkers);
            if (tid == 0) mbar_arrive(bars.bfull(pb));
            ++pc;
          }
        }
        if (tid == 0) stamp(a, p, 1);
        // read the accumulators (segment s by group s & 1), publish, reduce
        for (int s = grp; s < ns; s += 2) {
          const StepJob &J = P.jobs[segs[s].job];
          const GemvArgs &g = J.g;
          const int my_sc = sc + s;
          const int acc = my_sc % kNAcc;
          mbar_wait_bounded(bars.accfull(acc), (my_sc / kNAcc) & 1, a.err);
          tc_fence_after();
          const int quad = warp & 3;
          float v[32];
          tmem_ld32(tmem + acc * 32 + ((uint32_t)(quad * 32) << 16), v);   // columns 0..15 hi, 16..31 lo
          tc_fence_before();
          named_sync(2 + grp, 128);
          if (gtid == 0) mbar_arrive(bars.accempty(acc));
          float *mine = a.part + ((size_t)b * kStepMaxSeg + s) * kMaxT * kTile;
          const int row = quad * 32 + lane;
#pragma unroll
          for (int t = 0; t < 16; ++t)
            if (t < T) __stcg(mine + t * kTile + row, v[t] + v[16 + t]);
          __threadfence();
          named_sync(2 + grp, 128);
          // contributors of this tile: with at least as many chunks as CTAs every CTA
          // owns a non-empty range and they are the owners of the tile's first to
          // last chunk; with fewer, each chunk is one CTA's whole range
          const int tc0 = J.chunk0 + segs[s].tile * J.cpt;
          const bool dense = P.nchunks >= G;
          const int blo = step_owner(tc0, P.nchunks, G);
          const int ncontrib = dense ? step_owner(tc0 + J.cpt - 1, P.nchunks, G) - blo + 1 : J.cpt;
          if (gtid == 0) {
            int *tk = a.tickets + segs[s].gt;
            const int old = atomicAdd(tk, 1);
            const bool last = old == ncontrib - 1;
            if (last) atomicExch(tk, 0);
            flags[4 + grp] = last ? 1 : 0;
          }
          named_sync(2 + grp, 128);
          if (!flags[4 + grp]) continue;
          __threadfence();
          // the last contributor: partials in CTA order, then the fused epilogue
          const int m0 = segs[s].tile * kTile;
          const int gw = gtid >> 5;
          for (int t = gw; t < T; t += 4) {
            EpiIn in;
            epilogue_load(g, t, m0, in);
            float vv[4] = {0.f, 0.f, 0.f, 0.f};
            for (int i0 = 0; i0 < ncontrib; i0 += 8) {
              float4 pr[8];
#pragma unroll
              for (int x = 0; x < 8; ++x) {
                pr[x] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (i0 + x < ncontrib) {
                  const int bb = dense ? blo + i0 + x : step_owner(tc0 + i0 + x, P.nchunks, G);
                  // the segment index of this tile in CTA bb's list
                  const int si = segs[s].gt - step_tile(P, step_lo(bb, P.nchunks, G));
                  pr[x] = __ldcg(reinterpret_cast<const float4 *>(
                      a.part + (((size_t)bb * kStepMaxSeg + si) * kMaxT + t) * kTile + 4 * lane));
                }
              }
#pragma unroll
              for (int x = 0; x < 8; ++x) {
                vv[0] += pr[x].x; vv[1] += pr[x].y; vv[2] += pr[x].z; vv[3] += pr[x].w;
              }
            }
            epilogue_unit(g, t, m0, vv, segs[s].tile, in);
          }
          if (J.self_tail) {
            // the block attention of each head of this tile once its q, k and v tiles are all stored
            __threadfence();
            named_sync(2 + grp, 128);
            const int heads = kTile / g.hd;
            if (gtid == 0) {
              const int mseg = m0 % g.self_D;
              for (int i = 0; i < heads; ++i) {
                const int h = mseg / g.hd + i;
                int *tk = a.tickets + kStepTileTickets + h;
                const int old = atomicAdd(tk, 1);
                const bool last = old == 2;
                if (last) atomicExch(tk, 0);
                flags[8 + 2 * grp + i] = last ? h : -1;
              }
            }
            named_sync(2 + grp, 128);
            for (int i = 0; i < heads; ++i) {
              const int h = flags[8 + 2 * grp + i];
              if (h >= 0) {
                __threadfence();
                group_self_attention(g, h, T, reinterpret_cast<float *>(gbase + kOffScratch + grp * (kScratch / 2)),
                                     2 + grp, gtid);
              }
            }
          }
        }
        sc += ns;
      } else {
        // ------------------------------------------------------------ cross-attention
        const StepAttn &A = P.at;
        const int hd = A.hd;
        const bool active = b < A.n_heads * A.nsp;
        AttnItem it;
        if (active) it = attn_item(A, a.sp, b);
        const uint32_t tileb = kKeys * hd * 2;
        auto kbuf = [&](int i) { return scratch + 2 * i * tileb; };
        auto vbuf = [&](int i) { return scratch + (2 * i + 1) * tileb; };
        if (active) {
          // the rest of the first two stages (all of them if nothing was requested early)
          const int stable = A.prefetched ? a.sp->stable : 0;
          for (int st = 0; st < 2; ++st) {
            if (st < it.nst) {
              const int pre = max(0, min(kKeys, stable - (it.kbeg + st * kKeys)));
              if (pre < kKeys) attn_issue(A, it, st, kbuf(st), vbuf(st), pre, kKeys, tid);
            }
            cp_async_commit();
          }
          // queries -> f16 hi / lo tiles in the (idle) B piece area: [16 rows][hd], units permuted by row
          const uint32_t qhi = piece0, qlo = piece0 + 16 * hd * 2;
          const int q4 = hd / 4;
          for (int i = tid; i < 16 * q4; i += kWorkers) {
            const int t = i / q4, d = 4 * (i - t * q4);
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < T) x = __ldcg(reinterpret_cast<const float4 *>(A.Q + (size_t)t * A.ldq + it.head * hd + d));
            uint32_t h01, l01, h23, l23;
            split2_f16(x.x, x.y, h01, l01);
            split2_f16(x.z, x.w, h23, l23);
            const uint32_t off = kv_slot(t, d >> 3, hd) + (d & 7) * 2;
            asm volatile("st.shared.v2.u32 [%0], {%1,%2};\n" ::"r"(qhi + off), "r"(h01), "r"(h23));
            asm volatile("st.shared.v2.u32 [%0], {%1,%2};\n" ::"r"(qlo + off), "r"(l01), "r"(l23));
          }
          // per warp: keys 8w .. 8w + 7 of each stage; thread rows g and g + 8
          const int w = warp - 2, gq = lane >> 2, q = lane & 3;
          const int NT = hd / 8;
          float o[16][4];
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
          float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
          const int mi = lane >> 3, ri = lane & 7;
          for (int st = 0; st < it.nst; ++st) {
            cp_async_wait<1>();
            named_sync(1, kWorkers);
            const uint32_t kb = kbuf(st & 1), vb = vbuf(st & 1);
            const int key = 8 * w + ri;     // this lane's row address for ldmatrix
            float s4[4] = {0.f, 0.f, 0.f, 0.f};
            float s4b[4] = {0.f, 0.f, 0.f, 0.f};
            for (int ks = 0; ks < hd / 16; ks += 2) {
              uint32_t b0, b1, b2, b3;
              ldsm_x4(kb + kv_slot(key, 2 * ks + mi, hd), b0, b1, b2, b3);
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
            // scores (log2 domain), masked past kend; rows g (s[0], s[1]) and g + 8 (s[2], s[3])
            const int kabs = it.kbeg + st * kKeys + 8 * w + 2 * q;
            float s[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int kk = kabs + (e & 1);
              s[e] = kk < it.kend ? (s4[e] + s4b[e]) * A.scale_log2 : -INFINITY;
            }
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
            float pr[4];
            float rsum[2] = {0.f, 0.f};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float mm = m_r[e >> 1];
              pr[e] = mm == -INFINITY ? 0.f : exp2f(s[e] - mm);
              rsum[e >> 1] += pr[e];
            }
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              rsum[h2] += __shfl_xor_sync(0xffffffffu, rsum[h2], 1);
              rsum[h2] += __shfl_xor_sync(0xffffffffu, rsum[h2], 2);
              l_r[h2] = l_r[h2] * alpha[h2] + rsum[h2];
            }
            uint32_t ph0, pl0, ph1, pl1;
            split2_f16(pr[0], pr[1], ph0, pl0);   // row g, keys 2q, 2q + 1
            split2_f16(pr[2], pr[3], ph1, pl1);   // row g + 8
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
              if (nt < NT) {
                o[nt][0] *= alpha[0]; o[nt][1] *= alpha[0];
                o[nt][2] *= alpha[1]; o[nt][3] *= alpha[1];
              }
            }
            // O += P V: B = V[8 keys][8 dims] via ldmatrix.trans, four n-tiles per load
#pragma unroll
            for (int nt = 0; nt < 16; nt += 4) {
              if (nt < NT) {
                uint32_t v0, v1, v2, v3;
                asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                             : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                             : "r"(vb + kv_slot(key, nt + mi, hd)));
                mma_f16_k8(o[nt], ph0, ph1, v0);
                mma_f16_k8(o[nt], pl0, pl1, v0);
                mma_f16_k8(o[nt + 1], ph0, ph1, v1);
                mma_f16_k8(o[nt + 1], pl0, pl1, v1);
                mma_f16_k8(o[nt + 2], ph0, ph1, v2);
                mma_f16_k8(o[nt + 2], pl0, pl1, v2);
                mma_f16_k8(o[nt + 3], ph0, ph1, v3);
                mma_f16_k8(o[nt + 3], pl0, pl1, v3);
              }
            }
            named_sync(1, kWorkers);   // every warp is done with this stage's buffers
            if (st + 2 < it.nst) attn_issue(A, it, st + 2, kbuf(st & 1), vbuf(st & 1), 0, kKeys, tid);
            cp_async_commit();
          }
          cp_async_wait<0>();
          named_sync(1, kWorkers);
          // merge the eight warps in three halving rounds through the scratch
          float *mo = reinterpret_cast<float *>(gbase + kOffScratch);        // [4][16][hd]
          float *mml = mo + 4 * 16 * hd;                                     // [4][16][2]
          for (int half = 4; half >= 1; half >>= 1) {
            if (w >= half && w < 2 * half) {
              const int ww = w - half;
#pragma unroll
              for (int nt = 0; nt < 16; ++nt) {
                if (nt < NT) {
                  const int d = 8 * nt + 2 * q;
                  *reinterpret_cast<float2 *>(mo + (ww * 16 + gq) * hd + d) = make_float2(o[nt][0], o[nt][1]);
                  *reinterpret_cast<float2 *>(mo + (ww * 16 + gq + 8) * hd + d) = make_float2(o[nt][2], o[nt][3]);
                }
              }
              if (q == 0) {
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
                    const float2 x = *reinterpret_cast<const float2 *>(mo + (w * 16 + row) * hd + 8 * nt + 2 * q);
                    o[nt][2 * h2] = o[nt][2 * h2] * f1 + x.x * f2;
                    o[nt][2 * h2 + 1] = o[nt][2 * h2 + 1] * f1 + x.y * f2;
                  }
                }
              }
            }
            named_sync(1, kWorkers);
          }
          // this CTA's partial (unnormalised rows, max, sum) to global memory
          float *po = a.apart + (size_t)b * (kMaxT * hd + 2 * kMaxT);
          float *pml = po + kMaxT * hd;
          if (w == 0) {
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
              if (nt < NT) {
                const int d = 8 * nt + 2 * q;
                __stcg(reinterpret_cast<float2 *>(po + gq * hd + d), make_float2(o[nt][0], o[nt][1]));
                __stcg(reinterpret_cast<float2 *>(po + (gq + 8) * hd + d), make_float2(o[nt][2], o[nt][3]));
              }
            }
            if (q == 0) {
              __stcg(reinterpret_cast<float2 *>(pml + 2 * gq), make_float2(m_r[0], l_r[0]));
              __stcg(reinterpret_cast<float2 *>(pml + 2 * (gq + 8)), make_float2(m_r[1], l_r[1]));
            }
            __threadfence();
          }
          named_sync(1, kWorkers);
          if (tid == 0) {
            int *tk = a.tickets + kStepTileTickets + kStepHeadTickets + it.head;
            const int old = atomicAdd(tk, 1);
            const bool last = old == A.nsp - 1;
            if (last) atomicExch(tk, 0);
            flags[2] = last ? 1 : 0;
          }
          named_sync(1, kWorkers);
          if (flags[2]) {
            // the last CTA of the head merges the splits in order: per row the
            // weight of each split, exp2(m_s - M) / sum_s' exp2(m_s' - M) l_s', then
            // the weighted sum of the unnormalised rows
            __threadfence();
            const int b0 = it.head * A.nsp;
            const size_t stride = (size_t)kMaxT * hd + 2 * kMaxT;
            float *fw = reinterpret_cast<float *>(gbase + kOffScratch);   // [16][nsp]
            if (tid < 16) {
              const int t = tid;
              float M = -INFINITY;
              for (int sp = 0; sp < A.nsp; ++sp)
                M = fmaxf(M, __ldcg(a.apart + (b0 + sp) * stride + kMaxT * hd + 2 * t));
              float den = 0.f;
              for (int sp = 0; sp < A.nsp; ++sp) {
                const float2 ml = __ldcg(reinterpret_cast<const float2 *>(a.apart + (b0 + sp) * stride + kMaxT * hd + 2 * t));
                const float f = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
                fw[t * A.nsp + sp] = f;
                den += f * ml.y;
              }
              const float inv = 1.f / den;
              for (int sp = 0; sp < A.nsp; ++sp) fw[t * A.nsp + sp] *= inv;
            }
            named_sync(1, kWorkers);
            for (int i = tid; i < 16 * (hd / 4); i += kWorkers) {
              const int t = i / (hd / 4), d = 4 * (i - t * (hd / 4));
              if (t >= T) continue;
              float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int sp = 0; sp < A.nsp; ++sp) {
                const float f = fw[t * A.nsp + sp];
                const float4 x = __ldcg(reinterpret_cast<const float4 *>(a.apart + (b0 + sp) * stride + t * hd + d));
                acc4.x += f * x.x; acc4.y += f * x.y; acc4.z += f * x.z; acc4.w += f * x.w;
              }
              *reinterpret_cast<float4 *>(A.out + (size_t)t * A.ldo + it.head * hd + d) = acc4;
            }
          }
        } else {
          cp_async_wait<0>();
        }
      }
      // this phase is done here
      named_sync(1, kWorkers);
      if (tid == 0) {
        stamp(a, p, 2);
        grid_arrive(a.bar, G);
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_free<kTmemCols>(tmem);
  }
}

size_t step_smem_bytes() { return (size_t)kSmemBytes; }
size_t step_apart_floats(int hd) { return (size_t)kMaxT * hd + 2 * kMaxT; }

// attrs: bit 0 = cooperative launch (the driver co-schedules every CTA), bit 1 =
// programmatic stream serialisation (the CTAs may start while the previous
// kernel drains; they call griddepcontrol.wait before reading its results)
cudaError_t launch_step(const StepArgs &a, int grid, cudaStream_t st, int attrs) {
  cudaError_t e = cudaFuncSetAttribute(fm_draft_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kAll, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
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

int step_max_grid() {
  int n = 0;
  if (cudaFuncSetAttribute(fm_draft_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fm_draft_step_kernel, kAll, kSmemBytes) != cudaSuccess) return 0;
  return n;
}

}  // namespace fm
