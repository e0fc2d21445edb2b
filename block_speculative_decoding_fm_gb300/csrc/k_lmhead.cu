// k_lmhead.cu -- lm_head over the tied token table fused with the per-row
// argmax: tok[t] = argmax_v sum_k Y[t][k] E[v][k]   (ties -> lowest v).
//
// The pages run the 16 slots through the target's token-table matvec and a
// separate argmaxRows pass (flashmap_drafter.js ``draft``; the table is Q8_0 in
// the GGUF block format the MTP loader on ternary_bonsai_2_mtp.js repacks into
// an int8 plane and a scale plane).  Here one persistent kernel streams the
// table once and the logits never reach memory:
//   * Y is split into hi + lo 16-bit halves (by the head GEMV's epilogue, or
//     here) as the B operand (N = 32: per group of 8 slots, 8 hi rows then 8 lo
//     rows) in the tensor cores' 128-byte-swizzle K-major layout, streamed with
//     the table or kept resident in shared memory;
//   * a producer warp streams 128-row x 64-column table chunks with 1-D bulk
//     TMA copies into an mbarrier ring;
//   * bf16 table: the chunk is already a swizzled K-major tile; the MMA warp
//     (an elected lane issuing) runs tcgen05.mma (M = 128 table rows) into a
//     TMEM accumulator per tile;
//   * Q8_0 table: converter warps form each weight times its block scale in
//     f16 (one rounding: relative error <= 2^-11 per weight, so a logit's
//     relative error stays near 3e-4 for these sums; kWeightResidual adds the
//     exact f16 residual as a second A operand, at twice the converter and MMA
//     work) and store it into TMEM, which tcgen05.mma reads as the A operand, so
//     each tile's whole K accumulates into one f32 accumulator per issuing warp;
//   * each tile's rows keep a running (value, index) best per slot; pass two is
//     the last CTA reducing the per-CTA bests (one warp per slot).
#include <mutex>
#include <type_traits>

#include "dev_common.cuh"
#include "fm_internal.h"

namespace fm {

namespace {

constexpr int kChunk = 64;
// Q8_0: also feed the residual of each weight's f16 rounding (exact products, twice the converter work)
constexpr bool kWeightResidual = false;
constexpr int kBfStage = kTile * kChunk * 2;  // 16 KB bf16 chunk
constexpr int kYChunk = kLmYChunk;            // one 64-column chunk of the resident Y (32 rows x 128 B)
constexpr int kBfWorkers = 128;               // bf16: warps 2..5
constexpr int kBase = 64;                     // warp 0: producer, warp 1: TMEM owner + MMA issuer


// Four offset-binary bytes u = q + 128 (the repacked table's form) -> two f16x2
// words holding q exactly: each byte goes into the low mantissa bits of 1024.0
// (0x64 high byte), then 1024 + 128 is subtracted (the published "magic number"
// int-to-float conversion).  One byte permute per pair, no sign handling.
__device__ __forceinline__ void ob8x4_to_f16x4(uint32_t u, uint32_t &w01, uint32_t &w23) {
  const uint32_t h01 = __byte_perm(u, 0x64646464u, 0x4140);
  const uint32_t h23 = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  __half2 r01 = __hsub2(*reinterpret_cast<const __half2 *>(&h01), bias);
  __half2 r23 = __hsub2(*reinterpret_cast<const __half2 *>(&h23), bias);
  w01 = *reinterpret_cast<uint32_t *>(&r01);
  w23 = *reinterpret_cast<uint32_t *>(&r23);
}

// tcgen05.mma with A in tensor memory (lane = A row, 32-bit columns hold K pairs),
// issued by one elected lane of a warp that runs the issue loop together
__device__ __forceinline__ void umma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16], bool wait = true) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
  if (wait) asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}
// 16 columns of this thread's lane; the caller waits with tmem_ld_wait() before using them
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&f)[16]) {
  uint32_t v[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(v[i]);
}

// Y (f32 [T][ldy]) -> resident B operand: hi and lo halves (f16 for the Q8
// table, bf16 for the bf16 table), slots >= T zero.
template <bool Q8>
__device__ void stage_y(const LmArgs &a, uint32_t ybuf, int T, int tid, int nthreads) {
  const int q4 = a.H >> 2;
  constexpr int kBatch = 8;
  for (int i0 = tid; i0 < 16 * q4; i0 += nthreads * kBatch) {
    float4 y[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int i = i0 + b * nthreads;
      const int t = i / q4, k = (i - t * q4) * 4;
      y[b] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < 16 * q4 && t < T) y[b] = __ldcg(reinterpret_cast<const float4 *>(a.Y + (size_t)t * a.ldy + k));
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int i = i0 + b * nthreads;
      if (i >= 16 * q4) break;
      const int t = i / q4, k = (i - t * q4) * 4;
      const float v[4] = {y[b].x, y[b].y, y[b].z, y[b].w};
      uint32_t hw[2], lw[2];
      if (Q8) {
        split2_f16(v[0], v[1], hw[0], lw[0]);
        split2_f16(v[2], v[3], hw[1], lw[1]);
      } else {
        split2_bf16(v[0], v[1], hw[0], lw[0]);
        split2_bf16(v[2], v[3], hw[1], lw[1]);
      }
      const uint32_t cb = ybuf + (uint32_t)(k >> 6) * kYChunk;
      const int r = lm_yrow(t);
      asm volatile("st.shared.v2.u32 [%0], {%1,%2};\n" ::"r"(cb + sw128(r, k & 63)), "r"(hw[0]), "r"(hw[1]));
      asm volatile("st.shared.v2.u32 [%0], {%1,%2};\n" ::"r"(cb + sw128(r + 8, k & 63)), "r"(lw[0]), "r"(lw[1]));
    }
  }
}

// Per-CTA best per slot from the per-thread bests (each worker thread owns one
// table row per tile and NB slots starting at t0), then the cross-CTA pass.
template <int NB>
__device__ void finish_argmax(const LmArgs &a, int T, bool worker, int t0, float (&bv)[NB], int (&bi)[NB]) {
  __shared__ float s_v[4][16];
  __shared__ int s_i[4][16];
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, quad = (threadIdx.x >> 5) & 3;
  if (worker) {
#pragma unroll
    for (int j = 0; j < NB; ++j) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv[j], o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi[j], o);
        if (better(ov, oi, bv[j], bi[j])) { bv[j] = ov; bi[j] = oi; }
      }
      if (lane == 0) {
        s_v[quad][t0 + j] = bv[j];
        s_i[quad][t0 + j] = bi[j];
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < 16) {
    const int t = threadIdx.x;
    float v = s_v[0][t];
    int i = s_i[0][t];
    for (int qd = 1; qd < 4; ++qd)
      if (better(s_v[qd][t], s_i[qd][t], v, i)) { v = s_v[qd][t]; i = s_i[qd][t]; }
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
  // the last CTA: one warp per slot, the lanes take the CTAs' bests 32 apart with all
  // their loads in flight, then a shuffle reduction (ties -> lowest index, any order)
  const int wq = threadIdx.x >> 5, nwq = blockDim.x >> 5;
  constexpr int kPer = 8;   // per lane in flight: grids up to 256 CTAs in one round
  for (int t = wq; t < T; t += nwq) {
    float v = -INFINITY;
    int i = 0x7fffffff;
    float2 p[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int b = lane + 32 * j;
      p[j] = b < (int)gridDim.x ? __ldcg(a.part + b * kMaxT + t) : make_float2(-INFINITY, __int_as_float(0x7fffffff));
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int pi = __float_as_int(p[j].y);
      if (better(p[j].x, pi, v, i)) { v = p[j].x; i = pi; }
    }
    for (int b = lane + 32 * kPer; b < (int)gridDim.x; b += 32) {
      const float2 q = __ldcg(a.part + b * kMaxT + t);
      const int qi = __float_as_int(q.y);
      if (better(q.x, qi, v, i)) { v = q.x; i = qi; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, i, o);
      if (better(ov, oi, v, i)) { v = ov; i = oi; }
    }
    if (lane == 0) {
      int32_t *out = a.tokens ? a.tokens : a.sp->tokens;
      out[t] = i == 0x7fffffff ? -1 : i;
    }
  }
}

// The producer's copy of a pre-split Y (kLmYChunk per 64 columns) into the resident operand.
__device__ __forceinline__ void load_ylm(const LmArgs &a, uint32_t ybuf, uint32_t yfull) {
  const uint32_t bytes = (uint32_t)(a.H / kChunk) * kYChunk;
  mbar_expect_tx(yfull, bytes);
  for (uint32_t off = 0; off < bytes; off += 16384)
    bulk_g2s(ybuf + off, a.ylm + off, bytes - off < 16384 ? bytes - off : 16384, yfull);
}

__device__ __forceinline__ int my_tile_count(int n_tiles) {
  return (int)blockIdx.x < n_tiles ? (n_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
}

}  // namespace

// ---------------------------------------------------------------- Q8_0 table
// The block scale is folded into the A operand: for table row r and 32-column
// block b, the converters form w = q * d (int8 times the f16 block scale, exact
// in f32) as two f16 halves, hi = rn(q d) and lo = rn(q d - hi) (one f16
// multiply and one fused multiply-add; lo holds the exact residual, which has
// at most 9 significant bits), and write both to TMEM.  The MMAs then run the
// whole K extent of a tile into one f32 accumulator (A = hi, then A = lo, each
// against the Y hi/lo rows), so the epilogue touches each tile once.
// Roles: warp 0 streams the table, warp 1 owns TMEM and issues MMAs, warps
// 2..17 convert (two sets of 8: set h takes chunk h of each pair; in a set,
// one thread per table row and 32-column block), warps 18..21 read each
// finished tile and keep the per-row running best, warp 22 is the second MMA
// issuer (pairs alternate between the issuers, each with its own accumulator).
// Work moves in pairs of chunks (G = 2; G = 1 when a tile's chunk count is odd).
// TMEM columns: A slot i < kNA at kSlotW i (6 slots of 64 columns, so the
// converters can run five pairs ahead of the MMAs; 3 of 128 with the f16
// residual), chunk h of the pair at + kSlotW / 2 h, hi at + 0 (and lo at + 32)
// (16 columns per 32-column block); accumulators at 384 + 64 me + 32 db
// (issuer me, tile parity db), per group of 8 slots 8 hi then 8 lo columns.
// Y operand: kStreamY (Y pre-split in global memory): each ring stage carries
// the Y chunks its table chunks need, so the ring can be deep; otherwise Y is
// split here and stays resident, and the ring gets what shared memory is left.
constexpr int kQ8Conv = 16, kQ8Epi = 4;   // warps
constexpr int kQ8Issuer2 = 2 + kQ8Conv + kQ8Epi;
constexpr int kQ8Threads = kBase + 32 * (kQ8Conv + kQ8Epi + 1);

// bytes of one ring stage: (streamed Y chunks, then) U table chunks, 1024-aligned
__host__ __device__ constexpr int q8_stage_bytes(bool stream_y, int U) {
  return ((stream_y ? U * kYChunk : 0) + U * kQ8Chunk + 1023) / 1024 * 1024;
}

// position of a chunk in the ring: stage, offset inside the stage's unit, phase parity
struct RingPos {
  int st = 0, uo = 0;
  uint32_t par = 0;
  __device__ __forceinline__ void step(int n, int U, int S) {
    uo += n;
    while (uo >= U) {
      uo -= U;
      if (++st == S) { st = 0; par ^= 1; }
    }
  }
};

template <bool kStreamY>
__global__ void __launch_bounds__(kQ8Threads, 1) fm_lmhead_q8_kernel(const __grid_constant__ LmArgs a, const int S, const int U, const int NI, const int G) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  constexpr int SB = kQ8Chunk;
  // A slots: with the f16 residual a slot holds a pair's hi and lo halves (128 columns, 3 slots); without
  // it a pair's two chunks take 64 columns, so 6 slots fit and the converters run five pairs ahead
  constexpr int kNA = kWeightResidual ? 3 : 6;
  constexpr int kSlotW = kWeightResidual ? 128 : 64, kChunkW = kSlotW / 2;
  constexpr int kD = kSlotW * kNA;   // first accumulator column (384)
  constexpr uint32_t IDESC = umma_idesc(128, 32, false);
  const int H = a.H, kcs = H / kChunk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ybuf = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t ring = kStreamY ? ybuf : ybuf + kcs * kYChunk;
  // a ring stage holds U consecutive chunks of one tile, moved by one bulk copy: the
  // copy engine takes a roughly fixed time per copy, so fewer, larger copies stream faster
  const int SS = q8_stage_bytes(kStreamY, U);          // stage stride
  const int TOFF = kStreamY ? U * kYChunk : 0;         // table offset inside a stage
  const uint32_t bars = ring + S * SS;
  auto full = [&](int i) { return bars + 8 * i; };
  auto empty = [&](int i) { return bars + 8 * (S + i); };
  auto afull = [&](int i) { return bars + 8 * (2 * S + i); };
  auto aempty = [&](int i) { return bars + 8 * (2 * S + kNA + i); };
  auto dfull = [&](int j) { return bars + 8 * (2 * S + 2 * kNA + j); };
  auto dempty = [&](int j) { return bars + 8 * (2 * S + 2 * kNA + 2 + j); };
  const uint32_t yfull = bars + 8 * (2 * S + 2 * kNA + 4);
  const uint32_t tslot = yfull + 8;

  const int n_tiles = (a.V + kTile - 1) / kTile;
  const int tiles = my_tile_count(n_tiles);
  const int total = tiles * kcs;
  const int units = total / U;
  const int npairs = total / G;                        // G divides kcs
  const size_t tile_stride = (size_t)gridDim.x * kcs * SB;   // bytes between this CTA's tiles
  const uint8_t *first = a.q8 + (size_t)blockIdx.x * kcs * SB;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full(i), 1);
      // free once the converters that read its table chunks (one set per chunk, both
      // sets when a unit spans a pair) and, for streamed Y, the issuers' MMAs are done
      mbar_init(empty(i), (U == 1 ? kQ8Conv / 2 : kQ8Conv) + (kStreamY ? NI : 0));
    }
    for (int i = 0; i < kNA; ++i) {
      mbar_init(afull(i), (kQ8Conv / 2) * G);
      mbar_init(aempty(i), 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(dfull(j), NI);
      mbar_init(dempty(j), kQ8Epi);
    }
    mbar_init(yfull, 1);
    mbar_fence_init();
    // the table does not depend on earlier kernels; a CTA's units walk its tiles in order
    const uint8_t *src = first;
    int kc = 0;
    for (int j = 0; j < S && j < units; ++j) {
      // streamed Y: one expect for the stage's table and Y bytes; Y is copied after griddepcontrol.wait
      mbar_expect_tx(full(j), U * SB + (kStreamY ? U * kYChunk : 0));
      bulk_g2s(ring + j * SS + TOFF, src + (size_t)kc * SB, U * SB, full(j));
      kc += U;
      if (kc == kcs) { kc = 0; src += tile_stride; }
    }
  }
  if (warp == 1) tmem_alloc<512>(tslot);
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = lds32(tslot);
  pdl_wait();
  const int T = a.T_const > 0 ? a.T_const : a.sp->T;

  if (!kStreamY && warp >= 2) {
    stage_y<true>(a, ybuf, T, (int)threadIdx.x - kBase, kQ8Threads - kBase);
    fence_proxy_async();
    named_sync(1, kQ8Threads - kBase);
    if (threadIdx.x == kBase) mbar_arrive(yfull);
  }

  const int quad = warp & 3;   // TMEM lanes 32 quad .. + 31 belong to this warp
  const int r = 32 * quad + lane;
  const uint32_t lane_base = tmem + ((uint32_t)(32 * quad) << 16);
  float bv[16];
  int bi[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) { bv[i] = -INFINITY; bi[i] = 0x7fffffff; }

  // the MMA issuers: one code path per issuer, so that every value the MMAs take
  // (TMEM and shared-memory addresses) derives from compile-time constants and
  // warp-uniform counters
  auto issue = [&](auto me_c) {
    constexpr int me = decltype(me_c)::value;
    // the whole warp runs the issue loop (warp-uniform state); one elected lane issues.
    // Issuer me takes pairs me, me + NI, ...: a tile's pairs alternate between the
    // issuers (the launcher makes their count even).  Counters only: a division or
    // modulo by a runtime value in this loop slowed the MMA stream threefold.
    if (me < NI && mbar_wait_warp(yfull, 0, a.err)) {
      const int stride = G * NI;            // chunks from one of this issuer's pairs to the next
      int kc = G * me, tl = 0;              // the pair's first chunk in its tile; the tile
      int i = me, q = 0;                    // A slot (pair % kNA) and pair / kNA
      RingPos y;                            // ring position of the pair's first chunk
      y.step(G * me, U, S);
      for (int sc = me; sc < npairs; sc += NI) {
        const int db = tl & 1;
        const uint32_t d = tmem + kD + 64 * me + 32 * db;
        const bool first_in_tile = kc == G * me;
        if (first_in_tile && tl >= 2 && !mbar_wait_warp(dempty(db), ((tl >> 1) - 1) & 1, a.err)) break;
        if (!mbar_wait_warp(afull(i), (uint32_t)q & 1, a.err)) break;
        tc_fence_after();
        RingPos y2 = y;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h < G) {
            // (streamed Y: the converters' afull for this chunk implies its stage has landed)
            const uint64_t bd = umma_desc_sw128(kStreamY ? ring + y2.st * SS + y2.uo * kYChunk
                                                          : ybuf + (kc + h) * kYChunk);
            const uint32_t ah = tmem + kSlotW * i + kChunkW * h;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              umma_ts_elect(d, ah + 8 * kk, bd + 2 * kk, IDESC, (first_in_tile && h == 0 && kk == 0) ? 0u : 1u);
              if constexpr (kWeightResidual) umma_ts_elect(d, ah + 32 + 8 * kk, bd + 2 * kk, IDESC, 1u);
            }
            // one issuer: release the stage after its last chunk; two: each releases after its pair
            if (kStreamY && ((NI == 1 && y2.uo == U - 1) || (NI == 2 && h == G - 1))) umma_commit_elect(empty(y2.st));
            y2.step(1, U, S);
          }
        }
        umma_commit_elect(aempty(i));
        if (kc + stride >= kcs) umma_commit_elect(dfull(db));   // this issuer's last pair of the tile
        y.step(stride, U, S);
        kc += stride;
        if (kc >= kcs) { kc -= kcs; ++tl; }
        i += NI;
        if (i >= kNA) { i -= kNA; ++q; }
      }
    }
  };

  if (warp == 0) {
    if (lane == 0) {
      // split K (y_slice_tiles > 0): the rows of tile t hold K slice t / y_slice_tiles,
      // whose Y chunks follow the earlier slices' in the operand
      auto ychunk = [&](int tile, int c) {
        const int sl = a.y_slice_tiles > 0 ? tile / a.y_slice_tiles : 0;
        return a.ylm + ((size_t)sl * kcs + c) * kYChunk;
      };
      if (kStreamY) {
        // the Y chunks of the first stages (Y is this call's data: after griddepcontrol.wait)
        int kc = 0, tile = blockIdx.x;
        for (int j = 0; j < S && j < units; ++j) {
          bulk_g2s(ring + j * SS, ychunk(tile, kc), U * kYChunk, full(j));
          kc += U;
          if (kc == kcs) { kc = 0; tile += gridDim.x; }
        }
        mbar_arrive(yfull);
      }
      // unit j reuses stage j % S once unit j - S is released
      const uint8_t *src = first;
      int kc = 0, tile = blockIdx.x;
      for (int j = 0; j < S && j < units; ++j) {
        kc += U;
        if (kc == kcs) { kc = 0; src += tile_stride; tile += gridDim.x; }
      }
      int st = 0;
      uint32_t par = 0;
      for (int j = S; j < units; ++j) {
        if (!mbar_wait_bounded(empty(st), par, a.err)) break;
        mbar_expect_tx(full(st), U * SB + (kStreamY ? U * kYChunk : 0));
        bulk_g2s(ring + st * SS + TOFF, src + (size_t)kc * SB, U * SB, full(st));
        if (kStreamY) bulk_g2s(ring + st * SS, ychunk(tile, kc), U * kYChunk, full(st));
        kc += U;
        if (kc == kcs) { kc = 0; src += tile_stride; tile += gridDim.x; }
        if (++st == S) { st = 0; par ^= 1; }
      }
    }
  } else if (warp == 1) {
    issue(std::integral_constant<int, 0>());
  } else if (warp == kQ8Issuer2) {
    issue(std::integral_constant<int, 1>());
  } else if (warp < 2 + kQ8Conv) {
    // converters: set h takes chunk h of each pair; thread = (row r, block b) of the chunk
    const int h = (warp - 2) >> 3;
    const int b = ((warp - 2) >> 2) & 1;
    if (h < G) {
      const uint32_t x = (uint32_t)((r >> 1) & 3);
      const uint32_t o0 = (uint32_t)r * 64 + (((2 * b) ^ x) << 4), o1 = (uint32_t)r * 64 + (((2 * b + 1) ^ x) << 4);
      // the row's f16 block scale (two rows per 32-bit word in the chunk's scale plane)
      const uint32_t soff = (uint32_t)kTile * 64 + (uint32_t)b * 256 + (uint32_t)(r & ~1) * 2;
      const uint32_t dsel = (r & 1) ? 0x3232u : 0x1010u;   // this row's f16 scale, in both halves
      RingPos c;
      c.step(h, U, S);
      int i = 0;
      uint32_t apar = 0;
      for (int sc = 0; sc < npairs; ++sc) {
        if (sc >= kNA && !mbar_wait_bounded(aempty(i), apar ^ 1, a.err)) break;
        // first chunk of this set in the stage's unit: wait for the stage
        if (c.uo < G && !mbar_wait_bounded(full(c.st), c.par, a.err)) break;
        tc_fence_after();
        const uint32_t buf = ring + c.st * SS + TOFF + c.uo * SB;
        const uint4 v0 = lds128(buf + o0), v1 = lds128(buf + o1);
        const uint32_t sw = lds32(buf + soff);
        const uint32_t dpair = __byte_perm(sw, 0u, dsel);
        const __half2 d2 = *reinterpret_cast<const __half2 *>(&dpair);
        uint32_t w[16];
        ob8x4_to_f16x4(v0.x, w[0], w[1]);
        ob8x4_to_f16x4(v0.y, w[2], w[3]);
        ob8x4_to_f16x4(v0.z, w[4], w[5]);
        ob8x4_to_f16x4(v0.w, w[6], w[7]);
        ob8x4_to_f16x4(v1.x, w[8], w[9]);
        ob8x4_to_f16x4(v1.y, w[10], w[11]);
        ob8x4_to_f16x4(v1.z, w[12], w[13]);
        ob8x4_to_f16x4(v1.w, w[14], w[15]);
        // last chunk of this set in the unit: the stage may be refilled after these loads
        if (c.uo + G >= U) {
          __syncwarp();
          if (lane == 0) mbar_arrive(empty(c.st));
        }
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const __half2 q = *reinterpret_cast<const __half2 *>(&w[j]);
          const __half2 ph = __hmul2(q, d2);
          hi[j] = *reinterpret_cast<const uint32_t *>(&ph);
          if constexpr (kWeightResidual) {
            const __half2 pl = __hfma2(q, d2, __hneg2(ph));
            lo[j] = *reinterpret_cast<const uint32_t *>(&pl);
          }
        }
        const uint32_t ta = lane_base + kSlotW * i + kChunkW * h + 16 * b;
        if constexpr (kWeightResidual) {
          tmem_st16(ta, hi, false);
          tmem_st16(ta + 32, lo);
        } else {
          tmem_st16(ta, hi);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(afull(i));
        if (++i == kNA) { i = 0; apar ^= 1; }
        c.step(G, U, S);
      }
    }
  } else if (warp < 2 + kQ8Conv + kQ8Epi) {
    // epilogue: one finished tile at a time; row r, all 16 slots (8 hi then 8 lo columns per group)
    int tile = blockIdx.x;
    for (int tl = 0; tl < tiles; ++tl, tile += gridDim.x) {
      const int db = tl & 1;
      if (!mbar_wait_bounded(dfull(db), (tl >> 1) & 1, a.err)) break;
      tc_fence_after();
      const int v = tile * kTile + r;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        uint32_t d0[16], d1[16];
        tmem_ld16_async(lane_base + kD + 32 * db + 16 * g, d0);
        if (NI == 2) tmem_ld16_async(lane_base + kD + 64 + 32 * db + 16 * g, d1);
        tmem_ld_wait();
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          float l = __uint_as_float(d0[t]) + __uint_as_float(d0[8 + t]);
          if (NI == 2) l += __uint_as_float(d1[t]) + __uint_as_float(d1[8 + t]);
          const int slot = 8 * g + t;
          if (v < a.V && slot < T) {
            if (a.logits) a.logits[(size_t)slot * a.V + v] = l;
            if (better(l, v, bv[slot], bi[slot])) { bv[slot] = l; bi[slot] = v; }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dempty(db));
    }
  }
  finish_argmax<16>(a, T, warp >= 2 + kQ8Conv && warp < kQ8Issuer2, 0, bv, bi);
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_free<512>(tmem);
  }
}

// ---------------------------------------------------------------- bf16 table
// TMEM columns: per-tile accumulator, double buffered at 0 and 32.  Y either
// streams with the table (each stage: U Y chunks, then U table chunks) or stays
// resident, as in the Q8_0 kernel.
__host__ __device__ constexpr int bf_stage_bytes(bool stream_y, int U) {
  return (stream_y ? U * kYChunk : 0) + U * kBfStage;   // multiples of 1024
}

template <bool kStreamY>
__global__ void __launch_bounds__(kBase + kBfWorkers, 1) fm_lmhead_bf16_kernel(const __grid_constant__ LmArgs a, const int S, const int U) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  constexpr int SB = kBfStage;
  constexpr uint32_t IDESC = umma_idesc(128, 32, true);
  const int H = a.H, kcs = H / kChunk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ybuf = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t ring = kStreamY ? ybuf : ybuf + kcs * kYChunk;
  // a ring stage holds U consecutive chunks of one tile, moved by one bulk copy: the
  // copy engine takes a roughly fixed time per copy, so fewer, larger copies stream faster
  const int SS = bf_stage_bytes(kStreamY, U);
  const int TOFF = kStreamY ? U * kYChunk : 0;
  const uint32_t bars = ring + S * SS;
  auto full = [&](int i) { return bars + 8 * i; };
  auto empty = [&](int i) { return bars + 8 * (S + i); };
  auto dfull = [&](int j) { return bars + 8 * (2 * S + j); };
  auto dempty = [&](int j) { return bars + 8 * (2 * S + 2 + j); };
  const uint32_t yfull = bars + 8 * (2 * S + 4);
  const uint32_t tslot = yfull + 8;

  const int n_tiles = (a.V + kTile - 1) / kTile;
  const int tiles = my_tile_count(n_tiles);
  const int total = tiles * kcs;
  auto src_of = [&](int c) {
    const int tile = blockIdx.x + (c / kcs) * gridDim.x;
    return a.wb + ((size_t)tile * kcs + (c % kcs)) * SB;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(dfull(j), 1);
      mbar_init(dempty(j), kBfWorkers / 32);
    }
    mbar_init(yfull, 1);
    mbar_fence_init();
    for (int j = 0; j < S && j * U < total; ++j) {
      // streamed Y: one expect for the stage's table and Y bytes; Y is copied after griddepcontrol.wait
      mbar_expect_tx(full(j), U * SB + (kStreamY ? U * kYChunk : 0));
      bulk_g2s(ring + j * SS + TOFF, src_of(j * U), U * SB, full(j));
    }
  }
  if (warp == 1) tmem_alloc<64>(tslot);
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = lds32(tslot);
  pdl_wait();
  const int T = a.T_const > 0 ? a.T_const : a.sp->T;

  if (warp == 0) {
    if (lane == 0) {
      if (kStreamY) {
        for (int j = 0; j < S && j * U < total; ++j)
          bulk_g2s(ring + j * SS, a.ylm + (size_t)((j * U) % kcs) * kYChunk, U * kYChunk, full(j));
        mbar_arrive(yfull);
      } else if (a.ylm) {
        load_ylm(a, ybuf, yfull);
      }
      int st = 0;
      uint32_t par = 0;
      for (int j = S; j * U < total; ++j) {
        if (!mbar_wait_bounded(empty(st), par, a.err)) break;
        mbar_expect_tx(full(st), U * SB + (kStreamY ? U * kYChunk : 0));
        bulk_g2s(ring + st * SS + TOFF, src_of(j * U), U * SB, full(st));
        if (kStreamY) bulk_g2s(ring + st * SS, a.ylm + (size_t)((j * U) % kcs) * kYChunk, U * kYChunk, full(st));
        if (++st == S) { st = 0; par ^= 1; }
      }
    }
  } else if (warp == 1) {
    // the whole warp runs the issue loop (warp-uniform state); one elected lane issues
    if (mbar_wait_warp(yfull, 0, a.err)) {
      // counters instead of divisions
      int st = 0, uo = 0, kc = 0, ti = 0;
      uint32_t fpar = 0;
      for (int c = 0; c < total; ++c) {
        const int db = ti & 1;
        if (kc == 0 && ti >= 2 && !mbar_wait_warp(dempty(db), ((ti >> 1) - 1) & 1, a.err)) break;
        if (uo == 0 && !mbar_wait_warp(full(st), fpar, a.err)) break;
        tc_fence_after();
        const uint64_t ad = umma_desc_sw128(ring + st * SS + TOFF + uo * SB);
        const uint64_t bd = umma_desc_sw128(kStreamY ? ring + st * SS + uo * kYChunk : ybuf + kc * kYChunk);
#pragma unroll
        for (int kk = 0; kk < kChunk / 16; ++kk)
          umma_ss_elect(tmem + 32 * db, ad + 2 * kk, bd + 2 * kk, IDESC, (kc | kk) ? 1u : 0u);
        if (uo == U - 1) umma_commit_elect(empty(st));
        if (kc == kcs - 1) umma_commit_elect(dfull(db));
        if (++uo == U) { uo = 0; if (++st == S) { st = 0; fpar ^= 1; } }
        if (++kc == kcs) { kc = 0; ++ti; }
      }
    }
  }

  const int quad = warp & 3;
  const int r = 32 * quad + lane;
  float bv[16];
  int bi[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) { bv[i] = -INFINITY; bi[i] = 0x7fffffff; }
  if (warp >= 2) {
    if (!kStreamY && !a.ylm) {
      stage_y<false>(a, ybuf, T, (int)threadIdx.x - kBase, kBfWorkers);
      fence_proxy_async();
      named_sync(1, kBfWorkers);
      if (threadIdx.x == kBase) mbar_arrive(yfull);
    }
    const uint32_t lane_base = tmem + ((uint32_t)(32 * quad) << 16);
    for (int ti = 0; ti < tiles; ++ti) {
      const int db = ti & 1;
      if (!mbar_wait_bounded(dfull(db), (ti >> 1) & 1, a.err)) break;
      tc_fence_after();
      float d0[16], d1[16];
      tmem_ld16(lane_base + 32 * db, d0);        // slots 0..7 hi, lo
      tmem_ld16(lane_base + 32 * db + 16, d1);   // slots 8..15 hi, lo
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dempty(db));
      const int v = (blockIdx.x + ti * gridDim.x) * kTile + r;
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const float val = t < 8 ? d0[t] + d0[8 + t] : d1[t - 8] + d1[t];
        if (v < a.V && t < T) {
          if (a.logits) a.logits[(size_t)t * a.V + v] = val;
          if (better(val, v, bv[t], bi[t])) { bv[t] = val; bi[t] = v; }
        }
      }
    }
  }
  finish_argmax<16>(a, T, warp >= 2, 0, bv, bi);
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_free<64>(tmem);
  }
}

// Scratch of the lm_head entry point that allocates nothing: the completion
// ticket (first 256 bytes; it must read zero before a launch, and the last CTA
// of every launch puts it back to zero) followed by the per-CTA partial bests
// (grid x kMaxT float2).  Static device memory of this library: every device
// that loads it holds one copy until the process exits, shared by all calls.
constexpr size_t kStaticLmScratchBytes = 64 * 1024;
static __device__ __align__(256) unsigned char g_lm_scratch[kStaticLmScratchBytes];

int lmhead_static_max_grid() { return (int)((kStaticLmScratchBytes - 256) / (kMaxT * sizeof(float2))); }

cudaError_t lmhead_static_scratch(int grid, float2 **part, int32_t **ticket, cudaStream_t st) {
  if (grid < 1 || grid > lmhead_static_max_grid()) return cudaErrorInvalidValue;
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static unsigned char *addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned char *p = nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    p = addr[dev];
    if (!p) {
      // first call on this device (current): the symbol's device address, then a zero ticket
      e = cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_lm_scratch);
      if (e != cudaSuccess) return e;
      e = cudaMemsetAsync(p, 0, 256, st);
      if (e != cudaSuccess) return e;
      addr[dev] = p;
    }
  }
  *ticket = reinterpret_cast<int32_t *>(p);
  *part = reinterpret_cast<float2 *>(p + 256);
  return cudaSuccess;
}

int lmhead_grid(const LmArgs &a, int n_sm) {
  const int n_tiles = (a.V + kTile - 1) / kTile;
  return n_tiles < n_sm ? n_tiles : n_sm;
}

cudaError_t launch_lmhead(const LmArgs &a, int grid, cudaStream_t st, bool pdl) {
  const bool q8 = a.q8 != nullptr;
  const int kcs = a.H / kChunk;
  const size_t bars = 8 * (2 * 4 + 2 * 6 + 2) + 16;
  const size_t budget = 227 * 1024 - 2048;   // leaves room for the static shared arrays
  int U, S;
  size_t smem;
  const bool stream = a.ylm != nullptr;
  if (stream) {
    // several chunks (and their Y) per stage when the tile's chunk count allows
    U = q8 ? (kcs % 4 == 0 ? 4 : kcs % 2 == 0 ? 2 : 1) : (kcs % 2 == 0 ? 2 : 1);
    const size_t ss = q8 ? (size_t)q8_stage_bytes(true, U) : (size_t)bf_stage_bytes(true, U);
    S = (int)((budget - 1024 - bars) / (ss + 16));
    if (S > 8) S = 8;
    if (S < 2) return cudaErrorInvalidValue;
    smem = 1024 + bars + (size_t)S * (ss + 16);
  } else {
    const size_t ybytes = (size_t)kcs * kYChunk;
    const size_t fixed = 1024 + ybytes + bars;
    // two chunks per bulk copy when a tile's chunk count is even and three such stages fit
    U = kcs % 2 == 0 ? 2 : 1;
    size_t sb = q8 ? (size_t)q8_stage_bytes(false, U) : (size_t)U * kBfStage;
    if (U == 2 && fixed + 3 * (sb + 16) > budget) {
      U = 1;
      sb = q8 ? (size_t)q8_stage_bytes(false, 1) : (size_t)kBfStage;
    }
    if (fixed + 2 * (sb + 16) > budget) return cudaErrorInvalidValue;
    S = (int)((budget - fixed) / (sb + 16));
    if (S > 12) S = 12;
    smem = fixed + (size_t)S * (sb + 16);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(q8 ? kQ8Threads : kBase + kBfWorkers, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  auto go = [&](auto kern) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, kern, a, S, U);
  };
  // Q8_0: chunks move in pairs when a tile's chunk count is even; two MMA issuers when
  // Y streams in 4-chunk units (each unit = one pair per issuer) and a tile's pairs
  // split evenly between them
  const int G = kcs % 2 == 0 ? 2 : 1;
  const int NI = q8 && stream && U == 4 && (kcs / G) % 2 == 0 ? 2 : 1;
  auto goq = [&](auto kern) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, kern, a, S, U, NI, G);
  };
  if (q8) return stream ? goq(fm_lmhead_q8_kernel<true>) : goq(fm_lmhead_q8_kernel<false>);
  return stream ? go(fm_lmhead_bf16_kernel<true>) : go(fm_lmhead_bf16_kernel<false>);
}

}  // namespace fm
