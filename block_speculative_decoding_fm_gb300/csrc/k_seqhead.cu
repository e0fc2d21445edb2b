// k_seqhead.cu -- the sequential logit head and the confidence head of the
// DFlash drafter (module-dflash.ts: ``#markov``, ``#rnn``, ``#confidence`` and
// the greedy branch of ``forwardRows``).  Position k of the block is drafted
// after position k - 1: with prev the anchor (k = 0) or the token of k - 1,
//   e1 = markov.w1[prev];  Markov: bias = e1 markov.w2;
//   RNN: s_k = tanh(s_{k-1} rnn.wH + e1 + rnn.bH), bias = s_k rnn.wO;
//   token_k = argmax(base logits_k + bias);
//   conf_k = sigmoid([out_norm(block row k), e1] conf.w + conf.b);
// and confidence pruning ends the block at the first k >= 1 whose conf_k is
// below the position's threshold (later positions are not drafted).
// One launch per position streams the [r][V] bias matrix once (bf16, 16-byte
// loads) fused with the add and a two-pass argmax (per-CTA bests, the last CTA
// reduces, ties to the lower index); the last CTA then forms the confidence and
// the pruning decision.  A CTA owns 512 vocabulary columns and splits the rank
// over four row groups of 64 threads, each thread keeping eight loads in
// flight, so an SM holds enough bytes in flight to stream at the HBM rate.
#include "dev_common.cuh"
#include "fm_internal.h"

namespace fm {

namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 8;                 // vocabulary columns per thread (one 16-byte load)
constexpr int kGroups = 4;                    // rank row groups per CTA
constexpr int kColThreads = kThreads / kGroups;
constexpr int kCols = kColThreads * kPerThread;   // vocabulary columns per CTA
constexpr int kInflight = 8;                  // loads in flight per thread
constexpr int kMaxRank = 512;

__device__ __forceinline__ void best_reduce_block(float &bv, int &bi, float *sv, int *si) {
  // warp, then the block's warps, ties to the lower index
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) { sv[w] = bv; si[w] = bi; }
  __syncthreads();
  if (w == 0) {
    bv = lane < kThreads / 32 ? sv[lane] : -INFINITY;
    bi = lane < kThreads / 32 ? si[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
  }
}

__global__ void __launch_bounds__(kThreads) seq_bias_argmax_kernel(const __grid_constant__ SeqArgs a) {
  __shared__ float e[kMaxRank];
  __shared__ float red[kGroups][kCols];
  __shared__ float sv[kThreads / 32];
  __shared__ int si[kThreads / 32];
  __shared__ int last;
  if (a.flags[0]) return;   // pruning ended the block at an earlier position
  const int k = a.k;
  const int prev = k == 0 ? a.sp->anchor : a.sp->tokens[k - 1];
  for (int i = threadIdx.x; i < a.r; i += kThreads)
    e[i] = a.state ? a.state[i] : __bfloat162float(a.w1[(size_t)prev * a.r + i]);
  __syncthreads();
  // partial sums of row group g over its rows g, g + kGroups, ...
  const int g = threadIdx.x / kColThreads, ct = threadIdx.x % kColThreads;
  const int v0 = blockIdx.x * kCols + ct * kPerThread;
  float acc[kPerThread];
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) acc[j] = 0.f;
  if (v0 < a.V) {
    const __nv_bfloat16 *col = a.W + v0;
    for (int i0 = g; i0 < a.r; i0 += kGroups * kInflight) {
      uint4 u[kInflight];
#pragma unroll
      for (int x = 0; x < kInflight; ++x) {
        const int i = i0 + x * kGroups;
        u[x] = i < a.r ? __ldg(reinterpret_cast<const uint4 *>(col + (size_t)i * a.V)) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int x = 0; x < kInflight; ++x) {
        const int i = i0 + x * kGroups;
        const float ex = i < a.r ? e[i] : 0.f;
        const uint32_t w4[4] = {u[x].x, u[x].y, u[x].z, u[x].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[2 * j] += ex * __uint_as_float(w4[j] << 16);
          acc[2 * j + 1] += ex * __uint_as_float(w4[j] & 0xffff0000u);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) red[g][ct * kPerThread + j] = acc[j];
  __syncthreads();
  // each thread finishes two columns: the row groups in order, then the base logit
  float bv = -INFINITY;
  int bi = 0x7fffffff;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int c = 2 * threadIdx.x + q;
    const int v = blockIdx.x * kCols + c;
    if (v < a.V) {
      float b = red[0][c];
#pragma unroll
      for (int gg = 1; gg < kGroups; ++gg) b += red[gg][c];
      const float sc = __ldcg(a.base + (size_t)k * a.V + v) + b;
      if (better(sc, v, bv, bi)) { bv = sc; bi = v; }
    }
  }
  best_reduce_block(bv, bi, sv, si);
  if (threadIdx.x == 0) {
    a.part[blockIdx.x] = make_float2(bv, __int_as_float(bi));
    __threadfence();
    const int old = atomicAdd(a.ticket, 1);
    last = old == (int)gridDim.x - 1;
    if (last) atomicExch(a.ticket, 0);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  // the last CTA: the position's token over every CTA's best, in CTA order
  bv = -INFINITY;
  bi = 0x7fffffff;
  for (int b = threadIdx.x; b < (int)gridDim.x; b += kThreads) {
    const float2 p = __ldcg(a.part + b);
    if (better(p.x, __float_as_int(p.y), bv, bi)) { bv = p.x; bi = __float_as_int(p.y); }
  }
  best_reduce_block(bv, bi, sv, si);
  __syncthreads();
  if (threadIdx.x == 0) {
    a.sp->tokens[k] = bi;
    si[0] = bi;
  }
  if (!a.conf_w) {
    if (threadIdx.x == 0 && k == a.T - 1) {
      a.flags[1] = a.T;
      if (a.sp->length) *a.sp->length = a.T;
    }
    return;
  }
  // confidence of position k: sigmoid([out_norm(X_k), e1] conf.w + conf.b), with
  // e1 = markov.w1[prev] (both heads)
  float ss = 0.f;
  for (int i = threadIdx.x; i < a.d; i += kThreads) {
    const float x = a.X[(size_t)k * a.d + i];
    ss += x * x;
  }
  ss = warp_sum(ss);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sv[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) tot += sv[w];
  const float rs = rsqrtf(tot / (float)a.d + a.eps);
  float z = 0.f;
  for (int i = threadIdx.x; i < a.d; i += kThreads)
    z += a.X[(size_t)k * a.d + i] * rs * __bfloat162float(a.out_norm[i]) * __bfloat162float(a.conf_w[i]);
  for (int i = threadIdx.x; i < a.r; i += kThreads)
    z += __bfloat162float(a.w1[(size_t)prev * a.r + i]) * __bfloat162float(a.conf_w[a.d + i]);
  z = warp_sum(z);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sv[threadIdx.x >> 5] = z;
  __syncthreads();
  if (threadIdx.x == 0) {
    float zz = __bfloat162float(a.conf_b[0]);
    for (int w = 0; w < kThreads / 32; ++w) zz += sv[w];
    const float c = 1.f / (1.f + expf(-zz));
    if (a.sp->conf) a.sp->conf[k] = c;
    const float thr = a.sp->thr[k];
    if (k > 0 && thr == thr && c < thr) {   // thr == thr: not NaN (a threshold is set)
      a.flags[0] = 1;
      a.flags[1] = k;
    } else if (k == a.T - 1) {
      a.flags[1] = a.T;
    }
    if (a.sp->length && (a.flags[0] || k == a.T - 1)) *a.sp->length = a.flags[1];
  }
}

// s_k = tanh(s_{k-1} wH + w1[prev] + bH), one CTA: r / 8 threads cover a row
// of wH with 16-byte loads (eight columns each) and the CTA's 256 / (r / 8)
// row groups split the rows; the groups' sums meet in shared memory in order.
__global__ void __launch_bounds__(kThreads) rnn_step_kernel(const __grid_constant__ RnnArgs a) {
  __shared__ float red[kThreads * 8];      // [row group][r]: n_grp * r <= 8 * 256
  if (a.flags[0]) return;
  const int r = a.r;
  const int tpr = r / 8;                  // threads per row
  const int n_grp = kThreads / tpr;       // row groups
  const int t = threadIdx.x;
  const int grp = t / tpr, c8 = (t % tpr) * 8;
  const int prev = a.k == 0 ? a.sp->anchor : a.sp->tokens[a.k - 1];
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.f;
  if (a.k > 0 && grp < n_grp) {
    for (int i0 = grp; i0 < r; i0 += n_grp * kInflight) {
      uint4 u[kInflight];
      float si[kInflight];
#pragma unroll
      for (int x = 0; x < kInflight; ++x) {
        const int i = i0 + x * n_grp;
        u[x] = i < r ? __ldg(reinterpret_cast<const uint4 *>(a.wH + (size_t)i * r + c8)) : make_uint4(0u, 0u, 0u, 0u);
        si[x] = i < r ? __ldcg(a.s_in + i) : 0.f;
      }
#pragma unroll
      for (int x = 0; x < kInflight; ++x) {
        const uint32_t w4[4] = {u[x].x, u[x].y, u[x].z, u[x].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[2 * j] += si[x] * __uint_as_float(w4[j] << 16);
          acc[2 * j + 1] += si[x] * __uint_as_float(w4[j] & 0xffff0000u);
        }
      }
    }
  }
  if (grp < n_grp) {
#pragma unroll
    for (int j = 0; j < 8; ++j) red[grp * r + c8 + j] = acc[j];
  }
  __syncthreads();
  for (int j = t; j < r; j += kThreads) {
    float v = __bfloat162float(a.w1[(size_t)prev * r + j]) + __bfloat162float(a.bH[j]);
    for (int q = 0; q < n_grp; ++q) v += red[q * r + j];
    a.s_out[j] = tanhf(v);
  }
}

__global__ void seq_init_kernel(int32_t *flags, int32_t T) {
  flags[0] = 0;
  flags[1] = T;
}

}  // namespace

int seq_grid(int V) { return (V + kCols - 1) / kCols; }

cudaError_t launch_seq_bias_argmax(const SeqArgs &a, cudaStream_t s) {
  if (a.r > kMaxRank || a.V % kPerThread) return cudaErrorInvalidValue;
  seq_bias_argmax_kernel<<<seq_grid(a.V), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rnn_step(const RnnArgs &a, cudaStream_t s) {
  // whole 16-byte row pieces, and at least one row group per CTA
  if (a.r < 8 || a.r % 8 || a.r / 8 > kThreads || a.r > kMaxRank) return cudaErrorInvalidValue;
  rnn_step_kernel<<<1, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_seq_init(int32_t *flags, int32_t T, cudaStream_t s) {
  seq_init_kernel<<<1, 1, 0, s>>>(flags, T);
  return cudaGetLastError();
}

}  // namespace fm
