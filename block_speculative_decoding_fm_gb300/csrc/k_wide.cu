// k_wide.cu -- the small kernels of a batched draft, where the 16 slot rows of
// every sequence in the call (up to 512 rows) go through the tensor-core GEMM
// together (flashmap_drafter.js ``draft`` for many anchors at once; the page's
// ``runGemm`` takes over from the skinny products above 17 rows):
//   * wide_prep       every slot row starts at h0 (``init``: the jump from zero
//                     noise), and each sequence's anchor row is gathered from
//                     the f16 token table (the anchor_proj operand);
//   * wide_lnmod      adds the gated branch of the previous product to the
//                     residual stream (``gateAdd``) when that product wrote it
//                     apart (its tensor reduce-add copies otherwise added it
//                     already), then adaLN LayerNorm-modulate
//                     of each row (``lnMod``): two-pass mean / population
//                     variance, * (1 + scale) + shift, f16 out (the next
//                     product's operand);
//   * wide_self_attn  the block's self-attention per sequence and head (no
//                     mask, ``attn`` over the 16 slots), f16 out;
//   * wide_argmax     the per-row reduction of the lm_head's per-tile bests
//                     (lowest index on ties);
//   * q8_to_f16       the Q8_0 token table as f16(d * q) rows, each weight
//                     rounded once (the batched lm_head's operand).
#include "dev_common.cuh"
#include "fm_internal.h"

namespace fm {

namespace {

__global__ void wide_prep_kernel(const float *__restrict__ h0, int D, int T, float *__restrict__ X,
                                 const WideParams *__restrict__ wp, const __half *__restrict__ table, int H,
                                 __half *__restrict__ anc) {
  pdl_trigger();
  pdl_wait();
  const int n = wp->n;
  const int d4 = D / 4, h8 = H / 8;
  const size_t nx = (size_t)T * d4;
  const size_t total = nx + (size_t)n * h8;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    if (i < nx) {
      reinterpret_cast<float4 *>(X)[i] = reinterpret_cast<const float4 *>(h0)[i % d4];
    } else {
      const size_t j = i - nx;
      const int r = (int)(j / h8), c = (int)(j % h8);
      reinterpret_cast<uint4 *>(anc + (size_t)r * H)[c] =
          reinterpret_cast<const uint4 *>(table + (size_t)wp->anchor[r] * H)[c];
    }
  }
}

// Sum over the CTA (at most 8 warps) in warp order, the same value in every thread; slot k of red
// is this reduction's own, so two reductions need one barrier each.
__device__ __forceinline__ float block_sum(float v, float (*red)[8], int k) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) red[k][warp] = v;
  __syncthreads();
  float s = 0.f;
  for (int i = 0; i < nw; ++i) s += red[k][i];
  return s;
}

// one CTA per row of D columns (a multiple of 256, at most 4096): float4 i of the row goes to thread
// i % blockDim.x, at most 4 per thread.  With R: the residual stream first takes the gated branch the
// previous product wrote (X += R, stored back).  A thread's modulation columns (weights, not written by
// earlier kernels) are loaded before griddepcontrol.wait.
template <int Q>   // float4 per thread at most (2 for rows up to 2048 columns, else 4): the register budget
__global__ void __launch_bounds__(256) wide_lnmod_kernel(float *__restrict__ X, const float *__restrict__ R, int D,
                                                          int T, const float *__restrict__ scale,
                                                          const float *__restrict__ shift, float eps,
                                                          __half *__restrict__ out) {
  __shared__ float red[2][8];
  pdl_trigger();
  const int t = threadIdx.x, nt = blockDim.x, n4 = D / 4, row = blockIdx.x;
  float4 sc[Q], sh[Q], v[Q];
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    if (t + q * nt < n4) {
      sc[q] = reinterpret_cast<const float4 *>(scale)[t + q * nt];
      sh[q] = reinterpret_cast<const float4 *>(shift)[t + q * nt];
    }
  }
  pdl_wait();
  if (row >= T) return;
  float4 *x = reinterpret_cast<float4 *>(X + (size_t)row * D);
  const float4 *r = R ? reinterpret_cast<const float4 *>(R + (size_t)row * D) : nullptr;
  float4 g[Q];
#pragma unroll
  for (int q = 0; q < Q; ++q) {   // every load of the row before any store
    if (t + q * nt < n4) {
      v[q] = x[t + q * nt];
      if (r) g[q] = r[t + q * nt];
    }
  }
  float s = 0.f;
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    if (t + q * nt < n4) {
      if (r) {
        v[q].x += g[q].x;
        v[q].y += g[q].y;
        v[q].z += g[q].z;
        v[q].w += g[q].w;
        x[t + q * nt] = v[q];
      }
      s += (v[q].x + v[q].y) + (v[q].z + v[q].w);
    }
  }
  const float mean = block_sum(s, red, 0) / (float)D;
  float m2 = 0.f;
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    if (t + q * nt < n4) {
      const float a = v[q].x - mean, b = v[q].y - mean, c = v[q].z - mean, d = v[q].w - mean;
      m2 += (a * a + b * b) + (c * c + d * d);
    }
  }
  const float rstd = rsqrtf(block_sum(m2, red, 1) / (float)D + eps);
  __half *o = out + (size_t)row * D;
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    if (t + q * nt < n4) {
      const int i4 = t + q * nt;
      const __half2 h01 = __floats2half2_rn((v[q].x - mean) * rstd * (1.f + sc[q].x) + sh[q].x,
                                            (v[q].y - mean) * rstd * (1.f + sc[q].y) + sh[q].y);
      const __half2 h23 = __floats2half2_rn((v[q].z - mean) * rstd * (1.f + sc[q].z) + sh[q].z,
                                            (v[q].w - mean) * rstd * (1.f + sc[q].w) + sh[q].w);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t *>(&h01);
      pk.y = *reinterpret_cast<const uint32_t *>(&h23);
      *reinterpret_cast<uint2 *>(o + 4 * i4) = pk;
    }
  }
}

// one CTA (128 threads) per (sequence, head): O = softmax(q k^T / sqrt(128)) v over the B <= 16 slots.
// Scores: thread i takes the pairs (n, j) = (i / 16, i % 16) and (i / 16 + 8, i % 16) over the 128 dims
// with four partial sums; softmax: a half-warp per row (lane j holds score j), maximum and sum by
// shuffles inside the half; output: a warp per four rows, a lane per four dims.
__global__ void wide_self_attn_kernel(const float *__restrict__ qkv, int D, int B, __half *__restrict__ out) {
  constexpr int HD = 128, KS = HD + 4;   // padded q / k rows
  __shared__ __align__(16) float q[16][KS], k[16][KS], v[16][HD];
  __shared__ float p[16][17];
  pdl_trigger();
  pdl_wait();
  const int seq = blockIdx.x, head = blockIdx.y, t = threadIdx.x;
  const int r0 = seq * B;
  // 16 rows x 32 float4 per operand over 128 threads: every load issued before the shared-memory stores
  float4 lq[4], lk[4], lv[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = t + 128 * j, n = i / (HD / 4), c = (i % (HD / 4)) * 4;
    if (n < B) {
      const float *row = qkv + (size_t)(r0 + n) * 3 * D + head * HD + c;
      lq[j] = *reinterpret_cast<const float4 *>(row);
      lk[j] = *reinterpret_cast<const float4 *>(row + D);
      lv[j] = *reinterpret_cast<const float4 *>(row + 2 * D);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = t + 128 * j, n = i / (HD / 4), c = (i % (HD / 4)) * 4;
    if (n < B) {
      *reinterpret_cast<float4 *>(&q[n][c]) = lq[j];
      *reinterpret_cast<float4 *>(&k[n][c]) = lk[j];
      *reinterpret_cast<float4 *>(&v[n][c]) = lv[j];
    }
  }
  __syncthreads();
  const float scale = 0.08838834764831845f;   // 1 / sqrt(128)
  {
    const int j = t & 15;
#pragma unroll
    for (int y = 0; y < 2; ++y) {
      const int n = (t >> 4) + 8 * y;
      if (n < B && j < B) {
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll 8
        for (int d = 0; d < HD; d += 4) {
          const float4 a = *reinterpret_cast<const float4 *>(&q[n][d]);
          const float4 b = *reinterpret_cast<const float4 *>(&k[j][d]);
          s0 += a.x * b.x; s1 += a.y * b.y; s2 += a.z * b.z; s3 += a.w * b.w;
        }
        p[n][j] = ((s0 + s1) + (s2 + s3)) * scale;
      }
    }
  }
  __syncthreads();
  {
    const int lane = t & 31, j = lane & 15;
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      const int n = 2 * (t >> 5) + (lane >> 4) + 8 * pass;
      const bool on = n < B && j < B;
      const float sc = on ? p[n][j] : -INFINITY;
      float m = sc;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const float e = on ? expf(sc - m) : 0.f;
      float l = e;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      if (on) p[n][j] = e / l;
    }
  }
  __syncthreads();
  // warp w forms rows 4w .. 4w + 3, lane l dims 4l .. 4l + 3: one float4 of v and four probabilities per key
  const int lane = t & 31, n0 = 4 * (t >> 5);
  float o[4][4] = {};
  for (int j = 0; j < B; ++j) {
    const float4 vj = *reinterpret_cast<const float4 *>(&v[j][4 * lane]);
#pragma unroll
    for (int y = 0; y < 4; ++y) {
      const float pj = p[n0 + y][j];
      o[y][0] += pj * vj.x; o[y][1] += pj * vj.y; o[y][2] += pj * vj.z; o[y][3] += pj * vj.w;
    }
  }
#pragma unroll
  for (int y = 0; y < 4; ++y) {
    if (n0 + y < B) {
      const __half2 a = __floats2half2_rn(o[y][0], o[y][1]), b = __floats2half2_rn(o[y][2], o[y][3]);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t *>(&a);
      pk.y = *reinterpret_cast<const uint32_t *>(&b);
      *reinterpret_cast<uint2 *>(out + (size_t)(r0 + n0 + y) * D + head * HD + 4 * lane) = pk;
    }
  }
}

// one warp per row: the best (value, index) over the row's column-block bests, in block order
__global__ void wide_argmax_kernel(const float2 *__restrict__ part, int n_blocks, int T, const WideParams *wp) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + warp;
  if (row >= T) return;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int j = lane; j < n_blocks; j += 32) {
    const float2 e = part[(size_t)row * n_blocks + j];
    const int ei = __float_as_int(e.y);
    if (better(e.x, ei, bv, bi)) {
      bv = e.x;
      bi = ei;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
  if (lane == 0) wp->tokens[row] = bi;
}

// rows [0, V) from the Q8_0 blocks (f16 d, then 32 int8 q); rows [V, Vpad) zero
__global__ void q8_to_f16_kernel(const uint8_t *__restrict__ raw, int V, int H, int Vpad, __half *__restrict__ out) {
  const int nb = H / 32;
  const size_t total = (size_t)Vpad * nb;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / nb;
    __half *o = out + i * 32;
    if ((int)r >= V) {
      for (int e = 0; e < 32; ++e) o[e] = __float2half_rn(0.f);
      continue;
    }
    const uint8_t *blk = raw + i * 34;
    const float d = __half2float(__ushort_as_half((unsigned short)(blk[0] | (blk[1] << 8))));
    for (int e = 0; e < 32; ++e) o[e] = __float2half_rn(d * (float)(int8_t)blk[2 + e]);
  }
}

__global__ void f16_copy_pad_kernel(const __nv_bfloat16 *__restrict__ in, int V, int H, int Vpad,
                                    __half *__restrict__ out) {
  const size_t total = (size_t)Vpad * H;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x)
    out[i] = (int)(i / H) < V ? __float2half_rn(__bfloat162float(in[i])) : __float2half_rn(0.f);
}

cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, void **args, cudaStream_t s, size_t smem = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

cudaError_t launch_wide_prep(const float *h0, int D, int T, float *X, const WideParams *wp, int n_max,
                             const __half *table, int H, __half *anc, int n_sm, cudaStream_t s) {
  if (D % 4 || H % 8) return cudaErrorInvalidValue;
  const size_t total = (size_t)T * (D / 4) + (size_t)n_max * (H / 8);
  int grid = (int)((total + 255) / 256);
  if (grid > 4 * n_sm) grid = 4 * n_sm;
  void *args[] = {(void *)&h0, (void *)&D, (void *)&T, (void *)&X, (void *)&wp, (void *)&table, (void *)&H, (void *)&anc};
  return launch_pdl((const void *)wide_prep_kernel, dim3(grid), dim3(256), args, s);
}

cudaError_t launch_wide_lnmod(float *X, const float *R, int D, int T, const float *scale, const float *shift, float eps,
                              __half *out, cudaStream_t s) {
  if (D % 256 || D > 4096 || T < 1) return cudaErrorInvalidValue;
  void *args[] = {(void *)&X, (void *)&R, (void *)&D, (void *)&T, (void *)&scale, (void *)&shift, (void *)&eps,
                  (void *)&out};
  // D / 8 threads (two float4 each, whole warps) up to 256; wider rows give a thread up to four
  const int nt = D / 8 < 256 ? D / 8 : 256;
  return launch_pdl(D <= 2048 ? (const void *)wide_lnmod_kernel<2> : (const void *)wide_lnmod_kernel<4>, dim3(T),
                    dim3(nt), args, s, 0);
}

cudaError_t launch_wide_self_attn(const float *qkv, int D, int B, int n_seqs, int n_heads, __half *out, cudaStream_t s) {
  if (B < 1 || B > 16) return cudaErrorInvalidValue;
  void *args[] = {(void *)&qkv, (void *)&D, (void *)&B, (void *)&out};
  return launch_pdl((const void *)wide_self_attn_kernel, dim3(n_seqs, n_heads), dim3(128), args, s);
}

cudaError_t launch_wide_argmax(const float2 *part, int n_blocks, int T, const WideParams *wp, cudaStream_t s) {
  void *args[] = {(void *)&part, (void *)&n_blocks, (void *)&T, (void *)&wp};
  return launch_pdl((const void *)wide_argmax_kernel, dim3((T + 7) / 8), dim3(256), args, s);
}

cudaError_t launch_q8_to_f16(const uint8_t *raw, int V, int H, int Vpad, __half *out, cudaStream_t s) {
  if (H % 32) return cudaErrorInvalidValue;
  const size_t total = (size_t)Vpad * (H / 32);
  const unsigned grid = (unsigned)((total + 255) / 256 < 65536 ? (total + 255) / 256 : 65536);
  q8_to_f16_kernel<<<grid, 256, 0, s>>>(raw, V, H, Vpad, out);
  return cudaGetLastError();
}

cudaError_t launch_bf16_to_f16_pad(const __nv_bfloat16 *in, int V, int H, int Vpad, __half *out, cudaStream_t s) {
  const size_t total = (size_t)Vpad * H;
  const unsigned grid = (unsigned)((total + 255) / 256 < 65536 ? (total + 255) / 256 : 65536);
  f16_copy_pad_kernel<<<grid, 256, 0, s>>>(in, V, H, Vpad, out);
  return cudaGetLastError();
}

}  // namespace fm
