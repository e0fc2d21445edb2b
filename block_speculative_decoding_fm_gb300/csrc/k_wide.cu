// k_wide.cu -- the small kernels of a batched draft, where the 16 slot rows of
// every sequence in the call (up to 512 rows) go through the tensor-core GEMM
// together (flashmap_drafter.js ``draft`` for many anchors at once; the page's
// ``runGemm`` takes over from the skinny products above 17 rows):
//   * wide_prep       every slot row starts at h0 (``init``: the jump from zero
//                     noise), and each sequence's anchor row is gathered from
//                     the f16 token table (the anchor_proj operand);
//   * wide_lnmod      adds the gated branch of the previous product to the
//                     residual stream (``gateAdd``), then adaLN LayerNorm-modulate
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

// one warp per row; D <= 4096, a multiple of 128.  With R: the residual stream
// first takes the gated branch the previous product wrote (X += R, stored back).
// The modulation rows (weights, not written by earlier kernels) are staged in
// shared memory before griddepcontrol.wait.
__global__ void wide_lnmod_kernel(float *__restrict__ X, const float *__restrict__ R, int D, int T,
                                  const float *__restrict__ scale, const float *__restrict__ shift, float eps,
                                  __half *__restrict__ out) {
  extern __shared__ float4 mods[];   // [D / 4] scale, then [D / 4] shift
  pdl_trigger();
  {
    // all of a thread's loads first, then its shared-memory stores (D / 4 <= 1024 float4 per row over 128 threads)
    float4 sv[8], hv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = threadIdx.x + j * blockDim.x;
      if (i < D / 4) {
        sv[j] = reinterpret_cast<const float4 *>(scale)[i];
        hv[j] = reinterpret_cast<const float4 *>(shift)[i];
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = threadIdx.x + j * blockDim.x;
      if (i < D / 4) {
        mods[i] = sv[j];
        mods[D / 4 + i] = hv[j];
      }
    }
  }
  __syncthreads();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + warp;
  if (row >= T) return;
  const int per = D / 128;   // float4 per lane
  float4 *x = reinterpret_cast<float4 *>(X + (size_t)row * D);
  const float4 *r = R ? reinterpret_cast<const float4 *>(R + (size_t)row * D) : nullptr;
  float4 v[32];
  float s = 0.f;
  // every load of the row is issued before any store
#pragma unroll
  for (int u = 0; u < 32; ++u) {
    if (u < per) {
      v[u] = x[u * 32 + lane];
      if (r) {
        const float4 g = r[u * 32 + lane];
        v[u].x += g.x;
        v[u].y += g.y;
        v[u].z += g.z;
        v[u].w += g.w;
      }
      s += (v[u].x + v[u].y) + (v[u].z + v[u].w);
    }
  }
  if (r) {
#pragma unroll
    for (int u = 0; u < 32; ++u)
      if (u < per) x[u * 32 + lane] = v[u];
  }
  const float mean = warp_sum(s) / (float)D;
  float q = 0.f;
#pragma unroll
  for (int u = 0; u < 32; ++u) {
    if (u < per) {
      const float a = v[u].x - mean, b = v[u].y - mean, c = v[u].z - mean, d = v[u].w - mean;
      q += (a * a + b * b) + (c * c + d * d);
    }
  }
  const float rstd = rsqrtf(warp_sum(q) / (float)D + eps);
  __half *o = out + (size_t)row * D;
#pragma unroll
  for (int u = 0; u < 32; ++u) {
    if (u < per) {
      const int i4 = u * 32 + lane;
      const float4 sc = mods[i4];
      const float4 sh = mods[D / 4 + i4];
      const __half2 h01 = __floats2half2_rn((v[u].x - mean) * rstd * (1.f + sc.x) + sh.x,
                                            (v[u].y - mean) * rstd * (1.f + sc.y) + sh.y);
      const __half2 h23 = __floats2half2_rn((v[u].z - mean) * rstd * (1.f + sc.z) + sh.z,
                                            (v[u].w - mean) * rstd * (1.f + sc.w) + sh.w);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t *>(&h01);
      pk.y = *reinterpret_cast<const uint32_t *>(&h23);
      *reinterpret_cast<uint2 *>(o + 4 * i4) = pk;
    }
  }
}

// one CTA (128 threads) per (sequence, head): O = softmax(q k^T / sqrt(128)) v over the B slots
__global__ void wide_self_attn_kernel(const float *__restrict__ qkv, int D, int B, __half *__restrict__ out) {
  constexpr int HD = 128;
  __shared__ float q[16][HD], k[16][HD], v[16][HD];
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
  for (int pr = t; pr < B * B; pr += blockDim.x) {
    const int n = pr / B, j = pr % B;
    float s = 0.f;
#pragma unroll 8
    for (int d = 0; d < HD; ++d) s += q[n][(d + j) & (HD - 1)] * k[j][(d + j) & (HD - 1)];
    p[n][j] = s * scale;
  }
  __syncthreads();
  if (t < B) {
    float m = -INFINITY;
    for (int j = 0; j < B; ++j) m = fmaxf(m, p[t][j]);
    float l = 0.f;
    for (int j = 0; j < B; ++j) {
      const float e = expf(p[t][j] - m);
      p[t][j] = e;
      l += e;
    }
    const float inv = 1.f / l;
    for (int j = 0; j < B; ++j) p[t][j] *= inv;
  }
  __syncthreads();
  for (int n = 0; n < B; ++n) {
    float o = 0.f;
    for (int j = 0; j < B; ++j) o += p[n][j] * v[j][t];
    out[(size_t)(r0 + n) * D + head * HD + t] = __float2half_rn(o);
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
  if (D % 128 || D > 4096) return cudaErrorInvalidValue;
  void *args[] = {(void *)&X, (void *)&R, (void *)&D, (void *)&T, (void *)&scale, (void *)&shift, (void *)&eps,
                  (void *)&out};
  return launch_pdl((const void *)wide_lnmod_kernel, dim3((T + 3) / 4), dim3(128), args, s, (size_t)D * 8);
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
