// mtp.cu -- the MTP draft head (ternary_bonsai_2_mtp.js: the header's graph,
// MCFG, MTPHead.forward and its WGSL kernels, MTPRunner's draft loop).
//
// One Qwen-style decoder layer with Q8_0 weights over M <= 8 rows, chained in
// depth.  The Q8_0 products run on the lm_head kernel's tensor-core path
// (fm_lmhead_q8_kernel, f16 hi + lo activations, logits mode): its operand is
// the activations already split into the swizzled hi / lo rows, written by the
// kernel that produces them (the norms, the gated attention, the SiLU
// product).  Products with few 128-row tiles are split along K into slices
// (the table's tiles in slice order, each slice reading its own Y chunks), so
// that enough SMs stream the weights; the consumer of the output sums the
// slices.  The KV cache is f32, as the page keeps it.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/fm.h"
#include "dev_common.cuh"
#include "fm_internal.h"

namespace fm {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxRows = 8;

// the lm_head operand row of slot t (hi; lo is 8 rows further), 64-column chunks of kLmYChunk bytes
__device__ __forceinline__ void store_y8(uint8_t *ylm, int t, int col, const float (&v)[8]) {
  uint32_t hw[4], lw[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) split2_f16(v[2 * e], v[2 * e + 1], hw[e], lw[e]);
  uint8_t *cb = ylm + (size_t)(col >> 6) * kLmYChunk;
  const int r = lm_yrow(t);
  *reinterpret_cast<uint4 *>(cb + sw128(r, col & 63)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  *reinterpret_cast<uint4 *>(cb + sw128(r + 8, col & 63)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}
__device__ __forceinline__ void store_y1(uint8_t *ylm, int t, int col, float v) {
  const __half h = __float2half_rn(v);
  const __half l = __float2half_rn(v - __half2float(h));
  uint8_t *cb = ylm + (size_t)(col >> 6) * kLmYChunk;
  const int r = lm_yrow(t);
  *reinterpret_cast<__half *>(cb + sw128(r, col & 63)) = h;
  *reinterpret_cast<__half *>(cb + sw128(r + 8, col & 63)) = l;
}

__device__ __forceinline__ float block_sum(float v, float *red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < kThreads / 32; ++i) t += red[i];
  return t;
}

// Xc = [rms(E[x]; enorm) | rms(h; hnorm)] as the operand of eh_proj.  Block (2m + which).
__global__ void __launch_bounds__(kThreads) mtp_embed_norm_kernel(const __nv_bfloat16 *embd, const int32_t *tokens,
                                                                  int vocab, const float *hn, int ldh, const float *w_e,
                                                                  const float *w_h, int H, float eps, uint8_t *ylm,
                                                                  int32_t *err) {
  __shared__ float red[kThreads / 32];
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x >> 1, which = blockIdx.x & 1;
  int tok = which == 0 ? tokens[m] : 0;
  if (tok < 0 || tok >= vocab) {   // a token outside the table (a caller's, or a failed argmax): reported, row 0 read
    if (threadIdx.x == 0) atomicExch(err, 2);
    tok = 0;
  }
  float ss = 0.f;
  for (int c = threadIdx.x; c < H; c += kThreads) {
    const float x = which == 0 ? __bfloat162float(embd[(size_t)tok * H + c]) : __ldcg(hn + (size_t)m * ldh + c);
    ss += x * x;
  }
  const float r = rsqrtf(block_sum(ss, red) / (float)H + eps);
  const float *w = which == 0 ? w_e : w_h;
  for (int c0 = 8 * threadIdx.x; c0 < H; c0 += 8 * kThreads) {
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float x = which == 0 ? __bfloat162float(embd[(size_t)tok * H + c0 + e]) : __ldcg(hn + (size_t)m * ldh + c0 + e);
      v[e] = x * r * w[c0 + e];
    }
    store_y8(ylm, m, which * H + c0, v);
  }
}

// X = (X + ) sum of the product's K slices; then rms(X; w) as the next operand
// (and, for the head's output, as f32 rows).  Block m.
__global__ void __launch_bounds__(kThreads) mtp_add_norm_kernel(float *x, bool residual, const float *delta, int slices,
                                                                int H, const float *w, float eps, uint8_t *ylm,
                                                                float *out) {
  __shared__ float red[kThreads / 32];
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x;
  const int M = gridDim.x;
  float ss = 0.f;
  for (int c = threadIdx.x; c < H; c += kThreads) {
    float v = residual ? x[(size_t)m * H + c] : 0.f;
    for (int s = 0; s < slices; ++s) v += __ldcg(delta + (size_t)m * slices * H + (size_t)s * H + c);
    x[(size_t)m * H + c] = v;
    ss += v * v;
  }
  (void)M;
  const float r = rsqrtf(block_sum(ss, red) / (float)H + eps);   // (block_sum syncs: x rows are visible)
  for (int c0 = 8 * threadIdx.x; c0 < H; c0 += 8 * kThreads) {
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = x[(size_t)m * H + c0 + e] * r * w[c0 + e];
    if (ylm) store_y8(ylm, m, c0, v);
    if (out) {
#pragma unroll
      for (int e = 0; e < 8; ++e) out[(size_t)m * H + c0 + e] = v[e];
    }
  }
}

// Per head: RMSNorm over hd, NEOX RoPE on the first rot dims at the row's position;
// q heads -> Q, k heads -> the K cache row, v heads -> the V cache row.
// Block (m, j): j < nh a q head, then nkv k heads, then nkv v heads; thread = dim.
__global__ void mtp_qk_prep_kernel(const float *qkv, int ldq, int nh, int nkv, int hd, int rot, double theta, float eps,
                                   const float *w_q, const float *w_k, int pos0, float *Q, float *kc, float *vc) {
  __shared__ float sh[256];
  __shared__ float red[8];
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x, j = blockIdx.y, d = threadIdx.x;
  const int pos = pos0 + m;
  const float *row = qkv + (size_t)m * ldq;
  if (j >= nh + nkv) {
    const int g = j - nh - nkv;
    vc[(size_t)pos * nkv * hd + g * hd + d] = __ldcg(row + nh * 2 * hd + nkv * hd + g * hd + d);
    return;
  }
  const bool isq = j < nh;
  const float x = isq ? __ldcg(row + j * 2 * hd + d) : __ldcg(row + nh * 2 * hd + (j - nh) * hd + d);
  float ss = warp_sum(x * x);
  if ((d & 31) == 0) red[d >> 5] = ss;
  __syncthreads();
  ss = 0.f;
  for (int i = 0; i < hd / 32; ++i) ss += red[i];
  const float y = x * rsqrtf(ss / (float)hd + eps) * (isq ? w_q[d] : w_k[d]);
  sh[d] = y;
  __syncthreads();
  float out = y;
  if (d < rot) {
    const int half = rot >> 1, i = d < half ? d : d - half;
    // the angle in double, reduced to [-pi, pi] before the single-precision sine and cosine
    double ang = (double)pos * pow(theta, -2.0 * i / rot);
    ang -= 6.283185307179586 * rint(ang / 6.283185307179586);
    float sn, cs;
    sincosf((float)ang, &sn, &cs);
    out = d < half ? y * cs - sh[d + half] * sn : y * cs + sh[d - half] * sn;
  }
  if (isq)
    Q[(size_t)m * nh * hd + j * hd + d] = out;
  else
    kc[(size_t)pos * nkv * hd + (j - nh) * hd + d] = out;
}

// Causal attention of row m, q head h over cache rows kv_lo .. pos0 + m (KV head
// h / (nh / nkv)), online softmax over 256-key tiles, times sigmoid(gate); written
// as the operand of attn_output.  Block (m, h): warps score 32 keys each (lanes
// over the head dims), then thread = dim accumulates P.V.  (Scoring four keys per
// warp at a time, with the lanes on strided or on consecutive dims, was measured
// 9 % slower on the full head's draft.)
__global__ void __launch_bounds__(kThreads) mtp_attn_kernel(const float *Q, const float *qkv, int ldq, const float *kc,
                                                            const float *vc, int nh, int nkv, int hd, int pos0,
                                                            int kv_lo, float scale, uint8_t *ylm) {
  __shared__ float q[256];
  __shared__ float p[256];
  __shared__ float red[8];
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x, h = blockIdx.y, t = threadIdx.x, w = t >> 5, lane = t & 31;
  const int g = h / (nh / nkv), ldk = nkv * hd;
  if (t < hd) q[t] = Q[(size_t)m * nh * hd + h * hd + t];
  __syncthreads();
  const int last = pos0 + m;
  float mx = -INFINITY, l = 0.f, acc = 0.f;
  for (int t0 = kv_lo; t0 <= last; t0 += kThreads) {
    // scores of keys t0 + 32 w .. + 31
    for (int kk = 0; kk < 32; ++kk) {
      const int key = t0 + 32 * w + kk;
      float s = -INFINITY;
      if (key <= last) {
        const float *kr = kc + (size_t)key * ldk + g * hd;
        float dsum = 0.f;
        for (int e = lane; e < hd; e += 32) dsum += q[e] * kr[e];
        s = warp_sum(dsum) * scale;
      }
      if (lane == 0) p[32 * w + kk] = s;
    }
    __syncthreads();
    float tm = -INFINITY;
    for (int i = lane; i < kThreads; i += 32) tm = fmaxf(tm, p[i]);
    tm = warp_max(tm);
    const float nm = fmaxf(mx, tm);
    const float corr = mx == -INFINITY ? 0.f : expf(mx - nm);
    __syncthreads();
    const float pj = p[t] == -INFINITY ? 0.f : expf(p[t] - nm);
    __syncthreads();
    p[t] = pj;
    const float ts = block_sum(pj, red);
    l = l * corr + ts;
    acc *= corr;
    mx = nm;
    const int cnt = min(kThreads, last - t0 + 1);
    if (t < hd)
      for (int jj = 0; jj < cnt; ++jj) acc += p[jj] * vc[(size_t)(t0 + jj) * ldk + g * hd + t];
    __syncthreads();
  }
  if (t < hd) {
    const float gate = __ldcg(qkv + (size_t)m * ldq + h * 2 * hd + hd + t);
    store_y1(ylm, m, h * hd + t, acc / l / (1.f + expf(-gate)));
  }
}

// silu(gate) * up from the stacked gate / up product, as the operand of ffn_down.
__global__ void __launch_bounds__(kThreads) mtp_silu_mul_kernel(const float *gu, int I, uint8_t *ylm) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.y;
  const int c0 = 8 * (blockIdx.x * kThreads + threadIdx.x);
  if (c0 >= I) return;
  float v[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float gt = __ldcg(gu + (size_t)m * 2 * I + c0 + e);
    const float up = __ldcg(gu + (size_t)m * 2 * I + I + c0 + e);
    v[e] = gt / (1.f + expf(-gt)) * up;
  }
  store_y8(ylm, m, c0, v);
}

__global__ void mtp_copy_token_kernel(const int32_t *src, int32_t *dst) {
  pdl_trigger();
  pdl_wait();
  *dst = *src;
}

template <typename K, typename... Args>
cudaError_t launch(K kern, dim3 grid, dim3 block, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

thread_local std::string g_mtp_error;

}  // namespace
}  // namespace fm

using namespace fm;

struct fm_mtp {
  fm_mtp_config cfg{};
  std::string err;
  int n_sm = 0;
  std::vector<void *> allocs;
  // a Q8_0 product: the repacked table (slices of K in tile order), out features, in features, slices
  struct Lin {
    uint8_t *t = nullptr;
    int N = 0, K = 0, S = 1;
  };
  Lin eh, qkv, o, gu, down, lm;
  float *n_e = nullptr, *n_h = nullptr, *n_attn = nullptr, *n_q = nullptr, *n_k = nullptr, *n_post = nullptr,
        *n_shared = nullptr;
  __nv_bfloat16 *embd = nullptr;
  float *kc = nullptr, *vc = nullptr;
  float *x = nullptr, *hout = nullptr, *y = nullptr, *Q = nullptr;
  uint8_t *ylm = nullptr;
  float2 *part = nullptr;
  int32_t *ticket = nullptr, *tok = nullptr, *dev_err = nullptr;
  size_t y_floats = 0;
  int last_launches = 0;
};

namespace {

fm_status mfail(fm_mtp *m, fm_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (m)
    m->err = buf;
  else
    g_mtp_error = buf;
  return s;
}

#define MCK(expr)                                                                                   \
  do {                                                                                              \
    cudaError_t e_ = (expr);                                                                        \
    if (e_ != cudaSuccess) return mfail(m, FM_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_));   \
  } while (0)
#define MTRY(expr)                       \
  do {                                   \
    fm_status s_ = (expr);               \
    if (s_ != FM_OK) return s_;          \
  } while (0)

template <typename T>
fm_status malloc_dev(fm_mtp *m, T **p, size_t count) {
  void *q = nullptr;
  if (cudaMalloc(&q, (count ? count : 1) * sizeof(T)) != cudaSuccess) {
    cudaGetLastError();
    return mfail(m, FM_ERR_OOM, "device allocation of %zu bytes failed", count * sizeof(T));
  }
  m->allocs.push_back(q);
  *p = static_cast<T *>(q);
  return FM_OK;
}

const fm_tensor *find_tensor(const std::unordered_map<std::string, const fm_tensor *> &ts, const char *name) {
  auto it = ts.find(name);
  return it == ts.end() ? nullptr : it->second;
}

fm_status need(fm_mtp *m, const std::unordered_map<std::string, const fm_tensor *> &ts, const char *name,
               int32_t dtype, int64_t bytes, const fm_tensor **out) {
  const fm_tensor *t = find_tensor(ts, name);
  if (!t) return mfail(m, FM_ERR_INVALID_ARG, "missing tensor %s", name);
  if (t->dtype != dtype) return mfail(m, FM_ERR_INVALID_ARG, "tensor %s: dtype %d, expected %d", name, t->dtype, dtype);
  if (t->nbytes != bytes)
    return mfail(m, FM_ERR_INVALID_ARG, "tensor %s: %lld bytes, expected %lld", name, (long long)t->nbytes,
                 (long long)bytes);
  if (!t->data) return mfail(m, FM_ERR_INVALID_ARG, "tensor %s: null data", name);
  *out = t;
  return FM_OK;
}

// Q8_0 rows of the named tensors stacked along N, split along K into S slices
// (slice s = every row's blocks s K/S .. (s+1) K/S - 1, the slices one after
// another), repacked into the lm_head table layout.
fm_status load_lin(fm_mtp *m, const std::unordered_map<std::string, const fm_tensor *> &ts,
                   std::initializer_list<std::pair<const char *, int>> parts, int K, int S, fm_mtp::Lin *L,
                   cudaStream_t s) {
  int N = 0;
  for (auto &p : parts) N += p.second;
  const size_t row = (size_t)K / 32 * 34, srow = row / S;
  uint8_t *raw;
  MTRY(malloc_dev(m, &raw, (size_t)N * row));
  int r0 = 0;
  for (auto &p : parts) {
    const fm_tensor *t;
    MTRY(need(m, ts, p.first, FM_DTYPE_Q8_0, (int64_t)p.second * (int64_t)row, &t));
    for (int sl = 0; sl < S; ++sl)
      MCK(cudaMemcpy2DAsync(raw + ((size_t)sl * N + r0) * srow, srow, static_cast<const uint8_t *>(t->data) + sl * srow,
                            row, srow, p.second, cudaMemcpyDefault, s));
    r0 += p.second;
  }
  MTRY(malloc_dev(m, &L->t, q8_table_bytes(S * N, K / S)));
  MCK(launch_q8_repack(raw, S * N, K / S, L->t, s));
  MCK(cudaStreamSynchronize(s));
  cudaFree(raw);
  m->allocs.erase(std::find(m->allocs.begin(), m->allocs.end(), static_cast<void *>(raw)));
  L->N = N;
  L->K = K;
  L->S = S;
  return FM_OK;
}

fm_status load_f32(fm_mtp *m, const std::unordered_map<std::string, const fm_tensor *> &ts, const char *name, int n,
                   float **dst, cudaStream_t s) {
  const fm_tensor *t;
  MTRY(need(m, ts, name, FM_DTYPE_F32, (int64_t)n * 4, &t));
  MTRY(malloc_dev(m, dst, n));
  MCK(cudaMemcpyAsync(*dst, t->data, (size_t)n * 4, cudaMemcpyDefault, s));
  return FM_OK;
}

// slices for a product of N out features: enough 128-row tiles to cover the SMs,
// each slice at least 16 chunks of 64 columns
int pick_slices(int N, int K, int n_sm) {
  int S = 1;
  const int tiles = N / 128;
  while (tiles * S * 2 <= n_sm + n_sm / 4 && (K / (S * 2)) % 64 == 0 && K / (S * 2) >= 1024) S *= 2;
  return S;
}

// one Q8_0 product: out[t][s N + n] = slice s's partial sum for rows t < M
fm_status run_lin(fm_mtp *m, const fm_mtp::Lin &L, int M, float *out, int32_t *tokens, cudaStream_t s) {
  LmArgs a;
  memset(&a, 0, sizeof a);
  a.q8 = L.t;
  a.err = m->dev_err;
  a.V = L.S * L.N;
  a.H = L.K / L.S;
  a.T_const = M;
  a.ldy = a.H;
  a.ylm = m->ylm;
  a.part = m->part;
  a.ticket = m->ticket;
  a.tokens = tokens ? tokens : m->tok;
  a.logits = out;
  a.y_slice_tiles = L.S > 1 ? L.N / 128 : 0;
  MCK(launch_lmhead(a, lmhead_grid(a, m->n_sm), s, true));
  ++m->last_launches;
  return FM_OK;
}

// MTPHead.forward over M rows; drafts: per-row argmax of the lm_head, or null
fm_status mtp_pass(fm_mtp *m, int M, const int32_t *tokens, const float *hn, int ldh, int pos0, int kv_lo,
                   int32_t *drafts, cudaStream_t s) {
  const fm_mtp_config &c = m->cfg;
  const int H = c.hidden, I = c.inter, nh = c.n_heads, nkv = c.n_kv_heads, hd = c.head_dim;
  MCK(launch(mtp_embed_norm_kernel, dim3(2 * M), dim3(kThreads), s, (const __nv_bfloat16 *)m->embd, tokens, c.vocab,
             hn, ldh, (const float *)m->n_e, (const float *)m->n_h, H, c.eps, m->ylm, m->dev_err));
  ++m->last_launches;
  MTRY(run_lin(m, m->eh, M, m->y, nullptr, s));
  MCK(launch(mtp_add_norm_kernel, dim3(M), dim3(kThreads), s, m->x, false, (const float *)m->y, m->eh.S, H,
             (const float *)m->n_attn, c.eps, m->ylm, (float *)nullptr));
  ++m->last_launches;
  MTRY(run_lin(m, m->qkv, M, m->y, nullptr, s));
  MCK(launch(mtp_qk_prep_kernel, dim3(M, nh + 2 * nkv), dim3(hd), s, (const float *)m->y, m->qkv.N, nh, nkv, hd,
             c.rot_dims, (double)c.theta, c.eps, (const float *)m->n_q, (const float *)m->n_k, pos0, m->Q, m->kc, m->vc));
  ++m->last_launches;
  MCK(launch(mtp_attn_kernel, dim3(M, nh), dim3(kThreads), s, (const float *)m->Q, (const float *)m->y, m->qkv.N,
             (const float *)m->kc, (const float *)m->vc, nh, nkv, hd, pos0, kv_lo, 1.0f / sqrtf((float)hd), m->ylm));
  ++m->last_launches;
  // attn_output's slices land beside the q/k/v rows' gates (read above): a separate region
  float *yo = m->y + (size_t)kMaxRows * m->qkv.N;
  MTRY(run_lin(m, m->o, M, yo, nullptr, s));
  MCK(launch(mtp_add_norm_kernel, dim3(M), dim3(kThreads), s, m->x, true, (const float *)yo, m->o.S, H,
             (const float *)m->n_post, c.eps, m->ylm, (float *)nullptr));
  ++m->last_launches;
  MTRY(run_lin(m, m->gu, M, m->y, nullptr, s));
  MCK(launch(mtp_silu_mul_kernel, dim3((I / 8 + kThreads - 1) / kThreads, M), dim3(kThreads), s, (const float *)m->y, I,
             m->ylm));
  ++m->last_launches;
  MTRY(run_lin(m, m->down, M, yo, nullptr, s));
  MCK(launch(mtp_add_norm_kernel, dim3(M), dim3(kThreads), s, m->x, true, (const float *)yo, m->down.S, H,
             (const float *)m->n_shared, c.eps, m->ylm, m->hout));
  ++m->last_launches;
  // the lm_head (one slice): drafts per row
  MTRY(run_lin(m, m->lm, M, nullptr, drafts ? drafts : m->tok, s));
  return FM_OK;
}

fm_status mtp_checks(fm_mtp *m, int M, const int32_t *tokens, const float *hn, int pos0, int kv_lo) {
  const fm_mtp_config &c = m->cfg;
  if (M < 1 || M > c.max_rows) return mfail(m, FM_ERR_INVALID_ARG, "n_rows %d outside [1, %d]", M, c.max_rows);
  if (!tokens || !hn) return mfail(m, FM_ERR_INVALID_ARG, "null tokens or hidden rows");
  if (pos0 < 0 || kv_lo < 0 || kv_lo > pos0) return mfail(m, FM_ERR_INVALID_ARG, "kv_lo %d outside [0, pos0 %d]", kv_lo, pos0);
  if (pos0 + M > c.kv_cap) return mfail(m, FM_ERR_INVALID_ARG, "pos0 + n_rows = %d > kv_cap %d", pos0 + M, c.kv_cap);
  return FM_OK;
}

}  // namespace

extern "C" {

fm_status fm_mtp_create(const fm_mtp_config *cfg, const fm_tensor *weights, int32_t n_weights, void *stream,
                        fm_mtp **out) {
  if (!out) return mfail(nullptr, FM_ERR_INVALID_ARG, "null out");
  *out = nullptr;
  if (!cfg || (!weights && n_weights > 0) || n_weights < 0) return mfail(nullptr, FM_ERR_INVALID_ARG, "bad arguments");
  const fm_mtp_config c = *cfg;
  const int H = c.hidden, I = c.inter, nh = c.n_heads, nkv = c.n_kv_heads, hd = c.head_dim;
  if (H < 128 || H % 128 || I < 128 || I % 128 || nh < 1 || nkv < 1 || nh % nkv || hd < 32 || hd > 256 || hd % 32 ||
      c.rot_dims < 0 || c.rot_dims > hd || c.rot_dims % 2 || c.vocab < 1 || c.kv_cap < 1 || c.max_rows < 1 ||
      c.max_rows > kMaxRows || (nh * 2 * hd + 2 * nkv * hd) % 128 || (nh * hd) % 64 || !(c.eps > 0.f) ||
      !(c.theta > 0.f))
    return mfail(nullptr, FM_ERR_UNSUPPORTED, "MTP config outside the supported limits");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  fm_mtp *m = new fm_mtp();
  m->cfg = c;
  auto bail = [&](fm_status st) {
    g_mtp_error = m->err;
    for (void *p : m->allocs) cudaFree(p);
    delete m;
    return st;
  };
  std::unordered_map<std::string, const fm_tensor *> ts;
  for (int i = 0; i < n_weights; ++i)
    if (weights[i].name) ts[weights[i].name] = &weights[i];
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&m->n_sm, cudaDevAttrMultiProcessorCount, dev);
  fm_status st;
#define STEP(expr)              \
  if ((st = (expr)) != FM_OK) { \
    return bail(st);            \
  }
  STEP(load_lin(m, ts, {{"eh_proj", H}}, 2 * H, pick_slices(H, 2 * H, m->n_sm), &m->eh, s));
  // (the q/k/v and gate/up outputs are read by kernels that take one slice)
  STEP(load_lin(m, ts, {{"attn_q", nh * 2 * hd}, {"attn_k", nkv * hd}, {"attn_v", nkv * hd}}, H, 1, &m->qkv, s));
  STEP(load_lin(m, ts, {{"attn_output", H}}, nh * hd, pick_slices(H, nh * hd, m->n_sm), &m->o, s));
  STEP(load_lin(m, ts, {{"ffn_gate", I}, {"ffn_up", I}}, H, 1, &m->gu, s));
  STEP(load_lin(m, ts, {{"ffn_down", H}}, I, pick_slices(H, I, m->n_sm), &m->down, s));
  // the lm_head: vocab rows padded to whole tiles by the repack
  {
    const fm_tensor *t;
    const size_t row = (size_t)H / 32 * 34;
    STEP(need(m, ts, "lm_head", FM_DTYPE_Q8_0, (int64_t)c.vocab * (int64_t)row, &t));
    uint8_t *raw;
    STEP(malloc_dev(m, &raw, (size_t)c.vocab * row));
    if (cudaMemcpyAsync(raw, t->data, (size_t)c.vocab * row, cudaMemcpyDefault, s) != cudaSuccess)
      return bail(mfail(m, FM_ERR_CUDA, "lm_head upload failed"));
    STEP(malloc_dev(m, &m->lm.t, q8_table_bytes(c.vocab, H)));
    if (launch_q8_repack(raw, c.vocab, H, m->lm.t, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
      return bail(mfail(m, FM_ERR_CUDA, "lm_head repack failed"));
    cudaFree(raw);
    m->allocs.erase(std::find(m->allocs.begin(), m->allocs.end(), static_cast<void *>(raw)));
    m->lm.N = c.vocab;
    m->lm.K = H;
    m->lm.S = 1;
  }
  STEP(load_f32(m, ts, "enorm", H, &m->n_e, s));
  STEP(load_f32(m, ts, "hnorm", H, &m->n_h, s));
  STEP(load_f32(m, ts, "attn_norm", H, &m->n_attn, s));
  STEP(load_f32(m, ts, "post_attention_norm", H, &m->n_post, s));
  STEP(load_f32(m, ts, "shared_head_norm", H, &m->n_shared, s));
  STEP(load_f32(m, ts, "attn_q_norm", hd, &m->n_q, s));
  STEP(load_f32(m, ts, "attn_k_norm", hd, &m->n_k, s));
  {
    const fm_tensor *t;
    STEP(need(m, ts, "token_embd", FM_DTYPE_BF16, (int64_t)c.vocab * H * 2, &t));
    STEP(malloc_dev(m, &m->embd, (size_t)c.vocab * H));
    if (cudaMemcpyAsync(m->embd, t->data, (size_t)c.vocab * H * 2, cudaMemcpyDefault, s) != cudaSuccess)
      return bail(mfail(m, FM_ERR_CUDA, "token_embd upload failed"));
  }
  const size_t kvw = (size_t)nkv * hd;
  STEP(malloc_dev(m, &m->kc, (size_t)c.kv_cap * kvw));
  STEP(malloc_dev(m, &m->vc, (size_t)c.kv_cap * kvw));
  if (cudaMemsetAsync(m->kc, 0, (size_t)c.kv_cap * kvw * 4, s) != cudaSuccess ||
      cudaMemsetAsync(m->vc, 0, (size_t)c.kv_cap * kvw * 4, s) != cudaSuccess)
    return bail(mfail(m, FM_ERR_CUDA, "cache clear failed"));
  STEP(malloc_dev(m, &m->x, (size_t)kMaxRows * H));
  STEP(malloc_dev(m, &m->hout, (size_t)kMaxRows * H));
  STEP(malloc_dev(m, &m->Q, (size_t)kMaxRows * nh * hd));
  // product outputs: [rows][slices * N] for every product; attn_output / ffn_down after the q/k/v rows
  size_t yf = 0;
  for (const fm_mtp::Lin *L : {&m->eh, &m->qkv, &m->gu}) yf = std::max(yf, (size_t)kMaxRows * L->S * L->N);
  yf = std::max(yf, (size_t)kMaxRows * m->qkv.N + (size_t)kMaxRows * std::max(m->o.S, m->down.S) * H);
  m->y_floats = yf;
  STEP(malloc_dev(m, &m->y, yf));
  const int kmax = std::max(std::max(2 * H, I), nh * hd);
  STEP(malloc_dev(m, &m->ylm, (size_t)(kmax / 64) * kLmYChunk));
  if (cudaMemsetAsync(m->ylm, 0, (size_t)(kmax / 64) * kLmYChunk, s) != cudaSuccess)
    return bail(mfail(m, FM_ERR_CUDA, "operand clear failed"));
  STEP(malloc_dev(m, &m->part, (size_t)m->n_sm * kMaxT));
  STEP(malloc_dev(m, &m->ticket, 4));
  STEP(malloc_dev(m, &m->tok, 32));
  STEP(malloc_dev(m, &m->dev_err, 4));
  if (cudaMemsetAsync(m->ticket, 0, 16, s) != cudaSuccess || cudaMemsetAsync(m->dev_err, 0, 4, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return bail(mfail(m, FM_ERR_CUDA, "set-up failed"));
#undef STEP
  *out = m;
  return FM_OK;
}

fm_status fm_mtp_forward(fm_mtp *m, int32_t n_rows, const int32_t *tokens_dev, const float *hn_dev, int32_t pos0,
                         int32_t kv_lo, float *hout_dev, int32_t *drafts_dev, void *stream) {
  if (!m) return FM_ERR_INVALID_ARG;
  m->last_launches = 0;
  MTRY(mtp_checks(m, n_rows, tokens_dev, hn_dev, pos0, kv_lo));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MTRY(mtp_pass(m, n_rows, tokens_dev, hn_dev, m->cfg.hidden, pos0, kv_lo, drafts_dev, s));
  if (hout_dev)
    MCK(cudaMemcpyAsync(hout_dev, m->hout, (size_t)n_rows * m->cfg.hidden * 4, cudaMemcpyDeviceToDevice, s));
  return FM_OK;
}

fm_status fm_mtp_draft(fm_mtp *m, int32_t n_rows, const int32_t *tokens_dev, const float *hn_dev, int32_t pos0,
                       int32_t kv_lo, int32_t depth, int32_t *drafts_dev, void *stream) {
  if (!m) return FM_ERR_INVALID_ARG;
  m->last_launches = 0;
  MTRY(mtp_checks(m, n_rows, tokens_dev, hn_dev, pos0, kv_lo));
  if (!drafts_dev) return mfail(m, FM_ERR_INVALID_ARG, "null drafts");
  if (depth < 1 || pos0 + n_rows + depth - 1 > m->cfg.kv_cap)
    return mfail(m, FM_ERR_INVALID_ARG, "depth %d outside [1, %d]", depth, m->cfg.kv_cap - pos0 - n_rows + 1);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int H = m->cfg.hidden;
  MTRY(mtp_pass(m, n_rows, tokens_dev, hn_dev, H, pos0, kv_lo, nullptr, s));
  MCK(launch(mtp_copy_token_kernel, dim3(1), dim3(1), s, (const int32_t *)(m->tok + n_rows - 1), drafts_dev));
  ++m->last_launches;
  int last = n_rows - 1;
  for (int d = 1; d < depth; ++d) {
    // the previous draft, with the previous pass's last h' (row `last` of hout)
    MTRY(mtp_pass(m, 1, drafts_dev + d - 1, m->hout + (size_t)last * H, H, pos0 + n_rows + d - 1, kv_lo,
                  drafts_dev + d, s));
    last = 0;
  }
  return FM_OK;
}

fm_status fm_mtp_cache(fm_mtp *m, int32_t which, int32_t rows, float *dst, void *stream) {
  if (!m) return FM_ERR_INVALID_ARG;
  if ((which != 0 && which != 1) || rows < 0 || rows > m->cfg.kv_cap || !dst)
    return mfail(m, FM_ERR_INVALID_ARG, "bad cache copy arguments");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MCK(cudaMemcpyAsync(dst, which ? m->vc : m->kc, (size_t)rows * m->cfg.n_kv_heads * m->cfg.head_dim * 4,
                      cudaMemcpyDefault, s));
  MCK(cudaStreamSynchronize(s));
  int32_t e = 0;
  MCK(cudaMemcpy(&e, m->dev_err, 4, cudaMemcpyDeviceToHost));
  if (e) {
    cudaMemset(m->dev_err, 0, 4);
    return e == 2 ? mfail(m, FM_ERR_INVALID_ARG, "a token outside [0, vocab) reached the embedding")
                  : mfail(m, FM_ERR_TIMEOUT, "a bounded device wait gave up");
  }
  return FM_OK;
}

fm_status fm_mtp_last_launch_count(const fm_mtp *m, int32_t *count) {
  if (!m || !count) return FM_ERR_INVALID_ARG;
  *count = m->last_launches;
  return FM_OK;
}

const char *fm_mtp_last_error(const fm_mtp *m) { return m ? m->err.c_str() : g_mtp_error.c_str(); }

void fm_mtp_destroy(fm_mtp *m) {
  if (!m) return;
  cudaDeviceSynchronize();
  for (void *p : m->allocs) cudaFree(p);
  delete m;
}

}  // extern "C"
