// k_setup.cu -- one-time set-up kernels run by fm_create, and small kernels.
#include "dev_common.cuh"
#include "fm_internal.h"

namespace fm {

namespace {

// GGUF Q8_0 rows [V][nb * 34] -> the lm_head layout: per (128-row tile, 64-column
// chunk) 128 x 64 weights as offset-binary bytes q + 128 (pre-swizzled; rows past V
// hold q = 0, the byte 0x80) then the chunk's two blocks of f16 scales
// [2][128] (the MTP loader on ternary_bonsai_2_mtp.js splits the 34-byte blocks
// into an int8 plane and a scale plane; here both halves of a chunk sit together
// so one bulk copy fetches them).  One thread per block.
__global__ void q8_repack_kernel(const uint8_t *raw, int V, int H, uint8_t *dst) {
  const int nb = H / 32, nck = H / 64;
  const int Vpad = (V + 127) / 128 * 128;
  const long long id = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (id >= (long long)Vpad * nb) return;
  const int r = (int)(id / nb), b = (int)(id - (long long)r * nb);
  const int tile = r >> 7, rr = r & 127, kc = b >> 1, bb = b & 1;
  uint8_t *chunk = dst + ((size_t)tile * nck + kc) * kQ8Chunk;
  uint8_t q[32];
  unsigned short d = 0;
  if (r < V) {
    const uint8_t *src = raw + (size_t)r * nb * 34 + b * 34;
    d = (unsigned short)src[0] | ((unsigned short)src[1] << 8);
    for (int i = 0; i < 32; ++i) q[i] = src[2 + i];
  } else {
    for (int i = 0; i < 32; ++i) q[i] = 0;
  }
  // offset binary: the byte q + 128 (q ^ 0x80), so the converters place it straight into an f16 mantissa
  for (int i = 0; i < 32; ++i) chunk[q8_slot(rr, 32 * bb + i)] = (uint8_t)(q[i] ^ 0x80u);
  *reinterpret_cast<unsigned short *>(chunk + kTile * 64 + bb * 256 + rr * 2) = d;
}

// column sums in double over a slab of rows; partial[slab][col]
__global__ void colsum_q8_kernel(const uint8_t *raw, int V, int H, int rows_per_slab, double *partial) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= H) return;
  const int nb = H / 32;
  const int r0 = blockIdx.y * rows_per_slab, r1 = min(V, r0 + rows_per_slab);
  double s = 0.0;
  for (int r = r0; r < r1; ++r) {
    const uint8_t *blk = raw + (size_t)r * nb * 34 + (c >> 5) * 34;
    const unsigned short db = (unsigned short)blk[0] | ((unsigned short)blk[1] << 8);
    const float d = __half2float(__ushort_as_half(db));
    s += (double)(d * (float)(int8_t)blk[2 + (c & 31)]);
  }
  partial[(size_t)blockIdx.y * H + c] = s;
}

__global__ void colsum_bf16_kernel(const __nv_bfloat16 *w, int V, int H, int rows_per_slab, double *partial) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= H) return;
  const int r0 = blockIdx.y * rows_per_slab, r1 = min(V, r0 + rows_per_slab);
  double s = 0.0;
  for (int r = r0; r < r1; ++r) s += (double)__bfloat162float(w[(size_t)r * H + c]);
  partial[(size_t)blockIdx.y * H + c] = s;
}

__global__ void colmean_finish_kernel(const double *partial, int slabs, int H, int V, float *out) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= H) return;
  double s = 0.0;
  for (int i = 0; i < slabs; ++i) s += partial[(size_t)i * H + c];
  out[c] = (float)(s / (double)V);
}

// (cos, sin) of p * theta^(-2i / hd), angles in double
__global__ void rope_table_kernel(float2 *tab, int n_pos, int hd, double theta) {
  const int half = hd / 2;
  const long long id = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (id >= (long long)n_pos * half) return;
  const int p = (int)(id / half), i = (int)(id - (long long)p * half);
  const double inv = pow(theta, -2.0 * (double)i / (double)hd);
  double s, c;
  sincos((double)p * inv, &s, &c);
  tab[id] = make_float2((float)c, (float)s);
}

__global__ void transpose_bf16_kernel(const __nv_bfloat16 *in, int rows, int cols, __nv_bfloat16 *out, int ldo) {
  __shared__ __nv_bfloat16 t[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols) t[i][threadIdx.x] = in[(size_t)r * cols + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (r < rows && c < cols) out[(size_t)c * ldo + r] = t[threadIdx.x][i];
  }
}

// DFlash block rows 1 .. gamma-1: mask_emb[j-1] + block_pos[j] (module-dflash.ts #buildBlock)
__global__ void block_consts_kernel(const __nv_bfloat16 *mask_emb, const __nv_bfloat16 *block_pos, int gamma, int d,
                                    float *out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= gamma * d) return;
  const int j = i / d, k = i - j * d;
  out[i] = j == 0 ? 0.f : __bfloat162float(mask_emb[(size_t)(j - 1) * d + k]) + __bfloat162float(block_pos[i]);
}

// (mean, M2) of each row over each 128-column tile, two-pass (M2 = the sum of
// squared deviations from the tile mean): st[tile * kMaxT + row].  Consumers
// combine the tiles with the pairwise update of Chan, Golub and LeVeque.
__global__ void row_stats_kernel(const float *x, int rows, int d, float2 *st) {
  const int tile = blockIdx.x, row = blockIdx.y;
  const int lane = threadIdx.x;
  const int c0 = tile * kTile, c1 = min(d, (tile + 1) * kTile);
  float s = 0.f;
  for (int c = c0 + lane; c < c1; c += 32) s += x[(size_t)row * d + c];
  const float mean = warp_sum(s) / (float)(c1 - c0);
  float q = 0.f;
  for (int c = c0 + lane; c < c1; c += 32) {
    const float e = x[(size_t)row * d + c] - mean;
    q += e * e;
  }
  q = warp_sum(q);
  if (lane == 0 && row < rows) st[tile * kMaxT + row] = make_float2(mean, q);
}

// ---- time conditioning (flashmap_drafter.js, ``timeConditioning``): set-up only ----
// [cos a_i | sin a_i], a_i = time * time_scale * exp(-ln(10000) i / half), in double
__global__ void time_embed_kernel(float *e, int time_dim, double time_scale, double time) {
  const int half = time_dim / 2;
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    const double a = time * time_scale * exp(-log(10000.0) * (double)i / (double)half);
    e[i] = (float)cos(a);
    e[half + i] = (float)sin(a);
  }
}
__device__ __forceinline__ float silu(float v) { return v / (1.f + expf(-v)); }
// y[m] = sum_k W[m][k] x'[k] + b[m] (bf16 W [M][N], optional bias), one warp per
// row; x' = x (act 0), SiLU(x) (act 1) or SiLU(x + x2) (act 2)
__global__ void setup_linear_kernel(const __nv_bfloat16 *W, const __nv_bfloat16 *b, const float *x, const float *x2,
                                    int M, int N, int act, float *y) {
  const int m = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (m >= M) return;
  float acc = 0.f;
  for (int k = lane; k < N; k += 32) {
    float v = x[k];
    if (act == 1) v = silu(v);
    if (act == 2) v = silu(v + x2[k]);
    acc = fmaf(__bfloat162float(W[(size_t)m * N + k]), v, acc);
  }
  acc = warp_sum(acc);
  if (lane == 0) y[m] = acc + (b ? __bfloat162float(b[m]) : 0.f);
}

// The failure path of the bounded waits: one thread waits on an mbarrier phase
// that nothing completes, with a short budget; the wait gives up, raises the
// error word and the kernel returns (nothing hangs, nothing faults).
__global__ void wait_selftest_kernel(int32_t *err, long long budget_cycles) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(b, 0, err, budget_cycles);
  __syncthreads();
}

__global__ void accept_kernel(int n, int block, const int32_t *draft, const int32_t *target, const int32_t *k,
                              int32_t *acc, int32_t *bonus) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  int kk = k[i];
  kk = kk < 0 ? 0 : (kk > block ? block : kk);
  const int32_t *d = draft + (size_t)i * block, *t = target + (size_t)i * (block + 1);
  int a = 0;
  while (a < kk && d[a] == t[a]) ++a;
  acc[i] = a;
  bonus[i] = t[a];
}

// One 16-byte unit (8 bf16) per thread: row r, unit u of chunk kc of tile
// -> byte ((tile * nck + kc) * 16384) + sw128(r, 8u): the tensor cores'
// 128-byte-swizzle K-major layout, so a bulk copy lands a ready operand tile.
__global__ void tile_weights_kernel(const uint4 *src, int M, int K, uint8_t *dst) {
  const int nck = K / 64;
  const long long id = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const int n_tiles = (M + 127) / 128;
  if (id >= (long long)n_tiles * nck * 1024) return;
  const int u = (int)(id & 7), r = (int)((id >> 3) & 127);
  const long long tk = id >> 10;
  const int kc = (int)(tk % nck), tile = (int)(tk / nck);
  const int m = tile * 128 + r;
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (m < M) v = src[((size_t)m * K + (size_t)kc * 64 + u * 8) / 8];
  *reinterpret_cast<uint4 *>(dst + (size_t)tk * 16384 + sw128(r, 8 * u)) = v;
}

__global__ void fill_kernel(float *p, size_t n, float v) {
  const size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (i < n) p[i] = v;
}

}  // namespace

size_t q8_table_bytes(int32_t V, int32_t H) { return (size_t)((V + 127) / 128) * (H / 64) * kQ8Chunk; }

cudaError_t launch_q8_repack(const uint8_t *raw, int32_t V, int32_t H, uint8_t *dst, cudaStream_t s) {
  const long long n = (long long)((V + 127) / 128 * 128) * (H / 32);
  q8_repack_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(raw, V, H, dst);
  return cudaGetLastError();
}

static cudaError_t colmean_common(const void *a, const __half *sc, bool q8, int32_t V, int32_t H, float *out,
                                  cudaStream_t s) {
  const int slabs = 128;
  const int rps = (V + slabs - 1) / slabs;
  double *partial = nullptr;
  cudaError_t e = cudaMallocAsync(&partial, sizeof(double) * slabs * H, s);
  if (e != cudaSuccess) return e;
  dim3 grid((H + 127) / 128, slabs);
  if (q8)
    colsum_q8_kernel<<<grid, 128, 0, s>>>(static_cast<const uint8_t *>(a), V, H, rps, partial);
  else
    colsum_bf16_kernel<<<grid, 128, 0, s>>>(static_cast<const __nv_bfloat16 *>(a), V, H, rps, partial);
  colmean_finish_kernel<<<(H + 127) / 128, 128, 0, s>>>(partial, slabs, H, V, out);
  e = cudaGetLastError();
  cudaFreeAsync(partial, s);
  return e;
}

cudaError_t launch_colmean_q8(const uint8_t *raw, int32_t V, int32_t H, float *out, cudaStream_t s) {
  return colmean_common(raw, nullptr, true, V, H, out, s);
}

cudaError_t launch_colmean_bf16(const __nv_bfloat16 *w, int32_t V, int32_t H, float *out, cudaStream_t s) {
  return colmean_common(w, nullptr, false, V, H, out, s);
}

cudaError_t launch_rope_table(float2 *tab, int32_t n_pos, int32_t hd, float theta, cudaStream_t s) {
  const long long n = (long long)n_pos * (hd / 2);
  rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(tab, n_pos, hd, (double)theta);
  return cudaGetLastError();
}

cudaError_t launch_transpose_bf16(const __nv_bfloat16 *in, int32_t rows, int32_t cols, __nv_bfloat16 *out,
                                  int32_t ldo, cudaStream_t s) {
  dim3 grid((cols + 31) / 32, (rows + 31) / 32), block(32, 8);
  transpose_bf16_kernel<<<grid, block, 0, s>>>(in, rows, cols, out, ldo);
  return cudaGetLastError();
}

cudaError_t launch_block_consts(const __nv_bfloat16 *mask_emb, const __nv_bfloat16 *block_pos, int32_t gamma,
                                int32_t d, float *out, float2 *st, cudaStream_t s) {
  block_consts_kernel<<<(gamma * d + 255) / 256, 256, 0, s>>>(mask_emb, block_pos, gamma, d, out);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_row_stats(out, gamma, d, st, s);
}

cudaError_t launch_row_stats(const float *x, int32_t rows, int32_t d, float2 *st, cudaStream_t s) {
  dim3 grid((d + kTile - 1) / kTile, rows);
  row_stats_kernel<<<grid, 32, 0, s>>>(x, rows, d, st);
  return cudaGetLastError();
}

cudaError_t launch_accept(int32_t n, int32_t block, const int32_t *draft, const int32_t *target, const int32_t *k,
                          int32_t *acc, int32_t *bonus, cudaStream_t s) {
  accept_kernel<<<(n + 127) / 128, 128, 0, s>>>(n, block, draft, target, k, acc, bonus);
  return cudaGetLastError();
}

size_t tiled_bytes(int32_t M, int32_t K) { return (size_t)((M + 127) / 128) * (K / 64) * 16384; }

cudaError_t launch_tile_weights(const __nv_bfloat16 *src, int32_t M, int32_t K, uint8_t *dst, cudaStream_t s) {
  const long long n = (long long)((M + 127) / 128) * (K / 64) * 1024;
  tile_weights_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(reinterpret_cast<const uint4 *>(src), M, K, dst);
  return cudaGetLastError();
}

cudaError_t launch_fill_f32(float *p, size_t n, float v, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  fill_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(p, n, v);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int32_t *err, long long budget_cycles, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(err, budget_cycles);
  return cudaGetLastError();
}

cudaError_t launch_time_embed(float *e, int32_t time_dim, double time_scale, double time, cudaStream_t s) {
  time_embed_kernel<<<1, 256, 0, s>>>(e, time_dim, time_scale, time);
  return cudaGetLastError();
}

cudaError_t launch_setup_linear(const __nv_bfloat16 *W, const __nv_bfloat16 *b, const float *x, const float *x2,
                                int32_t M, int32_t N, int32_t act, float *y, cudaStream_t s) {
  setup_linear_kernel<<<(M + 7) / 8, 256, 0, s>>>(W, b, x, x2, M, N, act, y);
  return cudaGetLastError();
}

}  // namespace fm
