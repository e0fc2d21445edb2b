// fm_internal.h -- kernel argument blocks and launcher declarations shared by
// the host runtime (fm_api.cu) and the kernels.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace fm {

constexpr int kMaxT = 32;        // rows a skinny GEMV carries (two m16 MMA tiles)
constexpr int kTile = 128;       // output rows per GEMV tile (one 128-wide head)
constexpr int kMaxSegs = 16;     // row segments a GEMV epilogue distinguishes

// Device-resident per-call values.  The host fills one slot before each call
// so that launches (and captured graphs) stay fixed while positions move.
struct StepParams {
  int32_t T;        // rows in this chain: draft = block, append = n_rows
  int32_t pos;      // draft: the anchor's position
  int32_t L;        // cross-attention keys
  int32_t anchor;   // draft: anchor token id
  int32_t start;    // append: first position
  int32_t stable;   // cache rows < stable are not written by any kernel of this call
  int32_t pad1, pad2;
  const float *feats;  // append: feature rows [T][feat_dim]
  int32_t *tokens;     // draft: where the argmax tokens go [T]
  float *conf;         // sequential head: the confidence of each position [T], or null
  int32_t *length;     // sequential head: positions kept after pruning [1], or null
  float thr[16];       // sequential head: pruning threshold of each position (NaN: none)
};

// --- batched draft: many sequences' slot rows through the tensor-core GEMM ---
constexpr int kWideSeqs = 32;                  // sequences per batched pass
constexpr int kWideRows = kWideSeqs * 16;      // slot rows per pass
// Device-resident per-pass values of a batched draft (uploaded before the
// chain, so a captured chain stays fixed while positions move).
struct WideParams {
  int32_t n;                     // sequences in this pass
  int32_t pad[3];
  int32_t *tokens;               // [n][block] the drafted tokens
  int32_t seq[kWideSeqs];        // pass slot -> sequence id
  int32_t anchor[kWideSeqs];     // pass slot -> anchor token
  int32_t pos[kWideSeqs];        // pass slot -> anchor position (the context length before the draft)
  // cross-attention launch slots, longest context first: pass slot, sequence, keys
  int32_t z_call[kWideSeqs], z_seq[kWideSeqs], z_L[kWideSeqs];
  int32_t kv_seq[kWideSeqs];     // anchor rows' K/V: sequence and position
  int32_t kv_pos[kWideSeqs];
  int32_t row_pos[kWideRows];    // draft row -> RoPE position (pos + 1 + slot)
};
cudaError_t launch_wide_prep(const float *h0, int D, int T, float *X, const WideParams *wp, int n_max,
                             const __half *table, int H, __half *anc, int n_sm, cudaStream_t s);
cudaError_t launch_wide_lnmod(float *X, const float *R, int D, int T, const float *scale, const float *shift, float eps,
                              __half *out, cudaStream_t s);
cudaError_t launch_wide_self_attn(const float *qkv, int D, int B, int n_seqs, int n_heads, __half *out, cudaStream_t s);
cudaError_t launch_wide_argmax(const float2 *part, int n_blocks, int T, const WideParams *wp, cudaStream_t s);
cudaError_t launch_q8_to_f16(const uint8_t *raw, int V, int H, int Vpad, __half *out, cudaStream_t s);
cudaError_t launch_bf16_to_f16_pad(const __nv_bfloat16 *in, int V, int H, int Vpad, __half *out, cudaStream_t s);

// --- the DFlash sequential logit head and confidence (k_seqhead.cu) ---------
struct SeqArgs {
  const float *base;           // [T][V] base logits of the block
  int32_t V, r, k, d;          // vocab, rank, position, draft width
  const __nv_bfloat16 *w1;     // markov.w1 [V][r]
  const __nv_bfloat16 *W;      // markov.w2 or rnn.wO [r][V]
  const float *state;          // RNN: s_k [r]; null: Markov (e1 = w1[prev])
  const StepParams *sp;        // anchor (position 0's prev), tokens, conf, length, thr
  float2 *part;                // [gridDim] per-CTA bests
  int32_t *ticket;             // [1]
  int32_t *flags;              // [0]: decided (pruning ended the block), [1]: length so far
  // confidence
  const __nv_bfloat16 *conf_w, *conf_b;   // [d + r], [1] (null: no confidence head)
  const float *X;              // backbone rows before out_norm [T][d]
  const __nv_bfloat16 *out_norm;
  float eps;
  int32_t T;                   // positions in the block
};
struct RnnArgs {
  const __nv_bfloat16 *w1, *wH, *bH;   // [V][r], [r][r], [r]
  const float *s_in;           // s_{k-1} [r]
  float *s_out;                // s_k [r]
  int32_t r, k;
  const StepParams *sp;
  const int32_t *flags;
};
cudaError_t launch_seq_bias_argmax(const SeqArgs &a, cudaStream_t s);
int seq_grid(int V);
cudaError_t launch_rnn_step(const RnnArgs &a, cudaStream_t s);
cudaError_t launch_seq_init(int32_t *flags, int32_t T, cudaStream_t s);

// --- skinny GEMV: Y[t][m] = sum_k A[t][k] W[m][k] for t < T <= 32 ----------
enum AMode : int32_t {
  A_PLAIN = 0,     // A = X
  A_RMS = 1,       // A = X * w[k] * rsqrt(mean(x^2) + eps)         (RMSNorm)
  A_LNMOD = 2,     // A = (X - mu) * rstd * (1 + scale[k]) + shift[k] (adaLN)
  A_ROW_Q8 = 3,    // A row 0 = dequantised table row sp->anchor (Q8_0)
  A_ROW_BF16 = 4,  // A row 0 = table row sp->anchor (bf16)
  A_RMS2 = 5,      // A = RMSNorm(RMSNorm(X; nw); nw2): stats are (sum x^2, sum (x nw)^2)
};

enum SegKind : int32_t {
  SEG_F32 = 0,     // store f32 rows into Y (optionally head RMSNorm + RoPE)
  SEG_CACHE = 1,   // store f16 into a head-major cache [H][max_ctx][hd] (optionally norm + RoPE)
};

enum EMode : int32_t {
  E_STORE = 0,     // Y = y + b (out stats optional)
  E_GELU = 1,      // Y = gelu_erf(y + b)
  E_RESID = 2,     // Y = R + gate * (y + b)  (gate null -> 1), out stats
  E_SEGS = 3,      // per-segment f32 / cache stores with per-head RMSNorm + RoPE
  E_GEGLU = 4,     // tile = 64 gate rows + 64 up rows: Y[f] = gelu_tanh(g) * u
};

struct SegDesc {
  int32_t kind;                 // SegKind
  int32_t y_col;                // SEG_F32: column offset of the segment in Y
  int32_t rope;                 // apply RoPE after the norm
  int32_t pad;
  const __nv_bfloat16 *norm_w;  // per-head RMSNorm weight [hd] (null = none)
  __half *cache;                // SEG_CACHE: [n_heads][max_ctx][hd]
};

struct GemvArgs {
  const uint8_t *Wt;       // weights tiled [ceil(M/128)][K/64][16 KB]: 128 rows x 64 bf16, pre-swizzled
  int32_t *err;            // raised when a bounded wait gives up
  int32_t M, K, Kc, Kp;    // rows, cols, cols per CTA, cols per staged A piece
  int32_t ksplit;          // CTAs (one cluster) sharing a row tile
  int32_t T_const;         // > 0: fixed T, else sp->T
  const StepParams *sp;

  // prologue
  int32_t amode;
  const float *X;          // input rows X[t * ldx + k] (ldx 0 = one row broadcast)
  int32_t ldx;
  int32_t x_from_sp;       // X = sp->feats
  const float2 *st;        // input row stats: st[i * kMaxT + t] = (mean, M2) of tile i (128 columns), i < st_tiles
  int32_t st_tiles;
  int32_t st_bcast;        // stats of row 0 serve every row
  const __nv_bfloat16 *nw; // RMS weight (A_RMS, first weight of A_RMS2)
  const __nv_bfloat16 *nw2;// A_RMS2 second weight; + (m0 / nw_rows) * K for per-layer weights
  int32_t nw_rows;         // rows sharing one second norm weight (0 = one weight for all)
  const float *sc, *sh;    // A_LNMOD scale / shift [K]
  // A_RMS with two row sources: rows t >= split come from X2 (row t - split)
  // with their own statistics st2 and norm weight nw_alt
  int32_t split;           // 0 = one source
  const float *X2;
  const float2 *st2;
  const __nv_bfloat16 *nw_alt;
  float eps, inv_n;
  const uint8_t *tq8;      // A_ROW_Q8: the table in lm_head layout (see LmArgs)
  const uint8_t *tb;       // A_ROW_BF16: the table in GEMV tile layout

  // epilogue
  int32_t emode;
  const __nv_bfloat16 *bias;  // [M] or null
  float *Y;
  int32_t ldy;
  uint8_t *ylm;               // E_STORE: also write Y as the lm_head operand (kLmYChunk layout), or null
  int32_t ylm_f16;            // 1: f16 hi/lo halves (Q8_0 table), 0: bf16
  float2 *out_st;             // [M / 128][kMaxT] per-tile (mean, M2) of the stored rows, or null
  const __nv_bfloat16 *st_w;  // if set, out_st holds (sum v^2, sum (v st_w)^2) instead
  const float *gate;          // E_RESID gate [M] (null = 1)
  const float *R;             // E_RESID residual source R[t * ldr + m]
  int32_t ldr;
  // E_SEGS
  int32_t seg_rows, n_segs, hd, max_ctx;
  int32_t pos_src;            // 0: sp->pos, 1: sp->start, 2: sp->L, 3: t < split ? sp->start + t : sp->pos
  int32_t pos_add;            // position of row t = base + pos_add + t
  const float2 *rope;         // [positions][hd / 2] (cos, sin)
  float qk_eps;
  SegDesc segs[kMaxSegs];
  float *Y2;                  // E_RESID: a second copy of the stored rows (debug), or null
  int32_t ldy2;
  // self-attention handoff: after the q/k/v segments of a head are stored, the
  // last CTA to finish one computes that head's attention over the T rows.
  int32_t *tickets;           // [n_heads] zero-initialised, self-resetting
  float *attn_out;            // [T][D]
  int32_t self_D;             // width of one of q / k / v (0 = no attention tail)
  float attn_scale;
};

// --- flash-decode cross attention over a head-major f16 cache --------------
struct AttnArgs {
  const float *Q;          // [T][ldq] f32 queries (head h at column h * hd)
  int32_t ldq;
  const __half *Kc, *Vc;   // [n_heads][max_ctx][hd]
  int32_t max_ctx, n_heads, hd;
  int32_t splits;          // CTAs per head (one thread-block cluster, <= 8)
  int32_t T_const;
  int32_t L_src;           // 0: sp->L, 1: sp->pos + 1 (FlashMap keys 0..pos)
  int32_t L_add;
  const StepParams *sp;
  float scale_log2;        // log2(e) / sqrt(hd)
  float *out;              // [T][ldo]
  int32_t ldo;
};

// --- tensor-core attention over the cache, head dim 128 (k_xattn.cu) --------
constexpr int kMaxXSplits = 32;   // key ranges per head
struct XAttnArgs {
  CUtensorMap tm_k, tm_v;  // the K / V planes as [n_heads * max_ctx][128] f16, 128 x 64 boxes
  const float *Q;          // [T][ldq] f32 queries (head h at column h * 128)
  int32_t ldq;
  int32_t max_ctx, n_heads;
  int32_t splits;          // key ranges (CTAs) per head, <= kMaxXSplits
  int32_t T_const;
  int32_t L_src;           // 0: sp->L, 1: sp->pos + 1
  int32_t L_add;
  const StepParams *sp;
  float scale_log2;        // log2(e) / sqrt(128)
  float *out;              // [T][ldo]
  int32_t ldo;
  float *part_o;           // [n_heads][splits][16][128] unnormalised partial outputs
  float2 *part_ml;         // [n_heads][splits][16] (reference m, row sum l)
  int32_t *tickets;        // [n_heads], zero between launches
  int32_t *err;
  // Several sequences in one launch (grid z; null: one sequence, the fields
  // above): launch slot z serves the call's sequence bz_call[z] (its query rows
  // start at bz_call[z] * T_const) over the cache of sequence bz_seq[z], keys
  // 0 .. bz_L[z]-1.  The maps then cover the whole cache, [seqs * layers * 2 *
  // n_heads * max_ctx][128]: K rows of (sequence, layer) from
  // ((seq * n_layers + layer) * 2) * n_heads * max_ctx, V rows n_heads * max_ctx
  // further.  Partials, tickets and the output are per launch slot / call row.
  const int32_t *bz_call, *bz_seq, *bz_L;
  int32_t n_z, layer, n_layers;
  __half *out16;           // f16 output [rows][ldo] instead of out (null: f32 out)
};
cudaError_t launch_xattn(const XAttnArgs &a, int stages, bool cluster, cudaStream_t st, bool pdl);
size_t xattn_smem_bytes(int stages);
int xattn_max_active_clusters(int cluster, int n_heads);
bool make_cache_map(CUtensorMap *map, const __half *plane, int n_heads, int max_ctx);

// --- lm_head GEMV fused with the per-row argmax -----------------------------
// Q8_0 table layout: per (128-row tile, 64-column chunk) one contiguous 8704-byte
// block: 128 rows x 64 int8 (pre-swizzled, q8_slot) then the two 32-column
// blocks' f16 scales [2][128].  bf16 table: the GEMV tile layout.
constexpr int kQ8Chunk = kTile * 64 + 2 * kTile * 2;
// lm_head operand rows of Y: per 64 columns one 32-row x 128-byte block in the
// 128-byte-swizzle K-major layout; slot t has its hi half in row lm_yrow(t) and
// its lo half 8 rows further (f16 halves for the Q8_0 table, bf16 for bf16).
constexpr int kLmYChunk = 32 * 128;
struct LmArgs {
  const uint8_t *q8;         // Q8_0 table (layout above) or null
  const uint8_t *wb;         // bf16 table (GEMV tile layout) or null
  int32_t *err;
  int32_t V, H;
  int32_t T_const;
  const StepParams *sp;
  const float *Y;            // [T][H]
  int32_t ldy;
  const uint8_t *ylm;        // Y already split into the resident operand layout (kLmYChunk per 64 columns), or null
  float2 *part;              // [gridDim.x][kMaxT] (value, index-as-float bits)
  int32_t *ticket;           // [1]
  int32_t *tokens;           // [T]; null: sp->tokens
  float *logits;             // optional [T][V] store (debug, or the output of a Q8_0 linear layer)
  // Q8_0 with a pre-split Y only: a linear layer split along K into slices of H columns,
  // the table's tiles in slice order (y_slice_tiles tiles each) and Y holding every
  // slice's chunks in turn; the row v of tile t is slice t / y_slice_tiles's partial
  // sum (0: no split)
  int32_t y_slice_tiles;
};

// --- the persistent draft step (k_step.cu) -----------------------------------
// One launch runs a program of phases separated by grid-wide barriers, on
// clusters of kStepCS CTAs (one CTA per SM).  In a linear phase the 128-row
// weight tiles are dealt to clusters: tile i goes to cluster
// ((i % map_mod) + rot) % n_clusters.  Rank r of a cluster takes the same K
// slice [r cpt / kStepCS, (r + 1) cpt / kStepCS) of every tile its cluster
// owns, so it stages that slice of the activations once; the partial tiles
// meet through distributed shared memory and rank r finishes rows r and
// r + kStepCS of every tile (the fused epilogue).
constexpr int kStepCS = 8;          // CTAs per cluster
constexpr int kStepMaxTiles = 6;    // tiles one cluster may own in a phase
enum StepPrologue : int32_t { SP_NONE = 0, SP_SELF_ATTN = 1 };
enum StepTail : int32_t { ST_NONE = 0, ST_CROSS_ATTN = 1 };

struct StepAttn {
  int32_t max_ctx, n_heads, hd;
  int32_t L_src;              // cross keys: 0: sp->L, 1: sp->pos + 1 (plus L_add)
  int32_t L_add;
  float scale;                // 1 / sqrt(hd)
  float scale_log2;           // log2(e) / sqrt(hd)
  int32_t ldo;
  const __half *Kc, *Vc;      // cross: head-major caches [n_heads][max_ctx][hd]
  const float *Q;             // cross: queries [T][ldq] (head h at column h * hd)
  int32_t ldq;
  int32_t D;                  // self: width of each of q / k / v
  const float *qkv;           // self: [T][3 D] rows (q, k, v)
  float *out;                 // cross: attention rows [T][ldo]
};

struct StepPhase {
  GemvArgs g;
  int32_t cpt;        // chunks per tile (K / 64)
  int32_t ntiles;
  int32_t map_mod;    // tile i -> cluster ((i % map_mod) + rot) % n_clusters
  int32_t rot;
  int32_t prologue;   // StepPrologue: SP_SELF_ATTN forms the activations as the block self-attention of q/k/v
  int32_t tail;       // StepTail: ST_CROSS_ATTN attends the cluster's heads over the cache after the epilogue
  int32_t pad[2];
  StepAttn at;
};

struct StepArgs {
  const StepPhase *ph;
  int32_t n_phases;
  int32_t T;
  int32_t n_clusters;
  const StepParams *sp;
  uint32_t *bar;       // [0]: arrivals, [32]: generation (separate cache lines)
  int32_t *err;
  uint64_t *trace;     // null, or [n_phases][gridDim][kStepTraceSlots] globaltimer stamps (ns)
};
// trace slots per (phase, CTA): 0 workers start the phase (barrier passed),
// 1 staging done, 2 phase done (arrive), 3 the producer issued the phase's last
// copy, 4 the MMA warp committed the phase's last tile, 5 partials published,
// 6 epilogues done
constexpr int kStepTraceSlots = 8;

// the cluster that owns tile i of a phase
__host__ __device__ __forceinline__ int step_cluster_of(const StepPhase &P, int i, int ncl) {
  return ((i % P.map_mod) + P.rot) % ncl;
}
// chunk range of rank r in every tile: [step_klo(r), step_klo(r + 1))
__host__ __device__ __forceinline__ int step_klo(int r, int cpt) { return r * cpt / kStepCS; }

size_t step_smem_bytes();
// attrs: bit 0 = cooperative launch, bit 1 = programmatic stream serialisation
cudaError_t launch_step(const StepArgs &a, int clusters, cudaStream_t s, int attrs);
int step_max_clusters();   // clusters of the step kernel the device holds at once

// launchers (return cudaError_t of the launch)
cudaError_t launch_gemv(const GemvArgs &a, int n_tiles, cudaStream_t s, bool pdl);
size_t gemv_smem_bytes(const GemvArgs &a, int mt);
cudaError_t launch_attn(const AttnArgs &a, int L_now, cudaStream_t s, bool pdl);
cudaError_t launch_lmhead(const LmArgs &a, int grid, cudaStream_t s, bool pdl);
int lmhead_grid(const LmArgs &a, int n_sm);
// The static scratch of the lm_head entry point that allocates nothing: the
// largest grid it holds, and its ticket / partial-best pointers on the current
// device (the first call per device resolves the address and zeroes the ticket).
int lmhead_static_max_grid();
cudaError_t lmhead_static_scratch(int grid, float2 **part, int32_t **ticket, cudaStream_t st);

// set-up and small kernels
cudaError_t launch_q8_repack(const uint8_t *raw, int32_t V, int32_t H, uint8_t *dst, cudaStream_t s);
size_t q8_table_bytes(int32_t V, int32_t H);
cudaError_t launch_colmean_q8(const uint8_t *raw, int32_t V, int32_t H, float *out, cudaStream_t s);
cudaError_t launch_colmean_bf16(const __nv_bfloat16 *w, int32_t V, int32_t H, float *out, cudaStream_t s);
cudaError_t launch_rope_table(float2 *tab, int32_t n_pos, int32_t hd, float theta, cudaStream_t s);
cudaError_t launch_transpose_bf16(const __nv_bfloat16 *in, int32_t rows, int32_t cols, __nv_bfloat16 *out,
                                  int32_t ldo, cudaStream_t s);
cudaError_t launch_block_consts(const __nv_bfloat16 *mask_emb, const __nv_bfloat16 *block_pos, int32_t gamma,
                                int32_t d, float *out, float2 *st, cudaStream_t s);
cudaError_t launch_row_stats(const float *x, int32_t rows, int32_t d, float2 *st, cudaStream_t s);
cudaError_t launch_accept(int32_t n, int32_t block, const int32_t *draft, const int32_t *target,
                          const int32_t *k, int32_t *acc, int32_t *bonus, cudaStream_t s);
cudaError_t launch_wait_selftest(int32_t *err, long long budget_cycles, cudaStream_t s);
cudaError_t launch_time_embed(float *e, int32_t time_dim, double time_scale, double time, cudaStream_t s);
cudaError_t launch_setup_linear(const __nv_bfloat16 *W, const __nv_bfloat16 *b, const float *x, const float *x2,
                                int32_t M, int32_t N, int32_t act, float *y, cudaStream_t s);
cudaError_t launch_fill_f32(float *p, size_t n, float v, cudaStream_t s);
// [M][K] bf16 row-major -> GEMV tile layout (zero rows past M)
cudaError_t launch_tile_weights(const __nv_bfloat16 *src, int32_t M, int32_t K, uint8_t *dst, cudaStream_t s);
size_t tiled_bytes(int32_t M, int32_t K);

}  // namespace fm
