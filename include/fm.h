/*
 * fm.h -- C ABI of libfm.so, a GB300 (sm_103a) implementation of the forward
 * pass of a block-parallel speculative-decoding drafter of the FlashMap /
 * DFlash kind.  One process, one GPU; every compute step runs in the
 * library's own CUDA kernels.
 *
 * Sources (page title, file, section):
 *   [FM]  diskformer 0.5.4 -> 0.6.6, package/engines/flashmap_drafter.js
 *   [MTP] diskformer 0.5.3 -> 0.6.4, package/engines/ternary_bonsai_2_mtp.js
 *   [DF]  mlx-bun 0.4.0 -> 1.0.0, package/src/spec/dspark/module-dflash.ts
 *
 * Conventions
 *   - Pointers named *_dev are device pointers; *_host are host pointers.
 *     "stream" is a cudaStream_t passed as void* (NULL = legacy stream).
 *   - Every call checks its arguments on the host before it launches anything
 *     and returns an fm_status; nothing aborts and no C++ exception crosses the
 *     ABI.  On failure fm_last_error(h) holds a one-line reason.
 *   - All device work is ordered on the given stream; no call synchronises the
 *     host except fm_debug_copy (it copies to host memory), fm_synchronize and
 *     fm_create.
 *   - A handle is not thread-safe: one host thread at a time per handle.
 */
#ifndef FM_H_
#define FM_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FM_ABI_VERSION 1

/* exported from libfm.so; everything else in the library is hidden */
#if defined(__GNUC__)
#define FM_API __attribute__((visibility("default")))
#else
#define FM_API
#endif

typedef enum fm_status {
  FM_OK = 0,
  FM_ERR_INVALID_ARG = 1,   /* a null/misaligned pointer, a size or index out of range, a bad tensor */
  FM_ERR_UNSUPPORTED = 2,   /* a configuration the kernels do not handle (see fm_config) */
  FM_ERR_OOM = 3,           /* a device or pinned-host allocation failed */
  FM_ERR_CONTEXT_FULL = 4,  /* start + n_rows + block + 1 > max_ctx ([FM] extendContext's check) */
  FM_ERR_STATE = 5,         /* the call does not fit the sequence state (pos != length, start > length) */
  FM_ERR_CUDA = 6,          /* a CUDA runtime error; fm_last_error has the CUDA message */
  FM_ERR_TIMEOUT = 7        /* a bounded device-side wait gave up (reported, never hung) */
} fm_status;

/* fm_config.variant */
#define FM_VARIANT_FLASHMAP 0 /* adaLN DiT drafter with context injection [FM] */
#define FM_VARIANT_DFLASH 1   /* KV-injection drafter, Eq 2 / Eq 3 [DF] */

/* fm_config.lm_format: storage of the tied token table E [vocab][target_dim] */
#define FM_LM_BF16 0
#define FM_LM_Q8_0 1 /* GGUF Q8_0: per 32 values a little-endian f16 scale then 32 int8 (34 bytes) [MTP] */

/* fm_tensor.dtype */
#define FM_DTYPE_BF16 0
#define FM_DTYPE_Q8_0 1
#define FM_DTYPE_F32 2

typedef struct fm_config {
  int32_t variant;     /* FM_VARIANT_* */
  int32_t dim;         /* draft width D (multiple of 128) */
  int32_t n_heads;     /* D = n_heads * head_dim */
  int32_t head_dim;    /* 64 or 128 */
  int32_t n_layers;    /* DiT / backbone layers (1..64) */
  int32_t ff_dim;      /* MLP width (multiple of 128) */
  int32_t block;       /* draft slots: 16 for [FM], gamma for [DF]; 1..16 */
  int32_t target_dim;  /* the target's hidden width Ht (multiple of 64) */
  int32_t n_taps;      /* tapped target layers; feature rows are n_taps * target_dim wide */
  int32_t vocab;       /* rows of the token table */
  int32_t lm_format;   /* FM_LM_* */
  int32_t max_ctx;     /* cache rows per sequence (positions 0 .. max_ctx-1) */
  int32_t max_seqs;    /* independent sequences the handle holds caches for (>= 1) */
  float rope_theta;    /* RoPE base ([FM] CFG.theta) */
  float ln_eps;        /* adaLN LayerNorm eps ([FM] CFG.lnEps) */
  float rms_eps;       /* RMSNorm eps ([FM] CFG.rmsEps; [DF] the target's eps) */
  float qk_eps;        /* per-head q/k RMSNorm eps ([FM] CFG.qkEps) */
} fm_config;

/*
 * One named weight.  Names, shapes and layouts ([out][in] for [FM], [in][out]
 * for [DF]) are those of the drafter checkpoints:
 *   [FM]: fc.weight, hidden_norm.weight, anchor_proj.{weight,bias},
 *         anchor_norm.weight, state_norm.weight, x_embed.{weight,bias},
 *         layers.{l}.{self_attn,cross_attn}.{q,k,v,o}_proj.weight,
 *         layers.{l}.{self_attn,cross_attn}.{q,k}_norm.weight,
 *         layers.{l}.mlp.fc{1,2}.{weight,bias}, head.{weight,bias},
 *         token_embd.weight (the tied table; FM_DTYPE_Q8_0 or FM_DTYPE_BF16).
 *         A missing bias is read as zero.
 *   [DF]: bb.{i}.{attn_norm,q,k,v,o,ff_norm,gate,up,down}, W_c, ctx_norm,
 *         tok_proj, mask_emb, block_pos, out_norm, out_proj, token_embd.weight.
 * data is host memory (on_device = 0) or device memory (on_device = 1); the
 * library copies (and repacks) every tensor during fm_create, so the caller may
 * free it when fm_create returns.  nbytes must equal the tensor's size.
 */
typedef struct fm_tensor {
  const char *name;
  const void *data;
  int64_t nbytes;
  int32_t dtype;      /* FM_DTYPE_* */
  int32_t on_device;  /* 0 host, 1 device */
} fm_tensor;

typedef struct fm_handle fm_handle;

/*
 * fm_create -- take the configuration and the weights, build the device state
 * ([FM] FlashMapDrafter.load / upload / init; [DF] DflashDrafter.load).
 *   modulation_host: [FM] the adaLN table [(3*n_layers+1) * 3 * dim] f32 in
 *     blocks [scale dim | shift dim | gate dim] for (self, cross, mlp) of every
 *     layer and the final norm ([FM] timeConditioning output, e.g. from
 *     fm_time_conditioning); host or device memory; NULL for [DF].
 *   On success *out owns: the repacked weights, per-sequence caches of max_ctx
 *   rows, work buffers, and the constant start row h0 = x_embed(state_norm(
 *   mean row of E)) ([FM] init).  Synchronises the stream before returning.
 * Errors: FM_ERR_INVALID_ARG (null pointer, unknown/missing/mis-sized tensor,
 *   wrong dtype), FM_ERR_UNSUPPORTED (dims outside the limits above), FM_ERR_OOM,
 *   FM_ERR_CUDA.  *out is NULL on failure.
 */
FM_API fm_status fm_create(const fm_config *cfg, const fm_tensor *weights, int32_t n_weights,
                    const float *modulation_host, void *stream, fm_handle **out);

/*
 * fm_time_conditioning -- the adaLN table fm_create takes for [FM], computed
 * from the checkpoint's time-conditioning linears for the jump s -> t of the
 * flow map ([FM] timeConditioning; the page drafts with s = 0, t = 1):
 *   e(x) = [cos a_i | sin a_i], a_i = x * time_scale * exp(-ln(10000) i / half),
 *   half = time_dim / 2 ([FM] CFG.timeDim, CFG.timeScale);
 *   ts = time_embed.linear_2(SiLU(time_embed.linear_1(e(s)))), tj likewise with
 *   jump_embed and e(t); cond = SiLU(ts + tj), SiLU(x) = x / (1 + exp(-x));
 *   block n of the table = adaLN linear n of cond, n over
 *   layers.{l}.{self_attn_adaln,cross_attn_adaln,mlp_adaln}.linear then
 *   final_adaln.linear, each [scale dim | shift dim | gate dim].
 * weights: bf16 tensors (host or device) time_embed.linear_{1,2}.{weight,bias},
 *   jump_embed.linear_{1,2}.{weight,bias} (linear_1 [cond_dim][time_dim],
 *   linear_2 [cond_dim][cond_dim]) and every adaLN linear .weight
 *   [3 dim][cond_dim] / .bias [3 dim]; a missing bias is read as zero.  Other
 *   tensors in the list are ignored, so the full checkpoint list may be passed.
 * table_dev: device f32 [(3 n_layers + 1) * 3 * dim], caller-owned; pass it to
 *   fm_create as the modulation table (device memory is accepted there).
 * Set-up: allocates temporary device buffers and synchronises the stream.
 * Errors: FM_ERR_INVALID_ARG (null or misaligned pointer, odd time_dim,
 *   missing / mis-sized tensor, not [FM]), FM_ERR_OOM, FM_ERR_CUDA; the reason
 *   is in fm_last_error(NULL).
 */
FM_API fm_status fm_time_conditioning(const fm_config *cfg, const fm_tensor *weights, int32_t n_weights,
                                      int32_t time_dim, int32_t cond_dim, float time_scale, float s, float t,
                                      float *table_dev, void *stream);

/*
 * fm_context_append -- context injection ([FM] extendContext; [DF] Eq 2 and
 * projectContextRows): the target's tapped feature rows feats_dev
 * [n_rows][n_taps * target_dim] f32 (device, row-major, 16-byte aligned)
 * become cache rows start_pos .. start_pos + n_rows - 1 of sequence seq.
 *   [FM]: c = fc(f); cn = RMSNorm(c; hidden_norm); per layer k = RoPE(k_norm(
 *         k_proj cn)) at the row's position, v = v_proj cn; stored as f16.
 *   [DF]: H = RMSNorm(f W_c; ctx_norm); per layer K = attn_norm(H) W_k,
 *         V = attn_norm(H) W_v; stored as f16.
 * start_pos <= length is required; writing below the length rewinds (the
 * verify step re-appends from the anchor slot).  Afterwards length =
 * start_pos + n_rows.  n_rows may be 0 (only moves the length).
 * Errors: FM_ERR_INVALID_ARG (seq out of range, n_rows < 0, null feats with
 *   n_rows > 0), FM_ERR_STATE (start_pos > length or < 0),
 *   FM_ERR_CONTEXT_FULL (start_pos + n_rows + block + 1 > max_ctx), FM_ERR_CUDA.
 */
FM_API fm_status fm_context_append(fm_handle *h, int32_t seq, const float *feats_dev, int32_t n_rows,
                            int32_t start_pos, void *stream);

/*
 * fm_context_append_batched -- fm_context_append for several sequences in one
 * call.  Dense appends (>= 128 rows) run one after another through the
 * tensor-core prefill.  The shorter appends of 4 or more sequences, on a
 * FlashMap handle with max_seqs >= 2 and head_dim 128, share each weight
 * read: all their rows go through one fc GEMM and one K/V GEMM (per-row
 * sequence and position), in chunks of at most 16384 rows; otherwise each
 * runs on its sequence's own stream, concurrently (each reading the weights
 * itself).  feats_dev holds the rows of seq_ids[0], then seq_ids[1], ...;
 * n_rows_host[i] and start_host[i] are per sequence (host arrays of n_seqs).
 * Same checks per sequence; nothing is launched if any check fails.
 * Sequence ids must be distinct.  Batched calls on one handle run in stream
 * order on one stream (they share the handle's batched-pass buffers).
 */
FM_API fm_status fm_context_append_batched(fm_handle *h, int32_t n_seqs, const int32_t *seq_ids_host,
                                    const float *feats_dev, const int32_t *n_rows_host,
                                    const int32_t *start_host, void *stream);

/*
 * fm_draft -- draft `block` tokens after each anchor ([FM] draft; [DF]
 * forwardRows with the greedy argmax).  For sequence seq_ids[i] the anchor
 * token anchors[i] sits at position pos[i], which must equal that sequence's
 * length.  [FM] writes the anchor's own context slot (cache row pos) as the
 * page does; the length is unchanged (a later append from pos overwrites it).
 * tokens_dev: device int32 [n_seqs][block], written in stream order.
 * Host arrays: seq_ids, anchors, pos (n_seqs each; distinct seq ids).
 * Four or more sequences on a FlashMap handle with max_seqs >= 2 and
 * head_dim 128 draft together, in passes of up to 32: each pass runs every
 * product over all the pass's slot rows as one tensor-core GEMM (f16
 * operands), so each weight and the token table are read once per pass, and
 * one attention launch per layer serves every sequence's cache.  Fewer
 * sequences, or other handles, run one chain per sequence on the sequences'
 * own streams.
 * Errors: FM_ERR_INVALID_ARG (anchor outside [0, vocab), bad seq id, n_seqs
 *   outside [1, max_seqs], null tokens), FM_ERR_STATE (pos != length),
 *   FM_ERR_CONTEXT_FULL (pos + block + 1 > max_ctx), FM_ERR_CUDA.
 */
FM_API fm_status fm_draft(fm_handle *h, int32_t n_seqs, const int32_t *seq_ids_host, const int32_t *anchors_host,
                   const int32_t *pos_host, int32_t *tokens_dev, void *stream);

/*
 * Host-buffer forms of the three calls above, for callers whose feature rows
 * arrive in, and whose drafted tokens go to, host memory.  Each copies on the
 * stream with cudaMemcpyAsync: the rows into a handle-owned device staging
 * buffer (grown when a call needs more; it waits for the previous
 * host-buffer call's work before it is reused), then runs the device-pointer
 * call, whose checks, behaviour and errors it shares; fm_draft_host then
 * copies the tokens back.  With pinned host memory every copy is
 * asynchronous to the host: the rows must stay unchanged, and tokens_host
 * must not be read, until the stream has passed the call (fm_synchronize).
 * With pageable memory the runtime makes the copies synchronous instead.
 *   feats_host: host f32 rows laid out as in the device-pointer call (no
 *     alignment requirement).
 *   tokens_host: host int32 [n_seqs][block].
 * Errors: those of the device-pointer call; FM_ERR_INVALID_ARG (null
 *   feats_host with rows, null tokens_host); FM_ERR_OOM (the staging buffer
 *   could not grow); FM_ERR_CUDA (a copy failed).
 */
FM_API fm_status fm_context_append_host(fm_handle *h, int32_t seq, const float *feats_host, int32_t n_rows,
                                        int32_t start_pos, void *stream);
FM_API fm_status fm_context_append_batched_host(fm_handle *h, int32_t n_seqs, const int32_t *seq_ids_host,
                                                const float *feats_host, const int32_t *n_rows_host,
                                                const int32_t *start_host, void *stream);
FM_API fm_status fm_draft_host(fm_handle *h, int32_t n_seqs, const int32_t *seq_ids_host,
                               const int32_t *anchors_host, const int32_t *pos_host, int32_t *tokens_host,
                               void *stream);

/*
 * fm_draft_pruned -- [DF] the greedy draft of one sequence through the
 * sequential logit head, with the confidence head and confidence pruning
 * (module-dflash.ts: ``#markov`` (Eq 5), ``#rnn`` (Eq 6), ``#confidence`` and
 * the pruning of Alg 1 in ``forwardRows``).  Needs weights that hold
 * markov.w1 [V][r] (r <= 512, vocab % 8 == 0) and markov.w2 [r][V], or the RNN
 * head (rnn.wH [r][r], rnn.bH [r], rnn.wO [r][V]); conf.w [dim + r] and
 * conf.b [1] for conf_dev and any threshold.  With such weights fm_draft also
 * drafts through the sequential head (no pruning).
 * Position k (prev = anchor for k = 0, else token k - 1; e1 = markov.w1[prev]):
 *   Markov bias = e1 markov.w2; RNN s_k = tanh(s_{k-1} rnn.wH + e1 + rnn.bH),
 *   s_{-1} = 0, bias = s_k rnn.wO;  token_k = argmax(base logits_k + bias),
 *   ties to the lower index;  conf_k = sigmoid([out_norm(row k), e1] conf.w
 *   + conf.b).
 * Pruning: the threshold of position k is thresholds_host[k] (host float
 * [block], or NULL) unless that is NaN, else min_conf (NaN: none), as the
 * page's per-position lookup falls back to its uniform override.  The block ends at the
 * first k >= 1 with conf_k below its threshold (length = k).  Entries
 * 0 .. min(length, block - 1) of tokens_dev and conf_dev are written (the
 * cut position's own, whose confidence decided the cut, included); later
 * positions are not drafted and their entries are left as they were.
 * tokens_dev: device int32 [block]; conf_dev: device float [block] or NULL;
 * length_dev: device int32 [1] or NULL, the positions kept (block without
 * pruning).  All written in stream order.  Same argument checks as fm_draft;
 * FM_ERR_UNSUPPORTED without a sequential head, or without a confidence head
 * when conf_dev or a threshold is given.
 */
FM_API fm_status fm_draft_pruned(fm_handle *h, int32_t seq, int32_t anchor, int32_t pos,
                                 const float *thresholds_host, float min_conf, int32_t *tokens_dev,
                                 float *conf_dev, int32_t *length_dev, void *stream);

/*
 * fm_accept -- greedy acceptance ([FM] specGenerate verify step; [MTP] the
 * same rule): n_accepted = the longest prefix i < k with draft[i] == target[i];
 * bonus = target[n_accepted].  draft_host has k entries, target_host k + 1.
 * Pure host function.  Errors: FM_ERR_INVALID_ARG (null pointer, k < 0).
 */
FM_API fm_status fm_accept(const int32_t *draft_host, const int32_t *target_host, int32_t k, int32_t *n_accepted,
                    int32_t *bonus);

/*
 * fm_accept_batched -- fm_accept for n_seqs sequences on the device:
 * draft_dev [n_seqs][block], target_dev [n_seqs][block + 1], k_dev [n_seqs]
 * (each clamped to [0, block]); writes n_accepted_dev[n_seqs], bonus_dev[n_seqs].
 * Errors: FM_ERR_INVALID_ARG (null pointer, n_seqs < 1), FM_ERR_CUDA.
 */
FM_API fm_status fm_accept_batched(fm_handle *h, int32_t n_seqs, const int32_t *draft_dev, const int32_t *target_dev,
                            const int32_t *k_dev, int32_t *n_accepted_dev, int32_t *bonus_dev, void *stream);

/*
 * fm_lm_head_argmax_noalloc -- fm_draft's fused lm_head + per-row argmax on
 * rows the caller supplies: tokens[t] = argmax_v sum_k y[t][k] E[v][k]
 * (ties -> lowest v) over the handle's token table E.  The paper has no
 * counterpart to this entry point.  It is for callers that may not allocate
 * device memory while they run -- a serving loop whose memory is all handed
 * out up front by its own pool, or code running where cudaMalloc would stall
 * the device or could fail under memory pressure.  It allocates nothing: the
 * cross-CTA partial bests and the completion ticket live in a fixed 64 KB
 * block of static device memory inside the library, which every GPU that
 * loads the library keeps until the process exits.  That block holds at
 * most 255 CTAs of partials; larger grids are rejected with
 * FM_ERR_UNSUPPORTED.  The first call on a device looks up the block's
 * address and zeroes the ticket on the stream, so make that first call
 * before any stream capture.  Every call shares the block: calls that
 * overlap on the GPU (other streams, other handles on the same device) race
 * and must be serialised by the caller.
 * y_dev: device f32 [n_rows][target_dim], row-major, 16-byte aligned.
 * tokens_dev: device int32 [n_rows], 4-byte aligned, written in stream
 * order.  Both stay owned by the caller.  The handle's device must be the
 * current device.
 * Errors: FM_ERR_INVALID_ARG (null or misaligned pointer, n_rows outside
 *   1..16, the current device is not the handle's), FM_ERR_UNSUPPORTED (grid
 *   beyond the static block), FM_ERR_CUDA.  A device-side bounded wait that
 *   gives up inside the kernel is reported late: the call has already
 *   returned FM_OK, tokens_dev is then undefined, and the next
 *   fm_synchronize (or fm_debug_copy) on the handle returns FM_ERR_TIMEOUT.
 */
FM_API fm_status fm_lm_head_argmax_noalloc(fm_handle *h, const float *y_dev, int32_t n_rows, int32_t *tokens_dev,
                                    void *stream);

/*
 * fm_synchronize -- wait for the work on stream, then report whether a
 * device-side bounded wait gave up in any call since the last check (a wait
 * that exceeds its clock budget raises an error word on the device and its
 * kernel returns instead of hanging).  Clears the word.
 * Errors: FM_ERR_TIMEOUT (a wait gave up: the outputs of those calls are
 *   undefined; the handle stays usable), FM_ERR_CUDA, FM_ERR_INVALID_ARG.
 */
FM_API fm_status fm_synchronize(fm_handle *h, void *stream);

/*
 * fm_selftest_wait_timeout -- exercise the failure path of the bounded waits:
 * launches one CTA whose mbarrier wait can never complete, with a budget of
 * budget_us microseconds (1 .. 1e6); the wait gives up, raises the handle's
 * device error word and the kernel returns.  A following fm_synchronize
 * returns FM_ERR_TIMEOUT.  Nothing hangs and nothing faults.
 * Errors: FM_ERR_INVALID_ARG (budget out of range), FM_ERR_CUDA.
 */
FM_API fm_status fm_selftest_wait_timeout(fm_handle *h, int32_t budget_us, void *stream);

/*
 * The verify-length and fallback policy of the speculative loop ([FM]
 * specGenerate): a caller-owned record and four host functions, no device
 * work.  Per step of the loop fm_policy_next says whether to run a draft round
 * verifying k drafts (FM_ACT_ROUND), a step of a plain-decoding stretch
 * (FM_ACT_PLAIN: report it with fm_policy_after_plain), or a plain step at the
 * drafter's context limit (FM_ACT_PLAIN_LIMIT: position + 2 block + 2 >
 * max_ctx; no statistics).  After a round, fm_policy_after_round takes the
 * accepted count and the round's time.
 *   k: adaptive (verify = 0): block when the acceptance average >= 5, else 7;
 *      fixed: min(block, verify).
 *   averages: acceptance 0.6 / 0.4 (starts at 4), tokens per round
 *      0.75 / 0.25 of accepted + 1 (starts at 5), round time 0.6 / 0.4 (the
 *      first round after a stretch whose rows were handed to the drafter is left
 *      out), plain-step time 0.7 / 0.3 (starts at 30 ms).
 *   fallback: from the fourth round on, when tokens per round x plain-step time
 *      < 0.85 x round time, a plain stretch of probe_every steps starts (then
 *      one round probes again).
 * Errors: FM_ERR_INVALID_ARG (null pointer, block < 1, verify < 0,
 *   probe_every < 1, accepted < 0, a plain report outside a stretch).
 */
typedef struct fm_verify_policy {
  int32_t block, verify, fallback, probe_every;
  double ema;          /* acceptance average */
  double ema_tokens;   /* tokens-per-round average */
  double round_ms;     /* round-time average, < 0 until the first round */
  double step_ms;      /* plain-step time average */
  int32_t plain_left;  /* steps left in the current plain stretch */
  int32_t rounds;      /* rounds so far */
  int32_t catch_up;    /* the next round's time is left out of the average */
  int32_t pad;
} fm_verify_policy;
#define FM_ACT_ROUND 0
#define FM_ACT_PLAIN 1
#define FM_ACT_PLAIN_LIMIT 2
FM_API fm_status fm_policy_init(fm_verify_policy *p, int32_t block, int32_t verify, int32_t fallback,
                                int32_t probe_every);
FM_API fm_status fm_policy_next(const fm_verify_policy *p, int32_t position, int32_t max_ctx, int32_t *action,
                                int32_t *k);
FM_API fm_status fm_policy_after_round(fm_verify_policy *p, int32_t accepted, double ms);
FM_API fm_status fm_policy_after_plain(fm_verify_policy *p, double ms, int32_t rows_handed);

/* fm_debug_copy selectors ([FM] readOut / peek: look at working buffers) */
#define FM_DEBUG_HIDDEN 0   /* index = layer: the block's hidden rows after that layer [block][dim] f32 (last draft) */
#define FM_DEBUG_HEAD_OUT 1 /* the head output Y [block][target_dim] f32 (last draft of seq) */
#define FM_DEBUG_LOGITS 2   /* logits [block][vocab] f32 of the last draft's Y, recomputed without argmax */
#define FM_DEBUG_CACHE_K 3  /* index = layer: cache K of seq, [n_heads][max_ctx][head_dim] as f16 bits */
#define FM_DEBUG_CACHE_V 4  /* index = layer: cache V, same layout */
#define FM_DEBUG_H0 5       /* [FM] the constant start row h0 [dim] f32 */
#define FM_DEBUG_STEP_TRACE 6 /* [FM] persistent step trace of the last traced draft: u64 [phases][CTAs][8]
                                 (CTAs = the step's clusters x 8) globaltimer ns: 0 phase start, 1 staged,
                                 2 done, 3 last copy issued, 4 last MMA committed, 5 partials published,
                                 6 epilogues done; 0 = no event */

/*
 * fm_debug_copy -- copy nbytes of the selected buffer, starting at byte
 * offset, to dst_host.  Synchronises the stream.  After a batched draft,
 * FM_DEBUG_HEAD_OUT and FM_DEBUG_LOGITS read the sequence's rows of the last
 * pass of the last batched call (the logits recomputed by the batched
 * lm_head's product); a sequence of an earlier pass, or of an earlier batched
 * call, has no kept head output until its next draft (FM_ERR_UNSUPPORTED).
 * FM_DEBUG_HIDDEN is kept by single-sequence drafts only.
 * Errors: FM_ERR_INVALID_ARG (unknown selector, index or range outside the
 * buffer), FM_ERR_UNSUPPORTED (above), FM_ERR_CUDA, FM_ERR_TIMEOUT (a bounded
 * wait gave up in an earlier call).
 */
FM_API fm_status fm_debug_copy(fm_handle *h, int32_t what, int32_t seq, int32_t index, int64_t offset, void *dst_host,
                        int64_t nbytes, void *stream);

/* fm_set_debug flags */
#define FM_DEBUG_KEEP_HIDDEN 1 /* keep every layer's block hidden rows for FM_DEBUG_HIDDEN (adds copies) */
#define FM_DEBUG_PROFILE 2     /* bracket every kernel launch with CUDA events (serialises the chain) */
#define FM_DEBUG_TRACE 4       /* record per-phase timestamps of the persistent draft step (FM_DEBUG_STEP_TRACE) */

/* Debug switches for later calls (0 = the plain hot path).  Errors: FM_ERR_INVALID_ARG. */
FM_API fm_status fm_set_debug(fm_handle *h, int32_t flags);

/* Per-kernel timings gathered while FM_DEBUG_PROFILE is set: one entry per
 * kernel name, with the launches, their summed device time and the summed
 * algorithmic bytes they move (weights once, activations once); for the
 * tensor-core GEMMs (names containing "gemm") the field holds their summed
 * floating-point operations instead (2 M N K each).  Reading synchronises the
 * stream of the recorded launches and resets the record.
 * Errors: FM_ERR_INVALID_ARG (null pointers, cap < 0), FM_ERR_CUDA. */
typedef struct fm_kernel_time {
  char name[32];
  int32_t launches;
  float ms;
  double bytes;
} fm_kernel_time;
FM_API fm_status fm_profile_read(fm_handle *h, fm_kernel_time *out, int32_t cap, int32_t *n);

/* Current context length of a sequence.  Errors: FM_ERR_INVALID_ARG. */
FM_API fm_status fm_get_length(const fm_handle *h, int32_t seq, int32_t *length);

/* Device bytes the handle holds ([FM] gpuBytes). */
FM_API fm_status fm_memory_bytes(const fm_handle *h, int64_t *bytes);

/* Kernel launches issued by the last fm_context_append / fm_draft / batched call. */
FM_API fm_status fm_last_launch_count(const fm_handle *h, int32_t *count);

FM_API const char *fm_status_str(fm_status s);
FM_API const char *fm_last_error(const fm_handle *h);   /* never NULL; "" when no error; NULL h: the last failed
                                                            fm_create / fm_time_conditioning on this thread */

/* Free everything the handle owns.  NULL is ignored. */
FM_API void fm_destroy(fm_handle *h);

/* ------------------------------------------------------------------------
 * The MTP draft head ([MTP] ternary_bonsai_2_mtp.js: the header's graph,
 * MCFG, MTPHead.forward and its kernels, MTPRunner's draft loop): one
 * Qwen-style decoder layer with Q8_0 weights, chained in depth.  A second
 * drafter, with its own handle.
 *
 * One pass over M <= max_rows rows (tokens x at positions pos0 .. pos0+M-1,
 * each with h, the normed hidden of its previous position):
 *   Xc = [rms(E[x]; enorm) | rms(h; hnorm)];  X = eh_proj Xc
 *   A = rms(X; attn_norm);  [q | gate] per q head = attn_q A;  k, v = attn_k A, attn_v A
 *   per head RMSNorm over head_dim (attn_q_norm / attn_k_norm), NEOX RoPE on the
 *   first rot_dims (pairs i, i + rot_dims/2, angle pos * theta^(-2i/rot_dims));
 *   k, v rows stored in the head's own f32 cache at their positions
 *   O = softmax(q k^T / sqrt(head_dim)) v over cache rows kv_lo .. pos (KV head
 *   h / (n_heads / n_kv_heads)), times sigmoid(gate)
 *   X += attn_output O;  X += ffn_down(silu(ffn_gate A') * ffn_up A'), A' = rms(X; post_attention_norm)
 *   h' = rms(X; shared_head_norm);  draft = argmax(lm_head h'), ties to the lower index
 * ------------------------------------------------------------------------ */
typedef struct fm_mtp_config {
  int32_t hidden;      /* H (MCFG.H 5120); a multiple of 128 */
  int32_t inter;       /* I (17408); a multiple of 128 */
  int32_t n_heads;     /* q heads (24) */
  int32_t n_kv_heads;  /* KV heads (4); divides n_heads */
  int32_t head_dim;    /* 256; a multiple of 32, <= 256 */
  int32_t rot_dims;    /* NEOX-rotated dims per head (64); even, <= head_dim */
  float theta;         /* RoPE base (1e7) */
  float eps;           /* RMSNorm eps (1e-6) */
  int32_t vocab;       /* lm_head rows (248320) */
  int32_t kv_cap;      /* cache rows (positions) the head keeps */
  int32_t max_rows;    /* M per pass, <= 8 (MCFG.MAXM) */
} fm_mtp_config;

typedef struct fm_mtp fm_mtp;

/*
 * fm_mtp_create -- load the head.  weights (host or device, copied):
 *   Q8_0 (GGUF rows [N][K/32 * 34]): eh_proj [H][2H], attn_q [n_heads*2*head_dim][H]
 *     (per head the query rows, then its gate rows), attn_k / attn_v
 *     [n_kv_heads*head_dim][H], attn_output [H][n_heads*head_dim], ffn_gate /
 *     ffn_up [I][H], ffn_down [H][I], lm_head [vocab][H];
 *   FM_DTYPE_F32: enorm, hnorm, attn_norm, post_attention_norm, shared_head_norm [H],
 *     attn_q_norm, attn_k_norm [head_dim];
 *   FM_DTYPE_BF16: token_embd [vocab][H] (the rows the drafted tokens are embedded with).
 * Every 2-D product's N must be a multiple of 128 and its K of 64.
 * Errors: FM_ERR_INVALID_ARG (null, missing / mis-sized tensor, wrong dtype),
 *   FM_ERR_UNSUPPORTED (dims outside the limits above), FM_ERR_OOM, FM_ERR_CUDA.
 *   *out is NULL on failure; the reason is in fm_mtp_last_error(NULL).
 */
FM_API fm_status fm_mtp_create(const fm_mtp_config *cfg, const fm_tensor *weights, int32_t n_weights, void *stream,
                               fm_mtp **out);

/*
 * fm_mtp_forward -- MTPHead.forward: one pass over n_rows rows.  tokens_dev:
 * device int32 [n_rows]; hn_dev: device f32 [n_rows][H] (the normed hidden of
 * each row's previous position); writes cache rows pos0 .. pos0+n_rows-1 and,
 * when hout_dev is not NULL, h' (device f32 [n_rows][H]).  Attention reads rows
 * kv_lo .. pos; rows below pos0 must have been written by earlier passes.
 * drafts_dev (device int32 [n_rows] or NULL) receives argmax(lm_head h') per row.
 * Errors: FM_ERR_INVALID_ARG (n_rows outside [1, max_rows], null tokens / hn,
 *   kv_lo outside [0, pos0], pos0 + n_rows > kv_cap), FM_ERR_CUDA.
 */
FM_API fm_status fm_mtp_forward(fm_mtp *m, int32_t n_rows, const int32_t *tokens_dev, const float *hn_dev,
                                int32_t pos0, int32_t kv_lo, float *hout_dev, int32_t *drafts_dev, void *stream);

/*
 * fm_mtp_draft -- MTPRunner's draft: a pass over the n_rows pending rows (as
 * fm_mtp_forward), the draft of its last row, then depth - 1 single-row passes
 * at pos0 + n_rows, ..., each on the previous draft (embedded on the device)
 * and the previous pass's last h'.  drafts_dev: device int32 [depth].  No host
 * round trip between the passes.  Errors: as fm_mtp_forward, and depth outside
 * [1, kv_cap - pos0 - n_rows + 1].
 */
FM_API fm_status fm_mtp_draft(fm_mtp *m, int32_t n_rows, const int32_t *tokens_dev, const float *hn_dev,
                              int32_t pos0, int32_t kv_lo, int32_t depth, int32_t *drafts_dev, void *stream);

/* Copy the head's K (which = 0) or V (which = 1) cache rows [0, rows) ([rows][n_kv_heads * head_dim] f32,
   host or device dst) after the stream's work (synchronises it); for tests.  Also reports what the device
   raised since the last check: FM_ERR_INVALID_ARG for a token outside [0, vocab) that reached the embedding
   (row 0 was read instead), FM_ERR_TIMEOUT for a bounded wait that gave up.  Errors: FM_ERR_INVALID_ARG,
   FM_ERR_CUDA. */
FM_API fm_status fm_mtp_cache(fm_mtp *m, int32_t which, int32_t rows, float *dst, void *stream);

/* Kernel launches issued by the last fm_mtp_forward / fm_mtp_draft. */
FM_API fm_status fm_mtp_last_launch_count(const fm_mtp *m, int32_t *count);
FM_API const char *fm_mtp_last_error(const fm_mtp *m);   /* never NULL; NULL m: the last failed fm_mtp_create */
FM_API void fm_mtp_destroy(fm_mtp *m);

#ifdef __cplusplus
}
#endif
#endif /* FM_H_ */
