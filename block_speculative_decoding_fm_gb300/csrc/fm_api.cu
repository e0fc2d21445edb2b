// fm_api.cu -- host runtime behind the C ABI in include/fm.h: weight intake
// and repacking, the device buffer plan, and the launch sequences of context
// injection and drafting.  Every compute step is one of this library's
// kernels; the host only checks arguments, fills the per-call parameter slot
// and enqueues launches (chained with programmatic dependent launch).
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstddef>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <string>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "../../include/fm.h"
#include "fm_internal.h"
#include "tc_gemm.h"

using namespace fm;

namespace {

constexpr int kParamSlots = 64;

struct Seg2 {  // cache pointers of one sequence and layer
  __half *k, *v;
};

struct ProfRec {
  std::string name;
  cudaEvent_t e0, e1;
  double bytes;
};

}  // namespace

struct fm_handle {
  fm_config cfg{};
  std::string err;
  int n_sm = 148;
  int dev = 0;
  int64_t bytes = 0;
  int32_t debug = 0;
  int32_t last_launches = 0;
  std::vector<void *> allocs;

  // ---- weights (FlashMap) ----
  __nv_bfloat16 *w_fc = nullptr, *w_hn = nullptr, *w_ap = nullptr, *b_ap = nullptr, *w_an = nullptr;
  __nv_bfloat16 *w_sn = nullptr, *w_xe = nullptr, *b_xe = nullptr, *w_head = nullptr, *b_head = nullptr;
  __nv_bfloat16 *w_kvall = nullptr, *w_ckn = nullptr;
  std::vector<__nv_bfloat16 *> w_qkv, w_sqn, w_skn, w_so, w_cq, w_cqn, w_co, w_f1, b_f1, w_f2, b_f2;
  float *mod = nullptr;
  // ---- weights (DFlash) ----
  std::vector<__nv_bfloat16 *> w_o, w_gu, w_down;
  __nv_bfloat16 *attn_norm = nullptr, *ff_norm = nullptr, *ctx_norm = nullptr, *out_norm = nullptr;
  __nv_bfloat16 *w_c = nullptr, *w_tok = nullptr, *block_pos = nullptr, *w_out = nullptr;
  float *hinit = nullptr;
  // ---- token table (Q8_0: lm_head chunk layout; bf16: GEMV tile layout) ----
  uint8_t *tq8 = nullptr;
  uint8_t *tb = nullptr;
  int Vpad = 0;

  // ---- state ----
  __half *cache = nullptr;
  size_t cache_plane = 0;  // elements of one [H][max_ctx][hd] plane
  std::vector<int32_t> length;
  float2 *rope = nullptr;
  int rope_pos = 0;
  float *h0 = nullptr;

  // ---- work buffers ----
  float *X = nullptr, *qkv = nullptr, *qc = nullptr, *attn = nullptr, *u = nullptr, *Y = nullptr;
  uint8_t *ylm = nullptr;  // the head output as the lm_head operand (hi/lo halves, swizzled)
  float *ctx = nullptr, *actx = nullptr, *uni = nullptr, *hid = nullptr, *dbg_logits = nullptr;
  float2 *st_x = nullptr, *st_h0 = nullptr, *st_c = nullptr, *st_a = nullptr, *st_u = nullptr, *st_init = nullptr;
  float *part_o = nullptr;
  float2 *part_ml = nullptr, *lm_part = nullptr;
  int max_splits = 1;
  int32_t *tickets = nullptr;  // [0, H): self, [H, 2H): cross, [2H]: lm head
  float *xo = nullptr;         // cross-attention range partials of the current lane
  float2 *xml = nullptr;
  int32_t *xtickets = nullptr;
  int32_t *tok_tmp = nullptr;

  // ---- DFlash sequential logit head and confidence head (optional tensors) ----
  __nv_bfloat16 *seq_w1 = nullptr;   // markov.w1 [V][r]
  __nv_bfloat16 *seq_W = nullptr;    // markov.w2, or rnn.wO with the RNN head [r][V]
  __nv_bfloat16 *seq_wH = nullptr, *seq_bH = nullptr;  // RNN head only: [r][r], [r]
  __nv_bfloat16 *conf_w = nullptr, *conf_b = nullptr;  // [d + r], [1], or null
  int seq_rank = 0;                   // r; 0: no sequential head (each slot's argmax is its token)

  // ---- dense prefill (tcgen05) ----
  __half *w_fc16 = nullptr, *w_kv16 = nullptr;  // f16 copies of fc and the stacked cross K/V
  __half *pf_a = nullptr, *pf_c = nullptr;       // scratch: f16 feature rows, f16 weighted fc output
  float *pf_st = nullptr;                         // per-row partial sums of squares
  int32_t *pf_err = nullptr;
  int pf_rows = 0;                                // rows the scratch holds
  CUtensorMap tm_wfc{}, tm_wkv{}, tm_c{};

  int32_t *dev_err = nullptr;     // raised by a device-side bounded wait that gave up

  // ---- calls with host buffers: device copies of their feature rows and tokens ----
  float *stage_feats = nullptr;   // grown on demand
  size_t stage_cap = 0;           // floats stage_feats holds
  int32_t *stage_tok = nullptr;   // [max_seqs][block]
  cudaEvent_t stage_ev = nullptr; // recorded after the last host-buffer call's work

  // ---- the persistent draft step ----
  bool use_step = true;
  int step_attrs = 3;                 // launch attributes the device accepted (cooperative | PDL)
  int step_clusters = 0;              // co-resident clusters of the step kernel
  uint32_t *step_bar = nullptr;       // grid barrier words
  // device programs by (sequence, key splits, debug, parameter slot): the jobs
  // carry the address of the parameter slot their chain reads
  std::map<std::tuple<int, int, int, const void *>, StepPhase *> step_progs;
  uint64_t *step_trace = nullptr;     // FM_DEBUG_TRACE: per phase and CTA, globaltimer stamps
  int step_trace_phases = 0;
  int xattn_cluster = 0;              // the largest cross-attention cluster all heads' fit at once
  // several sequences' chains run at once (a batched call): each product then runs unsplit, on as
  // many CTAs as it has 128-row tiles, so that the chains fill the GPU side by side
  bool narrow = false;
  std::vector<void *> to_free;    // row-major staging copies released at the end of fm_create

  // ---- batched draft: the slot rows of up to kWideSeqs sequences go through the
  // tensor-core GEMM together, so each weight is read once per pass ----
  struct Wide {
    bool on = false;
    int Vn = 0;                                      // token table rows, padded to 256
    std::vector<__half *> qkv, so, cq, co, f1, f2;   // f16 copies of the layer weights, [N][K]
    __half *ap = nullptr, *head = nullptr, *table = nullptr;
    std::vector<CUtensorMap> t_qkv, t_so, t_cq, t_co, t_f1, t_f2;
    CUtensorMap t_ap{}, t_head{}, t_table{}, t_cache{};
    // activations: X [rows][D] f32; q/k/v and cross q f32; the head output f32 and f16
    float *X = nullptr, *qkv_out = nullptr, *qc = nullptr, *Y = nullptr, *kst = nullptr;
    float *br = nullptr;            // without tensor stores: a product's gated branch, added by the next adaLN
    __half *a16 = nullptr, *o16 = nullptr, *u16 = nullptr, *y16 = nullptr, *anc16 = nullptr, *kin16 = nullptr;
    CUtensorMap m_a16{}, m_o16{}, m_u16{}, m_y16{}, m_anc16{}, m_kin16{};
    float2 *amax = nullptr;         // lm_head per-row, per-column-block bests
    float *xo = nullptr;            // cross-attention range partials of every sequence
    float2 *xml = nullptr;
    int32_t *xtickets = nullptr;
    int xsplits = 1;                // key ranges per (sequence, head) (measured: 1 > 2 > 3 at 32 sequences)
    bool tstore = true;             // single-output epilogues write through tensor stores (FM_WIDE_TSTORE=0: plain)
    int max_ksplit = 4;             // K slices per GEMM tile at most (1, 2 or 4)
    WideParams *par = nullptr;      // device copy of the pass's values
    WideParams *par_host = nullptr; // pinned ring
    cudaEvent_t par_ev[kParamSlots]{};
    int par_next = 0;
    // batched append: per-row (sequence, position) of the rows' K/V
    int32_t *rows = nullptr, *rows_host = nullptr;
    int rows_cap = 0;
    cudaEvent_t rows_ev[kParamSlots]{};
    int rows_next = 0;
    std::vector<int> row_of;        // per sequence: its first row in the last batched pass; -1: its last
                                    // draft was not batched; -2: an earlier pass of the last batched call
    double keys = 0;                // the current pass's cache rows read per layer (profile bytes)
    float *dbg_logits = nullptr;    // FM_DEBUG_LOGITS of a batched draft: [block][Vn]
  } wide;

  // ---- per-sequence lanes ----
  // Each sequence has its own work buffers (and, with several sequences, its own
  // stream), so the chains of different sequences can run at the same time; the
  // fields X .. tickets above point at the lane whose chain is being built.
  struct Lane {
    float *X = nullptr, *qkv = nullptr, *qc = nullptr, *attn = nullptr, *u = nullptr, *Y = nullptr;
    float *ctx = nullptr, *actx = nullptr;
    uint8_t *ylm = nullptr;
    float2 *st_x = nullptr, *st_c = nullptr, *st_a = nullptr, *st_u = nullptr, *lm_part = nullptr;
    int32_t *tickets = nullptr;
    // sequential head: base logits [block][V], RNN states [2][r], per-CTA bests,
    // flags {decided, length, ticket, -, scratch tokens [kMaxT]}
    float *seq_base = nullptr, *seq_state = nullptr;
    float2 *seq_part = nullptr;
    int32_t *seq_flags = nullptr;
    // tensor-core cross-attention: per-range partials and per-head tickets
    float *xo = nullptr;
    float2 *xml = nullptr;
    int32_t *xtickets = nullptr;
    cudaStream_t stream = nullptr;
    cudaEvent_t done = nullptr;
    // a short append whose K/V projection waits for this sequence's next draft
    bool pending = false;
    int pend_start = 0, pend_n = 0;
  };
  std::vector<Lane> lanes;
  cudaEvent_t fork_ev = nullptr;

  // ---- captured chains ----
  struct GraphEntry {
    cudaGraphExec_t exec = nullptr;
    StepParams *sp = nullptr;
    int launches = 0;
  };
  std::unordered_map<uint64_t, GraphEntry> graphs;
  cudaStream_t cap = nullptr;
  bool use_graphs = true;
  bool use_prefill = true;
  bool use_defer = true;

  // ---- diagnostics ----
  std::vector<ProfRec> prof;
  std::vector<cudaEvent_t> ev_pool;

  // ---- per-call parameters ----
  StepParams *sp_dev = nullptr;
  StepParams *sp_host = nullptr;  // pinned
  cudaEvent_t sp_ev[kParamSlots]{};
  int sp_next = 0;

  Seg2 kv(int seq, int l) const {
    const size_t base = ((size_t)seq * cfg.n_layers + l) * 2 * cache_plane;
    return {cache + base, cache + base + cache_plane};
  }
};

namespace {

thread_local std::string g_create_error;  // reason of the last failed fm_create on this thread

// point the handle's work-buffer fields at sequence seq's lane
void use_lane(fm_handle *h, int seq) {
  const fm_handle::Lane &L = h->lanes[seq];
  h->X = L.X; h->qkv = L.qkv; h->qc = L.qc; h->attn = L.attn; h->u = L.u; h->Y = L.Y;
  h->ctx = L.ctx; h->actx = L.actx; h->ylm = L.ylm;
  h->st_x = L.st_x; h->st_c = L.st_c; h->st_a = L.st_a; h->st_u = L.st_u; h->lm_part = L.lm_part;
  h->tickets = L.tickets;
  h->xo = L.xo; h->xml = L.xml; h->xtickets = L.xtickets;
}

fm_status fail(fm_handle *h, fm_status s, const char *fmt, ...) {
  if (h) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    h->err = buf;
  }
  return s;
}

#define CK(expr)                                                                                     \
  do {                                                                                               \
    cudaError_t e_ = (expr);                                                                         \
    if (e_ != cudaSuccess) return fail(h, FM_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_));     \
  } while (0)

// Fault injection for the allocation path (host side only): FM_FAULT_INJECT=alloc:N
// makes the N-th device allocation of a handle report out-of-memory.
int fault_alloc_at() {
  const char *s = getenv("FM_FAULT_INJECT");
  if (!s || strncmp(s, "alloc:", 6) != 0) return -1;
  return atoi(s + 6);
}

template <typename T>
fm_status dalloc(fm_handle *h, T **p, size_t count) {
  const int inject = fault_alloc_at();
  if (inject >= 0 && (int)h->allocs.size() + 1 == inject) {
    *p = nullptr;
    return fail(h, FM_ERR_OOM, "injected allocation failure at allocation %d", inject);
  }
  const size_t bytes = count * sizeof(T) > 0 ? count * sizeof(T) : 16;
  void *q = nullptr;
  cudaError_t e = cudaMalloc(&q, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    return fail(h, FM_ERR_OOM, "cudaMalloc(%zu bytes): %s", bytes, cudaGetErrorString(e));
  }
  h->allocs.push_back(q);
  h->bytes += (int64_t)bytes;
  *p = static_cast<T *>(q);
  return FM_OK;
}

void dfree_later(fm_handle *h, void *p) {
  auto it = std::find(h->allocs.begin(), h->allocs.end(), p);
  if (it != h->allocs.end()) h->allocs.erase(it);
  h->to_free.push_back(p);
}

#define TRY(expr)                    \
  do {                               \
    fm_status s_ = (expr);           \
    if (s_ != FM_OK) return s_;      \
  } while (0)

struct TensorSet {
  std::unordered_map<std::string, const fm_tensor *> by_name;
};

fm_status find(fm_handle *h, const TensorSet &ts, const std::string &name, int64_t nbytes, int32_t dtype,
               bool required, const fm_tensor **out) {
  *out = nullptr;
  auto it = ts.by_name.find(name);
  if (it == ts.by_name.end()) {
    if (required) return fail(h, FM_ERR_INVALID_ARG, "missing tensor %s", name.c_str());
    return FM_OK;
  }
  const fm_tensor *t = it->second;
  if (t->dtype != dtype) return fail(h, FM_ERR_INVALID_ARG, "tensor %s: dtype %d, expected %d", name.c_str(), t->dtype, dtype);
  if (t->nbytes != nbytes)
    return fail(h, FM_ERR_INVALID_ARG, "tensor %s: %lld bytes, expected %lld", name.c_str(), (long long)t->nbytes,
                (long long)nbytes);
  if (!t->data) return fail(h, FM_ERR_INVALID_ARG, "tensor %s: null data", name.c_str());
  *out = t;
  return FM_OK;
}

// copy a bf16 tensor (required unless `optional`) to dst; absent optional -> zeros
fm_status put_bf16(fm_handle *h, const TensorSet &ts, const std::string &name, void *dst, int64_t elems,
                   cudaStream_t s, bool optional = false) {
  const fm_tensor *t;
  TRY(find(h, ts, name, elems * 2, FM_DTYPE_BF16, !optional, &t));
  if (!t) {
    CK(cudaMemsetAsync(dst, 0, elems * 2, s));
    return FM_OK;
  }
  CK(cudaMemcpyAsync(dst, t->data, elems * 2, cudaMemcpyDefault, s));
  return FM_OK;
}

// copy an [in][out] bf16 matrix transposed into dst ([out][in], row stride ldo)
fm_status put_bf16_t(fm_handle *h, const TensorSet &ts, const std::string &name, int rows, int cols,
                     __nv_bfloat16 *dst, int ldo, __nv_bfloat16 *tmp, cudaStream_t s) {
  const fm_tensor *t;
  TRY(find(h, ts, name, (int64_t)rows * cols * 2, FM_DTYPE_BF16, true, &t));
  CK(cudaMemcpyAsync(tmp, t->data, (size_t)rows * cols * 2, cudaMemcpyDefault, s));
  CK(launch_transpose_bf16(tmp, rows, cols, dst, ldo, s));
  return FM_OK;
}

// Replace a row-major [M][K] bf16 weight by its GEMV tile layout (same pointer slot).
fm_status tile_weight(fm_handle *h, __nv_bfloat16 **w, int M, int K, cudaStream_t s) {
  uint8_t *t;
  TRY(dalloc(h, &t, tiled_bytes(M, K)));
  CK(launch_tile_weights(*w, M, K, t, s));
  dfree_later(h, *w);
  *w = reinterpret_cast<__nv_bfloat16 *>(t);
  return FM_OK;
}

StepParams *next_params(fm_handle *h, const StepParams &p, cudaStream_t s, fm_status *st) {
  const int i = h->sp_next;
  h->sp_next = (h->sp_next + 1) % kParamSlots;
  cudaEventSynchronize(h->sp_ev[i]);  // the slot's previous copy has been consumed
  h->sp_host[i] = p;
  cudaError_t e = cudaMemcpyAsync(h->sp_dev + i, h->sp_host + i, sizeof(StepParams), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaEventRecord(h->sp_ev[i], s);
  if (e != cudaSuccess) {
    *st = fail(h, FM_ERR_CUDA, "parameter upload: %s", cudaGetErrorString(e));
    return nullptr;
  }
  *st = FM_OK;
  return h->sp_dev + i;
}

// Upload p into a fixed device slot through the pinned ring (stream ordered).
fm_status upload_params(fm_handle *h, const StepParams &p, StepParams *dst, cudaStream_t s) {
  const int i = h->sp_next;
  h->sp_next = (h->sp_next + 1) % kParamSlots;
  cudaEventSynchronize(h->sp_ev[i]);
  h->sp_host[i] = p;
  CK(cudaMemcpyAsync(dst, h->sp_host + i, sizeof(StepParams), cudaMemcpyHostToDevice, s));
  CK(cudaEventRecord(h->sp_ev[i], s));
  return FM_OK;
}

cudaEvent_t pool_event(fm_handle *h) {
  if (!h->ev_pool.empty()) {
    cudaEvent_t e = h->ev_pool.back();
    h->ev_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Optional event bracket around one launch (FM_DEBUG_PROFILE).
struct ProfScope {
  fm_handle *h;
  cudaStream_t s;
  ProfRec rec;
  bool on;
  ProfScope(fm_handle *h_, cudaStream_t s_, const char *name, double bytes) : h(h_), s(s_), on(h_->debug & FM_DEBUG_PROFILE) {
    if (!on) return;
    rec.name = name;
    rec.bytes = bytes;
    rec.e0 = pool_event(h);
    rec.e1 = pool_event(h);
    cudaEventRecord(rec.e0, s);
  }
  ~ProfScope() {
    if (!on) return;
    cudaEventRecord(rec.e1, s);
    h->prof.push_back(rec);
  }
};

GemvArgs gemv_base(const fm_handle *h, const __nv_bfloat16 *W, int M, int K, int T_const, const StepParams *sp) {
  GemvArgs a;
  memset(&a, 0, sizeof a);
  a.Wt = reinterpret_cast<const uint8_t *>(W);  // weight buffers hold the GEMV tile layout
  a.err = h->dev_err;
  a.M = M;
  a.K = K;
  a.T_const = T_const;
  a.sp = sp;
  const int tiles = (M + kTile - 1) / kTile;
  // split K over a cluster of up to 8 CTAs; unsplit when several sequences' chains run at once
  // (measured, 32 FlashMap-4B sequences: split as a single chain 76 steps/s, to one wave of
  // clusters 95, unsplit 109)
  int ks = 1;
  while (!h->narrow && ks < 8 && K % (64 * ks * 2) == 0 && tiles * ks * 2 <= 2 * h->n_sm) ks *= 2;
  a.ksplit = ks;
  a.Kc = K / ks;
  // activation pieces: 256 columns; 128 for 17..32 rows, which keeps two CTAs per SM
  const int kp = (T_const > 0 && T_const <= 16) ? 256 : 128;
  a.Kp = a.Kc < kp ? a.Kc : kp;
  a.hd = h->cfg.head_dim;
  a.max_ctx = h->cfg.max_ctx;
  a.rope = h->rope;
  a.qk_eps = h->cfg.qk_eps;
  a.eps = h->cfg.rms_eps;
  a.inv_n = 1.0f / (float)K;
  return a;
}

fm_status run_gemv(fm_handle *h, const GemvArgs &a, cudaStream_t s, const char *tag = "gemv", int T = 16) {
  const int tiles = (a.M + kTile - 1) / kTile;
  ProfScope ps(h, s, tag, (double)a.M * a.K * 2 + (double)T * (a.K + a.M) * 4);
  CK(launch_gemv(a, tiles, s, true));
  ++h->last_launches;
  return FM_OK;
}

// Key ranges per head for the cross-attention over L keys, and how they merge.
// Head dim 128 (tensor-core kernel): up to four 128-key tiles per range, the
// ranges of a head merged in a cluster (one-stage ring) no larger than lets every
// head's cluster run at once; longer contexts: one range per SM, three-stage
// rings, merged by the last range (ticket).
// Head dim 64: one cluster of at most 8 CTAs per head (16-CTA clusters were
// measured slower there: their scheduling and merge cost more than the shorter
// key loop saves).
struct AttnPlan {
  int splits;
  bool cluster;
};
AttnPlan attn_plan(const fm_handle *h, int L) {
  const int nt = (L + 127) / 128;
  if (h->cfg.head_dim != 128) return {nt < 1 ? 1 : nt > 8 ? 8 : nt, true};
  // the largest cluster of which every head's can run at once (measured on this GPU: 15
  // clusters of 7..9 ranges, 23 of 6, 7 of 16), then up to four tiles per range
  const int cl = nt < h->xattn_cluster ? nt : h->xattn_cluster;
  if (cl >= 1 && nt <= 4 * cl) return {cl, true};
  int cap = h->n_sm / h->cfg.n_heads;
  if (cap > kMaxXSplits) cap = kMaxXSplits;
  if (cap < 1) cap = 1;
  return {nt > cap ? cap : nt, false};
}
// the plan as one number (part of a captured chain's key)
int attn_splits(const fm_handle *h, int L) {
  const AttnPlan p = attn_plan(h, L);
  return p.splits + (p.cluster ? 0 : 64);
}

fm_status run_attn(fm_handle *h, const float *Q, int ldq, const Seg2 &kv, int T, int L_src, int L_add, int L_now,
                   const StepParams *sp, float *out, cudaStream_t s) {
  const fm_config &c = h->cfg;
  if (c.head_dim == 128) {
    XAttnArgs x;
    memset(&x, 0, sizeof x);
    if (!make_cache_map(&x.tm_k, kv.k, c.n_heads, c.max_ctx) || !make_cache_map(&x.tm_v, kv.v, c.n_heads, c.max_ctx))
      return fail(h, FM_ERR_CUDA, "cache tensor map encoding failed");
    x.Q = Q;
    x.ldq = ldq;
    x.max_ctx = c.max_ctx;
    x.n_heads = c.n_heads;
    const AttnPlan plan = attn_plan(h, L_now);
    x.splits = plan.splits;
    x.T_const = T;
    x.L_src = L_src;
    x.L_add = L_add;
    x.sp = sp;
    x.scale_log2 = (float)(1.4426950408889634 / std::sqrt(128.0));
    x.out = out;
    x.ldo = c.dim;
    x.part_o = h->xo;
    x.part_ml = h->xml;
    x.tickets = h->xtickets;
    x.err = h->dev_err;
    ProfScope ps(h, s, "attn.cross", (double)L_now * c.dim * 2 * 2 + 2.0 * T * c.dim * 4);
    CK(launch_xattn(x, plan.cluster ? 1 : 3, plan.cluster, s, true));
    ++h->last_launches;
    return FM_OK;
  }
  AttnArgs a;
  memset(&a, 0, sizeof a);
  a.Q = Q;
  a.ldq = ldq;
  a.Kc = kv.k;
  a.Vc = kv.v;
  a.max_ctx = c.max_ctx;
  a.n_heads = c.n_heads;
  a.hd = c.head_dim;
  a.splits = attn_plan(h, L_now).splits;
  a.T_const = T;
  a.L_src = L_src;
  a.L_add = L_add;
  a.sp = sp;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c.head_dim));
  a.out = out;
  a.ldo = c.dim;
  ProfScope ps(h, s, "attn.cross", (double)L_now * c.dim * 2 * 2 + 2.0 * T * c.dim * 4);
  CK(launch_attn(a, L_now, s, true));
  ++h->last_launches;
  return FM_OK;
}

fm_status run_lmhead(fm_handle *h, const float *Y, int T, const StepParams *sp, int32_t *tokens, float *logits,
                     cudaStream_t s, const uint8_t *ylm = nullptr) {
  const fm_config &c = h->cfg;
  LmArgs a;
  memset(&a, 0, sizeof a);
  if (c.lm_format == FM_LM_Q8_0)
    a.q8 = h->tq8;
  else
    a.wb = h->tb;
  a.err = h->dev_err;
  a.V = c.vocab;
  a.H = c.target_dim;
  a.T_const = T;
  a.sp = sp;
  a.Y = Y;
  a.ldy = c.target_dim;
  a.ylm = ylm;
  a.part = h->lm_part;
  a.ticket = h->tickets + 2 * c.n_heads;
  a.tokens = tokens;
  a.logits = logits;
  const double tb = c.lm_format == FM_LM_Q8_0 ? (double)c.vocab * (c.target_dim + c.target_dim / 16)
                                               : (double)c.vocab * c.target_dim * 2;
  ProfScope ps(h, s, "lm_head", tb + (double)T * c.target_dim * 4);
  CK(launch_lmhead(a, lmhead_grid(a, h->n_sm), s, true));
  ++h->last_launches;
  return FM_OK;
}

// ---------------------------------------------------------------- FlashMap

// fc (no bias) on the appended feature rows -> ctx rows + their row statistics
fm_status flashmap_fc_rows(fm_handle *h, const StepParams *sp, int T, cudaStream_t s) {
  const fm_config &c = h->cfg;
  const int D = c.dim, FW = c.n_taps * c.target_dim;
  GemvArgs a = gemv_base(h, h->w_fc, D, FW, 0, sp);
  a.amode = A_PLAIN;
  a.x_from_sp = 1;
  a.ldx = FW;
  a.emode = E_STORE;
  a.Y = h->ctx;
  a.ldy = D;
  a.out_st = h->st_c;
  return run_gemv(h, a, s, "gemv.fc", T);
}

// The stacked cross K/V of every layer over normalised rows: rows < split are
// ctx rows (hidden_norm, positions start + t); with an anchor row (split > 0 and
// T = split + 1) the last row is the anchor (anchor_norm, position pos).
GemvArgs flashmap_kv_args(fm_handle *h, int seq, const StepParams *sp, int T_const, int split) {
  const fm_config &c = h->cfg;
  const int D = c.dim, L = c.n_layers;
  GemvArgs b = gemv_base(h, h->w_kvall, L * 2 * D, D, T_const, sp);
  b.amode = A_RMS;
  b.X = split > 0 || T_const == 0 ? h->ctx : h->actx;
  b.ldx = D;
  b.st = split > 0 || T_const == 0 ? h->st_c : h->st_a;
  b.st_tiles = D / kTile;
  b.nw = split > 0 || T_const == 0 ? h->w_hn : h->w_an;
  b.inv_n = 1.0f / D;
  if (split > 0) {
    b.split = split;
    b.X2 = h->actx;
    b.st2 = h->st_a;
    b.nw_alt = h->w_an;
    b.pos_src = 3;
  } else {
    b.pos_src = T_const == 0 ? 1 : 0;
  }
  b.emode = E_SEGS;
  b.seg_rows = D;
  b.n_segs = 2 * L;
  for (int l = 0; l < L; ++l) {
    Seg2 kv = h->kv(seq, l);
    b.segs[2 * l] = {SEG_CACHE, 0, 1, 0, h->w_ckn + (size_t)l * c.head_dim, kv.k};
    b.segs[2 * l + 1] = {SEG_CACHE, 0, 0, 0, nullptr, kv.v};
  }
  return b;
}

// fc -> hidden_norm -> all layers' k / v (k_norm + RoPE) -> f16 cache rows
fm_status flashmap_append_rows(fm_handle *h, int seq, const StepParams *sp, int T, cudaStream_t s) {
  TRY(flashmap_fc_rows(h, sp, T, s));
  return run_gemv(h, flashmap_kv_args(h, seq, sp, 0, 0), s, "gemv.kv_append", T);
}

// The products of one FlashMap draft, in order: the anchor slot (anchor_proj,
// then the K/V of the pending rows and the anchor row), per layer the self
// q/k/v (+ the block attention tail), o, cross q, cross o, fc1 and fc2, then
// the head.  Shared by the launch-per-product chain and the persistent step.
struct FlashMapPlan {
  GemvArgs anchor, kv;
  std::vector<GemvArgs> qkv, o, cq, co, f1, f2;
  GemvArgs head;
};

FlashMapPlan flashmap_plan(fm_handle *h, int seq, const StepParams *sp, int n_pend) {
  const fm_config &c = h->cfg;
  const int D = c.dim, B = c.block, Ht = c.target_dim, F = c.ff_dim, L = c.n_layers;
  FlashMapPlan pl;
  // the anchor's context slot at pos: anchor_proj(E[anchor]) -> anchor_norm -> k / v of every layer
  GemvArgs a = gemv_base(h, h->w_ap, D, Ht, 1, sp);
  a.amode = c.lm_format == FM_LM_Q8_0 ? A_ROW_Q8 : A_ROW_BF16;
  a.tq8 = h->tq8;
  a.tb = h->tb;
  a.emode = E_STORE;
  a.bias = h->b_ap;
  a.Y = h->actx;
  a.ldy = D;
  a.out_st = h->st_a;
  pl.anchor = a;
  // the pending appended rows (deferred) and the anchor row share one pass over the cross K/V weights
  pl.kv = flashmap_kv_args(h, seq, sp, n_pend + 1, n_pend);

  const float attn_scale = (float)(1.0 / std::sqrt((double)c.head_dim));
  for (int l = 0; l < L; ++l) {
    const float *m_self = h->mod + (size_t)(3 * l + 0) * 3 * D;
    const float *m_cross = h->mod + (size_t)(3 * l + 1) * 3 * D;
    const float *m_mlp = h->mod + (size_t)(3 * l + 2) * 3 * D;
    const bool first = l == 0;
    // self-attention: adaLN -> q, k, v (+ q/k norm, RoPE at pos + 1 + t) -> attention tail
    GemvArgs q = gemv_base(h, h->w_qkv[l], 3 * D, D, B, sp);
    q.amode = A_LNMOD;
    q.X = first ? h->h0 : h->X;
    q.ldx = first ? 0 : D;
    q.st = first ? h->st_h0 : h->st_x;
    q.st_bcast = first ? 1 : 0;
    q.st_tiles = D / kTile;
    q.sc = m_self;
    q.sh = m_self + D;
    q.eps = c.ln_eps;
    q.inv_n = 1.0f / D;
    q.emode = E_SEGS;
    q.Y = h->qkv;
    q.ldy = 3 * D;
    q.seg_rows = D;
    q.n_segs = 3;
    q.segs[0] = {SEG_F32, 0, 1, 0, h->w_sqn[l], nullptr};
    q.segs[1] = {SEG_F32, D, 1, 0, h->w_skn[l], nullptr};
    q.segs[2] = {SEG_F32, 2 * D, 0, 0, nullptr, nullptr};
    q.pos_src = 0;
    q.pos_add = 1;
    q.tickets = h->tickets;
    q.attn_out = h->attn;
    q.self_D = D;
    q.attn_scale = attn_scale;
    pl.qkv.push_back(q);

    GemvArgs o = gemv_base(h, h->w_so[l], D, D, B, sp);
    o.amode = A_PLAIN;
    o.X = h->attn;
    o.ldx = D;
    o.emode = E_RESID;
    o.R = first ? h->h0 : h->X;
    o.ldr = first ? 0 : D;
    o.gate = m_self + 2 * D;
    o.Y = h->X;
    o.ldy = D;
    o.out_st = h->st_x;
    pl.o.push_back(o);

    // cross-attention over cache rows 0 .. pos
    GemvArgs cq = gemv_base(h, h->w_cq[l], D, D, B, sp);
    cq.amode = A_LNMOD;
    cq.X = h->X;
    cq.ldx = D;
    cq.st = h->st_x;
    cq.st_tiles = D / kTile;
    cq.sc = m_cross;
    cq.sh = m_cross + D;
    cq.eps = c.ln_eps;
    cq.inv_n = 1.0f / D;
    cq.emode = E_SEGS;
    cq.Y = h->qc;
    cq.ldy = D;
    cq.seg_rows = D;
    cq.n_segs = 1;
    cq.segs[0] = {SEG_F32, 0, 1, 0, h->w_cqn[l], nullptr};
    cq.pos_src = 0;
    cq.pos_add = 1;
    pl.cq.push_back(cq);

    GemvArgs co = gemv_base(h, h->w_co[l], D, D, B, sp);
    co.amode = A_PLAIN;
    co.X = h->attn;
    co.ldx = D;
    co.emode = E_RESID;
    co.R = h->X;
    co.ldr = D;
    co.gate = m_cross + 2 * D;
    co.Y = h->X;
    co.ldy = D;
    co.out_st = h->st_x;
    pl.co.push_back(co);

    // MLP: adaLN -> fc1 + bias -> exact GELU -> fc2 + bias -> gated residual
    GemvArgs f1 = gemv_base(h, h->w_f1[l], F, D, B, sp);
    f1.amode = A_LNMOD;
    f1.X = h->X;
    f1.ldx = D;
    f1.st = h->st_x;
    f1.st_tiles = D / kTile;
    f1.sc = m_mlp;
    f1.sh = m_mlp + D;
    f1.eps = c.ln_eps;
    f1.inv_n = 1.0f / D;
    f1.emode = E_GELU;
    f1.bias = h->b_f1[l];
    f1.Y = h->u;
    f1.ldy = F;
    pl.f1.push_back(f1);

    GemvArgs f2 = gemv_base(h, h->w_f2[l], D, F, B, sp);
    f2.amode = A_PLAIN;
    f2.X = h->u;
    f2.ldx = F;
    f2.emode = E_RESID;
    f2.bias = h->b_f2[l];
    f2.R = h->X;
    f2.ldr = D;
    f2.gate = m_mlp + 2 * D;
    f2.Y = h->X;
    f2.ldy = D;
    f2.out_st = h->st_x;
    pl.f2.push_back(f2);
  }
  // final adaLN -> head (its output also split into the lm_head operand)
  const float *m_fin = h->mod + (size_t)(3 * L) * 3 * D;
  GemvArgs hd = gemv_base(h, h->w_head, Ht, D, B, sp);
  hd.amode = A_LNMOD;
  hd.X = h->X;
  hd.ldx = D;
  hd.st = h->st_x;
  hd.st_tiles = D / kTile;
  hd.sc = m_fin;
  hd.sh = m_fin + D;
  hd.eps = c.ln_eps;
  hd.inv_n = 1.0f / D;
  hd.emode = E_STORE;
  hd.bias = h->b_head;
  hd.Y = h->Y;
  hd.ldy = Ht;
  hd.ylm = h->ylm;
  hd.ylm_f16 = c.lm_format == FM_LM_Q8_0;
  pl.head = hd;
  return pl;
}

// The persistent program of one FlashMap draft (layers + head): per layer the
// q/k/v product, o with the block self-attention as its prologue, cross-q with
// the cross-attention as its tail, cross-o, fc1 and fc2; then the head.
// Returns false when the shapes do not fit the kernel's limits (the caller
// then runs the launch-per-product chain).
bool flashmap_step_program(fm_handle *h, int seq, const FlashMapPlan &pl, std::vector<StepPhase> &ph) {
  const fm_config &c = h->cfg;
  const int D = c.dim, L = c.n_layers, hd = c.head_dim, ncl = h->step_clusters;
  if (ncl < 1 || c.block > 16) return false;
  int rot = 0;
  auto linear = [&](const GemvArgs &g, int map_mod) {
    StepPhase P;
    memset(&P, 0, sizeof P);
    P.g = g;
    P.cpt = g.K / 64;
    P.ntiles = (g.M + kTile - 1) / kTile;
    P.map_mod = map_mod > 0 ? map_mod : P.ntiles;
    P.rot = rot % ncl;
    rot += P.ntiles;   // the clusters that got an extra tile move on from phase to phase
    P.prologue = SP_NONE;
    P.tail = ST_NONE;
    ph.push_back(P);
    return &ph.back();
  };
  const float scale = (float)(1.0 / std::sqrt((double)hd));
  for (int l = 0; l < L; ++l) {
    linear(pl.qkv[l], 0);
    StepPhase *o = linear(pl.o[l], 0);
    o->prologue = SP_SELF_ATTN;
    o->at.hd = hd;
    o->at.scale = scale;
    o->at.D = D;
    o->at.qkv = h->qkv;
    StepPhase *q = linear(pl.cq[l], 0);
    q->tail = ST_CROSS_ATTN;
    Seg2 kv = h->kv(seq, l);
    q->at.max_ctx = c.max_ctx;
    q->at.n_heads = c.n_heads;
    q->at.hd = hd;
    q->at.L_src = 1;
    q->at.L_add = 0;
    q->at.scale = scale;
    q->at.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)hd));
    q->at.Kc = kv.k;
    q->at.Vc = kv.v;
    q->at.Q = h->qc;
    q->at.ldq = D;
    q->at.out = h->attn;
    q->at.ldo = D;
    linear(pl.co[l], 0);
    linear(pl.f1[l], 0);
    GemvArgs f2 = pl.f2[l];
    if (h->debug & FM_DEBUG_KEEP_HIDDEN) {
      f2.Y2 = h->hid + (size_t)l * kMaxT * D;
      f2.ldy2 = D;
    }
    linear(f2, 0);
  }
  linear(pl.head, 0);
  // the kernel's limits
  for (size_t i = 0; i < ph.size(); ++i) {
    const StepPhase &P = ph[i];
    if (P.g.K % 64 || P.cpt < 1) return false;
    std::vector<int> per(ncl, 0);
    for (int t = 0; t < P.ntiles; ++t) ++per[step_cluster_of(P, t, ncl)];
    const int most = *std::max_element(per.begin(), per.end());
    if (most > kStepMaxTiles) return false;
    // the rank's K slice fits one staged piece when it is formed in shared memory,
    // and the q, k, v rows of the heads it covers fit the partial area
    if (P.prologue == SP_SELF_ATTN) {
      if (D % hd) return false;
      for (int r = 0; r < kStepCS; ++r) {
        const int kb = step_klo(r, P.cpt) * 64, ncol = (step_klo(r + 1, P.cpt) - step_klo(r, P.cpt)) * 64;
        if (ncol == 0) continue;
        if (ncol > 256) return false;
        const int heads = (kb + ncol - 1) / hd - kb / hd + 1;
        if ((size_t)heads * 3 * 16 * (hd + 4) * 4 > 52 * 1024) return false;
      }
    }
    // the cross-attention tail requests its first key stage in the partial area
    // behind the previous phase's two tiles
    if (P.tail == ST_CROSS_ATTN) {
      if (most > 2 || i == 0 || hd % 16) return false;
      std::vector<int> prev(ncl, 0);
      for (int t = 0; t < ph[i - 1].ntiles; ++t) ++prev[step_cluster_of(ph[i - 1], t, ncl)];
      if (*std::max_element(prev.begin(), prev.end()) > 2) return false;
    }
  }
  return true;
}

fm_status run_step(fm_handle *h, int seq, const std::vector<StepPhase> &prog, const StepParams *sp, int T,
                   double bytes, cudaStream_t s) {
  const auto key = std::make_tuple(seq, 0, h->debug & FM_DEBUG_KEEP_HIDDEN, (const void *)sp);
  auto it = h->step_progs.find(key);
  if (it == h->step_progs.end()) {
    StepPhase *d = nullptr;
    TRY(dalloc(h, &d, prog.size()));
    CK(cudaMemcpy(d, prog.data(), prog.size() * sizeof(StepPhase), cudaMemcpyHostToDevice));
    it = h->step_progs.emplace(key, d).first;
  }
  StepArgs a;
  memset(&a, 0, sizeof a);
  a.ph = it->second;
  a.n_phases = (int)prog.size();
  a.T = T;
  a.n_clusters = h->step_clusters;
  a.sp = sp;
  a.bar = h->step_bar;
  a.err = h->dev_err;
  const int G = h->step_clusters * kStepCS;
  if (h->debug & FM_DEBUG_TRACE) {
    if (!h->step_trace || h->step_trace_phases < (int)prog.size()) {
      TRY(dalloc(h, &h->step_trace, (size_t)prog.size() * G * kStepTraceSlots));
      h->step_trace_phases = (int)prog.size();
    }
    CK(cudaMemsetAsync(h->step_trace, 0, (size_t)prog.size() * G * kStepTraceSlots * 8, s));
    a.trace = h->step_trace;
  }
  ProfScope ps(h, s, "draft_step", bytes);
  CK(launch_step(a, h->step_clusters, s, h->step_attrs));
  ++h->last_launches;
  return FM_OK;
}

fm_status flashmap_draft_launch(fm_handle *h, int seq, int pos, const StepParams *sp, int n_pend, cudaStream_t s) {
  const fm_config &c = h->cfg;
  const int D = c.dim, B = c.block, L = c.n_layers, Ht = c.target_dim, F = c.ff_dim;
  const FlashMapPlan pl = flashmap_plan(h, seq, sp, n_pend);
  TRY(run_gemv(h, pl.anchor, s, "gemv.anchor_proj", 1));
  TRY(run_gemv(h, pl.kv, s, n_pend ? "gemv.kv_fused" : "gemv.kv_anchor", n_pend + 1));

  if (h->use_step) {
    std::vector<StepPhase> prog;
    if (flashmap_step_program(h, seq, pl, prog)) {
      // algorithmic bytes: every weight of the layers and the head once, the keys and values read once
      // (q/k/v 3 D^2, o, cross q, cross o D^2 each, fc1 and fc2 F D per layer; the head Ht D; bf16)
      const double bytes = 2.0 * ((double)L * (6.0 * D * D + 2.0 * F * D) + (double)Ht * D) +
                           (double)L * (pos + 1) * D * 2 * 2;
      TRY(run_step(h, seq, prog, sp, B, bytes, s));
      return run_lmhead(h, h->Y, B, sp, nullptr, nullptr, s, h->ylm);
    }
  }

  for (int l = 0; l < L; ++l) {
    TRY(run_gemv(h, pl.qkv[l], s, "gemv.qkv_self"));
    TRY(run_gemv(h, pl.o[l], s, "gemv.o_self"));
    TRY(run_gemv(h, pl.cq[l], s, "gemv.q_cross"));
    TRY(run_attn(h, h->qc, D, h->kv(seq, l), B, 1, 0, pos + 1, sp, h->attn, s));
    TRY(run_gemv(h, pl.co[l], s, "gemv.o_cross"));
    TRY(run_gemv(h, pl.f1[l], s, "gemv.fc1"));
    TRY(run_gemv(h, pl.f2[l], s, "gemv.fc2"));
    if (h->debug & FM_DEBUG_KEEP_HIDDEN) {
      CK(cudaMemcpyAsync(h->hid + (size_t)l * kMaxT * D, h->X, (size_t)B * D * 4, cudaMemcpyDeviceToDevice, s));
    }
  }
  TRY(run_gemv(h, pl.head, s, "gemv.head"));
  return run_lmhead(h, h->Y, B, sp, nullptr, nullptr, s, h->ylm);
}

// ---------------------------------------------------------------- DFlash

// Eq 2 and the retained per-layer context K / V (projectContextRows)
fm_status dflash_append_rows(fm_handle *h, int seq, const StepParams *sp, cudaStream_t s) {
  const fm_config &c = h->cfg;
  const int d = c.dim, FW = c.n_taps * c.target_dim;
  GemvArgs a = gemv_base(h, h->w_c, d, FW, 0, sp);
  a.amode = A_PLAIN;
  a.x_from_sp = 1;
  a.ldx = FW;
  a.emode = E_STORE;
  a.Y = h->ctx;
  a.ldy = d;
  a.out_st = h->st_c;
  a.st_w = h->ctx_norm;
  TRY(run_gemv(h, a, s, "gemv.wc", 32));

  GemvArgs b = gemv_base(h, h->w_kvall, c.n_layers * 2 * d, d, 0, sp);
  b.amode = A_RMS2;
  b.X = h->ctx;
  b.ldx = d;
  b.st = h->st_c;
  b.st_tiles = d / kTile;
  b.nw = h->ctx_norm;
  b.nw2 = h->attn_norm;
  b.nw_rows = 2 * d;
  b.inv_n = 1.0f / d;
  b.emode = E_SEGS;
  b.seg_rows = d;
  b.n_segs = 2 * c.n_layers;
  b.pos_src = 1;
  for (int l = 0; l < c.n_layers; ++l) {
    Seg2 kv = h->kv(seq, l);
    b.segs[2 * l] = {SEG_CACHE, 0, 0, 0, nullptr, kv.k};
    b.segs[2 * l + 1] = {SEG_CACHE, 0, 0, 0, nullptr, kv.v};
  }
  return run_gemv(h, b, s, "gemv.kv_append", 32);
}

// The sequential head after the parallel block: the lm_head stores the block's
// base logits, then position k = 0 .. block-1 in turn adds its bias (Markov:
// markov.w1[prev] markov.w2; RNN: the recurrent state through rnn.wO) and takes
// the argmax, which is position k + 1's prev; the confidence head and the
// pruning decision ride on the same launch.  Positions after a pruned one see
// the decided flag and return at once.
fm_status dflash_seq_head(fm_handle *h, int seq, const StepParams *sp, cudaStream_t s) {
  const fm_config &c = h->cfg;
  const int G = c.block, V = c.vocab, r = h->seq_rank;
  fm_handle::Lane &ln = h->lanes[seq];
  TRY(run_lmhead(h, h->Y, G, sp, ln.seq_flags + 4, ln.seq_base, s, h->ylm));
  CK(launch_seq_init(ln.seq_flags, G, s));
  ++h->last_launches;
  SeqArgs q{};
  q.base = ln.seq_base;
  q.V = V;
  q.r = r;
  q.d = c.dim;
  q.w1 = h->seq_w1;
  q.W = h->seq_W;
  q.sp = sp;
  q.part = ln.seq_part;
  q.ticket = ln.seq_flags + 2;
  q.flags = ln.seq_flags;
  q.conf_w = h->conf_w;
  q.conf_b = h->conf_b;
  q.X = h->X;
  q.out_norm = h->out_norm;
  q.eps = c.rms_eps;
  q.T = G;
  for (int k = 0; k < G; ++k) {
    if (h->seq_wH) {
      RnnArgs ra{};
      ra.w1 = h->seq_w1;
      ra.wH = h->seq_wH;
      ra.bH = h->seq_bH;
      ra.s_in = ln.seq_state + (size_t)((k + 1) & 1) * r;
      ra.s_out = ln.seq_state + (size_t)(k & 1) * r;
      ra.r = r;
      ra.k = k;
      ra.sp = sp;
      ra.flags = ln.seq_flags;
      ProfScope ps(h, s, "seq.rnn", (double)r * r * 2 + (double)r * 2 * 2);
      CK(launch_rnn_step(ra, s));
      ++h->last_launches;
      q.state = ra.s_out;
    }
    q.k = k;
    ProfScope ps(h, s, "seq.bias_argmax", (double)r * V * 2 + (double)V * 4);
    CK(launch_seq_bias_argmax(q, s));
    ++h->last_launches;
  }
  return FM_OK;
}

fm_status dflash_draft_launch(fm_handle *h, int seq, int pos, const StepParams *sp, cudaStream_t s) {
  const fm_config &c = h->cfg;
  const int d = c.dim, G = c.block, H = c.target_dim, F = c.ff_dim, L = c.n_layers;

  // block row 0 = tok_proj(E[anchor]) + block_pos[0]; rows 1.. are constants
  GemvArgs a = gemv_base(h, h->w_tok, d, H, 1, sp);
  a.amode = c.lm_format == FM_LM_Q8_0 ? A_ROW_Q8 : A_ROW_BF16;
  a.tq8 = h->tq8;
  a.tb = h->tb;
  a.emode = E_STORE;
  a.bias = h->block_pos;
  a.Y = h->hinit;
  a.ldy = d;
  a.out_st = h->st_init;
  TRY(run_gemv(h, a, s, "gemv.tok_proj", 1));

  for (int l = 0; l < L; ++l) {
    const bool first = l == 0;
    Seg2 kv = h->kv(seq, l);
    GemvArgs q = gemv_base(h, h->w_qkv[l], 3 * d, d, G, sp);
    q.amode = A_RMS;
    q.X = first ? h->hinit : h->X;
    q.ldx = d;
    q.st = first ? h->st_init : h->st_x;
    q.st_tiles = d / kTile;
    q.nw = h->attn_norm + (size_t)l * d;
    q.inv_n = 1.0f / d;
    q.emode = E_SEGS;
    q.Y = h->qc;
    q.ldy = d;
    q.seg_rows = d;
    q.n_segs = 3;
    q.segs[0] = {SEG_F32, 0, 0, 0, nullptr, nullptr};
    q.segs[1] = {SEG_CACHE, 0, 0, 0, nullptr, kv.k};
    q.segs[2] = {SEG_CACHE, 0, 0, 0, nullptr, kv.v};
    q.pos_src = 2;
    q.pos_add = 0;
    TRY(run_gemv(h, q, s, "gemv.qkv", G));

    TRY(run_attn(h, h->qc, d, kv, G, 0, G, pos + G, sp, h->attn, s));

    GemvArgs o = gemv_base(h, h->w_o[l], d, d, G, sp);
    o.amode = A_PLAIN;
    o.X = h->attn;
    o.ldx = d;
    o.emode = E_RESID;
    o.R = first ? h->hinit : h->X;
    o.ldr = d;
    o.Y = h->X;
    o.ldy = d;
    o.out_st = h->st_x;
    TRY(run_gemv(h, o, s, "gemv.o", G));

    GemvArgs gu = gemv_base(h, h->w_gu[l], 2 * F, d, G, sp);
    gu.amode = A_RMS;
    gu.X = h->X;
    gu.ldx = d;
    gu.st = h->st_x;
    gu.st_tiles = d / kTile;
    gu.nw = h->ff_norm + (size_t)l * d;
    gu.inv_n = 1.0f / d;
    gu.emode = E_GEGLU;
    gu.Y = h->u;
    gu.ldy = F;
    TRY(run_gemv(h, gu, s, "gemv.gate_up", G));

    GemvArgs dn = gemv_base(h, h->w_down[l], d, F, G, sp);
    dn.amode = A_PLAIN;
    dn.X = h->u;
    dn.ldx = F;
    dn.emode = E_RESID;
    dn.R = h->X;
    dn.ldr = d;
    dn.Y = h->X;
    dn.ldy = d;
    dn.out_st = h->st_x;
    TRY(run_gemv(h, dn, s, "gemv.down", G));

    if (h->debug & FM_DEBUG_KEEP_HIDDEN) {
      CK(cudaMemcpyAsync(h->hid + (size_t)l * kMaxT * d, h->X, (size_t)G * d * 4, cudaMemcpyDeviceToDevice, s));
    }
  }
  GemvArgs op = gemv_base(h, h->w_out, H, d, G, sp);
  op.amode = A_RMS;
  op.X = h->X;
  op.ldx = d;
  op.st = h->st_x;
  op.st_tiles = d / kTile;
  op.nw = h->out_norm;
  op.inv_n = 1.0f / d;
  op.emode = E_STORE;
  op.Y = h->Y;
  op.ldy = H;
  op.ylm = h->ylm;
  op.ylm_f16 = c.lm_format == FM_LM_Q8_0;
  TRY(run_gemv(h, op, s, "gemv.out_proj", G));
  if (!h->seq_rank) return run_lmhead(h, h->Y, G, sp, nullptr, nullptr, s, h->ylm);
  return dflash_seq_head(h, seq, sp, s);
}

// ---------------------------------------------------------------- dense prefill

constexpr int kPrefillMin = 128;     // appends of at least this many rows use the tensor-core GEMMs
constexpr int kPrefillChunk = 16384; // rows per pass (bounds the scratch)

fm_status prefill_setup(fm_handle *h, cudaStream_t s) {
  if (h->pf_rows) return FM_OK;
  const fm_config &c = h->cfg;
  const int D = c.dim, FW = c.n_taps * c.target_dim, L = c.n_layers;
  if (D % 256) return fail(h, FM_ERR_UNSUPPORTED, "dense prefill needs dim % 256 == 0");
  const int rows = c.max_ctx < kPrefillChunk ? c.max_ctx : kPrefillChunk;
  if (!h->w_fc16) return fail(h, FM_ERR_UNSUPPORTED, "dense prefill weights were not prepared");
  TRY(dalloc(h, &h->pf_a, (size_t)rows * FW));
  TRY(dalloc(h, &h->pf_c, (size_t)rows * D));
  TRY(dalloc(h, &h->pf_st, (size_t)rows * (D / 256) * 4));   // up to 4 K-slice pieces per 256 columns
  TRY(dalloc(h, &h->pf_err, 4));
  CK(cudaMemsetAsync(h->pf_err, 0, 4, s));
  if (!make_tma_f16(&h->tm_wfc, h->w_fc16, D, FW, 256) || !make_tma_f16(&h->tm_wkv, h->w_kv16, (uint64_t)L * 2 * D, D, 256))
    return fail(h, FM_ERR_CUDA, "tensor map encoding failed");
  h->pf_rows = rows;
  return FM_OK;
}

// fc -> hidden_norm -> all layers' k / v for rows start .. start+n-1 on tcgen05
fm_status flashmap_prefill(fm_handle *h, int seq, const float *feats, int n, int start, cudaStream_t s) {
  TRY(prefill_setup(h, s));
  const fm_config &c = h->cfg;
  const int D = c.dim, FW = c.n_taps * c.target_dim, L = c.n_layers;
  for (int r0 = 0; r0 < n; r0 += h->pf_rows) {
    const int R = n - r0 < h->pf_rows ? n - r0 : h->pf_rows;
    {
      ProfScope ps(h, s, "prefill.f32_to_f16", (double)R * FW * 6);
      CK(launch_f32_to_f16(feats + (size_t)r0 * FW, h->pf_a, (size_t)R * FW, h->n_sm, s));
      ++h->last_launches;
    }
    TcGemmArgs g;
    memset(&g, 0, sizeof g);
    if (!make_tma_f16(&g.tma_a, h->pf_a, R, FW, 128)) return fail(h, FM_ERR_CUDA, "tensor map encoding failed");
    g.tma_b = h->tm_wfc;
    g.M = R;
    g.N = D;
    g.K = FW;
    g.epi = TC_EPI_FC;
    g.err = h->pf_err;
    g.colw = h->w_hn;
    g.out16 = h->pf_c;
    g.ldo = D;
    g.row_st = h->pf_st;
    g.st_ld = D / 256;
    {
      ProfScope ps(h, s, "prefill.gemm_fc", 2.0 * R * D * FW);
      CK(launch_tc_gemm(g, h->n_sm, s));
      ++h->last_launches;
    }
    TcGemmArgs k;
    memset(&k, 0, sizeof k);
    if (!make_tma_f16(&k.tma_a, h->pf_c, R, D, 128)) return fail(h, FM_ERR_CUDA, "tensor map encoding failed");
    k.tma_b = h->tm_wkv;
    k.M = R;
    k.N = L * 2 * D;
    k.K = D;
    k.epi = TC_EPI_KV;
    // the stacked K/V weights (L * 2 * D rows) outweigh the rows' A panel: the
    // CTAs in flight walk the row blocks of a 16 MB A panel under one B tile
    k.group_m = (int)((16u << 20) / ((size_t)128 * D * 2));
    if (k.group_m < 1) k.group_m = 1;
    k.err = h->pf_err;
    k.in_st = h->pf_st;
    k.in_st_n = D / 256;
    k.eps = c.rms_eps;
    k.inv_n = 1.0f / D;
    k.seg_cols = D;
    k.hd = c.head_dim;
    k.max_ctx = c.max_ctx;
    k.start = start + r0;
    k.rope = h->rope;
    k.qk_eps = c.qk_eps;
    k.kn_w = h->w_ckn;
    k.cache = h->kv(seq, 0).k;
    k.plane = h->cache_plane;
    {
      ProfScope ps(h, s, "prefill.gemm_kv", 2.0 * R * D * (2.0 * L * D));
      CK(launch_tc_gemm(k, h->n_sm, s));
      ++h->last_launches;
    }
  }
  // a bounded wait that gave up is reported, never hung
  int32_t flag = 0;
  CK(cudaMemcpyAsync(&flag, h->pf_err, 4, cudaMemcpyDeviceToHost, s));
  CK(cudaStreamSynchronize(s));
  if (flag) {
    cudaMemsetAsync(h->pf_err, 0, 4, s);
    return fail(h, FM_ERR_TIMEOUT, "prefill GEMM: a pipeline wait exceeded its budget");
  }
  return FM_OK;
}

// ---------------------------------------------------------------- chains

// Run one chain of launches.  The first time a key is seen the chain is
// captured into a CUDA graph on the capture stream (launches read their
// per-call values from a fixed device slot); later calls upload the values
// and replay the graph.  With FM_DEBUG_PROFILE the chain is launched directly.
template <typename Enqueue>
fm_status run_chain(fm_handle *h, uint64_t key, const StepParams &p, cudaStream_t s, Enqueue &&enqueue) {
  key |= (uint64_t)(h->narrow ? 1 : 0) << 55;   // the products' launch shapes depend on it
  if (h->use_graphs && !(h->debug & (FM_DEBUG_PROFILE | FM_DEBUG_TRACE))) {
    auto it = h->graphs.find(key);
    if (it == h->graphs.end()) {
      fm_handle::GraphEntry g;
      TRY(dalloc(h, &g.sp, 1));
      CK(cudaStreamBeginCapture(h->cap, cudaStreamCaptureModeRelaxed));
      const int before = h->last_launches;
      fm_status st = enqueue(g.sp, h->cap);
      cudaGraph_t graph = nullptr;
      cudaError_t e = cudaStreamEndCapture(h->cap, &graph);
      if (st != FM_OK) {
        if (graph) cudaGraphDestroy(graph);
        return st;
      }
      CK(e);
      e = cudaGraphInstantiate(&g.exec, graph, 0);
      cudaGraphDestroy(graph);
      CK(e);
      g.launches = h->last_launches - before;
      h->last_launches = before;
      it = h->graphs.emplace(key, g).first;
    }
    TRY(upload_params(h, p, it->second.sp, s));
    CK(cudaGraphLaunch(it->second.exec, s));
    h->last_launches += it->second.launches;
    return FM_OK;
  }
  fm_status st;
  const StepParams *sp = next_params(h, p, s, &st);
  if (!sp) return st;
  return enqueue(sp, s);
}

uint64_t chain_key(int kind, int seq, int T, int splits, int debug) {
  return ((uint64_t)kind << 56) | ((uint64_t)(uint32_t)seq << 24) | ((uint64_t)T << 12) | ((uint64_t)splits << 2) |
         (uint64_t)(debug & FM_DEBUG_KEEP_HIDDEN);
}

// Project the K/V rows of a deferred append (when no draft of that sequence
// follows it directly).
fm_status flush_pending(fm_handle *h, int seq, cudaStream_t s) {
  fm_handle::Lane &L = h->lanes[seq];
  if (!L.pending) return FM_OK;
  use_lane(h, seq);
  const int n = L.pend_n;
  StepParams p{};
  p.T = n;
  p.start = L.pend_start;
  L.pending = false;
  return run_chain(h, chain_key(4, seq, n, 0, 0), p, s, [&](const StepParams *sp, cudaStream_t st) {
    return run_gemv(h, flashmap_kv_args(h, seq, sp, 0, 0), st, "gemv.kv_append", n);
  });
}

// conf, length, thr: the sequential head's confidence outputs and pruning
// thresholds (thr[k] NaN: none), all optional
fm_status draft_one(fm_handle *h, int seq, int anchor, int pos, int32_t *tokens, cudaStream_t s,
                    float *conf = nullptr, int32_t *length = nullptr, const float *thr = nullptr) {
  const fm_config &c = h->cfg;
  fm_handle::Lane &lane = h->lanes[seq];
  if (h->wide.on) h->wide.row_of[seq] = -1;
  int n_pend = 0;
  if (lane.pending) {
    if (lane.pend_start + lane.pend_n == pos && c.variant == FM_VARIANT_FLASHMAP && lane.pend_n + 1 <= kMaxT) {
      n_pend = lane.pend_n;
    } else {
      TRY(flush_pending(h, seq, s));
    }
  }
  use_lane(h, seq);
  StepParams p{};
  p.start = n_pend ? lane.pend_start : 0;
  if (n_pend) lane.pending = false;
  // cache rows no kernel of this draft writes: below the pending rows / the anchor / the block
  p.stable = n_pend ? p.start : pos;
  p.T = c.block;
  p.pos = pos;
  p.anchor = anchor;
  p.tokens = tokens;
  p.conf = conf;
  p.length = length;
  for (int k = 0; k < 16; ++k) p.thr[k] = thr && k < c.block ? thr[k] : NAN;
  int L_now;
  if (c.variant == FM_VARIANT_FLASHMAP) {
    p.L = pos + 1;
    L_now = pos + 1;
  } else {
    p.L = pos;  // context rows 0 .. pos-1; the block's own keys go to rows pos .. pos+block-1
    L_now = pos + c.block;
  }
  const uint64_t key = chain_key(1, seq, c.block + 64 * n_pend, attn_splits(h, L_now), h->debug);
  return run_chain(h, key, p, s, [&](const StepParams *sp, cudaStream_t st) {
    return c.variant == FM_VARIANT_FLASHMAP ? flashmap_draft_launch(h, seq, pos, sp, n_pend, st)
                                            : dflash_draft_launch(h, seq, pos, sp, st);
  });
}

// ---------------------------------------------------------------- batched draft

// Several sequences drafting at once (flashmap_drafter.js ``draft`` per anchor;
// above 17 rows the page hands its products to ``runGemm``): the block rows of
// up to kWideSeqs sequences (16 each, 512 at most) go through every product as
// one tensor-core GEMM, so each weight and the token table are read once per
// pass instead of once per sequence.  Activations enter the tensor cores as
// f16 (one rounding per product, against the skinny path's hi + lo split);
// weights as f16 copies of the bf16 values and the Q8_0 table as f16(d * q).
constexpr int kWideMin = 4;   // sequences per call from which drafts take the batched path

bool wide_wanted(const fm_handle *h) {
  const fm_config &c = h->cfg;
  const char *e = getenv("FM_NO_WIDE");
  if (e && e[0] == '1') return false;
  const double cache_rows = (double)c.max_seqs * c.n_layers * 2 * c.n_heads * c.max_ctx;
  return c.variant == FM_VARIANT_FLASHMAP && c.max_seqs >= kWideMin && c.head_dim == 128 && c.dim % 256 == 0 &&
         c.ff_dim % 256 == 0 && c.target_dim % 256 == 0 && c.dim <= 4096 && c.max_ctx >= 128 &&
         cache_rows < 2147483647.0;
}

// A-operand buffer: [rows][cols] f16 with rows a multiple of 128 (whole TMA boxes)
fm_status wide_abuf(fm_handle *h, __half **p, CUtensorMap *m, int rows, int cols) {
  const int r = (rows + 127) / 128 * 128;
  TRY(dalloc(h, p, (size_t)r * cols));
  if (!make_tma_f16(m, *p, r, cols, 128)) return fail(h, FM_ERR_CUDA, "tensor map encoding failed");
  return FM_OK;
}

fm_status wide_weight(fm_handle *h, const __nv_bfloat16 *w, int N, int K, __half **out, CUtensorMap *m, cudaStream_t s) {
  TRY(dalloc(h, out, (size_t)N * K));
  CK(launch_bf16_to_f16(w, *out, (size_t)N * K, s));
  if (!make_tma_f16(m, *out, N, K, 256)) return fail(h, FM_ERR_CUDA, "tensor map encoding failed");
  return FM_OK;
}

// f16 copies of the layer weights (from the row-major bf16 staging copies,
// before they are tiled) and the batched path's buffers
fm_status create_wide(fm_handle *h, cudaStream_t s) {
  const fm_config &c = h->cfg;
  fm_handle::Wide &w = h->wide;
  const int D = c.dim, F = c.ff_dim, Ht = c.target_dim, L = c.n_layers, H = c.n_heads;
  const int ns = c.max_seqs < kWideSeqs ? c.max_seqs : kWideSeqs;
  const int T = ns * c.block;
  TRY(prefill_setup(h, s));
  w.qkv.resize(L); w.so.resize(L); w.cq.resize(L); w.co.resize(L); w.f1.resize(L); w.f2.resize(L);
  w.t_qkv.resize(L); w.t_so.resize(L); w.t_cq.resize(L); w.t_co.resize(L); w.t_f1.resize(L); w.t_f2.resize(L);
  for (int l = 0; l < L; ++l) {
    TRY(wide_weight(h, h->w_qkv[l], 3 * D, D, &w.qkv[l], &w.t_qkv[l], s));
    TRY(wide_weight(h, h->w_so[l], D, D, &w.so[l], &w.t_so[l], s));
    TRY(wide_weight(h, h->w_cq[l], D, D, &w.cq[l], &w.t_cq[l], s));
    TRY(wide_weight(h, h->w_co[l], D, D, &w.co[l], &w.t_co[l], s));
    TRY(wide_weight(h, h->w_f1[l], F, D, &w.f1[l], &w.t_f1[l], s));
    TRY(wide_weight(h, h->w_f2[l], D, F, &w.f2[l], &w.t_f2[l], s));
  }
  TRY(wide_weight(h, h->w_ap, D, Ht, &w.ap, &w.t_ap, s));
  TRY(wide_weight(h, h->w_head, Ht, D, &w.head, &w.t_head, s));
  if (!make_tma_f16(&w.t_table, w.table, w.Vn, Ht, 256)) return fail(h, FM_ERR_CUDA, "tensor map encoding failed");
  if (!make_cache_map(&w.t_cache, h->cache, c.max_seqs * L * 2 * H, c.max_ctx))
    return fail(h, FM_ERR_CUDA, "cache tensor map encoding failed");
  const int Tr = (T + 127) / 128 * 128;
  TRY(dalloc(h, &w.X, (size_t)Tr * D));
  TRY(dalloc(h, &w.br, (size_t)Tr * D));
  TRY(dalloc(h, &w.qkv_out, (size_t)Tr * 3 * D));
  TRY(dalloc(h, &w.qc, (size_t)Tr * D));
  TRY(dalloc(h, &w.Y, (size_t)Tr * Ht));
  TRY(dalloc(h, &w.kst, (size_t)128 * (D / 256) * 4));   // up to 4 K-slice pieces per 256 columns
  TRY(wide_abuf(h, &w.a16, &w.m_a16, T, D));
  TRY(wide_abuf(h, &w.o16, &w.m_o16, T, D));
  TRY(wide_abuf(h, &w.u16, &w.m_u16, T, F));
  TRY(wide_abuf(h, &w.y16, &w.m_y16, T, Ht));
  TRY(wide_abuf(h, &w.anc16, &w.m_anc16, ns, Ht));
  TRY(wide_abuf(h, &w.kin16, &w.m_kin16, ns, D));
  TRY(dalloc(h, &w.amax, (size_t)T * (w.Vn / 256)));
  TRY(dalloc(h, &w.xo, (size_t)ns * H * 8 * 16 * 128));
  TRY(dalloc(h, &w.xml, (size_t)ns * H * 8 * 16));
  TRY(dalloc(h, &w.xtickets, (size_t)ns * H));
  CK(cudaMemsetAsync(w.xtickets, 0, (size_t)ns * H * 4, s));
  const char *xs = getenv("FM_WIDE_XSPLITS");
  if (xs && atoi(xs) >= 1 && atoi(xs) <= 8) w.xsplits = atoi(xs);
  const char *mk = getenv("FM_WIDE_MAX_KSPLIT");
  if (mk && atoi(mk) >= 1 && atoi(mk) <= 4) w.max_ksplit = atoi(mk);
  const char *ts = getenv("FM_WIDE_TSTORE");
  w.tstore = !(ts && ts[0] == '0');
  TRY(dalloc(h, &w.par, 1));
  CK(cudaMallocHost(&w.par_host, sizeof(WideParams) * kParamSlots));
  w.rows_cap = h->pf_rows;
  TRY(dalloc(h, &w.rows, (size_t)2 * w.rows_cap));
  CK(cudaMallocHost(&w.rows_host, sizeof(int32_t) * 2 * w.rows_cap * kParamSlots));
  for (int i = 0; i < kParamSlots; ++i) {
    CK(cudaEventCreateWithFlags(&w.par_ev[i], cudaEventDisableTiming));
    CK(cudaEventCreateWithFlags(&w.rows_ev[i], cudaEventDisableTiming));
  }
  w.row_of.assign(c.max_seqs, -1);
  w.on = true;
  return FM_OK;
}

// device address of an int32 array inside the pass parameters
#define WIDE_FIELD(h, f) \
  reinterpret_cast<const int32_t *>(reinterpret_cast<const char *>((h)->wide.par) + offsetof(WideParams, f))

// one GEMM of the batched path: A [M][K] rows (map a) times the weight B [N][K] (map b)
TcGemmArgs wide_gemm(const fm_handle *h, const CUtensorMap &a, const CUtensorMap &b, int M, int N, int K, int epi) {
  TcGemmArgs g;
  memset(&g, 0, sizeof g);
  g.tma_a = a;
  g.tma_b = b;
  g.M = M;
  g.N = N;
  g.K = K;
  g.epi = epi;
  g.group_m = (M + 127) / 128;   // the row blocks that share a weight tile run side by side
  g.err = h->dev_err;
  // K slices (clusters of 2 or 4) fill the GPU when there are fewer tiles than SMs
  const int tiles = tc_gemm_tiles(M, N), nk = K / 64;
  int ks = 1;
  while (ks * 2 <= h->wide.max_ksplit && tiles * ks * 2 <= h->n_sm && ks * 2 <= nk) ks *= 2;
  g.ksplit = ks;
  g.hd = h->cfg.head_dim;
  g.max_ctx = h->cfg.max_ctx;
  g.rope = h->rope;
  g.qk_eps = h->cfg.qk_eps;
  return g;
}

fm_status run_tc(fm_handle *h, const TcGemmArgs &g, cudaStream_t s, const char *tag) {
  ProfScope ps(h, s, tag, 2.0 * g.M * g.N * g.K);   // GEMM records carry their FLOPs
  CK(launch_tc_gemm(g, h->n_sm, s));
  ++h->last_launches;
  return FM_OK;
}

// A single-output product of a batched pass stores its tile through tensor copies: the output's map
// covers the pass's rows, so a ragged last row block is clipped.
fm_status wide_tstore(fm_handle *h, TcGemmArgs &g, const void *out, int rows, int cols, bool f32) {
  if (!h->wide.tstore) return FM_OK;
  if (!make_tma_out(&g.tma_o, out, rows, cols, f32)) return fail(h, FM_ERR_CUDA, "tensor map encoding failed");
  g.tstore = 1;
  return FM_OK;
}

// A gated residual product: with tensor stores its tile is added into the residual stream X by tensor
// reduce-add copies (each element gets its one addend); otherwise it writes the branch to br, which the
// next adaLN adds.
fm_status wide_gated(fm_handle *h, TcGemmArgs &g, int T) {
  fm_handle::Wide &w = h->wide;
  g.ldo32 = h->cfg.dim;
  if (!w.tstore) {
    g.out32 = w.br;
    return FM_OK;
  }
  g.out32 = w.X;
  g.treduce = 1;
  return wide_tstore(h, g, w.X, T, h->cfg.dim, true);
}

// the residual stream takes the previous product's gated branch (when `add`), then adaLN
fm_status run_lnmod(fm_handle *h, const float *m, int T, bool add, cudaStream_t s) {
  const int D = h->cfg.dim;
  ProfScope ps(h, s, "wide.lnmod", (double)T * D * (add ? 14 : 6));
  CK(launch_wide_lnmod(h->wide.X, add ? h->wide.br : nullptr, D, T, m, m + D, h->cfg.ln_eps, h->wide.a16, s));
  ++h->last_launches;
  return FM_OK;
}

// The launches of one batched pass over n sequences (values from wide.par).
fm_status wide_chain(fm_handle *h, int n, int xs, cudaStream_t s) {
  const fm_config &c = h->cfg;
  fm_handle::Wide &w = h->wide;
  const int D = c.dim, B = c.block, Ht = c.target_dim, F = c.ff_dim, L = c.n_layers, H = c.n_heads;
  const int T = n * B;
  {
    ProfScope ps(h, s, "wide.prep", (double)T * D * 4 + (double)n * Ht * 4);
    CK(launch_wide_prep(h->h0, D, T, w.X, w.par, n, w.table, Ht, w.anc16, h->n_sm, s));
    ++h->last_launches;
  }
  // the anchors' context slots: anchor_proj + bias (anchor_norm folded in), then every layer's K / V at pos
  TcGemmArgs g = wide_gemm(h, w.m_anc16, w.t_ap, n, D, Ht, TC_EPI_FC);
  g.bias = h->b_ap;
  g.colw = h->w_an;
  g.out16 = w.kin16;
  g.ldo = D;
  g.row_st = w.kst;
  g.st_ld = D / 256 * g.ksplit;
  const int st_n = g.st_ld;
  TRY(run_tc(h, g, s, "wide.gemm_anchor_proj"));
  g = wide_gemm(h, w.m_kin16, h->tm_wkv, n, L * 2 * D, D, TC_EPI_KV);
  g.in_st = w.kst;
  g.in_st_n = st_n;
  g.eps = c.rms_eps;
  g.inv_n = 1.0f / D;
  g.seg_cols = D;
  g.kn_w = h->w_ckn;
  g.cache = h->cache;
  g.plane = h->cache_plane;
  g.row_seq = WIDE_FIELD(h, kv_seq);
  g.row_pos = WIDE_FIELD(h, kv_pos);
  g.seq_stride = (size_t)L * 2 * h->cache_plane;
  TRY(run_tc(h, g, s, "wide.gemm_kv_anchor"));
  for (int l = 0; l < L; ++l) {
    const float *ms = h->mod + (size_t)(3 * l + 0) * 3 * D;
    const float *mc = h->mod + (size_t)(3 * l + 1) * 3 * D;
    const float *mm = h->mod + (size_t)(3 * l + 2) * 3 * D;
    // self-attention over each sequence's block (the previous layer's MLP branch joins the stream first)
    TRY(run_lnmod(h, ms, T, l > 0 && !w.tstore, s));
    g = wide_gemm(h, w.m_a16, w.t_qkv[l], T, 3 * D, D, TC_EPI_SEGS);
    g.seg_cols = D;
    g.nw0 = h->w_sqn[l];
    g.nw1 = h->w_skn[l];
    g.out32 = w.qkv_out;
    g.ldo32 = 3 * D;
    g.row_pos = WIDE_FIELD(h, row_pos);
    TRY(wide_tstore(h, g, w.qkv_out, T, 3 * D, true));
    TRY(run_tc(h, g, s, "wide.gemm_qkv_self"));
    {
      ProfScope ps(h, s, "wide.attn_self", (double)T * D * 3 * 4 + (double)T * D * 2);
      CK(launch_wide_self_attn(w.qkv_out, D, B, n, H, w.o16, s));
      ++h->last_launches;
    }
    g = wide_gemm(h, w.m_o16, w.t_so[l], T, D, D, TC_EPI_GATED);
    g.gate = ms + 2 * D;
    TRY(wide_gated(h, g, T));
    TRY(run_tc(h, g, s, "wide.gemm_o_self"));
    // cross-attention over each sequence's own cache rows 0 .. pos
    TRY(run_lnmod(h, mc, T, !w.tstore, s));
    g = wide_gemm(h, w.m_a16, w.t_cq[l], T, D, D, TC_EPI_SEGS);
    g.seg_cols = D;
    g.nw0 = h->w_cqn[l];
    g.out32 = w.qc;
    g.ldo32 = D;
    g.row_pos = WIDE_FIELD(h, row_pos);
    TRY(wide_tstore(h, g, w.qc, T, D, true));
    TRY(run_tc(h, g, s, "wide.gemm_q_cross"));
    {
      XAttnArgs xa;
      memset(&xa, 0, sizeof xa);
      xa.tm_k = w.t_cache;
      xa.tm_v = w.t_cache;
      xa.Q = w.qc;
      xa.ldq = D;
      xa.max_ctx = c.max_ctx;
      xa.n_heads = H;
      xa.splits = xs;
      xa.T_const = B;
      xa.scale_log2 = (float)(1.4426950408889634 / std::sqrt(128.0));
      xa.out16 = w.o16;
      xa.ldo = D;
      xa.part_o = w.xo;
      xa.part_ml = w.xml;
      xa.tickets = w.xtickets;
      xa.err = h->dev_err;
      xa.bz_call = WIDE_FIELD(h, z_call);
      xa.bz_seq = WIDE_FIELD(h, z_seq);
      xa.bz_L = WIDE_FIELD(h, z_L);
      xa.n_z = n;
      xa.layer = l;
      xa.n_layers = L;
      ProfScope ps(h, s, "wide.attn_cross", w.keys * c.dim * 2 * 2 + 2.0 * T * D * (4 + 2));
      CK(launch_xattn(xa, 3, false, s, true));
      ++h->last_launches;
    }
    g = wide_gemm(h, w.m_o16, w.t_co[l], T, D, D, TC_EPI_GATED);
    g.gate = mc + 2 * D;
    TRY(wide_gated(h, g, T));
    TRY(run_tc(h, g, s, "wide.gemm_o_cross"));
    // MLP
    TRY(run_lnmod(h, mm, T, !w.tstore, s));
    g = wide_gemm(h, w.m_a16, w.t_f1[l], T, F, D, TC_EPI_F16);
    g.bias = h->b_f1[l];
    g.gelu = 1;
    g.out16 = w.u16;
    g.ldo = F;
    TRY(wide_tstore(h, g, w.u16, T, F, false));
    TRY(run_tc(h, g, s, "wide.gemm_fc1"));
    g = wide_gemm(h, w.m_u16, w.t_f2[l], T, D, F, TC_EPI_GATED);
    g.bias = h->b_f2[l];
    g.gate = mm + 2 * D;
    TRY(wide_gated(h, g, T));
    TRY(run_tc(h, g, s, "wide.gemm_fc2"));
  }
  // the last MLP branch joins the stream; final adaLN -> head -> lm_head with the per-row argmax
  TRY(run_lnmod(h, h->mod + (size_t)(3 * L) * 3 * D, T, !w.tstore, s));
  g = wide_gemm(h, w.m_a16, w.t_head, T, Ht, D, TC_EPI_F16);
  g.bias = h->b_head;
  g.out16 = w.y16;
  g.ldo = Ht;
  g.out32 = w.Y;
  g.ldo32 = Ht;
  TRY(run_tc(h, g, s, "wide.gemm_head"));
  g = wide_gemm(h, w.m_y16, w.t_table, T, w.Vn, Ht, TC_EPI_ARGMAX);
  g.amax = w.amax;
  g.amax_ld = w.Vn / 256;
  g.n_valid = c.vocab;
  TRY(run_tc(h, g, s, "wide.gemm_lm_head"));
  {
    ProfScope ps(h, s, "wide.argmax", (double)T * (w.Vn / 256) * 8);
    CK(launch_wide_argmax(w.amax, w.Vn / 256, T, w.par, s));
    ++h->last_launches;
  }
  return FM_OK;
}

// Capture a launch sequence into a CUDA graph the first time its key is seen,
// replay it afterwards (the per-call values travel through device buffers
// uploaded before the launch).
template <typename Enqueue>
fm_status run_graph(fm_handle *h, uint64_t key, cudaStream_t s, Enqueue &&enqueue) {
  if (!h->use_graphs || (h->debug & (FM_DEBUG_PROFILE | FM_DEBUG_TRACE))) return enqueue(s);
  auto it = h->graphs.find(key);
  if (it == h->graphs.end()) {
    fm_handle::GraphEntry g;
    CK(cudaStreamBeginCapture(h->cap, cudaStreamCaptureModeRelaxed));
    const int before = h->last_launches;
    fm_status st = enqueue(h->cap);
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(h->cap, &graph);
    if (st != FM_OK) {
      if (graph) cudaGraphDestroy(graph);
      return st;
    }
    CK(e);
    e = cudaGraphInstantiate(&g.exec, graph, 0);
    cudaGraphDestroy(graph);
    CK(e);
    g.launches = h->last_launches - before;
    h->last_launches = before;
    it = h->graphs.emplace(key, g).first;
  }
  CK(cudaGraphLaunch(it->second.exec, s));
  h->last_launches += it->second.launches;
  return FM_OK;
}

fm_status wide_upload(fm_handle *h, const WideParams &p, cudaStream_t s) {
  fm_handle::Wide &w = h->wide;
  const int i = w.par_next;
  w.par_next = (i + 1) % kParamSlots;
  cudaEventSynchronize(w.par_ev[i]);   // the slot's previous copy has been consumed
  w.par_host[i] = p;
  CK(cudaMemcpyAsync(w.par, w.par_host + i, sizeof(WideParams), cudaMemcpyHostToDevice, s));
  CK(cudaEventRecord(w.par_ev[i], s));
  return FM_OK;
}

// Batched draft of n sequences (arguments checked by the caller), in passes of kWideSeqs.
fm_status wide_draft(fm_handle *h, int n, const int32_t *ids, const int32_t *anchors, const int32_t *pos,
                     int32_t *tokens, cudaStream_t s) {
  const fm_config &c = h->cfg;
  fm_handle::Wide &w = h->wide;
  for (int i = 0; i < n; ++i) TRY(flush_pending(h, ids[i], s));
  for (int &r : w.row_of)
    if (r >= 0) r = -2;   // this call overwrites the head output of the previous batched call
  for (int p0 = 0; p0 < n; p0 += kWideSeqs) {
    const int m = n - p0 < kWideSeqs ? n - p0 : kWideSeqs;
    WideParams p;
    memset(&p, 0, sizeof p);
    p.n = m;
    p.tokens = tokens + (size_t)p0 * c.block;
    std::vector<int> order(m);
    for (int i = 0; i < m; ++i) {
      p.seq[i] = ids[p0 + i];
      p.anchor[i] = anchors[p0 + i];
      p.pos[i] = pos[p0 + i];
      p.kv_seq[i] = ids[p0 + i];
      p.kv_pos[i] = pos[p0 + i];
      for (int t = 0; t < c.block; ++t) p.row_pos[i * c.block + t] = pos[p0 + i] + 1 + t;
      order[i] = i;
    }
    // the cross-attention hands out its CTAs longest context first
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return p.pos[a] > p.pos[b]; });
    for (int z = 0; z < m; ++z) {
      p.z_call[z] = order[z];
      p.z_seq[z] = p.seq[order[z]];
      p.z_L[z] = p.pos[order[z]] + 1;
    }
    TRY(wide_upload(h, p, s));
    w.keys = 0;
    for (int i = 0; i < m; ++i) w.keys += p.pos[i] + 1;
    const int xs = w.xsplits;
    TRY(run_graph(h, chain_key(6, 0, m, xs, 0), s, [&](cudaStream_t st) { return wide_chain(h, m, xs, st); }));
    // the head output of the last pass stays readable; earlier passes' rows are overwritten (-2)
    for (int i = 0; i < m; ++i) w.row_of[ids[p0 + i]] = p0 + m == n ? i * c.block : -2;
  }
  return FM_OK;
}

// Batched append of small row counts: every row of every sequence through one
// fc GEMM and one K/V GEMM (per-row sequence and position), in chunks of the
// prefill scratch.  feats: the rows of sequence i start at feats + offs[i].
fm_status wide_append(fm_handle *h, int n, const int32_t *ids, const float *feats, const size_t *offs,
                      const int32_t *n_rows, const int32_t *start, cudaStream_t s) {
  const fm_config &c = h->cfg;
  fm_handle::Wide &w = h->wide;
  const int D = c.dim, FW = c.n_taps * c.target_dim, L = c.n_layers;
  for (int i = 0; i < n; ++i) TRY(flush_pending(h, ids[i], s));
  // rows in call order: (sequence index, row within it)
  std::vector<std::pair<int, int>> rows;
  for (int i = 0; i < n; ++i)
    for (int r = 0; r < n_rows[i]; ++r) rows.emplace_back(i, r);
  const int R = (int)rows.size();
  for (int r0 = 0; r0 < R; r0 += h->pf_rows) {
    const int Rc = R - r0 < h->pf_rows ? R - r0 : h->pf_rows;
    // f32 -> f16 rows, one launch per run of rows adjacent in the caller's buffer
    for (int a = 0; a < Rc;) {
      const float *src = feats + offs[rows[r0 + a].first] + (size_t)rows[r0 + a].second * FW;
      int b = a + 1;
      while (b < Rc && feats + offs[rows[r0 + b].first] + (size_t)rows[r0 + b].second * FW == src + (size_t)(b - a) * FW) ++b;
      ProfScope ps(h, s, "append.f32_to_f16", (double)(b - a) * FW * 6);
      CK(launch_f32_to_f16(src, h->pf_a + (size_t)a * FW, (size_t)(b - a) * FW, h->n_sm, s));
      ++h->last_launches;
      a = b;
    }
    // per-row targets
    const int slot = w.rows_next;
    w.rows_next = (slot + 1) % kParamSlots;
    cudaEventSynchronize(w.rows_ev[slot]);
    int32_t *hs = w.rows_host + (size_t)slot * 2 * w.rows_cap;
    for (int r = 0; r < Rc; ++r) {
      const int i = rows[r0 + r].first;
      hs[r] = ids[i];
      hs[w.rows_cap + r] = start[i] + rows[r0 + r].second;
    }
    CK(cudaMemcpyAsync(w.rows, hs, (size_t)Rc * 4, cudaMemcpyHostToDevice, s));
    CK(cudaMemcpyAsync(w.rows + w.rows_cap, hs + w.rows_cap, (size_t)Rc * 4, cudaMemcpyHostToDevice, s));
    CK(cudaEventRecord(w.rows_ev[slot], s));
    // whole 128-row boxes: the maps span at least 128 rows of the scratch (rows past Rc are masked)
    const int Rm = Rc < 128 ? 128 : Rc;
    CUtensorMap ma;
    if (!make_tma_f16(&ma, h->pf_a, Rm, FW, 128)) return fail(h, FM_ERR_CUDA, "tensor map encoding failed");
    TcGemmArgs g = wide_gemm(h, ma, h->tm_wfc, Rc, D, FW, TC_EPI_FC);
    g.colw = h->w_hn;
    g.out16 = h->pf_c;
    g.ldo = D;
    g.row_st = h->pf_st;
    g.st_ld = D / 256 * g.ksplit;
    const int st_n = g.st_ld;
    TRY(run_tc(h, g, s, "append.gemm_fc"));
    CUtensorMap mc;
    if (!make_tma_f16(&mc, h->pf_c, Rm, D, 128)) return fail(h, FM_ERR_CUDA, "tensor map encoding failed");
    g = wide_gemm(h, mc, h->tm_wkv, Rc, L * 2 * D, D, TC_EPI_KV);
    g.in_st = h->pf_st;
    g.in_st_n = st_n;
    g.eps = c.rms_eps;
    g.inv_n = 1.0f / D;
    g.seg_cols = D;
    g.kn_w = h->w_ckn;
    g.cache = h->cache;
    g.plane = h->cache_plane;
    g.row_seq = w.rows;
    g.row_pos = w.rows + w.rows_cap;
    g.seq_stride = (size_t)L * 2 * h->cache_plane;
    TRY(run_tc(h, g, s, "append.gemm_kv"));
  }
  for (int i = 0; i < n; ++i) h->length[ids[i]] = start[i] + n_rows[i];
  return FM_OK;
}

// ---------------------------------------------------------------- create

fm_status check_config(fm_handle *h, const fm_config &c) {
  if (c.variant != FM_VARIANT_FLASHMAP && c.variant != FM_VARIANT_DFLASH)
    return fail(h, FM_ERR_INVALID_ARG, "unknown variant %d", c.variant);
  if (c.head_dim != 64 && c.head_dim != 128) return fail(h, FM_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (c.n_heads < 1 || c.n_heads * c.head_dim != c.dim) return fail(h, FM_ERR_INVALID_ARG, "dim != n_heads * head_dim");
  if (c.dim % kTile || c.ff_dim % kTile || c.dim < kTile)
    return fail(h, FM_ERR_UNSUPPORTED, "dim and ff_dim must be multiples of 128");
  if (c.target_dim % 64 || c.target_dim < 64) return fail(h, FM_ERR_UNSUPPORTED, "target_dim must be a multiple of 64");
  if (c.n_taps < 1) return fail(h, FM_ERR_INVALID_ARG, "n_taps < 1");
  if (c.n_layers < 1 || c.n_layers > kMaxSegs / 2)
    return fail(h, FM_ERR_UNSUPPORTED, "n_layers must be in 1..%d", kMaxSegs / 2);
  if (c.block < 1 || c.block > 16) return fail(h, FM_ERR_UNSUPPORTED, "block must be in 1..16");
  if (c.vocab < 1) return fail(h, FM_ERR_INVALID_ARG, "vocab < 1");
  if (c.lm_format != FM_LM_BF16 && c.lm_format != FM_LM_Q8_0) return fail(h, FM_ERR_INVALID_ARG, "lm_format");
  if (c.max_seqs < 1) return fail(h, FM_ERR_INVALID_ARG, "max_seqs < 1");
  if (c.max_ctx < c.block + 2) return fail(h, FM_ERR_INVALID_ARG, "max_ctx < block + 2");
  if (c.target_dim > 3072)
    return fail(h, FM_ERR_UNSUPPORTED, "target_dim above 3072 (the lm_head keeps the slot rows in shared memory)");
  return FM_OK;
}

fm_status create_common(fm_handle *h, cudaStream_t s) {
  const fm_config &c = h->cfg;
  const int D = c.dim, Ht = c.target_dim, F = c.ff_dim;
  h->length.assign(c.max_seqs, 0);
  h->cache_plane = (size_t)c.n_heads * c.max_ctx * c.head_dim;
  TRY(dalloc(h, &h->cache, (size_t)c.max_seqs * c.n_layers * 2 * h->cache_plane));
  CK(cudaMemsetAsync(h->cache, 0, (size_t)c.max_seqs * c.n_layers * 2 * h->cache_plane * 2, s));
  h->rope_pos = c.max_ctx + c.block + 2;
  TRY(dalloc(h, &h->rope, (size_t)h->rope_pos * c.head_dim / 2));
  CK(launch_rope_table(h->rope, h->rope_pos, c.head_dim, c.rope_theta, s));
  const int wmax = 3 * D > F ? (3 * D > Ht ? 3 * D : Ht) : (F > Ht ? F : Ht);
  const int tiles_max = (wmax + kTile - 1) / kTile + 64;
  h->lanes.resize(c.max_seqs);
  for (int i = 0; i < c.max_seqs; ++i) {
    fm_handle::Lane &L = h->lanes[i];
    TRY(dalloc(h, &L.X, (size_t)kMaxT * D));
    TRY(dalloc(h, &L.qkv, (size_t)kMaxT * 3 * D));
    TRY(dalloc(h, &L.qc, (size_t)kMaxT * D));
    TRY(dalloc(h, &L.attn, (size_t)kMaxT * D));
    TRY(dalloc(h, &L.u, (size_t)kMaxT * (F > wmax ? F : wmax)));
    TRY(dalloc(h, &L.Y, (size_t)kMaxT * Ht));
    // the head's output also split into the lm_head operand; rows of unused slots stay zero
    TRY(dalloc(h, &L.ylm, (size_t)(Ht / 64) * kLmYChunk));
    CK(cudaMemsetAsync(L.ylm, 0, (size_t)(Ht / 64) * kLmYChunk, s));
    TRY(dalloc(h, &L.ctx, (size_t)kMaxT * D));
    TRY(dalloc(h, &L.actx, (size_t)kMaxT * D));
    CK(cudaMemsetAsync(L.X, 0, (size_t)kMaxT * D * 4, s));
    float2 **sts[] = {&L.st_x, &L.st_c, &L.st_a, &L.st_u};
    for (float2 **p : sts) {
      TRY(dalloc(h, p, (size_t)tiles_max * kMaxT));
      CK(cudaMemsetAsync(*p, 0, (size_t)tiles_max * kMaxT * sizeof(float2), s));
    }
    TRY(dalloc(h, &L.lm_part, (size_t)h->n_sm * kMaxT));
    TRY(dalloc(h, &L.tickets, (size_t)2 * c.n_heads + 8));
    CK(cudaMemsetAsync(L.tickets, 0, ((size_t)2 * c.n_heads + 8) * 4, s));
    if (c.head_dim == 128) {
      TRY(dalloc(h, &L.xo, (size_t)c.n_heads * kMaxXSplits * 16 * 128));
      TRY(dalloc(h, &L.xml, (size_t)c.n_heads * kMaxXSplits * 16));
      TRY(dalloc(h, &L.xtickets, (size_t)c.n_heads));
      CK(cudaMemsetAsync(L.xtickets, 0, (size_t)c.n_heads * 4, s));
    }
    if (c.max_seqs > 1) {
      CK(cudaStreamCreateWithFlags(&L.stream, cudaStreamNonBlocking));
      CK(cudaEventCreateWithFlags(&L.done, cudaEventDisableTiming));
    }
  }
  if (c.max_seqs > 1) CK(cudaEventCreateWithFlags(&h->fork_ev, cudaEventDisableTiming));
  use_lane(h, 0);
  TRY(dalloc(h, &h->hid, (size_t)c.n_layers * kMaxT * D));
  CK(cudaMemsetAsync(h->hid, 0, (size_t)c.n_layers * kMaxT * D * 4, s));
  float2 **sts[] = {&h->st_h0, &h->st_init};
  for (float2 **p : sts) {
    TRY(dalloc(h, p, (size_t)tiles_max * kMaxT));
    CK(cudaMemsetAsync(*p, 0, (size_t)tiles_max * kMaxT * sizeof(float2), s));
  }
  h->max_splits = 2 * h->n_sm / c.n_heads;
  if (h->max_splits < 1) h->max_splits = 1;
  if (c.head_dim == 128) {
    // cross-attention clusters: the largest size (<= 16) of which all n_heads clusters are co-resident
    h->xattn_cluster = 0;
    for (int cs = 16; cs >= 1 && !h->xattn_cluster; --cs)
      if (xattn_max_active_clusters(cs, c.n_heads) >= c.n_heads) h->xattn_cluster = cs;
  }
  TRY(dalloc(h, &h->tok_tmp, (size_t)kMaxT));
  TRY(dalloc(h, &h->dev_err, 4));
  CK(cudaMemsetAsync(h->dev_err, 0, 4, s));
  TRY(dalloc(h, &h->step_bar, 64));
  CK(cudaMemsetAsync(h->step_bar, 0, 64 * 4, s));
  TRY(dalloc(h, &h->sp_dev, kParamSlots));
  CK(cudaMallocHost(&h->sp_host, sizeof(StepParams) * kParamSlots));
  memset(h->sp_host, 0, sizeof(StepParams) * kParamSlots);
  for (int i = 0; i < kParamSlots; ++i) CK(cudaEventCreateWithFlags(&h->sp_ev[i], cudaEventDisableTiming));
  CK(cudaStreamCreateWithFlags(&h->cap, cudaStreamNonBlocking));
  const char *g = getenv("FM_NO_GRAPHS");
  h->use_graphs = !(g && g[0] == '1');
  const char *df = getenv("FM_NO_DEFER");
  h->use_defer = !(df && df[0] == '1');
  const char *pf = getenv("FM_NO_TC_PREFILL");
  h->use_prefill = !(pf && pf[0] == '1');
  // the persistent draft step needs one co-resident CTA per SM; an empty program
  // finds the launch attributes the device takes (outside any stream capture)
  const char *ps = getenv("FM_PERSISTENT");
  h->step_clusters = c.variant == FM_VARIANT_FLASHMAP ? step_max_clusters() : 0;
  h->use_step = (ps && ps[0] == '1') && h->step_clusters >= 1;
  if (h->use_step) {
    StepArgs a;
    memset(&a, 0, sizeof a);
    a.n_clusters = h->step_clusters;
    a.bar = h->step_bar;
    a.err = h->dev_err;
    h->step_attrs = -1;
    for (int attrs : {3, 1, 2, 0}) {
      if (launch_step(a, h->step_clusters, s, attrs) == cudaSuccess && cudaStreamSynchronize(s) == cudaSuccess) {
        h->step_attrs = attrs;
        break;
      }
      cudaGetLastError();
    }
    if (h->step_attrs < 0) h->use_step = false;
  }
  return FM_OK;
}

fm_status create_table(fm_handle *h, const TensorSet &ts, cudaStream_t s) {
  const fm_config &c = h->cfg;
  const int V = c.vocab, H = c.target_dim;
  h->Vpad = (V + kTile - 1) / kTile * kTile;
  TRY(dalloc(h, &h->uni, H));
  if (c.lm_format == FM_LM_Q8_0) {
    const fm_tensor *t;
    TRY(find(h, ts, "token_embd.weight", (int64_t)V * (H / 32) * 34, FM_DTYPE_Q8_0, true, &t));
    uint8_t *raw;
    TRY(dalloc(h, &raw, (size_t)V * (H / 32) * 34));
    CK(cudaMemcpyAsync(raw, t->data, (size_t)V * (H / 32) * 34, cudaMemcpyDefault, s));
    TRY(dalloc(h, &h->tq8, q8_table_bytes(V, H)));
    CK(launch_q8_repack(raw, V, H, h->tq8, s));
    CK(launch_colmean_q8(raw, V, H, h->uni, s));
    if (wide_wanted(h)) {
      h->wide.Vn = (V + 255) / 256 * 256;
      TRY(dalloc(h, &h->wide.table, (size_t)h->wide.Vn * H));
      CK(launch_q8_to_f16(raw, V, H, h->wide.Vn, h->wide.table, s));
    }
    dfree_later(h, raw);
  } else {
    __nv_bfloat16 *tb;
    TRY(dalloc(h, &tb, (size_t)V * H));
    TRY(put_bf16(h, ts, "token_embd.weight", tb, (int64_t)V * H, s));
    CK(launch_colmean_bf16(tb, V, H, h->uni, s));
    if (wide_wanted(h)) {
      h->wide.Vn = (V + 255) / 256 * 256;
      TRY(dalloc(h, &h->wide.table, (size_t)h->wide.Vn * H));
      CK(launch_bf16_to_f16_pad(tb, V, H, h->wide.Vn, h->wide.table, s));
    }
    TRY(tile_weight(h, &tb, V, H, s));
    h->tb = reinterpret_cast<uint8_t *>(tb);
  }
  return FM_OK;
}

fm_status create_flashmap(fm_handle *h, const TensorSet &ts, const float *modulation, cudaStream_t s) {
  const fm_config &c = h->cfg;
  const int D = c.dim, Ht = c.target_dim, F = c.ff_dim, L = c.n_layers, hd = c.head_dim;
  const int FW = c.n_taps * Ht;
  if (!modulation) return fail(h, FM_ERR_INVALID_ARG, "FlashMap needs the modulation table");
  TRY(create_table(h, ts, s));
  TRY(dalloc(h, &h->w_fc, (size_t)D * FW));
  TRY(put_bf16(h, ts, "fc.weight", h->w_fc, (int64_t)D * FW, s));
  TRY(dalloc(h, &h->w_hn, D));
  TRY(put_bf16(h, ts, "hidden_norm.weight", h->w_hn, D, s));
  TRY(dalloc(h, &h->w_ap, (size_t)D * Ht));
  TRY(put_bf16(h, ts, "anchor_proj.weight", h->w_ap, (int64_t)D * Ht, s));
  TRY(dalloc(h, &h->b_ap, D));
  TRY(put_bf16(h, ts, "anchor_proj.bias", h->b_ap, D, s, true));
  TRY(dalloc(h, &h->w_an, D));
  TRY(put_bf16(h, ts, "anchor_norm.weight", h->w_an, D, s));
  TRY(dalloc(h, &h->w_sn, Ht));
  TRY(put_bf16(h, ts, "state_norm.weight", h->w_sn, Ht, s));
  TRY(dalloc(h, &h->w_xe, (size_t)D * Ht));
  TRY(put_bf16(h, ts, "x_embed.weight", h->w_xe, (int64_t)D * Ht, s));
  TRY(dalloc(h, &h->b_xe, D));
  TRY(put_bf16(h, ts, "x_embed.bias", h->b_xe, D, s, true));
  TRY(dalloc(h, &h->w_head, (size_t)Ht * D));
  TRY(put_bf16(h, ts, "head.weight", h->w_head, (int64_t)Ht * D, s));
  TRY(dalloc(h, &h->b_head, Ht));
  TRY(put_bf16(h, ts, "head.bias", h->b_head, Ht, s, true));
  TRY(dalloc(h, &h->w_kvall, (size_t)L * 2 * D * D));
  TRY(dalloc(h, &h->w_ckn, (size_t)L * hd));
  const size_t DD = (size_t)D * D;
  for (int l = 0; l < L; ++l) {
    const std::string p = "layers." + std::to_string(l) + ".";
    __nv_bfloat16 *w;
    TRY(dalloc(h, &w, 3 * DD));
    TRY(put_bf16(h, ts, p + "self_attn.q_proj.weight", w, DD, s));
    TRY(put_bf16(h, ts, p + "self_attn.k_proj.weight", w + DD, DD, s));
    TRY(put_bf16(h, ts, p + "self_attn.v_proj.weight", w + 2 * DD, DD, s));
    h->w_qkv.push_back(w);
    TRY(dalloc(h, &w, hd));
    TRY(put_bf16(h, ts, p + "self_attn.q_norm.weight", w, hd, s));
    h->w_sqn.push_back(w);
    TRY(dalloc(h, &w, hd));
    TRY(put_bf16(h, ts, p + "self_attn.k_norm.weight", w, hd, s));
    h->w_skn.push_back(w);
    TRY(dalloc(h, &w, DD));
    TRY(put_bf16(h, ts, p + "self_attn.o_proj.weight", w, DD, s));
    h->w_so.push_back(w);
    TRY(dalloc(h, &w, DD));
    TRY(put_bf16(h, ts, p + "cross_attn.q_proj.weight", w, DD, s));
    h->w_cq.push_back(w);
    TRY(put_bf16(h, ts, p + "cross_attn.k_proj.weight", h->w_kvall + (size_t)(2 * l) * DD, DD, s));
    TRY(put_bf16(h, ts, p + "cross_attn.v_proj.weight", h->w_kvall + (size_t)(2 * l + 1) * DD, DD, s));
    TRY(dalloc(h, &w, hd));
    TRY(put_bf16(h, ts, p + "cross_attn.q_norm.weight", w, hd, s));
    h->w_cqn.push_back(w);
    TRY(put_bf16(h, ts, p + "cross_attn.k_norm.weight", h->w_ckn + (size_t)l * hd, hd, s));
    TRY(dalloc(h, &w, DD));
    TRY(put_bf16(h, ts, p + "cross_attn.o_proj.weight", w, DD, s));
    h->w_co.push_back(w);
    TRY(dalloc(h, &w, (size_t)F * D));
    TRY(put_bf16(h, ts, p + "mlp.fc1.weight", w, (int64_t)F * D, s));
    h->w_f1.push_back(w);
    TRY(dalloc(h, &w, F));
    TRY(put_bf16(h, ts, p + "mlp.fc1.bias", w, F, s, true));
    h->b_f1.push_back(w);
    TRY(dalloc(h, &w, (size_t)D * F));
    TRY(put_bf16(h, ts, p + "mlp.fc2.weight", w, (int64_t)D * F, s));
    h->w_f2.push_back(w);
    TRY(dalloc(h, &w, D));
    TRY(put_bf16(h, ts, p + "mlp.fc2.bias", w, D, s, true));
    h->b_f2.push_back(w);
  }
  const size_t nmod = (size_t)(3 * L + 1) * 3 * D;
  TRY(dalloc(h, &h->mod, nmod));
  CK(cudaMemcpyAsync(h->mod, modulation, nmod * 4, cudaMemcpyDefault, s));
  TRY(create_common(h, s));

  // f16 row-major copies for the dense prefill, then every GEMV weight to its tile layout
  if (D % 256 == 0 && c.max_ctx >= 128) {
    TRY(dalloc(h, &h->w_fc16, (size_t)D * FW));
    TRY(dalloc(h, &h->w_kv16, (size_t)L * 2 * D * D));
    CK(launch_bf16_to_f16(h->w_fc, h->w_fc16, (size_t)D * FW, s));
    CK(launch_bf16_to_f16(h->w_kvall, h->w_kv16, (size_t)L * 2 * D * D, s));
  }
  if (wide_wanted(h)) TRY(create_wide(h, s));
  TRY(tile_weight(h, &h->w_fc, D, FW, s));
  TRY(tile_weight(h, &h->w_ap, D, Ht, s));
  TRY(tile_weight(h, &h->w_xe, D, Ht, s));
  TRY(tile_weight(h, &h->w_head, Ht, D, s));
  TRY(tile_weight(h, &h->w_kvall, L * 2 * D, D, s));
  for (int l = 0; l < L; ++l) {
    TRY(tile_weight(h, &h->w_qkv[l], 3 * D, D, s));
    TRY(tile_weight(h, &h->w_so[l], D, D, s));
    TRY(tile_weight(h, &h->w_cq[l], D, D, s));
    TRY(tile_weight(h, &h->w_co[l], D, D, s));
    TRY(tile_weight(h, &h->w_f1[l], F, D, s));
    TRY(tile_weight(h, &h->w_f2[l], D, F, s));
  }

  // h0 = x_embed(state_norm(mean row of E)) + bias, and its row statistics
  TRY(dalloc(h, &h->h0, D));
  CK(launch_row_stats(h->uni, 1, Ht, h->st_u, s));
  StepParams p{};
  p.T = 1;
  fm_status st;
  const StepParams *sp = next_params(h, p, s, &st);
  if (!sp) return st;
  GemvArgs a = gemv_base(h, h->w_xe, D, Ht, 1, sp);
  a.amode = A_RMS;
  a.X = h->uni;
  a.ldx = Ht;
  a.st = h->st_u;
  a.st_tiles = (Ht + kTile - 1) / kTile;
  a.nw = h->w_sn;
  a.inv_n = 1.0f / Ht;
  a.emode = E_STORE;
  a.bias = h->b_xe;
  a.Y = h->h0;
  a.ldy = D;
  a.out_st = h->st_h0;
  CK(launch_gemv(a, (D + kTile - 1) / kTile, s, false));
  return FM_OK;
}

// The sequential logit head is present when the weights hold markov.w1 [V][r]
// (bf16, r <= 512): the Markov head with markov.w2 [r][V], or the RNN head when
// rnn.wH [r][r], rnn.bH [r] and rnn.wO [r][V] are there too; conf.w [d + r] and
// conf.b [1] add the confidence head.
fm_status create_seq_head(fm_handle *h, const TensorSet &ts, cudaStream_t s) {
  const fm_config &c = h->cfg;
  const int V = c.vocab, G = c.block;
  auto it = ts.by_name.find("markov.w1");
  if (it == ts.by_name.end()) return FM_OK;
  const fm_tensor *t = it->second;
  if (t->dtype != FM_DTYPE_BF16 || t->nbytes <= 0 || t->nbytes % ((int64_t)2 * V))
    return fail(h, FM_ERR_INVALID_ARG, "markov.w1: expected bf16 [%d][r]", V);
  const int r = (int)(t->nbytes / ((int64_t)2 * V));
  if (r > 512) return fail(h, FM_ERR_UNSUPPORTED, "sequential head rank %d > 512", r);
  if (V % 8) return fail(h, FM_ERR_UNSUPPORTED, "sequential head needs vocab %% 8 == 0 (vocab %d)", V);
  h->seq_rank = r;
  const size_t rv = (size_t)r * V;
  TRY(dalloc(h, &h->seq_w1, rv));
  TRY(put_bf16(h, ts, "markov.w1", h->seq_w1, (int64_t)rv, s));
  TRY(dalloc(h, &h->seq_W, rv));
  if (ts.by_name.count("rnn.wH")) {
    TRY(dalloc(h, &h->seq_wH, (size_t)r * r));
    TRY(put_bf16(h, ts, "rnn.wH", h->seq_wH, (int64_t)r * r, s));
    TRY(dalloc(h, &h->seq_bH, (size_t)r));
    TRY(put_bf16(h, ts, "rnn.bH", h->seq_bH, r, s));
    TRY(put_bf16(h, ts, "rnn.wO", h->seq_W, (int64_t)rv, s));
  } else {
    TRY(put_bf16(h, ts, "markov.w2", h->seq_W, (int64_t)rv, s));
  }
  if (ts.by_name.count("conf.w")) {
    TRY(dalloc(h, &h->conf_w, (size_t)c.dim + r));
    TRY(put_bf16(h, ts, "conf.w", h->conf_w, (int64_t)c.dim + r, s));
    TRY(dalloc(h, &h->conf_b, 1));
    TRY(put_bf16(h, ts, "conf.b", h->conf_b, 1, s));
  }
  for (fm_handle::Lane &L : h->lanes) {
    TRY(dalloc(h, &L.seq_base, (size_t)G * V));
    TRY(dalloc(h, &L.seq_state, (size_t)2 * r));
    TRY(dalloc(h, &L.seq_part, (size_t)seq_grid(V)));
    TRY(dalloc(h, &L.seq_flags, (size_t)4 + kMaxT));
    CK(cudaMemsetAsync(L.seq_flags, 0, ((size_t)4 + kMaxT) * 4, s));
  }
  return FM_OK;
}

fm_status create_dflash(fm_handle *h, const TensorSet &ts, cudaStream_t s) {
  const fm_config &c = h->cfg;
  const int d = c.dim, H = c.target_dim, F = c.ff_dim, L = c.n_layers, G = c.block;
  const int mH = c.n_taps * H;
  TRY(create_table(h, ts, s));
  size_t tmp_elems = (size_t)mH * d;
  if ((size_t)d * F > tmp_elems) tmp_elems = (size_t)d * F;
  if ((size_t)H * d > tmp_elems) tmp_elems = (size_t)H * d;
  __nv_bfloat16 *tmp, *tmp2;
  TRY(dalloc(h, &tmp, tmp_elems));
  TRY(dalloc(h, &tmp2, (size_t)d * F));
  const size_t dd = (size_t)d * d;
  TRY(dalloc(h, &h->attn_norm, (size_t)L * d));
  TRY(dalloc(h, &h->ff_norm, (size_t)L * d));
  TRY(dalloc(h, &h->w_kvall, (size_t)L * 2 * dd));
  for (int l = 0; l < L; ++l) {
    const std::string p = "bb." + std::to_string(l) + ".";
    TRY(put_bf16(h, ts, p + "attn_norm", h->attn_norm + (size_t)l * d, d, s));
    TRY(put_bf16(h, ts, p + "ff_norm", h->ff_norm + (size_t)l * d, d, s));
    __nv_bfloat16 *w;
    TRY(dalloc(h, &w, 3 * dd));
    TRY(put_bf16_t(h, ts, p + "q", d, d, w, d, tmp, s));
    TRY(put_bf16_t(h, ts, p + "k", d, d, w + dd, d, tmp, s));
    TRY(put_bf16_t(h, ts, p + "v", d, d, w + 2 * dd, d, tmp, s));
    CK(cudaMemcpyAsync(h->w_kvall + (size_t)(2 * l) * dd, w + dd, 2 * dd * 2, cudaMemcpyDeviceToDevice, s));
    h->w_qkv.push_back(w);
    TRY(dalloc(h, &w, dd));
    TRY(put_bf16_t(h, ts, p + "o", d, d, w, d, tmp, s));
    h->w_o.push_back(w);
    // gate / up interleaved per 64 features: tile j = gate rows 64j.. then up rows 64j..
    TRY(dalloc(h, &w, (size_t)2 * F * d));
    TRY(put_bf16_t(h, ts, p + "gate", d, F, tmp2, d, tmp, s));
    for (int j = 0; j < F / 64; ++j)
      CK(cudaMemcpyAsync(w + (size_t)(128 * j) * d, tmp2 + (size_t)(64 * j) * d, (size_t)64 * d * 2,
                         cudaMemcpyDeviceToDevice, s));
    TRY(put_bf16_t(h, ts, p + "up", d, F, tmp2, d, tmp, s));
    for (int j = 0; j < F / 64; ++j)
      CK(cudaMemcpyAsync(w + (size_t)(128 * j + 64) * d, tmp2 + (size_t)(64 * j) * d, (size_t)64 * d * 2,
                         cudaMemcpyDeviceToDevice, s));
    h->w_gu.push_back(w);
    TRY(dalloc(h, &w, (size_t)d * F));
    TRY(put_bf16_t(h, ts, p + "down", F, d, w, F, tmp, s));
    h->w_down.push_back(w);
  }
  TRY(dalloc(h, &h->w_c, (size_t)d * mH));
  TRY(put_bf16_t(h, ts, "W_c", mH, d, h->w_c, mH, tmp, s));
  TRY(dalloc(h, &h->ctx_norm, d));
  TRY(put_bf16(h, ts, "ctx_norm", h->ctx_norm, d, s));
  TRY(dalloc(h, &h->w_tok, (size_t)d * H));
  TRY(put_bf16_t(h, ts, "tok_proj", H, d, h->w_tok, H, tmp, s));
  __nv_bfloat16 *mask_emb;
  TRY(dalloc(h, &mask_emb, (size_t)(G > 1 ? G - 1 : 1) * d));
  if (G > 1) TRY(put_bf16(h, ts, "mask_emb", mask_emb, (int64_t)(G - 1) * d, s));
  TRY(dalloc(h, &h->block_pos, (size_t)G * d));
  TRY(put_bf16(h, ts, "block_pos", h->block_pos, (int64_t)G * d, s));
  TRY(dalloc(h, &h->out_norm, d));
  TRY(put_bf16(h, ts, "out_norm", h->out_norm, d, s));
  TRY(dalloc(h, &h->w_out, (size_t)H * d));
  TRY(put_bf16_t(h, ts, "out_proj", d, H, h->w_out, d, tmp, s));
  TRY(create_common(h, s));
  TRY(create_seq_head(h, ts, s));
  TRY(dalloc(h, &h->hinit, (size_t)kMaxT * d));
  CK(cudaMemsetAsync(h->hinit, 0, (size_t)kMaxT * d * 4, s));
  CK(launch_block_consts(mask_emb, h->block_pos, G, d, h->hinit, h->st_init, s));
  for (int l = 0; l < L; ++l) {
    TRY(tile_weight(h, &h->w_qkv[l], 3 * d, d, s));
    TRY(tile_weight(h, &h->w_o[l], d, d, s));
    TRY(tile_weight(h, &h->w_gu[l], 2 * F, d, s));
    TRY(tile_weight(h, &h->w_down[l], d, F, s));
  }
  TRY(tile_weight(h, &h->w_kvall, L * 2 * d, d, s));
  TRY(tile_weight(h, &h->w_c, d, mH, s));
  TRY(tile_weight(h, &h->w_tok, d, H, s));
  TRY(tile_weight(h, &h->w_out, H, d, s));
  dfree_later(h, tmp);
  dfree_later(h, tmp2);
  CK(cudaStreamSynchronize(s));
  return FM_OK;
}

fm_status check_seq(fm_handle *h, int32_t seq) {
  if (seq < 0 || seq >= h->cfg.max_seqs) return fail(h, FM_ERR_INVALID_ARG, "seq %d outside [0, %d)", seq, h->cfg.max_seqs);
  return FM_OK;
}

fm_status append_checks(fm_handle *h, int32_t seq, const float *feats, int32_t n, int32_t start) {
  TRY(check_seq(h, seq));
  if (n < 0) return fail(h, FM_ERR_INVALID_ARG, "n_rows < 0");
  if (n > 0 && !feats) return fail(h, FM_ERR_INVALID_ARG, "null feature rows");
  if (n > 0 && (reinterpret_cast<uintptr_t>(feats) & 15)) return fail(h, FM_ERR_INVALID_ARG, "feature rows not 16-byte aligned");
  if (start < 0 || start > h->length[seq])
    return fail(h, FM_ERR_STATE, "start %d outside [0, length %d]", start, h->length[seq]);
  if ((int64_t)start + n + h->cfg.block + 1 > h->cfg.max_ctx)
    return fail(h, FM_ERR_CONTEXT_FULL, "context full: %d + %d + %d + 1 > %d", start, n, h->cfg.block, h->cfg.max_ctx);
  return FM_OK;
}

fm_status append_one(fm_handle *h, int32_t seq, const float *feats, int32_t n, int32_t start, cudaStream_t s) {
  const int FW = h->cfg.n_taps * h->cfg.target_dim;
  TRY(flush_pending(h, seq, s));
  use_lane(h, seq);
  if (h->cfg.variant == FM_VARIANT_FLASHMAP && n > 0 && n < kMaxT && h->use_defer) {
    // fc now; the K/V projection joins the next draft of this sequence
    StepParams p{};
    p.T = n;
    p.start = start;
    p.feats = feats;
    TRY(run_chain(h, chain_key(3, seq, n, 0, 0), p, s, [&](const StepParams *sp, cudaStream_t st) {
      return flashmap_fc_rows(h, sp, n, st);
    }));
    fm_handle::Lane &L = h->lanes[seq];
    L.pending = true;
    L.pend_start = start;
    L.pend_n = n;
    h->length[seq] = start + n;
    return FM_OK;
  }
  if (h->cfg.variant == FM_VARIANT_FLASHMAP && n >= kPrefillMin && h->cfg.dim % 256 == 0 && h->use_prefill) {
    TRY(flashmap_prefill(h, seq, feats, n, start, s));
    h->length[seq] = start + n;
    return FM_OK;
  }
  for (int r0 = 0; r0 < n; r0 += kMaxT) {
    const int rows = n - r0 < kMaxT ? n - r0 : kMaxT;
    StepParams p{};
    p.T = rows;
    p.start = start + r0;
    p.feats = feats + (size_t)r0 * FW;
    const uint64_t key = chain_key(2, seq, rows, 0, 0);
    TRY(run_chain(h, key, p, s, [&](const StepParams *sp, cudaStream_t st) {
      return h->cfg.variant == FM_VARIANT_FLASHMAP ? flashmap_append_rows(h, seq, sp, rows, st)
                                                   : dflash_append_rows(h, seq, sp, st);
    }));
  }
  h->length[seq] = start + n;
  return FM_OK;
}

// The device copy of a host-buffer call's feature rows (n floats), made on stream s after the
// previous host-buffer call's work: the staging buffer is grown (once that work has finished) when
// it is too small.  Asynchronous to the host when the rows are in pinned memory.
fm_status stage_rows(fm_handle *h, const float *host, size_t n, cudaStream_t s, const float **dev) {
  if (!h->stage_ev) CK(cudaEventCreateWithFlags(&h->stage_ev, cudaEventDisableTiming));
  CK(cudaStreamWaitEvent(s, h->stage_ev, 0));
  if (n > h->stage_cap) {
    CK(cudaEventSynchronize(h->stage_ev));
    if (h->stage_feats) {
      auto it = std::find(h->allocs.begin(), h->allocs.end(), static_cast<void *>(h->stage_feats));
      if (it != h->allocs.end()) h->allocs.erase(it);
      h->bytes -= (int64_t)(h->stage_cap * sizeof(float));
      cudaFree(h->stage_feats);
      h->stage_feats = nullptr;
      h->stage_cap = 0;
    }
    const size_t cap = n < ((size_t)1 << 20) ? (size_t)1 << 20 : n;
    TRY(dalloc(h, &h->stage_feats, cap));
    h->stage_cap = cap;
  }
  if (n) CK(cudaMemcpyAsync(h->stage_feats, host, n * sizeof(float), cudaMemcpyHostToDevice, s));
  *dev = h->stage_feats;
  return FM_OK;
}

}  // namespace

// Run body(i, stream) for the n sequences ids[0..n): one sequence on the caller's
// stream as is; several on their lanes' streams, forked from and joined back into
// the caller's stream, so independent sequences' chains overlap on the GPU.
template <typename F>
fm_status run_lanes(fm_handle *h, int n, const int32_t *ids, cudaStream_t s, F body) {
  if (n == 1 || h->lanes.size() < 2) {
    for (int i = 0; i < n; ++i) TRY(body(i, s));
    return FM_OK;
  }
  CK(cudaEventRecord(h->fork_ev, s));
  fm_status st = FM_OK;
  int started = 0;
  for (int i = 0; i < n && st == FM_OK; ++i, ++started) {
    fm_handle::Lane &L = h->lanes[ids[i]];
    if (cudaStreamWaitEvent(L.stream, h->fork_ev, 0) != cudaSuccess) {
      st = fail(h, FM_ERR_CUDA, "stream wait failed");
      break;
    }
    st = body(i, L.stream);
  }
  for (int i = 0; i < started; ++i) {
    fm_handle::Lane &L = h->lanes[ids[i]];
    if (cudaEventRecord(L.done, L.stream) != cudaSuccess || cudaStreamWaitEvent(s, L.done, 0) != cudaSuccess)
      if (st == FM_OK) st = fail(h, FM_ERR_CUDA, "stream join failed");
  }
  return st;
}

extern "C" {

fm_status fm_create(const fm_config *cfg, const fm_tensor *weights, int32_t n_weights, const float *modulation,
                    void *stream, fm_handle **out) {
  if (!out) return FM_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || (!weights && n_weights > 0) || n_weights < 0) return FM_ERR_INVALID_ARG;
  fm_handle *h = new (std::nothrow) fm_handle();
  if (!h) return FM_ERR_OOM;
  h->cfg = *cfg;
  fm_status st = check_config(h, *cfg);
  if (st != FM_OK) {
    g_create_error = h->err;
    fm_destroy(h);
    return st;
  }
  cudaGetDevice(&h->dev);
  cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, h->dev);
  TensorSet ts;
  for (int i = 0; i < n_weights; ++i) {
    if (!weights[i].name) {
      fm_destroy(h);
      return FM_ERR_INVALID_ARG;
    }
    ts.by_name[weights[i].name] = &weights[i];
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = cfg->variant == FM_VARIANT_FLASHMAP ? create_flashmap(h, ts, modulation, s) : create_dflash(h, ts, s);
  if (st == FM_OK) {
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) st = fail(h, FM_ERR_CUDA, "create: %s", cudaGetErrorString(e));
  }
  cudaStreamSynchronize(s);
  for (void *p : h->to_free) cudaFree(p);
  h->to_free.clear();
  if (st != FM_OK) {
    g_create_error = h->err;
    fm_destroy(h);
    return st;
  }
  g_create_error.clear();
  *out = h;
  return FM_OK;
}

fm_status fm_context_append(fm_handle *h, int32_t seq, const float *feats, int32_t n_rows, int32_t start_pos,
                            void *stream) {
  if (!h) return FM_ERR_INVALID_ARG;
  h->last_launches = 0;
  TRY(append_checks(h, seq, feats, n_rows, start_pos));
  h->narrow = false;
  return append_one(h, seq, feats, n_rows, start_pos, static_cast<cudaStream_t>(stream));
}

constexpr int kNarrowSeqs = 8;   // sequences per call from which the products run unsplit

fm_status fm_context_append_batched(fm_handle *h, int32_t n_seqs, const int32_t *seq_ids, const float *feats,
                                    const int32_t *n_rows, const int32_t *start, void *stream) {
  if (!h) return FM_ERR_INVALID_ARG;
  h->last_launches = 0;
  if (n_seqs < 1 || n_seqs > h->cfg.max_seqs || !seq_ids || !n_rows || !start)
    return fail(h, FM_ERR_INVALID_ARG, "bad batched append arguments");
  std::vector<char> seen(h->cfg.max_seqs, 0);
  size_t off = 0;
  for (int i = 0; i < n_seqs; ++i) {
    TRY(append_checks(h, seq_ids[i], feats ? feats + off : nullptr, n_rows[i], start[i]));
    if (seen[seq_ids[i]]) return fail(h, FM_ERR_INVALID_ARG, "repeated seq id %d", seq_ids[i]);
    seen[seq_ids[i]] = 1;
    off += (size_t)n_rows[i] * h->cfg.n_taps * h->cfg.target_dim;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::vector<size_t> offs(n_seqs);
  off = 0;
  for (int i = 0; i < n_seqs; ++i) {
    offs[i] = off;
    off += (size_t)n_rows[i] * h->cfg.n_taps * h->cfg.target_dim;
  }
  // dense appends share the prefill scratch: they run first, one after the other, on the caller's stream
  std::vector<int32_t> rest;
  std::vector<int> rest_i;
  for (int i = 0; i < n_seqs; ++i) {
    if (n_rows[i] >= kPrefillMin) {
      TRY(append_one(h, seq_ids[i], feats + offs[i], n_rows[i], start[i], s));
    } else {
      rest.push_back(seq_ids[i]);
      rest_i.push_back(i);
    }
  }
  if (rest.empty()) return FM_OK;
  if (h->wide.on && (int)rest.size() >= kWideMin && h->use_prefill) {
    std::vector<size_t> ro(rest.size());
    std::vector<int32_t> rn(rest.size()), rs(rest.size());
    for (size_t j = 0; j < rest.size(); ++j) {
      ro[j] = offs[rest_i[j]];
      rn[j] = n_rows[rest_i[j]];
      rs[j] = start[rest_i[j]];
    }
    return wide_append(h, (int)rest.size(), rest.data(), feats, ro.data(), rn.data(), rs.data(), s);
  }
  h->narrow = (int)rest.size() >= kNarrowSeqs && h->lanes.size() > 1;
  return run_lanes(h, (int)rest.size(), rest.data(), s, [&](int j, cudaStream_t ls) {
    const int i = rest_i[j];
    return append_one(h, seq_ids[i], feats + offs[i], n_rows[i], start[i], ls);
  });
}

fm_status fm_draft(fm_handle *h, int32_t n_seqs, const int32_t *seq_ids, const int32_t *anchors, const int32_t *pos,
                   int32_t *tokens, void *stream) {
  if (!h) return FM_ERR_INVALID_ARG;
  h->last_launches = 0;
  if (n_seqs < 1 || n_seqs > h->cfg.max_seqs || !seq_ids || !anchors || !pos || !tokens)
    return fail(h, FM_ERR_INVALID_ARG, "bad draft arguments");
  std::vector<char> seen(h->cfg.max_seqs, 0);
  for (int i = 0; i < n_seqs; ++i) {
    TRY(check_seq(h, seq_ids[i]));
    if (seen[seq_ids[i]]) return fail(h, FM_ERR_INVALID_ARG, "repeated seq id %d", seq_ids[i]);
    seen[seq_ids[i]] = 1;
    if (anchors[i] < 0 || anchors[i] >= h->cfg.vocab)
      return fail(h, FM_ERR_INVALID_ARG, "anchor %d outside [0, %d)", anchors[i], h->cfg.vocab);
    if (pos[i] != h->length[seq_ids[i]])
      return fail(h, FM_ERR_STATE, "pos %d != length %d", pos[i], h->length[seq_ids[i]]);
    if ((int64_t)pos[i] + h->cfg.block + 1 > h->cfg.max_ctx)
      return fail(h, FM_ERR_CONTEXT_FULL, "context full at pos %d", pos[i]);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (h->wide.on && !h->use_step && n_seqs >= kWideMin) return wide_draft(h, n_seqs, seq_ids, anchors, pos, tokens, s);
  h->narrow = !h->use_step && n_seqs >= kNarrowSeqs && h->lanes.size() > 1;
  if (h->use_step) {
    // the persistent step holds every SM: sequences draft one after another on the caller's stream
    for (int i = 0; i < n_seqs; ++i)
      TRY(draft_one(h, seq_ids[i], anchors[i], pos[i], tokens + (size_t)i * h->cfg.block, s));
    return FM_OK;
  }
  return run_lanes(h, n_seqs, seq_ids, s, [&](int i, cudaStream_t ls) {
    return draft_one(h, seq_ids[i], anchors[i], pos[i], tokens + (size_t)i * h->cfg.block, ls);
  });
}

fm_status fm_context_append_host(fm_handle *h, int32_t seq, const float *feats_host, int32_t n_rows,
                                 int32_t start_pos, void *stream) {
  if (!h) return FM_ERR_INVALID_ARG;
  h->last_launches = 0;
  if (n_rows > 0 && !feats_host) return fail(h, FM_ERR_INVALID_ARG, "null feature rows");
  TRY(check_seq(h, seq));
  if (n_rows < 0) return fail(h, FM_ERR_INVALID_ARG, "n_rows < 0");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float *dev = nullptr;
  TRY(stage_rows(h, feats_host, (size_t)n_rows * h->cfg.n_taps * h->cfg.target_dim, s, &dev));
  const fm_status st = fm_context_append(h, seq, n_rows > 0 ? dev : nullptr, n_rows, start_pos, stream);
  CK(cudaEventRecord(h->stage_ev, s));
  return st;
}

fm_status fm_context_append_batched_host(fm_handle *h, int32_t n_seqs, const int32_t *seq_ids,
                                         const float *feats_host, const int32_t *n_rows, const int32_t *start,
                                         void *stream) {
  if (!h) return FM_ERR_INVALID_ARG;
  h->last_launches = 0;
  if (n_seqs < 1 || n_seqs > h->cfg.max_seqs || !seq_ids || !n_rows || !start)
    return fail(h, FM_ERR_INVALID_ARG, "bad batched append arguments");
  size_t total = 0;
  for (int i = 0; i < n_seqs; ++i) {
    if (n_rows[i] < 0) return fail(h, FM_ERR_INVALID_ARG, "n_rows < 0");
    total += (size_t)n_rows[i];
  }
  if (total > 0 && !feats_host) return fail(h, FM_ERR_INVALID_ARG, "null feature rows");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float *dev = nullptr;
  TRY(stage_rows(h, feats_host, total * h->cfg.n_taps * h->cfg.target_dim, s, &dev));
  const fm_status st = fm_context_append_batched(h, n_seqs, seq_ids, total > 0 ? dev : nullptr, n_rows, start,
                                                 stream);
  CK(cudaEventRecord(h->stage_ev, s));
  return st;
}

fm_status fm_draft_host(fm_handle *h, int32_t n_seqs, const int32_t *seq_ids, const int32_t *anchors,
                        const int32_t *pos, int32_t *tokens_host, void *stream) {
  if (!h) return FM_ERR_INVALID_ARG;
  h->last_launches = 0;
  if (!tokens_host) return fail(h, FM_ERR_INVALID_ARG, "null tokens");
  if (n_seqs < 1 || n_seqs > h->cfg.max_seqs) return fail(h, FM_ERR_INVALID_ARG, "n_seqs outside [1, max_seqs]");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!h->stage_ev) CK(cudaEventCreateWithFlags(&h->stage_ev, cudaEventDisableTiming));
  if (!h->stage_tok) TRY(dalloc(h, &h->stage_tok, (size_t)h->cfg.max_seqs * h->cfg.block));
  CK(cudaStreamWaitEvent(s, h->stage_ev, 0));
  TRY(fm_draft(h, n_seqs, seq_ids, anchors, pos, h->stage_tok, stream));
  CK(cudaMemcpyAsync(tokens_host, h->stage_tok, (size_t)n_seqs * h->cfg.block * sizeof(int32_t),
                     cudaMemcpyDeviceToHost, s));
  CK(cudaEventRecord(h->stage_ev, s));
  return FM_OK;
}

fm_status fm_draft_pruned(fm_handle *h, int32_t seq, int32_t anchor, int32_t pos, const float *thresholds,
                          float min_conf, int32_t *tokens, float *conf, int32_t *length, void *stream) {
  if (!h) return FM_ERR_INVALID_ARG;
  h->last_launches = 0;
  const fm_config &c = h->cfg;
  if (!h->seq_rank) return fail(h, FM_ERR_UNSUPPORTED, "the weights hold no sequential head (markov.w1)");
  if (!tokens) return fail(h, FM_ERR_INVALID_ARG, "null tokens");
  TRY(check_seq(h, seq));
  if (anchor < 0 || anchor >= c.vocab) return fail(h, FM_ERR_INVALID_ARG, "anchor %d outside [0, %d)", anchor, c.vocab);
  if (pos != h->length[seq]) return fail(h, FM_ERR_STATE, "pos %d != length %d", pos, h->length[seq]);
  if ((int64_t)pos + c.block + 1 > c.max_ctx) return fail(h, FM_ERR_CONTEXT_FULL, "context full at pos %d", pos);
  float thr[16];
  bool any = false;
  for (int k = 0; k < 16; ++k) {
    // a position without a threshold of its own (NaN) takes min_conf
    thr[k] = k >= c.block ? NAN : thresholds && thresholds[k] == thresholds[k] ? thresholds[k] : min_conf;
    any = any || thr[k] == thr[k];
  }
  if (!h->conf_w && (any || conf))
    return fail(h, FM_ERR_UNSUPPORTED, "the weights hold no confidence head (conf.w, conf.b)");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  h->narrow = false;
  return draft_one(h, seq, anchor, pos, tokens, s, conf, length, thr);
}

fm_status fm_accept(const int32_t *draft, const int32_t *target, int32_t k, int32_t *n_accepted, int32_t *bonus) {
  if (!draft || !target || !n_accepted || !bonus || k < 0) return FM_ERR_INVALID_ARG;
  int32_t a = 0;
  while (a < k && draft[a] == target[a]) ++a;
  *n_accepted = a;
  *bonus = target[a];
  return FM_OK;
}

fm_status fm_accept_batched(fm_handle *h, int32_t n_seqs, const int32_t *draft, const int32_t *target,
                            const int32_t *k, int32_t *acc, int32_t *bonus, void *stream) {
  if (!h) return FM_ERR_INVALID_ARG;
  if (n_seqs < 1 || !draft || !target || !k || !acc || !bonus) return fail(h, FM_ERR_INVALID_ARG, "bad accept arguments");
  CK(launch_accept(n_seqs, h->cfg.block, draft, target, k, acc, bonus, static_cast<cudaStream_t>(stream)));
  return FM_OK;
}

// The fused lm_head + argmax on caller rows, with its cross-CTA scratch in the
// library's static device memory instead of the handle's buffers.
fm_status fm_lm_head_argmax_noalloc(fm_handle *h, const float *y_dev, int32_t n_rows, int32_t *tokens_dev,
                                     void *stream) {
  if (!h) return FM_ERR_INVALID_ARG;
  h->last_launches = 0;
  if (!y_dev || !tokens_dev || n_rows < 1 || n_rows > 16)
    return fail(h, FM_ERR_INVALID_ARG, "bad lm_head arguments (n_rows must be in 1..16)");
  // the kernel reads the rows as float4 and writes the tokens as int32
  if (reinterpret_cast<uintptr_t>(y_dev) & 15) return fail(h, FM_ERR_INVALID_ARG, "y_dev is not 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(tokens_dev) & 3) return fail(h, FM_ERR_INVALID_ARG, "tokens_dev is not 4-byte aligned");
  // the table and the static scratch are those of the current device: it must be the handle's
  int cur = -1;
  CK(cudaGetDevice(&cur));
  if (cur != h->dev)
    return fail(h, FM_ERR_INVALID_ARG, "the current device (%d) is not the handle's device (%d)", cur, h->dev);
  const fm_config &c = h->cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LmArgs a;
  memset(&a, 0, sizeof a);
  if (c.lm_format == FM_LM_Q8_0)
    a.q8 = h->tq8;
  else
    a.wb = h->tb;
  a.err = h->dev_err;
  a.V = c.vocab;
  a.H = c.target_dim;
  a.T_const = n_rows;
  a.Y = y_dev;
  a.ldy = c.target_dim;
  a.tokens = tokens_dev;
  const int grid = lmhead_grid(a, h->n_sm);
  if (grid > lmhead_static_max_grid())
    return fail(h, FM_ERR_UNSUPPORTED, "lm_head grid of %d CTAs exceeds the static scratch (at most %d)", grid,
                lmhead_static_max_grid());
  CK(lmhead_static_scratch(grid, &a.part, &a.ticket, s));
  CK(launch_lmhead(a, grid, s, false));
  ++h->last_launches;
  return FM_OK;
}

fm_status fm_time_conditioning(const fm_config *cfg, const fm_tensor *weights, int32_t n_weights, int32_t time_dim,
                               int32_t cond_dim, float time_scale, float s_time, float t_time, float *table_dev,
                               void *stream) {
  fm_handle tmp;   // holds the temporary buffers and the error text
  fm_handle *h = &tmp;
  auto done = [&](fm_status st) {
    for (void *p : tmp.allocs) cudaFree(p);
    tmp.allocs.clear();
    if (st != FM_OK) g_create_error = tmp.err;
    return st;
  };
  if (!cfg || (!weights && n_weights > 0) || n_weights < 0 || !table_dev) return FM_ERR_INVALID_ARG;
  tmp.cfg = *cfg;
  if (cfg->variant != FM_VARIANT_FLASHMAP) return done(fail(h, FM_ERR_INVALID_ARG, "time conditioning is FlashMap's"));
  if (cfg->dim < 1 || cfg->n_layers < 1 || time_dim < 2 || time_dim % 2 || cond_dim < 1)
    return done(fail(h, FM_ERR_INVALID_ARG, "bad dims (time_dim must be even, all dims positive)"));
  if (reinterpret_cast<uintptr_t>(table_dev) & 3) return done(fail(h, FM_ERR_INVALID_ARG, "table_dev not 4-byte aligned"));
  TensorSet ts;
  for (int i = 0; i < n_weights; ++i) {
    if (!weights[i].name) return done(fail(h, FM_ERR_INVALID_ARG, "unnamed tensor"));
    ts.by_name[weights[i].name] = &weights[i];
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int L = cfg->n_layers, D3 = 3 * cfg->dim, nb = 3 * L + 1;
  struct Lin {
    __nv_bfloat16 *w = nullptr, *b = nullptr;
  };
  auto load = [&](const std::string &name, int M, int N, Lin &out) -> fm_status {
    TRY(dalloc(h, &out.w, (size_t)M * N));
    TRY(put_bf16(h, ts, name + ".weight", out.w, (int64_t)M * N, s));
    TRY(dalloc(h, &out.b, M));
    return put_bf16(h, ts, name + ".bias", out.b, M, s, true);
  };
  Lin te1, te2, je1, je2;
  fm_status st;
  if ((st = load("time_embed.linear_1", cond_dim, time_dim, te1)) != FM_OK ||
      (st = load("time_embed.linear_2", cond_dim, cond_dim, te2)) != FM_OK ||
      (st = load("jump_embed.linear_1", cond_dim, time_dim, je1)) != FM_OK ||
      (st = load("jump_embed.linear_2", cond_dim, cond_dim, je2)) != FM_OK)
    return done(st);
  std::vector<Lin> ada(nb);
  for (int n = 0; n < nb; ++n) {
    const std::string name = n < 3 * L ? "layers." + std::to_string(n / 3) + "." +
                                             (n % 3 == 0 ? "self_attn_adaln" : n % 3 == 1 ? "cross_attn_adaln" : "mlp_adaln") +
                                             ".linear"
                                       : "final_adaln.linear";
    if ((st = load(name, D3, cond_dim, ada[n])) != FM_OK) return done(st);
  }
  float *e = nullptr, *hid = nullptr, *tsv = nullptr, *tjv = nullptr;
  if ((st = dalloc(h, &e, time_dim)) != FM_OK || (st = dalloc(h, &hid, cond_dim)) != FM_OK ||
      (st = dalloc(h, &tsv, cond_dim)) != FM_OK || (st = dalloc(h, &tjv, cond_dim)) != FM_OK)
    return done(st);
  auto run = [&]() -> cudaError_t {
    cudaError_t r;
    // ts = linear_2(SiLU(linear_1(embed(s)))), tj likewise for t
    if ((r = launch_time_embed(e, time_dim, time_scale, s_time, s)) != cudaSuccess) return r;
    if ((r = launch_setup_linear(te1.w, te1.b, e, nullptr, cond_dim, time_dim, 0, hid, s)) != cudaSuccess) return r;
    if ((r = launch_setup_linear(te2.w, te2.b, hid, nullptr, cond_dim, cond_dim, 1, tsv, s)) != cudaSuccess) return r;
    if ((r = launch_time_embed(e, time_dim, time_scale, t_time, s)) != cudaSuccess) return r;
    if ((r = launch_setup_linear(je1.w, je1.b, e, nullptr, cond_dim, time_dim, 0, hid, s)) != cudaSuccess) return r;
    if ((r = launch_setup_linear(je2.w, je2.b, hid, nullptr, cond_dim, cond_dim, 1, tjv, s)) != cudaSuccess) return r;
    // every adaLN block from cond = SiLU(ts + tj)
    for (int n = 0; n < nb; ++n)
      if ((r = launch_setup_linear(ada[n].w, ada[n].b, tsv, tjv, D3, cond_dim, 2, table_dev + (size_t)n * D3, s)) !=
          cudaSuccess)
        return r;
    return cudaStreamSynchronize(s);
  };
  const cudaError_t r = run();
  if (r != cudaSuccess) return done(fail(h, FM_ERR_CUDA, "time conditioning: %s", cudaGetErrorString(r)));
  return done(FM_OK);
}

fm_status fm_synchronize(fm_handle *h, void *stream) {
  if (!h) return FM_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t flag = 0;
  CK(cudaMemcpyAsync(&flag, h->dev_err, 4, cudaMemcpyDeviceToHost, s));
  CK(cudaStreamSynchronize(s));
  if (flag) {
    CK(cudaMemsetAsync(h->dev_err, 0, 4, s));
    // a draft step that wound down early left its grid barrier's arrival count off
    if (h->step_bar) CK(cudaMemsetAsync(h->step_bar, 0, 64 * 4, s));
    CK(cudaStreamSynchronize(s));
    return fail(h, FM_ERR_TIMEOUT, "a device-side bounded wait gave up; the outputs of the calls since the last check "
                                   "are undefined");
  }
  return FM_OK;
}

fm_status fm_selftest_wait_timeout(fm_handle *h, int32_t budget_us, void *stream) {
  if (!h) return FM_ERR_INVALID_ARG;
  if (budget_us < 1 || budget_us > 1000000) return fail(h, FM_ERR_INVALID_ARG, "budget_us outside [1, 1000000]");
  int khz = 0;
  CK(cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, h->dev));
  if (khz <= 0) khz = 2000000;
  const long long cycles = (long long)budget_us * (khz / 1000);
  CK(launch_wait_selftest(h->dev_err, cycles, static_cast<cudaStream_t>(stream)));
  h->last_launches = 1;
  return FM_OK;
}

fm_status fm_debug_copy(fm_handle *h, int32_t what, int32_t seq, int32_t index, int64_t offset, void *dst,
                        int64_t nbytes, void *stream) {
  if (!h) return FM_ERR_INVALID_ARG;
  if (!dst || nbytes < 0 || offset < 0) return fail(h, FM_ERR_INVALID_ARG, "bad debug copy arguments");
  const fm_config &c = h->cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void *src = nullptr;
  int64_t size = 0;
  switch (what) {
    case FM_DEBUG_HIDDEN:
      if (index < 0 || index >= c.n_layers) return fail(h, FM_ERR_INVALID_ARG, "layer %d", index);
      src = h->hid + (size_t)index * kMaxT * c.dim;
      size = (int64_t)c.block * c.dim * 4;
      break;
    case FM_DEBUG_HEAD_OUT:
      TRY(check_seq(h, seq));
      use_lane(h, seq);
      src = h->Y;
      if (h->wide.on && h->wide.row_of[seq] == -2)
        return fail(h, FM_ERR_UNSUPPORTED, "the head output of an earlier batched pass is not kept");
      if (h->wide.on && h->wide.row_of[seq] >= 0) src = h->wide.Y + (size_t)h->wide.row_of[seq] * c.target_dim;
      size = (int64_t)c.block * c.target_dim * 4;
      break;
    case FM_DEBUG_LOGITS: {
      TRY(check_seq(h, seq));
      if (h->wide.on && h->wide.row_of[seq] == -2)
        return fail(h, FM_ERR_UNSUPPORTED, "the head output of an earlier batched pass is not kept");
      if (h->wide.on && h->wide.row_of[seq] >= 0) {
        // the batched lm_head's product for this sequence's rows, stored instead of reduced
        fm_handle::Wide &w = h->wide;
        if (!w.dbg_logits) TRY(dalloc(h, &w.dbg_logits, (size_t)c.block * w.Vn));
        if (!h->dbg_logits) TRY(dalloc(h, &h->dbg_logits, (size_t)kMaxT * c.vocab));
        TcGemmArgs g = wide_gemm(h, w.m_y16, w.t_table, c.block, w.Vn, c.target_dim, TC_EPI_F16);
        g.a_row0 = w.row_of[seq];
        g.out32 = w.dbg_logits;
        g.ldo32 = w.Vn;
        TRY(run_tc(h, g, s, "wide.gemm_logits"));
        CK(cudaMemcpy2DAsync(h->dbg_logits, (size_t)c.vocab * 4, w.dbg_logits, (size_t)w.Vn * 4, (size_t)c.vocab * 4,
                             c.block, cudaMemcpyDeviceToDevice, s));
        src = h->dbg_logits;
        size = (int64_t)c.block * c.vocab * 4;
        break;
      }
      use_lane(h, seq);
      if (!h->dbg_logits) TRY(dalloc(h, &h->dbg_logits, (size_t)kMaxT * c.vocab));
      StepParams p{};
      p.T = c.block;
      fm_status st;
      const StepParams *sp = next_params(h, p, s, &st);
      if (!sp) return st;
      TRY(run_lmhead(h, h->Y, c.block, sp, h->tok_tmp, h->dbg_logits, s, h->ylm));
      src = h->dbg_logits;
      size = (int64_t)c.block * c.vocab * 4;
      break;
    }
    case FM_DEBUG_CACHE_K:
    case FM_DEBUG_CACHE_V: {
      TRY(check_seq(h, seq));
      TRY(flush_pending(h, seq, s));
      if (index < 0 || index >= c.n_layers) return fail(h, FM_ERR_INVALID_ARG, "layer %d", index);
      Seg2 kv = h->kv(seq, index);
      src = what == FM_DEBUG_CACHE_K ? kv.k : kv.v;
      size = (int64_t)h->cache_plane * 2;
      break;
    }
    case FM_DEBUG_STEP_TRACE:
      if (!h->step_trace) return fail(h, FM_ERR_INVALID_ARG, "no trace recorded (set FM_DEBUG_TRACE before a draft)");
      src = h->step_trace;
      size = (int64_t)h->step_trace_phases * h->step_clusters * kStepCS * kStepTraceSlots * 8;
      break;
    case FM_DEBUG_H0:
      if (!h->h0) return fail(h, FM_ERR_INVALID_ARG, "no h0 for this variant");
      src = h->h0;
      size = (int64_t)c.dim * 4;
      break;
    default:
      return fail(h, FM_ERR_INVALID_ARG, "unknown debug selector %d", what);
  }
  if (offset + nbytes > size) return fail(h, FM_ERR_INVALID_ARG, "range beyond the buffer (%lld bytes)", (long long)size);
  CK(cudaMemcpyAsync(dst, static_cast<const char *>(src) + offset, nbytes, cudaMemcpyDeviceToHost, s));
  int32_t flag = 0;
  CK(cudaMemcpyAsync(&flag, h->dev_err, 4, cudaMemcpyDeviceToHost, s));
  CK(cudaStreamSynchronize(s));
  if (flag) return fail(h, FM_ERR_TIMEOUT, "a device-side bounded wait gave up in an earlier call");
  return FM_OK;
}

fm_status fm_set_debug(fm_handle *h, int32_t flags) {
  if (!h) return FM_ERR_INVALID_ARG;
  h->debug = flags;
  return FM_OK;
}

fm_status fm_profile_read(fm_handle *h, fm_kernel_time *out, int32_t cap, int32_t *n) {
  if (!h || !n || cap < 0 || (cap > 0 && !out)) return FM_ERR_INVALID_ARG;
  std::vector<fm_kernel_time> agg;
  for (ProfRec &r : h->prof) {
    CK(cudaEventSynchronize(r.e1));
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, r.e0, r.e1));
    fm_kernel_time *k = nullptr;
    for (auto &a : agg)
      if (r.name == a.name) k = &a;
    if (!k) {
      agg.emplace_back();
      k = &agg.back();
      memset(k, 0, sizeof *k);
      snprintf(k->name, sizeof k->name, "%s", r.name.c_str());
    }
    k->launches += 1;
    k->ms += ms;
    k->bytes += r.bytes;
    h->ev_pool.push_back(r.e0);
    h->ev_pool.push_back(r.e1);
  }
  h->prof.clear();
  *n = (int32_t)agg.size();
  for (int i = 0; i < (int)agg.size() && i < cap; ++i) out[i] = agg[i];
  return FM_OK;
}

fm_status fm_get_length(const fm_handle *h, int32_t seq, int32_t *length) {
  if (!h || !length || seq < 0 || seq >= h->cfg.max_seqs) return FM_ERR_INVALID_ARG;
  *length = h->length[seq];
  return FM_OK;
}

fm_status fm_memory_bytes(const fm_handle *h, int64_t *bytes) {
  if (!h || !bytes) return FM_ERR_INVALID_ARG;
  *bytes = h->bytes;
  return FM_OK;
}

fm_status fm_last_launch_count(const fm_handle *h, int32_t *count) {
  if (!h || !count) return FM_ERR_INVALID_ARG;
  *count = h->last_launches;
  return FM_OK;
}

const char *fm_status_str(fm_status s) {
  switch (s) {
    case FM_OK: return "ok";
    case FM_ERR_INVALID_ARG: return "invalid argument";
    case FM_ERR_UNSUPPORTED: return "unsupported configuration";
    case FM_ERR_OOM: return "out of memory";
    case FM_ERR_CONTEXT_FULL: return "context full";
    case FM_ERR_STATE: return "bad sequence state";
    case FM_ERR_CUDA: return "CUDA error";
    case FM_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

// With a null handle: the reason the last failed fm_create or fm_time_conditioning on this thread.
const char *fm_last_error(const fm_handle *h) { return h ? h->err.c_str() : g_create_error.c_str(); }

void fm_destroy(fm_handle *h) {
  if (!h) return;
  for (void *p : h->allocs) cudaFree(p);
  for (void *p : h->to_free) cudaFree(p);
  if (h->sp_host) cudaFreeHost(h->sp_host);
  for (int i = 0; i < kParamSlots; ++i)
    if (h->sp_ev[i]) cudaEventDestroy(h->sp_ev[i]);
  for (ProfRec &r : h->prof) {
    cudaEventDestroy(r.e0);
    cudaEventDestroy(r.e1);
  }
  for (cudaEvent_t e : h->ev_pool) cudaEventDestroy(e);
  for (auto &kv : h->graphs)
    if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
  if (h->cap) cudaStreamDestroy(h->cap);
  for (fm_handle::Lane &L : h->lanes) {
    if (L.stream) cudaStreamDestroy(L.stream);
    if (L.done) cudaEventDestroy(L.done);
  }
  if (h->fork_ev) cudaEventDestroy(h->fork_ev);
  if (h->stage_ev) cudaEventDestroy(h->stage_ev);
  if (h->wide.par_host) cudaFreeHost(h->wide.par_host);
  if (h->wide.rows_host) cudaFreeHost(h->wide.rows_host);
  for (int i = 0; i < kParamSlots; ++i) {
    if (h->wide.par_ev[i]) cudaEventDestroy(h->wide.par_ev[i]);
    if (h->wide.rows_ev[i]) cudaEventDestroy(h->wide.rows_ev[i]);
  }
  delete h;
}

}  // extern "C"
