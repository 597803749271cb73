// Host side of the FlashMap C ABI (include/flashmap.h): argument validation, the
// load-time precompute, workspace carving and the launch sequence of each call.
// Every call validates first and launches nothing on an invalid argument.

#include <algorithm>
#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include "common.cuh"
#include "internal.h"

using fm::Launch;
using fm::Weight;

namespace {

thread_local std::string g_last_error;

flashmap_status fail(flashmap_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

#define FM_CUDA(call)                                                                          \
  do {                                                                                         \
    cudaError_t e_ = (call);                                                                   \
    if (e_ != cudaSuccess) return fail(FLASHMAP_E_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_)); \
  } while (0)

size_t dt_size(int dtype) { return dtype == FLASHMAP_F32 ? 4 : dtype == FLASHMAP_BF16 ? 2 : 1; }

inline size_t align_up(size_t x, size_t a = 256) { return (x + a - 1) / a * a; }

// Carves 256-byte aligned sub-buffers out of one allocation (or measures the total).
struct Carver {
  uint8_t* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<uint8_t*>(b)) {}
  template <typename P>
  P* take(size_t bytes) {
    off = align_up(off);
    P* p = base ? reinterpret_cast<P*>(base + off) : nullptr;
    off += bytes;
    return p;
  }
};

struct LayerW {
  Weight qkv, o, cq, co, fc1, fc2;
  float *qn = nullptr, *kn = nullptr, *cqn = nullptr;
  float* mods = nullptr;  // [9][D]: (1+scale, shift, gate) x (self, cross, mlp)
  float *fc1_b = nullptr, *fc2_beta = nullptr;
};

}  // namespace

struct flashmap_model {
  flashmap_config cfg;
  int device = 0, num_sms = 0;
  int adt = FLASHMAP_F32, wdt = FLASHMAP_F32, kdt = FLASHMAP_F32;  // activations, GEMM weights, KV pool
  int H = 0, Lt = 0, D = 0, L = 0, nh = 0, hd = 0, F = 0, K = 0, V = 0, Vd = 0, P = 0, maxpos = 0;
  void* arena = nullptr;
  unsigned* dev_err = nullptr;
  Weight fc, ap, ctx_kv, chol, xe, head;
  std::vector<LayerW> layers;
  float *hidden_norm_w = nullptr, *anchor_norm_w = nullptr, *noise_norm_w = nullptr;
  float *ap_b = nullptr, *xe_b = nullptr, *head_b = nullptr, *ctx_knorm = nullptr;
  float *final_mods = nullptr, *u = nullptr;
  float gate = 1.f;
  int64_t* hot = nullptr;
  int32_t* inv_hot = nullptr;
  float2* rope = nullptr;
  const void* embedding = nullptr;
  // several jumps (num_steps > 1): per jump (s, t) its modulations, final AdaLN and
  // fc2 bias terms; the embedding transposed (the GEMM's weight for [posterior; state]
  // @ E) and the full-vocabulary folded head for the state update between jumps
  int steps = 1;
  float grid[5] = {0.f, 1.f, 0.f, 0.f, 0.f};
  float step_gate[4] = {1.f, 1.f, 1.f, 1.f};
  float *step_mods = nullptr, *step_final = nullptr, *step_fc2_beta = nullptr;  // [steps][L][9][D], [steps][2][D], [steps][L][D]
  Weight et, full_head;
  float *full_head_b = nullptr, *state_norm_w = nullptr;
  // folded-noise eigenbasis (noise_path 1): M = diag(sqrt lam) Q^T diag(w) W_x^T as a
  // GEMM weight (D out, H in), lam / H, x_embed(u); the eigensolver's sweep count
  int noise_path = 0, eig_sweeps = 0;
  Weight fold;
  float *fold_var = nullptr, *fold_xu = nullptr;
  // the anchor branch of a draft runs on this stream, forked from and joined back to
  // the caller's stream with the two events
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  // launch timing (flashmap_profile_start / stop)
  bool prof_on = false;
  int prof_cap = 0;
  std::vector<cudaEvent_t> prof_events;
  std::vector<flashmap_launch_record> prof_recs;
  Launch launch(cudaStream_t s) const { return Launch{s, num_sms, dev_err}; }
};

// The draft's anchor branch on the side stream (1) or in line (0), and the tcgen05
// GEMM CTAs per SM while both branches run.
#ifndef FM_DRAFT_FORK
#define FM_DRAFT_FORK 1
#endif
#ifndef FM_FORK_CTAS_PER_SM
#define FM_FORK_CTAS_PER_SM 1
#endif
// Cross-attention at small batches: K/V requested before the dependency wait when the
// draft is forked.
#ifndef FM_XATTN_EARLY
#define FM_XATTN_EARLY 1
#endif
// Cross-attention items handed out through a counter (1) or by fixed stride (0).
#ifndef FM_XATTN_DYNAMIC
#define FM_XATTN_DYNAMIC 1
#endif

namespace {
// Records an event pair around one launch while profiling is on.
struct Prof {
  flashmap_model* m;
  cudaStream_t s;
  bool on;
  Prof(flashmap_model* m_, cudaStream_t s_, int kind, int layer, int rows = 0, int n = 0, int k = 0)
      : m(m_), s(s_), on(m_->prof_on && static_cast<int>(m_->prof_recs.size()) < m_->prof_cap) {
    if (!on) return;
    const size_t i = m->prof_recs.size();
    if (m->prof_events.size() < 2 * (i + 1)) {
      cudaEvent_t a, b;
      cudaEventCreate(&a);
      cudaEventCreate(&b);
      m->prof_events.push_back(a);
      m->prof_events.push_back(b);
    }
    m->prof_recs.push_back(flashmap_launch_record{kind, layer, rows, n, k, 0.f});
    cudaEventRecord(m->prof_events[2 * i], s);
  }
  ~Prof() {
    if (on) cudaEventRecord(m->prof_events[2 * (m->prof_recs.size() - 1) + 1], s);
  }
};
}  // namespace

#define PROF(kind, layer, ...) Prof prof_##__LINE__(m, s, kind, layer, ##__VA_ARGS__)
#define TIMED(kind, layer, call) \
  do {                           \
    PROF(kind, layer);           \
    FM_CUDA(call);               \
  } while (0)
#define TIMED_GEMM(layer, W, rows, call)       \
  do {                                         \
    PROF(FLASHMAP_KIND_GEMM, layer, rows, (W).N, (W).K); \
    FM_CUDA(call);                             \
  } while (0)

namespace {

bool is_act(int d) { return d == FLASHMAP_F32 || d == FLASHMAP_BF16; }

// configuration_flashmap.py, DEFAULT_JUMP_GRIDS: jump times for 1..4 steps.
constexpr float kJumpGrids[4][5] = {
    {0.0f, 1.0f},
    {0.0f, 0.8172569274902344f, 1.0f},
    {0.0f, 0.8010796308517456f, 0.8310279846191406f, 1.0f},
    {0.0f, 0.7906050682067871f, 0.8172569274902344f, 0.8379518389701843f, 1.0f},
};

flashmap_status validate(const flashmap_config* c) {
  if (!c) return fail(FLASHMAP_E_INVALID, "config is NULL");
  const int dims[] = {c->target_hidden, c->num_target_layers, c->hidden, c->num_layers, c->num_heads, c->head_dim,
                      c->intermediate, c->cond_dim, c->time_embed_dim, c->block_size, c->vocab_size,
                      c->page_size, c->max_position};
  for (int d : dims)
    if (d <= 0) return fail(FLASHMAP_E_INVALID, "every size in the config must be positive");
  if (c->draft_vocab_size < 0) return fail(FLASHMAP_E_INVALID, "draft_vocab_size must be >= 0");
  if (c->noise_path != 0 && c->noise_path != 1)
    return fail(FLASHMAP_E_INVALID, "noise_path must be 0 (z L^T) or 1 (folded eigenbasis)");
  if (c->noise_path == 1 && c->num_steps != 1)
    return fail(FLASHMAP_E_UNSUPPORTED, "the folded-noise path is a one-jump path (num_steps = 1)");
  if (c->num_steps < 1 || c->num_steps > 4)
    return fail(FLASHMAP_E_UNSUPPORTED, "num_steps must be 1..4 (the printed jump grids); got " +
                                            std::to_string(c->num_steps));
  if (c->hidden != c->num_heads * c->head_dim) return fail(FLASHMAP_E_INVALID, "hidden != num_heads * head_dim");
  if (c->head_dim != 32 && c->head_dim != 64 && c->head_dim != 128)
    return fail(FLASHMAP_E_UNSUPPORTED, "head_dim must be 32, 64 or 128");
  if (c->block_size > 16) return fail(FLASHMAP_E_UNSUPPORTED, "block_size must be <= 16");
  if (c->page_size % 16) return fail(FLASHMAP_E_UNSUPPORTED, "page_size must be a multiple of 16");
  if (c->time_embed_dim % 2) return fail(FLASHMAP_E_INVALID, "time_embed_dim must be even");
  if (c->cond_dim > 8192 || c->time_embed_dim > 8192) return fail(FLASHMAP_E_UNSUPPORTED, "cond_dim too large");
  if (!is_act(c->act_dtype)) return fail(FLASHMAP_E_INVALID, "act_dtype must be F32 or BF16");
  if (c->weight_dtype != c->act_dtype && !(c->weight_dtype == FLASHMAP_E4M3 && c->act_dtype == FLASHMAP_BF16))
    return fail(FLASHMAP_E_INVALID, "weight_dtype must equal act_dtype (or E4M3 with BF16 activations)");
  if (c->kv_dtype != c->act_dtype && !(c->kv_dtype == FLASHMAP_E4M3 && c->act_dtype == FLASHMAP_BF16))
    return fail(FLASHMAP_E_INVALID, "kv_dtype must equal act_dtype (or E4M3 with BF16 activations)");
  if (c->weight_dtype == FLASHMAP_E4M3 && (c->target_hidden % 16 || c->hidden % 16 || c->intermediate % 16))
    return fail(FLASHMAP_E_UNSUPPORTED, "E4M3 weights need target_hidden, hidden and intermediate multiples of 16");
  {
    const int a[] = {c->target_hidden, c->hidden, c->intermediate};
    for (int d : a)
      if (d % 8) return fail(FLASHMAP_E_UNSUPPORTED, "target_hidden, hidden and intermediate must be multiples of 8");
    // the state rows feed a GEMM over the vocabulary; a row spreads over at most 8 CTAs
    if (c->num_steps > 1 && (c->vocab_size % 8 || c->vocab_size > 393216))
      return fail(FLASHMAP_E_UNSUPPORTED, "several jumps need vocab_size a multiple of 8 and <= 393216");
    if (c->target_hidden > 16384 || c->hidden > 16384)
      return fail(FLASHMAP_E_UNSUPPORTED, "target_hidden and hidden must be <= 16384");
  }
  if (c->max_position > (1 << 18)) return fail(FLASHMAP_E_UNSUPPORTED, "max_position must be <= 262144");
  if (!(c->rope_theta > 0) || !(c->time_scale >= 0) || !(c->rms_norm_eps >= 0) || !(c->qk_norm_eps >= 0) ||
      !(c->layer_norm_eps >= 0))
    return fail(FLASHMAP_E_INVALID, "rope_theta, time_scale and eps values must be non-negative");
  return FLASHMAP_OK;
}

int draft_vocab(const flashmap_config* c) {
  return (c->draft_vocab_size > 0 && c->draft_vocab_size < c->vocab_size) ? c->draft_vocab_size : c->vocab_size;
}

// The rotary table: inv_freq_i = float32(theta^(-2i/hd)) computed in float64; the
// angle of position p is the float32 product float32(p) * inv_freq_i; cos and sin of
// that angle are evaluated in float64 and stored as float32
// (flashmap/modeling_flashmap.py, rope_tables: float32 angles).
std::vector<float2> rope_table(int maxpos, int hd, double theta) {
  std::vector<float> inv(hd / 2);
  for (int i = 0; i < hd / 2; ++i) inv[i] = static_cast<float>(1.0 / std::pow(theta, (2.0 * i) / hd));
  std::vector<float2> t(static_cast<size_t>(maxpos) * (hd / 2));
  for (int p = 0; p < maxpos; ++p) {
    for (int i = 0; i < hd / 2; ++i) {
      volatile float a = static_cast<float>(p) * inv[i];
      const double ad = static_cast<double>(a);
      t[static_cast<size_t>(p) * (hd / 2) + i] = make_float2(static_cast<float>(std::cos(ad)), static_cast<float>(std::sin(ad)));
    }
  }
  return t;
}

struct DraftWs {
  float *x, *acc_big, *acc_d, *acc_a, *acc_kv;
  void *act, *e_rows;
  void* kv_in;  // rows the all-layer context K/V GEMM projects: the anchors, then a deferred write's
  // a deferred verify-window write (draft with write): its fc accumulator, the committed
  // rows gathered, their window rows, their count and anchors + count
  float* acc_fc = nullptr;
  void* xc = nullptr;
  int32_t* row_src = nullptr;
  int *wcnt = nullptr, *wtotal = nullptr;
  void* act_f;  // the MLP's hidden activations GELU(fc1), [R][F] act dtype
  int32_t *exp_pos, *exp_rpi;  // per-block request arrays of a multi-candidate draft
  // GEMM split-tile scratch of the main stream and of the anchor branch
  fm::GemmScratch red_main, red_side;
  // several jumps: the state (R x V float32), [posterior; state] in act dtype (2R x V),
  // their embeddings (2R x H float32) and the full-vocabulary logits (R x V float32)
  float *state = nullptr, *emb = nullptr, *logits_full = nullptr;
  void* xbuf = nullptr;
  int* plan;
  float *part_o, *part_ml;
  unsigned* xnext;  // the cross-attention items kernel's work counter
  size_t bytes;
};

bool write_can_compact(const flashmap_model* m);

// bs: the blocks drafted; wrows: the rows of a deferred verify-window write (0: none).
DraftWs carve_draft(const flashmap_model* m, int bs, void* base, int wrows = 0) {
  Carver c(base);
  const size_t R = static_cast<size_t>(bs) * m->K, es = dt_size(m->adt);
  const size_t big = std::max(3 * static_cast<size_t>(m->D), static_cast<size_t>(m->H));  // qkv, or the noise z L^T
  const size_t wide = std::max(static_cast<size_t>(m->D), static_cast<size_t>(m->H));  // the MLP's F: act_f
  DraftWs w;
  w.x = c.take<float>(R * m->D * 4);
  w.acc_big = c.take<float>(R * big * 4);
  w.acc_d = c.take<float>(R * m->D * 4);
  w.acc_a = c.take<float>(static_cast<size_t>(bs) * m->D * 4);
  w.acc_kv = c.take<float>(static_cast<size_t>(bs + wrows) * 2 * m->L * m->D * 4);
  w.act = c.take<void>(R * wide * es);
  w.act_f = c.take<void>(R * static_cast<size_t>(m->F) * es);
  w.e_rows = c.take<void>(static_cast<size_t>(bs) * m->H * es);
  w.kv_in = c.take<void>(static_cast<size_t>(bs + wrows) * m->D * es);
  if (wrows > 0) {
    w.acc_fc = c.take<float>(static_cast<size_t>(wrows) * m->D * 4);
    if (write_can_compact(m)) {
      w.xc = c.take<void>(static_cast<size_t>(wrows) * m->Lt * m->H * es);
      w.row_src = c.take<int32_t>(static_cast<size_t>(wrows) * 4);
      w.wcnt = c.take<int>(4);
      w.wtotal = c.take<int>(4);
    }
  }
  w.exp_pos = c.take<int32_t>(static_cast<size_t>(bs) * 4);
  w.exp_rpi = c.take<int32_t>(static_cast<size_t>(bs) * 4);
  if (m->steps > 1) {
    const size_t V = static_cast<size_t>(m->V);
    w.state = c.take<float>(R * V * 4);
    w.xbuf = c.take<void>(2 * R * V * es);
    w.emb = c.take<float>(2 * R * m->H * 4);
    w.logits_full = c.take<float>(R * V * 4);
  }
  w.plan = c.take<int>(fm::xattn_plan_ints(m->num_sms, m->nh, bs) * 4);
  const size_t chunks = fm::xattn_max_chunks(m->num_sms, m->nh, bs);
  w.part_o = c.take<float>(chunks * m->nh * 16 * m->hd * 4);
  w.part_ml = c.take<float>(chunks * m->nh * 32 * 4);
  w.xnext = c.take<unsigned>(4);
  {
    const int main_rows = static_cast<int>(m->steps > 1 ? 2 * R : R);
    w.red_main = fm::gemm_scratch_carve(c.take<uint8_t>(fm::gemm_scratch_bytes(main_rows, m->num_sms)), main_rows,
                                        m->num_sms);
    w.red_side = fm::gemm_scratch_carve(c.take<uint8_t>(fm::gemm_scratch_bytes(bs + wrows, m->num_sms)), bs + wrows,
                                        m->num_sms);
  }
  w.bytes = align_up(c.off);
  return w;
}

// A verify-window write of at least this many columns projects only the committed
// ones (compacted on the device); smaller ones project every column and skip the
// uncommitted ones at the scatter.
#ifndef FM_WRITE_COMPACT_MIN_ROWS
#define FM_WRITE_COMPACT_MIN_ROWS 48
#endif
struct WriteWs {
  float *acc_fc, *acc_kv;
  void* ctx;
  void* xc = nullptr;           // the committed rows of the target hidden states
  int32_t* row_src = nullptr;   // their window rows
  int* rows_dev = nullptr;      // their count
  fm::GemmScratch red;          // GEMM split-tile scratch
};
// The compacted write needs the tcgen05 GEMMs (device row counts).
bool write_can_compact(const flashmap_model* m) { return m->wdt != FLASHMAP_F32; }
size_t write_row_bytes(const flashmap_model* m) {
  const size_t xrow = static_cast<size_t>(m->Lt) * m->H * dt_size(m->adt);
  return static_cast<size_t>(m->D) * 4 + static_cast<size_t>(m->D) * dt_size(m->adt) +
         static_cast<size_t>(2) * m->L * m->D * 4 + (write_can_compact(m) ? xrow + 4 : 0);
}
WriteWs carve_write(const flashmap_model* m, int rows, void* base, size_t* bytes) {
  Carver c(base);
  WriteWs w;
  w.acc_fc = c.take<float>(static_cast<size_t>(rows) * m->D * 4);
  w.ctx = c.take<void>(static_cast<size_t>(rows) * m->D * dt_size(m->adt));
  w.acc_kv = c.take<float>(static_cast<size_t>(rows) * 2 * m->L * m->D * 4);
  if (write_can_compact(m)) {
    w.xc = c.take<void>(static_cast<size_t>(rows) * m->Lt * m->H * dt_size(m->adt));
    w.row_src = c.take<int32_t>(static_cast<size_t>(rows) * 4);
    w.rows_dev = c.take<int>(4);
  }
  w.red = fm::gemm_scratch_carve(c.take<uint8_t>(fm::gemm_scratch_bytes(rows, m->num_sms)), rows, m->num_sms);
  *bytes = align_up(c.off);
  return w;
}

// sample workspace: the row keys and counters of the split sampler, then the draft
// logits unless the caller takes them
struct SampleWs {
  unsigned long long* keys;
  unsigned* counters;
  float* logits;
  fm::GemmScratch red;  // GEMM split-tile scratch
  size_t bytes;
};
SampleWs carve_sample(const flashmap_model* m, int bs, bool own_logits, void* base) {
  Carver c(base);
  const size_t R = static_cast<size_t>(bs) * m->K;
  SampleWs w;
  w.keys = c.take<unsigned long long>(R * 8);
  w.counters = c.take<unsigned>(R * 4);
  w.logits = own_logits ? c.take<float>(R * m->Vd * 4) : nullptr;
  w.red = fm::gemm_scratch_carve(c.take<uint8_t>(fm::gemm_scratch_bytes(static_cast<int>(R), m->num_sms)),
                                 static_cast<int>(R), m->num_sms);
  w.bytes = align_up(c.off);
  return w;
}

flashmap_status check_weight_map(Weight& w, int dtype, std::string* err) {
  w.dtype = dtype;
  if (dtype == FLASHMAP_BF16) {
    if (!fm::make_tmap_bf16(&w.map, w.ptr, w.N, w.K, w.K, 128, err)) return FLASHMAP_E_CUDA;
    w.has_map = true;
  } else if (dtype == FLASHMAP_E4M3) {
    if (!fm::make_tmap_e4m3(&w.map, w.ptr, w.N, w.K, err)) return FLASHMAP_E_CUDA;
    w.has_map = true;
  }
  return FLASHMAP_OK;
}

}  // namespace

extern "C" {

const char* flashmap_last_error(void) { return g_last_error.c_str(); }

flashmap_status flashmap_validate_config(const flashmap_config* cfg) {
  g_last_error.clear();
  return validate(cfg);
}

flashmap_status flashmap_pool_bytes(const flashmap_config* cfg, int64_t num_pages, size_t* bytes) {
  g_last_error.clear();
  flashmap_status st = validate(cfg);
  if (st != FLASHMAP_OK) return st;
  if (!bytes || num_pages <= 0) return fail(FLASHMAP_E_INVALID, "num_pages must be positive and bytes non-NULL");
  *bytes = static_cast<size_t>(cfg->num_layers) * 2 * static_cast<size_t>(num_pages) * cfg->num_heads *
           cfg->page_size * cfg->head_dim * dt_size(cfg->kv_dtype);
  return FLASHMAP_OK;
}

flashmap_status flashmap_get_config(const flashmap_model* model, flashmap_config* cfg) {
  if (!model || !cfg) return fail(FLASHMAP_E_INVALID, "NULL argument");
  *cfg = model->cfg;
  return FLASHMAP_OK;
}

flashmap_status flashmap_free(flashmap_model* model) {
  if (!model) return FLASHMAP_OK;
  if (model->arena) cudaFree(model->arena);
  for (cudaEvent_t e : model->prof_events) cudaEventDestroy(e);
  if (model->ev_fork) cudaEventDestroy(model->ev_fork);
  if (model->ev_join) cudaEventDestroy(model->ev_join);
  if (model->side) cudaStreamDestroy(model->side);
  delete model;
  return FLASHMAP_OK;
}

flashmap_status flashmap_load_weights(const flashmap_config* cfg, const flashmap_weights* w, const void* embedding,
                                      const void* lm_head, const int64_t* vocab_ranking, flashmap_stream stream,
                                      flashmap_model** out) {
  g_last_error.clear();
  flashmap_status st = validate(cfg);
  if (st != FLASHMAP_OK) return st;
  if (!w || !embedding || !lm_head || !out || !w->layers) return fail(FLASHMAP_E_INVALID, "NULL argument");
  {
    const void* req[] = {w->fc_w, w->hidden_norm_w, w->anchor_proj_w, w->anchor_proj_b, w->anchor_norm_w,
                         w->state_norm_w, w->noise_norm_w, w->noise_gate, w->x_embed_w, w->x_embed_b,
                         w->time_l1_w, w->time_l1_b, w->time_l2_w, w->time_l2_b, w->jump_l1_w, w->jump_l1_b,
                         w->jump_l2_w, w->jump_l2_b, w->final_adaln_w, w->final_adaln_b, w->head_w, w->head_b};
    for (const void* p : req)
      if (!p) return fail(FLASHMAP_E_INVALID, "a weight pointer is NULL");
    for (int l = 0; l < cfg->num_layers; ++l) {
      const flashmap_layer_weights& lw = w->layers[l];
      const void* lr[] = {lw.self_adaln_w, lw.self_adaln_b, lw.self_q_w, lw.self_k_w, lw.self_v_w, lw.self_o_w,
                          lw.self_q_norm_w, lw.self_k_norm_w, lw.cross_adaln_w, lw.cross_adaln_b, lw.cross_q_w,
                          lw.cross_k_w, lw.cross_v_w, lw.cross_o_w, lw.cross_q_norm_w, lw.cross_k_norm_w,
                          lw.mlp_adaln_w, lw.mlp_adaln_b, lw.fc1_w, lw.fc1_b, lw.fc2_w, lw.fc2_b};
      for (const void* p : lr)
        if (!p) return fail(FLASHMAP_E_INVALID, "a layer weight pointer is NULL (layer " + std::to_string(l) + ")");
    }
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto* m = new flashmap_model();
  auto cleanup = [&](flashmap_status code) {
    flashmap_free(m);
    return code;
  };
  m->cfg = *cfg;
  m->adt = cfg->act_dtype;
  m->wdt = cfg->weight_dtype;
  m->kdt = cfg->kv_dtype;
  m->H = cfg->target_hidden;
  m->Lt = cfg->num_target_layers;
  m->D = cfg->hidden;
  m->L = cfg->num_layers;
  m->nh = cfg->num_heads;
  m->hd = cfg->head_dim;
  m->F = cfg->intermediate;
  m->K = cfg->block_size;
  m->V = cfg->vocab_size;
  m->Vd = vocab_ranking ? draft_vocab(cfg) : cfg->vocab_size;  // no ranking: the full vocabulary
  m->P = cfg->page_size;
  m->maxpos = cfg->max_position;
  m->steps = cfg->num_steps;
  m->noise_path = cfg->noise_path;
  for (int i = 0; i <= m->steps; ++i) m->grid[i] = kJumpGrids[m->steps - 1][i];
  m->embedding = embedding;
  if (cudaGetDevice(&m->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device) != cudaSuccess)
    return cleanup(fail(FLASHMAP_E_CUDA, "no CUDA device"));
  if (cudaStreamCreateWithFlags(&m->side, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&m->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&m->ev_join, cudaEventDisableTiming) != cudaSuccess)
    return cleanup(fail(FLASHMAP_E_CUDA, "could not create the model's side stream and events"));
  const int adt = m->adt;
  const bool e4m3 = m->wdt == FLASHMAP_E4M3;
  const size_t es = dt_size(adt);
  const int64_t H = m->H, D = m->D, L = m->L, F = m->F, Vd = m->Vd, V = m->V, hd = m->hd, C = cfg->cond_dim;

  // ---- arena layout. With e4m3 weights every large GEMM weight (all but the noise
  // factor L) is stored as e4m3 plus one float32 scale per output channel
  // (flashmap/sglang/model.py, _quantize_fp8).
  auto layout = [&](Carver& c) {
    auto big = [&](Weight& W, int64_t rows, int64_t cols) {
      W.ptr = c.take<void>(rows * cols * (e4m3 ? 1 : es));
      W.wscale = e4m3 ? c.take<float>(rows * 4) : nullptr;
    };
    big(m->fc, D, m->Lt * H);
    big(m->ap, D, H);
    big(m->ctx_kv, 2 * L * D, D);
    m->chol.ptr = c.take<void>(H * H * es);
    big(m->xe, D, H);
    big(m->head, Vd, D);
    m->layers.resize(L);
    for (auto& lw : m->layers) {
      big(lw.qkv, 3 * D, D);
      big(lw.o, D, D);
      big(lw.cq, D, D);
      big(lw.co, D, D);
      big(lw.fc1, F, D);
      big(lw.fc2, D, F);
      lw.qn = c.take<float>(hd * 4);
      lw.kn = c.take<float>(hd * 4);
      lw.cqn = c.take<float>(hd * 4);
      lw.mods = c.take<float>(9 * D * 4);
      lw.fc1_b = c.take<float>(F * 4);
      lw.fc2_beta = c.take<float>(D * 4);
    }
    m->hidden_norm_w = c.take<float>(D * 4);
    m->anchor_norm_w = c.take<float>(D * 4);
    m->noise_norm_w = c.take<float>(H * 4);
    m->ap_b = c.take<float>(D * 4);
    m->xe_b = c.take<float>(D * 4);
    m->head_b = c.take<float>(Vd * 4);
    m->ctx_knorm = c.take<float>(L * hd * 4);
    m->final_mods = c.take<float>(2 * D * 4);
    m->u = c.take<float>(H * 4);
    m->hot = c.take<int64_t>(Vd * 8);
    m->inv_hot = c.take<int32_t>(V * 4);
    m->rope = c.take<float2>(static_cast<size_t>(m->maxpos) * (hd / 2) * 8);
    m->dev_err = c.take<unsigned>(256);
    if (m->steps > 1) {
      m->et.ptr = c.take<void>(H * V * es);
      m->full_head.ptr = c.take<void>(V * D * es);
      m->full_head_b = c.take<float>(V * 4);
      m->state_norm_w = c.take<float>(H * 4);
      m->step_mods = c.take<float>(static_cast<size_t>(m->steps) * L * 9 * D * 4);
      m->step_final = c.take<float>(static_cast<size_t>(m->steps) * 2 * D * 4);
      m->step_fc2_beta = c.take<float>(static_cast<size_t>(m->steps) * L * D * 4);
    }
    if (m->noise_path == 1) {
      m->fold.ptr = c.take<void>(D * H * es);
      m->fold_var = c.take<float>(H * 4);
      m->fold_xu = c.take<float>(D * 4);
    }
  };
  Carver measure(nullptr);
  layout(measure);
  if (cudaMalloc(&m->arena, measure.off) != cudaSuccess) {
    cudaGetLastError();
    m->arena = nullptr;
    return cleanup(fail(FLASHMAP_E_NOMEM, "cannot allocate " + std::to_string(measure.off) + " bytes of weights"));
  }
  Carver arena(m->arena);
  layout(arena);

  // Load-time scratch: gram (float64 H x H), column sums, conditioning, fc2 bias.
  void* scratch = nullptr;
  const size_t fold_bytes = m->noise_path == 1 ? align_up(fm::folded_scratch_bytes(static_cast<int>(H))) : 0;
  const size_t scratch_bytes =
      align_up(H * H * 8) + align_up(static_cast<size_t>(fm::colsum_doubles(m->V, m->H)) * 8) + align_up(C * 8) +
      align_up(std::max(D, H) * 4) + fold_bytes;
  if (cudaMalloc(&scratch, scratch_bytes) != cudaSuccess) {
    cudaGetLastError();
    return cleanup(fail(FLASHMAP_E_NOMEM, "cannot allocate load-time scratch"));
  }
  struct ScratchGuard {
    void* p;
    ~ScratchGuard() { cudaFree(p); }
  } guard{scratch};
  Carver sc(scratch);
  double* gram = sc.take<double>(H * H * 8);
  double* colsum = sc.take<double>(static_cast<size_t>(fm::colsum_doubles(m->V, m->H)) * 8);
  double* cond = sc.take<double>(C * 8);
  float* tmp_d = sc.take<float>(std::max(D, H) * 4);  // D or H floats of scratch
  void* fold_scratch = fold_bytes ? sc.take<void>(fold_bytes) : nullptr;
  // e4m3: each weight is assembled in act_dtype (the folded head in float32) in one
  // staging buffer, then quantized into the arena; stream order serializes the reuse.
  void* stage = nullptr;
  if (e4m3) {
    const size_t stage_bytes = std::max({static_cast<size_t>(D * m->Lt * H) * es, static_cast<size_t>(2 * L * D * D) * es,
                                         static_cast<size_t>(3 * D * D) * es, static_cast<size_t>(F * D) * es,
                                         static_cast<size_t>(D * H) * es, static_cast<size_t>(Vd * D) * 4});
    if (cudaMalloc(&stage, stage_bytes) != cudaSuccess) {
      cudaGetLastError();
      return cleanup(fail(FLASHMAP_E_NOMEM, "cannot allocate the e4m3 staging buffer"));
    }
  }
  struct StageGuard {
    void* p;
    ~StageGuard() {
      if (p) cudaFree(p);
    }
  } stage_guard{stage};

#define LCHK(call)                                                                                  \
  do {                                                                                              \
    cudaError_t e_ = (call);                                                                        \
    if (e_ != cudaSuccess) return cleanup(fail(FLASHMAP_E_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_))); \
  } while (0)

  LCHK(fm::gemm_prepare());
  LCHK(fm::xattn_prepare());
  if (m->steps > 1) LCHK(fm::jumps_prepare(m->V));
  LCHK(cudaMemsetAsync(m->dev_err, 0, 4, s));
  auto copy = [&](void* dst, const void* src, size_t bytes) { return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s); };
  auto bytes_of = [&](int64_t rows, int64_t cols) { return static_cast<size_t>(rows) * cols * es; };
  // where a weight's raw values go: its arena slot, or the staging buffer (e4m3)
  auto dst = [&](Weight& W) { return static_cast<uint8_t*>(e4m3 ? stage : const_cast<void*>(W.ptr)); };
  // e4m3: quantize the staged weight (rows x cols, src_dtype) into its arena slot
  auto finish = [&](Weight& W, int64_t rows, int64_t cols, int src_dtype) -> cudaError_t {
    if (!e4m3) return cudaSuccess;
    return fm::quantize_e4m3(s, stage, src_dtype, static_cast<int>(rows), static_cast<int>(cols),
                             const_cast<void*>(W.ptr), const_cast<float*>(W.wscale));
  };
  // ---- copies: the all-layer context K/V weight [k_0; v_0; ...] and fused q/k/v
  LCHK(copy(dst(m->fc), w->fc_w, bytes_of(D, m->Lt * H)));
  LCHK(finish(m->fc, D, m->Lt * H, adt));
  LCHK(copy(dst(m->ap), w->anchor_proj_w, bytes_of(D, H)));
  LCHK(finish(m->ap, D, H, adt));
  LCHK(copy(dst(m->xe), w->x_embed_w, bytes_of(D, H)));
  LCHK(finish(m->xe, D, H, adt));
  {
    uint8_t* ck = dst(m->ctx_kv);
    for (int l = 0; l < L; ++l) {
      LCHK(copy(ck + bytes_of(2 * l * D, D), w->layers[l].cross_k_w, bytes_of(D, D)));
      LCHK(copy(ck + bytes_of((2 * l + 1) * D, D), w->layers[l].cross_v_w, bytes_of(D, D)));
    }
    LCHK(finish(m->ctx_kv, 2 * L * D, D, adt));
  }
  for (int l = 0; l < L; ++l) {
    const flashmap_layer_weights& lw = w->layers[l];
    LayerW& d = m->layers[l];
    uint8_t* q = dst(d.qkv);
    LCHK(copy(q, lw.self_q_w, bytes_of(D, D)));
    LCHK(copy(q + bytes_of(D, D), lw.self_k_w, bytes_of(D, D)));
    LCHK(copy(q + bytes_of(2 * D, D), lw.self_v_w, bytes_of(D, D)));
    LCHK(finish(d.qkv, 3 * D, D, adt));
    LCHK(copy(dst(d.o), lw.self_o_w, bytes_of(D, D)));
    LCHK(finish(d.o, D, D, adt));
    LCHK(copy(dst(d.cq), lw.cross_q_w, bytes_of(D, D)));
    LCHK(finish(d.cq, D, D, adt));
    LCHK(copy(dst(d.co), lw.cross_o_w, bytes_of(D, D)));
    LCHK(finish(d.co, D, D, adt));
    LCHK(copy(dst(d.fc1), lw.fc1_w, bytes_of(F, D)));
    LCHK(finish(d.fc1, F, D, adt));
    LCHK(copy(dst(d.fc2), lw.fc2_w, bytes_of(D, F)));
    LCHK(finish(d.fc2, D, F, adt));
    LCHK(fm::to_f32(s, lw.self_q_norm_w, adt, hd, d.qn));
    LCHK(fm::to_f32(s, lw.self_k_norm_w, adt, hd, d.kn));
    LCHK(fm::to_f32(s, lw.cross_q_norm_w, adt, hd, d.cqn));
    LCHK(fm::to_f32(s, lw.cross_k_norm_w, adt, hd, m->ctx_knorm + l * hd));
    LCHK(fm::to_f32(s, lw.fc1_b, adt, F, d.fc1_b));
  }
  LCHK(fm::to_f32(s, w->hidden_norm_w, adt, D, m->hidden_norm_w));
  LCHK(fm::to_f32(s, w->anchor_norm_w, adt, D, m->anchor_norm_w));
  LCHK(fm::to_f32(s, w->noise_norm_w, adt, H, m->noise_norm_w));
  LCHK(fm::to_f32(s, w->anchor_proj_b, adt, D, m->ap_b));
  LCHK(fm::to_f32(s, w->x_embed_b, adt, D, m->xe_b));

  // ---- AdaLN modulations of the jump 0 -> 1
  fm::TimeCondArgs ta{w->time_l1_w, w->time_l1_b, w->time_l2_w, w->time_l2_b, w->jump_l1_w, w->jump_l1_b,
                      w->jump_l2_w, w->jump_l2_b, adt, cfg->cond_dim, cfg->time_embed_dim, 0.0, 1.0,
                      static_cast<double>(cfg->time_scale)};
  LCHK(fm::time_cond(s, ta, cond));
  for (int l = 0; l < L; ++l) {
    const flashmap_layer_weights& lw = w->layers[l];
    LayerW& d = m->layers[l];
    const void* aw[3] = {lw.self_adaln_w, lw.cross_adaln_w, lw.mlp_adaln_w};
    const void* ab[3] = {lw.self_adaln_b, lw.cross_adaln_b, lw.mlp_adaln_b};
    for (int j = 0; j < 3; ++j)
      LCHK(fm::adaln(s, aw[j], ab[j], adt, cfg->cond_dim, m->D, cond, d.mods + (3 * j) * D, d.mods + (3 * j + 1) * D,
                     d.mods + (3 * j + 2) * D));
    // fc2's bias enters the gated residual as gate * b2
    LCHK(fm::to_f32(s, lw.fc2_b, adt, D, tmp_d));
    LCHK(fm::mul_vec(s, d.mods + 8 * D, tmp_d, d.fc2_beta, m->D));
  }
  LCHK(fm::adaln(s, w->final_adaln_w, w->final_adaln_b, adt, cfg->cond_dim, m->D, cond, m->final_mods,
                 m->final_mods + D, nullptr));
  // ---- several jumps: the conditioning of every jump (s, t) of the grid
  for (int st = 0; m->steps > 1 && st < m->steps; ++st) {
    fm::TimeCondArgs tj = ta;
    tj.s = m->grid[st];
    tj.t = m->grid[st + 1];
    LCHK(fm::time_cond(s, tj, cond));
    for (int l = 0; l < L; ++l) {
      const flashmap_layer_weights& lw = w->layers[l];
      float* md = m->step_mods + (static_cast<size_t>(st) * L + l) * 9 * D;
      const void* aw[3] = {lw.self_adaln_w, lw.cross_adaln_w, lw.mlp_adaln_w};
      const void* ab[3] = {lw.self_adaln_b, lw.cross_adaln_b, lw.mlp_adaln_b};
      for (int j = 0; j < 3; ++j)
        LCHK(fm::adaln(s, aw[j], ab[j], adt, cfg->cond_dim, m->D, cond, md + (3 * j) * D, md + (3 * j + 1) * D,
                       md + (3 * j + 2) * D));
      LCHK(fm::to_f32(s, lw.fc2_b, adt, D, tmp_d));
      LCHK(fm::mul_vec(s, md + 8 * D, tmp_d, m->step_fc2_beta + (static_cast<size_t>(st) * L + l) * D, m->D));
    }
    float* fin = m->step_final + static_cast<size_t>(st) * 2 * D;
    LCHK(fm::adaln(s, w->final_adaln_w, w->final_adaln_b, adt, cfg->cond_dim, m->D, cond, fin, fin + D, nullptr));
  }

  // ---- the uniform posterior's embedding and the Cholesky factor of E^T E
  LCHK(fm::to_f32(s, w->state_norm_w, adt, H, tmp_d));
  LCHK(fm::uniform_constant(s, embedding, adt, V, m->H, tmp_d, cfg->rms_norm_eps, colsum, m->u));
  if (m->noise_path == 1) {  // the eigenbasis is sensitive to the gram: float64 products and sums
    LCHK(fm::gram_f64(s, embedding, adt, V, m->H, gram));
  } else {  // float32 partial sums of 1024 products, added in float64 in order
    LCHK(fm::simt_gemm(s, m->H, m->H, m->V, embedding, adt, nullptr, 1, H, embedding, adt, H, 1, gram, FLASHMAP_F32, H, 2));
  }
  LCHK(fm::cholesky_f64(s, gram, m->H, m->dev_err));
  LCHK(fm::chol_store(s, gram, m->H, adt, const_cast<void*>(m->chol.ptr)));
  if (m->noise_path == 1) {
    // the eigenbasis of E^T E from X = L^T (the factor's storage is taken over), then
    // the folded projection, lam / H and x_embed(u)
    std::string eerr;
    const cudaError_t e = fm::folded_noise_constants(s, gram, m->H, fold_scratch, m->noise_norm_w, w->x_embed_w,
                                                     w->x_embed_b, adt, m->D, m->u, const_cast<void*>(m->fold.ptr),
                                                     m->fold_var, m->fold_xu, &m->eig_sweeps, &eerr);
    if (e != cudaSuccess)
      return cleanup(fail(FLASHMAP_E_CUDA, eerr.empty() ? std::string("folded noise: ") + cudaGetErrorString(e) : eerr));
  }

  // ---- draft vocabulary and the folded head
  {
    std::vector<int64_t> hot(Vd);
    if (Vd < V) {
      std::vector<int64_t> rank(V);
      LCHK(cudaMemcpyAsync(rank.data(), vocab_ranking, V * 8, cudaMemcpyDeviceToHost, s));
      LCHK(cudaStreamSynchronize(s));
      std::copy(rank.begin(), rank.begin() + Vd, hot.begin());
      std::sort(hot.begin(), hot.end());
      for (int64_t i = 0; i < Vd; ++i)
        if (hot[i] < 0 || hot[i] >= V || (i && hot[i] == hot[i - 1]))
          return cleanup(fail(FLASHMAP_E_INVALID, "vocab_ranking must hold distinct token ids in [0, V)"));
    } else {
      for (int64_t i = 0; i < V; ++i) hot[i] = i;
    }
    std::vector<int32_t> inv(V, -1);
    for (int64_t i = 0; i < m->Vd; ++i) inv[hot[i]] = static_cast<int32_t>(i);
    LCHK(cudaMemcpyAsync(m->hot, hot.data(), m->Vd * 8, cudaMemcpyHostToDevice, s));
    LCHK(cudaMemcpyAsync(m->inv_hot, inv.data(), V * 4, cudaMemcpyHostToDevice, s));
    // W_f = LM[hot] W_head (Vd x D), b_f = LM[hot] b_head, float32 accumulation
    LCHK(fm::simt_gemm(s, m->Vd, m->D, m->H, lm_head, adt, m->hot, H, 1, w->head_w, adt, D, 1, dst(m->head),
                       e4m3 ? FLASHMAP_F32 : adt, D, 1));
    LCHK(finish(m->head, Vd, D, FLASHMAP_F32));
    LCHK(fm::simt_gemm(s, m->Vd, 1, m->H, lm_head, adt, m->hot, H, 1, w->head_b, adt, 1, 0, m->head_b,
                       FLASHMAP_F32, 1, 0));
    if (m->steps > 1) {
      // E^T (H x V) for [posterior; state] @ E, and the full-vocabulary folded head
      // LM (W_head, b_head) for the state update between jumps (float32 accumulation)
      LCHK(fm::transpose(s, adt, embedding, V, H, const_cast<void*>(m->et.ptr)));
      LCHK(fm::simt_gemm(s, m->V, m->D, m->H, lm_head, adt, nullptr, H, 1, w->head_w, adt, D, 1,
                         const_cast<void*>(m->full_head.ptr), adt, D, 1));
      LCHK(fm::simt_gemm(s, m->V, 1, m->H, lm_head, adt, nullptr, H, 1, w->head_b, adt, 1, 0, m->full_head_b,
                         FLASHMAP_F32, 1, 0));
      LCHK(fm::to_f32(s, w->state_norm_w, adt, H, m->state_norm_w));
    }
    // rotary table
    std::vector<float2> rt = rope_table(m->maxpos, m->hd, cfg->rope_theta);
    LCHK(cudaMemcpyAsync(m->rope, rt.data(), rt.size() * sizeof(float2), cudaMemcpyHostToDevice, s));
    // the noise gate of the jump 0 -> 1: noise_gate * (t - s) = noise_gate
    float ng = 1.f;
    if (adt == FLASHMAP_F32) {
      LCHK(cudaMemcpyAsync(&ng, w->noise_gate, 4, cudaMemcpyDeviceToHost, s));
      LCHK(cudaStreamSynchronize(s));
    } else {
      __nv_bfloat16 b;
      LCHK(cudaMemcpyAsync(&b, w->noise_gate, 2, cudaMemcpyDeviceToHost, s));
      LCHK(cudaStreamSynchronize(s));
      ng = __bfloat162float(b);
    }
    m->gate = cfg->noise_gate_constant ? ng : ng * (1.0f - 0.0f);
    for (int st = 0; st < m->steps; ++st)  // the noise weight of jump st: noise_gate * (t - s), or noise_gate
      m->step_gate[st] = cfg->noise_gate_constant ? ng : ng * (m->grid[st + 1] - m->grid[st]);
    LCHK(cudaStreamSynchronize(s));  // host vectors above must outlive their copies
  }

  // ---- GEMM descriptors
  m->fc.N = m->D, m->fc.K = m->Lt * m->H;
  m->ap.N = m->D, m->ap.K = m->H;
  m->ctx_kv.N = 2 * m->L * m->D, m->ctx_kv.K = m->D;
  m->chol.N = m->H, m->chol.K = m->H;
  m->xe.N = m->D, m->xe.K = m->H;
  m->head.N = m->Vd, m->head.K = m->D;
  std::string err;
  Weight* ws[] = {&m->fc, &m->ap, &m->ctx_kv, &m->xe, &m->head};
  for (Weight* x : ws)
    if (check_weight_map(*x, m->wdt, &err) != FLASHMAP_OK) return cleanup(fail(FLASHMAP_E_CUDA, err));
  if (check_weight_map(m->chol, adt, &err) != FLASHMAP_OK) return cleanup(fail(FLASHMAP_E_CUDA, err));
  if (m->noise_path == 1) {
    m->fold.N = m->D, m->fold.K = m->H;
    if (check_weight_map(m->fold, adt, &err) != FLASHMAP_OK) return cleanup(fail(FLASHMAP_E_CUDA, err));
  }
  if (m->steps > 1) {
    m->et.N = m->H, m->et.K = m->V;
    m->full_head.N = m->V, m->full_head.K = m->D;
    if (check_weight_map(m->et, adt, &err) != FLASHMAP_OK || check_weight_map(m->full_head, adt, &err) != FLASHMAP_OK)
      return cleanup(fail(FLASHMAP_E_CUDA, err));
  }
  for (auto& d : m->layers) {
    d.qkv.N = 3 * m->D, d.qkv.K = m->D;
    d.o.N = m->D, d.o.K = m->D;
    d.cq.N = m->D, d.cq.K = m->D;
    d.co.N = m->D, d.co.K = m->D;
    d.fc1.N = m->F, d.fc1.K = m->D;
    d.fc2.N = m->D, d.fc2.K = m->F;
    Weight* lws[] = {&d.qkv, &d.o, &d.cq, &d.co, &d.fc1, &d.fc2};
    for (Weight* x : lws)
      if (check_weight_map(*x, m->wdt, &err) != FLASHMAP_OK) return cleanup(fail(FLASHMAP_E_CUDA, err));
  }
  LCHK(cudaStreamSynchronize(s));
  LCHK(cudaGetLastError());
  unsigned derr = 0;
  LCHK(cudaMemcpy(&derr, m->dev_err, 4, cudaMemcpyDeviceToHost));
  if (derr) return cleanup(fail(FLASHMAP_E_DEVICE, "E^T E is not positive definite (Cholesky pivot <= 0)"));
#undef LCHK
  *out = m;
  return FLASHMAP_OK;
}

flashmap_status flashmap_workspace_size(const flashmap_model* m, int32_t max_bs, int32_t max_write_rows,
                                        size_t* bytes) {
  g_last_error.clear();
  if (!m || !bytes || max_bs <= 0 || max_write_rows < 0) return fail(FLASHMAP_E_INVALID, "bad workspace query");
  size_t wb = 0;
  carve_write(m, std::max(max_write_rows, 1), nullptr, &wb);
  *bytes = std::max({carve_draft(m, max_bs, nullptr, max_write_rows).bytes, carve_sample(m, max_bs, true, nullptr).bytes,
                     wb});
  return FLASHMAP_OK;
}

flashmap_status flashmap_write_context_kv(flashmap_model* m, const flashmap_kv_pool* pool, const void* target_hidden,
                                          int32_t bs, int32_t W, const int32_t* req_pool_idx,
                                          const int32_t* start_pos, const int32_t* commit_lens,
                                          const int32_t* req_to_page, int32_t req_to_page_stride, int64_t* out_loc,
                                          void* workspace, size_t workspace_bytes, flashmap_stream stream) {
  g_last_error.clear();
  if (!m || !pool || !target_hidden || !req_pool_idx || !start_pos || !req_to_page || !workspace)
    return fail(FLASHMAP_E_INVALID, "NULL argument");
  if (bs <= 0 || W <= 0 || req_to_page_stride <= 0) return fail(FLASHMAP_E_INVALID, "bs, W and the page-table stride must be positive");
  if (pool->dtype != m->kdt || !pool->base || pool->num_pages <= 0)
    return fail(FLASHMAP_E_INVALID, "pool dtype must equal kv_dtype, with pages");
  if (m->adt == FLASHMAP_BF16 && (reinterpret_cast<uintptr_t>(target_hidden) & 15))
    return fail(FLASHMAP_E_INVALID, "target_hidden must be 16-byte aligned");
  const int64_t total = static_cast<int64_t>(bs) * W;
  const size_t per_row = write_row_bytes(m) + 3 * 256;
  int64_t chunk = static_cast<int64_t>(workspace_bytes / per_row);
  chunk = std::min<int64_t>(chunk, total);
  size_t need = 0;
  while (chunk > 0) {
    carve_write(m, static_cast<int>(chunk), nullptr, &need);
    if (need <= workspace_bytes) break;
    --chunk;
  }
  if (chunk <= 0) return fail(FLASHMAP_E_INVALID, "workspace too small for one write row");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const Launch Lh = m->launch(s);
  const size_t xrow = static_cast<size_t>(m->Lt) * m->H * dt_size(m->adt);
  for (int64_t r0 = 0; r0 < total; r0 += chunk) {
    const int rows = static_cast<int>(std::min<int64_t>(chunk, total - r0));
    size_t b = 0;
    WriteWs ws = carve_write(m, rows, workspace, &b);
    Launch Lw = Lh;
    Lw.red = ws.red;
    fm::ZeroList z;  // the GEMMs' split-tile counters (their outputs are written whole)
    z.add(reinterpret_cast<float*>(ws.red.cnt), ws.red.cnt_cap);  // zero bits
    TIMED(FLASHMAP_KIND_MEMSET, -1, fm::zero_ranges(Lw, z));
    const void* x = static_cast<const uint8_t*>(target_hidden) + r0 * xrow;
    // A large window projects only its committed columns: their rows are gathered in
    // order and counted on the device, and every kernel below takes that count
    // (uncommitted columns get out_loc -1 here).
    const bool compact = commit_lens && write_can_compact(m) && rows >= FM_WRITE_COMPACT_MIN_ROWS;
    const int* rows_dev = nullptr;
    if (compact) {
      TIMED(FLASHMAP_KIND_ROWS, -1, fm::window_compact(Lh, commit_lens, W, r0, rows, ws.row_src, ws.rows_dev, out_loc));
      TIMED(FLASHMAP_KIND_ROWS, -1, fm::gather_window_rows(Lh, target_hidden, static_cast<int64_t>(xrow), ws.row_src,
                                                           ws.rows_dev, rows, ws.xc));
      x = ws.xc;
      rows_dev = ws.rows_dev;
    }
    // ctx = RMSNorm_hidden(fc(x)); kv = W_ctx ctx
    TIMED_GEMM(-1, m->fc, rows, fm::linear(Lw, m->fc, x, rows, m->Lt * m->H, ws.acc_fc, m->D, nullptr, nullptr, fm::Out::Store,
                                           rows_dev));
    TIMED(FLASHMAP_KIND_ROWS, -1, fm::rms_rows(Lh, m->adt, ws.acc_fc, rows, m->D, m->hidden_norm_w, m->cfg.rms_norm_eps,
                                               1.f, nullptr, 0.f, ws.ctx, m->D, rows_dev));
    TIMED_GEMM(-1, m->ctx_kv, rows, fm::linear(Lw, m->ctx_kv, ws.ctx, rows, m->D, ws.acc_kv, 2 * m->L * m->D, nullptr,
                                               nullptr, fm::Out::Store, rows_dev));
    fm::KvWriteArgs a;
    a.acc = ws.acc_kv;
    a.ld = 2LL * m->L * m->D;
    a.rows = rows;
    a.W = W;
    a.row0 = r0;
    a.start_pos = start_pos;
    a.commit_lens = commit_lens;
    a.req_pool_idx = req_pool_idx;
    a.req_to_page = req_to_page;
    a.r2p_stride = req_to_page_stride;
    a.L = m->L;
    a.nh = m->nh;
    a.hd = m->hd;
    a.P = m->P;
    a.num_pages = pool->num_pages;
    a.k_norm = m->ctx_knorm;
    a.eps = m->cfg.qk_norm_eps;
    a.rope = m->rope;
    a.max_pos = m->maxpos;
    a.pool = pool->base;
    a.out_loc = out_loc;
    if (compact) {
      a.row_src = ws.row_src;
      a.rows_dev = rows_dev;
    }
    TIMED(FLASHMAP_KIND_ROWS, -1, fm::kv_write(Lh, m->kdt, a));
  }
  return FLASHMAP_OK;
}

// The draft of n_cand candidate blocks per request (1: flashmap_draft_block): the anchor
// rows once per request, then the noise (keyed by the candidate) and the DiT on
// bs * n_cand blocks, block bc being candidate bc % n_cand of request bc / n_cand.
static flashmap_status draft_impl(flashmap_model* m, const flashmap_kv_pool* pool, const flashmap_pending_write* pw,
                                  int32_t bs, int32_t n_cand,
                                  const int64_t* anchor_ids, const int32_t* anchor_pos, const int32_t* req_pool_idx,
                                  const int32_t* req_to_page, int32_t req_to_page_stride, const uint64_t* seeds,
                                  float noise_scale, void* hidden_out, int64_t* anchor_loc_out, void* workspace,
                                  size_t workspace_bytes, flashmap_stream stream) {
  g_last_error.clear();
  if (!m || !pool || !anchor_ids || !anchor_pos || !req_pool_idx || !req_to_page || !seeds || !hidden_out || !workspace)
    return fail(FLASHMAP_E_INVALID, "NULL argument");
  if (bs <= 0 || req_to_page_stride <= 0) return fail(FLASHMAP_E_INVALID, "bs and the page-table stride must be positive");
  if (n_cand < 1 || static_cast<int64_t>(bs) * n_cand * m->K > (1 << 24))
    return fail(FLASHMAP_E_INVALID, "n_cand must be >= 1 and bs * n_cand * block_size <= 2^24");
  if (n_cand > 1 && m->steps > 1)  // flashmap/sglang/model.py: several candidates take one jump
    return fail(FLASHMAP_E_UNSUPPORTED, "candidate drafts take one jump (num_steps = 1)");
  if (pool->dtype != m->kdt || !pool->base || pool->num_pages <= 0)
    return fail(FLASHMAP_E_INVALID, "pool dtype must equal kv_dtype, with pages");
  if (!std::isfinite(noise_scale)) return fail(FLASHMAP_E_INVALID, "noise_scale must be finite");
  int wrows = 0;  // rows of a deferred verify-window write
  if (pw) {
    if (!pw->target_hidden || !pw->start_pos || pw->W <= 0)
      return fail(FLASHMAP_E_INVALID, "the pending write needs target_hidden, start_pos and W > 0");
    if (m->adt == FLASHMAP_BF16 && (reinterpret_cast<uintptr_t>(pw->target_hidden) & 15))
      return fail(FLASHMAP_E_INVALID, "target_hidden must be 16-byte aligned");
    if (static_cast<int64_t>(bs) * pw->W > (1 << 24)) return fail(FLASHMAP_E_INVALID, "bs * W must be <= 2^24");
    wrows = bs * pw->W;
  }
  const int bsc = bs * n_cand;  // blocks
  const DraftWs need = carve_draft(m, bsc, nullptr, wrows);
  if (workspace_bytes < need.bytes)
    return fail(FLASHMAP_E_INVALID, "workspace too small: need " + std::to_string(need.bytes) + " bytes");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const DraftWs ws = carve_draft(m, bsc, workspace, wrows);
  const Launch Lh = [&] {
    Launch l = m->launch(s);
    l.red = ws.red_main;
    return l;
  }();
  const int R = bsc * m->K, D = m->D, H = m->H, adt = m->adt;
  {
    // counters only: every GEMM output is written whole (the residual stream starts as
    // x_embed's output, stored)
    fm::ZeroList z;
    z.add(reinterpret_cast<float*>(ws.xnext), 1);  // zero bits
    z.add(reinterpret_cast<float*>(ws.red_main.cnt), ws.red_main.cnt_cap);
    z.add(reinterpret_cast<float*>(ws.red_side.cnt), ws.red_side.cnt_cap);
    TIMED(FLASHMAP_KIND_MEMSET, -1, fm::zero_ranges(Lh, z));
  }
  // the blocks' request arrays (candidates of a request share its position and pages)
  const int32_t *pos_x = anchor_pos, *rpi_x = req_pool_idx;
  if (n_cand > 1) {
    TIMED(FLASHMAP_KIND_ROWS, -1, fm::expand_requests(Lh, anchor_pos, req_pool_idx, bs, n_cand, ws.exp_pos, ws.exp_rpi));
    pos_x = ws.exp_pos;
    rpi_x = ws.exp_rpi;
  }
  // split-KV plan of the cross-attention, shared by every layer
  TIMED(FLASHMAP_KIND_ROWS, -1, fm::xattn_plan(Lh, pos_x, bsc, m->nh, ws.plan, n_cand));
  // 1. anchor row: anchor_norm(anchor_proj(E[anchor])) -> every layer's context K/V at p.
  // Nothing before layer 0's cross-attention reads it, so it runs on the model's side
  // stream beside the noise embedding and layer 0's self-attention half: the two
  // branches fill each other's gaps between weight-streaming GEMMs. Their GEMMs take one
  // CTA per SM so that one of each branch fits on an SM at once. (Not while launches are
  // being timed one by one.)
  const bool fork = FM_DRAFT_FORK && !m->prof_on;
  const Launch La = [&] {
    Launch l = m->launch(fork ? m->side : s);
    if (fork) l.ctas_per_sm = FM_FORK_CTAS_PER_SM;
    l.red = ws.red_side;
    return l;
  }();
  Launch Lm = Lh;  // the main branch until the join
  if (fork) {
    Lm.ctas_per_sm = FM_FORK_CTAS_PER_SM;
    FM_CUDA(cudaEventRecord(m->ev_fork, s));
    FM_CUDA(cudaStreamWaitEvent(m->side, m->ev_fork, 0));
  }
  TIMED(FLASHMAP_KIND_ROWS, -1, fm::gather_rows(La, adt, m->embedding, m->V, H, anchor_ids, bs, ws.e_rows));
  TIMED_GEMM(-1, m->ap, bs, fm::linear(La, m->ap, ws.e_rows, bs, H, ws.acc_a, D, nullptr, m->ap_b, fm::Out::Store));
  TIMED(FLASHMAP_KIND_ROWS, -1, fm::rms_rows(La, adt, ws.acc_a, bs, D, m->anchor_norm_w, m->cfg.rms_norm_eps, 1.f, nullptr, 0.f, ws.kv_in, D));
  // A deferred verify-window write (flashmap/vllm/model.py, defer_context_kv /
  // _prologue): its rows hidden_norm(fc(target hidden)) follow the anchor rows, and one
  // all-layer context K/V GEMM projects both. A large window lists its committed
  // columns first (as flashmap_write_context_kv does); the GEMM then takes the anchors
  // plus their count from the device.
  int kv_rows = bs;
  const int* kv_rows_dev = nullptr;
  bool wcompact = false;
  if (wrows > 0) {
    const void* xw = pw->target_hidden;
    const int* wdev = nullptr;
    wcompact = pw->commit_lens && write_can_compact(m) && wrows >= FM_WRITE_COMPACT_MIN_ROWS;
    if (wcompact) {
      const size_t xrow = static_cast<size_t>(m->Lt) * H * dt_size(adt);
      TIMED(FLASHMAP_KIND_ROWS, -1, fm::window_compact(La, pw->commit_lens, pw->W, 0, wrows, ws.row_src, ws.wcnt,
                                                       pw->out_loc, ws.wtotal, bs));
      TIMED(FLASHMAP_KIND_ROWS, -1, fm::gather_window_rows(La, pw->target_hidden, static_cast<int64_t>(xrow),
                                                           ws.row_src, ws.wcnt, wrows, ws.xc));
      xw = ws.xc;
      wdev = ws.wcnt;
      kv_rows_dev = ws.wtotal;
    }
    TIMED_GEMM(-1, m->fc, wrows, fm::linear(La, m->fc, xw, wrows, m->Lt * H, ws.acc_fc, D, nullptr, nullptr,
                                             fm::Out::Store, wdev));
    TIMED(FLASHMAP_KIND_ROWS, -1, fm::rms_rows(La, adt, ws.acc_fc, wrows, D, m->hidden_norm_w, m->cfg.rms_norm_eps,
                                               1.f, nullptr, 0.f,
                                               static_cast<uint8_t*>(ws.kv_in) + static_cast<size_t>(bs) * D * dt_size(adt),
                                               D, wdev));
    kv_rows = bs + wrows;
  }
  TIMED_GEMM(-1, m->ctx_kv, kv_rows, fm::linear(La, m->ctx_kv, ws.kv_in, kv_rows, D, ws.acc_kv, 2 * m->L * D, nullptr,
                                                nullptr, fm::Out::Store, kv_rows_dev));
  if (wrows > 0) {
    fm::KvWriteArgs a;
    a.acc = ws.acc_kv + static_cast<size_t>(bs) * 2 * m->L * D;
    a.ld = 2LL * m->L * D;
    a.rows = wrows;
    a.W = pw->W;
    a.row0 = 0;
    a.start_pos = pw->start_pos;
    a.commit_lens = pw->commit_lens;
    a.req_pool_idx = req_pool_idx;
    a.req_to_page = req_to_page;
    a.r2p_stride = req_to_page_stride;
    a.L = m->L;
    a.nh = m->nh;
    a.hd = m->hd;
    a.P = m->P;
    a.num_pages = pool->num_pages;
    a.k_norm = m->ctx_knorm;
    a.eps = m->cfg.qk_norm_eps;
    a.rope = m->rope;
    a.max_pos = m->maxpos;
    a.pool = pool->base;
    a.out_loc = pw->out_loc;
    if (wcompact) {
      a.row_src = ws.row_src;
      a.rows_dev = ws.wcnt;
    }
    TIMED(FLASHMAP_KIND_ROWS, -1, fm::kv_write(La, m->kdt, a));
  }
  {
    fm::KvWriteArgs a;
    a.acc = ws.acc_kv;
    a.ld = 2LL * m->L * D;
    a.rows = bs;
    a.W = 1;
    a.row0 = 0;
    a.start_pos = anchor_pos;
    a.req_pool_idx = req_pool_idx;
    a.req_to_page = req_to_page;
    a.r2p_stride = req_to_page_stride;
    a.L = m->L;
    a.nh = m->nh;
    a.hd = m->hd;
    a.P = m->P;
    a.num_pages = pool->num_pages;
    a.k_norm = m->ctx_knorm;
    a.eps = m->cfg.qk_norm_eps;
    a.rope = m->rope;
    a.max_pos = m->maxpos;
    a.pool = pool->base;
    a.out_loc = anchor_loc_out;
    TIMED(FLASHMAP_KIND_ROWS, -1, fm::kv_write(La, m->kdt, a));
  }
  if (fork) FM_CUDA(cudaEventRecord(m->ev_join, m->side));
  bool joined = !fork;
  // 3. the DiT blocks (launches on Lc: the main branch's configuration until the join)
  Launch Lc = Lm;
  const float eps_ln = m->cfg.layer_norm_eps, eps_qk = m->cfg.qk_norm_eps;
  // the pool as rows of head_dim channels for the TMA-fed cross-attention (bf16)
  CUtensorMap kvmap;
  bool kvmap_ok = false;
  {
    const int64_t rows = 2LL * m->L * pool->num_pages * m->nh * m->P;
    std::string err;
    if (m->kdt == FLASHMAP_BF16 && (m->hd == 64 || m->hd == 128) && rows < (1LL << 31))
      kvmap_ok = fm::make_tmap_bf16(&kvmap, pool->base, rows, m->hd, m->hd, 16, &err);
  }
  fm::XattnArgs xa;
  xa.pool = pool->base;
  xa.num_pages = pool->num_pages;
  xa.bs = bsc;
  xa.n_cand = n_cand;
  xa.K = m->K;
  xa.nh = m->nh;
  xa.hd = m->hd;
  xa.P = m->P;
  xa.anchor_pos = pos_x;
  xa.req_pool_idx = rpi_x;
  xa.req_to_page = req_to_page;
  xa.r2p_stride = req_to_page_stride;
  xa.plan = ws.plan;
  xa.part_o = ws.part_o;
  xa.part_ml = ws.part_ml;
  xa.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(m->hd)));
  xa.qacc = ws.acc_d;
  xa.eps = eps_qk;
  xa.rope = m->rope;
  xa.max_pos = m->maxpos;
  // Forked: the anchor rows are joined before layer 0's cross-attention and everything
  // else its items kernels read before their dependency wait (plan, page table, pool)
  // was complete before the fork; each later items kernel starts after layer 0's did.
  // (The block self-attention reads the positions early on the same grounds: the
  // caller's anchor positions, or a multi-candidate draft's per-block copies once the
  // anchor branch has joined.)
  xa.early = FM_XATTN_EARLY && fork ? 1 : 0;
  // (one block: every item is the same length, and a fixed stride needs no counter)
  xa.next_item = FM_XATTN_DYNAMIC && bsc > 1 ? ws.xnext : nullptr;
  // The residual stream x: x_embed (or the folded noise) stores its start, the gated o,
  // cross-o and fc2 outputs are added to it once per element.
  auto resid_linear = [&](const Launch& Lx, int layer, const Weight& W, const void* in, int ldx, const float* alpha,
                          const float* beta, bool add) -> flashmap_status {
    TIMED_GEMM(layer, W, R, fm::linear(Lx, W, in, R, ldx, ws.x, D, alpha, beta, add ? fm::Out::Add : fm::Out::Store));
    return FLASHMAP_OK;
  };
  auto ln_mod = [&](const Launch& Lx, int layer, const float* scale, const float* shift, void* out) -> flashmap_status {
    TIMED(FLASHMAP_KIND_ROWS, layer, fm::ln_mod_rows(Lx, adt, ws.x, R, D, scale, shift, eps_ln, out));
    return FLASHMAP_OK;
  };
#define FM_TRY(call)                             \
  do {                                           \
    const flashmap_status st_ = (call);          \
    if (st_ != FLASHMAP_OK) return st_;          \
  } while (0)
  // the DiT blocks and the final AdaLN with one jump's modulations (null: the one jump's)
  auto dit = [&](const float* mods_all, const float* beta_all, const float* fin, void* out) -> flashmap_status {
    for (int l = 0; l < m->L; ++l) {
      const LayerW& lw = m->layers[l];
      const float* md = mods_all ? mods_all + static_cast<size_t>(l) * 9 * D : lw.mods;
      const float* fc2_beta = beta_all ? beta_all + static_cast<size_t>(l) * D : lw.fc2_beta;
      FM_TRY(ln_mod(Lc, l, md + 0 * D, md + 1 * D, ws.act));
      TIMED_GEMM(l, lw.qkv, R, fm::linear(Lc, lw.qkv, ws.act, R, D, ws.acc_big, 3 * D, nullptr, nullptr, fm::Out::Store));
      TIMED(FLASHMAP_KIND_SELF_ATTN, l, fm::self_attention(Lc, adt, ws.acc_big, bsc, m->K, m->nh, m->hd, lw.qn, lw.kn, eps_qk, m->rope, m->maxpos,
                                 pos_x, ws.act, xa.early != 0 && (n_cand == 1 || l > 0)));
      FM_TRY(resid_linear(Lc, l, lw.o, ws.act, D, md + 2 * D, nullptr, true));
      FM_TRY(ln_mod(Lc, l, md + 3 * D, md + 4 * D, ws.act));
      TIMED_GEMM(l, lw.cq, R, fm::linear(Lc, lw.cq, ws.act, R, D, ws.acc_d, D, nullptr, nullptr, fm::Out::Store));
      if (!joined) {  // the anchor rows are in the pool from here on
        FM_CUDA(cudaStreamWaitEvent(s, m->ev_join, 0));
        joined = true;
        Lc = Lh;
      }
      xa.layer = l;
      xa.q_norm = lw.cqn;
      TIMED(FLASHMAP_KIND_XATTN, l, fm::xattn_items(Lc, m->kdt, xa, kvmap_ok ? &kvmap : nullptr));
      TIMED(FLASHMAP_KIND_XCOMBINE, l, fm::xattn_combine(Lc, adt, xa, ws.act));
      FM_TRY(resid_linear(Lc, l, lw.co, ws.act, D, md + 5 * D, nullptr, true));
      FM_TRY(ln_mod(Lc, l, md + 6 * D, md + 7 * D, ws.act));
      // fc1 + bias + GELU in the GEMM's epilogue, written in the activation dtype
      TIMED_GEMM(l, lw.fc1, R, fm::linear(Lc, lw.fc1, ws.act, R, D, ws.act_f, m->F, nullptr, lw.fc1_b, fm::Out::GeluAct));
      FM_TRY(resid_linear(Lc, l, lw.fc2, ws.act_f, m->F, md + 8 * D, fc2_beta, true));
    }
    if (!joined) {
      FM_CUDA(cudaStreamWaitEvent(s, m->ev_join, 0));
      joined = true;
      Lc = Lh;
    }
    FM_TRY(ln_mod(Lc, -1, fin, fin + D, out));
    return FLASHMAP_OK;
  };
  if (m->steps == 1 && m->noise_path == 1) {
    // 2'. folded noise: z (Philox, as below) scaled by gate * rsqrt(sum(lam z^2) / H + eps),
    // then one GEMM through M onto x_embed(u)
    TIMED(FLASHMAP_KIND_ROWS, -1, fm::folded_noise(Lc, adt, seeds, anchor_pos, bs, m->K, H, n_cand, noise_scale,
                                                   m->fold_var, m->cfg.rms_norm_eps, m->gate, ws.act));
    FM_TRY(resid_linear(Lc, -1, m->fold, ws.act, H, nullptr, m->fold_xu, false));
    return dit(nullptr, nullptr, m->final_mods, hidden_out);
  }
  if (m->steps == 1) {
    // 2. noise: z (Philox, keyed by seed and slot position) -> z L^T -> u + gate * noise_norm -> x_embed
    TIMED(FLASHMAP_KIND_ROWS, -1, fm::draft_noise(Lc, adt, seeds, anchor_pos, bs, m->K, H, ws.act, n_cand));
    TIMED_GEMM(-1, m->chol, R, fm::linear(Lc, m->chol, ws.act, R, H, ws.acc_big, H, nullptr, nullptr, fm::Out::Store));
    TIMED(FLASHMAP_KIND_ROWS, -1, fm::rms_rows(Lc, adt, ws.acc_big, R, H, m->noise_norm_w, m->cfg.rms_norm_eps, noise_scale, m->u, m->gate,
                         ws.act, H));
    FM_TRY(resid_linear(Lc, -1, m->xe, ws.act, H, nullptr, m->xe_b, false));
    return dit(nullptr, nullptr, m->final_mods, hidden_out);
  }
  // several jumps: the state starts as V-wide noise keyed like the one-jump noise
  const int64_t V = m->V;
  const size_t es = dt_size(adt);
  uint8_t* xpost = static_cast<uint8_t*>(ws.xbuf);
  uint8_t* xstate = xpost + static_cast<size_t>(R) * V * es;
  TIMED(FLASHMAP_KIND_ROWS, -1, fm::draft_noise(Lc, FLASHMAP_F32, seeds, anchor_pos, bs, m->K, static_cast<int>(V),
                                                ws.state, 1, noise_scale));
  for (int st = 0; st < m->steps; ++st) {
    const float s0 = m->grid[st];
    const float ev = s0 > 0.f ? s0 / ((1.f - s0 > 1e-3f ? 1.f - s0 : 1e-3f) * (1.f - s0 > 1e-3f ? 1.f - s0 : 1e-3f))
                              : 0.f;
    // the previous jump's state update, then this jump's posterior and state in act dtype
    TIMED(FLASHMAP_KIND_ROWS, -1, fm::state_prep(Lc, adt, ws.state, ws.logits_full, m->full_head_b, R,
                                                 static_cast<int>(V), st > 0, st > 0 ? m->grid[st - 1] : 0.f, s0, ev,
                                                 xpost, xstate, V));
    // [posterior; state] @ E (at s = 0 only the state: the posterior is uniform)
    if (s0 > 0.f) {
      TIMED_GEMM(-1, m->et, 2 * R, fm::linear(Lc, m->et, xpost, 2 * R, static_cast<int>(V), ws.emb, H, nullptr,
                                              nullptr, fm::Out::Store));
    } else {
      TIMED_GEMM(-1, m->et, R, fm::linear(Lc, m->et, xstate, R, static_cast<int>(V), ws.emb + static_cast<size_t>(R) * H,
                                          H, nullptr, nullptr, fm::Out::Store));
    }
    TIMED(FLASHMAP_KIND_ROWS, -1, fm::mix_state(Lc, adt, s0 > 0.f ? ws.emb : nullptr, ws.emb + static_cast<size_t>(R) * H,
                                                R, H, m->u, m->state_norm_w, m->noise_norm_w, m->cfg.rms_norm_eps,
                                                m->step_gate[st], ws.act));
    // the residual stream (re)starts at x_embed of this jump's input
    FM_TRY(resid_linear(Lc, -1, m->xe, ws.act, H, nullptr, m->xe_b, false));
    const bool last = st + 1 == m->steps;
    const size_t L = static_cast<size_t>(m->L);
    const flashmap_status r = dit(m->step_mods + st * L * 9 * D, m->step_fc2_beta + st * L * D,
                                  m->step_final + static_cast<size_t>(st) * 2 * D, last ? hidden_out : ws.act);
    if (r != FLASHMAP_OK) return r;
    if (!last)  // the full-vocabulary logits that move the state
      TIMED_GEMM(-1, m->full_head, R, fm::linear(Lc, m->full_head, ws.act, R, D, ws.logits_full,
                                                 static_cast<int>(V), nullptr, nullptr, fm::Out::Store));
  }
  return FLASHMAP_OK;
}

flashmap_status flashmap_draft_block(flashmap_model* m, const flashmap_kv_pool* pool, int32_t bs,
                                     const int64_t* anchor_ids, const int32_t* anchor_pos,
                                     const int32_t* req_pool_idx, const int32_t* req_to_page,
                                     int32_t req_to_page_stride, const uint64_t* seeds, float noise_scale,
                                     void* hidden_out, int64_t* anchor_loc_out, void* workspace,
                                     size_t workspace_bytes, flashmap_stream stream) {
  return draft_impl(m, pool, nullptr, bs, 1, anchor_ids, anchor_pos, req_pool_idx, req_to_page, req_to_page_stride,
                    seeds, noise_scale, hidden_out, anchor_loc_out, workspace, workspace_bytes, stream);
}

flashmap_status flashmap_draft_block_with_write(flashmap_model* m, const flashmap_kv_pool* pool,
                                                const flashmap_pending_write* pending, int32_t bs,
                                                const int64_t* anchor_ids, const int32_t* anchor_pos,
                                                const int32_t* req_pool_idx, const int32_t* req_to_page,
                                                int32_t req_to_page_stride, const uint64_t* seeds, float noise_scale,
                                                void* hidden_out, int64_t* anchor_loc_out, void* workspace,
                                                size_t workspace_bytes, flashmap_stream stream) {
  if (!pending) {
    g_last_error.clear();
    return fail(FLASHMAP_E_INVALID, "NULL pending write");
  }
  return draft_impl(m, pool, pending, bs, 1, anchor_ids, anchor_pos, req_pool_idx, req_to_page, req_to_page_stride,
                    seeds, noise_scale, hidden_out, anchor_loc_out, workspace, workspace_bytes, stream);
}

flashmap_status flashmap_draft_candidates(flashmap_model* m, const flashmap_kv_pool* pool, int32_t bs,
                                          int32_t n_cand, const int64_t* anchor_ids, const int32_t* anchor_pos,
                                          const int32_t* req_pool_idx, const int32_t* req_to_page,
                                          int32_t req_to_page_stride, const uint64_t* seeds, float noise_scale,
                                          void* hidden_out, int64_t* anchor_loc_out, void* workspace,
                                          size_t workspace_bytes, flashmap_stream stream) {
  return draft_impl(m, pool, nullptr, bs, n_cand, anchor_ids, anchor_pos, req_pool_idx, req_to_page,
                    req_to_page_stride, seeds, noise_scale, hidden_out, anchor_loc_out, workspace, workspace_bytes,
                    stream);
}

flashmap_status flashmap_sample_block(flashmap_model* m, int32_t bs, const void* hidden, const int32_t* anchor_pos,
                                      const float* temperature, const uint8_t* greedy, const uint64_t* seeds,
                                      uint64_t step, int64_t* tokens_out, float* draft_logits_out,
                                      float* full_logits_out, void* workspace, size_t workspace_bytes,
                                      flashmap_stream stream) {
  g_last_error.clear();
  if (!m || !hidden || !anchor_pos || !temperature || !greedy || !seeds || !tokens_out)
    return fail(FLASHMAP_E_INVALID, "NULL argument");
  if (bs <= 0) return fail(FLASHMAP_E_INVALID, "bs must be positive");
  if (m->adt == FLASHMAP_BF16 && (reinterpret_cast<uintptr_t>(hidden) & 15))
    return fail(FLASHMAP_E_INVALID, "hidden must be 16-byte aligned");
  const SampleWs need = carve_sample(m, bs, draft_logits_out == nullptr, nullptr);
  if (!workspace || workspace_bytes < need.bytes)
    return fail(FLASHMAP_E_INVALID, "workspace too small: need " + std::to_string(need.bytes) + " bytes");
  const SampleWs ws = carve_sample(m, bs, draft_logits_out == nullptr, workspace);
  float* logits = draft_logits_out ? draft_logits_out : ws.logits;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Launch Lh = m->launch(s);
  Lh.red = ws.red;
  const int R = bs * m->K;
  {
    fm::ZeroList z;
    z.add(reinterpret_cast<float*>(ws.keys), 2LL * R);
    z.add(reinterpret_cast<float*>(ws.counters), R);
    z.add(reinterpret_cast<float*>(ws.red.cnt), ws.red.cnt_cap);
    TIMED(FLASHMAP_KIND_MEMSET, -1, fm::zero_ranges(Lh, z));
  }
  TIMED_GEMM(-1, m->head, R, fm::linear(Lh, m->head, hidden, R, m->D, logits, m->Vd, nullptr, m->head_b, fm::Out::Store));
  TIMED(FLASHMAP_KIND_SAMPLE, -1, fm::sample_rows(Lh, logits, R, m->Vd, m->K, temperature, greedy, seeds, anchor_pos,
                                                   static_cast<uint32_t>(step), m->hot, tokens_out, ws.keys,
                                                   ws.counters));
  if (full_logits_out)
    TIMED(FLASHMAP_KIND_SAMPLE, -1, fm::full_scatter(Lh, logits, R, m->Vd, m->inv_hot, m->V, full_logits_out));
  return FLASHMAP_OK;
}

flashmap_status flashmap_sample_logits_static(flashmap_model* m, int32_t bs, const float* logits,
                                             const int32_t* anchor_pos, const float* temperature,
                                             const uint8_t* greedy, const uint64_t* seeds, uint64_t step,
                                             int64_t* tokens_out, flashmap_stream stream) {
  g_last_error.clear();
  if (!m || !logits || !anchor_pos || !temperature || !greedy || !seeds || !tokens_out)
    return fail(FLASHMAP_E_INVALID, "NULL argument");
  if (bs <= 0) return fail(FLASHMAP_E_INVALID, "bs must be positive");
  const int64_t rows = static_cast<int64_t>(bs) * m->K;
  if (rows > fm::kStaticSampleRows)
    return fail(FLASHMAP_E_INVALID, "bs * block_size = " + std::to_string(rows) + " rows exceeds the " +
                                        std::to_string(fm::kStaticSampleRows) + " rows of the static sampler scratch");
  // The array's address is looked up for the current device: it must be the model's.
  int dev = -1;
  FM_CUDA(cudaGetDevice(&dev));
  if (dev != m->device)
    return fail(FLASHMAP_E_INVALID, "the current device (" + std::to_string(dev) + ") is not the model's device (" +
                                        std::to_string(m->device) + ")");
  void* scratch = nullptr;
  FM_CUDA(fm::static_sample_scratch(&scratch));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const Launch Lh = m->launch(s);
  auto* keys = static_cast<unsigned long long*>(scratch);
  auto* counters = reinterpret_cast<unsigned*>(static_cast<unsigned char*>(scratch) + rows * 8);
  fm::ZeroList z;  // the array keeps the last call's contents
  z.add(reinterpret_cast<float*>(keys), 2 * rows);
  z.add(reinterpret_cast<float*>(counters), rows);
  FM_CUDA(fm::zero_ranges(Lh, z));
  FM_CUDA(fm::sample_rows(Lh, logits, static_cast<int>(rows), m->Vd, m->K, temperature, greedy, seeds, anchor_pos,
                          static_cast<uint32_t>(step), m->hot, tokens_out, keys, counters));
  return FLASHMAP_OK;
}

flashmap_status flashmap_get_device_error(flashmap_model* m, flashmap_stream stream, uint32_t* code) {
  g_last_error.clear();
  if (!m || !code) return fail(FLASHMAP_E_INVALID, "NULL argument");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned v = 0;
  FM_CUDA(cudaStreamSynchronize(s));
  FM_CUDA(cudaMemcpy(&v, m->dev_err, 4, cudaMemcpyDeviceToHost));
  FM_CUDA(cudaMemset(m->dev_err, 0, 4));
  *code = v;
  if (v) return fail(FLASHMAP_E_DEVICE, "device error bits " + std::to_string(v));
  return FLASHMAP_OK;
}

flashmap_status flashmap_profile_start(flashmap_model* m, int32_t capacity) {
  g_last_error.clear();
  if (!m || capacity < 0) return fail(FLASHMAP_E_INVALID, "bad argument");
  m->prof_recs.clear();
  m->prof_cap = capacity;
  m->prof_on = true;
  return FLASHMAP_OK;
}

flashmap_status flashmap_profile_stop(flashmap_model* m, flashmap_launch_record* out, int32_t capacity,
                                      int32_t* count) {
  g_last_error.clear();
  if (!m || !count) return fail(FLASHMAP_E_INVALID, "bad argument");
  m->prof_on = false;
  const int n = static_cast<int>(m->prof_recs.size());
  for (int i = 0; i < n; ++i) {
    FM_CUDA(cudaEventSynchronize(m->prof_events[2 * i + 1]));
    float ms = 0.f;
    FM_CUDA(cudaEventElapsedTime(&ms, m->prof_events[2 * i], m->prof_events[2 * i + 1]));
    m->prof_recs[i].ms = ms;
  }
  if (out)
    for (int i = 0; i < std::min(n, static_cast<int>(capacity)); ++i) out[i] = m->prof_recs[i];
  *count = n;
  return FLASHMAP_OK;
}

flashmap_status flashmap_profile_gemm_chain(flashmap_model* m, int32_t bs, int32_t window, const void* hidden,
                                           void* workspace, size_t workspace_bytes, int64_t* bytes_out,
                                           int32_t* launches_out, flashmap_stream stream) {
  g_last_error.clear();
  if (!m || !hidden || !workspace || !bytes_out || !launches_out || bs <= 0 || window < 0)
    return fail(FLASHMAP_E_INVALID, "bad argument");
  if (reinterpret_cast<uintptr_t>(hidden) & 15) return fail(FLASHMAP_E_INVALID, "hidden must be 16-byte aligned");
  if (m->steps != 1 || m->wdt == FLASHMAP_F32)
    return fail(FLASHMAP_E_UNSUPPORTED, "the GEMM chain covers one-jump drafts with tcgen05 weights");
  const int64_t wrows = static_cast<int64_t>(bs) * window;
  if (wrows > (1 << 24)) return fail(FLASHMAP_E_INVALID, "bs * window must be <= 2^24");
  const DraftWs need = carve_draft(m, bs, nullptr, static_cast<int>(wrows));
  const SampleWs sneed = carve_sample(m, bs, true, nullptr);
  if (workspace_bytes < std::max(need.bytes, sneed.bytes))
    return fail(FLASHMAP_E_INVALID, "workspace too small for the chain");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int R = bs * m->K, D = m->D, H = m->H;
  const size_t es = dt_size(m->adt);
  int64_t bytes = 0;
  int32_t n = 0;
  // algorithmic bytes of one launch: weights once (e4m3: one byte and a float32 scale
  // per output channel), activations read, outputs written (float32, or act dtype)
  // the residual-stream linears: x_embed stores, the gated outputs add
  auto resid = [&](const Launch& L, const Weight& W, const void* in, int rows, int ldx, float* x, const float* alpha,
                   const float* beta, bool add) -> cudaError_t {
    return fm::linear(L, W, in, rows, ldx, x, D, alpha, beta, add ? fm::Out::Add : fm::Out::Store);
  };
  auto count = [&](const Weight& W, int rows, size_t out_es) {
    const size_t wb = W.dtype == FLASHMAP_E4M3 ? static_cast<size_t>(W.N) * W.K + static_cast<size_t>(W.N) * 4
                                                : static_cast<size_t>(W.N) * W.K * es;
    bytes += static_cast<int64_t>(wb + static_cast<size_t>(rows) * W.K * es + static_cast<size_t>(rows) * W.N * out_es);
    ++n;
  };
  {
    // the draft with the verify-window write deferred into it (as the step runs it): fc
    // over the window rows, the anchor projection, then one all-layer context K/V GEMM
    // over the anchors and the window rows
    const DraftWs ws = carve_draft(m, bs, workspace, static_cast<int>(wrows));
    // the anchor branch and the main branch up to layer 0's cross-attention run side by
    // side in a draft, one GEMM CTA per SM each; the rest with the kernel's own maximum
    Launch L = m->launch(s);
    L.red = ws.red_main;
    L.ctas_per_sm = FM_DRAFT_FORK ? FM_FORK_CTAS_PER_SM : 0;
    Launch La = L;
    La.red = ws.red_side;
    FM_CUDA(cudaMemsetAsync(ws.red_main.cnt, 0, static_cast<size_t>(ws.red_main.cnt_cap) * 4, s));
    FM_CUDA(cudaMemsetAsync(ws.red_side.cnt, 0, static_cast<size_t>(ws.red_side.cnt_cap) * 4, s));
    if (wrows > 0) {
      FM_CUDA(fm::linear(La, m->fc, ws.xc, static_cast<int>(wrows), m->Lt * H, ws.acc_fc, D, nullptr, nullptr,
                         fm::Out::Store));
      count(m->fc, static_cast<int>(wrows), 4);
    }
    FM_CUDA(fm::linear(La, m->ap, ws.e_rows, bs, H, ws.acc_a, D, nullptr, m->ap_b, fm::Out::Store));
    count(m->ap, bs, 4);
    FM_CUDA(fm::linear(La, m->ctx_kv, ws.kv_in, bs + static_cast<int>(wrows), D, ws.acc_kv, 2 * m->L * D, nullptr,
                       nullptr, fm::Out::Store));
    count(m->ctx_kv, bs + static_cast<int>(wrows), 4);
    if (m->noise_path == 1) {
      FM_CUDA(resid(L, m->fold, ws.act, R, H, ws.x, nullptr, m->fold_xu, false));
      count(m->fold, R, 4);
    } else {
      FM_CUDA(fm::linear(L, m->chol, ws.act, R, H, ws.acc_big, H, nullptr, nullptr, fm::Out::Store));
      count(m->chol, R, 4);
      FM_CUDA(resid(L, m->xe, ws.act, R, H, ws.x, nullptr, m->xe_b, false));
      count(m->xe, R, 4);
    }
    for (int l = 0; l < m->L; ++l) {
      const LayerW& lw = m->layers[l];
      FM_CUDA(fm::linear(L, lw.qkv, ws.act, R, D, ws.acc_big, 3 * D, nullptr, nullptr, fm::Out::Store));
      count(lw.qkv, R, 4);
      FM_CUDA(resid(L, lw.o, ws.act, R, D, ws.x, lw.mods + 2 * D, nullptr, true));
      count(lw.o, R, 4);
      FM_CUDA(fm::linear(L, lw.cq, ws.act, R, D, ws.acc_d, D, nullptr, nullptr, fm::Out::Store));
      count(lw.cq, R, 4);
      L.ctas_per_sm = 0;  // the branches have joined
      FM_CUDA(resid(L, lw.co, ws.act, R, D, ws.x, lw.mods + 5 * D, nullptr, true));
      count(lw.co, R, 4);
      FM_CUDA(fm::linear(L, lw.fc1, ws.act, R, D, ws.act_f, m->F, nullptr, lw.fc1_b, fm::Out::GeluAct));
      count(lw.fc1, R, es);
      FM_CUDA(resid(L, lw.fc2, ws.act_f, R, m->F, ws.x, lw.mods + 8 * D, lw.fc2_beta, true));
      count(lw.fc2, R, 4);
    }
  }
  {
    const SampleWs ws = carve_sample(m, bs, true, workspace);
    Launch L = m->launch(s);
    L.red = ws.red;
    FM_CUDA(cudaMemsetAsync(ws.red.cnt, 0, static_cast<size_t>(ws.red.cnt_cap) * 4, s));
    FM_CUDA(fm::linear(L, m->head, hidden, R, D, ws.logits, m->Vd, nullptr, m->head_b, fm::Out::Store));
    count(m->head, R, 4);
  }
  *bytes_out = bytes;
  *launches_out = n;
  return FLASHMAP_OK;
}

flashmap_status flashmap_build_tree(const int64_t* candidates, int32_t bs, int32_t n_cand, int32_t block_size,
                                    int32_t width, int64_t* tokens_out, int64_t* ids_out, int64_t* stats_out,
                                    flashmap_stream stream) {
  g_last_error.clear();
  if (!candidates || !tokens_out || !ids_out || !stats_out || bs <= 0)
    return fail(FLASHMAP_E_INVALID, "NULL argument or bs <= 0");
  if (n_cand < 1 || n_cand > fm::kTreeMaxCandidates || block_size < 1 ||
      static_cast<int64_t>(n_cand) * block_size > fm::kTreeMaxNodes || width < 2 || width > fm::kTreeMaxNodes + 1)
    return fail(FLASHMAP_E_INVALID, "need 1 <= n_cand <= 64, n_cand * block_size <= 1024, 2 <= width <= 1025");
  int dev = 0, sms = 0;
  FM_CUDA(cudaGetDevice(&dev));
  FM_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  Launch Lh{reinterpret_cast<cudaStream_t>(stream), sms, nullptr, true};
  FM_CUDA(fm::build_tree(Lh, candidates, bs, n_cand, block_size, width, tokens_out, ids_out, stats_out));
  return FLASHMAP_OK;
}

flashmap_status flashmap_debug_philox(const uint64_t* seeds, const uint32_t* ctr, int64_t n, uint32_t* out,
                                      float* normals, flashmap_stream stream) {
  g_last_error.clear();
  if (!seeds || !ctr || !out || n < 0) return fail(FLASHMAP_E_INVALID, "bad argument");
  FM_CUDA(fm::philox_export(reinterpret_cast<cudaStream_t>(stream), seeds, ctr, n, out, normals));
  return FLASHMAP_OK;
}

flashmap_status flashmap_debug_linear(int32_t dtype, const void* x, const void* w, int32_t rows, int32_t in_features,
                                      int32_t out_features, float* out, flashmap_stream stream) {
  g_last_error.clear();
  if (!x || !w || !out || rows <= 0 || in_features <= 0 || out_features <= 0 ||
      !(is_act(dtype) || dtype == FLASHMAP_E4M3))
    return fail(FLASHMAP_E_INVALID, "bad argument");
  if (dtype != FLASHMAP_F32 && in_features % (dtype == FLASHMAP_E4M3 ? 16 : 8))
    return fail(FLASHMAP_E_INVALID, "in_features must be a multiple of 8 (16 for E4M3)");
  int dev = 0, sms = 0;
  FM_CUDA(cudaGetDevice(&dev));
  FM_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  FM_CUDA(fm::gemm_prepare());
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Weight W;
  W.ptr = w;
  W.N = out_features;
  W.K = in_features;
  void* q = nullptr;
  if (dtype == FLASHMAP_E4M3) {  // w is bf16: quantize it as flashmap_load_weights does
    const size_t qbytes = align_up(static_cast<size_t>(out_features) * in_features);
    FM_CUDA(cudaMallocAsync(&q, qbytes + static_cast<size_t>(out_features) * 4, s));
    float* scale = reinterpret_cast<float*>(static_cast<uint8_t*>(q) + qbytes);
    FM_CUDA(fm::quantize_e4m3(s, w, FLASHMAP_BF16, out_features, in_features, q, scale));
    W.ptr = q;
    W.wscale = scale;
  }
  std::string err;
  if (check_weight_map(W, dtype, &err) != FLASHMAP_OK) {
    if (q) cudaFreeAsync(q, s);
    return fail(FLASHMAP_E_CUDA, err);
  }
  Launch Lh{s, sms, nullptr, true};
  // the GEMM's split-tile scratch (a test hook: it keeps one buffer per device, grown
  // when a call needs more, so that timing it measures the kernel, not allocation)
  static std::vector<std::pair<void*, size_t>> scratch(64, {nullptr, 0});
  const size_t red_bytes = fm::gemm_scratch_bytes(rows, sms);
  cudaError_t e = cudaSuccess;
  if (dev < 0 || dev >= 64) e = cudaErrorInvalidDevice;
  if (e == cudaSuccess && scratch[dev].second < red_bytes) {
    if (scratch[dev].first) cudaFree(scratch[dev].first);  // synchronizes: a test hook
    scratch[dev] = {nullptr, 0};
    e = cudaMalloc(&scratch[dev].first, red_bytes);
    if (e == cudaSuccess) {
      scratch[dev].second = red_bytes;
      e = cudaMemset(scratch[dev].first, 0, red_bytes);  // counters start at zero; launches leave them so
    }
  }
  if (e == cudaSuccess) {
    Lh.red = fm::gemm_scratch_carve(scratch[dev].first, rows, sms);
    e = fm::linear(Lh, W, x, rows, in_features, out, out_features, nullptr, nullptr, fm::Out::Add);
  }
  if (q) cudaFreeAsync(q, s);
  FM_CUDA(e);
  return FLASHMAP_OK;
}

flashmap_status flashmap_debug_wait_timeout(flashmap_model* m, uint64_t limit_ns, flashmap_stream stream) {
  g_last_error.clear();
  if (!m) return fail(FLASHMAP_E_INVALID, "NULL model");
  if (limit_ns == 0 || limit_ns > 100000000ull) return fail(FLASHMAP_E_INVALID, "limit_ns must be in (0, 100 ms]");
  FM_CUDA(fm::wait_timeout_probe(m->launch(reinterpret_cast<cudaStream_t>(stream)), limit_ns));
  return FLASHMAP_OK;
}

flashmap_status flashmap_debug_constants(const flashmap_model* m, float* chol, float* uniform, int64_t* hot_ids,
                                         flashmap_stream stream) {
  g_last_error.clear();
  if (!m) return fail(FLASHMAP_E_INVALID, "NULL model");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (chol) FM_CUDA(fm::to_f32(s, m->chol.ptr, m->adt, static_cast<int64_t>(m->H) * m->H, chol));
  if (uniform) FM_CUDA(cudaMemcpyAsync(uniform, m->u, static_cast<size_t>(m->H) * 4, cudaMemcpyDeviceToDevice, s));
  if (hot_ids) FM_CUDA(cudaMemcpyAsync(hot_ids, m->hot, static_cast<size_t>(m->Vd) * 8, cudaMemcpyDeviceToDevice, s));
  return FLASHMAP_OK;
}

flashmap_status flashmap_debug_folded(const flashmap_model* m, float* variance, float* embedded_uniform, void* proj,
                                      int32_t* sweeps, flashmap_stream stream) {
  g_last_error.clear();
  if (!m) return fail(FLASHMAP_E_INVALID, "NULL model");
  if (m->noise_path != 1) return fail(FLASHMAP_E_INVALID, "the model was loaded without the folded-noise path");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (variance) FM_CUDA(cudaMemcpyAsync(variance, m->fold_var, static_cast<size_t>(m->H) * 4, cudaMemcpyDeviceToDevice, s));
  if (embedded_uniform)
    FM_CUDA(cudaMemcpyAsync(embedded_uniform, m->fold_xu, static_cast<size_t>(m->D) * 4, cudaMemcpyDeviceToDevice, s));
  if (proj)
    FM_CUDA(cudaMemcpyAsync(proj, m->fold.ptr, static_cast<size_t>(m->D) * m->H * dt_size(m->adt),
                            cudaMemcpyDeviceToDevice, s));
  if (sweeps) *sweeps = m->eig_sweeps;
  return FLASHMAP_OK;
}

}  // extern "C"
