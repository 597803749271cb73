// Host-side interfaces shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "flashmap.h"

namespace fm {

// Scratch of the tcgen05 GEMM's fixed-order split-tile sums: four counters per CTA of
// a launch (one per epilogue warp, i.e. per 32 output channels of a tile) and two
// partial-tile slots per CTA (BN x 128 float32 each). The counters must be zero when a
// launch starts; every launch that completes leaves them zero. One scratch serves one
// stream: launches that may overlap on the GPU need their own.
struct GemmScratch {
  unsigned* cnt = nullptr;
  float* slots = nullptr;
  int64_t cnt_cap = 0, slot_cap = 0;  // capacities in counters and in floats
};

struct Launch {
  cudaStream_t stream;
  int num_sms;
  unsigned* dev_err;  // the model's device error word (may be null in debug calls)
  bool pdl = true;    // launch with programmatic stream serialization
  int ctas_per_sm = 0;  // tcgen05 GEMM CTAs per SM (0: the kernel's own maximum)
  GemmScratch red;      // the tcgen05 GEMM's split-tile scratch on this stream
};

// Launches `kernel` on L.stream, with programmatic stream serialization when L.pdl,
// in thread-block clusters of `cluster` CTAs along x when cluster > 1.
template <typename... KArgs, typename... Args>
cudaError_t launch_kc(const Launch& L, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, int cluster,
                      Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_k(const Launch& L, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     Args&&... args) {
  return launch_kc(L, kernel, grid, block, smem, 1, static_cast<Args&&>(args)...);
}

// Zeroes up to kZeroRanges float32 ranges in one launch (accumulators a call sums into).
struct ZeroList {
  static constexpr int kZeroRanges = 12;
  float* ptr[kZeroRanges];
  int64_t n[kZeroRanges];
  int count = 0;
  void add(float* p, int64_t len) {
    if (len > 0 && count < kZeroRanges) {
      ptr[count] = p;
      n[count] = len;
      ++count;
    }
  }
};
cudaError_t zero_ranges(const Launch& L, const ZeroList& z);
// One warp waiting limit_ns on an mbarrier nothing arrives on (sets the TIMEOUT bit).
cudaError_t wait_timeout_probe(const Launch& L, uint64_t limit_ns);

// A GEMM weight W (N out, K in), row-major in device memory.
struct Weight {
  const void* ptr = nullptr;
  int N = 0, K = 0;
  int dtype = FLASHMAP_F32;      // F32, BF16, or E4M3 (expanded to bf16 in shared memory by the GEMM)
  const float* wscale = nullptr; // per-output-channel scale of an E4M3 weight
  bool has_map = false;
  CUtensorMap map;  // BF16: box 64 x 128, 128B swizzle; E4M3: box 64 bytes x 128 rows, no swizzle
};

// Encodes the tensor map of a row-major bf16 matrix (rows x cols, leading dim ld
// elements) read in boxes of box_rows x 64 columns with 128-byte swizzle.
bool make_tmap_bf16(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld,
                    int box_rows, std::string* err);
// The same for a dense row-major e4m3 matrix (cols a multiple of 16), box 64 x 128.
bool make_tmap_e4m3(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, std::string* err);

// Sets the kernel attributes the tcgen05 GEMM needs on the current device (call once
// per device before launching; not during stream capture).
cudaError_t gemm_prepare();

// What a linear does with y[r][n] = alpha[n] * sum_k x[r * ldx + k] * W[n][k] + beta[n]:
//   Add:      float32 out[r * ldo + n] += y  (one addition per element: the residual stream)
//   Store:    float32 out[r * ldo + n]  = y
//   GeluAct:  out[r * ldo + n] = GELU_erf(y) in the activation dtype (bf16 for tcgen05
//             weights, float32 for float32 weights)
// Every element is finished by one thread with a fixed summation order, so results do
// not change from run to run.
enum class Out { Add = 0, Store = 1, GeluAct = 2 };

// Sizes (bytes) of the GEMM scratch for launches of at most max_rows activation rows,
// and its carving out of `base` (256-byte aligned; counters first).
size_t gemm_scratch_bytes(int max_rows, int num_sms);
GemmScratch gemm_scratch_carve(void* base, int max_rows, int num_sms);

// y = x W^T (+ alpha, beta) for r < rows, n < N, written as `mode` says. alpha / beta may
// be null (1 / 0). x has W.dtype (bf16 for E4M3 weights). rows_dev (tcgen05 weights
// only): the rows actually present, counted on the device, at most `rows` (the launch
// is sized for `rows`). tcgen05 launches need L.red large enough for `rows`.
cudaError_t linear(const Launch& L, const Weight& W, const void* x, int rows, int ldx, void* out, int ldo,
                   const float* alpha, const float* beta, Out mode, const int* rows_dev = nullptr);

// General strided SIMT GEMM for load-time work, float32 accumulation:
// C(m, n) = sum_k A(m, k) B(k, n), A(m, k) = a[arow(m) * sam + k * sak] with
// arow(m) = a_rows ? a_rows[m] : m, B(k, n) = b[k * sbk + n * sbn]; types by dtype codes.
// mode 0: c_f32[m * ldc + n] = acc;  mode 1: c (dtype c_dtype) = acc;  mode 2:
// c_f64[m * ldc + n] = the float64 sum, in k order, of float32 sums over 1024-long k
// chunks (deterministic).
cudaError_t simt_gemm(cudaStream_t s, int M, int N, int K, const void* a, int a_dtype, const int64_t* a_rows,
                      int64_t sam, int64_t sak, const void* b, int b_dtype, int64_t sbk, int64_t sbn, void* c,
                      int c_dtype, int64_t ldc, int mode);

}  // namespace fm

namespace fm {

// ------------------------------------------------------------------ rows.cu
struct KvWriteArgs {
  const float* acc = nullptr;  // [rows][ld] float32 projections: per layer [k (D) | v (D)]
  int64_t ld = 0;
  int rows = 0, W = 1;   // local row i is global row row0 + i = column % W of request / W
  int64_t row0 = 0;
  const int32_t* start_pos = nullptr;   // [bs] position of column 0
  const int32_t* commit_lens = nullptr; // [bs] or null (all columns)
  const int32_t* req_pool_idx = nullptr;
  const int32_t* req_to_page = nullptr;
  int r2p_stride = 0;
  int L = 0, nh = 0, hd = 0, P = 0;
  int64_t num_pages = 0;
  const float* k_norm = nullptr;  // [L][hd]
  float eps = 0.f;
  const float2* rope = nullptr;   // [max_pos][hd / 2] (cos, sin)
  int max_pos = 0;
  void* pool = nullptr;
  int64_t* out_loc = nullptr;
  // compacted rows (window_compact): local row i is global row row_src[i], for
  // i < *rows_dev (null: every local row, global row row0 + i)
  const int32_t* row_src = nullptr;
  const int* rows_dev = nullptr;
  unsigned* dev_err = nullptr;
};
cudaError_t kv_write(const Launch& L, int dtype, const KvWriteArgs& a);
// The committed columns of window rows [r0, r0 + rows) (global row g is column g % W of
// request g / W, committed when the column is below commit_lens[g / W]), in order:
// row_src[k] = the k-th one's global row, *rows_dev = their count; out_loc[g] = -1 for
// the others (out_loc may be null); *total_dev = total_base + the count when total_dev
// is given. One CTA.
cudaError_t window_compact(const Launch& L, const int32_t* commit_lens, int W, int64_t r0, int rows,
                           int32_t* row_src, int* rows_dev, int64_t* out_loc, int* total_dev = nullptr,
                           int total_base = 0);
// xc[k] = x[row_src[k]] for k < *rows_dev; rows of row_bytes bytes (a multiple of 16,
// 16-byte aligned). One CTA per row of the largest count.
cudaError_t gather_window_rows(const Launch& L, const void* x, int64_t row_bytes, const int32_t* row_src,
                               const int* rows_dev, int max_rows, void* xc);
cudaError_t ln_mod_rows(const Launch& L, int dtype, const float* x, int rows, int width, const float* ms,
                        const float* mh, float eps, void* out);
cudaError_t rms_rows(const Launch& L, int dtype, const float* acc, int rows, int width, const float* w, float eps,
                     float prescale, const float* add, float gate, void* out, int ldo,
                     const int* rows_dev = nullptr);  // rows_dev: only rows below *rows_dev
cudaError_t gather_rows(const Launch& L, int dtype, const void* table, int64_t nrows, int width, const int64_t* ids,
                        int n, void* out);
cudaError_t draft_noise(const Launch& L, int dtype, const uint64_t* seeds, const int32_t* anchor_pos, int bs, int K,
                        int H, void* out, int n_cand = 1, float scale = 1.f);
// z (keyed like draft_noise) scaled per row by gate * rsqrt(sum(variance z^2) + eps): the
// folded projection's input (rows.cu)
cudaError_t folded_noise(const Launch& L, int dtype, const uint64_t* seeds, const int32_t* anchor_pos, int bs, int K,
                         int H, int n_cand, float scale, const float* variance, float eps, float gate, void* out);
// several jumps (jumps.cu); jumps_prepare sets state_prep's shared-memory limit for a
// vocabulary of V entries (once per device, not during capture)
cudaError_t jumps_prepare(int V);
cudaError_t state_prep(const Launch& L, int dtype, float* state, float* logits, const float* bias, int rows,
                       int V, bool upd, float s, float t, float ev, void* x_post, void* x_state, int64_t ld);
cudaError_t mix_state(const Launch& L, int dtype, float* emb_post, float* emb_state, int rows, int H, const float* u,
                      const float* state_w, const float* noise_w, float eps, float gate, void* out);
cudaError_t transpose(cudaStream_t s, int dtype, const void* in, int64_t rows, int64_t cols, void* out);
cudaError_t expand_requests(const Launch& L, const int32_t* anchor_pos, const int32_t* req_pool_idx, int bs,
                            int n_cand, int32_t* pos_out, int32_t* rpi_out);
cudaError_t philox_export(cudaStream_t s, const uint64_t* seeds, const uint32_t* ctr, int64_t n, uint32_t* out,
                          float* normals);

// ------------------------------------------------------------------ attention.cu
struct XattnArgs {
  const float* qacc = nullptr;  // [bs * K][D] float32 query projections
  const float* q_norm = nullptr;  // [hd] the layer's cross-attention q_norm weight
  float eps = 0.f;
  const float2* rope = nullptr;   // [max_pos][hd / 2]
  int max_pos = 0;
  const void* pool = nullptr;
  int64_t num_pages = 0;
  int bs = 0, K = 0, nh = 0, hd = 0, P = 0, layer = 0;
  const int32_t* anchor_pos = nullptr;
  const int32_t* req_pool_idx = nullptr;
  const int32_t* req_to_page = nullptr;
  int r2p_stride = 0;
  const int* plan = nullptr;
  float* part_o = nullptr;   // [chunks * nh][16][hd]
  float* part_ml = nullptr;  // [chunks * nh][16][2]
  float scale_log2 = 0.f;    // hd^-1/2 * log2(e)
  int n_cand = 1;            // blocks per request: a tree draft's candidates share a context
  // 1: the pool, the plan and the page table were complete before the items kernel could
  // start (only the queries come from the kernel just before it), so its first K/V
  // blocks are requested before it waits for that kernel
  int early = 0;
  // zeroed counter of the items handed out beyond each CTA's first (both items
  // kernels); the combine that follows zeroes it again. Null: items by fixed stride.
  unsigned* next_item = nullptr;
  unsigned* dev_err = nullptr;
};
cudaError_t self_attention(const Launch& L, int dtype, const float* qkv, int bs, int K, int nh, int hd, const float* qn,
                           const float* kn, float eps, const float2* rope, int max_pos, const int32_t* anchor_pos,
                           void* out, bool early = false);
int xattn_max_chunks(int num_sms, int nh, int bs);
size_t xattn_plan_ints(int num_sms, int nh, int bs);
// n_cand: blocks per request (consecutive blocks of a request share its context)
cudaError_t xattn_plan(const Launch& L, const int32_t* anchor_pos, int bs, int nh, int* plan, int n_cand = 1);
// kvmap: the bf16 pool as rows of head_dim channels (box 64 x 16, 128B swizzle) for the
// TMA-fed kernel, or null for the cp.async one.
cudaError_t xattn_items(const Launch& L, int dtype, const XattnArgs& a, const CUtensorMap* kvmap = nullptr);
cudaError_t xattn_prepare();  // kernel attributes, once per device (not during capture)
cudaError_t xattn_combine(const Launch& L, int dtype, const XattnArgs& a, void* out);

// ------------------------------------------------------------------ sample.cu
// keys: [rows] uint64 + counters [rows] uint32, zero before the first call; the
// sampler leaves them zero again.
int sample_splits(int Vd, int rows, int num_sms);
// Sampler merge slots in a static device array (no allocation): rows <= kStaticSampleRows.
constexpr int kStaticSampleRows = 8192;
cudaError_t static_sample_scratch(void** out);
cudaError_t sample_rows(const Launch& L, const float* logits, int rows, int Vd, int K, const float* temps,
                        const uint8_t* greedy, const uint64_t* seeds, const int32_t* anchor_pos, uint32_t step,
                        const int64_t* hot, int64_t* tokens, unsigned long long* keys, unsigned* counters);
// The verify tree of N candidate blocks of K tokens per request (tree.cu).
constexpr int kTreeMaxCandidates = 64, kTreeMaxNodes = 1024;  // N, N * K
cudaError_t build_tree(const Launch& L, const int64_t* candidates, int bs, int N, int K, int width, int64_t* tokens,
                       int64_t* ids, int64_t* stats);
cudaError_t full_scatter(const Launch& L, const float* logits, int rows, int Vd, const int32_t* inv, int V,
                         float* full);

// ------------------------------------------------------------------ loadtime.cu
struct TimeCondArgs {
  const void *te_l1_w, *te_l1_b, *te_l2_w, *te_l2_b, *je_l1_w, *je_l1_b, *je_l2_w, *je_l2_b;
  int dtype, C, Te;
  double s, t, time_scale;
};
cudaError_t to_f32(cudaStream_t s, const void* src, int dtype, int64_t n, float* dst);
cudaError_t mul_vec(cudaStream_t s, const float* a, const float* b, float* out, int n);
cudaError_t time_cond(cudaStream_t s, const TimeCondArgs& a, double* cond);
cudaError_t adaln(cudaStream_t s, const void* w, const void* b, int dtype, int C, int D, const double* cond,
                  float* s1, float* sh, float* gate);
cudaError_t uniform_constant(cudaStream_t s, const void* E, int dtype, int64_t V, int H, const float* w, float eps,
                             double* colsum, float* u);
// The doubles uniform_constant's colsum scratch holds (per-row-block column sums).
int64_t colsum_doubles(int64_t V, int H);
cudaError_t cholesky_f64(cudaStream_t s, double* A, int n, unsigned* err);
// folded-noise eigenbasis (eigen.cu): from the Cholesky factor's storage X (row-major
// L, n x n float64; overwritten), the folded projection proj (D x n, dtype), lam / n
// and x_embed(u); scratch of folded_scratch_bytes(n). Synchronizes s.
size_t folded_scratch_bytes(int n);
// E^T E (H x H) with float64 products and sums (eigen.cu)
cudaError_t gram_f64(cudaStream_t s, const void* E, int dtype, int64_t V, int H, double* G);
cudaError_t folded_noise_constants(cudaStream_t s, double* X, int n, void* scratch, const float* noise_w,
                                   const void* xw, const void* xb, int dtype, int D, const float* u, void* proj,
                                   float* variance, float* xu, int* sweeps_out, std::string* err);
cudaError_t chol_store(cudaStream_t s, const double* A, int n, int dtype, void* out);
cudaError_t quantize_e4m3(cudaStream_t s, const void* w, int dtype, int rows, int cols, void* q, float* scale);

}  // namespace fm
