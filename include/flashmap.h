/*
 * flashmap.h -- C ABI of the GB300-native FlashMap one-jump block-draft step.
 *
 * FlashMap drafts the block_size tokens after each request's last verified token
 * (the anchor) with a flow map: a small DiT that jumps once from Gaussian noise at
 * time 0 to per-slot token distributions at time 1, conditioned on the target
 * model's hidden states through paged cross-attention (flashmap/modeling_flashmap.py,
 * module docstring; flashmap/sglang/model.py, module docstring).
 *
 * The step has four calls, in the order a serving loop makes them:
 *   flashmap_write_context_kv  committed target hidden states -> paged context K/V
 *   flashmap_draft_block       anchor row, noise embedding, the DiT -> final hidden
 *   flashmap_sample_block      folded head logits -> one token per slot
 * after a one-time flashmap_load_weights.
 *
 * Conventions for every call:
 *   - Pointers marked (device) are CUDA device pointers on the current device;
 *     (host) pointers are ordinary host memory. The caller owns every buffer it
 *     passes; the model owns only what flashmap_load_weights derives.
 *   - Calls other than load/free/get_device_error enqueue work on `stream` and
 *     return without synchronizing the host; they allocate nothing, so they may be
 *     captured in a CUDA graph (workspace and outputs are caller-owned).
 *   - Arguments are validated on the host before anything is launched: an invalid
 *     call returns FLASHMAP_E_INVALID (or E_UNSUPPORTED) and enqueues nothing;
 *     flashmap_last_error() then describes the problem.
 *   - Values only the device can check (page ids, positions, token ids read from
 *     device arrays) are checked by the kernels: an out-of-range value skips the
 *     access it guards and sets the model's device error word, read back with
 *     flashmap_get_device_error(). No kernel traps or spins without a time limit.
 *   - Matrices are row-major. "rows" of the draft are request-major:
 *     row b * block_size + k is slot k of request b.
 *   - flashmap_draft_block and flashmap_draft_candidates run part of their work on a
 *     stream the model owns, forked from `stream` by an event and joined back before
 *     the call returns; work enqueued on `stream` after the call still sees all of it.
 *     Drafts of one model must therefore be enqueued from one host thread at a time.
 */
#ifndef FLASHMAP_H_
#define FLASHMAP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* flashmap_stream; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  FLASHMAP_OK = 0,
  FLASHMAP_E_INVALID = 1,     /* bad argument, shape or configuration */
  FLASHMAP_E_UNSUPPORTED = 2, /* valid for FlashMap, not built here (e.g. more jumps) */
  FLASHMAP_E_CUDA = 3,        /* a CUDA runtime call failed */
  FLASHMAP_E_NOMEM = 4,       /* device allocation failed (load only) */
  FLASHMAP_E_DEVICE = 5       /* a kernel reported an out-of-range value or a timeout */
} flashmap_status;

typedef enum { FLASHMAP_F32 = 0, FLASHMAP_BF16 = 1, FLASHMAP_E4M3 = 2 } flashmap_dtype;

/* Device error word bits (flashmap_get_device_error). */
#define FLASHMAP_DEVERR_PAGE 1u      /* a page id outside [0, num_pages) */
#define FLASHMAP_DEVERR_POSITION 2u  /* a position outside [0, max_position) */
#define FLASHMAP_DEVERR_TOKEN 4u     /* an anchor token id outside [0, vocab_size) */
#define FLASHMAP_DEVERR_TIMEOUT 8u   /* a pipeline wait gave up (kernel returned early) */
#define FLASHMAP_DEVERR_NUMERIC 16u  /* a non-positive pivot in the load-time Cholesky */

/*
 * FlashMapConfig (flashmap/configuration_flashmap.py, FlashMapConfig) restricted to
 * the one-jump draft, plus the draft pool's paging and the compute dtypes.
 *   target_hidden        H, the target model's hidden size
 *   num_target_layers    Lt, target layers whose outputs are concatenated (fc input Lt*H)
 *   hidden               D = num_heads * head_dim, the DiT width
 *   num_layers           L, DiT blocks
 *   intermediate         F, MLP width
 *   cond_dim, time_embed_dim, time_scale   time conditioning (FlashMapTimeEmbedding)
 *   block_size           K, draft slots per request
 *   vocab_size           V; draft_vocab_size Vd (0 or >= V: the full vocabulary)
 *   num_steps            jumps per draft, 1..4, on the printed grids
 *                        (flashmap/configuration_flashmap.py, DEFAULT_JUMP_GRIDS). One
 *                        jump reads its noise as z L^T (z ~ N(0, I_H)); several jumps
 *                        keep a vocabulary-sized float32 state per drafted row
 *                        (flashmap/modeling_flashmap.py, draft / embed_state / mix_state):
 *                        the load then also keeps E^T and the full-vocabulary folded
 *                        head, and the workspace the state, its posterior and logits.
 *   noise_gate_constant  0: gate noise_gate*(t-s) ("jump"); 1: noise_gate ("constant")
 *   page_size            P, positions per pool page (a multiple of 16)
 *   max_position         positions are < max_position (sizes the RoPE table)
 *   rope_theta, rms_norm_eps, qk_norm_eps, layer_norm_eps   as in FlashMapConfig
 *   act_dtype            F32 or BF16: activations, raw weights and the KV pool
 *   weight_dtype         act_dtype, or E4M3 (bf16 activations only): at load, every
 *                        large GEMM weight (fc, anchor_proj, x_embed, the all-layer
 *                        context K/V, each block's q/k/v, o, cross q and o, fc1, fc2,
 *                        and the folded head after folding) is quantized to e4m3fn
 *                        with one float32 scale per output channel, scale = max|w|/448
 *                        (1 for an all-zero row), q = w / scale rounded to nearest
 *                        even and saturated (flashmap/sglang/model.py, _quantize_fp8).
 *                        The noise factor L stays bf16. Activations stay bf16 and
 *                        accumulation float32 (W8A16): the GEMM expands each e4m3 tile
 *                        to bf16 on chip and applies the scale to its output. Needs
 *                        target_hidden, hidden and intermediate multiples of 16.
 *   kv_dtype             the draft KV pool's element type: act_dtype, or E4M3 (bf16
 *                        activations only): keys (after k-norm and RoPE) and values
 *                        are stored as e4m3fn with scale 1, rounded to nearest even
 *                        and saturated at +-448, and the cross-attention quantizes each
 *                        request's queries per head to e4m3 with scale
 *                        max(max|q|, 1e-12) / 448 over the block's slots and channels,
 *                        descaling the scores by it (flashmap/sglang/model.py,
 *                        _paged_cross_attention_fp8). Halves the pool's bytes.
 *   noise_path           how one jump reads its noise: 0, as z L^T then noise_norm and
 *                        x_embed; 1, the folded eigenbasis (flashmap/sglang/model.py,
 *                        noise_basis / _folded_noise): at load E^T E = Q diag(lam) Q^T
 *                        (float64 one-sided Jacobi; lam ascending, each eigenvector's
 *                        entry of largest magnitude positive), M = diag(sqrt lam) Q^T
 *                        diag(noise_norm w) W_x^T kept in act_dtype, lam / H and
 *                        x_embed(u); per step x = x_embed(u) + gate * r * (z @ M),
 *                        r = rsqrt(sum(lam z^2) / H + eps): one GEMM instead of two and
 *                        a row norm. Same z as path 0, the same law of x, other samples.
 *                        One jump only (num_steps = 1).
 */
typedef struct {
  int32_t target_hidden, num_target_layers, hidden, num_layers, num_heads, head_dim;
  int32_t intermediate, cond_dim, time_embed_dim, block_size, vocab_size, draft_vocab_size;
  int32_t num_steps, noise_gate_constant, page_size, max_position;
  float time_scale, rope_theta, rms_norm_eps, qk_norm_eps, layer_norm_eps;
  int32_t act_dtype, weight_dtype, kv_dtype;
  int32_t noise_path;
} flashmap_config;

/* One DiT block's raw weights (flashmap/modeling_flashmap.py, FlashMapLayer), all
 * (device) in act_dtype, shapes (out, in): adaln w (3D, cond_dim), b (3D); q/k/v/o
 * (D, D); q_norm/k_norm (head_dim); fc1 (F, D) + (F); fc2 (D, F) + (D). */
typedef struct {
  const void *self_adaln_w, *self_adaln_b;
  const void *self_q_w, *self_k_w, *self_v_w, *self_o_w, *self_q_norm_w, *self_k_norm_w;
  const void *cross_adaln_w, *cross_adaln_b;
  const void *cross_q_w, *cross_k_w, *cross_v_w, *cross_o_w, *cross_q_norm_w, *cross_k_norm_w;
  const void *mlp_adaln_w, *mlp_adaln_b;
  const void *fc1_w, *fc1_b, *fc2_w, *fc2_b;
} flashmap_layer_weights;

/* The drafter's raw weights (flashmap/modeling_flashmap.py, FlashMapDraftModel),
 * all (device) in act_dtype: fc (D, Lt*H); hidden_norm (D); anchor_proj (D, H) + (D);
 * anchor_norm (D); state_norm, noise_norm (H); noise_gate (1); x_embed (D, H) + (D);
 * time_embed / jump_embed linear_1 (C, Te) + (C), linear_2 (C, C) + (C);
 * final_adaln (3D, C) + (3D); head (H, D) + (H). `layers` is a (host) array of
 * num_layers entries. They are read during flashmap_load_weights only. */
typedef struct {
  const void *fc_w, *hidden_norm_w, *anchor_proj_w, *anchor_proj_b, *anchor_norm_w;
  const void *state_norm_w, *noise_norm_w, *noise_gate, *x_embed_w, *x_embed_b;
  const void *time_l1_w, *time_l1_b, *time_l2_w, *time_l2_b;
  const void *jump_l1_w, *jump_l1_b, *jump_l2_w, *jump_l2_b;
  const void *final_adaln_w, *final_adaln_b, *head_w, *head_b;
  const flashmap_layer_weights* layers;
} flashmap_weights;

/*
 * The paged draft KV pool (flashmap/sglang/model.py, _fused_write_args: per layer
 * keys and values; tokenspeed dflash.py: req_to_page / page_size addressing).
 * Layout (device, kv_dtype): [num_layers][2 (key, value)][num_pages][num_heads]
 * [page_size][head_dim]; the slot of position pos of the request in page-table row
 * r is req_to_page[r][pos / P] * P + pos % P. An E4M3 pool stores each (page, head)
 * block of VALUES channel-major instead, [head_dim][page_size] (keys as above), and
 * within every 16 positions of a channel row position 2t + e at byte 4t + e and
 * position 8 + 2t + e at byte 4t + 2 + e (t < 4, e < 2): the order in which the
 * cross-attention's value product takes them, so that it reads the block without a
 * transpose. The size is the same either way. Caller-owned; size it with
 * flashmap_pool_bytes.
 */
typedef struct {
  void* base;
  int64_t num_pages;
  int32_t dtype; /* must equal kv_dtype */
} flashmap_kv_pool;

typedef struct flashmap_model flashmap_model;

/* Bytes of a pool of num_pages pages for cfg (host-only; no GPU needed). */
flashmap_status flashmap_pool_bytes(const flashmap_config* cfg, int64_t num_pages, size_t* bytes);

/* Checks cfg as flashmap_load_weights does (host-only; no GPU needed). */
flashmap_status flashmap_validate_config(const flashmap_config* cfg);

/*
 * Loads a drafter and precomputes everything a one-jump draft reads that depends
 * only on weights (flashmap/sglang/model.py, load_weights / prepare /
 * _jump_constants / _fold_lm_head; flashmap/vllm/model.py, prepare):
 *   - the all-layer context K/V weight [k_0; v_0; ...; k_{L-1}; v_{L-1}] (2LD, D) and
 *     each block's fused q/k/v weight (3D, D);
 *   - every AdaLN modulation of the jump 0 -> 1 as (1 + scale, shift, gate);
 *   - the uniform posterior's embedding state_norm(mean row of E) and the Cholesky
 *     factor L of E^T E (gram accumulated on the GPU, factored in float64);
 *   - the draft vocabulary hot = sort(vocab_ranking[:Vd]) and the folded head
 *     W_f = LM[hot] W_head (Vd, D), b_f = LM[hot] b_head, folded in float32;
 *   - the float32 RoPE table (cos, sin) for positions < max_position.
 * embedding (device, (V, H) act_dtype) is BORROWED: the draft reads anchor rows from
 * it, so it must outlive the model. lm_head (device, (V, H)) is read here only.
 * vocab_ranking (device int64 (V), most frequent first) may be NULL: full vocabulary.
 * Synchronizes `stream`. Returns E_NOMEM if device memory runs out, E_DEVICE if the
 * gram is not positive definite.
 */
flashmap_status flashmap_load_weights(const flashmap_config* cfg, const flashmap_weights* weights,
                                      const void* embedding, const void* lm_head,
                                      const int64_t* vocab_ranking, flashmap_stream stream,
                                      flashmap_model** out);

flashmap_status flashmap_free(flashmap_model* model);

/* The model's config (host copy). */
flashmap_status flashmap_get_config(const flashmap_model* model, flashmap_config* cfg);

/* Workspace bytes needed by write/draft/sample for batches of up to max_bs requests
 * and writes of up to max_write_rows (bs * window) rows at once, including a draft
 * with a deferred write of up to max_write_rows rows (flashmap_draft_block_with_write,
 * which does not split its write into chunks). */
flashmap_status flashmap_workspace_size(const flashmap_model* model, int32_t max_bs,
                                        int32_t max_write_rows, size_t* bytes);

/*
 * Context-KV write (flashmap/sglang/model.py, write_target_hidden_kv / _write_context;
 * flashmap/modeling_flashmap.py, extend_context): for request b and window column
 * c < W at position start_pos[b] + c, if c < commit_lens[b] (every column when
 * commit_lens is NULL):
 *   ctx = RMSNorm_hidden(fc(target_hidden[b, c]))           (eps rms_norm_eps)
 *   per layer l, head h: key = RoPE_pos(RMSNorm_{k_norm_l}(k_l ctx)) (eps qk_norm_eps),
 *   value = v_l ctx; both stored at slot(req_pool_idx[b], pos).
 * Uncommitted columns are neither written nor waited for (no host sync).
 *   target_hidden  (device) [bs][W][Lt*H] act_dtype
 *   req_pool_idx   (device) int32 [bs], page-table row of each request
 *   start_pos      (device) int32 [bs], position of window column 0
 *   commit_lens    (device) int32 [bs] in [0, W], or NULL
 *   req_to_page    (device) int32 [rows][req_to_page_stride]
 *   out_loc        (device) int64 [bs][W]: the slot written, -1 if skipped; or NULL
 * Rows are processed in chunks of max_write_rows (flashmap_workspace_size). A chunk of
 * 48 or more rows with commit_lens (bf16 or e4m3 GEMM weights) projects only its
 * committed columns, listed and counted on the device; the results are the same.
 */
flashmap_status flashmap_write_context_kv(flashmap_model* model, const flashmap_kv_pool* pool,
                                          const void* target_hidden, int32_t bs, int32_t W,
                                          const int32_t* req_pool_idx, const int32_t* start_pos,
                                          const int32_t* commit_lens, const int32_t* req_to_page,
                                          int32_t req_to_page_stride, int64_t* out_loc,
                                          void* workspace, size_t workspace_bytes,
                                          flashmap_stream stream);

/*
 * One jump from t = 0 for bs requests (flashmap/sglang/model.py, forward / _draft_impl
 * / _denoise; flashmap/modeling_flashmap.py, draft / FlashMapLayer):
 *   1. the anchor row anchor_norm(anchor_proj(E[anchor_ids[b]])) is projected by every
 *      layer's context key/value weights, k-normed, rotated at anchor_pos[b] and
 *      written at slot(req_pool_idx[b], anchor_pos[b]) (later overwritten by the
 *      verified hidden state);
 *   2. slot k of request b sits at position p = anchor_pos[b] + 1 + k; its noise
 *      z ~ N(0, I_H) is Philox4x32-10 keyed by (seeds[b], p); the embedded state is
 *      u + gate * RMSNorm_noise(noise_scale * z L^T), then x_embed;
 *   3. every DiT block: modulated LayerNorm -> self-attention across the request's
 *      K slots (q/k RMSNorm, RoPE) -> gated residual; modulated LayerNorm -> paged
 *      cross-attention onto pool positions 0..anchor_pos[b] -> gated residual;
 *      modulated LayerNorm -> fc1, GELU, fc2 -> gated residual;
 *   4. the final modulated LayerNorm -> hidden_out.
 *   anchor_ids  (device) int64 [bs]; anchor_pos (device) int32 [bs]
 *   seeds       (device) uint64 [bs]; noise_scale 1 (0: a deterministic draft)
 *   hidden_out  (device) [bs * K][D] act_dtype
 *   anchor_loc_out (device) int64 [bs] slot of the anchor row, or NULL
 */
flashmap_status flashmap_draft_block(flashmap_model* model, const flashmap_kv_pool* pool, int32_t bs,
                                     const int64_t* anchor_ids, const int32_t* anchor_pos,
                                     const int32_t* req_pool_idx, const int32_t* req_to_page,
                                     int32_t req_to_page_stride, const uint64_t* seeds,
                                     float noise_scale, void* hidden_out, int64_t* anchor_loc_out,
                                     void* workspace, size_t workspace_bytes, flashmap_stream stream);

/* A verify-window context-KV write handed to the next draft instead of run on its
 * own (flashmap/vllm/model.py, defer_context_kv): the fields of
 * flashmap_write_context_kv for bs requests (the draft's bs, req_pool_idx and page
 * table). */
typedef struct {
  const void* target_hidden;   /* (device) [bs][W][Lt*H] act_dtype, 16-byte aligned */
  int32_t W;                   /* window columns per request */
  const int32_t* start_pos;    /* (device) int32 [bs], position of window column 0 */
  const int32_t* commit_lens;  /* (device) int32 [bs] in [0, W], or NULL (every column) */
  int64_t* out_loc;            /* (device) int64 [bs][W]: the slot written, -1 if skipped; or NULL */
} flashmap_pending_write;

/*
 * flashmap_draft_block with a pending verify-window write done in the same call
 * (flashmap/vllm/model.py, defer_context_kv and _prologue: the pending context rows
 * and the anchors go through one GEMM over the all-layer context K/V weight). The
 * window's committed columns are written exactly as flashmap_write_context_kv writes
 * them (same slots, keys and values, out_loc) and the anchors as flashmap_draft_block
 * writes them; the all-layer context K/V weight is read once for both instead of once
 * per call. The write completes before any cross-attention reads the pool. The
 * workspace must hold the draft and the bs * W write rows at once
 * (flashmap_workspace_size with max_write_rows >= bs * W); the write is not chunked.
 */
flashmap_status flashmap_draft_block_with_write(flashmap_model* model, const flashmap_kv_pool* pool,
                                                const flashmap_pending_write* pending, int32_t bs,
                                                const int64_t* anchor_ids, const int32_t* anchor_pos,
                                                const int32_t* req_pool_idx, const int32_t* req_to_page,
                                                int32_t req_to_page_stride, const uint64_t* seeds,
                                                float noise_scale, void* hidden_out, int64_t* anchor_loc_out,
                                                void* workspace, size_t workspace_bytes, flashmap_stream stream);

/*
 * Whole-block sampling (flashmap/sglang/sampler.py, FlashMapDraftSampler, fused
 * variant; flashmap/sglang/model.py, head_logits): logits l = W_f hidden + b_f over
 * the draft vocabulary, then for row r = b * K + k at position p = anchor_pos[b]+1+k:
 * greedy[b] != 0 or temperature[b] <= 0 -> j = argmax_j l_j; otherwise
 * j = argmax_j (l_j / temperature[b] + G_j), G_j = -ln(-ln U_j), U_j from Philox4x32-10
 * keyed by seeds[b] with counter (j / 4, p, 1, step), word j mod 4; ties go to the
 * lowest j. tokens_out[r] = hot[j].
 *   hidden       (device) [bs * K][D] act_dtype (flashmap_draft_block's output)
 *   temperature  (device) float32 [bs]; greedy (device) uint8 [bs]; seeds (device) uint64 [bs]
 *   step         caller counter, advanced per call so rounds draw fresh noise
 *   tokens_out   (device) int64 [bs * K]
 *   draft_logits_out (device) float32 [bs * K][Vd], or NULL
 *   full_logits_out  (device) float32 [bs * K][V]: the draft logits at their token ids,
 *                    -inf elsewhere (flashmap/sglang/sampler.py, _FullLogits), or NULL
 *   workspace    (device) per-row merge slots of the split sampler, plus the logits
 *                when draft_logits_out is NULL (flashmap_workspace_size covers both)
 */
flashmap_status flashmap_sample_block(flashmap_model* model, int32_t bs, const void* hidden,
                                      const int32_t* anchor_pos, const float* temperature,
                                      const uint8_t* greedy, const uint64_t* seeds, uint64_t step,
                                      int64_t* tokens_out, float* draft_logits_out,
                                      float* full_logits_out, void* workspace,
                                      size_t workspace_bytes, flashmap_stream stream);

/*
 * flashmap_sample_block's sampling step for callers that cannot allocate device
 * memory: for example a host runtime that owns every device allocation and hands a
 * plugin only its input and output buffers, or code running where a device
 * allocation would not be allowed. The paper has no counterpart; this is a
 * library-level addition. The caller passes the draft-vocabulary logits (device,
 * float32 [bs * K][Vd], e.g. flashmap_sample_block's draft_logits_out) and the same
 * per-request inputs as flashmap_sample_block; tokens_out (device, int64 [bs * K])
 * receives the same token ids flashmap_sample_block draws from those logits. The
 * per-row merge slots live in a fixed array inside the library (96 KB on every GPU
 * that loads it, kept until the process exits), so bs * block_size may not exceed
 * 8192 rows (E_INVALID otherwise). The model's device must be the current device
 * (E_INVALID otherwise: the array's address is per device). The first call on a
 * device looks up that array's
 * device address; make it before any stream capture on that device. The array is
 * shared by every call and keeps the last call's contents (the call clears what it
 * uses): calls that overlap on the GPU, on any stream, race and give wrong tokens.
 */
flashmap_status flashmap_sample_logits_static(flashmap_model* model, int32_t bs, const float* logits,
                                             const int32_t* anchor_pos, const float* temperature,
                                             const uint8_t* greedy, const uint64_t* seeds, uint64_t step,
                                             int64_t* tokens_out, flashmap_stream stream);

/*
 * flashmap_draft_block for n_cand candidate blocks per request, drafted from
 * independent noise (tree drafting: flashmap/sglang/model.py, _draft_impl with
 * n_cand > 1). The anchor rows are computed and written once per request; block bc =
 * b * n_cand + c (candidate c of request b) has the request's positions and context,
 * and its noise takes Philox counter word 3 = c, so candidate 0 is the block
 * flashmap_draft_block drafts. The candidates of a request share its context: when
 * n_cand is a multiple of 2 or 4, the cross-attention serves 2 or 4 of them from one
 * read of each K/V block (bf16 and e4m3 pools); otherwise each reads it.
 *   hidden_out  (device) [bs * n_cand * K][D] act_dtype, candidate-major per request
 * Size the workspace with flashmap_workspace_size(max_bs = bs * n_cand). The blocks'
 * tokens come from flashmap_sample_block over bs * n_cand blocks (with each request's
 * position, seed and temperature repeated n_cand times); flashmap_build_tree merges
 * them into the verify tree.
 */
flashmap_status flashmap_draft_candidates(flashmap_model* model, const flashmap_kv_pool* pool, int32_t bs,
                                          int32_t n_cand, const int64_t* anchor_ids, const int32_t* anchor_pos,
                                          const int32_t* req_pool_idx, const int32_t* req_to_page,
                                          int32_t req_to_page_stride, const uint64_t* seeds, float noise_scale,
                                          void* hidden_out, int64_t* anchor_loc_out, void* workspace,
                                          size_t workspace_bytes, flashmap_stream stream);

/*
 * The verify tree of a multi-candidate draft (flashmap/sglang/tree.py, build_tree_abi;
 * flashmap/sglang/model.py, _draft_tree). For each request, n_cand candidate blocks
 * of block_size tokens drafted after its anchor (the tree's root) form a trie with a
 * node per distinct prefix; a node's vote is the number of candidates through it. The
 * width - 1 nodes with the most votes (ties: shallower, then lower candidate) are
 * kept -- every kept node's parent is kept too -- and listed by depth, then by the
 * lowest candidate through them, numbered 1.. (the root is 0). A trie with fewer nodes
 * is padded with copies of the first listed node (a child of the root).
 *   candidates  (device) int64 [bs][n_cand][block_size] token ids
 *   tokens_out  (device) int64 [bs][width - 1] the nodes' tokens
 *   ids_out     (device) int64 [bs][width - 1] parent * width + number
 *   stats_out   (device) int64 [bs][2] (trie nodes before the cut, distinct candidates)
 * Limits: 1 <= n_cand <= 64, n_cand * block_size <= 1024, 2 <= width <= 1025.
 * Allocates nothing; enqueued on `stream`.
 */
flashmap_status flashmap_build_tree(const int64_t* candidates, int32_t bs, int32_t n_cand, int32_t block_size,
                                    int32_t width, int64_t* tokens_out, int64_t* ids_out, int64_t* stats_out,
                                    flashmap_stream stream);

/* The device error word (FLASHMAP_DEVERR_* bits), then clears it. Synchronizes
 * `stream`. Returns E_DEVICE when the word was non-zero. */
flashmap_status flashmap_get_device_error(flashmap_model* model, flashmap_stream stream,
                                          uint32_t* code);

/* A description of the last failed call on this thread ("" if none). */
const char* flashmap_last_error(void);

/* ----------------------------------------------------------------------------------
 * Launch timing. While profiling is on, the write/draft/sample calls of `model`
 * record a CUDA event pair on their stream around every kernel launch, with the
 * launch's kind and GEMM shape. Calls stay asynchronous; do not profile inside a
 * stream capture. Kinds: */
#define FLASHMAP_KIND_GEMM 0       /* tcgen05 (bf16) or SIMT (float32) linear */
#define FLASHMAP_KIND_XATTN 1      /* paged cross-attention items */
#define FLASHMAP_KIND_XCOMBINE 2   /* split-KV combine */
#define FLASHMAP_KIND_SELF_ATTN 3  /* block self-attention */
#define FLASHMAP_KIND_ROWS 4       /* norms, RoPE, GELU, noise, gather, KV write, plan */
#define FLASHMAP_KIND_SAMPLE 5     /* sampler and full-vocabulary scatter */
#define FLASHMAP_KIND_MEMSET 6     /* accumulator clears */

typedef struct {
  int32_t kind;
  int32_t layer;      /* DiT block of the launch, -1 outside the blocks */
  int32_t rows, n, k; /* GEMM: activation rows x out features x in features; else 0 */
  float ms;           /* event-timed duration */
} flashmap_launch_record;

/* Starts recording up to `capacity` launches (host-side events; no device memory). */
flashmap_status flashmap_profile_start(flashmap_model* model, int32_t capacity);
/* Stops, synchronizes the recorded events and copies up to `capacity` records (host)
 * to `out`; *count receives the number recorded. */
flashmap_status flashmap_profile_stop(flashmap_model* model, flashmap_launch_record* out, int32_t capacity,
                                      int32_t* count);

/* The tcgen05 GEMM launches of one one-jump step of `bs` requests, with the shapes,
 * weights and launch configuration the calls use, back to back on `stream` and with
 * nothing else between them: flashmap_draft_block_with_write's linears (fc over the
 * bs * window verify-window rows, none when window = 0; the anchor projection; one
 * all-layer context K/V GEMM over the anchors and the window rows; the noise and DiT
 * linears) and the sampler's folded head (reading `hidden`, device [bs * K][D] act
 * dtype). The linears a draft runs on its two branches side by side take one CTA per
 * SM here too. They read and write the workspace (sized for bs requests and bs *
 * window write rows); what they leave there is not a result, and the chain clears
 * only the GEMMs' own counters (three small memsets). A measurement hook: captured in a CUDA graph and
 * replayed, it times the GEMM kernel the way a step runs it, without the time of
 * the kernels between the GEMMs. *bytes_out receives the chain's algorithmic bytes
 * (each weight once, e4m3 weights one byte and a float32 scale per output channel;
 * activations read; outputs written), *launches_out the number of GEMM launches.
 * E_UNSUPPORTED for several-jump drafts and float32 weights. */
flashmap_status flashmap_profile_gemm_chain(flashmap_model* model, int32_t bs, int32_t window, const void* hidden,
                                           void* workspace, size_t workspace_bytes, int64_t* bytes_out,
                                           int32_t* launches_out, flashmap_stream stream);

/* ----------------------------------------------------------------------------------
 * Test and inspection exports. They run the library's own kernels on small inputs.
 * ---------------------------------------------------------------------------------- */

/* The timeout path of the kernels' pipeline waits, exercised without any fault: one
 * warp on `stream` waits limit_ns (at most 100 ms, else E_INVALID) on an mbarrier
 * that nothing arrives on, through the same bounded wait every pipeline uses, gives
 * up, sets FLASHMAP_DEVERR_TIMEOUT in the model's device error word and returns (read
 * it with flashmap_get_device_error). No copy or MMA is issued. Test-only. */
flashmap_status flashmap_debug_wait_timeout(flashmap_model* model, uint64_t limit_ns, flashmap_stream stream);

/* Raw Philox4x32-10 words (Salmon et al., SC'11, section 3) for n (key, counter)
 * pairs: seeds (device) uint64 [n] (key = lo32, hi32), ctr (device) uint32 [n][4];
 * out (device) uint32 [n][4]; normals (device) float32 [n][4] (Box-Muller on the word
 * pairs, the draft noise transform) or NULL. */
flashmap_status flashmap_debug_philox(const uint64_t* seeds, const uint32_t* ctr, int64_t n,
                                      uint32_t* out, float* normals, flashmap_stream stream);

/* out[r][n] += sum_k x[r][k] w[n][k] for r < rows, n < out_features, through the same
 * GEMM the draft uses for dtype (F32: SIMT; BF16: tcgen05). x (device) [rows][in]
 * and w (device) [out][in] in dtype; out (device) float32 [rows][out_features].
 * dtype E4M3: x and w are bf16; w is first quantized per output channel exactly as
 * flashmap_load_weights does for E4M3 weights, and the e4m3 tcgen05 GEMM computes
 * out += x (q * scale)^T (stream-ordered temporary allocation for q and scale). */
flashmap_status flashmap_debug_linear(int32_t dtype, const void* x, const void* w, int32_t rows,
                                      int32_t in_features, int32_t out_features, float* out,
                                      flashmap_stream stream);

/* The model's derived tensors, copied to caller buffers (device): the Cholesky
 * factor L (H, H) float32, the uniform constant u (H) float32, hot ids (Vd) int64.
 * Any pointer may be NULL. */
flashmap_status flashmap_debug_constants(const flashmap_model* model, float* chol, float* uniform,
                                         int64_t* hot_ids, flashmap_stream stream);

/* The folded-noise constants of a model loaded with noise_path 1, copied to caller
 * buffers (device): variance = lam / H (H) float32 in ascending order, x_embed(u) (D)
 * float32, the projection as the GEMM holds it, M^T (D, H) in act_dtype; sweeps (host)
 * the Jacobi sweeps the load took. Any pointer may be NULL. E_INVALID when the model
 * was loaded with noise_path 0. */
flashmap_status flashmap_debug_folded(const flashmap_model* model, float* variance, float* embedded_uniform,
                                      void* proj, int32_t* sweeps, flashmap_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* FLASHMAP_H_ */
