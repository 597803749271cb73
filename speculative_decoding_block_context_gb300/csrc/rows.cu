// Row-wise kernels of the FlashMap step: modulated LayerNorm, RMSNorm variants
// (context, anchor, noise embedding), the seeded draft noise, per-head q/k RMSNorm +
// interleaved RoPE, and the paged context-KV write. The float32 GEMM outputs they read
// are written whole by their GEMM (every element once), so nothing here clears them.

#include <algorithm>
#include <climits>

#include "common.cuh"
#include "internal.h"
#include "philox.cuh"

namespace fm {
namespace {

// Loads the EPL channels lane*EPL.. of one head vector (L2).
template <int EPL>
__device__ __forceinline__ void load_head(const float* src, float (&v)[EPL], int lane) {
  const float* p = src + lane * EPL;
  if constexpr (EPL == 4) {
    const float4 t = LDCG(reinterpret_cast<const float4*>(p));
    v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
  } else if constexpr (EPL == 2) {
    const float2 t = LDCG(reinterpret_cast<const float2*>(p));
    v[0] = t.x, v[1] = t.y;
  } else {
    v[0] = LDCG(p);
  }
}

template <typename T, int N>
__device__ __forceinline__ void store_vec(T* dst, const float* v) {
  if constexpr (sizeof(T) == 2 && N == 4) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&a);
    u.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(dst) = u;
  } else if constexpr (sizeof(T) == 4 && N == 4) {
    *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
  } else if constexpr (sizeof(T) == 1) {  // e4m3 pool: scale 1, nearest even, saturated at +-448
    uint32_t u = 0;
#pragma unroll
    for (int e = 0; e < N; ++e)
      u |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(v[e], __NV_SATFINITE, __NV_E4M3)) << (8 * (e & 3));
    if constexpr (N == 4)
      *reinterpret_cast<uint32_t*>(dst) = u;
    else if constexpr (N == 2)
      *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(u);
    else
      dst[0] = static_cast<T>(u);
  } else {
#pragma unroll
    for (int e = 0; e < N; ++e) dst[e] = from_f32<T>(v[e]);
  }
}

// ------------------------------------------------------------------ context-KV write

// One CTA per (row, layer), one warp per head. Thread 0 resolves the row's slot (the
// request's start position, commit length, page-table row and page: four dependent
// loads of per-request scalars) and hands it to the CTA through shared memory, while
// every warp already streams its head's key and value from the accumulator. Loading
// the scalars once per CTA instead of once per warp keeps thousands of CTAs from
// queueing on the same few L2 sectors.
template <typename T, int EPL>
__global__ void __launch_bounds__(1024, 2) kv_write_kernel(KvWriteArgs a) {
  constexpr int HD = EPL * 32;
  __shared__ int64_t s_slot;
  __shared__ int s_pos;
  pdl_trigger();
  pdl_wait();
  const int il = blockIdx.x, l = blockIdx.y;
  if (a.rows_dev && il >= LDCG(a.rows_dev)) return;  // past the compacted rows (CTA-uniform)
  const int64_t i = a.row_src ? static_cast<int64_t>(LDCG(a.row_src + il)) : a.row0 + il;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int D = a.nh * HD;
  const float* row = a.acc + static_cast<int64_t>(il) * a.ld + static_cast<int64_t>(l) * 2 * D;
  // this warp's first head, loaded before the slot is known
  float k[EPL], v[EPL], kw[EPL];
  if (warp < a.nh) {
    load_head<EPL>(row + warp * HD, k, lane);
    load_head<EPL>(row + D + warp * HD, v, lane);
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) kw[e] = a.k_norm[static_cast<int64_t>(l) * HD + lane * EPL + e];
  if (threadIdx.x == 0) {
    const int b = static_cast<int>(i / a.W), c = static_cast<int>(i - static_cast<int64_t>(b) * a.W);
    // the three per-request scalars in one round trip, then the page
    const int start = LDCG(a.start_pos + b);
    const int clen = a.commit_lens ? LDCG(a.commit_lens + b) : INT_MAX;
    const int rrow = a.req_pool_idx ? LDCG(a.req_pool_idx + b) : b;
    const int pos = start + c;
    int64_t slot = -1;
    if (c < clen) {
      const int pi = pos >= 0 ? pos / a.P : -1;
      if (pos < 0 || pos >= a.max_pos || pi >= a.r2p_stride || rrow < 0) {
        if (l == 0) set_dev_error(a.dev_err, FLASHMAP_DEVERR_POSITION);
      } else {
        const int page = LDCG(a.req_to_page + static_cast<int64_t>(rrow) * a.r2p_stride + pi);
        if (page < 0 || page >= a.num_pages) {
          if (l == 0) set_dev_error(a.dev_err, FLASHMAP_DEVERR_PAGE);
        } else {
          slot = static_cast<int64_t>(page) * a.P + (pos - pi * a.P);
        }
      }
    }
    if (a.out_loc && l == 0) a.out_loc[i] = slot;
    s_slot = slot;
    s_pos = pos;
  }
  __syncthreads();
  const int64_t slot = s_slot;
  if (slot < 0) return;
  const float2* rope = a.rope + static_cast<int64_t>(s_pos) * (HD / 2);
  T* pool = static_cast<T*>(a.pool);
  const int64_t page = slot / a.P, off = slot - page * a.P;
  const int64_t kv_stride = a.num_pages * a.nh * a.P;  // pool rows between a layer's keys and values
  const int64_t kbase = (static_cast<int64_t>(l) * 2 * a.num_pages + page) * a.nh * a.P + off;
  for (int h = warp; h < a.nh; h += nw) {
    if (h != warp) {  // more heads than warps
      load_head<EPL>(row + h * HD, k, lane);
      load_head<EPL>(row + D + h * HD, v, lane);
    }
    head_norm_rope_w<EPL>(k, kw, a.eps, rope, lane);
    const int64_t r = kbase + static_cast<int64_t>(h) * a.P;
    store_vec<T, EPL>(pool + r * HD + lane * EPL, k);
    if constexpr (sizeof(T) == 1) {
      // an e4m3 pool keeps each (page, head) block of values channel-major: channel c of
      // the block's positions is a row of P bytes, and within each 16 positions position
      // 2t + e sits at byte 4t + e and position 8 + 2t + e at 4t + 2 + e (t < 4, e < 2),
      // the order in which the cross-attention's P V product takes them (a plain
      // ldmatrix gives each thread 4 consecutive bytes)
      const int o16 = static_cast<int>(off & 15);
      T* vb = pool + (r - off + kv_stride) * HD + (off & ~15LL) + (4 * ((o16 & 7) >> 1) + 2 * (o16 >> 3) + (o16 & 1));
#pragma unroll
      for (int e = 0; e < EPL; ++e)
        vb[static_cast<int64_t>(lane * EPL + e) * a.P] =
            static_cast<T>(__nv_cvt_float_to_fp8(v[e], __NV_SATFINITE, __NV_E4M3));
    } else {
      store_vec<T, EPL>(pool + (r + kv_stride) * HD + lane * EPL, v);
    }
  }
}

// ------------------------------------------------------------------ row norms
//
// One CTA of 256 threads per row; thread t holds the float4 groups t, t + 256, ...
// (NV of them) in registers: the row is read once, both statistics come from the
// registers, and the result is written once.

constexpr int kRowThreads = 256;

// constants (weights, modulations) may use any load; rows produced in the step use L2
template <int NV, bool kCoherent>
__device__ __forceinline__ void load_row4(const float* src, int w4, float4 (&v)[NV]) {
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int f = threadIdx.x + i * kRowThreads;
    const float4* p = reinterpret_cast<const float4*>(src) + f;
    v[i] = f < w4 ? (kCoherent ? LDCG(p) : *p) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Merges (count, mean, M2) statistics b into a: the combined count, mean and sum of
// squared deviations (Chan, Golub and LeVeque's pairwise update).
__device__ __forceinline__ void merge_mean_m2(float& n, float& mean, float& m2, float nb, float meanb, float m2b) {
  const float nt = n + nb;
  if (nt > 0.f) {
    const float d = meanb - mean, f = nb / nt;
    mean = fmaf(d, f, mean);
    m2 = m2 + m2b + d * d * n * f;
    n = nt;
  }
}

// Block-wide merge of every thread's (count, mean, M2); every thread gets the same
// result (the warps' partials are merged in warp order). red: >= 3 * warps floats.
__device__ __forceinline__ void block_mean_m2(float& n, float& mean, float& m2, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float nb = __shfl_xor_sync(0xffffffffu, n, o), mb = __shfl_xor_sync(0xffffffffu, mean, o),
                qb = __shfl_xor_sync(0xffffffffu, m2, o);
    merge_mean_m2(n, mean, m2, nb, mb, qb);
  }
  if (lane == 0) {
    red[3 * warp] = n;
    red[3 * warp + 1] = mean;
    red[3 * warp + 2] = m2;
  }
  __syncthreads();
  n = 0.f, mean = 0.f, m2 = 0.f;
  for (int w = 0; w < nw; ++w) merge_mean_m2(n, mean, m2, red[3 * w], red[3 * w + 1], red[3 * w + 2]);
}

// out = LayerNorm(x) * mscale + mshift   (no affine; biased variance)
template <typename T, int NV>
__global__ void __launch_bounds__(kRowThreads) ln_mod_kernel(const float* __restrict__ x, int width,
                                                             const float* __restrict__ ms,
                                                             const float* __restrict__ mh, float eps,
                                                             T* __restrict__ out) {
  __shared__ float red[32];
  pdl_trigger();
  const int w4 = width >> 2;
  float4 m1[NV], m2[NV], v[NV];
  load_row4<NV, false>(ms, w4, m1);  // constants: read before waiting
  load_row4<NV, false>(mh, w4, m2);
  pdl_wait();
  load_row4<NV, true>(x + static_cast<int64_t>(blockIdx.x) * width, w4, v);
  // the row's mean and squared deviations in one block reduction: each thread's own
  // (count, mean, M2) in two passes over its registers, merged pairwise (Chan et al.)
  float s = 0.f, cnt = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    if (threadIdx.x + i * kRowThreads < w4) {
      s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
      cnt += 4.f;
    }
  }
  float mean = cnt > 0.f ? s / cnt : 0.f, dev2 = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    if (threadIdx.x + i * kRowThreads < w4) {
      const float a = v[i].x - mean, b = v[i].y - mean, c = v[i].z - mean, d = v[i].w - mean;
      dev2 += (a * a + b * b) + (c * c + d * d);
    }
  }
  block_mean_m2(cnt, mean, dev2, red);
  const float rstd = rsqrtf(dev2 / width + eps);
  T* o = out + static_cast<int64_t>(blockIdx.x) * width;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int f = threadIdx.x + i * kRowThreads;
    if (f < w4) {
      const float r[4] = {fmaf((v[i].x - mean) * rstd, m1[i].x, m2[i].x), fmaf((v[i].y - mean) * rstd, m1[i].y, m2[i].y),
                          fmaf((v[i].z - mean) * rstd, m1[i].z, m2[i].z), fmaf((v[i].w - mean) * rstd, m1[i].w, m2[i].w)};
      store_vec<T, 4>(o + 4 * f, r);
    }
  }
}

// y = prescale * acc; v = y * w * rsqrt(mean(y^2) + eps); out = add ? add + gate * v : v.
template <typename T, int NV>
__global__ void __launch_bounds__(kRowThreads) rms_rows_kernel(const float* __restrict__ acc, int width,
                                                               const float* __restrict__ w, float eps,
                                                               float prescale, const float* __restrict__ add,
                                                               float gate, T* __restrict__ out, int ldo,
                                                               const int* __restrict__ rows_dev) {
  __shared__ float red[32];
  pdl_trigger();
  const int w4 = width >> 2;
  float4 wv[NV], av[NV], v[NV];
  load_row4<NV, false>(w, w4, wv);
  if (add) load_row4<NV, false>(add, w4, av);
  pdl_wait();
  if (rows_dev && static_cast<int>(blockIdx.x) >= LDCG(rows_dev)) return;  // CTA-uniform
  const float* ar = acc + static_cast<int64_t>(blockIdx.x) * width;
  load_row4<NV, true>(ar, w4, v);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    v[i].x *= prescale, v[i].y *= prescale, v[i].z *= prescale, v[i].w *= prescale;
    s += (v[i].x * v[i].x + v[i].y * v[i].y) + (v[i].z * v[i].z + v[i].w * v[i].w);
  }
  const float r = rsqrtf(block_sum(s, red) / width + eps);
  T* o = out + static_cast<int64_t>(blockIdx.x) * ldo;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int f = threadIdx.x + i * kRowThreads;
    if (f < w4) {
      float q[4] = {v[i].x * r * wv[i].x, v[i].y * r * wv[i].y, v[i].z * r * wv[i].z, v[i].w * r * wv[i].w};
      if (add) {
        q[0] = fmaf(gate, q[0], av[i].x);
        q[1] = fmaf(gate, q[1], av[i].y);
        q[2] = fmaf(gate, q[2], av[i].z);
        q[3] = fmaf(gate, q[3], av[i].w);
      }
      store_vec<T, 4>(o + 4 * f, q);
    }
  }
}

// The committed columns of a verify-window chunk, in order (sglang/model.py,
// write_target_hidden_kv: only committed columns are written): an exclusive scan of
// the keep flags, 1024 rows at a time.
__global__ void __launch_bounds__(1024) window_compact_kernel(const int32_t* __restrict__ commit_lens, int W,
                                                              int64_t r0, int rows, int32_t* __restrict__ row_src,
                                                              int* __restrict__ rows_dev,
                                                              int64_t* __restrict__ out_loc, int* __restrict__ total_dev,
                                                              int total_base) {
  __shared__ int scan[1024];
  __shared__ int carry;
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < rows; base += 1024) {
    const int t = base + static_cast<int>(threadIdx.x);
    const int64_t g = r0 + t;
    int keep = 0;
    if (t < rows) {
      const int64_t b = g / W;
      keep = g - b * W < LDCG(commit_lens + b) ? 1 : 0;
      if (!keep && out_loc) out_loc[g] = -1;
    }
    scan[threadIdx.x] = keep;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
      const int x = threadIdx.x >= static_cast<unsigned>(off) ? scan[threadIdx.x - off] : 0;
      __syncthreads();
      scan[threadIdx.x] += x;
      __syncthreads();
    }
    if (keep) row_src[carry + scan[threadIdx.x] - 1] = static_cast<int32_t>(g);
    __syncthreads();
    if (threadIdx.x == 1023) carry += scan[1023];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    *rows_dev = carry;
    if (total_dev) *total_dev = total_base + carry;
  }
}

__global__ void __launch_bounds__(256) gather_window_rows_kernel(const uint8_t* __restrict__ x, int64_t row_bytes,
                                                                 const int32_t* __restrict__ row_src,
                                                                 const int* __restrict__ rows_dev,
                                                                 uint8_t* __restrict__ xc) {
  pdl_trigger();
  pdl_wait();
  const int k = blockIdx.x;
  if (k >= LDCG(rows_dev)) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(LDCG(row_src + k)) * row_bytes);
  uint4* dst = reinterpret_cast<uint4*>(xc + static_cast<int64_t>(k) * row_bytes);
  for (int64_t i = threadIdx.x; i < row_bytes / 16; i += blockDim.x) dst[i] = src[i];
}

// Row copies in 16-byte chunks: grid (rows, chunk blocks).
__global__ void gather_rows_kernel(const uint4* __restrict__ table, int64_t nrows, int chunks,
                                   const int64_t* __restrict__ ids, uint4* __restrict__ out, unsigned* dev_err) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  const int64_t id = LDCG(ids + b);
  const bool ok = id >= 0 && id < nrows;
  if (!ok && threadIdx.x == 0 && blockIdx.y == 0) set_dev_error(dev_err, FLASHMAP_DEVERR_TOKEN);
  const int c = blockIdx.y * blockDim.x + threadIdx.x;
  if (c < chunks) out[static_cast<int64_t>(b) * chunks + c] = ok ? table[id * chunks + c] : make_uint4(0, 0, 0, 0);
}

// z[b*K + k][j] ~ N(0, 1) keyed by (seeds[b], position anchor_pos[b] + 1 + k): counter
// (j / 4, position, 0, 0), normal j % 4 from the Box-Muller pairs (w0, w1), (w2, w3).
template <typename T>
// Row r is slot k = r % K of block r / K; with n_cand candidates per request, block
// bc is candidate bc % n_cand of request bc / n_cand, keyed by counter word 3 = the
// candidate (0 for a single draft).
__global__ void draft_noise_kernel(const uint64_t* __restrict__ seeds, const int32_t* __restrict__ anchor_pos,
                                   int K, int n_cand, int H, int64_t total, float scale, T* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int n4 = (H + 3) >> 2;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int row = static_cast<int>(t / n4), j4 = static_cast<int>(t - static_cast<int64_t>(row) * n4);
    const int bc = row / K, k = row - bc * K;
    const int b = bc / n_cand, c = bc - b * n_cand;
    const uint32_t pos = static_cast<uint32_t>(LDCG(anchor_pos + b) + 1 + k);
    const uint4 w = philox_seeded(LDCG(seeds + b), static_cast<uint32_t>(j4), pos, kDomainDraftNoise,
                                  static_cast<uint32_t>(c));
    const float2 n01 = box_muller(w.x, w.y), n23 = box_muller(w.z, w.w);
    const float v[4] = {scale * n01.x, scale * n01.y, scale * n23.x, scale * n23.y};
    T* o = out + static_cast<int64_t>(row) * H + 4 * j4;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (4 * j4 + e < H) o[e] = from_f32<T>(v[e]);
  }
}

// The folded path's noise input, one CTA per drafted row: z (the draft_noise
// normals of the row, times scale) and r = rsqrt(sum_i variance_i z_i^2 + eps), written
// as z * gate * r (flashmap/sglang/model.py, _folded_noise; flashmap/vllm/model.py,
// _one_jump). A thread holds up to kFoldPer groups of 4 normals between the sum and
// the store (H <= 4 * kFoldPer * blockDim).
constexpr int kFoldThreads = 1024, kFoldPer = 4;

template <typename T>
__global__ void __launch_bounds__(kFoldThreads) folded_noise_kernel(const uint64_t* __restrict__ seeds,
                                                                    const int32_t* __restrict__ anchor_pos, int K,
                                                                    int n_cand, int H, float scale,
                                                                    const float* __restrict__ variance, float eps,
                                                                    float gate, T* __restrict__ out) {
  __shared__ float red[32];
  __shared__ uint64_t s_seed;
  __shared__ uint32_t s_pos;
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x, bc = row / K, k = row - bc * K;
  const int b = bc / n_cand, c = bc - b * n_cand;
  if (threadIdx.x == 0) {
    s_seed = LDCG(seeds + b);
    s_pos = static_cast<uint32_t>(LDCG(anchor_pos + b) + 1 + k);
  }
  __syncthreads();
  const int n4 = H >> 2;
  const float4* var4 = reinterpret_cast<const float4*>(variance);
  float4 z[kFoldPer];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kFoldPer; ++i) {
    const int j4 = threadIdx.x + i * blockDim.x;
    if (j4 < n4) {
      const uint4 w = philox_seeded(s_seed, static_cast<uint32_t>(j4), s_pos, kDomainDraftNoise,
                                    static_cast<uint32_t>(c));
      const float2 n01 = box_muller(w.x, w.y), n23 = box_muller(w.z, w.w);
      z[i] = make_float4(scale * n01.x, scale * n01.y, scale * n23.x, scale * n23.y);
      const float4 v = var4[j4];
      ss = fmaf(v.x, z[i].x * z[i].x, ss);
      ss = fmaf(v.y, z[i].y * z[i].y, ss);
      ss = fmaf(v.z, z[i].z * z[i].z, ss);
      ss = fmaf(v.w, z[i].w * z[i].w, ss);
    }
  }
  ss = block_sum(ss, red);
  const float f = gate * rsqrtf(ss + eps);
  T* o = out + static_cast<int64_t>(row) * H;
#pragma unroll
  for (int i = 0; i < kFoldPer; ++i) {
    const int j4 = threadIdx.x + i * blockDim.x;
    if (j4 < n4) {
      o[4 * j4 + 0] = from_f32<T>(z[i].x * f);
      o[4 * j4 + 1] = from_f32<T>(z[i].y * f);
      o[4 * j4 + 2] = from_f32<T>(z[i].z * f);
      o[4 * j4 + 3] = from_f32<T>(z[i].w * f);
    }
  }
}

// The timeout path of a pipeline wait, exercised on purpose: one warp waits on an
// mbarrier that nothing arrives on, with the given limit, through the same bounded
// wait the pipelines use; the wait gives up and the kernel reports
// FLASHMAP_DEVERR_TIMEOUT in the error word and returns. No copy or MMA is issued.
__global__ void wait_timeout_probe_kernel(uint64_t limit_ns, unsigned* dev_err) {
  __shared__ uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  const bool ok = mbar_wait_for(&bar, 0, &abort_flag, limit_ns);
  if (threadIdx.x == 0 && !ok) set_dev_error(dev_err, FLASHMAP_DEVERR_TIMEOUT);
}

__global__ void zero_kernel(ZeroList z) {
  pdl_trigger();
  pdl_wait();
  for (int r = 0; r < z.count; ++r) {
    float4* p = reinterpret_cast<float4*>(z.ptr[r]);
    const int64_t n4 = (reinterpret_cast<uintptr_t>(z.ptr[r]) & 15) ? 0 : z.n[r] >> 2;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
      p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t i = (n4 << 2) + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < z.n[r];
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
      z.ptr[r][i] = 0.f;
  }
}

}  // namespace

// ------------------------------------------------------------------ launchers

cudaError_t wait_timeout_probe(const Launch& L, uint64_t limit_ns) {
  return launch_k(L, wait_timeout_probe_kernel, dim3(1), dim3(32), 0, limit_ns, L.dev_err);
}

cudaError_t zero_ranges(const Launch& L, const ZeroList& z) {
  int64_t total = 0;
  for (int r = 0; r < z.count; ++r) total += z.n[r];
  if (total <= 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>((total / 4 + 255) / 256 + 1, static_cast<int64_t>(L.num_sms) * 8));
  return launch_k(L, zero_kernel, dim3(blocks), dim3(256), 0, z);
}

#define FM_DISPATCH_T(dtype, ...)                 \
  do {                                            \
    if ((dtype) == FLASHMAP_F32) {                \
      using T = float;                            \
      __VA_ARGS__;                                \
    } else {                                      \
      using T = __nv_bfloat16;                    \
      __VA_ARGS__;                                \
    }                                             \
  } while (0)

#define FM_DISPATCH_EPL(hd, ...)                  \
  do {                                            \
    if ((hd) == 32) {                             \
      constexpr int EPL = 1;                      \
      __VA_ARGS__;                                \
    } else if ((hd) == 64) {                      \
      constexpr int EPL = 2;                      \
      __VA_ARGS__;                                \
    } else {                                      \
      constexpr int EPL = 4;                      \
      __VA_ARGS__;                                \
    }                                             \
  } while (0)

cudaError_t window_compact(const Launch& L, const int32_t* commit_lens, int W, int64_t r0, int rows,
                           int32_t* row_src, int* rows_dev, int64_t* out_loc, int* total_dev, int total_base) {
  if (rows <= 0 || W <= 0) return cudaSuccess;
  return launch_k(L, window_compact_kernel, dim3(1), dim3(1024), 0, commit_lens, W, r0, rows, row_src, rows_dev,
                  out_loc, total_dev, total_base);
}

cudaError_t gather_window_rows(const Launch& L, const void* x, int64_t row_bytes, const int32_t* row_src,
                               const int* rows_dev, int max_rows, void* xc) {
  if (max_rows <= 0) return cudaSuccess;
  if ((row_bytes & 15) || (reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(xc) & 15))
    return cudaErrorInvalidValue;
  return launch_k(L, gather_window_rows_kernel, dim3(max_rows), dim3(256), 0, static_cast<const uint8_t*>(x),
                  row_bytes, row_src, rows_dev, static_cast<uint8_t*>(xc));
}

cudaError_t kv_write(const Launch& L, int dtype, const KvWriteArgs& a) {
  if (a.rows <= 0) return cudaSuccess;
  KvWriteArgs b = a;
  b.dev_err = L.dev_err;
  dim3 grid(a.rows, a.L);
  cudaError_t e = cudaSuccess;
  const dim3 block(32 * std::min(a.nh, 32));
  if (dtype == FLASHMAP_E4M3) {
    using T = uint8_t;
    FM_DISPATCH_EPL(a.hd, (e = launch_k(L, kv_write_kernel<T, EPL>, grid, block, 0, b)));
  } else {
    FM_DISPATCH_T(dtype, FM_DISPATCH_EPL(a.hd, (e = launch_k(L, kv_write_kernel<T, EPL>, grid, block, 0, b))));
  }
  return e;
}

#define FM_DISPATCH_NV(width, ...)                                          \
  do {                                                                      \
    const int nv_ = ((width) / 4 + kRowThreads - 1) / kRowThreads;          \
    if (nv_ <= 1) {                                                         \
      constexpr int NV = 1;                                                 \
      __VA_ARGS__;                                                          \
    } else if (nv_ <= 2) {                                                  \
      constexpr int NV = 2;                                                 \
      __VA_ARGS__;                                                          \
    } else if (nv_ <= 4) {                                                  \
      constexpr int NV = 4;                                                 \
      __VA_ARGS__;                                                          \
    } else if (nv_ <= 8) {                                                  \
      constexpr int NV = 8;                                                 \
      __VA_ARGS__;                                                          \
    } else {                                                                \
      constexpr int NV = 16;                                                \
      __VA_ARGS__;                                                          \
    }                                                                       \
  } while (0)

// width % 4 == 0 and width <= 16384 (checked at load)
cudaError_t ln_mod_rows(const Launch& L, int dtype, const float* x, int rows, int width, const float* ms,
                        const float* mh, float eps, void* out) {
  if (rows <= 0) return cudaSuccess;
  cudaError_t e = cudaSuccess;
  FM_DISPATCH_T(dtype, FM_DISPATCH_NV(width, (e = launch_k(L, ln_mod_kernel<T, NV>, dim3(rows), dim3(kRowThreads), 0,
                                                          x, width, ms, mh, eps, static_cast<T*>(out)))));
  return e;
}

cudaError_t rms_rows(const Launch& L, int dtype, const float* acc, int rows, int width, const float* w, float eps,
                     float prescale, const float* add, float gate, void* out, int ldo, const int* rows_dev) {
  if (rows <= 0) return cudaSuccess;
  cudaError_t e = cudaSuccess;
  FM_DISPATCH_T(dtype, FM_DISPATCH_NV(width, (e = launch_k(L, rms_rows_kernel<T, NV>, dim3(rows), dim3(kRowThreads),
                                                          0, acc, width, w, eps, prescale, add, gate,
                                                          static_cast<T*>(out), ldo, rows_dev))));
  return e;
}

// width * element size must be a multiple of 16 bytes (checked at load)
cudaError_t gather_rows(const Launch& L, int dtype, const void* table, int64_t nrows, int width, const int64_t* ids,
                        int n, void* out) {
  if (n <= 0) return cudaSuccess;
  const int chunks = width * (dtype == FLASHMAP_F32 ? 4 : 2) / 16;
  return launch_k(L, gather_rows_kernel, dim3(n, (chunks + 255) / 256), dim3(256), 0,
                  static_cast<const uint4*>(table), nrows, chunks, ids, static_cast<uint4*>(out), L.dev_err);
}

cudaError_t draft_noise(const Launch& L, int dtype, const uint64_t* seeds, const int32_t* anchor_pos, int bs, int K,
                        int H, void* out, int n_cand, float scale) {
  const int64_t total = static_cast<int64_t>(bs) * n_cand * K * ((H + 3) / 4);
  if (total <= 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(L.num_sms) * 16));
  cudaError_t e = cudaSuccess;
  FM_DISPATCH_T(dtype, (e = launch_k(L, draft_noise_kernel<T>, dim3(blocks), dim3(256), 0, seeds, anchor_pos, K,
                                     n_cand, H, total, scale, static_cast<T*>(out))));
  return e;
}

cudaError_t folded_noise(const Launch& L, int dtype, const uint64_t* seeds, const int32_t* anchor_pos, int bs, int K,
                         int H, int n_cand, float scale, const float* variance, float eps, float gate, void* out) {
  const int rows = bs * n_cand * K;
  if (rows <= 0) return cudaSuccess;
  if (H % 4 || H > 4 * kFoldPer * kFoldThreads) return cudaErrorInvalidValue;
  const int threads = std::min(kFoldThreads, std::max(32, ((H / 4 + kFoldPer - 1) / kFoldPer + 31) / 32 * 32));
  cudaError_t e = cudaSuccess;
  FM_DISPATCH_T(dtype, (e = launch_k(L, folded_noise_kernel<T>, dim3(rows), dim3(threads), 0, seeds, anchor_pos, K,
                                     n_cand, H, scale, variance, eps, gate, static_cast<T*>(out))));
  return e;
}

// Per-block copies of the request arrays for a draft of n_cand candidates per request:
// block bc = candidate bc % n_cand of request bc / n_cand.
__global__ void expand_kernel(const int32_t* __restrict__ anchor_pos, const int32_t* __restrict__ req_pool_idx,
                              int bs, int n_cand, int32_t* __restrict__ pos_out, int32_t* __restrict__ rpi_out) {
  pdl_trigger();
  pdl_wait();
  for (int bc = blockIdx.x * blockDim.x + threadIdx.x; bc < bs * n_cand; bc += gridDim.x * blockDim.x) {
    const int b = bc / n_cand;
    pos_out[bc] = LDCG(anchor_pos + b);
    rpi_out[bc] = req_pool_idx ? LDCG(req_pool_idx + b) : b;
  }
}

cudaError_t expand_requests(const Launch& L, const int32_t* anchor_pos, const int32_t* req_pool_idx, int bs,
                            int n_cand, int32_t* pos_out, int32_t* rpi_out) {
  const int n = bs * n_cand;
  return launch_k(L, expand_kernel, dim3((n + 255) / 256), dim3(256), 0, anchor_pos, req_pool_idx, bs, n_cand, pos_out,
                  rpi_out);
}

// ------------------------------------------------------------------ Philox export

namespace {
__global__ void philox_export_kernel(const uint64_t* seeds, const uint32_t* ctr, int64_t n, uint32_t* out,
                                     float* normals) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 w = philox_seeded(seeds[i], ctr[4 * i], ctr[4 * i + 1], ctr[4 * i + 2], ctr[4 * i + 3]);
    out[4 * i] = w.x;
    out[4 * i + 1] = w.y;
    out[4 * i + 2] = w.z;
    out[4 * i + 3] = w.w;
    if (normals) {
      const float2 a = box_muller(w.x, w.y), b = box_muller(w.z, w.w);
      normals[4 * i] = a.x;
      normals[4 * i + 1] = a.y;
      normals[4 * i + 2] = b.x;
      normals[4 * i + 3] = b.y;
    }
  }
}
}  // namespace

cudaError_t philox_export(cudaStream_t s, const uint64_t* seeds, const uint32_t* ctr, int64_t n, uint32_t* out,
                          float* normals) {
  if (n <= 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 4096));
  philox_export_kernel<<<blocks, 256, 0, s>>>(seeds, ctr, n, out, normals);
  return cudaGetLastError();
}

}  // namespace fm
