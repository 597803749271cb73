// Attention of the FlashMap DiT.
//
// Self-attention (flashmap/sglang/model.py, _denoise: block_self_attention) is
// non-causal across the block_size slots of one request: per (request, head), q and k
// are RMS-normed and rotated at the slot positions, and the K x K softmax is tiny.
//
// Cross-attention (flashmap/sglang/model.py, _paged_cross_attention; flashmap/vllm/
// model.py, paged_cross_attention) reads each request's context positions 0..p
// (anchor included) of one layer straight from the paged pool. The work is split
// flash-decoding style: a per-step plan (computed on the device once and shared by
// every layer, like the pages' FlashAttention scheduler metadata) cuts each request's
// context into chunks sized so the whole batch yields a few waves of (chunk, head)
// items; a persistent grid walks the items, each producing an unnormalized partial
// (O, running max, running sum) in base-2 exponent form; a combine pass merges a
// request's chunks per head.

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace fm {
namespace {

// ------------------------------------------------------------------ block self-attention

template <typename T, int EPL>
__global__ void self_attn_kernel(float* __restrict__ qkv, int K, int nh, const float* __restrict__ qn,
                                 const float* __restrict__ kn, float eps, const float2* __restrict__ rope_tab,
                                 int max_pos, const int32_t* __restrict__ anchor_pos, T* __restrict__ out,
                                 unsigned* dev_err) {
  constexpr int HD = EPL * 32;
  extern __shared__ float sm[];
  float* sq = sm;                  // [K][HD + 1]
  float* sk = sq + K * (HD + 1);   // [K][HD + 1]
  float* sv = sk + K * (HD + 1);   // [K][HD]
  const int b = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int D = nh * HD;
  const int k = warp;  // one warp per slot
  const int row = b * K + k;
  int pos = anchor_pos[b] + 1 + k;
  if (pos < 0 || pos >= max_pos) {
    if (lane == 0) set_dev_error(dev_err, FLASHMAP_DEVERR_POSITION);
    pos = 0;
  }
  const float2* rope = rope_tab + static_cast<int64_t>(pos) * (HD / 2);
  float* base = qkv + static_cast<int64_t>(row) * 3 * D + h * HD;
  float v[EPL];
#pragma unroll
  for (int part = 0; part < 3; ++part) {
    float* src = base + part * D;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      v[e] = src[lane * EPL + e];
      src[lane * EPL + e] = 0.f;
    }
    if (part < 2) {  // q or k: RMSNorm then rotation (the pair partner may be another lane)
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) ss = fmaf(v[e], v[e], ss);
      ss = warp_sum(ss);
      const float r = rsqrtf(ss * (1.f / HD) + eps);
      const float* w = part == 0 ? qn : kn;
#pragma unroll
      for (int e = 0; e < EPL; ++e) v[e] *= r * w[lane * EPL + e];
      if constexpr (EPL >= 2) {
#pragma unroll
        for (int e = 0; e < EPL; e += 2) {
          const float2 cs = rope[(lane * EPL + e) >> 1];
          const float x1 = v[e], x2 = v[e + 1];
          v[e] = x1 * cs.x - x2 * cs.y;
          v[e + 1] = x2 * cs.x + x1 * cs.y;
        }
      } else {
        const float other = __shfl_xor_sync(0xffffffffu, v[0], 1);
        const float2 cs = rope[lane >> 1];
        v[0] = (lane & 1) ? (v[0] * cs.x + other * cs.y) : (v[0] * cs.x - other * cs.y);
      }
    }
    float* dst = part == 0 ? sq + k * (HD + 1) : part == 1 ? sk + k * (HD + 1) : sv + k * HD;
#pragma unroll
    for (int e = 0; e < EPL; ++e) dst[lane * EPL + e] = v[e];
  }
  __syncthreads();
  // scores of slot k against slot j = lane
  const float scale = rsqrtf(static_cast<float>(HD));
  float s = -INFINITY;
  if (lane < K) {
    float acc = 0.f;
    const float* qr = sq + k * (HD + 1);
    const float* kr = sk + lane * (HD + 1);
    for (int d = 0; d < HD; ++d) acc = fmaf(qr[d], kr[d], acc);
    s = acc * scale;
  }
  const float m = warp_max(s);
  float p = lane < K ? expf(s - m) : 0.f;
  p /= warp_sum(p);
  T* o = out + static_cast<int64_t>(row) * D + h * HD;
  for (int d = lane; d < HD; d += 32) {
    float acc = 0.f;
    for (int j = 0; j < K; ++j) acc = fmaf(__shfl_sync(0xffffffffu, p, j), sv[j * HD + d], acc);
    o[d] = from_f32<T>(acc);
  }
}

// ------------------------------------------------------------------ split-KV plan

// plan (int32): [0] items = chunks * nh, [1] chunk length, [2] chunks,
// [3 .. 3 + bs] first chunk of each request (bs + 1 entries), then per chunk g the
// pair (request, chunk index within the request) at [4 + bs + 2g].
__global__ void __launch_bounds__(1024) xattn_plan_kernel(const int32_t* __restrict__ anchor_pos, int bs, int nh,
                                                          int target_items, int max_chunks, int* __restrict__ plan,
                                                          unsigned* dev_err) {
  __shared__ float red[32];
  __shared__ int carry;
  float t16 = 0.f;
  for (int b = threadIdx.x; b < bs; b += blockDim.x) t16 += static_cast<float>((max(anchor_pos[b] + 1, 1) + 15) / 16);
  const float total16 = block_sum(t16, red);
  const int64_t need = static_cast<int64_t>(total16) * nh;
  int bpc = static_cast<int>((need + target_items - 1) / target_items);
  bpc = max(bpc, 16);
  const int chunk_len = 16 * bpc;
  if (threadIdx.x == 0) carry = 0;
  int* first = plan + 3;
  int* pairs = plan + 4 + bs;
  __syncthreads();
  // exclusive scan of the per-request chunk counts, 1024 requests at a time
  __shared__ int scan[1024];
  for (int b0 = 0; b0 < bs; b0 += blockDim.x) {
    const int b = b0 + threadIdx.x;
    const int n = b < bs ? max(anchor_pos[b] + 1, 1) : 0;
    const int cnt = b < bs ? (n + chunk_len - 1) / chunk_len : 0;
    scan[threadIdx.x] = cnt;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
      const int x = threadIdx.x >= off ? scan[threadIdx.x - off] : 0;
      __syncthreads();
      scan[threadIdx.x] += x;
      __syncthreads();
    }
    const int excl = carry + scan[threadIdx.x] - cnt;
    if (b < bs) {
      first[b] = excl;
      for (int c = 0; c < cnt; ++c) {
        const int g = excl + c;
        if (g < max_chunks) {
          pairs[2 * g] = b;
          pairs[2 * g + 1] = c;
        }
      }
    }
    __syncthreads();
    if (threadIdx.x == 1023) carry += scan[1023];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    int chunks = carry;
    if (chunks > max_chunks) {
      set_dev_error(dev_err, FLASHMAP_DEVERR_POSITION);
      chunks = max_chunks;
    }
    first[bs] = chunks;
    plan[0] = chunks * nh;
    plan[1] = chunk_len;
    plan[2] = chunks;
  }
}

// ------------------------------------------------------------------ paged cross-attention items (SIMT)

template <typename T, int HD>
__global__ void __launch_bounds__(128) xattn_items_simt_kernel(XattnArgs a) {
  __shared__ float sq[16][HD];
  __shared__ float sk[16][HD + 1];
  __shared__ float sv[16][HD];
  __shared__ float ss[16][17];
  __shared__ float sm[16], sl[16], scorr[16];
  const int tid = threadIdx.x;
  const int K = a.K, nh = a.nh, D = nh * HD;
  const int items = a.plan[0], chunk_len = a.plan[1];
  const int* pairs = a.plan + 4 + a.bs;
  const T* pool = static_cast<const T*>(a.pool);
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int g = item / nh, h = item - g * nh;
    const int b = pairs[2 * g], c = pairs[2 * g + 1];
    const int n = a.anchor_pos[b] + 1;
    const int p0 = c * chunk_len, p1 = min(n, p0 + chunk_len);
    const int rrow = a.req_pool_idx ? a.req_pool_idx[b] : b;
    const T* qb = static_cast<const T*>(a.q) + static_cast<int64_t>(b) * K * D + h * HD;
    __syncthreads();
    for (int i = tid; i < 16 * HD; i += blockDim.x) {
      const int qi = i / HD, d = i - qi * HD;
      sq[qi][d] = qi < K ? to_f32(qb[static_cast<int64_t>(qi) * D + d]) * a.scale_log2 : 0.f;
    }
    if (tid < 16) {
      sm[tid] = -INFINITY;
      sl[tid] = 0.f;
    }
    float o[16];
#pragma unroll
    for (int qi = 0; qi < 16; ++qi) o[qi] = 0.f;
    for (int blk = p0; blk < p1; blk += 16) {
      // the 16 positions blk..blk+15 lie in one page (page_size is a multiple of 16)
      const int pi = blk / a.P;
      int page = pi < a.r2p_stride ? a.req_to_page[static_cast<int64_t>(rrow) * a.r2p_stride + pi] : -1;
      const bool ok = page >= 0 && page < a.num_pages;
      if (!ok && tid == 0) set_dev_error(a.dev_err, FLASHMAP_DEVERR_PAGE);
      const int off = blk - pi * a.P;
      const int64_t kb = ((((static_cast<int64_t>(a.layer) * 2 + 0) * a.num_pages + (ok ? page : 0)) * nh + h) * a.P + off) * HD;
      const int64_t vb = ((((static_cast<int64_t>(a.layer) * 2 + 1) * a.num_pages + (ok ? page : 0)) * nh + h) * a.P + off) * HD;
      __syncthreads();
      for (int i = tid; i < 16 * HD; i += blockDim.x) {
        const int j = i / HD, d = i - j * HD;
        const bool valid = ok && blk + j < p1;
        sk[j][d] = valid ? to_f32(pool[kb + i]) : 0.f;
        sv[j][d] = valid ? to_f32(pool[vb + i]) : 0.f;
      }
      __syncthreads();
      for (int i = tid; i < 256; i += blockDim.x) {
        const int qi = i >> 4, j = i & 15;
        float acc = 0.f;
#pragma unroll 8
        for (int d = 0; d < HD; ++d) acc = fmaf(sq[qi][d], sk[j][d], acc);
        ss[qi][j] = (blk + j < p1 && ok) ? acc : -INFINITY;
      }
      __syncthreads();
      if (tid < 16) {
        const int qi = tid;
        float mx = sm[qi];
        for (int j = 0; j < 16; ++j) mx = fmaxf(mx, ss[qi][j]);
        const float corr = mx == -INFINITY ? 1.f : exp2f(sm[qi] - mx);
        float sum = 0.f;
        for (int j = 0; j < 16; ++j) {
          const float p = ss[qi][j] == -INFINITY ? 0.f : exp2f(ss[qi][j] - mx);
          ss[qi][j] = p;
          sum += p;
        }
        sl[qi] = sl[qi] * corr + sum;
        sm[qi] = mx;
        scorr[qi] = corr;
      }
      __syncthreads();
      for (int d = tid; d < HD; d += blockDim.x) {
#pragma unroll
        for (int qi = 0; qi < 16; ++qi) {
          float acc = o[qi] * scorr[qi];
          for (int j = 0; j < 16; ++j) acc = fmaf(ss[qi][j], sv[j][d], acc);
          o[qi] = acc;
        }
      }
    }
    const int64_t pidx = static_cast<int64_t>(g) * nh + h;
    float* po = a.part_o + pidx * 16 * HD;
    for (int d = tid; d < HD; d += blockDim.x) {
#pragma unroll
      for (int qi = 0; qi < 16; ++qi) po[qi * HD + d] = o[qi];
    }
    __syncthreads();
    if (tid < 16) {
      a.part_ml[pidx * 32 + 2 * tid] = sm[tid];
      a.part_ml[pidx * 32 + 2 * tid + 1] = sl[tid];
    }
  }
}

// ------------------------------------------------------------------ combine

template <typename T, int HD>
__global__ void __launch_bounds__(HD) xattn_combine_kernel(XattnArgs a, T* __restrict__ out) {
  const int b = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  const int nh = a.nh, D = nh * HD;
  const int* first = a.plan + 3;
  const int g0 = first[b], g1 = first[b + 1];
  for (int qi = 0; qi < a.K; ++qi) {
    float M = -INFINITY;
    for (int g = g0; g < g1; ++g) M = fmaxf(M, a.part_ml[(static_cast<int64_t>(g) * nh + h) * 32 + 2 * qi]);
    float L = 0.f, acc = 0.f;
    for (int g = g0; g < g1; ++g) {
      const int64_t pidx = static_cast<int64_t>(g) * nh + h;
      const float m = a.part_ml[pidx * 32 + 2 * qi];
      if (m == -INFINITY) continue;
      const float w = exp2f(m - M);
      L = fmaf(a.part_ml[pidx * 32 + 2 * qi + 1], w, L);
      acc = fmaf(a.part_o[pidx * 16 * HD + qi * HD + d], w, acc);
    }
    out[(static_cast<int64_t>(b) * a.K + qi) * D + h * HD + d] = from_f32<T>(L > 0.f ? acc / L : 0.f);
  }
}

}  // namespace

#define FM_DISPATCH_T2(dtype, ...)  \
  do {                              \
    if ((dtype) == FLASHMAP_F32) {  \
      using T = float;              \
      __VA_ARGS__;                  \
    } else {                        \
      using T = __nv_bfloat16;      \
      __VA_ARGS__;                  \
    }                               \
  } while (0)

#define FM_DISPATCH_HD(hd, ...)     \
  do {                              \
    if ((hd) == 32) {               \
      constexpr int HD = 32;        \
      __VA_ARGS__;                  \
    } else if ((hd) == 64) {        \
      constexpr int HD = 64;        \
      __VA_ARGS__;                  \
    } else {                        \
      constexpr int HD = 128;       \
      __VA_ARGS__;                  \
    }                               \
  } while (0)

cudaError_t self_attention(const Launch& L, int dtype, float* qkv, int bs, int K, int nh, int hd, const float* qn,
                           const float* kn, float eps, const float2* rope, int max_pos, const int32_t* anchor_pos,
                           void* out) {
  if (bs <= 0) return cudaSuccess;
  dim3 grid(bs, nh);
  const size_t smem = static_cast<size_t>(K) * ((hd + 1) * 2 + hd) * sizeof(float);
  if (hd == 32) {
    FM_DISPATCH_T2(dtype, (self_attn_kernel<T, 1><<<grid, 32 * K, smem, L.stream>>>(
                              qkv, K, nh, qn, kn, eps, rope, max_pos, anchor_pos, static_cast<T*>(out), L.dev_err)));
  } else if (hd == 64) {
    FM_DISPATCH_T2(dtype, (self_attn_kernel<T, 2><<<grid, 32 * K, smem, L.stream>>>(
                              qkv, K, nh, qn, kn, eps, rope, max_pos, anchor_pos, static_cast<T*>(out), L.dev_err)));
  } else {
    FM_DISPATCH_T2(dtype, (self_attn_kernel<T, 4><<<grid, 32 * K, smem, L.stream>>>(
                              qkv, K, nh, qn, kn, eps, rope, max_pos, anchor_pos, static_cast<T*>(out), L.dev_err)));
  }
  return cudaGetLastError();
}

int xattn_target_items(int num_sms) { return num_sms * 8; }
int xattn_max_chunks(int num_sms, int nh, int bs) { return xattn_target_items(num_sms) / nh + bs + 1; }
size_t xattn_plan_ints(int num_sms, int nh, int bs) { return 4 + bs + 2 * static_cast<size_t>(xattn_max_chunks(num_sms, nh, bs)); }

cudaError_t xattn_plan(const Launch& L, const int32_t* anchor_pos, int bs, int nh, int* plan) {
  xattn_plan_kernel<<<1, 1024, 0, L.stream>>>(anchor_pos, bs, nh, xattn_target_items(L.num_sms),
                                              xattn_max_chunks(L.num_sms, nh, bs), plan, L.dev_err);
  return cudaGetLastError();
}

cudaError_t xattn_items(const Launch& L, int dtype, const XattnArgs& args) {
  XattnArgs a = args;
  a.dev_err = L.dev_err;
  const int grid = L.num_sms * 4;
  FM_DISPATCH_T2(dtype, FM_DISPATCH_HD(a.hd, (xattn_items_simt_kernel<T, HD><<<grid, 128, 0, L.stream>>>(a))));
  return cudaGetLastError();
}

cudaError_t xattn_combine(const Launch& L, int dtype, const XattnArgs& args, void* out) {
  XattnArgs a = args;
  a.dev_err = L.dev_err;
  dim3 cgrid(a.bs, a.nh);
  FM_DISPATCH_T2(dtype, FM_DISPATCH_HD(a.hd, (xattn_combine_kernel<T, HD><<<cgrid, HD, 0, L.stream>>>(
                                                 a, static_cast<T*>(out)))));
  return cudaGetLastError();
}

}  // namespace fm
