// Row-wise kernels of the FlashMap step: modulated LayerNorm, RMSNorm variants
// (context, anchor, noise embedding), GELU, the seeded draft noise, per-head q/k
// RMSNorm + interleaved RoPE, and the paged context-KV write. Every kernel that
// reads a GEMM's float32 accumulator also clears it, so the next GEMM into the same
// buffer starts from zero.

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "philox.cuh"

namespace fm {
namespace {

template <typename T, int EPL>
__device__ __forceinline__ void store_head(T* dst, const float (&v)[EPL], int lane) {
#pragma unroll
  for (int e = 0; e < EPL; ++e) dst[lane * EPL + e] = from_f32<T>(v[e]);
}

template <int EPL>
__device__ __forceinline__ void load_clear_head(float* src, float (&v)[EPL], int lane) {
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    v[e] = src[lane * EPL + e];
    src[lane * EPL + e] = 0.f;
  }
}

// ------------------------------------------------------------------ context-KV write

template <typename T, int EPL>
__global__ void __launch_bounds__(128) kv_write_kernel(KvWriteArgs a) {
  constexpr int HD = EPL * 32;
  pdl_trigger();
  pdl_wait();
  const int il = blockIdx.x, l = blockIdx.y;
  const int64_t i = a.row0 + il;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = static_cast<int>(i / a.W), c = static_cast<int>(i - static_cast<int64_t>(b) * a.W);
  const int pos = a.start_pos[b] + c;
  bool write = a.commit_lens == nullptr || c < a.commit_lens[b];
  int64_t slot = -1;
  if (write) {
    const int rrow = a.req_pool_idx ? a.req_pool_idx[b] : b;
    const int pi = pos >= 0 ? pos / a.P : -1;
    if (pos < 0 || pos >= a.max_pos || pi >= a.r2p_stride || rrow < 0) {
      if (threadIdx.x == 0 && l == 0) set_dev_error(a.dev_err, FLASHMAP_DEVERR_POSITION);
      write = false;
    } else {
      const int page = a.req_to_page[static_cast<int64_t>(rrow) * a.r2p_stride + pi];
      if (page < 0 || page >= a.num_pages) {
        if (threadIdx.x == 0 && l == 0) set_dev_error(a.dev_err, FLASHMAP_DEVERR_PAGE);
        write = false;
      } else {
        slot = static_cast<int64_t>(page) * a.P + (pos - pi * a.P);
      }
    }
  }
  if (a.out_loc && l == 0 && threadIdx.x == 0) a.out_loc[i] = write ? slot : -1;
  const int D = a.nh * HD;
  float* row = a.acc + static_cast<int64_t>(il) * a.ld + static_cast<int64_t>(l) * 2 * D;
  const float* kw = a.k_norm + static_cast<int64_t>(l) * HD;
  const float2* rope = write ? a.rope + static_cast<int64_t>(pos) * (HD / 2) : nullptr;
  T* pool = static_cast<T*>(a.pool);
  const int64_t page = write ? slot / a.P : 0, off = write ? slot - page * a.P : 0;
  for (int h = warp; h < a.nh; h += 4) {
    float k[EPL], v[EPL];
    load_clear_head<EPL>(row + h * HD, k, lane);
    load_clear_head<EPL>(row + D + h * HD, v, lane);
    if (!write) continue;
    head_norm_rope<EPL>(k, kw, a.eps, rope, lane);
    const int64_t kbase = (((static_cast<int64_t>(l) * 2 + 0) * a.num_pages + page) * a.nh + h) * a.P;
    const int64_t vbase = (((static_cast<int64_t>(l) * 2 + 1) * a.num_pages + page) * a.nh + h) * a.P;
    store_head<T, EPL>(pool + (kbase + off) * HD, k, lane);
    store_head<T, EPL>(pool + (vbase + off) * HD, v, lane);
  }
}

// ------------------------------------------------------------------ row norms

// out = LayerNorm(x) * mscale + mshift   (no affine; biased variance)
template <typename T>
__global__ void __launch_bounds__(256) ln_mod_kernel(const float* __restrict__ x, int width,
                                                     const float* __restrict__ ms, const float* __restrict__ mh,
                                                     float eps, T* __restrict__ out) {
  __shared__ float red[32];
  pdl_trigger();
  pdl_wait();
  const float* xr = x + static_cast<int64_t>(blockIdx.x) * width;
  float s = 0.f;
  for (int i = threadIdx.x; i < width; i += blockDim.x) s += xr[i];
  const float mean = block_sum(s, red) / width;
  float s2 = 0.f;
  for (int i = threadIdx.x; i < width; i += blockDim.x) {
    const float d = xr[i] - mean;
    s2 = fmaf(d, d, s2);
  }
  const float rstd = rsqrtf(block_sum(s2, red) / width + eps);
  T* o = out + static_cast<int64_t>(blockIdx.x) * width;
  for (int i = threadIdx.x; i < width; i += blockDim.x) o[i] = from_f32<T>(fmaf((xr[i] - mean) * rstd, ms[i], mh[i]));
}

// y = prescale * acc; v = y * w * rsqrt(mean(y^2) + eps); out = add ? add + gate * v : v
template <typename T>
__global__ void __launch_bounds__(256) rms_rows_kernel(float* __restrict__ acc, int width,
                                                       const float* __restrict__ w, float eps, float prescale,
                                                       const float* __restrict__ add, float gate,
                                                       T* __restrict__ out, int ldo) {
  __shared__ float red[32];
  pdl_trigger();
  pdl_wait();
  float* ar = acc + static_cast<int64_t>(blockIdx.x) * width;
  float s = 0.f;
  for (int i = threadIdx.x; i < width; i += blockDim.x) {
    const float y = prescale * ar[i];
    s = fmaf(y, y, s);
  }
  const float r = rsqrtf(block_sum(s, red) / width + eps);
  T* o = out + static_cast<int64_t>(blockIdx.x) * ldo;
  for (int i = threadIdx.x; i < width; i += blockDim.x) {
    float v = prescale * ar[i] * r * w[i];
    if (add) v = fmaf(gate, v, add[i]);
    o[i] = from_f32<T>(v);
    ar[i] = 0.f;
  }
}

template <typename T>
__global__ void gelu_kernel(float* __restrict__ acc, int64_t n, T* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float x = acc[i];
    out[i] = from_f32<T>(0.5f * x * (1.f + erff(x * 0.70710678118654752f)));
    acc[i] = 0.f;
  }
}

template <typename T>
__global__ void gather_rows_kernel(const T* __restrict__ table, int64_t nrows, int width,
                                   const int64_t* __restrict__ ids, T* __restrict__ out, unsigned* dev_err) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  int64_t id = ids[b];
  const bool ok = id >= 0 && id < nrows;
  if (!ok && threadIdx.x == 0) set_dev_error(dev_err, FLASHMAP_DEVERR_TOKEN);
  const T* src = table + (ok ? id : 0) * width;
  T* dst = out + static_cast<int64_t>(b) * width;
  for (int i = threadIdx.x; i < width; i += blockDim.x) dst[i] = ok ? src[i] : from_f32<T>(0.f);
}

// z[b*K + k][j] ~ N(0, 1) keyed by (seeds[b], position anchor_pos[b] + 1 + k): counter
// (j / 4, position, 0, 0), normal j % 4 from the Box-Muller pairs (w0, w1), (w2, w3).
template <typename T>
__global__ void draft_noise_kernel(const uint64_t* __restrict__ seeds, const int32_t* __restrict__ anchor_pos,
                                   int K, int H, int64_t total, T* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int n4 = (H + 3) >> 2;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int row = static_cast<int>(t / n4), j4 = static_cast<int>(t - static_cast<int64_t>(row) * n4);
    const int b = row / K, k = row - b * K;
    const uint32_t pos = static_cast<uint32_t>(anchor_pos[b] + 1 + k);
    const uint4 w = philox_seeded(seeds[b], static_cast<uint32_t>(j4), pos, kDomainDraftNoise, 0u);
    const float2 n01 = box_muller(w.x, w.y), n23 = box_muller(w.z, w.w);
    const float v[4] = {n01.x, n01.y, n23.x, n23.y};
    T* o = out + static_cast<int64_t>(row) * H + 4 * j4;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (4 * j4 + e < H) o[e] = from_f32<T>(v[e]);
  }
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

cudaError_t kv_write(const Launch& L, int dtype, const KvWriteArgs& a) {
  if (a.rows <= 0) return cudaSuccess;
  KvWriteArgs b = a;
  b.dev_err = L.dev_err;
  dim3 grid(a.rows, a.L);
  cudaError_t e = cudaSuccess;
  FM_DISPATCH_T(dtype, FM_DISPATCH_EPL(a.hd, (e = launch_k(L, kv_write_kernel<T, EPL>, grid, dim3(128), 0, b))));
  return e;
}

cudaError_t ln_mod_rows(const Launch& L, int dtype, const float* x, int rows, int width, const float* ms,
                        const float* mh, float eps, void* out) {
  if (rows <= 0) return cudaSuccess;
  cudaError_t e = cudaSuccess;
  FM_DISPATCH_T(dtype, (e = launch_k(L, ln_mod_kernel<T>, dim3(rows), dim3(256), 0, x, width, ms, mh, eps,
                                     static_cast<T*>(out))));
  return e;
}

cudaError_t rms_rows(const Launch& L, int dtype, float* acc, int rows, int width, const float* w, float eps,
                     float prescale, const float* add, float gate, void* out, int ldo) {
  if (rows <= 0) return cudaSuccess;
  cudaError_t e = cudaSuccess;
  FM_DISPATCH_T(dtype, (e = launch_k(L, rms_rows_kernel<T>, dim3(rows), dim3(256), 0, acc, width, w, eps, prescale,
                                     add, gate, static_cast<T*>(out), ldo)));
  return e;
}

cudaError_t gelu_rows(const Launch& L, int dtype, float* acc, int64_t n, void* out) {
  if (n <= 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, static_cast<int64_t>(L.num_sms) * 16));
  cudaError_t e = cudaSuccess;
  FM_DISPATCH_T(dtype, (e = launch_k(L, gelu_kernel<T>, dim3(blocks), dim3(256), 0, acc, n, static_cast<T*>(out))));
  return e;
}

cudaError_t gather_rows(const Launch& L, int dtype, const void* table, int64_t nrows, int width, const int64_t* ids,
                        int n, void* out) {
  if (n <= 0) return cudaSuccess;
  cudaError_t e = cudaSuccess;
  FM_DISPATCH_T(dtype, (e = launch_k(L, gather_rows_kernel<T>, dim3(n), dim3(256), 0, static_cast<const T*>(table),
                                     nrows, width, ids, static_cast<T*>(out), L.dev_err)));
  return e;
}

cudaError_t draft_noise(const Launch& L, int dtype, const uint64_t* seeds, const int32_t* anchor_pos, int bs, int K,
                        int H, void* out) {
  const int64_t total = static_cast<int64_t>(bs) * K * ((H + 3) / 4);
  if (total <= 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(L.num_sms) * 16));
  cudaError_t e = cudaSuccess;
  FM_DISPATCH_T(dtype, (e = launch_k(L, draft_noise_kernel<T>, dim3(blocks), dim3(256), 0, seeds, anchor_pos, K, H,
                                     total, static_cast<T*>(out))));
  return e;
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
