// Drafting in several jumps (flashmap/modeling_flashmap.py, FlashMapDraftModel.draft,
// embed_state, mix_state; flashmap/vllm/model.py, _embed_state and the jump loop).
// The state is vocabulary-sized: per drafted row, V float32 values. Each jump s -> t
// reads it through the target's embedding E twice -- as the posterior
// softmax(state * s / max(1 - s, 1e-3)^2) and linearly -- and, before t = 1, moves it
// toward the DiT's full-vocabulary distribution:
//   state <- ((1 - t) state + (t - s) softmax(logits)) / (1 - s).
// Row kernels here: the state update fused with the next jump's posterior and the
// bf16 copies the embedding GEMM reads, and the mix of the two embeddings.

#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace fm {
namespace {

namespace cg = cooperative_groups;

constexpr int kPrepThreads = 512;
constexpr int kPrepMaxCluster = 8;  // portable cluster size
constexpr int kPrepMinChunk = 2048;  // vocabulary entries below which a row takes one CTA

// The row split of state_prep: C CTAs of a cluster, each holding `chunk` entries
// (a multiple of 4) of the row in shared memory.
struct PrepSplit {
  int C, chunk;
};

PrepSplit prep_split(int V) {
  const int C = std::max(1, std::min(kPrepMaxCluster, (V + kPrepMinChunk - 1) / kPrepMinChunk));
  const int chunk = ((V + C - 1) / C + 3) & ~3;
  return {C, chunk};
}

// (m, l) of a softmax over a union of parts: max and sum of exp(x - max).
__device__ __forceinline__ void ml_merge(float& m, float& l, float m2, float l2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;  // both parts empty
  l = l * expf(m - M) + l2 * expf(m2 - M);
  m = M;
}

__device__ __forceinline__ void warp_ml(float& m, float& l) {
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off), l2 = __shfl_xor_sync(0xffffffffu, l, off);
    ml_merge(m, l, m2, l2);
  }
}

// Merges every thread's (m, l) over the block, then over the cluster through each
// CTA's `slot` (a distinct slot per call: a peer may still be reading the last one).
__device__ float2 cluster_ml(float m, float l, float2* slot, float2* red, float2* bcast, cg::cluster_group& cl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  warp_ml(m, l);
  if (lane == 0) red[warp] = make_float2(m, l);
  __syncthreads();
  if (warp == 0) {
    const float2 p = lane < static_cast<int>(blockDim.x >> 5) ? red[lane] : make_float2(-INFINITY, 0.f);
    m = p.x, l = p.y;
    warp_ml(m, l);
    if (lane == 0) *slot = make_float2(m, l);
  }
  cl.sync();
  if (warp == 0) {
    const float2 p = lane < static_cast<int>(cl.num_blocks()) ? *cl.map_shared_rank(slot, lane)
                                                              : make_float2(-INFINITY, 0.f);
    m = p.x, l = p.y;
    warp_ml(m, l);
    if (lane == 0) *bcast = make_float2(m, l);
  }
  __syncthreads();
  return *bcast;
}

__device__ __forceinline__ float max4(float4 v) { return fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)); }

template <typename T>
__device__ __forceinline__ void store4(T* p, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&a);
  u.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// Row y of the state, split over the cluster's C CTAs (x = rank), each with its
// `chunk` entries in shared memory, so every entry is read and written once.
// upd: first apply the jump s -> t with the row's logits (+ bias), the softmax's
// max and sum merged over the cluster; then write the state as T (the linear read)
// and, when ev > 0, the posterior softmax(state * ev) as T (the posterior read).
template <typename T>
__global__ void __launch_bounds__(kPrepThreads) state_prep_kernel(float* __restrict__ state,
                                                                  float* __restrict__ logits,
                                                                  const float* __restrict__ bias, int V, int chunk,
                                                                  int upd, float s, float t, float ev,
                                                                  T* __restrict__ x_post, T* __restrict__ x_state,
                                                                  int64_t ld) {
  extern __shared__ float4 buf[];
  __shared__ float2 part[2], red[32], bcast;
  cg::cluster_group cl = cg::this_cluster();
  pdl_trigger();
  pdl_wait();
  const int64_t row = blockIdx.y;
  const int v0 = static_cast<int>(cl.block_rank()) * chunk;
  const int n4 = max(0, min(chunk, V - v0)) >> 2;
  float4* st4 = reinterpret_cast<float4*>(state + row * V + v0);
  if (upd) {
    const float4* lg4 = reinterpret_cast<const float4*>(logits + row * V + v0);  // the GEMM's output
    const float4* b4 = reinterpret_cast<const float4*>(bias + v0);
    float m = -INFINITY, l = 0.f;
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
      const float4 g = __ldcg(lg4 + i), b = b4[i];
      const float4 x = make_float4(g.x + b.x, g.y + b.y, g.z + b.z, g.w + b.w);
      buf[i] = x;
      m = fmaxf(m, max4(x));
    }
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
      const float4 x = buf[i];
      l += expf(x.x - m) + expf(x.y - m) + expf(x.z - m) + expf(x.w - m);
    }
    const float2 tot = cluster_ml(m, l, &part[0], red, &bcast, cl);
    const float inv_l = 1.f / tot.y, keep = 1.f - t, move = (t - s) * inv_l, inv_1s = 1.f / (1.f - s);
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
      const float4 x = buf[i], o = __ldcg(st4 + i);
      const float4 y = make_float4((keep * o.x + move * expf(x.x - tot.x)) * inv_1s,
                                   (keep * o.y + move * expf(x.y - tot.x)) * inv_1s,
                                   (keep * o.z + move * expf(x.z - tot.x)) * inv_1s,
                                   (keep * o.w + move * expf(x.w - tot.x)) * inv_1s);
      st4[i] = y;
      buf[i] = y;
    }
  } else {
    for (int i = threadIdx.x; i < n4; i += blockDim.x) buf[i] = __ldcg(st4 + i);
  }
  // each thread reads back only the entries it wrote: no block barrier needed
  T* xs = x_state + row * ld + v0;
  float m2 = -INFINITY;
  for (int i = threadIdx.x; i < n4; i += blockDim.x) {
    const float4 x = buf[i];
    store4<T>(xs + 4 * i, x);
    m2 = fmaxf(m2, max4(x) * ev);  // ev > 0 whenever it is used
  }
  if (ev > 0.f) {
    float l2 = 0.f;
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
      const float4 x = buf[i];
      l2 += expf(x.x * ev - m2) + expf(x.y * ev - m2) + expf(x.z * ev - m2) + expf(x.w * ev - m2);
    }
    const float2 tot = cluster_ml(m2, l2, &part[1], red, &bcast, cl);
    const float inv = 1.f / tot.y;
    T* xp = x_post + row * ld + v0;
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
      const float4 x = buf[i];
      store4<T>(xp + 4 * i, make_float4(expf(x.x * ev - tot.x) * inv, expf(x.y * ev - tot.x) * inv,
                                        expf(x.z * ev - tot.x) * inv, expf(x.w * ev - tot.x) * inv));
    }
  }
  cl.sync();  // no CTA leaves while a peer may still read its partials
}

// The DiT input of a jump, per row (one CTA): state_norm(emb_post) (or the uniform
// constant u when the posterior is uniform) + gate * noise_norm(emb_state), from the
// float32 embeddings the GEMM through E^T wrote.
template <typename T>
__global__ void __launch_bounds__(256) mix_state_kernel(float* __restrict__ emb_post, float* __restrict__ emb_state,
                                                        int H, const float* __restrict__ u,
                                                        const float* __restrict__ state_w,
                                                        const float* __restrict__ noise_w, float eps, float gate,
                                                        T* __restrict__ out) {
  __shared__ float red[32];
  pdl_trigger();
  pdl_wait();
  const int64_t row = blockIdx.x;
  const float* ep = emb_post ? emb_post + row * H : nullptr;
  const float* es = emb_state + row * H;
  float ss_p = 0.f, ss_s = 0.f;
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    const float a = LDCG(es + h);
    ss_s = fmaf(a, a, ss_s);
    if (ep) {
      const float b = LDCG(ep + h);
      ss_p = fmaf(b, b, ss_p);
    }
  }
  ss_s = block_sum(ss_s, red);
  if (ep) ss_p = block_sum(ss_p, red);
  const float rs = rsqrtf(ss_s / H + eps), rp = ep ? rsqrtf(ss_p / H + eps) : 0.f;
  T* o = out + row * H;
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    const float post = ep ? LDCG(ep + h) * rp * state_w[h] : u[h];
    const float noise = LDCG(es + h) * rs * noise_w[h];
    o[h] = from_f32<T>(post + gate * noise);
  }
}

// out[c][r] = in[r][c] for a rows x cols matrix of 2- or 4-byte elements (load time).
template <typename T>
__global__ void transpose_kernel(const T* __restrict__ in, int64_t rows, int64_t cols, T* __restrict__ out) {
  __shared__ T tile[32][33];
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 32, c0 = static_cast<int64_t>(blockIdx.x) * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int64_t r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[i][threadIdx.x] = in[r * cols + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int64_t c = c0 + i, r = r0 + threadIdx.x;
    if (r < rows && c < cols) out[c * rows + r] = tile[threadIdx.x][i];
  }
}

#define FM_DISPATCH_TJ(dtype, ...)  \
  do {                              \
    if ((dtype) == FLASHMAP_F32) {  \
      using T = float;              \
      __VA_ARGS__;                  \
    } else {                        \
      using T = __nv_bfloat16;      \
      __VA_ARGS__;                  \
    }                               \
  } while (0)

}  // namespace

cudaError_t state_prep(const Launch& L, int dtype, float* state, float* logits, const float* bias, int rows,
                       int V, bool upd, float s, float t, float ev, void* x_post, void* x_state, int64_t ld) {
  if (rows <= 0) return cudaSuccess;
  const PrepSplit sp = prep_split(V);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sp.C, rows);
  cfg.blockDim = dim3(kPrepThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(sp.chunk) * 4;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = sp.C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaSuccess;
  FM_DISPATCH_TJ(dtype, (e = cudaLaunchKernelEx(&cfg, state_prep_kernel<T>, state, logits, bias, V, sp.chunk,
                                                upd ? 1 : 0, s, t, ev, static_cast<T*>(x_post),
                                                static_cast<T*>(x_state), ld)));
  return e;
}

size_t state_prep_smem(int V) { return static_cast<size_t>(prep_split(V).chunk) * 4; }

cudaError_t jumps_prepare(int V) {
  const int smem = static_cast<int>(state_prep_smem(V));
  cudaError_t e = cudaFuncSetAttribute(state_prep_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(state_prep_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  return e;
}

cudaError_t mix_state(const Launch& L, int dtype, float* emb_post, float* emb_state, int rows, int H, const float* u,
                      const float* state_w, const float* noise_w, float eps, float gate, void* out) {
  if (rows <= 0) return cudaSuccess;
  cudaError_t e = cudaSuccess;
  FM_DISPATCH_TJ(dtype, (e = launch_k(L, mix_state_kernel<T>, dim3(rows), dim3(256), 0, emb_post, emb_state, H, u,
                                      state_w, noise_w, eps, gate, static_cast<T*>(out))));
  return e;
}

cudaError_t transpose(cudaStream_t s, int dtype, const void* in, int64_t rows, int64_t cols, void* out) {
  dim3 grid(static_cast<unsigned>((cols + 31) / 32), static_cast<unsigned>((rows + 31) / 32));
  if (dtype == FLASHMAP_F32)
    transpose_kernel<float><<<grid, dim3(32, 8), 0, s>>>(static_cast<const float*>(in), rows, cols,
                                                         static_cast<float*>(out));
  else
    transpose_kernel<__nv_bfloat16><<<grid, dim3(32, 8), 0, s>>>(static_cast<const __nv_bfloat16*>(in), rows, cols,
                                                                 static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace fm
