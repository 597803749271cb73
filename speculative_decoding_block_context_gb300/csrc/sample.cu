// Whole-block sampling (flashmap/sglang/sampler.py, FlashMapDraftSampler, fused
// variant): a few CTAs per block row take the row's argmax (greedy rows) or its
// Gumbel-max at the request's temperature with Philox noise drawn in the kernel, and
// map the drafted index to a token id; and the optional full-vocabulary logits with
// -inf outside the draft vocabulary (flashmap/sglang/sampler.py, _FullLogits).

#include <algorithm>
#include <climits>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "philox.cuh"

namespace fm {
namespace {

__device__ __forceinline__ bool better(float v, int j, float bv, int bj) { return v > bv || (v == bv && j < bj); }

// A float's bits mapped so that unsigned order is float order.
__device__ __forceinline__ uint32_t orderable(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Row r is scanned by `splits` CTAs (blockIdx.y), each over a contiguous slice of the
// draft vocabulary. Each slice's best (value, lowest index) is merged into keys[r] by
// one 64-bit atomicMax on (orderable(value) << 32 | ~index), so larger values win and
// equal values go to the lowest index. The CTA that finishes a row last (a counter,
// no waiting) writes the token and clears the row's key and counter for the next call.
template <bool kVec>
__global__ void __launch_bounds__(256) sample_kernel(const float* __restrict__ logits, int Vd, int K,
                                                     const float* __restrict__ temps,
                                                     const uint8_t* __restrict__ greedy,
                                                     const uint64_t* __restrict__ seeds,
                                                     const int32_t* __restrict__ anchor_pos, uint32_t step,
                                                     const int64_t* __restrict__ hot, int64_t* __restrict__ tokens,
                                                     unsigned long long* keys, unsigned* counters) {
  __shared__ float rv[32];
  __shared__ int rj[32];
  __shared__ float s_T;
  __shared__ int s_pos, s_greedy;
  __shared__ uint64_t s_seed;
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x, b = row / K, k = row - b * K;
  const int splits = gridDim.y, sp = blockIdx.y;
  // the request's scalars, loaded once per CTA (every CTA of a request reads the same
  // few bytes; per-warp loads would queue on one L2 sector)
  if (threadIdx.x == 0) {
    s_T = LDCG(temps + b);
    s_greedy = LDCG(greedy + b);
    s_seed = LDCG(seeds + b);
    s_pos = LDCG(anchor_pos + b);
  }
  const float* lr = logits + static_cast<int64_t>(row) * Vd;
  const int n4 = (Vd + 3) >> 2;
  const int j4_0 = static_cast<int>(static_cast<int64_t>(n4) * sp / splits);
  const int j4_1 = static_cast<int>(static_cast<int64_t>(n4) * (sp + 1) / splits);
  // kVec: every row starts 16-byte aligned and holds whole float4 groups
  float4 lv = make_float4(0.f, 0.f, 0.f, 0.f);
  if (kVec && j4_0 + static_cast<int>(threadIdx.x) < j4_1)
    lv = LDCG(reinterpret_cast<const float4*>(lr) + j4_0 + threadIdx.x);
  __syncthreads();
  const float T = s_T;
  const bool argmax_only = s_greedy != 0 || !(T > 0.f);
  const uint64_t seed = s_seed;
  const uint32_t pos = static_cast<uint32_t>(s_pos + 1 + k);
  float bv = -INFINITY;
  int bj = INT_MAX;
  for (int j4 = j4_0 + threadIdx.x; j4 < j4_1; j4 += blockDim.x) {
    float ls[4];
    if constexpr (kVec) {
      ls[0] = lv.x, ls[1] = lv.y, ls[2] = lv.z, ls[3] = lv.w;
      if (j4 + static_cast<int>(blockDim.x) < j4_1) lv = LDCG(reinterpret_cast<const float4*>(lr) + j4 + blockDim.x);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) ls[e] = 4 * j4 + e < Vd ? LDCG(lr + 4 * j4 + e) : -INFINITY;
    }
    uint4 w = make_uint4(0, 0, 0, 0);
    if (!argmax_only) w = philox_seeded(seed, static_cast<uint32_t>(j4), pos, kDomainGumbel, step);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = 4 * j4 + e;
      if (!kVec && j >= Vd) break;
      const float l = ls[e];
      const float v = argmax_only ? l : __fdiv_rn(l, T) + gumbel_of_word(ws[e]);
      if (better(v, j, bv, bj)) {
        bv = v;
        bj = j;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
    if (better(ov, oj, bv, bj)) {
      bv = ov;
      bj = oj;
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    rv[warp] = bv;
    rj[warp] = bj;
  }
  __syncthreads();
  if (warp != 0) return;
  const int nw = blockDim.x >> 5;
  bv = lane < nw ? rv[lane] : -INFINITY;
  bj = lane < nw ? rj[lane] : INT_MAX;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
    if (better(ov, oj, bv, bj)) {
      bv = ov;
      bj = oj;
    }
  }
  if (lane != 0) return;
  const unsigned long long key = (static_cast<unsigned long long>(orderable(bv)) << 32) |
                                 static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(bj));
  atomicMax(keys + row, key);
  __threadfence();
  if (atomicAdd(counters + row, 1u) == static_cast<unsigned>(splits - 1)) {
    __threadfence();
    const unsigned long long best = atomicExch(keys + row, 0ull);
    counters[row] = 0;
    uint32_t j = 0xFFFFFFFFu - static_cast<uint32_t>(best & 0xFFFFFFFFull);
    if (j >= static_cast<uint32_t>(Vd)) j = 0;  // every value NaN
    tokens[row] = hot ? hot[j] : static_cast<int64_t>(j);
  }
}

__global__ void full_scatter_kernel(const float* __restrict__ logits, int Vd, const int32_t* __restrict__ inv,
                                    int V, float* __restrict__ full) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.y;
  const float* lr = logits + static_cast<int64_t>(row) * Vd;
  float* fr = full + static_cast<int64_t>(row) * V;
  for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < V; v += gridDim.x * blockDim.x) {
    const int j = inv[v];
    fr[v] = j >= 0 ? LDCG(lr + j) : -INFINITY;
  }
}

// The same with V a multiple of 4 and 16-byte aligned rows: each thread maps 4
// consecutive vocabulary entries (one int4 of the inverse map, read once) for
// kScatterRows rows (one float4 streaming store per row: the full logits are written
// once and not re-read here).
constexpr int kScatterRows = 8;
__global__ void __launch_bounds__(256) full_scatter4_kernel(const float* __restrict__ logits, int Vd,
                                                            const int32_t* __restrict__ inv, int V, int rows,
                                                            float* __restrict__ full) {
  pdl_trigger();
  const int v4 = blockIdx.x * blockDim.x + threadIdx.x;  // group of 4 entries
  const bool live = v4 * 4 < V;
  const int4 j = live ? *reinterpret_cast<const int4*>(inv + 4 * v4) : make_int4(-1, -1, -1, -1);
  pdl_wait();
  if (!live) return;
  const int r0 = blockIdx.y * kScatterRows, r1 = min(rows, r0 + kScatterRows);
  for (int r = r0; r < r1; ++r) {
    const float* lr = logits + static_cast<int64_t>(r) * Vd;
    float4 o;
    o.x = j.x >= 0 ? LDCG(lr + j.x) : -INFINITY;
    o.y = j.y >= 0 ? LDCG(lr + j.y) : -INFINITY;
    o.z = j.z >= 0 ? LDCG(lr + j.z) : -INFINITY;
    o.w = j.w >= 0 ? LDCG(lr + j.w) : -INFINITY;
    __stcs(reinterpret_cast<float4*>(full + static_cast<int64_t>(r) * V) + v4, o);
  }
}

}  // namespace

// Merge slots of the sampler for callers that cannot allocate device memory: one
// 8-byte key and one 4-byte counter per row, kStaticSampleRows rows, in a file-scope
// array that every GPU loading the library holds until the process exits.
static __device__ __align__(256) unsigned char g_sample_scratch[kStaticSampleRows * 12];

// The device address of g_sample_scratch on the current device. The host-side name
// of the array is only a stand-in: the address comes from cudaGetSymbolAddress,
// looked up once per device (with that device current) and cached.
cudaError_t static_sample_scratch(void** out) {
  static std::mutex mu;
  static void* cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_sample_scratch);
    if (e != cudaSuccess) return e;
    cache[dev] = p;
  }
  *out = cache[dev];
  return cudaSuccess;
}

// CTAs per row: up to one per 2048 draft-vocabulary entries, and no more than keep
// about 16 CTAs per SM in all (a few rows are split widely; thousands of rows are not,
// where one CTA per row already fills the GPU and the extra CTAs cost more to schedule
// than they save).
int sample_splits(int Vd, int rows, int num_sms) {
  const int by_vocab = std::max(1, std::min(32, (Vd + 2047) / 2048));
  const int by_grid = std::max(1, (16 * num_sms + rows - 1) / rows);
  return std::min(by_vocab, by_grid);
}

cudaError_t sample_rows(const Launch& L, const float* logits, int rows, int Vd, int K, const float* temps,
                        const uint8_t* greedy, const uint64_t* seeds, const int32_t* anchor_pos, uint32_t step,
                        const int64_t* hot, int64_t* tokens, unsigned long long* keys, unsigned* counters) {
  if (rows <= 0) return cudaSuccess;
  const bool vec = Vd % 4 == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0;
  return launch_k(L, vec ? sample_kernel<true> : sample_kernel<false>, dim3(rows, sample_splits(Vd, rows, L.num_sms)), dim3(256), 0,
                  logits, Vd, K, temps, greedy, seeds, anchor_pos, step, hot, tokens, keys, counters);
}

cudaError_t full_scatter(const Launch& L, const float* logits, int rows, int Vd, const int32_t* inv, int V,
                         float* full) {
  if (rows <= 0) return cudaSuccess;
  if (V % 4 == 0 && (reinterpret_cast<uintptr_t>(full) & 15) == 0 && (reinterpret_cast<uintptr_t>(inv) & 15) == 0) {
    dim3 grid((V / 4 + 255) / 256, (rows + kScatterRows - 1) / kScatterRows);
    return launch_k(L, full_scatter4_kernel, grid, dim3(256), 0, logits, Vd, inv, V, rows, full);
  }
  dim3 grid(std::min((V + 255) / 256, 64), rows);
  return launch_k(L, full_scatter_kernel, grid, dim3(256), 0, logits, Vd, inv, V, full);
}

}  // namespace fm
