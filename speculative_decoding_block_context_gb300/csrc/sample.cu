// Whole-block sampling (flashmap/sglang/sampler.py, FlashMapDraftSampler, fused
// variant): one CTA per block row takes the row's argmax (greedy rows) or its
// Gumbel-max at the request's temperature with Philox noise drawn in the kernel, and
// maps the drafted index to a token id; and the optional full-vocabulary logits with
// -inf outside the draft vocabulary (flashmap/sglang/sampler.py, _FullLogits).

#include <climits>

#include "common.cuh"
#include "internal.h"
#include "philox.cuh"

namespace fm {
namespace {

__device__ __forceinline__ bool better(float v, int j, float bv, int bj) { return v > bv || (v == bv && j < bj); }

__global__ void __launch_bounds__(256) sample_kernel(const float* __restrict__ logits, int Vd, int K,
                                                     const float* __restrict__ temps,
                                                     const uint8_t* __restrict__ greedy,
                                                     const uint64_t* __restrict__ seeds,
                                                     const int32_t* __restrict__ anchor_pos, uint32_t step,
                                                     const int64_t* __restrict__ hot, int64_t* __restrict__ tokens) {
  __shared__ float rv[32];
  __shared__ int rj[32];
  const int row = blockIdx.x, b = row / K, k = row - b * K;
  const float T = temps[b];
  const bool argmax_only = greedy[b] != 0 || !(T > 0.f);
  const uint64_t seed = seeds[b];
  const uint32_t pos = static_cast<uint32_t>(anchor_pos[b] + 1 + k);
  const float* lr = logits + static_cast<int64_t>(row) * Vd;
  float bv = -INFINITY;
  int bj = INT_MAX;
  const int n4 = (Vd + 3) >> 2;
  for (int j4 = threadIdx.x; j4 < n4; j4 += blockDim.x) {
    uint4 w = make_uint4(0, 0, 0, 0);
    if (!argmax_only) w = philox_seeded(seed, static_cast<uint32_t>(j4), pos, kDomainGumbel, step);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = 4 * j4 + e;
      if (j >= Vd) break;
      const float l = lr[j];
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
  if (warp == 0) {
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
    if (lane == 0) {
      if (bj == INT_MAX) bj = 0;  // every value NaN
      tokens[row] = hot ? hot[bj] : bj;
    }
  }
}

__global__ void full_scatter_kernel(const float* __restrict__ logits, int Vd, const int32_t* __restrict__ inv,
                                    int V, float* __restrict__ full) {
  const int row = blockIdx.y;
  const float* lr = logits + static_cast<int64_t>(row) * Vd;
  float* fr = full + static_cast<int64_t>(row) * V;
  for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < V; v += gridDim.x * blockDim.x) {
    const int j = inv[v];
    fr[v] = j >= 0 ? lr[j] : -INFINITY;
  }
}

}  // namespace

cudaError_t sample_rows(const Launch& L, const float* logits, int rows, int Vd, int K, const float* temps,
                        const uint8_t* greedy, const uint64_t* seeds, const int32_t* anchor_pos, uint32_t step,
                        const int64_t* hot, int64_t* tokens) {
  if (rows <= 0) return cudaSuccess;
  sample_kernel<<<rows, 256, 0, L.stream>>>(logits, Vd, K, temps, greedy, seeds, anchor_pos, step, hot, tokens);
  return cudaGetLastError();
}

cudaError_t full_scatter(const Launch& L, const float* logits, int rows, int Vd, const int32_t* inv, int V,
                         float* full) {
  if (rows <= 0) return cudaSuccess;
  dim3 grid(std::min((V + 255) / 256, 64), rows);
  full_scatter_kernel<<<grid, 256, 0, L.stream>>>(logits, Vd, inv, V, full);
  return cudaGetLastError();
}

}  // namespace fm
