// The verify tree of a multi-candidate draft (flashmap/sglang/tree.py, build_tree_abi):
// per request, N candidate blocks of K tokens drafted after the anchor become a trie
// (a node per distinct prefix), cut to the width - 1 nodes with the most votes, and
// listed in EAGLE's encoding: tokens and ids parent * width + number.
//
// One CTA per request, everything in shared memory (N * K <= kTreeMaxNodes):
//   lcp[i][j]    the length of the common prefix of candidates i and j;
//   node (i, d)  the prefix c_i[0..d]; its votes are #{j : lcp[i][j] > d}, its
//                representative the lowest such j; it is "real" (stands for its trie
//                node) when that is i itself;
//   key          votes, then shallower, then lower candidate, packed so that larger
//                is better and real nodes never tie; a node is kept when fewer than
//                width - 1 real nodes have a larger key, and numbered by
//                (depth, candidate) among the kept.

#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace fm {
namespace {

constexpr int kTreeThreads = 256;

__global__ void __launch_bounds__(kTreeThreads) build_tree_kernel(const int64_t* __restrict__ cand, int N, int K,
                                                                  int width, int64_t* __restrict__ tokens,
                                                                  int64_t* __restrict__ ids,
                                                                  int64_t* __restrict__ stats) {
  __shared__ int64_t c[kTreeMaxNodes];
  __shared__ uint8_t lcp[kTreeMaxCandidates * kTreeMaxCandidates];
  __shared__ int key[kTreeMaxNodes], first[kTreeMaxNodes], number[kTreeMaxNodes];
  __shared__ uint8_t kept[kTreeMaxNodes];
  __shared__ int s_real, s_distinct, s_kept, s_first_slot;
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, t = threadIdx.x;
  const int nk = N * K, m = width - 1;
  const int64_t* cb = cand + static_cast<int64_t>(b) * nk;
  for (int i = t; i < nk; i += blockDim.x) c[i] = LDCG(cb + i);
  if (t == 0) s_real = s_distinct = s_kept = 0, s_first_slot = -1;
  __syncthreads();
  for (int p = t; p < N * N; p += blockDim.x) {
    const int i = p / N, j = p - i * N;
    int l = 0;
    while (l < K && c[i * K + l] == c[j * K + l]) ++l;
    lcp[p] = static_cast<uint8_t>(l);
  }
  __syncthreads();
  for (int u = t; u < nk; u += blockDim.x) {  // node u = (candidate i, depth d)
    const int i = u / K, d = u - i * K;
    int votes = 0, f = N;
    for (int j = 0; j < N; ++j)
      if (lcp[i * N + j] > d) {
        ++votes;
        f = min(f, j);
      }
    first[u] = f;
    const bool real = f == i;
    key[u] = real ? votes * nk + (K - 1 - d) * N + (N - 1 - i) : -1;
    if (real) atomicAdd(&s_real, 1);
    if (real && d == K - 1) atomicAdd(&s_distinct, 1);
  }
  __syncthreads();
  // kept: fewer than m real nodes rank above it
  for (int u = t; u < nk; u += blockDim.x) {
    number[u] = 0;
    kept[u] = 0;
    if (key[u] < 0) continue;
    int above = 0;
    for (int v = 0; v < nk; ++v) above += key[v] > key[u];
    if (above < m) {
      kept[u] = 1;
      atomicAdd(&s_kept, 1);
    }
  }
  __syncthreads();
  // number: 1 + the kept nodes listed before it (shallower, or as deep with a lower candidate)
  for (int u = t; u < nk; u += blockDim.x) {
    if (!kept[u]) continue;
    const int i = u / K, d = u - i * K;
    int before = 0;
    for (int v = 0; v < nk; ++v) {
      const int iv = v / K, dv = v - iv * K;
      before += kept[v] && (dv < d || (dv == d && iv < i));
    }
    number[u] = before + 1;
  }
  __syncthreads();
  const int64_t base = static_cast<int64_t>(b) * m;
  for (int u = t; u < nk; u += blockDim.x) {
    const int q = number[u];
    if (q == 0) continue;
    const int i = u / K, d = u - i * K;
    const int parent = d == 0 ? 0 : number[first[i * K + d - 1] * K + d - 1];
    tokens[base + q - 1] = c[u];
    ids[base + q - 1] = static_cast<int64_t>(parent) * width + q;
    if (q == 1) s_first_slot = u;
  }
  __syncthreads();
  for (int q = s_kept + 1 + t; q <= m; q += blockDim.x) {  // padding: the first node under the root
    tokens[base + q - 1] = c[s_first_slot];
    ids[base + q - 1] = q;
  }
  if (t == 0) {
    stats[2 * b] = s_real;
    stats[2 * b + 1] = s_distinct;
  }
}

}  // namespace

cudaError_t build_tree(const Launch& L, const int64_t* candidates, int bs, int N, int K, int width, int64_t* tokens,
                       int64_t* ids, int64_t* stats) {
  if (bs <= 0) return cudaSuccess;
  return launch_k(L, build_tree_kernel, dim3(bs), dim3(kTreeThreads), 0, candidates, N, K, width, tokens, ids,
                  stats);
}

}  // namespace fm
