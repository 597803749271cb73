// The folded-noise eigenbasis (flashmap/sglang/model.py, noise_basis and _folded_noise):
// E^T E = Q diag(lam) Q^T in float64, then the per-step constants of the folded path
//   variance = lam / H,  M = diag(sqrt lam) Q^T diag(w) W_x^T,  x_embed(u),
// with the eigenpairs listed by ascending lam and each eigenvector signed so that its
// entry of largest magnitude (the first such) is positive.
//
// The eigensolver is Hestenes' one-sided Jacobi method on a square root X of the
// gram (X^T X = E^T E; here X = L^T from the load-time Cholesky factor): plane
// rotations applied to column pairs of X drive its columns to mutual orthogonality;
// the same rotations accumulated into V (starting at I) give the eigenvectors, and the
// squared column norms the eigenvalues (Hestenes 1958; parallel ordering of Brent and
// Luk 1985). Here the columns are grouped in blocks of 4. Each round pairs every
// block with another by the round-robin (circle) schedule. A CTA takes the 8 columns
// of one block pair. It forms their 8 x 8 gram in one pass over the rows, runs one
// cyclic sweep of 2 x 2 rotations on that gram in shared memory, and applies the
// product R of the rotations to the 8 columns of X and of V in a second pass. A sweep
// is nb - 1 rounds (nb blocks). The sweeps stop when no column pair's cosine
// |x_a . x_b| / (|x_a| |x_b|) exceeds the tolerance.
//
// All arithmetic is float64. Load time only.

#include <algorithm>
#include <cmath>
#include <cstring>
#include <numeric>
#include <string>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace fm {
namespace {

constexpr int kJb = 4;          // columns per block
constexpr int kJw = 2 * kJb;    // columns per block pair
constexpr int kJg = kJw * (kJw + 1) / 2;  // distinct gram entries of a pair
constexpr int kJThreads = 256;

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Block pair k of round `round` (0 <= round < nb - 1) of the circle schedule over nb
// blocks (nb even): block nb - 1 stays put and meets `round`; the others pair up as
// round + k and round - k (mod nb - 1). Over nb - 1 rounds every pair meets once.
__device__ __forceinline__ void circle_pair(int nb, int round, int k, int& I, int& J) {
  const int m = nb - 1;
  if (k == 0) {
    I = m;
    J = round;
  } else {
    I = (round + k) % m;
    J = (round - k + m) % m;
  }
}

// X and V are n x n, column-major (column j at j * n). off_bits collects the largest
// pair cosine seen before rotating (a non-negative double, ordered as its bits).
__global__ void __launch_bounds__(kJThreads) jacobi_round_kernel(double* __restrict__ X, double* __restrict__ V,
                                                                 int n, int nb, int round, double tol,
                                                                 unsigned long long* off_bits) {
  __shared__ double red[kJThreads / 32][kJg];
  __shared__ double g[kJw][kJw + 1];
  __shared__ double R[kJw][kJw + 1];
  __shared__ int s_any;
  int I, J;
  circle_pair(nb, round, blockIdx.x, I, J);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int col[kJw];
#pragma unroll
  for (int a = 0; a < kJw; ++a) {
    const int c = a < kJb ? I * kJb + a : J * kJb + (a - kJb);
    col[a] = c < n ? c : -1;
  }
  // pass 1: the gram of the 8 columns (upper triangle, row-major packing)
  double acc[kJg];
#pragma unroll
  for (int q = 0; q < kJg; ++q) acc[q] = 0.0;
  for (int r = tid; r < n; r += blockDim.x) {
    double x[kJw];
#pragma unroll
    for (int a = 0; a < kJw; ++a) x[a] = col[a] >= 0 ? X[static_cast<int64_t>(col[a]) * n + r] : 0.0;
    int q = 0;
#pragma unroll
    for (int a = 0; a < kJw; ++a)
#pragma unroll
      for (int b = a; b < kJw; ++b, ++q) acc[q] = fma(x[a], x[b], acc[q]);
  }
#pragma unroll
  for (int q = 0; q < kJg; ++q) acc[q] = warp_sum_d(acc[q]);
  if (lane == 0)
#pragma unroll
    for (int q = 0; q < kJg; ++q) red[warp][q] = acc[q];
  __syncthreads();
  if (tid < kJg) {
    double sum = 0.0;
    for (int w = 0; w < kJThreads / 32; ++w) sum += red[w][tid];
    int a = 0, q = tid;
    while (q >= kJw - a) q -= kJw - a, ++a;
    const int b = a + q;
    g[a][b] = sum;
    g[b][a] = sum;
  }
  if (tid < kJw * kJw) R[tid / kJw][tid % kJw] = (tid / kJw == tid % kJw) ? 1.0 : 0.0;
  __syncthreads();
  if (warp == 0) {
    // the largest cosine among the pairs before rotating (zero columns excluded)
    double off = 0.0;
    for (int p = lane; p < kJw * kJw; p += 32) {
      const int a = p / kJw, b = p % kJw;
      if (a < b && col[a] >= 0 && col[b] >= 0 && g[a][a] > 0.0 && g[b][b] > 0.0)
        off = fmax(off, fabs(g[a][b]) / sqrt(g[a][a] * g[b][b]));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) off = fmax(off, __shfl_xor_sync(0xffffffffu, off, o));
    if (lane == 0) atomicMax(off_bits, static_cast<unsigned long long>(__double_as_longlong(off)));
    // one cyclic sweep of rotations on the 8 x 8 gram, accumulated into R
    int any = 0;
    for (int a = 0; a < kJw - 1; ++a) {
      for (int b = a + 1; b < kJw; ++b) {
        if (col[a] < 0 || col[b] < 0) continue;
        const double alpha = g[a][a], beta = g[b][b], gam = g[a][b];
        if (!(fabs(gam) > tol * sqrt(alpha * beta))) continue;
        // x_a' = c x_a - s x_b, x_b' = s x_a + c x_b with x_a' . x_b' = 0:
        // t = s / c the smaller root of t^2 + 2 zeta t - 1 = 0
        const double zeta = (beta - alpha) / (2.0 * gam);
        const double t = (zeta >= 0.0 ? 1.0 : -1.0) / (fabs(zeta) + sqrt(1.0 + zeta * zeta));
        const double c = 1.0 / sqrt(1.0 + t * t), s = c * t;
        any = 1;
        if (lane < kJw) {  // columns a, b of g and R
          const double gp = g[lane][a], gq = g[lane][b];
          g[lane][a] = c * gp - s * gq;
          g[lane][b] = s * gp + c * gq;
          const double rp = R[lane][a], rq = R[lane][b];
          R[lane][a] = c * rp - s * rq;
          R[lane][b] = s * rp + c * rq;
        }
        __syncwarp();
        if (lane < kJw) {  // rows a, b of g
          const double gp = g[a][lane], gq = g[b][lane];
          g[a][lane] = c * gp - s * gq;
          g[b][lane] = s * gp + c * gq;
        }
        __syncwarp();
      }
    }
    if (lane == 0) s_any = any;
  }
  __syncthreads();
  if (!s_any) return;
  // pass 2: the 8 columns of X and of V times R
  for (int mtx = 0; mtx < 2; ++mtx) {
    double* A = mtx == 0 ? X : V;
    for (int r = tid; r < n; r += blockDim.x) {
      double x[kJw];
#pragma unroll
      for (int a = 0; a < kJw; ++a) x[a] = col[a] >= 0 ? A[static_cast<int64_t>(col[a]) * n + r] : 0.0;
#pragma unroll
      for (int b = 0; b < kJw; ++b) {
        if (col[b] < 0) continue;
        double y = 0.0;
#pragma unroll
        for (int a = 0; a < kJw; ++a) y = fma(x[a], R[a][b], y);
        A[static_cast<int64_t>(col[b]) * n + r] = y;
      }
    }
  }
}

// Row-major lower factor L (upper triangle holding leftovers) -> X = L^T column-major:
// the same storage with the upper triangle zeroed.
__global__ void tril_kernel(double* A, int n) {
  const int64_t total = static_cast<int64_t>(n) * n;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / n, c = i - r * n;
    if (c > r) A[i] = 0.0;
  }
}

__global__ void eye_kernel(double* A, int n) {
  const int64_t total = static_cast<int64_t>(n) * n;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    A[i] = (i / n == i % n) ? 1.0 : 0.0;
}

// lam[j] = |x_j|^2; sign[j] = the sign of v_j's entry of largest magnitude (the
// first such). One CTA per column.
__global__ void __launch_bounds__(256) column_stats_kernel(const double* __restrict__ X, const double* __restrict__ V,
                                                           int n, double* __restrict__ lam, int* __restrict__ sign) {
  __shared__ double rs[8];
  __shared__ double rm[8];
  __shared__ int ri[8];
  const int j = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const double* x = X + static_cast<int64_t>(j) * n;
  const double* v = V + static_cast<int64_t>(j) * n;
  double ss = 0.0, best = -1.0;
  int bi = n;
  for (int r = tid; r < n; r += blockDim.x) {
    ss = fma(x[r], x[r], ss);
    const double m = fabs(v[r]);
    if (m > best) best = m, bi = r;  // rows ascend per thread: the first wins ties
  }
  ss = warp_sum_d(ss);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const double m2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    if (m2 > best || (m2 == best && i2 < bi)) best = m2, bi = i2;
  }
  if (lane == 0) rs[warp] = ss, rm[warp] = best, ri[warp] = bi;
  __syncthreads();
  if (tid == 0) {
    double s = 0.0, b = -1.0;
    int i = n;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
      s += rs[w];
      if (rm[w] > b || (rm[w] == b && ri[w] < i)) b = rm[w], i = ri[w];
    }
    lam[j] = s;
    sign[j] = (i < n && v[i] < 0.0) ? -1 : 1;
  }
}

// A[i][k] = sign_p sqrt(lam_p) v_p[k] w[k] (p = perm[i]): the rows of
// diag(sqrt lam) Q^T diag(w) in ascending order, float32, row-major.
__global__ void __launch_bounds__(256) assemble_kernel(const double* __restrict__ V, const double* __restrict__ lam,
                                                       const int* __restrict__ sign, const int* __restrict__ perm,
                                                       const float* __restrict__ w, int n, float* __restrict__ A) {
  const int i = blockIdx.x, p = perm[i];
  const double f = sign[p] * sqrt(fmax(lam[p], 0.0));
  const double* v = V + static_cast<int64_t>(p) * n;
  for (int k = threadIdx.x; k < n; k += blockDim.x)
    A[static_cast<int64_t>(i) * n + k] = static_cast<float>(f * v[k] * static_cast<double>(w[k]));
}

// out[d] = sum_k W[d][k] u[k] + b[d] (W, b in dtype; u float32), float64 sums; one warp per d.
__global__ void affine_kernel(const void* W, const void* b, int dtype, int D, int K, const float* __restrict__ u,
                              float* __restrict__ out) {
  const int d = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (d >= D) return;
  double s = 0.0;
  for (int k = lane; k < K; k += 32)
    s += static_cast<double>(load_as_f32(W, dtype, static_cast<int64_t>(d) * K + k)) * u[k];
  s = warp_sum_d(s);
  if (lane == 0) out[d] = static_cast<float>(s + load_as_f32(b, dtype, d));
}

// G = E^T E (H x H, float64, both triangles) with float64 products and sums: bf16 and
// float32 entries multiply exactly in float64, so G is the exact gram up to the
// rounding of its sums, as the pages form it (flashmap/sglang/model.py,
// _embedding_gram). One CTA per 64 x 64 tile on or above the diagonal; each thread
// holds a 4 x 4 block of it; E is staged 16 rows at a time.
constexpr int kGt = 64, kGk = 16;

__global__ void __launch_bounds__(256) gram_f64_kernel(const void* __restrict__ E, int dtype, int64_t V, int H,
                                                       double* __restrict__ G) {
  __shared__ double si[kGk][kGt + 1], sj[kGk][kGt + 1];
  // tile index -> (ti <= tj) over the upper triangle of tiles, row by row
  const int nt = (H + kGt - 1) / kGt;
  int ti = 0, rem = blockIdx.x;
  while (rem >= nt - ti) rem -= nt - ti, ++ti;
  const int tj = ti + rem;
  const int i0 = ti * kGt, j0 = tj * kGt;
  const int tid = threadIdx.x, tr = tid >> 4, tc = tid & 15;
  double acc[4][4] = {};
  for (int64_t v0 = 0; v0 < V; v0 += kGk) {
    for (int e = tid; e < kGk * kGt; e += blockDim.x) {
      const int kk = e / kGt, c = e - kk * kGt;
      const int64_t v = v0 + kk;
      const bool ok = v < V;
      si[kk][c] = ok && i0 + c < H ? static_cast<double>(load_as_f32(E, dtype, v * H + i0 + c)) : 0.0;
      sj[kk][c] = ok && j0 + c < H ? static_cast<double>(load_as_f32(E, dtype, v * H + j0 + c)) : 0.0;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kGk; ++kk) {
      double a[4], b[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) a[x] = si[kk][tr * 4 + x], b[x] = sj[kk][tc * 4 + x];
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = fma(a[x], b[y], acc[x][y]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < 4; ++y) {
      const int i = i0 + tr * 4 + x, j = j0 + tc * 4 + y;
      if (i < H && j < H) {
        G[static_cast<int64_t>(i) * H + j] = acc[x][y];
        G[static_cast<int64_t>(j) * H + i] = acc[x][y];
      }
    }
}

}  // namespace

cudaError_t gram_f64(cudaStream_t s, const void* E, int dtype, int64_t V, int H, double* G) {
  const int nt = (H + kGt - 1) / kGt;
  gram_f64_kernel<<<nt * (nt + 1) / 2, 256, 0, s>>>(E, dtype, V, H, G);
  return cudaGetLastError();
}

size_t folded_scratch_bytes(int n) {
  return static_cast<size_t>(n) * n * 8 + static_cast<size_t>(n) * (8 + 4 + 4) + 64;
}

cudaError_t folded_noise_constants(cudaStream_t s, double* X, int n, void* scratch, const float* noise_w,
                                   const void* xw, const void* xb, int dtype, int D, const float* u, void* proj,
                                   float* variance, float* xu, int* sweeps_out, std::string* err) {
  uint8_t* sc = static_cast<uint8_t*>(scratch);
  double* Vm = reinterpret_cast<double*>(sc);
  double* lam = reinterpret_cast<double*>(sc + static_cast<size_t>(n) * n * 8);
  int* sign = reinterpret_cast<int*>(lam + n);
  int* perm = sign + n;
  unsigned long long* off_bits = reinterpret_cast<unsigned long long*>(
      (reinterpret_cast<uintptr_t>(perm + n) + 15) & ~static_cast<uintptr_t>(15));
  cudaError_t e;
#define FM_EIG(call)               \
  do {                             \
    if ((e = (call)) != cudaSuccess) return e; \
  } while (0)
  tril_kernel<<<1024, 256, 0, s>>>(X, n);
  eye_kernel<<<1024, 256, 0, s>>>(Vm, n);
  FM_EIG(cudaGetLastError());
  const int nb = 2 * ((((n + kJb - 1) / kJb) + 1) / 2);
  // a pair cosine below this is round-off of the n-long dot products
  const double tol = 2e-15 * std::sqrt(static_cast<double>(n));
  int sweep = 0;
  double off = 1.0;
  for (; sweep < 60 && off > tol; ++sweep) {
    FM_EIG(cudaMemsetAsync(off_bits, 0, 8, s));
    for (int round = 0; round < nb - 1; ++round)
      jacobi_round_kernel<<<nb / 2, kJThreads, 0, s>>>(X, Vm, n, nb, round, tol, off_bits);
    FM_EIG(cudaGetLastError());
    unsigned long long bits = 0;
    FM_EIG(cudaMemcpyAsync(&bits, off_bits, 8, cudaMemcpyDeviceToHost, s));
    FM_EIG(cudaStreamSynchronize(s));
    std::memcpy(&off, &bits, 8);
    if (!(off == off)) break;  // NaN: stop, reported below
  }
  if (sweeps_out) *sweeps_out = sweep;
  if (!(off <= tol)) {
    if (err) *err = "folded noise: the Jacobi eigensolver did not converge (largest cosine " + std::to_string(off) + ")";
    return cudaErrorUnknown;
  }
  column_stats_kernel<<<n, 256, 0, s>>>(X, Vm, n, lam, sign);
  FM_EIG(cudaGetLastError());
  std::vector<double> hl(n);
  FM_EIG(cudaMemcpyAsync(hl.data(), lam, static_cast<size_t>(n) * 8, cudaMemcpyDeviceToHost, s));
  FM_EIG(cudaStreamSynchronize(s));
  std::vector<int> order(n);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return hl[a] < hl[b]; });
  std::vector<float> hv(n);
  for (int i = 0; i < n; ++i) hv[i] = static_cast<float>(std::max(hl[order[i]], 0.0) / n);
  FM_EIG(cudaMemcpyAsync(perm, order.data(), static_cast<size_t>(n) * 4, cudaMemcpyHostToDevice, s));
  FM_EIG(cudaMemcpyAsync(variance, hv.data(), static_cast<size_t>(n) * 4, cudaMemcpyHostToDevice, s));
  // A (float32, n x n) over X's storage, which is no longer needed
  float* A = reinterpret_cast<float*>(X);
  assemble_kernel<<<n, 256, 0, s>>>(Vm, lam, sign, perm, noise_w, n, A);
  FM_EIG(cudaGetLastError());
  // proj (D x n, row-major in dtype) = W_x A^T: proj[d][i] = sum_k W_x[d][k] A[i][k]
  FM_EIG(simt_gemm(s, D, n, n, xw, dtype, nullptr, n, 1, A, FLASHMAP_F32, 1, n, proj, dtype, n, 1));
  affine_kernel<<<(D + 7) / 8, 256, 0, s>>>(xw, xb, dtype, D, n, u, xu);
  FM_EIG(cudaGetLastError());
  FM_EIG(cudaStreamSynchronize(s));  // the host vectors above must outlive their copies
#undef FM_EIG
  return cudaSuccess;
}

}  // namespace fm
