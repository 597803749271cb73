// Load-time precompute (flashmap/sglang/model.py, _jump_constants / _embedding_gram /
// _fold_lm_head; flashmap/modeling_flashmap.py, time_conditioning / target_constants).
// None of this runs per step.

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace fm {
namespace {

__device__ __forceinline__ double silu_d(double x) { return x / (1.0 + exp(-x)); }

__global__ void to_f32_kernel(const void* src, int dtype, int64_t n, float* dst) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    dst[i] = load_as_f32(src, dtype, i);
}

__global__ void mul_vec_kernel(const float* a, const float* b, float* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = a[i] * b[i];
}

// cond = time_embed(s) + jump_embed(t) (modeling_flashmap.py, FlashMapTimeEmbedding):
// sinusoidal features of t * time_scale, freqs exp(-ln(1e4) i / half), [cos, sin],
// then linear_1 -> SiLU -> linear_2. One block; float64.
__global__ void time_cond_kernel(TimeCondArgs a, double* cond) {
  extern __shared__ double sh[];
  double* emb = sh;               // [Te]
  double* hid = emb + a.Te;       // [C]
  const int half = a.Te / 2;
  for (int i = threadIdx.x; i < a.C; i += blockDim.x) cond[i] = 0.0;
  __syncthreads();
  for (int which = 0; which < 2; ++which) {
    const double t = which == 0 ? a.s : a.t;
    const void* l1w = which == 0 ? a.te_l1_w : a.je_l1_w;
    const void* l1b = which == 0 ? a.te_l1_b : a.je_l1_b;
    const void* l2w = which == 0 ? a.te_l2_w : a.je_l2_w;
    const void* l2b = which == 0 ? a.te_l2_b : a.je_l2_b;
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
      const double f = exp(-log(10000.0) * static_cast<double>(i) / half);
      const double arg = t * a.time_scale * f;
      emb[i] = cos(arg);
      emb[half + i] = sin(arg);
    }
    for (int i = 2 * half + threadIdx.x; i < a.Te; i += blockDim.x) emb[i] = 0.0;
    __syncthreads();
    for (int j = threadIdx.x; j < a.C; j += blockDim.x) {
      double acc = load_as_f32(l1b, a.dtype, j);
      for (int i = 0; i < 2 * half; ++i) acc += load_as_f32(l1w, a.dtype, static_cast<int64_t>(j) * a.Te + i) * emb[i];
      hid[j] = silu_d(acc);
    }
    __syncthreads();
    for (int j = threadIdx.x; j < a.C; j += blockDim.x) {
      double acc = load_as_f32(l2b, a.dtype, j);
      for (int i = 0; i < a.C; ++i) acc += load_as_f32(l2w, a.dtype, static_cast<int64_t>(j) * a.C + i) * hid[i];
      cond[j] += acc;
    }
    __syncthreads();
  }
}

// AdaLN modulation linear(SiLU(cond)) -> (1 + scale, shift, gate), one warp per output.
__global__ void adaln_kernel(const void* w, const void* b, int dtype, int C, int D, const double* cond, float* s1,
                             float* sh, float* gate) {
  const int j = static_cast<int>((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (j >= 3 * D) return;
  double acc = 0.0;
  for (int c = lane; c < C; c += 32) acc += load_as_f32(w, dtype, static_cast<int64_t>(j) * C + c) * silu_d(cond[c]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane) return;
  acc += load_as_f32(b, dtype, j);
  if (j < D)
    s1[j] = static_cast<float>(1.0 + acc);
  else if (j < 2 * D)
    sh[j - D] = static_cast<float>(acc);
  else if (gate)
    gate[j - 2 * D] = static_cast<float>(acc);
}

constexpr int kColsumRows = 2048;

// Column sums of E in float64 over blocks of rows: out[block][col] (summed in block
// order by uniform_kernel, so the result does not depend on scheduling).
__global__ void colsum_kernel(const void* E, int dtype, int64_t V, int H, int rows_per_block, double* out) {
  const int col = blockIdx.x * blockDim.x + threadIdx.x;
  if (col >= H) return;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_block;
  const int64_t r1 = r0 + rows_per_block < V ? r0 + rows_per_block : V;
  double acc = 0.0;
  for (int64_t r = r0; r < r1; ++r) acc += load_as_f32(E, dtype, r * H + col);
  out[static_cast<int64_t>(blockIdx.y) * H + col] = acc;
}

// u = state_norm(colsum / V): RMSNorm with weight w (float32 out), colsum the column
// sums of `blocks` row blocks, added in block order first. One block.
__global__ void uniform_kernel(double* colsum, int blocks, int64_t V, int H, const float* w, float eps, float* u) {
  __shared__ double red[32];
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    double c = colsum[i];
    for (int b = 1; b < blocks; ++b) c += colsum[static_cast<int64_t>(b) * H + i];
    colsum[i] = c;
  }
  double s = 0.0;
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    const double m = colsum[i] / static_cast<double>(V);
    s += m * m;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    double t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const double r = 1.0 / sqrt(red[0] / H + static_cast<double>(eps));
  for (int i = threadIdx.x; i < H; i += blockDim.x) u[i] = static_cast<float>(colsum[i] / static_cast<double>(V) * r * w[i]);
}

// ------------------------------------------------------------------ float64 blocked Cholesky (right-looking)

constexpr int NB = 32;

__global__ void potrf_diag_kernel(double* A, int n, int j0, int nb, unsigned* err) {
  __shared__ double a[NB][NB + 1];
  const int tid = threadIdx.x;
  for (int i = tid; i < nb * nb; i += blockDim.x) {
    const int r = i / nb, c = i - r * nb;
    a[r][c] = A[static_cast<int64_t>(j0 + r) * n + j0 + c];
  }
  __syncthreads();
  for (int k = 0; k < nb; ++k) {
    if (tid == 0) {
      double d = a[k][k];
      if (!(d > 0.0)) {
        set_dev_error(err, FLASHMAP_DEVERR_NUMERIC);
        d = 1e-300;
      }
      a[k][k] = sqrt(d);
    }
    __syncthreads();
    for (int i = k + 1 + tid; i < nb; i += blockDim.x) a[i][k] /= a[k][k];
    __syncthreads();
    for (int i = tid; i < nb * nb; i += blockDim.x) {
      const int r = i / nb, c = i - r * nb;
      if (c > k && r >= c) a[r][c] -= a[r][k] * a[c][k];
    }
    __syncthreads();
  }
  for (int i = tid; i < nb * nb; i += blockDim.x) {
    const int r = i / nb, c = i - r * nb;
    if (r >= c) A[static_cast<int64_t>(j0 + r) * n + j0 + c] = a[r][c];
  }
}

// Rows below the diagonal block: L21 = A21 L11^-T (forward substitution per row).
__global__ void trsm_panel_kernel(double* A, int n, int j0, int nb) {
  __shared__ double l11[NB][NB + 1];
  for (int i = threadIdx.x; i < nb * nb; i += blockDim.x) {
    const int r = i / nb, c = i - r * nb;
    l11[r][c] = r >= c ? A[static_cast<int64_t>(j0 + r) * n + j0 + c] : 0.0;
  }
  __syncthreads();
  const int i = j0 + nb + blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  double x[NB];
  double* row = A + static_cast<int64_t>(i) * n + j0;
  for (int c = 0; c < nb; ++c) x[c] = row[c];
  for (int c = 0; c < nb; ++c) {
    double s = x[c];
    for (int k = 0; k < c; ++k) s -= x[k] * l11[c][k];
    x[c] = s / l11[c][c];
  }
  for (int c = 0; c < nb; ++c) row[c] = x[c];
}

// Trailing update A22 -= L21 L21^T on the lower triangle, 32 x 32 tiles.
__global__ void syrk_update_kernel(double* A, int n, int j0, int nb) {
  __shared__ double pi[NB][NB + 1], pj[NB][NB + 1];
  const int t0 = j0 + nb;
  // triangular tile index -> (ti >= tj)
  const int64_t idx = blockIdx.x;
  int ti = static_cast<int>((sqrt(8.0 * static_cast<double>(idx) + 1.0) - 1.0) / 2.0);
  while (static_cast<int64_t>(ti) * (ti + 1) / 2 > idx) --ti;
  while (static_cast<int64_t>(ti + 1) * (ti + 2) / 2 <= idx) ++ti;
  const int tj = static_cast<int>(idx - static_cast<int64_t>(ti) * (ti + 1) / 2);
  const int r0 = t0 + ti * NB, c0 = t0 + tj * NB;
  for (int i = threadIdx.x; i < NB * nb; i += blockDim.x) {
    const int r = i / nb, k = i - r * nb;
    pi[r][k] = r0 + r < n ? A[static_cast<int64_t>(r0 + r) * n + j0 + k] : 0.0;
    pj[r][k] = c0 + r < n ? A[static_cast<int64_t>(c0 + r) * n + j0 + k] : 0.0;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < NB * NB; i += blockDim.x) {
    const int r = i / NB, c = i - r * NB;
    const int gr = r0 + r, gc = c0 + c;
    if (gr >= n || gc >= n || gc > gr) continue;
    double s = 0.0;
    for (int k = 0; k < nb; ++k) s += pi[r][k] * pj[c][k];
    A[static_cast<int64_t>(gr) * n + gc] -= s;
  }
}

template <typename T>
__global__ void chol_store_kernel(const double* A, int n, T* out) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < static_cast<int64_t>(n) * n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / n), c = static_cast<int>(i - static_cast<int64_t>(r) * n);
    out[i] = from_f32<T>(c <= r ? static_cast<float>(A[i]) : 0.f);
  }
}

// e4m3 copy of a weight with one float32 scale per output row: scale = max|w| / 448
// (1 for an all-zero row), q = e4m3(w / scale) rounded to nearest even, saturating.
__global__ void quantize_e4m3_kernel(const void* w, int dtype, int rows, int cols, uint8_t* q, float* scale) {
  __shared__ float red[32];
  const int r = blockIdx.x;
  float amax = 0.f;
  for (int c = threadIdx.x; c < cols; c += blockDim.x)
    amax = fmaxf(amax, fabsf(load_as_f32(w, dtype, static_cast<int64_t>(r) * cols + c)));
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    t = warp_max(t);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const float s = red[0] > 0.f ? __fdiv_rn(red[0], 448.f) : 1.f;
  if (threadIdx.x == 0) scale[r] = s;
  for (int c = threadIdx.x; c < cols; c += blockDim.x) {
    const float x = __fdiv_rn(load_as_f32(w, dtype, static_cast<int64_t>(r) * cols + c), s);
    q[static_cast<int64_t>(r) * cols + c] = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);  // nearest even
  }
}

}  // namespace

cudaError_t to_f32(cudaStream_t s, const void* src, int dtype, int64_t n, float* dst) {
  if (n <= 0) return cudaSuccess;
  to_f32_kernel<<<static_cast<int>(std::min<int64_t>((n + 255) / 256, 4096)), 256, 0, s>>>(src, dtype, n, dst);
  return cudaGetLastError();
}

cudaError_t mul_vec(cudaStream_t s, const float* a, const float* b, float* out, int n) {
  if (n <= 0) return cudaSuccess;
  mul_vec_kernel<<<(n + 255) / 256, 256, 0, s>>>(a, b, out, n);
  return cudaGetLastError();
}

cudaError_t time_cond(cudaStream_t s, const TimeCondArgs& a, double* cond) {
  const size_t smem = static_cast<size_t>(a.Te + a.C) * sizeof(double);
  time_cond_kernel<<<1, 256, smem, s>>>(a, cond);
  return cudaGetLastError();
}

cudaError_t adaln(cudaStream_t s, const void* w, const void* b, int dtype, int C, int D, const double* cond,
                  float* s1, float* sh, float* gate) {
  const int64_t threads = static_cast<int64_t>(3) * D * 32;
  adaln_kernel<<<static_cast<int>((threads + 255) / 256), 256, 0, s>>>(w, b, dtype, C, D, cond, s1, sh, gate);
  return cudaGetLastError();
}

int64_t colsum_doubles(int64_t V, int H) { return (V + kColsumRows - 1) / kColsumRows * H; }

cudaError_t uniform_constant(cudaStream_t s, const void* E, int dtype, int64_t V, int H, const float* w, float eps,
                             double* colsum, float* u) {
  const int blocks = static_cast<int>((V + kColsumRows - 1) / kColsumRows);
  dim3 grid((H + 255) / 256, static_cast<unsigned>(blocks));
  colsum_kernel<<<grid, 256, 0, s>>>(E, dtype, V, H, kColsumRows, colsum);
  uniform_kernel<<<1, 1024, 0, s>>>(colsum, blocks, V, H, w, eps, u);
  return cudaGetLastError();
}

cudaError_t cholesky_f64(cudaStream_t s, double* A, int n, unsigned* err) {
  for (int j0 = 0; j0 < n; j0 += NB) {
    const int nb = std::min(NB, n - j0);
    potrf_diag_kernel<<<1, 256, 0, s>>>(A, n, j0, nb, err);
    const int rest = n - j0 - nb;
    if (rest > 0) {
      trsm_panel_kernel<<<(rest + 127) / 128, 128, 0, s>>>(A, n, j0, nb);
      const int64_t t = (rest + NB - 1) / NB;
      syrk_update_kernel<<<static_cast<unsigned>(t * (t + 1) / 2), 256, 0, s>>>(A, n, j0, nb);
    }
  }
  return cudaGetLastError();
}

cudaError_t chol_store(cudaStream_t s, const double* A, int n, int dtype, void* out) {
  const int blocks = 4096;
  if (dtype == FLASHMAP_F32)
    chol_store_kernel<float><<<blocks, 256, 0, s>>>(A, n, static_cast<float*>(out));
  else
    chol_store_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(A, n, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

cudaError_t quantize_e4m3(cudaStream_t s, const void* w, int dtype, int rows, int cols, void* q, float* scale) {
  quantize_e4m3_kernel<<<rows, 256, 0, s>>>(w, dtype, rows, cols, static_cast<uint8_t*>(q), scale);
  return cudaGetLastError();
}

}  // namespace fm
