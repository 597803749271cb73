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

// One head vector (channels lane*EPL..) of a step-produced float32 row: one L2 load.
template <int EPL>
__device__ __forceinline__ void load_head_vec(const float* src, float (&v)[EPL], int lane) {
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

// ------------------------------------------------------------------ block self-attention

#ifndef FM_SA_WIDE_CTAS_PER_SM
#define FM_SA_WIDE_CTAS_PER_SM 4
#endif

// One CTA per (request, head); warp w holds slots w * SPW .. w * SPW + SPW - 1 (two
// per warp at large batches: twice the loads in flight per thread, half the threads
// per CTA, so more CTAs fit on an SM).
template <typename T, int EPL, int SPW>
__global__ void self_attn_kernel(const float* __restrict__ qkv, int K, int nh, const float* __restrict__ qn,
                                 const float* __restrict__ kn, float eps, const float2* __restrict__ rope_tab,
                                 int max_pos, const int32_t* __restrict__ anchor_pos, T* __restrict__ out,
                                 int early, unsigned* dev_err) {
  constexpr int HD = EPL * 32;
  extern __shared__ float sm[];
  constexpr int LDQ = HD + 4;      // 16-byte rows, 4 banks apart: conflict-free float4 reads
  float* sq = sm;                  // [K][LDQ]
  float* sk = sq + K * LDQ;        // [K][LDQ]
  float* sv = sk + K * LDQ;        // [K][HD]
  pdl_trigger();
  const int b = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float wq[EPL], wk[EPL];  // the norm weights: constants, read before waiting
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    wq[e] = qn[lane * EPL + e];
    wk[e] = kn[lane * EPL + e];
  }
  __shared__ int s_anchor;
  // early: the positions were written before the kernel just before this one started
  if (early && threadIdx.x == 0) s_anchor = LDCG(anchor_pos + b);
  pdl_wait();
  const int D = nh * HD;
  // q, k and v of this warp's slots and head: all loads first (one vector per lane and
  // part), then the request's position (once per CTA) and the norms, so the L2 round
  // trips overlap
  float v[SPW][3][EPL];
#pragma unroll
  for (int i = 0; i < SPW; ++i) {
    const int k = warp * SPW + i;
    if (k < K) {  // warp-uniform
      const float* base = qkv + static_cast<int64_t>(b * K + k) * 3 * D + h * HD;
#pragma unroll
      for (int part = 0; part < 3; ++part) load_head_vec<EPL>(base + part * D, v[i][part], lane);
    }
  }
  if (!early && threadIdx.x == 0) s_anchor = LDCG(anchor_pos + b);
  __syncthreads();
#pragma unroll
  for (int i = 0; i < SPW; ++i) {
    const int k = warp * SPW + i;
    if (k >= K) continue;
    int pos = s_anchor + 1 + k;
    if (pos < 0 || pos >= max_pos) {
      if (lane == 0) set_dev_error(dev_err, FLASHMAP_DEVERR_POSITION);
      pos = 0;
    }
    const float2* rope = rope_tab + static_cast<int64_t>(pos) * (HD / 2);
    if constexpr (EPL >= 2) {  // the slot's rotation pairs, requested before q, k and v are used
      float2 cs[EPL / 2];
#pragma unroll
      for (int c = 0; c < EPL / 2; ++c) cs[c] = rope[(lane * EPL >> 1) + c];
      head_norm_rot<EPL>(v[i][0], wq, eps, cs);
      head_norm_rot<EPL>(v[i][1], wk, eps, cs);
    } else {
      head_norm_rope_w<EPL>(v[i][0], wq, eps, rope, lane);
      head_norm_rope_w<EPL>(v[i][1], wk, eps, rope, lane);
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      sq[k * LDQ + lane * EPL + e] = v[i][0][e];
      sk[k * LDQ + lane * EPL + e] = v[i][1][e];
      sv[k * HD + lane * EPL + e] = v[i][2][e];
    }
  }
  __syncthreads();
  const float scale = rsqrtf(static_cast<float>(HD));
#pragma unroll
  for (int i = 0; i < SPW; ++i) {
    const int k = warp * SPW + i;
    if (k >= K) continue;
    // scores of slot k against slot j = lane (four partial sums: a short dependency chain)
    float s = -INFINITY;
    if (lane < K) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const float4* qr = reinterpret_cast<const float4*>(sq + k * LDQ);
      const float4* kr = reinterpret_cast<const float4*>(sk + lane * LDQ);
#pragma unroll
      for (int d4 = 0; d4 < HD / 4; ++d4) {
        const float4 a4 = qr[d4], b4 = kr[d4];
        float& c = acc[d4 & 3];
        c = fmaf(a4.x, b4.x, c);
        c = fmaf(a4.y, b4.y, c);
        c = fmaf(a4.z, b4.z, c);
        c = fmaf(a4.w, b4.w, c);
      }
      s = ((acc[0] + acc[1]) + (acc[2] + acc[3])) * scale;
    }
    const float m = warp_max(s);
    float p = lane < K ? expf(s - m) : 0.f;
    p /= warp_sum(p);
    // the probabilities of all K (<= 16) slots in every lane, then each lane's channels
    float pj[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) pj[j] = __shfl_sync(0xffffffffu, p, j);
    T* o = out + static_cast<int64_t>(b * K + k) * D + h * HD;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const int d = lane + 32 * e;
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < K) acc = fmaf(pj[j], sv[j * HD + d], acc);
      o[d] = from_f32<T>(acc);
    }
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
  pdl_trigger();
  pdl_wait();
  float t16 = 0.f;
  for (int b = threadIdx.x; b < bs; b += blockDim.x) t16 += static_cast<float>((max(LDCG(anchor_pos + b) + 1, 1) + 15) / 16);
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
    const int n = b < bs ? max(LDCG(anchor_pos + b) + 1, 1) : 0;
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

// ------------------------------------------------------------------ cross-attention queries

// The layer's cross-attention queries of request b, head h, in float32 sq[16][HD]
// (rows >= K zero): q = RoPE(RMSNorm_{q_norm}(W_q n)) at the slot positions
// p + 1 + k (flashmap/modeling_flashmap.py, FlashMapAttention.forward). Every item of a
// (request, head) derives them from the projection accumulator; 128 threads.
template <int HD, bool kQuant = false>
__device__ __forceinline__ float load_queries(const XattnArgs& a, int b, int h, float* sq, int anchor) {
  constexpr int EPL = HD / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int D = a.nh * HD;
  float v[4][EPL];
  // every load of the warp's four rows first, then the reductions
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int q = warp + 4 * i;
    const float* src = a.qacc + static_cast<int64_t>(b * a.K + q) * D + h * HD + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) v[i][e] = q < a.K ? LDCG(src + e) : 0.f;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int q = warp + 4 * i;
    if (q < a.K) {  // warp-uniform
      int pos = anchor + 1 + q;
      if (pos < 0 || pos >= a.max_pos) {
        if (lane == 0) set_dev_error(a.dev_err, FLASHMAP_DEVERR_POSITION);
        pos = 0;
      }
      head_norm_rope<EPL>(v[i], a.q_norm, a.eps, a.rope + static_cast<int64_t>(pos) * (HD / 2), lane);
    }
  }
  float qscale = 1.f;
  if constexpr (kQuant) {
    // e4m3 queries for an e4m3 pool: one scale per (request, head), max|q| / 448 over
    // the block's slots and channels (flashmap/sglang/model.py, _paged_cross_attention_fp8)
    __shared__ float red[4];
    float mx = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int e = 0; e < EPL; ++e) mx = fmaxf(mx, fabsf(v[i][e]));
    mx = warp_max(mx);
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    qscale = __fdiv_rn(fmaxf(mx, 1e-12f), 448.f);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const __nv_fp8_storage_t q8 = __nv_cvt_float_to_fp8(__fdiv_rn(v[i][e], qscale), __NV_SATFINITE, __NV_E4M3);
        v[i][e] = __half2float(__half(__nv_cvt_fp8_to_halfraw(q8, __NV_E4M3)));
      }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int q = warp + 4 * i;
#pragma unroll
    for (int e = 0; e < EPL; ++e) sq[q * HD + lane * EPL + e] = v[i][e];
  }
  return qscale;
}

// ------------------------------------------------------------------ paged cross-attention items (SIMT)

template <typename T, int HD>
__global__ void __launch_bounds__(128) xattn_items_simt_kernel(XattnArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sq[16][HD];
  __shared__ float sk[16][HD + 1];
  __shared__ float sv[16][HD];
  __shared__ float ss[16][17];
  __shared__ float sm[16], sl[16], scorr[16];
  const int tid = threadIdx.x;
  const int nh = a.nh;
  const int items = LDCG(a.plan), chunk_len = LDCG(a.plan + 1);
  const int* pairs = a.plan + 4 + a.bs;
  const T* pool = static_cast<const T*>(a.pool);
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int g = item / nh, h = item - g * nh;
    const int b = LDCG(pairs + 2 * g), c = LDCG(pairs + 2 * g + 1);
    const int n = LDCG(a.anchor_pos + b) + 1;
    const int p0 = c * chunk_len, p1 = min(n, p0 + chunk_len);
    const int rrow = a.req_pool_idx ? LDCG(a.req_pool_idx + b) : b;
    __syncthreads();
    load_queries<HD>(a, b, h, &sq[0][0], LDCG(a.anchor_pos + b));
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
      int page = pi < a.r2p_stride ? LDCG(a.req_to_page + static_cast<int64_t>(rrow) * a.r2p_stride + pi) : -1;
      const bool ok = page >= 0 && page < a.num_pages;
      if (!ok && tid == 0) set_dev_error(a.dev_err, FLASHMAP_DEVERR_PAGE);
      const int off = blk - pi * a.P;
      const int64_t kb = ((((static_cast<int64_t>(a.layer) * 2 + 0) * a.num_pages + (ok ? page : 0)) * nh + h) * a.P + off) * HD;
      const int64_t vb = ((((static_cast<int64_t>(a.layer) * 2 + 1) * a.num_pages + (ok ? page : 0)) * nh + h) * a.P + off) * HD;
      __syncthreads();
      for (int i = tid; i < 16 * HD; i += blockDim.x) {
        const int j = i / HD, d = i - j * HD;
        const bool valid = ok && blk + j < p1;
        sk[j][d] = valid ? to_f32(LDCG(pool + kb + i)) : 0.f;
        sv[j][d] = valid ? to_f32(LDCG(pool + vb + i)) : 0.f;
      }
      __syncthreads();
      for (int i = tid; i < 256; i += blockDim.x) {
        const int qi = i >> 4, j = i & 15;
        float acc = 0.f;
#pragma unroll 8
        for (int d = 0; d < HD; ++d) acc = fmaf(sq[qi][d], sk[j][d], acc);
        ss[qi][j] = (blk + j < p1 && ok) ? acc * a.scale_log2 : -INFINITY;
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

// ------------------------------------------------------------------ paged cross-attention items (tensor cores)
//
// bf16 path. The 16 queries of a (request, head) are exactly the M = 16 of
// mma.sync.m16n8k16, so S = Q K^T and O += P V run on the tensor cores without
// padding (tcgen05's smallest tile would waste 3/4 of its rows here). Each warp
// streams its own 16-position blocks of K and V (4 KB each at hd 128: one page
// slice) through a 3-deep cp.async ring in XOR-swizzled shared memory (16-byte
// chunk c of row r stored at c ^ (r & 7): conflict-free ldmatrix), keeps the running
// max / sum / O of its blocks in registers (base-2 exponents), and the CTA merges its
// four warps before writing the item's partial.

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// 2^x (ex2.approx, subnormal results flushed to zero; -inf -> 0).
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Four e4m3 values (one word, lowest byte first) -> two half2 words (exact).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
// D += A B with e4m3 A (16 x 32, row) and B (32 x 8, col), float32 accumulation.
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Four e4m3-representable floats -> four e4m3 bytes (exact), lowest first.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xFFFFu) | (hi << 16);
}
// bf16 operands for a bf16 pool; half for an e4m3 pool (e4m3 widens to half in one
// conversion per pair, and the e4m3 queries and the probabilities are exact or finer
// in half)
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return F16 ? pack_f16(lo, hi) : pack_bf16(lo, hi);
}
template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (F16)
    mma_f16_16816(d, a, b0, b1);
  else
    mma_bf16_16816(d, a, b0, b1);
}

// The byte of position p (< 16) in a 16-byte row of an e4m3 pool's channel-major values.
__device__ __forceinline__ int vbyte_of(int p) { return 4 * ((p & 7) >> 1) + 2 * (p >> 3) + (p & 1); }

constexpr float kLazyLog2 = 8.f;  // the running max's slack: p <= 2^8
constexpr int kXStages = 3;   // bf16 pool, one candidate: cp.async stages per warp
constexpr int kXStages8 = 4;  // e4m3 pool (half the bytes per stage; 3 CTAs per SM)

__device__ __forceinline__ void bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// A CTA's 4 warps serve NC blocks that share one context: NC = 1 for a draft (one
// block per request), 2 or 4 for the candidate blocks of a tree draft. The warps of a
// candidate (WPC = 4 / NC of them) split the chunk's 16-position blocks by block lane
// (warp % WPC); the NC warps of one block lane share a ring of K/V blocks, each issuing
// part of every block's copies, so the context is read once for the NC candidates.
// Ring layout: 16-byte chunks XOR-swizzled by row. For an e4m3 pool the keys feed the
// e4m3 tensor-core product as stored, and the values arrive channel-major (the pool
// keeps each (page, head) block of values that way): one 16-byte row per channel holds
// the block's 16 positions, so a plain ldmatrix hands each thread four consecutive
// bytes of one channel, widened to half in registers for the half product with the
// probabilities. The pool orders each 16 positions so that bytes 4t..4t+3 are positions
// 2t, 2t+1, 2t+8, 2t+9, the k rows the product's fragment wants from thread t.
template <int HD, bool F8 = false, int NC = 1>
struct XCfg {
  static constexpr int WPC = 4 / NC;      // warps per candidate = rings per CTA
  static constexpr int ROWB = HD * 2;     // bytes of one bf16 position row
  static constexpr int BLK = 16 * ROWB;   // one 16-position block of K (or V), bf16
  static constexpr int CH = HD / 8;       // 16-byte chunks per bf16 row
  static constexpr int ROWB8 = HD;        // bytes of one e4m3 row
  static constexpr int BLK8 = 16 * ROWB8;
  static constexpr int CH8 = HD / 16;     // 16-byte chunks per e4m3 row
  static constexpr int STAGES = NC == 1 ? (F8 ? kXStages8 : kXStages) : NC == 4 ? 8 : (F8 ? 6 : 4);
  static constexpr int STAGE = F8 ? 2 * BLK8 : 2 * BLK;
  static constexpr int WORK = 0;
  // e4m3 rows are HD bytes: chunk c of row r sits at c ^ ((r >> SW8) & (CH8 - 1)), so the
  // 8 rows an ldmatrix reads fall on distinct banks (128-byte rows: r & 7; 64-byte: r/2 & 3)
  static constexpr int SW8 = CH8 >= 8 ? 0 : (CH8 == 4 ? 1 : 2);
  static constexpr int RING = STAGES * STAGE + WORK;
  static constexpr int SMEM_RING = WPC * RING;
  static constexpr int SQ_OFF = SMEM_RING;          // the candidates' queries, beside the rings
  static constexpr int SMEM_Q = SQ_OFF + NC * 16 * HD * 4;
  static constexpr int SMEM_MERGE = 4 * 16 * (HD + 2) * 4;
  static constexpr int SMEM = SMEM_Q > SMEM_MERGE ? SMEM_Q : SMEM_MERGE;
};

template <int HD, bool F8, int NC>
__global__ void __launch_bounds__(128, F8 ? 3 : 2) xattn_items_mma_kernel(XattnArgs a) {
  using C = XCfg<HD, F8, NC>;
  constexpr int WPC = C::WPC;
  extern __shared__ __align__(128) uint8_t xsm[];
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int cw = warp / WPC, lw = warp - cw * WPC;  // this warp's candidate and block lane
  const int nh = a.nh;
  const int chunk_len = LDCG(a.plan + 1), chunks = LDCG(a.plan + 2);
  const int* first = a.plan + 3;
  const int* pairs = a.plan + 4 + a.bs;
  const uint8_t* pool = static_cast<const uint8_t*>(a.pool);  // element e at byte e * (F8 ? 1 : 2)
  constexpr int ES = F8 ? 1 : 2;
  const uint32_t ring = smem_u32(xsm) + lw * C::RING;
  // candidate groups of NC blocks of one request (NC > 1): a.n_cand blocks per request
  const int ncand = NC > 1 ? a.n_cand : 1, groups = ncand / NC, nreq = a.bs / ncand;
  const int total = NC > 1 ? (chunks / ncand) * nh * groups : LDCG(a.plan);
  // Items are handed out in order as CTAs free up (item lengths vary by orders of
  // magnitude across a ragged batch): each CTA starts at its own index and claims its
  // next one from the shared counter while it works on the current one.
  __shared__ int s_next;
  for (int v = blockIdx.x; v < total;) {
    int claimed = 0;
    if (a.next_item && threadIdx.x == 0) claimed = static_cast<int>(gridDim.x + atomicAdd(a.next_item, 1u));
    int h, b, c, gk[NC];  // head, this warp's block, chunk; every candidate's pair index
    if constexpr (NC == 1) {
      const int g = v / nh;
      h = v - g * nh;
      b = LDCG(pairs + 2 * g);
      c = LDCG(pairs + 2 * g + 1);
      gk[0] = g;
    } else {
      const int grp = v % groups, t = v / groups;
      h = t % nh;
      const int q = t / nh;  // the request chunk: request r's chunks are q in [F(r), F(r + 1))
      int lo = 0, hi = nreq - 1;  // F(r) = first[r * ncand] / ncand, the largest r with F(r) <= q
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (LDCG(first + mid * ncand) / ncand <= q) lo = mid; else hi = mid - 1;
      }
      c = q - LDCG(first + lo * ncand) / ncand;
#pragma unroll
      for (int k = 0; k < NC; ++k) gk[k] = LDCG(first + lo * ncand + grp * NC + k) + c;
      b = lo * ncand + grp * NC + cw;
    }
    const int n = LDCG(a.anchor_pos + b) + 1;
    const int p0 = c * chunk_len, p1 = min(n, p0 + chunk_len);
    const int nblk = (p1 - p0 + 15) >> 4;
    const int rrow = a.req_pool_idx ? LDCG(a.req_pool_idx + b) : b;
    // The first blocks of keys and values are requested before the queries are
    // prepared (the two do not depend on each other).
    const int nj = lw < nblk ? (nblk - lw + WPC - 1) / WPC : 0;
    // The page ids of this lane's blocks, 32 blocks at a time, one per lane: loaded
    // ahead so that no page-table load sits between a block's issue and the next.
    const int32_t* r2p = a.req_to_page + static_cast<int64_t>(rrow) * a.r2p_stride;
    auto page_ids = [&](int j0) {
      const int j = j0 + lane;
      if (j >= nj) return -1;
      const int pi = (p0 + ((lw + WPC * j) << 4)) / a.P;
      return pi < a.r2p_stride ? LDCG(r2p + pi) : -1;
    };
    int pg = page_ids(0), pg_group = 0;
    // element offsets: K of (layer, page, head, position) = head_base + page * page_stride
    // + position * HD; V sits kv_stride further
    const int64_t page_stride = static_cast<int64_t>(nh) * a.P * HD;
    const int64_t head_base = (static_cast<int64_t>(a.layer) * 2 * a.num_pages * nh + h) * a.P * HD;
    const int64_t kv_stride = static_cast<int64_t>(a.num_pages) * page_stride;
    // the ring's NC warps split a block's 16-byte chunks: this warp's first chunk and stride
    const int ci0 = (NC > 1 ? cw * 32 : 0) + lane;
    const int p_shift = (a.P & (a.P - 1)) == 0 ? __ffs(a.P) - 1 : -1;  // a power-of-two page size
    auto issue = [&](int j) {
      if (j < nj) {
        if ((j >> 5) != pg_group) {  // warp-uniform: more than 32 blocks per lane
          pg_group = j >> 5;
          pg = page_ids(j & ~31);
        }
        const int blk = p0 + ((lw + WPC * j) << 4);
        const int pi = p_shift >= 0 ? blk >> p_shift : blk / a.P;
        const int page = __shfl_sync(0xffffffffu, pg, j & 31);
        const bool ok = page >= 0 && page < a.num_pages;
        if (!ok && lane == 0 && cw == 0) set_dev_error(a.dev_err, FLASHMAP_DEVERR_PAGE);
        const int off = blk - pi * a.P;
        const int64_t kb = head_base + (ok ? page : 0) * page_stride + off * HD;
        const int64_t vb = kb + kv_stride;
        const uint32_t st = ring + (j % C::STAGES) * C::STAGE;
        if constexpr (F8) {
          // keys: rows of 16-byte chunks, swizzled
#pragma unroll
          for (int i = ci0; i < 16 * C::CH8; i += 32 * NC) {
            const int r = i / C::CH8, ch = i - r * C::CH8;
            const uint32_t bytes = (ok && blk + r < p1) ? 16u : 0u;
            const uint32_t dst = st + r * C::ROWB8 + ((ch ^ ((r >> C::SW8) & (C::CH8 - 1))) << 4);
            cp_async16(dst, pool + (kb + r * HD) * ES + ch * 16, bytes);
          }
          // values: channel c of the block is 16 bytes at c * P + off in the (page, head)
          // block (an invalid page's zero-filled; positions past the chunk are zeroed
          // once they have landed)
          const int64_t vblk = kb - off * HD + kv_stride;
          const uint32_t vbytes = ok ? 16u : 0u;
#pragma unroll
          for (int i = ci0; i < HD; i += 32 * NC)
            cp_async16(st + C::BLK8 + i * 16, pool + vblk + static_cast<int64_t>(i) * a.P + off, vbytes);
        } else {
#pragma unroll
          for (int i = ci0; i < 16 * C::CH; i += 32 * NC) {
            const int r = i / C::CH, ch = i - r * C::CH;
            const uint32_t bytes = (ok && blk + r < p1) ? 16u : 0u;
            const uint32_t dst = st + r * C::ROWB + ((ch ^ (r & 7)) << 4);
            cp_async16(dst, pool + (kb + r * HD) * ES + ch * 16, bytes);
            cp_async16(dst + C::BLK, pool + (vb + r * HD) * ES + ch * 16, bytes);
          }
        }
      }
      cp_async_commit();
    };
#pragma unroll
    for (int j = 0; j < C::STAGES - 1; ++j) issue(j);
    // every candidate's Q (normed, rotated; e4m3-rounded for an e4m3 pool), rows >= K zero
    float* sq = reinterpret_cast<float*>(xsm + C::SQ_OFF);
    float qscale = 1.f;
    if constexpr (NC == 1) {
      qscale = load_queries<HD, F8>(a, b, h, sq, LDCG(a.anchor_pos + b));  // 1 unless e4m3 queries
    } else {
#pragma unroll 1
      for (int k = 0; k < NC; ++k) {
        const float s = load_queries<HD, F8>(a, b - cw + k, h, sq + k * 16 * HD, LDCG(a.anchor_pos + b - cw + k));
        if (k == cw) qscale = s;
      }
    }
    const float s_scale = a.scale_log2 * qscale;
    __syncthreads();
    const float* sqw = sq + cw * 16 * HD;
    // A fragments: bf16 (m16n8k16) for a bf16 pool; e4m3 (m16n8k32: a register holds
    // 4 channels, rows g8 / g8 + 8, channels 4 t4 + 0..3 and + 16) for an e4m3 pool
    constexpr int KQ = F8 ? HD / 32 : HD / 16;
    uint32_t qa[KQ][4];
#pragma unroll
    for (int kk = 0; kk < KQ; ++kk) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int row = g8 + ((j & 1) << 3);
        if constexpr (F8) {
          const float* q4 = sqw + row * HD + kk * 32 + ((j >> 1) << 4) + 4 * t4;
          qa[kk][j] = pack_e4m3x4(q4[0], q4[1], q4[2], q4[3]);
        } else {
          const int col = kk * 16 + ((j >> 1) << 3) + 2 * t4;
          qa[kk][j] = pack2<F8>(sqw[row * HD + col], sqw[row * HD + col + 1]);
        }
      }
    }
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[HD / 8][4];
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    for (int j = 0; j < nj; ++j) {
      if constexpr (NC == 1) {
        issue(j + C::STAGES - 1);
        cp_async_wait<C::STAGES - 1>();
        __syncwarp();
      } else {
        // block j landed (every warp waited for its part; the barrier joins them), and
        // every warp of the ring is done with block j - 1, whose stage is refilled next
        cp_async_wait<C::STAGES - 2>();
        bar_sync(1 + lw, 32 * NC);
        issue(j + C::STAGES - 1);
      }
      const int blk = p0 + ((lw + WPC * j) << 4);
      const uint32_t kst = ring + (j % C::STAGES) * C::STAGE;
      uint32_t vst = kst + C::BLK;
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if constexpr (F8) {
        // S = Q K^T on the e4m3 keys as stored: per 32 channels one ldmatrix.x4 of the
        // two 8-position halves x two 16-channel chunks gives both B fragments (a b16
        // matrix row of 16 bytes = 16 e4m3 channels; a thread's word = 4 channels)
#pragma unroll
        for (int kk = 0; kk < HD / 32; ++kk) {
          const int r = (lane & 7) + ((lane >> 4) << 3);
          const int ch = kk * 2 + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kst + r * C::ROWB8 + ((ch ^ ((r >> C::SW8) & (C::CH8 - 1))) << 4), b0, b1, b2, b3);
          mma_e4m3_16832(s[0], qa[kk], b0, b1);
          mma_e4m3_16832(s[1], qa[kk], b2, b3);
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const int r = (lane & 7) + ((lane >> 4) << 3);
          const int ch = kk * 2 + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kst + r * C::ROWB + ((ch ^ (r & 7)) << 4), b0, b1, b2, b3);
          mma16816<F8>(s[0], qa[kk], b0, b1);
          mma16816<F8>(s[1], qa[kk], b2, b3);
        }
      }
      if constexpr (F8) {
        vst = kst + C::BLK8;  // the channel-major e4m3 values
        if (blk + 16 > p1) {  // the chunk's last block: zero the values of positions past it
          const int valid = max(0, p1 - blk);
          uint8_t* vrow = xsm + (vst - smem_u32(xsm));
          for (int ch = lane; ch < HD; ch += 32)
            for (int p = valid; p < 16; ++p) vrow[ch * 16 + vbyte_of(p)] = 0;
          __syncwarp();
        }
      }
      // scale to base 2 and mask positions past the chunk (the last block only)
      if (blk + 16 <= p1) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[nt][e] *= s_scale;
      } else {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int pos = blk + nt * 8 + 2 * t4 + (e & 1);
            s[nt][e] = pos < p1 ? s[nt][e] * s_scale : -INFINITY;
          }
      }
      float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
      float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      // The reference max of a row moves only when a score passes it by more than
      // kLazyLog2 (base 2): then every row of the warp takes its running max and o, l
      // are rescaled; otherwise p <= 2^kLazyLog2 (well inside the half / bf16 range) and the
      // rescale is skipped. The sum is the same softmax; only its reference differs.
      if (__any_sync(0xffffffffu, mx0 > m0 + kLazyLog2 || mx1 > m1 + kLazyLog2)) {
        const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
        const float c0 = n0 == -INFINITY ? 1.f : ex2f(m0 - n0);
        const float c1 = n1 == -INFINITY ? 1.f : ex2f(m1 - n1);
        l0 *= c0;
        l1 *= c1;
        m0 = n0;
        m1 = n1;
#pragma unroll
        for (int i = 0; i < HD / 8; ++i) {
          o[i][0] *= c0;
          o[i][1] *= c0;
          o[i][2] *= c1;
          o[i][3] *= c1;
        }
      }
      const float z0 = m0 == -INFINITY ? 0.f : m0, z1 = m1 == -INFINITY ? 0.f : m1;  // -inf rows: p = 0
      float p[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        p[nt][0] = ex2f(s[nt][0] - z0);
        p[nt][1] = ex2f(s[nt][1] - z0);
        p[nt][2] = ex2f(s[nt][2] - z1);
        p[nt][3] = ex2f(s[nt][3] - z1);
      }
      l0 += p[0][0] + p[0][1] + p[1][0] + p[1][1];
      l1 += p[0][2] + p[0][3] + p[1][2] + p[1][3];
      const uint32_t pa[4] = {pack2<F8>(p[0][0], p[0][1]), pack2<F8>(p[0][2], p[0][3]), pack2<F8>(p[1][0], p[1][1]),
                              pack2<F8>(p[1][2], p[1][3])};
      if constexpr (F8) {
        // P V with the channel-major e4m3 values: per 32 channels one ldmatrix.x4 (lane L
        // addresses channel row 32 g + L) gives each thread 4 positions of 4 channels;
        // each word widens (exactly) to the two half pairs of one B fragment
#pragma unroll
        for (int g = 0; g < HD / 32; ++g) {
          uint32_t w[4];
          ldsm_x4(vst + (g * 32 + lane) * 16, w[0], w[1], w[2], w[3]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t b0, b1;
            e4m3x4_to_f16x4(w[i], b0, b1);
            mma16816<F8>(o[4 * g + i], pa, b0, b1);
          }
        }
      } else {
#pragma unroll
        for (int dn = 0; dn < HD / 16; ++dn) {
          const int r = (lane & 7) + (((lane >> 3) & 1) << 3);
          const int ch = dn * 2 + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vst + r * C::ROWB + ((ch ^ (r & 7)) << 4), b0, b1, b2, b3);
          mma16816<F8>(o[2 * dn], pa, b0, b1);
          mma16816<F8>(o[2 * dn + 1], pa, b2, b3);
        }
      }
      __syncwarp();
    }
    cp_async_wait<0>();
    // row sums over the quad
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    __syncthreads();  // every warp is done with its ring: reuse it for the merge
    float* mm = reinterpret_cast<float*>(xsm);        // [4][16] max
    float* ll = mm + 64;                               // [4][16] sum
    float* oo = ll + 64;                               // [4][16][HD]
    if (t4 == 0) {
      mm[warp * 16 + g8] = m0;
      mm[warp * 16 + g8 + 8] = m1;
      ll[warp * 16 + g8] = l0;
      ll[warp * 16 + g8 + 8] = l1;
    }
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      float* r0 = oo + (warp * 16 + g8) * HD + i * 8 + 2 * t4;
      float* r1 = oo + (warp * 16 + g8 + 8) * HD + i * 8 + 2 * t4;
      r0[0] = o[i][0];
      r0[1] = o[i][1];
      r1[0] = o[i][2];
      r1[1] = o[i][3];
    }
    __syncthreads();
    // each candidate's partial: its WPC warps merged
#pragma unroll 1
    for (int k = 0; k < NC; ++k) {
      const int64_t pidx = static_cast<int64_t>(gk[k]) * nh + h;
      const int w0 = k * WPC;
      const int q = threadIdx.x >> 3, d0 = (threadIdx.x & 7) * (HD / 8);
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < WPC; ++w) M = fmaxf(M, mm[(w0 + w) * 16 + q]);
      float wgt[WPC], L = 0.f;
#pragma unroll
      for (int w = 0; w < WPC; ++w) {
        const float mw = mm[(w0 + w) * 16 + q];
        wgt[w] = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
        L = fmaf(wgt[w], ll[(w0 + w) * 16 + q], L);
      }
      float* po = a.part_o + pidx * 16 * HD + q * HD;
      for (int d = d0; d < d0 + HD / 8; ++d) {
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < WPC; ++w) acc = fmaf(wgt[w], oo[((w0 + w) * 16 + q) * HD + d], acc);
        po[d] = acc;
      }
      if ((threadIdx.x & 7) == 0) {
        a.part_ml[pidx * 32 + 2 * q] = M;
        a.part_ml[pidx * 32 + 2 * q + 1] = L;
      }
    }
    if (threadIdx.x == 0) s_next = a.next_item ? claimed : v + static_cast<int>(gridDim.x);
    __syncthreads();
    v = s_next;
  }
}

// ------------------------------------------------------------------ paged cross-attention items (TMA-fed)
//
// bf16 pool, head_dim 64 or 128. The same items and arithmetic as the cp.async kernel
// above, but each warp's 16-position blocks of K and V are fetched by one lane with
// TMA tensor copies (the pool viewed as rows of head_dim channels; one 64-channel box
// of 16 rows per copy, 128-byte swizzled for conflict-free ldmatrix) into a per-warp
// ring completed on mbarriers: a block costs the warp 2 * HD / 64 copy instructions
// instead of 16 per-lane cp.async with their address arithmetic. Rows past the chunk
// (or of an invalid page) arrive as whatever the pool holds there: their scores are
// masked and, in partial blocks, their value rows are zeroed before use.

constexpr int kXattnTmaMaxBatch = 8;

template <int HD>
struct XTCfg {
  static constexpr int BOX = 16 * 128;         // 16 rows x 64 bf16 channels, 128B-swizzled
  static constexpr int NB = HD / 64;           // boxes per block of K (or V)
  static constexpr int BLK = NB * BOX;
  static constexpr int STAGES = 3;
  static constexpr int STAGE = 2 * BLK;        // K then V
  static constexpr int RING = STAGES * STAGE;  // per warp
  static constexpr int SMEM_RING = 4 * RING;
  static constexpr int SQ_OFF = SMEM_RING;
  static constexpr int SMEM_Q = SQ_OFF + 16 * HD * 4;
  static constexpr int SMEM_MERGE = 4 * 16 * (HD + 2) * 4;
  static constexpr int SMEM = (SMEM_Q > SMEM_MERGE ? SMEM_Q : SMEM_MERGE) + 1024;  // + alignment slack
};

// byte offset of 16-byte chunk ch (0 .. HD/8-1) of row r in a block of XTCfg layout
__device__ __forceinline__ uint32_t xt_off(int r, int ch) {
  return static_cast<uint32_t>((ch >> 3) * (16 * 128) + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

template <int HD>
__global__ void __launch_bounds__(128, 2) xattn_items_tma_kernel(const __grid_constant__ CUtensorMap kvmap,
                                                                 XattnArgs a) {
  using C = XTCfg<HD>;
  extern __shared__ uint8_t xraw[];
  __shared__ uint64_t bars[4][C::STAGES];
  __shared__ volatile int abort_flag;
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g8 = lane >> 2, t4 = lane & 3;
  const uint32_t raw = smem_u32(xraw);
  uint8_t* xsm = xraw + (((raw + 1023u) & ~1023u) - raw);  // 1024-aligned: the swizzle atom
  if (threadIdx.x == 0) {
    for (int w = 0; w < 4; ++w)
      for (int st = 0; st < C::STAGES; ++st) mbar_init(&bars[w][st], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // early: nothing read before the wait below (plan, page table, pool) comes from the
  // kernel just before this one, so the first blocks are requested while it finishes
  bool waited = a.early == 0;
  if (waited) pdl_wait();
  const int nh = a.nh;
  const int items = LDCG(a.plan), chunk_len = LDCG(a.plan + 1);
  const int* pairs = a.plan + 4 + a.bs;
  const uint32_t ring = smem_u32(xsm) + warp * C::RING;
  uint8_t* ring_ptr = xsm + warp * C::RING;
  const int64_t rows_per_kv = a.num_pages * nh * a.P;  // pool rows between a layer's keys and values
  uint32_t jt = 0;      // blocks this warp has issued (and consumed), over all its items
  uint32_t okm = 0;     // bit st: the block in stage st comes from a valid page
  const uint64_t pol = l2_policy_evict_first();  // keys and values are read once
  // items from the work counter after each CTA's first, as in the cp.async kernel (the
  // claim follows the dependency wait: the counter is zeroed by the previous combine)
  __shared__ int s_next;
  for (int item = blockIdx.x; item < items;) {
    const int g = item / nh, h = item - g * nh;
    const int b = LDCG(pairs + 2 * g), c = LDCG(pairs + 2 * g + 1);
    const int n = LDCG(a.anchor_pos + b) + 1;
    const int p0 = c * chunk_len, p1 = min(n, p0 + chunk_len);
    const int nblk = (p1 - p0 + 15) >> 4;
    const int rrow = a.req_pool_idx ? LDCG(a.req_pool_idx + b) : b;
    const int nj = warp < nblk ? (nblk - warp + 3) >> 2 : 0;
    const int32_t* r2p = a.req_to_page + static_cast<int64_t>(rrow) * a.r2p_stride;
    auto page_ids = [&](int j0) {
      const int j = j0 + lane;
      if (j >= nj) return -1;
      const int pi = (p0 + ((warp + 4 * j) << 4)) / a.P;
      return pi < a.r2p_stride ? LDCG(r2p + pi) : -1;
    };
    int pg = page_ids(0), pg_group = 0;
    // the page of block j of this item (warp-uniform; -1 if invalid)
    auto page_of = [&](int j) {
      if ((j >> 5) != pg_group) {
        pg_group = j >> 5;
        pg = page_ids(j & ~31);
      }
      const int page = __shfl_sync(0xffffffffu, pg, j & 31);
      return (page >= 0 && page < a.num_pages) ? page : -1;
    };
    auto issue = [&](int j) {
      if (j >= nj) return;
      const int blk = p0 + ((warp + 4 * j) << 4);
      const int pi = blk / a.P;
      const int page = page_of(j);
      if (page < 0 && lane == 0) set_dev_error(a.dev_err, FLASHMAP_DEVERR_PAGE);
      const uint32_t st = (jt + j) % C::STAGES;
      okm = page < 0 ? (okm & ~(1u << st)) : (okm | (1u << st));
      if (lane == 0) {
        const int64_t krow = ((static_cast<int64_t>(a.layer) * 2 * a.num_pages + (page < 0 ? 0 : page)) * nh + h) * a.P +
                             (blk - pi * a.P);
        uint8_t* dst = ring_ptr + st * C::STAGE;
        mbar_arrive_expect_tx(&bars[warp][st], C::STAGE);
#pragma unroll
        for (int bx = 0; bx < C::NB; ++bx) {
          tma_load_2d(dst + bx * C::BOX, &kvmap, &bars[warp][st], bx * 64, static_cast<int>(krow), pol);
          tma_load_2d(dst + C::BLK + bx * C::BOX, &kvmap, &bars[warp][st], bx * 64,
                      static_cast<int>(krow + rows_per_kv), pol);
        }
      }
    };
#pragma unroll
    for (int j = 0; j < C::STAGES - 1; ++j) issue(j);
    if (!waited) {  // the queries (and every buffer written below) follow the kernel before
      pdl_wait();
      waited = true;
    }
    int claimed = 0;
    if (a.next_item && threadIdx.x == 0) claimed = static_cast<int>(gridDim.x + atomicAdd(a.next_item, 1u));
    // Q (normed, rotated, rounded to bf16) as A fragments; rows >= K are zero
    float* sq = reinterpret_cast<float*>(xsm + C::SQ_OFF);
    load_queries<HD>(a, b, h, sq, n - 1);  // n - 1: the anchor position, read above
    __syncthreads();
    uint32_t qa[HD / 16][4];
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int row = g8 + ((j & 1) << 3);
        const int col = kk * 16 + ((j >> 1) << 3) + 2 * t4;
        qa[kk][j] = pack_bf16(sq[row * HD + col], sq[row * HD + col + 1]);
      }
    }
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[HD / 8][4];
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    int jdone = 0;  // blocks of this item consumed
    for (int j = 0; j < nj; ++j) {
      issue(j + C::STAGES - 1);
      const uint32_t st = (jt + j) % C::STAGES, par = ((jt + j) / C::STAGES) & 1;
      if (!mbar_wait(&bars[warp][st], par, &abort_flag)) break;
      jdone = j + 1;
      const int blk = p0 + ((warp + 4 * j) << 4);
      const uint32_t kst = ring + st * C::STAGE, vst = kst + C::BLK;
      const int valid = (okm >> st) & 1u ? min(16, p1 - blk) : 0;  // rows holding positions of the chunk
      if (valid < 16) {  // warp-uniform: zero the value rows past them
        uint8_t* v = ring_ptr + st * C::STAGE + C::BLK;
        for (int i = lane; i < 16 * (HD / 8); i += 32) {
          const int r = i / (HD / 8), ch = i - r * (HD / 8);
          if (r >= valid) *reinterpret_cast<uint4*>(v + xt_off(r, ch)) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const int r = (lane & 7) + ((lane >> 4) << 3);
        const int ch = kk * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kst + xt_off(r, ch), b0, b1, b2, b3);
        mma_bf16_16816(s[0], qa[kk], b0, b1);
        mma_bf16_16816(s[1], qa[kk], b2, b3);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = nt * 8 + 2 * t4 + (e & 1);
          s[nt][e] = r < valid ? s[nt][e] * a.scale_log2 : -INFINITY;
        }
      float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
      float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
      const float c0 = n0 == -INFINITY ? 1.f : exp2f(m0 - n0);
      const float c1 = n1 == -INFINITY ? 1.f : exp2f(m1 - n1);
      float p[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        p[nt][0] = n0 == -INFINITY ? 0.f : exp2f(s[nt][0] - n0);
        p[nt][1] = n0 == -INFINITY ? 0.f : exp2f(s[nt][1] - n0);
        p[nt][2] = n1 == -INFINITY ? 0.f : exp2f(s[nt][2] - n1);
        p[nt][3] = n1 == -INFINITY ? 0.f : exp2f(s[nt][3] - n1);
      }
      l0 = l0 * c0 + p[0][0] + p[0][1] + p[1][0] + p[1][1];
      l1 = l1 * c1 + p[0][2] + p[0][3] + p[1][2] + p[1][3];
      m0 = n0;
      m1 = n1;
#pragma unroll
      for (int i = 0; i < HD / 8; ++i) {
        o[i][0] *= c0;
        o[i][1] *= c0;
        o[i][2] *= c1;
        o[i][3] *= c1;
      }
      const uint32_t pa[4] = {pack_bf16(p[0][0], p[0][1]), pack_bf16(p[0][2], p[0][3]), pack_bf16(p[1][0], p[1][1]),
                              pack_bf16(p[1][2], p[1][3])};
#pragma unroll
      for (int dn = 0; dn < HD / 16; ++dn) {
        const int r = (lane & 7) + (((lane >> 3) & 1) << 3);
        const int ch = dn * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vst + xt_off(r, ch), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dn], pa, b0, b1);
        mma_bf16_16816(o[2 * dn + 1], pa, b2, b3);
      }
      __syncwarp();
    }
    if (jdone < nj) {
      // a wait gave up: wait (bounded) for this warp's copies still in flight, so that
      // none lands after the CTA has moved on; the CTA then stops after this item
      const int issued = min(nj, jdone + C::STAGES - 1 + 1);
      for (int q = jdone; q < issued; ++q) {
        const uint32_t st = (jt + q) % C::STAGES, par = ((jt + q) / C::STAGES) & 1;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&bars[warp][st], par) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
      if (lane == 0) set_dev_error(a.dev_err, FLASHMAP_DEVERR_TIMEOUT);
    }
    jt += nj;
    // row sums over the quad
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    __syncthreads();  // every warp is done with its ring: reuse it for the merge
    float* mm = reinterpret_cast<float*>(xsm);        // [4][16] max
    float* ll = mm + 64;                               // [4][16] sum
    float* oo = ll + 64;                               // [4][16][HD]
    if (t4 == 0) {
      mm[warp * 16 + g8] = m0;
      mm[warp * 16 + g8 + 8] = m1;
      ll[warp * 16 + g8] = l0;
      ll[warp * 16 + g8 + 8] = l1;
    }
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      float* r0 = oo + (warp * 16 + g8) * HD + i * 8 + 2 * t4;
      float* r1 = oo + (warp * 16 + g8 + 8) * HD + i * 8 + 2 * t4;
      r0[0] = o[i][0];
      r0[1] = o[i][1];
      r1[0] = o[i][2];
      r1[1] = o[i][3];
    }
    __syncthreads();
    const int64_t pidx = static_cast<int64_t>(g) * nh + h;
    {
      const int q = threadIdx.x >> 3, d0 = (threadIdx.x & 7) * (HD / 8);
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) M = fmaxf(M, mm[w * 16 + q]);
      float wgt[4], L = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float mw = mm[w * 16 + q];
        wgt[w] = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
        L = fmaf(wgt[w], ll[w * 16 + q], L);
      }
      float* po = a.part_o + pidx * 16 * HD + q * HD;
      for (int d = d0; d < d0 + HD / 8; ++d) {
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) acc = fmaf(wgt[w], oo[(w * 16 + q) * HD + d], acc);
        po[d] = acc;
      }
      if ((threadIdx.x & 7) == 0) {
        a.part_ml[pidx * 32 + 2 * q] = M;
        a.part_ml[pidx * 32 + 2 * q + 1] = L;
      }
    }
    if (threadIdx.x == 0) s_next = a.next_item ? claimed : item + static_cast<int>(gridDim.x);
    __syncthreads();
    if (abort_flag) break;  // the same value in every warp after the barrier
    item = s_next;
  }
  if (!waited) pdl_wait();  // no item: the grid still completes after the kernel before
}

// ------------------------------------------------------------------ combine

// One CTA of 64 threads per (request, head, 4 query rows): the chunks' running maxima
// and sums are reduced per query row (16 threads per row), then each thread sums
// HD / 16 channels of its row over the chunks with the chunk weights 2^(m_c - M) / L.
constexpr int kMaxChunksPerRequest = 1024;  // max_position <= 262144, chunks >= 256 positions
constexpr int kCombineRowsMaxBatch = 4;     // up to this batch the one-row-per-CTA combine is faster

template <typename T, int HD>
__global__ void __launch_bounds__(64) xattn_combine_kernel(XattnArgs a, T* __restrict__ out) {
  __shared__ float sw[4][kMaxChunksPerRequest];  // per row: the chunks' maxima, then weights
  __shared__ int s_g[2];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, h = blockIdx.y, t = threadIdx.x;
  const int nh = a.nh, D = nh * HD;
  if (a.next_item && (b | h | blockIdx.z | t) == 0) *a.next_item = 0;  // for the next items launch
  if (t < 2) s_g[t] = LDCG(a.plan + 3 + b + t);  // the request's chunk range
  __syncthreads();
  const int g0 = s_g[0], nc = min(s_g[1] - g0, kMaxChunksPerRequest);
  const int ql = t >> 4, q = blockIdx.z * 4 + ql, j = t & 15;  // query row, lane within its 16 threads
  float* w = sw[ql];
  const float* ml = a.part_ml + (static_cast<int64_t>(g0) * nh + h) * 32 + 2 * q;
  const int64_t mls = static_cast<int64_t>(nh) * 32;  // between chunks
  float M = -INFINITY;
  for (int c = j; c < nc; c += 16) {
    const float m = LDCG(ml + c * mls);
    w[c] = m;
    M = fmaxf(M, m);
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));  // the row's 16 lanes
  float L = 0.f;
  for (int c = j; c < nc; c += 16) {
    const float m = w[c];
    const float wc = m == -INFINITY ? 0.f : exp2f(m - M);
    w[c] = wc;
    L = fmaf(wc, LDCG(ml + c * mls + 1), L);
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  __syncwarp();  // the row's weights are written by its own 16 lanes
  // channels d = j, j + 16, ...: independent loads over the chunks
  constexpr int NV = HD / 16;
  float acc[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) acc[v] = 0.f;
  const float* po = a.part_o + (static_cast<int64_t>(g0) * nh + h) * 16 * HD + q * HD + j;
  const int64_t pos_ = static_cast<int64_t>(nh) * 16 * HD;  // between chunks
#pragma unroll 2
  for (int c = 0; c < nc; ++c) {
    const float wc = w[c];
#pragma unroll
    for (int v = 0; v < NV; ++v) acc[v] = fmaf(wc, LDCG(po + c * pos_ + 16 * v), acc[v]);
  }
  if (q < a.K) {
    const int64_t r = (static_cast<int64_t>(b) * a.K + q) * D + h * HD + j;
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      out[r + 16 * v] = from_f32<T>(L > 0.f ? acc[v] * inv : 0.f);
    }
  }
}

// Small batches: one CTA of HD threads per (request, head, query row), one thread per
// channel, for more CTAs in flight when there are few requests. Each thread folds the
// chunks' partials into a running (max, sum, output) in one pass: every load is
// independent of the others, and no block reduction is needed.
template <typename T, int HD>
__global__ void __launch_bounds__(HD) xattn_combine_rows_kernel(XattnArgs a, T* __restrict__ out) {
  pdl_trigger();
  const int b = blockIdx.x, h = blockIdx.y, qi = blockIdx.z, d = threadIdx.x;
  const int nh = a.nh, D = nh * HD;
  int g0 = 0, g1 = 0;
  if (a.early) {  // the plan was complete before the items kernel started
    g0 = LDCG(a.plan + 3 + b);
    g1 = LDCG(a.plan + 4 + b);
  }
  pdl_wait();
  if (a.next_item && (b | h | qi | d) == 0) *a.next_item = 0;  // for the next items launch
  if (!a.early) {
    g0 = LDCG(a.plan + 3 + b);
    g1 = LDCG(a.plan + 4 + b);
  }
  const int nc = min(g1 - g0, kMaxChunksPerRequest);
  const float* mlp = a.part_ml + (static_cast<int64_t>(g0) * nh + h) * 32 + 2 * qi;
  const float* po = a.part_o + (static_cast<int64_t>(g0) * nh + h) * 16 * HD + qi * HD + d;
  const int64_t mls = static_cast<int64_t>(nh) * 32, ps = static_cast<int64_t>(nh) * 16 * HD;  // between chunks
  float M = -INFINITY, L = 0.f, acc = 0.f;
#pragma unroll 4
  for (int c = 0; c < nc; ++c) {
    const float2 ml = LDCG(reinterpret_cast<const float2*>(mlp + c * mls));  // (running max, sum) of chunk c
    const float o = LDCG(po + c * ps);
    if (ml.x == -INFINITY) continue;  // no position of the chunk: nothing to add
    const float nM = fmaxf(M, ml.x);
    const float s_old = exp2f(M - nM), s_new = exp2f(ml.x - nM);  // exp2(-inf) = 0
    L = fmaf(L, s_old, ml.y * s_new);
    acc = fmaf(acc, s_old, o * s_new);
    M = nM;
  }
  out[(static_cast<int64_t>(b) * a.K + qi) * D + h * HD + d] = from_f32<T>(L > 0.f ? acc / L : 0.f);
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

cudaError_t self_attention(const Launch& L, int dtype, const float* qkv, int bs, int K, int nh, int hd, const float* qn,
                           const float* kn, float eps, const float2* rope, int max_pos, const int32_t* anchor_pos,
                           void* out, bool early) {
  if (bs <= 0) return cudaSuccess;
  dim3 grid(bs, nh);
  const size_t smem = static_cast<size_t>(K) * ((hd + 4) * 2 + hd) * sizeof(float);
  cudaError_t e = cudaSuccess;
  const int ea = early ? 1 : 0;
  // two slots per warp once the grid alone holds a few CTAs per SM
  const bool wide = static_cast<int64_t>(bs) * nh >= static_cast<int64_t>(FM_SA_WIDE_CTAS_PER_SM) * L.num_sms;
#define FM_SA_LAUNCH(EPL_)                                                                                        \
  FM_DISPATCH_T2(dtype, (e = wide ? launch_k(L, self_attn_kernel<T, EPL_, 2>, grid, dim3(32 * ((K + 1) / 2)),   \
                                             smem, qkv, K, nh, qn, kn, eps, rope, max_pos, anchor_pos,          \
                                             static_cast<T*>(out), ea, L.dev_err)                               \
                                      : launch_k(L, self_attn_kernel<T, EPL_, 1>, grid, dim3(32 * K), smem, qkv, \
                                                 K, nh, qn, kn, eps, rope, max_pos, anchor_pos,                 \
                                                 static_cast<T*>(out), ea, L.dev_err)))
  if (hd == 32) {
    FM_SA_LAUNCH(1);
  } else if (hd == 64) {
    FM_SA_LAUNCH(2);
  } else {
    FM_SA_LAUNCH(4);
  }
#undef FM_SA_LAUNCH
  return e;
}

int xattn_target_items(int num_sms) { return num_sms * 16; }
// Room for the plan of a tree draft too, whose target is scaled by the candidates a CTA
// serves at once (at most 4)
int xattn_max_chunks(int num_sms, int nh, int bs) { return 4 * xattn_target_items(num_sms) / nh + bs + 1; }
int xattn_cands_per_cta(int n_cand) { return n_cand % 4 == 0 ? 4 : n_cand % 2 == 0 ? 2 : 1; }
size_t xattn_plan_ints(int num_sms, int nh, int bs) { return 4 + bs + 2 * static_cast<size_t>(xattn_max_chunks(num_sms, nh, bs)); }

cudaError_t xattn_plan(const Launch& L, const int32_t* anchor_pos, int bs, int nh, int* plan, int n_cand) {
  // a CTA serving NC candidates runs 1/NC of the items: NC times as many keep the SMs busy
  const int target = xattn_target_items(L.num_sms) * xattn_cands_per_cta(n_cand);
  return launch_k(L, xattn_plan_kernel, dim3(1), dim3(1024), 0, anchor_pos, bs, nh, target,
                  xattn_max_chunks(L.num_sms, nh, bs), plan, L.dev_err);
}

cudaError_t xattn_items(const Launch& L, int dtype, const XattnArgs& args, const CUtensorMap* kvmap) {
  XattnArgs a = args;
  a.dev_err = L.dev_err;
  const int grid = L.num_sms * 2;
  cudaError_t e = cudaSuccess;
  // TMA-fed at small batches (fewer instructions on the latency-bound path); the
  // cp.async kernel measured slightly faster once the pool streams at full rate
  const int nc = xattn_cands_per_cta(a.n_cand);
  if (nc > 1 && (dtype == FLASHMAP_BF16 || dtype == FLASHMAP_E4M3)) {
    // candidate blocks of a tree draft: NC of them per CTA share each K/V block
    const int g = L.num_sms * (dtype == FLASHMAP_E4M3 ? 3 : 2);
    if (dtype == FLASHMAP_BF16) {
      if (nc == 4)
        FM_DISPATCH_HD(a.hd, (e = launch_k(L, xattn_items_mma_kernel<HD, false, 4>, dim3(g), dim3(128),
                                           XCfg<HD, false, 4>::SMEM, a)));
      else
        FM_DISPATCH_HD(a.hd, (e = launch_k(L, xattn_items_mma_kernel<HD, false, 2>, dim3(g), dim3(128),
                                           XCfg<HD, false, 2>::SMEM, a)));
    } else {
      if (nc == 4)
        FM_DISPATCH_HD(a.hd, (e = launch_k(L, xattn_items_mma_kernel<HD, true, 4>, dim3(g), dim3(128),
                                           XCfg<HD, true, 4>::SMEM, a)));
      else
        FM_DISPATCH_HD(a.hd, (e = launch_k(L, xattn_items_mma_kernel<HD, true, 2>, dim3(g), dim3(128),
                                           XCfg<HD, true, 2>::SMEM, a)));
    }
  } else if (dtype == FLASHMAP_BF16 && kvmap && (a.hd == 64 || a.hd == 128) && a.bs <= kXattnTmaMaxBatch) {
    if (a.hd == 128)
      e = launch_k(L, xattn_items_tma_kernel<128>, dim3(grid), dim3(128), XTCfg<128>::SMEM, *kvmap, a);
    else
      e = launch_k(L, xattn_items_tma_kernel<64>, dim3(grid), dim3(128), XTCfg<64>::SMEM, *kvmap, a);
  } else if (dtype == FLASHMAP_BF16) {
    FM_DISPATCH_HD(a.hd, (e = launch_k(L, xattn_items_mma_kernel<HD, false, 1>, dim3(grid), dim3(128),
                                       XCfg<HD, false>::SMEM, a)));
  } else if (dtype == FLASHMAP_E4M3) {
    // three CTAs per SM: the e4m3 kernel is latency-bound per block, not byte-bound
    FM_DISPATCH_HD(a.hd, (e = launch_k(L, xattn_items_mma_kernel<HD, true, 1>, dim3(L.num_sms * 3), dim3(128),
                                       XCfg<HD, true>::SMEM, a)));
  } else {
    FM_DISPATCH_HD(a.hd, (e = launch_k(L, xattn_items_simt_kernel<float, HD>, dim3(grid), dim3(128), 0, a)));
  }
  return e;
}

cudaError_t xattn_prepare() {
  cudaError_t e = cudaSuccess;
#define FM_XATTR(HD_, F8_, NC_)                                                                                     \
  if (e == cudaSuccess)                                                                                             \
    e = cudaFuncSetAttribute(xattn_items_mma_kernel<HD_, F8_, NC_>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             XCfg<HD_, F8_, NC_>::SMEM);
#define FM_XATTR_NC(HD_, F8_) FM_XATTR(HD_, F8_, 1) FM_XATTR(HD_, F8_, 2) FM_XATTR(HD_, F8_, 4)
  FM_XATTR_NC(128, false) FM_XATTR_NC(64, false) FM_XATTR_NC(32, false) FM_XATTR_NC(128, true)
  FM_XATTR_NC(64, true) FM_XATTR_NC(32, true)
#undef FM_XATTR_NC
#undef FM_XATTR
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(xattn_items_tma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             XTCfg<128>::SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(xattn_items_tma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             XTCfg<64>::SMEM);
  return e;
}

cudaError_t xattn_combine(const Launch& L, int dtype, const XattnArgs& args, void* out) {
  XattnArgs a = args;
  a.dev_err = L.dev_err;
  cudaError_t e = cudaSuccess;
  if (a.bs <= kCombineRowsMaxBatch) {
    FM_DISPATCH_T2(dtype, FM_DISPATCH_HD(a.hd, (e = launch_k(L, xattn_combine_rows_kernel<T, HD>,
                                                             dim3(a.bs, a.nh, a.K), dim3(HD), 0, a,
                                                             static_cast<T*>(out)))));
    return e;
  }
  FM_DISPATCH_T2(dtype, FM_DISPATCH_HD(a.hd, (e = launch_k(L, xattn_combine_kernel<T, HD>, dim3(a.bs, a.nh, 4),
                                                           dim3(64), 0, a, static_cast<T*>(out)))));
  return e;
}

}  // namespace fm
