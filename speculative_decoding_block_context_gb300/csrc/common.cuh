// Shared device helpers of the FlashMap library (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "flashmap.h"

namespace fm {

// ------------------------------------------------------------------ dtypes

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float load_as_f32(const void* p, int dtype, int64_t i) {
  return dtype == FLASHMAP_F32 ? static_cast<const float*>(p)[i]
                               : __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

// ------------------------------------------------------------------ errors

__device__ __forceinline__ void set_dev_error(unsigned* err, unsigned bits) {
  if (err) atomicOr(err, bits);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Every pipeline wait gives up after this long and reports FLASHMAP_DEVERR_TIMEOUT.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

// ------------------------------------------------------------------ programmatic dependent launch
// Every kernel of a call is launched with programmatic stream serialization: it lets
// its dependents launch at once (their prologue, and a GEMM's weight prefetch,
// overlap its tail) and waits for its predecessors' completion before touching data
// they produce. Without a programmatic predecessor both are no-ops.

// Loads of data written earlier in the same chain of launches (accumulators, the
// residual stream, plans, partial results) and of per-call inputs go to L2
// (ld.global.cg): under programmatic dependent launch a CTA's L1 may still hold a
// line that other SMs have since changed in L2.
#define LDCG(p) __ldcg(p)

__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------------ stream-K partition
// (the tcgen05 GEMM's units (tile, 64-wide k block) cut into G contiguous ranges
// [T c / G, T (c + 1) / G); a reader of its split outputs repeats the same arithmetic)

// The CTA whose range holds unit u.
__host__ __device__ __forceinline__ int unit_owner(int64_t u, int64_t T, int G) {
  int c = static_cast<int>(u * G / T);
  while (c + 1 < G && T * (c + 1) / G <= u) ++c;
  while (c > 0 && T * c / G > u) --c;
  return c;
}
// The scratch slot of CTA c's part of tile `tile`: 2c for the first tile of its range,
// 2c + 1 for its last (ranges of at most a tile's k blocks touch two tiles).
__host__ __device__ __forceinline__ int64_t split_slot(int c, int64_t tile, int64_t T, int G, int KB) {
  return 2LL * c + ((T * c / G) / KB == tile ? 0 : 1);
}
__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// ------------------------------------------------------------------ reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sum over the block; `red` holds >= 32 floats. All threads get the result.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.f;
  t = warp_sum(t);
  return t;
}

// RMSNorm of one head vector held EPL-per-lane by a warp (lane owns channels
// lane*EPL .. lane*EPL+EPL-1), then the interleaved-pair rotation of the pairs
// (2i, 2i+1) by angle row `rope` (cos, sin per pair), if given
// (flashmap/modeling_flashmap.py, FlashMapRMSNorm and apply_rope).
template <int EPL>
__device__ __forceinline__ void head_norm_rope_w(float (&v)[EPL], const float (&w)[EPL], float eps,
                                                 const float2* __restrict__ rope, int lane) {
  constexpr int HD = EPL * 32;
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) ss = fmaf(v[e], v[e], ss);
  ss = warp_sum(ss);
  const float r = rsqrtf(ss * (1.f / HD) + eps);
#pragma unroll
  for (int e = 0; e < EPL; ++e) v[e] *= r * w[e];
  if (rope == nullptr) return;
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

// The same with the rotation's (cos, sin) pairs of this lane's channels already loaded
// (cs[i] for the pair (lane*EPL + 2i, lane*EPL + 2i + 1)); EPL >= 2.
template <int EPL>
__device__ __forceinline__ void head_norm_rot(float (&v)[EPL], const float (&w)[EPL], float eps,
                                              const float2 (&cs)[EPL / 2]) {
  static_assert(EPL >= 2, "pairs within a lane");
  constexpr int HD = EPL * 32;
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) ss = fmaf(v[e], v[e], ss);
  ss = warp_sum(ss);
  const float r = rsqrtf(ss * (1.f / HD) + eps);
#pragma unroll
  for (int e = 0; e < EPL; ++e) v[e] *= r * w[e];
#pragma unroll
  for (int e = 0; e < EPL; e += 2) {
    const float x1 = v[e], x2 = v[e + 1];
    v[e] = x1 * cs[e >> 1].x - x2 * cs[e >> 1].y;
    v[e + 1] = x2 * cs[e >> 1].x + x1 * cs[e >> 1].y;
  }
}

// The same with the norm weight read from memory (channels lane*EPL..).
template <int EPL>
__device__ __forceinline__ void head_norm_rope(float (&v)[EPL], const float* __restrict__ w, float eps,
                                               const float2* __restrict__ rope, int lane) {
  float wr[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) wr[e] = w[lane * EPL + e];
  head_norm_rope_w<EPL>(v, wr, eps, rope, lane);
}

// e4m3 x 16 (one 16-byte chunk) -> bf16 x 16 (two 16-byte chunks).
// Every e4m3 value is exact in half and in bf16.
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 u, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __half2_raw hr =
          __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * h)) & 0xFFFFu), __NV_E4M3);
      const float2 f = __half22float2(__half2(hr));
      const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
      o[2 * i + h] = *reinterpret_cast<const uint32_t*>(&b);
    }
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// e4m3 x 16 -> half x 16 (one conversion per pair; every e4m3 value is exact in half).
__device__ __forceinline__ void e4m3x16_to_f16(const uint4 u, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __half2_raw hr =
          __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * h)) & 0xFFFFu), __NV_E4M3);
      o[2 * i + h] = static_cast<uint32_t>(hr.x) | (static_cast<uint32_t>(hr.y) << 16);
    }
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// ------------------------------------------------------------------ shared memory / mbarrier

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase of `bar` with the given parity; gives up (returns false) after
// limit_ns or as soon as *abort is set, setting *abort itself on a timeout.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, volatile int* abort,
                                              uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort = 1;
      return false;
    }
  }
  return true;
}
// The pipelines' wait: kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return mbar_wait_for(bar, parity, abort, kWaitLimitNs);
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------------ tcgen05 (5th-generation tensor cores)

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA with
// 128-byte swizzle: rows of 64 bf16 (128 B), 8-row groups 1024 B apart (stride byte
// offset); the leading byte offset is unused for this layout; version 1 (bits 46-47);
// layout type 2 = SWIZZLE_128B (bits 61-63). Tiles must be 1024-byte aligned.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;          // leading byte offset (16 B, unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;  // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;          // descriptor version
  d |= static_cast<uint64_t>(2) << 61;          // SWIZZLE_128B
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: D float32, A and B bf16, both
// K-major, shape M x N (N multiple of 16 for M = 128).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                                  // D format: F32
         | (1u << 7)                                // A format: BF16
         | (1u << 10)                               // B format: BF16
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives on `bar` once every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns from TMEM (each thread: its lane).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace fm
