// Dense contractions of the FlashMap step.
//
// bf16 and e4m3 weights: a persistent, warp-specialized tcgen05 kernel. Every linear of
// the step is "weights x activations" with few activation rows (16 at batch 1), so the
// weight matrix W (N x K) is the MMA's A operand (M = 128 output channels per tile) and
// the activation rows are the B operand (N = 16..256 rows): the tensor core's large M
// dimension is spent on the weights and no row padding to 128 is needed. With at most
// half as many tiles as CTAs, a thread-block cluster splits each tile's k range and
// sums it through shared memory in rank order. Otherwise the iteration space (output
// tile, 64-wide k block) is cut into equal contiguous ranges, one per CTA (stream-K),
// so every SM streams the same number of weight bytes whatever the shape. A tile split
// over several CTAs is summed in a fixed order, so results repeat bit for bit: every
// CTA but one leaves its partial tile in a scratch slot and counts it; the CTA holding
// the tile's first k blocks (it reaches them last, at the end of its range) finds the
// others counted, adds their partials in CTA order while its own MMAs finish, then adds
// its own and writes the tile. If it arrives before all the others it leaves its
// partial too, and whichever arrives last sums the slots in the same order. No CTA
// waits for another's counter.
// Above 128 rows, bf16 GEMMs with at least 32 tiles of 256 x 256 run on SM pairs
// instead (tc_pair_kernel, tcgen05 cta_group::2: half of both operands per SM).
// Roles: warp 0 issues TMA loads (128B-swizzled, weights with an evict-first L2
// policy), warp 1 owns TMEM and issues tcgen05.mma, warps 2-5 drain the double-
// buffered TMEM accumulator (tcgen05.ld) into global memory, each warp its own 32
// output channels of a tile (split-tile counting is per warp as well).
//
// float32: SIMT kernels (the float32 path must match a float64 reference to 1e-4,
// which TF32 tensor cores cannot), and a general strided SIMT GEMM for load-time work.

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace fm {
namespace {

// Warps: 0 TMA producer, 1 MMA issuer, 2-5 epilogue, and for e4m3 weights 6-9
// converters (e4m3 weight tile -> bf16 tile in the MMA's swizzled layout).
constexpr int kTcThreads = 192;
constexpr int kTcThreadsF8 = 320;

// Pipeline depth of the narrow (<= 32 activation rows) GEMMs, and CTAs launched per SM.
#ifndef FM_TC_STAGES_NARROW
#define FM_TC_STAGES_NARROW 4
#endif
#ifndef FM_TC_CTAS_PER_SM
#define FM_TC_CTAS_PER_SM 2
#endif
// Whole tiles of 64 rows or more added onto the output by read-add-write (1) or by L2
// reductions (0).
#ifndef FM_GEMM_ADD_RMW
#define FM_GEMM_ADD_RMW 1
#endif
// Largest thread-block cluster of the cluster split-K mode (0: stream-K only; above 8
// needs the non-portable cluster sizes, at most 16).
#ifndef FM_GEMM_CLUSTER_MAX
#define FM_GEMM_CLUSTER_MAX 8
#endif
// The fewest 256 x 256 tiles with which a GEMM of more than 128 rows (bf16 weights)
// runs on SM pairs (tcgen05 cta_group::2): with 32, 64 SMs or more hold a tile (512
// rows x 4096 channels), and the pairs still beat the one-SM kernel's cluster split
// (batch-32 GEMMs 1.57 -> 1.48 ms per step); 0 turns the pair kernel off.
#ifndef FM_GEMM_PAIR_MIN_TILES
#define FM_GEMM_PAIR_MIN_TILES 32
#endif


// One pipeline stage: the bf16 weight tile (A, 128 x 64, 128B-swizzled), the
// activation tile (B, BN x 64, 128B-swizzled) and, for e4m3 weights, the raw e4m3
// weight tile as TMA wrote it (128 rows x 64 bytes, unswizzled) that the converter
// warps expand into A.
template <int BN, bool F8>
struct TcCfg {
  static constexpr int STAGES = F8 ? (BN <= 32 ? 4 : BN <= 64 ? 3 : BN <= 128 ? 5 : 4)
                                   : (BN <= 32 ? FM_TC_STAGES_NARROW : BN <= 64 ? 4 : BN <= 128 ? 6 : 4);
  static constexpr int A_BYTES = 128 * 64 * 2;
  static constexpr int B_BYTES = BN * 64 * 2;
  static constexpr int A8_BYTES = F8 ? 128 * 64 : 0;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + A8_BYTES;
  static constexpr uint32_t TX_BYTES = (F8 ? A8_BYTES : A_BYTES) + B_BYTES;  // bytes TMA writes per stage
  // Narrow bf16 tiles sum a cluster split-K tile by pushing: each rank stores its
  // partial of rank o's channels into o's receive area (one slot per sending rank,
  // channel-major, rows padded by 4), beside the ring.
  static constexpr bool PUSH = !F8 && BN <= 32 && FM_GEMM_CLUSTER_MAX >= 2;
  static constexpr int RECV_BYTES = PUSH ? (128 + FM_GEMM_CLUSTER_MAX) * (BN + 4) * 4 : 0;
  static constexpr int SMEM = STAGES * STAGE_BYTES + RECV_BYTES + 1024;
  static constexpr uint32_t TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;
  static constexpr int THREADS = F8 ? kTcThreadsF8 : kTcThreads;
  static constexpr int FIT = (228 * 1024) / (SMEM + 1024);
  static constexpr int PER_SM = FIT < FM_TC_CTAS_PER_SM ? (FIT < 1 ? 1 : FIT) : FM_TC_CTAS_PER_SM;
};


__device__ __forceinline__ bool mbar_wait_timed(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ float gelu_erf(float x) { return 0.5f * x * (1.f + erff(x * 0.70710678118654752f)); }

// A tile's final value y of (row, n), written as `mode` (an Out) says.
__device__ __forceinline__ void emit_out(int mode, void* out, int ldo, int row, int n, float y) {
  const int64_t o = static_cast<int64_t>(row) * ldo + n;
  if (mode == static_cast<int>(Out::Add))  // the one addition this element gets: a reduction, no return value
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(static_cast<float*>(out) + o), "f"(y) : "memory");
  else if (mode == static_cast<int>(Out::Store))
    static_cast<float*>(out)[o] = y;
  else
    static_cast<__nv_bfloat16*>(out)[o] = __float2bfloat16_rn(gelu_erf(y));
}

// Thread-block clusters: every thread of every CTA of the cluster arrives, then waits
// (release / acquire: shared-memory writes before it are visible to the cluster after).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// A 16-byte store into a peer CTA's shared memory that counts its bytes on the peer's
// mbarrier (both addresses shared::cluster).
__device__ __forceinline__ void st_async4(uint32_t addr, float a, float b, float c, float d, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
               "f"(a), "f"(b), "f"(c), "f"(d), "r"(bar)
               : "memory");
}
// Waits (at most kWaitLimitNs) for a phase completed by other CTAs of the cluster.
__device__ __forceinline__ bool mbar_wait_cluster_timed(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_dsmem4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// s[0..15] = sum over the CTAs c_lo + 1 .. c_hi, in that order, of their partials of
// `tile` (rows c0 .. c0 + 15 of this thread's channel). Stream-K ranges of at least a
// tile's k blocks give a split tile two parts, so this is one partial's loads.
template <int BN>
__device__ __forceinline__ void sum_partials(const float* __restrict__ slots, int c_lo, int c_hi, int64_t tile,
                                             int64_t T, int G, int KB, int chan, int c0, float (&s)[16]) {
  float4 acc[4];
  for (int c = c_lo + 1; c <= c_hi; ++c) {
    const float4* p = reinterpret_cast<const float4*>(slots + split_slot(c, tile, T, G, KB) * (BN * 128) +
                                                      static_cast<int64_t>(chan) * BN + c0);
    float4 t[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) t[i] = __ldcg(p + i);
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = c == c_lo + 1 ? t[i] : add4(acc[i], t[i]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    s[4 * i] = acc[i].x, s[4 * i + 1] = acc[i].y, s[4 * i + 2] = acc[i].z, s[4 * i + 3] = acc[i].w;
  }
}

template <int BN, bool F8>
__global__ void __launch_bounds__(TcCfg<BN, F8>::THREADS, TcCfg<BN, F8>::PER_SM)
    tc_linear_kernel(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapX,
                     void* __restrict__ out, int ldo, int R, int N, int K, const float* __restrict__ alpha,
                     const float* __restrict__ beta, const float* __restrict__ wscale, int mode,
                     const int* __restrict__ rows_dev, unsigned* red_cnt, float* red_slots, int cs,
                     unsigned* dev_err) {
  using C = TcCfg<BN, F8>;
  extern __shared__ uint8_t smem_raw[];
  // full: TMA bytes landed; conv (e4m3 only): the bf16 weight tile is written;
  // empty: the MMAs reading the stage completed
  __shared__ uint64_t full_bar[C::STAGES], conv_bar[C::STAGES], empty_bar[C::STAGES], acc_full[2], acc_empty[2],
      drain_bar, recv_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ int64_t issued, consumed;

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // rows_dev: the activation rows are counted on the device by the kernel before this
  // one (at most R; the partition below follows the count, so no weight is streamed
  // for absent rows and none is requested before the wait)
  if (rows_dev) {
    pdl_wait();
    R = min(R, LDCG(rows_dev));
  }
  // tiles are numbered weight tile fastest (tile = r * mt + m): the CTAs running at the
  // same time hold neighbouring ranges, so the row tiles that need one weight tile ask
  // for it together and DRAM serves it once
  const int mt = (N + 127) >> 7, rt = (R + BN - 1) / BN, KB = (K + 63) >> 6;
  const int64_t T = static_cast<int64_t>(mt) * rt * KB;
  int64_t it0, it1;
  if (cs) {
    // cluster split-K (fewer tiles than CTAs): cluster c takes tile c, its cs CTAs one
    // share of the k blocks each, in rank order; the tile is summed through the
    // cluster's shared memory below. A cluster past the tiles present leaves whole.
    const int c = blockIdx.x / cs, rk = blockIdx.x - c * cs;
    if (c >= mt * rt) return;
    it0 = static_cast<int64_t>(c) * KB + KB * rk / cs;
    it1 = static_cast<int64_t>(c) * KB + KB * (rk + 1) / cs;
  } else {
    it0 = T * blockIdx.x / gridDim.x;
    it1 = T * (blockIdx.x + 1) / gridDim.x;
    if (it0 == it1) return;  // fewer units than CTAs (a device row count below the launch's)
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&conv_bar[s], 4);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    issued = 0;
    consumed = 0;
    if (C::PUSH && cs) {
      // every rank's share of this rank's channels: cs x nch x BN floats
      const int rk = blockIdx.x % cs, nch = 128 * (rk + 1) / cs - 128 * rk / cs;
      mbar_init(&recv_bar, 1);
      mbar_arrive_expect_tx(&recv_bar, static_cast<uint32_t>(cs * nch * BN * 4));
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  // push mode: the peers push only after this barrier phase, once every receive
  // barrier of the cluster is initialised
  if (C::PUSH && cs) cluster_arrive_relaxed();

  pdl_trigger();
  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      const uint64_t pol_w = l2_policy_evict_first(), pol_x = l2_policy_evict_last();
      // The weights depend on no earlier kernel: the first stages' weight tiles are
      // requested before waiting for the kernel that produced the activations.
      const int pre = static_cast<int>(min(static_cast<int64_t>(C::STAGES), it1 - it0));
      for (int i = 0; i < pre; ++i) {
        const int64_t tile = (it0 + i) / KB;
        const int kb = static_cast<int>(it0 + i - tile * KB);
        const int m = static_cast<int>(tile % mt);
        mbar_arrive_expect_tx(&full_bar[i], C::TX_BYTES);
        tma_load_2d(smem + i * C::STAGE_BYTES + (F8 ? C::A_BYTES + C::B_BYTES : 0), &mapW, &full_bar[i], kb * 64,
                    m * 128, pol_w);
      }
      pdl_wait();
      for (int i = 0; i < pre; ++i) {
        const int64_t tile = (it0 + i) / KB;
        const int kb = static_cast<int>(it0 + i - tile * KB);
        const int r = static_cast<int>(tile / mt);
        tma_load_2d(smem + i * C::STAGE_BYTES + C::A_BYTES, &mapX, &full_bar[i], kb * 64, r * BN, pol_x);
      }
      issued = pre;
      int stage = pre % C::STAGES;
      uint32_t phase = pre == C::STAGES ? 1u : 0u;
      for (int64_t it = it0 + pre; it < it1; ++it) {
        const int64_t tile = it / KB;
        const int kb = static_cast<int>(it - tile * KB);
        const int r = static_cast<int>(tile / mt), m = static_cast<int>(tile - static_cast<int64_t>(r) * mt);
        if (!mbar_wait(&empty_bar[stage], phase ^ 1u, &abort_flag)) break;
        uint8_t* sa = smem + stage * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&full_bar[stage], C::TX_BYTES);
        tma_load_2d(sa + (F8 ? C::A_BYTES + C::B_BYTES : 0), &mapW, &full_bar[stage], kb * 64, m * 128, pol_w);
        tma_load_2d(sa + C::A_BYTES, &mapX, &full_bar[stage], kb * 64, r * BN, pol_x);
        ++issued;
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(128, BN);
      int stage = 0;
      uint32_t phase = 0;
      int seg = 0;
      int64_t it = it0;
      bool ok = true;
      while (ok && it < it1) {
        const int64_t tile = it / KB;
        const int64_t seg_end = min(it1, (tile + 1) * KB);
        const int buf = seg & 1;
        const uint32_t aph = (seg >> 1) & 1;
        if (!mbar_wait(&acc_empty[buf], aph ^ 1u, &abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(buf * BN);
        bool first = true;
        for (; it < seg_end; ++it) {
          if (!mbar_wait(F8 ? &conv_bar[stage] : &full_bar[stage], phase, &abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          ++consumed;
          const uint32_t sa = base + stage * C::STAGE_BYTES;
          const uint64_t ad = sdesc_sw128(sa), bd = sdesc_sw128(sa + C::A_BYTES);
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // 4 x (K = 16) per 64-wide block; +32 B per step
            umma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (first && k == 0) ? 0u : 1u);
          }
          first = false;
          umma_commit(&empty_bar[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&acc_full[buf]);
        ++seg;
      }
      umma_commit(&drain_bar);  // every MMA issued above has completed past this wait
      if (!mbar_wait_timed(&drain_bar, 0)) abort_flag = 1;
    }
  } else if (F8 && warp >= 6) {  // converters: warps 6..9, 128 threads
    const int t = threadIdx.x - 192;
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t it = it0; it < it1; ++it) {
      if (!mbar_wait(&full_bar[stage], phase, &abort_flag)) break;
      const uint8_t* a8 = smem + stage * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES;
      uint8_t* a16 = smem + stage * C::STAGE_BYTES;
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // 512 chunks of 16 e4m3: row = chunk / 4, 16-byte column c = chunk % 4
        const int chunk = t + 128 * j, row = chunk >> 2, c = chunk & 3;
        uint4 lo, hi;
        e4m3x16_to_bf16(*reinterpret_cast<const uint4*>(a8 + row * 64 + c * 16), lo, hi);
        // 128B swizzle: 16-byte chunk q of row `row` sits at q ^ (row % 8)
        *reinterpret_cast<uint4*>(a16 + row * 128 + (((2 * c) ^ (row & 7)) << 4)) = lo;
        *reinterpret_cast<uint4*>(a16 + row * 128 + (((2 * c + 1) ^ (row & 7)) << 4)) = hi;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(&conv_bar[stage]);
      if (++stage == C::STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  } else {  // epilogue: warps 2..5, TMEM lane quadrant warp % 4, output channels q*32..q*32+31
    pdl_wait();
    const int q = warp & 3, chan = q * 32 + lane, G = gridDim.x, bid = blockIdx.x;
    auto emit = [&](int row, int n, float y) { emit_out(mode, out, ldo, row, n, y); };
    if (C::PUSH && cs) {  // one segment: each channel's partial goes to the rank that sums it
      cluster_wait();
      if (mbar_wait(&acc_full[0], 0, &abort_flag)) {
        tc_fence_after();
        const int rk = bid % cs, nmax = (128 + cs - 1) / cs;
        const int o = ((chan + 1) * cs - 1) >> 7;  // the largest o with 128 o / cs <= chan
        const uint32_t slot = smem_u32(smem + C::STAGES * C::STAGE_BYTES) +
                              static_cast<uint32_t>(((rk * nmax + chan - 128 * o / cs) * (BN + 4)) * 4);
        const uint32_t dst = cluster_map(slot, static_cast<uint32_t>(o));
        const uint32_t bar = cluster_map(smem_u32(&recv_bar), static_cast<uint32_t>(o));
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 16) {
          float v[16];
          tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c0), v);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            st_async4(dst + static_cast<uint32_t>((c0 + 4 * i) * 4), v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3],
                      bar);
        }
      }
    } else if (cs) {  // one segment: the raw partial goes to this CTA's shared memory (stage
                      // area, free once the MMAs completed), channel-major, rows padded by 4
      if (mbar_wait(&acc_full[0], 0, &abort_flag)) {
        tc_fence_after();
        float* part = reinterpret_cast<float*>(smem) + chan * (BN + 4);
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 16) {
          float v[16];
          tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c0), v);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            reinterpret_cast<float4*>(part + c0)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
      }
    }
    int seg = 0;
    int64_t it = cs ? it1 : it0;
    while (it < it1) {
      const int64_t tile = it / KB;
      const int kb0 = static_cast<int>(it - tile * KB);
      const int64_t tile_end = (tile + 1) * KB;
      const int64_t seg_end = min(it1, tile_end);
      const int r = static_cast<int>(tile / mt), m = static_cast<int>(tile - static_cast<int64_t>(r) * mt);
      const int buf = seg & 1;
      const uint32_t aph = (seg >> 1) & 1;
      const int n = m * 128 + chan;
      float a = 1.f, b = 0.f;
      if (n < N) {
        if (alpha) a = alpha[n];
        if (F8) a *= wscale[n];  // the weight's per-output-channel scale
        if (beta) b = beta[n];
      }
      const bool head = kb0 == 0, tail = seg_end == tile_end;
      const uint32_t tacc = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN);
      if (head && tail) {  // the whole k range is here
        if (!mbar_wait(&acc_full[buf], aph, &abort_flag)) break;
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 16) {
          const int row0 = r * BN + c0;
          if (FM_GEMM_ADD_RMW && BN >= 64 && mode == static_cast<int>(Out::Add)) {
            // one writer per element: read, add and write back (the 16 rows' loads
            // issued together, before the accumulator read) instead of L2 reductions
            float o16[16];
            float* op = static_cast<float*>(out) + static_cast<int64_t>(row0) * ldo + n;
#pragma unroll
            for (int j = 0; j < 16; ++j) o16[j] = (n < N && row0 + j < R) ? __ldcg(op + static_cast<int64_t>(j) * ldo) : 0.f;
            float v[16];
            tmem_ld16(tacc + static_cast<uint32_t>(c0), v);
            if (n < N) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (row0 + j < R) op[static_cast<int64_t>(j) * ldo] = o16[j] + fmaf(a, v[j], b);
            }
            continue;
          }
          float v[16];
          tmem_ld16(tacc + static_cast<uint32_t>(c0), v);
          if (n < N) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (row0 + j < R) emit(row0 + j, n, fmaf(a, v[j], b));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      } else {  // a split tile: CTAs c_lo .. c_hi hold its k range in order
        const int c_lo = head ? bid : unit_owner(tile * KB, T, G);
        const int c_hi = tail ? bid : unit_owner(tile_end - 1, T, G);
        unsigned* cnt = red_cnt + 4 * c_lo + q;
        float* mine = red_slots + split_slot(bid, tile, T, G, KB) * (BN * 128) + static_cast<int64_t>(chan) * BN;
        // The first k blocks' CTA (head) comes here at the end of its range, after the
        // others; once it sees all of them counted it is the one that sums, and it
        // loads their partials while its own MMAs finish (narrow tiles: in registers).
        bool reduce_here = false;
        constexpr int PRE = 16;
        float pre[PRE];
        if (head) {
          // every lane reads the count with acquire order; all must see it complete
          reduce_here = __all_sync(0xffffffffu, ld_acquire_u32(cnt) == static_cast<unsigned>(c_hi - c_lo));
          if (reduce_here && BN == 16) {
#pragma unroll
            for (int c0 = 0; c0 < PRE; c0 += 16) {
              float s16[16];
              sum_partials<BN>(red_slots, c_lo, c_hi, tile, T, G, KB, chan, c0, s16);
#pragma unroll
              for (int j = 0; j < 16; ++j) pre[c0 + j] = s16[j];
            }
          }
        }
        if (!mbar_wait(&acc_full[buf], aph, &abort_flag)) break;
        tc_fence_after();
        if (reduce_here) {  // (others, in CTA order) + own, written out
          if constexpr (BN == 16) {
            float v[16];
            tmem_ld16(tacc, v);
            const int row0 = r * BN;
            if (n < N) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (row0 + j < R) emit(row0 + j, n, fmaf(a, pre[j] + v[j], b));
            }
          } else if (c_hi == c_lo + 1) {
            // the usual case (tiles at least as many as CTAs: two parts): the other
            // part's next 16 rows are requested while this chunk is summed
            const float4* op = reinterpret_cast<const float4*>(
                red_slots + split_slot(c_hi, tile, T, G, KB) * (BN * 128) + static_cast<int64_t>(chan) * BN);
            float4 cur[4], nxt[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) cur[i] = __ldcg(op + i);
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 16) {
              if (c0 + 16 < BN) {
#pragma unroll
                for (int i = 0; i < 4; ++i) nxt[i] = __ldcg(op + (c0 + 16) / 4 + i);
              }
              float v[16];
              tmem_ld16(tacc + static_cast<uint32_t>(c0), v);
              const float o16[16] = {cur[0].x, cur[0].y, cur[0].z, cur[0].w, cur[1].x, cur[1].y, cur[1].z, cur[1].w,
                                     cur[2].x, cur[2].y, cur[2].z, cur[2].w, cur[3].x, cur[3].y, cur[3].z, cur[3].w};
              const int row0 = r * BN + c0;
              if (n < N) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  if (row0 + j < R) emit(row0 + j, n, fmaf(a, o16[j] + v[j], b));
              }
#pragma unroll
              for (int i = 0; i < 4; ++i) cur[i] = nxt[i];
            }
          } else {
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 16) {
              float v[16], s16[16];
              tmem_ld16(tacc + static_cast<uint32_t>(c0), v);
              sum_partials<BN>(red_slots, c_lo, c_hi, tile, T, G, KB, chan, c0, s16);
              const int row0 = r * BN + c0;
              if (n < N) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  if (row0 + j < R) emit(row0 + j, n, fmaf(a, s16[j] + v[j], b));
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&acc_empty[buf]);
            *cnt = 0;  // every other CTA of the tile has counted: ready for the next launch
          }
        } else {  // leave the partial and count it; the last to count sums
#pragma unroll 1
          for (int c0 = 0; c0 < BN; c0 += 16) {
            float v[16];
            tmem_ld16(tacc + static_cast<uint32_t>(c0), v);
            float4* p = reinterpret_cast<float4*>(mine + c0);
#pragma unroll
            for (int i = 0; i < 4; ++i) p[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);
          __threadfence();  // this lane's partial is visible before the count
          __syncwarp();
          unsigned ticket = 0;
          if (lane == 0) {
            ticket = atomicAdd(cnt, 1u);
            __threadfence();
          }
          ticket = __shfl_sync(0xffffffffu, ticket, 0);
          if (ticket == static_cast<unsigned>(c_hi - c_lo)) {  // last of all c_hi - c_lo + 1 CTAs
            __threadfence();
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 16) {
              float s16[16];
              sum_partials<BN>(red_slots, c_lo, c_hi, tile, T, G, KB, chan, c0, s16);
              const float4* p0 = reinterpret_cast<const float4*>(
                  red_slots + split_slot(c_lo, tile, T, G, KB) * (BN * 128) + static_cast<int64_t>(chan) * BN + c0);
              float v[16];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float4 t = __ldcg(p0 + i);
                v[4 * i] = t.x, v[4 * i + 1] = t.y, v[4 * i + 2] = t.z, v[4 * i + 3] = t.w;
              }
              const int row0 = r * BN + c0;
              if (n < N) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  if (row0 + j < R) emit(row0 + j, n, fmaf(a, s16[j] + v[j], b));
              }
            }
            __syncwarp();
            if (lane == 0) *cnt = 0;
          }
        }
      }
      it = seg_end;
      ++seg;
    }
  }

  __syncthreads();
  if (C::PUSH && cs) {
    // Rank rk sums channels [128 rk / cs, 128 (rk + 1) / cs) over the ranks' slots in
    // rank order once its receive barrier has counted every byte. The barrier phase
    // after it keeps every CTA resident until all pushes have landed.
    if (warp >= 2 && warp < 6) {
      const bool got = mbar_wait_cluster_timed(&recv_bar, 0);
      cluster_arrive();
      if (got) {
        const int c = blockIdx.x / cs, rk = blockIdx.x - c * cs, nmax = (128 + cs - 1) / cs;
        const int rtile = c / mt, m = c - rtile * mt;
        const int ch0 = 128 * rk / cs, nch = 128 * (rk + 1) / cs - ch0, groups = BN / 4;
        const float* recv = reinterpret_cast<const float*>(smem + C::STAGES * C::STAGE_BYTES);
        for (int i = threadIdx.x - 64; i < nch * groups; i += 128) {
          const int g = i / nch, ch = i - g * nch;  // neighbouring threads: neighbouring channels
          const float* src = recv + ch * (BN + 4) + 4 * g;
          float4 acc = *reinterpret_cast<const float4*>(src);
          for (int k = 1; k < cs; ++k)
            acc = add4(acc, *reinterpret_cast<const float4*>(src + k * nmax * (BN + 4)));
          const int n = m * 128 + ch0 + ch;
          if (n < N) {
            const float a = alpha ? alpha[n] : 1.f, b = beta ? beta[n] : 0.f;
            const int row0 = rtile * BN + 4 * g;
            const float v4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (row0 + e < R) emit_out(mode, out, ldo, row0 + e, n, fmaf(a, v4[e], b));
          }
        }
      } else if (threadIdx.x == 64) {
        abort_flag = 1;
      }
    } else {
      cluster_wait();  // the first phase (the epilogue warps waited before pushing)
      cluster_arrive();
    }
    cluster_wait();
  } else if (cs) {
    // Every rank's partial is in its shared memory after the first cluster barrier;
    // rank rk sums channels [128 rk / cs, 128 (rk + 1) / cs) of the tile over ranks
    // 0..cs-1 in order and writes them; the second barrier keeps each CTA's shared
    // memory alive until its peers have read it.
    tc_fence_before();
    cluster_sync_all();
    if (warp >= 2 && warp < 6) {
      const int c = blockIdx.x / cs, rk = blockIdx.x - c * cs;
      const int rtile = c / mt, m = c - rtile * mt;
      const int ch0 = 128 * rk / cs, nch = 128 * (rk + 1) / cs - ch0, groups = BN / 4;
      const uint32_t pbase = smem_u32(smem);
      for (int i = threadIdx.x - 64; i < nch * groups; i += 128) {
        const int g = i / nch, ch = ch0 + (i - g * nch);  // neighbouring threads: neighbouring channels
        const uint32_t off = pbase + static_cast<uint32_t>((ch * (BN + 4) + 4 * g) * 4);
        // every rank's value requested before the in-order sum (one round trip, not cs)
        constexpr int kMaxCs = FM_GEMM_CLUSTER_MAX > 8 ? 16 : 8;
        float4 t[kMaxCs];
#pragma unroll
        for (int k = 0; k < kMaxCs; ++k)
          if (k < cs) t[k] = ld_dsmem4(cluster_map(off, static_cast<uint32_t>(k)));
        float4 acc = t[0];
#pragma unroll
        for (int k = 1; k < kMaxCs; ++k)
          if (k < cs) acc = add4(acc, t[k]);
        const int n = m * 128 + ch;
        if (n < N) {
          float a = alpha ? alpha[n] : 1.f;
          if (F8) a *= wscale[n];
          const float b = beta ? beta[n] : 0.f;
          const int row0 = rtile * BN + 4 * g;
          const float v4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (row0 + e < R) emit_out(mode, out, ldo, row0 + e, n, fmaf(a, v4[e], b));
        }
      }
    }
    __syncwarp();
    cluster_sync_all();
  }
  if (threadIdx.x == 0 && abort_flag) {
    // Wait (bounded) for the TMA loads still in flight before the CTA exits.
    for (int64_t i = consumed; i < issued; ++i) {
      mbar_wait_timed(&full_bar[i % C::STAGES], static_cast<uint32_t>((i / C::STAGES) & 1));
    }
    set_dev_error(dev_err, FLASHMAP_DEVERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ CTA-pair GEMM (tcgen05 cta_group::2)
//
// Activation tiles of 256 rows on two SMs: a cluster of two CTAs computes one tile of
// 256 weight channels x 256 activation rows. Rank k keeps weight channels 128 k ..
// 128 k + 127 of the tile (A) and activation rows 128 k .. 128 k + 127 (B) in its own
// shared memory; rank 0 issues one M = 256, N = 256 MMA per 16-wide k step, which
// reads both ranks' halves and leaves each rank's 128 channels x 256 rows in that
// rank's TMEM. Per SM and 64-wide k block that is 32 KB of operands for 4.2 MFLOP,
// against 48 KB for the one-SM 128 x 256 tile. Both ranks' loads of a stage count
// their bytes on rank 0's mbarrier (the pair form of the TMA copy), and rank 0's MMA
// commits free the stage and hand over the accumulator on both ranks (multicast
// commits). Whole tiles: pair p takes tiles p, p + P, ..., numbered activation tile
// fastest. Every tcgen05 instruction of the kernel is of the pair form.

// Pair pipeline depth (6 x 32 KB) and threads: warp 0 TMA, warp 1 MMA (rank 0),
// warps 2-5 epilogue.
constexpr int kPairStages = 6;
constexpr int kPairThreads = 192;
struct PairCfg {
  static constexpr int A_BYTES = 128 * 64 * 2;
  static constexpr int B_BYTES = 128 * 64 * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TX_BYTES = 2 * STAGE_BYTES;  // both ranks' bytes of a stage, counted at rank 0
  // The whole of the SM's shared memory (227 KB less the static part): no CTA of
  // another kernel shares an SM with a pair CTA. (It also leaves 16 KB and more past the
  // ring, so a 256-row read of the last stage's B operand would stay inside it.)
  static constexpr int SMEM = 227 * 1024 - 1024;
  static constexpr uint32_t TMEM_COLS = 512;  // two 256-column accumulators
};

// A TMA tile load into this CTA's shared memory whose bytes count on an mbarrier of
// either CTA of the pair (bar: shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives on `bar` (the same shared-memory offset) in both ranks once the MMAs issued
// so far complete.
__device__ __forceinline__ void umma_commit_pair_both(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}
__device__ __forceinline__ void umma_commit_pair_self(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// One arrive on an mbarrier of a CTA of the cluster (shared::cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cl_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cl_addr) : "memory");
}
// The pipelines' wait for a phase completed from another CTA of the cluster (the
// clock is read only once the first try fails).
__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cl(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait_cl(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_cl(bar, parity)) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      return false;
    }
  }
  return true;
}

__global__ void __launch_bounds__(kPairThreads, 1)
    tc_pair_kernel(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapX,
                   void* __restrict__ out, int ldo, int R, int N, int K, const float* __restrict__ alpha,
                   const float* __restrict__ beta, int mode, unsigned* dev_err) {
  using C = PairCfg;
  constexpr int S = kPairStages;
  extern __shared__ uint8_t smem_raw[];
  // full (rank 0): both ranks' TMA bytes of the stage landed; empty: the MMAs reading
  // the stage completed (both ranks)
  __shared__ uint64_t full_bar[S], empty_bar[S], acc_full[2], acc_empty[2], drain_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ int issued, consumed;

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // the same offset in both ranks
  uint8_t* smem = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = blockIdx.x >> 1, P = gridDim.x >> 1;
  const int mt2 = (N + 255) >> 8, rt = (R + 255) >> 8, KB = (K + 63) >> 6;
  // Whole tiles, numbered activation tile fastest (t = m2 * rt + r) so that the pairs
  // running together share a few weight tiles: pair p takes tiles p, p + P, ...
  const int T2 = mt2 * rt;
  const int ntile = pair < T2 ? (T2 - 1 - pair) / P + 1 : 0;
  const int total = ntile * KB;  // this pair's units (64-wide k blocks)
  if (total == 0) return;        // both ranks of the pair
  auto seg_tile = [&](int g) { return pair + g * P; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 8);  // 4 epilogue warps per rank
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    issued = 0;
    consumed = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both ranks' barriers exist before any remote arrive or commit
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  pdl_trigger();
  if (warp == 0) {
    if (lane == 0) {  // TMA producer of this rank's halves
      const uint64_t pol_w = l2_policy_evict_first(), pol_x = l2_policy_evict_last();
      const uint32_t full0 = cluster_map(smem_u32(&full_bar[0]), 0u);  // rank 0's barriers
      const int row_off = static_cast<int>(rank) * 128;
      // the position advances by one unit per stage; the tile's (m2, r) is recomputed
      // once per segment (no division per stage on this single thread)
      struct Cur {
        int u, g, kb, m2, r;
      };
      auto enter = [&](Cur& c, int g) {
        c.g = g;
        const int t = seg_tile(g);
        c.m2 = t / rt;
        c.r = t - c.m2 * rt;
        c.kb = 0;
      };
      auto next = [&](Cur& c) {
        ++c.u;
        if (++c.kb == KB && c.u < total) enter(c, c.g + 1);
      };
      const int pre = min(S, total);
      Cur c;
      c.u = 0;
      enter(c, 0);
      for (int i = 0; i < pre; ++i, next(c)) {  // weights first: they depend on no earlier kernel
        if (rank == 0) mbar_arrive_expect_tx(&full_bar[i], C::TX_BYTES);
        tma_load_2d_pair(smem + i * C::STAGE_BYTES, &mapW, full0 + i * 8, c.kb * 64, c.m2 * 256 + row_off, pol_w);
      }
      pdl_wait();
      c.u = 0;
      enter(c, 0);
      for (int i = 0; i < pre; ++i, next(c))
        tma_load_2d_pair(smem + i * C::STAGE_BYTES + C::A_BYTES, &mapX, full0 + i * 8, c.kb * 64, c.r * 256 + row_off,
                         pol_x);
      issued = pre;
      int stage = pre % S;
      uint32_t phase = pre == S ? 1u : 0u;
      for (; c.u < total; next(c)) {
        if (!mbar_wait(&empty_bar[stage], phase ^ 1u, &abort_flag)) break;
        uint8_t* sa = smem + stage * C::STAGE_BYTES;
        if (rank == 0) mbar_arrive_expect_tx(&full_bar[stage], C::TX_BYTES);
        tma_load_2d_pair(sa, &mapW, full0 + stage * 8, c.kb * 64, c.m2 * 256 + row_off, pol_w);
        tma_load_2d_pair(sa + C::A_BYTES, &mapX, full0 + stage * 8, c.kb * 64, c.r * 256 + row_off, pol_x);
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {  // the MMA issuer for the pair: one accumulator per tile
      constexpr uint32_t idesc = idesc_bf16_f32(256, 256);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int g = 0; ok && g < ntile; ++g) {
        const int buf = g & 1;
        const uint32_t aph = (g >> 1) & 1;
        if (!mbar_wait_cl(&acc_empty[buf], aph ^ 1u, &abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(buf * 256);
        for (int k64 = 0; k64 < KB; ++k64) {
          if (!mbar_wait_cl(&full_bar[stage], phase, &abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          ++consumed;
          const uint32_t sa = base + stage * C::STAGE_BYTES;
          const uint64_t ad = sdesc_sw128(sa), bd = sdesc_sw128(sa + C::A_BYTES);
#pragma unroll
          for (int k = 0; k < 4; ++k) umma_bf16_pair(d, ad + 2 * k, bd + 2 * k, idesc, (k64 == 0 && k == 0) ? 0u : 1u);
          umma_commit_pair_both(&empty_bar[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_both(&acc_full[buf]);
      }
      umma_commit_pair_self(&drain_bar);  // every MMA issued above has completed past this wait
      if (!mbar_wait_timed(&drain_bar, 0)) abort_flag = 1;
    }
  } else {  // epilogue: warps 2..5, TMEM lane quadrant warp % 4 = 32 of this rank's channels
    pdl_wait();
    const int q = warp & 3, chan = q * 32 + lane;
    const uint32_t empty0 = cluster_map(smem_u32(&acc_empty[0]), 0u);
    const bool add = mode == static_cast<int>(Out::Add);
    for (int g = 0; g < ntile; ++g) {
      const int t = seg_tile(g), m2 = t / rt, r = t - m2 * rt;
      const int n = m2 * 256 + static_cast<int>(rank) * 128 + chan;
      float a = 1.f, b = 0.f;
      if (n < N) {
        if (alpha) a = alpha[n];
        if (beta) b = beta[n];
      }
      const int buf = g & 1;
      const uint32_t tacc = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * 256);
      float* op = static_cast<float*>(out) + static_cast<int64_t>(r) * 256 * ldo + n;  // (row r * 256, n)
      // the 16 output values of rows c0 .. c0 + 15 that an addition reads (issued a
      // chunk ahead)
      auto load_out = [&](int c0, float (&o16)[16]) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          o16[j] = (n < N && r * 256 + c0 + j < R) ? __ldcg(op + static_cast<int64_t>(c0 + j) * ldo) : 0.f;
      };
      const int nrows = min(256, R - r * 256);  // rows of this tile present (> 0)
      float on[16];
      if (add) load_out(0, on);  // the first chunk's output, before the accumulator wait
      if (!mbar_wait(&acc_full[buf], (g >> 1) & 1, &abort_flag)) break;
      tc_fence_after();
#pragma unroll 1
      for (int c0 = 0; c0 < nrows; c0 += 16) {
        float o16[16], v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) o16[j] = on[j];
        if (add && c0 + 16 < nrows) load_out(c0 + 16, on);
        tmem_ld16(tacc + static_cast<uint32_t>(c0), v);
        if (n < N) {  // rows c0 .. c0 + 15 of this channel: y = a v + b, added onto o16 or written
          const int row0 = r * 256 + c0;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (row0 + j >= R) break;
            if (add)
              op[static_cast<int64_t>(c0 + j) * ldo] = o16[j] + fmaf(a, v[j], b);
            else
              emit_out(mode, out, ldo, row0 + j, n, fmaf(a, v[j], b));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(empty0 + static_cast<uint32_t>(buf * 8));
    }
  }

  if (threadIdx.x == 0 && abort_flag) set_dev_error(dev_err, FLASHMAP_DEVERR_TIMEOUT);
  if (threadIdx.x == 0 && rank == 0 && abort_flag) {
    // Wait (bounded) for the loads still in flight: rank 0's stage barriers count both
    // ranks' bytes of every stage it armed.
    for (int i = consumed; i < issued; ++i) mbar_wait_timed(&full_bar[i % S], static_cast<uint32_t>((i / S) & 1));
  }
  tc_fence_before();
  __syncthreads();
  // rank 0's MMAs (which read rank 1's shared memory) are drained, and rank 1 stays
  // until rank 0 has seen every armed stage land
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ SIMT linear (float32 path)

template <typename T>
__global__ void __launch_bounds__(256) linear_warp_kernel(const T* __restrict__ x, int R, int ldx,
                                                          const T* __restrict__ w, int N, int K,
                                                          void* __restrict__ out, int ldo,
                                                          const float* __restrict__ alpha,
                                                          const float* __restrict__ beta, int mode) {
  constexpr int RB = 4;
  pdl_trigger();
  pdl_wait();
  const int n = static_cast<int>((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (n >= N) return;
  const T* wr = w + static_cast<int64_t>(n) * K;
  const float a = alpha ? alpha[n] : 1.f, b = beta ? beta[n] : 0.f;
  for (int r0 = 0; r0 < R; r0 += RB) {
    float acc[RB] = {0.f, 0.f, 0.f, 0.f};
    for (int k = lane; k < K; k += 32) {
      const float wv = to_f32(wr[k]);
#pragma unroll
      for (int j = 0; j < RB; ++j)
        if (r0 + j < R) acc[j] = fmaf(wv, to_f32(LDCG(x + static_cast<int64_t>(r0 + j) * ldx + k)), acc[j]);
    }
#pragma unroll
    for (int j = 0; j < RB; ++j) {
      const float s = warp_sum(acc[j]);
      if (lane == 0 && r0 + j < R) {  // one writer per element
        const int64_t o = static_cast<int64_t>(r0 + j) * ldo + n;
        const float y = fmaf(a, s, b);
        if (mode == static_cast<int>(Out::Add))
          static_cast<float*>(out)[o] = LDCG(static_cast<const float*>(out) + o) + y;
        else if (mode == static_cast<int>(Out::Store))
          static_cast<float*>(out)[o] = y;
        else
          static_cast<T*>(out)[o] = from_f32<T>(gelu_erf(y));
      }
    }
  }
}

// ------------------------------------------------------------------ general strided SIMT GEMM (load time)

__device__ __forceinline__ float ld_any(const void* p, int dt, int64_t i) {
  return dt == FLASHMAP_F32 ? static_cast<const float*>(p)[i]
                            : __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

__global__ void __launch_bounds__(256) simt_gemm_kernel(int M, int N, int K, int kchunk, const void* a, int adt,
                                                        const int64_t* __restrict__ arows, int64_t sam,
                                                        int64_t sak, const void* b, int bdt, int64_t sbk,
                                                        int64_t sbn, void* c, int cdt, int64_t ldc, int mode) {
  __shared__ float As[16][65], Bs[16][65];
  const int tid = threadIdx.x, tm = tid >> 4, tn = tid & 15;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  // mode 2: the k range in chunks of kchunk, each summed in float32 and added into
  // float64 in chunk order (one block owns its tile: no atomics, a fixed order)
  const int nchunks = mode == 2 ? (K + kchunk - 1) / kchunk : 1;
  double acc64[4][4] = {};
  float acc[4][4];
  for (int chunk = 0; chunk < nchunks; ++chunk) {
  const int kbeg = mode == 2 ? chunk * kchunk : blockIdx.z * kchunk, kend = min(K, kbeg + kchunk);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int k0 = kbeg; k0 < kend; k0 += 16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = tid + 256 * i;
      int mm, kk;
      if (sak == 1) {
        kk = e & 15;
        mm = e >> 4;
      } else {
        mm = e & 63;
        kk = e >> 6;
      }
      const int gm = m0 + mm, gk = k0 + kk;
      float v = 0.f;
      if (gm < M && gk < kend) {
        const int64_t row = arows ? arows[gm] : gm;
        v = ld_any(a, adt, row * sam + static_cast<int64_t>(gk) * sak);
      }
      As[kk][mm] = v;
      int nn;
      if (sbn == 1) {
        nn = e & 63;
        kk = e >> 6;
      } else {
        kk = e & 15;
        nn = e >> 4;
      }
      const int gn = n0 + nn, gk2 = k0 + kk;
      float u = 0.f;
      if (gn < N && gk2 < kend) u = ld_any(b, bdt, static_cast<int64_t>(gk2) * sbk + static_cast<int64_t>(gn) * sbn);
      Bs[kk][nn] = u;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][tm * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tn * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  if (mode == 2) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc64[i][j] += static_cast<double>(acc[i][j]);
  }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + tm * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tn * 4 + j;
      if (gn >= N) continue;
      const int64_t idx = static_cast<int64_t>(gm) * ldc + gn;
      if (mode == 0) {
        static_cast<float*>(c)[idx] = acc[i][j];
      } else if (mode == 1) {
        if (cdt == FLASHMAP_F32)
          static_cast<float*>(c)[idx] = acc[i][j];
        else
          static_cast<__nv_bfloat16*>(c)[idx] = __float2bfloat16_rn(acc[i][j]);
      } else {
        static_cast<double*>(c)[idx] = acc64[i][j];
      }
    }
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

template <int BN, bool F8>
cudaError_t launch_tc(const Launch& L, const Weight& W, const void* x, int R, int ldx, void* out, int ldo,
                      const float* alpha, const float* beta, Out mode, const int* rows_dev) {
  using C = TcCfg<BN, F8>;
  CUtensorMap mapX;
  std::string err;
  if (!make_tmap_bf16(&mapX, x, R, W.K, ldx, BN, &err)) return cudaErrorInvalidValue;
  const int64_t mt = (W.N + 127) / 128, rt = (R + BN - 1) / BN, KB = (W.K + 63) / 64;
  const int64_t T = mt * rt * KB;
  const int per_sm = L.ctas_per_sm > 0 ? std::min(L.ctas_per_sm, C::PER_SM) : C::PER_SM;
  const int64_t Gmax = static_cast<int64_t>(L.num_sms) * per_sm, tiles = mt * rt;
  // At most half as many tiles as CTAs: cluster split-K, cs CTAs per tile (cs <= 8, a
  // portable cluster), summed in the cluster's shared memory. Otherwise stream-K over
  // every CTA, whose ranges then cover at least half a tile's k blocks each.
  const int cs = FM_GEMM_CLUSTER_MAX >= 2 && 2 * tiles <= Gmax && KB >= 2
                     ? static_cast<int>(std::min<int64_t>({FM_GEMM_CLUSTER_MAX, Gmax / tiles, KB}))
                     : 0;
  // Between half as many tiles as CTAs and as many: one whole tile per CTA (stream-K
  // over all the CTAs would give a tile up to three parts, summed at the end of the
  // kernel by its last CTA). From as many tiles as CTAs up: stream-K, two parts at most.
  const int G = cs ? static_cast<int>(tiles * cs)
                   : static_cast<int>(tiles < Gmax ? std::min<int64_t>(tiles, T) : std::min<int64_t>(T, Gmax));
  // the stream-K split-tile scratch: four counters and two BN x 128 slots per CTA
  if (!cs && (!L.red.cnt || !L.red.slots || 4LL * G > L.red.cnt_cap || 2LL * G * BN * 128 > L.red.slot_cap))
    return cudaErrorInvalidValue;
  return launch_kc(L, tc_linear_kernel<BN, F8>, dim3(G), dim3(C::THREADS), C::SMEM, cs, W.map, mapX, out, ldo, R,
                  W.N, W.K, alpha, beta, W.wscale, static_cast<int>(mode), rows_dev, L.red.cnt, L.red.slots, cs,
                  L.dev_err);
}

int tc_bn(int rows) { return rows <= 16 ? 16 : rows <= 32 ? 32 : rows <= 64 ? 64 : rows <= 128 ? 128 : 256; }

// Clusters of two that fit at once (one CTA per SM; SMs that cannot be paired in their
// GPC stay out), cached per device.
int pair_clusters(int num_sms) {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (num_sms / 2));
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = PairCfg::SMEM;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc_pair_kernel, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = num_sms / 2;
  }
  cached[dev] = std::min(n, num_sms / 2);
  return cached[dev];
}

// The pair kernel for bf16 weights at more than 128 rows (host row count), with at
// least FM_GEMM_PAIR_MIN_TILES tiles.
cudaError_t launch_pair(const Launch& L, const Weight& W, const void* x, int R, int ldx, void* out, int ldo,
                        const float* alpha, const float* beta, Out mode, bool* used) {
  *used = false;
  const int64_t T2 = ((W.N + 255) / 256) * static_cast<int64_t>((R + 255) / 256);
  const int pairs = pair_clusters(L.num_sms);
  if (FM_GEMM_PAIR_MIN_TILES <= 0 || T2 < FM_GEMM_PAIR_MIN_TILES) return cudaSuccess;
  CUtensorMap mapX;
  std::string err;
  if (!make_tmap_bf16(&mapX, x, R, W.K, ldx, 128, &err)) return cudaErrorInvalidValue;
  const int P = static_cast<int>(std::min<int64_t>(T2, pairs));
  *used = true;
  return launch_kc(L, tc_pair_kernel, dim3(2 * P), dim3(kPairThreads), PairCfg::SMEM, 2, W.map, mapX, out, ldo, R,
                   W.N, W.K, alpha, beta, static_cast<int>(mode), L.dev_err);
}

template <bool F8>
cudaError_t launch_tc_rows(const Launch& L, const Weight& W, const void* x, int rows, int ldx, void* out, int ldo,
                           const float* alpha, const float* beta, Out mode, const int* rows_dev) {
  if (!F8 && !rows_dev && rows > 128) {
    bool used = false;
    const cudaError_t e = launch_pair(L, W, x, rows, ldx, out, ldo, alpha, beta, mode, &used);
    if (used || e != cudaSuccess) return e;
  }
  switch (tc_bn(rows)) {
    case 16: return launch_tc<16, F8>(L, W, x, rows, ldx, out, ldo, alpha, beta, mode, rows_dev);
    case 32: return launch_tc<32, F8>(L, W, x, rows, ldx, out, ldo, alpha, beta, mode, rows_dev);
    case 64: return launch_tc<64, F8>(L, W, x, rows, ldx, out, ldo, alpha, beta, mode, rows_dev);
    case 128: return launch_tc<128, F8>(L, W, x, rows, ldx, out, ldo, alpha, beta, mode, rows_dev);
    default: return launch_tc<256, F8>(L, W, x, rows, ldx, out, ldo, alpha, beta, mode, rows_dev);
  }
}

// The most CTAs a launch of BN-row tiles can have (either weight type).
template <int BN>
int64_t tc_max_ctas(int num_sms) {
  return static_cast<int64_t>(num_sms) * std::max(TcCfg<BN, false>::PER_SM, TcCfg<BN, true>::PER_SM);
}
int64_t tc_slot_floats(int bn, int num_sms) {
  switch (bn) {
    case 16: return 2 * tc_max_ctas<16>(num_sms) * 16 * 128;
    case 32: return 2 * tc_max_ctas<32>(num_sms) * 32 * 128;
    case 64: return 2 * tc_max_ctas<64>(num_sms) * 64 * 128;
    case 128: return 2 * tc_max_ctas<128>(num_sms) * 128 * 128;
    default: return 2 * tc_max_ctas<256>(num_sms) * 256 * 128;
  }
}
int64_t tc_cnt_entries(int num_sms) { return 4LL * num_sms * FM_TC_CTAS_PER_SM; }

template <int BN, bool F8>
cudaError_t set_tc_attr() {
  cudaError_t e = cudaFuncSetAttribute(tc_linear_kernel<BN, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TcCfg<BN, F8>::SMEM);
  if (e == cudaSuccess && FM_GEMM_CLUSTER_MAX > 8)
    e = cudaFuncSetAttribute(tc_linear_kernel<BN, F8>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

template <bool F8>
cudaError_t set_tc_attrs() {
  cudaError_t e;
  if ((e = set_tc_attr<16, F8>()) != cudaSuccess) return e;
  if ((e = set_tc_attr<32, F8>()) != cudaSuccess) return e;
  if ((e = set_tc_attr<64, F8>()) != cudaSuccess) return e;
  if ((e = set_tc_attr<128, F8>()) != cudaSuccess) return e;
  return set_tc_attr<256, F8>();
}

}  // namespace

cudaError_t gemm_prepare() {
  cudaError_t e = set_tc_attrs<false>();
  if (e == cudaSuccess) e = set_tc_attrs<true>();
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PairCfg::SMEM);
  return e;
}

bool make_tmap_bf16(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_rows,
                    std::string* err) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    if (err) *err = "cuTensorMapEncodeTiled is not available from the driver";
    return false;
  }
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) || ((ld * 2) & 15) || cols <= 0 || rows <= 0) {
    if (err) *err = "tensor map operand must be 16-byte aligned with a 16-byte multiple row pitch";
    return false;
  }
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (err) *err = "cuTensorMapEncodeTiled failed (" + std::to_string(static_cast<int>(r)) + ")";
    return false;
  }
  return true;
}

bool make_tmap_e4m3(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, std::string* err) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    if (err) *err = "cuTensorMapEncodeTiled is not available from the driver";
    return false;
  }
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) || (cols & 15) || cols <= 0 || rows <= 0) {
    if (err) *err = "an e4m3 weight must be 16-byte aligned with a multiple of 16 columns";
    return false;
  }
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
  const cuuint32_t box[2] = {64, 128};  // 64 bytes x 128 rows, unswizzled
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (err) *err = "cuTensorMapEncodeTiled failed (" + std::to_string(static_cast<int>(r)) + ")";
    return false;
  }
  return true;
}

size_t gemm_scratch_bytes(int max_rows, int num_sms) {
  int64_t slots = 0;
  for (int bn = 16; bn <= tc_bn(std::max(max_rows, 1)); bn *= 2) slots = std::max(slots, tc_slot_floats(bn, num_sms));
  const size_t cnt = (static_cast<size_t>(tc_cnt_entries(num_sms)) * 4 + 255) / 256 * 256;
  return cnt + static_cast<size_t>(slots) * 4;
}

GemmScratch gemm_scratch_carve(void* base, int max_rows, int num_sms) {
  GemmScratch g;
  const size_t cnt = (static_cast<size_t>(tc_cnt_entries(num_sms)) * 4 + 255) / 256 * 256;
  g.cnt = static_cast<unsigned*>(base);
  g.cnt_cap = tc_cnt_entries(num_sms);
  g.slots = reinterpret_cast<float*>(static_cast<uint8_t*>(base) + cnt);
  g.slot_cap = static_cast<int64_t>((gemm_scratch_bytes(max_rows, num_sms) - cnt) / 4);
  return g;
}

cudaError_t linear(const Launch& L, const Weight& W, const void* x, int rows, int ldx, void* out, int ldo,
                   const float* alpha, const float* beta, Out mode, const int* rows_dev) {
  if (rows <= 0 || W.N <= 0) return cudaSuccess;
  if (W.dtype == FLASHMAP_BF16) {
    if (!W.has_map) return cudaErrorInvalidValue;
    return launch_tc_rows<false>(L, W, x, rows, ldx, out, ldo, alpha, beta, mode, rows_dev);
  }
  if (W.dtype == FLASHMAP_E4M3) {  // e4m3 weights, bf16 activations
    if (!W.has_map || !W.wscale) return cudaErrorInvalidValue;
    return launch_tc_rows<true>(L, W, x, rows, ldx, out, ldo, alpha, beta, mode, rows_dev);
  }
  if (rows_dev) return cudaErrorInvalidValue;  // device row counts: tcgen05 weights only
  if (W.dtype == FLASHMAP_F32) {
    const int64_t threads = static_cast<int64_t>(W.N) * 32;
    const int blocks = static_cast<int>((threads + 255) / 256);
    return launch_k(L, linear_warp_kernel<float>, dim3(blocks), dim3(256), 0, static_cast<const float*>(x), rows,
                    ldx, static_cast<const float*>(W.ptr), W.N, W.K, out, ldo, alpha, beta, static_cast<int>(mode));
  }
  return cudaErrorInvalidValue;
}

cudaError_t simt_gemm(cudaStream_t s, int M, int N, int K, const void* a, int a_dtype, const int64_t* a_rows,
                      int64_t sam, int64_t sak, const void* b, int b_dtype, int64_t sbk, int64_t sbn, void* c,
                      int c_dtype, int64_t ldc, int mode) {
  if (M <= 0 || N <= 0 || K <= 0) return cudaSuccess;
  // mode 2: float32 partial sums over 1024-long k ranges, added in float64 in order
  const int kchunk = mode == 2 ? 1024 : K;
  dim3 grid((N + 63) / 64, (M + 63) / 64, 1);
  simt_gemm_kernel<<<grid, 256, 0, s>>>(M, N, K, kchunk, a, a_dtype, a_rows, sam, sak, b, b_dtype, sbk, sbn, c,
                                        c_dtype, ldc, mode);
  return cudaGetLastError();
}

}  // namespace fm
