// Split-K FP8 decode GEMM (m <= 64) on tcgen05 tensor cores: the same linear
// and the same split-K partition as decode_gemm.cu (see there), for the m where
// the warp-level mma.sync path cannot keep up with HBM.
//
//   Y[m, o] = bf16_rne( sum_kb s[o/128, kb] * sum_{i in kb} x[m, i] * e4m3(q[o, i]) )
//
// Swap-AB: the weight rows are the MMA's M = 128 dimension and the
// activations its N = 16..64 dimension (m rounded up to 16).
//   * warp 0, one thread: TMA producer. Per unit (256 weight rows x 128 K) it
//     loads the e4m3 weight slab (128-byte swizzle) and the raw bf16 activation
//     slab [N, 128] into one of 4-5 shared-memory stages.
//   * warps 2-9 (each owns one quarter of the TMEM lanes of one of the unit's
//     two 128-row tiles): convert every weight row exactly (e4m3 -> f16)
//     straight into TMEM, where it is the MMA's A
//     operand, and the activations (bf16 -> f16, saturating) into the 128-byte
//     swizzled B layout in shared memory; then, one unit behind, read the MMA's
//     per-slab result from TMEM and add it, times the slab's 128 x 128 block
//     scale, into fp32 registers (exact block scaling, as in the prefill GEMM).
//   * warp 1: allocates TMEM and issues tcgen05.mma kind::f16 with A in TMEM:
//     2 tiles x 8 MMAs (128 x N x 16) per unit into two D buffers.
// Converted weights never pass through shared memory, so shared-memory traffic
// stays at about 2 bytes per weight byte (TMA write + conversion read).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "decode_common.cuh"
#include "ptx.cuh"
#include "sws_internal.h"

namespace sws {
namespace {

using namespace dec;

constexpr int kTcRows = 256;  // weight rows per unit: two 128-row MMA tiles
constexpr int kTcWarps = 10;  // 0 producer, 1 MMA, 2..9 workers (one per tile and TMEM lane quarter)
constexpr int kWorkers = 8;
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTmemCols = 512;

template <int N>
struct TcCfg {
  static constexpr int kWBytes = kTcRows * kSlabK;     // e4m3 weight slab
  static constexpr int kXRawBytes = N * kSlabK * 2;    // bf16 activations [N][128]
  static constexpr int kStageBytes = kWBytes + kXRawBytes;
  static constexpr int kXBytes = N * kSlabK * 2;       // f16 B operand: two 128-byte atoms per row
  static constexpr int kStages = N <= 32 ? 5 : 4;
  static constexpr int kSmem = kStages * kStageBytes + 2 * kXBytes + 1024;
  static constexpr int kSlotFloats = kTcRows * N;      // partial-sum slot of one CTA
};

__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);  // start address
  d |= (uint64_t)1 << 16;                  // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;        // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                  // descriptor version
  d |= (uint64_t)2 << 61;                  // SWIZZLE_128B
  return d;
}

// kind::f16 instruction descriptor: A, B f16, D f32, K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D (TMEM) (+)= A (TMEM) x B (shared memory).
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   dev::smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Barrier among the 8 worker warps only (named barrier 1).
__device__ __forceinline__ void workers_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Scale of 128-row tile t of a unit (0 past the last row).
__device__ __forceinline__ float tile_scale(const DecodeParams& p, const UnitPos& up, int t) {
  const DecodeEntry& e = p.e[up.j];
  const int64_t row0 = up.rbl * kTcRows + t * 128;
  return row0 < e.rows ? __ldg(e.scales + (row0 >> 7) * e.scale_cols + up.kb) : 0.f;
}

// Each worker thread owns row `row` of tile `t` (0 or 1) of every unit.
template <int N>
__device__ __forceinline__ void tc_write_y(const float (&acc)[N], const DecodeParams& p, const UnitPos& up, int t,
                                           int row) {
  const DecodeEntry& e = p.e[up.j];
  const int64_t o = up.rbl * kTcRows + t * 128 + row;
  if (o < e.rows) {
#pragma unroll
    for (int mm = 0; mm < N; ++mm)
      if (mm < p.m) {
        const __nv_bfloat16 b = __float2bfloat16_rn(acc[mm]);
        e.y[(int64_t)mm * e.rows + o] = *reinterpret_cast<const uint16_t*>(&b);
      }
  }
}

template <int N>
__device__ __forceinline__ void tc_end_run(float (&acc)[N], const DecodeParams& p, const RunGeom& geo,
                                           const UnitPos& up, int t, int row) {
  if (!geo.partial(p, up.rbg)) {
    tc_write_y<N>(acc, p, up, t, row);
  } else {
    float4* d = reinterpret_cast<float4*>(p.partials + geo.slot(p, geo.c, up.rbg) * (int64_t)TcCfg<N>::kSlotFloats +
                                          (t * 128 + row) * N);
#pragma unroll
    for (int q = 0; q < N / 4; ++q) d[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
  }
#pragma unroll
  for (int mm = 0; mm < N; ++mm) acc[mm] = 0.f;
}

// After the CTA's last unit: arrival counts on its (at most two) partial row
// blocks; the last CTA to arrive adds the partials in K order and writes Y.
template <int N>
__device__ __forceinline__ void tc_settle(const DecodeParams& p, const RunGeom& geo, int64_t u_first,
                                          int64_t u_last, int wt, int t, int row, int* s_last) {
  const UnitPos uf = unit_pos(p, u_first), ul = unit_pos(p, u_last);
  const bool pf = geo.partial(p, uf.rbg), pl = ul.rbg != uf.rbg && geo.partial(p, ul.rbg);
  if (!pf && !pl) return;
  __threadfence();
  workers_sync();
  if (wt == 0) {
    int last = 0;
    if (pf)
      last |= (atomicAdd(p.counters + uf.rbg, 1) == (int)(geo.last_cta(p, uf.rbg) - geo.first_cta(p, uf.rbg)));
    if (pl)
      last |= (atomicAdd(p.counters + ul.rbg, 1) == (int)(geo.last_cta(p, ul.rbg) - geo.first_cta(p, ul.rbg))) << 1;
    *s_last = last;
  }
  workers_sync();
  const int last = *s_last;
  if (!last) return;
  __threadfence();
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {
    if (!(last & (1 << which))) continue;
    const UnitPos& up = which == 0 ? uf : ul;
    const int64_t cf = geo.first_cta(p, up.rbg), cl = geo.last_cta(p, up.rbg);
    float acc[N];
#pragma unroll
    for (int mm = 0; mm < N; ++mm) acc[mm] = 0.f;
    for (int64_t cc = cf; cc <= cl; ++cc) {  // K order: the sum does not depend on who arrived last
      const float4* s4 = reinterpret_cast<const float4*>(
          p.partials + geo.slot(p, cc, up.rbg) * (int64_t)TcCfg<N>::kSlotFloats + (t * 128 + row) * N);
#pragma unroll
      for (int q = 0; q < N / 4; ++q) {
        const float4 v = __ldcg(s4 + q);
        acc[4 * q] += v.x;
        acc[4 * q + 1] += v.y;
        acc[4 * q + 2] += v.z;
        acc[4 * q + 3] += v.w;
      }
    }
    tc_write_y<N>(acc, p, up, t, row);
    if (wt == 0) p.counters[up.rbg] = 0;
  }
}

template <int N>
__global__ void __launch_bounds__(kTcThreads, 1) decode_tc_kernel(const __grid_constant__ DecodeParams p) {
  using Cf = TcCfg<N>;
  constexpr int S = Cf::kStages;
  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t sfull[S], sempty[S], abfull[2], abempty[2], dfull[2], dempty[2], mdone;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ int s_last;
  // Swizzled TMA tiles and MMA operands need 1024-byte aligned bases.
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  uint8_t* xbuf = smem + S * Cf::kStageBytes;  // two f16 B operands
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t U = p.units, G = gridDim.x, c = blockIdx.x;
  const int64_t u0 = c * U / G, u1 = (c + 1) * U / G, n = u1 - u0;

  if (tid == 0) {
    dev::trace_start(p.trace);
    for (int s = 0; s < S; ++s) {
      dev::mbar_init(&sfull[s], 1);
      dev::mbar_init(&sempty[s], kWorkers);
    }
    for (int b = 0; b < 2; ++b) {
      dev::mbar_init(&abfull[b], kWorkers);
      dev::mbar_init(&abempty[b], 1);
      dev::mbar_init(&dfull[b], 1);
      dev::mbar_init(&dempty[b], kWorkers);
    }
    dev::mbar_init(&mdone, 1);
    dev::fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dev::smem_addr(&s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const RunGeom geo{G, U, c};

  if (warp == 0) {
    // ---- TMA producer ------------------------------------------------------
    if (lane == 0) {
      int64_t i = 0;
      for (; i < n && !s_abort; ++i) {
        const int s = (int)(i % S);
        if (!dev::mbar_wait(&sempty[s], (uint32_t)(((i / S) & 1) ^ 1), kWaitLimitNs)) {
          dev::set_status(p.status, SWS_E_TIMEOUT);
          s_abort = 1;
          break;
        }
        const UnitPos up = unit_pos(p, u0 + i);
        const DecodeEntry& e = p.e[up.j];
        uint8_t* st = smem + s * Cf::kStageBytes;
        dev::mbar_arrive_expect_tx(&sfull[s], Cf::kStageBytes);
        tma_load_2d(st, &e.tmap, (int32_t)(up.kb * kSlabK), (int32_t)(up.rbl * kTcRows), &sfull[s]);
        tma_load_2d(st + Cf::kWBytes, &e.xmap, (int32_t)(up.kb * kSlabK), 0, &sfull[s]);
      }
      // Before the CTA may exit, every issued stage must have landed.
      for (int64_t k = i - S; k < i; ++k)
        if (k >= 0) dev::mbar_wait(&sfull[(int)(k % S)], (uint32_t)((k / S) & 1), kWaitLimitNs / 4);
    }
  } else if (warp == 1) {
    // ---- MMA issuer ----------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(128, N);
      bool issued = false;
      for (int64_t i = 0; i < n && !s_abort; ++i) {
        const int b = (int)(i & 1);
        if (!dev::mbar_wait(&abfull[b], (uint32_t)((i >> 1) & 1), kWaitLimitNs) ||
            !dev::mbar_wait(&dempty[b], (uint32_t)(((i >> 1) & 1) ^ 1), kWaitLimitNs)) {
          dev::set_status(p.status, SWS_E_TIMEOUT);
          s_abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t xs = dev::smem_addr(xbuf + b * Cf::kXBytes);
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int k = 0; k < kSlabK / 16; ++k)
            mma_f16_ta(tmem + 256 + b * 2 * N + t * N, tmem + b * 128 + t * 64 + k * 8,
                       smem_desc_sw128(xs + (k >> 2) * (N * 128) + (k & 3) * 32), idesc, k > 0);
        mma_commit(&abempty[b]);
        mma_commit(&dfull[b]);
        issued = true;
      }
      if (issued) {  // all MMAs of this CTA complete before TMEM is released
        mma_commit(&mdone);
        dev::mbar_wait(&mdone, 0, kWaitLimitNs);
      }
    }
  } else {
    // ---- workers: convert unit i, promote unit i - 1 ---------------------------------
    const int q = warp & 3;          // TMEM lane quarter of this warp
    const int t = (warp - 2) >> 2;   // the unit's 128-row tile this warp works on
    const int row = q * 32 + lane;   // row inside the tile = TMEM lane
    const int wt = tid - 64;         // worker thread 0..255
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    float acc[N];
#pragma unroll
    for (int mm = 0; mm < N; ++mm) acc[mm] = 0.f;
    float sc_new = 0.f, sc_old = 0.f;
    bool ok = true;
    for (int64_t i = 0; i <= n && ok; ++i) {
      if (i < n) {
        const int s = (int)(i % S), b = (int)(i & 1);
        if (!dev::mbar_wait(&sfull[s], (uint32_t)((i / S) & 1), kWaitLimitNs) ||
            !dev::mbar_wait(&abempty[b], (uint32_t)(((i >> 1) & 1) ^ 1), kWaitLimitNs)) {
          dev::set_status(p.status, SWS_E_TIMEOUT);
          s_abort = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const UnitPos up = unit_pos(p, u0 + i);
        sc_new = tile_scale(p, up, t);  // used when this unit is promoted, one step later
        const uint8_t* st = smem + s * Cf::kStageBytes;
        // weight row `row` of tile t, e4m3 -> f16 into TMEM (A operand)
        const int r = t * 128 + row;
        const uint8_t* wr = st + r * kSlabK;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t h[32];
#pragma unroll
          for (int cq = 0; cq < 4; ++cq) {
            const int cc = hh * 4 + cq;
            const uint4 w = *reinterpret_cast<const uint4*>(wr + ((cc ^ (r & 7)) << 4));
            h[cq * 8 + 0] = e4m3x2_to_f16x2(w.x);
            h[cq * 8 + 1] = e4m3x2_to_f16x2(w.x >> 16);
            h[cq * 8 + 2] = e4m3x2_to_f16x2(w.y);
            h[cq * 8 + 3] = e4m3x2_to_f16x2(w.y >> 16);
            h[cq * 8 + 4] = e4m3x2_to_f16x2(w.z);
            h[cq * 8 + 5] = e4m3x2_to_f16x2(w.z >> 16);
            h[cq * 8 + 6] = e4m3x2_to_f16x2(w.w);
            h[cq * 8 + 7] = e4m3x2_to_f16x2(w.w >> 16);
          }
          tmem_st32(tmem + lane_off + b * 128 + t * 64 + hh * 32, h);
        }
        // activations: bf16 [N][128] -> f16 B operand (two 128-byte swizzled atoms per row)
        uint8_t* xb = xbuf + b * Cf::kXBytes;
#pragma unroll
        for (int k = wt; k < N * 16; k += 32 * kWorkers) {
          const int xr = k >> 4, hc = k & 15, atom = hc >> 3, cc = hc & 7;
          const uint4 raw = *reinterpret_cast<const uint4*>(st + Cf::kWBytes + xr * 256 + hc * 16);
          uint4 o;
          o.x = bf16x2_to_f16x2(raw.x);
          o.y = bf16x2_to_f16x2(raw.y);
          o.z = bf16x2_to_f16x2(raw.z);
          o.w = bf16x2_to_f16x2(raw.w);
          *reinterpret_cast<uint4*>(xb + atom * (N * 128) + xr * 128 + ((cc ^ (xr & 7)) << 4)) = o;
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        dev::fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          dev::mbar_arrive(&sempty[s]);
          dev::mbar_arrive(&abfull[b]);
        }
      }
      if (i >= 1) {
        const int64_t ip = i - 1;
        const int b = (int)(ip & 1);
        if (!dev::mbar_wait(&dfull[b], (uint32_t)((ip >> 1) & 1), kWaitLimitNs)) {
          dev::set_status(p.status, SWS_E_TIMEOUT);
          s_abort = 1;
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < N / 16; ++c0) {
          float v[16];
          tmem_ld16(tmem + lane_off + 256 + b * 2 * N + t * N + c0 * 16, v);
#pragma unroll
          for (int k = 0; k < 16; ++k) acc[c0 * 16 + k] = fmaf(sc_old, v[k], acc[c0 * 16 + k]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(&dempty[b]);
        const UnitPos up = unit_pos(p, u0 + ip);
        if (ip + 1 == n || up.kb + 1 == p.e[up.j].slabs) tc_end_run<N>(acc, p, geo, up, t, row);
      }
      sc_old = sc_new;
    }
    if (ok && n > 0) tc_settle<N>(p, geo, u0, u1 - 1, wt, t, row, &s_last);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  if (tid == 0) {
    __threadfence();
    dev::trace_end(p.trace, p.tag);
  }
}

template <int N>
cudaError_t launch_tc_n(const DecodeParams& p, int64_t grid_cap, cudaStream_t s) {
  constexpr int kSmem = TcCfg<N>::kSmem;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(decode_tc_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (attr != cudaSuccess) return attr;
  const int64_t grid = std::min<int64_t>({p.units, (int64_t)device_sm_count(), (int64_t)kMaxGrid, grid_cap});
  decode_tc_kernel<N><<<(unsigned)grid, kTcThreads, kSmem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

namespace dec {
cudaError_t launch_decode_tc(const DecodeParams& p, int64_t grid_cap, cudaStream_t s) {
  const int npad = ((p.m + 15) / 16) * 16;
  switch (npad) {
    case 16: return launch_tc_n<16>(p, grid_cap, s);
    case 32: return launch_tc_n<32>(p, grid_cap, s);
    case 48: return launch_tc_n<48>(p, grid_cap, s);
    default: return launch_tc_n<64>(p, grid_cap, s);
  }
}
int64_t tc_slot_bytes(int64_t m) { return (int64_t)kTcRows * (((m + 15) / 16) * 16) * 4; }
}  // namespace dec

}  // namespace sws
