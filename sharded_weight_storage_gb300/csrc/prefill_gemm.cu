// Block-scaled FP8 prefill GEMM (m > 64) on tcgen05 tensor cores and TMEM.
//
//   Y[m, n] = bf16_rne( sum_kb ex[m, kb] * s_w[n / 128, kb] * sum_{k in kb} xq[m, k] * wq[n, k] )
//
// xq / ex come from the activation quantiser (e4m3 codes with a power-of-two
// scale per row and 128-column group); wq / s_w are the weight view and its
// 128 x 128 float32 block scales. This is the linear of the weight-sharding
// blog (section "核心抽象": Y = X W^T on the full W) at prefill sizes, where
// the GEMM is a dense contraction and the gather is easy to hide (section
// "提前一层：lookahead 与 ping-pong slot").
//
// Design (one persistent CTA per SM, 10 warps, warp-specialised):
//   * warp 0, one thread: TMA producer. Per 128-K slab it loads the 128 x 128
//     activation tile and the 256 x 128 weight tile (e4m3, 128-byte swizzle,
//     zero fill past the edges) into one of 4 shared-memory stages.
//   * warp 1: allocates 512 TMEM columns; one thread issues the MMAs:
//     4 x tcgen05.mma kind::f8f6f4 (128 x 256 x 32) per slab into one of two
//     TMEM slab buffers (128 lanes x 256 fp32 columns each), then commits to
//     the stage's "empty" barrier and the buffer's "full" barrier.
//   * warps 2-9: promotion. The weight scales are not powers of two, so they
//     cannot feed the MMA's own block scaling; each slab result is read from
//     TMEM (tcgen05.ld) and added into fp32 registers with the factor
//     ex[m, kb] * s_w[n/128, kb] (each thread owns one row m and 128 columns).
//     After the last slab of a tile the row is rounded to bf16 and stored.
//   * Every mbarrier wait is bounded; a wait that runs out records
//     SWS_E_TIMEOUT and the CTA finishes with TMEM released.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "ptx.cuh"
#include "sws_internal.h"

namespace sws {
namespace {

constexpr int kBM = 128;          // activation rows per tile (MMA M)
constexpr int kBN = 256;          // weight rows per tile (MMA N)
constexpr int kBK = 128;          // K per slab = one scale block
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK;  // 16 KB
constexpr int kBBytes = kBN * kBK;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kEpiWarps = 8;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr int kTmemCols = 512;  // two slab buffers of kBN columns
constexpr int kSmemBytes = kStages * kStageBytes + 1024;

struct PrefillParams {
  CUtensorMap tmap_x;  // xq [M, K] u8, box {128, 128}
  CUtensorMap tmap_w;  // wq [N, K] u8, box {128, 256}
  const float* ex;     // [M, K/128]
  const float* sw;     // [ceil(N/128), K/128]
  uint16_t* y;         // bf16 [M, N]
  int64_t M, N, K;
  int32_t kslabs, m_tiles, n_tiles;
  int32_t* status;
  uint64_t* trace;
  uint64_t tag;
};

// ---- tcgen05 helpers ----------------------------------------------------------

// Shared-memory matrix descriptor: K-major operand tile stored as 128-byte rows
// with the 128-byte swizzle, 8-row groups 1024 bytes apart (SM100 layout type
// 2 = SWIZZLE_128B, descriptor version 1).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);      // start address
  d |= (uint64_t)1 << 16;                      // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;            // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                      // descriptor version
  d |= (uint64_t)2 << 61;                      // SWIZZLE_128B
  return d;
}

// Instruction descriptor for kind::f8f6f4: A and B e4m3, D f32, both K-major.
__host__ __device__ constexpr uint32_t idesc_f8(int m, int n) {
  return (1u << 4)                     // D format: f32
         | (0u << 7) | (0u << 10)      // A, B format: e4m3
         | ((uint32_t)(n >> 3) << 17)  // N / 8
         | ((uint32_t)(m >> 4) << 24); // M / 16
}

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// Arrives once on `bar` when all previously issued MMAs of this thread finish.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   dev::smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 16 consecutive fp32 columns: thread (lane i) gets row i's values.
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

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(dev::smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(dev::smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void set_abort(const PrefillParams& p, volatile int* s_abort) {
  dev::set_status(p.status, SWS_E_TIMEOUT);
  *s_abort = 1;
}

__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], mdone;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  // 128-byte swizzled TMA tiles need a 1024-byte aligned destination.
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles;
  const int G = p.kslabs;

  if (threadIdx.x == 0) {
    dev::trace_start(p.trace);
    for (int s = 0; s < kStages; ++s) {
      dev::mbar_init(&full[s], 1);
      dev::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      dev::mbar_init(&tfull[b], 1);
      dev::mbar_init(&tempty[b], kEpiWarps);
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

  if (warp == 0) {
    // ---- TMA producer ----------------------------------------------------
    if (lane == 0) {
      int64_t it = 0;
      for (int64_t tile = blockIdx.x; tile < tiles && !s_abort; tile += gridDim.x) {
        const int32_t mt = (int32_t)(tile % p.m_tiles), nt = (int32_t)(tile / p.m_tiles);
        for (int kb = 0; kb < G; ++kb, ++it) {
          const int s = (int)(it % kStages);
          if (!dev::mbar_wait(&empty[s], (uint32_t)(((it / kStages) & 1) ^ 1), kWaitLimitNs)) {
            set_abort(p, &s_abort);
            break;
          }
          uint8_t* st = smem + s * kStageBytes;
          dev::mbar_arrive_expect_tx(&full[s], kStageBytes);
          tma_load_2d(st, &p.tmap_x, kb * kBK, mt * kBM, &full[s]);
          tma_load_2d(st + kABytes, &p.tmap_w, kb * kBK, nt * kBN, &full[s]);
        }
      }
      // Before the CTA may exit, every issued stage must have landed.
      for (int64_t k = it - kStages; k < it; ++k)
        if (k >= 0) dev::mbar_wait(&full[(int)(k % kStages)], (uint32_t)((k / kStages) & 1), kWaitLimitNs / 4);
    }
  } else if (warp == 1) {
    // ---- MMA issuer ------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f8(kBM, kBN);
      int64_t it = 0;
      bool issued = false;
      for (int64_t tile = blockIdx.x; tile < tiles && !s_abort; tile += gridDim.x) {
        for (int kb = 0; kb < G && !s_abort; ++kb, ++it) {
          const int s = (int)(it % kStages), buf = (int)(it & 1);
          if (!dev::mbar_wait(&tempty[buf], (uint32_t)(((it >> 1) & 1) ^ 1), kWaitLimitNs)) {
            set_abort(p, &s_abort);
            break;
          }
          tc_fence_after();
          if (!dev::mbar_wait(&full[s], (uint32_t)((it / kStages) & 1), kWaitLimitNs)) {
            set_abort(p, &s_abort);
            break;
          }
          tc_fence_after();
          const uint32_t a = dev::smem_addr(smem + s * kStageBytes), b = a + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk)
            mma_f8(tmem + buf * kBN, smem_desc_sw128(a + kk * 32), smem_desc_sw128(b + kk * 32), idesc, kk > 0);
          mma_commit(&empty[s]);
          mma_commit(&tfull[buf]);
          issued = true;
        }
      }
      if (issued) {  // all MMAs of this CTA complete before TMEM is released
        mma_commit(&mdone);
        dev::mbar_wait(&mdone, 0, kWaitLimitNs);
      }
    }
  } else {
    // ---- promotion and output -------------------------------------------------
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;   // which 128 of the tile's 256 columns
    const int row = q * 32 + lane;   // tile row = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + h * 128;
    const int64_t sw_rows = (p.N + 127) / 128;
    int64_t it = 0;
    for (int64_t tile = blockIdx.x; tile < tiles && !s_abort; tile += gridDim.x) {
      const int32_t mt = (int32_t)(tile % p.m_tiles), nt = (int32_t)(tile / p.m_tiles);
      const int64_t m = (int64_t)mt * kBM + row;
      const int64_t n0 = (int64_t)nt * kBN + h * 128, nb = n0 / 128;
      const float* exr = p.ex + (m < p.M ? m : 0) * G;
      const float* swr = p.sw + (nb < sw_rows ? nb : 0) * G;
      const bool live = m < p.M && nb < sw_rows;
      // Raw scale loads, multiplied only when used: a product taken at load
      // time would make the thread wait for both loads right away.
      auto load_ex = [&](int kb) -> float { return (live && kb < G) ? __ldg(exr + kb) : 0.f; };
      auto load_sw = [&](int kb) -> float { return (live && kb < G) ? __ldg(swr + kb) : 0.f; };
      float acc[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0.f;
      // Scale factors are fetched four slabs ahead (rings fe[d], fw[d] hold slab kb0 + d).
      float fe[4], fw[4];
#pragma unroll
      for (int d = 0; d < 4; ++d) {
        fe[d] = load_ex(d);
        fw[d] = load_sw(d);
      }
      bool ok = true;
      for (int kb0 = 0; kb0 < G && ok; kb0 += 4) {
#pragma unroll
        for (int d = 0; d < 4; ++d) {
          const int kb = kb0 + d;
          if (kb < G && ok) {
            const int buf = (int)(it & 1);
            ok = dev::mbar_wait(&tfull[buf], (uint32_t)((it >> 1) & 1), kWaitLimitNs);
            if (!ok) {
              set_abort(p, &s_abort);
            } else {
              tc_fence_after();
              const float fk = fe[d] * fw[d];
              fe[d] = load_ex(kb + 4);
              fw[d] = load_sw(kb + 4);
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                float v[16];
                tmem_ld16(lane_base + buf * kBN + c * 16, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[c * 16 + i] = fmaf(fk, v[i], acc[c * 16 + i]);
              }
              tc_fence_before();
              __syncwarp();
              if (lane == 0) dev::mbar_arrive(&tempty[buf]);
              ++it;
            }
          }
        }
      }
      if (!ok) break;
      // ---- the tile row: bf16, 128 columns -------------------------------------
      if (m < p.M) {
        uint16_t* yrow = p.y + m * p.N + n0;
        const int64_t ncols = p.N - n0 < 128 ? p.N - n0 : 128;
        if (ncols == 128 && (p.N & 7) == 0) {
#pragma unroll
          for (int i = 0; i < 128; i += 8) {
            uint4 o;
            uint32_t* w = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[i + 2 * t], acc[i + 2 * t + 1]);
              w[t] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            *reinterpret_cast<uint4*>(yrow + i) = o;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i < ncols) {
              const __nv_bfloat16 b = __float2bfloat16_rn(acc[i]);
              yrow[i] = *reinterpret_cast<const uint16_t*>(&b);
            }
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  if (threadIdx.x == 0) {
    __threadfence();
    dev::trace_end(p.trace, p.tag);
  }
}

}  // namespace

int launch_prefill(const PrefillLaunch& a, cudaStream_t s) {
  if (a.m <= 0 || a.rows <= 0) return SWS_OK;
  if (a.cols <= 0 || a.cols % 128 != 0)
    return fail(SWS_E_UNSUPPORTED, "prefill: cols=%lld is not a positive multiple of 128", (long long)a.cols);
  if (!aligned16(a.w) || !aligned16(a.xq) || !aligned16(a.y) || !aligned16(a.ex) || !aligned16(a.scales))
    return fail(SWS_E_ALIGN, "prefill: pointer not 16-byte aligned");
  PrefillParams p;
  int rc = encode_u8_tile_map(&p.tmap_x, a.xq, a.m, a.cols, kBM);
  if (rc != SWS_OK) return rc;
  rc = encode_u8_tile_map(&p.tmap_w, a.w, a.rows, a.cols, kBN);
  if (rc != SWS_OK) return rc;
  p.ex = a.ex;
  p.sw = a.scales;
  p.y = a.y;
  p.M = a.m;
  p.N = a.rows;
  p.K = a.cols;
  p.kslabs = (int32_t)(a.cols / kBK);
  p.m_tiles = (int32_t)cdiv(a.m, kBM);
  p.n_tiles = (int32_t)cdiv(a.rows, kBN);
  p.status = a.status;
  p.trace = a.trace;
  p.tag = a.tag;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr != cudaSuccess) return cuda_fail(attr, "prefill: cudaFuncSetAttribute");
  const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles;
  const int64_t grid = std::min<int64_t>(tiles, device_sm_count());
  prefill_kernel<<<(unsigned)grid, kThreads, kSmemBytes, s>>>(p);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SWS_OK : cuda_fail(e, "prefill kernel launch");
}

}  // namespace sws
