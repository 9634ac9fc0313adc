// Prefill path: activation quantiser (and, in prefill_gemm.cu, the tcgen05
// block-scaled FP8 GEMM).
//
// Quantiser: for each row m and 128-column group g,
//   ex[m, g] = 2^k, k the smallest integer with amax <= 448 * 2^k (1 if the
//   group is all zero),  xq[m, i] = e4m3_rne(x[m, i] / ex[m, g]).
// Dividing by a power of two is exact, so the only rounding is the e4m3 one,
// and the result is reproducible bit for bit.
#include <cuda_runtime.h>

#include <algorithm>

#include "ptx.cuh"
#include "sws_internal.h"

namespace sws {
namespace {

// 2^e as a float, exactly for e in [-149, 127]; 0 below (float32 underflow).
__device__ __forceinline__ float exp2_exact(int e) {
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : e >= -149 ? __uint_as_float(1u << (e + 149)) : 0.f;
}

// Eight consecutive threads per (row, 128-column group), 16 columns each
// (two 16-byte loads, one 16-byte store); a grid-stride loop over the groups.
__global__ void __launch_bounds__(256) quantize_x_kernel(const uint16_t* __restrict__ x, int64_t m, int64_t k,
                                                         int64_t groups, uint8_t* __restrict__ xq,
                                                         float* __restrict__ ex) {
  const int g = threadIdx.x & 7;
  const int64_t tasks = m * groups;
  const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 3);
  for (int64_t task = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 3; task < tasks; task += stride) {
    const int64_t row = task / groups, grp = task - row * groups;
    const int64_t col = grp * 128 + g * 16;
    float v[16];
    const bool valid = col < k;  // k % 16 == 0: 16 columns are all in or all out
    if (valid) {
      const uint4* src = reinterpret_cast<const uint4*>(x + row * k + col);
      const uint4 r0 = __ldcs(src), r1 = __ldcs(src + 1);
      const uint32_t u[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[2 * i] = __uint_as_float(u[i] << 16);
        v[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0.f;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    // Lanes 8t..8t+7 hold one task and run the loop together; other tasks of
    // the warp may have left it, so the shuffles name only these eight lanes.
    const uint32_t mask = 0xffu << ((threadIdx.x & 31) & 24);
    amax = fmaxf(amax, __shfl_xor_sync(mask, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(mask, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(mask, amax, 4));
    // k = smallest integer with amax <= 448 * 2^k: for amax = 1.f x 2^E that is
    // E - 8 when 1.f <= 1.75 (448 = 1.75 x 2^8), else E - 7. Subnormal amax: frexp.
    int kexp = 0;
    const uint32_t bits = __float_as_uint(amax);
    if (bits >= 0x00800000u) {
      const int E = (int)(bits >> 23) - 127;
      kexp = (bits & 0x007fffffu) <= 0x00600000u ? E - 8 : E - 7;
    } else if (amax > 0.f) {
      int p;
      const float f = frexpf(amax, &p);  // amax = f * 2^p, f in [0.5, 1); 448 = 0.875 * 2^9
      kexp = (f <= 0.875f) ? p - 9 : p - 8;
    }
    if (valid) {
      uint32_t w[4];
      if (-kexp >= -126 && -kexp <= 127) {  // x * 2^-k with one exact multiply
        const float inv = __uint_as_float((uint32_t)(127 - kexp) << 23);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint16_t lo, hi;
          asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(v[4 * i + 1] * inv), "f"(v[4 * i] * inv));
          asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(v[4 * i + 3] * inv), "f"(v[4 * i + 2] * inv));
          w[i] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
      } else {  // 2^-k is not a normal float: scale in two exact steps
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint16_t lo, hi;
          const float q0 = ldexpf(v[4 * i], -kexp), q1 = ldexpf(v[4 * i + 1], -kexp);
          const float q2 = ldexpf(v[4 * i + 2], -kexp), q3 = ldexpf(v[4 * i + 3], -kexp);
          asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(q1), "f"(q0));
          asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(q3), "f"(q2));
          w[i] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
      }
      *reinterpret_cast<uint4*>(xq + row * k + col) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (g == 0) ex[row * groups + grp] = exp2_exact(kexp);
  }
}

}  // namespace

int launch_quantize_x(const uint16_t* x, int64_t m, int64_t k, uint8_t* xq, float* ex, cudaStream_t s) {
  if (m < 0 || k < 0) return fail(SWS_E_INVALID, "quantize_x: m=%lld k=%lld", (long long)m, (long long)k);
  if (k % 16 != 0) return fail(SWS_E_UNSUPPORTED, "quantize_x: k=%lld is not a multiple of 16", (long long)k);
  const int64_t groups = cdiv(k, 128);
  const int64_t tasks = m * groups;  // one task (8 threads) per (row, group)
  if (tasks == 0) return SWS_OK;
  if (!aligned16(x) || !aligned16(xq) || !aligned16(ex)) return fail(SWS_E_ALIGN, "quantize_x: pointer not 16-byte aligned");
  const int64_t blocks = std::min<int64_t>(cdiv(tasks, 32), (int64_t)device_sm_count() * 8);
  cudaError_t e = launch_high(quantize_x_kernel, dim3((unsigned)blocks), dim3(256), 0, s, x, m, k, groups, xq, ex);
  return e == cudaSuccess ? SWS_OK : cuda_fail(e, "quantize_x kernel launch");
}

}  // namespace sws
