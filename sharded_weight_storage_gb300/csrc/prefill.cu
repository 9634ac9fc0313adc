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

// One warp per (row, 128-column group); each lane owns 4 consecutive columns.
__global__ void __launch_bounds__(256) quantize_x_kernel(const uint16_t* __restrict__ x, int64_t m, int64_t k,
                                                         int64_t groups, uint8_t* __restrict__ xq,
                                                         float* __restrict__ ex) {
  const int64_t wid = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= m * groups) return;
  const int64_t row = wid / groups, grp = wid - row * groups;
  const int64_t col = grp * 128 + lane * 4;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  const bool valid = col < k;  // k % 16 == 0, so 4 columns are all in or all out
  if (valid) {
    const uint2 raw = *reinterpret_cast<const uint2*>(x + row * k + col);
    v[0] = __uint_as_float(raw.x << 16);
    v[1] = __uint_as_float(raw.x & 0xffff0000u);
    v[2] = __uint_as_float(raw.y << 16);
    v[3] = __uint_as_float(raw.y & 0xffff0000u);
  }
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  int kexp = 0;
  if (amax > 0.f) {
    int p;
    const float f = frexpf(amax, &p);  // amax = f * 2^p, f in [0.5, 1); 448 = 0.875 * 2^9
    kexp = (f <= 0.875f) ? p - 9 : p - 8;
  }
  if (valid) {
    uint16_t lo, hi;
    const float q0 = ldexpf(v[0], -kexp), q1 = ldexpf(v[1], -kexp);
    const float q2 = ldexpf(v[2], -kexp), q3 = ldexpf(v[3], -kexp);
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(q1), "f"(q0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(q3), "f"(q2));
    *reinterpret_cast<uint32_t*>(xq + row * k + col) = (uint32_t)lo | ((uint32_t)hi << 16);
  }
  if (lane == 0) ex[row * groups + grp] = ldexpf(1.0f, kexp);
}

}  // namespace

int launch_quantize_x(const uint16_t* x, int64_t m, int64_t k, uint8_t* xq, float* ex, cudaStream_t s) {
  if (m < 0 || k < 0) return fail(SWS_E_INVALID, "quantize_x: m=%lld k=%lld", (long long)m, (long long)k);
  if (k % 16 != 0) return fail(SWS_E_UNSUPPORTED, "quantize_x: k=%lld is not a multiple of 16", (long long)k);
  const int64_t groups = cdiv(k, 128);
  const int64_t warps = m * groups;
  if (warps == 0) return SWS_OK;
  if (!aligned16(x) || !aligned16(xq) || !aligned16(ex)) return fail(SWS_E_ALIGN, "quantize_x: pointer not 16-byte aligned");
  quantize_x_kernel<<<(unsigned)cdiv(warps, 8), 256, 0, s>>>(x, m, k, groups, xq, ex);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SWS_OK : cuda_fail(e, "quantize_x kernel launch");
}

}  // namespace sws
