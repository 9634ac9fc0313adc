// SiLU(gate) * up between the two linears of a shared expert (the second
// workload shape: gate_up -> SiLU * up -> down, bf16 tensors in between).
//
//   act[m, j] = bf16_rne( g / (1 + e^-g) * u ),  g = gu[m, j], u = gu[m, F + j]
//
// computed in fp32. HBM-bound: 6 bytes in and 2 out per output element; each
// thread handles 8 consecutive columns with 16-byte loads and stores, over a
// grid-stride loop sized to the SM count.
//
// Also here: the bf16 -> f16 rounding of activations that meet f16 weights at
// prefill sizes (the tensor cores take both operands of one MMA in the same
// 16-bit format), 2 bytes in and 2 out per element.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "sws_internal.h"

namespace sws {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t silu_mul2(uint32_t g, uint32_t u) {
  const float g0 = bf16_lo(g), g1 = bf16_hi(g), u0 = bf16_lo(u), u1 = bf16_hi(u);
  const float a0 = g0 / (1.0f + expf(-g0)) * u0;
  const float a1 = g1 / (1.0f + expf(-g1)) * u1;
  const __nv_bfloat162 r = __floats2bfloat162_rn(a0, a1);
  return *reinterpret_cast<const uint32_t*>(&r);
}

__global__ void __launch_bounds__(256) silu_mul_kernel(const uint16_t* __restrict__ gu, int64_t m, int64_t f,
                                                        uint16_t* __restrict__ act) {
  const int64_t per_row = f / 8;  // 8-column groups per row
  const int64_t n = m * per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / per_row, c = (i - r * per_row) * 8;
    const uint4 g = __ldg(reinterpret_cast<const uint4*>(gu + r * 2 * f + c));
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(gu + r * 2 * f + f + c));
    uint4 o;
    o.x = silu_mul2(g.x, u.x);
    o.y = silu_mul2(g.y, u.y);
    o.z = silu_mul2(g.z, u.z);
    o.w = silu_mul2(g.w, u.w);
    *reinterpret_cast<uint4*>(act + r * f + c) = o;
  }
}

// Each bf16 value rounded to nearest even f16 (overflow to +-inf).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  const __half2 h = __floats2half2_rn(bf16_lo(v), bf16_hi(v));
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(256) to_f16_kernel(const uint16_t* __restrict__ x, int64_t n8,
                                                      uint16_t* __restrict__ out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x) + i);
    uint4 o;
    o.x = bf16x2_to_f16x2(v.x);
    o.y = bf16x2_to_f16x2(v.y);
    o.z = bf16x2_to_f16x2(v.z);
    o.w = bf16x2_to_f16x2(v.w);
    reinterpret_cast<uint4*>(out)[i] = o;
  }
}

}  // namespace

int launch_to_f16(const uint16_t* x, int64_t n, uint16_t* out, cudaStream_t s) {
  if (n < 0 || n % 8 != 0) return fail(SWS_E_UNSUPPORTED, "to_f16: n=%lld is not a multiple of 8", (long long)n);
  if (n == 0) return SWS_OK;
  if (!aligned16(x) || !aligned16(out)) return fail(SWS_E_ALIGN, "to_f16: pointer not 16-byte aligned");
  const int64_t blocks = std::min<int64_t>(cdiv(n / 8, 256), (int64_t)device_sm_count() * 8);
  cudaError_t e = launch_high(to_f16_kernel, dim3((unsigned)blocks), dim3(256), 0, s, x, n / 8, out);
  return e == cudaSuccess ? SWS_OK : cuda_fail(e, "to_f16 kernel launch");
}

int launch_silu_mul(const uint16_t* gu, int64_t m, int64_t f, uint16_t* act, cudaStream_t s) {
  if (m < 0 || f < 0) return fail(SWS_E_INVALID, "silu_mul: m=%lld f=%lld", (long long)m, (long long)f);
  if (f % 8 != 0) return fail(SWS_E_UNSUPPORTED, "silu_mul: f=%lld is not a multiple of 8", (long long)f);
  if (m == 0 || f == 0) return SWS_OK;
  if (!gu || !act) return fail(SWS_E_INVALID, "silu_mul: NULL pointer");
  if (!aligned16(gu) || !aligned16(act)) return fail(SWS_E_ALIGN, "silu_mul: pointer not 16-byte aligned");
  const int64_t groups = m * (f / 8);
  const int64_t blocks = std::min<int64_t>(cdiv(groups, 256), (int64_t)device_sm_count() * 8);
  cudaError_t e = launch_high(silu_mul_kernel, dim3((unsigned)blocks), dim3(256), 0, s, gu, m, f, act);
  return e == cudaSuccess ? SWS_OK : cuda_fail(e, "silu_mul kernel launch");
}

}  // namespace sws
