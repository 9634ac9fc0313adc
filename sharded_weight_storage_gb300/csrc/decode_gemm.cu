// Split-K FP8 skinny decode GEMM (m <= 64) on zero-copy weight views.
//
//   Y[m, o] = bf16_rne( sum_kb s[o/128, kb] * sum_{i in kb} x[m, i] * e4m3(q[o, i]) )
//
// The linear the weight-sharding blog keeps unchanged (section "核心抽象":
// the GEMM sees the full W; Y = X W^T with W [out, in]); block scales are
// 128 x 128, float32.
//
// Design (HBM-bound at decode sizes; every weight byte is read exactly once):
//   * Swap-AB warp-level tensor-core MMA (mma.sync m16n8k16, f16 operands,
//     fp32 accumulate): the weight supplies 16-row A tiles, the activations the
//     8-column B tiles, so m <= 64 costs 1..8 n-tiles.
//   * Weights stream straight from HBM into registers with 16-byte
//     non-allocating loads (one slab of 128 K ahead), and are widened with the
//     exact e4m3x2 -> f16x2 conversion. Because a dot product does not care
//     about the order of k, each thread reads contiguous bytes and the
//     activations use the same permutation of k.
//   * Activations are converted bf16 -> f16 once per CTA and staged in shared
//     memory (double-buffered, XOR-swizzled so that fragment loads are free of
//     bank conflicts); one __syncthreads per 128-K slab.
//   * Block scales: a warp's rows lie inside one 128-row scale block, so the
//     scale is one scalar per warp and slab. The accumulator holds
//     sum_b (s_b / s_cur) P_b and is rescaled by s_prev / s_cur when the scale
//     changes, then multiplied by the last scale at the end of a run.
//   * Split-K across CTAs: the (row block, K slab) units are cut into equal
//     contiguous ranges, one per CTA of a grid sized to the SM count. A CTA that
//     covers a whole row block writes Y directly; partial runs write fp32 sums
//     to the workspace and the last CTA to arrive on a row block (atomic
//     counter, no waiting) adds them in K order and writes Y.
//   * Fused variant: the same kernel reads each 16-byte weight piece from the
//     chunk that holds it (byte g of T lives in chunk g / C at g % C), so no
//     slot is written.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "ptx.cuh"
#include "sws_internal.h"

namespace sws {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSlabK = 128;
constexpr int kMaxGrid = 256;  // upper bound used to size the workspace

struct DecodeParams {
  const uint8_t* w;
  const uint8_t* chunks[256];
  int64_t chunk_bytes;
  int64_t t_offset;
  const float* scales;
  int64_t scale_cols;
  const uint16_t* x;
  uint16_t* y;
  int64_t rows, cols;
  int32_t m;
  int32_t slabs;       // ceil(cols / 128)
  int64_t units;       // row blocks * slabs
  int32_t* counters;
  float* partials;
  uint64_t* trace;
  uint64_t tag;
};

__device__ __forceinline__ uint4 ldg_stream(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)two_bytes));
  return r;
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  const float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xffff0000u);
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Which CTA's unit range [u*G/U ...) contains unit u.
__device__ __forceinline__ int64_t cta_of(int64_t u, int64_t G, int64_t U) { return ((u + 1) * G - 1) / U; }

template <int NT, int R, bool FUSED>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int kRowsWarp = 16 * R;
  constexpr int kRowsCta = kWarps * kRowsWarp;
  constexpr int kXRows = NT * 8;
  constexpr int kXUnits = kXRows * 16;  // 16-byte units per X slab
  constexpr int kXPer = (kXUnits + kThreads - 1) / kThreads;
  constexpr int kSlot = kWarps * R * NT * 32 * 4;  // floats per partial slot

  __shared__ __align__(16) uint4 xs[2][kXUnits];
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tig = lane & 3;
  const int64_t U = p.units, G = gridDim.x, c = blockIdx.x;
  const int64_t u0 = c * U / G, u1 = (c + 1) * U / G;
  if (tid == 0) dev::trace_start(p.trace);
  const int64_t C = p.chunk_bytes;

  // ---- weight loads ------------------------------------------------------
  // Thread (g, tig) of warp w, row tile rt, half h (rows g and g+8) reads the
  // 16 bytes at k = kb*128 + l*64 + 16*tig for l = 0, 1.
  auto load_w = [&](int64_t u, uint4 (&dst)[R][2][2]) {
    const int64_t rb = u / p.slabs, kb = u - rb * p.slabs;
#pragma unroll
    for (int rt = 0; rt < R; ++rt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t o = rb * kRowsCta + warp * kRowsWarp + rt * 16 + g + 8 * h;
#pragma unroll
        for (int l = 0; l < 2; ++l) {
          const int64_t k = kb * kSlabK + l * 64 + 16 * tig;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (o < p.rows && k < p.cols) {
            if (FUSED) {
              const int64_t gb = p.t_offset + o * p.cols + k;
              const int64_t ci = gb / C;
              v = ldg_stream(p.chunks[ci] + (gb - ci * C));
            } else {
              v = ldg_stream(p.w + o * p.cols + k);
            }
          }
          dst[rt][h][l] = v;
        }
      }
  };
  // ---- activation staging (bf16 -> f16, swizzled) --------------------------
  auto load_x = [&](int64_t u, uint4 (&dst)[kXPer]) {
    const int64_t kb = u % p.slabs;
#pragma unroll
    for (int i = 0; i < kXPer; ++i) {
      const int v = tid + i * kThreads;
      const int mrow = v >> 4, q = v & 15;
      const int64_t k = kb * kSlabK + q * 8;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (v < kXUnits && mrow < p.m && k < p.cols)
        val = __ldg(reinterpret_cast<const uint4*>(p.x + (int64_t)mrow * p.cols + k));
      dst[i] = val;
    }
  };
  auto store_x = [&](int buf, const uint4 (&src)[kXPer]) {
#pragma unroll
    for (int i = 0; i < kXPer; ++i) {
      const int v = tid + i * kThreads;
      if (v < kXUnits) {
        const int mrow = v >> 4, q = v & 15;
        uint4 h;
        h.x = bf16x2_to_f16x2(src[i].x);
        h.y = bf16x2_to_f16x2(src[i].y);
        h.z = bf16x2_to_f16x2(src[i].z);
        h.w = bf16x2_to_f16x2(src[i].w);
        xs[buf][mrow * 16 + (q ^ (mrow & 1))] = h;
      }
    }
  };

  float acc[R][NT][4];
#pragma unroll
  for (int rt = 0; rt < R; ++rt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[rt][nt][e] = 0.f;
  float cs = 0.f;  // scale the accumulator currently refers to

  uint4 wcur[R][2][2], wnxt[R][2][2];
  uint4 xst[kXPer];
  if (u0 < u1) {
    load_w(u0, wcur);
    load_x(u0, xst);
    store_x(0, xst);
  }

  for (int64_t u = u0; u < u1; ++u) {
    const int buf = (int)((u - u0) & 1);
    __syncthreads();  // xs[buf] is complete; xs[buf ^ 1] is no longer read
    const bool more = u + 1 < u1;
    if (more) {
      load_w(u + 1, wnxt);
      load_x(u + 1, xst);
    }
    const int64_t rb = u / p.slabs, kb = u - rb * p.slabs;
    const int64_t row0 = rb * kRowsCta + warp * kRowsWarp;
    const bool run_start = (u == u0) || kb == 0;
    const bool run_end = (u + 1 == u1) || kb + 1 == p.slabs;
    if (run_start) cs = 0.f;
    // ---- this warp's scale for the slab, and the accumulator rescale ----
    float s = 0.f;
    if (row0 < p.rows) s = __ldg(p.scales + (row0 >> 7) * p.scale_cols + kb);
    if (s != 0.f) {
      if (cs != 0.f && s != cs) {
        const float ratio = cs / s;
#pragma unroll
        for (int rt = 0; rt < R; ++rt)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[rt][nt][e] *= ratio;
      }
      cs = s;
      // ---- MMAs over the slab: two 64-K halves of four k16 steps ----
      const uint4* xb = xs[buf];
#pragma unroll
      for (int l = 0; l < 2; ++l) {
        uint32_t a[R][2][8];  // [rt][row g / g+8][f16x2 words for k positions]
#pragma unroll
        for (int rt = 0; rt < R; ++rt)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 wv = wcur[rt][h][l];
            a[rt][h][0] = e4m3x2_to_f16x2(wv.x);
            a[rt][h][1] = e4m3x2_to_f16x2(wv.x >> 16);
            a[rt][h][2] = e4m3x2_to_f16x2(wv.y);
            a[rt][h][3] = e4m3x2_to_f16x2(wv.y >> 16);
            a[rt][h][4] = e4m3x2_to_f16x2(wv.z);
            a[rt][h][5] = e4m3x2_to_f16x2(wv.z >> 16);
            a[rt][h][6] = e4m3x2_to_f16x2(wv.w);
            a[rt][h][7] = e4m3x2_to_f16x2(wv.w >> 16);
          }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int mrow = nt * 8 + g;
          const int u0x = 8 * l + 2 * tig;
          const uint4 b0 = xb[mrow * 16 + (u0x ^ (mrow & 1))];
          const uint4 b1 = xb[mrow * 16 + ((u0x + 1) ^ (mrow & 1))];
          const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int rt = 0; rt < R; ++rt)
              mma16816(acc[rt][nt], a[rt][0][2 * kk], a[rt][1][2 * kk], a[rt][0][2 * kk + 1], a[rt][1][2 * kk + 1],
                       bw[2 * kk], bw[2 * kk + 1]);
        }
      }
    }
    if (more) store_x(buf ^ 1, xst);

    if (run_end) {
      // ---- finish the run: apply the last scale, then write or reduce ----
#pragma unroll
      for (int rt = 0; rt < R; ++rt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[rt][nt][e] *= cs;
      const int64_t ks = rb * p.slabs;
      const int64_t cf = cta_of(ks, G, U), cl = cta_of(ks + p.slabs - 1, G, U);
      bool write_y = true;
      if (cf != cl) {
        // partial run: publish, count arrivals; the last CTA sums in K order
        const int64_t my_first_rb = u0 / p.slabs;
        float* slot = p.partials + (2 * c + (rb == my_first_rb ? 0 : 1)) * (int64_t)kSlot;
#pragma unroll
        for (int rt = 0; rt < R; ++rt)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            reinterpret_cast<float4*>(slot)[((warp * R + rt) * NT + nt) * 32 + lane] =
                make_float4(acc[rt][nt][0], acc[rt][nt][1], acc[rt][nt][2], acc[rt][nt][3]);
        __threadfence();
        __syncthreads();
        if (tid == 0) {
          const int old = atomicAdd(p.counters + rb, 1);
          s_last = (old == (int)(cl - cf));
        }
        __syncthreads();
        write_y = s_last != 0;
        if (write_y) {
          __threadfence();
#pragma unroll
          for (int rt = 0; rt < R; ++rt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[rt][nt][e] = 0.f;
          for (int64_t cc = cf; cc <= cl; ++cc) {
            const int64_t first_rb = (cc * U / G) / p.slabs;
            const float* sl = p.partials + (2 * cc + (rb == first_rb ? 0 : 1)) * (int64_t)kSlot;
#pragma unroll
            for (int rt = 0; rt < R; ++rt)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(sl) + ((warp * R + rt) * NT + nt) * 32 + lane);
                acc[rt][nt][0] += v.x;
                acc[rt][nt][1] += v.y;
                acc[rt][nt][2] += v.z;
                acc[rt][nt][3] += v.w;
              }
          }
          if (tid == 0) p.counters[rb] = 0;
        }
      }
      if (write_y) {
#pragma unroll
        for (int rt = 0; rt < R; ++rt)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int64_t o = row0 + rt * 16 + g + 8 * (e >> 1);
              const int mm = nt * 8 + 2 * tig + (e & 1);
              if (o < p.rows && mm < p.m) {
                const __nv_bfloat16 b = __float2bfloat16_rn(acc[rt][nt][e]);
                p.y[(int64_t)mm * p.rows + o] = *reinterpret_cast<const uint16_t*>(&b);
              }
            }
      }
#pragma unroll
      for (int rt = 0; rt < R; ++rt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[rt][nt][e] = 0.f;
    }
    if (more) {
#pragma unroll
      for (int rt = 0; rt < R; ++rt)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int l = 0; l < 2; ++l) wcur[rt][h][l] = wnxt[rt][h][l];
    }
  }
  if (tid == 0) {
    __threadfence();
    dev::trace_end(p.trace, p.tag);
  }
}

template <int NT>
constexpr int rows_per_warp_tiles() { return NT <= 2 ? 4 : 2; }

template <int NT, bool FUSED>
cudaError_t launch_nt(const DecodeParams& p0, int64_t row_blocks, cudaStream_t s) {
  constexpr int R = rows_per_warp_tiles<NT>();
  DecodeParams p = p0;
  p.units = row_blocks * p.slabs;
  const int64_t grid = std::min<int64_t>({p.units, (int64_t)device_sm_count(), (int64_t)kMaxGrid});
  decode_kernel<NT, R, FUSED><<<(unsigned)grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

int nt_for(int64_t m) { return m <= 8 ? 1 : m <= 16 ? 2 : m <= 32 ? 4 : 8; }
int rows_per_cta(int nt) { return kWarps * 16 * (nt <= 2 ? 4 : 2); }

}  // namespace

int decode_workspace_bytes(int64_t m, int64_t rows, int64_t cols, int64_t* bytes) {
  (void)cols;
  if (m < 0 || m > 64) return fail(SWS_E_INVALID, "decode: m=%lld outside [0, 64]", (long long)m);
  const int nt = nt_for(std::max<int64_t>(m, 1));
  const int r = nt <= 2 ? 4 : 2;
  const int64_t slot_floats = (int64_t)kWarps * r * nt * 32 * 4;
  const int64_t row_blocks = cdiv(rows, rows_per_cta(nt));
  if (row_blocks > kMaxCounters) return fail(SWS_E_UNSUPPORTED, "decode: %lld rows is too many", (long long)rows);
  *bytes = kCtlBytes + kMaxCounters * 4 + 2 * (int64_t)kMaxGrid * slot_floats * 4;
  return SWS_OK;
}

int launch_decode(const DecodeLaunch& a, cudaStream_t s) {
  if (a.m <= 0 || a.rows == 0) return SWS_OK;
  if (a.cols % 16 != 0) return fail(SWS_E_UNSUPPORTED, "decode: cols=%lld is not a multiple of 16", (long long)a.cols);
  int64_t need = 0;
  int rc = decode_workspace_bytes(a.m, a.rows, a.cols, &need);
  if (rc != SWS_OK) return rc;
  if (a.workspace_bytes < need)
    return fail(SWS_E_WORKSPACE, "decode: workspace %lld < %lld bytes", (long long)a.workspace_bytes, (long long)need);
  if (a.cols == 0) {
    cudaError_t e = cudaMemsetAsync(a.y, 0, (size_t)(a.m * a.rows * 2), s);
    return e == cudaSuccess ? SWS_OK : cuda_fail(e, "decode: cudaMemsetAsync");
  }
  DecodeParams p;
  p.w = a.w;
  const bool fused = a.w == nullptr;
  for (int i = 0; i < 256; ++i) p.chunks[i] = i < a.n_chunks ? a.chunks[i] : nullptr;
  p.chunk_bytes = a.chunk_bytes > 0 ? a.chunk_bytes : 1;
  p.t_offset = a.t_offset;
  p.scales = a.scales;
  p.scale_cols = cdiv(a.cols, 128);
  p.x = a.x;
  p.y = a.y;
  p.rows = a.rows;
  p.cols = a.cols;
  p.m = (int32_t)a.m;
  p.slabs = (int32_t)cdiv(a.cols, kSlabK);
  p.counters = reinterpret_cast<int32_t*>(a.workspace + kCtlBytes);
  p.partials = reinterpret_cast<float*>(a.workspace + kCtlBytes + kMaxCounters * 4);
  p.trace = a.trace;
  p.tag = a.tag;
  const int nt = nt_for(a.m);
  const int64_t row_blocks = cdiv(a.rows, rows_per_cta(nt));
  cudaError_t e;
  switch (nt) {
    case 1: e = fused ? launch_nt<1, true>(p, row_blocks, s) : launch_nt<1, false>(p, row_blocks, s); break;
    case 2: e = fused ? launch_nt<2, true>(p, row_blocks, s) : launch_nt<2, false>(p, row_blocks, s); break;
    case 4: e = fused ? launch_nt<4, true>(p, row_blocks, s) : launch_nt<4, false>(p, row_blocks, s); break;
    default: e = fused ? launch_nt<8, true>(p, row_blocks, s) : launch_nt<8, false>(p, row_blocks, s); break;
  }
  return e == cudaSuccess ? SWS_OK : cuda_fail(e, "decode kernel launch");
}

}  // namespace sws

// ---------------------------------------------------------------------------
// Decode linear that allocates nothing.
//
// Some callers cannot hand this library a workspace or let it allocate one: an
// inference engine that sizes its KV-cache pool from the free memory left after
// the weights are placed has no headroom for allocations made later, and a
// cudaMalloc issued in the middle of a decode step can synchronise the whole
// device. This variant of the split-K decode kernel keeps its scratch (the
// split-K partial sums and the per-row-block arrival counters) in a fixed
// array that lives in the library's device image, so a call needs only the
// caller's inputs and outputs.
//
// The array is shared by every call on a device and keeps the last call's
// contents; the arrival counters are cleared on the stream before each launch.
// Two calls whose work overlaps on the GPU race on the array.
// ---------------------------------------------------------------------------
namespace sws {
namespace {

constexpr int64_t kNoAllocPartialBytes = int64_t(8) << 20;  // 8 MiB of fp32 partial sums
constexpr int64_t kNoAllocCounters = 4096;                    // row blocks, one int32 each
constexpr int64_t kNoAllocScratchBytes = kNoAllocPartialBytes + kNoAllocCounters * 4;
constexpr int kMaxDevices = 64;

// Partial sums first (256-byte aligned), counters after them.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device. The first call on
// a device resolves it with cudaGetSymbolAddress (with that device current);
// later calls reuse the cached address.
int noalloc_scratch(uint8_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "linear_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(SWS_E_UNSUPPORTED, "linear_noalloc: device %d", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "linear_noalloc: cudaGetSymbolAddress(scratch)");
    g_noalloc_addr[dev] = p;
  }
  *out = static_cast<uint8_t*>(g_noalloc_addr[dev]);
  return SWS_OK;
}

template <int NT>
cudaError_t launch_noalloc_nt(DecodeParams p, int64_t row_blocks, cudaStream_t s) {
  constexpr int R = rows_per_warp_tiles<NT>();
  constexpr int64_t kSlotBytes = int64_t(kWarps) * R * NT * 32 * 4 * 4;
  constexpr int64_t kGridCap = kNoAllocPartialBytes / (2 * kSlotBytes);  // two partial slots per CTA
  p.units = row_blocks * p.slabs;
  const int64_t grid = std::min<int64_t>({p.units, (int64_t)device_sm_count(), (int64_t)kMaxGrid, kGridCap});
  decode_kernel<NT, R, false><<<(unsigned)grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace
}  // namespace sws

extern "C" int sws_linear_noalloc(const void* w, const float* scales, int64_t rows, int64_t cols, const void* x,
                                  int64_t m, void* y, sws_stream_t stream) {
  using namespace sws;
  if (m < 0 || m > 64) return fail(SWS_E_INVALID, "linear_noalloc: m=%lld outside [0, 64]", (long long)m);
  if (rows < 0 || cols < 0) return fail(SWS_E_INVALID, "linear_noalloc: shape [%lld, %lld]", (long long)rows,
                                        (long long)cols);
  if (cols % 16 != 0)
    return fail(SWS_E_UNSUPPORTED, "linear_noalloc: cols=%lld is not a multiple of 16", (long long)cols);
  if (m == 0 || rows == 0) return SWS_OK;
  if (!w || !scales || !x || !y) return fail(SWS_E_INVALID, "linear_noalloc: NULL pointer");
  if (!aligned16(w) || !aligned16(scales) || !aligned16(x) || !aligned16(y))
    return fail(SWS_E_ALIGN, "linear_noalloc: a pointer is not 16-byte aligned");
  const int nt = nt_for(m);
  const int64_t row_blocks = cdiv(rows, rows_per_cta(nt));
  if (row_blocks > kNoAllocCounters)
    return fail(SWS_E_INVALID, "linear_noalloc: rows=%lld exceeds the limit of %lld rows at m=%lld",
                (long long)rows, (long long)(kNoAllocCounters * rows_per_cta(nt)), (long long)m);
  int rc = check_device();
  if (rc != SWS_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  if (cols == 0) {
    cudaError_t e = cudaMemsetAsync(y, 0, (size_t)(m * rows * 2), s);
    return e == cudaSuccess ? SWS_OK : cuda_fail(e, "linear_noalloc: cudaMemsetAsync(y)");
  }
  uint8_t* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc != SWS_OK) return rc;
  int32_t* counters = reinterpret_cast<int32_t*>(scratch + kNoAllocPartialBytes);
  cudaError_t e = cudaMemsetAsync(counters, 0, (size_t)(row_blocks * 4), s);
  if (e != cudaSuccess) return cuda_fail(e, "linear_noalloc: cudaMemsetAsync(counters)");
  DecodeParams p;
  p.w = static_cast<const uint8_t*>(w);
  for (int i = 0; i < 256; ++i) p.chunks[i] = nullptr;
  p.chunk_bytes = 1;
  p.t_offset = 0;
  p.scales = scales;
  p.scale_cols = cdiv(cols, 128);
  p.x = static_cast<const uint16_t*>(x);
  p.y = static_cast<uint16_t*>(y);
  p.rows = rows;
  p.cols = cols;
  p.m = (int32_t)m;
  p.slabs = (int32_t)cdiv(cols, kSlabK);
  p.counters = counters;
  p.partials = reinterpret_cast<float*>(scratch);
  p.trace = nullptr;
  p.tag = 0;
  switch (nt) {
    case 1: e = launch_noalloc_nt<1>(p, row_blocks, s); break;
    case 2: e = launch_noalloc_nt<2>(p, row_blocks, s); break;
    case 4: e = launch_noalloc_nt<4>(p, row_blocks, s); break;
    default: e = launch_noalloc_nt<8>(p, row_blocks, s); break;
  }
  return e == cudaSuccess ? SWS_OK : cuda_fail(e, "linear_noalloc: kernel launch");
}
