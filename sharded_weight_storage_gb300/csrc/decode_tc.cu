// Split-K FP8 decode GEMM (m <= 64) on tcgen05 tensor cores: the same linear
// and the same split-K partition as decode_gemm.cu (see there), for the m where
// the warp-level mma.sync path cannot keep up with HBM. A bf16-weight variant
// and an fp16-weight variant (WT = 1, 2) share everything but the operands: x
// itself (as bf16, or rounded to f16) is the B operand (split_x_16_kernel),
// the MMAs are kind::f16 and no scales apply.
//
//   Y[m, o] = bf16_rne( sum_kb s[o/128, kb] * sum_{i in kb} x[m, i] * e4m3(q[o, i]) )
//
// The weights are never converted: the e4m3 weight slab goes from HBM (TMA,
// 128-byte swizzle) straight into the MMA as its A operand, and the MMA is
// tcgen05.mma kind::f8f6f4. The bf16 activations are made FP8 without loss:
// per (row m, 128-K slab) with a power-of-two scale e = 2^(floor(log2 amax) - 7)
// every x/e lies in [-256, 256) and is the exact sum of two e4m3 numbers,
//   x/e = hi + lo,  hi = e4m3_rne(x/e),  lo = e4m3_rne(x/e - hi),
// for all |x| >= amax / 1024 (smaller elements keep an error below
// e * 2^-10 <= amax * 2^-17). So sum_i x_i w_i = e * (sum_i hi_i w_i + sum_i lo_i w_i):
// the two terms are two more columns of the MMA, added when the result is
// read out.
//
// A launch is three kernels on the stream:
//   1. split_x_kernel: every (entry, K slab) block of activations -> its hi and
//      lo e4m3 operands (already in the 128-byte swizzled order of a
//      1024-byte aligned shared-memory tile) and the scales e, in the workspace.
//      This is m x K work per linear, done once instead of once per row block.
//   2. decode_tc_kernel, launched as a programmatic dependent of (1): its
//      weight loads start while (1) runs; only the activation loads wait for
//      (1) to finish (griddepcontrol.wait). Row blocks that one CTA covers
//      whole are written to Y; a CTA's first and last run may share their row
//      block with neighbouring CTAs (split-K) and store fp32 partial sums.
//   3. settle_kernel, a programmatic dependent of (2): adds the partial sums
//      of every shared row block in K order and writes Y. Settling in its own
//      grid keeps the GEMM free of fences, atomics and cold code at its end.
//      The GEMM releases it once every CTA has read all its weights, and it
//      releases its own dependents at once, so a gather that follows on the
//      stream (the next step's) overlaps the GEMM's tail and the settle.
// decode_tc_kernel (swap-AB: weight rows are the MMA's M = 128 dimension, the
// activations its N = 16..64 dimension, m rounded up to 16):
//   * warp 0, one thread: producer. Per unit (256 weight rows x 128 K) one TMA
//     load of the weight slab, one bulk copy of the slab's split block and two
//     4-byte async copies of the unit's weight scales, into one of 4 stages.
//   * warp 1: allocates TMEM and issues, per unit, 2 tiles x 4 MMAs
//     (128 x 2N x 32: the hi and lo operands side by side as one 2N-row B
//     operand, so each weight byte is read from shared memory once) into one
//     of two to four D buffers.
//   * warps 2-9 (each one quarter of the TMEM lanes of one 128-row tile): read
//     the unit's result from TMEM and add hi + lo, times s[o/128, kb] * e[m], into
//     fp32 registers; at the end of a run, write Y or the partial sums.
// Shared-memory traffic is one TMA write and one MMA read per weight byte.
// Every wait is bounded; a wait that runs out records SWS_E_TIMEOUT and the
// CTA finishes with its copies landed and TMEM released.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <memory>
#include <mutex>
#include <vector>

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

__host__ __device__ constexpr int pow2_at_least(int v) {
  int r = 32;
  while (r < v) r *= 2;
  return r;
}

// WB = false: e4m3 weights, activations split into two e4m3 terms (hi, lo)
// and a scale per row; WB = true: 16-bit (bf16 or f16) weights (64 K per
// 128-byte slab row) and the activations themselves, in the weights' format,
// as the one B operand, no scales.
template <int N, bool WB = false>
struct TcCfg {
  static constexpr int kWBytes = kTcRows * kSlabK;  // weight slab, 128-byte swizzle
  static constexpr int kTermBytes = N * kSlabK;     // one B operand [N][128 bytes]
  static constexpr int kXBytes = WB ? kTermBytes : (int)tc_split_block_bytes(N);  // (hi, lo, e) or x
  static constexpr int kSwOff = kWBytes + kXBytes;  // four fp32 weight scales
  static constexpr int kStageBytes = (kSwOff + 16 + 1023) / 1024 * 1024;
  // 4 stages hold 128 KB of weights in flight per SM (measured as fast as 5
  // or 6) and leave room beside the CTA for a shared-SM gather CTA up to N = 32.
  static constexpr int kStages = 4;
  static constexpr int kSmem = kStages * kStageBytes + 1024;
  static constexpr int kDCols = WB ? 2 * N : 4 * N;  // one TMEM accumulator buffer: 2 tiles x (2N or N) columns
  static constexpr int kDBufs = N <= 32 ? 4 : 2;
  static constexpr int kTmemCols = pow2_at_least(kDBufs * kDCols);
  // Partial-sum slot of one CTA run: the sums of its 256 rows x N columns as
  // float4 groups, group q of row r at q * 256 + r, so a warp's 32 rows are
  // 512 contiguous bytes for both the GEMM's stores and the settle's loads.
  static constexpr int kSlotFloats = kTcRows * N;
};
static_assert(TcCfg<16>::kSmem + 1024 <= 227 * 1024, "decode_tc: shared memory");
static_assert(TcCfg<32>::kSmem + 1024 <= 227 * 1024, "decode_tc: shared memory");
static_assert(TcCfg<48>::kSmem + 1024 <= 227 * 1024, "decode_tc: shared memory");
static_assert(TcCfg<64>::kSmem + 1024 <= 227 * 1024, "decode_tc: shared memory");
static_assert(TcCfg<64>::kTmemCols <= 512, "decode_tc: TMEM columns");
// A shared-SM gather CTA (3 x 16 KB stages) fits beside one GEMM CTA up to N = 32
// (228 KB of shared memory per SM, 1 KB reserved per CTA).
static_assert(TcCfg<32>::kSmem + 1024 + 3 * 16384 + 1024 <= 228 * 1024, "decode_tc: room for a gather CTA");

__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);  // start address
  d |= (uint64_t)1 << 16;                  // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;        // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                  // descriptor version
  d |= (uint64_t)2 << 61;                  // SWIZZLE_128B
  return d;
}

// kind::f8f6f4 instruction descriptor: A, B e4m3, D f32, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f8(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
// kind::f16 instruction descriptor: A, B bf16 (or f16 when f16 is set), D f32,
// both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_16(int m, int n, bool f16) {
  return (1u << 4) | (f16 ? 0u : (1u << 7) | (1u << 10)) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D (TMEM) (+)= A (shared memory) x B (shared memory).
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   dev::smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 16 consecutive fp32 columns, without waiting for completion.
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 4-byte async copy global -> shared (zero fill when src_bytes == 0).
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gsrc, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dev::smem_addr(smem_dst)), "l"(gsrc),
               "r"(src_bytes)
               : "memory");
}
// Arrives on `bar` once this thread's earlier cp.async copies have landed
// (the arrival counts toward the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(dev::smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Two fp32 lanes per instruction (packed .f32x2 arithmetic, each lane rounded
// as the scalar instruction would): a += (s * e) * (h + l) for a pair of
// columns, the same three roundings in the same order as the scalar form.
__device__ __forceinline__ void promote2(float& a0, float& a1, uint64_t ss, float e0, float e1, uint32_t h0,
                                         uint32_t h1, uint32_t l0, uint32_t l1) {
  uint64_t acc, ee, hh, ll;
  asm("mov.b64 %0, {%1, %2};" : "=l"(acc) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(ee) : "f"(e0), "f"(e1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(hh) : "r"(h0), "r"(h1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(ll) : "r"(l0), "r"(l1));
  asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(ee) : "l"(ss));
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(hh) : "l"(ll));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(ee), "l"(hh));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(acc));
}

// Every lane waits; the warp fails if any lane ran out of time.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  const bool ok = dev::mbar_wait(bar, parity, kWaitLimitNs);
  return __all_sync(0xffffffffu, ok);
}

// Two fp32 -> e4m3 (round to nearest even, saturating); `lo` in the low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two_bytes) {
  const uint32_t h = e4m3x2_to_f16x2(two_bytes);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// ---- 1. activation split ---------------------------------------------------------

// What the split kernels read: the linears whose activations they split, with
// the first thread of each (a few hundred bytes of launch parameters instead
// of the GEMM's tensor maps).
struct SplitLinear {
  const uint16_t* x;  // bf16 [m, cols]
  uint8_t* xs;        // its split blocks, one per K slab
  int64_t cols;
  int64_t thread_end;  // one past the last thread of this linear
};
struct SplitParams {
  SplitLinear l[kMaxDecodeGroup];
  int32_t n;  // linears
  int32_t m;
  uint64_t* trace;
};
// The linear of thread `tid`, or -1 past the last one; `first` receives its first thread.
__device__ __forceinline__ int split_linear_of(const SplitParams& sp, int64_t tid, int64_t* first) {
  int64_t b = 0;
  for (int j = 0; j < sp.n; ++j) {
    if (tid < sp.l[j].thread_end) {
      *first = b;
      return j;
    }
    b = sp.l[j].thread_end;
  }
  return -1;
}

// Eight consecutive threads per (entry, K slab, row), 16 activations each. The
// thread count is a multiple of 128, so whole warps are either in or out.
__global__ void __launch_bounds__(256) split_x_kernel(const __grid_constant__ SplitParams sp, int32_t n_pad) {
  // Let the GEMM launch now: it waits for this grid's results before it reads them.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) dev::trace_start(sp.trace);  // the linear's trace spans all three kernels
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int g = (int)(tid & 7);
  int64_t first = 0;
  const int j = split_linear_of(sp, tid, &first);
  if (j < 0) return;
  const SplitLinear& e = sp.l[j];
  const int64_t task = (tid - first) >> 3;  // (slab, row) of the linear
  const int64_t kb = task / n_pad;
  const int r = (int)(task - kb * n_pad);
  const int64_t col = kb * kSlabK + g * 16;
  float v[16];
  if (r < sp.m && col < e.cols) {  // cols is a multiple of 16: a group is all in or all out
    const uint4* src = reinterpret_cast<const uint4*>(e.x + (int64_t)r * e.cols + col);
    const uint4 r0 = __ldg(src), r1 = __ldg(src + 1);
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
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(v[i]));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
  // e = 2^(E - 134) for amax with biased exponent E, so amax / e is in
  // [128, 256); 1 for an all-zero (or below 2^-119) row slab.
  const uint32_t E = __float_as_uint(a) >> 23;
  const bool big = E > 7;
  const float es = big ? __uint_as_float((E - 7) << 23) : 1.f;
  const float inv = big ? __uint_as_float((261 - E) << 23) : 1.f;
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float s0 = v[4 * i] * inv, s1 = v[4 * i + 1] * inv;
    const float s2 = v[4 * i + 2] * inv, s3 = v[4 * i + 3] * inv;
    const uint32_t h01 = f32x2_to_e4m3x2(s0, s1), h23 = f32x2_to_e4m3x2(s2, s3);
    const float2 b01 = e4m3x2_to_f32x2(h01), b23 = e4m3x2_to_f32x2(h23);
    const uint32_t l01 = f32x2_to_e4m3x2(s0 - b01.x, s1 - b01.y);
    const uint32_t l23 = f32x2_to_e4m3x2(s2 - b23.x, s3 - b23.y);
    hi[i] = h01 | (h23 << 16);
    lo[i] = l01 | (l23 << 16);
  }
  // Row r at r * 128, 16-byte chunk g at (g ^ (r & 7)) * 16: the 128-byte
  // swizzle of a 1024-byte aligned tile.
  uint8_t* blk = e.xs + kb * tc_split_block_bytes(n_pad);
  const int off = r * 128 + ((g ^ (r & 7)) << 4);
  *reinterpret_cast<uint4*>(blk + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  *reinterpret_cast<uint4*>(blk + n_pad * 128 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  if (g == 0) reinterpret_cast<float*>(blk + 2 * n_pad * 128)[r] = es;
}

// 16-bit weights: the B operand of a (entry, 64-K slab) block is the
// activations themselves - as bf16, or rounded to f16 (to_f16) for f16
// weights - [n_pad rows][128 bytes] in the 128-byte swizzled order, zero past m
// and past cols. Eight threads per (entry, slab, row), one 16-byte piece each.
__global__ void __launch_bounds__(256) split_x_16_kernel(const __grid_constant__ SplitParams sp, int32_t n_pad,
                                                          int32_t to_f16) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) dev::trace_start(sp.trace);
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int g = (int)(tid & 7);
  int64_t first = 0;
  const int j = split_linear_of(sp, tid, &first);
  if (j < 0) return;
  const SplitLinear& e = sp.l[j];
  const int64_t task = (tid - first) >> 3;
  const int64_t kb = task / n_pad;
  const int r = (int)(task - kb * n_pad);
  const int64_t col = kb * 64 + g * 8;
  uint4 v = make_uint4(0, 0, 0, 0);
  if (r < sp.m && col < e.cols) v = __ldg(reinterpret_cast<const uint4*>(e.x + (int64_t)r * e.cols + col));
  if (to_f16) {
    v.x = bf16x2_to_f16x2(v.x);
    v.y = bf16x2_to_f16x2(v.y);
    v.z = bf16x2_to_f16x2(v.z);
    v.w = bf16x2_to_f16x2(v.w);
  }
  *reinterpret_cast<uint4*>(e.xs + kb * (int64_t)n_pad * 128 + r * 128 + ((g ^ (r & 7)) << 4)) = v;
}

// ---- 2. GEMM ---------------------------------------------------------------------

// Walks a CTA's consecutive units like an odometer (K slab, then row block,
// then entry), so the per-unit loop needs no division and reads the launch
// parameters only when the entry changes.
struct UnitCursor {
  int j;
  int64_t rbl, kb;
  int32_t slabs;
  int64_t nrb, rb_begin, rows, scale_cols, row_base, unit_begin, y_rows;
  const float* scales;
  const uint8_t* xs;
  uint16_t* y;
  __device__ __forceinline__ void load(const DecodeParams& p) {
    const DecodeEntry& e = p.e[j];
    slabs = e.slabs;
    rows = e.rows;
    row_base = e.row_base;
    unit_begin = e.unit_begin;
    y_rows = e.y_rows;
    y = e.y;
    nrb = (e.rows + kTcRows - 1) / kTcRows;
    rb_begin = e.rb_begin;
    scale_cols = e.scale_cols;
    scales = e.scales;
    xs = e.xs;
  }
  __device__ __forceinline__ void init(const DecodeParams& p, int64_t u) {
    const UnitPos up = unit_pos(p, u);
    j = up.j;
    rbl = up.rbl;
    kb = up.kb;
    load(p);
  }
  __device__ __forceinline__ void next(const DecodeParams& p) {
    if (++kb < slabs) return;
    kb = 0;
    if (++rbl < nrb) return;
    rbl = 0;
    if (++j < p.n_entries) load(p);
  }
};

// End of a run of units on one row block (acc holds its sums): a run that
// covers the whole row block writes Y; a partial run stores its sums in the
// CTA's slot (first or last run) for the settle kernel. Everything comes from
// the cursor's registers: no launch-parameter reads at the end of a run.
template <int N>
__device__ __forceinline__ void tc_end_run(float (&acc)[N], const DecodeParams& p, const RunGeom& geo,
                                           const UnitCursor& cur, int64_t first_rbg, int t, int row) {
  const int64_t fu = cur.unit_begin + cur.rbl * cur.slabs;  // the row block's first unit
  const bool partial = cta_of(fu, geo.G, geo.U) != cta_of(fu + cur.slabs - 1, geo.G, geo.U);
  const int64_t o = cur.rbl * kTcRows + t * 128 + row;      // row of the entry
  if (!partial) {
    if (o < cur.rows) {
      const int m = p.m;
#pragma unroll
      for (int mm = 0; mm < N; ++mm)
        if (mm < m) {
          const __nv_bfloat16 b = __float2bfloat16_rn(acc[mm]);
          cur.y[(int64_t)mm * cur.y_rows + cur.row_base + o] = *reinterpret_cast<const uint16_t*>(&b);
        }
    }
  } else {
    const int64_t slot = 2 * geo.c + (cur.rb_begin + cur.rbl == first_rbg ? 0 : 1);
    float4* d = reinterpret_cast<float4*>(p.partials + slot * (int64_t)TcCfg<N>::kSlotFloats) + (t * 128 + row);
#pragma unroll
    for (int q = 0; q < N / 4; ++q)
      d[q * kTcRows] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
  }
#pragma unroll
  for (int mm = 0; mm < N; ++mm) acc[mm] = 0.f;
}

template <int N, int WT>
__global__ void __launch_bounds__(kTcThreads, 1) decode_tc_kernel(const __grid_constant__ DecodeParams p) {
  constexpr bool WB = WT != 0;  // 16-bit weights, no scales
  using Cf = TcCfg<N, WB>;
  constexpr int S = Cf::kStages;
  extern __shared__ uint8_t dsm[];
  constexpr int kDBufs = Cf::kDBufs;
  __shared__ __align__(8) uint64_t sfull[S], sempty[S], dfull[kDBufs], dempty[kDBufs], mdone;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  // Swizzled TMA tiles and MMA operands need 1024-byte aligned bases.
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t U = p.units, G = gridDim.x, c = blockIdx.x;
  const int64_t u0 = c * U / G, u1 = (c + 1) * U / G, n = u1 - u0;

  if (tid == 0) {
    dev::trace_start(p.trace);
    for (int s = 0; s < S; ++s) {
      dev::mbar_init(&sfull[s], 2);              // expect_tx arrival + the scale copies' arrival
      dev::mbar_init(&sempty[s], 1 + kWorkers);  // MMA commit + the workers (they read e)
    }
    for (int b = 0; b < kDBufs; ++b) {
      dev::mbar_init(&dfull[b], 1);
      dev::mbar_init(&dempty[b], kWorkers);
    }
    dev::mbar_init(&mdone, 1);
    dev::fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dev::smem_addr(&s_tmem)),
                 "r"(Cf::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const RunGeom geo{G, U, c};

  if (warp == 0) {
    // ---- producer ------------------------------------------------------------
    if (lane == 0) {
      for (int j = 0; j < p.n_entries; ++j)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.e[j].tmap)) : "memory");
      const uint64_t stream_policy = l2_evict_first_policy();
      // Split-block copies of the first stages wait for the split kernel; the
      // weight loads of those stages go out before it has finished.
      const uint8_t* pend_src[S];
      bool split_ready = false;
      auto finish_split = [&](int64_t issued) {
        grid_dependency_wait();
        split_ready = true;
        for (int64_t k = 0; k < issued; ++k)
          dev::bulk_g2s(smem + k * Cf::kStageBytes + Cf::kWBytes, pend_src[k], Cf::kXBytes, &sfull[k]);
      };
      UnitCursor cur;
      cur.init(p, u0);
      int64_t i = 0;
      for (; i < n && !s_abort; ++i, cur.next(p)) {
        if (!split_ready && i == S) finish_split(S);  // stage 0's reuse needs its split data
        const int s = (int)(i % S);
        if (!dev::mbar_wait(&sempty[s], (uint32_t)(((i / S) & 1) ^ 1), kWaitLimitNs)) {
          dev::set_status(p.status, SWS_E_TIMEOUT);
          s_abort = 1;
          break;
        }
        uint8_t* st = smem + s * Cf::kStageBytes;
        dev::mbar_arrive_expect_tx(&sfull[s], Cf::kWBytes + Cf::kXBytes);
        tma_load_2d_hint(st, &p.e[cur.j].tmap, (int32_t)(cur.kb * kSlabK), (int32_t)(cur.rbl * kTcRows), &sfull[s],
                         stream_policy);
        // Block scales of each 128-row tile's first and last row (a segment's
        // tile may cross a 128-row scale block of its linear).
        float* sw = reinterpret_cast<float*>(st + Cf::kSwOff);
        if constexpr (!WB) {  // bf16 weights have no scales
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int64_t lr0 = cur.rbl * kTcRows + t * 128;  // first row of the tile in the entry
            const bool in = lr0 < cur.rows;
            const int64_t g0 = cur.row_base + lr0;
            const int64_t g1 = cur.row_base + (lr0 + 127 < cur.rows ? lr0 + 127 : cur.rows - 1);
            cp_async4(sw + 2 * t, cur.scales + (in ? (g0 >> 7) * cur.scale_cols + cur.kb : 0), in ? 4u : 0u);
            cp_async4(sw + 2 * t + 1, cur.scales + (in ? (g1 >> 7) * cur.scale_cols + cur.kb : 0), in ? 4u : 0u);
          }
        }
        cp_async_arrive_noinc(&sfull[s]);  // (with no copies pending it arrives at once)
        const uint8_t* src = cur.xs + cur.kb * Cf::kXBytes;
        if (split_ready)
          dev::bulk_g2s(st + Cf::kWBytes, src, Cf::kXBytes, &sfull[s]);
        else
          pend_src[i] = src;
      }
      if (!split_ready) finish_split(i);  // also completes the stages of an early abort
      // Before the CTA may exit, every issued stage must have landed.
      for (int64_t k = i - S; k < i; ++k)
        if (k >= 0) dev::mbar_wait(&sfull[(int)(k % S)], (uint32_t)((k / S) & 1), kWaitLimitNs / 4);
      // This CTA reads nothing more from the weights: once every CTA is here,
      // the settle grid may launch (it waits for this grid's results), and
      // with it a gather that follows on the stream may overwrite the slot.
      asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
  } else if (warp == 1) {
    // ---- MMA issuer ----------------------------------------------------------
    if (lane == 0) {
      // B is the split block's hi and lo operands as one 2N-row operand, so
      // each weight tile is read once: D[:, 0:N] = A hi^T, D[:, N:2N] = A lo^T.
      // bf16: B is x itself, D[:, 0:N] = A x^T, 16 K per MMA.
      constexpr uint32_t idesc = WB ? idesc_16(128, N, WT == 2) : idesc_f8(128, 2 * N);
      bool issued = false;
      for (int64_t i = 0; i < n && !s_abort; ++i) {
        const int s = (int)(i % S), b = (int)(i % kDBufs);
        if (!dev::mbar_wait(&sfull[s], (uint32_t)((i / S) & 1), kWaitLimitNs) ||
            !dev::mbar_wait(&dempty[b], (uint32_t)(((i / kDBufs) & 1) ^ 1), kWaitLimitNs)) {
          dev::set_status(p.status, SWS_E_TIMEOUT);
          s_abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t wa = dev::smem_addr(smem + s * Cf::kStageBytes);
        const uint32_t xb = wa + Cf::kWBytes;
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int k = 0; k < kSlabK / 32; ++k) {  // 32 bytes of K per MMA
            const uint32_t d = tmem + b * Cf::kDCols + t * (Cf::kDCols / 2);
            if constexpr (WB)
              mma_16(d, smem_desc_sw128(wa + t * (128 * kSlabK) + k * 32), smem_desc_sw128(xb + k * 32), idesc,
                     k != 0);
            else
              mma_f8(d, smem_desc_sw128(wa + t * (128 * kSlabK) + k * 32), smem_desc_sw128(xb + k * 32), idesc,
                     k != 0);
          }
        mma_commit(&sempty[s]);
        mma_commit(&dfull[b]);
        issued = true;
      }
      if (issued) {  // all MMAs of this CTA complete before TMEM is released
        mma_commit(&mdone);
        dev::mbar_wait(&mdone, 0, kWaitLimitNs);
      }
    }
  } else {
    // ---- workers: promote each unit's slab result ---------------------------------
    const int q = warp & 3;         // TMEM lane quarter of this warp
    const int t = (warp - 2) >> 2;  // the unit's 128-row tile this warp promotes
    const int row = q * 32 + lane;  // row inside the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    float acc[N];
#pragma unroll
    for (int mm = 0; mm < N; ++mm) acc[mm] = 0.f;
    bool fail = false;
    UnitCursor cur;
    cur.init(p, u0);
    const int64_t first_rbg = cur.rb_begin + cur.rbl;
    for (int64_t i = 0; i < n; ++i, cur.next(p)) {
      const int s = (int)(i % S), b = (int)(i % kDBufs);
      fail = !warp_wait(&sfull[s], (uint32_t)((i / S) & 1)) || !warp_wait(&dfull[b], (uint32_t)((i / kDBufs) & 1));
      if (fail) break;
      tc_fence_after();
      const uint8_t* st = smem + s * Cf::kStageBytes;
      const uint32_t dcol = tmem + lane_off + b * Cf::kDCols + t * (Cf::kDCols / 2);
      if constexpr (WB) {  // no scales: the slab's products add straight in
#pragma unroll
        for (int c0 = 0; c0 < N; c0 += 16) {
          uint32_t rh[16];
          tmem_ld16_nowait(dcol + c0, rh);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 16; ++k) acc[c0 + k] += __uint_as_float(rh[k]);
        }
      } else {
        const float* ex = reinterpret_cast<const float*>(st + Cf::kWBytes + 2 * Cf::kTermBytes);
        // this row's 128-row scale block: the tile's first or last one
        const float* swt = reinterpret_cast<const float*>(st + Cf::kSwOff) + 2 * t;
        const int64_t g0 = cur.row_base + cur.rbl * kTcRows + t * 128;
        const float sw = ((g0 + row) >> 7) == (g0 >> 7) ? swt[0] : swt[1];
        uint64_t ss;  // (sw, sw) for the packed multiply
        asm("mov.b64 %0, {%1, %1};" : "=l"(ss) : "f"(sw));
#pragma unroll
        for (int c0 = 0; c0 < N; c0 += 16) {  // hi columns; lo N further
          uint32_t rh[16], rl[16];
          tmem_ld16_nowait(dcol + c0, rh);
          tmem_ld16_nowait(dcol + N + c0, rl);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 16; k += 2)
            promote2(acc[c0 + k], acc[c0 + k + 1], ss, ex[c0 + k], ex[c0 + k + 1], rh[k], rh[k + 1], rl[k], rl[k + 1]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        dev::mbar_arrive(&dempty[b]);
        dev::mbar_arrive(&sempty[s]);
      }
      if (i + 1 == n || cur.kb + 1 == cur.slabs) tc_end_run<N>(acc, p, geo, cur, first_rbg, t, row);
    }
    if (fail) {
      dev::set_status(p.status, SWS_E_TIMEOUT);
      s_abort = 1;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(Cf::kTmemCols)
                 : "memory");
  }
  if (p.trace && tid == 0) {  // the record's end stamp after this kernel's writes
    __threadfence();
    dev::trace_end(p.trace, p.tag);
  }
}

// ---- 3. split-K settle ------------------------------------------------------------

// A row block that the GEMM's partition split between CTAs, worked out on the
// host from the same partition, with everything its settle block needs: the
// block's one read of its task is all the launch-parameter traffic it makes.
struct SettleTask {
  uint16_t* y;      // Y[0, first row of the row block] (bf16, rows `ystride` apart in m)
  int32_t ystride;  // rows of the linear
  int32_t rows;     // rows of the row block inside its entry (<= 256)
  int32_t cf, cl;   // the CTAs that share it, in K order
  int32_t cf_slot;  // partial slot of CTA cf (its first or its second run); a later CTA's is its first, 2c
  int32_t pad;
};
struct SettlePlan {
  int32_t n;  // tasks
  int32_t m;
  const float* partials;
  uint64_t* trace;
  uint64_t tag;
  SettleTask task[kMaxGrid];
};

// Adds the partial sums of one settle task in K (CTA) order, so the result does
// not depend on timing, and writes Y for columns [c0, c0 + C). Thread r owns row
// r of the row block; it issues the loads of up to KB contributions before
// adding them.
template <int N, int C>
__device__ __forceinline__ void settle_task(const SettleTask& tk, const float* partials, int m, int c0) {
  constexpr int KB = C <= 16 ? 4 : C <= 32 ? 2 : 1;  // contributions loaded at once: 12-16 float4 a thread
  constexpr int64_t kSlot = TcCfg<N>::kSlotFloats;
  const int row = threadIdx.x;
  if (row >= tk.rows) return;  // past the entry (segment); straddling rows are in none
  float4 acc[C / 4];
#pragma unroll
  for (int q = 0; q < C / 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int32_t cb = tk.cf; cb <= tk.cl; cb += KB) {
    float4 v[KB][C / 4];
#pragma unroll
    for (int k = 0; k < KB; ++k)
      if (cb + k <= tk.cl) {
        const int64_t slot = cb + k == tk.cf ? tk.cf_slot : 2 * (int64_t)(cb + k);
        const float4* s4 = reinterpret_cast<const float4*>(partials + slot * kSlot) + (c0 / 4) * kTcRows + row;
#pragma unroll
        for (int q = 0; q < C / 4; ++q) v[k][q] = __ldcg(s4 + q * kTcRows);
      }
#pragma unroll
    for (int k = 0; k < KB; ++k)
      if (cb + k <= tk.cl) {
#pragma unroll
        for (int q = 0; q < C / 4; ++q) {
          acc[q].x += v[k][q].x;
          acc[q].y += v[k][q].y;
          acc[q].z += v[k][q].z;
          acc[q].w += v[k][q].w;
        }
      }
  }
#pragma unroll
  for (int q = 0; q < C / 4; ++q) {
    const float a[4] = {acc[q].x, acc[q].y, acc[q].z, acc[q].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int mm = c0 + 4 * q + k;
      if (mm < m) {
        const __nv_bfloat16 b = __float2bfloat16_rn(a[k]);
        tk.y[(int64_t)mm * tk.ystride + row] = *reinterpret_cast<const uint16_t*>(&b);
      }
    }
  }
}

__device__ __forceinline__ void settle_trace_end(const SettlePlan& sp) {
  __syncwarp();
  if (sp.trace && (threadIdx.x & 31) == 0) {  // the record's end stamp after this kernel's writes
    __threadfence();
    dev::trace_end(sp.trace, sp.tag);
  }
}

// Slot path: one block per settle task, all N columns (a launch has fewer
// tasks than CTAs, so the grid is one wave).
template <int N>
__global__ void __launch_bounds__(kTcRows) settle_kernel(const __grid_constant__ SettlePlan sp) {
  // A gather launched next on the stream (programmatic serialisation) may
  // start now: this grid launched once every GEMM CTA had read all its
  // weights, the gather writes a slot, which nothing here reads, and reads
  // chunks, which nothing here writes; later stream work still waits for
  // this grid.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  grid_dependency_wait();  // the GEMM's results are complete and visible
  settle_task<N, N>(sp.task[blockIdx.x], sp.partials, sp.m, 0);
  settle_trace_end(sp);
}

// Chunk-map path: the settle tasks as above, then one block per straddling row
// and 16-column group: that row is in no segment, so the block computes it
// directly from the chunks (straddle_row).
template <int N, int WT>
__device__ void straddle_row(const DecodeParams& p, int sidx, int c0);

template <int N, int WT>
__global__ void __launch_bounds__(kTcRows) settle_fused_kernel(const __grid_constant__ DecodeParams p,
                                                               const __grid_constant__ SettlePlan sp) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // as in settle_kernel
  grid_dependency_wait();
  const int b = (int)blockIdx.x;
  if (b < sp.n)
    settle_task<N, N>(sp.task[b], sp.partials, sp.m, 0);
  else
    straddle_row<N, WT>(p, (b - sp.n) / (N / 16), (b - sp.n) % (N / 16) * 16);
  settle_trace_end(sp);
}

// Row st.row of a linear, read through the chunk map (a chunk boundary falls
// inside it), for outputs m = c0 .. c0 + 15. The block stages the row in 4 KB
// windows (32 slabs of 128 bytes; 16-byte pieces never straddle a boundary,
// which is a multiple of 16), so each window costs one memory round trip. Warp
// w takes slabs w, w + 8, ... of a window and each lane four weights of a slab
// (e4m3: 4 bytes, times the slab's block scale; bf16: 8 bytes, no scale); a
// lane accumulates x * w over its slabs for every m, and the warps' sums are
// added once at the end, warp by warp in a fixed order.
template <int N, int WT>
__device__ void straddle_row(const DecodeParams& p, int sidx, int c0) {
  constexpr bool WB = WT != 0;
  constexpr int kWin = 32 * kSlabK;  // bytes per window
  constexpr int kWarps = kTcRows / 32;
  constexpr int kElem = WB ? 2 : 1;
  __shared__ __align__(16) uint8_t wbuf[kWin];
  __shared__ float sbuf[32];
  __shared__ float part[kWarps][16];
  const DecodeEntry& e = p.e[p.st.entry[sidx]];  // a segment of the linear: its pointers
  const int64_t r = p.st.row[sidx];                // row of the linear
  const int64_t cols = e.cols, rowb = cols * kElem, rows = e.y_rows, C = p.chunk_bytes;
  const int64_t t0 = e.t_offset + r * rowb;
  const float* srow = WB ? nullptr : e.scales + (r >> 7) * e.scale_cols;
  uint16_t* const y = e.y;
  const int slabs = e.slabs, m = p.m;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float acc[16];
#pragma unroll
  for (int h = 0; h < 16; ++h) acc[h] = 0.f;
  for (int64_t w0 = 0; w0 < rowb; w0 += kWin) {
    __syncthreads();  // the previous window is consumed
    for (int t = threadIdx.x; t < kWin / 16; t += blockDim.x) {
      const int64_t k = w0 + 16 * t;
      if (k < rowb) {
        const int64_t g = t0 + k;
        *reinterpret_cast<uint4*>(wbuf + 16 * t) = *reinterpret_cast<const uint4*>(p.chunks[g / C] + g % C);
      }
    }
    const int kb0 = (int)(w0 / kSlabK);
    if (!WB && threadIdx.x < 32)
      sbuf[threadIdx.x] = kb0 + (int)threadIdx.x < slabs ? __ldg(srow + kb0 + threadIdx.x) : 0.f;
    __syncthreads();
    for (int sl = warp; sl < 32; sl += kWarps) {
      if constexpr (WB) {
        // 64 bf16 weights per slab: lane takes weights 2*lane, 2*lane + 1 (one
        // 4-byte word), k = (w0 + sl*128)/2 + 2*lane
        const int64_t kb = w0 + sl * kSlabK + lane * 4;  // byte offset in the row
        if (kb >= rowb) break;
        const int64_t k = kb / 2;
        const uint32_t w2 = *reinterpret_cast<const uint32_t*>(wbuf + sl * kSlabK + lane * 4);
        float a0, a1;
        if constexpr (WT == 2) {  // f16 weights; x takes the f16 operand's rounding too
          const float2 wf = __half22float2(*reinterpret_cast<const __half2*>(&w2));
          a0 = wf.x;
          a1 = wf.y;
        } else {
          a0 = __uint_as_float(w2 << 16);
          a1 = __uint_as_float(w2 & 0xffff0000u);
        }
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          if (c0 + h < m) {
            uint32_t x2 = *reinterpret_cast<const uint32_t*>(e.x + (int64_t)(c0 + h) * cols + k);
            float x0, x1;
            if constexpr (WT == 2) {
              x2 = bf16x2_to_f16x2(x2);
              const float2 xf = __half22float2(*reinterpret_cast<const __half2*>(&x2));
              x0 = xf.x;
              x1 = xf.y;
            } else {
              x0 = __uint_as_float(x2 << 16);
              x1 = __uint_as_float(x2 & 0xffff0000u);
            }
            acc[h] = fmaf(x1, a1, fmaf(x0, a0, acc[h]));
          }
        }
      } else {
        const int64_t k = w0 + sl * kSlabK + lane * 4;
        if (k >= cols) break;  // cols % 16 == 0: four weights are all in or all out
        const uint32_t w4 = *reinterpret_cast<const uint32_t*>(wbuf + sl * kSlabK + lane * 4);
        const float2 w01 = e4m3x2_to_f32x2(w4), w23 = e4m3x2_to_f32x2(w4 >> 16);
        const float sc = sbuf[sl];
        const float a0 = sc * w01.x, a1 = sc * w01.y, a2 = sc * w23.x, a3 = sc * w23.y;
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          if (c0 + h < m) {
            const uint2 x4 = *reinterpret_cast<const uint2*>(e.x + (int64_t)(c0 + h) * cols + k);
            float v = acc[h];
            v = fmaf(__uint_as_float(x4.x << 16), a0, v);
            v = fmaf(__uint_as_float(x4.x & 0xffff0000u), a1, v);
            v = fmaf(__uint_as_float(x4.y << 16), a2, v);
            acc[h] = fmaf(__uint_as_float(x4.y & 0xffff0000u), a3, v);
          }
        }
      }
    }
  }
#pragma unroll
  for (int h = 0; h < 16; ++h) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], off);
    if (lane == 0) part[warp][h] = acc[h];
  }
  __syncthreads();
  if (threadIdx.x < 16) {
    const int h = threadIdx.x;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) v += part[w][h];
    if (c0 + h < m && r < rows) {
      const __nv_bfloat16 b = __float2bfloat16_rn(v);
      y[(int64_t)(c0 + h) * rows + r] = *reinterpret_cast<const uint16_t*>(&b);
    }
  }
}

// Host copy of the partition's arithmetic (unit_pos, cta_of, RunGeom).
void settle_plan(const DecodeParams& p, int64_t G, SettlePlan* sp) {
  const int64_t U = p.units;
  auto pos = [&](int64_t u) {
    int j = 0;
    for (int q = 1; q < p.n_entries && u >= p.e[q].unit_begin; ++q) j = q;
    const int64_t local = u - p.e[j].unit_begin;
    UnitPos r;
    r.j = j;
    r.rbl = local / p.e[j].slabs;
    r.kb = local - r.rbl * p.e[j].slabs;
    r.rbg = p.e[j].rb_begin + r.rbl;
    return r;
  };
  auto cta = [&](int64_t u) { return ((u + 1) * G - 1) / U; };
  sp->n = 0;
  sp->m = p.m;
  sp->partials = p.partials;
  sp->trace = p.trace;
  sp->tag = p.tag;
  for (int64_t c = 1; c < G; ++c) {
    const UnitPos up = pos(c * U / G);
    if (up.kb == 0) continue;  // the boundary is a row-block start: nothing is split here
    if (c > 1) {               // an earlier boundary inside the same row block settles it
      const UnitPos prev = pos((c - 1) * U / G);
      if (prev.rbg == up.rbg && prev.kb != 0) continue;
    }
    const DecodeEntry& e = p.e[up.j];
    const int64_t fu = e.unit_begin + up.rbl * e.slabs;
    SettleTask& t = sp->task[sp->n++];
    t.y = e.y + e.row_base + up.rbl * kTcRows;
    t.ystride = (int32_t)e.y_rows;
    t.rows = (int32_t)std::min<int64_t>(kTcRows, e.rows - up.rbl * kTcRows);
    t.cf = (int32_t)cta(fu);
    t.cl = (int32_t)cta(fu + e.slabs - 1);
    // CTA cf holds the row block's first units: its first run if its range
    // starts inside the row block, else its last (second) run.
    t.cf_slot = 2 * t.cf + (pos(t.cf * U / G).rbg == up.rbg ? 0 : 1);
    t.pad = 0;
  }
}

// The split kernels' parameters: the linears whose activations a launch splits
// (the owner entry of each; chunk-map segments of one linear share its blocks).
// A group has at most kMaxDecodeGroup linears; more owners leave sp.n at -1.
SplitParams split_params(const DecodeParams& p, int64_t n_pad, bool w16) {
  SplitParams sp = {};
  sp.m = p.m;
  sp.trace = p.trace;
  int64_t end = 0;
  for (int j = 0; j < p.n_entries; ++j) {
    if (!p.e[j].split_owner) continue;
    if (sp.n == kMaxDecodeGroup) {
      sp.n = -1;
      return sp;
    }
    SplitLinear& l = sp.l[sp.n++];
    l.x = p.e[j].x;
    l.xs = p.e[j].xs;
    l.cols = p.e[j].cols;
    // one thread per 16 (e4m3 split) or 8 (16-bit copy) activations of a slab row
    end += (int64_t)p.e[j].slabs * n_pad * 8;
    l.thread_end = end;
  }
  (void)w16;
  return sp;
}

template <int N, bool FUSED, int WT>
cudaError_t launch_tc_n(const DecodeParams& p, int64_t grid_cap, cudaStream_t s) {
  constexpr bool WB = WT != 0;
  constexpr int kSmem = TcCfg<N, WB>::kSmem;
  static PerDevice once;
  const cudaError_t attr = once.run([] {
    cudaError_t a = cudaFuncSetAttribute(decode_tc_kernel<N, WT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (a == cudaSuccess)  // an SM running this CTA can still take a gather CTA
      a = cudaFuncSetAttribute(decode_tc_kernel<N, WT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
    return a;
  });
  if (attr != cudaSuccess) return attr;
  // 1. split the activations of every linear
  const SplitParams spl = split_params(p, N, WB);
  if (spl.n < 1 || spl.n > kMaxDecodeGroup) return cudaErrorInvalidValue;
  const int64_t threads = spl.l[spl.n - 1].thread_end;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributePriority;
  at[0].val.priority = high_priority();
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((threads + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;  // priority only
  cudaError_t e = WB ? cudaLaunchKernelEx(&cfg, split_x_16_kernel, spl, (int)N, (int)(WT == 2))
                     : cudaLaunchKernelEx(&cfg, split_x_kernel, spl, (int)N);
  if (e != cudaSuccess) return e;
  // 2. the GEMM, as a programmatic dependent launch of (1)
  const int64_t grid = std::min<int64_t>({p.units, (int64_t)device_sm_count(), (int64_t)kMaxGrid, grid_cap});
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.numAttrs = 2;  // priority + programmatic stream serialization
  e = cudaLaunchKernelEx(&cfg, decode_tc_kernel<N, WT>, p);
  // 3. the split-K settle (and the straddling rows of a chunk-map launch), as
  //    a programmatic dependent launch of (2)
  if (e != cudaSuccess) return e;
  SettlePlan sp;
  settle_plan(p, grid, &sp);
  const int64_t blocks = sp.n + (FUSED ? (int64_t)p.st.n * (N / 16) : 0);
  if (blocks < 1) return cudaSuccess;
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kTcRows);
  cfg.dynamicSmemBytes = 0;
  if constexpr (FUSED)
    return cudaLaunchKernelEx(&cfg, settle_fused_kernel<N, WT>, p, sp);
  else
    return cudaLaunchKernelEx(&cfg, settle_kernel<N>, sp);
}

template <bool FUSED, int WT>
cudaError_t launch_tc(const DecodeParams& p, int64_t grid_cap, cudaStream_t s) {
  switch ((int)tc_n_pad(p.m)) {
    case 16: return launch_tc_n<16, FUSED, WT>(p, grid_cap, s);
    case 32: return launch_tc_n<32, FUSED, WT>(p, grid_cap, s);
    case 48: return launch_tc_n<48, FUSED, WT>(p, grid_cap, s);
    default: return launch_tc_n<64, FUSED, WT>(p, grid_cap, s);
  }
}

}  // namespace

namespace dec {
cudaError_t launch_decode_tc(const DecodeParams& p, bool fused, int wtype, int64_t grid_cap, cudaStream_t s) {
  switch (wtype) {
    case 1: return fused ? launch_tc<true, 1>(p, grid_cap, s) : launch_tc<false, 1>(p, grid_cap, s);
    case 2: return fused ? launch_tc<true, 2>(p, grid_cap, s) : launch_tc<false, 2>(p, grid_cap, s);
    default: return fused ? launch_tc<true, 0>(p, grid_cap, s) : launch_tc<false, 0>(p, grid_cap, s);
  }
}
int64_t tc_slot_bytes(int64_t m) { return (int64_t)kTcRows * tc_n_pad(m) * 4; }
}  // namespace dec

}  // namespace sws

// Test hook (host only): the settle tasks of a tcgen05 decode launch from
// slot views of the given linears on `grid` CTAs. The unit space is laid out
// as a slot-view launch lays it out (each linear's 256-row blocks in turn,
// ceil(cols * elem_bytes / 128) K slabs each) and settle_plan runs on it;
// the outputs are stand-ins in a host array, so each task's Y pointer tells
// its linear and row block. Writes 6 values per task (linear, row block,
// rows, first CTA, last CTA, partial slot of the first CTA) and returns the
// number of tasks, or a negative status.
extern "C" int sws_test_settle_plan(int32_t n_linears, const int64_t* rows, const int64_t* cols, int32_t elem_bytes,
                                    int64_t grid, int32_t* out, int32_t capacity) {
  using namespace sws;
  using namespace sws::dec;
  if (n_linears < 1 || n_linears > kMaxDecodeGroup || !rows || !cols || !out || capacity < 0)
    return fail(SWS_E_INVALID, "test_settle_plan: %d linears", n_linears);
  if (elem_bytes != 1 && elem_bytes != 2) return fail(SWS_E_INVALID, "test_settle_plan: elem_bytes %d", elem_bytes);
  int64_t total_rows = 0;
  for (int i = 0; i < n_linears; ++i) {
    if (rows[i] < 1 || rows[i] > ((int64_t)1 << 24) || cols[i] < 16 || cols[i] % 16 != 0 || cols[i] > ((int64_t)1 << 24))
      return fail(SWS_E_INVALID, "test_settle_plan: linear %d is [%lld, %lld]", i, (long long)rows[i],
                  (long long)cols[i]);
    total_rows += rows[i];
  }
  std::unique_ptr<DecodeParams> p(new DecodeParams());
  std::vector<uint16_t> ybuf((size_t)total_rows);
  std::vector<int64_t> first_row(n_linears);
  p->n_entries = n_linears;
  p->m = 1;
  p->units = 0;
  int64_t rb = 0, off = 0;
  for (int i = 0; i < n_linears; ++i) {
    DecodeEntry& e = p->e[i];
    e.y = ybuf.data() + off;
    first_row[i] = off;
    e.rows = rows[i];
    e.row_base = 0;
    e.y_rows = rows[i];
    e.linear = i;
    e.split_owner = 1;
    e.cols = cols[i];
    e.slabs = (int32_t)cdiv(cols[i] * elem_bytes, kSlabK);
    e.unit_begin = p->units;
    e.rb_begin = rb;
    const int64_t nrb = cdiv(rows[i], kTcUnitRows);
    rb += nrb;
    p->units += nrb * e.slabs;
    off += rows[i];
  }
  if (grid < 1 || grid > std::min<int64_t>(p->units, kMaxGrid))
    return fail(SWS_E_INVALID, "test_settle_plan: grid %lld for %lld units", (long long)grid, (long long)p->units);
  std::unique_ptr<SettlePlan> sp(new SettlePlan());
  settle_plan(*p, grid, sp.get());
  if (sp->n > capacity) return fail(SWS_E_INVALID, "test_settle_plan: %d tasks, room for %d", sp->n, capacity);
  for (int t = 0; t < sp->n; ++t) {
    const SettleTask& k = sp->task[t];
    const int64_t d = k.y - ybuf.data();
    int i = n_linears - 1;
    while (i > 0 && d < first_row[i]) --i;
    int32_t* o = out + 6 * t;
    o[0] = i;
    o[1] = (int32_t)((d - first_row[i]) / kTcRows);
    o[2] = k.rows;
    o[3] = k.cf;
    o[4] = k.cl;
    o[5] = k.cf_slot;
  }
  return sp->n;
}
