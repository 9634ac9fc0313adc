// Split-K FP8 skinny decode GEMM (m <= 64) on zero-copy weight views, on
// warp-level mma.sync (the tcgen05 kernel in decode_tc.cu is the default).
//
//   Y[m, o] = bf16_rne( sum_kb s[o/128, kb] * sum_{i in kb} x[m, i] * e4m3(q[o, i]) )
//
// (bf16 or f16 weights, WT = 1 or 2: the same without scales, 64 K per
// 128-byte slab row; for f16 weights x is rounded to f16.)
//
// The linear the weight-sharding blog keeps unchanged (section "核心抽象":
// the GEMM sees the full W; Y = X W^T with W [out, in]); block scales are
// 128 x 128, float32. One launch computes a group of up to eight such linears
// (all linears of a layer share m), so launch, ramp-up and drain are paid once.
//
// Design (HBM-bound at decode sizes; every weight byte is read exactly once):
//   * Swap-AB warp-level tensor-core MMA (mma.sync m16n8k16, f16 operands,
//     fp32 accumulate): the weight supplies 16-row A tiles, the activations the
//     8-column B tiles, so m <= 64 costs 1..8 n-tiles. e4m3 -> f16 is exact
//     (one cvt per two weights); the dot product ignores the order of k, so
//     each thread takes 32 contiguous weight bytes per 128-K slab and the
//     activations use the same permutation of k.
//   * Slot path: 128-K weight slabs of the CTA's rows are staged in shared
//     memory by 2-D TMA (128-byte swizzle, zero fill past the edges) through a
//     ring of 3-6 stages with mbarrier completion, issued by one thread, so
//     that >= 128 KB per SM are in flight without holding registers.
//   * Fused path (no slot): the same ring and arithmetic, but every thread
//     copies 16-byte weight pieces with cp.async straight from the chunk that
//     holds them (byte g of T lives in chunk g / C at offset g % C), walking
//     the chunk map incrementally down its rows.
//   * Activations are converted bf16 -> f16 once per CTA and staged in shared
//     memory (double-buffered, XOR-swizzled so that fragment loads are free of
//     bank conflicts); one CTA barrier per 128-K slab.
//   * Block scales: a warp's rows lie inside one 128-row scale block, so the
//     scale is one scalar per warp and slab. The accumulator holds
//     sum_b (s_b / s_cur) P_b and is rescaled by s_prev / s_cur when the scale
//     changes, then multiplied by the last scale at the end of a run.
//   * Split-K across CTAs: the (row block, K slab) units of all linears of the
//     group are concatenated and cut into equal contiguous ranges, one per CTA
//     of a grid sized to the SM count. A CTA that covers a whole row block
//     writes Y directly; partial runs store fp32 sums in the workspace and, once
//     the CTA has streamed all its weights, the last CTA to arrive on a row
//     block (atomic counter, no waiting) adds them in K order and writes Y.
#include <cuda.h>
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

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

// Weight element types: WB = false for e4m3 codes (128 K per 128-byte slab
// row, block scales), WB = true for 16-bit weights (64 K per slab row, no
// scales). Either way a slab row is 128 bytes, so the staging, the swizzle and
// the TMA boxes are the same.
template <bool WB>
__host__ __device__ constexpr int slab_elems() { return WB ? 64 : 128; }

// Position of 16-byte activation unit u (8 elements of k) in row m of a staged
// slab: spreads the units a quarter-warp reads, and neighbouring rows, over all
// 32 banks. e4m3 slabs have 16 units per row, bf16 slabs 8.
template <bool WB>
__device__ __forceinline__ int xpos(int u, int m) {
  if constexpr (WB)
    return u ^ (m & 7);
  else
    return u ^ (((u >> 3) & 1) << 1) ^ (m & 1);
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- activation staging: one slab of bf16 X -> shared (as f16 for e4m3
// weights, as bf16 for bf16 weights) ------------------------------------------
template <int NT, int WT>
struct XStage {
  static constexpr bool WB = WT != 0;
  static constexpr int kRowUnits = slab_elems<WB>() / 8;  // 16-byte units per row
  static constexpr int kUnits = NT * 8 * kRowUnits;         // 16-byte units per slab
  static constexpr int kPer = (kUnits + kThreads - 1) / kThreads;
  uint4 r[kPer];

  __device__ __forceinline__ void load(const DecodeEntry& e, int m, int64_t kb, int tid) {
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int v = tid + i * kThreads;
      const int mrow = v / kRowUnits, q = v % kRowUnits;
      const int64_t k = kb * slab_elems<WB>() + q * 8;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (v < kUnits && mrow < m && k < e.cols)
        val = __ldg(reinterpret_cast<const uint4*>(e.x + (int64_t)mrow * e.cols + k));
      r[i] = val;
    }
  }
  __device__ __forceinline__ void store(uint4* xs, int tid) const {
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int v = tid + i * kThreads;
      if (v < kUnits) {
        const int mrow = v / kRowUnits, q = v % kRowUnits;
        uint4 h = r[i];
        if constexpr (WT != 1) {  // f16 operands: e4m3 and f16 weights
          h.x = bf16x2_to_f16x2(r[i].x);
          h.y = bf16x2_to_f16x2(r[i].y);
          h.z = bf16x2_to_f16x2(r[i].z);
          h.w = bf16x2_to_f16x2(r[i].w);
        }
        xs[mrow * kRowUnits + xpos<WB>(q, mrow)] = h;
      }
    }
  }
};

// ---- MMAs of one 64-K half-slab ---------------------------------------------
// wq[rt][h] holds the 16 weight bytes of row (g + 8h) of row tile rt at
// k = 32*tig + 16*l + [0, 16); the activation fragments come from units
// 4*tig + 2*l and 4*tig + 2*l + 1 of each n-tile row.
template <int NT, int R>
__device__ __forceinline__ void mma_half_e4m3(float (&acc)[R][NT][4], const uint4 (&wq)[R][2], const uint4* xb, int l,
                                              int g, int tig) {
  uint32_t a[R][2][8];
#pragma unroll
  for (int rt = 0; rt < R; ++rt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 wv = wq[rt][h];
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
    const int u = 4 * tig + 2 * l;
    const uint4 b0 = xb[mrow * 16 + xpos<false>(u, mrow)];
    const uint4 b1 = xb[mrow * 16 + xpos<false>(u + 1, mrow)];
    const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int rt = 0; rt < R; ++rt)
        mma16816(acc[rt][nt], a[rt][0][2 * kk], a[rt][1][2 * kk], a[rt][0][2 * kk + 1], a[rt][1][2 * kk + 1],
                 bw[2 * kk], bw[2 * kk + 1]);
  }
}

// 16-bit weights: wq[rt][h] holds the 8 weights of row (g + 8h) of row tile
// rt at k = 16*tig + 8*l + [0, 8); the activations come from unit 2*tig + l
// (bf16, or f16 for f16 weights).
template <int NT, int R, bool F16>
__device__ __forceinline__ void mma_half_16(float (&acc)[R][NT][4], const uint4 (&wq)[R][2], const uint4* xb, int l,
                                            int g, int tig) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int mrow = nt * 8 + g;
    const uint4 b = xb[mrow * 8 + xpos<true>(2 * tig + l, mrow)];
#pragma unroll
    for (int rt = 0; rt < R; ++rt) {
      if constexpr (F16) {
        mma16816(acc[rt][nt], wq[rt][0].x, wq[rt][1].x, wq[rt][0].y, wq[rt][1].y, b.x, b.y);
        mma16816(acc[rt][nt], wq[rt][0].z, wq[rt][1].z, wq[rt][0].w, wq[rt][1].w, b.z, b.w);
      } else {
        mma16816_bf16(acc[rt][nt], wq[rt][0].x, wq[rt][1].x, wq[rt][0].y, wq[rt][1].y, b.x, b.y);
        mma16816_bf16(acc[rt][nt], wq[rt][0].z, wq[rt][1].z, wq[rt][0].w, wq[rt][1].w, b.z, b.w);
      }
    }
  }
}

template <int NT, int R, int WT>
__device__ __forceinline__ void mma_half(float (&acc)[R][NT][4], const uint4 (&wq)[R][2], const uint4* xb, int l,
                                         int g, int tig) {
  if constexpr (WT == 1)
    mma_half_16<NT, R, false>(acc, wq, xb, l, g, tig);
  else if constexpr (WT == 2)
    mma_half_16<NT, R, true>(acc, wq, xb, l, g, tig);
  else
    mma_half_e4m3<NT, R>(acc, wq, xb, l, g, tig);
}

template <int NT, int R>
__device__ __forceinline__ void rescale(float (&acc)[R][NT][4], float f) {
#pragma unroll
  for (int rt = 0; rt < R; ++rt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[rt][nt][e] *= f;
}

template <int NT, int R>
__device__ __forceinline__ void zero(float (&acc)[R][NT][4]) {
#pragma unroll
  for (int rt = 0; rt < R; ++rt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[rt][nt][e] = 0.f;
}

// Scale bookkeeping for one slab of a warp; returns false when the slab's
// scale is zero (it contributes nothing and is skipped).
template <int NT, int R>
__device__ __forceinline__ bool apply_scale(float (&acc)[R][NT][4], float& cs, float s) {
  if (s == 0.f) return false;
  if (cs != 0.f && s != cs) rescale<NT, R>(acc, cs / s);
  cs = s;
  return true;
}

// ---- end of a run -------------------------------------------------------------
// Runs that cover a whole row block write Y at once. A partial run only stores
// its fp32 sums in its slot (first or last run of the CTA); the arrival count
// and the reduction wait until the CTA has streamed all its weights, so no
// fence, barrier or atomic round trip stalls the weight pipeline mid-stream.
template <int NT, int R>
__device__ __forceinline__ void write_y(const float (&acc)[R][NT][4], const DecodeEntry& e, int m, int64_t row0,
                                        int g, int tig) {
  // Into registers first: a store could alias the parameter block, and the
  // compiler would read these again after every store.
  uint16_t* const y = e.y;
  const int64_t rows = e.rows;
#pragma unroll
  for (int rt = 0; rt < R; ++rt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t o = row0 + rt * 16 + g + 8 * (q >> 1);
        const int mm = nt * 8 + 2 * tig + (q & 1);
        if (o < rows && mm < m) {
          const __nv_bfloat16 b = __float2bfloat16_rn(acc[rt][nt][q]);
          y[(int64_t)mm * rows + o] = *reinterpret_cast<const uint16_t*>(&b);
        }
      }
}

template <int NT, int R>
__device__ __forceinline__ void end_run(float (&acc)[R][NT][4], const DecodeParams& p, const RunGeom& geo,
                                        const UnitPos& up, int64_t row0, int warp, int lane) {
  constexpr int kSlot = kWarps * R * NT * 32 * 4;  // floats per partial slot
  if (!geo.partial(p, up.rbg)) {
    write_y<NT, R>(acc, p.e[up.j], p.m, row0, lane >> 2, lane & 3);
  } else {
    float4* slot = reinterpret_cast<float4*>(p.partials + geo.slot(p, geo.c, up.rbg) * (int64_t)kSlot);
#pragma unroll
    for (int rt = 0; rt < R; ++rt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        slot[((warp * R + rt) * NT + nt) * 32 + lane] =
            make_float4(acc[rt][nt][0], acc[rt][nt][1], acc[rt][nt][2], acc[rt][nt][3]);
  }
  zero<NT, R>(acc);
}

// After the CTA's last slab: count arrivals on the (at most two) partial row
// blocks of this CTA; the last CTA to arrive on one adds the partials of all
// its contributors in K order and writes Y, then re-arms the counter.
template <int NT, int R, int kRowsCta, int kRowsWarp>
__device__ __forceinline__ void settle_partials(const DecodeParams& p, const RunGeom& geo, int64_t rb_first,
                                                int64_t rb_last, int warp, int lane, int* s_last) {
  constexpr int kSlot = kWarps * R * NT * 32 * 4;
  const int tid = warp * 32 + lane;
  const bool pf = geo.partial(p, rb_first), pl = rb_last != rb_first && geo.partial(p, rb_last);
  if (!pf && !pl) return;
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    int last = 0;
    if (pf)
      last |= (atomicAdd(p.counters + rb_first, 1) == (int)(geo.last_cta(p, rb_first) - geo.first_cta(p, rb_first)));
    if (pl)
      last |= (atomicAdd(p.counters + rb_last, 1) == (int)(geo.last_cta(p, rb_last) - geo.first_cta(p, rb_last)))
              << 1;
    *s_last = last;
  }
  __syncthreads();
  const int last = *s_last;
  if (!last) return;
  __threadfence();
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {
    if (!(last & (1 << which))) continue;
    const int64_t rbg = which == 0 ? rb_first : rb_last;
    const int j = entry_of_rb(p, rbg);
    const int64_t cf = geo.first_cta(p, rbg), cl = geo.last_cta(p, rbg);
    float acc[R][NT][4];
    zero<NT, R>(acc);
    // Per accumulator tile, the loads of up to four contributors are issued
    // together and added in K order, so the sum does not depend on which CTA
    // arrived last.
    for (int64_t c0 = cf; c0 <= cl; c0 += 4) {
      const float4* sl[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t cc = c0 + q <= cl ? c0 + q : cl;
        sl[q] = reinterpret_cast<const float4*>(p.partials + geo.slot(p, cc, rbg) * (int64_t)kSlot);
      }
      const int nq = (int)(cl - c0 + 1 < 4 ? cl - c0 + 1 : 4);
#pragma unroll
      for (int rt = 0; rt < R; ++rt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int idx = ((warp * R + rt) * NT + nt) * 32 + lane;
          float4 v[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) v[q] = __ldcg(sl[q] + idx);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (q < nq) {
              acc[rt][nt][0] += v[q].x;
              acc[rt][nt][1] += v[q].y;
              acc[rt][nt][2] += v[q].z;
              acc[rt][nt][3] += v[q].w;
            }
        }
    }
    write_y<NT, R>(acc, p.e[j], p.m, (rbg - p.e[j].rb_begin) * kRowsCta + warp * kRowsWarp, lane >> 2, lane & 3);
    if (tid == 0) p.counters[rbg] = 0;
  }
}

// ---- the kernel ---------------------------------------------------------------
// FUSED = false: weight slabs come from the views by TMA (thread 0 issues).
// FUSED = true:  every thread copies 16-byte pieces straight from the chunks
//                with cp.async into the same swizzled layout.
// WT: 0 e4m3 codes with block scales; 1 bf16, 2 f16 weights (no scales).
template <int NT, int R, int S, bool FUSED, int WT>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int kRowsWarp = 16 * R;
  constexpr int kRowsCta = kWarps * kRowsWarp;
  constexpr int kStage = kRowsCta * kSlabK;  // bytes of one staged weight slab
  constexpr int kBoxRows = kRowsCta > 256 ? 256 : kRowsCta;
  constexpr int kBoxes = kRowsCta / kBoxRows;
  using XS = XStage<NT, WT>;
  constexpr bool WB = WT != 0;
  constexpr int kElem = WB ? 2 : 1;  // bytes per weight

  extern __shared__ uint8_t dsm[];
  __shared__ __align__(16) uint4 xs[2][XS::kUnits];
  __shared__ __align__(8) uint64_t full[S];
  __shared__ int s_last;
  // 128-byte swizzled TMA tiles need a 1024-byte aligned destination.
  uint8_t* wst = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tig = lane & 3;
  const int64_t U = p.units, G = gridDim.x, c = blockIdx.x;
  const int64_t u0 = c * U / G, u1 = (c + 1) * U / G, n = u1 - u0;
  if (tid == 0) {
    dev::trace_start(p.trace);
    if (!FUSED) {
      for (int s = 0; s < S; ++s) dev::mbar_init(&full[s], 1);
      dev::fence_mbar_init();
    }
  }
  __syncthreads();

  // Stage slab i (unit u0 + i) into ring slot i % S.
  auto issue = [&](int64_t i) {
    const UnitPos up = unit_pos(p, u0 + i);
    const DecodeEntry& e = p.e[up.j];
    uint8_t* dst = wst + (int)(i % S) * kStage;
    if (!FUSED) {
      uint64_t* bar = &full[(int)(i % S)];
      dev::mbar_arrive_expect_tx(bar, kStage);
#pragma unroll
      for (int b = 0; b < kBoxes; ++b)
        tma_load_2d(dst + b * kBoxRows * kSlabK, &e.tmap, (int32_t)(up.kb * kSlabK),
                    (int32_t)(up.rbl * kRowsCta + b * kBoxRows), bar);
    } else {
      // thread -> 16-byte column piece cu of rows rr, rr + 32, ...; byte
      // g = t_offset + o * cols + k of T lives in chunk g / C at g % C.
      const int cu = tid & 7;
      const int64_t rowb = e.cols * kElem;  // bytes per weight row
      const int64_t k = up.kb * kSlabK + 16 * cu;
      const int64_t C = p.chunk_bytes;
      int64_t gb = e.t_offset + (up.rbl * kRowsCta + (tid >> 3)) * rowb + k;
      int64_t ci = gb / C, off = gb - ci * C;
      const int64_t step = 32 * rowb;
#pragma unroll 4
      for (int jr = 0; jr < kRowsCta / 32; ++jr) {
        const int rr = (tid >> 3) + 32 * jr;
        const int64_t o = up.rbl * kRowsCta + rr;
        const bool valid = o < e.rows && k < rowb;
        const uint8_t* src = p.chunks[valid ? ci : 0] + (valid ? off : 0);
        dev::cp_async16(dst + rr * kSlabK + ((cu ^ (rr & 7)) << 4), src, valid ? 16u : 0u);
        off += step;
        while (off >= C) {
          off -= C;
          ++ci;
        }
      }
      dev::cp_async_commit();
    }
  };

  if (FUSED) {
    for (int64_t i = 0; i < S - 1; ++i) {
      if (i < n) issue(i); else dev::cp_async_commit();
    }
  } else if (tid == 0) {
    for (int64_t i = 0; i < n && i < S - 1; ++i) issue(i);
  }

  // Activations are fetched two slabs ahead (register sets xa / xb take turns,
  // the loop is unrolled by two so they stay in registers), and block scales
  // 32 slabs at a time, one per lane, a block ahead, so no global-load latency
  // sits on the per-slab path.
  XS xa, xb;
  auto stage_x = [&](XS& dst, int64_t i) {
    const UnitPos up = unit_pos(p, u0 + i);
    dst.load(p.e[up.j], p.m, up.kb, tid);
  };
  auto scale_of = [&](int64_t i) -> float {
    if (i >= n) return 0.f;
    const UnitPos up = unit_pos(p, u0 + i);
    const DecodeEntry& e = p.e[up.j];
    const int64_t row0 = up.rbl * kRowsCta + warp * kRowsWarp;
    if (WB) return row0 < e.rows ? 1.f : 0.f;
    return row0 < e.rows ? __ldg(e.scales + (row0 >> 7) * e.scale_cols + up.kb) : 0.f;
  };
  float sc_cur = scale_of(lane), sc_next = scale_of(32 + lane);
  if (n > 0) {
    stage_x(xa, 0);
    xa.store(xs[0], tid);
  }
  if (n > 1) stage_x(xb, 1);
  float acc[R][NT][4];
  zero<NT, R>(acc);
  float cs = 0.f;  // scale the accumulator currently refers to
  const RunGeom geo{G, U, c};
  bool timed_out = false;

  // One slab: `nx` receives slab i + 2 (it held slab i, already staged);
  // `cx` holds slab i + 1, staged at the end.
  auto slab = [&](int64_t i, XS& nx, XS& cx) {
    const int st = (int)(i % S);
    bool ok = true;
    if (FUSED) dev::cp_async_wait<S - 2>();
    else ok = dev::mbar_wait(&full[st], (uint32_t)((i / S) & 1), kWaitLimitNs);
    // Slab i has landed for everyone; slab i-1's stage and X buffer are free.
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        dev::set_status(p.status, SWS_E_TIMEOUT);
        for (int64_t jj = i; jj < n && jj < i + S - 1; ++jj)  // drain copies still in flight (bounded)
          dev::mbar_wait(&full[(int)(jj % S)], (uint32_t)((jj / S) & 1), kWaitLimitNs / 4);
      }
      timed_out = true;
      return;
    }
    if (FUSED) {
      if (i + S - 1 < n) issue(i + S - 1); else dev::cp_async_commit();
    } else if (tid == 0 && i + S - 1 < n) {
      issue(i + S - 1);
    }
    if (i + 2 < n) stage_x(nx, i + 2);
    if ((i & 31) == 0 && i > 0) {
      sc_cur = sc_next;
      sc_next = scale_of(i + 32 + lane);
    }
    const float s = __shfl_sync(0xffffffffu, sc_cur, (int)(i & 31));
    const UnitPos up = unit_pos(p, u0 + i);
    const int64_t row0 = up.rbl * kRowsCta + warp * kRowsWarp;
    if (i == 0 || up.kb == 0) cs = 0.f;
    if (apply_scale<NT, R>(acc, cs, s)) {
      const uint8_t* wb = wst + st * kStage;
#pragma unroll
      for (int l = 0; l < 2; ++l) {
        uint4 wq[R][2];
#pragma unroll
        for (int rt = 0; rt < R; ++rt)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int r = warp * kRowsWarp + rt * 16 + g + 8 * h;
            wq[rt][h] = *reinterpret_cast<const uint4*>(wb + r * kSlabK + (((2 * tig + l) ^ g) << 4));
          }
        mma_half<NT, R, WT>(acc, wq, xs[i & 1], l, g, tig);
      }
    }
    if (i + 1 < n) cx.store(xs[(i + 1) & 1], tid);
    if (i + 1 == n || up.kb + 1 == p.e[up.j].slabs) {
      rescale<NT, R>(acc, cs);
      end_run<NT, R>(acc, p, geo, up, row0, warp, lane);
    }
  };
  for (int64_t i = 0; i < n && !timed_out; i += 2) {
    slab(i, xa, xb);
    if (i + 1 < n && !timed_out) slab(i + 1, xb, xa);
  }
  if (!timed_out && n > 0)
    settle_partials<NT, R, kRowsCta, kRowsWarp>(p, geo, unit_pos(p, u0).rbg, unit_pos(p, u1 - 1).rbg, warp, lane,
                                                &s_last);
  if (FUSED) dev::cp_async_wait<0>();
  if (p.trace && tid == 0) {  // the record's end stamp after this kernel's writes
    __threadfence();
    dev::trace_end(p.trace, p.tag);
  }
}

template <int NT>
constexpr int rows_per_warp_tiles() { return NT <= 2 ? 4 : 2; }
// Ring depth: 192 KB of weight stages, leaving room for the staged activations.
template <int NT>
constexpr int stages_for() { return NT <= 2 ? 3 : NT == 4 ? 6 : 5; }

int nt_for(int64_t m) { return m <= 8 ? 1 : m <= 16 ? 2 : m <= 32 ? 4 : 8; }
int rows_per_cta(int nt) { return kWarps * 16 * (nt <= 2 ? 4 : 2); }
constexpr int64_t slot_bytes_for(int nt) { return (int64_t)kWarps * (nt <= 2 ? 4 : 2) * nt * 32 * 4 * 4; }

template <int NT, bool FUSED, int WT>
cudaError_t launch_nt(const DecodeParams& p, int64_t grid_cap, cudaStream_t s) {
  constexpr int R = rows_per_warp_tiles<NT>();
  constexpr int S = stages_for<NT>();
  constexpr int kRowsCta = kWarps * 16 * R;
  constexpr int kSmem = S * kRowsCta * kSlabK + 1024;
  auto kern = decode_kernel<NT, R, S, FUSED, WT>;
  static PerDevice once;
  const cudaError_t attr =
      once.run([&] { return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem); });
  if (attr != cudaSuccess) return attr;
  const int64_t grid = std::min<int64_t>({p.units, (int64_t)device_sm_count(), (int64_t)kMaxGrid, grid_cap});
  return launch_high(kern, dim3((unsigned)grid), dim3(kThreads), kSmem, s, p);
}

template <int WT>
cudaError_t dispatch_w(const DecodeParams& p, int nt, bool fused, int64_t grid_cap, cudaStream_t s) {
  switch (nt) {
    case 1: return fused ? launch_nt<1, true, WT>(p, grid_cap, s) : launch_nt<1, false, WT>(p, grid_cap, s);
    case 2: return fused ? launch_nt<2, true, WT>(p, grid_cap, s) : launch_nt<2, false, WT>(p, grid_cap, s);
    case 4: return fused ? launch_nt<4, true, WT>(p, grid_cap, s) : launch_nt<4, false, WT>(p, grid_cap, s);
    default: return fused ? launch_nt<8, true, WT>(p, grid_cap, s) : launch_nt<8, false, WT>(p, grid_cap, s);
  }
}
cudaError_t dispatch(const DecodeParams& p, int nt, bool fused, int wtype, int64_t grid_cap, cudaStream_t s) {
  switch (wtype) {
    case 1: return dispatch_w<1>(p, nt, fused, grid_cap, s);
    case 2: return dispatch_w<2>(p, nt, fused, grid_cap, s);
    default: return dispatch_w<0>(p, nt, fused, grid_cap, s);
  }
}

// Validates a group and fills the kernel parameters, except the scratch
// pointers. *empty is set when nothing is left to launch (every item has no
// rows or no columns; outputs of zero-column items are zeroed on `s`).
int build_params(DecodeParams& p, const DecodeGroup& g, int64_t* row_blocks, bool* empty, cudaStream_t s,
                 uint8_t* tc_split = nullptr) {
  const bool tc = tc_split != nullptr;
  *empty = true;
  if (g.n < 1 || g.n > kMaxDecodeGroup) return fail(SWS_E_INVALID, "decode: group of %d linears", g.n);
  if (g.m < 0 || g.m > 64) return fail(SWS_E_INVALID, "decode: m=%lld outside [0, 64]", (long long)g.m);
  const int nt = nt_for(std::max<int64_t>(g.m, 1));
  const int rows_cta = tc ? kTcUnitRows : rows_per_cta(nt);
  p.n_entries = 0;
  p.m = (int32_t)g.m;
  p.units = 0;
  for (int i = 0; i < 256; ++i) p.chunks[i] = i < g.n_chunks ? g.chunks[i] : nullptr;
  p.chunk_bytes = g.chunk_bytes > 0 ? g.chunk_bytes : 1;
  int64_t rb = 0;
  for (int i = 0; i < g.n; ++i) {
    const DecodeItem& it = g.item[i];
    if (it.cols % 16 != 0)
      return fail(SWS_E_UNSUPPORTED, "decode: cols=%lld is not a multiple of 16", (long long)it.cols);
    if (g.m == 0 || it.rows == 0) continue;
    if (it.cols == 0) {
      cudaError_t e = cudaMemsetAsync(it.y, 0, (size_t)(g.m * it.rows * 2), s);
      if (e != cudaSuccess) return cuda_fail(e, "decode: cudaMemsetAsync");
      continue;
    }
    DecodeEntry& e = p.e[p.n_entries++];
    const int64_t elem = (g.wtype != 0 ? 2 : 1);
    if (!g.fused) {  // the weight as bytes: one 128-byte slab row is 128 e4m3 or 64 bf16 weights
      int rc = encode_u8_tile_map(&e.tmap, it.w, it.rows, it.cols * elem, std::min(256, rows_cta));
      if (rc != SWS_OK) return rc;
    }
    e.xs = nullptr;
    if (tc) {  // the entry's activation blocks, one per K slab: (hi, lo, e) for e4m3 weights, x for bf16
      e.xs = tc_split;
      tc_split += cdiv(it.cols * elem, kSlabK) * tc_x_block_bytes(tc_n_pad(g.m), g.wtype != 0);
    }
    e.scales = it.scales;
    e.x = it.x;
    e.y = it.y;
    e.rows = it.rows;
    e.row_base = 0;
    e.y_rows = it.rows;
    e.linear = i;
    e.split_owner = 1;
    e.cols = it.cols;
    e.t_offset = it.t_offset;
    e.scale_cols = cdiv(it.cols, 128);
    e.slabs = (int32_t)cdiv(it.cols * elem, kSlabK);
    e.unit_begin = p.units;
    e.rb_begin = rb;
    const int64_t nrb = cdiv(it.rows, rows_cta);
    rb += nrb;
    p.units += nrb * e.slabs;
  }
  if (rb > kMaxCounters) return fail(SWS_E_UNSUPPORTED, "decode: %lld row blocks in one launch", (long long)rb);
  if (p.units >= ((int64_t)1 << 31)) return fail(SWS_E_UNSUPPORTED, "decode: group too large");
  *row_blocks = rb;
  *empty = p.n_entries == 0;
  return SWS_OK;
}

}  // namespace

namespace {
std::atomic<int> g_decode_kernel{kDecodeAuto};  // SWS_OPT_DECODE_KERNEL
}

void set_decode_kernel(int k) { g_decode_kernel.store(k, std::memory_order_relaxed); }

// The tcgen05 kernel streams the weights at the HBM rate for every m <= 64
// (its MMAs and activation split are small next to the weight bytes); the
// mma.sync kernel serves chunk-map launches beyond the tcgen05 segment tables
// and can be selected for comparison.
int decode_kernel_for(int64_t m) {
  const int k = g_decode_kernel.load(std::memory_order_relaxed);
  if (k != kDecodeAuto) return k;
  (void)m;
  return kDecodeTc;
}

int64_t decode_split_bytes(int64_t m, int64_t slabs) {
  return slabs * tc_split_block_bytes(tc_n_pad(std::max<int64_t>(m, 1)));
}

int decode_workspace_bytes(int64_t m, int64_t* bytes) {
  if (m < 0 || m > 64) return fail(SWS_E_INVALID, "decode: m=%lld outside [0, 64]", (long long)m);
  const int64_t mm = std::max<int64_t>(m, 1);
  const int64_t slot = std::max<int64_t>(slot_bytes_for(nt_for(mm)), tc_slot_bytes(mm));
  *bytes = kCtlBytes + kMaxCounters * 4 + 2 * (int64_t)kMaxGrid * slot;
  return SWS_OK;
}

// Chunk-map (fused) launch on the tcgen05 path. Each linear becomes one entry
// per chunk it has whole rows in (a segment: rows rf..rl, a tensor map over
// that chunk's bytes), so no unit reads across a chunk boundary; the rows a
// boundary splits are listed for the settle kernel. `lin` holds the group's
// linears as build_params made them (with their split blocks); *ok stays false
// when the segments or split rows exceed the tables (the mma.sync kernel then
// serves the launch).
int build_fused_segments(DecodeParams& p, const DecodeParams& lin, const DecodeGroup& g, bool* ok) {
  *ok = false;
  p = lin;
  p.n_entries = 0;
  p.units = 0;
  p.st.n = 0;
  const int64_t C = g.chunk_bytes;
  int64_t rb = 0;
  for (int j = 0; j < lin.n_entries; ++j) {
    const DecodeEntry& L = lin.e[j];
    // byte arithmetic: `cols` here is the row length in bytes
    const int64_t o = L.t_offset, cols = L.cols * ((g.wtype != 0 ? 2 : 1)), rows = L.rows, end = o + rows * cols;
    const int64_t c0 = o / C, c1 = (end - 1) / C;
    bool owner = true;
    for (int64_t c = c0; c <= c1; ++c) {
      const int64_t lo = c * C, hi = lo + C;
      if (c > c0 && (lo - o) % cols != 0) {  // the boundary at lo splits row (lo - o) / cols
        if (p.st.n >= kMaxStraddle) return SWS_OK;
        p.st.row[p.st.n] = (lo - o) / cols;
        p.st.entry[p.st.n] = -1 - j;  // resolved to a segment of linear j below
        ++p.st.n;
      }
      const int64_t rf = lo <= o ? 0 : (lo - o + cols - 1) / cols;
      const int64_t rl = std::min<int64_t>(rows, (hi - o) / cols) - 1;
      if (rf > rl) continue;
      if (p.n_entries >= kMaxDecodeEntries) return SWS_OK;
      if (c >= g.n_chunks || !g.chunks[c]) return fail(SWS_E_INVALID, "decode: chunk %lld is missing", (long long)c);
      DecodeEntry& e = p.e[p.n_entries];
      e = L;
      int rc = encode_u8_tile_map(&e.tmap, g.chunks[c] + (o + rf * cols - lo), rl - rf + 1, cols, kTcUnitRows);
      if (rc != SWS_OK) return rc;
      e.rows = rl - rf + 1;
      e.row_base = rf;
      e.y_rows = rows;
      e.linear = j;
      e.split_owner = owner ? 1 : 0;
      owner = false;
      e.unit_begin = p.units;
      e.rb_begin = rb;
      const int64_t nrb = cdiv(e.rows, kTcUnitRows);
      rb += nrb;
      p.units += nrb * e.slabs;
      ++p.n_entries;
    }
    if (owner) return SWS_OK;  // no whole row of this linear in any chunk
  }
  for (int k = 0; k < p.st.n; ++k) {  // any segment of the linear gives the straddling row's pointers
    const int j = -1 - p.st.entry[k];
    for (int q = 0; q < p.n_entries; ++q)
      if (p.e[q].linear == j) {
        p.st.entry[k] = q;
        break;
      }
  }
  if (rb > kMaxCounters || p.units >= ((int64_t)1 << 31)) return SWS_OK;
  *ok = true;
  return SWS_OK;
}

int launch_decode(const DecodeGroup& g, cudaStream_t s) {
  if (g.m == 0) return SWS_OK;
  int64_t dec = 0;
  int rc = decode_workspace_bytes(g.m, &dec);
  if (rc != SWS_OK) return rc;
  int64_t split = 0;  // the activation split region follows the partial sums
  for (int i = 0; i < g.n; ++i)
    split += cdiv(g.item[i].cols * ((g.wtype != 0 ? 2 : 1)), kSlabK) * tc_x_block_bytes(tc_n_pad(std::max<int64_t>(g.m, 1)), g.wtype != 0);
  bool tc = decode_kernel_for(g.m) == kDecodeTc;
  const int64_t need = dec + (tc ? split : 0);
  if (g.workspace_bytes < need)
    return fail(SWS_E_WORKSPACE, "decode: workspace %lld < %lld bytes", (long long)g.workspace_bytes, (long long)need);
  DecodeParams p;
  int64_t row_blocks = 0;
  bool empty = true;
  rc = build_params(p, g, &row_blocks, &empty, s, tc ? g.workspace + dec : nullptr);
  if (rc != SWS_OK || empty) return rc;
  if (tc && g.fused) {
    DecodeParams lin = p;
    bool ok = false;
    rc = build_fused_segments(p, lin, g, &ok);
    if (rc != SWS_OK) return rc;
    if (!ok) {  // beyond the chunk-map tables: the mma.sync kernel reads this group
      tc = false;
      rc = build_params(p, g, &row_blocks, &empty, s, nullptr);
      if (rc != SWS_OK || empty) return rc;
    }
  }
  p.counters = reinterpret_cast<int32_t*>(g.workspace + kCtlBytes);
  p.partials = reinterpret_cast<float*>(g.workspace + kCtlBytes + kMaxCounters * 4);
  p.status = reinterpret_cast<int32_t*>(g.workspace);
  p.trace = g.trace;
  p.tag = g.tag | ((tc ? (g.fused ? kTraceTcFused : kTraceTc) : (g.fused ? kTraceMmaFused : kTraceMma)) << 48);
  cudaError_t e =
      tc ? launch_decode_tc(p, g.fused, g.wtype, kMaxGrid, s) : dispatch(p, nt_for(g.m), g.fused, g.wtype, kMaxGrid, s);
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
// split-K partial sums, the per-row-block arrival counters and a status word)
// in a fixed array that lives in the library's device image, so a call needs
// only the caller's inputs and outputs.
//
// The array is shared by every call on a device and keeps the last call's
// contents; the arrival counters are cleared on the stream before each launch.
// Two calls whose work overlaps on the GPU race on the array.
// ---------------------------------------------------------------------------
namespace sws {
namespace {

// fp32 partial sums: two slots of the largest size (m > 32) for each of up to
// kMaxGrid CTAs, so the grid is never narrowed to fit the array.
constexpr int64_t kNoAllocPartialBytes = 2 * (int64_t)kMaxGrid * slot_bytes_for(8);  // 32 MiB
static_assert(kNoAllocPartialBytes == (int64_t(32) << 20), "noalloc partial-sum region");
constexpr int64_t kNoAllocCounters = 4096;  // row blocks, one int32 each
constexpr int64_t kNoAllocStatusOffset = kNoAllocPartialBytes + kNoAllocCounters * 4;
// [partial sums | counters | status word (int32) and padding]
constexpr int64_t kNoAllocScratchBytes = kNoAllocStatusOffset + 256;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device. The first use on
// a device resolves it with cudaGetSymbolAddress (with that device current) and
// clears the status word on `s`; later uses reuse the cached address.
int noalloc_scratch(uint8_t** out, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "linear_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(SWS_E_UNSUPPORTED, "linear_noalloc: device %d", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "linear_noalloc: cudaGetSymbolAddress(scratch)");
    e = cudaMemsetAsync(static_cast<uint8_t*>(p) + kNoAllocStatusOffset, 0, 4, s);
    if (e != cudaSuccess) return cuda_fail(e, "linear_noalloc: cudaMemsetAsync(status)");
    g_noalloc_addr[dev] = p;
  }
  *out = static_cast<uint8_t*>(g_noalloc_addr[dev]);
  return SWS_OK;
}

}  // namespace

int noalloc_status_word(int32_t** out, cudaStream_t s) {
  uint8_t* scratch = nullptr;
  const int rc = noalloc_scratch(&scratch, s);
  if (rc != SWS_OK) return rc;
  *out = reinterpret_cast<int32_t*>(scratch + kNoAllocStatusOffset);
  return SWS_OK;
}

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
  DecodeGroup g;
  g.n = 1;
  g.m = m;
  g.fused = false;
  g.item[0] = DecodeItem{static_cast<const uint8_t*>(w), scales, static_cast<const uint16_t*>(x),
                         static_cast<uint16_t*>(y), rows, cols, 0};
  DecodeParams p;
  int64_t nrb = 0;
  bool empty = true;
  rc = build_params(p, g, &nrb, &empty, s);
  if (rc != SWS_OK || empty) return rc;
  uint8_t* scratch = nullptr;
  rc = noalloc_scratch(&scratch, s);
  if (rc != SWS_OK) return rc;
  int32_t* counters = reinterpret_cast<int32_t*>(scratch + kNoAllocPartialBytes);
  cudaError_t e = cudaMemsetAsync(counters, 0, (size_t)(nrb * 4), s);
  if (e != cudaSuccess) return cuda_fail(e, "linear_noalloc: cudaMemsetAsync(counters)");
  p.counters = counters;
  p.partials = reinterpret_cast<float*>(scratch);
  // A wait that runs out records SWS_E_TIMEOUT here (read by sws_noalloc_status).
  p.status = reinterpret_cast<int32_t*>(scratch + kNoAllocStatusOffset);
  p.trace = nullptr;
  p.tag = 0;
  // Two partial slots per CTA fit in the fixed array for every grid up to kMaxGrid.
  const int64_t grid_cap = kNoAllocPartialBytes / (2 * slot_bytes_for(nt));
  e = dispatch(p, nt, false, 0, grid_cap, s);
  return e == cudaSuccess ? SWS_OK : cuda_fail(e, "linear_noalloc: kernel launch");
}

extern "C" int sws_noalloc_status(int32_t clear, int32_t* status) {
  using namespace sws;
  if (!status) return fail(SWS_E_INVALID, "noalloc_status: status is NULL");
  *status = 0;
  int32_t* word = nullptr;
  int rc = noalloc_status_word(&word, nullptr);
  if (rc != SWS_OK) return rc;
  int dev = 0;
  SWS_CUDA_TRY(cudaGetDevice(&dev));
  rc = device_sync_deadline(dev, "noalloc_status");
  if (rc != SWS_OK) return rc;
  int32_t v = 0;
  SWS_CUDA_TRY(cudaMemcpy(&v, word, sizeof v, cudaMemcpyDeviceToHost));
  if (clear) {
    SWS_CUDA_TRY(cudaMemset(word, 0, sizeof v));
    SWS_CUDA_TRY(cudaStreamSynchronize(nullptr));  // cleared before any later launch
  }
  *status = v;
  return SWS_OK;
}
