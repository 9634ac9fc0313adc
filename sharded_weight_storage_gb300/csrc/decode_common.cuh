// Shared pieces of the decode linears (m <= 64): launch parameters of a group
// of linears, the (row block, K slab) unit space of the split-K partition, and
// small conversion / copy helpers. Included by decode_gemm.cu (mma.sync
// kernel) and decode_tc.cu (tcgen05 kernel).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"
#include "sws_internal.h"

namespace sws {
namespace dec {

constexpr int kSlabK = 128;
constexpr int kMaxGrid = 256;  // upper bound used to size the workspace

// One linear of a group, or (tcgen05 chunk-map launches) one segment of a
// linear: the rows of the linear that lie whole inside one chunk.
struct DecodeEntry {
  CUtensorMap tmap;   // 2-D map of the weight rows [rows, cols] u8 (slot view, or the segment in its chunk)
  const float* scales;
  const uint16_t* x;  // bf16 [m, cols]
  uint16_t* y;        // bf16 [m, rows]
  int64_t rows, cols;  // rows of this entry / segment
  int64_t row_base;    // first row of the linear this entry covers (segments), else 0
  int64_t y_rows;      // rows of the linear: the row stride of y (and of the scale rows)
  int32_t linear;      // which linear of the group
  int32_t split_owner; // 1 for the entry that splits the linear's activations
  uint8_t* xs;         // tcgen05 path: the linear's activation split blocks (one per K slab)
  int64_t t_offset;    // fused path: o_j, the entry's offset in T
  int64_t scale_cols;  // ceil(cols / 128)
  int64_t unit_begin;  // first unit of this entry in the group's unit space
  int64_t rb_begin;    // first row block of this entry in the group
  int32_t slabs;       // ceil(cols / 128)
};

// Chunk-map (fused) reads on the tcgen05 path: every entry is a segment (the
// rows of a linear that lie whole inside one chunk, with a tensor map over that
// chunk), so no unit reads across a chunk boundary. A row that a boundary
// splits (a "straddling" row) belongs to no segment: the settle kernel
// computes that row of Y directly.
constexpr int kMaxDecodeEntries = 40;
constexpr int kMaxStraddle = 32;
struct Straddles {
  int32_t n;
  int32_t entry[kMaxStraddle];  // an entry (segment) of the linear, for its pointers
  int64_t row[kMaxStraddle];    // the row within the linear
};

struct DecodeParams {
  DecodeEntry e[kMaxDecodeEntries];
  int32_t n_entries;
  int32_t m;
  int64_t units;  // total units (row block x K slab) of the group
  const uint8_t* chunks[256];  // fused path: the layer's chunks
  int64_t chunk_bytes;
  Straddles st;   // tcgen05 chunk-map launches only
  int32_t* counters;
  float* partials;
  int32_t* status;
  uint64_t* trace;
  uint64_t tag;
};

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)two_bytes));
  return r;
}

// bf16 pair -> f16 pair: exact for |x| in [2^-24, 65504]; larger magnitudes
// saturate to +-65504, smaller ones round to the f16 subnormal grid.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  const float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xffff0000u);
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(dev::smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(dev::smem_addr(bar))
      : "memory");
}

// Same, with an L2 cache policy (from createpolicy) for the loaded lines.
__device__ __forceinline__ void tma_load_2d_hint(void* smem_dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                 uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dev::smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(dev::smem_addr(bar)), "l"(policy)
      : "memory");
}

// L2 policy for data read once (a streamed weight): evict first, so the small
// data that is read again (activations, scales, partial sums) stays in L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Which CTA's unit range [c*U/G, (c+1)*U/G) contains unit u.
__device__ __forceinline__ int64_t cta_of(int64_t u, int64_t G, int64_t U) { return ((u + 1) * G - 1) / U; }

// Where a unit of the group's unit space lies.
struct UnitPos {
  int j;        // entry
  int64_t rbl;  // row block inside the entry
  int64_t kb;   // K slab
  int64_t rbg;  // row block in the group
};

__device__ __forceinline__ int entry_of_unit(const DecodeParams& p, int64_t u) {
  int j = 0;
  for (int q = 1; q < p.n_entries && u >= p.e[q].unit_begin; ++q) j = q;
  return j;
}

__device__ __forceinline__ int entry_of_rb(const DecodeParams& p, int64_t rbg) {
  int j = 0;
  for (int q = 1; q < p.n_entries && rbg >= p.e[q].rb_begin; ++q) j = q;
  return j;
}

__device__ __forceinline__ UnitPos unit_pos(const DecodeParams& p, int64_t u) {
  UnitPos r;
  r.j = entry_of_unit(p, u);
  const DecodeEntry& e = p.e[r.j];
  const uint32_t local = (uint32_t)(u - e.unit_begin);  // units per entry < 2^31
  const uint32_t rbl = local / (uint32_t)e.slabs;
  r.rbl = rbl;
  r.kb = local - rbl * (uint32_t)e.slabs;
  r.rbg = e.rb_begin + r.rbl;
  return r;
}

// Row-block bookkeeping of the split-K partition (all in group row blocks).
struct RunGeom {
  int64_t G, U, c;
  __device__ __forceinline__ int64_t first_unit(const DecodeParams& p, int64_t rbg) const {
    const DecodeEntry& e = p.e[entry_of_rb(p, rbg)];
    return e.unit_begin + (rbg - e.rb_begin) * e.slabs;
  }
  __device__ __forceinline__ int64_t first_cta(const DecodeParams& p, int64_t rbg) const {
    return cta_of(first_unit(p, rbg), G, U);
  }
  __device__ __forceinline__ int64_t last_cta(const DecodeParams& p, int64_t rbg) const {
    const DecodeEntry& e = p.e[entry_of_rb(p, rbg)];
    return cta_of(first_unit(p, rbg) + e.slabs - 1, G, U);
  }
  __device__ __forceinline__ bool partial(const DecodeParams& p, int64_t rbg) const {
    return first_cta(p, rbg) != last_cta(p, rbg);
  }
  // Partial slot of CTA cc for row block rbg: 0 for its first run, 1 otherwise.
  __device__ __forceinline__ int64_t slot(const DecodeParams& p, int64_t cc, int64_t rbg) const {
    return 2 * cc + (rbg == unit_pos(p, cc * U / G).rbg ? 0 : 1);
  }
};

// tcgen05 decode kernel (decode_tc.cu): units of 256 weight rows. A launch
// first splits the activations into per-slab blocks (xs of every entry), then
// runs the GEMM on them; the params must have been built with that unit height.
constexpr int kTcUnitRows = 256;
__host__ __device__ constexpr int64_t tc_n_pad(int64_t m) { return (m + 15) / 16 * 16; }
// Split block of one entry and K slab for n_pad = m rounded up to 16:
// [hi e4m3 n_pad x 128 | lo e4m3 n_pad x 128 | e fp32 n_pad].
__host__ __device__ constexpr int64_t tc_split_block_bytes(int64_t n_pad) { return 260 * n_pad; }
// Activation block of one entry and 128-byte weight slab: the split block for
// e4m3 weights, the 16-bit activations [n_pad][64] (128 bytes a row) for bf16
// or f16 weights.
__host__ __device__ constexpr int64_t tc_x_block_bytes(int64_t n_pad, bool w16) {
  return w16 ? 128 * n_pad : tc_split_block_bytes(n_pad);
}
// wtype: 0 e4m3 weights with block scales, 1 bf16 weights, 2 f16 weights.
cudaError_t launch_decode_tc(const DecodeParams& p, bool fused, int wtype, int64_t grid_cap, cudaStream_t s);
int64_t tc_slot_bytes(int64_t m);

}  // namespace dec
}  // namespace sws
