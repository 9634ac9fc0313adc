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
// Two kernels compute it; both are persistent and warp-specialised: one
// thread loads operand tiles with TMA, one thread issues the MMAs into TMEM
// slab buffers (one buffer per 128-K slab), and promotion warps turn each slab
// into fp32 register sums. The weight scales are not powers of two, so they
// cannot feed the MMA's own block scaling: each slab result is read from TMEM
// (tcgen05.ld) and added with the factor ex[m, kb] * s_w[n/128, kb] (each
// promotion thread owns one row m and a run of columns). After the last slab
// of a tile the rows are rounded to bf16 and stored. The factors reach the
// promotion threads through a shared-memory ring filled by cp.async eight
// slabs ahead.
//
// prefill_kernel: one CTA per 128 x 256 tile (128 activation rows, 256 weight
// rows); 4 stages of 48 KB; 4 x tcgen05.mma kind::f8f6f4 (128 x 256 x 32)
// per slab into one of two 256-column buffers; 8 promotion warps x 128
// columns.
//
// prefill_pair_kernel (selected by option; slower here, see below): a cluster
// of two CTAs on an SM pair per 256 x 256 tile, with tcgen05 .cta_group::2.
// Each CTA loads 128 activation rows and 128 weight rows per slab (32 KB)
// into one of 6 stages; the pair's MMA (256 x 256 x 32) reads each CTA's
// activation half and both weight halves, so an SM takes in 32 KB from L2
// per 128 x 256 x 128 slab of work instead of 48 KB. Both CTAs' copies
// complete on the first CTA's stage barrier; its MMA thread commits to the
// empty and slab barriers of both CTAs (multicast); each CTA's 16 promotion
// warps (64 columns each) read their own TMEM lanes and release the buffer
// on the first CTA's barrier. With two slab buffers, every slab's MMA waits
// for the promotion of the slab two back in both CTAs, and that cross-SM
// round trip costs more than the L2 traffic saves: on the KDA-like linears
// it reaches about 41% of the FP8 peak where the one-CTA kernel reaches 47%.
//
// Every mbarrier wait is bounded; a wait that runs out records SWS_E_TIMEOUT
// and the CTA (or pair) finishes with TMEM released.
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

constexpr int kBK = 128;  // K per slab = one scale block

// One CTA per 128 x 256 tile: A = 128 activation rows, B = 256 weight rows,
// two TMEM slab buffers of 256 columns, 8 promotion warps x 128 columns.
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK;  // 16 KB
constexpr int kBBytes = kBN * kBK;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kEpiWarps = 8;
constexpr int kThreads = (2 + kEpiWarps) * 32;
// The FP8 kernel adds one warp that loads the scale factors.
constexpr int kFp8Threads = (3 + kEpiWarps) * 32;

// A CTA pair per 256 x 256 tile: each CTA loads 128 activation rows and 128
// weight rows per slab (32 KB); two TMEM slab buffers of 256 columns; 16
// promotion warps x 64 columns per CTA.
constexpr int kPairM = 256, kPairN = 256;
constexpr int kPairStages = 6;
constexpr int kPairABytes = (kPairM / 2) * kBK;         // 16 KB
constexpr int kPairBBytes = (kPairN / 2) * kBK;         // 16 KB
constexpr int kPairStageBytes = kPairABytes + kPairBBytes;
constexpr int kPairEpiWarps = 16;
constexpr int kPairThreads = (3 + kPairEpiWarps) * 32;  // with a scale warp

constexpr int kTmemCols = 512;

// Slabs of scale factors kept in flight ahead of the promotion warps, and the
// shared memory the one-CTA kernel sets aside for them (its output staging
// follows this space).
constexpr int kScaleDepth = 8;
__host__ __device__ constexpr int scale_ring_bytes(int epi_warps) { return kScaleDepth * (epi_warps * 32 + epi_warps) * 4; }
// Factor ring of the one-CTA FP8 kernel, filled by its scale warp: per slab
// (kScaleDepth of them in flight, across tiles) ex[m, kb] of the tile's 128
// rows and s_w[nb, kb] of its two 128-column blocks.
constexpr int kFactorSlot = kBM + 2;  // floats
constexpr int kFactorRingBytes = kScaleDepth * kFactorSlot * 4;
static_assert(kFactorRingBytes <= scale_ring_bytes(kEpiWarps), "factor ring fits the scale ring's space");
// Output staging of the one-CTA kernel: per promotion warp, 32 rows x 32 bf16
// columns (64 bytes a row) at a time.
constexpr int kOutChunk = 32;
constexpr int kOutWarpBytes = 32 * kOutChunk * 2;
constexpr int kSmemBytes = kStages * kStageBytes + scale_ring_bytes(kEpiWarps) + kEpiWarps * kOutWarpBytes + 1024;
constexpr int kPairSmemBytes = kPairStages * kPairStageBytes + kScaleDepth * (kBM + 2) * 4 + 1024;

struct PrefillParams {
  CUtensorMap tmap_x;  // xq [M, K] u8
  CUtensorMap tmap_w;  // wq [N, K] u8
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

// 32 lanes x 16 consecutive fp32 columns (thread = lane = row), without
// waiting (tmem_wait_ld).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// 32 lanes x 32 consecutive fp32 columns, without waiting (tmem_wait_ld).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(dev::smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(dev::smem_addr(bar))
      : "memory");
}

// ---- CTA-pair helpers ---------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Every thread of both CTAs arrives; memory before it is visible after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of `p` (a shared variable of this CTA) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(dev::smem_addr(p)), "r"(rank));
  return r;
}
// TMA tile load into this CTA's shared memory whose completion is counted on
// an mbarrier that may sit in the peer CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                 uint32_t cluster_bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dev::smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(cluster_bar)
      : "memory");
}
__device__ __forceinline__ void mma_f8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
// Arrives once on `bar` in both CTAs of the pair when the pair's previously
// issued MMAs finish.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  const uint16_t both = 0x3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          dev::smem_addr(bar)),
      "h"(both)
      : "memory");
}

__device__ __forceinline__ void set_abort(const PrefillParams& p, volatile int* s_abort) {
  dev::set_status(p.status, SWS_E_TIMEOUT);
  *s_abort = 1;
}

// a += f * v on two fp32 lanes at once (packed fma.rn.f32x2: each lane rounds
// exactly like fmaf), so the promotion issues half as many FMA instructions.
__device__ __forceinline__ void fma2(float& a0, float& a1, uint64_t ff, uint32_t v0, uint32_t v1) {
  uint64_t acc, vv;
  asm("mov.b64 %0, {%1, %2};" : "=l"(acc) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(vv) : "r"(v0), "r"(v1));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(ff), "l"(vv));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(acc));
}

// Row m, columns n0 .. n0+kCols-1 of Y as bf16 (round to nearest even).
template <int kCols>
__device__ __forceinline__ void store_row(const PrefillParams& p, const float (&acc)[kCols], int64_t m, int64_t n0) {
  if (m >= p.M || n0 >= p.N) return;
  uint16_t* yrow = p.y + m * p.N + n0;
  const int64_t ncols = p.N - n0 < kCols ? p.N - n0 : kCols;
  if (ncols == kCols && (p.N & 7) == 0) {
#pragma unroll
    for (int i = 0; i < kCols; i += 8) {
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
    for (int i = 0; i < kCols; ++i)
      if (i < ncols) {
        const __nv_bfloat16 b = __float2bfloat16_rn(acc[i]);
        yrow[i] = *reinterpret_cast<const uint16_t*>(&b);
      }
  }
}

// One promotion thread's share of a tile: TMEM lane `row` of the tile, kCols
// columns from `lane_base` within each slab buffer (two buffers, kBN columns
// apart, used in turn). For each K slab kb it waits for the slab buffer and
// for the slab's factors in the ring the scale warp fills (slot
// it % kScaleDepth: fslot_full says it is filled, fslot_empty takes one
// arrival per promotion warp once read), adds the buffer into acc scaled by
// ex[m, kb] * s_w[nb, kb], and releases the buffer once per warp. `g` is the
// warp's kCols-column group of the tile; release0 is the address of the first
// slab buffer's empty barrier (the second's follows it), this CTA's or, for a
// pair, the first CTA's through its cluster address. Returns false if a wait
// ran out.
template <int kCols, bool kPair = false>
__device__ __forceinline__ bool promote_tile_ring(const PrefillParams& p, float (&acc)[kCols], int row, int g,
                                                  uint32_t lane_base, uint64_t* tfull, uint32_t release0,
                                                  const float* ring, uint64_t* fslot_full, uint64_t* fslot_empty,
                                                  int64_t& it, int lane, volatile int* s_abort) {
  const int G = p.kslabs;
  const int nbi = g * kCols / 128;  // the tile's 128-column block of these columns
#pragma unroll
  for (int i = 0; i < kCols; ++i) acc[i] = 0.f;
  for (int kb = 0; kb < G; ++kb) {
    const int buf = (int)(it & 1), d = (int)(it % kScaleDepth);
    if (!dev::mbar_wait(&fslot_full[d], (uint32_t)((it / kScaleDepth) & 1), kWaitLimitNs) ||
        !dev::mbar_wait(&tfull[buf], (uint32_t)((it >> 1) & 1), kWaitLimitNs)) {
      set_abort(p, s_abort);
      return false;
    }
    tc_fence_after();
    const float* slot = ring + d * kFactorSlot;
    const float fk = slot[row] * slot[kBM + nbi];
    __syncwarp();
    if (lane == 0) dev::mbar_arrive(&fslot_empty[d]);
    uint64_t ff;  // (fk, fk) for the packed FMAs
    asm("mov.b64 %0, {%1, %1};" : "=l"(ff) : "f"(fk));
#pragma unroll
    for (int c = 0; c < kCols / 16; ++c) {
      uint32_t v[16];
      tmem_ld16(lane_base + buf * kBN + c * 16, v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; i += 2) fma2(acc[c * 16 + i], acc[c * 16 + i + 1], ff, v[i], v[i + 1]);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      const uint32_t rel = release0 + 8u * (uint32_t)buf;  // the two slab buffers' barriers are adjacent
      if (kPair)  // the first CTA's barrier, through its cluster address
        asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(rel) : "memory");
      else
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(rel) : "memory");
    }
    ++it;
  }
  return true;
}

// One 32-column chunk of the warp's 32 rows (this lane's row as 16 bf16-pair
// words, columns nc .. nc+31, all inside Y) through `stage`: written row by
// row (16-byte piece i of row r at slot i ^ ((r >> 1) & 3), so neither the
// writes nor the reads conflict on banks), read back so that one store
// instruction covers 8 rows x 64 contiguous bytes instead of 32 rows x 16.
__device__ __forceinline__ void store_chunk_staged(const PrefillParams& p, const uint32_t (&w)[16], int64_t m0,
                                                   int64_t nc, int lane, uint32_t sbase) {
  __syncwarp();  // the previous chunk has been read back
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t a = sbase + lane * 64 + ((i ^ ((lane >> 1) & 3)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w[4 * i]), "r"(w[4 * i + 1]),
                 "r"(w[4 * i + 2]), "r"(w[4 * i + 3])
                 : "memory");
  }
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 4; ++j) {  // rows 8j .. 8j+7, four lanes a row
    const int r = j * 8 + (lane >> 2), i = lane & 3;
    const uint32_t a = sbase + r * 64 + ((i ^ ((r >> 1) & 3)) << 4);
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a)
                 : "memory");
    const int64_t m = m0 + r;
    if (m < p.M) *reinterpret_cast<uint4*>(p.y + m * p.N + nc + i * 8) = v;
  }
}

// The warp's 32 rows m0 .. m0+31 (row m0 + lane in this lane's acc), columns
// n0 .. n0+kCols-1 of Y as bf16, 32 columns at a time through `stage`
// (kOutWarpBytes); store_row where the columns are ragged.
template <int kCols>
__device__ __forceinline__ void store_rows_staged(const PrefillParams& p, const float (&acc)[kCols], int64_t m0,
                                                  int64_t n0, int lane, uint8_t* stage) {
  if (n0 + kCols > p.N || (p.N & 7) != 0) {
    store_row<kCols>(p, acc, m0 + lane, n0);
    return;
  }
  const uint32_t sbase = dev::smem_addr(stage);
#pragma unroll
  for (int c = 0; c < kCols / kOutChunk; ++c) {
    uint32_t w[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[c * kOutChunk + 2 * t], acc[c * kOutChunk + 2 * t + 1]);
      w[t] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    store_chunk_staged(p, w, m0, n0 + c * kOutChunk, lane, sbase);
  }
}

__global__ void __launch_bounds__(kFp8Threads, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], mdone;
  __shared__ __align__(8) uint64_t ffull[kScaleDepth], fempty[kScaleDepth];
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
    for (int d = 0; d < kScaleDepth; ++d) {
      dev::mbar_init(&ffull[d], 32);  // every lane of the scale warp
      dev::mbar_init(&fempty[d], kEpiWarps);
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
  } else if (warp == 2 + kEpiWarps) {
    // ---- scale warp: each slab's factors into the ring, kScaleDepth ahead ---
    float* ring = reinterpret_cast<float*>(smem + kStages * kStageBytes);
    const int64_t sw_rows = (p.N + 127) / 128;
    int64_t it = 0;
    for (int64_t tile = blockIdx.x; tile < tiles && !s_abort; tile += gridDim.x) {
      const int32_t mt = (int32_t)(tile % p.m_tiles), nt = (int32_t)(tile / p.m_tiles);
      const int64_t m0 = (int64_t)mt * kBM + lane * 4, nb0 = (int64_t)nt * (kBN / 128);
      bool ok = true;
      for (int kb = 0; kb < G; ++kb, ++it) {
        const int d = (int)(it % kScaleDepth);
        if (!dev::mbar_wait(&fempty[d], (uint32_t)(((it / kScaleDepth) & 1) ^ 1), kWaitLimitNs)) {
          set_abort(p, &s_abort);
          ok = false;
          break;
        }
        float* slot = ring + d * kFactorSlot;
#pragma unroll
        for (int r = 0; r < 4; ++r) slot[lane * 4 + r] = m0 + r < p.M ? __ldg(p.ex + (m0 + r) * G + kb) : 0.f;
        if (lane < 2) slot[kBM + lane] = nb0 + lane < sw_rows ? __ldg(p.sw + (nb0 + lane) * G + kb) : 0.f;
        dev::mbar_arrive(&ffull[d]);  // each lane, after its own stores
      }
      if (!ok) break;
    }
  } else {
    // ---- promotion and output: 8 warps, thread = tile row, 128 columns -------
    constexpr int kCols = kBN / (kEpiWarps / 4);
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int g = (warp - 2) >> 2;   // which kCols of the tile's kBN columns
    const int row = q * 32 + lane;   // tile row = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + g * kCols;
    const float* ring = reinterpret_cast<const float*>(smem + kStages * kStageBytes);
    uint8_t* stage = smem + kStages * kStageBytes + scale_ring_bytes(kEpiWarps) + (warp - 2) * kOutWarpBytes;
    int64_t it = 0;
    for (int64_t tile = blockIdx.x; tile < tiles && !s_abort; tile += gridDim.x) {
      const int32_t mt = (int32_t)(tile % p.m_tiles), nt = (int32_t)(tile / p.m_tiles);
      const int64_t m = (int64_t)mt * kBM + row;
      const int64_t n0 = (int64_t)nt * kBN + g * kCols;
      float acc[kCols];
      if (!promote_tile_ring<kCols>(p, acc, row, g, lane_base, tfull, dev::smem_addr(&tempty[0]), ring, ffull,
                                    fempty, it, lane, &s_abort))
        break;
      store_rows_staged<kCols>(p, acc, m - lane, n0, lane, stage);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  if (p.trace && threadIdx.x == 0) {  // the record's end stamp after this kernel's writes
    __threadfence();
    dev::trace_end(p.trace, p.tag);
  }
}

// ---- CTA-pair kernel ------------------------------------------------------------
// Cluster rank 0 of each pair holds the stage "full" barriers that count both
// CTAs' copies and the slab-buffer "empty" barriers that count both CTAs'
// promotion warps, and its MMA thread issues the pair's MMAs. Tiles of
// 256 x 256 outputs go to clusters round-robin; CTA r of a pair owns
// activation rows mt*256 + r*128 .. +127 (its TMEM lanes) and loads weight
// rows nt*256 + r*128 .. +127 (the pair's MMA reads both weight halves).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    prefill_pair_kernel(const __grid_constant__ PrefillParams p) {
  constexpr int kNBuf = kTmemCols / kPairN;  // 2 slab buffers
  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t full[kPairStages], empty[kPairStages], tfull[kNBuf], tempty[kNBuf], mdone;
  __shared__ __align__(8) uint64_t ffull[kScaleDepth], fempty[kScaleDepth];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_cta_rank();
  const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles;
  const int64_t first = cluster_index(), stride = cluster_count();
  const int G = p.kslabs;

  if (threadIdx.x == 0) {
    dev::trace_start(p.trace);
    for (int s = 0; s < kPairStages; ++s) {
      dev::mbar_init(&full[s], 1);
      dev::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < kNBuf; ++b) {
      dev::mbar_init(&tfull[b], 1);
      dev::mbar_init(&tempty[b], 2 * kPairEpiWarps);
    }
    for (int d = 0; d < kScaleDepth; ++d) {
      dev::mbar_init(&ffull[d], 32);  // every lane of this CTA's scale warp
      dev::mbar_init(&fempty[d], kPairEpiWarps);
    }
    dev::mbar_init(&mdone, 1);
    dev::fence_mbar_init();
    s_abort = 0;
  }
  // Both CTAs' barriers are initialised, and both CTAs are running, before any
  // arrival crosses the pair and before the paired TMEM allocation.
  cluster_sync();
  if (warp == 1) {  // the same 512 columns in both CTAs' TMEM
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dev::smem_addr(&s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    // ---- TMA producer (both CTAs) ----------------------------------------
    if (lane == 0) {
      int64_t it = 0;
      for (int64_t tile = first; tile < tiles && !s_abort; tile += stride) {
        const int32_t mt = (int32_t)(tile % p.m_tiles), nt = (int32_t)(tile / p.m_tiles);
        const int32_t ya = mt * kPairM + (int32_t)rank * (kPairM / 2);
        const int32_t yb = nt * kPairN + (int32_t)rank * (kPairN / 2);
        for (int kb = 0; kb < G; ++kb, ++it) {
          const int s = (int)(it % kPairStages);
          if (!dev::mbar_wait(&empty[s], (uint32_t)(((it / kPairStages) & 1) ^ 1), kWaitLimitNs)) {
            set_abort(p, &s_abort);
            break;
          }
          if (rank == 0) dev::mbar_arrive_expect_tx(&full[s], 2 * kPairStageBytes);
          const uint32_t bar = cluster_addr(&full[s], 0);
          uint8_t* st = smem + s * kPairStageBytes;
          tma_load_2d_pair(st, &p.tmap_x, kb * kBK, ya, bar);
          tma_load_2d_pair(st + kPairABytes, &p.tmap_w, kb * kBK, yb, bar);
        }
      }
      // Rank 0 sees every stage land (both halves) before the pair may exit.
      if (rank == 0)
        for (int64_t k = it - kPairStages; k < it; ++k)
          if (k >= 0) dev::mbar_wait(&full[(int)(k % kPairStages)], (uint32_t)((k / kPairStages) & 1), kWaitLimitNs / 4);
    }
  } else if (warp == 1) {
    // ---- MMA issuer (rank 0 only) ------------------------------------------
    if (rank == 0 && lane == 0) {
      constexpr uint32_t idesc = idesc_f8(kPairM, kPairN);
      int64_t it = 0;
      bool issued = false;
      for (int64_t tile = first; tile < tiles && !s_abort; tile += stride) {
        for (int kb = 0; kb < G && !s_abort; ++kb, ++it) {
          const int s = (int)(it % kPairStages), buf = (int)(it % kNBuf);
          if (!dev::mbar_wait(&tempty[buf], (uint32_t)(((it / kNBuf) & 1) ^ 1), kWaitLimitNs)) {
            set_abort(p, &s_abort);
            break;
          }
          tc_fence_after();
          if (!dev::mbar_wait(&full[s], (uint32_t)((it / kPairStages) & 1), kWaitLimitNs)) {
            set_abort(p, &s_abort);
            break;
          }
          tc_fence_after();
          const uint32_t a = dev::smem_addr(smem + s * kPairStageBytes), b = a + kPairABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk)
            mma_f8_pair(tmem + buf * kPairN, smem_desc_sw128(a + kk * 32), smem_desc_sw128(b + kk * 32), idesc,
                        kk > 0);
          mma_commit_pair(&empty[s]);
          mma_commit_pair(&tfull[buf]);
          issued = true;
        }
      }
      if (issued) {  // the pair's MMAs complete before either CTA releases TMEM
        mma_commit_pair(&mdone);
        dev::mbar_wait(&mdone, 0, kWaitLimitNs);
      }
    }
  } else if (warp == 2 + kPairEpiWarps) {
    // ---- scale warp (both CTAs): this CTA's factors into its ring ------------
    float* ring = reinterpret_cast<float*>(smem + kPairStages * kPairStageBytes);
    const int64_t sw_rows = (p.N + 127) / 128;
    int64_t it = 0;
    for (int64_t tile = first; tile < tiles && !s_abort; tile += stride) {
      const int32_t mt = (int32_t)(tile % p.m_tiles), nt = (int32_t)(tile / p.m_tiles);
      const int64_t m0 = (int64_t)mt * kPairM + (int64_t)rank * (kPairM / 2) + lane * 4;
      const int64_t nb0 = (int64_t)nt * (kPairN / 128);
      bool ok = true;
      for (int kb = 0; kb < G; ++kb, ++it) {
        const int d = (int)(it % kScaleDepth);
        if (!dev::mbar_wait(&fempty[d], (uint32_t)(((it / kScaleDepth) & 1) ^ 1), kWaitLimitNs)) {
          set_abort(p, &s_abort);
          ok = false;
          break;
        }
        float* slot = ring + d * kFactorSlot;
#pragma unroll
        for (int r = 0; r < 4; ++r) slot[lane * 4 + r] = m0 + r < p.M ? __ldg(p.ex + (m0 + r) * G + kb) : 0.f;
        if (lane < 2) slot[kBM + lane] = nb0 + lane < sw_rows ? __ldg(p.sw + (nb0 + lane) * G + kb) : 0.f;
        dev::mbar_arrive(&ffull[d]);  // each lane, after its own stores
      }
      if (!ok) break;
    }
  } else {
    // ---- promotion and output (both CTAs): 16 warps, 64 columns each ------------
    constexpr int kCols = kPairN / (kPairEpiWarps / 4);
    const int q = warp & 3;
    const int g = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + g * kCols;
    const float* ring = reinterpret_cast<const float*>(smem + kPairStages * kPairStageBytes);
    int64_t it = 0;
    for (int64_t tile = first; tile < tiles && !s_abort; tile += stride) {
      const int32_t mt = (int32_t)(tile % p.m_tiles), nt = (int32_t)(tile / p.m_tiles);
      const int64_t m = (int64_t)mt * kPairM + (int64_t)rank * (kPairM / 2) + row;
      const int64_t n0 = (int64_t)nt * kPairN + g * kCols;
      float acc[kCols];
      if (!promote_tile_ring<kCols, true>(p, acc, row, g, lane_base, tfull, cluster_addr(&tempty[0], 0), ring,
                                          ffull, fempty, it, lane, &s_abort))
        break;
      store_row<kCols>(p, acc, m, n0);
    }
  }
  __syncthreads();
  if (s_abort && threadIdx.x == 0) {
    // After a timeout this CTA may have copies in flight whose barrier is the
    // peer's: give them a millisecond to land before the memory is released.
    const uint64_t t0 = dev::globaltimer();
    while (dev::globaltimer() - t0 < 1000000ull) {
    }
  }
  __syncthreads();
  cluster_sync();  // both CTAs are done with TMEM and with each other's barriers
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  if (p.trace && threadIdx.x == 0) {  // the record's end stamp after this kernel's writes
    __threadfence();
    dev::trace_end(p.trace, p.tag);
  }
}

// ---- 16-bit weights -------------------------------------------------------------
// Y = X W^T with bf16 X [M, K] and bf16 W [N, K] (or both f16), no scales: the whole K of a
// tile accumulates in TMEM (tcgen05.mma kind::f16, 128 x 256 x 16), and the
// tile is read out once. One CTA per 128 x 256 tile; a slab is 64 K (one
// 128-byte row of each operand), 4 stages of 48 KB; the two TMEM buffers hold
// consecutive tiles, so the read-out of tile t overlaps the MMAs of tile t+1.
// 8 read-out warps: thread = tile row (TMEM lane), 128 columns each.
constexpr int kBf16SlabK = 64;

__host__ __device__ constexpr uint32_t idesc_16(int m, int n, bool f16) {
  return (1u << 4)                                      // D format: f32
         | (f16 ? 0u : (1u << 7) | (1u << 10))          // A, B format: f16 (0) or bf16 (1)
         | ((uint32_t)(n >> 3) << 17)  // N / 8
         | ((uint32_t)(m >> 4) << 24); // M / 16
}

__device__ __forceinline__ void mma_16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

template <bool F16>
__global__ void __launch_bounds__(kThreads, 1) prefill_16_kernel(const __grid_constant__ PrefillParams p) {
  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], mdone;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles;
  const int G = p.kslabs;  // 64-K slabs

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
          // x coordinates are in bytes of the [rows, 2K] byte view: 128 per slab
          tma_load_2d(st, &p.tmap_x, kb * 128, mt * kBM, &full[s]);
          tma_load_2d(st + kABytes, &p.tmap_w, kb * 128, nt * kBN, &full[s]);
        }
      }
      for (int64_t k = it - kStages; k < it; ++k)
        if (k >= 0) dev::mbar_wait(&full[(int)(k % kStages)], (uint32_t)((k / kStages) & 1), kWaitLimitNs / 4);
    }
  } else if (warp == 1) {
    // ---- MMA issuer: a tile's slabs accumulate into TMEM buffer t % 2 -------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_16(kBM, kBN, F16);
      int64_t it = 0, t = 0;
      bool issued = false;
      for (int64_t tile = blockIdx.x; tile < tiles && !s_abort; tile += gridDim.x, ++t) {
        const int buf = (int)(t & 1);
        if (!dev::mbar_wait(&tempty[buf], (uint32_t)(((t >> 1) & 1) ^ 1), kWaitLimitNs)) {
          set_abort(p, &s_abort);
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < G && !s_abort; ++kb, ++it) {
          const int s = (int)(it % kStages);
          if (!dev::mbar_wait(&full[s], (uint32_t)((it / kStages) & 1), kWaitLimitNs)) {
            set_abort(p, &s_abort);
            break;
          }
          tc_fence_after();
          const uint32_t a = dev::smem_addr(smem + s * kStageBytes), b = a + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBf16SlabK / 16; ++kk)  // 16 K = 32 bytes per MMA
            mma_16(tmem + buf * kBN, smem_desc_sw128(a + kk * 32), smem_desc_sw128(b + kk * 32), idesc,
                     (kb > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&empty[s]);
          issued = true;
        }
        if (s_abort) break;
        mma_commit(&tfull[buf]);
      }
      if (issued) {
        mma_commit(&mdone);
        dev::mbar_wait(&mdone, 0, kWaitLimitNs);
      }
    }
  } else {
    // ---- read-out: thread = tile row, 128 columns ----------------------------
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + h * 128;
    const uint32_t stage_addr =
        dev::smem_addr(smem + kStages * kStageBytes + scale_ring_bytes(kEpiWarps) + (warp - 2) * kOutWarpBytes);
    int64_t t = 0;
    for (int64_t tile = blockIdx.x; tile < tiles && !s_abort; tile += gridDim.x, ++t) {
      const int buf = (int)(t & 1);
      if (!dev::mbar_wait(&tfull[buf], (uint32_t)((t >> 1) & 1), kWaitLimitNs)) {
        set_abort(p, &s_abort);
        break;
      }
      tc_fence_after();
      const int32_t mt = (int32_t)(tile % p.m_tiles), nt = (int32_t)(tile / p.m_tiles);
      const int64_t m = (int64_t)mt * kBM + row;
      const int64_t n0 = (int64_t)nt * kBN + h * 128;
      const bool vec = (p.N & 7) == 0;
      if (vec && n0 + 128 <= p.N) {  // whole columns: through shared memory, 8 rows x 64 bytes a store
#pragma unroll 1
        for (int c = 0; c < 128 / kOutChunk; ++c) {
          uint32_t v[32], w[16];
          tmem_ld16(lane_base + buf * kBN + c * kOutChunk, *reinterpret_cast<uint32_t(*)[16]>(v));
          tmem_ld16(lane_base + buf * kBN + c * kOutChunk + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
          tmem_wait_ld();
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * t]), __uint_as_float(v[2 * t + 1]));
            w[t] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          store_chunk_staged(p, w, m - lane, n0 + c * kOutChunk, lane, stage_addr);
        }
      } else {
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t v[16];
        tmem_ld16(lane_base + buf * kBN + c * 16, v);
        tmem_wait_ld();
        const int64_t nc = n0 + c * 16;
        if (m < p.M && nc < p.N) {
          uint16_t* yp = p.y + m * p.N + nc;
          uint32_t w[8];
#pragma unroll
          for (int t2 = 0; t2 < 8; ++t2) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * t2]), __uint_as_float(v[2 * t2 + 1]));
            w[t2] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          if (vec && nc + 16 <= p.N) {
            reinterpret_cast<uint4*>(yp)[0] = make_uint4(w[0], w[1], w[2], w[3]);
            reinterpret_cast<uint4*>(yp)[1] = make_uint4(w[4], w[5], w[6], w[7]);
          } else {
            for (int i = 0; i < 16 && nc + i < p.N; ++i) yp[i] = (uint16_t)(w[i >> 1] >> ((i & 1) * 16));
          }
        }
      }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(&tempty[buf]);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  if (p.trace && threadIdx.x == 0) {  // the record's end stamp after this kernel's writes
    __threadfence();
    dev::trace_end(p.trace, p.tag);
  }
}

std::atomic<int> g_prefill_kernel{kPrefillAuto};  // SWS_OPT_PREFILL_KERNEL

// Clusters of two prefill_pair_kernel CTAs that fit on the current device at
// once (0 if none; cached per device).
int pair_cluster_capacity() {
  static int cache[64];
  static bool known[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!known[dev]) {
    int n = 0;
    if (cudaFuncSetAttribute(prefill_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmemBytes) ==
        cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * (unsigned)device_sm_count(), 1, 1);
      cfg.blockDim = dim3(kPairThreads, 1, 1);
      cfg.dynamicSmemBytes = kPairSmemBytes;
      if (cudaOccupancyMaxActiveClusters(&n, prefill_pair_kernel, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();  // a failed query leaves no sticky error
    cache[dev] = n;
    known[dev] = true;
  }
  return cache[dev];
}

}  // namespace

void set_prefill_kernel(int k) { g_prefill_kernel.store(k, std::memory_order_relaxed); }

int launch_prefill(const PrefillLaunch& a, cudaStream_t s) {
  if (a.m <= 0 || a.rows <= 0) return SWS_OK;
  if (a.cols <= 0 || a.cols % 128 != 0)
    return fail(SWS_E_UNSUPPORTED, "prefill: cols=%lld is not a positive multiple of 128", (long long)a.cols);
  if (!aligned16(a.w) || !aligned16(a.xq) || !aligned16(a.y) || !aligned16(a.ex) || !aligned16(a.scales))
    return fail(SWS_E_ALIGN, "prefill: pointer not 16-byte aligned");
  const int choice = g_prefill_kernel.load(std::memory_order_relaxed);
  const int clusters = choice == kPrefillPair ? pair_cluster_capacity() : 0;
  if (choice == kPrefillPair && clusters <= 0)
    return fail(SWS_E_UNSUPPORTED, "prefill: no cluster of two CTAs fits on this device");
  const bool pair = clusters > 0 && choice == kPrefillPair;
  PrefillParams p;
  int rc = encode_u8_tile_map(&p.tmap_x, a.xq, a.m, a.cols, pair ? kPairM / 2 : kBM);
  if (rc != SWS_OK) return rc;
  rc = encode_u8_tile_map(&p.tmap_w, a.w, a.rows, a.cols, pair ? kPairN / 2 : kBN);
  if (rc != SWS_OK) return rc;
  p.ex = a.ex;
  p.sw = a.scales;
  p.y = a.y;
  p.M = a.m;
  p.N = a.rows;
  p.K = a.cols;
  p.kslabs = (int32_t)(a.cols / kBK);
  p.m_tiles = (int32_t)cdiv(a.m, pair ? kPairM : kBM);
  p.n_tiles = (int32_t)cdiv(a.rows, pair ? kPairN : kBN);
  p.status = a.status;
  p.trace = a.trace;
  p.tag = pair ? (a.tag & ~(0xFFull << 48)) | (kTracePrefillPair << 48) : a.tag;
  const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles;
  if (pair) {
    const int64_t n_clusters = std::min<int64_t>(tiles, clusters);
    cudaError_t le = launch_high(prefill_pair_kernel, dim3((unsigned)(2 * n_clusters)), dim3(kPairThreads),
                                 kPairSmemBytes, s, p);
    if (le != cudaSuccess) return cuda_fail(le, "prefill pair kernel launch");
  } else {
    static PerDevice once;
    const cudaError_t attr = once.run(
        [] { return cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes); });
    if (attr != cudaSuccess) return cuda_fail(attr, "prefill: cudaFuncSetAttribute");
    const int64_t grid = std::min<int64_t>(tiles, device_sm_count());
    cudaError_t le = launch_high(prefill_kernel, dim3((unsigned)grid), dim3(kFp8Threads), kSmemBytes, s, p);
    if (le != cudaSuccess) return cuda_fail(le, "prefill kernel launch");
  }
  return SWS_OK;
}

int launch_prefill_16(const PrefillLaunch& a, bool f16, cudaStream_t s) {
  if (a.m <= 0 || a.rows <= 0) return SWS_OK;
  if (a.cols <= 0 || a.cols % 8 != 0)
    return fail(SWS_E_UNSUPPORTED, "prefill: 16-bit cols=%lld is not a positive multiple of 8", (long long)a.cols);
  if (!aligned16(a.w) || !aligned16(a.xq) || !aligned16(a.y))
    return fail(SWS_E_ALIGN, "prefill: pointer not 16-byte aligned");
  PrefillParams p;
  // 16-bit rows as bytes: 128-byte boxes (64 K) of [rows, 2K] byte tensors
  int rc = encode_u8_tile_map(&p.tmap_x, a.xq, a.m, 2 * a.cols, kBM);
  if (rc != SWS_OK) return rc;
  rc = encode_u8_tile_map(&p.tmap_w, a.w, a.rows, 2 * a.cols, kBN);
  if (rc != SWS_OK) return rc;
  p.ex = nullptr;
  p.sw = nullptr;
  p.y = a.y;
  p.M = a.m;
  p.N = a.rows;
  p.K = a.cols;
  p.kslabs = (int32_t)cdiv(a.cols, kBf16SlabK);
  p.m_tiles = (int32_t)cdiv(a.m, kBM);
  p.n_tiles = (int32_t)cdiv(a.rows, kBN);
  p.status = a.status;
  p.trace = a.trace;
  p.tag = a.tag;
  static PerDevice once;
  const cudaError_t attr = once.run([] {
    cudaError_t a = cudaFuncSetAttribute(prefill_16_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (a == cudaSuccess)
      a = cudaFuncSetAttribute(prefill_16_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    return a;
  });
  if (attr != cudaSuccess) return cuda_fail(attr, "prefill: cudaFuncSetAttribute (16-bit)");
  const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles;
  const int64_t grid = std::min<int64_t>(tiles, device_sm_count());
  cudaError_t e = f16 ? launch_high(prefill_16_kernel<true>, dim3((unsigned)grid), dim3(kThreads), kSmemBytes, s, p)
                      : launch_high(prefill_16_kernel<false>, dim3((unsigned)grid), dim3(kThreads), kSmemBytes, s, p);
  return e == cudaSuccess ? SWS_OK : cuda_fail(e, "prefill 16-bit kernel launch");
}

}  // namespace sws
