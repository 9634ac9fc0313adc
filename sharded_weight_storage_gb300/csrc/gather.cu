// Chunk -> slot gather and the one-time relayout, for sm_103a.
//
// gather: the single-GPU stand-in for the per-layer all_gather_into_tensor of
// the weight-sharding blog (section "一层一次 AllGather：flat layout", step 3):
// slot[i*C : (i+1)*C] = chunk_i. It is a pure byte copy, so the kernel is built
// for HBM bandwidth: each CTA runs a ring of shared-memory stages; one thread
// issues bulk TMA loads (global -> shared, completion on an mbarrier) and bulk
// TMA stores (shared -> global) so that several tiles per SM are in flight
// without occupying registers. Tiles are assigned round-robin over a grid
// sized to the SM count. Two shapes: 2 CTAs per SM with 3 x 32 KB stages (the
// fastest alone), and 1 CTA per SM with 3 x 16 KB stages, which fits in the
// shared memory a decode GEMM CTA leaves free, so that a lookahead gather and
// the current layer's linears run on the same SMs at the same time instead of
// one after the other. Both ask for the largest shared-memory carveout, so an
// SM that runs one of them can still take the other's CTAs.
//
// relayout: section "加载：行 shard 先行，finalize 再重排", step 2 - the one-time
// remap of per-weight row shards into flat chunks, expressed by the host as a
// list of contiguous copy / zero-fill segments.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "ptx.cuh"
#include "sws_internal.h"

namespace sws {

// ---------------------------------------------------------------------------
// device properties
// ---------------------------------------------------------------------------
int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

// The highest stream priority of the current device (the numerically smallest
// value; cached per device). The linears' kernels are launched with it so that,
// when a gather on another stream competes for SMs, the block scheduler
// places the linears' CTAs first; the gather keeps the default priority.
int high_priority() {
  static int cache[64];
  static bool known[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!known[dev]) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) greatest = 0;
    cache[dev] = greatest;
    known[dev] = true;
  }
  return cache[dev];
}

int check_device() {
  int dev = 0, major = 0, minor = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(major)");
  e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(minor)");
  if (major != 10 || minor != 3)
    return fail(SWS_E_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major, minor);
  return SWS_OK;
}

// ---------------------------------------------------------------------------
// gather
// ---------------------------------------------------------------------------
namespace {

constexpr int kGatherTile = 32 * 1024;  // bytes per stage
constexpr int kGatherStages = 3;
constexpr int kGatherCtasPerSm = 2;
constexpr int kSharedTile = 16 * 1024;  // the shared-SM variant
constexpr int kSharedStages = 3;
constexpr int kSharedCtasPerSm = 1;

struct GatherParams {
  const uint8_t* chunks[256];
  int64_t chunk_bytes;
  int64_t tiles_per_chunk;
  int64_t total_tiles;
  uint8_t* dst;
  int32_t* status;
  uint64_t* trace;
  uint64_t tag;
};

template <int TILE, int STAGES>
__global__ void __launch_bounds__(32) gather_kernel(const __grid_constant__ GatherParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[STAGES];
  if (threadIdx.x != 0) return;
  dev::trace_start(p.trace);
  const int64_t G = gridDim.x, b = blockIdx.x;
  const int64_t n_my = (b < p.total_tiles) ? (p.total_tiles - 1 - b) / G + 1 : 0;
  for (int s = 0; s < STAGES; ++s) dev::mbar_init(&bars[s], 1);
  dev::fence_mbar_init();

  auto tile_of = [&](int64_t k, const uint8_t** src, uint8_t** dst, uint32_t* bytes) {
    const int64_t t = b + k * G;
    const int64_t ci = t / p.tiles_per_chunk;
    const int64_t off = (t - ci * p.tiles_per_chunk) * TILE;
    *bytes = (uint32_t)min((int64_t)TILE, p.chunk_bytes - off);
    *src = p.chunks[ci] + off;
    *dst = p.dst + ci * p.chunk_bytes + off;
  };
  auto issue_load = [&](int64_t k) {
    const uint8_t* src;
    uint8_t* dst;
    uint32_t bytes;
    tile_of(k, &src, &dst, &bytes);
    const int s = (int)(k % STAGES);
    dev::mbar_arrive_expect_tx(&bars[s], bytes);
    dev::bulk_g2s(smem + s * TILE, src, bytes, &bars[s]);
  };

  const int64_t pre = n_my < STAGES ? n_my : STAGES;
  for (int64_t k = 0; k < pre; ++k) issue_load(k);
  int64_t issued = pre;
  bool ok = true;
  for (int64_t k = 0; k < n_my; ++k) {
    const int s = (int)(k % STAGES);
    if (!dev::mbar_wait(&bars[s], (uint32_t)((k / STAGES) & 1), kWaitLimitNs)) {
      ok = false;
      break;
    }
    dev::fence_proxy_async_smem();
    const uint8_t* src;
    uint8_t* dst;
    uint32_t bytes;
    tile_of(k, &src, &dst, &bytes);
    dev::bulk_s2g(dst, smem + s * TILE, bytes);
    dev::bulk_commit();
    // Refill the stage of tile k-1 once its store has finished reading it.
    if (k >= 1 && issued < n_my) {
      dev::bulk_wait_read<1>();
      issue_load(issued);
      ++issued;
    }
  }
  if (!ok) {
    dev::set_status(p.status, SWS_E_TIMEOUT);
    // Drain loads still in flight (bounded), so no copy targets freed smem.
    for (int64_t k = 0; k < issued; ++k) {
      const int s = (int)(k % STAGES);
      dev::mbar_wait(&bars[s], (uint32_t)((k / STAGES) & 1), kWaitLimitNs / 4);
    }
  }
  dev::bulk_wait<0>();
  dev::trace_end(p.trace, p.tag);
}

template <int TILE, int STAGES, int CTAS_PER_SM>
cudaError_t launch_gather_shape(const GatherLaunch& a, cudaStream_t stream) {
  GatherParams p;
  for (int i = 0; i < a.n; ++i) p.chunks[i] = a.chunks[i];
  p.chunk_bytes = a.chunk_bytes;
  p.tiles_per_chunk = cdiv(a.chunk_bytes, TILE);
  p.total_tiles = p.tiles_per_chunk * a.n;
  p.dst = a.dst;
  p.status = a.status;
  p.trace = a.trace;
  p.tag = a.tag;
  if (p.total_tiles == 0) return cudaSuccess;
  auto kern = gather_kernel<TILE, STAGES>;
  constexpr int smem = TILE * STAGES;
  static PerDevice once;
  const cudaError_t attr_err = once.run([&] {
    cudaError_t a = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (a == cudaSuccess)
      a = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
    return a;
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t grid = std::min<int64_t>(p.total_tiles, (int64_t)device_sm_count() * CTAS_PER_SM);
  // With overlap_prev, programmatic stream serialisation: when the previous
  // kernel on the stream is a decode launch's settle grid (which releases its
  // dependents at once), the gather overlaps it; after any other kernel it
  // starts as usual, when that kernel completes. The gather never waits on
  // its predecessor's data.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = a.overlap_prev ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

cudaError_t launch_gather(const GatherLaunch& a, cudaStream_t stream) {
  return a.shared_sm ? launch_gather_shape<kSharedTile, kSharedStages, kSharedCtasPerSm>(a, stream)
                     : launch_gather_shape<kGatherTile, kGatherStages, kGatherCtasPerSm>(a, stream);
}

// ---------------------------------------------------------------------------
// relayout
// ---------------------------------------------------------------------------
namespace {

constexpr int kSegBatch = 512;
constexpr int64_t kPiece = 32 * 1024;

struct RelayoutParams {
  CopySeg seg[kSegBatch];
  int32_t piece_prefix[kSegBatch + 1];  // pieces before segment i
  int32_t n;
};

__global__ void __launch_bounds__(256) relayout_kernel(const __grid_constant__ RelayoutParams p) {
  const int32_t piece = blockIdx.x;
  // segment holding this piece: last i with prefix[i] <= piece
  int lo = 0, hi = p.n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (p.piece_prefix[mid] <= piece) lo = mid; else hi = mid - 1;
  }
  const CopySeg sg = p.seg[lo];
  const int64_t begin = (int64_t)(piece - p.piece_prefix[lo]) * kPiece;
  const int64_t len = min(kPiece, sg.len - begin);
  uint8_t* dst = sg.dst + begin;
  const uint8_t* src = sg.src ? sg.src + begin : nullptr;
  const bool vec = ((reinterpret_cast<uintptr_t>(dst) | (src ? reinterpret_cast<uintptr_t>(src) : 0) | (uintptr_t)len) & 15) == 0;
  if (vec) {
    uint4* d = reinterpret_cast<uint4*>(dst);
    const int64_t nv = len >> 4;
    if (src) {
      const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll 4
      for (int64_t i = threadIdx.x; i < nv; i += blockDim.x) d[i] = __ldg(s + i);
    } else {
      for (int64_t i = threadIdx.x; i < nv; i += blockDim.x) d[i] = make_uint4(0, 0, 0, 0);
    }
  } else {
    for (int64_t i = threadIdx.x; i < len; i += blockDim.x) dst[i] = src ? src[i] : 0;
  }
}

}  // namespace

cudaError_t launch_relayout(const std::vector<CopySeg>& segs, cudaStream_t stream) {
  size_t i = 0;
  while (i < segs.size()) {
    RelayoutParams p;
    int n = 0;
    int64_t pieces = 0;
    while (i < segs.size() && n < kSegBatch) {
      const CopySeg& s = segs[i];
      if (s.len <= 0) { ++i; continue; }
      const int64_t np = cdiv(s.len, kPiece);
      if (pieces + np > (int64_t)1 << 30) break;
      p.seg[n] = s;
      p.piece_prefix[n] = (int32_t)pieces;
      pieces += np;
      ++n;
      ++i;
    }
    if (n == 0) break;
    p.piece_prefix[n] = (int32_t)pieces;
    p.n = n;
    relayout_kernel<<<(unsigned)pieces, 256, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ---------------------------------------------------------------------------
// trace records
// ---------------------------------------------------------------------------
namespace {
__global__ void trace_reset_kernel(uint64_t* rec, int32_t n) {
  for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    rec[4 * i + 0] = 0;
    rec[4 * i + 1] = ~0ull;
    rec[4 * i + 2] = 0;
    rec[4 * i + 3] = 0;
  }
}
// A wait on an mbarrier that nothing arrives at, with the same bounded wait
// every kernel of the library uses: it gives up after limit_ns and records
// SWS_E_TIMEOUT in the status word, then the kernel returns normally.
__global__ void bounded_wait_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  dev::mbar_init(&bar, 1);
  dev::fence_mbar_init();
  if (!dev::mbar_wait(&bar, 0, limit_ns)) dev::set_status(status, SWS_E_TIMEOUT);
}
}  // namespace

cudaError_t launch_bounded_wait(int32_t* status, uint64_t limit_ns, cudaStream_t s) {
  bounded_wait_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_trace_reset(uint64_t* rec, int32_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  trace_reset_kernel<<<(unsigned)std::min<int64_t>(cdiv(n, 256), 1024), 256, 0, s>>>(rec, n);
  return cudaGetLastError();
}

}  // namespace sws
