// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <utility>
#include <stdint.h>

#include <string>
#include <vector>

#include "sws.h"

namespace sws {

// ---- errors -----------------------------------------------------------------
// Records a message for sws_last_error() and returns `code`.
int fail(int code, const char* fmt, ...);
int cuda_fail(cudaError_t e, const char* what);
void clear_error();  // empties sws_last_error() on the calling thread
#define SWS_CUDA_TRY(expr)                                   \
  do {                                                       \
    cudaError_t _e = (expr);                                 \
    if (_e != cudaSuccess) return ::sws::cuda_fail(_e, #expr); \
  } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t roundup(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int elem_bytes(int32_t dtype);  // 0 for an unknown type

// ---- plan ------------------------------------------------------------------
struct EntryPlan {
  int32_t layer = 0, dtype = 0;
  int64_t rows = 0, cols = 0, elem = 1, bytes = 0;
  bool sharded = false;
  int64_t offset = -1;       // o_j inside the layer's T, -1 if replicated
  int32_t index_in_layer = 0; // position among all entries of the layer
  // SWS_SCALES_IN_T: the entry's fp32 block scales [ceil(rows/128),
  // ceil(cols/128)] as their own entry of T right after the weight (-1 when
  // the scales are not in T), their size, and where the chunk-map path stages
  // them in the workspace (offset inside the layer's staging area).
  int64_t scale_offset = -1, scale_bytes = 0, scale_stage = 0;
};

struct LayerPlan {
  std::vector<int32_t> sharded;  // entry ids packed into T, in order
  std::vector<int32_t> all;      // every entry id of the layer, in order
  int64_t total = 0, chunk = 0;
  int64_t scale_stage_bytes = 0;  // SWS_SCALES_IN_T: staging area of the layer's scales (chunk-map path)
};

// ---- device status word and trace records (inside the workspace) -----------
// Workspace layout (bytes):
//   [0, 256)        control: status word (int32 at 0)
//   [256, 256+CNT)  split-K arrival counters (int32 per row block)
//   then            split-K partial sums (fp32)
//   then            tcgen05 decode: activation split blocks
//   then            prefill quantiser output (xq bytes, then ex floats)
constexpr int64_t kCtlBytes = 256;
constexpr int64_t kMaxCounters = 1 << 16;

// Kinds written into trace tags.
constexpr uint64_t kTraceGather = 1, kTraceLinear = 2;
// Kernel of a linear launch, in bits 48..55 of its trace tag.
constexpr uint64_t kTraceMma = 1, kTraceMmaFused = 2, kTraceTc = 3, kTraceTcFused = 4, kTracePrefill = 5,
                   kTracePrefillPair = 6;

// Device-side wait limit for mbarrier / TMA waits, in nanoseconds of
// %globaltimer. A wait that runs out sets the status word and the kernel exits.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// 2-D tensor map of a byte matrix [rows, cols] (row stride cols, cols % 16 ==
// 0): boxes of box_cols (128 or 64) bytes by box_rows rows, with the swizzle of
// that width (128- or 64-byte), zero fill outside.
int encode_u8_tile_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows,
                       int box_cols = 128);

// Runs a set-up step (kernel attributes such as the dynamic shared-memory
// limit, which the runtime keeps per device) once for each device it is called
// on - the current one - and returns that device's result on every later call.
struct PerDevice {
  static constexpr int kMaxDevices = 64;
  std::mutex mu;
  bool done[kMaxDevices] = {};
  cudaError_t err[kMaxDevices] = {};
  template <typename F>
  cudaError_t run(F&& f) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
      err[dev] = f();
      done[dev] = true;
    }
    return err[dev];
  }
};

// Host-side waits for the device (sws_run_timing, sws_ctx_status,
// sws_noalloc_status) give up after this many milliseconds with SWS_E_TIMEOUT
// (SWS_OPT_HOST_WAIT_MS; the default is well above the device-side limit).
int host_wait_ms();
// Polls `ev` (cudaEventQuery) until it has completed or host_wait_ms() passed.
int wait_event_deadline(cudaEvent_t ev, const char* what);
// Waits for all work queued on `device` (cudaDeviceSynchronize on a helper
// thread) for at most host_wait_ms(); SWS_E_TIMEOUT when it did not finish.
int device_sync_deadline(int device, const char* what);

// ---- kernel launchers (defined in the .cu files) -----------------------------
int device_sm_count();
int high_priority();  // launch priority of the linears' kernels (see gather.cu)

// Launch with the high priority (kernels of the linears and their helpers).
template <typename... KArgs, typename... Args>
cudaError_t launch_high(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                        Args&&... args) {
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributePriority;
  at[0].val.priority = high_priority();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
int check_device();  // SWS_OK if the current device is sm_103, else an error code

struct GatherLaunch {
  const uint8_t* chunks[256];
  int32_t n;
  int64_t chunk_bytes;
  uint8_t* dst;
  int32_t* status;
  uint64_t* trace;  // record (4 x u64) or nullptr
  uint64_t tag;     // written into the record's tag field
  bool shared_sm = false;  // the small-footprint variant that fits beside a decode GEMM CTA
  bool overlap_prev = false;  // programmatic stream serialisation: may overlap a predecessor that allows it
};
cudaError_t launch_gather(const GatherLaunch& a, cudaStream_t s);

struct CopySeg {
  const uint8_t* src;  // nullptr: fill with zeros
  uint8_t* dst;
  int64_t len;
};
cudaError_t launch_relayout(const std::vector<CopySeg>& segs, cudaStream_t s);
// Appends the copy segments that move T bytes [g0, g1) of a layer with chunk
// size c between the chunks and a linear buffer `lin` (lin holds byte g0 at
// its start): to_chunks copies lin -> chunks, else chunks -> lin; lin ==
// nullptr with to_chunks fills the chunk bytes with zeros.
void chunk_segments(int64_t g0, int64_t g1, int64_t c, void* const* chunks, const uint8_t* lin_src, uint8_t* lin_dst,
                    std::vector<CopySeg>* segs);
// SWS_OPT_CHECK_BOUNDS: a buffer [lo, hi) that copy segments may read or write.
struct Extent {
  const uint8_t* lo;
  const uint8_t* hi;
};
bool check_bounds();
void set_check_bounds(bool on);
// SWS_E_INVALID (naming `what` and the segment) if a segment reads outside
// every extent of `srcs` (zero fills read nothing) or writes outside every
// extent of `dsts`; SWS_OK otherwise.
int check_segments(const std::vector<CopySeg>& segs, std::vector<Extent> srcs, std::vector<Extent> dsts,
                   const char* what);
// The extents of a layer's N chunks of c bytes.
std::vector<Extent> chunk_extents(void* const* chunks, int32_t n, int64_t c);

// Decode linears (m <= 64): a group of up to kMaxDecodeGroup linears that
// share m runs as one launch. Slot path: each item's weight is a view `w`
// [rows, cols] (TMA). Fused path: each item's bytes are T[t_offset, ...) read
// through the layer's chunks (byte g of T lives in chunks[g / C] at g % C).
constexpr int kMaxDecodeGroup = 8;
struct DecodeItem {
  const uint8_t* w;  // slot / replicated view (unused on the fused path)
  const float* scales;
  const uint16_t* x;  // bf16 [m, cols]
  uint16_t* y;        // bf16 [m, rows]
  int64_t rows, cols;
  int64_t t_offset;  // fused path: o_j
};
struct DecodeGroup {
  DecodeItem item[kMaxDecodeGroup];
  int32_t n = 0;
  int64_t m = 0;
  bool fused = false;
  int wtype = 0;  // every item's weight: 0 e4m3 codes with block scales, 1 bf16, 2 f16 (no scales)
  const uint8_t* chunks[256];
  int32_t n_chunks = 0;
  int64_t chunk_bytes = 0;
  uint8_t* workspace = nullptr;  // control + counters + partials
  int64_t workspace_bytes = 0;
  uint64_t* trace = nullptr;
  uint64_t tag = 0;
};
// Workspace a decode launch with this m needs (independent of the shapes, up
// to kMaxCounters row blocks per launch).
int decode_workspace_bytes(int64_t m, int64_t* bytes);
// Activation split region a tcgen05 decode launch needs after that workspace:
// one block per K slab of its linears (slabs = sum of ceil(cols / 128)).
int64_t decode_split_bytes(int64_t m, int64_t slabs);
int launch_decode(const DecodeGroup& g, cudaStream_t s);
// Which decode kernel serves a view-path launch: SWS_DECODE_AUTO picks by m.
enum DecodeKernel { kDecodeAuto = 0, kDecodeMma = 1, kDecodeTc = 2 };
void set_decode_kernel(int k);
int decode_kernel_for(int64_t m);

int launch_quantize_x(const uint16_t* x, int64_t m, int64_t k, uint8_t* xq, float* ex, cudaStream_t s);
int launch_silu_mul(const uint16_t* gu, int64_t m, int64_t f, uint16_t* act, cudaStream_t s);
// bf16 -> f16 (round to nearest even) of n elements, n % 8 == 0.
int launch_to_f16(const uint16_t* x, int64_t n, uint16_t* out, cudaStream_t s);

struct PrefillLaunch {
  const uint8_t* w;      // fp8 [rows, cols] (slot view or replicated buffer)
  const float* scales;   // [ceil(rows/128), cols/128]
  const uint8_t* xq;     // fp8 [m, cols]
  const float* ex;       // [m, cols/128]
  uint16_t* y;           // bf16 [m, rows]
  int64_t m, rows, cols;
  int32_t* status;
  uint64_t* trace;
  uint64_t tag;
};
enum PrefillKernel { kPrefillAuto = 0, kPrefillSingle = 1, kPrefillPair = 2 };
void set_prefill_kernel(int k);
int launch_prefill(const PrefillLaunch& a, cudaStream_t s);
// 16-bit weights: `xq` is the activation X [m, cols] in the weights' format
// (bf16, or f16 when f16 is set), `w` [rows, cols]; ex and scales are unused.
int launch_prefill_16(const PrefillLaunch& a, bool f16, cudaStream_t s);

cudaError_t launch_trace_reset(uint64_t* rec, int32_t n, cudaStream_t s);
// The status word inside sws_linear_noalloc's fixed scratch on the current
// device (set up on `s` at the first use on that device).
int noalloc_status_word(int32_t** out, cudaStream_t s);
cudaError_t launch_bounded_wait(int32_t* status, uint64_t limit_ns, cudaStream_t s);

}  // namespace sws

struct sws_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

struct sws_plan {
  int32_t n_shards = 1;
  uint32_t flags = 0;
  std::vector<sws::EntryPlan> entries;
  std::vector<sws::LayerPlan> layers;
  int64_t slot_bytes = 0;
};
