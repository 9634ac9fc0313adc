// Context, linear dispatch and the lookahead slot scheduler.
//
// Scheduler: weight-sharding blog (zdszero.github.io/weight_sharding.html),
// sections "提前一层：lookahead 与 ping-pong slot" and "SGLang 中的实现":
//   pre_dispatch(first): gather the first layer on the side stream;
//   per layer l: maybe_dispatch(l+1) - the side stream waits done(l-1), the
//   gate on the slot that layer l-1 read, then gathers layer l+1 into it and
//   records ready(l+1); the layer waits ready(l) once ("wait_ready_once",
//   section "CUDA graph 与 draft 模型"), runs its linears and records done(l).
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <chrono>
#include <condition_variable>
#include <memory>
#include <new>
#include <thread>

#include "sws_internal.h"

using namespace sws;

namespace sws {

// Process-wide options are atomics: a thread may set one while another is
// inside a call, which then sees the old value or the new one.
namespace {
std::atomic<int> g_host_wait_ms{10000};  // SWS_OPT_HOST_WAIT_MS
}

int host_wait_ms() { return g_host_wait_ms.load(std::memory_order_relaxed); }

int wait_event_deadline(cudaEvent_t ev, const char* what) {
  const auto t0 = std::chrono::steady_clock::now();
  const int wait_ms = host_wait_ms();
  const auto limit = std::chrono::milliseconds(wait_ms);
  for (int spin = 0;; ++spin) {
    const cudaError_t e = cudaEventQuery(ev);
    if (e == cudaSuccess) return SWS_OK;
    if (e != cudaErrorNotReady) return cuda_fail(e, what);
    if (std::chrono::steady_clock::now() - t0 > limit)
      return fail(SWS_E_TIMEOUT, "%s: the device had not reached the event after %d ms (host wait limit)", what,
                  wait_ms);
    if (spin > 64) std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
}

int device_sync_deadline(int device, const char* what) {
  // cudaDeviceSynchronize cannot be polled, so a helper thread makes the call
  // and this thread waits for it with the limit; after a timeout the helper
  // returns by itself once the device has finished the work queued before it.
  struct State {
    std::mutex mu;
    std::condition_variable cv;
    bool done = false;
    cudaError_t err = cudaSuccess;
  };
  auto st = std::make_shared<State>();
  try {
    std::thread([st, device] {
      cudaError_t e = cudaSetDevice(device);
      if (e == cudaSuccess) e = cudaDeviceSynchronize();
      std::lock_guard<std::mutex> lock(st->mu);
      st->err = e;
      st->done = true;
      st->cv.notify_all();
    }).detach();
  } catch (...) {
    return fail(SWS_E_INVALID, "%s: could not start the wait thread", what);
  }
  std::unique_lock<std::mutex> lock(st->mu);
  const int wait_ms = host_wait_ms();
  if (!st->cv.wait_for(lock, std::chrono::milliseconds(wait_ms), [&] { return st->done; }))
    return fail(SWS_E_TIMEOUT, "%s: the device had not finished its queued work after %d ms (host wait limit)", what,
                wait_ms);
  return st->err == cudaSuccess ? SWS_OK : cuda_fail(st->err, what);
}

}  // namespace sws

struct sws_ctx {
  const sws_plan* plan = nullptr;
  int device = 0;
  std::vector<uint8_t*> chunks;  // [n_layers * N]
  uint8_t* slot[2] = {nullptr, nullptr};
  int32_t slot_tag[2] = {-1, -1};
  std::vector<const float*> scales;
  std::vector<const uint8_t*> replicated;
  uint8_t* ws = nullptr;
  int64_t ws_bytes = 0;
  int64_t ws_decode = 0;  // bytes of the decode region at the start of ws
  int64_t ws_scales = 0;  // SWS_SCALES_IN_T: the scale staging area (the workspace's last bytes)
  cudaEvent_t ready[2] = {nullptr, nullptr}, done[2] = {nullptr, nullptr};
  cudaEvent_t call_start = nullptr, join = nullptr;
  // timing of the last SWS_RUN_TIMING run
  std::vector<cudaEvent_t> t_wait, t_begin, t_end;
  int32_t timed_n = 0;
  // device trace records
  uint64_t* trace = nullptr;
  int32_t trace_cap = 0, trace_next = 0;
  // prefill layers: the next linear's activations are quantised on qstream
  // while the current GEMM runs (two workspace buffers)
  cudaStream_t qstream = nullptr;
  cudaEvent_t q_done[2] = {nullptr, nullptr}, g_done[2] = {nullptr, nullptr};
  // layer prefetched into each slot by sws_prefetch_layer and not consumed
  // yet (-1: none), and the event its gather recorded
  int32_t prefetch_layer[2] = {-1, -1};
  cudaEvent_t prefetched[2] = {nullptr, nullptr};
};

namespace {

int32_t* status_word(sws_ctx* c) { return reinterpret_cast<int32_t*>(c->ws); }

uint64_t* next_trace(sws_ctx* c) {
  if (!c->trace || c->trace_next >= c->trace_cap) return nullptr;
  return c->trace + 4 * (int64_t)(c->trace_next++);
}

// Workspace one prefill linear's activations need: E4M3 entries the
// quantiser's xq and ex, F16 entries x rounded to f16; BF16 entries none.
int64_t prefill_bytes(int32_t dtype, int64_t m, int64_t cols) {
  if (m <= 64) return 0;
  if (dtype == SWS_F16) return roundup(2 * m * cols, 256);
  if (dtype != SWS_E4M3) return 0;
  return roundup(m * cols, 256) + roundup(m * cdiv(cols, 128) * 4, 256);
}

// Weight type of a decode group: 0 e4m3 codes with block scales, 1 bf16, 2 f16.
int weight_type(int32_t dtype) { return dtype == SWS_BF16 ? 1 : dtype == SWS_F16 ? 2 : 0; }

int ensure_events(sws_ctx* c, size_t n) {
  while (c->t_wait.size() < n) {
    cudaEvent_t a, b, d;
    SWS_CUDA_TRY(cudaEventCreate(&a));
    SWS_CUDA_TRY(cudaEventCreate(&b));
    SWS_CUDA_TRY(cudaEventCreate(&d));
    c->t_wait.push_back(a);
    c->t_begin.push_back(b);
    c->t_end.push_back(d);
  }
  return SWS_OK;
}

std::atomic<int> g_gather_engine{SWS_GATHER_TMA};

// overlap_prev: launch the kernel with programmatic stream serialisation (see
// launch_gather); only the stand-alone gather call asks for it. Inside
// run_layers the gathers sit behind event waits on the side stream, where it
// gains nothing, and a captured programmatic edge there slowed graph replays.
int gather_impl(sws_ctx* c, int32_t layer, int32_t slot, cudaStream_t s, bool overlap_prev = false) {
  const sws_plan* p = c->plan;
  const LayerPlan& lp = p->layers[layer];
  c->slot_tag[slot] = layer;
  c->prefetch_layer[slot] = -1;  // whatever was prefetched into this slot is overwritten
  if (lp.total == 0) return SWS_OK;
  GatherLaunch g;
  g.n = p->n_shards;
  for (int i = 0; i < g.n; ++i) {
    g.chunks[i] = c->chunks[(int64_t)layer * g.n + i];
    if (!g.chunks[i]) return fail(SWS_E_INVALID, "gather: chunk %d of layer %d is NULL", i, layer);
  }
  g.chunk_bytes = lp.chunk;
  g.dst = c->slot[slot];
  if (check_bounds()) {  // slot[i*C : (i+1)*C] = chunk i, inside the slot's plan.slot_bytes
    std::vector<CopySeg> segs;
    for (int i = 0; i < g.n; ++i) segs.push_back(CopySeg{g.chunks[i], g.dst + (int64_t)i * lp.chunk, lp.chunk});
    std::vector<Extent> srcs;
    for (int i = 0; i < g.n; ++i) srcs.push_back({g.chunks[i], g.chunks[i] + lp.chunk});
    const int rc = check_segments(segs, srcs, {Extent{g.dst, g.dst + p->slot_bytes}}, "gather");
    if (rc != SWS_OK) return rc;
  }
  const int engine = g_gather_engine.load(std::memory_order_relaxed);
  if (engine == SWS_GATHER_COPY_ENGINE) {  // slot[i*C : (i+1)*C] = chunk i, by the copy engines
    for (int i = 0; i < g.n; ++i) {
      cudaError_t e = cudaMemcpyAsync(g.dst + (int64_t)i * lp.chunk, g.chunks[i], (size_t)lp.chunk,
                                      cudaMemcpyDeviceToDevice, s);
      if (e != cudaSuccess) return cuda_fail(e, "gather: cudaMemcpyAsync");
    }
    return SWS_OK;
  }
  g.status = status_word(c);
  g.trace = next_trace(c);
  g.tag = (kTraceGather << 56) | ((uint64_t)layer << 32) | (uint64_t)(uint32_t)slot;
  g.shared_sm = engine == SWS_GATHER_TMA_SHARED_SM;
  g.overlap_prev = overlap_prev;
  cudaError_t e = launch_gather(g, s);
  return e == cudaSuccess ? SWS_OK : cuda_fail(e, "gather kernel launch");
}

// Layer `layer` in slot `slot` for work on `s`: if sws_prefetch_layer left it
// there, `s` waits for that gather once; otherwise (cold start) `s` waits for
// the slot's last reader and gathers inline. *cold tells which.
int take_prefetch(sws_ctx* c, int32_t layer, int32_t slot, cudaStream_t s, bool* cold) {
  if (c->prefetch_layer[slot] == layer) {
    *cold = false;
    c->prefetch_layer[slot] = -1;
    SWS_CUDA_TRY(cudaStreamWaitEvent(s, c->prefetched[slot], 0));
    return SWS_OK;
  }
  *cold = true;
  SWS_CUDA_TRY(cudaStreamWaitEvent(s, c->done[slot], 0));
  return gather_impl(c, layer, slot, s);
}

// Where entry j's weight lives for source `src`: a view (slot or replicated
// buffer) or, for the fused source, the chunks of its layer.
int weight_source(sws_ctx* c, int32_t j, int32_t src, const uint8_t** w, bool* fused) {
  const EntryPlan& e = c->plan->entries[j];
  *w = nullptr;
  *fused = false;
  if (!e.sharded) {
    *w = c->replicated[j];
    if (!*w) return fail(SWS_E_INVALID, "linear: replicated entry %d has no buffer", j);
  } else if (src == SWS_SRC_SLOT0 || src == SWS_SRC_SLOT1) {
    if (c->slot_tag[src] != e.layer)
      return fail(SWS_E_STATE, "linear: slot %d holds layer %d, entry %d belongs to layer %d", src, c->slot_tag[src], j,
                  e.layer);
    *w = c->slot[src] + e.offset;
  } else if (src == SWS_SRC_FUSED) {
    *fused = true;
  } else {
    return fail(SWS_E_INVALID, "linear: src=%d", src);
  }
  return SWS_OK;
}

// Where entry j's block scales live for source `src`: the caller's replicated
// buffer, or - with SWS_SCALES_IN_T - T itself: the slot that holds the
// weight, or the workspace copy staged from the chunks (stage_scales) for the
// chunk-map source.
const float* scale_source(sws_ctx* c, int32_t j, int32_t src) {
  const EntryPlan& e = c->plan->entries[j];
  if (e.scale_offset < 0) return c->scales[j];
  if (src == SWS_SRC_FUSED) return reinterpret_cast<const float*>(c->ws + c->ws_scales + e.scale_stage);
  return reinterpret_cast<const float*>(c->slot[src] + e.scale_offset);
}

// SWS_SCALES_IN_T, chunk-map source: copies the layer's scale regions from its
// chunks into the workspace staging area, on `s` before the linears that read
// them (T bytes [o, o + size) of each scale entry, cut at chunk boundaries).
int stage_scales(sws_ctx* c, int32_t layer, cudaStream_t s) {
  const sws_plan* p = c->plan;
  const LayerPlan& lp = p->layers[layer];
  if (lp.scale_stage_bytes == 0) return SWS_OK;
  void* const* chunks = reinterpret_cast<void* const*>(&c->chunks[(size_t)layer * p->n_shards]);
  std::vector<CopySeg> segs;
  for (int32_t j : lp.sharded) {
    const EntryPlan& e = p->entries[j];
    if (e.scale_offset < 0 || e.scale_bytes == 0) continue;
    chunk_segments(e.scale_offset, e.scale_offset + e.scale_bytes, lp.chunk, chunks, nullptr,
                   c->ws + c->ws_scales + e.scale_stage, &segs);
  }
  if (check_bounds()) {  // chunks -> the workspace's staging area (its last bytes)
    const int rc = check_segments(segs, chunk_extents(chunks, p->n_shards, lp.chunk),
                                  {Extent{c->ws + c->ws_scales, c->ws + c->ws_bytes}}, "linear: scale staging");
    if (rc != SWS_OK) return rc;
  }
  const cudaError_t ce = launch_relayout(segs, s);
  return ce == cudaSuccess ? SWS_OK : cuda_fail(ce, "linear: scale staging kernel");
}

int check_linear_args(sws_ctx* c, int32_t j, const void* x, int64_t m, void* y) {
  const sws_plan* p = c->plan;
  if (j < 0 || j >= (int32_t)p->entries.size()) return fail(SWS_E_INVALID, "linear: entry %d", j);
  const EntryPlan& e = p->entries[j];
  if (e.dtype != SWS_E4M3 && e.dtype != SWS_BF16 && e.dtype != SWS_F16)
    return fail(SWS_E_UNSUPPORTED, "linear: entry %d is not E4M3, BF16 or F16", j);
  if (m < 0 || m >= ((int64_t)1 << 31)) return fail(SWS_E_INVALID, "linear: m=%lld", (long long)m);
  if (m == 0 || e.rows == 0) return SWS_OK;
  if (!x || !y) return fail(SWS_E_INVALID, "linear: x or y is NULL");
  if (!aligned16(x) || !aligned16(y)) return fail(SWS_E_ALIGN, "linear: x or y is not 16-byte aligned");
  if (e.dtype == SWS_E4M3 && !c->scales[j] && e.scale_offset < 0)
    return fail(SWS_E_INVALID, "linear: entry %d has no scales", j);
  if (e.cols % 16 != 0) return fail(SWS_E_UNSUPPORTED, "linear: cols=%lld is not a multiple of 16", (long long)e.cols);
  return SWS_OK;
}

void init_group(sws_ctx* c, DecodeGroup& g, int32_t layer, int64_t m, bool fused) {
  const sws_plan* p = c->plan;
  g.n = 0;
  g.m = m;
  g.fused = fused;
  for (int i = 0; i < 256; ++i) g.chunks[i] = nullptr;
  g.n_chunks = 0;
  if (fused) {
    g.n_chunks = p->n_shards;
    for (int i = 0; i < p->n_shards; ++i) g.chunks[i] = c->chunks[(int64_t)layer * p->n_shards + i];
  }
  g.chunk_bytes = p->layers[layer].chunk;
  g.workspace = c->ws;
  g.workspace_bytes = c->ws_decode;
}

int launch_group(sws_ctx* c, DecodeGroup& g, int32_t layer, int32_t first_entry, cudaStream_t s) {
  if (g.n == 0) return SWS_OK;
  if (g.fused)
    for (int i = 0; i < g.n_chunks; ++i)
      if (!g.chunks[i]) return fail(SWS_E_INVALID, "linear: chunk %d of layer %d is NULL", i, layer);
  g.trace = next_trace(c);
  g.tag = (kTraceLinear << 56) | ((uint64_t)layer << 32) | (uint64_t)(uint32_t)first_entry;
  int rc = launch_decode(g, s);
  g.n = 0;
  return rc;
}

// Activations of a prefill linear in the workspace: for E4M3 weights the
// quantiser's xq [m, cols] then ex [m, cols/128]; for F16 weights x as f16
// [m, cols] at xq.
struct PrefillBuf {
  uint8_t* xq;
  float* ex;
};
PrefillBuf prefill_buf(sws_ctx* c, int b, int64_t per_buf, int64_t m, int64_t cols) {
  PrefillBuf r;
  r.xq = c->ws + c->ws_decode + b * per_buf;
  r.ex = reinterpret_cast<float*>(r.xq + roundup(m * cols, 256));
  return r;
}

int prefill_gemm(sws_ctx* c, int32_t j, int32_t src, const uint8_t* w, const PrefillBuf& q, int64_t m, void* y,
                 cudaStream_t s) {
  const EntryPlan& e = c->plan->entries[j];
  PrefillLaunch pl;
  pl.w = w;
  pl.scales = scale_source(c, j, src);
  pl.xq = q.xq;
  pl.ex = q.ex;
  pl.y = static_cast<uint16_t*>(y);
  pl.m = m;
  pl.rows = e.rows;
  pl.cols = e.cols;
  pl.status = status_word(c);
  pl.trace = next_trace(c);
  pl.tag = (kTraceLinear << 56) | (kTracePrefill << 48) | ((uint64_t)e.layer << 32) | (uint64_t)(uint32_t)j;
  return launch_prefill(pl, s);
}

// 16-bit weights at prefill sizes: no quantiser, the activations (bf16 as
// given, or already rounded to f16 for f16 weights) feed the tensor cores.
int prefill_linear_16(sws_ctx* c, int32_t j, const uint8_t* w, const void* x, int64_t m, void* y, cudaStream_t s) {
  const EntryPlan& e = c->plan->entries[j];
  PrefillLaunch pl;
  pl.w = w;
  pl.scales = nullptr;
  pl.xq = static_cast<const uint8_t*>(x);
  pl.ex = nullptr;
  pl.y = static_cast<uint16_t*>(y);
  pl.m = m;
  pl.rows = e.rows;
  pl.cols = e.cols;
  pl.status = status_word(c);
  pl.trace = next_trace(c);
  pl.tag = (kTraceLinear << 56) | (kTracePrefill << 48) | ((uint64_t)e.layer << 32) | (uint64_t)(uint32_t)j;
  return launch_prefill_16(pl, e.dtype == SWS_F16, s);
}

int prefill_linear(sws_ctx* c, int32_t j, int32_t src, const uint8_t* w, const void* x, int64_t m, void* y,
                   cudaStream_t s) {
  const EntryPlan& e = c->plan->entries[j];
  if (e.dtype == SWS_BF16) return prefill_linear_16(c, j, w, x, m, y, s);
  if (e.dtype == SWS_E4M3 && e.cols % 128 != 0)
    return fail(SWS_E_UNSUPPORTED, "linear: prefill needs cols %% 128 == 0");
  const int64_t need = c->ws_decode + prefill_bytes(e.dtype, m, e.cols);
  if (c->ws_bytes < need)
    return fail(SWS_E_WORKSPACE, "linear: workspace %lld < %lld bytes for m=%lld", (long long)c->ws_bytes,
                (long long)need, (long long)m);
  const PrefillBuf q = prefill_buf(c, 0, 0, m, e.cols);
  if (e.dtype == SWS_F16) {
    int rc = launch_to_f16(static_cast<const uint16_t*>(x), m * e.cols, reinterpret_cast<uint16_t*>(q.xq), s);
    if (rc != SWS_OK) return rc;
    return prefill_linear_16(c, j, w, q.xq, m, y, s);
  }
  int rc = launch_quantize_x(static_cast<const uint16_t*>(x), m, e.cols, q.xq, q.ex, s);
  if (rc != SWS_OK) return rc;
  return prefill_gemm(c, j, src, w, q, m, y, s);
}

int linear_impl(sws_ctx* c, int32_t j, int32_t src, const void* x, int64_t m, void* y, cudaStream_t s);

// A prefill layer: the q-th E4M3 linear's activations are quantised (the q-th
// F16 linear's rounded to f16) on the context's side stream into buffer q % 2
// while the previous GEMM runs on `s`; GEMM q waits for its quantiser, and
// quantiser q waits for GEMM q - 2, the last reader of its buffer. BF16
// linears need neither and run on `s` in order. Without room for two buffers
// the linears run one after another.
int prefill_layer(sws_ctx* c, const LayerPlan& lp, int32_t src, const sws_layer_io& io, cudaStream_t s) {
  const int64_t m = io.m;
  int64_t per_buf = 0;
  int n_q = 0;  // linears whose activations go through the side stream
  for (int32_t j : lp.all) {
    const EntryPlan& e = c->plan->entries[j];
    if (e.dtype != SWS_E4M3 && e.dtype != SWS_F16) continue;
    if (e.dtype == SWS_E4M3 && e.cols % 128 != 0)
      return fail(SWS_E_UNSUPPORTED, "linear: prefill needs cols %% 128 == 0");
    per_buf = std::max(per_buf, prefill_bytes(e.dtype, m, e.cols));
    ++n_q;
  }
  if (n_q < 2 || c->ws_bytes < c->ws_decode + 2 * per_buf) {
    for (size_t k = 0; k < lp.all.size(); ++k) {
      int rc = linear_impl(c, lp.all[k], src, io.x[k], m, io.y[k], s);
      if (rc != SWS_OK) return rc;
    }
    return SWS_OK;
  }
  cudaError_t ce = cudaEventRecord(c->call_start, s);  // the activations are ready in s's order
  if (ce == cudaSuccess) ce = cudaStreamWaitEvent(c->qstream, c->call_start, 0);
  if (ce != cudaSuccess) return cuda_fail(ce, "prefill layer: stream order");
  int qi = 0;  // E4M3 and F16 linears so far
  for (size_t k = 0; k < lp.all.size(); ++k) {
    const int32_t j = lp.all[k];
    int rc = check_linear_args(c, j, io.x[k], m, io.y[k]);
    if (rc != SWS_OK) return rc;
    const EntryPlan& e = c->plan->entries[j];
    if (e.rows == 0) continue;
    const uint8_t* w = nullptr;
    bool fused = false;
    rc = weight_source(c, j, src, &w, &fused);
    if (rc != SWS_OK) return rc;
    if (fused) return fail(SWS_E_UNSUPPORTED, "linear: the fused source is for decode (m <= 64)");
    if (e.dtype == SWS_BF16) {
      rc = prefill_linear_16(c, j, w, io.x[k], m, io.y[k], s);
      if (rc != SWS_OK) return rc;
      continue;
    }
    const int b = qi & 1;
    const PrefillBuf q = prefill_buf(c, b, per_buf, m, e.cols);
    if (qi >= 2 && (ce = cudaStreamWaitEvent(c->qstream, c->g_done[b], 0)) != cudaSuccess)
      return cuda_fail(ce, "prefill layer: wait");
    ++qi;
    const bool f16 = e.dtype == SWS_F16;
    rc = f16 ? launch_to_f16(static_cast<const uint16_t*>(io.x[k]), m * e.cols, reinterpret_cast<uint16_t*>(q.xq),
                             c->qstream)
             : launch_quantize_x(static_cast<const uint16_t*>(io.x[k]), m, e.cols, q.xq, q.ex, c->qstream);
    if (rc != SWS_OK) return rc;
    if ((ce = cudaEventRecord(c->q_done[b], c->qstream)) != cudaSuccess ||
        (ce = cudaStreamWaitEvent(s, c->q_done[b], 0)) != cudaSuccess)
      return cuda_fail(ce, "prefill layer: quantiser order");
    rc = f16 ? prefill_linear_16(c, j, w, q.xq, m, io.y[k], s) : prefill_gemm(c, j, src, w, q, m, io.y[k], s);
    if (rc != SWS_OK) return rc;
    if ((ce = cudaEventRecord(c->g_done[b], s)) != cudaSuccess) return cuda_fail(ce, "prefill layer: record");
  }
  return SWS_OK;
}

int linear_impl(sws_ctx* c, int32_t j, int32_t src, const void* x, int64_t m, void* y, cudaStream_t s) {
  int rc = check_linear_args(c, j, x, m, y);
  if (rc != SWS_OK) return rc;
  const EntryPlan& e = c->plan->entries[j];
  if (m == 0 || e.rows == 0) return SWS_OK;
  const uint8_t* w = nullptr;
  bool fused = false;
  rc = weight_source(c, j, src, &w, &fused);
  if (rc != SWS_OK) return rc;
  if (m > 64) {
    if (fused) return fail(SWS_E_UNSUPPORTED, "linear: the fused source is for decode (m <= 64)");
    return prefill_linear(c, j, src, w, x, m, y, s);
  }
  if (fused && e.scale_offset >= 0) {
    rc = stage_scales(c, e.layer, s);
    if (rc != SWS_OK) return rc;
  }
  DecodeGroup g;
  init_group(c, g, e.layer, m, fused);
  g.wtype = weight_type(e.dtype);
  g.item[g.n++] = DecodeItem{w, scale_source(c, j, src), static_cast<const uint16_t*>(x), static_cast<uint16_t*>(y),
                             e.rows, e.cols, e.offset};
  return launch_group(c, g, e.layer, j, s);
}

// All linears of a layer: decode-sized ones go out as grouped launches, one
// group per (views by TMA or chunk-map reads) x (E4M3, BF16 or F16 weights),
// up to kMaxDecodeGroup per launch.
int layer_linears(sws_ctx* c, int32_t layer, int32_t src, const sws_layer_io& io, cudaStream_t s) {
  const LayerPlan& lp = c->plan->layers[layer];
  if (lp.all.empty()) return SWS_OK;
  if (!io.x || !io.y) return fail(SWS_E_INVALID, "run_layers: io of layer %d has NULL arrays", layer);
  const int64_t m = io.m;
  if (m > 64) return prefill_layer(c, lp, src, io, s);
  if (m > 0 && src == SWS_SRC_FUSED) {  // scales in T read through the chunk map: staged once for the layer
    int rc = stage_scales(c, layer, s);
    if (rc != SWS_OK) return rc;
  }
  constexpr int kGroups = 6;  // index: fused * 3 + weight type
  DecodeGroup grp[kGroups];
  int32_t first[kGroups] = {-1, -1, -1, -1, -1, -1};
  for (int q = 0; q < kGroups; ++q) {
    init_group(c, grp[q], layer, m, q >= 3);
    grp[q].wtype = q % 3;
  }
  for (size_t k = 0; k < lp.all.size(); ++k) {
    const int32_t j = lp.all[k];
    int rc = check_linear_args(c, j, io.x[k], m, io.y[k]);
    if (rc != SWS_OK) return rc;
    const EntryPlan& e = c->plan->entries[j];
    if (m == 0 || e.rows == 0) continue;
    const uint8_t* w = nullptr;
    bool fused = false;
    rc = weight_source(c, j, src, &w, &fused);
    if (rc != SWS_OK) return rc;
    const int q = (fused ? 3 : 0) + weight_type(e.dtype);
    DecodeGroup& g = grp[q];
    if (g.n == kMaxDecodeGroup) {
      rc = launch_group(c, g, layer, first[q], s);
      if (rc != SWS_OK) return rc;
    }
    if (g.n == 0) first[q] = j;
    g.item[g.n++] = DecodeItem{w, scale_source(c, j, src), static_cast<const uint16_t*>(io.x[k]),
                               static_cast<uint16_t*>(io.y[k]), e.rows, e.cols, e.offset};
  }
  for (int q = 0; q < kGroups; ++q) {
    int rc = launch_group(c, grp[q], layer, first[q], s);
    if (rc != SWS_OK) return rc;
  }
  return SWS_OK;
}

// Activation split region of the tcgen05 decode path: enough for the largest
// layer (all of a layer's linears in one launch).
int64_t split_region_bytes(const sws_plan* p, int64_t m) {
  int64_t most = 0;
  for (const LayerPlan& l : p->layers) {
    int64_t slabs = 0;
    for (int32_t j : l.all) slabs += cdiv(p->entries[j].cols, 128);
    most = std::max(most, slabs);
  }
  return decode_split_bytes(m, most);
}

// SWS_SCALES_IN_T: staging area for the chunk-map source, the largest layer's.
int64_t scale_stage_region_bytes(const sws_plan* p) {
  int64_t most = 0;
  for (const LayerPlan& l : p->layers) most = std::max(most, l.scale_stage_bytes);
  return roundup(most, 256);
}

}  // namespace

extern "C" {

int64_t sws_workspace_bytes(const sws_plan* p, int64_t max_m) {
  if (!p || max_m < 0) return -1;
  const int64_t mm = std::min<int64_t>(std::max<int64_t>(max_m, 1), 64);
  int64_t dec = 0;
  if (decode_workspace_bytes(mm, &dec) != SWS_OK) return -1;
  int64_t pre = 0;
  for (const EntryPlan& e : p->entries)
    pre = std::max(pre, prefill_bytes(e.dtype, max_m, e.cols));
  // two prefill buffers: quantiser k + 1 beside GEMM k; the scale staging
  // area (chunk-map decode only, never in use beside a prefill linear) last
  return dec + split_region_bytes(p, mm) + 2 * pre + scale_stage_region_bytes(p);
}

int sws_ctx_create(const sws_plan* plan, void* const* chunks, void* slot0, void* slot1, const float* const* scales,
                   const void* const* replicated, void* workspace, int64_t workspace_bytes, sws_ctx** out) {
  if (!out) return fail(SWS_E_INVALID, "ctx_create: out is NULL");
  *out = nullptr;
  if (!plan) return fail(SWS_E_INVALID, "ctx_create: plan is NULL");
  int rc = check_device();
  if (rc != SWS_OK) return rc;
  const int32_t n = plan->n_shards, L = (int32_t)plan->layers.size(), E = (int32_t)plan->entries.size();
  if (L > 0 && !chunks) return fail(SWS_E_INVALID, "ctx_create: chunks is NULL");
  for (int32_t l = 0; l < L; ++l)
    for (int32_t i = 0; i < n; ++i) {
      void* ptr = chunks[(int64_t)l * n + i];
      if (plan->layers[l].total > 0 && !ptr) return fail(SWS_E_INVALID, "ctx_create: chunk (%d, %d) is NULL", l, i);
      if (ptr && !aligned16(ptr)) return fail(SWS_E_ALIGN, "ctx_create: chunk (%d, %d) is not 16-byte aligned", l, i);
    }
  if (plan->slot_bytes > 0 && (!slot0 || !slot1)) return fail(SWS_E_INVALID, "ctx_create: a slot is NULL");
  if (!aligned16(slot0) || !aligned16(slot1)) return fail(SWS_E_ALIGN, "ctx_create: slot not 16-byte aligned");
  if (E > 0 && !scales) return fail(SWS_E_INVALID, "ctx_create: scales is NULL");
  for (int32_t j = 0; j < E; ++j) {
    if (plan->entries[j].dtype == SWS_E4M3 && !scales[j] && plan->entries[j].scale_offset < 0)
      return fail(SWS_E_INVALID, "ctx_create: E4M3 entry %d has no scales", j);
    if (scales[j] && !aligned16(scales[j])) return fail(SWS_E_ALIGN, "ctx_create: scales of entry %d unaligned", j);
    if (!plan->entries[j].sharded) {
      const void* r = replicated ? replicated[j] : nullptr;
      if (r && !aligned16(r)) return fail(SWS_E_ALIGN, "ctx_create: replicated buffer of entry %d unaligned", j);
    }
  }
  const int64_t need = sws_workspace_bytes(plan, 1);
  if (!workspace || workspace_bytes < need)
    return fail(SWS_E_WORKSPACE, "ctx_create: workspace %lld < %lld bytes", (long long)workspace_bytes,
                (long long)need);
  if (!aligned16(workspace)) return fail(SWS_E_ALIGN, "ctx_create: workspace not 16-byte aligned");
  sws_ctx* c = new (std::nothrow) sws_ctx();
  if (!c) return fail(SWS_E_INVALID, "ctx_create: out of host memory");
  c->plan = plan;
  cudaGetDevice(&c->device);
  c->chunks.assign((size_t)L * n, nullptr);
  for (int64_t i = 0; i < (int64_t)L * n; ++i) c->chunks[i] = static_cast<uint8_t*>(chunks[i]);
  c->slot[0] = static_cast<uint8_t*>(slot0);
  c->slot[1] = static_cast<uint8_t*>(slot1);
  c->scales.assign(E, nullptr);
  c->replicated.assign(E, nullptr);
  for (int32_t j = 0; j < E; ++j) {
    c->scales[j] = scales[j];
    if (replicated && !plan->entries[j].sharded) c->replicated[j] = static_cast<const uint8_t*>(replicated[j]);
  }
  c->ws = static_cast<uint8_t*>(workspace);
  c->ws_bytes = workspace_bytes;
  int64_t dec64 = 0;
  decode_workspace_bytes(64, &dec64);
  // The scale staging area (SWS_SCALES_IN_T) is the workspace's last bytes:
  // decode launches for every m the workspace was sized for end before it.
  c->ws_scales = (workspace_bytes - scale_stage_region_bytes(plan)) & ~int64_t(15);
  c->ws_decode = std::min(dec64 + split_region_bytes(plan, 64), c->ws_scales);
  // Only the status word and the split-K arrival counters must start at zero.
  cudaError_t e = cudaMemset(workspace, 0, (size_t)(kCtlBytes + kMaxCounters * 4));
  if (e != cudaSuccess) {
    delete c;
    return cuda_fail(e, "ctx_create: cudaMemset(workspace)");
  }
  for (int s = 0; s < 2; ++s) {
    if ((e = cudaEventCreateWithFlags(&c->ready[s], cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&c->done[s], cudaEventDisableTiming)) != cudaSuccess) {
      sws_ctx_destroy(c);
      return cuda_fail(e, "ctx_create: cudaEventCreate");
    }
  }
  if ((e = cudaEventCreateWithFlags(&c->call_start, cudaEventDisableTiming)) != cudaSuccess ||
      (e = cudaEventCreateWithFlags(&c->join, cudaEventDisableTiming)) != cudaSuccess ||
      (e = cudaEventCreateWithFlags(&c->prefetched[0], cudaEventDisableTiming)) != cudaSuccess ||
      (e = cudaEventCreateWithFlags(&c->prefetched[1], cudaEventDisableTiming)) != cudaSuccess) {
    sws_ctx_destroy(c);
    return cuda_fail(e, "ctx_create: cudaEventCreate");
  }
  for (int b = 0; b < 2; ++b)
    if ((e = cudaEventCreateWithFlags(&c->q_done[b], cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&c->g_done[b], cudaEventDisableTiming)) != cudaSuccess) {
      sws_ctx_destroy(c);
      return cuda_fail(e, "ctx_create: cudaEventCreate");
    }
  if ((e = cudaStreamCreateWithFlags(&c->qstream, cudaStreamNonBlocking)) != cudaSuccess) {
    sws_ctx_destroy(c);
    return cuda_fail(e, "ctx_create: cudaStreamCreate");
  }
  *out = c;
  return SWS_OK;
}

void sws_ctx_destroy(sws_ctx* c) {
  if (!c) return;
  for (int s = 0; s < 2; ++s) {
    if (c->ready[s]) cudaEventDestroy(c->ready[s]);
    if (c->done[s]) cudaEventDestroy(c->done[s]);
  }
  if (c->call_start) cudaEventDestroy(c->call_start);
  if (c->join) cudaEventDestroy(c->join);
  for (int s = 0; s < 2; ++s)
    if (c->prefetched[s]) cudaEventDestroy(c->prefetched[s]);
  for (int b = 0; b < 2; ++b) {
    if (c->q_done[b]) cudaEventDestroy(c->q_done[b]);
    if (c->g_done[b]) cudaEventDestroy(c->g_done[b]);
  }
  if (c->qstream) cudaStreamDestroy(c->qstream);
  for (size_t i = 0; i < c->t_wait.size(); ++i) {
    cudaEventDestroy(c->t_wait[i]);
    cudaEventDestroy(c->t_begin[i]);
    cudaEventDestroy(c->t_end[i]);
  }
  delete c;
}

int sws_gather_to_slot(sws_ctx* c, int32_t layer, int32_t slot, sws_stream_t stream) {
  if (!c) return fail(SWS_E_INVALID, "gather_to_slot: ctx is NULL");
  if (layer < 0 || layer >= (int32_t)c->plan->layers.size()) return fail(SWS_E_INVALID, "gather_to_slot: layer %d", layer);
  if (slot != 0 && slot != 1) return fail(SWS_E_INVALID, "gather_to_slot: slot %d", slot);
  return gather_impl(c, layer, slot, (cudaStream_t)stream, /*overlap_prev=*/true);
}

int sws_linear(sws_ctx* c, int32_t entry, int32_t src, const void* x, int64_t m, void* y, sws_stream_t stream) {
  if (!c) return fail(SWS_E_INVALID, "linear: ctx is NULL");
  return linear_impl(c, entry, src, x, m, y, (cudaStream_t)stream);
}

int sws_layer_linears(sws_ctx* c, int32_t layer, int32_t src, const sws_layer_io* io, sws_stream_t stream) {
  if (!c) return fail(SWS_E_INVALID, "layer_linears: ctx is NULL");
  if (layer < 0 || layer >= (int32_t)c->plan->layers.size())
    return fail(SWS_E_INVALID, "layer_linears: layer %d", layer);
  if (!io) return fail(SWS_E_INVALID, "layer_linears: io is NULL");
  return layer_linears(c, layer, src, *io, (cudaStream_t)stream);
}

int sws_run_layers(sws_ctx* c, int32_t first, int32_t last, const sws_layer_io* io, uint32_t flags,
                   sws_stream_t main_s, sws_stream_t side_s) {
  if (!c) return fail(SWS_E_INVALID, "run_layers: ctx is NULL");
  const int32_t L = (int32_t)c->plan->layers.size();
  if (last < first) return SWS_OK;
  if (first < 0 || last >= L) return fail(SWS_E_INVALID, "run_layers: range [%d, %d] outside [0, %d)", first, last, L);
  if (!io) return fail(SWS_E_INVALID, "run_layers: io is NULL");
  if (flags & ~(SWS_RUN_FUSED | SWS_RUN_TIMING | SWS_RUN_FIRST_PREFETCHED))
    return fail(SWS_E_INVALID, "run_layers: flags 0x%x", flags);
  if ((flags & SWS_RUN_FUSED) && (flags & SWS_RUN_FIRST_PREFETCHED))
    return fail(SWS_E_INVALID, "run_layers: SWS_RUN_FIRST_PREFETCHED needs the slot path");
  cudaStream_t ms = (cudaStream_t)main_s, ss = (cudaStream_t)side_s;
  const bool timing = (flags & SWS_RUN_TIMING) != 0;
  const int32_t n = last - first + 1;
  if (timing) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    SWS_CUDA_TRY(cudaStreamIsCapturing(ms, &cap));
    if (cap != cudaStreamCaptureStatusNone)
      return fail(SWS_E_INVALID, "run_layers: SWS_RUN_TIMING records timing events and cannot be captured");
    int rc = ensure_events(c, (size_t)n);
    if (rc != SWS_OK) return rc;
    c->timed_n = n;
  } else {
    c->timed_n = 0;
  }
  if (flags & SWS_RUN_FUSED) {
    for (int32_t l = first; l <= last; ++l) {
      if (timing) {
        SWS_CUDA_TRY(cudaEventRecord(c->t_wait[l - first], ms));
        SWS_CUDA_TRY(cudaEventRecord(c->t_begin[l - first], ms));
      }
      int rc = layer_linears(c, l, SWS_SRC_FUSED, io[l - first], ms);
      if (rc != SWS_OK) return rc;
      if (timing) SWS_CUDA_TRY(cudaEventRecord(c->t_end[l - first], ms));
    }
    return SWS_OK;
  }
  if (ss == ms) return fail(SWS_E_INVALID, "run_layers: main and side streams must differ");
  auto slot_of = [&](int32_t l) { return (l - first) & 1; };
  // pre_dispatch(first): the side stream starts after work already on main.
  SWS_CUDA_TRY(cudaEventRecord(c->call_start, ms));
  if (timing) SWS_CUDA_TRY(cudaEventRecord(c->t_wait[0], ms));
  SWS_CUDA_TRY(cudaStreamWaitEvent(ss, c->call_start, 0));
  int rc = SWS_OK;
  if (flags & SWS_RUN_FIRST_PREFETCHED) {  // blog "CUDA graph 与 draft 模型": the first layer was prefetched
    bool cold = false;
    rc = take_prefetch(c, first, slot_of(first), ss, &cold);
  } else {
    rc = gather_impl(c, first, slot_of(first), ss);
  }
  if (rc != SWS_OK) return rc;
  SWS_CUDA_TRY(cudaEventRecord(c->ready[slot_of(first)], ss));
  for (int32_t l = first; l <= last; ++l) {
    const int32_t nxt = l + 1;
    if (nxt <= last) {  // maybe_dispatch(l + 1)
      if (l - 1 >= first) SWS_CUDA_TRY(cudaStreamWaitEvent(ss, c->done[slot_of(l - 1)], 0));
      rc = gather_impl(c, nxt, slot_of(nxt), ss);
      if (rc != SWS_OK) return rc;
      SWS_CUDA_TRY(cudaEventRecord(c->ready[slot_of(nxt)], ss));
    }
    if (timing && l > first) SWS_CUDA_TRY(cudaEventRecord(c->t_wait[l - first], ms));
    SWS_CUDA_TRY(cudaStreamWaitEvent(ms, c->ready[slot_of(l)], 0));  // wait once
    if (timing) SWS_CUDA_TRY(cudaEventRecord(c->t_begin[l - first], ms));
    rc = layer_linears(c, l, slot_of(l), io[l - first], ms);
    if (rc != SWS_OK) return rc;
    if (timing) SWS_CUDA_TRY(cudaEventRecord(c->t_end[l - first], ms));
    SWS_CUDA_TRY(cudaEventRecord(c->done[slot_of(l)], ms));  // update_done_event(l)
  }
  SWS_CUDA_TRY(cudaEventRecord(c->join, ss));
  SWS_CUDA_TRY(cudaStreamWaitEvent(ms, c->join, 0));
  return SWS_OK;
}

int sws_graph_capture(sws_ctx* c, int32_t first, int32_t last, const sws_layer_io* io, uint32_t flags,
                      sws_stream_t main_s, sws_stream_t side_s, sws_graph** out) {
  if (!out) return fail(SWS_E_INVALID, "graph_capture: out is NULL");
  *out = nullptr;
  if (!c) return fail(SWS_E_INVALID, "graph_capture: ctx is NULL");
  if (flags & (SWS_RUN_TIMING | SWS_RUN_FIRST_PREFETCHED))
    return fail(SWS_E_INVALID, "graph_capture: SWS_RUN_TIMING and SWS_RUN_FIRST_PREFETCHED are eager-only");
  cudaStream_t ms = (cudaStream_t)main_s;
  if (!ms) return fail(SWS_E_INVALID, "graph_capture: the legacy default stream cannot capture");
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  SWS_CUDA_TRY(cudaStreamIsCapturing(ms, &cap));
  if (cap != cudaStreamCaptureStatusNone) return fail(SWS_E_STATE, "graph_capture: main is already capturing");
  // Host-side bookkeeping runs in issue order, but nothing captured has run:
  // on failure it is put back; on success the slots' layers are unknown until
  // the next gather (a launch of the graph leaves them as the capture did).
  const int32_t tag0 = c->slot_tag[0], tag1 = c->slot_tag[1];
  const int32_t pre0 = c->prefetch_layer[0], pre1 = c->prefetch_layer[1];
  const int32_t trace_next = c->trace_next;
  auto restore = [&] {
    c->slot_tag[0] = tag0;
    c->slot_tag[1] = tag1;
    c->prefetch_layer[0] = pre0;
    c->prefetch_layer[1] = pre1;
    c->trace_next = trace_next;
  };
  SWS_CUDA_TRY(cudaStreamBeginCapture(ms, cudaStreamCaptureModeThreadLocal));
  const int rc = sws_run_layers(c, first, last, io, flags, main_s, side_s);
  cudaGraph_t g = nullptr;
  const cudaError_t ee = cudaStreamEndCapture(ms, &g);  // always ends it, so `main` is usable again
  if (rc != SWS_OK || ee != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    restore();
    return rc != SWS_OK ? rc : cuda_fail(ee, "graph_capture: cudaStreamEndCapture");
  }
  c->slot_tag[0] = c->slot_tag[1] = -1;
  cudaGraphExec_t x = nullptr;
  const cudaError_t ie = cudaGraphInstantiateWithFlags(&x, g, cudaGraphInstantiateFlagUseNodePriority);
  if (ie != cudaSuccess) {
    cudaGraphDestroy(g);
    restore();
    return cuda_fail(ie, "graph_capture: cudaGraphInstantiateWithFlags");
  }
  sws_graph* h = new (std::nothrow) sws_graph;
  if (!h) {
    cudaGraphExecDestroy(x);
    cudaGraphDestroy(g);
    return fail(SWS_E_INVALID, "graph_capture: out of host memory");
  }
  h->graph = g;
  h->exec = x;
  *out = h;
  return SWS_OK;
}

int sws_graph_launch(sws_graph* g, sws_stream_t stream) {
  if (!g) return fail(SWS_E_INVALID, "graph_launch: graph is NULL");
  SWS_CUDA_TRY(cudaGraphLaunch(g->exec, (cudaStream_t)stream));
  return SWS_OK;
}

void sws_graph_destroy(sws_graph* g) {
  if (!g) return;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  delete g;
}

int sws_run_timing(sws_ctx* c, float* exposed_ms, float* layer_ms, int32_t n) {
  if (!c) return fail(SWS_E_INVALID, "run_timing: ctx is NULL");
  if (c->timed_n == 0) return fail(SWS_E_STATE, "run_timing: the last run had no SWS_RUN_TIMING");
  if (n < c->timed_n) return fail(SWS_E_INVALID, "run_timing: n=%d < %d layers", n, c->timed_n);
  const int rc = wait_event_deadline(c->t_end[c->timed_n - 1], "run_timing");
  if (rc != SWS_OK) return rc;
  for (int32_t i = 0; i < c->timed_n; ++i) {
    float a = 0.f, b = 0.f;
    SWS_CUDA_TRY(cudaEventElapsedTime(&a, c->t_wait[i], c->t_begin[i]));
    SWS_CUDA_TRY(cudaEventElapsedTime(&b, c->t_begin[i], c->t_end[i]));
    if (exposed_ms) exposed_ms[i] = a;
    if (layer_ms) layer_ms[i] = b;
  }
  return SWS_OK;
}

int sws_quantize_x(const void* x, int64_t m, int64_t k, void* xq, float* ex, sws_stream_t stream) {
  return launch_quantize_x(static_cast<const uint16_t*>(x), m, k, static_cast<uint8_t*>(xq), ex,
                           (cudaStream_t)stream);
}

int sws_prefetch_layer(sws_ctx* c, int32_t layer, int32_t slot, sws_stream_t stream) {
  if (!c) return fail(SWS_E_INVALID, "prefetch_layer: ctx is NULL");
  if (layer < 0 || layer >= (int32_t)c->plan->layers.size())
    return fail(SWS_E_INVALID, "prefetch_layer: layer %d", layer);
  if (slot != 0 && slot != 1) return fail(SWS_E_INVALID, "prefetch_layer: slot %d", slot);
  cudaStream_t s = (cudaStream_t)stream;
  SWS_CUDA_TRY(cudaStreamWaitEvent(s, c->done[slot], 0));  // the slot's last reader in this context
  int rc = gather_impl(c, layer, slot, s);
  if (rc != SWS_OK) return rc;
  SWS_CUDA_TRY(cudaEventRecord(c->prefetched[slot], s));
  c->prefetch_layer[slot] = layer;
  return SWS_OK;
}

int sws_wait_prefetch(sws_ctx* c, int32_t layer, int32_t slot, sws_stream_t stream) {
  if (!c) return fail(SWS_E_INVALID, "wait_prefetch: ctx is NULL");
  if (layer < 0 || layer >= (int32_t)c->plan->layers.size())
    return fail(SWS_E_INVALID, "wait_prefetch: layer %d", layer);
  if (slot != 0 && slot != 1) return fail(SWS_E_INVALID, "wait_prefetch: slot %d", slot);
  bool cold = false;
  int rc = take_prefetch(c, layer, slot, (cudaStream_t)stream, &cold);
  if (rc != SWS_OK) return rc;
  return cold ? SWS_W_COLD : SWS_OK;
}

int sws_test_bounded_wait(sws_ctx* c, int64_t limit_ns, sws_stream_t stream) {
  if (limit_ns < 0 || limit_ns > 100000000) return fail(SWS_E_INVALID, "test_bounded_wait: limit %lld ns", (long long)limit_ns);
  int32_t* status = nullptr;
  if (c) {
    status = status_word(c);
  } else {  // the status word of sws_linear_noalloc's fixed scratch on the current device
    const int rc = noalloc_status_word(&status, (cudaStream_t)stream);
    if (rc != SWS_OK) return rc;
  }
  cudaError_t e = launch_bounded_wait(status, (uint64_t)limit_ns, (cudaStream_t)stream);
  return e == cudaSuccess ? SWS_OK : cuda_fail(e, "test_bounded_wait: launch");
}

int sws_silu_mul(const void* gu, int64_t m, int64_t f, void* act, sws_stream_t stream) {
  return launch_silu_mul(static_cast<const uint16_t*>(gu), m, f, static_cast<uint16_t*>(act), (cudaStream_t)stream);
}

int sws_ctx_status(sws_ctx* c, int32_t clear) {
  if (!c) return fail(SWS_E_INVALID, "ctx_status: ctx is NULL");
  clear_error();  // a message after this call comes from the call itself, not from the status word
  int32_t v = 0;
  const int rc = device_sync_deadline(c->device, "ctx_status");
  if (rc != SWS_OK) return rc;
  SWS_CUDA_TRY(cudaMemcpy(&v, c->ws, sizeof v, cudaMemcpyDeviceToHost));
  if (clear) {
    SWS_CUDA_TRY(cudaMemset(c->ws, 0, sizeof v));
    SWS_CUDA_TRY(cudaStreamSynchronize(nullptr));  // cleared before any later launch
  }
  return v;
}

int sws_trace_begin(sws_ctx* c, uint64_t* records, int32_t capacity, sws_stream_t stream) {
  if (!c) return fail(SWS_E_INVALID, "trace_begin: ctx is NULL");
  if (records && (capacity < 0 || !aligned16(records))) return fail(SWS_E_INVALID, "trace_begin: bad buffer");
  c->trace = records;
  c->trace_cap = records ? capacity : 0;
  c->trace_next = 0;
  if (records) {
    cudaError_t e = launch_trace_reset(records, capacity, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "trace_begin: reset kernel");
  }
  return SWS_OK;
}

int32_t sws_trace_count(const sws_ctx* c) { return c ? c->trace_next : -1; }

int sws_set_option(int32_t option, int64_t value) {
  switch (option) {
    case SWS_OPT_DECODE_KERNEL:
      if (value < SWS_DECODE_AUTO || value > SWS_DECODE_TCGEN05)
        return fail(SWS_E_INVALID, "set_option: decode kernel %lld", (long long)value);
      set_decode_kernel((int)value);
      return SWS_OK;
    case SWS_OPT_PREFILL_KERNEL:
      if (value < SWS_PREFILL_AUTO || value > SWS_PREFILL_PAIR)
        return fail(SWS_E_INVALID, "set_option: prefill kernel %lld", (long long)value);
      set_prefill_kernel((int)value);
      return SWS_OK;
    case SWS_OPT_HOST_WAIT_MS:
      if (value < 1 || value > 3600000) return fail(SWS_E_INVALID, "set_option: host wait %lld ms", (long long)value);
      g_host_wait_ms.store((int)value, std::memory_order_relaxed);
      return SWS_OK;
    case SWS_OPT_CHECK_BOUNDS:
      if (value != 0 && value != 1) return fail(SWS_E_INVALID, "set_option: check bounds %lld", (long long)value);
      set_check_bounds(value != 0);
      return SWS_OK;
    case SWS_OPT_GATHER_ENGINE:
      if (value != SWS_GATHER_TMA && value != SWS_GATHER_COPY_ENGINE && value != SWS_GATHER_TMA_SHARED_SM)
        return fail(SWS_E_INVALID, "set_option: gather engine %lld", (long long)value);
      g_gather_engine.store((int)value, std::memory_order_relaxed);
      return SWS_OK;
    default:
      return fail(SWS_E_INVALID, "set_option: unknown option %d", option);
  }
}

}  // extern "C"
