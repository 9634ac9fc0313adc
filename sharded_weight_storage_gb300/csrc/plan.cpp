// Host-side flat-layout planner and the relayout segment builder.
//
// Layout rule: weight-sharding blog (zdszero.github.io/weight_sharding.html),
// section "一层一次 AllGather：flat layout", steps 1-2: a layer's weights are
// concatenated in order, each padded to 16 bytes, the total padded to a
// multiple of 16*N, and T is cut into N byte-equal chunks of C = |T|/N.
// Eligibility: section "只 shard 真正 replicated 的权重": weights whose row
// count does not divide by N are skipped (kept replicated) with a warning.
// Relayout: section "加载：行 shard 先行，finalize 再重排", step 2.
#include <stdarg.h>
#include <stdio.h>

#include <algorithm>
#include <new>

#include "sws_internal.h"

namespace sws {

static thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

void clear_error() { g_last_error.clear(); }

int cuda_fail(cudaError_t e, const char* what) {
  return fail(SWS_E_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

int elem_bytes(int32_t dtype) {
  switch (dtype) {
    case SWS_E4M3: return 1;
    case SWS_BF16: return 2;
    case SWS_F32: return 4;
    case SWS_U8: return 1;
    case SWS_F16: return 2;
    default: return 0;
  }
}

}  // namespace sws

using namespace sws;

namespace sws {
void chunk_segments(int64_t g0, int64_t g1, int64_t c, void* const* chunks, const uint8_t* lin_src, uint8_t* lin_dst,
                    std::vector<CopySeg>* segs) {
  while (g0 < g1) {
    const int64_t ci = g0 / c, in_chunk = g0 - ci * c;
    const int64_t len = std::min(g1 - g0, c - in_chunk);
    uint8_t* ch = static_cast<uint8_t*>(chunks[ci]) + in_chunk;
    if (lin_dst) {
      segs->push_back(CopySeg{ch, lin_dst, len});
      lin_dst += len;
    } else {
      segs->push_back(CopySeg{lin_src, ch, len});
      if (lin_src) lin_src += len;
    }
    g0 += len;
  }
}

namespace {
std::atomic<bool> g_check_bounds{false};  // SWS_OPT_CHECK_BOUNDS
}  // namespace
bool check_bounds() { return g_check_bounds.load(std::memory_order_relaxed); }
void set_check_bounds(bool on) { g_check_bounds.store(on, std::memory_order_relaxed); }

std::vector<Extent> chunk_extents(void* const* chunks, int32_t n, int64_t c) {
  std::vector<Extent> x;
  for (int32_t i = 0; i < n; ++i) {
    const uint8_t* b = static_cast<const uint8_t*>(chunks[i]);
    x.push_back({b, b + c});
  }
  return x;
}

int check_segments(const std::vector<CopySeg>& segs, std::vector<Extent> srcs, std::vector<Extent> dsts,
                   const char* what) {
  auto by_lo = [](const Extent& a, const Extent& b) { return a.lo < b.lo; };
  std::sort(srcs.begin(), srcs.end(), by_lo);
  std::sort(dsts.begin(), dsts.end(), by_lo);
  // [a, a + len) inside some extent: the last extent starting at or before a must reach a + len
  auto inside = [&](const std::vector<Extent>& xs, const uint8_t* a, int64_t len) {
    auto it = std::upper_bound(xs.begin(), xs.end(), Extent{a, a}, by_lo);
    if (it == xs.begin()) return false;
    --it;
    return a >= it->lo && a + len <= it->hi;
  };
  for (size_t i = 0; i < segs.size(); ++i) {
    const CopySeg& g = segs[i];
    if (g.len <= 0) continue;
    if (!inside(dsts, g.dst, g.len))
      return fail(SWS_E_INVALID, "%s: copy segment %zu writes [%p, +%lld) outside its buffer", what, i,
                  static_cast<void*>(g.dst), (long long)g.len);
    if (g.src && !inside(srcs, g.src, g.len))
      return fail(SWS_E_INVALID, "%s: copy segment %zu reads [%p, +%lld) outside its buffer", what, i,
                  static_cast<const void*>(g.src), (long long)g.len);
  }
  return SWS_OK;
}

namespace {
// The copy segments of sws_relayout for one layer, with the extents of the
// row shards they read.
void relayout_segments(const sws_plan* p, int32_t layer, const void* const* row_shards, void* const* chunks,
                       std::vector<CopySeg>* segs, std::vector<Extent>* shard_extents) {
  const LayerPlan& lp = p->layers[layer];
  const int32_t n = p->n_shards;
  const int64_t c = lp.chunk;
  // Walk T once, cutting it into maximal runs that stay inside one chunk and
  // one source (a row shard, or padding; with SWS_SCALES_IN_T the scale
  // regions are written as zeros here and filled by sws_relayout_scales).
  auto emit = [&](int64_t g0, int64_t g1, const uint8_t* src) {  // T bytes [g0, g1)
    chunk_segments(g0, g1, c, chunks, src, nullptr, segs);
  };
  for (size_t k = 0; k < lp.sharded.size(); ++k) {
    const EntryPlan& e = p->entries[lp.sharded[k]];
    const int64_t per = e.bytes / n;  // bytes of one row shard
    for (int32_t r = 0; r < n && per > 0; ++r) {
      const uint8_t* sh = static_cast<const uint8_t*>(row_shards[k * n + r]);
      emit(e.offset + r * per, e.offset + (r + 1) * per, sh);
      shard_extents->push_back({sh, sh + per});
    }
    const int64_t end = e.offset + e.bytes;
    const int64_t next = (k + 1 < lp.sharded.size()) ? p->entries[lp.sharded[k + 1]].offset : lp.total;
    if (next > end) emit(end, next, nullptr);  // padding after the entry
  }
  if (lp.sharded.empty()) emit(0, lp.total, nullptr);
}
}  // namespace
}  // namespace sws

extern "C" {

const char* sws_last_error(void) { return g_last_error.c_str(); }

int32_t sws_version(void) { return 100; }

int sws_plan_create(const sws_entry* entries, int32_t n_entries, int32_t n_shards, uint32_t flags,
                    sws_plan** out) {
  if (!out) return fail(SWS_E_INVALID, "plan_create: out is NULL");
  *out = nullptr;
  if (n_entries < 0 || (n_entries > 0 && !entries)) return fail(SWS_E_INVALID, "plan_create: bad entry list");
  if (n_shards < 1 || n_shards > 256) return fail(SWS_E_INVALID, "plan_create: N=%d outside [1, 256]", n_shards);
  if (flags & ~SWS_SCALES_IN_T) return fail(SWS_E_INVALID, "plan_create: unknown flags 0x%x", flags);
  sws_plan* p = new (std::nothrow) sws_plan();
  if (!p) return fail(SWS_E_INVALID, "plan_create: out of host memory");
  p->n_shards = n_shards;
  p->flags = flags;
  int32_t n_layers = 0;
  for (int32_t j = 0; j < n_entries; ++j) {
    const sws_entry& e = entries[j];
    int eb = elem_bytes(e.dtype);
    if (e.layer < 0 || e.layer >= (1 << 20) || e.rows < 0 || e.cols < 0 || eb == 0 ||
        (e.cols > 0 && e.rows > (int64_t(1) << 40) / (e.cols * eb))) {
      delete p;
      return fail(SWS_E_INVALID, "plan_create: entry %d has layer %d, shape [%lld, %lld], dtype %d", j, e.layer,
                  (long long)e.rows, (long long)e.cols, e.dtype);
    }
    n_layers = std::max(n_layers, e.layer + 1);
  }
  p->layers.resize(n_layers);
  p->entries.resize(n_entries);
  bool skipped = false;
  for (int32_t j = 0; j < n_entries; ++j) {
    const sws_entry& e = entries[j];
    EntryPlan& ep = p->entries[j];
    LayerPlan& lp = p->layers[e.layer];
    ep.layer = e.layer;
    ep.dtype = e.dtype;
    ep.rows = e.rows;
    ep.cols = e.cols;
    ep.elem = elem_bytes(e.dtype);
    ep.bytes = e.rows * e.cols * ep.elem;
    ep.sharded = (e.rows % n_shards) == 0;
    ep.index_in_layer = (int32_t)lp.all.size();
    lp.all.push_back(j);
    if (!ep.sharded) {
      skipped = true;
      continue;
    }
    ep.offset = lp.total;           // o_j
    lp.total += roundup(ep.bytes, 16);  // each entry padded to 16 B
    lp.sharded.push_back(j);
    if ((flags & SWS_SCALES_IN_T) && e.dtype == SWS_E4M3) {
      // the weight's block scales follow it as their own entry, padded to 16 B
      ep.scale_bytes = cdiv(e.rows, 128) * cdiv(e.cols, 128) * 4;
      ep.scale_offset = lp.total;
      lp.total += roundup(ep.scale_bytes, 16);
      ep.scale_stage = lp.scale_stage_bytes;
      lp.scale_stage_bytes += roundup(ep.scale_bytes, 16);
    }
  }
  for (LayerPlan& lp : p->layers) {
    lp.total = roundup(lp.total, 16 * (int64_t)n_shards);  // total padded to 16*N
    lp.chunk = lp.total / n_shards;                         // C = |T|/N
    p->slot_bytes = std::max(p->slot_bytes, lp.total);
  }
  *out = p;
  if (skipped) {
    fail(SWS_W_SKIPPED, "plan_create: some entries have rows %% N != 0 and stay replicated");
    return SWS_W_SKIPPED;
  }
  return SWS_OK;
}

int sws_plan_info(const sws_plan* p, int32_t* n_layers, int32_t* n_shards, int32_t* n_entries) {
  if (!p) return fail(SWS_E_INVALID, "plan_info: plan is NULL");
  if (n_layers) *n_layers = (int32_t)p->layers.size();
  if (n_shards) *n_shards = p->n_shards;
  if (n_entries) *n_entries = (int32_t)p->entries.size();
  return SWS_OK;
}

int sws_plan_layer(const sws_plan* p, int32_t layer, int64_t* total, int64_t* chunk, int32_t* n_entries) {
  if (!p) return fail(SWS_E_INVALID, "plan_layer: plan is NULL");
  if (layer < 0 || layer >= (int32_t)p->layers.size()) return fail(SWS_E_INVALID, "plan_layer: layer %d", layer);
  const LayerPlan& lp = p->layers[layer];
  if (total) *total = lp.total;
  if (chunk) *chunk = lp.chunk;
  if (n_entries) *n_entries = (int32_t)lp.all.size();
  return SWS_OK;
}

int sws_plan_entry(const sws_plan* p, int32_t j, int64_t* offset, int64_t* nbytes, int32_t* sharded) {
  if (!p) return fail(SWS_E_INVALID, "plan_entry: plan is NULL");
  if (j < 0 || j >= (int32_t)p->entries.size()) return fail(SWS_E_INVALID, "plan_entry: entry %d", j);
  const EntryPlan& e = p->entries[j];
  if (offset) *offset = e.offset;
  if (nbytes) *nbytes = e.bytes;
  if (sharded) *sharded = e.sharded ? 1 : 0;
  return SWS_OK;
}

int sws_plan_scales(const sws_plan* p, int32_t j, int64_t* offset, int64_t* nbytes) {
  if (!p) return fail(SWS_E_INVALID, "plan_scales: plan is NULL");
  if (j < 0 || j >= (int32_t)p->entries.size()) return fail(SWS_E_INVALID, "plan_scales: entry %d", j);
  const EntryPlan& e = p->entries[j];
  if (offset) *offset = e.scale_offset;
  if (nbytes) *nbytes = e.scale_offset >= 0 ? e.scale_bytes : 0;
  return SWS_OK;
}

int64_t sws_plan_slot_bytes(const sws_plan* p) { return p ? p->slot_bytes : -1; }

void sws_plan_destroy(sws_plan* p) { delete p; }

int sws_relayout(const sws_plan* p, int32_t layer, const void* const* row_shards, void* const* chunks,
                 sws_stream_t stream) {
  if (!p) return fail(SWS_E_INVALID, "relayout: plan is NULL");
  if (layer < 0 || layer >= (int32_t)p->layers.size()) return fail(SWS_E_INVALID, "relayout: layer %d", layer);
  const LayerPlan& lp = p->layers[layer];
  const int32_t n = p->n_shards;
  if (lp.total == 0) return SWS_OK;
  if (!chunks) return fail(SWS_E_INVALID, "relayout: chunks is NULL");
  if (!lp.sharded.empty() && !row_shards) return fail(SWS_E_INVALID, "relayout: row_shards is NULL");
  for (int32_t i = 0; i < n; ++i) {
    if (!chunks[i]) return fail(SWS_E_INVALID, "relayout: chunk %d is NULL", i);
    if (!aligned16(chunks[i])) return fail(SWS_E_ALIGN, "relayout: chunk %d is not 16-byte aligned", i);
  }
  for (size_t k = 0; k < lp.sharded.size(); ++k)
    for (int32_t r = 0; r < n; ++r)
      if (p->entries[lp.sharded[k]].bytes > 0 && !row_shards[k * n + r])
        return fail(SWS_E_INVALID, "relayout: row shard %d of sharded entry %zu is NULL", r, k);
  std::vector<CopySeg> segs;
  std::vector<Extent> shards;
  relayout_segments(p, layer, row_shards, chunks, &segs, &shards);
  if (check_bounds()) {
    const int rc = check_segments(segs, shards, chunk_extents(chunks, n, lp.chunk), "relayout");
    if (rc != SWS_OK) return rc;
  }
  cudaError_t e = launch_relayout(segs, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "relayout kernel launch");
  return SWS_OK;
}


int sws_relayout_scales(const sws_plan* p, int32_t layer, const float* const* scales, void* const* chunks,
                        sws_stream_t stream) {
  if (!p) return fail(SWS_E_INVALID, "relayout_scales: plan is NULL");
  if (layer < 0 || layer >= (int32_t)p->layers.size()) return fail(SWS_E_INVALID, "relayout_scales: layer %d", layer);
  const LayerPlan& lp = p->layers[layer];
  if (!(p->flags & SWS_SCALES_IN_T) || lp.total == 0) return SWS_OK;
  if (!chunks || !scales) return fail(SWS_E_INVALID, "relayout_scales: chunks or scales is NULL");
  for (int32_t i = 0; i < p->n_shards; ++i) {
    if (!chunks[i]) return fail(SWS_E_INVALID, "relayout_scales: chunk %d is NULL", i);
    if (!aligned16(chunks[i])) return fail(SWS_E_ALIGN, "relayout_scales: chunk %d is not 16-byte aligned", i);
  }
  // Each rank holds the full (replicated) scale tensor and copies out the
  // bytes that fall into its window [i*C, (i+1)*C) of T.
  std::vector<CopySeg> segs;
  std::vector<Extent> srcs;
  for (size_t k = 0; k < lp.all.size(); ++k) {
    const EntryPlan& e = p->entries[lp.all[k]];
    if (e.scale_offset < 0 || e.scale_bytes == 0) continue;
    if (!scales[k]) return fail(SWS_E_INVALID, "relayout_scales: entry %zu of layer %d has no scales", k, layer);
    const uint8_t* sc = reinterpret_cast<const uint8_t*>(scales[k]);
    chunk_segments(e.scale_offset, e.scale_offset + e.scale_bytes, lp.chunk, chunks, sc, nullptr, &segs);
    srcs.push_back({sc, sc + e.scale_bytes});
  }
  if (segs.empty()) return SWS_OK;
  if (check_bounds()) {
    const int rc = check_segments(segs, srcs, chunk_extents(chunks, p->n_shards, lp.chunk), "relayout_scales");
    if (rc != SWS_OK) return rc;
  }
  cudaError_t e = launch_relayout(segs, (cudaStream_t)stream);
  return e == cudaSuccess ? SWS_OK : cuda_fail(e, "relayout_scales kernel launch");
}

int sws_test_check_relayout(const sws_plan* p, int32_t layer, int64_t chunk_bytes) {
  if (!p) return fail(SWS_E_INVALID, "test_check_relayout: plan is NULL");
  if (layer < 0 || layer >= (int32_t)p->layers.size())
    return fail(SWS_E_INVALID, "test_check_relayout: layer %d", layer);
  const LayerPlan& lp = p->layers[layer];
  const int32_t n = p->n_shards;
  // Stand-in addresses, never dereferenced: row shards and chunks 2^36 bytes
  // apart (more than any of them holds), from 2^52 up.
  auto at = [](uint64_t i) { return reinterpret_cast<uint8_t*>(((uint64_t)1 << 52) + (i << 36)); };
  if ((lp.sharded.size() + 1) * (size_t)n >= ((size_t)1 << 14))
    return fail(SWS_E_INVALID, "test_check_relayout: too many row shards for the stand-in addresses");
  std::vector<const void*> shards(lp.sharded.size() * (size_t)n);
  for (size_t i = 0; i < shards.size(); ++i) shards[i] = at(i);
  std::vector<void*> chunks(n);
  for (int32_t i = 0; i < n; ++i) chunks[i] = at(shards.size() + i);
  std::vector<CopySeg> segs;
  std::vector<Extent> srcs;
  relayout_segments(p, layer, shards.data(), chunks.data(), &segs, &srcs);
  return check_segments(segs, srcs, chunk_extents(chunks.data(), n, chunk_bytes), "relayout");
}

}  // extern "C"
