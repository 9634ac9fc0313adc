/*
 * sws.h - C ABI of the sharded weight storage library ("store sharded,
 * compute full"), for NVIDIA GB300 (sm_103a).
 *
 * The method (weight-sharding blog, zdszero.github.io/weight_sharding.html):
 * every layer's replicated weights are packed into one flat byte stream T
 * (section "一层一次 AllGather：flat layout"); T is cut into N equal chunks, one
 * per rank; before a layer runs, one gather restores T into one of two
 * ping-pong slots (section "提前一层：lookahead 与 ping-pong slot") and the
 * layer's linears read zero-copy views of the slot. Here the N ranks are N
 * device buffers on one GPU and the AllGather is an on-GPU copy kernel.
 *
 * Conventions for every call:
 *   - Return value: SWS_OK (0), a positive warning, or a negative error code.
 *     The message of the last error on the calling thread is available from
 *     sws_last_error(). No C++ exception crosses this boundary and no kernel
 *     traps; faults of queued GPU work surface as SWS_E_CUDA on a later call.
 *   - Memory: the caller allocates and owns every device buffer (chunks, row
 *     shards, slots, scales, activations, outputs, workspace) and keeps it
 *     alive until the work queued on it has finished. The library allocates
 *     host objects, CUDA events and one CUDA stream per context (prefill
 *     layers quantise the next linear's activations on it); it never calls
 *     cudaMalloc.
 *   - Alignment: every device pointer passed in must be 16-byte aligned
 *     (SWS_E_ALIGN otherwise).
 *   - Streams: sws_stream_t is a cudaStream_t; NULL is the legacy default
 *     stream. All device work is asynchronous with respect to the host.
 *   - Element types: SWS_E4M3 is OCP FP8 E4M3FN (1 byte), SWS_BF16 2 bytes,
 *     SWS_F32 4 bytes, SWS_U8 1 byte, SWS_F16 IEEE binary16 (2 bytes).
 */
#ifndef SWS_H_
#define SWS_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define SWS_OK 0
/* Some entry has rows % N != 0 and stays replicated, outside T (the blog's
 * section "只 shard 真正 replicated 的权重": such weights are skipped with a
 * warning). The plan is still created. */
#define SWS_W_SKIPPED 1
#define SWS_W_COLD 2 /* sws_wait_prefetch: nothing was prefetched, the gather ran inline */
#define SWS_E_INVALID (-1)     /* bad argument: N, shape, index, size, layout */
#define SWS_E_ALIGN (-2)       /* a device pointer is not 16-byte aligned */
#define SWS_E_STATE (-3)       /* slot holds another layer, or calls out of order */
#define SWS_E_CUDA (-4)        /* a CUDA runtime call failed (message has the name) */
#define SWS_E_TIMEOUT (-5)     /* a device-side wait gave up (see sws_ctx_status) */
#define SWS_E_UNSUPPORTED (-6) /* device is not sm_103, or shape outside a kernel's range */
#define SWS_E_WORKSPACE (-7)   /* workspace smaller than sws_workspace_bytes() */

/* ---- element types ----------------------------------------------------- */
#define SWS_E4M3 0
#define SWS_BF16 1
#define SWS_F32 2
#define SWS_U8 3
#define SWS_F16 4

/* ---- linear weight sources --------------------------------------------- */
#define SWS_SRC_SLOT0 0 /* view of slot 0 (must hold the entry's layer) */
#define SWS_SRC_SLOT1 1 /* view of slot 1 (must hold the entry's layer) */
#define SWS_SRC_FUSED 2 /* read the layer's chunks directly through the chunk map */

/* ---- plan flags -------------------------------------------------------- */
/* Block scales inside T: each sharded E4M3 entry's fp32 block-scale tensor
 * [ceil(rows/128), ceil(cols/128)] becomes an entry of T of its own, right
 * after the weight (16-byte padded like every entry), so the gather restores
 * the scales with the weights and the linears read them from the slot (or
 * through the chunk map). Off by default: the blog keeps scales replicated,
 * outside the flat layout (section "加载：行 shard 先行，finalize 再重排", the
 * quantisation variants). */
#define SWS_SCALES_IN_T 1u

/* ---- run_layers flags -------------------------------------------------- */
#define SWS_RUN_FUSED 1u  /* no gather: every linear reads the chunks directly */
#define SWS_RUN_TIMING 2u /* record per-layer CUDA events (see sws_run_timing) */
#define SWS_RUN_FIRST_PREFETCHED 4u /* the first layer was prefetched into slot 0 (sws_prefetch_layer):
                                       wait for it instead of gathering it (cold start: gather) */

typedef struct CUstream_st* sws_stream_t;
typedef struct sws_plan sws_plan;
typedef struct sws_ctx sws_ctx;
typedef struct sws_graph sws_graph;

/* One weight declared to the planner. rows = out_features (dimension 0, the
 * one row shards split), cols = in_features; row-major [rows, cols]. */
typedef struct sws_entry {
  int32_t layer; /* layer id, 0 <= layer < 2^20 */
  int32_t dtype; /* SWS_E4M3, SWS_BF16, SWS_F32, SWS_U8 or SWS_F16 */
  int64_t rows;
  int64_t cols;
} sws_entry;

/* Activations and outputs of one layer for sws_run_layers: x[k] / y[k] belong
 * to the k-th entry of that layer in declaration order (replicated entries
 * included), each x bf16 [m, cols], each y bf16 [m, rows]. */
typedef struct sws_layer_io {
  const void* const* x;
  void* const* y;
  int64_t m;
} sws_layer_io;

/* ---- planner (host only, no GPU needed) -------------------------------- */

/* Flat layout (blog section "flat layout", steps 1-2): the sharded entries of
 * each layer are concatenated in declaration order at offsets o_j that are
 * multiples of 16 (every entry's byte size is rounded up to 16), |T| is
 * rounded up to a multiple of 16*N, and C = |T|/N. An entry is sharded iff
 * rows % N == 0; otherwise it is replicated and the call returns
 * SWS_W_SKIPPED. n_shards in [1, 256]; rows, cols >= 0; flags 0 or
 * SWS_SCALES_IN_T (then each sharded E4M3 entry is followed in T by its
 * block-scale tensor, 16-byte padded; sws_plan_scales gives where).
 * On success *out receives a plan owned by the caller (sws_plan_destroy). */
int sws_plan_create(const sws_entry* entries, int32_t n_entries, int32_t n_shards, uint32_t flags,
                    sws_plan** out);
/* Number of layers (highest layer id + 1) and shards. */
int sws_plan_info(const sws_plan* plan, int32_t* n_layers, int32_t* n_shards, int32_t* n_entries);
/* |T| of a layer and its chunk size C (both 0 for a layer with no sharded
 * entry) and how many entries (sharded or not) the layer has. */
int sws_plan_layer(const sws_plan* plan, int32_t layer, int64_t* total_bytes, int64_t* chunk_bytes,
                   int32_t* n_entries);
/* Offset o_j of entry j inside its layer's T (-1 if replicated), its size in
 * bytes and whether it is sharded. */
int sws_plan_entry(const sws_plan* plan, int32_t j, int64_t* offset, int64_t* nbytes, int32_t* sharded);
/* With SWS_SCALES_IN_T: offset inside its layer's T of entry j's block-scale
 * tensor (float32 [ceil(rows/128), ceil(cols/128)] row-major, 16-byte
 * aligned) and its size in bytes; offset -1 and size 0 when the entry's
 * scales are not in T (flag off, not E4M3, or a replicated entry). */
int sws_plan_scales(const sws_plan* plan, int32_t j, int64_t* offset, int64_t* nbytes);
/* max over layers of |T| - the size each of the two slots needs. */
int64_t sws_plan_slot_bytes(const sws_plan* plan);
void sws_plan_destroy(sws_plan* plan);

/* ---- one-time relayout -------------------------------------------------- */

/* Remaps a layer from the loader's per-weight row shards to flat chunks (blog
 * section "加载：行 shard 先行，finalize 再重排", step 2): chunk i receives T
 * bytes [i*C, (i+1)*C); a byte at local offset u of sharded entry j comes from
 * row shard u / (s_j/N) at offset u % (s_j/N); padding bytes are written as 0.
 *   row_shards: host array of device pointers, [k*N + r] = shard r of the k-th
 *               sharded entry of the layer (declaration order), each
 *               (rows/N)*cols*elem bytes, contiguous. Any alignment.
 *   chunks:     host array of N device pointers, C bytes each, 16-B aligned.
 * Enqueued on `stream`; source and destination must not overlap. */
int sws_relayout(const sws_plan* plan, int32_t layer, const void* const* row_shards, void* const* chunks,
                 sws_stream_t stream);

/* With SWS_SCALES_IN_T: fills the scale regions of a layer's chunks. Block
 * FP8 keeps its scales at full shape on every rank (the blog's block-FP8
 * variant slices at finalize, from the full tensor), so each chunk i receives
 * the bytes of each scale tensor that fall into its window [i*C, (i+1)*C).
 *   scales: host array [n entries of the layer, declaration order] of device
 *           pointers to the full float32 scale tensors; NULL where the entry's
 *           scales are not in T. Any 4-byte alignment.
 *   chunks: as for sws_relayout.
 * sws_relayout writes the scale regions as zeros, so call this after it, on
 * the same stream. A no-op for plans without the flag. */
int sws_relayout_scales(const sws_plan* plan, int32_t layer, const float* const* scales, void* const* chunks,
                        sws_stream_t stream);

/* ---- context: resident chunks, two slots, scales, workspace ------------- */

/* Bytes of workspace a context needs for linears with up to max_m rows of
 * activations (split-K partial sums, counters, the tcgen05 decode path's
 * activation split blocks, with SWS_SCALES_IN_T a staging area for one
 * layer's scales read through the chunk map, two buffers of prefill
 * activations - the quantiser's output for E4M3 entries, x rounded to f16 for
 * F16 entries - and the device status word). */
int64_t sws_workspace_bytes(const sws_plan* plan, int64_t max_m);

/* Creates a context over caller-owned device memory:
 *   chunks:     host array [n_layers * N] of device pointers, layer-major;
 *               chunk (l, i) holds C_l bytes. Entries for layers without
 *               sharded weights may be NULL.
 *   slot0/1:    two device buffers of at least sws_plan_slot_bytes() bytes.
 *   scales:     host array [n_entries] of device pointers to float32 block
 *               scales [ceil(rows/128), ceil(cols/128)] row-major for E4M3
 *               entries (NULL for other types). With SWS_SCALES_IN_T the
 *               linears of sharded E4M3 entries read their scales from T
 *               (slot + scale offset, or the chunks), and their pointers here
 *               may be NULL; replicated E4M3 entries still need theirs.
 *   replicated: host array [n_entries] of device pointers to the full weight
 *               of each replicated entry (NULL for sharded ones); may be NULL
 *               when every entry is sharded.
 *   workspace:  device buffer of workspace_bytes >= sws_workspace_bytes(plan,
 *               max_m) for the largest m later passed to sws_linear. It is
 *               zeroed here on the legacy default stream, synchronously.
 * Every pointer array is copied; the plan must outlive the context. */
int sws_ctx_create(const sws_plan* plan, void* const* chunks, void* slot0, void* slot1,
                   const float* const* scales, const void* const* replicated, void* workspace,
                   int64_t workspace_bytes, sws_ctx** out);
void sws_ctx_destroy(sws_ctx* ctx);

/* One layer's gather (blog "flat layout" step 3, all_gather_into_tensor):
 * slot[i*C : (i+1)*C] = chunk(layer, i) for i in [0, N), a pure byte copy on
 * `stream`, by the TMA bulk-copy kernel or, with SWS_OPT_GATHER_ENGINE =
 * SWS_GATHER_COPY_ENGINE, by N cudaMemcpyAsync copies. Tags the slot with
 * `layer` (host-side, in issue order). The kernel is launched with
 * programmatic stream serialisation: right after a decode linear of this
 * library on `stream`, it may start while that launch's last (settle) kernel,
 * which reads no slot and writes only y, finishes; after any other work it
 * starts when that work completes, and work queued after it still waits for
 * everything before it. */
int sws_gather_to_slot(sws_ctx* ctx, int32_t layer, int32_t slot, sws_stream_t stream);

/* Y = X W_j^T for entry j (blog section "核心抽象": the GEMM sees the full W),
 * fp32 accumulation, Y rounded to bf16 (nearest even):
 *   E4M3 entries: Y[m, o] = sum_i x[m, i] * e4m3(q[o, i]) * s[o/128, i/128];
 *   BF16 entries: Y[m, o] = sum_i x[m, i] * w[o, i]  (no scales; the blog's
 *                 unquantised variant goes through the same flat layout);
 *   F16 entries:  Y[m, o] = sum_i f16(x[m, i]) * w[o, i]  (w IEEE binary16,
 *                 x rounded to nearest even f16 first, the tensor cores'
 *                 operands of one MMA sharing one format).
 * W_j is the view slot + o_j (src = SWS_SRC_SLOT0/1; the slot's tag must equal
 * the entry's layer, else SWS_E_STATE), the chunks themselves
 * (SWS_SRC_FUSED), or the replicated buffer for entries outside T (src
 * ignored). x: bf16 [m, cols] row-major; y: bf16 [m, rows] row-major.
 * m in [0, 2^31). m <= 64 runs a split-K decode launch, by default on the
 * tcgen05 kernel (SWS_OPT_DECODE_KERNEL): for E4M3 with x split exactly into
 * two e4m3 terms (kind::f8f6f4), for BF16 / F16 on bf16 / f16 operands
 * (kind::f16), from views or through the chunk map (SWS_SRC_FUSED).
 * m > 64 runs the prefill path: E4M3 quantises x (sws_quantize_x into the
 * workspace) and runs the tcgen05 block-scaled FP8 GEMM; BF16 runs a tcgen05
 * bf16 GEMM on x directly; F16 rounds x to f16 into the workspace and runs
 * the same GEMM on f16 operands. Requires E4M3, BF16 or F16 weights (else
 * SWS_E_UNSUPPORTED), cols % 16 == 0, and, for E4M3 with m > 64,
 * cols % 128 == 0; E4M3 entries need their scales. With SWS_SCALES_IN_T a
 * sharded E4M3 entry's scales come from T: from the same slot as the weight,
 * or - on the chunk-map source - copied from the chunks into the workspace by
 * a small copy kernel queued before the linear's kernels. Linears that share
 * a context must not overlap on the GPU (they share the workspace). */
int sws_linear(sws_ctx* ctx, int32_t entry, int32_t src, const void* x, int64_t m, void* y,
               sws_stream_t stream);

/* Every linear of one layer (declaration order, replicated entries included),
 * with io->x[k] / io->y[k] for its k-th entry and a common m: the decode-sized
 * ones (m <= 64) run as grouped launches, up to 8 linears per launch, one
 * group per weight source (views: slot src or replicated buffers; chunk-map
 * reads: SWS_SRC_FUSED) and weight type (E4M3, BF16, F16), so a layer pays one
 * launch instead of one per weight. Same results and rules as sws_linear for
 * each entry. */
int sws_layer_linears(sws_ctx* ctx, int32_t layer, int32_t src, const sws_layer_io* io, sws_stream_t stream);

/* Decode linear that allocates nothing. The paper has no counterpart to this
 * call; it serves callers that cannot give the library memory. An inference engine
 * that sizes its KV-cache pool from the memory left free after loading the
 * weights has no headroom for allocations made later, and a device allocation
 * in the middle of a decode step can stall the whole GPU; such a caller passes
 * only its inputs and outputs here. Same result as sws_linear for m <= 64
 * (within rounding: the split-K partition may differ), on the warp-level
 * mma.sync decode kernel:
 *   w:      E4M3 weight [rows, cols] row-major (e.g. a slot view slot + o_j),
 *   scales: float32 block scales [ceil(rows/128), ceil(cols/128)],
 *   x:      bf16 [m, cols], y: bf16 [m, rows]; all 16-byte aligned.
 * Limits: 0 <= m <= 64, cols % 16 == 0, at most 4096 row blocks (2,097,152
 * rows for m <= 16, 1,048,576 rows for 16 < m <= 64); anything larger is
 * rejected with SWS_E_INVALID / SWS_E_UNSUPPORTED before any launch.
 * Scratch: a fixed array of 32 MiB + 16 KiB + 256 B inside the library's
 * device image (every GPU that loads the library holds it until the process
 * exits): split-K partial sums (two 64 KiB slots for each of up to 256 CTAs,
 * so the grid is the same as sws_linear's), one arrival counter per row block
 * and one int32 status word. It is shared by all calls on a device and keeps
 * the last call's contents; the arrival counters are cleared on `stream`
 * before each launch. Calls whose work overlaps on the GPU race on it, so
 * serialise them (one stream).
 * Status: a device-side wait of the kernel that runs out (2 s) records
 * SWS_E_TIMEOUT in the status word, and the rows it left unwritten stay as
 * they were; the call itself has already returned SWS_OK by then, so read the
 * word with sws_noalloc_status. It stays set until cleared there.
 * The first call on a device looks up the array's device address with
 * cudaGetSymbolAddress (with that device current) and clears the status word
 * on `stream`; make that first call before any stream capture. No cudaMalloc /
 * cudaFree is ever called. */
int sws_linear_noalloc(const void* w, const float* scales, int64_t rows, int64_t cols, const void* x, int64_t m,
                       void* y, sws_stream_t stream);
/* Status word of sws_linear_noalloc's scratch on the current device: *status
 * receives 0, or the SWS_E_* code one of its kernels recorded since the last
 * clear (e.g. SWS_E_TIMEOUT). Waits for the device's queued work first, at
 * most the host wait limit (SWS_OPT_HOST_WAIT_MS): past it the call returns
 * SWS_E_TIMEOUT itself and *status is not read. `clear` != 0 resets the word.
 * Returns SWS_OK when *status was read. Allocates nothing. */
int sws_noalloc_status(int32_t clear, int32_t* status);

/* Lookahead over layers first..last (blog "提前一层" and "SGLang 中的实现"):
 * gather(first) is issued on `side` after `side` waits for work already
 * queued on `main`; then for each layer l: `side` waits done(l-1) and gathers
 * layer l+1 into slot (l+1-first) % 2, recording ready(l+1); `main` waits
 * ready(l) once, runs every linear of layer l on slot (l-first) % 2 and
 * records done(l). At most two layers' full weights are resident. With
 * SWS_RUN_FUSED no gather runs and the linears read the chunks directly.
 * io[l - first] gives layer l's activations and outputs. On return `main`
 * carries all the work (side-stream work is joined into it). The linears'
 * kernels are launched with the device's highest stream priority and the
 * gather with the default one, so that the block scheduler gives the SMs to
 * the linears first when both wait for them.
 * Stream capture: without SWS_RUN_TIMING the call only enqueues kernels and
 * event record/wait pairs (no synchronisation, no allocation, no query), so
 * it records into a CUDA graph when `main` is capturing: the fork to `side`
 * and the join back are captured edges, and replaying the graph repeats the
 * run on the pointers given at capture time (activations and outputs are read
 * and written in place, so refill x between replays). SWS_RUN_TIMING records
 * timing events and is not capturable (SWS_E_INVALID while capturing). */
int sws_run_layers(sws_ctx* ctx, int32_t first, int32_t last, const sws_layer_io* io, uint32_t flags,
                   sws_stream_t main, sws_stream_t side);

/* Draft-model first-layer prefetch (blog "CUDA graph 与 draft 模型": the draft
 * model's layer 0 has no previous layer to hide its gather behind, so the
 * gather is taken out of the graph and issued early on a dedicated stream;
 * a shared side stream would queue it behind the target model's gathers).
 * sws_prefetch_layer: `stream` waits for the last reader of `slot` in this
 * context (its done event), gathers `layer` into `slot` and records an event;
 * the slot is marked as holding a prefetched `layer`.
 * sws_wait_prefetch: `stream` waits once for that gather if `layer` is the
 * prefetched one (returns SWS_OK); otherwise - a cold start, or another gather
 * into the slot since - `stream` waits for the slot's last reader and gathers
 * `layer` inline (returns SWS_W_COLD). run_layers with
 * SWS_RUN_FIRST_PREFETCHED does the same for its first layer (slot 0) on the
 * side stream. Host-side bookkeeping in issue order; meant for eager launches
 * outside a captured graph, as the blog does. */
int sws_prefetch_layer(sws_ctx* ctx, int32_t layer, int32_t slot, sws_stream_t stream);
int sws_wait_prefetch(sws_ctx* ctx, int32_t layer, int32_t slot, sws_stream_t stream);

/* After a run with SWS_RUN_TIMING: waits for the recorded events (polling, at
 * most the host wait limit SWS_OPT_HOST_WAIT_MS, else SWS_E_TIMEOUT with a
 * message saying so) and writes, per layer of that run (n values each,
 * n = last - first + 1):
 *   exposed_ms[l] - time `main` stood waiting for ready(l) (from the end of
 *                   layer l-1's linears to the start of layer l's; for the
 *                   first layer, from the run's start),
 *   layer_ms[l]   - time from the start to the end of layer l's linears. */
int sws_run_timing(sws_ctx* ctx, float* exposed_ms, float* layer_ms, int32_t n);

/* A lookahead run recorded once as a CUDA graph (blog "CUDA graph 与 draft
 * 模型": the per-layer schedule is fixed, so it is replayed instead of
 * re-issued). sws_graph_capture captures sws_run_layers(ctx, first, last, io,
 * flags, main, side) on `main` (thread-local capture mode; `main` must not be
 * the legacy default stream nor already capturing, else SWS_E_INVALID /
 * SWS_E_STATE) and instantiates it with per-node priorities kept
 * (cudaGraphInstantiateFlagUseNodePriority), so the linears' kernels keep the
 * higher launch priority they have in eager runs. SWS_RUN_TIMING and
 * SWS_RUN_FIRST_PREFETCHED are not allowed (SWS_E_INVALID). Nothing runs at
 * capture; each sws_graph_launch replays the run on `stream` on the pointers
 * given at capture (refill the activations in place between launches). The
 * graph uses the context's events, slots and workspace: replays of graphs of
 * one context, and eager calls on it, must not overlap on the GPU. On error
 * *out is NULL, any partial capture is discarded and the context's host-side
 * state (slot tags, prefetch marks, trace position) is as before the call. On
 * success the slots' layer tags become unknown: an eager sws_linear from a
 * slot needs a sws_gather_to_slot (or a run_layers) first, else SWS_E_STATE.
 * The caller destroys the graph (sws_graph_destroy, NULL allowed) before the
 * context. */
int sws_graph_capture(sws_ctx* ctx, int32_t first, int32_t last, const sws_layer_io* io, uint32_t flags,
                      sws_stream_t main, sws_stream_t side, sws_graph** out);
int sws_graph_launch(sws_graph* graph, sws_stream_t stream);
void sws_graph_destroy(sws_graph* graph);

/* Prefill activation quantiser: for each row m and 128-column group g,
 * ex[m, g] = 2^k with k the smallest integer such that amax <= 448 * 2^k
 * (1 when the group is all zero), and xq[m, i] = e4m3_rne(x[m, i] / ex[m, g])
 * (ties to even, saturating). x bf16 [m, k] row-major, xq u8 [m, k],
 * ex float32 [m, ceil(k/128)]; k % 16 == 0. */
int sws_quantize_x(const void* x, int64_t m, int64_t k, void* xq, float* ex, sws_stream_t stream);

/* SiLU(gate) * up, the step between a shared expert's two linears (gate_up ->
 * SiLU * up -> down; the blog's shared-expert layer, the second workload):
 *   act[m, j] = bf16_rne( g / (1 + e^-g) * u ),  g = gu[m, j], u = gu[m, f + j],
 * computed in fp32. gu bf16 [m, 2f] row-major with the gate half first (the
 * gate_up linear's output), act bf16 [m, f]; f % 8 == 0, both 16-byte aligned
 * (else SWS_E_UNSUPPORTED / SWS_E_ALIGN). Runs on `stream`. */
int sws_silu_mul(const void* gu, int64_t m, int64_t f, void* act, sws_stream_t stream);

/* Device-side status of a context: 0, or the SWS_E_* code a kernel recorded
 * (e.g. SWS_E_TIMEOUT when a wait on a TMA completion gave up). Waits for all
 * work queued on the context's device first, at most the host wait limit
 * (SWS_OPT_HOST_WAIT_MS): past it the call returns SWS_E_TIMEOUT without
 * reading the word, the device's work continues, and a later call reads it.
 * The call empties sws_last_error() first, so after it a non-empty message
 * means the call itself failed (host wait, CUDA error) and an empty one that
 * the value is the word. `clear` != 0 resets the word. */
int sws_ctx_status(sws_ctx* ctx, int32_t clear);

/* ---- tracing ------------------------------------------------------------ */

/* Optional device timestamps: each later gather / linear launch of the
 * context appends one record of 4 uint64 to `records` (device memory,
 * capacity records): {tag, start_ns, end_ns, 0} where tag = kind << 56 |
 * kernel << 48 | layer << 32 | entry (kind 1 = gather, 2 = linear; kernel, for
 * linears: 1 mma.sync on views, 2 mma.sync through the chunk map, 3 tcgen05
 * on views, 4 tcgen05 through the chunk map, 5 prefill, 6 prefill on a CTA
 * pair), start_ns is the earliest
 * %globaltimer read by any CTA at entry and end_ns the latest at exit. Passing
 * NULL turns tracing off. Records are reset (start = ~0, end = 0) on `stream`.
 * Returns the number of records written so far through sws_trace_count. */
int sws_trace_begin(sws_ctx* ctx, uint64_t* records, int32_t capacity, sws_stream_t stream);
int32_t sws_trace_count(const sws_ctx* ctx);

/* ---- options -------------------------------------------------------------- */
#define SWS_OPT_DECODE_KERNEL 1 /* which kernel serves decode linears (m <= 64) from views */
#define SWS_DECODE_AUTO 0       /* the library's choice (default): tcgen05 */
#define SWS_DECODE_MMA 1        /* warp-level mma.sync kernel */
#define SWS_DECODE_TCGEN05 2    /* tcgen05 / TMEM kernel */
#define SWS_OPT_PREFILL_KERNEL 2 /* which kernel serves prefill linears (m > 64) */
#define SWS_PREFILL_AUTO 0       /* the library's choice (default): one CTA per tile */
#define SWS_PREFILL_SINGLE 1     /* one CTA per 128 x 256 output tile */
#define SWS_PREFILL_PAIR 2       /* a cluster of two CTAs (tcgen05 .cta_group::2) per 256 x 256 tile;
                                    SWS_E_UNSUPPORTED at launch if no such cluster fits */
#define SWS_OPT_GATHER_ENGINE 3 /* what copies the chunks into a slot (sws_gather_to_slot, run_layers) */
#define SWS_GATHER_TMA 0        /* default: the TMA bulk-copy kernel (uses SMs, writes a trace record) */
#define SWS_GATHER_COPY_ENGINE 1 /* N cudaMemcpyAsync device-to-device copies of C bytes on the stream:
                                    the copy engines move the bytes and no SM is used (the pages'
                                    all-gather runs on copy engines too); no trace record */
#define SWS_GATHER_TMA_SHARED_SM 2 /* the TMA kernel with one 48 KB CTA per SM, which fits beside a
                                      decode GEMM CTA (m <= 32): run_layers' lookahead gather then
                                      shares the SMs with the current layer's linears instead of
                                      waiting for them; slower than SWS_GATHER_TMA on its own */
#define SWS_OPT_HOST_WAIT_MS 4 /* limit of the host-side waits (sws_run_timing, sws_ctx_status,
                                  sws_noalloc_status), in ms, 1..3600000; default 10000 */
#define SWS_OPT_CHECK_BOUNDS 5 /* 0 (default) or 1: a self-check of the library's copy plans.
                                  Before sws_relayout, sws_relayout_scales, the scale staging of
                                  a chunk-map linear and a gather launch anything, every copy
                                  segment is checked against the buffer it reads (a row shard, a
                                  scale tensor, a chunk of C bytes) and the one it writes (a
                                  chunk, the slot, the workspace's staging area); a segment that
                                  leaves one fails the call with SWS_E_INVALID (the message names
                                  it) and nothing is launched. For debugging; it costs host time. */
/* Process-wide options, read at each launch. Both decode kernels compute the
 * same linear (sws_linear) within the same tolerance, from views and through
 * the chunk map (a chunk-map launch whose segments or split rows exceed the
 * tcgen05 launch's tables runs on the mma.sync kernel). A tcgen05 launch is
 * three kernels on the stream (activation split, GEMM, split-K settle); an
 * mma.sync launch is one.
 * Both prefill kernels compute the same sums in the same slab order per output
 * element and give bit-identical results.
 * An option may be set from any thread; a call running at the same time on
 * another thread sees its old value or its new one.
 * SWS_E_INVALID for an unknown option or value. */
int sws_set_option(int32_t option, int64_t value);

/* Test hook of SWS_OPT_CHECK_BOUNDS (host only, no device memory): builds the
 * copy segments sws_relayout would launch for `layer`, with stand-in
 * addresses for the row shards and for N chunks of `chunk_bytes` bytes each,
 * and checks them as that option does. SWS_OK when every segment stays inside
 * its buffers (chunk_bytes >= the plan's C), SWS_E_INVALID otherwise. */
int sws_test_check_relayout(const sws_plan* plan, int32_t layer, int64_t chunk_bytes);

/* Test hook of the decode launch's split-K bookkeeping (host only, no device
 * memory): lays out the units of `n_linears` linears (rows[i] x cols[i],
 * elem_bytes 1 for E4M3 or 2 for BF16/F16 weights) as a tcgen05 decode launch
 * from slot views does - each linear's 256-row blocks in turn, each block
 * ceil(cols * elem_bytes / 128) K slabs, CTA c of `grid` taking units
 * [c*U/grid, (c+1)*U/grid) - and writes the settle tasks that launch would
 * run: one per row block that more than one CTA works on, 6 int32 each
 * (linear, row block, rows, first CTA, last CTA, partial slot of the first
 * CTA: 2c for its first run, 2c+1 for its last). Returns the number of tasks
 * (at most `capacity`), or SWS_E_INVALID for 1 <= n_linears <= 8,
 * cols % 16 == 0 or 1 <= grid <= min(U, 256) not holding. */
int sws_test_settle_plan(int32_t n_linears, const int64_t* rows, const int64_t* cols, int32_t elem_bytes,
                         int64_t grid, int32_t* out, int32_t capacity);

/* Failure-detection check: one kernel waits, with the bounded wait every
 * kernel of the library uses, on a barrier that nothing arrives at; after
 * limit_ns (0..1e8) it records SWS_E_TIMEOUT in the context's status word (as
 * a kernel whose TMA copy never landed would) and returns. The context stays
 * usable; sws_ctx_status reports and clears the code. With ctx == NULL the
 * code goes to the status word of sws_linear_noalloc's scratch on the current
 * device (read with sws_noalloc_status). */
int sws_test_bounded_wait(sws_ctx* ctx, int64_t limit_ns, sws_stream_t stream);

/* ---- misc --------------------------------------------------------------- */
const char* sws_last_error(void);
/* Library version as major*10000 + minor*100 + patch. */
int32_t sws_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SWS_H_ */
