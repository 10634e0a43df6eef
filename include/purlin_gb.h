/*
 * purlin_gb.h - C ABI of the collective datapath for one GB300 (sm_103a).
 *
 * What the library computes.  Purlin's collectives (Purlin README, purlin
 * 0.6.4: summary paragraph and "Key Idea") are built from two datapath
 * primitives, a copy and an N-to-1 reduce that sums several input buffers into
 * one output, driven by layouts that say which bytes go where and whether they
 * are copied or reduced, and by the Stage, Notify And Consume (SNAC) protocol.
 * Here the `world` ranks of a collective are `world` separate buffers in the
 * HBM of one GPU: rank r's input is src[r] and its output is dst[r].
 *
 * Semantics of each collective follow AWS Neuron NKI, "Collective
 * Communication Kernels API Reference" (dim-0 definitions and the worked
 * all-reduce example); the V variants are named in the Purlin README summary.
 * Reductions are deterministic (Purlin README, "Reduction determinism"): every
 * output element is the binary32 left fold, in ascending rank order starting
 * from rank 0's value, of the ranks' elements, rounded once to the output type
 * (bf16: nearest, ties to even).  Results are bit-identical from call to call.
 *
 * Conventions shared by every entry point:
 *   - Pointers in src[] / dst[] are owned by the caller and point to memory
 *     the handle's device can address: its own device memory, managed
 *     memory, or pinned host memory (cudaHostAlloc, or pageable memory after
 *     cudaHostRegister).  The kernel reads and writes host memory in place
 *     over the host link (no staging copies; such calls run on the register
 *     path).  Any other pointer -- unregistered pageable memory included --
 *     returns PL_ERR_INVALID_ARG.  The host arrays src[], dst[], bytes[] are
 *     read during the call only.
 *   - `bytes` arguments count bytes, not elements.
 *   - Every collective is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  Argument errors are returned at once and
 *     nothing is launched.  Errors found on the device (a SNAC wait that ran
 *     out of time) are recorded in the handle's device status word and
 *     reported by purlin_status_get().
 *   - A call that moves zero bytes returns PL_OK without launching anything.
 *   - Destination ranges must not overlap each other or any source range.
 *     The one exception is in-place AllReduce, src[r] == dst[r].
 *   - Sizes whose sums (a V collective's totals, an AllGather's world x bytes)
 *     or whose buffer ends do not fit in 64 bits return PL_ERR_INVALID_ARG.
 *     The library cannot see how large the caller's allocations are: byte
 *     counts larger than the buffers they describe are the caller's error.
 *   - Reductions need every pointer aligned to the element size; copies take
 *     any byte alignment.  16-byte alignment of every address is the fast path.
 *   - Calls on one handle must be ordered (one stream, or streams the caller
 *     orders): they share the handle's workspace.  They must be made with the
 *     handle's device current (the one current at purlin_initialize); other
 *     calls return PL_ERR_INVALID_ARG.
 *   - The first call of a given shape builds its plan (a small host
 *     computation plus one upload); make it before capturing the stream into
 *     a CUDA graph.
 */
#ifndef PURLIN_GB_H
#define PURLIN_GB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PURLIN_MAX_WORLD 16
/* SNAC flags of the workspace the library allocates when purlin_initialize is
 * given none (8 MiB of flags): the two-shot and ring AllReduce layouts at the
 * tuning table's tile sizes for up to 8 ranks of about 9 GiB each, or 16
 * ranks of about 4 GiB. */
#define PURLIN_DEFAULT_WORKSPACE_FLAGS 2097152u

typedef struct purlin_ctx* purlin_handle;
typedef void* purlin_stream_t; /* a cudaStream_t */

typedef enum {
  PL_OK = 0,
  PL_ERR_INVALID_ARG = 1,  /* null pointer, bad world, sizes that do not split or overflow, overlap */
  PL_ERR_ALIGNMENT = 2,    /* a reduce pointer or size not aligned to the element size */
  PL_ERR_UNSUPPORTED = 3,  /* e.g. a reduction over PL_U8, an unknown mode or layout */
  PL_ERR_WORKSPACE = 4,    /* caller-provided workspace too small for this call */
  PL_ERR_CUDA = 5,         /* a CUDA runtime call failed */
  PL_ERR_LAUNCH = 6,       /* the kernel could not be launched */
  PL_ERR_TIMEOUT = 7,      /* device: a SNAC consume wait gave up */
  PL_ERR_FINALIZED = 8,    /* the handle was finalized */
  PL_ERR_BOUNDS = 9        /* device, checking build only: a work item reached outside a rank buffer */
} purlin_status;

typedef enum { PL_U8 = 0, PL_F32 = 1, PL_BF16 = 2 } purlin_dtype;

/* Purlin README, "Reduction determinism".  Only the deterministic mode exists
 * here: the other mode of the pages needs a multicast fabric across GPUs. */
typedef enum { PL_DETERMINISTIC = 0 } purlin_mode;

typedef enum {
  PL_COLL_ALL_REDUCE = 0,
  PL_COLL_REDUCE_SCATTER = 1,
  PL_COLL_ALL_GATHER = 2,
  PL_COLL_ALL_TO_ALL = 3,
  PL_COLL_ALL_GATHER_V = 4,
  PL_COLL_ALL_TO_ALL_V = 5,
  PL_COLL_REDUCE_SCATTER_V = 6,
  PL_COLL_ATOM_COPY = 7,
  PL_COLL_ATOM_REDUCE = 8
} purlin_coll;

/* AllReduce layouts (Iris docs, "Device Context", all_reduce_one_shot,
 * all_reduce_two_shot and all_reduce_ring).  One-shot: every byte range is
 * reduced once and the sum stored to all ranks.  Two-shot: rank o reduces
 * range o into its own output and notifies; a consumer then copies that range
 * to every other rank.  Ring: per tile, a running sum handed from rank to
 * rank -- stage k adds rank k's elements to the sum the previous stage left
 * in the outputs, each stage waiting for the previous one's flag -- then the
 * finished tile is passed around the ring, output to output.  The running sum
 * is kept in binary32 (for bf16 data as two 16-bit halves in two ranks'
 * outputs) and every tile is walked from rank 0 upwards, so all three
 * layouts give the ascending-rank fold described above, bit for bit.  The
 * ring moves about three times the bytes of the one-shot layout; only on
 * request, AUTO never picks it.  Register path only (PL_ERR_UNSUPPORTED
 * otherwise). */
typedef enum {
  PL_LAYOUT_AUTO = 0,
  PL_LAYOUT_ONE_SHOT = 1,
  PL_LAYOUT_TWO_SHOT = 2,
  PL_LAYOUT_RING = 3,
  /* The two-shot layout with fused items: after a first wave of reduces, each
   * item reduces one owner tile and, in the same pass, copies a tile another
   * CTA reduced one wave earlier (its SNAC wait), so every CTA streams the
   * one-shot layout's mix of reads and writes.  Same results.  Register path,
   * item schedule and store_hint 3 only (PL_ERR_UNSUPPORTED otherwise); only on
   * request. */
  PL_LAYOUT_TWO_SHOT_FUSED = 4
} purlin_layout;

/* Tuning of one call (the role of Purlin's host tuning policies).  A zero field
 * means "take the tuning table's value". */
typedef struct {
  int layout;       /* purlin_layout; AllReduce only */
  int ctas_per_sm;  /* persistent CTAs per SM (grid = ctas_per_sm x SMs, capped by work) */
  int threads;      /* threads per CTA: a multiple of 32 in [64, 512] */
  int unroll;       /* 16-byte vectors in flight per thread per source, 1..8 */
  int path;         /* 1 = register path, 2 = TMA bulk pipeline through shared memory */
  int chunk_bytes;  /* TMA stage size per source, or SNAC tile size of the two-shot and ring
                       layouts (ring default: a 64th of bytes_per_rank / world, kept
                       between 64 and 128 KiB) */
  int stages;       /* TMA pipeline depth, 2..8 */
  int store_hint;   /* register path: 1 = write-back stores, 2 = streaming (evict-first)
                       stores; 3 = L2 priorities of the two-shot AllReduce (only there,
                       else PL_ERR_INVALID_ARG): reduce inputs loaded evict-first, owner
                       tiles stored evict-last until their copies have read them, copies
                       stored evict-first */
  int min_cta_bytes;/* fewest work bytes given to one CTA before the grid shrinks */
  int interleave_bytes; /* a multiple of 512: the work is cut into k x grid parts of about
                           this size and CTA c takes parts c, c + grid, ...; -1: one
                           contiguous share per CTA (0 = the table's choice) */
  int max_ctas;     /* > 0: at most this many CTAs (fewer concurrent DRAM streams) */
  int schedule;     /* purlin_schedule: how CTAs walk their items */
  int snac_lag;     /* two-shot and ring AllReduce: a flag's consumer comes about snac_lag x
                       grid / 2 places after its producer in the items' order (1..64;
                       table: 2, one wave of CTAs) */
} purlin_tune;

/* How the CTAs of a launch walk the plan's work items (purlin_tune.schedule).
 * PL_SCHED_ITEM: each CTA runs its own share one item at a time (on the bulk
 * path every item fills and drains its own pipeline).  PL_SCHED_STREAM: a
 * CTA's items flow through one continuous bulk pipeline.  PL_SCHED_QUEUE:
 * streamed, and CTAs take items in order from a counter the grid shares
 * (the plan's parts are about interleave_bytes, else 256 KiB), so CTAs that
 * get more DRAM bandwidth take more items.  STREAM serves copy collectives on
 * the bulk path (path = 2).  QUEUE serves every collective on the register
 * path (path = 1; two-shot SNAC plans included: an item only waits on
 * earlier items, so the earliest unfinished item always runs) and copy
 * collectives on the bulk path.  QUEUE_GUIDED is the queue with parts that
 * shrink as the work runs out: each is 1/(2 x grid) of what is left, kept
 * between T and 4 T bytes (T = interleave_bytes, else 256 KiB), so the
 * first parts are larger (fewer items) and the last ones small (CTAs that
 * run slower finish at nearly the same time).  Other combinations return
 * PL_ERR_UNSUPPORTED. */
typedef enum { PL_SCHED_ITEM = 1, PL_SCHED_STREAM = 2, PL_SCHED_QUEUE = 3, PL_SCHED_QUEUE_GUIDED = 4 } purlin_schedule;

/* One work item of a plan, as purlin_plan_describe reports it. */
typedef struct {
  uint64_t src_off;  /* byte offset into every source buffer the item reads */
  uint64_t dst_off;  /* byte offset into every destination buffer it writes */
  uint64_t len;      /* bytes */
  uint32_t src_mask; /* bit r (r < 16): input of rank r; bit 16 + r: output of rank r.
                        Several bits = N-to-1 reduce in ascending bit order. */
  uint32_t dst_mask; /* bit r (r < 16): output of rank r.  Bits 30 and 31 mark the ring
                        layout's reduce items over bf16 data, whose running binary32 sum is
                        kept as two 16-bit halves in two neighbouring ranks' outputs (low
                        half in the lower rank): bit 30, the item's two output sources are
                        those halves; bit 31, its two destinations receive the halves of
                        the new sum instead of a rounded bf16 value.  Bit 29 marks a fused
                        two-shot item: it reduces the tile at src_off (its input bits) into
                        the output of its one destination bit and, in the same pass, copies
                        the tile at dst_off from the output of its output source bit to
                        every other rank's output; it notifies the flag of the tile it
                        reduces and waits for the flag of the tile it copies. */
  uint32_t wait;     /* 0, or 1 + index of the SNAC flag consumed before the item */
  uint32_t notify;   /* 0, or 1 + index of the SNAC flag raised after the item */
  uint32_t cta;      /* CTA that runs the item; 0xFFFFFFFF under PL_SCHED_QUEUE (any CTA) */
  uint32_t order;    /* position of the item in that CTA's sequence (in the queue) */
} purlin_item;

/* ---------------------------------------------------------------- set-up */

/* Bytes of workspace a handle needs for collectives of up to
 * `max_bytes_per_rank` per rank (the SNAC signal flags plus a status word).
 * Role of the pages' workspace of staging and signal buffers (purlin 0.6.5,
 * "Host-side").  Returns 0 for a world outside [1, PURLIN_MAX_WORLD]. */
size_t purlin_workspace_bytes(int world, size_t max_bytes_per_rank);

/* Create a handle for `world` ranks on the current CUDA device (purlin 0.6.5,
 * "Host-side": create once, reuse for every collective).  `workspace` is
 * device memory owned by the caller, of `workspace_bytes` bytes, 256-byte
 * aligned; it never grows, and a call whose plan needs more flags than it
 * holds returns PL_ERR_WORKSPACE.  Pass NULL to let the library allocate its
 * own: workspace_bytes, or PURLIN_DEFAULT_WORKSPACE_FLAGS flags if that is
 * larger (size it with purlin_workspace_bytes for the largest call you will
 * make).  A later call that needs more flags than a library-owned workspace
 * holds grows it, once per growth: the call waits for `stream`, allocates a
 * larger workspace, zeroes it and frees the old one (cudaMalloc and cudaFree
 * may synchronise the whole device); under stream capture it returns
 * PL_ERR_WORKSPACE instead.  purlin_workspace_query reports the size and the
 * growths.  The workspace is zeroed on `stream` before the call returns.  On
 * success *out holds the handle. */
purlin_status purlin_initialize(int world, void* workspace, size_t workspace_bytes,
                                purlin_stream_t stream, purlin_handle* out);

/* Free what the library allocated for the handle, after work queued on
 * `stream` is done (purlin 0.6.5, "Host-side": finalize after the last
 * collective).  Returns the first device error still pending, if any. */
purlin_status purlin_finalize(purlin_handle h, purlin_stream_t stream);

/* ----------------------------------------------------------- collectives */

/* AllReduce (NKI all_reduce_hbm_kernel: sum tensors across ranks): dst[r][i] =
 * sum over s of src[s][i] for every r, folded as described at the top, in
 * every layout (purlin_layout).  bytes_per_rank = size of each input and each
 * output.  dtype PL_F32 or PL_BF16.  In-place (src[r] == dst[r]) is allowed. */
purlin_status purlin_all_reduce(purlin_handle h, const void* const* src, void* const* dst,
                                size_t bytes_per_rank, purlin_dtype dtype, purlin_mode mode,
                                purlin_stream_t stream);

/* ReduceScatter (NKI reduce_scatter_hbm_kernel: sum, then dim 0 is split into
 * world chunks): dst[r][j] = sum over s of src[s][r*c + j], c = elements per
 * chunk.  in_bytes_per_rank must split into world chunks of whole elements;
 * each output holds in_bytes_per_rank / world bytes. */
purlin_status purlin_reduce_scatter(purlin_handle h, const void* const* src, void* const* dst,
                                    size_t in_bytes_per_rank, purlin_dtype dtype, purlin_mode mode,
                                    purlin_stream_t stream);

/* AllGather (NKI all_gather_hbm_kernel: gather along dim 0): dst[r] = src[0] ||
 * src[1] || ... || src[world-1] for every r.  in_bytes_per_rank is the size of
 * each input; each output holds world * in_bytes_per_rank bytes. */
purlin_status purlin_all_gather(purlin_handle h, const void* const* src, void* const* dst,
                                size_t in_bytes_per_rank, purlin_stream_t stream);

/* AllToAll (NKI all_to_all_hbm_kernel: rank i receives chunk i of every
 * input): dst[d][s*c .. s*c+c) = src[s][d*c .. d*c+c), c = bytes_per_rank /
 * world.  bytes_per_rank (each input and each output) must split into world
 * equal chunks. */
purlin_status purlin_all_to_all(purlin_handle h, const void* const* src, void* const* dst,
                                size_t bytes_per_rank, purlin_stream_t stream);

/* AllGatherV (Purlin README: variable-length AllGather): dst[r] = the first
 * bytes[0] bytes of src[0] || ... || the first bytes[world-1] bytes of
 * src[world-1], packed in rank order, for every r.  bytes has world entries. */
purlin_status purlin_all_gather_v(purlin_handle h, const void* const* src, void* const* dst,
                                  const size_t* bytes, purlin_stream_t stream);

/* AllToAllV (Purlin README: variable-length AllToAll).  bytes[s*world + d]
 * bytes go from rank s to rank d.  Rank s sends its block for d from offset
 * sum_{d'<d} bytes[s*world+d']; rank d stores the block from s at offset
 * sum_{s'<s} bytes[s'*world+d]. */
purlin_status purlin_all_to_all_v(purlin_handle h, const void* const* src, void* const* dst,
                                  const size_t* bytes, purlin_stream_t stream);

/* ReduceScatterV (Purlin README: variable-length ReduceScatter).  Every input
 * holds sum_r bytes[r] bytes; dst[r] receives bytes[r] bytes, the sum over s
 * of src[s] from offset sum_{r'<r} bytes[r'].  Each bytes[r] must be a whole
 * number of elements. */
purlin_status purlin_reduce_scatter_v(purlin_handle h, const void* const* src, void* const* dst,
                                      const size_t* bytes, purlin_dtype dtype, purlin_mode mode,
                                      purlin_stream_t stream);

/* ----------------------------------------------------------------- Atoms */

/* Copy Atom (purlin 0.6.5, "Samples": threads of a CTA copy one slice; src
 * and dst may be anywhere in device memory): dst[d][0..bytes) =
 * src[0..bytes) for each of the ndst destinations, spread over the grid. */
purlin_status purlin_atom_copy(purlin_handle h, const void* src, void* const* dst, int ndst,
                               size_t bytes, purlin_stream_t stream);

/* N-to-1 reduce Atom (Purlin README: combines several input buffers into one
 * output): dst[d][i] = sum over s < nsrc of src[s][i] (ascending fold) for each
 * of the ndst destinations.  bytes = size of each buffer. */
purlin_status purlin_atom_reduce(purlin_handle h, const void* const* src, int nsrc,
                                 void* const* dst, int ndst, size_t bytes, purlin_dtype dtype,
                                 purlin_stream_t stream);

/* ------------------------------------------------------ status and tuning */

/* Wait for `stream`'s queued work, then report (and clear) the first error
 * recorded on the device since the last call: *device_status = PL_OK or
 * PL_ERR_TIMEOUT.  Returns PL_OK when the query itself worked. */
purlin_status purlin_status_get(purlin_handle h, purlin_stream_t stream, int* device_status);

const char* purlin_status_string(purlin_status s);

/* The tuning the handle would use for a call: table entry, then the
 * handle's override, then the layout's own defaults (two-shot and ring
 * AllReduce) and the thread cap of the register path beyond 8 sources. */
purlin_status purlin_tune_get(purlin_handle h, purlin_coll coll, purlin_dtype dtype,
                              size_t bytes_per_rank, purlin_tune* out);

/* Override the tuning table for every later call on the handle (non-zero
 * fields win); NULL restores the table.  Used by the tuning sweep. */
purlin_status purlin_tune_override(purlin_handle h, const purlin_tune* t);

/* Test hook of the checking build (libpurlin_gb_debug.so, compiled with
 * PURLIN_DEBUG): every kernel checks each work item against the byte count
 * of every rank buffer it touches before it moves any data; an item that
 * would reach outside is skipped (its SNAC notify still raised) and the
 * device status reads PL_ERR_BOUNDS.  This hook makes the next launch on the
 * handle believe that buffer `rank` (an input if is_output is 0, else an
 * output) holds only `bytes` bytes, so a test can see the check fire without
 * any access outside a buffer.  In the normal build the call is accepted and
 * has no effect (there is no check to fire). */
purlin_status purlin_debug_limit_buffer(purlin_handle h, int is_output, int rank, uint64_t bytes);

/* Test hook: set the SNAC epoch counter of the handle (the epoch the last
 * launch with SNAC flags used), in stream order.  Launches of SNAC plans use
 * epochs 1 .. 0xFFFFFFFF, one per launch, and flags are ready when they hold
 * the launch's epoch; the launch that used 0xFFFFFFFF clears every flag and
 * publishes 0, and the counter starts again at 1.  Setting the counter near
 * the end of the cycle lets a test run that wrap without 2^32 launches.  The
 * counter only ever holds 0 .. 0xFFFFFFFE: 0xFFFFFFFF is refused
 * (PL_ERR_INVALID_ARG; the next launch would take epoch 0, the value of a
 * cleared flag, and its consumers would not wait).  Waits for the stream;
 * refused (PL_ERR_INVALID_ARG) while the stream is being captured. */
purlin_status purlin_debug_set_epoch(purlin_handle h, uint32_t epoch, purlin_stream_t stream);

/* The same for purlin_all_reduce_noalloc's scratch on the current device. */
purlin_status purlin_debug_noalloc_set_epoch(uint32_t epoch, purlin_stream_t stream);

/* Test hook for purlin_all_reduce_noalloc: its next call (on any device) waits
 * at most `timeout_ns` in each SNAC consume (0: the default 2 s) and skips the
 * notify of the reduce of flag `drop_tile` (owner o's tile t is flag
 * o x T + t, T = tiles of the largest owner range; -1: none), so a test can
 * make a wait run out and read PL_ERR_TIMEOUT from its status word.  Applies
 * to one call, then clears.  drop_tile >= 16384 returns PL_ERR_INVALID_ARG. */
purlin_status purlin_debug_noalloc_next(uint64_t timeout_ns, long long drop_tile);

/* Time limit of every SNAC consume wait, in nanoseconds (default 2e9). */
purlin_status purlin_set_wait_timeout_ns(purlin_handle h, uint64_t ns);

/* Test hook: the next launch on the handle skips the notify of its item with
 * index `item` (plan order), so the consumer of that flag runs out of time and
 * the device status reads PL_ERR_TIMEOUT.  -1 clears. */
purlin_status purlin_debug_drop_notify(purlin_handle h, long long item);

/* Trace every work item of later calls on the handle into `buffer`, device
 * memory owned by the caller, 8-byte aligned, `buffer_bytes` long (Iris docs,
 * "Device Context": device-side event tracing of a collective).  Layout: one
 * 64-bit count of records, then 32-byte records {u64 start_ns, u64 end_ns,
 * u32 cta, u32 item, u32 wait_ns, u32 length_KiB} in completion order, times
 * from %globaltimer.  The caller zeroes the count before the calls it wants
 * traced; records beyond the buffer's capacity are counted, not written.
 * NULL stops tracing. */
purlin_status purlin_trace_enable(purlin_handle h, void* buffer, size_t buffer_bytes);

/* Workspace of the handle: its size in bytes and how many times the library
 * has grown it (always 0 for a caller's workspace).  Either pointer may be NULL. */
purlin_status purlin_workspace_query(purlin_handle h, size_t* bytes, int* grown);

/* Device facts the handle uses: SM count, compute capability (major*10+minor),
 * and the largest number of CTAs of the reduce kernel resident per SM. */
purlin_status purlin_query(purlin_handle h, int* sm_count, int* arch, int* max_ctas_per_sm);

/* ------------------------------------------------- allocation-free variant */

/* AllReduce (two-shot layout, same results as purlin_all_reduce: the
 * ascending-rank binary32 fold, bit for bit) for callers that must not
 * allocate device memory once running -- a runtime whose memory is fixed at
 * start-up, a plug-in that has to stay inside its host framework's memory
 * pool, code that cannot take the device-wide synchronisation cudaMalloc /
 * cudaFree may cause.  The source pages have no counterpart to this call.
 *
 * It needs no handle and calls no allocating routine.  Its scratch (SNAC
 * flags and control words, about 64 KiB) is a static array in the library,
 * present on every GPU that loads it until the process exits.  The first call
 * on a device looks up that array's device address and zeroes it on `stream`;
 * make that first call before any stream capture.  Every call on a device
 * shares the array: calls that overlap on the GPU (unordered streams) race
 * and must not be made; calls ordered on one stream are fine.
 *
 * world in [1, PURLIN_MAX_WORLD]; src / dst as for purlin_all_reduce (in place
 * allowed).  Size limit: world * ceil(largest rank share / 64 KiB) <= 16384
 * tiles, where a rank share is bytes_per_rank / world rounded up to whole
 * elements -- about 1 GiB per rank; larger sizes return PL_ERR_WORKSPACE and
 * launch nothing.  device_status: NULL, or device memory the caller owns that
 * receives PL_OK or PL_ERR_TIMEOUT (a SNAC wait gave up after 2 s) when the
 * kernel ends.  A call that timed out leaves its outputs partly written; with
 * a NULL device_status nothing reports it (the failure is kept only in the
 * library's scratch, which no call reads back), so pass a status word
 * wherever a time-out must be noticed.  Asynchronous on `stream`. */
purlin_status purlin_all_reduce_noalloc(int world, const void* const* src, void* const* dst,
                                        size_t bytes_per_rank, purlin_dtype dtype, int* device_status,
                                        purlin_stream_t stream);

/* ------------------------------------------------------- host-only plans */

/* The plan a call would run, computed on the host with no GPU: the layout
 * (pieces of copy / reduce work, Purlin README "Key Idea": layouts describe
 * the collective) split into per-CTA work items.  `sizes` is the size
 * argument of the collective: one value (bytes per rank) for AllReduce,
 * ReduceScatter, AllGather, AllToAll; `world` values for AllGatherV and
 * ReduceScatterV; world*world values for AllToAllV.  `src_addr` / `dst_addr`
 * (world entries each, may be NULL = all 256-byte aligned) supply the buffer
 * addresses whose low bits decide alignment.  `tune` may be NULL (table).
 * Writes up to `cap` items; *n_items receives the total, *grid the CTA count,
 * *n_flags the SNAC flags used. */
purlin_status purlin_plan_describe(purlin_coll coll, int world, purlin_dtype dtype,
                                   const size_t* sizes, const uint64_t* src_addr,
                                   const uint64_t* dst_addr, int sm_count,
                                   const purlin_tune* tune, purlin_item* items, size_t cap,
                                   size_t* n_items, int* grid, int* n_flags);

#ifdef __cplusplus
}
#endif

#endif /* PURLIN_GB_H */
