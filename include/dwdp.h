/*
 * dwdp.h: C ABI of libdwdp.so, the single-rank hot path of DWDP
 * (Distributed Weight Data Parallelism) on one GB300 (sm_103a).
 *
 * Sources, cited by page title and section:
 *   [DWDP] "DWDP: Distributed Weight Data Parallelism for High-Performance LLM
 *          Inference on NVL72" (arXiv 2604.01621), as summarised on its
 *          summary pages;
 *   [news] the thecoregrid.dev news summary of the same paper.
 *
 * One rank runs one MoE block per layer.  Some experts of each layer are
 * resident ("local"); the others live on peers and are pulled into one of the
 * staging buffers (two by default: double buffering) by asynchronous copies
 * while the previous layer computes ([DWDP] §2 Methodology Overview).  The grouped GEMM reads each expert from
 * whichever buffer holds it through a per-expert table, with no merge copy
 * ([DWDP] §4.2).  Copies are cut into fixed-size slices issued round-robin
 * over the sources ([DWDP] §4.3.2; [news]).  On one GPU the peers are emulated
 * by separate device-memory pools.
 *
 * Conventions for every call:
 *   - bf16 tensors are raw 16-bit IEEE bfloat16; every matrix is row-major
 *     with no padding between rows.
 *   - "device" pointers point into the current CUDA device's global memory
 *     and must be 16-byte aligned; the caller owns every buffer it passes and
 *     keeps it alive until the work enqueued on it has finished.  Buffers
 *     the GEMMs read through TMA tensor maps (x, the workspace, the router
 *     weight, the local pool, the shared expert, the staging buffers) are
 *     checked to be device memory of the context's (current) device, else
 *     INVALID_ARG: the kernels never read another GPU's or the host's memory
 *     through a tensor map.  Only peer pools, which are copied from and
 *     never read by a kernel, may live elsewhere.
 *   - The context owns its CUDA events, tensor-map descriptors, its small
 *     device tables and error word, and the copy plans.  Use one context from
 *     one host thread at a time.
 *   - Every call validates its arguments on the host first.  A negative
 *     return means nothing was enqueued; dwdp_last_error() says why.
 *     Asynchronous CUDA faults surface as DWDP_ERR_CUDA from a later call.
 *   - Kernels never trap.  A bounded wait inside a kernel that runs out sets
 *     the context's device error word and returns; dwdp_device_status()
 *     reports it as DWDP_ERR_DEVICE_CHECK.
 *
 * Weight layouts:
 *   w13 of one expert : [2I][H]  rows 0..I-1 = W_gate^T, rows I..2I-1 = W_up^T
 *   w2  of one expert : [H][I]   = W_down^T
 *   a pool            : w13 [n_slots][2I][H] and w2 [n_slots][H][I]
 *   router weight     : [E][H]   row e = column e of the H x E gate matrix
 * Expert weights are bf16, 1-byte E4M3 codes in an E4M3 context, or NVFP4
 * slots (see DWDP_DTYPE_NVFP4) in an NVFP4 context; the router weight and
 * the activations passed in and out are always bf16.
 */
#ifndef DWDP_H_
#define DWDP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DWDP_ABI_VERSION 5
#define DWDP_MAX_EXPERTS 1024
#define DWDP_MAX_TOPK 32
#define DWDP_MAX_LAYERS 256
#define DWDP_MAX_PEERS 64

typedef struct dwdp_ctx dwdp_ctx;
/* Same object as cudaStream_t; NULL = the legacy default stream. */
typedef struct CUstream_st* dwdp_stream_t;

typedef enum {
    DWDP_OK = 0,
    DWDP_ERR_INVALID_ARG = -1,  /* bad pointer, size, index or alignment */
    DWDP_ERR_NOT_MAPPED = -2,   /* layer has no expert map, or stage holds another layer */
    DWDP_ERR_CUDA = -3,         /* a CUDA runtime call failed */
    DWDP_ERR_TIMEOUT = -4,      /* dwdp_wait_stage ran out of time */
    DWDP_ERR_UNSUPPORTED = -5,  /* shape outside what the kernels handle */
    DWDP_ERR_DEVICE_CHECK = -6  /* a kernel reported a failed check or wait */
} dwdp_status;

typedef struct {
    int32_t hidden;       /* H: multiple of 64 (NVFP4: of 256) */
    int32_t inter;        /* I: expert intermediate size, multiple of 64 (NVFP4: of 256) */
    int32_t n_experts;    /* E: routed experts, 1..DWDP_MAX_EXPERTS */
    int32_t top_k;        /* k: 1..min(E, DWDP_MAX_TOPK) */
    int32_t n_shared;     /* always-on shared experts: 0 or 1 */
    int32_t max_tokens;   /* largest T any call will pass */
    int32_t n_layers;     /* layers that get an expert map: 1..DWDP_MAX_LAYERS */
    int32_t stage_slots;  /* experts each staging buffer holds (0 = no staging) */
    int32_t weight_dtype; /* DWDP_DTYPE_BF16, DWDP_DTYPE_E4M3 or DWDP_DTYPE_NVFP4 */
    int32_t n_stages;     /* staging buffers: 0 = 2 (the pages' double buffering); 1..DWDP_MAX_STAGES */
    int32_t flags;        /* DWDP_FLAG_* (0 = defaults) */
} dwdp_config;

/* NVFP4 contexts: the gate/up GEMM drains its one TMEM accumulator with
 * eight epilogue warps (two per lane quarter) instead of four, so the next
 * tile's MMAs start sooner.  Faster when the GEMM runs alone; on one GPU a
 * copy-engine prefetch running beside it then gets much less of the memory
 * system (the copy, and with it the overlapped layer, takes longer), so it
 * is off by default.  Ignored by bf16 and E4M3 contexts. */
#define DWDP_FLAG_WIDE_EPILOGUE 1

#define DWDP_MAX_STAGES 4

/* Expert weight types.  DWDP_DTYPE_E4M3 (an FP8 variant of the layer; the
 * pages run NVFP4 expert weights, DWDP §5.1): pools and stage buffers hold
 * 1-byte E4M3 codes (w = code * scale, one scale per expert tensor, given by
 * dwdp_set_expert_scales); the layer quantizes its activations per row to
 * E4M3 (scale = row amax / 448, binary32, round-to-nearest-even,
 * saturating) before each expert GEMM, and the GEMMs run on FP8 tensor
 * cores.  Routing stays bf16. */
#define DWDP_DTYPE_BF16 0
#define DWDP_DTYPE_E4M3 1
/* DWDP_DTYPE_NVFP4 (the format the pages run DeepSeek-R1's MoE weights in,
 * DWDP §5.1): a weight is an E2M1 code (4 bits) times an E4M3 scale shared by
 * 16 consecutive elements along K, times one binary32 scale per expert tensor
 * (dwdp_set_expert_scales).  One pool slot of a [rows][K] tensor (w13: rows =
 * 2I, K = H; w2: rows = H, K = I) is rows * K * 9 / 16 bytes:
 *   - codes [rows][K / 2] bytes, element 2i of a row in the low nibble of
 *     byte i, 2i + 1 in the high nibble;
 *   - then the block scales in 512-byte chunks, one per (row block rb of 128
 *     rows, K step ks of 64 elements), chunk (rb, ks) at (rb * K / 64 + ks) *
 *     512; in it the scale of row 128 rb + 32 m1 + m0 and 16-element block kb
 *     of the step is byte 16 m0 + 4 m1 + kb.
 * The layer quantizes its activations per row to NVFP4 before each expert
 * GEMM (row scale = row amax / 2688 in binary32; block scale = E4M3 of block
 * amax / (6 * row scale); code = E2M1 of v / (block scale * row scale), round
 * to nearest even, saturating) and the GEMMs run on the block-scaled FP4
 * tensor cores.  H and I must be multiples of 256. */
#define DWDP_DTYPE_NVFP4 2

/* One buffer of experts: w13 [n_slots][2I][H], w2 [n_slots][H][I] (device;
 * NVFP4: n_slots slots of the sizes given at DWDP_DTYPE_NVFP4). */
typedef struct {
    const void* w13;
    const void* w2;
    int32_t n_slots;
} dwdp_pool;

/* Routing results (all device pointers, written by dwdp_route).
 *   topk_ids [T][k]  chosen experts of each token, ascending expert id
 *   topk_w   [T][k]  their weights: softmax renormalised over the chosen k
 *   counts   [E]     (token, slot) pairs routed to each expert
 *   offsets  [E+1]   exclusive scan of counts; offsets[E] = T*k
 *   perm     [T*k]   flat index t*k+j of the pair at grouped row r; within an
 *                    expert, rows keep ascending flat index
 *   inv_perm [T*k]   grouped row of pair t*k+j
 *   logits   [T][E]  fp32 router logits x.Wr (+ bias); NULL = not returned.
 *                    With few tokens the router GEMM splits K into up to 4
 *                    parts summed in order: the logits are the ones the
 *                    choice was made on, deterministic for a given device
 *                    and shape. */
typedef struct {
    int32_t* topk_ids;
    float* topk_w;
    int32_t* counts;
    int32_t* offsets;
    int32_t* perm;
    int32_t* inv_perm;
    float* logits;
} dwdp_route_out;

/* One slice of a prefetch copy plan.  tensor 0 = w13, 1 = w2; offsets are in
 * bytes from the start of the peer pool's tensor and the stage buffer's
 * tensor. */
typedef struct {
    int32_t peer;
    int32_t tensor;
    int64_t src_offset;
    int64_t dst_offset;
    int64_t nbytes;
} dwdp_copy_slice;

/* ABI version of the loaded library (DWDP_ABI_VERSION). */
int32_t dwdp_version(void);

/* Create a context on the current CUDA device.  stage_w13[s] / stage_w2[s]
 * (s = 0 .. n_stages - 1, n_stages = cfg->n_stages or 2 when that is 0) are
 * the caller's staging buffers ([DWDP] §2: double buffering; a third stage
 * lets the copy of layer l + 2 start while layer l computes, so the copy
 * stream can run back to back), each [stage_slots][2I][H] /
 * [stage_slots][H][I] in the weight format; they may be NULL when
 * cfg->stage_slots == 0.  On success *out owns the events and descriptors
 * listed above.  Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
int32_t dwdp_create(const dwdp_config* cfg, void* const stage_w13[], void* const stage_w2[],
                    dwdp_ctx** out);

/* Destroy a context (waits for nothing; the caller synchronises first). */
void dwdp_destroy(dwdp_ctx* ctx);

/* Text of the last error on this context (or of the last failed
 * dwdp_create / host helper when ctx is NULL).  Never NULL. */
const char* dwdp_last_error(const dwdp_ctx* ctx);

/* Device workspace, in bytes, that dwdp_route and dwdp_moe_layer need for T
 * tokens (the larger of the two; both may share one buffer when they run in
 * order on one stream). */
size_t dwdp_workspace_bytes(const dwdp_ctx* ctx, int32_t T);

/* Where dwdp_moe_layer keeps each intermediate of a T-token layer in its
 * workspace (instrumentation: after the layer has run, and until the next
 * call that uses the workspace, the caller may read them back).  Regions,
 * with rows_r = T k routed rows in expert order (dwdp_route's grouped rows)
 * and rows_all = T (k + n_shared) (the shared expert's rows after them):
 *   DWDP_WS_XP  [rows_r][H] x in expert order (bf16, E4M3 or NVFP4 codes)
 *   DWDP_WS_A   [rows_all][I] bf16 a = SiLU(gate) * up
 *   DWDP_WS_Y   [rows_all][H] bf16 expert outputs y
 *   DWDP_WS_XQ  [T][H] x's codes (E4M3 / NVFP4 contexts)
 *   DWDP_WS_SX, DWDP_WS_SXP  fp32 row scales of x by token / in expert order
 *   DWDP_WS_AQ  [rows_all][I] a's codes; DWDP_WS_SA [rows_all] fp32 a's row scales
 *   DWDP_WS_SFX, DWDP_WS_SFA  NVFP4 block scales of the gate/up and down
 *     GEMMs' A operands in the 512-byte chunk layout, chunk (tile, ks) at
 *     (tile * K / 64 + ks) * 512, where the A tiles are numbered expert by
 *     expert (ceil(rows_e / 128) tiles each, in expert order), then the
 *     shared expert's ceil(T / 128) tiles.
 * Writes the byte offset from ws and the region's size (0 when the context's
 * weight type has no such region).  Errors: INVALID_ARG. */
#define DWDP_WS_XP 0
#define DWDP_WS_A 1
#define DWDP_WS_Y 2
#define DWDP_WS_XQ 3
#define DWDP_WS_SX 4
#define DWDP_WS_SXP 5
#define DWDP_WS_AQ 6
#define DWDP_WS_SA 7
#define DWDP_WS_SFX 8
#define DWDP_WS_SFA 9
int32_t dwdp_workspace_region(const dwdp_ctx* ctx, int32_t T, int32_t region, size_t* offset, size_t* bytes);

/* Placement of layer `layer` ([DWDP] §2: experts partitioned across peers,
 * placement need not be disjoint; a redundant expert is read from its local
 * copy).  For each routed expert e:
 *   local_slot[e] >= 0  -> resident in `local` at that slot;
 *   otherwise peer_id[e] in [0, n_peers) and peer_slot[e] name its copy in
 *   peers[peer_id[e]], and it is staged by dwdp_prefetch_layer.
 * local_slot, peer_id, peer_slot are host arrays [E]; local and peers are host
 * structs describing device buffers (a peer pool may instead be pinned host
 * memory: its slices then cross the host link, and only their writes land in
 * this GPU's memory).  shared_w13 [2I][H] / shared_w2 [H][I]
 * (device) are the layer's shared expert, required iff n_shared == 1.  The
 * non-resident experts take stage slots 0, 1, ... in ascending id, at most
 * stage_slots of them.  Replaces any earlier map of the layer (the caller
 * makes sure no enqueued work still uses it).  Errors: INVALID_ARG, CUDA. */
int32_t dwdp_set_expert_map(dwdp_ctx* ctx, int32_t layer, const dwdp_pool* local,
                            const dwdp_pool* peers, int32_t n_peers, const int32_t* local_slot,
                            const int32_t* peer_id, const int32_t* peer_slot,
                            const void* shared_w13, const void* shared_w2);

/* Per-expert-tensor weight scales of layer `layer` for DWDP_DTYPE_E4M3 and
 * DWDP_DTYPE_NVFP4 contexts: expert e's gate/up weights are the w13 codes'
 * values * w13_scale[e], its down weights the w2 codes' values * w2_scale[e]
 * (host arrays [E]; NVFP4: on top of the block scales); shared_* for the
 * shared expert (ignored when n_shared == 0).  Required before
 * dwdp_moe_layer on such a context; kept until replaced.  Errors:
 * INVALID_ARG (bf16 context, bad layer, non-finite or non-positive scale). */
int32_t dwdp_set_expert_scales(dwdp_ctx* ctx, int32_t layer, const float* w13_scale, const float* w2_scale,
                               float shared_w13_scale, float shared_w2_scale);

/* Top-k routing with a deterministic grouping of the (token, slot) pairs by
 * expert.  x [T][H] bf16 and w_router [E][H] bf16 are device pointers;
 * logit_bias [E] fp32 (device) or NULL is added to every logit before the
 * choice.  The chosen experts are the k largest logits (softmax is
 * monotone), ties to the lower id, decided on the fp32 logits; weights are
 * exp(z_j - z_max) / sum over the chosen set.  ws (device, ws_bytes >=
 * dwdp_workspace_bytes) is scratch.  Enqueued on `stream`.  A token with
 * a logit that is not finite (NaN or +-inf, e.g. from a NaN in x) has no
 * defined choice: it still gets k distinct experts, but its ids and weights
 * are unspecified and the device error word is set (dwdp_device_status:
 * DEVICE_CHECK).  x and w_router must be device memory of the context's
 * device (they are read through TMA tensor maps).
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
int32_t dwdp_route(dwdp_ctx* ctx, const void* x, int32_t T, const void* w_router,
                   const float* logit_bias, const dwdp_route_out* out, void* ws, size_t ws_bytes,
                   dwdp_stream_t stream);

/* Pull layer `layer`'s non-resident experts from their peer pools into stage
 * buffer `stage` ([DWDP] §2: asynchronous prefetch of layer l+1 during layer
 * l, double-buffered; §4.3.2: fixed-size slices, round-robin over sources).
 * Each slice is one memcpy node (copy engine, no SMs) of at
 * most chunk_bytes in a CUDA graph that the context builds on first use for
 * this (chunk_bytes, stage, n_copy_streams) and keeps until the layer's map
 * is replaced; slices from peer p form chain p % n_copy_streams of the graph
 * (chains may run on separate copy engines), each chain in plan order.  The
 * graph is launched on copy_streams[0] (the other streams are not used)
 * after that stream waits until the last dwdp_moe_layer that read this
 * stage has finished reading it; completion is recorded as the stage's
 * "ready" event.  Errors: INVALID_ARG, NOT_MAPPED, CUDA. */
int32_t dwdp_prefetch_layer(dwdp_ctx* ctx, int32_t layer, int32_t stage, size_t chunk_bytes,
                            dwdp_stream_t const* copy_streams, int32_t n_copy_streams);

/* One MoE layer for T tokens on `stream` ([DWDP] §2 and §4.2):
 *   xp  = x rows copied into expert order (row route->inv_perm[t*k+j] = x[t])
 *   a   = SiLU(xp W_gate) * (xp W_up)          per expert, bf16
 *   y   = a W_down                             per expert, bf16
 *   out[t] = sum_j topk_w[t][j] y[inv_perm[t*k+j]] + y_shared[t]  (fp32 sum, bf16)
 * Each expert's weights come from the local pool or from stage `stage`, per
 * the layer's map; before the gate/up GEMM the stream waits for that stage's
 * "ready" event when the layer has non-resident experts (per-layer arrival,
 * [DWDP] §2).  route
 * holds dwdp_route's outputs for the same x (offsets, inv_perm and topk_w are
 * read; NVFP4 contexts also read topk_ids).  In E4M3 and NVFP4 contexts x
 * and a are quantized per row first (see DWDP_DTYPE_*) and the GEMMs run on
 * the codes.  out [T][H] bf16 (device).  An inv_perm entry outside
 * [0, T*k) is not followed: the kernels skip it (the token's output then
 * lacks that expert) and set the device error word, which
 * dwdp_device_status reports as DEVICE_CHECK.
 * Errors: INVALID_ARG, NOT_MAPPED, UNSUPPORTED, CUDA. */
int32_t dwdp_moe_layer(dwdp_ctx* ctx, int32_t layer, int32_t stage, const void* x, int32_t T,
                       const dwdp_route_out* route, void* out, void* ws, size_t ws_bytes,
                       dwdp_stream_t stream);

/* Activation quantization on its own, the same kernels and decisions as
 * dwdp_moe_layer applies to x and to a: x [rows][K] bf16 (device) to
 *   DWDP_DTYPE_E4M3: codes [rows][K] E4M3 bytes, row_scale [rows] fp32
 *     (amax / 448; block_scales unused);
 *   DWDP_DTYPE_NVFP4: codes [rows][K / 2] (two E2M1 codes per byte, element
 *     2i in the low nibble), row_scale [rows] fp32 (amax / 2688) and
 *     block_scales in the 512-byte chunk layout of DWDP_DTYPE_NVFP4 for a
 *     tensor of ceil(rows / 128) * 128 rows (bytes of rows past `rows` are
 *     not written).
 * K a multiple of 64; rows < 2^31.  All pointers device, 16-byte aligned.
 * Enqueued on `stream`; needs no context.  Errors: INVALID_ARG, CUDA. */
int32_t dwdp_quantize_rows(int32_t weight_dtype, const void* x, int64_t rows, int32_t K, void* codes,
                           void* block_scales, float* row_scale, dwdp_stream_t stream);

/* Host-side bounded wait for stage `stage`'s last prefetch: returns OK when
 * it has finished, TIMEOUT after timeout_ms (>= 0), CUDA on a fault. */
int32_t dwdp_wait_stage(dwdp_ctx* ctx, int32_t stage, int32_t timeout_ms);

/* Layer whose experts stage `stage` holds (or is being filled with), -1 if
 * none.  Host-side bookkeeping only. */
int32_t dwdp_stage_layer(const dwdp_ctx* ctx, int32_t stage);

/* Read and clear the device error word (synchronises the device).  OK, or
 * DEVICE_CHECK with the failing check described by dwdp_last_error: bits
 * 0-5 a bounded wait inside the grouped GEMM ran out, bit 6 an index outside
 * its buffer was skipped, bit 7 a router logit was not finite, bit 8 the
 * wait of dwdp_selftest_bounded_wait ran out (as that call intends). */
int32_t dwdp_device_status(dwdp_ctx* ctx);

/* Diagnostic (the pages have no counterpart): enqueues on `stream` one
 * one-thread kernel that waits, with the same bounded mbarrier wait every
 * grouped-GEMM role uses, for a barrier phase that nothing completes.  The
 * wait gives up after limit_us microseconds, sets bit 8 of the context's
 * device error word and the kernel returns: no trap, no hang, the context
 * stays usable.  The next dwdp_device_status then returns DEVICE_CHECK
 * (and clears the word).  limit_us in [1, 1000000].  Errors: INVALID_ARG,
 * CUDA. */
int32_t dwdp_selftest_bounded_wait(dwdp_ctx* ctx, uint32_t limit_us, dwdp_stream_t stream);

/* Optional phase timing.  events is a host array of DWDP_PHASE_EVENTS
 * caller-owned cudaEvent_t (or NULL to stop).  While set, dwdp_route records
 * events[0] at its start and events[1] at its end on its stream, and
 * dwdp_moe_layer records events[2] once x is in expert order (E4M3 / NVFP4:
 * quantized), events[3] after waiting for its stage (the layer puts x in
 * expert order before it waits: only the GEMMs read staged weights),
 * events[4] after the gate/up GEMM, events[5] after the down GEMM and
 * events[6] after the combine.  The context keeps the pointers
 * until the next call; the caller keeps the events alive.  Errors:
 * INVALID_ARG (a NULL event or a wrong count; the previous events, or
 * none, stay in effect). */
#define DWDP_PHASE_EVENTS 7
int32_t dwdp_set_phase_events(dwdp_ctx* ctx, void* const* events, int32_t n_events);

/* Split-pointer grouped GEMM on its own ([DWDP] §4.2: one kernel over several
 * weight buffers, no merge).  For each group g in [0, G):
 *   rows r in [row_offsets[g], row_offsets[g+1]) of a [rows][K] bf16:
 *   d[r][n] = sum_k a[r][k] * B_g[n][k],  B_g = slot buf_slot[2g+1] of
 *   buffer bufs[buf_slot[2g]] (each buffer [n_slots][N_b][K] bf16).
 * epilogue 0: d bf16 [rows][N], B_g has N rows.
 * epilogue 1: d bf16 [rows][N] = SiLU(gate) * up with gate = rows 0..N-1 and
 *             up = rows N..2N-1 of B_g (B_g has 2N rows).
 * epilogue 2: d fp32 [rows][N], B_g has N rows.
 * row_offsets is a DEVICE array [G+1] (non-decreasing, row_offsets[G] <=
 * a_rows; rows outside [0, a_rows) are not stored and raise DEVICE_CHECK);
 * buf_slot is a HOST array [2G]; bufs is a host array of n_bufs <= 3 buffers
 * of which only .w13 (the base) and .n_slots are read.
 * K and N multiples of 64 (epilogue 2: N any value >= 1).  Enqueued on
 * `stream`; uses no workspace.  Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
int32_t dwdp_grouped_gemm(dwdp_ctx* ctx, int32_t epilogue, const void* a, int64_t a_rows, int32_t K,
                          int32_t N, const int32_t* row_offsets, int32_t G, const dwdp_pool* bufs,
                          int32_t n_bufs, const int32_t* buf_slot, void* d, dwdp_stream_t stream);

/* Routing that allocates no device memory (the paper has no counterpart: it
 * serves callers that cannot call cudaMalloc where they route tokens, e.g. a
 * framework whose caching allocator owns all device memory, a latency-bound
 * serving loop that cannot afford the synchronisation cudaMalloc may imply,
 * or a host with a memory budget fixed at start-up).
 * Computes exactly what dwdp_route computes (same kernels, same results) for
 * x [T][hidden], w_router [n_experts][hidden], logit_bias [n_experts] or
 * NULL, without a context or workspace; out->logits is ignored (the logits
 * stay in the scratch).  Its scratch is one file-scope device array of
 * 32 MiB + 256 bytes: DWDP_STATIC_SCRATCH_BYTES (16 MiB) of fp32 logits, as
 * much again for the router GEMM's partial sums (its K may be split into
 * parts as in dwdp_route, which always fit on GPUs with up to 256 SMs) and a
 * 256-byte error word, held by every GPU that loads this library until the
 * process exits, so T * n_experts * 4 must not exceed
 * DWDP_STATIC_SCRATCH_BYTES (else INVALID_ARG, nothing enqueued).  The first
 * call on each device (of this entry point or of dwdp_route_static_status)
 * looks up the array's device address (cudaGetSymbolAddress) with that
 * device current and keeps it for the life of the process; make that first
 * call before any stream capture, and do not use these two calls on a
 * device after cudaDeviceReset (the address belonged to the context the
 * reset destroyed).  Every call on a device shares the one array and it
 * keeps the last call's contents (the error word is cleared on `stream` at
 * the start of each call): calls whose work overlaps on the GPU (other
 * streams, other threads) race on it.  Device-side failures (a non-finite
 * logit as in dwdp_route, a bounded wait that ran out) set the array's
 * error word: read it with dwdp_route_static_status.  Calls no cudaMalloc,
 * cudaFree or other allocating routine.  Errors (text in
 * dwdp_last_error(NULL)): INVALID_ARG, UNSUPPORTED, CUDA. */
#define DWDP_STATIC_SCRATCH_BYTES (16u << 20)
int32_t dwdp_route_static(const void* x, int32_t T, int32_t hidden, int32_t n_experts, int32_t top_k,
                          const void* w_router, const float* logit_bias, const dwdp_route_out* out,
                          dwdp_stream_t stream);

/* The device error word of dwdp_route_static on the current device (no
 * counterpart in the paper; dwdp_route_static has no context whose
 * dwdp_device_status could report it).  Waits for the work already enqueued
 * on `stream` (not allowed while `stream` is being captured), reads the word
 * and, when it is non-zero, clears it on `stream`.  *bits (may be NULL)
 * receives the raw bits (as for dwdp_device_status).  Returns OK for a zero
 * word, DEVICE_CHECK otherwise (text in dwdp_last_error(NULL)).  Allocates
 * nothing.  Errors: CUDA, UNSUPPORTED. */
int32_t dwdp_route_static_status(dwdp_stream_t stream, int32_t* bits);

/* Host-only (no GPU needed): the prefetch copy plan dwdp_prefetch_layer
 * issues for a map ([DWDP] §4.3.2).  The non-resident experts (local_slot <
 * 0) take stage slots in ascending id; each peer's work is its w13 copies then
 * its w2 copies in ascending expert id, merged where contiguous in both
 * source and destination, cut into slices of chunk_bytes (the last one
 * short); slices are emitted round-robin over peers 0..n_peers-1.  Writes up
 * to max_out slices to out (may be NULL when max_out == 0) and the full count
 * to *n_out.  weight_dtype (DWDP_DTYPE_*) sets the bytes of one expert
 * tensor.  Errors: INVALID_ARG (bad map or a non-resident expert with no
 * peer copy). */
int32_t dwdp_plan_prefetch(int32_t n_experts, int32_t hidden, int32_t inter, int32_t weight_dtype,
                           const int32_t* local_slot, const int32_t* peer_id,
                           const int32_t* peer_slot, int32_t n_peers, size_t chunk_bytes,
                           dwdp_copy_slice* out, int64_t max_out, int64_t* n_out);

/* Host-only (no GPU needed): the expert map of rank `rank` in a DWDP group
 * of n_ranks ranks ([DWDP] §2: each rank keeps a partition of the experts
 * and pulls the rest from its peers; §4.3.1-§4.3.2: the pulls of several
 * destinations from one source contend, so slices are issued round-robin).
 * Rank q hosts experts [floor(q E / N), floor((q + 1) E / N)) in slots
 * 0, 1, ... of its pool.  Fills local_slot [E] (the slot for this rank's own
 * experts, else -1), and for the others peer_id [E] and peer_slot [E] (-1 for
 * own experts), numbering this rank's peers from the next rank on: peer p
 * is rank (rank + 1 + p) mod n_ranks, so the peers array given to
 * dwdp_set_expert_map lists the other ranks' pools in that order.  With this
 * numbering the round-robin of dwdp_plan_prefetch has every rank, at the
 * same step of its plan, pulling from a different source (when every rank
 * hosts the same number of experts), so no source serves two destinations
 * at once.  A map for placement only: the pulls themselves are copy-engine
 * memcpy nodes whose source may be any memory the copy engine reaches.
 * Errors: INVALID_ARG. */
int32_t dwdp_group_map(int32_t n_experts, int32_t n_ranks, int32_t rank, int32_t* local_slot, int32_t* peer_id,
                       int32_t* peer_slot);

#ifdef __cplusplus
}
#endif

#endif /* DWDP_H_ */
