/*
 * moe.h -- C ABI of libmoe_gb300.so: a routed Mixture-of-Experts layer with
 * Q8_0 (or Q4_0) SwiGLU experts, hand-written for NVIDIA GB300 (sm_103a).
 *
 * The layer (qwen3_moe geometry: d_model 2048, d_ff 768, 128 experts, top-8,
 * 48 layers -- amalgafy.com/evidence, "Historical baseline environment"):
 *
 *   router   l[t][e] = x[t] . Wr[e] (+ bias[e])        "LinearGate" routing,
 *                                                        amalgafy.com/evidence
 *   top-k    the k largest logits, ties to the lower expert id, ordered by
 *            descending logit; weights w_i = exp(l_i - l_max) / sum_sel exp(.)
 *            ("GPU router/top-k", amalgafy.com/technical-overview)
 *   bucket   (token, slot) pairs grouped by expert, stable in (token, slot)
 *            order ("compact expert grouping", expxa.com
 *            reuse-ordering-qualification, "What changed from the first
 *            experiment")
 *   experts  y = Wd (silu(Wg x) * (Wu x)), every weight dequantised exactly:
 *            Q8_0 w = q * d (native Q8_0 weights, amalgafy.com/technical-
 *            overview, "Validated GPU foundation") or Q4_0 w = (n - 8) * d
 *            (layout below); down projection K=768 -> 2048 rows (expxa.com,
 *            "What changed from the first experiment")
 *   combine  out[t] = (residual ? x[t] : 0) + sum_slot w[t][slot] * y
 *            ("weighted combine", amalgafy.com/technical-overview,
 *            "Execution architecture")
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers owned by the caller unless stated
 *    otherwise.  The library allocates no device memory: scratch comes from a
 *    caller workspace sized by moe_workspace_size().
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call only enqueues work on it: it never synchronises the
 *    device or the stream and never reads results back to the host.
 *  - The return value is a MOE_* code.  Host-side argument checks run before
 *    anything is enqueued; MOE_ERR_CUDA reports a launch error.
 *  - Problems the device finds (an expert id out of range, a duplicate id in
 *    one token's selection) are OR-ed into an optional caller-owned int32
 *    status word (MOE_STATUS_*); the caller reads it whenever it likes.
 *  - The library holds no per-call state; calls on different streams with
 *    different buffers may run concurrently.
 *  - Alignment: every float / int32 array 16-byte aligned; qs and d arrays
 *    16-byte aligned; d_model and d_ff multiples of 32.
 *
 * Device weight layout, Q8_0 (moe_layer_w.wfmt = MOE_WFMT_Q8_0, produced by
 * moe_pack_q8 from the 34-byte blocks):
 *   qs  bytes    [E][rows][K]       the 32 int8 values q of each block, along
 *                                   K, each stored as the byte q + 128 (its
 *                                   sign bit flipped: offset binary), the
 *                                   form the exact dequantisation takes; the
 *                                   weight is (u - 128) * d
 *   d   fp16 bits[E][rows][K/32]    one scale per 32-wide block
 * Q4_0 (MOE_WFMT_Q4_0, produced by moe_pack_q4 from 18-byte blocks):
 *   qs  bytes    [E][rows][K/2]     each block's 16 bytes, unchanged: byte j
 *                                   of block b holds element 32b+j in its low
 *                                   nibble and 32b+16+j in its high nibble,
 *                                   unsigned; the weight is (n - 8) * d
 *   d   fp16 bits[E][rows][K/32]    one scale per 32-wide block
 *   gate, up: rows = d_ff, K = d_model;  down: rows = d_model, K = d_ff.
 * The pages name a 4-bit expert format as the next execution stage ("Q4
 * expert execution", amalgafy.com/technical-overview, "Execution
 * architecture") without giving its layout; Q4_0 here is the plain 4-bit
 * sibling of Q8_0 (same 32-wide blocks and fp16 scale, values offset by 8).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ---------------------------------------------------- */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1  /* null/misaligned pointer, bad size, k > E, ... */
#define MOE_ERR_UNSUPPORTED 2  /* device is not sm_100/sm_103, or a mode not built */
#define MOE_ERR_CUDA 3         /* a launch failed (cudaGetLastError) */
#define MOE_ERR_WORKSPACE 4    /* workspace null or smaller than moe_workspace_size() */

/* ---- device status bits (OR-ed into *status) ------------------------- */
#define MOE_STATUS_BAD_INDEX 1 /* an expert id outside [0, E), or repeated in one token */
#define MOE_STATUS_TIMEOUT 2   /* a bounded on-device wait (grid barrier, mbarrier) gave up after
                                  2 s; that call's outputs are invalid */
#define MOE_STATUS_ARENA_FULL 4 /* an arena admission had more missed experts than evictable slots;
                                   the experts left without a slot are skipped (wrong outputs) */

/* ---- expert-input precision ------------------------------------------ */
#define MOE_ACT_F32 0  /* fp32 activations, CUDA-core contraction (decode) */
#define MOE_ACT_BF16 1 /* bf16 activations and weights on tcgen05 tensor cores (prefill), Q8_0 or
                          Q4_0; batches of fewer than 128 pairs, or d_model / d_ff not multiples
                          of 256, run the fp32 path (more accurate, and memory-bound at that
                          size anyway) */

/* ---- expert weight formats (moe_layer_w.wfmt) ------------------------- */
#define MOE_WFMT_Q8_0 0 /* every path */
#define MOE_WFMT_Q4_0 1 /* fp32 lane-per-row kernels, any T; needs d_model and d_ff multiples of
                           256 (else MOE_ERR_UNSUPPORTED); one or two tokens with d_model a multiple
                           of 1024 (at most 2048): the single-launch decode kernel; MOE_ACT_BF16 at
                           128+ pairs: the tensor-core kernels */

/* ---- flags ----------------------------------------------------------- */
#define MOE_FLAG_DETERMINISTIC 1 /* combine by a fixed-order sum instead of atomics */
#define MOE_FLAG_REUSE_ORDER 2   /* opt-in: the tensor-core down projection walks each expert's
                                    work in bands of four output-row tiles across all its token
                                    chunks (the reuse-ordering traversal of
                                    expxa.com/research/reuse-ordering-qualification); the same
                                    tiles with the same arithmetic in another order (bit-identical
                                    with MOE_FLAG_DETERMINISTIC).  Off by default */

/* Limits: E <= 256, k <= 32, k <= E, d_model and d_ff multiples of 32,
 * d_model <= 8192, d_ff <= 8192, T <= 65536. */
#define MOE_MAX_EXPERTS 256
#define MOE_MAX_TOPK 32

/* One quantised matrix family (all E experts), device layout above; qs
 * holds int8 values (Q8_0) or packed nibbles (Q4_0). */
typedef struct {
    const int8_t* qs;
    const uint16_t* d;
} moe_q8_mat;

/* One layer's weights.  router_w: fp32 [E][d_model]; router_bias: fp32 [E]
 * or NULL; wfmt: MOE_WFMT_* of gate, up and down.
 * expert_slot (device int32 [E]) or NULL: with NULL, gate/up/down hold the E
 * experts in expert order; otherwise they are an expert arena of n_slots
 * slots ([n_slots][rows][...]) and expert e's matrices sit in slot
 * expert_slot[e] (moe_arena_admit writes such a map).  A slot outside
 * [0, n_slots) means "not resident": that expert's pairs are skipped. */
typedef struct {
    int E, k, d_model, d_ff;
    moe_q8_mat gate, up, down;
    const float* router_w;
    const float* router_bias;
    int wfmt;
    int n_slots;
    const int32_t* expert_slot;
} moe_layer_w;

/*
 * Bytes of workspace the calls below need for T tokens (0 if the arguments
 * are invalid).  act: MOE_ACT_*; flags: MOE_FLAG_*.  The workspace must be
 * 256-byte aligned.  It holds the routing results, the bucketing, the SwiGLU
 * activations h and, for MOE_FLAG_DETERMINISTIC, the per-pair outputs.
 */
MOE_API size_t moe_workspace_size(int T, const moe_layer_w* w, int act, int flags);

/*
 * Repack Q8_0 weights from the pages' 34-byte blocks (fp16 scale d, little
 * endian, then 32 int8 values q along K) into the device layout.
 *   blocks: device bytes, rows * (K/32) blocks, row-major (any alignment)
 *   qs: bytes q + 128 [rows][K] (16-byte aligned); d: fp16 bits [rows][K/32]
 * rows may span several experts ([E*rows_per_expert]).  Exact: the scale
 * bits are copied and each value's sign bit is flipped.
 */
MOE_API int moe_pack_q8(const uint8_t* blocks, long long rows, int K, int8_t* qs, uint16_t* d, void* stream);

/*
 * Repack Q4_0 weights from 18-byte blocks (fp16 scale d, little endian, then
 * 16 bytes of 4-bit values, layout above) into the device layout.
 *   blocks: device bytes, rows * (K/32) blocks, row-major (any alignment)
 *   qs: bytes [rows][K/2] (16-byte aligned); d: fp16 bits [rows][K/32]
 * Bit-exact copy.
 */
MOE_API int moe_pack_q4(const uint8_t* blocks, long long rows, int K, uint8_t* qs, uint16_t* d, void* stream);

/*
 * Router: logits x . Wr^T (+ bias) in fp32, top-k (ties to the lower id,
 * descending logit), renormalised softmax weights.
 *   x: fp32 [T][d_model]; idx: int32 [T][k]; wts: fp32 [T][k].
 * Deterministic: the same inputs give bit-identical idx and wts.
 */
MOE_API int moe_route(const float* x, int T, const moe_layer_w* w, int32_t* idx, float* wts, void* stream);

/*
 * Compact expert grouping: a stable counting sort of the T*k pairs by expert.
 *   idx: int32 [T][k] expert ids.
 *   offsets: int32 [E+1], offsets[e] = number of pairs with expert < e
 *   pair_tok, pair_slot: int32 [T*k], the pairs in bucket order, ascending
 *       (token, slot) within one expert
 *   pos: int32 [T*k], pos[t*k+s] = bucket position of pair (t, s)
 *   status: optional; MOE_STATUS_BAD_INDEX if an id is out of range or
 *       repeated within a token (such pairs are dropped; outputs then only
 *       stay in bounds)
 * Deterministic (no atomics decide any position).
 */
MOE_API int moe_bucket(const int32_t* idx, int T, int k, int E, int32_t* offsets, int32_t* pair_tok, int32_t* pair_slot,
               int32_t* pos, int32_t* status, void* stream);

/*
 * Expert SwiGLU FFNs over the bucketed pairs, dequantisation (Q8_0 or Q4_0,
 * w->wfmt) fused into the contractions.
 *   x: fp32 [T][d_model] expert inputs (token-indexed)
 *   offsets, pair_tok, pair_slot, pos, wts: from moe_bucket / moe_route.
 *       Every bucket is clamped into [0, T*k] and token / slot ids are
 *       range-checked, so offsets that are not a valid bucketing give wrong
 *       values but no access outside the arrays.
 *   act: MOE_ACT_F32 (fp32 FMA) or MOE_ACT_BF16 (tcgen05, bf16 operands,
 *        fp32 accumulation)
 *   fuse_combine = 1: out_or_ypairs is out fp32 [T][d_model]; it is
 *        overwritten with (residual ? x : 0) + sum_slot w * y (fp32 atomic
 *        adds, so the last bits may vary run to run)
 *   fuse_combine = 0: out_or_ypairs is ypairs fp32 [T*k][d_model], row p
 *        holding y of the pair in bucket position p (bit-reproducible);
 *        `residual` is ignored.  Combine with moe_combine().
 *   ws / ws_bytes: workspace of at least moe_workspace_size(T, w, act, 0).
 * out must not alias x.
 */
MOE_API int moe_expert_ffn_q8(const float* x, int T, const moe_layer_w* w, const int32_t* offsets, const int32_t* pair_tok,
                      const int32_t* pair_slot, const float* wts, int act, int fuse_combine, float* out_or_ypairs,
                      int residual, void* ws, size_t ws_bytes, int32_t* status, void* stream);

/*
 * Weighted combine in a fixed order (bit-reproducible):
 *   out[t][o] = (residual ? residual[t][o] : 0) + sum_{s=0..k-1} wts[t][s] * ypairs[pos[t*k+s]][o]
 *   ypairs fp32 [T*k][d_model]; residual fp32 [T][d_model] or NULL.
 */
MOE_API int moe_combine(const float* ypairs, const float* wts, const int32_t* pos, int T, int k, int d_model,
                const float* residual, float* out, void* stream);

/*
 * The whole layer: route -> bucket -> gate/up -> down + combine.
 *   x: fp32 [T][d_model]; out: fp32 [T][d_model], must not alias x.
 *       x is only read, with plain loads, so it may also be a page-locked
 *       host buffer the GPU addresses directly (on GB300 the host memory is
 *       coherent with the GPU over NVLink-C2C); that pays off only for a
 *       token or two, where it saves a separate copy.
 * Paths: one or two tokens on the fp32 path without MOE_FLAG_DETERMINISTIC
 * run as ONE cooperative kernel (router, top-k, bucketing, gate/up, down and
 * combine) with one grid-wide exchange of launch-tagged words kept in the
 * workspace: nothing is cleared between calls and any prior workspace
 * content is safe (shapes that kernel does not take -- d_model not a
 * multiple of 512, or of 1024 for Q4_0 -- use an older single-launch kernel
 * whose 8-byte barrier words are cleared by a memset before it, where it
 * fits, and the separate kernels otherwise).  The kernel is
 * launched as a programmatic dependent of the previous kernel in the stream:
 * its blocks may become resident while that kernel's last blocks run, but
 * everything it reads that a previous kernel may have written (x, the
 * weights, the workspace) is read after that kernel has completed.
 * Otherwise router, bucketing and the expert kernels (tcgen05 for
 * MOE_ACT_BF16 with >= 128 pairs), each a programmatic dependent of the one
 * before: the first reads x only after the caller's previous kernel has
 * completed, and a later one reads early only what an earlier kernel of the
 * same call was done with before it let that one launch (the tcgen05
 * kernels stream weights while the previous kernel of the call finishes).
 * Grid exchanges and mbarrier waits are bounded (MOE_STATUS_TIMEOUT).
 *   act: MOE_ACT_F32 or MOE_ACT_BF16; flags: MOE_FLAG_*
 *   residual: 1 adds x to the output (a residual stream between layers)
 *   idx_out [T][k], wts_out [T][k], offsets_out [E+1]: optional copies of the
 *       routing and bucketing (NULL to skip)
 *   ws / ws_bytes: at least moe_workspace_size(T, w, act, flags)
 * Enqueues a fixed sequence of kernels (no host synchronisation), so the call
 * can be captured into a CUDA graph and replayed.
 */
MOE_API int moe_layer_forward(const float* x, int T, const moe_layer_w* w, int act, int flags, int residual, float* out,
                      int32_t* idx_out, float* wts_out, int32_t* offsets_out, void* ws, size_t ws_bytes,
                      int32_t* status, void* stream);

/*
 * moe_layer_forward without a caller workspace, for callers that cannot
 * allocate device memory where they run the layer (a latency-critical loop
 * that must not enter an allocator, a plugin inside a runtime that owns all
 * device memory).  The pages have no counterpart; this is a convenience of
 * this library.
 *
 * Same arguments and results as moe_layer_forward with idx_out, wts_out and
 * offsets_out NULL; the scratch comes from one fixed region of
 * MOE_STATIC_SCRATCH_BYTES compiled into the library (held on every GPU that
 * loads it, until the process exits).
 *  - Returns MOE_ERR_WORKSPACE when moe_workspace_size(T, w, act, flags)
 *    exceeds MOE_STATIC_SCRATCH_BYTES (for the qwen3_moe geometry, T <= 64
 *    fits with or without MOE_FLAG_DETERMINISTIC).
 *  - Allocates nothing.  The first call on each device looks up the region's
 *    device address (cudaGetSymbolAddress) with that device current; make it
 *    before any stream capture.
 *  - Every call shares the region: calls whose GPU work may overlap (other
 *    streams, other host threads, same device) race and must be serialised
 *    by the caller.
 */
#define MOE_STATIC_SCRATCH_BYTES (8u << 20)
MOE_API int moe_layer_forward_static(const float* x, int T, const moe_layer_w* w, int act, int flags, int residual,
                                     float* out, int32_t* status, void* stream);

/*
 * ---- Expert arena: device-resident slots with a host-memory miss path ----
 *
 * "Managed VRAM expert arena" and the miss path that "changes residency
 * beneath the compute plane" (amalgafy.com/technical-overview, "VRAM budget
 * policy", "Execution architecture"), reduced to one GPU: every expert of
 * every layer lives in host memory as one page-aligned blob; the arena holds
 * n_slots of them in HBM.  Each layer call admits the experts its bucketing
 * routes to: hits keep their slot, misses take the least recently used
 * evictable slots and their blobs are copied in by the GPU itself, reading
 * the page-locked host memory directly (on GB300 host memory is coherent
 * with the GPU over NVLink-C2C), so no host synchronisation or readback is
 * involved and the admission can be captured in a CUDA graph.
 *
 * Replacement (one admission, for layer l with active experts A ascending):
 *   clock += 1; every resident e in A: its slot's stamp = clock (a hit);
 *   the missed experts, ascending, take the evictable slots (stamp != clock)
 *   in ascending (stamp, slot) order -- empty slots have stamp 0 -- evicting
 *   their previous owners; each taken slot's stamp = clock.
 *
 * Blob (host memory, moe_arena_blob_bytes() each, blob index l*E + e): a
 * 4 KiB header page (uint32 words: magic 0x424f454d, version 1, wfmt,
 * layer, expert, d_model, d_ff, payload bytes) and the payload: gate qs,
 * up qs, down qs, gate d, up d, down d of that expert, in the device layout
 * above, back to back, the whole blob a multiple of 4 KiB.  For Q8_0 at
 * d_model 2048, d_ff 768 the payload is 5,013,504 B and the blob 5,017,600 B.
 *
 * State (device memory, moe_arena_state_bytes()): starts with
 * moe_arena_stats, then the residency tables; the caller may read the
 * stats whenever it likes (e.g. with a device-to-host copy).
 */
typedef struct {
    unsigned long long hits;      /* admitted experts that were resident */
    unsigned long long misses;    /* admitted experts copied in */
    unsigned long long bytes_in;  /* payload bytes copied from host memory */
    unsigned int clock;           /* admissions so far */
    int layers, experts, slots;
    int last_misses;              /* misses of the latest admission */
    int full_events;              /* admissions that ran out of evictable slots */
    int reserved[2];
} moe_arena_stats;

/* Bytes of one expert blob for the geometry and format of w (0 if invalid). */
MOE_API size_t moe_arena_blob_bytes(const moe_layer_w* w);

/* Device bytes of the arena state for `layers` x `experts` and `slots` (0 if invalid;
 * experts <= 256, slots <= 65536). */
MOE_API size_t moe_arena_state_bytes(int layers, int experts, int slots);

/* Reset the state: every slot empty, clock and stats zero. */
MOE_API int moe_arena_init(void* state, int layers, int experts, int slots, void* stream);

/*
 * Write the blob of expert e of layer `layer` from a layer's resident weights
 * w (device layout, expert order; w->expert_slot must be NULL) into `blob`
 * (device memory, or page-locked host memory the GPU can address).
 */
MOE_API int moe_arena_pack_blob(const moe_layer_w* w, int layer, int e, void* blob, void* stream);

/*
 * One admission (replacement rule above) for layer `layer`, whose bucketing
 * is `offsets` (int32 [E+1], buckets clamped into [0, P]).
 *   host_blobs: the blobs of all layers x experts, blob index l*E + e
 *       (page-locked host memory, or device memory), read by the GPU
 *   arena: geometry, format and the slot arrays (gate/up/down with
 *       arena->n_slots slots); its expert_slot is ignored
 *   slot_map: int32 [E] out, the map for the FFN (arena->expert_slot):
 *       every admitted expert's slot, -1 for experts left without one
 *   status: optional; MOE_STATUS_ARENA_FULL when misses exceed the evictable slots
 * Two kernels: the admission (one CTA) and the copy of the missed blobs.
 */
MOE_API int moe_arena_admit(void* state, int layer, const int32_t* offsets, int P, const void* host_blobs,
                            const moe_layer_w* arena, int32_t* slot_map, int32_t* status, void* stream);

/*
 * The layer forward through the arena: route -> bucket -> admit -> expert
 * FFNs reading the arena slots -> combine.  Same arguments as
 * moe_layer_forward, plus the arena state, the layer index and the host
 * blobs; w is the arena (router of this layer, gate/up/down with n_slots
 * slots).  Never takes the single-launch decode kernel.
 */
MOE_API int moe_layer_forward_arena(const float* x, int T, const moe_layer_w* w, int act, int flags, int residual,
                                    float* out, void* state, int layer, const void* host_blobs, void* ws,
                                    size_t ws_bytes, int32_t* status, void* stream);

/* Library version string (static storage). */
MOE_API const char* moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
