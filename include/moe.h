/*
 * libmoe — routed mixture-of-experts FFN of a decode step, on one GB300 (sm_103a).
 *
 * Per layer and token the library computes what the TurboFieldfare write-up
 * ("Optimizing a 14.3 GB model for an 8 GB machine") and the video
 * walkthrough of the same project (the yousumm.com transcript) describe for
 * Gemma 4 26B-A4B:
 *
 *   - a router over E experts (128 in that model) of which only the k best
 *     (8 there) are evaluated, as the video's account of one token step
 *     explains, with softmax gates over the k picked logits;
 *   - for each picked expert and for the shared expert, which the video
 *     describes as evaluated for every token whatever the router picks: an int4-affine gate and up
 *     projection (groups of 64 inputs with a 16-bit scale and bias each,
 *     section "Vectorization helped when it respected the storage layout"),
 *     the GELU-gated product GELU(gate) * up, and the down projection;
 *   - the combine y = y_shared + sum_j gate_j * y_{e_j};
 *   - optionally, a per-layer bounded expert-slot cache with LRU eviction
 *     that stages missing experts into fixed device slots (section "MoE
 *     needed parallel work, reuse, and coarse overlap"; goinfer, "When the
 *     model doesn't fit"), the copies overlapped with the shared expert.
 *     The cache can evict by LFU instead, and the staging can be done by a
 *     device kernel instead of host-issued copies.  The experts can also
 *     live in a file read by bounded parallel pread (section "Explicit reads
 *     made expert streaming work"), optionally behind a pinned host tier.
 *     Prefill on such a context goes a chunk at a time, each layer staging
 *     the union of the chunk's experts once.
 *
 * Conventions for every entry point:
 *   - Every call returns a moe_status and never aborts, throws or exits.
 *   - Argument errors (MOE_EINVAL) are detected before anything is enqueued
 *     or allocated.
 *   - A failed CUDA call or an expired bounded wait poisons the context:
 *     every later call on it returns MOE_ESTATE until moe_destroy.
 *   - One context is used by one host thread at a time.
 *   - "device" pointers are CUDA device (or managed) memory on the context's
 *     device; "host" pointers are ordinary or pinned host memory.
 *   - Nothing in the library ever falls back to a CPU implementation.
 */
#ifndef LIBMOE_MOE_H
#define LIBMOE_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_ctx moe_ctx; /* opaque, owned by the library */

typedef enum {
    MOE_OK = 0,
    MOE_EINVAL = 1,   /* invalid argument; nothing enqueued, nothing changed */
    MOE_ENOMEM = 2,   /* computed budget exceeds free device memory, or an allocation failed;
                         the context is unchanged */
    MOE_ECUDA = 3,    /* a CUDA call failed; the context is now poisoned */
    MOE_ESTATE = 4,   /* poisoned context, or a call in the wrong state (layer not initialised,
                         slots not set) */
    MOE_ETIMEOUT = 5, /* a bounded wait expired; the context is now poisoned */
    MOE_EDOMAIN = 6,  /* the device saw a value outside a documented domain: a router input
                         outside the exact fixed-point domain (|W_r[e,i] * x[i]| >= 2^11 or
                         non-finite), an fp16 matrix operand outside [-65504, 65504] (prefill
                         and the clustered one-token kernel), or a clustered-kernel partial
                         layer output with |y| >= 2^17; reported by moe_sync */
    MOE_EIO = 7       /* a read or write of the expert file failed or came up short; the
                         context (if any) is now poisoned */
} moe_status;

enum { MOE_RESIDENT_HBM = 0, MOE_HOST_POOL = 1, MOE_FILE_POOL = 2 };
enum { MOE_FILE_DIRECT = 1 };   /* moe_set_expert_file flag: read misses with O_DIRECT */
enum { MOE_STAGING_HOST = 0, MOE_STAGING_DEVICE = 1, MOE_STAGING_FUSED = 2 };   /* moe_set_staging modes */
enum { MOE_CACHE_LRU = 0, MOE_CACHE_LFU = 1 };
enum { MOE_GELU_ERF = 0, MOE_GELU_TANH = 1 };

/* Model dimensions.  Constraints (checked by moe_create): d, f and f_shared
 * are multiples of 64; group == 64; 1 <= top_k <= n_experts <= 256;
 * d <= 3072 (keeps the int64 router sum exact); n_layers >= 1;
 * 1 <= max_tokens <= 65536. */
typedef struct {
    int32_t d;            /* hidden size */
    int32_t f;            /* routed-expert intermediate size */
    int32_t f_shared;     /* shared-expert intermediate size */
    int32_t n_experts;    /* E */
    int32_t top_k;        /* k */
    int32_t group;        /* int4 affine group length along the input dimension (64) */
    int32_t n_layers;     /* layers held by the context */
    int32_t gelu_variant; /* MOE_GELU_ERF (exact erf form) or MOE_GELU_TANH */
    int32_t prenorm;      /* 1: a layer's FFN input is x = bf16(h / sqrt(mean(h^2) + norm_eps));
                             0: the FFN input is h itself */
    int32_t max_tokens;   /* largest B of moe_decode_step and T of moe_prefill */
    float norm_eps;       /* epsilon of the RMS normalisation (used when prenorm = 1) */
} moe_config;

/* One expert's weights in canonical layout.  Every projection is row-major
 * [out][in]; int4 values are unsigned 0..15 packed two per byte (byte m of a
 * row holds element 2m in its low nibble, 2m+1 in its high nibble); each run
 * of 64 consecutive inputs of a row has an fp16 (scale, bias) pair, stored
 * sb[row][in/64][2]; the weight is scale * q + bias.
 *   gate_q [f][d/2]  gate_sb [f][d/64][2]
 *   up_q   [f][d/2]  up_sb   [f][d/64][2]
 *   down_q [d][f/2]  down_sb [d][f/64][2]
 * (f is f_shared for the shared expert.) */
typedef struct {
    const uint8_t *gate_q;
    const uint16_t *gate_sb;
    const uint8_t *up_q;
    const uint16_t *up_sb;
    const uint8_t *down_q;
    const uint16_t *down_sb;
} moe_expert_weights;

/* One record per (token step, layer, top-k position) of the slot cache. */
typedef struct {
    int32_t token;   /* step counter value of the decode call (see moe_decode_step) */
    int32_t layer;
    int32_t k_pos;   /* top-k position j, 0 = highest logit */
    int32_t expert;  /* picked expert */
    int32_t hit;     /* 1 if the expert was already in a slot */
    int32_t slot;    /* slot index that holds it after the step */
    int32_t evicted; /* expert that a miss replaced, or -1 (slot was empty, or hit) */
} moe_trace_rec;

typedef struct {
    int64_t steps;         /* decode calls on a host-pool context since create/reset */
    int64_t hits;          /* summed over layers */
    int64_t misses;
    int64_t staged_bytes;  /* routed-expert bytes copied to the device: decode misses into
                              slots, and chunked-prefill unions into the prefill arena */
    int64_t n_slots;
    int64_t expert_bytes;  /* bytes of one routed expert (device layout == canonical size) */
    int64_t shared_bytes;
    int64_t device_bytes;  /* device memory held by the context */
    int64_t host_pool_bytes;
    int64_t file_read_bytes;  /* expert-file contexts: routed-expert bytes read from the file */
    int64_t host_tier_hits;   /* expert-file contexts: slot-cache misses served by the host tier */
    int64_t host_tier_bytes;  /* pinned bytes of the host tier (moe_set_file_cache) */
} moe_stats;

/* Create a context on CUDA device `device`.  Allocates the per-call scratch
 * sized for cfg->max_tokens.  MOE_EINVAL on a bad config, MOE_ENOMEM if the
 * scratch does not fit.  The config carries the model geometry the video
 * walkthrough gives for Gemma 4 26B-A4B (30 layers, 128 experts per layer, 8
 * picked, one shared expert) and the quantisation of the write-up's section
 * "Vectorization helped when it respected the storage layout" (int4 weights,
 * one 16-bit scale and bias per group of 64); every field can be set
 * independently within the limits checked here. */
moe_status moe_create(const moe_config *cfg, int device, moe_ctx **out);

/* Copy one layer's weights into the context (synchronous; the caller may free
 * its buffers on return).  Pointers may be host or device memory.
 *   router_w: fp16 [n_experts][d], row-major
 *   experts:  array of n_experts moe_expert_weights (canonical layout above)
 *   shared:   the shared expert (intermediate size f_shared)
 *   residency: MOE_RESIDENT_HBM keeps every expert in device memory;
 *              MOE_HOST_POOL keeps routed experts in a pinned host pool and
 *              serves them from per-layer device slots (see moe_set_slots);
 *              MOE_FILE_POOL writes them to the expert file instead (see
 *              moe_set_expert_file, which must come first) and serves them
 *              the same way.  All layers of a context use the same residency.
 * The library repacks the weights into its own device layout: a permutation
 * of the same bytes (nibbles and (scale, bias) pairs), never a re-encoding.
 * This follows the write-up's section "Explicit reads made expert streaming
 * work" and the video walkthrough's account of the file format: the weights
 * are stored in exactly the order the kernels read them, so that staging an
 * expert (slot copy, file read) is one contiguous copy with no conversion. */
moe_status moe_init_layer(moe_ctx *ctx, int layer, const uint16_t *router_w,
                          const moe_expert_weights *experts, const moe_expert_weights *shared,
                          int residency);

/* Host-pool and expert-file contexts: give every layer n_slots device slots (top_k <= n_slots
 * <= n_experts) and empty the LRU tables.  The byte budget
 * n_layers * n_slots * expert_bytes is checked against free device memory
 * before anything is allocated (MOE_ENOMEM, context unchanged).
 * goinfer, "When the model doesn't fit": the slot count is the lever of a
 * paged MoE (its table sweeps 8 to 128 slots per layer), and the budget guard
 * must be keyed on bytes the program computes itself, because a guard on the
 * operating system's resident-set figure inverted at the failure point; the
 * write-up's section "MoE needed parallel work, reuse, and coarse overlap"
 * gives the per-layer bounded cache (16 of 128 experts there). */
moe_status moe_set_slots(moe_ctx *ctx, int n_slots);

/* Run layers [layer_begin, layer_end) for B tokens, each layer
 *   x = prenorm ? bf16(RMSNorm(h)) : h;  y = MoE-FFN(x);  h <- bf16(h + y).
 * The per-layer step is the one the video walkthrough narrates for a token
 * passing the 30 layers in order (the router names 8 of 128 experts, which
 * run together with the shared expert) and the write-up's section "MoE needed
 * parallel work, reuse, and coarse overlap" restructures (routed experts from
 * the cache first, misses after; the shared expert overlapped with the
 * reads).  The RMS pre-norm between layers stands in for the attention block
 * the pages place there, which is outside this library.
 *   h_in:  device bf16 [B][d] residual entering layer_begin (not modified)
 *   h_out: device bf16 [B][d] residual after layer_end - 1 (may equal h_in)
 *   logit_bias: device fp32 [layer_end - layer_begin][B][n_experts] added to the
 *          router logits, or NULL
 *   y_last: device fp32 [B][d], the FFN output y of the last layer, or NULL
 *   trace / trace_cap / trace_len: host-pool contexts only, host array that
 *          receives (layer_end - layer_begin) * top_k records, or NULL
 *   stream: cudaStream_t to run on (NULL = legacy default stream)
 * Resident contexts accept 1 <= B <= min(max_tokens, 32) and return without
 * synchronising.  B == 1 runs every layer in one cooperative launch: the
 * clustered kernel (clusters of four CTAs, one per SM, when the device and
 * the shape allow it: at most 6 (shared or top-k position, int4 group) units
 * per cluster and layer, n_experts <= CTAs), else the per-SM persistent
 * kernel.  The clustered kernel multiplies fp16 activations (x and the GELU
 * product, the latter as an fp16 hi + lo pair), sums the layer output as
 * integers on a 2^-32 grid (deterministic), and reports a launch without its
 * cluster shape as MOE_ECUDA from moe_sync.  From 16 tokens on (when the
 * shape allows it) a step runs through the same grouped tcgen05 path as
 * moe_prefill, with the same exact routing.  Host-pool and expert-file
 * contexts need B == 1 and slots set; every call is one cache step (the step
 * counter increments per call).  With host staging (the default) the call
 * returns after the last layer's staging decision, with the compute still
 * enqueued; an expert-file context reads its misses on the calling thread
 * meanwhile.  With MOE_STAGING_DEVICE (moe_set_staging) it returns once every
 * layer is enqueued, or after the step when a trace is asked for.  Waits
 * inside the call are bounded (MOE_ETIMEOUT). */
moe_status moe_decode_step(moe_ctx *ctx, const void *h_in, int B, int layer_begin, int layer_end,
                           const float *logit_bias, void *h_out, float *y_last, moe_trace_rec *trace,
                           int trace_cap, int *trace_len, void *stream);

/* Prefill: T tokens at once through layers [layer_begin, layer_end)
 * ("Optimizing a 14.3 GB model for an 8 GB machine", section "Splitting the
 * work improved attention and prefill": dequantise a small 16-bit tile, run
 * the matrix primitive, discard the tile).  1 <= T <= max_tokens; h, h_out
 * bf16 [T][d] and y_last fp32 [T][d] (nullable)
 * on the device; logit_bias (nullable) fp32 [layer_end - layer_begin][T][E].
 * When d % 128 == 0 and n_experts <= 128 (else the batched decode kernels run,
 * 32 tokens at a time): the routing is exact (the same ids and gates as
 * moe_decode_step), the (token, k) pairs are grouped by expert, and each
 * expert's rows run through int4 -> fp16 tiles on tcgen05 tensor cores with
 * fp32 accumulation (weights rounded once to fp16, activations in fp16), then
 * are combined per token as shared + routed outputs in top-k order; an fp16
 * operand outside [-65504, 65504] is reported by moe_sync as MOE_EDOMAIN.  The
 * first call allocates scratch for max_tokens tokens (about 180 KB per token at
 * the full shape).  Returns without synchronising.
 * Host-pool and expert-file contexts (chunked prefill, same write-up and
 * section: the prompt goes through in bounded batches instead of one token at
 * a time, here with only the experts a batch picks in device memory): the
 * call is one chunk.  Per layer the T tokens
 * are routed, the union of the experts they pick is staged once (from the
 * pinned pool, or read from the expert file) into a one-layer arena of
 * n_experts device records (made on the first call), and the same grouped
 * GEMMs run over it, so the outputs are bit-identical to a resident context's;
 * the shared expert's gate/up runs while the union is staged.  The host waits
 * for each layer's routing (bounded: MOE_ETIMEOUT), so the call returns after
 * the last layer's staging.  The decode slot cache is neither read nor
 * changed; staged bytes count in moe_stats.  Needs the tensor-core path
 * (d % 128 == 0, n_experts <= 128), else MOE_EINVAL. */
moe_status moe_prefill(moe_ctx *ctx, const void *h, int T, int layer_begin, int layer_end,
                       const float *logit_bias, void *h_out, float *y_last, void *stream);

/* Capture per-layer values of the next decode/prefill calls into caller device
 * buffers (any may be NULL; max_layers bounds the layers written):
 *   x_layers  bf16 [max_layers][B][d]   FFN input of each layer
 *   ids       int32 [max_layers][B][k]  picked experts, top-k order
 *   gates     fp32 [max_layers][B][k]
 *   y_layers  fp32 [max_layers][B][d]   FFN output of each layer
 * Pass all NULL to stop capturing. */
/* Capture the router logits of the next calls (bias included, units of 2^-40,
 * layout int64 [max_layers][B][n_experts], max_layers from moe_set_debug;
 * NULL stops).  The decode kernels write every expert's exact logit.  The
 * prefill router evaluates exactly only the experts its error bound cannot
 * rule out; the others read INT64_MIN.  Takes effect only while moe_set_debug
 * has a non-zero max_layers. */
moe_status moe_set_debug_logits(moe_ctx *ctx, int64_t *logits);

moe_status moe_set_debug(moe_ctx *ctx, uint16_t *x_layers, int32_t *ids, float *gates,
                         float *y_layers, int max_layers);

/* Synchronise `stream`, then report device-side conditions raised since the
 * last moe_sync: MOE_EDOMAIN (a value outside a documented domain, see
 * moe_status), MOE_ETIMEOUT (a device wait ran out; poisons), MOE_ECUDA (the
 * clustered kernel ran without its cluster shape and did nothing; poisons).
 * Clears the reported conditions. */
moe_status moe_sync(moe_ctx *ctx, void *stream);

moe_status moe_get_stats(moe_ctx *ctx, moe_stats *out);

/* Host-pool contexts: copy layer `layer`'s slot table to host arrays of
 * n_slots entries (expert_of_slot: -1 = empty; last_use: step counter, -1 = empty). */
moe_status moe_get_cache_state(moe_ctx *ctx, int layer, int32_t *expert_of_slot, int64_t *last_use);

/* Empty every slot table and the LFU use counts, zero the counters and the step counter. */
moe_status moe_reset_cache(moe_ctx *ctx);

/* Host-pool contexts: the slot cache's eviction policy, then an empty cache
 * (as moe_reset_cache).  MOE_CACHE_LRU (the default; goinfer, "When the model
 * doesn't fit": plain LRU over the slots): a miss takes the slot least
 * recently used.  MOE_CACHE_LFU (the TurboFieldfare video walkthrough: the
 * expert used least often leaves): every pick adds one to its expert's
 * whole-run count, and a miss takes the slot with the smallest (count of its
 * expert, last use, slot index); an empty slot counts -1.  In both, hits are
 * taken first and misses in top-k order among the slots this step has not
 * touched.  MOE_EINVAL for an unknown policy, MOE_ESTATE for a resident
 * context. */
moe_status moe_set_cache_policy(moe_ctx *ctx, int policy);

/* Expert file tier ("Optimizing a 14.3 GB model for an 8 GB machine", section
 * "Explicit reads made expert streaming work": routed experts are read from
 * the model file on a miss with a bounded number of parallel pread calls into
 * per-layer slots, instead of being mapped and paged in).  Call before the
 * first moe_init_layer of a context whose layers use residency
 * MOE_FILE_POOL: `path` is created (or truncated); moe_init_layer then writes
 * each routed expert of the layer, in the device layout, to the record at
 * byte offset (layer * n_experts + expert) * record_stride (record_stride =
 * the expert's device bytes rounded up to 4096) instead of keeping it in a
 * pinned host pool.  Such a context behaves like a MOE_HOST_POOL context
 * (moe_set_slots, moe_set_cache_policy, traces, one token per decode call)
 * except that a miss is read from the file by `n_threads` (1..64) host
 * threads in chunks of `chunk_bytes` (0 = 512 KiB; multiple of 4096) into
 * pinned staging memory (2 * top_k records, owned by the library), from which
 * the staging copy to the slot is issued.  The host pool's bytes are 0.
 * flags: MOE_FILE_DIRECT reads whole records through a second descriptor
 * opened with O_DIRECT (past the page cache; MOE_EINVAL where the file system
 * refuses it), else 0.
 * Errors: MOE_EINVAL (NULL path, bad counts, layers already initialised, or
 * the file cannot be created), MOE_ENOMEM (staging memory, or the reader
 * threads cannot be started), MOE_EIO later
 * (a record read or write that fails or comes up short). */
moe_status moe_set_expert_file(moe_ctx *ctx, const char *path, int n_threads, uint64_t chunk_bytes, int flags);

/* Host-pool contexts: who stages the slot cache's misses.  MOE_STAGING_HOST
 * (the default; the TurboFieldfare write-up's "coarse overlap": the host
 * waits for each layer's routing, then issues the copies on a side stream
 * while the shared expert and the hits are computed).  MOE_STAGING_DEVICE:
 * no host round trip per layer; a staging kernel on the side stream, ordered
 * after the layer's router kernel, reads the miss record and copies the
 * missed experts from the pinned pool (mapped into the device address space,
 * read through the host link) into their slots, so moe_decode_step enqueues
 * all layers and returns at once (after the step completes when a trace is
 * asked for, to fill it).  MOE_STAGING_FUSED: the whole step is one launch
 * of the clustered decode kernel (the write-up's section "MoE needed parallel
 * work, reuse, and coarse overlap": persistent workers, the cache first, the
 * shared expert overlapped with the reads): every layer's router and top-k,
 * the slot-cache step (run once, in cluster 0, which publishes each rank's
 * slot and hit to every CTA), hits loaded from their slots, and misses read
 * by the consumer warps from the mapped pool straight into their stage
 * buffers and written into the slots on the way.  Needs the clustered kernel
 * (B = 1, d <= 2816, its shape limits) and returns once the step is enqueued
 * (after it completes when a trace is asked for).  All three modes give the
 * same cache decisions and traces; HOST and DEVICE run the per-layer kernels,
 * FUSED the clustered kernel, whose outputs equal a resident context's
 * clustered kernel bit for bit.  Empties the cache as moe_reset_cache.
 * Errors: MOE_EINVAL (unknown mode), MOE_ESTATE (not a host-pool context, a
 * pool the device cannot address, or FUSED without the clustered kernel). */
moe_status moe_set_staging(moe_ctx *ctx, int mode);

/* Two-tier cache (expert file -> pinned host records -> HBM slots): keeps
 * `n_host` records per layer of an expert-file context in pinned host memory
 * in front of the file, so the slot cache's misses come from the file only
 * when the host tier misses too.  The pages keep a bounded set of experts in
 * memory in front of the SSD (the TurboFieldfare video walkthrough: 16 per
 * layer; the goinfer chapter "When the model doesn't fit": weights on disk or
 * in host memory, streamed as needed); with device memory apart from host
 * memory, that level sits between the file and the device slots, here
 * explicit, pinned and bounded.  The host tier follows the slot cache's LRU
 * rules one level down:
 * per layer and step, the misses it holds refresh their record's last use
 * (the step counter); the others, in top-k order, take the record with the
 * smallest (last use, record index) among those the step has not touched
 * (empty records, last use -1, first) and are read from the file into it; the
 * staging copy to the slot then comes from that record.  n_host = 0 removes
 * the tier (misses go through the two staging halves again).  Any call empties
 * the tier; moe_reset_cache, moe_set_slots and moe_set_cache_policy do too.
 * Call between steps.  Errors: MOE_ESTATE (no expert file), MOE_EINVAL
 * (n_host outside {0} + [top_k, n_experts]), MOE_ENOMEM (n_layers * n_host
 * records of pinned memory). */
moe_status moe_set_file_cache(moe_ctx *ctx, int n_host);

/* Reads bytes [offset, offset + bytes) of the file at `path` into host
 * memory `dst` with `n_threads` (1..64) threads taking chunks of
 * `chunk_bytes` (0 = one chunk), restarting short reads: the expert file
 * tier's read engine on its own.  No context, no GPU.  MOE_EINVAL for bad
 * arguments or a file that cannot be opened, MOE_ENOMEM if the threads cannot
 * be started, MOE_EIO for a failed or short read (past the end of the file). */
moe_status moe_pread_parallel(const char *path, uint64_t offset, uint64_t bytes, void *dst, int n_threads,
                              uint64_t chunk_bytes);

/* Read rate of the host link as the fused host-pool step uses it: plain
 * 16-byte loads from every SM of the current device over `bytes` (a multiple
 * of 16) of page-locked host memory at host_buf (16-byte aligned; allocated
 * with cudaHostAlloc / cudaMallocHost or registered, so the device reads it
 * through the host link), repeated `reps` times after one untimed pass on
 * `stream`; *gbs receives bytes * reps / time in GB/s (CUDA events on the
 * stream).  A measurement for the pool workload's roofline, not part of the
 * FFN.  MOE_EINVAL for bad arguments or memory the device cannot read,
 * MOE_ECUDA on a failed CUDA call (no context to poison). */
moe_status moe_host_read_rate(const void *host_buf, uint64_t bytes, int reps, void *stream, double *gbs);

/* Bytes of one routed expert / of the shared expert for a config (0 on a bad config). */
int64_t moe_expert_bytes(const moe_config *cfg);
int64_t moe_shared_bytes(const moe_config *cfg);

/* Routing only (logits, top-k, gates) without any device allocation.  The
 * write-ups this library follows have no counterpart to this call.  It is for
 * callers that cannot call cudaMalloc where they route: a host that reserves
 * all device memory up front and forbids later allocation, or a real-time
 * serving loop that cannot afford cudaMalloc's blocking, its implicit device
 * synchronisation or its failure under memory pressure.  The caller passes
 * every input and output; the arithmetic is that of the router phase of
 * moe_decode_step (optional RMS norm, exact fixed-point logits, top-k with
 * lower-index ties, softmax gates over the k picked).
 *   cfg:        d, n_experts, top_k, group, prenorm and norm_eps are used:
 *               group == 64, d a multiple of 64 and at most 3072,
 *               1 <= n_experts <= 256, 1 <= top_k <= min(n_experts, 32),
 *               prenorm 0 or 1; anything else returns MOE_EINVAL
 *   router_w:   device fp16 [n_experts][d], 16-byte aligned
 *   h:          device bf16 [B][d], 16-byte aligned
 *   logit_bias: device fp32 [B][n_experts], or NULL
 *   ids:        device int32 [B][top_k] (output); gates: device fp32 [B][top_k] (output)
 *   B:          1 <= B <= MOE_ROUTE_NOALLOC_MAX_B; a larger B returns MOE_EINVAL
 * A misaligned router_w or h (or ids, gates, logit_bias not 4-byte aligned)
 * returns MOE_EINVAL.
 * Runs on the current CUDA device, on `stream`.  Its only scratch is a fixed
 * 131,328-byte device array that every GPU loading this library holds until
 * the process exits.  The first call on each device looks up that array's
 * address once (cudaGetSymbolAddress), so make the first call on a device
 * before any stream capture.  All calls share the array and it keeps the last
 * call's contents: calls that overlap on the GPU (unordered streams) race.
 * Router products outside the exact domain (|W_r[e,i] * x[i]| >= 2^11) are
 * dropped rather than reported, and so is a logit_bias entry with
 * |b| >= 2^20 or a NaN (the logit then takes no bias).  Returns MOE_EINVAL or MOE_ECUDA on failure
 * (there is no context to poison). */
#define MOE_ROUTE_NOALLOC_MAX_B 64

moe_status moe_route_noalloc(const moe_config *cfg, const uint16_t *router_w, const void *h, int B,
                             const float *logit_bias, int32_t *ids, float *gates, void *stream);

/* Per-kernel timing.  While enabled, decode and prefill calls launch their
 * kernels one by one (no graph replay), record a CUDA event pair around every
 * launch on the call's stream, and synchronise that stream before returning
 * to add the durations to the running totals.  kind: 0 router/top-k/plan,
 * 1 gate/up GEMV, 2 down GEMV + combine, 3 persistent one-token decode
 * (all layers), 4 prefill routing and grouping (norm, router, expert
 * grouping, gather; one pair of events per layer), 5 prefill GEMMs (the four
 * tcgen05 GEMMs of one layer), 6 prefill combine, 7 small-batch grouped GEMVs
 * (the gate/up and the down launch of one layer of a call of at most 32
 * tokens). */
typedef struct {
    int64_t launches;
    double total_ms;
} moe_kernel_time;

#define MOE_N_KERNEL_KINDS 8

moe_status moe_profile(moe_ctx *ctx, int enable);

/* Copy min(n, MOE_N_KERNEL_KINDS) totals to out and reset them. */
moe_status moe_get_profile(moe_ctx *ctx, moe_kernel_time *out, int n);

/* Test hook.  hook 1: the next host-pool staging copy reports a CUDA error
 * (the call returns MOE_ECUDA and poisons the context).  hook 2: host waits
 * use a limit of `value` microseconds; value -1 makes the next host wait
 * report a timeout (after letting the awaited work finish).  hook 6: budget
 * checks see `value` bytes of free device memory (-1 restores the real
 * figure).  hook 3: programmatic dependent launch
 * between consecutive kernels on (value != 0, the default) or off.  hook 4:
 * the single-launch kernels for resident one-token decode on (value != 0, the
 * default) or off (per-layer kernels).  hook 9: among those, the clustered
 * kernel (value != 0, the default when available) or the per-SM persistent
 * kernel (0).  hook 5: `value` is the address of a caller device buffer of
 * event times (%globaltimer ns), 0 stops it.  Clustered kernel: 152 rows of
 * 32 uint64, row = CTA, columns 0..21 the first (or, for the "last" events,
 * the latest) time of each event of the call's third layer, columns 24..30
 * summed stage times (see decode_cluster.cu).  Per-SM kernel: 2 * n_layers *
 * 16 uint64, rows [0, n_layers) min or max over CTAs, rows [n_layers,
 * 2 n_layers) steps of the first routed CTA; with 2 * n_layers + gridDim.x
 * rows also per-CTA times of the third layer (see persistent.cu).
 * hook 4, 7 or 9 with a value selecting a kernel path that cannot run on the
 * configuration returns MOE_ESTATE.  hook 7: the grouped path (routing and
 * expert grouping, then tcgen05 GEMMs or small-batch GEMVs) for prefill and for
 * batched decode steps on (value != 0, the default when the shape allows it)
 * or off (per-layer batched decode kernels).
 * hook 8: `value` is a caller device buffer of 4 * 16 uint64 receiving event
 * times of CTA (0, 0) of each prefill GEMM of the first layer of a call, or
 * 0 to stop.  hook 10: every bounded device wait of the two persistent
 * decode kernels gives up after `value` SM cycles (<= 0 restores the default,
 * 4e9 cycles, about two seconds); a wait that runs out sets the abort flag,
 * every CTA drains its own copies in flight and leaves, the last one out
 * resets the launch words, and moe_sync returns MOE_ETIMEOUT and poisons the
 * context.  hook 11 (value ignored, allowed on a poisoned context): waits for
 * the device, then MOE_OK if the persistent kernels' exit counters, abort
 * flags, dependency counters and fixed-point output sums are all zero, else
 * MOE_ESTATE.  hook 12 (allowed on a poisoned context): waits for the device,
 * writes the clustered kernel's wait diagnostic into the host uint32 at
 * address `value` and clears it: 0 if no wait ran out, else (site << 16) |
 * CTA of the first wait that did (sites are listed in decode_cluster.cu).
 * hook 13: decode steps of 2 to 32 tokens and prefill calls of at most 32
 * tokens run their matrix products as small-batch grouped GEMVs (value != 0,
 * the default when the shape allows it) or as the tcgen05 GEMMs (decode: from
 * 16 tokens on, else the per-layer GEMVs); MOE_ESTATE when asked for where
 * they cannot run.
 * hook 14: resident decode steps of 2 to 4 tokens run one clustered-kernel
 * launch per token (value != 0, the default, where that kernel can run) or
 * take the batched paths of hook 13 (0).
 * Other hooks: MOE_EINVAL. */
moe_status moe_test_hook(moe_ctx *ctx, int hook, int64_t value);

const char *moe_status_string(moe_status s);

/* Last error message of the context (static string if ctx is NULL). */
const char *moe_last_error(const moe_ctx *ctx);

void moe_destroy(moe_ctx *ctx);

#ifdef __cplusplus
}
#endif

#endif /* LIBMOE_MOE_H */
