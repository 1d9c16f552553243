/*
 * moe_cache.h -- C ABI of libmoecache.so: one MoE layer over a GPU-memory cache
 * whose slots each hold one whole (layer, expert), for one GB300 (sm_103a).
 *
 * What the library computes (FreeToken, as described on four web pages):
 *
 *  - Every routed expert of the model is kept in host memory, and that copy is
 *    authoritative.  The GPU memory reserved for experts forms a single LRU
 *    cache whose slots each hold one whole expert; every table is indexed by
 *    f = layer * E + expert.  (snackonai deep dive "FreeToken, or why your
 *    laptop was never the bottleneck", sections "What It Actually Does" and
 *    "The Architecture, Unpacked".)
 *  - For each decode layer, a single kernel on the device removes duplicate
 *    routed ids, looks each one up in the residency table, computes the miss
 *    split q, finds the K slots used longest ago in a single pass, and turns
 *    each expert id into a slot id or a mark for the CPU; the host never
 *    waits on it.
 *    (same page, "The Architecture, Unpacked", decision three; ai.thesatyajit
 *    article "FreeToken: a 753B model on one GPU ...", section "Residency that
 *    follows the router", last paragraph.)
 *  - The split: q* = round(m * B_pcie / (B_pcie + B_cpu)) with B_cpu the
 *    residual host bandwidth B_H - B_P, rounded half to even, then
 *    max(1, min(q*, m)) when m > 0, then capped by K and by the evictable
 *    slots.  (snackonai, "The split policy itself"; thesatyajit, "Decode: the
 *    one equation".)
 *  - Hits and filled experts run as grouped SwiGLU work on the GPU; fills
 *    copy complete experts host -> GPU on a side stream; the combine merges
 *    the GPU partial sums with caller-supplied partial sums of CPU-assigned
 *    experts, weighted by the router gates, in fixed top-k order.
 *    (snackonai, "The split policy itself", closing note; "What It Actually
 *    Does": the merge of the partial sums is exact.)
 *  - Prefill: the slot pool lends room for two whole layers; layer l+1's
 *    experts all load on a copy stream while layer l is computed; if two
 *    layers do not fit, the routed experts load as they are needed.  (thesatyajit, "Prefill: hide the
 *    pool behind the wire"; snackonai, decision two.)
 *  - Resize: rebuild the cache for a new slot count without touching the
 *    host pool.  (snackonai, "Resizing the cache without a restart";
 *    thesatyajit, "Elastic memory, because the machine is not yours".)
 *  - Calibration: measure B_P (host -> GPU expert transfer) and B_H (host
 *    expert read) and recommend the hybrid backend iff B_H > 2 * B_P.
 *    (snackonai, "Calibration decides the backend, not the GPU".)
 *
 * Conventions for every call:
 *  - Device pointers ("_dev") are caller-owned device memory of the cache's
 *    device; host pointers ("_host") are caller-owned host memory.  The
 *    library owns the slot pool, its tables, streams and events.
 *  - Returns a moe_status; on failure moe_last_error() gives a message
 *    (thread-local, valid until the next call on the same thread).
 *  - A decode or prefill call only enqueues work on the caller's stream (a
 *    cudaStream_t passed as void*, NULL = legacy default stream) and never
 *    blocks the host.  Every other call synchronises the library's streams.
 *  - Range violations the GPU detects (an expert id outside [0, E), a
 *    CPU-assigned pair with no CPU partial sums) set an error word; the next
 *    call on the cache returns MOE_EDEVICE and clears it.  The affected
 *    outputs are left defined (id -> CPU flag, missing partial -> 0).
 *  - Not thread-safe per cache: one caller thread at a time.
 */
#ifndef MOE_CACHE_H
#define MOE_CACHE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_cache moe_cache;   /* opaque; created and freed by the library */

typedef enum moe_status {
  MOE_OK = 0,
  MOE_EINVAL = 1,     /* a bad argument (shape, pointer, layer, T, config) */
  MOE_ENOMEM = 2,     /* device or pinned host allocation failed */
  MOE_ECUDA = 3,      /* a CUDA runtime error (message has the CUDA error string) */
  MOE_ECAPACITY = 4,  /* the slot pool cannot hold what the call needs */
  MOE_EBUSY = 5,      /* reserved: a safe-point call while work is in flight */
  MOE_EDEVICE = 6     /* the GPU flagged a range violation in an earlier call */
} moe_status;

typedef enum moe_dtype {
  MOE_F32 = 0,            /* IEEE binary32 */
  MOE_BF16 = 1,           /* bfloat16 */
  MOE_FP8E4M3_B128 = 2,   /* OCP e4m3 codes with one fp32 scale per 128x128 block */
  MOE_NVFP4 = 3,          /* e2m1 codes, one e4m3 scale per 16 row elements, one fp32 scale per matrix */
  MOE_MXFP4 = 4           /* OCP MX: e2m1 codes, one e8m0 scale per 32 row elements */
} moe_dtype;

/*
 * Expert blob ("bank layout"), S bytes, one per flat id, 16-byte aligned:
 *   W_gu [2I, H] row-major in wdtype (rows 0..I-1 gate, rows I..2I-1 up),
 *   W_d  [H, I]  row-major in wdtype,
 *   MOE_FP8E4M3_B128 only: s_gu [2I/128, H/128] fp32, s_d [H/128, I/128] fp32.
 *   MOE_NVFP4: W_gu and W_d hold two e2m1 codes per byte (the even element in
 *   the low nibble), then s_gu [2I, H/16] and s_d [H, I/16] e4m3 codes (one per
 *   16 consecutive elements of a row), then fp32 g_gu, g_d and 8 bytes of zero;
 *   a weight is e2m1(code) * e4m3(its block's scale) * g of its matrix.
 *   MOE_MXFP4 (the OCP Microscaling format, one of the formats FreeToken
 *   serves: "FreeToken: a 753B model on one GPU ...", "Why this one
 *   matters"): W_gu and W_d packed as for MOE_NVFP4, then s_gu [2I, H/32] and
 *   s_d [H, I/32] e8m0 codes (one per 32 consecutive elements of a row); a
 *   weight is e2m1(code) * 2^(scale code - 127), scale code 255 being NaN.
 * S = 3*I*H*sizeof(w) (+ 4*(2I*H + H*I)/16384 for fp8; 3*I*H/2 + 3*I*H/16 + 16
 * for nvfp4; 3*I*H/2 + 3*I*H/32 for mxfp4).  H and I must be multiples of 128
 * (fp8), 32 (nvfp4, mxfp4) or 8 (f32, bf16), and S a multiple of 16 bytes (for
 * fp8: the scale count (2I/128)(H/128) + (H/128)(I/128) a multiple of 4);
 * otherwise moe_cache_create and moe_layer_ffn_noalloc return MOE_EINVAL.
 * NVFP4 and MXFP4 experts stay 4-bit in the slots and are decoded chunk by
 * chunk inside the decode GEMVs (any batch); their prefill decodes each
 * layer's routed experts to bf16 for the grouped GEMM (see moe_layer_prefill).
 */
typedef struct moe_config {
  int32_t n_layers;       /* L */
  int32_t n_experts;      /* E routed experts per layer (1..4096) */
  int32_t hidden;         /* H */
  int32_t inter;          /* I, SwiGLU intermediate size */
  int32_t top_k;          /* k (1..E) */
  int32_t max_tokens;     /* largest T of a decode call (1..1024) */
  int32_t max_fetch;      /* K: fills per layer per call; < 0 = min(E, max_tokens * k) */
  int32_t wdtype;         /* moe_dtype of the expert weights */
  int32_t adtype;         /* activations: MOE_F32 or MOE_BF16 (prefill needs MOE_BF16 and bf16 / nvfp4 / mxfp4 weights) */
  int32_t n_shared;       /* 0, or 1 always-resident shared expert per layer (gate 1.0) */
  uint32_t bw_pcie_mbps;  /* B_pcie in MB/s (> 0 unless bw_cpu_mbps > 0) */
  uint32_t bw_cpu_mbps;   /* B_cpu = B_H - B_P in MB/s; 0 = offload mode (every miss fills, up to K) */
  int32_t device;         /* CUDA device ordinal */
  int32_t max_prefill_tokens; /* largest T of a prefill call; 0 = prefill disabled */
} moe_config;

/*
 * Create a cache of n_slots slots on cfg->device.
 *   host_pool       caller-owned host memory holding the expert blobs; the
 *                   caller keeps it alive and unchanged until destroy.  If it
 *                   is not page-locked already the library registers it
 *                   (mapped, read-only) and unregisters it at destroy.
 *   host_pool_bytes its size.
 *   blob_offsets    L*E byte offsets (host array, copied), blob f at
 *                   host_pool + blob_offsets[f]; each a multiple of 16 and
 *                   offset + S <= host_pool_bytes.  NULL = dense, f * S.
 *   shared_host     n_shared == 1: L shared-expert blobs back to back (host,
 *                   copied to GPU memory at create); otherwise NULL.
 *   n_slots         C >= 1 and < 2^20.  Slots start empty (cold start).
 * Errors: MOE_EINVAL (config), MOE_ENOMEM, MOE_ECUDA.
 */
moe_status moe_cache_create(const moe_config* cfg, const void* host_pool, uint64_t host_pool_bytes,
                            const uint64_t* blob_offsets, const void* shared_host, uint64_t n_slots,
                            moe_cache** out);

/* Free everything the cache owns (synchronises its streams first).  NULL is a no-op. */
moe_status moe_cache_destroy(moe_cache* cache);

/*
 * Safe-point rebuild for n_slots slots: keeps the min(n_slots, resident) most
 * recently used experts, packed into slots 0.. in ascending old-slot order
 * with their recency; the other slots start empty.  Synchronises the device.
 * Errors: MOE_EINVAL (n_slots == 0 or >= 2^20), MOE_ENOMEM (old pool is kept).
 */
moe_status moe_cache_resize(moe_cache* cache, uint64_t n_slots);

/*
 * One MoE layer of decode for T tokens (0 <= T <= max_tokens), enqueued on `stream`.
 *   x_dev        [T, H] in adtype
 *   topk_ids_dev [T, k] int32 routed expert ids of this layer (0..E-1, distinct per token)
 *   topk_w_dev   [T, k] fp32 router gates
 *   cpu_part_dev [T, k, H] fp32 unweighted outputs of the CPU-assigned pairs, read
 *                only where the slot map says CPU; may be NULL when no pair can be
 *                CPU-assigned (offload mode with K >= k*T and enough slots)
 *   out_dev      [T, H] fp32: sum_j w[t,j] * y[t,j] in j order (+ shared expert)
 *   slot_map_dev [T, k] int32 out, may be NULL: the slot each pair ran from, -1 = CPU
 * x_dev, cpu_part_dev and out_dev must be 16-byte aligned, the int32 / fp32
 * arrays 4-byte aligned (MOE_EINVAL otherwise, before anything is enqueued).
 * Errors: MOE_EINVAL, MOE_EDEVICE (earlier violation), MOE_ECUDA.
 * The resident experts run as a gate/up grid then a down + combine grid.  With
 * MOE_DECODE_RESIDENT=fused (or MOE_DECODE_FUSED=1) in the environment when the
 * cache is created, one-token calls on bf16 caches with at most top-8 routed
 * experts and no shared expert run both in one launch with a grid-wide barrier
 * between them instead (same outputs bit for bit).
 * With a CPU branch registered (moe_cache_set_cpu_branch) cpu_part_dev is
 * ignored.
 */
moe_status moe_layer_decode(moe_cache* cache, int32_t layer, int32_t T, const void* x_dev,
                            const int32_t* topk_ids_dev, const float* topk_w_dev,
                            const float* cpu_part_dev, float* out_dev, int32_t* slot_map_dev,
                            void* stream);

/*
 * One MoE layer of a prefill chunk of T tokens (1 <= T <= max_prefill_tokens), bf16
 * activations and bf16, nvfp4 or mxfp4 weights.  Full-layer mode (C >= 2E): makes
 * layer `layer` resident, starts loading all of layer+1 on the transfer stream, runs
 * the grouped GEMM on `stream`, and marks the layer's E experts used.  C < 2E: loads
 * the routed experts of the layer on demand, at most C at a time.  4-bit experts stay
 * 4-bit in their slots (the host link carries 4-bit blobs); before the GEMMs each
 * routed expert is decoded to a bf16 blob in a device staging area of E * 6*I*H
 * bytes that the cache allocates at create time (MXFP4 values are exact in bf16,
 * NVFP4 values e2m1 * e4m3 * g are rounded to nearest bf16).
 *   x_dev [T, H] bf16, topk_ids_dev / topk_w_dev [T, k], out_dev [T, H] fp32 (overwritten).
 * x_dev and out_dev 16-byte aligned, topk_ids_dev / topk_w_dev 4-byte aligned.
 * Errors: MOE_EINVAL, MOE_EDEVICE, MOE_ECUDA.
 */
moe_status moe_layer_prefill(moe_cache* cache, int32_t layer, int32_t T, const void* x_dev,
                             const int32_t* topk_ids_dev, const float* topk_w_dev, float* out_dev,
                             void* stream);

/*
 * The second prefill buffer on (on = 1, the default) or off (on = 0), for the
 * no-second-buffer comparison of ai.thesatyajit.com "FreeToken: a 753B model
 * on one GPU, and the two bandwidths that decide everything", section
 * "Prefill: hide the pool behind the wire" (also snackonai "FreeToken, or why
 * your laptop was never the bottleneck", section "It In Action").  Off, a
 * full-layer prefill call loads only the missing experts of its own layer,
 * into victims that exclude that layer's slots, and its GEMMs start once those
 * loads are done: nothing of the next layer loads while this one computes.
 * Takes effect from the next prefill call.  Errors: MOE_EINVAL (NULL cache,
 * prefill disabled, on not 0 or 1).
 */
moe_status moe_cache_set_prefill_prefetch(moe_cache* cache, int32_t on);

/*
 * Copy the residency state to host arrays (synchronises the device); any pointer may be NULL.
 *   slot_to_expert_host [C] int32 (-1 = empty), stamps_host [C] uint64 (0 = empty; a
 *   larger stamp = more recently used), expert_to_slot_host [L*E] int32 (-1 = not resident),
 *   counters_host [8] uint64: unique hits, unique misses, fills, CPU-assigned, pair reads
 *   that hit, pair reads that missed, decode calls, experts loaded by prefill;
 *   clock_host: the last stamp handed out.
 */
moe_status moe_cache_get_state(moe_cache* cache, int32_t* slot_to_expert_host, uint64_t* stamps_host,
                               int32_t* expert_to_slot_host, uint64_t* counters_host,
                               uint64_t* clock_host);

/*
 * The last decode call's plan (synchronises the device); any pointer may be NULL.
 *   scalars_host [8] int32: layer, unique u, hits h, misses m, fills q, CPU-assigned,
 *                GPU experts run (h + q + shared), 0.
 *   victims_host [K] int32: the K least-recently-used evictable slots in eviction
 *                order (key (stamp, slot) ascending, this call's hits excluded), -1 padded.
 *   fills_host   [2K] int32: (flat id, slot) of the q fills, in fill order.
 *   y_host       [T, k, H] fp32: the GPU partial sum of each GPU-run pair (unweighted),
 *                undefined for CPU-assigned pairs.
 */
moe_status moe_cache_get_plan(moe_cache* cache, int32_t* scalars_host, int32_t* victims_host,
                              int32_t* fills_host, float* y_host);

/*
 * Sizes of a cache: info_host[8] uint64: slot bytes S, slots C, K, L*E,
 * device bytes held, host pool bytes, kernel launches of one decode call of
 * max_tokens tokens (with a CPU branch registered: its combine kernel
 * included), and how such a call runs its resident experts: 0 = a gate/up grid
 * then a down + combine grid, 1 = one launch with a grid-wide barrier between
 * gate/up and down + combine.
 */
moe_status moe_cache_info(moe_cache* cache, uint64_t* info_host);

/*
 * Kernel timing with CUDA event pairs around every kernel group the cache
 * launches.  mode 1: start (reset; 4096 event pairs are created here, so a
 * stream capture that follows records into existing events); mode 3: pause
 * (keep the pairs recorded so far, e.g. those captured into a graph, record no
 * new ones); mode 2: synchronise and read the sums over the recorded pairs
 * (after each replay of a captured graph its pairs hold that replay's times);
 * mode 0: stop, read and reset.  Per kind the summed milliseconds and the
 * number of timed groups: 0 control, 1 fill (with the gate/up GEMV of the
 * filled experts), 2 GEMV of the resident experts (gate/up, and, when the down
 * projection is split, their down projection + combine), 3 down-projection GEMV
 * of the filled experts (split), 4 down-projection GEMV of every GPU expert +
 * combine (not split), 5 prefill control, 6 prefill load, 7 prefill grouped GEMM.  ms_host[8] and
 * launches_host[8] may be NULL.
 */
moe_status moe_cache_profile(moe_cache* cache, int32_t mode, double* ms_host, uint64_t* launches_host);

/*
 * Calibrate on `device` with expert-sized blobs of expert_bytes (rounded up to 16).
 *   b_pcie_gbs         B_P: host -> GPU expert transfer, GB/s (1e9 B/s), through the
 *                      library's own fill path (SM copy from page-locked host memory)
 *   b_host_gbs         B_H: host-side expert read bandwidth, GB/s (all host threads
 *                      streaming the pool, the bytes an in-place CPU expert reads)
 *   recommend_hybrid   1 iff B_H > 2.0 * B_P, else 0
 * Any output may be NULL.  Allocates and frees its own buffers.  Synchronises.
 */
moe_status bench_bw(int32_t device, uint64_t expert_bytes, double* b_pcie_gbs, double* b_host_gbs,
                    int32_t* recommend_hybrid);

/*
 * One MoE layer's expert SwiGLU + combine without allocating any GPU memory.
 * (This call has no counterpart on the pages; it is an addition for callers
 * that may not allocate.)
 *
 * Who it is for: code that may not call cudaMalloc -- a plug-in running inside
 * another framework's memory pool, a process that reserved all GPU memory at
 * start-up, or a runtime that forbids allocations after start so its memory
 * use stays fixed.  The caller passes inputs and outputs only; every
 * intermediate lives in one fixed 16 MiB device array inside this library
 * (every GPU that loads the library holds it until the process exits).
 *
 * What it computes: the same output as moe_layer_decode when every routed
 * expert of the layer is resident and nothing is CPU-assigned:
 *   out[t] = sum_j w[t,j] * SwiGLU_{ids[t,j]}(x[t]), summed in j order in fp32.
 *   experts_dev  the layer's E expert blobs back to back (bank layout above,
 *                S bytes each), device memory, 16-byte aligned
 *   x_dev [T, H] in adtype, topk_ids_dev / topk_w_dev [T, k], out_dev [T, H] fp32
 *   (x_dev and out_dev 16-byte aligned, the id and gate arrays 4-byte aligned)
 * Ids outside [0, E) contribute nothing.  Enqueued on `stream`; never blocks.
 * wdtype MOE_F32, MOE_BF16 or MOE_FP8E4M3_B128 (MOE_NVFP4 and MOE_MXFP4 are
 * MOE_EINVAL here).
 *
 * Limits and sharing:
 *   - scratch needed ~ T * top_k * (H + I) * 4 bytes plus small lists; a call
 *     that needs more than 16 MiB, or that routes more than 9216 pairs
 *     (T * top_k), returns MOE_ECAPACITY with a message.
 *   - range violations the GPU finds in this call (an id outside [0, E)) are
 *     not reported: such a pair contributes nothing and no later call returns
 *     MOE_EDEVICE for it.
 *   - every call on a device uses the same scratch array and leaves its
 *     contents behind; each call rewrites everything it reads first, so
 *     nothing needs clearing, but calls that overlap on the GPU (different
 *     streams, no ordering between them) race and corrupt each other.
 *   - the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 */
moe_status moe_layer_ffn_noalloc(int32_t n_experts, int32_t hidden, int32_t inter, int32_t top_k,
                                 int32_t wdtype, int32_t adtype, const void* experts_dev, int32_t T,
                                 const void* x_dev, const int32_t* topk_ids_dev, const float* topk_w_dev,
                                 float* out_dev, void* stream);

/*
 * The CPU branch of the decode step.  The CPU-assigned experts run on the host,
 * started from a host-function node of the same captured graph, between a copy
 * to the host of what they read and a copy back of their partial sums; the GPU
 * path runs beside them and the exact merge waits for both, so a layer costs the
 * longer of the two branches.  (ai.thesatyajit.com "FreeToken: a 753B model on
 * one GPU ...", section "Residency that follows the router", last paragraph;
 * snackonai "FreeToken, or why your laptop was never the bottleneck", section
 * "It In Action".)  The library has no CPU expert executor of its own: the
 * caller registers the function that computes the CPU-assigned pairs.
 *
 * With fn registered, every moe_layer_decode call on the cache enqueues, after
 * its control kernel and on a stream of the library: copies of x, the routed
 * ids and the slot map into page-locked memory the library owns; a host
 * function (cudaLaunchHostFunc) that calls
 *   fn(user, layer, T, x_host [T, H] in adtype, topk_ids_host [T, k] int32,
 *      slot_map_host [T, k] int32, cpu_part_host [T, k, H] fp32)
 * which must write cpu_part_host[t, j, :], the unweighted output of expert
 * topk_ids[t, j] applied to x[t], wherever slot_map_host[t, j] < 0 (other
 * entries are not read); then a copy of cpu_part_host to device memory the
 * library owns.  The down kernels of the call only store the GPU pairs'
 * outputs; one combine kernel on the caller's stream waits for both branches
 * and forms out in top-k order.  The call's cpu_part_dev argument is ignored.
 * fn runs on a CUDA driver thread, must not call CUDA, and must not wait on
 * anything that waits on the stream; the pointers it gets are valid only
 * during the call.  Everything is stream-ordered and capturable in a CUDA
 * graph (the host function becomes a host node; a graph captured before fn is
 * registered again must be captured again).  fn NULL removes the branch.
 * Synchronises the device.  Errors: MOE_EINVAL (NULL cache), MOE_ENOMEM.
 */
typedef void (*moe_cpu_branch_fn)(void* user, int32_t layer, int32_t T, const void* x_host,
                                  const int32_t* topk_ids_host, const int32_t* slot_map_host,
                                  float* cpu_part_host);
moe_status moe_cache_set_cpu_branch(moe_cache* cache, moe_cpu_branch_fn fn, void* user);

/* The message of the last failed call on this thread ("" if none). */
const char* moe_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_CACHE_H */
