/*
 * moe.h -- C ABI of the GB300 MoE expert-parallel layer forward (libmoe.so).
 *
 * The layer the pages describe, on one GPU:
 *   route          gate a batch of hidden states, top-k          (moe_route)
 *   plan dispatch  group token rows per expert into batches      (moe_plan_dispatch)
 *   expert FFN     run every batch through its SwiGLU expert     (moe_expert_ffn)
 *   combine        gate-weighted sum + shared expert (+residual) (moe_combine)
 *   layer forward  all four in one stream-ordered sequence       (moe_layer_forward)
 * Sources: "Distributed MoE" (tenzro docs) -- the RPC list (route, execute,
 * forward), the tenzro_moePlanDispatch records, the router-families and
 * expert-host-runtime paragraphs; "Expert-Sharded Swarm Inference: The Design"
 * (kvasir) -- the layer pseudocode; "Expert-sharding" (kvasir wiki), section
 * "Twee rollen" -- the worker request (n_used, n_tokens, cur, sel).
 *
 * Conventions for every call
 *   - Pointers are DEVICE pointers unless stated otherwise; the caller owns every
 *     buffer.  The library allocates no device memory: scratch comes from the
 *     caller's workspace, sized by moe_workspace_size().
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every call is asynchronous and stream-ordered; no call synchronizes the
 *     device except moe_get_device_status().  The calls can be captured in a
 *     CUDA graph.
 *   - Argument errors are returned synchronously, before anything is launched.
 *     A failed launch returns MOE_ERR_CUDA.  Problems only the device can see
 *     (an expert id out of range, a bounded wait that expired) set a sticky
 *     flag in the workspace that moe_get_device_status() reports.  No exception
 *     or abort crosses the ABI.
 *   - T = 0 is a valid no-op (MOE_OK, nothing launched).
 *   - All pointers must be 16-byte aligned; row-major tensors are contiguous.
 *
 * Layouts (row-major; the expert index is the outermost dimension, so each
 * expert's weights are one contiguous slab -- "Expert-Sharded Swarm Inference:
 * The Design", slicing paragraph; projections are Y = X * W^T with W stored
 * [out, in] -- "Distributed MoE", compute-seam paragraph):
 *   x        [T, d]          dtype                 hidden states (already normed)
 *   Wr       [E, d]          dtype                 router
 *   Wg, Wu   [E+S, I, d]     dtype                 gate / up projections
 *   Wd       [E+S, d, I]     dtype                 down projection
 *   experts 0..E-1 are routed, E..E+S-1 are the shared experts.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment or flag */
  MOE_ERR_UNSUPPORTED = 2,  /* valid but not supported (see constraints) */
  MOE_ERR_WORKSPACE = 3,    /* workspace missing or smaller than moe_workspace_size() */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
  MOE_ERR_TIMEOUT = 5,      /* device: a bounded wait inside a kernel expired */
  MOE_ERR_DEVICE_INPUT = 6  /* device: an input value was out of range (e.g. expert id) */
} moe_status;

/* Gating families ("Distributed MoE", router-families paragraph). */
typedef enum {
  /* Qwen layout: w = softmax(logits)[top-k of logits]; renormalised over the
     top-k only when norm_topk != 0; times routed_scaling (1.0 normally). */
  MOE_GATE_SOFTMAX_TOPK = 0,
  /* DeepSeek / Kimi layout: s = sigmoid(logits); the top-k of s + sel_bias is
     selected; w = s[sel] (divided by its sum over the selection when
     norm_topk != 0) times routed_scaling.  The bias only selects. */
  MOE_GATE_SIGMOID_BIAS = 1
} moe_gate_kind;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* The self-describing layer record: shapes plus gating metadata
   ("Distributed MoE", router-families paragraph: the gate blob carries its
   bias and scaling metadata). */
typedef struct {
  int32_t layer;           /* carried for the caller's bookkeeping; not used */
  int32_t T;               /* tokens in the batch (>= 0) */
  int32_t d;               /* hidden size */
  int32_t E;               /* routed experts */
  int32_t k;               /* experts per token, 1 <= k <= min(E, 32) */
  int32_t I;               /* SwiGLU intermediate size (routed and shared) */
  int32_t S;               /* shared experts, 0 <= S <= 4, weight 1.0 each */
  int32_t gate;            /* moe_gate_kind */
  int32_t norm_topk;       /* 0 / 1 */
  float routed_scaling;    /* multiplies the routed gate weights */
  int32_t dtype;           /* moe_dtype of x and of every weight */
} moe_layer_desc;

/* Constraints: dtype MOE_BF16 needs d % 64 == 0 and I % 64 == 0 (tensor-core
   path) and (E+S) * min(d, I) >= 128; MOE_F32 needs d % 8 == 0 and
   I % 4 == 0.  E <= 1024, T * (k + S) <= 2^30.  Violations return
   MOE_ERR_UNSUPPORTED.  Routing ids handed to moe_plan_dispatch must be
   distinct within a token (as any top-k is). */

/* Bytes of workspace any call below needs for this layer (0 when T == 0).
   The same buffer may be reused by every call on the same stream. */
moe_status moe_workspace_size(const moe_layer_desc* desc, size_t* bytes);

/* Clears the workspace's device-status flag (asynchronously, on `stream`).
   moe_layer_forward clears it itself; call this once on a fresh workspace
   before using the individual calls with moe_get_device_status(). */
moe_status moe_workspace_init(void* workspace, size_t ws_bytes, void* stream);

/* moe_route -- gate a batch ("Distributed MoE", RPC list: route; layer
   pseudocode: ids, p = top_k(softmax(cur @ router), k)).
     logit_bias [E] fp32 or NULL: added to every token's router logits
                 (a per-expert logit offset, both families).
     sel_bias   [E] fp32 or NULL: selection bias, sigmoid family only
                 (MOE_ERR_INVALID_ARG with the softmax family).
     topk_ids   [T, k] int32 out: descending selection score, ties to the
                 lower expert index.
     topk_w     [T, k] fp32 out: gate weights of those experts.            */
moe_status moe_route(const moe_layer_desc* desc, const void* x, const void* Wr,
                     const float* logit_bias, const float* sel_bias, int32_t* topk_ids,
                     float* topk_w, void* workspace, size_t ws_bytes, void* stream);

/* moe_plan_dispatch -- invert the routing into per-expert batches
   ("Distributed MoE", tenzro_moePlanDispatch records: batches of
   token_indices per (layer, expert) and per-token slot assignments).
   Pairs (t, j), j < k routed (expert topk_ids[t, j]) and j = k + s shared
   (expert E + s), are placed by a stable counting sort in token-major order:
     expert_offsets [E+S+1] int32 out: batch e = rows offsets[e] .. offsets[e+1]
     token_indices  [T*(k+S)] int32 out: token of each batch row, ascending
                    inside every batch
     slot_row       [T, k+S] int32 out: batch row of pair (t, j) (the token
                    assignments; token_indices[slot_row[t, j]] == t)
     active_ids     [E+S] int32 out (or NULL): experts with a non-empty batch,
                    ascending; n_active [1] int32 out (or NULL) their count.
     topk_w         [T, k] fp32 in (or NULL), slot_w [T*(k+S)] fp32 out (or
                    NULL): the gate weight of every batch row (1.0 for shared
                    rows), for moe_expert_ffn's optional row scaling.
   An id outside [0, E) sets MOE_ERR_DEVICE_INPUT in the workspace flag; that
   pair is dropped (slot_row = -1) and nothing is written out of bounds.     */
moe_status moe_plan_dispatch(const moe_layer_desc* desc, const int32_t* topk_ids,
                             const float* topk_w, int32_t* expert_offsets,
                             int32_t* token_indices, int32_t* slot_row, int32_t* active_ids,
                             int32_t* n_active, float* slot_w, void* workspace, size_t ws_bytes,
                             void* stream);

/* moe_expert_ffn -- run every batch through its expert ("Distributed MoE",
   RPC list: execute; expert-host-runtime paragraph: SwiGLU over gate/up/down;
   "Expert-sharding", section "Twee rollen": the worker's three mat-muls):
     y_perm[r] = slot_w[r] * Wd_e (silu(Wg_e x_t) * (Wu_e x_t)),
   for every batch row r of expert e with token t = token_indices[r];
   slot_w NULL means a factor of 1.  y_perm is [T*(k+S), d] in the layer's
   dtype (bf16 rows for MOE_BF16, fp32 for MOE_F32).                      */
moe_status moe_expert_ffn(const moe_layer_desc* desc, const void* x,
                          const int32_t* expert_offsets, const int32_t* token_indices,
                          const float* slot_w, const void* Wg, const void* Wu, const void* Wd,
                          void* y_perm, void* workspace, size_t ws_bytes, void* stream);

/* moe_expert_ffn_noalloc -- moe_expert_ffn for callers that cannot allocate
   device memory.  The pages have no counterpart to this call; it exists for
   callers that cannot lend the library a workspace: code inside a host
   application that owns all device memory through its own allocator and
   offers no way to get more, or latency-critical code that must never call
   cudaMalloc (which may synchronize the device).  Inputs, outputs and results
   are those of moe_expert_ffn; the scratch (gathered rows and the SwiGLU
   intermediate) lives in a fixed 64 MiB array inside the library instead:
     - a layer needing more (256 B + two buffers of round32(T*(k+S)) + 256 rows
       of d and of I elements) returns MOE_ERR_UNSUPPORTED, launching nothing;
     - every GPU that loads the library's device code holds the array until
       the process exits;
     - all calls on a device share the array and it keeps the last call's
       contents: calls that overlap on the GPU race, so the caller must order
       them (one stream, or explicit dependencies);
     - the first call on each device looks up the array's address with that
       device current and keeps it; make that first call before any stream
       capture; the kept address does not survive a device reset
       (cudaDeviceReset), so the call must not be used on a device after it
       has been reset;
     - device-detected problems (bad token indices, timeouts) are not reported
       by this call; use moe_expert_ffn with a workspace to see them.
   Nothing is allocated: no cudaMalloc, cudaFree or allocating library call. */
moe_status moe_expert_ffn_noalloc(const moe_layer_desc* desc, const void* x,
                                  const int32_t* expert_offsets, const int32_t* token_indices,
                                  const float* slot_w, const void* Wg, const void* Wu,
                                  const void* Wd, void* y_perm, void* stream);

/* moe_combine -- gate-weighted sum per token plus the shared experts
   ("Distributed MoE", expert-host-runtime paragraph: recombine weighted by
   the gate probabilities; layer pseudocode: combine(p, partials) + shared):
     y[t] = sum_{j<k} topk_w[t, j] * y_perm[slot_row[t, j]]
            + sum_{s<S} y_perm[slot_row[t, k+s]]  (+ residual[t])
   summed in that fixed order in fp32.  topk_w NULL means the rows are
   already weighted (moe_expert_ffn with slot_w).  residual [T, d] fp32 or
   NULL; y [T, d] fp32 out.  Rows whose slot_row is -1 are skipped.        */
moe_status moe_combine(const moe_layer_desc* desc, const void* y_perm, const int32_t* slot_row,
                       const float* topk_w, const float* residual, float* y, void* stream);

/* moe_combine_partial -- the combine when some experts did not respond
   ("Distributed MoE", failover paragraph: allow_partial renormalises the gate
   weights over the experts that responded and reports the unserved
   (expert, token) pairs as missing -- serving with a reduced top-k).
     topk_ids         [T, k] int32 and topk_w [T, k] fp32: the routing.
     expert_available [E+S] int32: nonzero for experts whose rows in y_perm
                      are valid (rows of the others are never read).
     missing          [T, k+S] int32 out (or NULL): 1 for every slot whose
                      expert was unavailable, else 0.
   For token t, mass = sum_j topk_w[t, j] and resp = the same sum over the
   available routed slots (slot order, fp32); an available routed slot
   weighs topk_w[t, j] * (mass / resp), so the token keeps its routed gate
   mass and, with every expert available, the result is moe_combine's
   exactly.  A token with no available routed expert gets no routed term;
   an unavailable shared expert is left out.  y and residual as in
   moe_combine; y_perm rows must not be pre-weighted. */
moe_status moe_combine_partial(const moe_layer_desc* desc, const void* y_perm,
                               const int32_t* slot_row, const int32_t* topk_ids,
                               const float* topk_w, const int32_t* expert_available,
                               const float* residual, float* y, int32_t* missing,
                               void* stream);

/* moe_partial_missing_pairs -- the unserved pairs of a partial combine as a
   list ("Distributed MoE", failover paragraph: allow_partial reports the
   (expert, token) pairs it could not serve under `missing`).
     topk_ids [T, k] int32: the routing given to moe_combine_partial.
     missing  [T, k+S] int32: the mask moe_combine_partial wrote.
     pairs    [T*(k+S), 2] int32 out (8-byte aligned): (expert, token) of
              every flagged slot, ordered by token, then slot (the shared
              expert s of a token is expert E+s); entries past the count are
              left untouched.
     n_pairs  [1] int32 out: the number of pairs.
   Device pointers, caller-owned; stream-ordered.  T == 0 writes a count of
   0.  Argument errors return before any launch. */
moe_status moe_partial_missing_pairs(const moe_layer_desc* desc, const int32_t* topk_ids,
                                     const int32_t* missing, int32_t* pairs, int32_t* n_pairs,
                                     void* stream);

/* moe_layer_forward -- gate -> plan -> expert FFN -> combine ("Distributed
   MoE", RPC list: forward).  topk_ids_out [T, k] / topk_w_out [T, k] may be
   NULL; everything else as in the calls above.                             */
moe_status moe_layer_forward(const moe_layer_desc* desc, const void* x, const void* Wr,
                             const float* logit_bias, const float* sel_bias, const void* Wg,
                             const void* Wu, const void* Wd, const float* residual, float* y,
                             int32_t* topk_ids_out, float* topk_w_out, void* workspace,
                             size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- Q8_0 expert weights
   ("Distributed MoE", quantization table: Q8_0 = 32-element blocks with one
   f16 scale, about 8.5 bits per weight; the prepare job block-quantizes
   each expert projection, and a holder decodes it with its dequant path.)
   The block contents are GGUF's; the arrangement is planar for the GPU:
     q     int8 codes in the weight's own layout, [n_mats, rows, K]
     scale f16 bit patterns, transposed per matrix, [n_mats, K/32, rows]
   Block b of row r represents scale[m][b][r] * q[m][r][32b .. 32b+31]. */
typedef struct {
  const void* q;      /* int8  [E+S, rows, K] */
  const void* scale;  /* f16   [E+S, K/32, rows] */
} moe_q8_weight;

/* moe_quantize_q8_0 -- quantize n_mats row-major [rows, K] matrices (fp32 or
   bf16, src_dtype a moe_dtype) into Q8_0: for each 32-element block,
   d = max|w| / 127, q = round-half-away(w / d) computed as w * (1/d) in fp32,
   scale = f16(d).  K % 32 == 0.  q and scale are device outputs sized as in
   moe_q8_weight. */
moe_status moe_quantize_q8_0(int n_mats, int rows, int K, int src_dtype, const void* w, void* q,
                             void* scale, void* stream);

/* moe_expert_ffn_q8 / moe_layer_forward_q8 -- moe_expert_ffn and
   moe_layer_forward with Q8_0 expert projections (router weights stay in the
   layer's dtype).  desc->dtype must be MOE_BF16 (activations); each weight
   is dequantized on chip (scale * q rounded to bf16) and fed to the same
   tensor-core path.  Wg/Wu have rows = I and K = d; Wd has rows = d, K = I. */
moe_status moe_expert_ffn_q8(const moe_layer_desc* desc, const void* x,
                             const int32_t* expert_offsets, const int32_t* token_indices,
                             const float* slot_w, const moe_q8_weight* Wg,
                             const moe_q8_weight* Wu, const moe_q8_weight* Wd, void* y_perm,
                             void* workspace, size_t ws_bytes, void* stream);
moe_status moe_layer_forward_q8(const moe_layer_desc* desc, const void* x, const void* Wr,
                                const float* logit_bias, const float* sel_bias,
                                const moe_q8_weight* Wg, const moe_q8_weight* Wu,
                                const moe_q8_weight* Wd, const float* residual, float* y,
                                int32_t* topk_ids_out, float* topk_w_out, void* workspace,
                                size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- expert tier in host memory
   ("Distributed MoE", expert-residency paragraph: experts are kept in a
   byte-bounded, least-recently-used memory tier over a colder tier, and
   before a forward dispatches, readahead brings in the experts the routing
   decision selected; "Module expert_store" (ferrox-core docs), design list:
   a lease pins an entry against eviction while work still reads it, and a
   step whose experts do not all fit still succeeds, at the cost of more
   transfers.)
   Here the colder tier is host memory (on GB300 the Grace memory, read over
   NVLink-C2C) and the bounded tier is a pool of expert slots in HBM. */
typedef struct {
  uint64_t steps;         /* assignments made (forwards and prefetches) */
  uint64_t hits;          /* experts already resident when a step needed them */
  uint64_t misses;        /* experts brought into a slot */
  uint64_t evictions;     /* resident experts displaced to make room */
  uint64_t extra_passes;  /* FFN passes beyond the first: a step needed more experts than slots */
  uint64_t bytes_loaded;  /* host -> device weight bytes (a bare slot cache reports 0) */
  int32_t n_slots;
  int32_t resident;       /* slots holding an expert */
} moe_tier_stats;

/* The residency logic on its own (host only, no device needed).  A cache of
   n_slots slots over experts 0 .. n_experts-1 (1 <= n_slots <= n_experts).
   moe_slot_cache_assign gives one step's n distinct experts their slots:
   slot[i]; load[i] = 1 when expert i's bytes must be brought into that slot
   (a miss), 0 when it is resident (a hit); pass[i], the pass that uses it.
   Pass 0 holds every hit and as many misses as fit; a miss takes a free
   slot, else the least recently used slot not pinned by the current pass
   (its expert is evicted); when every slot is pinned, a new pass starts and
   the pins are dropped.  Passes must run one after another.  *n_passes is
   the number of passes (0 for n = 0).  A repeated or out-of-range expert is
   MOE_ERR_INVALID_ARG with the cache unchanged.  Thread-safe per cache.
   moe_slot_cache_slot_of: an expert's slot, or -1 when not resident. */
typedef struct moe_slot_cache moe_slot_cache;
moe_status moe_slot_cache_create(int n_slots, int n_experts, moe_slot_cache** out);
moe_status moe_slot_cache_destroy(moe_slot_cache* cache);
moe_status moe_slot_cache_assign(moe_slot_cache* cache, const int32_t* experts, int n,
                                 int32_t* slot, int32_t* load, int32_t* pass,
                                 int32_t* n_passes);
moe_status moe_slot_cache_slot_of(moe_slot_cache* cache, int expert, int32_t* slot);
moe_status moe_slot_cache_get_stats(moe_slot_cache* cache, moe_tier_stats* out);

/* Host memory for the tier's expert projections: page-locked, aligned to the
   host's transparent-huge-page size and backed by huge pages where the host
   allows it (zero-filled).  Host -> device copies from such memory keep the
   link's bandwidth even on first touch of a large region; copies from
   base-page memory can run at half of it.  Free with moe_host_free (which
   rejects pointers it did not hand out).  Host only; MOE_ERR_CUDA when the
   allocation or page-locking fails. */
moe_status moe_host_alloc(size_t bytes, void** out);
moe_status moe_host_free(void* ptr);

/* The expert tier.  moe_tier_create keeps pointers to the layer's expert
   projections in HOST memory (bf16, layouts as in moe_layer_forward:
   Wg/Wu [E+S, I, d], Wd [E+S, d, I]); the caller keeps them alive and
   unchanged until moe_tier_destroy (moe_host_alloc memory is the fast
   choice).  The tier page-locks them if they are not already (and unlocks
   what it locked on destroy), and allocates
   n_slots = min(E+S, floor(hbm_budget_bytes / (6 I d))) expert slots in
   HBM on the current device (MOE_ERR_INVALID_ARG below one slot).  desc
   fixes d, E, k, I, S, gate and dtype (MOE_BF16 only; other dtypes are
   MOE_ERR_UNSUPPORTED); its T is ignored.

   moe_tier_forward is moe_layer_forward over the tier, with desc giving
   this call's T: route and plan on the device; the routing decision (the
   expert batch sizes) is copied to the host, which WAITS for the stream
   once; slots are assigned (moe_slot_cache_assign), the missing experts
   are copied into their slots (on a copy stream of the tier's, ordered
   after the work already on `stream`), and the FFN runs once per pass
   over the experts of that pass; then the combine.  The result equals
   moe_layer_forward's bit for bit.  Calls on one tier are serialized
   (the tier orders its work after its previous call's, whatever stream).
   moe_tier_prefetch brings up to n_slots of the listed experts in ahead of
   use (a caller-supplied hotlist), asynchronously, ordered after `stream`.
   moe_tier_destroy waits for the tier's outstanding work. */
typedef struct moe_expert_tier moe_expert_tier;
moe_status moe_tier_create(const moe_layer_desc* desc, const void* Wg_host, const void* Wu_host,
                           const void* Wd_host, size_t hbm_budget_bytes, moe_expert_tier** out);
moe_status moe_tier_destroy(moe_expert_tier* tier);
moe_status moe_tier_prefetch(moe_expert_tier* tier, const int32_t* experts, int n, void* stream);
moe_status moe_tier_forward(moe_expert_tier* tier, const moe_layer_desc* desc, const void* x,
                            const void* Wr, const float* logit_bias, const float* sel_bias,
                            const float* residual, float* y, int32_t* topk_ids_out,
                            float* topk_w_out, void* workspace, size_t ws_bytes, void* stream);
moe_status moe_tier_get_stats(moe_expert_tier* tier, moe_tier_stats* out);

/* The layer call with host buffers (the pages' forward RPC, its input and
   output on the host side): x_host ([T, d], the layer's dtype) is copied into
   the workspace, the layer runs exactly as moe_layer_forward (or
   moe_layer_forward_q8) on it, and y ([T, d] fp32) is copied to y_host; all
   enqueued on `stream`, asynchronously, so y_host holds the result once the
   stream has passed the call (page-locked host buffers make the copies
   asynchronous).  The other pointers (weights, biases, residual, top-k
   outputs) are device memory as for moe_layer_forward.  Errors as
   moe_layer_forward; MOE_ERR_INVALID_ARG for a NULL host buffer. */
moe_status moe_layer_forward_host(const moe_layer_desc* desc, const void* x_host,
                                  const void* Wr, const float* logit_bias,
                                  const float* sel_bias, const void* Wg, const void* Wu,
                                  const void* Wd, const float* residual, float* y_host,
                                  int32_t* topk_ids_out, float* topk_w_out, void* workspace,
                                  size_t ws_bytes, void* stream);
moe_status moe_layer_forward_q8_host(const moe_layer_desc* desc, const void* x_host,
                                     const void* Wr, const float* logit_bias,
                                     const float* sel_bias, const moe_q8_weight* Wg,
                                     const moe_q8_weight* Wu, const moe_q8_weight* Wd,
                                     const float* residual, float* y_host,
                                     int32_t* topk_ids_out, float* topk_w_out, void* workspace,
                                     size_t ws_bytes, void* stream);

/* A run of n_steps layer calls with host buffers, the copies overlapped with
   the neighbouring steps' compute (a serving loop over batches of T tokens
   that live in host memory, as the forward RPC delivers them).  Step i reads
   x_host[i] ([T, d], the layer's dtype) and writes y_host[i] ([T, d] fp32);
   its layer is exactly moe_layer_forward's (moe_layer_forward_q8's) on that
   input, with no residual and no top-k outputs, so y_host[i] equals the
   single call's result bit for bit.  The layer runs on `stream`; two copy
   streams owned by the call move the data: step i + 1's input goes up while
   step i computes, step i's output comes down while step i + 1 computes (two
   x and two y stages in the workspace).  Ordering: the run starts after the
   work enqueued on `stream` before the call, and `stream` waits for the last
   copy, so work enqueued on it after the call sees every y_host[i] written.
   Host buffers should be page-locked (otherwise the copies serialize with
   the host).  x_host and y_host are host arrays of n_steps pointers; an entry
   may repeat (the copies of one direction run in step order).  n_steps == 0
   or T == 0: MOE_OK, nothing enqueued.  Errors as moe_layer_forward;
   MOE_ERR_INVALID_ARG for n_steps < 0 or a NULL array or entry. */
moe_status moe_layer_forward_host_pipelined(const moe_layer_desc* desc, int n_steps,
                                            const void* const* x_host, const void* Wr,
                                            const float* logit_bias, const float* sel_bias,
                                            const void* Wg, const void* Wu, const void* Wd,
                                            float* const* y_host, void* workspace,
                                            size_t ws_bytes, void* stream);
moe_status moe_layer_forward_q8_host_pipelined(const moe_layer_desc* desc, int n_steps,
                                               const void* const* x_host, const void* Wr,
                                               const float* logit_bias, const float* sel_bias,
                                               const moe_q8_weight* Wg, const moe_q8_weight* Wu,
                                               const moe_q8_weight* Wd, float* const* y_host,
                                               void* workspace, size_t ws_bytes, void* stream);

/* Synchronizes `stream`, then reports the sticky device flag held in the
   workspace: MOE_OK, MOE_ERR_DEVICE_INPUT or MOE_ERR_TIMEOUT (MOE_ERR_CUDA if
   the copy itself fails).  clear != 0 resets the flag afterwards.          */
moe_status moe_get_device_status(void* workspace, size_t ws_bytes, int clear, void* stream);

/* Failure-detection self-check (no counterpart in the pages: it exercises the
   library's own error path).  Enqueues on `stream` one small kernel that
   waits on an mbarrier whose phase nothing completes, using the bounded wait
   named by `which`: 0 the single-thread wait, 1 the warp-wide wait, 2 the
   wind-down wait, 3 a warp-wide and a single-thread wait sharing one abort
   flag.  The wait expires after about one second, sets the timeout bit of the
   workspace's device flag and the kernel ends normally, so the CUDA context
   stays usable; moe_get_device_status() then reports MOE_ERR_TIMEOUT.
   Returns MOE_ERR_WORKSPACE for a missing, short (< 16 bytes) or unaligned
   workspace, MOE_ERR_INVALID_ARG for another `which`, MOE_ERR_CUDA if the
   launch fails, else MOE_OK. */
moe_status moe_check_bounded_wait(void* workspace, size_t ws_bytes, int which, void* stream);

/* Human-readable name of a status; never NULL. */
const char* moe_status_string(moe_status status);

/* Kernel launches made by this library since it was loaded (all threads). */
int64_t moe_launch_count(void);

/* Profiling.  moe_profile_enable(1) starts recording a CUDA event pair around
   every kernel this library launches (on the launching stream) and clears
   earlier records; moe_profile_enable(2) does the same for the launches that
   state the bytes they move only (the expert tier's loads), so the other
   kernels' streams get no extra events; moe_profile_enable(0) stops.  moe_profile_query()
   synchronizes on the recorded events and returns, for the named kernel, the
   number of recorded launches and their summed device time in milliseconds.
   Kernel names: router_logits_splitk, router_logits_tc, router_topk,
   plan_small, plan_mark, plan_scan, plan_place, gather_rows, scatter_rows,
   ffn_gateup_simt, ffn_down_simt, ffn_gateup_tc, ffn_down_tc,
   ffn_gateup_tc_q8, ffn_down_tc_q8, quantize_q8_0, combine, combine_partial,
   missing_pairs, load_experts (the expert tier's loads of host-resident
   experts into HBM slots).
   moe_profile_list() gives the named kernel's recorded launches one by one,
   in launch order: the first max_n durations (ms) and the bytes each launch
   moves where its launcher states them (load_experts: the experts' three
   projections; 0 otherwise); *n_out = the number of recorded launches. */
moe_status moe_profile_enable(int on);
moe_status moe_profile_query(const char* kernel, int32_t* launches, float* total_ms);
moe_status moe_profile_list(const char* kernel, int32_t max_n, float* ms, uint64_t* bytes,
                            int32_t* n_out);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
