/*
 * moe_layer.h -- C ABI of a GB300 (sm_103a) library for the forward pass of
 * one Mixture-of-Experts FFN layer during LLM serving.
 *
 * The problem, as the pages state it: token activations x [T x m], a router
 * W_r [m x E] and E experts, each a two-layer MLP x.W1.W2 with W1 of shape
 * m x p and W2 of shape p x m (HARMOEny write-up, part 3.2 "expert prefetch"),
 * or the gated three-matrix form of Mixtral / Phi-3.5-MoE experts
 * (expert-cache article, sections 1 and 5.1).  The router scores every token,
 * each token goes to its k best experts, and the weighted expert outputs are
 * gathered back in token order (HARMOEny write-up, part 1 "What is MoE" and
 * part 3.3 steps 1, 4, 5, 6).
 *
 * The forward pass runs, in order:
 *   router GEMM -> softmax + top-k (moe_route)
 *   -> per-expert histogram, exclusive scan, stable permute (moe_route)
 *   -> expert up-projection + activation -> down-projection scaled by the
 *      routing weight -> weighted un-permute and combine (moe_forward).
 *
 * Conventions shared by every entry point:
 *   - All pointers named "host" are host memory read during the call only.
 *     All other buffers are caller-owned DEVICE memory on the layer's device.
 *   - Matrices are row-major.  bf16 data is IEEE bfloat16 bit patterns.
 *   - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream.  Every call is stream-ordered and returns before the GPU work
 *     completes; nothing is synchronised on the host except where stated.
 *   - Every call validates its arguments before launching anything and
 *     returns a status; no exception crosses the ABI.  After MOE_ERR_CUDA the
 *     text of the CUDA error is available from moe_last_error().
 *   - A layer is not thread-safe: one host thread at a time per layer.
 *   - Routing problems that only the device can see (an expert id out of
 *     range or repeated within a token in moe_route_from_topk, a gather index
 *     out of range in moe_forward) never cause an out-of-bounds access: the
 *     kernel skips or clamps the access and sets a bit in the layer's device
 *     error word, which moe_layer_sync_check() reports as
 *     MOE_ERR_INVALID_ARG.
 */
#ifndef MOE_LAYER_H
#define MOE_LAYER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_layer moe_layer_t; /* opaque */
typedef struct moe_pool moe_pool_t;   /* opaque: paged expert-slot pool */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* bad pointer, size, shape or routing data   */
    MOE_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement */
    MOE_ERR_OOM = 3,          /* device or pinned-host allocation failed     */
    MOE_ERR_CUDA = 4,         /* a CUDA runtime call failed                  */
    MOE_ERR_TIMEOUT = 5,      /* a bounded host or device wait gave up       */
    MOE_ERR_INTERNAL = 6      /* library invariant broken                    */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_I8 = 2 } moe_dtype_t;

typedef enum {
    MOE_EXPERT_RELU2 = 0,  /* y = ReLU(x.W1).W2                              */
    MOE_EXPERT_SWIGLU = 1  /* y = (SiLU(x.W1) * (x.W3)).W2; W1 gate, W3 up   */
} moe_expert_t;

/* Layer configuration, fixed at create time.
 *   m: hidden size, p: expert FFN size, E: experts (1..64), k: experts per
 *   token (1..min(E, 8)), max_tokens: largest T any later call may pass.
 *   act_dtype: F32 or BF16 -- type of x, y and the router weights.
 *   weight_dtype: F32 (needs act F32), BF16 or I8 (both need act BF16).
 *     I8 means the library quantises the given bf16 weights per output
 *     column, symmetrically: scale = max|W[:,c]| / 127, code =
 *     round-half-even(W / scale) clamped to [-127, 127], in fp32.
 *   has_router_bias: 1 if b_router is given to moe_layer_create.
 *   paged: 1 to keep the expert weights in pinned host memory and serve them
 *     through a moe_pool_t (expert-cache article, sections 2.2 and 3.2). */
typedef struct {
    int m, p, E, k, max_tokens;
    moe_dtype_t act_dtype;
    moe_dtype_t weight_dtype;
    moe_expert_t expert;
    int has_router_bias;
    int paged;
} moe_config_t;

/* Routing tables: caller-owned device buffers, sized for max_tokens.
 * moe_route* fill them; moe_forward reads them.
 *   topk_ids      [T*k] int32   expert of slot j of token t at t*k + j;
 *                               slot 0 has the largest logit, ties to the
 *                               lower expert id
 *   topk_w        [T*k] fp32    softmax renormalised over the k chosen
 *   counts        [E]   int32   tokens routed to each expert; sum = T*k
 *   offsets       [E+1] int32   exclusive prefix sum of counts
 *   gather_index  [T*k] int32   flat index i = t*k + j at permuted position
 *                               pos; expert segments in expert order, flat
 *                               index ascending inside a segment
 *   scatter_index [T*k] int32   inverse: permuted position of flat index i
 *   logits        [T*E] fp32    optional (NULL to skip): the router logits
 *                               written by moe_route
 *   T                           set by moe_route* to the token count */
typedef struct {
    int32_t *topk_ids;
    float *topk_w;
    int32_t *counts;
    int32_t *offsets;
    int32_t *gather_index;
    int32_t *scatter_index;
    float *logits;
    int T;
} moe_routing_t;

/* Create a layer on the current CUDA device.
 *   w_router: host, m x E in act_dtype.  b_router: host, E fp32, or NULL.
 *   w1, w3: host arrays of E pointers to m x p matrices; w2: E pointers to
 *   p x m matrices; element type F32 if weight_dtype is F32, else BF16.
 *   w3 must be NULL for MOE_EXPERT_RELU2 and non-NULL for MOE_EXPERT_SWIGLU.
 *   The host weights are read during the call only: the library copies them
 *   to the device, transposes each matrix so that the reduction dimension is
 *   contiguous for every output (DeepSpeed-Inference article, part 3,
 *   SBI-GeMM "full cache lines"), and quantises them for I8.  The layer owns
 *   that copy and a workspace sized from max_tokens.
 *   pool: NULL unless cfg->paged; then the expert weights stay in pinned host
 *   memory owned by the layer and are brought into the pool's slots on demand.
 *   layer_id: the layer's index in the model (selects the pool set).
 * Returns MOE_ERR_INVALID_ARG for a bad shape or pointer, MOE_ERR_UNSUPPORTED
 * for an unsupported dtype/shape combination, MOE_ERR_OOM if memory runs out
 * (nothing is leaked), MOE_ERR_CUDA on a CUDA failure. */
moe_status_t moe_layer_create(const moe_config_t *cfg, const void *w_router,
                              const float *b_router, const void *const *w1,
                              const void *const *w2, const void *const *w3,
                              moe_pool_t *pool, int layer_id, moe_layer_t **out);

/* Free everything the layer owns (synchronises the device first). NULL is OK. */
moe_status_t moe_destroy(moe_layer_t *layer);

/* Router GEMM + softmax + top-k, then histogram, scan and stable permute.
 *   x: device [T x m] in act_dtype.  1 <= T <= max_tokens; T = 0 is allowed
 *   and writes counts = 0, offsets = 0.  Fills every table of `r` (logits
 *   only if r->logits is not NULL) and sets r->T. */
moe_status_t moe_route(moe_layer_t *layer, const void *x, int T, moe_routing_t *r,
                       void *stream);

/* Top-k + permute from given fp32 logits (device [T x E]); same outputs as
 * moe_route except r->logits, which is not written. */
moe_status_t moe_route_from_logits(moe_layer_t *layer, const float *logits, int T,
                                   moe_routing_t *r, void *stream);

/* Permute from a given top-k choice: ids device [T*k] int32, w device [T*k]
 * fp32.  The ids are copied into r->topk_ids and the weights into r->topk_w.
 * An id out of [0, E) is routed to expert 0 and flagged; a repeated id within
 * a token is flagged (see moe_layer_sync_check). */
moe_status_t moe_route_from_topk(moe_layer_t *layer, const int32_t *ids, const float *w,
                                 int T, moe_routing_t *r, void *stream);

/* Expert MLPs and combine: y[t] = sum_j topk_w[t,j] * expert_{ids[t,j]}(x[t]),
 * summed over ascending j in fp32 and rounded once to act_dtype.
 *   x: device [r->T x m] (the same x that was routed); y: device [r->T x m].
 *   The regime (decode: weight-streaming GEMV; batch: grouped tensor-core
 *   GEMM) is chosen on the host from T alone, so a resident layer never
 *   synchronises the host.  A paged layer copies counts to the host once to
 *   decide which experts to fetch, and the host waits for that copy: it runs
 *   on the stream of the routing call that wrote r (when r comes from this
 *   layer's last routing call; else on `stream`), and `stream` waits for it
 *   before any expert kernel.  A caller that knows the routing early can
 *   route on a side stream ahead of time, so that the wait does not also wait
 *   for the compute already queued on `stream`. */
moe_status_t moe_forward(moe_layer_t *layer, const void *x, const moe_routing_t *r,
                         void *y, void *stream);

/* Forward pass that allocates nothing and uses no layer workspace.
 * No counterpart in the source paper: this entry point exists for callers
 * that cannot call cudaMalloc while they run -- a serving engine whose own
 * allocator holds all free device memory, a latency-critical loop that cannot
 * take cudaMalloc's implicit synchronisation, code that runs where allocating
 * is not allowed.  Such a caller creates the layer up front and then calls
 * this instead of moe_forward.
 *   Same arguments, same kernels and same results as moe_forward in the decode
 *   regime, but its scratch (expert hidden rows and split-reduction partial
 *   sums) lives in a 16 MiB array compiled into the library, one per device,
 *   held until the process exits.  No cudaMalloc, cudaFree or other
 *   allocating routine is called.
 *   Limits: resident bf16/int8 layers only; T*k at most 512 and a scratch
 *   need of at most 16 MiB, where, with R = T*k and the decode plan's
 *   reduction splits S_up and S_down (moe_plan_forward, regime 1), the need is
 *     r256(2*R*p) + r256(4*S_down*R*m) + (S_up > 1 ? 2*r256(4*S_up*R*p) : 0)
 *   bytes (r256 rounds up to a multiple of 256; the last term holds the split
 *   up projection's gate and up partial sums) -- e.g. T <= 16 for a
 *   Mixtral-shaped layer.  Larger requests return MOE_ERR_INVALID_ARG with
 *   both sizes in moe_last_error().
 *   The call must be made with the layer's device current (else
 *   MOE_ERR_INVALID_ARG).  The first call on a device looks up the array's
 *   device address with that device current; make it before any stream
 *   capture begins.  The address is cached for the process: after a device
 *   reset the library has to be unloaded and loaded again.
 *   Every call on a device uses the same array: calls whose GPU work overlaps
 *   (other streams, other host threads) race on it and must be serialised.
 *   Nothing needs clearing between calls. */
moe_status_t moe_forward_static_scratch(moe_layer_t *layer, const void *x, const moe_routing_t *r,
                                        void *y, void *stream);

/* Options.
 *   MOE_OPT_REGIME: 0 = automatic (default), 1 = always the decode kernels,
 *     2 = always the batch (tensor-core) kernels.
 *   MOE_OPT_TIMING: 1 = bracket every kernel launch of this layer with a pair
 *     of CUDA events recorded on the launch stream (read with
 *     moe_layer_timings); 0 = off (default).
 *   MOE_OPT_PAIR_TILES: 1 (default) = the up projection's 256-token
 *     tensor-core tiles run on pairs of CTAs (tcgen05 cta_group::2, 256 x 256
 *     tiles over two SMs) where the shapes allow (resident bf16 layers,
 *     stored rows a multiple of 256); 0 = one CTA per 128 x 256 tile.  Both
 *     give the same results up to the order of fp32 additions inside the
 *     MMA.
 *   MOE_OPT_HOST_TIMEOUT_MS: the longest a call of this layer waits on the
 *     host for device work (the paged forward's read of the token counts and
 *     of its previous call's timing events), polling the event; past it the
 *     call returns MOE_ERR_TIMEOUT having changed no slot state, and the layer
 *     stays usable.  Milliseconds >= 0, or -1 for no limit; default 120000. */
typedef enum {
    MOE_OPT_REGIME = 1,
    MOE_OPT_TIMING = 2,
    MOE_OPT_PAIR_TILES = 3,
    MOE_OPT_HOST_TIMEOUT_MS = 4
} moe_option_t;
moe_status_t moe_layer_set_option(moe_layer_t *layer, moe_option_t opt, int value);

/* Launch plan of moe_forward for T tokens: which expert-MLP kernels run and
 * how their work is cut.  It is the same host arithmetic that moe_forward
 * performs (moe_forward takes its plan from this function), computed here
 * from the configuration alone, without a layer or a device -- for capacity
 * planning, and so that the choice can be checked off the GPU.
 *   cfg: a layer configuration (checked as moe_layer_create checks it).
 *   T: 0 <= T <= cfg->max_tokens.  num_sms: SMs of the device, >= 1 (152 on
 *   a GB300; moe_layer_info reports a layer's).  regime and pair_tiles: the
 *   values of MOE_OPT_REGIME (0, 1, 2) and MOE_OPT_PAIR_TILES (0, 1) the
 *   layer would have.
 * The decode regime runs the weight-streaming GEMV: token passes of 8, 16,
 * 24 or 32 tokens, sized to the mean count per expert plus 1.5 standard
 * deviations under uniform routing (an expert with more tokens takes further
 * passes); the batch regime runs the tcgen05 grouped GEMM with token tiles of
 * N = 16 .. 256 (int8: <= 192).
 * Automatic choice: the GEMV while ceil(T*k/E) <= 4 (bf16 weights) or <= 12
 * (int8 weights) and T*k <= 512, the tensor cores beyond, where the shapes
 * allow (2p or p, m and for int8 p multiples of 128).
 * Returns MOE_ERR_INVALID_ARG for a bad cfg, T, num_sms, regime or
 * pair_tiles; MOE_ERR_UNSUPPORTED where moe_forward would refuse the request
 * (a forced regime the shapes or T do not allow).  Pure host arithmetic. */
typedef enum {
    MOE_PATH_NONE = 0,   /* T = 0: no expert kernel runs                      */
    MOE_PATH_SIMT = 1,   /* fp32 layers: CUDA-core expert kernels             */
    MOE_PATH_GEMV = 2,   /* decode regime: weight-streaming GEMV              */
    MOE_PATH_TENSOR = 3  /* batch regime: tcgen05 grouped GEMM                */
} moe_path_t;
typedef struct {
    int path;                    /* a moe_path_t                                   */
    int mean_tokens;             /* ceil(T*k / E), the count the regime follows    */
    int tile_up, tile_down;      /* tokens per GEMV pass or per tensor-core tile   */
    int splits_up, splits_down;  /* reduction splits of each projection (1: none)  */
    int pair_up;                 /* 1: up-projection tiles on CTA pairs            */
} moe_plan_t;
moe_status_t moe_plan_forward(const moe_config_t *cfg, int T, int num_sms, int regime,
                              int pair_tiles, moe_plan_t *out);

/* Per-phase device time of the layer's kernels, from the events that
 * MOE_OPT_TIMING records.  Waits for the recorded events, sums the elapsed
 * time of every launch per phase, and (reset != 0) forgets them. */
typedef enum {
    MOE_PHASE_ROUTER = 0,   /* router GEMM + softmax + top-k (or its variants) */
    MOE_PHASE_PERMUTE = 1,  /* histogram + scan + stable scatter               */
    MOE_PHASE_GATHER = 2,   /* token rows into expert order (batch regime)     */
    MOE_PHASE_UP = 3,       /* expert up-projection + activation               */
    MOE_PHASE_UP_FINISH = 4,/* split-reduction finish of the up-projection     */
    MOE_PHASE_DOWN = 5,     /* expert down-projection x routing weight         */
    MOE_PHASE_COMBINE = 6,  /* weighted un-permute and combine                 */
    MOE_PHASE_COPY = 7,     /* paged weight copies (copy stream)               */
    MOE_NUM_PHASES = 8
} moe_phase_t;
typedef struct {
    double ms[MOE_NUM_PHASES];
    uint64_t launches[MOE_NUM_PHASES];
} moe_timings_t;
moe_status_t moe_layer_timings(moe_layer_t *layer, moe_timings_t *out, int reset);

/* Static facts about a layer.  expert_bytes: device bytes of one expert's
 * weights as stored (codes plus scales for I8).  workspace_bytes: device
 * workspace owned by the layer. */
typedef struct {
    size_t expert_bytes;
    size_t weight_bytes;
    size_t workspace_bytes;
    int decode_splits_up, decode_splits_down;
    int num_sms;
} moe_layer_info_t;
moe_status_t moe_layer_info(const moe_layer_t *layer, moe_layer_info_t *out);

/* Counters since create.  The slot and copy counters are zero for resident
 * layers. */
typedef struct {
    uint64_t kernel_launches; /* every kernel this layer launched (all calls) */
    uint64_t forwards;
    uint64_t slot_hits, slot_misses;
    uint64_t h2d_bytes;
    double h2d_ms;       /* summed duration of the copy-stream transfers   */
    double forward_ms;   /* summed duration of paged forward calls         */
    uint64_t prefetch_copies; /* experts this layer's calls prefetched for the next layer */
    uint64_t prefetch_hits;   /* lookups of this layer served by a prefetched expert      */
    uint64_t gemv_runs;       /* expert-MLP passes on the weight-streaming GEMV (decode regime) */
    uint64_t tc_runs;         /* expert-MLP passes on the tensor-core grouped GEMM (batch regime) */
} moe_stats_t;
moe_status_t moe_layer_stats(moe_layer_t *layer, moe_stats_t *out);

/* Bits of a layer's device error word (reported by moe_layer_sync_check). */
typedef enum {
    MOE_FLAG_EXPERT_ID = 1u << 0,     /* expert id outside [0, E): routed to expert 0      */
    MOE_FLAG_DUPLICATE_ID = 1u << 1,  /* the same expert twice in one token's top-k      */
    MOE_FLAG_GATHER_INDEX = 1u << 2,  /* gather index outside [0, T*k): access skipped   */
    MOE_FLAG_OFFSETS = 1u << 3,       /* offsets not monotone or out of range: clamped   */
    MOE_FLAG_WAIT_TIMEOUT = 1u << 4,  /* a bounded device wait gave up (a bug or a hang) */
    MOE_FLAG_TMEM_ALLOC = 1u << 5     /* tensor-memory allocation did not succeed        */
} moe_flag_t;

/* Wait (up to timeout_ms, polling) for the layer's last launched work, then
 * read and clear the device error word.  The wait covers everything queued on
 * the stream of the layer's last route or forward call up to this call (that
 * stream must still exist; a stream being captured into a graph is refused
 * with MOE_ERR_INVALID_ARG).  Returns MOE_ERR_TIMEOUT if the work did not
 * finish in time or a kernel's bounded wait gave up (MOE_FLAG_WAIT_TIMEOUT),
 * MOE_ERR_INVALID_ARG if a kernel flagged bad routing data (the other flags),
 * MOE_OK otherwise; the flag bits are written to *flags if flags is not NULL. */
moe_status_t moe_layer_sync_check(moe_layer_t *layer, int timeout_ms, uint32_t *flags);

/* Copy one stored expert matrix back to the host, in the user's orientation
 * (m x p for which = 1 or 3, p x m for which = 2).  For I8 layers `values`
 * receives the int8 codes and `scales` (length = number of columns) the fp32
 * per-column scales; for other layers `values` receives act-typed elements
 * and `scales` is ignored. */
moe_status_t moe_layer_read_expert(const moe_layer_t *layer, int expert, int which,
                                   void *values, float *scales);

/* ---- paged weights (expert-cache article, sections 2.2, 3.1, 3.2) --------
 * A pool is a fixed budget of device expert slots arranged as N sets
 * (indices) x M ways.  A layer with id l uses set l mod N; inside a set the
 * least recently used expert is replaced.  Misses are copied from the
 * layer's pinned host copy on a separate copy stream, one event per page,
 * and the compute stream waits for each expert's pages before its kernels.
 *
 * moe_pool_geometry: S = floor(budget_bytes / expert_bytes) slots,
 * N = floor(S / ways) sets, usable slots N * ways.  Pure host arithmetic.
 * Returns MOE_ERR_INVALID_ARG if fewer than one set fits. */
moe_status_t moe_pool_geometry(size_t budget_bytes, size_t expert_bytes, int ways,
                               int *n_index, int *usable_slots);

/* Create a pool for layers whose experts occupy expert_bytes each (see
 * moe_layer_info) on the current device: N * M slots of expert_bytes rounded
 * up to 256 plus 768 bytes of alignment room, and a copy stream.
 * page_bytes: granularity of the host-to-device copies (0 = 16 MiB; a
 * multiple of 256).  Paged layers created with this pool keep their experts
 * in pinned host memory; moe_forward on such a layer copies the routing
 * counts to the host (synchronising the caller's stream once), brings the
 * missing experts in on the copy stream, and runs each expert's kernels as
 * soon as its copy has landed, so copies overlap compute.  A slot is never
 * overwritten while a kernel may still read it.  Results are bit-identical
 * to a resident layer's.  A pool may serve many layers (set = layer_id mod N)
 * but one host thread at a time; destroy the layers before the pool.
 * Fault injection for tests: if the environment variable MOE_FAULT_COPY_FAIL
 * holds n when the pool is created, the pool's n-th page copy (0-based,
 * counting every page of every expert copy) is not issued and the forward call
 * that needed it returns MOE_ERR_CUDA; the slot it was filling is emptied, so
 * a later call copies that expert again.  No GPU operation fails. */
moe_status_t moe_pool_create(size_t budget_bytes, size_t expert_bytes, int ways,
                             size_t page_bytes, moe_pool_t **out);
moe_status_t moe_pool_destroy(moe_pool_t *pool);

/* Cross-layer prefetch (HARMOEny write-up, part 3.2; expert-cache article,
 * section 2.1: consecutive layers often pick the same experts).  With
 * max_experts > 0, every paged forward of layer l, after its own lookups,
 * copies in for layer l + 1 (when attached to this pool and mapped to a
 * different set) the max_experts experts that had the most tokens in this
 * call (ties to the lower id) and are not resident for l + 1.  Each takes an
 * empty or the least recently used way of l + 1's set.  0 (the default)
 * turns it off.  Host-only; takes effect from the next forward call. */
moe_status_t moe_pool_set_prefetch(moe_pool_t *pool, int max_experts);

/* The pool's lookups and prefetch inserts since creation, oldest first (at
 * most 2^20 kept): for entry i, the layer id, the expert, the kind -- 0 miss,
 * 1 hit, 2 prefetch insert, 3 hit on a prefetched expert not used before --
 * and the slot (set * M + way).  Any output pointer may be NULL.  *n_out
 * receives the number written (<= max).  Host-only. */
moe_status_t moe_pool_query_log(moe_pool_t *pool, int32_t *layer, int32_t *expert, int32_t *hit,
                                int32_t *slot, int max, int *n_out);

/* Status text, and the message of the last failure on this host thread. */
const char *moe_status_string(moe_status_t s);
const char *moe_last_error(void);

/* Self-test of the device-side wait limit.  Every wait in the library's
 * kernels polls its mbarrier a bounded number of times and, if the phase has
 * not completed, sets MOE_FLAG_WAIT_TIMEOUT, releases what it holds and
 * returns, so a lost signal ends as an error status instead of a hung GPU.
 * This launches one CTA whose threads wait, with that same bounded loop, on
 * an mbarrier phase that nothing completes, giving up after `polls` polls
 * (1 <= polls <= 2^24), and copies the resulting error bits to *flags (may be
 * NULL).  Synchronises `stream`.  Returns MOE_ERR_TIMEOUT when the wait gave
 * up (the expected outcome) and MOE_ERR_INTERNAL if it did not; the CUDA
 * context stays usable either way. */
moe_status_t moe_selftest_bounded_wait(uint32_t polls, uint32_t *flags, void *stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LAYER_H */
