/*
 * moe.h -- C ABI of the OEA MoE decode layer for one GB300 (sm_103a).
 *
 * The layer is the decode-time Mixture-of-Experts block described on the
 * page "Opportunistic Expert Activation (OEA)" (zhaifeiyue.github.io,
 * papers/2511.02237/detail.html):
 *   1. router scores and per-token top-k (section 2, Q1/Q2);
 *   2. optionally the OEA two-phase re-route: each token keeps its top-n_i
 *      experts, n_i = min(k0, t_i) with t_i an adaptive top-p count, the
 *      batch union S_base of those baselines is formed, and each token then
 *      adds experts from its own ranked list only if they are already in
 *      S_base, so T = |S_base| does not grow; kept scores are renormalised
 *      (section 2 Q2, section 3);
 *   3. grouping of (token, slot) pairs by expert (the per-expert loads
 *      cnt_e of the cost model, section 4);
 *   4. the expert FFN of every activated expert, each expert's weights read
 *      from HBM once (section 2 Q1, section 4 check 4), in the SwiGLU form
 *      of the Qwen3 experts the page measures:
 *      y = W_down (silu(W_gate x) * (W_up x));
 *   5. the weighted combine out_i = sum_j w_ij y_{e_ij}(x_i).
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller, 16-byte
 *     aligned, row-major and densely packed.  Buffers whose size is a
 *     multiple of B may be NULL when B == 0.  The library allocates no
 *     device memory; per-call scratch lives in the caller's workspace.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default
 *     stream).  Nothing synchronises except moe_device_status().
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns MOE_ERR_ARG and launches nothing.  Conditions only
 *     the GPU can see (a non-finite router score, a wait that timed out)
 *     set bits in a flag word in the workspace and never trap; read them
 *     with moe_device_status().
 *   - Results are deterministic: the same inputs give the same bits.
 *   - Not thread-safe per workspace: calls that share a workspace must be
 *     ordered on one stream.
 */
#ifndef OEA_MOE_H
#define OEA_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st *moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_ARG = 1,          /* invalid argument; nothing was launched       */
    MOE_ERR_CUDA = 2,         /* a CUDA runtime call failed                   */
    MOE_ERR_DEVICE_CHECK = 3, /* the GPU raised a flag (moe_device_status)    */
    MOE_ERR_WORKSPACE = 4,    /* workspace missing, misaligned or too small   */
    MOE_ERR_UNSUPPORTED = 5   /* valid but not supported on this device       */
} moe_status;

typedef enum { MOE_MODE_TOPK = 0, MOE_MODE_OEA = 1 } moe_mode;

/* Element type of hidden states, router and expert weights and output. */
typedef enum { MOE_DTYPE_BF16 = 0, MOE_DTYPE_F32 = 1 } moe_dtype;

/* Device flag bits reported by moe_device_status(). */
#define MOE_FLAG_NONFINITE_SCORE 0x1u  /* a router score was NaN or +-inf     */
#define MOE_FLAG_WAIT_TIMEOUT 0x2u     /* an in-kernel wait gave up           */
#define MOE_FLAG_BAD_INDEX 0x4u        /* an index failed its range check     */

/* Size limits. */
#define MOE_MAX_TOKENS 256
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_SLOTS 32

/*
 * Routing parameters (OEA page, section 2 Q2; sections 4-5 and 7 for maxP,
 * k^max and the padding mask).
 *   B        tokens in the batch, 0..MOE_MAX_TOKENS.
 *   B_valid  tokens 0..B_valid-1 are real; tokens B_valid..B-1 are padding
 *            and select no expert, so they cannot enlarge T (OEA page,
 *            section 7, implementation detail 1).  Negative: B.
 *   d        hidden size; a multiple of 64.
 *   N        experts, 1..MOE_MAX_EXPERTS.
 *   k        experts per token of the plain router, 1..min(N, 32).
 *   mode     MOE_MODE_TOPK or MOE_MODE_OEA.
 *   k0       OEA baseline cap, 1..k; <= 0 chooses it from the batch
 *            (section 7, implementation detail 2: piggybacking adds nothing
 *            for a single token, and smaller batches want a larger, safer
 *            k0): B_valid <= 1 routes as plain top-k (k0 = k, top-p off),
 *            2..15 real tokens take k0 = ceil(5k/8), 16 or more
 *            ceil(3k/8) -- for k = 8 the page's settings 5 and 3.
 *   p        OEA top-p threshold in (0, 1]; p >= 1 switches top-p off
 *            (t_i = N), as in the simplified router of section 5.
 *   maxP     OEA: deepest rank of the token's own list that phase 2 may
 *            take an expert from; <= 0 or >= N means N (no limit).
 *   kmax     OEA: experts per token after phase 2 (k^max); <= 0 means k;
 *            otherwise k0..min(N, 32).
 *   dtype    moe_dtype of hidden, router weights, expert weights and output.
 * Slots per token: kslots = k for MOE_MODE_TOPK, kmax for MOE_MODE_OEA
 * (moe_num_slots()).
 */
typedef struct {
    int32_t B;
    int32_t B_valid;
    int32_t d;
    int32_t N;
    int32_t k;
    int32_t mode;
    int32_t k0;
    float p;
    int32_t maxP;
    int32_t kmax;
    int32_t dtype;
} moe_route_params;

/*
 * Routing results: device buffers owned by the caller, written by
 * moe_route().  Ranks and ties: experts are ranked by score, larger first,
 * equal scores by the lower expert id.
 *   expert_idx [B][kslots] int32  chosen experts in rank order, -1 in unused
 *                                 slots (a token keeps min(kmax, T) experts
 *                                 in OEA mode; padding tokens keep none).
 *   weights    [B][kslots] fp32   renormalised scores (softmax over the kept
 *                                 scores), 0 in unused slots.
 *   T          [1] int32          number of distinct activated experts.
 *   active     [N] int32          activated experts, ascending id; entries
 *                                 T..N-1 are -1.
 *   counts     [N] int32          cnt_e, tokens routed to expert e.
 *   offsets    [N+1] int32        exclusive prefix sum of counts.
 *   perm       [B*kslots] int32   token*kslots+slot grouped by expert
 *                                 (ascending id), tokens ascending within an
 *                                 expert; entries offsets[N].. are unused.
 *   n_base     [B] int32          nullable; n_i (k in top-k mode, 0 for
 *                                 padding tokens).
 *   logits     [B][N] fp32        nullable; router scores (bias included).
 */
typedef struct {
    int32_t *expert_idx;
    float *weights;
    int32_t *T;
    int32_t *active;
    int32_t *counts;
    int32_t *offsets;
    int32_t *perm;
    int32_t *n_base;
    float *logits;
} moe_routing;

/* Slots per token for these parameters (k or kmax), or -1 if invalid. */
int32_t moe_num_slots(const moe_route_params *params);

/*
 * Kernels that one moe_decode_layer() call launches for these parameters
 * and expert FFN width on the current device, or -1 if the parameters are
 * invalid.  bf16 batches of up to 32 tokens with N <= 128 score and route
 * in one cluster launch, so a layer is two kernels.  Otherwise the router
 * and the routing are separate launches: three kernels with bf16 experts,
 * five on the fp32 path (three expert kernels).  An empty batch launches
 * only the routing kernel.
 */
int32_t moe_layer_launches(const moe_route_params *params, int32_t d_ff);

/*
 * Bytes of device workspace needed by moe_route / moe_expert_ffn /
 * moe_decode_layer for these parameters and expert FFN width d_ff (pass
 * d_ff = 0 when only moe_route is used).  Returns 0 if the parameters are
 * invalid.  The workspace must be 256-byte aligned and zero-filled once
 * before its first use; the library leaves it ready for the next call.
 */
size_t moe_workspace_bytes(const moe_route_params *params, int32_t d_ff);

/*
 * Router + routing (steps 1-3 above).
 *   hidden      [B][d]  dtype   token hidden states.
 *   w_router    [N][d]  dtype   router (gate) weights.
 *   router_bias [N]     fp32    nullable; added to every score.
 *   routing                     outputs, see moe_routing.
 * Scores are accumulated in fp32.  Routing decisions compare those fp32
 * scores exactly; the top-p prefix is computed in fp32.
 */
moe_status moe_route(const void *hidden, const void *w_router, const float *router_bias,
                     const moe_route_params *params, const moe_routing *routing,
                     void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * Expert FFN + weighted combine (steps 4-5) for a batch routed by
 * moe_route() with the same params and the same workspace: besides the
 * routing outputs it reads the per-pair positions, per-expert records and
 * per-(token, 128 rows of d) combine counters that moe_route left in the
 * workspace, so no other call may use that workspace in between.  A
 * completed call leaves them as it found them, so it may be repeated on the
 * same routing.  Reads only activated experts, each expert's three
 * matrices once from HBM.  With OEA routing of up to 64 tokens, the call
 * starts on the activated experts' weights as soon as the preceding
 * moe_route() on this workspace and stream has fixed them (its phase 1),
 * before that routing call's kernel ends; it recognises that call's
 * published set by a per-call tag the library keeps for the workspace.
 *   hidden  [B][d]        dtype  the hidden states given to moe_route.
 *   w_gate  [N][d_ff][d]  dtype  expert gate projections.
 *   w_up    [N][d_ff][d]  dtype  expert up projections.  bf16: where w_gate
 *           and w_up are distinct and less than 2^40 bytes apart (two halves
 *           of one allocation always are), one tensor map reads both and a
 *           pipeline stage of an expert tile is a single copy; otherwise
 *           (for instance separate allocations in distant address ranges)
 *           each stage takes 16 smaller copies, and such tiles run about
 *           20 % slower.  Results are the same.
 *   w_down  [N][d][d_ff]  dtype  expert down projections.
 *   d_ff    expert FFN width, a multiple of 64.
 *   routing the results of moe_route (expert_idx, weights, T, active,
 *           counts, offsets, perm are read).
 *   out     [B][d]        dtype  written; padding tokens get zeros.
 * bf16: products in fp32 on tensor cores, the SwiGLU activation h rounded
 * to bf16 before the down projection, sums in fp32, output rounded once.
 * fp32: all arithmetic in fp32 on CUDA cores.
 */
moe_status moe_expert_ffn(const void *hidden, const void *w_gate, const void *w_up,
                          const void *w_down, int32_t d_ff, const moe_route_params *params,
                          const moe_routing *routing, void *out, void *workspace,
                          size_t workspace_bytes, moe_stream_t stream);

/*
 * Mixed-precision experts (DynaExq page, section 3.2: frequently used experts
 * in high precision, the others in a 4-bit version).  Hot experts keep bf16
 * weights in w_gate / w_up / w_down (laid out as for moe_expert_ffn, with
 * n_hot experts); cold experts are INT4 with one bf16 scale per row and
 * 128-column group of the contraction dimension (d for W_gate / W_up, d_ff
 * for W_down): w = q * s, q in -7..7.  An INT4 expert is
 * 3 * (d * d_ff / 2 + d * d_ff / 64) bytes (moe_pack_int4 makes images).
 *   slot    [N] int32, device: for expert e, slot[e] >= 0 is its index among
 *           the bf16 experts, slot[e] < 0 means INT4 expert -1 - slot[e].
 *           An out-of-range slot raises MOE_FLAG_BAD_INDEX.
 *   q_gate, q_up  [n_cold] packed images of the [d_ff][d] matrices,
 *   q_down        [n_cold] packed images of the [d][d_ff] matrices.
 * Packed image of a matrix [rows][cols] with chunk height rb (64 for W_gate
 * and W_up, 128 for W_down): chunks of rb rows x 128 columns (one scale
 * group) in row-block-major, column-group order; a chunk is rb*64 bytes of
 * codes then rb bf16 scales (one per row: the row's scale of the group).
 * In a chunk row, local column c is the 4-bit field at bit
 * 4*((c%8)/2) + 16*(c%2) of little-endian 32-bit word c/8 of the row's 64
 * bytes, holding q + 8.
 * Requirements: dtype bf16, d and d_ff multiples of 128, n_hot >= 1,
 * 16-byte aligned images.  Results as moe_expert_ffn; each INT4 weight is
 * decoded to q exactly and multiplied by its group scale with one rounding
 * to bf16 before the tensor-core products (fp32 accumulation).
 */
typedef struct {
    const int32_t *slot;
    const void *q_gate;
    const void *q_up;
    const void *q_down;
    int32_t n_hot;
    int32_t n_cold;
} moe_mixed_experts;

moe_status moe_expert_ffn_mixed(const void *hidden, const void *w_gate, const void *w_up, const void *w_down,
                                const moe_mixed_experts *mixed, int32_t d_ff, const moe_route_params *params,
                                const moe_routing *routing, void *out, void *workspace, size_t workspace_bytes,
                                moe_stream_t stream);

/*
 * Makes the packed INT4 image of one bf16 matrix on the device: the 4-bit
 * version of an expert matrix that moe_expert_ffn_mixed reads (DynaExq
 * page, section 3.2, INT4 tier; section 2.4: a new version is prepared
 * off the request path and only then published, here by writing the
 * expert's slot).  Per row and 128-column group:
 *   s = max|w| / 7, the quotient taken in double and rounded to nearest
 *       even, first to fp32, then to bf16;
 *   q = rint(w / s) in double (ties to even), clamped to -7..7; q = 0
 *       where s = 0.
 *   w     [rows][cols] bf16, device, 16-byte aligned.
 *   rows  a multiple of rb.  cols: a multiple of 128.
 *   rb    chunk height of the image: 64 for W_gate / W_up, 128 for W_down
 *         (any multiple of 8 is accepted).
 *   out   rows*cols/2 + rows*(cols/128)*2 bytes, device, 16-byte aligned.
 * Asynchronous on `stream`; allocates nothing.
 */
moe_status moe_pack_int4(const void *w, int32_t rows, int32_t cols, int32_t rb, void *out, moe_stream_t stream);

/*
 * The whole layer with mixed-precision experts in one call: moe_route, then
 * moe_expert_ffn_mixed, on the same stream and workspace.  `mixed` is the
 * per-expert descriptor of the DynaExq page's stable expert handles
 * (section 2.2; section 3.2 for the precision tiers): for every expert id,
 * its slot says where its current version lives -- a bf16 expert of
 * w_gate / w_up / w_down, or a packed INT4 image -- so the kernels resolve
 * each activated expert through the table and a caller switches an
 * expert's version by rewriting its slot (and image) between calls.
 * Arguments, layouts and results as moe_route and moe_expert_ffn_mixed;
 * every argument, the descriptor included, is checked before anything is
 * launched.  With OEA routing of up to 64 tokens the expert kernel starts
 * on the activated experts before the routing kernel ends, as for
 * moe_expert_ffn.
 */
moe_status moe_decode_layer_mixed(const void *hidden, const void *w_router, const float *router_bias,
                                  const void *w_gate, const void *w_up, const void *w_down,
                                  const moe_mixed_experts *mixed, int32_t d_ff,
                                  const moe_route_params *params, const moe_routing *routing, void *out,
                                  void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * Expert residency at run time (DynaExq page, sections 2.2-2.5 and 3.2-3.5):
 * which experts of one layer keep their bf16 version, decided from the
 * routing as the layer runs, and changed without stopping it.
 *   - Handles: `slot` is the table moe_expert_ffn_mixed / moe_decode_layer_mixed
 *     read (pass it as moe_mixed_experts.slot with n_hot = n_hot, n_cold = N
 *     and INT4 images of all N experts, image i = expert i).  The kernels
 *     resolve every activated expert through it at every call.
 *   - Pools: the caller's bf16 pool of n_hot slots (fixed budget) and INT4
 *     images of all experts, which stay resident as the version every handle
 *     can fall back to.
 *   - Hotness (section 2.5): moe_residency_observe adds a call's per-expert
 *     counts (moe_routing.counts) on the device; every update_every calls the
 *     interval's counts c are copied to `snapshot` (pinned host memory) and
 *     cleared, without waiting; when they have arrived,
 *     S_e <- alpha S_e + (1 - alpha) c_e (S starts at 0).
 *   - Selection with hysteresis (section 3.5): while the best expert outside
 *     the bf16 set (highest S, ties to the lower id) scores more than
 *     `margin` above the weakest member (lowest S, ties to the higher id),
 *     the two swap places (moe_residency_select).  A selection runs only
 *     when no transition is pending.
 *   - Transitions (sections 2.4, 3.4): a demotion redirects the handle to
 *     the INT4 image on the caller's stream, then the freed slot receives
 *     the promoted expert's bf16 weights: an asynchronous copy from the
 *     caller's pinned host memory on the residency's own migration stream,
 *     which waits for the redirect.  The handle is pointed at the new slot
 *     only after that copy's completion event has been seen (by a later
 *     observe or flush), so no kernel reads a partly copied version; until
 *     then the expert runs in INT4.  At most max_inflight copies are in
 *     flight; further swaps wait in a queue.
 * The library allocates no device memory for this: the accumulator and the
 * snapshot are the caller's.  Not thread-safe; calls on one residency must
 * use one stream.
 * Reading of the page: the update interval is counted in routing calls
 * (the page uses a time interval); the INT4 images of all experts stay on
 * the device, so a demotion moves no data.
 */
typedef struct {
    int32_t N;             /* experts, 2..MOE_MAX_EXPERTS                          */
    int32_t n_hot;         /* bf16 slots (the budget), 1..N-1                      */
    int32_t d, d_ff;       /* multiples of 128                                     */
    double alpha;          /* weight of the old score, 0 <= alpha < 1              */
    double margin;         /* hysteresis margin, in selections per interval, >= 0 */
    int32_t update_every;  /* routing calls per update interval, >= 1             */
    int32_t max_inflight;  /* promotion copies in flight at once, >= 1            */
    int32_t *slot;         /* [N] device: the handle table                         */
    uint32_t *counts_acc;  /* [N] device: counts of the current interval           */
    uint32_t *snapshot;    /* [N] pinned host: counts of the last interval         */
    void *hot_gate;        /* device bf16 pool: [n_hot][d_ff][d]                   */
    void *hot_up;          /*                   [n_hot][d_ff][d]                   */
    void *hot_down;        /*                   [n_hot][d][d_ff]                   */
    const void *host_gate; /* pinned host bf16 weights of all experts: [N][d_ff][d] */
    const void *host_up;   /*                                          [N][d_ff][d] */
    const void *host_down; /*                                          [N][d][d_ff] */
} moe_residency_config;

typedef struct moe_residency moe_residency;

/* Residency states reported by moe_residency_query. */
#define MOE_RESIDENT_LO 0
#define MOE_RESIDENT_HI 1
#define MOE_PROMOTING 2

/*
 * Creates a residency whose bf16 set starts as initial_hot[n_hot] (expert
 * initial_hot[k] in slot k; the caller has filled the pool accordingly).
 * Writes the handle table and clears the accumulator on `stream` and waits
 * for them.
 */
moe_status moe_residency_create(const moe_residency_config *cfg, const int32_t *initial_hot,
                                moe_residency **out, moe_stream_t stream);

/* After a routing call on `stream`: adds its counts[N] (device), publishes
 * completed promotions, updates the scores when a snapshot has arrived,
 * selects and issues transitions.  Never waits for the GPU. */
moe_status moe_residency_observe(moe_residency *r, const int32_t *counts, moe_stream_t stream);

/* Waits for every queued and in-flight transition and publishes it. */
moe_status moe_residency_flush(moe_residency *r, moe_stream_t stream);

/* Host copies of the per-expert state (MOE_RESIDENT_*, nullable [N]), the
 * scores S (nullable [N]) and, in stats[5] (nullable): routing calls seen,
 * score updates, promotions, demotions, transitions queued or in flight. */
moe_status moe_residency_query(const moe_residency *r, int32_t *state, double *scores, uint64_t *stats);

moe_status moe_residency_destroy(moe_residency *r);

/*
 * The selection step alone, on the host: in_hot[N] (0/1) is updated in
 * place and the swaps are written to promote / demote (nullable, [N]) in
 * the order they are made.  Returns their number, or -1 for bad arguments.
 */
int32_t moe_residency_select(const double *S, int32_t N, double margin, uint8_t *in_hot, int32_t *promote,
                             int32_t *demote);

/* moe_route followed by moe_expert_ffn on the same stream. */
moe_status moe_decode_layer(const void *hidden, const void *w_router, const float *router_bias,
                            const void *w_gate, const void *w_up, const void *w_down,
                            int32_t d_ff, const moe_route_params *params,
                            const moe_routing *routing, void *out, void *workspace,
                            size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_decode_layer for callers that cannot allocate device memory.  The
 * pages have no counterpart: this is a property of the library, not of the
 * method.  A plugin whose host engine owns all device memory, a runtime
 * that freezes allocation after start-up, or code without access to its
 * framework's allocator may have no way to provide a workspace.  This call
 * takes its scratch from one fixed array in the library's own device memory
 * (MOE_STATIC_SCRATCH_BYTES, held by every GPU that loads the library until
 * the process exits) and allocates nothing.  Inputs, routing buffers and
 * output are the caller's, exactly as for moe_decode_layer.
 *   - A batch whose workspace (moe_workspace_bytes) exceeds
 *     MOE_STATIC_SCRATCH_BYTES is rejected with MOE_ERR_WORKSPACE before
 *     anything is launched.
 *   - Every call looks up the array's device address on the current device
 *     (no allocation).  The first call on a device may load the library's
 *     device code, so make it before any stream capture.  After a reset of
 *     the device (cudaDeviceReset, or the primary context torn down and
 *     recreated) the next call finds the array again, zeroed.
 *   - All calls on a device share its array, which keeps the last call's
 *     contents; the counters at its front are cleared on `stream` at every
 *     call.  Calls that overlap on the GPU (for example on two streams) race
 *     with each other: serialise them.
 *   - Device flags raised by these calls accumulate in the array until
 *     moe_device_status_static() reads and clears them.
 */
#define MOE_STATIC_SCRATCH_BYTES (32u << 20)
moe_status moe_decode_layer_static(const void *hidden, const void *w_router, const float *router_bias,
                                   const void *w_gate, const void *w_up, const void *w_down,
                                   int32_t d_ff, const moe_route_params *params,
                                   const moe_routing *routing, void *out, moe_stream_t stream);

/*
 * moe_device_status for moe_decode_layer_static: synchronises `stream`,
 * returns the device flag word (MOE_FLAG_*) that calls of
 * moe_decode_layer_static raised on the current device since the last
 * read, and clears it.  Returns MOE_ERR_DEVICE_CHECK if any flag was set.
 * Allocates nothing.  (No counterpart on the pages.)
 */
moe_status moe_device_status_static(moe_stream_t stream, uint32_t *flags);

/*
 * Synchronises `stream`, returns the device flag word (MOE_FLAG_*) that the
 * calls on this workspace raised since the last read, and clears it.
 * Returns MOE_ERR_DEVICE_CHECK if any flag was set.
 */
moe_status moe_device_status(void *workspace, moe_stream_t stream, uint32_t *flags);

/*
 * Bound, in microseconds, of every wait inside the library's kernels: the
 * expert kernel's CTAs wait for one another (hidden states copied, h rows
 * written, y slices stored) and, with the early start, for the routing
 * kernel's published union.  A healthy layer's waits last microseconds.  A
 * wait that reaches the bound gives up: the kernel raises
 * MOE_FLAG_WAIT_TIMEOUT, every later wait in the same CTA returns at once,
 * the call's output is not valid, and the kernel still ends and leaves the
 * workspace ready for the next call.  Default 2,000,000 (two seconds);
 * 0 restores it.  The bound is counted in SM clock cycles at 2,000 per
 * microsecond (the clock runs at up to 2.07 GHz), so it lasts at least
 * about the given time.  Applies to calls launched afterwards, process
 * wide.  Short bounds are for tests of the failure path: a layer whose CTA
 * is delayed for longer than the bound (for example by a long kernel on
 * another stream occupying its SM) would fail with the flag.
 * (No counterpart on the pages.)
 */
moe_status moe_set_wait_timeout_us(uint32_t microseconds);

/*
 * Seeded synthetic tensor fill (for benchmarks and tests; not part of the
 * layer).  Writes elements start..start+n-1 of the counter-based stream:
 * SplitMix64 (Steele, Lea & Flood, OOPSLA 2014) output i for initial state
 * `seed`, its four 16-bit fields summed and centred (an Irwin-Hall sum),
 * times `scale` in fp32, rounded to bf16 (nearest even) when dtype is bf16.
 * dst must hold n elements of dtype.
 */
moe_status moe_synth_normal(void *dst, int32_t dtype, uint64_t n, uint64_t start, uint64_t seed,
                            float scale, moe_stream_t stream);

/* Human-readable name of a status, and the last error detail on this thread. */
const char *moe_status_string(moe_status status);
const char *moe_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* OEA_MOE_H */
