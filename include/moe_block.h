/*
 * moe_block.h -- C ABI of the block-coreset sparse mixture-of-experts FFN
 * (libmoeblock.so, CUDA, sm_103a).
 *
 * The layer, as the source pages state it:
 *   - model card "Clover-35B-A3B-Preview -- CMF", intro: an MoE with 256
 *     experts, top-8, plus one shared expert, evaluated on every denoising
 *     pass over a block of 32 rows;
 *   - same page, Usage: the block's experts are restricted to the set that
 *     carries 90% of its routing; block size 8, 16 or 32;
 *   - InfiniLM PR #604 (Clover on Hygon DCUs), Summary and Notes: preview
 *     passes route through the block coreset, the commit pass replays the
 *     full route (coreset disabled).
 * The pages give no API; the three calls below follow that statement of the
 * problem: route every row, restrict each block to its coreset, evaluate the
 * experts and the shared expert.
 *
 * Conventions for every call:
 *   - Pointers named x, y, w_*, topk_*, keep, core_size, block_offsets,
 *     workspace ... are DEVICE pointers owned by the caller; the library
 *     allocates no device memory and keeps no pointer beyond the call, except
 *     the weight pointers given to moe_plan_create (kept for the plan's life).
 *   - bf16 tensors are row-major with the last dimension contiguous.
 *   - Every call validates its arguments on the host first; on error it
 *     returns a negative moe_status, launches nothing, and moe_last_error()
 *     returns a message (thread-local).  On success the work is enqueued on
 *     `stream` and the call returns without synchronising; nothing is copied
 *     back to the host.
 *   - Anomalies that only the device can see (an expert id out of range,
 *     non-finite logits, block offsets that are not monotone, a row whose
 *     coreset weights are all zero, a pipeline wait that gave up) are counted
 *     in a status word inside the workspace; read it with
 *     moe_read_device_status().  No kernel traps.
 *   - Calls on one stream with one workspace are ordered; calls that share a
 *     workspace must not run concurrently on different streams.
 */
#ifndef MOE_BLOCK_H
#define MOE_BLOCK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (NULL = the legacy default stream). */
typedef struct CUstream_st* moe_stream_t;

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,  /* null/misaligned pointer, bad size or value */
    MOE_ERR_UNSUPPORTED = -2,  /* shape outside what the kernels implement */
    MOE_ERR_WORKSPACE = -3,    /* workspace too small or misaligned */
    MOE_ERR_CUDA = -4          /* a CUDA runtime or driver call failed */
} moe_status;

/* Layer shape and the largest call the workspace must hold.
 *   H   hidden size; multiple of 256 (the router's summation stripes)
 *   E   routed experts; 1..1024
 *   k   experts per row; 1..32 and <= E
 *   I   routed-expert intermediate size; multiple of 64
 *   Is  shared-expert intermediate size; multiple of 64
 *   max_rows    largest R of any call (1 .. 2^21)
 *   max_blocks  largest nb of any call (>= 1) */
typedef struct moe_dims {
    int32_t H, E, k, I, Is;
    int32_t max_rows, max_blocks;
} moe_dims;

/* Opaque host object: the shape, the weight pointers and their TMA tensor maps. */
typedef struct moe_plan moe_plan;

/* Device status word (uint32 counters), see moe_read_device_status. */
enum {
    MOE_STATUS_NONFINITE_LOGITS = 0,  /* logits that were NaN or +-inf */
    MOE_STATUS_BAD_EXPERT_ID = 1,     /* top-k ids outside [0, E) (skipped) */
    MOE_STATUS_BAD_OFFSETS = 2,       /* blocks with offsets out of order/range */
    MOE_STATUS_EMPTY_ROWS = 3,        /* rows left with only the shared expert */
    MOE_STATUS_WAIT_TIMEOUT = 4,      /* GEMM pipeline waits that gave up */
    MOE_STATUS_NONFINITE_OUTPUT = 5,  /* 256-column pieces of y with a non-finite value */
    MOE_STATUS_BAD_UNIT = 6,          /* GEMM work units found invalid and skipped: the
                                         workspace was overwritten during the call (e.g.
                                         by work on another stream not ordered before it) */
    MOE_STATUS_WORDS = 8
};

/* Bytes of device workspace needed for calls up to `dims`; 0 on invalid dims.
 * The workspace must be 256-byte aligned.  Its status counters are whatever
 * the memory held: zero them once (moe_clear_device_status or a memset)
 * before reading them. */
size_t moe_workspace_bytes(const moe_dims* dims);

/* Create a plan.  Weights (device, bf16, row-major, 16-byte aligned):
 *   w_router [E, H]   router (one row per expert)
 *   w_gate   [E, I, H], w_up [E, I, H], w_down [E, H, I]   routed experts
 *   ws_gate  [Is, H],   ws_up [Is, H],   ws_down [H, Is]     shared expert
 * Expert e computes  W_down[e] (silu(W_gate[e] x) * (W_up[e] x)).
 * Must be called with the device that owns the weights current.  On success
 * *out receives a plan that the caller frees with moe_plan_destroy. */
moe_status moe_plan_create(const moe_dims* dims, const void* w_router, const void* w_gate,
                           const void* w_up, const void* w_down, const void* ws_gate,
                           const void* ws_up, const void* ws_down, moe_plan** out);

void moe_plan_destroy(moe_plan* plan);

/* Quantised expert weights (model card "Clover-35B-A3B-Preview -- CMF",
 * Files: the 8-bit and 4-bit expert files; the page gives no codec).  Along
 * each weight row's input dimension, blocks of 32 weights share one bf16 scale
 * d; a weight is stored as a signed integer q and stands for q * d rounded
 * once to bf16 (round to nearest, ties to even).  bits == 8: q is int8;
 * bits == 4: q is a 4-bit two's-complement nibble, two per byte, the even
 * element in the low nibble, so the last dimension below is halved (in bytes).
 * Scales are bf16, block-major: d[block][row] (the scales of consecutive rows
 * of one block of 32 are contiguous).  The gate and up matrices of an expert
 * are one tensor (codes, and scales), their rows interleaved in groups of 64:
 * rows 128 j .. 128 j + 63 are gate rows 64 j .. 64 j + 63 and rows
 * 128 j + 64 .. 128 j + 127 the up rows of the same indices (so I and Is are
 * multiples of 64); one 128-row tile is then the gate and up rows a GEMM stage
 * needs.  Device pointers, 16-byte aligned:
 *   gate_up         [E, 2I, H]   codes       gate_up_scale           [E, H/32, 2I]
 *   down            [E, H, I]    codes       down_scale              [E, I/32, H]
 *   shared_gate_up  [2Is, H]     codes       shared_gate_up_scale    [H/32, 2Is]
 *   shared_down     [H, Is]      codes       shared_down_scale       [Is/32, H]
 * The router stays bf16. */
typedef struct moe_quant_weights {
    int32_t bits;
    const void *gate_up, *down, *gate_up_scale, *down_scale;
    const void *shared_gate_up, *shared_down, *shared_gate_up_scale, *shared_down_scale;
} moe_quant_weights;

/* Create a plan whose routed and shared experts are quantised (see
 * moe_quant_weights); w_router is bf16 [E, H] as for moe_plan_create.  Every
 * call works on such a plan as on a bf16 one: the routing is the same, and
 * the expert GEMMs read the codes and scales (half or a quarter of the bf16
 * bytes) and turn them into bf16 weights in shared memory before the tensor
 * cores use them.  All call sizes run the streaming kernels (units of 32
 * rows).  Errors: MOE_ERR_UNSUPPORTED for bits other than 8 or 4, or I or Is
 * not a multiple of 64; otherwise as moe_plan_create. */
moe_status moe_plan_create_quantized(const moe_dims* dims, const void* w_router,
                                     const moe_quant_weights* qw, moe_plan** out);

/* Router: logits, top-k and weights for every row.
 * (Model card, intro: "256 experts top-8".)
 *   x             [R, H] bf16 rows; R <= max_rows
 *   block_offsets [nb + 1] int32: block b holds rows block_offsets[b] ..
 *                 block_offsets[b+1]-1; 0 = first <= ... <= last = R
 *   logit_bias    [nb, E] fp32 added to row r's logits for r in block b, or NULL
 *   topk_idx      [R, k] int32 out: experts by (logit desc, id asc)
 *   topk_w        [R, k] fp32 out: softmax over the k selected logits
 * Logits are fp32 sums of exact bf16 products in a fixed order (stripes of 256
 * along H; lane p of 32 owns elements 8p..8p+7 of each stripe and adds them in
 * ascending H; the 32 partial sums combine by an xor butterfly), so top-k ids
 * are reproducible bit for bit.  NaN logits rank last (counted). */
moe_status moe_block_route(const moe_plan* plan, const void* x, int32_t R,
                           const int32_t* block_offsets, int32_t nb, const float* logit_bias,
                           int32_t* topk_idx, float* topk_w, void* workspace,
                           size_t workspace_bytes, moe_stream_t stream);

/* Router with the probability mass (the other reading of the coreset's mass).
 * (InfiniLM PR #604, Summary: preview passes use "block coreset routing";
 * model card, Usage: "90% of its routing".  The pages do not say whether a
 * slot's mass is its renormalised top-k weight or its probability under the
 * softmax over all experts; moe_block_route serves the first reading, this
 * call the second.)
 * As moe_block_route, and in addition
 *   topk_p  [R, k] fp32 out (device): p_j = a_j / D, the selected experts'
 *           probabilities under the softmax over all E experts, with
 *           a_j = exp_c(z_j - z_0) as for topk_w and D = sum over every expert e
 *           of exp_c(z_e - z_0) in a fixed order (lane p of 32 adds the experts
 *           p, p + 32, ... in ascending e; the 32 lane sums combine by the xor
 *           butterfly of the logits), then one IEEE division.
 * topk_idx and topk_w are bit-identical to moe_block_route's.  D needs the exact
 * logit of every expert, so calls of >= 256 rows take the fixed-order router
 * for all experts instead of the tensor-core screen (slower, same ids).
 * topk_p NULL: this is moe_block_route.  Errors as moe_block_route. */
moe_status moe_block_route_probs(const moe_plan* plan, const void* x, int32_t R,
                                 const int32_t* block_offsets, int32_t nb, const float* logit_bias,
                                 int32_t* topk_idx, float* topk_w, float* topk_p, void* workspace,
                                 size_t workspace_bytes, moe_stream_t stream);

/* Block coreset and renormalisation.
 * (Model card, Usage: the block's experts restricted to the set carrying 90% of
 * its routing; InfiniLM PR #604, Notes: full-route replay = coreset disabled.)
 * Per block: mass q = floor(w * 2^32) per (row, slot) as exact integers,
 * Q_e = sum over the block's rows; theta = ceil(tau * sum_e Q_e) exactly;
 * experts ordered by (Q desc, id asc); the coreset is the shortest prefix whose
 * mass reaches theta.  tau >= 1 (or +inf) disables the coreset: every touched
 * expert is kept and w_renorm = topk_w bit for bit.  Otherwise each row's
 * surviving weights are divided by their sum (fp32, rank order); dropped slots
 * get 0; a row with no surviving weight keeps only the shared expert.
 *   tau        (0, inf]; NaN or <= 0 is rejected
 *   keep       [nb, ceil(E/32)] uint32 out: bit e of block b = expert e kept
 *   core_size  [nb] int32 out: coreset size
 *   w_renorm   [R, k] fp32 out
 *   n_empty    [nb] int32 out (or NULL): rows left with only the shared expert */
moe_status moe_block_coreset(const moe_plan* plan, int32_t R, const int32_t* block_offsets,
                             int32_t nb, const int32_t* topk_idx, const float* topk_w,
                             float tau, uint32_t* keep, int32_t* core_size, float* w_renorm,
                             int32_t* n_empty, void* workspace, size_t workspace_bytes,
                             moe_stream_t stream);

/* Block coreset under an expert budget.
 * (InfiniLM PR #604, Summary: preview passes use block coreset routing with an
 * "expert-budget"; the pages name the budget without defining it.  Reading:
 * a cap on the number of experts a block keeps.)
 * As moe_block_coreset, and then at most max_experts experts per block are
 * kept: the first ones of the same (Q desc, id asc) order.  With tau >= 1 the
 * budget applies to the touched experts.  The rows keep topk_w bit for bit
 * only when tau >= 1 and the budget drops nothing; otherwise they are
 * renormalised as above.
 *   max_experts  >= 1: the cap; 0: no cap (= moe_block_coreset); < 0 rejected */
moe_status moe_block_coreset_budget(const moe_plan* plan, int32_t R, const int32_t* block_offsets,
                                    int32_t nb, const int32_t* topk_idx, const float* topk_w,
                                    float tau, int32_t max_experts, uint32_t* keep,
                                    int32_t* core_size, float* w_renorm, int32_t* n_empty,
                                    void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* Block coreset with the slots' masses given apart from the weights.
 * (InfiniLM PR #604, Summary; model card, Usage: the mass "90% of its routing"
 * is read either as the renormalised weights -- moe_block_coreset -- or as the
 * probabilities under the full softmax -- topk_mass = the topk_p of
 * moe_block_route_probs.)
 * As moe_block_coreset_budget, with q = floor(topk_mass * 2^32) per (row, slot)
 * in place of floor(topk_w * 2^32); a mass outside [0, 1] (or NaN) counts as 0.
 * The renormalisation still divides topk_w (w_renorm is the same function of
 * topk_w and the kept set); tau >= 1 with nothing dropped keeps topk_w bit for
 * bit.
 *   topk_mass  [R, k] fp32 (device), or NULL: the masses are topk_w
 * Other arguments, outputs and errors: moe_block_coreset_budget. */
moe_status moe_block_coreset_mass(const moe_plan* plan, int32_t R, const int32_t* block_offsets,
                                  int32_t nb, const int32_t* topk_idx, const float* topk_w,
                                  const float* topk_mass, float tau, int32_t max_experts,
                                  uint32_t* keep, int32_t* core_size, float* w_renorm,
                                  int32_t* n_empty, void* workspace, size_t workspace_bytes,
                                  moe_stream_t stream);

/* Expert evaluation and combine.
 * (Model card, intro: top-8 experts plus a shared expert.)
 *   y[r] = S(x[r]) + sum over slots j of row r whose expert is kept for r's
 *          block of w_renorm[r, j] * E_{topk_idx[r, j]}(x[r])
 * with S the shared expert.  bf16 MMA with fp32 accumulation; a routed pair's
 * SwiGLU activations enter the down projection in bf16, the shared expert's
 * as two bf16 parts (hi + lo, about 16 significant bits: its output enters
 * every row with weight 1); each expert's weighted output and the shared output are
 * staged in fp16 (|value| < 65504) and summed in fp32 per row in a fixed order
 * (shared expert, then the row's slots in rank order), so y is reproducible.
 *   y      [R, H] bf16 out
 *   y_f32  [R, H] fp32 out (the sum before the bf16 rounding), or NULL
 * Each touched expert's weights are streamed from HBM once per call. */
moe_status moe_block_forward(const moe_plan* plan, const void* x, int32_t R,
                             const int32_t* block_offsets, int32_t nb, const int32_t* topk_idx,
                             const float* w_renorm, const uint32_t* keep, void* y, float* y_f32,
                             void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* One denoising pass of the layer: route, coreset and forward in one call.
 * (Model card, Hardware: every pass as one GPU submission; intro and Usage for
 * the three steps.)
 * Does what moe_block_route_probs, moe_block_coreset_mass and
 * moe_block_forward do in sequence, with the same arguments, outputs and
 * errors (topk_p NULL: the weight mass; non-NULL: the probability mass, and
 * topk_p is written), bit for bit the same results, with one validation and
 * the kernels enqueued back to back (programmatic dependent launch between
 * them, no host synchronisation).  All outputs (topk_idx, topk_w, topk_p,
 * keep, core_size, w_renorm, n_empty, y, y_f32) are written as by those
 * calls. */
moe_status moe_block_pass(const moe_plan* plan, const void* x, int32_t R,
                          const int32_t* block_offsets, int32_t nb, const float* logit_bias,
                          float tau, int32_t max_experts, int32_t* topk_idx, float* topk_w,
                          float* topk_p, uint32_t* keep, int32_t* core_size, float* w_renorm,
                          int32_t* n_empty, void* y, float* y_f32, void* workspace,
                          size_t workspace_bytes, moe_stream_t stream);

/* Live-row reuse (InfiniLM pull 604 "Clover MoE": Summary, Motivation and the
 * benchmark table's "expert budget/live reuse" rows).  The pages name live-row
 * reuse with a refresh interval of five passes and define neither the live
 * set nor the reuse; the reading taken here: between refreshes, a denoising
 * pass recomputes the MoE output of the rows still live (positions not yet
 * resolved) and keeps the cached output of the others.  The refresh policy
 * (a full moe_block_forward every fifth pass) belongs to the caller.
 *   live  [R] uint8 device: row r is evaluated iff live[r] != 0; NULL = every
 *         row (then this is moe_block_forward).
 * For a live row r, y[r] (and y_f32[r]) is what moe_block_forward writes, bit
 * for bit, given the same keep mask.  For a dead row, y[r] and y_f32[r] are
 * not written: they hold whatever the caller left there (the cached output).
 * Dead rows contribute no (row, expert) pair and are not fed to the shared
 * expert, so a pass with few live rows streams only the experts their pairs
 * touch (plus the shared expert).  keep is not recomputed: pass the coreset
 * the caller wants (e.g. one computed over the live rows only).  Other
 * arguments, errors and the workspace are those of moe_block_forward. */
moe_status moe_block_forward_live(const moe_plan* plan, const void* x, int32_t R,
                                  const int32_t* block_offsets, int32_t nb,
                                  const int32_t* topk_idx, const float* w_renorm,
                                  const uint32_t* keep, const uint8_t* live, void* y,
                                  float* y_f32, void* workspace, size_t workspace_bytes,
                                  moe_stream_t stream);

/* Router for callers that cannot allocate device memory (no counterpart on the
 * pages: an addition for deployment).  Some callers cannot hand the library a
 * workspace, e.g. an engine that reserves all of its device memory up front,
 * or a plugin allowed to touch only the buffers it is given.  This call does
 * what moe_block_route does, with bit-identical outputs, through the
 * fixed-order (SIMT) router (never the tensor-core screen that
 * moe_block_route takes from 256 rows on, so it is slower there), and
 * keeps the router's scratch (logits and tickets) in a 1 MiB array
 * compiled into the library, which every GPU that loads the library holds
 * until the library is unloaded.  The caller still passes x, block_offsets,
 * logit_bias, topk_idx and topk_w as for moe_block_route.
 *   - Allocates nothing and calls no allocating routine.
 *   - Rejects with MOE_ERR_UNSUPPORTED any call whose scratch
 *     (4*R*E + 4*R rounded up to 256, + 256 bytes) exceeds 1 MiB:
 *     at E = 256, R <= 1019.
 *   - All calls share the array.  The tickets are cleared on `stream` at the
 *     start of each call; calls that overlap on the GPU (other streams, other
 *     host threads) race on the array and must not be issued.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address; make it before any stream capture.  Calls
 *     outside a capture look it up again; calls inside one reuse the last.
 *   - Non-finite logits are counted in the array, not reported. */
moe_status moe_block_route_noalloc(const moe_plan* plan, const void* x, int32_t R,
                                   const int32_t* block_offsets, int32_t nb,
                                   const float* logit_bias, int32_t* topk_idx, float* topk_w,
                                   moe_stream_t stream);

/* Same type as cudaEvent_t. */
typedef struct CUevent_st* moe_event_t;

/* Optional per-kernel timing of moe_block_forward and moe_block_pass.  With
 * n_events == 5 the call records, on its stream, events[0] before the pair
 * scatter (moe_block_pass: before the router), events[1] before the gate/up GEMM,
 * events[2] before the down GEMM, events[3] before the final bf16 store and
 * events[4] after it.  The events
 * belong to the caller and must outlive every forward that records them;
 * n_events == 0 (events NULL) turns the recording off.  Not thread-safe
 * against concurrent forwards on the same plan. */
moe_status moe_plan_set_forward_events(moe_plan* plan, moe_event_t const* events,
                                       int32_t n_events);

/* Limit of the kernels' pipeline waits, for tests of the failure path.
 * (No counterpart on the pages: part of this library's failure handling.)
 * Every wait of the GEMM and tensor-core router pipelines gives up after a
 * limit (built in: 2 s, far beyond any legal wait); the kernel then counts
 * MOE_STATUS_WAIT_TIMEOUT, leaves its loops, waits for its own copies and
 * MMAs in flight (with their own fixed limit) and releases its tensor memory,
 * so the call returns and the context stays usable; the outputs of that call
 * are not valid.  A test sets a tiny limit to make the waits run out and
 * checks that path; limit_ns == 0 restores the built-in limit.  Applies to
 * calls enqueued after it; not thread-safe against concurrent calls on the
 * plan. */
moe_status moe_plan_set_wait_limit(moe_plan* plan, uint64_t limit_ns);

/* Copy the MOE_STATUS_WORDS counters to out[] (host); synchronises `stream`. */
moe_status moe_read_device_status(const void* workspace, moe_stream_t stream, uint32_t* out);

/* Zero the status counters (enqueued on `stream`). */
moe_status moe_clear_device_status(void* workspace, moe_stream_t stream);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char* moe_last_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_BLOCK_H */
