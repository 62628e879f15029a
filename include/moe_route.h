/*
 * moe_route.h - C ABI of the GB300 (sm_103a) MoE token-routing library
 * (libmoe_route.so).
 *
 * The library implements the data-parallel routing path of a
 * MegaBlocks-style Mixture-of-Experts layer:
 *   [top-k gating] -> route build -> binned / padded gather (permute)
 *   -> [expert FFN, not here] -> binned / padded scatter (combine)
 *   -> router-weight gradient and expert-row gradient (weighted gather),
 * plus the dense routing-map -> fixed-width top-k compaction and its
 * backward. Sources, by page title and section:
 *   [binned] "Build Triton-Ascend Binned MoE Routing": Goal, Workflow,
 *            Implementation Pattern, Ascend Guardrails, Verification.
 *   [padded] "Build Triton-Ascend Padded MoE Routing": Goal, Workflow,
 *            Implementation Pattern, Ascend Guardrails, Verification.
 *   [mok]    Megatron-Core API docs, core.transformer.moe.megakernel.mok.
 *            route_adapter: RoutingMapToIndices, routing_map_to_mok_inputs.
 *   [dispatch] "Fused MoE Dispatch (Triton, universal)": pipeline and usage.
 *
 * Conventions (all entry points):
 *  - Every pointer is a DEVICE pointer owned by the caller. The library
 *    allocates no memory: scratch space is passed in through `workspace`,
 *    sized by the matching *_workspace_size() call.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and runs asynchronously. No entry point synchronises the host.
 *  - Outputs are written completely, zeros included; callers need not clear
 *    them. Inputs are read-only. Outputs must not alias inputs or each other.
 *  - Assignment id a = t * top_k + k for token t and slot k; n = T * top_k.
 *    Index vectors are int32 and n must fit in int32.
 *  - dtype selects the activation type: MOE_F32 (float) or MOE_BF16
 *    (__nv_bfloat16 bits). Router weights, wgrad and all compaction floats
 *    are fp32. Activations are row-major [rows, hidden].
 *  - Return value: MOE_OK, or an MOE_ERR_* code. Argument errors are found
 *    on the host before anything is enqueued; MOE_ERR_CUDA reports a launch
 *    failure (cudaGetLastError).
 *  - Errors in device-resident data (an expert id outside [0, E), bins that
 *    are not monotonic, an index outside its range) cannot be reported
 *    synchronously. Entry points that read such data take `d_status`: a
 *    nullable device int32 into which kernels OR MOE_STATUS_* bits. Kernels
 *    never trap; they skip the offending element, keep every access in
 *    bounds, and leave the affected outputs unspecified. The caller clears
 *    *d_status before the calls it wants to check.
 */
#ifndef MOE_ROUTE_H
#define MOE_ROUTE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* moe_stream_t;

enum moe_error {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null required pointer, size out of range, n overflowing int32 */
  MOE_ERR_UNSUPPORTED = 2, /* dtype, or a pointer not aligned to its element size */
  MOE_ERR_CUDA = 3         /* a kernel launch failed */
};

enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1 };

/* Bits OR-ed into *d_status by kernels that meet invalid device data. */
enum moe_device_status {
  MOE_STATUS_BAD_EXPERT = 1,   /* expert id outside [0, E) */
  MOE_STATUS_BAD_INDEX = 2,    /* an index or position outside its range, or a positions
                                   entry that indices does not map back
                                   (indices[positions[a]] != a) */
  MOE_STATUS_BAD_BINS = 4,     /* bins / padded_bins not monotonic or not consistent */
  MOE_STATUS_ROWS_MISMATCH = 8, /* padded_bins[E-1] exceeds the rows the caller provided */
  MOE_STATUS_TIMEOUT = 16       /* a bounded wait gave up (on an asynchronous copy, or at a grid
                                   barrier of the one-launch route build + gather): the
                                   launch's outputs are unspecified and the stream must be
                                   treated as failed (a copy may still be landing) */
};

/* Library limits (inclusive). */
#define MOE_MAX_EXPERTS 4096
#define MOE_MAX_TOP_K 64

/* Human-readable name of an MOE_ERR_* code (static string). */
const char* moe_error_string(int code);

/* Library version as major*10000 + minor*100 + patch. */
int moe_version(void);

/*
 * Route build ([padded] Workflow steps 1-3; [binned] Workflow steps 1-2).
 * Stable counting sort of the n = T*top_k expert choices by expert id.
 *   top_expert  [n] int32   expert of assignment a (row-major [T, top_k]).
 *   indices     [n] int32   out: assignment id at each sorted position;
 *                           within an expert, ids ascend (stable).
 *   bin_ids     [n] int32   out: expert of each sorted position
 *                           (nondecreasing).
 *   bins        [E] int32   out: inclusive cumulative count through expert e
 *                           (bins[E-1] == n).
 *   padded_bins [E] int32   out, nullable: inclusive cumulative sum of each
 *                           count rounded up to a multiple of pad_multiple
 *                           (an empty expert stays 0 rows).
 *   positions   [n] int32   out, nullable: inverse of indices
 *                           (positions[indices[i]] == i). Passing it to the
 *                           scatter entry points saves them a pass.
 *   workspace   >= moe_route_build_workspace_size(n, E) bytes of device
 *                           scratch, 4-byte aligned; contents need no
 *                           initialisation and are clobbered.
 * Requires 0 <= n <= INT32_MAX, 1 <= E <= MOE_MAX_EXPERTS, pad_multiple >= 1
 * and n + E*(pad_multiple-1) <= INT32_MAX. An expert id outside [0, E) sets
 * MOE_STATUS_BAD_EXPERT and is left out of every output (outputs are then
 * unspecified).
 */
size_t moe_route_build_workspace_size(int64_t n, int32_t num_experts);
int moe_route_build(const int32_t* top_expert, int64_t n, int32_t num_experts,
                    int32_t pad_multiple, int32_t* indices, int32_t* bin_ids,
                    int32_t* bins, int32_t* padded_bins, int32_t* positions,
                    void* workspace, size_t workspace_bytes, int32_t* d_status,
                    moe_stream_t stream);

/*
 * Route build that allocates nothing. The pages have no counterpart: this is
 * a convenience of this library, not part of the method.
 * Same arguments, outputs and device-status behaviour as moe_route_build,
 * minus the workspace. It is meant for callers that cannot hand the library
 * any scratch memory: a plain C host that owns only its inputs and outputs,
 * a plugin running under a framework that holds the whole device memory pool
 * without exposing an allocator, or a hot loop that must not call cudaMalloc
 * (which may synchronise the device).
 *  - The scratch is a static device array of MOE_ROUTE_BUILD_NOALLOC_MAX_BYTES
 *    inside the library; every GPU on which the library is loaded keeps it
 *    reserved until the process exits. No cudaMalloc / cudaFree is called.
 *  - Size limit: returns MOE_ERR_INVALID_ARG, without enqueuing anything,
 *    when moe_route_build_workspace_size(n, num_experts) exceeds
 *    MOE_ROUTE_BUILD_NOALLOC_MAX_BYTES (for E = 256 that is n above about
 *    one million assignments); use moe_route_build with a caller workspace
 *    then.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) and caches it; make that first call before any
 *    stream capture on that device. It returns MOE_ERR_CUDA if the lookup
 *    fails. The cached address is kept for the life of the process: after a
 *    cudaDeviceReset the library's device image is loaded again and the
 *    array may move, so do not call this entry point on a device that has
 *    been reset since its first call.
 *  - All calls on a device share the one array, which keeps the last call's
 *    contents (nothing in it needs to start at zero). Calls whose work
 *    overlaps on the GPU - on different streams without ordering between
 *    them - race on it and produce wrong results: order them on one stream
 *    or with events.
 */
#define MOE_ROUTE_BUILD_NOALLOC_MAX_BYTES (1u << 20)
int moe_route_build_noalloc(const int32_t* top_expert, int64_t n,
                            int32_t num_experts, int32_t pad_multiple,
                            int32_t* indices, int32_t* bin_ids, int32_t* bins,
                            int32_t* padded_bins, int32_t* positions,
                            int32_t* d_status, moe_stream_t stream);

/*
 * Routing check ([binned] Guardrails: bins monotonic, bins[-1] == n, bin_ids
 * aligned with the bin boundaries; [padded] Guardrails: padded segments no
 * shorter than the counts; [padded] Workflow step 1: sorted by expert, in
 * increasing assignment id within an expert). ORs into *d_status (the
 * caller zeroes it first; required):
 *   MOE_STATUS_BAD_BINS    bins[0] < 0, bins decreasing, bins[E-1] != n,
 *                          padded_bins decreasing or a padded segment shorter
 *                          than its count, or a sorted position outside the
 *                          segment of its bin_ids entry;
 *   MOE_STATUS_BAD_EXPERT  a bin_ids entry outside [0, E);
 *   MOE_STATUS_BAD_INDEX   an indices entry outside [0, n), indices not
 *                          increasing inside a run of equal bin_ids, or
 *                          (positions given) positions[indices[i]] != i —
 *                          with positions this certifies that indices is a
 *                          permutation.
 *   indices, bin_ids [n]; bins [E]; padded_bins [E] and positions [n]
 *   nullable (their conditions are then skipped). One launch, no host sync.
 */
int moe_check_routing(const int32_t* indices, const int32_t* bin_ids,
                      const int32_t* bins, const int32_t* padded_bins,
                      const int32_t* positions, int64_t n, int32_t num_experts,
                      int32_t* d_status, moe_stream_t stream);

/*
 * Binned gather ([binned] Goal, Workflow step 3, Implementation Pattern,
 * Guardrails). For expert e and slot j < capacity:
 *   out[e, j, :] = x[indices[bins[e-1] + j] / top_k, :]  if j < count_e,
 *                  0                                      otherwise,
 * with bins[-1] read as 0. Assignments beyond capacity are dropped.
 *   x    [T, H] dtype;  out [E, capacity, H] dtype (fully written).
 *   indices [n], bins [E] from moe_route_build; n = T*top_k.
 *   positions [n] int32, nullable: the inverse permutation of indices
 *   (positions[indices[i]] = i), as moe_route_build writes it. Every entry
 *   is checked against indices before it is followed.
 * capacity >= 0; capacity == 0 writes nothing.
 * Schedule (the result does not depend on it): with positions, one launch
 * that copies each token row once to all of its kept rows and zero-fills
 * the rest. Without them, when out holds more than 4n bytes plus one row,
 * the gather first stores the inverse permutation of indices in the last 4n
 * bytes of out (16-byte aligned), then copies each token row once to all of
 * its kept rows, then writes the rows that overlap those bytes; three
 * launches, no workspace. out must not alias any input.
 * A sorted position that does not map back to its assignment (indices not a
 * permutation) sets MOE_STATUS_BAD_INDEX; bins that decrease or pass n set
 * MOE_STATUS_BAD_BINS. The same holds for every gather below.
 */
int moe_binned_gather(const void* x, int32_t dtype, const int32_t* indices,
                      const int32_t* bins, const int32_t* positions,
                      int64_t num_tokens, int64_t hidden, int32_t num_experts,
                      int32_t capacity, int32_t top_k, void* out,
                      int32_t* d_status, moe_stream_t stream);

/*
 * Padded gather ([padded] Goal, Workflow steps 4-5, Implementation Pattern,
 * Guardrails). Row padded_bins[e-1] + j of out receives
 * x[indices[bins[e-1] + j] / top_k] for j < count_e; padding rows are zero.
 *   out [out_rows, H] dtype. out_rows is the caller's row count, normally
 *   padded_bins[E-1] (read back by the caller to size the buffer). Rows at
 *   or beyond padded_bins[E-1] are zero-filled; if padded_bins[E-1] exceeds
 *   out_rows, rows past out_rows are not written and MOE_STATUS_ROWS_MISMATCH
 *   is set.
 */
int moe_padded_gather(const void* x, int32_t dtype, const int32_t* indices,
                      const int32_t* bins, const int32_t* padded_bins,
                      const int32_t* positions, int64_t num_tokens,
                      int64_t hidden, int32_t num_experts, int32_t top_k,
                      void* out, int64_t out_rows, int32_t* d_status,
                      moe_stream_t stream);

/*
 * Weighted gather: the gradient of the combine (moe_*_scatter with weights)
 * with respect to the expert rows. The pages define the combine ([binned]
 * Workflow step 5; [padded] Workflow step 6); its derivative with respect to
 * the row of a kept assignment a is weights[a] * dy[a / top_k]:
 *   out[row(a), :] = fl(weights[a] * dy[a / top_k, :])  for kept a,
 *   0                                                 for every other row,
 * each product rounded to nearest in fp32, then to dtype (nearest even).
 * Same layout, arguments and row mapping as the plain gathers, with dy [T, H]
 * in place of x and weights [n] fp32 (required when T > 0). The gradient of
 * an unweighted combine is the plain gather of dy.
 */
int moe_binned_gather_weighted(const void* dy, int32_t dtype,
                               const int32_t* indices, const int32_t* bins,
                               const float* weights, const int32_t* positions,
                               int64_t num_tokens, int64_t hidden,
                               int32_t num_experts, int32_t capacity,
                               int32_t top_k, void* out, int32_t* d_status,
                               moe_stream_t stream);
int moe_padded_gather_weighted(const void* dy, int32_t dtype,
                               const int32_t* indices, const int32_t* bins,
                               const int32_t* padded_bins, const float* weights,
                               const int32_t* positions, int64_t num_tokens,
                               int64_t hidden, int32_t num_experts,
                               int32_t top_k, void* out, int64_t out_rows,
                               int32_t* d_status, moe_stream_t stream);

/*
 * Route build and gather in one call ([padded] Workflow steps 1-5;
 * [binned] Workflow steps 1-3): exactly moe_route_build of
 * top_expert [n = T*top_k] (all five outputs, positions required) followed
 * by moe_binned_gather / moe_padded_gather of x given those positions, with
 * the same results, x read once per token.
 *   One launch when the bulk-copy gather applies (rows a multiple of 16
 *   bytes, x and out 16-byte aligned), E <= 1024, the workspace is 8-byte
 *   aligned and holds moe_route_build_gather_workspace_size(n, E) bytes,
 *   and the device accepts a cooperative launch (all CTAs resident): the
 *   CTAs count, scan and scatter the routing data between grid-wide
 *   barriers and then copy the rows. Each barrier wait is bounded; a CTA
 *   that gives up sets MOE_STATUS_TIMEOUT and stops (outputs then
 *   unspecified). The barrier word in the workspace needs no
 *   initialisation, but two such calls must not use one workspace at the
 *   same time. A CUDA graph may capture the call and replay it (each
 *   launch leaves the word clear for the next); after a timeout the word
 *   stays marked, so replays of that captured launch keep reporting
 *   MOE_STATUS_TIMEOUT until a new call (or a new capture) is made.
 *   Otherwise three or four launches (the route build's two or three and
 *   the gather's token pass, chained by programmatic dependent launch),
 *   needing only moe_route_build_workspace_size(n, E) bytes of workspace.
 *   On GB300 the chained launches measured faster at every batch size tried
 *   (16 to 8192 tokens of the DeepSeek-V3 shape: the single launch's three
 *   grid barriers cost more than the launches they replace), so the larger
 *   workspace is for callers that want exactly one kernel.
 *   padded: out has out_rows rows; the caller does not know
 *   padded_bins[E-1] before the call, so out_rows is a bound, such as
 *   n + E*(pad_multiple-1) (every padded total is at most that); rows at
 *   or beyond padded_bins[E-1] are zero-filled, and MOE_STATUS_ROWS_MISMATCH
 *   is set if padded_bins[E-1] exceeds out_rows.
 * Errors as for the two calls; argument errors return before anything is
 * enqueued. An expert id outside [0, E) sets MOE_STATUS_BAD_EXPERT (its
 * position entry is -1 on the one-launch path; outputs unspecified).
 */
size_t moe_route_build_gather_workspace_size(int64_t n, int32_t num_experts);
/*
 * Testing only: raises the target of every grid barrier of the one-launch
 * route build + gather by `extra` arrivals (0 restores it), so that the
 * bounded waits run out and the call reports MOE_STATUS_TIMEOUT without any
 * fault. Process-wide; not for concurrent use with real calls.
 */
void moe_test_barrier_slack(uint32_t extra);
int moe_route_build_binned_gather(const int32_t* top_expert, const void* x,
                                  int32_t dtype, int64_t num_tokens,
                                  int64_t hidden, int32_t num_experts,
                                  int32_t top_k, int32_t capacity,
                                  int32_t pad_multiple, int32_t* indices,
                                  int32_t* bin_ids, int32_t* bins,
                                  int32_t* padded_bins, int32_t* positions,
                                  void* out, void* workspace,
                                  size_t workspace_bytes, int32_t* d_status,
                                  moe_stream_t stream);
int moe_route_build_padded_gather(const int32_t* top_expert, const void* x,
                                  int32_t dtype, int64_t num_tokens,
                                  int64_t hidden, int32_t num_experts,
                                  int32_t top_k, int32_t pad_multiple,
                                  int32_t* indices, int32_t* bin_ids,
                                  int32_t* bins, int32_t* padded_bins,
                                  int32_t* positions, void* out,
                                  int64_t out_rows, void* workspace,
                                  size_t workspace_bytes, int32_t* d_status,
                                  moe_stream_t stream);

/*
 * Scatter / combine ([binned] Workflow step 5, Guardrails; [padded]
 * Workflow step 6, Guardrails). For each token t:
 *   out[t, :] = sum_{k=0..top_k-1, slot kept} s_a * xe[row(a), :],
 *   a = t*top_k + k, s_a = weights[a] (or 1 when weights == NULL),
 * accumulated in fp32 in increasing k starting from +0.0, each weighted
 * term rounded as fl(s_a * v) (no fused multiply-add), then rounded to
 * dtype (nearest even). A slot is kept when its offset in its expert is
 * below capacity (binned) or always (padded); dropped slots add nothing,
 * so a token whose slots are all dropped gets +0.0.
 *   xe  [E, capacity, H] (binned) or [xe_rows, H] (padded), dtype;
 *   out [T, H] dtype; weights [n] fp32 nullable, indexed by assignment id.
 *   positions [n] nullable: the inverse permutation from moe_route_build.
 *   When NULL it is rebuilt in `workspace`
 *   (>= moe_scatter_workspace_size(n) bytes); otherwise workspace may be
 *   NULL. Every entry is checked against indices before it is followed
 *   (indices[positions[a]] must equal a): a positions vector from another
 *   routing, or one with entries exchanged, sets MOE_STATUS_BAD_INDEX in
 *   d_status and the mismatched slots contribute nothing.
 */
size_t moe_scatter_workspace_size(int64_t n);
int moe_binned_scatter(const void* xe, int32_t dtype, const int32_t* indices,
                       const int32_t* bin_ids, const int32_t* bins,
                       const float* weights, const int32_t* positions,
                       int64_t num_tokens, int64_t hidden, int32_t num_experts,
                       int32_t capacity, int32_t top_k, void* out,
                       void* workspace, size_t workspace_bytes,
                       int32_t* d_status, moe_stream_t stream);
int moe_padded_scatter(const void* xe, int32_t dtype, const int32_t* indices,
                       const int32_t* bin_ids, const int32_t* bins,
                       const int32_t* padded_bins, const float* weights,
                       const int32_t* positions, int64_t num_tokens,
                       int64_t hidden, int32_t num_experts, int32_t top_k,
                       int64_t xe_rows, void* out, void* workspace,
                       size_t workspace_bytes, int32_t* d_status,
                       moe_stream_t stream);

/*
 * Router-weight gradient ([binned] Workflow step 6, Guardrails; [padded]
 * Workflow step 6, Guardrails). For every sorted position i with
 * assignment a = indices[i]:
 *   wgrad[a] = dot(xe[row(i), :], grad[a / top_k, :])  if i is kept,
 *              0                                        otherwise.
 * Accumulated in fp32 with compensated (error-free transformation)
 * summation, so the result is close to the correctly rounded dot.
 *   xe as for scatter; grad [T, H] dtype; wgrad [n] fp32 (fully written).
 * No workspace. moe_padded_wgrad visits assignments in id order so that
 * each gradient row is read about once; it takes positions (nullable, the
 * inverse permutation of indices as moe_route_build writes it, each entry
 * checked against indices): with them, one launch; without them, two (the
 * first stores the inverse permutation in wgrad itself, n 32-bit slots, the
 * second reads each slot once and overwrites it with the result).
 * moe_binned_wgrad is one launch: for E <= 1024 its warps visit only the
 * kept rows (a thread per sorted position writes the dropped slots' 0),
 * otherwise every sorted position. wgrad must not
 * alias any input; its contents are meaningful only once the call's work
 * has run. In the padded call a position that does not map back to its
 * assignment (indices not a permutation) sets MOE_STATUS_BAD_INDEX and that
 * slot's result is 0.
 */
int moe_binned_wgrad(const void* xe, const void* grad, int32_t dtype,
                     const int32_t* indices, const int32_t* bin_ids,
                     const int32_t* bins, int64_t num_tokens, int64_t hidden,
                     int32_t num_experts, int32_t capacity, int32_t top_k,
                     float* wgrad, int32_t* d_status, moe_stream_t stream);
int moe_padded_wgrad(const void* xe, const void* grad, int32_t dtype,
                     const int32_t* indices, const int32_t* bin_ids,
                     const int32_t* bins, const int32_t* padded_bins,
                     const int32_t* positions, int64_t num_tokens,
                     int64_t hidden, int32_t num_experts, int32_t top_k,
                     int64_t xe_rows, float* wgrad, int32_t* d_status,
                     moe_stream_t stream);

/*
 * Router top-k gating: the step before the route build ("Fused MoE Dispatch
 * (Triton, universal)": pipeline "router scores -> top-k gating -> permute",
 * usage gating="softmax" | "sigmoid"). For each token t:
 *   top_expert[t, 0..top_k) = the top_k experts by logit, decreasing, ties to
 *                             the lower expert id (NaN counts as -inf);
 *   weights[t, k]           = score of expert top_expert[t, k]:
 *       MOE_GATING_SOFTMAX: softmax over all E logits of the row,
 *       MOE_GATING_SIGMOID: 1 / (1 + exp(-logit)),
 *     divided by the sum of the chosen scores when normalize != 0.
 * Rows with every logit -inf (or chosen scores summing to 0) take the limit
 * of equal logits: a uniform softmax and weights 1 / top_k. Scores are
 * computed in fp32 (the selection is an exact comparison of the fp32
 * logits). top_expert is the route build's input (n = T * top_k) and weights
 * the combine's.
 *   logits [T, E] fp32; top_expert [T, top_k] int32 out; weights [T, top_k]
 *   fp32 out. 1 <= top_k <= min(E, MOE_MAX_TOP_K); E <= MOE_GATING_MAX_EXPERTS
 *   (else MOE_ERR_UNSUPPORTED).
 */
enum moe_gating { MOE_GATING_SOFTMAX = 0, MOE_GATING_SIGMOID = 1 };
#define MOE_GATING_MAX_EXPERTS 1024
int moe_topk_gating(const float* logits, int64_t num_tokens,
                    int32_t num_experts, int32_t top_k, int32_t mode,
                    int32_t normalize, int32_t* top_expert, float* weights,
                    moe_stream_t stream);

/*
 * Dense routing map -> fixed-width compaction ([mok] RoutingMapToIndices,
 * forward; routing_map_to_mok_inputs). Row t lists the experts e with
 * routing_map[t, e] != 0 in increasing e; the first topk of them give
 *   indices[t, j] = e,  probs_indices[t, j] = probs[t, e];
 * the remaining slots get -1 and 0.0f. Routes beyond topk are dropped.
 *   probs [T, E] fp32; routing_map [T, E] int8 (a bool map has the same
 *   bytes); probs_indices [T, topk] fp32 out; indices [T, topk] int32 out.
 * T >= 0, E >= 1, topk >= 1 (topk may exceed E: extra slots are padding).
 */
int moe_routing_map_to_indices_fwd(const float* probs, const int8_t* routing_map,
                                   int64_t num_tokens, int32_t num_experts,
                                   int32_t topk, float* probs_indices,
                                   int32_t* indices, moe_stream_t stream);

/*
 * Backward of the compaction ([mok] RoutingMapToIndices, backward):
 *   grad_probs[t, :] = 0;  grad_probs[t, indices[t, j]] = grad_probs_indices[t, j]
 * for every slot with indices[t, j] != -1 (the gradient for the integer
 * indices has no meaning and is not taken). With repeated indices in a row
 * the highest j wins. An index outside [-1, E) sets MOE_STATUS_BAD_INDEX and
 * is skipped.
 *   grad_probs_indices [T, topk] fp32; indices [T, topk] int32;
 *   grad_probs [T, E] fp32 out (fully written).
 */
int moe_routing_map_to_indices_bwd(const float* grad_probs_indices,
                                   const int32_t* indices, int64_t num_tokens,
                                   int32_t num_experts, int32_t topk,
                                   float* grad_probs, int32_t* d_status,
                                   moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTE_H */
