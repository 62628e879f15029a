/*
 * CPU oracle for MegaBlocks-style MoE token routing.
 *
 * TEST INFRASTRUCTURE ONLY. Plain, slow, single-threaded loops that restate
 * what the pages define, so that the CUDA library can be checked against
 * them. Only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use this file. It shares no code, header, table or helper with the CUDA
 * library, and the library never calls it.
 *
 * Sources (page title, section):
 *   [binned]  "Build Triton-Ascend Binned MoE Routing" (SKILL.md):
 *             Goal; Workflow steps 1-6; Implementation Pattern; Ascend
 *             Guardrails; Verification.
 *   [padded]  "Build Triton-Ascend Padded MoE Routing" (SKILL.md):
 *             Goal; Workflow steps 1-6; Implementation Pattern; Ascend
 *             Guardrails; Verification.
 *   [mok]     Megatron-Core API docs, "core.transformer.moe.megakernel.mok.
 *             route_adapter": RoutingMapToIndices (class summary, forward,
 *             backward) and routing_map_to_mok_inputs (Parameters, Returns).
 *
 * Readings where the pages leave a step open:
 *   - the sort by expert is stable: within an expert, assignments keep
 *     increasing assignment id, so capacity keeps the earliest tokens (the
 *     only deterministic choice; it decides which assignments survive);
 *   - an expert with no assignment gets a padded segment of length zero;
 *   - the TOP_K slots of a token are summed in fp32 in slot order
 *     k = 0..TOP_K-1, starting from +0.0, skipping dropped slots; a weighted
 *     slot contributes fl(w * v); no fused multiply-add (build with
 *     -ffp-contract=off);
 *   - wgrad of an assignment that was dropped by capacity is 0; wgrad of a
 *     kept one is the dot product accumulated in double and rounded to fp32
 *     once (more accurate than the fp32 the pages ask of the kernel, so the
 *     kernel is judged by a tolerance);
 *   - compaction keeps the first `topk` routes in increasing expert order and
 *     drops the rest; the backward writes every entry of the dense gradient,
 *     zero where no compact slot points.
 *
 * Element types: dtype 0 = fp32, dtype 1 = bf16 stored as uint16 bit
 * patterns. Router weights, wgrad and every compaction float are fp32.
 * Index vectors are int32; assignment id a = t*TOP_K + k.
 *
 * Every function returns 0 on success and a nonzero code when its inputs
 * break the invariants it relies on (it then leaves outputs unspecified but
 * never reads or writes out of bounds).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

/* bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 word. */
static float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even; NaN stays NaN (quiet). */
static uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

static float load_elem(const void* base, int dtype, int64_t idx) {
    if (dtype == ORC_F32) return ((const float*)base)[idx];
    return bf16_to_f32(((const uint16_t*)base)[idx]);
}

static void store_elem(void* base, int dtype, int64_t idx, float v) {
    if (dtype == ORC_F32) ((float*)base)[idx] = v;
    else ((uint16_t*)base)[idx] = f32_to_bf16(v);
}

static size_t elem_size(int dtype) { return dtype == ORC_F32 ? 4 : 2; }

/* Start of expert e's real segment in sorted order: 0 for e = 0, else
 * bins[e-1] ([binned] Implementation Pattern, expert_start). */
static int64_t seg_start(const int32_t* cum, int32_t e) { return e == 0 ? 0 : cum[e - 1]; }

/*
 * Route build ([padded] Workflow steps 1-3; [binned] Workflow steps 1-2).
 * indices: the assignment ids ordered by expert, ascending assignment id
 *          within an expert (stable);
 * bin_ids: the expert of each sorted position (nondecreasing);
 * bins:    inclusive cumulative count through expert e;
 * padded_bins: inclusive cumulative sum of each count rounded up to a
 *          multiple of m;
 * positions: inverse of indices (positions[indices[i]] = i).
 * Written as the definition: for each expert in turn, list its assignments
 * in increasing id. Returns 1 if an expert id is outside [0, E).
 */
int oracle_route_build(const int32_t* top_expert, int64_t n, int32_t E, int32_t m,
                       int32_t* indices, int32_t* bin_ids, int32_t* bins,
                       int32_t* padded_bins, int32_t* positions) {
    if (E < 1 || m < 1 || n < 0) return 2;
    for (int64_t a = 0; a < n; ++a)
        if (top_expert[a] < 0 || top_expert[a] >= E) return 1;
    int64_t i = 0, padded_total = 0;
    for (int32_t e = 0; e < E; ++e) {
        int64_t count = 0;
        for (int64_t a = 0; a < n; ++a) {
            if (top_expert[a] == e) {
                indices[i] = (int32_t)a;
                bin_ids[i] = e;
                ++i;
                ++count;
            }
        }
        bins[e] = (int32_t)i;
        padded_total += ((count + m - 1) / m) * m;
        padded_bins[e] = (int32_t)padded_total;
    }
    for (int64_t j = 0; j < n; ++j) positions[indices[j]] = (int32_t)j;
    return 0;
}

/*
 * Row of the expert tensor that sorted position i lands in, or -1 when the
 * assignment is dropped.
 *   binned ([binned] Implementation Pattern): offset = i - expert_start;
 *          kept iff offset < capacity; row = expert * capacity + offset.
 *   padded ([padded] Implementation Pattern / Workflow step 4):
 *          row = padded_start + (i - real_start); always kept.
 * padded_bins == NULL selects the binned rule.
 */
static int64_t expert_row(int64_t i, const int32_t* bin_ids, const int32_t* bins,
                          const int32_t* padded_bins, int32_t capacity) {
    int32_t e = bin_ids[i];
    int64_t offset = i - seg_start(bins, e);
    if (padded_bins == NULL) {
        if (offset >= capacity) return -1;
        return (int64_t)e * capacity + offset;
    }
    return seg_start(padded_bins, e) + offset;
}

/* Checks the aligned-vector preconditions the gather/scatter steps rely on
 * ([binned] Guardrails: bins monotonic, bins[-1] == len(indices), bin_ids
 * consistent with bin boundaries; [padded] Guardrails: padded segments no
 * shorter than real counts) plus index ranges, so that no access below goes
 * out of bounds. */
static int check_bins(const int32_t* indices, const int32_t* bin_ids, const int32_t* bins,
                      const int32_t* padded_bins, int64_t n, int32_t E) {
    for (int32_t e = 0; e < E; ++e) {
        if (seg_start(bins, e) > bins[e]) return 3;
        if (padded_bins) {
            if (seg_start(padded_bins, e) > padded_bins[e]) return 3;
            if (padded_bins[e] - seg_start(padded_bins, e) < bins[e] - seg_start(bins, e)) return 3;
        }
    }
    if (E > 0 && bins[E - 1] != n) return 3;
    for (int64_t i = 0; i < n; ++i) {
        int32_t e = bin_ids[i];
        if (e < 0 || e >= E) return 4;
        if (i < seg_start(bins, e) || i >= bins[e]) return 4;
        if (indices[i] < 0 || indices[i] >= n) return 5;
    }
    return 0;
}

/*
 * Routing check ([binned] Guardrails: bins monotonic, bins[-1] ==
 * len(indices), bin_ids aligned with the bin boundaries; [padded]
 * Guardrails: padded segments no shorter than the real counts; [padded]
 * Workflow step 1: assignments sorted by expert, in increasing id within an
 * expert). Returns the OR of status bits, 0 for a consistent routing:
 *   4 (bins):   bins[0] < 0, bins decreasing, bins[E-1] != n, padded_bins
 *               decreasing or a padded segment shorter than its count,
 *               sorted position i outside the segment of bin_ids[i];
 *   1 (expert): bin_ids[i] outside [0, E);
 *   2 (index):  indices[i] outside [0, n), indices not increasing inside a
 *               run of equal bin_ids, or (positions given)
 *               positions[indices[i]] != i.
 * Every condition is tested for every element; nothing stops early.
 */
int oracle_check_routing(const int32_t* indices, const int32_t* bin_ids, const int32_t* bins,
                         const int32_t* padded_bins, const int32_t* positions, int64_t n, int32_t E) {
    int bits = 0;
    for (int32_t e = 0; e < E; ++e) {
        int64_t start = seg_start(bins, e);
        if (bins[e] < start || (e == 0 && bins[0] < 0)) bits |= 4;
        if (padded_bins) {
            int64_t pstart = seg_start(padded_bins, e);
            if (padded_bins[e] < pstart || padded_bins[e] - pstart < (int64_t)bins[e] - start) bits |= 4;
        }
    }
    if (E > 0 && bins[E - 1] != n) bits |= 4;
    for (int64_t i = 0; i < n; ++i) {
        int32_t e = bin_ids[i];
        if (e < 0 || e >= E) {
            bits |= 1;
        } else if (i < seg_start(bins, e) || i >= bins[e]) {
            bits |= 4;
        }
        int32_t a = indices[i];
        if (a < 0 || a >= n) {
            bits |= 2;
        } else if (positions && positions[a] != i) {
            bits |= 2;
        }
        if (i > 0 && bin_ids[i] == bin_ids[i - 1] && a <= indices[i - 1]) bits |= 2;
    }
    return bits;
}

/*
 * Gather ([binned] Goal, Workflow step 3, Guardrails; [padded] Goal,
 * Workflow steps 4-5, Guardrails). out has out_rows rows of H elements:
 * E*capacity rows (binned, padded_bins == NULL) or padded_bins[E-1] rows
 * (padded). It is zero-initialised, then every kept sorted position i copies
 * token indices[i] / TOP_K into its expert row.
 */
static int gather(const void* x, int dtype, const int32_t* indices, const int32_t* bin_ids,
                  const int32_t* bins, const int32_t* padded_bins, int64_t T, int64_t H,
                  int32_t E, int32_t capacity, int32_t top_k, void* out, int64_t out_rows) {
    int64_t n = T * top_k;
    int rc = check_bins(indices, bin_ids, bins, padded_bins, n, E);
    if (rc) return rc;
    size_t b = elem_size(dtype);
    memset(out, 0, (size_t)out_rows * (size_t)H * b);
    for (int64_t i = 0; i < n; ++i) {
        int64_t row = expert_row(i, bin_ids, bins, padded_bins, capacity);
        if (row < 0) continue;
        if (row >= out_rows) return 6;
        int64_t token = indices[i] / top_k;
        memcpy((char*)out + (size_t)row * H * b, (const char*)x + (size_t)token * H * b, (size_t)H * b);
    }
    return 0;
}

/*
 * Weighted gather: the gradient of the combine with respect to the expert
 * rows. The pages give the combine ([binned] Workflow step 5; [padded]
 * Workflow step 6: y[t] = sum over kept slots of weights[a] * row(a)); its
 * derivative with respect to row(a) is weights[a] * dy[a / TOP_K]. So out
 * is zero-filled and every kept sorted position i writes
 * fl(weights[indices[i]] * dy[indices[i] / TOP_K]) to its expert row,
 * rounded to dtype. weights == NULL gives the plain gather.
 */
static int gather_weighted(const void* dy, int dtype, const int32_t* indices, const int32_t* bin_ids,
                           const int32_t* bins, const int32_t* padded_bins, const float* weights,
                           int64_t T, int64_t H, int32_t E, int32_t capacity, int32_t top_k, void* out,
                           int64_t out_rows) {
    int64_t n = T * top_k;
    int rc = check_bins(indices, bin_ids, bins, padded_bins, n, E);
    if (rc) return rc;
    memset(out, 0, (size_t)out_rows * (size_t)H * elem_size(dtype));
    for (int64_t i = 0; i < n; ++i) {
        int64_t row = expert_row(i, bin_ids, bins, padded_bins, capacity);
        if (row < 0) continue;
        if (row >= out_rows) return 6;
        int64_t a = indices[i];
        int64_t token = a / top_k;
        for (int64_t h = 0; h < H; ++h) {
            float v = load_elem(dy, dtype, token * H + h);
            float scaled = weights ? weights[a] * v : v;
            store_elem(out, dtype, row * H + h, scaled);
        }
    }
    return 0;
}

int oracle_binned_gather_weighted(const void* dy, int dtype, const int32_t* indices, const int32_t* bin_ids,
                                  const int32_t* bins, const float* weights, int64_t T, int64_t H, int32_t E,
                                  int32_t capacity, int32_t top_k, void* out) {
    if (capacity < 0) return 2;
    return gather_weighted(dy, dtype, indices, bin_ids, bins, NULL, weights, T, H, E, capacity, top_k, out,
                           (int64_t)E * capacity);
}

int oracle_padded_gather_weighted(const void* dy, int dtype, const int32_t* indices, const int32_t* bin_ids,
                                  const int32_t* bins, const int32_t* padded_bins, const float* weights,
                                  int64_t T, int64_t H, int32_t E, int32_t top_k, void* out, int64_t out_rows) {
    return gather_weighted(dy, dtype, indices, bin_ids, bins, padded_bins, weights, T, H, E, 0, top_k, out,
                           out_rows);
}

int oracle_binned_gather(const void* x, int dtype, const int32_t* indices, const int32_t* bin_ids,
                         const int32_t* bins, int64_t T, int64_t H, int32_t E, int32_t capacity,
                         int32_t top_k, void* out) {
    if (capacity < 0) return 2;
    return gather(x, dtype, indices, bin_ids, bins, NULL, T, H, E, capacity, top_k, out,
                  (int64_t)E * capacity);
}

int oracle_padded_gather(const void* x, int dtype, const int32_t* indices, const int32_t* bin_ids,
                         const int32_t* bins, const int32_t* padded_bins, int64_t T, int64_t H,
                         int32_t E, int32_t top_k, void* out, int64_t out_rows) {
    return gather(x, dtype, indices, bin_ids, bins, padded_bins, T, H, E, 0, top_k, out, out_rows);
}

/*
 * Scatter / combine ([binned] Workflow step 5, Guardrails "accumulate
 * weighted values in float32"; [padded] Workflow step 6, Guardrails on
 * weight indexing weights[indices[position]]).
 * Step 1: every kept sorted position stores its expert row into the unique
 *         slot of its assignment id indices[i] (here: records which row).
 * Step 2: for each token, the TOP_K slots are optionally scaled by the
 *         router weight of the assignment and summed in fp32, k ascending.
 * weights == NULL means unscaled.
 */
static int scatter(const void* xe, int dtype, const int32_t* indices, const int32_t* bin_ids,
                   const int32_t* bins, const int32_t* padded_bins, const float* weights,
                   int64_t T, int64_t H, int32_t E, int32_t capacity, int32_t top_k,
                   int64_t xe_rows, void* out) {
    int64_t n = T * top_k;
    int rc = check_bins(indices, bin_ids, bins, padded_bins, n, E);
    if (rc) return rc;
    int64_t* slot_row = (int64_t*)malloc((size_t)(n > 0 ? n : 1) * sizeof(int64_t));
    float* acc = (float*)malloc((size_t)(H > 0 ? H : 1) * sizeof(float));
    if (!slot_row || !acc) { free(slot_row); free(acc); return 7; }
    for (int64_t a = 0; a < n; ++a) slot_row[a] = -1;
    for (int64_t i = 0; i < n; ++i) {
        int64_t row = expert_row(i, bin_ids, bins, padded_bins, capacity);
        if (row >= xe_rows) { free(slot_row); free(acc); return 6; }
        slot_row[indices[i]] = row;
    }
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) acc[h] = 0.0f;
        for (int32_t k = 0; k < top_k; ++k) {
            int64_t a = t * top_k + k;
            int64_t row = slot_row[a];
            if (row < 0) continue;
            for (int64_t h = 0; h < H; ++h) {
                float v = load_elem(xe, dtype, row * H + h);
                if (weights) {
                    float scaled = weights[a] * v;
                    acc[h] = acc[h] + scaled;
                } else {
                    acc[h] = acc[h] + v;
                }
            }
        }
        for (int64_t h = 0; h < H; ++h) store_elem(out, dtype, t * H + h, acc[h]);
    }
    free(slot_row);
    free(acc);
    return 0;
}

int oracle_binned_scatter(const void* xe, int dtype, const int32_t* indices, const int32_t* bin_ids,
                          const int32_t* bins, const float* weights, int64_t T, int64_t H,
                          int32_t E, int32_t capacity, int32_t top_k, void* out) {
    if (capacity < 0) return 2;
    return scatter(xe, dtype, indices, bin_ids, bins, NULL, weights, T, H, E, capacity, top_k,
                   (int64_t)E * capacity, out);
}

int oracle_padded_scatter(const void* xe, int dtype, const int32_t* indices, const int32_t* bin_ids,
                          const int32_t* bins, const int32_t* padded_bins, const float* weights,
                          int64_t T, int64_t H, int32_t E, int32_t top_k, int64_t xe_rows,
                          void* out) {
    return scatter(xe, dtype, indices, bin_ids, bins, padded_bins, weights, T, H, E, 0, top_k,
                   xe_rows, out);
}

/*
 * Router-weight gradient ([binned] Goal, Workflow step 6; [padded] Workflow
 * step 6, Guardrails on unique assignment ids and column-tile reduction).
 * For each kept sorted position i: wgrad[indices[i]] = dot(expert row of i,
 * grad[indices[i] / TOP_K]). Accumulated in double, rounded to fp32 once.
 * Assignments dropped by capacity get 0.
 */
static int wgrad(const void* xe, const void* grad, int dtype, const int32_t* indices,
                 const int32_t* bin_ids, const int32_t* bins, const int32_t* padded_bins,
                 int64_t T, int64_t H, int32_t E, int32_t capacity, int32_t top_k,
                 int64_t xe_rows, float* out) {
    int64_t n = T * top_k;
    int rc = check_bins(indices, bin_ids, bins, padded_bins, n, E);
    if (rc) return rc;
    for (int64_t a = 0; a < n; ++a) out[a] = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        int64_t row = expert_row(i, bin_ids, bins, padded_bins, capacity);
        if (row < 0) continue;
        if (row >= xe_rows) return 6;
        int64_t token = indices[i] / top_k;
        double dot = 0.0;
        for (int64_t h = 0; h < H; ++h)
            dot += (double)load_elem(xe, dtype, row * H + h) * (double)load_elem(grad, dtype, token * H + h);
        out[indices[i]] = (float)dot;
    }
    return 0;
}

int oracle_binned_wgrad(const void* xe, const void* grad, int dtype, const int32_t* indices,
                        const int32_t* bin_ids, const int32_t* bins, int64_t T, int64_t H,
                        int32_t E, int32_t capacity, int32_t top_k, float* out) {
    if (capacity < 0) return 2;
    return wgrad(xe, grad, dtype, indices, bin_ids, bins, NULL, T, H, E, capacity, top_k,
                 (int64_t)E * capacity, out);
}

int oracle_padded_wgrad(const void* xe, const void* grad, int dtype, const int32_t* indices,
                        const int32_t* bin_ids, const int32_t* bins, const int32_t* padded_bins,
                        int64_t T, int64_t H, int32_t E, int32_t top_k, int64_t xe_rows,
                        float* out) {
    return wgrad(xe, grad, dtype, indices, bin_ids, bins, padded_bins, T, H, E, 0, top_k,
                 xe_rows, out);
}

/*
 * Dense routing map -> fixed-width compaction ([mok] RoutingMapToIndices
 * summary and forward; routing_map_to_mok_inputs Returns). Row t lists the
 * experts e with routing_map[t][e] != 0 in increasing e; the first topk
 * become indices[t][j] = e with probs_indices[t][j] = probs[t][e]; the
 * remaining slots are -1 and 0.0f.
 */
int oracle_routing_map_to_indices_fwd(const float* probs, const int8_t* routing_map, int64_t T,
                                      int32_t E, int32_t topk, float* probs_indices,
                                      int32_t* indices) {
    if (T < 0 || E < 1 || topk < 1) return 2;
    for (int64_t t = 0; t < T; ++t) {
        int32_t j = 0;
        for (int32_t e = 0; e < E; ++e) {
            if (routing_map[t * E + e] != 0 && j < topk) {
                indices[t * topk + j] = e;
                probs_indices[t * topk + j] = probs[t * E + e];
                ++j;
            }
        }
        for (; j < topk; ++j) {
            indices[t * topk + j] = -1;
            probs_indices[t * topk + j] = 0.0f;
        }
    }
    return 0;
}

/*
 * Backward of the compaction ([mok] RoutingMapToIndices backward;
 * _routing_map_to_indices_backward_kernel): grad_probs starts at zero and
 * each compact slot with a valid index writes its gradient to
 * grad_probs[t][indices[t][j]] (slots visited j ascending, so with repeated
 * indices the last one wins). Slots holding -1 contribute nothing; an index
 * outside [-1, E) returns 1 and is skipped.
 */
int oracle_routing_map_to_indices_bwd(const float* grad_probs_indices, const int32_t* indices,
                                      int64_t T, int32_t E, int32_t topk, float* grad_probs) {
    if (T < 0 || E < 1 || topk < 1) return 2;
    int rc = 0;
    for (int64_t q = 0; q < T * E; ++q) grad_probs[q] = 0.0f;
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < topk; ++j) {
            int32_t e = indices[t * topk + j];
            if (e == -1) continue;
            if (e < -1 || e >= E) { rc = 1; continue; }
            grad_probs[t * E + e] = grad_probs_indices[t * topk + j];
        }
    }
    return rc;
}

/*
 * Router top-k gating ("Fused MoE Dispatch (Triton, universal)": the
 * pipeline "router scores -> top-k gating -> permute", usage example with
 * gating="softmax" or "sigmoid"). Per token t:
 *   - the top_k experts with the largest logits, in decreasing logit order,
 *     ties to the lower expert id (a NaN logit counts as -infinity); both
 *     scores below increase with the logit, so this is the top_k by score;
 *   - score of expert e: softmax over all E logits (mode 0) or the logistic
 *     sigmoid of its logit (mode 1), in double;
 *   - weights[t][k] = score of the k-th chosen expert, divided by the sum of
 *     the chosen scores when normalize != 0; rounded to fp32 once.
 * Degenerate rows (every logit -inf or NaN, or chosen scores summing to 0)
 * take the limit of equal logits: a uniform softmax, weights 1 / top_k.
 * Requires 1 <= top_k <= E.
 */
int oracle_topk_gating(const float* logits, int64_t T, int32_t E, int32_t top_k, int mode, int normalize,
                       int32_t* top_expert, float* weights) {
    if (T < 0 || E < 1 || top_k < 1 || top_k > E || (mode != 0 && mode != 1)) return 2;
    char* chosen = (char*)malloc((size_t)E);
    double* score = (double*)malloc((size_t)E * sizeof(double));
    if (!chosen || !score) { free(chosen); free(score); return 7; }
    for (int64_t t = 0; t < T; ++t) {
        const float* l = logits + t * E;
        double lmax = -INFINITY;
        for (int32_t e = 0; e < E; ++e) {
            double v = isnan(l[e]) ? -INFINITY : (double)l[e];
            if (v > lmax) lmax = v;
        }
        double z = 0.0;
        for (int32_t e = 0; e < E; ++e) {
            double v = isnan(l[e]) ? -INFINITY : (double)l[e];
            if (mode == 0) {
                /* every logit -inf: the limit of equal logits, a uniform softmax */
                score[e] = lmax == -INFINITY ? 1.0 : exp(v - lmax);
                z += score[e];
            } else {
                score[e] = 1.0 / (1.0 + exp(-v));
            }
        }
        if (mode == 0)
            for (int32_t e = 0; e < E; ++e) score[e] /= z;
        memset(chosen, 0, (size_t)E);
        double chosen_sum = 0.0;
        for (int32_t k = 0; k < top_k; ++k) {
            int32_t best = -1;
            float bv = 0.0f;
            for (int32_t e = 0; e < E; ++e) {
                if (chosen[e]) continue;
                float v = isnan(l[e]) ? -INFINITY : l[e];
                if (best < 0 || v > bv) { best = e; bv = v; }
            }
            chosen[best] = 1;
            top_expert[t * top_k + k] = best;
            chosen_sum += score[best];
        }
        for (int32_t k = 0; k < top_k; ++k) {
            double w = score[top_expert[t * top_k + k]];
            /* chosen scores all zero: the limit of equal scores, 1 / top_k each */
            if (normalize) w = chosen_sum > 0.0 ? w / chosen_sum : 1.0 / top_k;
            weights[t * top_k + k] = (float)w;
        }
    }
    free(chosen);
    free(score);
    return 0;
}

/* Round fp32 values to bf16 bits (test helper for expected outputs). */
void oracle_f32_to_bf16(const float* in, int64_t count, uint16_t* out) {
    for (int64_t q = 0; q < count; ++q) out[q] = f32_to_bf16(in[q]);
}
