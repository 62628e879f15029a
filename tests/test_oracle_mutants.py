"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check
that at least two independent pins catch every one of them: a dropped term,
a wrong index, an unstable sort, an off-by-one capacity test, a transposed
operand, a wrong rounding rule and so on. The committed oracle is never
modified."""
import json
import os
import subprocess
import sys
import textwrap

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

# (name, text in oracle.c, replacement); each text must occur exactly once.
MUTANTS = [
    ("unstable_sort",
     "for (int64_t a = 0; a < n; ++a) {\n            if (top_expert[a] == e) {",
     "for (int64_t a = n - 1; a >= 0; --a) {\n            if (top_expert[a] == e) {"),
    ("exclusive_bins", "bins[e] = (int32_t)i;", "bins[e] = (int32_t)(i - count);"),
    ("pad_round_down", "padded_total += ((count + m - 1) / m) * m;", "padded_total += (count / m) * m;"),
    ("pad_always_extra", "padded_total += ((count + m - 1) / m) * m;", "padded_total += (count / m + 1) * m;"),
    ("capacity_off_by_one", "if (offset >= capacity) return -1;", "if (offset > capacity) return -1;"),
    ("padded_row_real_start", "return seg_start(padded_bins, e) + offset;", "return seg_start(bins, e) + offset;"),
    ("binned_row_transposed", "return (int64_t)e * capacity + offset;", "return (int64_t)offset * capacity + e;"),
    ("gather_token_mod", "int64_t token = indices[i] / top_k;\n        memcpy",
     "int64_t token = indices[i] % top_k;\n        memcpy"),
    ("gather_no_zero", "memset(out, 0, (size_t)out_rows * (size_t)H * b);",
     "memset(out, 1, (size_t)out_rows * (size_t)H * b);"),
    ("wgather_no_zero", "memset(out, 0, (size_t)out_rows * (size_t)H * elem_size(dtype));",
     "memset(out, 1, (size_t)out_rows * (size_t)H * elem_size(dtype));"),
    ("scatter_weight_index", "float scaled = weights[a] * v;", "float scaled = weights[(a + 1) % n] * v;"),
    ("scatter_drop_term", "acc[h] = acc[h] + scaled;", "acc[h] = scaled;"),
    ("scatter_unweighted_drop_term", "acc[h] = acc[h] + v;", "acc[h] = v;"),
    ("scatter_reversed_slots", "for (int32_t k = 0; k < top_k; ++k) {\n            int64_t a = t * top_k + k;",
     "for (int32_t k = top_k - 1; k >= 0; --k) {\n            int64_t a = t * top_k + k;"),
    ("scatter_skip_first_slot", "for (int32_t k = 0; k < top_k; ++k) {\n            int64_t a = t * top_k + k;",
     "for (int32_t k = (top_k > 1 ? 1 : 0); k < top_k; ++k) {\n            int64_t a = t * top_k + k;"),
    ("wgrad_token_mod", "int64_t token = indices[i] / top_k;\n        double dot",
     "int64_t token = indices[i] % top_k;\n        double dot"),
    ("wgrad_reversed_operand", "(double)load_elem(grad, dtype, token * H + h);",
     "(double)load_elem(grad, dtype, token * H + (H - 1 - h));"),
    ("wgrad_slot_by_position", "out[indices[i]] = (float)dot;", "out[i] = (float)dot;"),
    ("positions_not_inverse", "positions[indices[j]] = (int32_t)j;", "positions[j] = indices[j];"),
    ("compaction_descending",
     "for (int32_t e = 0; e < E; ++e) {\n            if (routing_map[t * E + e] != 0 && j < topk) {",
     "for (int32_t e = E - 1; e >= 0; --e) {\n            if (routing_map[t * E + e] != 0 && j < topk) {"),
    ("compaction_pad_zero", "indices[t * topk + j] = -1;", "indices[t * topk + j] = 0;"),
    ("compaction_keep_last", "if (routing_map[t * E + e] != 0 && j < topk) {",
     "if (routing_map[t * E + e] != 0 && (j < topk || (j = topk - 1) >= 0)) {"),
    ("compaction_bwd_slot_swap", "grad_probs[t * E + e] = grad_probs_indices[t * topk + j];",
     "grad_probs[t * E + e] = grad_probs_indices[t * topk + (topk - 1 - j)];"),
    ("bf16_round_half_up", "u += 0x7fffu + lsb;", "u += 0x8000u;"),
    ("gating_ties_to_higher_id", "if (best < 0 || v > bv) { best = e; bv = v; }",
     "if (best < 0 || v >= bv) { best = e; bv = v; }"),
    ("gating_sigmoid_sign", "score[e] = 1.0 / (1.0 + exp(-v));", "score[e] = 1.0 / (1.0 + exp(v));"),
    ("gating_no_normalize", "if (normalize) w = chosen_sum > 0.0 ? w / chosen_sum : 1.0 / top_k;",
     "if (normalize) w = chosen_sum > 0.0 ? w : 1.0 / top_k;"),
    ("gating_weight_of_slot", "double w = score[top_expert[t * top_k + k]];", "double w = score[k];"),
    ("gating_softmax_unscaled", "for (int32_t e = 0; e < E; ++e) score[e] /= z;",
     "for (int32_t e = 0; e < E; ++e) score[e] /= 1.0;"),
    ("wgather_weight_by_position", "float scaled = weights ? weights[a] * v : v;",
     "float scaled = weights ? weights[i] * v : v;"),
    ("wgather_unscaled", "float scaled = weights ? weights[a] * v : v;", "float scaled = weights ? v : v;"),
    ("wgather_token_mod", "int64_t a = indices[i];\n        int64_t token = a / top_k;",
     "int64_t a = indices[i];\n        int64_t token = a % top_k;"),
    ("check_ignores_positions", "} else if (positions && positions[a] != i) {", "} else if (0) {"),
    ("check_no_order", "if (i > 0 && bin_ids[i] == bin_ids[i - 1] && a <= indices[i - 1]) bits |= 2;", ""),
    ("check_no_end", "if (E > 0 && bins[E - 1] != n) bits |= 4;", ""),
]

_RUNNER = textwrap.dedent("""
    import json, sys
    sys.path.insert(0, %(root)r); sys.path.insert(0, %(tests)r)
    import oracle, pins
    caught = {}
    for name, path in json.loads(sys.argv[1]).items():
        lib = oracle.load(path)
        caught[name] = []
        for check in pins.ALL_CHECKS:
            try:
                check(lib)
            except (AssertionError, oracle.OracleError) as exc:
                caught[name].append(check.__name__)
    print(json.dumps(caught))
""")


def test_every_planted_mistake_is_caught(tmp_path):
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    libs = {}
    for name, old, new in MUTANTS:
        assert src.count(old) == 1, "mutation site for %s not unique" % name
        mpath = tmp_path / (name + ".c")
        mpath.write_text(src.replace(old, new))
        libs[name] = oracle.build(force=True, src=str(mpath), out=str(tmp_path / (name + ".so")))
    res = subprocess.run([sys.executable, "-c", _RUNNER % {"root": ROOT, "tests": HERE}, json.dumps(libs)],
                         capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stderr[-3000:]
    caught = json.loads(res.stdout.strip().splitlines()[-1])
    # every planted mistake must fail at least two independent pins
    weak = {k: v for k, v in caught.items() if len(v) < 2}
    assert not weak, "planted mistakes caught by fewer than two pins: %s" % weak
