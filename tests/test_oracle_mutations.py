"""Plant plausible mistakes in copies of the oracle and show that a pin catches each.

Every mutation is applied to a fresh copy of the oracle module (on the CPU); the
real oracle is never modified.
"""
import inspect
import types

import pytest

from oracle import hashattn_oracle as O
import oracle_pins as P

SOURCE = inspect.getsource(O)

# (name, text in the oracle source, replacement)
MUTATIONS = [
    ("popcount_drops_bit31", "for j in range(32):", "for j in range(31):"),
    ("distance_and_not_xor", "return popcount32(k ^ q)", "return popcount32(k & q)"),
    ("keeps_largest_distance", "order = np.lexsort((np.arange(n), dist))",
     "order = np.lexsort((np.arange(n), -dist))"),
    ("tie_break_index_descending", "order = np.lexsort((np.arange(n), dist))",
     "order = np.lexsort((-np.arange(n), dist))"),
    ("budget_off_by_one", "k = max(0, min(int(m), n))", "k = max(0, min(int(m), n) - 1)"),
    ("local_window_off_by_one", "local = np.arange(max(0, n - int(n_local)), n, dtype=np.int64)",
     "local = np.arange(max(0, n - int(n_local) + 1), n, dtype=np.int64)"),
    ("sink_not_clamped", "sink = np.arange(0, max(0, min(int(n_sink), n)), dtype=np.int64)",
     "sink = np.arange(0, int(n_sink), dtype=np.int64)"),
    ("intersection_not_union", "return np.union1d(top, win).astype(np.int64)",
     "return np.intersect1d(top, win).astype(np.int64)"),
    ("windows_dropped", "    win = window_positions(n, n_sink, n_local)\n    if exclusive:",
     "    win = np.zeros(0, dtype=np.int64)\n    if exclusive:"),
    ("exclusive_ignores_windows", "top = outside[top_m_by_score(dist[outside], m)]", "top = top_m_by_score(dist, m)"),
    ("per_head_budget_ignored", "            mb = int(m_per_head[b, h])", "            mb = mb"),
    ("missing_sqrt_d_scale", "z = k_rows @ q / math.sqrt(d)", "z = k_rows @ q"),
    ("scale_by_d", "z = k_rows @ q / math.sqrt(d)", "z = k_rows @ q / d"),
    ("lse_drops_max", "lse = z_max + math.log(total)", "lse = math.log(total)"),
    ("values_from_keys", "out = (w / total) @ v_rows", "out = (w / total) @ k_rows"),
    ("unnormalised_output", "out = (w / total) @ v_rows", "out = w @ v_rows"),
    ("merge_weights_swapped", "out = (wa * out_a + wb * out_b) / (wa + wb)",
     "out = (wb * out_a + wa * out_b) / (wa + wb)"),
    ("merge_lse_is_max", "return out, top + math.log(wa + wb)", "return out, top"),
    ("gate_sign_flipped", "g = 1.0 / (1.0 + math.exp(-(lse_a - lse_loc)))",
     "g = 1.0 / (1.0 + math.exp(lse_a - lse_loc))"),
    ("gqa_head_modulo", "g = h // G", "g = h % Hkv"),
    ("merge_segments_mean_not_mass", "merged = sum(m_s * outs[s] for m_s, s in zip(mass, live)) / norm",
     "merged = sum(outs[s] for s in live) / len(live)"),
    ("merge_segments_lse_without_peak", "return merged, peak + math.log(norm)", "return merged, math.log(norm)"),
    ("exact_topm_smallest_scores", "order = np.lexsort((np.arange(n), -z))  # score descending",
     "order = np.lexsort((np.arange(n), z))  # score descending"),
    ("exact_topm_ties_to_larger_index", "order = np.lexsort((np.arange(n), -z))  # score descending",
     "order = np.lexsort((-np.arange(n), -z))  # score descending"),
    ("recall_over_selected", "    return hit / ref.size", "    return hit / max(1, np.unique(np.asarray(selected)).size)"),
    ("wide_distance_first_word_only", "    return popcount32(k ^ q).sum(axis=1)", "    return popcount32(k ^ q)[:, 0]"),
    ("encode_zero_sets_bit", "        if proj[j] > 0.0:", "        if proj[j] >= 0.0:"),
    ("encode_bit_order_reversed", "            code |= 1 << j", "            code |= 1 << (31 - j)"),
    ("mlp_first_relu_dropped", "h1 = np.maximum(np.asarray(W1, np.float64) @ x + np.asarray(b1, np.float64), 0.0)",
     "h1 = np.asarray(W1, np.float64) @ x + np.asarray(b1, np.float64)"),
    ("mlp_second_relu_dropped", "h2 = np.maximum(np.asarray(W2, np.float64) @ h1 + np.asarray(b2, np.float64), 0.0)",
     "h2 = np.asarray(W2, np.float64) @ h1 + np.asarray(b2, np.float64)"),
    ("mlp_second_bias_dropped", "@ h1 + np.asarray(b2, np.float64), 0.0)", "@ h1, 0.0)"),
    ("mlp_second_layer_transposed", "np.asarray(W2, np.float64) @ h1", "np.asarray(W2, np.float64).T @ h1"),
    ("mlp_zero_sets_bit", "        if f[j] > 0.0:", "        if f[j] >= 0.0:"),
    ("encode_transposed_projection", "proj = np.asarray(W, dtype=np.float64) @ np.asarray(x, dtype=np.float64)",
     "proj = np.asarray(x, dtype=np.float64) @ np.asarray(W, dtype=np.float64)[:, :1].repeat(32, axis=1)"),
]


def _mutant(old, new):
    assert SOURCE.count(old) >= 1, old
    mod = types.ModuleType("oracle_mutant")
    exec(compile(SOURCE.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


def test_real_oracle_passes_every_pin():
    assert P.failing_checks(O) == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(name, old, new):
    bad = P.failing_checks(_mutant(old, new))
    assert bad, f"no pin caught the planted mistake {name}"
