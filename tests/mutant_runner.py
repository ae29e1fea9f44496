"""Runs the oracle pins against one mutant oracle library (a subprocess of
tests/test_oracle_mutants.py) and prints the names of the pins that failed,
as JSON, on the last line of stdout."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from oracle.oracle import Oracle  # noqa: E402
from tests import test_oracle_pins as pins  # noqa: E402

CHECKS = [
    ("routing_golden", lambda o: pins.test_routing_golden_cases(o)),
    ("all_equal_renorm", lambda o: pins.test_all_equal_logits_closed_form(o, True)),
    ("all_equal_no_renorm", lambda o: pins.test_all_equal_logits_closed_form(o, False)),
    ("two_expert_sigmoid", lambda o: pins.test_two_expert_sigmoid_closed_form(o)),
    ("nan_ranks_last", lambda o: pins.test_nan_ranks_last(o)),
    ("topk_vs_sort", lambda o: pins.test_topk_matches_library_sort_and_softmax(o, "coarse", 64, 6)),
    ("dispatch_vs_argsort", lambda o: pins.test_dispatch_matches_stable_argsort(o, 333, 64, 6)),
    ("swiglu_golden", lambda o: pins.test_swiglu_golden(o)),
    ("logits_vs_matmul", lambda o: pins.test_logits_match_float64_matmul(o)),
    ("dense_mlp_E1", lambda o: pins.test_dense_mlp_when_one_expert(o)),
    ("soft_mixture_kE", lambda o: pins.test_soft_mixture_when_k_equals_E(o)),
    ("brute_force", lambda o: pins.test_brute_force_tiny_layer(o, False)),
    ("brute_force_bias", lambda o: pins.test_brute_force_tiny_layer(o, True)),
    ("token_outputs_rows", lambda o: pins.test_token_outputs_equal_forward_rows(o)),
    ("input_scaled_dense", lambda o: pins.test_input_scaled_equals_dense_no_dispatch(o, 6, 2, True)),
    ("input_scaled_kE", lambda o: pins.test_input_scaled_equals_dense_no_dispatch(o, 6, 6, False)),
    ("input_scaled_one_expert", lambda o: pins.test_input_scaled_single_expert_is_plain_mlp(o)),
    ("combine_one_hot", lambda o: pins.test_combine_one_hot_rows(o, False)),
    ("combine_one_hot_scaled", lambda o: pins.test_combine_one_hot_rows(o, True)),
    ("combine_vs_einsum", lambda o: pins.test_combine_matches_einsum_on_random_rows(o)),
    ("ffn_rows", lambda o: pins.test_expert_ffn_rows_equal_single_rows(o)),
]

if __name__ == "__main__":
    o = Oracle(sys.argv[1])
    failed = []
    for name, check in CHECKS:
        try:
            check(o)
        except AssertionError:
            failed.append(name)
    print(json.dumps(failed))
