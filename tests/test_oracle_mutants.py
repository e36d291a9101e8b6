"""The oracle's pins catch planted mistakes.

Each case plants one plausible mistake in the oracle (a dropped scale, a log2 LSE, an
off-by-one KV chunk, transposed operands, a merge that drops a chunk or keeps only the
max, a flipped sign on D, swapped dK/dV, unnormalised P), by wrapping the oracle's own
function on the CPU, and requires that every pin named for it then fails.  A pin that
still passed would not be pinning what it claims to.
"""
import dataclasses
import math

import numpy as np
import pytest

import oracle
from tests import test_oracle as pins

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

FWD, MERGE, DQ, DKDV = oracle.forward, oracle.merge, oracle.backward_dq, oracle.backward_dkdv


def _shorter(item):
    if item.kv_hi <= item.kv_lo:
        return item
    return dataclasses.replace(item, kv_hi=item.kv_hi - 1)


def fwd_no_scale(q, k, v, item, scale, rows=None):
    return FWD(q, k, v, item, 1.0, rows)


def fwd_log2(q, k, v, item, scale, rows=None):
    O, L = FWD(q, k, v, item, scale, rows)
    return O, L / math.log(2.0)


def fwd_short_chunk(q, k, v, item, scale, rows=None):
    return FWD(q, k, v, _shorter(item), scale, rows)


def fwd_swapped_kv(q, k, v, item, scale, rows=None):
    return FWD(q, v, k, item, scale, rows)


def merge_drops_last(parts):
    return MERGE(parts[:-1]) if len(parts) > 1 else MERGE(parts)


def merge_lse_is_max(parts):
    O, _ = MERGE(parts)
    return O, np.stack([p[1] for p in parts]).max(axis=0)


def dq_flipped_d(q, k, v, do_rows, o_rows, lse_rows, item, scale, rows):
    return DQ(q, k, v, do_rows, -np.asarray(o_rows), lse_rows, item, scale, rows)


def dq_no_scale(q, k, v, do_rows, o_rows, lse_rows, item, scale, rows):
    return DQ(q, k, v, do_rows, o_rows, lse_rows, item, scale, rows) / scale


def dkdv_swapped(q, k, v, do_all, o_all, lse_all, item, scale, kv_rows=None):
    dK, dV = DKDV(q, k, v, do_all, o_all, lse_all, item, scale, kv_rows)
    return dV, dK


def dkdv_flipped_d(q, k, v, do_all, o_all, lse_all, item, scale, kv_rows=None):
    return DKDV(q, k, v, do_all, -np.asarray(o_all), lse_all, item, scale, kv_rows)


def prob_unnormalised(q, k, item, h, scale, rows=None):
    rows = np.arange(item.q_lo, item.q_hi) if rows is None else np.asarray(rows)
    S = oracle.scores(q, k, item, h, rows, scale)
    return np.exp(S - S.max(axis=1, keepdims=True))


FD = pins.test_gradients_match_central_differences
GOLDEN = pins.test_golden_worked_example
MERGE_PIN = pins.test_merge_of_any_k_split_equals_unsplit

CASES = {
    "forward drops the scale": ("forward", fwd_no_scale, [
        (pins.test_forward_matches_brute_force_tiny_mixed,), (GOLDEN, "worked_example_scale2.json"),
        (pins.test_matches_torch_sdpa_float64_with_autograd,)]),
    "forward LSE in log2": ("forward", fwd_log2, [
        (pins.test_forward_matches_brute_force_tiny_mixed,), (GOLDEN, "worked_example.json"),
        (pins.test_zero_query_gives_mean_and_log_count,)]),
    "forward KV chunk one short": ("forward", fwd_short_chunk, [
        (pins.test_forward_matches_brute_force_tiny_mixed,), (pins.test_single_key_gives_that_value,),
        (pins.test_zero_query_gives_mean_and_log_count,)]),
    "forward with K and V transposed": ("forward", fwd_swapped_kv, [
        (pins.test_forward_matches_brute_force_tiny_mixed,), (GOLDEN, "worked_example.json")]),
    "merge drops the last chunk": ("merge", merge_drops_last, [
        (MERGE_PIN, [0, 128, 256]), (MERGE_PIN, [0, 1, 255, 256]),
        (pins.test_forward_matches_brute_force_tiny_mixed,)]),
    "merge keeps only the max as LSE": ("merge", merge_lse_is_max, [
        (MERGE_PIN, [0, 128, 256]), (pins.test_forward_matches_brute_force_tiny_mixed,)]),
    "dQ with the sign of D flipped": ("backward_dq", dq_flipped_d, [
        (FD, "whole"), (FD, "ksplit"), (GOLDEN, "worked_example.json"),
        (pins.test_matches_torch_sdpa_float64_with_autograd,)]),
    "dQ without the scale": ("backward_dq", dq_no_scale, [
        (FD, "qsplit"), (GOLDEN, "worked_example_scale2.json")]),
    "dK and dV swapped": ("backward_dkdv", dkdv_swapped, [
        (FD, "whole"), (pins.test_gradient_sums_over_whole_item,), (GOLDEN, "worked_example.json")]),
    "dK/dV with the sign of D flipped": ("backward_dkdv", dkdv_flipped_d, [
        (FD, "hsplit"), (pins.test_gradient_sums_over_whole_item,),
        (pins.test_matches_torch_sdpa_float64_with_autograd,)]),
    "P not normalised": ("probabilities", prob_unnormalised, [
        (pins.test_probability_rows_sum_to_one,)]),
}


@pytest.mark.parametrize("name", list(CASES))
def test_pins_catch_planted_mistake(name, monkeypatch):
    attr, mutant, catchers = CASES[name]
    monkeypatch.setattr(oracle, attr, mutant)
    for pin, *args in catchers:
        with pytest.raises(AssertionError):
            pin(*args)


def test_pins_pass_on_the_oracle_itself():
    # the same pins with nothing planted (the control)
    for _, _, catchers in CASES.values():
        for pin, *args in catchers:
            pin(*args)
