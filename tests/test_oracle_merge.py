"""Pins of the attention-state merge.

"Deep Dive - FlashInfer", section "A worked split-KV example": chunk A
(o=[1,0], b=2) merged with chunk B (o=[0,1], b=1) gives [2/3, 1/3] and
2 + log2(1.5); empty states are the identity; 1e308 payloads do not overflow;
168 split/direct cases drawn with random.Random(7) agree to 1e-10; an
overlapping split turns 0.5 into 0.6667 and a natural-log producer turns
0.6667 into 0.6179.
"""
import json
import math
import os
import random

import numpy as np
import pytest

from oracle import ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
G = json.load(open(os.path.join(GOLDEN, "merge_state_example.json")))


def test_worked_merge():
    a, b = G["chunk_a"], G["chunk_b"]
    o, lse = ref.merge_state(a["o"], a["b"], b["o"], b["b"])
    assert abs(o[0] - 2 / 3) < 1e-12 and abs(o[1] - 1 / 3) < 1e-12
    assert abs(lse - (2 + math.log2(1.5))) < 1e-12
    assert [round(float(x), 4) for x in o] == G["printed_merged_o_4dp"]
    assert round(lse, 3) == G["printed_merged_b_3dp"]


def test_empty_states_are_identity():
    o, lse = ref.merge_state([1.0, 0.0], 2.0, [0.0, 1.0], 1.0)
    o2, lse2 = ref.merge_state([0.0, 0.0], -math.inf, o, lse)
    assert np.array_equal(o2, o) and lse2 == lse
    o3, lse3 = ref.merge_state(o, lse, [0.0, 0.0], -math.inf)
    assert np.array_equal(o3, o) and lse3 == lse
    o4, lse4 = ref.merge_state([0.0, 0.0], -math.inf, [0.0, 0.0], -math.inf)
    assert np.array_equal(o4, [0.0, 0.0]) and lse4 == -math.inf


def test_large_payload_does_not_overflow():
    o, _ = ref.merge_state([1e308], 0.0, [1e308], 0.0)
    assert o[0] == 1e308


@pytest.mark.parametrize("bad", [
    ([1.0], 0.0, [1.0, 2.0], 0.0),           # dimension mismatch
    ([], 0.0, [], 0.0),                      # empty vector
    ([math.nan], 0.0, [1.0], 0.0),           # non-finite payload
    ([1.0], math.inf, [1.0], 0.0),           # +inf statistic
    ([1.0], -math.inf, [1.0], 0.0),          # empty state with non-zero vector
])
def test_invalid_states_rejected(bad):
    with pytest.raises(ValueError):
        ref.merge_state(*bad)


def test_split_direct_sweep():
    sd = G["split_direct"]
    rng = random.Random(sd["seed"])
    cases = 0
    for length in sd["lengths"]:
        for offset in sd["offsets"]:
            scores = [offset + rng.uniform(*sd["score_uniform"]) for _ in range(length)]
            values = [[rng.uniform(*sd["value_uniform"]), rng.uniform(*sd["value_uniform"])]
                      for _ in scores]
            vals = np.array(values, dtype=np.float64).reshape(-1, 2)
            eo, eb = ref.direct_state(scores, vals)
            for cut in range(length + 1):
                left = ref.direct_state(scores[:cut], vals[:cut])
                right = ref.direct_state(scores[cut:], vals[cut:])
                o, b = ref.merge_state(*left, *right)
                assert np.max(np.abs(o - eo)) < sd["tolerance"]
                assert abs(b - eb) < sd["tolerance"]
                cases += 1
    assert cases == sd["printed_cases"]


def test_overlap_and_wrong_base_are_detected():
    scores, values = [0.0, 0.0], np.array([[1.0, 0.0], [0.0, 1.0]])
    whole = ref.direct_state(scores, values)
    assert abs(whole[0][0] - 0.5) < 1e-12
    dup = ref.merge_state(*whole, *ref.direct_state(scores[:1], values[:1]))
    assert round(float(dup[0][0]), 4) == G["printed_overlap_changes_0.5_to"]
    correct = ref.merge_state([1.0, 0.0], 2.0, [0.0, 1.0], 1.0)
    wrong = ref.merge_state([1.0, 0.0], 2 * math.log(2), [0.0, 1.0], math.log(2))
    assert abs(wrong[0][0] - correct[0][0]) > 0.04
    assert round(float(wrong[0][0]), 4) == G["printed_wrong_base_changes_0.6667_to"]


def test_direct_state_lse_closed_form():
    # constant scores s over n keys: lse2 = s / ln 2 + log2(n), output = mean of values
    for s, n in ((0.0, 1), (3.5, 7), (-20.0, 33)):
        vals = np.arange(2 * n, dtype=np.float64).reshape(n, 2)
        o, b = ref.direct_state([s] * n, vals)
        assert abs(b - (s / math.log(2) + math.log2(n))) < 1e-12
        assert np.allclose(o, vals.mean(axis=0), atol=1e-12)


def test_multiway_fold_equals_direct():
    rng = np.random.default_rng(3)
    s = rng.normal(size=40) * 3
    v = rng.normal(size=(40, 5))
    eo, eb = ref.direct_state(s, v)
    cuts = [0, 3, 3, 17, 18, 40]  # includes an empty chunk
    states = [ref.direct_state(s[a:b], v[a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
    o, b = ref.merge_states(states)
    assert np.max(np.abs(o - eo)) < 1e-12 and abs(b - eb) < 1e-12
