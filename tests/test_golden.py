"""Checks against the stored fixtures under tests/golden/.

  * tie_rule_examples.json: selection orders worked by hand from the tie rule of the
    sparse-delta-memory CHANGELOG (2.0.0 > Upgrading from v1); the oracle must give them.
  * oracle_regression_tiny.json: the oracle's outputs on one small seeded stream, written
    by tests/golden/make_oracle_regression.py (which calls only the oracle); any change
    of the oracle's arithmetic shows here.
"""

import json
import os

import numpy as np

import oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


def test_tie_rule_examples_worked_by_hand():
    fx = _load("tie_rule_examples.json")
    assert fx["examples"]
    for ex in fx["examples"]:
        s_list = [np.asarray(s, np.float32) for s in ex["factor_scores"]]
        ranks = [oracle.factor_ranks(s) for s in s_list]
        assert [list(r) for r in ranks] == ex["factor_ranks"], ex["name"]
        S = oracle.slot_scores(s_list)
        order = [int(i) for i in oracle.topk_slots(S, ranks, ex["k"], prefilter=False)]
        assert order == ex["expected_order"], ex["name"]


def test_oracle_reproduces_its_stored_outputs():
    import sys
    sys.path.insert(0, HERE)
    import make_oracle_regression as gen
    stored = _load("oracle_regression_tiny.json")
    fresh = json.loads(json.dumps(gen.build()))
    for k in ("config", "idx_w", "idx_r", "wt_w", "wt_r", "y", "bank_rows", "bank_sample"):
        assert fresh[k] == stored[k], k
