"""Writes oracle_regression_tiny.json: the oracle's outputs on one small seeded stream.

Calls only ``oracle/`` and the seeded input generator.  The stored values pin the
oracle against unintended changes of its arithmetic: a later change to the oracle that
alters them must say, in its commit message, which passage of the pages justifies it.
Run from the repository root:  python tests/golden/make_oracle_regression.py
"""

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import sdm_inputs  # noqa: E402

T = 6
SAMPLE_ROWS = 6


def build() -> dict:
    cfg = sdm_inputs.CONFIGS["tiny"].replace(B=1, H=1, T=T)
    d = sdm_inputs.make_inputs(cfg)
    out = oracle.sdm_write_read(d["q_w"], d["q_r"], d["k_val"], d["gates"], d["subkeys"], d["bank_init"],
                                factor_dims=cfg.factor_dims, W=cfg.W, R=cfg.R,
                                act_dtype=cfg.act_dtype, bank_dtype=cfg.bank_dtype)[(0, 0)]
    rows = sorted(set(int(i) for i in out["idx_w"].ravel()))[:SAMPLE_ROWS]
    hexs = lambda a: [float(x).hex() for x in np.asarray(a, np.float64).ravel()]
    return {
        "config": {"name": cfg.name, "B": 1, "H": 1, "T": T, "seed": cfg.seed},
        "idx_w": out["idx_w"].tolist(), "idx_r": out["idx_r"].tolist(),
        "wt_w": hexs(out["wt_w"]), "wt_r": hexs(out["wt_r"]),
        "y": hexs(out["y"]),
        "bank_rows": rows, "bank_sample": hexs(out["bank"][rows]),
    }


if __name__ == "__main__":
    path = os.path.join(HERE, "oracle_regression_tiny.json")
    with open(path, "w") as f:
        json.dump(build(), f, indent=0)
    print(path)
