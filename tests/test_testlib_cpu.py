"""The parity rules of sdm_testlib, exercised on the CPU with the oracle standing in for
the GPU: its own outputs pass, a planted error fails, and a different valid pick at an
exact tie is followed to the end of the stream (y and the final bank still compared)."""

import numpy as np
import pytest
import torch

import oracle
import sdm_inputs
from sdm_inputs import CONFIGS
from sdm_testlib import compare_stream


def _as_gpu(cfg, d, out):
    """Oracle outputs of every stream laid out like gpu_write_read's CPU tensors."""
    B, T, H = cfg.B, d["q_w"].shape[1], cfg.H
    act = torch.float32 if cfg.act_dtype == "f32" else torch.bfloat16
    g = {"y": torch.zeros(B, T, H, cfg.d_v, dtype=act), "bank": torch.zeros(B, H, cfg.N, cfg.d_v),
         "idx_w": torch.zeros(B, T, H, cfg.W, dtype=torch.int32), "wt_w": torch.zeros(B, T, H, cfg.W),
         "idx_r": torch.zeros(B, T, H, cfg.R, dtype=torch.int32), "wt_r": torch.zeros(B, T, H, cfg.R)}
    for (b, h), o in out.items():
        g["y"][b, :, h] = torch.from_numpy(o["y"]).to(act)
        g["bank"][b, h] = torch.from_numpy(o["bank"]).float()
        for k in ("idx_w", "idx_r"):
            g[k][b, :, h] = torch.from_numpy(o[k]).int()
        for k in ("wt_w", "wt_r"):
            g[k][b, :, h] = torch.from_numpy(o[k]).float()
    return g


def _run(cfg, d):
    return oracle.sdm_write_read(d["q_w"], d["q_r"], d["k_val"], d["gates"], d["subkeys"], d["bank_init"],
                                 factor_dims=cfg.factor_dims, W=cfg.W, R=cfg.R, act_dtype=cfg.act_dtype,
                                 bank_dtype=cfg.bank_dtype)


def test_oracle_outputs_pass_the_parity_rules():
    cfg = CONFIGS["tiny"].replace(T=24, H=2)
    d = sdm_inputs.make_inputs(cfg)
    g = _as_gpu(cfg, d, _run(cfg, d))
    for h in range(cfg.H):
        r = compare_stream(cfg, d, g, 0, h)
        assert r == {"rows": cfg.T, "near_ties": 0, "near_tie_tokens": []}


def test_a_planted_error_in_y_or_the_bank_fails():
    cfg = CONFIGS["tiny"].replace(T=24)
    d = sdm_inputs.make_inputs(cfg)
    g = _as_gpu(cfg, d, _run(cfg, d))
    g["y"][0, 20, 0, 3] += 1e-3
    with pytest.raises(AssertionError, match="y"):
        compare_stream(cfg, d, g, 0, 0)
    g = _as_gpu(cfg, d, _run(cfg, d))
    g["bank"][0, 0, 7, 1] += 1e-3
    with pytest.raises(AssertionError, match="bank"):
        compare_stream(cfg, d, g, 0, 0)


def test_a_different_pick_with_a_clear_margin_fails():
    cfg = CONFIGS["tiny"].replace(T=8)
    d = sdm_inputs.make_inputs(cfg)
    g = _as_gpu(cfg, d, _run(cfg, d))
    sel = g["idx_w"][0, 3, 0].clone()
    outside = next(n for n in range(cfg.N) if n not in set(sel.tolist()))
    g["idx_w"][0, 3, 0, -1] = outside
    with pytest.raises(AssertionError):
        compare_stream(cfg, d, g, 0, 0)


def test_a_valid_pick_at_an_exact_tie_is_followed_to_the_end():
    # two sub-keys of the first factor made identical: slots (a, x) and (a', x) score the
    # same, so swapping the k-th write slot for its tied twin is another valid top-k;
    # the "GPU" below took that pick at token 2 and ran on from it
    cfg = CONFIGS["tiny"].replace(T=10, W=4, R=4)
    d = sdm_inputs.make_inputs(cfg)
    K = d["subkeys"][0].double().numpy()
    t = 2
    q = d["q_w"][0, t, 0].double().numpy()
    idx, _, _ = oracle.select(q, K, cfg.factor_dims, cfg.d_sub, cfg.W)
    a, x = divmod(int(idx[-1]), cfg.factor_dims[1])
    sel_a = {int(s) // cfg.factor_dims[1] for s in idx}
    twin = next(i for i in range(cfg.factor_dims[0]) if i not in sel_a)
    d["subkeys"][0, twin] = d["subkeys"][0, a]
    idx, _, _ = oracle.select(d["q_w"][0, t, 0].double().numpy(), d["subkeys"][0].double().numpy(),
                              cfg.factor_dims, cfg.d_sub, cfg.W)
    last = int(idx[-1])
    a, x = divmod(last, cfg.factor_dims[1])
    other = (twin if a != twin else int(idx[-1]) // cfg.factor_dims[1]) * cfg.factor_dims[1] + x
    assert other not in set(idx.tolist())

    def follow(tt, which, i, w):
        if tt == t and which == 0:
            return np.concatenate([i[:-1], [other]])
        return None

    M = d["bank_init"][0].double().numpy().copy()
    o = oracle.run_stream(M, d["q_w"][0, :, 0].double().numpy(), d["q_r"][0, :, 0].double().numpy(),
                          d["k_val"][0, :, 0].double().numpy(), d["gates"][0, :, 0].double().numpy(),
                          d["subkeys"][0].double().numpy(), factor_dims=cfg.factor_dims, d_sub=cfg.d_sub,
                          W=cfg.W, R=cfg.R, act_dtype=cfg.act_dtype, bank_dtype=cfg.bank_dtype, pick=follow)
    o["bank"] = M
    g = _as_gpu(cfg, d, {(0, 0): o})
    r = compare_stream(cfg, d, g, 0, 0)
    assert r["rows"] == cfg.T and r["near_ties"] == 1 and r["near_tie_tokens"] == [t]
    # and the history after the pick really differs from the oracle's own
    own = _run(cfg, d)[(0, 0)]
    assert not np.allclose(own["bank"], M)
