"""Step 1 on its own: the GPU's factor scores against the oracle's correctly rounded ones.

The oracle's score s* is the float64 dot product rounded once to float32
(oracle.factor_scores).  The GPU's scorers meet it within stated bounds, with u = 2^-24
(half an ulp of 1 in float32) and A = sum_d |q_d| |k_d| (the scale of every rounding
inside a dot product):

  * tensor cores, bfloat16 inputs: the products are exact; the float32 accumulator of
    d_sub/16 MMA steps rounds (or truncates) at most once per step, so
        |s - s*| <= (d_sub/16 + 1) * 2u * A;
  * tensor cores, float32 inputs (the error-free fixed-point split into four 8-bit
    slices per value): every level sum is exact for d_sub <= 128, so s is the correctly
    rounded value of the dot product less a truncation below
    tau = 2^-29 * d_sub * max_d |q_d| * max_d |k_d|, and
        |s - s*| <= 2u * |s*| + 2 tau   (+ (d_sub/16) * 2u * A when d_sub > 128),
    and at these sizes at least 90% of the scores equal the oracle's bit for bit;
  * CUDA cores (forced by the test hook), float32 inputs, compensated sums:
        |s - s*| <= 2u * |s*| + 64u^2 * A;
    bfloat16 inputs, plain float32 sums over blocks of 32 terms folded into a
    compensated total:
        |s - s*| <= 2u * |s*| + 32u * A.

On grid-valued inputs (sdm_inputs, grid=True) every score is exact in float32, so the
GPU's must equal the oracle's bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
import sdm_inputs
from sdm_inputs import CONFIGS

pytestmark = pytest.mark.gpu

U = 2.0 ** -24

# (name, config overrides): shapes that exercise the split's zero padding (d_sub = 32, 40),
# scalar loads (d_sub % 8 != 0), ragged token tiles (B*T not a multiple of 128), several N
# tiles per factor (n_f = 256 > 128 for the split path), unequal factors and the ring of
# k blocks (d_sub = 512).
SHAPES = {
    "tiny": ("tiny", dict(T=200)),
    "three_factor": ("three_factor", dict(T=256, H=2)),
    "layer_f32": ("layer", dict(B=1, T=130, d_v=64, act_dtype="f32")),
    "ragged_d_sub": ("tiny", dict(B=2, T=77, H=3, factor_dims=(16, 48), d_sub=40)),
    "layer_bf16": ("layer", dict(B=1, T=130, d_v=64)),
}


@pytest.fixture(scope="module")
def sdm():
    import gated_delta_rule_factor_gb300 as m
    yield m
    m.test_force_simt_scorer(False)


def _gpu_scores(sdm, cfg, d):
    q_w, q_r, sk = (d[k].cuda() for k in ("q_w", "q_r", "subkeys"))
    s = sdm.test_factor_scores(q_w, q_r, sk, factor_dims=cfg.factor_dims)
    torch.cuda.synchronize()
    return s.cpu().numpy().astype(np.float64)


def _oracle_scores(cfg, d):
    """oracle.factor_scores of every row; A = |q| . |k| and max|q_f| * max|k| of every
    score (float64)."""
    B, T, H = d["q_w"].shape[:3]
    ntot = sum(cfg.factor_dims)
    want = np.zeros((2, B * T * H, ntot))
    scale = np.zeros((2, B * T * H, ntot))
    peak = np.zeros((2, B * T * H, ntot))
    K = [d["subkeys"][h].double().numpy() for h in range(H)]
    kmax = [np.abs(k).max(axis=1) for k in K]
    for qsel, name in enumerate(("q_w", "q_r")):
        Q = d[name].double().numpy()
        for b in range(B):
            for t in range(T):
                for h in range(H):
                    r = (b * T + t) * H + h
                    q = Q[b, t, h]
                    want[qsel, r] = np.concatenate(oracle.factor_scores(q, K[h], cfg.factor_dims, cfg.d_sub))
                    off = 0
                    for f, n in enumerate(cfg.factor_dims):
                        qf = np.abs(q[f * cfg.d_sub:(f + 1) * cfg.d_sub])
                        scale[qsel, r, off:off + n] = np.abs(K[h][off:off + n]) @ qf
                        peak[qsel, r, off:off + n] = qf.max() * kmax[h][off:off + n]
                        off += n
    return want, scale, peak


def _bound(cfg, tensor_cores, want, scale, peak):
    if not tensor_cores:
        return 2 * U * np.abs(want) + (32 * U if cfg.act_dtype == "bf16" else 64 * U * U) * scale
    if cfg.act_dtype == "bf16":
        return (-(-cfg.d_sub // 16) + 1) * 2 * U * scale
    tau = 2.0 ** -29 * cfg.d_sub * peak
    extra = (cfg.d_sub // 16) * 2 * U * scale if cfg.d_sub > 128 else 0.0
    return 2 * U * np.abs(want) + 2 * tau + extra


@pytest.mark.parametrize("name", sorted(SHAPES))
@pytest.mark.parametrize("scorer", ["tensor_cores", "cuda_cores"])
def test_factor_scores_within_the_stated_bound(sdm, name, scorer):
    base, over = SHAPES[name]
    cfg = CONFIGS[base].replace(**over)
    d = sdm_inputs.make_inputs(cfg)
    sdm.test_force_simt_scorer(scorer == "cuda_cores")
    try:
        got = _gpu_scores(sdm, cfg, d)
    finally:
        sdm.test_force_simt_scorer(False)
    want, scale, peak = _oracle_scores(cfg, d)
    err = np.abs(got - want)
    bound = _bound(cfg, scorer == "tensor_cores", want, scale, peak)
    worst = float(np.max(err / (U * scale)))
    exact = float(np.mean(err == 0))
    print(f"{name}/{scorer}: max |s - s*| = {err.max():.3g}, max |s - s*| / (u A) = {worst:.3g}, "
          f"bitwise equal {exact:.5f}")
    bad = err > bound
    assert not bad.any(), (f"{int(bad.sum())}/{err.size} scores beyond the bound; worst "
                           f"{float(np.max(err - bound)):.3g} past it")
    if scorer == "tensor_cores" and cfg.act_dtype == "f32" and cfg.d_sub <= 128:
        assert exact >= 0.9, exact


@pytest.mark.parametrize("name", ["three_factor", "tiny", "layer_bf16", "layer_f32"])
def test_grid_scores_are_exact(sdm, name):
    base, over = SHAPES[name]
    cfg = CONFIGS[base].replace(**over)
    d = sdm_inputs.make_inputs(cfg, grid=True)
    got = _gpu_scores(sdm, cfg, d)
    want = _oracle_scores(cfg, d)[0]
    np.testing.assert_array_equal(got, want)


def test_factor_scores_refusals(sdm):
    cfg = CONFIGS["tiny"]
    d = sdm_inputs.make_inputs(cfg)
    q_w, q_r, sk = (d[k].cuda() for k in ("q_w", "q_r", "subkeys"))
    with pytest.raises(sdm.SdmError):
        sdm.test_factor_scores(q_w, q_r, sk, factor_dims=cfg.factor_dims,
                               workspace=torch.empty(64, dtype=torch.uint8, device="cuda"))
