"""Pins of the oracle's backward (oracle/sdm_backward.py) against facts that do not come
from the backward itself.

  * Central finite differences of the oracle's forward (run in float64 with float64
    scores, so that only the arithmetic is differentiated): the directional derivative
    of L = <c_y, y> + <c_M, final bank> along a random direction of each input matches
    <gradient, direction>.  A dropped term, a wrong sign, a transposed operand or a
    gradient sent to the wrong slot fails this.
  * Closed forms: with alpha = 1, beta = 0 the bank gradient is the read's scatter of
    r_j dy plus the final-bank gradient, the value and write-query gradients are zero
    and the beta gradient is sum_j w_j <G_j, v - p>; a single full-strength write
    (W = 1, beta = 1) passes the whole row gradient to its value and none to the row
    before it.
  * The reverse sweep restores the bank exactly from the snapshots.
"""

import numpy as np
import pytest

from oracle import sdm_backward as bwd
from oracle import sdm_oracle as fwd_oracle


def _problem(seed, factor_dims=(6, 7), d_sub=4, d_v=5, T=6, W=3, R=4, spread=2.0):
    rng = np.random.default_rng(seed)
    N = int(np.prod(factor_dims))
    F = len(factor_dims)
    return {
        "factor_dims": factor_dims, "d_sub": d_sub, "W": W, "R": R,
        "q_w": rng.normal(0, spread, (T, F * d_sub)), "q_r": rng.normal(0, spread, (T, F * d_sub)),
        "k_val": rng.normal(0, 1, (T, d_v)),
        "gates": np.stack([rng.uniform(0.3, 0.95, T), rng.uniform(0.2, 0.9, T)], axis=1),
        "subkeys": rng.normal(0, 1 / np.sqrt(d_sub), (sum(factor_dims), d_sub)),
        "bank": rng.normal(0, 0.5, (N, d_v)),
        "c_y": rng.normal(0, 1, (T, d_v)), "c_M": rng.normal(0, 1, (N, d_v)),
    }


def _loss(p, **over):
    x = dict(p, **over)
    M = x["bank"].copy()
    out = bwd.stream_forward(M, x["q_w"], x["q_r"], x["k_val"], x["gates"], x["subkeys"],
                             factor_dims=x["factor_dims"], d_sub=x["d_sub"], W=x["W"], R=x["R"],
                             act_dtype="f64", bank_dtype="f64", exact=True)
    sel = [(r["w"]["idx"].tolist(), r["r"]["idx"].tolist()) for r in out["rec"]]
    return float(np.sum(p["c_y"] * out["y"]) + np.sum(p["c_M"] * M)), sel


def _grads(p):
    M = p["bank"].copy()
    out = bwd.stream_forward(M, p["q_w"], p["q_r"], p["k_val"], p["gates"], p["subkeys"],
                             factor_dims=p["factor_dims"], d_sub=p["d_sub"], W=p["W"], R=p["R"],
                             act_dtype="f64", bank_dtype="f64", exact=True)
    g = bwd.stream_backward(M, out, p["c_y"], p["c_M"], p["q_w"], p["q_r"], p["k_val"], p["gates"],
                            p["subkeys"], factor_dims=p["factor_dims"], d_sub=p["d_sub"])
    return g, M


INPUTS = ["bank", "k_val", "gates", "q_w", "q_r", "subkeys"]


@pytest.mark.parametrize("seed,factor_dims", [(1, (6, 7)), (2, (6, 7)), (3, (4, 3, 5))])
def test_gradients_match_central_differences(seed, factor_dims):
    p = _problem(seed, factor_dims=factor_dims)
    g, _ = _grads(p)
    rng = np.random.default_rng(100 + seed)
    _, sel0 = _loss(p)
    for name in INPUTS:
        d = rng.normal(0, 1, p[name].shape)
        eps = 1e-6
        lp, selp = _loss(p, **{name: p[name] + eps * d})
        lm, selm = _loss(p, **{name: p[name] - eps * d})
        assert selp == sel0 and selm == sel0, f"{name}: selection moved under the perturbation"
        fd = (lp - lm) / (2 * eps)
        an = float(np.sum(g[name] * d))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, fd, an)


def test_each_gradient_is_nonzero_somewhere():
    # guards the finite-difference test against a vacuous pass
    g, _ = _grads(_problem(1))
    for name in INPUTS:
        assert np.abs(g[name]).max() > 1e-3, name


def test_reverse_sweep_restores_the_bank_exactly():
    p = _problem(4)
    _, M = _grads(p)
    assert np.array_equal(M, p["bank"])
    # also through the rounded (float32 bank) forward used for parity
    M = p["bank"].astype(np.float32).astype(np.float64)
    start = M.copy()
    out = bwd.stream_forward(M, p["q_w"], p["q_r"], p["k_val"], p["gates"], p["subkeys"],
                             factor_dims=p["factor_dims"], d_sub=p["d_sub"], W=p["W"], R=p["R"])
    assert not np.array_equal(M, start)
    bwd.stream_backward(M, out, p["c_y"], p["c_M"], p["q_w"], p["q_r"], p["k_val"], p["gates"],
                        p["subkeys"], factor_dims=p["factor_dims"], d_sub=p["d_sub"])
    assert np.array_equal(M, start)


def test_recording_forward_is_the_oracle_forward():
    p = _problem(5)
    M1 = p["bank"].astype(np.float32).astype(np.float64)
    M2 = M1.copy()
    a = bwd.stream_forward(M1, p["q_w"], p["q_r"], p["k_val"], p["gates"], p["subkeys"],
                           factor_dims=p["factor_dims"], d_sub=p["d_sub"], W=p["W"], R=p["R"])
    b = fwd_oracle.run_stream(M2, p["q_w"], p["q_r"], p["k_val"], p["gates"], p["subkeys"],
                              factor_dims=p["factor_dims"], d_sub=p["d_sub"], W=p["W"], R=p["R"],
                              act_dtype="f32", bank_dtype="f32")
    assert np.array_equal(a["y"], b["y"]) and np.array_equal(M1, M2)
    for t, r in enumerate(a["rec"]):
        assert np.array_equal(r["w"]["idx"], b["idx_w"][t]) and np.array_equal(r["r"]["idx"], b["idx_r"][t])


def test_supplied_slots_follow_the_forward_oracle():
    """A pick that hands back slots (its own, then a reordered and a substituted set) gives
    the records run_stream computes for the same picks: same weights, y and bank."""
    p = _problem(6)

    def swap(t, which, idx, w):
        if t % 3 == 0:
            return None
        alt = np.array(idx, dtype=np.int64)
        if t % 3 == 1:
            alt[[0, 1]] = alt[[1, 0]]
        else:
            others = np.setdiff1d(np.arange(int(np.prod(p["factor_dims"]))), alt)
            alt[-1] = others[0]
        return alt

    M1 = p["bank"].astype(np.float32).astype(np.float64)
    M2 = M1.copy()
    a = bwd.stream_forward(M1, p["q_w"], p["q_r"], p["k_val"], p["gates"], p["subkeys"],
                           factor_dims=p["factor_dims"], d_sub=p["d_sub"], W=p["W"], R=p["R"], pick=swap)
    b = fwd_oracle.run_stream(M2, p["q_w"], p["q_r"], p["k_val"], p["gates"], p["subkeys"],
                              factor_dims=p["factor_dims"], d_sub=p["d_sub"], W=p["W"], R=p["R"],
                              act_dtype="f32", bank_dtype="f32", pick=swap)
    assert np.array_equal(a["y"], b["y"]) and np.array_equal(M1, M2)
    for t, r in enumerate(a["rec"]):
        assert np.array_equal(r["w"]["idx"], b["idx_w"][t]) and np.array_equal(r["w"]["w"], b["wt_w"][t])
        assert np.array_equal(r["r"]["idx"], b["idx_r"][t]) and np.array_equal(r["r"]["w"], b["wt_r"][t])
        dig = np.stack(np.unravel_index(r["w"]["idx"], p["factor_dims"]), axis=1)
        assert np.array_equal(r["w"]["digits"], dig)
    own = bwd.record_of(p["q_w"][0], p["subkeys"], p["factor_dims"], p["d_sub"], a["rec"][0]["w"]["idx"])
    for k in ("idx", "digits", "w", "S"):
        assert np.array_equal(own[k], a["rec"][0]["w"][k]), k


def test_identity_write_closed_form():
    # alpha = 1, beta = 0: the bank never changes; y_t = sum_j r_j M[i^r_j].  Then
    # dL/dM = c_M + sum_t scatter(i^r_t, r_t dy_t); the write passes nothing to the bank.
    p = _problem(6)
    p["gates"][:, 0] = 1.0
    p["gates"][:, 1] = 0.0
    g, _ = _grads(p)
    M = p["bank"].copy()
    out = bwd.stream_forward(M, p["q_w"], p["q_r"], p["k_val"], p["gates"], p["subkeys"],
                             factor_dims=p["factor_dims"], d_sub=p["d_sub"], W=p["W"], R=p["R"],
                             act_dtype="f64", bank_dtype="f64", exact=True)
    want = p["c_M"].copy()
    for t, r in enumerate(out["rec"]):
        for j, n in enumerate(r["r"]["idx"]):
            want[n] += r["r"]["w"][j] * p["c_y"][t]
    assert np.allclose(g["bank"], want, rtol=1e-13, atol=1e-13)
    assert np.all(g["k_val"] == 0)
    assert np.all(g["q_w"] == 0)   # the write weights do not reach the loss
    # dL/dbeta_t = sum_j w_j <G_t[i_j], v_t - sum_k w_k M[i_k]>, G_t = c_M plus the reads
    # at t and later (the rows never change)
    for t, r in enumerate(out["rec"]):
        Gt = p["c_M"].copy()
        for t2 in range(t, len(out["rec"])):
            for j, n in enumerate(out["rec"][t2]["r"]["idx"]):
                Gt[n] += out["rec"][t2]["r"]["w"][j] * p["c_y"][t2]
        w, iw = r["w"]["w"], r["w"]["idx"]
        u = p["k_val"][t] - w @ p["bank"][iw]
        assert np.isclose(g["gates"][t, 1], np.sum(w * (Gt[iw] @ u)), rtol=1e-12, atol=1e-13)


def test_full_strength_single_write_closed_form():
    # W = 1, beta = 1: the written row becomes v exactly, whatever it held, so its value
    # takes the row's whole gradient and the row before the write gets none of it.
    p = _problem(7, W=1, R=2, T=1)
    p["gates"][:, 1] = 1.0
    g, _ = _grads(p)
    M = p["bank"].copy()
    out = bwd.stream_forward(M, p["q_w"], p["q_r"], p["k_val"], p["gates"], p["subkeys"],
                             factor_dims=p["factor_dims"], d_sub=p["d_sub"], W=1, R=2,
                             act_dtype="f64", bank_dtype="f64", exact=True)
    rec = out["rec"][0]
    n = int(rec["w"]["idx"][0])
    G = p["c_M"][n].copy()
    for j, m in enumerate(rec["r"]["idx"]):
        if m == n:
            G += rec["r"]["w"][j] * p["c_y"][0]
    assert np.allclose(g["k_val"][0], G, rtol=1e-13, atol=1e-13)
    assert np.allclose(g["bank"][n], 0.0, atol=1e-13)
    assert abs(g["gates"][0, 0]) < 1e-13     # alpha is multiplied away by (1 - beta)


def test_batched_entry_sums_subkey_gradients_over_batch():
    rng = np.random.default_rng(8)
    B, T, H, fd, d_sub, d_v, W, R = 2, 3, 2, (5, 6), 3, 4, 2, 3
    N, F = 30, 2
    q_w = rng.normal(0, 2, (B, T, H, F * d_sub))
    q_r = rng.normal(0, 2, (B, T, H, F * d_sub))
    k_val = rng.normal(0, 1, (B, T, H, d_v))
    gates = rng.uniform(0.2, 0.9, (B, T, H, 2))
    subkeys = rng.normal(0, 0.5, (H, sum(fd), d_sub))
    bank = rng.normal(0, 0.5, (B, H, N, d_v)).astype(np.float32).astype(np.float64)
    dy = rng.normal(0, 1, (B, T, H, d_v))
    dbank = rng.normal(0, 1, (B, H, N, d_v))
    out = bwd.sdm_write_read_backward(q_w, q_r, k_val, gates, subkeys, bank, dy, dbank, factor_dims=fd,
                                      W=W, R=R)
    dK = np.zeros_like(subkeys)
    for b in range(B):
        for h in range(H):
            M = bank[b, h].copy()
            f = bwd.stream_forward(M, q_w[b, :, h], q_r[b, :, h], k_val[b, :, h], gates[b, :, h], subkeys[h],
                                   factor_dims=fd, d_sub=d_sub, W=W, R=R)
            g = bwd.stream_backward(M, f, dy[b, :, h], dbank[b, h], q_w[b, :, h], q_r[b, :, h],
                                    k_val[b, :, h], gates[b, :, h], subkeys[h], factor_dims=fd, d_sub=d_sub)
            assert np.array_equal(out["bank"][b, h], g["bank"])
            assert np.array_equal(out["q_w"][b, :, h], g["q_w"])
            dK[h] += g["subkeys"]
    assert np.array_equal(out["subkeys"], dK)


def _batched(seed, bank_dtype, snapshot_dtype=None):
    rng = np.random.default_rng(seed)
    B, T, H, fd, d_sub, d_v, W, R = 1, 4, 2, (6, 5), 4, 8, 3, 3
    N = 30
    q_w = rng.normal(0, 2, (B, T, H, 2 * d_sub))
    q_r = rng.normal(0, 2, (B, T, H, 2 * d_sub))
    k_val = rng.normal(0, 1, (B, T, H, d_v))
    gates = rng.uniform(0.2, 0.9, (B, T, H, 2))
    subkeys = rng.normal(0, 0.5, (H, sum(fd), d_sub))
    bank = fwd_oracle.round_to(rng.normal(0, 0.5, (B, H, N, d_v)), bank_dtype)
    dy = rng.normal(0, 1, (B, T, H, d_v))
    dbank = rng.normal(0, 1, (B, H, N, d_v))
    return bwd.sdm_write_read_backward(q_w, q_r, k_val, gates, subkeys, bank, dy, dbank, factor_dims=fd,
                                       W=W, R=R, bank_dtype=bank_dtype, snapshot_dtype=snapshot_dtype)


def test_bf16_snapshot_on_a_bf16_bank_changes_nothing():
    # CHANGELOG 2.0.0 > Package: on a bfloat16 bank the bf16 snapshot is bit-identical to
    # the default one (the rows it keeps are bfloat16 already)
    a = _batched(9, "bf16")
    b = _batched(9, "bf16", "bf16")
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_bf16_snapshot_on_a_float32_bank_moves_only_the_gradients_that_read_it():
    # the value gradient never reads the rows before the write; the gate and query
    # gradients do, and move by about bfloat16's rounding of those rows
    a = _batched(10, "f32")
    b = _batched(10, "f32", "bf16")
    assert np.array_equal(a["k_val"], b["k_val"])
    for k in ("gates", "q_w"):
        diff = np.abs(a[k] - b[k]).max()
        assert 0 < diff <= 2.0 ** -6 * np.abs(a[k]).max(), (k, diff)
