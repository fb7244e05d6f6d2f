"""Pins of the layer oracle (oracle/sdm_layer.py) against the op oracle and closed forms.

sparse-delta-memory README > usage example: the layer maps x [batch, tokens, dim] to the
same shape through the op.  With 0/1 selection weights the projections pick coordinates
of x exactly and the output projection places the read back into chosen coordinates, so
the layer must reduce to the op oracle on slices of x (a transposed weight, a swapped
projection or a wrong head order fails); the gates' sigmoid is checked on exact logits.
"""

import numpy as np
import pytest

from oracle import sdm_layer, sdm_oracle


def _select(rows: int, dim: int, cols) -> np.ndarray:
    """[rows, dim] 0/1 matrix whose row i picks coordinate cols[i] of x."""
    w = np.zeros((rows, dim))
    w[np.arange(rows), cols] = 1.0
    return w


def _problem(seed=0, B=2, T=12, H=2, factor_dims=(4, 5), d_sub=3, d_v=4, dim=61):
    rng = np.random.default_rng(seed)
    F = len(factor_dims)
    N = int(np.prod(factor_dims))
    x = rng.normal(0, 1, (B, T, dim))
    perm = rng.permutation(dim)
    dq = H * F * d_sub
    cq_w, cq_r, cv = perm[:dq], perm[dq:2 * dq], perm[2 * dq:2 * dq + H * d_v]
    w_qw, w_qr, w_v = _select(dq, dim, cq_w), _select(dq, dim, cq_r), _select(H * d_v, dim, cv)
    out_cols = rng.permutation(dim)[:H * d_v]
    w_o = np.zeros((dim, H * d_v))
    w_o[out_cols, np.arange(H * d_v)] = 1.0
    subkeys = rng.normal(0, 1 / np.sqrt(d_sub), (H, sum(factor_dims), d_sub))
    bank = rng.normal(0, 0.5, (H, N, d_v))
    return dict(x=x, w_qw=w_qw, w_qr=w_qr, w_v=w_v, w_o=w_o, cq_w=cq_w, cq_r=cq_r, cv=cv, out_cols=out_cols,
                subkeys=subkeys, bank=bank, factor_dims=factor_dims, B=B, T=T, H=H, d_v=d_v, dim=dim, F=F,
                d_sub=d_sub)


def test_selection_weights_reduce_the_layer_to_the_op():
    p = _problem()
    B, T, H, F, d_sub, d_v = p["B"], p["T"], p["H"], p["F"], p["d_sub"], p["d_v"]
    w_g = np.zeros((2 * H, p["dim"]))                            # gates = sigmoid(0) = 1/2
    got = sdm_layer.layer_forward(p["x"], p["w_qw"], p["w_qr"], p["w_v"], w_g, p["w_o"], p["subkeys"], p["bank"],
                                  factor_dims=p["factor_dims"], W=3, R=4)
    q_w = p["x"][..., p["cq_w"]].reshape(B, T, H, F * d_sub)
    q_r = p["x"][..., p["cq_r"]].reshape(B, T, H, F * d_sub)
    k_val = p["x"][..., p["cv"]].reshape(B, T, H, d_v)
    gates = np.full((B, T, H, 2), 0.5)
    assert np.array_equal(got["q_w"], sdm_oracle.round_to(q_w, "f32"))
    assert np.array_equal(got["q_r"], sdm_oracle.round_to(q_r, "f32"))
    assert np.array_equal(got["k_val"], sdm_oracle.round_to(k_val, "f32"))
    assert np.array_equal(got["gates"], gates)
    op = sdm_oracle.sdm_write_read(sdm_oracle.round_to(q_w, "f32"), sdm_oracle.round_to(q_r, "f32"),
                                   sdm_oracle.round_to(k_val, "f32"), gates, p["subkeys"], p["bank"],
                                   factor_dims=p["factor_dims"], W=3, R=4)
    out = np.zeros((B, T, p["dim"]))
    for b in range(B):
        for h in range(H):
            assert np.array_equal(got["y"][b, :, h], op[(b, h)]["y"])
            out[b][:, p["out_cols"][h * d_v:(h + 1) * d_v]] = op[(b, h)]["y"]
    assert np.array_equal(got["out"], out)


def test_given_inputs_replace_the_projections_only_for_the_op():
    p = _problem(1)
    w_g = np.zeros((2 * p["H"], p["dim"]))
    base = sdm_layer.layer_forward(p["x"], p["w_qw"], p["w_qr"], p["w_v"], w_g, p["w_o"], p["subkeys"], p["bank"],
                                   factor_dims=p["factor_dims"], W=3, R=4)
    alt_k = base["k_val"] * 2.0
    got = sdm_layer.layer_forward(p["x"], p["w_qw"], p["w_qr"], p["w_v"], w_g, p["w_o"], p["subkeys"], p["bank"],
                                  factor_dims=p["factor_dims"], W=3, R=4, given={"k_val": alt_k})
    assert np.array_equal(got["k_val"], base["k_val"])          # the oracle's own projection is reported
    assert not np.array_equal(got["y"], base["y"])              # the op ran on the given values


def test_gate_sigmoid_on_exact_logits():
    # logits ln 3 and -ln 3 give 3/4 and 1/4 exactly in float32
    x = np.array([[np.log(3.0), 0.0]])
    w_g = np.array([[1.0, 0.0], [-1.0, 0.0], [0.0, 1.0]])
    g = sdm_layer.gates_of(x, w_g)
    assert np.array_equal(g, np.array([[0.75, 0.25, 0.5]]))


def test_output_projection_is_linear_in_its_weight():
    p = _problem(2)
    rng = np.random.default_rng(5)
    w_g = rng.normal(0, 0.3, (2 * p["H"], p["dim"]))
    w_o1 = rng.normal(0, 1, (p["dim"], p["H"] * p["d_v"]))
    w_o2 = rng.normal(0, 1, (p["dim"], p["H"] * p["d_v"]))
    kw = dict(factor_dims=p["factor_dims"], W=3, R=4, act_dtype="f64", bank_dtype="f64")
    args = (p["x"], p["w_qw"], p["w_qr"], p["w_v"], w_g)
    a = sdm_layer.layer_forward(*args, w_o1, p["subkeys"], p["bank"], **kw)["out"]
    b = sdm_layer.layer_forward(*args, w_o2, p["subkeys"], p["bank"], **kw)["out"]
    c = sdm_layer.layer_forward(*args, w_o1 + w_o2, p["subkeys"], p["bank"], **kw)["out"]
    assert np.allclose(a + b, c, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- the layer's backward

from oracle import sdm_backward  # noqa: E402

GROUPS = ("x", "w_qw", "w_qr", "w_v", "w_g", "w_o", "subkeys", "bank_init")


def _train_problem(seed=3, B=2, T=6, H=2, factor_dims=(4, 5), d_sub=3, d_v=4, dim=9):
    rng = np.random.default_rng(seed)
    F = len(factor_dims)
    N = int(np.prod(factor_dims))
    dq = H * F * d_sub
    p = {"x": rng.normal(0, 1, (B, T, dim)), "w_qw": rng.normal(0, 0.6, (dq, dim)),
         "w_qr": rng.normal(0, 0.6, (dq, dim)), "w_v": rng.normal(0, 0.5, (H * d_v, dim)),
         "w_g": rng.normal(0, 0.5, (2 * H, dim)), "w_o": rng.normal(0, 0.5, (dim, H * d_v)),
         "subkeys": rng.normal(0, 1 / np.sqrt(d_sub), (H, sum(factor_dims), d_sub)),
         "bank_init": rng.normal(0, 0.5, (H, N, d_v))}
    c_out = rng.normal(0, 1, (B, T, dim))
    c_M = rng.normal(0, 1, (B, H, N, d_v))
    return p, c_out, c_M, dict(factor_dims=factor_dims, W=3, R=4)


def _exact_loss(p, c_out, c_M, kw):
    """sum(c_out * out) + sum(c_M * final banks), the layer in float64 with float64 scores."""
    B, T, dim = p["x"].shape
    H = p["subkeys"].shape[0]
    X = p["x"].reshape(B * T, dim)
    q_w = (X @ p["w_qw"].T).reshape(B, T, H, -1)
    q_r = (X @ p["w_qr"].T).reshape(B, T, H, -1)
    k_val = (X @ p["w_v"].T).reshape(B, T, H, -1)
    gates = (1.0 / (1.0 + np.exp(-(X @ p["w_g"].T)))).reshape(B, T, H, 2)
    d_v = p["bank_init"].shape[-1]
    Y = np.zeros((B, T, H, d_v))
    loss = 0.0
    for b in range(B):
        for h in range(H):
            M = p["bank_init"][h].copy()
            rec = sdm_backward.stream_forward(M, q_w[b, :, h], q_r[b, :, h], k_val[b, :, h], gates[b, :, h],
                                              p["subkeys"][h], factor_dims=kw["factor_dims"], d_sub=p["subkeys"].shape[2],
                                              W=kw["W"], R=kw["R"], act_dtype="f64", bank_dtype="f64", exact=True)
            Y[b, :, h] = rec["y"]
            loss += float(np.sum(c_M[b, h] * M))
    out = Y.reshape(B * T, -1) @ p["w_o"].T
    return loss + float(np.sum(c_out.reshape(B * T, dim) * out))


@pytest.mark.parametrize("group", GROUPS)
def test_layer_gradients_match_directional_differences(group):
    """<grad, v> against the central difference of the exact layer loss along a random
    direction v of one parameter group: a dropped term, a transposed weight or a wrong
    sigmoid derivative moves it far beyond the difference's error."""
    p, c_out, c_M, kw = _train_problem()
    g = sdm_layer.layer_backward(p["x"], p["w_qw"], p["w_qr"], p["w_v"], p["w_g"], p["w_o"], p["subkeys"],
                                 p["bank_init"], c_out, dbank=c_M, act_dtype="f64", bank_dtype="f64", exact=True, **kw)
    rng = np.random.default_rng(11)
    v = rng.normal(0, 1, p[group].shape)
    eps = 1e-6
    hi, lo = dict(p), dict(p)
    hi[group] = p[group] + eps * v
    lo[group] = p[group] - eps * v
    fd = (_exact_loss(hi, c_out, c_M, kw) - _exact_loss(lo, c_out, c_M, kw)) / (2 * eps)
    an = float(np.sum(g[group] * v))
    assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (group, fd, an)


def test_learned_table_gradient_is_the_batch_sum():
    p, c_out, c_M, kw = _train_problem(4)
    g = sdm_layer.layer_backward(p["x"], p["w_qw"], p["w_qr"], p["w_v"], p["w_g"], p["w_o"], p["subkeys"],
                                 p["bank_init"], c_out, dbank=c_M, act_dtype="f64", bank_dtype="f64", exact=True, **kw)
    assert np.array_equal(g["bank_init"], g["bank"].sum(axis=0))
