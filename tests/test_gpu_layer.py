"""The layer forward around the op (sdm_layer_forward) on the GPU against oracle/sdm_layer.py.

README > usage example: x [batch, tokens, dim] -> y [batch, tokens, dim], the bank
advancing in place.  Checked in three parts, each on the GPU's own inputs to that part:
  * the projections (cuBLASLt GEMMs) and the gates (this library's kernel) against the
    oracle's float64 products of the same x and weights, rounded once: within one
    rounding of the activation type (rtol 1e-5 float32, 2e-2 bfloat16, measured as
    |gpu - oracle| <= rtol * (|oracle| + rms));
  * the op on the GPU's projections, with the op's parity rules (compare_stream);
  * the output projection of the GPU's read against the oracle's product of it.
Plus bitwise repeatability, and the README call at full size on sampled rows and a
sampled stream.
"""

import numpy as np
import pytest
import torch

import sdm_inputs
from oracle import sdm_layer
from sdm_inputs import CONFIGS
from sdm_testlib import RTOL, _f64, assert_close, compare_stream, to_device

pytestmark = pytest.mark.gpu

KEEP = ("q_w", "q_r", "k_val", "gates", "y")


def run_layer(cfg, L, dim):
    import gated_delta_rule_factor_gb300 as sdm
    g = to_device(L)
    B, T = g["x"].shape[:2]
    act = g["x"].dtype
    bank = torch.empty((B, cfg.H, cfg.N, cfg.d_v), dtype=g["bank_init"].dtype, device="cuda")
    keep = {"q_w": torch.empty((B, T, cfg.H, cfg.F * cfg.d_sub), dtype=act, device="cuda"),
            "q_r": torch.empty((B, T, cfg.H, cfg.F * cfg.d_sub), dtype=act, device="cuda"),
            "k_val": torch.empty((B, T, cfg.H, cfg.d_v), dtype=act, device="cuda"),
            "gates": torch.empty((B, T, cfg.H, 2), dtype=torch.float32, device="cuda"),
            "y": torch.empty((B, T, cfg.H, cfg.d_v), dtype=act, device="cuda")}
    sh = sdm.make_shape(B=B, T=T, H=cfg.H, factor_dims=cfg.factor_dims, d_sub=cfg.d_sub, d_v=cfg.d_v, W=cfg.W,
                        R=cfg.R, chunk_size=cfg.chunk_size, act_dtype=0 if cfg.act_dtype == "f32" else 1,
                        bank_dtype=0 if cfg.bank_dtype == "f32" else 1)
    ws = torch.empty(sdm.layer_workspace_size(sh, dim), dtype=torch.uint8, device="cuda")
    out = sdm.sdm_layer_forward(g["x"], g["w_qw"], g["w_qr"], g["w_v"], g["w_g"], g["w_o"], g["subkeys"], bank,
                                cfg.chunk_size, cfg.W, cfg.R, factor_dims=cfg.factor_dims,
                                bank_init=g["bank_init"], keep=keep, workspace=ws)
    torch.cuda.synchronize()
    assert sdm.last_device_error(ws) == 0
    res = {k: v.cpu() for k, v in keep.items()}
    res["out"] = out.cpu()
    res["bank"] = bank
    return res


def check_projections(cfg, L, gpu, rows=None):
    """GPU projections and gates against the oracle's products of the same x (rows: a
    sample of token rows b*T + t, else all)."""
    B, T, dim = L["x"].shape
    X = _f64(L["x"]).reshape(B * T, dim)
    sel = np.arange(B * T) if rows is None else np.asarray(rows)
    rt = RTOL[cfg.act_dtype]
    for name, w in (("q_w", "w_qw"), ("q_r", "w_qr"), ("k_val", "w_v")):
        want = sdm_layer.project(X[sel], L[w], cfg.act_dtype)
        got = gpu[name].reshape(B * T, -1)[torch.as_tensor(sel)]
        assert_close(got, want, rt, name)
    assert_close(gpu["gates"].reshape(B * T, -1)[torch.as_tensor(sel)], sdm_layer.gates_of(X[sel], L["w_g"]),
                 1e-6, "gates")


def check_output(cfg, L, gpu, rows=None):
    B, T, dim = L["x"].shape
    Y = _f64(gpu["y"]).reshape(B * T, -1)
    sel = np.arange(B * T) if rows is None else np.asarray(rows)
    want = sdm_layer.project(Y[sel], L["w_o"], cfg.act_dtype)
    assert_close(gpu["out"].reshape(B * T, dim)[torch.as_tensor(sel)], want, RTOL[cfg.act_dtype], "out")


def op_inputs_of(gpu, L):
    """The op's inputs as the GPU produced them, in make_inputs' layout."""
    return {"q_w": gpu["q_w"], "q_r": gpu["q_r"], "k_val": gpu["k_val"], "gates": gpu["gates"],
            "subkeys": L["subkeys"], "bank_init": L["bank_init"]}


LAYERS = {
    "tiny_f32": (dict(), 96),
    "small_bf16": (dict(act_dtype="bf16", factor_dims=(16, 16), d_sub=32, d_v=64, H=2, B=2, T=48, W=16, R=16), 128),
    "bf16_bank": (dict(act_dtype="bf16", bank_dtype="bf16", d_v=128, W=64, R=64, T=40), 160),
    "three_factors": (dict(factor_dims=(8, 8, 8), d_sub=16, W=16, R=12, T=60), 72),
}


@pytest.mark.parametrize("name", sorted(LAYERS))
def test_layer_matches_oracle(name):
    kw, dim = LAYERS[name]
    cfg = CONFIGS["tiny"].replace(**kw)
    L = sdm_inputs.make_layer_inputs(cfg, dim)
    gpu = run_layer(cfg, L, dim)
    check_projections(cfg, L, gpu)
    d = op_inputs_of(gpu, L)
    res = [compare_stream(cfg, d, {**gpu, "bank": gpu["bank"].cpu(), **_selections(cfg, d)}, b, h)
           for b in range(cfg.B) for h in range(cfg.H)]
    assert sum(r["near_ties"] for r in res) <= 2, res
    check_output(cfg, L, gpu)


def _selections(cfg, d):
    """The op's selections on the GPU's projections (sdm_write_read on the same inputs, the
    same kernels the layer ran): compare_stream checks them against the oracle."""
    from sdm_testlib import gpu_write_read
    g = gpu_write_read(cfg, d)
    return {k: g[k] for k in ("idx_w", "wt_w", "idx_r", "wt_r")}


def test_layer_is_bitwise_repeatable():
    kw, dim = LAYERS["small_bf16"]
    cfg = CONFIGS["tiny"].replace(**kw)
    L = sdm_inputs.make_layer_inputs(cfg, dim)
    a = run_layer(cfg, L, dim)
    b = run_layer(cfg, L, dim)
    for k in KEEP + ("out",):
        assert torch.equal(a[k], b[k]), k
    assert torch.equal(a["bank"], b["bank"])


def test_readme_call_full_size():
    """The README call: dim=2048, num_heads=2, 65536 slots per head, W=R=64, chunk 64,
    B=2, T=4096, bf16 activations (float32 bank); projections and output on 64 sampled
    token rows, the op on one whole sampled stream."""
    cfg = CONFIGS["layer"]
    dim = 2048
    L = sdm_inputs.make_layer_inputs(cfg, dim)
    gpu = run_layer(cfg, L, dim)
    rows = np.random.default_rng(7).choice(cfg.B * cfg.T, 64, replace=False)
    check_projections(cfg, L, gpu, rows)
    check_output(cfg, L, gpu, rows)
    d = op_inputs_of(gpu, L)
    sel = _selections(cfg, d)
    r = compare_stream(cfg, d, {"y": gpu["y"], "bank": gpu["bank"].cpu(), **sel}, 1, 0)
    assert r["rows"] == cfg.T
    print(f"README call: stream (1, 0) compared over {r['rows']} tokens, {r['near_ties']} near-tie picks")


# ---------------------------------------------------------------- training through the layer

GRAD_RTOL = {"f32": 1e-4, "bf16": 3e-2}
LAYER_GRADS = ("x", "w_qw", "w_qr", "w_v", "w_g", "w_o", "subkeys", "bank", "bank_init")


def run_layer_train(cfg, L, dim, dout, snapshot_dtype=torch.float32):
    import gated_delta_rule_factor_gb300 as sdm
    g = to_device(L)
    B = g["x"].shape[0]
    bank = torch.empty((B, cfg.H, cfg.N, cfg.d_v), dtype=g["bank_init"].dtype, device="cuda")
    out, saved = sdm.sdm_layer_forward_train(g["x"], g["w_qw"], g["w_qr"], g["w_v"], g["w_g"], g["w_o"],
                                             g["subkeys"], bank, cfg.chunk_size, cfg.W, cfg.R,
                                             factor_dims=cfg.factor_dims, bank_init=g["bank_init"],
                                             snapshot_dtype=snapshot_dtype)
    torch.cuda.synchronize()
    bank_after = bank.clone()
    grads = sdm.sdm_layer_backward(g["x"], g["w_qw"], g["w_qr"], g["w_v"], g["w_g"], g["w_o"], g["subkeys"], bank,
                                   dout.cuda(), saved, cfg.chunk_size, cfg.W, cfg.R, factor_dims=cfg.factor_dims)
    torch.cuda.synchronize()
    assert sdm.last_device_error(grads["workspace"]) == 0
    res = {"out": out.cpu(), "bank_after": bank_after, "bank_restored": bank,
           "saved": {k: v.cpu() for k, v in saved.items() if isinstance(v, torch.Tensor) and k != "snapshot"}}
    res.update({k: grads[k].cpu() for k in LAYER_GRADS})
    return res


def oracle_layer_backward(cfg, L, dout, gpu):
    """The oracle's layer gradients on the GPU's intermediates, following its near-tie picks."""
    from oracle import sdm_layer
    sv = gpu["saved"]
    K = {h: _f64(L["subkeys"][h]) for h in range(cfg.H)}
    near = []

    def pick_for(b, h):
        q = (_f64(sv["q_w"][b, :, h]), _f64(sv["q_r"][b, :, h]))
        gi = (sv["idx_w"][b, :, h].numpy(), sv["idx_r"][b, :, h].numpy())
        gw = (sv["wt_w"][b, :, h].numpy(), sv["wt_r"][b, :, h].numpy())

        def pick(t, which, idx, w):
            from sdm_testlib import check_selection
            if check_selection(cfg, q[which][t], K[h], (cfg.W, cfg.R)[which], gi[which][t], gw[which][t], idx, w):
                return None
            near.append((b, h, t))
            return np.asarray(gi[which][t], dtype=np.int64)
        return pick

    given = {k: sv[k] for k in ("q_w", "q_r", "k_val", "gates", "y")}
    o = sdm_layer.layer_backward(L["x"], L["w_qw"], L["w_qr"], L["w_v"], L["w_g"], L["w_o"], L["subkeys"],
                                 L["bank_init"], dout, factor_dims=cfg.factor_dims, W=cfg.W, R=cfg.R,
                                 act_dtype=cfg.act_dtype, bank_dtype=cfg.bank_dtype, given=given, pick=pick_for)
    return o, len(near)


def compare_layer_grads(cfg, gpu, o):
    rt = GRAD_RTOL["bf16" if "bf16" in (cfg.act_dtype, cfg.bank_dtype) else "f32"]
    for k in LAYER_GRADS:
        assert_close(gpu[k], o[k], rt, f"d_{k}")


LAYER_TRAIN = {
    "tiny_f32": (dict(), 96),
    "small_bf16": (dict(act_dtype="bf16", factor_dims=(16, 16), d_sub=32, d_v=64, H=2, B=2, T=48, W=16, R=16), 128),
    "bf16_bank": (dict(act_dtype="bf16", bank_dtype="bf16", d_v=128, W=64, R=64, T=40), 160),
    "three_factors": (dict(factor_dims=(8, 8, 8), d_sub=16, W=16, R=12, T=60), 72),
}


@pytest.mark.parametrize("name", sorted(LAYER_TRAIN))
def test_layer_backward_matches_oracle(name):
    kw, dim = LAYER_TRAIN[name]
    cfg = CONFIGS["tiny"].replace(**kw)
    L = sdm_inputs.make_layer_inputs(cfg, dim)
    dout = sdm_inputs.make_grad_inputs(cfg.replace(d_v=dim, H=1), dbank=False)["dy"].reshape(cfg.B, cfg.T, dim)
    gpu = run_layer_train(cfg, L, dim, dout)
    assert torch.equal(gpu["bank_restored"], to_device(L)["bank_init"].unsqueeze(0).expand_as(gpu["bank_restored"]))
    o, near = oracle_layer_backward(cfg, L, dout, gpu)
    assert near <= 2, near
    compare_layer_grads(cfg, gpu, o)


def test_layer_training_is_bitwise_repeatable():
    kw, dim = LAYER_TRAIN["small_bf16"]
    cfg = CONFIGS["tiny"].replace(**kw)
    L = sdm_inputs.make_layer_inputs(cfg, dim)
    dout = sdm_inputs.make_grad_inputs(cfg.replace(d_v=dim, H=1), dbank=False)["dy"].reshape(cfg.B, cfg.T, dim)
    a = run_layer_train(cfg, L, dim, dout)
    b = run_layer_train(cfg, L, dim, dout)
    for k in LAYER_GRADS + ("out",):
        assert torch.equal(a[k], b[k]), k


def test_readme_call_training_full_width():
    """The README call's shapes (dim 2048, 2 heads of d_v 1024, 65536 slots per head,
    W = R = 64, bf16) at T = 1024, forward and backward, every gradient against the oracle."""
    cfg = CONFIGS["layer"].replace(T=1024)
    dim = 2048
    L = sdm_inputs.make_layer_inputs(cfg, dim)
    dout = sdm_inputs.make_grad_inputs(cfg.replace(d_v=dim, H=1), dbank=False)["dy"].reshape(cfg.B, cfg.T, dim)
    gpu = run_layer_train(cfg, L, dim, dout)
    o, near = oracle_layer_backward(cfg, L, dout, gpu)
    print(f"README call training: {near} near-tie picks followed")
    compare_layer_grads(cfg, gpu, o)
