"""The deterministic sparse backward on the GPU against the oracle's reverse sweep.

sdm_write_read_train (the forward with a snapshot of the rows each token overwrites)
followed by sdm_write_read_backward, compared with oracle.sdm_backward on the same
seeded inputs and loss gradients (sparse-delta-memory CHANGELOG > 2.0.0 > New:
deterministic sparse backward; > Behavior changes: the first backward restores the bank
in place; > Package: bf16 snapshots).

Rules:
  * selections are checked as in the forward parity tests (check_selection); at a valid
    near tie the oracle takes the GPU's slots, so every token stays compared;
  * gradients match within GRAD_RTOL, measured as in the forward tests:
    |gpu - oracle| <= rtol * (|oracle| + rms(oracle)) per tensor;
  * the bank comes back bit for bit (float32 snapshot, or any snapshot of a bfloat16
    bank); with a bfloat16 snapshot of a float32 bank the rows the forward wrote come
    back rounded to bfloat16 and every other row is untouched;
  * gradients are bitwise repeatable and do not depend on the forward's chunk size.
"""

import numpy as np
import pytest
import torch

import sdm_inputs
from oracle import sdm_backward as obwd
from sdm_inputs import CONFIGS
from sdm_testlib import _f64, assert_close, check_selection, to_device

pytestmark = pytest.mark.gpu

# Gradient tolerance.  Every gradient is a float32 chain of sums whose length grows with
# the sequence: G accumulates r_j dy and alpha-scaled updates over every later token that
# touches the row, dalpha/dbeta/dw sum W*d_v products, ds subtracts the weighted mean of
# dw (cancellation), and dK sums over all 2*B*T query rows.  With float32 rounding
# u = 2^-24 and sums of length n <= 2^16 the forward error bound n*u is ~4e-3 in the
# worst case and ~sqrt(n)*u ~ 1.5e-5 typically; 1e-4 of the tensor's rms leaves room for
# the cancellation in ds.  bfloat16 activations or banks carry the forward's 2e-2.
GRAD_RTOL = {"f32": 1e-4, "bf16": 3e-2}
GRAD_KEYS = ("k_val", "gates", "q_w", "q_r", "subkeys", "bank")
_T = {"f32": torch.float32, "bf16": torch.bfloat16}


def gpu_train_backward(cfg, d, gr, *, snapshot_dtype="f32", chunk_size=None, device="cuda"):
    """Forward with snapshot, then backward, on CPU inputs ``d`` and gradients ``gr``."""
    import gated_delta_rule_factor_gb300 as sdm
    g = to_device(d, device)
    gg = to_device(gr, device)
    B, T, H = g["q_w"].shape[:3]
    bank = g["bank_init"].unsqueeze(0).expand(B, *g["bank_init"].shape).contiguous()
    bank0 = bank.clone()
    saved = sdm.sdm_write_read_train(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], bank,
                                     chunk_size or cfg.chunk_size, cfg.W, cfg.R, factor_dims=cfg.factor_dims,
                                     snapshot_dtype=_T[snapshot_dtype])
    torch.cuda.synchronize()
    bank_after = bank.clone()
    dbank = gg["dbank"].clone()
    grads = sdm.sdm_write_read_backward(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], bank,
                                        gg["dy"], saved, cfg.W, cfg.R, factor_dims=cfg.factor_dims, dbank=dbank)
    torch.cuda.synchronize()
    assert sdm.last_device_error(grads["workspace"]) == 0
    out = {k: grads[k] for k in GRAD_KEYS}
    out.update(y=saved["y"], bank0=bank0, bank_after=bank_after, bank_restored=bank,
               idx_w=saved["idx_w"], wt_w=saved["wt_w"], idx_r=saved["idx_r"], wt_r=saved["wt_r"])
    return out


def oracle_backward(cfg, d, gr, gpu, *, stream=None, snapshot_dtype=None):
    """The oracle's gradients on the same inputs, following the GPU's valid near-tie picks.

    stream=(b, h): only that stream, from its own slices of the inputs (results shaped
    with B = H = 1).  Returns (gradients, number of near-tie picks)."""
    near = []
    if stream is not None:
        b0, h0 = stream
        d = {"q_w": d["q_w"][b0:b0 + 1, :, h0:h0 + 1], "q_r": d["q_r"][b0:b0 + 1, :, h0:h0 + 1],
             "k_val": d["k_val"][b0:b0 + 1, :, h0:h0 + 1], "gates": d["gates"][b0:b0 + 1, :, h0:h0 + 1],
             "subkeys": d["subkeys"][h0:h0 + 1], "bank_init": d["bank_init"][h0:h0 + 1]}
        gr = {"dy": gr["dy"][b0:b0 + 1, :, h0:h0 + 1], "dbank": gr["dbank"][b0:b0 + 1, h0:h0 + 1]}
    else:
        b0 = h0 = 0
    K = {h: _f64(d["subkeys"][h]) for h in range(d["subkeys"].shape[0])}
    sel = {k: gpu[k].cpu() for k in ("idx_w", "wt_w", "idx_r", "wt_r")}

    def pick_for(b, h):
        q = (_f64(d["q_w"][b, :, h]), _f64(d["q_r"][b, :, h]))
        gi = (sel["idx_w"][b + b0, :, h + h0].numpy(), sel["idx_r"][b + b0, :, h + h0].numpy())
        gw = (sel["wt_w"][b + b0, :, h + h0].numpy(), sel["wt_r"][b + b0, :, h + h0].numpy())
        ks = (cfg.W, cfg.R)

        def pick(t, which, idx, w):
            if check_selection(cfg, q[which][t], K[h], ks[which], gi[which][t], gw[which][t], idx, w):
                return None
            near.append((b + b0, h + h0, t))
            return np.asarray(gi[which][t], dtype=np.int64)
        return pick

    B = d["q_w"].shape[0]
    bank = d["bank_init"].unsqueeze(0).expand(B, *d["bank_init"].shape)
    o = obwd.sdm_write_read_backward(d["q_w"], d["q_r"], d["k_val"], d["gates"], d["subkeys"], bank, gr["dy"],
                                     gr["dbank"], factor_dims=cfg.factor_dims, W=cfg.W, R=cfg.R,
                                     act_dtype=cfg.act_dtype, bank_dtype=cfg.bank_dtype,
                                     snapshot_dtype=snapshot_dtype, pick=pick_for)
    return o, len(near)


def _rtol(cfg):
    return GRAD_RTOL["bf16" if "bf16" in (cfg.act_dtype, cfg.bank_dtype) else "f32"]


def compare_grads(cfg, gpu, o, *, stream=None):
    """All streams (and the sub-key gradient), or one sampled stream (b, h) whose oracle
    results have B = H = 1 (the sub-key gradient then sums other streams too: skipped)."""
    rt = _rtol(cfg)
    worst = {}

    def close(got, want, what):
        g64, w64 = _f64(got), _f64(want)
        scale = np.sqrt(np.mean(w64 ** 2)) if w64.size else 0.0
        if w64.size:
            worst[what.split("[")[0]] = max(worst.get(what.split("[")[0], 0.0),
                                            float(np.max(np.abs(g64 - w64) / (np.abs(w64) + scale + 1e-300))))
        assert_close(got, want, rt, what)
    pairs = [((b, h), (b, h)) for b in range(cfg.B) for h in range(cfg.H)] if stream is None else [(stream, (0, 0))]
    for (b, h), (ob, oh) in pairs:
        for k in ("k_val", "gates", "q_w", "q_r"):
            close(gpu[k][b, :, h].cpu(), o[k][ob, :, oh], f"d_{k}[{b},:,{h}]")
        close(gpu["bank"][b, h].cpu(), o["bank"][ob, oh], f"d_bank[{b},{h}]")
    if stream is None:
        close(gpu["subkeys"].cpu(), o["subkeys"], "d_subkeys")
    print("worst error / (|oracle| + rms):", {k: f"{v:.2e}" for k, v in worst.items()})


def check_restored(cfg, gpu, snapshot_dtype):
    b0, br = gpu["bank0"], gpu["bank_restored"]
    if snapshot_dtype == "bf16" and cfg.bank_dtype == "f32":
        written = torch.zeros(br.shape[:3], dtype=torch.bool, device=br.device)
        B, T, H = gpu["idx_w"].shape[:3]
        for b in range(B):
            for h in range(H):
                written[b, h, gpu["idx_w"][b, :, h].reshape(-1).long()] = True
        rounded = b0.to(torch.bfloat16).float()
        assert written.any()
        assert torch.equal(br[written], rounded[written])
        assert torch.equal(br[~written], b0[~written])
    else:
        assert torch.equal(br, b0)


SMALL = {
    "tiny": dict(),
    "w64_r64": dict(W=64, R=64, T=40),
    "w48_r64_ragged": dict(W=48, R=64, T=37),
    "w128_r96": dict(factor_dims=(64, 64), W=128, R=96, T=24, d_v=64),
    "w3_r5": dict(W=3, R=5, T=30),
    "bf16_bank_bf16_acts": dict(act_dtype="bf16", bank_dtype="bf16", W=64, R=32, T=40, d_v=128),
    "f32_acts_bf16_bank": dict(bank_dtype="bf16", d_v=128, T=32),
    "bf16_acts_f32_bank": dict(act_dtype="bf16", d_v=96, W=24, R=40, T=40),
    "three_factors": dict(factor_dims=(8, 8, 8), d_sub=16, W=16, R=12),
    "many_streams": dict(B=3, H=2, T=50, W=64, R=64),
    "partial_last_piece_bf16": dict(d_v=72, bank_dtype="bf16", act_dtype="bf16", T=30),
    "every_slot": dict(factor_dims=(4, 4), W=16, R=16, T=24),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_gradients_match_oracle(name):
    cfg = CONFIGS["tiny"].replace(**SMALL[name])
    d = sdm_inputs.make_inputs(cfg)
    gr = sdm_inputs.make_grad_inputs(cfg)
    gpu = gpu_train_backward(cfg, d, gr)
    o, near = oracle_backward(cfg, d, gr, gpu)
    assert near <= 2, near
    compare_grads(cfg, gpu, o)
    check_restored(cfg, gpu, "f32")


def test_subkey_gradient_over_several_splits():
    """2*B*T = 2400 query rows: the sub-key gradient runs as three splits of 1024 rows,
    added in split order."""
    cfg = CONFIGS["tiny"].replace(B=2, T=600, W=16, R=16, d_v=32)
    d = sdm_inputs.make_inputs(cfg)
    gr = sdm_inputs.make_grad_inputs(cfg)
    gpu = gpu_train_backward(cfg, d, gr)
    o, near = oracle_backward(cfg, d, gr, gpu)
    assert near <= 2, near
    compare_grads(cfg, gpu, o)


@pytest.mark.parametrize("bank_dtype", ["f32", "bf16"])
def test_bf16_snapshot(bank_dtype):
    """bf16 snapshots: the forward is bit-identical to the float32-snapshot run; on a
    float32 bank the gradients that read the rounded rows match the oracle with
    snapshot_dtype="bf16"; on a bfloat16 bank the gradients and the restored bank are
    bit-identical to the float32 snapshot's."""
    cfg = CONFIGS["tiny"].replace(W=64, R=64, T=60, d_v=128, bank_dtype=bank_dtype)
    d = sdm_inputs.make_inputs(cfg)
    gr = sdm_inputs.make_grad_inputs(cfg)
    full = gpu_train_backward(cfg, d, gr, snapshot_dtype="f32")
    half = gpu_train_backward(cfg, d, gr, snapshot_dtype="bf16")
    for k in ("y", "bank_after", "idx_w", "wt_w", "idx_r", "wt_r"):
        assert torch.equal(full[k], half[k]), k
    check_restored(cfg, half, "bf16")
    if bank_dtype == "bf16":
        for k in GRAD_KEYS + ("bank_restored",):
            assert torch.equal(full[k], half[k]), k
    else:
        o, near = oracle_backward(cfg, d, gr, half, snapshot_dtype="bf16")
        assert near <= 2, near
        compare_grads(cfg, half, o)


def test_train_forward_is_the_plain_forward():
    """sdm_write_read_train leaves y, the bank and the selections bitwise as sdm_write_read."""
    from sdm_testlib import gpu_write_read
    cfg = CONFIGS["tiny"].replace(W=64, R=64, B=2, H=2, T=80, d_v=128)
    d = sdm_inputs.make_inputs(cfg)
    gr = sdm_inputs.make_grad_inputs(cfg)
    plain = gpu_write_read(cfg, d, bank_init=False)
    train = gpu_train_backward(cfg, d, gr)
    assert torch.equal(plain["y"], train["y"].cpu())
    assert torch.equal(plain["bank"], train["bank_after"].cpu())
    for k in ("idx_w", "wt_w", "idx_r", "wt_r"):
        assert torch.equal(plain[k], train[k].cpu()), k


def test_bitwise_repeatable_and_chunk_independent():
    cfg = CONFIGS["tiny"].replace(W=64, R=64, B=2, H=2, T=120, d_v=256)
    d = sdm_inputs.make_inputs(cfg)
    gr = sdm_inputs.make_grad_inputs(cfg)
    first = gpu_train_backward(cfg, d, gr)
    for chunk in (64, 1, 17, 256):
        again = gpu_train_backward(cfg, d, gr, chunk_size=chunk)
        for k in GRAD_KEYS + ("bank_restored",):
            assert torch.equal(first[k], again[k]), (chunk, k)


def test_second_backward_is_refused():
    """The snapshot serves one backward: a second one records SDM_DEVERR_SNAPSHOT and
    touches neither the bank nor the bank gradient."""
    import gated_delta_rule_factor_gb300 as sdm
    cfg = CONFIGS["tiny"].replace(T=40)
    d = to_device(sdm_inputs.make_inputs(cfg))
    gr = to_device(sdm_inputs.make_grad_inputs(cfg))
    bank = d["bank_init"].unsqueeze(0).contiguous()
    saved = sdm.sdm_write_read_train(d["q_w"], d["q_r"], d["k_val"], d["gates"], d["subkeys"], bank,
                                     cfg.chunk_size, cfg.W, cfg.R, factor_dims=cfg.factor_dims)
    g1 = sdm.sdm_write_read_backward(d["q_w"], d["q_r"], d["k_val"], d["gates"], d["subkeys"], bank, gr["dy"],
                                     saved, cfg.W, cfg.R, factor_dims=cfg.factor_dims, dbank=gr["dbank"].clone())
    assert sdm.last_device_error(g1["workspace"]) == 0
    bank_before, dbank = bank.clone(), g1["bank"].clone()
    g2 = sdm.sdm_write_read_backward(d["q_w"], d["q_r"], d["k_val"], d["gates"], d["subkeys"], bank, gr["dy"],
                                     saved, cfg.W, cfg.R, factor_dims=cfg.factor_dims, dbank=dbank)
    assert sdm.last_device_error(g2["workspace"]) == 4          # SDM_DEVERR_SNAPSHOT
    assert torch.equal(bank, bank_before)
    assert torch.equal(dbank, g1["bank"])


@pytest.mark.parametrize("name,T,stream", [("layer", 4096, (1, 0)), ("train_fwd", 1024, (5, 1))])
def test_full_size_sampled_stream(name, T, stream):
    """Full-size shapes (N = 65536 slots, d_v = 1024, W = R = 64, every stream on the
    GPU); one sampled stream compared with the oracle, every token of it."""
    cfg = CONFIGS[name].replace(T=T)
    d = sdm_inputs.make_inputs(cfg)
    gr = sdm_inputs.make_grad_inputs(cfg, dbank=False)
    gpu = gpu_train_backward(cfg, d, gr)
    check_restored(cfg, gpu, "f32")
    o, near = oracle_backward(cfg, d, gr, gpu, stream=stream)
    print(f"{name}: {T} tokens of stream {stream} compared, {near} near-tie picks followed")
    compare_grads(cfg, gpu, o, stream=stream)
