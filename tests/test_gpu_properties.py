"""Properties of the CUDA path that hold at any size: bitwise repeatability, chunk-size
independence, the identity update, decode copy == donate, in-place donation, the
decode step against the oracle and against the write/read op, refusals with real
tensors, launch counting and per-kernel timing."""

import numpy as np
import pytest
import torch

import oracle
import sdm_inputs
from sdm_inputs import CONFIGS
from sdm_testlib import RTOL, assert_close, check_selection, gpu_write_read, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdm():
    import gated_delta_rule_factor_gb300 as m
    return m


def _same(a: dict, b: dict):
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_bitwise_repeatable_layer_shape():
    cfg = CONFIGS["layer"]
    d = sdm_inputs.make_inputs(cfg)
    first = gpu_write_read(cfg, d)
    for _ in range(2):
        _same(first, gpu_write_read(cfg, d))


@pytest.mark.parametrize("name,T", [("tiny", 256), ("three_factor", 1024)])
def test_chunk_size_changes_nothing(name, T):
    # the planner's chunk only groups tokens for staging; tokens still apply one at a time
    cfg = CONFIGS[name]
    d = sdm_inputs.make_inputs(cfg, T=T)
    ref = gpu_write_read(cfg, d, chunk_size=64)
    for c in (1, 3, 17, 128, 256):
        _same(ref, gpu_write_read(cfg, d, chunk_size=c))


def test_forget_one_input_zero_leaves_bank_bitwise_unchanged():
    cfg = CONFIGS["tiny"].replace(B=2, H=2, T=64)
    d = sdm_inputs.make_inputs(cfg)
    d["gates"][..., 0] = 1.0
    d["gates"][..., 1] = 0.0
    out = gpu_write_read(cfg, d)
    want = d["bank_init"].unsqueeze(0).expand(2, *d["bank_init"].shape)
    assert torch.equal(out["bank"], want)


def test_identity_update_reads_a_weighted_gather():
    cfg = CONFIGS["tiny"].replace(T=32)
    d = sdm_inputs.make_inputs(cfg)
    d["gates"][..., 0] = 1.0
    d["gates"][..., 1] = 0.0
    out = gpu_write_read(cfg, d)
    M = d["bank_init"][0].double()
    idx, w = out["idx_r"][0, :, 0].long(), out["wt_r"][0, :, 0].double()
    want = (w[..., None] * M[idx]).sum(1)
    assert_close(out["y"][0, :, 0], want, 1e-5, "y")


def test_single_full_strength_write_stores_the_value():
    cfg = CONFIGS["tiny"].replace(W=1, R=1, T=32)
    d = sdm_inputs.make_inputs(cfg)
    d["gates"][..., 1] = 1.0
    d["q_r"] = d["q_w"].clone()
    out = gpu_write_read(cfg, d)
    # W = 1, beta = 1: the written row becomes v; reading the same slot returns it
    assert torch.equal(out["idx_w"], out["idx_r"])
    assert torch.equal(out["wt_w"], torch.ones_like(out["wt_w"]))
    # fl(m + fl(v - m)) is v up to one rounding of the float32 update
    assert_close(out["y"], d["k_val"], 1e-6, "y = v")


def test_refusals_with_real_tensors(sdm):
    cfg = CONFIGS["tiny"]
    g = to_device(sdm_inputs.make_inputs(cfg, T=8))
    bank = torch.zeros((1, 1, cfg.N, cfg.d_v), device="cuda")
    with pytest.raises(sdm.SdmError) as e:
        sdm.sdm_write_read(g["q_w"].half(), g["q_r"].half(), g["k_val"].half(), g["gates"],
                           g["subkeys"].half(), bank, 64, 8, 8, factor_dims=cfg.factor_dims)
    assert e.value.status == 2
    with pytest.raises(sdm.SdmError) as e:
        sdm.sdm_write_read(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], bank, 64,
                           2000, 8, factor_dims=cfg.factor_dims)
    assert e.value.status == 1
    with pytest.raises(sdm.SdmError) as e:   # y written over the values
        sdm.sdm_write_read(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], bank, 64,
                           8, 8, factor_dims=cfg.factor_dims, y=g["k_val"])
    assert e.value.status == 3


def test_launch_count_and_kernel_timing(sdm):
    cfg = CONFIGS["tiny"]
    g = to_device(sdm_inputs.make_inputs(cfg))
    bank = torch.empty((1, 1, cfg.N, cfg.d_v), device="cuda")
    before = sdm.launch_count()
    sdm.profile_begin()
    for _ in range(3):
        sdm.sdm_write_read(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], bank, 64, 8, 8,
                           factor_dims=cfg.factor_dims, bank_init=g["bank_init"])
    times = sdm.profile_end()
    assert sdm.launch_count() - before == 18    # copy, score, select, 2 plan kernels, write/read
    for k in ("bank_copy", "score", "select", "plan_sort", "plan_link", "write_read"):
        assert times[k][0] == 3 and times[k][1] > 0


def test_non_default_stream(sdm):
    cfg = CONFIGS["tiny"]
    d = sdm_inputs.make_inputs(cfg)
    ref = gpu_write_read(cfg, d)
    g = to_device(d)
    bank = torch.empty((1, 1, cfg.N, cfg.d_v), device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = sdm.sdm_write_read(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], bank, 64, 8,
                               8, factor_dims=cfg.factor_dims, bank_init=g["bank_init"], stream=s)
    s.synchronize()
    assert torch.equal(y.cpu(), ref["y"]) and torch.equal(bank.cpu(), ref["bank"])


# --------------------------------------------------------------------------- decode

def _step_inputs(g, t):
    """Token t of every stream, as contiguous [B, H, ...] tensors."""
    return tuple(g[k][:, t].contiguous() for k in ("q_w", "q_r", "k_val", "gates"))


def _decode_steps(sdm, cfg, d, steps, donate, sel=None):
    """Run `steps` decode steps; every step writes its selections into fresh buffers and
    its workspace flag is read back (a kernel-side error fails the test).  With a dict
    `sel`, the per-step idx_w, wt_w, idx_r, wt_r [B, steps, H, k] are stored in it."""
    g = to_device(d)
    state = g["bank"].clone()
    B, H = cfg.B, cfg.H
    ys, got = [], {k: [] for k in ("idx_w", "wt_w", "idx_r", "wt_r")}
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    for t in range(steps):
        out = {"idx_w": torch.empty((B, H, cfg.W), dtype=torch.int32, device="cuda"),
               "wt_w": torch.empty((B, H, cfg.W), dtype=torch.float32, device="cuda"),
               "idx_r": torch.empty((B, H, cfg.R), dtype=torch.int32, device="cuda"),
               "wt_r": torch.empty((B, H, cfg.R), dtype=torch.float32, device="cuda")}
        y, new = sdm.sdm_decode_step(*_step_inputs(g, t), g["subkeys"], state, cfg.W, cfg.R,
                                     factor_dims=cfg.factor_dims, donate=donate, workspace=ws, **out)
        assert (new.data_ptr() == state.data_ptr()) == donate   # in place exactly when donating
        assert sdm.last_device_error(ws) == 0, f"step {t}: kernel-side error"
        ys.append(y.clone())
        for k in got:
            got[k].append(out[k].cpu())
        state = new
    torch.cuda.synchronize()
    if sel is not None:
        sel.update({k: torch.stack(v, 1) for k, v in got.items()})
    return torch.stack(ys, 1).cpu(), state.cpu()


def _check_decode_selections(cfg, d, sel, t):
    """Step t's selections of every stream against the oracle's (exact under the margin
    rule; a valid near-tie alternative is counted and returned)."""
    near = 0
    for b in range(cfg.B):
        for h in range(cfg.H):
            K = d["subkeys"][h].float().double().numpy()
            for name, wname, qk, k in (("idx_w", "wt_w", "q_w", cfg.W), ("idx_r", "wt_r", "q_r", cfg.R)):
                q = d[qk][b, t, h].float().double().numpy()
                oi, ow, _ = oracle.select(q, K, cfg.factor_dims, cfg.d_sub, k)
                near += 0 if check_selection(cfg, q, K, k, sel[name][b, t, h].numpy(),
                                             sel[wname][b, t, h].numpy(), oi, ow) else 1
    return near


def test_decode_copy_equals_donate_bitwise(sdm):
    cfg = CONFIGS["decode"]
    d = sdm_inputs.make_decode_inputs(cfg, steps=16)
    y_c, b_c = _decode_steps(sdm, cfg, d, 16, donate=False)
    y_d, b_d = _decode_steps(sdm, cfg, d, 16, donate=True)
    assert torch.equal(y_c, y_d) and torch.equal(b_c, b_d)


def test_decode_copy_leaves_the_old_state_and_donate_reuses_it(sdm):
    cfg = CONFIGS["decode"].replace(B=4)
    d = sdm_inputs.make_decode_inputs(cfg, steps=2)
    g = to_device(d)
    bank = g["bank"].clone()
    keep = bank.clone()
    y, new = sdm.sdm_decode_step(*_step_inputs(g, 0), g["subkeys"], bank, cfg.W, cfg.R,
                                 factor_dims=cfg.factor_dims)
    assert new.data_ptr() != bank.data_ptr() and torch.equal(bank, keep)
    y2, same = sdm.sdm_decode_step(*_step_inputs(g, 0), g["subkeys"], bank, cfg.W, cfg.R,
                                   factor_dims=cfg.factor_dims, donate=True)
    assert same.data_ptr() == bank.data_ptr()
    assert torch.equal(same, new) and torch.equal(y, y2)
    assert not torch.equal(bank, keep)              # the predecessor really was overwritten


def test_decode_from_a_learned_table_never_writes_it(sdm):
    cfg = CONFIGS["decode"].replace(B=3)
    d = sdm_inputs.make_decode_inputs(cfg, steps=3)
    g = to_device(d)
    table = g["bank"][0].clone()                     # [H, N, d_v]
    table_keep = table.clone()
    state = table.unsqueeze(0).expand(cfg.B, *table.shape)   # init_state's broadcast
    for t in range(3):
        y, state = sdm.sdm_decode_step(*_step_inputs(g, t), g["subkeys"], state, cfg.W, cfg.R,
                                       factor_dims=cfg.factor_dims, donate=True)
    assert torch.equal(table, table_keep)
    # and the result equals stepping from materialised tables
    y_ref, b_ref = _decode_steps(sdm, cfg, d, 3, donate=False)
    assert torch.equal(state.cpu(), b_ref)


def _decode_against_oracle(sdm, cfg, d, steps, tol):
    """Donated steps against the oracle: selections (exact under the margin rule), y and
    the final bank.  The oracle's bank follows the GPU's selection when a step took a
    valid near-tie alternative, so the comparison never stops early."""
    sel = {}
    y_gpu, b_gpu = _decode_steps(sdm, cfg, d, steps, donate=True, sel=sel)
    bank = d["bank"].float().double().numpy().copy()
    near = 0
    for t in range(steps):
        near += _check_decode_selections(cfg, d, sel, t)
        y_o = np.zeros((cfg.B, cfg.H, cfg.d_v))
        for b in range(cfg.B):
            for h in range(cfg.H):
                gi = {0: sel["idx_w"][b, t, h].numpy(), 1: sel["idx_r"][b, t, h].numpy()}

                def follow(tt, which, idx, w, gi=gi):
                    return None if np.array_equal(gi[which], idx) else gi[which]

                K = d["subkeys"][h].float().double().numpy()
                res = oracle.run_stream(bank[b, h], d["q_w"][b, t:t + 1, h].float().double().numpy(),
                                        d["q_r"][b, t:t + 1, h].float().double().numpy(),
                                        d["k_val"][b, t:t + 1, h].float().double().numpy(),
                                        d["gates"][b, t:t + 1, h].double().numpy(), K,
                                        factor_dims=cfg.factor_dims, d_sub=cfg.d_sub, W=cfg.W, R=cfg.R,
                                        act_dtype=cfg.act_dtype, bank_dtype=cfg.bank_dtype, pick=follow)
                y_o[b, h] = res["y"][0]
        assert_close(y_gpu[:, t], y_o, tol, f"decode y step {t}")
    assert_close(b_gpu, bank, tol, "decode bank")
    return near


def test_decode_matches_oracle(sdm):
    cfg = CONFIGS["decode"].replace(B=16)
    d = sdm_inputs.make_decode_inputs(cfg, steps=3)
    assert _decode_against_oracle(sdm, cfg, d, 3, RTOL["f32"]) <= 1


def test_decode_grid_inputs_select_identically(sdm):
    # exact scores (grid inputs): the decode step's selections equal the oracle's bit for
    # bit, order and ties included
    cfg = CONFIGS["decode"].replace(B=8)
    d = sdm_inputs.make_decode_inputs(cfg, steps=2, grid=True)
    sel = {}
    _decode_steps(sdm, cfg, d, 2, donate=True, sel=sel)
    ties = 0
    for t in range(2):
        for b in range(cfg.B):
            for h in range(cfg.H):
                K = d["subkeys"][h].float().double().numpy()
                for name, qk, k in (("idx_w", "q_w", cfg.W), ("idx_r", "q_r", cfg.R)):
                    q = d[qk][b, t, h].float().double().numpy()
                    oi, _, S_sel = oracle.select(q, K, cfg.factor_dims, cfg.d_sub, k)
                    np.testing.assert_array_equal(sel[name][b, t, h].numpy(), oi, err_msg=f"{name} {b},{t},{h}")
                    ties += int(len(np.unique(S_sel)) < len(S_sel))
    assert ties > 0, "grid inputs produced no tie inside the top k"
    assert _decode_against_oracle(sdm, cfg, d, 2, RTOL["f32"]) == 0


def test_decode_steps_equal_the_write_read_op(sdm):
    cfg = CONFIGS["tiny"].replace(B=2, H=2, T=12)
    d = sdm_inputs.make_inputs(cfg)
    wr = gpu_write_read(cfg, d)
    dd = dict(d)
    bi = dd.pop("bank_init")
    dd["bank"] = bi.unsqueeze(0).expand(cfg.B, *bi.shape).contiguous()
    y_dec, b_dec = _decode_steps(sdm, cfg.replace(T=1), dd, cfg.T, donate=True)
    assert_close(y_dec, wr["y"], 1e-5, "decode vs write_read y")
    assert_close(b_dec, wr["bank"], 1e-5, "decode vs write_read bank")


def test_decode_bf16(sdm):
    cfg = CONFIGS["decode"].replace(B=8, act_dtype="bf16", bank_dtype="bf16")
    d = sdm_inputs.make_decode_inputs(cfg, steps=2)
    y_c, b_c = _decode_steps(sdm, cfg, d, 2, donate=False)
    y_d, b_d = _decode_steps(sdm, cfg, d, 2, donate=True)
    assert torch.equal(y_c, y_d) and torch.equal(b_c, b_d)
    assert _decode_against_oracle(sdm, cfg, d, 2, RTOL["bf16"]) <= 1


# Decode shapes beyond the benchmark's: bfloat16 rows (8 per 16-byte group), a d_v whose
# last column block is partly past the row end, W != R with three factors, and the
# largest k.  Each runs donated and copying steps (bit-equal) against the oracle.
_DECODE_SHAPES = {
    "bf16_bank_and_acts": dict(act_dtype="bf16", bank_dtype="bf16", B=4),
    "ragged_d_v": dict(d_v=104, B=3),
    "bf16_bank_ragged_d_v": dict(bank_dtype="bf16", d_v=72, B=3),
    "w_ne_r_three_factors": dict(factor_dims=(8, 8, 16), d_sub=32, W=8, R=24, B=3),
    "max_k": dict(W=128, R=128, B=2),
}


@pytest.mark.parametrize("name", sorted(_DECODE_SHAPES))
def test_decode_shapes_against_oracle(sdm, name):
    cfg = CONFIGS["decode"].replace(**_DECODE_SHAPES[name])
    steps = 3
    d = sdm_inputs.make_decode_inputs(cfg, steps=steps)
    y_d, b_d = _decode_steps(sdm, cfg, d, steps, donate=True)
    y_c, b_c = _decode_steps(sdm, cfg, d, steps, donate=False)
    assert torch.equal(y_d, y_c) and torch.equal(b_d, b_c)
    tol = RTOL[cfg.bank_dtype if cfg.bank_dtype == "bf16" else cfg.act_dtype]
    assert _decode_against_oracle(sdm, cfg, d, steps, tol) <= 1


def test_decode_copy_wait_that_runs_out_reports_timeout_and_the_context_survives(sdm):
    # The copy thread's bounded mbarrier wait is made to run out (a barrier nothing
    # arrives at): the step completes, the workspace flag reads SDM_DEVERR_TIMEOUT, and
    # the next step on the same context is correct again.
    SDM_DEVERR_TIMEOUT = 3
    cfg = CONFIGS["decode"].replace(B=2)
    d = to_device(sdm_inputs.make_decode_inputs(cfg, steps=1))
    inp = tuple(d[k][:, 0].contiguous() for k in ("q_w", "q_r", "k_val", "gates"))
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    y_ref, out_ref = sdm.sdm_decode_step(*inp, d["subkeys"], d["bank"], cfg.W, cfg.R,
                                         factor_dims=cfg.factor_dims, donate=False, workspace=ws)
    torch.cuda.synchronize()
    assert sdm.last_device_error(ws) == 0
    sdm.test_stall_decode_copy(True)
    try:
        sdm.sdm_decode_step(*inp, d["subkeys"], d["bank"], cfg.W, cfg.R, factor_dims=cfg.factor_dims,
                            donate=False, workspace=ws)
        torch.cuda.synchronize()
        assert sdm.last_device_error(ws) == SDM_DEVERR_TIMEOUT
    finally:
        sdm.test_stall_decode_copy(False)
    y, out = sdm.sdm_decode_step(*inp, d["subkeys"], d["bank"], cfg.W, cfg.R, factor_dims=cfg.factor_dims,
                                 donate=False, workspace=ws)
    torch.cuda.synchronize()
    assert sdm.last_device_error(ws) == 0
    assert torch.equal(y, y_ref) and torch.equal(out, out_ref)
