"""CUDA-graph capture of the write/read op and of the decode step.

A call allocates nothing and never synchronises; after the first call of a shape the
library makes only stream-ordered CUDA calls (kernel launches, one memset of the error
flag, and the event fork/join of the bank-copy side stream).  A captured call must
therefore replay exactly the work of an eager call: the tests compare bit for bit, and
also after new inputs are copied into the captured buffers.
"""

import pytest
import torch

import sdm_inputs
from sdm_inputs import CONFIGS
from sdm_testlib import to_device

pytestmark = pytest.mark.gpu

_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def sdm():
    import gated_delta_rule_factor_gb300 as m
    return m


def _write_read_buffers(sdm, cfg, g):
    B, T, H = g["q_w"].shape[:3]
    bank = torch.empty((B, H, cfg.N, cfg.d_v), dtype=_TORCH[cfg.bank_dtype], device="cuda")
    y = torch.empty_like(g["k_val"])
    sh = sdm.make_shape(B=B, T=T, H=H, factor_dims=cfg.factor_dims, d_sub=cfg.d_sub, d_v=cfg.d_v,
                        W=cfg.W, R=cfg.R, chunk_size=cfg.chunk_size,
                        act_dtype=0 if cfg.act_dtype == "f32" else 1,
                        bank_dtype=0 if cfg.bank_dtype == "f32" else 1)
    ws = torch.empty(sdm.write_read_workspace_size(sh), dtype=torch.uint8, device="cuda")
    return bank, y, ws


@pytest.mark.parametrize("name,T", [("tiny", 200), ("layer", 128)])
def test_write_read_graph_replay_is_bitwise_eager(sdm, name, T):
    cfg = CONFIGS[name]
    g = to_device(sdm_inputs.make_inputs(cfg, T=T))
    bank, y, ws = _write_read_buffers(sdm, cfg, g)

    def call():
        sdm.sdm_write_read(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], bank, cfg.chunk_size,
                           cfg.W, cfg.R, factor_dims=cfg.factor_dims, bank_init=g["bank_init"], y=y,
                           workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):      # warm-up off the capture, as torch asks
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    want_y, want_bank = y.clone(), bank.clone()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    y.zero_()
    bank.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert sdm.last_device_error(ws) == 0
    assert torch.equal(y, want_y) and torch.equal(bank, want_bank)

    # new inputs in the captured buffers: the replay follows them
    fresh = to_device(sdm_inputs.make_inputs(cfg, T=T, seed=cfg.seed + 11))
    for k in ("q_w", "q_r", "k_val", "gates"):
        g[k].copy_(fresh[k])
    graph.replay()
    torch.cuda.synchronize()
    got_y, got_bank = y.clone(), bank.clone()
    call()
    torch.cuda.synchronize()
    assert torch.equal(got_y, y) and torch.equal(got_bank, bank)
    assert not torch.equal(got_y, want_y)


def test_decode_graph_steps_are_bitwise_eager(sdm):
    cfg = CONFIGS["decode"].replace(B=8)
    steps = 6
    d = to_device(sdm_inputs.make_decode_inputs(cfg, steps=steps))
    per_step = [tuple(d[k][:, t].contiguous() for k in ("q_w", "q_r", "k_val", "gates")) for t in range(steps)]
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")

    # eager reference: donated steps from the same start
    state = d["bank"].clone()
    ys = []
    for t in range(steps):
        y, state = sdm.sdm_decode_step(*per_step[t], d["subkeys"], state, cfg.W, cfg.R,
                                       factor_dims=cfg.factor_dims, donate=True, workspace=ws)
        ys.append(y.clone())
    torch.cuda.synchronize()

    # captured: one donated step on fixed input buffers, replayed per token
    inp = tuple(x.clone() for x in per_step[0])
    gstate = d["bank"].clone()
    gy = torch.empty_like(ys[0])

    def call():
        _, out = sdm.sdm_decode_step(*inp, d["subkeys"], gstate, cfg.W, cfg.R, factor_dims=cfg.factor_dims,
                                     donate=True, y=gy, workspace=ws)
        assert out.data_ptr() == gstate.data_ptr()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    warm = gstate.clone()
    with torch.cuda.stream(side):      # warm-up on a copy of the state
        sdm.sdm_decode_step(*inp, d["subkeys"], warm, cfg.W, cfg.R, factor_dims=cfg.factor_dims,
                            donate=True, y=gy, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for t in range(steps):
        for buf, x in zip(inp, per_step[t]):
            buf.copy_(x)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(gy, ys[t]), t
    assert torch.equal(gstate, state)
    assert sdm.last_device_error(ws) == 0


def test_decode_copy_form_captures(sdm):
    cfg = CONFIGS["decode"].replace(B=4)
    d = to_device(sdm_inputs.make_decode_inputs(cfg, steps=1))
    inp = tuple(d[k][:, 0].contiguous() for k in ("q_w", "q_r", "k_val", "gates"))
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    y_e, out_e = sdm.sdm_decode_step(*inp, d["subkeys"], d["bank"], cfg.W, cfg.R, factor_dims=cfg.factor_dims,
                                     donate=False, workspace=ws)
    torch.cuda.synchronize()
    out = torch.empty_like(out_e)
    y = torch.empty_like(y_e)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        sdm.sdm_decode_step(*inp, d["subkeys"], d["bank"], cfg.W, cfg.R, factor_dims=cfg.factor_dims,
                            donate=False, bank_out=out, y=y, workspace=ws)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, out_e) and torch.equal(y, y_e)
    assert sdm.last_device_error(ws) == 0


def _capture_and_compare(call, outputs, check):
    """Warm up off the capture, capture one call, zero the outputs, replay: the replay
    gives the eager results bit for bit."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    want = {k: v.clone() for k, v in outputs.items()}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for v in outputs.values():
        v.zero_()
    graph.replay()
    torch.cuda.synchronize()
    check()
    for k, v in outputs.items():
        assert torch.equal(v, want[k]), k
    return graph


def test_training_step_graph_replay_is_bitwise_eager(sdm):
    """The training pair (forward with snapshot, dL/d(final bank) = 0, backward) captured as
    one graph: every replay arms and spends the snapshot, restores the bank and gives the
    eager gradients bit for bit."""
    cfg = CONFIGS["tiny"].replace(W=64, R=64, T=96, d_v=128, act_dtype="bf16", bank_dtype="bf16")
    g = to_device(sdm_inputs.make_inputs(cfg))
    gr = to_device(sdm_inputs.make_grad_inputs(cfg, dbank=False))
    bank, y, ws = _write_read_buffers(sdm, cfg, g)
    shape = sdm.make_shape(B=cfg.B, T=cfg.T, H=cfg.H, factor_dims=cfg.factor_dims, d_sub=cfg.d_sub, d_v=cfg.d_v,
                           W=cfg.W, R=cfg.R, chunk_size=cfg.chunk_size, act_dtype=1, bank_dtype=1)
    bws = torch.empty(sdm.backward_workspace_size(shape), dtype=torch.uint8, device="cuda")
    dbank = torch.zeros((cfg.B, cfg.H, cfg.N, cfg.d_v), dtype=torch.float32, device="cuda")
    saved = sdm.sdm_write_read_train(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], bank, cfg.chunk_size,
                                     cfg.W, cfg.R, factor_dims=cfg.factor_dims, bank_init=g["bank_init"],
                                     snapshot_dtype=torch.bfloat16, y=y, workspace=ws)
    grads = sdm.sdm_write_read_backward(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], bank, gr["dy"],
                                        saved, cfg.W, cfg.R, factor_dims=cfg.factor_dims, dbank=dbank,
                                        workspace=bws)
    grads.pop("workspace")

    def call():
        sdm.sdm_write_read_train(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], bank, cfg.chunk_size,
                                 cfg.W, cfg.R, factor_dims=cfg.factor_dims, bank_init=g["bank_init"],
                                 snapshot_dtype=torch.bfloat16, saved=saved, y=y, workspace=ws)
        dbank.zero_()
        sdm.sdm_write_read_backward(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], bank, gr["dy"],
                                    saved, cfg.W, cfg.R, factor_dims=cfg.factor_dims, dbank=dbank, grads=grads,
                                    workspace=bws)

    outs = {("d_" + k): v for k, v in grads.items()}          # d_bank is the gradient table
    outs.update(y=y, bank=bank)

    def check():
        assert sdm.last_device_error(ws) == 0 and sdm.last_device_error(bws) == 0

    _capture_and_compare(call, outs, check)
    assert torch.equal(bank, g["bank_init"].unsqueeze(0).expand_as(bank))   # restored


def test_layer_forward_graph_replay_is_bitwise_eager(sdm):
    """The layer forward (cuBLASLt projections included) captured and replayed."""
    cfg = CONFIGS["tiny"].replace(act_dtype="bf16", factor_dims=(16, 16), d_sub=32, d_v=64, H=2, B=2, T=48,
                                  W=16, R=16)
    dim = 128
    L = to_device(sdm_inputs.make_layer_inputs(cfg, dim))
    bank = torch.empty((cfg.B, cfg.H, cfg.N, cfg.d_v), dtype=L["bank_init"].dtype, device="cuda")
    out = torch.empty_like(L["x"])
    shape = sdm.make_shape(B=cfg.B, T=cfg.T, H=cfg.H, factor_dims=cfg.factor_dims, d_sub=cfg.d_sub, d_v=cfg.d_v,
                           W=cfg.W, R=cfg.R, chunk_size=cfg.chunk_size, act_dtype=1, bank_dtype=0)
    ws = torch.empty(sdm.layer_workspace_size(shape, dim), dtype=torch.uint8, device="cuda")

    def call():
        sdm.sdm_layer_forward(L["x"], L["w_qw"], L["w_qr"], L["w_v"], L["w_g"], L["w_o"], L["subkeys"], bank,
                              cfg.chunk_size, cfg.W, cfg.R, factor_dims=cfg.factor_dims, bank_init=L["bank_init"],
                              out=out, workspace=ws)

    _capture_and_compare(call, {"out": out, "bank": bank}, lambda: None)
    assert sdm.last_device_error(ws) == 0
