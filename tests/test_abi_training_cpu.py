"""Host-side tests of the training pair, the layer entry and the factor-score hook that
need no GPU.

Every refusal of sdm_write_read_train, sdm_write_read_backward, sdm_layer_forward and
sdm_test_factor_scores is decided on the host before any CUDA call or launch, so these
calls pass fake (never dereferenced) device addresses, as in test_abi_cpu.py.  Also
checked: the snapshot size follows the documented layout, the workspace sizes depend only
on the shape, and a float32 shape's workspace holds the scorer's split of the queries.
"""

import ctypes

import pytest

from test_abi_cpu import fake, lib, shape, ws_size  # noqa: F401  (lib is a fixture)

from gated_delta_rule_factor_gb300 import _abi  # noqa: E402


def snap_bytes(lib, sh, dt):
    n = ctypes.c_size_t(0)
    st = lib.sdm_snapshot_bytes(ctypes.byref(sh), dt, ctypes.byref(n))
    return st, n.value


def bwd_ws(lib, sh):
    n = ctypes.c_size_t(0)
    st = lib.sdm_write_read_backward_workspace_size(ctypes.byref(sh), ctypes.byref(n))
    return st, n.value


@pytest.mark.parametrize("bank_dtype", [_abi.SDM_F32, _abi.SDM_BF16])
def test_snapshot_size_follows_the_documented_layout(lib, bank_dtype):
    # a 256-byte header, then per stream, token and 32-byte piece of a row, the W rows'
    # pieces in the snapshot type
    sh = shape(B=3, T=10, H=2, d_v=72, W=5, bank_dtype=bank_dtype)
    eb = 4 if bank_dtype == _abi.SDM_F32 else 2
    pieces = -(-(72 * eb) // 32)
    cols = 32 // eb
    for dt, se in ((_abi.SDM_F32, 4), (_abi.SDM_BF16, 2)):
        st, n = snap_bytes(lib, sh, dt)
        assert st == _abi.SDM_OK
        assert n == 256 + 3 * 2 * 10 * pieces * 5 * cols * se
    assert snap_bytes(lib, sh, _abi.SDM_F16)[0] == _abi.SDM_ERR_UNSUPPORTED
    assert snap_bytes(lib, sh, 9)[0] == _abi.SDM_ERR_INVALID_ARG


def test_backward_workspace_size_depends_only_on_shape(lib):
    sizes = {bwd_ws(lib, shape())[1] for _ in range(3)}
    assert len(sizes) == 1 and sizes.pop() > 0
    assert bwd_ws(lib, shape(T=4096))[1] > bwd_ws(lib, shape())[1]


def call_train(lib, sh, **over):
    st, nb = snap_bytes(lib, sh, _abi.SDM_F32)
    assert st == _abi.SDM_OK
    p = dict(q_w=fake(1), q_r=fake(2), k_val=fake(3), gates=fake(4), subkeys=fake(5), bank_init=None,
             bank=fake(6), y=fake(7), idx_w=fake(9), wt_w=fake(10), idx_r=fake(11), wt_r=fake(12),
             snap=fake(13), snap_bytes=nb, snap_dt=_abi.SDM_F32, ws=fake(8), ws_bytes=ws_size(lib, sh)[1])
    p.update(over)
    return lib.sdm_write_read_train(ctypes.byref(sh), p["q_w"], p["q_r"], p["k_val"], p["gates"], p["subkeys"],
                                    p["bank_init"], p["bank"], p["y"], p["idx_w"], p["wt_w"], p["idx_r"],
                                    p["wt_r"], p["snap"], p["snap_bytes"], p["snap_dt"], p["ws"], p["ws_bytes"],
                                    None)


@pytest.mark.parametrize("over,status", [
    (dict(snap=None), _abi.SDM_ERR_INVALID_ARG),
    (dict(snap=fake(13) + 8), _abi.SDM_ERR_INVALID_ARG),          # misaligned
    (dict(snap_bytes=1024), _abi.SDM_ERR_INVALID_ARG),             # short
    (dict(snap_dt=_abi.SDM_F16), _abi.SDM_ERR_UNSUPPORTED),
    (dict(idx_w=None), _abi.SDM_ERR_INVALID_ARG),                  # the backward reads the selections
    (dict(wt_r=fake(12) + 4), _abi.SDM_ERR_INVALID_ARG),           # 16-byte aligned here
    (dict(snap=fake(6)), _abi.SDM_ERR_ALIAS),                      # snapshot over the bank
])
def test_train_refusals_enqueue_nothing(lib, over, status):
    before = lib.sdm_launch_count()
    assert call_train(lib, shape(), **over) == status, lib.sdm_last_error_message()
    assert lib.sdm_launch_count() == before


def call_backward(lib, sh, **over):
    st, nb = snap_bytes(lib, sh, _abi.SDM_F32)
    p = dict(q_w=fake(1), q_r=fake(2), k_val=fake(3), gates=fake(4), subkeys=fake(5), idx_w=fake(9),
             wt_w=fake(10), idx_r=fake(11), wt_r=fake(12), snap=fake(13), snap_bytes=nb, snap_dt=_abi.SDM_F32,
             bank=fake(6), dy=fake(14), dbank=fake(15), d_kv=fake(16), d_g=fake(17), d_qw=fake(18),
             d_qr=fake(19), d_sk=fake(20), ws=fake(8), ws_bytes=bwd_ws(lib, sh)[1])
    p.update(over)
    return lib.sdm_write_read_backward(
        ctypes.byref(sh), p["q_w"], p["q_r"], p["k_val"], p["gates"], p["subkeys"], p["idx_w"], p["wt_w"],
        p["idx_r"], p["wt_r"], p["snap"], p["snap_bytes"], p["snap_dt"], p["bank"], p["dy"], p["dbank"],
        p["d_kv"], p["d_g"], p["d_qw"], p["d_qr"], p["d_sk"], p["ws"], p["ws_bytes"], None)


@pytest.mark.parametrize("over,status", [
    (dict(snap=None), _abi.SDM_ERR_INVALID_ARG),
    (dict(dy=None), _abi.SDM_ERR_INVALID_ARG),
    (dict(dbank=fake(15) + 4), _abi.SDM_ERR_INVALID_ARG),          # misaligned
    (dict(snap_bytes=512), _abi.SDM_ERR_INVALID_ARG),              # short snapshot
    (dict(snap_dt=_abi.SDM_F16), _abi.SDM_ERR_UNSUPPORTED),
    (dict(ws=None), _abi.SDM_ERR_WORKSPACE),
    (dict(ws_bytes=1024), _abi.SDM_ERR_WORKSPACE),
    (dict(dbank=fake(6)), _abi.SDM_ERR_ALIAS),                     # gradient table over the bank
    (dict(d_qw=fake(1)), _abi.SDM_ERR_ALIAS),                      # an output over an input
    (dict(d_sk=fake(16) + 256), _abi.SDM_ERR_ALIAS),               # two outputs overlapping
])
def test_backward_refusals_enqueue_nothing(lib, over, status):
    before = lib.sdm_launch_count()
    assert call_backward(lib, shape(), **over) == status, lib.sdm_last_error_message()
    assert lib.sdm_launch_count() == before


def layer_ws(lib, sh, dim):
    n = ctypes.c_size_t(0)
    st = lib.sdm_layer_workspace_size(ctypes.byref(sh), dim, ctypes.byref(n))
    return st, n.value


def call_layer(lib, sh, dim=96, **over):
    p = dict(x=fake(1), w_qw=fake(2), w_qr=fake(3), w_v=fake(4), w_g=fake(5), w_o=fake(6), subkeys=fake(7),
             bank_init=None, bank=fake(9), out=fake(10), q_w=None, q_r=None, k_val=None, gates=None, y=None,
             ws=fake(11), ws_bytes=layer_ws(lib, sh, dim)[1])
    p.update(over)
    return lib.sdm_layer_forward(ctypes.byref(sh), dim, p["x"], p["w_qw"], p["w_qr"], p["w_v"], p["w_g"], p["w_o"],
                                 p["subkeys"], p["bank_init"], p["bank"], p["out"], p["q_w"], p["q_r"],
                                 p["k_val"], p["gates"], p["y"], p["ws"], p["ws_bytes"], None)


def test_layer_workspace_size(lib):
    st, n = layer_ws(lib, shape(), 96)
    assert st == _abi.SDM_OK and n > ws_size(lib, shape())[1]
    assert layer_ws(lib, shape(), 0)[0] == _abi.SDM_ERR_INVALID_ARG


@pytest.mark.parametrize("over,status", [
    (dict(dim=0), _abi.SDM_ERR_INVALID_ARG),
    (dict(x=None), _abi.SDM_ERR_INVALID_ARG),
    (dict(w_o=fake(6) + 8), _abi.SDM_ERR_INVALID_ARG),             # misaligned
    (dict(ws_bytes=4096), _abi.SDM_ERR_WORKSPACE),
    (dict(ws=fake(11) + 16), _abi.SDM_ERR_WORKSPACE),              # the layer wants 256-byte alignment
    (dict(out=fake(1)), _abi.SDM_ERR_ALIAS),                       # out over x
    (dict(q_w=fake(2)), _abi.SDM_ERR_ALIAS),                       # a kept intermediate over a weight
])
def test_layer_refusals_enqueue_nothing(lib, over, status):
    before = lib.sdm_launch_count()
    dim = over.pop("dim", 96)
    assert call_layer(lib, shape(), dim=dim, **over) == status, lib.sdm_last_error_message()
    assert lib.sdm_launch_count() == before


def call_scores(lib, sh, **over):
    p = dict(q_w=fake(1), q_r=fake(2), subkeys=fake(5), scores=fake(9), ws=fake(8), ws_bytes=ws_size(lib, sh)[1])
    p.update(over)
    return lib.sdm_test_factor_scores(ctypes.byref(sh), p["q_w"], p["q_r"], p["subkeys"], p["scores"], p["ws"],
                                      p["ws_bytes"], None)


@pytest.mark.parametrize("act", [_abi.SDM_F32, _abi.SDM_BF16])
def test_float32_workspace_holds_the_score_split(lib, act):
    # float32 queries are split into four bfloat16 slices for the tensor cores (plus one
    # exponent per segment) inside the op's workspace; bfloat16 queries need no split
    sh = shape(act_dtype=act, d_sub=40)
    n_f32 = ws_size(lib, shape(act_dtype=_abi.SDM_F32, d_sub=40))[1]
    n_bf16 = ws_size(lib, shape(act_dtype=_abi.SDM_BF16, d_sub=40))[1]
    segments = 2 * sh.B * sh.T * sh.H * 2 + sh.H * 32        # query factor slices + sub-key rows
    assert n_f32 - n_bf16 >= segments * (4 * 64 * 2 + 4)      # d_sub 40 padded to 64
    assert ws_size(lib, sh)[0] == _abi.SDM_OK


@pytest.mark.parametrize("over,status", [
    (dict(q_w=None), _abi.SDM_ERR_INVALID_ARG),
    (dict(scores=None), _abi.SDM_ERR_INVALID_ARG),
    (dict(subkeys=fake(5) + 8), _abi.SDM_ERR_INVALID_ARG),         # misaligned
    (dict(ws_bytes=1024), _abi.SDM_ERR_WORKSPACE),
    (dict(ws=None), _abi.SDM_ERR_WORKSPACE),
    (dict(scores=fake(1)), _abi.SDM_ERR_ALIAS),                    # scores over q_w
    (dict(ws=fake(9)), _abi.SDM_ERR_ALIAS),                        # workspace over scores
])
def test_factor_score_hook_refusals_enqueue_nothing(lib, over, status):
    before = lib.sdm_launch_count()
    assert call_scores(lib, shape(), **over) == status, lib.sdm_last_error_message()
    assert lib.sdm_launch_count() == before
