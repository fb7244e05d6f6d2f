"""sdm_write_read_static: the write/read op on the library's fixed scratch array.

The entry allocates nothing; it runs the same kernels as sdm_write_read with its
scratch in a device array of the library.  The GPU test compares it with
sdm_write_read (caller workspace) on two calls in a row and wants every output bit for
bit; the CPU test checks the size refusal, which is decided before any CUDA call.  This file is collected last so that it also runs after every other test.
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import sdm_inputs

from sdm_testlib import to_device

_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16}


def _lib():
    import __graft_entry__
    __graft_entry__._build_script().build()
    from gated_delta_rule_factor_gb300 import _abi
    return _abi, _abi.load()


def _shape(_abi, cfg, T):
    sh = _abi.SdmShape()
    sh.B, sh.T, sh.H, sh.d_sub, sh.d_v = cfg.B, T, cfg.H, cfg.d_sub, cfg.d_v
    sh.F = len(cfg.factor_dims)
    for i, n in enumerate(cfg.factor_dims):
        sh.factor_dims[i] = n
    sh.W, sh.R, sh.chunk_size = cfg.W, cfg.R, cfg.chunk_size
    sh.act_dtype = 0 if cfg.act_dtype == "f32" else 1
    sh.bank_dtype = 0 if cfg.bank_dtype == "f32" else 1
    return sh


def test_static_scratch_refuses_shapes_beyond_its_size():
    _abi, lib = _lib()
    cfg = sdm_inputs.CONFIGS["layer"]
    sh = _shape(_abi, cfg, cfg.T)
    need = ctypes.c_size_t()
    assert lib.sdm_write_read_workspace_size(ctypes.byref(sh), ctypes.byref(need)) == _abi.SDM_OK
    assert need.value > _abi.STATIC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 40)
    st = lib.sdm_write_read_static(ctypes.byref(sh), fake, fake, fake, fake, fake, None, fake, fake,
                                   None, None, None, None, None)
    assert st == _abi.SDM_ERR_WORKSPACE
    msg = lib.sdm_last_error_message().decode()
    assert "static array" in msg and str(need.value) in msg


def _outputs(cfg, B, T, H, dev):
    return {"bank": torch.empty((B, H, cfg.N, cfg.d_v), dtype=_TORCH[cfg.bank_dtype], device=dev),
            "y": torch.empty((B, T, H, cfg.d_v), dtype=_TORCH[cfg.act_dtype], device=dev),
            "idx_w": torch.empty((B, T, H, cfg.W), dtype=torch.int32, device=dev),
            "wt_w": torch.empty((B, T, H, cfg.W), dtype=torch.float32, device=dev),
            "idx_r": torch.empty((B, T, H, cfg.R), dtype=torch.int32, device=dev),
            "wt_r": torch.empty((B, T, H, cfg.R), dtype=torch.float32, device=dev)}


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_on_two_calls_in_a_row():
    import gated_delta_rule_factor_gb300 as sdm
    from gated_delta_rule_factor_gb300 import _abi
    cfg = sdm_inputs.CONFIGS["layer"]
    T = 256
    dev = torch.device("cuda")
    inputs = [to_device(sdm_inputs.make_inputs(cfg, seed=cfg.seed + s, T=T)) for s in (11, 12)]
    B, H = cfg.B, cfg.H
    sh = sdm.make_shape(B=B, T=T, H=H, factor_dims=cfg.factor_dims, d_sub=cfg.d_sub, d_v=cfg.d_v,
                        W=cfg.W, R=cfg.R, chunk_size=cfg.chunk_size,
                        act_dtype=0 if cfg.act_dtype == "f32" else 1,
                        bank_dtype=0 if cfg.bank_dtype == "f32" else 1)
    assert sdm.write_read_workspace_size(sh) <= _abi.STATIC_SCRATCH_BYTES
    stat = [_outputs(cfg, B, T, H, dev) for _ in inputs]
    ref = [_outputs(cfg, B, T, H, dev) for _ in inputs]
    stream = torch.cuda.current_stream()

    def static_call(g, o):
        sdm.sdm_write_read_static(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], o["bank"],
                                  cfg.chunk_size, cfg.W, cfg.R, factor_dims=cfg.factor_dims,
                                  bank_init=g["bank_init"], y=o["y"], idx_w=o["idx_w"], wt_w=o["wt_w"],
                                  idx_r=o["idx_r"], wt_r=o["wt_r"], stream=stream)

    # the first call on the device does the set-up; the two calls compared come after it
    static_call(inputs[0], stat[0])
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for g, o in zip(inputs, stat):            # two calls in a row on the static scratch
        static_call(g, o)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "the static entry changed free device memory"

    for g, o in zip(inputs, ref):
        ws = torch.empty(sdm.write_read_workspace_size(sh), dtype=torch.uint8, device=dev)
        sdm.sdm_write_read(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], o["bank"],
                           cfg.chunk_size, cfg.W, cfg.R, factor_dims=cfg.factor_dims,
                           bank_init=g["bank_init"], y=o["y"], idx_w=o["idx_w"], wt_w=o["wt_w"],
                           idx_r=o["idx_r"], wt_r=o["wt_r"], workspace=ws, stream=stream)
        torch.cuda.synchronize()
        assert sdm.last_device_error(ws) == 0

    # the static entry runs the same kernels on the same inputs as sdm_write_read: every
    # output, the whole bank included, must be bitwise identical (this is also the only
    # check of the static path, whose kernel-side error flag no call can read)
    for i, (s, r) in enumerate(zip(stat, ref)):
        for k in ("y", "idx_w", "wt_w", "idx_r", "wt_r", "bank"):
            assert torch.equal(s[k], r[k]), f"call {i}: {k} differs from sdm_write_read"
    assert not np.array_equal(stat[0]["y"].float().cpu().numpy(), stat[1]["y"].float().cpu().numpy())
