"""Torch-tensor front end of the C ABI: sdm_write_read and sdm_decode_step.

Argument marshalling only.  Every step of the op runs in the CUDA library
(libsdm_gb300.so); PyTorch only supplies device memory and the current stream.
There is no CPU path: without the library, importing the package fails.
"""

from __future__ import annotations

import ctypes
import math
from typing import Optional, Sequence

import torch

from . import _abi

_DT = {torch.float32: _abi.SDM_F32, torch.bfloat16: _abi.SDM_BF16, torch.float16: _abi.SDM_F16}


def _dtype_code(t: torch.Tensor, name: str) -> int:
    if t.dtype not in _DT:
        raise TypeError(f"{name}: dtype {t.dtype} is not float32 or bfloat16")
    return _DT[t.dtype]


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream: Optional[torch.cuda.Stream], device: torch.device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _require_cuda_contig(name: str, t: Optional[torch.Tensor], device) -> None:
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def make_shape(*, B: int, T: int, H: int, factor_dims: Sequence[int], d_sub: int, d_v: int,
               W: int, R: int, chunk_size: int, act_dtype: int, bank_dtype: int) -> _abi.SdmShape:
    if len(factor_dims) > _abi.MAX_FACTORS:
        # let the library refuse it with its own status
        dims = list(factor_dims)[:_abi.MAX_FACTORS]
        F = len(factor_dims)
    else:
        dims = list(factor_dims) + [1] * (_abi.MAX_FACTORS - len(factor_dims))
        F = len(factor_dims)
    sh = _abi.SdmShape()
    sh.B, sh.T, sh.H, sh.d_sub, sh.d_v = int(B), int(T), int(H), int(d_sub), int(d_v)
    sh.F = F
    for i, n in enumerate(dims):
        sh.factor_dims[i] = int(n)
    sh.W, sh.R, sh.chunk_size = int(W), int(R), int(chunk_size)
    sh.act_dtype, sh.bank_dtype = int(act_dtype), int(bank_dtype)
    return sh


def write_read_workspace_size(shape: _abi.SdmShape) -> int:
    n = ctypes.c_size_t(0)
    _abi.check(_abi.load().sdm_write_read_workspace_size(ctypes.byref(shape), ctypes.byref(n)),
               "sdm_write_read_workspace_size")
    return int(n.value)


def decode_workspace_size(shape: _abi.SdmShape) -> int:
    n = ctypes.c_size_t(0)
    _abi.check(_abi.load().sdm_decode_workspace_size(ctypes.byref(shape), ctypes.byref(n)),
               "sdm_decode_workspace_size")
    return int(n.value)


def _shape_of(q_w, k_val, bank_dtype_t, factor_dims, W, R, chunk_size, T=None) -> _abi.SdmShape:
    F = len(factor_dims)
    if q_w.dim() != 4 and T is None:
        raise ValueError("q_w must be [B, T, H, F*d_sub]")
    B, Tq, H, D = q_w.shape if T is None else (q_w.shape[0], 1, q_w.shape[1], q_w.shape[2])
    if F == 0 or D % F != 0:
        raise ValueError(f"query width {D} is not a multiple of F={F}")
    return make_shape(B=B, T=Tq, H=H, factor_dims=factor_dims, d_sub=D // F, d_v=k_val.shape[-1],
                      W=W, R=R, chunk_size=chunk_size, act_dtype=_dtype_code(q_w, "q_w"),
                      bank_dtype=_dtype_code(bank_dtype_t, "bank"))


def sdm_write_read(q_w: torch.Tensor, q_r: torch.Tensor, k_val: torch.Tensor, gates: torch.Tensor,
                   subkeys: torch.Tensor, bank: torch.Tensor, chunk_size: int, W: int, R: int, *,
                   factor_dims: Sequence[int], bank_init: Optional[torch.Tensor] = None,
                   y: Optional[torch.Tensor] = None, idx_w: Optional[torch.Tensor] = None,
                   wt_w: Optional[torch.Tensor] = None, idx_r: Optional[torch.Tensor] = None,
                   wt_r: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """The chunked write/read op; the bank advances in place.  Returns y [B, T, H, d_v].

    q_w, q_r [B,T,H,F*d_sub]; k_val [B,T,H,d_v]; gates [B,T,H,2] float32 (alpha, beta);
    subkeys [H, sum(factor_dims), d_sub]; bank [B,H,N,d_v] (float32 or bfloat16).
    bank_init: optional learned table [H,N,d_v] copied into every stream's bank first.
    idx_w/wt_w/idx_r/wt_r: optional output buffers for the selections.
    """
    dev = q_w.device
    for name, t in (("q_w", q_w), ("q_r", q_r), ("k_val", k_val), ("gates", gates),
                    ("subkeys", subkeys), ("bank", bank), ("bank_init", bank_init), ("y", y),
                    ("idx_w", idx_w), ("wt_w", wt_w), ("idx_r", idx_r), ("wt_r", wt_r),
                    ("workspace", workspace)):
        _require_cuda_contig(name, t, dev)
    if gates.dtype != torch.float32:
        raise TypeError("gates must be float32")
    shape = _shape_of(q_w, k_val, bank, factor_dims, W, R, chunk_size)
    if y is None:
        y = torch.empty_like(k_val)
    if workspace is None:
        workspace = torch.empty(write_read_workspace_size(shape), dtype=torch.uint8, device=dev)
    st = _abi.load().sdm_write_read(
        ctypes.byref(shape), _ptr(q_w), _ptr(q_r), _ptr(k_val), _ptr(gates), _ptr(subkeys),
        _ptr(bank_init), _ptr(bank), _ptr(y), _ptr(idx_w), _ptr(wt_w), _ptr(idx_r), _ptr(wt_r),
        _ptr(workspace), workspace.numel(), _stream_handle(stream, dev))
    _abi.check(st, "sdm_write_read")
    return y


def sdm_write_read_static(q_w: torch.Tensor, q_r: torch.Tensor, k_val: torch.Tensor, gates: torch.Tensor,
                          subkeys: torch.Tensor, bank: torch.Tensor, chunk_size: int, W: int, R: int, *,
                          factor_dims: Sequence[int], bank_init: Optional[torch.Tensor] = None,
                          y: torch.Tensor, idx_w: Optional[torch.Tensor] = None,
                          wt_w: Optional[torch.Tensor] = None, idx_r: Optional[torch.Tensor] = None,
                          wt_r: Optional[torch.Tensor] = None,
                          stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """sdm_write_read on the library's own fixed scratch array: allocates nothing, so the
    caller passes every output buffer, y included.  Shapes needing more scratch than
    _abi.STATIC_SCRATCH_BYTES are refused; calls must be ordered on one stream."""
    dev = q_w.device
    for name, t in (("q_w", q_w), ("q_r", q_r), ("k_val", k_val), ("gates", gates),
                    ("subkeys", subkeys), ("bank", bank), ("bank_init", bank_init), ("y", y),
                    ("idx_w", idx_w), ("wt_w", wt_w), ("idx_r", idx_r), ("wt_r", wt_r)):
        _require_cuda_contig(name, t, dev)
    if gates.dtype != torch.float32:
        raise TypeError("gates must be float32")
    shape = _shape_of(q_w, k_val, bank, factor_dims, W, R, chunk_size)
    st = _abi.load().sdm_write_read_static(
        ctypes.byref(shape), _ptr(q_w), _ptr(q_r), _ptr(k_val), _ptr(gates), _ptr(subkeys),
        _ptr(bank_init), _ptr(bank), _ptr(y), _ptr(idx_w), _ptr(wt_w), _ptr(idx_r), _ptr(wt_r),
        _stream_handle(stream, dev))
    _abi.check(st, "sdm_write_read_static")
    return y


_SNAP_DT = {"f32": _abi.SDM_F32, "bf16": _abi.SDM_BF16, torch.float32: _abi.SDM_F32,
            torch.bfloat16: _abi.SDM_BF16}


def _snap_code(snapshot_dtype) -> int:
    if snapshot_dtype in (_abi.SDM_F32, _abi.SDM_BF16) and isinstance(snapshot_dtype, int):
        return snapshot_dtype
    if snapshot_dtype not in _SNAP_DT:
        raise TypeError(f"snapshot_dtype {snapshot_dtype!r} is not float32 or bfloat16")
    return _SNAP_DT[snapshot_dtype]


def snapshot_bytes(shape: _abi.SdmShape, snapshot_dtype=torch.float32) -> int:
    n = ctypes.c_size_t(0)
    _abi.check(_abi.load().sdm_snapshot_bytes(ctypes.byref(shape), _snap_code(snapshot_dtype), ctypes.byref(n)),
               "sdm_snapshot_bytes")
    return int(n.value)


def backward_workspace_size(shape: _abi.SdmShape) -> int:
    n = ctypes.c_size_t(0)
    _abi.check(_abi.load().sdm_write_read_backward_workspace_size(ctypes.byref(shape), ctypes.byref(n)),
               "sdm_write_read_backward_workspace_size")
    return int(n.value)


def sdm_write_read_train(q_w: torch.Tensor, q_r: torch.Tensor, k_val: torch.Tensor, gates: torch.Tensor,
                         subkeys: torch.Tensor, bank: torch.Tensor, chunk_size: int, W: int, R: int, *,
                         factor_dims: Sequence[int], bank_init: Optional[torch.Tensor] = None,
                         snapshot_dtype=torch.float32, y: Optional[torch.Tensor] = None,
                         saved: Optional[dict] = None, workspace: Optional[torch.Tensor] = None,
                         stream: Optional[torch.cuda.Stream] = None) -> dict:
    """sdm_write_read that keeps what its backward needs: the selections and a snapshot of
    the rows each token overwrites (float32, exact, or bfloat16).  The bank advances in
    place.  Returns {"y", "idx_w", "wt_w", "idx_r", "wt_r", "snapshot", "snapshot_dtype"}
    (``saved`` may pass those buffers in to be reused)."""
    dev = q_w.device
    shape = _shape_of(q_w, k_val, bank, factor_dims, W, R, chunk_size)
    code = _snap_code(snapshot_dtype)
    B, T, H = shape.B, shape.T, shape.H
    if saved is None:
        saved = {
            "idx_w": torch.empty((B, T, H, W), dtype=torch.int32, device=dev),
            "wt_w": torch.empty((B, T, H, W), dtype=torch.float32, device=dev),
            "idx_r": torch.empty((B, T, H, R), dtype=torch.int32, device=dev),
            "wt_r": torch.empty((B, T, H, R), dtype=torch.float32, device=dev),
            "snapshot": torch.empty(snapshot_bytes(shape, code), dtype=torch.uint8, device=dev),
        }
    saved = dict(saved)
    saved["snapshot_dtype"] = code
    saved["y"] = torch.empty_like(k_val) if y is None else y
    for name, t in (("q_w", q_w), ("q_r", q_r), ("k_val", k_val), ("gates", gates), ("subkeys", subkeys),
                    ("bank", bank), ("bank_init", bank_init), ("y", saved["y"]), ("idx_w", saved["idx_w"]),
                    ("wt_w", saved["wt_w"]), ("idx_r", saved["idx_r"]), ("wt_r", saved["wt_r"]),
                    ("snapshot", saved["snapshot"]), ("workspace", workspace)):
        _require_cuda_contig(name, t, dev)
    if gates.dtype != torch.float32:
        raise TypeError("gates must be float32")
    if workspace is None:
        workspace = torch.empty(write_read_workspace_size(shape), dtype=torch.uint8, device=dev)
    snap = saved["snapshot"]
    st = _abi.load().sdm_write_read_train(
        ctypes.byref(shape), _ptr(q_w), _ptr(q_r), _ptr(k_val), _ptr(gates), _ptr(subkeys), _ptr(bank_init),
        _ptr(bank), _ptr(saved["y"]), _ptr(saved["idx_w"]), _ptr(saved["wt_w"]), _ptr(saved["idx_r"]),
        _ptr(saved["wt_r"]), _ptr(snap), snap.numel() * snap.element_size(), code, _ptr(workspace),
        workspace.numel(), _stream_handle(stream, dev))
    _abi.check(st, "sdm_write_read_train")
    return saved


def sdm_write_read_backward(q_w: torch.Tensor, q_r: torch.Tensor, k_val: torch.Tensor, gates: torch.Tensor,
                            subkeys: torch.Tensor, bank: torch.Tensor, dy: torch.Tensor, saved: dict,
                            W: int, R: int, *, factor_dims: Sequence[int], dbank: Optional[torch.Tensor] = None,
                            grads: Optional[dict] = None, workspace: Optional[torch.Tensor] = None,
                            stream: Optional[torch.cuda.Stream] = None) -> dict:
    """The backward of one sdm_write_read_train call (``saved`` is what it returned).

    bank: the bank the forward left; restored in place to the bank before it.  dy:
    dL/dy.  dbank: float32 dL/d(final bank) (zeros when None), overwritten in place with
    dL/d(initial bank).  Returns float32 gradients {"bank", "k_val", "gates", "q_w",
    "q_r", "subkeys"} (``grads`` may pass those buffers in).  A second backward through
    the same ``saved`` is refused by the library (SDM_DEVERR_SNAPSHOT, bank untouched).
    """
    dev = q_w.device
    shape = _shape_of(q_w, k_val, bank, factor_dims, W, R, 1)
    f32 = dict(dtype=torch.float32, device=dev)
    if dbank is None:
        dbank = torch.zeros(bank.shape, **f32)
    if grads is None:
        grads = {"k_val": torch.empty(k_val.shape, **f32), "gates": torch.empty(gates.shape, **f32),
                 "q_w": torch.empty(q_w.shape, **f32), "q_r": torch.empty(q_r.shape, **f32),
                 "subkeys": torch.empty(subkeys.shape, **f32)}
    grads = dict(grads)
    grads["bank"] = dbank
    snap = saved["snapshot"]
    for name, t in (("q_w", q_w), ("q_r", q_r), ("k_val", k_val), ("gates", gates), ("subkeys", subkeys),
                    ("bank", bank), ("dy", dy), ("dbank", dbank), ("snapshot", snap), ("workspace", workspace),
                    ("idx_w", saved["idx_w"]), ("wt_w", saved["wt_w"]), ("idx_r", saved["idx_r"]),
                    ("wt_r", saved["wt_r"])) + tuple((f"grads[{k}]", v) for k, v in grads.items()):
        _require_cuda_contig(name, t, dev)
    if dbank.dtype != torch.float32 or any(g.dtype != torch.float32 for g in grads.values()):
        raise TypeError("gradient buffers must be float32")
    if dy.dtype != k_val.dtype:
        raise TypeError("dy must have the activations' dtype")
    if workspace is None:
        workspace = torch.empty(backward_workspace_size(shape), dtype=torch.uint8, device=dev)
    st = _abi.load().sdm_write_read_backward(
        ctypes.byref(shape), _ptr(q_w), _ptr(q_r), _ptr(k_val), _ptr(gates), _ptr(subkeys),
        _ptr(saved["idx_w"]), _ptr(saved["wt_w"]), _ptr(saved["idx_r"]), _ptr(saved["wt_r"]), _ptr(snap),
        snap.numel() * snap.element_size(), int(saved["snapshot_dtype"]), _ptr(bank), _ptr(dy), _ptr(dbank),
        _ptr(grads["k_val"]), _ptr(grads["gates"]), _ptr(grads["q_w"]), _ptr(grads["q_r"]),
        _ptr(grads["subkeys"]), _ptr(workspace), workspace.numel(), _stream_handle(stream, dev))
    _abi.check(st, "sdm_write_read_backward")
    grads["workspace"] = workspace
    return grads


def layer_workspace_size(shape: _abi.SdmShape, dim: int) -> int:
    n = ctypes.c_size_t(0)
    _abi.check(_abi.load().sdm_layer_workspace_size(ctypes.byref(shape), int(dim), ctypes.byref(n)),
               "sdm_layer_workspace_size")
    return int(n.value)


def sdm_layer_forward(x: torch.Tensor, w_qw: torch.Tensor, w_qr: torch.Tensor, w_v: torch.Tensor,
                      w_g: torch.Tensor, w_o: torch.Tensor, subkeys: torch.Tensor, bank: torch.Tensor,
                      chunk_size: int, W: int, R: int, *, factor_dims: Sequence[int],
                      bank_init: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                      keep: Optional[dict] = None, workspace: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """The SDM layer forward around the op: x [B,T,dim] -> out [B,T,dim]; the bank advances in
    place (bank_init, if given, is copied into it first).  Weights are [out, in]: w_qw, w_qr
    [H*F*d_sub, dim], w_v [H*d_v, dim], w_g [2H, dim] (rows: alpha, beta of each head), w_o
    [dim, H*d_v].  ``keep``: optional dict of buffers receiving the intermediates "q_w",
    "q_r", "k_val", "gates" (float32) and "y"."""
    dev = x.device
    B, T, dim = x.shape
    H, d_sub = subkeys.shape[0], subkeys.shape[2]
    F = len(factor_dims)
    d_v = bank.shape[-1]
    sh = make_shape(B=B, T=T, H=H, factor_dims=factor_dims, d_sub=d_sub, d_v=d_v, W=W, R=R,
                    chunk_size=chunk_size, act_dtype=_dtype_code(x, "x"), bank_dtype=_dtype_code(bank, "bank"))
    keep = keep or {}
    if out is None:
        out = torch.empty_like(x)
    for name, t in (("x", x), ("w_qw", w_qw), ("w_qr", w_qr), ("w_v", w_v), ("w_g", w_g), ("w_o", w_o),
                    ("subkeys", subkeys), ("bank", bank), ("bank_init", bank_init), ("out", out),
                    ("workspace", workspace)) + tuple((f"keep[{k}]", v) for k, v in keep.items()):
        _require_cuda_contig(name, t, dev)
    for name, t, rows in (("w_qw", w_qw, H * F * d_sub), ("w_qr", w_qr, H * F * d_sub), ("w_v", w_v, H * d_v),
                          ("w_g", w_g, 2 * H), ("w_o", w_o, dim)):
        cols = H * d_v if name == "w_o" else dim
        if tuple(t.shape) != (rows, cols):
            raise ValueError(f"{name} must be [{rows}, {cols}], got {tuple(t.shape)}")
        if t.dtype != x.dtype:
            raise TypeError(f"{name} must have x's dtype")
    if workspace is None:
        workspace = torch.empty(layer_workspace_size(sh, dim), dtype=torch.uint8, device=dev)
    st = _abi.load().sdm_layer_forward(
        ctypes.byref(sh), int(dim), _ptr(x), _ptr(w_qw), _ptr(w_qr), _ptr(w_v), _ptr(w_g), _ptr(w_o),
        _ptr(subkeys), _ptr(bank_init), _ptr(bank), _ptr(out), _ptr(keep.get("q_w")), _ptr(keep.get("q_r")),
        _ptr(keep.get("k_val")), _ptr(keep.get("gates")), _ptr(keep.get("y")), _ptr(workspace),
        workspace.numel(), _stream_handle(stream, dev))
    _abi.check(st, "sdm_layer_forward")
    return out


def layer_backward_workspace_size(shape: _abi.SdmShape, dim: int) -> int:
    n = ctypes.c_size_t(0)
    _abi.check(_abi.load().sdm_layer_backward_workspace_size(ctypes.byref(shape), int(dim), ctypes.byref(n)),
               "sdm_layer_backward_workspace_size")
    return int(n.value)


def _layer_shape(x, subkeys, bank, factor_dims, W, R, chunk_size):
    B, T, _ = x.shape
    return make_shape(B=B, T=T, H=subkeys.shape[0], factor_dims=factor_dims, d_sub=subkeys.shape[2],
                      d_v=bank.shape[-1], W=W, R=R, chunk_size=chunk_size, act_dtype=_dtype_code(x, "x"),
                      bank_dtype=_dtype_code(bank, "bank"))


def _saved_struct(saved: dict) -> _abi.SdmLayerSaved:
    sv = _abi.SdmLayerSaved()
    for k in ("q_w", "q_r", "k_val", "gates", "y", "idx_w", "wt_w", "idx_r", "wt_r", "snapshot"):
        setattr(sv, k, _ptr(saved[k]))
    sv.snapshot_bytes = saved["snapshot"].numel() * saved["snapshot"].element_size()
    sv.snapshot_dtype = int(saved["snapshot_dtype"])
    return sv


def sdm_layer_forward_train(x: torch.Tensor, w_qw: torch.Tensor, w_qr: torch.Tensor, w_v: torch.Tensor,
                            w_g: torch.Tensor, w_o: torch.Tensor, subkeys: torch.Tensor, bank: torch.Tensor,
                            chunk_size: int, W: int, R: int, *, factor_dims: Sequence[int],
                            bank_init: Optional[torch.Tensor] = None, snapshot_dtype=torch.float32,
                            out: Optional[torch.Tensor] = None, saved: Optional[dict] = None,
                            workspace: Optional[torch.Tensor] = None,
                            stream: Optional[torch.cuda.Stream] = None):
    """sdm_layer_forward that keeps what sdm_layer_backward needs.  Returns (out, saved):
    saved holds the intermediates, the selections and the snapshot (pass it back in to
    reuse its buffers)."""
    dev = x.device
    sh = _layer_shape(x, subkeys, bank, factor_dims, W, R, chunk_size)
    B, T, dim = x.shape
    H, F, d_sub, d_v = sh.H, len(factor_dims), sh.d_sub, sh.d_v
    code = _snap_code(snapshot_dtype)
    if saved is None:
        f32, i32 = dict(dtype=torch.float32, device=dev), dict(dtype=torch.int32, device=dev)
        saved = {"q_w": torch.empty((B, T, H, F * d_sub), dtype=x.dtype, device=dev),
                 "q_r": torch.empty((B, T, H, F * d_sub), dtype=x.dtype, device=dev),
                 "k_val": torch.empty((B, T, H, d_v), dtype=x.dtype, device=dev),
                 "gates": torch.empty((B, T, H, 2), **f32), "y": torch.empty((B, T, H, d_v), dtype=x.dtype, device=dev),
                 "idx_w": torch.empty((B, T, H, W), **i32), "wt_w": torch.empty((B, T, H, W), **f32),
                 "idx_r": torch.empty((B, T, H, R), **i32), "wt_r": torch.empty((B, T, H, R), **f32),
                 "snapshot": torch.empty(snapshot_bytes(sh, code), dtype=torch.uint8, device=dev)}
    saved = dict(saved)
    saved["snapshot_dtype"] = code
    if out is None:
        out = torch.empty_like(x)
    for name, t in (("x", x), ("w_qw", w_qw), ("w_qr", w_qr), ("w_v", w_v), ("w_g", w_g), ("w_o", w_o),
                    ("subkeys", subkeys), ("bank", bank), ("bank_init", bank_init), ("out", out),
                    ("workspace", workspace)) + tuple((f"saved[{k}]", v) for k, v in saved.items()
                                                      if isinstance(v, torch.Tensor)):
        _require_cuda_contig(name, t, dev)
    if workspace is None:
        workspace = torch.empty(layer_workspace_size(sh, dim), dtype=torch.uint8, device=dev)
    sv = _saved_struct(saved)
    st = _abi.load().sdm_layer_forward_train(
        ctypes.byref(sh), int(dim), _ptr(x), _ptr(w_qw), _ptr(w_qr), _ptr(w_v), _ptr(w_g), _ptr(w_o), _ptr(subkeys),
        _ptr(bank_init), _ptr(bank), _ptr(out), ctypes.byref(sv), _ptr(workspace), workspace.numel(),
        _stream_handle(stream, dev))
    _abi.check(st, "sdm_layer_forward_train")
    return out, saved


def sdm_layer_backward(x: torch.Tensor, w_qw: torch.Tensor, w_qr: torch.Tensor, w_v: torch.Tensor,
                       w_g: torch.Tensor, w_o: torch.Tensor, subkeys: torch.Tensor, bank: torch.Tensor,
                       dout: torch.Tensor, saved: dict, chunk_size: int, W: int, R: int, *,
                       factor_dims: Sequence[int], dbank: Optional[torch.Tensor] = None, learned_table: bool = True,
                       grads: Optional[dict] = None, workspace: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None) -> dict:
    """The backward of one sdm_layer_forward_train call for the loss gradient dout [B,T,dim].
    Returns {"x" (activation dtype), "w_qw", "w_qr", "w_v", "w_g", "w_o", "subkeys", "bank" (the
    float32 gradient table: dbank in, zeros when None), "bank_init" (its sum over the batch,
    when learned_table)}; the bank is restored in place."""
    dev = x.device
    sh = _layer_shape(x, subkeys, bank, factor_dims, W, R, chunk_size)
    dim = x.shape[-1]
    f32 = dict(dtype=torch.float32, device=dev)
    if dbank is None:
        dbank = torch.zeros(bank.shape, **f32)
    if grads is None:
        grads = {"x": torch.empty_like(x), "w_qw": torch.empty(w_qw.shape, **f32),
                 "w_qr": torch.empty(w_qr.shape, **f32), "w_v": torch.empty(w_v.shape, **f32),
                 "w_g": torch.empty(w_g.shape, **f32), "w_o": torch.empty(w_o.shape, **f32),
                 "subkeys": torch.empty(subkeys.shape, **f32)}
        if learned_table:
            grads["bank_init"] = torch.empty(bank.shape[1:], **f32)
    grads = dict(grads)
    grads["bank"] = dbank
    for name, t in (("x", x), ("w_o", w_o), ("subkeys", subkeys), ("bank", bank), ("dout", dout),
                    ("workspace", workspace)) + tuple((f"grads[{k}]", v) for k, v in grads.items()):
        _require_cuda_contig(name, t, dev)
    if workspace is None:
        workspace = torch.empty(layer_backward_workspace_size(sh, dim), dtype=torch.uint8, device=dev)
    gs = _abi.SdmLayerGrads()
    gs.dx, gs.dw_qw, gs.dw_qr = _ptr(grads["x"]), _ptr(grads["w_qw"]), _ptr(grads["w_qr"])
    gs.dw_v, gs.dw_g, gs.dw_o = _ptr(grads["w_v"]), _ptr(grads["w_g"]), _ptr(grads["w_o"])
    gs.d_subkeys, gs.dbank, gs.d_bank_init = _ptr(grads["subkeys"]), _ptr(dbank), _ptr(grads.get("bank_init"))
    sv = _saved_struct(saved)
    st = _abi.load().sdm_layer_backward(
        ctypes.byref(sh), int(dim), _ptr(x), _ptr(w_qw), _ptr(w_qr), _ptr(w_v), _ptr(w_g), _ptr(w_o),
        _ptr(subkeys), _ptr(bank), _ptr(dout), ctypes.byref(sv), ctypes.byref(gs), _ptr(workspace),
        workspace.numel(), _stream_handle(stream, dev))
    _abi.check(st, "sdm_layer_backward")
    grads["workspace"] = workspace
    return grads


def _owns_storage(t: torch.Tensor) -> bool:
    """True when writing into t cannot reach another tensor's data (the donate guards).

    A view (including a broadcast with a zero stride) may share its storage with a table
    that is not the stream's own, and a tensor autograd records must not change under
    it (lumen PR #29, Donating is a permission).
    """
    if t._base is not None:
        return False
    if any(s == 0 for s, n in zip(t.stride(), t.shape) if n > 1):
        return False
    if t.requires_grad:
        return False
    return t.is_contiguous()


def sdm_decode_step(q_w: torch.Tensor, q_r: torch.Tensor, k_val: torch.Tensor, gates: torch.Tensor,
                    subkeys: torch.Tensor, bank: torch.Tensor, W: int, R: int, *,
                    factor_dims: Sequence[int], donate: bool = False,
                    bank_out: Optional[torch.Tensor] = None, y: Optional[torch.Tensor] = None,
                    idx_w: Optional[torch.Tensor] = None, wt_w: Optional[torch.Tensor] = None,
                    idx_r: Optional[torch.Tensor] = None, wt_r: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None):
    """One decode step for every stream.  Returns (y [B,H,d_v], successor bank).

    q_w, q_r [B,H,F*d_sub]; k_val [B,H,d_v]; gates [B,H,2]; bank [B,H,N,d_v], or a
    learned table [H,N,d_v] / its broadcast view that every stream starts from.
    donate=True lets the step write the successor into `bank` itself; it is honoured only
    when `bank` owns its storage (not a view, not a broadcast, not recorded by autograd),
    otherwise the step copies, as a permission and not a demand.
    """
    dev = q_w.device
    B, H = q_w.shape[0], q_w.shape[1]
    shared = False
    bank_in = bank
    if bank.dim() == 3:
        shared = True
    elif bank.dim() == 4 and bank.shape[0] == B and bank.stride(0) == 0 and B > 1:
        bank_in = bank[0]               # a broadcast of one [H,N,d_v] table
        shared = True
    if shared:
        if not bank_in.is_contiguous():
            bank_in = bank_in.contiguous()
        donate = False
    elif donate and not _owns_storage(bank):
        donate = False
    for name, t in (("q_w", q_w), ("q_r", q_r), ("k_val", k_val), ("gates", gates),
                    ("subkeys", subkeys), ("bank", bank_in), ("bank_out", bank_out), ("y", y),
                    ("idx_w", idx_w), ("wt_w", wt_w), ("idx_r", idx_r), ("wt_r", wt_r),
                    ("workspace", workspace)):
        _require_cuda_contig(name, t, dev)
    shape = _shape_of(q_w, k_val, bank_in, factor_dims, W, R, 1, T=1)
    N = math.prod(int(n) for n in factor_dims)
    if donate:
        bank_out = bank
    elif bank_out is None:
        bank_out = torch.empty((B, H, N, k_val.shape[-1]), dtype=bank_in.dtype, device=dev)
    if y is None:
        y = torch.empty_like(k_val)
    if workspace is None:
        workspace = torch.empty(decode_workspace_size(shape), dtype=torch.uint8, device=dev)
    st = _abi.load().sdm_decode_step(
        ctypes.byref(shape), _ptr(q_w), _ptr(q_r), _ptr(k_val), _ptr(gates), _ptr(subkeys),
        _ptr(bank_in), 1 if shared else 0, _ptr(bank_out), 1 if donate else 0, _ptr(y),
        _ptr(idx_w), _ptr(wt_w), _ptr(idx_r), _ptr(wt_r), _ptr(workspace), workspace.numel(),
        _stream_handle(stream, dev))
    _abi.check(st, "sdm_decode_step")
    return y, bank_out


def last_device_error(workspace: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> int:
    """Kernel-side error code of the last call that used `workspace` (0 = none); syncs."""
    code = ctypes.c_int32(0)
    st = _abi.load().sdm_last_device_error(_ptr(workspace), workspace.numel(), ctypes.byref(code),
                                           _stream_handle(stream, workspace.device))
    if st not in (_abi.SDM_OK, _abi.SDM_ERR_DEVICE):
        _abi.check(st, "sdm_last_device_error")
    return int(code.value)


def launch_count() -> int:
    return int(_abi.load().sdm_launch_count())


def test_stall_decode_copy(on: bool) -> None:
    """Test hook of the device failure path (see sdm_test_stall_decode_copy in sdm.h)."""
    _abi.check(_abi.load().sdm_test_stall_decode_copy(1 if on else 0), "sdm_test_stall_decode_copy")


def test_force_write_read_layout(slice_bytes: int = 0, stage_tokens: int = 0) -> None:
    """Test hook: force the write/read kernel's row slice per CTA (32, 128 or 256 bytes)
    and cap its stage length; 0 restores the automatic choice (sdm.h)."""
    _abi.check(_abi.load().sdm_test_force_write_read_layout(int(slice_bytes), int(stage_tokens)),
               "sdm_test_force_write_read_layout")


def test_force_simt_scorer(on: bool) -> None:
    """Test hook: score on the CUDA-core scorer instead of the tensor cores (sdm.h)."""
    _abi.check(_abi.load().sdm_test_force_simt_scorer(1 if on else 0), "sdm_test_force_simt_scorer")


def test_factor_scores(q_w: torch.Tensor, q_r: torch.Tensor, subkeys: torch.Tensor, *,
                       factor_dims: Sequence[int], workspace: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Test hook: the factor scores of step 1, [2, B*T*H, sum(factor_dims)] float32 (q_w rows,
    then q_r rows), from the scorer sdm_write_read would use (sdm.h)."""
    dev = q_w.device
    for name, t in (("q_w", q_w), ("q_r", q_r), ("subkeys", subkeys)):
        _require_cuda_contig(name, t, dev)
    B, T, H, D = q_w.shape
    F = len(factor_dims)
    if F == 0 or D % F != 0:
        raise ValueError(f"query width {D} is not a multiple of F={F}")
    act = _dtype_code(q_w, "q_w")
    shape = make_shape(B=B, T=T, H=H, factor_dims=factor_dims, d_sub=D // F, d_v=8, W=1, R=1, chunk_size=64,
                       act_dtype=act, bank_dtype=act)
    scores = torch.empty((2, B * T * H, sum(factor_dims)), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(write_read_workspace_size(shape), dtype=torch.uint8, device=dev)
    st = _abi.load().sdm_test_factor_scores(ctypes.byref(shape), _ptr(q_w), _ptr(q_r), _ptr(subkeys), _ptr(scores),
                                            _ptr(workspace), workspace.numel(), _stream_handle(stream, dev))
    _abi.check(st, "sdm_test_factor_scores")
    return scores


def profile_begin() -> None:
    _abi.check(_abi.load().sdm_profile_begin(), "sdm_profile_begin")


def profile_end() -> dict:
    """{kernel name: (launches, total ms)} of the launches since profile_begin."""
    out = _abi.KernelTimes()
    _abi.check(_abi.load().sdm_profile_end(ctypes.byref(out)), "sdm_profile_end")
    return {name: (int(out.launches[i]), float(out.ms[i])) for i, name in enumerate(_abi.KERNEL_KINDS)}
