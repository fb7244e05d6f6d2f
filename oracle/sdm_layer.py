"""CPU oracle of the SDM layer forward around the write/read op.

TEST INFRASTRUCTURE ONLY, like sdm_oracle.py: nothing in the product path imports it.

What the pages fix (page title > section): sparse-delta-memory README > usage example: a
layer built from dim, num_heads, slots_per_head, num_writes, num_reads and chunk_size
maps x [batch, tokens, dim] to y of the same shape, and the bank advances in place.
Readings where the pages are silent (the plainest layer that the op's inputs imply):
  * four input projections of x without bias: the write and read queries
    [H*F*d_sub], the values [H*d_v], and two gate logits per head whose sigmoids are
    (alpha, beta); weights stored [out, in];
  * an output projection of the heads' reads [H*d_v] back to dim, without bias;
  * projections accumulate exactly (float64 here) and round once to the activation
    type; the gates round once to float32;
  * the backward (README > usage example: backward() through the layer) is the chain rule
    through these maps around the op's backward (sdm_backward), every rounding passing
    the gradient unchanged; the gradients that cross between the dense products and the op
    are held in the activation type, as the op's activations are (dy = dout w_o, and the
    query, value and gate-logit gradients before they meet the weights), so they round
    once to it there; the learned table's gradient is the sum over the batch of the
    streams' bank gradients.
"""

from __future__ import annotations

from typing import Iterable, Optional

import numpy as np

from . import sdm_backward
from .sdm_oracle import _f64, round_to, sdm_write_read

__all__ = ["project", "gates_of", "layer_forward", "layer_backward"]


def project(x: np.ndarray, w: np.ndarray, act_dtype: str) -> np.ndarray:
    """x [rows, in] times w [out, in] transposed, rounded once to the activation type."""
    return round_to(_f64(x) @ _f64(w).T, act_dtype)


def gates_of(x: np.ndarray, w_g: np.ndarray) -> np.ndarray:
    """sigmoid(x w_g^T) [rows, 2H] in float64, rounded once to float32."""
    z = _f64(x) @ _f64(w_g).T
    return round_to(1.0 / (1.0 + np.exp(-z)), "f32")


def layer_forward(x, w_qw, w_qr, w_v, w_g, w_o, subkeys, bank_init, *, factor_dims, W: int, R: int,
                  chunk_size: int = 64, act_dtype: str = "f32", bank_dtype: str = "f32",
                  streams: Optional[Iterable] = None, given: Optional[dict] = None) -> dict:
    """The layer forward of x [B, T, dim]: projections, the op (sdm_oracle.sdm_write_read,
    every stream starting from the learned table bank_init [H, N, d_v]) and the output
    projection.

    ``given`` may hold the op's inputs "q_w", "q_r", "k_val", "gates" ([B,T,H,...]) to use
    instead of the oracle's own projections (to check the op and the output projection
    on another path's projections); the oracle's own projections are returned either way.
    Returns float64 arrays: q_w, q_r, k_val, gates, y [B,T,H,d_v], out [B,T,dim] (out and
    y only for the listed streams' heads when ``streams`` is given: other entries zero),
    and the per-stream op results under "op".
    """
    x = _f64(x)
    B, T, dim = x.shape
    H, _, d_sub = np.shape(subkeys)
    F = len(factor_dims)
    d_v = np.shape(bank_init)[-1]
    X = x.reshape(B * T, dim)
    own = {
        "q_w": project(X, w_qw, act_dtype).reshape(B, T, H, F * d_sub),
        "q_r": project(X, w_qr, act_dtype).reshape(B, T, H, F * d_sub),
        "k_val": project(X, w_v, act_dtype).reshape(B, T, H, d_v),
        "gates": gates_of(X, w_g).reshape(B, T, H, 2),
    }
    src = dict(own)
    if given:
        src.update({k: _f64(v) for k, v in given.items()})
    op = sdm_write_read(src["q_w"], src["q_r"], src["k_val"], src["gates"], subkeys, bank_init,
                        factor_dims=factor_dims, W=W, R=R, chunk_size=chunk_size, act_dtype=act_dtype,
                        bank_dtype=bank_dtype, streams=streams)
    y = np.zeros((B, T, H, d_v))
    for (b, h), res in op.items():
        y[b, :, h] = res["y"]
    out = project(y.reshape(B * T, H * d_v), w_o, act_dtype).reshape(B, T, dim)
    return dict(own, y=y, out=out, op=op)


def layer_backward(x, w_qw, w_qr, w_v, w_g, w_o, subkeys, bank_init, dout, *, factor_dims, W: int, R: int,
                   act_dtype: str = "f32", bank_dtype: str = "f32", snapshot_dtype: Optional[str] = None,
                   dbank=None, given: Optional[dict] = None, pick=None, exact: bool = False) -> dict:
    """Gradients of a loss with respect to the layer's inputs, for dout = dL/d(out) [B,T,dim]
    (and dbank = dL/d(final bank) [B,H,N,d_v], zeros when None).

    ``given`` as in layer_forward (the op's inputs and its read y: the backward then runs the
    op's backward on them and the output projection's backward on y); ``pick`` goes to
    sdm_backward.sdm_write_read_backward; ``exact``: float64 everywhere with float64 scores
    (for finite differences; act_dtype and bank_dtype should then be "f64").
    Returns float64 arrays keyed x, w_qw, w_qr, w_v, w_g, w_o, subkeys, bank ([B,H,N,d_v]),
    bank_init ([H,N,d_v]), and the op's gradients under "op".
    """
    x = _f64(x)
    B, T, dim = x.shape
    H, _, d_sub = np.shape(subkeys)
    F = len(factor_dims)
    d_v = np.shape(bank_init)[-1]
    BT, dq, dv = B * T, H * F * d_sub, H * d_v
    X = x.reshape(BT, dim)
    w_qw, w_qr, w_v, w_g, w_o = (_f64(w) for w in (w_qw, w_qr, w_v, w_g, w_o))
    if exact:
        ins = {"q_w": (X @ w_qw.T).reshape(B, T, H, F * d_sub), "q_r": (X @ w_qr.T).reshape(B, T, H, F * d_sub),
               "k_val": (X @ w_v.T).reshape(B, T, H, d_v),
               "gates": (1.0 / (1.0 + np.exp(-(X @ w_g.T)))).reshape(B, T, H, 2)}
    else:
        ins = {"q_w": project(X, w_qw, act_dtype).reshape(B, T, H, F * d_sub),
               "q_r": project(X, w_qr, act_dtype).reshape(B, T, H, F * d_sub),
               "k_val": project(X, w_v, act_dtype).reshape(B, T, H, d_v),
               "gates": gates_of(X, w_g).reshape(B, T, H, 2)}
    if given:
        ins.update({k: _f64(v) for k, v in given.items() if k != "y"})
    if given and "y" in given:
        Y = _f64(given["y"]).reshape(BT, dv)
    else:
        bank = np.broadcast_to(_f64(bank_init)[None], (B, H) + np.shape(bank_init)[1:])
        fwd = {}
        for b in range(B):
            for h in range(H):
                M = np.array(bank[b, h])
                rec = sdm_backward.stream_forward(M, ins["q_w"][b, :, h], ins["q_r"][b, :, h], ins["k_val"][b, :, h],
                                                  ins["gates"][b, :, h], _f64(subkeys)[h], factor_dims=factor_dims,
                                                  d_sub=d_sub, W=W, R=R, act_dtype=act_dtype, bank_dtype=bank_dtype,
                                                  exact=exact, pick=None if pick is None else pick(b, h))
                fwd[(b, h)] = rec["y"]
        Y = np.zeros((B, T, H, d_v))
        for (b, h), yy in fwd.items():
            Y[b, :, h] = yy
        Y = Y.reshape(BT, dv)
    D = _f64(dout).reshape(BT, dim)
    dY = D @ w_o                                        # [BT, H d_v]: the op's dy
    if not exact:
        dY = round_to(dY, act_dtype)                    # the op takes dy in the activation type
    dw_o = D.T @ Y                                      # [dim, H d_v]
    bank = np.broadcast_to(_f64(bank_init)[None], (B, H) + np.shape(bank_init)[1:])
    db = np.zeros(bank.shape) if dbank is None else _f64(dbank)
    g = sdm_backward.sdm_write_read_backward(ins["q_w"], ins["q_r"], ins["k_val"], ins["gates"], subkeys, bank,
                                             dY.reshape(B, T, H, d_v), db, factor_dims=factor_dims, W=W, R=R,
                                             act_dtype=act_dtype, bank_dtype=bank_dtype,
                                             snapshot_dtype=snapshot_dtype, pick=pick, exact=exact)
    z = X @ w_g.T
    s = 1.0 / (1.0 + np.exp(-z))
    dz = g["gates"].reshape(BT, 2 * H) * s * (1.0 - s)
    d_qw, d_qr, d_kv = g["q_w"].reshape(BT, dq), g["q_r"].reshape(BT, dq), g["k_val"].reshape(BT, dv)
    if not exact:                                       # the projections' gradients meet the
        d_qw, d_qr, d_kv, dz = (round_to(a, act_dtype)  # weights in the activation type
                                for a in (d_qw, d_qr, d_kv, dz))
    dx = d_qw @ w_qw + d_qr @ w_qr + d_kv @ w_v + dz @ w_g
    return {"x": dx.reshape(B, T, dim), "w_qw": d_qw.T @ X, "w_qr": d_qr.T @ X, "w_v": d_kv.T @ X,
            "w_g": dz.T @ X, "w_o": dw_o, "subkeys": g["subkeys"], "bank": g["bank"],
            "bank_init": g["bank"].sum(axis=0), "op": g}
