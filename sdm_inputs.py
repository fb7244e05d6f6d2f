"""Seeded synthetic inputs for the Sparse Delta Memory (SDM) write/read op.

This module only draws random numbers and casts them; it holds none of the
method's arithmetic (no scoring, no top-k, no update).  Both the CPU oracle
(``oracle/``) and the CUDA path (``gated_delta_rule_factor_gb300``) take their
inputs from here, so that the two see identical bits.

Workloads follow the shapes the SDM pages describe: the README layer call
(2 heads of 1024, 65536 slots per head from two factors of 256, 64 writes and
reads per token, chunk 64), the lumen decode step (128 streams, d_model 512,
2 heads, 32x32 slots), the 32K-token training shape and a three-factor
configuration.  Distributions: queries and values N(0, 1); sub-keys
N(0, 1/d_sub); gates sigmoid(N(0, 1)) for the forget gate alpha and the input
gate beta independently; the bank N(0, 0.02^2) (standard deviation 0.02).

``grid=True`` quantises queries and sub-keys to a coarse binary grid (see
``_grid``) on which every factor score, and every float32 sum of factor scores,
is exactly representable: any summation order then gives the same bits, so the
product-key selection is unique and the tie rule is exercised by real ties.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = ["SdmConfig", "CONFIGS", "make_inputs", "make_decode_inputs", "grid_exponents"]


@dataclasses.dataclass(frozen=True)
class SdmConfig:
    name: str
    B: int
    T: int
    H: int
    factor_dims: tuple
    d_sub: int
    d_v: int
    W: int
    R: int
    chunk_size: int
    act_dtype: str      # "f32" or "bf16"
    bank_dtype: str     # "f32" or "bf16"
    seed: int
    low_rank_queries: bool = False
    learned_bank: bool = True   # bank given as a learned [H, N, d_v] table copied per stream

    @property
    def F(self) -> int:
        return len(self.factor_dims)

    @property
    def N(self) -> int:
        return int(math.prod(self.factor_dims))

    def replace(self, **kw) -> "SdmConfig":
        return dataclasses.replace(self, **kw)


# The five workloads, in the order the task description lists them; seed = 1000 + position.
CONFIGS = {
    "tiny": SdmConfig("tiny", B=1, T=256, H=1, factor_dims=(32, 32), d_sub=32, d_v=64,
                      W=8, R=8, chunk_size=64, act_dtype="f32", bank_dtype="f32", seed=1001),
    "layer": SdmConfig("layer", B=2, T=4096, H=2, factor_dims=(256, 256), d_sub=512, d_v=1024,
                       W=64, R=64, chunk_size=64, act_dtype="bf16", bank_dtype="f32", seed=1002),
    "decode": SdmConfig("decode", B=128, T=1, H=2, factor_dims=(32, 32), d_sub=128, d_v=256,
                        W=64, R=64, chunk_size=1, act_dtype="f32", bank_dtype="f32", seed=1003),
    "train_fwd": SdmConfig("train_fwd", B=8, T=4096, H=2, factor_dims=(256, 256), d_sub=512,
                           d_v=1024, W=64, R=64, chunk_size=64, act_dtype="bf16",
                           bank_dtype="bf16", seed=1004),
    "three_factor": SdmConfig("three_factor", B=1, T=8192, H=4, factor_dims=(64, 64, 64),
                              d_sub=64, d_v=256, W=64, R=64, chunk_size=128, act_dtype="f32",
                              bank_dtype="f32", seed=1005, low_rank_queries=True),
}

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def grid_exponents(d_sub: int):
    """Binary exponents (e_q, e_k) of the query and sub-key grids.

    Queries are multiples of 2**-e_q and sub-keys multiples of 2**-e_k, each with an
    integer numerator of magnitude <= 127 (exact in bfloat16 and float32).  A factor
    score is then an integer times 2**-(e_q+e_k) of magnitude <= d_sub*127*127, which
    float32 holds exactly while F*d_sub*127*127 < 2**24.
    """
    e_q = 4                                   # N(0,1) at 1/16 resolution, range +-7.9
    sigma_k = 1.0 / math.sqrt(d_sub)
    e_k = int(math.floor(math.log2(127.0 / (8.0 * sigma_k))))
    return e_q, e_k


def _grid(x: torch.Tensor, e: int) -> torch.Tensor:
    scale = float(2 ** e)
    return torch.clamp(torch.round(x * scale), -127, 127) / scale


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def make_inputs(cfg: SdmConfig, *, seed: Optional[int] = None, grid: bool = False,
                T: Optional[int] = None, B: Optional[int] = None) -> dict:
    """Draw one batch of inputs for ``cfg`` on the CPU.

    Returns a dict of CPU tensors:
      q_w, q_r   [B, T, H, F*d_sub]  act dtype
      k_val      [B, T, H, d_v]      act dtype
      gates      [B, T, H, 2]        float32, (alpha, beta) in (0, 1)
      subkeys    [H, sum(n_f), d_sub] act dtype; factor f at row offset sum_{g<f} n_g
      bank_init  [H, N, d_v]         bank dtype (the learned initial table)
    ``T``/``B`` override the config's sequence length / batch (prefix-compatible:
    the first T tokens of a longer draw are not reused, each call draws afresh).
    """
    seed = cfg.seed if seed is None else seed
    B = cfg.B if B is None else B
    T = cfg.T if T is None else T
    g = _gen(seed)
    F, H, d_sub, d_v = cfg.F, cfg.H, cfg.d_sub, cfg.d_v
    D = F * d_sub
    n_tot = sum(cfg.factor_dims)
    act = _TORCH_DTYPE[cfg.act_dtype]
    bank_t = _TORCH_DTYPE[cfg.bank_dtype]

    subkeys = torch.randn(H, n_tot, d_sub, generator=g) / math.sqrt(d_sub)
    if cfg.low_rank_queries:
        # q_t = 2 z_t U + eps_t, U fixed per head (entries N(0,1)), z_t ~ N(0, I_2),
        # eps ~ N(0, 0.25 I): tokens prefer the same sub-keys, so slots collide often.
        U = torch.randn(H, 2, D, generator=g)
        z_w = torch.randn(B, T, H, 2, generator=g)
        z_r = torch.randn(B, T, H, 2, generator=g)
        q_w = 2.0 * torch.einsum("bthz,hzd->bthd", z_w, U) + 0.5 * torch.randn(B, T, H, D, generator=g)
        q_r = 2.0 * torch.einsum("bthz,hzd->bthd", z_r, U) + 0.5 * torch.randn(B, T, H, D, generator=g)
    else:
        q_w = torch.randn(B, T, H, D, generator=g)
        q_r = torch.randn(B, T, H, D, generator=g)
    k_val = torch.randn(B, T, H, d_v, generator=g)
    gates = torch.sigmoid(torch.randn(B, T, H, 2, generator=g))
    bank_init = 0.02 * torch.randn(H, cfg.N, d_v, generator=g)

    if grid:
        e_q, e_k = grid_exponents(d_sub)
        q_w = _grid(q_w, e_q)
        q_r = _grid(q_r, e_q)
        subkeys = _grid(subkeys, e_k)

    return {
        "q_w": q_w.to(act).contiguous(),
        "q_r": q_r.to(act).contiguous(),
        "k_val": k_val.to(act).contiguous(),
        "gates": gates.to(torch.float32).contiguous(),
        "subkeys": subkeys.to(act).contiguous(),
        "bank_init": bank_init.to(bank_t).contiguous(),
    }


def make_decode_inputs(cfg: SdmConfig, steps: int, *, seed: Optional[int] = None,
                       grid: bool = False) -> dict:
    """Inputs for ``steps`` consecutive single-token decode steps of ``cfg``.

    Same tensors as ``make_inputs`` with T = steps; step s uses token s.  The bank is
    returned per stream ([B, H, N, d_v]), already broadcast from the learned table,
    since a decode state owns its table.
    """
    d = make_inputs(cfg, seed=seed, grid=grid, T=steps)
    bank = d.pop("bank_init")
    d["bank"] = bank.unsqueeze(0).expand(cfg.B, *bank.shape).contiguous()
    return d


def make_grad_inputs(cfg: SdmConfig, *, seed: Optional[int] = None, T: Optional[int] = None,
                     B: Optional[int] = None, dbank: bool = True) -> dict:
    """Loss gradients for the backward of one ``make_inputs`` batch (CPU tensors).

      dy     [B, T, H, d_v]  act dtype, N(0, 1): dL/dy
      dbank  [B, H, N, d_v]  float32, N(0, 0.01^2): dL/d(final bank), or zeros when
             ``dbank`` is False (y the only output that matters)
    Drawn from a generator of its own (seed + 500), so the forward's inputs are the same
    whether or not gradients are drawn.
    """
    seed = (cfg.seed if seed is None else seed) + 500
    B = cfg.B if B is None else B
    T = cfg.T if T is None else T
    g = _gen(seed)
    dy = torch.randn(B, T, cfg.H, cfg.d_v, generator=g).to(_TORCH_DTYPE[cfg.act_dtype]).contiguous()
    if dbank:
        db = 0.01 * torch.randn(B, cfg.H, cfg.N, cfg.d_v, generator=g)
    else:
        db = torch.zeros(B, cfg.H, cfg.N, cfg.d_v)
    return {"dy": dy, "dbank": db.to(torch.float32).contiguous()}


def make_layer_inputs(cfg: SdmConfig, dim: int, *, seed: Optional[int] = None, T: Optional[int] = None,
                      B: Optional[int] = None) -> dict:
    """Inputs of the layer around the op, for ``cfg``'s op shape and model width ``dim``
    (CPU tensors, activation dtype unless noted).

      x      [B, T, dim]            N(0, 1)
      w_qw, w_qr [H*F*d_sub, dim]   N(0, 1/dim): projected queries ~ N(0, 1)
      w_v    [H*d_v, dim]           N(0, 1/dim)
      w_g    [2H, dim]              N(0, 1/dim): gate logits ~ N(0, 1), as the op's gates
      w_o    [dim, H*d_v]           N(0, 1/(H*d_v))
      subkeys, bank_init            as make_inputs
    Drawn from a generator of its own (seed + 900).
    """
    base = make_inputs(cfg, seed=seed, T=1, B=1)
    seed = (cfg.seed if seed is None else seed) + 900
    B = cfg.B if B is None else B
    T = cfg.T if T is None else T
    g = _gen(seed)
    act = _TORCH_DTYPE[cfg.act_dtype]
    H, dq, dv = cfg.H, cfg.H * cfg.F * cfg.d_sub, cfg.H * cfg.d_v
    s = 1.0 / math.sqrt(dim)
    out = {
        "x": torch.randn(B, T, dim, generator=g),
        "w_qw": s * torch.randn(dq, dim, generator=g),
        "w_qr": s * torch.randn(dq, dim, generator=g),
        "w_v": s * torch.randn(dv, dim, generator=g),
        "w_g": s * torch.randn(2 * H, dim, generator=g),
        "w_o": torch.randn(dim, dv, generator=g) / math.sqrt(dv),
    }
    out = {k: v.to(act).contiguous() for k, v in out.items()}
    out["subkeys"] = base["subkeys"]
    out["bank_init"] = base["bank_init"]
    return out
