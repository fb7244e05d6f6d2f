"""Shared helpers of the GPU tests: run the CUDA op and the oracle on the same inputs
and compare them under the parity rules.

Parity rules (floating point from the task's stated tolerances):
  * selected slot ids are compared exactly wherever the oracle's k-th and (k+1)-th
    slot scores differ by more than 1e-6 relative; at a closer call the GPU's set must
    still be a valid top-k of the oracle's scores within that margin;
  * y and the final bank match within rtol = 1e-5 (float32) or 2e-2 (bfloat16),
    measured as |gpu - oracle| <= rtol * (|oracle| + rms(oracle)) elementwise (the rms
    term keeps entries near zero from demanding an absolute precision the other entries
    never had);
  * where the GPU's pick is a valid alternative at a near tie, the oracle continues on
    the GPU's slots (their weights from the oracle's own scores), so y and the final
    bank stay compared through the last token of every stream.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
import sdm_inputs

RTOL = {"f32": 1e-5, "bf16": 2e-2}
MARGIN = 1e-6
_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16}


def to_device(d: dict, device="cuda") -> dict:
    return {k: v.to(device) for k, v in d.items()}


def gpu_write_read(cfg, d: dict, *, chunk_size=None, bank_init=True, device="cuda"):
    """Run sdm_write_read on ``d`` (CPU tensors); returns CPU results."""
    import gated_delta_rule_factor_gb300 as sdm
    g = to_device(d, device)
    B, T, H = g["q_w"].shape[0], g["q_w"].shape[1], g["q_w"].shape[2]
    bank = torch.empty((B, H, cfg.N, cfg.d_v), dtype=_TORCH[cfg.bank_dtype], device=device)
    idx_w = torch.empty((B, T, H, cfg.W), dtype=torch.int32, device=device)
    wt_w = torch.empty((B, T, H, cfg.W), dtype=torch.float32, device=device)
    idx_r = torch.empty((B, T, H, cfg.R), dtype=torch.int32, device=device)
    wt_r = torch.empty((B, T, H, cfg.R), dtype=torch.float32, device=device)
    if not bank_init:
        bank.copy_(g["bank_init"].unsqueeze(0).expand_as(bank))
    sh = sdm.make_shape(B=B, T=T, H=H, factor_dims=cfg.factor_dims, d_sub=cfg.d_sub, d_v=cfg.d_v,
                        W=cfg.W, R=cfg.R, chunk_size=chunk_size or cfg.chunk_size,
                        act_dtype=0 if cfg.act_dtype == "f32" else 1,
                        bank_dtype=0 if cfg.bank_dtype == "f32" else 1)
    ws = torch.empty(sdm.write_read_workspace_size(sh), dtype=torch.uint8, device=device)
    y = sdm.sdm_write_read(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], bank,
                           chunk_size or cfg.chunk_size, cfg.W, cfg.R, factor_dims=cfg.factor_dims,
                           bank_init=g["bank_init"] if bank_init else None, idx_w=idx_w, wt_w=wt_w,
                           idx_r=idx_r, wt_r=wt_r, workspace=ws)
    torch.cuda.synchronize()
    assert sdm.last_device_error(ws) == 0
    return {"y": y.cpu(), "bank": bank.cpu(), "idx_w": idx_w.cpu(), "wt_w": wt_w.cpu(),
            "idx_r": idx_r.cpu(), "wt_r": wt_r.cpu()}


def _f64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.float().numpy().astype(np.float64) if t.dtype == torch.bfloat16 else t.numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def assert_close(got, want, rtol, what):
    got, want = _f64(got), _f64(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    scale = np.sqrt(np.mean(want ** 2)) if want.size else 0.0
    err = np.abs(got - want)
    bound = rtol * (np.abs(want) + scale)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())}/{err.size} beyond rtol {rtol}; worst at {i}: "
                             f"got {got[i]!r} want {want[i]!r} (rms {scale:.3g})")


def oracle_keys(cfg, q: np.ndarray, subkeys_h: np.ndarray, k: int):
    """The oracle's top-(k+1) slots and their scores for one query (margin checks)."""
    s_list = oracle.factor_scores(q, subkeys_h, cfg.factor_dims, cfg.d_sub)
    ranks = [oracle.factor_ranks(s) for s in s_list]
    S = oracle.slot_scores(s_list)
    kk = min(k + 1, S.shape[0])
    idx = oracle.topk_slots(S, ranks, kk)
    return idx, S


def check_selection(cfg, q: np.ndarray, subkeys_h: np.ndarray, k: int, gpu_idx: np.ndarray,
                    gpu_wt: np.ndarray, ora_idx: np.ndarray, ora_wt: np.ndarray) -> bool:
    """Compare one row's selection.  Returns True if it matches exactly, False if it is a
    valid near-tie alternative (then the histories may diverge); raises otherwise."""
    gpu_idx = np.asarray(gpu_idx, dtype=np.int64)
    if np.array_equal(gpu_idx, ora_idx):
        assert_close(gpu_wt, ora_wt, 1e-5, "selection weights")
        return True
    idx_k1, S = oracle_keys(cfg, q, subkeys_h, k)
    if set(gpu_idx.tolist()) == set(ora_idx.tolist()):
        # same slots in another order: only slots whose scores tie within the margin may swap
        g_scores = S[gpu_idx].astype(np.float64)
        scale = max(abs(float(g_scores.max())), 1e-30)
        assert np.all(np.diff(g_scores) <= MARGIN * scale), "GPU order not by score"
        go, oo = np.argsort(gpu_idx), np.argsort(ora_idx)
        assert_close(np.asarray(gpu_wt)[go], np.asarray(ora_wt)[oo], 1e-5, "selection weights")
        return True
    s_sel = S[ora_idx].astype(np.float64)
    scale = max(abs(float(s_sel[0])), 1e-30)
    kth = float(S[idx_k1[k - 1]])
    nxt = float(S[idx_k1[k]]) if len(idx_k1) > k else -np.inf
    margin_ok = (kth - nxt) > MARGIN * scale
    if margin_ok and set(gpu_idx.tolist()) != set(ora_idx.tolist()):
        raise AssertionError(f"selected set differs with a clear margin ({kth - nxt:.3g}): "
                             f"gpu {sorted(gpu_idx.tolist())[:8]}... oracle {sorted(ora_idx.tolist())[:8]}...")
    # valid top-k within the margin: every GPU pick scores at least the oracle's k-th - margin,
    # the GPU order is non-increasing within the margin, the ids are distinct and in range
    assert len(set(gpu_idx.tolist())) == k
    assert gpu_idx.min() >= 0 and gpu_idx.max() < S.shape[0]
    g_scores = S[gpu_idx].astype(np.float64)
    assert np.all(g_scores >= kth - MARGIN * scale - 1e-30), "a GPU pick scores below the k-th"
    assert np.all(np.diff(g_scores) <= MARGIN * scale), "GPU order not by score"
    return False


def compare_stream(cfg, d: dict, gpu: dict, b: int, h: int, *, T=None) -> dict:
    """Run the oracle on stream (b, h) and compare every token's selection, y and the
    final bank with the GPU's.

    The oracle is driven token by token: where the GPU's selection is exact it keeps
    its own; where the GPU took a different valid top-k at a near tie (check_selection)
    it continues on the GPU's slots, so the histories stay the same and nothing after
    the tie goes uncompared.  Returns {'rows': tokens compared, 'near_ties': number of
    such picks, 'near_tie_tokens': their tokens}."""
    T = gpu["y"].shape[1] if T is None else T
    q_w = _f64(d["q_w"][b, :T, h])
    q_r = _f64(d["q_r"][b, :T, h])
    K = _f64(d["subkeys"][h])
    bank0 = d["bank_init"][h] if "bank_init" in d else d["bank"][b, h]
    M = _f64(bank0).copy()
    near = []
    g_idx = (gpu["idx_w"][b, :T, h].numpy(), gpu["idx_r"][b, :T, h].numpy())
    g_wt = (gpu["wt_w"][b, :T, h].numpy(), gpu["wt_r"][b, :T, h].numpy())
    qs, ks = (q_w, q_r), (cfg.W, cfg.R)

    def pick(t, which, idx, w):
        gi = g_idx[which][t]
        exact = check_selection(cfg, qs[which][t], K, ks[which], gi, g_wt[which][t], idx, w)
        if exact:
            return None
        near.append(t)
        return np.asarray(gi, dtype=np.int64)

    o = oracle.run_stream(M, q_w, q_r, _f64(d["k_val"][b, :T, h]), _f64(d["gates"][b, :T, h]), K,
                          factor_dims=cfg.factor_dims, d_sub=cfg.d_sub, W=cfg.W, R=cfg.R,
                          act_dtype=cfg.act_dtype, bank_dtype=cfg.bank_dtype, pick=pick)
    assert_close(gpu["y"][b, :T, h], o["y"], RTOL[cfg.act_dtype], f"y[{b},:,{h}]")
    if T == gpu["y"].shape[1]:
        assert_close(gpu["bank"][b, h], M, RTOL[cfg.bank_dtype], f"bank[{b},{h}]")
    return {"rows": T, "near_ties": len(near), "near_tie_tokens": sorted(set(near))}
