"""CPU oracle for the Sparse Delta Memory (SDM) write/read op and decode step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module: only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference arm of
``bench.py`` call it.  It shares no code with the CUDA path.

It is a plain, slow restatement of what the op computes, token by token, for one
stream (batch element b, head h) at a time, scoring ALL N slots by brute force.
Floating point is float64 except where the pages fix float32 (the slot score is
"the float32 sum of the factor scores"), and where a stored value is rounded to
its storage type (bank rows after each token's update, the read output).

Sources (page title > section):
  * sparse-delta-memory README > introduction: SDM reads and writes a large sparse
    memory addressed by product keys, with gated (forget/input) delta-rule updates;
    README > prior ideas: product-key memory (Lample et al.) and the gated delta
    rule (Yang et al.).
  * sparse-delta-memory CHANGELOG > 2.0.0 > Upgrading from v1: exact top-k ties go
    to the larger rank sum, then the larger first rank; the slot score is the
    float32 sum of the factor scores; chunk_size changes outputs only through
    rounding.
  * CHANGELOG > 2.0.0 > New: any number of product-key factors of any widths,
    exact product-key top-k.
  * CHANGELOG > 2.0.0 > Removed: reads happen inside the write/read call.
  * lumen PR #29 > Donating is a permission: the in-place (donated) and copying
    step run one body and agree bit for bit.

Readings where the pages are silent:
  * update: the coupled gated delta rule restricted to the W selected rows,
        m_j = alpha * M[i_j];  p = sum_j w_j m_j;  M[i_j] <- m_j + beta w_j (v - p)
    (the forget gate decays only the selected rows);
  * write/read weights: softmax of the selected slot scores, no temperature;
  * gates: the op takes post-sigmoid values (alpha, beta), one pair per token and head;
  * "rank" in the tie rule: a factor's ascending score rank (larger = larger
    score), equal factor scores ordered by index; ties left after the first rank
    are broken by the second rank, then the third, ... (larger first);
  * slot id: mixed radix over the factor indices, the first factor most significant;
  * the read follows the token's own write;
  * a bank stored in bfloat16 is rounded to bfloat16 after every token.

Parity pins: see tests/test_oracle_pins.py (brute-force vs product-key top-k, the
tie rule on constructed ties, alpha=1/beta=0 identity, single full-strength write,
the scalar closed form of repeated single-slot writes, the dense-matrix form of
the gated delta rule, the read as a weighted gather).  The choice of the coupled
update (first reading above) among the update rules the pages' words allow is
not pinned by the pages: "parity unpinned" for that reading.
"""

from __future__ import annotations

import math
from typing import Callable, Iterable, Optional

import numpy as np

__all__ = [
    "round_to_bf16", "round_to", "factor_scores", "factor_ranks", "slot_scores",
    "slot_tie_keys", "topk_slots", "softmax_weights", "select", "weights_of", "gated_delta_write",
    "weighted_read", "run_stream", "sdm_write_read", "sdm_decode_step",
]


# --------------------------------------------------------------------------- rounding

def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even), returned as float64.

    One rounding from float64 (a float64 -> float32 -> bfloat16 chain would round
    twice).  bfloat16 keeps 8 significant bits and float32's exponent range; the
    values here stay far from the subnormal and overflow ranges.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                     # x = m * 2**e, 0.5 <= |m| < 1
    r = np.rint(np.ldexp(m, 8))            # 8 significant bits, ties to even
    return np.ldexp(r, e - 8)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round to a storage type ("f32", "bf16" or "f64"), returned as float64."""
    if dtype == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
    if dtype == "bf16":
        return round_to_bf16(x)
    if dtype == "f64":
        return np.asarray(x, dtype=np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


# --------------------------------------------------------------------------- scoring

def factor_scores(q: np.ndarray, subkeys: np.ndarray, factor_dims, d_sub: int) -> list:
    """Per-factor sub-key scores of one query (product-key memory, Lample et al.).

    q: [F*d_sub] query; subkeys: [sum(n_f), d_sub] of one head, factor f at row
    offset sum_{g<f} n_g.  s_f[a] = <q[f*d_sub:(f+1)*d_sub], K_f[a]>, the dot product
    taken in float64 and rounded once to float32.
    """
    q = np.asarray(q, dtype=np.float64)
    out = []
    off = 0
    for f, n in enumerate(factor_dims):
        qf = q[f * d_sub:(f + 1) * d_sub]
        Kf = np.asarray(subkeys[off:off + n], dtype=np.float64)
        out.append((Kf @ qf).astype(np.float32))
        off += n
    return out


def factor_ranks(s: np.ndarray) -> np.ndarray:
    """Ascending rank of each sub-key score: #{a' : (s[a'], a') < (s[a], a)}.

    A larger rank means a larger score; equal scores are ordered by index.
    """
    n = s.shape[0]
    order = np.lexsort((np.arange(n), s))       # primary key s, then index, ascending
    rank = np.empty(n, dtype=np.int64)
    rank[order] = np.arange(n)
    return rank


def slot_scores(s_list: list) -> np.ndarray:
    """Score of every slot: the float32 sum of its factor scores, left to right.

    Slot n = (...(a_1 n_2 + a_2) n_3 + a_3 ...) (first factor most significant);
    S[n] = fl32(fl32(s_1[a_1] + s_2[a_2]) + s_3[a_3]) ...
    """
    S = np.asarray(s_list[0], dtype=np.float32)
    for s in s_list[1:]:
        S = (S[:, None] + np.asarray(s, dtype=np.float32)[None, :]).reshape(-1)
    return S


def slot_tie_keys(rank_list: list, slots: np.ndarray) -> tuple:
    """Rank sum and per-factor ranks of the given slots (slot layout of ``slot_scores``)."""
    dims = [r.shape[0] for r in rank_list]
    digits = np.unravel_index(np.asarray(slots, dtype=np.int64), dims)   # (a_1, ..., a_F)
    per_factor = [rank_list[f][digits[f]] for f in range(len(dims))]
    rank_sum = np.zeros(len(slots), dtype=np.int64)
    for r in per_factor:
        rank_sum = rank_sum + r
    return rank_sum, per_factor


def topk_slots(S: np.ndarray, ranks: list, k: int, prefilter: bool = True) -> np.ndarray:
    """Exact top-k slot ids, best first.

    Order (CHANGELOG > Upgrading from v1): larger slot score; on equal score the
    larger rank sum; then the larger first rank; then the larger second rank, ...
    With ``prefilter`` the full sort runs only over slots whose score is at least
    the k-th largest score: every slot of the top k is among them, since the k
    best slots carry the k largest scores.
    """
    N = S.shape[0]
    if prefilter and N > 4 * k:
        kth = np.partition(S, N - k)[N - k]
        cand = np.nonzero(S >= kth)[0]
    else:
        cand = np.arange(N)
    rank_sum, per_factor = slot_tie_keys(ranks, cand)
    keys = [-r for r in reversed(per_factor)] + [-rank_sum, -S[cand].astype(np.float64)]
    order = np.lexsort(tuple(keys))             # last key primary, all ascending
    return cand[order[:k]]


def softmax_weights(S_sel: np.ndarray) -> np.ndarray:
    """w_j = exp(S_j - S_0) / sum_i exp(S_i - S_0) over the selected slots (float64)."""
    x = np.asarray(S_sel, dtype=np.float64)
    e = np.exp(x - x[0])
    return e / e.sum()


def select(q: np.ndarray, subkeys: np.ndarray, factor_dims, d_sub: int, k: int,
           prefilter: bool = True):
    """Product-key scoring and exact top-k of one query: (slot ids, weights, scores)."""
    s_list = factor_scores(q, subkeys, factor_dims, d_sub)
    ranks = [factor_ranks(s) for s in s_list]
    S = slot_scores(s_list)
    idx = topk_slots(S, ranks, k, prefilter=prefilter)
    w = softmax_weights(S[idx])
    return idx, w, S[idx]


def weights_of(q: np.ndarray, subkeys: np.ndarray, factor_dims, d_sub: int, idx) -> np.ndarray:
    """Softmax weights of the given slots, in the given order, from this query's slot scores.

    Used when a caller supplies the selected slots itself: at a near tie several
    slot sets are valid top-k answers, and the rest of the arithmetic (weights,
    update, read) is the same for any of them.
    """
    S = slot_scores(factor_scores(q, subkeys, factor_dims, d_sub))
    return softmax_weights(S[np.asarray(idx, dtype=np.int64)])


# --------------------------------------------------------------------------- update / read

def gated_delta_write(M: np.ndarray, idx: np.ndarray, w: np.ndarray, alpha: float,
                      beta: float, v: np.ndarray, bank_dtype: str) -> None:
    """Gated delta-rule write of one token into the selected rows of M (in place).

    m_j = alpha M[i_j];  p = sum_j w_j m_j;  M[i_j] <- round(m_j + beta w_j (v - p)).
    This is S' = S D (I - beta k k^T) + beta v k^T for S = M^T, key k = w on the
    selected slots and D = identity with alpha on the selected slots.  The W slots
    are distinct, so the rows update independently of their order.
    """
    m = float(alpha) * M[idx]                       # [W, d_v]
    p = w @ m                                       # [d_v]
    M[idx] = round_to(m + float(beta) * w[:, None] * (np.asarray(v, np.float64) - p)[None, :],
                      bank_dtype)


def weighted_read(M: np.ndarray, idx: np.ndarray, r: np.ndarray) -> np.ndarray:
    """y = sum_j r_j M[i_j] (float64, unrounded)."""
    return r @ M[idx]


def run_stream(M: np.ndarray, q_w: np.ndarray, q_r: np.ndarray, k_val: np.ndarray,
               gates: np.ndarray, subkeys: np.ndarray, *, factor_dims, d_sub: int, W: int,
               R: int, act_dtype: str, bank_dtype: str, prefilter: bool = True,
               pick: Optional[Callable] = None) -> dict:
    """Run T tokens of one stream through the op, in token order; M advances in place.

    q_w, q_r: [T, F*d_sub]; k_val: [T, d_v]; gates: [T, 2] = (alpha, beta);
    subkeys: [sum(n_f), d_sub] of this head; M: [N, d_v] float64 holding values of
    the bank type.  Returns y [T, d_v] (rounded to the activation type), the write
    and read slot ids and weights.

    ``pick(t, which, idx, w)`` (which = 0 for the write query, 1 for the read query),
    if given, sees each exact top-k and may return other slot ids to use instead (a
    different valid answer at a near tie); their weights are then the softmax of
    their own slot scores (``weights_of``), and the update and read run on them.
    Returning None keeps the exact top-k.
    """
    T = q_w.shape[0]
    d_v = M.shape[1]
    y = np.zeros((T, d_v), dtype=np.float64)
    idx_w = np.zeros((T, W), dtype=np.int64)
    idx_r = np.zeros((T, R), dtype=np.int64)
    wt_w = np.zeros((T, W), dtype=np.float64)
    wt_r = np.zeros((T, R), dtype=np.float64)
    for t in range(T):
        iw, ww, _ = select(q_w[t], subkeys, factor_dims, d_sub, W, prefilter)
        ir, rr, _ = select(q_r[t], subkeys, factor_dims, d_sub, R, prefilter)
        if pick is not None:
            alt = pick(t, 0, iw, ww)
            if alt is not None:
                iw = np.asarray(alt, dtype=np.int64)
                ww = weights_of(q_w[t], subkeys, factor_dims, d_sub, iw)
            alt = pick(t, 1, ir, rr)
            if alt is not None:
                ir = np.asarray(alt, dtype=np.int64)
                rr = weights_of(q_r[t], subkeys, factor_dims, d_sub, ir)
        alpha, beta = float(gates[t, 0]), float(gates[t, 1])
        gated_delta_write(M, iw, ww, alpha, beta, k_val[t], bank_dtype)
        y[t] = round_to(weighted_read(M, ir, rr), act_dtype)
        idx_w[t], wt_w[t], idx_r[t], wt_r[t] = iw, ww, ir, rr
    return {"y": y, "idx_w": idx_w, "wt_w": wt_w, "idx_r": idx_r, "wt_r": wt_r}


def _f64(x) -> np.ndarray:
    """float64 view of a numpy array or a (CPU) torch tensor of any float type."""
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if str(x.dtype) in ("torch.bfloat16", "torch.float16"):
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def sdm_write_read(q_w, q_r, k_val, gates, subkeys, bank, *, factor_dims, W: int, R: int,
                   chunk_size: int = 64, act_dtype: str = "f32", bank_dtype: str = "f32",
                   streams: Optional[Iterable] = None, T_limit: Optional[int] = None,
                   prefilter: bool = True) -> dict:
    """The chunked write/read op over all (or the listed) streams.

    q_w, q_r [B,T,H,F*d_sub]; k_val [B,T,H,d_v]; gates [B,T,H,2]; subkeys [H,sum n_f,d_sub];
    bank [B,H,N,d_v] (per-stream tables) or [H,N,d_v] (a learned table each stream
    starts from).  ``chunk_size`` is accepted and has no effect: the oracle has no
    chunks, it applies tokens one at a time (CHANGELOG > Upgrading from v1: the chunk
    size changes outputs only through rounding).  ``streams``: iterable of (b, h) to
    run (default all); ``T_limit``: run only the first T_limit tokens.

    Returns a dict of float64 / int64 arrays keyed by (b, h):
      out[(b, h)] = {"y": [T, d_v], "bank": [N, d_v], "idx_w", "wt_w", "idx_r", "wt_r"}.
    """
    del chunk_size
    q_w, q_r, k_val, gates = _f64(q_w), _f64(q_r), _f64(k_val), _f64(gates)
    subkeys = _f64(subkeys)
    B, T, H, _ = q_w.shape
    d_sub = subkeys.shape[2]
    if T_limit is not None:
        T = min(T, T_limit)
    if streams is None:
        streams = [(b, h) for b in range(B) for h in range(H)]
    out = {}
    for (b, h) in streams:
        M = _f64(bank[h] if bank.ndim == 3 else bank[b, h]).copy()   # one stream at a time
        res = run_stream(M, q_w[b, :T, h], q_r[b, :T, h], k_val[b, :T, h], gates[b, :T, h],
                         subkeys[h], factor_dims=factor_dims, d_sub=d_sub, W=W, R=R,
                         act_dtype=act_dtype, bank_dtype=bank_dtype, prefilter=prefilter)
        res["bank"] = M
        out[(b, h)] = res
    return out


def sdm_decode_step(q_w, q_r, k_val, gates, subkeys, bank: np.ndarray, *, factor_dims,
                    W: int, R: int, donate: bool = False, act_dtype: str = "f32",
                    bank_dtype: str = "f32"):
    """One single-token step for every stream: (y [B,H,d_v], successor bank).

    q_w, q_r [B,H,F*d_sub]; k_val [B,H,d_v]; gates [B,H,2]; bank [B,H,N,d_v] float64.
    With ``donate`` the successor is written into ``bank`` itself and returned;
    without it ``bank`` is left untouched and a new table is returned.  Both run the
    same body, so they agree bit for bit (lumen PR #29 > Donating is a permission).
    """
    q_w, q_r, k_val, gates, subkeys = _f64(q_w), _f64(q_r), _f64(k_val), _f64(gates), _f64(subkeys)
    out = bank if donate else bank.copy()
    B, H = q_w.shape[0], q_w.shape[1]
    d_sub = subkeys.shape[2]
    y = np.zeros((B, H, out.shape[-1]), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            res = run_stream(out[b, h], q_w[b, h][None], q_r[b, h][None], k_val[b, h][None],
                             gates[b, h][None], subkeys[h], factor_dims=factor_dims,
                             d_sub=d_sub, W=W, R=R, act_dtype=act_dtype, bank_dtype=bank_dtype)
            y[b, h] = res["y"][0]
    return y, out

