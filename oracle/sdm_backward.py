"""CPU oracle for the backward of the SDM write/read op (gradients of a scalar loss).

TEST INFRASTRUCTURE ONLY, like sdm_oracle.py: nothing in the product path imports it.

What the pages fix (page title > section):
  * sparse-delta-memory CHANGELOG > 2.0.0 > New: exact product-key top-k with a
    deterministic sparse backward; > Deterministic: every gradient is bitwise
    repeatable (v1 used float atomics);
  * CHANGELOG > 2.0.0 > Package (bf16 snapshots): training saves a snapshot of the rows
    a step overwrites (float32 by default) for the backward;
  * CHANGELOG > 2.0.0 > Behavior changes: the first backward restores the bank in place
    (a second backward through the same call is refused).

The gradient itself is the plain chain rule through the oracle's forward
(sdm_oracle.run_stream), taken in float64; the pages print no formulas for it, so it
is pinned against central finite differences of that forward (tests/test_oracle_backward.py).
Readings where the pages are silent:
  * the selected slot ids are piecewise constant in the queries and sub-keys: the
    gradient flows through the softmax weights of the selected slots only;
  * the float32 rounding of factor and slot scores and the rounding of stored bank rows
    and outputs are passed straight through (their derivative is taken as 1);
  * gates are the post-sigmoid values (alpha, beta) the op takes, so their gradient is
    with respect to those values;
  * snapshot precision (CHANGELOG > 2.0.0 > Package, bf16 snapshots): the snapshot of the
    rows a token overwrites holds them exactly by default (a float32 snapshot of a float32
    or bfloat16 bank), or rounded to ``snapshot_dtype`` ("bf16");
    the backward reads the snapshot wherever it needs the rows before the write (the
    alpha, beta and weight gradients, so those of the gates and queries) and restores
    the bank from it.  On a bfloat16 bank the rows are already bfloat16, so a bfloat16
    snapshot changes nothing (the pages state this, bit for bit).

Per token t of one stream, with X_j the W rows before the write (the snapshot),
m_j = alpha X_j, p = sum_j w_j m_j, u = v - p, M'[i_j] = m_j + beta w_j u, and
y = sum_j r_j M'[i^r_j], given G = dL/dM' (all rows) and dy:
  read:   G[i^r_j] += r_j dy;            dr_j = <dy, M'[i^r_j]>
  write:  G_j = G[i_j];  dv = beta sum_j w_j G_j;  dp = -dv;  dbeta = sum_j w_j <G_j, u>
          dm_j = G_j + w_j dp;  dw_j = beta <G_j, u> + <dp, m_j>;  dalpha = sum_j <dm_j, X_j>
          G[i_j] <- alpha dm_j  (the gradient with respect to the rows before the write)
  softmax: dS_j = w_j (dw_j - sum_k w_k dw_k)   (the same for the read weights)
  scores:  S_j = sum_f s_f[a_f(j)]  ->  ds_f[a] += dS_j;  s_f[a] = <q_f, K_f[a]>
           -> dq_f += ds_f[a] K_f[a],  dK_f[a] += ds_f[a] q_f.
"""

from __future__ import annotations

from typing import Callable, Iterable, Optional

import numpy as np

from .sdm_oracle import (_f64, factor_ranks, round_to, slot_scores, softmax_weights,
                         topk_slots)

__all__ = ["select_record", "record_of", "stream_forward", "stream_backward", "sdm_write_read_backward"]


def _factor_scores(q: np.ndarray, subkeys: np.ndarray, factor_dims, d_sub: int, exact: bool) -> list:
    """Per-factor scores, rounded to float32 as the forward does unless ``exact``."""
    out, off = [], 0
    for f, n in enumerate(factor_dims):
        s = np.asarray(subkeys[off:off + n], np.float64) @ np.asarray(q[f * d_sub:(f + 1) * d_sub], np.float64)
        out.append(s if exact else s.astype(np.float32).astype(np.float64))
        off += n
    return out


def select_record(q: np.ndarray, subkeys: np.ndarray, factor_dims, d_sub: int, k: int,
                  exact: bool = False) -> dict:
    """Selection of one query with what its backward needs.

    Returns slot ids (best first), their factor indices [k, F], softmax weights and slot
    scores.  With ``exact`` the factor scores and slot scores stay float64 (for the
    finite-difference checks); otherwise this is sdm_oracle.select.
    """
    s_list = _factor_scores(q, subkeys, factor_dims, d_sub, exact)
    ranks = [factor_ranks(s) for s in s_list]
    if exact:
        S = s_list[0]
        for s in s_list[1:]:
            S = (S[:, None] + s[None, :]).reshape(-1)
    else:
        S = slot_scores(s_list).astype(np.float64)
    idx = topk_slots(S, ranks, k)
    digits = np.stack(np.unravel_index(idx, tuple(int(n) for n in factor_dims)), axis=1)
    return {"idx": idx, "digits": digits, "w": softmax_weights(S[idx]), "S": S[idx]}


def record_of(q: np.ndarray, subkeys: np.ndarray, factor_dims, d_sub: int, idx) -> dict:
    """select_record for slots a caller supplies (in its order), scored as the forward does."""
    idx = np.asarray(idx, dtype=np.int64)
    S = slot_scores(_factor_scores(q, subkeys, factor_dims, d_sub, False)).astype(np.float64)
    digits = np.stack(np.unravel_index(idx, tuple(int(n) for n in factor_dims)), axis=1)
    return {"idx": idx, "digits": digits, "w": softmax_weights(S[idx]), "S": S[idx]}


def stream_forward(M: np.ndarray, q_w, q_r, k_val, gates, subkeys, *, factor_dims, d_sub: int, W: int,
                   R: int, act_dtype: str = "f32", bank_dtype: str = "f32", exact: bool = False,
                   snapshot_dtype: Optional[str] = None, pick: Optional[Callable] = None) -> dict:
    """The forward of one stream (M advances in place), keeping the backward's record.

    Same arithmetic as sdm_oracle.run_stream; additionally stores per token the write
    and read selections and the snapshot of the W rows before the write: exact, or
    rounded to ``snapshot_dtype`` (the forward itself uses the rows as they are).
    ``exact``: float64 scores (bank_dtype / act_dtype "f64" then make the whole forward
    float64).  ``pick(t, which, idx, w)``: as in sdm_oracle.run_stream, may return other
    slot ids (a different valid top-k at a near tie) whose weights are then the softmax
    of their own slot scores.
    """
    T, d_v = q_w.shape[0], M.shape[1]
    y = np.zeros((T, d_v))
    rec = []
    for t in range(T):
        sw = select_record(q_w[t], subkeys, factor_dims, d_sub, W, exact)
        sr = select_record(q_r[t], subkeys, factor_dims, d_sub, R, exact)
        if pick is not None:
            alt = pick(t, 0, sw["idx"], sw["w"])
            if alt is not None:
                sw = record_of(q_w[t], subkeys, factor_dims, d_sub, alt)
            alt = pick(t, 1, sr["idx"], sr["w"])
            if alt is not None:
                sr = record_of(q_r[t], subkeys, factor_dims, d_sub, alt)
        alpha, beta = float(gates[t, 0]), float(gates[t, 1])
        X = M[sw["idx"]].copy()
        m = alpha * X
        p = sw["w"] @ m
        M[sw["idx"]] = round_to(m + beta * sw["w"][:, None] * (np.asarray(k_val[t], np.float64) - p)[None, :],
                                bank_dtype)
        y[t] = round_to(sr["w"] @ M[sr["idx"]], act_dtype)
        rec.append({"w": sw, "r": sr, "X": X if snapshot_dtype is None else round_to(X, snapshot_dtype)})
    return {"y": y, "rec": rec}


def _scores_backward(sel: dict, dsel_w: np.ndarray, q: np.ndarray, subkeys: np.ndarray, factor_dims,
                     d_sub: int, dq: np.ndarray, dK: np.ndarray) -> None:
    """Softmax and score backward of one selection: accumulates into dq [F*d_sub], dK."""
    w = sel["w"]
    dS = w * (dsel_w - np.dot(w, dsel_w))
    offs = np.concatenate([[0], np.cumsum(factor_dims)[:-1]]).astype(np.int64)
    for f in range(len(factor_dims)):
        ds = np.zeros(int(factor_dims[f]))
        np.add.at(ds, sel["digits"][:, f], dS)
        Kf = np.asarray(subkeys[offs[f]:offs[f] + int(factor_dims[f])], np.float64)
        qf = np.asarray(q[f * d_sub:(f + 1) * d_sub], np.float64)
        dq[f * d_sub:(f + 1) * d_sub] += ds @ Kf
        dK[offs[f]:offs[f] + int(factor_dims[f])] += ds[:, None] * qf[None, :]


def stream_backward(M: np.ndarray, fwd: dict, dy: np.ndarray, dM: np.ndarray, q_w, q_r, k_val, gates,
                    subkeys, *, factor_dims, d_sub: int) -> dict:
    """Reverse sweep over the tokens of one stream.

    M: the bank after the forward (float64), restored in place to the bank before it
    from the snapshots; dy [T, d_v]: dL/dy; dM [N, d_v]: dL/d(final bank).  Returns the
    gradients with respect to the initial bank, k_val, gates (alpha, beta), q_w, q_r and
    the head's sub-keys.
    """
    T = dy.shape[0]
    G = np.array(dM, dtype=np.float64)
    d_kv = np.zeros((T, M.shape[1]))
    d_g = np.zeros((T, 2))
    d_qw = np.zeros(np.shape(q_w))
    d_qr = np.zeros(np.shape(q_r))
    d_K = np.zeros(np.shape(subkeys))
    for t in range(T - 1, -1, -1):
        rc = fwd["rec"][t]
        sw, sr, X = rc["w"], rc["r"], rc["X"]
        alpha, beta = float(gates[t, 0]), float(gates[t, 1])
        v = np.asarray(k_val[t], np.float64)
        # read (after the write): rows of M are the post-write values here
        rows_r = M[sr["idx"]]
        dr = rows_r @ dy[t]
        np.add.at(G, sr["idx"], sr["w"][:, None] * dy[t][None, :])
        # write
        w = sw["w"]
        m = alpha * X
        u = v - w @ m
        Gj = G[sw["idx"]]
        dv = beta * (w @ Gj)
        dp = -dv
        dm = Gj + w[:, None] * dp[None, :]
        d_kv[t] = dv
        d_g[t, 1] = float(np.sum(w * (Gj @ u)))
        d_g[t, 0] = float(np.sum(dm * X))
        dw = beta * (Gj @ u) + m @ dp
        G[sw["idx"]] = alpha * dm
        M[sw["idx"]] = X                                            # restore from the snapshot
        _scores_backward(sr, dr, q_r[t], subkeys, factor_dims, d_sub, d_qr[t], d_K)
        _scores_backward(sw, dw, q_w[t], subkeys, factor_dims, d_sub, d_qw[t], d_K)
    return {"bank": G, "k_val": d_kv, "gates": d_g, "q_w": d_qw, "q_r": d_qr, "subkeys": d_K}


def sdm_write_read_backward(q_w, q_r, k_val, gates, subkeys, bank, dy, dbank, *, factor_dims, W: int, R: int,
                            act_dtype: str = "f32", bank_dtype: str = "f32", snapshot_dtype: Optional[str] = None,
                            streams: Optional[Iterable] = None, pick: Optional[Callable] = None,
                            exact: bool = False) -> dict:
    """Gradients of the write/read op over all (or the listed) streams.

    Inputs as sdm_oracle.sdm_write_read (bank [B,H,N,d_v] per stream); dy [B,T,H,d_v] and
    dbank [B,H,N,d_v]: the loss gradients with respect to y and the final bank.  Runs the
    forward with its record, then the reverse sweep, stream by stream.  Sub-key gradients
    of one head are summed over batch elements in increasing b.  Returns float64 arrays
    shaped like the inputs.  ``pick(b, h)``, if given, returns the per-stream pick
    passed to stream_forward (or None); ``exact`` is stream_forward's (float64 scores).
    """
    q_w, q_r, k_val, gates, subkeys = _f64(q_w), _f64(q_r), _f64(k_val), _f64(gates), _f64(subkeys)
    bank, dy, dbank = _f64(bank), _f64(dy), _f64(dbank)
    B, T, H, _ = q_w.shape
    d_sub = subkeys.shape[2]
    if streams is None:
        streams = [(b, h) for b in range(B) for h in range(H)]
    out = {"bank": np.zeros_like(bank), "k_val": np.zeros_like(k_val), "gates": np.zeros_like(gates),
           "q_w": np.zeros_like(q_w), "q_r": np.zeros_like(q_r), "subkeys": np.zeros_like(subkeys)}
    for (b, h) in sorted(streams):
        M = bank[b, h].copy()
        fwd = stream_forward(M, q_w[b, :, h], q_r[b, :, h], k_val[b, :, h], gates[b, :, h], subkeys[h],
                             factor_dims=factor_dims, d_sub=d_sub, W=W, R=R, act_dtype=act_dtype,
                             bank_dtype=bank_dtype, snapshot_dtype=snapshot_dtype, exact=exact,
                             pick=None if pick is None else pick(b, h))
        g = stream_backward(M, fwd, dy[b, :, h], dbank[b, h], q_w[b, :, h], q_r[b, :, h], k_val[b, :, h],
                            gates[b, :, h], subkeys[h], factor_dims=factor_dims, d_sub=d_sub)
        out["bank"][b, h] = g["bank"]
        out["k_val"][b, :, h] = g["k_val"]
        out["gates"][b, :, h] = g["gates"]
        out["q_w"][b, :, h] = g["q_w"]
        out["q_r"][b, :, h] = g["q_r"]
        out["subkeys"][h] += g["subkeys"]
    return out
