"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test fixes part of what the oracle computes by an independent route: a
hand-worked example of a rule the SDM pages state, a closed form, a special case
that reduces to a library routine, a different algorithm (product-key pruning
instead of brute force), or the dense-matrix form of the gated delta rule.  Each
is chosen so that a plausible slip in the oracle (a dropped term, a flipped sign
or rank direction, a transposed slot layout, reading before writing) fails it.
"""

import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import sdm_inputs


# --------------------------------------------------------------------------- helpers

def _nearest_f32(x: Fraction) -> np.float32:
    """Correctly rounded float32 of an exact rational (ties to even)."""
    approx = np.float32(float(x))
    cands = {approx, np.nextafter(approx, np.float32(np.inf)), np.nextafter(approx, np.float32(-np.inf))}
    best = None
    for c in sorted(cands):
        d = abs(Fraction(float(c)) - x)
        if best is None or d < best[0] or (d == best[0] and (c.view(np.uint32) & 1) == 0):
            best = (d, c)
    return best[1]


def _product_key_topk(s_list, k):
    """Independent product-key top-k (Lample et al.) with rank-dominance pruning.

    Each factor is sorted best first by (score, index); a tuple of positions
    (p_1..p_F) can be in the top k only if prod(p_f + 1) <= k, because every tuple
    it dominates position-wise scores at least as high (float addition is monotone)
    and wins any tie on the rank sum.  The survivors are ordered by the key of the
    tie rule: score, rank sum, first rank, second rank, ... all larger first.
    """
    F = len(s_list)
    dims = [len(s) for s in s_list]
    orders, ranks = [], []
    for s in s_list:
        n = len(s)
        desc = sorted(range(n), key=lambda a: (float(s[a]), a), reverse=True)
        orders.append(desc)
        r = [0] * n
        for pos, a in enumerate(desc):
            r[a] = n - 1 - pos                # ascending rank
        ranks.append(r)
    kf = [min(k, n) for n in dims]
    cands = []
    for pos in itertools.product(*[range(x) for x in kf]):
        if math.prod(p + 1 for p in pos) > k:
            continue
        a = [orders[f][pos[f]] for f in range(F)]
        S = np.float32(s_list[0][a[0]])
        for f in range(1, F):
            S = np.float32(S + np.float32(s_list[f][a[f]]))
        slot = 0
        for f in range(F):
            slot = slot * dims[f] + a[f]
        rk = [ranks[f][a[f]] for f in range(F)]
        cands.append(((float(S), sum(rk), *rk), slot))
    cands.sort(key=lambda c: c[0], reverse=True)
    return [slot for _, slot in cands[:k]]


def _random_subkeys(rng, dims, d_sub):
    return rng.standard_normal((sum(dims), d_sub)) / math.sqrt(d_sub)


# --------------------------------------------------------------------------- scoring

def test_factor_score_uses_each_factor_slice_and_offset():
    # A one-hot query e_{f*d_sub+d} makes s_f[a] = K_f[a, d] and every other factor 0.
    rng = np.random.default_rng(0)
    dims, d_sub = (3, 5, 4), 6
    K = _random_subkeys(rng, dims, d_sub).astype(np.float32)
    offs = [0, 3, 8]
    for f in range(3):
        for d in range(d_sub):
            q = np.zeros(3 * d_sub, dtype=np.float32)
            q[f * d_sub + d] = 1.0
            s = oracle.factor_scores(q, K, dims, d_sub)
            for g in range(3):
                want = K[offs[g]:offs[g] + dims[g], d] if g == f else np.zeros(dims[g], np.float32)
                np.testing.assert_array_equal(s[g], want)


def test_factor_score_is_the_correctly_rounded_dot_product():
    rng = np.random.default_rng(1)
    dims, d_sub = (7, 9), 40
    K = _random_subkeys(rng, dims, d_sub).astype(np.float32)
    for _ in range(5):
        q = rng.standard_normal(2 * d_sub).astype(np.float32)
        s = oracle.factor_scores(q, K, dims, d_sub)
        off = 0
        for f, n in enumerate(dims):
            for a in range(n):
                exact = sum(Fraction(float(q[f * d_sub + d])) * Fraction(float(K[off + a, d]))
                            for d in range(d_sub))
                assert s[f][a] == _nearest_f32(exact)
            off += n


def test_factor_ranks_hand_example():
    # ascending (score, index): (-1,1) (0.5,0) (0.5,2) (2,3)
    s = np.array([0.5, -1.0, 0.5, 2.0], dtype=np.float32)
    assert list(oracle.factor_ranks(s)) == [1, 0, 2, 3]


def test_slot_layout_first_factor_most_significant():
    # n = (2, 3): slot = a1 * 3 + a2.  Best is a1 = 1 (score 10), a2 = 2 (score 1).
    s1 = np.array([0.0, 10.0], dtype=np.float32)
    s2 = np.array([0.0, 0.0, 1.0], dtype=np.float32)
    S = oracle.slot_scores([s1, s2])
    assert S.dtype == np.float32 and S.shape == (6,)
    assert int(np.argmax(S)) == 5
    assert S[3] == 10.0 and S[2] == 1.0


def test_slot_score_is_float32_sum_left_to_right():
    # fl(fl(a + b) + c) differs from the exact sum and from fl(a + fl(b + c)) here.
    a, b, c = np.float32(1.0), np.float32(2.0 ** -24), np.float32(2.0 ** -24)
    S = oracle.slot_scores([np.array([a]), np.array([b]), np.array([c])])
    assert S[0] == np.float32(1.0)                   # 1 + 2^-24 rounds to 1, twice
    assert np.float32(a + np.float32(b + c)) != S[0]


# --------------------------------------------------------------------------- tie rule

def _select_from_scores(s_list, k):
    ranks = [oracle.factor_ranks(np.asarray(s, np.float32)) for s in s_list]
    S = oracle.slot_scores([np.asarray(s, np.float32) for s in s_list])
    return list(oracle.topk_slots(S, ranks, k, prefilter=False))


def test_tie_rule_equal_scores_two_factors():
    # All scores equal: ranks follow the index.  (1,1) has rank sum 2; (1,0) and
    # (0,1) tie on rank sum 1 and the larger first rank puts (1,0) first.
    assert _select_from_scores([[0.0, 0.0], [0.0, 0.0]], 4) == [3, 2, 1, 0]


def test_tie_rule_equal_scores_three_factors():
    # Rank sum 3: (1,1,1)=7.  Sum 2: (1,1,0)=6 and (1,0,1)=5 share first rank 1, the
    # second rank decides; then (0,1,1)=3.  Sum 1: (1,0,0)=4, (0,1,0)=2, (0,0,1)=1.
    assert _select_from_scores([[0.0, 0.0]] * 3, 8) == [7, 6, 5, 3, 4, 2, 1, 0]


def test_tie_rule_score_tie_between_different_combinations():
    # s1 = [1, 0], s2 = [0, 1]: S(0,1) = 2; S(0,0) = S(1,1) = 1 with rank sums 1 and 1,
    # first ranks 1 and 0, so (0,0) precedes (1,1); S(1,0) = 0 last.
    assert _select_from_scores([[1.0, 0.0], [0.0, 1.0]], 4) == [1, 0, 3, 2]


@pytest.mark.parametrize("dims,k", [((6, 5), 7), ((8, 8), 16), ((4, 5, 3), 9), ((6, 6, 6), 20),
                                    ((3, 4, 2, 3), 10), ((16,), 5)])
def test_brute_force_equals_product_key_topk(dims, k):
    rng = np.random.default_rng(sum(dims) * 31 + k)
    d_sub = 4
    F = len(dims)
    for trial in range(25):
        K = _random_subkeys(rng, dims, d_sub).astype(np.float32)
        if trial % 5 == 1:
            K[1] = K[0]                          # duplicate sub-keys -> equal factor scores
        if trial % 5 == 2:
            K = np.round(K * 2) / 2              # coarse grid -> many equal slot scores
        q = rng.standard_normal(F * d_sub).astype(np.float32)
        if trial % 5 == 3:
            q[:] = 0.0                           # every slot score equal
        s_list = oracle.factor_scores(q, K, dims, d_sub)
        idx, w, S_sel = oracle.select(q, K, dims, d_sub, k, prefilter=False)
        assert list(idx) == _product_key_topk(s_list, k)
        idx2, _, _ = oracle.select(q, K, dims, d_sub, k, prefilter=True)
        assert list(idx2) == list(idx)


def test_grid_inputs_make_scores_exact_in_any_order():
    cfg = sdm_inputs.CONFIGS["layer"].replace(B=1, T=4)
    d = sdm_inputs.make_inputs(cfg, grid=True)
    q = d["q_w"][0, 0, 0].float().numpy()
    K = d["subkeys"][0].float().numpy()
    s = oracle.factor_scores(q, K, cfg.factor_dims, cfg.d_sub)
    # float32 accumulation forward and backward gives the same bits as the oracle's
    for f in range(2):
        prod = (K[f * 256:(f + 1) * 256] * q[f * 512:(f + 1) * 512][None, :]).astype(np.float32)
        fwd = np.zeros(256, np.float32)
        bwd = np.zeros(256, np.float32)
        for d_ in range(512):
            fwd = np.float32(fwd + prod[:, d_])
            bwd = np.float32(bwd + prod[:, 511 - d_])
        np.testing.assert_array_equal(fwd, s[f])
        np.testing.assert_array_equal(bwd, s[f])


# --------------------------------------------------------------------------- weights

def test_softmax_weights_properties():
    S = np.array([3.0, 2.5, 2.5, -1.0], dtype=np.float32)
    w = oracle.softmax_weights(S)
    assert abs(w.sum() - 1.0) < 1e-15
    assert w[1] == w[2]
    assert abs(w[0] / w[3] - math.exp(4.0)) < 1e-9
    assert abs(w[0] - 1.0 / (1.0 + 2 * math.exp(-0.5) + math.exp(-4.0))) < 1e-15


# --------------------------------------------------------------------------- rounding

def test_round_to_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000)).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    np.testing.assert_array_equal(oracle.round_to_bf16(x.astype(np.float64)), want)


def test_round_to_bf16_rounds_once_from_float64():
    x = 1.0 + 2.0 ** -8 + 2.0 ** -30          # just above the bf16 midpoint of [1, 1+2^-7]
    assert oracle.round_to_bf16(np.array([x]))[0] == 1.0 + 2.0 ** -7
    # float32 first would land exactly on the midpoint and tie to even (1.0)
    assert torch.tensor([x], dtype=torch.float32).to(torch.bfloat16).item() == 1.0


# --------------------------------------------------------------------------- update / read

def _tiny_stream(seed, T=12, dims=(8, 8), d_sub=8, d_v=16, W=4, R=4):
    rng = np.random.default_rng(seed)
    F = len(dims)
    K = _random_subkeys(rng, dims, d_sub)
    return dict(
        M=0.02 * rng.standard_normal((math.prod(dims), d_v)),
        q_w=rng.standard_normal((T, F * d_sub)), q_r=rng.standard_normal((T, F * d_sub)),
        k_val=rng.standard_normal((T, d_v)), K=K, dims=dims, d_sub=d_sub, W=W, R=R,
        gates=1.0 / (1.0 + np.exp(-rng.standard_normal((T, 2)))))


def _run(st, gates, bank_dtype="f64", act_dtype="f64"):
    M = st["M"].copy()
    res = oracle.run_stream(M, st["q_w"], st["q_r"], st["k_val"], gates, st["K"],
                            factor_dims=st["dims"], d_sub=st["d_sub"], W=st["W"], R=st["R"],
                            act_dtype=act_dtype, bank_dtype=bank_dtype)
    return M, res


def test_forget_one_input_zero_leaves_bank_unchanged_and_reads_are_a_weighted_gather():
    st = _tiny_stream(4)
    gates = np.tile([1.0, 0.0], (12, 1))
    M0 = st["M"].copy()
    M0r = oracle.round_to(M0, "f32")
    M2 = M0r.copy()
    res2 = oracle.run_stream(M2, st["q_w"], st["q_r"], st["k_val"], gates, st["K"],
                             factor_dims=st["dims"], d_sub=st["d_sub"], W=4, R=4,
                             act_dtype="f64", bank_dtype="f32")
    np.testing.assert_array_equal(M2, M0r)                 # bit-identical bank
    # read = embedding_bag(sum) of the bank rows with per-sample weights (library routine)
    bag = torch.nn.functional.embedding_bag(
        torch.from_numpy(res2["idx_r"].reshape(-1)), torch.from_numpy(M0r),
        offsets=torch.arange(0, res2["idx_r"].size, 4),
        per_sample_weights=torch.from_numpy(res2["wt_r"].reshape(-1)), mode="sum").numpy()
    np.testing.assert_allclose(res2["y"], bag, rtol=0, atol=1e-15)


def test_single_full_strength_write_sets_row_to_value():
    # W = 1: the only weight is 1; beta = 1 gives m + (v - m) = v for any alpha.
    st = _tiny_stream(5, W=1, R=1)
    rng = np.random.default_rng(5)
    gates = np.stack([rng.uniform(0.1, 1.0, 12), np.ones(12)], axis=1)
    for bank_dtype in ("f32", "bf16", "f64"):
        M = oracle.round_to(st["M"], bank_dtype)
        for t in range(12):
            iw, ww, _ = oracle.select(st["q_w"][t], st["K"], st["dims"], st["d_sub"], 1)
            assert ww[0] == 1.0
            v = oracle.round_to(st["k_val"][t], bank_dtype)
            m = gates[t, 0] * M[iw[0]]
            oracle.gated_delta_write(M, iw, ww, gates[t, 0], 1.0, v, bank_dtype)
            if bank_dtype == "f64":
                # fl(m + fl(v - m)) is within 2 ulp of max(|m|, |v|) of v
                bound = 2 * np.spacing(np.maximum(np.abs(m), np.abs(v)))
                assert np.all(np.abs(M[iw[0]] - v) <= bound)
            else:
                # v - m and m + (v - m) are exact in float64 for float32/bfloat16 values,
                # so the stored row is v itself
                np.testing.assert_array_equal(M[iw[0]], v)


def test_repeated_single_slot_writes_follow_the_scalar_closed_form():
    # One slot always wins (its sub-keys dominate for positive queries); with W = 1
    # the row follows M_t = alpha_t (1 - beta_t) M_{t-1} + beta_t v_t, whose unrolled
    # form is M_T = prod_t a_t(1-b_t) M_0 + sum_t b_t v_t prod_{s>t} a_s(1-b_s).
    rng = np.random.default_rng(6)
    T, d_v = 40, 8
    dims, d_sub = (4, 4), 2
    K = np.zeros((8, d_sub))
    K[0] = K[4] = [3.0, 3.0]
    K[1:4] = K[5:8] = rng.uniform(-1, 1, (3, d_sub))
    q = np.abs(rng.standard_normal((T, 2 * d_sub))) + 0.5
    v = rng.standard_normal((T, d_v))
    g = rng.uniform(0.05, 0.95, (T, 2))
    M = rng.standard_normal((16, d_v))
    M0 = M[0].copy()
    oracle.run_stream(M, q, q, v, g, K, factor_dims=dims, d_sub=d_sub, W=1, R=1,
                      act_dtype="f64", bank_dtype="f64")
    decay = g[:, 0] * (1.0 - g[:, 1])
    want = np.prod(decay) * M0
    for t in range(T):
        want = want + g[t, 1] * v[t] * np.prod(decay[t + 1:])
    np.testing.assert_allclose(M[0], want, rtol=1e-12, atol=1e-12)


def test_sparse_update_equals_dense_gated_delta_rule():
    # S_t = S_{t-1} D_t (I - beta k k^T) + beta v k^T, y_t = S_t r  (S = M^T, d_v x N),
    # k = write weights scattered on the written slots, D_t = I except alpha on them.
    st = _tiny_stream(7, T=30, dims=(32, 32), d_sub=8, d_v=64, W=8, R=8)
    M, res = _run(st, st["gates"])
    N = 1024
    S = st["M"].T.copy()
    I = np.eye(N)
    for t in range(30):
        k = np.zeros(N)
        k[res["idx_w"][t]] = res["wt_w"][t]
        D = np.eye(N)
        D[res["idx_w"][t], res["idx_w"][t]] = st["gates"][t, 0]
        beta = st["gates"][t, 1]
        S = S @ D @ (I - beta * np.outer(k, k)) + beta * np.outer(st["k_val"][t], k)
        r = np.zeros(N)
        r[res["idx_r"][t]] = res["wt_r"][t]
        np.testing.assert_allclose(res["y"][t], S @ r, rtol=0, atol=1e-12)
    np.testing.assert_allclose(M, S.T, rtol=0, atol=1e-12)


def test_read_sees_the_same_tokens_write():
    # q_r = q_w and R = W = 1 with beta = 1: the read returns exactly the written value.
    st = _tiny_stream(8, W=1, R=1)
    st["q_r"] = st["q_w"]
    st["k_val"] = oracle.round_to(st["k_val"], "f32")
    st["M"] = oracle.round_to(st["M"], "f32")
    gates = np.tile([0.7, 1.0], (12, 1))
    _, res = _run(st, gates, bank_dtype="f32")
    np.testing.assert_array_equal(res["y"], st["k_val"])


# --------------------------------------------------------------------------- op level

def test_chunk_size_has_no_effect_and_decode_equals_write_read():
    cfg = sdm_inputs.CONFIGS["tiny"].replace(T=6)
    d = sdm_inputs.make_inputs(cfg)
    kw = dict(factor_dims=cfg.factor_dims, W=cfg.W, R=cfg.R)
    a = oracle.sdm_write_read(d["q_w"], d["q_r"], d["k_val"], d["gates"], d["subkeys"],
                              d["bank_init"], chunk_size=1, **kw)
    b = oracle.sdm_write_read(d["q_w"], d["q_r"], d["k_val"], d["gates"], d["subkeys"],
                              d["bank_init"], chunk_size=64, **kw)
    np.testing.assert_array_equal(a[(0, 0)]["y"], b[(0, 0)]["y"])
    np.testing.assert_array_equal(a[(0, 0)]["bank"], b[(0, 0)]["bank"])
    # the same six tokens as six decode steps, copying and donating
    bank = d["bank_init"].double().numpy()[None].copy()
    bank_keep = bank.copy()
    bank_don = bank.copy()
    for t in range(6):
        args = (d["q_w"][:, t], d["q_r"][:, t], d["k_val"][:, t], d["gates"][:, t], d["subkeys"])
        y_c, new = oracle.sdm_decode_step(*args, bank_keep, donate=False, **kw)
        assert new is not bank_keep
        bank_keep = new
        y_d, same = oracle.sdm_decode_step(*args, bank_don, donate=True, **kw)
        assert same is bank_don
        np.testing.assert_array_equal(y_c, y_d)
        np.testing.assert_array_equal(y_c[0, 0], a[(0, 0)]["y"][t])
    np.testing.assert_array_equal(bank_keep, bank_don)
    np.testing.assert_array_equal(bank_keep[0, 0], a[(0, 0)]["bank"])
    np.testing.assert_array_equal(bank, d["bank_init"].double().numpy()[None])  # copy left it


def test_bf16_bank_rows_are_rounded_after_every_token():
    cfg = sdm_inputs.CONFIGS["tiny"].replace(T=8, bank_dtype="bf16", act_dtype="bf16")
    d = sdm_inputs.make_inputs(cfg)
    out = oracle.sdm_write_read(d["q_w"], d["q_r"], d["k_val"], d["gates"], d["subkeys"],
                                d["bank_init"], factor_dims=cfg.factor_dims, W=cfg.W, R=cfg.R,
                                act_dtype="bf16", bank_dtype="bf16")
    M = out[(0, 0)]["bank"]
    np.testing.assert_array_equal(oracle.round_to_bf16(M), M)
    y = out[(0, 0)]["y"]
    np.testing.assert_array_equal(oracle.round_to_bf16(y), y)
