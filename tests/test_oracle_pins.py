"""Pins for the CPU oracle: each test ties it to something other than itself.

Pins used: the hand-worked example under tests/golden (values derived by hand
from the definitions), closed forms (SiLU values, column norms, the FFN rate
the POP notes print), brute force on tiny inputs (pure-Python loops, pairwise
rank counting, subset enumeration), and invariants the method fixes (r = 0 is
the dense FFN, gamma = 0 is a static mask, |R| + k = keep, period 1 is per-step
POP, permutation equivariance, scaling of W2).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth


def _tiny_layer(seed, D, N, scale=1.0):
    Wg, W1, W2 = synth.ffn_weights(seed, D, N)
    Wg, W1, W2 = (synth.bf16_to_f64(w) * (scale / synth.WEIGHT_STD) for w in (Wg, W1, W2))
    return Wg, W1, W2


def _x(seed, T, D, step=None):
    sc = synth.dim_scales(seed, D)
    u = synth.prompt(seed, T, sc) if step is None else synth.decode_input(seed, step, T, sc)
    return synth.bf16_to_f64(u)


# ----------------------------------------------------------------- worked example

def test_worked_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "tiny_worked_example.json")))
    Wg, W1, W2 = (np.array(g[k], dtype=np.float64) for k in ("Wg", "W1", "W2"))
    X = np.array(g["prompt_x"], dtype=np.float64)
    pre = oracle.prefill(Wg, W1, W2, X, g["r"], g["gamma"])
    np.testing.assert_allclose(pre["Z"][0], g["z_prefill"], rtol=1e-15)
    np.testing.assert_allclose(oracle.column_norms(W2), g["n2"], rtol=1e-15)
    np.testing.assert_allclose(pre["I"], g["importance"], rtol=1e-15)
    c = pre["counts"]
    assert (c.n_P, c.n_R, c.n_C, c.keep, c.k) == tuple(g["counts"][k] for k in ("n_P", "n_R", "n_C", "keep", "k"))
    assert pre["R"].tolist() == g["R"] and pre["C"].tolist() == g["C"] and pre["P"].tolist() == g["P"]
    s = oracle.PopSession(Wg, W1, W2, pre["R"], pre["C"], c.k)
    y = s.step(np.array(g["decode_x"], dtype=np.float64))
    RC = np.concatenate([s.C, s.R])
    for pos, ch in enumerate(RC):
        assert s.last_z[0, pos] == pytest.approx(g["z_decode_RC"][str(ch)], rel=1e-15)
    np.testing.assert_allclose(s.last_scores, g["scores_C"], rtol=1e-15)
    assert s.C[s.S].tolist() == g["S_channels"]
    assert s.kept_channels().tolist() == g["kept_channels"]
    np.testing.assert_allclose(y, g["y_decode"], rtol=1e-14, atol=1e-15)


# ----------------------------------------------------------------- closed forms

def test_silu_closed_form():
    v = oracle.silu(np.array([0.0, 1.0, -1.0, 2.0, 40.0, -40.0]))
    assert v[0] == 0.0
    assert v[1] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    assert v[2] == pytest.approx(-1.0 / (1.0 + math.e), rel=1e-15)
    assert v[1] - v[2] == pytest.approx(1.0, rel=1e-15)        # SiLU(x) - SiLU(-x) = x
    assert v[4] == pytest.approx(40.0, rel=1e-15)               # -> identity for large x
    assert abs(v[5]) < 1e-15                                    # -> 0 for very negative x


def test_column_norms_orientation():
    # W2 is [D, D_FF]; the importance weight factor is the norm over D of column i.
    W2 = np.array([[3.0, 0.0, 1.0], [4.0, 2.0, 0.0]])
    np.testing.assert_array_equal(oracle.column_norms(W2), [5.0, 2.0, 1.0])


def test_importance_closed_form():
    # two tokens; channel norms over tokens: sqrt(3^2+4^2) = 5, sqrt(0+1) = 1, 0
    Z = np.array([[3.0, 0.0, 0.0], [4.0, -1.0, 0.0]])
    W2 = np.array([[1.0, 0.0, 7.0], [0.0, 2.0, 0.0]])
    ss, I = oracle.channel_importance(W2, Z)
    np.testing.assert_array_equal(ss, [25.0, 1.0, 0.0])
    np.testing.assert_array_equal(I, [5.0, 2.0, 0.0])


def test_ffn_rate_matches_pages(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "pages_numbers.json")))["ffn_rate_llama2_7b"]
    D, N = g["D"], g["D_FF"]
    rate = g["global_rate"] * (4 * D * D + 3 * D * N) / (3 * D * N)
    assert abs(rate - g["value"]) <= g["print_precision"]


def test_candidate_share_matches_pages(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "pages_numbers.json")))["candidate_share"]
    for N, r in [(11008, 0.299), (11008, 0.5), (28672, 0.5), (14336, 0.3), (1024, 0.3)]:
        c = oracle.region_counts(N, r, g["gamma"])
        assert abs(c.n_C / N - g["value"]) <= g["print_precision"]


def test_counts_equal_linear_quantiles():
    # On the five workload shapes, count-based cut-offs equal the sets that linear-interpolated
    # quantiles give on distinct scores (in general the two readings can differ by one channel
    # when (r +- gamma) * (N - 1) lands on an integer).
    rng = np.random.default_rng(1)
    for N, r, gamma in [(1024, 0.3, 0.1), (11008, 0.299, 0.1), (11008, 0.5, 0.1), (28672, 0.5, 0.1),
                        (14336, 0.3, 0.1)]:
        I = rng.permutation(N).astype(np.float64) + 0.5
        c = oracle.region_counts(N, r, gamma)
        lo = np.quantile(I, r - gamma, method="linear")
        hi = np.quantile(I, r + gamma, method="linear")
        assert int(np.sum(I <= lo)) == c.n_P
        assert int(np.sum(I >= hi)) == c.n_R
        assert c.n_R + c.k == c.keep == N - int(round(r * N))


def test_counts_edges():
    c = oracle.region_counts(100, 0.0, 0.1)
    assert (c.n_P, c.k, c.keep) == (0, c.n_C, 100)
    c = oracle.region_counts(100, 0.3, 0.0)
    assert c.n_C == 0 and c.k == 0 and c.n_R == c.keep == 70
    c = oracle.region_counts(100, 0.5, 0.5)
    assert c.n_P == 0 and c.n_R == 0 and c.n_C == 100 and c.k == 50
    c = oracle.region_counts(0, 0.3, 0.1)
    assert c.keep == 0 and c.n_C == 0
    with pytest.raises(ValueError):
        oracle.region_counts(10, 1.5, 0.1)


# ----------------------------------------------------------------- brute force

def test_ffn_activations_bruteforce():
    D, N, T = 5, 7, 3
    Wg, W1, W2 = _tiny_layer(3, D, N, scale=0.5)
    X = _x(3, T, D)
    Z = oracle.ffn_activations(Wg, W1, X)
    for t in range(T):
        for i in range(N):
            g = sum(Wg[i][d] * X[t][d] for d in range(D))
            u = sum(W1[i][d] * X[t][d] for d in range(D))
            assert Z[t, i] == pytest.approx(g / (1.0 + math.exp(-g)) * u, rel=1e-12, abs=1e-14)
    Y = oracle.dense_ffn(Wg, W1, W2, X)
    for t in range(T):
        for d in range(D):
            assert Y[t, d] == pytest.approx(sum(Z[t][i] * W2[d][i] for i in range(N)), rel=1e-12, abs=1e-14)


def _rank_least_important_first(I32):
    # rank = how many channels are less important: lower score, or equal score and higher index
    N = len(I32)
    return [sum(1 for j in range(N) if I32[j] < I32[i] or (I32[j] == I32[i] and j > i)) for i in range(N)]


def test_partition_pairwise_ranks():
    rng = np.random.default_rng(7)
    for N, r, gamma in [(40, 0.3, 0.1), (37, 0.5, 0.2), (64, 0.299, 0.1), (20, 0.0, 0.1), (20, 0.9, 0.3)]:
        I = rng.integers(0, 9, size=N).astype(np.float64) * 0.25  # many exact ties
        c = oracle.region_counts(N, r, gamma)
        R, C, P = oracle.partition(I, c)
        rank = _rank_least_important_first(np.asarray(I, dtype=np.float32).tolist())
        assert sorted(rank) == list(range(N))
        assert P.tolist() == [i for i in range(N) if rank[i] < c.n_P]
        assert R.tolist() == [i for i in range(N) if rank[i] >= N - c.n_R]
        assert C.tolist() == [i for i in range(N) if c.n_P <= rank[i] < N - c.n_R]
        # threshold semantics: R at or above every C, C at or above every P
        if R.size and C.size:
            assert I[R].min() >= I[C].max()
        if C.size and P.size:
            assert I[C].min() >= I[P].max()


def test_topk_subset_enumeration():
    rng = np.random.default_rng(11)
    for n in range(0, 11):
        for k in range(0, n + 1):
            a = rng.random(n)
            S = oracle.select_topk(a, k)
            best = max((sum(a[list(s)]) for s in itertools.combinations(range(n), k)), default=0.0)
            assert sum(a[S]) == pytest.approx(best, rel=1e-12)
            winners = [s for s in itertools.combinations(range(n), k) if abs(sum(a[list(s)]) - best) < 1e-12]
            assert len(winners) == 1 and list(winners[0]) == S.tolist()
    # ties: equal scores go to the lower position
    a = np.array([1.0, 2.0, 2.0, 2.0, 0.5])
    assert oracle.select_topk(a, 2).tolist() == [1, 2]
    assert oracle.select_topk(a, 4).tolist() == [0, 1, 2, 3]


def test_decode_mask_enumeration():
    # D <= 8, N <= 16: S must maximise the score mass over all masks R <= M <= R u C with |M| = keep.
    D, N = 6, 14
    Wg, W1, W2 = _tiny_layer(5, D, N, scale=0.7)
    pre = oracle.prefill(Wg, W1, W2, _x(5, 4, D), r=0.4, gamma=0.2)
    c = pre["counts"]
    s = oracle.PopSession(Wg, W1, W2, pre["R"], pre["C"], c.k)
    n2 = oracle.column_norms(W2)
    for t in range(3):
        x = _x(5, 2, D, step=t)
        y = s.step(x)
        # scores recomputed by brute force from the definition over C only
        a = []
        for ch in s.C:
            zb = []
            for b in range(x.shape[0]):
                g = sum(Wg[ch][d] * x[b][d] for d in range(D))
                u = sum(W1[ch][d] * x[b][d] for d in range(D))
                zb.append(abs(g / (1 + math.exp(-g)) * u))
            a.append(max(zb) * n2[ch])
        a = np.array(a)
        best = None
        for M in itertools.combinations(range(len(s.C)), c.k):
            v = a[list(M)].sum()
            if best is None or v > best[0] + 1e-12:
                best = (v, M)
        assert list(best[1]) == s.S.tolist()
        kept = s.kept_channels()
        assert len(kept) == c.keep and set(s.R.tolist()) <= set(kept.tolist())
        # y by loops over the kept channels
        for b in range(x.shape[0]):
            for d in range(D):
                ref = 0.0
                for ch in kept:
                    g = sum(Wg[ch][e] * x[b][e] for e in range(D))
                    u = sum(W1[ch][e] * x[b][e] for e in range(D))
                    ref += g / (1 + math.exp(-g)) * u * W2[d][ch]
                assert y[b, d] == pytest.approx(ref, rel=1e-11, abs=1e-13)


# ----------------------------------------------------------------- invariants

@pytest.mark.parametrize("B", [1, 3])
def test_rate_zero_is_dense(B):
    D, N = 16, 48
    Wg, W1, W2 = _tiny_layer(9, D, N)
    pre = oracle.prefill(Wg, W1, W2, _x(9, 8, D), r=0.0, gamma=0.1)
    c = pre["counts"]
    assert c.n_P == 0 and c.k == c.n_C
    s = oracle.PopSession(Wg, W1, W2, pre["R"], pre["C"], c.k)
    for t in range(3):
        x = _x(9, B, D, step=t)
        y = s.step(x)
        np.testing.assert_array_equal(y, oracle.dense_ffn(Wg, W1, W2, x))


def test_gamma_zero_is_static_mask():
    D, N = 16, 50
    Wg, W1, W2 = _tiny_layer(10, D, N)
    pre = oracle.prefill(Wg, W1, W2, _x(10, 8, D), r=0.3, gamma=0.0)
    c = pre["counts"]
    assert c.n_C == 0 and c.k == 0
    s = oracle.PopSession(Wg, W1, W2, pre["R"], pre["C"], c.k)
    top_keep = np.sort(np.lexsort((np.arange(N), -pre["I"].astype(np.float32)))[:c.keep])
    for t in range(4):
        s.step(_x(10, 2, D, step=t))
        assert s.kept_channels().tolist() == top_keep.tolist()


def test_keep_count_and_cover():
    D, N = 32, 200
    Wg, W1, W2 = _tiny_layer(12, D, N)
    pre = oracle.prefill(Wg, W1, W2, _x(12, 16, D), r=0.299, gamma=0.1)
    c = pre["counts"]
    allc = np.concatenate([pre["R"], pre["C"], pre["P"]])
    assert np.array_equal(np.sort(allc), np.arange(N))
    s = oracle.PopSession(Wg, W1, W2, pre["R"], pre["C"], c.k)
    for t in range(5):
        s.step(_x(12, 4, D, step=t))
        kept = s.kept_channels()
        assert len(kept) == c.n_R + c.k == c.keep
        assert not set(kept.tolist()) & set(pre["P"].tolist())


def test_full_reevaluation_variant():
    # gamma >= max(r, 1-r): R = P = empty and every step takes the top-keep over all channels.
    D, N = 12, 30
    Wg, W1, W2 = _tiny_layer(13, D, N)
    pre = oracle.prefill(Wg, W1, W2, _x(13, 4, D), r=0.4, gamma=0.6)
    c = pre["counts"]
    assert c.n_R == 0 and c.n_P == 0 and c.n_C == N and c.k == c.keep
    s = oracle.PopSession(Wg, W1, W2, pre["R"], pre["C"], c.k)
    n2 = oracle.column_norms(W2)
    for t in range(3):
        x = _x(13, 1, D, step=t)
        s.step(x)
        z = oracle.ffn_activations(Wg, W1, x)[0]
        score = np.abs(z) * n2
        ranked = sorted(range(N), key=lambda i: (-np.float32(score[i]), i))
        assert s.kept_channels().tolist() == sorted(ranked[:c.keep])


def test_period_one_is_per_step_and_memory_sums():
    D, N, P = 16, 60, 4
    Wg, W1, W2 = _tiny_layer(14, D, N)
    pre = oracle.prefill(Wg, W1, W2, _x(14, 8, D), r=0.5, gamma=0.1)
    c = pre["counts"]
    s1 = oracle.PopSession(Wg, W1, W2, pre["R"], pre["C"], c.k, period=1)
    sP = oracle.PopSession(Wg, W1, W2, pre["R"], pre["C"], c.k, period=P)
    history = []
    for t in range(10):
        x = _x(14, 3, D, step=t)
        y1 = s1.step(x)
        # per-step: selection = top-k of this step's scores
        assert s1.S.tolist() == oracle.select_topk(s1.last_scores, c.k).tolist()
        history.append(s1.last_scores.copy())
        sP.step(x)
        np.testing.assert_array_equal(sP.last_scores, s1.last_scores)
        if t % P == 0:
            window = history[max(0, t - P + 1):t + 1] if t else history[:1]
            mem = np.sum(window, axis=0)
            ranked = sorted(range(len(mem)), key=lambda i: (-np.float32(mem[i]), i))
            assert sP.S.tolist() == sorted(ranked[:c.k])
            held = sP.S.copy()
        else:
            assert sP.S.tolist() == held.tolist()
    # P = 1 session equals a session built with period 1 explicitly and fresh memory each step
    assert y1.shape == (3, D)


def test_permutation_equivariance():
    D, N = 16, 64
    Wg, W1, W2 = _tiny_layer(15, D, N)
    X = _x(15, 8, D)
    perm = np.random.default_rng(0).permutation(N)
    pre = oracle.prefill(Wg, W1, W2, X, r=0.3, gamma=0.1)
    preP = oracle.prefill(Wg[perm], W1[perm], W2[:, perm], X, r=0.3, gamma=0.1)
    inv = np.argsort(perm)
    for name in ("R", "C", "P"):
        assert np.sort(perm[preP[name]]).tolist() == pre[name].tolist()
    np.testing.assert_allclose(preP["Y"], pre["Y"], rtol=1e-12, atol=1e-14)
    s = oracle.PopSession(Wg, W1, W2, pre["R"], pre["C"], pre["counts"].k)
    sP = oracle.PopSession(Wg[perm], W1[perm], W2[:, perm], preP["R"], preP["C"], preP["counts"].k)
    for t in range(3):
        x = _x(15, 2, D, step=t)
        y = s.step(x)
        yP = sP.step(x)
        np.testing.assert_allclose(yP, y, rtol=1e-12, atol=1e-14)
        assert np.sort(perm[sP.kept_channels()]).tolist() == s.kept_channels().tolist()
    assert inv.shape == perm.shape


def test_w2_scaling():
    D, N = 16, 64
    Wg, W1, W2 = _tiny_layer(16, D, N)
    X = _x(16, 8, D)
    pre = oracle.prefill(Wg, W1, W2, X, r=0.3, gamma=0.1)
    pre2 = oracle.prefill(Wg, W1, 2.0 * W2, X, r=0.3, gamma=0.1)
    for name in ("R", "C", "P"):
        assert pre2[name].tolist() == pre[name].tolist()
    s = oracle.PopSession(Wg, W1, W2, pre["R"], pre["C"], pre["counts"].k)
    s2 = oracle.PopSession(Wg, W1, 2.0 * W2, pre["R"], pre["C"], pre["counts"].k)
    for t in range(3):
        x = _x(16, 2, D, step=t)
        np.testing.assert_allclose(s2.step(x), 2.0 * s.step(x), rtol=1e-14, atol=1e-16)
        assert s2.S.tolist() == s.S.tolist()


def test_moe_route():
    logits = np.array([[0.1, 2.0, 2.0, -1.0], [3.0, 1.0, 0.0, 1.0]])
    e, w = oracle.moe_route(logits)
    assert e.tolist() == [[1, 2], [0, 1]]
    np.testing.assert_allclose(w.sum(axis=1), 1.0)
    assert w[0, 0] == pytest.approx(0.5)
    assert w[1, 0] == pytest.approx(1.0 / (1.0 + math.exp(-2.0)))


# ----------------------------------------------------------------- MoE experts (reading 7)

def _moe_experts(E, D, N, same=False):
    return [_tiny_layer(40 if same else 40 + e, D, N) for e in range(E)]


def test_moe_route_against_pairwise_brute_force():
    rng = np.random.default_rng(7)
    L = np.round(rng.normal(size=(200, 6)), 1)  # one decimal: many exact ties
    e, w = oracle.moe_route(L)
    for t in range(L.shape[0]):
        # brute force over ordered pairs (a, b), a != b: a beats every other expert, b every other but a;
        # "beats" = larger logit, or equal logit and lower index
        def beats(i, j):
            return L[t, i] > L[t, j] or (L[t, i] == L[t, j] and i < j)
        pairs = [(a, b) for a in range(6) for b in range(6) if a != b
                 and all(beats(a, c) for c in range(6) if c != a)
                 and all(beats(b, c) for c in range(6) if c not in (a, b))]
        assert len(pairs) == 1 and tuple(e[t]) == pairs[0]
        d = L[t, e[t, 1]] - L[t, e[t, 0]]
        assert w[t, 0] == pytest.approx(1.0 / (1.0 + math.exp(d)), rel=1e-14)
        assert w[t, 1] == pytest.approx(math.exp(d) / (1.0 + math.exp(d)), rel=1e-14)


def test_moe_identical_dense_experts_are_the_dense_ffn():
    # r = 0 keeps every channel; identical experts and weights summing to one give the plain FFN
    D, N, E = 16, 40, 4
    ex = _moe_experts(E, D, N, same=True)
    X = _x(41, 12, D)
    L = np.random.default_rng(1).normal(size=(12, E))
    pre = oracle.moe_prefill(ex, X, L, r=0.0, gamma=0.1)
    Wg, W1, W2 = ex[0]
    np.testing.assert_allclose(pre["Y"], oracle.dense_ffn(Wg, W1, W2, X), rtol=1e-12, atol=1e-14)
    sess = oracle.MoeSession([oracle.PopSession(*ex[e], pre["parts"][e]["R"], pre["parts"][e]["C"],
                                                pre["parts"][e]["counts"].k) for e in range(E)])
    for t in range(3):
        x = _x(41, 5, D, step=t)
        y = sess.step(x, np.random.default_rng(10 + t).normal(size=(5, E)))
        np.testing.assert_allclose(y, oracle.dense_ffn(Wg, W1, W2, x), rtol=1e-12, atol=1e-14)


def test_moe_two_identical_experts_equal_one_pruned_layer():
    # E = 2 with top-2 routing sends every token to both experts, so each sees the whole prompt,
    # takes the single-layer partition and selection, and the weights sum to one
    D, N = 16, 64
    ex = _moe_experts(2, D, N, same=True)
    X = _x(42, 10, D)
    L = np.random.default_rng(2).normal(size=(10, 2))
    pre = oracle.moe_prefill(ex, X, L, r=0.3, gamma=0.1)
    single = oracle.prefill(*ex[0], X, 0.3, 0.1)
    for p in pre["parts"]:
        for name in ("R", "C", "P"):
            assert p[name].tolist() == single[name].tolist()
    np.testing.assert_allclose(pre["Y"], single["Y"], rtol=1e-12, atol=1e-14)
    moe = oracle.MoeSession([oracle.PopSession(*ex[e], single["R"], single["C"], single["counts"].k)
                             for e in range(2)])
    one = oracle.PopSession(*ex[0], single["R"], single["C"], single["counts"].k)
    for t in range(4):
        x = _x(42, 3, D, step=t)
        np.testing.assert_allclose(moe.step(x, np.random.default_rng(20 + t).normal(size=(3, 2))), one.step(x),
                                   rtol=1e-12, atol=1e-14)


def test_moe_idle_expert_split_is_the_index_tie_rule():
    # experts 2 and 3 never receive a token: s = 0, I = 0, so R is the n_R lowest indices, P the n_P
    # highest, and every decode step selects the k lowest candidate positions (all scores 0)
    D, N, E = 8, 30, 4
    ex = _moe_experts(E, D, N)
    X = _x(43, 9, D)
    L = np.full((9, E), -5.0)
    L[:, 0], L[:, 1] = 1.0, 0.5
    pre = oracle.moe_prefill(ex, X, L, r=0.3, gamma=0.1)
    c = oracle.region_counts(N, 0.3, 0.1)
    for e in (2, 3):
        p = pre["parts"][e]
        assert p["tokens"].size == 0
        assert p["R"].tolist() == list(range(c.n_R))
        assert p["P"].tolist() == list(range(N - c.n_P, N))
        assert p["C"].tolist() == list(range(c.n_R, N - c.n_P))
    sess = [oracle.PopSession(*ex[e], pre["parts"][e]["R"], pre["parts"][e]["C"], pre["parts"][e]["counts"].k)
            for e in range(E)]
    moe = oracle.MoeSession(sess)
    busy = [oracle.PopSession(*ex[e], pre["parts"][e]["R"], pre["parts"][e]["C"], pre["parts"][e]["counts"].k)
            for e in range(2)]
    for t in range(3):
        x = _x(43, 4, D, step=t)
        Lt = np.full((4, E), -5.0)
        Lt[:, 0], Lt[:, 1] = 2.0, 1.0
        y = moe.step(x, Lt)
        w0 = 1.0 / (1.0 + math.exp(-1.0))
        np.testing.assert_allclose(y, w0 * busy[0].step(x) + (1.0 - w0) * busy[1].step(x), rtol=1e-12, atol=1e-14)
        for e in (2, 3):
            assert sess[e].S.tolist() == list(range(c.k))
            assert sess[e].t == t + 1


def test_moe_token_permutation_permutes_outputs():
    D, N, E = 16, 48, 4
    ex = _moe_experts(E, D, N)
    X = _x(44, 14, D)
    L = np.random.default_rng(4).normal(size=(14, E))
    perm = np.random.default_rng(5).permutation(14)
    a = oracle.moe_prefill(ex, X, L, 0.3, 0.1)
    b = oracle.moe_prefill(ex, X[perm], L[perm], 0.3, 0.1)
    np.testing.assert_allclose(b["Y"], a["Y"][perm], rtol=1e-12, atol=1e-14)
    for pa, pb in zip(a["parts"], b["parts"]):
        for name in ("R", "C", "P"):
            assert pa[name].tolist() == pb[name].tolist()
    sa = oracle.MoeSession([oracle.PopSession(*ex[e], a["parts"][e]["R"], a["parts"][e]["C"],
                                              a["parts"][e]["counts"].k) for e in range(E)])
    sb = oracle.MoeSession([oracle.PopSession(*ex[e], a["parts"][e]["R"], a["parts"][e]["C"],
                                              a["parts"][e]["counts"].k) for e in range(E)])
    x = _x(44, 6, D, step=0)
    Lt = np.random.default_rng(6).normal(size=(6, E))
    q = np.random.default_rng(7).permutation(6)
    np.testing.assert_allclose(sb.step(x[q], Lt[q]), sa.step(x, Lt)[q], rtol=1e-12, atol=1e-14)


def test_moe_decode_expert_major_equals_stepping_the_layer():
    D, N, E = 16, 48, 4
    ex = _moe_experts(E, D, N)
    pre = oracle.moe_prefill(ex, _x(45, 12, D), np.random.default_rng(8).normal(size=(12, E)), 0.3, 0.1)
    k = pre["parts"][0]["counts"].k
    xs = [_x(45, 5, D, step=t) for t in range(4)]
    Ls = [np.random.default_rng(30 + t).normal(size=(5, E)) for t in range(4)]
    ys, per = oracle.moe_decode(lambda e: ex[e], pre["parts"], xs, Ls, k, period=2)
    sess = oracle.MoeSession([oracle.PopSession(*ex[e], pre["parts"][e]["R"], pre["parts"][e]["C"], k, period=2)
                              for e in range(E)])
    for t in range(4):
        np.testing.assert_array_equal(ys[t], sess.step(xs[t], Ls[t]))
        for e in range(E):
            s = sess.sessions[e]
            assert per[e][t]["S"].tolist() == s.C[s.S].tolist()


# ----------------------------------------------------------------- periodic skip variant (reading 8)

def _skip_pair(period, seed=50, D=12, N=60, B=3):
    Wg, W1, W2 = _tiny_layer(seed, D, N)
    pre = oracle.prefill(Wg, W1, W2, _x(seed, 10, D), r=0.3, gamma=0.1)
    k = pre["counts"].k
    full = oracle.PopSession(Wg, W1, W2, pre["R"], pre["C"], k, period=period)
    skip = oracle.PopSession(Wg, W1, W2, pre["R"], pre["C"], k, period=period, skip=True)
    xs = [_x(seed, B, D, step=t) for t in range(3 * period + 1)]
    return full, skip, xs


def test_skip_with_period_one_is_per_step_pop():
    full, skip, xs = _skip_pair(1)
    for x in xs:
        np.testing.assert_array_equal(skip.step(x), full.step(x))
        assert skip.S.tolist() == full.S.tolist()


def test_skip_steps_give_the_held_mask_output_and_memory_of_s_only():
    # until the first update after t = 0 both variants hold the same S, so y agrees; the skip
    # variant's memory is the full variant's per-step scores summed over those steps, on S only
    P = 4
    full, skip, xs = _skip_pair(P)
    acc = np.zeros(full.C.shape[0])
    for t in range(P):
        y_full, y_skip = full.step(xs[t]), skip.step(xs[t])
        np.testing.assert_allclose(y_skip, y_full, rtol=1e-12, atol=1e-14)
        if t > 0:
            acc += full.last_scores
    mask = np.zeros(full.C.shape[0], dtype=bool)
    mask[skip.S] = True
    np.testing.assert_allclose(skip.memory, np.where(mask, acc, 0.0), rtol=1e-12, atol=1e-15)
    # the update step selects from the memory plus this step's full scores, by the top-k rule
    skip.step(xs[P])
    full.step(xs[P])
    a = full.last_scores
    expect = oracle.select_topk(np.where(mask, acc, 0.0) + a, full.k)
    assert skip.S.tolist() == expect.tolist()
    np.testing.assert_array_equal(skip.memory, np.zeros_like(skip.memory))
