"""Pins of the fp64 CPU oracle against what the pages and the mathematics fix.

None of these checks re-types the oracle's formulas: each compares it with a closed form, a
value printed on the pages, an invariant, a special case, or brute force on tiny inputs. Page
citations are the page title and section (see each golden fixture for its own).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import moe_inputs
import oracle
from oracle import OracleCfg

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _zeros_inputs(T, d, Ks, N, I, dtype=np.float32):
    E = Ks + N
    return {"u": np.zeros((T, d), dtype), "centroids": np.zeros((N, d), dtype), "bias": None,
            "w_gate": np.zeros((E, I, d), dtype), "w_up": np.zeros((E, I, d), dtype),
            "w_down": np.zeros((E, d, I), dtype)}


def _rand_inputs(rng, T, d, Ks, N, I):
    E = Ks + N
    f = np.float32
    return {"u": rng.standard_normal((T, d)).astype(f),
            "centroids": (rng.standard_normal((N, d)) / math.sqrt(d)).astype(f),
            "bias": None,
            "w_gate": (rng.standard_normal((E, I, d)) / math.sqrt(d)).astype(f),
            "w_up": (rng.standard_normal((E, I, d)) / math.sqrt(d)).astype(f),
            "w_down": (rng.standard_normal((E, d, I)) / math.sqrt(I)).astype(f)}


# ------------------------------------------------------------------------- routing pins ----

def test_router_closed_form(oracle_lib):
    g = _golden("router_closed_form.json")
    cfg = OracleCfg(T=1, d=2, n_shared=0, n_routed=3, inter=16, top_k=2)
    e = np.array([[math.log(v), 0.0] for v in g["centroids_ln_of"]], np.float32)
    u = np.array(g["u"], np.float32)
    r = oracle.route(cfg, u, e, want_scores=True)
    tol = g["tolerance"]
    np.testing.assert_allclose(r["scores"][0], g["expect_scores"], atol=tol)
    assert list(r["topk_idx"][0]) == g["expect_topk_idx"]
    np.testing.assert_allclose(r["topk_gate"][0], g["expect_gate"], atol=tol)
    assert abs(r["margin"][0] - g["expect_margin"]) < tol
    cfg.renormalize = 1
    r = oracle.route(cfg, u, e)
    np.testing.assert_allclose(r["topk_gate"][0], g["expect_gate_renorm"], atol=tol)


def test_all_ties_pick_lowest_index(oracle_lib):
    """Zero centroids make every affinity exactly 1/N': ranks fall back to the index order."""
    T, d, N, K = 5, 8, 7, 3
    cfg = OracleCfg(T=T, d=d, n_shared=0, n_routed=N, inter=16, top_k=K)
    u = np.random.default_rng(0).standard_normal((T, d)).astype(np.float32)
    r = oracle.route(cfg, u, np.zeros((N, d), np.float32), want_scores=True)
    assert np.all(r["scores"] == 1.0 / N)
    assert np.all(r["topk_idx"] == np.arange(K))
    assert np.all(r["topk_gate"] == 1.0 / N)
    assert list(r["counts"]) == [T] * K + [0] * (N - K)
    np.testing.assert_allclose(r["psum"], T / N, rtol=1e-15)
    assert np.all(r["margin"] == 0.0)


def test_logit_bias_enters_softmax(oracle_lib):
    """With zero centroids and b_j = ln w_j, the affinity is w_j / sum(w)."""
    w = np.array([1.0, 2.0, 3.0, 4.0])
    cfg = OracleCfg(T=2, d=4, n_shared=0, n_routed=4, inter=16, top_k=2)
    u = np.ones((2, 4), np.float32)
    bias = np.log(w).astype(np.float32)
    r = oracle.route(cfg, u, np.zeros((4, 4), np.float32), bias, want_scores=True)
    np.testing.assert_allclose(r["scores"], np.tile(w / w.sum(), (2, 1)), atol=1e-7)
    assert np.all(r["topk_idx"] == [3, 2])


def test_softmax_invariants(oracle_lib):
    """s sums to 1, and log(s_i / s_j) equals the logit difference (u.e_i - u.e_j)."""
    rng = np.random.default_rng(1)
    T, d, N = 16, 32, 9
    inp = _rand_inputs(rng, T, d, 0, N, 16)
    cfg = OracleCfg(T=T, d=d, n_shared=0, n_routed=N, inter=16, top_k=2)
    r = oracle.route(cfg, inp["u"], inp["centroids"], want_scores=True)
    s = r["scores"]
    np.testing.assert_allclose(s.sum(axis=1), 1.0, atol=1e-14)
    z = inp["u"].astype(np.float64) @ inp["centroids"].astype(np.float64).T
    np.testing.assert_allclose(np.log(s[:, 1:] / s[:, :1]), z[:, 1:] - z[:, :1], atol=1e-12)


@pytest.mark.parametrize("N,K", [(6, 1), (6, 2), (7, 3), (8, 4), (9, 9), (15, 3)])
def test_topk_is_brute_force_argmax(oracle_lib, N, K):
    """The top-K' set is the unique subset of K' experts with the largest total affinity
    (checked over all C(N', K') subsets), listed by affinity descending."""
    rng = np.random.default_rng(N * 31 + K)
    T, d = 12, 16
    inp = _rand_inputs(rng, T, d, 0, N, 16)
    cfg = OracleCfg(T=T, d=d, n_shared=0, n_routed=N, inter=16, top_k=K)
    r = oracle.route(cfg, inp["u"], inp["centroids"], want_scores=True)
    for t in range(T):
        s = r["scores"][t]
        best = max(itertools.combinations(range(N), K), key=lambda S: sum(s[i] for i in S))
        assert set(r["topk_idx"][t]) == set(best)
        assert np.all(np.diff(s[r["topk_idx"][t]]) <= 0)
        np.testing.assert_allclose(r["topk_gate"][t], s[r["topk_idx"][t]], rtol=1e-15)
        srt = np.sort(s)[::-1]
        gaps = srt[:-1] - srt[1:]
        expect_margin = gaps[:K].min() if K < N else (gaps[:K - 1].min() if K > 1 else np.inf)
        assert r["margin"][t] == pytest.approx(expect_margin, rel=1e-12, abs=1e-300)


def test_renormalised_gates_sum_to_one(oracle_lib):
    rng = np.random.default_rng(2)
    inp = _rand_inputs(rng, 20, 16, 0, 10, 16)
    cfg = OracleCfg(T=20, d=16, n_shared=0, n_routed=10, inter=16, top_k=4, renormalize=1)
    r = oracle.route(cfg, inp["u"], inp["centroids"])
    np.testing.assert_allclose(r["topk_gate"].sum(axis=1), 1.0, atol=1e-14)
    cfg.top_k, cfg.renormalize = 10, 0   # K' = N': plain softmax gates already sum to 1
    r = oracle.route(cfg, inp["u"], inp["centroids"])
    np.testing.assert_allclose(r["topk_gate"].sum(axis=1), 1.0, atol=1e-14)


def test_counts_and_psum_totals(oracle_lib):
    sh = moe_inputs.CONFIGS["tiny_f32"]
    inp = moe_inputs.make_inputs(sh)
    cfg = OracleCfg.from_shape(sh)
    r = oracle.route(cfg, inp["u"], inp["centroids"], want_scores=True)
    assert r["counts"].sum() == sh.T * sh.top_k
    hist = np.bincount(r["topk_idx"].ravel(), minlength=sh.n_routed)
    assert np.array_equal(hist, r["counts"])
    assert r["psum"].sum() == pytest.approx(sh.T, rel=1e-13)
    np.testing.assert_allclose(r["psum"], r["scores"].sum(axis=0), rtol=1e-13)


# ------------------------------------------------------------------------ permutation pins ----

@pytest.mark.parametrize("T,N,K", [(1, 4, 1), (37, 5, 2), (256, 15, 3), (100, 9, 9)])
def test_permutation_invariants(oracle_lib, T, N, K):
    rng = np.random.default_rng(T + N + K)
    idx = np.stack([rng.permutation(N)[:K] for _ in range(T)]).astype(np.int32)
    cfg = OracleCfg(T=T, d=4, n_shared=0, n_routed=N, inter=16, top_k=K)
    p = oracle.permute(cfg, idx)
    off, pt, ps = p["offsets"], p["perm_token"], p["perm_slot"]
    assert off[0] == 0 and off[-1] == T * K and np.all(np.diff(off) >= 0)
    assert np.array_equal(np.diff(off), np.bincount(idx.ravel(), minlength=N))
    assert sorted(ps.tolist()) == list(range(T * K))          # a bijection onto the rows
    # row r holds assignment (t, k): its token is t, its expert's segment contains r
    for t in range(T):
        for k in range(K):
            r = ps[t * K + k]
            assert pt[r] == t
            assert off[idx[t, k]] <= r < off[idx[t, k] + 1]
    # brute force: rows are the assignments sorted by (expert, token)
    expect = sorted((idx[t, k], t) for t in range(T) for k in range(K))
    assert [t for _, t in expect] == pt.tolist()


def test_permutation_rejects_bad_ids(oracle_lib):
    cfg = OracleCfg(T=2, d=4, n_shared=0, n_routed=4, inter=16, top_k=1)
    with pytest.raises(ValueError):
        oracle.permute(cfg, np.array([[0], [4]], np.int32))


# --------------------------------------------------------------- expert FFN / layer pins ----

def test_ffn_one_hot_closed_form(oracle_lib):
    g = _golden("ffn_one_hot.json")
    d, I, Ks, N = g["d"], g["inter"], g["n_shared"], g["n_routed"]
    inp = _zeros_inputs(1, d, Ks, N, I)
    for key, name in (("w_gate_nonzero", "w_gate"), ("w_up_nonzero", "w_up"),
                      ("w_down_nonzero", "w_down")):
        for e, a, b, v in g[key]:
            inp[name][e, a, b] = v
    inp["u"][0] = [0.0, 1.0, math.log(3)]
    inp["centroids"][:] = np.float32(0.5)
    cfg = OracleCfg(T=1, d=d, n_shared=Ks, n_routed=N, inter=I, top_k=g["top_k"])
    out = oracle.forward_tokens(cfg, inp, [0])
    np.testing.assert_allclose(out["h"][0], g["expect_h"], atol=g["tolerance"])


@pytest.mark.parametrize("m", [2, 4])
def test_segmentation_identity(oracle_lib, m):
    """Splitting an expert's intermediate dimension into m segments that are all active with
    equal gates reproduces the unsplit expert (fine-grained segmentation keeps the function)."""
    rng = np.random.default_rng(10 + m)
    T, d, I = 6, 24, 8
    # split side: m shared experts of width I, and m routed experts of width I that are all
    # selected with equal affinity 1/m (zero centroids, K' = N' = m)
    split = _rand_inputs(rng, T, d, m, m, I)
    split["centroids"][:] = 0
    cfg_split = OracleCfg(T=T, d=d, n_shared=m, n_routed=m, inter=I, top_k=m)
    h_split = oracle.forward_tokens(cfg_split, split, range(T))["h"]
    # unsplit side: one shared expert of width m*I (segments stacked), one routed expert of
    # width m*I whose W_down carries the common gate 1/m (exact for m a power of two)
    def stack(lo):
        wg = np.concatenate([split["w_gate"][e] for e in range(lo, lo + m)], axis=0)
        wu = np.concatenate([split["w_up"][e] for e in range(lo, lo + m)], axis=0)
        wd = np.concatenate([split["w_down"][e] for e in range(lo, lo + m)], axis=1)
        return wg, wu, wd
    sg, su, sd = stack(0)
    rg, ru, rd = stack(m)
    whole = {"u": split["u"], "centroids": np.zeros((1, d), np.float32), "bias": None,
             "w_gate": np.stack([sg, rg]), "w_up": np.stack([su, ru]),
             "w_down": np.stack([sd, (rd / m).astype(np.float32)])}
    cfg_whole = OracleCfg(T=T, d=d, n_shared=1, n_routed=1, inter=m * I, top_k=1)
    h_whole = oracle.forward_tokens(cfg_whole, whole, range(T))["h"]
    np.testing.assert_allclose(h_split, h_whole, rtol=1e-12, atol=1e-12)


def test_identical_routed_experts_reduce_to_one_ffn(oracle_lib):
    """Coarse top-k routing without shared experts (K_s = 0, the GShard-style special case):
    with all routed experts identical and renormalised gates, h = u + FFN(u), where FFN(u) is
    what the same weights give as a shared expert."""
    rng = np.random.default_rng(3)
    T, d, I, N, K = 8, 16, 8, 6, 2
    base = _rand_inputs(rng, T, d, 0, 1, I)
    routed = {"u": base["u"], "centroids": (rng.standard_normal((N, d)) / 4).astype(np.float32),
              "bias": None, "w_gate": np.repeat(base["w_gate"], N, 0),
              "w_up": np.repeat(base["w_up"], N, 0), "w_down": np.repeat(base["w_down"], N, 0)}
    cfg_r = OracleCfg(T=T, d=d, n_shared=0, n_routed=N, inter=I, top_k=K, renormalize=1)
    h_r = oracle.forward_tokens(cfg_r, routed, range(T))["h"]
    shared = {"u": base["u"], "centroids": np.zeros((1, d), np.float32), "bias": None,
              "w_gate": np.concatenate([base["w_gate"], base["w_gate"]]),
              "w_up": np.concatenate([base["w_up"], base["w_up"]]),
              "w_down": np.concatenate([base["w_down"], np.zeros_like(base["w_down"])])}
    cfg_s = OracleCfg(T=T, d=d, n_shared=1, n_routed=1, inter=I, top_k=1)
    h_s = oracle.forward_tokens(cfg_s, shared, range(T))["h"]
    np.testing.assert_allclose(h_r, h_s, rtol=1e-12, atol=1e-12)
    # without renormalisation the routed part is scaled by the selected affinity mass
    cfg_r.renormalize = 0
    out = oracle.forward_tokens(cfg_r, routed, range(T))
    mass = out["topk_gate"].sum(axis=1, keepdims=True)
    u64 = base["u"].astype(np.float64)
    np.testing.assert_allclose(out["h"] - u64, mass * (h_s - u64), rtol=1e-11, atol=1e-12)


def test_dense_limit_is_softmax_mixture(oracle_lib):
    """K' = N' (every routed expert active) gives the dense softmax mixture. With
    W_down,j = c_j W_down,0 the FFNs are c_j FFN_0, so h - u = (sum_j s_j c_j) FFN_0."""
    rng = np.random.default_rng(4)
    T, d, I, N = 5, 16, 8, 5
    inp = _rand_inputs(rng, T, d, 0, N, I)
    c = np.array([1.0, -2.0, 0.5, 4.0, 0.25], np.float32)
    for j in range(N):
        inp["w_gate"][j] = inp["w_gate"][0]
        inp["w_up"][j] = inp["w_up"][0]
        inp["w_down"][j] = inp["w_down"][0] * c[j]
    cfg = OracleCfg(T=T, d=d, n_shared=0, n_routed=N, inter=I, top_k=N)
    out = oracle.forward_tokens(cfg, inp, range(T))
    s = oracle.route(cfg, inp["u"], inp["centroids"], want_scores=True)["scores"]
    one = OracleCfg(T=T, d=d, n_shared=0, n_routed=N, inter=I, top_k=1)
    for t in range(T):
        ffn0 = oracle.expert_ffn(one, inp, 0, inp["u"][t].astype(np.float64))
        np.testing.assert_allclose(out["h"][t] - inp["u"][t], (s[t] @ c) * ffn0,
                                   rtol=1e-11, atol=1e-12)


def test_shared_isolation(oracle_lib):
    """With every routed W_down zero, h = u + sum of the K_s shared experts, whatever routing
    does; K_s identical shared experts give K_s times one of them."""
    rng = np.random.default_rng(5)
    T, d, I, Ks, N = 4, 16, 8, 3, 4
    inp = _rand_inputs(rng, T, d, Ks, N, I)
    inp["w_down"][Ks:] = 0
    for e in range(1, Ks):
        inp["w_gate"][e], inp["w_up"][e], inp["w_down"][e] = (inp["w_gate"][0], inp["w_up"][0],
                                                              inp["w_down"][0])
    cfg = OracleCfg(T=T, d=d, n_shared=Ks, n_routed=N, inter=I, top_k=2)
    out = oracle.forward_tokens(cfg, inp, range(T), want_parts=True)
    for t in range(T):
        one = oracle.expert_ffn(cfg, inp, 0, inp["u"][t].astype(np.float64))
        np.testing.assert_allclose(out["h"][t] - inp["u"][t], Ks * one, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(out["shared"][t], Ks * one, rtol=1e-12, atol=1e-13)
        assert np.all(out["routed"][t] == 0)


def test_forward_matches_route(oracle_lib):
    """Per-token routing inside the forward agrees with the all-token router."""
    sh = moe_inputs.CONFIGS["tiny_f32"]
    inp = moe_inputs.make_inputs(sh)
    cfg = OracleCfg.from_shape(sh)
    r = oracle.route(cfg, inp["u"], inp["centroids"])
    fw = oracle.forward_tokens(cfg, inp, range(0, sh.T, 7))
    assert np.array_equal(fw["topk_idx"], r["topk_idx"][::7])
    assert np.array_equal(fw["topk_gate"], r["topk_gate"][::7])


# -------------------------------------------------------------------- balance-loss pins ----

def test_balance_hand_example(oracle_lib):
    g = _golden("balance_hand_example.json")
    cfg = OracleCfg(T=g["T"], d=4, n_shared=0, n_routed=g["n_routed"], inter=16,
                    top_k=g["top_k"], n_groups=g["n_groups"], alpha1=g["alpha1"],
                    alpha2=g["alpha2"])
    st = oracle.balance_stats(cfg, g["counts"], g["psum"])
    for k in ("f", "P", "fg", "Pg", "losses"):
        np.testing.assert_allclose(st[k], g["expect_" + k], rtol=1e-15, atol=1e-15)


@pytest.mark.parametrize("N,K,D", [(15, 3, 4), (64, 6, 8), (63, 7, 8), (128, 12, 8), (8, 8, 1)])
def test_balanced_routing_gives_alpha(oracle_lib, N, K, D):
    """Perfect balance (count_j = K'T/N', uniform affinity 1/N') gives f_j = 1, P_j = 1/N',
    L_ExpBal = alpha1 and L_DevBal = alpha2; the N'/K' factor makes f independent of N'."""
    T = N * 4
    cfg = OracleCfg(T=T, d=4, n_shared=0, n_routed=N, inter=16, top_k=K, n_groups=D,
                    alpha1=0.01, alpha2=0.05)
    st = oracle.balance_stats(cfg, np.full(N, K * T // N), np.full(N, T / N))
    np.testing.assert_allclose(st["f"], 1.0, rtol=1e-15)
    np.testing.assert_allclose(st["losses"], [0.01, 0.05], rtol=1e-13)


def test_f_sums_to_n_routed(oracle_lib):
    sh = moe_inputs.CONFIGS["tiny_f32"]
    inp = moe_inputs.make_inputs(sh)
    cfg = OracleCfg.from_shape(sh)
    r = oracle.route(cfg, inp["u"], inp["centroids"])
    st = oracle.balance_stats(cfg, r["counts"], r["psum"])
    assert st["f"].sum() == pytest.approx(sh.n_routed, rel=1e-14)
    assert st["P"].sum() == pytest.approx(1.0, rel=1e-13)
    assert st["Pg"].sum() == pytest.approx(1.0, rel=1e-13)


@pytest.mark.parametrize("N,D,sizes", [(15, 4, [4, 4, 4, 3]), (63, 8, [8] * 7 + [7]),
                                       (64, 8, [8] * 8), (10, 3, [4, 3, 3])])
def test_group_partition(oracle_lib, N, D, sizes):
    got = [oracle.group_range(N, D, g) for g in range(D)]
    assert [s for _, s in got] == sizes
    assert [f for f, _ in got] == list(np.concatenate([[0], np.cumsum(sizes)[:-1]]))


# -------------------------------------------------------------------- printed constants ----

def test_printed_constants():
    g = _golden("printed_constants.json")
    assert math.comb(16, 2) == g["comb_16_2"]
    assert abs(math.comb(64, 8) - g["comb_64_8_approx"]) / g["comb_64_8_approx"] < 0.01
    for key, name in (("layer_2b", "2b_bf16"), ("layer_16b", "16b_bf16")):
        sh = moe_inputs.CONFIGS[name]
        for f, v in g[key].items():
            assert getattr(sh, f) == v
    assert moe_inputs.CONFIGS["145b_zipf_bf16"].d == g["layer_145b"]["d"]


# ------------------------------------------------------------------- ablation options ----
# "DeepSeekMoE 论文解读" §专家特化深度分析: the analysis disables each token's top routed experts
# (routing falls to the next-ranked ones) and, separately, disables the shared experts.

def test_skip_top_closed_form(oracle_lib):
    """With s = (1, 2, 3)/6 (router fixture), disabling the top expert routes top-1 to expert 1
    with gate 1/3 (renormalised: 1); the decision depends on the gaps of ranks 1-2 and 2-3."""
    g = _golden("router_closed_form.json")
    e = np.array([[math.log(v), 0.0] for v in g["centroids_ln_of"]], np.float32)
    u = np.array(g["u"], np.float32)
    cfg = OracleCfg(T=1, d=2, n_shared=0, n_routed=3, inter=16, top_k=1, skip_top=1)
    r = oracle.route(cfg, u, e)
    assert list(r["topk_idx"][0]) == [1]
    assert abs(r["topk_gate"][0, 0] - 1 / 3) < 1e-7
    assert abs(r["margin"][0] - 1 / 6) < 1e-7
    cfg.renormalize = 1
    assert oracle.route(cfg, u, e)["topk_gate"][0, 0] == pytest.approx(1.0, abs=1e-12)
    with pytest.raises(ValueError):   # skip_top + K' beyond N'
        oracle.route(OracleCfg(T=1, d=2, n_shared=0, n_routed=3, inter=16, top_k=2, skip_top=2),
                     u, e)


@pytest.mark.parametrize("N,K,r", [(8, 2, 1), (9, 3, 2), (15, 3, 4), (6, 1, 5)])
def test_skip_top_is_next_ranked_set(oracle_lib, N, K, r):
    """The routed set with the r best experts disabled is top-(r+K') minus top-r (brute force over
    subsets for both), gates are the unchanged affinities, and ties fall to lower indices."""
    rng = np.random.default_rng(100 + N + K + r)
    T, d = 10, 16
    inp = _rand_inputs(rng, T, d, 0, N, 16)
    base = OracleCfg(T=T, d=d, n_shared=0, n_routed=N, inter=16, top_k=K)
    skip = OracleCfg(T=T, d=d, n_shared=0, n_routed=N, inter=16, top_k=K, skip_top=r)
    rs = oracle.route(skip, inp["u"], inp["centroids"], want_scores=True)
    for t in range(T):
        s = rs["scores"][t]
        def best(k):
            return set(max(itertools.combinations(range(N), k),
                           key=lambda S: sum(s[i] for i in S))) if k else set()
        assert set(rs["topk_idx"][t]) == best(r + K) - best(r)
        np.testing.assert_allclose(rs["topk_gate"][t], s[rs["topk_idx"][t]], rtol=1e-15)
    # all-equal affinities: ranks follow the index, so the chosen experts are r .. r+K'-1
    rz = oracle.route(skip, inp["u"], np.zeros((N, d), np.float32))
    assert np.all(rz["topk_idx"] == np.arange(r, r + K))
    # the softmax itself does not change
    rb = oracle.route(base, inp["u"], inp["centroids"], want_scores=True)
    np.testing.assert_array_equal(rb["psum"], rs["psum"])


def test_drop_shared_equals_zeroed_shared_experts(oracle_lib):
    """Disabling the shared experts gives the layer whose shared W_down is zero."""
    rng = np.random.default_rng(21)
    T, d, I, Ks, N = 6, 16, 8, 2, 5
    inp = _rand_inputs(rng, T, d, Ks, N, I)
    cfg = OracleCfg(T=T, d=d, n_shared=Ks, n_routed=N, inter=I, top_k=2, drop_shared=1)
    h_drop = oracle.forward_tokens(cfg, inp, range(T))["h"]
    zeroed = dict(inp)
    zeroed["w_down"] = inp["w_down"].copy()
    zeroed["w_down"][:Ks] = 0
    cfg0 = OracleCfg(T=T, d=d, n_shared=Ks, n_routed=N, inter=I, top_k=2)
    np.testing.assert_array_equal(h_drop, oracle.forward_tokens(cfg0, zeroed, range(T))["h"])


# ----------------------------------------------------------------- bf16 input path pins ----
# bf16 inputs reach the oracle as raw 16-bit patterns, widened to double inside it. These pins
# fix that widening against hand-written IEEE bf16 encodings and against fp32 inputs that hold
# the same values.

_BF16 = {1.0: 0x3F80, 1.5: 0x3FC0, -3.0: 0xC040, 0.5: 0x3F00, -0.5: 0xBF00, 2.0: 0x4000,
         0.0: 0x0000}


def test_bf16_bit_patterns_widen_to_their_values(oracle_lib):
    """u = (1.5, -3.0) and centroids e0 = (1, 0), e1 = (0, 1), e2 = (0.5, 0.5), all given as bf16
    bit patterns, make the logits (1.5, -3.0, -0.75): the log-ratios of the affinities are the
    logit differences 4.5 and 2.25, so a wrong half-word, shift or sign of the widening fails."""
    b = _BF16
    u = np.array([[b[1.5], b[-3.0]]], np.uint16)
    e = np.array([[b[1.0], b[0.0]], [b[0.0], b[1.0]], [b[0.5], b[0.5]]], np.uint16)
    cfg = OracleCfg(T=1, d=2, n_shared=0, n_routed=3, inter=16, top_k=2, dtype="bf16")
    r = oracle.route(cfg, u, e, want_scores=True)
    s = r["scores"][0]
    assert math.log(s[0] / s[1]) == pytest.approx(4.5, abs=1e-12)
    assert math.log(s[0] / s[2]) == pytest.approx(2.25, abs=1e-12)
    assert list(r["topk_idx"][0]) == [0, 2]


def test_bf16_expert_weights_widen_to_their_values(oracle_lib):
    """The one-hot layer of ffn_one_hot.json with every weight and token given as bf16 patterns of
    the same (bf16-exact) values gives the same h, bit for bit, as with fp32 inputs."""
    import torch
    g = _golden("ffn_one_hot.json")
    d, I, Ks, N = g["d"], g["inter"], g["n_shared"], g["n_routed"]
    inp = _zeros_inputs(1, d, Ks, N, I)
    for key, name in (("w_gate_nonzero", "w_gate"), ("w_up_nonzero", "w_up"),
                      ("w_down_nonzero", "w_down")):
        for e, a, bb, v in g[key]:
            inp[name][e, a, bb] = v
    inp["u"][0] = [0.0, 1.0, 1.5]
    inp["centroids"][:] = np.float32(0.5)
    exact = {k: torch.from_numpy(v).to(torch.bfloat16) for k, v in inp.items() if v is not None}
    for k, v in exact.items():   # every value is exact in bf16, so the fp32 twin holds the same
        assert np.array_equal(v.to(torch.float32).numpy(), inp[k])
    exact["bias"] = None
    f32 = {k: (None if v is None else v.to(torch.float32)) for k, v in exact.items()}
    cfg16 = OracleCfg(T=1, d=d, n_shared=Ks, n_routed=N, inter=I, top_k=g["top_k"], dtype="bf16")
    cfg32 = OracleCfg(T=1, d=d, n_shared=Ks, n_routed=N, inter=I, top_k=g["top_k"])
    h16 = oracle.forward_tokens(cfg16, exact, [0])["h"]
    h32 = oracle.forward_tokens(cfg32, f32, [0])["h"]
    np.testing.assert_array_equal(h16, h32)
    assert np.any(h16 != inp["u"])   # the experts contribute


def test_bf16_inputs_equal_fp32_inputs_of_the_same_values(oracle_lib):
    """Seeded bf16 tensors of the 2B-like layer (sub-sampled) against fp32 tensors holding the
    same values: routing, margins, sums and h agree exactly."""
    import torch
    sh = moe_inputs.CONFIGS["2b_bf16"].with_(T=12, d=64, n_routed=16, inter=32, top_k=4,
                                            n_groups=4)
    inp = moe_inputs.make_inputs(sh)
    f32 = {k: (None if v is None else v.to(torch.float32)) for k, v in inp.items()}
    f32["bias"] = inp["bias"]
    c16 = OracleCfg.from_shape(sh)
    c32 = OracleCfg.from_shape(sh.with_(dtype="f32"))
    r16 = oracle.route(c16, inp["u"], inp["centroids"], want_scores=True)
    r32 = oracle.route(c32, f32["u"], f32["centroids"], want_scores=True)
    for k in ("scores", "topk_idx", "topk_gate", "margin", "counts", "psum"):
        np.testing.assert_array_equal(r16[k], r32[k])
    toks = np.arange(sh.T)
    np.testing.assert_array_equal(oracle.forward_tokens(c16, inp, toks)["h"],
                                  oracle.forward_tokens(c32, f32, toks)["h"])
