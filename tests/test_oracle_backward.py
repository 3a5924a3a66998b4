"""Pins of the oracle's backward pass by central finite differences of the oracle's forward.

The objective is Lambda = sum_t dh_t . h_t + L_ExpBal + L_DevBal, with the expert selection and
the selection counts held at their unperturbed values ("DeepSeekMoE 论文解读" §方法细节: f_i is a
selection frequency, P_i a mean affinity; the loss gradient flows through P). Every check below
evaluates only the forward (h, the affinity sums, the balance statistics), so it is independent
of the backward's own formulas."""
import math

import numpy as np
import pytest

import oracle
from oracle import OracleCfg


def _inputs(rng, T, d, Ks, N, I):
    E = Ks + N
    f = np.float32
    return {"u": rng.standard_normal((T, d)).astype(f),
            "centroids": (rng.standard_normal((N, d)) * 1.5 / math.sqrt(d)).astype(f),
            "bias": (rng.standard_normal(N) * 0.5).astype(f),
            "w_gate": (rng.standard_normal((E, I, d)) / math.sqrt(d)).astype(f),
            "w_up": (rng.standard_normal((E, I, d)) / math.sqrt(d)).astype(f),
            "w_down": (rng.standard_normal((E, d, I)) / math.sqrt(I)).astype(f)}


def _objective(cfg, inp, dh, counts):
    fw = oracle.forward_tokens(cfg, inp, np.arange(cfg.T))
    r = oracle.route(cfg, inp["u"], inp["centroids"], inp["bias"])
    assert np.array_equal(r["counts"], counts), "a perturbation changed the routing"
    st = oracle.balance_stats(cfg, counts, r["psum"])
    return float(np.sum(dh * fw["h"]) + st["losses"].sum())


def _fd(cfg, inp, dh, counts, key, index, eps=2e-3):
    """Central difference of the objective along one fp32 input element, using the exactly
    representable perturbed values."""
    arr = inp[key]
    x0 = arr[index]
    xp, xm = np.float32(x0 + eps), np.float32(x0 - eps)
    arr[index] = xp
    fp = _objective(cfg, inp, dh, counts)
    arr[index] = xm
    fm = _objective(cfg, inp, dh, counts)
    arr[index] = x0
    return (fp - fm) / (float(xp) - float(xm))


CASES = [
    dict(renormalize=0, skip_top=0, drop_shared=0),
    dict(renormalize=1, skip_top=0, drop_shared=0),
    dict(renormalize=0, skip_top=1, drop_shared=1),
    dict(renormalize=1, skip_top=2, drop_shared=0),
]


@pytest.mark.parametrize("opts", CASES)
def test_backward_matches_finite_differences(oracle_lib, opts):
    T, d, Ks, N, I, K = 6, 8, 1, 6, 4, 2
    cfg = OracleCfg(T=T, d=d, n_shared=Ks, n_routed=N, inter=I, top_k=K, n_groups=2,
                    alpha1=0.3, alpha2=0.7, **opts)
    for seed in range(100):   # the first seeded input that routes far from any tie
        rng = np.random.default_rng(1000 * seed + 7 + 10 * opts["renormalize"] + opts["skip_top"])
        inp = _inputs(rng, T, d, Ks, N, I)
        r = oracle.route(cfg, inp["u"], inp["centroids"], inp["bias"])
        if r["margin"].min() > 5e-3:
            break
    assert r["margin"].min() > 5e-3
    counts = r["counts"]
    dh = rng.standard_normal((T, d))
    g = oracle.backward(cfg, inp, dh, counts)
    probes = [("u", (0, 0)), ("u", (3, 5)), ("u", (5, 7)),
              ("centroids", (0, 1)), ("centroids", (4, 6)), ("bias", (2,)), ("bias", (5,)),
              ("w_gate", (0, 1, 2)), ("w_gate", (3, 2, 7)), ("w_up", (0, 3, 0)),
              ("w_up", (4, 1, 4)), ("w_down", (0, 5, 3)), ("w_down", (2, 0, 1)),
              ("w_down", (6, 7, 2))]
    names = {"u": "du", "centroids": "d_centroids", "bias": "d_bias", "w_gate": "dw_gate",
             "w_up": "dw_up", "w_down": "dw_down"}
    for key, index in probes:
        fd = _fd(cfg, inp, dh, counts, key, index)
        an = g[names[key]][index]
        assert an == pytest.approx(fd, rel=2e-4, abs=2e-6), (key, index, an, fd)


def test_backward_is_affine_in_dh(oracle_lib):
    """The upstream part of every gradient is linear in dh; the balance-loss part does not
    depend on dh: g(2 dh) - g(dh) = g(dh) - g(0)."""
    rng = np.random.default_rng(3)
    T, d, Ks, N, I, K = 5, 8, 2, 5, 4, 2
    inp = _inputs(rng, T, d, Ks, N, I)
    cfg = OracleCfg(T=T, d=d, n_shared=Ks, n_routed=N, inter=I, top_k=K, n_groups=5,
                    alpha1=0.2, alpha2=0.1)
    dh = rng.standard_normal((T, d))
    g0, g1, g2 = (oracle.backward(cfg, inp, a * dh) for a in (0.0, 1.0, 2.0))
    for k in g0:
        np.testing.assert_allclose(g2[k] - g1[k], g1[k] - g0[k], rtol=1e-9, atol=1e-12)
    # with dh = 0 only the balance losses act: no expert weight receives a gradient
    for k in ("dw_gate", "dw_up", "dw_down"):
        assert np.all(g0[k] == 0)
    assert np.abs(g0["d_centroids"]).max() > 0


def test_du_of_a_token_needs_only_counts_and_T(oracle_lib):
    """du_t depends on the other tokens only through the selection counts (held fixed) and the
    1/T of the balance statistics. The balance part of the affinity gradient,
    (a1 f_j + a2 f'_g) / T with f proportional to count / T, scales as 1 / T^2. The rows of a
    batch's du are recovered from a sub-batch run with the batch's counts, once with dh and
    once with dh = 0, by rescaling the latter by (T_s / T)^2. The full-size GPU check of the
    backward rests on this."""
    rng = np.random.default_rng(9)
    T, d, Ks, N, I, K = 12, 8, 1, 6, 4, 2
    inp = _inputs(rng, T, d, Ks, N, I)
    cfg = OracleCfg(T=T, d=d, n_shared=Ks, n_routed=N, inter=I, top_k=K, n_groups=3,
                    alpha1=0.3, alpha2=0.6)
    dh = rng.standard_normal((T, d))
    counts = oracle.route(cfg, inp["u"], inp["centroids"], inp["bias"])["counts"]
    full = oracle.backward(cfg, inp, dh, counts)
    sample = np.array([0, 4, 11])
    sub = dict(inp)
    sub["u"] = inp["u"][sample]
    cs = OracleCfg(T=len(sample), d=d, n_shared=Ks, n_routed=N, inter=I, top_k=K, n_groups=3,
                   alpha1=0.3, alpha2=0.6)
    w1 = oracle.backward(cs, sub, dh[sample], counts)
    w0 = oracle.backward(cs, sub, np.zeros((len(sample), d)), counts)
    want = w1["du"] - (1.0 - (len(sample) / T) ** 2) * w0["du"]
    np.testing.assert_allclose(want, full["du"][sample], rtol=1e-10, atol=1e-12)
    assert np.abs(w0["du"]).max() > 0   # the balance part is present and rescaled
