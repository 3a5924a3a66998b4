"""Helpers of the GPU parity tests: run the CUDA layer through the C ABI, run the oracle on the
same bytes, and compare what must be identical (routing on tokens without a near-tie, counts and
the permutation) and what must agree within the floating-point tolerance."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle import OracleCfg

# Tokens whose oracle affinity gap between neighbouring ranks 1..K'+1 is below this are near-ties:
# their selection is decided by rounding, so they are excluded from the exact routing check.
NEAR_TIE = 1e-6
# rel-L2 tolerances of h: fp32 layers / bf16 layers.
TOL = {"f32": 1e-4, "bf16": 2e-2}
# The same bound per token (on h and on h - u of every compared token), so that an error confined
# to a few tokens or one expert cannot hide inside the aggregate.
TOL_TOKEN = {"f32": 1e-3, "bf16": 5e-2}


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.to(torch.float32)
    return t.numpy()


def run_layer(shape, inputs, T=None, stream=None):
    """moe_layer_forward on cuda:0; returns the layer object (outputs on the device)."""
    from fine_grained_moe_softmax_b300 import MoEConfig, MoELayer
    cfg = MoEConfig.from_shape(shape, T=T)
    layer = MoELayer(cfg, inputs["centroids"], inputs["w_gate"], inputs["w_up"], inputs["w_down"],
                     inputs.get("bias"))
    u = inputs["u"].to("cuda")
    layer.forward(u, stream=stream)
    torch.cuda.synchronize()
    return layer, u


def check_routing(cfg: OracleCfg, ref: dict, idx_gpu: np.ndarray, gate_gpu: np.ndarray,
                  counts_gpu: np.ndarray, gate_atol: float = 2e-5):
    """Exact top-k on tokens without a near-tie; gates within gate_atol; counts == histogram of
    the GPU's own indices. Returns the boolean mask of compared (non-near-tie) tokens."""
    ok = ref["margin"] >= NEAR_TIE
    assert ok.mean() > 0.99, f"too many near-ties: {(~ok).sum()}"
    bad = np.nonzero(ok & np.any(idx_gpu != ref["topk_idx"], axis=1))[0]
    assert bad.size == 0, (f"{bad.size} tokens route differently, first {bad[:5]}: "
                           f"gpu {idx_gpu[bad[:1]]} oracle {ref['topk_idx'][bad[:1]]}")
    err = np.abs(gate_gpu[ok] - ref["topk_gate"][ok]).max() if ok.any() else 0.0
    assert err <= gate_atol, f"gate max abs error {err}"
    hist = np.bincount(idx_gpu.ravel(), minlength=cfg.n_routed)
    assert np.array_equal(hist, counts_gpu)
    return ok


def check_permutation(cfg: OracleCfg, idx_gpu, offsets, perm_token, perm_slot):
    """Bit-exact against the oracle's counting sort of the GPU's own indices."""
    ref = oracle.permute(cfg, idx_gpu)
    assert np.array_equal(ref["offsets"], offsets)
    assert np.array_equal(ref["perm_token"], perm_token)
    assert np.array_equal(ref["perm_slot"], perm_slot)


def per_token_rel_l2(got, want) -> np.ndarray:
    """rel-L2 of each row of got against the same row of want."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    den = np.linalg.norm(want, axis=1)
    return np.linalg.norm(got - want, axis=1) / np.where(den > 0, den, 1.0)
