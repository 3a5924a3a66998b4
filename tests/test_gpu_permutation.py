"""Bit-exact dispatch permutation at the token counts the benchmark and the full-size workloads use.

moe_route and moe_permute run through the C ABI on the workloads' full batches (up to 512 router
tiles, so the finalize kernel's scan crosses its 128-tile chunks and carries totals between them,
and a ragged last tile). Offsets, perm_token and perm_slot must equal, bit for bit, the oracle's
counting sort of the GPU's own expert indices, and the GPU's indices must equal the oracle's on
every token without a near-tie. moe_permute_static, the same permutation without a caller
workspace, must give the same bytes wherever its fixed scratch is large enough.
"""
import ctypes

import numpy as np
import pytest
import torch

import moe_inputs
import oracle
from oracle import OracleCfg
from parity import check_permutation, check_routing, to_np

pytestmark = pytest.mark.gpu

C = moe_inputs.CONFIGS


def _route_and_permute(shape, T):
    import fine_grained_moe_softmax_b300 as moe
    inputs = moe_inputs.make_inputs(shape, T=T)
    T = inputs["u"].shape[0]
    cfg = moe.MoEConfig.from_shape(shape, T=T)
    dev, i32, f32 = "cuda", torch.int32, torch.float32
    K, N = shape.top_k, shape.n_routed
    # a workspace for the router and permutation only: these stages use its status word and its
    # per-tile tables, which sit at the front of the full layer workspace
    ws = torch.empty(moe.moe_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    out = {"idx": torch.empty(T, K, dtype=i32, device=dev),
           "gate": torch.empty(T, K, dtype=f32, device=dev),
           "counts": torch.empty(N, dtype=i32, device=dev),
           "psum": torch.empty(N, dtype=f32, device=dev),
           "offsets": torch.full((N + 1,), -7, dtype=i32, device=dev),
           "perm_token": torch.full((T * K,), -7, dtype=i32, device=dev),
           "perm_slot": torch.full((T * K,), -7, dtype=i32, device=dev)}
    bias = None if inputs["bias"] is None else inputs["bias"].to(dev)
    moe.moe_route(cfg, inputs["u"].to(dev), inputs["centroids"].to(dev), bias, out["idx"],
                  out["gate"], out["counts"], out["psum"], ws)
    moe.moe_permute(cfg, out["idx"], out["counts"], out["offsets"], out["perm_token"],
                    out["perm_slot"], ws)
    torch.cuda.synchronize()
    assert moe.moe_device_status(ws) == 0
    return cfg, inputs, out, ws


def _permute_static(cfg, idx, counts):
    from fine_grained_moe_softmax_b300 import binding as B
    fn = B.lib().moe_permute_static
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(B.MoEConfig)] + [ctypes.c_void_p] * 7
    T, K, N = cfg.T, cfg.top_k, cfg.n_routed
    dev = "cuda"
    off = torch.full((N + 1,), -7, dtype=torch.int32, device=dev)
    pt = torch.full((T * K,), -7, dtype=torch.int32, device=dev)
    ps = torch.full((T * K,), -7, dtype=torch.int32, device=dev)
    status = torch.full((1,), -9, dtype=torch.int32, device=dev)
    rc = fn(ctypes.byref(cfg), *[ctypes.c_void_p(t.data_ptr()) for t in (idx, counts, off, pt, ps,
                                                                         status)],
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, B.status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return off, pt, ps


@pytest.mark.parametrize("name,T", [
    ("16b_bf16", None),             # 128 tiles: the benchmark's batch
    ("16b_bf16", 65459),            # 512 tiles, four scan chunks, a ragged last tile (51 tokens)
    ("145b_zipf_bf16", None),       # 64 tiles, 128 experts, K' = 12, skewed counts
    ("2b_bf16", None),              # 64 tiles, 63 experts, K' = 7
    ("2b_gshard_top2_bf16", None),  # 16 experts, K' = 2
    ("tiny_f32", 20000),            # fp32 router, 157 tiles
])
def test_full_size_permutation_is_bit_exact(name, T):
    shape = C[name]
    cfg, inputs, out, _ = _route_and_permute(shape, T)
    ocfg = OracleCfg.from_shape(shape, T=cfg.T)
    ref = oracle.route(ocfg, inputs["u"], inputs["centroids"], inputs["bias"])
    idx = to_np(out["idx"])
    check_routing(ocfg, ref, idx, to_np(out["gate"]), to_np(out["counts"]))
    np.testing.assert_allclose(to_np(out["psum"]), ref["psum"], rtol=2e-4, atol=1e-5)
    off, pt, ps = to_np(out["offsets"]), to_np(out["perm_token"]), to_np(out["perm_slot"])
    check_permutation(ocfg, idx, off, pt, ps)
    # the static-scratch version on the same routing
    s_off, s_pt, s_ps = _permute_static(cfg, out["idx"], out["counts"])
    assert torch.equal(s_off, out["offsets"])
    assert torch.equal(s_pt, out["perm_token"])
    assert torch.equal(s_ps, out["perm_slot"])


def test_permutation_of_adversarial_routing_at_full_size():
    """Routing that no seeded router output produces: at T = 16384 x 4 every token picks experts
    from a skewed table (one expert takes most tokens, several take none), crossing the scan's
    chunk boundaries with very uneven per-tile counts."""
    import fine_grained_moe_softmax_b300 as moe
    shape = C["16b_bf16"]
    T, K, N = 65536, shape.top_k, shape.n_routed
    g = torch.Generator().manual_seed(123)
    w = torch.zeros(N)
    w[:8] = torch.tensor([64.0, 16, 8, 4, 2, 1, 1, 1])
    w[40] = 32.0
    w[63] = 0.5
    idx = torch.multinomial(w.expand(T, N), K, replacement=False, generator=g).to(torch.int32)
    counts = torch.bincount(idx.flatten().long(), minlength=N).to(torch.int32)
    cfg = moe.MoEConfig.from_shape(shape, T=T)
    dev = "cuda"
    ws = torch.empty(moe.moe_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    off = torch.empty(N + 1, dtype=torch.int32, device=dev)
    pt = torch.empty(T * K, dtype=torch.int32, device=dev)
    ps = torch.empty(T * K, dtype=torch.int32, device=dev)
    idx_d, counts_d = idx.to(dev), counts.to(dev)
    moe.moe_permute(cfg, idx_d, counts_d, off, pt, ps, ws)
    torch.cuda.synchronize()
    assert moe.moe_device_status(ws) == 0
    ocfg = OracleCfg.from_shape(shape, T=T)
    check_permutation(ocfg, idx.numpy(), to_np(off), to_np(pt), to_np(ps))
    s_off, s_pt, s_ps = _permute_static(cfg, idx_d, counts_d)
    assert torch.equal(s_off, off) and torch.equal(s_pt, pt) and torch.equal(s_ps, ps)
