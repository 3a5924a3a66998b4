"""moe_permute_static: the permutation for callers that cannot allocate device scratch memory
(for example code that runs after its engine has reserved all device memory, or a plugin that
only receives its input and output buffers). Its scratch lives in a fixed array inside the
library, so the caller passes no workspace. These tests compare it, through the C ABI, with
moe_permute on the same routing, on consecutive calls that reuse the array."""
import ctypes

import numpy as np
import pytest
import torch

import moe_inputs

pytestmark = pytest.mark.gpu


def _lib():
    from fine_grained_moe_softmax_b300 import binding as B
    lib = B.lib()
    fn = lib.moe_permute_static
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(B.MoEConfig)] + [ctypes.c_void_p] * 7
    return B, fn


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _routed(B, shape, T, seed):
    """topk_idx and counts from moe_route on seeded tokens."""
    cfg = B.MoEConfig.from_shape(shape, T=T)
    inputs = moe_inputs.make_inputs(shape, T=T, seed=seed)
    dev = "cuda"
    ws = torch.empty(B.moe_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    idx = torch.empty(T, shape.top_k, dtype=torch.int32, device=dev)
    gate = torch.empty(T, shape.top_k, dtype=torch.float32, device=dev)
    counts = torch.empty(shape.n_routed, dtype=torch.int32, device=dev)
    psum = torch.empty(shape.n_routed, dtype=torch.float32, device=dev)
    bias = None if inputs["bias"] is None else inputs["bias"].to(dev)
    B.moe_route(cfg, inputs["u"].to(dev), inputs["centroids"].to(dev), bias, idx, gate, counts,
                psum, ws)
    return cfg, ws, idx, counts


def _run_both(B, fn, cfg, ws, idx, counts):
    T, K, N = cfg.T, cfg.top_k, cfg.n_routed
    dev = "cuda"
    out = {}
    for name in ("ref", "static"):
        off = torch.full((N + 1,), -7, dtype=torch.int32, device=dev)
        pt = torch.full((T * K,), -7, dtype=torch.int32, device=dev)
        ps = torch.full((T * K,), -7, dtype=torch.int32, device=dev)
        status = torch.full((1,), -9, dtype=torch.int32, device=dev)
        if name == "ref":
            B.moe_permute(cfg, idx, counts, off, pt, ps, ws)
        else:
            rc = fn(ctypes.byref(cfg), _p(idx), _p(counts), _p(off), _p(pt), _p(ps), _p(status),
                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
            assert rc == 0, B.status_string(rc)
        torch.cuda.synchronize()
        out[name] = (off.cpu(), pt.cpu(), ps.cpu(), status.cpu())
    out["ws_status"] = B.moe_device_status(ws)   # moe_permute's own status word
    return out


@pytest.mark.parametrize("name,T", [("16b_bf16", 1000), ("145b_zipf_bf16", 700),
                                    ("tiny_f32", 256)])
def test_static_matches_workspace_version_on_consecutive_calls(name, T):
    B, fn = _lib()
    shape = moe_inputs.CONFIGS[name]
    for seed in (1, 2):   # the second call reuses the array the first one left behind
        cfg, ws, idx, counts = _routed(B, shape, T, seed)
        out = _run_both(B, fn, cfg, ws, idx, counts)
        for a, b in zip(out["ref"][:3], out["static"][:3]):
            assert torch.equal(a, b)
        assert out["ws_status"] == 0
        assert int(out["static"][3][0]) == 0


def test_static_reports_corrupt_counts_and_rejects_oversized():
    B, fn = _lib()
    shape = moe_inputs.CONFIGS["2b_bf16"]
    cfg, ws, idx, counts = _routed(B, shape, 300, 3)
    bad = counts.clone()
    bad[0] += 1
    out = _run_both(B, fn, cfg, ws, idx, bad)
    assert out["ws_status"] == -6          # both versions flag the inconsistent counts
    assert int(out["static"][3][0]) == -6
    for a, b in zip(out["ref"][:3], out["static"][:3]):
        assert torch.equal(a, b)
    big = B.MoEConfig.from_shape(shape, T=128 * 2100)   # 2100 tiles x 63 experts > the limit
    assert fn(ctypes.byref(big), _p(idx), _p(counts), _p(idx), _p(idx), _p(idx), None,
              None) == -2


def test_static_at_its_size_limit():
    """ceil(T / 128) * N' exactly at the documented limit of 131072 table entries (8192 tiles of
    128 tokens, N' = 16) reaches the far end of both tables in the fixed array; the result must
    equal moe_permute's and the oracle's counting sort. One token more must be refused."""
    import oracle
    from oracle import OracleCfg
    B, fn = _lib()
    shape = moe_inputs.MoEShape("limit", T=128 * 8192, d=64, n_shared=0, n_routed=16, inter=16,
                                top_k=2, n_groups=1, dtype="bf16", seed=0)
    T, K, N = shape.T, shape.top_k, shape.n_routed
    g = torch.Generator().manual_seed(77)
    first = torch.randint(0, N, (T,), generator=g)
    second = (first + torch.randint(1, N, (T,), generator=g)) % N
    idx = torch.stack([first, second], 1).to(torch.int32)
    counts = torch.bincount(idx.flatten().long(), minlength=N).to(torch.int32)
    cfg = B.MoEConfig.from_shape(shape)
    dev = "cuda"
    ws = torch.empty(B.moe_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    out = _run_both(B, fn, cfg, ws, idx.to(dev), counts.to(dev))
    for a, b in zip(out["ref"][:3], out["static"][:3]):
        assert torch.equal(a, b)
    assert out["ws_status"] == 0 and int(out["static"][3][0]) == 0
    want = oracle.permute(OracleCfg.from_shape(shape), idx.numpy())
    off, pt, ps = (t.numpy() for t in out["static"][:3])
    assert np.array_equal(off, want["offsets"])
    assert np.array_equal(pt, want["perm_token"])
    assert np.array_equal(ps, want["perm_slot"])
    over = B.MoEConfig.from_shape(shape, T=T + 1)   # 8193 tiles x 16 experts
    d_idx = idx.to(dev)
    assert fn(ctypes.byref(over), _p(d_idx), _p(d_idx), _p(d_idx), _p(d_idx), _p(d_idx), None,
              None) == -2
