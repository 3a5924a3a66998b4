"""The C-ABI library loads and exports every function of include/moe_b300.h; host-side argument
validation and size queries behave as documented. No compute call is made (no GPU needed)."""
import ctypes
import subprocess

import pytest

import moe_inputs

B = pytest.importorskip("fine_grained_moe_softmax_b300.binding")

from fine_grained_moe_softmax_b300 import build as build_mod  # noqa: E402

EXPECTED = {"moe_workspace_bytes", "moe_packed_weight_bytes", "moe_pack_weights", "moe_route",
            "moe_permute", "moe_expert_ffn", "moe_combine", "moe_balance_stats",
            "moe_layer_forward", "moe_device_status", "moe_status_string", "moe_launch_count",
            "moe_profile_enable", "moe_profile_read", "moe_profile_read_gate_up",
            "moe_selftest_bounded_wait", "moe_layer_routing"}


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.lib()


def test_header_declares_the_abi():
    assert EXPECTED <= set(B.header_functions())


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [f for f in B.header_functions() if f not in exported]
    assert not missing, missing
    for f in B.header_functions():
        assert getattr(lib, f) is not None


def test_status_strings(lib):
    assert B.status_string(0) == "MOE_OK"
    for code, name in [(-1, "INVALID_ARG"), (-2, "UNSUPPORTED"), (-3, "WORKSPACE"), (-4, "CUDA"),
                       (-5, "TIMEOUT"), (-6, "CORRUPT_INPUT")]:
        assert name in B.status_string(code)


@pytest.mark.parametrize("name", sorted(moe_inputs.CONFIGS))
def test_sizes(lib, name):
    sh = moe_inputs.CONFIGS[name]
    cfg = B.MoEConfig.from_shape(sh)
    es = 4 if sh.dtype == "f32" else 2
    assert B.moe_packed_weight_bytes(cfg) == 3 * sh.n_experts * sh.inter * sh.d * es
    ws = B.moe_workspace_bytes(cfg)
    TK = sh.T * sh.top_k
    # at least the permuted token rows, routed activations/outputs and the shared intermediates
    assert ws >= es * (TK * sh.d * 2 + TK * sh.inter + sh.T * sh.n_shared * sh.inter + sh.T * sh.d)
    assert ws % 256 == 0


def _cfg(**kw):
    base = dict(T=16, d=128, n_shared=1, n_routed=8, inter=32, top_k=2, renormalize=0,
                n_groups=2, alpha1=0.01, alpha2=0.05, dtype=B.MOE_DTYPE_BF16)
    base.update(kw)
    return B.MoEConfig(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(top_k=9), -1), (dict(top_k=0), -1), (dict(T=-1), -1), (dict(n_groups=9), -1),
    (dict(n_groups=0), -1), (dict(renormalize=2), -1), (dict(dtype=7), -1),
    (dict(n_routed=0), -1), (dict(d=96), -2), (dict(inter=24), -2),
    (dict(n_routed=300, n_groups=2), -2), (dict(n_routed=64, top_k=17), -2),
    (dict(skip_top=-1), -1), (dict(skip_top=7), -1), (dict(drop_shared=2), -1),
    (dict(n_routed=64, top_k=8, skip_top=9), -2),
])
def test_config_validation(lib, kw, code):
    cfg = _cfg(**kw)
    assert lib.moe_workspace_bytes(ctypes.byref(cfg)) == 0
    rc = lib.moe_route(ctypes.byref(cfg), None, None, None, None, None, None, None, None, 0, None)
    assert rc == code


def test_null_and_workspace_errors(lib):
    cfg = _cfg()
    P = ctypes.c_void_p
    fake = P(1 << 20)   # never dereferenced: validation fails first
    # missing tensors
    assert lib.moe_route(ctypes.byref(cfg), None, fake, None, fake, fake, fake, fake, fake,
                         1 << 30, None) == -1
    # workspace too small / misaligned
    small = lib.moe_workspace_bytes(ctypes.byref(cfg)) - 1
    assert lib.moe_route(ctypes.byref(cfg), fake, fake, None, fake, fake, fake, fake, fake,
                         small, None) == -3
    assert lib.moe_route(ctypes.byref(cfg), fake, fake, None, fake, fake, fake, fake,
                         P((1 << 20) + 16), 1 << 30, None) == -3
    # misaligned tensor
    assert lib.moe_layer_forward(ctypes.byref(cfg), P((1 << 20) + 2), fake, None, fake, fake, fake,
                                 fake, fake, fake, fake, fake, fake, 1 << 30, None) == -1
    assert lib.moe_balance_stats(ctypes.byref(cfg), None, fake, fake, fake, fake, None) == -1
    assert lib.moe_pack_weights(ctypes.byref(cfg), fake, None, fake, fake, None) == -1
    assert lib.moe_device_status(None, None) == -1
    assert lib.moe_profile_enable(1, 0) == -1
    assert lib.moe_selftest_bounded_wait(None, 256, 1000, None) == -3
    assert lib.moe_selftest_bounded_wait(P((1 << 20) + 8), 256, 1000, None) == -3


def test_profile_read_without_calls(lib):
    assert lib.moe_profile_enable(0, 0) == 0
    ms = (ctypes.c_float * B.N_STAGES)()
    n = ctypes.c_int(-1)
    assert lib.moe_profile_read(ms, ctypes.byref(n)) == 0
    assert n.value == 0 and list(ms) == [0.0] * B.N_STAGES
    gu, n_split = ctypes.c_float(-1.0), ctypes.c_int(-1)
    assert lib.moe_profile_read_gate_up(ctypes.byref(gu), ctypes.byref(n),
                                        ctypes.byref(n_split)) == 0
    assert n.value == 0 and n_split.value == 0 and gu.value == 0.0
    assert lib.moe_profile_read_gate_up(None, ctypes.byref(n), ctypes.byref(n_split)) == -1


def test_layer_routing_views_stay_inside_the_workspace(lib):
    """moe_layer_routing only hands out pointers into the caller's workspace (nothing is
    dereferenced, so a fake aligned address stands in for device memory): the four tables lie
    inside [ws, ws + moe_workspace_bytes), do not overlap, are 256-byte aligned, and have room for
    their sizes. NULL outputs are allowed; a bad config or workspace is refused."""
    P = ctypes.c_void_p
    for sh in (moe_inputs.CONFIGS["16b_bf16"], moe_inputs.CONFIGS["tiny_f32"]):
        cfg = B.MoEConfig.from_shape(sh)
        base, nbytes = 1 << 30, lib.moe_workspace_bytes(ctypes.byref(cfg))
        out = [P() for _ in range(4)]
        assert lib.moe_layer_routing(ctypes.byref(cfg), P(base), nbytes,
                                     *[ctypes.byref(p) for p in out]) == 0
        TK, N = sh.T * sh.top_k, sh.n_routed
        spans = sorted((p.value, p.value + 4 * n) for p, n in zip(out, (N + 1, TK, TK, N)))
        for lo, hi in spans:
            assert base <= lo and hi <= base + nbytes and lo % 256 == 0
        for (lo1, hi1), (lo2, _) in zip(spans, spans[1:]):
            assert hi1 <= lo2
        assert lib.moe_layer_routing(ctypes.byref(cfg), P(base), nbytes, None, None, None,
                                     None) == 0
        assert lib.moe_layer_routing(ctypes.byref(cfg), P(base), nbytes - 1,
                                     *[ctypes.byref(p) for p in out]) == -3
        assert lib.moe_layer_routing(ctypes.byref(cfg), P(base + 16), nbytes,
                                     *[ctypes.byref(p) for p in out]) == -3
    assert lib.moe_layer_routing(ctypes.byref(_cfg(top_k=9)), P(1 << 30), 1 << 30, None, None,
                                 None, None) == -1
