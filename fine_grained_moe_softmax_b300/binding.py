"""ctypes binding of ``libmoe_b300.so`` with the C ABI's own names (include/moe_b300.h).

Argument marshalling only: tensors become device pointers, the stream defaults to torch's current
stream, and a negative status raises ``MoEError``. Every step of the layer runs in the library's
CUDA kernels; there is no other implementation behind these functions. If the library is missing
or cannot be loaded, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "moe_b300.h")

MOE_DTYPE_F32, MOE_DTYPE_BF16 = 0, 1
N_STAGES = 7
STAGE_NAMES = ("router", "permute", "gather", "gemm_gate_up", "gemm_down", "combine", "stats")


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class MoEConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("n_routed", ctypes.c_int32), ("inter", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("renormalize", ctypes.c_int32), ("n_groups", ctypes.c_int32),
                ("alpha1", ctypes.c_float), ("alpha2", ctypes.c_float), ("dtype", ctypes.c_int32),
                ("skip_top", ctypes.c_int32), ("drop_shared", ctypes.c_int32)]

    @classmethod
    def from_shape(cls, shape, T: Optional[int] = None) -> "MoEConfig":
        return cls(shape.T if T is None else T, shape.d, shape.n_shared, shape.n_routed,
                   shape.inter, shape.top_k, shape.renormalize, shape.n_groups, shape.alpha1,
                   shape.alpha2, MOE_DTYPE_F32 if shape.dtype == "f32" else MOE_DTYPE_BF16,
                   getattr(shape, "skip_top", 0), getattr(shape, "drop_shared", 0))

    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == MOE_DTYPE_F32 else torch.bfloat16


_lib = None
_P = ctypes.c_void_p
_CFG = ctypes.POINTER(MoEConfig)
_SIG = {
    "moe_workspace_bytes": (ctypes.c_size_t, [_CFG]),
    "moe_packed_weight_bytes": (ctypes.c_size_t, [_CFG]),
    "moe_pack_weights": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P]),
    "moe_route": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_permute": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_expert_ffn": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_combine": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_balance_stats": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P]),
    "moe_layer_forward": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                         ctypes.c_size_t, _P]),
    "moe_layer_routing": (ctypes.c_int, [_CFG, _P, ctypes.c_size_t, ctypes.POINTER(_P),
                                         ctypes.POINTER(_P), ctypes.POINTER(_P),
                                         ctypes.POINTER(_P)]),
    "moe_backward_workspace_bytes": (ctypes.c_size_t, [_CFG]),
    "moe_packed_backward_bytes": (ctypes.c_size_t, [_CFG]),
    "moe_pack_weights_backward": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P]),
    "moe_layer_backward": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                          _P, ctypes.c_size_t, _P]),
    "moe_layer_forward_train": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                               _P, ctypes.c_size_t, _P]),
    "moe_layer_backward_saved": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                                _P, ctypes.c_size_t, _P]),
    "moe_device_status": (ctypes.c_int, [_P, _P]),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_selftest_bounded_wait": (ctypes.c_int, [_P, ctypes.c_size_t, ctypes.c_uint64, _P]),
    "moe_launch_count": (ctypes.c_uint64, []),
    "moe_profile_enable": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
    "moe_profile_read": (ctypes.c_int, [ctypes.POINTER(ctypes.c_float),
                                        ctypes.POINTER(ctypes.c_int)]),
    "moe_profile_read_gate_up": (ctypes.c_int, [ctypes.POINTER(ctypes.c_float),
                                                ctypes.POINTER(ctypes.c_int),
                                                ctypes.POINTER(ctypes.c_int)]),
}


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m fine_grained_moe_softmax_b300.build` (nvcc, sm_103a)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIG.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def header_functions() -> list:
    """Names of the functions declared in include/moe_b300.h."""
    with open(HEADER) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(moe_[a-z_0-9]+)\s*\(",
                                 text, flags=re.M)))


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(rc: int, where: str):
    if rc != 0:
        raise MoEError(rc, where)


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


# ---------------------------------------------------------------------- C ABI, same names ----

def moe_workspace_bytes(cfg: MoEConfig) -> int:
    return int(lib().moe_workspace_bytes(ctypes.byref(cfg)))


def moe_packed_weight_bytes(cfg: MoEConfig) -> int:
    return int(lib().moe_packed_weight_bytes(ctypes.byref(cfg)))


def moe_pack_weights(cfg, w_gate, w_up, w_down, packed, stream=None):
    _check(lib().moe_pack_weights(ctypes.byref(cfg), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                  _ptr(packed), _stream(stream)), "moe_pack_weights")


def moe_route(cfg, u, centroids, logit_bias, topk_idx, topk_gate, counts, psum, ws, stream=None):
    _check(lib().moe_route(ctypes.byref(cfg), _ptr(u), _ptr(centroids), _ptr(logit_bias),
                           _ptr(topk_idx), _ptr(topk_gate), _ptr(counts), _ptr(psum), _ptr(ws),
                           _nbytes(ws), _stream(stream)), "moe_route")


def moe_permute(cfg, topk_idx, counts, offsets, perm_token, perm_slot, ws, stream=None):
    _check(lib().moe_permute(ctypes.byref(cfg), _ptr(topk_idx), _ptr(counts), _ptr(offsets),
                             _ptr(perm_token), _ptr(perm_slot), _ptr(ws), _nbytes(ws),
                             _stream(stream)), "moe_permute")


def moe_expert_ffn(cfg, u, packed_w, offsets, perm_token, y_routed, y_shared, ws, stream=None):
    _check(lib().moe_expert_ffn(ctypes.byref(cfg), _ptr(u), _ptr(packed_w), _ptr(offsets),
                                _ptr(perm_token), _ptr(y_routed), _ptr(y_shared), _ptr(ws),
                                _nbytes(ws), _stream(stream)), "moe_expert_ffn")


def moe_combine(cfg, u, y_routed, y_shared, perm_slot, topk_gate, h, ws, stream=None):
    _check(lib().moe_combine(ctypes.byref(cfg), _ptr(u), _ptr(y_routed), _ptr(y_shared),
                             _ptr(perm_slot), _ptr(topk_gate), _ptr(h), _ptr(ws), _nbytes(ws),
                             _stream(stream)), "moe_combine")


def moe_balance_stats(cfg, counts, psum, f, P, losses, stream=None):
    _check(lib().moe_balance_stats(ctypes.byref(cfg), _ptr(counts), _ptr(psum), _ptr(f), _ptr(P),
                                   _ptr(losses), _stream(stream)), "moe_balance_stats")


def moe_layer_forward(cfg, u, centroids, logit_bias, packed_w, h, topk_idx, topk_gate, counts, f,
                      P, losses, ws, stream=None):
    _check(lib().moe_layer_forward(ctypes.byref(cfg), _ptr(u), _ptr(centroids), _ptr(logit_bias),
                                   _ptr(packed_w), _ptr(h), _ptr(topk_idx), _ptr(topk_gate),
                                   _ptr(counts), _ptr(f), _ptr(P), _ptr(losses), _ptr(ws),
                                   _nbytes(ws), _stream(stream)), "moe_layer_forward")


def moe_layer_routing(cfg, ws) -> dict:
    """Views into ``ws`` of the routing tables the last moe_layer_forward on it left there:
    offsets [N'+1], perm_token [T*K'], perm_slot [T*K'] (int32) and psum [N'] (fp32)."""
    ptrs = [ctypes.c_void_p() for _ in range(4)]
    _check(lib().moe_layer_routing(ctypes.byref(cfg), _ptr(ws), _nbytes(ws),
                                   *[ctypes.byref(p) for p in ptrs]), "moe_layer_routing")
    base = ws.data_ptr()
    TK, N = cfg.T * cfg.top_k, cfg.n_routed
    out = {}
    for name, p, n, dt in (("offsets", ptrs[0], N + 1, torch.int32),
                           ("perm_token", ptrs[1], TK, torch.int32),
                           ("perm_slot", ptrs[2], TK, torch.int32),
                           ("psum", ptrs[3], N, torch.float32)):
        off = p.value - base
        out[name] = ws[off:off + 4 * n].view(dt)
    return out


def moe_backward_workspace_bytes(cfg: MoEConfig) -> int:
    return int(lib().moe_backward_workspace_bytes(ctypes.byref(cfg)))


def moe_packed_backward_bytes(cfg: MoEConfig) -> int:
    return int(lib().moe_packed_backward_bytes(ctypes.byref(cfg)))


def moe_pack_weights_backward(cfg, w_gate, w_up, w_down, packed_bwd, stream=None):
    _check(lib().moe_pack_weights_backward(ctypes.byref(cfg), _ptr(w_gate), _ptr(w_up),
                                           _ptr(w_down), _ptr(packed_bwd), _stream(stream)),
           "moe_pack_weights_backward")


def moe_layer_backward(cfg, u, centroids, logit_bias, packed_w, packed_bwd, dh, du, d_centroids,
                       d_bias, dw_gate, dw_up, dw_down, ws, stream=None):
    _check(lib().moe_layer_backward(ctypes.byref(cfg), _ptr(u), _ptr(centroids), _ptr(logit_bias),
                                    _ptr(packed_w), _ptr(packed_bwd), _ptr(dh), _ptr(du),
                                    _ptr(d_centroids), _ptr(d_bias), _ptr(dw_gate), _ptr(dw_up),
                                    _ptr(dw_down), _ptr(ws), _nbytes(ws), _stream(stream)),
           "moe_layer_backward")


def moe_layer_forward_train(cfg, u, centroids, logit_bias, packed_w, h, topk_idx, topk_gate,
                            counts, f, P, losses, ws, stream=None):
    _check(lib().moe_layer_forward_train(ctypes.byref(cfg), _ptr(u), _ptr(centroids),
                                         _ptr(logit_bias), _ptr(packed_w), _ptr(h), _ptr(topk_idx),
                                         _ptr(topk_gate), _ptr(counts), _ptr(f), _ptr(P),
                                         _ptr(losses), _ptr(ws), _nbytes(ws), _stream(stream)),
           "moe_layer_forward_train")


def moe_layer_backward_saved(cfg, u, centroids, logit_bias, packed_bwd, dh, du, d_centroids,
                             d_bias, dw_gate, dw_up, dw_down, ws, stream=None):
    _check(lib().moe_layer_backward_saved(ctypes.byref(cfg), _ptr(u), _ptr(centroids),
                                          _ptr(logit_bias), _ptr(packed_bwd), _ptr(dh), _ptr(du),
                                          _ptr(d_centroids), _ptr(d_bias), _ptr(dw_gate),
                                          _ptr(dw_up), _ptr(dw_down), _ptr(ws), _nbytes(ws),
                                          _stream(stream)),
           "moe_layer_backward_saved")


def moe_device_status(ws, stream=None) -> int:
    return int(lib().moe_device_status(_ptr(ws), _stream(stream)))


def moe_status_string(status: int) -> str:
    return status_string(status)


def moe_selftest_bounded_wait(ws, timeout_ns: int, stream=None):
    _check(lib().moe_selftest_bounded_wait(_ptr(ws), _nbytes(ws), int(timeout_ns),
                                           _stream(stream)), "moe_selftest_bounded_wait")


def moe_launch_count() -> int:
    return int(lib().moe_launch_count())


def moe_profile_enable(enable: bool, max_calls: int = 64):
    _check(lib().moe_profile_enable(int(bool(enable)), int(max_calls)), "moe_profile_enable")


def moe_profile_read():
    """(per-stage summed milliseconds as a dict, number of recorded calls)."""
    ms = (ctypes.c_float * N_STAGES)()
    n = ctypes.c_int()
    _check(lib().moe_profile_read(ms, ctypes.byref(n)), "moe_profile_read")
    return dict(zip(STAGE_NAMES, list(ms))), n.value


def moe_profile_read_gate_up():
    """(summed milliseconds of the gate/up launch over the routed groups, recorded calls, calls
    whose shared group had a gate/up launch of its own)."""
    ms = ctypes.c_float()
    n, n_split = ctypes.c_int(), ctypes.c_int()
    _check(lib().moe_profile_read_gate_up(ctypes.byref(ms), ctypes.byref(n), ctypes.byref(n_split)),
           "moe_profile_read_gate_up")
    return ms.value, n.value, n_split.value
