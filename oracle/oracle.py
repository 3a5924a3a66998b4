"""ctypes front end of the fp64 CPU oracle (``moe_oracle.c``). Test infrastructure only.

Arrays go in as numpy arrays or CPU torch tensors: fp32 values, or bf16 tensors, whose bit
patterns are handed over unchanged and widened to double inside the oracle. Everything comes
back as numpy arrays (fp64 for real values).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")
_lib = None

F32, BF16 = 0, 1


def lib_path() -> str:
    return _LIB_PATH


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, OpenMP over tokens, IEEE arithmetic)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC",
                        "-shared", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Cfg(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("d", ctypes.c_int), ("n_shared", ctypes.c_int),
                ("n_routed", ctypes.c_int), ("inter", ctypes.c_int), ("top_k", ctypes.c_int),
                ("renormalize", ctypes.c_int), ("n_groups", ctypes.c_int),
                ("alpha1", ctypes.c_double), ("alpha2", ctypes.c_double), ("dtype", ctypes.c_int),
                ("skip_top", ctypes.c_int), ("drop_shared", ctypes.c_int)]


@dataclass
class OracleCfg:
    T: int
    d: int
    n_shared: int
    n_routed: int
    inter: int
    top_k: int
    renormalize: int = 0
    n_groups: int = 1
    alpha1: float = 0.01
    alpha2: float = 0.05
    dtype: str = "f32"
    skip_top: int = 0
    drop_shared: int = 0

    @classmethod
    def from_shape(cls, shape, T: Optional[int] = None) -> "OracleCfg":
        return cls(T=shape.T if T is None else T, d=shape.d, n_shared=shape.n_shared,
                   n_routed=shape.n_routed, inter=shape.inter, top_k=shape.top_k,
                   renormalize=shape.renormalize, n_groups=shape.n_groups, alpha1=shape.alpha1,
                   alpha2=shape.alpha2, dtype=shape.dtype,
                   skip_top=getattr(shape, "skip_top", 0),
                   drop_shared=getattr(shape, "drop_shared", 0))

    def c(self) -> _Cfg:
        return _Cfg(self.T, self.d, self.n_shared, self.n_routed, self.inter, self.top_k,
                    self.renormalize, self.n_groups, self.alpha1, self.alpha2,
                    F32 if self.dtype == "f32" else BF16, self.skip_top, self.drop_shared)


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        cfgp = ctypes.POINTER(_Cfg)
        lib.oracle_route.argtypes = [cfgp, P, P, P, P, P, P, P, P, P]
        lib.oracle_permute.argtypes = [cfgp, P, P, P, P]
        lib.oracle_forward_tokens.argtypes = [cfgp, P, P, P, P, P, P, ctypes.c_int, P, P, P, P,
                                              P, P, P]
        lib.oracle_balance_stats.argtypes = [cfgp, P, P, P, P, P, P, P]
        lib.oracle_expert_ffn.argtypes = [cfgp, P, P, P, ctypes.c_int, P, P]
        lib.oracle_expert_ffn.restype = None
        lib.oracle_group_range.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P]
        lib.oracle_group_range.restype = None
        lib.oracle_threads.restype = ctypes.c_int
        lib.oracle_backward.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, P, P, P, P, P]
        _lib = lib
    return _lib


def threads() -> int:
    return int(_load().oracle_threads())


def _raw(x, dtype: str) -> np.ndarray:
    """Contiguous numpy view holding fp32 values (f32) or bf16 bit patterns (bf16)."""
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                if dtype != "bf16":
                    raise TypeError("bf16 tensor given to an f32 oracle config")
                return x.view(torch.int16).numpy().view(np.uint16)
            if dtype == "bf16":
                raise TypeError("bf16 oracle config needs bf16 tensors")
            return np.ascontiguousarray(x.to(torch.float32).numpy())
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if dtype == "bf16":
        if x.dtype != np.uint16:
            raise TypeError("bf16 oracle config needs uint16 bit patterns")
        return x
    return x.astype(np.float32, copy=False)


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bias(b):
    if b is None:
        return None
    try:
        import torch
        if isinstance(b, torch.Tensor):
            b = b.detach().cpu().to(torch.float32).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(b, dtype=np.float32)


def route(cfg: OracleCfg, u, centroids, bias=None, want_scores: bool = False) -> dict:
    """Affinities, top-k, gates, near-tie margins, counts and affinity sums for all T tokens."""
    lib = _load()
    T, N, K = cfg.T, cfg.n_routed, cfg.top_k
    u_, e_, b_ = _raw(u, cfg.dtype), _raw(centroids, cfg.dtype), _bias(bias)
    assert u_.size == T * cfg.d and e_.size == N * cfg.d
    out = {"topk_idx": np.zeros((T, K), np.int32), "topk_gate": np.zeros((T, K), np.float64),
           "margin": np.zeros(T, np.float64), "counts": np.zeros(N, np.int64),
           "psum": np.zeros(N, np.float64)}
    scores = np.zeros((T, N), np.float64) if want_scores else None
    c = cfg.c()
    rc = lib.oracle_route(ctypes.byref(c), _p(u_), _p(e_), _p(b_), _p(out["topk_idx"]),
                          _p(out["topk_gate"]), _p(out["margin"]), _p(out["counts"]),
                          _p(out["psum"]), _p(scores))
    if rc != 0:
        raise ValueError("oracle_route rejected its arguments")
    if want_scores:
        out["scores"] = scores
    return out


def permute(cfg: OracleCfg, topk_idx) -> dict:
    """Stable counting sort of the (token, slot) assignments by routed expert."""
    lib = _load()
    idx = np.ascontiguousarray(np.asarray(topk_idx), dtype=np.int32)
    assert idx.size == cfg.T * cfg.top_k
    out = {"offsets": np.zeros(cfg.n_routed + 1, np.int32),
           "perm_token": np.zeros(cfg.T * cfg.top_k, np.int32),
           "perm_slot": np.zeros(cfg.T * cfg.top_k, np.int32)}
    c = cfg.c()
    rc = lib.oracle_permute(ctypes.byref(c), _p(idx), _p(out["offsets"]), _p(out["perm_token"]),
                            _p(out["perm_slot"]))
    if rc != 0:
        raise ValueError("oracle_permute: expert id out of range")
    return out


def forward_tokens(cfg: OracleCfg, inputs: dict, tokens: Sequence[int],
                   want_parts: bool = False) -> dict:
    """h (and routing) for the listed tokens, each routed on its own."""
    lib = _load()
    tok = np.ascontiguousarray(np.asarray(tokens), dtype=np.int32)
    n, d, K = tok.size, cfg.d, cfg.top_k
    u_ = _raw(inputs["u"], cfg.dtype)
    e_ = _raw(inputs["centroids"], cfg.dtype)
    b_ = _bias(inputs.get("bias"))
    wg, wu, wd = (_raw(inputs[k], cfg.dtype) for k in ("w_gate", "w_up", "w_down"))
    E = cfg.n_shared + cfg.n_routed
    assert wg.size == E * cfg.inter * d and wd.size == E * d * cfg.inter
    out = {"h": np.zeros((n, d), np.float64), "topk_idx": np.zeros((n, K), np.int32),
           "topk_gate": np.zeros((n, K), np.float64), "margin": np.zeros(n, np.float64)}
    if want_parts:
        out["shared"] = np.zeros((n, d), np.float64)
        out["routed"] = np.zeros((n, K, d), np.float64)
    c = cfg.c()
    rc = lib.oracle_forward_tokens(ctypes.byref(c), _p(u_), _p(e_), _p(b_), _p(wg), _p(wu), _p(wd),
                                   n, _p(tok), _p(out["h"]), _p(out.get("shared")),
                                   _p(out.get("routed")), _p(out["topk_idx"]),
                                   _p(out["topk_gate"]), _p(out["margin"]))
    if rc != 0:
        raise ValueError("oracle_forward_tokens: token id out of range")
    return out


def expert_ffn(cfg: OracleCfg, inputs: dict, expert: int, x) -> np.ndarray:
    """FFN of one expert (global id) applied to an fp64 vector x [d]."""
    lib = _load()
    wg, wu, wd = (_raw(inputs[k], cfg.dtype) for k in ("w_gate", "w_up", "w_down"))
    x_ = np.ascontiguousarray(x, dtype=np.float64)
    y = np.zeros(cfg.d, np.float64)
    c = cfg.c()
    lib.oracle_expert_ffn(ctypes.byref(c), _p(wg), _p(wu), _p(wd), int(expert), _p(x_), _p(y))
    return y


def balance_stats(cfg: OracleCfg, counts, psum) -> dict:
    """f, P, group f', group P', and (L_ExpBal, L_DevBal)."""
    lib = _load()
    N, D = cfg.n_routed, cfg.n_groups
    cnt = np.ascontiguousarray(np.asarray(counts), dtype=np.int64)
    ps = np.ascontiguousarray(np.asarray(psum), dtype=np.float64)
    out = {"f": np.zeros(N), "P": np.zeros(N), "fg": np.zeros(D), "Pg": np.zeros(D),
           "losses": np.zeros(2)}
    c = cfg.c()
    rc = lib.oracle_balance_stats(ctypes.byref(c), _p(cnt), _p(ps), _p(out["f"]), _p(out["P"]),
                                  _p(out["fg"]), _p(out["Pg"]), _p(out["losses"]))
    if rc != 0:
        raise ValueError("oracle_balance_stats rejected its arguments")
    return out


def group_range(n_routed: int, n_groups: int, g: int):
    lib = _load()
    first, size = ctypes.c_int(), ctypes.c_int()
    lib.oracle_group_range(n_routed, n_groups, g, ctypes.byref(first), ctypes.byref(size))
    return first.value, size.value


def layer_forward(cfg: OracleCfg, inputs: dict, tokens: Optional[Sequence[int]] = None) -> dict:
    """The whole layer: routing and statistics over all T tokens, h for ``tokens`` (all if None)."""
    r = route(cfg, inputs["u"], inputs["centroids"], inputs.get("bias"))
    perm = permute(cfg, r["topk_idx"])
    st = balance_stats(cfg, r["counts"], r["psum"])
    toks = np.arange(cfg.T, dtype=np.int32) if tokens is None else np.asarray(tokens, np.int32)
    fw = forward_tokens(cfg, inputs, toks)
    out = dict(r)
    out.update(perm)
    out.update(st)
    out["tokens"] = toks
    out["h"] = fw["h"]
    return out


def backward(cfg: OracleCfg, inputs: dict, dh, counts=None) -> dict:
    """Gradients of sum_t dh_t . h_t + L_ExpBal + L_DevBal (selection and counts held fixed)."""
    lib = _load()
    T, d, N, I = cfg.T, cfg.d, cfg.n_routed, cfg.inter
    E = cfg.n_shared + N
    u_ = _raw(inputs["u"], cfg.dtype)
    e_ = _raw(inputs["centroids"], cfg.dtype)
    b_ = _bias(inputs.get("bias"))
    wg, wu, wd = (_raw(inputs[k], cfg.dtype) for k in ("w_gate", "w_up", "w_down"))
    dh_ = np.ascontiguousarray(np.asarray(dh, dtype=np.float64).reshape(T, d))
    cnt = None if counts is None else np.ascontiguousarray(np.asarray(counts), dtype=np.int64)
    out = {"du": np.zeros((T, d)), "d_centroids": np.zeros((N, d)), "d_bias": np.zeros(N),
           "dw_gate": np.zeros((E, I, d)), "dw_up": np.zeros((E, I, d)),
           "dw_down": np.zeros((E, d, I))}
    c = cfg.c()
    rc = lib.oracle_backward(ctypes.byref(c), _p(u_), _p(e_), _p(b_), _p(wg), _p(wu), _p(wd),
                             _p(dh_), _p(cnt), _p(out["du"]), _p(out["d_centroids"]),
                             _p(out["d_bias"]), _p(out["dw_gate"]), _p(out["dw_up"]),
                             _p(out["dw_down"]))
    if rc != 0:
        raise ValueError("oracle_backward rejected its arguments")
    return out
