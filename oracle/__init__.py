"""CPU oracle of the mHC sublayer boundary -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline
(and its ``--impl reference`` arm) may import this package.  The product
path (``mhc_residual_boundary_gb300``) never imports it and shares no code
with it.

The arithmetic lives in ``mhc_oracle.c`` (plain C, FP32 one operation at a
time, built with contraction off); this module only builds that file with
gcc and marshals NumPy arrays through ctypes.  ``truth.py`` is a separate
FP64 statement of the same steps used to bound the FP32 oracle's rounding.

Pages cited by the C file:
  [GLM] vllm.models.glm5next.nvidia.specialized_decode.all_reduce_mhc
  [DSV] vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

HC = 4
MIX = 24

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mhc_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmhc_oracle.so")
_lock = threading.Lock()
_lib = None

# Flags: ISO C, no contraction of a*b+c into an FMA, no fast-math, so every
# FP32 expression in the C file rounds exactly as written on x86-64 and
# aarch64 alike.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build (idempotent)."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(
                     os.path.join(_HERE, "mhc_oracle.h")))
        if force or stale:
            os.makedirs(_BUILD_DIR, exist_ok=True)
            tmp = _LIB_PATH + f".{os.getpid()}.tmp"
            subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OracleConfig(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int32),
        ("tp", ctypes.c_int32),
        ("m", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("rows_per_rank", ctypes.c_int32),
        ("sinkhorn_repeat", ctypes.c_int32),
        ("rms_eps", ctypes.c_float),
        ("hc_eps", ctypes.c_float),
        ("post_mult", ctypes.c_float),
        ("norm_eps", ctypes.c_float),
    ]


class OracleIO(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in (
        "partials", "routed", "idx", "weights", "shared", "residual", "post",
        "comb", "hc_fn", "hc_fn_bf16", "scale", "base", "gamma", "residual_out",
        "layer_input", "post_out", "comb_out", "mixes", "pre", "reduced",
        "mx_values", "mx_scales", "pre_in")]


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
        cfgp = ctypes.POINTER(OracleConfig)
        lib.oracle_bf16_to_f32.argtypes, lib.oracle_bf16_to_f32.restype = [ctypes.c_uint16], f32
        lib.oracle_f32_to_bf16.argtypes, lib.oracle_f32_to_bf16.restype = [f32], ctypes.c_uint16
        lib.oracle_f32_to_e4m3.argtypes, lib.oracle_f32_to_e4m3.restype = [f32], ctypes.c_uint8
        lib.oracle_e4m3_to_f64.argtypes, lib.oracle_e4m3_to_f64.restype = [ctypes.c_uint8], ctypes.c_double
        lib.oracle_ue8m0_of_amax.argtypes, lib.oracle_ue8m0_of_amax.restype = [f32], ctypes.c_uint8
        lib.oracle_mxfp8_scale_bytes.argtypes, lib.oracle_mxfp8_scale_bytes.restype = [i32, i32], ctypes.c_size_t
        lib.oracle_swizzle_128x4.argtypes, lib.oracle_swizzle_128x4.restype = [i32, i32, i32], ctypes.c_size_t
        for name in ("oracle_f32_to_bf16_array", "oracle_f32_to_e4m3_array"):
            getattr(lib, name).argtypes = [ctypes.c_size_t, vp, vp]
            getattr(lib, name).restype = None
        steps = {
            "oracle_stage1": 2, "oracle_moe_fold": 5, "oracle_post_mix": 5,
            "oracle_prenorm_gemv": 4, "oracle_prenorm_gemv_bf16": 4, "oracle_mixes_and_pre": 6,
            "oracle_post_from_mixes": 4, "oracle_sinkhorn": 4,
            "oracle_collapse_norm": 4,
        }
        for name, nptr in steps.items():
            fn = getattr(lib, name)
            fn.argtypes = [cfgp, i32, i32] + [vp] * nptr
            fn.restype = None
        lib.oracle_mxfp8.argtypes = [cfgp, i32, i32, vp, vp, vp, ctypes.c_int]
        lib.oracle_mxfp8.restype = None
        lib.oracle_boundary.argtypes = [cfgp, i32, i32, ctypes.c_int, ctypes.POINTER(OracleIO)]
        lib.oracle_boundary.restype = ctypes.c_int
        _lib = lib
    return _lib


@dataclass
class Problem:
    """Sizes and scalars of one boundary problem (mirrors the C config)."""
    hidden: int
    tp: int
    m: int
    top_k: int = 0
    rows_per_rank: int = 0
    sinkhorn_repeat: int = 20
    rms_eps: float = 1e-6
    hc_eps: float = 1e-6
    post_mult: float = 2.0
    norm_eps: float = 1e-6

    def c(self) -> OracleConfig:
        return OracleConfig(self.hidden, self.tp, self.m, self.top_k,
                            self.rows_per_rank, self.sinkhorn_repeat,
                            self.rms_eps, self.hc_eps, self.post_mult,
                            self.norm_eps)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _arr(a, dtype, shape=None):
    a = np.ascontiguousarray(a, dtype=dtype)
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {a.shape}")
    return a


# ----------------------------------------------------------------- scalars
def bf16_to_f32(bits: int) -> float:
    return _load().oracle_bf16_to_f32(int(bits))


def f32_to_bf16(value: float) -> int:
    return _load().oracle_f32_to_bf16(float(value))


def f32_to_e4m3(value: float) -> int:
    return _load().oracle_f32_to_e4m3(float(value))


def e4m3_to_f64(bits: int) -> float:
    return _load().oracle_e4m3_to_f64(int(bits))


def ue8m0_of_amax(amax: float) -> int:
    return _load().oracle_ue8m0_of_amax(float(amax))


def mxfp8_scale_bytes(m: int, hidden: int) -> int:
    return _load().oracle_mxfp8_scale_bytes(m, hidden)


def swizzle_128x4(row: int, col: int, scale_cols: int) -> int:
    return _load().oracle_swizzle_128x4(row, col, scale_cols)


def f32_to_bf16_array(values) -> np.ndarray:
    x = _arr(values, np.float32).reshape(-1)
    out = np.zeros(x.shape, np.uint16)
    _load().oracle_f32_to_bf16_array(x.size, _p(x), _p(out))
    return out


def f32_to_e4m3_array(values) -> np.ndarray:
    x = _arr(values, np.float32).reshape(-1)
    out = np.zeros(x.shape, np.uint8)
    _load().oracle_f32_to_e4m3_array(x.size, _p(x), _p(out))
    return out


# ------------------------------------------------------------------- steps
def stage1(partials) -> np.ndarray:
    tp, m, hidden = partials.shape
    x = _arr(partials, np.uint16)
    y = np.zeros((m, hidden), np.uint16)
    cfg = Problem(hidden, tp, m).c()
    _load().oracle_stage1(ctypes.byref(cfg), 0, m, _p(x), _p(y))
    return y


def moe_fold(routed, idx, weights, shared) -> np.ndarray:
    tp, rows, hidden = routed.shape
    _, m, k = idx.shape
    routed = _arr(routed, np.uint16)
    idx = _arr(idx, np.int32, (tp, m, k))
    weights = _arr(weights, np.float32, (m, k))
    shared = _arr(shared, np.uint16, (tp, m, hidden))
    if np.any(idx < -1) or np.any(idx >= rows):
        raise ValueError("route index out of range")
    y = np.zeros((m, hidden), np.uint16)
    cfg = Problem(hidden, tp, m, top_k=k, rows_per_rank=rows).c()
    _load().oracle_moe_fold(ctypes.byref(cfg), 0, m, _p(routed), _p(idx), _p(weights), _p(shared), _p(y))
    return y


def post_mix(y, residual, post, comb) -> np.ndarray:
    m, hidden = y.shape
    y = _arr(y, np.uint16)
    residual = _arr(residual, np.uint16, (m, HC, hidden))
    post = _arr(post, np.float32).reshape(m, HC)
    comb = _arr(comb, np.float32, (m, HC, HC))
    out = np.zeros((m, HC, hidden), np.uint16)
    cfg = Problem(hidden, 1, m).c()
    _load().oracle_post_mix(ctypes.byref(cfg), 0, m, _p(y), _p(residual), _p(post), _p(comb), _p(out))
    return out


def prenorm_gemv(streams, hc_fn):
    m, _, hidden = streams.shape
    streams = _arr(streams, np.uint16)
    hc_fn = _arr(hc_fn, np.float32, (HC * hidden, MIX))
    raw = np.zeros((m, MIX), np.float32)
    ss = np.zeros((m,), np.float32)
    cfg = Problem(hidden, 1, m).c()
    _load().oracle_prenorm_gemv(ctypes.byref(cfg), 0, m, _p(streams), _p(hc_fn), _p(raw), _p(ss))
    return raw, ss


def consume(problem: Problem, inputs: dict, pre, *, moe: bool = False, mxfp8_out: bool = False,
            residual_only: bool = False) -> dict:
    """[DSV] AllReduceMHC's delayed-mHC consumer: stage 1 (or the MoE fold),
    the post-mix, and the collapse + RMSNorm with the carried pre-mix ``pre``
    [m][4] (no GEMV, no mixes); with ``residual_only`` the post-mixed streams
    alone."""
    m, hidden = problem.m, problem.hidden
    outputs = {"residual_out": np.zeros((m, HC, hidden), np.uint16),
               "reduced": np.zeros((m, hidden), np.uint16)}
    if not residual_only:
        outputs["layer_input"] = np.zeros((m, hidden), np.uint16)
        if mxfp8_out:
            outputs["mx_values"] = np.zeros((m, hidden), np.uint8)
            outputs["mx_scales"] = np.full((mxfp8_scale_bytes(m, hidden),), 0xAB, np.uint8)
    ins = dict(inputs)
    ins["pre_in"] = _arr(pre, np.float32, (m, HC))
    return boundary(problem, ins, moe=moe, mxfp8_out=mxfp8_out and not residual_only, outputs=outputs)


def prenorm_gemv_bf16(streams, fn):
    """The GEMV with the weight as BF16 [24][4H] (the GLM page's layout)."""
    m, _, hidden = streams.shape
    streams = _arr(streams, np.uint16)
    fn = _arr(fn, np.uint16, (MIX, HC * hidden))
    raw = np.zeros((m, MIX), np.float32)
    ss = np.zeros((m,), np.float32)
    cfg = Problem(hidden, 1, m).c()
    _load().oracle_prenorm_gemv_bf16(ctypes.byref(cfg), 0, m, _p(streams), _p(fn), _p(raw), _p(ss))
    return raw, ss


def mixes_and_pre(raw, ss, scale, base, hidden, rms_eps=1e-6, hc_eps=1e-6):
    m = raw.shape[0]
    raw = _arr(raw, np.float32, (m, MIX))
    ss = _arr(ss, np.float32, (m,))
    scale = _arr(scale, np.float32, (3,))
    base = _arr(base, np.float32, (MIX,))
    mixes = np.zeros((m, MIX), np.float32)
    pre = np.zeros((m, HC), np.float32)
    cfg = Problem(hidden, 1, m, rms_eps=rms_eps, hc_eps=hc_eps).c()
    _load().oracle_mixes_and_pre(ctypes.byref(cfg), 0, m, _p(raw), _p(ss), _p(scale), _p(base), _p(mixes), _p(pre))
    return mixes, pre


def post_from_mixes(mixes, scale, base, post_mult=2.0):
    m = mixes.shape[0]
    mixes = _arr(mixes, np.float32, (m, MIX))
    out = np.zeros((m, HC), np.float32)
    cfg = Problem(8, 1, m, post_mult=post_mult).c()
    _load().oracle_post_from_mixes(ctypes.byref(cfg), 0, m, _p(mixes), _p(_arr(scale, np.float32, (3,))),
                                   _p(_arr(base, np.float32, (MIX,))), _p(out))
    return out


def sinkhorn(mixes, scale, base, hc_eps=1e-6, repeat=20):
    m = mixes.shape[0]
    mixes = _arr(mixes, np.float32, (m, MIX))
    out = np.zeros((m, HC, HC), np.float32)
    cfg = Problem(8, 1, m, hc_eps=hc_eps, sinkhorn_repeat=repeat).c()
    _load().oracle_sinkhorn(ctypes.byref(cfg), 0, m, _p(mixes), _p(_arr(scale, np.float32, (3,))),
                            _p(_arr(base, np.float32, (MIX,))), _p(out))
    return out


def collapse_norm(streams, pre, gamma, norm_eps=1e-6):
    m, _, hidden = streams.shape
    streams = _arr(streams, np.uint16)
    pre = _arr(pre, np.float32, (m, HC))
    gamma = _arr(gamma, np.uint16, (hidden,))
    out = np.zeros((m, hidden), np.uint16)
    cfg = Problem(hidden, 1, m, norm_eps=norm_eps).c()
    _load().oracle_collapse_norm(ctypes.byref(cfg), 0, m, _p(streams), _p(pre), _p(gamma), _p(out))
    return out


def mxfp8(layer_input, pad: bool = True):
    m, hidden = layer_input.shape
    if hidden % 128:
        raise ValueError("MXFP8 needs hidden % 128 == 0")
    x = _arr(layer_input, np.uint16)
    values = np.zeros((m, hidden), np.uint8)
    scales = np.full((mxfp8_scale_bytes(m, hidden),), 0xAB, np.uint8)
    cfg = Problem(hidden, 1, m).c()
    _load().oracle_mxfp8(ctypes.byref(cfg), 0, m, _p(x), _p(values), _p(scales), int(pad))
    return values, scales


# ------------------------------------------------------------ whole boundary
def boundary(problem: Problem, inputs: dict, *, moe: bool = False,
             mxfp8_out: bool = False, t0: int = 0, t1: int | None = None,
             outputs: dict | None = None) -> dict:
    """Runs every step for tokens [t0, t1) into ``outputs`` (allocated here
    when not given).  ``inputs`` holds NumPy arrays named as in the C-ABI."""
    p = problem
    m, hidden = p.m, p.hidden
    t1 = m if t1 is None else t1
    if outputs is None:
        outputs = {
            "residual_out": np.zeros((m, HC, hidden), np.uint16),
            "layer_input": np.zeros((m, hidden), np.uint16),
            "post_out": np.zeros((m, HC), np.float32),
            "comb_out": np.zeros((m, HC, HC), np.float32),
            "mixes": np.zeros((m, MIX), np.float32),
            "pre": np.zeros((m, HC), np.float32),
            "reduced": np.zeros((m, hidden), np.uint16),
        }
        if mxfp8_out:
            outputs["mx_values"] = np.zeros((m, hidden), np.uint8)
            outputs["mx_scales"] = np.full((mxfp8_scale_bytes(m, hidden),), 0xAB, np.uint8)
    keep = {}

    def ptr(name, dtype, src):
        a = src.get(name)
        if a is None:
            return None
        a = np.ascontiguousarray(a, dtype=dtype)
        keep[name] = a
        return a.ctypes.data_as(ctypes.c_void_p)

    io = OracleIO()
    for name, dtype in (("partials", np.uint16), ("routed", np.uint16), ("idx", np.int32),
                        ("weights", np.float32), ("shared", np.uint16), ("residual", np.uint16),
                        ("post", np.float32), ("comb", np.float32), ("hc_fn", np.float32),
                        ("hc_fn_bf16", np.uint16), ("pre_in", np.float32),
                        ("scale", np.float32), ("base", np.float32), ("gamma", np.uint16)):
        setattr(io, name, ptr(name, dtype, inputs))
    for name in ("residual_out", "layer_input", "post_out", "comb_out", "mixes", "pre",
                 "reduced", "mx_values", "mx_scales"):
        a = outputs.get(name)
        if a is not None:
            if not a.flags["C_CONTIGUOUS"]:
                raise ValueError(f"{name} must be C-contiguous")
            setattr(io, name, a.ctypes.data_as(ctypes.c_void_p))
    cfg = p.c()
    status = _load().oracle_boundary(ctypes.byref(cfg), t0, t1, int(moe), ctypes.byref(io))
    if status != 0:
        raise ValueError(f"oracle_boundary failed with status {status}")
    return outputs
