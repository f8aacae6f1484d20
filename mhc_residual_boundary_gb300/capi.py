"""ctypes binding of include/mhc_boundary.h (argument marshalling only).

The functions keep the C names; every step of the boundary runs in the CUDA
library.  Loading fails loudly when the library has not been built: there is
no CPU or PyTorch fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch  # loads the CUDA runtime the library links against

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libmhc_boundary.so")

MHC_OK = 0
STATUS = {0: "MHC_OK", 1: "MHC_ERR_INVALID_ARG", 2: "MHC_ERR_UNSUPPORTED", 3: "MHC_ERR_CAPACITY",
          4: "MHC_ERR_CUDA", 5: "MHC_ERR_OOM", 6: "MHC_ERR_TIMEOUT"}
MHC_FLAG_MXFP8 = 1 << 0
MHC_FLAG_SYNC_MIXES = 1 << 1
MHC_FLAG_HOST_STAGING = 1 << 2
MHC_FLAG_SIDE_MIXES = 1 << 3
MHC_FLAG_STATIC_WEIGHT = 1 << 4
MHC_FLAG_OWNER_REDUCE = 1 << 5
MHC_FLAG_CHECK_ERRORS = 1 << 6


class MhcError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class mhc_boundary_config_t(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("hc_mult", ctypes.c_int32), ("tp", ctypes.c_int32),
                ("max_num_tokens", ctypes.c_int32), ("sinkhorn_repeat", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("hc_eps", ctypes.c_float),
                ("post_mult", ctypes.c_float), ("norm_eps", ctypes.c_float), ("flags", ctypes.c_uint32)]


RUN_FIELDS = ("partials", "residual", "post", "comb", "hc_fn", "scale", "base", "norm_weight",
              "residual_out", "layer_input", "post_out", "comb_out", "pre_out", "mixes_out",
              "reduced_out", "mxfp8_values", "mxfp8_scales", "hc_fn_bf16")


class mhc_run_args_t(ctypes.Structure):
    _fields_ = [("m", ctypes.c_int32)] + [(f, ctypes.c_void_p) for f in RUN_FIELDS]


class mhc_moe_args_t(ctypes.Structure):
    _fields_ = [("run", mhc_run_args_t), ("rows_per_rank", ctypes.c_int32),
                ("routed", ctypes.c_void_p), ("idx", ctypes.c_void_p),
                ("weights", ctypes.c_void_p), ("shared", ctypes.c_void_p)]


class mhc_consume_args_t(ctypes.Structure):
    _fields_ = [("m", ctypes.c_int32), ("partials", ctypes.c_void_p), ("rows_per_rank", ctypes.c_int32)] + [
        (f, ctypes.c_void_p) for f in ("routed", "idx", "weights", "shared", "residual", "post", "comb", "pre",
                                      "norm_weight", "residual_out", "layer_input", "reduced_out",
                                      "mxfp8_values", "mxfp8_scales")]


class mhc_profile_t(ctypes.Structure):
    _fields_ = [("calls", ctypes.c_int32), ("stage_ms", ctypes.c_float), ("finish_ms", ctypes.c_float),
                ("mixes_ms", ctypes.c_float)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with mhc_residual_boundary_gb300.build.build() "
                "(nvcc for sm_103a); there is no fallback path")
        h = ctypes.CDLL(LIB_PATH)
        vp, st = ctypes.c_void_p, ctypes.c_int
        h.mhc_boundary_create.argtypes = [ctypes.POINTER(mhc_boundary_config_t), ctypes.c_int, ctypes.POINTER(vp)]
        h.mhc_boundary_run.argtypes = [vp, ctypes.POINTER(mhc_run_args_t), vp]
        h.mhc_boundary_run_host.argtypes = [vp, ctypes.POINTER(mhc_run_args_t), vp]
        h.mhc_boundary_finalize_moe.argtypes = [vp, ctypes.POINTER(mhc_moe_args_t), vp]
        h.mhc_boundary_join.argtypes = [vp, vp]
        h.mhc_boundary_consume.argtypes = [vp, ctypes.POINTER(mhc_consume_args_t), vp]
        h.mhc_boundary_check_errors.argtypes = [vp]
        h.mhc_boundary_destroy.argtypes = [vp]
        h.mhc_boundary_profile_begin.argtypes = [vp, ctypes.c_int32]
        h.mhc_boundary_profile_end.argtypes = [vp, ctypes.POINTER(mhc_profile_t)]
        for name in ("mhc_boundary_create", "mhc_boundary_run", "mhc_boundary_run_host",
                     "mhc_boundary_finalize_moe", "mhc_boundary_consume", "mhc_boundary_join",
                     "mhc_boundary_check_errors",
                     "mhc_boundary_destroy", "mhc_boundary_profile_begin", "mhc_boundary_profile_end"):
            getattr(h, name).restype = st
        h.mhc_boundary_run_static.argtypes = [ctypes.POINTER(mhc_boundary_config_t),
                                               ctypes.POINTER(mhc_run_args_t), vp, ctypes.c_char_p,
                                               ctypes.c_size_t]
        h.mhc_boundary_run_static.restype = st
        h.mhc_mxfp8_scale_bytes.argtypes = [ctypes.c_int32, ctypes.c_int32]
        h.mhc_test_stall_stage_copies.argtypes = [ctypes.c_int32]
        h.mhc_test_stall_stage_copies.restype = st
        h.mhc_mxfp8_scale_bytes.restype = ctypes.c_size_t
        h.mhc_boundary_launches_per_call.argtypes = [vp]
        h.mhc_boundary_launches_per_call.restype = ctypes.c_int32
        h.mhc_status_string.argtypes = [st]
        h.mhc_status_string.restype = ctypes.c_char_p
        h.mhc_last_error.argtypes = [vp]
        h.mhc_last_error.restype = ctypes.c_char_p
        _lib = h
    return _lib


def _check(status: int, handle) -> None:
    if status != MHC_OK:
        raise MhcError(status, lib().mhc_last_error(handle).decode())


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    return ctypes.c_void_p(int(stream))


def mhc_boundary_create(config: mhc_boundary_config_t, device: int) -> ctypes.c_void_p:
    handle = ctypes.c_void_p()
    status = lib().mhc_boundary_create(ctypes.byref(config), int(device), ctypes.byref(handle))
    _check(status, None)
    return handle


def mhc_boundary_run(handle, args: mhc_run_args_t, stream=None) -> None:
    _check(lib().mhc_boundary_run(handle, ctypes.byref(args), _stream_ptr(stream)), handle)


def mhc_boundary_run_host(handle, args: mhc_run_args_t, stream=None) -> None:
    _check(lib().mhc_boundary_run_host(handle, ctypes.byref(args), _stream_ptr(stream)), handle)


def mhc_boundary_finalize_moe(handle, args: mhc_moe_args_t, stream=None) -> None:
    _check(lib().mhc_boundary_finalize_moe(handle, ctypes.byref(args), _stream_ptr(stream)), handle)


def mhc_boundary_consume(handle, args: mhc_consume_args_t, stream=None) -> None:
    _check(lib().mhc_boundary_consume(handle, ctypes.byref(args), _stream_ptr(stream)), handle)


def mhc_boundary_join(handle, stream=None) -> None:
    _check(lib().mhc_boundary_join(handle, _stream_ptr(stream)), handle)


def mhc_boundary_check_errors(handle) -> None:
    _check(lib().mhc_boundary_check_errors(handle), handle)


def mhc_boundary_destroy(handle) -> None:
    _check(lib().mhc_boundary_destroy(handle), None)


def mhc_boundary_run_static(config: mhc_boundary_config_t, args: mhc_run_args_t, stream=None) -> None:
    """The allocation-free call: no handle, scratch in the library's static
    device array (see include/mhc_boundary.h)."""
    err = ctypes.create_string_buffer(512)
    status = lib().mhc_boundary_run_static(ctypes.byref(config), ctypes.byref(args), _stream_ptr(stream),
                                           err, len(err))
    if status != MHC_OK:
        raise MhcError(status, err.value.decode())


def mhc_test_stall_stage_copies(on: bool) -> None:
    """Test hook (include/mhc_boundary_test.h): the stage kernels launched
    from now on issue no input copies, so their bounded waits run out."""
    status = lib().mhc_test_stall_stage_copies(1 if on else 0)
    if status != MHC_OK:
        raise MhcError(status, "could not set the stall flag")


def mhc_boundary_profile_begin(handle, max_calls: int) -> None:
    _check(lib().mhc_boundary_profile_begin(handle, int(max_calls)), handle)


def mhc_boundary_profile_end(handle) -> mhc_profile_t:
    out = mhc_profile_t()
    _check(lib().mhc_boundary_profile_end(handle, ctypes.byref(out)), handle)
    return out


def mhc_mxfp8_scale_bytes(m: int, hidden: int) -> int:
    return int(lib().mhc_mxfp8_scale_bytes(m, hidden))


def mhc_boundary_launches_per_call(handle) -> int:
    return int(lib().mhc_boundary_launches_per_call(handle))


def mhc_status_string(status: int) -> str:
    return lib().mhc_status_string(status).decode()


def mhc_last_error(handle=None) -> str:
    return lib().mhc_last_error(handle).decode()
