"""PyTorch-facing wrapper of the boundary library: tensors in, tensors out.

PyTorch supplies device memory and streams; the wrapper checks shapes and
dtypes (so that every pointer it hands over covers the sizes the C ABI
assumes) and passes raw pointers.  All arithmetic runs in the CUDA kernels.
Interface after [GLM] AllReduceMhcBoundary (vllm.models.glm5next.nvidia.
specialized_decode.all_reduce_mhc) and [DSV] AllReduceMHC (vllm.models.
deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc).
"""
from __future__ import annotations

import torch

from . import capi

HC = 4
MIX = 24

INPUT_SPECS = {
    # name: (dtype, shape as a function of (tp, m, H, K, rows))
    "partials": (torch.bfloat16, lambda tp, m, H, K, R: (tp, m, H)),
    "residual": (torch.bfloat16, lambda tp, m, H, K, R: (m, HC, H)),
    "post": (torch.float32, lambda tp, m, H, K, R: (m, HC)),
    "comb": (torch.float32, lambda tp, m, H, K, R: (m, HC, HC)),
    "hc_fn": (torch.float32, lambda tp, m, H, K, R: (HC * H, MIX)),
    "hc_fn_bf16": (torch.bfloat16, lambda tp, m, H, K, R: (MIX, HC * H)),
    "scale": (torch.float32, lambda tp, m, H, K, R: (3,)),
    "base": (torch.float32, lambda tp, m, H, K, R: (MIX,)),
    "norm_weight": (torch.bfloat16, lambda tp, m, H, K, R: (H,)),
    "routed": (torch.bfloat16, lambda tp, m, H, K, R: (tp, R, H)),
    "idx": (torch.int32, lambda tp, m, H, K, R: (tp, m, K)),
    "weights": (torch.float32, lambda tp, m, H, K, R: (m, K)),
    "shared": (torch.bfloat16, lambda tp, m, H, K, R: (tp, m, H)),
}

OUTPUT_SPECS = {
    "residual_out": (torch.bfloat16, lambda m, H: (m, HC, H)),
    "layer_input": (torch.bfloat16, lambda m, H: (m, H)),
    "post_out": (torch.float32, lambda m, H: (m, HC)),
    "comb_out": (torch.float32, lambda m, H: (m, HC, HC)),
    "pre_out": (torch.float32, lambda m, H: (m, HC)),
    "pre": (torch.float32, lambda m, H: (m, HC)),
    "mixes_out": (torch.float32, lambda m, H: (m, MIX)),
    "reduced_out": (torch.bfloat16, lambda m, H: (m, H)),
    "mxfp8_values": (torch.uint8, lambda m, H: (m, H)),
    "mxfp8_scales": (torch.uint8, lambda m, H: (capi.mhc_mxfp8_scale_bytes(m, H),)),
}

REQUIRED_OUTPUTS = ("residual_out", "layer_input", "post_out", "comb_out")


class Boundary:
    """One boundary instance: it serves every call of up to max_num_tokens
    tokens ([GLM] AllReduceMhcBoundary: one instance serves every boundary
    of the model, one after another).

    Flags (include/mhc_boundary.h): mxfp8 (accept the MXFP8 outputs),
    sync_mixes / side_mixes (post and Sinkhorn in a separate kernel on the
    caller's stream / a side stream), host_staging (allow run_host),
    static_weight (the prenorm weight is a layer weight, staged while the
    kernel before the call finishes), owner_reduce (the two-shot reduction:
    an owner-reduce kernel sums the partials first).  All give the same
    results."""

    def __init__(self, *, hidden: int, tp: int, max_num_tokens: int, sinkhorn_repeat: int = 20,
                 top_k: int = 0, rms_eps: float = 1e-6, hc_eps: float = 1e-6,
                 post_mult: float = 2.0, norm_eps: float = 1e-6, mxfp8: bool = False,
                 sync_mixes: bool = False, side_mixes: bool = False, host_staging: bool = False,
                 static_weight: bool = False, owner_reduce: bool = False, device=None):
        if device is None:
            device = torch.cuda.current_device()
        self.device = torch.device("cuda", int(torch.device("cuda", device).index
                                               if not isinstance(device, int) else device))
        flags = ((capi.MHC_FLAG_MXFP8 if mxfp8 else 0) | (capi.MHC_FLAG_SYNC_MIXES if sync_mixes else 0)
                 | (capi.MHC_FLAG_HOST_STAGING if host_staging else 0)
                 | (capi.MHC_FLAG_SIDE_MIXES if side_mixes else 0)
                 | (capi.MHC_FLAG_STATIC_WEIGHT if static_weight else 0)
                 | (capi.MHC_FLAG_OWNER_REDUCE if owner_reduce else 0))
        self.config = capi.mhc_boundary_config_t(hidden, HC, tp, max_num_tokens, sinkhorn_repeat, top_k,
                                                 rms_eps, hc_eps, post_mult, norm_eps, flags)
        self.hidden, self.tp, self.top_k, self.capacity = hidden, tp, top_k, max_num_tokens
        self.handle = capi.mhc_boundary_create(self.config, self.device.index)

    # ------------------------------------------------------------ lifecycle
    def close(self) -> None:
        if getattr(self, "handle", None):
            capi.mhc_boundary_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -------------------------------------------------------------- helpers
    def supports(self, tokens: int) -> bool:
        return 1 <= tokens <= self.capacity

    def empty_outputs(self, m: int, *, extras: bool = False, mxfp8: bool = False,
                      device=None, pin_memory: bool = False) -> dict:
        """Output tensors of an m-token call (device tensors unless device='cpu')."""
        device = self.device if device is None else torch.device(device)
        names = list(REQUIRED_OUTPUTS)
        if extras:
            names += ["pre_out", "mixes_out", "reduced_out"]
        if mxfp8:
            names += ["mxfp8_values", "mxfp8_scales"]
        out = {}
        for n in names:
            dtype, shape = OUTPUT_SPECS[n]
            out[n] = torch.empty(shape(m, self.hidden), dtype=dtype, device=device,
                                 pin_memory=pin_memory and device.type == "cpu")
        return out

    def _args(self, inputs: dict, outputs: dict, moe: bool, where: str) -> tuple:
        m = outputs["layer_input"].shape[0]
        K = self.top_k
        rows = inputs["routed"].shape[1] if moe else 0
        args = capi.mhc_run_args_t()
        args.m = m
        # the prenorm weight: FP32 [4H][24] (hc_fn) or BF16 [24][4H] (hc_fn_bf16)
        weight = "hc_fn_bf16" if inputs.get("hc_fn_bf16") is not None else "hc_fn"
        names = ["residual", "post", "comb", weight, "scale", "base", "norm_weight"]
        names += ["routed", "idx", "weights", "shared"] if moe else ["partials"]
        for n in names:
            t = inputs[n]
            dtype, shape = INPUT_SPECS[n]
            want = shape(self.tp, m, self.hidden, K, rows)
            if t.dtype != dtype or tuple(t.shape) != want or not t.is_contiguous():
                raise ValueError(f"{n}: expected contiguous {dtype} {want}, got {t.dtype} {tuple(t.shape)}")
            self._check_place(n, t, where)
        for n in names:
            if n in capi.RUN_FIELDS:
                setattr(args, n, inputs[n].data_ptr())
        for n, t in outputs.items():
            dtype, shape = OUTPUT_SPECS[n]
            if t.dtype != dtype or tuple(t.shape) != shape(m, self.hidden) or not t.is_contiguous():
                raise ValueError(f"{n}: expected contiguous {dtype} {shape(m, self.hidden)}")
            self._check_place(n, t, where)
            setattr(args, n, t.data_ptr())
        return args, rows

    def _check_place(self, n: str, t: torch.Tensor, where: str) -> None:
        # the kernels dereference every pointer on this boundary's GPU: a
        # device call takes tensors on that GPU, a host call host tensors
        if where == "device":
            if t.device != self.device:
                raise ValueError(f"{n} must be a tensor on {self.device}, got {t.device}")
        elif t.device.type != "cpu":
            raise ValueError(f"{n} must be a host tensor, got {t.device}")

    # ---------------------------------------------------------------- calls
    def run(self, inputs: dict, outputs: dict, stream=None) -> dict:
        """One boundary call; post_out / comb_out need join() (or the next call)
        before the caller's stream reads them."""
        args, _ = self._args(inputs, outputs, False, "device")
        capi.mhc_boundary_run(self.handle, args, stream)
        return outputs

    def finalize_moe(self, inputs: dict, outputs: dict, stream=None) -> dict:
        run, rows = self._args(inputs, outputs, True, "device")
        args = capi.mhc_moe_args_t()
        args.run = run
        args.run.partials = None
        args.rows_per_rank = rows
        for n in ("routed", "idx", "weights", "shared"):
            setattr(args, n, inputs[n].data_ptr())
        capi.mhc_boundary_finalize_moe(self.handle, args, stream)
        return outputs

    def consume(self, inputs: dict, outputs: dict, stream=None) -> dict:
        """The delayed-mHC consumer ([DSV] AllReduceMHC.__call__ / finalize):
        inputs hold partials (or routed / idx / weights / shared), residual,
        post, comb and, unless residual only, pre [m][4] and norm_weight;
        outputs hold residual_out and, with pre, layer_input (optionally
        reduced_out, mxfp8_values / mxfp8_scales)."""
        m = outputs["residual_out"].shape[0]
        a = capi.mhc_consume_args_t()
        a.m = m
        moe = inputs.get("partials") is None
        K = self.top_k
        rows = inputs["routed"].shape[1] if moe else 0
        names = ["residual", "post", "comb"]
        names += ["routed", "idx", "weights", "shared"] if moe else ["partials"]
        if inputs.get("pre") is not None:
            names += ["pre", "norm_weight"]
        for n in names:
            t = inputs[n]
            dtype, shape = INPUT_SPECS[n] if n in INPUT_SPECS else OUTPUT_SPECS[n]
            want = shape(self.tp, m, self.hidden, K, rows) if n in INPUT_SPECS else shape(m, self.hidden)
            if t.dtype != dtype or tuple(t.shape) != want or not t.is_contiguous():
                raise ValueError(f"{n}: expected contiguous {dtype} {want}")
            self._check_place(n, t, "device")
            setattr(a, n, t.data_ptr())
        a.rows_per_rank = rows
        for n, t in outputs.items():
            dtype, shape = OUTPUT_SPECS[n]
            if t.dtype != dtype or tuple(t.shape) != shape(m, self.hidden) or not t.is_contiguous():
                raise ValueError(f"{n}: expected contiguous {dtype} {shape(m, self.hidden)}")
            self._check_place(n, t, "device")
            setattr(a, n, t.data_ptr())
        capi.mhc_boundary_consume(self.handle, a, stream)
        return outputs

    def run_host(self, inputs: dict, outputs: dict, stream=None) -> dict:
        """The call on host tensors (pinned for asynchronous copies); returns
        when the outputs are in host memory."""
        args, _ = self._args(inputs, outputs, False, "host")
        capi.mhc_boundary_run_host(self.handle, args, stream)
        return outputs

    def join(self, stream=None) -> None:
        capi.mhc_boundary_join(self.handle, stream)

    def check_errors(self) -> None:
        capi.mhc_boundary_check_errors(self.handle)

    def profile_begin(self, max_calls: int) -> None:
        capi.mhc_boundary_profile_begin(self.handle, max_calls)

    def profile_end(self) -> dict:
        p = capi.mhc_boundary_profile_end(self.handle)
        return {"calls": p.calls, "stage_ms": p.stage_ms, "finish_ms": p.finish_ms, "mixes_ms": p.mixes_ms}

    def launches_per_call(self) -> int:
        return capi.mhc_boundary_launches_per_call(self.handle)
