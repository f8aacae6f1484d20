"""FP64 statement of the mHC boundary -- TEST INFRASTRUCTURE ONLY.

The same steps as ``mhc_oracle.c`` with every FP32 operation replaced by
FP64 and every BF16 rounding point kept (rounded straight from the FP64
value).  It bounds the rounding of the FP32 oracle: on small problems the
two must agree within the tolerances stated in the tests.  It is written
separately (vectorised NumPy, no shared helpers) so that a slip in one
statement is unlikely to be repeated in the other.

Pages: [GLM] vllm.models.glm5next.nvidia.specialized_decode.all_reduce_mhc,
[DSV] vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc.
"""
from __future__ import annotations

import numpy as np

HC = 4
MIX = 24


def bf16_bits_to_f64(bits) -> np.ndarray:
    bits = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def round_bf16(x) -> np.ndarray:
    """Nearest BF16 (8 significant bits, FP32 exponent range), ties to even,
    as an FP64 array."""
    x = np.asarray(x, np.float64)
    mant, exp = np.frexp(x)                      # x = mant * 2^exp, |mant| in [0.5, 1)
    quantum_exp = np.maximum(exp - 8, -133)       # BF16 subnormal spacing is 2^-133
    out = np.ldexp(np.rint(np.ldexp(x, -quantum_exp)), quantum_exp)
    out = np.where(np.abs(out) > 3.3895313892515355e38, np.copysign(np.inf, x), out)
    return np.where(x == 0, x, out)


def bf16_bits(x64) -> np.ndarray:
    """BF16 bit patterns of FP64 values that are already BF16-representable."""
    return (np.asarray(x64, np.float64).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def stage1(partials) -> np.ndarray:
    x = bf16_bits_to_f64(partials)               # [tp, m, H]
    return round_bf16(x.sum(axis=0))             # exact in FP64 for tp <= 8 and these ranges


def moe_fold(routed, idx, weights, shared) -> np.ndarray:
    routed = bf16_bits_to_f64(routed)            # [tp, rows, H]
    shared = bf16_bits_to_f64(shared)            # [tp, m, H]
    weights = np.asarray(weights, np.float64)    # [m, K]
    tp, m, k = idx.shape
    total = np.zeros(shared.shape[1:], np.float64)
    for r in range(tp):
        acc = np.zeros_like(total)
        for kk in range(k):
            rows = idx[r, :, kk]
            held = rows >= 0
            acc[held] += routed[r, rows[held]] * weights[held, kk][:, None]
        total += round_bf16(acc + shared[r])
    return round_bf16(total)


def post_mix(y64, residual, post, comb) -> np.ndarray:
    res = bf16_bits_to_f64(residual)             # [m, 4, H]
    post = np.asarray(post, np.float64).reshape(-1, HC)
    comb = np.asarray(comb, np.float64)          # [m, source, target]
    mixed = y64[:, None, :] * post[:, :, None] + np.einsum("mkh,mkj->mjh", res, comb)
    return round_bf16(mixed)                      # [m, 4, H]


def prenorm(new64, hc_fn):
    m, _, hidden = new64.shape
    flat = new64.reshape(m, HC * hidden)
    raw = flat @ np.asarray(hc_fn, np.float64)
    ss = (flat * flat).sum(axis=1)
    return raw, ss


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def mixes_and_pre(raw, ss, scale, base, hidden, rms_eps, hc_eps):
    rstd = 1.0 / np.sqrt(ss / (HC * hidden) + rms_eps)
    mixes = raw * rstd[:, None]
    pre = sigmoid(mixes[:, :HC] * scale[0] + base[:HC]) + hc_eps
    return mixes, pre


def post_from_mixes(mixes, scale, base, post_mult):
    return sigmoid(mixes[:, HC:2 * HC] * scale[1] + base[HC:2 * HC]) * post_mult


def sinkhorn(mixes, scale, base, eps, repeat):
    c = (mixes[:, 2 * HC:] * scale[2] + base[2 * HC:]).reshape(-1, HC, HC)
    c = np.exp(c - c.max(axis=2, keepdims=True))
    c = c / c.sum(axis=2, keepdims=True) + eps
    for it in range(repeat):
        if it > 0:
            c = c / (c.sum(axis=2, keepdims=True) + eps)
        c = c / (c.sum(axis=1, keepdims=True) + eps)
    return c


def collapse_norm(new64, pre, gamma, hidden, norm_eps):
    c = round_bf16(np.einsum("mjh,mj->mh", new64, pre))
    inv = 1.0 / np.sqrt((c * c).sum(axis=1) / hidden + norm_eps)
    return round_bf16(c * inv[:, None] * bf16_bits_to_f64(gamma)[None, :])


def boundary(problem, inputs: dict, *, moe: bool = False) -> dict:
    p = problem
    if moe:
        y = moe_fold(inputs["routed"], inputs["idx"], inputs["weights"], inputs["shared"])
    else:
        y = stage1(inputs["partials"])
    new = post_mix(y, inputs["residual"], inputs["post"], inputs["comb"])
    raw, ss = prenorm(new, inputs["hc_fn"])
    scale = np.asarray(inputs["scale"], np.float64)
    base = np.asarray(inputs["base"], np.float64)
    mixes, pre = mixes_and_pre(raw, ss, scale, base, p.hidden, p.rms_eps, p.hc_eps)
    out = collapse_norm(new, pre, inputs["gamma"], p.hidden, p.norm_eps)
    return {
        "reduced": y, "residual_out": new, "mixes": mixes, "pre": pre,
        "layer_input": out,
        "post_out": post_from_mixes(mixes, scale, base, p.post_mult),
        "comb_out": sinkhorn(mixes, scale, base, p.hc_eps, p.sinkhorn_repeat),
    }
