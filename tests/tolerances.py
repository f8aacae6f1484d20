"""Comparison helpers shared by the oracle and GPU parity tests.

Tolerances (derived from the arithmetic; the parity bar of each output):

* stage-1 sum and MoE fold (``reduced``): bit-exact -- both sides add the
  same FP32 values in the same rank / route order with IEEE rounding.
* post-mixed streams: at most 2 BF16 ulp (both sides take the same multiply
  and four fused multiply-adds, so they are normally bit-identical).
* layer input: at most 2 BF16 ulp, the ulp taken at
  max(|ref|, 2^-8 * T), where T is the largest of the four collapse terms
  |new_j * pre_j| after normalisation (times |gamma|).  pre comes out of an
  FP32 reduction of 4H products whose order differs between the two sides,
  so it agrees only to ~1e-7 relative; where the collapse cancels to below
  1/256 of its largest term, that difference is amplified more than 256x
  relative to the result and a plain 2-ulp bound at |ref| would be a bound on
  the summation order, not on the method.
  The floor is meant for rare cancelling elements: the parity tests count
  the elements that exceed 2 ulp at |ref| and pass only through the floor,
  and require that count to stay at most FLOOR_ONLY_FRACTION of the
  elements (at least FLOOR_ONLY_MIN, for the few-element edge cases).  For
  N(0, 1) streams the estimate is about 1e-5: a 1e-7 relative difference of
  pre moves c by more than 2 ulp of |c| only where |c| < T / 80000.
* pre / post / comb (FP32): relative 1e-4, absolute floor 1e-6.
* raw mixes (FP32, before the sigmoid): relative 1e-4, absolute floor 1e-5
  (the mixes are ~N(0, 1) and carry the FP32 reduction-order error).
"""
import numpy as np

HC = 4


def f32(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def ulp_diff(a, b):
    """|a - b| in BF16 ulps (order-preserving integer map of the patterns)."""
    def key(x):
        x = np.asarray(x, np.uint16).astype(np.int64)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7fff), 0x8000 + x)
    return np.abs(key(a) - key(b))


def bf16_ulp(x):
    """Spacing of BF16 numbers at |x| (8 significant bits)."""
    x = np.abs(np.asarray(x, np.float64))
    _, e = np.frexp(np.maximum(x, 2.0 ** -126))
    return np.ldexp(1.0, e - 8)


def collapse_scale(streams, pre, gamma):
    """T of the layer-input tolerance: largest |new_j * pre_j| of each element
    times inv_rms * |gamma| (inv_rms from the collapse itself)."""
    new = f32(streams).astype(np.float64)                        # [m, 4, H]
    p = np.asarray(pre, np.float64)[:, :, None]
    terms = np.abs(new * p)
    c = (new * p).sum(axis=1)
    inv = 1.0 / np.sqrt((c * c).mean(axis=1) + 1e-30)
    return terms.max(axis=1) * inv[:, None] * np.abs(f32(gamma).astype(np.float64))[None, :]


def layer_input_ok(got, ref, streams, pre, gamma, floor=2.0 ** -8, ulps=2, scale=None):
    """Boolean mask of elements within the layer-input tolerance (`scale`:
    collapse_scale(streams, pre, gamma) if already computed)."""
    g = f32(got).astype(np.float64)
    r = f32(ref).astype(np.float64)
    t = collapse_scale(streams, pre, gamma) if scale is None else scale
    at = np.maximum(np.abs(r), floor * t)
    return np.abs(g - r) <= ulps * bf16_ulp(at)


FLOOR_ONLY_FRACTION = 1e-4
FLOOR_ONLY_MIN = 2


def floor_use(got, ref, streams, pre, gamma, ulps=2):
    """How the layer-input tolerance was met: the number of elements beyond
    `ulps` ulp at |ref| that pass only through the cancellation floor, their
    largest ulp difference and the largest T / |ref| among them."""
    t = collapse_scale(streams, pre, gamma)
    ok = layer_input_ok(got, ref, streams, pre, gamma, ulps=ulps, scale=t)
    plain = layer_input_ok(got, ref, streams, pre, gamma, floor=0.0, ulps=ulps, scale=t)
    only = ok & ~plain
    n = int(only.sum())
    rep = {"elements": int(ok.size), "floor_only": n, "floor_only_max_ulp": 0, "floor_only_worst_t_over_ref": 0.0}
    if n:
        rep["floor_only_max_ulp"] = int(ulp_diff(got, ref)[only].max())
        r = np.abs(f32(ref).astype(np.float64))
        rep["floor_only_worst_t_over_ref"] = float((t[only] / np.maximum(r[only], 1e-30)).max())
    return rep


def floor_use_allowed(rep):
    return rep["floor_only"] <= max(FLOOR_ONLY_FRACTION * rep["elements"], FLOOR_ONLY_MIN)


def close_f32(got, ref, rtol, atol):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return np.abs(got - ref) <= atol + rtol * np.abs(ref)
