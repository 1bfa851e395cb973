"""Planted mistakes in the oracle must be caught by its pins.

Each mutant is a copy of the oracle's source with one plausible slip (a dropped
term, a wrong sign or index, a transposed operand, a wrong order of steps).  The
whole pin suite runs against the mutant on the CPU and at least one pin must
fail.  This is what shows the pins are strong enough to trust the oracle.
"""
import os
import types

import pytest

import oracle
from tests import oracle_pins

SRC_PATH = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.py")

MUTANTS = [
    ("bit stream read big-endian", 'axis=-1, bitorder="little")', 'axis=-1, bitorder="big")'),
    ("code bits reversed", "(digits << np.arange(bits, dtype=np.int64))",
     "(digits << np.arange(bits, dtype=np.int64)[::-1])"),
    ("code width ignored", "n = stream.shape[-1] // bits\n", "bits = 4\n    n = stream.shape[-1] // bits\n"),
    ("dequant drops bias", "return s_full * q + b_full", "return s_full * q"),
    ("group index k % groups", "s_full = np.repeat(s, group, axis=-1)", "s_full = np.tile(s, group)"),
    ("bias leaks into weights", "w = s[ids]", "w = keys[ids]"),
    ("normalise after scaling",
     "    w = w * float(spec.routed_scale)\n    return ids, w",
     "    w = w * float(spec.routed_scale)\n    if spec.renormalize:\n        w = w / w.sum()\n"
     "    return ids, w"),
    ("ties to the higher index", "(0, -keys[e], e)", "(0, -keys[e], -e)"),
    ("non-finite keys first", "else (1, 0.0, e)", "else (-1, 0.0, e)"),
    ("relu instead of relu^2", "return r * r", "return r"),
    ("silu dropped", "return (g / (1.0 + np.exp(-g))) * u", "return g * u"),
    ("silu sign", "return (g / (1.0 + np.exp(-g))) * u", "return (g / (1.0 + np.exp(g))) * u"),
    ("gate and up swapped", "h = activation(cache.spec, u, g)", "h = activation(cache.spec, g, u) if g is not None else activation(cache.spec, u, g)"),
    ("fc2 replaced by fc1 transposed", "r = W2 @ y if sp.latent else y", "r = W1.T @ y if sp.latent else y"),
    ("fc1 replaced by fc2 transposed", "xin = W1 @ xt if sp.latent else xt", "xin = W2.T @ xt if sp.latent else xt"),
    ("residual dropped", "out[t] = xt + r + shared_output(layer, xt)", "out[t] = r + shared_output(layer, xt)"),
    ("shared expert dropped", "out[t] = xt + r + shared_output(layer, xt)", "out[t] = xt + r"),
    ("combine weights dropped", "y = y + w[j] * expert_output(cache, int(ids[j]), xin)",
     "y = y + expert_output(cache, int(ids[j]), xin)"),
    ("softmax not renormalised", "denom = ez[ids].sum() if spec.renormalize else ez.sum()", "denom = ez.sum()"),
    ("sigmoid sign", "return 1.0 / (1.0 + np.exp(-z))", "return 1.0 / (1.0 + np.exp(z))"),
    ("selection ignores the bias", "s = s + np.asarray(bias, dtype=np.float64)", "s = s"),
    ("last pick dropped", "for j in range(k):", "for j in range(k - 1):"),
    ("margin one rank too low", "return float(srt[k - 1] - srt[k])", "return float(srt[k] - srt[k + 1])"),
    ("margin one rank too high", "return float(srt[k - 1] - srt[k])", "return float(srt[k - 2] - srt[k - 1])"),
    ("margin on the logits", "keys = selection_keys(z, spec, bias)\n    k = spec.top_k",
     "keys = np.asarray(z, dtype=np.float64)\n    k = spec.top_k"),
    ("margin ranks NaN first", "ranked = np.where(np.isfinite(keys), keys, -np.inf)",
     "ranked = np.where(np.isnan(keys), np.inf, keys)"),
    ("margin zero past the finite keys", "return math.inf if srt[k - 1] > -np.inf else 0.0",
     "return 0.0"),
    ("shared gate/up swapped", "    h = activation(sp, u, g)\n    return widen(layer.sh_down, dt) @ h",
     "    h = activation(sp, g, u) if g is not None else activation(sp, u, g)\n"
     "    return widen(layer.sh_down, dt) @ h"),
    ("E2M1 exponent bias dropped", "np.exp2(ef - 1.0) * (1.0 + 0.5 * mf)", "np.exp2(ef) * (1.0 + 0.5 * mf)"),
    ("E2M1 subnormal as normal", "mag = np.where(ef == 0, 0.5 * mf, ", "mag = np.where(ef < 0, 0.5 * mf, "),
    ("E2M1 sign ignored", "    return np.where(sign == 1, -mag, mag)\n\n\ndef e4m3_values",
     "    return mag\n\n\ndef e4m3_values"),
    ("E2M1 exponent bits swapped", "ef = (c >> 2 & 1) * 2 + (c >> 1 & 1)", "ef = (c >> 1 & 1) * 2 + (c >> 2 & 1)"),
    ("E4M3 exponent bias 8", "(1.0 + mf / 8.0) * np.exp2(ef - 7.0)", "(1.0 + mf / 8.0) * np.exp2(ef - 8.0)"),
    ("E4M3 subnormal off by a power of two", "(mf / 8.0) * 2.0 ** -6", "(mf / 8.0) * 2.0 ** -7"),
    ("E4M3 mantissa of 4 bits", "mf = v & 7\n", "mf = v & 15\n"),
    ("NVFP4 blocks of 32", "np.repeat(s, 16, axis=-1) * float", "np.repeat(s, 32, axis=-1)[..., : q.shape[-1]] * float"),
    ("E8M0 bias 128", "np.exp2(v - 127.0))", "np.exp2(v - 128.0))"),
    ("MXFP4 blocks of 16", "q * np.repeat(s, 32, axis=-1)", "q * np.repeat(s, 16, axis=-1)[..., : q.shape[-1]]"),
    ("E8M0 NaN at zero", "np.where(v == 255, np.nan", "np.where(v == 0, np.nan"),
    ("NVFP4 matrix scale dropped", "return q * np.repeat(s, 16, axis=-1) * float(np.float32(matrix_scale))",
     "return q * np.repeat(s, 16, axis=-1)"),
]


def _mutant_module(old, new):
    src = open(SRC_PATH).read()
    assert src.count(old) == 1, f"snippet not unique in the oracle: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    mod.__file__ = SRC_PATH
    exec(compile(src.replace(old, new), SRC_PATH + " (mutant)", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new):
    mod = _mutant_module(old, new)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mod)
        except Exception as exc:  # an assertion or a crash both count as caught
            failed.append((pin.__name__, type(exc).__name__))
    assert failed, f"no pin caught the planted mistake: {name}"


def test_unmutated_copy_passes():
    """The same exec path with no change passes every pin (the harness itself
    does not make pins fail)."""
    mod = _mutant_module("import math", "import math")
    for pin in oracle_pins.ALL_PINS:
        pin(mod)
