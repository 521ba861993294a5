"""Plants plausible mistakes in the oracle (on the CPU, one at a time) and
checks that its pins catch each one: a pin that cannot fail proves nothing."""
import numpy as np
import pytest

import oracle
import oracle.nvfp4_ref as R
from tests import test_oracle as P


def _set(mp, name, fn):
    """Patch the oracle module and the package's re-export alike."""
    mp.setattr(R, name, fn)
    if hasattr(oracle, name):
        mp.setattr(oracle, name, fn)


def _ties_away(mag, values, codes):
    mag = np.asarray(mag, dtype=np.float64)
    n = len(values)
    hi = np.clip(np.searchsorted(values, mag, side="left"), 0, n - 1)
    lo = np.clip(hi - 1, 0, n - 1)
    take_hi = (values[hi] - mag) <= (mag - values[lo])
    return np.where(take_hi, codes[hi], codes[lo])


def _pack_swapped(codes):
    c = np.asarray(codes, dtype=np.uint8)
    return (c[:, 1::2] | (c[:, 0::2] << 4)).astype(np.uint8)


def _e4m3_bias8(code):
    c = np.asarray(code, dtype=np.int64) & 0xFF
    e, m = (c >> 3) & 0xF, c & 7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -7), np.ldexp(1.0 + m / 8.0, e - 8))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(((c >> 7) & 1) == 1, -mag, mag)


def _e2m1_no_signed_zero(q):
    q = np.asarray(q, dtype=np.float32)
    mag = R._nearest_even(np.abs(q).astype(np.float64), R._E2M1_POS_VALUES, R._E2M1_POS_CODES)
    return (mag | (((q < 0) & (mag > 0)).astype(np.int64) << 3)).astype(np.uint8)


def _tensor_scale_448(x):
    x = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0)
    return np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(448.0))


def _gemm_drops_tensor_scale(x, w):
    return np.asarray(x, dtype=np.float64) @ (R.decode(w) / np.float64(w.s_t)).T


def _route_renormalised(logits, topk):
    ids, w = _ORIG_ROUTE(logits, topk)
    return ids, w / w.sum(axis=1, keepdims=True)


_ORIG_ROUTE = R.moe_route


def _argmax_first_position(logits, rows):
    logits = np.asarray(logits, dtype=np.float64)
    pos = logits.argmax(axis=1)
    return np.asarray(rows)[pos], logits.max(axis=1)


def _moe_w4a4_mutant(quant_x=True, quant_h=True, per_expert_h=False, swap_gu=False):
    """The R10 layer with one planted mistake."""
    def f(x, ids, weights, w13, w2):
        x = np.asarray(x, dtype=np.float32)
        ids = np.asarray(ids)
        weights = np.asarray(weights, dtype=np.float64)
        xd = R.decode(R.quantize(x)) if quant_x else x.astype(np.float64)
        tok, slot = np.nonzero(ids >= 0)
        exp = ids[tok, slot]
        inter = w13[0].shape[0] // 2
        h = np.zeros((tok.size, inter))
        for e in np.unique(exp):
            r = np.nonzero(exp == e)[0]
            gu = xd[tok[r]] @ R.decode(w13[e]).T
            g, u = (gu[:, inter:], gu[:, :inter]) if swap_gu else (gu[:, :inter], gu[:, inter:])
            h[r] = R.bf16_round(R.silu(g) * u)
        if quant_h and not per_expert_h:
            h = R.decode(R.quantize(h.astype(np.float32)))
        out = np.zeros((x.shape[0], w2[0].shape[0]))
        for e in np.unique(exp):
            r = np.nonzero(exp == e)[0]
            he = R.decode(R.quantize(h[r].astype(np.float32))) if per_expert_h else h[r]
            np.add.at(out, tok[r], weights[tok[r], slot[r]][:, None] * (he @ R.decode(w2[e]).T))
        return out
    return f


def _golden_all():
    for blk in P.load_blocks():
        P.test_golden_block(blk)


MUTANTS = {
    "e2m1 ties away from zero": (
        lambda mp: _set(mp, "_nearest_even", _ties_away),
        [_golden_all, P.test_e2m1_encode_brute_force]),
    "nibbles swapped": (
        lambda mp: _set(mp, "pack_codes", _pack_swapped),
        [_golden_all]),
    "E4M3 bias 8": (
        lambda mp: _set(mp, "e4m3_value", _e4m3_bias8),
        [P.test_e4m3_decode_matches_torch_float8, P.test_e4m3_known_values]),
    "sign of zero dropped": (
        lambda mp: _set(mp, "e2m1_encode", _e2m1_no_signed_zero),
        [_golden_all, P.test_e2m1_encode_ties_and_signed_zero]),
    "tensor scale amax/448": (
        lambda mp: _set(mp, "tensor_scale", _tensor_scale_448),
        [P.test_tensor_scale_closed_form, P.test_largest_block_gets_scale_448_when_dynamic]),
    "GEMM drops s_t": (
        lambda mp: _set(mp, "gemm_w4a16", _gemm_drops_tensor_scale),
        [P.test_full_k16_code_enumeration_single_row]),
    "routing renormalised": (
        lambda mp: _set(mp, "moe_route", _route_renormalised),
        [P.test_route_matches_sorting]),
    "W4A4 MoE input not quantised": (
        lambda mp: _set(mp, "moe_forward_w4a4", _moe_w4a4_mutant(quant_x=False)),
        [P.test_moe_w4a4_sees_only_the_quantised_input]),
    "W4A4 MoE h not quantised": (
        lambda mp: _set(mp, "moe_forward_w4a4", _moe_w4a4_mutant(quant_h=False)),
        [P.test_moe_w4a4_is_near_the_w4a16_layer_on_the_quantised_input,
         P.test_moe_w4a4_h_scale_is_shared_by_all_routed_rows]),
    "W4A4 MoE h scale per expert": (
        lambda mp: _set(mp, "moe_forward_w4a4", _moe_w4a4_mutant(per_expert_h=True)),
        [P.test_moe_w4a4_h_scale_is_shared_by_all_routed_rows]),
    "W4A4 MoE gate and up swapped": (
        lambda mp: _set(mp, "moe_forward_w4a4", _moe_w4a4_mutant(swap_gu=True)),
        [P.test_moe_w4a4_is_near_the_w4a16_layer_on_the_quantised_input]),
    "argmax by first position": (
        lambda mp: _set(mp, "argmax_lowest_id", _argmax_first_position),
        [P.test_argmax_ties_go_to_lowest_vocab_id]),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    patch, pins = MUTANTS[name]
    patch(monkeypatch)
    caught = 0
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError):
            caught += 1
    assert caught > 0, f"no pin caught the planted mistake: {name}"
