"""The pins must fail when a plausible mistake is planted in the oracle (CPU only).

Each case monkeypatches one oracle function with a wrong variant (a flipped sign, a dropped
term, a transposed pairing, a patch that is rotated too, a double rounding, an off-by-one
slot) and checks that at least one pin in tests/test_oracle_pins.py then fails.
"""
import numpy as np
import pytest

from oracle import kamera_oracle as ora
from tests import test_oracle_pins as pins


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def wrong_sign_rotate(x, delta, theta, style):
    return ora_rotate_orig(x, -delta, theta, style)


def dropped_term_rotate(x, delta, theta, style):
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    if delta == 0:
        return out
    d = x.shape[-1]
    phi = float(delta) * ora.inv_freq(theta, d)
    c, s = np.cos(phi), np.sin(phi)
    ia, ib = ora.rope_pairs(d, style)
    a, b = x[..., ia], x[..., ib]
    out[..., ia] = a * c            # "- b sin φ" dropped
    out[..., ib] = b * c + a * s
    return out


def swapped_pairs(d, style):
    k = np.arange(d // 2)
    if style == ora.NEOX_HALF:      # interleaved pairing where NeoX-half is meant
        return 2 * k, 2 * k + 1
    return k, k + d // 2


def wrong_freq(theta, d):
    i = np.arange(d // 2, dtype=np.float64)
    return np.power(float(theta), -1.0 * i / d)   # exponent -i/d instead of -2i/d


def double_rounding(x):
    return ora_f64_to_bf16_orig(np.asarray(x, np.float64).astype(np.float32).astype(np.float64))


def off_by_one_slot(page_table, req, tok, page_size):
    return int(page_table[req][tok // page_size]) * page_size + (tok + 1) % page_size


ora_rotate_orig = ora.rotate_band
ora_f64_to_bf16_orig = ora.f64_to_bf16


CASES = [
    ("rotate_band", wrong_sign_rotate, [pins.test_rotation_equals_complex_multiplication,
                                        pins.test_pair_zero_turns_by_exactly_delta]),
    ("rotate_band", dropped_term_rotate, [pins.test_inverse_and_norm_preservation,
                                          pins.test_rotation_equals_complex_multiplication]),
    ("rope_pairs", swapped_pairs, [pins.test_rotation_equals_complex_multiplication]),
    ("inv_freq", wrong_freq, [pins.test_inv_freq_closed_forms,
                              pins.test_rotation_equals_complex_multiplication]),
    ("f64_to_bf16", double_rounding, [pins.test_bf16_ties_to_even_and_single_rounding]),
    ("slot_of", off_by_one_slot, [pins.test_slots_match_independent_page_expansion,
                                  pins.test_identity_mode_scatter_is_byte_exact]),
]


@pytest.mark.parametrize("name,bad,checks", CASES, ids=[f"{c[0]}-{c[1].__name__}" for c in CASES])
def test_planted_mistake_is_caught(monkeypatch, name, bad, checks):
    monkeypatch.setattr(ora, name, bad)
    caught = [c.__name__ for c in checks if _fails(c)]
    assert caught, f"no pin caught the planted {bad.__name__}"


def test_transposed_patch_is_caught(monkeypatch):
    def transposed_vt(layout, vt_layer, m, g):
        _, _, (w0, w1) = ora.widths(layout)
        w = w0 if g == 0 else w1
        off = 0 if g == 0 else m * w0
        # reads the factor as [W][m] (V_m instead of V_mᵀ)
        return np.asarray(vt_layer)[off: off + m * w].reshape(w, m).T
    monkeypatch.setattr(ora, "vt_of_group", transposed_vt)
    assert _fails(pins.test_patch_by_pure_python_sums) or \
        _fails(pins.test_full_rank_patch_reconstructs_conditioned_kv)


def test_rotated_patch_is_caught(monkeypatch):
    orig = ora.reuse_layer

    def patch_then_rotate(layout, item, layer, channel, tokens=None):
        # adds the patch before the rotation, so the patch gets rotated too
        from types import SimpleNamespace
        unrot = SimpleNamespace(**{**vars(item), "delta": 0})
        vals, mask = orig(layout, unrot, layer, channel, tokens)
        if channel == 0 and item.delta != 0:
            for c0, d in ora.rope_bands(layout):
                vals[:, c0:c0 + d] = ora.rotate_band(vals[:, c0:c0 + d], item.delta,
                                                     layout.rope_theta, layout.rope_style)
                mask[c0:c0 + d] = False
        return vals, mask
    monkeypatch.setattr(ora, "reuse_layer", patch_then_rotate)
    assert _fails(pins.test_patch_added_after_rotation_not_rotated) or \
        _fails(pins.test_full_rank_patch_reconstructs_conditioned_kv)
