"""The pins must fail when a plausible mistake is planted in the oracle (CPU only).

Each case monkeypatches one oracle function with a wrong variant and checks that at least one
pin in tests/test_oracle_pins.py then fails. The variants: a flipped sign, a dropped term, a
transposed pairing, a patch that is rotated too, a double rounding, an off-by-one slot, M-RoPE
offsets or sections taken wrongly, a re-anchoring position of the wrong sign or with its
coordinates reversed, attention without its scale, an unnormalised split merge, singular
values in ascending order, the opposite sign convention, an error scale built from the product
of the factor sums or counting a turned pair twice, a re-anchoring that skips the values, a
bf16 spacing that is wrong at zero or one bit short, a patch range that takes in its end
layer, the factors of the next layer, a survivor turned by -δ, an in-place patch that ignores
its sign, query heads dealt to KV heads round-robin instead of in groups, MLA's rotation
applied to the latent instead of k_pe, every column rounded instead of the untouched ones
copied, and the deficit taken the wrong way round.
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


def offsets_ignore_sections(layout, item, npairs):
    return int(item.delta)            # every pair turns by δ_t, the h and w offsets dropped


def sections_off_by_one(npairs, sections, style):
    s_t, s_h, s_w = (int(v) for v in sections)
    if style == ora.MROPE_CONTIGUOUS:  # the t section one pair too long
        return np.array([0] * (s_t + 1) + [1] * (s_h - 1) + [2] * s_w)
    return ora_axes_orig(npairs, sections, style)


def token_offsets_wrong_sign(layout, position, npairs):
    off = ora_token_offsets_orig(layout, position, npairs)
    return -off if np.ndim(off) == 0 else [-v for v in off]


def token_offsets_reversed_coords(layout, position, npairs):
    if not ora.has_mrope(layout):
        return int(position)
    return ora_token_offsets_orig(layout, list(position)[::-1], npairs)  # (w, h, t) for (t, h, w)


def attend_without_scale(k, v, q, scale):
    return ora_attend_orig(k, v, q, 1.0)


def merge_unnormalised(parts):
    lses = np.array([l for _, l in parts], dtype=np.float64)
    m = np.max(lses)
    w = np.exp(lses - m)
    o = sum(wi * np.asarray(oi, np.float64) for wi, (oi, _) in zip(w, parts))  # no / sum(w)
    return o, m + np.log(np.sum(w))


def randomized_ascending(delta, omega, m, q):
    # eigenvalues taken in ascending order: the smallest directions of the sketch
    a = np.asarray(delta, np.float64)
    q_, _ = np.linalg.qr(a @ np.asarray(omega, np.float64))
    for _ in range(q):
        z, _ = np.linalg.qr(a.T @ q_)
        q_, _ = np.linalg.qr(a @ z)
    bt = a.T @ q_
    lam, ut = np.linalg.eigh(bt.T @ bt)
    sig = np.sqrt(np.maximum(lam[:m], 0.0))
    us = (q_ @ ut[:, :m]) * sig[None, :]
    with np.errstate(divide="ignore", invalid="ignore"):
        vt = np.where(sig[:, None] > 0, (bt @ ut[:, :m]).T / sig[:, None], 0.0)
    return us, vt, sig


def sign_rows_flipped(us, vt):
    us, vt = ora_sign_rows_orig(us, vt)
    return -us, -vt                   # the largest entry of each row made negative


def magnitude_product_of_sums(layout, item, layer, channel, tokens=None):
    # Σ_j|U_tj| · Σ_j|Vt_jc| in place of Σ_j |U_tj · Vt_jc| for the patch term
    mag = ora_magnitude_orig(layout, ora.as_item(**{**vars(item), "patch_m": 0}), layer, channel,
                             tokens)
    if ora.layer_patched(item, layer):
        li = layer - item.patch_l0
        for c0, w, g in ora.channel_groups(layout, channel):
            u = np.abs(ora.factor_f64(item.patch_u[li][g]))
            vt = np.abs(ora.factor_f64(ora.vt_of_group(layout, item.patch_vt[li], item.patch_m, g)))
            mag[:, c0:c0 + w] += u.sum(axis=1, keepdims=True) * vt.sum(axis=0, keepdims=True)
    return mag


def magnitude_pair_twice(layout, item, layer, channel, tokens=None):
    # |x| kept and |a| + |b| added on top for turned pairs (the element counted twice)
    mag = ora_magnitude_orig(layout, item, layer, channel, tokens)
    if channel == 0 and ora.item_rotates(layout, item):
        canon = np.asarray(item.canon_k[layer])
        x = np.abs(ora.bf16_to_f64(canon if tokens is None else canon[np.asarray(tokens)]))
        for c0, d in ora.rope_bands(layout):
            mag[:, c0:c0 + d] += x[:, c0:c0 + d]
    return mag


def ulp_from_frexp_alone(y):
    ay = np.abs(np.asarray(y, dtype=np.float64))
    _, E = np.frexp(ay)                      # zero is taken as if it were in [0.5, 1)
    return np.ldexp(1.0, np.maximum(E - 1, -126) - 7)


def ulp_one_bit_short(y):
    return 2.0 * ora_ulp_orig(y)             # the spacing of a 7-bit significand


def reanchor_skips_values(layout, item, k_pool, v_pool, page_table):
    ora_apply_reanchor_orig(layout, item, k_pool, None, page_table)


def patched_through_l1(item, layer):
    return item.patch_m > 0 and item.patch_l0 <= layer <= item.patch_l1


def factors_of_the_next_layer(layout, item, layer, channel, tokens=None):
    from types import SimpleNamespace
    if item.patch_m > 0 and item.patch_l1 - item.patch_l0 > 1:
        pu, pv = list(item.patch_u), list(item.patch_vt)
        item = SimpleNamespace(**{**vars(item), "patch_u": pu[1:] + pu[:1],
                                  "patch_vt": pv[1:] + pv[:1]})
    return ora_reuse_layer_orig(layout, item, layer, channel, tokens)


def relocate_backwards(layout, k_pool, page_table, req, start_tok, num_tokens, delta):
    ora_relocate_orig(layout, k_pool, page_table, req, start_tok, num_tokens, -delta)


def patch_inplace_ignores_sign(layout, k_pool, v_pool, page_table, req, start_tok, num_tokens,
                               patch_u, patch_vt, m, l0, l1, sign=1):
    ora_patch_inplace_orig(layout, k_pool, v_pool, page_table, req, start_tok, num_tokens,
                           patch_u, patch_vt, m, l0, l1, 1)


def heads_round_robin(layout, h, num_q_heads):
    if layout.kind == ora.GQA:      # head h to KV head h % H_kv instead of h // (H_q / H_kv)
        c0 = (h % layout.num_kv_heads) * layout.head_dim
        return (c0, layout.head_dim), (c0, layout.head_dim), 1
    return ora_head_columns_orig(layout, h, num_q_heads)


def bands_on_the_latent(layout):
    if layout.kind == ora.MLA:      # the first rope_dim columns of the row: the c_KV latent
        return [(0, layout.rope_dim)]
    return ora_rope_bands_orig(layout)


def every_column_rounded(layout, item, layer, channel, tokens=None):
    vals, _ = ora.reuse_layer(layout, item, layer, channel, tokens)
    return ora.f64_to_bf16(vals)    # no byte copy where nothing is computed


def deficit_reversed(kv_cond, kv_solo_relocated, m):
    return ora_form_patch_orig(kv_solo_relocated, kv_cond, m)


ora_rotate_orig = ora.rotate_band
ora_magnitude_orig = ora.magnitude_layer
ora_apply_reanchor_orig = ora.apply_reanchor
ora_f64_to_bf16_orig = ora.f64_to_bf16
ora_axes_orig = ora.mrope_pair_axes
ora_token_offsets_orig = ora.token_offsets
ora_attend_orig = ora.attend
ora_sign_rows_orig = ora._sign_rows
ora_ulp_orig = ora.bf16_ulp
ora_reuse_layer_orig = ora.reuse_layer
ora_relocate_orig = ora.relocate
ora_patch_inplace_orig = ora.patch_inplace
ora_head_columns_orig = ora.head_columns
ora_rope_bands_orig = ora.rope_bands
ora_form_patch_orig = ora.form_patch


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
    ("pair_offsets", offsets_ignore_sections,
     [lambda: pins.test_mrope_pair_turns_by_its_section_offset(ora.MROPE_CONTIGUOUS,
                                                               (16, 24, 24))]),
    ("mrope_pair_axes", sections_off_by_one, [pins.test_mrope_sections_match_printed_counts]),
    ("token_offsets", token_offsets_wrong_sign,
     [pins.test_reanchor_turns_each_token_by_its_own_position]),
    ("token_offsets", token_offsets_reversed_coords, [pins.test_reanchor_mrope_coordinates]),
    ("attend", attend_without_scale, [pins.test_attention_closed_forms,
                                      pins.test_decode_attention_gathers_heads_and_pages]),
    ("lse_merge", merge_unnormalised, [pins.test_attention_of_a_union_is_the_lse_merge_of_its_parts]),
    ("form_patch_randomized", randomized_ascending,
     [pins.test_randomized_patch_recovers_an_exactly_low_rank_deficit,
      pins.test_randomized_patch_residual_near_the_eckart_young_optimum]),
    ("_sign_rows", sign_rows_flipped,
     [pins.test_randomized_patch_recovers_an_exactly_low_rank_deficit]),
    ("magnitude_layer", magnitude_product_of_sums,
     [lambda: pins.test_magnitude_scale_by_explicit_loops("gqa", ora.NEOX_HALF, 0),
      lambda: pins.test_magnitude_scale_by_explicit_loops("mla", ora.NEOX_HALF, 31)]),
    ("magnitude_layer", magnitude_pair_twice,
     [lambda: pins.test_magnitude_scale_by_explicit_loops("gqa", ora.NEOX_HALF, 777)]),
    ("apply_reanchor", reanchor_skips_values, [pins.test_reanchored_items_land_at_their_slots]),
    ("slot_of", off_by_one_slot, [pins.test_reanchored_items_land_at_their_slots]),
    ("bf16_ulp", ulp_from_frexp_alone, [pins.test_bf16_ulp_is_the_gap_to_the_next_pattern]),
    ("bf16_ulp", ulp_one_bit_short, [pins.test_bf16_ulp_is_the_gap_to_the_next_pattern]),
    ("layer_patched", patched_through_l1, [pins.test_layers_outside_the_patch_range_are_unpatched]),
    ("reuse_layer", factors_of_the_next_layer, [pins.test_patch_by_pure_python_sums,
                                                pins.test_mla_kpe_band_gets_its_own_patch_group]),
    ("relocate", relocate_backwards, [pins.test_relocate_in_place_rotates_only_rope_columns]),
    ("patch_inplace", patch_inplace_ignores_sign,
     [pins.test_patch_inplace_sign_symmetry_and_pure_python_sums,
      pins.test_patch_add_then_remove_is_within_two_roundings]),
    ("head_columns", heads_round_robin, [pins.test_decode_attention_gathers_heads_and_pages]),
    ("rope_bands", bands_on_the_latent, [pins.test_mla_latent_copied_byte_exact_and_only_kpe_turns,
                                         pins.test_layout_reading_matches_printed_shapes]),
    ("reuse_layer_bits", every_column_rounded, [pins.test_delta_zero_rank_zero_is_bitwise_identity]),
    ("form_patch", deficit_reversed, [pins.test_full_rank_patch_reconstructs_conditioned_kv,
                                      pins.test_eckart_young_residual]),
]


@pytest.mark.parametrize("name,bad,checks", CASES, ids=[f"{c[0]}-{c[1].__name__}" for c in CASES])
def test_planted_mistake_is_caught(monkeypatch, name, bad, checks):
    monkeypatch.setattr(ora, name, bad)
    caught = [getattr(c, "__name__", "pin") for c in checks if _fails(c)]
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
