"""Pins of the float64 oracle against what the Kamera pages and the mathematics fix.

Nothing here retypes the oracle's own formulas: rotations are checked against an explicit
dense rotation matrix built from scalar ``math`` calls and against complex multiplication,
the patch against pure-Python sums and Eckart–Young (with singular values taken from an
eigen-decomposition, not the SVD the oracle calls), rounding against brute-force neighbour
search and torch's float32 -> bf16 conversion, slots against an independent page expansion,
and the layout against the shapes printed on the pages (tests/golden/).
"""
import cmath
import math
import os

import numpy as np
import pytest
import torch

from oracle import kamera_oracle as ora

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def ns_layout(**kw):
    from types import SimpleNamespace
    base = dict(kind=ora.GQA, num_layers=1, page_size=4, num_kv_heads=1, head_dim=8,
                latent_dim=0, rope_dim=8, rope_style=ora.NEOX_HALF, rope_theta=1e4)
    base.update(kw)
    return SimpleNamespace(**base)


def rand_bf16_bits(shape, scale=1.0, rng=RNG):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------------------------------
# bf16 rounding
# ------------------------------------------------------------------------------------------

def test_bf16_known_bit_patterns():
    vals = [1.0, -2.0, 0.0, -0.0, math.inf, -math.inf, 3.3895313892515355e38, 2.0 ** -133,
            -(2.0 ** -126), 0.5]
    want = [0x3F80, 0xC000, 0x0000, 0x8000, 0x7F80, 0xFF80, 0x7F7F, 0x0001, 0x8080, 0x3F00]
    got = ora.f64_to_bf16(np.array(vals)).tolist()
    assert got == want
    assert ora.f64_to_bf16(np.array([math.nan]))[0] & 0x7FFF > 0x7F80


def test_bf16_ties_to_even_and_single_rounding():
    # exact halfway cases go to the even neighbour
    assert ora.f64_to_bf16(np.array([1 + 2 ** -8]))[0] == 0x3F80
    assert ora.f64_to_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 0x3F82
    # just above the halfway point: one rounding goes up; rounding through float32 first
    # would land exactly on the tie and then on the even value 1.0
    assert ora.f64_to_bf16(np.array([1 + 2 ** -8 + 2 ** -40]))[0] == 0x3F81
    assert ora.f64_to_bf16(np.array([-(1 + 2 ** -8 + 2 ** -40)]))[0] == 0xBF81
    # overflow: above max + half ulp is infinity, below stays max
    mx = 3.3895313892515355e38
    half_ulp = 2.0 ** 119
    assert ora.f64_to_bf16(np.array([mx + half_ulp]))[0] == 0x7F80
    assert ora.f64_to_bf16(np.array([mx + half_ulp * 0.99]))[0] == 0x7F7F


def test_bf16_matches_torch_on_float32_inputs():
    x = np.concatenate([RNG.standard_normal(50000) * 10.0 ** RNG.integers(-40, 38, 50000),
                        RNG.standard_normal(2000) * 1e-39,  # subnormal float32 range
                        RNG.standard_normal(2000)]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = ora.f64_to_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_bf16_nearest_by_brute_force_neighbours():
    y = RNG.standard_normal(4000) * 10.0 ** RNG.uniform(-30, 30, 4000)
    bits = ora.f64_to_bf16(y)
    got = ora.bf16_to_f64(bits)
    # the two neighbours of the chosen value, by stepping the bit pattern
    mag = bits & 0x7FFF
    up = ora.bf16_to_f64((bits & 0x8000) | np.minimum(mag + 1, 0x7F7F))
    dn = ora.bf16_to_f64((bits & 0x8000) | np.maximum(mag.astype(np.int32) - 1, 0).astype(np.uint16))
    err = np.abs(got - y)
    assert np.all(err <= np.abs(up - y))
    assert np.all(err <= np.abs(dn - y))
    # ties never occur for these draws; the chosen value is strictly nearest or equal
    assert np.all(err <= 0.5 * ora.bf16_ulp(got) * (1 + 1e-12))


def test_bf16_ulp_is_the_gap_to_the_next_pattern():
    """bf16_ulp(y) is the distance from y to the next larger bf16 value, found by stepping
    the bit pattern, for every finite non-negative bf16 value including zero and the
    subnormals; negative values take their magnitude's spacing."""
    bits = np.arange(0x0000, 0x7F7F, dtype=np.uint32).astype(np.uint16)
    y = ora.bf16_to_f64(bits)
    nxt = ora.bf16_to_f64((bits + 1).astype(np.uint16))
    np.testing.assert_array_equal(ora.bf16_ulp(y), nxt - y)
    np.testing.assert_array_equal(ora.bf16_ulp(-y), nxt - y)
    assert ora.bf16_ulp(0.0) == 2.0 ** -133 and ora.bf16_ulp(1.0) == 2.0 ** -7


def test_bf16_decode_encode_roundtrip_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = ora.bf16_to_f64(bits)
    back = ora.f64_to_bf16(vals)
    ok = ~np.isnan(vals)
    np.testing.assert_array_equal(back[ok], bits[ok])


# ------------------------------------------------------------------------------------------
# RoPE relocation R(δ)
# ------------------------------------------------------------------------------------------

def dense_rotation(d, delta, theta, style):
    """Explicit d×d block rotation with 2×2 blocks [[c, -s], [s, c]] on each pair (the
    textbook RoPE of Su et al.: x1' = x1 cos - x2 sin, x2' = x2 cos + x1 sin), built from
    scalar math calls."""
    M = [[0.0] * d for _ in range(d)]
    for k in range(d // 2):
        phi = delta * math.pow(theta, -2.0 * k / d)
        c, s = math.cos(phi), math.sin(phi)
        if style == ora.NEOX_HALF:
            a, b = k, k + d // 2
        else:
            a, b = 2 * k, 2 * k + 1
        M[a][a], M[a][b] = c, -s
        M[b][a], M[b][b] = s, c
    return np.array(M)


@pytest.mark.parametrize("style", [ora.NEOX_HALF, ora.INTERLEAVED])
@pytest.mark.parametrize("d", [2, 4, 8])
@pytest.mark.parametrize("delta", [1, -7, 1000, 131071])
def test_rotation_equals_dense_matrix(style, d, delta):
    x = RNG.standard_normal((3, d))
    want = x @ dense_rotation(d, delta, 1e4, style).T
    got = ora.rotate_band(x, delta, 1e4, style)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_rotation_equals_complex_multiplication():
    d, theta = 16, 1e6
    x = RNG.standard_normal((5, d))
    for delta in (3, -576, 32768):
        got = ora.rotate_band(x, delta, theta, ora.NEOX_HALF)
        for t in range(5):
            for k in range(d // 2):
                z = complex(x[t, k], x[t, k + d // 2])
                w = z * cmath.exp(1j * delta * theta ** (-2.0 * k / d))
                assert abs(got[t, k] - w.real) < 1e-12
                assert abs(got[t, k + d // 2] - w.imag) < 1e-12


def test_inv_freq_closed_forms():
    np.testing.assert_allclose(ora.inv_freq(1e4, 4), [1.0, 0.01], rtol=1e-15)
    f = ora.inv_freq(1e6, 128)
    assert f[0] == 1.0 and len(f) == 64
    np.testing.assert_allclose(f[1:] / f[:-1], 1e6 ** (-2 / 128), rtol=1e-13)
    np.testing.assert_allclose(f[-1], 1e6 ** (-126 / 128), rtol=1e-13)


def test_pair_zero_turns_by_exactly_delta():
    # inv_freq_0 = 1: the first pair of a unit key turns by δ radians
    for style in (ora.NEOX_HALF, ora.INTERLEAVED):
        for delta in (1, -1, 1000, 131071, -131071):
            e = np.zeros(8)
            a, b = ora.rope_pairs(8, style)
            e[a[0]] = 1.0
            r = ora.rotate_band(e, delta, 1e4, style)
            assert abs(r[a[0]] - math.cos(delta)) < 1e-12
            assert abs(r[b[0]] - math.sin(delta)) < 1e-12


DELTAS = [0, 1, -1, 576, -576, 32768, -32768, 131071]


@pytest.mark.parametrize("style", [ora.NEOX_HALF, ora.INTERLEAVED])
def test_composition_identity(style):
    # R(δ) R(p) = R(p + δ)  (§1, §3: RoPE composes exactly)
    x = RNG.standard_normal((4, 64))
    for p in DELTAS:
        xp = ora.rotate_band(x, p, 1e4, style)
        for d in DELTAS:
            lhs = ora.rotate_band(xp, d, 1e4, style)
            rhs = ora.rotate_band(x, p + d, 1e4, style)
            np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-9)


def test_inverse_and_norm_preservation():
    x = RNG.standard_normal((4, 128))
    for d in DELTAS:
        y = ora.rotate_band(x, d, 1e6, ora.NEOX_HALF)
        np.testing.assert_allclose(ora.rotate_band(y, -d, 1e6, ora.NEOX_HALF), x, atol=1e-12)
        a, b = ora.rope_pairs(128, ora.NEOX_HALF)
        np.testing.assert_allclose(np.hypot(y[:, a], y[:, b]), np.hypot(x[:, a], x[:, b]),
                                   rtol=1e-13)


def test_relocation_from_bf16_storage_matches_direct_placement():
    # keys stored rotated at p (bf16), relocated by δ, against keys rotated directly to p+δ
    x = RNG.standard_normal((256, 128))
    for p, d in [(0, 1000), (5000, -576), (100, 131071 - 100)]:
        stored = ora.f64_to_bf16(ora.rotate_band(x, p, 1e4, ora.NEOX_HALF))
        moved = ora.f64_to_bf16(ora.rotate_band(ora.bf16_to_f64(stored), d, 1e4, ora.NEOX_HALF))
        direct = ora.rotate_band(x, p + d, 1e4, ora.NEOX_HALF)
        got = ora.bf16_to_f64(moved)
        rel = np.linalg.norm(got - direct) / np.linalg.norm(direct)
        assert rel < 2 ** -8
        # the storage rounding (at most half an ulp on each pair member) turns with the pair,
        # so each element may move by both halves; the final rounding adds half an ulp
        sv = ora.bf16_to_f64(stored)
        a, b = ora.rope_pairs(128, ora.NEOX_HALF)
        pair_err = 0.5 * (ora.bf16_ulp(sv[:, a]) + ora.bf16_ulp(sv[:, b]))
        bound = np.empty_like(direct)
        bound[:, a] = pair_err
        bound[:, b] = pair_err
        bound += 0.5 * ora.bf16_ulp(got)
        assert np.all(np.abs(got - direct) <= bound * (1 + 1e-9))


# ------------------------------------------------------------------------------------------
# the operator on items
# ------------------------------------------------------------------------------------------

def gqa_item(L=2, T=6, H=2, hd=8, m=0, l0=0, l1=0, delta=0, rng=RNG, float_factors=False):
    lay = ns_layout(num_layers=L, num_kv_heads=H, head_dim=hd, rope_dim=hd)
    W = H * hd
    k = rand_bf16_bits((L, T, W), rng=rng)
    v = rand_bf16_bits((L, T, W), rng=rng)
    pu = pv = None
    if m:
        if float_factors:
            pu = rng.standard_normal((l1 - l0, 2, T, m))
            pv = rng.standard_normal((l1 - l0, m * 2 * W))
        else:
            pu = rand_bf16_bits((l1 - l0, 2, T, m), rng=rng)
            pv = rand_bf16_bits((l1 - l0, m * 2 * W), 0.1, rng=rng)
    it = ora.as_item(canon_k=k, canon_v=v, patch_u=pu, patch_vt=pv, delta=delta, patch_m=m,
                     patch_l0=l0, patch_l1=l1)
    return lay, it


def test_delta_zero_rank_zero_is_bitwise_identity():
    lay, it = gqa_item(delta=0)
    # plant signed zeros and a NaN payload: a byte copy keeps them
    it.canon_k[0, 0, :4] = [0x8000, 0x0000, 0x8000, 0x7FC3]
    it.canon_v[1, 2, :2] = [0x8000, 0xFFC1]
    for layer in range(2):
        np.testing.assert_array_equal(ora.reuse_layer_bits(lay, it, layer, 0), it.canon_k[layer])
        np.testing.assert_array_equal(ora.reuse_layer_bits(lay, it, layer, 1), it.canon_v[layer])


def test_values_untouched_by_delta():
    # §3: V is untouched by relocation; with no patch the V bytes equal the stored ones
    lay, it = gqa_item(delta=12345)
    for layer in range(2):
        np.testing.assert_array_equal(ora.reuse_layer_bits(lay, it, layer, 1), it.canon_v[layer])
        assert not np.array_equal(ora.reuse_layer_bits(lay, it, layer, 0), it.canon_k[layer])


def test_patch_by_pure_python_sums():
    # δ = 0 isolates the patch: out[t][c] = x[t][c] + Σ_j U[t][j] Vt[j][c] per channel group
    lay, it = gqa_item(L=3, T=3, H=1, hd=4, m=2, l0=1, l1=3, delta=0)
    W = 4
    for layer in range(3):
        for ch in range(2):
            vals, _ = ora.reuse_layer(lay, it, layer, ch)
            canon = (it.canon_k if ch == 0 else it.canon_v)[layer]
            for t in range(3):
                for c in range(W):
                    want = float(ora.bf16_to_f64(canon[t, c]))
                    if 1 <= layer < 3:
                        li = layer - 1
                        for j in range(2):
                            u = float(ora.bf16_to_f64(it.patch_u[li, ch, t, j]))
                            vt = float(ora.bf16_to_f64(it.patch_vt[li, ch * 2 * W + j * W + c]))
                            want += u * vt
                    assert abs(vals[t, c] - want) <= 1e-12 * max(1.0, abs(want))


def test_layers_outside_the_patch_range_are_unpatched():
    # Eq. 1 adds U_m V_m^T only on the patched layers [l0, l1): the layers on either side are
    # the relocated canonical alone (the same item at rank zero), bit for bit. The factor
    # arrays hold an entry for every layer, so a boundary taken one layer off reads real
    # factors instead of failing to index them.
    from types import SimpleNamespace
    rng = np.random.default_rng(77)
    lay, it = gqa_item(L=4, T=5, H=1, hd=8, delta=777, rng=rng)
    m = 2
    it = SimpleNamespace(**{**vars(it), "patch_m": m, "patch_l0": 1, "patch_l1": 3,
                            "patch_u": rand_bf16_bits((4, 2, 5, m), rng=rng),
                            "patch_vt": rand_bf16_bits((4, m * 2 * 8), 0.5, rng=rng)})
    bare = SimpleNamespace(**{**vars(it), "patch_m": 0, "patch_l0": 0, "patch_l1": 0})
    for layer in range(4):
        for ch in range(2):
            got = ora.reuse_layer_bits(lay, it, layer, ch)
            ref = ora.reuse_layer_bits(lay, bare, layer, ch)
            if layer in (0, 3):
                np.testing.assert_array_equal(got, ref)
            else:
                assert not np.array_equal(got, ref), f"layer {layer} channel {ch} unpatched"


def test_full_rank_patch_reconstructs_conditioned_kv():
    # App. A: Δ = KV(B|A) - R(δ)KV(B|∅); the patch from the full SVD of Δ added after the
    # rotation gives back KV(B|A) exactly (float64).
    T, H, hd = 12, 2, 8
    W = H * hd
    delta = 777
    lay, it = gqa_item(L=1, T=T, H=H, hd=hd, delta=delta)
    cond_k = RNG.standard_normal((T, W))
    cond_v = RNG.standard_normal((T, W))
    solo_k = ora.bf16_to_f64(it.canon_k[0])
    rel_k = np.concatenate([ora.rotate_band(solo_k[:, h * hd:(h + 1) * hd], delta, 1e4,
                                            ora.NEOX_HALF) for h in range(H)], axis=1)
    solo_v = ora.bf16_to_f64(it.canon_v[0])
    m = min(T, W)
    uk, vk = ora.form_patch(cond_k, rel_k, m)
    uv, vv = ora.form_patch(cond_v, solo_v, m)
    it.patch_u = np.stack([uk, uv])[None]
    it.patch_vt = np.concatenate([vk.ravel(), vv.ravel()])[None]
    it.patch_m, it.patch_l0, it.patch_l1 = m, 0, 1
    got_k, _ = ora.reuse_layer(lay, it, 0, 0)
    got_v, _ = ora.reuse_layer(lay, it, 0, 1)
    np.testing.assert_allclose(got_k, cond_k, atol=1e-12)
    np.testing.assert_allclose(got_v, cond_v, atol=1e-12)


def test_low_rank_deficit_recovered_by_any_rank_at_least_r():
    T, W, r = 20, 16, 3
    base = RNG.standard_normal((T, W))
    deficit = RNG.standard_normal((T, r)) @ RNG.standard_normal((r, W))
    for m in (r, r + 1, W):
        u, vt = ora.form_patch(base + deficit, base, m)
        np.testing.assert_allclose(u @ vt, deficit, atol=1e-11)


def test_eckart_young_residual():
    T, W = 40, 24
    d = RNG.standard_normal((T, W))
    lam = np.sort(np.linalg.eigvalsh(d.T @ d))[::-1]  # σ_i² from the Gram matrix
    for m in (1, 4, 8, 23):
        u, vt = ora.form_patch(d, np.zeros_like(d), m)
        res = np.linalg.norm(d - u @ vt)
        assert abs(res - math.sqrt(max(lam[m:].sum(), 0.0))) < 1e-9 * np.linalg.norm(d)
        # no other rank-m product of random factors does better
        q = RNG.standard_normal((T, m)) @ RNG.standard_normal((m, W))
        a = np.linalg.lstsq(q.reshape(-1, 1), d.reshape(-1), rcond=None)[0]
        assert res <= np.linalg.norm(d - a * q) + 1e-12


def test_patch_added_after_rotation_not_rotated():
    # a patch that only touches one rope pair: rotating it too would change the result
    lay, it = gqa_item(L=1, T=2, H=1, hd=4, m=1, l0=0, l1=1, delta=3, float_factors=True)
    it.patch_u = np.zeros((1, 2, 2, 1)); it.patch_u[0, 0, :, 0] = 1.0
    it.patch_vt = np.zeros((1, 1 * 2 * 4)); it.patch_vt[0, 0] = 1.0  # K column 0 only
    vals, _ = ora.reuse_layer(lay, it, 0, 0)
    rot = ora.rotate_band(ora.bf16_to_f64(it.canon_k[0]), 3, 1e4, ora.NEOX_HALF)
    np.testing.assert_allclose(vals[:, 0], rot[:, 0] + 1.0, atol=1e-14)
    np.testing.assert_allclose(vals[:, 1:], rot[:, 1:], atol=1e-14)


# ------------------------------------------------------------------------------------------
# MLA
# ------------------------------------------------------------------------------------------

def mla_item(L=3, T=5, latent=16, rope=8, m=2, l0=1, l1=2, delta=0):
    from types import SimpleNamespace
    lay = SimpleNamespace(kind=ora.MLA, num_layers=L, page_size=4, num_kv_heads=0, head_dim=0,
                          latent_dim=latent, rope_dim=rope, rope_style=ora.NEOX_HALF,
                          rope_theta=1e4)
    k = rand_bf16_bits((L, T, latent + rope))
    pu = rand_bf16_bits((l1 - l0, 2, T, m))
    pv = rand_bf16_bits((l1 - l0, m * (latent + rope)), 0.1)
    return lay, ora.as_item(canon_k=k, patch_u=pu, patch_vt=pv, delta=delta, patch_m=m,
                            patch_l0=l0, patch_l1=l1)


def test_mla_latent_copied_byte_exact_and_only_kpe_turns():
    lay, it = mla_item(delta=-4321)
    for layer in (0, 2):  # unpatched layers
        out = ora.reuse_layer_bits(lay, it, layer, 0)
        np.testing.assert_array_equal(out[:, :16], it.canon_k[layer][:, :16])
        assert np.mean(out[:, 16:] != it.canon_k[layer][:, 16:]) > 0.5


def test_mla_latent_independent_of_delta():
    lay, a = mla_item(delta=5)
    b = ora.as_item(**{**vars(a), "delta": -9999})
    for layer in range(3):
        oa = ora.reuse_layer_bits(lay, a, layer, 0)
        ob = ora.reuse_layer_bits(lay, b, layer, 0)
        np.testing.assert_array_equal(oa[:, :16], ob[:, :16])
        assert not np.array_equal(oa[:, 16:], ob[:, 16:])


def test_mla_kpe_band_gets_its_own_patch_group():
    lay, it = mla_item(delta=0, m=2, l0=0, l1=3)
    vals, _ = ora.reuse_layer(lay, it, 1, 0)
    x = ora.bf16_to_f64(it.canon_k[1])
    u = ora.bf16_to_f64(it.patch_u[1])
    vt = ora.bf16_to_f64(it.patch_vt[1])
    for t in range(5):
        for c in range(24):
            g, cc, w = (0, c, 16) if c < 16 else (1, c - 16, 8)
            off = 0 if g == 0 else 2 * 16
            want = x[t, c] + sum(u[g, t, j] * vt[off + j * w + cc] for j in range(2))
            assert abs(vals[t, c] - want) < 1e-12


# ------------------------------------------------------------------------------------------
# slots and the pool
# ------------------------------------------------------------------------------------------

def test_slots_match_independent_page_expansion():
    ps = 16
    pt = RNG.permutation(40).reshape(5, 8).astype(np.int32)
    flat = (pt[:, :, None].astype(np.int64) * ps + np.arange(ps)).reshape(5, -1)
    for r in range(5):
        for t in range(8 * ps):
            assert ora.slot_of(pt, r, t, ps) == flat[r, t]


def test_identity_mode_scatter_is_byte_exact():
    # δ = 0, m = 0, canonicals encode (item, layer, token): the pool must equal a scatter
    # built from the page expansion; every other slot keeps the sentinel.
    ps, L, H, hd = 4, 2, 1, 8
    lay = ns_layout(num_layers=L, page_size=ps, num_kv_heads=H, head_dim=hd, rope_dim=hd)
    W = H * hd
    pt = RNG.permutation(12).reshape(2, 6).astype(np.int32)
    flat = (pt[:, :, None].astype(np.int64) * ps + np.arange(ps)).reshape(2, -1)
    k_pool = np.full((L, 48, W), 0x5A5A, np.uint16)
    v_pool = k_pool.copy()
    want_k, want_v = k_pool.copy(), v_pool.copy()
    items = []
    for i, (req, start, T) in enumerate([(0, 0, 7), (0, 9, 5), (1, 3, 13)]):
        code = lambda ch: np.array([[[(i << 12) | (l << 10) | (t << 3) | (c & 7) | (ch << 15)
                                      for c in range(W)] for t in range(T)] for l in range(L)],
                                   dtype=np.uint16)
        k, v = code(0), code(1)
        items.append(ora.as_item(canon_k=k, canon_v=v, delta=0, req=req, start_tok=start,
                                 num_tokens=T))
        for l in range(L):
            for t in range(T):
                want_k[l, flat[req, start + t]] = k[l, t]
                want_v[l, flat[req, start + t]] = v[l, t]
    ora.batch_reuse(lay, items, k_pool, v_pool, pt)
    np.testing.assert_array_equal(k_pool, want_k)
    np.testing.assert_array_equal(v_pool, want_v)


def test_relocate_in_place_rotates_only_rope_columns():
    from types import SimpleNamespace
    lay = SimpleNamespace(kind=ora.MLA, num_layers=2, page_size=4, num_kv_heads=0,
                          head_dim=0, latent_dim=8, rope_dim=8, rope_style=ora.INTERLEAVED,
                          rope_theta=1e4)
    pool = rand_bf16_bits((2, 16, 16))
    before = pool.copy()
    pt = np.array([[3, 1, 0, 2]], np.int32)
    ora.relocate(lay, pool, pt, 0, 2, 9, -576)
    touched = {ora.slot_of(pt, 0, t, 4) for t in range(2, 11)}
    for s in range(16):
        np.testing.assert_array_equal(pool[:, s, :8], before[:, s, :8])
        if s not in touched:
            np.testing.assert_array_equal(pool[:, s], before[:, s])
        else:
            for l in range(2):
                want = ora.f64_to_bf16(ora.rotate_band(ora.bf16_to_f64(before[l, s, 8:]), -576,
                                                       1e4, ora.INTERLEAVED))
                np.testing.assert_array_equal(pool[l, s, 8:], want)


# ------------------------------------------------------------------------------------------
# reversible switch: the patch re-added in place (App. E)
# ------------------------------------------------------------------------------------------

def switch_setup(kind="gqa", delta=0, m=3):
    """A chunk written clean (rank 0) into a pool, and the patch of its layers 1..2."""
    if kind == "gqa":
        lay, it = gqa_item(L=3, T=7, H=2, hd=8, m=m, l0=1, l1=3, delta=delta)
        W0 = W1 = 16
        rk, rv = 16, 16
    else:
        lay, it = mla_item(L=3, T=7, latent=16, rope=8, m=m, l0=1, l1=3, delta=delta)
        W0, W1 = 16, 8
        rk, rv = 24, 0
    lay.page_size = 4
    pt = np.array([[5, 2, 7], [0, 3, 1]], np.int32)
    k_pool = np.full((3, 32, rk), 0x5A5A, np.uint16)
    v_pool = np.full((3, 32, rv), 0x5A5A, np.uint16) if rv else None
    clean = ora.as_item(**{**vars(it), "patch_m": 0, "patch_l0": 0, "patch_l1": 0,
                           "req": 0, "start_tok": 2})
    ora.apply_reuse(lay, clean, k_pool, v_pool, pt)
    patched = ora.as_item(**{**vars(clean), "patch_m": m, "patch_l0": 1, "patch_l1": 3})
    return lay, it, pt, k_pool, v_pool, clean, patched


@pytest.mark.parametrize("kind", ["gqa", "mla"])
def test_patch_readd_on_clean_view_equals_reuse_with_patch(kind):
    # App. E: the clean view is the stored canonical (an exact copy at δ = 0); re-adding the
    # rank-m patch on it gives exactly the patched reuse, one rounding each
    lay, it, pt, k_pool, v_pool, clean, patched = switch_setup(kind, delta=0)
    ora.patch_inplace(lay, k_pool, v_pool, pt, 0, 2, 7, it.patch_u, it.patch_vt, it.patch_m,
                      1, 3)
    want_k = np.full_like(k_pool, 0x5A5A)
    want_v = None if v_pool is None else np.full_like(v_pool, 0x5A5A)
    ora.apply_reuse(lay, patched, want_k, want_v, pt)
    np.testing.assert_array_equal(k_pool, want_k)
    if v_pool is not None:
        np.testing.assert_array_equal(v_pool, want_v)


def test_patch_inplace_sign_symmetry_and_pure_python_sums():
    lay, it, pt, k_pool, v_pool, clean, patched = switch_setup("gqa", delta=777, m=2)
    before_k, before_v = k_pool.copy(), v_pool.copy()
    a_k, a_v = k_pool.copy(), v_pool.copy()
    b_k, b_v = k_pool.copy(), v_pool.copy()
    neg_u = it.patch_u ^ np.uint16(0x8000)  # exact negation of every bf16 factor
    ora.patch_inplace(lay, a_k, a_v, pt, 0, 2, 7, it.patch_u, it.patch_vt, 2, 1, 3, sign=-1)
    ora.patch_inplace(lay, b_k, b_v, pt, 0, 2, 7, neg_u, it.patch_vt, 2, 1, 3, sign=+1)
    np.testing.assert_array_equal(a_k, b_k)
    np.testing.assert_array_equal(a_v, b_v)
    # element by element: x - Σ_j U_tj Vt_jc, rounded once; untouched rows and layers stay
    W = 16
    for layer in range(3):
        for ch, (pool, before) in enumerate(((a_k, before_k), (a_v, before_v))):
            for t in range(7):
                s = ora.slot_of(pt, 0, 2 + t, 4)
                for c in range(W):
                    x = float(ora.bf16_to_f64(before[layer, s, c]))
                    if 1 <= layer < 3:
                        li = layer - 1
                        for j in range(2):
                            x -= (float(ora.bf16_to_f64(it.patch_u[li, ch, t, j])) *
                                  float(ora.bf16_to_f64(it.patch_vt[li, ch * 2 * W + j * W + c])))
                    assert pool[layer, s, c] == ora.f64_to_bf16(np.array([x]))[0]
    touched = {ora.slot_of(pt, 0, 2 + t, 4) for t in range(7)}
    for s in set(range(32)) - touched:
        np.testing.assert_array_equal(a_k[:, s], before_k[:, s])


def test_patch_add_then_remove_is_within_two_roundings():
    # the inverse of a re-add is the subtraction of the same patch, exact up to rounding
    lay, it, pt, k_pool, v_pool, clean, patched = switch_setup("gqa", delta=-31, m=3)
    before = ora.bf16_to_f64(k_pool).copy()
    ora.patch_inplace(lay, k_pool, v_pool, pt, 0, 2, 7, it.patch_u, it.patch_vt, 3, 1, 3)
    mid = ora.bf16_to_f64(k_pool).copy()
    ora.patch_inplace(lay, k_pool, v_pool, pt, 0, 2, 7, it.patch_u, it.patch_vt, 3, 1, 3,
                      sign=-1)
    after = ora.bf16_to_f64(k_pool)
    bound = 0.5 * ora.bf16_ulp(mid) + 0.5 * ora.bf16_ulp(after)
    assert np.all(np.abs(after - before) <= bound * (1 + 1e-9))
    assert not np.array_equal(mid[1:], before[1:])


# ------------------------------------------------------------------------------------------
# patch forming from a given deficit (App. A form_patch; randomized range finder)
# ------------------------------------------------------------------------------------------

def test_randomized_patch_recovers_an_exactly_low_rank_deficit():
    # a deficit of rank r <= k lies in the sketch's range: the randomized factors equal the
    # truncated SVD's (Eckart–Young), whatever the test matrix
    rng = np.random.default_rng(11)
    T, W, r, m, k = 60, 40, 6, 4, 10
    delta = rng.standard_normal((T, r)) @ np.diag([9, 7, 5, 3, 2, 1.0]) @ rng.standard_normal((r, W))
    for q in (0, 1):
        us, vt, sig = ora.form_patch_randomized(delta, rng.standard_normal((W, k)), m, q)
        us0, vt0, sig0 = ora.form_patch_svd(delta, m)
        np.testing.assert_allclose(sig, sig0, rtol=1e-10)
        np.testing.assert_allclose(us, us0, atol=1e-9)
        np.testing.assert_allclose(vt, vt0, atol=1e-9)
        np.testing.assert_allclose(vt @ vt.T, np.eye(m), atol=1e-10)
        # the sign convention: each row's largest-magnitude entry is positive
        for row in (vt, vt0):
            assert np.all(row[np.arange(m), np.argmax(np.abs(row), axis=1)] > 0)


def test_randomized_patch_residual_near_the_eckart_young_optimum():
    # a decaying spectrum: with power iterations the residual approaches sqrt(sum_{i>m} s_i^2)
    rng = np.random.default_rng(12)
    T, W, m, k = 120, 80, 8, 16
    u, _ = np.linalg.qr(rng.standard_normal((T, W)))
    v, _ = np.linalg.qr(rng.standard_normal((W, W)))
    s = 0.8 ** np.arange(W)
    delta = (u * s) @ v.T
    best = np.sqrt(np.sum(s[m:] ** 2))
    # the exact SVD returns the planted spectrum and the planted rank-m truncation
    us0, vt0, sig0 = ora.form_patch_svd(delta, m)
    np.testing.assert_allclose(sig0, s[:m], rtol=1e-12)
    np.testing.assert_allclose(us0 @ vt0, (u[:, :m] * s[:m]) @ v[:, :m].T, atol=1e-12)
    prev = np.inf
    for q in (0, 1, 2):
        us, vt, sig = ora.form_patch_randomized(delta, rng.standard_normal((W, k)), m, q)
        res = np.linalg.norm(delta - us @ vt)
        assert best - 1e-12 <= res <= 1.01 * best if q >= 1 else res <= 1.5 * best
        assert res <= prev * (1 + 1e-9)
        prev = res
    np.testing.assert_allclose(sig, s[:m], rtol=1e-3)


def test_randomized_patch_zero_deficit_gives_zero_factors():
    us, vt, sig = ora.form_patch_randomized(np.zeros((10, 6)), np.ones((6, 4)), 3, 1)
    assert np.all(us == 0) and np.all(vt == 0) and np.all(sig == 0)


# ------------------------------------------------------------------------------------------
# shapes and sizes printed on the pages
# ------------------------------------------------------------------------------------------

def read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("|")[0].strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split("=")
            out[k.strip()] = int(v)
    return out


def test_layout_reading_matches_printed_shapes():
    g = read_golden("pages_shapes.txt")
    qwen = ns_layout(num_kv_heads=g["qwen25vl_kv_heads"], head_dim=g["qwen25vl_head_dim"],
                     rope_dim=g["qwen25vl_head_dim"])
    row_k, row_v, (w0, w1) = ora.widths(qwen)
    assert row_k == row_v == w0 == w1 == g["qwen25vl_k_width"]
    bands = ora.rope_bands(qwen)
    assert all(len(ora.rope_pairs(d, ora.NEOX_HALF)[0]) == g["qwen25vl_rope_pairs_per_head"]
               for _, d in bands)
    q3 = ns_layout(num_kv_heads=g["qwen3vl_kv_heads"], head_dim=128, rope_dim=128)
    assert ora.widths(q3)[0] == g["qwen3vl_k_width"]
    from types import SimpleNamespace
    kimi = SimpleNamespace(kind=ora.MLA, num_kv_heads=0, head_dim=0,
                           latent_dim=g["kimivl_ckv_dim"], rope_dim=g["kimivl_krope_dim"])
    row, _, (c, r) = ora.widths(kimi)
    assert (c, r) == (512, 64) and row == 576
    (c0, d), = ora.rope_bands(kimi)
    assert c0 == 512 and len(ora.rope_pairs(d, ora.NEOX_HALF)[0]) == g["kimivl_krope_pairs"]


# ------------------------------------------------------------------------------------------
# M-RoPE sections (Fig. 2: 16|24|24 and 24|20|20 pairs over t, h, w)
# ------------------------------------------------------------------------------------------

def mrope_layout(style, sections, theta=1e6, heads=2):
    return ns_layout(num_kv_heads=heads, head_dim=128, rope_dim=128, rope_theta=theta,
                     mrope_section=tuple(sections), mrope_style=style)


def test_mrope_sections_match_printed_counts():
    g = read_golden("pages_shapes.txt")
    npairs = g["qwen25vl_rope_pairs_per_head"]
    blocked = [g["qwen25vl_mrope_t"], g["qwen25vl_mrope_h"], g["qwen25vl_mrope_w"]]
    inter = [g["qwen3vl_mrope_t"], g["qwen3vl_mrope_h"], g["qwen3vl_mrope_w"]]
    assert sum(blocked) == sum(inter) == npairs
    for style, sec in ((ora.MROPE_CONTIGUOUS, blocked), (ora.MROPE_INTERLEAVED, inter)):
        axes = ora.mrope_pair_axes(npairs, sec, style)
        assert [int(np.sum(axes == a)) for a in range(3)] == sec
    # blocked: t, then h, then w, in the printed order
    axes = ora.mrope_pair_axes(npairs, blocked, ora.MROPE_CONTIGUOUS)
    assert np.all(np.diff(axes) >= 0) and axes[0] == 0 and axes[-1] == 2
    # interleaved: h and w alternate with t across the pairs, never two h or two w adjacent
    axes = ora.mrope_pair_axes(npairs, inter, ora.MROPE_INTERLEAVED)
    assert all(not (axes[i] == axes[i + 1] and axes[i] != 0) for i in range(npairs - 1))
    with pytest.raises(ValueError):
        ora.mrope_pair_axes(npairs, [16, 24, 23], ora.MROPE_CONTIGUOUS)


@pytest.mark.parametrize("style,sections", [(ora.MROPE_CONTIGUOUS, (16, 24, 24)),
                                            (ora.MROPE_INTERLEAVED, (24, 20, 20))])
def test_mrope_equal_offsets_are_one_dimensional_rope(style, sections):
    # Fig. 2 caption: relocation advances all three coordinates together, so the layout of
    # the sections does not matter: the result equals 1-D RoPE by the same delta, bit for bit
    lay = mrope_layout(style, sections)
    flat = mrope_layout(style, (0, 0, 0))
    T = 5
    canon = ora.f64_to_bf16(RNG.standard_normal((1, T, 256)))
    for delta in (1, -77, 123457):
        a = ora.as_item(canon_k=canon, canon_v=canon, delta=delta, num_tokens=T)
        b = ora.as_item(canon_k=canon, canon_v=canon, delta=delta, delta_h=delta, delta_w=delta,
                        num_tokens=T)
        assert np.array_equal(ora.reuse_layer_bits(lay, a, 0, 0), ora.reuse_layer_bits(flat, a, 0, 0))
        assert np.array_equal(ora.reuse_layer_bits(lay, b, 0, 0), ora.reuse_layer_bits(flat, a, 0, 0))


@pytest.mark.parametrize("style,sections", [(ora.MROPE_CONTIGUOUS, (16, 24, 24)),
                                            (ora.MROPE_INTERLEAVED, (24, 20, 20))])
def test_mrope_pair_turns_by_its_section_offset(style, sections):
    # each pair, taken one at a time in pure Python: a complex multiplication by
    # exp(i * delta_section * theta^(-2k/d)) with delta_section chosen by the pair's section
    lay = mrope_layout(style, sections, heads=1)
    d = 128
    offs = (1000, -3, 41)
    x = RNG.standard_normal((2, d))
    it = ora.as_item(canon_k=None, delta=offs[0], delta_h=offs[1], delta_w=offs[2], num_tokens=2)
    got = ora.rotate_band(x, ora.pair_offsets(lay, it, d // 2), lay.rope_theta, ora.NEOX_HALF)
    axes = ora.mrope_pair_axes(d // 2, sections, style)
    for k in range(d // 2):
        phi = offs[axes[k]] * lay.rope_theta ** (-2.0 * k / d)
        for r in range(2):
            z = complex(x[r, k], x[r, k + d // 2]) * cmath.exp(1j * phi)
            assert abs(got[r, k] - z.real) <= 1e-12 and abs(got[r, k + d // 2] - z.imag) <= 1e-12
    # a temporal move (delta_t only) leaves every h and w pair exactly as it was
    it_t = ora.as_item(canon_k=None, delta=500, delta_h=0, delta_w=0, num_tokens=2)
    got_t = ora.rotate_band(x, ora.pair_offsets(lay, it_t, d // 2), lay.rope_theta, ora.NEOX_HALF)
    still = np.flatnonzero(axes != 0)
    assert np.array_equal(got_t[:, still], x[:, still])
    assert np.array_equal(got_t[:, still + d // 2], x[:, still + d // 2])
    assert not np.allclose(got_t[:, np.flatnonzero(axes == 0)], x[:, np.flatnonzero(axes == 0)])


def test_mrope_offsets_compose_per_section():
    lay = mrope_layout(ora.MROPE_INTERLEAVED, (24, 20, 20), heads=1)
    x = RNG.standard_normal((3, 128))
    a = ora.as_item(canon_k=None, delta=7, delta_h=-2000, delta_w=31, num_tokens=3)
    b = ora.as_item(canon_k=None, delta=-900, delta_h=5, delta_w=1 << 20, num_tokens=3)
    ab = ora.as_item(canon_k=None, delta=7 - 900, delta_h=-2000 + 5, delta_w=31 + (1 << 20),
                     num_tokens=3)
    po = lambda it: ora.pair_offsets(lay, it, 64)
    two = ora.rotate_band(ora.rotate_band(x, po(a), 1e6, ora.NEOX_HALF), po(b), 1e6, ora.NEOX_HALF)
    one = ora.rotate_band(x, po(ab), 1e6, ora.NEOX_HALF)
    np.testing.assert_allclose(two, one, atol=1e-9)


# ------------------------------------------------------------------------------------------
# re-anchoring keys stored before rotation (QV-PIC, Eq. 2)
# ------------------------------------------------------------------------------------------

def anchor_item(layout, T, positions, seed=0):
    rng = np.random.default_rng(seed)
    row = layout.num_kv_heads * layout.head_dim if layout.kind == ora.GQA else \
        layout.latent_dim + layout.rope_dim
    k = ora.f64_to_bf16(rng.standard_normal((1, T, row)))
    v = ora.f64_to_bf16(rng.standard_normal((1, T, row))) if layout.kind == ora.GQA else None
    from types import SimpleNamespace
    return SimpleNamespace(canon_k=k, canon_v=v, positions=np.asarray(positions), num_tokens=T,
                           req=0, start_tok=0)


def test_reanchor_turns_each_token_by_its_own_position():
    lay = ns_layout(num_kv_heads=2, head_dim=16, rope_dim=16)
    pos = [0, 5, -3, 1 << 20, 77]
    it = anchor_item(lay, len(pos), pos)
    vals, mask = ora.reanchor_layer(lay, it, 0, 0)
    assert not mask.any()
    x = ora.bf16_to_f64(it.canon_k[0])
    d = 16
    for j, p in enumerate(pos):
        for h in range(2):
            for k in range(d // 2):
                z = complex(x[j, h * d + k], x[j, h * d + k + d // 2]) * \
                    cmath.exp(1j * p * 1e4 ** (-2.0 * k / d))
                assert abs(vals[j, h * d + k] - z.real) <= 1e-12
                assert abs(vals[j, h * d + k + d // 2] - z.imag) <= 1e-12
    assert np.array_equal(vals[0], x[0])                      # position 0: unchanged
    vbits = ora.reanchor_layer_bits(lay, it, 0, 1)
    assert np.array_equal(vbits, it.canon_v[0])               # values: byte copies


def test_reanchor_mrope_coordinates():
    sec = (16, 24, 24)
    lay = mrope_layout(ora.MROPE_CONTIGUOUS, sec, heads=1)
    flat = mrope_layout(ora.MROPE_CONTIGUOUS, (0, 0, 0), heads=1)
    pos3 = [(3, 40, 41), (0, 0, 0), (1000, -5, 7)]
    it = anchor_item(lay, 3, pos3)
    vals, _ = ora.reanchor_layer(lay, it, 0, 0)
    x = ora.bf16_to_f64(it.canon_k[0])
    axes = ora.mrope_pair_axes(64, sec, ora.MROPE_CONTIGUOUS)
    for j, p in enumerate(pos3):
        for k in (0, 15, 16, 39, 40, 63):
            z = complex(x[j, k], x[j, k + 64]) * cmath.exp(1j * p[axes[k]] * 1e6 ** (-k / 64))
            assert abs(vals[j, k] - z.real) <= 1e-12 and abs(vals[j, k + 64] - z.imag) <= 1e-12
    # equal coordinates: 1-D RoPE at that position, bit for bit
    same = anchor_item(lay, 3, [(p, p, p) for p in (9, -2, 123456)], seed=1)
    flat_it = anchor_item(flat, 3, [9, -2, 123456], seed=1)
    assert np.array_equal(ora.reanchor_layer_bits(lay, same, 0, 0),
                          ora.reanchor_layer_bits(flat, flat_it, 0, 0))


def test_reanchor_then_relocate_is_reanchor_at_moved_positions():
    # R(δ) R(P) K̄ = R(P + δ) K̄: Kamera's relocation of a re-anchored key moves its anchor
    lay = ns_layout(num_kv_heads=1, head_dim=32, rope_dim=32)
    pos = np.array([4, 100, -7, 65536])
    it = anchor_item(lay, 4, pos)
    moved = anchor_item(lay, 4, pos + 999)
    a, _ = ora.reanchor_layer(lay, it, 0, 0)
    b, _ = ora.reanchor_layer(lay, moved, 0, 0)
    np.testing.assert_allclose(ora.rotate_band(a, 999, 1e4, ora.NEOX_HALF), b, atol=1e-9)


def test_reanchor_mla_rotates_only_k_pe():
    lay = ns_layout(kind=ora.MLA, num_kv_heads=0, head_dim=0, latent_dim=32, rope_dim=16)
    it = anchor_item(lay, 3, [1, 2, 3])
    bits = ora.reanchor_layer_bits(lay, it, 0, 0)
    assert np.array_equal(bits[:, :32], it.canon_k[0][:, :32])
    assert not np.array_equal(bits[:, 32:], it.canon_k[0][:, 32:])


def test_reanchored_items_land_at_their_slots():
    # every token's re-anchored row is written at slot_of(req, start_tok + j) of each layer and
    # channel (an independent page expansion), and no other slot changes
    ps, L = 4, 2
    lay = ns_layout(num_layers=L, page_size=ps, num_kv_heads=2, head_dim=8, rope_dim=8)
    W = 16
    pt = RNG.permutation(12).reshape(2, 6).astype(np.int32)
    flat = (pt[:, :, None].astype(np.int64) * ps + np.arange(ps)).reshape(2, -1)
    k_pool = np.full((L, 48, W), 0x5A5A, np.uint16)
    v_pool = k_pool.copy()
    want_k, want_v = k_pool.copy(), v_pool.copy()
    from types import SimpleNamespace
    for i, (req, start, T) in enumerate([(0, 1, 7), (1, 5, 9)]):
        rng = np.random.default_rng(40 + i)
        k = ora.f64_to_bf16(rng.standard_normal((L, T, W)))
        v = ora.f64_to_bf16(rng.standard_normal((L, T, W)))
        it = SimpleNamespace(canon_k=k, canon_v=v, positions=rng.integers(-50, 50, T),
                             num_tokens=T, req=req, start_tok=start)
        ora.apply_reanchor(lay, it, k_pool, v_pool, pt)
        for layer in range(L):
            kb = ora.reanchor_layer_bits(lay, it, layer, 0)
            vb = ora.reanchor_layer_bits(lay, it, layer, 1)
            for j in range(T):
                want_k[layer, flat[req, start + j]] = kb[j]
                want_v[layer, flat[req, start + j]] = vb[j]
    np.testing.assert_array_equal(k_pool, want_k)
    np.testing.assert_array_equal(v_pool, want_v)
    # MLA: one pool, only the k_pe band turns
    mla = ns_layout(kind=ora.MLA, num_layers=1, page_size=ps, num_kv_heads=0, head_dim=0,
                    latent_dim=16, rope_dim=8)
    pool = np.full((1, 48, 24), 0x5A5A, np.uint16)
    want = pool.copy()
    it = SimpleNamespace(canon_k=ora.f64_to_bf16(RNG.standard_normal((1, 5, 24))), canon_v=None,
                         positions=np.array([3, -1, 0, 7, 100]), num_tokens=5, req=1, start_tok=2)
    ora.apply_reanchor(mla, it, pool, None, pt)
    bits = ora.reanchor_layer_bits(mla, it, 0, 0)
    for j in range(5):
        want[0, flat[1, 2 + j]] = bits[j]
    np.testing.assert_array_equal(pool, want)


# ------------------------------------------------------------------------------------------
# the error scale the GPU tolerance multiplies (§6 "within one bf16 ULP")
# ------------------------------------------------------------------------------------------

def _magnitude_by_hand(lay, it, layer, ch):
    """The scale of the terms of every result element, by explicit loops: |x| of the element,
    or |a| + |b| of its rope pair when the pair turns, plus the sum over j of |U_tj * Vt_jc|."""
    canon = (it.canon_k if ch == 0 else it.canon_v)[layer]
    T, row = canon.shape
    x = [[float(ora.bf16_to_f64(canon[t, c])) for c in range(row)] for t in range(T)]
    out = [[abs(x[t][c]) for c in range(row)] for t in range(T)]
    if ch == 0 and it.delta != 0:
        if lay.kind == ora.GQA:
            bands = [(h * lay.head_dim, lay.head_dim) for h in range(lay.num_kv_heads)]
        else:
            bands = [(lay.latent_dim, lay.rope_dim)]
        for c0, d in bands:
            for k in range(d // 2):
                a, b = (c0 + k, c0 + k + d // 2) if lay.rope_style == ora.NEOX_HALF else \
                    (c0 + 2 * k, c0 + 2 * k + 1)
                for t in range(T):
                    out[t][a] = out[t][b] = abs(x[t][a]) + abs(x[t][b])
    if it.patch_m and it.patch_l0 <= layer < it.patch_l1:
        li, m = layer - it.patch_l0, it.patch_m
        if lay.kind == ora.GQA:
            groups = [(0, row, ch)]
        else:
            groups = [(0, lay.latent_dim, 0), (lay.latent_dim, lay.rope_dim, 1)]
        w0 = lay.num_kv_heads * lay.head_dim if lay.kind == ora.GQA else lay.latent_dim
        for c0, w, g in groups:
            off = 0 if g == 0 else m * w0
            for t in range(T):
                for c in range(w):
                    for j in range(m):
                        u = float(ora.bf16_to_f64(it.patch_u[li][g][t][j]))
                        v = float(ora.bf16_to_f64(it.patch_vt[li][off + j * w + c]))
                        out[t][c0 + c] += abs(u * v)
    return np.array(out)


@pytest.mark.parametrize("kind,style,delta", [("gqa", ora.NEOX_HALF, 777), ("gqa", ora.NEOX_HALF, 0),
                                              ("gqa", ora.INTERLEAVED, -5), ("mla", ora.NEOX_HALF, 31),
                                              ("mla", ora.INTERLEAVED, 0)])
def test_magnitude_scale_by_explicit_loops(kind, style, delta):
    if kind == "gqa":
        lay, it = gqa_item(L=3, T=4, H=2, hd=8, m=3, l0=1, l1=3, delta=delta)
        lay.rope_style = style
    else:
        lay, it = mla_item(L=3, T=4, latent=16, rope=8, m=2, l0=1, l1=2, delta=delta)
        lay.rope_style = style
    # signs on both sides of zero in the factors: a product of sums would not match
    n_ch = 2 if kind == "gqa" else 1
    for layer in range(3):
        for ch in range(n_ch):
            got = ora.magnitude_layer(lay, it, layer, ch)
            np.testing.assert_allclose(got, _magnitude_by_hand(lay, it, layer, ch), rtol=1e-12,
                                       atol=0)


# ------------------------------------------------------------------------------------------
# consumer check: decode attention and the log-sum-exp merge (§1)
# ------------------------------------------------------------------------------------------

def test_attention_of_a_union_is_the_lse_merge_of_its_parts():
    rng = np.random.default_rng(21)
    k = rng.standard_normal((50, 16))
    v = rng.standard_normal((50, 8))
    q = rng.standard_normal(16)
    whole = ora.attend(k, v, q, 0.3)
    for cut in ((20,), (1, 49), (10, 11, 30)):
        bounds = (0,) + cut + (50,)
        parts = [ora.attend(k[a:b], v[a:b], q, 0.3) for a, b in zip(bounds[:-1], bounds[1:])]
        o, l = ora.lse_merge(parts)
        np.testing.assert_allclose(o, whole[0], atol=1e-12)
        assert abs(l - whole[1]) <= 1e-12
    # the two-part form printed on the page: o = (1 - mu) o_B + mu o_A, mu = A's softmax mass
    (oa, la), (ob, lb) = ora.attend(k[:20], v[:20], q, 0.3), ora.attend(k[20:], v[20:], q, 0.3)
    mu = math.exp(la) / (math.exp(la) + math.exp(lb))
    np.testing.assert_allclose((1 - mu) * ob + mu * oa, whole[0], atol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(22)
    v = rng.standard_normal((7, 5))
    # one key: the output is its value, lse its score
    o, l = ora.attend(np.ones((1, 3)), v[:1], np.array([1.0, 2.0, 3.0]), 0.5)
    np.testing.assert_array_equal(o, v[0])
    assert l == 3.0
    # equal scores: the mean of the values, lse = s + log T
    o, l = ora.attend(np.zeros((7, 3)), v, np.ones(3), 1.0)
    np.testing.assert_allclose(o, v.mean(axis=0), atol=1e-15)
    assert abs(l - math.log(7)) <= 1e-15
    # a dominant key takes all the mass; an empty context gives (0, -inf)
    k = np.zeros((7, 2))
    k[4] = [100.0, 0.0]
    o, _ = ora.attend(k, v, np.array([1.0, 0.0]), 1.0)
    np.testing.assert_allclose(o, v[4], atol=1e-30)
    o, l = ora.attend(np.zeros((0, 2)), np.zeros((0, 5)), np.ones(2), 1.0)
    assert np.all(o == 0) and l == -np.inf
    o, l = ora.lse_merge([(np.zeros(5), -np.inf), (np.zeros(5), -np.inf)])
    assert np.all(o == 0) and l == -np.inf


def test_decode_attention_gathers_heads_and_pages():
    # brute force on a tiny pool: GQA head grouping and the MLA absorbed form against explicit
    # loops over tokens
    rng = np.random.default_rng(23)
    pt = np.array([[2, 0], [1, 3]])
    gqa = ns_layout(num_kv_heads=2, head_dim=4, rope_dim=4, page_size=2)
    kp = ora.f64_to_bf16(rng.standard_normal((1, 8, 8)))
    vp = ora.f64_to_bf16(rng.standard_normal((1, 8, 8)))
    q = rng.standard_normal((4, 4))
    o, l = ora.decode_attention(gqa, kp, vp, pt, 1, 3, q, 0.5, 0)
    slots = [1 * 2 + 0, 1 * 2 + 1, 3 * 2 + 0]
    for h in range(4):
        kvh = h // 2
        s = [0.5 * sum(ora.bf16_to_f64(kp[0][t][kvh * 4 + d]) * q[h][d] for d in range(4))
             for t in slots]
        w = [math.exp(x - max(s)) for x in s]
        for d in range(4):
            ref = sum(wi * ora.bf16_to_f64(vp[0][t][kvh * 4 + d]) for wi, t in zip(w, slots)) / sum(w)
            assert abs(o[h][d] - ref) <= 1e-12
        assert abs(l[h] - (max(s) + math.log(sum(w)))) <= 1e-12
    mla = ns_layout(kind=ora.MLA, num_kv_heads=0, head_dim=0, latent_dim=4, rope_dim=2,
                    page_size=2)
    kp = ora.f64_to_bf16(rng.standard_normal((1, 8, 6)))
    qm = rng.standard_normal((3, 6))
    o, l = ora.decode_attention(mla, kp, None, pt, 0, 4, qm, 1.0, 0)
    rows = ora.bf16_to_f64(kp[0][[4, 5, 0, 1]])
    for h in range(3):
        ref_o, ref_l = ora.attend(rows, rows[:, :4], qm[h], 1.0)
        np.testing.assert_allclose(o[h], ref_o, atol=1e-12)


def test_patch_byte_fraction_matches_printed_values():
    with open(os.path.join(GOLDEN, "patch_fraction.txt")) as f:
        rows = [l.split("|")[0] for l in f if l.strip() and not l.startswith("#")]
    for r in rows:
        m, frac, tol = (float(x) for x in r.split(","))
        assert abs(ora.patch_byte_fraction(512, 512, int(m)) - frac) <= tol
