"""GPU parity of the C-ABI calls against the float64 oracle, at sizes the oracle finishes in
seconds that span several tiles, ragged tails, unaligned page starts and both layouts.

Every slot of both pools is compared: written rows against the oracle (bit-exact where no
arithmetic happens, else the tolerance in kamera_testlib), untouched slots against the
sentinel they were filled with.
"""
import dataclasses

import numpy as np
import pytest
import torch

import position_independent_multimodal_gb300 as km
import workloads as wl
from oracle import kamera_oracle as ora
from tests import kamera_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda(cuda_ok):
    return cuda_ok


def gqa_layout(L=3, H=2, hd=64, style=wl.NEOX_HALF, theta=1e4, page=16):
    return wl.Layout(kind=wl.GQA, num_layers=L, page_size=page, num_kv_heads=H, head_dim=hd,
                     rope_dim=hd, rope_style=style, rope_theta=theta)


def mla_layout(L=3, style=wl.NEOX_HALF, page=16, latent=512, rope=64):
    return wl.Layout(kind=wl.MLA, num_layers=L, page_size=page, latent_dim=latent,
                     rope_dim=rope, rope_style=style, rope_theta=1e4)


def ragged(layout, m, name, seed=0, strong=True):
    # five placements of four chunks of ragged length into three requests, starting mid-page
    Ts = [1, 37, 130, 300]
    placements = [(0, 0, 5, 0), (1, 0, 40, -1), (2, 1, 0, 131071), (3, 2, 7, -32768),
                  (1, 1, 300, 17)]
    return wl.reuse_workload(name, layout, n_chunks=4, T=Ts, placements=placements, m=m,
                             l0=1, l1=layout.num_layers, seed=seed, strong=strong,
                             patch_per_item=True, extra_pages=3)


def run_and_check(w, batch=True, **options):
    h = km.create(w.layout, **options)
    items = tl.to_device_items(w.items)
    if batch:
        k, v, status, _ = tl.run_batch(h, w.layout, items, w.page_table, w.num_slots)
    else:
        k, v, status = tl.run_single(h, w.layout, items, w.page_table, w.num_slots)
    assert status == 0
    return tl.check_full(w.layout, w.items, w.page_table, k, v)


@pytest.mark.parametrize("strong", [False, True])
@pytest.mark.parametrize("batch", [False, True])
def test_config1_tiny_gqa(strong, batch):
    st = run_and_check(wl.config1(strong=strong), batch=batch)
    assert st.computed > 0


@pytest.mark.parametrize("m", [0, 3, 8, 12, 16, 24, 32, 64])
@pytest.mark.parametrize("style", [wl.NEOX_HALF, wl.INTERLEAVED])
def test_gqa_ragged_batch(m, style):
    # ranks 3 and 12 take the CUDA-core path, multiples of 8 the tensor-core path
    run_and_check(ragged(gqa_layout(style=style), m, f"gqa{m}{style}"))


@pytest.mark.parametrize("kind", ["gqa", "mla"])
def test_fma_engine_matches_oracle(kind):
    # the CUDA-core engine for every patched tile (the ablation of the tensor-core path)
    lay = gqa_layout(L=2, H=4, hd=128) if kind == "gqa" else mla_layout(L=2)
    run_and_check(ragged(lay, 32, f"fma{kind}"), patch_engine=km.KAMERA_ENGINE_CUDA_CORES)


@pytest.mark.parametrize("m", [0, 8, 32, 128])
def test_gqa_wide_heads_and_big_rank(m):
    lay = gqa_layout(L=2, H=8, hd=128, theta=1e6)
    run_and_check(ragged(lay, m, f"gqaw{m}"))


@pytest.mark.parametrize("m", [0, 16, 32])
@pytest.mark.parametrize("style", [wl.NEOX_HALF, wl.INTERLEAVED])
def test_mla_ragged_batch(m, style):
    run_and_check(ragged(mla_layout(style=style), m, f"mla{m}{style}"))


def with_mrope_offsets(w, seed):
    """Give every item its own (δ_t, δ_h, δ_w): a temporal move (h, w still), a move of all
    three together, a move with t still, and independent offsets, in turn."""
    rng = np.random.default_rng(seed)
    out = []
    for i, it in enumerate(w.items):
        kind = i % 4
        if kind == 0:
            dh = dw = 0
        elif kind == 1:
            dh = dw = it.delta
        elif kind == 2:
            it = dataclasses.replace(it, delta=0)
            dh, dw = int(rng.integers(1, 5000)), -int(rng.integers(1, 5000))
        else:  # within ±2^20, where the float64 angle of the oracle is exact to ~1e-10 rad
            dh, dw = int(rng.integers(-(1 << 20), 1 << 20)), int(rng.integers(-70000, 70000))
        out.append(dataclasses.replace(it, delta_h=dh, delta_w=dw))
    w.items = out
    return w


def mrope_layout(style, sections, H, theta, rope_style=wl.NEOX_HALF, L=3):
    return wl.Layout(kind=wl.GQA, num_layers=L, page_size=16, num_kv_heads=H, head_dim=128,
                     rope_dim=128, rope_style=rope_style, rope_theta=theta,
                     mrope_section=sections, mrope_style=style)


@pytest.mark.parametrize("m", [0, 12, 32])
@pytest.mark.parametrize("which", ["blocked-16-24-24", "interleaved-24-20-20"])
@pytest.mark.parametrize("batch", [False, True])
def test_mrope_per_section_offsets(which, m, batch):
    # Fig. 2: Qwen2.5-VL's 16|24|24 blocked sections (4 KV heads, θ = 1e6) and Qwen3-VL's
    # 24|20|20 interleaved sections (8 KV heads, θ = 5e6), every pair turning by its
    # section's offset; rank 32 takes the tensor cores, rank 12 the CUDA cores, rank 0 only
    # the copy kernel
    if which.startswith("blocked"):
        lay = mrope_layout(wl.MROPE_CONTIGUOUS, (16, 24, 24), 4, 1e6)
    else:
        lay = mrope_layout(wl.MROPE_INTERLEAVED, (24, 20, 20), 8, 5e6)
    w = with_mrope_offsets(ragged(lay, m, f"mrope{which}{m}"), seed=m)
    st = run_and_check(w, batch=batch)
    assert st.computed > 0


def test_mrope_with_interleaved_pairing_takes_the_general_kernel():
    # interleaved (2i, 2i+1) pairing is served by the general pipeline
    lay = mrope_layout(wl.MROPE_CONTIGUOUS, (16, 24, 24), 2, 1e6, rope_style=wl.INTERLEAVED)
    run_and_check(with_mrope_offsets(ragged(lay, 32, "mropeil"), seed=3))


def test_mla_latent_is_byte_exact_on_unpatched_layers():
    w = ragged(mla_layout(L=4), 32, "mlab")
    w.items = [it for it in w.items]
    for it in w.items:
        it.patch_l0, it.patch_l1 = 2, 4
        if it.patch_u is not None:
            it.patch_u, it.patch_vt = it.patch_u[1:3], it.patch_vt[1:3]
    h = km.create(w.layout)
    k, _, status, _ = tl.run_batch(h, w.layout, tl.to_device_items(w.items), w.page_table,
                                   w.num_slots)
    assert status == 0
    kb = wl.bf16_bits(k)
    pt = w.page_table.numpy()
    for it in w.items:
        sl = tl.slots_of(pt, it.req, it.start_tok, it.num_tokens, 16)
        cb = wl.bf16_bits(it.canon_k)
        for layer in (0, 1):
            np.testing.assert_array_equal(kb[layer, sl, :512], cb[layer, :, :512])


def test_identity_mode_exhaustive_scatter():
    # δ = 0 and m = 0: the pool must hold the canonical bit patterns at the mapped slots;
    # canonicals encode (chunk, layer, token) and include signed zeros and NaN payloads.
    lay = gqa_layout(L=2, H=1, hd=16, page=4)
    w = wl.reuse_workload("ident", lay, n_chunks=3, T=[9, 4, 13],
                          placements=[(0, 0, 1, 0), (1, 0, 12, 0), (2, 1, 3, 0)], m=0, l0=0,
                          l1=0, seed=5, extra_pages=2)
    for c, it in enumerate(w.items):
        for name in ("canon_k", "canon_v"):
            t = getattr(it, name)
            L, T, W = t.shape
            code = (torch.arange(L).view(L, 1, 1) * 4096 + torch.arange(T).view(1, T, 1) * 64
                    + torch.arange(W).view(1, 1, W) + c * 16384).to(torch.int32)
            bits = (code & 0x7FFF) | (0x8000 if name == "canon_v" else 0)
            bits = bits.to(torch.int32)
            bits[0, 0, 0] = 0x8000            # -0
            bits[0, 0, 1] = 0x7FC3            # NaN with payload
            setattr(it, name, bits.to(torch.int16).view(torch.bfloat16))
    h = km.create(lay)
    k, v, status, _ = tl.run_batch(h, lay, tl.to_device_items(w.items), w.page_table,
                                   w.num_slots)
    assert status == 0
    kb, vb = wl.bf16_bits(k), wl.bf16_bits(v)
    wk = np.full_like(kb, wl.POOL_SENTINEL_BITS)
    wv = wk.copy()
    pt = w.page_table.numpy()
    for it in w.items:
        sl = tl.slots_of(pt, it.req, it.start_tok, it.num_tokens, 4)
        wk[:, sl] = wl.bf16_bits(it.canon_k)
        wv[:, sl] = wl.bf16_bits(it.canon_v)
    np.testing.assert_array_equal(kb, wk)
    np.testing.assert_array_equal(vb, wv)


def _relocate_case(lay, delta, seed=3):
    g = torch.Generator().manual_seed(seed)
    n_req, pages_per_req = 3, 12
    pt = wl.shuffled_page_table(n_req, pages_per_req, g, n_req * pages_per_req + 4)
    num_slots = (n_req * pages_per_req + 4) * lay.page_size
    k = wl.normal_bf16((lay.num_layers, num_slots, lay.row_k), 1.0, g, "cpu")
    spans = [(0, 3, 90), (1, 16, 100), (2, 0, 1)]
    before = wl.bf16_bits(k)
    kd = k.cuda()
    vd = None
    if lay.kind == wl.GQA:  # a V tensor must be given for GQA; it is never touched
        vd = torch.full((1, 1, 8), 7, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    pool = km.Pool(kd, vd, pt.cuda(), num_slots)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    h = km.create(lay)
    for req, start, T in spans:
        km.kamera_relocate(h, pool, req, start, T, delta, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    if vd is not None:
        assert torch.all(vd.view(torch.int16) == 7)
    want = before.copy()
    for req, start, T in spans:
        ora.relocate(lay, want, pt.numpy(), req, start, T, delta)
    got = wl.bf16_bits(kd)
    return before, got, want, pt.numpy(), spans


def _rotation_tolerance(lay, x, y):
    """ulp_bf16(y) + 8 * 2^-24 * (|a| + |b|) per rotated element."""
    S = np.abs(x).copy()
    for c0, d in ora.rope_bands(lay):
        ia, ib = ora.rope_pairs(d, lay.rope_style)
        ab = np.abs(x[:, c0 + ia]) + np.abs(x[:, c0 + ib])
        S[:, c0 + ia] = ab
        S[:, c0 + ib] = ab
    return ora.bf16_ulp(y) + 8 * 2.0 ** -24 * S


@pytest.mark.parametrize("style", [wl.NEOX_HALF, wl.INTERLEAVED])
@pytest.mark.parametrize("delta", [-576, 1, 131071])
def test_relocate_gqa_in_place(style, delta):
    lay = gqa_layout(L=2, H=4, hd=128, style=style, theta=1e4)
    before, got, want, pt, spans = _relocate_case(lay, delta)
    touched = np.zeros(got.shape[1], bool)
    for req, start, T in spans:
        touched[tl.slots_of(pt, req, start, T, 16)] = True
    np.testing.assert_array_equal(got[:, ~touched], before[:, ~touched])
    for layer in range(2):
        x = ora.bf16_to_f64(before[layer, touched])
        y = x.copy()
        for c0, d in ora.rope_bands(lay):
            y[:, c0:c0 + d] = ora.rotate_band(x[:, c0:c0 + d], delta, 1e4, style)
        g = ora.bf16_to_f64(got[layer, touched])
        assert np.all(np.abs(g - y) <= _rotation_tolerance(lay, x, y))
        r = ora.bf16_to_f64(want[layer, touched])
        assert np.linalg.norm(g - r) / np.linalg.norm(r) < 1e-3


@pytest.mark.parametrize("style", [wl.NEOX_HALF, wl.INTERLEAVED])
def test_relocate_mla_only_kpe(style):
    lay = mla_layout(L=2, style=style)
    before, got, want, pt, spans = _relocate_case(lay, -12345)
    np.testing.assert_array_equal(got[:, :, :512], before[:, :, :512])
    diff = got[:, :, 512:] != want[:, :, 512:]
    # the GPU rounds float32 results; allow one-ulp disagreements with the float64 oracle
    gv, wv = ora.bf16_to_f64(got[:, :, 512:]), ora.bf16_to_f64(want[:, :, 512:])
    assert np.all(np.abs(gv - wv)[diff] <= ora.bf16_ulp(wv)[diff])
    assert diff.mean() < 0.05


def test_relocate_delta_zero_is_a_no_op():
    lay = gqa_layout(L=1, H=1, hd=16)
    before, got, _, _, _ = _relocate_case(lay, 0)
    np.testing.assert_array_equal(got, before)


@pytest.mark.parametrize("theta,d", [(1e4, 64), (1e6, 128), (5e6, 128)])
def test_rope_phases_range_reduction(theta, d):
    lay = gqa_layout(H=1, hd=d, theta=theta)
    h = km.create(lay)
    # |delta| up to 2^31: the Q0.64 table then carries < 2^-33 turns of error
    deltas = np.array([0, 1, -1, 576, -576, 1000, 2048, 32767, -32768, 65536, 131071, -131071,
                       1 << 20, -(1 << 24) + 7, (1 << 31) - 1, -(1 << 31)], dtype=np.int64)
    out = torch.empty(len(deltas), d // 2, 2, dtype=torch.float32, device="cuda")
    km.kamera_rope_phases(h, torch.from_numpy(deltas).cuda(), out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    want = phase_reference(theta, d, deltas)
    bad = np.argwhere(np.abs(got - want) > 2.0 ** -22)
    assert bad.size == 0, [(int(deltas[a]), int(i), got[a, i], want[a, i]) for a, i, _ in bad[:5]]


def phase_reference(theta, d, deltas):
    """(cos, sin) of δ·inv_freq_i with the angle reduced exactly: δ times the float64 inv_freq_i
    as a rational number of turns of the float64 2π, the fractional turn taken exactly."""
    import math
    from fractions import Fraction
    inv = [Fraction(float(x)) for x in ora.inv_freq(theta, d)]
    two_pi = Fraction(2 * math.pi)
    out = np.empty((len(deltas), d // 2, 2))
    for a, dl in enumerate(deltas):
        for i, f in enumerate(inv):
            turns = Fraction(int(dl)) * f / two_pi
            frac = float(turns - math.floor(turns))
            out[a, i] = (math.cos(2 * math.pi * frac), math.sin(2 * math.pi * frac))
    return out


@pytest.mark.parametrize("workload", ["tiny", "reorder", "mla_recall", "sliding_window",
                                      "recall_sweep"])
def test_rope_phases_every_offset_of_the_reference_workloads(workload):
    # every (δ, pair) the five reference workloads use, with their θ and rotary width, against
    # the exactly reduced angle; 2^-22 absolute: one float32 ulp near 1 of the sincospi result
    # plus the Q0.64 table's |δ|·2^-65 turns
    theta, d, deltas = {
        "tiny": (1e4, 64, [1000]),
        "reorder": (1e6, 128, [0, 1024, 2048]),
        "mla_recall": (1e4, 64, wl.config3_deltas()),
        "sliding_window": (1e4, 128, [-576]),
        "recall_sweep": (1e6, 128, wl.config5_deltas()),
    }[workload]
    h = km.create(gqa_layout(H=1, hd=d, theta=theta))
    dl = np.asarray(deltas, dtype=np.int64)
    out = torch.empty(len(dl), d // 2, 2, dtype=torch.float32, device="cuda")
    km.kamera_rope_phases(h, torch.from_numpy(dl).cuda(), out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    want = phase_reference(theta, d, dl)
    bad = np.argwhere(np.abs(got - want) > 2.0 ** -22)
    assert bad.size == 0, [(int(dl[a]), int(i), got[a, i], want[a, i]) for a, i, _ in bad[:5]]


def test_empty_inputs_launch_nothing():
    lay = gqa_layout(L=1, H=1, hd=16)
    h = km.create(lay)
    k, v = tl.sentinel_pool(lay, 64)
    pt = torch.arange(4, dtype=torch.int32, device="cuda").view(1, 4)
    pool = km.Pool(k, v, pt, 64)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_items = torch.zeros(64, dtype=torch.uint8, device="cuda")
    km.kamera_batch_reuse(h, d_items, 0, 16, 0, pool, status)
    km.kamera_relocate(h, pool, 0, 0, 0, 5, status)
    c = torch.zeros(1, 0, 16, dtype=torch.bfloat16, device="cuda")
    it = wl.Item(canon_k=c, canon_v=c, patch_u=None, patch_vt=None, delta=3, num_tokens=0,
                 req=0, start_tok=0)
    km.kamera_reuse(h, it, pool, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.all(k.view(torch.int16) == wl.POOL_SENTINEL_BITS)


# ------------------------------------------------------------------------------------------
# reversible switch: patch re-added (and removed) in place on cached rows
# ------------------------------------------------------------------------------------------

def _inplace_expected(lay, before_k, before_v, pt, it, sign):
    """Oracle result of one in-place add on a host copy of the pools, plus the float64 values
    and error scale of the touched rows (for the tolerance)."""
    k, v = before_k.copy(), None if before_v is None else before_v.copy()
    u = wl.bf16_bits(it.patch_u)
    vt = wl.bf16_bits(it.patch_vt)
    ora.patch_inplace(lay, k, v, pt, it.req, it.start_tok, it.num_tokens, u, vt, it.patch_m,
                      it.patch_l0, it.patch_l1, sign)
    slots = tl.slots_of(pt, it.req, it.start_tok, it.num_tokens, lay.page_size)
    vals, mags = {}, {}
    for layer in range(it.patch_l0, it.patch_l1):
        li = layer - it.patch_l0
        for ch in range(2 if lay.kind == wl.GQA else 1):
            pool = before_k if ch == 0 else before_v
            x = ora.bf16_to_f64(pool[layer, slots])
            y, s = x.copy(), np.abs(x)
            for c0, w, g in ora.channel_groups(lay, ch):
                uu = ora.factor_f64(u[li][g])
                vv = ora.factor_f64(ora.vt_of_group(lay, vt[li], it.patch_m, g))
                y[:, c0:c0 + w] += sign * (uu @ vv)
                s[:, c0:c0 + w] += np.abs(uu) @ np.abs(vv)
            vals[(layer, ch)], mags[(layer, ch)] = y, s
    return k, v, slots, vals, mags


def _check_inplace(lay, it, got_k, got_v, want_k, want_v, slots, vals, mags):
    m = it.patch_m
    for (layer, ch), y in vals.items():
        got = ora.bf16_to_f64((got_k if ch == 0 else got_v)[layer, slots])
        tol = ora.bf16_ulp(y) + (2 * m + 8) * 2.0 ** -24 * mags[(layer, ch)]
        assert np.all(np.abs(got - y) <= tol), (layer, ch)
    # everything else: the bytes the oracle leaves (untouched rows and layers)
    mask = np.ones(want_k.shape[:2], dtype=bool)
    for layer in range(it.patch_l0, it.patch_l1):
        mask[layer, slots] = False
    np.testing.assert_array_equal(got_k[mask], want_k[mask])
    if want_v is not None:
        np.testing.assert_array_equal(got_v[mask], want_v[mask])


@pytest.mark.parametrize("kind,m", [("gqa", 8), ("gqa", 12), ("gqa", 32), ("gqai", 16),
                                    ("mla", 32), ("mla", 24)])
def test_patch_inplace_add_then_remove(kind, m):
    lay = {"gqa": gqa_layout(), "gqai": gqa_layout(style=wl.INTERLEAVED),
           "mla": mla_layout()}[kind]
    w = ragged(lay, m, f"inplace{kind}{m}")
    h = km.create(lay)
    items = tl.to_device_items(w.items)
    clean = [dataclasses.replace(it, patch_m=0, patch_l0=0, patch_l1=0, patch_u=None,
                                 patch_vt=None) for it in items]
    k, v, status, (_, pt_dev) = tl.run_batch(h, lay, clean, w.page_table, w.num_slots)
    assert status == 0
    pt = w.page_table.numpy()
    pool = km.Pool(k, v, pt_dev, w.num_slots)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for it in items:
        if it.num_tokens < 2:
            continue
        for sign in (1, -1):
            before_k = wl.bf16_bits(k)
            before_v = None if v is None else wl.bf16_bits(v)
            km.kamera_patch_inplace(h, pool, it.req, it.start_tok, it.num_tokens, it.patch_u,
                                    it.patch_vt, it.patch_m, it.patch_l0, it.patch_l1, sign, st)
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            want = _inplace_expected(lay, before_k, before_v, pt, it, sign)
            _check_inplace(lay, it, wl.bf16_bits(k), None if v is None else wl.bf16_bits(v),
                           *want)


def test_patch_inplace_on_clean_view_matches_reuse_with_patch():
    # δ = 0: the clean view is an exact copy, so re-adding the patch must give the bytes the
    # patched reuse writes (both round x + U V_m^T once, on the same kernel path)
    lay = gqa_layout(L=3, H=2, hd=128)
    w = wl.reuse_workload("sw0", lay, n_chunks=2, T=[200, 64],
                          placements=[(0, 0, 0, 0), (1, 1, 16, 0)], m=16, l0=1, l1=3, seed=9,
                          strong=True, patch_per_item=True)
    h = km.create(lay)
    items = tl.to_device_items(w.items)
    clean = [dataclasses.replace(it, patch_m=0, patch_l0=0, patch_l1=0, patch_u=None,
                                 patch_vt=None) for it in items]
    k, v, status, (_, pt_dev) = tl.run_batch(h, lay, clean, w.page_table, w.num_slots)
    assert status == 0
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = km.Pool(k, v, pt_dev, w.num_slots)
    for it in items:
        km.kamera_patch_inplace(h, pool, it.req, it.start_tok, it.num_tokens, it.patch_u,
                                it.patch_vt, it.patch_m, it.patch_l0, it.patch_l1, 1, st)
    k2, v2, status2, _ = tl.run_batch(h, lay, items, w.page_table, w.num_slots)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and status2 == 0
    assert torch.equal(k.view(torch.int16), k2.view(torch.int16))
    assert torch.equal(v.view(torch.int16), v2.view(torch.int16))


@pytest.mark.parametrize("kind", ["gqa", "mla"])
def test_batch_patch_inplace_matches_oracle_and_single_calls(kind):
    lay = gqa_layout() if kind == "gqa" else mla_layout()
    w = ragged(lay, 16, f"binplace{kind}")
    h = km.create(lay)
    items = tl.to_device_items(w.items)
    clean = [dataclasses.replace(it, patch_m=0, patch_l0=0, patch_l1=0, patch_u=None,
                                 patch_vt=None) for it in items]
    k, v, status, (_, pt_dev) = tl.run_batch(h, lay, clean, w.page_table, w.num_slots)
    assert status == 0
    k1, v1 = k.clone(), None if v is None else v.clone()
    before_k, before_v = wl.bf16_bits(k), None if v is None else wl.bf16_bits(v)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_items = km.pack_items(items).cuda()
    km.kamera_batch_patch_inplace(h, d_items, len(items), max(it.num_tokens for it in items), 16,
                                  km.Pool(k, v, pt_dev, w.num_slots), -1, st)
    for it in items:  # the same edits one chunk at a time
        km.kamera_patch_inplace(h, km.Pool(k1, v1, pt_dev, w.num_slots), it.req, it.start_tok,
                                it.num_tokens, it.patch_u, it.patch_vt, it.patch_m, it.patch_l0,
                                it.patch_l1, -1, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(k.view(torch.int16), k1.view(torch.int16))
    if v is not None:
        assert torch.equal(v.view(torch.int16), v1.view(torch.int16))
    # against the oracle, item by item (items cover disjoint rows)
    pt = w.page_table.numpy()
    want_k, want_v = before_k.copy(), None if before_v is None else before_v.copy()
    gk, gv = wl.bf16_bits(k), None if v is None else wl.bf16_bits(v)
    for it in items:
        res = _inplace_expected(lay, want_k, want_v, pt, it, -1)
        want_k, want_v = res[0], res[1]
        for (layer, ch), y in res[3].items():
            got = ora.bf16_to_f64((gk if ch == 0 else gv)[layer, res[2]])
            tol = ora.bf16_ulp(y) + (2 * 16 + 8) * 2.0 ** -24 * res[4][(layer, ch)]
            assert np.all(np.abs(got - y) <= tol)


def test_batch_patch_inplace_rejects_a_bad_item_on_device():
    lay = gqa_layout()
    w = ragged(lay, 8, "binplacebad")
    h = km.create(lay)
    items = tl.to_device_items(w.items)
    k, v, status, (_, pt_dev) = tl.run_batch(h, lay, items, w.page_table, w.num_slots)
    assert status == 0
    before = k.clone()
    bad = [dataclasses.replace(items[2], req=99)]  # a request outside the page table
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    km.kamera_batch_patch_inplace(h, km.pack_items(bad).cuda(), 1, 512, 8,
                                  km.Pool(k, v, pt_dev, w.num_slots), 1, st)
    torch.cuda.synchronize()
    assert int(st.item()) == km.KAMERA_DEVICE_BAD_ITEM
    assert torch.equal(k.view(torch.int16), before.view(torch.int16))
