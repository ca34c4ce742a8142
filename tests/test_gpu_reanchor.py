"""GPU parity of kamera_reanchor (keys stored before rotation, re-anchored at per-token request
positions; QV-PIC Eq. 2) against the float64 oracle, through the C ABI.

Every slot of both pools is checked: written rows against the oracle and all other slots
against the sentinel they were filled with. Rotated columns must be within
ulp_bf16(y) + 8·2⁻²⁴·S of the oracle's exact value y (S = |a| + |b| of the pair: one float32
rotation with float32 cos/sin, then one rounding); all other columns are byte copies.
"""
import dataclasses
from types import SimpleNamespace

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


GRIDS = [(1, 1, 1), (1, 1, 37), (1, 10, 13), (3, 10, 10)]          # T = 1, 37, 130, 300
PLACEMENTS = [(0, 0, 5, 0), (1, 0, 40, 3), (2, 1, 0, 100), (3, 2, 7, -50), (1, 1, 300, 7)]


def workload(layout, name, seed=0, random_positions=True):
    w = wl.anchor_workload(name, layout, grids=GRIDS, placements=PLACEMENTS, seed=seed,
                           extra_pages=2)
    if random_positions:
        # positions need not follow the grid: each token anywhere within ±2^20 (where the
        # float64 angle of the oracle stays exact to ~1e-10 rad)
        rng = np.random.default_rng(seed + 1)
        w.items = [dataclasses.replace(it, positions=torch.as_tensor(
            rng.integers(-(1 << 20), 1 << 20, tuple(it.positions.shape)), dtype=torch.int64))
            for it in w.items]
    return w


def run(w, items=None, pools=None):
    items = w.items if items is None else items
    lay = w.layout
    h = km.create(lay)
    k, v = pools if pools is not None else tl.sentinel_pool(lay, w.num_slots)
    dev_items = [dataclasses.replace(it, canon_k=it.canon_k.cuda(),
                                     canon_v=None if it.canon_v is None else it.canon_v.cuda(),
                                     positions=it.positions.cuda()) for it in items]
    d = km.pack_anchor_items(dev_items).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    km.kamera_reanchor(h, d, len(items), max(it.num_tokens for it in items),
                       km.Pool(k, v, w.page_table.cuda(), w.num_slots), status)
    torch.cuda.synchronize()
    return k, v, int(status.item()), dev_items


def oracle_item(it):
    return SimpleNamespace(canon_k=wl.bf16_bits(it.canon_k),
                           canon_v=None if it.canon_v is None else wl.bf16_bits(it.canon_v),
                           positions=it.positions.cpu().numpy(), num_tokens=it.num_tokens,
                           req=it.req, start_tok=it.start_tok)


def check_rows(lay, oi, layer, ch, got):
    vals, copy_mask = ora.reanchor_layer(lay, oi, layer, ch)
    canon = oi.canon_k if ch == 0 else oi.canon_v
    src = canon[layer]
    assert np.array_equal(got[:, copy_mask], src[:, copy_mask])
    if copy_mask.all():
        return 0
    x = ora.bf16_to_f64(src)
    mag = np.abs(x)
    for c0, d in ora.rope_bands(lay):
        ia, ib = ora.rope_pairs(d, lay.rope_style)
        ab = np.abs(x[:, c0 + ia]) + np.abs(x[:, c0 + ib])
        mag[:, c0 + ia] = ab
        mag[:, c0 + ib] = ab
    y = vals[:, ~copy_mask]
    g = ora.bf16_to_f64(got[:, ~copy_mask])
    tol = ora.bf16_ulp(y) + 8 * 2.0 ** -24 * mag[:, ~copy_mask]
    bad = ~(np.abs(g - y) <= tol)
    assert not bad.any(), (layer, ch, int(bad.sum()), np.argwhere(bad)[:3])
    return int((~copy_mask).sum()) * got.shape[0]


def check_all(w, k, v, skip=()):
    lay = w.layout
    pt = w.page_table.numpy()
    kb = wl.bf16_bits(k)
    vb = wl.bf16_bits(v) if v is not None else None
    written = np.zeros(kb.shape[1], dtype=bool)
    computed = 0
    for idx, it in enumerate(w.items):
        if idx in skip:
            continue
        oi = oracle_item(it)
        sl = tl.slots_of(pt, it.req, it.start_tok, it.num_tokens, lay.page_size)
        written[sl] = True
        for layer in range(lay.num_layers):
            for ch, pool in ((0, kb), (1, vb)):
                if pool is None:
                    continue
                computed += check_rows(lay, oi, layer, ch, pool[layer, sl])
    for pool in (kb, vb):
        if pool is not None:
            assert np.all(pool[:, ~written] == wl.POOL_SENTINEL_BITS)
    return computed


def gqa(H=2, hd=64, style=wl.NEOX_HALF, L=3, **kw):
    return wl.Layout(kind=wl.GQA, num_layers=L, page_size=16, num_kv_heads=H, head_dim=hd,
                     rope_dim=hd, rope_style=style, rope_theta=1e4, **kw)


@pytest.mark.parametrize("style", [wl.NEOX_HALF, wl.INTERLEAVED])
def test_reanchor_gqa_per_token_positions(style):
    w = workload(gqa(style=style), f"anc{style}")
    k, v, status, _ = run(w)
    assert status == 0
    assert check_all(w, k, v) > 0


def test_reanchor_layers_beyond_one_block_group():
    # 9 layers: a CTA takes seven, the next group the last two
    w = workload(gqa(H=1, L=9), "ancl9")
    k, v, status, _ = run(w)
    assert status == 0
    assert check_all(w, k, v) > 0


@pytest.mark.parametrize("mstyle,sections,H", [(wl.MROPE_CONTIGUOUS, (16, 24, 24), 4),
                                               (wl.MROPE_INTERLEAVED, (24, 20, 20), 8)])
def test_reanchor_mrope_coordinates(mstyle, sections, H):
    lay = gqa(H=H, hd=128, mrope_section=sections, mrope_style=mstyle)
    for random_positions in (False, True):  # grid coordinates, then arbitrary (t, h, w)
        w = workload(lay, f"ancm{mstyle}", random_positions=random_positions)
        assert w.items[0].positions.dim() == 2
        k, v, status, _ = run(w)
        assert status == 0
        assert check_all(w, k, v) > 0


def test_reanchor_mla_latent_copied_k_pe_rotated():
    lay = wl.Layout(kind=wl.MLA, num_layers=2, page_size=16, latent_dim=512, rope_dim=64,
                    rope_theta=1e4)
    w = workload(lay, "ancmla")
    k, _, status, _ = run(w)
    assert status == 0
    assert check_all(w, k, None) > 0


def test_reanchor_rejects_bad_items_and_out_of_range_pages():
    w = workload(gqa(), "ancbad")
    items = list(w.items)
    # item 1: positions not 8-byte aligned -> rejected on the device, nothing written
    pos = torch.zeros(items[1].num_tokens * 8 + 8, dtype=torch.uint8).cuda()
    bad = dataclasses.replace(items[1], positions=pos[4:].view(-1))
    k, v = tl.sentinel_pool(w.layout, w.num_slots)
    h = km.create(w.layout)
    dev = [dataclasses.replace(it, canon_k=it.canon_k.cuda(), canon_v=it.canon_v.cuda(),
                               positions=it.positions.cuda()) for it in items]
    dev[1] = dataclasses.replace(dev[1], positions=bad.positions)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    km.kamera_reanchor(h, km.pack_anchor_items(dev).cuda(), len(dev), 300,
                       km.Pool(k, v, w.page_table.cuda(), w.num_slots), status)
    torch.cuda.synchronize()
    assert int(status.item()) == km.KAMERA_DEVICE_BAD_ITEM
    check_all(w, k, v, skip=(1,))
    # a page id beyond the pool: those rows are skipped, the bit is set, the rest is written
    pt = w.page_table.clone()
    pt[2, 0] = 10 ** 6
    k2, v2 = tl.sentinel_pool(w.layout, w.num_slots)
    status.zero_()
    km.kamera_reanchor(h, km.pack_anchor_items(dev[:1]).cuda(), 1, 300,
                       km.Pool(k2, v2, pt.cuda(), w.num_slots), status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0  # item 0 (request 0) never touches request 2
    items3 = [dev[3]]  # request 2, tokens 7..306: page 0 holds tokens 7..15
    status.zero_()
    km.kamera_reanchor(h, km.pack_anchor_items(items3).cuda(), 1, 300,
                       km.Pool(k2, v2, pt.cuda(), w.num_slots), status)
    torch.cuda.synchronize()
    assert int(status.item()) == km.KAMERA_DEVICE_SLOT_OOB
    kb = wl.bf16_bits(k2)
    it = w.items[3]
    toks = np.arange(9, it.num_tokens)  # logical tokens 16.. onwards are on valid pages
    sl = tl.slots_of(pt.numpy(), it.req, it.start_tok, it.num_tokens, 16)[9:]
    oi = oracle_item(it)
    for layer in range(3):
        vals = ora.reanchor_layer_bits(w.layout, oi, layer, 0, tokens=toks)
        g = kb[layer, sl]
        assert np.all(np.abs(ora.bf16_to_f64(g) - ora.bf16_to_f64(vals)) <=
                      2 * ora.bf16_ulp(ora.bf16_to_f64(vals)) + 1e-30)
