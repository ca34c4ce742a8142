"""Batches whose items share a chunk (Kamera §5 "Reorder": one orbit patch serves every
ordering of a chunk). kamera_batch_reuse reads and computes such rows once per group and
writes them to every member's slots; the bytes must be exactly those of separate
kamera_reuse calls (which never group), and match the float64 oracle on every slot.

Cases: all six orderings of three ragged chunks behind an unaligned prefix (members that
share the offset on K, all placements of a chunk on V), GQA with 64- and 128-column tiles and
MLA (only the k_pe tile turns), ranks 0 / 8 / 32 and a CUDA-core rank, more items than one
share block, an invalid item with the same sources ahead of its group, an out-of-range page
in one member, per-item patches over one canonical, and M-RoPE items that share δ but not δ_h.
"""
import dataclasses
import itertools

import numpy as np
import pytest
import torch

import position_independent_multimodal_gb300 as km
import workloads as wl
from tests import kamera_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda(cuda_ok):
    return cuda_ok


def gqa(L=3, H=2, hd=64, page=16):
    return wl.Layout(kind=wl.GQA, num_layers=L, page_size=page, num_kv_heads=H, head_dim=hd,
                     rope_dim=hd, rope_style=wl.NEOX_HALF, rope_theta=1e4)


def mla(L=3):
    return wl.Layout(kind=wl.MLA, num_layers=L, page_size=16, latent_dim=512, rope_dim=64,
                     rope_style=wl.NEOX_HALF, rope_theta=1e4)


def orderings(layout, m, name, Ts=(130, 256, 77), prefix=5, patch_per_item=False):
    """Three chunks in all six orderings, one request per ordering, after a ``prefix``-token
    prefix; a chunk stored at position 0 and placed at logical token s has δ = s."""
    placements = []
    for r, perm in enumerate(itertools.permutations(range(3))):
        s = prefix
        for c in perm:
            placements.append((c, r, s, s))
            s += Ts[c]
    return wl.reuse_workload(name, layout, n_chunks=3, T=list(Ts), placements=placements, m=m,
                             l0=1, l1=layout.num_layers, seed=3, strong=True,
                             patch_per_item=patch_per_item, extra_pages=2)


def batch_pools(w, items, options=None, **kw):
    h = km.create(w.layout, **(options or {}))
    return tl.run_batch(h, w.layout, items, w.page_table, w.num_slots, **kw)


def single_pools(w, items, options=None):
    h = km.create(w.layout, **(options or {}))
    return tl.run_single(h, w.layout, items, w.page_table, w.num_slots)


def same_bytes(a, b):
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def check_grouped(w, n_shared_min=1, options=None):
    items = tl.to_device_items(w.items)
    ptrs = {(it.canon_k.data_ptr(), it.delta) for it in items}
    assert len(ptrs) <= len(items) - n_shared_min, "the workload has no shared rows"
    k, v, status, _ = batch_pools(w, items, options)
    assert status == 0
    tl.check_full(w.layout, w.items, w.page_table, k, v)
    k1, v1, s1 = single_pools(w, items, options)
    assert s1 == 0
    same_bytes(k, k1)
    if v is not None:
        same_bytes(v, v1)
    # the same batch with every item on its own copies (no group forms) writes the same bytes
    k2, v2, s2, _ = batch_pools(w, tl.to_device_items(w.items, keep_sharing=False), options)
    assert s2 == 0
    same_bytes(k, k2)
    if v is not None:
        same_bytes(v, v2)


@pytest.mark.parametrize("m", [0, 8, 12, 32])
@pytest.mark.parametrize("shape", ["gqa64", "gqa128", "mla"])
def test_all_orderings_of_three_chunks(shape, m):
    lay = {"gqa64": gqa(), "gqa128": gqa(H=4, hd=128), "mla": mla()}[shape]
    check_grouped(orderings(lay, m, f"share{shape}{m}"), n_shared_min=4)


def test_more_items_than_one_share_block():
    # one 70-token chunk in 40 requests at three offsets: blocks of 32 and 8 items, each with
    # three K groups and one V group
    lay = gqa(L=2, H=4, hd=128)
    placements = [(0, r, 16 * (r % 3) + 1, [0, 700, -70000][r % 3]) for r in range(40)]
    w = wl.reuse_workload("share40", lay, n_chunks=1, T=70, placements=placements, m=16,
                          l0=0, l1=2, seed=4, strong=True, extra_pages=1)
    check_grouped(w, n_shared_min=30)


def test_per_item_patches_share_only_unpatched_layers():
    check_grouped(orderings(gqa(L=4), 16, "sharepp", patch_per_item=True), n_shared_min=4)


def test_mrope_items_share_delta_but_not_delta_h():
    lay = dataclasses.replace(gqa(L=2, H=4, hd=128), mrope_section=(16, 24, 24),
                              mrope_style=wl.MROPE_CONTIGUOUS)
    w = orderings(lay, 32, "sharemrope")
    # within each ordering h and w move with the position; the first request keeps them still
    w.items = [dataclasses.replace(it, delta_h=(0 if it.req == 0 else it.delta // 7),
                                   delta_w=-it.delta) for it in w.items]
    check_grouped(w, n_shared_min=4)


def test_invalid_item_ahead_of_its_group_is_skipped():
    # item 0 names the same rows and offset as items 1 and 2 but an unknown request: it is
    # reported and skipped, and the group it would have led is still written
    lay = gqa(L=2, H=4, hd=128)
    w = wl.reuse_workload("sharebad", lay, n_chunks=1, T=150,
                          placements=[(0, 0, 3, 40), (0, 1, 3, 40), (0, 2, 20, 40)], m=8,
                          l0=1, l1=2, seed=5, strong=True, extra_pages=1)
    items = tl.to_device_items(w.items)
    bad = dataclasses.replace(items[0], req=99)
    k, v, status, _ = batch_pools(w, [bad] + items[1:])
    assert status == km.KAMERA_DEVICE_BAD_ITEM
    k1, v1, s1 = single_pools(w, items[1:])
    assert s1 == 0
    same_bytes(k, k1)
    same_bytes(v, v1)
    tl.check_full(w.layout, w.items[1:], w.page_table, k, v)


def test_out_of_range_page_in_one_member():
    # two placements with the same rows and offset; one page of the second request points
    # outside the pool: only that member's rows on that page are skipped
    lay = gqa(L=2, H=4, hd=128)
    w = wl.reuse_workload("shareoob", lay, n_chunks=1, T=200,
                          placements=[(0, 0, 0, 9), (0, 1, 0, 9)], m=32, l0=1, l1=2, seed=6,
                          strong=True, extra_pages=1)
    pt = w.page_table.clone()
    pt[1, 3] = 10 ** 6                      # tokens 48..63 of request 1
    w = dataclasses.replace(w, page_table=pt)
    items = tl.to_device_items(w.items)
    k, v, status, _ = batch_pools(w, items)
    assert status == km.KAMERA_DEVICE_SLOT_OOB
    k1, v1, s1 = single_pools(w, items)
    assert s1 == km.KAMERA_DEVICE_SLOT_OOB
    same_bytes(k, k1)
    same_bytes(v, v1)
    kb = wl.bf16_bits(k)
    ptn = pt.numpy()
    oi = tl.oracle_item(w.items[0])
    sl = tl.slots_of(ptn, 0, 0, 200, 16)
    for layer in range(2):
        tl.check_rows(lay, oi, layer, 0, None, kb[layer, sl])
    changed = np.any(kb != wl.POOL_SENTINEL_BITS, axis=(0, 2))
    assert changed.sum() == 200 + 200 - 16


@pytest.mark.parametrize("m", [0, 16])
def test_interleaved_pairing_groups_in_the_copy_kernel(m):
    # interleaved pairs take the general patched-layer kernel (no groups there); unpatched
    # layers still go through the grouped copy kernel
    lay = dataclasses.replace(gqa(H=2, hd=64), rope_style=wl.INTERLEAVED)
    check_grouped(orderings(lay, m, f"shareil{m}"), n_shared_min=4)


@pytest.mark.parametrize("kind", ["gqa", "mla"])
def test_cuda_core_engine_with_shared_chunks(kind):
    # the CUDA-core patch engine (general kernel) beside the grouped copy kernel
    lay = gqa(H=4, hd=128) if kind == "gqa" else mla()
    check_grouped(orderings(lay, 16, f"sharefma{kind}"), n_shared_min=4,
                  options=dict(patch_engine=km.KAMERA_ENGINE_CUDA_CORES))


@pytest.mark.parametrize("runs", [(1, 1), (6, 8), (32, 3)])
def test_run_sizes_write_the_same_bytes(runs):
    # any run size (1: no groups) writes what separate calls write
    patched, unpatched = runs
    check_grouped(orderings(gqa(H=4, hd=128), 16, f"runs{patched}"), n_shared_min=4,
                  options=dict(share_run_patched=patched, share_run_unpatched=unpatched))
