"""Device-side error reporting, with the faults made on the host: a page-table entry that
points outside the pool, and batch items that break the item rules. The kernels must skip
exactly the affected rows or items, set the status bit, and write everything else correctly.
Nothing here can fault the GPU: every bad index is caught by the kernels' own checks before
any access."""
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


def small():
    lay = wl.Layout(kind=wl.GQA, num_layers=2, page_size=16, num_kv_heads=2, head_dim=64,
                    rope_dim=64, rope_style=wl.NEOX_HALF, rope_theta=1e4)
    return wl.reuse_workload("err", lay, n_chunks=3, T=[40, 64, 20],
                             placements=[(0, 0, 0, 9), (1, 1, 0, -9), (2, 2, 3, 100)], m=16,
                             l0=1, l1=2, seed=11, patch_per_item=True, extra_pages=2)


@pytest.mark.parametrize("bad_page", [-1, 10 ** 6])
def test_out_of_range_page_skips_its_rows(bad_page):
    w = small()
    pt = w.page_table.clone()
    pt[1, 2] = bad_page                     # tokens 32..47 of request 1
    h = km.create(w.layout)
    k, v, status, _ = tl.run_batch(h, w.layout, tl.to_device_items(w.items), pt, w.num_slots)
    assert status & km.KAMERA_DEVICE_SLOT_OOB
    kb, vb = wl.bf16_bits(k), wl.bf16_bits(v)
    ptn = pt.numpy()
    for idx, it in enumerate(w.items):
        oi = tl.oracle_item(it)
        toks = np.arange(it.num_tokens)
        ok = ~((idx == 1) & ((toks + it.start_tok) // 16 == 2))
        sl = tl.slots_of(np.where(ptn < 0, 0, np.minimum(ptn, 10 ** 5)), it.req, it.start_tok,
                         it.num_tokens, 16)
        for layer in range(2):
            for ch, pool in ((0, kb), (1, vb)):
                tl.check_rows(w.layout, oi, layer, ch, toks[ok], pool[layer, sl[ok]])
    # nothing else was written: count the slots that left the sentinel
    changed = np.any(kb != wl.POOL_SENTINEL_BITS, axis=(0, 2))
    assert changed.sum() == 40 + 64 - 16 + 20


@pytest.mark.parametrize("breakage", ["req", "canon_v", "rank", "tokens", "layers", "align"])
def test_bad_batch_item_is_skipped(breakage):
    w = small()
    items = tl.to_device_items(w.items)
    bad = items[1]
    if breakage == "req":
        bad.req = 99
    elif breakage == "canon_v":
        bad.canon_v = None
    elif breakage == "rank":
        bad.patch_m = 32                    # above max_patch_m given below
    elif breakage == "tokens":
        bad.num_tokens = 65                 # above max_tokens given below
    elif breakage == "layers":
        bad.patch_l1 = 3
    elif breakage == "align":
        # a canonical that starts 2 bytes into an allocation is not 16-byte aligned; the item
        # check rejects it before any load
        base = torch.empty(bad.canon_k.numel() + 8, dtype=torch.bfloat16, device="cuda")
        bad.canon_k = base[1:1 + bad.canon_k.numel()].view(bad.canon_k.shape)
    h = km.create(w.layout)
    k, v, status, _ = tl.run_batch(h, w.layout, items, w.page_table, w.num_slots, max_m=16,
                                   max_tokens=64)
    assert status == km.KAMERA_DEVICE_BAD_ITEM
    kb = wl.bf16_bits(k)
    ptn = w.page_table.numpy()
    sl_bad = tl.slots_of(ptn, 1, 0, 64, 16)
    assert np.all(kb[:, sl_bad] == wl.POOL_SENTINEL_BITS)
    for idx in (0, 2):
        it = w.items[idx]
        oi = tl.oracle_item(it)
        sl = tl.slots_of(ptn, it.req, it.start_tok, it.num_tokens, 16)
        for layer in range(2):
            tl.check_rows(w.layout, oi, layer, 0, None, kb[layer, sl])


def test_host_errors_raise_and_launch_nothing():
    w = small()
    h = km.create(w.layout)
    k, v = tl.sentinel_pool(w.layout, w.num_slots)
    pool = km.Pool(k, v, w.page_table.cuda(), w.num_slots)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    it = tl.to_device_items(w.items)[0]
    it.req = 7
    with pytest.raises(km.KameraError) as e:
        km.kamera_reuse(h, it, pool, status)
    assert e.value.status == km.KAMERA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(k.view(torch.int16) == wl.POOL_SENTINEL_BITS)
    assert int(status.item()) == 0
