"""Helpers shared by the GPU parity tests: run the library through the C ABI on seeded
workloads and compare with the float64 oracle.

Tolerance (per element, for every column some arithmetic touches):

    |gpu - y| <= ulp_bf16(y) + (2m + 8) * 2^-24 * S

y is the oracle's exact float64 value, S the oracle's error scale (|a|+|b| on rotated pairs,
|x| elsewhere, plus Σ_j |U_tj Vt_jc|). The first term is the "one bf16 ulp" of the pages
(Kamera §6 "Recompute-free on a live engine"); the second bounds the float32 evaluation
(rotation: a few roundings plus float32 cos/sin error; rank-m accumulation: at most m+1
roundings, doubled for truncating accumulators) and only matters under cancellation. Columns
no arithmetic touches must be bit-exact, and every (item, layer, channel) must also meet a
relative Frobenius error <= 1e-3 against the oracle's bf16 result.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import position_independent_multimodal_gb300 as km
import workloads as wl
from oracle import kamera_oracle as ora

REL_FROB = 1e-3


class LazyLayers:
    """Indexable view of a device tensor [L][...] that copies one layer to host bits on
    demand (the oracle reads ``x[layer]``)."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, l):
        return wl.bf16_bits(self.t[l])

    def __len__(self):
        return self.t.shape[0]


def oracle_item(it: wl.Item, lazy: bool = False):
    conv = (lambda t: None if t is None else LazyLayers(t)) if lazy else \
        (lambda t: None if t is None else wl.bf16_bits(t))
    return ora.as_item(canon_k=conv(it.canon_k), canon_v=conv(it.canon_v),
                       patch_u=conv(it.patch_u), patch_vt=conv(it.patch_vt), delta=it.delta,
                       num_tokens=it.num_tokens, req=it.req, start_tok=it.start_tok,
                       patch_m=it.patch_m, patch_l0=it.patch_l0, patch_l1=it.patch_l1,
                       delta_h=it.delta_h, delta_w=it.delta_w)


def sentinel_pool(layout: wl.Layout, num_slots: int, device="cuda"):
    k = torch.full((layout.num_layers, num_slots, layout.row_k), wl.POOL_SENTINEL_BITS,
                   dtype=torch.int16, device=device).view(torch.bfloat16)
    v = None
    if layout.kind == wl.GQA:
        v = torch.full((layout.num_layers, num_slots, layout.row_v), wl.POOL_SENTINEL_BITS,
                       dtype=torch.int16, device=device).view(torch.bfloat16)
    return k, v


def to_device_items(items, device="cuda", keep_sharing=True):
    """Items with their tensors on the device. Tensors that several host items share stay
    shared (one device copy), as a caller's chunk store would be, unless ``keep_sharing`` is
    False (every item gets its own copies, so no two items name the same rows)."""
    out = []
    copies = {}

    def mv(t):
        if t is None:
            return None
        if not keep_sharing:
            return t.to(device)
        if id(t) not in copies:
            copies[id(t)] = (t, t.to(device))
        return copies[id(t)][1]

    for it in items:
        out.append(dataclasses.replace(it, canon_k=mv(it.canon_k), canon_v=mv(it.canon_v),
                                       patch_u=mv(it.patch_u), patch_vt=mv(it.patch_vt)))
    return out


def run_batch(handle, layout, items, page_table, num_slots, pools=None, max_m=None,
              max_tokens=None, device="cuda"):
    """kamera_batch_reuse over device items; returns (k_pool, v_pool, status)."""
    k, v = pools if pools is not None else sentinel_pool(layout, num_slots, device)
    pt = page_table.to(device)
    pool = km.Pool(k, v, pt, num_slots)
    d_items = km.pack_items(items).to(device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    mm = max_m if max_m is not None else max([it.patch_m for it in items] + [0])
    mt = max_tokens if max_tokens is not None else max([it.num_tokens for it in items] + [0])
    km.kamera_batch_reuse(handle, d_items, len(items), mt, mm, pool, status)
    torch.cuda.synchronize()
    return k, v, int(status.item()), (d_items, pt)


def run_single(handle, layout, items, page_table, num_slots, device="cuda"):
    k, v = sentinel_pool(layout, num_slots, device)
    pt = page_table.to(device)
    pool = km.Pool(k, v, pt, num_slots)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    for it in items:
        km.kamera_reuse(handle, it, pool, status)
    torch.cuda.synchronize()
    return k, v, int(status.item())


@dataclasses.dataclass
class Stats:
    elems: int = 0
    computed: int = 0
    not_rne_equal: int = 0
    max_ulps: float = 0.0
    worst_rel_frob: float = 0.0

    def add(self, other: "Stats"):
        self.elems += other.elems
        self.computed += other.computed
        self.not_rne_equal += other.not_rne_equal
        self.max_ulps = max(self.max_ulps, other.max_ulps)
        self.worst_rel_frob = max(self.worst_rel_frob, other.worst_rel_frob)


def check_rows(layout, oitem, layer: int, ch: int, tokens, got_bits: np.ndarray) -> Stats:
    """Compare the GPU rows of (item, layer, channel) at ``tokens`` with the oracle."""
    vals, copy_mask = ora.reuse_layer(layout, oitem, layer, ch, tokens)
    want_bits = ora.reuse_layer_bits(layout, oitem, layer, ch, tokens)
    st = Stats(elems=got_bits.size)
    # untouched columns: byte copies
    if copy_mask.any():
        np.testing.assert_array_equal(got_bits[:, copy_mask], want_bits[:, copy_mask],
                                      err_msg=f"copy columns differ (layer {layer}, ch {ch})")
    comp = ~copy_mask
    if not comp.any():
        return st
    g = ora.bf16_to_f64(got_bits[:, comp])
    y = vals[:, comp]
    S = ora.magnitude_layer(layout, oitem, layer, ch, tokens)[:, comp]
    m = oitem.patch_m if ora.layer_patched(oitem, layer) else 0
    tol = ora.bf16_ulp(y) + (2 * m + 8) * 2.0 ** -24 * S
    err = np.abs(g - y)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"layer {layer} ch {ch}: {int(bad.sum())} elements outside tolerance; first "
            f"{[(int(i), int(j), float(g[i, j]), float(y[i, j]), float(tol[i, j])) for i, j in idx]}")
    st.computed = int(comp.sum()) * got_bits.shape[0]
    st.not_rne_equal = int((got_bits[:, comp] != want_bits[:, comp]).sum())
    st.max_ulps = float(np.max(err / ora.bf16_ulp(y)))
    # relative Frobenius error against the oracle's own bf16 result: rounding to bf16 alone
    # moves a layer by ~1.6e-3 (RMS) from the exact values, so the bound compares outputs
    r = ora.bf16_to_f64(want_bits[:, comp])
    nr = np.linalg.norm(r)
    rel = np.linalg.norm(g - r) / nr if nr > 0 else np.linalg.norm(g - r)
    st.worst_rel_frob = float(rel)
    assert rel <= REL_FROB, f"layer {layer} ch {ch}: relative Frobenius error {rel:.3e}"
    return st


def mini_item(layout, it: wl.Item, layer: int, toks: np.ndarray):
    """An oracle item holding only ``toks`` rows of one layer (host bits), so a sample of a
    full-size item is checked without copying the whole item to the host."""
    idx = torch.as_tensor(np.asarray(toks), device=it.canon_k.device)
    ck = {layer: wl.bf16_bits(it.canon_k[layer].index_select(0, idx))}
    cv = None if it.canon_v is None else {layer: wl.bf16_bits(it.canon_v[layer].index_select(0, idx))}
    pu = pv = None
    if it.patch_m > 0 and it.patch_l0 <= layer < it.patch_l1:
        li = layer - it.patch_l0
        pu = {li: [wl.bf16_bits(it.patch_u[li, g].index_select(0, idx)) for g in range(2)]}
        pv = {li: wl.bf16_bits(it.patch_vt[li])}
    return ora.as_item(canon_k=ck, canon_v=cv, patch_u=pu, patch_vt=pv, delta=it.delta,
                       num_tokens=len(toks), req=it.req, start_tok=0, patch_m=it.patch_m,
                       patch_l0=it.patch_l0, patch_l1=it.patch_l1, delta_h=it.delta_h,
                       delta_w=it.delta_w)


def check_sampled(layout, it: wl.Item, layer: int, ch: int, toks, pool: torch.Tensor,
                  page_table: np.ndarray) -> Stats:
    """Check the rows of sampled tokens of one (item, layer, channel) in a device pool."""
    toks = np.asarray(sorted(set(int(t) for t in toks)))
    logical = it.start_tok + toks
    sl = (page_table[it.req, logical // layout.page_size].astype(np.int64) * layout.page_size
          + logical % layout.page_size)
    got = wl.bf16_bits(pool[layer].index_select(0, torch.as_tensor(sl, device=pool.device)))
    return check_rows(layout, mini_item(layout, it, layer, toks), layer, ch, None, got)


def slots_of(page_table: np.ndarray, req: int, start: int, T: int, page: int) -> np.ndarray:
    toks = start + np.arange(T)
    return page_table[req, toks // page].astype(np.int64) * page + toks % page


def check_full(layout, items, page_table, k_pool, v_pool) -> Stats:
    """Every slot of both pools: written rows against the oracle, all others the sentinel."""
    pt = page_table.cpu().numpy()
    kb = wl.bf16_bits(k_pool)
    vb = wl.bf16_bits(v_pool) if v_pool is not None else None
    written = np.zeros(kb.shape[1], dtype=bool)
    st = Stats()
    for it in items:
        oi = oracle_item(it)
        sl = slots_of(pt, it.req, it.start_tok, it.num_tokens, layout.page_size)
        assert not written[sl].any(), "test workload maps two tokens to one slot"
        written[sl] = True
        for layer in range(layout.num_layers):
            for ch in range(2 if layout.kind == wl.GQA else 1):
                pool = kb if ch == 0 else vb
                st.add(check_rows(layout, oi, layer, ch, None, pool[layer, sl]))
    assert np.all(kb[:, ~written] == wl.POOL_SENTINEL_BITS), "stray writes in the K pool"
    if vb is not None:
        assert np.all(vb[:, ~written] == wl.POOL_SENTINEL_BITS), "stray writes in the V pool"
    return st
