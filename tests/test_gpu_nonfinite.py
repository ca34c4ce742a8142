"""Non-finite canonical values propagate as in IEEE arithmetic, element by element, through the
GPU path (a float64 oracle of the same definition decides every element).

+Inf, -Inf and NaN payloads are planted in the canonical rows of: a patched V tile, a patched K
tile whose offset is zero (nothing turns; the staged row is added to the patch), a patched K tile
that turns, an MLA c_KV tile and k_pe band on a patched layer, and unpatched layers (byte copies).
An element whose exact result is non-finite must come out NaN where the oracle gives NaN and the
same infinity where it gives one; every other element of the row, including the other columns of
its 16-column block, must stay finite and within the parity tolerance.
"""
import numpy as np
import pytest
import torch

import position_independent_multimodal_gb300 as km
import workloads as wl
from oracle import kamera_oracle as ora
from tests import kamera_testlib as tl

pytestmark = pytest.mark.gpu

# bit patterns planted: +Inf, -Inf, a quiet NaN with a payload, a negative NaN with a payload
PLANTS = [0x7F80, 0xFF80, 0x7FC3, 0xFFA1]


@pytest.fixture(scope="module", autouse=True)
def _cuda(cuda_ok):
    return cuda_ok


def plant(t: torch.Tensor, layer: int, seed: int):
    """Write the PLANTS patterns at seeded (token, column) positions of one layer of a bf16
    canonical tensor [L][T][row], several per 16-column block somewhere in the row."""
    rng = np.random.default_rng(seed)
    bits = t.view(torch.int16)
    T, row = t.shape[1], t.shape[2]
    for i in range(12):
        tok = int(rng.integers(0, T))
        col = int(rng.integers(0, row))
        v = PLANTS[i % len(PLANTS)]
        bits[layer, tok, col] = v - 0x10000 if v >= 0x8000 else v


def check(layout, items, page_table, k_pool, v_pool):
    pt = page_table.cpu().numpy()
    kb = wl.bf16_bits(k_pool)
    vb = wl.bf16_bits(v_pool) if v_pool is not None else None
    n_nonfinite = 0
    for it in items:
        oi = tl.oracle_item(it)
        sl = tl.slots_of(pt, it.req, it.start_tok, it.num_tokens, layout.page_size)
        for layer in range(layout.num_layers):
            for ch in range(2 if layout.kind == wl.GQA else 1):
                got = (kb if ch == 0 else vb)[layer, sl]
                vals, copy_mask = ora.reuse_layer(layout, oi, layer, ch)
                want = ora.reuse_layer_bits(layout, oi, layer, ch)
                if copy_mask.any():  # byte copies keep NaN payloads and signs
                    np.testing.assert_array_equal(got[:, copy_mask], want[:, copy_mask])
                comp = ~copy_mask
                if not comp.any():
                    continue
                y = vals[:, comp]
                with np.errstate(invalid="ignore"):
                    g = ora.bf16_to_f64(got[:, comp])
                fin = np.isfinite(y)
                n_nonfinite += int((~fin).sum())
                assert np.array_equal(np.isnan(g), np.isnan(y)), \
                    f"layer {layer} ch {ch}: NaN where the oracle has none, or the reverse"
                inf = np.isinf(y)
                assert np.array_equal(g[inf], y[inf]), f"layer {layer} ch {ch}: infinities differ"
                assert np.all(np.isfinite(g[fin])), f"layer {layer} ch {ch}: a finite result lost"
                S = ora.magnitude_layer(layout, oi, layer, ch)[:, comp]
                m = oi.patch_m if ora.layer_patched(oi, layer) else 0
                tol = ora.bf16_ulp(y) + (2 * m + 8) * 2.0 ** -24 * S
                assert np.all(np.abs(g[fin] - y[fin]) <= tol[fin]), \
                    f"layer {layer} ch {ch}: finite elements outside the tolerance"
    return n_nonfinite


def workload(layout, m, name):
    # chunk 0 placed at offset 0 (nothing turns) and chunk 1 moved by 1000, patched on layers
    # 1..L-1; layer 0 is unpatched (the copy kernel)
    placements = [(0, 0, 0, 0), (1, 0, 256, 1000), (0, 1, 16, 0)]
    w = wl.reuse_workload(name, layout, n_chunks=2, T=200, placements=placements, m=m, l0=1,
                          l1=layout.num_layers, seed=5, strong=True)
    cks = {id(it.canon_k): it.canon_k for it in w.items}
    cvs = {id(it.canon_v): it.canon_v for it in w.items if it.canon_v is not None}
    for i, t in enumerate(cks.values()):
        for layer in range(layout.num_layers):
            plant(t, layer, seed=100 * i + layer)
    for i, t in enumerate(cvs.values()):
        for layer in range(layout.num_layers):
            plant(t, layer, seed=1000 + 100 * i + layer)
    return w


@pytest.mark.parametrize("kind,m", [("gqa128", 32), ("gqa64", 16), ("mla", 32), ("gqa128", 12)])
@pytest.mark.parametrize("batch", [True, False])
def test_nonfinite_canonicals_propagate_element_by_element(kind, m, batch):
    if kind == "mla":
        lay = wl.Layout(kind=wl.MLA, num_layers=3, page_size=16, latent_dim=512, rope_dim=64,
                        rope_style=wl.NEOX_HALF, rope_theta=1e4)
    else:
        hd = 128 if kind == "gqa128" else 64
        lay = wl.Layout(kind=wl.GQA, num_layers=3, page_size=16, num_kv_heads=4 if hd == 128 else 2,
                        head_dim=hd, rope_dim=hd, rope_style=wl.NEOX_HALF, rope_theta=1e6)
    w = workload(lay, m, f"nonfinite{kind}{m}")
    h = km.create(lay)
    items = tl.to_device_items(w.items)
    if batch:
        k, v, status, _ = tl.run_batch(h, lay, items, w.page_table, w.num_slots)
    else:
        k, v, status = tl.run_single(h, lay, items, w.page_table, w.num_slots)
    assert status == 0
    assert check(lay, w.items, w.page_table, k, v) > 0
