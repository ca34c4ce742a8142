"""Parity at the full sizes of the five reference workloads, through the same C-ABI calls the
benchmark times. Sampled rows are compared with the float64 oracle one by one (the oracle
cannot redo a whole workload in seconds); whole-pool properties are checked on the device:
every slot of every request written, untouched rows unchanged, and the byte-copy columns
(V and the MLA latent on unpatched layers) equal to the canonical bytes."""
import numpy as np
import pytest
import torch

import position_independent_multimodal_gb300 as km
import workloads as wl
from oracle import kamera_oracle as ora
from tests import kamera_testlib as tl

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _cuda(cuda_ok):
    yield
    torch.cuda.empty_cache()


def run_batch(w, items, workspace=False):
    """The batch call over the items; with `workspace`, through a batch workspace (the
    persistent path the benchmark times), whose plan header is returned as well."""
    lay = w.layout
    k, v = tl.sentinel_pool(lay, w.num_slots)
    h = km.create(lay)
    ws = None
    if workspace:
        ws = torch.full((km.kamera_batch_workspace_bytes(h, len(items)),), 0xFF,
                        dtype=torch.uint8, device="cuda")
        km.kamera_set_batch_workspace(h, ws)
    pt = w.page_table.cuda()
    d_items = km.pack_items(items).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    max_t = max(it.num_tokens for it in items)
    max_m = max(it.patch_m for it in items)
    km.kamera_batch_reuse(h, d_items, len(items), max_t, max_m, km.Pool(k, v, pt, w.num_slots),
                          status)
    torch.cuda.synchronize()
    if workspace:
        return k, v, int(status.item()), ws[:28].view(torch.int32).cpu().tolist()
    return k, v, int(status.item())


def unwritten_rows(pool):
    return int((pool.view(torch.int16) == wl.POOL_SENTINEL_BITS).all(dim=-1).sum().item())


def item_slots(w, it):
    toks = it.start_tok + np.arange(it.num_tokens)
    pt = w.page_table.numpy()
    ps = w.layout.page_size
    return torch.as_tensor(pt[it.req, toks // ps].astype(np.int64) * ps + toks % ps, device="cuda")


def sample_tokens(rng, T, n=40):
    return np.unique(np.concatenate([[0, T - 1, 127, 128], rng.integers(0, T, n)]))


def check_units(w, items, k, v, n_units, seed, layers=None):
    rng = np.random.default_rng(seed)
    lay = w.layout
    pt = w.page_table.numpy()
    n_ch = 2 if lay.kind == wl.GQA else 1
    layer_pool = layers if layers is not None else range(lay.num_layers)
    st = tl.Stats()
    for _ in range(n_units):
        it = items[int(rng.integers(len(items)))]
        layer = int(rng.choice(list(layer_pool)))
        ch = int(rng.integers(n_ch))
        pool = k if ch == 0 else v
        st.add(tl.check_sampled(lay, it, layer, ch, sample_tokens(rng, it.num_tokens), pool, pt))
    return st


def test_config2_mrope_reorder_full():
    # the reorder workload with blocked 16|24|24 M-RoPE sections and different t / h,w offsets
    w = wl.config2_mrope(device="cuda")
    assert any(it.delta_h != it.delta for it in w.items)
    k, v, status = run_batch(w, w.items)
    assert status == 0
    assert unwritten_rows(k) == 0 and unwritten_rows(v) == 0
    st = check_units(w, w.items, k, v, 40, seed=12)
    assert st.computed > 0


def test_config2_gqa_reorder_full():
    w = wl.config2(device="cuda")
    k, v, status = run_batch(w, w.items)
    assert status == 0
    assert unwritten_rows(k) == 0 and unwritten_rows(v) == 0
    st = check_units(w, w.items, k, v, 40, seed=2)
    assert st.computed > 0
    # unpatched layers: V is a byte copy of the canonical values
    for it in w.items[:6]:
        sl = item_slots(w, it)
        for layer in (0, 7, 13):
            assert torch.equal(v[layer].index_select(0, sl), it.canon_v[layer])
    del k, v, w
    torch.cuda.empty_cache()


@pytest.mark.parametrize("make", [wl.config2, wl.config2_mrope], ids=["rope", "mrope"])
def test_config2_reorder_full_persistent(make):
    # the timed launch configuration: 14 patched layers x (9 K runs of 2 + 6 V runs of 3) =
    # 210 task rows of 8 token tiles x 4 column tiles, every row the same length, so the plan
    # deals two rows to each set and hands the tiles of the rest out one at a time
    w = make(device="cuda")
    k, v, status, head = run_batch(w, w.items, workspace=True)
    rows, tiles, _weight, s1, n_dyn, ntt, stride = head
    assert status == 0
    assert (rows, tiles, ntt) == (210, 6720, 8)
    # token-tile positions: whole rows to the sets, the rest claimed one at a time
    assert stride >= 1 and s1 % ntt == 0 and n_dyn > 0 and s1 + n_dyn == rows * ntt
    k0, v0, status0 = run_batch(w, w.items)
    assert status0 == 0
    assert torch.equal(k.view(torch.int16), k0.view(torch.int16))
    assert torch.equal(v.view(torch.int16), v0.view(torch.int16))
    del k0, v0
    torch.cuda.empty_cache()
    st = check_units(w, w.items, k, v, 40, seed=22, layers=range(14, 28))
    assert st.computed > 0
    del k, v, w
    torch.cuda.empty_cache()


def test_config3_mla_recall_full():
    w = wl.config3(device="cuda")
    k, _, status = run_batch(w, w.items)
    assert status == 0
    assert unwritten_rows(k) == 0
    check_units(w, w.items, k, None, 40, seed=3)
    # the latent c_KV is copied byte for byte on unpatched layers (0-12)
    for it in w.items[::8]:
        sl = item_slots(w, it)
        for layer in range(0, 13, 4):
            assert torch.equal(k[layer].index_select(0, sl)[:, :512], it.canon_k[layer][:, :512])
    del k, w
    torch.cuda.empty_cache()


def test_config4_sliding_window_survivors_full():
    w = wl.config4(device="cuda")
    lay = w.layout
    pt = w.page_table.numpy()
    rng = np.random.default_rng(4)
    ps = lay.page_size
    # sampled rows before the slide: survivor tokens and evicted-chunk tokens
    probes = []
    for _ in range(24):
        req = int(rng.integers(len(w.spans)))
        tok = int(rng.integers(0, w.meta["chunk"] * w.meta["window"]))
        layer = int(rng.integers(lay.num_layers))
        slot = int(pt[req, tok // ps]) * ps + tok % ps
        probes.append((req, tok, layer, slot, wl.bf16_bits(w.k_pool[layer, slot])))
    h = km.create(lay)
    vd = torch.zeros(1, 1, 8, dtype=torch.bfloat16, device="cuda")  # GQA needs a V; untouched
    pool = km.Pool(w.k_pool, vd, w.page_table.cuda(), w.num_slots)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for sp in w.spans:
        km.kamera_relocate(h, pool, sp.req, sp.start_tok, sp.num_tokens, sp.delta, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for req, tok, layer, slot, before in probes:
        got = wl.bf16_bits(w.k_pool[layer, slot])
        if tok < w.meta["chunk"]:  # the evicted chunk's rows are not touched
            np.testing.assert_array_equal(got, before)
            continue
        x = ora.bf16_to_f64(before)[None]
        y = x.copy()
        for c0, d in ora.rope_bands(lay):
            y[:, c0:c0 + d] = ora.rotate_band(x[:, c0:c0 + d], -w.meta["chunk"], lay.rope_theta,
                                              lay.rope_style)
        g = ora.bf16_to_f64(got)[None]
        S = np.abs(x).copy()
        for c0, d in ora.rope_bands(lay):
            ia, ib = ora.rope_pairs(d, lay.rope_style)
            S[:, c0 + ia] = S[:, c0 + ib] = np.abs(x[:, c0 + ia]) + np.abs(x[:, c0 + ib])
        assert np.all(np.abs(g - y) <= ora.bf16_ulp(y) + 8 * 2.0 ** -24 * S)
    del w, pool
    torch.cuda.empty_cache()


def test_config5_recall_sweep_full():
    w = wl.config5(device="cuda")
    Ls = w.meta["layer_slices"]
    for launch in range(w.meta["full_layout"].num_layers // Ls):
        items = wl.config5_launch_items(w, launch)
        k, v, status = run_batch(w, items)
        assert status == 0
        assert unwritten_rows(k) == 0 and unwritten_rows(v) == 0
        if launch in (0, 3, 4, 7):  # unpatched and patched slices
            check_units(w, items, k, v, 10, seed=50 + launch)
        del k, v
    del w
    torch.cuda.empty_cache()


def test_reanchor_full():
    # the QV-PIC re-anchoring workload at bench size, in the bench's single launch: every slot
    # written, sampled rows against the oracle (rotated columns within one ulp plus the float32
    # rotation bound, V byte copies)
    from types import SimpleNamespace
    w = wl.config_reanchor(device="cuda")
    lay = w.layout
    k, v = tl.sentinel_pool(lay, w.num_slots)
    h = km.create(lay)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    km.kamera_reanchor(h, km.pack_anchor_items(w.items).cuda(), len(w.items), 1024,
                       km.Pool(k, v, w.page_table.cuda(), w.num_slots), status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # every slot an item covers is written; only the 16-token prefix of each request is not
    uncovered = lay.num_layers * (w.num_slots - sum(it.num_tokens for it in w.items))
    assert unwritten_rows(k) == uncovered and unwritten_rows(v) == uncovered
    rng = np.random.default_rng(31)
    pt = w.page_table.numpy()
    for _ in range(24):
        it = w.items[int(rng.integers(len(w.items)))]
        layer = int(rng.integers(lay.num_layers))
        toks = sample_tokens(rng, it.num_tokens)
        idx = torch.as_tensor(toks, device="cuda")
        oi = SimpleNamespace(canon_k={layer: wl.bf16_bits(it.canon_k[layer].index_select(0, idx))},
                             canon_v={layer: wl.bf16_bits(it.canon_v[layer].index_select(0, idx))},
                             positions=it.positions.cpu().numpy()[toks], num_tokens=len(toks))
        sl = torch.as_tensor(pt[it.req, (it.start_tok + toks) // lay.page_size].astype(np.int64)
                             * lay.page_size + (it.start_tok + toks) % lay.page_size,
                             device="cuda")
        for ch, pool in ((0, k), (1, v)):
            got = wl.bf16_bits(pool[layer].index_select(0, sl))
            vals, copy_mask = ora.reanchor_layer(lay, oi, layer, ch)
            src = (oi.canon_k if ch == 0 else oi.canon_v)[layer]
            assert np.array_equal(got[:, copy_mask], src[:, copy_mask])
            if not copy_mask.all():
                x = ora.bf16_to_f64(src)
                S = np.abs(x)
                for c0, d in ora.rope_bands(lay):
                    ia, ib = ora.rope_pairs(d, lay.rope_style)
                    S[:, c0 + ia] = S[:, c0 + ib] = np.abs(x[:, c0 + ia]) + np.abs(x[:, c0 + ib])
                y = vals[:, ~copy_mask]
                g = ora.bf16_to_f64(got[:, ~copy_mask])
                assert np.all(np.abs(g - y) <= ora.bf16_ulp(y) + 8 * 2.0 ** -24 * S[:, ~copy_mask])
    del k, v, w
    torch.cuda.empty_cache()


def test_decode_attention_full():
    # decode attention over the reorder pool at bench size (6 requests x 3072 tokens, 28 query
    # heads over 4 KV heads), sampled layers, against float64 attention over the same pool
    from tests.test_gpu_attention import compare
    w = wl.config2(device="cuda")
    lay = w.layout
    k, v, status = run_batch(w, w.items)
    assert status == 0
    h = km.create(lay)
    reqs, hq, ctx = int(w.page_table.shape[0]), 28, 3 * 1024
    q = wl.normal_bf16((reqs, hq, lay.head_dim), 1.0, torch.Generator().manual_seed(8), "cpu")
    ws = torch.empty(km.kamera_decode_attention_workspace(h, reqs, hq, ctx), dtype=torch.uint8,
                     device="cuda")
    kb, vb = wl.bf16_bits(k), wl.bf16_bits(v)
    for layer in (0, 14, 27):
        out = torch.full((reqs, hq, lay.head_dim), float("nan"), device="cuda")
        lse = torch.full((reqs, hq), float("nan"), device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        km.kamera_decode_attention(h, km.Pool(k, v, w.page_table.cuda(), w.num_slots), layer,
                                   q.cuda(), torch.full((reqs,), ctx, dtype=torch.int32,
                                                        device="cuda"),
                                   ctx, lay.head_dim ** -0.5, out, lse, ws, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        compare(lay, kb, vb, kb, vb, w.page_table.numpy(), q, [ctx] * reqs,
                lay.head_dim ** -0.5, layer, out.cpu().numpy(), lse.cpu().numpy(),
                pool_diff=False)
    del k, v, w
    torch.cuda.empty_cache()


def test_form_patch_full():
    # patch forming at bench size (84 deficits of 1024 x 512, k = 40, m = 32, q = 1), in the
    # bench's single launch; three sampled problems against the oracle on the same inputs
    from tests.test_gpu_form import check_problem
    n, T, W, k, q, m = 84, 1024, 512, 40, 1, 32
    delta, omega = wl.deficit_problems(n, T, W, k=k, rank=64, decay=0.9, noise=1e-2, seed=0,
                                       device="cuda")
    u = torch.full((n, T, m), float("nan"), dtype=torch.bfloat16, device="cuda")
    vt = torch.full((n, m, W), float("nan"), dtype=torch.bfloat16, device="cuda")
    sig = torch.full((n, m), float("nan"), device="cuda")
    ws = torch.empty(km.kamera_form_patch_workspace(n, T, W, k), dtype=torch.uint8, device="cuda")
    km.kamera_form_patch(delta, omega, k, q, m, u, vt, sig, ws, num_problems=n, T=T, W=W, ld=W,
                         delta_stride=T * W, omega_stride=0, u_stride=T * m, vt_stride=m * W)
    torch.cuda.synchronize()
    assert not torch.isnan(u.float()).any() and not torch.isnan(vt.float()).any()
    om64 = omega.double().cpu().numpy()
    for i in (0, 41, 83):
        check_problem(delta[i].double().cpu().numpy(), om64, q, m,
                      u[i].float().double().cpu().numpy(), vt[i].float().double().cpu().numpy(),
                      sig[i].double().cpu().numpy(), need_columns=8)
    del delta, u, vt, ws
    torch.cuda.empty_cache()
