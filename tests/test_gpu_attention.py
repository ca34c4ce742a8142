"""Consumer check: kamera_decode_attention over the paged pool against float64 attention.

Two comparisons:
  * kernel parity, same pool: the GPU's attention and the oracle's attention read the same
    pool bits. With B = max_t (Dk + 1)·2⁻²⁴·scale·Σ_d |q_d k_td| (float32 dot accumulation),
    every output element is within (8B + 1e-4)·max|V| and the lse within 4B + 1e-5·(1 + |lse|):
    a score error B moves each softmax weight by about 2B relatively, and the remaining
    float32 sums (one split's ≤ 256 terms, then the split merge) stay below 1e-4.
  * GQA with head_dim 128 runs on the tensor cores, which take the softmax weights as bf16:
    the normaliser sums the same rounded weights, so each weight of the convex combination is
    off by at most 2·2⁻⁹ relatively, adding 2⁻⁸·max|V| to the output and 2⁻⁸ to the lse bound.
  * consumer check: the GPU attends over the pool the GPU reuse call wrote, the oracle over
    the pool the oracle's reuse wrote. The two pools differ by at most about one and a half
    bf16 ulps per element (≤ 2⁻⁷ relative), which adds 2·B_pool·max|V| + 2⁻⁷·max|V| to the
    output bound (B_pool = 2⁻⁷·scale·max_t Σ_d |q_d k_td|) and 2·B_pool to the lse bound.
"""
import math

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


def gpu_attention(lay, k, v, pt, num_slots, q, ctx, max_ctx, scale, layer):
    h = km.create(lay)
    R, hq = q.shape[0], q.shape[1]
    dv = lay.head_dim if lay.kind == wl.GQA else lay.latent_dim
    out = torch.full((R, hq, dv), float("nan"), device="cuda")
    lse = torch.full((R, hq), float("nan"), device="cuda")
    ws_bytes = km.kamera_decode_attention_workspace(h, R, hq, max_ctx)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    km.kamera_decode_attention(h, km.Pool(k, v, pt.cuda(), num_slots), layer, q.cuda(),
                               torch.as_tensor(ctx, dtype=torch.int32, device="cuda"), max_ctx,
                               scale, out, lse, ws, st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy(), int(st.item())


def score_bound(lay, kbits, pt, req, ctx, qv, scale, layer, hq, rel):
    """max over tokens of rel·scale·Σ_d |q_d k_td| for each query head."""
    if ctx == 0:
        return np.zeros(hq)
    slots = [ora.slot_of(pt, req, t, lay.page_size) for t in range(ctx)]
    rows = np.abs(ora.bf16_to_f64(kbits[layer][slots]))
    out = []
    for h in range(hq):
        (k0, dk), _, _ = ora.head_columns(lay, h, hq)
        out.append(rel(dk) * scale * np.max(rows[:, k0:k0 + dk] @ np.abs(qv[h])))
    return np.array(out)


def vmax(lay, kbits, vbits, pt, req, ctx, layer, hq):
    if ctx == 0:
        return np.zeros(hq)
    slots = [ora.slot_of(pt, req, t, lay.page_size) for t in range(ctx)]
    out = []
    for h in range(hq):
        _, (v0, dv), vch = ora.head_columns(lay, h, hq)
        src = vbits if vch == 1 else kbits
        out.append(np.max(np.abs(ora.bf16_to_f64(src[layer][slots][:, v0:v0 + dv]))))
    return np.array(out)


def compare(lay, kb_gpu, vb_gpu, kb_ref, vb_ref, pt, q, ctx, scale, layer, o_g, l_g, pool_diff,
            reqs=None):
    qv = ora.bf16_to_f64(wl.bf16_bits(q))
    hq = q.shape[1]
    for r, c in enumerate(ctx):
        if reqs is not None and r not in reqs:
            continue
        o_r, l_r = ora.decode_attention(lay, kb_ref, vb_ref, pt, r, c, qv[r], scale, layer)
        if c == 0:
            assert np.all(o_g[r] == 0) and np.all(np.isneginf(l_g[r]))
            continue
        B = score_bound(lay, kb_gpu, pt, r, c, qv[r], scale, layer, hq,
                        lambda dk: (dk + 1) * 2.0 ** -24)
        Vm = vmax(lay, kb_gpu, vb_gpu, pt, r, c, layer, hq)
        tol_o = (8 * B + 1e-4) * Vm
        tol_l = 4 * B + 1e-5 * (1 + np.abs(l_r))
        if tensor_path(lay):
            tol_o = tol_o + 2.0 ** -8 * Vm
            tol_l = tol_l + 2.0 ** -8
        if pool_diff:
            Bp = score_bound(lay, kb_gpu, pt, r, c, qv[r], scale, layer, hq, lambda dk: 2.0 ** -7)
            tol_o = tol_o + (2 * Bp + 2.0 ** -7) * Vm
            tol_l = tol_l + 2 * Bp
        err_o = np.max(np.abs(o_g[r] - o_r), axis=1)
        assert np.all(err_o <= tol_o), (r, c, err_o, tol_o)
        assert np.all(np.abs(l_g[r] - l_r) <= tol_l), (r, c, l_g[r], l_r)


def tensor_path(lay):
    return lay.kind == wl.GQA and lay.head_dim == 128


def random_pool(lay, R, pages_per_req, seed):
    g = torch.Generator().manual_seed(seed)
    n = R * pages_per_req * lay.page_size
    k = wl.normal_bf16((lay.num_layers, n, lay.row_k), 1.0, g, "cpu")
    v = wl.normal_bf16((lay.num_layers, n, lay.row_v), 1.0, g, "cpu") if lay.kind == wl.GQA \
        else None
    pt = wl.shuffled_page_table(R, pages_per_req, g)
    return k, v, pt, n


CASES = {
    "gqa-64-group3": (wl.Layout(kind=wl.GQA, num_layers=2, page_size=16, num_kv_heads=2,
                                head_dim=64, rope_dim=64, rope_theta=1e4), 6),
    "gqa-128-group7": (wl.Layout(kind=wl.GQA, num_layers=2, page_size=16, num_kv_heads=4,
                                 head_dim=128, rope_dim=128, rope_theta=1e6), 28),
    "mla-16-heads": (wl.Layout(kind=wl.MLA, num_layers=2, page_size=16, latent_dim=512,
                               rope_dim=64, rope_theta=1e4), 16),
    "mla-20-heads": (wl.Layout(kind=wl.MLA, num_layers=2, page_size=16, latent_dim=512,
                               rope_dim=64, rope_theta=1e4), 20),
}


@pytest.mark.parametrize("sharp", [1.0, 8.0])
@pytest.mark.parametrize("case", sorted(CASES))
def test_decode_attention_matches_oracle_on_the_same_pool(case, sharp):
    # contexts: empty, one token, one split less one, one split plus one, several splits
    lay, hq = CASES[case]
    ctx = [0, 1, 255, 257, 700]
    k, v, pt, n = random_pool(lay, len(ctx), 45, seed=hq)
    dk = lay.head_dim if lay.kind == wl.GQA else lay.latent_dim + lay.rope_dim
    g = torch.Generator().manual_seed(7)
    q = wl.normal_bf16((len(ctx), hq, dk), sharp, g, "cpu")
    scale = 1.0 / math.sqrt(dk)
    layer = 1
    o_g, l_g, st = gpu_attention(lay, k.cuda(), None if v is None else v.cuda(), pt, n, q, ctx,
                                 max(ctx), scale, layer)
    assert st == 0
    kb = wl.bf16_bits(k)
    vb = wl.bf16_bits(v) if v is not None else None
    compare(lay, kb, vb, kb, vb, pt.numpy(), q, ctx, scale, layer, o_g, l_g, pool_diff=False)


def back_to_back(lay, m, name):
    # two requests whose contexts are filled by chunks placed back to back from token 0
    T = [37, 130, 300, 64]
    placements = [(0, 0, 0, 0), (1, 0, 37, 37), (2, 0, 167, 167),
                  (2, 1, 0, 0), (3, 1, 300, 300), (0, 1, 364, 364)]
    return wl.reuse_workload(name, lay, n_chunks=4, T=T, placements=placements, m=m, l0=0,
                             l1=lay.num_layers, seed=3, strong=True, patch_per_item=True), \
        [467, 401]


@pytest.mark.parametrize("case", ["gqa-128-group7", "mla-16-heads"])
def test_consumer_check_over_the_pool_written_by_reuse(case):
    # relocated + patched rows written by kamera_batch_reuse, read back by the attention
    # kernel, against the oracle's attention over the oracle's own pool
    lay, hq = CASES[case]
    w, ctx = back_to_back(lay, 32, f"cons{case}")
    h = km.create(lay)
    k, v, status, _ = tl.run_batch(h, lay, tl.to_device_items(w.items), w.page_table,
                                   w.num_slots)
    assert status == 0
    kb_ref = np.full((lay.num_layers, w.num_slots, lay.row_k), wl.POOL_SENTINEL_BITS,
                     dtype=np.uint16)
    vb_ref = np.full((lay.num_layers, w.num_slots, lay.row_v), wl.POOL_SENTINEL_BITS,
                     dtype=np.uint16) if lay.kind == wl.GQA else None
    ora.batch_reuse(lay, [tl.oracle_item(it) for it in w.items], kb_ref, vb_ref,
                    w.page_table.numpy())
    dk = lay.head_dim if lay.kind == wl.GQA else lay.latent_dim + lay.rope_dim
    q = wl.normal_bf16((len(ctx), hq, dk), 1.0, torch.Generator().manual_seed(9), "cpu")
    scale = 1.0 / math.sqrt(dk)
    for layer in range(lay.num_layers):
        o_g, l_g, st = gpu_attention(lay, k, v, w.page_table, w.num_slots, q, ctx, max(ctx),
                                     scale, layer)
        assert st == 0
        compare(lay, wl.bf16_bits(k), wl.bf16_bits(v) if v is not None else None, kb_ref,
                vb_ref, w.page_table.numpy(), q, ctx, scale, layer, o_g, l_g, pool_diff=True)


def test_context_longer_than_max_is_rejected_on_the_device():
    lay, hq = CASES["gqa-64-group3"]
    ctx = [300, 20]
    k, v, pt, n = random_pool(lay, 2, 20, seed=1)
    q = wl.normal_bf16((2, hq, 64), 1.0, torch.Generator().manual_seed(2), "cpu")
    o_g, l_g, st = gpu_attention(lay, k.cuda(), v.cuda(), pt, n, q, ctx, 256, 0.125, 0)
    assert st == km.KAMERA_DEVICE_BAD_ITEM
    assert np.all(np.isnan(o_g[0])) and np.all(np.isnan(l_g[0]))   # request 0 not written
    kb, vb = wl.bf16_bits(k), wl.bf16_bits(v)
    compare(lay, kb, vb, kb, vb, pt.numpy(), q, ctx, 0.125, 0, o_g, l_g, pool_diff=False,
            reqs=[1])
