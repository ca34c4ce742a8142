"""GPU parity of kamera_form_patch (patch forming from a given deficit) against the float64
oracle ``form_patch_randomized`` on the same Δ and Ω.

Tolerances, derived from the arithmetic (the kernel runs float32, the oracle float64, and the
outputs are bf16):
  * σ: |σ_gpu − σ| <= 1e-4·σ_1. The float32 path evaluates every product with at most
    max(T, W) accumulations per element (relative error well below 1e-4 at these sizes);
    the orthonormalisations and Jacobi add a few ulps of float32.
  * the patch U·Σ·V_mᵀ formed from the bf16 outputs: relative Frobenius error <= 5e-3 against
    the oracle's float64 product. Each factor is rounded once to bf16 (2⁻⁹ relative per
    element), so the product carries about 2·2⁻⁹ ≈ 3.9e-3 at worst.
  * single factors are unique (up to the sign the convention fixes) only for a singular value
    separated from its neighbours; for those with σ_j >= 0.01·σ_1 and both gaps >= 0.02·σ_1,
    every element obeys |gpu − ref| <= 2⁻⁸·|ref| + 1e-4·max|ref column| (one bf16 ulp plus
    the float32 path's error amplified by at most σ_1/gap = 50).
"""
import numpy as np
import pytest
import torch

import position_independent_multimodal_gb300 as km
import workloads as wl
from oracle import kamera_oracle as ora

pytestmark = pytest.mark.gpu

SIG_TOL = 1e-4
PROD_TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda(cuda_ok):
    return cuda_ok


def bf16_to_f64(t):
    return t.float().double().cpu().numpy()


def form(delta, omega, k, q, m, *, u=None, vt=None, u_off=0, vt_off=0, u_stride=None,
         vt_stride=None, shared=True):
    """Run kamera_form_patch on n = delta.shape[0] problems; returns (u, vt, sigma) tensors.
    When u / vt are given, results go to them at the offsets and strides (elements)."""
    n, T, W = delta.shape
    dev = "cuda"
    d = delta.to(dev).contiguous()
    o = omega.to(dev).contiguous()
    u_stride = T * m if u_stride is None else u_stride
    vt_stride = m * W if vt_stride is None else vt_stride
    if u is None:
        u = torch.full((n * T * m,), float("nan"), dtype=torch.bfloat16, device=dev)
    if vt is None:
        vt = torch.full((n * m * W,), float("nan"), dtype=torch.bfloat16, device=dev)
    sig = torch.full((n, m), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(km.kamera_form_patch_workspace(n, T, W, k), dtype=torch.uint8, device=dev)
    km.kamera_form_patch(d, o, k, q, m, u.view(-1)[u_off:], vt.view(-1)[vt_off:], sig, ws,
                         num_problems=n, T=T, W=W, ld=W, delta_stride=T * W,
                         omega_stride=0 if shared else W * k, u_stride=u_stride,
                         vt_stride=vt_stride)
    torch.cuda.synchronize()
    return u, vt, sig


def well_separated(s, j):
    s1 = s[0]
    lo = s[j] - s[j + 1] if j + 1 < len(s) else np.inf
    hi = s[j - 1] - s[j] if j > 0 else np.inf
    return s[j] >= 0.01 * s1 and min(lo, hi) >= 0.02 * s1


def check_problem(d64, om64, q, m, us_g, vt_g, sig_g, *, need_columns=1):
    k = om64.shape[1]
    # all k values of the sketch's spectrum decide which of the first m columns are unique;
    # the oracle's first m factors do not depend on how many it is asked for
    us_k, vt_k, s_k = ora.form_patch_randomized(d64, om64, k, q)
    us, vt, s = us_k[:, :m], vt_k[:m], s_k[:m]
    assert np.all(np.abs(sig_g - s) <= SIG_TOL * s[0] + 1e-12), (sig_g[:4], s[:4])
    p_ref = us @ vt
    p_gpu = us_g @ vt_g
    den = np.linalg.norm(p_ref)
    if den == 0:
        assert np.all(p_gpu == 0)
        return
    assert np.linalg.norm(p_gpu - p_ref) <= PROD_TOL * den
    checked = 0
    for j in range(m):
        if not well_separated(s_k, j):
            continue
        checked += 1
        for got, ref in ((vt_g[j], vt[j]), (us_g[:, j], us[:, j])):
            tol = 2.0 ** -8 * np.abs(ref) + 1e-4 * np.max(np.abs(ref))
            bad = np.abs(got - ref) > tol
            assert not bad.any(), (j, np.flatnonzero(bad)[:5], got[bad][:3], ref[bad][:3])
    assert checked >= need_columns


def unpack(u, vt, sig, n, T, W, m, u_off=0, vt_off=0, u_stride=None, vt_stride=None):
    u_stride = T * m if u_stride is None else u_stride
    vt_stride = m * W if vt_stride is None else vt_stride
    uf = u.view(-1)
    vf = vt.view(-1)
    out = []
    for i in range(n):
        us = bf16_to_f64(uf[u_off + i * u_stride: u_off + i * u_stride + T * m]).reshape(T, m)
        v = bf16_to_f64(vf[vt_off + i * vt_stride: vt_off + i * vt_stride + m * W]).reshape(m, W)
        out.append((us, v, sig[i].double().cpu().numpy()))
    return out


def test_form_patch_gqa_into_store_layout():
    """Two patched GQA layers (K and V groups, W = 2 heads x 128) formed straight into the
    kamera_item patch layout: patch_u [layers][2][T][m], patch_vt [layers][m*(W0+W1)].
    T = 300 spans four 64-row GEMM blocks and a ragged tail."""
    L, T, W, m, k, q = 2, 300, 256, 16, 24, 1
    delta, omega = wl.deficit_problems(2 * L, T, W, k=k, rank=32, decay=0.85, noise=1e-3,
                                       seed=1)
    dev = "cuda"
    pu = torch.full((L, 2, T, m), float("nan"), dtype=torch.bfloat16, device=dev)
    pv = torch.full((L, m * 2 * W), float("nan"), dtype=torch.bfloat16, device=dev)
    sigs = []
    for g in range(2):  # problems of group g: layers 0..L-1, deficit index 2*l + g
        dg = delta[g::2].contiguous()
        _, _, sig = form(dg, omega, k, q, m, u=pu, vt=pv, u_off=g * T * m, vt_off=g * m * W,
                         u_stride=2 * T * m, vt_stride=2 * m * W)
        sigs.append(sig)
    assert not torch.isnan(pu.float()).any() and not torch.isnan(pv.float()).any()
    om64 = omega.double().numpy()
    for g in range(2):
        res = unpack(pu, pv, sigs[g], L, T, W, m, u_off=g * T * m, vt_off=g * m * W,
                     u_stride=2 * T * m, vt_stride=2 * m * W)
        for l, (us, v, s) in enumerate(res):
            check_problem(delta[2 * l + g].double().numpy(), om64, q, m, us, v, s,
                          need_columns=4)


def test_form_patch_mla_two_group_widths_per_problem_omega():
    """MLA groups of different widths (c_KV 512, k_pe 64) in one patch store, each problem
    with its own Ω; two power iterations."""
    L, T, m, k, q = 3, 200, 8, 24, 2
    W0, W1 = 512, 64
    dev = "cuda"
    pu = torch.full((L, 2, T, m), float("nan"), dtype=torch.bfloat16, device=dev)
    pv = torch.full((L, m * (W0 + W1)), float("nan"), dtype=torch.bfloat16, device=dev)
    for g, W in enumerate((W0, W1)):
        delta, omega = wl.deficit_problems(L, T, W, k=k, rank=20, decay=0.8, noise=1e-3,
                                           seed=10 + g, shared_omega=False)
        _, _, sig = form(delta, omega, k, q, m, u=pu, vt=pv, u_off=g * T * m,
                         vt_off=g * m * W0, u_stride=2 * T * m, vt_stride=m * (W0 + W1),
                         shared=False)
        res = unpack(pu, pv, sig, L, T, W, m, u_off=g * T * m, vt_off=g * m * W0,
                     u_stride=2 * T * m, vt_stride=m * (W0 + W1))
        for i, (us, v, s) in enumerate(res):
            check_problem(delta[i].double().numpy(), omega[i].double().numpy(), q, m, us, v, s,
                          need_columns=3)
    assert not torch.isnan(pu.float()).any() and not torch.isnan(pv.float()).any()


def test_form_patch_exact_low_rank_and_zero_deficit():
    """A deficit of exact rank 5 < m: the first five factors match, σ past the rank is at
    the float32 noise level; an all-zero deficit gives all-zero factors and σ."""
    T, W, m, k, q = 160, 96, 8, 12, 0
    delta, omega = wl.deficit_problems(2, T, W, k=k, rank=5, decay=0.6, noise=0.0, seed=3)
    delta[1].zero_()
    u, vt, sig = form(delta, omega, k, q, m)
    res = unpack(u, vt, sig, 2, T, W, m)
    us, v, s = res[0]
    s_ref = np.linalg.svd(delta[0].double().numpy(), compute_uv=False)
    assert np.all(s[5:] <= 1e-5 * s_ref[0])
    check_problem(delta[0].double().numpy(), omega.double().numpy(), q, m, us, v, s,
                  need_columns=3)
    us0, v0, s0 = res[1]
    assert np.all(us0 == 0) and np.all(v0 == 0) and np.all(s0 == 0)


@pytest.mark.parametrize("T,W,k,m,q", [(40, 700, 13, 13, 1), (700, 40, 17, 9, 3),
                                       (64, 64, 64, 32, 1)])
def test_form_patch_edge_shapes(T, W, k, m, q):
    """Odd k (a dummy index in the Jacobi rounds), m = k, k = T = W, W > T and T > W."""
    delta, omega = wl.deficit_problems(3, T, W, k=k, rank=min(T, W, 48), decay=0.8,
                                       noise=1e-3, seed=T + W + k)
    u, vt, sig = form(delta, omega, k, q, m)
    for i, (us, v, s) in enumerate(unpack(u, vt, sig, 3, T, W, m)):
        check_problem(delta[i].double().numpy(), omega.double().numpy(), q, m, us, v, s)


def test_form_patch_is_deterministic():
    delta, omega = wl.deficit_problems(4, 256, 128, k=20, rank=24, decay=0.85, noise=1e-3,
                                       seed=7)
    a = form(delta, omega, 20, 1, 12)
    b = form(delta, omega, 20, 1, 12)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y)
