"""kamera_form_patch_static_scratch: patch forming with the library's fixed device scratch (no
device allocation at the call), compared with kamera_form_patch and a caller workspace.

The file name puts it last in collection on purpose: the scratch is one array per device shared
by every call, and these tests must pass both alone in a fresh process and after all the
others. Tolerance: the factor tolerance of the patch-forming parity tests, per element
|got − ref| <= 2⁻⁸·|ref| + 1e-4·max|ref column| and σ within 1e-4·σ₁ (both entry points run
the same kernel, so in practice they agree bit for bit).
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import position_independent_multimodal_gb300 as km
import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _case(n, T, W, k, m, q, shared, seed):
    delta, omega = wl.deficit_problems(n, T, W, k=k, rank=min(64, T, W), decay=0.9,
                                       noise=1e-2, seed=seed, shared_omega=shared)
    dev = "cuda"
    return dict(n=n, T=T, W=W, k=k, m=m, q=q, shared=shared, delta=delta.to(dev),
                omega=omega.to(dev),
                out=lambda: (torch.full((n, T, m), float("nan"), dtype=torch.bfloat16,
                                        device=dev),
                             torch.full((n, m, W), float("nan"), dtype=torch.bfloat16,
                                        device=dev),
                             torch.full((n, m), float("nan"), dtype=torch.float32,
                                        device=dev)))


def _kw(c):
    n, T, W, k, m = c["n"], c["T"], c["W"], c["k"], c["m"]
    return dict(num_problems=n, T=T, W=W, ld=W, delta_stride=T * W,
                omega_stride=0 if c["shared"] else W * k, u_stride=T * m, vt_stride=m * W)


def _with_workspace(c):
    u, vt, sig = c["out"]()
    ws = torch.empty(km.kamera_form_patch_workspace(c["n"], c["T"], c["W"], c["k"]),
                     dtype=torch.uint8, device="cuda")
    km.kamera_form_patch(c["delta"], c["omega"], c["k"], c["q"], c["m"], u, vt, sig, ws,
                         **_kw(c))
    torch.cuda.synchronize()
    return u, vt, sig


def _static(c, outs):
    u, vt, sig = outs
    km.kamera_form_patch_static_scratch(c["delta"], c["omega"], c["k"], c["q"], c["m"], u, vt,
                                        sig, **_kw(c))


def _assert_close(ref, got):
    ur, vr, sr = (x.double().cpu().numpy() for x in ref)
    ug, vg, sg = (x.double().cpu().numpy() for x in got)
    assert np.all(np.isfinite(ug)) and np.all(np.isfinite(vg)) and np.all(np.isfinite(sg))
    assert np.all(np.abs(sg - sr) <= 1e-4 * sr[:, :1])
    # u [n][T][m]: columns are axis 1; vt [n][m][W]: rows are axis 2
    assert np.all(np.abs(ug - ur) <= 2.0 ** -8 * np.abs(ur) +
                  1e-4 * np.abs(ur).max(axis=1, keepdims=True))
    assert np.all(np.abs(vg - vr) <= 2.0 ** -8 * np.abs(vr) +
                  1e-4 * np.abs(vr).max(axis=2, keepdims=True))


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_on_two_calls_in_a_row(cuda_ok):
    # the 84 deficits of the reorder workload (30.1 MB of scratch), then a smaller problem set
    # with per-problem test matrices and two power iterations, issued back to back
    a = _case(84, 1024, 512, 40, 32, 1, True, seed=21)
    b = _case(5, 300, 256, 24, 16, 2, False, seed=22)
    ref_a, ref_b = _with_workspace(a), _with_workspace(b)
    out_a, out_b = a["out"](), b["out"]()
    _static(a, out_a)
    _static(b, out_b)
    torch.cuda.synchronize()
    _assert_close(ref_a, out_a)
    _assert_close(ref_b, out_b)
    # once set up, a call takes no device memory: free memory is unchanged around it
    out_c = b["out"]()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    _static(b, out_c)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    _assert_close(ref_b, out_c)


_FRESH = r"""
import sys
import torch
sys.path.insert(0, sys.argv[1])
import position_independent_multimodal_gb300 as km
import workloads as wl
torch.cuda.set_device(0)
n, T, W, k, m = 84, 1024, 512, 40, 32
delta, omega = wl.deficit_problems(n, T, W, k=k, rank=64, decay=0.9, noise=1e-2, seed=21,
                                   shared_omega=True)
delta, omega = delta.cuda(), omega.cuda()
u = torch.empty(n, T, m, dtype=torch.bfloat16, device="cuda")
vt = torch.empty(n, m, W, dtype=torch.bfloat16, device="cuda")
sig = torch.empty(n, m, dtype=torch.float32, device="cuda")
kw = dict(T=T, W=W, ld=W, delta_stride=T * W, omega_stride=0, u_stride=T * m, vt_stride=m * W)
def call(nprob):
    km.kamera_form_patch_static_scratch(delta, omega, k, 1, m, u, vt, sig, num_problems=nprob,
                                        **kw)
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
free1 = call(0)   # the set-up alone
free2 = call(n)
free3 = call(n)
print(free0 - free1, free1 - free2, free1 - free3)
"""


@pytest.mark.gpu
def test_static_scratch_takes_no_memory_after_its_set_up_in_a_fresh_process(cuda_ok):
    # The engine's order of events: a call with no problems (the set-up, made at start-up),
    # then the real calls, which must take no device memory. A fresh process, so that no earlier
    # test has done the set-up already. (The set-up itself reserves the array when CUDA loads
    # the library's device code lazily; with eager loading that happened with the context.)
    out = subprocess.run([sys.executable, "-c", _FRESH, ROOT], capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    setup, first, second = (int(v) for v in out.stdout.split()[-3:])
    assert setup in (0,) or setup >= km.KAMERA_FORM_PATCH_SCRATCH_BYTES - (2 << 20)
    assert first == 0 and second == 0


def test_static_scratch_checks_arguments_before_its_limit():
    # 200 deficits of 1024 x 512 at k = 40 need 71.7 MB of workspace, above the 32 MiB array:
    # with valid arguments that is UNSUPPORTED; a bad argument is reported first, as
    # kamera_form_patch reports it. Nothing is launched or set up, so no GPU is needed.
    n, T, W, k, m = 200, 1024, 512, 40, 32
    assert km.kamera_form_patch_workspace(n, T, W, k) > km.KAMERA_FORM_PATCH_SCRATCH_BYTES
    fake = 1 << 20  # aligned addresses that are never dereferenced

    def call(mm=m, u_stride=T * m):
        return km.lib().kamera_form_patch_static_scratch(
            fake, W, T * W, n, T, W, fake, 0, k, 1, mm, fake, u_stride, fake, mm * W, None, None)
    assert call() == km.KAMERA_ERR_UNSUPPORTED
    assert call(mm=k + 1) == km.KAMERA_ERR_INVALID_ARG       # m > k
    assert call(u_stride=1) == km.KAMERA_ERR_INVALID_ARG     # outputs of problems overlap
