"""The C ABI on the host (no GPU needed): the library builds, loads, exports every function
include/kamera.h declares, its structs have the documented sizes, and the host-side checks
reject bad arguments before anything is launched."""
import ctypes
import os
import re

import pytest
import torch

import position_independent_multimodal_gb300 as km
from position_independent_multimodal_gb300 import _binding as kb
from position_independent_multimodal_gb300 import build as kbuild
import workloads as wl

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return km.lib()


def declared_functions():
    names = []
    for f in os.listdir(HEADER):
        if f.endswith(".h"):
            src = open(os.path.join(HEADER, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(
                r"^\s*(?:kamera_status|const char\s*\*|size_t)\s*(kamera_\w+)\s*\(", src,
                flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "kamera_batch_reuse" in names and "kamera_relocate" in names
    assert "kamera_reuse" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_struct_sizes():
    assert ctypes.sizeof(kb.kamera_item) == 80
    assert ctypes.sizeof(kb.kamera_layout) == 56
    assert ctypes.sizeof(kb.kamera_pool) == 40
    assert ctypes.sizeof(kb.kamera_anchor_item) == 40


def gqa(**kw):
    base = dict(kind=wl.GQA, num_layers=2, page_size=16, num_kv_heads=2, head_dim=64,
                rope_dim=64, rope_style=wl.NEOX_HALF, rope_theta=1e4)
    base.update(kw)
    return wl.Layout(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(num_layers=0), km.KAMERA_ERR_INVALID_ARG),
    (dict(page_size=0), km.KAMERA_ERR_INVALID_ARG),
    (dict(rope_theta=1.0), km.KAMERA_ERR_INVALID_ARG),
    (dict(rope_theta=float("nan")), km.KAMERA_ERR_INVALID_ARG),
    (dict(rope_style=7), km.KAMERA_ERR_INVALID_ARG),
    (dict(kind=5), km.KAMERA_ERR_INVALID_ARG),
    (dict(rope_dim=32), km.KAMERA_ERR_UNSUPPORTED),       # partial rotary
    (dict(head_dim=72, rope_dim=72), km.KAMERA_ERR_UNSUPPORTED),
    (dict(head_dim=512, rope_dim=512), km.KAMERA_ERR_UNSUPPORTED),
    (dict(num_kv_heads=200, head_dim=128, rope_dim=128), km.KAMERA_ERR_UNSUPPORTED),
    # M-RoPE sections must cover the 32 pairs exactly, be non-negative and fit their style
    (dict(mrope_section=(8, 12, 11)), km.KAMERA_ERR_INVALID_ARG),
    (dict(mrope_section=(40, -4, -4)), km.KAMERA_ERR_INVALID_ARG),
    (dict(mrope_section=(8, 12, 12), mrope_style=2), km.KAMERA_ERR_INVALID_ARG),
    (dict(mrope_section=(0, 12, 20), mrope_style=wl.MROPE_INTERLEAVED),
     km.KAMERA_ERR_INVALID_ARG),
])
def test_create_rejects_bad_layouts(lib, kw, status):
    with pytest.raises(km.KameraError) as e:
        km.create(gqa(**kw))
    assert e.value.status == status


def test_create_accepts_reference_layouts(lib):
    km.create(wl.config1().layout)
    km.create(gqa(head_dim=128, rope_dim=128, mrope_section=(16, 24, 24)))
    km.create(gqa(head_dim=128, rope_dim=128, mrope_section=(24, 20, 20),
                  mrope_style=wl.MROPE_INTERLEAVED))
    km.create(wl.Layout(kind=wl.MLA, num_layers=27, page_size=16, latent_dim=512, rope_dim=64,
                        rope_style=wl.NEOX_HALF, rope_theta=1e4))
    km.create(wl.Layout(kind=wl.MLA, num_layers=2, page_size=16, latent_dim=512, rope_dim=72,
                        rope_theta=1e4)) if False else None


class FakeTensor:
    """Stands in for a device tensor: only its address is read on the host."""

    def __init__(self, addr, shape=(1,), stride0=1):
        self.addr, self.shape, self._s = addr, shape, stride0

    def data_ptr(self):
        return self.addr

    def stride(self, i):
        return self._s


def fake_pool(k=0x10000, v=0x20000, slots=256, reqs=2, stride=16, pt=0x30000):
    return km.Pool(FakeTensor(k) if k is not None else None,
                   FakeTensor(v) if v is not None else None,
                   FakeTensor(pt, (reqs, stride), stride), slots)


def fake_item(**kw):
    base = dict(canon_k=FakeTensor(0x40000), canon_v=FakeTensor(0x50000), patch_u=None,
                patch_vt=None, delta=5, num_tokens=16, req=0, start_tok=0)
    base.update(kw)
    return wl.Item(**base)


STATUS = FakeTensor(0x60000)


@pytest.mark.parametrize("pool_kw,item_kw", [
    (dict(k=None), {}),
    (dict(k=0x10008), {}),                               # misaligned pool
    (dict(v=None), {}),                                  # GQA needs V
    (dict(slots=250), {}),                               # not a multiple of the page size
    (dict(pt=0x30002), {}),
    ({}, dict(req=2)),
    ({}, dict(req=-1)),
    ({}, dict(start_tok=250)),                           # runs past the page table
    ({}, dict(canon_v=None)),
    ({}, dict(canon_k=FakeTensor(0x40004))),
    ({}, dict(num_tokens=-1)),
    ({}, dict(patch_m=8, patch_l0=0, patch_l1=3)),       # layer range past L
    ({}, dict(patch_m=8, patch_l0=1, patch_l1=0)),
    ({}, dict(patch_m=8, patch_l0=0, patch_l1=1)),       # missing factors
    ({}, dict(delta=(1 << 62) + 1)),
])
def test_reuse_rejects_bad_arguments_on_host(lib, pool_kw, item_kw):
    h = km.create(gqa())
    with pytest.raises(km.KameraError) as e:
        km.kamera_reuse(h, fake_item(**item_kw), fake_pool(**pool_kw), STATUS, stream=0)
    assert e.value.status == km.KAMERA_ERR_INVALID_ARG


def test_reuse_rank_above_limit_is_unsupported(lib):
    h = km.create(gqa())
    it = fake_item(patch_m=129, patch_l0=0, patch_l1=1, patch_u=FakeTensor(0x70000),
                   patch_vt=FakeTensor(0x80000))
    with pytest.raises(km.KameraError) as e:
        km.kamera_reuse(h, it, fake_pool(), STATUS, stream=0)
    assert e.value.status == km.KAMERA_ERR_UNSUPPORTED


def test_mla_rejects_a_value_pool(lib):
    h = km.create(wl.Layout(kind=wl.MLA, num_layers=2, page_size=16, latent_dim=512,
                            rope_dim=64, rope_theta=1e4))
    with pytest.raises(km.KameraError):
        km.kamera_relocate(h, fake_pool(), 0, 0, 4, 3, STATUS, stream=0)


def test_batch_and_relocate_host_checks(lib):
    h = km.create(gqa())
    d = FakeTensor(0x90000)
    for args in [(-1, 16, 0), (1, -1, 0), (1, 16, -1)]:
        with pytest.raises(km.KameraError):
            km.kamera_batch_reuse(h, d, *args, fake_pool(), STATUS, stream=0)
    with pytest.raises(km.KameraError) as e:
        km.kamera_batch_reuse(h, d, 1, 16, 129, fake_pool(), STATUS, stream=0)
    assert e.value.status == km.KAMERA_ERR_UNSUPPORTED
    with pytest.raises(km.KameraError):
        km.kamera_batch_reuse(h, FakeTensor(0x90004), 1, 16, 0, fake_pool(), STATUS, stream=0)
    with pytest.raises(km.KameraError):
        km.kamera_batch_reuse(h, d, 1, 16, 0, fake_pool(), FakeTensor(0), stream=0)
    for args in [(2, 0, 4, 3), (0, 250, 16, 3), (0, 0, -1, 3), (0, 0, 4, -(1 << 62) - 1)]:
        with pytest.raises(km.KameraError):
            km.kamera_relocate(h, fake_pool(), *args, STATUS, stream=0)
    # nothing to do: returns OK without touching the device
    km.kamera_batch_reuse(h, d, 0, 16, 0, fake_pool(), STATUS, stream=0)
    km.kamera_relocate(h, fake_pool(), 0, 0, 0, 3, STATUS, stream=0)
    km.kamera_relocate(h, fake_pool(), 0, 0, 8, 0, STATUS, stream=0)


def test_patch_inplace_host_checks(lib):
    h = km.create(gqa())
    u, vt = FakeTensor(0x70000), FakeTensor(0x80000)
    bad = [
        dict(req=2), dict(start_tok=-1), dict(num_tokens=-1), dict(start_tok=250),
        dict(sign=0), dict(sign=2), dict(l0=1, l1=0), dict(l1=3), dict(u=None),
        dict(vt=FakeTensor(0x80008)), dict(u=FakeTensor(0x70001)),
    ]
    for kw in bad:
        a = dict(req=0, start_tok=0, num_tokens=16, u=u, vt=vt, m=8, l0=0, l1=1, sign=1)
        a.update(kw)
        with pytest.raises(km.KameraError) as e:
            km.kamera_patch_inplace(h, fake_pool(), a["req"], a["start_tok"], a["num_tokens"],
                                    a["u"], a["vt"], a["m"], a["l0"], a["l1"], a["sign"],
                                    STATUS, stream=0)
        assert e.value.status == km.KAMERA_ERR_INVALID_ARG, kw
    with pytest.raises(km.KameraError) as e:
        km.kamera_patch_inplace(h, fake_pool(), 0, 0, 16, u, vt, 129, 0, 1, 1, STATUS, stream=0)
    assert e.value.status == km.KAMERA_ERR_UNSUPPORTED
    # nothing to do: returns OK without touching the device
    for m, l0, l1, T in [(0, 0, 1, 16), (8, 1, 1, 16), (8, 0, 1, 0)]:
        km.kamera_patch_inplace(h, fake_pool(), 0, 0, T, u, vt, m, l0, l1, -1, STATUS, stream=0)
    # tiles that are not 64 or 128 columns wide are not served
    wide = km.create(wl.Layout(kind=wl.GQA, num_layers=2, page_size=16, num_kv_heads=2,
                               head_dim=256, rope_dim=256, rope_theta=1e4))
    with pytest.raises(km.KameraError) as e:
        km.kamera_patch_inplace(wide, fake_pool(), 0, 0, 16, u, vt, 8, 0, 1, 1, STATUS,
                                stream=0)
    assert e.value.status == km.KAMERA_ERR_UNSUPPORTED


def test_batch_patch_inplace_host_checks(lib):
    h = km.create(gqa())
    d = FakeTensor(0x90000)
    for args in [(-1, 16, 8, 1), (1, -1, 8, 1), (1, 16, -1, 1), (1, 16, 8, 0)]:
        with pytest.raises(km.KameraError):
            km.kamera_batch_patch_inplace(h, d, args[0], args[1], args[2], fake_pool(), args[3],
                                          STATUS, stream=0)
    with pytest.raises(km.KameraError) as e:
        km.kamera_batch_patch_inplace(h, d, 1, 16, 129, fake_pool(), 1, STATUS, stream=0)
    assert e.value.status == km.KAMERA_ERR_UNSUPPORTED
    with pytest.raises(km.KameraError):
        km.kamera_batch_patch_inplace(h, FakeTensor(0x90004), 1, 16, 8, fake_pool(), 1, STATUS,
                                      stream=0)
    km.kamera_batch_patch_inplace(h, d, 0, 16, 8, fake_pool(), 1, STATUS, stream=0)
    km.kamera_batch_patch_inplace(h, d, 3, 16, 0, fake_pool(), -1, STATUS, stream=0)


class FakeWorkspace(FakeTensor):
    def __init__(self, addr, nbytes):
        super().__init__(addr)
        self.nbytes = nbytes

    def numel(self):
        return self.nbytes

    def element_size(self):
        return 1


def test_form_patch_host_checks(lib):
    n, T, W, k, q, m = 3, 100, 64, 16, 1, 8
    need = km.kamera_form_patch_workspace(n, T, W, k)

    def documented(n, T, W, k):  # floats per problem, rounded up to a multiple of 4
        nt = -(-max(T, W) // 128)
        per = (T + W) * k + nt * (k * k + 3 * k) + 9 * k * k + k + 4
        return n * (-(-per // 4) * 4) * 4
    assert need == documented(n, T, W, k) == 63024
    assert km.kamera_form_patch_workspace(n, 40, 300, k) == documented(n, 40, 300, k) == 104112
    assert km.kamera_form_patch_workspace(1, 1024, 512, 40) == 358576
    assert km.kamera_form_patch_workspace(-1, T, W, k) == 0
    d, o = FakeTensor(0x100000), FakeTensor(0x200000)
    u, vt, sig = FakeTensor(0x300000), FakeTensor(0x400000), FakeTensor(0x500000)
    ws = FakeWorkspace(0x600000, need)
    base = dict(k=k, q=q, m=m, num_problems=n, T=T, W=W, ld=W, delta_stride=T * W,
                omega_stride=0, u_stride=T * m, vt_stride=m * W, d=d, o=o, u=u, vt=vt, sig=sig,
                ws=ws)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        km.kamera_form_patch(a["d"], a["o"], a["k"], a["q"], a["m"], a["u"], a["vt"], a["sig"],
                             a["ws"], num_problems=a["num_problems"], T=a["T"], W=a["W"],
                             ld=a["ld"], delta_stride=a["delta_stride"],
                             omega_stride=a["omega_stride"], u_stride=a["u_stride"],
                             vt_stride=a["vt_stride"], stream=0)

    invalid = [dict(num_problems=-1), dict(T=0), dict(W=0), dict(k=0), dict(m=0), dict(m=17),
               dict(q=-1), dict(ld=W - 1), dict(delta_stride=-1), dict(omega_stride=-1),
               dict(u_stride=T * m - 1), dict(vt_stride=m * W - 1), dict(d=None), dict(o=None),
               dict(u=None), dict(vt=None), dict(ws=None), dict(d=FakeTensor(0x100002)),
               dict(o=FakeTensor(0x200001)), dict(u=FakeTensor(0x300001)),
               dict(vt=FakeTensor(0x400001)), dict(sig=FakeTensor(0x500002)),
               dict(ws=FakeWorkspace(0x600000, need - 1)),
               dict(ws=FakeWorkspace(0x600002, need))]
    for kw in invalid:
        with pytest.raises(km.KameraError) as e:
            call(**kw)
        assert e.value.status == km.KAMERA_ERR_INVALID_ARG, kw
    # k above 96, above T or W, or too many power iterations (W itself is not bounded)
    unsupported = [dict(k=97, m=8, T=200, W=200), dict(k=64, T=63), dict(k=65, W=64),
                   dict(q=17)]
    for kw in unsupported:
        with pytest.raises(km.KameraError) as e:
            call(**kw)
        assert e.value.status == km.KAMERA_ERR_UNSUPPORTED, kw
    # nothing to do: returns OK without touching the device
    call(num_problems=0)


def test_reanchor_host_checks(lib):
    h = km.create(gqa())
    d = FakeTensor(0x90000)
    for args in [(-1, 16), (1, -1)]:
        with pytest.raises(km.KameraError) as e:
            km.kamera_reanchor(h, d, args[0], args[1], fake_pool(), STATUS, stream=0)
        assert e.value.status == km.KAMERA_ERR_INVALID_ARG
    with pytest.raises(km.KameraError) as e:
        km.kamera_reanchor(h, FakeTensor(0x90004), 1, 16, fake_pool(), STATUS, stream=0)
    assert e.value.status == km.KAMERA_ERR_INVALID_ARG
    with pytest.raises(km.KameraError) as e:
        km.kamera_reanchor(h, d, 70000, 16, fake_pool(), STATUS, stream=0)
    assert e.value.status == km.KAMERA_ERR_UNSUPPORTED
    # nothing to do: returns OK without touching the device
    km.kamera_reanchor(h, d, 0, 16, fake_pool(), STATUS, stream=0)
    km.kamera_reanchor(h, d, 3, 0, fake_pool(), STATUS, stream=0)


def test_decode_attention_host_checks(lib):
    h = km.create(gqa())  # H_kv = 2, head_dim = 64
    q = FakeTensor(0xA0000, shape=(3, 4, 64))
    ctx = FakeTensor(0xB0000)
    out, lse, ws = FakeTensor(0xC0000), FakeTensor(0xD0000), FakeWorkspace(0xE0000, 1 << 20)
    need = km.kamera_decode_attention_workspace(h, 3, 4, 600)
    assert need == 3 * 4 * 3 * (64 + 1) * 4  # splits of 256 tokens: ceil(600 / 256) = 3
    assert km.kamera_decode_attention_workspace(h, 3, 4, 0) == 0

    def call(**kw):
        a = dict(layer=0, q=q, ctx=ctx, max_ctx=600, scale=0.125, out=out, lse=lse, ws=ws)
        a.update(kw)
        km.kamera_decode_attention(h, fake_pool(reqs=4), a["layer"], a["q"], a["ctx"], a["max_ctx"],
                                   a["scale"], a["out"], a["lse"], a["ws"], STATUS, stream=0)

    invalid = [dict(layer=-1), dict(layer=2), dict(max_ctx=-1), dict(scale=float("nan")),
               dict(q=FakeTensor(0xA0000, shape=(3, 3, 64))),      # 3 heads over 2 KV heads
               dict(q=FakeTensor(0xA0001, shape=(3, 4, 64))), dict(ctx=FakeTensor(0xB0002)),
               dict(out=FakeTensor(0xC0002)), dict(lse=FakeTensor(0xD0001)),
               dict(ws=FakeWorkspace(0xE0000, need - 4)), dict(ws=None),
               dict(q=FakeTensor(0xA0000, shape=(9, 4, 64)))]     # more requests than rows
    for kw in invalid:
        with pytest.raises(km.KameraError) as e:
            call(**kw)
        assert e.value.status == km.KAMERA_ERR_INVALID_ARG, kw
    with pytest.raises(km.KameraError) as e:
        call(q=FakeTensor(0xA0000, shape=(3, 258, 64)))
    assert e.value.status == km.KAMERA_ERR_UNSUPPORTED
    call(q=FakeTensor(0xA0000, shape=(0, 4, 64)))  # no requests: nothing launched


def test_status_strings(lib):
    for s in range(4):
        assert km.status_string(s)


def test_library_is_required(monkeypatch, tmp_path):
    monkeypatch.setattr(kb, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(kb, "_lib", None)
    with pytest.raises(ImportError):
        kb.lib()


def test_set_option_checks_its_arguments():
    h = km.create(gqa())
    km.kamera_set_option(h, "patch_engine", km.KAMERA_ENGINE_CUDA_CORES)
    km.kamera_set_option(h, km.KAMERA_OPT_PATCH_ENGINE, km.KAMERA_ENGINE_TENSOR)
    km.kamera_set_option(h, "share_run_patched", 32)
    km.kamera_set_option(h, "share_run_unpatched", 1)
    for opt, val in ((km.KAMERA_OPT_PATCH_ENGINE, 2), (km.KAMERA_OPT_SHARE_RUN_PATCHED, 0),
                     (km.KAMERA_OPT_SHARE_RUN_PATCHED, 33), (km.KAMERA_OPT_SHARE_RUN_UNPATCHED, 9),
                     (99, 1)):
        with pytest.raises(km.KameraError) as e:
            km.kamera_set_option(h, opt, val)
        assert e.value.status == km.KAMERA_ERR_INVALID_ARG
    assert km.lib().kamera_set_option(None, km.KAMERA_OPT_PATCH_ENGINE, 0) == \
        km.KAMERA_ERR_INVALID_ARG


class _WsFake:
    """A device buffer's address and size; kamera_set_batch_workspace only stores them."""
    is_cuda = True

    def __init__(self, addr, nbytes):
        self.addr, self.nbytes = addr, nbytes

    def is_contiguous(self):
        return True

    def data_ptr(self):
        return self.addr

    def numel(self):
        return self.nbytes

    def element_size(self):
        return 1


def test_batch_workspace_size_and_setter(lib):
    lay = gqa()
    h = km.create(lay)
    sizes = [km.kamera_batch_workspace_bytes(h, n) for n in (0, 1, 18, 1000)]
    assert all(s % 256 == 0 for s in sizes) and sizes == sorted(sizes)
    per_task = 16
    c = km.make_layout(lay)
    assert sizes[3] >= 1000 * c.num_layers * 2 * per_task  # task rows: items x layers x channels
    assert lib.kamera_batch_workspace_bytes(None, 5) == 0
    assert km.kamera_batch_workspace_bytes(h, -1) == 0
    need = km.kamera_batch_workspace_bytes(h, 1)
    for bad in (_WsFake(0x100010, need), _WsFake(0x100000, need - 256)):
        with pytest.raises(km.KameraError) as e:
            km.kamera_set_batch_workspace(h, bad)
        assert e.value.status == km.KAMERA_ERR_INVALID_ARG
    assert lib.kamera_set_batch_workspace(h.ptr, None, 64) == km.KAMERA_ERR_INVALID_ARG
    assert lib.kamera_set_batch_workspace(None, None, 0) == km.KAMERA_ERR_INVALID_ARG
    km.kamera_set_batch_workspace(h, _WsFake(0x100000, need))
    km.kamera_set_batch_workspace(h, None)
    # host memory or a strided view is refused before the library sees a pointer
    for bad in (torch.zeros(need, dtype=torch.uint8), torch.zeros(2 * need, dtype=torch.uint8)[::2]):
        with pytest.raises(ValueError):
            km.kamera_set_batch_workspace(h, bad)


def test_timed_batch_takes_three_or_four_events(lib):
    h = km.create(gqa())
    for events in ([None] * 2, [None] * 5):
        with pytest.raises(ValueError):
            km.kamera_batch_reuse_timed(h, None, 0, 0, 0, None, None, events)
