"""Thin ctypes binding of libkamera.so: argument marshalling only.

Every function here has the name of the C entry point it calls (include/kamera.h) and does
nothing but convert PyTorch tensors and Python numbers into pointers and sizes. All work runs
in the CUDA kernels; if the library is missing or a call fails, an exception is raised: there
is no other code path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libkamera.so")

KAMERA_OK = 0
KAMERA_ERR_INVALID_ARG = 1
KAMERA_ERR_UNSUPPORTED = 2
KAMERA_ERR_CUDA = 3
KAMERA_DEVICE_SLOT_OOB = 0x1
KAMERA_DEVICE_BAD_ITEM = 0x2
KAMERA_GQA = 0
KAMERA_MLA = 1
KAMERA_ROPE_NEOX_HALF = 0
KAMERA_ROPE_INTERLEAVED = 1
KAMERA_MROPE_CONTIGUOUS = 0
KAMERA_MROPE_INTERLEAVED = 1
KAMERA_FORM_PATCH_SCRATCH_BYTES = 32 << 20
KAMERA_OPT_PATCH_ENGINE = 1
KAMERA_OPT_SHARE_RUN_PATCHED = 2
KAMERA_OPT_SHARE_RUN_UNPATCHED = 3
KAMERA_ENGINE_TENSOR = 0
KAMERA_ENGINE_CUDA_CORES = 1


class KameraError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({status_string(status)})")
        self.status = status


class kamera_layout(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("num_layers", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("latent_dim", ctypes.c_int32),
                ("rope_dim", ctypes.c_int32), ("rope_style", ctypes.c_int32),
                ("rope_theta", ctypes.c_double), ("mrope_section", ctypes.c_int32 * 3),
                ("mrope_style", ctypes.c_int32)]


class kamera_item(ctypes.Structure):
    _fields_ = [("canon_k", ctypes.c_void_p), ("canon_v", ctypes.c_void_p),
                ("patch_u", ctypes.c_void_p), ("patch_vt", ctypes.c_void_p),
                ("delta", ctypes.c_int64), ("num_tokens", ctypes.c_int32),
                ("req", ctypes.c_int32), ("start_tok", ctypes.c_int32),
                ("patch_m", ctypes.c_int32), ("patch_l0", ctypes.c_int32),
                ("patch_l1", ctypes.c_int32), ("delta_h", ctypes.c_int64),
                ("delta_w", ctypes.c_int64)]


class kamera_pool(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("num_slots", ctypes.c_int64),
                ("page_table", ctypes.c_void_p), ("num_reqs", ctypes.c_int32),
                ("pt_stride", ctypes.c_int32)]


class kamera_anchor_item(ctypes.Structure):
    _fields_ = [("canon_k", ctypes.c_void_p), ("canon_v", ctypes.c_void_p),
                ("positions", ctypes.c_void_p), ("num_tokens", ctypes.c_int32),
                ("req", ctypes.c_int32), ("start_tok", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


ITEM_BYTES = ctypes.sizeof(kamera_item)
_lib = None


def lib() -> ctypes.CDLL:
    """Load libkamera.so (built in-tree by ``build()``); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "position_independent_multimodal_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.kamera_create.argtypes = [ctypes.POINTER(kamera_layout), ctypes.POINTER(vp)]
        L.kamera_destroy.argtypes = [vp]
        L.kamera_status_string.argtypes = [ctypes.c_int]
        L.kamera_status_string.restype = ctypes.c_char_p
        L.kamera_set_option.argtypes = [vp, i32, i32]
        L.kamera_batch_workspace_bytes.argtypes = [vp, i32]
        L.kamera_batch_workspace_bytes.restype = ctypes.c_size_t
        L.kamera_set_batch_workspace.argtypes = [vp, vp, ctypes.c_size_t]
        L.kamera_relocate.argtypes = [vp, ctypes.POINTER(kamera_pool), i32, i32, i32, i64, vp, vp]
        L.kamera_reuse.argtypes = [vp, ctypes.POINTER(kamera_item), ctypes.POINTER(kamera_pool),
                                   vp, vp]
        L.kamera_batch_reuse.argtypes = [vp, vp, i32, i32, i32, ctypes.POINTER(kamera_pool), vp,
                                         vp]
        L.kamera_rope_phases.argtypes = [vp, vp, i32, vp, vp]
        L.kamera_batch_reuse_timed.argtypes = [vp, vp, i32, i32, i32,
                                               ctypes.POINTER(kamera_pool), vp, vp,
                                               ctypes.POINTER(vp)]
        L.kamera_patch_inplace.argtypes = [vp, ctypes.POINTER(kamera_pool), i32, i32, i32, vp,
                                           vp, i32, i32, i32, i32, vp, vp]
        L.kamera_batch_patch_inplace.argtypes = [vp, vp, i32, i32, i32,
                                                 ctypes.POINTER(kamera_pool), i32, vp, vp]
        L.kamera_reanchor.argtypes = [vp, vp, i32, i32, ctypes.POINTER(kamera_pool), vp, vp]
        L.kamera_decode_attention_workspace.argtypes = [vp, i32, i32, i32]
        L.kamera_decode_attention_workspace.restype = ctypes.c_size_t
        L.kamera_decode_attention.argtypes = [vp, ctypes.POINTER(kamera_pool), i32, vp, i32, i32,
                                              vp, i32, ctypes.c_float, vp, vp, vp,
                                              ctypes.c_size_t, vp, vp]
        L.kamera_form_patch_workspace.argtypes = [i32, i32, i32, i32]
        L.kamera_form_patch_workspace.restype = ctypes.c_size_t
        L.kamera_form_patch.argtypes = [vp, i64, i64, i32, i32, i32, vp, i64, i32, i32, i32, vp,
                                        i64, vp, i64, vp, vp, ctypes.c_size_t, vp]
        L.kamera_form_patch_static_scratch.argtypes = [vp, i64, i64, i32, i32, i32, vp, i64,
                                                       i32, i32, i32, vp, i64, vp, i64, vp, vp]
        for f in ("kamera_create", "kamera_destroy", "kamera_relocate", "kamera_reuse",
                  "kamera_set_option", "kamera_set_batch_workspace",
                  "kamera_batch_reuse", "kamera_rope_phases", "kamera_batch_reuse_timed",
                  "kamera_patch_inplace", "kamera_batch_patch_inplace", "kamera_form_patch",
                  "kamera_form_patch_static_scratch", "kamera_reanchor",
                  "kamera_decode_attention"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().kamera_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != KAMERA_OK:
        raise KameraError(status, what)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_layout(layout) -> kamera_layout:
    """Any object with the descriptor's fields -> the C struct (M-RoPE fields optional)."""
    sec = tuple(int(x) for x in getattr(layout, "mrope_section", (0, 0, 0)))
    return kamera_layout(int(layout.kind), int(layout.num_layers), int(layout.page_size),
                         int(layout.num_kv_heads), int(layout.head_dim), int(layout.latent_dim),
                         int(layout.rope_dim), int(layout.rope_style), float(layout.rope_theta),
                         (ctypes.c_int32 * 3)(*sec), int(getattr(layout, "mrope_style", 0)))


class Handle:
    """Owns a kamera_handle (created by kamera_create, freed by kamera_destroy)."""

    def __init__(self, layout):
        self.layout = layout
        self._c = make_layout(layout)
        h = ctypes.c_void_p()
        _check(lib().kamera_create(ctypes.byref(self._c), ctypes.byref(h)), "kamera_create")
        self.ptr = h

    def close(self):
        if self.ptr:
            lib().kamera_destroy(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def create(layout, **options) -> Handle:
    """kamera_create, then kamera_set_option for each keyword: patch_engine,
    share_run_patched, share_run_unpatched."""
    h = Handle(layout)
    for name, value in options.items():
        kamera_set_option(h, name, value)
    return h


_OPTIONS = {"patch_engine": KAMERA_OPT_PATCH_ENGINE,
            "share_run_patched": KAMERA_OPT_SHARE_RUN_PATCHED,
            "share_run_unpatched": KAMERA_OPT_SHARE_RUN_UNPATCHED}


def kamera_set_option(handle: Handle, option, value: int) -> None:
    """kamera_set_option; `option` is a KAMERA_OPT_* value or its keyword name."""
    opt = _OPTIONS[option] if isinstance(option, str) else int(option)
    _check(lib().kamera_set_option(handle.ptr, opt, int(value)), "kamera_set_option")


def kamera_batch_workspace_bytes(handle: Handle, num_items: int) -> int:
    """kamera_batch_workspace_bytes: workspace bytes for batches of up to num_items items."""
    return int(lib().kamera_batch_workspace_bytes(handle.ptr, int(num_items)))


def kamera_set_batch_workspace(handle: Handle, workspace: Optional[torch.Tensor]) -> None:
    """kamera_set_batch_workspace with a device tensor (its bytes), or None to remove it. The
    handle object keeps a reference to the tensor while the library holds its pointer."""
    if workspace is None:
        _check(lib().kamera_set_batch_workspace(handle.ptr, None, 0), "kamera_set_batch_workspace")
    else:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("the batch workspace must be a contiguous CUDA tensor")
        nbytes = workspace.numel() * workspace.element_size()
        _check(lib().kamera_set_batch_workspace(handle.ptr, workspace.data_ptr(), nbytes),
               "kamera_set_batch_workspace")
    handle.batch_workspace = workspace


class Pool:
    """The paged pool: k, v tensors [L][num_slots][row] and the int32 page table."""

    def __init__(self, k: torch.Tensor, v: Optional[torch.Tensor], page_table: torch.Tensor,
                 num_slots: Optional[int] = None):
        self.k, self.v, self.page_table = k, v, page_table
        self.num_slots = int(num_slots if num_slots is not None else k.shape[1])

    def c(self) -> kamera_pool:
        pt = self.page_table
        return kamera_pool(_ptr(self.k), _ptr(self.v), self.num_slots, _ptr(pt),
                           int(pt.shape[0]), int(pt.stride(0)))


def make_item(it) -> kamera_item:
    """An object with the kamera_item fields (tensors for the pointers) -> the C struct.
    ``delta_h`` / ``delta_w`` default to ``delta`` (all M-RoPE coordinates move together)."""
    dh = getattr(it, "delta_h", None)
    dw = getattr(it, "delta_w", None)
    return kamera_item(_ptr(it.canon_k), _ptr(getattr(it, "canon_v", None)),
                       _ptr(getattr(it, "patch_u", None)), _ptr(getattr(it, "patch_vt", None)),
                       int(it.delta), int(it.num_tokens), int(it.req), int(it.start_tok),
                       int(getattr(it, "patch_m", 0)), int(getattr(it, "patch_l0", 0)),
                       int(getattr(it, "patch_l1", 0)), int(it.delta if dh is None else dh),
                       int(it.delta if dw is None else dw))


def pack_items(items: Sequence) -> torch.Tensor:
    """Pack items into a host uint8 tensor of ``len(items) * sizeof(kamera_item)`` bytes."""
    arr = (kamera_item * len(items))(*[make_item(it) for it in items])
    return torch.frombuffer(bytearray(bytes(arr)), dtype=torch.uint8)


def kamera_relocate(handle: Handle, pool: Pool, req: int, start_tok: int, num_tokens: int,
                    delta: int, status: torch.Tensor, stream=None) -> None:
    p = pool.c()
    _check(lib().kamera_relocate(handle.ptr, ctypes.byref(p), int(req), int(start_tok),
                                 int(num_tokens), int(delta), _ptr(status), _stream(stream)),
           "kamera_relocate")


def kamera_reuse(handle: Handle, item, pool: Pool, status: torch.Tensor, stream=None) -> None:
    c = make_item(item)
    p = pool.c()
    _check(lib().kamera_reuse(handle.ptr, ctypes.byref(c), ctypes.byref(p), _ptr(status),
                              _stream(stream)), "kamera_reuse")


def kamera_batch_reuse(handle: Handle, d_items: torch.Tensor, num_items: int, max_tokens: int,
                       max_patch_m: int, pool: Pool, status: torch.Tensor, stream=None) -> None:
    p = pool.c()
    _check(lib().kamera_batch_reuse(handle.ptr, _ptr(d_items), int(num_items), int(max_tokens),
                                    int(max_patch_m), ctypes.byref(p), _ptr(status),
                                    _stream(stream)), "kamera_batch_reuse")


def kamera_patch_inplace(handle: Handle, pool: Pool, req: int, start_tok: int, num_tokens: int,
                         patch_u: torch.Tensor, patch_vt: torch.Tensor, patch_m: int,
                         patch_l0: int, patch_l1: int, sign: int, status: torch.Tensor,
                         stream=None) -> None:
    p = pool.c()
    _check(lib().kamera_patch_inplace(handle.ptr, ctypes.byref(p), int(req), int(start_tok),
                                      int(num_tokens), _ptr(patch_u), _ptr(patch_vt),
                                      int(patch_m), int(patch_l0), int(patch_l1), int(sign),
                                      _ptr(status), _stream(stream)), "kamera_patch_inplace")


def kamera_batch_patch_inplace(handle: Handle, d_items: torch.Tensor, num_items: int,
                               max_tokens: int, max_patch_m: int, pool: Pool, sign: int,
                               status: torch.Tensor, stream=None) -> None:
    p = pool.c()
    _check(lib().kamera_batch_patch_inplace(handle.ptr, _ptr(d_items), int(num_items),
                                            int(max_tokens), int(max_patch_m), ctypes.byref(p),
                                            int(sign), _ptr(status), _stream(stream)),
           "kamera_batch_patch_inplace")


def pack_anchor_items(items: Sequence) -> torch.Tensor:
    """Objects with canon_k, canon_v, positions (tensors), num_tokens, req, start_tok -> a host
    uint8 tensor of packed kamera_anchor_item structs."""
    arr = (kamera_anchor_item * len(items))(*[
        kamera_anchor_item(_ptr(it.canon_k), _ptr(getattr(it, "canon_v", None)),
                           _ptr(it.positions), int(it.num_tokens), int(it.req),
                           int(it.start_tok), 0) for it in items])
    return torch.frombuffer(bytearray(bytes(arr)), dtype=torch.uint8)


def kamera_reanchor(handle: Handle, d_items: torch.Tensor, num_items: int, max_tokens: int,
                    pool: Pool, status: torch.Tensor, stream=None) -> None:
    p = pool.c()
    _check(lib().kamera_reanchor(handle.ptr, _ptr(d_items), int(num_items), int(max_tokens),
                                 ctypes.byref(p), _ptr(status), _stream(stream)),
           "kamera_reanchor")


def kamera_decode_attention_workspace(handle: Handle, num_reqs: int, num_q_heads: int,
                                      max_ctx: int) -> int:
    return int(lib().kamera_decode_attention_workspace(handle.ptr, int(num_reqs),
                                                       int(num_q_heads), int(max_ctx)))


def kamera_decode_attention(handle: Handle, pool: Pool, layer: int, q: torch.Tensor,
                            ctx_len: torch.Tensor, max_ctx: int, scale: float,
                            out: torch.Tensor, lse: torch.Tensor,
                            workspace: Optional[torch.Tensor], status: torch.Tensor,
                            stream=None) -> None:
    """Decode attention of ``q`` [R][H_q][Dk] over pool layer ``layer`` (requests = page-table
    rows 0..R-1, contexts ``ctx_len`` int32 [R]) into ``out`` float32 [R][H_q][Dv] and ``lse``
    float32 [R][H_q]."""
    p = pool.c()
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().kamera_decode_attention(handle.ptr, ctypes.byref(p), int(layer), _ptr(q),
                                         int(q.shape[0]), int(q.shape[1]), _ptr(ctx_len),
                                         int(max_ctx), float(scale), _ptr(out), _ptr(lse),
                                         _ptr(workspace), int(nbytes), _ptr(status),
                                         _stream(stream)), "kamera_decode_attention")


def kamera_rope_phases(handle: Handle, d_deltas: torch.Tensor, d_out: torch.Tensor,
                       stream=None) -> None:
    """(cos, sin) per (delta, pair) into ``d_out`` float32 [n][rope_dim/2][2]."""
    _check(lib().kamera_rope_phases(handle.ptr, _ptr(d_deltas), int(d_deltas.numel()),
                                    _ptr(d_out), _stream(stream)), "kamera_rope_phases")


def kamera_batch_reuse_timed(handle: Handle, d_items: torch.Tensor, num_items: int,
                             max_tokens: int, max_patch_m: int, pool: Pool, status: torch.Tensor,
                             events, stream=None) -> None:
    """kamera_batch_reuse recording torch.cuda.Event objects (or None): before its first kernel,
    between the unpatched and the patched layers, after the planning kernel of the persistent
    path, and after its last kernel (a list of three leaves out the third)."""
    ev = list(events)
    if len(ev) == 3:
        ev = [ev[0], ev[1], None, ev[2]]
    if len(ev) != 4:
        raise ValueError("kamera_batch_reuse_timed takes three or four events")
    for e in ev:
        if e is not None and not e.cuda_event:
            e.record()  # torch creates an event's CUDA event at its first record
    arr = (ctypes.c_void_p * 4)(*[None if e is None else e.cuda_event for e in ev])
    p = pool.c()
    _check(lib().kamera_batch_reuse_timed(handle.ptr, _ptr(d_items), int(num_items),
                                          int(max_tokens), int(max_patch_m), ctypes.byref(p),
                                          _ptr(status), _stream(stream), arr),
           "kamera_batch_reuse_timed")


def kamera_form_patch_workspace(num_problems: int, T: int, W: int, k: int) -> int:
    """Bytes of device workspace ``kamera_form_patch`` needs."""
    return int(lib().kamera_form_patch_workspace(int(num_problems), int(T), int(W), int(k)))


def kamera_form_patch(delta: torch.Tensor, omega: torch.Tensor, k: int, q: int, m: int,
                      u: torch.Tensor, vt: torch.Tensor, sigma: Optional[torch.Tensor],
                      workspace: Optional[torch.Tensor], *, num_problems: int, T: int, W: int,
                      ld: int, delta_stride: int, omega_stride: int, u_stride: int,
                      vt_stride: int, stream=None) -> None:
    """Top-m factors of ``num_problems`` float32 deficits into bf16 ``u`` / ``vt`` (strides in
    elements, as in the C call); ``workspace`` is a device buffer of at least
    ``kamera_form_patch_workspace`` bytes."""
    _check(lib().kamera_form_patch(_ptr(delta), int(ld), int(delta_stride), int(num_problems),
                                   int(T), int(W), _ptr(omega), int(omega_stride), int(k),
                                   int(q), int(m), _ptr(u), int(u_stride), _ptr(vt),
                                   int(vt_stride), _ptr(sigma), _ptr(workspace),
                                   0 if workspace is None else
                                   int(workspace.numel() * workspace.element_size()),
                                   _stream(stream)), "kamera_form_patch")


def kamera_form_patch_static_scratch(delta: torch.Tensor, omega: torch.Tensor, k: int, q: int,
                                     m: int, u: torch.Tensor, vt: torch.Tensor,
                                     sigma: Optional[torch.Tensor], *, num_problems: int, T: int,
                                     W: int, ld: int, delta_stride: int, omega_stride: int,
                                     u_stride: int, vt_stride: int, stream=None) -> None:
    """``kamera_form_patch`` with the library's fixed device scratch instead of a caller
    workspace (no device allocation at the call; at most ``KAMERA_FORM_PATCH_SCRATCH_BYTES``
    of workspace; calls on one device must not overlap in time)."""
    _check(lib().kamera_form_patch_static_scratch(
        _ptr(delta), int(ld), int(delta_stride), int(num_problems), int(T), int(W),
        _ptr(omega), int(omega_stride), int(k), int(q), int(m), _ptr(u), int(u_stride),
        _ptr(vt), int(vt_stride), _ptr(sigma), _stream(stream)),
        "kamera_form_patch_static_scratch")
