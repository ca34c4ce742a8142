"""Kamera relocate + patch operator for NVIDIA GB300 (sm_103a).

``KV^(B|A) = R(δ)·KV(B|∅) + U_m·V_mᵀ`` written into a paged KV pool, as hand-written CUDA
kernels behind a C ABI (include/kamera.h). This package is the Python binding: it marshals
PyTorch tensors into the C calls and nothing more. Build the library with ``build.build()``.
"""
from ._binding import (  # noqa: F401
    ITEM_BYTES, KAMERA_DEVICE_BAD_ITEM, KAMERA_DEVICE_SLOT_OOB, KAMERA_ERR_CUDA,
    KAMERA_FORM_PATCH_SCRATCH_BYTES,
    KAMERA_ERR_INVALID_ARG, KAMERA_ERR_UNSUPPORTED, KAMERA_GQA, KAMERA_MLA,
    KAMERA_ENGINE_CUDA_CORES, KAMERA_ENGINE_TENSOR, KAMERA_OPT_PATCH_ENGINE,
    KAMERA_OPT_SHARE_RUN_PATCHED, KAMERA_OPT_SHARE_RUN_UNPATCHED, kamera_set_option,
    KAMERA_MROPE_CONTIGUOUS, KAMERA_MROPE_INTERLEAVED, KAMERA_OK,
    KAMERA_ROPE_INTERLEAVED, KAMERA_ROPE_NEOX_HALF, LIB_PATH, Handle, KameraError, Pool,
    create, kamera_batch_patch_inplace, kamera_batch_reuse, kamera_batch_reuse_timed,
    kamera_batch_workspace_bytes, kamera_set_batch_workspace,
    kamera_form_patch, kamera_form_patch_static_scratch, kamera_form_patch_workspace,
    kamera_decode_attention, kamera_decode_attention_workspace, kamera_patch_inplace,
    kamera_reanchor, pack_anchor_items, kamera_relocate,
    kamera_reuse, kamera_rope_phases, lib, make_item, make_layout,
    pack_items, status_string,
)
