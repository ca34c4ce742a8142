"""Float64 CPU oracle of the Kamera reuse operator.

TEST INFRASTRUCTURE ONLY. This module is imported by ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``, and by nothing else. It
shares no code with the CUDA library: it imports only NumPy and the standard library, and it
takes plain arrays (bf16 values as ``uint16`` bit patterns) and plain numbers.

What it computes (Kamera: Unified Position-Invariant Multimodal KV Cache for Training-Free
Reuse, Eq. 1 in §1 and §3; App. A "Forming and applying the patch"):

    KV^(B|A) = R(δ) · KV(B|∅) + U_m · V_mᵀ

  * R(δ) re-rotates the RoPE phase of the stored keys by the integer offset δ = p1 - p0
    (§3 "Relocate"); RoPE composes, R(δ)R(p0) = R(p1), so this is exact algebra. Values and
    the MLA latent c_KV are never rotated (§3 "One mechanism for MLA, GQA, and MHA"; Fig. 2).
  * U_m V_mᵀ is the rank-m patch: the left factor carries the singular values (U·Σ, [T×m]) and
    the stored V_m is kept transposed as Vt [m×W] (App. A ``form_patch``); the patch is added
    after the rotation, in the target frame (App. A ``apply_reuse``: rotate, then add).
  * The result is written into a paged KV pool at the chunk's new slots (§6 "Recompute-free
    on a live engine": SGLang's paged KV pool).

Also: re-anchoring of keys stored before rotation to per-token request positions (QV-PIC,
"Model-Native Template-Conditioned Compilation", Eq. 2), per-section M-RoPE offsets (Kamera
Fig. 2), and patch forming from a given deficit (App. A ``form_patch``).

Readings taken where the pages are silent:
  * inv_freq_i = θ^(-2i/d), i < d/2, d = rotary dim (head_dim for GQA/MHA, the 64-dim k_pe band
    for MLA); the angle δ·inv_freq_i is formed in float64 and cos/sin taken in float64.
  * NeoX-half pairing pairs dim i with i + d/2 inside a rope band; interleaved pairs 2i, 2i+1.
  * GQA/MHA: every K head is rotated over its whole head_dim; one patch group per (layer,
    channel) spans all KV heads (W = H_kv·head_dim). MLA: row = c_KV ‖ k_pe (k_pe trailing),
    group 0 = c_KV (W = latent), group 1 = k_pe (W = rope_dim).
  * δ = 0 is R(0) = I exactly: no arithmetic, bit patterns kept (signed zeros included).
    Channels that neither rotate nor receive a patch are byte copies.
  * One rounding: the float64 result is rounded once, to nearest-even bf16.
  * slot(req, tok) = page_table[req][tok // page_size] * page_size + tok % page_size.
"""
from __future__ import annotations

import math
from types import SimpleNamespace

import numpy as np

GQA = 0
MLA = 1
NEOX_HALF = 0
INTERLEAVED = 1
MROPE_CONTIGUOUS = 0
MROPE_INTERLEAVED = 1


# ----------------------------------------------------------------------------------------
# bf16 encode / decode
# ----------------------------------------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    """Decode bf16 bit patterns (uint16) to float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    """Round float64 values once to the nearest bf16, ties to even; returns uint16 bits.

    bf16 keeps 8 significant bits and float32's exponent range, so the spacing at |x| is
    2^(e-7) with e = floor(log2|x|) clamped at -126 (subnormal spacing 2^-133). The value is
    rounded on that grid (NumPy rounds halves to even), overflow goes to infinity, and the
    (now exactly representable) value is encoded through float32.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    neg = np.signbit(x)
    finite = np.isfinite(x)
    safe = np.where(finite, ax, 0.0)
    _, E = np.frexp(safe)
    e = np.maximum(E - 1, -126)
    q = np.ldexp(1.0, e - 7)
    r = np.round(safe / q) * q
    big = r >= 2.0 ** 128
    with np.errstate(over="ignore"):
        r32 = np.where(big, np.float32(np.inf), r.astype(np.float32))
    bits = (r32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    bits = np.where(finite, bits, np.where(np.isnan(x), np.uint16(0x7FC0), np.uint16(0x7F80)))
    return (bits | (neg.astype(np.uint16) << np.uint16(15))).astype(np.uint16)


def factor_f64(a) -> np.ndarray:
    """A stored factor as float64: bf16 bit patterns (uint16) are decoded, floats are taken as
    they are (the pins feed float64 factors straight from an SVD)."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return bf16_to_f64(a)
    return a.astype(np.float64)


def bf16_ulp(y) -> np.ndarray:
    """Spacing of bf16 numbers at |y| (the unit in the last place of a bf16 value): 2^(e-7)
    for |y| in [2^e, 2^(e+1)), and the subnormal spacing 2^-133 below 2^-126 and at zero."""
    ay = np.abs(np.asarray(y, dtype=np.float64))
    _, E = np.frexp(ay)
    e = np.where(ay == 0, -126, np.maximum(E - 1, -126))
    return np.ldexp(1.0, e - 7)


# ----------------------------------------------------------------------------------------
# RoPE relocation R(δ)
# ----------------------------------------------------------------------------------------

def inv_freq(theta: float, d: int) -> np.ndarray:
    """inv_freq_i = θ^(-2i/d) for i < d/2, in float64."""
    i = np.arange(d // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / d)


def rope_pairs(d: int, style: int):
    """Index arrays (a, b) of the rotation pairs of a d-dim band; pair k uses frequency k."""
    k = np.arange(d // 2)
    if style == NEOX_HALF:
        return k, k + d // 2
    if style == INTERLEAVED:
        return 2 * k, 2 * k + 1
    raise ValueError("unknown rope style")


def rotate_band(x, delta, theta: float, style: int) -> np.ndarray:
    """Apply R(δ) to the last axis of ``x`` (a full rope band of even width d).

    Each pair (a, b) turns by φ_k = δ·inv_freq_k:  a' = a cos φ - b sin φ,  b' = b cos φ + a sin φ
    (§3 "Relocate": re-rotate B's keys by δ). ``delta`` is one integer for every pair, or one
    integer per pair (M-RoPE: each pair takes its section's offset). All zero returns the
    input unchanged.
    """
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    d = x.shape[-1]
    if np.ndim(delta) == 0:
        if delta == 0:
            return out
        phi = float(delta) * inv_freq(theta, d)
    else:
        offs = [int(v) for v in delta]
        if len(offs) != d // 2:
            raise ValueError("one offset per rope pair")
        if not any(offs):
            return out
        phi = np.array([float(v) for v in offs]) * inv_freq(theta, d)
    c, s = np.cos(phi), np.sin(phi)
    ia, ib = rope_pairs(d, style)
    a, b = x[..., ia], x[..., ib]
    out[..., ia] = a * c - b * s
    out[..., ib] = b * c + a * s
    return out


def mrope_pair_axes(npairs: int, sections, style: int) -> np.ndarray:
    """M-RoPE section of each rope pair: 0 = t, 1 = h, 2 = w (Kamera Fig. 2: the 64 rope pairs
    of a 128-d head split 16|24|24 or 24|20|20 over t, h, w).

    Contiguous: the first s_t pairs are t, the next s_h are h, the last s_w are w.
    Interleaved: h takes every third pair from pair 1 (s_h of them), w every third pair from
    pair 2 (s_w of them), and t takes the rest.
    """
    s_t, s_h, s_w = (int(v) for v in sections)
    if min(s_t, s_h, s_w) < 0 or s_t + s_h + s_w != npairs:
        raise ValueError("M-RoPE sections must sum to the rope pairs")
    if style == MROPE_CONTIGUOUS:
        return np.array([0] * s_t + [1] * s_h + [2] * s_w)
    if style == MROPE_INTERLEAVED:
        axes = np.zeros(npairs, dtype=int)
        h = list(range(1, npairs, 3))[:s_h]
        w = list(range(2, npairs, 3))[:s_w]
        if len(h) != s_h or len(w) != s_w:
            raise ValueError("interleaved M-RoPE sections do not fit the rope pairs")
        axes[h] = 1
        axes[w] = 2
        return axes
    raise ValueError("unknown M-RoPE style")


def has_mrope(layout) -> bool:
    return any(int(v) != 0 for v in getattr(layout, "mrope_section", (0, 0, 0)))


def pair_offsets(layout, item, npairs: int):
    """The relocation offset of each rope pair of a band: the item's δ for every pair under
    1-D RoPE; under M-RoPE, pair k takes (δ_t, δ_h, δ_w)[section of k], where δ_t = delta and
    δ_h, δ_w default to delta (all three coordinates advance together, Fig. 2 "relocate: +δ to
    the (t,h,w) position id")."""
    if not has_mrope(layout):
        return int(item.delta)
    dh = getattr(item, "delta_h", None)
    dw = getattr(item, "delta_w", None)
    offs = (int(item.delta), int(item.delta if dh is None else dh),
            int(item.delta if dw is None else dw))
    axes = mrope_pair_axes(npairs, layout.mrope_section, getattr(layout, "mrope_style", 0))
    return [offs[a] for a in axes]


def item_rotates(layout, item) -> bool:
    """Whether any rope pair of the item turns."""
    if not has_mrope(layout):
        return int(item.delta) != 0
    return any(v != 0 for v in pair_offsets(layout, item, int(sum(layout.mrope_section))))


# ----------------------------------------------------------------------------------------
# layout reading: content | rope split (§3, Fig. 2)
# ----------------------------------------------------------------------------------------

def widths(layout):
    """(row of channel 0, row of channel 1 or 0, group widths (W0, W1))."""
    if layout.kind == GQA:
        w = layout.num_kv_heads * layout.head_dim
        return w, w, (w, w)
    return layout.latent_dim + layout.rope_dim, 0, (layout.latent_dim, layout.rope_dim)


def rope_bands(layout):
    """(first column, width) of every rope band of the channel-0 row (K, or c_KV ‖ k_pe)."""
    if layout.kind == GQA:
        return [(h * layout.head_dim, layout.head_dim) for h in range(layout.num_kv_heads)]
    return [(layout.latent_dim, layout.rope_dim)]


def channel_groups(layout, channel: int):
    """Patch groups of a channel's row as (first column, width, group index)."""
    if layout.kind == GQA:
        w = layout.num_kv_heads * layout.head_dim
        return [(0, w, channel)]
    return [(0, layout.latent_dim, 0), (layout.latent_dim, layout.rope_dim, 1)]


def vt_of_group(layout, vt_layer, m: int, g: int) -> np.ndarray:
    """V_mᵀ of group g from one layer's packed factor ([m×W0] then [m×W1])."""
    _, _, (w0, w1) = widths(layout)
    flat = np.asarray(vt_layer)
    if g == 0:
        return flat[: m * w0].reshape(m, w0)
    return flat[m * w0: m * (w0 + w1)].reshape(m, w1)


# ----------------------------------------------------------------------------------------
# the operator
# ----------------------------------------------------------------------------------------

def layer_patched(item, layer: int) -> bool:
    return item.patch_m > 0 and item.patch_l0 <= layer < item.patch_l1


def reuse_layer(layout, item, layer: int, channel: int, tokens=None):
    """Exact result of one (item, layer, channel) before rounding.

    Returns (values float64 [t][row], copy_mask bool [row]) where ``copy_mask`` marks the
    columns that no arithmetic touches (bytes copied verbatim). ``tokens`` selects rows.
    """
    canon = item.canon_k if channel == 0 else item.canon_v
    rows = np.asarray(canon[layer])
    if tokens is not None:
        rows = rows[np.asarray(tokens)]
    x = bf16_to_f64(rows)
    copy_mask = np.ones(x.shape[-1], dtype=bool)
    if channel == 0 and item_rotates(layout, item):
        for c0, d in rope_bands(layout):
            x[:, c0:c0 + d] = rotate_band(x[:, c0:c0 + d], pair_offsets(layout, item, d // 2),
                                          layout.rope_theta, layout.rope_style)
            copy_mask[c0:c0 + d] = False
    if layer_patched(item, layer):
        m = item.patch_m
        li = layer - item.patch_l0
        for c0, w, g in channel_groups(layout, channel):
            u = factor_f64(item.patch_u[li][g])
            if tokens is not None:
                u = u[np.asarray(tokens)]
            vt = factor_f64(vt_of_group(layout, item.patch_vt[li], m, g))
            x[:, c0:c0 + w] = x[:, c0:c0 + w] + u @ vt
            copy_mask[c0:c0 + w] = False
    return x, copy_mask


def reuse_layer_bits(layout, item, layer: int, channel: int, tokens=None) -> np.ndarray:
    """bf16 bits the operator writes for one (item, layer, channel): one rounding, byte copy
    where nothing is computed."""
    vals, copy_mask = reuse_layer(layout, item, layer, channel, tokens)
    canon = item.canon_k if channel == 0 else item.canon_v
    src = np.asarray(canon[layer])
    if tokens is not None:
        src = src[np.asarray(tokens)]
    bits = f64_to_bf16(vals)
    bits[:, copy_mask] = src[:, copy_mask]
    return bits


def magnitude_layer(layout, item, layer: int, channel: int, tokens=None) -> np.ndarray:
    """Scale of the terms that make each result element: |a| + |b| on rotated pairs (an error
    in cos φ or sin φ multiplies both pair members), |x| elsewhere, plus Σ_j |U_tj · Vt_jc|.
    Float rounding errors of any evaluation order are bounded by a multiple of this."""
    canon = item.canon_k if channel == 0 else item.canon_v
    rows = np.asarray(canon[layer])
    if tokens is not None:
        rows = rows[np.asarray(tokens)]
    x = bf16_to_f64(rows)
    mag = np.abs(x)
    if channel == 0 and item_rotates(layout, item):
        for c0, d in rope_bands(layout):
            ia, ib = rope_pairs(d, layout.rope_style)
            ab = np.abs(x[:, c0 + ia]) + np.abs(x[:, c0 + ib])
            mag[:, c0 + ia] = ab
            mag[:, c0 + ib] = ab
    if layer_patched(item, layer):
        m = item.patch_m
        li = layer - item.patch_l0
        for c0, w, g in channel_groups(layout, channel):
            u = np.abs(factor_f64(item.patch_u[li][g]))
            if tokens is not None:
                u = u[np.asarray(tokens)]
            vt = np.abs(factor_f64(vt_of_group(layout, item.patch_vt[li], m, g)))
            mag[:, c0:c0 + w] += u @ vt
    return mag


def slot_of(page_table, req: int, tok: int, page_size: int) -> int:
    """Physical slot of logical token ``tok`` of request ``req``."""
    return int(page_table[req][tok // page_size]) * page_size + tok % page_size


def apply_reuse(layout, item, k_pool, v_pool, page_table) -> None:
    """Write one placed chunk into the pools (``uint16 [L][slots][row]``), every layer."""
    page = layout.page_size
    slots = [slot_of(page_table, item.req, item.start_tok + t, page)
             for t in range(item.num_tokens)]
    n_ch = 2 if layout.kind == GQA else 1
    for layer in range(layout.num_layers):
        for ch in range(n_ch):
            bits = reuse_layer_bits(layout, item, layer, ch)
            pool = k_pool if ch == 0 else v_pool
            for t, s in enumerate(slots):
                pool[layer, s, :] = bits[t]


def batch_reuse(layout, items, k_pool, v_pool, page_table) -> None:
    for it in items:
        apply_reuse(layout, it, k_pool, v_pool, page_table)


def relocate(layout, k_pool, page_table, req: int, start_tok: int, num_tokens: int,
             delta: int) -> None:
    """Survivor relocation in place: rotate the rope columns of K (GQA/MHA) or of the k_pe
    band (MLA) at the span's slots by δ; all other columns and V are left alone
    (§5 "Sliding-window survival": keep the survivor's KV as-is and apply R(δ); Fig. 2
    ``rotate_k_pe_inplace``)."""
    if delta == 0:
        return
    page = layout.page_size
    for layer in range(layout.num_layers):
        for t in range(num_tokens):
            s = slot_of(page_table, req, start_tok + t, page)
            row = bf16_to_f64(k_pool[layer, s, :])
            for c0, d in rope_bands(layout):
                rot = rotate_band(row[c0:c0 + d], delta, layout.rope_theta, layout.rope_style)
                k_pool[layer, s, c0:c0 + d] = f64_to_bf16(rot)


def patch_inplace(layout, k_pool, v_pool, page_table, req: int, start_tok: int,
                  num_tokens: int, patch_u, patch_vt, m: int, l0: int, l1: int,
                  sign: int = 1) -> None:
    """Conditioning switched back on in place: the rank-m patch added to the cached rows of a
    chunk (App. E "Context management as reversible state edits": re-applying conditioning
    is a single rank-m add; the clean view it starts from is the stored canonical). For each
    layer in [l0, l1) and each patch group, the rows of logical tokens
    [start_tok, start_tok + num_tokens) of request ``req`` become row + sign · U·Vt, computed
    in float64 and rounded once to bf16. ``sign = -1`` subtracts the same patch. Nothing
    rotates; columns outside the groups do not exist (the groups tile the row)."""
    if m <= 0 or l1 <= l0 or num_tokens <= 0:
        return
    page = layout.page_size
    slots = [slot_of(page_table, req, start_tok + t, page) for t in range(num_tokens)]
    n_ch = 2 if layout.kind == GQA else 1
    for layer in range(l0, l1):
        li = layer - l0
        for ch in range(n_ch):
            pool = k_pool if ch == 0 else v_pool
            rows = bf16_to_f64(np.stack([pool[layer, s, :] for s in slots]))
            for c0, w, g in channel_groups(layout, ch):
                u = factor_f64(patch_u[li][g])
                vt = factor_f64(vt_of_group(layout, patch_vt[li], m, g))
                rows[:, c0:c0 + w] = rows[:, c0:c0 + w] + sign * (u @ vt)
            bits = f64_to_bf16(rows)
            for t, s in enumerate(slots):
                pool[layer, s, :] = bits[t]


# ----------------------------------------------------------------------------------------
# re-anchoring keys stored before rotation (QV-PIC, Eq. 2)
# ----------------------------------------------------------------------------------------

def token_offsets(layout, position, npairs: int):
    """The rotation of every rope pair of one token at an absolute ``position``: one integer
    under 1-D RoPE; under M-RoPE ``position`` is (t, h, w) and pair k takes the coordinate of
    its section."""
    if not has_mrope(layout):
        return int(position)
    axes = mrope_pair_axes(npairs, layout.mrope_section, getattr(layout, "mrope_style", 0))
    coords = [int(v) for v in position]
    return [coords[a] for a in axes]


def reanchor_layer(layout, item, layer: int, channel: int, tokens=None):
    """Exact result of re-anchoring one (item, layer, channel) before rounding (QV-PIC,
    "Model-Native Template-Conditioned Compilation", Eq. 2: K = R(K̄, P(q)), keys stored before
    rotation turned to each token's request position; values position-independent).

    ``item.positions`` holds one position per token ([T], or [T][3] = (t, h, w) under M-RoPE).
    Token j's rope pairs turn from zero by its own position; values and the MLA latent are
    copied. Returns (values float64 [t][row], copy_mask bool [row]).
    """
    canon = item.canon_k if channel == 0 else item.canon_v
    rows = np.asarray(canon[layer])
    pos = np.asarray(item.positions, dtype=np.int64)
    if tokens is not None:
        rows = rows[np.asarray(tokens)]
        pos = pos[np.asarray(tokens)]
    x = bf16_to_f64(rows)
    copy_mask = np.ones(x.shape[-1], dtype=bool)
    if channel == 0:
        for c0, d in rope_bands(layout):
            for j in range(x.shape[0]):
                x[j, c0:c0 + d] = rotate_band(x[j, c0:c0 + d], token_offsets(layout, pos[j], d // 2),
                                              layout.rope_theta, layout.rope_style)
            copy_mask[c0:c0 + d] = False
    return x, copy_mask


def reanchor_layer_bits(layout, item, layer: int, channel: int, tokens=None) -> np.ndarray:
    """bf16 bits re-anchoring writes for one (item, layer, channel): one rounding of the rotated
    columns, byte copies elsewhere."""
    vals, copy_mask = reanchor_layer(layout, item, layer, channel, tokens)
    canon = item.canon_k if channel == 0 else item.canon_v
    src = np.asarray(canon[layer])
    if tokens is not None:
        src = src[np.asarray(tokens)]
    bits = f64_to_bf16(vals)
    bits[:, copy_mask] = src[:, copy_mask]
    return bits


def apply_reanchor(layout, item, k_pool, v_pool, page_table) -> None:
    """Write one re-anchored item into the pools at its slots (all layers, both channels)."""
    n_layers = len(item.canon_k)
    for layer in range(n_layers):
        for channel, pool in ((0, k_pool), (1, v_pool)):
            if channel == 1 and (layout.kind != GQA or pool is None):
                continue
            bits = reanchor_layer_bits(layout, item, layer, channel)
            for j in range(item.num_tokens):
                pool[layer][slot_of(page_table, item.req, item.start_tok + j,
                                    layout.page_size)] = bits[j]


# ----------------------------------------------------------------------------------------
# consumer check: decode attention over the pool (§1, the log-sum-exp readout merge)
# ----------------------------------------------------------------------------------------

def attend(k, v, q, scale: float):
    """Attention of one query over key rows ``k`` [T][Dk] and value rows ``v`` [T][Dv], float64:
    s = scale·k q, o = softmax(s)·v, lse = log Σ_t exp(s_t). No keys: o = 0, lse = -inf."""
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    if k.shape[0] == 0:
        return np.zeros(v.shape[-1]), -np.inf
    s = scale * (k @ np.asarray(q, np.float64))
    m = np.max(s)
    p = np.exp(s - m)
    return (p @ v) / np.sum(p), m + np.log(np.sum(p))


def lse_merge(parts):
    """Attention over the union of disjoint key sets from each set's (o, lse): weights
    exp(lse_s - lse) with lse = log Σ_s exp(lse_s) (§1: attention over KV(A) ‖ KV(B) equals
    attending each part and merging by softmax mass, o = (1 - μ) o_B + μ o_A)."""
    lses = np.array([l for _, l in parts], dtype=np.float64)
    if len(parts) == 0 or np.all(np.isneginf(lses)):
        dv = parts[0][0].shape[-1] if parts else 0
        return np.zeros(dv), -np.inf
    m = np.max(lses)
    w = np.exp(lses - m)
    o = sum(wi * np.asarray(oi, np.float64) for wi, (oi, _) in zip(w, parts)) / np.sum(w)
    return o, m + np.log(np.sum(w))


def head_columns(layout, h: int, num_q_heads: int):
    """Columns of query head h's key and value in the pool rows: ((k0, dk), (v0, dv), channel of
    V). GQA/MHA: head h // (H_q / H_kv) of the K and V rows. MLA (absorbed form): K is the whole
    c_KV ‖ k_pe row and V its c_KV part, both in channel 0."""
    if layout.kind == GQA:
        group = num_q_heads // layout.num_kv_heads
        c0 = (h // group) * layout.head_dim
        return (c0, layout.head_dim), (c0, layout.head_dim), 1
    return (0, layout.latent_dim + layout.rope_dim), (0, layout.latent_dim), 0


def decode_attention(layout, k_pool, v_pool, page_table, req: int, ctx_len: int, q,
                     scale: float, layer: int):
    """One query token per query head attending over logical tokens [0, ctx_len) of page-table
    row ``req`` in pool layer ``layer``. ``q`` [H_q][Dk] (values); pools hold bf16 bits.
    Returns (o [H_q][Dv], lse [H_q])."""
    q = np.asarray(q, np.float64)
    hq = q.shape[0]
    slots = [slot_of(page_table, req, t, layout.page_size) for t in range(ctx_len)]
    krows = bf16_to_f64(np.asarray(k_pool[layer])[slots]) if slots else None
    vrows = None
    if layout.kind == GQA and slots:
        vrows = bf16_to_f64(np.asarray(v_pool[layer])[slots])
    outs, lses = [], []
    for h in range(hq):
        (k0, dk), (v0, dv), vch = head_columns(layout, h, hq)
        if not slots:
            outs.append(np.zeros(dv))
            lses.append(-np.inf)
            continue
        src_v = vrows if vch == 1 else krows
        o, l = attend(krows[:, k0:k0 + dk], src_v[:, v0:v0 + dv], q[h], scale)
        outs.append(o)
        lses.append(l)
    return np.array(outs), np.array(lses)


# ----------------------------------------------------------------------------------------
# compile side, for the pins only (App. A ``form_patch``)
# ----------------------------------------------------------------------------------------

def form_patch(kv_cond, kv_solo_relocated, m: int):
    """The compile step of App. A from its two prefills: the deficit between the conditioned KV
    and the relocated context-free KV, replaced by its best rank-m approximation (Eckart–Young:
    the m leading singular triplets), with the singular values carried by the left factor.
    Returns (U·Σ [T×m], V_mᵀ [m×W]); see ``form_patch_svd`` for the sign convention."""
    deficit = np.asarray(kv_cond, np.float64) - np.asarray(kv_solo_relocated, np.float64)
    us, vt, _ = form_patch_svd(deficit, m)
    return us, vt


def _sign_rows(us, vt):
    """Fix the SVD sign freedom: the entry of largest magnitude in each row of Vt is made
    positive (the matching column of U·Σ flips with it)."""
    if vt.shape[0] == 0:
        return us, vt
    idx = np.argmax(np.abs(vt), axis=1)
    sgn = np.where(vt[np.arange(vt.shape[0]), idx] < 0, -1.0, 1.0)
    return us * sgn[None, :], vt * sgn[:, None]


def form_patch_svd(delta, m: int):
    """``form_patch`` on a given deficit Δ with the sign convention of ``_sign_rows``:
    (U·Σ [T×m], Vt [m×W], σ [m]) from the full SVD (numpy.linalg.svd, float64)."""
    u, s, vt = np.linalg.svd(np.asarray(delta, np.float64), full_matrices=False)
    us, vt = _sign_rows(u[:, :m] * s[:m], vt[:m])
    return us, vt, s[:m]


def form_patch_randomized(delta, omega, m: int, q: int):
    """Top-m patch of a deficit Δ [T×W] by the randomized range finder with q power
    iterations (Halko, Martinsson & Tropp, SIAM Review 2011, Alg. 4.4), then the SVD of the
    small projection B = QᵀΔ (their Alg. 5.1), in float64. ``omega`` [W×k] is the random
    test matrix (k ≥ m columns), drawn by the caller. Steps:
      Y = Δ Ω; Q = orth(Y); q times: Z = orth(ΔᵀQ), Q = orth(Δ Z);
      Bᵀ = ΔᵀQ; B Bᵀ = Ũ Λ Ũᵀ (eigenvalues descending); σ = √Λ;
      U·Σ = Q Ũ_m Σ_m, V_mᵀ = Σ_m⁻¹ Ũ_mᵀ B; signs as in ``_sign_rows``.
    Columns of σ = 0 give zero factors. Returns (U·Σ, Vt, σ)."""
    a = np.asarray(delta, np.float64)
    om = np.asarray(omega, np.float64)
    q_, _ = np.linalg.qr(a @ om)
    for _ in range(q):
        z, _ = np.linalg.qr(a.T @ q_)
        q_, _ = np.linalg.qr(a @ z)
    bt = a.T @ q_
    lam, ut = np.linalg.eigh(bt.T @ bt)
    order = np.argsort(lam)[::-1]
    lam, ut = lam[order], ut[:, order]
    sig = np.sqrt(np.maximum(lam[:m], 0.0))
    us = (q_ @ ut[:, :m]) * sig[None, :]
    with np.errstate(divide="ignore", invalid="ignore"):
        vt = np.where(sig[:, None] > 0, (bt @ ut[:, :m]).T / sig[:, None], 0.0)
    us, vt = _sign_rows(us, vt)
    return us, vt, sig


def patch_byte_fraction(T: int, W: int, m: int) -> float:
    """Bytes of a rank-m patch (U [T×m] and Vt [m×W]) over the bytes of the [T×W] page it
    patches, same element type on both sides: m·(T + W) / (T·W)."""
    return m * (T + W) / (T * W)


def as_item(**kw) -> SimpleNamespace:
    """Convenience record with the fields the oracle reads."""
    base = dict(canon_v=None, patch_u=None, patch_vt=None, patch_m=0, patch_l0=0, patch_l1=0,
                req=0, start_tok=0, delta_h=None, delta_w=None)
    base.update(kw)
    if "num_tokens" not in base:
        base["num_tokens"] = int(np.asarray(base["canon_k"]).shape[1])
    return SimpleNamespace(**base)


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("math", "np",
                                                                  "SimpleNamespace",
                                                                  "annotations")]
