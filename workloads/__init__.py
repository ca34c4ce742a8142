"""Seeded synthetic inputs for the Kamera relocate + patch operator.

This module is shared by the tests, the benchmark and the smoke run. It holds shapes, value
distributions and random draws only: no rotation, no patch product, no slot arithmetic and no
rounding of results. Both the float64 oracle and the CUDA library consume what it returns.

Shapes follow the workloads the Kamera paper measures ("Kamera: Unified Position-Invariant
Multimodal KV Cache for Training-Free Reuse"): 1024-token video segments (§1), 576-token
images, K=3 reorders (§5, Reorder), sliding-window survivors (§5, Sliding-window survival)
and recalls at large offsets (§5, Recall). No dataset is read: every value is drawn here.

Conventions of the generated data:
  * bf16 tensors hold the round-to-nearest-even bf16 of float32 normal draws (torch does the
    conversion);
  * a canonical chunk is stored as ``[L][T][row]``; GQA/MHA keeps K and V separately
    (row = H_kv * head_dim), MLA keeps one tensor with row = latent ‖ rope band;
  * a patch is stored per item as ``patch_u [l1-l0][2][T][m]`` (U·Σ) and
    ``patch_vt [l1-l0][m*(W0+W1)]`` where group 0 (K or c_KV, width W0) is followed by
    group 1 (V or k_pe, width W1), each ``[m][W_g]`` row-major (= V_mᵀ);
  * pools are ``[L][num_slots][row]``; a page is ``page_size`` consecutive slots; the page
    table is ``int32 [num_reqs][pt_stride]`` holding physical page ids.
"""
from __future__ import annotations

import dataclasses
import itertools
import zlib
from typing import Optional

import numpy as np
import torch

GQA = 0
MLA = 1
NEOX_HALF = 0
INTERLEAVED = 1
MROPE_CONTIGUOUS = 0
MROPE_INTERLEAVED = 1

# sentinel bf16 bit pattern that untouched pool slots keep; chosen finite and unlikely
POOL_SENTINEL_BITS = 0x5A5A


@dataclasses.dataclass(frozen=True)
class Layout:
    kind: int
    num_layers: int
    page_size: int
    num_kv_heads: int = 0
    head_dim: int = 0
    latent_dim: int = 0
    rope_dim: int = 0
    rope_style: int = NEOX_HALF
    rope_theta: float = 10000.0
    mrope_section: tuple = (0, 0, 0)      # M-RoPE pairs of t, h, w; (0, 0, 0) = 1-D RoPE
    mrope_style: int = 0                  # MROPE_CONTIGUOUS or MROPE_INTERLEAVED

    # widths of the stored rows and of the two patch groups (pure shape bookkeeping)
    @property
    def row_k(self) -> int:
        if self.kind == GQA:
            return self.num_kv_heads * self.head_dim
        return self.latent_dim + self.rope_dim

    @property
    def row_v(self) -> int:
        return self.num_kv_heads * self.head_dim if self.kind == GQA else 0

    @property
    def group_widths(self) -> tuple[int, int]:
        if self.kind == GQA:
            w = self.num_kv_heads * self.head_dim
            return (w, w)
        return (self.latent_dim, self.rope_dim)


@dataclasses.dataclass
class Item:
    """One chunk placement: canonical -> pool, relocated by ``delta`` and patched."""
    canon_k: torch.Tensor                 # bf16 [L][T][row_k]
    canon_v: Optional[torch.Tensor]       # bf16 [L][T][row_v] (GQA) or None (MLA)
    patch_u: Optional[torch.Tensor]       # bf16 [l1-l0][2][T][m] or None
    patch_vt: Optional[torch.Tensor]      # bf16 [l1-l0][m*(W0+W1)] or None
    delta: int
    num_tokens: int
    req: int
    start_tok: int
    patch_m: int = 0
    patch_l0: int = 0
    patch_l1: int = 0
    chunk_id: int = -1                    # which distinct canonical this item reads
    delta_h: Optional[int] = None         # M-RoPE h / w offsets (None: same as delta)
    delta_w: Optional[int] = None


@dataclasses.dataclass
class AnchorItem:
    """One placement of keys stored before rotation, re-anchored at per-token positions."""
    canon_k: torch.Tensor                 # bf16 [L][T][row_k], unrotated keys
    canon_v: Optional[torch.Tensor]       # bf16 [L][T][row_v] (GQA) or None (MLA)
    positions: torch.Tensor               # int64 [T] (1-D RoPE) or [T][3] (t, h, w; M-RoPE)
    num_tokens: int
    req: int
    start_tok: int
    chunk_id: int = -1


@dataclasses.dataclass
class Span:
    """A run of tokens already in the pool, to be relocated in place (survivors)."""
    req: int
    start_tok: int
    num_tokens: int
    delta: int


@dataclasses.dataclass
class Workload:
    name: str
    layout: Layout
    items: list
    page_table: torch.Tensor              # int32 [num_reqs][pt_stride]
    num_slots: int
    spans: list = dataclasses.field(default_factory=list)
    k_pool: Optional[torch.Tensor] = None  # pre-filled pool (relocate workloads)
    meta: dict = dataclasses.field(default_factory=dict)


def sub_seed(seed: int, *tags) -> int:
    """Deterministic 63-bit seed for one random stream, from the base seed and role tags."""
    key = repr((int(seed),) + tuple(tags)).encode()
    ss = np.random.SeedSequence([zlib.crc32(key), int(seed) & 0xFFFFFFFF, len(key)])
    return int(ss.generate_state(2, dtype=np.uint64)[0] & ((1 << 63) - 1))


def _gen(device, seed: int, *tags) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(sub_seed(seed, *tags))
    return g


def normal_bf16(shape, std: float, gen: torch.Generator, device, chunk_elems: int = 1 << 28) -> torch.Tensor:
    """bf16 RNE of N(0, std²) float32 draws, generated in slices to bound temporaries."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        tmp = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        flat[s:e].copy_(tmp)  # float32 -> bf16 conversion is round-to-nearest-even
        del tmp
    return out


def shuffled_page_table(num_reqs: int, pages_per_req: int, gen: torch.Generator,
                        total_pages: Optional[int] = None) -> torch.Tensor:
    """Page table whose entries are a seeded random permutation of the pool's pages."""
    total = total_pages if total_pages is not None else num_reqs * pages_per_req
    perm = torch.randperm(total, generator=gen, device="cpu", dtype=torch.int64)
    return perm[: num_reqs * pages_per_req].to(torch.int32).view(num_reqs, pages_per_req).contiguous()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def patch_tensors(layout: Layout, T: int, m: int, n_layers: int, gen, device,
                  strong: bool, std_weak: float = 0.02):
    """U·Σ and V_mᵀ factors for ``n_layers`` patched layers.

    weak: U, Vt ~ N(0, std_weak²) (the tiny reference config);
    strong: U ~ N(0,1), Vt ~ N(0, (0.3/sqrt(m))²): |U Vt| of order 0.3, inside the deficit
    norms the paper reports for deep layers (§4, 0.08 -> 0.49).
    """
    w0, w1 = layout.group_widths
    su, sv = (1.0, 0.3 / np.sqrt(m)) if strong else (std_weak, std_weak)
    u = normal_bf16((n_layers, 2, T, m), su, gen, device)
    vt = normal_bf16((n_layers, m * (w0 + w1)), sv, gen, device)
    return u, vt


def _outlier_scale_(x: torch.Tensor, frac: float, factor: float, gen: torch.Generator):
    """Scale ``frac`` of the last-dim channels of each [L] slice by ``factor`` (in place)."""
    L, _, W = x.shape
    k = max(1, int(round(frac * W)))
    for l in range(L):
        ch = torch.randperm(W, generator=gen, device="cpu")[:k].to(x.device)
        x[l, :, ch] = (x[l, :, ch].float() * factor).to(torch.bfloat16)


# --------------------------------------------------------------------------------------
# generic builders
# --------------------------------------------------------------------------------------

def reuse_workload(name: str, layout: Layout, *, n_chunks: int, T: int, placements,
                   m: int, l0: int, l1: int, seed: int, device="cpu", strong=True,
                   std_weak=0.02, pages_per_req: Optional[int] = None,
                   extra_pages: int = 0, outliers: bool = False,
                   patch_per_item: bool = False) -> Workload:
    """Items that place ``n_chunks`` distinct canonicals into requests.

    ``T`` is one chunk length or a list with one length per chunk (ragged batches).
    ``placements`` is a list of (chunk, req, start_tok, delta). One patch per chunk is shared
    by every placement of it (the paper's orbit patch, §5 Reorder) unless ``patch_per_item``.
    """
    L = layout.num_layers
    Ts = list(T) if isinstance(T, (list, tuple)) else [int(T)] * n_chunks
    canon_k, canon_v, patches = [], [], []
    for c in range(n_chunks):
        gk = _gen(device, seed, name, "canon_k", c)
        k = normal_bf16((L, Ts[c], layout.row_k), 1.0, gk, device)
        if outliers:
            _outlier_scale_(k, 0.01, 8.0, _gen("cpu", seed, name, "outk", c))
        canon_k.append(k)
        if layout.kind == GQA:
            gv = _gen(device, seed, name, "canon_v", c)
            v = normal_bf16((L, Ts[c], layout.row_v), 1.0, gv, device)
            if outliers:
                _outlier_scale_(v, 0.01, 8.0, _gen("cpu", seed, name, "outv", c))
            canon_v.append(v)
        else:
            canon_v.append(None)
    n_patch_sets = len(placements) if patch_per_item else n_chunks
    if m > 0 and l1 > l0:
        for c in range(n_patch_sets):
            gp = _gen(device, seed, name, "patch", c)
            Tc = Ts[placements[c][0]] if patch_per_item else Ts[c]
            patches.append(patch_tensors(layout, Tc, m, l1 - l0, gp, device, strong, std_weak))
    reqs = max(p[1] for p in placements) + 1 if placements else 0
    if pages_per_req is None:
        end = max((p[2] + Ts[p[0]] for p in placements), default=0)
        pages_per_req = max(1, -(-end // layout.page_size))
    total_pages = reqs * pages_per_req + extra_pages
    pt = shuffled_page_table(reqs, pages_per_req, _gen("cpu", seed, name, "pages"), total_pages)
    items = []
    for idx, (c, r, s, d) in enumerate(placements):
        pu = pv = None
        if patches:
            pu, pv = patches[idx if patch_per_item else c]
        items.append(Item(canon_k=canon_k[c], canon_v=canon_v[c], patch_u=pu, patch_vt=pv,
                          delta=int(d), num_tokens=Ts[c], req=r, start_tok=s,
                          patch_m=m if pu is not None else 0,
                          patch_l0=l0 if pu is not None else 0,
                          patch_l1=l1 if pu is not None else 0, chunk_id=c))
    return Workload(name=name, layout=layout, items=items, page_table=pt,
                    num_slots=total_pages * layout.page_size,
                    meta=dict(n_chunks=n_chunks, T=Ts, m=m, l0=l0, l1=l1, seed=seed))


# --------------------------------------------------------------------------------------
# the five reference workloads
# --------------------------------------------------------------------------------------

def config1(seed: int = 0, device="cpu", strong: bool = False) -> Workload:
    """Tiny GQA reuse: 2 layers, one chunk T=256, H_kv=2, hd=64, NeoX-half RoPE θ=1e4,
    canonical at p=0 relocated by δ=1000, K/V ~ N(0,1), rank-8 patch on both layers with
    U, V ~ N(0, 0.02²) (``strong`` switches to the strong-patch variant), 16 shuffled pages."""
    lay = Layout(kind=GQA, num_layers=2, page_size=16, num_kv_heads=2, head_dim=64,
                 rope_dim=64, rope_style=NEOX_HALF, rope_theta=1e4)
    return reuse_workload("cfg1" + ("_strong" if strong else ""), lay, n_chunks=1, T=256,
                          placements=[(0, 0, 0, 1000)], m=8, l0=0, l1=2, seed=seed,
                          device=device, strong=strong)


def config2(seed: int = 0, device="cpu") -> Workload:
    """GQA reorder (Qwen2-VL-7B-like): 28 layers, H_kv=4, hd=128, θ=1e6, three T=1024 chunks
    (1% outlier channels ×8) placed in all 6 orderings (18 placements), one orbit patch per
    chunk with m=32 on layers 14–27, page size 16. Canonicals sit at p0=0, so position j of an
    ordering gets δ = j·1024."""
    lay = Layout(kind=GQA, num_layers=28, page_size=16, num_kv_heads=4, head_dim=128,
                 rope_dim=128, rope_style=NEOX_HALF, rope_theta=1e6)
    T = 1024
    placements = []
    for r, perm in enumerate(itertools.permutations(range(3))):
        for j, c in enumerate(perm):
            placements.append((c, r, j * T, j * T))
    return reuse_workload("cfg2", lay, n_chunks=3, T=T, placements=placements, m=32,
                          l0=14, l1=28, seed=seed, device=device, outliers=True)


def config2_mrope(seed: int = 0, device="cpu") -> Workload:
    """The GQA reorder workload with Qwen2.5-VL's M-RoPE: sections of 16|24|24 rope pairs over
    t, h, w (Fig. 2), blocked. Each chunk is a 1024-token video segment of 4 × 16 × 16 merged
    tokens; position j of an ordering moves its t coordinate by j·1024 (as the 1-D workload
    does) and its h and w coordinates by j·16 (one 16 × 16 grid per segment), so the three
    sections turn by different offsets."""
    w = config2(seed, device)
    lay = dataclasses.replace(w.layout, mrope_section=(16, 24, 24), mrope_style=MROPE_CONTIGUOUS)
    items = [dataclasses.replace(it, delta_h=(it.delta // 1024) * 16,
                                 delta_w=(it.delta // 1024) * 16) for it in w.items]
    return dataclasses.replace(w, name="cfg2_mrope", layout=lay, items=items)


def image_positions(layout: Layout, base: int, grid) -> torch.Tensor:
    """Request positions of the tokens of one image or video segment placed at ``base``:
    [T] = base + token index under 1-D RoPE; [T][3] = (base + frame, base + row, base + col)
    for a (frames, rows, cols) grid of merged tokens under M-RoPE (Fig. 2 (a): every merged
    token gets a (t, h, w) coordinate)."""
    f, r, c = grid
    if not any(layout.mrope_section):
        return base + torch.arange(f * r * c, dtype=torch.int64)
    ft, rt, ct = torch.meshgrid(torch.arange(f), torch.arange(r), torch.arange(c), indexing="ij")
    return base + torch.stack([ft, rt, ct], dim=-1).reshape(-1, 3).to(torch.int64)


def anchor_workload(name: str, layout: Layout, *, grids, placements, seed: int = 0,
                    device="cpu", extra_pages: int = 0) -> Workload:
    """Keys stored before rotation (one per grid), placed by ``placements`` =
    [(chunk, req, start_tok, base_position)] and re-anchored at their request positions."""
    g = _gen(device, seed, name, "canon")
    Ts = [f * r * c for f, r, c in grids]
    canon_k = [normal_bf16((layout.num_layers, T, layout.row_k), 1.0, g, device) for T in Ts]
    canon_v = [normal_bf16((layout.num_layers, T, layout.row_v), 1.0, g, device)
               if layout.kind == GQA else None for T in Ts]
    reqs = max(p[1] for p in placements) + 1
    end = max(p[2] + Ts[p[0]] for p in placements)
    pages_per_req = (end + layout.page_size - 1) // layout.page_size + extra_pages
    pt = shuffled_page_table(reqs, pages_per_req, _gen("cpu", seed, name, "pages"))
    items = [AnchorItem(canon_k=canon_k[c], canon_v=canon_v[c],
                        positions=image_positions(layout, base, grids[c]).to(device),
                        num_tokens=Ts[c], req=r, start_tok=s, chunk_id=c)
             for c, r, s, base in placements]
    return Workload(name=name, layout=layout, items=items, page_table=pt,
                    num_slots=reqs * pages_per_req * layout.page_size)


def config_reanchor(seed: int = 0, device="cpu") -> Workload:
    """QV-PIC-style re-anchoring on the reorder shape: Qwen2.5-VL layout (28 layers, H_kv=4 x
    128, θ=1e6, M-RoPE 16|24|24), three rendered images of 32 x 32 merged tokens (T = 1024)
    stored before rotation, placed in all 6 orderings (18 placements) after a 16-token prefix;
    the image at ordering position j starts at position 16 + 33·j (an image spans 32 rows /
    columns, and the next starts one past its largest coordinate)."""
    lay = Layout(kind=GQA, num_layers=28, page_size=16, num_kv_heads=4, head_dim=128,
                 rope_dim=128, rope_style=NEOX_HALF, rope_theta=1e6, mrope_section=(16, 24, 24),
                 mrope_style=MROPE_CONTIGUOUS)
    placements = []
    for r, perm in enumerate(itertools.permutations(range(3))):
        for j, c in enumerate(perm):
            placements.append((c, r, 16 + j * 1024, 16 + 33 * j))
    return anchor_workload("reanchor", lay, grids=[(1, 32, 32)] * 3, placements=placements,
                           seed=seed, device=device)


def config3_deltas(seed: int = 0, n_chunks: int = 64) -> list:
    """The MLA recall workload's offsets: δ ~ U[-32768, 32768] per chunk."""
    g = _gen("cpu", seed, "cfg3", "delta")
    return torch.randint(-32768, 32769, (n_chunks,), generator=g).tolist()


def config5_deltas(seed: int = 0, n_items: int = 1024) -> list:
    """The recall sweep's offsets: δ ~ U[0, 131072) per item."""
    g = _gen("cpu", seed, "cfg5", "delta")
    return torch.randint(0, 131072, (n_items,), generator=g).tolist()


def config3(seed: int = 0, device="cpu", n_chunks: int = 64) -> Workload:
    """MLA (DeepSeek-V2-Lite-shaped): 27 layers, c_KV 512 ‖ k_pe 64, θ=1e4, T=1024 chunks each
    recalled into its own request at δ ~ U[-32768, 32768], m=32 on both groups for layers
    13–26. The paper's setting is one chunk; ``n_chunks`` of them form the batch."""
    lay = Layout(kind=MLA, num_layers=27, page_size=16, latent_dim=512, rope_dim=64,
                 rope_style=NEOX_HALF, rope_theta=1e4)
    deltas = config3_deltas(seed, n_chunks)
    placements = [(c, c, 0, deltas[c]) for c in range(n_chunks)]
    return reuse_workload("cfg3", lay, n_chunks=n_chunks, T=1024, placements=placements,
                          m=32, l0=13, l1=27, seed=seed, device=device)


def config4(seed: int = 0, device="cpu", n_seq: int = 64, layers: int = 32,
            heads: int = 32) -> Workload:
    """MHA sliding-window survival: 32 layers, 32 heads, hd=128, θ=1e4, 64 sequences with a
    window of 8 chunks × 576 tokens already in the K pool; the window slides by one chunk, so
    tokens [576, 4608) of each sequence are re-rotated in place by δ=-576 (no patch; V is
    neither read nor allocated)."""
    lay = Layout(kind=GQA, num_layers=layers, page_size=16, num_kv_heads=heads, head_dim=128,
                 rope_dim=128, rope_style=NEOX_HALF, rope_theta=1e4)
    chunk, window = 576, 8
    tokens = chunk * window
    ppr = tokens // lay.page_size
    pt = shuffled_page_table(n_seq, ppr, _gen("cpu", seed, "cfg4", "pages"))
    num_slots = n_seq * ppr * lay.page_size
    pool = normal_bf16((layers, num_slots, lay.row_k), 1.0, _gen(device, seed, "cfg4", "pool"),
                       device)
    spans = [Span(req=r, start_tok=chunk, num_tokens=tokens - chunk, delta=-chunk)
             for r in range(n_seq)]
    return Workload(name="cfg4", layout=lay, items=[], page_table=pt, num_slots=num_slots,
                    spans=spans, k_pool=pool, meta=dict(chunk=chunk, window=window, seed=seed))


def config5(seed: int = 0, device="cpu", n_req: int = 256, recalls: int = 4,
            layer_slices: int = 8) -> Workload:
    """Batched GQA recall sweep: 64 layers, H_kv=8, hd=128, θ=1e6, 256 requests × 4 recalls of
    T=1024 at δ ~ U[0, 131072), a fresh m=64 patch per item on layers 32–63, shuffled pages.

    Capacity staging: the literal pool (256 GiB) and store do not fit next to each other, so
    the 64 layers run as 8 launches of an 8-layer slice. Each item's canonical holds 8 layer
    slices that every launch reads again (launch g covers layers 8g..8g+7), the pool holds 8
    layers that every launch overwrites, and the patch store holds all 32 patched layers.
    Every (item, layer) still reads and writes its own HBM bytes."""
    T, L, Ls = 1024, 64, layer_slices
    lay_full = Layout(kind=GQA, num_layers=L, page_size=16, num_kv_heads=8, head_dim=128,
                      rope_dim=128, rope_style=NEOX_HALF, rope_theta=1e6)
    lay = dataclasses.replace(lay_full, num_layers=Ls)
    n_items = n_req * recalls
    deltas = config5_deltas(seed, n_items)
    ppr = recalls * T // lay.page_size
    pt = shuffled_page_table(n_req, ppr, _gen("cpu", seed, "cfg5", "pages"))
    W = lay.row_k
    m, pl0, pl1 = 64, 32, 64
    canon_k = normal_bf16((n_items, Ls, T, W), 1.0, _gen(device, seed, "cfg5", "ck"), device)
    canon_v = normal_bf16((n_items, Ls, T, W), 1.0, _gen(device, seed, "cfg5", "cv"), device)
    gp = _gen(device, seed, "cfg5", "patch")
    su, sv = 1.0, 0.3 / np.sqrt(m)
    pu = normal_bf16((n_items, pl1 - pl0, 2, T, m), su, gp, device)
    pv = normal_bf16((n_items, pl1 - pl0, m * 2 * W), sv, gp, device)
    items = []
    for i in range(n_items):
        items.append(Item(canon_k=canon_k[i], canon_v=canon_v[i], patch_u=pu[i], patch_vt=pv[i],
                          delta=int(deltas[i]), num_tokens=T, req=i // recalls,
                          start_tok=(i % recalls) * T, patch_m=m, patch_l0=pl0, patch_l1=pl1,
                          chunk_id=i))
    return Workload(name="cfg5", layout=lay, items=items, page_table=pt,
                    num_slots=n_req * ppr * lay.page_size,
                    meta=dict(full_layout=lay_full, layer_slices=Ls, m=m, l0=pl0, l1=pl1,
                              canon_k=canon_k, canon_v=canon_v, patch_u=pu, patch_vt=pv,
                              seed=seed))


def config5_launch_items(wl: Workload, launch: int) -> list:
    """Items of launch ``launch`` of the staged 64-layer sweep: layers 8g..8g+7 of the full
    model, expressed against the 8-layer slice layout (canonical slices reused, patch layers
    offset into the patch store)."""
    Ls = wl.meta["layer_slices"]
    pl0, pl1 = wl.meta["l0"], wl.meta["l1"]
    lo, hi = launch * Ls, (launch + 1) * Ls
    a, b = max(lo, pl0), min(hi, pl1)
    out = []
    for it in wl.items:
        if a < b:
            pu = it.patch_u[a - pl0: b - pl0]
            pv = it.patch_vt[a - pl0: b - pl0]
            out.append(dataclasses.replace(it, patch_u=pu, patch_vt=pv, patch_l0=a - lo,
                                           patch_l1=b - lo))
        else:
            out.append(dataclasses.replace(it, patch_u=None, patch_vt=None, patch_m=0,
                                           patch_l0=0, patch_l1=0))
    return out


def deficit_problems(n: int, T: int, W: int, *, k: int, rank: int, decay: float,
                     noise: float, seed: int = 0, shared_omega: bool = True, scale: float = 0.3,
                     device="cpu"):
    """Synthetic conditioning deficits for patch forming and their random test matrices.

    Δ_i = A_i diag(scale·decay^j) B_iᵀ + noise·E_i with A_i ~ N(0, 1/T) [T × rank],
    B_i ~ N(0, 1/W) [W × rank] and E_i ~ N(0, 1/max(T, W)) [T × W]: a geometric spectrum of
    ``rank`` terms whose leading value is about ``scale`` (the deficit norms the pages report
    for deep layers, §4: 0.08 to 0.49) over a noise floor of about 2·noise. Returns
    (delta float32 [n][T][W], omega float32 [W][k] when shared, else [n][W][k]); Ω ~ N(0, 1).
    """
    g = _gen("cpu", seed, "deficit", n, T, W, rank)
    s = scale * decay ** torch.arange(rank, dtype=torch.float64)
    a = torch.randn(n, T, rank, generator=g, dtype=torch.float64) / np.sqrt(T)
    b = torch.randn(n, W, rank, generator=g, dtype=torch.float64) / np.sqrt(W)
    e = torch.randn(n, T, W, generator=g, dtype=torch.float64) / np.sqrt(max(T, W))
    delta = (torch.einsum("ntr,r,nwr->ntw", a, s, b) + noise * e).to(torch.float32)
    go = _gen("cpu", seed, "omega", n, W, k, bool(shared_omega))
    omega = torch.randn((W, k) if shared_omega else (n, W, k), generator=go, dtype=torch.float32)
    return delta.to(device), omega.to(device)


CONFIGS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}
