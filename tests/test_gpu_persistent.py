"""The persistent path of the patched layers: a handle with a batch workspace plans a GQA/MHA
batch on the device (groups, task rows, one range of token tiles per set of CTAs) and runs the
patched layers as a persistent kernel. Every byte it writes must equal what the grid path (the
same handle without a workspace) writes, and the rows must match the float64 oracle of Eq. 1
(Kamera §5 "Reorder": one orbit patch serves every ordering of a chunk).

Each case also reads the plan's header (task rows and tiles) back from the workspace, so a
silent fall-back to the grid path cannot pass for the persistent one, and the cases that must
fall back (MLA, runs above 4) check that the header was left alone.

Cases: the six orderings of three ragged chunks (GQA with 64- and 128-column tiles; MLA falls
back) at ranks 8 and 32 and a CUDA-core rank 12; equal lengths, whose last sixth of row tiles
is handed out a tile at a time; the plan's task and tile counts; run sizes 1 to 4 (6 falls
back); M-RoPE items that share δ but not δ_h; an invalid item ahead of its group and an
out-of-range page; one batch mixing ranks, lengths and unpatched items; a batch of many
one-tile task rows, more per CTA than the kernel keeps in shared memory at once; a workspace
too small and a rank too high (both fall back); successive batches on one workspace; a
call replayed from a CUDA graph; and the timed call of the benchmark's per-kernel split, with
and without a workspace.
"""
import dataclasses
import itertools

import pytest
import torch

import position_independent_multimodal_gb300 as km
import workloads as wl
from tests import kamera_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda(cuda_ok):
    return cuda_ok


def gqa(L=3, H=2, hd=64):
    return wl.Layout(kind=wl.GQA, num_layers=L, page_size=16, num_kv_heads=H, head_dim=hd,
                     rope_dim=hd, rope_style=wl.NEOX_HALF, rope_theta=1e4)


def mla(L=3):
    return wl.Layout(kind=wl.MLA, num_layers=L, page_size=16, latent_dim=512, rope_dim=64,
                     rope_style=wl.NEOX_HALF, rope_theta=1e4)


def orderings(layout, m, name, Ts=(130, 256, 77), prefix=5):
    placements = []
    for r, perm in enumerate(itertools.permutations(range(3))):
        s = prefix
        for c in perm:
            placements.append((c, r, s, s))
            s += Ts[c]
    return wl.reuse_workload(name, layout, n_chunks=3, T=list(Ts), placements=placements, m=m,
                             l0=1, l1=layout.num_layers, seed=3, strong=True, extra_pages=2)


def run(w, items, workspace, options=None):
    """kamera_batch_reuse of the items; with `workspace`, through a batch workspace whose
    header is returned (task rows, tiles, weight, static positions, tail positions, token tiles
    per row when every row has the same), else Nones."""
    h = km.create(w.layout, **(options or {}))
    ws = None
    if workspace:
        ws = torch.full((km.kamera_batch_workspace_bytes(h, len(items)),), 0xFF,
                        dtype=torch.uint8, device="cuda")
        km.kamera_set_batch_workspace(h, ws)
    k, v, status, _ = tl.run_batch(h, w.layout, items, w.page_table, w.num_slots)
    head = (None,) * 6
    if ws is not None:
        head = tuple(ws[:24].view(torch.int32).cpu().tolist())
    return k, v, status, head


def same_bytes(a, b):
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def compare(w, items=None, options=None, status=0, oracle_items=None, persistent=True,
            tail=None):
    items = items if items is not None else tl.to_device_items(w.items)
    k, v, st, head = run(w, items, True, options)
    n_tasks, n_tiles = head[:2]
    k0, v0, st0, _ = run(w, items, False, options)
    assert st == status and st0 == status
    if persistent:
        assert n_tasks > 0 and n_tiles >= n_tasks, "the persistent path did not run"
        if tail is not None:
            assert (head[4] > 0) == tail, "tail positions handed out" if tail else "no tail"
    else:
        assert (n_tasks, n_tiles) == (-1, -1), "the persistent path ran"
    same_bytes(k, k0)
    if v is not None:
        same_bytes(v, v0)
    if oracle_items is not None:
        tl.check_full(w.layout, oracle_items, w.page_table, k, v)
    return n_tasks, n_tiles


@pytest.mark.parametrize("m", [8, 12, 32])
@pytest.mark.parametrize("shape", ["gqa64", "gqa128", "mla"])
def test_orderings_match_the_grid_path_and_the_oracle(shape, m):
    lay = {"gqa64": gqa(), "gqa128": gqa(H=4, hd=128), "mla": mla()}[shape]
    w = orderings(lay, m, f"pers{shape}{m}")
    compare(w, oracle_items=w.items, persistent=shape != "mla")


@pytest.mark.parametrize("m", [12, 32])
@pytest.mark.parametrize("shape", ["gqa64", "gqa128"])
def test_equal_lengths_hand_out_a_tail(shape, m):
    # every chunk 300 tokens (3 token tiles a row): the last sixth of the row tiles is handed
    # out one at a time, here with runs of 2 (K) and 3 (V) members
    lay = {"gqa64": gqa(), "gqa128": gqa(H=4, hd=128)}[shape]
    w = orderings(lay, m, f"perstail{shape}{m}", Ts=(300, 300, 300))
    compare(w, oracle_items=w.items, tail=True)


def test_task_and_tile_counts_of_the_plan():
    # GQA, 2 heads of 128 -> 2 column tiles; layers 1 and 2 patched. K groups: placements with
    # equal (chunk, offset); V groups: every placement of a chunk; each taken in runs of 3
    w = orderings(gqa(H=2, hd=128), 32, "perscount")

    def runs_and_tiles(key):
        groups = {}
        for it in w.items:
            groups.setdefault(key(it), []).append(it)
        runs = sum(-(-len(g) // 3) for g in groups.values())
        tiles = sum(-(-len(g) // 3) * -(-g[0].num_tokens // 128) for g in groups.values())
        return runs, tiles

    k_runs, k_tiles = runs_and_tiles(lambda it: (id(it.canon_k), it.delta))
    v_runs, v_tiles = runs_and_tiles(lambda it: id(it.canon_v))
    assert (k_runs, v_runs) == (12, 6)
    n_rows, n_tiles = compare(w, tail=False)
    assert n_rows == 2 * (k_runs + v_runs)  # task rows: 2 patched layers
    assert n_tiles == 2 * 2 * (k_tiles + v_tiles)  # x 2 column tiles


@pytest.mark.parametrize("run_patched", [1, 2, 4, 6])
def test_run_sizes(run_patched):
    w = orderings(gqa(H=4, hd=128), 16, f"persrun{run_patched}")
    compare(w, options=dict(share_run_patched=run_patched), persistent=run_patched <= 4,
            oracle_items=w.items if run_patched == 2 else None)


def test_mrope_items_share_delta_but_not_delta_h():
    lay = dataclasses.replace(gqa(L=2, H=4, hd=128), mrope_section=(16, 24, 24),
                              mrope_style=wl.MROPE_CONTIGUOUS)
    w = orderings(lay, 32, "persmrope")
    w.items = [dataclasses.replace(it, delta_h=(0 if it.req == 0 else it.delta // 7),
                                   delta_w=-it.delta) for it in w.items]
    compare(w, oracle_items=w.items)


def test_invalid_item_ahead_of_its_group():
    lay = gqa(L=2, H=4, hd=128)
    w = wl.reuse_workload("persbad", lay, n_chunks=1, T=150,
                          placements=[(0, 0, 3, 40), (0, 1, 3, 40), (0, 2, 20, 40)], m=8,
                          l0=1, l1=2, seed=5, strong=True, extra_pages=1)
    items = tl.to_device_items(w.items)
    bad = dataclasses.replace(items[0], req=99)
    compare(w, items=[bad] + items[1:], status=km.KAMERA_DEVICE_BAD_ITEM,
            oracle_items=w.items[1:])


def test_out_of_range_page_in_one_member():
    lay = gqa(L=2, H=4, hd=128)
    w = wl.reuse_workload("persoob", lay, n_chunks=1, T=200,
                          placements=[(0, 0, 0, 9), (0, 1, 0, 9)], m=32, l0=1, l1=2, seed=6,
                          strong=True, extra_pages=1)
    pt = w.page_table.clone()
    pt[1, 3] = 10 ** 6
    w = dataclasses.replace(w, page_table=pt)
    compare(w, status=km.KAMERA_DEVICE_SLOT_OOB)


def test_mixed_ranks_lengths_and_unpatched_items():
    # one batch: ranks 8, 16, 32 (tensor cores) and 12 (CUDA cores), lengths from 1 to 300
    # tokens, an item without a patch and one with no tokens; the persistent CTAs cross tasks of
    # different rank, length and engine
    lay = gqa(L=3, H=2, hd=128)
    Ts = [300, 1, 127, 128, 129, 64]
    placements = [(c, c, 3 + 16 * c, 1000 * c - 2500) for c in range(len(Ts))]
    w = wl.reuse_workload("persmix", lay, n_chunks=len(Ts), T=Ts, placements=placements, m=32,
                          l0=0, l1=3, seed=8, strong=True, extra_pages=1)
    ranks = [8, 16, 32, 12, 0, 32]
    items = []
    for it, m in zip(w.items, ranks):
        if m == 0:
            items.append(dataclasses.replace(it, patch_m=0, patch_u=None, patch_vt=None))
        else:
            u = it.patch_u[..., :m].contiguous()
            W0 = lay.num_kv_heads * lay.head_dim
            vt = it.patch_vt.view(lay.num_layers, 2, 32, W0)[:, :, :m].contiguous()
            vt = vt.view(lay.num_layers, -1)
            items.append(dataclasses.replace(it, patch_m=m, patch_u=u, patch_vt=vt))
    items.append(dataclasses.replace(items[0], num_tokens=0, req=5))
    w = dataclasses.replace(w, items=items)
    compare(w, items=tl.to_device_items(items), oracle_items=items[:-1])


def test_many_one_tile_tasks_refetch_their_records():
    # 400 short chunks, each in its own request, 10 layers (9 patched): 400 x 9 x 2 = 7200
    # one-tile task rows over two column tiles (4 heads of 64, two per tile); each CTA's own
    # range holds about 40 of them, more than one fetch of records, and the last sixth of the
    # positions is handed out one tile at a time
    lay = gqa(L=10, H=4, hd=64)
    n = 400
    Ts = [16 + (i * 37) % 100 for i in range(n)]
    placements = [(i, i, 0, 7 * i - 300) for i in range(n)]
    w = wl.reuse_workload("persmany", lay, n_chunks=n, T=Ts, placements=placements, m=8, l0=1,
                          l1=10, seed=9, strong=False, extra_pages=0)
    n_rows, n_tiles = compare(w, tail=True)
    assert n_rows == n * 9 * 2 and n_tiles == 2 * n_rows
    k, v, _, _ = run(w, tl.to_device_items(w.items), True)
    tl.check_full(lay, w.items, w.page_table, k, v)


def test_too_small_a_workspace_or_too_high_a_rank_falls_back():
    # a workspace sized for one item cannot hold the plan of 18 (the grid path runs and the
    # workspace is left alone); rank 64 at 128-column tiles leaves no room for two V_m^T
    # buffers beside two CTAs per SM
    w = orderings(gqa(H=4, hd=128), 16, "perssmall")
    items = tl.to_device_items(w.items)
    h = km.create(w.layout)
    ws = torch.full((km.kamera_batch_workspace_bytes(h, 1),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    km.kamera_set_batch_workspace(h, ws)
    k, v, st, _ = tl.run_batch(h, w.layout, items, w.page_table, w.num_slots)
    assert st == 0 and ws[:8].view(torch.int32).tolist() == [-1, -1]
    k0, v0, _, _ = run(w, items, False)
    same_bytes(k, k0)
    same_bytes(v, v0)
    w64 = orderings(gqa(H=4, hd=128), 64, "pers64")
    compare(w64, persistent=False)


def test_one_workspace_for_successive_batches():
    # two different batches, one after the other on one handle: the second plan replaces the
    # first in the workspace, and each call writes its own bytes
    lay = gqa(H=4, hd=128)
    w1 = orderings(lay, 32, "perssucc1", Ts=(300, 300, 300))
    w2 = orderings(lay, 8, "perssucc2")
    h = km.create(lay)
    n = max(len(w1.items), len(w2.items))
    ws = torch.full((km.kamera_batch_workspace_bytes(h, n),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    km.kamera_set_batch_workspace(h, ws)
    outs = []
    for w in (w1, w2, w1):
        k, v, st, _ = tl.run_batch(h, lay, tl.to_device_items(w.items), w.page_table,
                                   w.num_slots)
        assert st == 0
        outs.append((k, v))
    for (k, v), w in zip(outs, (w1, w2, w1)):
        k0, v0, _, _ = run(w, tl.to_device_items(w.items), False)
        same_bytes(k, k0)
        same_bytes(v, v0)


def test_replayed_from_a_cuda_graph():
    # the planning and persistent kernels are stream work only (the plan resets the tail
    # counters itself), so one captured call replays to the same bytes
    w = orderings(gqa(H=4, hd=128), 32, "persgraph", Ts=(300, 300, 300))
    lay = w.layout
    items = tl.to_device_items(w.items)
    h = km.create(lay)
    ws = torch.full((km.kamera_batch_workspace_bytes(h, len(items)),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    km.kamera_set_batch_workspace(h, ws)
    k, v = tl.sentinel_pool(lay, w.num_slots)
    pool = km.Pool(k, v, w.page_table.cuda(), w.num_slots)
    d_items = km.pack_items(items).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # one call outside the graph loads the kernels
        km.kamera_batch_reuse(h, d_items, len(items), 300, 32, pool, status, s)
    s.synchronize()
    k.fill_(0)
    v.fill_(0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        km.kamera_batch_reuse(h, d_items, len(items), 300, 32, pool, status, s)
    for _ in range(2):
        k.fill_(0)
        v.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        k0, v0, _, _ = run(w, items, False)
        written = k0.view(torch.int16) != wl.POOL_SENTINEL_BITS
        assert torch.equal(k.view(torch.int16)[written], k0.view(torch.int16)[written])
        assert torch.equal(v.view(torch.int16)[written], v0.view(torch.int16)[written])


@pytest.mark.parametrize("workspace", [True, False])
def test_timed_call_writes_the_same_bytes_and_orders_its_marks(workspace):
    # the per-kernel split of the benchmark: events never recorded before (the binding creates
    # them), marks before the copy kernel, between the layers, after the planning kernel (on
    # the grid path at the same point) and after the last kernel, in that order
    w = orderings(gqa(H=4, hd=128), 32, f"perstimed{int(workspace)}")
    lay = w.layout
    items = tl.to_device_items(w.items)
    h = km.create(lay)
    ws = None
    if workspace:
        ws = torch.full((km.kamera_batch_workspace_bytes(h, len(items)),), 0xFF,
                        dtype=torch.uint8, device="cuda")
        km.kamera_set_batch_workspace(h, ws)
    k, v = tl.sentinel_pool(lay, w.num_slots)
    pool = km.Pool(k, v, w.page_table.cuda(), w.num_slots)
    d_items = km.pack_items(items).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    max_t = max(it.num_tokens for it in items)
    km.kamera_batch_reuse_timed(h, d_items, len(items), max_t, 32, pool, status, ev)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    if workspace:
        assert int(ws[:4].view(torch.int32).item()) > 0, "the persistent path did not run"
    gaps = [ev[i].elapsed_time(ev[i + 1]) for i in range(3)]
    assert all(g >= 0 for g in gaps) and sum(gaps) > 0
    k0, v0, st0, _ = run(w, items, False)
    assert st0 == 0
    same_bytes(k, k0)
    same_bytes(v, v0)
