// The fused relocate + patch + scatter kernel of the Kamera operator (Eq. 1; App. A
// "apply_reuse": a per-layer RoPE rotation plus a rank-m GEMM into the paged KV cache).
//
// Work decomposition. A task is (item, layer, channel, column tile of whole heads); its tiles
// are the chunk's tokens in runs of 128. The grid is persistent: CTA b takes tasks b, b + G,
// b + 2G, ... and walks their tiles in order through two shared-memory stages. Everything a
// tile needs -- canonical rows, page ids, U rows (A operand), V_m^T columns (B operand, only
// when the stage held another task), cos/sin table -- is issued by cp.async two tiles ahead,
// so tile k+1's data is in flight while tile k is multiplied, rotated and stored.
//
// Per tile: on patched layers one thread issues tcgen05.mma (A = U rows as K-major core
// matrices, B = V_m^T rows as MN-major core matrices, copied straight from the store) into a
// TMEM accumulator [128 lanes = tokens][tile columns]. The epilogue gives each token row to
// two threads (warps w and w+4 share TMEM lanes 32(w%4)..): they read their accumulator
// columns with tcgen05.ld, rotate the canonical row from shared memory, add, round once to
// bf16 and write the row back in place; the CTA then stores all rows to their pages with
// coalesced 16-byte stores. Tiles that neither rotate nor receive a patch are byte copies.
// Ranks that are not a multiple of 8 (or the CUDA-core engine) take the same pipeline with the
// contraction done by FMAs from the staged operands.
#include "kamera_dev.cuh"
#include "kamera_ptx.cuh"

namespace kamera {

namespace {

constexpr int kThr = 256;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any MMA of one tile

__device__ __forceinline__ uint4 lds16(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ void sts16(uint32_t a, const uint4 &v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts_u16(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"((unsigned short)v) : "memory");
}
__device__ __forceinline__ void stg16(void *p, const uint4 &v) {
  *reinterpret_cast<uint4 *>(p) = v;
}
__device__ __forceinline__ uint32_t ldg_u16(const __nv_bfloat16 *p) {
  return __ldg(reinterpret_cast<const unsigned short *>(p));
}
__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// Everything a tile needs besides the staged arrays, kept in shared memory per stage.
struct TileDesc {
  kamera_item it;
  int layer, ch, coltile, t0, rows, task;
  int valid;     // 0: no tile (the CTA's sequence has ended)
  int patched;   // this layer receives the patch
  int tensor;    // the contraction runs on tcgen05 (else FMAs)
  int off0;      // position of the tile's first token inside its first page
  int pad[2];
};

// Position in this CTA's sequence of tiles.
struct Cursor {
  int task;  // current task (>= n_tasks: finished)
  int tt;    // token tile within the task
  int ntt;   // token tiles of the task
  kamera_item it;
};

__device__ __forceinline__ void task_coords(const ReuseArgs &a, int task, int *item, int *layer,
                                            int *ch, int *coltile) {
  const int ntile = a.lay.ntile;
  *coltile = task % ntile;
  const int rest = task / ntile;
  *item = rest % a.n_items;
  const int lc = rest / a.n_items;
  *layer = lc / a.lay.n_ch;
  *ch = lc - *layer * a.lay.n_ch;
}

// Move the cursor to the first tile of the next task with work (from `task` on).
__device__ __forceinline__ void cursor_seek(const ReuseArgs &a, int n_tasks, Cursor *cur,
                                            int task) {
  for (; task < n_tasks; task += gridDim.x) {
    int item, layer, ch, ct;
    task_coords(a, task, &item, &layer, &ch, &ct);
    const kamera_item it = a.items ? a.items[item] : a.single;
    if (a.items && item_check(it, a.lay, a.pool, a.max_tokens, a.max_m) != 0) {
      if (layer == 0 && ch == 0 && ct == 0 && threadIdx.x == 0)
        atomicOr(a.status, KAMERA_DEVICE_BAD_ITEM);
      continue;
    }
    if (it.num_tokens <= 0) continue;
    cur->task = task;
    cur->tt = 0;
    cur->ntt = (it.num_tokens + kTileRows - 1) / kTileRows;
    cur->it = it;
    return;
  }
  cur->task = n_tasks;
}

__device__ __forceinline__ void cursor_next(const ReuseArgs &a, int n_tasks, Cursor *cur) {
  if (++cur->tt >= cur->ntt) cursor_seek(a, n_tasks, cur, cur->task + gridDim.x);
}

// e -> (e / n, e % n) with a shift when n is a power of two
struct DivMod {
  int n, sh;  // sh >= 0: n == 1 << sh
  __device__ __forceinline__ explicit DivMod(int n_) : n(n_), sh(-1) {
    if ((n_ & (n_ - 1)) == 0) {
      sh = 0;
      while ((1 << sh) < n_) ++sh;
    }
  }
  __device__ __forceinline__ void split(int e, int *q, int *r) const {
    if (sh >= 0) {
      *q = e >> sh;
      *r = e & (n - 1);
    } else {
      *q = e / n;
      *r = e - *q * n;
    }
  }
};

// Stage the cursor's tile into stage s (cp.async, no wait) and record its descriptor.
// b_task[s] remembers which task's B operand stage s holds.
__device__ __forceinline__ void issue_tile(const ReuseArgs &a, int n_tasks, const Cursor &cur,
                                           int s, uint32_t s0, unsigned char *smem,
                                           int *b_task) {
  const SmemPlan &P = a.smem;
  TileDesc *dsc = reinterpret_cast<TileDesc *>(smem + P.desc) + s;
  const int tid = threadIdx.x;
  if (cur.task >= n_tasks) {
    if (tid == 0) dsc->valid = 0;
    return;
  }
  int item, layer, ch, ct;
  task_coords(a, cur.task, &item, &layer, &ch, &ct);
  const kamera_item &it = cur.it;
  const int t0 = cur.tt * kTileRows;
  const int rows = min(kTileRows, it.num_tokens - t0);
  const bool rotate = ch == 0 && it.delta != 0;
  const Tile tile = tile_of(a.lay, ch, ct, rotate);
  const int row = ch == 0 ? a.lay.row_k : a.lay.row_v;
  // canonical rows
  const __nv_bfloat16 *canon = static_cast<const __nv_bfloat16 *>(ch == 0 ? it.canon_k
                                                                           : it.canon_v) +
                               ((long long)layer * it.num_tokens + t0) * row + tile.col0;
  const DivMod cpr(tile.ncols >> 3);
  const uint32_t c_dst = s0 + P.canon + s * P.stage;
  for (int e = tid; e < rows * cpr.n; e += kThr) {
    int r, ck;
    cpr.split(e, &r, &ck);
    ptx::cp_async16(c_dst + r * P.pitch + ck * 16, canon + (long long)r * row + 8 * ck, 16u);
  }
  // page ids of the tile's tokens
  const unsigned tok0 = (unsigned)it.start_tok + (unsigned)t0;
  const unsigned ps = (unsigned)a.lay.page_size;
  const unsigned p_first = tok0 / ps, off0 = tok0 - p_first * ps;
  const int npages = (int)((off0 + rows - 1) / ps) + 1;
  const int32_t *pt = a.pool.pt + (long long)it.req * a.pool.pt_stride + p_first;
  for (int e = tid; e < npages; e += kThr)
    ptx::cp_async4(s0 + P.pages + s * P.pages_stage + 4 * e, pt + e);
  // patch operands
  const bool patched = layer_patched(it, layer);
  const bool tensor = patched && a.engine == kEngineTensor && (it.patch_m & 7) == 0 &&
                      aligned16(it.patch_u);
  if (patched) {
    const int m = it.patch_m, Kp = (m + 15) & ~15;
    const int li = layer - it.patch_l0;
    const __nv_bfloat16 *U = static_cast<const __nv_bfloat16 *>(it.patch_u) +
                             ((long long)(li * 2 + tile.group) * it.num_tokens + t0) * m;
    const uint32_t a_dst = s0 + P.a_op + s * P.a_stage;
    // A: element (r, k) at ((k/8)*16 + r/8)*128 + (r%8)*16 + (k%8)*2; zero past rows and m
    if (tensor) {
      const DivMod kcs(Kp >> 3);
      for (int e = tid; e < kTileRows * kcs.n; e += kThr) {
        int r, kc;
        kcs.split(e, &r, &kc);
        const bool ok = r < rows && kc * 8 < m;
        ptx::cp_async16(a_dst + ((kc * 16 + (r >> 3)) << 7) + ((r & 7) << 4),
                        ok ? (const void *)(U + (long long)r * m + kc * 8) : (const void *)U,
                        ok ? 16u : 0u);
      }
    } else {
      for (int e = tid; e < kTileRows * Kp; e += kThr) {
        const int r = e / Kp, k = e - r * Kp;
        const uint32_t v = (r < rows && k < m) ? ldg_u16(U + (long long)r * m + k) : 0u;
        sts_u16(a_dst + (((k >> 3) * 16 + (r >> 3)) << 7) + ((r & 7) << 4) + ((k & 7) << 1), v);
      }
    }
    // B: V_m^T rows as MN-major core matrices: element (n, k) at
    // (k/8)*(NC/8)*128 + (n/8)*128 + (k%8)*16 + (n%8)*2; a 16-byte run of a V_m^T row is one
    // core-matrix row
    if (b_task[s] != cur.task) {
      const int wg = tile.group == 0 ? a.lay.w0 : a.lay.w1;
      const __nv_bfloat16 *vt = static_cast<const __nv_bfloat16 *>(it.patch_vt) +
                                (long long)li * m * (a.lay.w0 + a.lay.w1) +
                                (tile.group == 0 ? 0 : (long long)m * a.lay.w0) + tile.gcol0;
      const uint32_t b_dst = s0 + P.b_op + s * P.b_stage;
      const int ncore = cpr.n;
      for (int e = tid; e < Kp * ncore; e += kThr) {
        int k, j;
        cpr.split(e, &k, &j);
        const bool ok = k < m;
        ptx::cp_async16(b_dst + (((k >> 3) * ncore + j) << 7) + ((k & 7) << 4),
                        ok ? (const void *)(vt + (long long)k * wg + 8 * j) : (const void *)vt,
                        ok ? 16u : 0u);
      }
      b_task[s] = cur.task;
    }
  }
  // cos/sin of the tile's rotation
  if (tile.band) {
    float2 *cs = reinterpret_cast<float2 *>(smem + P.cs + s * P.cs_stage);
    for (int i = tid; i < a.lay.npairs; i += kThr) cs[i] = rope_phase(a.freq.q[i], it.delta);
  }
  if (tid == 0) {
    dsc->it = it;
    dsc->layer = layer;
    dsc->ch = ch;
    dsc->coltile = ct;
    dsc->t0 = t0;
    dsc->rows = rows;
    dsc->task = cur.task;
    dsc->valid = 1;
    dsc->patched = patched;
    dsc->tensor = tensor;
    dsc->off0 = (int)off0;
  }
}

// Patch value of 8 consecutive tile columns [n0, n0+8) of row r from the staged operands
// (the CUDA-core contraction).
__device__ __forceinline__ void fma_patch8(uint32_t a_base, uint32_t b_base, int r, int n0, int m,
                                           int ncore, float *p) {
#pragma unroll
  for (int e = 0; e < 8; ++e) p[e] = 0.f;
  for (int k = 0; k < m; ++k) {
    const float u = bf16_bits_to_float(
        lds_u16(a_base + (((k >> 3) * 16 + (r >> 3)) << 7) + ((r & 7) << 4) + ((k & 7) << 1)));
    float v[8];
    unpack8(lds16(b_base + (((k >> 3) * ncore + (n0 >> 3)) << 7) + ((k & 7) << 4)), v);
#pragma unroll
    for (int e = 0; e < 8; ++e) p[e] = fmaf(u, v[e], p[e]);
  }
}

struct PatchSrc {
  bool on, tensor;
  uint32_t trow;  // TMEM address of this row (lane) at column 0
  uint32_t a_base, b_base;
  int r, m, ncore;
};

__device__ __forceinline__ void patch8(const PatchSrc &ps, int col, float *p) {
  if (ps.tensor) {
    uint32_t acc[8];
    ptx::tmem_ld8(ps.trow + col, acc);
    ptx::tmem_ld_wait(acc);
#pragma unroll
    for (int e = 0; e < 8; ++e) p[e] = __uint_as_float(acc[e]);
  } else {
    fma_patch8(ps.a_base, ps.b_base, ps.r, col, ps.m, ps.ncore, p);
  }
}

__device__ __forceinline__ void patch16(const PatchSrc &ps, int ca, int cb, float *pa,
                                        float *pb) {
  if (ps.tensor) {  // both loads in flight before one wait
    uint32_t acc[16];
    ptx::tmem_ld8(ps.trow + ca, acc);
    ptx::tmem_ld8(ps.trow + cb, acc + 8);
    ptx::tmem_ld_wait(acc);
    ptx::tmem_ld_wait(acc + 8);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      pa[e] = __uint_as_float(acc[e]);
      pb[e] = __uint_as_float(acc[8 + e]);
    }
  } else {
    patch8(ps, ca, pa);
    patch8(ps, cb, pb);
  }
}

// Rotate and/or patch one row of the tile in place, one rounding (this thread's half of the
// units). NeoX bands: groups of 8 pairs (columns i..i+7 with partners i+band/2..); interleaved
// bands and unrotated tiles: 8-column chunks. Half h takes units u with u % 2 == h; tcgen05.ld
// is warp-collective, so all lanes of a warp walk the same units.
__device__ __forceinline__ void epilogue_row(uint32_t crow, const Tile &tile, int style,
                                             int half, const PatchSrc &ps, const float2 *cs) {
  const int NC = tile.ncols, band = tile.band;
  if (band != 0 && style == KAMERA_ROPE_NEOX_HALF) {
    const int hb = band >> 1;
    const int ngroups = NC >> 4;
    for (int g = half; g < ngroups; g += 2) {
      const int p0 = g * 8;
      const int head = p0 / hb, i = p0 - head * hb;
      const int ca = head * band + i, cb = ca + hb;
      float xa[8], xb[8];
      unpack8(lds16(crow + ca * 2), xa);
      unpack8(lds16(crow + cb * 2), xb);
      if (ps.on) {
        float pa[8], pb[8];
        patch16(ps, ca, cb, pa, pb);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          rot_pair(xa[e], xb[e], cs[i + e]);
          xa[e] += pa[e];
          xb[e] += pb[e];
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) rot_pair(xa[e], xb[e], cs[i + e]);
      }
      sts16(crow + ca * 2, pack8_rn(xa));
      sts16(crow + cb * 2, pack8_rn(xb));
    }
  } else {
    const int nchunks = NC >> 3;
    for (int ck = half; ck < nchunks; ck += 2) {
      const int col = ck * 8;
      float x[8];
      unpack8(lds16(crow + col * 2), x);
      if (band != 0) {  // interleaved pairs (2i, 2i+1)
        const int f0 = (col % band) >> 1;
#pragma unroll
        for (int e = 0; e < 8; e += 2) rot_pair(x[e], x[e + 1], cs[f0 + (e >> 1)]);
      }
      if (ps.on) {
        float p[8];
        patch8(ps, col, p);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] += p[e];
      }
      sts16(crow + col * 2, pack8_rn(x));
    }
  }
}

__global__ void __launch_bounds__(kThr, 2) reuse_kernel(const __grid_constant__ ReuseArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const SmemPlan &P = a.smem;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int n_tasks = a.lay.ntile * a.n_items * a.lay.L * a.lay.n_ch;
  const uint32_t s0 = ptx::smem_addr(smem);
  const uint32_t s_tmem = s0 + P.misc, s_bar = s0 + P.misc + 8;
  long long *slots = reinterpret_cast<long long *>(smem + P.slots);
  const TileDesc *descs = reinterpret_cast<const TileDesc *>(smem + P.desc);

  Cursor cur;
  cursor_seek(a, n_tasks, &cur, blockIdx.x);
  if (cur.task >= n_tasks) return;  // nothing for this CTA (uniform)

  if (P.tmem_cols > 0 && warp == 0) {
    ptx::tmem_alloc(s_tmem, P.tmem_cols);
    ptx::tmem_relinquish();
  }
  if (tid == 0) {
    ptx::mbar_init(s_bar, 1);
    ptx::fence_mbar_init();
  }
  int b_task[2] = {-1, -1};
  // prologue: tiles 0 and 1 in flight
  issue_tile(a, n_tasks, cur, 0, s0, smem, b_task);
  ptx::cp_async_commit();
  cursor_next(a, n_tasks, &cur);
  issue_tile(a, n_tasks, cur, 1, s0, smem, b_task);
  ptx::cp_async_commit();
  cursor_next(a, n_tasks, &cur);
  ptx::tc_fence_before();
  __syncthreads();  // TMEM address and the barrier initialisation visible
  ptx::tc_fence_after();
  const uint32_t tmem =
      P.tmem_cols > 0 ? *reinterpret_cast<volatile uint32_t *>(smem + P.misc) : 0u;

  uint32_t mma_phase = 0;
  bool timed_out = false;
  const int r = ((warp & 3) << 5) + (tid & 31);  // epilogue row (TMEM lane)
  const int half = warp >> 2;

  for (int k = 0;; ++k) {
    const int s = k & 1;
    ptx::cp_async_wait_group1();
    ptx::fence_proxy_async_smem();
    __syncthreads();  // tile k's operands, rows, page ids, cos/sin and descriptor visible
    const TileDesc &d = descs[s];
    if (!d.valid) break;
    const bool rotate = d.ch == 0 && d.it.delta != 0;
    const Tile tile = tile_of(a.lay, d.ch, d.coltile, rotate);
    const bool tensor = d.patched && d.tensor && !timed_out;
    const uint32_t a_op = s0 + P.a_op + s * P.a_stage, b_op = s0 + P.b_op + s * P.b_stage;
    if (tensor) {
      ptx::tc_fence_after();
      if (tid == 0) {
        const int Kp = (d.it.patch_m + 15) & ~15, ncore = tile.ncols >> 3;
        // B is MN-major: instruction-descriptor bit 16 set. In the no-swizzle MN-major layout
        // the descriptor's leading offset is the K-direction step between core matrices and
        // the stride offset the MN-direction step (K-major: LBO along K, SBO along M).
        const uint32_t idesc = ptx::idesc_bf16_f32(kTileRows, tile.ncols) | (1u << 16);
        const uint32_t lbo_a = 16 * 128, sbo_a = 128;
        const uint32_t k_step_b = ncore * 128, mn_step_b = 128;
        for (int ks = 0; ks < Kp / 16; ++ks) {
          const uint64_t ad = ptx::smem_desc(a_op + ks * 2 * lbo_a, lbo_a, sbo_a);
          const uint64_t bd = ptx::smem_desc(b_op + ks * 2 * k_step_b, k_step_b, mn_step_b);
          ptx::mma_bf16(tmem, ad, bd, idesc, ks > 0 ? 1u : 0u);
        }
        ptx::mma_commit(s_bar);
      }
      if (!ptx::mbar_wait(s_bar, mma_phase, kWaitLimitNs)) {
        timed_out = true;
        if (tid == 0) atomicOr(a.status, KAMERA_DEVICE_TIMEOUT);
      }
      mma_phase ^= 1;
      ptx::tc_fence_after();
    }
    const bool write = !(d.patched && timed_out);
    const uint32_t c_stage = s0 + P.canon + s * P.stage;
    if (write && (d.patched || tile.band)) {
      PatchSrc ps;
      ps.on = d.patched;
      ps.tensor = tensor;
      ps.trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
      ps.a_base = a_op;
      ps.b_base = b_op;
      ps.r = r;
      ps.m = d.it.patch_m;
      ps.ncore = tile.ncols >> 3;
      const float2 *cs = reinterpret_cast<const float2 *>(smem + P.cs + s * P.cs_stage);
      if (r < d.rows || tensor)
        epilogue_row(c_stage + r * P.pitch, tile, a.lay.style, half, ps, cs);
    }
    if (half == 0 && r < d.rows) {  // slot of this row, checked against the pool
      const int ps_ = a.lay.page_size;
      const int rel = d.off0 + r;
      const int pg = rel / ps_;
      const int page = reinterpret_cast<const int *>(smem + P.pages + s * P.pages_stage)[pg];
      long long slot = -1;
      if (page >= 0 && (long long)(page + 1) * ps_ <= a.pool.num_slots)
        slot = (long long)page * ps_ + (rel - pg * ps_);
      else
        atomicOr(a.status, KAMERA_DEVICE_SLOT_OOB);
      slots[r] = slot;
    }
    if (tensor) ptx::tc_fence_before();
    __syncthreads();  // rows complete
    if (write) {      // consecutive threads take consecutive 16-byte chunks of a row
      const DivMod cpr(tile.ncols >> 3);
      const int row = d.ch == 0 ? a.lay.row_k : a.lay.row_v;
      __nv_bfloat16 *pool = (d.ch == 0 ? a.pool.k : a.pool.v) +
                            (long long)d.layer * a.pool.num_slots * row + tile.col0;
      for (int e = tid; e < d.rows * cpr.n; e += kThr) {
        int rr, ck;
        cpr.split(e, &rr, &ck);
        const long long slot = slots[rr];
        if (slot < 0) continue;
        stg16(pool + slot * row + 8 * ck, lds16(c_stage + rr * P.pitch + ck * 16));
      }
    }
    __syncthreads();  // stage s is free
    issue_tile(a, n_tasks, cur, s, s0, smem, b_task);
    ptx::cp_async_commit();
    cursor_next(a, n_tasks, &cur);
  }
  ptx::cp_async_wait_all();
  if (P.tmem_cols > 0) {
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, P.tmem_cols);
  }
}

int align128(int x) { return (x + 127) & ~127; }

}  // namespace

SmemPlan reuse_smem_plan(const DevLayout &l, int max_m) {
  SmemPlan p;
  int widest = l.tw;
  if (l.kind == KAMERA_MLA && l.rope_d > widest) widest = l.rope_d;
  const int kp = max_m > 0 ? ((max_m + 15) & ~15) : 0;
  p.pitch = widest * 2 + 16;  // one 16-byte pad per row: rows land on different bank groups
  p.stage = align128(kTileRows * p.pitch);
  p.a_stage = align128(kTileRows * kp * 2);
  p.b_stage = align128(widest * kp * 2);
  p.cs_stage = align128(l.npairs * 8);
  p.pages_stage = align128((kTileRows / l.page_size + 2) * 4);
  // the B operands come first: every descriptor offset stays inside the allocation
  int off = 0;
  p.b_op = off;
  off += 2 * p.b_stage;
  p.a_op = off;
  off += 2 * p.a_stage;
  p.canon = off;
  off += 2 * p.stage;
  p.cs = off;
  off += 2 * p.cs_stage;
  p.pages = off;
  off += 2 * p.pages_stage;
  p.desc = off;
  off = align128(off + 2 * (int)sizeof(TileDesc));
  p.slots = off;
  off = align128(off + kTileRows * 8);
  p.misc = off;
  off = align128(off + 16);
  p.total = off;
  int cols = 0;
  if (kp > 0) {
    cols = 32;
    while (cols < widest) cols <<= 1;
  }
  p.tmem_cols = cols;
  return p;
}

cudaError_t launch_reuse(const ReuseArgs &a, int n_items, cudaStream_t s) {
  static int configured_smem[64] = {0};
  static int sm_count[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured_smem[dev] == 0) {
    e = cudaFuncSetAttribute(reuse_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    configured_smem[dev] = 1;
  }
  if (a.smem.total > configured_smem[dev] && a.smem.total > 48 * 1024) {
    e = cudaFuncSetAttribute(reuse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             a.smem.total);
    if (e != cudaSuccess) return e;
    configured_smem[dev] = a.smem.total;
  }
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reuse_kernel, kThr, a.smem.total);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  // TMEM holds 512 columns per SM; each resident CTA takes tmem_cols of them
  if (a.smem.tmem_cols > 0 && per_sm * a.smem.tmem_cols > 512) per_sm = 512 / a.smem.tmem_cols;
  const long long tasks = (long long)a.lay.ntile * n_items * a.lay.L * a.lay.n_ch;
  const long long cap = (long long)sm_count[dev] * per_sm;
  const long long grid = tasks < cap ? tasks : cap;
  reuse_kernel<<<(unsigned)grid, kThr, a.smem.total, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kamera
