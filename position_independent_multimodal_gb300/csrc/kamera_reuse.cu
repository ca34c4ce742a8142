// The fused relocate + patch + scatter kernel of the Kamera operator (Eq. 1; App. A
// "apply_reuse": a per-layer RoPE rotation plus a rank-m GEMM into the paged KV cache).
//
// One CTA of 128 threads takes one tile: (item, layer, channel, 128 tokens, a column tile of
// whole heads). Three paths, chosen per tile:
//   * unpatched layers: a streaming rotate/copy with 16-byte vectors (no shared memory);
//   * patched layers, rank a multiple of 8: U (the A operand) and V_m^T (the B operand) are
//     staged as K-major core matrices, one thread issues tcgen05.mma into a TMEM accumulator
//     [128 lanes = tokens][tile columns], and each thread then owns one token row: it reads
//     its accumulator row with tcgen05.ld, rotates its canonical row (staged in XOR-swizzled
//     shared memory by cp.async), adds, rounds once to bf16 and writes the row back in place;
//     the warps then store their 32 rows to the pages with coalesced 16-byte stores;
//   * patched layers with any other rank (or the FMA engine): float32 FMAs per element.
#include "kamera_dev.cuh"
#include "kamera_ptx.cuh"

namespace kamera {

namespace {

constexpr int kThr = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any MMA of one tile

__device__ __forceinline__ uint4 ldg16(const void *p) {
  return __ldg(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void stg16(void *p, const uint4 &v) {
  *reinterpret_cast<uint4 *>(p) = v;
}
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
__device__ __forceinline__ uint32_t ldg_u16(const __nv_bfloat16 *p) {
  return __ldg(reinterpret_cast<const unsigned short *>(p));
}

struct TileCtx {
  const DevLayout *lay;
  int ch, layer, t0, rows, row;
  bool rotate;
  Tile tile;
  const __nv_bfloat16 *canon;  // first row of the tile's tokens in this layer
  __nv_bfloat16 *pool;         // this layer's pool
  const long long *slots;
  const float2 *cs;
};

// ---- unpatched tiles: rotate (K / k_pe band) or copy, 16-byte vectors, 4 units in flight ----
__device__ void stream_tile(const TileCtx &c) {
  const int ppr = c.tile.ncols >> 4;
  const int u0 = c.tile.col0 >> 4;
  const int n = c.rows * ppr;
  constexpr int B = 4;
  for (int base = threadIdx.x; base < n; base += kThr * B) {
    uint4 ra[B], rb[B];
    ColUnit cu[B];
    long long sl[B];
#pragma unroll
    for (int k = 0; k < B; ++k) {
      const int w = base + k * kThr;
      sl[k] = -1;
      if (w < n) {
        const int r = w / ppr;
        cu[k] = col_unit(*c.lay, c.ch, u0 + (w - r * ppr), c.rotate);
        sl[k] = c.slots[r];
        const __nv_bfloat16 *src = c.canon + (long long)r * c.row;
        ra[k] = ldg16(src + cu[k].ca);
        rb[k] = ldg16(src + cu[k].cb);
      }
    }
#pragma unroll
    for (int k = 0; k < B; ++k) {
      if (sl[k] < 0) continue;
      __nv_bfloat16 *dst = c.pool + sl[k] * c.row;
      if (cu[k].rot == 0) {
        stg16(dst + cu[k].ca, ra[k]);
        stg16(dst + cu[k].cb, rb[k]);
      } else {
        float xa[8], xb[8];
        unpack8(ra[k], xa);
        unpack8(rb[k], xb);
        rotate_unit(cu[k], c.cs, xa, xb);
        stg16(dst + cu[k].ca, pack8_rn(xa));
        stg16(dst + cu[k].cb, pack8_rn(xb));
      }
    }
  }
}

// ---- patched tiles on CUDA cores (any rank) ----
__device__ void fma_tile(const TileCtx &c, const kamera_item &it) {
  const DevLayout &lay = *c.lay;
  const int m = it.patch_m;
  const int li = c.layer - it.patch_l0;
  const int g = c.tile.group;
  const __nv_bfloat16 *U = static_cast<const __nv_bfloat16 *>(it.patch_u) +
                           ((long long)(li * 2 + g) * it.num_tokens + c.t0) * m;
  const int wg = g == 0 ? lay.w0 : lay.w1;
  const __nv_bfloat16 *vt = static_cast<const __nv_bfloat16 *>(it.patch_vt) +
                            (long long)li * m * (lay.w0 + lay.w1) +
                            (g == 0 ? 0 : (long long)m * lay.w0);
  const int ppr = c.tile.ncols >> 4;
  const int u0 = c.tile.col0 >> 4;
  for (int w = threadIdx.x; w < c.rows * ppr; w += kThr) {
    const int r = w / ppr;
    const long long slot = c.slots[r];
    if (slot < 0) continue;
    const ColUnit cu = col_unit(lay, c.ch, u0 + (w - r * ppr), c.rotate);
    const __nv_bfloat16 *src = c.canon + (long long)r * c.row;
    float xa[8], xb[8];
    unpack8(ldg16(src + cu.ca), xa);
    unpack8(ldg16(src + cu.cb), xb);
    rotate_unit(cu, c.cs, xa, xb);
    float pa[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float pb[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const __nv_bfloat16 *ur = U + (long long)r * m;
    for (int j = 0; j < m; ++j) {
      const float uj = __bfloat162float(ur[j]);
      float va[8], vb[8];
      unpack8(ldg16(vt + (long long)j * wg + cu.gca), va);
      unpack8(ldg16(vt + (long long)j * wg + cu.gcb), vb);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        pa[e] = fmaf(uj, va[e], pa[e]);
        pb[e] = fmaf(uj, vb[e], pb[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      xa[e] += pa[e];
      xb[e] += pb[e];
    }
    __nv_bfloat16 *dst = c.pool + slot * c.row;
    stg16(dst + cu.ca, pack8_rn(xa));
    stg16(dst + cu.cb, pack8_rn(xb));
  }
}

// ---- patched tiles on the tensor cores ----
__device__ __forceinline__ void add_acc(float *x, const uint32_t *acc) {
#pragma unroll
  for (int e = 0; e < 8; ++e) x[e] += __uint_as_float(acc[e]);
}

__device__ void mma_tile(const TileCtx &c, const kamera_item &it, const SmemPlan &P,
                         unsigned char *smem, unsigned *status) {
  const DevLayout &lay = *c.lay;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t s0 = ptx::smem_addr(smem);
  const uint32_t s_canon = s0 + P.canon, s_a = s0 + P.a_op, s_b = s0 + P.b_op;
  const uint32_t s_tmem = s0 + P.misc, s_bar = s0 + P.misc + 8;
  const int m = it.patch_m, Kp = (m + 15) & ~15, NC = c.tile.ncols;
  uint32_t ncols_alloc = 32;
  while (ncols_alloc < (uint32_t)NC) ncols_alloc <<= 1;

  if (warp == 0) {
    ptx::tmem_alloc(s_tmem, ncols_alloc);
    ptx::tmem_relinquish();
  }
  if (tid == 0) {
    ptx::mbar_init(s_bar, 1);
    ptx::fence_mbar_init();
  }

  // canonical tile -> shared (rows past the chunk's end are zero), chunk c of row r stored
  // at chunk (c ^ (r & 7)) so row-per-thread reads hit 8 distinct bank groups
  const int cpr = NC >> 3;
  for (int e = tid; e < kTileRows * cpr; e += kThr) {
    const int r = e / cpr, ck = e - r * cpr;
    const bool ok = r < c.rows;
    const __nv_bfloat16 *src = c.canon + (long long)(ok ? r : 0) * c.row + c.tile.col0 + 8 * ck;
    ptx::cp_async16(s_canon + r * P.pitch + ((ck ^ (r & 7)) << 4), src, ok ? 16u : 0u);
  }
  // A operand: U rows of this tile (group g), core matrix (r/8, k/8) at ((k/8)*16 + r/8)*128
  const int g = c.tile.group;
  const int li = c.layer - it.patch_l0;
  const __nv_bfloat16 *U = static_cast<const __nv_bfloat16 *>(it.patch_u) +
                           ((long long)(li * 2 + g) * it.num_tokens + c.t0) * m;
  const int kcs = Kp >> 3;
  for (int e = tid; e < kTileRows * kcs; e += kThr) {
    const int r = e / kcs, kc = e - r * kcs;
    const bool ok = r < c.rows && kc * 8 < m;
    ptx::cp_async16(s_a + ((kc * 16 + (r >> 3)) << 7) + ((r & 7) << 4),
                    ok ? (const void *)(U + (long long)r * m + kc * 8) : (const void *)U,
                    ok ? 16u : 0u);
  }
  ptx::cp_async_commit();
  // B operand: element (n, k) = V_m^T[k][gcol0 + n]; core matrix (n/8, k/8) at
  // ((k/8)*(NC/8) + n/8)*128; gathered down the columns of V_m^T (coalesced along n)
  const int wg = g == 0 ? lay.w0 : lay.w1;
  const __nv_bfloat16 *vt = static_cast<const __nv_bfloat16 *>(it.patch_vt) +
                            (long long)li * m * (lay.w0 + lay.w1) +
                            (g == 0 ? 0 : (long long)m * lay.w0) + c.tile.gcol0;
  const int ncore = NC >> 3;
  for (int e = tid; e < kcs * NC; e += kThr) {
    const int kb = e / NC, n = e - kb * NC;
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      const int k0 = kb * 8 + j;
      const uint32_t lo = k0 < m ? ldg_u16(vt + (long long)k0 * wg + n) : 0u;
      const uint32_t hi = k0 + 1 < m ? ldg_u16(vt + (long long)(k0 + 1) * wg + n) : 0u;
      w[j >> 1] = lo | (hi << 16);
    }
    sts16(s_b + ((kb * ncore + (n >> 3)) << 7) + ((n & 7) << 4), make_uint4(w[0], w[1], w[2], w[3]));
  }
  ptx::cp_async_wait_all();
  ptx::fence_proxy_async_smem();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + P.misc);

  if (tid == 0) {
    const uint32_t idesc = ptx::idesc_bf16_f32(kTileRows, NC);
    const uint32_t lbo_a = 16 * 128, lbo_b = ncore * 128, sbo = 128;
    for (int ks = 0; ks < Kp / 16; ++ks) {
      const uint64_t ad = ptx::smem_desc(s_a + ks * 2 * lbo_a, lbo_a, sbo);
      const uint64_t bd = ptx::smem_desc(s_b + ks * 2 * lbo_b, lbo_b, sbo);
      ptx::mma_bf16(tmem, ad, bd, idesc, ks > 0 ? 1u : 0u);
    }
    ptx::mma_commit(s_bar);
  }
  const bool done = ptx::mbar_wait(s_bar, 0, kWaitLimitNs);
  ptx::tc_fence_after();

  if (done) {
    // epilogue: this thread owns token row tid = TMEM lane tid
    const int r = tid;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    const uint32_t crow = s_canon + r * P.pitch;
    const int sw = r & 7;
    const int band = c.tile.band;
    if (band == 0) {
      for (int ck = 0; ck < cpr; ck += 2) {
        uint32_t acc[16];
        ptx::tmem_ld8(trow + ck * 8, acc);
        ptx::tmem_ld8(trow + ck * 8 + 8, acc + 8);
        ptx::tmem_ld_wait(acc);
        ptx::tmem_ld_wait(acc + 8);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint32_t addr = crow + (((ck + q) ^ sw) << 4);
          float x[8];
          unpack8(lds16(addr), x);
          add_acc(x, acc + 8 * q);
          sts16(addr, pack8_rn(x));
        }
      }
    } else if (lay.style == KAMERA_ROPE_NEOX_HALF) {
      const int half = band >> 1;
      for (int h0 = 0; h0 < NC; h0 += band) {
        for (int i = 0; i < half; i += 8) {
          const int ca = h0 + i, cb = ca + half;
          uint32_t acc[16];
          ptx::tmem_ld8(trow + ca, acc);
          ptx::tmem_ld8(trow + cb, acc + 8);
          ptx::tmem_ld_wait(acc);
          ptx::tmem_ld_wait(acc + 8);
          const uint32_t aa = crow + (((ca >> 3) ^ sw) << 4);
          const uint32_t ab = crow + (((cb >> 3) ^ sw) << 4);
          float xa[8], xb[8];
          unpack8(lds16(aa), xa);
          unpack8(lds16(ab), xb);
#pragma unroll
          for (int e = 0; e < 8; ++e) rot_pair(xa[e], xb[e], c.cs[i + e]);
          add_acc(xa, acc);
          add_acc(xb, acc + 8);
          sts16(aa, pack8_rn(xa));
          sts16(ab, pack8_rn(xb));
        }
      }
    } else {  // interleaved pairs (2i, 2i+1) of each band
      for (int ck = 0; ck < cpr; ++ck) {
        uint32_t acc[8];
        ptx::tmem_ld8(trow + ck * 8, acc);
        ptx::tmem_ld_wait(acc);
        const uint32_t addr = crow + ((ck ^ sw) << 4);
        float x[8];
        unpack8(lds16(addr), x);
        const int f0 = ((ck * 8) % band) >> 1;
#pragma unroll
        for (int e = 0; e < 8; e += 2) rot_pair(x[e], x[e + 1], c.cs[f0 + (e >> 1)]);
        add_acc(x, acc);
        sts16(addr, pack8_rn(x));
      }
    }
    __syncwarp();
    // store this warp's 32 rows: consecutive lanes take consecutive 16-byte chunks of a row
    for (int e = lane; e < 32 * cpr; e += 32) {
      const int rr = warp * 32 + e / cpr, ck = e % cpr;
      if (rr >= c.rows) continue;
      const long long slot = c.slots[rr];
      if (slot < 0) continue;
      const uint4 v = lds16(s_canon + rr * P.pitch + ((ck ^ (rr & 7)) << 4));
      stg16(c.pool + slot * c.row + c.tile.col0 + 8 * ck, v);
    }
  } else if (tid == 0) {
    atomicOr(status, KAMERA_DEVICE_TIMEOUT);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tmem, ncols_alloc);
}

__global__ void __launch_bounds__(kThr) reuse_kernel(const __grid_constant__ ReuseArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const DevLayout &lay = a.lay;
  const bool batch = a.items != nullptr;
  const kamera_item it = batch ? a.items[blockIdx.y] : a.single;
  if (batch && item_check(it, lay, a.pool, a.max_tokens, a.max_m) != 0) {
    if (blockIdx.x == 0 && blockIdx.z == 0 && threadIdx.x == 0)
      atomicOr(a.status, KAMERA_DEVICE_BAD_ITEM);
    return;
  }
  const int layer = blockIdx.z / lay.n_ch;
  const int ch = blockIdx.z - layer * lay.n_ch;
  const int tt = blockIdx.x / lay.ntile;
  const int ti = blockIdx.x - tt * lay.ntile;
  const int T = it.num_tokens;
  const int t0 = tt * kTileRows;
  if (t0 >= T) return;

  TileCtx c;
  c.lay = &lay;
  c.ch = ch;
  c.layer = layer;
  c.t0 = t0;
  c.rows = min(kTileRows, T - t0);
  c.row = ch == 0 ? lay.row_k : lay.row_v;
  c.rotate = ch == 0 && it.delta != 0;
  c.tile = tile_of(lay, ch, ti, c.rotate);
  c.canon = static_cast<const __nv_bfloat16 *>(ch == 0 ? it.canon_k : it.canon_v) +
            ((long long)layer * T + t0) * c.row;
  c.pool = (ch == 0 ? a.pool.k : a.pool.v) + (long long)layer * a.pool.num_slots * c.row;
  float2 *cs = reinterpret_cast<float2 *>(smem + a.smem.cs);
  long long *slots = reinterpret_cast<long long *>(smem + a.smem.slots);
  c.cs = cs;
  c.slots = slots;

  const int tid = threadIdx.x;
  if (c.tile.band)
    for (int i = tid; i < lay.npairs; i += kThr) cs[i] = rope_phase(a.freq.q[i], it.delta);
  for (int r = tid; r < c.rows; r += kThr)
    slots[r] = slot_of(a.pool, lay.page_size, it.req, (long long)it.start_tok + t0 + r, a.status);
  __syncthreads();

  if (!layer_patched(it, layer)) {
    stream_tile(c);
    return;
  }
  const bool tensor = a.engine == kEngineTensor && (it.patch_m & 7) == 0 &&
                      aligned16(it.patch_u);
  if (!tensor) {
    fma_tile(c, it);
    return;
  }
  mma_tile(c, it, a.smem, smem, a.status);
}

int align128(int x) { return (x + 127) & ~127; }

}  // namespace

SmemPlan reuse_smem_plan(const DevLayout &l, int max_m) {
  SmemPlan p;
  int widest = l.tw;
  if (l.kind == KAMERA_MLA && l.rope_d > widest) widest = l.rope_d;
  const int kp = max_m > 0 ? ((max_m + 15) & ~15) : 0;
  p.pitch = align128(widest * 2);
  int off = 0;
  p.canon = off;
  off += kp > 0 ? kTileRows * p.pitch : 0;
  p.a_op = off;
  off = align128(off + kTileRows * kp * 2);
  p.b_op = off;
  off = align128(off + widest * kp * 2);
  p.cs = off;
  off = align128(off + l.npairs * 8);
  p.slots = off;
  off = align128(off + kTileRows * 8);
  p.misc = off;
  off = align128(off + 16);
  p.total = off;
  return p;
}

cudaError_t launch_reuse(const ReuseArgs &a, int token_tiles, int n_items, cudaStream_t s) {
  static int configured_smem[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && a.smem.total > configured_smem[dev] && a.smem.total > 48 * 1024) {
    e = cudaFuncSetAttribute(reuse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             a.smem.total);
    if (e != cudaSuccess) return e;
    configured_smem[dev] = a.smem.total;
  }
  dim3 grid(token_tiles * a.lay.ntile, n_items, a.lay.L * a.lay.n_ch);
  reuse_kernel<<<grid, kThr, a.smem.total, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kamera
