// The fused relocate + patch + scatter kernel of the Kamera operator on patched layers (Eq. 1;
// App. A "apply_reuse": a per-layer RoPE rotation plus a rank-m GEMM into the paged KV cache).
//
// One CTA of 256 threads per task = (item, layer, channel, column tile of whole heads). The CTA
// stages the task's V_m^T columns (the B operand, MN-major core matrices copied straight from
// the store) and cos/sin table once, then walks the chunk's tokens in tiles of 128 through two
// shared-memory stages: tile t+2's canonical rows and page ids are in flight (cp.async) while
// tile t is multiplied and stored, and tile t+1's U rows (the A operand, K-major core matrices)
// land while tile t's epilogue runs.
//
// Per tile one thread issues tcgen05.mma into a TMEM accumulator [128 lanes = tokens][tile
// columns]. Each token row then belongs to two threads (warps w and w+4 share TMEM lanes
// 32(w%4)..): they read their accumulator columns with tcgen05.ld, rotate the canonical row
// from shared memory, add, round once to bf16 and write the row back in place; the CTA stores
// the rows to their pages with coalesced 16-byte stores. Ranks that are not a multiple of 8
// (or the CUDA-core engine) run the same pipeline with the contraction done by FMAs from the
// staged operands. Unpatched layers never reach this kernel (see reuse_copy_kernel).
#include "kamera_dev.cuh"
#include "kamera_ptx.cuh"
#include "kamera_smem.cuh"

namespace kamera {

namespace {

constexpr int kThr = 256;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any MMA of one tile

struct PatchSrc {
  bool tensor;
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

// Rotate + patch one row of the tile in place, one rounding (this thread's half of the units).
// NeoX bands: groups of 8 pairs (columns i..i+7 with partners i+band/2..) in packed f32x2
// arithmetic: a' = b*(-sin) + (a*cos + p_a), b' = a*sin + (b*cos + p_b). Interleaved bands
// and unrotated tiles: 8-column chunks. Half h takes units u with u % 2 == h; tcgen05.ld is
// warp-collective, so all lanes of a warp walk the same units. `rot` holds cos[npairs],
// sin[npairs] and -sin[npairs] of the item's offset.
__device__ __forceinline__ void epilogue_row(uint32_t crow, const Tile &tile, int style,
                                             int half, const PatchSrc &ps, const float *rot,
                                             int npairs) {
  const int NC = tile.ncols, band = tile.band;
  if (band != 0 && style == KAMERA_ROPE_NEOX_HALF) {
    const int hb = band >> 1;
    const DivMod hbd(hb);
    const int ngroups = NC >> 4;
    for (int g = half; g < ngroups; g += 2) {
      int head, i;
      hbd.split(g * 8, &head, &i);
      const int ca = head * band + i, cb = ca + hb;
      float pa[8], pb[8];
      patch16(ps, ca, cb, pa, pb);
      const uint4 ra = lds16(crow + ca * 2), rb = lds16(crow + cb * 2);
      const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
      const float4 *cv = reinterpret_cast<const float4 *>(rot + i);
      const float4 *sv = reinterpret_cast<const float4 *>(rot + npairs + i);
      const float4 *nv = reinterpret_cast<const float4 *>(rot + 2 * npairs + i);
      uint32_t oa[4], ob[4];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float4 c4 = cv[q], s4 = sv[q], n4 = nv[q];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int j = 2 * q + h2;  // word j holds elements 2j, 2j+1
          const f32x2 c = h2 ? f2(c4.z, c4.w) : f2(c4.x, c4.y);
          const f32x2 sn = h2 ? f2(s4.z, s4.w) : f2(s4.x, s4.y);
          const f32x2 ns = h2 ? f2(n4.z, n4.w) : f2(n4.x, n4.y);
          const f32x2 a = bf2_to_f2(wa[j]), b = bf2_to_f2(wb[j]);
          const f32x2 na = fma2(b, ns, fma2(a, c, f2(pa[2 * j], pa[2 * j + 1])));
          const f32x2 nb = fma2(a, sn, fma2(b, c, f2(pb[2 * j], pb[2 * j + 1])));
          oa[j] = f2_to_bf2(na);
          ob[j] = f2_to_bf2(nb);
        }
      }
      sts16(crow + ca * 2, make_uint4(oa[0], oa[1], oa[2], oa[3]));
      sts16(crow + cb * 2, make_uint4(ob[0], ob[1], ob[2], ob[3]));
    }
  } else {
    const int nchunks = NC >> 3;
    for (int ck = half; ck < nchunks; ck += 2) {
      const int col = ck * 8;
      float p[8];
      patch8(ps, col, p);
      const uint4 rw = lds16(crow + col * 2);
      const uint32_t w[4] = {rw.x, rw.y, rw.z, rw.w};
      uint32_t o[4];
      if (band != 0) {  // interleaved pairs (2i, 2i+1)
        const int f0 = (col % band) >> 1;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float x0 = __uint_as_float(w[j] << 16), x1 = __uint_as_float(w[j] & 0xFFFF0000u);
          rot_pair(x0, x1, make_float2(rot[f0 + j], rot[npairs + f0 + j]));
          o[j] = pack2_rn(x0 + p[2 * j], x1 + p[2 * j + 1]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          o[j] = f2_to_bf2(add2(bf2_to_f2(w[j]), f2(p[2 * j], p[2 * j + 1])));
      }
      sts16(crow + col * 2, make_uint4(o[0], o[1], o[2], o[3]));
    }
  }
}

// Epilogue of one row for a compile-time tile shape: NC columns, NeoX bands of width BAND
// (0: nothing rotates), accumulator in TMEM. Half h takes the contiguous half of the units:
// NeoX pairs [h*NC/4, (h+1)*NC/4) with their partners, or 8-column chunks
// [h*NC/16, (h+1)*NC/16); every offset is a constant of the unrolled loop.
template <int NC, int BAND>
__device__ __forceinline__ void epilogue_fixed(uint32_t crow, int half, uint32_t trow,
                                               const float *rot, int npairs) {
  if constexpr (BAND > 0) {
    constexpr int HB = BAND / 2, PAIRS_HALF = NC / 4, GROUPS = PAIRS_HALF / 8;
#pragma unroll
    for (int q = 0; q < GROUPS; ++q) {
      const int p = half * PAIRS_HALF + q * 8;  // first pair of the group
      const int head = p / HB, i = p % HB;
      const int ca = head * BAND + i, cb = ca + HB;
      uint32_t acc[16];
      ptx::tmem_ld8(trow + ca, acc);
      ptx::tmem_ld8(trow + cb, acc + 8);
      const uint4 ra = lds16(crow + ca * 2), rb = lds16(crow + cb * 2);
      const float4 *cv = reinterpret_cast<const float4 *>(rot + i);
      const float4 *sv = reinterpret_cast<const float4 *>(rot + npairs + i);
      const float4 *nv = reinterpret_cast<const float4 *>(rot + 2 * npairs + i);
      ptx::tmem_ld_wait(acc);
      ptx::tmem_ld_wait(acc + 8);
      const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
      uint32_t oa[4], ob[4];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const float4 c4 = cv[h2], s4 = sv[h2], n4 = nv[h2];
#pragma unroll
        for (int g2 = 0; g2 < 2; ++g2) {
          const int j = 2 * h2 + g2;  // word j holds elements 2j, 2j+1
          const f32x2 c = g2 ? f2(c4.z, c4.w) : f2(c4.x, c4.y);
          const f32x2 sn = g2 ? f2(s4.z, s4.w) : f2(s4.x, s4.y);
          const f32x2 ns = g2 ? f2(n4.z, n4.w) : f2(n4.x, n4.y);
          const f32x2 a = bf2_to_f2(wa[j]), b = bf2_to_f2(wb[j]);
          const f32x2 pa = f2(__uint_as_float(acc[2 * j]), __uint_as_float(acc[2 * j + 1]));
          const f32x2 pb =
              f2(__uint_as_float(acc[8 + 2 * j]), __uint_as_float(acc[8 + 2 * j + 1]));
          oa[j] = f2_to_bf2(fma2(b, ns, fma2(a, c, pa)));
          ob[j] = f2_to_bf2(fma2(a, sn, fma2(b, c, pb)));
        }
      }
      sts16(crow + ca * 2, make_uint4(oa[0], oa[1], oa[2], oa[3]));
      sts16(crow + cb * 2, make_uint4(ob[0], ob[1], ob[2], ob[3]));
    }
  } else {
    constexpr int CH_HALF = NC / 16;  // 8-column chunks per half
#pragma unroll
    for (int q = 0; q < CH_HALF; q += 2) {
      const int col = (half * CH_HALF + q) * 8;
      uint32_t acc[16];
      ptx::tmem_ld8(trow + col, acc);
      ptx::tmem_ld8(trow + col + 8, acc + 8);
      const uint4 r0 = lds16(crow + col * 2), r1 = lds16(crow + col * 2 + 16);
      ptx::tmem_ld_wait(acc);
      ptx::tmem_ld_wait(acc + 8);
      const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
      uint32_t o[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        o[j] = f2_to_bf2(add2(bf2_to_f2(w[j]),
                              f2(__uint_as_float(acc[2 * j]), __uint_as_float(acc[2 * j + 1]))));
      sts16(crow + col * 2, make_uint4(o[0], o[1], o[2], o[3]));
      sts16(crow + col * 2 + 16, make_uint4(o[4], o[5], o[6], o[7]));
    }
  }
}

// Everything one CTA does for its task. NC > 0 fixes the tile width and BAND the NeoX band
// width at compile time (the tensor-core epilogue is then fully unrolled); NC == 0 is the
// general path for any tile, band, pairing and engine.
template <int NC, int BAND>
__device__ __forceinline__ void run_task(const ReuseArgs &a, unsigned char *smem,
                                         const kamera_item &it, int layer, int ch,
                                         const Tile &tile) {
  constexpr bool kFixed = NC > 0;
  const SmemPlan &P = a.smem;
  const DevLayout &lay = a.lay;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int T = it.num_tokens, m = it.patch_m, Kp = (m + 15) & ~15;
  const int ncols = kFixed ? NC : tile.ncols;
  const int ncore = ncols >> 3;
  const int row = ch == 0 ? lay.row_k : lay.row_v;
  const bool tensor = a.engine == kEngineTensor && (m & 7) == 0 && aligned16(it.patch_u);
  const bool u2 = P.u_bufs == 2;  // U of tile t+2 staged with its rows (else one buffer)
  const int li = layer - it.patch_l0;
  const __nv_bfloat16 *canon = static_cast<const __nv_bfloat16 *>(ch == 0 ? it.canon_k
                                                                           : it.canon_v) +
                               (long long)layer * T * row + tile.col0;
  const __nv_bfloat16 *U = static_cast<const __nv_bfloat16 *>(it.patch_u) +
                           (long long)(li * 2 + tile.group) * T * m;
  const int wg = tile.group == 0 ? lay.w0 : lay.w1;
  const __nv_bfloat16 *vt = static_cast<const __nv_bfloat16 *>(it.patch_vt) +
                            (long long)li * m * (lay.w0 + lay.w1) +
                            (tile.group == 0 ? 0 : (long long)m * lay.w0) + tile.gcol0;
  __nv_bfloat16 *pool = (ch == 0 ? a.pool.k : a.pool.v) +
                        (long long)layer * a.pool.num_slots * row + tile.col0;
  const int ntt = (T + kTileRows - 1) / kTileRows;
  const uint32_t s0 = ptx::smem_addr(smem);
  const uint32_t b_op = s0 + P.b_op, c_op = s0 + P.canon, pg_op = s0 + P.pages;
  const uint32_t s_tmem = s0 + P.misc, s_bar = s0 + P.misc + 8;  // two MMA barriers
  const DivMod cpr(ncore);
  const DivMod psd(lay.page_size);
  // fixed 16-byte chunk per thread for row copies: rows my_r0, my_r0 + rs, ...
  const int rs = (kThr % ncore == 0) ? kThr / ncore : 0;
  int my_r0 = 0, my_ck = 0;
  if (rs) cpr.split(tid, &my_r0, &my_ck);
  const int r = ((warp & 3) << 5) + (tid & 31);  // epilogue row (TMEM lane)
  const int half = warp >> 2;
  __nv_bfloat16 **rowptr = reinterpret_cast<__nv_bfloat16 **>(smem + P.slots);
  float *rot = reinterpret_cast<float *>(smem + P.cs);  // cos[np] | sin[np] | -sin[np]
  auto a_buf = [&](int t) { return s0 + P.a_op + (u2 ? (t & 1) * P.a_stage : 0); };

  // canonical rows and page ids of tile t into stage s
  auto issue_canon = [&](int t, int s) {
    const int t0 = t * kTileRows;
    const int rows = min(kTileRows, T - t0);
    const uint32_t dst0 = c_op + s * P.stage;
    if (rs) {
      const __nv_bfloat16 *src = canon + (long long)(t0 + my_r0) * row + 8 * my_ck;
      uint32_t dst = dst0 + my_r0 * P.pitch + my_ck * 16;
      for (int rr = my_r0; rr < rows; rr += rs, src += (long long)rs * row, dst += rs * P.pitch)
        ptx::cp_async16(dst, src, 16u);
    } else {
      for (int e = tid; e < rows * ncore; e += kThr) {
        int rr, ck;
        cpr.split(e, &rr, &ck);
        ptx::cp_async16(dst0 + rr * P.pitch + ck * 16, canon + (long long)(t0 + rr) * row + 8 * ck,
                        16u);
      }
    }
    int p_first, off0;
    psd.split(it.start_tok + t0, &p_first, &off0);
    int npages, dummy;
    psd.split(off0 + rows - 1, &npages, &dummy);
    const int32_t *pt = a.pool.pt + (long long)it.req * a.pool.pt_stride + p_first;
    for (int e = tid; e <= npages; e += kThr)
      ptx::cp_async4(pg_op + s * P.pages_stage + 4 * e, pt + e);
  };
  // U rows of tile t as the A operand (rows past the chunk and ranks past m are zero)
  auto issue_u = [&](int t) {
    const int t0 = t * kTileRows;
    const int rows = min(kTileRows, T - t0);
    const __nv_bfloat16 *Ut = U + (long long)t0 * m;
    const uint32_t a_op = a_buf(t);
    if (tensor) {
      const DivMod kcs(Kp >> 3);
      for (int e = tid; e < kTileRows * kcs.n; e += kThr) {
        int rr, kc;
        kcs.split(e, &rr, &kc);
        const bool ok = rr < rows && kc * 8 < m;
        ptx::cp_async16(a_op + ((kc * 16 + (rr >> 3)) << 7) + ((rr & 7) << 4),
                        ok ? (const void *)(Ut + (long long)rr * m + kc * 8) : (const void *)Ut,
                        ok ? 16u : 0u);
      }
    } else {
      for (int e = tid; e < kTileRows * Kp; e += kThr) {
        const int rr = e / Kp, k = e - rr * Kp;
        const uint32_t v = (rr < rows && k < m) ? ldg_u16(Ut + (long long)rr * m + k) : 0u;
        sts_u16(a_op + (((k >> 3) * 16 + (rr >> 3)) << 7) + ((rr & 7) << 4) + ((k & 7) << 1), v);
      }
    }
  };
  uint32_t tmem = 0;
  const uint32_t idesc = ptx::idesc_bf16_f32(kTileRows, ncols) | (1u << 16);  // B MN-major
  // MMA of tile t into accumulator t & 1 (one thread); arrives on barrier t & 1
  auto issue_mma = [&](int t) {
    ptx::tc_fence_after();
    // In the no-swizzle MN-major layout the descriptor's leading offset is the K-direction
    // step between core matrices and the stride offset the MN-direction step (K-major A:
    // LBO along K, SBO along M).
    const uint32_t lbo_a = 16 * 128, sbo_a = 128;
    const uint32_t k_step_b = ncore * 128, mn_step_b = 128;
    const uint32_t a_op = a_buf(t);
    const uint32_t d = tmem + (t & 1) * P.acc_cols;
    for (int ks = 0; ks < Kp / 16; ++ks) {
      const uint64_t ad = ptx::smem_desc(a_op + ks * 2 * lbo_a, lbo_a, sbo_a);
      const uint64_t bd = ptx::smem_desc(b_op + ks * 2 * k_step_b, k_step_b, mn_step_b);
      ptx::mma_bf16(d, ad, bd, idesc, ks > 0 ? 1u : 0u);
    }
    ptx::mma_commit(s_bar + 8 * (t & 1));
  };

  if (warp == 0) {
    ptx::tmem_alloc(s_tmem, P.tmem_cols);
    ptx::tmem_relinquish();
  }
  if (tid == 0) {
    ptx::mbar_init(s_bar, 1);
    ptx::mbar_init(s_bar + 8, 1);
    ptx::fence_mbar_init();
  }
  if (tile.band)  // cos/sin of each pair's offset, once per CTA
    for (int i = tid; i < lay.npairs; i += kThr) {
      const float2 c = rope_phase(a.freq.q[i], pair_delta(it, lay, i));
      rot[i] = c.x;
      rot[lay.npairs + i] = c.y;
      rot[2 * lay.npairs + i] = -c.y;
    }
  // B operand, once per CTA: a 16-byte run of a V_m^T row is one core-matrix row
  for (int e = tid; e < Kp * ncore; e += kThr) {
    int k, j;
    cpr.split(e, &k, &j);
    const bool ok = k < m;
    ptx::cp_async16(b_op + (((k >> 3) * ncore + j) << 7) + ((k & 7) << 4),
                    ok ? (const void *)(vt + (long long)k * wg + 8 * j) : (const void *)vt,
                    ok ? 16u : 0u);
  }
  issue_canon(0, 0);
  issue_u(0);
  ptx::cp_async_commit();
  if (ntt > 1) {
    issue_canon(1, 1);
    if (u2) issue_u(1);
  }
  ptx::cp_async_commit();
  ptx::cp_async_wait_group1();  // tile 0 (and B)
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();  // TMEM address, barriers, tile 0 visible
  ptx::tc_fence_after();
  tmem = *reinterpret_cast<volatile uint32_t *>(smem + P.misc);
  bool timed_out = false;
  if (tensor && tid == 0) issue_mma(0);
  const uint32_t trow0 = tmem + ((uint32_t)((warp & 3) * 32) << 16);

  for (int t = 0; t < ntt; ++t) {
    const int s = t & 1;
    const int t0 = t * kTileRows;
    const int rows = min(kTileRows, T - t0);
    const bool use_tc = tensor && !timed_out;
    if (use_tc) {  // warp 0 waits for MMA(t); the other warps sleep at the barrier
      if (warp == 0) {
        const bool ok = ptx::mbar_wait(s_bar + 8 * s, (t >> 1) & 1, kWaitLimitNs);
        if (tid == 0) *reinterpret_cast<volatile int *>(smem + P.misc + 4) = ok ? 0 : 1;
      }
      ptx::tc_fence_before();
      __syncthreads();
      ptx::tc_fence_after();
      if (*reinterpret_cast<volatile int *>(smem + P.misc + 4)) {
        timed_out = true;
        if (tid == 0) atomicOr(a.status, KAMERA_DEVICE_TIMEOUT);
      }
      // one U buffer: MMA(t) has read it, so U of tile t+1 may land now
      if (!u2 && t + 1 < ntt) issue_u(t + 1);
      ptx::cp_async_commit();
    }
    const bool write = !(tensor && timed_out);
    const uint32_t c_row = c_op + s * P.stage + r * P.pitch;
    if (write && (r < rows || use_tc)) {
      bool done = false;
      if constexpr (kFixed) {
        if (use_tc) {
          epilogue_fixed<NC, BAND>(c_row, half, trow0 + s * P.acc_cols, rot, lay.npairs);
          done = true;
        }
      }
      if (!done) {
        PatchSrc ps;
        ps.tensor = use_tc;
        ps.trow = trow0 + s * P.acc_cols;
        ps.a_base = a_buf(t);
        ps.b_base = b_op;
        ps.r = r;
        ps.m = m;
        ps.ncore = ncore;
        epilogue_row(c_row, tile, lay.style, half, ps, rot, lay.npairs);
      }
    }
    if (half == 0 && r < rows) {  // the row's owner finds its slot
      int pg, in_page;
      psd.split(it.start_tok + t0 + r, &pg, &in_page);
      int p_first, off0;
      psd.split(it.start_tok + t0, &p_first, &off0);
      int page;
      asm volatile("ld.shared.b32 %0, [%1];"
                   : "=r"(page)
                   : "r"(pg_op + s * P.pages_stage + 4 * (pg - p_first)));
      __nv_bfloat16 *dst = nullptr;
      if (page >= 0 && (long long)(page + 1) * lay.page_size <= a.pool.num_slots)
        dst = pool + ((long long)page * lay.page_size + in_page) * row;
      else
        atomicOr(a.status, KAMERA_DEVICE_SLOT_OOB);
      rowptr[r] = dst;
    }
    // the CUDA-core path with one U buffer reads U(t) in the epilogue: U(t+1) after it
    if (!u2 && !tensor && t + 1 < ntt) {
      __syncthreads();
      issue_u(t + 1);
      ptx::cp_async_commit();
    }
    ptx::cp_async_wait_all();  // tile t+1's rows, pages and U
    ptx::fence_proxy_async_smem();
    if (use_tc) ptx::tc_fence_before();
    __syncthreads();  // rows of tile t complete, tile t+1 staged
    if (tensor && !timed_out && t + 1 < ntt && tid == 0) issue_mma(t + 1);
    if (write) {  // fixed 16-byte chunk per thread, coalesced along each row
      const uint32_t st0 = c_op + s * P.stage;
      if (rs) {
        uint32_t src = st0 + my_r0 * P.pitch + my_ck * 16;
        for (int rr = my_r0; rr < rows; rr += rs, src += rs * P.pitch) {
          __nv_bfloat16 *dst = rowptr[rr];
          if (dst) stg16(dst + 8 * my_ck, lds16(src));
        }
      } else {
        for (int e = tid; e < rows * ncore; e += kThr) {
          int rr, ck;
          cpr.split(e, &rr, &ck);
          __nv_bfloat16 *dst = rowptr[rr];
          if (dst) stg16(dst + 8 * ck, lds16(st0 + rr * P.pitch + ck * 16));
        }
      }
    }
    __syncthreads();  // stage s is free
    if (t + 2 < ntt) {
      issue_canon(t + 2, s);
      if (u2) issue_u(t + 2);
    }
    ptx::cp_async_commit();
  }
  ptx::cp_async_wait_all();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tmem, P.tmem_cols);
}

__global__ void __launch_bounds__(kThr, 2) reuse_kernel(const __grid_constant__ ReuseArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const DevLayout &lay = a.lay;
  // this CTA's task: column tile, item, (layer, channel)
  const int ct = blockIdx.x, item = blockIdx.y;
  const int layer = lay.L - 1 - (int)blockIdx.z / lay.n_ch;  // top layers first (see the tile kernel)
  const int ch = (int)blockIdx.z % lay.n_ch;
  const kamera_item it = a.items ? a.items[item] : a.single;
  if (a.items && item_check(it, lay, a.pool, a.max_tokens, a.max_m) != 0) {
    if (ct == 0 && blockIdx.z == 0 && threadIdx.x == 0) atomicOr(a.status, KAMERA_DEVICE_BAD_ITEM);
    return;
  }
  if (it.num_tokens <= 0 || !layer_patched(it, layer)) return;  // the copy kernel's work
  const bool rotate = ch == 0 && item_rotates(it, lay);
  const Tile tile = tile_of(lay, ch, ct, rotate);
  // compile-time shapes of the reference layouts; everything else takes the general path
  // (NeoX tiles of 64 or 128 columns with the tensor engine run in reuse_fast_kernel)
  if (tile.ncols == 128 && tile.band == 0) {
    run_task<128, 0>(a, smem, it, layer, ch, tile);
  } else if (tile.ncols == 64 && tile.band == 0) {
    run_task<64, 0>(a, smem, it, layer, ch, tile);
  } else {
    run_task<0, 0>(a, smem, it, layer, ch, tile);
  }
}

int align128(int x) { return (x + 127) & ~127; }

}  // namespace

SmemPlan reuse_smem_plan(const DevLayout &l, int max_m) {
  SmemPlan p{};
  int widest = l.tw;
  if (l.kind == KAMERA_MLA && l.rope_d > widest) widest = l.rope_d;
  const int kp = max_m > 0 ? ((max_m + 15) & ~15) : 0;
  p.pitch = widest * 2 + 16;  // one 16-byte pad per row: rows land on different bank groups
  p.stage = align128(kTileRows * p.pitch);
  p.a_stage = align128(kTileRows * kp * 2);
  p.b_stage = align128(widest * kp * 2);
  p.cs_stage = align128(l.npairs * 12);
  p.pages_stage = align128((kTileRows / l.page_size + 2) * 4);
  const int fixed = p.b_stage + 2 * p.stage + p.cs_stage + 2 * p.pages_stage +
                    align128(kTileRows * 8) + 128;
  // two U buffers when two CTAs still fit on an SM (227 KB of shared memory, 1 KB reserved
  // per CTA), else one
  p.u_bufs = (fixed + 2 * p.a_stage + 1024) * 2 <= 227 * 1024 ? 2 : 1;
  // B first: every descriptor offset stays inside the allocation
  int off = 0;
  p.b_op = off;
  off += p.b_stage;
  p.a_op = off;
  off += p.u_bufs * p.a_stage;
  p.canon = off;
  off += 2 * p.stage;
  p.cs = off;
  off += p.cs_stage;
  p.pages = off;
  off += 2 * p.pages_stage;
  p.desc = off;   // unused
  p.slots = off;  // row pointers of the tile being stored
  off = align128(off + kTileRows * 8);
  p.misc = off;   // TMEM address, timeout flag, two MMA barriers
  off = align128(off + 32);
  p.total = off;
  int cols = 0;
  if (kp > 0) {
    cols = 32;
    while (cols < widest) cols <<= 1;
  }
  p.acc_cols = cols;       // one accumulator
  p.tmem_cols = 2 * cols;  // two: MMA of the next tile runs under this tile's stores
  return p;
}

cudaError_t launch_reuse(const ReuseArgs &a, int n_items, cudaStream_t s) {
  static int configured_smem[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured_smem[dev] == 0) {
    e = cudaFuncSetAttribute(reuse_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured_smem[dev] = 1;
  }
  if (a.smem.total > configured_smem[dev] && a.smem.total > 48 * 1024) {
    e = cudaFuncSetAttribute(reuse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             a.smem.total);
    if (e != cudaSuccess) return e;
    configured_smem[dev] = a.smem.total;
  }
  dim3 grid(a.lay.ntile, n_items, a.lay.L * a.lay.n_ch);
  reuse_kernel<<<grid, kThr, a.smem.total, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kamera
