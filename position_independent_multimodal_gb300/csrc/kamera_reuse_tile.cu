// Patched-layer kernel of the Kamera reuse operator for the common layouts (Eq. 1,
// KV^(B|A) = R(delta) KV(B|empty) + U_m V_m^T written into the paged KV pool; App. A
// "apply_reuse": a per-layer RoPE rotation plus a rank-m GEMM into the paged KV cache).
//
// Layouts served: NeoX-half pairing with column tiles of 64 or 128 columns holding whole heads
// (GQA/MHA head_dim 64 or 128; MLA c_KV tiles of 64 or 128 and a k_pe band of 64 or 128),
// tensor engine. Unpatched layers stream through reuse_copy_kernel; other layouts use
// reuse_kernel.
//
// One CTA of 256 threads per task (item, patched layer, channel, column tile) walks the
// chunk's tokens in tiles of 128 through two shared-memory stages; two CTAs share an SM. The
// canonical rows of tile t+2 and their page ids are in flight (cp.async) while tile t is
// finished, and U of tile t+1 lands during tile t's epilogue. Canonical tiles are staged in the
// tensor core's 128-byte swizzled K-major layout (rows of 128 bytes per 64-column atom, 16-byte
// chunk j of row r at chunk j ^ (r % 8)), so copies in and out move 4 rows x 128 bytes per
// warp instruction and a thread that owns a row reads and writes its chunks without bank
// conflicts. U rows (A operand) and V_m^T columns (B operand, staged once per task) are
// no-swizzle core matrices. Per tile one thread issues tcgen05.mma of the patch U V_m^T into
// one of two TMEM accumulators [128 lanes = tokens][tile columns] (float32); the MMA of tile t+1
// runs while tile t is stored. In the epilogue each token row belongs to two threads (TMEM lane
// quarter warp % 4, half warp / 4 of the columns): the staged row, rotated on the CUDA cores
// where it turns, plus the patch in packed f32x2 arithmetic, one rounding to bf16, written back
// in place. Ranks that are not a multiple of 8 form the patch on the CUDA cores from the staged
// operands.
#include "kamera_dev.cuh"
#include "kamera_ptx.cuh"
#include "kamera_smem.cuh"

namespace kamera {

namespace {

constexpr int kThrT = 256;
constexpr uint64_t kWaitNsT = 2000000000ull;  // 2 s: far beyond one MMA
constexpr int kAtomT = kTileRows * 128;       // one 64-column swizzle atom of a 128-row tile

// Shared address of 16-byte chunk j (8 columns) of row r in a swizzled tile at x.
__device__ __forceinline__ uint32_t swz(uint32_t x, int r, int j) {
  return x + (j >> 3) * kAtomT + r * 128 + (((j & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ int lds_i32t(uint32_t a) {
  int v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts_i32t(uint32_t a, int v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Unrotated tile: the staged row plus the patch from TMEM in packed f32x2 arithmetic, one
// rounding, written back in place. Half h owns the contiguous chunks [h*NC/16, (h+1)*NC/16).
// Each element is its own sum, so a non-finite value stays in its own column.
template <int NC>
__device__ __forceinline__ void epi_add(uint32_t x, int r, int half, uint32_t trow) {
  constexpr int CH = NC / 16;
#pragma unroll 1
  for (int q0 = 0; q0 < CH; q0 += 2) {
    const int j0 = half * CH + q0;
    uint32_t acc[16];
    ptx::tmem_ld16(trow + j0 * 8, acc);
    const uint32_t a0 = swz(x, r, j0), a1 = swz(x, r, j0 + 1);
    const uint4 x0 = lds16(a0), x1 = lds16(a1);
    ptx::tmem_ld_wait(acc);
    ptx::tmem_ld_wait(acc + 8);
    const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    uint32_t o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
      o[e] = f2_to_bf2(add2(bf2_to_f2(w[e]), f2(__uint_as_float(acc[2 * e]),
                                                 __uint_as_float(acc[2 * e + 1]))));
    sts16(a0, make_uint4(o[0], o[1], o[2], o[3]));
    sts16(a1, make_uint4(o[4], o[5], o[6], o[7]));
  }
}

// NeoX bands of width BAND, patch from TMEM: groups of 8 pairs (columns ca..ca+7, partners
// cb = ca + BAND/2), a' = b*(-sin) + (a*cos + p_a), b' = a*sin + (b*cos + p_b) in packed f32x2
// arithmetic, one rounding. Half h owns pairs [h*NC/4, (h+1)*NC/4). `rot` holds
// cos[np] | sin[np] | -sin[np].
template <int NC, int BAND>
__device__ __forceinline__ void epi_rot(uint32_t x, int r, int half, uint32_t trow,
                                        const float *rot, int np) {
  constexpr int HB = BAND / 2, PAIRS_HALF = NC / 4, GROUPS = PAIRS_HALF / 8;
#pragma unroll 1
  for (int q = 0; q < GROUPS; ++q) {
    const int p = half * PAIRS_HALF + q * 8;
    const int head = p / HB, i = p % HB;
    const int ca = head * BAND + i, cb = ca + HB;
    uint32_t acc[16];
    ptx::tmem_ld8(trow + ca, acc);
    ptx::tmem_ld8(trow + cb, acc + 8);
    const uint32_t aa = swz(x, r, ca >> 3), ab = swz(x, r, cb >> 3);
    const uint4 ra = lds16(aa), rb = lds16(ab);
    const float4 *cv = reinterpret_cast<const float4 *>(rot + i);
    const float4 *sv = reinterpret_cast<const float4 *>(rot + np + i);
    const float4 *nv = reinterpret_cast<const float4 *>(rot + 2 * np + i);
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
        const f32x2 av = bf2_to_f2(wa[j]), bv = bf2_to_f2(wb[j]);
        const f32x2 pa = f2(__uint_as_float(acc[2 * j]), __uint_as_float(acc[2 * j + 1]));
        const f32x2 pb = f2(__uint_as_float(acc[8 + 2 * j]), __uint_as_float(acc[8 + 2 * j + 1]));
        oa[j] = f2_to_bf2(fma2(bv, ns, fma2(av, c, pa)));
        ob[j] = f2_to_bf2(fma2(av, sn, fma2(bv, c, pb)));
      }
    }
    sts16(aa, make_uint4(oa[0], oa[1], oa[2], oa[3]));
    sts16(ab, make_uint4(ob[0], ob[1], ob[2], ob[3]));
  }
}

// CUDA-core contraction (ranks that are not a multiple of 8): the patch of row r from the
// staged operands, added to the staged row (rotated first when band > 0), one rounding. Each
// half owns the chunks of epi_add / epi_rot.
__device__ __noinline__ void epi_fma(uint32_t x, int r, int half, int nc, int band,
                                     uint32_t a_op, uint32_t b_op, int m, const float *rot,
                                     int np) {
  const int ncore = nc >> 3;
  if (band > 0) {
    const int hb = band >> 1, pairs_half = nc >> 2;
    for (int g = 0; g < pairs_half / 8; ++g) {
      const int p = half * pairs_half + g * 8;
      const int head = p / hb, i = p % hb;
      const int ca = head * band + i, cb = ca + hb;
      float pa[8], pb[8], xa[8], xb[8];
      fma_patch8(a_op, b_op, r, ca, m, ncore, pa);
      fma_patch8(a_op, b_op, r, cb, m, ncore, pb);
      const uint32_t aa = swz(x, r, ca >> 3), ab = swz(x, r, cb >> 3);
      unpack8(lds16(aa), xa);
      unpack8(lds16(ab), xb);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        rot_pair(xa[e], xb[e], make_float2(rot[i + e], rot[np + i + e]));
        xa[e] += pa[e];
        xb[e] += pb[e];
      }
      sts16(aa, pack8_rn(xa));
      sts16(ab, pack8_rn(xb));
    }
  } else {
    const int per_half = ncore >> 1;
    for (int j = half * per_half; j < (half + 1) * per_half; ++j) {
      float p[8], xv[8];
      fma_patch8(a_op, b_op, r, 8 * j, m, ncore, p);
      const uint32_t ad = swz(x, r, j);
      unpack8(lds16(ad), xv);
#pragma unroll
      for (int e = 0; e < 8; ++e) xv[e] += p[e];
      sts16(ad, pack8_rn(xv));
    }
  }
}

// The tile is computed from item `it` and stored to its slots or, when MULTI, to the slots of
// nmem group members, whose requests and first tokens are in shared memory at P.members
// (member 0 is `it`).
template <int NC, int BAND, bool INPLACE, bool MULTI>
__device__ __forceinline__ void task_loop(const ReuseArgs &a, uint32_t s0, unsigned char *sp,
                                          const kamera_item &it, int layer, int ch,
                                          const Tile &tile, int nmem) {
  constexpr int ATOMS = NC / 64;
  constexpr int NCORE = NC / 8;
  const SmemPlan &P = a.smem;
  const DevLayout &lay = a.lay;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = it.num_tokens, m = it.patch_m, Kp = (m + 15) & ~15, m8 = m >> 3;
  const int row = ch == 0 ? lay.row_k : lay.row_v;
  const bool tensor = (m & 7) == 0 && aligned16(it.patch_u);
  const bool u2 = P.u_bufs == 2;  // U of tile t+2 staged with its rows (else one buffer)
  const int ps = lay.page_size;
  const int ntt = (T + kTileRows - 1) / kTileRows;
  const uint32_t x_op = s0 + P.canon, v_op = s0 + P.b_op;
  const uint32_t pg_op = s0 + P.pages;
  const uint32_t s_tmem = s0 + P.misc, s_bar = s0 + P.misc + 8;  // two MMA barriers
  volatile int *flag = reinterpret_cast<volatile int *>(sp + P.misc + 4);
  // MULTI: int slot [member][row] (-1 skips); else the global address of each row (0 skips)
  unsigned long long *rowptr = reinterpret_cast<unsigned long long *>(sp + P.slots);
  const uint32_t slots = s0 + P.slots;
  auto mreq = [&](int f) { return lds_i32t(s0 + P.members + 4 * f); };
  auto mstart = [&](int f) { return lds_i32t(s0 + P.members + 4 * (kShareBlock + f)); };
  float *rot = reinterpret_cast<float *>(sp + P.cs);
  const int li = layer - it.patch_l0;
  const __nv_bfloat16 *U = static_cast<const __nv_bfloat16 *>(it.patch_u) +
                           (long long)(li * 2 + tile.group) * T * m;
  const __nv_bfloat16 *canon = INPLACE ? nullptr
                                         : static_cast<const __nv_bfloat16 *>(
                                               ch == 0 ? it.canon_k : it.canon_v) +
                                               (long long)layer * T * row + tile.col0;
  const __nv_bfloat16 *pool_ch = ch == 0 ? a.pool.k : a.pool.v;
  auto u_buf = [&](int t) { return s0 + P.a_op + (u2 ? (t & 1) * P.a_stage : 0); };
  const int lc = tid & 7, lr = tid >> 3;  // copies: chunk of an atom row, row of each pass
  const uint32_t swc = (uint32_t)((lc ^ (lr & 7)) << 4);
  const DivMod md(m8 > 0 ? m8 : 1);
  const DivMod psd(ps);

  // canonical rows of tile t into stage s (4 rows x 128 bytes per warp instruction) and the
  // page ids of its tokens
  auto issue_x = [&](int t, int s) {
    const int t0 = t * kTileRows, rows = min(kTileRows, T - t0);
    const uint32_t dst = x_op + s * P.stage + lr * 128 + swc;
    if constexpr (!INPLACE) {
      const __nv_bfloat16 *src = canon + (long long)(t0 + lr) * row + 8 * lc;
      const long long step = 32ll * row;
#pragma unroll
      for (int pr = 0; pr < 4; ++pr) {
        if (lr + 32 * pr < rows) {
#pragma unroll
          for (int at = 0; at < ATOMS; ++at)
            ptx::cp_async16(dst + at * kAtomT + pr * 32 * 128, src + pr * step + at * 64, 16u);
        }
      }
    } else {  // the cached rows themselves, gathered through the page table
      const int32_t *ptab = a.pool.pt + (long long)it.req * a.pool.pt_stride;
#pragma unroll
      for (int pr = 0; pr < 4; ++pr) {
        const int rr = lr + 32 * pr;
        if (rr < rows) {
          int pg, in_page;
          psd.split(it.start_tok + t0 + rr, &pg, &in_page);
          const int page = __ldg(ptab + pg);
          if (page >= 0 && (long long)(page + 1) * ps <= a.pool.num_slots) {
            const __nv_bfloat16 *src =
                pool_ch + ((long long)layer * a.pool.num_slots + (long long)page * ps + in_page) *
                              row + tile.col0 + 8 * lc;
#pragma unroll
            for (int at = 0; at < ATOMS; ++at)
              ptx::cp_async16(dst + at * kAtomT + pr * 32 * 128, src + at * 64, 16u);
          }
        }
      }
    }
    if constexpr (MULTI) {  // page ids of each member's tokens [t0, t0 + rows)
      const int pgs = P.pg_per_member;
      for (int e = tid; e < nmem * pgs; e += kThrT) {
        const int f = e / pgs, k = e - f * pgs;
        int p_first, off0, npages, dummy;
        psd.split(mstart(f) + t0, &p_first, &off0);
        psd.split(off0 + rows - 1, &npages, &dummy);
        if (k <= npages)
          ptx::cp_async4(pg_op + s * P.pages_stage + 4 * e,
                         a.pool.pt + (long long)mreq(f) * a.pool.pt_stride + p_first + k);
      }
    } else {
      int p_first, off0, npages, dummy;
      psd.split(it.start_tok + t0, &p_first, &off0);
      psd.split(off0 + rows - 1, &npages, &dummy);
      const int32_t *ptab = a.pool.pt + (long long)it.req * a.pool.pt_stride + p_first;
      for (int e = tid; e <= npages; e += kThrT)
        ptx::cp_async4(pg_op + s * P.pages_stage + 4 * e, ptab + e);
    }
  };
  // U rows of tile t as the A operand (K-major core matrices). Rows past the chunk stay stale
  // (their accumulator rows are never stored); the rank padding was zeroed once.
  auto issue_u = [&](int t) {
    const int t0 = t * kTileRows, rows = min(kTileRows, T - t0);
    const __nv_bfloat16 *Ut = U + (long long)t0 * m;
    const uint32_t ub = u_buf(t);
    if (tensor) {
      for (int e = tid; e < rows * m8; e += kThrT) {
        int rr, kc;
        md.split(e, &rr, &kc);
        ptx::cp_async16(ub + ((kc * 16 + (rr >> 3)) << 7) + ((rr & 7) << 4),
                        Ut + (long long)rr * m + kc * 8, 16u);
      }
    } else {
      for (int e = tid; e < kTileRows * Kp; e += kThrT) {
        const int rr = e / Kp, k = e - rr * Kp;
        const uint32_t v = (rr < rows && k < m) ? ldg_u16(Ut + (long long)rr * m + k) : 0u;
        sts_u16(ub + (((k >> 3) * 16 + (rr >> 3)) << 7) + ((rr & 7) << 4) + ((k & 7) << 1), v);
      }
    }
  };
  uint32_t tmem = 0;
  // MMA of tile t into accumulator t & 1 (one thread); arrives on barrier t & 1
  auto issue_mma = [&](int t) {
    ptx::tc_fence_after();
    const uint32_t ub = u_buf(t), d = tmem + (t & 1) * P.acc_cols;
    // no-swizzle layouts: K-major A with the K step (2048) as leading offset and the M step
    // (128) as stride; MN-major B with the K step as leading offset and the N step as stride
    const uint32_t idesc = ptx::idesc_bf16_f32(kTileRows, NC) | (1u << 16);
    for (int ks = 0; ks < Kp / 16; ++ks)
      ptx::mma_bf16(d, ptx::smem_desc(ub + ks * 2 * 2048, 2048, 128),
                    ptx::smem_desc(v_op + ks * 2 * NCORE * 128, NCORE * 128, 128), idesc,
                    ks > 0 ? 1u : 0u);
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
    *flag = 0;
  }
  if (BAND > 0)  // cos/sin of each pair's offset, once per CTA
    for (int i = tid; i < lay.npairs; i += kThrT) {
      const float2 c = rope_phase(a.freq.q[i], pair_delta(it, lay, i));
      rot[i] = c.x;
      rot[lay.npairs + i] = c.y;
      rot[2 * lay.npairs + i] = -c.y;
    }
  if (tensor && (Kp >> 3) > m8)  // rank padding of the U buffers: zero (meets zero V_m^T rows)
    for (int e = tid; e < (u2 ? 2 : 1) * kTileRows; e += kThrT) {
      const int b = e >> 7, rr = e & 127;
      sts16(s0 + P.a_op + b * P.a_stage + ((m8 * 16 + (rr >> 3)) << 7) + ((rr & 7) << 4),
            make_uint4(0u, 0u, 0u, 0u));
    }
  {  // V_m^T of the tile, once: MN-major core matrices, ranks past m zero
    const int wg = tile.group == 0 ? lay.w0 : lay.w1;
    const __nv_bfloat16 *vt = static_cast<const __nv_bfloat16 *>(it.patch_vt) +
                              (long long)li * m * (lay.w0 + lay.w1) +
                              (tile.group == 0 ? 0 : (long long)m * lay.w0) + tile.gcol0;
    for (int e = tid; e < Kp * NCORE; e += kThrT) {
      const int k = e / NCORE, j = e % NCORE;
      const bool ok = k < m;
      ptx::cp_async16(v_op + ((k >> 3) * NCORE + j) * 128 + (k & 7) * 16,
                      ok ? (const void *)(vt + (long long)k * wg + 8 * j) : (const void *)vt,
                      ok ? 16u : 0u);
    }
  }
  issue_x(0, 0);
  issue_u(0);
  ptx::cp_async_commit();
  if (ntt > 1) {
    issue_x(1, 1);
    if (u2) issue_u(1);
  }
  ptx::cp_async_commit();
  ptx::cp_async_wait_group1();  // tile 0 (and V_m^T)
  if (INPLACE && a.sign < 0)  // subtraction: negate V_m^T exactly (bf16 sign bits)
    for (int e = tid; e < Kp * NCORE * 4; e += kThrT) {
      const uint32_t ad = v_op + 4 * e;
      uint32_t w;
      asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w) : "r"(ad));
      asm volatile("st.shared.b32 [%0], %1;" ::"r"(ad), "r"(w ^ 0x80008000u) : "memory");
    }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();  // TMEM address, barriers, table, tile 0 visible
  ptx::tc_fence_after();
  tmem = *reinterpret_cast<volatile uint32_t *>(sp + P.misc);
  bool timed_out = false;
  if (tensor && tid == 0) issue_mma(0);
  const int r = ((warp & 3) << 5) + lane;  // epilogue row (TMEM lane)
  const int half = warp >> 2;
  const uint32_t trow0 = tmem + ((uint32_t)((warp & 3) * 32) << 16);

  for (int t = 0; t < ntt; ++t) {
    const int s = t & 1;
    const int t0 = t * kTileRows, rows = min(kTileRows, T - t0);
    const bool use_tc = tensor && !timed_out;
    if (use_tc) {  // warp 0 waits for MMA(t); the other warps sleep at the barrier
      if (warp == 0) {
        const bool ok = ptx::mbar_wait(s_bar + 8 * s, (t >> 1) & 1, kWaitNsT);
        if (lane == 0 && !ok) *flag = 1;
      }
      ptx::tc_fence_before();
      __syncthreads();
      ptx::tc_fence_after();
      if (*flag) {
        timed_out = true;
        if (tid == 0) atomicOr(a.status, KAMERA_DEVICE_TIMEOUT);
      }
      // one U buffer: MMA(t) has read it, so U of tile t+1 may land now
      if (!u2 && t + 1 < ntt) issue_u(t + 1);
      ptx::cp_async_commit();
    }
    const bool write = !(tensor && timed_out);
    const uint32_t xs = x_op + s * P.stage;
    if (write) {
      if (use_tc) {
        if constexpr (BAND == 0)
          epi_add<NC>(xs, r, half, trow0 + s * P.acc_cols);
        else
          epi_rot<NC, BAND>(xs, r, half, trow0 + s * P.acc_cols, rot, lay.npairs);
      } else if (!tensor && r < rows) {
        epi_fma(xs, r, half, NC, BAND, u_buf(t), v_op, m, rot, lay.npairs);
      }
    }
    if constexpr (MULTI) {
      if (r < rows)  // the row's two owners find its slot in each member (alternating)
        for (int f = half; f < nmem; f += 2) {
          int pg, in_page, p_first, off0;
          const int st = mstart(f);
          psd.split(st + t0 + r, &pg, &in_page);
          psd.split(st + t0, &p_first, &off0);
          const int page = lds_i32t(pg_op + s * P.pages_stage +
                                    4 * (f * P.pg_per_member + pg - p_first));
          int slot = -1;
          if (page >= 0 && (long long)(page + 1) * ps <= a.pool.num_slots)
            slot = page * ps + in_page;
          else
            atomicOr(a.status, KAMERA_DEVICE_SLOT_OOB);
          sts_i32t(slots + 4 * (f * kTileRows + r), slot);
        }
    } else if (half == 0 && r < rows) {  // the row's owner finds its slot
      int pg, in_page, p_first, off0;
      psd.split(it.start_tok + t0 + r, &pg, &in_page);
      psd.split(it.start_tok + t0, &p_first, &off0);
      const int page = lds_i32t(pg_op + s * P.pages_stage + 4 * (pg - p_first));
      unsigned long long dst = 0;
      if (page >= 0 && (long long)(page + 1) * ps <= a.pool.num_slots)
        dst = static_cast<unsigned long long>(__cvta_generic_to_global(
            (ch == 0 ? a.pool.k : a.pool.v) +
            ((long long)layer * a.pool.num_slots + (long long)page * ps + in_page) * row +
            tile.col0));
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
    if (write && !MULTI) {  // 4 rows x 128 bytes per warp instruction
      const uint32_t src = xs + lr * 128 + swc;
#pragma unroll
      for (int pr = 0; pr < 4; ++pr) {
        const int rr = lr + 32 * pr;
        if (rr < rows) {
          const unsigned long long dst = rowptr[rr];
          if (dst) {
#pragma unroll
            for (int at = 0; at < ATOMS; ++at)
              stg16_global(reinterpret_cast<void *>(dst + 128ull * at + 16ull * lc),
                           lds16(src + at * kAtomT + pr * 32 * 128));
          }
        }
      }
    } else if (write) {  // the same, once per member
      const uint32_t src = xs + lr * 128 + swc;
      const unsigned long long out_base = static_cast<unsigned long long>(
          __cvta_generic_to_global(pool_ch + (long long)layer * a.pool.num_slots * row + tile.col0));
      for (int f = 0; f < nmem; ++f) {
#pragma unroll
        for (int pr = 0; pr < 4; ++pr) {
          const int rr = lr + 32 * pr;
          if (rr < rows) {
            const int slot = lds_i32t(slots + 4 * (f * kTileRows + rr));
            if (slot >= 0) {
              const unsigned long long dst = out_base + (unsigned long long)slot * (2ull * row);
#pragma unroll
              for (int at = 0; at < ATOMS; ++at)
                stg16_global(reinterpret_cast<void *>(dst + 128ull * at + 16ull * lc),
                             lds16(src + at * kAtomT + pr * 32 * 128));
            }
          }
        }
      }
    }
    __syncthreads();  // stage s is free
    if (t + 2 < ntt) {
      issue_x(t + 2, s);
      if (u2) issue_u(t + 2);
    }
    ptx::cp_async_commit();
  }
  ptx::cp_async_wait_all();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tmem, P.tmem_cols);
}

template <bool INPLACE, bool MULTI>
__device__ __forceinline__ void run_task(const ReuseArgs &a, uint32_t s0, unsigned char *sp,
                                         const kamera_item &it, int layer, int ch,
                                         const Tile &tile, int nmem) {
  if constexpr (MULTI) {
    if (tile.band == 0) {
      if (tile.ncols == 128)
        task_loop<128, 0, false, true>(a, s0, sp, it, layer, ch, tile, nmem);
      else
        task_loop<64, 0, false, true>(a, s0, sp, it, layer, ch, tile, nmem);
    } else if (tile.ncols == 128 && tile.band == 128) {
      task_loop<128, 128, false, true>(a, s0, sp, it, layer, ch, tile, nmem);
    } else if (tile.ncols == 128) {
      task_loop<128, 64, false, true>(a, s0, sp, it, layer, ch, tile, nmem);
    } else {
      task_loop<64, 64, false, true>(a, s0, sp, it, layer, ch, tile, nmem);
    }
  } else if (INPLACE || tile.band == 0) {
    if (tile.ncols == 128)
      task_loop<128, 0, INPLACE, false>(a, s0, sp, it, layer, ch, tile, 1);
    else
      task_loop<64, 0, INPLACE, false>(a, s0, sp, it, layer, ch, tile, 1);
  } else if constexpr (!INPLACE) {
    if (tile.ncols == 128 && tile.band == 128)
      task_loop<128, 128, false, false>(a, s0, sp, it, layer, ch, tile, 1);
    else if (tile.ncols == 128)
      task_loop<128, 64, false, false>(a, s0, sp, it, layer, ch, tile, 1);
    else
      task_loop<64, 64, false, false>(a, s0, sp, it, layer, ch, tile, 1);
  }
}

__global__ void __launch_bounds__(kThrT, 2) reuse_tile_kernel(const __grid_constant__ ReuseArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t s0 = (raw + 1023u) & ~1023u;  // the swizzle atoms need 1024-byte alignment
  unsigned char *sp = smem_raw + (s0 - raw);
  const DevLayout &lay = a.lay;
  const int ct = blockIdx.x, item = blockIdx.y;
  // top layers first: the reference models patch the upper layers, so the CTAs of unpatched
  // layers (which return at once) come last, into the slots the tail leaves idle, instead of
  // filling the machine before any work starts (9 us of the reorder step's 162)
  const int layer = lay.L - 1 - (int)blockIdx.z / lay.n_ch;
  const int ch = (int)blockIdx.z % lay.n_ch;
  // canonical pointers of the block's items for the group search, loaded with the item
  kamera_item cand;
  const bool has_cand = share_candidate(a.items, a.n_items, item, a.smem.run > 1, &cand);
  const kamera_item it = a.items ? a.items[item] : a.single;
  // rejected items are reported by the copy kernel; unpatched layers are its work too
  if (a.items && item_check(it, lay, a.pool, a.max_tokens, a.max_m) != 0) return;
  if (it.num_tokens <= 0 || !layer_patched(it, layer)) return;
  const bool rotate = ch == 0 && item_rotates(it, lay);
  const Tile tile = tile_of(lay, ch, ct, rotate);
  // the tile holds rope columns (all of GQA channel 0, MLA's k_pe tile): group members need
  // the same offsets as well as the same canonical, length, factors and patched layers
  const bool has_rope = tile_of(lay, ch, ct, true).band > 0;
  const void *src = ch == 0 ? it.canon_k : it.canon_v;
  int nmem = 1;
  if (a.items && a.smem.run > 1) {
    // every warp finds the run (the same answer from the same items), so that no barrier is
    // needed unless the tile has several members; warp 0 records them
    nmem = share_run(item, it, src, ch, has_cand, cand, a.smem.run,
                     reinterpret_cast<int *>(sp + a.smem.members), threadIdx.x < 32,
                     [&](const kamera_item &o) {
                       return o.num_tokens == it.num_tokens && o.patch_u == it.patch_u &&
                              o.patch_vt == it.patch_vt && o.patch_m == it.patch_m &&
                              o.patch_l0 == it.patch_l0 && o.patch_l1 == it.patch_l1 &&
                              (!has_rope || same_offsets(o, it, lay)) &&
                              item_check(o, lay, a.pool, a.max_tokens, a.max_m) == 0;
                     });
    if (nmem == 0) return;       // another CTA writes this tile
    if (nmem > 1) __syncthreads();  // the members' requests and first tokens are visible
  }
  // the single-member branch first: the member loops placed ahead of it slowed it by 5 %
  if (nmem == 1)
    run_task<false, false>(a, s0, sp, it, layer, ch, tile, 1);
  else
    run_task<false, true>(a, s0, sp, it, layer, ch, tile, nmem);
}

// The patch re-added in place on cached rows: every tile unrotated, rows gathered from and
// written back to the pool (no groups: each item's rows are its own).
__global__ void __launch_bounds__(kThrT, 2) patch_inplace_kernel(const __grid_constant__ ReuseArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t s0 = (raw + 1023u) & ~1023u;
  unsigned char *sp = smem_raw + (s0 - raw);
  const DevLayout &lay = a.lay;
  const int ct = blockIdx.x, item = blockIdx.y;
  const int layer = lay.L - 1 - (int)blockIdx.z / lay.n_ch;  // top layers first, as above
  const int ch = (int)blockIdx.z % lay.n_ch;
  const kamera_item it = a.items ? a.items[item] : a.single;
  if (a.items && inplace_item_check(it, lay, a.pool, a.max_tokens, a.max_m) != 0) {
    if (ct == 0 && blockIdx.z == 0 && threadIdx.x == 0) atomicOr(a.status, KAMERA_DEVICE_BAD_ITEM);
    return;
  }
  if (it.num_tokens <= 0 || !layer_patched(it, layer)) return;
  const Tile tile = tile_of(lay, ch, ct, false);
  run_task<true, false>(a, s0, sp, it, layer, ch, tile, 1);
}

int align128t(int x) { return (x + 127) & ~127; }

}  // namespace

bool fast_layout(const DevLayout &l) {
  if (l.style != KAMERA_ROPE_NEOX_HALF) return false;
  if (l.tw != 64 && l.tw != 128) return false;
  if (l.kind == KAMERA_GQA) return (l.hd == 64 || l.hd == 128) && l.hd <= l.tw && l.row_k % l.tw == 0;
  return l.latent % l.tw == 0 && (l.rope_d == 64 || l.rope_d == 128);
}

// The in-place patch add never rotates, so any pairing and head width will do as long as
// every column tile is 64 or 128 columns wide.
bool inplace_layout(const DevLayout &l) {
  if (l.tw != 64 && l.tw != 128) return false;
  if (l.kind == KAMERA_GQA) return l.row_k % l.tw == 0;
  return l.latent % l.tw == 0 && (l.rope_d == 64 || l.rope_d == 128);
}

namespace {

// Offsets for runs of up to `run` group members per CTA with `u_bufs` U buffers.
SmemPlan tile_plan_with(const DevLayout &l, int max_m, int run, int u_bufs) {
  SmemPlan p{};
  int widest = l.tw;
  if (l.kind == KAMERA_MLA && l.rope_d > widest) widest = l.rope_d;
  const int kp = max_m > 0 ? ((max_m + 15) & ~15) : 16;
  p.fast = 1;
  p.run = run;
  p.u_bufs = u_bufs;
  p.pitch = widest * 2;
  p.stage = kTileRows * widest * 2;  // a multiple of 1024: the swizzle atoms stay aligned
  p.a_stage = align128t(kTileRows * kp * 2);
  p.b_stage = align128t(widest * kp * 2);
  p.cs_stage = align128t(l.npairs * 12);
  p.pg_per_member = kTileRows / l.page_size + 2;
  p.pages_stage = align128t(run * p.pg_per_member * 4);
  int off = 0;
  p.canon = off;  // two stages of swizzled tiles, first so they stay 1024-aligned
  off += 2 * p.stage;
  p.b_op = off;
  off += p.b_stage;
  p.a_op = off;
  off += p.u_bufs * p.a_stage;
  p.cs = off;
  off += p.cs_stage;
  p.pages = off;
  off += 2 * p.pages_stage;
  p.slots = off;  // slot of each row of the tile being stored, per member
  off += align128t(run * kTileRows * 4 > kTileRows * 8 ? run * kTileRows * 4 : kTileRows * 8);
  p.members = off;  // members' requests and first tokens
  off += 2 * kShareBlock * 4;
  p.misc = off;   // TMEM address, timeout flag, two MMA barriers, member count
  off += 128;
  p.total = off + 1024;  // slack to align the base to 1024 bytes
  int cols = 32;
  while (cols < widest) cols <<= 1;
  p.acc_cols = cols;
  p.tmem_cols = 2 * cols;
  return p;
}

// CTAs of a plan per SM (227 KB of shared memory, 1 KB reserved per CTA; at most 2).
int tile_ctas(const SmemPlan &p) {
  const int n = (227 * 1024) / (p.total + 1024);
  return n < 2 ? n : 2;
}

}  // namespace

// Two U buffers when two CTAs still fit on an SM, else one. Runs of group members grow (up to
// max_run) while the plan keeps its U buffers and CTAs per SM.
SmemPlan reuse_tile_plan(const DevLayout &l, int max_m, int max_run) {
  SmemPlan base = tile_plan_with(l, max_m, 1, 2);
  if (tile_ctas(base) < 2) base = tile_plan_with(l, max_m, 1, 1);
  SmemPlan best = base;
  for (int r = 2; r <= max_run && r <= kShareBlock; ++r) {
    const SmemPlan p = tile_plan_with(l, max_m, r, base.u_bufs);
    if (tile_ctas(p) < tile_ctas(base)) break;
    best = p;
  }
  return best;
}

cudaError_t launch_reuse_tile(const ReuseArgs &a, int n_items, cudaStream_t s) {
  static int configured_smem[2][64] = {{0}};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int which = a.inplace ? 1 : 0;
  void (*kernel)(const ReuseArgs) = which ? patch_inplace_kernel : reuse_tile_kernel;
  if (a.smem.total > configured_smem[which][dev] && a.smem.total > 48 * 1024) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, a.smem.total);
    if (e != cudaSuccess) return e;
    configured_smem[which][dev] = a.smem.total;
  }
  dim3 grid(a.lay.ntile, n_items, a.lay.L * a.lay.n_ch);
  kernel<<<grid, kThrT, a.smem.total, s>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------
// Persistent path of the patched layers (kamera_batch_reuse with a batch workspace; GQA/MHA
// layouts, whose column tiles all have one width and one group rule per channel).
//
// The grid kernel above pays per task a prologue (group search, TMEM and barriers, phase
// table, V_m^T, the first two tiles' loads and their latency) and ends in a tail as long as a
// task; in a batch of shared chunks most of its CTAs only search their group and exit. Here a
// planning kernel (one CTA) forms the groups once and lists the task rows: (top-first patched
// layer, channel, the first item of a run), each covering every column tile of its rows, as
// self-contained 128-byte records. The persistent CTAs come in Q sets of `ntile`, one CTA per
// column tile; a set's CTAs walk the same row tiles side by side, so the column pieces of
// each pool row are written together, as in the grid kernel.
// - When every task row has the same number of token tiles, set q owns whole rows q, q + Q,
//   q + 2Q, ... (about five sixths of the rows): the sets work through neighbouring rows at
//   the same time, so the runs of one chunk, which are neighbouring rows, read its canonical
//   rows once from DRAM. The tiles of the rows left over are handed out one at a time from a
//   counter per column tile, so CTAs that ran slower take fewer of them.
// - Otherwise each set owns one contiguous range of row tiles of equal weight (a token tile
//   of a run of r members weighing 5 + r) and nothing is handed out.
// Each CTA walks its tiles with the grid kernel's two-stage pipeline, carried across task
// boundaries: the next task's record, first tiles and V_m^T (two buffers, by task parity) are
// loaded while the previous task's last tiles are finished, and TMEM and the barriers are set
// up once. Each tile's bytes are those of the grid kernel.
// ---------------------------------------------------------------------------------------

namespace {

constexpr int kRunCapP = 4;           // most group members of one task
constexpr int kRecSlots = 32;         // task records held in shared memory
constexpr int kRecFetch = 16;         // task records fetched at a time
constexpr int kMaxPersistCtas = 1024;
constexpr int kPlanThreads = 1024;
constexpr int kMaxPlanItems = 512;
constexpr int kMaxPlanRows = 8192;    // task rows of one batch

// A task row in the workspace and in shared memory (128 bytes): the run's first item, the
// row's layer and channel, its members' requests and first tokens.
struct TaskRec {
  kamera_item it;
  int code;        // layer << 16 | channel << 8 (the CTA adds its column tile)
  int nmem;        // members of the run
  int ntt;         // token tiles
  int pad;
  int req[kRunCapP], start[kRunCapP];
};
static_assert(sizeof(kamera_item) == 80, "kamera_item layout");
static_assert(sizeof(TaskRec) == 128, "task record layout");

// Plan header, the first 256 bytes of the workspace.
struct PlanHead {
  int rows;      // task rows
  int tiles;     // tiles of all tasks (rows' token tiles x column tiles)
  int weight;    // total weight of the rows' token tiles
  int s1;        // token-tile positions [0, s1) go to the sets
  int n_dyn;     // positions [s1, s1 + n_dyn) are handed out one at a time
  int ntt;       // token tiles of every row (0: rows differ)
  int stride;    // when ntt > 0, set q owns rows q, q + Q, ..., `stride` of them (otherwise set
                 // q owns the range of row tiles starts[q] .. starts[q + 1])
};

// Byte offsets of the batch workspace for n items.
struct WsLayout {
  size_t counters;  // int [kMaxPersistCtas]: handed-out positions per column tile
  size_t starts;    // int2 [kMaxPersistCtas + 1]: (row, tile) where each set's range begins
  size_t rows;      // TaskRec [min(n * L * 2, kMaxPlanRows)]
  size_t total;
};
__host__ __device__ inline WsLayout ws_layout(const DevLayout &l, long long n) {
  WsLayout w;
  w.counters = 256;
  w.starts = w.counters + 4 * (size_t)kMaxPersistCtas;
  size_t off = w.starts + 8 * (size_t)(kMaxPersistCtas + 1);
  off = (off + 255) & ~(size_t)255;
  w.rows = off;
  long long rows = n * l.L * 2;
  if (rows > kMaxPlanRows) rows = kMaxPlanRows;
  off += (size_t)rows * sizeof(TaskRec);
  w.total = (off + 255) & ~(size_t)255;
  return w;
}

// Whether item o joins item me's group on channel ch (channel 0 turns: the same offsets as
// well): the grid kernel's group rule for GQA column tiles.
__device__ __forceinline__ bool same_group(const kamera_item &me, const kamera_item &o, int ch,
                                           const DevLayout &lay) {
  return (ch == 0 ? o.canon_k == me.canon_k : o.canon_v == me.canon_v) &&
         o.num_tokens == me.num_tokens && o.patch_u == me.patch_u &&
         o.patch_vt == me.patch_vt && o.patch_m == me.patch_m && o.patch_l0 == me.patch_l0 &&
         o.patch_l1 == me.patch_l1 && (ch != 0 || same_offsets(o, me, lay));
}

__host__ __device__ __forceinline__ int tile_weight(int nmem) { return 5 + nmem; }

// Candidate rows of a batch of n items (every layer, both channels), at most kMaxPlanRows.
__host__ __device__ inline int plan_rows(const DevLayout &l, int n) {
  const long long r = (long long)n * l.L * 2;
  return r < kMaxPlanRows ? (int)r : kMaxPlanRows;
}

// Shared memory of the planning kernel: the items, their lengths and layers, run sizes and
// members, then per task row its weight prefix and (token tiles << 8 | members), and the scan.
size_t plan_smem_bytes(const DevLayout &l, int n) {
  return 96 * (size_t)n + (((size_t)n * 2 + 15) & ~(size_t)15) + 64 * (size_t)n +
         8 * (size_t)(plan_rows(l, n) + 1) + 6 * 32 * 4;
}

// One CTA of kPlanThreads: the groups, the task rows, the range of each of Q sets of CTAs and
// the handed-out tail, into the workspace a.plan_ws. Rows past kMaxPlanRows are not planned
// (the host sizes batches below it).
__global__ void __launch_bounds__(kPlanThreads) reuse_plan_kernel(const __grid_constant__ ReuseArgs a,
                                                                  int Q) {
  extern __shared__ __align__(16) unsigned char psm[];
  const DevLayout &lay = a.lay;
  const int n = a.n_items, tid = threadIdx.x, run = a.smem.run;
  const int warp = tid >> 5, lane = tid & 31;
  unsigned char *ws = static_cast<unsigned char *>(a.plan_ws);
  const WsLayout W = ws_layout(lay, n);
  PlanHead *head = reinterpret_cast<PlanHead *>(ws);
  int *counters = reinterpret_cast<int *>(ws + W.counters);
  int2 *starts = reinterpret_cast<int2 *>(ws + W.starts);
  TaskRec *rows = reinterpret_cast<TaskRec *>(ws + W.rows);
  const int RC = plan_rows(lay, n);
  kamera_item *items = reinterpret_cast<kamera_item *>(psm);  // the batch, staged once
  int4 *info = reinterpret_cast<int4 *>(psm + 80 * n);  // (tokens, or -1 when skipped; m, l0, l1)
  signed char *nm = reinterpret_cast<signed char *>(psm + 96 * n);  // run size per (item, ch)
  int2 *members = reinterpret_cast<int2 *>(psm + 96 * n + ((2 * n + 15) & ~15));  // [2n][4]
  int *wpre = reinterpret_cast<int *>(members + 8 * n);  // weight prefix of the task rows
  int *rinfo = wpre + RC + 1;                            // token tiles << 8 | members
  int *scan = rinfo + RC;  // [3][32], then min and max token tiles
  {  // 16-byte words (the item array is 16-byte aligned and 80 bytes an item)
    const uint4 *src = reinterpret_cast<const uint4 *>(a.items);
    uint4 *dst = reinterpret_cast<uint4 *>(items);
    for (int q = tid; q < 5 * n; q += kPlanThreads) dst[q] = src[q];
  }
  for (int c = tid; c < lay.ntile; c += kPlanThreads) counters[c] = 0;
  if (tid == 0) {
    scan[96] = 0x7fffffff;
    scan[97] = 0;
  }
  __syncthreads();
  for (int i = tid; i < n; i += kPlanThreads) {
    const kamera_item &it = items[i];
    const bool ok = item_check(it, lay, a.pool, a.max_tokens, a.max_m) == 0 &&
                    it.num_tokens > 0 && it.patch_m > 0 && it.patch_l1 > it.patch_l0;
    info[i] = make_int4(ok ? it.num_tokens : -1, it.patch_m, it.patch_l0, it.patch_l1);
  }
  __syncthreads();
  // runs, one warp per (item, channel): the members of the item's group in its aligned block,
  // in item order, taken `run` at a time; the first item of each run leads it
  for (int j = warp; j < 2 * n; j += kPlanThreads / 32) {
    const int i = j >> 1, ch = j & 1;
    int nmem = 0;
    if (info[i].x > 0) {
      const kamera_item &me = items[i];
      const int b0 = i & ~(kShareBlock - 1), o = b0 + lane;
      const bool mem = o == i || (run > 1 && o < n && info[o].x > 0 &&
                                  same_group(me, items[o], ch, lay));
      const unsigned mask = __ballot_sync(0xffffffffu, mem);
      const int f_self = __popc(mask & ((1u << (i - b0)) - 1u));
      if (f_self % run == 0) {
        nmem = min(run, __popc(mask) - f_self);
        const int f = __popc(mask & ((1u << lane) - 1u)) - f_self;
        if (mem && f >= 0 && f < nmem)
          members[j * kRunCapP + f] = make_int2(items[o].req, items[o].start_tok);
      }
    }
    if (lane == 0) nm[j] = static_cast<signed char>(nmem);
  }
  __syncthreads();
  // task rows: candidates (top-first layer, channel, item), each thread a contiguous share
  const int R = lay.L * 2 * n;
  const int per = (R + kPlanThreads - 1) / kPlanThreads;
  const int r0 = min(R, tid * per), r1 = min(R, r0 + per);
  auto task_row = [&](int rr, int *i, int *layer, int *ch) {
    const int z = rr / n;
    *i = rr - z * n;
    *layer = lay.L - 1 - (z >> 1);
    *ch = z & 1;
    const int4 in = info[*i];
    return in.x > 0 && *layer >= in.z && *layer < in.w && nm[(*i << 1) | *ch] > 0;
  };
  int cnt = 0, wsum = 0, tsum = 0, tmin = 0x7fffffff, tmax = 0;
  for (int rr = r0; rr < r1; ++rr) {
    int i, layer, ch;
    if (task_row(rr, &i, &layer, &ch)) {
      const int ntt = (info[i].x + kTileRows - 1) / kTileRows;
      ++cnt;
      tsum += ntt;
      wsum += ntt * tile_weight(nm[(i << 1) | ch]);
      tmin = min(tmin, ntt);
      tmax = max(tmax, ntt);
    }
  }
  if (cnt > 0) {
    atomicMin(&scan[96], tmin);
    atomicMax(&scan[97], tmax);
  }
  int v0 = cnt, v1 = wsum, v2 = tsum;  // inclusive scans, warp then block
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int x0 = __shfl_up_sync(0xffffffffu, v0, d), x1 = __shfl_up_sync(0xffffffffu, v1, d),
              x2 = __shfl_up_sync(0xffffffffu, v2, d);
    if (lane >= d) {
      v0 += x0;
      v1 += x1;
      v2 += x2;
    }
  }
  if (lane == 31) {
    scan[warp] = v0;
    scan[32 + warp] = v1;
    scan[64 + warp] = v2;
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int c = 0; c < 3; ++c) {
      int x = scan[32 * c + lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int px = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += px;
      }
      scan[32 * c + lane] = x;
    }
  }
  __syncthreads();
  const int NR = min(scan[31], RC), WT = scan[63], NT = scan[95];
  int k = (warp > 0 ? scan[warp - 1] : 0) + v0 - cnt;
  int wp = (warp > 0 ? scan[32 + warp - 1] : 0) + v1 - wsum;
  for (int rr = r0; rr < r1 && k < NR; ++rr) {
    int i, layer, ch;
    if (task_row(rr, &i, &layer, &ch)) {
      const int ntt = (info[i].x + kTileRows - 1) / kTileRows, j = (i << 1) | ch;
      TaskRec rec;
      rec.it = items[i];
      rec.code = (layer << 16) | (ch << 8);
      rec.nmem = nm[j];
      rec.ntt = ntt;
      rec.pad = 0;
#pragma unroll
      for (int f = 0; f < kRunCapP; ++f) {
        const int2 mm = f < rec.nmem ? members[j * kRunCapP + f] : make_int2(0, 0);
        rec.req[f] = mm.x;
        rec.start[f] = mm.y;
      }
      rows[k] = rec;
      wpre[k] = wp;
      rinfo[k] = (ntt << 8) | rec.nmem;
      wp += ntt * tile_weight(nm[j]);
      ++k;
    }
  }
  if (tid == 0) wpre[NR] = WT;
  __syncthreads();
  // When every row has the same token tiles, set q owns whole rows q, q + Q, q + 2Q, ... (the
  // sets work through neighbouring rows at the same time, so the runs of one chunk, which are
  // neighbouring rows, read its canonical rows from L2 after the first), about five sixths of
  // all rows, and the tiles of the rows left over are handed out one at a time, in order (a
  // position names its row and tile by division). Otherwise each set owns one contiguous range
  // of row tiles of equal weight and nothing is handed out.
  const int uni = (NR > 0 && scan[96] == scan[97]) ? scan[97] : 0;
  const int stride = uni > 0 ? (int)((long long)NR * 5 / (6ll * Q)) : 0;
  const int s1 = uni > 0 ? Q * stride * uni : NT;
  const int n_dyn = NT - s1;
  const int w1 = uni > 0 ? wpre[s1 / uni] + (s1 % uni) * (s1 / uni < NR
                                                                ? tile_weight(rinfo[s1 / uni] & 0xff)
                                                                : 0)
                         : WT;
  const int2 s1pos = uni > 0 ? make_int2(s1 / uni, s1 % uni) : make_int2(NR, 0);
  // set q begins at the first row tile whose weight prefix is at least floor(q * w1 / Q)
  for (int q = tid; q <= Q; q += kPlanThreads) {
    const int target = (int)((long long)q * w1 / Q);
    int lo = 0, hi = NR;  // the first row r with wpre[r + 1] > target
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (wpre[mid + 1] > target)
        hi = mid;
      else
        lo = mid + 1;
    }
    int2 st = s1pos;
    if (lo < NR && q < Q) {
      const int ntt = rinfo[lo] >> 8, w = tile_weight(rinfo[lo] & 0xff);
      const int d = target - wpre[lo], t = d <= 0 ? 0 : (d + w - 1) / w;
      st = t < ntt ? make_int2(lo, t) : make_int2(lo + 1, 0);
      if (st.x > s1pos.x || (st.x == s1pos.x && st.y > s1pos.y)) st = s1pos;
    }
    starts[q] = st;
  }
  if (tid == 0) {
    head->rows = NR;
    head->tiles = NT * lay.ntile;
    head->weight = WT;
    head->s1 = s1;
    head->n_dyn = n_dyn;
    head->ntt = uni;
    head->stride = stride;
  }
}

// What the loops need of a task record at column tile ct.
struct TaskV {
  int layer, ch, nmem, T, m, row, li, tensor;
  Tile tile;
};
__device__ __forceinline__ TaskV task_v(const TaskRec &r, const DevLayout &lay, int engine,
                                        int ct) {
  TaskV v;
  v.layer = r.code >> 16;
  v.ch = (r.code >> 8) & 0xff;
  v.nmem = r.nmem;
  v.T = r.it.num_tokens;
  v.m = r.it.patch_m;
  v.row = v.ch == 0 ? lay.row_k : lay.row_v;
  v.li = v.layer - r.it.patch_l0;
  v.tile = tile_of(lay, v.ch, ct, v.ch == 0 && item_rotates(r.it, lay));
  v.tensor = engine == kEngineTensor && (v.m & 7) == 0 && aligned16(r.it.patch_u);
  return v;
}

__global__ void __launch_bounds__(kThrT, 2) reuse_persist_kernel(const __grid_constant__ ReuseArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t s0 = (raw + 1023u) & ~1023u;  // the swizzle atoms need 1024-byte alignment
  unsigned char *sp = smem_raw + (s0 - raw);
  const SmemPlan &P = a.smem;
  const DevLayout &lay = a.lay;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char *ws = static_cast<unsigned char *>(a.plan_ws);
  const WsLayout W = ws_layout(lay, a.n_items);
  const uint32_t s_tmem = s0 + P.misc, s_bar = s0 + P.misc + 8;  // two MMA barriers
  volatile int *flag = reinterpret_cast<volatile int *>(sp + P.misc + 4);
  if (warp == 0) {
    ptx::tmem_alloc(s_tmem, P.tmem_cols);
    ptx::tmem_relinquish();
  }
  if (tid == 0) {
    ptx::mbar_init(s_bar, 1);
    ptx::mbar_init(s_bar + 8, 1);
    ptx::fence_mbar_init();
    *flag = 0;
  }
  const PlanHead head = *reinterpret_cast<const PlanHead *>(ws);
  int *counter = reinterpret_cast<int *>(ws + W.counters);
  const int2 *starts = reinterpret_cast<const int2 *>(ws + W.starts);
  const TaskRec *grow = reinterpret_cast<const TaskRec *>(ws + W.rows);
  // this CTA: column tile c of set q; its own range runs from token tile b.y of task row b.x
  // to token tile e.y of row e.x (exclusive), then it takes tail positions of column c
  const int nt = lay.ntile, q = blockIdx.x / nt, c = blockIdx.x - q * nt;
  const int Q = gridDim.x / nt;
  const int2 b = starts[q], e = starts[q + 1];
  const bool own = head.ntt > 0 ? head.stride > 0 : !(b.x == e.x && b.y == e.y);
  // nothing to do: free TMEM (the barrier orders the allocation's write of its address)
  auto leave = [&]() {
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 0) ptx::tmem_dealloc(*reinterpret_cast<volatile uint32_t *>(sp + P.misc),
                                     P.tmem_cols);
  };
  if (!own && head.n_dyn == 0) {
    leave();
    return;
  }
  // tasks of the own rows (every stride-th row) or of the own range
  const int n_own = !own ? 0 : head.ntt > 0 ? head.stride : e.x - b.x + (e.y > 0 ? 1 : 0);
  auto own_row = [&](int j) { return head.ntt > 0 ? q + j * Q : b.x + j; };
  TaskRec *rec = reinterpret_cast<TaskRec *>(sp + P.recs);
  // local task j: record slot j % kRecSlots; its row and token tiles [t_lo, t_hi)
  int *l_row = reinterpret_cast<int *>(sp + P.misc + 128);
  int *l_lo = l_row + kRecSlots, *l_hi = l_lo + kRecSlots;
  volatile int *s_nlocal = reinterpret_cast<volatile int *>(sp + P.misc + 32);
  volatile int *s_final = reinterpret_cast<volatile int *>(sp + P.misc + 36);
  // copies of task rows into record slots: 8 threads per record (16-byte words)
  auto copy_rec = [&](int j, int row, int part) {
    ptx::cp_async16(s0 + P.recs + (j % kRecSlots) * 128 + 16 * part,
                    reinterpret_cast<const unsigned char *>(grow + row) + 16 * part, 16u);
  };
  // own tasks [j0, j1) (own rows or own range): records and tile ranges, then wait (every
  // thread calls)
  auto fetch_own = [&](int j0, int j1) {
    for (int x = tid; x < 8 * (j1 - j0); x += kThrT)
      copy_rec(j0 + (x >> 3), own_row(j0 + (x >> 3)), x & 7);
    ptx::cp_async_commit();
    ptx::cp_async_wait_all();
    __syncthreads();
    for (int j = j0 + tid; j < j1; j += kThrT) {
      const int row = own_row(j);
      const bool ranged = head.ntt == 0;
      l_row[j % kRecSlots] = row;
      l_lo[j % kRecSlots] = ranged && j == 0 ? b.y : 0;
      l_hi[j % kRecSlots] = ranged && row == e.x ? e.y : rec[j % kRecSlots].ntt;
    }
    __syncthreads();
  };
  // tail positions of column c (thread 0): `res` is the position reserved by the last
  // increment; taking it appends a one-tile task (its record copied by thread 0) or ends the
  // list
  int res = 0;
  auto take = [&](int n_local) -> bool {  // thread 0; returns false when the tail is used up
    const int pos = res;
    if (pos >= head.n_dyn) return false;
    const int p = head.s1 + pos, row = p / head.ntt, j = n_local;
    l_row[j % kRecSlots] = row;
    l_lo[j % kRecSlots] = p - row * head.ntt;
    l_hi[j % kRecSlots] = p - row * head.ntt + 1;
    for (int part = 0; part < 8; ++part) copy_rec(j, row, part);
    ptx::cp_async_commit();
    res = atomicAdd(counter + c, 1);
    return true;
  };
  if (tid == 0 && head.n_dyn > 0) res = atomicAdd(counter + c, 1);
  int loaded = min(n_own, kRecFetch);
  if (loaded > 0) fetch_own(0, loaded);
  if (tid == 0) {
    int nl = n_own, fin = head.n_dyn == 0 ? 1 : 0;
    while (!fin && nl < 3) {  // no own range (or a short one): start on the tail
      if (take(nl))
        ++nl;
      else
        fin = 1;
    }
    *s_nlocal = nl;
    *s_final = fin;
  }
  ptx::cp_async_wait_all();
  __syncthreads();
  int n_local = *s_nlocal;
  if (n_local == 0) {  // the tail was used up before this CTA started
    leave();
    return;
  }

  const uint32_t x_op = s0 + P.canon, pg_op = s0 + P.pages, slots = s0 + P.slots;
  const bool u2 = P.u_bufs == 2;
  const int ps = lay.page_size;
  const DivMod psd(ps);
  const int lc = tid & 7, lr = tid >> 3;  // copies: chunk of an atom row, row of each pass
  const uint32_t swc = (uint32_t)((lc ^ (lr & 7)) << 4);
  auto rec_of = [&](int j) -> const TaskRec & { return rec[j % kRecSlots]; };
  auto u_buf = [&](int g) { return s0 + P.a_op + (u2 ? (g & 1) * P.a_stage : 0); };
  auto vt_buf = [&](int j) { return s0 + P.b_op + (j & 1) * P.b_stage; };
  auto rot_of = [&](int j) { return reinterpret_cast<float *>(sp + P.cs + (j & 1) * P.cs_stage); };

  // canonical rows of token tile t of task j into stage s, and the page ids of its members
  auto issue_x = [&](int j, int t, int s) {
    const TaskRec &R = rec_of(j);
    const TaskV v = task_v(R, lay, a.engine, c);
    const int t0 = t * kTileRows, rows = min(kTileRows, v.T - t0);
    const int atoms = v.tile.ncols >> 6;
    const __nv_bfloat16 *src =
        static_cast<const __nv_bfloat16 *>(v.ch == 0 ? R.it.canon_k : R.it.canon_v) +
        ((long long)v.layer * v.T + t0 + lr) * v.row + v.tile.col0 + 8 * lc;
    const uint32_t dst = x_op + s * P.stage + lr * 128 + swc;
    const long long step = 32ll * v.row;
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
      if (lr + 32 * pr < rows) {
#pragma unroll
        for (int at = 0; at < 2; ++at)
          if (at < atoms)
            ptx::cp_async16(dst + at * kAtomT + pr * 32 * 128, src + pr * step + at * 64, 16u);
      }
    }
    const int pgs = P.pg_per_member;
    for (int x = tid; x < v.nmem * pgs; x += kThrT) {
      const int f = x / pgs, kk = x - f * pgs;
      int p_first, off0, npages, dummy;
      psd.split(R.start[f] + t0, &p_first, &off0);
      psd.split(off0 + rows - 1, &npages, &dummy);
      if (kk <= npages)
        ptx::cp_async4(pg_op + s * P.pages_stage + 4 * x,
                       a.pool.pt + (long long)R.req[f] * a.pool.pt_stride + p_first + kk);
    }
  };
  // U rows of token tile t of task j as the A operand in buffer ub; rank padding zeroed
  auto issue_u = [&](int j, int t, uint32_t ub) {
    const TaskRec &R = rec_of(j);
    const TaskV v = task_v(R, lay, a.engine, c);
    const int t0 = t * kTileRows, rows = min(kTileRows, v.T - t0);
    const int m = v.m, m8 = m >> 3, Kp = (m + 15) & ~15;
    const __nv_bfloat16 *Ut = static_cast<const __nv_bfloat16 *>(R.it.patch_u) +
                              ((long long)(v.li * 2 + v.tile.group) * v.T + t0) * m;
    if (v.tensor) {
      const DivMod md(m8);
      for (int x = tid; x < rows * m8; x += kThrT) {
        int rr, kc;
        md.split(x, &rr, &kc);
        ptx::cp_async16(ub + ((kc * 16 + (rr >> 3)) << 7) + ((rr & 7) << 4),
                        Ut + (long long)rr * m + kc * 8, 16u);
      }
      for (int x = tid; x < kTileRows * ((Kp >> 3) - m8); x += kThrT) {
        const int kc = m8 + (x >> 7), rr = x & 127;
        sts16(ub + ((kc * 16 + (rr >> 3)) << 7) + ((rr & 7) << 4), make_uint4(0u, 0u, 0u, 0u));
      }
    } else {
      for (int x = tid; x < kTileRows * Kp; x += kThrT) {
        const int rr = x / Kp, kk = x - rr * Kp;
        const uint32_t val = (rr < rows && kk < m) ? ldg_u16(Ut + (long long)rr * m + kk) : 0u;
        sts_u16(ub + (((kk >> 3) * 16 + (rr >> 3)) << 7) + ((rr & 7) << 4) + ((kk & 7) << 1), val);
      }
    }
  };
  // a new task: its phase table (plain stores) and V_m^T (copies) in the task-parity buffers
  auto prepare = [&](int j) {
    const TaskRec &R = rec_of(j);
    const TaskV v = task_v(R, lay, a.engine, c);
    if (v.tile.band > 0) {
      float *rot = rot_of(j);
      for (int i = tid; i < lay.npairs; i += kThrT) {
        const float2 cs = rope_phase(a.freq.q[i], pair_delta(R.it, lay, i));
        rot[i] = cs.x;
        rot[lay.npairs + i] = cs.y;
        rot[2 * lay.npairs + i] = -cs.y;
      }
    }
    const int m = v.m, Kp = (m + 15) & ~15, ncore = v.tile.ncols >> 3;
    const int wg = v.tile.group == 0 ? lay.w0 : lay.w1;
    const __nv_bfloat16 *vt = static_cast<const __nv_bfloat16 *>(R.it.patch_vt) +
                              (long long)v.li * m * (lay.w0 + lay.w1) +
                              (v.tile.group == 0 ? 0 : (long long)m * lay.w0) + v.tile.gcol0;
    const uint32_t vb = vt_buf(j);
    for (int x = tid; x < Kp * ncore; x += kThrT) {
      const int kk = x / ncore, jj = x - kk * ncore;
      const bool ok = kk < m;
      ptx::cp_async16(vb + ((kk >> 3) * ncore + jj) * 128 + (kk & 7) * 16,
                      ok ? (const void *)(vt + (long long)kk * wg + 8 * jj) : (const void *)vt,
                      ok ? 16u : 0u);
    }
  };
  uint32_t tmem = 0;
  // MMA of tile g (task j) into accumulator g & 1 (one thread); arrives on barrier g & 1
  auto issue_mma = [&](int j, int g) {
    const TaskRec &R = rec_of(j);
    const TaskV v = task_v(R, lay, a.engine, c);
    const int Kp = (v.m + 15) & ~15, ncore = v.tile.ncols >> 3;
    ptx::tc_fence_after();
    const uint32_t ub = u_buf(g), vb = vt_buf(j), d = tmem + (g & 1) * P.acc_cols;
    const uint32_t idesc = ptx::idesc_bf16_f32(kTileRows, v.tile.ncols) | (1u << 16);
    for (int ks = 0; ks < Kp / 16; ++ks)
      ptx::mma_bf16(d, ptx::smem_desc(ub + ks * 2 * 2048, 2048, 128),
                    ptx::smem_desc(vb + ks * 2 * ncore * 128, ncore * 128, 128), idesc,
                    ks > 0 ? 1u : 0u);
    ptx::mma_commit(s_bar + 8 * (g & 1));
  };
  // the tile after (j, t); true when it begins task j + 1 (whose first tile is read from the
  // task list when that task is reached)
  auto next = [&](int &j, int &t) -> bool {
    if (++t == l_hi[j % kRecSlots]) {
      ++j;
      return true;
    }
    return false;
  };

  int ck = 0, ctl = l_lo[0];  // the tile being finished (local task, token tile)
  int lk = 0, lt = ctl;       // the next tile to load
  prepare(lk);
  issue_x(lk, lt, 0);
  issue_u(lk, lt, u_buf(0));
  ptx::cp_async_commit();
  bool fresh = next(lk, lt);
  if (lk < n_local) {
    if (fresh) {
      lt = l_lo[lk % kRecSlots];
      prepare(lk);
    }
    issue_x(lk, lt, 1);
    if (u2) issue_u(lk, lt, u_buf(1));
    fresh = next(lk, lt);
  }
  ptx::cp_async_commit();
  ptx::cp_async_wait_group1();  // tile 0, its U and V_m^T
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();  // TMEM address, barriers, tables, tile 0 visible
  ptx::tc_fence_after();
  tmem = *reinterpret_cast<volatile uint32_t *>(sp + P.misc);
  bool timed_out = false;
  uint32_t ph = 0;  // parity of each MMA barrier's next phase
  if (tid == 0 && task_v(rec_of(ck), lay, a.engine, c).tensor) issue_mma(ck, 0);
  const int r = ((warp & 3) << 5) + lane;  // epilogue row (TMEM lane)
  const int half = warp >> 2;
  const uint32_t trow0 = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  const unsigned long long pool_k =
      static_cast<unsigned long long>(__cvta_generic_to_global(a.pool.k));
  const unsigned long long pool_v =
      a.pool.v ? static_cast<unsigned long long>(__cvta_generic_to_global(a.pool.v)) : 0ull;

  for (int g = 0; ck < n_local; ++g) {
    const int s = g & 1;
    const TaskRec &R = rec_of(ck);
    const TaskV v = task_v(R, lay, a.engine, c);
    const int t0 = ctl * kTileRows, rows = min(kTileRows, v.T - t0);
    int nk = ck, ntl = ctl;
    if (next(nk, ntl) && nk < n_local) ntl = l_lo[nk % kRecSlots];
    const bool has_next = nk < n_local;
    const bool use_tc = v.tensor && !timed_out;
    if (use_tc) {  // warp 0 waits for MMA(g); the other warps sleep at the barrier
      if (warp == 0) {
        const bool ok = ptx::mbar_wait(s_bar + 8 * s, (ph >> s) & 1u, kWaitNsT);
        if (lane == 0 && !ok) *flag = 1;
      }
      ph ^= 1u << s;
      ptx::tc_fence_before();
    }
    __syncthreads();
    n_local = *s_nlocal;  // the task list as thread 0 left it in the last iteration
    if (use_tc) {
      ptx::tc_fence_after();
      if (*flag) {
        timed_out = true;
        if (tid == 0) atomicOr(a.status, KAMERA_DEVICE_TIMEOUT);
      }
    }
    // one U buffer: MMA(g) has read it, so U of the next tile may land now
    if (!u2 && v.tensor && has_next) {
      issue_u(nk, ntl, u_buf(g + 1));
      ptx::cp_async_commit();
    }
    const bool write = !(v.tensor && timed_out);
    const uint32_t xs = x_op + s * P.stage;
    if (write) {
      const uint32_t trow = trow0 + s * P.acc_cols;
      const float *rot = rot_of(ck);
      if (use_tc) {
        if (v.tile.ncols == 128) {
          if (v.tile.band == 0)
            epi_add<128>(xs, r, half, trow);
          else if (v.tile.band == 128)
            epi_rot<128, 128>(xs, r, half, trow, rot, lay.npairs);
          else
            epi_rot<128, 64>(xs, r, half, trow, rot, lay.npairs);
        } else {
          if (v.tile.band == 0)
            epi_add<64>(xs, r, half, trow);
          else
            epi_rot<64, 64>(xs, r, half, trow, rot, lay.npairs);
        }
      } else if (!v.tensor && r < rows) {
        epi_fma(xs, r, half, v.tile.ncols, v.tile.band, u_buf(g), vt_buf(ck), v.m, rot,
                lay.npairs);
      }
    }
    if (r < rows)  // the row's two owners find its slot in each member (alternating)
      for (int f = half; f < v.nmem; f += 2) {
        int pg, in_page, p_first, off0;
        const int st = R.start[f];
        psd.split(st + t0 + r, &pg, &in_page);
        psd.split(st + t0, &p_first, &off0);
        const int page = lds_i32t(pg_op + s * P.pages_stage +
                                  4 * (f * P.pg_per_member + pg - p_first));
        int slot = -1;
        if (page >= 0 && (long long)(page + 1) * ps <= a.pool.num_slots)
          slot = page * ps + in_page;
        else
          atomicOr(a.status, KAMERA_DEVICE_SLOT_OOB);
        sts_i32t(slots + 4 * (f * kTileRows + r), slot);
      }
    // the CUDA-core path with one U buffer reads U(g) in the epilogue: U of the next tile after
    if (!u2 && !v.tensor && has_next) {
      __syncthreads();
      issue_u(nk, ntl, u_buf(g + 1));
      ptx::cp_async_commit();
    }
    ptx::cp_async_wait_all();  // the next tile's rows, pages, U and V_m^T; new task records
    ptx::fence_proxy_async_smem();
    if (use_tc) ptx::tc_fence_before();
    __syncthreads();  // rows of tile g complete, the next tile staged
    if (has_next && !timed_out && tid == 0 && task_v(rec_of(nk), lay, a.engine, c).tensor)
      issue_mma(nk, g + 1);
    if (write) {  // 4 rows x 128 bytes per warp instruction, once per member
      const uint32_t src = xs + lr * 128 + swc;
      const int atoms = v.tile.ncols >> 6;
      const unsigned long long out_base =
          (v.ch == 0 ? pool_k : pool_v) +
          2ull * ((unsigned long long)v.layer * (unsigned long long)a.pool.num_slots * v.row +
                  v.tile.col0);
      for (int f = 0; f < v.nmem; ++f) {
#pragma unroll
        for (int pr = 0; pr < 4; ++pr) {
          const int rr = lr + 32 * pr;
          if (rr < rows) {
            const int slot = lds_i32t(slots + 4 * (f * kTileRows + rr));
            if (slot >= 0) {
              const unsigned long long dst = out_base + (unsigned long long)slot * (2ull * v.row);
#pragma unroll
              for (int at = 0; at < 2; ++at)
                if (at < atoms)
                  stg16_global(reinterpret_cast<void *>(dst + 128ull * at + 16ull * lc),
                               lds16(src + at * kAtomT + pr * 32 * 128));
            }
          }
        }
      }
    }
    // keep two tasks past the load cursor listed: take a tail position (thread 0; the others
    // read the list after the next barrier); lk moves by at most one task an iteration, so the
    // task it loads next was listed (and its record landed) at least one iteration before
    if (tid == 0 && !*s_final && n_local - lk < 2) {
      if (take(n_local))
        *s_nlocal = n_local + 1;
      else
        *s_final = 1;
    }
    // The tile after the next one goes into stage s with no barrier first: each thread loads
    // exactly the chunks of the stage that it stored from (the same row and chunk mapping),
    // after its own reads of them; the epilogue's other mapping finished before the last
    // barrier, and the page ids of stage s were read before it.
    if (lk < n_local) {
      if (fresh) {       // starts a task
        if (lk < n_own && lk >= loaded) {
          const int j1 = min(n_own, lk + kRecFetch);
          fetch_own(lk, j1);
          loaded = j1;
        }
        lt = l_lo[lk % kRecSlots];
        prepare(lk);
      }
      issue_x(lk, lt, s);
      if (u2) issue_u(lk, lt, u_buf(g));
      fresh = next(lk, lt);
    }
    ptx::cp_async_commit();
    ck = nk;
    ctl = ntl;
  }
  ptx::cp_async_wait_all();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tmem, P.tmem_cols);
}

// Offsets of the persistent kernel's shared memory: the tile kernel's stages and U buffers,
// two V_m^T buffers and two phase tables (by task parity), the task records and the task list.
SmemPlan persist_plan_with(const DevLayout &l, int max_m, int run, int u_bufs) {
  SmemPlan p{};
  int widest = l.tw;
  if (l.kind == KAMERA_MLA && l.rope_d > widest) widest = l.rope_d;
  const int kp = max_m > 0 ? ((max_m + 15) & ~15) : 16;
  p.fast = 1;
  p.run = run;
  p.u_bufs = u_bufs;
  p.pitch = widest * 2;
  p.stage = kTileRows * widest * 2;
  p.a_stage = align128t(kTileRows * kp * 2);
  p.b_stage = align128t(widest * kp * 2);
  p.cs_stage = align128t(l.npairs * 12);
  p.pg_per_member = kTileRows / l.page_size + 2;
  p.pages_stage = align128t(run * p.pg_per_member * 4);
  int off = 0;
  p.canon = off;
  off += 2 * p.stage;
  p.b_op = off;
  off += 2 * p.b_stage;
  p.a_op = off;
  off += u_bufs * p.a_stage;
  p.cs = off;
  off += 2 * p.cs_stage;
  p.pages = off;
  off += 2 * p.pages_stage;
  p.slots = off;
  off += align128t(run * kTileRows * 4);
  p.recs = off;
  off += kRecSlots * (int)sizeof(TaskRec);
  // TMEM address, timeout flag, two MMA barriers, the task count and end flag, and each local
  // task's row and token tiles (three int [kRecSlots] from +128)
  p.misc = off;
  off += 128 + 3 * 4 * kRecSlots;
  p.total = off + 1024;
  int cols = 32;
  while (cols < widest) cols <<= 1;
  p.acc_cols = cols;
  p.tmem_cols = 2 * cols;
  return p;
}

}  // namespace

size_t persist_workspace_bytes(const DevLayout &l, long long n_items) {
  return ws_layout(l, n_items < 0 ? 0 : n_items).total;
}

SmemPlan reuse_persist_plan(const DevLayout &l, int max_m, int run) {
  SmemPlan p{};
  if (!fast_layout(l) || run < 1 || run > kRunCapP) return p;
  p = persist_plan_with(l, max_m, run, 2);
  if (tile_ctas(p) < 2) p = persist_plan_with(l, max_m, run, 1);
  if (tile_ctas(p) < 2) p.fast = 0;
  return p;
}

bool persist_batch_ok(const DevLayout &l, const SmemPlan &p, int n_items, int max_tokens) {
  const long long rows = (long long)n_items * l.L * 2;
  const long long ntt = ((long long)max_tokens + kTileRows - 1) / kTileRows;
  return p.fast && l.kind == KAMERA_GQA && n_items >= 1 && n_items <= kMaxPlanItems &&
         rows <= kMaxPlanRows && rows * ntt * tile_weight(kRunCapP) < (1ll << 31) &&
         rows * ntt < (1ll << 31) / l.ntile && l.ntile <= kMaxPersistCtas &&
         plan_smem_bytes(l, n_items) <= 227 * 1024;
}

cudaError_t launch_reuse_persist(const ReuseArgs &a, cudaStream_t s, cudaEvent_t planned) {
  static int configured[2][64] = {{0}};
  static int sm_count[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!sm_count[dev]) {
    e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  const int plan_smem = (int)plan_smem_bytes(a.lay, a.n_items);
  if (plan_smem > configured[0][dev] && plan_smem > 48 * 1024) {
    e = cudaFuncSetAttribute(reuse_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             plan_smem);
    if (e != cudaSuccess) return e;
    configured[0][dev] = plan_smem;
  }
  if (a.smem.total > configured[1][dev] && a.smem.total > 48 * 1024) {
    e = cudaFuncSetAttribute(reuse_persist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             a.smem.total);
    if (e != cudaSuccess) return e;
    configured[1][dev] = a.smem.total;
  }
  // sets of ntile CTAs (one per column tile), as many as fill two CTAs per SM
  const int Q = max(1, min(kMaxPersistCtas, tile_ctas(a.smem) * sm_count[dev]) / a.lay.ntile);
  reuse_plan_kernel<<<1, kPlanThreads, plan_smem, s>>>(a, Q);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (planned) {
    e = cudaEventRecord(planned, s);
    if (e != cudaSuccess) return e;
  }
  reuse_persist_kernel<<<Q * a.lay.ntile, kThrT, a.smem.total, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kamera
