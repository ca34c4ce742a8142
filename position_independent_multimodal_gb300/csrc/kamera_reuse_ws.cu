// Persistent, warp-specialised kernel of the Kamera reuse operator for the common layouts
// (Eq. 1, KV^(B|A) = R(delta) KV(B|empty) + U_m V_m^T, written into the paged KV pool; App. A
// "apply_reuse": a per-layer RoPE rotation plus a rank-m GEMM into the paged KV cache).
//
// Layouts served: NeoX-half pairing with column tiles of 64 or 128 columns holding whole
// heads (GQA/MHA head_dim 64 or 128; MLA c_KV tiles of 64 or 128 and a k_pe band of 64 or
// 128), tensor engine. Every layer of every item runs here, patched or not; other layouts use
// reuse_copy_kernel and reuse_kernel.
//
// One CTA per SM walks a static list of tasks (item, layer, channel, column tile; task k goes
// to CTA k mod grid) and the 128-token tiles of each. Its warps have fixed roles and hand
// tiles on through mbarriers (every wait bounded):
//   warps 0-2  producers: cp.async of the canonical tile into a stage, in the tensor core's
//              128-byte swizzled K-major layout (rows of 128 bytes per 64-column atom, 16-byte
//              chunk j of row r at chunk j ^ (r % 8)); the U rows (A operand) and, when the
//              task changes, the V_m^T columns (B operand) as no-swizzle core matrices; the
//              tile's page ids; the cos/sin table of the item's offset.
//   warp 3     MMA issuer: tcgen05.mma into one of two TMEM accumulators [128 lanes = tokens]
//              [tile columns]: the patch U V_m^T and, on tiles that do not rotate, the canonical
//              tile itself as X I per 16-column block (I a 16 x 16 identity; exact products,
//              float32 accumulation).
//   warps 4-11 epilogue and stores: one token row per thread and half of its columns (TMEM
//              lane quarter warp % 4): round the accumulator (folded tiles), or rotate the
//              staged row on the CUDA cores and add the patch, one rounding to bf16, written
//              back in place; the row's owner looks up its page slot; then the 256 threads store
//              the tile, 4 rows x 128 bytes per warp instruction, and release the stage.
// Unpatched tiles skip the MMA: a tile that neither rotates nor takes a patch goes from global
// memory to shared memory and back untouched (a byte copy).
#include "kamera_dev.cuh"
#include "kamera_ptx.cuh"
#include "kamera_smem.cuh"

namespace kamera {

namespace {

constexpr int kWarpsW = 12;
constexpr int kThrW = kWarpsW * 32;
constexpr int kProdWarps = 3;     // warps 0..2
constexpr int kProdThreads = kProdWarps * 32;
constexpr int kMmaWarp = 3;
constexpr int kEpiWarp0 = 4;      // warps 4..11
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr uint64_t kWaitNsW = 2000000000ull;  // 2 s: far beyond any tile
constexpr int kAtomW = kTileRows * 128;       // one 64-column swizzle atom of a 128-row tile
constexpr int kMaxStagesW = 6;

enum TileKind { kCopy = 0, kRot = 1, kFold = 2, kPatchRot = 3, kFmaPatch = 4 };

// Shared address of 16-byte chunk j (8 columns) of row r in a swizzled tile at x.
__device__ __forceinline__ uint32_t swz(uint32_t x, int r, int j) {
  return x + (j >> 3) * kAtomW + r * 128 + (((j & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ int lds_i32(uint32_t a) {
  int v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts_i32(uint32_t a, int v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Everything a role needs about task k; every role decodes the same list the same way.
struct Task {
  kamera_item it;
  Tile tile;
  int item, layer, ch, kind, ntt, row;
  bool ok, report;
};

__device__ __forceinline__ Task decode(const ReuseArgs &a, int k) {
  Task d;
  const DevLayout &lay = a.lay;
  const int per_z = a.n_items * lay.ntile;
  const int z = k / per_z;
  const int rem = k - z * per_z;
  const int item = rem / lay.ntile;
  const int ct = rem - item * lay.ntile;
  d.item = item;
  d.layer = z / lay.n_ch;
  d.ch = z - d.layer * lay.n_ch;
  d.it = a.items ? a.items[item] : a.single;
  d.ok = !(a.items && item_check(d.it, lay, a.pool, a.max_tokens, a.max_m) != 0);
  d.report = !d.ok && ct == 0 && z == 0;
  d.ntt = d.ok ? (d.it.num_tokens + kTileRows - 1) / kTileRows : 0;
  const bool rotate = d.ch == 0 && d.it.delta != 0;
  d.tile = tile_of(lay, d.ch, ct, rotate);
  d.row = d.ch == 0 ? lay.row_k : lay.row_v;
  const bool patched = layer_patched(d.it, d.layer);
  const bool tensor = (d.it.patch_m & 7) == 0 && aligned16(d.it.patch_u);
  d.kind = !patched ? (d.tile.band ? kRot : kCopy)
                    : (!tensor ? kFmaPatch : (d.tile.band ? kPatchRot : kFold));
  return d;
}

// Calls f(task, k, t, n) for every tile of this CTA in order (n counts them); stops when f
// returns false. `reporter` flags rejected batch items in the status word.
template <typename F>
__device__ __forceinline__ void for_each_tile(const ReuseArgs &a, int ntasks, bool reporter,
                                              F &&f) {
  int n = 0;
  for (int k = blockIdx.x; k < ntasks; k += gridDim.x) {
    const Task d = decode(a, k);
    if (d.report && reporter) atomicOr(a.status, KAMERA_DEVICE_BAD_ITEM);
    for (int t = 0; t < d.ntt; ++t, ++n)
      if (!f(d, k, t, n)) return;
  }
}

// Bounded wait; on a timeout the CTA's abort flag and the status bit are set.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, uint32_t abort_flag,
                                         unsigned *status) {
  if (lds_i32(abort_flag)) return false;
  if (ptx::mbar_wait(bar, parity, kWaitNsW)) return true;
  sts_i32(abort_flag, 1);
  atomicOr(status, KAMERA_DEVICE_TIMEOUT);
  return false;
}

// ---- epilogues (thread = token row r, half h of its columns) ----

// Canonical folded into the accumulator: round and write back. Half h owns the contiguous
// chunks [h*NC/16, (h+1)*NC/16).
template <int NC>
__device__ __forceinline__ void epi_fold(uint32_t x, int r, int half, uint32_t trow) {
  constexpr int CH = NC / 16;
#pragma unroll
  for (int q0 = 0; q0 < CH; q0 += 4) {
    const int j0 = half * CH + q0;
    uint32_t acc[32];
    ptx::tmem_ld32(trow + j0 * 8, acc);
    ptx::tmem_ld_wait(acc);
    ptx::tmem_ld_wait(acc + 8);
    ptx::tmem_ld_wait(acc + 16);
    ptx::tmem_ld_wait(acc + 24);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        o[e] = pack2_rn(__uint_as_float(acc[8 * q + 2 * e]),
                        __uint_as_float(acc[8 * q + 2 * e + 1]));
      sts16(swz(x, r, j0 + q), make_uint4(o[0], o[1], o[2], o[3]));
    }
  }
}

// NeoX bands of width BAND: groups of 8 pairs (columns ca..ca+7, partners cb = ca + BAND/2),
// a' = b*(-sin) + (a*cos + p_a), b' = a*sin + (b*cos + p_b) in packed f32x2 arithmetic, one
// rounding; p from TMEM when PATCH. Half h owns pairs [h*NC/4, (h+1)*NC/4). `rot` holds
// cos[np] | sin[np] | -sin[np].
template <int NC, int BAND, bool PATCH>
__device__ __forceinline__ void epi_rot(uint32_t x, int r, int half, uint32_t trow,
                                        const float *rot, int np) {
  constexpr int HB = BAND / 2, PAIRS_HALF = NC / 4, GROUPS = PAIRS_HALF / 8;
#pragma unroll
  for (int q = 0; q < GROUPS; ++q) {
    const int p = half * PAIRS_HALF + q * 8;
    const int head = p / HB, i = p % HB;
    const int ca = head * BAND + i, cb = ca + HB;
    uint32_t acc[16];
    if (PATCH) {
      ptx::tmem_ld8(trow + ca, acc);
      ptx::tmem_ld8(trow + cb, acc + 8);
    }
    const uint32_t aa = swz(x, r, ca >> 3), ab = swz(x, r, cb >> 3);
    const uint4 ra = lds16(aa), rb = lds16(ab);
    const float4 *cv = reinterpret_cast<const float4 *>(rot + i);
    const float4 *sv = reinterpret_cast<const float4 *>(rot + np + i);
    const float4 *nv = reinterpret_cast<const float4 *>(rot + 2 * np + i);
    if (PATCH) {
      ptx::tmem_ld_wait(acc);
      ptx::tmem_ld_wait(acc + 8);
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e] = 0u;
    }
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
// staged operands, added to the staged row (rotated first when band > 0), one rounding. The
// chunks each half owns are those of epi_fold / epi_rot.
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

template <int NC, int BAND>
__device__ __forceinline__ void epilogue_tile(int kind, uint32_t x, int r, int half,
                                              uint32_t trow, const float *rot, int np) {
  if constexpr (BAND == 0) {
    if (kind == kFold) epi_fold<NC>(x, r, half, trow);
  } else {
    if (kind == kPatchRot)
      epi_rot<NC, BAND, true>(x, r, half, trow, rot, np);
    else if (kind == kRot)
      epi_rot<NC, BAND, false>(x, r, half, trow, rot, np);
  }
}

__device__ __forceinline__ void bar_epilogue() {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}

__global__ void __launch_bounds__(kThrW, 1) reuse_ws_kernel(const __grid_constant__ ReuseArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t s0 = (raw + 1023u) & ~1023u;  // the swizzle atoms need 1024-byte alignment
  unsigned char *sp = smem_raw + (s0 - raw);
  const SmemPlan &P = a.smem;
  const DevLayout &lay = a.lay;
  const int NS = P.nstages;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntasks = lay.ntile * a.n_items * lay.L * lay.n_ch;
  // barriers: full[NS] (kProdThreads cp.async completions + one release by producer lane 0),
  // empty[NS] (the 8 epilogue warps, after storing), acc_full[2] (MMA commit or arrive),
  // acc_empty[2] (the 8 epilogue warps)
  const uint32_t s_tmem = s0 + P.misc, s_abort = s0 + P.misc + 4;
  const uint32_t b_full = s0 + P.misc + 16, b_empty = b_full + 8 * NS;
  const uint32_t b_accf = b_empty + 8 * NS, b_acce = b_accf + 16;
  const uint32_t b_tag = b_acce + 16;  // producer-private tags: V_m^T task [3][NS], cos/sin item [NS]
  const uint32_t x_op = s0 + P.canon, u_op = s0 + P.a_op, v_op = s0 + P.b_op;
  const uint32_t id_op = s0 + P.desc, pg_op = s0 + P.pages;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(b_full + 8 * s, kProdThreads + 1);
      ptx::mbar_init(b_empty + 8 * s, kEpiWarps);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(b_accf + 8 * i, 1);
      ptx::mbar_init(b_acce + 8 * i, kEpiWarps);
    }
    ptx::fence_mbar_init();
    sts_i32(s_abort, 0);
  }
  if (tid < (kProdWarps + 1) * kMaxStagesW) sts_i32(b_tag + 4 * tid, -1);
  // operand buffers start at zero: padding ranks and rows stay finite for the tensor core
  for (int e = tid * 16; e < NS * (P.a_stage + P.b_stage); e += kThrW * 16)
    sts16(u_op + e, make_uint4(0u, 0u, 0u, 0u));
  if (tid < 256) {  // 16 x 16 identity, MN-major core matrices (element (n, k))
    const int n = tid & 15, k = tid >> 4;
    sts_u16(id_op + ((k >> 3) * 2 + (n >> 3)) * 128 + (k & 7) * 16 + (n & 7) * 2,
            n == k ? 0x3F80u : 0u);
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(s_tmem, P.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sp + P.misc);
  const int ps = lay.page_size;
  const DivMod psd(ps);

  if (warp < kProdWarps) {
    // ---------------- producers ----------------
    const int pt = tid;  // 0 .. kProdThreads-1
    const int lc = pt & 7, lr = pt >> 3;  // chunk of an atom row; first row of this thread
    constexpr int kRowStep = kProdThreads / 8;
    for_each_tile(a, ntasks, pt == 0, [&](const Task &d, int k, int t, int n) -> bool {
      const int s = n % NS;
      if (n >= NS && !wait_bar(b_empty + 8 * s, ((n / NS) & 1) ^ 1, s_abort, a.status))
        return false;
      const kamera_item &it = d.it;
      const int T = it.num_tokens, t0 = t * kTileRows, rows = min(kTileRows, T - t0);
      const int row = d.row, nc = d.tile.ncols;
      // canonical rows: 12 rows x 128 bytes per pass of the producer threads
      const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(d.ch == 0 ? it.canon_k
                                                                             : it.canon_v) +
                                 ((long long)d.layer * T + t0 + lr) * row + d.tile.col0 + 8 * lc;
      const long long step = (long long)kRowStep * row;
      const uint32_t xs = x_op + s * P.stage;
      for (int rr = lr; rr < rows; rr += kRowStep, src += step) {
        const uint32_t dst = xs + rr * 128 + ((lc ^ (rr & 7)) << 4);
        ptx::cp_async16(dst, src, 16u);
        if (nc == 128) ptx::cp_async16(dst + kAtomW, src + 64, 16u);
      }
      // page ids of the tile's tokens
      {
        int p_first, off0, npages, dummy;
        psd.split(it.start_tok + t0, &p_first, &off0);
        psd.split(off0 + rows - 1, &npages, &dummy);
        const int32_t *ptab = a.pool.pt + (long long)it.req * a.pool.pt_stride + p_first;
        for (int e = pt; e <= npages; e += kProdThreads)
          ptx::cp_async4(pg_op + s * P.pages_stage + 4 * e, ptab + e);
      }
      if (d.kind >= kFold) {  // patched: U rows and (when the task changed) V_m^T
        const int m = it.patch_m, m8 = m >> 3;
        const int li = d.layer - it.patch_l0;
        const __nv_bfloat16 *Ut = static_cast<const __nv_bfloat16 *>(it.patch_u) +
                                  (long long)(li * 2 + d.tile.group) * T * m + (long long)t0 * m;
        const uint32_t us = u_op + s * P.a_stage;
        if (d.kind != kFmaPatch) {
          const DivMod md(m8);
          for (int e = pt; e < rows * m8; e += kProdThreads) {
            int rr, kc;
            md.split(e, &rr, &kc);
            ptx::cp_async16(us + ((kc * 16 + (rr >> 3)) << 7) + ((rr & 7) << 4),
                            Ut + (long long)rr * m + kc * 8, 16u);
          }
        } else if (warp == 0) {  // element copies; published by lane 0's release below
          const int kp = (m + 15) & ~15;
          for (int e = lane; e < kTileRows * kp; e += 32) {
            const int rr = e / kp, kk = e - rr * kp;
            const uint32_t v = (rr < rows && kk < m) ? ldg_u16(Ut + (long long)rr * m + kk) : 0u;
            sts_u16(us + (((kk >> 3) * 16 + (rr >> 3)) << 7) + ((rr & 7) << 4) + ((kk & 7) << 1), v);
          }
        }
        const uint32_t tag = b_tag + 4 * (warp * kMaxStagesW + s);
        if (lds_i32(tag) != k) {  // this warp's share of V_m^T: MN-major core matrices
          const int wg = d.tile.group == 0 ? lay.w0 : lay.w1;
          const __nv_bfloat16 *vt = static_cast<const __nv_bfloat16 *>(it.patch_vt) +
                                    (long long)li * m * (lay.w0 + lay.w1) +
                                    (d.tile.group == 0 ? 0 : (long long)m * lay.w0) + d.tile.gcol0;
          const int ncore = nc >> 3, kpad = (m + 15) & ~15;
          const uint32_t vs = v_op + s * P.b_stage;
          for (int e = pt; e < kpad * ncore; e += kProdThreads) {
            const int kk = e / ncore, j = e - kk * ncore;
            const bool ok = kk < m;
            ptx::cp_async16(vs + ((kk >> 3) * ncore + j) * 128 + (kk & 7) * 16,
                            ok ? (const void *)(vt + (long long)kk * wg + 8 * j) : (const void *)vt,
                            ok ? 16u : 0u);
          }
          sts_i32(tag, k);  // every lane keeps the same tag (no cross-lane read)
        }
      }
      if (d.tile.band && warp == 0) {  // cos/sin of the item's offset (cached per stage)
        const uint32_t tag = b_tag + 4 * (kProdWarps * kMaxStagesW + s);
        if (lds_i32(tag) != d.item) {  // the table depends on the item's offset only
          float *rot = reinterpret_cast<float *>(sp + P.cs + s * P.cs_stage);
          for (int i = lane; i < lay.npairs; i += 32) {
            const float2 c = rope_phase(a.freq.q[i], it.delta);
            rot[i] = c.x;
            rot[lay.npairs + i] = c.y;
            rot[2 * lay.npairs + i] = -c.y;
          }
          __syncwarp();  // the table is complete before any lane moves on
          sts_i32(tag, d.item);
        }
      }
      ptx::cp_async_mbar_arrive(b_full + 8 * s);
      if (warp == 0) {
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(b_full + 8 * s);
      }
      return true;
    });
    ptx::cp_async_wait_all();
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      for_each_tile(a, ntasks, false, [&](const Task &d, int k, int t, int n) -> bool {
        const int s = n % NS, acc = n & 1;
        if (!wait_bar(b_full + 8 * s, (n / NS) & 1, s_abort, a.status)) return false;
        if (n >= 2 && !wait_bar(b_acce + 8 * acc, ((n >> 1) & 1) ^ 1, s_abort, a.status))
          return false;
        if (d.kind == kFold || d.kind == kPatchRot) {
          ptx::tc_fence_after();
          ptx::fence_proxy_async_smem();
          const int nc = d.tile.ncols, ncore = nc >> 3;
          const int kp = (d.it.patch_m + 15) & ~15;
          const uint32_t dt = tmem + acc * P.acc_cols;
          const uint32_t us = u_op + s * P.a_stage, vs = v_op + s * P.b_stage;
          // no-swizzle layouts: K-major A with the K step (2048) as leading offset and the M
          // step (128) as stride; MN-major B with the K step as leading offset, N step stride
          const uint32_t idesc = ptx::idesc_bf16_f32(kTileRows, nc) | (1u << 16);
          for (int ks = 0; ks < kp / 16; ++ks)
            ptx::mma_bf16(dt, ptx::smem_desc(us + ks * 2 * 2048, 2048, 128),
                          ptx::smem_desc(vs + ks * 2 * ncore * 128, ncore * 128, 128), idesc,
                          ks > 0 ? 1u : 0u);
          if (d.kind == kFold) {  // D[:, 16j..16j+15] += X[:, 16j..16j+15] * I
            const uint32_t idesc16 = ptx::idesc_bf16_f32(kTileRows, 16) | (1u << 16);
            const uint64_t bd = ptx::smem_desc(id_op, 256, 128);
            const uint32_t xs = x_op + s * P.stage;
            for (int j = 0; j < nc / 16; ++j)
              ptx::mma_bf16(dt + 16 * j,
                            ptx::smem_desc_sw128(xs + (j >> 2) * kAtomW + (j & 3) * 32), bd,
                            idesc16, 1u);
          }
          ptx::mma_commit(b_accf + 8 * acc);
        } else {
          ptx::mbar_arrive(b_accf + 8 * acc);
        }
        return true;
      });
    }
    __syncwarp();
  } else {
    // ---------------- epilogue and stores ----------------
    // Every epilogue warp passes the same named barrier once per tile, whatever happens, so
    // an abort can never leave one waiting.
    const int et = tid - kEpiWarp0 * 32;  // 0..255
    const int r = ((warp & 3) << 5) + lane;  // token row = TMEM lane
    const int half = (warp - kEpiWarp0) >> 2;
    const uint32_t trow0 = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int lc = et & 7, lr = et >> 3;  // stores: chunk of an atom row, row of each pass
    for_each_tile(a, ntasks, false, [&](const Task &d, int k, int t, int n) -> bool {
      const int s = n % NS, acc = n & 1;
      const bool ok = wait_bar(b_full + 8 * s, (n / NS) & 1, s_abort, a.status) &&
                      wait_bar(b_accf + 8 * acc, (n >> 1) & 1, s_abort, a.status);
      const uint32_t xs = x_op + s * P.stage;
      const int nc = d.tile.ncols, band = d.tile.band;
      const int t0 = t * kTileRows, rows = min(kTileRows, d.it.num_tokens - t0);
      unsigned long long *rowptr =
          reinterpret_cast<unsigned long long *>(sp + P.slots) + (n & 1) * kTileRows;
      if (ok) {
        ptx::tc_fence_after();
        const uint32_t trow = trow0 + acc * P.acc_cols;
        const float *rot = reinterpret_cast<const float *>(sp + P.cs + s * P.cs_stage);
        if (d.kind == kFmaPatch) {
          if (r < rows)
            epi_fma(xs, r, half, nc, band, u_op + s * P.a_stage, v_op + s * P.b_stage,
                    d.it.patch_m, rot, lay.npairs);
        } else if (d.kind != kCopy) {
          if (nc == 128) {
            if (band == 0)
              epilogue_tile<128, 0>(d.kind, xs, r, half, trow, rot, lay.npairs);
            else if (band == 128)
              epilogue_tile<128, 128>(d.kind, xs, r, half, trow, rot, lay.npairs);
            else
              epilogue_tile<128, 64>(d.kind, xs, r, half, trow, rot, lay.npairs);
          } else {
            if (band == 0)
              epilogue_tile<64, 0>(d.kind, xs, r, half, trow, rot, lay.npairs);
            else
              epilogue_tile<64, 64>(d.kind, xs, r, half, trow, rot, lay.npairs);
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(b_acce + 8 * acc);
        if (half == 0 && r < rows) {  // the row's owner finds its slot
          int pg, in_page, p_first, off0;
          psd.split(d.it.start_tok + t0 + r, &pg, &in_page);
          psd.split(d.it.start_tok + t0, &p_first, &off0);
          const int page = lds_i32(pg_op + s * P.pages_stage + 4 * (pg - p_first));
          unsigned long long dst = 0;
          if (page >= 0 && (long long)(page + 1) * ps <= a.pool.num_slots)
            dst = static_cast<unsigned long long>(__cvta_generic_to_global(
                (d.ch == 0 ? a.pool.k : a.pool.v) +
                ((long long)d.layer * a.pool.num_slots + (long long)page * ps + in_page) * d.row +
                d.tile.col0));
          else
            atomicOr(a.status, KAMERA_DEVICE_SLOT_OOB);
          rowptr[r] = dst;
        }
      }
      bar_epilogue();  // every row of the tile finished, its slot known
      if (ok) {  // 4 rows x 128 bytes per warp instruction
        const int atoms = nc >> 6;
        for (int rr = lr; rr < rows; rr += 32) {
          const unsigned long long dst = rowptr[rr];
          if (dst) {
            const uint32_t src = xs + rr * 128 + ((lc ^ (rr & 7)) << 4);
            stg16_global(reinterpret_cast<void *>(dst + 16ull * lc), lds16(src));
            if (atoms == 2)
              stg16_global(reinterpret_cast<void *>(dst + 128ull + 16ull * lc), lds16(src + kAtomW));
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(b_empty + 8 * s);
      }
      return true;
    });
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, P.tmem_cols);
}

int align128w(int x) { return (x + 127) & ~127; }

}  // namespace

bool fast_layout(const DevLayout &l) {
  if (l.style != KAMERA_ROPE_NEOX_HALF) return false;
  if (l.tw != 64 && l.tw != 128) return false;
  if (l.kind == KAMERA_GQA) return (l.hd == 64 || l.hd == 128) && l.hd <= l.tw && l.row_k % l.tw == 0;
  return l.latent % l.tw == 0 && (l.rope_d == 64 || l.rope_d == 128);
}

SmemPlan reuse_ws_plan(const DevLayout &l, int max_m) {
  SmemPlan p{};
  int widest = l.tw;
  if (l.kind == KAMERA_MLA && l.rope_d > widest) widest = l.rope_d;
  const int kp = max_m > 0 ? ((max_m + 15) & ~15) : 0;
  p.fast = 1;
  p.pitch = widest * 2;
  p.stage = kTileRows * widest * 2;  // a multiple of 1024: every swizzle atom stays aligned
  p.a_stage = align128w(kTileRows * kp * 2);
  p.b_stage = align128w(widest * kp * 2);
  p.cs_stage = align128w(l.npairs * 12);
  p.pages_stage = align128w((kTileRows / l.page_size + 2) * 4);
  const int per_stage = p.stage + p.a_stage + p.b_stage + p.cs_stage + p.pages_stage;
  const int fixed = 512 + 2048 + 512 + 1024;  // identity, row addresses, barriers and tags, alignment
  int ns = (227 * 1024 - fixed) / per_stage;
  if (ns > kMaxStagesW) ns = kMaxStagesW;
  p.nstages = ns;  // >= 2 for every rank <= 128
  int off = 0;
  p.canon = off;
  off += ns * p.stage;
  p.a_op = off;  // U stages, then V_m^T stages (zeroed together at start)
  off += ns * p.a_stage;
  p.b_op = off;
  off += ns * p.b_stage;
  p.cs = off;
  off += ns * p.cs_stage;
  p.pages = off;
  off += ns * p.pages_stage;
  p.desc = off;  // the 16 x 16 identity operand
  off += 512;
  p.slots = off;  // two buffers of the global addresses of a tile's rows
  off += 2 * kTileRows * 8;
  p.misc = off;  // TMEM address, abort flag, barriers, tags
  off += 512;
  p.total = off + 1024;
  p.acc_cols = widest;
  p.tmem_cols = 2 * widest;
  return p;
}

cudaError_t launch_reuse_ws(const ReuseArgs &a, cudaStream_t s) {
  static int configured_smem[64] = {0};
  static int sm_count[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (sm_count[dev] == 0) {
    e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  if (a.smem.total > configured_smem[dev]) {
    e = cudaFuncSetAttribute(reuse_ws_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             a.smem.total);
    if (e != cudaSuccess) return e;
    configured_smem[dev] = a.smem.total;
  }
  const long long ntasks = (long long)a.lay.ntile * a.n_items * a.lay.L * a.lay.n_ch;
  const int grid = (int)(ntasks < sm_count[dev] ? ntasks : sm_count[dev]);
  if (grid <= 0) return cudaSuccess;
  reuse_ws_kernel<<<grid, kThrW, a.smem.total, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kamera
