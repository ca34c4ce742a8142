// Streaming kernels of the Kamera operator (CUDA cores only).
//
//  * relocate_kernel: the survivor path, rotating the rope columns of pool rows in place
//    (§5 "Sliding-window survival"; Fig. 2 rotate_k_pe_inplace).
//  * reuse_copy_kernel: the unpatched layers of reuse items (rotate + copy to the slots).
//  * rope_phases_kernel: the (cos, sin) table of any offsets, as the other kernels compute it.
#include "kamera_dev.cuh"

namespace kamera {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void st16(void *p, const uint4 &v) {
  *reinterpret_cast<uint4 *>(p) = v;
}

constexpr int kRelocTile = 32;

// In place: 4 units (8 vectors) are loaded before any is written back, so each thread keeps
// 128 bytes in flight. kFixed: the row's rope units divide the block, so every thread keeps one
// column unit and walks rows (at most 85 registers: 3 CTAs per SM); otherwise (row, unit) pairs are
// dealt out in turn.
template <bool kFixed>
__global__ void __launch_bounds__(kThreads, kFixed ? 3 : 1) relocate_kernel(const __grid_constant__ RelocArgs a) {
  __shared__ float2 cs[kMaxPairs];
  __shared__ long long slots[kRelocTile];
  const DevLayout &lay = a.lay;
  const int layer = blockIdx.y;
  const int t0 = blockIdx.x * kRelocTile;
  const int rows = min(kRelocTile, a.T - t0);
  const int tid = threadIdx.x;
  for (int i = tid; i < lay.npairs; i += kThreads) cs[i] = rope_phase(a.freq.q[i], a.delta);
  for (int r = tid; r < rows; r += kThreads)
    slots[r] = slot_of(a.pool, lay.page_size, a.req, (long long)a.start_tok + t0 + r, a.status);
  __syncthreads();
  // rope units of the K row: every unit for GQA, the k_pe band's units for MLA
  const int u_first = lay.kind == KAMERA_GQA ? 0 : (lay.latent >> 4);
  const int n_units = lay.kind == KAMERA_GQA ? (lay.row_k >> 4) : (lay.rope_d >> 4);
  __nv_bfloat16 *pool = a.pool.k + (long long)layer * a.pool.num_slots * lay.row_k;
  constexpr int B = 4;
  if constexpr (kFixed) {
    // the units divide the block: every thread keeps one column unit and walks rows, B rows
    // loaded before any is written back
    const int rstep = kThreads / n_units;
    const ColUnit cu = col_unit(lay, 0, u_first + tid % n_units, true);
    for (int rb = tid / n_units; rb < rows; rb += rstep * B) {
      uint4 ra[B], rb_[B];
      __nv_bfloat16 *p[B];
#pragma unroll
      for (int k = 0; k < B; ++k) {
        const int r = rb + k * rstep;
        p[k] = nullptr;
        if (r < rows && slots[r] >= 0) {
          p[k] = pool + slots[r] * lay.row_k;
          ra[k] = *reinterpret_cast<const uint4 *>(p[k] + cu.ca);
          rb_[k] = *reinterpret_cast<const uint4 *>(p[k] + cu.cb);
        }
      }
#pragma unroll
      for (int k = 0; k < B; ++k) {
        if (!p[k]) continue;
        float xa[8], xb[8];
        unpack8(ra[k], xa);
        unpack8(rb_[k], xb);
        rotate_unit(cu, cs, xa, xb);
        st16(p[k] + cu.ca, pack8_rn(xa));
        st16(p[k] + cu.cb, pack8_rn(xb));
      }
    }
    return;
  }
  const int n = rows * n_units;
  for (int base = tid; base < n; base += kThreads * B) {
    uint4 ra[B], rb[B];
    ColUnit cu[B];
    __nv_bfloat16 *p[B];
#pragma unroll
    for (int k = 0; k < B; ++k) {
      const int w = base + k * kThreads;
      p[k] = nullptr;
      if (w < n) {
        const int r = w / n_units;
        const long long slot = slots[r];
        if (slot >= 0) {
          cu[k] = col_unit(lay, 0, u_first + (w - r * n_units), true);
          p[k] = pool + slot * lay.row_k;
          ra[k] = *reinterpret_cast<const uint4 *>(p[k] + cu[k].ca);
          rb[k] = *reinterpret_cast<const uint4 *>(p[k] + cu[k].cb);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < B; ++k) {
      if (!p[k]) continue;
      float xa[8], xb[8];
      unpack8(ra[k], xa);
      unpack8(rb[k], xb);
      rotate_unit(cu[k], cs, xa, xb);
      st16(p[k] + cu[k].ca, pack8_rn(xa));
      st16(p[k] + cu[k].cb, pack8_rn(xb));
    }
  }
}

constexpr int kCopyRows = 128;
constexpr int kCopyRun = 8;  // most group members one CTA of the copy kernel writes

// Unpatched layers of reuse items: the canonical rows of (item, layer, channel) stream through
// registers to their slots, rope columns rotated on the way (R(delta) with no patch term),
// everything else copied byte for byte. One CTA per 128 rows of an (item, layer, channel) that
// leads a run of group members; each row, rotated once, is stored at every member's slot
// (rowoff[f][r]: element offset of row r of member f in the layer's pool, -1 skips). The grid
// runs items fastest after the row blocks, so placements that share a canonical but not a run
// read it from L2. Patched layers are left to the tensor-core kernel.
template <bool kFixedUnit, bool kMulti>
__device__ __forceinline__ void copy_rows(const DevLayout &lay, int ch, bool rotate, int rows,
                                          int row, const __nv_bfloat16 *src0,
                                          __nv_bfloat16 *pool, const long long (*rowoff)[kCopyRows],
                                          int nmem, const float2 *cs) {
  const int tid = threadIdx.x;
  const int upr = row >> 4;
  constexpr int B = 2;  // two units (four 16-byte vectors) in flight per thread
  // one unit of row r (offset off of member 0), rotated if it holds rope pairs, to its slots
  auto put = [&](const ColUnit &cu, int r, long long off, uint4 va, uint4 vb) {
    if (cu.rot != 0) {
      float xa[8], xb[8];
      unpack8(va, xa);
      unpack8(vb, xb);
      rotate_unit(cu, cs, xa, xb);
      va = pack8_rn(xa);
      vb = pack8_rn(xb);
    }
    if (off >= 0) {
      st16(pool + off + cu.ca, va);
      st16(pool + off + cu.cb, vb);
    }
    if (kMulti)
      for (int f = 1; f < nmem; ++f) {
        const long long o = rowoff[f][r];
        if (o < 0) continue;
        st16(pool + o + cu.ca, va);
        st16(pool + o + cu.cb, vb);
      }
  };
  if (kFixedUnit) {
    // upr divides the block: every thread keeps one column unit and walks rows
    const int u = tid % upr, r0 = tid / upr, rstep = kThreads / upr;
    const ColUnit cu = col_unit(lay, ch, u, rotate);
    for (int rb = r0; rb < rows; rb += rstep * B) {
      uint4 ra[B], rb_[B];
      long long off[B];
#pragma unroll
      for (int k = 0; k < B; ++k) {
        const int r = rb + k * rstep;
        off[k] = -1;
        if (r < rows) {
          off[k] = rowoff[0][r];
          const __nv_bfloat16 *src = src0 + (long long)r * row;
          ra[k] = __ldg(reinterpret_cast<const uint4 *>(src + cu.ca));
          rb_[k] = __ldg(reinterpret_cast<const uint4 *>(src + cu.cb));
        }
      }
#pragma unroll
      for (int k = 0; k < B; ++k) {
        const int r = rb + k * rstep;
        if (r < rows && (kMulti || off[k] >= 0)) put(cu, r, off[k], ra[k], rb_[k]);
      }
    }
  } else {
    const int n = rows * upr;
    for (int base = tid; base < n; base += kThreads * B) {
      uint4 ra[B], rb_[B];
      ColUnit cu[B];
      long long off[B];
      int rr[B];
#pragma unroll
      for (int k = 0; k < B; ++k) {
        const int w = base + k * kThreads;
        rr[k] = -1;
        off[k] = -1;
        if (w < n) {
          const int r = w / upr;
          rr[k] = r;
          cu[k] = col_unit(lay, ch, w - r * upr, rotate);
          off[k] = rowoff[0][r];
          const __nv_bfloat16 *src = src0 + (long long)r * row;
          ra[k] = __ldg(reinterpret_cast<const uint4 *>(src + cu[k].ca));
          rb_[k] = __ldg(reinterpret_cast<const uint4 *>(src + cu[k].cb));
        }
      }
#pragma unroll
      for (int k = 0; k < B; ++k)
        if (rr[k] >= 0 && (kMulti || off[k] >= 0)) put(cu[k], rr[k], off[k], ra[k], rb_[k]);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 4) reuse_copy_kernel(const __grid_constant__ ReuseArgs a) {
  __shared__ float2 cs[kMaxPairs];
  __shared__ long long rowoff[kCopyRun][kCopyRows];  // member f, row r (-1: skipped)
  __shared__ int members[2 * kShareBlock];  // requests, then first tokens, of the run
  __shared__ int s_nmem;
  const DevLayout &lay = a.lay;
  const int tid = threadIdx.x;
  const int item = blockIdx.y;
  const int layer = blockIdx.z / lay.n_ch;
  const int ch = blockIdx.z - layer * lay.n_ch;
  // canonical pointers of the block's items for the group search, loaded with the item
  kamera_item cand;
  const bool has_cand = share_candidate(a.items, a.n_items, item, a.run_copy > 1 && tid < 32,
                                        &cand);
  const kamera_item it = a.items ? a.items[item] : a.single;
  if (a.items && item_check(it, lay, a.pool, a.max_tokens, a.max_m) != 0) {
    if (blockIdx.x == 0 && blockIdx.z == 0 && tid == 0) atomicOr(a.status, KAMERA_DEVICE_BAD_ITEM);
    return;
  }
  const int t0 = blockIdx.x * kCopyRows;
  if (t0 >= it.num_tokens || layer_patched(it, layer)) return;
  const int rows = min(kCopyRows, it.num_tokens - t0);
  const bool rotate = ch == 0 && item_rotates(it, lay);
  const int row = ch == 0 ? lay.row_k : lay.row_v;
  const void *src = ch == 0 ? it.canon_k : it.canon_v;
  if (tid < 32) {
    // group: valid items of the block with this channel's canonical and length, unpatched on
    // this layer too, and (channel 0, which holds the rope columns) the same offsets
    int n = 1;
    if (a.items && a.run_copy > 1)
      n = share_run(item, it, src, ch, has_cand, cand, a.run_copy, members, true,
                    [&](const kamera_item &o) {
                      return o.num_tokens == it.num_tokens && !layer_patched(o, layer) &&
                             (ch != 0 || same_offsets(o, it, lay)) &&
                             item_check(o, lay, a.pool, a.max_tokens, a.max_m) == 0;
                    });
    if (tid == 0) s_nmem = n;
  } else if (rotate) {
    for (int i = tid - 32; i < lay.npairs; i += kThreads - 32)
      cs[i] = rope_phase(a.freq.q[i], pair_delta(it, lay, i));
  }
  // member 0 of every run is the CTA's own item: its slots are looked up meanwhile
  for (int r = tid; r < rows; r += kThreads) {
    const long long slot =
        slot_of(a.pool, lay.page_size, it.req, (long long)it.start_tok + t0 + r, a.status);
    rowoff[0][r] = slot < 0 ? -1 : slot * row;
  }
  __syncthreads();
  const int nmem = s_nmem;
  if (nmem == 0) return;  // another CTA writes these rows
  if (nmem > 1) {
    for (int e = kCopyRows + tid; e < nmem * kCopyRows; e += kThreads) {
      const int f = e / kCopyRows, r = e - f * kCopyRows;
      if (r < rows) {
        const long long slot = slot_of(a.pool, lay.page_size, members[f],
                                       (long long)members[kShareBlock + f] + t0 + r, a.status);
        rowoff[f][r] = slot < 0 ? -1 : slot * row;
      }
    }
    __syncthreads();
  }
  const __nv_bfloat16 *src0 = static_cast<const __nv_bfloat16 *>(src) +
                              ((long long)layer * it.num_tokens + t0) * row;
  __nv_bfloat16 *pool = (ch == 0 ? a.pool.k : a.pool.v) + (long long)layer * a.pool.num_slots * row;
  const bool fixed = kThreads % (row >> 4) == 0;
  if (nmem > 1) {
    if (fixed)
      copy_rows<true, true>(lay, ch, rotate, rows, row, src0, pool, rowoff, nmem, cs);
    else
      copy_rows<false, true>(lay, ch, rotate, rows, row, src0, pool, rowoff, nmem, cs);
  } else {
    if (fixed)
      copy_rows<true, false>(lay, ch, rotate, rows, row, src0, pool, rowoff, 1, cs);
    else
      copy_rows<false, false>(lay, ch, rotate, rows, row, src0, pool, rowoff, 1, cs);
  }
}

__global__ void rope_phases_kernel(const __grid_constant__ FreqQ64 f, int npairs,
                                   const long long *deltas, int n, float *out) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (long long)n * npairs) return;
  const int d = (int)(e / npairs), i = (int)(e - (long long)d * npairs);
  const long long delta = deltas[d];
  float2 cs = make_float2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
  if (delta <= (1ll << 62) && delta >= -(1ll << 62)) cs = rope_phase(f.q[i], delta);
  out[2 * e] = cs.x;
  out[2 * e + 1] = cs.y;
}

}  // namespace

cudaError_t launch_rope_phases(const FreqQ64 &f, int npairs, const long long *deltas, int n,
                               float *out, cudaStream_t s) {
  const long long total = (long long)n * npairs;
  const int threads = 256;
  rope_phases_kernel<<<(unsigned)((total + threads - 1) / threads), threads, 0, s>>>(
      f, npairs, deltas, n, out);
  return cudaGetLastError();
}

cudaError_t launch_reuse_copy(const ReuseArgs &a, cudaStream_t s) {
  dim3 grid((a.max_tokens + kCopyRows - 1) / kCopyRows, a.n_items, a.lay.L * a.lay.n_ch);
  reuse_copy_kernel<<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_relocate(const RelocArgs &a, cudaStream_t s) {
  dim3 grid((a.T + kRelocTile - 1) / kRelocTile, a.lay.L);
  const int n_units = a.lay.kind == KAMERA_GQA ? (a.lay.row_k >> 4) : (a.lay.rope_d >> 4);
  if (kThreads % n_units == 0)
    relocate_kernel<true><<<grid, kThreads, 0, s>>>(a);
  else
    relocate_kernel<false><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kamera
