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
// 128 bytes in flight.
__global__ void __launch_bounds__(kThreads) relocate_kernel(const __grid_constant__ RelocArgs a) {
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
  const int n = rows * n_units;
  constexpr int B = 4;
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

// Unpatched layers of reuse items: the canonical rows of (item, layer, channel) stream through
// registers to their slots, rope columns rotated on the way (R(delta) with no patch term),
// everything else copied byte for byte. One CTA per 128 rows of an (item, layer, channel);
// the grid runs items fastest after the row blocks, so placements that share a canonical read
// it from L2. Patched layers are left to the tensor-core kernel.
template <bool kFixedUnit>
__device__ __forceinline__ void copy_rows(const DevLayout &lay, int ch, bool rotate, int rows,
                                          int row, const __nv_bfloat16 *src0,
                                          __nv_bfloat16 *pool, const long long *rowoff,
                                          const float2 *cs) {
  const int tid = threadIdx.x;
  const int upr = row >> 4;
  constexpr int B = 2;  // two units (four 16-byte vectors) in flight per thread
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
          off[k] = rowoff[r];
          const __nv_bfloat16 *src = src0 + (long long)r * row;
          ra[k] = __ldg(reinterpret_cast<const uint4 *>(src + cu.ca));
          rb_[k] = __ldg(reinterpret_cast<const uint4 *>(src + cu.cb));
        }
      }
#pragma unroll
      for (int k = 0; k < B; ++k) {
        if (off[k] < 0) continue;
        __nv_bfloat16 *dst = pool + off[k];
        if (cu.rot == 0) {
          st16(dst + cu.ca, ra[k]);
          st16(dst + cu.cb, rb_[k]);
        } else {
          float xa[8], xb[8];
          unpack8(ra[k], xa);
          unpack8(rb_[k], xb);
          rotate_unit(cu, cs, xa, xb);
          st16(dst + cu.ca, pack8_rn(xa));
          st16(dst + cu.cb, pack8_rn(xb));
        }
      }
    }
  } else {
    const int n = rows * upr;
    for (int base = tid; base < n; base += kThreads * B) {
      uint4 ra[B], rb_[B];
      ColUnit cu[B];
      long long off[B];
#pragma unroll
      for (int k = 0; k < B; ++k) {
        const int w = base + k * kThreads;
        off[k] = -1;
        if (w < n) {
          const int r = w / upr;
          cu[k] = col_unit(lay, ch, w - r * upr, rotate);
          off[k] = rowoff[r];
          const __nv_bfloat16 *src = src0 + (long long)r * row;
          ra[k] = __ldg(reinterpret_cast<const uint4 *>(src + cu[k].ca));
          rb_[k] = __ldg(reinterpret_cast<const uint4 *>(src + cu[k].cb));
        }
      }
#pragma unroll
      for (int k = 0; k < B; ++k) {
        if (off[k] < 0) continue;
        __nv_bfloat16 *dst = pool + off[k];
        if (cu[k].rot == 0) {
          st16(dst + cu[k].ca, ra[k]);
          st16(dst + cu[k].cb, rb_[k]);
        } else {
          float xa[8], xb[8];
          unpack8(ra[k], xa);
          unpack8(rb_[k], xb);
          rotate_unit(cu[k], cs, xa, xb);
          st16(dst + cu[k].ca, pack8_rn(xa));
          st16(dst + cu[k].cb, pack8_rn(xb));
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads) reuse_copy_kernel(const __grid_constant__ ReuseArgs a) {
  __shared__ float2 cs[kMaxPairs];
  __shared__ long long rowoff[kCopyRows];  // element offset of each row in the layer's pool
  const DevLayout &lay = a.lay;
  const int tid = threadIdx.x;
  const int item = blockIdx.y;
  const int layer = blockIdx.z / lay.n_ch;
  const int ch = blockIdx.z - layer * lay.n_ch;
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
  if (rotate)
    for (int i = tid; i < lay.npairs; i += kThreads)
      cs[i] = rope_phase(a.freq.q[i], pair_delta(it, lay, i));
  for (int r = tid; r < rows; r += kThreads) {
    const long long slot =
        slot_of(a.pool, lay.page_size, it.req, (long long)it.start_tok + t0 + r, a.status);
    rowoff[r] = slot < 0 ? -1 : slot * row;
  }
  __syncthreads();
  const __nv_bfloat16 *src0 = static_cast<const __nv_bfloat16 *>(ch == 0 ? it.canon_k
                                                                          : it.canon_v) +
                              ((long long)layer * it.num_tokens + t0) * row;
  __nv_bfloat16 *pool = (ch == 0 ? a.pool.k : a.pool.v) + (long long)layer * a.pool.num_slots * row;
  if (kThreads % (row >> 4) == 0)
    copy_rows<true>(lay, ch, rotate, rows, row, src0, pool, rowoff, cs);
  else
    copy_rows<false>(lay, ch, rotate, rows, row, src0, pool, rowoff, cs);
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
  relocate_kernel<<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kamera
