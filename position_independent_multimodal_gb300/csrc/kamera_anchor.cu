// Re-anchoring of keys stored before rotation: every token's rope pairs turn from zero to the
// token's own absolute position (QV-PIC, "Model-Native Template-Conditioned Compilation",
// Eq. 2: K = R(K_bar, P(q)), the model-native M-RoPE operator applied at the request
// positions). Values and the MLA latent are position-independent and are copied byte for byte.
//
// One CTA of 256 threads per 32 rows of an (item, channel) and seven layers. For K it first
// builds the per-row phase table [32][npairs] in shared memory (each (row, pair) from the
// token's position on the pair's M-RoPE section, by the exact Q0.64 range reduction the other
// kernels use); every head and every one of the seven layers then reads the same phases, and
// the rows' page slots are resolved once for all seven. Rows stream through registers to their
// slots in 16-byte vectors: where the row's 16-column units divide the block, a thread keeps
// one unit and has four rows in flight; otherwise it walks (row, unit) pairs, two at a time.
#include "kamera_dev.cuh"

namespace kamera {

namespace {

constexpr int kThr = 256;
constexpr int kRows = 32;    // rows per CTA: the phase table is kRows x npairs float2
constexpr int kLayers = 7;   // layers per CTA: the phase table and the slots serve them all

__device__ __forceinline__ void st16(void *p, const uint4 &v) {
  *reinterpret_cast<uint4 *>(p) = v;
}

__device__ __forceinline__ void store_unit(__nv_bfloat16 *dst, const ColUnit &cu, const uint4 &ra,
                                           const uint4 &rb, const float2 *cs) {
  if (cu.rot == 0) {
    st16(dst + cu.ca, ra);
    st16(dst + cu.cb, rb);
  } else {
    float xa[8], xb[8];
    unpack8(ra, xa);
    unpack8(rb, xb);
    rotate_unit(cu, cs, xa, xb);
    st16(dst + cu.ca, pack8_rn(xa));
    st16(dst + cu.cb, pack8_rn(xb));
  }
}

__global__ void __launch_bounds__(kThr) reanchor_kernel(const __grid_constant__ AnchorArgs a) {
  __shared__ float2 cs[kRows * kMaxPairs];
  __shared__ long long rowoff[kRows];  // element offset of each row in a layer's pool
  const DevLayout &lay = a.lay;
  const int tid = threadIdx.x;
  const int item = blockIdx.y;
  const int ch = blockIdx.z % lay.n_ch;
  const int l0 = (blockIdx.z / lay.n_ch) * kLayers;
  const int l1 = min(lay.L, l0 + kLayers);
  const kamera_anchor_item it = a.items[item];
  if (anchor_item_check(it, lay, a.pool, a.max_tokens) != 0) {
    if (blockIdx.x == 0 && blockIdx.z == 0 && tid == 0) atomicOr(a.status, KAMERA_DEVICE_BAD_ITEM);
    return;
  }
  const int t0 = blockIdx.x * kRows;
  if (t0 >= it.num_tokens) return;
  const int rows = min(kRows, it.num_tokens - t0);
  const bool rotate = ch == 0;
  const int row = ch == 0 ? lay.row_k : lay.row_v;
  const int np = lay.npairs;
  if (rotate) {
    const int stride = lay.mrope ? 3 : 1;  // [T] positions, or [T][3] (t, h, w) for M-RoPE
    const long long *pos =
        reinterpret_cast<const long long *>(it.positions) + (long long)t0 * stride;
    for (int e = tid; e < rows * np; e += kThr) {
      const int r = e / np, i = e - r * np;
      const int axis = lay.mrope ? mrope_axis(lay, i) : 0;
      cs[e] = rope_phase(a.freq.q[i], __ldg(pos + (long long)r * stride + axis));
    }
  }
  for (int r = tid; r < rows; r += kThr) {
    const long long slot =
        slot_of(a.pool, lay.page_size, it.req, (long long)it.start_tok + t0 + r, a.status);
    rowoff[r] = slot < 0 ? -1 : slot * row;
  }
  __syncthreads();
  const __nv_bfloat16 *canon = static_cast<const __nv_bfloat16 *>(ch == 0 ? it.canon_k
                                                                           : it.canon_v);
  __nv_bfloat16 *pool0 = ch == 0 ? a.pool.k : a.pool.v;
  const int upr = row >> 4;  // 16-column units per row
  if (kThr % upr == 0 && kRows % (kThr / upr) == 0) {
    // every thread keeps one column unit and walks the rows r0, r0 + rstep, ...; a row's
    // phases are read once into registers and turn the row in all of the CTA's layers, whose
    // loads are all in flight before the first store
    const int u = tid % upr, r0 = tid / upr, rstep = kThr / upr;
    const ColUnit cu = col_unit(lay, ch, u, rotate);
    const int nl = l1 - l0;
    for (int r = r0; r < rows; r += rstep) {
      const long long off = rowoff[r];
      if (off < 0) continue;
      uint4 ra[kLayers], rb[kLayers];
#pragma unroll
      for (int l = 0; l < kLayers; ++l) {
        if (l < nl) {
          const __nv_bfloat16 *src = canon + ((long long)(l0 + l) * it.num_tokens + t0 + r) * row;
          ra[l] = __ldg(reinterpret_cast<const uint4 *>(src + cu.ca));
          rb[l] = __ldg(reinterpret_cast<const uint4 *>(src + cu.cb));
        }
      }
      float2 c[8];
      if (cu.rot != 0) unit_phases(cu, cs + r * np, c);
#pragma unroll
      for (int l = 0; l < kLayers; ++l) {
        if (l >= nl) break;
        __nv_bfloat16 *dst = pool0 + (long long)(l0 + l) * a.pool.num_slots * row + off;
        if (cu.rot == 0) {
          st16(dst + cu.ca, ra[l]);
          st16(dst + cu.cb, rb[l]);
        } else {
          float xa[8], xb[8];
          unpack8(ra[l], xa);
          unpack8(rb[l], xb);
          rotate_unit_with(cu, c, xa, xb);
          st16(dst + cu.ca, pack8_rn(xa));
          st16(dst + cu.cb, pack8_rn(xb));
        }
      }
    }
  } else {
    const int n = rows * upr;
    constexpr int B = 2;
    for (int layer = l0; layer < l1; ++layer) {
      const __nv_bfloat16 *src0 = canon + ((long long)layer * it.num_tokens + t0) * row;
      __nv_bfloat16 *pool = pool0 + (long long)layer * a.pool.num_slots * row;
      for (int base = tid; base < n; base += kThr * B) {
        uint4 ra[B], rb[B];
        ColUnit cu[B];
        int rr[B];
#pragma unroll
        for (int k = 0; k < B; ++k) {
          const int w = base + k * kThr;
          rr[k] = -1;
          if (w < n) {
            const int r = w / upr;
            rr[k] = r;
            cu[k] = col_unit(lay, ch, w - r * upr, rotate);
            const __nv_bfloat16 *src = src0 + (long long)r * row;
            ra[k] = __ldg(reinterpret_cast<const uint4 *>(src + cu[k].ca));
            rb[k] = __ldg(reinterpret_cast<const uint4 *>(src + cu[k].cb));
          }
        }
#pragma unroll
        for (int k = 0; k < B; ++k)
          if (rr[k] >= 0 && rowoff[rr[k]] >= 0)
            store_unit(pool + rowoff[rr[k]], cu[k], ra[k], rb[k], cs + rr[k] * np);
      }
    }
  }
}

}  // namespace

cudaError_t launch_reanchor(const AnchorArgs &a, cudaStream_t s) {
  const int groups = (a.lay.L + kLayers - 1) / kLayers;
  const dim3 grid((unsigned)((a.max_tokens + kRows - 1) / kRows), (unsigned)a.n_items,
                  (unsigned)(groups * a.lay.n_ch));
  reanchor_kernel<<<grid, kThr, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kamera
