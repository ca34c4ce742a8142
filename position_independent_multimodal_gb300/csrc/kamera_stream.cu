// Streaming kernels of the Kamera operator (CUDA cores only).
//
//  * relocate_kernel: the survivor path, rotating the rope columns of pool rows in place
//    (§5 "Sliding-window survival"; Fig. 2 rotate_k_pe_inplace).
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

cudaError_t launch_relocate(const RelocArgs &a, cudaStream_t s) {
  dim3 grid((a.T + kRelocTile - 1) / kRelocTile, a.lay.L);
  relocate_kernel<<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kamera
