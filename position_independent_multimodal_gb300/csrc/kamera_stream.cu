// Streaming kernels of the Kamera operator (CUDA cores only).
//
//  * reuse_stream_kernel: canonical -> pool for one (item, layer, channel, 32-token tile):
//    R(delta) on the rope columns, the rank-m patch as float32 FMAs, one RNE to bf16, 16-byte
//    stores at the token's slot (Kamera, App. A "apply_reuse"; Eq. 1). It serves every rank;
//    the tensor-core kernel takes over the patched layers at larger ranks.
//  * relocate_kernel: the survivor path, rotating the rope columns of pool rows in place
//    (§5 "Sliding-window survival"; Fig. 2 rotate_k_pe_inplace).
#include "kamera_dev.cuh"

namespace kamera {

namespace {

constexpr int kTile = 32;      // tokens per CTA
constexpr int kThreads = 256;

__device__ __forceinline__ uint4 ld16(const void *p) {
  return __ldg(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void st16(void *p, const uint4 &v) {
  *reinterpret_cast<uint4 *>(p) = v;
}

__global__ void __launch_bounds__(kThreads)
    reuse_stream_kernel(const __grid_constant__ ReuseArgs a) {
  extern __shared__ float u_tile[];  // [groups of this channel][kTile][m]
  __shared__ float2 cs[kMaxPairs];
  __shared__ long long slots[kTile];

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
  const int T = it.num_tokens;
  const int t0 = blockIdx.x * kTile;
  if (t0 >= T) return;
  const int rows = min(kTile, T - t0);
  const bool rotate = (ch == 0) && it.delta != 0;
  const bool patched = layer_patched(it, layer);
  const int m = it.patch_m;
  const int tid = threadIdx.x;

  if (rotate)
    for (int i = tid; i < lay.npairs; i += kThreads) cs[i] = rope_phase(a.freq.q[i], it.delta);
  for (int r = tid; r < rows; r += kThreads)
    slots[r] = slot_of(a.pool, lay.page_size, it.req, (long long)it.start_tok + t0 + r,
                       a.status);
  // groups of this channel: GQA K -> {0}, GQA V -> {1}, MLA -> {0, 1}
  const int g_first = (lay.kind == KAMERA_GQA) ? ch : 0;
  const int n_groups = (lay.kind == KAMERA_GQA) ? 1 : 2;
  const __nv_bfloat16 *vt_layer = nullptr;
  if (patched) {
    const int li = layer - it.patch_l0;
    const __nv_bfloat16 *pu = static_cast<const __nv_bfloat16 *>(it.patch_u);
    for (int gi = 0; gi < n_groups; ++gi) {
      const __nv_bfloat16 *src = pu + ((long long)(li * 2 + g_first + gi) * T + t0) * m;
      float *dst = u_tile + gi * kTile * m;
      for (int e = tid; e < rows * m; e += kThreads) dst[e] = __bfloat162float(src[e]);
    }
    vt_layer = static_cast<const __nv_bfloat16 *>(it.patch_vt) +
               (long long)li * m * (lay.w0 + lay.w1);
  }
  __syncthreads();

  const int row = ch == 0 ? lay.row_k : lay.row_v;
  const __nv_bfloat16 *canon =
      static_cast<const __nv_bfloat16 *>(ch == 0 ? it.canon_k : it.canon_v) +
      ((long long)layer * T + t0) * row;
  __nv_bfloat16 *pool = (ch == 0 ? a.pool.k : a.pool.v) + (long long)layer * a.pool.num_slots * row;
  const int upr = row >> 4;

  for (int w = tid; w < rows * upr; w += kThreads) {
    const int r = w / upr;
    const int u = w - r * upr;
    const long long slot = slots[r];
    if (slot < 0) continue;
    const ColUnit c = col_unit(lay, ch, u, rotate);
    const __nv_bfloat16 *src = canon + (long long)r * row;
    __nv_bfloat16 *dst = pool + slot * row;
    const uint4 ra = ld16(src + c.ca), rb = ld16(src + c.cb);
    if (c.rot == 0 && !patched) {  // byte copy: nothing to compute
      st16(dst + c.ca, ra);
      st16(dst + c.cb, rb);
      continue;
    }
    float xa[8], xb[8];
    unpack8(ra, xa);
    unpack8(rb, xb);
    rotate_unit(c, cs, xa, xb);
    if (patched) {
      const int g = c.group;
      const int wg = g == 0 ? lay.w0 : lay.w1;
      const __nv_bfloat16 *vt = vt_layer + (g == 0 ? 0 : (long long)m * lay.w0);
      const float *ur = u_tile + (g - g_first) * kTile * m + r * m;
      float pa[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      float pb[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int j = 0; j < m; ++j) {
        const float uj = ur[j];
        float va[8], vb[8];
        unpack8(ld16(vt + (long long)j * wg + c.gca), va);
        unpack8(ld16(vt + (long long)j * wg + c.gcb), vb);
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
    }
    st16(dst + c.ca, pack8_rn(xa));
    st16(dst + c.cb, pack8_rn(xb));
  }
}

constexpr int kRelocTile = 16;

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
  for (int w = tid; w < rows * n_units; w += kThreads) {
    const int r = w / n_units;
    const int u = u_first + (w - r * n_units);
    const long long slot = slots[r];
    if (slot < 0) continue;
    const ColUnit c = col_unit(lay, 0, u, true);
    __nv_bfloat16 *p = pool + slot * lay.row_k;
    const uint4 ra = *reinterpret_cast<const uint4 *>(p + c.ca);
    const uint4 rb = *reinterpret_cast<const uint4 *>(p + c.cb);
    float xa[8], xb[8];
    unpack8(ra, xa);
    unpack8(rb, xb);
    rotate_unit(c, cs, xa, xb);
    st16(p + c.ca, pack8_rn(xa));
    st16(p + c.cb, pack8_rn(xb));
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

cudaError_t launch_reuse_stream(const ReuseArgs &a, int tiles, int n_items, cudaStream_t s) {
  const int n_groups = a.lay.kind == KAMERA_GQA ? 1 : 2;
  const size_t smem = (size_t)n_groups * kTile * a.max_m * sizeof(float);
  dim3 grid(tiles, n_items, a.lay.L * a.lay.n_ch);
  reuse_stream_kernel<<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_relocate(const RelocArgs &a, cudaStream_t s) {
  dim3 grid((a.T + kRelocTile - 1) / kRelocTile, a.lay.L);
  relocate_kernel<<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

int reuse_stream_tile() { return kTile; }

}  // namespace kamera
