// Shared-memory access, packed float32 arithmetic and index helpers used by the reuse kernels.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "kamera_dev.cuh"

namespace kamera {

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
// 16-byte store to global memory (the address is a global-space pointer)
__device__ __forceinline__ void stg16_global(void *p, const uint4 &v) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint32_t ldg_u16(const __nv_bfloat16 *p) {
  return __ldg(reinterpret_cast<const unsigned short *>(p));
}
__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// Two float32 lanes in one 64-bit register, for the packed f32x2 arithmetic of sm_100+.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 f2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(f32x2 v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// bf16 pair (low, high half of a 32-bit word) -> two float32 lanes
__device__ __forceinline__ f32x2 bf2_to_f2(uint32_t w) {
  return f2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ uint32_t f2_to_bf2(f32x2 v) {
  float lo, hi;
  f2_split(v, lo, hi);
  return pack2_rn(lo, hi);
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

// Patch value of 8 consecutive tile columns [n0, n0+8) of row r from the staged operands
// (the CUDA-core contraction). A: element (r, k) at ((k/8)*16 + r/8)*128 + (r%8)*16 +
// (k%8)*2; B (MN-major): element (n, k) at ((k/8)*ncore + n/8)*128 + (k%8)*16 + (n%8)*2.
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

}  // namespace kamera
