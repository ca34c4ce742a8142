// Patch forming on the device: the top-m factors of a conditioning deficit, written in the
// patch store's format (Kamera, App. A "form_patch": Δ = KV(B|A) − R(δ)KV(B|∅), keep
// U[:, :m]·S[:m] and Vt[:m]; §3 "Forming and applying the patch").
//
// The factors come from the randomized range finder with q power iterations (Halko,
// Martinsson & Tropp, "Finding structure with randomness", SIAM Review 2011, Alg. 4.4) and the
// SVD of the small projection (their Alg. 5.1):
//   Y = Δ Ω; Q = orth(Y); q times: Z = orth(ΔᵀQ), Q = orth(Δ Z);
//   Bᵀ = ΔᵀQ = V_B Σ Ũᵀ; U·Σ = Q Ũ_m Σ_m; V_mᵀ = (Bᵀ Ũ_m)ᵀ Σ_m⁻¹.
// Ω [W × k] is the caller's random test matrix. Each row of V_mᵀ is signed so that its entry
// of largest magnitude is positive (the first such entry on a tie); U·Σ's column flips with it.
//
// Everything is float32: GB300 runs float64 at a small fraction of its float32 rate, and the
// steps below stay accurate in float32.
//   orth() is shifted CholeskyQR3 (Fukaya, Kannan, Nakatsukasa, Yamamoto & Yanagisawa,
//   "Shifted Cholesky QR for computing the QR factorization of ill-conditioned matrices",
//   SIAM J. Sci. Comput. 2020): one Cholesky QR pass on G = YᵀY + sI with
//   s = 11 (M k + k (k + 1)) u ‖Y‖² (u = 2⁻²⁴, ‖Y‖² bounded by trace G), then two plain passes.
//   A pivot that is not positive (a zero column) drops its column: the column becomes zero and
//   no later column is reduced against it.
//   The SVD of the k-column Bᵀ is one-sided cyclic Jacobi (Hestenes 1958; Demmel & Veselić
//   1992): pairs of columns are rotated until every pair is orthogonal to within √W·2⁻²³ of
//   their norms (at most 30 sweeps); the rotations accumulate into Ũ and σ_j is the norm of
//   column j.
//
// One CTA of 256 threads per problem (one (layer, group) deficit [T × W]). The tall sketches
// live in a caller-provided workspace (two [max(T, W) × k] float32 buffers per problem);
// products go through a shared-memory tiled CTA GEMM; Bᵀ, its rotations and the k × k
// factors stay in shared memory.
#include <mutex>

#include "kamera_dev.cuh"

namespace kamera {

namespace {

constexpr int kThr = 256;
constexpr int kWarps = kThr / 32;
constexpr int kBM = 128, kBK = 32;  // GEMM: 128 rows of C per block, K in steps of 32
constexpr int kAPitch = kBM + 1;    // op(A) tile [kBK][kAPitch]: conflict-free stores and reads
constexpr int kStageF = kBK * kAPitch + kBK * kMaxSketch;  // floats of one GEMM stage

// Float offsets of the dynamic shared memory (one plan for host and device).
struct FormPlan {
  int tiles;     // GEMM: two stages of op(A) [kBK][kAPitch] and B [kBK][kMaxSketch]
  int g, r;      // k × k: Gram matrix / Cholesky factor, and the triangular inverse
  int v;         // k × k: Jacobi rotations Ũ, column-major
  int bc;        // W × k: Bᵀ, column-major (column j at bc + j*W)
  int nrm;       // k: column norms σ
  int sc_u;      // k: U·Σ column scales (sign · σ)
  int order;     // k ints: columns by σ, descending
  int total;     // floats
};

__host__ __device__ inline FormPlan form_plan(int W, int k) {
  FormPlan p;
  int o = 0;
  p.tiles = o;
  o += 2 * kStageF;
  p.g = o;
  o += k * k;
  p.r = o;
  o += k * k;
  p.v = o;
  o += k * k;
  p.bc = o;
  o += W * k;
  p.nrm = o;
  o += k;
  p.sc_u = o;
  o += k;
  p.order = o;
  o += k;
  p.total = o;
  return p;
}

template <typename Out>
__device__ __forceinline__ Out to_out(float x);
template <>
__device__ __forceinline__ float to_out<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// C = op(A) · B with float32 accumulation, by all threads of the CTA.
//   op(A) [M × K]: A itself (row stride lda) or, when TA, the transpose of A stored [K × M].
//   B [K × N], row stride ldb, N <= kMaxSketch (global or shared memory).
//   Element (i, j) goes to C[i*ldc + j], or to C[j*ldc + i] when TC, multiplied by scale[j]
//   when scale is given. C overlaps neither A nor B.
// Blocks of 128 rows of C; warp w owns columns [w·cpt, (w+1)·cpt) (cpt = ceil(N / 8)) and lane
// l rows l, l + 32, l + 64, l + 96, so op(A) reads are conflict-free and B reads broadcast.
// K advances in steps of 32 through two shared-memory stages: the next step's global loads
// are in registers while the current step computes, one barrier per step.
template <bool TA, bool TC, typename Out>
__device__ void cta_gemm(const float *A, long long lda, const float *B, long long ldb, Out *C,
                         long long ldc, int M, int N, int K, const float *scale, float *sm) {
  constexpr int kAper = kBK * kBM / kThr;          // op(A) elements a thread stages per step
  constexpr int kBper = kBK * kMaxSketch / kThr;   // B elements (upper bound) per step
  constexpr int kCols = kMaxSketch / 8;            // columns a warp can own
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cpt = (N + 7) / 8, c0 = warp * cpt;
  for (int m0 = 0; m0 < M; m0 += kBM) {
    float acc[4][kCols];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < kCols; ++c) acc[r][c] = 0.f;
    float ra[kAper], rb[kBper];
    auto load = [&](int k0) {  // global -> registers (zero outside the matrices)
#pragma unroll
      for (int j = 0; j < kAper; ++j) {
        const int e = tid + j * kThr;
        int kk, mm;
        if (TA) {  // A is [K × M]: consecutive threads walk M
          kk = e / kBM;
          mm = e - kk * kBM;
        } else {   // A is [M × K]: consecutive threads walk K
          mm = e / kBK;
          kk = e - mm * kBK;
        }
        const int gm = m0 + mm, gk = k0 + kk;
        ra[j] = (gm < M && gk < K) ? (TA ? A[(long long)gk * lda + gm] : A[(long long)gm * lda + gk])
                                   : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kBper; ++j) {
        const int e = tid + j * kThr;
        const int kk = e / kMaxSketch, n = e - kk * kMaxSketch;
        const int gk = k0 + kk;
        rb[j] = (n < N && gk < K) ? B[(long long)gk * ldb + n] : 0.f;
      }
    };
    auto store = [&](int st) {  // registers -> stage st
      float *ta = sm + st * kStageF, *tb = ta + kBK * kAPitch;
#pragma unroll
      for (int j = 0; j < kAper; ++j) {
        const int e = tid + j * kThr;
        int kk, mm;
        if (TA) {
          kk = e / kBM;
          mm = e - kk * kBM;
        } else {
          mm = e / kBK;
          kk = e - mm * kBK;
        }
        ta[kk * kAPitch + mm] = ra[j];
      }
#pragma unroll
      for (int j = 0; j < kBper; ++j) tb[tid + j * kThr] = rb[j];
    };
    __syncthreads();  // the previous use of the stages is over
    load(0);
    store(0);
    __syncthreads();
    int st = 0;
    for (int k0 = 0; k0 < K; k0 += kBK, st ^= 1) {
      const bool more = k0 + kBK < K;
      if (more) load(k0 + kBK);
      const float *ta = sm + st * kStageF, *tb = ta + kBK * kAPitch;
      const int kend = min(kBK, K - k0);
#pragma unroll 4
      for (int kk = 0; kk < kend; ++kk) {
        float av[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) av[r] = ta[kk * kAPitch + lane + 32 * r];
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          if (c < cpt) {
            const float bv = tb[kk * kMaxSketch + c0 + c];
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[r][c] = fmaf(av[r], bv, acc[r][c]);
          }
        }
      }
      if (more) store(st ^ 1);
      __syncthreads();
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int gi = m0 + lane + 32 * r;
      if (gi < M) {
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          const int col = c0 + c;
          if (c < cpt && col < N) {
            const float x = scale ? acc[r][c] * scale[col] : acc[r][c];
            if (TC)
              C[(long long)col * ldc + gi] = to_out<Out>(x);
            else
              C[(long long)gi * ldc + col] = to_out<Out>(x);
          }
        }
      }
    }
  }
  __syncthreads();
}

// G [k × k] (shared, row-major) = Yᵀ Y for Y [M × k] (row stride k). Each thread owns a 4 × 4
// block of the upper block triangle and a share of the rows (S row subsets when the blocks
// leave threads over); the subsets' partial blocks meet in `scratch` (S · k² floats) and the
// lower triangle is mirrored from the upper one.
__device__ void cta_gram(const float *Y, int M, int k, float *g, float *scratch) {
  const int tid = threadIdx.x;
  const int nb = (k + 3) >> 2, nblk = nb * (nb + 1) / 2;
  const int S = max(1, kThr / nblk);
  for (int w = tid; w < S * nblk; w += kThr) {
    const int sub = w / nblk;
    int b = w - sub * nblk, bi = 0;
    while (b >= nb - bi) {  // block b of the upper block triangle, row by row
      b -= nb - bi;
      ++bi;
    }
    const int bj = bi + b;
    const int i0 = 4 * bi, j0 = 4 * bj;
    float acc[4][4];
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) acc[x][y] = 0.f;
#pragma unroll 2
    for (int r = sub; r < M; r += S) {
      const float *row = Y + (long long)r * k;
      float u[4], v[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        u[x] = i0 + x < k ? row[i0 + x] : 0.f;
        v[x] = j0 + x < k ? row[j0 + x] : 0.f;
      }
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(u[x], v[y], acc[x][y]);
    }
    float *out = scratch + (long long)sub * k * k;
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y)
        if (i0 + x < k && j0 + y < k) out[(i0 + x) * k + j0 + y] = acc[x][y];
  }
  __syncthreads();
  for (int e = tid; e < k * k; e += kThr) {
    int i = e / k, j = e - i * k;
    if ((i >> 2) > (j >> 2)) {  // below the block diagonal: the mirror entry was computed
      const int t = i;
      i = j;
      j = t;
    }
    float sum = 0.f;
    for (int sub = 0; sub < S; ++sub) sum += scratch[(long long)sub * k * k + i * k + j];
    g[e] = sum;
  }
  __syncthreads();
}

// One Cholesky QR pass: dst [M × k] = src · L⁻ᵀ where L Lᵀ = srcᵀ src (+ sI when shifted).
// Row stride k for both; src and dst are distinct buffers.
__device__ void cholqr_pass(const float *src, float *dst, int M, int k, bool shifted, float *sm,
                            const FormPlan &p) {
  float *g = sm + p.g;  // row-major k × k; its lower triangle becomes L
  float *r = sm + p.r;  // r[c*k + j] = (L⁻¹)[j][c]: the [k × k] operand of dst = src · L⁻ᵀ
  cta_gram(src, M, k, g, sm + p.tiles);
  const int tid = threadIdx.x;
  if (shifted) {
    if (tid < 32) {
      float tr = 0.f;
      for (int j = tid; j < k; j += 32) tr += g[j * k + j];
      for (int o = 16; o > 0; o >>= 1) tr += __shfl_xor_sync(0xffffffffu, tr, o);
      const float s = 11.f * ((float)M * k + (float)k * (k + 1)) * 5.9604645e-8f * tr;
      __syncwarp();
      for (int j = tid; j < k; j += 32) g[j * k + j] += s;
    }
    __syncthreads();
  }
  // right-looking Cholesky on the lower triangle, all threads: scale column j by its pivot,
  // then update the trailing triangle
  for (int j = 0; j < k; ++j) {
    const float d = g[j * k + j];
    const float ljj = d > 0.f ? sqrtf(d) : 0.f;  // not positive (or NaN): drop column j
    const float inv = ljj > 0.f ? 1.f / ljj : 0.f;
    for (int i = j + 1 + tid; i < k; i += kThr) g[i * k + j] *= inv;
    __syncthreads();
    if (tid == 0) g[j * k + j] = ljj;
    const int rem = k - j - 1;
    for (int e = tid; e < rem * rem; e += kThr) {
      const int i = j + 1 + e / rem, l = j + 1 + e % rem;
      if (l <= i) g[i * k + l] -= g[i * k + j] * g[l * k + j];
    }
    __syncthreads();
  }
  // column c of L⁻¹ solves L x = e_c (forward substitution), one thread per column; a dropped
  // pivot gives x = 0. Four partial sums shorten the dependent chain.
  for (int c = tid; c < k; c += kThr) {
    for (int i = 0; i < c; ++i) r[c * k + i] = 0.f;
    for (int i = c; i < k; ++i) {
      float a0 = i == c ? 1.f : 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
      int l = c;
      for (; l + 3 < i; l += 4) {
        a0 -= g[i * k + l] * r[c * k + l];
        a1 -= g[i * k + l + 1] * r[c * k + l + 1];
        a2 -= g[i * k + l + 2] * r[c * k + l + 2];
        a3 -= g[i * k + l + 3] * r[c * k + l + 3];
      }
      for (; l < i; ++l) a0 -= g[i * k + l] * r[c * k + l];
      const float lii = g[i * k + i];
      r[c * k + i] = lii > 0.f ? ((a0 + a1) + (a2 + a3)) / lii : 0.f;
    }
  }
  __syncthreads();
  cta_gemm<false, false, float>(src, k, r, k, dst, k, M, k, k, nullptr, sm);
}

// Orthonormal basis of the columns of a [M × k] (row stride k) by shifted CholeskyQR3, with b
// as the second buffer. The basis ends in b.
__device__ void orth(float *a, float *b, int M, int k, float *sm, const FormPlan &p) {
  cholqr_pass(a, b, M, k, true, sm, p);
  cholqr_pass(b, a, M, k, false, sm, p);
  cholqr_pass(a, b, M, k, false, sm, p);
}

// Pair i of round `round` in the round-robin schedule over n (even) indices: every pair
// (p, q), p != q, meets once in n - 1 rounds and no index appears twice in one round.
__device__ __forceinline__ void rr_pair(int n, int round, int i, int &p, int &q) {
  if (i == 0) {
    p = n - 1;
    q = round;
  } else {
    p = (round + i) % (n - 1);
    q = (round - i + n - 1) % (n - 1);
  }
}

// One-sided Jacobi on the columns of bc [W × k] (column-major), rotations accumulated into
// v [k × k] (column-major, set to I here). A warp owns one pair for its whole rotation.
__device__ void jacobi_svd(float *bc, float *v, int W, int k) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int e = tid; e < k * k; e += kThr) v[e] = (e / k == e % k) ? 1.f : 0.f;
  __syncthreads();
  const int n = k + (k & 1);  // an odd k plays a dummy column
  const float tol = sqrtf((float)W) * 1.1920929e-7f;
  for (int sweep = 0; sweep < 30; ++sweep) {
    int rotated = 0;
    for (int round = 0; round < n - 1; ++round) {
      for (int i = warp; i < n / 2; i += kWarps) {
        int pc, qc;
        rr_pair(n, round, i, pc, qc);
        if (pc >= k || qc >= k) continue;
        float *x = bc + (long long)pc * W, *y = bc + (long long)qc * W;
        float a = 0.f, b = 0.f, c = 0.f;
        for (int w = lane; w < W; w += 32) {
          const float xv = x[w], yv = y[w];
          a = fmaf(xv, xv, a);
          b = fmaf(yv, yv, b);
          c = fmaf(xv, yv, c);
        }
        for (int o = 16; o > 0; o >>= 1) {
          a += __shfl_xor_sync(0xffffffffu, a, o);
          b += __shfl_xor_sync(0xffffffffu, b, o);
          c += __shfl_xor_sync(0xffffffffu, c, o);
        }
        if (!(fabsf(c) > tol * sqrtf(a) * sqrtf(b))) continue;  // orthogonal, or a zero column
        const float zeta = (b - a) / (2.f * c);
        const float t = copysignf(1.f, zeta) / (fabsf(zeta) + sqrtf(fmaf(zeta, zeta, 1.f)));
        const float cs = 1.f / sqrtf(fmaf(t, t, 1.f)), sn = cs * t;
        __syncwarp();
        for (int w = lane; w < W; w += 32) {
          const float xv = x[w], yv = y[w];
          x[w] = cs * xv - sn * yv;
          y[w] = sn * xv + cs * yv;
        }
        float *vx = v + pc * k, *vy = v + qc * k;
        for (int j = lane; j < k; j += 32) {
          const float xv = vx[j], yv = vy[j];
          vx[j] = cs * xv - sn * yv;
          vy[j] = sn * xv + cs * yv;
        }
        rotated = 1;
        __syncwarp();
      }
      __syncthreads();
    }
    if (!__syncthreads_or(rotated)) break;
  }
}

__global__ void __launch_bounds__(kThr, 1) form_patch_kernel(const __grid_constant__ FormArgs a) {
  extern __shared__ __align__(16) float sm[];
  const FormPlan p = form_plan(a.W, a.k);
  const int prob = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, W = a.W, k = a.k, m = a.m;
  const float *D = a.delta + (long long)prob * a.delta_stride;
  const float *om = a.omega + (long long)prob * a.omega_stride;
  const long long buf = (long long)max(T, W) * k;
  float *y = a.work + (long long)prob * 2 * buf;  // the basis Q ends here after every orth
  float *z = y + buf;

  cta_gemm<false, false, float>(D, a.ld, om, k, z, k, T, k, W, nullptr, sm);  // Y = Δ Ω
  orth(z, y, T, k, sm, p);
  for (int it = 0; it < a.q; ++it) {
    cta_gemm<true, false, float>(D, a.ld, y, k, z, k, W, k, T, nullptr, sm);  // Z = Δᵀ Q
    orth(z, y, W, k, sm, p);                                                   // Z = orth(Z)
    cta_gemm<false, false, float>(D, a.ld, y, k, z, k, T, k, W, nullptr, sm);  // Y = Δ Z
    orth(z, y, T, k, sm, p);                                                   // Q = orth(Y)
  }
  float *bc = sm + p.bc, *v = sm + p.v;
  cta_gemm<true, true, float>(D, a.ld, y, k, bc, W, W, k, T, nullptr, sm);  // Bᵀ = Δᵀ Q
  jacobi_svd(bc, v, W, k);

  // σ_j = ‖Bᵀ ũ_j‖, then the columns by σ (descending, ties by column index)
  float *nrm = sm + p.nrm, *sc_u = sm + p.sc_u;
  int *order = reinterpret_cast<int *>(sm + p.order);
  for (int j = warp; j < k; j += kWarps) {
    const float *x = bc + (long long)j * W;
    float s = 0.f;
    for (int w = lane; w < W; w += 32) s = fmaf(x[w], x[w], s);
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) nrm[j] = sqrtf(s);
  }
  __syncthreads();
  for (int j = tid; j < k; j += kThr) {
    int rank = 0;
    for (int i = 0; i < k; ++i) rank += (nrm[i] > nrm[j]) || (nrm[i] == nrm[j] && i < j);
    order[rank] = j;
  }
  __syncthreads();
  // rows of V_mᵀ, signed by their largest-magnitude entry; the U·Σ column scales
  __nv_bfloat16 *vt = a.vt + (long long)prob * a.vt_stride;
  for (int j = warp; j < m; j += kWarps) {
    const int c = order[j];
    const float sig = nrm[c];
    const float *x = bc + (long long)c * W;
    float best = -1.f, bval = 0.f;
    int bidx = 0x7fffffff;
    for (int w = lane; w < W; w += 32) {
      const float mag = fabsf(x[w]);
      if (mag > best) {  // w grows along a lane, so a lane keeps its first maximum
        best = mag;
        bval = x[w];
        bidx = w;
      }
    }
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const float ov = __shfl_xor_sync(0xffffffffu, bval, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
      if (ob > best || (ob == best && oi < bidx)) {
        best = ob;
        bval = ov;
        bidx = oi;
      }
    }
    const float sgn = bval < 0.f ? -1.f : 1.f;
    const float sv = sig > 0.f ? sgn / sig : 0.f;
    for (int w = lane; w < W; w += 32) vt[(long long)j * W + w] = __float2bfloat16_rn(x[w] * sv);
    if (lane == 0) {
      sc_u[j] = sgn * sig;
      if (a.sigma) a.sigma[(long long)prob * m + j] = sig;
    }
  }
  // the columns of Ũ_m in σ order as the [k × m] operand of U·Σ = Q Ũ_m (scaled per column)
  float *um = sm + p.g;
  for (int e = tid; e < k * m; e += kThr) {
    const int i = e / m, j = e - i * m;
    um[e] = v[order[j] * k + i];
  }
  __syncthreads();
  cta_gemm<false, false, __nv_bfloat16>(y, k, um, m, a.u + (long long)prob * a.u_stride, m, T, m,
                                        k, sc_u, sm);
}

}  // namespace

size_t form_patch_workspace(long long n, int T, int W, int k) {
  const size_t rows = (size_t)(T > W ? T : W);
  return (size_t)n * 2 * rows * (size_t)k * sizeof(float);
}

size_t form_patch_smem(int W, int k) { return (size_t)form_plan(W, k).total * sizeof(float); }

namespace {

int g_form_configured[64] = {0};  // per device: the kernel's dynamic shared-memory limit
std::mutex g_form_mu;

// Once per device: the kernel is loaded and may use the device's opt-in shared memory.
cudaError_t configure_form(int dev) {
  std::lock_guard<std::mutex> lock(g_form_mu);
  if (g_form_configured[dev]) return cudaSuccess;
  int optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, form_patch_kernel);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(form_patch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e != cudaSuccess) return e;
  g_form_configured[dev] = optin;
  return cudaSuccess;
}

}  // namespace

cudaError_t prepare_form_patch() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  return configure_form(dev);
}

cudaError_t launch_form_patch(const FormArgs &a, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const size_t smem = form_patch_smem(a.W, a.k);
  e = configure_form(dev);
  if (e != cudaSuccess) return e;
  if ((size_t)g_form_configured[dev] < smem) return cudaErrorInvalidValue;
  if (a.n == 0) return cudaSuccess;
  form_patch_kernel<<<a.n, kThr, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kamera

// ---------------------------------------------------------------------------------------
// kamera_form_patch_static_scratch: kamera_form_patch with its workspace in a fixed array of
// this library's device memory, for callers that cannot allocate device memory where they call
// it (see include/kamera.h). One array per device, shared by every call on that device.
// ---------------------------------------------------------------------------------------

namespace {

static __device__ __align__(256) float g_form_scratch[KAMERA_FORM_PATCH_SCRATCH_BYTES /
                                                      sizeof(float)];

// Set-up, once per device with that device current: the array's device address (the lookup
// also makes CUDA load this file's device code, which reserves the array) and the kernel,
// loaded and configured. Later calls on the device reuse the address.
cudaError_t form_scratch(void **out) {
  static void *ptrs[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_form_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    e = kamera::prepare_form_patch();
    if (e != cudaSuccess) return e;
    ptrs[dev] = p;
  }
  *out = ptrs[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" kamera_status kamera_form_patch_static_scratch(
    const float *d_delta, int64_t ld, int64_t delta_stride, int32_t num_problems, int32_t T,
    int32_t W, const float *d_omega, int64_t omega_stride, int32_t k, int32_t q, int32_t m,
    void *d_u, int64_t u_stride, void *d_vt, int64_t vt_stride, float *d_sigma,
    kamera_stream_t stream) {
  const kamera_status st =
      kamera::form_patch_args(d_delta, ld, delta_stride, num_problems, T, W, d_omega,
                              omega_stride, k, q, m, d_u, u_stride, d_vt, vt_stride, d_sigma);
  if (st != KAMERA_OK) return st;
  if (kamera::form_patch_workspace(num_problems, T, W, k) > KAMERA_FORM_PATCH_SCRATCH_BYTES)
    return KAMERA_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  if (form_scratch(&scratch) != cudaSuccess) return KAMERA_ERR_CUDA;  // set-up on a first call
  if (num_problems == 0) return KAMERA_OK;
  return kamera_form_patch(d_delta, ld, delta_stride, num_problems, T, W, d_omega, omega_stride,
                           k, q, m, d_u, u_stride, d_vt, vt_stride, d_sigma, scratch,
                           KAMERA_FORM_PATCH_SCRATCH_BYTES, stream);
}
