// Patch forming on the device: the top-m factors of a conditioning deficit, written in the
// patch store's format (Kamera, App. A "form_patch": Δ = KV(B|A) − R(δ)KV(B|∅), keep
// U[:, :m]·S[:m] and Vt[:m]; §3 "Forming and applying the patch").
//
// The factors come from the randomized range finder with q power iterations (Halko,
// Martinsson & Tropp, "Finding structure with randomness", SIAM Review 2011, Alg. 4.4) and the
// SVD of the small projection (their Alg. 5.1):
//   Y = Δ Ω; Q = orth(Y); q times: Z = orth(ΔᵀQ), Q = orth(Δ Z);
//   Bᵀ = ΔᵀQ = V_B Σ Ũᵀ; U·Σ = Q Ũ_m Σ_m; V_mᵀ = the first m columns of V_B, transposed.
// Ω [W × k] is the caller's random test matrix. Each row of V_mᵀ is signed so that its entry
// of largest magnitude is positive (the first such entry on a tie); U·Σ's column flips with it.
//
// One problem's work is spread over tiles of 128 rows, one CTA per tile, in a chain of kernels
// on the caller's stream:
//   * Products with Δ: Y = Δ X over tiles of T (K = W) and Z = Δᵀ X over tiles of W (K = T),
//     as tcgen05 MMAs of kind tf32 with float32 accumulators in TMEM. Each float32 operand x
//     is split into two tf32 numbers, hi = rn(x) and lo = rn(x − hi), so that x = hi + lo to
//     about 2⁻²² relative; the three products hi·hi + hi·lo + lo·hi give float32-accurate
//     results (the dropped lo·lo term is 2⁻²² relative).
//   * orth() is shifted CholeskyQR3 (Fukaya, Kannan, Nakatsukasa, Yamamoto & Yanagisawa,
//     "Shifted Cholesky QR for computing the QR factorization of ill-conditioned matrices",
//     SIAM J. Sci. Comput. 2020). Each kernel that writes a tall matrix X also writes the
//     partial Gram matrix of each of its tiles; the CTA that finishes last for a problem (an
//     atomic count, no waiting) adds them in tile order, so results do not depend on
//     scheduling, factors G = L Lᵀ and stores L⁻ᵀ for the next kernel, which multiplies its
//     tiles by it. The first pass of each orth adds s = 11 (M k + k (k + 1)) u ‖X‖² to the
//     diagonal (u = 2⁻²⁴, ‖X‖² bounded by trace G). A pivot that is not positive (a zero
//     column) drops its column: the column becomes zero and no later column is reduced
//     against it. The third pass is folded into the consumer: a product with Δ multiplies its
//     output tile by L⁻ᵀ instead, since Δᵀ(X L⁻ᵀ) = (ΔᵀX) L⁻ᵀ.
//   * The SVD of the k-column Bᵀ goes through its QR factorisation (Chan, "An improved
//     algorithm for computing the singular value decomposition", ACM TOMS 1982): CholeskyQR3
//     gives Bᵀ = Q_B R_B with R_B = L3ᵀ L2ᵀ L1ᵀ, and one-sided cyclic Jacobi (Hestenes 1958;
//     Demmel & Veselić 1992) on the k × k factor gives R_B Ṽ = U_R Σ. So V_B = Q_B U_R and
//     Ũ = Ṽ; σ_j is the norm of column j of R_B Ṽ. Jacobi rotates a pair of columns until
//     they are orthogonal to within √k·2⁻²³ of their norms (at most 30 sweeps).
//   * V_B = B₂ (L3⁻ᵀ U_R) over tiles of W (B₂: Bᵀ after two passes): each tile writes its
//     rows of V_mᵀ and the largest-magnitude entry of each of its columns; the last CTA picks
//     each column's sign from those and flips the rows that need it (exact on bf16).
//   * U·Σ = Y₂ (L⁻ᵀ Ũ_m Σ_m S), with Y₂ the range basis before its folded third pass and S
//     the signs, over tiles of T.
// Everything is float32: GB300 runs float64 at a small fraction of its float32 rate, and the
// steps above stay accurate in float32.
//
// A device-side wait that runs out of time (2 s; far beyond any MMA here) writes NaN into the
// tile it was producing, which carries through to the problem's outputs.
#include <math.h>
#include <mutex>

#include "kamera_dev.cuh"
#include "kamera_ptx.cuh"
#include "kamera_smem.cuh"

namespace kamera {

namespace {

constexpr int kThr = 256;
constexpr int kWarps = kThr / 32;
constexpr int kRows = 128;  // rows of a tile: one CTA, the MMA's M
constexpr int kCk = 32;     // K columns per staged chunk (128 bytes of float32 per row)
constexpr uint64_t kWaitNsF = 2000000000ull;

// Odd row pitch (floats) of a [128 × k] float32 tile in shared memory: threads that own
// consecutive rows reach different banks.
__host__ __device__ inline int tile_pitch(int k) { return (k & 1) ? k + 2 : k + 1; }
__host__ __device__ inline int pad16(int k) { return (k + 15) & ~15; }
__host__ __device__ inline int ntiles(int M) { return (M + kRows - 1) / kRows; }

// Row subsets of the partial Gram: threads own 4 × 4 blocks of the upper block triangle, and
// blocks are repeated over S subsets of the rows when they leave threads over.
__host__ __device__ inline int gram_subsets(int k) {
  const int nb = (k + 3) >> 2, nblk = nb * (nb + 1) / 2;
  return kThr / nblk > 1 ? kThr / nblk : 1;
}

}  // namespace

// Per-problem workspace (floats): the T-side range basis, the W-side basis (then Bᵀ), the
// per-tile partial Gram matrices, two L⁻ᵀ slots used in turn along the chain, L⁻ᵀ of the
// T-side basis's third pass, the three factors of Bᵀ's CholeskyQR, N = L3⁻ᵀ U_R and Ũ_m
// (k × m each), the k × m matrix that maps Y₂ to U·Σ, σ, the per-tile sign candidates of V_B
// (3 values per tile and column) and the count of finished CTAs.
struct FormWs {
  long long t, w, g, li0, li1, ly, lb1, lb2, lb3, nm, vs, mu, sig, cand, cnt, per;
};

__host__ __device__ inline FormWs form_ws(int T, int W, int k) {
  FormWs s;
  const long long k2 = (long long)k * k;
  const long long nt = ntiles(T > W ? T : W);
  long long o = 0;
  s.t = o;
  o += (long long)T * k;
  s.w = o;
  o += (long long)W * k;
  s.g = o;
  o += nt * k2;
  s.li0 = o;
  o += k2;
  s.li1 = o;
  o += k2;
  s.ly = o;
  o += k2;
  s.lb1 = o;
  o += k2;
  s.lb2 = o;
  o += k2;
  s.lb3 = o;
  o += k2;
  s.nm = o;
  o += k2;
  s.vs = o;
  o += k2;
  s.mu = o;
  o += k2;
  s.sig = o;
  o += k;
  s.cand = o;
  o += 3 * nt * k;
  s.cnt = o;
  o += 4;
  s.per = (o + 3) & ~3ll;
  return s;
}

namespace {

// ---------------------------------------------------------------------------------------
// k × k helpers (shared memory, all threads of the CTA)
// ---------------------------------------------------------------------------------------

// g = the sum of the nt partial Gram matrices at parts (tile t at parts + t·k²), in tile order.
// The parts were written by other CTAs of the same kernel: read them from L2, eight tiles of
// an element in flight at once.
__device__ void gram_sum(const float *parts, int nt, int k, float *g) {
  const int k2 = k * k;
  for (int e = threadIdx.x; e < k2; e += kThr) {
    float s = 0.f;
    for (int t0 = 0; t0 < nt; t0 += 8) {
      float v[8];
#pragma unroll
      for (int t = 0; t < 8; ++t)
        v[t] = t0 + t < nt ? __ldcg(parts + (long long)(t0 + t) * k2 + e) : 0.f;
#pragma unroll
      for (int t = 0; t < 8; ++t) s += v[t];
    }
    g[e] = s;
  }
  __syncthreads();
}

// Cholesky factor and its inverse together, in place on h (k × k, row-major, symmetric on
// entry), after adding 11 (M k + k (k + 1)) u trace(h) to the diagonal when shift_rows = M > 0.
// On return the lower triangle of h (with the diagonal) is L⁻¹, its strict upper triangle is
// Lᵀ, and d[j] = L[j][j]. A pivot that is not positive (or NaN) gives a zero column of L and a
// zero row of L⁻¹.
// Elimination by row operations: step j takes the pivot p = h[j][j] and, for every row i > j,
// f_i = h[j][i] / p (row j's trailing part equals column j by symmetry, and row j is not
// written during the step), then h[i][c] −= f_i h[j][c] over all columns c: for c < j that is
// L⁻¹'s row operation, for c > j the trailing update of the Gram matrix, and column j becomes
// L⁻¹'s −f_i. Row j is scaled by 1/√p one step later, when nothing reads it: its first j + 1
// entries become row j of L⁻¹ and the rest column j of L. Thread (column c, row group q) takes
// rows j + 1 + q, j + 1 + q + G, ... (G = 256 / k), so a step needs one barrier.
__device__ void chol_inverse(float *h, float *d, int k, int shift_rows) {
  const int tid = threadIdx.x;
  if (shift_rows > 0) {
    if (tid < 32) {
      float t = 0.f;
      for (int j = tid; j < k; j += 32) t += h[j * k + j];
      for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      const float s = 11.f * ((float)shift_rows * k + (float)k * (k + 1)) * 5.9604645e-8f * t;
      __syncwarp();
      for (int j = tid; j < k; j += 32) h[j * k + j] += s;
    }
    __syncthreads();
  }
  const int G = kThr / k;
  const int c = tid % k, q = tid / k;
  float prev = 0.f;
  for (int j = 0; j < k; ++j) {
    const float p = h[j * k + j];
    // 1/√p from the hardware reciprocal square root (a few ulp; the next CholeskyQR pass
    // absorbs it)
    const float iv = p > 0.f ? rsqrtf(p) : 0.f;
    const float ip = iv * iv;
    if (q < G) {
      const float hj = c == j ? 1.f : h[j * k + c];
      for (int i = j + 1 + q; i < k; i += G) {
        const float f = h[j * k + i] * ip;
        const float x = h[i * k + c];
        h[i * k + c] = c == j ? -f : fmaf(-f, hj, x);
      }
    }
    if (j > 0 && tid < k) h[(j - 1) * k + tid] = tid == j - 1 ? prev : h[(j - 1) * k + tid] * prev;
    if (tid == 0) d[j] = p > 0.f ? p * iv : 0.f;
    prev = iv;
    __syncthreads();
  }
  if (tid < k) h[(k - 1) * k + tid] = tid == k - 1 ? prev : h[(k - 1) * k + tid] * prev;
  __syncthreads();
}

// The factor step that ends a kernel writing a tall matrix. Every CTA has written its tile's
// partial Gram matrix; the CTA that counts last (of nt for this problem) adds them up,
// factors (with the shift when shift_rows > 0), stores L⁻ᵀ at li_out and, when l_out is
// given, L (lower triangle, zeros above), and resets the count for the next kernel. No CTA
// waits for another. g, li: k × k shared scratch; s_last: one shared int.
struct Factor {
  float *li_out, *l_out;
  int shift_rows;
};

__device__ void factor_if_last(const float *parts, int nt, int k, const Factor &f, int *cnt,
                               float *g, float *li, int *s_last) {
  const int tid = threadIdx.x;
  __threadfence();  // this CTA's partial Gram matrix, before its count
  __syncthreads();
  if (tid == 0) *s_last = atomicAdd(cnt, 1) == nt - 1;
  __syncthreads();
  if (!*s_last) return;
  __threadfence();
  gram_sum(parts, nt, k, g);
  chol_inverse(g, li, k, f.shift_rows);  // g: L⁻¹ below and on the diagonal, Lᵀ above; li: L's
                                          // diagonal
  for (int l = tid >> 5; l < k; l += kWarps)  // L⁻ᵀ: li_out[l·k + j] = L⁻¹[j][l]
    for (int j = tid & 31; j < k; j += 32) f.li_out[l * k + j] = l <= j ? g[j * k + l] : 0.f;
  if (f.l_out)  // L, zeros above the diagonal
    for (int i = tid >> 5; i < k; i += kWarps)
      for (int j = tid & 31; j < k; j += 32)
        f.l_out[i * k + j] = j < i ? g[j * k + i] : (j == i ? li[i] : 0.f);
  if (tid == 0) *cnt = 0;
}

// ---------------------------------------------------------------------------------------
// [128 × k] tile helpers (shared memory tile with row pitch P)
// ---------------------------------------------------------------------------------------

// gout (global, k × k, full) = Σ_r y[r]ᵀ y[r] over the first `rows` rows of the tile; scratch
// holds gram_subsets(k) · k² floats.
__device__ void tile_gram(const float *y, int P, int rows, int k, float *gout, float *scratch) {
  const int tid = threadIdx.x;
  const int nb = (k + 3) >> 2, nblk = nb * (nb + 1) / 2;
  const int S = gram_subsets(k);
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
      for (int z = 0; z < 4; ++z) acc[x][z] = 0.f;
    for (int r = sub; r < rows; r += S) {
      const float *row = y + r * P;
      float u[4], v[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        u[x] = i0 + x < k ? row[i0 + x] : 0.f;
        v[x] = j0 + x < k ? row[j0 + x] : 0.f;
      }
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int z = 0; z < 4; ++z) acc[x][z] = fmaf(u[x], v[z], acc[x][z]);
    }
    float *out = scratch + (long long)sub * k * k;
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int z = 0; z < 4; ++z)
        if (i0 + x < k && j0 + z < k) out[(i0 + x) * k + j0 + z] = acc[x][z];
  }
  __syncthreads();
  for (int i = tid >> 5; i < k; i += kWarps)
    for (int j = tid & 31; j < k; j += 32) {
      // below the block diagonal, the mirror entry was computed
      const bool lower = (i >> 2) > (j >> 2);
      const int e = lower ? j * k + i : i * k + j;
      float sum = 0.f;
      for (int sub = 0; sub < S; ++sub) sum += scratch[(long long)sub * k * k + e];
      gout[i * k + j] = sum;
    }
}

// Rows [0, rows) of a row-major [· × k] global matrix into the tile by cp.async, rows past
// `rows` zero. The caller commits the copies and waits for them.
__device__ void load_tile(const float *src, int rows, int k, float *y, int P) {
  for (int r = threadIdx.x >> 5; r < kRows; r += kWarps)
    for (int j = threadIdx.x & 31; j < k; j += 32) {
      if (r < rows)
        ptx::cp_async4(ptx::smem_addr(y + r * P + j), src + r * k + j);
      else
        y[r * P + j] = 0.f;
    }
}

// n floats from global memory into shared memory by cp.async (the caller commits and waits).
__device__ void load_vec(const float *src, int n, float *dst) {
  for (int e = threadIdx.x; e < n; e += kThr) ptx::cp_async4(ptx::smem_addr(dst + e), src + e);
}

// The first `rows` rows of the tile to global memory at dst (row stride k).
__device__ void store_tile(const float *y, int P, int rows, int k, float *dst) {
  for (int r = threadIdx.x >> 5; r < rows; r += kWarps)
    for (int j = threadIdx.x & 31; j < k; j += 32) dst[r * k + j] = y[r * P + j];
}

// dst tile = src tile · L⁻ᵀ (li[l·k + j] = L⁻¹[j][l]), all 128 rows. Thread (lane, warp) owns
// rows lane + 32i (i < 4) and the NC columns warp + 8c of its warp (NC = ⌈(k − warp) / 8⌉, a
// compile-time count so that no product slot is idle): each step over l reads four tile values
// and NC L⁻ᵀ values (the same for the whole warp) for 4·NC products.
template <int NC>
__device__ void apply_linv_cols(const float *src, float *dst, int P, int k, const float *li,
                                int rg, int cg) {
  float acc[4][NC];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < NC; ++c) acc[i][c] = 0.f;
  for (int l = 0; l < k; ++l) {
    float x[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = src[(rg + 32 * i) * P + l];
    const float *w = li + l * k + cg;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const float wc = w[8 * c];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i][c] = fmaf(x[i], wc, acc[i][c]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < NC; ++c) dst[(rg + 32 * i) * P + cg + 8 * c] = acc[i][c];
}

__device__ void apply_linv(const float *src, float *dst, int P, int k, const float *li) {
  const int rg = threadIdx.x & 31, cg = threadIdx.x >> 5;
  switch ((k - cg + 7) >> 3) {  // warp-uniform
    case 1: apply_linv_cols<1>(src, dst, P, k, li, rg, cg); break;
    case 2: apply_linv_cols<2>(src, dst, P, k, li, rg, cg); break;
    case 3: apply_linv_cols<3>(src, dst, P, k, li, rg, cg); break;
    case 4: apply_linv_cols<4>(src, dst, P, k, li, rg, cg); break;
    case 5: apply_linv_cols<5>(src, dst, P, k, li, rg, cg); break;
    case 6: apply_linv_cols<6>(src, dst, P, k, li, rg, cg); break;
    case 7: apply_linv_cols<7>(src, dst, P, k, li, rg, cg); break;
    case 8: apply_linv_cols<8>(src, dst, P, k, li, rg, cg); break;
    case 9: apply_linv_cols<9>(src, dst, P, k, li, rg, cg); break;
    case 10: apply_linv_cols<10>(src, dst, P, k, li, rg, cg); break;
    case 11: apply_linv_cols<11>(src, dst, P, k, li, rg, cg); break;
    case 12: apply_linv_cols<12>(src, dst, P, k, li, rg, cg); break;
    default: break;  // k − warp ≤ 0: no columns
  }
}

// ---------------------------------------------------------------------------------------
// products with Δ on the tensor cores
// ---------------------------------------------------------------------------------------

// C [M × k] tile rows [128·blockIdx.x, +128) of problem blockIdx.y:
//   TRANS = false: C = Δ X (M = T, K = W);  TRANS = true: C = Δᵀ X (M = W, K = T);
// X [K × k] row-major (row stride k). With li_in, the output is multiplied by that L⁻ᵀ (the
// folded third CholeskyQR pass of X). Each tile's partial Gram matrix goes to gparts; the last
// CTA of the problem factors their sum (`fac`).
struct ProdArgs {
  const float *delta;
  long long ld, delta_stride;
  const float *x;
  long long x_stride;
  float *c;           // per problem at c + i·ws_stride
  const float *li_in; // L⁻ᵀ to fold in, or null
  float *ly_out;      // tile 0 copies li_in here (or null)
  float *gparts;      // per-tile partial Gram matrices of C
  Factor fac;         // pointers of problem 0; the kernel adds i·ws_stride
  int *cnt;
  long long ws_stride;
  int n, T, W, k, kp;
};

struct ProdPlan {
  uint32_t stage, a_lo, b_hi, b_lo, g, li, bars, total;
};
// (bars: two stage barriers, then the TMEM address, the time-out flag and the last-CTA flag)

__host__ __device__ inline ProdPlan prod_plan(int k) {
  ProdPlan p;
  const int kp = pad16(k);
  p.a_lo = kRows * 128;
  p.b_hi = 2 * kRows * 128;
  p.b_lo = p.b_hi + kp * 128;
  p.stage = p.b_lo + kp * 128;  // a multiple of 1024
  p.g = 2 * p.stage;
  p.li = p.g + 4 * k * k;
  p.bars = (p.li + 4 * k * k + 15) & ~15u;
  p.total = p.bars + 64;
  return p;
}

template <bool TRANS, bool VEC>
__global__ void __launch_bounds__(kThr, 2) form_prod_kernel(const __grid_constant__ ProdArgs a) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  const uint32_t raw = ptx::smem_addr(smraw);
  const uint32_t s0 = (raw + 1023u) & ~1023u;
  unsigned char *sp = smraw + (s0 - raw);
  const int k = a.k, kp = a.kp;
  const ProdPlan P = prod_plan(k);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int prob = blockIdx.y, tile = blockIdx.x;
  const int M = TRANS ? a.W : a.T, K = TRANS ? a.T : a.W;
  const int m0 = tile * kRows, rows = min(kRows, M - m0);
  const float *D = a.delta + (long long)prob * a.delta_stride;
  const float *X = a.x + (long long)prob * a.x_stride;
  const long long wo = (long long)prob * a.ws_stride;
  float *g = reinterpret_cast<float *>(sp + P.g);
  float *li = reinterpret_cast<float *>(sp + P.li);
  const uint32_t bar = s0 + P.bars;  // two stage barriers
  volatile uint32_t *s_tmem = reinterpret_cast<volatile uint32_t *>(sp + P.bars + 16);
  volatile int *flag = reinterpret_cast<volatile int *>(sp + P.bars + 20);
  int *s_last = reinterpret_cast<int *>(sp + P.bars + 24);

  if (warp == 0) {
    ptx::tmem_alloc(s0 + P.bars + 16, 128);
    ptx::tmem_relinquish();
  }
  if (tid == 0) {
    ptx::mbar_init(bar, 1);
    ptx::mbar_init(bar + 8, 1);
    ptx::fence_mbar_init();
    *flag = 0;
  }
  if (a.li_in) load_vec(a.li_in + wo, k * k, li);  // the folded third pass: L⁻ᵀ of X's Gram
  ptx::cp_async_commit();
  ptx::cp_async_wait_all();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (a.li_in && tile == 0 && a.ly_out)
    for (int e = tid; e < k * k; e += kThr) a.ly_out[wo + e] = li[e];
  const uint32_t tmem = *s_tmem;

  // ---- staging: chunk c holds K columns [32c, 32c + 32) of A (128 rows) and of Bᵀ (kp rows).
  // Every thread loads four float4 of A:
  //   !TRANS: row f >> 3, 16-byte chunk f & 7 of that row (f = tid + 256 i);
  //   TRANS: A's rows are Δ's columns: K rows t0..t0+3 (t0 = 4·warp) of Δ at columns
  //   w0..w0+3 (w0 = 4·lane), turned in registers into four 16-byte chunks of A rows w0..w0+3.
  // Threads tb < 8·kp/4 load four float4 of X the same way (K rows 4·(tb / nq) + 0..3,
  // columns 4·(tb % nq) + 0..3, nq = kp / 4) and write four chunks of Bᵀ rows.
  const int nq = kp >> 2;
  const bool b_thread = tid < 8 * nq;
  const int bkg = b_thread ? tid / nq : 0, bq = b_thread ? tid - bkg * nq : 0;
  const bool xvec = (k & 3) == 0 && (reinterpret_cast<uintptr_t>(X) & 15u) == 0;
  auto ld4 = [](const float *src, int valid) {  // four floats, `valid` of them in range
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid > 0) v.x = __ldg(src);
    if (valid > 1) v.y = __ldg(src + 1);
    if (valid > 2) v.z = __ldg(src + 2);
    if (valid > 3) v.w = __ldg(src + 3);
    return v;
  };
  auto load = [&](int c, float4 *ra, float4 *rb) {
    const int k0 = c * kCk;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int gr, gc;  // Δ row and column of the float4's first element
      if (!TRANS) {
        const int f = tid + kThr * i;
        gr = m0 + (f >> 3);
        gc = k0 + 4 * (f & 7);
      } else {
        gr = k0 + 4 * warp + i;
        gc = m0 + 4 * lane;
      }
      const int nrow = TRANS ? K : M, ncol = TRANS ? M : K;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (gr < nrow) {
        const float *src = D + (long long)gr * a.ld + gc;
        if (VEC && gc + 3 < ncol)
          v = __ldg(reinterpret_cast<const float4 *>(src));
        else
          v = ld4(src, ncol - gc);
      }
      ra[i] = v;
    }
    if (b_thread) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kk = k0 + 4 * bkg + e, n = 4 * bq;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (kk < K) {
          const float *src = X + (long long)kk * k + n;
          if (xvec && n + 3 < k)
            v = __ldg(reinterpret_cast<const float4 *>(src));
          else
            v = ld4(src, k - n);
        }
        rb[e] = v;
      }
    }
  };
  auto split = [](float x, uint32_t &hi, uint32_t &lo) {
    hi = ptx::to_tf32(x);
    lo = ptx::to_tf32(x - __uint_as_float(hi));
  };
  auto comp = [](const float4 &v, int d) {  // component d of v
    return d == 0 ? v.x : d == 1 ? v.y : d == 2 ? v.z : v.w;
  };
  // the 16-byte chunk of row `row` holding K elements 4·kg..4·kg+3 (values q[0..3]), hi and lo
  auto put = [&](uint32_t base_hi, uint32_t base_lo, int row, int kg, const float *q) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) split(q[e], h[e], l[e]);
    const uint32_t o = row * 128 + ((kg ^ (row & 7)) << 4);
    sts16(base_hi + o, make_uint4(h[0], h[1], h[2], h[3]));
    sts16(base_lo + o, make_uint4(l[0], l[1], l[2], l[3]));
  };
  auto store = [&](int s, const float4 *ra, const float4 *rb) {
    const uint32_t st = s0 + s * P.stage;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (!TRANS) {  // row r, 16-byte chunk j of the 128-byte row
        const int f = tid + kThr * i;
        const float q[4] = {ra[i].x, ra[i].y, ra[i].z, ra[i].w};
        put(st, st + P.a_lo, f >> 3, f & 7, q);
      } else {  // row w0 + d takes component d of the four loaded rows; d turns with the lane
        const int d = (i + lane) & 3;
        const float q[4] = {comp(ra[0], d), comp(ra[1], d), comp(ra[2], d), comp(ra[3], d)};
        put(st, st + P.a_lo, 4 * lane + d, warp, q);
      }
    }
    if (b_thread) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int d = (i + bq) & 3;
        const float q[4] = {comp(rb[0], d), comp(rb[1], d), comp(rb[2], d), comp(rb[3], d)};
        put(st + P.b_hi, st + P.b_lo, 4 * bq + d, bkg, q);
      }
    }
  };
  const uint32_t idesc = ptx::idesc_tf32_f32(kRows, kp);
  auto issue = [&](int c) {
    const uint32_t st = s0 + (c & 1) * P.stage;
#pragma unroll
    for (int ks = 0; ks < kCk / 8; ++ks) {  // 8 tf32 = 32 bytes of K per MMA
      const uint64_t ah = ptx::smem_desc_sw128(st + ks * 32);
      const uint64_t al = ptx::smem_desc_sw128(st + P.a_lo + ks * 32);
      const uint64_t bh = ptx::smem_desc_sw128(st + P.b_hi + ks * 32);
      const uint64_t bl = ptx::smem_desc_sw128(st + P.b_lo + ks * 32);
      ptx::mma_tf32(tmem, al, bh, idesc, (c > 0 || ks > 0) ? 1u : 0u);
      ptx::mma_tf32(tmem, ah, bl, idesc, 1u);
      ptx::mma_tf32(tmem, ah, bh, idesc, 1u);
    }
    ptx::mma_commit(bar + 8 * (c & 1));
  };

  const int nc = (K + kCk - 1) / kCk;
  bool ok = true;
  float4 ra0[4], ra1[4], rb0[4], rb1[4];
  load(0, ra0, rb0);
  if (nc > 1) load(1, ra1, rb1);
  auto step = [&](int c, float4 *ra, float4 *rb) {
    const int s = c & 1;
    if (c >= 2 && !ptx::mbar_wait(bar + 8 * s, ((c - 2) >> 1) & 1, kWaitNsF)) ok = false;
    store(s, ra, rb);
    if (c + 2 < nc) load(c + 2, ra, rb);
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      ptx::tc_fence_after();
      issue(c);
    }
  };
  for (int c = 0; c < nc; c += 2) {
    step(c, ra0, rb0);
    if (c + 1 < nc) step(c + 1, ra1, rb1);
  }
  if (!ptx::mbar_wait(bar + 8 * ((nc - 1) & 1), ((nc - 1) >> 1) & 1, kWaitNsF)) ok = false;
  if (!ok) *flag = 1;
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const bool timed_out = *flag != 0;

  // ---- epilogue: TMEM rows -> (· L⁻ᵀ) -> output tile in the stage area
  const int Pt = tile_pitch(k);
  float *ct = reinterpret_cast<float *>(sp);
  float *scratch = ct + kRows * Pt;
  {
    const int r = ((warp & 3) << 5) + lane, h = warp >> 2;
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int half = kp >> 1;  // a multiple of 8
    for (int j0 = h * half; j0 < (h + 1) * half; j0 += 8) {
      float o[8];
      if (!a.li_in) {
        uint32_t v[8];
        ptx::tmem_ld8(trow + j0, v);
        ptx::tmem_ld_wait(v);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = __uint_as_float(v[e]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = 0.f;
        for (int l0 = 0; l0 < kp && l0 <= j0 + 7; l0 += 8) {
          uint32_t v[8];
          ptx::tmem_ld8(trow + l0, v);
          ptx::tmem_ld_wait(v);
#pragma unroll
          for (int l = 0; l < 8; ++l) {
            const int ll = l0 + l;
            if (ll < k) {
              const float xv = __uint_as_float(v[l]);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (j0 + e < k) o[e] = fmaf(xv, li[ll * k + j0 + e], o[e]);
            }
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (j0 + e < k) ct[r * Pt + j0 + e] = timed_out ? __int_as_float(0x7fc00000) : o[e];
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tmem, 128);
  store_tile(ct, Pt, rows, k, a.c + wo + (long long)m0 * k);
  tile_gram(ct, Pt, rows, k, a.gparts + wo + (long long)tile * k * k, scratch);
  Factor f = a.fac;
  f.li_out += wo;
  if (f.l_out) f.l_out += wo;
  factor_if_last(a.gparts + wo, gridDim.x, k, f, a.cnt + wo, g, li, s_last);
}

// ---------------------------------------------------------------------------------------
// one CholeskyQR pass over a tile, in place (CUDA cores)
// ---------------------------------------------------------------------------------------

struct PassArgs {
  float *x;            // [M × k] row-major, problem i at x + i·ws_stride
  const float *li_in;  // L⁻ᵀ of this pass (from the kernel before)
  float *gparts;       // partial Gram matrices of the result
  Factor fac;          // the next factor (pointers of problem 0)
  int *cnt;
  long long ws_stride;
  int n, M, k;
};

__host__ __device__ inline size_t pass_smem(int k) {
  return 4 * ((size_t)2 * kRows * tile_pitch(k) + (size_t)gram_subsets(k) * k * k + 2 * k * k) +
         16;
}

__global__ void __launch_bounds__(kThr, 2) form_pass_kernel(const __grid_constant__ PassArgs a) {
  extern __shared__ __align__(16) float fsm[];
  const int k = a.k, Pt = tile_pitch(k);
  const int prob = blockIdx.y, tile = blockIdx.x;
  const int m0 = tile * kRows, rows = min(kRows, a.M - m0);
  const long long wo = (long long)prob * a.ws_stride;
  float *xin = fsm, *xout = xin + kRows * Pt, *scratch = xout + kRows * Pt;
  float *g = scratch + gram_subsets(k) * k * k, *li = g + k * k;
  int *s_last = reinterpret_cast<int *>(li + k * k);
  float *x = a.x + wo + (long long)m0 * k;
  load_tile(x, rows, k, xin, Pt);
  load_vec(a.li_in + wo, k * k, li);
  ptx::cp_async_commit();
  ptx::cp_async_wait_all();
  __syncthreads();
  apply_linv(xin, xout, Pt, k, li);
  __syncthreads();
  store_tile(xout, Pt, rows, k, x);
  tile_gram(xout, Pt, rows, k, a.gparts + wo + (long long)tile * k * k, scratch);
  Factor f = a.fac;
  f.li_out += wo;
  if (f.l_out) f.l_out += wo;
  factor_if_last(a.gparts + wo, gridDim.x, k, f, a.cnt + wo, g, li, s_last);
}

// ---------------------------------------------------------------------------------------
// the small SVD and V_mᵀ (one CTA per problem)
// ---------------------------------------------------------------------------------------

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

// One-sided Jacobi on the columns of a [k × k] (column-major), rotations accumulated into
// v [k × k] (column-major, set to I here); pairs: (k + 1)² / 4 int2 of shared scratch for the
// round-robin schedule, computed once. Eight lanes own one pair for its whole rotation, so a
// warp turns four pairs at once; the pair's columns stay in registers from the dot products to
// the rotation. The rotation's parameters use the hardware reciprocal and reciprocal square
// root (a few ulp): any rotation with cs² + sn² = 1 to that accuracy serves, as the columns are
// orthogonalised, not the angles reproduced.
__device__ void jacobi_small(float *a, float *v, int k, int2 *pairs) {
  constexpr int G = 8, PW = 32 / G, E = (kMaxSketch + G - 1) / G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sub = lane % G, slot = lane / G;
  const int n = k + (k & 1), h = n / 2;  // an odd k plays a dummy column
  for (int e = tid; e < (n - 1) * h; e += kThr) {
    const int round = e / h, i = e - round * h;
    int p, q;
    rr_pair(n, round, i, p, q);
    pairs[e] = (p < k && q < k) ? make_int2(p, q) : make_int2(-1, -1);
  }
  for (int e = tid; e < k * k; e += kThr) v[e] = (e / k == e % k) ? 1.f : 0.f;
  __syncthreads();
  const float tol2 = (float)k * 1.1920929e-7f * 1.1920929e-7f;  // (√k·2⁻²³)²
  for (int sweep = 0; sweep < 30; ++sweep) {
    int rotated = 0;
    for (int round = 0; round < n - 1; ++round) {
      for (int i0 = PW * warp; i0 < h; i0 += PW * kWarps) {  // warp-uniform
        const int i = i0 + slot;
        const int2 pq = i < h ? pairs[round * h + i] : make_int2(-1, -1);
        const bool live = pq.x >= 0;
        float *x = a + (long long)(live ? pq.x : 0) * k, *y = a + (long long)(live ? pq.y : 0) * k;
        float xr[E], yr[E], al = 0.f, be = 0.f, ga = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int w = sub + G * e;
          xr[e] = (live && w < k) ? x[w] : 0.f;
          yr[e] = (live && w < k) ? y[w] : 0.f;
        }
#pragma unroll
        for (int e = 0; e < E; ++e) {
          al = fmaf(xr[e], xr[e], al);
          be = fmaf(yr[e], yr[e], be);
          ga = fmaf(xr[e], yr[e], ga);
        }
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) {
          al += __shfl_xor_sync(0xffffffffu, al, o);
          be += __shfl_xor_sync(0xffffffffu, be, o);
          ga += __shfl_xor_sync(0xffffffffu, ga, o);
        }
        // |γ| > tol·√(αβ): not yet orthogonal (a zero column never is rotated)
        if (live && ga * ga > tol2 * al * be) {
          const float zeta = (be - al) * __frcp_rn(2.f * ga);
          const float t =
              copysignf(1.f, zeta) * __frcp_rn(fabsf(zeta) + sqrtf(fmaf(zeta, zeta, 1.f)));
          const float cs = rsqrtf(fmaf(t, t, 1.f)), sn = cs * t;
          float *vx = v + (long long)pq.x * k, *vy = v + (long long)pq.y * k;
          float vxr[E], vyr[E];
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const int w = sub + G * e;
            vxr[e] = w < k ? vx[w] : 0.f;
            vyr[e] = w < k ? vy[w] : 0.f;
          }
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const int w = sub + G * e;
            if (w < k) {
              x[w] = cs * xr[e] - sn * yr[e];
              y[w] = sn * xr[e] + cs * yr[e];
              vx[w] = cs * vxr[e] - sn * vyr[e];
              vy[w] = sn * vxr[e] + cs * vyr[e];
            }
          }
          rotated = 1;
        }
      }
      __syncthreads();
    }
    if (!__syncthreads_or(rotated)) break;
  }
}

struct SvdArgs {
  const float *lb1, *lb2, *lb3;  // Bᵀ's CholeskyQR factors (lower, zeros above)
  const float *li3;              // L3⁻ᵀ
  float *nm;                     // out: N = L3⁻ᵀ U_R[:, order] [k × m]
  float *vs;                     // out: Ũ[:, order] [k × m]
  float *sig;                    // out: σ in order [m]
  long long ws_stride;           // per problem, for all of the above
  int n, k, m;
};

__host__ __device__ inline size_t svd_smem(int k) {
  return 4 * ((size_t)4 * k * k + 2 * k + 8) + 8 * (size_t)((k + 1) / 2) * (k + 1);
}

__global__ void __launch_bounds__(kThr, 1) form_svd_kernel(const __grid_constant__ SvdArgs a) {
  extern __shared__ __align__(16) float fsm[];
  const int k = a.k, m = a.m;
  const int prob = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long wo = (long long)prob * a.ws_stride;
  float *r = fsm, *v = r + k * k, *t1 = v + k * k, *l3 = t1 + k * k;
  float *nrm = l3 + k * k;
  int *order = reinterpret_cast<int *>(nrm + k);
  int2 *pairs = reinterpret_cast<int2 *>(fsm + ((4 * k * k + 2 * k + 8 + 1) & ~1));
  const float *L1 = r, *L2 = v;  // staged where R_B and Ṽ go later
  load_vec(a.lb1 + wo, k * k, r);
  load_vec(a.lb2 + wo, k * k, v);
  load_vec(a.lb3 + wo, k * k, l3);
  ptx::cp_async_commit();
  ptx::cp_async_wait_all();
  __syncthreads();
  // R_B = L3ᵀ (L2ᵀ L1ᵀ), column-major in r; t1 = L2ᵀ L1ᵀ, t1[i][j] = Σ_l L2[l][i] L1[j][l]
  for (int e = tid; e < k * k; e += kThr) {
    const int i = e / k, j = e - i * k;
    float s = 0.f;
    for (int l = i; l <= j; ++l) s = fmaf(L2[l * k + i], L1[j * k + l], s);
    t1[e] = s;
  }
  __syncthreads();
  for (int e = tid; e < k * k; e += kThr) {  // R[i][j] = Σ_{l ≥ i} L3[l][i] t1[l][j]
    const int j = e / k, i = e - j * k;
    float s = 0.f;
    for (int l = i; l <= j; ++l) s = fmaf(l3[l * k + i], t1[l * k + j], s);
    r[e] = s;
  }
  __syncthreads();
  jacobi_small(r, v, k, pairs);

  // σ_j = ‖column j‖, then the columns by σ (descending, ties by column index)
  for (int j = warp; j < k; j += kWarps) {
    float s = 0.f;
    for (int w = lane; w < k; w += 32) s = fmaf(r[j * k + w], r[j * k + w], s);
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
  // N = L3⁻ᵀ U_R[:, order] (U_R's column c = R_B Ṽ's column c / σ_c, zero when σ_c = 0), the
  // kept columns of Ũ, and σ
  float *li3 = t1;
  load_vec(a.li3 + wo, k * k, li3);
  ptx::cp_async_commit();
  ptx::cp_async_wait_all();
  __syncthreads();
  for (int e = tid; e < k * m; e += kThr) {
    const int i = e / m, jj = e - i * m;
    const int c = order[jj];
    const float sg = nrm[c];
    const float inv = sg > 0.f ? 1.f / sg : 0.f;
    float s = 0.f;
    for (int l = i; l < k; ++l) s = fmaf(li3[i * k + l], r[c * k + l], s);
    a.nm[wo + e] = s * inv;
    a.vs[wo + e] = v[c * k + i];
  }
  for (int j = tid; j < m; j += kThr) a.sig[wo + j] = nrm[order[j]];
}

// ---------------------------------------------------------------------------------------
// V_mᵀ = (B₂ N)ᵀ over tiles of W, signed by the last CTA of each problem
// ---------------------------------------------------------------------------------------

struct VArgs {
  const float *b2;      // Bᵀ after two passes [W × k]
  const float *nm, *vs, *sig, *ly;  // from the SVD kernel; L⁻ᵀ of the T-side third pass
  float *cand;          // per tile and column: largest magnitude, its row, its value
  float *mu;            // out: [k × m], U·Σ = Y₂ · mu
  int *cnt;
  long long ws_stride;  // per problem, for all of the above
  __nv_bfloat16 *vt;    // out: V_mᵀ [m × W] at vt + i·vt_stride
  long long vt_stride;
  float *sigma;         // out: [n][m] or null
  int n, W, k, m;
};

__host__ __device__ inline size_t v_smem(int k, int m) {
  return 4 * ((size_t)kRows * tile_pitch(k) + (size_t)k * m + (size_t)m * (kRows + 1) + m + 8);
}

__global__ void __launch_bounds__(kThr, 1) form_v_kernel(const __grid_constant__ VArgs a) {
  extern __shared__ __align__(16) float fsm[];
  const int k = a.k, m = a.m, W = a.W, Pt = tile_pitch(k);
  const int prob = blockIdx.y, tile = blockIdx.x, tid = threadIdx.x, warp = tid >> 5,
            lane = tid & 31;
  const int w0 = tile * kRows, rows = min(kRows, W - w0);
  const long long wo = (long long)prob * a.ws_stride;
  float *bt = fsm, *N = bt + kRows * Pt, *vtile = N + k * m, *sgn = vtile + m * (kRows + 1);
  int *s_last = reinterpret_cast<int *>(sgn + m);
  load_tile(a.b2 + wo + (long long)w0 * k, rows, k, bt, Pt);
  load_vec(a.nm + wo, k * m, N);
  ptx::cp_async_commit();
  ptx::cp_async_wait_all();
  __syncthreads();
  // V_B rows of the tile: thread (row, column half), rows along lanes
  __nv_bfloat16 *vt = a.vt + (long long)prob * a.vt_stride;
  {
    const int rr = tid & (kRows - 1);
    for (int j = tid >> 7; j < m; j += 2) {
      float s = 0.f;
      for (int i = 0; i < k; ++i) s = fmaf(bt[rr * Pt + i], N[i * m + j], s);
      vtile[j * (kRows + 1) + rr] = s;
      if (rr < rows) vt[(long long)j * W + w0 + rr] = __float2bfloat16_rn(s);
    }
  }
  __syncthreads();
  // each column's entry of largest magnitude in the tile (the first row on a tie)
  float *cand = a.cand + wo + (long long)tile * 3 * m;
  for (int j = warp; j < m; j += kWarps) {
    float mb = -1.f, vb = 0.f;
    int ib = 0x7fffffff;
    for (int rr = lane; rr < rows; rr += 32) {  // rows grow along a lane: keep its first
      const float x = vtile[j * (kRows + 1) + rr];
      if (fabsf(x) > mb) {
        mb = fabsf(x);
        vb = x;
        ib = w0 + rr;
      }
    }
    for (int o = 16; o > 0; o >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, mb, o);
      const float ov = __shfl_xor_sync(0xffffffffu, vb, o);
      const int oi = __shfl_xor_sync(0xffffffffu, ib, o);
      if (om > mb || (om == mb && oi < ib)) {
        mb = om;
        vb = ov;
        ib = oi;
      }
    }
    if (lane == 0) {
      cand[3 * j] = mb;
      cand[3 * j + 1] = __int_as_float(ib);
      cand[3 * j + 2] = vb;
    }
  }
  // the last CTA of the problem: signs over all tiles (tile order; the first row on a tie),
  // rows of V_mᵀ flipped where the sign is negative (exact on bf16), U·Σ's map and σ
  __threadfence();
  __syncthreads();
  if (tid == 0) *s_last = atomicAdd(a.cnt + wo, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!*s_last) return;
  __threadfence();
  const float *call = a.cand + wo;
  for (int j = tid; j < m; j += kThr) {
    float mb = -1.f, vb = 0.f;
    int ib = 0x7fffffff;
    for (int t = 0; t < (int)gridDim.x; ++t) {
      const float cm = __ldcg(call + (long long)t * 3 * m + 3 * j);
      const int ci = __float_as_int(__ldcg(call + (long long)t * 3 * m + 3 * j + 1));
      if (cm > mb || (cm == mb && ci < ib)) {
        mb = cm;
        ib = ci;
        vb = __ldcg(call + (long long)t * 3 * m + 3 * j + 2);
      }
    }
    sgn[j] = vb < 0.f ? -1.f : 1.f;
  }
  __syncthreads();
  for (int j = warp; j < m; j += kWarps) {
    if (sgn[j] < 0.f) {
      unsigned short *row = reinterpret_cast<unsigned short *>(vt + (long long)j * W);
      for (int w = lane; w < W; w += 32) row[w] = __ldcg(row + w) ^ 0x8000u;
    }
  }
  float *ly = bt, *vs = vtile;  // the tiles are done with
  load_vec(a.ly + wo, k * k, ly);
  load_vec(a.vs + wo, k * m, vs);
  ptx::cp_async_commit();
  ptx::cp_async_wait_all();
  __syncthreads();
  for (int e = tid; e < k * m; e += kThr) {
    const int i = e / m, j = e - i * m;
    float s = 0.f;
    for (int l = i; l < k; ++l) s = fmaf(ly[i * k + l], vs[l * m + j], s);
    a.mu[wo + e] = s * sgn[j] * a.sig[wo + j];
  }
  if (a.sigma)
    for (int j = tid; j < m; j += kThr) a.sigma[(long long)prob * m + j] = a.sig[wo + j];
  if (tid == 0) a.cnt[wo] = 0;
}

// ---------------------------------------------------------------------------------------
// U·Σ = Y₂ · mu over tiles of T
// ---------------------------------------------------------------------------------------

struct UArgs {
  const float *y;  // Y₂ [T × k], problem i at + i·ws_stride
  const float *mu; // [k × m]
  long long ws_stride;
  __nv_bfloat16 *u;  // U·Σ [T × m] at u + i·u_stride
  long long u_stride;
  int n, T, k, m;
};

__host__ __device__ inline size_t u_smem(int k, int m) {
  return 4 * ((size_t)kRows * tile_pitch(k) + (size_t)k * m);
}

__global__ void __launch_bounds__(kThr, 1) form_u_kernel(const __grid_constant__ UArgs a) {
  extern __shared__ __align__(16) float fsm[];
  const int k = a.k, m = a.m, Pt = tile_pitch(k);
  const int prob = blockIdx.y, tile = blockIdx.x, tid = threadIdx.x;
  const int t0 = tile * kRows, rows = min(kRows, a.T - t0);
  const long long wo = (long long)prob * a.ws_stride;
  float *yt = fsm, *mu = yt + kRows * Pt;
  load_tile(a.y + wo + (long long)t0 * k, rows, k, yt, Pt);
  load_vec(a.mu + wo, k * m, mu);
  ptx::cp_async_commit();
  ptx::cp_async_wait_all();
  __syncthreads();
  const int S = kThr / m, jj = tid % m, part = tid / m;
  if (part >= S) return;
  __nv_bfloat16 *u = a.u + (long long)prob * a.u_stride + (long long)t0 * m;
  for (int rr = part; rr < rows; rr += S) {
    float s = 0.f;
    for (int i = 0; i < k; ++i) s = fmaf(yt[rr * Pt + i], mu[i * m + jj], s);
    u[(long long)rr * m + jj] = __float2bfloat16_rn(s);
  }
}

size_t prod_smem(int k) { return (size_t)prod_plan(k).total + 1024; }

int g_form_configured[64] = {0};  // per device: the kernels' dynamic shared-memory limit
std::mutex g_form_mu;

template <typename K>
cudaError_t allow_smem(K kernel, int optin) {
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, kernel);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
}

// Once per device: the kernels are loaded and may use the device's opt-in shared memory.
cudaError_t configure_form(int dev) {
  std::lock_guard<std::mutex> lock(g_form_mu);
  if (g_form_configured[dev]) return cudaSuccess;
  int optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess) e = allow_smem(form_prod_kernel<false, false>, optin);
  if (e == cudaSuccess) e = allow_smem(form_prod_kernel<false, true>, optin);
  if (e == cudaSuccess) e = allow_smem(form_prod_kernel<true, false>, optin);
  if (e == cudaSuccess) e = allow_smem(form_prod_kernel<true, true>, optin);
  if (e == cudaSuccess) e = allow_smem(form_pass_kernel, optin);
  if (e == cudaSuccess) e = allow_smem(form_svd_kernel, optin);
  if (e == cudaSuccess) e = allow_smem(form_v_kernel, optin);
  if (e == cudaSuccess) e = allow_smem(form_u_kernel, optin);
  if (e != cudaSuccess) return e;
  g_form_configured[dev] = optin;
  return cudaSuccess;
}

}  // namespace

size_t form_patch_workspace(long long n, int T, int W, int k) {
  return (size_t)n * (size_t)form_ws(T, W, k).per * sizeof(float);
}

size_t form_patch_smem(int k) {
  size_t s = prod_smem(k);
  const size_t o[4] = {pass_smem(k), svd_smem(k), v_smem(k, k), u_smem(k, k)};
  for (size_t x : o) s = s > x ? s : x;
  return s;
}

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
  e = configure_form(dev);
  if (e != cudaSuccess) return e;
  if ((size_t)g_form_configured[dev] < form_patch_smem(a.k)) return cudaErrorInvalidValue;
  if (a.n == 0) return cudaSuccess;
  const int T = a.T, W = a.W, k = a.k, n = a.n;
  const FormWs L = form_ws(T, W, k);
  float *ws = a.work;
  float *bt = ws + L.t, *bw = ws + L.w;
  float *li[2] = {ws + L.li0, ws + L.li1};
  int *cnt = reinterpret_cast<int *>(ws + L.cnt);
  const bool vec = (reinterpret_cast<uintptr_t>(a.delta) & 15u) == 0 && (a.ld & 3) == 0 &&
                   (a.delta_stride & 3) == 0;
  // the finished-CTA counts start at zero (every last CTA puts its count back to zero)
  e = cudaMemset2DAsync(cnt, (size_t)L.per * sizeof(float), 0, 4 * sizeof(int), n, s);
  if (e != cudaSuccess) return e;

  int cur = 0;  // the L⁻ᵀ slot the next kernel reads; the factor step writes the other
  auto fac = [&](int shift_rows, float *l_out) {
    Factor f;
    f.li_out = li[cur ^ 1];
    f.l_out = l_out;
    f.shift_rows = shift_rows;
    return f;
  };
  // products with Δ: C = Δ X (trans = false) or Δᵀ X; with fold, · L⁻ᵀ of the slot `cur`
  auto prod = [&](bool trans, const float *x, long long x_stride, float *c, bool fold,
                  float *ly_out, int shift_rows, float *l_out) -> cudaError_t {
    ProdArgs p;
    p.delta = a.delta;
    p.ld = a.ld;
    p.delta_stride = a.delta_stride;
    p.x = x;
    p.x_stride = x_stride;
    p.c = c;
    p.li_in = fold ? li[cur] : nullptr;
    p.ly_out = ly_out;
    p.gparts = ws + L.g;
    p.fac = fac(shift_rows, l_out);
    p.cnt = cnt;
    p.ws_stride = L.per;
    p.n = n;
    p.T = T;
    p.W = W;
    p.k = k;
    p.kp = pad16(k);
    const dim3 grid(ntiles(trans ? W : T), n);
    const size_t smem = prod_smem(k);
    if (trans) {
      if (vec)
        form_prod_kernel<true, true><<<grid, kThr, smem, s>>>(p);
      else
        form_prod_kernel<true, false><<<grid, kThr, smem, s>>>(p);
    } else {
      if (vec)
        form_prod_kernel<false, true><<<grid, kThr, smem, s>>>(p);
      else
        form_prod_kernel<false, false><<<grid, kThr, smem, s>>>(p);
    }
    cur ^= 1;
    return cudaGetLastError();
  };
  // one CholeskyQR pass in place over x [M × k], by the factor in slot `cur`
  auto pass = [&](float *x, int M, int shift_rows, float *l_out) -> cudaError_t {
    PassArgs p;
    p.x = x;
    p.li_in = li[cur];
    p.gparts = ws + L.g;
    p.fac = fac(shift_rows, l_out);
    p.cnt = cnt;
    p.ws_stride = L.per;
    p.n = n;
    p.M = M;
    p.k = k;
    form_pass_kernel<<<dim3(ntiles(M), n), kThr, pass_smem(k), s>>>(p);
    cur ^= 1;
    return cudaGetLastError();
  };
  // Y = Δ Ω and its shifted factor; two explicit passes (the third factor is folded into the
  // next product)
  if (e == cudaSuccess) e = prod(false, a.omega, a.omega_stride, bt, false, nullptr, T, nullptr);
  if (e == cudaSuccess) e = pass(bt, T, 0, nullptr);
  if (e == cudaSuccess) e = pass(bt, T, 0, nullptr);
  for (int it = 0; it < a.q && e == cudaSuccess; ++it) {
    e = prod(true, bt, L.per, bw, true, nullptr, W, nullptr);  // Z = Δᵀ Q
    if (e == cudaSuccess) e = pass(bw, W, 0, nullptr);
    if (e == cudaSuccess) e = pass(bw, W, 0, nullptr);
    if (e == cudaSuccess) e = prod(false, bw, L.per, bt, true, nullptr, T, nullptr);  // Y = Δ Z
    if (e == cudaSuccess) e = pass(bt, T, 0, nullptr);
    if (e == cudaSuccess) e = pass(bt, T, 0, nullptr);
  }
  // Bᵀ = Δᵀ Q (Q's L⁻ᵀ kept for U·Σ) and two passes of its QR, keeping the three factors
  if (e == cudaSuccess) e = prod(true, bt, L.per, bw, true, ws + L.ly, W, ws + L.lb1);
  if (e == cudaSuccess) e = pass(bw, W, 0, ws + L.lb2);
  if (e == cudaSuccess) e = pass(bw, W, 0, ws + L.lb3);
  if (e != cudaSuccess) return e;
  SvdArgs sv;
  sv.lb1 = ws + L.lb1;
  sv.lb2 = ws + L.lb2;
  sv.lb3 = ws + L.lb3;
  sv.li3 = li[cur];
  sv.nm = ws + L.nm;
  sv.vs = ws + L.vs;
  sv.sig = ws + L.sig;
  sv.ws_stride = L.per;
  sv.n = n;
  sv.k = k;
  sv.m = a.m;
  form_svd_kernel<<<n, kThr, svd_smem(k), s>>>(sv);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  VArgs va;
  va.b2 = bw;
  va.nm = ws + L.nm;
  va.vs = ws + L.vs;
  va.sig = ws + L.sig;
  va.ly = ws + L.ly;
  va.cand = ws + L.cand;
  va.mu = ws + L.mu;
  va.cnt = cnt;
  va.ws_stride = L.per;
  va.vt = a.vt;
  va.vt_stride = a.vt_stride;
  va.sigma = a.sigma;
  va.n = n;
  va.W = W;
  va.k = k;
  va.m = a.m;
  form_v_kernel<<<dim3(ntiles(W), n), kThr, v_smem(k, a.m), s>>>(va);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  UArgs ua;
  ua.y = bt;
  ua.mu = ws + L.mu;
  ua.ws_stride = L.per;
  ua.u = a.u;
  ua.u_stride = a.u_stride;
  ua.n = n;
  ua.T = T;
  ua.k = k;
  ua.m = a.m;
  form_u_kernel<<<dim3(ntiles(T), n), kThr, u_smem(k, a.m), s>>>(ua);
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
// also makes CUDA load this file's device code, which reserves the array) and the kernels,
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
