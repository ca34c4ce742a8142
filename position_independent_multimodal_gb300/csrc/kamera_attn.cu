// Decode attention over the paged pool: the consumer of the rows the reuse, relocation and
// re-anchoring calls write. One query token per (request, query head):
//   s_t = scale * q . K_t,  o = sum_t softmax(s)_t V_t,  lse = log sum_t exp(s_t)
// over the request's logical tokens, gathered through its page-table row.
//
// The context is cut into splits of 256 tokens. attn_split_kernel computes each split's
// normalised output and log-sum-exp independently; attn_merge_kernel combines the splits by
// their softmax mass, the log-sum-exp merge the Kamera page uses to argue that attention over
// KV(A) || KV(B) equals attending each part and merging (§1: o = (1 - mu) o_B + mu o_A).
//
// attn_split_kernel: one CTA of 256 threads per (split, group of <= 8 query heads sharing a KV
// head, request). Scores: thread t owns token t of the split, streams its K row (16-byte
// loads, eight in flight) and forms the dots with the group's queries held in shared memory.
// The softmax statistics are CTA reductions. P·V: each thread owns an 8-column chunk of V and
// a subset of the tokens (a warp reads whole V rows; eight rows in flight per thread), with
// the partial sums reduced through shared memory.
// Float32 throughout; the bf16 K and V are read once per (split, query group).
#include <mutex>

#include "kamera_dev.cuh"
#include "kamera_ptx.cuh"
#include "kamera_smem.cuh"

namespace kamera {

namespace {

constexpr int kThr = 256;
constexpr int kSplit = 256;  // tokens per split: one token per thread in the score pass
constexpr int kGq = 8;       // query heads per CTA (a multiple of 4)
constexpr int kBatch = 8;    // 16-byte loads a thread keeps in flight

// Byte offsets of the split kernel's dynamic shared memory.
struct AttnPlan {
  int q;      // f32x2 [kGq][dk / 2]: the group's queries, dims paired
  int p;      // float [kSplit][kGq]: scores, then exp(s - m), token-major
  int slot;   // long long [kSplit]: pool slot of each token, -1 when left out
  int red;    // float [TL / 2][kGq][dv]: partial P·V sums, two token lanes per warp added
  int stat;   // float [2][kGq] (m, l) and [kGq][kThr / 32] warp partials
  int total;
};

__host__ __device__ inline int attn_lanes(int dv) { return kThr / (dv / 8); }

// Whether a warp holds two token lanes of the same columns (8-column chunks a power of two
// up to 16), so that the pair is added by a shuffle before the shared-memory reduction.
__host__ __device__ inline bool attn_pairs(int dv) {
  const int chunks = dv / 8;
  return chunks <= 16 && (chunks & (chunks - 1)) == 0;
}

__host__ __device__ inline AttnPlan attn_plan(int dk, int dv) {
  AttnPlan p;
  const int lanes = attn_lanes(dv);
  const int rl = attn_pairs(dv) ? lanes / 2 : lanes;
  int o = 0;
  p.q = o;
  o += kGq * dk * 4;
  p.p = o;
  o += kGq * kSplit * 4;
  p.slot = o;
  o += kSplit * 8;
  p.red = o;
  o += rl * kGq * dv * 4;
  p.stat = o;
  o += (2 * kGq + kGq * (kThr / 32)) * 4;
  p.total = o;
  return p;
}

// The query heads of a CTA and where their K and V columns sit in the pool rows.
struct QGroup {
  int h0, n;          // first query head and how many (<= kGq)
  int kcol, vcol;     // first column of K in a K row, of V in a V row (MLA: in the K row)
};

__device__ __forceinline__ QGroup qgroup(const AttnArgs &a, int y) {
  const DevLayout &l = a.lay;
  const int n_kv = l.kind == KAMERA_GQA ? l.H : 1;
  const int group = a.hq / n_kv;
  const int cpk = (group + kGq - 1) / kGq;
  const int kvh = y / cpk, j = y - kvh * cpk;
  QGroup g;
  g.h0 = kvh * group + j * kGq;
  g.n = min(kGq, group - j * kGq);
  g.kcol = l.kind == KAMERA_GQA ? kvh * l.hd : 0;
  g.vcol = g.kcol;
  return g;
}

__global__ void __launch_bounds__(kThr, 2) attn_split_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const AttnPlan P = attn_plan(a.dk, a.dv);
  f32x2 *qs = reinterpret_cast<f32x2 *>(smem + P.q);
  float *ps = reinterpret_cast<float *>(smem + P.p);
  long long *slots = reinterpret_cast<long long *>(smem + P.slot);
  float *red = reinterpret_cast<float *>(smem + P.red);
  float *stat = reinterpret_cast<float *>(smem + P.stat);  // m[kGq], l[kGq], warp partials
  const DevLayout &lay = a.lay;
  const int split = blockIdx.x, r = blockIdx.z, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int ctx = a.ctx_len[r];
  if (ctx < 0 || ctx > a.max_ctx) {
    if (split == 0 && blockIdx.y == 0 && tid == 0) atomicOr(a.status, KAMERA_DEVICE_BAD_ITEM);
    return;
  }
  const int s0 = split * kSplit;
  if (s0 >= ctx) return;  // the merge reads only the splits that hold tokens
  const int n = min(kSplit, ctx - s0);
  const QGroup qg = qgroup(a, blockIdx.y);  // a.split == kSplit on this path
  const int dk = a.dk, dv = a.dv, G = qg.n;
  const int dk2 = dk >> 1;

  const __nv_bfloat16 *q = a.q + ((long long)r * a.hq + qg.h0) * dk;
  for (int e = tid; e < kGq * dk2; e += kThr) {  // heads past G are zero
    const int g = e / dk2, d = 2 * (e - g * dk2);
    qs[e] = g < G ? f2(__bfloat162float(q[g * dk + d]), __bfloat162float(q[g * dk + d + 1]))
                  : f2(0.f, 0.f);
  }
  if (tid < n)
    slots[tid] = slot_of(a.pool, lay.page_size, r, (long long)s0 + tid, a.status);
  __syncthreads();

  // scores: thread t owns token t; dims in pairs, q read as 16-byte broadcasts
  f32x2 acc2[kGq];
#pragma unroll
  for (int g = 0; g < kGq; ++g) acc2[g] = f2(0.f, 0.f);
  const long long slot = tid < n ? slots[tid] : -1;
  if (slot >= 0) {
    const __nv_bfloat16 *krow =
        a.pool.k + ((long long)a.layer * a.pool.num_slots + slot) * lay.row_k + qg.kcol;
    for (int d0 = 0; d0 < dk; d0 += 8 * kBatch) {  // kBatch 16-byte loads in flight
      uint4 buf[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (d0 + 8 * j < dk) buf[j] = __ldg(reinterpret_cast<const uint4 *>(krow + d0 + 8 * j));
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (d0 + 8 * j >= dk) break;
        const f32x2 x0 = bf2_to_f2(buf[j].x), x1 = bf2_to_f2(buf[j].y);
        const f32x2 x2 = bf2_to_f2(buf[j].z), x3 = bf2_to_f2(buf[j].w);
        const int pair = (d0 + 8 * j) >> 1;
#pragma unroll
        for (int g = 0; g < kGq; ++g) {
          const ulonglong2 qa = *reinterpret_cast<const ulonglong2 *>(qs + g * dk2 + pair);
          const ulonglong2 qb = *reinterpret_cast<const ulonglong2 *>(qs + g * dk2 + pair + 2);
          acc2[g] = fma2(qa.x, x0, acc2[g]);
          acc2[g] = fma2(qa.y, x1, acc2[g]);
          acc2[g] = fma2(qb.x, x2, acc2[g]);
          acc2[g] = fma2(qb.y, x3, acc2[g]);
        }
      }
    }
  }
  const float neg_inf = -__int_as_float(0x7f800000);
  float sc[kGq];
#pragma unroll
  for (int g = 0; g < kGq; ++g) {
    float lo, hi;
    f2_split(acc2[g], lo, hi);
    sc[g] = slot >= 0 && g < G ? (lo + hi) * a.scale : neg_inf;
  }
  // softmax statistics per query head: m = max_t s_t, then l = sum_t exp(s_t - m)
  float *m = stat, *l = stat + kGq, *wp = stat + 2 * kGq;
#pragma unroll
  for (int g = 0; g < kGq; ++g) {
    float w = sc[g];
    for (int o = 16; o > 0; o >>= 1) w = fmaxf(w, __shfl_xor_sync(0xffffffffu, w, o));
    if (lane == 0) wp[g * (kThr / 32) + warp] = w;
  }
  __syncthreads();
  if (tid < kGq) {
    float w = neg_inf;
    for (int i = 0; i < kThr / 32; ++i) w = fmaxf(w, wp[tid * (kThr / 32) + i]);
    m[tid] = w;
  }
  __syncthreads();
  float ex[kGq];
#pragma unroll
  for (int g = 0; g < kGq; ++g) {
    ex[g] = (slot >= 0 && g < G && m[g] > neg_inf) ? expf(sc[g] - m[g]) : 0.f;
    float w = ex[g];
    for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
    if (lane == 0) wp[g * (kThr / 32) + warp] = w;
  }
  {
    float4 *pt = reinterpret_cast<float4 *>(ps + tid * kGq);
#pragma unroll
    for (int g4 = 0; g4 < kGq; g4 += 4)
      pt[g4 / 4] = make_float4(ex[g4], ex[g4 + 1], ex[g4 + 2], ex[g4 + 3]);
  }
  __syncthreads();
  if (tid < kGq) {
    float w = 0.f;
    for (int i = 0; i < kThr / 32; ++i) w += wp[tid * (kThr / 32) + i];
    l[tid] = w;
  }

  // P·V: thread (c, tl) owns columns [8c, 8c + 8) and tokens tl, tl + TL, ...
  const int chunks = dv >> 3, lanes = kThr / chunks;
  const int c = tid % chunks, tl = tid / chunks;
  f32x2 o8[kGq][4];
#pragma unroll
  for (int g = 0; g < kGq; ++g)
#pragma unroll
    for (int e = 0; e < 4; ++e) o8[g][e] = f2(0.f, 0.f);
  const __nv_bfloat16 *vbase;
  long long vrow;
  if (lay.kind == KAMERA_GQA) {
    vbase = a.pool.v + (long long)a.layer * a.pool.num_slots * lay.row_v + qg.vcol + 8 * c;
    vrow = lay.row_v;
  } else {
    vbase = a.pool.k + (long long)a.layer * a.pool.num_slots * lay.row_k + 8 * c;
    vrow = lay.row_k;
  }
  if (tl < lanes) {
    for (int t0 = tl; t0 < n; t0 += lanes * kBatch) {  // kBatch rows in flight
      uint4 buf[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int t = t0 + j * lanes;
        const long long st = t < n ? slots[t] : -1;
        if (st >= 0) buf[j] = __ldg(reinterpret_cast<const uint4 *>(vbase + st * vrow));
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int t = t0 + j * lanes;
        if (t >= n || slots[t] < 0) continue;
        const f32x2 x0 = bf2_to_f2(buf[j].x), x1 = bf2_to_f2(buf[j].y);
        const f32x2 x2 = bf2_to_f2(buf[j].z), x3 = bf2_to_f2(buf[j].w);
        float pg[kGq];
#pragma unroll
        for (int g4 = 0; g4 < kGq; g4 += 4) {
          const float4 p4 = *reinterpret_cast<const float4 *>(ps + t * kGq + g4);
          pg[g4] = p4.x;
          pg[g4 + 1] = p4.y;
          pg[g4 + 2] = p4.z;
          pg[g4 + 3] = p4.w;
        }
#pragma unroll
        for (int g = 0; g < kGq; ++g) {
          const f32x2 pp = f2(pg[g], pg[g]);
          o8[g][0] = fma2(pp, x0, o8[g][0]);
          o8[g][1] = fma2(pp, x1, o8[g][1]);
          o8[g][2] = fma2(pp, x2, o8[g][2]);
          o8[g][3] = fma2(pp, x3, o8[g][3]);
        }
      }
    }
  }
  // two token lanes share a warp when a warp spans two lanes' column ranges: add them first
  const bool pairs = attn_pairs(dv);
  if (pairs) {
#pragma unroll
    for (int g = 0; g < kGq; ++g)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float lo, hi;
        f2_split(o8[g][e], lo, hi);
        lo += __shfl_xor_sync(0xffffffffu, lo, chunks);
        hi += __shfl_xor_sync(0xffffffffu, hi, chunks);
        o8[g][e] = f2(lo, hi);
      }
  }
  const int rl = pairs ? lanes / 2 : lanes;
  const int slot_l = pairs ? tl / 2 : tl;
  if (tl < lanes && (!pairs || (tl & 1) == 0)) {
#pragma unroll
    for (int g = 0; g < kGq; ++g) {
      if (g < G) {
        float4 *dst = reinterpret_cast<float4 *>(red + ((long long)slot_l * kGq + g) * dv + 8 * c);
        float v[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) f2_split(o8[g][e], v[2 * e], v[2 * e + 1]);
        dst[0] = make_float4(v[0], v[1], v[2], v[3]);
        dst[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
    }
  }
  __syncthreads();
  float *po = a.part_o, *pl = a.part_lse;
  for (int e = tid; e < G * dv; e += kThr) {
    const int g = e / dv, d = e - g * dv;
    float sum = 0.f;
    for (int i = 0; i < rl; ++i) sum += red[((long long)i * kGq + g) * dv + d];
    const long long idx = ((long long)r * a.hq + qg.h0 + g) * a.n_splits + split;
    po[idx * dv + d] = l[g] > 0.f ? sum / l[g] : 0.f;
    if (d == 0) pl[idx] = l[g] > 0.f ? m[g] + logf(l[g]) : neg_inf;
  }
}

// ---------------------------------------------------------------------------------------
// Tensor-core split kernel (GQA, head_dim 128): one CTA of two warpgroups (256 threads) per
// (split of two 128-token tiles, up to 16 query heads of one KV head, request). Warpgroup g
// takes tile g: the two run side by side, so one's loads and MMA waits overlap the other's
// softmax. A warpgroup's stage holds K_i, then V_i: V_i is loaded once S_i is computed, while
// the softmax runs, so that two CTAs fit on an SM. Per tile i:
//   S_i^T [128 tokens x 16 heads] = K_i [128 x 128] · Q^T   (tcgen05, M = 128 tokens, N = 16)
//   softmax statistics of the tile: m_i = max_t s, P_i = bf16(exp(s - m_i)), l_i = sum_t P_i
//   O_i^T [128 dims x 16 heads] = V_i^T · P_i              (tcgen05, M = 128 dims, N = 16)
// and thread d of the warpgroup folds O_i into its running output with the log-sum-exp
// rescaling (o <- o e^(M - M') + O_i e^(m_i - M')); the two warpgroups' states are merged the
// same way at the end. Operands in the no-swizzle core-matrix layouts (8 rows x 16 bytes): K
// K-major (token rows), Q K-major (head rows), V MN-major (a 16-byte chunk of a V row is one
// core-matrix row, so V lands unchanged), P K-major (head rows of bf16 probabilities). The
// normaliser sums the same bf16-rounded weights the MMA uses.
// ---------------------------------------------------------------------------------------

constexpr int kTcWg = 2;                  // warpgroups per CTA
constexpr int kTcThr = 128 * kTcWg;
constexpr int kTcTok = 128;    // tokens per tile: the first MMA's M
constexpr int kTcTiles = 2;    // tiles per split: one per warpgroup
constexpr int kTcHeads = 16;   // query heads per CTA: both MMAs' N
constexpr int kTcDim = 128;    // head_dim served by this path: the second MMA's M
constexpr unsigned long long kTcWaitNs = 2000000000ull;

struct TcPlan {
  int q;           // Q operand [16 heads x 128]
  int p;           // P operand per warpgroup [16 heads x 128 tokens]
  int slot;        // long long [kTcTiles][kTcTok]
  int stat;        // per warpgroup: float m[16], l[16], wmax[4][16], wsum[4][16]
  int merge;       // float [128 dims][16] output and [16] (m, l) of warpgroup 1
  int bar;         // per warpgroup: mbarriers of S and O
  int misc;        // TMEM address, timeout flag
  int k, v;        // per warpgroup: the K tile, then the V tile in the same place
  int total;
};

__host__ __device__ inline TcPlan tc_plan() {
  TcPlan p;
  int o = 0;
  p.q = o;
  o += kTcHeads * kTcDim * 2;
  p.p = o;
  o += kTcWg * kTcHeads * kTcTok * 2;
  p.slot = o;
  o += kTcTiles * kTcTok * 8;
  p.stat = o;
  o += kTcWg * (2 * kTcHeads + 8 * kTcHeads) * 4;
  p.merge = o;
  o += (kTcDim * kTcHeads + 2 * kTcHeads) * 4;
  p.bar = o;
  o += kTcWg * 16;
  p.misc = o;
  o += 16;
  o = (o + 127) & ~127;
  p.k = o;
  o += kTcWg * kTcTok * kTcDim * 2;
  p.v = p.k;  // V_i lands where K_i was once S_i is computed: two CTAs fit on an SM
  p.total = o;
  return p;
}

__device__ __forceinline__ void wg_sync(int wg) {  // named barrier of one warpgroup
  asm volatile("bar.sync %0, 128;" ::"r"(1 + wg) : "memory");
}

__global__ void __launch_bounds__(kTcThr) attn_tc_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ __align__(128) unsigned char smem_tc[];
  unsigned char *smem = smem_tc;
  const TcPlan P = tc_plan();
  const uint32_t sb = ptx::smem_addr(smem);
  const DevLayout &lay = a.lay;
  const int split = blockIdx.x, r = blockIdx.z, tid = threadIdx.x;
  const int wg = tid >> 7, wt = tid & 127;          // warpgroup, thread within it (TMEM lane)
  const int wq = wt >> 5, lane = tid & 31;          // warp within the warpgroup
  const int ctx = a.ctx_len[r];
  if (ctx < 0 || ctx > a.max_ctx) {
    if (split == 0 && blockIdx.y == 0 && tid == 0) atomicOr(a.status, KAMERA_DEVICE_BAD_ITEM);
    return;
  }
  const int s0 = split * kTcTok * kTcTiles;
  if (s0 >= ctx) return;  // the merge reads only the splits that hold tokens
  const int ntile = min(kTcTiles, (ctx - s0 + kTcTok - 1) / kTcTok);
  const int group = a.hq / lay.H;
  const int cpk = (group + kTcHeads - 1) / kTcHeads;
  const int kvh = blockIdx.y / cpk, jg = blockIdx.y - kvh * cpk;
  const int h0 = kvh * group + jg * kTcHeads, G = min(kTcHeads, group - jg * kTcHeads);
  long long *slots = reinterpret_cast<long long *>(smem + P.slot);
  float *st = reinterpret_cast<float *>(smem + P.stat) + wg * (10 * kTcHeads);
  float *m_i = st, *l_i = st + kTcHeads, *wmax = st + 2 * kTcHeads, *wsum = wmax + 4 * kTcHeads;
  float *mo = reinterpret_cast<float *>(smem + P.merge);  // warpgroup 1's state
  volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(smem + P.misc);
  constexpr int nc = kTcDim / 8;  // 16-byte chunks per row
  constexpr int kStage = kTcTok * kTcDim * 2;
  const uint32_t qb = sb + P.q, bar = sb + P.bar + 16 * wg;
  const uint32_t kb = sb + P.k + wg * kStage, vb = sb + P.v + wg * kStage;
  const uint32_t pb = sb + P.p + wg * kTcHeads * kTcTok * 2;
  const __nv_bfloat16 *kbase =
      a.pool.k + (long long)a.layer * a.pool.num_slots * lay.row_k + kvh * kTcDim;
  const __nv_bfloat16 *vbase =
      a.pool.v + (long long)a.layer * a.pool.num_slots * lay.row_v + kvh * kTcDim;

  if (tid < 32) {
    ptx::tmem_alloc(sb + P.misc, 64);  // warpgroup g: S in columns 32g..32g+15, O in +16..+31
    ptx::tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < 2 * kTcWg; ++b) ptx::mbar_init(sb + P.bar + 8 * b, 1);
    ptx::fence_mbar_init();
    misc[1] = 0;
  }
  for (int e = tid; e < kTcHeads * nc; e += kTcThr) {  // Q, K-major over 16 head rows
    const int h = e % kTcHeads, c = e / kTcHeads;
    const bool ok = h < G;
    ptx::cp_async16(qb + ((c * (kTcHeads / 8) + (h >> 3)) << 7) + ((h & 7) << 4),
                    ok ? a.q + ((long long)r * a.hq + h0 + h) * kTcDim + 8 * c : a.q,
                    ok ? 16u : 0u);
  }
  for (int t = tid; t < kTcTiles * kTcTok; t += kTcThr)  // every slot of the split, once
    slots[t] = s0 + t < ctx ? slot_of(a.pool, lay.page_size, r, (long long)s0 + t, a.status) : -1;
  ptx::cp_async_commit();
  __syncthreads();
  // K of tile i into this warpgroup's stage; tokens left out are zero-filled
  auto issue_k = [&](int i) {
    const long long *sl = slots + i * kTcTok;
    for (int e = wt; e < kTcTok * nc; e += 128) {  // K-major: a warp takes 8 tokens x 4 chunks
      const int t = (e & 7) + 8 * ((e >> 5) & 15), c = ((e >> 3) & 3) + 4 * (e >> 9);
      const long long sl_t = sl[t];
      ptx::cp_async16(kb + ((c * (kTcTok / 8) + (t >> 3)) << 7) + ((t & 7) << 4),
                      sl_t >= 0 ? kbase + sl_t * lay.row_k + 8 * c : a.pool.k,
                      sl_t >= 0 ? 16u : 0u);
    }
    ptx::cp_async_commit();
  };
  // V of tile i into the same stage, once S_i is computed (K_i is no longer read)
  auto issue_v = [&](int i) {
    const long long *sl = slots + i * kTcTok;
    for (int e = wt; e < kTcTok * nc; e += 128) {  // MN-major: 8 tokens x 4 chunks
      const int t = (e & 7) + 8 * (e / (8 * nc)), c = (e >> 3) % nc;
      const long long sl_t = sl[t];
      ptx::cp_async16(vb + (((t >> 3) * nc + c) << 7) + ((t & 7) << 4),
                      sl_t >= 0 ? vbase + sl_t * lay.row_v + 8 * c : a.pool.v,
                      sl_t >= 0 ? 16u : 0u);
    }
    ptx::cp_async_commit();
  };
  if (wg < ntile) issue_k(wg);

  const float neg_inf = -__int_as_float(0x7f800000);
  float acc[kTcHeads], run_m[kTcHeads], run_l[kTcHeads];  // thread wt: dimension wt
#pragma unroll
  for (int h = 0; h < kTcHeads; ++h) {
    acc[h] = 0.f;
    run_m[h] = neg_inf;
    run_l[h] = 0.f;
  }
  ptx::cp_async_wait_all();  // Q (issued by every thread) and this warpgroup's first tile
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = misc[0];
  const uint32_t ts = tmem + 32 * wg, to = ts + 16;
  const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
  bool timed_out = false;
  int k = 0;  // this warpgroup's tile count (the barriers' phase)
  for (int i = wg; i < ntile; i += kTcWg, ++k) {
    const int n = min(kTcTok, ctx - (s0 + i * kTcTok));
    if (k > 0) {  // the tile issued after the previous one completed
      ptx::cp_async_wait_all();
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      wg_sync(wg);
      ptx::tc_fence_after();
    }
    if (wt == 0 && !timed_out) {  // S_i^T = K_i Q^T
      const uint32_t idesc = ptx::idesc_bf16_f32(kTcTok, kTcHeads);
      for (int ks = 0; ks < kTcDim / 16; ++ks)
        ptx::mma_bf16(ts, ptx::smem_desc(kb + ks * 2 * (kTcTok / 8) * 128, (kTcTok / 8) * 128, 128),
                      ptx::smem_desc(qb + ks * 2 * (kTcHeads / 8) * 128, (kTcHeads / 8) * 128, 128),
                      idesc, ks > 0 ? 1u : 0u);
      ptx::mma_commit(bar);
    }
    if (wq == 0 && !timed_out) {
      const bool ok = ptx::mbar_wait(bar, k & 1, kTcWaitNs);
      if (lane == 0 && !ok) misc[1] = 1;
    }
    ptx::tc_fence_before();
    wg_sync(wg);
    ptx::tc_fence_after();
    timed_out = misc[1] != 0;
    issue_v(i);  // in flight during the softmax

    // the tile's softmax statistics; thread wt holds token wt (TMEM lane wt)
    const bool live = wt < n && slots[i * kTcTok + wt] >= 0 && !timed_out;
    float sc[kTcHeads];
    {
      uint32_t rr[kTcHeads];
      ptx::tmem_ld16(ts + lane_off, rr);
      ptx::tmem_ld_wait(rr);
      ptx::tmem_ld_wait(rr + 8);
#pragma unroll
      for (int h = 0; h < kTcHeads; ++h)
        sc[h] = live ? __uint_as_float(rr[h]) * a.scale : neg_inf;
    }
    {  // column maxima: the 16 heads' butterflies interleaved step by step
      float w[kTcHeads];
#pragma unroll
      for (int h = 0; h < kTcHeads; ++h) w[h] = sc[h];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int h = 0; h < kTcHeads; ++h) w[h] = fmaxf(w[h], __shfl_xor_sync(0xffffffffu, w[h], o));
      if (lane < kTcHeads) {
        float v = w[0];
#pragma unroll
        for (int h = 1; h < kTcHeads; ++h) v = lane == h ? w[h] : v;
        wmax[wq * kTcHeads + lane] = v;
      }
    }
    wg_sync(wg);
    if (wt < kTcHeads)
      m_i[wt] = fmaxf(fmaxf(wmax[wt], wmax[kTcHeads + wt]),
                      fmaxf(wmax[2 * kTcHeads + wt], wmax[3 * kTcHeads + wt]));
    wg_sync(wg);
    {
      float w[kTcHeads];
#pragma unroll
      for (int h = 0; h < kTcHeads; ++h) {
        const float mh = m_i[h];
        const float e = live && mh > neg_inf ? expf(sc[h] - mh) : 0.f;
        const __nv_bfloat16 pb16 = __float2bfloat16_rn(e);
        sts_u16(pb + (((wt >> 3) * (kTcHeads / 8) + (h >> 3)) << 7) + ((h & 7) << 4) +
                    ((wt & 7) << 1),
                __bfloat16_as_ushort(pb16));
        w[h] = __bfloat162float(pb16);  // the normaliser sums the weights the MMA uses
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int h = 0; h < kTcHeads; ++h) w[h] += __shfl_xor_sync(0xffffffffu, w[h], o);
      if (lane < kTcHeads) {
        float v = w[0];
#pragma unroll
        for (int h = 1; h < kTcHeads; ++h) v = lane == h ? w[h] : v;
        wsum[wq * kTcHeads + lane] = v;
      }
    }
    ptx::cp_async_wait_all();  // V_i
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    wg_sync(wg);
    ptx::tc_fence_after();
    if (wt < kTcHeads)
      l_i[wt] = wsum[wt] + wsum[kTcHeads + wt] + wsum[2 * kTcHeads + wt] +
                wsum[3 * kTcHeads + wt];
    if (wt == 0 && !timed_out) {  // O_i^T = V_i^T P_i
      const uint32_t idesc = ptx::idesc_bf16_f32(kTcDim, kTcHeads) | (1u << 15);  // A MN-major
      for (int ks = 0; ks < kTcTok / 16; ++ks)
        ptx::mma_bf16(to, ptx::smem_desc(vb + ks * 2 * nc * 128, nc * 128, 128),
                      ptx::smem_desc(pb + ks * 2 * (kTcHeads / 8) * 128, (kTcHeads / 8) * 128, 128),
                      idesc, ks > 0 ? 1u : 0u);
      ptx::mma_commit(bar + 8);
    }
    if (wq == 0 && !timed_out) {
      const bool ok = ptx::mbar_wait(bar + 8, k & 1, kTcWaitNs);
      if (lane == 0 && !ok) misc[1] = 1;
    }
    ptx::tc_fence_before();
    wg_sync(wg);  // O_i complete: the stage (V_i, P_i) is free; l_i visible
    ptx::tc_fence_after();
    timed_out = misc[1] != 0;
    if (i + kTcWg < ntile) issue_k(i + kTcWg);  // in flight while O_i is folded
    uint32_t ro[kTcHeads];
    ptx::tmem_ld16(to + lane_off, ro);
    ptx::tmem_ld_wait(ro);
    ptx::tmem_ld_wait(ro + 8);
#pragma unroll
    for (int h = 0; h < kTcHeads; ++h) {
      const float mi = m_i[h];
      if (mi > neg_inf) {  // a head with no live token in the tile keeps its running state
        const float mn = fmaxf(run_m[h], mi);
        const float a_old = run_m[h] > neg_inf ? expf(run_m[h] - mn) : 0.f;
        const float a_new = expf(mi - mn);
        acc[h] = acc[h] * a_old + __uint_as_float(ro[h]) * a_new;
        run_l[h] = run_l[h] * a_old + l_i[h] * a_new;
        run_m[h] = mn;
      }
    }
  }
  // warpgroup 1 hands its state over; warpgroup 0 merges and writes
  if (wg == 1) {
#pragma unroll
    for (int h = 0; h < kTcHeads; ++h) mo[wt * kTcHeads + h] = acc[h];
    if (wt == 0)
#pragma unroll
      for (int h = 0; h < kTcHeads; ++h) {
        mo[kTcDim * kTcHeads + h] = run_m[h];
        mo[kTcDim * kTcHeads + kTcHeads + h] = run_l[h];
      }
  }
  __syncthreads();
  timed_out = misc[1] != 0;
  if (wg == 0) {
    if (timed_out && tid == 0) atomicOr(a.status, KAMERA_DEVICE_TIMEOUT);
    const long long base = ((long long)r * a.hq + h0) * a.n_splits + split;
#pragma unroll
    for (int h = 0; h < kTcHeads; ++h) {
      if (h >= G) continue;
      const float m1 = mo[kTcDim * kTcHeads + h], l1 = mo[kTcDim * kTcHeads + kTcHeads + h];
      const float mn = fmaxf(run_m[h], m1);
      const float a0 = run_m[h] > neg_inf ? expf(run_m[h] - mn) : 0.f;
      const float a1 = m1 > neg_inf ? expf(m1 - mn) : 0.f;
      const float L = run_l[h] * a0 + l1 * a1;
      const bool ok = !timed_out && L > 0.f;
      a.part_o[(base + (long long)h * a.n_splits) * kTcDim + wt] =
          ok ? (acc[h] * a0 + mo[wt * kTcHeads + h] * a1) / L : 0.f;
      if (wt == 0) a.part_lse[base + (long long)h * a.n_splits] = ok ? mn + logf(L) : neg_inf;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (tid < 32) ptx::tmem_dealloc(tmem, 64);
}

// One warp per (request, query head): the splits' outputs weighted by exp(lse_s - lse).
__global__ void __launch_bounds__(kThr) attn_merge_kernel(const __grid_constant__ AttnArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long rh = (long long)blockIdx.x * (kThr / 32) + warp;
  if (rh >= (long long)a.n_reqs * a.hq) return;
  const int r = (int)(rh / a.hq);
  const int ctx = a.ctx_len[r];
  if (ctx < 0 || ctx > a.max_ctx) return;  // reported by the split kernel
  const int ns = (ctx + a.split - 1) / a.split;
  const float neg_inf = -__int_as_float(0x7f800000);
  const float *pl = a.part_lse + rh * a.n_splits;
  float mx = neg_inf;
  for (int s = lane; s < ns; s += 32) mx = fmaxf(mx, pl[s]);
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float wsum = 0.f;
  for (int s = lane; s < ns; s += 32) wsum += mx > neg_inf ? expf(pl[s] - mx) : 0.f;
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  const float *po = a.part_o + rh * a.n_splits * a.dv;
  float *out = a.out + rh * a.dv;
  for (int d = lane; d < a.dv; d += 32) {
    float acc = 0.f;
    if (wsum > 0.f)
      for (int s = 0; s < ns; ++s) {
        const float w = expf(pl[s] - mx);
        if (w > 0.f) acc = fmaf(w, po[(long long)s * a.dv + d], acc);
      }
    out[d] = wsum > 0.f ? acc / wsum : 0.f;
  }
  if (lane == 0) a.lse[rh] = wsum > 0.f ? mx + logf(wsum) : neg_inf;
}

}  // namespace

size_t attn_workspace(long long n_reqs, int hq, int max_ctx, int dv) {
  const long long ns = (max_ctx + kSplit - 1) / kSplit;  // the smaller of the two split sizes
  return (size_t)(n_reqs * hq * ns * (dv + 1)) * sizeof(float);
}

size_t attn_smem(int dk, int dv) { return (size_t)attn_plan(dk, dv).total; }

bool attn_tensor_path(const DevLayout &l) { return l.kind == KAMERA_GQA && l.hd == kTcDim; }

int attn_split_tokens(const DevLayout &l) {
  return attn_tensor_path(l) ? kTcTok * kTcTiles : kSplit;
}

cudaError_t launch_attention(const AttnArgs &a, cudaStream_t s) {
  static int configured[64] = {0};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const bool tc = attn_tensor_path(a.lay);
  const int smem = tc ? tc_plan().total : (int)attn_smem(a.dk, a.dv);
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev]) {
      e = cudaFuncSetAttribute(attn_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)attn_smem(1024, 1024));
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               tc_plan().total);
      if (e != cudaSuccess) return e;
      configured[dev] = 1;
    }
  }
  const int n_kv = a.lay.kind == KAMERA_GQA ? a.lay.H : 1;
  const int group = a.hq / n_kv;
  const int per = tc ? kTcHeads : kGq;
  const int cpk = (group + per - 1) / per;
  if (a.n_splits > 0) {
    const dim3 grid((unsigned)a.n_splits, (unsigned)(n_kv * cpk), (unsigned)a.n_reqs);
    if (tc)
      attn_tc_kernel<<<grid, kTcThr, smem, s>>>(a);
    else
      attn_split_kernel<<<grid, kThr, smem, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const long long pairs = (long long)a.n_reqs * a.hq;
  attn_merge_kernel<<<(unsigned)((pairs + kThr / 32 - 1) / (kThr / 32)), kThr, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kamera
