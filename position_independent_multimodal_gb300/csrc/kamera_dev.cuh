// Internal definitions shared by the host API and the kernels of the Kamera library.
//
// Operator: Kamera (Unified Position-Invariant Multimodal KV Cache for Training-Free Reuse),
// Eq. 1: KV^(B|A) = R(delta) * KV(B|empty) + U_m V_m^T, written into a paged KV pool.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kamera.h"

namespace kamera {

constexpr int kMaxPairs = 128;  // rope_dim <= 256
constexpr int kMaxRank = 128;
constexpr int kMaxRow = 16384;

// Layout with every derived width spelled out (filled once by kamera_create).
struct DevLayout {
  int kind, L, page_size, H, hd, latent, rope_d, style;
  int row_k, row_v;  // row widths of channel 0 (K, or c_KV || k_pe) and channel 1 (V)
  int w0, w1;        // patch group widths
  int npairs;        // rope pairs per band (rope_d / 2)
  int n_ch;          // 2 for GQA (K, V), 1 for MLA
  // column tiles of the fused kernel: GQA rows split into tiles of `tw` columns holding whole
  // heads; MLA rows into latent tiles of `tw` plus one tile for the k_pe band
  int tw;            // tile width (<= 256, multiple of 16)
  int ntile;         // tiles per row (same for both GQA channels)
  int mrope;         // 1: M-RoPE sections (each rope pair turns by its section's offset)
  int mrope_t, mrope_h, mrope_w, mrope_style;  // pairs per section, KAMERA_MROPE_*
};

// Engines for patched tiles.
constexpr int kEngineTensor = 0;  // tcgen05 MMA into TMEM (rank a multiple of 8)
constexpr int kEngineFma = 1;     // float32 FMAs on CUDA cores (any rank)

// Rows per tile of the fused kernel: the MMA's M and the TMEM lanes.
constexpr int kTileRows = 128;

// Byte offsets of the fused kernel's dynamic shared memory.
struct SmemPlan {
  int b_op, b_stage;     // B operand (V_m^T rows): MN-major core matrices [Kp/8][tw/8][128 B]
  int a_op, a_stage;     // one or two A operands (U rows): K-major core matrices [Kp/8][16][128 B]
  int canon, stage;      // two stages of [128][pitch] bf16 canonical rows
  int pitch;             // row pitch in bytes (tile width * 2 + 16: rows land on distinct banks)
  int cs, cs_stage;      // two float2 cos/sin tables [npairs]
  int pages, pages_stage;  // two stages of page ids of the tile's tokens, per run member
  int pg_per_member;     // page ids per member and stage (tile rows / page size + 2)
  int desc;              // two stage descriptors
  int slots;             // slots (fast plan: int [run][128], -1 skips) of the tile's rows
  int members;           // run members' (req, start_tok): int [2][kShareBlock]
  int run;               // most group members one CTA writes (1: no groups)
  int misc;              // TMEM address (4 B), the MMA mbarrier and the two stage mbarriers
  int total;
  int tmem_cols;         // TMEM columns to allocate (0: no patched tiles possible)
  int acc_cols;          // TMEM columns of one accumulator
  int u_bufs;            // U buffers (2: staged two tiles ahead; 1: after each MMA)
  int fast;              // 1: plan of the tile kernels (swizzled canonical stages)
  int recs;              // persistent kernel: task records in shared memory
};

// A column tile: [col0, col0 + ncols) of a channel's row.
struct Tile {
  int col0, ncols;
  int group, gcol0;  // patch group and the tile's first column inside it
  int band;          // width of the rope bands it holds (0: nothing rotates in this tile)
};

__host__ __device__ inline Tile tile_of(const DevLayout &l, int ch, int ti, bool rotate) {
  Tile t;
  if (l.kind == KAMERA_GQA) {
    t.col0 = ti * l.tw;
    t.ncols = (l.row_k - t.col0) < l.tw ? (l.row_k - t.col0) : l.tw;
    t.group = ch;
    t.gcol0 = t.col0;
    t.band = (ch == 0 && rotate) ? l.hd : 0;
  } else {
    const int nlat = (l.latent + l.tw - 1) / l.tw;
    if (ti < nlat) {
      t.col0 = ti * l.tw;
      t.ncols = (l.latent - t.col0) < l.tw ? (l.latent - t.col0) : l.tw;
      t.group = 0;
      t.gcol0 = t.col0;
      t.band = 0;
    } else {
      t.col0 = l.latent;
      t.ncols = l.rope_d;
      t.group = 1;
      t.gcol0 = 0;
      t.band = rotate ? l.rope_d : 0;
    }
  }
  return t;
}

// Per-pair rotation speed in turns per token, as an unsigned Q0.64 fixed-point fraction:
// q_i = round(inv_freq_i / (2 pi) * 2^64). The angle of offset delta is delta * q_i mod 2^64,
// an exact modular product, so the range reduction of large |delta| loses nothing.
struct FreqQ64 {
  unsigned long long q[kMaxPairs];
};

struct DevPool {
  __nv_bfloat16 *k;
  __nv_bfloat16 *v;
  long long num_slots;
  const int32_t *pt;
  int num_reqs, pt_stride;
};

struct ReuseArgs {
  DevLayout lay;
  DevPool pool;
  kamera_item single;        // used when items == nullptr
  const kamera_item *items;  // device array (batch)
  int n_items;
  int max_tokens;
  int max_m;
  int engine;                // kEngineTensor or kEngineFma for patched tiles
  int inplace;               // 1: patch re-add on cached rows (read from and written to the pool)
  int sign;                  // inplace: +1 adds U V_m^T, -1 subtracts it
  int run_copy;              // most group members one CTA of the copy kernel writes
  void *plan_ws;             // batch workspace: patched layers take the persistent kernel
  SmemPlan smem;
  unsigned *status;
  FreqQ64 freq;
};

struct RelocArgs {
  DevLayout lay;
  DevPool pool;
  int req, start_tok, T;
  long long delta;
  unsigned *status;
  FreqQ64 freq;
};

struct AnchorArgs {
  DevLayout lay;
  DevPool pool;
  const kamera_anchor_item *items;
  int n_items, max_tokens;
  unsigned *status;
  FreqQ64 freq;
};

struct AttnArgs {
  DevLayout lay;
  DevPool pool;
  int layer;
  const __nv_bfloat16 *q;  // [n_reqs][hq][dk]
  const int *ctx_len;      // [n_reqs]
  int n_reqs, hq, dk, dv, max_ctx, n_splits;
  int split;               // tokens per split (the kernel's; n_splits = ceil(max_ctx / split))
  float scale;
  float *part_o, *part_lse;  // workspace: [n_reqs][hq][n_splits][dv], [n_reqs][hq][n_splits]
  float *out, *lse;          // [n_reqs][hq][dv], [n_reqs][hq]
  unsigned *status;
};

// The rules an item must satisfy (host: kamera_reuse; device: each batch item).
__host__ __device__ inline bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

__host__ __device__ inline int item_check(const kamera_item &it, const DevLayout &lay,
                                          const DevPool &pool, int max_tokens, int max_m) {
  // returns 0 when valid, else a kamera_status code
  if (it.num_tokens < 0 || it.num_tokens > max_tokens) return KAMERA_ERR_INVALID_ARG;
  if (it.patch_m < 0 || it.patch_m > kMaxRank) return KAMERA_ERR_UNSUPPORTED;
  if (it.patch_m > max_m) return KAMERA_ERR_INVALID_ARG;
  if (it.delta > (1ll << 62) || it.delta < -(1ll << 62)) return KAMERA_ERR_INVALID_ARG;
  if (lay.mrope && (it.delta_h > (1ll << 62) || it.delta_h < -(1ll << 62) ||
                    it.delta_w > (1ll << 62) || it.delta_w < -(1ll << 62)))
    return KAMERA_ERR_INVALID_ARG;
  if (it.num_tokens == 0) return 0;
  if (!it.canon_k || !aligned16(it.canon_k)) return KAMERA_ERR_INVALID_ARG;
  if (lay.kind == KAMERA_GQA) {
    if (!it.canon_v || !aligned16(it.canon_v)) return KAMERA_ERR_INVALID_ARG;
  } else if (it.canon_v) {
    return KAMERA_ERR_INVALID_ARG;
  }
  if (it.req < 0 || it.req >= pool.num_reqs || it.start_tok < 0) return KAMERA_ERR_INVALID_ARG;
  if ((long long)it.start_tok + it.num_tokens > (long long)pool.pt_stride * lay.page_size)
    return KAMERA_ERR_INVALID_ARG;
  if (it.patch_m > 0) {
    if (it.patch_l0 < 0 || it.patch_l1 < it.patch_l0 || it.patch_l1 > lay.L)
      return KAMERA_ERR_INVALID_ARG;
    if (it.patch_l1 > it.patch_l0) {
      if (!it.patch_u || !it.patch_vt || !aligned16(it.patch_vt) ||
          (reinterpret_cast<uintptr_t>(it.patch_u) & 1u))
        return KAMERA_ERR_INVALID_ARG;
    }
  }
  return 0;
}

// The rules of an item of an in-place patch re-add: the canonical pointers and the offset are
// not read; tokens, request, rank, layers and factors as for reuse.
__host__ __device__ inline int inplace_item_check(const kamera_item &it, const DevLayout &lay,
                                                  const DevPool &pool, int max_tokens,
                                                  int max_m) {
  if (it.num_tokens < 0 || it.num_tokens > max_tokens) return KAMERA_ERR_INVALID_ARG;
  if (it.patch_m < 0 || it.patch_m > kMaxRank) return KAMERA_ERR_UNSUPPORTED;
  if (it.patch_m > max_m) return KAMERA_ERR_INVALID_ARG;
  if (it.num_tokens == 0 || it.patch_m == 0) return 0;
  if (it.req < 0 || it.req >= pool.num_reqs || it.start_tok < 0) return KAMERA_ERR_INVALID_ARG;
  if ((long long)it.start_tok + it.num_tokens > (long long)pool.pt_stride * lay.page_size)
    return KAMERA_ERR_INVALID_ARG;
  if (it.patch_l0 < 0 || it.patch_l1 < it.patch_l0 || it.patch_l1 > lay.L)
    return KAMERA_ERR_INVALID_ARG;
  if (it.patch_l1 > it.patch_l0 &&
      (!it.patch_u || !it.patch_vt || !aligned16(it.patch_vt) ||
       (reinterpret_cast<uintptr_t>(it.patch_u) & 1u)))
    return KAMERA_ERR_INVALID_ARG;
  return 0;
}

// M-RoPE section of rope pair i: 0 t, 1 h, 2 w. Contiguous: [0, t) t, then h, then w;
// interleaved: h at i % 3 == 1 below 3h, w at i % 3 == 2 below 3w, t elsewhere.
__host__ __device__ __forceinline__ int mrope_axis(const DevLayout &l, int i) {
  if (l.mrope_style == KAMERA_MROPE_INTERLEAVED) {
    const int r = i % 3;
    return (r == 1 && i < 3 * l.mrope_h) ? 1 : (r == 2 && i < 3 * l.mrope_w) ? 2 : 0;
  }
  return i < l.mrope_t ? 0 : (i < l.mrope_t + l.mrope_h ? 1 : 2);
}

// Offset of rope pair i: the item's delta under 1-D RoPE; under M-RoPE, delta, delta_h or
// delta_w by the pair's section.
__host__ __device__ __forceinline__ long long pair_delta(const kamera_item &it,
                                                         const DevLayout &l, int i) {
  if (!l.mrope) return it.delta;
  const int axis = mrope_axis(l, i);
  return axis == 0 ? it.delta : (axis == 1 ? it.delta_h : it.delta_w);
}

// Whether any rope pair of the item turns.
__host__ __device__ __forceinline__ bool item_rotates(const kamera_item &it,
                                                      const DevLayout &l) {
  return it.delta != 0 || (l.mrope && (it.delta_h != 0 || it.delta_w != 0));
}

// The rules of a re-anchoring item (checked on the device for every item).
__host__ __device__ inline int anchor_item_check(const kamera_anchor_item &it,
                                                 const DevLayout &lay, const DevPool &pool,
                                                 int max_tokens) {
  if (it.num_tokens < 0 || it.num_tokens > max_tokens) return KAMERA_ERR_INVALID_ARG;
  if (it.num_tokens == 0) return 0;
  if (!it.canon_k || !aligned16(it.canon_k)) return KAMERA_ERR_INVALID_ARG;
  if (lay.kind == KAMERA_GQA) {
    if (!it.canon_v || !aligned16(it.canon_v)) return KAMERA_ERR_INVALID_ARG;
  } else if (it.canon_v) {
    return KAMERA_ERR_INVALID_ARG;
  }
  if (!it.positions || (reinterpret_cast<uintptr_t>(it.positions) & 7u))
    return KAMERA_ERR_INVALID_ARG;
  if (it.req < 0 || it.req >= pool.num_reqs || it.start_tok < 0) return KAMERA_ERR_INVALID_ARG;
  if ((long long)it.start_tok + it.num_tokens > (long long)pool.pt_stride * lay.page_size)
    return KAMERA_ERR_INVALID_ARG;
  return 0;
}

__device__ __forceinline__ bool layer_patched(const kamera_item &it, int layer) {
  return it.patch_m > 0 && layer >= it.patch_l0 && layer < it.patch_l1;
}

// Shared chunks in a batch. Placements of one chunk (the reorder of §5 puts each chunk in
// several orderings; one orbit patch serves them all) read the same canonical rows and add the
// same patch, and where nothing in a tile turns, or it turns by the same offsets, they produce
// the same bytes. The batch kernels therefore group the items of each aligned block of
// consecutive items (at most kShareBlock): the lowest valid item of a set of equal sources
// reads and computes the rows once and writes them to every member's slots.
constexpr int kShareBlock = 32;

__device__ __forceinline__ bool same_offsets(const kamera_item &a, const kamera_item &b,
                                             const DevLayout &l) {
  return a.delta == b.delta && (!l.mrope || (a.delta_h == b.delta_h && a.delta_w == b.delta_w));
}

// Lane j of a warp loads item (self's aligned block of kShareBlock items) + j for the group
// search, with the CTA's own item: the whole item, so that the search needs one round trip.
// Returns false (and leaves *o alone) when there is no such item or `on` is false.
__device__ __forceinline__ bool share_candidate(const kamera_item *items, int n_items, int self,
                                                bool on, kamera_item *o) {
  const int j = (self & ~(kShareBlock - 1)) + (int)(threadIdx.x & 31);
  if (!on || !items || j >= n_items || j == self) return false;
  *o = items[j];
  return true;
}

// Called by whole warps for item `self` (its item `me`, its channel's canonical `src`, and
// each lane's share_candidate item `cand` when `has_cand`) of a batch: the group of self is
// every valid item of self's aligned block of kShareBlock items with the same canonical for
// which `same` holds; its members, in item order, are split into runs of `run` items, and the
// CTA of each run's first item takes the run. Every lane returns the size of self's run (0:
// self belongs to a run that another CTA takes). When `record`, the run's requests and first
// tokens are written to members[f] and members[kShareBlock + f] (f = 0 is self).
template <class Same>
__device__ __forceinline__ int share_run(int self, const kamera_item &me, const void *src, int ch,
                                         bool has_cand, const kamera_item &cand, int run,
                                         int *members, bool record, Same same) {
  const int lane = threadIdx.x & 31;
  const int b0 = self & ~(kShareBlock - 1);
  const int j = b0 + lane;
  bool mem = j == self;
  int req = me.req, start = me.start_tok;
  if (has_cand && (ch == 0 ? cand.canon_k : cand.canon_v) == src && same(cand)) {
    mem = true;
    req = cand.req;
    start = cand.start_tok;
  }
  const unsigned mask = __ballot_sync(0xffffffffu, mem);
  const int f_self = __popc(mask & ((1u << (self - b0)) - 1u));
  if (f_self % run != 0) return 0;
  if (mem && record) {
    const int f = __popc(mask & ((1u << lane) - 1u)) - f_self;
    if (f >= 0 && f < run) {
      members[f] = req;
      members[kShareBlock + f] = start;
    }
  }
  const int left = __popc(mask) - f_self;
  return left < run ? left : run;
}

// cos/sin of delta * inv_freq_i: exact modular range reduction in Q0.64 turns, then the
// CUDA single-precision sincospi on the reduced angle (|angle| <= pi).
__device__ __forceinline__ float2 rope_phase(unsigned long long q, long long delta) {
  const unsigned long long turns = static_cast<unsigned long long>(delta) * q;
  const long long centred = static_cast<long long>(turns);   // [-1/2, 1/2) turn
  const float x = static_cast<float>(centred) * 0x1p-63f;   // angle / pi in [-1, 1)
  float s, c;
  sincospif(x, &s, &c);
  return make_float2(c, s);
}

// Physical slot of logical token tok of request req; -1 (and the OOB status bit) when the
// page-table entry points outside the pool.
__device__ __forceinline__ long long slot_of(const DevPool &p, int page_size, int req,
                                             long long tok, unsigned *status) {
  const long long pi = tok / page_size;
  if (pi >= p.pt_stride) {
    atomicOr(status, KAMERA_DEVICE_SLOT_OOB);
    return -1;
  }
  const int page = __ldg(p.pt + (long long)req * p.pt_stride + pi);
  if (page < 0 || (long long)(page + 1) * page_size > p.num_slots) {
    atomicOr(status, KAMERA_DEVICE_SLOT_OOB);
    return -1;
  }
  return (long long)page * page_size + tok % page_size;
}

// Columns are processed in units of 16: two 8-column (16-byte) chunks at ca and cb that are
// closed under rope pairing. NeoX-half: chunk cb holds the partners (d/2 apart) of chunk ca.
// Interleaved: each chunk pairs its own neighbours. Non-rope units: two consecutive chunks.
struct ColUnit {
  int ca, cb;    // first columns in the row
  int rot;       // 0 none, 1 NeoX-half (xa[e] with xb[e]), 2 interleaved (within chunks)
  int fa, fb;    // first frequency index of chunk a / b
  int group;     // patch group
  int gca, gcb;  // columns inside the patch group
};

// Unit u of a region [c0, c0 + w) that does not rotate: two 8-column chunks from the same
// 128-column group, half a group apart, so 8 consecutive units cover whole 128-byte lines
// (the last group may be narrower).
__device__ __forceinline__ void plain_unit(int c0, int w, int u, int *ca, int *cb) {
  const int gbase = (u >> 3) * 128;
  const int gw = (w - gbase) < 128 ? (w - gbase) : 128;
  *ca = c0 + gbase + 8 * (u & 7);
  *cb = *ca + (gw >> 1);
}

__device__ __forceinline__ int units_per_row(const DevLayout &l, int ch) {
  return (ch == 0 ? l.row_k : l.row_v) >> 4;
}

__device__ __forceinline__ ColUnit col_unit(const DevLayout &l, int ch, int u, bool rotate) {
  ColUnit c;
  if (l.kind == KAMERA_GQA) {
    if (ch == 1 || !rotate) {
      plain_unit(0, ch == 0 ? l.row_k : l.row_v, u, &c.ca, &c.cb);
      c.rot = 0;
      c.fa = c.fb = 0;
    } else {
      const int per_head = l.hd >> 4;
      const int h = u / per_head, q = u - h * per_head;
      if (l.style == KAMERA_ROPE_NEOX_HALF) {
        c.ca = h * l.hd + 8 * q;
        c.cb = c.ca + (l.hd >> 1);
        c.rot = 1;
        c.fa = 8 * q;
        c.fb = 8 * q;
      } else {
        c.ca = h * l.hd + 16 * q;
        c.cb = c.ca + 8;
        c.rot = 2;
        c.fa = 8 * q;
        c.fb = 8 * q + 4;
      }
    }
    c.group = ch;
    c.gca = c.ca;
    c.gcb = c.cb;
  } else {
    const int lat_units = l.latent >> 4;
    if (u < lat_units) {
      plain_unit(0, l.latent, u, &c.ca, &c.cb);
      c.rot = 0;
      c.fa = c.fb = 0;
      c.group = 0;
      c.gca = c.ca;
      c.gcb = c.cb;
    } else {
      const int r = u - lat_units;
      if (!rotate) {
        plain_unit(l.latent, l.rope_d, r, &c.ca, &c.cb);
        c.rot = 0;
        c.fa = c.fb = 0;
      } else if (l.style == KAMERA_ROPE_NEOX_HALF) {
        c.ca = l.latent + 8 * r;
        c.cb = c.ca + (l.rope_d >> 1);
        c.rot = 1;
        c.fa = c.fb = 8 * r;
      } else {
        c.ca = l.latent + 16 * r;
        c.cb = c.ca + 8;
        c.rot = 2;
        c.fa = 8 * r;
        c.fb = 8 * r + 4;
      }
      c.group = 1;
      c.gca = c.ca - l.latent;
      c.gcb = c.cb - l.latent;
    }
  }
  return c;
}

__device__ __forceinline__ void unpack8(const uint4 &v, float *x) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack2_rn(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint4 pack8_rn(const float *x) {
  uint4 v;
  v.x = pack2_rn(x[0], x[1]);
  v.y = pack2_rn(x[2], x[3]);
  v.z = pack2_rn(x[4], x[5]);
  v.w = pack2_rn(x[6], x[7]);
  return v;
}

// (a, b) -> (a cos - b sin, b cos + a sin)
__device__ __forceinline__ void rot_pair(float &a, float &b, float2 cs) {
  const float na = fmaf(a, cs.x, -b * cs.y);
  const float nb = fmaf(b, cs.x, a * cs.y);
  a = na;
  b = nb;
}

__device__ __forceinline__ void rotate_unit(const ColUnit &c, const float2 *cs, float *xa,
                                            float *xb) {
  if (c.rot == 1) {
#pragma unroll
    for (int e = 0; e < 8; ++e) rot_pair(xa[e], xb[e], cs[c.fa + e]);
  } else if (c.rot == 2) {
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      rot_pair(xa[e], xa[e + 1], cs[c.fa + (e >> 1)]);
      rot_pair(xb[e], xb[e + 1], cs[c.fb + (e >> 1)]);
    }
  }
}

// The eight (cos, sin) a unit's rotation reads, for keeping in registers while a thread turns
// the same unit of many rows: NeoX pairs fa..fa+7; interleaved fa..fa+3, then fb..fb+3.
__device__ __forceinline__ void unit_phases(const ColUnit &c, const float2 *cs, float2 *p) {
#pragma unroll
  for (int e = 0; e < 8; ++e)
    p[e] = c.rot == 1 ? cs[c.fa + e] : cs[(e < 4 ? c.fa : c.fb - 4) + e];
}

// rotate_unit with the phases of unit_phases.
__device__ __forceinline__ void rotate_unit_with(const ColUnit &c, const float2 *p, float *xa,
                                                 float *xb) {
  if (c.rot == 1) {
#pragma unroll
    for (int e = 0; e < 8; ++e) rot_pair(xa[e], xb[e], p[e]);
  } else if (c.rot == 2) {
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      rot_pair(xa[e], xa[e + 1], p[e >> 1]);
      rot_pair(xb[e], xb[e + 1], p[4 + (e >> 1)]);
    }
  }
}

// Patch forming (kamera_form.cu): one problem is a float32 deficit [T x W].
constexpr int kMaxSketch = 96;            // sketch width k
constexpr int kMaxFormSmem = 232448;      // shared memory per block (opt-in limit of sm_103a)

struct FormArgs {
  const float *delta;       // problem i at delta + i*delta_stride, row stride ld
  long long ld, delta_stride;
  const float *omega;       // [W x k] row-major, problem i at omega + i*omega_stride
  long long omega_stride;
  int n, T, W, k, q, m;
  __nv_bfloat16 *u;         // U*Sigma [T x m] at u + i*u_stride
  long long u_stride;
  __nv_bfloat16 *vt;        // V_m^T [m x W] at vt + i*vt_stride
  long long vt_stride;
  float *sigma;             // [n][m] or null
  float *work;              // 2 * max(T, W) * k floats per problem
};

// Kernel launchers.
size_t form_patch_workspace(long long n, int T, int W, int k);  // kamera_form.cu
size_t form_patch_smem(int k);  // the largest of the patch-forming kernels
cudaError_t launch_form_patch(const FormArgs &a, cudaStream_t s);
cudaError_t prepare_form_patch();  // loads the kernel and sets its shared-memory limit
// The argument checks of kamera_form_patch other than those of the workspace.
kamera_status form_patch_args(const float *d_delta, int64_t ld, int64_t delta_stride,
                              int32_t num_problems, int32_t T, int32_t W, const float *d_omega,
                              int64_t omega_stride, int32_t k, int32_t q, int32_t m,
                              const void *d_u, int64_t u_stride, const void *d_vt,
                              int64_t vt_stride, const float *d_sigma);
SmemPlan reuse_smem_plan(const DevLayout &l, int max_m);           // kamera_reuse.cu
cudaError_t launch_reuse(const ReuseArgs &a, int n_items, cudaStream_t s);
bool fast_layout(const DevLayout &l);                               // kamera_reuse_tile.cu
bool inplace_layout(const DevLayout &l);
SmemPlan reuse_tile_plan(const DevLayout &l, int max_m, int max_run);
cudaError_t launch_reuse_tile(const ReuseArgs &a, int n_items, cudaStream_t s);
// The persistent path of patched layers (kamera_reuse_tile.cu): workspace bytes for batches of
// up to n_items items, its plan (fast == 0 when the layout, rank or run does not fit it), and
// the launch of the planning and persistent kernels on `s` (a.plan_ws set; `planned`, when
// not null, recorded between them).
size_t persist_workspace_bytes(const DevLayout &l, long long n_items);
SmemPlan reuse_persist_plan(const DevLayout &l, int max_m, int run);
bool persist_batch_ok(const DevLayout &l, const SmemPlan &p, int n_items, int max_tokens);
cudaError_t launch_reuse_persist(const ReuseArgs &a, cudaStream_t s,
                                 cudaEvent_t planned = nullptr);
cudaError_t launch_relocate(const RelocArgs &a, cudaStream_t s);   // kamera_stream.cu
cudaError_t launch_reuse_copy(const ReuseArgs &a, cudaStream_t s);  // kamera_stream.cu
cudaError_t launch_reanchor(const AnchorArgs &a, cudaStream_t s);   // kamera_anchor.cu
size_t attn_workspace(long long n_reqs, int hq, int max_ctx, int dv);  // kamera_attn.cu
size_t attn_smem(int dk, int dv);
int attn_split_tokens(const DevLayout &l);
cudaError_t launch_attention(const AttnArgs &a, cudaStream_t s);
cudaError_t launch_rope_phases(const FreqQ64 &f, int npairs, const long long *deltas, int n,
                               float *out, cudaStream_t s);

}  // namespace kamera
