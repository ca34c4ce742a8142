// Host side of the Kamera C ABI: descriptor checks, RoPE frequency precomputation, argument
// checks and kernel launches. See include/kamera.h for the contract of every call.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "kamera_dev.cuh"

struct kamera_handle {
  kamera_layout desc;
  kamera::DevLayout lay;
  kamera::FreqQ64 freq;
  int engine;     // engine of patched tiles (KAMERA_OPT_PATCH_ENGINE)
  int run_tile;   // most members of a group written from one computed tile, patched layers
  int run_copy;   // the same on unpatched layers
  void *ws = nullptr;     // batch workspace (kamera_set_batch_workspace), device memory
  size_t ws_bytes = 0;
};

namespace {

using kamera::DevLayout;
using kamera::DevPool;

bool is_mult16(int x) { return x > 0 && (x % 16) == 0; }

kamera_status fill_layout(const kamera_layout &d, DevLayout *out) {
  DevLayout l{};
  if (d.num_layers < 1 || d.page_size < 1) return KAMERA_ERR_INVALID_ARG;
  if (!(d.rope_theta > 1.0) || !std::isfinite(d.rope_theta)) return KAMERA_ERR_INVALID_ARG;
  if (d.rope_style != KAMERA_ROPE_NEOX_HALF && d.rope_style != KAMERA_ROPE_INTERLEAVED)
    return KAMERA_ERR_INVALID_ARG;
  l.kind = d.kind;
  l.L = d.num_layers;
  l.page_size = d.page_size;
  l.style = d.rope_style;
  if (d.kind == KAMERA_GQA) {
    if (d.num_kv_heads < 1 || d.head_dim < 1) return KAMERA_ERR_INVALID_ARG;
    if (d.rope_dim != d.head_dim) return KAMERA_ERR_UNSUPPORTED;  // partial rotary
    if (!is_mult16(d.head_dim) || d.head_dim > 2 * kamera::kMaxPairs)
      return KAMERA_ERR_UNSUPPORTED;
    if ((long long)d.num_kv_heads * d.head_dim > kamera::kMaxRow) return KAMERA_ERR_UNSUPPORTED;
    l.H = d.num_kv_heads;
    l.hd = d.head_dim;
    l.rope_d = d.head_dim;
    l.latent = 0;
    l.row_k = l.row_v = l.H * l.hd;
    l.w0 = l.w1 = l.row_k;
    l.n_ch = 2;
    // tiles of whole heads, about 128 columns wide
    l.tw = l.hd >= 128 ? l.hd : l.hd * (128 / l.hd);
    if (l.tw > l.row_k) l.tw = l.row_k;
    l.ntile = (l.row_k + l.tw - 1) / l.tw;
  } else if (d.kind == KAMERA_MLA) {
    if (d.latent_dim < 1 || d.rope_dim < 1) return KAMERA_ERR_INVALID_ARG;
    if (!is_mult16(d.latent_dim) || !is_mult16(d.rope_dim) ||
        d.rope_dim > 2 * kamera::kMaxPairs)
      return KAMERA_ERR_UNSUPPORTED;
    if (d.latent_dim + d.rope_dim > kamera::kMaxRow) return KAMERA_ERR_UNSUPPORTED;
    l.H = 0;
    l.hd = 0;
    l.latent = d.latent_dim;
    l.rope_d = d.rope_dim;
    l.row_k = d.latent_dim + d.rope_dim;
    l.row_v = 0;
    l.w0 = d.latent_dim;
    l.w1 = d.rope_dim;
    l.n_ch = 1;
    l.tw = d.latent_dim < 128 ? d.latent_dim : 128;
    l.ntile = (d.latent_dim + l.tw - 1) / l.tw + 1;
  } else {
    return KAMERA_ERR_INVALID_ARG;
  }
  l.npairs = l.rope_d / 2;
  // M-RoPE sections: pairs of t, h, w summing to the band's pairs (Fig. 2 "16|24|24")
  const int st = d.mrope_section[0], sh = d.mrope_section[1], sw = d.mrope_section[2];
  l.mrope = 0;
  if (st != 0 || sh != 0 || sw != 0) {
    if (st < 0 || sh < 0 || sw < 0 || st + sh + sw != l.npairs) return KAMERA_ERR_INVALID_ARG;
    if (d.mrope_style == KAMERA_MROPE_INTERLEAVED) {
      if (3 * sh > l.npairs + 1 || 3 * sw > l.npairs) return KAMERA_ERR_INVALID_ARG;
    } else if (d.mrope_style != KAMERA_MROPE_CONTIGUOUS) {
      return KAMERA_ERR_INVALID_ARG;
    }
    l.mrope = 1;
    l.mrope_t = st;
    l.mrope_h = sh;
    l.mrope_w = sw;
    l.mrope_style = d.mrope_style;
  }
  *out = l;
  return KAMERA_OK;
}

// 1/(2 pi) as an unevaluated sum of two doubles (106 significant bits).
constexpr double kInvTwoPiHi = 0.15915494309189535;
constexpr double kInvTwoPiLo = -9.839338337591243e-18;

// q_i = round(inv_freq_i / (2 pi) * 2^64), inv_freq_i = theta^(-2i/d) in double. The product
// with 1/(2 pi) is carried in two doubles (exact product by fma, plus the low constant), so
// q_i is the double inv_freq_i over 2 pi to within half a unit of 2^-64: a relocation by
// delta then carries at most |delta| * 2^-65 turns of error from the table.
void fill_freq(const kamera_layout &d, const DevLayout &l, kamera::FreqQ64 *f) {
  std::memset(f, 0, sizeof(*f));
  for (int i = 0; i < l.npairs; ++i) {
    const double inv = std::pow(d.rope_theta, -2.0 * i / l.rope_d);
    const double x = std::ldexp(inv, 64);                 // exact scaling, < 2^64
    const double p = x * kInvTwoPiHi;                     // < 2^62
    const double e = std::fma(x, kInvTwoPiHi, -p) + x * kInvTwoPiLo;
    const double ip = std::floor(p);
    const long long frac = std::llround((p - ip) + e);    // p - ip is exact
    f->q[i] = static_cast<unsigned long long>(ip) + static_cast<unsigned long long>(frac);
  }
}

kamera_status check_pool(const DevLayout &l, const kamera_pool *p, DevPool *out) {
  if (!p) return KAMERA_ERR_INVALID_ARG;
  if (!p->k || !kamera::aligned16(p->k)) return KAMERA_ERR_INVALID_ARG;
  if (l.kind == KAMERA_GQA) {
    if (!p->v || !kamera::aligned16(p->v)) return KAMERA_ERR_INVALID_ARG;
  } else if (p->v) {
    return KAMERA_ERR_INVALID_ARG;
  }
  if (p->num_slots <= 0 || p->num_slots % l.page_size != 0) return KAMERA_ERR_INVALID_ARG;
  if (p->num_slots > 0x7FFFFFFFll) return KAMERA_ERR_UNSUPPORTED;  // slots are int32 on device
  if (!p->page_table || p->num_reqs < 1 || p->pt_stride < 1) return KAMERA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(p->page_table) & 3u) != 0) return KAMERA_ERR_INVALID_ARG;
  DevPool d;
  d.k = static_cast<__nv_bfloat16 *>(p->k);
  d.v = static_cast<__nv_bfloat16 *>(p->v);
  d.num_slots = p->num_slots;
  d.pt = p->page_table;
  d.num_reqs = p->num_reqs;
  d.pt_stride = p->pt_stride;
  *out = d;
  return KAMERA_OK;
}

kamera_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KAMERA_OK : KAMERA_ERR_CUDA; }

// A side stream per device on which the copy kernel runs next to the patched-layer kernel (the
// two write disjoint layers). The caller's stream forks into it and joins it again through two
// events, so work issued on the caller's stream afterwards waits for both kernels. Created on
// the first call that needs it on that device; a failure to create it only serialises the two
// kernels on the caller's stream.
struct SideStream {
  std::mutex mu;
  bool tried = false;
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
SideStream g_side[64];

SideStream *side_stream() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  SideStream &ss = g_side[dev];
  std::lock_guard<std::mutex> lock(ss.mu);
  if (!ss.tried) {
    ss.tried = true;
    if (cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess) {
      ss.stream = nullptr;
    }
  }
  return ss.stream ? &ss : nullptr;
}

// Patched layers: the persistent kernel when the batch has a workspace, else the grid kernel
// on the layouts it serves, else the general pipeline.
// `planned` (may be null) is recorded after the planning kernel of the persistent path, or
// before the patched-layer kernel on the other paths.
cudaError_t launch_patched(const kamera::ReuseArgs &a, int n_items, cudaStream_t s,
                           cudaEvent_t planned = nullptr) {
  if (a.smem.fast && a.plan_ws) return kamera::launch_reuse_persist(a, s, planned);
  if (planned) {
    const cudaError_t e = cudaEventRecord(planned, s);
    if (e != cudaSuccess) return e;
  }
  return a.smem.fast ? kamera::launch_reuse_tile(a, n_items, s)
                     : kamera::launch_reuse(a, n_items, s);
}

// Patched layers on the caller's stream, unpatched layers on the side stream at the same time
// (layouts served by the tile kernel); otherwise the two kernels in order on the caller's
// stream. `unpatched` false (a single item patched on every layer, checked on the host): the
// copy kernel would have nothing to do, so only the patched-layer kernel is launched.
cudaError_t launch_both(const kamera::ReuseArgs &a, int n_items, bool patched, cudaStream_t s,
                        bool unpatched = true) {
  if (patched && !unpatched) return launch_patched(a, n_items, s);
  SideStream *ss = (a.smem.fast && patched) ? side_stream() : nullptr;
  if (!ss) {
    cudaError_t e = kamera::launch_reuse_copy(a, s);
    if (e == cudaSuccess && patched) e = launch_patched(a, n_items, s);
    return e;
  }
  std::lock_guard<std::mutex> lock(ss->mu);  // one fork/join at a time per device
  cudaError_t e = cudaEventRecord(ss->fork, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ss->stream, ss->fork, 0);
  if (e == cudaSuccess) e = launch_patched(a, n_items, s);
  if (e == cudaSuccess) e = kamera::launch_reuse_copy(a, ss->stream);
  if (e == cudaSuccess) e = cudaEventRecord(ss->join, ss->stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ss->join, 0);
  return e;
}

// Unpatched layers always stream through the copy kernel. Patched layers take the per-tile
// tensor-core kernel on the layouts it serves (with the tensor engine), else the general
// patched pipeline.
kamera::SmemPlan reuse_plan(const kamera_handle *h, int max_m, int max_run) {
  if (h->engine == kamera::kEngineTensor && kamera::fast_layout(h->lay))
    return kamera::reuse_tile_plan(h->lay, max_m, max_run);
  return kamera::reuse_smem_plan(h->lay, max_m);
}


// Defaults of the handle options (measured on the reorder workload: runs of 3 on patched layers,
// 2 on unpatched ones give the fastest kernels).
constexpr int kDefaultRunTile = 3;
constexpr int kDefaultRunCopy = 2;
constexpr int kMaxRunCopy = 8;

}  // namespace

extern "C" {

kamera_status kamera_create(const kamera_layout *layout, kamera_handle **out) {
  if (!layout || !out) return KAMERA_ERR_INVALID_ARG;
  *out = nullptr;
  DevLayout l;
  const kamera_status st = fill_layout(*layout, &l);
  if (st != KAMERA_OK) return st;
  kamera_handle *h = new (std::nothrow) kamera_handle;
  if (!h) return KAMERA_ERR_INVALID_ARG;
  h->desc = *layout;
  h->lay = l;
  fill_freq(*layout, l, &h->freq);
  h->engine = kamera::kEngineTensor;
  h->run_tile = kDefaultRunTile;
  h->run_copy = kDefaultRunCopy;
  *out = h;
  return KAMERA_OK;
}

kamera_status kamera_set_option(kamera_handle *h, int32_t option, int32_t value) {
  if (!h) return KAMERA_ERR_INVALID_ARG;
  switch (option) {
    case KAMERA_OPT_PATCH_ENGINE:
      if (value != KAMERA_ENGINE_TENSOR && value != KAMERA_ENGINE_CUDA_CORES)
        return KAMERA_ERR_INVALID_ARG;
      h->engine = value == KAMERA_ENGINE_TENSOR ? kamera::kEngineTensor : kamera::kEngineFma;
      return KAMERA_OK;
    case KAMERA_OPT_SHARE_RUN_PATCHED:
      if (value < 1 || value > kamera::kShareBlock) return KAMERA_ERR_INVALID_ARG;
      h->run_tile = value;
      return KAMERA_OK;
    case KAMERA_OPT_SHARE_RUN_UNPATCHED:
      if (value < 1 || value > kMaxRunCopy) return KAMERA_ERR_INVALID_ARG;
      h->run_copy = value;
      return KAMERA_OK;
  }
  return KAMERA_ERR_INVALID_ARG;
}

size_t kamera_batch_workspace_bytes(const kamera_handle *h, int32_t num_items) {
  if (!h || num_items < 0) return 0;
  return kamera::persist_workspace_bytes(h->lay, num_items);
}

kamera_status kamera_set_batch_workspace(kamera_handle *h, void *d_workspace, size_t bytes) {
  if (!h) return KAMERA_ERR_INVALID_ARG;
  if (!d_workspace) {
    if (bytes != 0) return KAMERA_ERR_INVALID_ARG;
    h->ws = nullptr;
    h->ws_bytes = 0;
    return KAMERA_OK;
  }
  if ((reinterpret_cast<uintptr_t>(d_workspace) & 255u) != 0 ||
      bytes < kamera::persist_workspace_bytes(h->lay, 1))
    return KAMERA_ERR_INVALID_ARG;
  h->ws = d_workspace;
  h->ws_bytes = bytes;
  return KAMERA_OK;
}

kamera_status kamera_destroy(kamera_handle *handle) {
  delete handle;
  return KAMERA_OK;
}

const char *kamera_status_string(kamera_status s) {
  switch (s) {
    case KAMERA_OK: return "ok";
    case KAMERA_ERR_INVALID_ARG: return "invalid argument";
    case KAMERA_ERR_UNSUPPORTED: return "unsupported layout or size";
    case KAMERA_ERR_CUDA: return "CUDA runtime error";
  }
  return "unknown status";
}

kamera_status kamera_relocate(const kamera_handle *h, const kamera_pool *pool, int32_t req,
                              int32_t start_tok, int32_t num_tokens, int64_t delta,
                              uint32_t *d_status, kamera_stream_t stream) {
  if (!h || !d_status) return KAMERA_ERR_INVALID_ARG;
  kamera::RelocArgs a;
  a.lay = h->lay;
  kamera_status st = check_pool(h->lay, pool, &a.pool);
  if (st != KAMERA_OK) return st;
  if (num_tokens < 0 || start_tok < 0 || req < 0 || req >= pool->num_reqs)
    return KAMERA_ERR_INVALID_ARG;
  if ((long long)start_tok + num_tokens > (long long)pool->pt_stride * h->lay.page_size)
    return KAMERA_ERR_INVALID_ARG;
  if (delta > (1ll << 62) || delta < -(1ll << 62)) return KAMERA_ERR_INVALID_ARG;
  if (num_tokens == 0 || delta == 0) return KAMERA_OK;  // R(0) = I
  a.req = req;
  a.start_tok = start_tok;
  a.T = num_tokens;
  a.delta = delta;
  a.status = d_status;
  a.freq = h->freq;
  return from_cuda(kamera::launch_relocate(a, reinterpret_cast<cudaStream_t>(stream)));
}

kamera_status kamera_reuse(const kamera_handle *h, const kamera_item *item,
                           const kamera_pool *pool, uint32_t *d_status, kamera_stream_t stream) {
  if (!h || !item || !d_status) return KAMERA_ERR_INVALID_ARG;
  kamera::ReuseArgs a;
  std::memset(&a, 0, sizeof(a));
  a.lay = h->lay;
  kamera_status st = check_pool(h->lay, pool, &a.pool);
  if (st != KAMERA_OK) return st;
  const int chk = kamera::item_check(*item, h->lay, a.pool, 1 << 30, kamera::kMaxRank);
  if (chk != 0) return static_cast<kamera_status>(chk);
  if (item->num_tokens == 0) return KAMERA_OK;
  a.single = *item;
  a.items = nullptr;
  a.n_items = 1;
  a.max_tokens = item->num_tokens;
  a.max_m = item->patch_m;
  a.engine = h->engine;
  a.smem = reuse_plan(h, a.max_m, 1);
  a.status = d_status;
  a.freq = h->freq;
  const cudaStream_t strm = reinterpret_cast<cudaStream_t>(stream);
  // unpatched layers stream through registers; patched layers take the tensor-core pipeline
  const bool patched = item->patch_m > 0 && item->patch_l1 > item->patch_l0;
  const bool all_patched = patched && item->patch_l0 == 0 && item->patch_l1 == h->lay.L;
  return from_cuda(launch_both(a, 1, patched, strm, !all_patched));
}

namespace {

kamera_status batch_reuse(const kamera_handle *h, const kamera_item *d_items, int32_t num_items,
                          int32_t max_tokens, int32_t max_patch_m, const kamera_pool *pool,
                          uint32_t *d_status, kamera_stream_t stream, void *const *events) {
  if (!h || !d_status) return KAMERA_ERR_INVALID_ARG;
  if (num_items < 0 || max_tokens < 0 || max_patch_m < 0) return KAMERA_ERR_INVALID_ARG;
  if (max_patch_m > kamera::kMaxRank) return KAMERA_ERR_UNSUPPORTED;
  kamera::ReuseArgs a;
  std::memset(&a, 0, sizeof(a));
  a.lay = h->lay;
  kamera_status st = check_pool(h->lay, pool, &a.pool);
  if (st != KAMERA_OK) return st;
  if (num_items == 0 || max_tokens == 0) return KAMERA_OK;
  if (!d_items || (reinterpret_cast<uintptr_t>(d_items) & 7u)) return KAMERA_ERR_INVALID_ARG;
  if (num_items > 65535) return KAMERA_ERR_UNSUPPORTED;
  a.items = d_items;
  a.n_items = num_items;
  a.max_tokens = max_tokens;
  a.max_m = max_patch_m;
  a.engine = h->engine;
  a.smem = reuse_plan(h, a.max_m, h->run_tile);
  a.run_copy = h->run_copy;
  a.status = d_status;
  a.freq = h->freq;
  if ((long long)h->lay.ntile * num_items * h->lay.L * h->lay.n_ch > 0x7FFFFFFFll)
    return KAMERA_ERR_UNSUPPORTED;
  if (h->ws && a.smem.fast && max_patch_m > 0 &&
      (reinterpret_cast<uintptr_t>(d_items) & 15u) == 0 &&
      h->ws_bytes >= kamera::persist_workspace_bytes(h->lay, num_items)) {
    const kamera::SmemPlan pp = kamera::reuse_persist_plan(h->lay, a.max_m, h->run_tile);
    if (kamera::persist_batch_ok(h->lay, pp, num_items, max_tokens)) {
      a.smem = pp;
      a.plan_ws = h->ws;
    }
  }
  const cudaStream_t strm = reinterpret_cast<cudaStream_t>(stream);
  auto mark = [&](int i) -> cudaError_t {
    if (!events || !events[i]) return cudaSuccess;
    return cudaEventRecord(static_cast<cudaEvent_t>(events[i]), strm);
  };
  if (!events) return from_cuda(launch_both(a, num_items, max_patch_m > 0, strm));
  // timed: the two kernels in order on the caller's stream, marks around each
  cudaError_t e = mark(0);
  if (e == cudaSuccess) e = kamera::launch_reuse_copy(a, strm);
  if (e == cudaSuccess) e = mark(1);
  if (e == cudaSuccess && max_patch_m > 0)
    e = launch_patched(a, num_items, strm, static_cast<cudaEvent_t>(events[2]));
  else if (e == cudaSuccess)
    e = mark(2);
  if (e == cudaSuccess) e = mark(3);
  return from_cuda(e);
}

}  // namespace

kamera_status kamera_batch_reuse(const kamera_handle *h, const kamera_item *d_items,
                                 int32_t num_items, int32_t max_tokens, int32_t max_patch_m,
                                 const kamera_pool *pool, uint32_t *d_status,
                                 kamera_stream_t stream) {
  return batch_reuse(h, d_items, num_items, max_tokens, max_patch_m, pool, d_status, stream,
                     nullptr);
}

kamera_status kamera_batch_reuse_timed(const kamera_handle *h, const kamera_item *d_items,
                                       int32_t num_items, int32_t max_tokens, int32_t max_patch_m,
                                       const kamera_pool *pool, uint32_t *d_status,
                                       kamera_stream_t stream, void *const events[4]) {
  return batch_reuse(h, d_items, num_items, max_tokens, max_patch_m, pool, d_status, stream,
                     events);
}

kamera_status kamera_patch_inplace(const kamera_handle *h, const kamera_pool *pool, int32_t req,
                                   int32_t start_tok, int32_t num_tokens, const void *patch_u,
                                   const void *patch_vt, int32_t patch_m, int32_t patch_l0,
                                   int32_t patch_l1, int32_t sign, uint32_t *d_status,
                                   kamera_stream_t stream) {
  if (!h || !d_status) return KAMERA_ERR_INVALID_ARG;
  kamera::ReuseArgs a;
  std::memset(&a, 0, sizeof(a));
  a.lay = h->lay;
  kamera_status st = check_pool(h->lay, pool, &a.pool);
  if (st != KAMERA_OK) return st;
  if (sign != 1 && sign != -1) return KAMERA_ERR_INVALID_ARG;
  kamera_item it;
  std::memset(&it, 0, sizeof(it));
  it.patch_u = patch_u;
  it.patch_vt = patch_vt;
  it.num_tokens = num_tokens;
  it.req = req;
  it.start_tok = start_tok;
  it.patch_m = patch_m;
  it.patch_l0 = patch_l0;
  it.patch_l1 = patch_l1;
  const int chk = kamera::inplace_item_check(it, h->lay, a.pool, 1 << 30, kamera::kMaxRank);
  if (chk != 0) return static_cast<kamera_status>(chk);
  if (patch_m == 0 || patch_l0 == patch_l1 || num_tokens == 0) return KAMERA_OK;
  if (!kamera::inplace_layout(h->lay)) return KAMERA_ERR_UNSUPPORTED;
  a.single = it;
  a.items = nullptr;
  a.n_items = 1;
  a.max_tokens = num_tokens;
  a.max_m = patch_m;
  a.engine = kamera::kEngineTensor;
  a.smem = kamera::reuse_tile_plan(h->lay, patch_m, 1);
  a.inplace = 1;
  a.sign = sign;
  a.status = d_status;
  a.freq = h->freq;
  return from_cuda(kamera::launch_reuse_tile(a, 1, reinterpret_cast<cudaStream_t>(stream)));
}

kamera_status kamera_batch_patch_inplace(const kamera_handle *h, const kamera_item *d_items,
                                         int32_t num_items, int32_t max_tokens,
                                         int32_t max_patch_m, const kamera_pool *pool,
                                         int32_t sign, uint32_t *d_status,
                                         kamera_stream_t stream) {
  if (!h || !d_status) return KAMERA_ERR_INVALID_ARG;
  if (num_items < 0 || max_tokens < 0 || max_patch_m < 0) return KAMERA_ERR_INVALID_ARG;
  if (max_patch_m > kamera::kMaxRank) return KAMERA_ERR_UNSUPPORTED;
  if (sign != 1 && sign != -1) return KAMERA_ERR_INVALID_ARG;
  kamera::ReuseArgs a;
  std::memset(&a, 0, sizeof(a));
  a.lay = h->lay;
  kamera_status st = check_pool(h->lay, pool, &a.pool);
  if (st != KAMERA_OK) return st;
  if (num_items == 0 || max_tokens == 0 || max_patch_m == 0) return KAMERA_OK;
  if (!d_items || (reinterpret_cast<uintptr_t>(d_items) & 7u)) return KAMERA_ERR_INVALID_ARG;
  if (num_items > 65535) return KAMERA_ERR_UNSUPPORTED;
  if (!kamera::inplace_layout(h->lay)) return KAMERA_ERR_UNSUPPORTED;
  if ((long long)h->lay.ntile * num_items * h->lay.L * h->lay.n_ch > 0x7FFFFFFFll)
    return KAMERA_ERR_UNSUPPORTED;
  a.items = d_items;
  a.n_items = num_items;
  a.max_tokens = max_tokens;
  a.max_m = max_patch_m;
  a.engine = kamera::kEngineTensor;
  a.smem = kamera::reuse_tile_plan(h->lay, max_patch_m, 1);
  a.inplace = 1;
  a.sign = sign;
  a.status = d_status;
  a.freq = h->freq;
  return from_cuda(
      kamera::launch_reuse_tile(a, num_items, reinterpret_cast<cudaStream_t>(stream)));
}

kamera_status kamera_reanchor(const kamera_handle *h, const kamera_anchor_item *d_items,
                              int32_t num_items, int32_t max_tokens, const kamera_pool *pool,
                              uint32_t *d_status, kamera_stream_t stream) {
  if (!h || !d_status) return KAMERA_ERR_INVALID_ARG;
  if (num_items < 0 || max_tokens < 0) return KAMERA_ERR_INVALID_ARG;
  kamera::AnchorArgs a;
  std::memset(&a, 0, sizeof(a));
  a.lay = h->lay;
  kamera_status st = check_pool(h->lay, pool, &a.pool);
  if (st != KAMERA_OK) return st;
  if (num_items == 0 || max_tokens == 0) return KAMERA_OK;
  if (!d_items || (reinterpret_cast<uintptr_t>(d_items) & 7u)) return KAMERA_ERR_INVALID_ARG;
  if (num_items > 65535 || (long long)h->lay.L * h->lay.n_ch > 65535)
    return KAMERA_ERR_UNSUPPORTED;
  a.items = d_items;
  a.n_items = num_items;
  a.max_tokens = max_tokens;
  a.status = d_status;
  a.freq = h->freq;
  return from_cuda(kamera::launch_reanchor(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t kamera_decode_attention_workspace(const kamera_handle *h, int32_t num_reqs,
                                         int32_t num_q_heads, int32_t max_ctx) {
  if (!h || num_reqs < 0 || num_q_heads < 0 || max_ctx < 0) return 0;
  const int dv = h->lay.kind == KAMERA_GQA ? h->lay.hd : h->lay.latent;
  return kamera::attn_workspace(num_reqs, num_q_heads, max_ctx, dv);
}

kamera_status kamera_decode_attention(const kamera_handle *h, const kamera_pool *pool,
                                      int32_t layer, const void *d_q, int32_t num_reqs,
                                      int32_t num_q_heads, const int32_t *d_ctx_len,
                                      int32_t max_ctx, float scale, float *d_out, float *d_lse,
                                      void *d_workspace, size_t workspace_bytes,
                                      uint32_t *d_status, kamera_stream_t stream) {
  if (!h || !d_status) return KAMERA_ERR_INVALID_ARG;
  kamera::AttnArgs a;
  std::memset(&a, 0, sizeof(a));
  a.lay = h->lay;
  kamera_status st = check_pool(h->lay, pool, &a.pool);
  if (st != KAMERA_OK) return st;
  const kamera::DevLayout &l = h->lay;
  if (layer < 0 || layer >= l.L || num_reqs < 0 || num_q_heads < 1 || max_ctx < 0)
    return KAMERA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return KAMERA_ERR_INVALID_ARG;
  if (num_q_heads > 256) return KAMERA_ERR_UNSUPPORTED;
  if (l.kind == KAMERA_GQA && num_q_heads % l.H != 0) return KAMERA_ERR_INVALID_ARG;
  const int dk = l.kind == KAMERA_GQA ? l.hd : l.latent + l.rope_d;
  const int dv = l.kind == KAMERA_GQA ? l.hd : l.latent;
  if (dk > 1024 || (dv & 7) != 0) return KAMERA_ERR_UNSUPPORTED;
  if (num_reqs > a.pool.num_reqs) return KAMERA_ERR_INVALID_ARG;
  if (num_reqs > 65535) return KAMERA_ERR_UNSUPPORTED;
  if (num_reqs == 0) return KAMERA_OK;
  auto mis = [](const void *p, uintptr_t al) { return !p || (reinterpret_cast<uintptr_t>(p) & (al - 1)); };
  if (mis(d_q, 2) || mis(d_ctx_len, 4) || mis(d_out, 4) || mis(d_lse, 4))
    return KAMERA_ERR_INVALID_ARG;
  const size_t need = kamera::attn_workspace(num_reqs, num_q_heads, max_ctx, dv);
  if (need > 0 && (mis(d_workspace, 4) || workspace_bytes < need)) return KAMERA_ERR_INVALID_ARG;
  a.layer = layer;
  a.q = static_cast<const __nv_bfloat16 *>(d_q);
  a.ctx_len = d_ctx_len;
  a.n_reqs = num_reqs;
  a.hq = num_q_heads;
  a.dk = dk;
  a.dv = dv;
  a.max_ctx = max_ctx;
  a.split = kamera::attn_split_tokens(l);
  a.n_splits = (max_ctx + a.split - 1) / a.split;
  a.scale = scale;
  a.part_o = static_cast<float *>(d_workspace);
  a.part_lse = a.part_o + (size_t)num_reqs * num_q_heads * a.n_splits * dv;
  a.out = d_out;
  a.lse = d_lse;
  a.status = d_status;
  return from_cuda(kamera::launch_attention(a, reinterpret_cast<cudaStream_t>(stream)));
}

kamera_status kamera_rope_phases(const kamera_handle *h, const int64_t *d_deltas,
                                 int32_t num_deltas, float *d_out, kamera_stream_t stream) {
  if (!h || num_deltas < 0) return KAMERA_ERR_INVALID_ARG;
  if (num_deltas == 0) return KAMERA_OK;
  if (!d_deltas || !d_out || (reinterpret_cast<uintptr_t>(d_deltas) & 7u) ||
      (reinterpret_cast<uintptr_t>(d_out) & 3u))
    return KAMERA_ERR_INVALID_ARG;
  return from_cuda(kamera::launch_rope_phases(h->freq, h->lay.npairs,
                                              reinterpret_cast<const long long *>(d_deltas),
                                              num_deltas, d_out,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace kamera {

kamera_status form_patch_args(const float *d_delta, int64_t ld, int64_t delta_stride,
                              int32_t num_problems, int32_t T, int32_t W, const float *d_omega,
                              int64_t omega_stride, int32_t k, int32_t q, int32_t m,
                              const void *d_u, int64_t u_stride, const void *d_vt,
                              int64_t vt_stride, const float *d_sigma) {
  if (num_problems < 0 || T < 1 || W < 1) return KAMERA_ERR_INVALID_ARG;
  if (k < 1 || m < 1 || m > k || q < 0) return KAMERA_ERR_INVALID_ARG;
  if (k > kMaxSketch || k > T || k > W || q > 16) return KAMERA_ERR_UNSUPPORTED;
  if (form_patch_smem(k) > (size_t)kMaxFormSmem) return KAMERA_ERR_UNSUPPORTED;
  if (ld < W || delta_stride < 0 || omega_stride < 0 || u_stride < 0 || vt_stride < 0)
    return KAMERA_ERR_INVALID_ARG;
  if (num_problems > 1 && (u_stride < (int64_t)T * m || vt_stride < (int64_t)m * W))
    return KAMERA_ERR_INVALID_ARG;
  if (num_problems == 0) return KAMERA_OK;
  auto mis = [](const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (!d_delta || !d_omega || !d_u || !d_vt) return KAMERA_ERR_INVALID_ARG;
  if (mis(d_delta, 4) || mis(d_omega, 4) || mis(d_u, 2) || mis(d_vt, 2) ||
      (d_sigma && mis(d_sigma, 4)))
    return KAMERA_ERR_INVALID_ARG;
  return KAMERA_OK;
}

}  // namespace kamera

extern "C" {

size_t kamera_form_patch_workspace(int32_t num_problems, int32_t T, int32_t W, int32_t k) {
  if (num_problems < 0 || T < 0 || W < 0 || k < 0) return 0;
  return kamera::form_patch_workspace(num_problems, T, W, k);
}

kamera_status kamera_form_patch(const float *d_delta, int64_t ld, int64_t delta_stride,
                                int32_t num_problems, int32_t T, int32_t W, const float *d_omega,
                                int64_t omega_stride, int32_t k, int32_t q, int32_t m, void *d_u,
                                int64_t u_stride, void *d_vt, int64_t vt_stride, float *d_sigma,
                                void *d_workspace, size_t workspace_bytes,
                                kamera_stream_t stream) {
  const kamera_status st =
      kamera::form_patch_args(d_delta, ld, delta_stride, num_problems, T, W, d_omega,
                              omega_stride, k, q, m, d_u, u_stride, d_vt, vt_stride, d_sigma);
  if (st != KAMERA_OK || num_problems == 0) return st;
  if (!d_workspace || (reinterpret_cast<uintptr_t>(d_workspace) & 3u)) return KAMERA_ERR_INVALID_ARG;
  if (workspace_bytes < kamera::form_patch_workspace(num_problems, T, W, k))
    return KAMERA_ERR_INVALID_ARG;
  kamera::FormArgs a;
  a.delta = d_delta;
  a.ld = ld;
  a.delta_stride = delta_stride;
  a.omega = d_omega;
  a.omega_stride = omega_stride;
  a.n = num_problems;
  a.T = T;
  a.W = W;
  a.k = k;
  a.q = q;
  a.m = m;
  a.u = static_cast<__nv_bfloat16 *>(d_u);
  a.u_stride = u_stride;
  a.vt = static_cast<__nv_bfloat16 *>(d_vt);
  a.vt_stride = vt_stride;
  a.sigma = d_sigma;
  a.work = static_cast<float *>(d_workspace);
  return from_cuda(kamera::launch_form_patch(a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
