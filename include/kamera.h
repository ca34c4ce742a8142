/*
 * kamera.h — C ABI of the Kamera relocate + patch operator for NVIDIA GB300 (sm_103a).
 *
 * The operator is Eq. 1 of "Kamera: Unified Position-Invariant Multimodal KV Cache for
 * Training-Free Reuse" (§1, §3):
 *
 *     KV^(B|A) = R(delta) * KV(B|empty) + U_m * V_m^T
 *
 * R(delta) re-rotates the RoPE phase of a chunk's stored (canonical) keys by the integer offset
 * delta = p1 - p0 (§3 "Relocate"; exact because RoPE composes, R(delta)R(p0) = R(p1)); values
 * and the MLA latent are never rotated. U_m V_m^T is the rank-m conditioning patch formed at
 * compile time from the top-m SVD of the deficit (§3 "Forming and applying the patch";
 * App. A). The serve step applies both and writes the result into a paged KV pool (App. A
 * "apply_reuse": a per-layer RoPE rotation plus a GEMM into the paged KV cache).
 *
 * Conventions shared by every call:
 *   - All tensors are device memory owned by the caller. The library allocates no device
 *     memory, keeps no pointer after a call returns and never modifies the canonical or patch
 *     stores. The first reuse call on a device that runs both of its kernels creates one
 *     non-blocking stream and two events for that device, kept until the process exits: the
 *     kernel for unpatched layers runs there beside the one for patched layers, forked from and
 *     joined back into the caller's stream, so stream order is as if both ran on it.
 *   - bf16 everywhere for data; float32 arithmetic inside, one round-to-nearest-even to bf16.
 *   - Calls are asynchronous on the given stream (NULL = the legacy default stream).
 *   - Host-checkable errors return synchronously and launch nothing.
 *   - Device-detected errors never trap: the affected rows are not written and a bit is ORed
 *     into the caller's device status word (KAMERA_DEVICE_*). Read it after the stream syncs.
 *   - Destinations of different tokens must not overlap (two tokens mapped to one slot give an
 *     unspecified winner).
 */
#ifndef KAMERA_H
#define KAMERA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* The same object as cudaStream_t. */
typedef struct CUstream_st *kamera_stream_t;

typedef enum kamera_status {
  KAMERA_OK = 0,
  KAMERA_ERR_INVALID_ARG = 1, /* a bad pointer, size, index or descriptor field         */
  KAMERA_ERR_UNSUPPORTED = 2, /* well-formed but outside what the kernels implement      */
  KAMERA_ERR_CUDA = 3         /* a CUDA runtime call failed (launch, attribute, device)  */
} kamera_status;

/* Bits ORed into the device status word. */
#define KAMERA_DEVICE_SLOT_OOB 0x1u /* a page id or page index fell outside the pool or the
                                       page table; that token's row was not written          */
#define KAMERA_DEVICE_BAD_ITEM 0x2u /* kamera_batch_reuse: an item failed the checks that
                                       kamera_reuse makes on the host; none of it was written */
#define KAMERA_DEVICE_TIMEOUT 0x4u  /* a tensor-core tile did not complete within 2 s; its
                                       rows were not written (never expected)               */

/* Attention families (§3 "One mechanism for MLA, GQA, and MHA"). MHA is GQA with one KV head
 * per query head. */
#define KAMERA_GQA 0
#define KAMERA_MLA 1

/* RoPE pairing inside a rope band of width d (the pages do not fix it; both are served):
 * NEOX_HALF pairs dim i with dim i + d/2, INTERLEAVED pairs 2i with 2i+1; pair i turns at
 * inv_freq_i = theta^(-2i/d). */
#define KAMERA_ROPE_NEOX_HALF 0
#define KAMERA_ROPE_INTERLEAVED 1

/* Assignment of rope pairs to the M-RoPE sections (see kamera_layout). */
#define KAMERA_MROPE_CONTIGUOUS 0
#define KAMERA_MROPE_INTERLEAVED 1

/*
 * Layout descriptor: the content | rope split of §3 and Fig. 2.
 *   GQA/MHA: K row = V row = num_kv_heads * head_dim; every K head rotates over its whole
 *            head_dim (rope_dim must equal head_dim); V never rotates.
 *   MLA:     one row = latent_dim (c_KV, never rotated) followed by rope_dim (the decoupled
 *            k_pe band, rotated); there is no V tensor.
 * Patch groups (one rank-m patch each, per patched layer): GQA group 0 = K (width W0 =
 * num_kv_heads*head_dim), group 1 = V (W1 = W0); MLA group 0 = c_KV (W0 = latent_dim),
 * group 1 = k_pe (W1 = rope_dim).
 * Limits: head_dim, latent_dim, rope_dim multiples of 16; rope_dim <= 256; rows <= 16384.
 * M-RoPE (§3 "One mechanism for MLA, GQA, and MHA"; Fig. 2, "64 rope pairs of the 128-d head
 * (16|24|24 -> t,h,w)" and "(24|20|20 -> t,h,w)"): mrope_section = pairs of the t, h and w
 * sections, summing to rope_dim/2, or all zero for 1-D RoPE. Which pair belongs to which
 * section: KAMERA_MROPE_CONTIGUOUS gives pairs [0, s_t) to t, the next s_h to h, the last s_w
 * to w; KAMERA_MROPE_INTERLEAVED gives pair i to h when i % 3 == 1 and i < 3*s_h, to w when
 * i % 3 == 2 and i < 3*s_w, and to t otherwise. A pair of section s turns by delta_s (the
 * item's delta, delta_h or delta_w) times its frequency.
 */
typedef struct kamera_layout {
  int32_t kind;         /* KAMERA_GQA or KAMERA_MLA                                       */
  int32_t num_layers;   /* L >= 1                                                         */
  int32_t page_size;    /* tokens per page >= 1                                           */
  int32_t num_kv_heads; /* GQA: H_kv >= 1; MLA: ignored                                   */
  int32_t head_dim;     /* GQA: head dim; MLA: ignored                                    */
  int32_t latent_dim;   /* MLA: c_KV width; GQA: ignored                                  */
  int32_t rope_dim;     /* GQA: == head_dim; MLA: k_pe width (64 for DeepSeek-V2-style)   */
  int32_t rope_style;   /* KAMERA_ROPE_*                                                  */
  double rope_theta;    /* RoPE base theta > 1                                            */
  int32_t mrope_section[3]; /* M-RoPE pairs of t, h, w; {0, 0, 0} = 1-D RoPE             */
  int32_t mrope_style;  /* KAMERA_MROPE_*; ignored for 1-D RoPE                           */
} kamera_layout;

/*
 * One chunk placement (App. A "apply_reuse(stored, delta, U, V, layer)" for all layers).
 * canon_k : bf16 [L][T][row_k] canonical keys KV(B|empty), stored rotated at p0 (MLA: the
 *           whole c_KV || k_pe row).
 * canon_v : bf16 [L][T][row_v] canonical values (GQA); must be NULL for MLA.
 * patch_u : bf16 [l1-l0][2][T][m]: U*Sigma of group 0 then group 1, per patched layer.
 * patch_vt: bf16 [l1-l0][m*W0 + m*W1]: per patched layer V_m^T of group 0 ([m][W0],
 *           row-major) followed by V_m^T of group 1 ([m][W1]).
 *           Both patch pointers are ignored when patch_m == 0 or patch_l0 == patch_l1.
 * delta   : p1 - p0, any sign (|delta| < 2^62). With M-RoPE, the offset of the t section.
 * delta_h, delta_w: with M-RoPE, the offsets of the h and w sections (|.| < 2^62); ignored for
 *           1-D RoPE. Moving a chunk along the sequence advances all three coordinates
 *           (delta_h = delta_w = delta, Fig. 2 "relocate: +delta to the (t,h,w) position id");
 *           a temporal move changes t alone.
 * num_tokens, req, start_tok: the chunk's T tokens go to logical tokens
 *           [start_tok, start_tok + T) of page-table row req.
 * patch_m : rank, 0 (no patch) or 1..128. Layers in [patch_l0, patch_l1) get the patch.
 * All pointers 16-byte aligned.
 */
typedef struct kamera_item {
  const void *canon_k;
  const void *canon_v;
  const void *patch_u;
  const void *patch_vt;
  int64_t delta;
  int32_t num_tokens;
  int32_t req;
  int32_t start_tok;
  int32_t patch_m;
  int32_t patch_l0;
  int32_t patch_l1;
  int64_t delta_h;
  int64_t delta_w;
} kamera_item;

/*
 * The paged KV pool (§6: the engine's paged KV pool; page size 16 in the reference workloads).
 * k, v      : bf16 [L][num_slots][row]; v is NULL for MLA. 16-byte aligned.
 * num_slots : slots per layer; a multiple of page_size, below 2^31 (UNSUPPORTED otherwise).
 * page_table: int32 [num_reqs][pt_stride] of physical page ids; logical token t of request r
 *             lives at slot page_table[r][t / page_size] * page_size + t % page_size.
 * All device memory, read by the kernels only (page_table) or written (k, v).
 */
typedef struct kamera_pool {
  void *k;
  void *v;
  int64_t num_slots;
  const int32_t *page_table;
  int32_t num_reqs;
  int32_t pt_stride;
} kamera_pool;

typedef struct kamera_handle kamera_handle;

/* Validate a layout and precompute its RoPE frequencies (host only; touches no device).
 * Returns INVALID_ARG / UNSUPPORTED for a bad layout. *out must be freed by kamera_destroy. */
kamera_status kamera_create(const kamera_layout *layout, kamera_handle **out);

/* Free a handle (NULL is accepted). */
kamera_status kamera_destroy(kamera_handle *handle);

/* Short English text for a status code (static storage). */
const char *kamera_status_string(kamera_status status);

/*
 * Options of a handle, for ablations and tuning; a new handle has the defaults, and every call
 * made with the handle after kamera_set_option uses the new value. Not thread-safe against
 * calls that use the same handle at the same time. The pages have no counterpart: these select
 * between implementations of the same operation.
 *   KAMERA_OPT_PATCH_ENGINE: KAMERA_ENGINE_TENSOR (default) forms the rank-m patch on the tensor
 *     cores where the rank is a multiple of 8; KAMERA_ENGINE_CUDA_CORES forms every patch with
 *     float32 FMAs on the CUDA cores (the ablation of the tensor-core path).
 *   KAMERA_OPT_SHARE_RUN_PATCHED: in kamera_batch_reuse, the most members of a group of
 *     placements of one chunk (see kamera_batch_reuse) written from one computed tile on
 *     patched layers, 1..32 (default 3; 1 groups nothing).
 *   KAMERA_OPT_SHARE_RUN_UNPATCHED: the same on layers without a patch, 1..8 (default 2).
 * The bytes written do not depend on any option beyond the rounding of float32 sums. An unknown
 * option or a value out of range returns KAMERA_ERR_INVALID_ARG and changes nothing.
 */
#define KAMERA_OPT_PATCH_ENGINE 1
#define KAMERA_OPT_SHARE_RUN_PATCHED 2
#define KAMERA_OPT_SHARE_RUN_UNPATCHED 3
#define KAMERA_ENGINE_TENSOR 0
#define KAMERA_ENGINE_CUDA_CORES 1

kamera_status kamera_set_option(kamera_handle *handle, int32_t option, int32_t value);

/*
 * Batch workspace of a handle (the pages have no counterpart: it selects how the patched layers
 * of kamera_batch_reuse are scheduled, not what they compute). With a workspace of at least
 * kamera_batch_workspace_bytes(handle, num_items) bytes, a kamera_batch_reuse call of the
 * handle first plans the batch on the device (its groups and a list of its patched rows,
 * written into the workspace) and then runs the patched layers as a persistent kernel: sets of
 * CTAs, one per column tile, each set walking an equal share of the rows' token tiles. Without
 * a workspace, or when the batch does not fit this path, the call runs them as one CTA per
 * (item, layer, channel, column tile) as before. The bytes written to the pool are the same
 * either way.
 * Batches that take the persistent path: GQA/MHA layouts whose patched layers run on the
 * tensor-core tile kernel (NeoX-half pairing, column tiles of 64 or 128 whole-head columns),
 * d_items 16-byte aligned, at most 512 items and num_items x num_layers x 2 <= 8192,
 * KAMERA_OPT_SHARE_RUN_PATCHED at most 4, and a rank small enough for two V_m^T buffers and
 * two CTAs per SM in shared memory (max_patch_m <= 48 where a column tile is 128 wide).
 * kamera_batch_workspace_bytes: bytes for batches of up to num_items items (0 for a NULL
 * handle or num_items < 0).
 * kamera_set_batch_workspace: d_workspace is device memory owned by the caller, 256-byte
 * aligned, of `bytes` bytes (at least kamera_batch_workspace_bytes(handle, 1)); the handle
 * keeps the pointer until it is set again or the handle is destroyed. NULL with bytes 0
 * removes it. Calls that use the same handle's workspace must not run at the same time on
 * the device: order them on one stream (a later call overwrites the plan of an earlier one).
 * Returns KAMERA_ERR_INVALID_ARG (and changes nothing) for a NULL handle, a misaligned or too
 * small workspace, or NULL with bytes != 0.
 */
size_t kamera_batch_workspace_bytes(const kamera_handle *handle, int32_t num_items);
kamera_status kamera_set_batch_workspace(kamera_handle *handle, void *d_workspace, size_t bytes);

/*
 * Survivor relocation, in place (§5 "Sliding-window survival": keep the survivor's KV as-is
 * and apply R(delta); Fig. 2: rotate_k_pe_inplace). Rotates the rope columns of K (GQA/MHA:
 * every head; MLA: the k_pe band only) of logical tokens [start_tok, start_tok+num_tokens)
 * of request req by delta. V and c_KV are neither read nor written. delta == 0 or
 * num_tokens == 0 launches nothing.
 */
kamera_status kamera_relocate(const kamera_handle *handle, const kamera_pool *pool, int32_t req,
                              int32_t start_tok, int32_t num_tokens, int64_t delta,
                              uint32_t *d_status, kamera_stream_t stream);

/*
 * Reorder / recall of one chunk (§5 "Reorder", "Recall"): canonical -> pool with rotation and
 * patch, every layer, K and V (or the MLA row). The item lives in host memory and is checked
 * on the host.
 */
kamera_status kamera_reuse(const kamera_handle *handle, const kamera_item *item,
                           const kamera_pool *pool, uint32_t *d_status, kamera_stream_t stream);

/*
 * Many chunks and requests in one launch. d_items is a device array of num_items items; the
 * host cannot see them, so each is checked on the device against the same rules as
 * kamera_reuse plus num_tokens <= max_tokens and patch_m <= max_patch_m (a failing item sets
 * KAMERA_DEVICE_BAD_ITEM and is skipped). max_tokens sizes the grid; max_patch_m picks the
 * kernel (0..128).
 * Shared chunks (§5 "Reorder": one orbit patch serves every ordering of a chunk): valid items
 * of the same aligned block of 32 consecutive items (items 0-31, 32-63, ...) that name the
 * same canonical rows, length, factors and patched layers (and, for the columns that turn,
 * the same offsets) form a group. A group's members, in item order, are taken a few at a
 * time (3 on patched layers, 2 on the others): each such run is read and computed once and
 * written to each member's own slots. The bytes written are those of separate calls; only
 * the reads and arithmetic are shared.
 */
kamera_status kamera_batch_reuse(const kamera_handle *handle, const kamera_item *d_items,
                                 int32_t num_items, int32_t max_tokens, int32_t max_patch_m,
                                 const kamera_pool *pool, uint32_t *d_status,
                                 kamera_stream_t stream);

/*
 * kamera_batch_reuse with timing marks. The call runs its kernels one after the other on the
 * stream: the layers without a patch (rotation and copies), then the patched layers (tensor-core
 * patch; with a batch workspace, the planning kernel and then the persistent kernel).
 * events[0..3] are CUDA events (cudaEvent_t) recorded before the first kernel, between the
 * unpatched and the patched layers, after the planning kernel (recorded together with events[1]
 * when the batch does not take the persistent path), and after the last kernel; any entry may
 * be NULL, and a NULL `events` makes this call kamera_batch_reuse itself (the kernels side by
 * side). The work done is identical to kamera_batch_reuse.
 */
kamera_status kamera_batch_reuse_timed(const kamera_handle *handle, const kamera_item *d_items,
                                       int32_t num_items, int32_t max_tokens, int32_t max_patch_m,
                                       const kamera_pool *pool, uint32_t *d_status,
                                       kamera_stream_t stream, void *const events[4]);

/*
 * Conditioning switched back on in place (App. E "Context management as reversible state
 * edits": reverting to the context-clean view is a copy of the stored canonical, which
 * kamera_reuse with patch_m = 0 performs; re-applying conditioning is a single rank-m add).
 * For every layer in [patch_l0, patch_l1) and both patch groups (GQA: K and V; MLA: c_KV and
 * k_pe), the cached rows of logical tokens [start_tok, start_tok + num_tokens) of request req
 * become bf16(row + sign * U V_m^T), with one rounding. Nothing rotates: the rows are already
 * in their place. sign = -1 subtracts the same patch.
 * patch_u, patch_vt: the chunk's factors in the kamera_item layout ([l1-l0][2][T][m] and
 * [l1-l0][m*W0 + m*W1], bf16, device), with T = num_tokens.
 * Returns UNSUPPORTED for layouts whose column tiles are not 64 or 128 columns wide (GQA rows
 * not a multiple of the tile width, head_dim 256; MLA k_pe other than 64 or 128). Rows whose
 * page falls outside the pool are skipped with KAMERA_DEVICE_SLOT_OOB. patch_m == 0,
 * patch_l0 == patch_l1 or num_tokens == 0 launches nothing.
 */
kamera_status kamera_patch_inplace(const kamera_handle *handle, const kamera_pool *pool,
                                   int32_t req, int32_t start_tok, int32_t num_tokens,
                                   const void *patch_u, const void *patch_vt, int32_t patch_m,
                                   int32_t patch_l0, int32_t patch_l1, int32_t sign,
                                   uint32_t *d_status, kamera_stream_t stream);

/*
 * kamera_patch_inplace for many chunks in one launch. d_items is a device array of
 * kamera_item; only num_tokens, req, start_tok, patch_u, patch_vt, patch_m, patch_l0 and
 * patch_l1 are read (the canonical pointers and delta are ignored). Each item is checked on
 * the device against the rules of kamera_patch_inplace plus num_tokens <= max_tokens and
 * patch_m <= max_patch_m; a failing item sets KAMERA_DEVICE_BAD_ITEM and is skipped. Items
 * must not cover the same rows.
 */
kamera_status kamera_batch_patch_inplace(const kamera_handle *handle, const kamera_item *d_items,
                                         int32_t num_items, int32_t max_tokens,
                                         int32_t max_patch_m, const kamera_pool *pool,
                                         int32_t sign, uint32_t *d_status,
                                         kamera_stream_t stream);

/*
 * The RoPE phases the kernels use: for each of num_deltas offsets d_deltas[n] (device int64)
 * and each rope pair i of the layout, (cos, sin) of delta * inv_freq_i with inv_freq_i =
 * theta^(-2i/d), written as float32 pairs to d_out[n][rope_dim/2][2] (device). The angle is
 * range-reduced exactly (a Q0.64 fixed-point product modulo one turn) before a float32
 * sincospi, so large |delta| loses no accuracy (§3 "Relocate" re-rotates by delta;
 * inv_freq from the standard RoPE of Su et al.). Offsets with |delta| > 2^62 give NaN.
 */
kamera_status kamera_rope_phases(const kamera_handle *handle, const int64_t *d_deltas,
                                 int32_t num_deltas, float *d_out, kamera_stream_t stream);

/*
 * Re-anchoring of keys stored before rotation (QV-PIC, "Model-Native Template-Conditioned
 * Compilation", Eq. 2: K = R(K_bar, P(q)); values are position-independent and stitched as
 * they are). Each token is rotated from zero to its own absolute position, so there is no
 * common offset:
 * canon_k  : bf16 [L][T][row_k] keys before any rotation (MLA: the whole c_KV || k_pe row).
 * canon_v  : bf16 [L][T][row_v] values (GQA); must be NULL for MLA.
 * positions: int64, device. 1-D RoPE: [T], the position of each token. M-RoPE layouts:
 *            [T][3], the (t, h, w) position of each token; a pair of section s turns by
 *            position[s] times its frequency. Any int64 (the angle is reduced exactly).
 * num_tokens, req, start_tok: the T tokens go to logical tokens [start_tok, start_tok + T) of
 *            page-table row req.
 * canon_k / canon_v 16-byte aligned, positions 8-byte aligned.
 */
typedef struct kamera_anchor_item {
  const void *canon_k;
  const void *canon_v;
  const int64_t *positions;
  int32_t num_tokens;
  int32_t req;
  int32_t start_tok;
  int32_t reserved; /* set to 0 */
} kamera_anchor_item;

/*
 * Re-anchors num_items items (a device array of kamera_anchor_item) into the pool in one
 * launch: rope columns of K rotated per token (one float32 rotation, one rounding to bf16),
 * the MLA latent and all of V copied byte for byte. Items are checked on the device (the rules
 * above, plus num_tokens <= max_tokens); a failing item sets KAMERA_DEVICE_BAD_ITEM and is
 * skipped. Rows whose page falls outside the pool are skipped with KAMERA_DEVICE_SLOT_OOB.
 * max_tokens sizes the grid. Items must not map tokens to the same slot.
 */
kamera_status kamera_reanchor(const kamera_handle *handle, const kamera_anchor_item *d_items,
                              int32_t num_items, int32_t max_tokens, const kamera_pool *pool,
                              uint32_t *d_status, kamera_stream_t stream);

/*
 * Decode attention over the paged pool: the consumer-side check that the rows the other calls
 * write are the KV an attention kernel reads (§1: attention over KV(A) || KV(B) equals
 * attending each part separately and merging by softmax mass, o = (1 - mu) o_B + mu o_A, the
 * log-sum-exp merge of FlashAttention). One query token per request and query head:
 *   s_t = scale * q . K_t,  o = sum_t softmax(s)_t V_t,  lse = log sum_t exp(s_t),
 * over the request's logical tokens [0, ctx_len[r]) of pool layer `layer`, gathered through
 * page-table row r. The context is cut into splits of 256 tokens; each split's (o, lse) is
 * computed independently and the splits are merged by their log-sum-exp.
 *   GQA: K_t, V_t = head (h / (num_q_heads / num_kv_heads)) of the K and V rows; Dk = Dv =
 *        head_dim; num_q_heads a multiple of num_kv_heads.
 *   MLA: the absorbed form: K_t = the whole c_KV || k_pe row (Dk = latent + rope), V_t = its
 *        c_KV part (Dv = latent); every query head reads the one latent head.
 * d_q      : bf16 [num_reqs][num_q_heads][Dk], device.
 * d_ctx_len: int32 [num_reqs], device; each in [0, max_ctx] (a larger one sets
 *            KAMERA_DEVICE_BAD_ITEM and that request's outputs are not written).
 * d_out    : float32 [num_reqs][num_q_heads][Dv]; d_lse: float32 [num_reqs][num_q_heads]
 *            (natural log). An empty context gives o = 0 and lse = -inf.
 * d_workspace: at least kamera_decode_attention_workspace(handle, num_reqs, num_q_heads,
 *            max_ctx) bytes of device memory, 4-byte aligned (0 bytes when max_ctx is 0);
 *            contents ignored and left undefined.
 * Requests are page-table rows 0 .. num_reqs - 1 (num_reqs <= the pool's num_reqs).
 * Pages outside the pool set KAMERA_DEVICE_SLOT_OOB and their tokens are left out. Limits:
 * num_q_heads <= 256 (GQA: a multiple of num_kv_heads), Dk <= 1024.
 */
size_t kamera_decode_attention_workspace(const kamera_handle *handle, int32_t num_reqs,
                                         int32_t num_q_heads, int32_t max_ctx);

kamera_status kamera_decode_attention(const kamera_handle *handle, const kamera_pool *pool,
                                      int32_t layer, const void *d_q, int32_t num_reqs,
                                      int32_t num_q_heads, const int32_t *d_ctx_len,
                                      int32_t max_ctx, float scale, float *d_out, float *d_lse,
                                      void *d_workspace, size_t workspace_bytes,
                                      uint32_t *d_status, kamera_stream_t stream);

/*
 * Patch forming (§3 "Forming and applying the patch"; App. A "form_patch"): for each of
 * num_problems deficits Delta = KV(B|A) - R(delta)KV(B|empty), one (layer, group) each, the
 * top-m factors U*Sigma [T x m] and V_m^T [m x W] in the patch store's bf16 format. The
 * factors come from the randomized range finder with q power iterations and the SVD of the
 * small projection (Halko, Martinsson & Tropp, SIAM Review 2011, Alg. 4.4 and 5.1):
 *   Y = Delta Omega; Q = orth(Y); q times: Z = orth(Delta^T Q), Q = orth(Delta Z);
 *   B^T = Delta^T Q = V_B Sigma Ut^T; U*Sigma = Q Ut_m Sigma_m; V_m^T = (B^T Ut_m)^T / Sigma_m,
 * sigma descending, each row of V_m^T signed so that its largest-magnitude entry (the first on
 * a tie) is positive, the matching column of U*Sigma flipped with it. float32 arithmetic; the
 * products with Delta run on the tensor cores with float32 operands split into two tf32 terms,
 * which keeps them float32-accurate. A chain of kernels is launched on `stream`; the call
 * returns once they are queued.
 *   d_delta     : float32; problem i is the [T][W] matrix at d_delta + i*delta_stride with row
 *                 stride ld >= W (elements).
 *   d_omega     : float32 [W][k] random test matrix of problem i at d_omega + i*omega_stride
 *                 (omega_stride 0: one matrix for all problems), drawn by the caller.
 *   k           : sketch width, m <= k <= min(T, W, 96).
 *   q           : power iterations, 0..16.   m : rank kept, 1..k.
 *   d_u, d_vt   : bf16 outputs, problem i's U*Sigma [T][m] at d_u + i*u_stride and V_m^T
 *                 [m][W] at d_vt + i*vt_stride (elements). The strides place the results
 *                 straight into a kamera_item's patch_u / patch_vt: for group g of layers
 *                 l0..l1, u at patch_u + g*T*m with u_stride 2*T*m, vt at patch_vt + g*m*W0 with
 *                 vt_stride m*(W0 + W1). Outputs of different problems must not overlap.
 *   d_sigma     : float32 [num_problems][m] singular values, or NULL.
 *   d_workspace : device scratch of at least kamera_form_patch_workspace(num_problems, T, W, k)
 *                 bytes, 4-byte aligned; contents on entry are ignored and left undefined.
 *                 That is num_problems * 4 bytes * ((T + W) * k + nt * (k^2 + 3k) + 9k^2 + k
 *                 + 4) with nt = ceil(max(T, W) / 128), the float count per problem rounded up
 *                 to a multiple of 4.
 * Columns past the numerical rank of Delta come out with sigma near zero (zero factors for an
 * exactly zero deficit). Host checks return INVALID_ARG (bad pointer, size, stride, too small
 * a workspace) or UNSUPPORTED (k above the limit) and launch nothing. A device-side wait that
 * runs out of time (2 s) leaves NaN in the problem's outputs.
 */
size_t kamera_form_patch_workspace(int32_t num_problems, int32_t T, int32_t W, int32_t k);

kamera_status kamera_form_patch(const float *d_delta, int64_t ld, int64_t delta_stride,
                                int32_t num_problems, int32_t T, int32_t W, const float *d_omega,
                                int64_t omega_stride, int32_t k, int32_t q, int32_t m, void *d_u,
                                int64_t u_stride, void *d_vt, int64_t vt_stride, float *d_sigma,
                                void *d_workspace, size_t workspace_bytes,
                                kamera_stream_t stream);

/*
 * kamera_form_patch without a caller workspace, for callers that cannot allocate device memory
 * where they call it: a serving engine that hands all device memory left after the weights to
 * its paged KV pool at start-up (so an allocation at patch-forming time would fail or evict
 * cache), or host code with no device allocator of its own. The Kamera paper has no
 * counterpart to this call; it is kamera_form_patch with the workspace taken from a fixed
 * array of KAMERA_FORM_PATCH_SCRATCH_BYTES in this library's device memory.
 *   - Allocates nothing: no cudaMalloc/cudaFree and no allocating library routine.
 *   - Arguments, outputs and results are those of kamera_form_patch, and so are its argument
 *     errors, which are checked first. Then a call whose kamera_form_patch_workspace(
 *     num_problems, T, W, k) exceeds KAMERA_FORM_PATCH_SCRATCH_BYTES (32 MiB: e.g. more than 93
 *     deficits of 1024 x 512 at k = 40) returns KAMERA_ERR_UNSUPPORTED and launches nothing.
 *   - Set-up: the first call on a device, with that device current, looks up the array's
 *     device address and loads and configures the kernels; a failure returns KAMERA_ERR_CUDA.
 *     CUDA reserves the array when it loads this library's device code, which by default
 *     (lazy module loading) happens at that set-up, not earlier. A call with num_problems = 0
 *     and otherwise valid arguments does the set-up alone: make one on each device before
 *     handing that device's free memory to a pool, and before any stream capture. After the
 *     set-up, calls take no device memory. A device reset (cudaDeviceReset) discards the
 *     set-up's address: do not use this call on a device after resetting it.
 *   - Nothing has to start at zero: the array's contents on entry are ignored and left
 *     undefined.
 *   - One array per device: calls on the same device that overlap in time (different
 *     streams, or host threads without ordering) race on it and give undefined results.
 *     Order them on one stream, or synchronise between them.
 */
#define KAMERA_FORM_PATCH_SCRATCH_BYTES (32u << 20)

kamera_status kamera_form_patch_static_scratch(const float *d_delta, int64_t ld,
                                               int64_t delta_stride, int32_t num_problems,
                                               int32_t T, int32_t W, const float *d_omega,
                                               int64_t omega_stride, int32_t k, int32_t q,
                                               int32_t m, void *d_u, int64_t u_stride,
                                               void *d_vt, int64_t vt_stride, float *d_sigma,
                                               kamera_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KAMERA_H */
