/*
 * g4attn — batch-invariant hybrid decoder attention for Gemma-4-31B-class models on one
 * NVIDIA GB300 (sm_103a). C ABI: plain pointers and sizes only.
 *
 * What it computes. The attention cores of the RL-Kernel RFC "[RFC][Gemma-4-31B-it]
 * [CUDA/ROCm] WS1/WS2 kernel roadmap, ablation matrix and integration plan":
 *   - section 2, "Checkpoint fingerprint" table: 32 query heads; sliding layers with 16 KV
 *     heads of dim 256, window 1024, standard RoPE theta 1e4; global layers with 4 KV heads
 *     of dim 512, K==V (attention_k_eq_v), proportional p-RoPE, partial factor 0.25,
 *     theta 1e6; 262144 positions;
 *   - section 5, work-item rows sliding_rope_d256, global_proportional_p_rope,
 *     sliding_attention_core, global_attention_core, hybrid_kv_cache_contract and
 *     global_k_eq_v_projection;
 *   - section 4, "Numerical contract": fixed fp32 accumulation; a reduction order that does
 *     not depend on batch size, batch position, packing, launch geometry, SM count or
 *     occupancy; no dynamic split-KV and no cross-CTA atomics in the arithmetic; no TF32 or
 *     fast-math; casts only at declared points; unsupported geometry fails closed; runtime
 *     provenance.
 *
 * Arithmetic (fixed for every call):
 *   q' = RoPE(q, pos), k' = RoPE(k, pos) on the leading R half-split pairs (element t pairs
 *   with t + D/2; pair t turns by pos * theta^(-2t/D); R = D/2 on sliding layers, D/8 on
 *   global ones; the other pairs pass unchanged). Query i sees keys j <= i, and on sliding
 *   layers only i - j <= window - 1. o_i = sum_j softmax_j(scale * q'_i . k'_j) v_j, with
 *   v_j = the stored V (sliding) or the stored un-rotated S (global, K==V).
 *   Declared bf16 (round-to-nearest-even) casts: roped q, roped sliding K written to the
 *   cache, roped global K columns, the softmax probabilities P before P.V, and the output.
 *   Everything else accumulates in fp32. The softmax exponentials are the multi-function
 *   unit's 2^x (PTX ex2.approx.ftz.f32, deterministic; weights below 2^-126 flush to zero), a
 *   declared choice that g4attn_provenance records.
 *
 * Memory. Every tensor is a device buffer owned by the caller. The library allocates no
 * device memory: its only device-side state is static (the RoPE cos/sin tables, filled once
 * per device on the first call, one 32-bit error word, and the scratch buffer of
 * g4attn_decode_static). All calls are stream-ordered
 * on `stream` (a cudaStream_t; NULL = the legacy default stream) and never synchronise,
 * except g4attn_status_sync.
 *
 * Layouts (row-major, bf16 = IEEE bfloat16 in 2 bytes):
 *   q, out         [T][n_q_heads][head_dim]           query rows / output rows
 *   k, v           [T][n_kv_heads][head_dim]          new key / value rows of a prefill
 *   k_new, v_new   [B][n_kv_heads][head_dim]          the decode token's key / value
 *   cache->k       one page-head block of 16 keys x head_dim dims per (page, KV head),
 *                  16*head_dim contiguous bf16 at k + (page*n_kv_heads + head)*16*head_dim,
 *                  stored as 8x8 core matrices (key j, dim d):
 *                    sliding (D 256): [j/8][d/8][j%8][d%8]            = [2][32][8][8]
 *                    global  (D 512): [d/256][j/8][(d%256)/8][j%8][d%8] = [2][2][32][8][8]
 *                  sliding K' (roped) or global S (un-rotated, K==V)
 *   cache->v       sliding: V, 16 keys x 256 dims per (page, KV head) at the same place as k's
 *                  block, stored as two contiguous 128-dim halves of 8x8 core matrices:
 *                    [d/128][j/8][(d%128)/8][j%8][d%8]                 = [2][2][16][8][8]
 *                  global: NULL
 *   cache->k_rot   global only (NULL on sliding layers): p-RoPE(S) on the 128 rotated
 *                  columns d in [0,64) U [256,320), 2048 bf16 per (page, KV head) at
 *                  k_rot + (page*n_kv_heads + head)*2048, as [d/256][j/8][(d%64)/8][j%8][d%8].
 *                  Written by the library with S; it spares the prefill kernels from
 *                  rotating every key tile again for every query tile and head.
 *   page_table     int32 [B][max_pages]: physical page of logical page i of sequence b
 *                  (keys 16i .. 16i+15). Entries that no call needs may hold anything.
 *   All pointers 16-byte aligned.
 *
 * Errors. Host-side checks run before any launch and return G4_ERR_INVALID (bad pointer,
 * size or alignment) or G4_ERR_UNSUPPORTED (a geometry other than the two layer kinds
 * below); nothing is launched then. Problems only the device can see (a page-table entry
 * outside [0, num_pages), a position >= 262144 or beyond the page table, a bad image span
 * (g4attn_prefill_vision), a bounded wait that ran out) set bits in a device error word, and the
 * affected work is skipped; read and clear the word with g4attn_status_sync. Kernels never trap.
 * (The sliding prefill kernel also refuses, as G4_ERR_DEVICE, a launch whose dynamic shared
 * memory does not start 1024-byte aligned; a kernel without static shared memory always does.)
 */
#ifndef G4ATTN_H
#define G4ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  G4_OK = 0,
  G4_ERR_INVALID = 1,      /* bad argument: NULL pointer, size, alignment, range */
  G4_ERR_UNSUPPORTED = 2,  /* geometry or dtype outside the two supported layer kinds */
  G4_ERR_CUDA = 3,         /* a CUDA runtime call failed (launch, table upload) */
  G4_ERR_TIMEOUT = 4,      /* a bounded device wait ran out (device error word) */
  G4_ERR_DEVICE = 5,       /* device-detected bad data: page index or position (error word) */
  G4_ERR_SCRATCH = 6       /* g4attn_decode_static: the step needs more than the static scratch */
} g4_status;

/* Size of the static device scratch buffer behind g4attn_decode_static (per device). */
#define G4ATTN_DECODE_STATIC_SCRATCH_BYTES ((size_t)32 << 20)

typedef enum { G4_SLIDING = 0, G4_GLOBAL = 1 } g4_kind;

/* One attention layer. Supported (anything else: G4_ERR_UNSUPPORTED):
 *   sliding: kind 0, n_q_heads 32, n_kv_heads 16, head_dim 256, 1 <= window <= 262144,
 *            rope_theta 1e4, rope_partial 1.0, kv_shared 0;
 *   global:  kind 1, n_q_heads 32, n_kv_heads 4, head_dim 512, window 0,
 *            rope_theta 1e6, rope_partial 0.25, kv_shared 1.
 * Or one tensor-parallel rank's slice of either (RFC section 5, ws2_tp2, ws2_tp4 and
 * ws2_tp8_kv_replication): with tp in {2, 4, 8} ranks, n_q_heads 32/tp and n_kv_heads 16/tp
 * (sliding) or max(1, 4/tp) (global; at tp = 8 ranks 2g and 2g+1 both hold KV head g). The rank's
 * q, out, k, v and cache hold only its heads, in the same layouts with those head counts; query
 * head h of the slice reads KV head h / (n_q_heads / n_kv_heads) of the slice. Each head's rows
 * get the bits the full layer gives that head: the arithmetic of a head never involves another.
 * softmax_scale: any finite value > 0 (1/sqrt(head_dim) is the model's). */
typedef struct {
  int32_t kind;
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t window;         /* keys seen including the query's own; 0 = unbounded */
  float rope_theta;
  float rope_partial;
  float softmax_scale;
  int32_t kv_shared;      /* 1: K==V, the cache holds one tensor S */
} g4attn_layer;

/* Optional per-head RMS norms of the raw projections, applied before RoPE (RFC section 5, work
 * item qk_rmsnorm_d256_d512; TensorFold "cuda gemma4: images on the 31B", tf_qk_rows_once, which
 * can also norm v by a unit RMS norm). For a head vector x of head_dim elements:
 *   n(x) = x / sqrt(mean(x^2) + eps), computed in fp32 before the rotation and the declared cast;
 *   q -> q_weight * n(q)   when q_weight is set,
 *   k -> k_weight * n(k)   when k_weight is set,
 *   v -> n(v)              when v_norm is 1 (a unit norm, no weight).
 * On a K==V (global) layer the one projection S gives K = k_weight * n(S) and V = n(S): the
 * cache stores n(S) once, the k_rot pages hold RoPE(k_weight * n(S)), and the library carries
 * k_weight into the queries' un-rotated dims, where the attention reads K from the stored S.
 * There k_weight and v_norm must come together (both or neither; G4_ERR_UNSUPPORTED otherwise).
 * The weights are whatever multiplies the normalised vector: for a checkpoint that stores a
 * zero-centred Gemma weight g, pass 1 + g. Decode queries are normed (and, on K==V layers,
 * multiplied by k_weight on their un-rotated dims) into `out` first, with a bf16 cast there,
 * one declared cast more than prefill has. */
typedef struct {
  const void* q_weight;   /* bf16 [head_dim], device, 16-byte aligned, or NULL: queries not normed */
  const void* k_weight;   /* bf16 [head_dim], device, 16-byte aligned, or NULL: keys not normed */
  int32_t v_norm;         /* 1: values get the unit RMS norm; 0: they do not */
  float eps;              /* added to the mean square; finite and > 0 (Gemma uses 1e-6) */
} g4attn_norms;

/* A paged bf16 KV cache of one layer (RFC section 5, hybrid_kv_cache_contract). */
typedef struct {
  void* k;                /* sliding: roped K'; global: the shared S */
  void* v;                /* sliding: V; global: NULL */
  void* k_rot;            /* global: roped rotated columns of S; sliding: NULL */
  int32_t num_pages;      /* physical pages in k (and v, k_rot) */
  int32_t page_size;      /* keys per page; must be 16 */
} g4attn_cache;

/* RoPE / p-RoPE of a [T][H][head_dim] bf16 tensor (RFC section 5, sliding_rope_d256 and
 * global_proportional_p_rope). out[r][h] = bf16(RoPE(x[r][h], pos[r])). Pairs t >= R are
 * copied bit for bit. x and out may be the same buffer. pos: int32 [T], device, each in
 * [0, 262144) (others set G4_ERR_DEVICE and leave the row unwritten). T >= 0, H >= 1. */
g4_status g4attn_rope_apply(const g4attn_layer* layer, const void* x, const int32_t* pos,
                            int32_t T, int32_t H, void* out, void* stream);

/* Prefill, or one chunk of a chunked prefill, for B sequences (RFC section 5,
 * sliding_attention_core / global_attention_core). Sequence b owns rows
 * q_start[b] .. q_start[b]+q_len[b]-1 of q, k, v and out; they are its positions
 * ctx_start[b] .. ctx_start[b]+q_len[b]-1. Keys at positions < ctx_start[b] must already be
 * in the cache. The call first writes the new rows' K'/V (sliding) or S (global) into the
 * cache through page_table, then computes out for those rows (two launches; the queries are
 * rotated inside the attention kernel). Rows of out that belong to no
 * sequence are not written. q_start, q_len, ctx_start: int32 [B], device, read on the device
 * (q_len 0 is allowed); sequences' row ranges must not overlap and must lie inside [0, T) (a
 * range that does not is refused on the device: none of its rows is read or written, and
 * G4_ERR_DEVICE is reported). T: rows in q/k/v/out.
 * v: NULL on global layers (K==V). Launch geometry depends on T, B and the layer only. */
g4_status g4attn_prefill(const g4attn_layer* layer, const void* q, const void* k, const void* v,
                         int32_t T, const int32_t* q_start, const int32_t* q_len,
                         const int32_t* ctx_start, int32_t B, const g4attn_cache* cache,
                         const int32_t* page_table, int32_t max_pages, void* out, void* stream);

/* g4attn_prefill in two steps, for callers that schedule or time them apart (RFC section 5,
 * hybrid_kv_cache_contract for the append, sliding_attention_core / global_attention_core and
 * sliding_rope_d256 / global_proportional_p_rope for the attention). g4attn_prefill is exactly
 * g4attn_kv_append followed by g4attn_prefill_attend with its q on one stream.
 * g4attn_prefill_attend: the attention step over the cache and page table the append filled; it
 *   writes the output rows of the sequences into `out` and no other row. Arguments as
 *   g4attn_prefill without k and v. q: the raw query rows [T][Hq][D] (16-byte aligned), which the
 *   attention kernel rotates itself, with the angles, rotation and bf16 cast of the declared
 *   roped-q cast point; or NULL, when g4attn_prefill_stage has staged the roped queries in `out`
 *   (the staged form, then overwritten with the output). out must be 16-byte aligned when T > 0.
 *   Calling it with q NULL on rows that were not staged gives meaningless (but bounded, fault-free)
 *   output.
 * g4attn_prefill_stage: the staged form's first step: the cache append of the new rows, plus the
 *   declared bf16 cast of the roped queries written into the sequences' rows of `out`. Arguments
 *   and errors as g4attn_prefill. Stage, then attend with q NULL, gives the same bits as
 *   g4attn_prefill; it costs one more pass over q and out. */
g4_status g4attn_prefill_stage(const g4attn_layer* layer, const void* q, const void* k, const void* v,
                               int32_t T, const int32_t* q_start, const int32_t* q_len,
                               const int32_t* ctx_start, int32_t B, const g4attn_cache* cache,
                               const int32_t* page_table, int32_t max_pages, void* out, void* stream);
g4_status g4attn_prefill_attend(const g4attn_layer* layer, const void* q, int32_t T, const int32_t* q_start,
                                const int32_t* q_len, const int32_t* ctx_start, int32_t B,
                                const g4attn_cache* cache, const int32_t* page_table, int32_t max_pages,
                                void* out, void* stream);

/* g4attn_prefill, g4attn_kv_append and g4attn_decode with the per-head norms of g4attn_norms
 * (RFC section 5, qk_rmsnorm_d256_d512, fused into the staging of each call) applied to the raw
 * q, k and v they are given (norms NULL: exactly the plain calls). A
 * sequence's history must have been appended with the same norms. Errors as the plain calls,
 * plus G4_ERR_INVALID for a bad eps, v_norm or weight alignment, and G4_ERR_UNSUPPORTED for a
 * K==V layer whose key norm and value norm do not come together. */
g4_status g4attn_prefill_normed(const g4attn_layer* layer, const g4attn_norms* norms, const void* q,
                                const void* k, const void* v, int32_t T, const int32_t* q_start,
                                const int32_t* q_len, const int32_t* ctx_start, int32_t B,
                                const g4attn_cache* cache, const int32_t* page_table, int32_t max_pages,
                                void* out, void* stream);
g4_status g4attn_kv_append_normed(const g4attn_layer* layer, const g4attn_norms* norms, const void* k,
                                  const void* v, int32_t T, const int32_t* q_start, const int32_t* q_len,
                                  const int32_t* ctx_start, int32_t B, const g4attn_cache* cache,
                                  const int32_t* page_table, int32_t max_pages, void* stream);
g4_status g4attn_decode_normed(const g4attn_layer* layer, const g4attn_norms* norms, const void* q,
                               const void* k_new, const void* v_new, const int32_t* seq_len, int32_t B,
                               const g4attn_cache* cache, const int32_t* page_table, int32_t max_pages,
                               void* out, void* workspace, size_t workspace_bytes, void* stream);

/* g4attn_prefill_normed with the vision-token mask: the tokens of one image see each other in
 * both directions, on top of the layer's own mask (model card "Gemma 4 31B":
 * use_bidirectional_attention="vision"; RFC section 5, multimodal_bidirectional_mask). Available
 * on both layer kinds: the RFC places the mask in global attention, TensorFold's engine on the
 * sliding layers (where an image row sees all of its image past the window); the caller passes
 * spans to the layers it wants.
 *   span  int32 [T][2], device, 8-byte aligned, or NULL (then exactly g4attn_prefill_normed).
 *         Row t (a memory row, indexed like q) holds the image span [s0, s1) of absolute
 *         positions that its token belongs to; s1 <= s0 marks a text row. Gap rows are not read.
 *         A row's span must hold the row's position and end by ctx_start + q_len of its
 *         sequence (an image lies within one call: its keys are appended by the same call), and
 *         all rows of one image carry the same span. Else the device sets G4_ERR_DEVICE (read by
 *         g4attn_status_sync); the row then falls back to the layer mask and its output is not
 *         the masked attention.
 * Each row then sees one run of keys, lo .. hi: the layer mask's run widened to its image. A
 * decode query is a text token, so decoding takes no spans. Other errors as
 * g4attn_prefill_normed; a misaligned span gives G4_ERR_INVALID before any launch. */
g4_status g4attn_prefill_vision(const g4attn_layer* layer, const g4attn_norms* norms, const void* q,
                                const void* k, const void* v, int32_t T, const int32_t* q_start,
                                const int32_t* q_len, const int32_t* ctx_start, int32_t B, const int32_t* span,
                                const g4attn_cache* cache, const int32_t* page_table, int32_t max_pages,
                                void* out, void* stream);

/* One decode step with the prefill's bits (RFC section 1: training and rollout give exactly equal
 * selected-token log-probabilities in strict mode; section 5, hybrid_kv_cache_contract: the
 * prefill / chunked-prefill / decode handoff). Same arguments and row conventions as
 * g4attn_decode_normed (norms may be NULL), but the step runs as B one-row prefill chunks through
 * the prefill kernels: request b's output row is bit for bit the row a prefill of its whole
 * sequence computes at position seq_len[b] - 1 (for any batch and chunking of that prefill),
 * which g4attn_decode's split-key kernels do not give. It costs more than g4attn_decode: a
 * query tile of the tensor-core kernels holds one row.
 *   workspace  device, 16-byte aligned, at least g4attn_decode_exact_workspace_bytes(B) bytes
 *              (the rows of the B chunks; a g4attn_decode workspace is always large enough).
 * A request with seq_len[b] < 1 computes nothing and sets G4_ERR_DEVICE. */
g4_status g4attn_decode_exact(const g4attn_layer* layer, const g4attn_norms* norms, const void* q,
                              const void* k_new, const void* v_new, const int32_t* seq_len, int32_t B,
                              const g4attn_cache* cache, const int32_t* page_table, int32_t max_pages,
                              void* out, void* workspace, size_t workspace_bytes, void* stream);
/* Bytes of workspace g4attn_decode_exact needs for B requests (RFC section 5,
 * hybrid_kv_cache_contract: the rows of the B one-row chunks and their page-table rows,
 * int32 [4][B]); 0 when B <= 0. */
size_t g4attn_decode_exact_workspace_bytes(int32_t B);

/* Writes the K'/V (sliding) or S (global) rows of a prefill batch into the paged cache
 * without computing attention: the first step of g4attn_prefill on its own (RFC section 5,
 * hybrid_kv_cache_contract). Same row conventions and errors as g4attn_prefill; v NULL on
 * global layers. */
g4_status g4attn_kv_append(const g4attn_layer* layer, const void* k, const void* v, int32_t T,
                           const int32_t* q_start, const int32_t* q_len, const int32_t* ctx_start,
                           int32_t B, const g4attn_cache* cache, const int32_t* page_table,
                           int32_t max_pages, void* stream);

/* Context parallelism of a global (K==V) layer over keys (RFC section 5, ws2_tp4_cp2 and
 * cp_sliding_window_policy; section 4 rule 3: a split is allowed only with a merge tree fixed by the
 * contract). A sequence's keys are split into contiguous ranges, each held by one rank (its cache
 * need hold only its range's keys); every rank computes, for the query rows it is given, a partial
 * over its own keys, and the partials are merged in rank order.
 * g4attn_prefill_partial: g4attn_prefill_attend (with raw q) restricted to keys
 *   key_begin[b] .. key_end[b]-1 of sequence b (int32 [B], device; the causal mask still applies,
 *   and a row with no such key gets an empty partial). Instead of bf16 output rows it writes, for
 *   every row of the sequences and each query head: o_part fp32 [T][n_q_heads][512], the output
 *   not yet divided by the softmax sum (16-byte aligned), and ml_part fp32 [T][n_q_heads][2], the
 *   running maximum of the scaled scores in log2 units (-inf for an empty partial) and the sum of
 *   2^(score - maximum) (8-byte aligned). The rows' keys in range must be in the cache (appended
 *   with g4attn_kv_append). Global layers only (G4_ERR_UNSUPPORTED otherwise: sliding layers split
 *   with a window halo); no image spans. Other arguments and errors as g4attn_prefill_attend.
 * g4attn_merge_partials: for every row of the sequences (q_start, q_len: int32 [B], device) and
 *   every head, merges the n_parts partials (1 <= n_parts <= 8; o_parts and ml_parts are HOST
 *   arrays of n_parts device pointers laid out as above) in the order given: M = max_r m_r, then
 *   O = sum_r o_r 2^(m_r - M) and L = sum_r l_r 2^(m_r - M) over r ascending, out = bf16(O / L)
 *   ([T][n_q_heads][512], 16-byte aligned). Rows of no sequence are not written. The order is
 *   fixed by the caller, not by timing, so the result does not depend on the batch around a row. */
g4_status g4attn_prefill_partial(const g4attn_layer* layer, const void* q, int32_t T, const int32_t* q_start,
                                 const int32_t* q_len, const int32_t* ctx_start, int32_t B,
                                 const int32_t* key_begin, const int32_t* key_end, const g4attn_cache* cache,
                                 const int32_t* page_table, int32_t max_pages, float* o_part, float* ml_part,
                                 void* stream);
g4_status g4attn_merge_partials(const g4attn_layer* layer, int32_t n_parts, const float* const* o_parts,
                                const float* const* ml_parts, int32_t T, const int32_t* q_start,
                                const int32_t* q_len, int32_t B, void* out, void* stream);

/* Bytes of device workspace g4attn_decode needs for B requests whose page table has
 * max_pages columns: the partial softmax states (m, l, O in fp32) of the fixed key chunks whose
 * split and ordered merge RFC section 4 rule 3 allows only when the merge tree is fixed by the
 * contract. The size is taken from the page-table width, the one context bound the host knows
 * without reading device memory (a context never exceeds 16 * max_pages keys, and never 262144);
 * it is 0 for an unsupported layer, B <= 0 or max_pages <= 0. */
size_t g4attn_decode_workspace_bytes(const g4attn_layer* layer, int32_t B, int32_t max_pages);

/* One decode step for B requests (RFC section 5, sliding_attention_core / global_attention_core
 * at one query row, and hybrid_kv_cache_contract: the decode side of the paged-cache handoff;
 * section 4 rules 2 and 3: a fixed chunk split with a fixed merge order, no split that depends on
 * the batch or the occupancy). Request b's new token sits at position seq_len[b]-1
 * (seq_len counts the new token); its key/value (k_new, v_new; v_new NULL on global layers)
 * are first written into the cache at that position, then out[b] = attention of q[b] over
 * positions 0 .. seq_len[b]-1 (the last `window` of them on sliding layers). Keys are split
 * into fixed chunks aligned to absolute position 0 (256 keys on sliding layers, 1024 on
 * global ones) and merged in ascending chunk order. seq_len: int32 [B], device, each in
 * [1, min(262144, 16*max_pages)]. workspace: device, >= g4attn_decode_workspace_bytes,
 * 16-byte aligned; its contents on entry do not matter. */
g4_status g4attn_decode(const g4attn_layer* layer, const void* q, const void* k_new,
                        const void* v_new, const int32_t* seq_len, int32_t B,
                        const g4attn_cache* cache, const int32_t* page_table, int32_t max_pages,
                        void* out, void* workspace, size_t workspace_bytes, void* stream);

/* g4attn_decode without a caller workspace. The RFC this library follows has no counterpart
 * of this call; it exists for callers that cannot allocate device memory when they decode:
 * a plain C host program with no device allocator of its own, or a serving process whose
 * device memory is reserved up front by its pooling allocator, where one more allocation
 * would fail or stall the step.
 *
 * The partial softmax states live in a static device buffer of the library,
 * G4ATTN_DECODE_STATIC_SCRATCH_BYTES (32 MiB) per device, and this call allocates nothing.
 * A step fits when g4attn_decode_workspace_bytes(layer, B, max_pages) is at most that size:
 * for example a sliding step (window 1024) of up to 203 requests, or a global step of up to
 * 15 requests with page tables of 2048 pages (32768 positions). A larger step returns
 * G4_ERR_SCRATCH and launches nothing; use g4attn_decode with a workspace for it.
 *
 * Arguments, layouts, arithmetic, results and other errors are those of g4attn_decode (the
 * same kernels run). Nothing in the scratch needs to start at zero: each call writes every
 * scratch entry it later reads.
 *
 * All calls on one device share the one buffer. Calls whose kernels may run at the same time
 * on the GPU (different streams with no ordering between them) race on it and give wrong
 * results; calls ordered on one stream do not. The first call on each device looks up the
 * buffer's address (and, like every first call, uploads the RoPE tables) with that device
 * current; make that first call before any stream capture. */
g4_status g4attn_decode_static(const g4attn_layer* layer, const void* q, const void* k_new,
                               const void* v_new, const int32_t* seq_len, int32_t B,
                               const g4attn_cache* cache, const int32_t* page_table,
                               int32_t max_pages, void* out, void* stream);

/* Runtime provenance (RFC section 4, rule 8): writes a NUL-terminated one-line record
 * (backend, kernel ids, schedule, split policy, accumulator, layer kind, device, dtype,
 * fallback state) into buf. Returns the record's length without the NUL, or -1 when the
 * layer is unsupported. Truncates to len-1 characters. */
int32_t g4attn_provenance(const g4attn_layer* layer, char* buf, size_t len);

/* The fail-closed report of RFC section 4 rule 7: problems only the device can see (a bad page,
 * position or image span, a bounded wait that ran out) are never absorbed by a silent fallback but
 * surface here. Synchronises `stream`, then reads and clears the device error word of the current
 * device: G4_OK, G4_ERR_TIMEOUT or G4_ERR_DEVICE (or G4_ERR_CUDA if a CUDA call failed). */
g4_status g4attn_status_sync(void* stream);

/* The bound of every wait in the kernels (RFC section 4 rule 7: a kernel that cannot make progress
 * fails closed instead of hanging). Each spin-wait of the kernels' barrier protocols gives up once
 * this many nanoseconds have passed since its first poll failed; the kernel then sets the timeout
 * bit of the device error word (G4_ERR_TIMEOUT from g4attn_status_sync), lets the copies and
 * tensor-core operations it already issued finish (those drains keep their own 2 s bound), frees
 * its tensor memory and returns; its output rows are then unspecified. Process-wide, read at each
 * launch; ns in [0, 2e9] (2e9, 2 s, is the default; 0 gives up at the first failed poll, which
 * exercises the fail-closed path of every kernel on purpose). Larger values: G4_ERR_INVALID.
 * g4attn_wait_limit_ns returns the current value. */
g4_status g4attn_set_wait_limit_ns(uint64_t ns);
uint64_t g4attn_wait_limit_ns(void);

/* A static, human-readable name for a status code (the failure half of the provenance that RFC
 * section 4 rules 7 and 8 ask for: what was refused, and why). Never NULL. */
const char* g4attn_status_string(g4_status s);

#ifdef __cplusplus
}
#endif

#endif /* G4ATTN_H */
