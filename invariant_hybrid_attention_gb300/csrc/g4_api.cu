// The C ABI of g4attn: argument validation (fail closed), dispatch to the kernels of the one
// supported layer kind, runtime provenance and the device error word.
//
// Fail-closed rule and provenance follow section 4 ("Numerical contract", rules 7 and 8) of
// the RL-Kernel RFC "[RFC][Gemma-4-31B-it] WS1/WS2 kernel roadmap": a geometry outside the
// two supported layer kinds is refused before any launch, and there is no other code path to
// fall back to.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "g4_internal.h"
#include "g4attn.h"

using namespace g4;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Head counts of the full layer or of one tensor-parallel rank slice (RFC section 5, ws2_tp2 / ws2_tp4
// / ws2_tp8_kv_replication): tp in {1, 2, 4, 8} ranks each hold 32 / tp query heads and the KV
// heads they read, 16 / tp on sliding layers and 4 / tp on global ones, at least one: at tp = 8
// two ranks hold a copy of the same global KV head.
bool tp_heads(int n_q, int n_kv, bool global) {
  for (int tp = 1; tp <= 8; tp *= 2) {
    const int kv = global ? (kGlobalHkv / tp > 0 ? kGlobalHkv / tp : 1) : kSlidingHkv / tp;
    if (n_q == kSlidingHq / tp && n_kv == kv) return true;
  }
  return false;
}

g4_status check_layer(const g4attn_layer* L, bool* global) {
  if (!L) return G4_ERR_INVALID;
  if (L->kind == G4_SLIDING) {
    if (!tp_heads(L->n_q_heads, L->n_kv_heads, false) || L->head_dim != kSlidingD || L->kv_shared != 0 ||
        L->rope_theta != 1.0e4f || L->rope_partial != 1.0f)
      return G4_ERR_UNSUPPORTED;
    if (L->window < 1 || L->window > kMaxPos) return G4_ERR_UNSUPPORTED;
    *global = false;
  } else if (L->kind == G4_GLOBAL) {
    if (!tp_heads(L->n_q_heads, L->n_kv_heads, true) || L->head_dim != kGlobalD || L->kv_shared != 1 ||
        L->rope_theta != 1.0e6f || L->rope_partial != 0.25f || L->window != 0)
      return G4_ERR_UNSUPPORTED;
    *global = true;
  } else {
    return G4_ERR_UNSUPPORTED;
  }
  if (!(L->softmax_scale > 0.f) || !isfinite(L->softmax_scale)) return G4_ERR_INVALID;
  return G4_OK;
}

g4_status check_cache(const g4attn_cache* c, bool global, const int32_t* page_table, int32_t max_pages) {
  if (!c || !c->k || !aligned16(c->k)) return G4_ERR_INVALID;
  if (global) {
    if (c->v != nullptr || !c->k_rot || !aligned16(c->k_rot)) return G4_ERR_INVALID;
  } else if (!c->v || !aligned16(c->v) || c->k_rot != nullptr) {
    return G4_ERR_INVALID;
  }
  if (c->page_size != kPage) return G4_ERR_UNSUPPORTED;
  if (c->num_pages <= 0 || max_pages <= 0 || !page_table) return G4_ERR_INVALID;
  return G4_OK;
}

float scale_log2(const g4attn_layer* L) { return (float)((double)L->softmax_scale * 1.4426950408889634); }

g4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? G4_OK : G4_ERR_CUDA; }

PagedCache paged(const g4attn_layer* L, const g4attn_cache* c, const int32_t* page_table, int32_t max_pages) {
  PagedCache pc;
  pc.k = c->k;
  pc.v = c->v;
  pc.krot = c->k_rot;
  pc.num_pages = c->num_pages;
  pc.page_table = page_table;
  pc.max_pages = max_pages;
  pc.hq = L->n_q_heads;
  pc.hkv = L->n_kv_heads;
  return pc;
}

g4_status check_rows(const void* q_or_k, int32_t T, const int32_t* q_start, const int32_t* q_len,
                     const int32_t* ctx_start, int32_t B) {
  if (T < 0 || B <= 0 || !q_start || !q_len || !ctx_start) return G4_ERR_INVALID;
  if (T > 0 && (!q_or_k || !aligned16(q_or_k))) return G4_ERR_INVALID;
  return G4_OK;
}

// Norm arguments, checked on the host before any launch. On a K==V layer the stored S serves as V,
// and the key norm's weight reaches K only through the queries' un-rotated dims, so the key norm
// and the unit value norm come together there (or neither does).
g4_status check_norms(const g4attn_norms* n, bool global, NormArgs* out) {
  *out = NormArgs{};
  if (!n) return G4_OK;
  if (!(n->eps > 0.f) || !isfinite(n->eps)) return G4_ERR_INVALID;
  if (n->v_norm != 0 && n->v_norm != 1) return G4_ERR_INVALID;
  if ((n->q_weight && !aligned16(n->q_weight)) || (n->k_weight && !aligned16(n->k_weight))) return G4_ERR_INVALID;
  if (global && (n->v_norm != 0) != (n->k_weight != nullptr)) return G4_ERR_UNSUPPORTED;
  out->wq = (const __nv_bfloat16*)n->q_weight;
  out->wk = (const __nv_bfloat16*)n->k_weight;
  out->v_norm = n->v_norm;
  out->eps = n->eps;
  return G4_OK;
}

// Scratch of g4attn_decode_static: the partial softmax states of one decode step, in a
// file-scope device array so that the call needs no allocation. One copy per device; its
// address is looked up once per device and cached.
static __device__ __align__(256) uint8_t g_decode_scratch[G4ATTN_DECODE_STATIC_SCRATCH_BYTES];

constexpr int kScratchDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kScratchDevices];

cudaError_t decode_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kScratchDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_decode_scratch)) != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

const char* g4attn_status_string(g4_status s) {
  switch (s) {
    case G4_OK: return "ok";
    case G4_ERR_INVALID: return "invalid argument";
    case G4_ERR_UNSUPPORTED: return "unsupported geometry";
    case G4_ERR_CUDA: return "CUDA runtime error";
    case G4_ERR_SCRATCH: return "decode step larger than the static scratch buffer";
    case G4_ERR_TIMEOUT: return "bounded device wait timed out";
    case G4_ERR_DEVICE: return "device-detected bad page index, position or image span";
  }
  return "unknown status";
}

g4_status g4attn_rope_apply(const g4attn_layer* layer, const void* x, const int32_t* pos, int32_t T, int32_t H,
                            void* out, void* stream) {
  bool global = false;
  g4_status s = check_layer(layer, &global);
  if (s != G4_OK) return s;
  if (T < 0 || H < 1) return G4_ERR_INVALID;
  if (T == 0) return G4_OK;
  if (!x || !out || !pos || !aligned16(x) || !aligned16(out)) return G4_ERR_INVALID;
  DeviceState st;
  if (device_state(&st) != cudaSuccess) return G4_ERR_CUDA;
  return from_cuda(launch_rope_apply(global, x, pos, T, H, out, st, (cudaStream_t)stream));
}

g4_status g4attn_kv_append_normed(const g4attn_layer* layer, const g4attn_norms* norms, const void* k,
                                  const void* v, int32_t T, const int32_t* q_start, const int32_t* q_len,
                                  const int32_t* ctx_start, int32_t B, const g4attn_cache* cache,
                                  const int32_t* page_table, int32_t max_pages, void* stream) {
  bool global = false;
  g4_status s = check_layer(layer, &global);
  if (s != G4_OK) return s;
  NormArgs nm;
  if ((s = check_norms(norms, global, &nm)) != G4_OK) return s;
  if ((s = check_rows(k, T, q_start, q_len, ctx_start, B)) != G4_OK) return s;
  if ((s = check_cache(cache, global, page_table, max_pages)) != G4_OK) return s;
  if (global ? v != nullptr : (T > 0 && (!v || !aligned16(v)))) return G4_ERR_INVALID;
  if (T == 0) return G4_OK;
  DeviceState st;
  if (device_state(&st) != cudaSuccess) return G4_ERR_CUDA;
  SeqRows rows{q_start, q_len, ctx_start, B, T};
  return from_cuda(launch_append_prefill(global, k, v, rows, paged(layer, cache, page_table, max_pages), st,
                                         (cudaStream_t)stream, nullptr, nullptr, nm));
}

g4_status g4attn_kv_append(const g4attn_layer* layer, const void* k, const void* v, int32_t T,
                           const int32_t* q_start, const int32_t* q_len, const int32_t* ctx_start, int32_t B,
                           const g4attn_cache* cache, const int32_t* page_table, int32_t max_pages, void* stream) {
  return g4attn_kv_append_normed(layer, nullptr, k, v, T, q_start, q_len, ctx_start, B, cache, page_table, max_pages,
                                 stream);
}

// pt_row: optional page-table row of each sequence (the exact decode's chunks, listed from the
// longest context down).
static g4_status prefill_stage(const g4attn_layer* layer, const g4attn_norms* norms, const void* q, const void* k,
                               const void* v, int32_t T, const int32_t* q_start, const int32_t* q_len,
                               const int32_t* ctx_start, int32_t B, const g4attn_cache* cache,
                               const int32_t* page_table, int32_t max_pages, void* out, void* stream,
                               const int32_t* pt_row = nullptr) {
  bool global = false;
  g4_status s = check_layer(layer, &global);
  if (s != G4_OK) return s;
  NormArgs nm;
  if ((s = check_norms(norms, global, &nm)) != G4_OK) return s;
  if ((s = check_rows(q, T, q_start, q_len, ctx_start, B)) != G4_OK) return s;
  if ((s = check_cache(cache, global, page_table, max_pages)) != G4_OK) return s;
  if (T > 0 && (!k || !aligned16(k) || !out || !aligned16(out))) return G4_ERR_INVALID;
  if (global ? v != nullptr : (T > 0 && (!v || !aligned16(v)))) return G4_ERR_INVALID;
  if (T == 0) return G4_OK;
  DeviceState st;
  if (device_state(&st) != cudaSuccess) return G4_ERR_CUDA;
  // Cache append, and the roped queries staged in `out`: each sequence row of `out` holds its
  // roped query until g4attn_prefill_attend overwrites it with the attention output.
  const SeqRows rows{q_start, q_len, ctx_start, B, T, nullptr, pt_row, pt_row != nullptr};
  return from_cuda(launch_append_prefill(global, k, v, rows, paged(layer, cache, page_table, max_pages), st,
                                         (cudaStream_t)stream, q, out, nm));
}

g4_status g4attn_prefill_stage(const g4attn_layer* layer, const void* q, const void* k, const void* v, int32_t T,
                               const int32_t* q_start, const int32_t* q_len, const int32_t* ctx_start, int32_t B,
                               const g4attn_cache* cache, const int32_t* page_table, int32_t max_pages, void* out,
                               void* stream) {
  return prefill_stage(layer, nullptr, q, k, v, T, q_start, q_len, ctx_start, B, cache, page_table, max_pages, out,
                       stream);
}

// The attention step. q: the raw query rows, rotated inside the attention kernel; NULL: the roped
// queries staged in `out` by prefill_stage (image spans come only with staged queries).
static g4_status prefill_attend(const g4attn_layer* layer, const void* q, int32_t T, const int32_t* q_start,
                                const int32_t* q_len, const int32_t* ctx_start, int32_t B, const int32_t* span,
                                const g4attn_cache* cache, const int32_t* page_table, int32_t max_pages, void* out,
                                void* stream, const int32_t* pt_row = nullptr) {
  bool global = false;
  g4_status s = check_layer(layer, &global);
  if (s != G4_OK) return s;
  if ((s = check_rows(out, T, q_start, q_len, ctx_start, B)) != G4_OK) return s;
  if ((s = check_cache(cache, global, page_table, max_pages)) != G4_OK) return s;
  if (span && (reinterpret_cast<uintptr_t>(span) & 7u)) return G4_ERR_INVALID;
  if (q && (!aligned16(q) || span)) return G4_ERR_INVALID;
  if (T == 0) return G4_OK;
  DeviceState st;
  if (device_state(&st) != cudaSuccess) return G4_ERR_CUDA;
  const SeqRows rows{q_start, q_len, ctx_start, B, T, span, pt_row, pt_row != nullptr};
  return from_cuda(launch_prefill(global, rows, global ? 0 : layer->window, scale_log2(layer),
                                  paged(layer, cache, page_table, max_pages), out, st, (cudaStream_t)stream, q));
}

g4_status g4attn_prefill_attend(const g4attn_layer* layer, const void* q, int32_t T, const int32_t* q_start,
                                const int32_t* q_len, const int32_t* ctx_start, int32_t B, const g4attn_cache* cache,
                                const int32_t* page_table, int32_t max_pages, void* out, void* stream) {
  return prefill_attend(layer, q, T, q_start, q_len, ctx_start, B, nullptr, cache, page_table, max_pages, out,
                        stream);
}

g4_status g4attn_prefill_vision(const g4attn_layer* layer, const g4attn_norms* norms, const void* q, const void* k,
                                const void* v, int32_t T, const int32_t* q_start, const int32_t* q_len,
                                const int32_t* ctx_start, int32_t B, const int32_t* span,
                                const g4attn_cache* cache, const int32_t* page_table, int32_t max_pages, void* out,
                                void* stream) {
  // The span check comes first, so that a refused call launches nothing.
  if (span && (reinterpret_cast<uintptr_t>(span) & 7u)) return G4_ERR_INVALID;
  bool global = false;
  g4_status s = check_layer(layer, &global);
  if (s != G4_OK) return s;
  NormArgs nm;
  if ((s = check_norms(norms, global, &nm)) != G4_OK) return s;
  if (!nm.any() && !span) {
    // Plain queries: the cache append, then the attention kernel on the raw queries, which it
    // rotates itself (the same bits as the staged form below, one pass over q and out less).
    if (T > 0 && (!q || !aligned16(q) || !out || !aligned16(out))) return G4_ERR_INVALID;
    if ((s = check_rows(q, T, q_start, q_len, ctx_start, B)) != G4_OK) return s;
    if ((s = check_cache(cache, global, page_table, max_pages)) != G4_OK) return s;
    if ((s = g4attn_kv_append(layer, k, v, T, q_start, q_len, ctx_start, B, cache, page_table, max_pages, stream)) !=
        G4_OK)
      return s;
    return prefill_attend(layer, q, T, q_start, q_len, ctx_start, B, nullptr, cache, page_table, max_pages, out,
                          stream);
  }
  s = prefill_stage(layer, norms, q, k, v, T, q_start, q_len, ctx_start, B, cache, page_table, max_pages, out, stream);
  if (s != G4_OK) return s;
  return prefill_attend(layer, nullptr, T, q_start, q_len, ctx_start, B, span, cache, page_table, max_pages, out,
                        stream);
}

g4_status g4attn_prefill_normed(const g4attn_layer* layer, const g4attn_norms* norms, const void* q, const void* k,
                                const void* v, int32_t T, const int32_t* q_start, const int32_t* q_len,
                                const int32_t* ctx_start, int32_t B, const g4attn_cache* cache,
                                const int32_t* page_table, int32_t max_pages, void* out, void* stream) {
  return g4attn_prefill_vision(layer, norms, q, k, v, T, q_start, q_len, ctx_start, B, nullptr, cache, page_table,
                               max_pages, out, stream);
}

g4_status g4attn_prefill(const g4attn_layer* layer, const void* q, const void* k, const void* v, int32_t T,
                         const int32_t* q_start, const int32_t* q_len, const int32_t* ctx_start, int32_t B,
                         const g4attn_cache* cache, const int32_t* page_table, int32_t max_pages, void* out,
                         void* stream) {
  return g4attn_prefill_normed(layer, nullptr, q, k, v, T, q_start, q_len, ctx_start, B, cache, page_table, max_pages,
                               out, stream);
}

g4_status g4attn_prefill_partial(const g4attn_layer* layer, const void* q, int32_t T, const int32_t* q_start,
                                 const int32_t* q_len, const int32_t* ctx_start, int32_t B, const int32_t* key_begin,
                                 const int32_t* key_end, const g4attn_cache* cache, const int32_t* page_table,
                                 int32_t max_pages, float* o_part, float* ml_part, void* stream) {
  bool global = false;
  g4_status s = check_layer(layer, &global);
  if (s != G4_OK) return s;
  if (!global) return G4_ERR_UNSUPPORTED;   // sliding layers split a sequence with a window halo instead
  if ((s = check_rows(q, T, q_start, q_len, ctx_start, B)) != G4_OK) return s;
  if ((s = check_cache(cache, global, page_table, max_pages)) != G4_OK) return s;
  if (!key_begin || !key_end) return G4_ERR_INVALID;
  if (T > 0 && (!o_part || !ml_part || !aligned16(o_part) || (reinterpret_cast<uintptr_t>(ml_part) & 7u)))
    return G4_ERR_INVALID;
  if (T == 0) return G4_OK;
  DeviceState st;
  if (device_state(&st) != cudaSuccess) return G4_ERR_CUDA;
  const SeqRows rows{q_start, q_len, ctx_start, B, T};
  const PartialOut part{key_begin, key_end, o_part, ml_part};
  return from_cuda(launch_prefill_global(rows, scale_log2(layer), paged(layer, cache, page_table, max_pages), nullptr,
                                         st, (cudaStream_t)stream, q, &part));
}

g4_status g4attn_merge_partials(const g4attn_layer* layer, int32_t n_parts, const float* const* o_parts,
                                const float* const* ml_parts, int32_t T, const int32_t* q_start, const int32_t* q_len,
                                int32_t B, void* out, void* stream) {
  bool global = false;
  g4_status s = check_layer(layer, &global);
  if (s != G4_OK) return s;
  if (!global) return G4_ERR_UNSUPPORTED;
  if (n_parts < 1 || n_parts > kMaxParts || !o_parts || !ml_parts) return G4_ERR_INVALID;
  if (T < 0 || B <= 0 || !q_start || !q_len) return G4_ERR_INVALID;
  if (T == 0) return G4_OK;
  if (!out || !aligned16(out)) return G4_ERR_INVALID;
  PartialSet ps{};
  ps.n = n_parts;
  for (int i = 0; i < n_parts; ++i) {
    if (!o_parts[i] || !ml_parts[i] || !aligned16(o_parts[i]) || (reinterpret_cast<uintptr_t>(ml_parts[i]) & 7u))
      return G4_ERR_INVALID;
    ps.o[i] = o_parts[i];
    ps.ml[i] = ml_parts[i];
  }
  DeviceState st;
  if (device_state(&st) != cudaSuccess) return G4_ERR_CUDA;
  const SeqRows rows{q_start, q_len, nullptr, B, T};
  return from_cuda(launch_merge_partials(ps, rows, layer->n_q_heads, out, st, (cudaStream_t)stream));
}

size_t g4attn_decode_workspace_bytes(const g4attn_layer* layer, int32_t B, int32_t max_pages) {
  bool global = false;
  if (check_layer(layer, &global) != G4_OK || B <= 0 || max_pages <= 0) return 0;
  return decode_workspace_bytes(global, B, max_pages, global ? 0 : layer->window, layer->n_q_heads);
}

g4_status g4attn_decode_normed(const g4attn_layer* layer, const g4attn_norms* norms, const void* q,
                               const void* k_new, const void* v_new, const int32_t* seq_len, int32_t B,
                               const g4attn_cache* cache, const int32_t* page_table, int32_t max_pages, void* out,
                               void* workspace, size_t workspace_bytes, void* stream) {
  bool global = false;
  g4_status s = check_layer(layer, &global);
  if (s != G4_OK) return s;
  NormArgs nm;
  if ((s = check_norms(norms, global, &nm)) != G4_OK) return s;
  if (B <= 0 || !q || !k_new || !seq_len || !out || !workspace) return G4_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(out) || !aligned16(workspace)) return G4_ERR_INVALID;
  if (global ? v_new != nullptr : (!v_new || !aligned16(v_new))) return G4_ERR_INVALID;
  if ((s = check_cache(cache, global, page_table, max_pages)) != G4_OK) return s;
  if (workspace_bytes < decode_workspace_bytes(global, B, max_pages, global ? 0 : layer->window, layer->n_q_heads))
    return G4_ERR_INVALID;
  DeviceState st;
  if (device_state(&st) != cudaSuccess) return G4_ERR_CUDA;
  const cudaStream_t cs = (cudaStream_t)stream;
  const PagedCache pc = paged(layer, cache, page_table, max_pages);
  // Normed queries go through `out`: the decode kernel reads them there before the merge writes
  // the output rows.
  const void* q_eff = q;
  if (nm.wq != nullptr || (global && nm.wk != nullptr)) {
    if (launch_norm_queries(global, q, out, B, layer->n_q_heads, nm, cs) != cudaSuccess) return G4_ERR_CUDA;
    q_eff = out;
  }
  cudaError_t e = launch_append_decode(global, k_new, v_new, seq_len, B, pc, st, cs, nm);
  if (e != cudaSuccess) return G4_ERR_CUDA;
  return from_cuda(launch_decode(global, q_eff, seq_len, B, global ? 0 : layer->window, scale_log2(layer), pc, out,
                                 workspace, st, cs));
}

g4_status g4attn_decode(const g4attn_layer* layer, const void* q, const void* k_new, const void* v_new,
                        const int32_t* seq_len, int32_t B, const g4attn_cache* cache, const int32_t* page_table,
                        int32_t max_pages, void* out, void* workspace, size_t workspace_bytes, void* stream) {
  return g4attn_decode_normed(layer, nullptr, q, k_new, v_new, seq_len, B, cache, page_table, max_pages, out,
                              workspace, workspace_bytes, stream);
}

size_t g4attn_decode_exact_workspace_bytes(int32_t B) {
  return B <= 0 ? 0 : ((size_t)B * 4 * sizeof(int32_t) + 15) / 16 * 16;
}

g4_status g4attn_decode_exact(const g4attn_layer* layer, const g4attn_norms* norms, const void* q, const void* k_new,
                              const void* v_new, const int32_t* seq_len, int32_t B, const g4attn_cache* cache,
                              const int32_t* page_table, int32_t max_pages, void* out, void* workspace,
                              size_t workspace_bytes, void* stream) {
  bool global = false;
  g4_status s = check_layer(layer, &global);
  if (s != G4_OK) return s;
  NormArgs nm;
  if ((s = check_norms(norms, global, &nm)) != G4_OK) return s;
  // Every check of the two prefill steps runs here, before the first launch.
  if (B <= 0 || !q || !k_new || !seq_len || !out || !workspace) return G4_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(out) || !aligned16(workspace)) return G4_ERR_INVALID;
  if (global ? v_new != nullptr : (!v_new || !aligned16(v_new))) return G4_ERR_INVALID;
  if ((s = check_cache(cache, global, page_table, max_pages)) != G4_OK) return s;
  if (workspace_bytes < g4attn_decode_exact_workspace_bytes(B)) return G4_ERR_INVALID;
  DeviceState st;
  if (device_state(&st) != cudaSuccess) return G4_ERR_CUDA;
  int32_t* rows = static_cast<int32_t*>(workspace);
  if (launch_decode_rows(seq_len, B, rows, st, (cudaStream_t)stream) != cudaSuccess) return G4_ERR_CUDA;
  if ((s = prefill_stage(layer, norms, q, k_new, v_new, B, rows, rows + B, rows + 2 * B, B, cache, page_table,
                         max_pages, out, stream, rows + 3 * B)) != G4_OK)
    return s;
  return prefill_attend(layer, nullptr, B, rows, rows + B, rows + 2 * B, B, nullptr, cache, page_table, max_pages, out,
                        stream, rows + 3 * B);
}

g4_status g4attn_decode_static(const g4attn_layer* layer, const void* q, const void* k_new, const void* v_new,
                               const int32_t* seq_len, int32_t B, const g4attn_cache* cache,
                               const int32_t* page_table, int32_t max_pages, void* out, void* stream) {
  bool global = false;
  g4_status s = check_layer(layer, &global);
  if (s != G4_OK) return s;
  if (B <= 0 || max_pages <= 0) return G4_ERR_INVALID;
  const size_t need = decode_workspace_bytes(global, B, max_pages, global ? 0 : layer->window, layer->n_q_heads);
  if (need > G4ATTN_DECODE_STATIC_SCRATCH_BYTES) return G4_ERR_SCRATCH;
  void* ws = nullptr;
  if (decode_scratch(&ws) != cudaSuccess) return G4_ERR_CUDA;
  return g4attn_decode(layer, q, k_new, v_new, seq_len, B, cache, page_table, max_pages, out, ws,
                       G4ATTN_DECODE_STATIC_SCRATCH_BYTES, stream);
}

int32_t g4attn_provenance(const g4attn_layer* layer, char* buf, size_t len) {
  bool global = false;
  if (check_layer(layer, &global) != G4_OK) return -1;
  char dev[320] = "unknown";
  int d = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&d) == cudaSuccess && cudaGetDeviceProperties(&prop, d) == cudaSuccess)
    snprintf(dev, sizeof(dev), "%s(sm_%d%d,%dSM)", prop.name, prop.major, prop.minor, prop.multiProcessorCount);
  char rec[1536];
  int n;
  if (global)
    n = snprintf(rec, sizeof(rec),
                 "requested=g4attn;actual=g4attn-cuda-sm_103a;layer=global;kernels=append_shared_s,"
                 "prefill_global_tcgen05_2sm_x2_rope_q,decode_global_mma_bf16,merge_ordered;schedule=qtile128@abs-pos,"
                 "ktile128@abs-pos,ascending;split=decode-fixed-chunk-1024@abs-key0,4-warp-round-robin,ordered-merge;"
                 "qrope=attention-kernel(plain),append-pass(normed,vision,exact-decode);"
                 "exact-decode=prefill-kernels-one-row-chunks;vision=image-span-per-row;"
                 "accumulator=fp32;casts=roped-q,roped-k,p,out:bf16-rne;exp=ex2.approx.ftz.f32;device=%s;dtype=bf16;"
                 "shape=Hq%d,Hkv%d,D512,k_eq_v,prope0.25,theta1e6,scale%.9g;fallback=none",
                 dev, layer->n_q_heads, layer->n_kv_heads, (double)layer->softmax_scale);
  else
    n = snprintf(rec, sizeof(rec),
                 "requested=g4attn;actual=g4attn-cuda-sm_103a;layer=sliding;kernels=append_kv_keygroups,"
                 "prefill_sliding_tcgen05_2sm_rope_q,decode_sliding_mma_bf16,merge_ordered;"
                 "schedule=qtile128@abs-pos,ktile128@abs-pos,ascending,window-skip;"
                 "split=decode-fixed-chunk-256@abs-key0,4-warp-round-robin,ordered-merge;"
                 "qrope=attention-kernel(plain),append-pass(normed,vision,exact-decode);"
                 "exact-decode=prefill-kernels-one-row-chunks;vision=image-span-per-row;"
                 "accumulator=fp32;casts=roped-q,roped-k,p,out:bf16-rne;exp=ex2.approx.ftz.f32;device=%s;dtype=bf16;"
                 "shape=Hq%d,Hkv%d,D256,W%d,theta1e4,scale%.9g;fallback=none",
                 dev, layer->n_q_heads, layer->n_kv_heads, layer->window, (double)layer->softmax_scale);
  if (n < 0) return -1;
  if (buf && len > 0) {
    const size_t c = (size_t)n < len - 1 ? (size_t)n : len - 1;
    memcpy(buf, rec, c);
    buf[c] = '\0';
  }
  return n;
}

g4_status g4attn_set_wait_limit_ns(uint64_t ns) {
  if (ns > kWaitLimitNs) return G4_ERR_INVALID;
  set_wait_limit_ns(ns);
  return G4_OK;
}

uint64_t g4attn_wait_limit_ns(void) { return wait_limit_ns(); }

g4_status g4attn_status_sync(void* stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return G4_ERR_CUDA;
  DeviceState st;
  if (device_state(&st) != cudaSuccess) return G4_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, st.err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return G4_ERR_CUDA;
  if (word != 0 && cudaMemset(st.err, 0, sizeof(word)) != cudaSuccess) return G4_ERR_CUDA;
  if (word & kErrTimeout) return G4_ERR_TIMEOUT;
  if (word & (kErrPage | kErrPos | kErrSpan)) return G4_ERR_DEVICE;
  return G4_OK;
}

}  // extern "C"
