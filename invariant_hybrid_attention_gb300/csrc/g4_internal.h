// Host-side interface between the g4attn translation units (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "g4_common.cuh"

namespace g4 {

// Static device state of the current device: the RoPE tables of both layer kinds and the
// error word. Filled on the first call per device (a synchronous upload; make that first
// call outside any stream capture).
struct DeviceState {
  RopeTables sliding;
  RopeTables global;
  uint32_t* err;
};
cudaError_t device_state(DeviceState* st);

// The limit of every protocol wait in the kernels launched from now on (process-wide; kWaitLimitNs
// unless g4attn_set_wait_limit_ns changed it).
unsigned long long wait_limit_ns();
void set_wait_limit_ns(unsigned long long ns);

// Row-to-sequence description of a prefill batch (all device pointers, int32 [B]).
struct SeqRows {
  const int32_t* q_start;
  const int32_t* q_len;
  const int32_t* ctx_start;
  int32_t B;
  int32_t T;
  // Optional int32 [T][2]: the image span [s0, s1) of absolute positions of each query row
  // (memory row index, like q); s1 <= s0 marks a text row. NULL: every row is text.
  const int32_t* span = nullptr;
  // Optional int32 [B]: the page-table row of each sequence (NULL: sequence b reads row b). The
  // exact decode lists its one-row chunks from the longest context down, for the schedule, and
  // keeps each request's own page-table row.
  const int32_t* pt_row = nullptr;
  // The sequences are listed from the most expensive down: a persistent schedule then walks its
  // rounds of units in a snake, which evens the clusters' shares.
  bool by_cost = false;
};

// A layer's paged cache and the head counts of the call: hkv KV heads in the cache (its page-head
// blocks), hq query heads in the q and out rows. The full geometry has 32 / 16 (sliding) or 32 / 4
// (global); a tensor-parallel rank slice has 32 / tp query heads and 16 / tp or max(1, 4 / tp) KV
// heads.
struct PagedCache {
  void* k;
  void* v;
  void* krot;   // global layers: p-RoPE(S) on the rotated columns (rot_offset layout)
  int32_t num_pages;
  const int32_t* page_table;
  int32_t max_pages;
  int32_t hq = 32;
  int32_t hkv = 16;
};

// Optional per-head RMS norms of a prefill or decode (device pointers to bf16 [D] weights; a null
// weight leaves that tensor un-normed). See the norm notes in g4_rope.cu.
struct NormArgs {
  const __nv_bfloat16* wq = nullptr;   // query weight
  const __nv_bfloat16* wk = nullptr;   // key weight
  int v_norm = 0;                      // unit RMS norm of the values (the stored S on K==V layers)
  float eps = 1e-6f;
  __host__ __device__ bool any() const { return wq != nullptr || wk != nullptr || v_norm != 0; }
};

cudaError_t launch_rope_apply(bool global, const void* x, const int32_t* pos, int T, int H, void* out,
                              const DeviceState& st, cudaStream_t s);

// Writes the rows' K'/V (or S) into the cache; with q_out set, also the rows' roped queries
// (bf16) into q_out, the staging the prefill attention kernel reads its queries from.
cudaError_t launch_append_prefill(bool global, const void* k, const void* v, const SeqRows& rows,
                                  const PagedCache& cache, const DeviceState& st, cudaStream_t s,
                                  const void* q = nullptr, void* q_out = nullptr, const NormArgs& nm = NormArgs{});

cudaError_t launch_append_decode(bool global, const void* k_new, const void* v_new, const int32_t* seq_len,
                                 int B, const PagedCache& cache, const DeviceState& st, cudaStream_t s,
                                 const NormArgs& nm = NormArgs{});

// The decode queries' norms, written to out (bf16), for the decode kernel to read as its q.
cudaError_t launch_norm_queries(bool global, const void* q, void* out, int B, int hq, const NormArgs& nm,
                                cudaStream_t s);

// Decode partials + ordered merge. ws must hold decode_workspace_bytes(global, B, max_pages, window, hq).
size_t decode_workspace_bytes(bool global, int B, int max_pages, int window, int hq);
cudaError_t launch_decode(bool global, const void* q, const int32_t* seq_len, int B, int window,
                          float scale_log2, const PagedCache& cache, void* out, void* ws,
                          const DeviceState& st, cudaStream_t s);

// Writes rows [3][B] (q_start, q_len, ctx_start) of a decode step taken as B one-row prefill chunks.
cudaError_t launch_decode_rows(const int32_t* seq_len, int B, int32_t* rows, const DeviceState& st, cudaStream_t s);

// Attention of the rows of a prefill batch, written into `out`. With q_raw set the kernel reads the raw
// query rows there and rotates them itself; otherwise it reads the roped queries that
// launch_append_prefill staged in `out` and writes the output rows over them.
cudaError_t launch_prefill(bool global, const SeqRows& rows, int window, float scale_log2, const PagedCache& cache,
                           void* out, const DeviceState& st, cudaStream_t s, const void* q_raw = nullptr);
// A partial global prefill (context parallelism over keys): sequence b attends only to its keys
// key_begin[b] .. key_end[b]-1 (device int32 [B]); the rows' un-normalised output o (fp32
// [T][hq][512]) and softmax state ml (fp32 [T][hq][2]) are written instead of bf16 output rows.
struct PartialOut {
  const int32_t* key_begin;
  const int32_t* key_end;
  float* o;
  float* ml;
};
cudaError_t launch_prefill_global(const SeqRows& rows, float scale_log2, const PagedCache& cache, void* out,
                                  const DeviceState& st, cudaStream_t s, const void* q_raw = nullptr,
                                  const PartialOut* part = nullptr);

// Merges n partials of a global prefill, in the order given, into bf16 output rows (the rows of
// the sequences only): M = max m_r, then O = sum_r o_r 2^(m_r - M) and L = sum_r l_r 2^(m_r - M),
// out = O / L.
constexpr int kMaxParts = 8;
struct PartialSet {
  const float* o[kMaxParts];
  const float* ml[kMaxParts];
  int n;
};
cudaError_t launch_merge_partials(const PartialSet& parts, const SeqRows& rows, int hq, void* out, const DeviceState& st,
                                  cudaStream_t s);

}  // namespace g4
