// Pieces shared by the prefill kernels (sliding and global): parameters, the work-unit
// enumeration, page lookups and the tensor map over the roped query rows.
#pragma once

#include "g4_internal.h"

namespace g4 {
namespace pf {

constexpr int kBM = 128;               // query rows per tile (aligned to absolute position)
constexpr int kBN = 64;                // keys per tile (aligned to absolute key 0)
constexpr float kLazyRescale = 8.0f;   // rescale O only when a row max grows by more than 2^8
constexpr int kSoftmaxThreads = 128;   // one thread per query row
constexpr int kQChunk = kBM * 128;     // roped Q: 128 rows x 64 dims per chunk, 128B swizzle

struct PrefillParams {
  SeqRows rows;
  int window;               // sliding W (0 on global layers)
  float scale_log2;
  const void* k_cache;      // sliding K' or global S
  const void* v_cache;      // sliding V (NULL on global layers)
  const void* krot_cache;   // global: roped rotated columns (NULL on sliding layers)
  int num_pages;
  const int32_t* page_table;
  int max_pages;
  __nv_bfloat16* out;
  RopeTables tb;
  uint32_t* err;
  int n_units;              // persistent sliding kernel: (query tile, KV head) units of the batch
};

// Finds this CTA's (sequence, query tile) among all sequences' tiles: slot s of sequence b
// is its tile (last - s), so every sequence is walked from its most expensive tile down.
// Warp-wide; returns b = -1 when the slot is past the last tile. The per-sequence arrays are
// read through the read-only path: a CTA reads them again for every unit it computes, and they
// then come from L1 instead of costing an L2 round trip each time.
// With `fields` set, the sequence's ctx_start, q_len and q_start come back in fields[0..2], read
// in the same round trip as the search. A sequence whose rows do not lie inside the T rows of q and
// out (q_start < 0 or q_start + q_len > T), or whose positions reach past the last usable one
// (ctx_start + q_len > 262144, tested without forming the sum, which could overflow), has no tiles:
// its rows are never read or written, and kErrPos is set.
inline __device__ void find_unit(const SeqRows& rows, int slot, int& out_b, int& out_t, uint32_t* err,
                                 int* fields = nullptr) {
  const int lane = threadIdx.x & 31;
  int base = 0;
  out_b = -1;
  out_t = 0;
  for (int b0 = 0; b0 < rows.B; b0 += 32) {
    const int b = b0 + lane;
    int cnt = 0, tl = 0, L = 0, cs = 0, qs = 0;
    if (b < rows.B) {
      L = __ldg(rows.q_len + b);
      cs = __ldg(rows.ctx_start + b);
      qs = __ldg(rows.q_start + b);
      if (L > 0 && cs >= 0 && qs >= 0 && L <= rows.T - qs && L <= kMaxPos && cs <= kMaxPos - L) {
        tl = (cs + L - 1) / kBM;
        cnt = tl - cs / kBM + 1;
      } else if (L > 0 && cs >= 0) {
        set_error(err, kErrPos);
      }
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    const int excl = incl - cnt;
    const bool mine = cnt > 0 && slot >= base + excl && slot < base + incl;
    const unsigned m = __ballot_sync(0xffffffffu, mine);
    if (m) {
      const int src = __ffs(m) - 1;
      const int e = __shfl_sync(0xffffffffu, excl, src);
      const int t_last = __shfl_sync(0xffffffffu, tl, src);
      out_b = b0 + src;
      out_t = t_last - (slot - base - e);
      if (fields) {
        fields[0] = __shfl_sync(0xffffffffu, cs, src);
        fields[1] = __shfl_sync(0xffffffffu, L, src);
        fields[2] = __shfl_sync(0xffffffffu, qs, src);
      }
      return;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
}

// Page-head block (physical page * hkv + g) holding keys key0 .. key0+15 of KV head g, or -1
// when the page lies outside [k_lo, k_hi]: such pages are never looked up nor copied.
inline __device__ int page_block(int key0, int k_lo, int k_hi, const int32_t* pt, int num_pages, int hkv,
                                          int g, uint32_t* err) {
  if (key0 + kPage - 1 < k_lo || key0 > k_hi) return -1;
  const int phys = pt[key0 >> 4];
  if (phys < 0 || phys >= num_pages) {
    set_error(err, kErrPage);
    return -1;
  }
  return phys * hkv + g;
}

// The same lookup in two steps, so that the page-table load can be issued a unit ahead of its
// use: page_raw returns the table entry of the page holding keys key0 .. key0+15 (kNoPage when
// the page lies outside [k_lo, k_hi]), page_check turns it into a page-head block index or -1
// (setting the error word for an entry outside the pool).
constexpr int kNoPage = -2147483647 - 1;
inline __device__ int page_raw(int key0, int k_lo, int k_hi, const int32_t* pt) {
  if (key0 + kPage - 1 < k_lo || key0 > k_hi) return kNoPage;
  const int v = __ldg(pt + (key0 >> 4));
  return v == kNoPage ? -1 : v;
}
inline __device__ int page_check(int raw, int num_pages, int hkv, int g, uint32_t* err) {
  if (raw == kNoPage) return -1;
  if (raw < 0 || raw >= num_pages) {
    set_error(err, kErrPage);
    return -1;
  }
  return raw * hkv + g;
}

// Keys [lo, hi] that the query at position pos (memory row `row`) sees, in a sequence whose keys
// end at ctx_end - 1: the layer's mask (causal; with a window W > 0 also pos - j <= W - 1),
// widened for an image token to every token of its image, in both directions (the model card's
// use_bidirectional_attention="vision"). As the layer mask already holds pos, the union is one run
// of keys. An image span must hold pos and end by ctx_end (its keys are in the cache); any other
// non-empty span sets kErrSpan and leaves the row to the layer mask.
inline __device__ void row_keys(const SeqRows& rows, int window, int row, int pos, int ctx_end, uint32_t* err,
                                int& lo, int& hi) {
  lo = window > 0 ? max(0, pos - window + 1) : 0;
  hi = pos;
  if (rows.span) {
    if ((unsigned)row >= (unsigned)rows.T) {   // a sequence laid out past the q rows
      set_error(err, kErrPos);
      return;
    }
    const int2 s = __ldg(reinterpret_cast<const int2*>(rows.span) + row);
    if (s.y > s.x) {
      if (s.x >= 0 && s.x <= pos && pos < s.y && s.y <= ctx_end) {
        lo = min(lo, s.x);
        hi = s.y - 1;
      } else {
        set_error(err, kErrSpan);
      }
    }
  }
}

inline __device__ uint32_t tmem_lane_base(int warp) { return (uint32_t)(32 * (warp & 3)) << 16; }

// Full cluster barrier (every thread of both CTAs); used once, after the mbarriers are set up.
inline __device__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 3-D map over q [T][Hq][D] (dims innermost first: D, Hq, T); box 64 dims x 1 head x 128 rows,
// 128-byte swizzle, zero fill outside.
inline bool q_map(CUtensorMap* m, const void* q, int T, int hq, int D) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)hq, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)hq * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kBM};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pf
}  // namespace g4
