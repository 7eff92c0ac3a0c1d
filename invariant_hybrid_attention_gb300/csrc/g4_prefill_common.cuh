// Pieces shared by the prefill kernels (sliding and global): parameters, the work-unit
// enumeration, page lookups, the query rotation and the tensor map over the query rows.
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
  int hq, hkv;              // query heads of the q and out rows; KV heads of the cache
  // Partial calls (global layers, context parallelism over keys): sequence b attends only to keys
  // key_begin[b] .. key_end[b]-1, and the rows' un-normalised output o_part (fp32 [T][hq][D]) and
  // softmax state ml_part (fp32 [T][hq][2]: running max in log2 units, sum) are written instead of
  // out. NULL otherwise.
  const int32_t* key_begin;
  const int32_t* key_end;
  float* o_part;
  float* ml_part;
  int n_units;              // persistent sliding kernel: (query tile, KV head) units of the batch
  unsigned long long wait_ns;   // limit of every protocol wait (g4attn_set_wait_limit_ns)
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

// The in-kernel query rotation. A 128-row query tile sits in shared memory as 128B-swizzled boxes
// of 64 dims x 128 rows (row r of a box at r * 128, its 16-byte piece j at piece j ^ (r % 8)). One
// thread rotates one pair t of rows r_begin .. r_begin + 16 NK - 1 (r_begin a multiple of 16). Row
// r sits at position p0 + r, with p0 a multiple of 128 (and p0 + 127 < 262144), so every row of the
// tile shares the coarse table entry, a 16-row group the mid entry and rows with one r % 16 the
// fine entry: the thread loads 1 + NK + 16 table entries (from the entry-major copies of the
// tables, R pairs per entry), all at once, instead of 3 per row, and keeps them in registers. The angle of row r is cmul(cmul(coarse, mid), fine), exactly as rope_cs
// forms it, and the rotation and the bf16 cast (round to nearest even) are those of the
// cache-append pass, so a query rotated here has the bits a staged one has. A 16-row group goes in
// three phases (all its loads, then the arithmetic, then all its stores): rotated in place, a row's
// stores could otherwise alias the next row's loads as far as the compiler can tell, and every row
// would pay a whole load-rotate-store latency. Every row turns, those outside the sequence too
// (their outputs are never written), so that no branch splits a group. lo_box is the box holding
// dim t, hi_box the one holding its partner t + D/2.
template <int NK, int R>
inline __device__ void rotate_q_pair(uint8_t* lo_box, uint8_t* hi_box, const RopeTables& tb, int t, int p0,
                                     int r_begin) {
  const int e = t & 63;
  const int k0 = r_begin >> 4;
  // the entry-major copies: lanes hold consecutive t, so each load is two whole lines
  const float2 c = __ldg(tb.coarse_t + (size_t)(p0 >> 8) * R + t);
  const int a0 = (p0 >> 4) & 15;
  float2 m[NK], f[16];
#pragma unroll
  for (int k = 0; k < NK; ++k) m[k] = __ldg(tb.mid_t + (a0 + k0 + k) * R + t);
#pragma unroll
  for (int b = 0; b < 16; ++b) f[b] = __ldg(tb.fine_t + b * R + t);
  uint8_t* lo = lo_box + ((e & 7) << 1);
  uint8_t* hi = hi_box + ((e & 7) << 1);
  const int piece = e >> 3;
  int sw[8];   // the swizzled piece offset of rows with r % 8 = j
#pragma unroll
  for (int j = 0; j < 8; ++j) sw[j] = (piece ^ j) << 4;
#pragma unroll 1
  for (int k = 0; k < NK; ++k) {
    float2 mk = m[0];   // m[k] by selects: a dynamic index would put m in local memory
#pragma unroll
    for (int j = 1; j < NK; ++j)
      if (k == j) mk = m[j];
    const float2 cm = cmul(c, mk);
    uint8_t* lo_k = lo + 16 * (k0 + k) * 128;
    uint8_t* hi_k = hi + 16 * (k0 + k) * 128;
    float x[16], y[16];
#pragma unroll
    for (int b = 0; b < 16; ++b) {
      x[b] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(lo_k + b * 128 + sw[b & 7]));
      y[b] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(hi_k + b * 128 + sw[b & 7]));
    }
#pragma unroll
    for (int b = 0; b < 16; ++b) rope_pair(x[b], y[b], cmul(cm, f[b]));
#pragma unroll
    for (int b = 0; b < 16; ++b) {
      *reinterpret_cast<__nv_bfloat16*>(lo_k + b * 128 + sw[b & 7]) = __float2bfloat16_rn(x[b]);
      *reinterpret_cast<__nv_bfloat16*>(hi_k + b * 128 + sw[b & 7]) = __float2bfloat16_rn(y[b]);
    }
  }
}

// Epilogue stores. Lane L of an epilogue warp holds row L's 16 packed words (32 dims) of an output
// chunk, and rows lie hq * D * 2 bytes apart, so a store per lane would touch 32 rows (32 cache
// lines) for 16 bytes each. Two xor-shuffle stages transpose the 16-byte pieces inside each group
// of four lanes (each stage swaps one bit of the lane index with the same bit of the piece index),
// after which lane 4a + i holds piece i of rows 4a .. 4a+3: each store then writes 64 contiguous
// bytes of eight rows.
template <int M>
inline __device__ void xpose_pieces(uint32_t (&w)[16], int lane) {
  const bool hi = (lane & M) != 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (j & M) continue;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t send = hi ? w[4 * j + k] : w[4 * (j | M) + k];
      const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, M);
      if (hi)
        w[4 * j + k] = recv;
      else
        w[4 * (j | M) + k] = recv;
    }
  }
}
// Stores dims col0 .. col0+31 of head h of the warp's 32 rows of out [rows][hq][D]; row0 is the
// warp's first row (may be out of range: only rows set in `valid` are written).
template <int D>
inline __device__ void store_rows32(uint32_t (&w)[16], __nv_bfloat16* out, long long row0, int hq, int h, int col0,
                                    unsigned valid, int lane) {
  xpose_pieces<1>(w, lane);
  xpose_pieces<2>(w, lane);
  const int a = lane >> 2, i = lane & 3;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int row = 4 * a + t;
    if ((valid >> row) & 1u) {
      __nv_bfloat16* dst = out + ((row0 + row) * hq + h) * D + col0 + 8 * i;
      *reinterpret_cast<uint4*>(dst) = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
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
