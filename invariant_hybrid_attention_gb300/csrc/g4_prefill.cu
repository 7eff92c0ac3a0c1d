// Sliding-layer prefill on the 5th-generation tensor cores (tcgen05, accumulators in tensor
// memory): a persistent kernel of 2-SM MMA units, one unit per pair of query heads.
//
// Sliding layer (RL-Kernel RFC "[RFC][Gemma-4-31B-it] WS1/WS2 kernel roadmap", section 5,
// sliding_attention_core: causal local attention, window 1024, 32 Q / 16 KV heads, D 256).
// Work unit: (sequence, query tile of 128 positions aligned to absolute position, KV head g),
// computed by a cluster of two CTAs; CTA rank r owns query head 2g + r, i.e. the two query
// heads that share K and V. Key tiles of 128 keys are aligned to absolute key 0 and visited in
// ascending order, so the arithmetic a row gets depends only on its own position, its
// sequence's keys and the window: not on the batch, the row's place in it, padding, packing, the
// launch grid or which cluster runs the unit. A key tile that holds no visible key for a row
// adds exact zeros to it (RFC section 4 rules 2, 3 and 6).
//
// Every tcgen05 MMA is one 2-SM operation (M = 256: the two heads' 128 rows each) issued by
// the even CTA. A (queries, P) and D (S, O) are split by rows, so each CTA keeps its own head's
// rows in its own tensor memory; B (K, V) is split by columns, so each CTA stages only half of
// every key tile: keys 64r .. 64r+63 of K (all dims) and dims 128r .. 128r+127 of V (all 128
// keys), 64 KB per tile instead of 128 KB. QK^T runs at N = 128 keys, P.V at N = 256 dims.
//
// The grid holds as many clusters as can be resident at once; cluster c computes units
// c, c + C, c + 2C, ... (a fixed assignment: no work queue, no atomics). The K and V rings and
// every barrier run on counters that continue across units, so the next unit's keys stream in
// while the current one finishes; its Q tile is copied into buffers of its own while the
// current unit runs, so that the softmax warps can turn it as soon as they are done with the
// current unit.
// Per CTA:
//   warp 0     this CTA's K half of each key tile (four 8 KB page-head blocks) into a 2-stage
//              ring (three stages measured the same), and each unit's Q tile: dims 0-127 into a
//              staging buffer, dims 128-255 into one of two buffers by unit parity, the next
//              unit's after this unit's second key tile, once this unit's Q has moved on;
//   warp 6     this CTA's V half of each key tile (eight 4 KB copies: sliding V pages store each
//              128-dim half of a page-head block contiguously) into a 2-stage ring;
//   warp 1     even CTA: issues S = Q K^T for the pair. Odd CTA: tells the even CTA when each
//              of its K ring slots has landed;
//   warp 7     zeroes value rows of this CTA's V half that hold no key of the sequence; then
//              the even CTA's issues O += P V for the pair, the odd CTA's tells the even CTA
//              that its V half is ready;
//   warps 2-5, 8-11  two threads per query row of this CTA's head, one per half of the
//              columns (warps w and w + 6 share the rows of quarter w % 4, the tensor-memory
//              lanes they may access): Q dims 0-127 into tensor memory, mask, online softmax
//              (lazy rescale, threshold 2^8; the halves agree on each tile's row max through a
//              barrier of their quarter), P (bf16), the O correction when needed, and the
//              epilogue O / l -> bf16 (the halves' sums added in a fixed order).
// Queries (kRope): the Q tile is copied from the raw query rows and rotated in place in shared
// memory before it moves: all 128 pairs (t, t + 128) turn, t in Q dims 0-127 (the staging buffer,
// bound for tensor memory) and t + 128 in the shared-memory half. Softmax thread i rotates pair
// i % 128 of rows 64 (i / 128) .. +63 (rotate_q_pair), the eight softmax warps meet on an
// mbarrier, and each thread then moves its half of its row. The angles, the rotation and the bf16 cast are those of the append
// pass, so the roped queries, and with them every output bit, are those a staged call gives. Otherwise (the staged form: normed queries,
// image spans, the exact decode) the append pass before this kernel wrote bf16(RoPE(q)) into the
// sequence rows of `out`, which the Q copies read; the epilogue later overwrites exactly those
// rows (each row belongs to one unit).
// Tensor memory (512 columns, allocated jointly by the pair): O [0,256), Q dims 0-127 [256,320)
// as bf16 pairs, P [320,384) as bf16 key pairs, S [384,512). With one S buffer, QK^T of tile
// j+1 is issued as soon as both CTAs' softmax threads have read S_j into registers, so it runs
// while they exponentiate; P has its own buffer, so it never waits for S to be consumed.
// An mbarrier parity wait cannot tell phases two apart, so every role that waits on a ring
// barrier waits on each of its phases in order, including phases it has no use for.
#include <math.h>

#include "g4_prefill_common.cuh"

namespace g4 {

namespace {

using namespace pf;

constexpr int kSD = kSlidingD;                    // 256
constexpr int kSN = 128;                          // keys per tile
constexpr int kNK = 2, kNV = 2;                   // K and V ring stages
constexpr int kPageBytes = kPage * kSD * 2;       // one tiled page-head block: 8 KB
constexpr int kKeyGroupBytes = 8 * kSD * 2;       // K: 8 keys x 256 dims, 4 KB
constexpr int kVGroupBytes = 8 * (kSD / 2) * 2;   // V half: 8 keys x 128 dims, 2 KB
constexpr int kVHalfPageBytes = 2 * kVGroupBytes; // V half of one page-head block: 4 KB
constexpr int kKStage = (kSN / 2 / kPage) * kPageBytes;   // 4 pages: 32 KB
constexpr int kVStage = (kSN / 8) * kVGroupBytes;         // 16 key groups: 32 KB
constexpr int kSmxWarps = 8;                      // softmax warps: two per row quarter, one per half of the columns
constexpr int kThreads = 128 + 32 * kSmxWarps;    // warps 0, 1, 6, 7 have roles; 2-5 and 8-11 run the softmax
constexpr uint32_t kTmO = 0, kTmQ = 256, kTmP = 320, kTmS = 384;
constexpr uint32_t kIdescQK = idesc_bf16(2 * kBM, kSN, false, false);   // M 256 over the pair, N 128 keys
constexpr uint32_t kIdescPV = idesc_bf16(2 * kBM, kSD, false, true);    // M 256, N 256 dims
constexpr uint16_t kBoth = 0x3;
constexpr uint32_t kPairWarps = 2 * kSmxWarps;   // softmax warps of both CTAs

struct alignas(1024) SlidingSmem {
  uint8_t qlo[2 * kQChunk];         // a unit's Q dims 0-127 (128B swizzle) until they move into tensor memory
  uint8_t qhi[2][2 * kQChunk];      // unit u's Q dims 128-255 in qhi[u & 1]: the shared-memory A operand
  uint8_t k[kNK][kKStage];          // K halves [8 key groups][32 dim groups][8][8]
  uint8_t v[kNV][kVStage];          // V halves [16 key groups][16 dim groups][8][8]
  uint64_t k_full[kNK], k_empty[kNK], k_peer[kNK];
  uint64_t v_full[kNV], v_empty[kNV], v_ready[kNV];
  uint64_t s_full, s_free, p_full, pv_done;
  uint64_t q_full, q_pair, q_free, o_free, q_read, q_rot, teardown;
  uint64_t xchg[4];                 // the two softmax warps of row quarter i have posted their halves
  float xv[2][2][kBM];              // [exchange parity][column half][row]: a half's row max, then its sum
  uint32_t tmem_base;
  int abort_flag;
};
constexpr size_t kSlidingSmemBytes = sizeof(SlidingSmem);   // the base must be 1024-aligned (checked)
static_assert(kSlidingSmemBytes <= 232448, "sliding prefill exceeds the 227 KB shared-memory limit");

// One unit as one CTA of its pair sees it.
struct Unit {
  int g, h, t, p_lo, p_hi, ctx_end, k_lo, k_hi, kt0, n_tiles, q_row0;
  const int32_t* pt;
};

// Warp-wide. False when unit u holds no rows (its slot is past the last query tile) or its
// positions are out of range (then the error word is set); every role skips such units alike.
// Not inlined: six roles call it, once per unit. kSpan: the batch may hold image rows.
template <bool kSpan>
__device__ __noinline__ bool sliding_unit(const PrefillParams& p, int u, uint32_t rank, Unit& o) {
  o.g = u % p.hkv;
  o.h = 2 * o.g + (int)rank;
  int b, t, f[3];
  find_unit(p.rows, u / p.hkv, b, t, p.err, f);
  if (b < 0) return false;
  const int cs = f[0], L = f[1], qs = f[2];
  o.t = t;
  o.p_lo = max(kBM * t, cs);
  o.p_hi = min(kBM * t + kBM - 1, cs + L - 1);
  o.ctx_end = cs + L;
  if (o.p_hi >= kMaxPos || (o.p_hi >> 4) >= p.max_pages) {
    if ((threadIdx.x & 31) == 0) set_error(p.err, kErrPos);
    return false;
  }
  const int W = p.window;
  o.q_row0 = qs + (kBM * t - cs);   // memory row of tile row 0 (may be negative)
  if constexpr (kSpan) {
    // The rows' key runs start no earlier than the first row's and end no later than the last
    // row's: the layer mask moves with the position, and an image holding a row inside the tile
    // and reaching past an end row holds that end row too.
    int lo_l, hi_f;
    row_keys(p.rows, W, o.q_row0 + (o.p_lo - kBM * t), o.p_lo, o.ctx_end, p.err, o.k_lo, hi_f);
    row_keys(p.rows, W, o.q_row0 + (o.p_hi - kBM * t), o.p_hi, o.ctx_end, p.err, lo_l, o.k_hi);
    if ((o.k_hi >> 4) >= p.max_pages) {   // an image past the page table (the rows' own pages fit)
      if ((threadIdx.x & 31) == 0) set_error(p.err, kErrPos);
      return false;
    }
  } else {
    o.k_lo = W > 0 ? max(0, o.p_lo - W + 1) : 0;
    o.k_hi = o.p_hi;
  }
  o.kt0 = o.k_lo / kSN;
  o.n_tiles = o.k_hi / kSN - o.kt0 + 1;
  o.pt = p.page_table + (size_t)(p.rows.pt_row ? __ldg(p.rows.pt_row + b) : b) * p.max_pages;
  return true;
}

template <bool kSpan, bool kRope>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_sliding_kernel(const __grid_constant__ CUtensorMap tmap_q, PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  // The Q buffers are 128B-swizzled tiles and want 1024-byte alignment, which the dynamic shared
  // memory of a kernel without static shared memory has; a launch without it is refused
  // (G4_ERR_DEVICE) before any barrier exists. There is no room for an alignment pad.
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) set_error(p.err, kErrPage | kErrPos);
    return;
  }
  SlidingSmem& sm = *reinterpret_cast<SlidingSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();   // which query head of the KV head's pair
  const uint32_t peer = rank ^ 1u;
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
  const int W = p.window;

  if (threadIdx.x == 32) {
    for (int s = 0; s < kNK; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);   // QK^T commits (both CTAs), or the local Q move
      mbar_init(&sm.k_peer[s], 1);    // even CTA: the odd CTA's slot has landed
    }
    for (int s = 0; s < kNV; ++s) {
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
      mbar_init(&sm.v_ready[s], 1);   // even CTA: the odd CTA's V half landed and was checked
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.s_free, kPairWarps);   // even CTA: both CTAs' softmax warps have read S
    mbar_init(&sm.p_full, kPairWarps);   // even CTA: both CTAs' P is in tensor memory
    mbar_init(&sm.pv_done, 1);
    mbar_init(&sm.q_full, 1);            // Q dims 128-255 landed
    mbar_init(&sm.q_pair, kPairWarps);   // even CTA: both CTAs' Q is in place
    mbar_init(&sm.q_free, 1);            // the unit's last QK^T is done: Q may be replaced
    mbar_init(&sm.o_free, kPairWarps);   // even CTA: both CTAs have read O out
    mbar_init(&sm.q_read, kSmxWarps);    // this CTA's softmax warps have moved Q dims 0-127 out of qlo
    mbar_init(&sm.q_rot, kSmxWarps);     // kRope: this CTA's softmax warps have rotated Q
    for (int i = 0; i < 4; ++i) mbar_init(&sm.xchg[i], 2);
    mbar_init(&sm.teardown, 2);          // on an abort both issuers commit
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc2(&sm.tmem_base, 512);
    tmem_relinquish2();
  }
  tc_fence_before();
  cluster_sync_all();   // both CTAs' barriers and tensor memory exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tm = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;
  // Arrive on one of the even CTA's barriers: locally there, remotely from the odd CTA.
  auto arrive_leader = [&](uint64_t* bar) {
    if (leader)
      mbar_arrive(bar);
    else
      mbar_arrive_remote(map_peer(smem_u32(bar), 0u));
  };
  uint32_t k_slots = 0, v_slots = 0, q_units = 0;   // ring slots used, units (warp 0 keeps them for the teardown)

  if (warp == 0 || warp == 6) {
    // ------------------------------------------------------------ copy producers
    // Block indices come from the page table ahead of use: lane l holds page (l & 7) of tile
    // (l >> 3) of the current group of 4 tiles; the next group is looked up one group early.
    // Warp 0 copies this CTA's K pages (4r .. 4r+3 of the tile's 8), lanes 0-3 one page each,
    // and each unit's roped Q tile; warp 6 the dims half r of every page of the tile, lanes
    // 0-7 one page each. Pages outside [k_lo, k_hi] are neither looked up nor copied.
    const bool is_v = (warp == 6);
    uint64_t* full = is_v ? sm.v_full : sm.k_full;
    uint64_t* empty = is_v ? sm.v_empty : sm.k_empty;
    const int n_st = is_v ? kNV : kNK;
    const bool mine = is_v ? lane < 8 : lane < 4;
    const int pg = is_v ? (lane & 7) : (int)(4 * rank) + (lane & 3);   // page of the tile this lane copies
    uint32_t c = 0, vt = 0, q_issued = 0;
    int uq = 0;
    bool ok = true;
    if (!is_v && lane == 0) prefetch_tmap(&tmap_q);
    auto next_valid = [&](int& uu, Unit& o) -> bool {   // this cluster's first unit >= uu with rows
      for (; uu < p.n_units; uu += n_clusters)
        if (sliding_unit<kSpan>(p, uu, rank, o)) return true;
      return false;
    };
    auto raw_blocks = [&](const Unit& o, int j0) -> int {   // raw table entry of this lane's page
      const int jt = j0 + (lane >> 3);
      if (jt >= o.n_tiles) return kNoPage;
      return page_raw((o.kt0 + jt) * kSN + (lane & 7) * kPage, o.k_lo, o.k_hi, o.pt);
    };
    // Q tiles (warp 0): unit u's dims 0-127 into qlo and dims 128-255 into qhi[u & 1], all four
    // boxes of 64 dims x 128 rows (rows outside T read as 0) counted on q_full. Unit 0's goes
    // first; unit u + 1's right after unit u's second K tile (its first, for a unit of one tile),
    // once unit u's Q has left qlo for tensor memory (q_read). qhi[(u + 1) & 1] was last read by
    // unit u - 1's QK^T, which are done by then: the move of unit u's Q waited for them. So the
    // tile lands while unit u runs, and its rotation can start as soon as the softmax warps are
    // done with unit u.
    auto issue_q = [&](const Unit& o, int uo) {   // lane 0
      mbar_arrive_expect_tx(&sm.q_full, 4 * kQChunk);
#pragma unroll
      for (int c2 = 0; c2 < kSD / 64; ++c2)
        tma_load_3d(c2 < 2 ? sm.qlo + c2 * kQChunk : sm.qhi[uo & 1] + (c2 - 2) * kQChunk, &tmap_q, 64 * c2, o.h,
                    o.q_row0, &sm.q_full);
    };
    // The next unit is looked up, and the page-table entries of its first two groups of tiles
    // loaded, once the current unit's first slot is issued: at the unit boundary nothing waits
    // for memory, and the lookup does not delay the first copy.
    int u = cluster;
    Unit un;
    bool have = next_valid(u, un);
    int raw0 = have ? raw_blocks(un, 0) : kNoPage, raw1 = have ? raw_blocks(un, 4) : kNoPage;
    if (!is_v && have) {
      if (lane == 0) issue_q(un, 0);
      q_issued = 1;
    }
    while (ok && have) {
      int u2 = u + n_clusters;
      Unit nx;
      bool have_n = false;
      int nraw0 = kNoPage, nraw1 = kNoPage;
      auto load_blocks = [&](int j0) -> int {
        return page_check(raw_blocks(un, j0), p.num_pages, p.hkv, un.g, p.err);
      };
      int blk_cur = page_check(raw0, p.num_pages, p.hkv, un.g, p.err);
      int blk_next = page_check(raw1, p.num_pages, p.hkv, un.g, p.err);
      for (int j = 0; j < un.n_tiles; ++j, ++c) {   // key tile j of the unit
        const int s = c % n_st;
        if (j > 0 && (j & 3) == 0) {
          blk_cur = blk_next;
          blk_next = load_blocks(j + 4);
        }
        const int my_blk = __shfl_sync(0xffffffffu, blk_cur, (j & 3) * 8 + (pg & 7));
        const unsigned live = __ballot_sync(0xffffffffu, mine && my_blk >= 0);
        bool okw = true;
        if (lane == 0 && c >= (uint32_t)n_st)
          okw = mbar_wait_ool(&empty[s], ((c / n_st) - 1) & 1, abort_flag, p.err, p.wait_ns);
        if (!__shfl_sync(0xffffffffu, okw, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[s], __popc(live) * (is_v ? kVHalfPageBytes : kPageBytes));
        __syncwarp();
        if (mine && my_blk >= 0) {
          if (is_v)   // dims 128r .. 128r+127 of page pg: key groups 2pg, 2pg+1
            bulk_g2s(sm.v[s] + pg * kVHalfPageBytes,
                     (const __nv_bfloat16*)p.v_cache + (size_t)my_blk * kPage * kSD + rank * (kVHalfPageBytes / 2),
                     kVHalfPageBytes, &full[s]);
          else
            bulk_g2s(sm.k[s] + (lane & 3) * kPageBytes,
                     (const __nv_bfloat16*)p.k_cache + (size_t)my_blk * kPage * kSD, kPageBytes, &full[s]);
        }
        __syncwarp();
        if (j == 0) {
          have_n = next_valid(u2, nx);
          if (have_n) {
            nraw0 = raw_blocks(nx, 0);
            nraw1 = raw_blocks(nx, 4);
          }
        }
        if (!is_v && have_n && j == min(1, un.n_tiles - 1)) {   // the next unit's Q (see issue_q)
          bool okq = true;
          if (lane == 0) {
            okq = mbar_wait_ool(&sm.q_read, uq & 1, abort_flag, p.err, p.wait_ns);
            if (okq) issue_q(nx, uq + 1);
          }
          if (!__shfl_sync(0xffffffffu, okq, 0)) {
            ok = false;
            break;
          }
          ++q_issued;
        }
      }
      if (!is_v) vt += un.n_tiles;
      ++uq;
      un = nx;
      u = u2;
      have = have_n;
      raw0 = nraw0;
      raw1 = nraw1;
    }
    if (lane == 0 && *abort_flag) {   // drain copies still in flight (bounded) before the CTA may exit
      const unsigned long long w0 = globaltimer();
      if (q_issued > 0) {
        while (!mbar_try_wait(smem_u32(&sm.q_full), (q_issued - 1) & 1) && globaltimer() - w0 < kWaitLimitNs) {
        }
      }
      for (uint32_t i = c > (uint32_t)n_st ? c - n_st : 0; i < c; ++i) {
        while (!mbar_try_wait(smem_u32(&full[i % n_st]), (i / n_st) & 1) && globaltimer() - w0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
    k_slots = c;
    v_slots = vt;
    q_units = (uint32_t)uq;
  } else if (warp == 1 && !leader) {
    // ------------------------------------------------------------ K relay (odd CTA)
    uint32_t c = 0;
    bool ok = true;
    for (int u = cluster; ok && u < p.n_units; u += n_clusters) {
      Unit un;
      if (!sliding_unit<kSpan>(p, u, rank, un)) continue;
      for (int idx = 0; idx < un.n_tiles; ++idx, ++c) {   // every K ring slot
        const int s = c % kNK;
        ok = __all_sync(0xffffffffu, mbar_wait_ool(&sm.k_full[s], (c / kNK) & 1, abort_flag, p.err, p.wait_ns));
        if (!ok) break;
        if (lane == 0) mbar_arrive_remote(map_peer(smem_u32(&sm.k_peer[s]), peer));
        __syncwarp();
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK^T issuer (even CTA)
    // Issuing a group of MMAs blocks for about as long as they run, so QK^T and P.V have one
    // issuer each: neither waits for its operands while the tensor pipe idles. Each commit
    // tracks its own thread's MMAs only. Waits are warp-uniform, so that every lane leaves the
    // loops together on an abort.
    auto slot_ready = [&](uint32_t c) -> bool {   // K ring slot c has landed in both CTAs
      return mbar_wait_ool(&sm.k_full[c % kNK], (c / kNK) & 1, abort_flag, p.err, p.wait_ns) &&
             mbar_wait_cl_ool(&sm.k_peer[c % kNK], (c / kNK) & 1, abort_flag, p.err, p.wait_ns);
    };
    uint32_t c0 = 0, jt = 0;
    int uq = 0;
    bool ok = true;
    for (int u = cluster; ok && u < p.n_units; u += n_clusters) {
      Unit un;
      if (!sliding_unit<kSpan>(p, u, rank, un)) continue;
      // the unit's Q: both CTAs' softmax warps have rotated it and moved dims 0-127
      ok = __all_sync(0xffffffffu, mbar_wait_cl_ool(&sm.q_pair, uq & 1, abort_flag, p.err, p.wait_ns));
      for (int j = 0; ok && j < un.n_tiles; ++j, ++jt) {
        const uint32_t c = c0 + j;
        const int s = c % kNK;
        // the single S buffer: both CTAs' softmax threads have read the previous S into registers
        ok = __all_sync(0xffffffffu,
                        slot_ready(c) && (jt == 0 || mbar_wait_cl_ool(&sm.s_free, (jt - 1) & 1, abort_flag, p.err, p.wait_ns)));
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t ka = smem_u32(sm.k[s]);
          const uint32_t qh = smem_u32(sm.qhi[uq & 1]);
#pragma unroll
          for (int k = 0; k < 8; ++k)   // dims 0-127: Q from tensor memory
            mma2_ts(tm + kTmS, tm + kTmQ + 8 * k, desc_tiled(ka + k * 256, 128, kKeyGroupBytes), kIdescQK,
                    k > 0 ? 1u : 0u);
#pragma unroll
          for (int k = 8; k < 16; ++k)  // dims 128-255: Q from shared memory
            mma2_ss(tm + kTmS, desc_sw128(qh + ((k - 8) >> 2) * kQChunk + (k & 3) * 32, 16, 1024),
                    desc_tiled(ka + k * 256, 128, kKeyGroupBytes), kIdescQK, 1u);
          mma2_commit_mc(&sm.s_full, kBoth);
          mma2_commit_mc(&sm.k_empty[s], kBoth);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) mma2_commit_mc(&sm.q_free, kBoth);   // done with this unit's Q once these QK^T are
      __syncwarp();
      c0 += un.n_tiles;
      ++uq;
    }
  } else if (warp == 7) {
    // ------------------------------------------------------------ V check (both CTAs), P.V issuer (even CTA)
    // Value rows of this CTA's V half for keys that hold no data of this sequence are zeroed
    // before P.V: pages outside the key range were not copied and keep an older tile, and slots
    // past the sequence's last key may hold anything (NaN); P = 0 there does not cancel NaN.
    uint32_t cv = 0, jt = 0;
    int uq = 0;
    bool ok = true;
    for (int u = cluster; ok && u < p.n_units; u += n_clusters) {
      Unit un;
      if (!sliding_unit<kSpan>(p, u, rank, un)) continue;
      for (int i = 0; i < un.n_tiles; ++i, ++cv, ++jt) {
        const int s = cv % kNV;
        ok = __all_sync(0xffffffffu, mbar_wait_ool(&sm.v_full[s], (cv / kNV) & 1, abort_flag, p.err, p.wait_ns));
        if (!ok) break;
        const int kb = (un.kt0 + i) * kSN;
        const int v0 = max(kb, (un.k_lo >> 4) * kPage);
        const int v1 = min(min(kb + kSN, ((un.k_hi >> 4) + 1) * kPage), un.ctx_end);
        if (v0 > kb || v1 < kb + kSN) {
          for (int idx = lane; idx < kSN * 16; idx += 32) {
            const int r = idx >> 4, dg = idx & 15;
            if (kb + r < v0 || kb + r >= v1)
              *reinterpret_cast<uint4*>(sm.v[s] + ((r >> 3) * 16 + dg) * 128 + (r & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async();
        }
        __syncwarp();
        if (!leader) {
          if (lane == 0) mbar_arrive_remote(map_peer(smem_u32(&sm.v_ready[s]), peer));
          __syncwarp();
          continue;
        }
        // P_i is in place in both CTAs, the odd CTA's V half is ready, and (first tile of a
        // unit) the previous unit's O has been read out before this P.V overwrites it
        ok = __all_sync(0xffffffffu, mbar_wait_cl_ool(&sm.p_full, jt & 1, abort_flag, p.err, p.wait_ns) &&
                                         mbar_wait_cl_ool(&sm.v_ready[s], (cv / kNV) & 1, abort_flag, p.err, p.wait_ns) &&
                                         (i > 0 || uq == 0 || mbar_wait_cl_ool(&sm.o_free, (uq - 1) & 1, abort_flag, p.err, p.wait_ns)));
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t va = smem_u32(sm.v[s]);
#pragma unroll
          for (int k = 0; k < kSN / 16; ++k)   // 16 keys (two key groups) per step
            mma2_ts(tm + kTmO, tm + kTmP + 8 * k, desc_tiled(va + k * 2 * kVGroupBytes, kVGroupBytes, 128), kIdescPV,
                    (i > 0 || k > 0) ? 1u : 0u);
          mma2_commit_mc(&sm.pv_done, kBoth);
          mma2_commit_mc(&sm.v_empty[s], kBoth);
        }
        __syncwarp();
      }
      ++uq;
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue warps
    // Two warps per row quarter: warp w (2-5, 8-11) owns rows 32 (w % 4) .. +31 (its tensor-memory
    // lanes) and one half of the columns, hc = w / 8: keys 64 hc .. 64 hc + 63 of each S tile (P
    // key pairs 32 hc .. +31), dims 128 hc .. 128 hc + 127 of O. The two halves of a row meet
    // once per key tile to agree on the row max (so both scale P, l and O alike) and once per
    // unit to add their sums; everything else a thread does is its own half's.
    const int r = 32 * (warp & 3) + lane;   // query row = tensor-memory lane
    const int hc = warp >> 3;               // column half
    const int sidx = 32 * (warp < 8 ? warp - 2 : warp - 4) + lane;   // softmax thread 0 .. 255
    const uint32_t tq = tm + tmem_lane_base(warp);
    uint64_t* const xb = &sm.xchg[warp & 3];
    const float cl2 = p.scale_log2;
    uint32_t jt = 0, xph = 0;   // xph: exchanges of this row quarter so far
    int uq = 0, u = cluster - n_clusters;
    bool ok = true;
    auto next_unit = [&](Unit& o) -> bool {   // this cluster's next unit with rows (warp-wide)
      for (u += n_clusters; u < p.n_units; u += n_clusters)
        if (sliding_unit<kSpan>(p, u, rank, o)) return true;
      return false;
    };
    // Post this half's value of row r, then return the two halves' values (half 0's first). The
    // values of one exchange sit in xv[xph & 1]: the partner reads them before it can post its
    // next pair, and the one after that reuses the slot only once both have passed this one.
    auto exchange = [&](float v, float& v0, float& v1) -> bool {
      sm.xv[xph & 1][hc][r] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive(xb);
      if (!__all_sync(0xffffffffu, mbar_wait_ool(xb, xph & 1, abort_flag, p.err, p.wait_ns))) return false;
      v0 = sm.xv[xph & 1][0][r];
      v1 = sm.xv[xph & 1][1][r];
      ++xph;
      return true;
    };
    // Unit o's Q (dims 0-127 in qlo, dims 128-255 in qhi[uqo & 1], 128B swizzle; copied while the
    // unit before ran): with kRope rotated in place first, then dims 0-127 into tensor memory as
    // bf16 pairs, the A operand of half of the QK^T k-steps, once the unit before's QK^T are all
    // done with the columns. Each warp moves dims 64 hc .. +63 of its rows; q_read tells the Q
    // copier that qlo is free again.
    auto move_q = [&](const Unit& o, int uqo) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait_ool(&sm.q_full, uqo & 1, abort_flag, p.err, p.wait_ns))) return false;
      const uint8_t* qrow = sm.qlo + r * 128;
      if constexpr (kRope) {
        // softmax thread i rotates pair i % 128 of rows 64 (i / 128) .. +63
        const int t = sidx & 127;
        rotate_q_pair<4, kSlidingR>(sm.qlo + (t >> 6) * kQChunk, sm.qhi[uqo & 1] + (t >> 6) * kQChunk, p.tb, t,
                                    kBM * o.t, 64 * (sidx >> 7));
        fence_proxy_async();   // QK^T reads the rewritten dims 128-255 through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.q_rot);
        if (!__all_sync(0xffffffffu, mbar_wait_ool(&sm.q_rot, uqo & 1, abort_flag, p.err, p.wait_ns))) return false;
      }
      if (uqo > 0 && !__all_sync(0xffffffffu, mbar_wait_ool(&sm.q_free, (uqo - 1) & 1, abort_flag, p.err, p.wait_ns)))
        return false;
      tc_fence_after();
      {
        uint32_t w[32];
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          const uint4 v = *reinterpret_cast<const uint4*>(qrow + hc * kQChunk + ((q8 ^ (r & 7)) * 16));
          w[4 * q8] = v.x;
          w[4 * q8 + 1] = v.y;
          w[4 * q8 + 2] = v.z;
          w[4 * q8 + 3] = v.w;
        }
        tmem_st32(tq + kTmQ + 32 * hc, w);   // dims 64hc .. 64hc+63 -> columns 32hc .. 32hc+31
      }
      tmem_st_wait();
      tc_fence_before();
      fence_proxy_async();   // qlo is next written by the Q copy (async proxy), after these reads
      __syncwarp();
      if (lane == 0) {
        arrive_leader(&sm.q_pair);
        mbar_arrive(&sm.q_read);
      }
      return true;
    };

    // The unit after the current one is looked up at the start of the current one, while the
    // softmax waits for its first scores, so that moving its Q never waits for the lookup.
    Unit cur, nxt;
    bool have = next_unit(cur);
    if (have) ok = move_q(cur, uq);
    bool have_n = have && next_unit(nxt);
    constexpr int kHN = kSN / 2;   // keys of one half
    while (ok && have) {
      const int pos = kBM * cur.t + r;
      const bool row_ok = pos >= cur.p_lo && pos <= cur.p_hi;
      int row_lo = W > 0 ? max(0, pos - W + 1) : 0, row_hi = pos;   // the row's keys
      if (kSpan && row_ok) {
        row_keys(p.rows, W, cur.q_row0 + r, pos, cur.ctx_end, p.err, row_lo, row_hi);
        if (row_lo < cur.k_lo || row_hi > cur.k_hi) {   // spans that disagree between rows
          set_error(p.err, kErrSpan);
          row_lo = max(row_lo, cur.k_lo);
          row_hi = min(row_hi, cur.k_hi);
        }
      }
      float m_used = -INFINITY, l_half = 0.f;
      for (int j = 0; j < cur.n_tiles; ++j, ++jt) {
        const int kb = (cur.kt0 + j) * kSN + kHN * hc;   // this half's first key
        // Waits are made warp-uniform so that every lane leaves the loop together on an abort.
        if (!__all_sync(0xffffffffu, mbar_wait_ool(&sm.s_full, jt & 1, abort_flag, p.err, p.wait_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[kHN];
#pragma unroll
        for (int c = 0; c < kHN / 32; ++c)
          tmem_ld32(tq + kTmS + kHN * hc + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_leader(&sm.s_free);   // S may now be overwritten by the next QK^T

        float s[kHN];
#pragma unroll
        for (int c = 0; c < kHN; ++c) s[c] = __uint_as_float(sr[c]);
        const bool full = kSpan ? row_ok && kb >= row_lo && kb + kHN - 1 <= row_hi
                                : row_ok && kb + kHN - 1 <= pos && (W == 0 || pos - kb <= W - 1);
        if (!full) {   // the row's visible keys in this half are one run of columns [lo, hi]
          int lo = kSpan ? max(0, row_lo - kb) : (W > 0 ? max(0, pos - W + 1 - kb) : 0);
          int hi = row_ok ? min(kHN - 1, (kSpan ? row_hi : pos) - kb) : -1;
          if (hi < lo) lo = hi = 1 << 20;   // none
          const unsigned span = (unsigned)(hi - lo);
#pragma unroll
          for (int c = 0; c < kHN; ++c) s[c] = ((unsigned)(c - lo) <= span) ? s[c] : -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          mx[i] = s[i];
#pragma unroll
          for (int c = 1; c < kHN / 8; ++c) mx[i] = fmaxf(mx[i], s[i + 8 * c]);
        }
        float m0, m1;   // the two halves' maxima of the row
        if (!exchange(fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                            fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))),
                      m0, m1)) {
          ok = false;
          break;
        }
        const float mt = fmaxf(m0, m1) * cl2;
        float alpha = 1.f;
        bool need_o = false;
        if (mt > m_used + kLazyRescale) {
          need_o = (m_used != -INFINITY);
          alpha = ex2(m_used - mt);
          m_used = mt;
        }
        const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
        uint32_t pw[kHN / 2];
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w = 0; w < kHN / 2; ++w) {
          const float e0 = ex2(fmaf(s[2 * w], cl2, neg_m));
          const float e1 = ex2(fmaf(s[2 * w + 1], cl2, neg_m));
          ls[w & 3] += e0;
          ls[w & 3] += e1;
          pw[w] = pack_bf16(e0, e1);   // declared cast: P in bf16 for P.V
        }
        l_half = fmaf(l_half, alpha, (ls[0] + ls[1]) + (ls[2] + ls[3]));

        // The previous P.V has completed: the P buffer is free and O holds every earlier tile.
        if (jt > 0 && !__all_sync(0xffffffffu, mbar_wait_ool(&sm.pv_done, (jt - 1) & 1, abort_flag, p.err, p.wait_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, need_o)) {   // O correction (rows whose max rose by more than 2^8)
          const float a = need_o ? alpha : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < kSD / 64; ++cc) {
            uint32_t o[32];
            tmem_ld32(tq + kTmO + (kSD / 2) * hc + 32 * cc, o);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * a);
            tmem_st32(tq + kTmO + (kSD / 2) * hc + 32 * cc, o);
          }
        }
        // This half of P_j (bf16 key pairs 32 hc .. +31): the A operand of P.V.
        tmem_st32(tq + kTmP + 32 * hc, *reinterpret_cast<const uint32_t(*)[32]>(&pw[0]));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_leader(&sm.p_full);
      }
      if (!ok) break;

      // The next unit's Q goes into tensor memory now (this unit's QK^T are all done), so that
      // its first QK^T runs while this unit's O is written out.
      if (have_n && !move_q(nxt, uq + 1)) {
        ok = false;
        break;
      }

      // Epilogue: O / l -> bf16, rows of this sequence only, this half's dims. Once O is in
      // registers the even CTA may start the next unit's P.V, which overwrites it.
      float l0, l1;   // the halves' sums, added in a fixed order
      if (!exchange(l_half, l0, l1) ||
          !__all_sync(0xffffffffu, mbar_wait_ool(&sm.pv_done, (jt - 1) & 1, abort_flag, p.err, p.wait_ns))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float l_run = l0 + l1;
      const float inv = (l_run > 0.f) ? __frcp_rn(l_run) : 0.f;
      const unsigned valid = __ballot_sync(0xffffffffu, row_ok);
      const long long wrow0 = (long long)cur.q_row0 + 32 * (warp & 3);
#pragma unroll 1
      for (int cc = 0; cc < kSD / 64; ++cc) {
        uint32_t o[32];
        tmem_ld32(tq + kTmO + (kSD / 2) * hc + 32 * cc, o);
        tmem_ld_wait();
        if (cc == kSD / 64 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_leader(&sm.o_free);
        }
        uint32_t w16[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          w16[c] = pack_bf16(__uint_as_float(o[2 * c]) * inv, __uint_as_float(o[2 * c + 1]) * inv);
        store_rows32<kSD>(w16, p.out, wrow0, p.hq, cur.h, (kSD / 2) * hc + 32 * cc, valid, lane);
      }
      ++uq;
      cur = nxt;
      have = have_n;
      if (have) have_n = next_unit(nxt);
    }
  }

  // ------------------------------------------------------------ teardown
  // Neither CTA may free its tensor memory or leave while the pair's MMAs or signals into it
  // are in flight: each waits (bounded) for the last stage releases and the last Q release it
  // was sent, an abort is passed to the peer so that its waits end early, and a cluster barrier
  // closes the pair. Aligned CTA barriers count whole warps: every warp arrives converged.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    if (*abort_flag) {
      st_peer_u32(map_peer(smem_u32(&sm.abort_flag), peer), 1u);
    } else {
      const unsigned long long w0 = globaltimer();
      for (uint32_t s = 0; s < (uint32_t)kNK && s < k_slots; ++s) {
        const uint32_t last = s + kNK * ((k_slots - 1 - s) / kNK);
        while (!mbar_try_wait(smem_u32(&sm.k_empty[s]), (last / kNK) & 1u) && globaltimer() - w0 < kWaitLimitNs) {
        }
      }
      for (uint32_t s = 0; s < (uint32_t)kNV && s < v_slots; ++s) {
        const uint32_t last = s + kNV * ((v_slots - 1 - s) / kNV);
        while (!mbar_try_wait(smem_u32(&sm.v_empty[s]), (last / kNV) & 1u) && globaltimer() - w0 < kWaitLimitNs) {
        }
      }
      const uint32_t units = q_units;
      if (units > 0) {
        while (!mbar_try_wait(smem_u32(&sm.q_free), (units - 1) & 1u) && globaltimer() - w0 < kWaitLimitNs) {
        }
      }
    }
  }
  __syncwarp();
  __syncthreads();
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1 || warp == 7) {
    tc_fence_after();
    if (sm.abort_flag) {   // let every issued MMA finish before the columns are freed
      if (leader && lane == 0) mma2_commit_mc(&sm.teardown, kBoth);   // both issuers
      __syncwarp();
      if (warp == 1) {
        const unsigned long long w0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&sm.teardown), 0) && globaltimer() - w0 < kWaitLimitNs) {
        }
      }
    }
    if (warp == 1) tmem_dealloc2(tm, 512);
  }
}

}  // namespace

cudaError_t launch_prefill(bool global, const SeqRows& rows, int window, float scale_log2, const PagedCache& cache,
                           void* out, const DeviceState& st, cudaStream_t s, const void* q_raw) {
  if (global) return launch_prefill_global(rows, scale_log2, cache, out, st, s, q_raw);
  PrefillParams p{};
  p.rows = rows;
  p.window = window;
  p.scale_log2 = scale_log2;
  p.num_pages = cache.num_pages;
  p.page_table = cache.page_table;
  p.max_pages = cache.max_pages;
  p.out = (__nv_bfloat16*)out;
  p.tb = st.sliding;
  p.err = st.err;
  p.wait_ns = wait_limit_ns();
  p.k_cache = cache.k;
  p.v_cache = cache.v;
  p.hq = cache.hq;
  p.hkv = cache.hkv;
  // Raw queries are rotated in the kernel; otherwise the staged roped queries are read from `out`.
  // Image spans come only with staged queries.
  if (rows.span && q_raw) return cudaErrorInvalidValue;
  CUtensorMap mq;
  if (!q_map(&mq, q_raw ? q_raw : out, rows.T, cache.hq, kSD)) return cudaErrorInvalidValue;
  // Batches with image rows take their own instantiation, so that the plain one carries no span code.
  auto kernel = rows.span ? prefill_sliding_kernel<true, false>
                          : (q_raw ? prefill_sliding_kernel<false, true> : prefill_sliding_kernel<false, false>);
  const int ki = rows.span ? 1 : (q_raw ? 2 : 0);
  static bool attr[64][3] = {};
  static int max_clusters[64][3] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr[dev][ki]) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSlidingSmemBytes);
    if (e != cudaSuccess) return e;
    // clusters that fit on the device at once: the persistent grid
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSlidingSmemBytes;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeClusterDimension;
    la[0].val.clusterDim.x = 2;
    la[0].val.clusterDim.y = 1;
    la[0].val.clusterDim.z = 1;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    if (e != cudaSuccess) return e;
    max_clusters[dev][ki] = n > 0 ? n : 1;
    attr[dev][ki] = true;
  }
  const long long slots = (long long)rows.T / kBM + 2LL * rows.B;
  const long long n_units = slots * cache.hkv;   // (query tile, KV head) units, one per cluster at a time
  if (n_units <= 0 || n_units > 0x3fffffffLL) return cudaErrorInvalidValue;
  p.n_units = (int)n_units;
  const int n_clusters = (int)(n_units < max_clusters[dev][ki] ? n_units : max_clusters[dev][ki]);
  kernel<<<2u * (unsigned)n_clusters, kThreads, kSlidingSmemBytes, s>>>(mq, p);
  return cudaGetLastError();
}

}  // namespace g4
