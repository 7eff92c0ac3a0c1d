// Global-layer prefill on tcgen05: full causal attention, 32 Q / 4 KV heads, head dim 512,
// K==V (RL-Kernel RFC "[RFC][Gemma-4-31B-it] WS1/WS2 kernel roadmap", section 5,
// global_attention_core and global_k_eq_v_projection; section 2: proportional p-RoPE, partial
// factor 0.25, theta 1e6).
//
// A 128 x 512 fp32 output tile fills all 512 tensor-memory columns of one SM, so no SM can hold
// both the output of its rows and their scores. The work of one unit, (sequence, 128-row query
// tile, pair of query heads 2i, 2i+1 of one KV head), is therefore split over a cluster of four
// CTAs forming two 2-SM MMA pairs:
//   - the score pair (ranks 0, 1; rank r owns head 2i + r): S = Q K^T as one cta_group::2 MMA
//     over both heads (M = 256, N = 128 keys, K = 512 dims; each CTA stages 64 keys of every
//     key tile, all dims), then the online softmax of its head's rows. Each CTA sends its bf16 P
//     tile and per-row (alpha, l) to the output CTA of its head by bulk copies into that CTA's
//     shared memory;
//   - the output pair (ranks 2, 3; rank 2 + r owns head 2i + r): O += P V as one cta_group::2
//     MMA (M = 256, N = 256 dims per instruction, two instructions per 16-key step), V being the
//     stored un-rotated S (each CTA stages its 256-dim half of every key). Its warps apply the
//     lazy O rescale that alpha asks for and write the output.
// The rotated quarter of K comes from the cache's k_rot side pages (p-RoPE(S), written with S by
// the append pass); the un-rotated dims of K and all of V come from the same stored S pages.
// Key tiles of 128 keys are aligned to absolute key 0 and visited in ascending order, query
// tiles to absolute position; every row's arithmetic depends only on its own position and its
// sequence's keys (section 4 rules 2, 3 and 6).
//
// Score CTA warps: 0 copies this CTA's K half of each key tile into a 3-stage ring; 7 copies each
// unit's Q tile (TMA) into K stages 1-2 as soon as every QK^T of the earlier unit is done; 6 (rank 0)
// waits for each tile's operands (the unit's Q in place, both CTAs' K halves, the S buffer read)
// and hands the tile to the issuer; 1 issues QK^T (rank 0) or tells rank 0 that its ring slot has
// landed (rank 1); 2-5 move Q into tensor memory, then run mask, online softmax and P (one thread
// per row). Output CTA warps: 0 copies this CTA's V half of each 64-key half tile into a 4-stage
// ring; 7 (rank 2) or 1 (rank 3) zeroes value rows that hold no key of the sequence, then hands the
// step to the P.V issuer once the rest of its operands are ready (rank 2) or tells rank 2 that its
// half is ready (rank 3); 1 (rank 2) issues P.V; 2-5 check alpha, rescale O when asked, and write
// the output; 6 hands P slots back to the score CTA once P.V has read them. Issuing a group of MMAs
// blocks the issuing thread for about as long as they run, so the issuers wait on one barrier each
// (their helpers wait on the rest, three of them at cluster scope), and the next tile's MMAs follow
// the last ones closely.
// Queries (kRope): the Q tile is copied from the raw query rows and its 64 turning pairs (dims 0-63
// with 256-319) are rotated in place in shared memory before the move into tensor memory: softmax
// thread i rotates pair i % 64 of rows 64 (i / 64) .. +63 (rotate_q_pair; rows outside the sequence
// turn too, harmlessly), and the four softmax warps meet on an mbarrier before each moves its row. The angles, rotation and bf16 cast are the
// append pass's, so the queries get the bits a staged call gives. Otherwise (the staged form: normed queries, image spans, the exact decode) the append pass
// wrote bf16(p-RoPE(q)) into the sequence rows of `out`, which the Q copies read.
// Tensor memory, score CTAs: Q [0,256) as bf16 pairs, two S buffers [256,384), [384,512).
// Output CTAs: O [0,512), where column c holds dim c for c < 128 or c >= 384, dim c + 128 for
// 128 <= c < 256 and dim c - 128 for 256 <= c < 384 (each instruction's N = 256 columns are
// 128 dims of rank 2's half followed by the same 128 dims of rank 3's half).
#include <math.h>

#include "g4_prefill_common.cuh"

namespace g4 {

namespace {

using namespace pf;

constexpr int kGD = kGlobalD;       // 512
constexpr int kHalf = kGD / 2;      // 256
constexpr int kTN = 128;            // keys per tile: N of QK^T over the score pair
constexpr int kVN = 64;             // keys per V stage
constexpr int kNK = 3;              // K ring stages (score CTAs)
constexpr int kNV = 4;              // V ring stages (output CTAs)
constexpr int kNP = 2;              // S buffers (score CTAs) and P slots (output CTAs)
constexpr int kThreads = 256;
constexpr uint16_t kScorePair = 0x3, kOutPair = 0xC;

// Score-CTA K stage: this CTA's 64 keys of a tile (4 pages), all 512 dims. Each page arrives as
// two tensor copies whose boxes put the key group outside the dim half, so that for either half
// the 8 key groups of the stage sit at one fixed stride (the matrix descriptor's SBO):
//   dims 64..255 of each half (from S): [page (4)][key group (2)][half (2)][dim group 8..31 (24)][8][8]
//   at 0, key-group stride 6 KB;
//   dims 0..63 of each half (from k_rot): [page (4)][key group (2)][half (2)][dim group (8)][8][8]
//   at kRotOff, key-group stride 2 KB.
constexpr int kUnrotCM = 24 * 128;               // 3 KB: 24 core matrices of one (key group, half)
constexpr int kUnrotKG = 2 * kUnrotCM;           // 6 KB
constexpr int kUnrotPage = 2 * kUnrotKG;         // 12 KB
constexpr int kRotCM = 8 * 128;                  // 1 KB
constexpr int kRotKG = 2 * kRotCM;               // 2 KB
constexpr int kRotPage = 2 * kRotKG;             // 4 KB
constexpr int kRotOff = 4 * kUnrotPage;          // 48 KB
constexpr int kKStage = kRotOff + 4 * kRotPage;  // 64 KB
constexpr int kKPageBytes = kUnrotPage + kRotPage;   // 16 KB: one page's share of a stage
// The Q tile (8 boxes of 64 dims x 128 rows, 128B swizzle) lands at the first 1024-byte
// boundary at or after K stage 1; it may reach up to 1008 bytes into the P staging area, which is
// first written after every softmax warp of both score CTAs has moved Q into tensor memory.
// P tile of one head: [row group (16)][key group (17)][8 rows][8 keys] bf16. Key groups 0-15 are
// P (the A operand of P.V, row-group stride kPRowGroup); key group 16 carries the row's softmax
// state instead: alpha (fp32) in bytes 0-3 and l (fp32) in bytes 4-7 of its 16-byte row. The
// rows of one softmax warp (4 row groups) are contiguous, so one bulk copy per warp carries them.
constexpr int kPRowGroup = 17 * 128;             // 2176 B
constexpr int kPSlot = 16 * kPRowGroup;          // 34 KB
constexpr int kPWarpBytes = kPSlot / 4;          // 8.5 KB
constexpr uint32_t kPSendBytes = kPSlot;         // bytes one tile's copies deliver into a P slot
// Output-CTA V stage: 64 keys x this CTA's 256 dims: [key group (8)][dim group (32)][8][8].
constexpr int kVKG = 32 * 128;                   // 4 KB
constexpr int kVStage = 8 * kVKG;                // 32 KB
constexpr int kVPageBytes = 2 * kVKG;            // 8 KB: one page's half-block
// Byte offsets in the data area. Score CTAs: K ring [0, 192K), P staging [192K, 226K).
// Output CTAs: V ring [0, 128K), two P slots [128K, 196K).
constexpr int kSOffStage = kNK * kKStage;
constexpr int kOOffP = kNV * kVStage;
constexpr int kDataBytes = kSOffStage + kPSlot;   // 226 KB
static_assert(kOOffP + kNP * kPSlot <= kDataBytes, "output CTA layout exceeds the data area");
static_assert(kKStage + 1023 + 8 * kQChunk <= kDataBytes, "Q must fit between K stage 1 and the end");

constexpr uint32_t kTmQ = 0, kTmS = 256, kTmO = 0;
constexpr uint32_t kIdescQK = idesc_bf16(2 * kBM, kTN, false, false);   // M 256 over the pair, N 128 keys
constexpr uint32_t kIdescPV = idesc_bf16(2 * kBM, 256, false, true);    // M 256, N 256 dims

struct Bars {
  // score CTAs
  uint64_t k_full[kNK], k_empty[kNK], k_peer[kNK];
  uint64_t s_full[kNP], s_free[kNP], p_free[kNP];
  uint64_t q_full, q_moved, q_pair, stg_free, q_rot, go[2];
  uint64_t q_free;           // score CTAs: every QK^T of the unit is done (the issuer's commit, both CTAs)
  // output CTAs
  uint64_t v_full[kNV], v_empty[kNV], v_ready[kNV];
  uint64_t p_full[kNP], o_ready[kNP], pv_done[kNP];
  uint64_t o_free;           // output CTAs (rank 2): both CTAs' epilogue warps have read O out
  uint64_t go_pv[kNV];       // output CTAs (rank 2): the helper has seen V stage s's P.V ready
  uint64_t teardown;
  uint32_t tmem_base;
  int abort_flag;
  int p_seen[kNP];   // output CTAs: phases of each P slot consumed (for the abort drain)
  int q_issued;      // score CTAs: Q tiles issued (by thread 64; read by the abort drain)
};

struct GlobalSmem {
  uint8_t data[kDataBytes];
  Bars bar;
};
// The data area needs 128-byte alignment only (bulk copies, matrix descriptors); the Q staging
// finds its own 1024-byte boundary.
constexpr size_t kGlobalSmemBytes = sizeof(GlobalSmem) + 128;
static_assert(kGlobalSmemBytes <= 232448, "global prefill exceeds the 227 KB shared-memory limit");

// Output-CTA tensor-memory column -> head dim (see the header).
__device__ __forceinline__ int o_dim(int col) {
  return (col < 128 || col >= 384) ? col : (col < 256 ? col + 128 : col - 128);
}

// One unit as the CTAs of its cluster see it: (sequence b, query tile t, head pair hp); this CTA's
// head h (of the pair) reads KV head g. Keys k_lo .. k_hi in n_tiles tiles from key tile kt0.
struct GUnit {
  int b, t, hp, h, g, p_lo, p_hi, ctx_end, q_row0, k_lo, k_hi, kt0, n_tiles;
  const int32_t* pt;
};

// Warp-wide. False when unit u holds no rows or is refused (the error word is then set); every role
// of the four CTAs skips such units alike, so all of them walk the same units in the same order. A
// partial call's unit may have no key of its range (n_tiles 0): the roles that write rows write an
// empty partial, the others skip it. Not inlined: nine roles call it.
template <bool kPart>
__device__ __noinline__ bool global_unit(const PrefillParams& p, int u, uint32_t pr, GUnit& o) {
  o.hp = u % (p.hq / 2);
  o.h = 2 * o.hp + (int)pr;
  o.g = o.h / (p.hq / p.hkv);   // both heads of the pair share KV head g
  int b, t, f[3];
  find_unit(p.rows, u / (p.hq / 2), b, t, p.err, f);
  if (b < 0) return false;
  const int cs = f[0], L = f[1], qs = f[2];
  o.b = b;
  o.t = t;
  o.p_lo = max(kBM * t, cs);
  o.p_hi = min(kBM * t + kBM - 1, cs + L - 1);
  o.ctx_end = cs + L;
  if (o.p_hi >= kMaxPos || (o.p_hi >> 4) >= p.max_pages) {
    if ((threadIdx.x & 31) == 0) set_error(p.err, kErrPos);
    return false;
  }
  o.q_row0 = qs + (kBM * t - cs);
  // Keys 0 .. k_hi: the last row's run ends no earlier than any other row's (an image holding a
  // row of the tile and reaching past the last row holds the last row too).
  int lo_unused;
  row_keys(p.rows, 0, o.q_row0 + (o.p_hi - kBM * t), o.p_hi, o.ctx_end, p.err, lo_unused, o.k_hi);
  if ((o.k_hi >> 4) >= p.max_pages) {   // an image past the page table (the rows' own pages fit)
    if ((threadIdx.x & 31) == 0) set_error(p.err, kErrPos);
    return false;
  }
  // kPart: only keys key_begin .. key_end-1 of the sequence; the tiles start at the one holding
  // key_begin (tile j of the unit is key tile kt0 + j).
  o.k_lo = 0;
  if (kPart) {
    o.k_lo = max(0, __ldg(p.key_begin + b));
    o.k_hi = min(o.k_hi, __ldg(p.key_end + b) - 1);
  }
  o.kt0 = o.k_lo / kTN;
  o.n_tiles = o.k_hi >= o.k_lo ? o.k_hi / kTN - o.kt0 + 1 : 0;
  o.pt = p.page_table + (size_t)(p.rows.pt_row ? __ldg(p.rows.pt_row + b) : b) * p.max_pages;
  return true;
}

// The k-th unit of cluster c of C: rounds of C units. When the units are listed from the most
// expensive down (the exact decode's chunks), odd rounds are walked backwards (a snake), so that
// the clusters' shares even out; otherwise every round is walked forwards, which keeps the clusters
// of one KV head on neighbouring units, reading the same key tiles from L2 at about the same time
// (the snake measured 2% slower on a causal prefill). A fixed assignment either way: which cluster
// computes a unit changes none of its bits.
__device__ __forceinline__ int unit_at(int k, int c, int C, bool snake) {
  return k * C + ((snake && (k & 1)) ? C - 1 - c : c);
}

template <bool kRope, bool kPart>
__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_global_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_s,
                          const __grid_constant__ CUtensorMap tmap_rot, PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  GlobalSmem& sm = *reinterpret_cast<GlobalSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint8_t* const base = sm.data;
  uint8_t* const q_stage = base + kKStage + ((1024u - (smem_u32(base + kKStage) & 1023u)) & 1023u);
  // When the Q staging is clear of the P staging (the data area is 1024-byte aligned, as it is in
  // practice), warp 7 copies each unit's Q as soon as every QK^T of the earlier unit is done;
  // otherwise softmax thread 64 does, once the last P copy has also left the staging. The same for
  // every CTA of the grid.
  const bool q_sep = q_stage + 8 * kQChunk <= base + kSOffStage;
  Bars& bar = sm.bar;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool is_out = rank >= 2;
  const uint32_t pr = rank & 1u;             // which head of the pair
  const uint32_t pair_peer = rank ^ 1u;      // the other CTA of this MMA pair
  const uint32_t partner = rank ^ 2u;        // score CTA r <-> output CTA r + 2 (same head)
  const bool leader = pr == 0;               // issues the pair's MMAs
  const int cluster = blockIdx.x >> 2, n_clusters = gridDim.x >> 2;

  // The output CTAs' P-slot warp counts the cluster's key tiles over all its units before the
  // cluster barrier: it posts the bytes of the first two tiles' P before any copy can arrive.
  int total_tiles = 0;
  if (is_out && warp == 6) {
    for (int k = 0, u = unit_at(0, cluster, n_clusters, p.rows.by_cost); u < p.n_units; u = unit_at(++k, cluster, n_clusters, p.rows.by_cost)) {
      GUnit o;
      if (global_unit<kPart>(p, u, pr, o)) total_tiles += o.n_tiles;
    }
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < kNK; ++s) {
      mbar_init(&bar.k_full[s], 1);
      mbar_init(&bar.k_empty[s], 1);
      mbar_init(&bar.k_peer[s], 1);
    }
    for (int s = 0; s < kNP; ++s) {
      mbar_init(&bar.s_full[s], 1);
      mbar_init(&bar.s_free[s], 8);    // rank 0: both score CTAs' softmax warps have read S
      mbar_init(&bar.p_free[s], 1);    // the output CTA's P.V has read this P slot
      mbar_init(&bar.p_full[s], 1);    // one local expect-tx arrive, then the score CTA's bytes
      mbar_init(&bar.o_ready[s], 8);   // rank 2: both output CTAs have checked alpha (and rescaled O)
      mbar_init(&bar.pv_done[s], 1);   // P.V of tiles of this parity
      bar.p_seen[s] = 0;
    }
    bar.q_issued = 0;
    mbar_init(&bar.q_full, 1);
    mbar_init(&bar.q_moved, kSoftmaxThreads / 32);
    mbar_init(&bar.q_pair, 8);
    mbar_init(&bar.stg_free, 1);
    mbar_init(&bar.q_free, 1);
    mbar_init(&bar.go[0], 1);
    for (int s = 0; s < kNV; ++s) mbar_init(&bar.go_pv[s], 1);
    mbar_init(&bar.go[1], 1);
    mbar_init(&bar.q_rot, kSoftmaxThreads / 32);   // kRope: the softmax warps have rotated Q
    for (int s = 0; s < kNV; ++s) {
      mbar_init(&bar.v_full[s], 1);
      mbar_init(&bar.v_empty[s], 1);
      mbar_init(&bar.v_ready[s], 1);
    }
    mbar_init(&bar.o_free, 8);   // rank 2: both output CTAs' epilogue warps have read O out
    mbar_init(&bar.teardown, 1);
    bar.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (is_out && threadIdx.x == 192) {   // the first two tiles' P may arrive once the cluster is up
    for (int s = 0; s < kNP && s < total_tiles; ++s) mbar_arrive_expect_tx(&bar.p_full[s], kPSendBytes);
  }
  if (warp == 1) {
    tmem_alloc2(&bar.tmem_base, 512);
    tmem_relinquish2();
  }
  tc_fence_before();
  cluster_sync_all();   // every CTA's barriers and tensor memory exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tm = bar.tmem_base;
  volatile int* abort_flag = &bar.abort_flag;
  auto arrive_leader = [&](uint64_t* br) {   // arrive on the pair leader's copy of a barrier
    if (leader)
      mbar_arrive(br);
    else
      mbar_arrive_remote(map_peer(smem_u32(br), pair_peer));
  };
  // Copies in flight at an abort, kept by the producer warps (lane 0 is thread 0).
  uint32_t kuse[kNK] = {0u, 0u, 0u};   // score CTAs: uses of each K stage (each unit starts at stage 0)
  uint32_t vc_total = 0;               // output CTAs: V stages issued

  if (!is_out) {
    // ================================================================ score CTAs
    if (warp == 0) {
      // ------------------------------------------------------------ K copies
      if (lane == 0) {
        prefetch_tmap(&tmap_s);
        prefetch_tmap(&tmap_rot);
      }
      const int pl = lane & 3;
      bool ok = true;
      for (int k = 0, ui = 0, u = unit_at(0, cluster, n_clusters, p.rows.by_cost); ok && u < p.n_units; u = unit_at(++k, cluster, n_clusters, p.rows.by_cost)) {
        GUnit un;
        if (!global_unit<kPart>(p, u, pr, un) || un.n_tiles == 0) continue;
        // Lanes 0-3 copy the un-rotated dims of page `lane` of this CTA's 64 keys, lanes 4-7 its
        // k_rot block. Pages outside [k_lo, k_hi] are neither looked up nor copied. Block indices
        // come from the page table ahead of use: lane l holds page (l & 3) of tile (l >> 2) of the
        // current group of 8 tiles, and the next group is looked up one group early.
        auto load_blocks = [&](int j0) -> int {
          const int jt = j0 + (lane >> 2);
          if (jt >= un.n_tiles) return -1;
          return page_block((un.kt0 + jt) * kTN + 64 * (int)pr + kPage * (lane & 3), un.k_lo, un.k_hi, un.pt,
                            p.num_pages, p.hkv, un.g, p.err);
        };
        int blk_cur = load_blocks(0), blk_next = load_blocks(8);
        for (int j = 0; j < un.n_tiles; ++j) {
          const int s = j % kNK;
          if (j > 0 && (j & 7) == 0) {
            blk_cur = blk_next;
            blk_next = load_blocks(j + 8);
          }
          const int bl = __shfl_sync(0xffffffffu, blk_cur, (j & 7) * 4 + (lane & 3));
          const unsigned live = __ballot_sync(0xffffffffu, lane < 4 && bl >= 0);
          const int blk = __shfl_sync(0xffffffffu, bl, pl);
          bool okw = true;
          if (lane == 0) {
            // Stages 1-2 hold the unit's Q until the softmax warps have moved it; Q landed there
            // only after the earlier tiles in them were read, so tile 2 needs no wait of its own.
            if (j == 1)
              okw = mbar_wait(&bar.q_moved, ui & 1, abort_flag, p.err, p.wait_ns);
            else if (j != 2 && kuse[s] > 0)
              okw = mbar_wait(&bar.k_empty[s], (kuse[s] - 1) & 1, abort_flag, p.err, p.wait_ns);
          }
          if (!__shfl_sync(0xffffffffu, okw, 0)) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(&bar.k_full[s], __popc(live) * kKPageBytes);
          __syncwarp();
          if (lane < 8 && blk >= 0) {
            uint8_t* st = base + s * kKStage;
            if (lane < 4)   // box {64, 24 dim groups from 8, 2 halves, 2 key groups, 1 block}
              tma_load_5d(st + pl * kUnrotPage, &tmap_s, 0, 8, 0, 0, blk, &bar.k_full[s]);
            else            // box {64, 8 dim groups, 2 halves, 2 key groups, 1 block}
              tma_load_5d(st + kRotOff + pl * kRotPage, &tmap_rot, 0, 0, 0, 0, blk, &bar.k_full[s]);
          }
          __syncwarp();
          ++kuse[s];
        }
        // (A unit of one tile never waits on q_moved; still, this warp is never two phases of it
        // ahead, which a parity wait could not tell apart: the next unit's tile 0 waits for stage
        // 0's last use, whose QK^T came after that unit's Q had moved.)
        ++ui;
      }
    } else if (warp == 1 && !leader) {
      // ------------------------------------------------------------ K relay (rank 1)
      bool ok = true;
      for (int k = 0, u = unit_at(0, cluster, n_clusters, p.rows.by_cost); ok && u < p.n_units; u = unit_at(++k, cluster, n_clusters, p.rows.by_cost)) {
        GUnit un;
        if (!global_unit<kPart>(p, u, pr, un) || un.n_tiles == 0) continue;
        for (int j = 0; j < un.n_tiles; ++j) {
          const int s = j % kNK;
          if (!__all_sync(0xffffffffu, mbar_wait(&bar.k_full[s], kuse[s] & 1, abort_flag, p.err, p.wait_ns))) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_remote(map_peer(smem_u32(&bar.k_peer[s]), pair_peer));
          __syncwarp();
          ++kuse[s];
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ QK^T issuer (rank 0)
      bool ok = true;
      int tc = 0;
      for (int k = 0, ui = 0, u = unit_at(0, cluster, n_clusters, p.rows.by_cost); ok && u < p.n_units; u = unit_at(++k, cluster, n_clusters, p.rows.by_cost)) {
        GUnit un;
        if (!global_unit<kPart>(p, u, pr, un) || un.n_tiles == 0) continue;
        for (int j = 0; ok && j < un.n_tiles; ++j) {
          const int s = j % kNK, gt = tc + j, sb = gt % kNP;
          // the helper warp has seen this tile's operands ready
          ok = __all_sync(0xffffffffu, mbar_wait(&bar.go[gt & 1], (gt >> 1) & 1, abort_flag, p.err, p.wait_ns));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t st = smem_u32(base + s * kKStage);
            const uint32_t sd = tm + kTmS + kTN * sb;
#pragma unroll
            for (int ks = 0; ks < kGD / 16; ++ks) {   // dims 16ks .. 16ks+15
              const int hh = ks >> 4, kk = ks & 15;
              const uint64_t bd = kk < 4 ? desc_tiled(st + kRotOff + hh * kRotCM + kk * 256, 128, kRotKG)
                                         : desc_tiled(st + hh * kUnrotCM + (kk - 4) * 256, 128, kUnrotKG);
              mma2_ts(sd, tm + kTmQ + 8 * ks, bd, kIdescQK, ks > 0 ? 1u : 0u);
            }
            mma2_commit_mc(&bar.s_full[sb], kScorePair);
            mma2_commit_mc(&bar.k_empty[s], kScorePair);
          }
          __syncwarp();
          ++kuse[s];
        }
        if (!ok) break;
        if (q_sep && lane == 0) mma2_commit_mc(&bar.q_free, kScorePair);   // the unit's QK^T are all done
        __syncwarp();
        tc += un.n_tiles;
        ++ui;
      }
    } else if (warp == 7 && q_sep) {
      // ------------------------------------------------------------ Q copies (each score CTA)
      // The unit's Q goes into K stages 1-2 as soon as every QK^T of the earlier unit is done.
      bool ok = true;
      int ui = 0;
      for (int k = 0, u = unit_at(0, cluster, n_clusters, p.rows.by_cost); ok && u < p.n_units; u = unit_at(++k, cluster, n_clusters, p.rows.by_cost)) {
        GUnit un;
        if (!global_unit<kPart>(p, u, pr, un) || un.n_tiles == 0) continue;
        if (ui > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bar.q_free, (ui - 1) & 1, abort_flag, p.err, p.wait_ns));
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar.q_full, 8 * kQChunk);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            tma_load_3d(q_stage + c * kQChunk, &tmap_q, 64 * c, un.h, un.q_row0, &bar.q_full);
          bar.q_issued = ui + 1;
        }
        __syncwarp();
        ++ui;
      }
      // the last unit's commit lands before the CTA may leave
      if (ok && ui > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bar.q_free, (ui - 1) & 1, abort_flag, p.err, p.wait_ns));
    } else if (warp == 6 && leader) {
      // ------------------------------------------------------------ QK^T helper (rank 0)
      bool ok = true;
      int tc = 0;
      for (int k = 0, ui = 0, u = unit_at(0, cluster, n_clusters, p.rows.by_cost); ok && u < p.n_units; u = unit_at(++k, cluster, n_clusters, p.rows.by_cost)) {
        GUnit un;
        if (!global_unit<kPart>(p, u, pr, un) || un.n_tiles == 0) continue;
        ok = __all_sync(0xffffffffu, mbar_wait_cl(&bar.q_pair, ui & 1, abort_flag, p.err, p.wait_ns));
        for (int j = 0; ok && j < un.n_tiles; ++j) {
          const int s = j % kNK, gt = tc + j, sb = gt % kNP;
          ok = __all_sync(0xffffffffu,
                          mbar_wait(&bar.k_full[s], kuse[s] & 1, abort_flag, p.err, p.wait_ns) &&
                              mbar_wait_cl(&bar.k_peer[s], kuse[s] & 1, abort_flag, p.err, p.wait_ns) &&
                              (gt < kNP ||
                               mbar_wait_cl(&bar.s_free[sb], ((gt - kNP) / kNP) & 1, abort_flag, p.err, p.wait_ns)));
          if (!ok) break;
          if (lane == 0) mbar_arrive(&bar.go[gt & 1]);
          __syncwarp();
          ++kuse[s];
        }
        tc += un.n_tiles;
        ++ui;
      }
    } else if (warp >= 2 && warp <= 5) {
      // ------------------------------------------------------------ Q issue and move, softmax, P
      const int r = 32 * (warp & 3) + lane;   // query row = tensor-memory lane
      const int wq = warp & 3;
      const uint32_t tq = tm + tmem_lane_base(warp);
      const uint32_t p_dst = map_peer(smem_u32(base + kOOffP), partner);
      const uint32_t pfull_dst = map_peer(smem_u32(&bar.p_full[0]), partner);
      uint8_t* stg = base + kSOffStage;
      const float cl2 = p.scale_log2;
      bool ok = true;
      int tc = 0;
      uint32_t kq[kNK] = {0u, 0u, 0u};   // uses of each K stage by the earlier units (thread 64)
      if (threadIdx.x == 64) prefetch_tmap(&tmap_q);
      for (int k = 0, ui = 0, u = unit_at(0, cluster, n_clusters, p.rows.by_cost); ok && u < p.n_units; u = unit_at(++k, cluster, n_clusters, p.rows.by_cost)) {
        GUnit un;
        if (!global_unit<kPart>(p, u, pr, un)) continue;
        const int pos = kBM * un.t + r;
        const bool row_ok = pos >= un.p_lo && pos <= un.p_hi;
        if (un.n_tiles == 0) {   // kPart: no key of the range: an empty partial
          if (row_ok)
            reinterpret_cast<float2*>(p.ml_part)[(size_t)(un.q_row0 + r) * p.hq + un.h] = make_float2(-INFINITY, 0.f);
          continue;
        }
        // Without q_sep, the unit's Q (8 boxes of 64 dims x 128 rows, rows outside T read as 0) reaches
        // into the first bytes of the P staging: it goes into K stages 1-2 once the earlier units' key
        // tiles there have been read by QK^T and the last P copy has left the staging. Thread 64
        // issues it then: the softmax warps wait every phase of the staging barrier in order, so
        // this wait is one phase ahead at most.
        if (threadIdx.x == 64 && !q_sep) {
          bool okq = true;
          for (int s = 1; okq && s <= 2; ++s)
            if (kq[s] > 0) okq = mbar_wait(&bar.k_empty[s], (kq[s] - 1) & 1, abort_flag, p.err, p.wait_ns);
          if (okq && tc > 0) okq = mbar_wait_cl(&bar.stg_free, (tc - 1) & 1, abort_flag, p.err, p.wait_ns);
          if (okq) {
            mbar_arrive_expect_tx(&bar.q_full, 8 * kQChunk);
#pragma unroll
            for (int c = 0; c < 8; ++c)
              tma_load_3d(q_stage + c * kQChunk, &tmap_q, 64 * c, un.h, un.q_row0, &bar.q_full);
            bar.q_issued = ui + 1;
          }
        }
        for (int j = 0; j < un.n_tiles; ++j) ++kq[j % kNK];
        int row_hi = pos, row_lo = un.k_lo;   // the row sees keys row_lo .. row_hi
        if (kPart) row_hi = min(pos, un.k_hi);
        if (p.rows.span && row_ok) {
          int span_lo;   // 0 on a global layer
          row_keys(p.rows, 0, un.q_row0 + r, pos, un.ctx_end, p.err, span_lo, row_hi);
          if (row_hi > un.k_hi) {   // spans that disagree between rows
            set_error(p.err, kErrSpan);
            row_hi = un.k_hi;
          }
        }
        // The earlier unit's QK^T are all done (its last S was read), so Q may be replaced.
        ok = __all_sync(0xffffffffu, mbar_wait(&bar.q_full, ui & 1, abort_flag, p.err, p.wait_ns));
        if (kRope && ok) {   // thread i rotates pair i % 64 of rows 64 (i / 64) .. + 63
          const int qi = threadIdx.x - 64;
          rotate_q_pair<4, kGlobalR>(q_stage, q_stage + 4 * kQChunk, p.tb, qi & 63, kBM * un.t, 64 * (qi >> 6));
          fence_proxy_async();   // the K copies that later refill this area write through the async proxy
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar.q_rot);
          ok = __all_sync(0xffffffffu, mbar_wait(&bar.q_rot, ui & 1, abort_flag, p.err, p.wait_ns));
        }
        if (!ok) break;
        {   // Q (128B-swizzled boxes in K stages 1-2) -> tensor memory, bf16 pairs
          const uint8_t* qrow = q_stage + r * 128;
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t w[32];
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) {
              const uint4 v = *reinterpret_cast<const uint4*>(qrow + c * kQChunk + ((q8 ^ (r & 7)) * 16));
              w[4 * q8] = v.x;
              w[4 * q8 + 1] = v.y;
              w[4 * q8 + 2] = v.z;
              w[4 * q8 + 3] = v.w;
            }
            tmem_st32(tq + kTmQ + 32 * c, w);   // dims 64c .. 64c+63 -> columns 32c .. 32c+31
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&bar.q_moved);
            arrive_leader(&bar.q_pair);
          }
        }
        float m_used = -INFINITY, l_run = 0.f;
        for (int j = 0; ok && j < un.n_tiles; ++j) {
          const int gt = tc + j, sb = gt % kNP;
          const int kb = (un.kt0 + j) * kTN;
          // Waits are made warp-uniform so that every lane leaves the loop together on an abort.
          if (!__all_sync(0xffffffffu, mbar_wait(&bar.s_full[sb], (gt / kNP) & 1, abort_flag, p.err, p.wait_ns))) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t sr[kTN];
#pragma unroll
          for (int c = 0; c < kTN / 32; ++c)
            tmem_ld32(tq + kTmS + kTN * sb + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_leader(&bar.s_free[sb]);   // buffer sb may take QK^T of tile gt+2

          float s[kTN];
#pragma unroll
          for (int c = 0; c < kTN; ++c) s[c] = __uint_as_float(sr[c]);
          if constexpr (kPart) {   // the row's keys in this tile: one run [lo, hi] of columns
            if (!(row_ok && kb >= row_lo && kb + kTN - 1 <= row_hi)) {
              int lo = row_lo - kb, hi = row_ok ? row_hi - kb : -1;
              if (hi < lo) lo = hi = 1 << 20;   // none
              const unsigned span = (unsigned)(hi - lo);
#pragma unroll
              for (int c = 0; c < kTN; ++c) s[c] = ((unsigned)(c - lo) <= span) ? s[c] : -INFINITY;
            }
          } else if (!(row_ok && kb + kTN - 1 <= row_hi)) {   // causal mask (and rows outside the sequence)
            const int hi = row_ok ? row_hi - kb : -1;
#pragma unroll
            for (int c = 0; c < kTN; ++c) s[c] = (c <= hi) ? s[c] : -INFINITY;
          }
          float mx[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            mx[i] = s[i];
#pragma unroll
            for (int c = 1; c < kTN / 8; ++c) mx[i] = fmaxf(mx[i], s[i + 8 * c]);
          }
          const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * cl2;
          float alpha = 1.f;   // O rescale owed before P_j V_j (1 unless the reference rose by > 2^8)
          if (mt > m_used + kLazyRescale) {
            if (m_used != -INFINITY) alpha = ex2(m_used - mt);
            m_used = mt;
          }
          const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
          uint32_t pw[kTN / 2];
          float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int w = 0; w < kTN / 2; ++w) {
            const float e0 = ex2(fmaf(s[2 * w], cl2, neg_m));
            const float e1 = ex2(fmaf(s[2 * w + 1], cl2, neg_m));
            ls[w & 3] += e0;
            ls[w & 3] += e1;
            pw[w] = pack_bf16(e0, e1);   // declared cast: P in bf16 for P.V
          }
          l_run = fmaf(l_run, alpha, (ls[0] + ls[1]) + (ls[2] + ls[3]));

          // The staging area is free once the previous tile's copies have landed.
          if (gt > 0 &&
              !__all_sync(0xffffffffu, mbar_wait_cl(&bar.stg_free, (gt - 1) & 1, abort_flag, p.err, p.wait_ns))) {
            ok = false;
            break;
          }
          uint8_t* prow = stg + (r >> 3) * kPRowGroup + (r & 7) * 16;
#pragma unroll
          for (int kg = 0; kg < kTN / 8; ++kg)   // keys 8kg .. 8kg+7 of row r: one core-matrix row
            *reinterpret_cast<uint4*>(prow + kg * 128) =
                make_uint4(pw[4 * kg], pw[4 * kg + 1], pw[4 * kg + 2], pw[4 * kg + 3]);
          *reinterpret_cast<uint4*>(prow + 16 * 128) = make_uint4(__float_as_uint(alpha), __float_as_uint(l_run), 0u, 0u);
          fence_proxy_async();   // the bulk copies read what the generic stores wrote
          __syncwarp();
          bool okp = true;
          if (lane == 0) {
            // P slot sb of the output CTA was last read by P.V of tile gt-2
            okp = gt < kNP || mbar_wait_cl(&bar.p_free[sb], ((gt - kNP) / kNP) & 1, abort_flag, p.err, p.wait_ns);
            if (okp)
              bulk_s2peer(p_dst + sb * kPSlot + wq * kPWarpBytes, stg + wq * kPWarpBytes, kPWarpBytes,
                          pfull_dst + sb * 8);
          }
          if (!__shfl_sync(0xffffffffu, okp, 0)) ok = false;
        }
        // kPart: the row's softmax state; O (in the output CTA) is relative to the same running max
        if (kPart && ok && row_ok)
          reinterpret_cast<float2*>(p.ml_part)[(size_t)(un.q_row0 + r) * p.hq + un.h] = make_float2(m_used, l_run);
        tc += un.n_tiles;
        ++ui;
      }
    }
  } else {
    // ================================================================ output CTAs
    const int hv = (int)pr;   // this CTA stages dims 256 hv .. 256 hv + 255 of V
    if (warp == 0) {
      // ------------------------------------------------------------ V copies
      const __nv_bfloat16* sc = (const __nv_bfloat16*)p.k_cache;
      bool ok = true;
      for (int k = 0, u = unit_at(0, cluster, n_clusters, p.rows.by_cost); ok && u < p.n_units; u = unit_at(++k, cluster, n_clusters, p.rows.by_cost)) {
        GUnit un;
        if (!global_unit<kPart>(p, u, pr, un) || un.n_tiles == 0) continue;
        // Block indices ahead of use: lane l holds page (l & 3) of stage (l >> 2) of the current
        // group of 8 stages; the next group is looked up one group early.
        const int n_st = 2 * un.n_tiles;
        auto load_blocks = [&](int c0) -> int {
          const int cs2 = c0 + (lane >> 2);
          if (cs2 >= n_st) return -1;
          return page_block(un.kt0 * kTN + cs2 * kVN + kPage * (lane & 3), un.k_lo, un.k_hi, un.pt, p.num_pages,
                            p.hkv, un.g, p.err);
        };
        int blk_cur = load_blocks(0), blk_next = load_blocks(8);
        for (int c = 0; c < n_st; ++c) {
          const uint32_t vc = vc_total;
          const int s = vc % kNV;
          if (c > 0 && (c & 7) == 0) {
            blk_cur = blk_next;
            blk_next = load_blocks(c + 8);
          }
          const int bl0 = __shfl_sync(0xffffffffu, blk_cur, (c & 7) * 4 + (lane & 3));
          const int bl = lane < 4 ? bl0 : -1;
          const unsigned live = __ballot_sync(0xffffffffu, bl >= 0);
          bool okw = true;
          if (lane == 0 && vc >= (uint32_t)kNV)
            okw = mbar_wait(&bar.v_empty[s], ((vc / kNV) - 1) & 1, abort_flag, p.err, p.wait_ns);
          if (!__shfl_sync(0xffffffffu, okw, 0)) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(&bar.v_full[s], __popc(live) * kVPageBytes);
          __syncwarp();
          if (bl >= 0)
            bulk_g2s(base + s * kVStage + lane * kVPageBytes, sc + (size_t)bl * (kPage * kGD) + hv * (kPage * kHalf),
                     kVPageBytes, &bar.v_full[s]);
          __syncwarp();
          ++vc_total;
        }
      }
    } else if ((warp == 1 && !leader) || (warp == 7 && leader)) {
      // ------------------------------------------------------------ V check; P.V helper (rank 2) or relay (rank 3)
      // Value rows of keys that hold no data of this sequence are zeroed before P.V: pages past
      // the last needed one were not copied and keep an older tile, and slots past the
      // sequence's last key may hold anything (NaN); P = 0 there does not cancel NaN.
      bool ok = true;
      uint32_t vc = 0;
      int tc = 0;
      for (int k = 0, ui = 0, u = unit_at(0, cluster, n_clusters, p.rows.by_cost); ok && u < p.n_units; u = unit_at(++k, cluster, n_clusters, p.rows.by_cost)) {
        GUnit un;
        if (!global_unit<kPart>(p, u, pr, un) || un.n_tiles == 0) continue;
        const int n_st = 2 * un.n_tiles;
        for (int c = 0; ok && c < n_st; ++c, ++vc) {
          const int s = vc % kNV, j = c >> 1, e = c & 1, gt = tc + j;
          ok = __all_sync(0xffffffffu, mbar_wait(&bar.v_full[s], (vc / kNV) & 1, abort_flag, p.err, p.wait_ns));
          if (!ok) break;
          const int kb = un.kt0 * kTN + c * kVN;
          // kPart: a rank's cache may hold another rank's keys, or nothing, around its range
          const int v0 = kPart ? un.k_lo : 0;
          const int v1 = kPart ? min(kb + kVN, un.k_hi + 1)
                               : min(min(kb + kVN, ((un.k_hi >> 4) + 1) * kPage), un.ctx_end);
          if (v0 > kb || v1 < kb + kVN) {
            uint8_t* vt = base + s * kVStage;
            for (int idx = lane; idx < kVN * 32; idx += 32) {
              const int rr = idx >> 5, dg = idx & 31;
              if (kb + rr < v0 || kb + rr >= v1)
                *reinterpret_cast<uint4*>(vt + (rr >> 3) * kVKG + dg * 128 + (rr & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async();
          }
          __syncwarp();
          if (!leader) {
            if (lane == 0) mbar_arrive_remote(map_peer(smem_u32(&bar.v_ready[s]), pair_peer));
            __syncwarp();
            continue;
          }
          // rank 3's half is ready; at a tile's first half, both CTAs have P_j and have applied
          // alpha; at a unit's first step, both have read the earlier unit's O out
          ok = __all_sync(0xffffffffu,
                          mbar_wait_cl(&bar.v_ready[s], (vc / kNV) & 1, abort_flag, p.err, p.wait_ns) &&
                              (e == 1 ||
                               mbar_wait_cl(&bar.o_ready[gt % kNP], (gt / kNP) & 1, abort_flag, p.err, p.wait_ns)) &&
                              (c > 0 || ui == 0 || mbar_wait_cl(&bar.o_free, (ui - 1) & 1, abort_flag, p.err, p.wait_ns)));
          if (!ok) break;
          if (lane == 0) mbar_arrive(&bar.go_pv[s]);
          __syncwarp();
        }
        tc += un.n_tiles;
        ++ui;
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ P.V issuer (rank 2)
      bool ok = true;
      uint32_t vc = 0;
      int tc = 0;
      for (int k = 0, u = unit_at(0, cluster, n_clusters, p.rows.by_cost); ok && u < p.n_units; u = unit_at(++k, cluster, n_clusters, p.rows.by_cost)) {
        GUnit un;
        if (!global_unit<kPart>(p, u, pr, un) || un.n_tiles == 0) continue;
        const int n_st = 2 * un.n_tiles;
        for (int c = 0; ok && c < n_st; ++c, ++vc) {
          const int s = vc % kNV, j = c >> 1, e = c & 1, gt = tc + j;
          ok = __all_sync(0xffffffffu, mbar_wait(&bar.go_pv[s], (vc / kNV) & 1, abort_flag, p.err, p.wait_ns));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t va = smem_u32(base + s * kVStage);
            const uint32_t pa = smem_u32(base + kOOffP + (gt % kNP) * kPSlot);
#pragma unroll
            for (int k = 0; k < kVN / 16; ++k) {   // 16 keys (two key groups) per step
              const uint32_t acc = (j > 0 || e > 0 || k > 0) ? 1u : 0u;
              const uint64_t ad = desc_tiled(pa + (4 * e + k) * 256, 128, kPRowGroup);
              mma2_ss(tm + kTmO, ad, desc_tiled(va + k * 2 * kVKG, kVKG, 128), kIdescPV, acc);
              mma2_ss(tm + kTmO + 256, ad, desc_tiled(va + k * 2 * kVKG + 2048, kVKG, 128), kIdescPV, acc);
            }
            mma2_commit_mc(&bar.v_empty[s], kOutPair);
            if (e == 1) mma2_commit_mc(&bar.pv_done[gt % kNP], kOutPair);
          }
          __syncwarp();
        }
        tc += un.n_tiles;
      }
    } else if (warp >= 2 && warp <= 5) {
      // ------------------------------------------------------------ alpha, O rescale, epilogue
      const int r = 32 * (warp & 3) + lane;
      const uint32_t tq = tm + tmem_lane_base(warp);
      const uint32_t stg_free_dst = map_peer(smem_u32(&bar.stg_free), partner);
      bool ok = true;
      int tc = 0;
      for (int k = 0, u = unit_at(0, cluster, n_clusters, p.rows.by_cost); ok && u < p.n_units; u = unit_at(++k, cluster, n_clusters, p.rows.by_cost)) {
        GUnit un;
        if (!global_unit<kPart>(p, u, pr, un)) continue;
        const int pos = kBM * un.t + r;
        const bool row_ok = pos >= un.p_lo && pos <= un.p_hi;
        if (un.n_tiles == 0) {   // kPart: no key of the range: an empty partial
          if (row_ok) {
            float4* dst = reinterpret_cast<float4*>(p.o_part + ((size_t)(un.q_row0 + r) * p.hq + un.h) * kGD);
            for (int i = 0; i < kGD / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
          continue;
        }
        float l_last = 0.f;
        for (int j = 0; j < un.n_tiles; ++j) {
          const int gt = tc + j, sb = gt % kNP;
          if (!__all_sync(0xffffffffu, mbar_wait_cl(&bar.p_full[sb], (gt / kNP) & 1, abort_flag, p.err, p.wait_ns))) {
            ok = false;
            break;
          }
          const float2 ax = *reinterpret_cast<const float2*>(base + kOOffP + sb * kPSlot + (r >> 3) * kPRowGroup +
                                                            16 * 128 + (r & 7) * 16);
          if (threadIdx.x == 64) {
            bar.p_seen[sb] = gt / kNP + 1;
            mbar_arrive_remote(stg_free_dst);   // the score CTA may refill its staging
          }
          l_last = ax.y;
          const bool need = j > 0 && ax.x != 1.f;
          if (__any_sync(0xffffffffu, need)) {   // O correction, after P_{j-1} V_{j-1} has landed
            const int gp = gt - 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&bar.pv_done[gp % kNP], (gp / kNP) & 1, abort_flag, p.err,
                                                   p.wait_ns))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const float a = need ? ax.x : 1.f;
#pragma unroll 1
            for (int cc = 0; cc < kGD / 32; ++cc) {
              uint32_t o[32];
              tmem_ld32(tq + kTmO + 32 * cc, o);
              tmem_ld_wait();
#pragma unroll
              for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * a);
              tmem_st32(tq + kTmO + 32 * cc, o);
            }
            tmem_st_wait();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_leader(&bar.o_ready[sb]);
        }
        if (!ok) break;
        // Epilogue: O / l -> bf16 rows of this sequence only, row-contiguous stores (kPart: the
        // un-normalised fp32 rows). Once O is in registers, the next unit's first P.V (which
        // overwrites it) may start.
        const int gl = tc + un.n_tiles - 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&bar.pv_done[gl % kNP], (gl / kNP) & 1, abort_flag, p.err, p.wait_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float inv = (l_last > 0.f) ? __frcp_rn(l_last) : 0.f;
        const unsigned valid = __ballot_sync(0xffffffffu, row_ok);
        const long long wrow0 = (long long)un.q_row0 + 32 * (warp & 3);
        float* prow = kPart ? p.o_part + ((size_t)(un.q_row0 + r) * p.hq + un.h) * kGD : nullptr;
        tmem_ld_stream64<kGD / 64>(
            tq + kTmO,
            [&]() {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) arrive_leader(&bar.o_free);
            },
            [&](int c, const uint32_t(&o)[64]) {
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                const int d0 = o_dim(64 * c + 32 * half);   // 32 consecutive dims
                if constexpr (kPart) {
                  if (row_ok) {
                    float4* dst = reinterpret_cast<float4*>(prow + d0);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                      dst[i] = make_float4(__uint_as_float(o[32 * half + 4 * i]), __uint_as_float(o[32 * half + 4 * i + 1]),
                                           __uint_as_float(o[32 * half + 4 * i + 2]),
                                           __uint_as_float(o[32 * half + 4 * i + 3]));
                  }
                } else {
                  uint32_t w16[16];
#pragma unroll
                  for (int k = 0; k < 16; ++k)
                    w16[k] = pack_bf16(__uint_as_float(o[32 * half + 2 * k]) * inv,
                                       __uint_as_float(o[32 * half + 2 * k + 1]) * inv);
                  store_rows32<kGD>(w16, p.out, wrow0, p.hq, un.h, d0, valid, lane);
                }
              }
            });
        tc += un.n_tiles;
      }
    } else if (warp == 6) {
      // ------------------------------------------------------------ P slot hand-back
      // Once P.V of tile gt has completed, its P slot takes tile gt+2 (of this unit or a later
      // one): post the bytes that tile's copies will deliver, then tell the score CTA (posting
      // first keeps the count ahead).
      if (lane == 0) {
        const uint32_t pfree_dst = map_peer(smem_u32(&bar.p_free[0]), partner);
        for (int gt = 0; gt < total_tiles; ++gt) {
          if (!mbar_wait(&bar.pv_done[gt % kNP], (gt / kNP) & 1, abort_flag, p.err, p.wait_ns)) break;
          if (gt + kNP < total_tiles) {
            mbar_arrive_expect_tx(&bar.p_full[gt % kNP], kPSendBytes);
            mbar_arrive_remote(pfree_dst + (gt % kNP) * 8);
          }
        }
      }
      __syncwarp();
    }
  }

  // ------------------------------------------------------------ teardown
  // No CTA may free its tensor memory or leave while MMAs, copies or signals into it are in
  // flight. On an abort the flag is passed to the other three CTAs (their waits then end
  // early), copies this CTA issued are drained (bounded), and a cluster barrier closes the cluster.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (!*abort_flag && threadIdx.x == 0) {   // the last stage releases (MMA commits) have arrived
    const unsigned long long w0 = globaltimer();
    if (is_out) {
      for (uint32_t s = 0; s < (uint32_t)kNV && s < vc_total; ++s) {
        const uint32_t last = s + kNV * ((vc_total - 1 - s) / kNV);
        while (!mbar_try_wait(smem_u32(&bar.v_empty[s]), (last / kNV) & 1) && globaltimer() - w0 < kWaitLimitNs) {
        }
      }
    } else {
      for (int s = 0; s < kNK; ++s)
        if (kuse[s] > 0)
          while (!mbar_try_wait(smem_u32(&bar.k_empty[s]), (kuse[s] - 1) & 1) && globaltimer() - w0 < kWaitLimitNs) {
          }
    }
  }
  if (*abort_flag) {
    if (threadIdx.x == 0) {
      for (uint32_t q = 0; q < 4; ++q)
        if (q != rank) st_peer_u32(map_peer(smem_u32(&bar.abort_flag), q), 1u);
    }
    if (threadIdx.x == 0) {   // copies into this CTA's shared memory that may still be in flight
      const unsigned long long w0 = globaltimer();
      auto drain = [&](uint64_t* br, uint32_t par) {
        while (!mbar_try_wait_cluster(smem_u32(br), par) && globaltimer() - w0 < kWaitLimitNs) {
        }
      };
      if (!is_out) {
        if (bar.q_issued > 0) drain(&bar.q_full, (bar.q_issued - 1) & 1);
        for (int s = 0; s < kNK; ++s)
          if (kuse[s] > 0) drain(&bar.k_full[s], (kuse[s] - 1) & 1);
      } else {
        for (uint32_t i = vc_total > (uint32_t)kNV ? vc_total - kNV : 0; i < vc_total; ++i)
          drain(&bar.v_full[i % kNV], (i / kNV) & 1);
        for (int s = 0; s < kNP; ++s) drain(&bar.p_full[s], bar.p_seen[s] & 1);
      }
    }
  }
  __syncthreads();
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if (bar.abort_flag) {   // let every MMA the pair issued finish before the columns are freed
      if (leader && lane == 0) mma2_commit_mc(&bar.teardown, is_out ? kOutPair : kScorePair);
      __syncwarp();
      const unsigned long long w0 = globaltimer();
      while (!mbar_try_wait(smem_u32(&bar.teardown), 0) && globaltimer() - w0 < kWaitLimitNs) {
      }
    }
    tmem_dealloc2(tm, 512);
  }
}

// Tensor maps over the global cache's page-head blocks, as 5-D tensors (innermost first):
// 64 elements of a core matrix, dim group, dim half, key group, block (page * 4 + KV head). The
// dim half comes before the key group although its stride is larger, so that a box lands with the
// key group outermost (see the K stage layout). S: 32 dim groups per half, box from dim group 8;
// k_rot: 8 dim groups per half.
bool page_maps(CUtensorMap* ms, CUtensorMap* mr, const void* s_cache, const void* rot_cache, int num_pages, int hkv) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t blocks = (cuuint64_t)num_pages * hkv;
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  {
    const cuuint64_t dims[5] = {64, 32, 2, 2, blocks};
    const cuuint64_t strides[4] = {128, 2 * 32 * 128, 32 * 128, (cuuint64_t)kPage * kGD * 2};
    const cuuint32_t box[5] = {64, 24, 2, 2, 1};
    if (fn(ms, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(s_cache), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  {
    const cuuint64_t dims[5] = {64, 8, 2, 2, blocks};
    const cuuint64_t strides[4] = {128, 2 * 8 * 128, 8 * 128, (cuuint64_t)kRotPageElems * 2};
    const cuuint32_t box[5] = {64, 8, 2, 2, 1};
    if (fn(mr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(rot_cache), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

// ---------------------------------------------------------------- merge of partials (context parallelism)
// One CTA per query row: thread i merges dims 4i .. 4i+3 of every head of the row, over the parts in
// the order given. A row no sequence owns is not written.
__global__ void __launch_bounds__(kGD / 4) merge_partials_kernel(PartialSet parts, SeqRows rows, int hq,
                                                                 __nv_bfloat16* out) {
  const int r = blockIdx.x;
  __shared__ int owned;
  if (threadIdx.x < 32) {
    bool mine = false;
    for (int b0 = 0; b0 < rows.B && !mine; b0 += 32) {
      const int b = b0 + (int)threadIdx.x;
      if (b < rows.B) {
        const int s0 = rows.q_start[b], L = rows.q_len[b];
        mine = L > 0 && r >= s0 && r - s0 < L;
      }
      mine = __any_sync(0xffffffffu, mine);
    }
    if (threadIdx.x == 0) owned = mine ? 1 : 0;
  }
  __syncthreads();
  if (!owned) return;
  const int d0 = 4 * threadIdx.x;
  for (int h = 0; h < hq; ++h) {
    const size_t v = (size_t)r * hq + h;
    float M = -INFINITY;
    for (int i = 0; i < parts.n; ++i) M = fmaxf(M, parts.ml[i][2 * v]);
    float L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (M != -INFINITY) {
      for (int i = 0; i < parts.n; ++i) {
        const float mi = parts.ml[i][2 * v];
        if (mi == -INFINITY) continue;   // a part with no key for this row
        const float w = exp2f(mi - M);
        L = fmaf(parts.ml[i][2 * v + 1], w, L);
        const float4 o = *reinterpret_cast<const float4*>(parts.o[i] + v * kGD + d0);
        acc[0] = fmaf(o.x, w, acc[0]);
        acc[1] = fmaf(o.y, w, acc[1]);
        acc[2] = fmaf(o.z, w, acc[2]);
        acc[3] = fmaf(o.w, w, acc[3]);
      }
    }
    const float inv = (L > 0.f) ? __frcp_rn(L) : 0.f;
    uint2 pk;
    pk.x = pack_bf16(acc[0] * inv, acc[1] * inv);
    pk.y = pack_bf16(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(out + v * kGD + d0) = pk;
  }
}

}  // namespace

cudaError_t launch_merge_partials(const PartialSet& parts, const SeqRows& rows, int hq, void* out, const DeviceState& st,
                                  cudaStream_t s) {
  (void)st;
  if (rows.T <= 0) return cudaSuccess;
  merge_partials_kernel<<<(unsigned)rows.T, kGD / 4, 0, s>>>(parts, rows, hq, (__nv_bfloat16*)out);
  return cudaGetLastError();
}

cudaError_t launch_prefill_global(const SeqRows& rows, float scale_log2, const PagedCache& cache, void* out,
                                  const DeviceState& st, cudaStream_t s, const void* q_raw, const PartialOut* part) {
  PrefillParams p{};
  p.rows = rows;
  p.window = 0;
  p.scale_log2 = scale_log2;
  p.k_cache = cache.k;
  p.v_cache = nullptr;
  p.krot_cache = cache.krot;
  p.num_pages = cache.num_pages;
  p.page_table = cache.page_table;
  p.max_pages = cache.max_pages;
  p.out = (__nv_bfloat16*)out;
  p.tb = st.global;
  p.err = st.err;
  p.hq = cache.hq;
  p.hkv = cache.hkv;
  p.wait_ns = wait_limit_ns();
  if (part) {
    p.key_begin = part->key_begin;
    p.key_end = part->key_end;
    p.o_part = part->o;
    p.ml_part = part->ml;
  }
  // Raw queries are rotated in the kernel; otherwise the staged roped queries are read from `out`.
  // Partial calls take raw queries and no image spans.
  if (rows.span && q_raw) return cudaErrorInvalidValue;
  if (part && (!q_raw || rows.span)) return cudaErrorInvalidValue;
  CUtensorMap mq, ms, mr;   // queries (raw or staged), the cache's S and k_rot pages
  if (!q_map(&mq, q_raw ? q_raw : out, rows.T, cache.hq, kGD)) return cudaErrorInvalidValue;
  if (!page_maps(&ms, &mr, cache.k, cache.krot, cache.num_pages, cache.hkv)) return cudaErrorInvalidValue;
  auto kernel = part ? prefill_global_kernel<true, true>
                     : (q_raw ? prefill_global_kernel<true, false> : prefill_global_kernel<false, false>);
  const int ki = part ? 2 : (q_raw ? 1 : 0);
  static bool attr[64][3] = {};
  static int max_clusters[64][3] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr[dev][ki]) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGlobalSmemBytes);
    if (e != cudaSuccess) return e;
    // clusters that fit on the device at once: the persistent grid
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(4, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kGlobalSmemBytes;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeClusterDimension;
    la[0].val.clusterDim.x = 4;
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
  const long long n_units = slots * (cache.hq / 2);   // (query tile, head pair) units
  if (n_units <= 0 || n_units > 0x3fffffffLL) return cudaErrorInvalidValue;
  p.n_units = (int)n_units;
  const int n_clusters = (int)(n_units < max_clusters[dev][ki] ? n_units : max_clusters[dev][ki]);
  kernel<<<4u * (unsigned)n_clusters, kThreads, kGlobalSmemBytes, s>>>(mq, ms, mr, p);
  return cudaGetLastError();
}

}  // namespace g4
