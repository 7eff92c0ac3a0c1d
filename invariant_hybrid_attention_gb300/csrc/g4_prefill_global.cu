// Global-layer prefill on tcgen05: full causal attention, 32 Q / 4 KV heads, head dim 512,
// K==V (RL-Kernel RFC "[RFC][Gemma-4-31B-it] WS1/WS2 kernel roadmap", section 5,
// global_attention_core and global_k_eq_v_projection; section 2: proportional p-RoPE, partial
// factor 0.25, theta 1e6).
//
// A 128 x 512 fp32 output tile fills all of one SM's tensor memory, so each (query tile, head)
// runs on a cluster of two CTAs, each owning half of the head dims (rank r: dims 256r ..
// 256r+255):
//   - S_r = Q[:, half r] . K[:, half r]^T on the CTA's tensor cores; the two partial score
//     tiles are exchanged through distributed shared memory in 32-key halves (each warp stages
//     its 32 rows of a half and one bulk copy carries them to the peer), one half ahead of the
//     softmax, and both CTAs add them (IEEE addition commutes, so both hold the same S bits)
//     and run the same softmax;
//   - O[:, half r] += P . V[:, half r], V being the CTA's half of the un-rotated S tile: one
//     copy of each stored half-page serves V and the un-rotated 3/4 of K;
//   - the rotated quarter of K comes from the cache's k_rot side pages (p-RoPE(S), written
//     with S by the append pass), so no CTA re-rotates key tiles.
// Key tiles of 64 keys are aligned to absolute key 0 and visited in ascending order, query
// tiles are aligned to absolute position (section 4 rules 2, 3 and 6).
//
// Per CTA: warp 0 copies (roped Q tile by TMA; per key tile one 8 KB S half-page and one 2 KB
// rotated half-page per page, 4-stage ring), warp 1 issues the MMAs, warps 2-5 run the
// exchange, mask, online softmax, P (bf16, into tensor memory) and the epilogue.
// Tensor memory: O half [0,256), Q dims 0-127 of the half [256,320), three S/P buffers [320,512).
#include <math.h>

#include "g4_prefill_common.cuh"

namespace g4 {

namespace {

using namespace pf;

constexpr int kGD = kGlobalD;                          // 512
constexpr int kHalf = kGD / 2;                         // dims per CTA
constexpr int kNS = 4;                                 // key-tile ring stages
constexpr int kXCols = kBN / 2;                        // partial scores cross the pair in 32-key halves
constexpr int kNSP = 3;                                // S/P buffers
constexpr int kHalfPageBytes = kPage * kHalf * 2;      // 8 KB
constexpr int kRotHalfPageBytes = kPage * kGlobalR * 2;   // 2 KB
constexpr int kKG = 8 * kHalf * 2;                     // S half tile: bytes per key group (4 KB)
constexpr int kRotKG = 8 * kGlobalR * 2;               // rotated tile: bytes per key group (1 KB)
constexpr int kSTile = (kBN / kPage) * kHalfPageBytes;       // 32 KB
constexpr int kRotTile = (kBN / kPage) * kRotHalfPageBytes;  // 8 KB
constexpr int kStage = kSTile + kRotTile;              // 40 KB
constexpr int kThreads = 64 + kSoftmaxThreads;
constexpr uint32_t kTmO = 0, kTmQ = 256, kTmS = 320;
constexpr uint32_t kIdescQK = idesc_bf16(kBM, kBN, false, false);
constexpr uint32_t kIdescPV = idesc_bf16(kBM, kHalf, false, true);

struct GlobalSmem {
  uint8_t st[kNS][kStage];          // S half tile (V; K outside the rotated columns), rotated tile;
                                    // st[2] first holds Q dims 0-127 of the half
  uint8_t qhi[2 * kQChunk];         // Q dims 128-255 of the half (128B swizzle): an A operand
  float xbuf[2][kBM][kXCols];       // partial scores by 32-key half h: the peer's half h lands in
                                    // xbuf[h & 1]; this CTA's own half h is staged in xbuf[(h + 1) & 1]
  uint64_t full[kNS], empty[kNS];
  uint64_t s_full[kNSP], p_full[kNSP], pv_done[kNSP];
  uint64_t xfull[2];
  uint64_t q_full, q_ready, peer_done, teardown;
  uint32_t tmem_base;
  int abort_flag;
  int unit_b, unit_t;
};
static_assert(2 * kQChunk <= kStage, "Q dims 0-127 must fit in one ring stage");
constexpr size_t kGlobalSmemBytes = sizeof(GlobalSmem) + 1024;
static_assert(kGlobalSmemBytes <= 232448, "global prefill exceeds the 227 KB shared-memory limit");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_global_kernel(const __grid_constant__ CUtensorMap tmap_q, PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  GlobalSmem& sm = *reinterpret_cast<GlobalSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();   // which half of the head dims
  const uint32_t peer = rank ^ 1u;
  const int unit = blockIdx.x >> 1;
  const int h = unit % kGlobalHq;
  const int slot = unit / kGlobalHq;
  const int g = h / (kGlobalHq / kGlobalHkv);

  if (warp == 0) {
    int ub, ut;
    find_unit(p.rows, slot, ub, ut);
    if (lane == 0) {
      sm.unit_b = ub;
      sm.unit_t = ut;
    }
  }
  __syncthreads();
  const int b = sm.unit_b;   // both CTAs of the pair find the same unit
  if (b < 0) return;
  const int t = sm.unit_t;
  const int cs = p.rows.ctx_start[b], L = p.rows.q_len[b], qs = p.rows.q_start[b];
  const int p_lo = max(kBM * t, cs), p_hi = min(kBM * t + kBM - 1, cs + L - 1);
  const int ctx_end = cs + L;
  if (p_hi >= kMaxPos || (p_hi >> 4) >= p.max_pages) {
    if (threadIdx.x == 0 && h == 0 && rank == 0) set_error(p.err, kErrPos);
    return;
  }
  const int k_lo = 0, k_hi = p_hi;
  const int n_tiles = k_hi / kBN + 1;
  const int q_row0 = qs + (kBM * t - cs);
  const int32_t* pt = p.page_table + (size_t)b * p.max_pages;

  if (threadIdx.x == 32) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int s = 0; s < kNSP; ++s) {
      mbar_init(&sm.s_full[s], 1);
      mbar_init(&sm.p_full[s], kSoftmaxThreads);
      mbar_init(&sm.pv_done[s], 1);
    }
    for (int s = 0; s < 2; ++s) mbar_init(&sm.xfull[s], 1);   // one local arrive with the expected bytes
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_ready, kSoftmaxThreads);
    mbar_init(&sm.peer_done, 1);
    mbar_init(&sm.teardown, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync_all();   // the peer's barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tm = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ copy producer
    auto load_blocks = [&](int j0) -> int {
      const int jt = j0 + (lane >> 2);
      if (jt >= n_tiles) return -1;
      return page_block(jt * kBN + (lane & 3) * kPage, k_lo, k_hi, pt, p.num_pages, kGlobalHkv, g, p.err);
    };
    if (lane == 0) {   // roped Q dims 256r .. 256r+255: chunks 0-1 into stage 2, chunks 2-3 stay
      prefetch_tmap(&tmap_q);
      mbar_arrive_expect_tx(&sm.q_full, 4 * kQChunk);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tma_load_3d((c < 2 ? sm.st[2] + c * kQChunk : sm.qhi + (c - 2) * kQChunk), &tmap_q, kHalf * rank + 64 * c,
                    h, q_row0, &sm.q_full);
    }
    int blk_cur = load_blocks(0), blk_next = load_blocks(8);
    const __nv_bfloat16* sc = (const __nv_bfloat16*)p.k_cache;
    const __nv_bfloat16* rc = (const __nv_bfloat16*)p.krot_cache;
    int j = 0;
    for (; j < n_tiles; ++j) {
      const int s = j % kNS;
      if (j > 0 && (j & 7) == 0) {
        blk_cur = blk_next;
        blk_next = load_blocks(j + 8);
      }
      const int my_blk = __shfl_sync(0xffffffffu, blk_cur, (j & 7) * 4 + (lane & 3));
      const unsigned live = __ballot_sync(0xffffffffu, lane < 4 && my_blk >= 0);
      const uint32_t bytes = __popc(live) * (kHalfPageBytes + kRotHalfPageBytes);
      bool ok = (j < kNS) || lane != 0 || mbar_wait(&sm.empty[s], ((j / kNS) - 1) & 1, abort_flag, p.err);
      if (j == 2 && lane == 0) ok = ok && mbar_wait(&sm.q_ready, 0, abort_flag, p.err);   // Q left stage 2
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (lane == 0) mbar_arrive_expect_tx(&sm.full[s], bytes);
      __syncwarp();
      if (lane < 4 && my_blk >= 0) {
        bulk_g2s(sm.st[s] + lane * kHalfPageBytes, sc + (size_t)my_blk * kPage * kGD + rank * (kPage * kHalf),
                 kHalfPageBytes, &sm.full[s]);
        bulk_g2s(sm.st[s] + kSTile + lane * kRotHalfPageBytes,
                 rc + (size_t)my_blk * kRotPageElems + rank * (kPage * kGlobalR), kRotHalfPageBytes, &sm.full[s]);
      }
    }
    if (lane == 0 && *abort_flag) {   // drain copies still in flight (bounded) before the CTA may exit
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(smem_u32(&sm.q_full), 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
      for (int i = max(0, j - kNS); i < j; ++i) {
        while (!mbar_try_wait(smem_u32(&sm.full[i % kNS]), (i / kNS) & 1) && globaltimer() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    auto pv = [&](int i) -> bool {
      if (!mbar_wait(&sm.p_full[i % kNSP], (i / kNSP) & 1, abort_flag, p.err)) return false;
      const int kb = i * kBN;
      uint8_t* vt = sm.st[i % kNS];
      // V rows of keys that hold no data of this sequence are zeroed before P.V (pages past the
      // last needed one keep an older tile, slots past the last key may hold NaN). QK^T of this
      // tile has completed (the softmax read its S before arriving on p_full).
      const int v1 = min(min(kb + kBN, ((k_hi >> 4) + 1) * kPage), ctx_end);
      if (v1 < kb + kBN) {
        for (int idx = lane; idx < kBN * (kHalf / 8); idx += 32) {
          const int r = idx / (kHalf / 8), dg = idx % (kHalf / 8);
          if (kb + r >= v1)
            *reinterpret_cast<uint4*>(vt + (r >> 3) * kKG + dg * 128 + (r & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
        __syncwarp();
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t va = smem_u32(vt);
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k)   // V = the S half tile, MN-major: 16 keys (2 key groups) per step
          mma_ts(tm + kTmO, tm + kTmS + 64 * (i % kNSP) + 8 * k, desc_tiled(va + k * 2 * kKG, kKG, 128), kIdescPV,
                 (i > 0 || k > 0) ? 1u : 0u);
        mma_commit(&sm.pv_done[i % kNSP]);
        mma_commit(&sm.empty[i % kNS]);
      }
      __syncwarp();
      return true;
    };
    // QK^T runs two tiles ahead of P.V: the softmax sends tile j+1's partial scores while it
    // works on tile j, so S_{j+1} must be ready when tile j's softmax starts.
    auto qk = [&](int j) -> bool {
      const int s = j % kNS;
      if (!mbar_wait(&sm.full[s], (j / kNS) & 1, abort_flag, p.err)) return false;
      // S buffer j % 3 last held P_{j-3}: reuse it once P_{j-3} V_{j-3} has completed.
      if (j >= kNSP && !mbar_wait(&sm.pv_done[j % kNSP], ((j - kNSP) / kNSP) & 1, abort_flag, p.err)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t sa = smem_u32(sm.st[s]);
        const uint32_t ra = sa + kSTile;
        const uint32_t qh = smem_u32(sm.qhi);
        const uint32_t sd = tm + kTmS + 64 * (j % kNSP);
#pragma unroll
        for (int k = 0; k < 4; ++k)    // dims 0-63 of the half (the rotated ones): K from k_rot
          mma_ts(sd, tm + kTmQ + 8 * k, desc_tiled(ra + k * 256, 128, kRotKG), kIdescQK, k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 4; k < 8; ++k)    // dims 64-127: K = S
          mma_ts(sd, tm + kTmQ + 8 * k, desc_tiled(sa + k * 256, 128, kKG), kIdescQK, 1u);
#pragma unroll
        for (int k = 8; k < 16; ++k)   // dims 128-255: Q from shared memory, K = S
          mma_ss(sd, desc_sw128(qh + ((k - 8) >> 2) * kQChunk + (k & 3) * 32, 16, 1024),
                 desc_tiled(sa + k * 256, 128, kKG), kIdescQK, 1u);
        mma_commit(&sm.s_full[j % kNSP]);
      }
      __syncwarp();
      return true;
    };
    bool ok = mbar_wait(&sm.q_ready, 0, abort_flag, p.err);
    for (int j = 0; ok && j < 2 && j < n_tiles; ++j) ok = qk(j);
    for (int i = 0; ok && i < n_tiles; ++i) {
      if (!pv(i) || (i + 2 < n_tiles && !qk(i + 2))) ok = false;
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue warps
    const int r = 32 * (warp & 3) + lane;   // query row = tensor-memory lane
    const uint32_t tq = tm + tmem_lane_base(warp);
    const int pos = kBM * t + r;
    const bool row_ok = pos >= p_lo && pos <= p_hi;
    const uint32_t rsw = (uint32_t)(r & 7);   // 16-byte chunk swizzle of the exchange rows

    {   // Q dims 0-127 of the half: ring stage 2 -> tensor memory (bf16 pairs)
      const bool okq = mbar_wait(&sm.q_full, 0, abort_flag, p.err);
      const uint8_t* qrow = sm.st[2] + r * 128;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          const uint4 v = okq ? *reinterpret_cast<const uint4*>(qrow + c * kQChunk + ((q8 ^ (r & 7)) * 16))
                              : make_uint4(0, 0, 0, 0);
          w[4 * q8] = v.x;
          w[4 * q8 + 1] = v.y;
          w[4 * q8 + 2] = v.z;
          w[4 * q8 + 3] = v.w;
        }
        tmem_st32(tq + kTmQ + 32 * c, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sm.q_ready);
    }

    constexpr uint32_t kXBytes = kBM * kXCols * 4;      // one 32-key half of a partial score tile
    constexpr uint32_t kXWarpBytes = 32 * kXCols * 4;   // the 32 rows of one warp
    const uint32_t xrows = (uint32_t)(warp & 3) * kXWarpBytes;
    const uint32_t peer_xbuf = map_peer(smem_u32(&sm.xbuf[0][0][0]), peer) + xrows;
    const uint32_t peer_xfull = map_peer(smem_u32(&sm.xfull[0]), peer);
    const int n_halves = 2 * n_tiles;
    if (threadIdx.x == 64) {   // expect the peer's first two halves
      mbar_arrive_expect_tx(&sm.xfull[0], kXBytes);
      mbar_arrive_expect_tx(&sm.xfull[1], kXBytes);
    }
    // Exchange of partial scores in 32-key halves h = 2j + e (tile j, columns 32e..32e+31), one
    // half ahead of the softmax. The peer's half h lands in xbuf[h & 1]; this CTA's own half h is
    // staged in xbuf[(h + 1) & 1] and sent from there. Step h: wait for the peer's half h, read
    // this warp's rows of it into registers, stage and send own half h+1 from the buffer just
    // read, then run half h's softmax while that copy is in flight. Reuse is safe without a
    // separate free signal: the peer sends its half h+2 into xbuf[h & 1] only after it has
    // received all of this CTA's half h+1, whose copy read that buffer, and this CTA read the
    // peer's half h from it before staging.
    auto send_half = [&](int hh) -> bool {   // stage own half hh and copy it into the peer
      const int jt = hh >> 1, eh = hh & 1;
      if (eh == 0 &&
          !__all_sync(0xffffffffu, mbar_wait(&sm.s_full[jt % kNSP], (jt / kNSP) & 1, abort_flag, p.err)))
        return false;
      tc_fence_after();
      uint32_t sr[32];
      tmem_ld32(tq + kTmS + 64 * (jt % kNSP) + kXCols * eh, sr);
      tmem_ld_wait();
      const int sp = (hh + 1) & 1;
      float4* stg = reinterpret_cast<float4*>(&sm.xbuf[sp][r][0]);
#pragma unroll
      for (int c = 0; c < kXCols / 4; ++c)
        stg[c ^ rsw] = make_float4(__uint_as_float(sr[4 * c]), __uint_as_float(sr[4 * c + 1]),
                                   __uint_as_float(sr[4 * c + 2]), __uint_as_float(sr[4 * c + 3]));
      fence_proxy_async();
      __syncwarp();
      if (lane == 0)
        bulk_s2peer(peer_xbuf + (hh & 1) * kXBytes, reinterpret_cast<const uint8_t*>(&sm.xbuf[sp][0][0]) + xrows,
                    kXWarpBytes, peer_xfull + (hh & 1) * 8);
      return true;
    };

    const float cl2 = p.scale_log2;
    float m_used = -INFINITY, l_run = 0.f;
    bool ok = n_tiles > 0 && send_half(0);
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int sb = j % kNSP;
      float alpha_t = 1.f;   // O rescale owed for this tile (product over its halves)
      bool need_o = false;
#pragma unroll 1
      for (int e = 0; e < 2; ++e) {
        const int hh = 2 * j + e;
        const int par = hh & 1;
        const int kb = j * kBN + kXCols * e;   // first key of this half
        // Waits are made warp-uniform so that every lane leaves the loop together on an abort.
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.xfull[par], (hh >> 1) & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        if (hh + 2 < n_halves && threadIdx.x == 64) mbar_arrive_expect_tx(&sm.xfull[par], kXBytes);   // half h+2
        float pe[kXCols];
        {
          const float4* xr = reinterpret_cast<const float4*>(&sm.xbuf[par][r][0]);
#pragma unroll
          for (int c = 0; c < kXCols / 4; ++c) {
            const float4 o = xr[c ^ rsw];
            pe[4 * c] = o.x;
            pe[4 * c + 1] = o.y;
            pe[4 * c + 2] = o.z;
            pe[4 * c + 3] = o.w;
          }
        }
        if (hh + 1 < n_halves && !send_half(hh + 1)) {
          ok = false;
          break;
        }
        // S of this half: own partial (still in its tensor-memory buffer) + the peer's, the same
        // sum in either CTA.
        uint32_t sr[kXCols];
        tmem_ld32(tq + kTmS + 64 * sb + kXCols * e, sr);
        tmem_ld_wait();
        float s[kXCols];
#pragma unroll
        for (int c = 0; c < kXCols; ++c) s[c] = __uint_as_float(sr[c]) + pe[c];
        if (!(row_ok && kb + kXCols - 1 <= pos)) {   // causal mask (and rows outside the sequence)
#pragma unroll
          for (int c = 0; c < kXCols; ++c) s[c] = (row_ok && kb + c <= pos) ? s[c] : -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmaxf(fmaxf(s[i], s[i + 8]), fmaxf(s[i + 16], s[i + 24]));
        const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * cl2;
        float alpha = 1.f;
        bool raised = false;
        if (mt > m_used + kLazyRescale) {
          need_o = need_o || (m_used != -INFINITY);
          alpha = ex2(m_used - mt);
          m_used = mt;
          raised = true;
        }
        // The tile's first half of P was written against the old reference: rescale it too, so
        // that P_j V_j sees one reference per row.
        if (e == 1 && __any_sync(0xffffffffu, raised)) {
          uint32_t pw0[16];
          tmem_st_wait();   // the first half's own store has landed
          tmem_ld16(tq + kTmS + 64 * sb, pw0);
          tmem_ld_wait();
          const float a = raised ? alpha : 1.f;
#pragma unroll
          for (int w = 0; w < 16; ++w) pw0[w] = pack_bf16(bf16_lo(pw0[w]) * a, bf16_hi(pw0[w]) * a);
          tmem_st16(tq + kTmS + 64 * sb, pw0);
        }
        const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
        uint32_t pw[16];
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w = 0; w < 16; ++w) {
          const float e0 = ex2(fmaf(s[2 * w], cl2, neg_m));
          const float e1 = ex2(fmaf(s[2 * w + 1], cl2, neg_m));
          ls[w & 3] += e0;
          ls[w & 3] += e1;
          pw[w] = pack_bf16(e0, e1);   // declared cast: P in bf16 for P.V
        }
        l_run = fmaf(l_run, alpha, (ls[0] + ls[1]) + (ls[2] + ls[3]));
        alpha_t *= alpha;
        // P of this half (bf16 key pairs) over columns 16e.. of the tile's S buffer, whose S
        // values there are already consumed: the A operand of P.V.
        tmem_st16(tq + kTmS + 64 * sb + 16 * e, pw);
      }
      if (!ok) break;

      if (__any_sync(0xffffffffu, need_o)) {   // O correction after P_{j-1} V_{j-1} landed
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.pv_done[(j - 1) % kNSP], ((j - 1) / kNSP) & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float a = need_o ? alpha_t : 1.f;
#pragma unroll 1
        for (int cc = 0; cc < kHalf / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tq + kTmO + 32 * cc, o);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * a);
          tmem_st32(tq + kTmO + 32 * cc, o);
        }
        tmem_st_wait();
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sm.p_full[sb]);
    }

    // Epilogue: this CTA's 256 dims of O / l -> bf16, rows of this sequence only.
    if (ok && mbar_wait(&sm.pv_done[(n_tiles - 1) % kNSP], ((n_tiles - 1) / kNSP) & 1, abort_flag, p.err)) {
      tc_fence_after();
      const float inv = (l_run > 0.f) ? __frcp_rn(l_run) : 0.f;
      __nv_bfloat16* orow = p.out + ((size_t)(q_row0 + r) * kGlobalHq + h) * kGD + kHalf * rank;
#pragma unroll 1
      for (int cc = 0; cc < kHalf / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tq + kTmO + 32 * cc, o);
        tmem_ld_wait();
        uint32_t w16[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          w16[c] = pack_bf16(__uint_as_float(o[2 * c]) * inv, __uint_as_float(o[2 * c + 1]) * inv);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * cc);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w16[4 * i], w16[4 * i + 1], w16[4 * i + 2], w16[4 * i + 3]);
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if (sm.abort_flag) {   // let every issued MMA finish before the columns are freed
      if (lane == 0) mma_commit(&sm.teardown);
      __syncwarp();
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(smem_u32(&sm.teardown), 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
    tmem_dealloc(tm, 512);
  }
  // Neither CTA leaves while the other may still write into its shared memory: an abort is
  // passed on (so the peer's waits end early), then each side tells the other it is done.
  if (threadIdx.x == 0) {
    if (sm.abort_flag) st_peer_u32(map_peer(smem_u32(&sm.abort_flag), peer), 1u);
    mbar_arrive_peer(map_peer(smem_u32(&sm.peer_done), peer));
    const uint32_t a = smem_u32(&sm.peer_done);
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait_cluster(a, 0)) {
      if (globaltimer() - t0 > 2 * kWaitLimitNs) {
        set_error(p.err, kErrTimeout);
        break;
      }
    }
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_prefill_global(const SeqRows& rows, float scale_log2, const PagedCache& cache, void* out,
                                  const DeviceState& st, cudaStream_t s) {
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
  CUtensorMap mq;
  if (!q_map(&mq, out, rows.T, kGlobalHq, kGD)) return cudaErrorInvalidValue;
  static bool attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(prefill_global_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGlobalSmemBytes);
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  const long long slots = (long long)rows.T / kBM + 2LL * rows.B;
  const long long blocks = slots * kGlobalHq * 2;   // a pair of CTAs per (query tile, head)
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  prefill_global_kernel<<<(unsigned)blocks, kThreads, kGlobalSmemBytes, s>>>(mq, p);
  return cudaGetLastError();
}

}  // namespace g4
