// Prefill attention on the 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Work unit: (sequence, query tile of 128 positions aligned to absolute position, query head).
// Key tiles of 64 keys are aligned to absolute key 0 and visited in ascending order, so the
// arithmetic a row gets depends only on its own position, its sequence's keys and the window:
// not on the batch, the row's place in it, padding, packing or the launch grid (RL-Kernel RFC
// "[RFC][Gemma-4-31B-it] WS1/WS2 kernel roadmap", section 4 rules 2, 3 and 6).
//
// Sliding layer (RFC section 5, sliding_attention_core: causal local attention, window 1024,
// 32 Q / 16 KV heads, D 256). Per CTA:
//   warps 0, 6  copy producers (Q and K; V): the roped Q tile by TMA, then one bulk copy per
//           tiled page-head block (8 KB: 16 keys x 256 dims as 8x8 core matrices) into a
//           3-stage ring; pages outside the needed key range are never looked up nor copied;
//   warp 1  MMA issuer: S = Q K^T with Q in tensor memory and K (K-major, no swizzle) in shared
//           memory, O += P V with P in tensor memory and V (MN-major, no swizzle) in shared
//           memory; one elected lane issues, commits signal;
//   warps 2-5  one thread per query row: per key tile the mask, the online softmax (lazy
//           rescale, threshold 2^8), P (bf16) written over the tile's own S columns, the O
//           correction when needed, and the epilogue O / l -> bf16.
// The queries arrive already roped: the cache-append pass before this kernel wrote
// bf16(RoPE(q)) into the sequence rows of `out`; the producer's TMA loads the tile from there
// (into ring stage 2, which the softmax threads then empty into tensor memory), and the
// epilogue later overwrites exactly those rows (each row belongs to one CTA).
// Tensor memory (512 columns): O [0,256), Q dims 0-127 [256,320) as bf16 pairs, three S buffers
// [320,512) whose first 32 columns take P once the softmax has read S (three, so that QK^T of
// tile j+1 never waits on P.V of tile j-1). Shared memory: the 3-stage K/V ring and Q dims
// 128-255.
#include <math.h>

#include "g4_prefill_common.cuh"

namespace g4 {

namespace {

using namespace pf;

constexpr int kNS = 3;                    // K/V ring stages (stage 2 first holds the Q tile)
constexpr int kSlidingThreads = 64 + kSoftmaxThreads + 32;   // + the V producer warp (warp 6)

// ---------------------------------------------------------------- sliding layer geometry
constexpr int kSD = kSlidingD;            // 256
constexpr int kPageBytes = kPage * kSD * 2;       // one tiled page-head block: 8 KB
constexpr int kKeyGroupBytes = 8 * kSD * 2;       // 8 keys x all dims: 4 KB
constexpr int kSKTile = (kBN / kPage) * kPageBytes;   // 32 KB: 4 pages, key groups 0..7

constexpr int kNSP = 3;                   // S/P buffers in tensor memory
constexpr uint32_t kTmO = 0, kTmQ = 256, kTmS = 320;   // column offsets: O, Q dims 0-127, S/P x3
constexpr uint32_t kIdescQK = idesc_bf16(kBM, kBN, false, false);
constexpr uint32_t kIdescPV = idesc_bf16(kBM, kSD, false, true);

struct SlidingSmem {
  uint8_t st[kNS][2 * kSKTile];   // ring stage s: K tile, then V tile; st[2] first holds Q dims 0-127
  uint8_t qhi[2 * kQChunk];       // Q dims 128-255 (128B swizzle), the shared-memory A operand
  uint64_t k_full[kNS], k_empty[kNS], v_full[kNS], v_empty[kNS];
  uint64_t s_full[kNSP], p_full[kNSP], pv_done[kNSP];
  uint64_t q_full, q_ready, teardown;
  uint32_t tmem_base;
  int abort_flag;
  int unit_b, unit_t;
};
static_assert(2 * kQChunk <= 2 * kSKTile, "Q dims 0-127 must fit in one ring stage");
constexpr size_t kSlidingSmemBytes = sizeof(SlidingSmem) + 1024;
static_assert(kSlidingSmemBytes <= 232448, "sliding prefill exceeds the 227 KB shared-memory limit");

__global__ void __launch_bounds__(kSlidingThreads, 1)
    prefill_sliding_kernel(const __grid_constant__ CUtensorMap tmap_q, PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  SlidingSmem& sm =
      *reinterpret_cast<SlidingSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x % kSlidingHq;
  const int slot = blockIdx.x / kSlidingHq;
  const int g = h / (kSlidingHq / kSlidingHkv);

  if (warp == 0) {
    int ub, ut;
    find_unit(p.rows, slot, ub, ut);
    if (lane == 0) {
      sm.unit_b = ub;
      sm.unit_t = ut;
    }
  }
  __syncthreads();
  const int b = sm.unit_b;
  if (b < 0) return;
  const int t = sm.unit_t;
  const int cs = p.rows.ctx_start[b], L = p.rows.q_len[b], qs = p.rows.q_start[b];
  const int p_lo = max(kBM * t, cs), p_hi = min(kBM * t + kBM - 1, cs + L - 1);
  const int ctx_end = cs + L;
  if (p_hi >= kMaxPos || (p_hi >> 4) >= p.max_pages) {
    if (threadIdx.x == 0 && h == 0) set_error(p.err, kErrPos);
    return;
  }
  const int W = p.window;
  const int k_lo = W > 0 ? max(0, p_lo - W + 1) : 0;
  const int k_hi = p_hi;
  const int kt0 = k_lo / kBN;
  const int n_tiles = k_hi / kBN - kt0 + 1;
  const int q_row0 = qs + (kBM * t - cs);   // memory row of tile row 0 (may be negative)
  const int32_t* pt = p.page_table + (size_t)b * p.max_pages;

  if (threadIdx.x == 32) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
    }
    for (int s = 0; s < kNSP; ++s) {
      mbar_init(&sm.s_full[s], 1);
      mbar_init(&sm.p_full[s], kSoftmaxThreads);
      mbar_init(&sm.pv_done[s], 1);
    }
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_ready, kSoftmaxThreads);
    mbar_init(&sm.teardown, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == 0 || warp == 6) {
    // ------------------------------------------------------------ copy producers
    // Warp 0 loads the roped Q tile by TMA, then the K tiles; warp 6 loads the V tiles. Split
    // so that K, needed a tile earlier, never queues behind the release of a V stage. One bulk
    // copy per 8 KB tiled page-head block, lanes 0-3 one page each. Block indices come from the
    // page table ahead of use: lane l holds page (l & 3) of tile (l >> 2) of the current group
    // of 8 tiles, and the next group is looked up one group early.
    const bool is_v = (warp == 6);
    auto load_blocks = [&](int j0) -> int {
      const int jt = j0 + (lane >> 2);
      if (jt >= n_tiles) return -1;
      return page_block((kt0 + jt) * kBN + (lane & 3) * kPage, k_lo, k_hi, pt, p.num_pages, kSlidingHkv, g, p.err);
    };
    if (!is_v && lane == 0) {   // the roped Q tile: 4 boxes of 64 dims x 128 rows (rows outside T read as 0)
      prefetch_tmap(&tmap_q);
      mbar_arrive_expect_tx(&sm.q_full, (kSlidingD / 64) * kQChunk);
#pragma unroll
      for (int c = 0; c < kSlidingD / 64; ++c)
        tma_load_3d(c < 2 ? sm.st[2] + c * kQChunk : sm.qhi + (c - 2) * kQChunk, &tmap_q, 64 * c, h, q_row0, &sm.q_full);
    }
    int blk_cur = load_blocks(0), blk_next = load_blocks(8);
    const __nv_bfloat16* src = (const __nv_bfloat16*)(is_v ? p.v_cache : p.k_cache);
    uint64_t* full = is_v ? sm.v_full : sm.k_full;
    uint64_t* empty = is_v ? sm.v_empty : sm.k_empty;
    const int half = is_v ? kSKTile : 0;
    int j = 0;
    for (; j < n_tiles; ++j) {
      const int s = j % kNS;
      if (j > 0 && (j & 7) == 0) {
        blk_cur = blk_next;
        blk_next = load_blocks(j + 8);
      }
      const int my_blk = __shfl_sync(0xffffffffu, blk_cur, (j & 7) * 4 + (lane & 3));
      const unsigned live = __ballot_sync(0xffffffffu, lane < 4 && my_blk >= 0);
      const uint32_t bytes = __popc(live) * kPageBytes;
      bool ok = (j < kNS) || lane != 0 || mbar_wait(&empty[s], ((j / kNS) - 1) & 1, abort_flag, p.err);
      if (j == 2 && lane == 0) ok = ok && mbar_wait(&sm.q_ready, 0, abort_flag, p.err);   // Q left stage 2
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (lane == 0) mbar_arrive_expect_tx(&full[s], bytes);
      __syncwarp();
      if (lane < 4 && my_blk >= 0)
        bulk_g2s(sm.st[s] + half + lane * kPageBytes, src + (size_t)my_blk * kPage * kSD, kPageBytes, &full[s]);
    }
    if (lane == 0 && *abort_flag) {   // drain copies still in flight (bounded) before the CTA may exit
      const unsigned long long t0 = globaltimer();
      if (!is_v) {
        while (!mbar_try_wait(smem_u32(&sm.q_full), 0) && globaltimer() - t0 < kWaitLimitNs) {
        }
      }
      for (int i = max(0, j - kNS); i < j; ++i) {
        while (!mbar_try_wait(smem_u32(&full[i % kNS]), (i / kNS) & 1) && globaltimer() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    auto pv = [&](int i) -> bool {
      if (!mbar_wait(&sm.p_full[i % kNSP], (i / kNSP) & 1, abort_flag, p.err)) return false;
      if (!mbar_wait(&sm.v_full[i % kNS], (i / kNS) & 1, abort_flag, p.err)) return false;
      const int kb = (kt0 + i) * kBN;
      // V rows of keys that hold no data of this sequence are zeroed before P.V: pages that
      // were not copied (outside the needed key range) keep an older tile, and slots past the
      // sequence's last key may hold anything (NaN); P = 0 there does not cancel NaN.
      const int v0 = max(kb, (k_lo >> 4) * kPage), v1 = min(min(kb + kBN, ((k_hi >> 4) + 1) * kPage), ctx_end);
      if (v0 > kb || v1 < kb + kBN) {
        for (int idx = lane; idx < kBN * (kSD / 8); idx += 32) {
          const int r = idx / (kSD / 8), dg = idx % (kSD / 8);
          if (kb + r < v0 || kb + r >= v1)
            *reinterpret_cast<uint4*>(sm.st[i % kNS] + kSKTile + ((r >> 3) * (kSD / 8) + dg) * 128 + (r & 7) * 16) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
        __syncwarp();
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t va = smem_u32(sm.st[i % kNS] + kSKTile);
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k)
          mma_ts(tm + kTmO, tm + kTmS + 64 * (i % kNSP) + 8 * k,
                 desc_tiled(va + k * 2 * kKeyGroupBytes, kKeyGroupBytes, 128), kIdescPV, (i > 0 || k > 0) ? 1u : 0u);
        mma_commit(&sm.pv_done[i % kNSP]);
        mma_commit(&sm.v_empty[i % kNS]);
      }
      __syncwarp();
      return true;
    };
    bool ok = mbar_wait(&sm.q_ready, 0, abort_flag, p.err);
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int s = j % kNS;
      if (!mbar_wait(&sm.k_full[s], (j / kNS) & 1, abort_flag, p.err)) break;
      // S buffer j % 3 last held P_{j-3}: reuse it once P_{j-3} V_{j-3} has completed (issued two
      // MMA groups earlier, so this wait does not drain the tensor pipe).
      if (j >= kNSP && !mbar_wait(&sm.pv_done[j % kNSP], ((j - kNSP) / kNSP) & 1, abort_flag, p.err)) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t ka = smem_u32(sm.st[s]);
        const uint32_t qh = smem_u32(sm.qhi);
        const uint32_t sd = tm + kTmS + 64 * (j % kNSP);
#pragma unroll
        for (int k = 0; k < 8; ++k)   // dims 0-127: Q from tensor memory
          mma_ts(sd, tm + kTmQ + 8 * k, desc_tiled(ka + k * 256, 128, kKeyGroupBytes), kIdescQK, k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 8; k < 16; ++k)  // dims 128-255: Q from shared memory
          mma_ss(sd, desc_sw128(qh + ((k - 8) >> 2) * kQChunk + (k & 3) * 32, 16, 1024),
                 desc_tiled(ka + k * 256, 128, kKeyGroupBytes), kIdescQK, 1u);
        mma_commit(&sm.s_full[j % kNSP]);
        mma_commit(&sm.k_empty[s]);
      }
      __syncwarp();
      if (j >= 1 && !pv(j - 1)) {
        ok = false;
        break;
      }
      if (j == n_tiles - 1 && !pv(j)) ok = false;
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------ softmax / epilogue warps
    const int r = 32 * (warp & 3) + lane;   // query row = tensor-memory lane
    const uint32_t tq = tm + tmem_lane_base(warp);
    const int pos = kBM * t + r;
    const bool row_ok = pos >= p_lo && pos <= p_hi;

    // Q: the producer's TMA brought the roped tile in (4 chunks of 64 dims, 128B swizzle);
    // dims 0-127 sit in ring stage 2 and each thread moves its row of them into tensor memory
    // (an A operand in bf16 pairs), which frees stage 2 for keys and values. Dims 128-255 stay
    // in shared memory as the A operand of the other half of the QK^T k-steps.
    {
      const bool okq = mbar_wait(&sm.q_full, 0, abort_flag, p.err);
      const uint8_t* qrow = sm.st[2] + r * 128;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint4 v = okq ? *reinterpret_cast<const uint4*>(qrow + c * kQChunk + ((g ^ (r & 7)) * 16))
                              : make_uint4(0, 0, 0, 0);
          w[4 * g] = v.x;
          w[4 * g + 1] = v.y;
          w[4 * g + 2] = v.z;
          w[4 * g + 3] = v.w;
        }
        tmem_st32(tq + kTmQ + 32 * c, w);   // dims 64c .. 64c+63 -> columns 32c .. 32c+31
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sm.q_ready);
    }

    const float cl2 = p.scale_log2;
    float m_used = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int kb = (kt0 + j) * kBN;
      const int sb = j % kNSP;
      if (!mbar_wait(&sm.s_full[sb], (j / kNSP) & 1, abort_flag, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld32(tq + kTmS + 64 * sb, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(tq + kTmS + 64 * sb + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld_wait();

      float s[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(sr[c]);
      const bool full = row_ok && kb + kBN - 1 <= pos && (W == 0 || pos - kb <= W - 1);
      if (!full) {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int key = kb + c;
          const bool vis = row_ok && key <= pos && (W == 0 || pos - key <= W - 1);
          s[c] = vis ? s[c] : -INFINITY;
        }
      }
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        mx[i] = s[i];
#pragma unroll
        for (int c = 1; c < 8; ++c) mx[i] = fmaxf(mx[i], s[i + 8 * c]);
      }
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * cl2;
      float alpha = 1.f;
      bool need_o = false;
      if (mt > m_used + kLazyRescale) {
        need_o = (m_used != -INFINITY);
        alpha = ex2(m_used - mt);
        m_used = mt;
      }
      const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
      uint32_t pw[32];
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < 32; ++w) {
        const float e0 = ex2(fmaf(s[2 * w], cl2, neg_m));
        const float e1 = ex2(fmaf(s[2 * w + 1], cl2, neg_m));
        ls[w & 3] += e0;
        ls[w & 3] += e1;
        pw[w] = pack_bf16(e0, e1);   // declared cast: P in bf16 for P.V
      }
      l_run = fmaf(l_run, alpha, (ls[0] + ls[1]) + (ls[2] + ls[3]));

      // P_j (bf16 key pairs) over the first 32 columns of its own S buffer: the A operand of P.V.
      tmem_st32(tq + kTmS + 64 * sb, pw);

      // O correction (rows whose max rose by more than 2^8), after P_{j-1} V_{j-1} landed.
      if (__any_sync(0xffffffffu, need_o)) {
        if (!mbar_wait(&sm.pv_done[(j - 1) % kNSP], ((j - 1) / kNSP) & 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float a = need_o ? alpha : 1.f;
#pragma unroll 1
        for (int cc = 0; cc < kSD / 32; ++cc) {
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

    // Epilogue: O / l -> bf16, rows of this sequence only.
    if (ok && mbar_wait(&sm.pv_done[(n_tiles - 1) % kNSP], ((n_tiles - 1) / kNSP) & 1, abort_flag, p.err)) {
      tc_fence_after();
      const float inv = (l_run > 0.f) ? __frcp_rn(l_run) : 0.f;
      __nv_bfloat16* orow = p.out + ((size_t)(q_row0 + r) * kSlidingHq + h) * kSD;
#pragma unroll 1
      for (int cc = 0; cc < kSD / 32; ++cc) {
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
}

}  // namespace

cudaError_t launch_prefill(bool global, const SeqRows& rows, int window, float scale_log2, const PagedCache& cache,
                           void* out, const DeviceState& st, cudaStream_t s) {
  if (global) return launch_prefill_global(rows, scale_log2, cache, out, st, s);
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
  p.k_cache = cache.k;
  p.v_cache = cache.v;
  CUtensorMap mq;
  if (!q_map(&mq, out, rows.T, kSlidingHq, kSD)) return cudaErrorInvalidValue;
  static bool attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(prefill_sliding_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSlidingSmemBytes);
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  const long long slots = (long long)rows.T / kBM + 2LL * rows.B;
  const long long blocks = slots * kSlidingHq;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  prefill_sliding_kernel<<<(unsigned)blocks, kSlidingThreads, kSlidingSmemBytes, s>>>(mq, p);
  return cudaGetLastError();
}

}  // namespace g4
