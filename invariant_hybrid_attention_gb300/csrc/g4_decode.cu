// Paged decode: one query token per request against its cached keys, split into fixed key
// chunks aligned to absolute position 0 and merged in ascending chunk order.
//
// The RL-Kernel RFC "[RFC][Gemma-4-31B-it] WS1/WS2 kernel roadmap", section 4 rule 3, forbids
// split-KV unless the split and merge tree is fixed by the contract. Here the split is fixed:
// chunk c holds keys [C*c, C*c + C) (C = 256 sliding, 1024 global), whatever the batch, and
// inside a chunk the pages go round-robin to four warps whose states merge in warp order.
// Every number a request gets depends only on its own position, window and data.
//
// Both layer kinds run on warp-level bf16 MMA (m16n8k16) over bulk-copied page blocks. Global
// layers (8 query heads per KV head, K==V, 16 flop per byte): S^T = K q^T,
// where K is the stored S except on the 128 rotated dims (pairs t < 64: dims t and t+256),
// which come from the cache's k_rot side pages (p-RoPE(S), written with S by the append pass);
// then O^T += S^T' P^T with the un-rotated S rows as V.
#include <math.h>

#include "g4_internal.h"

namespace g4 {

namespace {

constexpr float kLazyRescale = 8.0f;   // rescale only when the running max grows by > 2^8

struct DecodeParams {
  const __nv_bfloat16* q;   // [B][32][D]
  const int32_t* seq_len;   // [B]
  int B;
  int window;               // sliding W; 0 on global layers
  float scale_log2;         // softmax_scale * log2(e)
  PagedCache cache;
  float* ws_ml;             // [B][32][NC][2]: running max (log2 units) and sum
  float* ws_o;              // [B][32][NC][D]: unnormalised output
  int NC;                   // chunk slots per (request, head)
  RopeTables tb;
  uint32_t* err;
  unsigned long long wait_ns;   // limit of every protocol wait (g4attn_set_wait_limit_ns)
};

// ---------------------------------------------------------------- sliding: D 256, Hkv 16, G 2
// One CTA per (fixed 256-key chunk, KV head, request); its pages (16 keys each) go round-robin
// to 4 warps. Pages arrive by bulk copy (8 KB of K' and 8 KB of V per page-head block) into a
// 6-stage ring shared by the warps: page i sits in stage i % 6, and the warp that consumed
// page i refills that stage with page i + 6. A per-stage count of issued pages lets the
// consumer of page i wait until page i has been issued before it tests the barrier: from then
// on the barrier is in phase i / 6 or the one after, which a parity wait tells apart (a
// parity wait cannot tell phases two apart, and the consumer of page i never saw page i - 6). Scores S^T = K q^T and O^T += V^T P^T run on
// warp-level bf16 MMA (m16n8k16) from ldmatrix on the tiled blocks; the two query heads of
// the KV head are columns 0-1 of the 8-wide N dimension (the other columns carry q = 0 and
// are never read out).
constexpr int kSD = kSlidingD;
constexpr int kSStages = 6;
constexpr int kSPageBytes = kPage * kSD * 2;      // one tiled page-head block (K' or V): 8 KB
constexpr int kSStageBytes = 2 * kSPageBytes;     // K' then V
constexpr int kSPRow = 48;                        // P^T staging row (8 heads x 16 keys bf16, padded)
constexpr int kSSmem = kSStages * kSStageBytes + 4 * 8 * kSPRow + kSStages * 8;

__global__ void __launch_bounds__(128, 2) decode_sliding_kernel(DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  uint8_t* p_s_all = smem + kSStages * kSStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(p_s_all + 4 * 8 * kSPRow);
  __shared__ int abort_flag;
  __shared__ int issued[kSStages];   // pages issued into each stage so far
  __shared__ float red_m[4][2], red_l[4][2];

  const int cr = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, cq = lane & 3;   // mma fragment coordinates

  const int pos = p.seq_len[b] - 1;
  if (pos < 0 || pos >= kMaxPos || (pos >> 4) >= p.cache.max_pages) {
    if (threadIdx.x == 0 && cr == 0 && g == 0) set_error(p.err, kErrPos);
    return;   // the merge writes zeros for this request
  }
  const int lo = max(0, pos - p.window + 1);
  const int c = lo / kDecodeChunkSliding + cr;
  const int k_begin = max(lo, c * kDecodeChunkSliding);
  const int k_end = min(pos, c * kDecodeChunkSliding + kDecodeChunkSliding - 1);   // inclusive
  if (k_begin > k_end) return;                                                       // unused slot

  const int pg0 = k_begin >> 4, pg1 = k_end >> 4;
  const int n_pages = pg1 - pg0 + 1;
  const int32_t* pt = p.cache.page_table + (size_t)b * p.cache.max_pages;
  bool bad = false;
  for (int i = pg0 + (int)threadIdx.x; i <= pg1; i += 128) {
    const int ph = pt[i];
    bad |= (ph < 0 || ph >= p.cache.num_pages);
  }
  if (threadIdx.x == 0) abort_flag = 0;
  if (threadIdx.x < kSStages) {
    mbar_init(&full[threadIdx.x], 1);
    issued[threadIdx.x] = 0;
  }
  fence_mbar_init();
  const size_t slot = (((size_t)b * p.cache.hq + 2 * g) * p.NC + cr);
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) {
      set_error(p.err, kErrPage);
      for (int hh = 0; hh < 2; ++hh) {
        p.ws_ml[(slot + (size_t)hh * p.NC) * 2 + 0] = -INFINITY;
        p.ws_ml[(slot + (size_t)hh * p.NC) * 2 + 1] = 0.f;
      }
    }
    return;
  }

  const __nv_bfloat16* kc = (const __nv_bfloat16*)p.cache.k;
  const __nv_bfloat16* vc = (const __nv_bfloat16*)p.cache.v;
  auto issue = [&](int i) {   // one thread
    const int st = i % kSStages;
    const size_t blk = (size_t)pt[pg0 + i] * p.cache.hkv + g;
    uint8_t* dst = ring + st * kSStageBytes;
    mbar_arrive_expect_tx(&full[st], kSStageBytes);
    bulk_g2s(dst, kc + blk * kPage * kSD, kSPageBytes, &full[st]);
    bulk_g2s(dst + kSPageBytes, vc + blk * kPage * kSD, kSPageBytes, &full[st]);
    __threadfence_block();
    *reinterpret_cast<volatile int*>(&issued[st]) = i / kSStages + 1;
  };
  if (threadIdx.x == 0)
    for (int i = 0; i < min(kSStages, n_pages); ++i) issue(i);

  // Roped query as B fragments: b0/b1 of k-step ks hold q[gq][16ks + 2cq (+8) .. +1] for
  // heads gq = 0, 1 (zero for the other columns). Pair t and t + 128 sit in k-steps ks and
  // ks + 8 of the same lane.
  uint32_t qb[16][2];
#pragma unroll
  for (int ks = 0; ks < 16; ++ks) qb[ks][0] = qb[ks][1] = 0u;
  if (gq < 2) {
    const __nv_bfloat16* qr = p.q + ((size_t)b * p.cache.hq + 2 * g + gq) * kSD;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int t = 16 * ks + 8 * hf + 2 * cq;
        const uint32_t xw = *reinterpret_cast<const uint32_t*>(qr + t);
        const uint32_t yw = *reinterpret_cast<const uint32_t*>(qr + t + kSD / 2);
        float x0 = bf16_lo(xw), x1 = bf16_hi(xw), y0 = bf16_lo(yw), y1 = bf16_hi(yw);
        rope_pair(x0, y0, rope_cs(p.tb, t, pos));
        rope_pair(x1, y1, rope_cs(p.tb, t + 1, pos));
        qb[ks][hf] = pack_bf16(x0, x1);   // declared cast: roped q in bf16
        qb[ks + 8][hf] = pack_bf16(y0, y1);
      }
    }
  }

  uint8_t* p_s = p_s_all + warp * 8 * kSPRow;
  const uint32_t p_addr = smem_u32(p_s);
  float o[16][4];
#pragma unroll
  for (int mt = 0; mt < 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  // ldmatrix lane addresses. K block [key group kg][dim group dg][8 keys][8 dims] (core matrices
  // of 128 B at (kg * 32 + dg) * 128): K as A takes tiles (keys 0-7 | 8-15) x (dims +0 | +8).
  // V block in 128-dim halves [half][kg][dg 0-15][8][8] (core matrix (kg, dg) at
  // ((dg / 16 * 2 + kg) * 16 + dg % 16) * 128): V^T as A (transposed) takes tiles (dims +0 | +8) x
  // (keys 0-7 | 8-15); dim tile mt starts at (mt / 8) * 4096 + (mt % 8) * 256.
  const uint32_t a_lane = (((lane >> 3) & 1) * 32 + (lane >> 4)) * 128 + (lane & 7) * 16;
  const uint32_t v_lane = (((lane >> 4) & 1) * 16 + ((lane >> 3) & 1)) * 128 + (lane & 7) * 16;

  for (int i = warp; i < n_pages; i += 4) {
    const int st = i % kSStages, ph = i / kSStages;
    if (ph > 0) {   // page i issued yet? (bounded)
      bool ok = true;
      const unsigned long long t0 = globaltimer();
      while (*reinterpret_cast<volatile int*>(&issued[st]) <= ph) {
        if (*reinterpret_cast<volatile int*>(&abort_flag)) {
          ok = false;
          break;
        }
        if (globaltimer() - t0 >= p.wait_ns) {
          abort_flag = 1;
          set_error(p.err, kErrTimeout);
          ok = false;
          break;
        }
      }
      if (!__all_sync(0xffffffffu, ok)) break;
      __threadfence_block();
    }
    if (!mbar_wait(&full[st], ph & 1, &abort_flag, p.err, p.wait_ns)) break;
    uint8_t* kp = ring + st * kSStageBytes;
    uint8_t* vp = kp + kSPageBytes;
    const int key0 = (pg0 + i) * kPage;
    if (key0 < k_begin || key0 + kPage - 1 > k_end) {   // V rows of keys outside the chunk: zero
      for (int idx = lane; idx < kPage * (kSD / 8); idx += 32) {
        const int r = idx / (kSD / 8), dg = idx % (kSD / 8);
        if (key0 + r < k_begin || key0 + r > k_end)
          *reinterpret_cast<uint4*>(vp + (((dg >> 4) * 2 + (r >> 3)) * 16 + (dg & 15)) * 128 + (r & 7) * 16) =
              make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }
    const uint32_t ka = smem_u32(kp), va = smem_u32(vp);

    // ---- S^T = K q^T (16 keys x 8 columns), two accumulation chains
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 16; ks += 2) {
      uint32_t a[4], a2[4];
      ldsm_x4(ka + a_lane + ks * 256, a[0], a[1], a[2], a[3]);
      ldsm_x4(ka + a_lane + (ks + 1) * 256, a2[0], a2[1], a2[2], a2[3]);
      mma16816(s0, a[0], a[1], a[2], a[3], qb[ks][0], qb[ks][1]);
      mma16816(s1, a2[0], a2[1], a2[2], a2[3], qb[ks + 1][0], qb[ks + 1][1]);
    }

    // ---- online softmax per column (heads 2cq, 2cq+1; keys gq, gq+8)
    float x[4];
    const bool v_lo = key0 + gq >= k_begin && key0 + gq <= k_end;
    const bool v_hi = key0 + gq + 8 >= k_begin && key0 + gq + 8 <= k_end;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float sv = s0[r] + s1[r];
      x[r] = ((r < 2) ? v_lo : v_hi) ? sv * p.scale_log2 : -INFINITY;
    }
    float pb[4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float mt = fmaxf(x[j], x[2 + j]);
#pragma unroll
      for (int m = 4; m <= 16; m <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, m));
      const float mn = fmaxf(m_run[j], mt);
      if (mn > m_run[j] + kLazyRescale) {
        const float al = exp2f(m_run[j] - mn);
        m_run[j] = mn;
        l_run[j] *= al;
#pragma unroll
        for (int mt2 = 0; mt2 < 16; ++mt2) {
          o[mt2][j] *= al;
          o[mt2][2 + j] *= al;
        }
      }
      pb[j] = (x[j] == -INFINITY) ? 0.f : round_bf16(exp2f(x[j] - m_run[j]));
      pb[2 + j] = (x[2 + j] == -INFINITY) ? 0.f : round_bf16(exp2f(x[2 + j] - m_run[j]));
      float ls = pb[j] + pb[2 + j];
#pragma unroll
      for (int m = 4; m <= 16; m <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, m);
      l_run[j] += ls;
    }
    // P^T into the B-fragment layout through a per-warp staging block [column][key].
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      *reinterpret_cast<__nv_bfloat16*>(p_s + (2 * cq + j) * kSPRow + gq * 2) = __float2bfloat16_rn(pb[j]);
      *reinterpret_cast<__nv_bfloat16*>(p_s + (2 * cq + j) * kSPRow + (gq + 8) * 2) = __float2bfloat16_rn(pb[2 + j]);
    }
    __syncwarp();
    uint32_t pb0, pb1;
    ldsm_x2(p_addr + (lane & 7) * kSPRow + ((lane >> 3) & 1) * 16, pb0, pb1);

    // ---- O^T += V^T P^T over the 16 dim tiles
#pragma unroll
    for (int mt = 0; mt < 16; ++mt) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(va + v_lane + (mt >> 3) * 4096 + (mt & 7) * 256, a0, a1, a2, a3);
      mma16816(o[mt], a0, a1, a2, a3, pb0, pb1);
    }
    __syncwarp();
    if (lane == 0 && i + kSStages < n_pages) {   // refill this stage with page i + 6
      fence_proxy_async();
      issue(i + kSStages);
    }
  }
  __syncthreads();
  if (abort_flag && threadIdx.x == 0) {   // after a timeout: wait (bounded) for copies in flight
    const unsigned long long t0 = globaltimer();
    for (int st = 0; st < kSStages; ++st)
      if (issued[st] > 0)
        while (!mbar_try_wait(smem_u32(&full[st]), (issued[st] - 1) & 1) && globaltimer() - t0 < kWaitLimitNs) {
        }
  }
  __syncthreads();   // all stages consumed: reuse the ring for the warp merge

  float* red_o = reinterpret_cast<float*>(ring);   // [warps][2 heads][256]
  if (lane == 0) {
    red_m[warp][0] = m_run[0];
    red_m[warp][1] = m_run[1];
    red_l[warp][0] = l_run[0];
    red_l[warp][1] = l_run[1];
  }
  if (cq == 0) {
#pragma unroll
    for (int mt = 0; mt < 16; ++mt) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int d = mt * 16 + gq + 8 * (r >> 1), hh = r & 1;
        red_o[(warp * 2 + hh) * kSD + d] = o[mt][r];
      }
    }
  }
  __syncthreads();
  // Merge the four warps in warp order; thread t writes 4 of the 2 x 256 outputs.
  for (int idx = threadIdx.x; idx < 2 * kSD; idx += 128) {
    const int hh = idx / kSD, d = idx % kSD;
    float M = red_m[0][hh];
#pragma unroll
    for (int w = 1; w < 4; ++w) M = fmaxf(M, red_m[w][hh]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float sc = (M == -INFINITY) ? 0.f : exp2f(red_m[w][hh] - M);
      L = fmaf(red_l[w][hh], sc, L);
      O = fmaf(red_o[(w * 2 + hh) * kSD + d], sc, O);
    }
    const size_t s = slot + (size_t)hh * p.NC;
    p.ws_o[s * kSD + d] = O;
    if (d == 0) {
      p.ws_ml[s * 2 + 0] = M;
      p.ws_ml[s * 2 + 1] = L;
    }
  }
}

// ---------------------------------------------------------------- global: D 512, Hkv 4, G 8, K==V
constexpr int kGD = kGlobalD;
constexpr int kGWarps = 4;
constexpr int kGStages = 5;                      // ring of page stages shared by the 4 warps
constexpr int kGSBytes = kPage * kGD * 2;        // one tiled page-head block of S: 16 KB
constexpr int kGRotBytes = kRotPageElems * 2;    // its k_rot block: 4 KB
constexpr int kGStageBytes = kGSBytes + kGRotBytes;
constexpr int kGRow = kGD * 2 + 16;              // padded query row: ldmatrix rows hit distinct banks
constexpr int kGQBytes = 8 * kGRow;              // the 8 roped query heads
constexpr int kGPRow = 48;                       // P^T staging row (8 heads x 16 keys bf16, padded)
constexpr int kGSmem = kGStages * kGStageBytes + kGQBytes + kGWarps * 8 * kGPRow + kGStages * 8;
static_assert(kGStages * kGStageBytes >= kGWarps * 8 * kGD * 4, "the warp merge reuses the ring");

// Page i of the chunk goes to warp i % 4 and sits in ring stage i % 5; the warp that consumed
// page i refills the stage with page i + 5. As in the sliding kernel, the consumer of page i
// first waits until page i has been issued (per-stage counts), so that a parity wait names
// the right phase. Two CTAs fit per SM.
__global__ void __launch_bounds__(128, 2) decode_global_kernel(DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stage_base = smem;
  uint8_t* q_s = smem + kGStages * kGStageBytes;
  uint8_t* p_s_all = q_s + kGQBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(p_s_all + kGWarps * 8 * kGPRow);
  __shared__ int abort_flag;
  __shared__ int issued[kGStages];   // pages issued into each stage so far
  __shared__ float red_m[kGWarps][8], red_l[kGWarps][8];

  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, cq = lane & 3;      // mma fragment coordinates

  const int pos = p.seq_len[b] - 1;
  if (pos < 0 || pos >= kMaxPos || (pos >> 4) >= p.cache.max_pages) {
    if (threadIdx.x == 0 && c == 0 && g == 0) set_error(p.err, kErrPos);
    return;
  }
  const int k_begin = c * kDecodeChunkGlobal;
  if (k_begin > pos) return;
  const int k_end = min(pos, k_begin + kDecodeChunkGlobal - 1);
  const int pg0 = k_begin >> 4, pg1 = k_end >> 4;
  const int32_t* pt = p.cache.page_table + (size_t)b * p.cache.max_pages;
  const int G = p.cache.hq / p.cache.hkv;   // query heads of KV head g: 8, or 4 on a tp = 8 rank slice
  const size_t slot = ((size_t)b * p.cache.hq + G * g) * p.NC + c;   // head G g + j adds j * NC

  bool bad = false;
  for (int i = pg0 + (int)threadIdx.x; i <= pg1; i += 128) {
    const int ph = pt[i];
    bad |= (ph < 0 || ph >= p.cache.num_pages);
  }
  if (threadIdx.x == 0) abort_flag = 0;
  if (threadIdx.x < kGStages) {
    mbar_init(&full[threadIdx.x], 1);
    issued[threadIdx.x] = 0;
  }
  fence_mbar_init();
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) {
      set_error(p.err, kErrPage);
      for (int j = 0; j < G; ++j) {
        p.ws_ml[(slot + (size_t)j * p.NC) * 2 + 0] = -INFINITY;
        p.ws_ml[(slot + (size_t)j * p.NC) * 2 + 1] = 0.f;
      }
    }
    return;
  }

  const int n_pages = pg1 - pg0 + 1;
  const __nv_bfloat16* sc = (const __nv_bfloat16*)p.cache.k;
  const __nv_bfloat16* rc = (const __nv_bfloat16*)p.cache.krot;
  auto issue = [&](int i) {   // one thread
    const int st = i % kGStages;
    const size_t blk = (size_t)pt[pg0 + i] * p.cache.hkv + g;
    uint8_t* dst = stage_base + st * kGStageBytes;
    mbar_arrive_expect_tx(&full[st], kGStageBytes);
    bulk_g2s(dst, sc + blk * kPage * kGD, kGSBytes, &full[st]);
    bulk_g2s(dst + kGSBytes, rc + blk * kRotPageElems, kGRotBytes, &full[st]);
    __threadfence_block();
    *reinterpret_cast<volatile int*>(&issued[st]) = i / kGStages + 1;
  };
  if (threadIdx.x == 0)
    for (int i = 0; i < min(kGStages, n_pages); ++i) issue(i);

  // Stage the G roped query heads (bf16) while the first pages are in flight; the columns of the
  // MMA past G (a rank slice's 4 heads) carry q = 0 and are never read out.
  {
    const __nv_bfloat16* qb = p.q + ((size_t)b * p.cache.hq + G * g) * kGD;
    for (int idx = threadIdx.x; idx < 8 * (kGD / 2); idx += 128) {
      const int h = idx / (kGD / 2), t = idx % (kGD / 2);
      float x = 0.f, y = 0.f;
      if (h < G) {
        x = bf16_to_f(qb[h * kGD + t]);
        y = bf16_to_f(qb[h * kGD + t + kGD / 2]);
      }
      if (t < kGlobalR) rope_pair(x, y, rope_cs(p.tb, t, pos));
      *reinterpret_cast<__nv_bfloat16*>(q_s + h * kGRow + t * 2) = __float2bfloat16_rn(x);
      *reinterpret_cast<__nv_bfloat16*>(q_s + h * kGRow + (t + kGD / 2) * 2) = __float2bfloat16_rn(y);
    }
  }
  __syncthreads();

  const uint32_t q_addr = smem_u32(q_s);
  uint8_t* p_s = p_s_all + warp * 8 * kGPRow;
  const uint32_t p_addr = smem_u32(p_s);
  float o[32][4];
#pragma unroll
  for (int mt = 0; mt < 32; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

  // ldmatrix lane addressing. A page stage is a tiled global page: two halves of 256 dims,
  // each [key group kg][dim group dg][8 keys][8 dims] (core matrices of 128 B at
  // ((half * 2 + kg) * 32 + dg) * 128): each 8x8 ldmatrix tile is one core matrix.
  // K as A (non-transposed): tiles (keys 0-7 | 8-15) x (dims +0 | +8);
  // V^T as A (transposed): tiles (dims +0 | +8) x (keys 0-7 | 8-15).
  // A 16-dim step s starts at byte (s / 16) * 8192 + (s % 16) * 256 of the stage.
  // The k_rot block after it holds the rotated dims as [half][kg][dg 0-7][8][8]: rotated step
  // s (s % 16 < 4) starts at byte 16384 + (s / 16) * 2048 + (s % 16) * 256, key groups 1 KB apart.
  const uint32_t a_lane = (((lane >> 3) & 1) * 32 + (lane >> 4)) * 128 + (lane & 7) * 16;
  const uint32_t r_lane = kGSBytes + (((lane >> 3) & 1) * 8 + (lane >> 4)) * 128 + (lane & 7) * 16;
  const uint32_t v_lane = (((lane >> 4) & 1) * 32 + ((lane >> 3) & 1)) * 128 + (lane & 7) * 16;
  auto step_off = [](int s16) -> uint32_t { return (uint32_t)((s16 >> 4) * 8192 + (s16 & 15) * 256); };
  const uint32_t q_lane = q_addr + (lane & 7) * kGRow + (lane >> 3) * 16;

  for (int i = warp; i < n_pages; i += kGWarps) {
    const int st = i % kGStages, ph = i / kGStages;
    if (ph > 0) {   // page i issued yet? (bounded)
      bool ok = true;
      const unsigned long long t0 = globaltimer();
      while (*reinterpret_cast<volatile int*>(&issued[st]) <= ph) {
        if (*reinterpret_cast<volatile int*>(&abort_flag)) {
          ok = false;
          break;
        }
        if (globaltimer() - t0 >= p.wait_ns) {
          abort_flag = 1;
          set_error(p.err, kErrTimeout);
          ok = false;
          break;
        }
      }
      if (!__all_sync(0xffffffffu, ok)) break;
      __threadfence_block();
    }
    if (!mbar_wait(&full[st], ph & 1, &abort_flag, p.err, p.wait_ns)) break;
    uint8_t* page = stage_base + st * kGStageBytes;
    const int key0 = (pg0 + i) * kPage;
    if (key0 + kPage - 1 > k_end) {   // zero stale rows (NaN-safe V), then make them visible
      for (int idx = lane; idx < kPage * (kGD / 8); idx += 32) {
        const int r = idx / (kGD / 8), dg = idx % (kGD / 8);
        if (key0 + r > k_end)
          *reinterpret_cast<uint4*>(page + (((dg >> 5) * 2 + (r >> 3)) * 32 + (dg & 31)) * 128 + (r & 7) * 16) =
              make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }
    const uint32_t pa = smem_u32(page);

    // ---- S^T = K q^T (16 keys x 8 heads), two accumulation chains
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {   // rotated k-steps: dims 16ks.. and their partners +256
      uint32_t a[4], h[4], bq0, bq1, bh0, bh1;
      ldsm_x4(pa + r_lane + ks * 256, a[0], a[1], a[2], a[3]);
      ldsm_x4(pa + r_lane + 2048 + ks * 256, h[0], h[1], h[2], h[3]);
      uint32_t t0, t1;
      ldsm_x4(q_lane + ks * 32, bq0, bq1, t0, t1);          // k-step ks (and ks+1, unused)
      ldsm_x4(q_lane + (ks + 16) * 32, bh0, bh1, t0, t1);   // k-step ks+16
      mma16816(s0, a[0], a[1], a[2], a[3], bq0, bq1);
      mma16816(s1, h[0], h[1], h[2], h[3], bh0, bh1);
    }
#pragma unroll
    for (int kp = 0; kp < 32; kp += 2) {   // plain k-steps, two at a time
      if ((kp >= 0 && kp < 4) || (kp >= 16 && kp < 20)) continue;
      uint32_t a[4], a2[4], b0, b1, b2, b3;
      ldsm_x4(pa + a_lane + step_off(kp), a[0], a[1], a[2], a[3]);
      ldsm_x4(pa + a_lane + step_off(kp + 1), a2[0], a2[1], a2[2], a2[3]);
      ldsm_x4(q_lane + kp * 32, b0, b1, b2, b3);
      mma16816(s0, a[0], a[1], a[2], a[3], b0, b1);
      mma16816(s1, a2[0], a2[1], a2[2], a2[3], b2, b3);
    }

    // ---- online softmax per head column (heads 2cq, 2cq+1; keys gq, gq+8)
    float x[4];
    const bool v_lo = key0 + gq <= k_end, v_hi = key0 + gq + 8 <= k_end;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float sv = s0[r] + s1[r];
      x[r] = ((r < 2) ? v_lo : v_hi) ? sv * p.scale_log2 : -INFINITY;
    }
    float pb[4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float mt = fmaxf(x[j], x[2 + j]);
#pragma unroll
      for (int m = 4; m <= 16; m <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, m));
      const float mn = fmaxf(m_run[j], mt);
      if (mn > m_run[j] + kLazyRescale) {
        const float al = exp2f(m_run[j] - mn);
        m_run[j] = mn;
        l_run[j] *= al;
#pragma unroll
        for (int mt2 = 0; mt2 < 32; ++mt2) {
          o[mt2][j] *= al;
          o[mt2][2 + j] *= al;
        }
      }
      pb[j] = (x[j] == -INFINITY) ? 0.f : round_bf16(exp2f(x[j] - m_run[j]));
      pb[2 + j] = (x[2 + j] == -INFINITY) ? 0.f : round_bf16(exp2f(x[2 + j] - m_run[j]));
      float ls = pb[j] + pb[2 + j];
#pragma unroll
      for (int m = 4; m <= 16; m <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, m);
      l_run[j] += ls;
    }
    // P^T into the B-fragment layout through a tiny per-warp staging block [head][key].
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      *reinterpret_cast<__nv_bfloat16*>(p_s + (2 * cq + j) * kGPRow + gq * 2) = __float2bfloat16_rn(pb[j]);
      *reinterpret_cast<__nv_bfloat16*>(p_s + (2 * cq + j) * kGPRow + (gq + 8) * 2) = __float2bfloat16_rn(pb[2 + j]);
    }
    __syncwarp();
    uint32_t pb0, pb1;
    ldsm_x2(p_addr + (lane & 7) * kGPRow + ((lane >> 3) & 1) * 16, pb0, pb1);

    // ---- O^T += V^T P^T over the 32 dim tiles (V = the same un-rotated S rows)
#pragma unroll
    for (int mt = 0; mt < 32; ++mt) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(pa + v_lane + step_off(mt), a0, a1, a2, a3);
      mma16816(o[mt], a0, a1, a2, a3, pb0, pb1);
    }
    __syncwarp();
    if (lane == 0 && i + kGStages < n_pages) {   // refill this stage with page i + 5
      fence_proxy_async();
      issue(i + kGStages);
    }
  }
  __syncthreads();
  if (abort_flag && threadIdx.x == 0) {   // after a timeout: wait (bounded) for copies in flight
    const unsigned long long t0 = globaltimer();
    for (int st = 0; st < kGStages; ++st)
      if (issued[st] > 0)
        while (!mbar_try_wait(smem_u32(&full[st]), (issued[st] - 1) & 1) && globaltimer() - t0 < kWaitLimitNs) {
        }
  }
  __syncthreads();   // all stages consumed: reuse them for the warp merge

  float* red_o = reinterpret_cast<float*>(stage_base);   // [warps][8 heads][512]
  if (gq == 0) {
    red_m[warp][2 * cq] = m_run[0];
    red_m[warp][2 * cq + 1] = m_run[1];
    red_l[warp][2 * cq] = l_run[0];
    red_l[warp][2 * cq + 1] = l_run[1];
  }
#pragma unroll
  for (int mt = 0; mt < 32; ++mt) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int d = mt * 16 + gq + 8 * (r >> 1), h = 2 * cq + (r & 1);
      red_o[(warp * 8 + h) * kGD + d] = o[mt][r];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * kGD; idx += 128) {
    const int h = idx / kGD, d = idx % kGD;
    float M = red_m[0][h];
#pragma unroll
    for (int w = 1; w < kGWarps; ++w) M = fmaxf(M, red_m[w][h]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kGWarps; ++w) {
      const float scw = (M == -INFINITY) ? 0.f : exp2f(red_m[w][h] - M);
      L = fmaf(red_l[w][h], scw, L);
      O = fmaf(red_o[(w * 8 + h) * kGD + d], scw, O);
    }
    const size_t s = slot + (size_t)h * p.NC;
    p.ws_o[s * kGD + d] = O;
    if (d == 0) {
      p.ws_ml[s * 2 + 0] = M;
      p.ws_ml[s * 2 + 1] = L;
    }
  }
}

// ---------------------------------------------------------------- ordered merge of the chunks
template <int D>
__global__ void __launch_bounds__(D / 4) decode_merge_kernel(const float* __restrict__ ws_ml,
                                                             const float* __restrict__ ws_o,
                                                             const int32_t* __restrict__ seq_len, int NC, int window,
                                                             int chunk, __nv_bfloat16* out) {
  const int h = blockIdx.x, b = blockIdx.y;
  const int d0 = threadIdx.x * 4;
  const int pos = seq_len[b] - 1;
  __nv_bfloat16* dst = out + ((size_t)b * gridDim.x + h) * D + d0;
  int n = 0;
  if (pos >= 0 && pos < kMaxPos) {
    const int lo = window > 0 ? max(0, pos - window + 1) : 0;
    n = min(NC, pos / chunk - lo / chunk + 1);
  }
  const size_t s0 = ((size_t)b * gridDim.x + h) * NC;
  float M = -INFINITY;
  for (int c = 0; c < n; ++c) M = fmaxf(M, ws_ml[(s0 + c) * 2]);
  float L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (M != -INFINITY) {
    for (int c = 0; c < n; ++c) {
      const float mc = ws_ml[(s0 + c) * 2];
      if (mc == -INFINITY) continue;   // an empty chunk: its output slot was never written
      const float w = exp2f(mc - M);
      L = fmaf(ws_ml[(s0 + c) * 2 + 1], w, L);
      const float4 ov = *reinterpret_cast<const float4*>(ws_o + (s0 + c) * D + d0);
      acc[0] = fmaf(ov.x, w, acc[0]);
      acc[1] = fmaf(ov.y, w, acc[1]);
      acc[2] = fmaf(ov.z, w, acc[2]);
      acc[3] = fmaf(ov.w, w, acc[3]);
    }
  }
  const float inv = (L > 0.f) ? __frcp_rn(L) : 0.f;
  uint2 pk;
  pk.x = pack_bf16(acc[0] * inv, acc[1] * inv);
  pk.y = pack_bf16(acc[2] * inv, acc[3] * inv);
  *reinterpret_cast<uint2*>(dst) = pk;
}

// Chunks a request can span: positions stop below kMaxPos, so a longer page table adds none.
int decode_chunks(bool global, int max_pages, int window) {
  const long long keys = (long long)max_pages * kPage < kMaxPos ? (long long)max_pages * kPage : kMaxPos;
  if (global) return (int)((keys + kDecodeChunkGlobal - 1) / kDecodeChunkGlobal);
  const int by_window = (window - 1) / kDecodeChunkSliding + 2;
  const int by_table = (int)((keys + kDecodeChunkSliding - 1) / kDecodeChunkSliding);
  return by_window < by_table ? by_window : by_table;
}

}  // namespace

size_t decode_workspace_bytes(bool global, int B, int max_pages, int window, int hq) {
  const size_t nc = (size_t)decode_chunks(global, max_pages, window);
  const size_t D = global ? kGD : kSD;
  const size_t ml = ((size_t)B * hq * nc * 2 * sizeof(float) + 255) / 256 * 256;
  return ml + (size_t)B * hq * nc * D * sizeof(float);
}

// A decode step laid out as B one-row prefill chunks: request b's query is row b, at position
// seq_len[b] - 1, and it reads page-table row b. The chunks are listed from the longest context
// down (ties by request index), so that the prefill kernels' fixed round-robin schedule gives
// every cluster a similar share of key tiles; a chunk's arithmetic does not depend on its place in
// the list. Steps of up to kSortedRows requests are sorted (each rank is a count over all of them);
// larger ones keep request order. A request with seq_len < 1 gets no row (and sets kErrPos).
constexpr int kSortedRows = 8192;
__global__ void decode_rows_kernel(const int32_t* seq_len, int B, int32_t* q_start, int32_t* q_len,
                                   int32_t* ctx_start, int32_t* pt_row, uint32_t* err) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int n = seq_len[b];
  int rank = b;
  if (B <= kSortedRows) {
    rank = 0;
    for (int i = 0; i < B; ++i) {
      const int m = __ldg(seq_len + i);
      rank += (m > n || (m == n && i < b)) ? 1 : 0;
    }
  }
  q_start[rank] = b;
  q_len[rank] = n >= 1 ? 1 : 0;
  ctx_start[rank] = n >= 1 ? n - 1 : 0;
  pt_row[rank] = b;
  if (n < 1) set_error(err, kErrPos);
}

cudaError_t launch_decode_rows(const int32_t* seq_len, int B, int32_t* rows, const DeviceState& st, cudaStream_t s) {
  decode_rows_kernel<<<(B + 127) / 128, 128, 0, s>>>(seq_len, B, rows, rows + B, rows + 2 * B, rows + 3 * B, st.err);
  return cudaGetLastError();
}

cudaError_t launch_decode(bool global, const void* q, const int32_t* seq_len, int B, int window, float scale_log2,
                          const PagedCache& cache, void* out, void* ws, const DeviceState& st, cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  DecodeParams p{};
  p.q = (const __nv_bfloat16*)q;
  p.seq_len = seq_len;
  p.B = B;
  p.window = global ? 0 : window;
  p.scale_log2 = scale_log2;
  p.cache = cache;
  p.NC = decode_chunks(global, cache.max_pages, window);
  const size_t ml = ((size_t)B * cache.hq * p.NC * 2 * sizeof(float) + 255) / 256 * 256;
  p.ws_ml = (float*)ws;
  p.ws_o = (float*)((uint8_t*)ws + ml);
  p.err = st.err;
  p.wait_ns = wait_limit_ns();
  if (global) {
    p.tb = st.global;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
      cudaError_t e = cudaFuncSetAttribute(decode_global_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmem);
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
    decode_global_kernel<<<dim3(p.NC, cache.hkv, B), 128, kGSmem, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_merge_kernel<kGD><<<dim3(cache.hq, B), kGD / 4, 0, s>>>(p.ws_ml, p.ws_o, seq_len, p.NC, 0,
                                                                    kDecodeChunkGlobal, (__nv_bfloat16*)out);
  } else {
    p.tb = st.sliding;
    static bool attr_set_s[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set_s[dev]) {
      cudaError_t e = cudaFuncSetAttribute(decode_sliding_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSSmem);
      if (e != cudaSuccess) return e;
      attr_set_s[dev] = true;
    }
    decode_sliding_kernel<<<dim3(p.NC, cache.hkv, B), 128, kSSmem, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_merge_kernel<kSD><<<dim3(cache.hq, B), kSD / 4, 0, s>>>(p.ws_ml, p.ws_o, seq_len, p.NC, window,
                                                                    kDecodeChunkSliding, (__nv_bfloat16*)out);
  }
  return cudaGetLastError();
}

}  // namespace g4
