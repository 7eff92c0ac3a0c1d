// Paged decode: one query token per request against its cached keys, split into fixed key
// chunks aligned to absolute position 0 and merged in ascending chunk order.
//
// The RL-Kernel RFC "[RFC][Gemma-4-31B-it] WS1/WS2 kernel roadmap", section 4 rule 3, forbids
// split-KV unless the split and merge tree is fixed by the contract. Here the split is fixed:
// chunk c holds keys [C*c, C*c + C) (C = 256 sliding, 1024 global), whatever the batch, and
// inside a chunk the pages go round-robin to four warps whose states merge in warp order.
// Every number a request gets depends only on its own position, window and data.
//
// Sliding layers (2 query heads per KV head, 2 flop per byte) run on CUDA cores. Global layers
// (8 query heads per KV head, K==V, 16 flop per byte) run on warp-level bf16 MMA: S^T = K q^T,
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
};

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ---------------------------------------------------------------- sliding: D 256, Hkv 16, G 2
constexpr int kSD = kSlidingD;

__global__ void __launch_bounds__(128) decode_sliding_kernel(DecodeParams p) {
  const int cr = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ float red_m[4][2], red_l[4][2];
  __shared__ float red_o[4][2][kSD];

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
  const int32_t* pt = p.cache.page_table + (size_t)b * p.cache.max_pages;
  bool bad = false;
  for (int i = pg0 + (int)threadIdx.x; i <= pg1; i += 128) {
    const int ph = pt[i];
    bad |= (ph < 0 || ph >= p.cache.num_pages);
  }
  const size_t slot = (((size_t)b * kSlidingHq + 2 * g) * p.NC + cr);
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

  // Roped query of both heads; lane owns dims 8*lane .. 8*lane+7 (pair t = 8*(lane%16) + i).
  float q0[8], q1[8];
  {
    const int t0 = (lane & 15) * 8;
    const bool hi = lane >= 16;
    const __nv_bfloat16* qb = p.q + ((size_t)b * kSlidingHq + 2 * g) * kSD;
    float2 cs[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) cs[i] = rope_cs(p.tb, t0 + i, pos);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const uint4 a4 = *reinterpret_cast<const uint4*>(qb + hh * kSD + t0);
      const uint4 b4 = *reinterpret_cast<const uint4*>(qb + hh * kSD + kSD / 2 + t0);
      const uint32_t* aw = reinterpret_cast<const uint32_t*>(&a4);
      const uint32_t* bw = reinterpret_cast<const uint32_t*>(&b4);
      float* qd = hh ? q1 : q0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float x = (i & 1) ? bf16_hi(aw[i >> 1]) : bf16_lo(aw[i >> 1]);
        float y = (i & 1) ? bf16_hi(bw[i >> 1]) : bf16_lo(bw[i >> 1]);
        rope_pair(x, y, cs[i]);
        qd[i] = round_bf16(hi ? y : x);   // declared cast: roped q in bf16
      }
    }
  }

  float m_run0 = -INFINITY, m_run1 = -INFINITY, l_run0 = 0.f, l_run1 = 0.f;
  float o0[8], o1[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) o0[i] = o1[i] = 0.f;

  const __nv_bfloat16* kc = (const __nv_bfloat16*)p.cache.k;
  const __nv_bfloat16* vc = (const __nv_bfloat16*)p.cache.v;
  for (int pg = pg0 + warp; pg <= pg1; pg += 4) {
    const size_t base = (((size_t)pt[pg] * kSlidingHkv + g) * kPage) * kSD;   // page-head block
    uint4 kr[16], vr[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) kr[j] = ldg_nc(kc + base + tiled_offset(j, lane * 8, kSD));
#pragma unroll
    for (int j = 0; j < 16; ++j) vr[j] = ldg_nc(vc + base + tiled_offset(j, lane * 8, kSD));

    // Partial dot products over this lane's 8 dims: index 2*key + head.
    float part[32];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t* w = reinterpret_cast<const uint32_t*>(&kr[j]);
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float kv = (i & 1) ? bf16_hi(w[i >> 1]) : bf16_lo(w[i >> 1]);
        s0 = fmaf(q0[i], kv, s0);
        s1 = fmaf(q1[i], kv, s1);
      }
      part[2 * j] = s0;
      part[2 * j + 1] = s1;
    }
    // Transposing reduction: afterwards lane l holds the full dot of index l.
#pragma unroll
    for (int m = 16, n = 32; m >= 1; m >>= 1, n >>= 1) {
      const bool upper = (lane & m) != 0;
#pragma unroll
      for (int i = 0; i < n / 2; ++i) {
        const float send = upper ? part[i] : part[i + n / 2];
        const float keep = upper ? part[i + n / 2] : part[i];
        part[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
      }
    }
    const int key = pg * kPage + (lane >> 1);
    const bool valid = key >= k_begin && key <= k_end;
    const float x = valid ? part[0] * p.scale_log2 : -INFINITY;

    float mt = x;
#pragma unroll
    for (int m = 2; m <= 16; m <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, m));
    const float mt_o = __shfl_xor_sync(0xffffffffu, mt, 1);
    const float mt0 = (lane & 1) ? mt_o : mt, mt1 = (lane & 1) ? mt : mt_o;
    const float mn0 = fmaxf(m_run0, mt0), mn1 = fmaxf(m_run1, mt1);
    if (mn0 > m_run0 + kLazyRescale) {
      const float a = exp2f(m_run0 - mn0);
      m_run0 = mn0;
      l_run0 *= a;
#pragma unroll
      for (int i = 0; i < 8; ++i) o0[i] *= a;
    }
    if (mn1 > m_run1 + kLazyRescale) {
      const float a = exp2f(m_run1 - mn1);
      m_run1 = mn1;
      l_run1 *= a;
#pragma unroll
      for (int i = 0; i < 8; ++i) o1[i] *= a;
    }
    const float pv = valid ? exp2f(x - ((lane & 1) ? m_run1 : m_run0)) : 0.f;
    float ls = pv;
#pragma unroll
    for (int m = 2; m <= 16; m <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, m);
    const float ls_o = __shfl_xor_sync(0xffffffffu, ls, 1);
    l_run0 += (lane & 1) ? ls_o : ls;
    l_run1 += (lane & 1) ? ls : ls_o;

#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float p0 = __shfl_sync(0xffffffffu, pv, 2 * j);
      const float p1 = __shfl_sync(0xffffffffu, pv, 2 * j + 1);
      const int kj = pg * kPage + j;
      if (kj >= k_begin && kj <= k_end) {   // stale slots may hold NaN: never multiply them
        const uint32_t* w = reinterpret_cast<const uint32_t*>(&vr[j]);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float vv = (i & 1) ? bf16_hi(w[i >> 1]) : bf16_lo(w[i >> 1]);
          o0[i] = fmaf(p0, vv, o0[i]);
          o1[i] = fmaf(p1, vv, o1[i]);
        }
      }
    }
  }

  if (lane == 0) {
    red_m[warp][0] = m_run0;
    red_m[warp][1] = m_run1;
    red_l[warp][0] = l_run0;
    red_l[warp][1] = l_run1;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    red_o[warp][0][lane * 8 + i] = o0[i];
    red_o[warp][1][lane * 8 + i] = o1[i];
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
      O = fmaf(red_o[w][hh][d], sc, O);
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
constexpr int kGStages = 2;                      // pages in flight per warp
constexpr int kGSBytes = kPage * kGD * 2;        // one tiled page-head block of S: 16 KB
constexpr int kGRotBytes = kRotPageElems * 2;    // its k_rot block: 4 KB
constexpr int kGStageBytes = kGSBytes + kGRotBytes;
constexpr int kGRow = kGD * 2 + 16;              // padded query row: ldmatrix rows hit distinct banks
constexpr int kGQBytes = 8 * kGRow;              // the 8 roped query heads
constexpr int kGPRow = 48;                       // P^T staging row (8 heads x 16 keys bf16, padded)
constexpr int kGSmem = kGWarps * kGStages * kGStageBytes + kGQBytes + kGWarps * 8 * kGPRow + 256;

__global__ void __launch_bounds__(128, 1) decode_global_kernel(DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stage_base = smem;
  uint8_t* q_s = smem + kGWarps * kGStages * kGStageBytes;
  uint8_t* p_s_all = q_s + kGQBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(p_s_all + kGWarps * 8 * kGPRow);   // [warps][stages]
  __shared__ int abort_flag;
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
  const size_t slot = ((size_t)b * kGlobalHq + 8 * g) * p.NC + c;   // head 8g + j adds j * NC

  bool bad = false;
  for (int i = pg0 + (int)threadIdx.x; i <= pg1; i += 128) {
    const int ph = pt[i];
    bad |= (ph < 0 || ph >= p.cache.num_pages);
  }
  if (threadIdx.x == 0) abort_flag = 0;
  if (threadIdx.x < kGWarps * kGStages) mbar_init(&bars[threadIdx.x], 1);
  fence_mbar_init();
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) {
      set_error(p.err, kErrPage);
      for (int j = 0; j < 8; ++j) {
        p.ws_ml[(slot + (size_t)j * p.NC) * 2 + 0] = -INFINITY;
        p.ws_ml[(slot + (size_t)j * p.NC) * 2 + 1] = 0.f;
      }
    }
    return;
  }

  // This warp's pages: pg0 + warp + 4*i.
  const int n_mine = (pg1 - pg0 - warp) >= 0 ? (pg1 - pg0 - warp) / kGWarps + 1 : 0;
  uint8_t* my_stages = stage_base + warp * kGStages * kGStageBytes;
  uint64_t* my_bars = bars + warp * kGStages;
  const __nv_bfloat16* sc = (const __nv_bfloat16*)p.cache.k;
  const __nv_bfloat16* rc = (const __nv_bfloat16*)p.cache.krot;
  auto issue = [&](int i) {   // lane 0 only
    const int pg = pg0 + warp + kGWarps * i;
    const size_t blk = (size_t)pt[pg] * kGlobalHkv + g;
    uint8_t* dst = my_stages + (i % kGStages) * kGStageBytes;
    uint64_t* bar = &my_bars[i % kGStages];
    mbar_arrive_expect_tx(bar, kGStageBytes);
    bulk_g2s(dst, sc + blk * kPage * kGD, kGSBytes, bar);
    bulk_g2s(dst + kGSBytes, rc + blk * kRotPageElems, kGRotBytes, bar);
  };
  int n_issued = 0, n_done = 0;   // lane 0's view of this warp's copies
  if (lane == 0)
    for (; n_issued < min(kGStages, n_mine); ++n_issued) issue(n_issued);

  // Stage the 8 roped query heads (bf16) while the first pages are in flight.
  {
    const __nv_bfloat16* qb = p.q + ((size_t)b * kGlobalHq + 8 * g) * kGD;
    for (int idx = threadIdx.x; idx < 8 * (kGD / 2); idx += 128) {
      const int h = idx / (kGD / 2), t = idx % (kGD / 2);
      float x = bf16_to_f(qb[h * kGD + t]), y = bf16_to_f(qb[h * kGD + t + kGD / 2]);
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

  for (int i = 0; i < n_mine; ++i) {
    const int st = i % kGStages;
    if (!mbar_wait(&my_bars[st], (i / kGStages) & 1, &abort_flag, p.err)) break;
    n_done = i + 1;
    uint8_t* page = my_stages + st * kGStageBytes;
    const int key0 = (pg0 + warp + kGWarps * i) * kPage;
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
    if (lane == 0 && i + kGStages < n_mine) {
      fence_proxy_async();
      issue(i + kGStages);
      n_issued = i + kGStages + 1;
    }
  }
  // After a timeout, wait (bounded) for this warp's copies still in flight before leaving.
  if (abort_flag && lane == 0) {
    const unsigned long long t0 = globaltimer();
    for (int i = n_done; i < n_issued; ++i) {
      while (!mbar_try_wait(smem_u32(&my_bars[i % kGStages]), (i / kGStages) & 1) &&
             globaltimer() - t0 < kWaitLimitNs) {
      }
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
  for (int idx = threadIdx.x; idx < 8 * kGD; idx += 128) {
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

size_t decode_workspace_bytes(bool global, int B, int max_pages, int window) {
  const size_t nc = (size_t)decode_chunks(global, max_pages, window);
  const size_t D = global ? kGD : kSD;
  const size_t ml = ((size_t)B * 32 * nc * 2 * sizeof(float) + 255) / 256 * 256;
  return ml + (size_t)B * 32 * nc * D * sizeof(float);
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
  const size_t ml = ((size_t)B * 32 * p.NC * 2 * sizeof(float) + 255) / 256 * 256;
  p.ws_ml = (float*)ws;
  p.ws_o = (float*)((uint8_t*)ws + ml);
  p.err = st.err;
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
    decode_global_kernel<<<dim3(p.NC, kGlobalHkv, B), 128, kGSmem, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_merge_kernel<kGD><<<dim3(kGlobalHq, B), kGD / 4, 0, s>>>(p.ws_ml, p.ws_o, seq_len, p.NC, 0,
                                                                    kDecodeChunkGlobal, (__nv_bfloat16*)out);
  } else {
    p.tb = st.sliding;
    decode_sliding_kernel<<<dim3(p.NC, kSlidingHkv, B), 128, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_merge_kernel<kSD><<<dim3(kSlidingHq, B), kSD / 4, 0, s>>>(p.ws_ml, p.ws_o, seq_len, p.NC, window,
                                                                    kDecodeChunkSliding, (__nv_bfloat16*)out);
  }
  return cudaGetLastError();
}

}  // namespace g4
