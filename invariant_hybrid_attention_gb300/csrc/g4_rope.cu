// RoPE / p-RoPE tables and the elementwise kernels: g4attn_rope_apply and the paged KV-cache
// append of prefill and decode.
//
// RoPE as the RL-Kernel RFC "[RFC][Gemma-4-31B-it] WS1/WS2 kernel roadmap" lists it (section 2
// fingerprint table; section 5 rows sliding_rope_d256 and global_proportional_p_rope):
// standard RoPE with theta 1e4 on the 256-dim sliding heads; proportional p-RoPE with
// partial factor 0.25 and theta 1e6 on the 512-dim global heads. Reading used here: element t
// pairs with t + D/2, pair t turns by pos * theta^(-2t/D) (frequency denominator = full D),
// and only pairs t < R turn (R = 128 sliding, 64 global); the rest are copied bit for bit.
//
// Angles: pos * f_t needs more than fp32 at large positions (about 0.016 rad of error at
// pos 2^18), so the tables hold (cos, sin) of 256*c*f_t, 16*a*f_t and b*f_t, computed in fp64
// on the host, and a lookup combines them by the angle-addition formula in fp32. The tables
// are static device arrays: the library allocates no device memory.
#include <math.h>

#include <atomic>
#include <mutex>
#include <type_traits>
#include <vector>

#include "g4_internal.h"

namespace g4 {

static __device__ float2 g_rope_sliding_coarse[kSlidingR * kRopeCoarse];
static __device__ float2 g_rope_sliding_mid[kSlidingR * kRopeMid];
static __device__ float2 g_rope_sliding_fine[kSlidingR * kRopeFine];
static __device__ float2 g_rope_global_coarse[kGlobalR * kRopeCoarse];
static __device__ float2 g_rope_global_mid[kGlobalR * kRopeMid];
static __device__ float2 g_rope_global_fine[kGlobalR * kRopeFine];
static __device__ float2 g_rope_sliding_coarse_t[kRopeCoarse * kSlidingR];
static __device__ float2 g_rope_sliding_mid_t[kRopeMid * kSlidingR];
static __device__ float2 g_rope_sliding_fine_t[kRopeFine * kSlidingR];
static __device__ float2 g_rope_global_coarse_t[kRopeCoarse * kGlobalR];
static __device__ float2 g_rope_global_mid_t[kRopeMid * kGlobalR];
static __device__ float2 g_rope_global_fine_t[kRopeFine * kGlobalR];
static __device__ uint32_t g_error_word;

namespace {

struct HostTables {
  std::vector<float2> coarse, mid, fine;
  std::vector<float2> coarse_t, mid_t, fine_t;   // the same values, entry-major
};

std::vector<float2> transpose(const std::vector<float2>& a, int rows, int cols) {
  std::vector<float2> t(a.size());
  for (int i = 0; i < rows; ++i)
    for (int j = 0; j < cols; ++j) t[(size_t)j * rows + i] = a[(size_t)i * cols + j];
  return t;
}

void build_tables(int D, int R, double theta, HostTables& h) {
  h.coarse.resize((size_t)R * kRopeCoarse);
  h.mid.resize((size_t)R * kRopeMid);
  h.fine.resize((size_t)R * kRopeFine);
  auto cs = [](double a) { return make_float2((float)cos(a), (float)sin(a)); };
  for (int t = 0; t < R; ++t) {
    const double f = pow(theta, -2.0 * t / (double)D);
    for (int c = 0; c < kRopeCoarse; ++c) h.coarse[(size_t)t * kRopeCoarse + c] = cs((256.0 * c) * f);
    for (int a = 0; a < kRopeMid; ++a) h.mid[(size_t)t * kRopeMid + a] = cs((16.0 * a) * f);
    for (int b = 0; b < kRopeFine; ++b) h.fine[(size_t)t * kRopeFine + b] = cs((double)b * f);
  }
  h.coarse_t = transpose(h.coarse, R, kRopeCoarse);
  h.mid_t = transpose(h.mid, R, kRopeMid);
  h.fine_t = transpose(h.fine, R, kRopeFine);
}

constexpr int kMaxDevices = 64;
std::atomic<unsigned long long> g_wait_ns{kWaitLimitNs};
std::mutex g_state_mutex;
bool g_state_ready[kMaxDevices];
DeviceState g_state[kMaxDevices];

}  // namespace

unsigned long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
void set_wait_limit_ns(unsigned long long ns) { g_wait_ns.store(ns, std::memory_order_relaxed); }

cudaError_t device_state(DeviceState* st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_state_mutex);
  if (!g_state_ready[dev]) {
    static HostTables hs, hg;
    if (hs.coarse.empty()) {
      build_tables(kSlidingD, kSlidingR, 1.0e4, hs);
      build_tables(kGlobalD, kGlobalR, 1.0e6, hg);
    }
    DeviceState s{};
    void* p = nullptr;
#define G4_UPLOAD(sym, vec)                                                                   \
  if ((e = cudaMemcpyToSymbol(sym, (vec).data(), (vec).size() * sizeof(float2))) != cudaSuccess) return e
#define G4_ADDR(sym, dst)                                                   \
  if ((e = cudaGetSymbolAddress(&p, sym)) != cudaSuccess) return e;         \
  dst = (const float2*)p
    G4_UPLOAD(g_rope_sliding_coarse, hs.coarse);
    G4_UPLOAD(g_rope_sliding_mid, hs.mid);
    G4_UPLOAD(g_rope_sliding_fine, hs.fine);
    G4_UPLOAD(g_rope_global_coarse, hg.coarse);
    G4_UPLOAD(g_rope_global_mid, hg.mid);
    G4_UPLOAD(g_rope_global_fine, hg.fine);
    G4_UPLOAD(g_rope_sliding_coarse_t, hs.coarse_t);
    G4_UPLOAD(g_rope_sliding_mid_t, hs.mid_t);
    G4_UPLOAD(g_rope_sliding_fine_t, hs.fine_t);
    G4_UPLOAD(g_rope_global_coarse_t, hg.coarse_t);
    G4_UPLOAD(g_rope_global_mid_t, hg.mid_t);
    G4_UPLOAD(g_rope_global_fine_t, hg.fine_t);
    G4_ADDR(g_rope_sliding_coarse, s.sliding.coarse);
    G4_ADDR(g_rope_sliding_mid, s.sliding.mid);
    G4_ADDR(g_rope_sliding_fine, s.sliding.fine);
    G4_ADDR(g_rope_global_coarse, s.global.coarse);
    G4_ADDR(g_rope_global_mid, s.global.mid);
    G4_ADDR(g_rope_global_fine, s.global.fine);
    G4_ADDR(g_rope_sliding_coarse_t, s.sliding.coarse_t);
    G4_ADDR(g_rope_sliding_mid_t, s.sliding.mid_t);
    G4_ADDR(g_rope_sliding_fine_t, s.sliding.fine_t);
    G4_ADDR(g_rope_global_coarse_t, s.global.coarse_t);
    G4_ADDR(g_rope_global_mid_t, s.global.mid_t);
    G4_ADDR(g_rope_global_fine_t, s.global.fine_t);
#undef G4_UPLOAD
#undef G4_ADDR
    const uint32_t zero = 0;
    if ((e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero))) != cudaSuccess) return e;
    if ((e = cudaGetSymbolAddress(&p, g_error_word)) != cudaSuccess) return e;
    s.err = (uint32_t*)p;
    g_state[dev] = s;
    g_state_ready[dev] = true;
  }
  *st = g_state[dev];
  return cudaSuccess;
}

// ---- one D-vector per warp ----------------------------------------------------------------------
// Lane l owns pairs t = l*P .. l*P+P-1 (P = D/64), i.e. P contiguous elements of each half.
// `Dst` maps a dim to its place: contiguous rows (rope_apply) or a key row of a tiled page.
struct RowDst {
  __nv_bfloat16* p;
  __device__ __forceinline__ __nv_bfloat16* at(int d) const { return p + d; }
};
template <int D>
struct PageDst {   // key slot j of a page-head block (see tiled_offset)
  __nv_bfloat16* block;
  int j;
  __device__ __forceinline__ __nv_bfloat16* at(int d) const { return block + tiled_offset(j, d, D); }
};

struct VDst {   // key slot j of a sliding V page-head block (see tiled_offset_v256)
  __nv_bfloat16* block;
  int j;
  __device__ __forceinline__ __nv_bfloat16* at(int d) const { return block + tiled_offset_v256(j, d); }
};

struct RotDst {   // key slot j of a rotated-column side page (see rot_offset); other dims dropped
  __nv_bfloat16* block;
  int j;
  __device__ __forceinline__ __nv_bfloat16* at(int d) const { return block + rot_offset(j, d); }
};

template <class Dst>
struct RotatedOnly {
  static constexpr bool value = false;
};
template <>
struct RotatedOnly<RotDst> {
  static constexpr bool value = true;
};

// (cos, sin) of this lane's P pairs at position pos (lanes whose pairs do not turn skip it). One
// row's vectors all turn by the same angles, so a row computes them once for all its heads.
template <int D, int R>
__device__ __forceinline__ void rope_cs_lane(const RopeTables& tb, int pos, float2 (&cs)[D / 64]) {
  constexpr int P = D / 64;
  const int t0 = (threadIdx.x & 31) * P;
  if (t0 < R) {
#pragma unroll
    for (int i = 0; i < P; ++i) cs[i] = rope_cs(tb, t0 + i, pos);
  }
}

template <int D, int R, class Dst>
__device__ __forceinline__ void rope_vec_warp_cs(const __nv_bfloat16* __restrict__ src, const Dst& dst,
                                                 const float2 (&cs)[D / 64]) {
  constexpr int P = D / 64;                    // 4 (D=256) or 8 (D=512)
  constexpr int half = D / 2;
  const int lane = threadIdx.x & 31;
  const int t0 = lane * P;
  using Vec = typename std::conditional<P == 8, uint4, uint2>::type;
  Vec lo = *reinterpret_cast<const Vec*>(src + t0);
  Vec hi = *reinterpret_cast<const Vec*>(src + half + t0);
  if (t0 < R) {                                 // R is a multiple of P: whole lanes turn or not
    uint32_t* lw = reinterpret_cast<uint32_t*>(&lo);
    uint32_t* hw = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
    for (int w = 0; w < P / 2; ++w) {
      float a0 = bf16_lo(lw[w]), a1 = bf16_hi(lw[w]);
      float b0 = bf16_lo(hw[w]), b1 = bf16_hi(hw[w]);
      rope_pair(a0, b0, cs[2 * w]);
      rope_pair(a1, b1, cs[2 * w + 1]);
      lw[w] = pack_bf16(a0, a1);
      hw[w] = pack_bf16(b0, b1);
    }
  }
  // P elements never cross an 8-dim group, so each half is one contiguous store either way.
  if (RotatedOnly<Dst>::value && t0 >= R) return;
  *reinterpret_cast<Vec*>(dst.at(t0)) = lo;
  *reinterpret_cast<Vec*>(dst.at(half + t0)) = hi;
}

template <int D, int R, class Dst>
__device__ __forceinline__ void rope_vec_warp(const __nv_bfloat16* __restrict__ src, const Dst& dst, int pos,
                                              const RopeTables& tb) {
  float2 cs[D / 64];
  rope_cs_lane<D, R>(tb, pos, cs);
  rope_vec_warp_cs<D, R>(src, dst, cs);
}

// The same rotation with 8 pairs per lane, so that every load and store is 16 bytes, one
// core-matrix row of a tiled page: D/16 lanes per vector, 32/(D/16) vectors per warp (two when
// D = 256). Lane l handles pairs (l % (D/16)) * 8 .. + 7 of vector l / (D/16); the caller passes
// that vector's source and destination. cs comes from rope_cs_lane8.
template <int D, int R>
__device__ __forceinline__ void rope_cs_lane8(const RopeTables& tb, int pos, float2 (&cs)[8]) {
  const int t0 = ((threadIdx.x & 31) % (D / 16)) * 8;
  if (t0 < R) {
#pragma unroll
    for (int i = 0; i < 8; ++i) cs[i] = rope_cs(tb, t0 + i, pos);
  }
}
template <int D, int R, class Dst>
__device__ __forceinline__ void rope_vec8_cs(const __nv_bfloat16* __restrict__ src, const Dst& dst,
                                             const float2 (&cs)[8]) {
  constexpr int half = D / 2;
  const int t0 = ((threadIdx.x & 31) % (D / 16)) * 8;
  uint4 lo = *reinterpret_cast<const uint4*>(src + t0);
  uint4 hi = *reinterpret_cast<const uint4*>(src + half + t0);
  if (t0 < R) {
    uint32_t* lw = reinterpret_cast<uint32_t*>(&lo);
    uint32_t* hw = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      float a0 = bf16_lo(lw[w]), a1 = bf16_hi(lw[w]);
      float b0 = bf16_lo(hw[w]), b1 = bf16_hi(hw[w]);
      rope_pair(a0, b0, cs[2 * w]);
      rope_pair(a1, b1, cs[2 * w + 1]);
      lw[w] = pack_bf16(a0, a1);
      hw[w] = pack_bf16(b0, b1);
    }
  }
  if (RotatedOnly<Dst>::value && t0 >= R) return;
  *reinterpret_cast<uint4*>(dst.at(t0)) = lo;
  *reinterpret_cast<uint4*>(dst.at(half + t0)) = hi;
}

template <int D, class Dst>
__device__ __forceinline__ void copy_vec_warp(const __nv_bfloat16* __restrict__ src, const Dst& dst) {
  constexpr int E = D / 32;                    // elements per lane: 8 or 16
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < E / 8; ++i) {
    const int d = (i * 32 + lane) * 8;
    *reinterpret_cast<uint4*>(dst.at(d)) = *reinterpret_cast<const uint4*>(src + d);
  }
}

// ---- optional per-head RMS norms, before the rotation --------------------------------------------
// Reading of the RFC work item qk_rmsnorm_d256_d512 and of TensorFold's tf_qk_rows_once (which
// "can norm v by a unit RMS norm"): a head vector x of D dims becomes (x * inv) * w with
// inv = 1/sqrt(mean(x^2) + eps), in fp32, before the rotation and the one declared bf16 cast; w
// is a per-dim weight for queries and keys, and 1 for the unit norm of values. On a K==V layer the
// stored S becomes n(S), which is V; the k_rot side pages hold RoPE(w_k n(S)); and the staged
// queries carry w_k on their un-rotated dims, where the attention kernels read K from the stored
// S: q . (w_k n(S)) = (q w_k) . n(S). The sum of squares is a fixed-order sum over the lane's 16
// elements followed by a butterfly over the vector's lanes; additions commute, so every lane gets
// the same bits, and a vector's result depends on that vector alone.
template <int D>
__device__ __forceinline__ void lane_weights(const __nv_bfloat16* w, float (&out)[16]) {
  const int t0 = ((threadIdx.x & 31) % (D / 16)) * 8;
  if (w == nullptr) {
#pragma unroll
    for (int i = 0; i < 16; ++i) out[i] = 1.f;
    return;
  }
  const uint4 lo = __ldg(reinterpret_cast<const uint4*>(w + t0));
  const uint4 hi = __ldg(reinterpret_cast<const uint4*>(w + D / 2 + t0));
  const uint32_t lw[4] = {lo.x, lo.y, lo.z, lo.w}, hw[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    out[2 * i] = bf16_lo(lw[i]);
    out[2 * i + 1] = bf16_hi(lw[i]);
    out[8 + 2 * i] = bf16_lo(hw[i]);
    out[8 + 2 * i + 1] = bf16_hi(hw[i]);
  }
}

// rope_vec8_cs with the norm: `norm` turns it on (weight w, all ones for a unit norm), pairs
// t < R rotate, and lanes whose pairs start at or after fold_from multiply by `fold` (w_k on the
// un-rotated dims of a K==V layer's queries; nullptr: no fold).
template <int D, int R, class Dst>
__device__ __forceinline__ void vec8_normed(const __nv_bfloat16* __restrict__ src, const Dst& dst,
                                            const float2 (&cs)[8], bool norm, float eps, const float (&w)[16],
                                            const float* fold, int fold_from) {
  constexpr int half = D / 2, LPV = D / 16;
  const int t0 = ((threadIdx.x & 31) % LPV) * 8;
  const uint4 lo = *reinterpret_cast<const uint4*>(src + t0);
  const uint4 hi = *reinterpret_cast<const uint4*>(src + half + t0);
  const uint32_t lw[4] = {lo.x, lo.y, lo.z, lo.w}, hw[4] = {hi.x, hi.y, hi.z, hi.w};
  float a[8], b[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a[2 * i] = bf16_lo(lw[i]);
    a[2 * i + 1] = bf16_hi(lw[i]);
    b[2 * i] = bf16_lo(hw[i]);
    b[2 * i + 1] = bf16_hi(hw[i]);
  }
  if (norm) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(a[i], a[i], ss);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(b[i], b[i], ss);
#pragma unroll
    for (int o = 1; o < LPV; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = __frsqrt_rn(fmaf(ss, 1.0f / (float)D, eps));   // ss / D is exact: D is a power of 2
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      a[i] = (a[i] * inv) * w[i];
      b[i] = (b[i] * inv) * w[8 + i];
    }
  }
  if (t0 < R) {
#pragma unroll
    for (int i = 0; i < 8; ++i) rope_pair(a[i], b[i], cs[i]);
  } else if (fold != nullptr && t0 >= fold_from) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      a[i] *= fold[i];
      b[i] *= fold[8 + i];
    }
  }
  if (RotatedOnly<Dst>::value && t0 >= R) return;
  uint4 olo, ohi;
  olo.x = pack_bf16(a[0], a[1]);
  olo.y = pack_bf16(a[2], a[3]);
  olo.z = pack_bf16(a[4], a[5]);
  olo.w = pack_bf16(a[6], a[7]);
  ohi.x = pack_bf16(b[0], b[1]);
  ohi.y = pack_bf16(b[2], b[3]);
  ohi.z = pack_bf16(b[4], b[5]);
  ohi.w = pack_bf16(b[6], b[7]);
  *reinterpret_cast<uint4*>(dst.at(t0)) = olo;
  *reinterpret_cast<uint4*>(dst.at(half + t0)) = ohi;
}

template <int D, int R>
__global__ void __launch_bounds__(256) rope_apply_kernel(const __nv_bfloat16* __restrict__ x,
                                                         const int32_t* __restrict__ pos, int T, int H,
                                                         __nv_bfloat16* out, RopeTables tb, uint32_t* err) {
  const long long vec = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (vec >= (long long)T * H) return;
  const int row = (int)(vec / H);
  const int p = pos[row];
  if (p < 0 || p >= kMaxPos) {
    if ((threadIdx.x & 31) == 0) set_error(err, kErrPos);
    return;
  }
  rope_vec_warp<D, R>(x + vec * D, RowDst{out + vec * D}, p, tb);
}

cudaError_t launch_rope_apply(bool global, const void* x, const int32_t* pos, int T, int H, void* out,
                              const DeviceState& st, cudaStream_t s) {
  const long long vecs = (long long)T * H;
  if (vecs == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((vecs + 7) / 8);
  if (global)
    rope_apply_kernel<kGlobalD, kGlobalR><<<blocks, 256, 0, s>>>((const __nv_bfloat16*)x, pos, T, H,
                                                                  (__nv_bfloat16*)out, st.global, st.err);
  else
    rope_apply_kernel<kSlidingD, kSlidingR><<<blocks, 256, 0, s>>>((const __nv_bfloat16*)x, pos, T, H,
                                                                    (__nv_bfloat16*)out, st.sliding, st.err);
  return cudaGetLastError();
}

// ---- paged KV append ----------------------------------------------------------------------------
// Writes one token's Hkv vectors into its page slot: sliding K' = bf16(RoPE(k)) and V as given;
// global S as given (K==V: the one stored projection, rotated only where it is read as K).
// cs: the lane's (cos, sin) at the token's position (rope_cs_lane); pos is in range.
template <int D, int R, bool SHARED, bool NORM>
__device__ __forceinline__ void append_token_cs(const __nv_bfloat16* k_row, const __nv_bfloat16* v_row, int b, int pos,
                                                const PagedCache& c, const float2 (&cs)[8], uint32_t* err,
                                                const NormArgs& nm, const float (&wk)[16], int g_begin, int g_end) {
  const int HKV = c.hkv;
  constexpr int VPW = 32 / (D / 16);   // vectors per warp instruction of rope_vec8_cs
  const int lane = threadIdx.x & 31;
  const int phys = c.page_table[(size_t)b * c.max_pages + (pos >> 4)];
  if (phys < 0 || phys >= c.num_pages) {
    if (lane == 0) set_error(err, kErrPage);
    return;
  }
  const int j = pos & 15;
  if (NORM) {   // the normed path: K' (or k_rot) from w_k n(k), V (or S) as n(v) when asked
    float ones[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) ones[i] = 1.f;
#pragma unroll 1
    for (int g0 = g_begin; g0 < g_end; g0 += VPW) {
      const int g = g0 + lane / (D / 16);
      const size_t blk = ((size_t)phys * HKV + g) * kPage * D;
      const __nv_bfloat16* kg = k_row + (size_t)g * D;
      if (SHARED) {
        vec8_normed<D, R>(kg, RotDst{(__nv_bfloat16*)c.krot + ((size_t)phys * HKV + g) * kRotPageElems, j}, cs,
                          nm.wk != nullptr, nm.eps, wk, nullptr, 0);
        if (nm.v_norm)
          vec8_normed<D, 0>(kg, PageDst<D>{(__nv_bfloat16*)c.k + blk, j}, cs, true, nm.eps, ones, nullptr, 0);
      } else {
        vec8_normed<D, R>(kg, PageDst<D>{(__nv_bfloat16*)c.k + blk, j}, cs, nm.wk != nullptr, nm.eps, wk, nullptr, 0);
        if (nm.v_norm)
          vec8_normed<D, 0>(v_row + (size_t)g * D, VDst{(__nv_bfloat16*)c.v + blk, j}, cs, true, nm.eps, ones,
                            nullptr, 0);
      }
      if (!nm.v_norm) {
#pragma unroll
        for (int gv = g0; gv < g0 + VPW; ++gv) {
          const size_t blkv = ((size_t)phys * HKV + gv) * kPage * D;
          if (SHARED)
            copy_vec_warp<D>(k_row + (size_t)gv * D, PageDst<D>{(__nv_bfloat16*)c.k + blkv, j});
          else
            copy_vec_warp<D>(v_row + (size_t)gv * D, VDst{(__nv_bfloat16*)c.v + blkv, j});
        }
      }
    }
    return;
  }
#pragma unroll 2
  for (int g0 = g_begin; g0 < g_end; g0 += VPW) {
    const int g = g0 + lane / (D / 16);   // this lane's KV head for the rotation
    const size_t blk = ((size_t)phys * HKV + g) * kPage * D;   // page-head block
    if (SHARED) {
      // The rotated columns once more, roped (the K side of K==V where it differs from S).
      rope_vec8_cs<D, R>(k_row + (size_t)g * D,
                         RotDst{(__nv_bfloat16*)c.krot + ((size_t)phys * HKV + g) * kRotPageElems, j}, cs);
    } else {
      rope_vec8_cs<D, R>(k_row + (size_t)g * D, PageDst<D>{(__nv_bfloat16*)c.k + blk, j}, cs);
    }
#pragma unroll
    for (int gv = g0; gv < g0 + VPW; ++gv) {   // S (global) or V (sliding) as given, a warp per vector
      const size_t blkv = ((size_t)phys * HKV + gv) * kPage * D;
      if (SHARED)
        copy_vec_warp<D>(k_row + (size_t)gv * D, PageDst<D>{(__nv_bfloat16*)c.k + blkv, j});
      else
        copy_vec_warp<D>(v_row + (size_t)gv * D, VDst{(__nv_bfloat16*)c.v + blkv, j});
    }
  }
}

template <int D, int R, bool SHARED, bool NORM>
__device__ __forceinline__ void append_token(const __nv_bfloat16* k_row, const __nv_bfloat16* v_row, int b, int pos,
                                             const PagedCache& c, const RopeTables& tb, uint32_t* err,
                                             const NormArgs& nm, int g_begin, int g_end) {
  const int lane = threadIdx.x & 31;
  if (pos < 0 || pos >= kMaxPos || (pos >> 4) >= c.max_pages) {
    if (lane == 0) set_error(err, kErrPos);
    return;
  }
  float2 cs[8];
  rope_cs_lane8<D, R>(tb, pos, cs);
  float wk[16];
  if (NORM) lane_weights<D>(nm.wk, wk);
  append_token_cs<D, R, SHARED, NORM>(k_row, v_row, b, pos, c, cs, err, nm, wk, g_begin, g_end);
}

// One warp per row of the prefill batch; the owning sequence is found by a scan over B.
// With q_out set, the row's query heads are also roped (declared bf16 cast) into q_out: the
// attention kernel that follows reads its queries already rotated.
template <int D, int R, bool SHARED, bool NORM>
__global__ void __launch_bounds__(256) append_prefill_kernel(const __nv_bfloat16* __restrict__ k,
                                                             const __nv_bfloat16* __restrict__ v,
                                                             const __nv_bfloat16* __restrict__ q,
                                                             __nv_bfloat16* q_out, SeqRows rows, PagedCache cache,
                                                             RopeTables tb, uint32_t* err, NormArgs nm, bool rows_kv) {
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int HQ = cache.hq, HKV = cache.hkv;
  if (r >= rows.T) return;
  int owner = -1;
  for (int b0 = 0; b0 < rows.B; b0 += 32) {
    const int b = b0 + lane;
    bool mine = false;
    if (b < rows.B) {
      const int s = rows.q_start[b], L = rows.q_len[b];
      mine = (L > 0 && r >= s && r - s < L);
    }
    const unsigned m = __ballot_sync(0xffffffffu, mine);
    if (m) {
      owner = b0 + __ffs(m) - 1;
      break;
    }
  }
  if (owner < 0) return;
  const long long pos64 = (long long)rows.ctx_start[owner] + (r - rows.q_start[owner]);   // no int overflow
  if (pos64 < 0 || pos64 >= kMaxPos || (int)(pos64 >> 4) >= cache.max_pages) {
    if (lane == 0) set_error(err, kErrPos);
    return;
  }
  const int pos = (int)pos64;
  float2 cs[8];   // the row's angles, shared by its query heads and its key heads
  rope_cs_lane8<D, R>(tb, pos, cs);
  float wk[16];
  if (NORM) lane_weights<D>(nm.wk, wk);
  if (q_out != nullptr) {
    constexpr int VPW = 32 / (D / 16);
    if (NORM) {
      float wq[16];
      lane_weights<D>(nm.wq, wq);
      const float* fold = (SHARED && nm.wk != nullptr) ? wk : nullptr;   // w_k on the un-rotated dims
#pragma unroll 2
      for (int h0 = 0; h0 < HQ; h0 += VPW) {
        const size_t v = (size_t)r * HQ + h0 + lane / (D / 16);
        vec8_normed<D, R>(q + v * D, RowDst{q_out + v * D}, cs, nm.wq != nullptr, nm.eps, wq, fold, R);
      }
    } else {
#pragma unroll 4
      for (int h0 = 0; h0 < HQ; h0 += VPW) {
        const size_t v = (size_t)r * HQ + h0 + lane / (D / 16);
        rope_vec8_cs<D, R>(q + v * D, RowDst{q_out + v * D}, cs);
      }
    }
  }
  if (rows_kv)
    append_token_cs<D, R, SHARED, NORM>(k + (size_t)r * HKV * D, SHARED ? nullptr : v + (size_t)r * HKV * D,
                                        rows.pt_row ? rows.pt_row[owner] : owner, pos, cache, cs, err, nm, wk, 0,
                                        HKV);
}

// ---- the sliding K'/V append by key groups ---------------------------------------------------------
// A page-head block stores 8 keys x 8 dims per 128-byte core matrix, so a warp that appends one key
// writes 16 bytes into each of its 32-byte sectors, and the L2 completes the sector with data read
// back from DRAM. This kernel gives each warp one group of 8 positions aligned to 8 (keys of one
// core-matrix row group) and 4 KV heads: lane (key kk = lane & 7, piece p = lane >> 3) handles dims
// 8(p + 4i) .. +7 and their pair partners 128 + 8(p + 4i) .. +7, i = 0..3, so one warp store writes
// four whole core matrices. The arithmetic per element is that of the per-row append: the same
// angles (rope_cs) and the same rotation (rope_pair), so the cache bits are the same.

// Key group `gi` of the batch: the groups of sequence b are its positions' groups ctx_start / 8 ..
// (ctx_start + q_len - 1) / 8, numbered in sequence order. Warp-wide; b = -1 past the last group.
// A sequence with a negative ctx_start, whose rows do not lie inside the T rows of k and v
// (q_start < 0 or q_start + q_len > T), or whose positions reach past the last usable one
// (ctx_start + q_len > 262144, tested without forming the sum), has no groups and sets kErrPos.
__device__ __forceinline__ void find_group(const SeqRows& rows, int gi, int& out_b, int& out_grp, uint32_t* err) {
  const int lane = threadIdx.x & 31;
  int base = 0;
  out_b = -1;
  out_grp = 0;
  for (int b0 = 0; b0 < rows.B; b0 += 32) {
    const int b = b0 + lane;
    int cnt = 0, first = 0;
    if (b < rows.B) {
      const int L = rows.q_len[b], cs = rows.ctx_start[b], qs = rows.q_start[b];
      if (L > 0 && cs >= 0 && qs >= 0 && L <= rows.T - qs && L <= kMaxPos && cs <= kMaxPos - L) {
        first = cs >> 3;
        cnt = ((cs + L - 1) >> 3) - first + 1;
      } else if (L > 0 && gi == 0) {
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
    const unsigned m = __ballot_sync(0xffffffffu, cnt > 0 && gi >= base + excl && gi < base + incl);
    if (m) {
      const int src = __ffs(m) - 1;
      out_b = b0 + src;
      out_grp = __shfl_sync(0xffffffffu, first, src) + (gi - base - __shfl_sync(0xffffffffu, excl, src));
      return;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
}

// kGroupHeads KV heads per warp (4; 2 for a cache of 2 KV heads, the sliding layer's tensor-parallel
// rank slice at tp = 8). Two blocks per SM (at most 128 registers a thread) with one iteration's
// loads in flight per warp measured faster than one block with two (111 against 124 us for the
// 4 x 4096 batch).
template <int D, int R, int kGroupHeads>
__global__ void __launch_bounds__(256, 2) append_kv_groups_kernel(const __nv_bfloat16* __restrict__ k,
                                                               const __nv_bfloat16* __restrict__ v, SeqRows rows,
                                                               PagedCache c, RopeTables tb, uint32_t* err) {
  static_assert(D == 256 && R == 128, "the group path serves the sliding geometry");
  const int lane = threadIdx.x & 31;
  const int HKV = c.hkv;   // a multiple of kGroupHeads
  const int unit = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int gi = unit / (HKV / kGroupHeads), g0 = (unit % (HKV / kGroupHeads)) * kGroupHeads;
  int b, grp;
  find_group(rows, gi, b, grp, err);
  if (b < 0) return;
  const int cs0 = rows.ctx_start[b], L = rows.q_len[b], qs = rows.q_start[b];
  const int key0 = 8 * grp;   // the 8 keys share one page (groups are aligned within pages)
  if (key0 >= kMaxPos || (key0 >> 4) >= c.max_pages) {
    if (lane == 0) set_error(err, kErrPos);
    return;
  }
  const int phys = c.page_table[(size_t)(rows.pt_row ? rows.pt_row[b] : b) * c.max_pages + (key0 >> 4)];
  if (phys < 0 || phys >= c.num_pages) {
    if (lane == 0) set_error(err, kErrPage);
    return;
  }
  const int kk = lane & 7, p = lane >> 3;
  const int pos = key0 + kk;
  if (pos < cs0 || pos >= cs0 + L) return;   // outside the call's rows (the group's ragged ends)
  const int j = pos & 15;
  const size_t row = (size_t)(qs + (pos - cs0));
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {
    const int d0 = 8 * (p + 4 * i);
    float2 cs[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) cs[e] = rope_cs(tb, d0 + e, pos);
    uint4 lo[kGroupHeads], hi[kGroupHeads], vl[kGroupHeads], vh[kGroupHeads];
#pragma unroll
    for (int hh = 0; hh < kGroupHeads; ++hh) {
      const size_t src = (row * HKV + g0 + hh) * D;
      lo[hh] = *reinterpret_cast<const uint4*>(k + src + d0);
      hi[hh] = *reinterpret_cast<const uint4*>(k + src + D / 2 + d0);
      vl[hh] = *reinterpret_cast<const uint4*>(v + src + d0);
      vh[hh] = *reinterpret_cast<const uint4*>(v + src + D / 2 + d0);
    }
#pragma unroll
    for (int hh = 0; hh < kGroupHeads; ++hh) {
      uint32_t* lw = reinterpret_cast<uint32_t*>(&lo[hh]);
      uint32_t* hw = reinterpret_cast<uint32_t*>(&hi[hh]);
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        float a0 = bf16_lo(lw[w]), a1 = bf16_hi(lw[w]);
        float b0 = bf16_lo(hw[w]), b1 = bf16_hi(hw[w]);
        rope_pair(a0, b0, cs[2 * w]);
        rope_pair(a1, b1, cs[2 * w + 1]);
        lw[w] = pack_bf16(a0, a1);
        hw[w] = pack_bf16(b0, b1);
      }
      const size_t blk = ((size_t)phys * HKV + g0 + hh) * kPage * D;
      __nv_bfloat16* kd = (__nv_bfloat16*)c.k + blk;
      __nv_bfloat16* vd = (__nv_bfloat16*)c.v + blk;
      *reinterpret_cast<uint4*>(kd + tiled_offset(j, d0, D)) = lo[hh];
      *reinterpret_cast<uint4*>(kd + tiled_offset(j, D / 2 + d0, D)) = hi[hh];
      *reinterpret_cast<uint4*>(vd + tiled_offset_v256(j, d0)) = vl[hh];
      *reinterpret_cast<uint4*>(vd + tiled_offset_v256(j, D / 2 + d0)) = vh[hh];
    }
  }
}

template <int D, int R, bool SHARED, bool NORM>
__global__ void __launch_bounds__(256) append_decode_kernel(const __nv_bfloat16* __restrict__ k,
                                                            const __nv_bfloat16* __restrict__ v,
                                                            const int32_t* __restrict__ seq_len, int B,
                                                            PagedCache cache, RopeTables tb, uint32_t* err,
                                                            NormArgs nm) {
  // One warp per (request, VPW KV heads): the heads of one request run in parallel, each with the
  // lane mapping and arithmetic of the one-warp-per-token append (so the same bits).
  constexpr int VPW = 32 / (D / 16);
  const int HKV = cache.hkv;   // a multiple of VPW
  const int NC = HKV / VPW;
  const int unit = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (unit >= B * NC) return;
  const int b = unit / NC, g0 = (unit % NC) * VPW;
  append_token<D, R, SHARED, NORM>(k + (size_t)b * HKV * D, SHARED ? nullptr : v + (size_t)b * HKV * D, b,
                                   seq_len[b] - 1, cache, tb, err, nm, g0, g0 + VPW);
}

// The decode queries' norm (and, on a K==V layer with a key norm, the fold of w_k into their
// un-rotated dims) ahead of the decode kernel, which ropes them itself: out[v] = bf16 of the
// normed query, one declared cast more than the prefill staging has. No rotation here.
template <int D, int R, bool SHARED>
__global__ void __launch_bounds__(256) norm_queries_kernel(const __nv_bfloat16* __restrict__ q, __nv_bfloat16* out,
                                                           int n_vec, NormArgs nm) {
  constexpr int VPW = 32 / (D / 16);
  const int lane = threadIdx.x & 31;
  const int v0 = (blockIdx.x * 8 + (threadIdx.x >> 5)) * VPW;   // n_vec is a multiple of VPW
  if (v0 >= n_vec) return;
  const size_t v = (size_t)v0 + lane / (D / 16);
  float wq[16], wk[16];
  lane_weights<D>(nm.wq, wq);
  lane_weights<D>(nm.wk, wk);
  float2 cs[8];   // unused: no rotation
  vec8_normed<D, 0>(q + v * D, RowDst{out + v * D}, cs, nm.wq != nullptr, nm.eps, wq,
                    (SHARED && nm.wk != nullptr) ? wk : nullptr, R);
}

// The global layer's S and k_rot append by key groups (plain calls): one warp per (group of 8
// positions aligned to 8, KV head). Lane (key kk = lane & 7, piece p = lane >> 3) copies dims
// 8(p + 4i) .. +7 of its key's S, i = 0..15, so one warp store writes four whole core matrices of the
// page-head block; the rotated pairs (t, t + 256), t < 64, are those of i = 0, 1 with i + 8, whose
// p-RoPE goes to the k_rot side page with the per-row append's angles (rope_cs), rotation
// (rope_pair) and cast, so the cache bits are the same.
// Eight blocks per SM (32 registers a thread), so that a 2 x 8192 batch's warps are all resident at
// once (42 against 48 us with five blocks and a second, partial wave).
template <int D, int R>
__global__ void __launch_bounds__(256, 8) append_s_groups_kernel(const __nv_bfloat16* __restrict__ k, SeqRows rows,
                                                             PagedCache c, RopeTables tb, uint32_t* err) {
  static_assert(D == 512 && R == 64, "the group path serves the global geometry");
  const int lane = threadIdx.x & 31;
  const int HKV = c.hkv;
  const int unit = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int gi = unit / HKV, g = unit % HKV;
  int b, grp;
  find_group(rows, gi, b, grp, err);
  if (b < 0) return;
  const int cs0 = rows.ctx_start[b], L = rows.q_len[b], qs = rows.q_start[b];
  const int key0 = 8 * grp;
  if (key0 >= kMaxPos || (key0 >> 4) >= c.max_pages) {
    if (lane == 0) set_error(err, kErrPos);
    return;
  }
  const int phys = c.page_table[(size_t)(rows.pt_row ? rows.pt_row[b] : b) * c.max_pages + (key0 >> 4)];
  if (phys < 0 || phys >= c.num_pages) {
    if (lane == 0) set_error(err, kErrPage);
    return;
  }
  const int kk = lane & 7, p = lane >> 3;
  const int pos = key0 + kk;
  if (pos < cs0 || pos >= cs0 + L) return;   // outside the call's rows (the group's ragged ends)
  const int j = pos & 15;
  const __nv_bfloat16* src = k + ((size_t)(qs + (pos - cs0)) * HKV + g) * D;
  uint4 s[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) s[i] = *reinterpret_cast<const uint4*>(src + 8 * (p + 4 * i));
  __nv_bfloat16* sd = (__nv_bfloat16*)c.k + ((size_t)phys * HKV + g) * kPage * D;
#pragma unroll
  for (int i = 0; i < 16; ++i) *reinterpret_cast<uint4*>(sd + tiled_offset(j, 8 * (p + 4 * i), D)) = s[i];
  __nv_bfloat16* rd = (__nv_bfloat16*)c.krot + ((size_t)phys * HKV + g) * kRotPageElems;
#pragma unroll
  for (int i = 0; i < 2; ++i) {   // pairs t = 8 (p + 4i) + e with t + 256
    const int t0 = 8 * (p + 4 * i);
    uint4 lo = s[i], hi = s[i + 8];
    uint32_t* lw = reinterpret_cast<uint32_t*>(&lo);
    uint32_t* hw = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      float a0 = bf16_lo(lw[w]), a1 = bf16_hi(lw[w]);
      float b0 = bf16_lo(hw[w]), b1 = bf16_hi(hw[w]);
      rope_pair(a0, b0, rope_cs(tb, t0 + 2 * w, pos));
      rope_pair(a1, b1, rope_cs(tb, t0 + 2 * w + 1, pos));
      lw[w] = pack_bf16(a0, a1);
      hw[w] = pack_bf16(b0, b1);
    }
    *reinterpret_cast<uint4*>(rd + rot_offset(j, t0)) = lo;
    *reinterpret_cast<uint4*>(rd + rot_offset(j, D / 2 + t0)) = hi;
  }
}

cudaError_t launch_append_prefill(bool global, const void* k, const void* v, const SeqRows& rows,
                                  const PagedCache& cache, const DeviceState& st, cudaStream_t s, const void* q,
                                  void* q_out, const NormArgs& nm) {
  if (rows.T <= 0 || rows.B <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((rows.T + 7) / 8);
  const __nv_bfloat16 *kb = (const __nv_bfloat16*)k, *vb = (const __nv_bfloat16*)v, *qb = (const __nv_bfloat16*)q;
  __nv_bfloat16* qo = (__nv_bfloat16*)q_out;
  if (global) {
    if (nm.any()) {
      append_prefill_kernel<kGlobalD, kGlobalR, true, true>
          <<<blocks, 256, 0, s>>>(kb, nullptr, qb, qo, rows, cache, st.global, st.err, nm, true);
    } else {
      // S and k_rot by key groups (whole-sector writes), the staged queries (if any) by rows.
      const long long groups = (long long)rows.T / 8 + 2LL * rows.B;   // a sequence adds at most two partial groups
      const long long units = groups * cache.hkv;
      if (units > 0x3fffffffLL) return cudaErrorInvalidValue;
      append_s_groups_kernel<kGlobalD, kGlobalR>
          <<<(unsigned)((units + 7) / 8), 256, 0, s>>>(kb, rows, cache, st.global, st.err);
      if (qo != nullptr)
        append_prefill_kernel<kGlobalD, kGlobalR, true, false>
            <<<blocks, 256, 0, s>>>(kb, nullptr, qb, qo, rows, cache, st.global, st.err, nm, false);
    }
  } else if (nm.any()) {
    append_prefill_kernel<kSlidingD, kSlidingR, false, true>
        <<<blocks, 256, 0, s>>>(kb, vb, qb, qo, rows, cache, st.sliding, st.err, nm, true);
  } else {
    // K' and V by key groups (whole-sector writes), the queries by rows.
    const int gh = cache.hkv % 4 == 0 ? 4 : 2;   // KV heads per warp
    const long long groups = (long long)rows.T / 8 + 2LL * rows.B;   // a sequence adds at most two partial groups
    const long long units = groups * (cache.hkv / gh);
    if (units > 0x3fffffffLL) return cudaErrorInvalidValue;
    const unsigned gblocks = (unsigned)((units + 7) / 8);
    if (gh == 4)
      append_kv_groups_kernel<kSlidingD, kSlidingR, 4><<<gblocks, 256, 0, s>>>(kb, vb, rows, cache, st.sliding, st.err);
    else
      append_kv_groups_kernel<kSlidingD, kSlidingR, 2><<<gblocks, 256, 0, s>>>(kb, vb, rows, cache, st.sliding, st.err);
    if (qo != nullptr)
      append_prefill_kernel<kSlidingD, kSlidingR, false, false>
          <<<blocks, 256, 0, s>>>(kb, vb, qb, qo, rows, cache, st.sliding, st.err, nm, false);
  }
  return cudaGetLastError();
}

cudaError_t launch_append_decode(bool global, const void* k_new, const void* v_new, const int32_t* seq_len,
                                 int B, const PagedCache& cache, const DeviceState& st, cudaStream_t s,
                                 const NormArgs& nm) {
  if (B <= 0) return cudaSuccess;
  // warps: B x (KV heads / heads per warp instruction)
  const int per_req = cache.hkv / (32 / ((global ? kGlobalD : kSlidingD) / 16));
  const unsigned blocks = (unsigned)(((long long)B * per_req + 7) / 8);
  const __nv_bfloat16 *kb = (const __nv_bfloat16*)k_new, *vb = (const __nv_bfloat16*)v_new;
  if (global) {
    if (nm.any())
      append_decode_kernel<kGlobalD, kGlobalR, true, true>
          <<<blocks, 256, 0, s>>>(kb, nullptr, seq_len, B, cache, st.global, st.err, nm);
    else
      append_decode_kernel<kGlobalD, kGlobalR, true, false>
          <<<blocks, 256, 0, s>>>(kb, nullptr, seq_len, B, cache, st.global, st.err, nm);
  } else {
    if (nm.any())
      append_decode_kernel<kSlidingD, kSlidingR, false, true>
          <<<blocks, 256, 0, s>>>(kb, vb, seq_len, B, cache, st.sliding, st.err, nm);
    else
      append_decode_kernel<kSlidingD, kSlidingR, false, false>
          <<<blocks, 256, 0, s>>>(kb, vb, seq_len, B, cache, st.sliding, st.err, nm);
  }
  return cudaGetLastError();
}

cudaError_t launch_norm_queries(bool global, const void* q, void* out, int B, int hq, const NormArgs& nm,
                                cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  const int n_vec = B * hq;
  if (global) {
    const unsigned blocks = (unsigned)((n_vec + 7) / 8);   // one vector per warp
    norm_queries_kernel<kGlobalD, kGlobalR, true><<<blocks, 256, 0, s>>>((const __nv_bfloat16*)q,
                                                                         (__nv_bfloat16*)out, n_vec, nm);
  } else {
    const unsigned blocks = (unsigned)((n_vec + 15) / 16);   // two vectors per warp
    norm_queries_kernel<kSlidingD, kSlidingR, false><<<blocks, 256, 0, s>>>((const __nv_bfloat16*)q,
                                                                            (__nv_bfloat16*)out, n_vec, nm);
  }
  return cudaGetLastError();
}

}  // namespace g4
