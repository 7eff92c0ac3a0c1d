// Device-side helpers shared by the g4attn kernels: bf16 packing, RoPE table lookups,
// bounded mbarrier waits, bulk/tensor copies (TMA) and tcgen05 (5th-generation tensor core)
// wrappers, all as inline PTX for sm_103a. No kernel here ever traps: a wait that runs out
// sets a bit in the caller-visible error word and returns false.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define G4_DEV __device__ __forceinline__

namespace g4 {

// ---- constants fixed by the two supported layer kinds ------------------------------------
constexpr int kPage = 16;                 // keys per cache page
constexpr int kMaxPos = 262144;           // positions 0 .. 262143
constexpr int kRopeCoarse = kMaxPos / 256;  // coarse table: angle of 256*c, 0 <= c < 1024
constexpr int kRopeMid = 16;                // mid table: angle of 16*a, 0 <= a < 16
constexpr int kRopeFine = 16;               // fine table: angle of b, 0 <= b < 16

constexpr int kSlidingHq = 32, kSlidingHkv = 16, kSlidingD = 256, kSlidingR = 128;
constexpr int kGlobalHq = 32, kGlobalHkv = 4, kGlobalD = 512, kGlobalR = 64;

constexpr int kDecodeChunkSliding = 256;  // keys per fixed decode chunk (aligned to key 0)
constexpr int kDecodeChunkGlobal = 1024;

// Error-word bits (g4attn_status_sync maps them to g4_status values).
enum : uint32_t { kErrTimeout = 1u, kErrPage = 2u, kErrPos = 4u, kErrSpan = 8u };

// Bounded waits give up after this long; nothing legitimate waits anywhere near it. The waits of
// the kernels' protocols take their limit from the launch (g4attn_set_wait_limit_ns; this is the
// default and the largest allowed); the drains of an aborted kernel (copies and MMAs it issued
// that must finish before it may leave) always use this one.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Cache page layout. One page of one KV head holds 16 keys x D dims as core matrices of
// 8 keys x 8 dims (128 contiguous bytes). Sliding pages (D = 256): key j, dim d sits at element
//   ((j / 8) * 32 + d / 8) * 64 + (j % 8) * 8 + d % 8
// of the page-head block, whose 16*D elements are contiguous at
//   cache + (page * Hkv + head) * 16 * D.
// Global pages (D = 512) are two such 256-dim halves one after the other, so that each half
// (8 KB) is contiguous: key j, dim d at
//   (((d / 256) * 2 + j / 8) * 32 + (d % 256) / 8) * 64 + (j % 8) * 8 + d % 8.
// One contiguous copy of a block (or half-block) lands in shared memory as an operand the
// tensor cores read directly (K-major for K, MN-major for V), and every 8x8 block is one
// ldmatrix tile.
__host__ __device__ constexpr int tiled_offset(int j, int d, int D) {
  return D == 512 ? ((((d >> 8) * 2 + (j >> 3)) * 32 + ((d & 255) >> 3)) * 64 + (j & 7) * 8 + (d & 7))
                  : (((j >> 3) * (D >> 3) + (d >> 3)) * 64 + (j & 7) * 8 + (d & 7));
}

// Sliding V pages are stored as two contiguous 128-dim halves (4 KB each) of the same 8x8 core
// matrices, so that each CTA of a prefill pair (one per half of the head dims) copies its half
// of a page with one bulk copy: key j, dim d at
//   (((d / 128) * 2 + j / 8) * 16 + (d % 128) / 8) * 64 + (j % 8) * 8 + d % 8.
__host__ __device__ constexpr int tiled_offset_v256(int j, int d) {
  return ((((d >> 7) * 2 + (j >> 3)) * 16 + ((d & 127) >> 3)) * 64 + (j & 7) * 8 + (d & 7));
}

// Rotated-column side pages of a global (K==V) cache: p-RoPE(S) on the 128 rotated dims
// d in [0, 64) U [256, 320), the only columns where K differs from the stored S. Key j, dim d
// sits at element (((d / 256) * 2 + j / 8) * 8 + (d % 64) / 8) * 64 + (j % 8) * 8 + d % 8 of a
// 2048-element page-head block at k_rot + (page * Hkv + head) * 2048.
constexpr int kRotPageElems = kPage * 2 * kGlobalR;   // 2048
__host__ __device__ constexpr int rot_offset(int j, int d) {
  return ((((d >> 8) * 2 + (j >> 3)) * 8 + ((d & 63) >> 3)) * 64 + (j & 7) * 8 + (d & 7));
}

// RoPE cos/sin tables for one layer kind, built in fp64 on the host and stored as fp32:
// coarse[t][c] = (cos, sin)(256*c*f_t), mid[t][a] = (cos, sin)(16*a*f_t) and
// fine[t][b] = (cos, sin)(b*f_t). The mid and fine tables are small enough to stay in L1.
// The same values are also kept transposed (entry-major, [entry][R]), for the prefill kernels'
// in-kernel query rotation, whose threads hold consecutive pairs t: there a warp's load of one
// entry for 32 pairs reads 256 contiguous bytes instead of 32 lines.
struct RopeTables {
  const float2* coarse;   // [R][kRopeCoarse]
  const float2* mid;      // [R][kRopeMid]
  const float2* fine;     // [R][kRopeFine]
  const float2* coarse_t; // [kRopeCoarse][R]
  const float2* mid_t;    // [kRopeMid][R]
  const float2* fine_t;   // [kRopeFine][R]
};

// ---- small helpers -------------------------------------------------------------------------
G4_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

G4_DEV unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

G4_DEV void set_error(uint32_t* err, uint32_t bits) {
  if (err) atomicOr(err, bits);   // error reporting only; never part of the arithmetic
}

G4_DEV float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
G4_DEV float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
G4_DEV float bf16_to_f(__nv_bfloat16 h) { return __bfloat162float(h); }

// Round-to-nearest-even pack of two fp32 values into bf16x2 (lo in the low half).
G4_DEV uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
G4_DEV float round_bf16(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// Complex product (cos a, sin a) * (cos b, sin b) = (cos, sin)(a + b), fp32.
G4_DEV float2 cmul(float2 a, float2 b) {
  return make_float2(fmaf(a.x, b.x, -(a.y * b.y)), fmaf(a.y, b.x, a.x * b.y));
}

// (cos, sin)(pos * f_t) from the three-level table by the angle-addition formula:
// pos = 256*c + 16*a + b, combined as (coarse * mid) * fine.
G4_DEV float2 rope_cs(const RopeTables& tb, int t, int pos) {
  const float2 c = __ldg(tb.coarse + (size_t)t * kRopeCoarse + (pos >> 8));
  const float2 m = __ldg(tb.mid + t * kRopeMid + ((pos >> 4) & 15));
  const float2 f = __ldg(tb.fine + t * kRopeFine + (pos & 15));
  return cmul(cmul(c, m), f);
}

// 2^x on the multi-function unit (PTX ex2.approx.ftz.f32; 2^-inf = +0). Results below 2^-126
// flush to zero: in the softmax they are weights under 2^-126 next to a row maximum of 1, far
// below what an fp32 accumulator or the bf16 output resolves. The non-flushing form costs
// about three times as much issue time here.
G4_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The rotation of one half-split pair, fp32 (the same expression everywhere in the library).
G4_DEV void rope_pair(float& lo, float& hi, float2 cs) {
  const float a = lo, b = hi;
  lo = fmaf(a, cs.x, -(b * cs.y));
  hi = fmaf(b, cs.x, a * cs.y);
}

// ---- mbarrier --------------------------------------------------------------------------------
G4_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
G4_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
G4_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
G4_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
G4_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of `bar` to complete. Gives up (returns false, sets *abort and the
// timeout bit) once limit_ns have passed since the first poll failed (limit 0: at once), or as
// soon as *abort is set by another thread.
G4_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* err,
                      unsigned long long limit_ns = kWaitLimitNs) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (abort && *abort) return false;
    if (globaltimer() - t0 >= limit_ns) {
      if (abort) *abort = 1;
      set_error(err, kErrTimeout);
      return false;
    }
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(a, parity)) return true;
  }
}

// Named barrier over `count` threads that also ANDs a predicate across them. Every thread of
// the group must reach it; the waits before it are bounded, so it is reached in bounded time.
G4_DEV bool named_barrier_and(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// ---- thread-block clusters (distributed shared memory between the two CTAs of a pair) ---------
G4_DEV uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address in CTA `rank`'s shared memory of the variable at local shared address `saddr`.
G4_DEV uint32_t map_peer(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Bulk copy of `bytes` from this CTA's shared memory into another CTA's (addresses 16-byte
// aligned, size a multiple of 16); completion counts the bytes on the receiver's mbarrier.
G4_DEV void bulk_s2peer(uint32_t dst_cluster, const void* src, uint32_t bytes, uint32_t peer_bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst_cluster),
               "r"(smem_u32(src)), "r"(bytes), "r"(peer_bar)
               : "memory");
}
G4_DEV void st_peer_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster, releasing this thread's prior writes.
G4_DEV void mbar_arrive_peer(uint32_t peer_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(peer_bar) : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster with the default (CTA-scope) release. About
// four times faster than the cluster-scope release above; for signals whose data is already
// complete when the arrive issues: registers read back (tcgen05.wait::ld), tensor-memory stores
// finished (tcgen05.wait::st), generic writes fenced to the async proxy, or copies observed
// complete. The waiter acquires at cluster scope.
G4_DEV void mbar_arrive_remote(uint32_t peer_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(peer_bar) : "memory");
}
G4_DEV bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// mbar_wait for barriers that the other CTA of the cluster arrives on: acquires their writes at
// cluster scope. Bounded like mbar_wait.
G4_DEV bool mbar_wait_cl(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* err,
                         unsigned long long limit_ns = kWaitLimitNs) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait_cluster(a, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (abort && *abort) return false;
    if (globaltimer() - t0 >= limit_ns) {
      if (abort) *abort = 1;
      set_error(err, kErrTimeout);
      return false;
    }
    for (int i = 0; i < 32; ++i) {
      if (mbar_try_wait_cluster(a, parity)) return true;
      __nanosleep(32);   // a cluster-scope poll does not suspend: leave issue slots to the other warps
    }
  }
}

// Out-of-line copies of the two waits, for kernels that wait in many places (one copy of each
// polling loop keeps their hot loops small enough for the instruction caches; a kernel whose
// inner loop waits on every step keeps the inlined form).
static __device__ __noinline__ bool mbar_wait_ool(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* err,
                                                  unsigned long long limit_ns) {
  return mbar_wait(bar, parity, abort, err, limit_ns);
}
static __device__ __noinline__ bool mbar_wait_cl_ool(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                     uint32_t* err, unsigned long long limit_ns) {
  return mbar_wait_cl(bar, parity, abort, err, limit_ns);
}

// ---- bulk copies (TMA) -------------------------------------------------------------------------
G4_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Contiguous global -> shared copy, completion counted on `bar` (bytes % 16 == 0, aligned).
G4_DEV void bulk_g2s(void* smem, const void* gmem, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem)),
      "l"(gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

G4_DEV void tma_load_3d(void* smem, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4}], [%5];" ::"r"(smem_u32(smem)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

G4_DEV void tma_load_5d(void* smem, const CUtensorMap* map, int c0, int c1, int c2, int c3, int c4, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5, %6}], [%7];" ::"r"(smem_u32(smem)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_u32(bar))
      : "memory");
}

// Tiled shared -> global store through a tensor map (bulk async-group completion). The
// innermost coordinate must keep the copy 16-byte aligned; no coordinate may be negative.
G4_DEV void tma_store_3d(const CUtensorMap* map, const void* smem, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(smem)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
G4_DEV void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed bulk store of this thread has finished reading shared memory.
G4_DEV void bulk_wait_group_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Prefetch of a tensor-map tile into L2 (no shared memory, no completion to wait for).
G4_DEV void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

G4_DEV void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- tcgen05: tensor memory, MMA, commit ------------------------------------------------------
G4_DEV void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {   // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
G4_DEV void tmem_relinquish() {   // whole warp
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
G4_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {   // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
G4_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
G4_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100-family layout: start>>4 at
// bits 0-13, leading byte offset>>4 at 16-29, stride byte offset>>4 at 32-45, version 1 at
// bit 46, swizzle mode 2 = 128B at bits 61-63). The tile base must be 1024-byte aligned.
G4_DEV uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Shared-memory matrix descriptor, no swizzle (core matrices of 8 rows x 16 bytes stored as
// 128 contiguous bytes). lbo = byte distance between core matrices adjacent along K,
// sbo = along M/N (both for K-major and MN-major operands).
G4_DEV uint64_t desc_tiled(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// Instruction descriptor of kind::f16 with bf16 A/B and an fp32 accumulator.
// a_mn / b_mn: operand stored MN-major (transposed) rather than K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4)                         // D format: f32
         | (1u << 7)                       // A format: bf16
         | (1u << 10)                      // B format: bf16
         | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16)
         | ((uint32_t)(N >> 3) << 17)      // N / 8
         | ((uint32_t)(M >> 4) << 24);     // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]
G4_DEV void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]
G4_DEV void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on `bar` when every tcgen05 op issued so far by this thread has completed.
G4_DEV void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// ---- 2-SM forms: the two CTAs of a cluster pair act as one MMA unit ----------------------------
// Allocation, relinquish and deallocation with cta_group::2 are collective: one warp of each CTA
// issues them and both CTAs get the same columns. An MMA is issued by the even CTA only: A and D
// are split by rows (each CTA holds its 128 rows of an M = 256 tile), B by columns (each CTA
// holds N/2 of the N columns, at the same shared-memory offset); the instruction descriptor
// carries M = 256 and the full N.
G4_DEV void tmem_alloc2(uint32_t* dst_smem, uint32_t ncols) {   // whole warp, in both CTAs
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
G4_DEV void tmem_relinquish2() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory"); }
G4_DEV void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {   // whole warp, in both CTAs
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
G4_DEV void mma2_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
G4_DEV void mma2_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
// Commit of the pair's MMAs issued so far by this thread: arrives on the mbarrier at `bar`'s
// offset in every CTA of `cta_mask`.
G4_DEV void mma2_commit_mc(uint64_t* bar, uint16_t cta_mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "h"(cta_mask)
               : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns; thread i of the warp gets lane (base + i).
G4_DEV void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns.
G4_DEV void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
G4_DEV void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
G4_DEV void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
G4_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 lanes x 64 consecutive 32-bit columns (asynchronous: read r only after tmem_ld_wait_on(r)).
G4_DEV void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
               : "r"(taddr)
               : "memory");
}
// tcgen05.wait::ld that also names the registers a load in flight writes, so that no use of
// them can be scheduled before the wait.
G4_DEV void tmem_ld_wait_on(uint32_t (&r)[64]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]), "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63])
               :
               : "memory");
}

// Reads columns [0, 64 NB) of this warp's 32 lanes, 64 at a time, the load of one batch in flight
// while the previous one is processed: fn(c, regs) gets batch c (columns 64c .. 64c+63), and
// loaded() runs once every column has been read into registers (the columns may then be
// overwritten). NB is even. Warp-wide.
template <int NB, class Loaded, class Fn>
G4_DEV void tmem_ld_stream64(uint32_t taddr, Loaded&& loaded, Fn&& fn) {
  static_assert(NB % 2 == 0, "batches come in pairs");
  uint32_t a[64], b[64];
  tmem_ld64(taddr, a);
  tmem_ld_wait_on(a);
#pragma unroll 1
  for (int c = 0; c < NB; c += 2) {
    tmem_ld64(taddr + 64 * (c + 1), b);
    fn(c, a);
    tmem_ld_wait_on(b);
    if (c + 2 < NB)
      tmem_ld64(taddr + 64 * (c + 2), a);
    else
      loaded();
    fn(c + 1, b);
    if (c + 2 < NB) tmem_ld_wait_on(a);
  }
}

G4_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---- legacy warp MMA (decode on the global layer) ----------------------------------------------
G4_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
G4_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
G4_DEV void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr)
               : "memory");
}
// D(16x8 f32) += A(16x16 bf16, row) * B(16x8 bf16, col)
G4_DEV void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, "
      "%1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace g4
