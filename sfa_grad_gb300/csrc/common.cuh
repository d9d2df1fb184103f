// Shared device helpers for the sm_103a kernels of the sparse flash-attention
// backward: mbarrier waits with a wall-clock limit, tcgen05 (TMEM allocation, MMA,
// commit, TMEM loads), cp.async with zero fill, and the 128-byte-swizzled
// shared-memory operand layouts the tensor-core descriptors describe.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace sfa {

// ------------------------------------------------------------------ limits
// Every pipeline wait gives up after a wall-clock limit (Prob::wait_ns,
// measured on %globaltimer); the kernel then records an error code and winds
// down instead of hanging.  The limit's resolution is one poll (a try_wait
// suspends for at most 10 us) plus the timer's update period.
constexpr unsigned long long kWaitNsDefault = 2000000000ull;   // 2 s
// Wind-down waits (for copies and MMAs already issued) ignore the abort flag
// and use this limit whatever the pipeline limit is.
constexpr unsigned long long kSettleNs = 2000000000ull;

// Kernels that allocate all 512 TMEM columns request at least this much
// dynamic shared memory so that no two of their CTAs share an SM.
constexpr int kOneCtaSmem = 120 * 1024;

// Device error codes written to the workspace error word.
constexpr int kErrTimeout = 1;       // a pipeline wait ran out
constexpr int kErrSeqLens = 2;       // TND lengths negative or not summing to T1/T2

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Nanoseconds of the GPU's global timer.
__device__ __forceinline__ unsigned long long gtime_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// n arrivals at once (n >= 1, at most the phase's pending count).
__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}
// try_wait may suspend the thread until the phase completes; the hint caps
// one suspension at 10 us so that the callers' wall-clock limits hold.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(10000u)
      : "memory");
  return ok != 0;
}
// Non-suspending poll (test_wait), for the single-thread MMA issuers: the
// tensor core keeps only a few MMAs queued, so every cycle the issuer spends
// waiting can leave it idle, and a suspending try_wait returns later than a
// poll.
__device__ __forceinline__ bool mbar_poll(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\n"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// What a pipeline wait needs besides the barrier: the CTA's abort flag (any
// warp may raise it), the global error word and the wall-clock limit.
struct Waiter {
  volatile int* abort;
  int* gerr;
  unsigned long long limit_ns;
};

// Bounded wait on phase `parity`.  Returns false when the wait was abandoned:
// another warp raised the abort flag, or the limit ran out (then this thread
// raises the flag and records a timeout).  A try_wait may suspend the thread
// for a while inside one poll, so those waits read the flag and the clock
// after every poll; the non-suspending polls of the MMA issuers every 32.
template <bool POLL>
__device__ __forceinline__ bool mbar_wait_t(uint64_t* bar, uint32_t parity, const Waiter& w) {
  const uint32_t a = smem_u32(bar);
  if (POLL ? mbar_poll(a, parity) : mbar_test(a, parity)) return true;
  const unsigned long long t0 = gtime_ns();
  for (uint32_t it = 1;; ++it) {
    if (POLL ? mbar_poll(a, parity) : mbar_test(a, parity)) return true;
    if (!POLL || (it & 31u) == 0) {
      if (*w.abort) return false;
      if (gtime_ns() - t0 > w.limit_ns) break;
    }
  }
  *w.abort = 1;
  atomicExch(w.gerr, kErrTimeout);
  return false;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const Waiter& w) {
  return mbar_wait_t<false>(bar, parity, w);
}
__device__ __forceinline__ bool mbar_wait_poll(uint64_t* bar, uint32_t parity, const Waiter& w) {
  return mbar_wait_t<true>(bar, parity, w);
}

// Wind-down wait for the completion of phase `parity` of `bar`, whatever the
// abort flag says: used before a CTA exits so that no TMA copy or MMA it
// issued is still writing its shared or tensor memory.  Gives up after
// kSettleNs (recording a timeout) so that it cannot hang either.
__device__ __forceinline__ void mbar_settle(uint64_t* bar, uint32_t parity, int* gerr) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = gtime_ns();
  for (;;) {
    if (mbar_test(a, parity)) return;
    if (gtime_ns() - t0 > kSettleNs) {
      atomicExch(gerr, kErrTimeout);
      return;
    }
  }
}

// Records, for a ring of up to 32 stage slots armed by one thread, the parity
// of the last phase armed on each slot; settle() then waits for each of them.
// A slot is only re-armed after its previous phase completed, so the last
// armed phase is the only one that can still have copies in flight.
struct ArmLog {
  uint32_t armed = 0, parity = 0;
  __device__ __forceinline__ void arm(int slot, uint32_t ph) {
    armed |= 1u << slot;
    parity = (parity & ~(1u << slot)) | ((ph & 1u) << slot);
  }
  __device__ __forceinline__ void settle(uint64_t* bars, int* gerr) const {
    for (int s = 0; s < 32; ++s)
      if (armed & (1u << s)) mbar_settle(&bars[s], (parity >> s) & 1u, gerr);
  }
};

// The last MMAs issued by this thread, settled: commits them to `bar` (a
// barrier of count 1 used for nothing else) and waits for its phase 0.
__device__ __forceinline__ void mma_settle(uint64_t* bar, int* gerr);

// ------------------------------------------------------------------ cp.async
// 16-byte global -> shared copy; src_bytes = 0 fills the destination with zeros
// without reading the source.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
// Makes this thread's completed generic-proxy shared writes visible to the
// tensor core (async proxy).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 16-byte shared-memory load and store at a shared-window address.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// ------------------------------------------------------------------ TMA
// Tensor maps of one call (2-D, 16-bit elements, 64-element = 128-byte inner
// box, 128-byte swizzle, so a box lands in shared memory exactly in the panel
// layout below).  Rows outside a map's extent (negative or past the end) are
// filled with zeros.
struct Maps {
  CUtensorMap q;    // (T1*G, 512), box 64 x GP
  CUtensorMap qr;   // (T1*G, 64),  box 64 x GP
  CUtensorMap dO;   // (T1*G, 512), box 64 x GP
  CUtensorMap k;    // (T2, 512),   box 64 x bs (block-sparse indices, bs >= 8), else unused
  CUtensorMap kr;   // (T2, 64),    box 64 x bs
  CUtensorMap v;    // (T2, 512),   box 64 x bs
  // staged P^T / dS^T, (chunk*Kpad rows, Gs heads), box 64 heads x 64 rows:
  // heads past Gs are outside the map and arrive as zeros
  CUtensorMap P;
  CUtensorMap dS;
  // q, qRope, dO with boxes of GK = G rounded up to 16 rows: the score
  // kernel loads only a token's own head rows (the padded rows up to GP stay
  // zero in its shared memory)
  CUtensorMap qg, qrg, dOg;
  // staged P^T / dS^T for the score kernel's stores: box 32 heads x 32 rows,
  // 64-byte swizzle (heads past Gs are outside the map and not written)
  CUtensorMap Pw, dSw;
  // dQ (T1*G, 512) and dQRope (T1*G, 64) for the stores of kvq's query side
  // (in the forward, dQw maps the output O for dq.cu's stores): box 32
  // features x 32 head rows, 64-byte swizzle
  CUtensorMap dQw, dQRw;
  // deterministic mode's bf16 partial rows (chunk*Kpad, 1088) for kvq's
  // drain stores: box 32 features x 32 slot rows, 64-byte swizzle
  CUtensorMap partw;
};

// Tensor maps of the key-major block kernel (kvb.cu).
struct BlkMaps {
  // q and dO as (64 features, T1*G rows, 8 panels): one box = all eight
  // 64-feature panels of one token's GK head rows (GK = G rounded up to 16),
  // landing as eight consecutive [GK x 64] panels
  CUtensorMap q;
  CUtensorMap qr;   // (T1*G, 64), box 64 x GK
  CUtensorMap dO;
  CUtensorMap P;    // staged P^T,  (chunk*Kpad, Gs), box 64 x 64 (as in Maps)
  CUtensorMap dS;   // staged dS^T, (chunk*Kpad, Gs), box 64 x 64
};

// Arrive once on `bar` and add `bytes` to the transaction count the phase
// waits for.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// One box at (x, y, z) of a 3-D map into shared memory at `dst`.
__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
// Store of the box at (x, y) from shared memory at `src` (bulk group of the
// issuing thread); x, y >= 0.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(x), "r"(y),
               "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The issuing thread's bulk stores have read their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// The issuing thread's bulk stores are complete.
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Prefetch of the box at (x, y) into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y) : "memory");
}
// One box at (x = column, y = row) into shared memory at `dst`.
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// ------------------------------------------------------------------ operand layouts
// All tensor-core operands live in shared memory as 128-byte swizzled rows:
// a "panel" holds R rows of 64 consecutive 16-bit elements (128 B per row),
// rows contiguous, 8-row atoms of 1024 B, and the 16-byte chunk c of row r is
// stored at chunk position c ^ (r & 7).  A K-major operand (K contiguous) with
// K > 64 is a sequence of panels along K; an MN-major operand (M or N
// contiguous) is a sequence of panels along MN whose rows are indexed by K.
// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}
// K-major panel of R rows starting at `panel`: K step ks (16 elements) inside
// the 64-wide panel advances the start by 32 B.
__device__ __forceinline__ uint64_t sdesc_kmajor(uint32_t panel, int ks) {
  return sdesc(panel + (uint32_t)ks * 32u, 16u, 1024u);
}
// MN-major operand made of panels of `krows` K-rows each (panel stride
// krows*128 B): K step ks (16 rows) advances the start by 2048 B.
__device__ __forceinline__ uint64_t sdesc_mnmajor(uint32_t base, int ks, uint32_t krows) {
  return sdesc(base + (uint32_t)ks * 2048u, krows * 128u, 1024u);
}

// Instruction descriptor for kind::f16 with fp32 accumulation.
// is_f16: operands are fp16 (else bf16); a_mn / b_mn: operand is MN-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool is_f16, bool a_mn, bool b_mn) {
  return (1u << 4) | ((is_f16 ? 0u : 1u) << 7) | ((is_f16 ? 0u : 1u) << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D(tmem) (+)= A(smem desc) * B(smem desc)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Four consecutive K steps (64 elements) into one accumulator.  `a` and `b`
// are the descriptors of step 0; each step advances the encoded start address
// by SA / SB units of 16 B (2 for a K-major 128-byte-swizzled panel, 128 for
// an MN-major one).  The MMA issue path is a single thread whose instruction
// latency is not hidden, so callers build descriptors once per stage and this
// only offsets them.
template <uint32_t SA, uint32_t SB>
__device__ __forceinline__ void mma_ss_k64(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc_first) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %3, 1;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %3, 1;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %10, %3, 1;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc_first), "l"(a + SA), "l"(b + SB), "l"(a + 2 * SA), "l"(b + 2 * SB),
      "l"(a + 3 * SA), "l"(b + 3 * SB)
      : "memory");
}
// Descriptor offset, in encoded 16-byte units, of a byte offset inside shared memory.
__device__ __forceinline__ uint64_t desc_off(uint32_t bytes) { return (uint64_t)(bytes >> 4); }
// Arrives on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mma_settle(uint64_t* bar, int* gerr) {
  mma_commit(bar);
  mbar_settle(bar, 0, gerr);
}

// 32 lanes x 32 consecutive fp32 columns: thread i of the warp gets lane
// (warp quadrant base + i), columns [col, col+32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 16 consecutive fp32 columns (thread i: lane base + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 2^x on the special-function unit (ex2.approx, flush-to-zero); 2^-inf = 0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ element types
template <typename T>
struct Elt;
template <>
struct Elt<__nv_bfloat16> {
  static constexpr bool is_f16 = false;
  __device__ static __forceinline__ uint32_t pack(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  // the two values pack() put in a word: a from the low half, b from the high
  // the two values of w times those of f, rounded once
  __device__ static __forceinline__ uint32_t mul2(uint32_t w, uint32_t f) {
    __nv_bfloat162 r = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&w), *reinterpret_cast<const __nv_bfloat162*>(&f));
    return *reinterpret_cast<uint32_t*>(&r);
  }
  __device__ static __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  __device__ static __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};
template <>
struct Elt<__half> {
  static constexpr bool is_f16 = true;
  __device__ static __forceinline__ uint32_t pack(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static __forceinline__ uint32_t mul2(uint32_t w, uint32_t f) {
    __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&w), *reinterpret_cast<const __half2*>(&f));
    return *reinterpret_cast<uint32_t*>(&r);
  }
  __device__ static __forceinline__ float to_f(__half x) { return __half2float(x); }
  __device__ static __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
};

// ------------------------------------------------------------------ problem view
// Per-token metadata built by the prep kernel: start row of the token's KV
// segment, and the largest key position the token may attend (-1: none).
struct TokMeta {
  int kv_start;
  int limit;
};

// Everything a kernel needs about one call (device pointers, sizes).
struct Prob {
  const void* q;    // (T1, G, 512)
  const void* qr;   // (T1, G, 64) or null
  const void* k;    // (T2, 512)
  const void* kr;   // (T2, 64) or null
  const void* v;    // (T2, 512)
  const void* dO;   // (T1, G, 512)
  const void* out;  // (T1, G, 512)
  const int* idx;   // (T1, Kidx)
  const float* smax;  // (T1, G)
  const float* ssum;  // (T1, G)
  const TokMeta* meta;  // (T1)
  const float* dsum;    // (T1, G)
  int* rowtab;          // (ntok, Kpad): kv row of every slot of the chunk, -1 if masked
  int T1, T2, G, Gp, Kidx, bs, Keff, Kpad;
  int Gs;   // heads per staged P^T / dS^T row: G rounded up to 16
  int has_rope;
  float scale;
  int tok0, ntok;  // token chunk processed by this launch
  unsigned long long wait_ns;   // limit of every pipeline wait
};

// Expanded key position of slot s of token t (64-bit: index + block offset
// cannot overflow) and whether it is attendable.
__device__ __forceinline__ int slot_row(const Prob& p, const TokMeta& m, int t, int s) {
  if (s >= p.Keff) return -1;
  const int r = __ldg(p.idx + (size_t)t * p.Kidx + s / p.bs);
  const long long j = (long long)r + (s % p.bs);
  if (j < 0 || j > (long long)m.limit) return -1;
  return m.kv_start + (int)j;
}

}  // namespace sfa
