// Key-side and query-side contractions of a token chunk in one launch.  Each
// CTA (one per SM) runs two independent tensor-core pipelines that share the
// SM:
//   key side:   dV_tile = P^T . dO and [dK|dKRope]_tile = dS^T . [q || qRope]
//               for 128 keys x 128 features, drained into the fp32 key-row
//               accumulator with vector reductions (deterministic mode:
//               stored as per-pair partial rows for the fixed-order sums);
//   query side: [dQ || dQRope](t) = dS(t) . [K || KRope]_sel, 192 features,
//               accumulated in tensor memory over all the token's keys.
// The key side is bound by the SM-to-L2 reduction path and leaves the tensor
// pipe mostly idle; the query side is bound by gathers and the tensor pipe.
// Running both in the same CTA overlaps the two.  The stores (dQ rows; in
// deterministic mode the partial rows) leave as TMA stores of 2 KB tiles
// staged in shared memory, which keeps them off the request path the
// reductions use.  Key-side items run
// token-major, or tile-group major when the accumulator rows a batch touches
// exceed L2.  (Block indices that many tokens select take kvb.cu for the key
// side and dqb.cu for dQ instead.)
//
// aclnnSparseFlashAttentionGrad doc, 阶段1 (dV = P^T dO) and 阶段3 (dQ, dK);
// MindSpore flash_attention_bwd.py, update_dVj / update_dQi / update_dKj.
#include "common.cuh"
#include "kernels.h"

namespace sfa {

namespace {

constexpr int kThreads = 640;   // 20 warps, roles below
// warp 0: key-side MMA issuer          warp 1: key-side TMA producer
// warp 2: query-side MMA issuer        warp 3: idle
// warps 4-11: key-side drain           warps 12-15: query-side epilogue
// warps 16-17: query-side gather producers, warps 18-19: idle
constexpr int kDrainThreads = 256;

constexpr int kKeys = 128;        // key-side tile (MMA M)
constexpr int kKvStages = 3;      // key-side A stages: 128 slots x 64 heads
constexpr int kKvChunks = 9;      // dK 4 x 128 + dKRope 64, dV 4 x 128
constexpr int kAccRow = 1088;
constexpr int kQSlots = 64;       // query-side keys per stage (MMA K extent)
constexpr int kQStages = 2;       // query-side stages next to the key side
constexpr int kQCol = 192;        // query-side features per item (MMA N)
constexpr int kQParts = 3;

// dynamic shared memory layout (offsets from a 1024-aligned base)
constexpr int kKvB = 0;                                   // 2 feature panels x 128 head rows
constexpr int kKvA = kKvB + 2 * 128 * 128;                // 3 stages x 16 KB
constexpr int kKvAStage = kKeys * 128;
constexpr int kKvStg = kKvA + kKvStages * kKvAStage;      // 8 warps x 32 rows x 32 floats
constexpr int kQ = kKvStg + 8 * 32 * 32 * 4;              // 2 stages x (A 16 KB + B 24 KB)
constexpr int kQA = 2 * kQSlots * 128;
constexpr int kQStage = kQA + (kQCol / 64) * kQSlots * 128;
constexpr int kSmemBytes = kQ + kQStages * kQStage + 1024;

// TMEM columns: key-side accumulators [0,128) and [128,256), query side [256,448)
constexpr uint32_t kQCol0 = 256;

__device__ __forceinline__ void kv_chunk(int ch, int& ncol, int& col0) {
  if (ch < 4) { ncol = 128; col0 = ch * 128; }
  else if (ch == 4) { ncol = 64; col0 = 512; }
  else { ncol = 128; col0 = 576 + (ch - 5) * 128; }
}

// Key-side work item: (tile group, token, feature chunk), tile-group major,
// `tg` tiles per group.  With sorted index lists a token's consecutive
// 128-slot tiles cover ascending key ranges, so while every SM works on the
// same group of tiles the reductions land in a narrow band of key rows that
// stays in L2 even when the whole accumulator does not fit.  When it does
// fit, one group spans all tiles (token-major order, the head rows of a
// chunk loaded once per token).
struct KvItem {
  int tl, ch, kt0, kt1;
};
__device__ __forceinline__ KvItem kv_item(int item, int ntok, int ntiles, int tg) {
  const int per = ntok * kKvChunks;
  const int grp = item / per, r = item - grp * per;
  KvItem it;
  it.tl = r / kKvChunks;
  it.ch = r - it.tl * kKvChunks;
  it.kt0 = grp * tg;
  it.kt1 = it.kt0 + tg < ntiles ? it.kt0 + tg : ntiles;
  return it;
}

__device__ __forceinline__ void red_add_v4(float* dst, float4 x) {
  asm volatile("red.global.add.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(dst), "f"(x.x), "f"(x.y), "f"(x.z), "f"(x.w)
               : "memory");
}

// BLK: block-sparse indices (sparseBlockSize >= 8): the query side loads key
// rows as one TMA box per selected block.  A compile-time switch: the unused
// branch in the row-gather loop alone costs the single-key path a quarter of
// its query-side throughput.
// PART (deterministic = 1): instead of reducing into the accumulator, the
// drain stores every valid (token, slot) pair's 1088-element row, rounded to
// bf16, as element (token_local * Kpad + slot) * 1088 of the bf16 array at
// acc (the partial rows the fixed-order reduction of det.cu sums in fp32);
// masked slots are not written.
template <typename T, int GP, bool BLK, bool PART>
__global__ void __launch_bounds__(kThreads, 1) kvq_kernel(const __grid_constant__ Maps maps, Prob p, float* acc,
                                                          T* dq, T* dqr, int tg, int* gerr) {
  using E = Elt<T>;
  constexpr int QST = kQStages;   // query-side stages
  constexpr int QOFF = kQ;        // offset of the query-side stages
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t kv_full[kKvStages], kv_empty[kKvStages], kv_tfull[2], kv_tempty[2], kv_bfull, kv_bempty;
  __shared__ uint64_t q_full[QST], q_empty[QST], q_tfull, q_tempty, kv_done, q_done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ __align__(16) int q_rows[QST][kQSlots];   // read and written as int2
  // query-side epilogue staging, 2 KB per warp, in the 64-byte swizzle of its
  // TMA stores; PART: the same for each partial-row drain warp
  __shared__ __align__(1024) uint4 q_stage[4][32 * 4];
  __shared__ __align__(1024) uint4 part_stage[PART ? 8 : 1][32 * 4];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = p.Kpad / kKeys;
  const int nkv = (ntiles + tg - 1) / tg * p.ntok * kKvChunks;
  const int qchunks = p.Kpad / kQSlots;
  const int nq = p.ntok * kQParts;

  if (GP == 64) {
    // query side: heads 64-127 do not exist, their A panel stays zero
    for (int s = 0; s < QST; ++s) {
      uint4* z = reinterpret_cast<uint4*>(smem + QOFF + s * kQStage + kQSlots * 128);
      for (int i = threadIdx.x; i < kQSlots * 128 / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
    }
  }
  // key side: the head-row panels start as zeros (the rope chunk loads one)
  for (int i = threadIdx.x; i < 2 * GP * 128 / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + kKvB)[i] = make_uint4(0, 0, 0, 0);
  fence_async_smem();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kKvStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_tfull[i], 1);
      mbar_init(&kv_tempty[i], kDrainThreads / 2);   // one drain group per TMEM set
    }
    mbar_init(&kv_bfull, 1);
    mbar_init(&kv_bempty, 1);
    for (int i = 0; i < QST; ++i) {
      mbar_init(&q_full[i], 32 + 1);   // the owning warp's lanes + the TMA transaction arrive
      mbar_init(&q_empty[i], 1);
    }
    mbar_init(&q_tfull, 1);
    mbar_init(&q_tempty, 128);
    mbar_init(&kv_done, 1);
    mbar_init(&q_done, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  const Waiter wt{&abort_flag, gerr, p.wait_ns};

  if (warp == 0) {
    // ================================================================ key side: MMA issuer
    if (lane == 0) {
      int stage = 0, tcount = 0, icount = 0;
      uint32_t phase = 0;
      bool ok = true;
      const uint64_t da0 = sdesc_kmajor(smem_u32(smem + kKvA), 0);
      const uint64_t db0 = sdesc_mnmajor(smem_u32(smem + kKvB), 0, GP);
      // Reductions: [key slots x features] = [dS | P]^T (K-major, slots on M)
      // . [q | qRope | dO] (MN-major, features on N).  Partial rows (PART):
      // the transpose, [features x key slots] with features on M, so that
      // the drain needs no shared-memory transposition; the rope chunk's
      // second feature panel then holds no data (zeros or an earlier item's
      // rows) and its rows of the result are not drained.
      for (int item = blockIdx.x; item < nkv && ok; item += gridDim.x, ++icount) {
        const KvItem ki = kv_item(item, p.ntok, ntiles, tg);
        int ncol, col0;
        kv_chunk(ki.ch, ncol, col0);
        const uint32_t idesc = PART ? idesc_f16(128, kKeys, E::is_f16, true, false)
                                    : idesc_f16(kKeys, ncol, E::is_f16, false, true);
        ok = mbar_wait_poll(&kv_bfull, icount & 1, wt);
        if (!ok) break;
        for (int kt = ki.kt0; kt < ki.kt1 && ok; ++kt, ++tcount) {
          const int set = tcount & 1;
          ok = mbar_wait_poll(&kv_tempty[set], ((tcount >> 1) & 1) ^ 1, wt);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tbase + set * 128;
          for (int hp = 0; hp < GP / 64 && ok; ++hp) {
            ok = mbar_wait_poll(&kv_full[stage], phase, wt);
            if (!ok) break;
            tc_fence_after();
            if constexpr (PART)
              mma_ss_k64<128, 2>(d, db0 + (uint64_t)(hp * 512), da0 + desc_off(stage * kKvAStage), idesc, hp > 0 ? 1u : 0u);
            else
              mma_ss_k64<2, 128>(d, da0 + desc_off(stage * kKvAStage), db0 + (uint64_t)(hp * 512), idesc, hp > 0 ? 1u : 0u);
            mma_commit(&kv_empty[stage]);
            if (++stage == kKvStages) { stage = 0; phase ^= 1; }
          }
          if (ok) mma_commit(&kv_tfull[set]);
        }
        if (ok) mma_commit(&kv_bempty);
      }
      mma_settle(&kv_done, gerr);   // no MMA still writing tensor memory at exit
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ key side: TMA producer
    // Per item: the token's head rows of q / qRope / dO for the chunk's
    // feature panels (B, kept for the whole item); per key tile and 64-head
    // panel: the staged dS^T or P^T rows (A, 128 slots x 64 heads).
    if (lane == 0) {
      int stage = 0, icount = 0;
      uint32_t phase = 0;
      bool ok = true;
      ArmLog alog_a, alog_b;
      const uint32_t b = smem_u32(smem + kKvB);
      for (int item = blockIdx.x; item < nkv && ok; item += gridDim.x, ++icount) {
        const KvItem ki = kv_item(item, p.ntok, ntiles, tg);
        const int tl = ki.tl, ch = ki.ch;
        const int t = p.tok0 + tl;
        int ncol, col0;
        kv_chunk(ch, ncol, col0);
        if (icount > 0) ok = mbar_wait(&kv_bempty, (icount - 1) & 1, wt);
        if (!ok) break;
        const int npan = ncol / 64;
        mbar_expect_tx(&kv_bfull, npan * GP * 128);
        alog_b.arm(0, (uint32_t)icount);
        for (int pb = 0; pb < npan; ++pb) {
          const CUtensorMap* mp;
          int x, y = t * p.G;
          if (ch >= 5) { mp = &maps.dO; x = col0 - 576 + pb * 64; }
          else if (ch < 4) { mp = &maps.q; x = col0 + pb * 64; }
          else if (p.has_rope) { mp = &maps.qr; x = 0; }
          else { mp = &maps.q; x = 0; y = -2 * GP; }   // no rope part: rows outside the map read as zeros
          tma_2d(b + pb * (GP * 128), mp, x, y, &kv_bfull);
        }
        const CUtensorMap* mA = ch < 5 ? &maps.dS : &maps.P;
        for (int kt = ki.kt0; kt < ki.kt1 && ok; ++kt) {
          const int y0 = tl * p.Kpad + kt * kKeys;
          for (int hp = 0; hp < GP / 64 && ok; ++hp) {
            ok = mbar_wait(&kv_empty[stage], phase ^ 1, wt);
            if (!ok) break;
            const uint32_t a = smem_u32(smem + kKvA + stage * kKvAStage);
            mbar_expect_tx(&kv_full[stage], kKvAStage);
            alog_a.arm(stage, phase);
            tma_2d(a, mA, hp * 64, y0, &kv_full[stage]);
            tma_2d(a + 64 * 128, mA, hp * 64, y0 + 64, &kv_full[stage]);
            if (++stage == kKvStages) { stage = 0; phase ^= 1; }
          }
        }
      }
      // no copy still landing in shared memory at exit
      alog_a.settle(kv_full, gerr);
      alog_b.settle(&kv_bfull, gerr);
    }
    __syncwarp();
  } else if (!PART && warp >= 4 && warp < 12) {
    // ================================================================ key side: reduction drain
    // Two groups of four warps take alternate tiles (group g drains TMEM
    // set g), so one group's reductions overlap the other group's TMEM loads
    // and staging instead of all eight warps pausing together.  Warp w of a
    // group reads TMEM lanes (key slots) 32*(w%4) .. +31 and all of the
    // chunk's columns; each 32-column slice is transposed through a per-warp
    // shared buffer (16-byte chunks XOR-swizzled by row) so that one
    // reduction instruction covers four key rows x 128 contiguous bytes.
    const int qd = warp & 3;
    const int grp = (warp - 4) >> 2;
    const int key = qd * 32 + lane;
    float* stg = reinterpret_cast<float*>(smem + kKvStg) + (warp - 4) * 32 * 32;
    int tcount = 0;
    // the row id of the group's next tile is loaded one tile ahead
    auto row_of = [&](int item, int kt) {
      return item < nkv ? p.rowtab[(size_t)kv_item(item, p.ntok, ntiles, tg).tl * p.Kpad + kt * kKeys + key] : -1;
    };
    auto advance = [&](int& item, int& kt) {
      if (++kt == kv_item(item, p.ntok, ntiles, tg).kt1) {
        item += gridDim.x;
        kt = kv_item(item, p.ntok, ntiles, tg).kt0;
      }
    };
    int nitem = blockIdx.x, nkt = kv_item(blockIdx.x, p.ntok, ntiles, tg).kt0;
    if (grp) advance(nitem, nkt);
    int next_row = row_of(nitem, nkt);
    for (int item = blockIdx.x; item < nkv && !abort_flag; item += gridDim.x) {
      const KvItem ki = kv_item(item, p.ntok, ntiles, tg);
      const int ch = ki.ch;
      int ncol, col0;
      kv_chunk(ch, ncol, col0);
      bool ok = true;
      for (int kt = ki.kt0; kt < ki.kt1; ++kt, ++tcount) {
        const int set = tcount & 1;
        if (set != grp) continue;
        const int row = next_row;
        advance(nitem, nkt);
        advance(nitem, nkt);
        next_row = row_of(nitem, nkt);
        ok = __all_sync(0xffffffffu, mbar_wait(&kv_tfull[set], (tcount >> 1) & 1, wt));
        if (!ok) break;
        tc_fence_after();
        const uint32_t td = tbase + set * 128 + ((uint32_t)(qd * 32) << 16);
        for (int c = 0; c < ncol; c += 32) {
          float v[32];
          tmem_ld32(td + c, v);
          float4* mine = reinterpret_cast<float4*>(stg + lane * 32);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            mine[u ^ (lane & 7)] = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
          __syncwarp();
#pragma unroll
          for (int rr = 0; rr < 8; ++rr) {
            const int rl = rr * 4 + (lane >> 3), c4 = lane & 7;
            const float4 x = reinterpret_cast<const float4*>(stg + rl * 32)[c4 ^ (rl & 7)];
            const int grow = __shfl_sync(0xffffffffu, row, rl);
            if (grow >= 0) red_add_v4(acc + (size_t)grow * kAccRow + col0 + c + c4 * 4, x);
          }
          __syncwarp();
        }
        tc_fence_before();
        mbar_arrive(&kv_tempty[set]);
      }
      if (!ok) break;
    }
  } else if (PART && warp >= 4 && warp < 12) {
    // ================================================================ key side: partial-row drain
    // Two groups of four warps take alternate tiles (group g drains TMEM
    // set g), so one group's reductions overlap the other group's TMEM loads
    // instead of all eight warps pausing together.  A tile is [features x
    // key slots]: warp w of a group reads TMEM lanes (features) 32*(w%4) ..
    // +31 and all 128 slot columns.  Adjacent lanes swap one value, so that
    // each lane holds two consecutive features of one pair's row; per 32
    // slots the warp stages its 32 rows x 32 features in a 2 KB buffer (the
    // 64-byte swizzle) and sends them with one TMA store.  Rows of masked
    // slots are written too; the fixed-order sum reads only valid pairs.
    const int qd = warp & 3;
    const int grp = (warp - 4) >> 2;
    const int odd = lane & 1;
    uint32_t* pst = reinterpret_cast<uint32_t*>(part_stage[PART ? warp - 4 : 0]);
    int tcount = 0;
    for (int item = blockIdx.x; item < nkv && !abort_flag; item += gridDim.x) {
      const KvItem ki = kv_item(item, p.ntok, ntiles, tg);
      const int ch = ki.ch;
      int ncol, col0;
      kv_chunk(ch, ncol, col0);
      // this lane's pair of features within the warp's 32
      const int fl = lane - odd;
      bool ok = true;
      for (int kt = ki.kt0; kt < ki.kt1; ++kt, ++tcount) {
        const int set = tcount & 1;
        if (set != grp) continue;
        ok = __all_sync(0xffffffffu, mbar_wait(&kv_tfull[set], (tcount >> 1) & 1, wt));
        if (!ok) break;
        tc_fence_after();
        if (qd * 32 < ncol) {   // the rope chunk has 64 features: lanes 64-127 hold no result
          const uint32_t td = tbase + set * 128 + ((uint32_t)(qd * 32) << 16);
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            float v[32];
            tmem_ld32(td + 32 * s, v);
            if (lane == 0) bulk_wait_read0();   // the buffer's previous store has read it
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              // even lane: features fl, fl+1 of slot j; odd lane: of slot j+1
              const float x = __shfl_xor_sync(0xffffffffu, odd ? v[j] : v[j + 1], 1);
              const float a = odd ? x : v[j], b = odd ? v[j + 1] : x;
              const int row = j + odd;
              pst[row * 16 + ((((fl >> 3) ^ ((row >> 1) & 3))) << 2) + ((fl & 7) >> 1)] =
                  Elt<__nv_bfloat16>::pack(a, b);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              // the pairs' rows rounded to bf16 (read back once, after this
              // kernel, and summed in fp32)
              tma_store_2d(&maps.partw, col0 + qd * 32, ki.tl * p.Kpad + kt * kKeys + 32 * s, smem_u32(pst));
              bulk_commit();
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&kv_tempty[set]);
      }
      if (!ok) break;
    }
    // the warp's stores are complete before the CTA exits
    if (lane == 0) bulk_wait0();
    __syncwarp();
  } else if (warp == 2) {
    // ================================================================ query side: MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, kQCol, E::is_f16, true, true);
      const uint64_t dqa0 = sdesc_mnmajor(smem_u32(smem + QOFF), 0, kQSlots);
      const uint64_t dqb0 = sdesc_mnmajor(smem_u32(smem + QOFF + kQA), 0, kQSlots);
      const uint32_t d = tbase + kQCol0;
      int it = 0, g = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < nq && ok; item += gridDim.x, ++it) {
        ok = mbar_wait_poll(&q_tempty, (it & 1) ^ 1, wt);
        if (!ok) break;
        tc_fence_after();
        for (int c = 0; c < qchunks; ++c, ++g) {
          const int slot = g % QST;
          ok = mbar_wait_poll(&q_full[slot], (g / QST) & 1, wt);
          if (!ok) break;
          tc_fence_after();
          static_assert(kQSlots == 64, "four K steps per stage");
          mma_ss_k64<128, 128>(d, dqa0 + desc_off(slot * kQStage), dqb0 + desc_off(slot * kQStage), idesc,
                               c == 0 ? 0u : 1u);
          mma_commit(&q_empty[slot]);
        }
        if (ok) mma_commit(&q_tfull);
      }
      mma_settle(&q_done, gerr);   // no MMA still writing tensor memory at exit
    }
    __syncwarp();
  } else if (warp >= 16 && warp < 16 + QST) {
    // ================================================================ query side: gather producers
    // Warp 16 + s owns stage slot s and takes every QST-th stage of 64 keys:
    // the staged dS^T rows as one TMA box per 64-head panel and the keys'
    // feature rows by cp.async; it waits only for its own copies, then fences
    // them for the tensor core and arrives.
    constexpr int kHP = GP / 64;
    constexpr int kCpr = kQCol / 8;
    const int me = warp - 16;
    const T* kmain = static_cast<const T*>(p.k);
    const T* krope = static_cast<const T*>(p.kr);
    const uint32_t a = smem_u32(smem + QOFF + me * kQStage);
    const uint32_t b = a + kQA;
    int* rows = q_rows[me];
    int g = 0;
    bool ok = true;
    ArmLog alog;
    for (int item = blockIdx.x; item < nq && ok; item += gridDim.x) {
      const int tl = item / kQParts, part = item % kQParts;
      const int f0 = part * kQCol;
      for (int c = 0; c < qchunks; ++c, ++g) {
        if (g % QST != me) continue;
        const int2 r2 = *reinterpret_cast<const int2*>(p.rowtab + (size_t)tl * p.Kpad + c * kQSlots + 2 * lane);
        if (lane == 0) ok = mbar_wait(&q_empty[me], ((g / QST) & 1) ^ 1, wt);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        *reinterpret_cast<int2*>(rows + 2 * lane) = r2;
        __syncwarp();
        if (!ok) break;
        constexpr bool blk = BLK;
        if (lane == 0) {
          mbar_expect_tx(&q_full[me], kHP * kQSlots * 128 + (blk ? (kQCol / 64) * kQSlots * 128 : 0));
          alog.arm(me, (uint32_t)(g / QST));
          for (int hp = 0; hp < kHP; ++hp)
            tma_2d(a + hp * (kQSlots * 128), &maps.dS, hp * 64, tl * p.Kpad + c * kQSlots, &q_full[me]);
        }
        if constexpr (blk) {
          // block-sparse indices: each selected block of bs kv rows is one TMA
          // box per 64-feature panel (lane i < 64/bs owns the stage's i-th
          // index); an index with no key at or above 0, past the last row or
          // past the index list reads zeros from below row 0
          __syncwarp();
          const int nidx = kQSlots / p.bs;
          if (lane < nidx) {
            const int i = (c * kQSlots) / p.bs + lane;
            const int t = p.tok0 + tl;
            int y = -p.bs;
            if (i < p.Kidx) {
              const int r = __ldg(p.idx + (size_t)t * p.Kidx + i);
              const long long yy = (long long)p.meta[t].kv_start + r;
              if ((long long)r + p.bs > 0 && yy < p.T2) y = (int)yy;
            }
            for (int pn = 0; pn < kQCol / 64; ++pn) {
              const int f = f0 + pn * 64;
              const uint32_t dst = b + pn * (kQSlots * 128) + lane * p.bs * 128;
              if (f < 512) tma_2d(dst, &maps.k, f, y, &q_full[me]);
              else tma_2d(dst, p.has_rope ? &maps.kr : &maps.k, p.has_rope ? f - 512 : 0, p.has_rope ? y : -p.bs,
                          &q_full[me]);
            }
          }
        } else if (lane < kCpr) {   // lane owns 16-byte piece `lane` of every gathered row
          const int f = f0 + lane * 8;
          const bool rope = f >= 512;
          const T* base = rope ? (p.has_rope ? krope + (f - 512) : kmain) : kmain + f;
          const int rlen = rope ? 64 : 512;
          const bool zero = rope && !p.has_rope;
          const uint32_t dst0 = b + (lane >> 3) * (kQSlots * 128);
          const uint32_t cc = lane & 7;
#pragma unroll 8
          for (int r = 0; r < kQSlots; ++r) {
            const int row = rows[r];
            cp_async16(dst0 + r * 128 + ((cc ^ (r & 7)) << 4), base + (size_t)(row < 0 ? 0 : row) * rlen,
                       (row < 0 || zero) ? 0u : 16u);
          }
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_async_smem();
        mbar_arrive(&q_full[me]);
        __syncwarp();
      }
    }
    alog.settle(q_full, gerr);   // no copy still landing in shared memory at exit
  } else if (warp >= 12 && warp < 16) {
    // ================================================================ query side: epilogue (thread = head)
    // A warp whose 32 heads all exist stages each 32-feature piece of its
    // head rows in a private 2 KB buffer (the 64-byte swizzle) and sends it
    // with one TMA store; a warp with heads past G stores from registers.
    const int ew = warp - 12;
    const int h = ew * 32 + lane;
    const bool tma_rows = ew * 32 + 32 <= p.G;
    uint4* stg = q_stage[ew];
    int it = 0;
    for (int item = blockIdx.x; item < nq && !abort_flag; item += gridDim.x, ++it) {
      const int tl = item / kQParts, part = item % kQParts;
      const int t = p.tok0 + tl;
      const bool ok = mbar_wait(&q_tfull, it & 1, wt);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t td = tbase + kQCol0 + ((uint32_t)(ew * 32) << 16);
      for (int c = 0; c < kQCol; c += 32) {
        float v[32];
        tmem_ld32(td + c, v);
        const int f = part * kQCol + c;
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = E::pack(v[2 * j], v[2 * j + 1]);
        if (tma_rows) {
          if (f >= 512 && !p.has_rope) continue;
          if (lane == 0) bulk_wait_read0();   // the buffer's previous store has read it
          __syncwarp();
#pragma unroll
          for (int u = 0; u < 4; ++u)
            stg[lane * 4 + (u ^ ((lane >> 1) & 3))] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (f < 512) tma_store_2d(&maps.dQw, f, t * p.G + ew * 32, smem_u32(stg));
            else tma_store_2d(&maps.dQRw, f - 512, t * p.G + ew * 32, smem_u32(stg));
            bulk_commit();
          }
          continue;
        }
        T* dst = nullptr;
        if (h < p.G) {
          if (f < 512) dst = dq + ((size_t)t * p.G + h) * 512 + f;
          else if (p.has_rope) dst = dqr + ((size_t)t * p.G + h) * 64 + (f - 512);
        }
        if (dst) {
          uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
          for (int u = 0; u < 4; ++u) d4[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&q_tempty);
    }
    // the warp's stores are complete before the CTA exits
    if (lane == 0) bulk_wait0();
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <typename T, int GP>
cudaError_t launch_gp(const Maps& maps, const Prob& p, float* acc, void* dq, void* dqr, int tile_group, bool part,
                      int* gerr, int nsm, cudaStream_t st) {
  if (tile_group < 1) return cudaErrorInvalidValue;
  auto kern = p.bs >= 8 ? (part ? kvq_kernel<T, GP, true, true> : kvq_kernel<T, GP, true, false>)
                        : (part ? kvq_kernel<T, GP, false, true> : kvq_kernel<T, GP, false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int nitems = p.ntok * kKvChunks;
  const int grid = nitems < nsm ? nitems : nsm;
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, kThreads, kSmemBytes, st>>>(maps, p, acc, static_cast<T*>(dq), static_cast<T*>(dqr), tile_group,
                                           gerr);
  return cudaGetLastError();
}

}  // namespace

template <typename T>
cudaError_t launch_kvq(const Maps& maps, const Prob& p, float* acc, void* dq, void* dqr, int tile_group, bool part,
                       int* gerr, int nsm, cudaStream_t st) {
  if (p.Gp == 64) return launch_gp<T, 64>(maps, p, acc, dq, dqr, tile_group, part, gerr, nsm, st);
  return launch_gp<T, 128>(maps, p, acc, dq, dqr, tile_group, part, gerr, nsm, st);
}

template cudaError_t launch_kvq<__nv_bfloat16>(const Maps&, const Prob&, float*, void*, void*, int, bool, int*, int,
                                               cudaStream_t);
template cudaError_t launch_kvq<__half>(const Maps&, const Prob&, float*, void*, void*, int, bool, int*, int,
                                        cudaStream_t);

}  // namespace sfa
