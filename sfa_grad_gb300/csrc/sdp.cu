// Score / softmax-gradient kernel: for one query token and a tile of 128 of its
// selected keys it recomputes
//     S^T = K_sel . [q || qRope]^T * scale        (tcgen05, keys on M, heads on N)
//     dP^T = V_sel . dO^T
// in tensor memory, then applies the saved softmax statistics:
//     P  = exp(S - softmaxMax) / softmaxSum                (masked keys -> 0)
//     dS = P * (dP - Dsum) * scale
// and writes P^T and dS^T (input dtype, heads contiguous, rows of G rounded
// up to 16 heads) for the later contractions.  The forward's one score pass
// reuses the score half: max/sum partials per 32 keys, with P staged relative
// to each partial's max.
//
// Pipeline: the contraction runs in stages of 128 features (64 for the rope
// part).  The gathered key/value rows (A) and the token's head rows (B) have
// separate rings.  A: four slots (five with 64 heads), each owned by a
// producer warp that takes every fourth (fifth) stage, copies 256 contiguous
// bytes per gathered row by cp.async (scattered 128-byte pieces halve the
// achievable gather rate) and waits only for its own copies, so up to four
// (five) gathers are in flight.  B: two slots
// filled by TMA from one thread.  Both operands of a stage complete on one
// barrier, so the MMA issuer waits once per stage.  Compile-time variants:
// value = key (one gathered stage feeds both contractions) and block indices
// (each selected block of rows arrives as one TMA box per panel).
//
// aclnnSparseFlashAttentionGrad doc, 功能说明 (gather by topkIndices) and
// 阶段1/阶段2 (dP, dS); MindSpore flash_attention_bwd.py, compute_Pij
// (P from saved max and sum) and compute_dSij.
#include "common.cuh"
#include "kernels.h"

namespace sfa {

namespace {

constexpr int kKeys = 128;           // keys per work item (MMA M)
constexpr int kBSlots = 2;           // head-row operand slots (TMA)
constexpr int kGatherWarps = 5;
constexpr int kMaxSlots = 5;         // barrier arrays sized for every ring layout
constexpr int kEpiThreads = 256;     // warps 4-11
// warp 0: MMA issuer; warps 1-3, 12 and 14: gather producers (slots 0-2, 3,
// 4; a warp without a slot of the layout idles); warps 4-11: epilogue;
// warp 13: TMA producer of the head-row operand
constexpr int kThreads = 15 * 32;

// The gathered rows are the stream that sets the kernel's pace (their bytes
// in flight per SM over the L2 latency), so they get the shared memory the
// head rows leave: four 32 KB slots with 128 heads, five with 64 (the head-row
// slots are half as large).
// SH: key and value are the same tensor.  A gathered stage of key rows then
// serves both the score and the dP contraction, so half as many rows are
// gathered; the rings become two gathered slots (two producer warps each,
// one half of the rows per warp) and four head-row slots (q and dO of a
// stage are both resident).
template <int GP, bool SH>
struct SdpSmem {
  static constexpr int kNA = SH ? 2 : (GP == 64 ? 5 : 4);   // gathered slots
  static constexpr int kNB = SH ? 4 : kBSlots;           // head-row slots
  static constexpr int kPanelA = kKeys * 128;   // 64 features x 128 key rows
  static constexpr int kPanelB = GP * 128;      // 64 features x GP head rows
  static constexpr int kA = 2 * kPanelA;                 // one gathered slot
  static constexpr int kB = 2 * kPanelB;                 // one head-row slot
  static constexpr int kBOff = kNA * kA;                 // B ring after the A ring
  static constexpr int kBytes = kBOff + kNB * kB + 1024;  // + alignment slack
};

// Stage c of an item: first source feature, 64-wide panel count, tensors.
struct Chunk {
  int f0;
  int npan;    // 2, or 1 for the rope part
  int kind;    // 0: k / q, 1: kRope / qRope, 2: v / dO
};
__device__ __forceinline__ Chunk chunk_of(int c, int nS) {
  if (c < 4) return Chunk{c * 128, 2, 0};
  if (c < nS) return Chunk{0, 1, 1};
  return Chunk{(c - nS) * 128, 2, 2};
}

// Reduce-scatter across the warp: on entry each lane holds 32 values (one
// per column j); on exit a[0] of lane j holds the max (MAX) or the sum of
// column j over all 32 lanes.  Five exchange steps, each lane keeping the half
// of its columns that its lane bit selects: 31 shuffles instead of 5 per
// column.
template <bool MAX>
__device__ __forceinline__ void butterfly_reduce(float (&a)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = up ? a[i] : a[i + w];
      const float keep = up ? a[i + w] : a[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, w);
      a[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
}

// BLK: block-sparse indices (sparseBlockSize >= 8), key/value rows by TMA boxes.
template <typename T, int GP, int MODE, bool SH, bool BLK>
__global__ void __launch_bounds__(kThreads, 1) sdp_kernel(const __grid_constant__ Maps maps, Prob p, float* tile_stats,
                                                          int* gerr) {
  using E = Elt<T>;
  using S = SdpSmem<GP, SH>;
  static_assert(!SH || MODE == kModeBwd, "the shared key/value layout serves the backward only");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // full_bar[s]: all operands of the stage in gathered slot s are in shared
  // memory (the gather warps' lanes + the head-row TMA transaction arrivals)
  __shared__ uint64_t full_bar[kMaxSlots], empty_bar[kMaxSlots], bempty_bar[kMaxSlots], tfull_bar[2], tempty_bar[2];
  __shared__ uint64_t done_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  // arrivals each producer made on full_bar (head-row TMA thread per slot;
  // gather warps), for the wind-down that completes every phase one of them
  // started
  __shared__ int arr_tma[kMaxSlots], arr_gat[kGatherWarps];
  __shared__ float stats_s[2][3 * GP];
  __shared__ __align__(16) int rows_s[kGatherWarps][kKeys];   // one per gather warp; read and written as int4
  // epilogue row transposition, 2 KB per warp, in the 64-byte swizzle of its TMA stores
  __shared__ __align__(1024) uint4 epi_stage[8][32 * 4];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool bwd = (MODE == kModeBwd);
  const int nS = p.has_rope ? 5 : 4;           // stages of the score contraction
  const int nchunks = bwd ? nS + 4 : nS;      // + 4 stages of dP
  const int ntiles = p.Kpad / kKeys;
  const int nitems = p.ntok * ntiles;
  // head rows per token as loaded (G rounded up to 16); the slot rows from gk
  // to GP are zeroed once here and never written, so padded heads score 0
  const int gk = (p.G + 15) / 16 * 16;
  if (gk < GP) {
    uint4* z = reinterpret_cast<uint4*>(smem + S::kBOff);
    for (int i = threadIdx.x; i < S::kNB * S::kB / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
    fence_async_smem();
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < S::kNA; ++i) {
      // SH: two gather warps + two head-row arrivals; else the owning warp + one
      mbar_init(&full_bar[i], SH ? 64 + 2 : 32 + 1);
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < S::kNB; ++i) mbar_init(&bempty_bar[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      mbar_init(&tempty_bar[i], kEpiThreads);
    }
    mbar_init(&done_bar, 1);
    for (int i = 0; i < kMaxSlots; ++i) arr_tma[i] = 0;
    for (int i = 0; i < kGatherWarps; ++i) arr_gat[i] = 0;
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
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kKeys, GP, E::is_f16, false, false);
      const uint64_t dbase = sdesc_kmajor(smem_u32(smem), 0);
      int it = 0, g = 0, gb = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x, ++it) {
        const int set = it & 1;
        ok = mbar_wait_poll(&tempty_bar[set], ((it >> 1) & 1) ^ 1, wt);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tS = tbase + set * (2 * GP);
        const uint32_t tP = tS + GP;
        if constexpr (SH) {
          // stage c: gathered key rows of chunk c; head rows q_c (and dO_c
          // for the 512-wide part, where the same rows act as value rows)
          for (int c = 0; c < nS; ++c, ++g) {
            const int slot = g % S::kNA;
            ok = mbar_wait_poll(&full_bar[slot], (g / S::kNA) & 1, wt);
            if (!ok) break;
            tc_fence_after();
            const Chunk ck = chunk_of(c, nS);
            const uint64_t da = dbase + desc_off(slot * S::kA);
            const int bs0 = gb % S::kNB;
            const uint64_t db0 = dbase + desc_off(S::kBOff + bs0 * S::kB);
            mma_ss_k64<2, 2>(tS, da, db0, idesc, c == 0 ? 0u : 1u);
            if (ck.npan == 2) mma_ss_k64<2, 2>(tS, da + desc_off(S::kPanelA), db0 + desc_off(S::kPanelB), idesc, 1u);
            mma_commit(&bempty_bar[bs0]);
            ++gb;
            if (ck.kind == 0) {
              const int bs1 = gb % S::kNB;
              const uint64_t db1 = dbase + desc_off(S::kBOff + bs1 * S::kB);
              mma_ss_k64<2, 2>(tP, da, db1, idesc, c == 0 ? 0u : 1u);
              mma_ss_k64<2, 2>(tP, da + desc_off(S::kPanelA), db1 + desc_off(S::kPanelB), idesc, 1u);
              mma_commit(&bempty_bar[bs1]);
              ++gb;
            }
            mma_commit(&empty_bar[slot]);
          }
        } else {
          for (int c = 0; c < nchunks; ++c, ++g) {
            const int slot = g % S::kNA, bslot = g % S::kNB;
            ok = mbar_wait_poll(&full_bar[slot], (g / S::kNA) & 1, wt);
            if (!ok) break;
            tc_fence_after();
            const Chunk ck = chunk_of(c, nS);
            const uint64_t da = dbase + desc_off(slot * S::kA);
            const uint64_t db = dbase + desc_off(S::kBOff + bslot * S::kB);
            const uint32_t d = c < nS ? tS : tP;
            const bool first = (c == 0 || c == nS);
            mma_ss_k64<2, 2>(d, da, db, idesc, first ? 0u : 1u);
            if (ck.npan == 2) mma_ss_k64<2, 2>(d, da + desc_off(S::kPanelA), db + desc_off(S::kPanelB), idesc, 1u);
            mma_commit(&empty_bar[slot]);
            mma_commit(&bempty_bar[bslot]);
          }
        }
        if (!ok) break;
        mma_commit(&tfull_bar[set]);
      }
      mma_settle(&done_bar, gerr);   // no MMA still writing tensor memory at exit
    }
    __syncwarp();
  } else if (warp == 13) {
    // ---------------------------------------------------------------- head-row operand (TMA)
    if (lane == 0) {
      int g = 0, gb = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x) {
        const int t = p.tok0 + item / ntiles;
        if constexpr (SH) {
          for (int c = 0; c < nS && ok; ++c, ++g) {
            const Chunk ck = chunk_of(c, nS);
            uint64_t* fb = &full_bar[g % S::kNA];
            const int nb = ck.kind == 0 ? 2 : 1;
            // The stage barrier's previous phase (stage g - 2) must be over
            // before this stage's transactions are posted on it; the head-row
            // slot waits alone do not imply that once a one-load rope stage
            // shifts the head-row sequence.
            ok = mbar_wait(&empty_bar[g % S::kNA], ((g / S::kNA) & 1) ^ 1, wt);
            if (!ok) break;
            for (int j = 0; j < nb && ok; ++j, ++gb) {
              const int bslot = gb % S::kNB;
              ok = mbar_wait(&bempty_bar[bslot], ((gb / S::kNB) & 1) ^ 1, wt);
              if (!ok) break;
              const uint32_t b = smem_u32(smem + S::kBOff + bslot * S::kB);
              mbar_expect_tx(fb, ck.npan * gk * 128);
              ++arr_tma[g % S::kNA];
              const CUtensorMap* mq = j == 1 ? &maps.dOg : ck.kind == 0 ? &maps.qg : &maps.qrg;
              for (int pn = 0; pn < ck.npan; ++pn) tma_2d(b + pn * S::kPanelB, mq, ck.f0 + pn * 64, t * p.G, fb);
            }
            if (ok && nb == 1) {   // the stage barrier counts two head-row arrivals
              mbar_arrive(fb);
              ++arr_tma[g % S::kNA];
            }
          }
        } else {
          for (int c = 0; c < nchunks && ok; ++c, ++g) {
            const int bslot = g % S::kNB;
            ok = mbar_wait(&bempty_bar[bslot], ((g / S::kNB) & 1) ^ 1, wt);
            if (!ok) break;
            const Chunk ck = chunk_of(c, nS);
            const uint32_t b = smem_u32(smem + S::kBOff + bslot * S::kB);
            uint64_t* fb = &full_bar[g % S::kNA];
            mbar_expect_tx(fb, ck.npan * gk * 128);
            ++arr_tma[g % S::kNA];
            const CUtensorMap* mq = ck.kind == 0 ? &maps.qg : ck.kind == 1 ? &maps.qrg : &maps.dOg;
            for (int pn = 0; pn < ck.npan; ++pn) tma_2d(b + pn * S::kPanelB, mq, ck.f0 + pn * 64, t * p.G, fb);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp <= 3 || warp == 12 || warp == 14) {
    // ---------------------------------------------------------------- gather producers
    // Without SH warp me owns slot me and all 128 rows of its stages; with SH
    // warps 2s and 2s+1 share slot s, one half of the rows each.
    const int me = warp == 12 ? 3 : warp == 14 ? 4 : warp - 1;
    const int slot = SH ? (me >> 1) : me;
    const int r0 = SH ? (me & 1) * (kKeys / 2) : 0;
    const int r1 = SH ? r0 + kKeys / 2 : kKeys;
    const int nst = SH ? nS : nchunks;           // stages that gather rows
    const T* k = static_cast<const T*>(p.k);
    const T* kr = static_cast<const T*>(p.kr);
    const T* v = static_cast<const T*>(p.v);
    const uint32_t a = smem_u32(smem + slot * S::kA);
    int* rows = rows_s[me];
    // Block-sparse indices (sparseBlockSize >= 8): a selected block is bs
    // contiguous kv rows, fetched as one TMA box per 64-feature panel.  Lane
    // i < nidx owns the i-th index of the warp's rows and keeps the first kv
    // row of its block; an index with no key at or above 0, or past the last
    // row, reads rows below row 0, which arrive as zeros.  Keys of a block
    // outside its segment or past the causal limit hold finite data and are
    // masked by the epilogue from the row table.
    constexpr bool blk = BLK;
    const int nidx = blk ? (r1 - r0) / p.bs : 0;
    // an item's 128 kv rows (-1: masked), or with block indices the lane's
    // first block row in .x, loaded one item ahead
    auto rows_of = [&](int item) {
      if (item >= nitems) return make_int4(-p.bs, -1, -1, -1);
      if constexpr (blk) {
        const int tl = item / ntiles, kt = item % ntiles, t = p.tok0 + tl;
        const int i = (kt * kKeys + r0) / p.bs + lane;
        int y = -p.bs;
        if (lane < nidx && i < p.Kidx) {
          // keys r .. r+bs-1; a start below 0 still covers keys 0 .. r+bs-1
          // (rows below the segment, or below row 0, are masked or zeros)
          const int r = __ldg(p.idx + (size_t)t * p.Kidx + i);
          const long long yy = (long long)p.meta[t].kv_start + r;
          if ((long long)r + p.bs > 0 && yy < p.T2) y = (int)yy;
        }
        return make_int4(y, -1, -1, -1);
      }
      return *reinterpret_cast<const int4*>(p.rowtab + (size_t)(item / ntiles) * p.Kpad + (item % ntiles) * kKeys +
                                            4 * lane);
    };
    int4 next4 = rows_of(blockIdx.x);
    int cur_y = -p.bs;
    int g = 0, loaded_item = -1;
    bool ok = true;
    for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x) {
      for (int c = 0; c < nst; ++c, ++g) {
        if (g % S::kNA != slot) continue;
        if (loaded_item != item) {
          if (blk) cur_y = next4.x;
          else *reinterpret_cast<int4*>(rows + 4 * lane) = next4;
          next4 = rows_of(item + gridDim.x);
          loaded_item = item;
        }
        if (lane == 0) ok = mbar_wait(&empty_bar[slot], ((g / S::kNA) & 1) ^ 1, wt);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();
        if (!ok) break;
        const Chunk ck = chunk_of(c, nS);
        if constexpr (blk) {
          if (lane == 0) mbar_expect_tx(&full_bar[slot], (uint32_t)(nidx * p.bs * 128 * ck.npan));
          __syncwarp();
          if (lane < nidx) {
            const CUtensorMap* mk = ck.kind == 0 ? &maps.k : ck.kind == 1 ? &maps.kr : &maps.v;
            const uint32_t dst = a + (uint32_t)(r0 + lane * p.bs) * 128;
            for (int pn = 0; pn < ck.npan; ++pn) tma_2d(dst + pn * S::kPanelA, mk, ck.f0 + pn * 64, cur_y, &full_bar[slot]);
          }
          if (lane != 0) mbar_arrive(&full_bar[slot]);
          if (lane == 0) arr_gat[me] += 32;
          continue;
        }
        // gathered rows, contiguous in global memory: with two panels a lane
        // owns 16-byte piece (lane & 15) of rows (lane >> 4) + 2i; with one
        // panel piece (lane & 7) of rows (lane >> 3) + 4i
        if (ck.npan == 2) {
          const T* base = (ck.kind == 0 ? k : v) + ck.f0 + (lane & 15) * 8;
          const uint32_t dst0 = a + ((lane >> 3) & 1) * S::kPanelA;
          const uint32_t c = lane & 7;
#pragma unroll 8
          for (int r = r0 + (lane >> 4); r < r1; r += 2) {
            const int row = rows[r];
            cp_async16(dst0 + r * 128 + ((c ^ (r & 7)) << 4), base + (size_t)(row < 0 ? 0 : row) * 512,
                       row < 0 ? 0u : 16u);
          }
        } else {
          const T* base = kr + (lane & 7) * 8;
          const uint32_t c = lane & 7;
#pragma unroll 8
          for (int r = r0 + (lane >> 3); r < r1; r += 4) {
            const int row = rows[r];
            cp_async16(a + r * 128 + ((c ^ (r & 7)) << 4), base + (size_t)(row < 0 ? 0 : row) * 64, row < 0 ? 0u : 16u);
          }
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_async_smem();
        mbar_arrive(&full_bar[slot]);
        if (lane == 0) arr_gat[me] += 32;
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ---------------------------------------------------------------- epilogue
    // Eight warps: warp w reads TMEM lanes (keys) 32*(w%4) .. +31 and the
    // head half (w-4)/4, i.e. heads [half*GP/2, (half+1)*GP/2).  Named
    // barriers between these warps run every item, so the trip count never
    // depends on the abort flag: an abandoned wait only skips the item's work.
    const int q = warp & 3;
    const int half = (warp - 4) >> 2;
    const int key = q * 32 + lane;
    const int etid = threadIdx.x - 128;
    constexpr int HH = GP / 2;
    const float sl2 = p.scale * kLog2e;
    // The next item's key validity and per-head statistics (softmaxMax,
    // softmaxSum, Dsum of head etid) are loaded one item ahead, so their
    // latency hides behind the current item's work.
    auto fetch = [&](int item, int& rowv, float& a, float& b, float& c) {
      rowv = -1;
      a = b = c = 0.f;
      if (item >= nitems) return;
      const int tl = item / ntiles, kt = item % ntiles;
      const int t = p.tok0 + tl;
      rowv = p.rowtab[(size_t)tl * p.Kpad + kt * kKeys + key];
      if (MODE != kModeFwdStats && etid < p.G) {
        a = __ldg(p.smax + (size_t)t * p.G + etid);
        b = __ldg(p.ssum + (size_t)t * p.G + etid);
        if (bwd) c = __ldg(p.dsum + (size_t)t * p.G + etid);
      }
    };
    // A lane holds 32 heads (64 bytes) of its own key row.  The warp's 32
    // rows go to a private shared buffer (16-byte piece u of row r at
    // position u ^ ((r >> 1) & 3): the 64-byte swizzle) and leave as one TMA
    // store of 32 rows x 32 heads, so the warp does not wait for them.
    // Staged rows hold Gs heads (G rounded up to 16); the store map ends at
    // Gs, so heads past it are not written.
    const int Gs = p.Gs;
    uint4* stg = epi_stage[warp - 4];
    // the buffer may be written once this warp's last store has read it
    auto stg_free = [&]() {
      if (lane == 0) bulk_wait_read0();
      __syncwarp();
    };
    auto put_rows = [&](const uint32_t* pk, const CUtensorMap* map, int x, int y) {
      stg_free();
#pragma unroll
      for (int u = 0; u < 4; ++u)
        stg[lane * 4 + (u ^ ((lane >> 1) & 3))] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(map, x, y, smem_u32(stg));
        bulk_commit();
      }
    };
    int nrow;
    float nmax, nsum, ndsum;
    fetch(blockIdx.x, nrow, nmax, nsum, ndsum);
    int it = 0;
    for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++it) {
      const int set = it & 1;
      const uint32_t tph = (it >> 1) & 1;
      const int tl = item / ntiles, kt = item % ntiles;
      const bool valid = nrow >= 0;
      float* st = stats_s[it & 1];
      if (MODE != kModeFwdStats && etid < GP) {
        // exponent offset, 1/sum (0 for an empty row or a padded head), Dsum * scale
        const bool live = nsum > 0.f;
        st[etid] = live ? nmax * kLog2e : 0.f;
        st[GP + etid] = live ? 1.f / nsum : 0.f;
        st[2 * GP + etid] = ndsum * p.scale;
      }
      fetch(item + gridDim.x, nrow, nmax, nsum, ndsum);
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
      const bool ok = __all_sync(0xffffffffu, !abort_flag && mbar_wait(&tfull_bar[set], tph, wt));
      if (ok) tc_fence_after();
      const uint32_t tS = tbase + set * (2 * GP) + ((uint32_t)(q * 32) << 16);
      const uint32_t tP = tS + GP;
      if (MODE == kModeFwdStats) {
        // Per head over the warp's 32 keys (one group of the token's slots):
        // m = max of the raw score s over the valid keys, l = sum of
        // exp((s - m) * scale), and P~ = exp((s - m) * scale) staged in the P
        // rows (0 for a masked key).  The P.V kernel rescales each group's P~
        // to the final statistics, so no second score pass is needed.
        const int row0 = tl * p.Kpad + kt * kKeys + q * 32;   // the warp's 32 staged rows
        float2* tsg = reinterpret_cast<float2*>(tile_stats) + ((size_t)tl * (ntiles * 4) + kt * 4 + q) * p.G;
#pragma unroll 1
        for (int c = 0; c < HH / 32; ++c) {
          const int h0 = half * HH + c * 32;
          if (h0 >= Gs) break;                       // padded heads only: nothing is staged
          // per-head max over the 32 lanes (keys): lane j ends with head j's;
          // every lane then reads all 32 from the warp's staging buffer.  The
          // scores are read from tensor memory twice (for the max, then for
          // the exponentials) so that one 32-value array is live at a time.
          float a[32];
          if (ok) tmem_ld32(tS + h0, a);
#pragma unroll
          for (int j = 0; j < 32; ++j) a[j] = (valid && ok) ? a[j] : -INFINITY;
          butterfly_reduce<true>(a, lane);
          const float gm = a[0];
          float* mrow = reinterpret_cast<float*>(stg);
          stg_free();
          mrow[lane] = gm;
          __syncwarp();
          if (ok) tmem_ld32(tS + h0, a);
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(mrow + j);
            const float mj[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) a[j + u] = (valid && ok) ? ex2((a[j + u] - mj[u]) * sl2) : 0.f;
            pk[j / 2] = E::pack(a[j], a[j + 1]);
            pk[j / 2 + 1] = E::pack(a[j + 2], a[j + 3]);
          }
          __syncwarp();
          butterfly_reduce<false>(a, lane);
          const float gl = a[0];
          if (ok) {
            if (h0 + lane < p.G) tsg[h0 + lane] = make_float2(gm, gl);   // raw score (unscaled), sum
            put_rows(pk, &maps.Pw, h0, row0);
          }
        }
        tc_fence_before();
        if (ok) mbar_arrive(&tempty_bar[set]);
        continue;
      }
      if (!ok) continue;
      const int row0 = tl * p.Kpad + kt * kKeys + q * 32;   // the warp's 32 staged rows
#pragma unroll 1
      for (int c = 0; c < HH / 32; ++c) {
        const int h0 = half * HH + c * 32;
        if (h0 >= Gs) break;                       // padded heads only: nothing is staged
        float s[32], dp[32];
        tmem_ld32(tS + h0, s);
        if (bwd) tmem_ld32(tP + h0, dp);
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          float pv[2], dv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int h = h0 + j + u;
            const float x = valid ? fmaf(s[j + u], sl2, -st[h]) : -INFINITY;
            const float pp = ex2(x) * st[GP + h];
            pv[u] = pp;
            // pp == 0 for a masked key: its dS is 0 even if the (unused) value
            // row it was computed from is not finite
            dv[u] = (bwd && pp != 0.f) ? pp * fmaf(dp[j + u], p.scale, -st[2 * GP + h]) : 0.f;
          }
          pk[j / 2] = E::pack(pv[0], pv[1]);
          dk[j / 2] = E::pack(dv[0], dv[1]);
        }
        put_rows(pk, &maps.Pw, h0, row0);
        if (bwd) put_rows(dk, &maps.dSw, h0, row0);
      }
      tc_fence_before();
      mbar_arrive(&tempty_bar[set]);
    }
    // the warp's stores are complete before the CTA exits
    if (lane == 0) bulk_wait0();
    __syncwarp();
  }
  // Wind-down.  A stage barrier collects arrivals from two producers (the
  // gather warps and the head-row TMA thread); after an abandoned wait one of
  // them may have started a phase the other never joined, with copies of the
  // first still in flight.  Thread 0 completes every started phase with the
  // missing arrivals and waits for each, so that no copy lands after the CTA
  // exits.  The producers' roles are one phase apart at most per slot.
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kNA; ++s) {
      constexpr int kTShare = SH ? 2 : 1;                // head-row arrivals per phase
      int n[3], sh[3], nr = 0;
      n[nr] = arr_tma[s], sh[nr++] = kTShare;
      for (int w = 0; w < kGatherWarps; ++w)
        if ((SH ? (w >> 1) : w) == s) n[nr] = arr_gat[w], sh[nr++] = 32;
      int klo = 1 << 30, khi = 0;
      for (int r = 0; r < nr; ++r) {
        klo = min(klo, n[r] / sh[r]);
        khi = max(khi, (n[r] + sh[r] - 1) / sh[r]);
      }
      if (klo >= 1) mbar_settle(&full_bar[s], (uint32_t)(klo - 1) & 1u, gerr);
      for (int k = klo; k < khi; ++k) {
        int missing = 0;
        for (int r = 0; r < nr; ++r) missing += sh[r] - min(max(n[r] - k * sh[r], 0), sh[r]);
        if (missing > 0) mbar_arrive_n(&full_bar[s], (uint32_t)missing);
        mbar_settle(&full_bar[s], (uint32_t)k & 1u, gerr);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <typename T, int GP, int MODE, bool SH = false>
cudaError_t launch_one(const Maps& maps, const Prob& p, float* tile_stats, int* gerr, int nsm,
                       cudaStream_t st) {
  auto kern = p.bs >= 8 ? sdp_kernel<T, GP, MODE, SH, true> : sdp_kernel<T, GP, MODE, SH, false>;
  using S = SdpSmem<GP, SH>;
  const int smem = S::kBytes > kOneCtaSmem ? S::kBytes : kOneCtaSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nitems = p.ntok * (p.Kpad / kKeys);
  const int grid = nitems < nsm ? nitems : nsm;
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, kThreads, smem, st>>>(maps, p, tile_stats, gerr);
  return cudaGetLastError();
}

}  // namespace

template <typename T>
cudaError_t launch_sdp(const Maps& maps, const Prob& p, int mode, float* tile_stats, int* gerr, int nsm,
                       cudaStream_t st) {
  // key and value given as the same tensor: gather the rows once per stage
  const bool shared_kv = p.k == p.v;
  if (p.Gp == 64) {
    if (mode == kModeBwd && shared_kv) return launch_one<T, 64, kModeBwd, true>(maps, p, tile_stats, gerr, nsm, st);
    if (mode == kModeBwd) return launch_one<T, 64, kModeBwd>(maps, p, tile_stats, gerr, nsm, st);
    if (mode == kModeFwdStats) return launch_one<T, 64, kModeFwdStats>(maps, p, tile_stats, gerr, nsm, st);
    return cudaErrorInvalidValue;
  }
  if (mode == kModeBwd && shared_kv) return launch_one<T, 128, kModeBwd, true>(maps, p, tile_stats, gerr, nsm, st);
  if (mode == kModeBwd) return launch_one<T, 128, kModeBwd>(maps, p, tile_stats, gerr, nsm, st);
  if (mode == kModeFwdStats) return launch_one<T, 128, kModeFwdStats>(maps, p, tile_stats, gerr, nsm, st);
  return cudaErrorInvalidValue;
}

template cudaError_t launch_sdp<__nv_bfloat16>(const Maps&, const Prob&, int, float*, int*, int, cudaStream_t);
template cudaError_t launch_sdp<__half>(const Maps&, const Prob&, int, float*, int*, int, cudaStream_t);

}  // namespace sfa
