// The companion forward's output over a token's selected keys, on the tensor
// cores:  O(t) = P(t) . V_sel  (2 items of 256 features per token).  The
// score kernel's statistics pass (sdp.cu) staged P~ = exp((s - m_g) * scale)
// relative to the max m_g of each group of 32 of the token's slots; the
// producers rescale every stage's P~ in shared memory by the group's factor
// exp((m_g - m) * scale) / l, which gives P for the final statistics m, l
// (softmaxMax = m * scale, softmaxSum = l) without a second score pass.
// Heads on M (padded to 128), features on N, keys (64 per pipeline stage) on
// K; the accumulator stays in tensor memory for the whole key loop and is
// written once.  (The backward's dQ has the same shape and runs in kvq.cu,
// next to the key side; block indices use dqb.cu for both.)
//
// aclnnSparseFlashAttentionGrad doc, 功能说明 (selectedValue gathered by
// topkIndices); MindSpore flash_attention_bwd.py, the forward's O = P V.
#include "common.cuh"
#include "kernels.h"

namespace sfa {

namespace {

constexpr int kSlots = 64;         // keys per pipeline stage (MMA K extent)
// A stage: the staged P of 64 keys (one 64-head panel per 64 heads),
// then the gathered rows' feature panels.  With 64 heads the MMA's rows
// 64-127 read the stage's first feature panel (the A operand's second
// 64-row atom lies one panel further on): finite data whose results are
// never stored; the stage is smaller and one more fits.
// warp 0: MMA issuer, warps 1..NST: producers (one per stage slot), then four
// epilogue warps (TMEM lane quadrant = warp % 4)
template <int NCOL, int GP>
struct DqSmem {
  static constexpr int kA = (GP / 64) * kSlots * 128;    // head panels
  static constexpr int kB = (NCOL / 64) * kSlots * 128;  // feature panels
  static constexpr int kStage = kA + kB;
  static constexpr int NST = GP == 64 ? 5 : 4;
  static constexpr int kBytes = NST * kStage + 1024;
  static constexpr int kThreads = (1 + NST + 4) * 32;
};

// BLK: block-sparse indices (sparseBlockSize >= 8): the key / value rows of a
// stage arrive as one TMA box per selected block and feature panel.
constexpr int NCOL = 256;     // features per item (MMA N)
constexpr int NPART = 2;      // items per token

template <typename T, int GP, bool BLK>
__global__ void __launch_bounds__(DqSmem<NCOL, GP>::kThreads, 1)
    dq_kernel(const __grid_constant__ Maps maps, Prob p, const float* part_stats, T* out, int* gerr) {
  using E = Elt<T>;
  using S = DqSmem<NCOL, GP>;
  constexpr int kStages = S::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // pfull_bar: the stage's staged P~ has landed (to be rescaled); full_bar:
  // the whole stage is ready for the MMA
  __shared__ uint64_t full_bar[kStages], pfull_bar[kStages], empty_bar[kStages], tfull_bar[2], tempty_bar[2], done_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ __align__(16) int rows_s[kStages][kSlots];   // read and written as int2
  // epilogue staging, 2 KB per warp, in the 64-byte swizzle of its TMA stores
  __shared__ __align__(1024) uint4 o_stage[4][32 * 4];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunks = p.Kpad / kSlots;
  const int nitems = p.ntok * NPART;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 32 + 1);   // the owning warp's lanes + one arrival with the value boxes' bytes
      mbar_init(&pfull_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      mbar_init(&tempty_bar[i], 128);
    }
    mbar_init(&done_bar, 1);
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
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, NCOL, E::is_f16, true, true);
      const uint64_t da0 = sdesc_mnmajor(smem_u32(smem), 0, kSlots);
      const uint64_t db0 = sdesc_mnmajor(smem_u32(smem + S::kA), 0, kSlots);
      int it = 0, g = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x, ++it) {
        const int set = it & 1;
        ok = mbar_wait_poll(&tempty_bar[set], ((it >> 1) & 1) ^ 1, wt);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tbase + set * 256;
        for (int c = 0; c < nchunks; ++c, ++g) {
          const int slot = g % kStages;
          ok = mbar_wait_poll(&full_bar[slot], (g / kStages) & 1, wt);
          if (!ok) break;
          tc_fence_after();
          static_assert(kSlots == 64, "four K steps per stage");
          mma_ss_k64<128, 128>(d, da0 + desc_off(slot * S::kStage), db0 + desc_off(slot * S::kStage), idesc,
                               c == 0 ? 0u : 1u);
          mma_commit(&empty_bar[slot]);
        }
        if (!ok) break;
        mma_commit(&tfull_bar[set]);
      }
      mma_settle(&done_bar, gerr);   // no MMA still writing tensor memory at exit
    }
    __syncwarp();
  } else if (warp <= kStages) {
    // ---------------------------------------------------------------- producers
    // Warp w owns stage slot w-1 and takes every NST-th stage of 64 keys: the
    // staged P~^T rows as one TMA box per 64-head panel, and the keys' value
    // rows gathered by cp.async (NCOL contiguous features per row).  While the
    // value rows are in flight the warp rescales the landed P~ in place (lane:
    // one 16-byte piece of 8 heads in kRPL consecutive rows, all in one group
    // of 32 slots), then waits for its own copies, fences them and its stores
    // for the tensor core and arrives.
    constexpr int kHP = GP / 64;
    constexpr int kCpr = NCOL / 8;            // 16-byte pieces per gathered row
    constexpr int kCPR = 8 * kHP;             // 16-byte pieces per staged P~ row
    constexpr int kRPL = kSlots * kCPR / 32;  // P~ rows per lane
    static_assert(kRPL == 16 || kRPL == 32, "a lane's rows lie in one group of 32 slots");
    const int pc = lane % kCPR, rs = lane / kCPR;
    const int hb = (pc >> 3) * 64 + (pc & 7) * 8;   // the lane's first head
    const int ngroups = p.Kpad / 32;
    const int me = warp - 1;
    const CUtensorMap* mA = &maps.P;
    const T* vrow = static_cast<const T*>(p.v);
    const uint32_t a = smem_u32(smem + me * S::kStage);
    const uint32_t b = a + S::kA;
    int* rows = rows_s[me];
    int g = 0;
    bool ok = true;
    ArmLog alog, plog;
    for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x) {
      const int tl = item / NPART, part = item % NPART;
      const int f0 = part * NCOL;
      // the final statistics of the lane's 8 heads: softmaxMax in log2 units
      // and 1 / softmaxSum (0 for a head past G or without a valid key)
      float nm[8], il[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int h = hb + u;
        const size_t o = (size_t)(p.tok0 + tl) * p.G + h;
        const float l = h < p.G ? __ldg(p.ssum + o) : 0.f;
        nm[u] = h < p.G ? __ldg(p.smax + o) * kLog2e : 0.f;
        il[u] = l > 0.f ? 1.f / l : 0.f;
      }
      for (int c = 0; c < nchunks; ++c, ++g) {
        if (g % kStages != me) continue;
        const int2 r2 = *reinterpret_cast<const int2*>(p.rowtab + (size_t)tl * p.Kpad + c * kSlots + 2 * lane);
        if (lane == 0) ok = mbar_wait(&empty_bar[me], ((g / kStages) & 1) ^ 1, wt);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        *reinterpret_cast<int2*>(rows + 2 * lane) = r2;
        __syncwarp();
        if (!ok) break;
        const uint32_t ph = (uint32_t)(g / kStages);
        if (lane == 0) {
          mbar_expect_tx(&pfull_bar[me], kHP * kSlots * 128);
          plog.arm(me, ph);
          for (int hp = 0; hp < kHP; ++hp)
            tma_2d(a + hp * (kSlots * 128), mA, hp * 64, tl * p.Kpad + c * kSlots, &pfull_bar[me]);
          mbar_expect_tx(&full_bar[me], BLK ? (NCOL / 64) * kSlots * 128 : 0);
          alog.arm(me, ph);
        }
        // the group maxima of the lane's 8 heads (-inf past the heads), loaded
        // now and used once the value rows are in flight
        float mg[8];
        {
          const int grp = (c * kSlots + rs * kRPL) / 32;
          const float* ps = part_stats + ((size_t)tl * ngroups + grp) * p.G * 2;
#pragma unroll
          for (int u = 0; u < 8; ++u) mg[u] = hb + u < p.G ? __ldg(ps + 2 * (hb + u)) : -INFINITY;
        }
        if constexpr (BLK) {
          // lane i < 64/bs owns the stage's i-th index: one box of bs rows per
          // feature panel (an index with no key at or above 0, past the last
          // row or past the index list reads zeros from below row 0)
          __syncwarp();
          const int nidx = kSlots / p.bs;
          if (lane < nidx) {
            const int i = (c * kSlots) / p.bs + lane;
            const int t = p.tok0 + tl;
            int y = -p.bs;
            if (i < p.Kidx) {
              const int r = __ldg(p.idx + (size_t)t * p.Kidx + i);
              const long long yy = (long long)p.meta[t].kv_start + r;
              if ((long long)r + p.bs > 0 && yy < p.T2) y = (int)yy;
            }
            for (int pn = 0; pn < NCOL / 64; ++pn) {
              const int f = f0 + pn * 64;
              const uint32_t dst = b + pn * (kSlots * 128) + lane * p.bs * 128;
              tma_2d(dst, &maps.v, f, y, &full_bar[me]);
            }
          }
        } else if (lane < kCpr) {   // lane < kCpr owns 16-byte piece `lane` of every gathered row
          const T* base = vrow + f0 + lane * 8;
          const uint32_t dst0 = b + (lane >> 3) * (kSlots * 128);
          const uint32_t c = lane & 7;
#pragma unroll 8
          for (int r = 0; r < kSlots; ++r) {
            const int row = rows[r];
            cp_async16(dst0 + r * 128 + ((c ^ (r & 7)) << 4), base + (size_t)(row < 0 ? 0 : row) * 512,
                       row < 0 ? 0u : 16u);
          }
        }
        cp_async_commit();
        // the factors exp((m_g - m) * scale) / l, as pairs in the input type
        // (0 past the heads, or for a group without a valid key, whose P~ is 0)
        uint32_t fac[4];
        {
          const float sl2 = p.scale * kLog2e;
          float f[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) f[u] = mg[u] == -INFINITY ? 0.f : ex2(fmaf(mg[u], sl2, -nm[u])) * il[u];
#pragma unroll
          for (int u = 0; u < 4; ++u) fac[u] = E::pack(f[2 * u], f[2 * u + 1]);
        }
        // P = P~ x factor, in place, once the staged rows have landed
        const bool pok = __all_sync(0xffffffffu, mbar_wait(&pfull_bar[me], ph & 1u, wt));
        if (pok) {
          // eight rows at a time: all loads, then all stores, so that the
          // loads overlap instead of each waiting behind the previous store
          const uint32_t pb = a + (pc >> 3) * (kSlots * 128) + (uint32_t)(rs * kRPL) * 128;
#pragma unroll
          for (int i0 = 0; i0 < kRPL; i0 += 8) {
            uint4 w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) w[j] = lds128(pb + (i0 + j) * 128 + (((pc & 7) ^ ((i0 + j) & 7)) << 4));
#pragma unroll
            for (int j = 0; j < 8; ++j)
              sts128(pb + (i0 + j) * 128 + (((pc & 7) ^ ((i0 + j) & 7)) << 4),
                     make_uint4(E::mul2(w[j].x, fac[0]), E::mul2(w[j].y, fac[1]), E::mul2(w[j].z, fac[2]),
                                E::mul2(w[j].w, fac[3])));
          }
        }
        cp_async_wait<0>();
        fence_async_smem();
        mbar_arrive(&full_bar[me]);
        __syncwarp();
        if (!pok) {
          ok = false;
          break;
        }
      }
    }
    // no copy still landing in shared memory at exit
    plog.settle(pfull_bar, gerr);
    alog.settle(full_bar, gerr);
  } else if (warp > kStages) {
    // ---------------------------------------------------------------- epilogue (thread = head)
    // A warp whose 32 heads all exist stages each 32-feature piece of its
    // head rows in a private 2 KB buffer (the 64-byte swizzle) and sends it
    // with one TMA store; a warp with heads past G stores from registers.
    const int ew = warp & 3;   // the TMEM lane quadrant this warp may read
    const int h = ew * 32 + lane;
    const bool tma_rows = ew * 32 + 32 <= p.G;
    uint4* stg = o_stage[ew];
    int it = 0;
    for (int item = blockIdx.x; item < nitems && !abort_flag; item += gridDim.x, ++it) {
      const int set = it & 1;
      const int tl = item / NPART, part = item % NPART;
      const int t = p.tok0 + tl;
      const bool ok = mbar_wait(&tfull_bar[set], (it >> 1) & 1, wt);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t td = tbase + set * 256 + ((uint32_t)(ew * 32) << 16);
      for (int c = 0; c < NCOL; c += 32) {
        float v[32];
        tmem_ld32(td + c, v);
        const int f = part * NCOL + c;
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = E::pack(v[2 * j], v[2 * j + 1]);
        if (tma_rows) {
          if (lane == 0) bulk_wait_read0();   // the buffer's previous store has read it
          __syncwarp();
#pragma unroll
          for (int u = 0; u < 4; ++u)
            stg[lane * 4 + (u ^ ((lane >> 1) & 3))] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&maps.dQw, f, t * p.G + ew * 32, smem_u32(stg));
            bulk_commit();
          }
          continue;
        }
        T* dst = h < p.G ? out + ((size_t)t * p.G + h) * 512 + f : nullptr;
        if (dst) {
          uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
          for (int u = 0; u < 4; ++u) d4[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty_bar[set]);
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
cudaError_t launch_one(const Maps& maps, const Prob& p, const float* part_stats, void* out, int* gerr, int nsm,
                       cudaStream_t st) {
  using S = DqSmem<NCOL, GP>;
  auto kern = p.bs >= 8 ? dq_kernel<T, GP, true> : dq_kernel<T, GP, false>;
  const int smem = S::kBytes > kOneCtaSmem ? S::kBytes : kOneCtaSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nitems = p.ntok * NPART;
  const int grid = nitems < nsm ? nitems : nsm;
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, S::kThreads, smem, st>>>(maps, p, part_stats, static_cast<T*>(out), gerr);
  return cudaGetLastError();
}

}  // namespace

template <typename T>
cudaError_t launch_pv(const Maps& maps, const Prob& p, const float* part_stats, void* out, int* gerr, int nsm,
                      cudaStream_t st) {
  if (p.Gp == 64) return launch_one<T, 64>(maps, p, part_stats, out, gerr, nsm, st);
  return launch_one<T, 128>(maps, p, part_stats, out, gerr, nsm, st);
}

template cudaError_t launch_pv<__nv_bfloat16>(const Maps&, const Prob&, const float*, void*, int*, int, cudaStream_t);
template cudaError_t launch_pv<__half>(const Maps&, const Prob&, const float*, void*, int*, int, cudaStream_t);

}  // namespace sfa
