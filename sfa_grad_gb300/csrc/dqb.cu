// dQ for block-sparse indices with at most 64 heads, features on the MMA's M:
//     [dQ || dQRope](t)^T = [K || KRope]_sel(t)^T . dS(t)^T
// (M = 128 features per tile, N = GN = G rounded up to 16 heads, K = keys),
// accumulated in tensor memory over all of the token's selected keys.
//
// With heads on M (the query side of kvq.cu) a token of G = 16 heads fills
// 16 of the MMA's 128 rows; here the 576 features fill M (four tiles of the
// 512-wide part, a fifth for the 64 rope features) and the heads are N, so
// no MMA row is padding.  The kernel is then bound by the L2-to-SM loads of
// the selected key rows (1152 B per key), so a stage carries all 576
// features of 64 keys and the token's staged dS rows once, and the ring is
// as deep as shared memory allows (two stages of 80 KB).
//
// PV: the companion forward's O(t)^T = V_sel(t)^T . P(t)^T with the same
// pipeline (value rows, the staged P rows, four feature tiles); P is staged
// relative to each (token, block) pair's max and rescaled here.
//
// aclnnSparseFlashAttentionGrad doc, 功能说明 (selected blocks of
// sparseBlockSize keys) and 阶段3 (dQ = dS . K * scale, with the scale folded
// into dS); MindSpore flash_attention_bwd.py, update_dQi.
#include "common.cuh"
#include "kernels.h"

namespace sfa {

namespace {

constexpr int kKeys = 64;                  // keys per stage (MMA K extent)
constexpr int kStages = 2;
constexpr int kPanel = kKeys * 128;        // 64 keys x 64 features (or heads), 8 KB
// stage layout, one panel each: [kRope | k 0-63 | ... | k 448-511 | dS].
// Feature tile m < 4 is panels 2m+1, 2m+2; the rope tile is panels 0, 1, so
// its rows 64-127 read k 0-63 (finite data whose results are never stored).
constexpr int kStageBytes = 10 * kPanel;
constexpr int kDsOff = 9 * kPanel;
// warp 0: MMA issuer, warps 1-2: TMA producers (one per stage slot),
// warps 3-6: epilogue (one per TMEM lane quadrant)
constexpr int kThreads = (1 + kStages + 4) * 32;
constexpr int kEpi0 = 1 + kStages;
constexpr int kSmemBytes = kStages * kStageBytes + 1024;

__device__ __forceinline__ uint32_t tile_off(int m) { return m < 4 ? (uint32_t)(2 * m + 1) * kPanel : 0u; }

template <typename T, int GN, bool PV>
__global__ void __launch_bounds__(kThreads, 1) dqb_kernel(const __grid_constant__ Maps maps, Prob p, T* dq, T* dqr,
                                                          const float* part_stats, int* gerr) {
  using E = Elt<T>;
  // five feature tiles per accumulator, each at a 32-column boundary
  constexpr int TS = (GN + 31) / 32 * 32;
  constexpr int kBufCols = 5 * TS;
  constexpr int NBUF = 2 * kBufCols <= 512 ? 2 : 1;        // accumulator buffers
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // PV: p_full (the stage's P box has landed, to be rescaled) and each
  // producer's factor table (blocks of the stage x heads)
  __shared__ uint64_t a_full[kStages], p_full[kStages], a_empty[kStages], t_full[NBUF], t_empty[NBUF], done_bar;
  __shared__ __align__(16) float fac_s[kStages][(kKeys / 16) * 64];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nst = p.Kpad / kKeys;          // stages per token
  const bool rope = !PV && p.has_rope;
  const int nt = rope ? 5 : 4;             // feature tiles

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&a_full[i], PV ? 1 + 32 : 1);   // PV: the arming lane + the rescaling lanes
      mbar_init(&p_full[i], 1);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < NBUF; ++i) {
      mbar_init(&t_full[i], 1);
      mbar_init(&t_empty[i], 128);
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
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, GN, E::is_f16, true, true);
      const uint64_t d0 = sdesc_mnmajor(smem_u32(smem), 0, kKeys);
      int g = 0, it = 0;
      bool ok = true;
      for (int tl = blockIdx.x; tl < p.ntok && ok; tl += gridDim.x, ++it) {
        const int buf = it % NBUF;
        ok = mbar_wait_poll(&t_empty[buf], ((it / NBUF) & 1) ^ 1, wt);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tbase + buf * kBufCols;
        for (int c = 0; c < nst; ++c, ++g) {
          const int slot = g % kStages;
          ok = mbar_wait_poll(&a_full[slot], (g / kStages) & 1, wt);
          if (!ok) break;
          tc_fence_after();
          const uint32_t so = slot * kStageBytes;
          const uint64_t db = d0 + desc_off(so + kDsOff);
          for (int m = 0; m < nt; ++m)
            mma_ss_k64<128, 128>(d + m * TS, d0 + desc_off(so + tile_off(m)), db, idesc, c == 0 ? 0u : 1u);
          mma_commit(&a_empty[slot]);
        }
        if (ok) mma_commit(&t_full[buf]);
      }
      mma_settle(&done_bar, gerr);   // no MMA still writing tensor memory at exit
    }
    __syncwarp();
  } else if (warp < kEpi0) {
    // ---------------------------------------------------------------- TMA producers
    // Producer w (warps 1-2) fills slot w-1 for every second stage: the
    // token's staged dS rows of 64 slots (one box; heads past Gs read as
    // zeros) and, per selected block of the stage, one box of bs key rows per
    // 64-feature panel.  An index with no key at or above 0, past the last
    // row or past the index list reads rows below row 0: zeros.
    const int me = warp - 1;
    const int nidx = kKeys / p.bs;
    const uint32_t tx = kPanel * (rope ? 10u : 9u);
    const CUtensorMap* mrow = PV ? &maps.v : &maps.k;
    const CUtensorMap* mcol = PV ? &maps.P : &maps.dS;
    // the stage's key (or value) rows: nidx blocks x (8 + rope) panel boxes
    auto issue_rows = [&](uint32_t st, int t, long long kv0, int c, uint64_t* bar) {
      for (int i = 0; i < nidx; ++i) {
        const int ii = c * nidx + i;
        int y = -p.bs;
        if (ii < p.Kidx) {
          const int r = __ldg(p.idx + (size_t)t * p.Kidx + ii);
          const long long yy = kv0 + r;
          if ((long long)r + p.bs > 0 && yy < p.T2) y = (int)yy;
        }
        const uint32_t dst = st + (uint32_t)(i * p.bs) * 128;
        for (int pn = 0; pn < 8; ++pn) tma_2d(dst + (1 + pn) * kPanel, mrow, pn * 64, y, bar);
        if (rope) tma_2d(dst, &maps.kr, 0, y, bar);
      }
    };
    if constexpr (!PV) {
      if (lane == 0) {
        int g = 0;
        bool ok = true;
        ArmLog alog;
        for (int tl = blockIdx.x; tl < p.ntok && ok; tl += gridDim.x) {
          const int t = p.tok0 + tl;
          const long long kv0 = p.meta[t].kv_start;
          for (int c = 0; c < nst && ok; ++c, ++g) {
            const int slot = g % kStages;
            if (slot != me) continue;
            ok = mbar_wait(&a_empty[slot], ((g / kStages) & 1) ^ 1, wt);
            if (!ok) break;
            mbar_expect_tx(&a_full[slot], tx);
            alog.arm(slot, (uint32_t)(g / kStages));
            const uint32_t st = smem_u32(smem + slot * kStageBytes);
            tma_2d(st + kDsOff, mcol, 0, tl * p.Kpad + c * kKeys, &a_full[slot]);
            issue_rows(st, t, kv0, c, &a_full[slot]);
          }
        }
        alog.settle(a_full, gerr);   // no copy still landing in shared memory at exit
      }
      __syncwarp();
    } else {
      // PV: the staged rows hold P~ relative to each (token, block) pair's max
      // (sdpb.cu's statistics pass).  The P box lands on its own barrier; the
      // warp builds the stage's factor table exp((m_pair - m) * scale) / l
      // (blocks x heads) meanwhile, rescales the box in place once it has
      // landed, fences its stores and arrives (one arrival per lane).
      constexpr int CPR = GN / 8;        // 16-byte pieces of a staged row that hold heads
      constexpr int NPL = kKeys * CPR / 32;
      constexpr int kFacPerLane = (kKeys / 16) * GN / 32;   // table entries per lane at bs = 16
      float* ft = fac_s[me];
      const float sl2 = p.scale * kLog2e;
      int g = 0;
      bool ok = true;
      ArmLog alog, plog;
      for (int tl = blockIdx.x; tl < p.ntok && ok; tl += gridDim.x) {
        const int t = p.tok0 + tl;
        const long long kv0 = p.meta[t].kv_start;
        for (int c = 0; c < nst && ok; ++c, ++g) {
          const int slot = g % kStages;
          if (slot != me) continue;
          const uint32_t ph = (uint32_t)(g / kStages);
          // the statistics behind the stage's factors (entry e = lane + 32 j:
          // block e / GN, head e % GN), loaded before the slot wait so that
          // their latency hides behind it
          float em[kFacPerLane], el[kFacPerLane], ex[kFacPerLane];
#pragma unroll
          for (int j = 0; j < kFacPerLane; ++j) {
            const int e = lane + 32 * j;
            const int i = e / GN, h = e - i * GN;
            const int ii = c * nidx + i;
            em[j] = -INFINITY;
            el[j] = 0.f;
            ex[j] = 0.f;
            if (e < nidx * GN && h < p.G && ii < p.Kidx) {
              const size_t o = (size_t)t * p.G + h;
              em[j] = __ldg(part_stats + (((size_t)tl * p.Kidx + ii) * p.G + h) * 2);
              el[j] = __ldg(p.ssum + o);
              ex[j] = __ldg(p.smax + o);
            }
          }
          bool w = true;
          if (lane == 0) w = mbar_wait(&a_empty[slot], (ph & 1u) ^ 1u, wt);
          ok = __shfl_sync(0xffffffffu, w, 0);
          if (!ok) break;
          const uint32_t st = smem_u32(smem + slot * kStageBytes);
          if (lane == 0) {
            mbar_expect_tx(&p_full[slot], kPanel);
            plog.arm(slot, ph);
            tma_2d(st + kDsOff, mcol, 0, tl * p.Kpad + c * kKeys, &p_full[slot]);
            mbar_expect_tx(&a_full[slot], tx - kPanel);
            alog.arm(slot, ph);
            issue_rows(st, t, kv0, c, &a_full[slot]);
            // the P box of this warp's next stage (kStages on), from HBM into
            // L2 now: the rescale waits on its copy, which then comes from L2
            int nc = c + kStages, ntl = tl;
            if (nc >= nst) {
              nc -= nst;
              ntl += gridDim.x;
            }
            if (nc < nst && ntl < p.ntok) tma_prefetch_2d(mcol, 0, ntl * p.Kpad + nc * kKeys);
          }
#pragma unroll
          for (int j = 0; j < kFacPerLane; ++j) {
            const int e = lane + 32 * j;
            if (e < nidx * GN)
              ft[e] = (em[j] != -INFINITY && el[j] > 0.f) ? ex2(fmaf(em[j], sl2, -ex[j] * kLog2e)) / el[j] : 0.f;
          }
          __syncwarp();
          const bool pok = __all_sync(0xffffffffu, mbar_wait(&p_full[slot], ph & 1u, wt));
          if (pok) {
            uint4 v[NPL];
#pragma unroll
            for (int j = 0; j < NPL; ++j) {
              const int e = lane + 32 * j, r = e / CPR, k = e - r * CPR;
              v[j] = lds128(st + kDsOff + r * 128 + ((k ^ (r & 7)) << 4));
            }
#pragma unroll
            for (int j = 0; j < NPL; ++j) {
              const int e = lane + 32 * j, r = e / CPR, k = e - r * CPR;
              const float* f = ft + (r / p.bs) * GN + 8 * k;
              const float4 f0 = *reinterpret_cast<const float4*>(f);
              const float4 f1 = *reinterpret_cast<const float4*>(f + 4);
              sts128(st + kDsOff + r * 128 + ((k ^ (r & 7)) << 4),
                     make_uint4(E::mul2(v[j].x, E::pack(f0.x, f0.y)), E::mul2(v[j].y, E::pack(f0.z, f0.w)),
                                E::mul2(v[j].z, E::pack(f1.x, f1.y)), E::mul2(v[j].w, E::pack(f1.z, f1.w))));
            }
          }
          fence_async_smem();
          mbar_arrive(&a_full[slot]);
          __syncwarp();
          if (!pok) {
            ok = false;
            break;
          }
        }
      }
      // no copy still landing in shared memory at exit
      plog.settle(p_full, gerr);
      alog.settle(a_full, gerr);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    // Warp w reads TMEM lane quadrant w % 4: thread = feature row f of a
    // tile, GN head columns; a warp store covers 32 consecutive features of
    // one head row (64 contiguous bytes).
    const int qd = warp & 3;
    int it = 0;
    for (int tl = blockIdx.x; tl < p.ntok && !abort_flag; tl += gridDim.x, ++it) {
      const int buf = it % NBUF;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&t_full[buf], (it / NBUF) & 1, wt));
      if (!ok) break;
      tc_fence_after();
      const size_t t = (size_t)(p.tok0 + tl);
      const uint32_t td = tbase + buf * kBufCols + ((uint32_t)(qd * 32) << 16);
      for (int m = 0; m < nt; ++m) {
        const int f = m * 128 + qd * 32 + lane;
        float v[GN];
#pragma unroll
        for (int c0 = 0; c0 + 32 <= GN; c0 += 32) tmem_ld32(td + m * TS + c0, v + c0);
        if constexpr (GN % 32 != 0) tmem_ld16(td + m * TS + (GN - 16), v + (GN - 16));
        T* dst = nullptr;
        size_t hs = 0;
        if (f < 512) {
          dst = dq + t * p.G * 512 + f;
          hs = 512;
        } else if (f < 576 && dqr) {
          dst = dqr + t * p.G * 64 + (f - 512);
          hs = 64;
        }
        if (dst) {
#pragma unroll
          for (int h = 0; h < GN; ++h)
            if (h < p.G) dst[h * hs] = E::from_f(v[h]);
        }
      }
      tc_fence_before();
      mbar_arrive(&t_empty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <typename T, int GN>
cudaError_t launch_g(const Maps& maps, const Prob& p, bool pv, void* dq, void* dqr, const float* part_stats, int* gerr,
                     int nsm, cudaStream_t st) {
  auto kern = pv ? dqb_kernel<T, GN, true> : dqb_kernel<T, GN, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = p.ntok < nsm ? p.ntok : nsm;
  kern<<<grid, kThreads, kSmemBytes, st>>>(maps, p, static_cast<T*>(dq), static_cast<T*>(dqr), part_stats, gerr);
  return cudaGetLastError();
}

}  // namespace

template <typename T>
cudaError_t launch_dqb(const Maps& maps, const Prob& p, bool pv, void* dq, void* dqr, const float* part_stats,
                       int* gerr, int nsm, cudaStream_t st) {
  if (p.ntok <= 0) return cudaSuccess;
  if (p.bs < 16 || p.bs > kKeys || kKeys % p.bs != 0 || p.Kpad % kKeys != 0 || p.G > 64) return cudaErrorInvalidValue;
  if (pv && !part_stats) return cudaErrorInvalidValue;
  switch (p.Gs) {
    case 16: return launch_g<T, 16>(maps, p, pv, dq, dqr, part_stats, gerr, nsm, st);
    case 32: return launch_g<T, 32>(maps, p, pv, dq, dqr, part_stats, gerr, nsm, st);
    case 48: return launch_g<T, 48>(maps, p, pv, dq, dqr, part_stats, gerr, nsm, st);
    default: return launch_g<T, 64>(maps, p, pv, dq, dqr, part_stats, gerr, nsm, st);
  }
}

template cudaError_t launch_dqb<__nv_bfloat16>(const Maps&, const Prob&, bool, void*, void*, const float*, int*, int,
                                               cudaStream_t);
template cudaError_t launch_dqb<__half>(const Maps&, const Prob&, bool, void*, void*, const float*, int*, int,
                                        cudaStream_t);

}  // namespace sfa
