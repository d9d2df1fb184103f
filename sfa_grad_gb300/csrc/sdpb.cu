// Key-major scores for block-sparse indices (sparseBlockSize >= 16, at most
// 64 heads), with several tokens packed into the MMA's M dimension.
//
// For every block start g that the chunk's tokens select (the groups formed
// for kvb.cu: the (token, index) pairs binned by start row), the block's bs
// key rows [k || kRope] and value rows stay in shared memory while the
// selecting tokens stream past in packs of TPK = 128 / GK tokens (GK = G
// rounded up to 16), so that a pack's token-heads fill M = 128 rows:
//     S  = [q || qRope]_pack . [k || kRope]_g^T     (M = token-heads, N = bs keys, K = 576)
//     dP = dO_pack . v_g^T                           (K = 512)
// in tensor memory; the epilogue (one thread per token-head row) forms
//     P  = exp(S * scale - softmaxMax) / softmaxSum  (masked keys -> 0)
//     dS = P * (dP - Dsum) * scale
// and writes each pair's bs staged P^T / dS^T rows (slots index*bs .. +bs-1,
// rows of Gs heads) with one bulk copy per pair and tensor.  The per-token
// score kernel (sdp.cu) instead loads a block's key and value rows once per
// selecting token; here they are loaded once per group.
//
// aclnnSparseFlashAttentionGrad doc, 功能说明 (selected blocks of
// sparseBlockSize keys) and 阶段1/阶段2 (dP, dS); MindSpore
// flash_attention_bwd.py, compute_Pij and compute_dSij.
#include "common.cuh"
#include "kernels.h"

namespace sfa {

namespace {

constexpr int kThreads = 256;   // warp 0: MMA issuer, warps 1-3: TMA producers, warps 4-7: epilogue
constexpr int kStages = 3;      // pack operand ring (one stage per producer warp)
constexpr int kRows = 128;      // MMA M: token-head rows of a pack
constexpr int kStageBytes = kRows * 128;   // one 64-feature panel of the pack

// dynamic shared memory: KV panels (17 x bs rows), ring, epilogue P and dS tiles
__host__ __device__ constexpr int kv_bytes(int bs) { return 17 * bs * 128; }
__host__ __device__ constexpr int epi_bytes(int bs) { return kRows * bs * 2; }
__host__ __device__ constexpr int smem_bytes(int bs) {
  return kv_bytes(bs) + kStages * kStageBytes + 2 * epi_bytes(bs) + 1024;
}

__device__ __forceinline__ void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <typename T, int BS, int GK>
__global__ void __launch_bounds__(kThreads, 1) sdpb_kernel(const __grid_constant__ Maps maps, Prob p, const int* groups,
                                                           const int* gbeg, const int* ngroups_p, const int* entries,
                                                           T* pst, T* dsst, int* gerr) {
  using E = Elt<T>;
  constexpr int TPK = kRows / GK;          // tokens per pack
  constexpr int kPanel = BS * 128;         // one 64-feature panel of the block's rows
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* kv = smem;
  uint8_t* ring = smem + kv_bytes(BS);
  T* epi_p = reinterpret_cast<T*>(ring + kStages * kStageBytes);
  T* epi_ds = epi_p + kRows * BS;
  __shared__ uint64_t kv_full, kv_empty, a_full[kStages], a_empty[kStages], t_full[2], t_empty[2], done_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = *ngroups_p;
  const int nS = p.has_rope ? 9 : 8;       // stages of the score contraction
  const int nc = nS + 8;                    // + 8 of dP
  const int Gs = p.Gs;

  // pack rows past TPK * GK (GK = 48) never receive a box: zero them once
  if (TPK * GK < kRows) {
    for (int s = 0; s < kStages; ++s) {
      uint4* z = reinterpret_cast<uint4*>(ring + s * kStageBytes + TPK * GK * 128);
      for (int i = threadIdx.x; i < (kRows - TPK * GK) * 128 / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
    }
  }
  // without rope the kRope panel stays zero
  if (!p.has_rope) {
    uint4* z = reinterpret_cast<uint4*>(kv + 8 * kPanel);
    for (int i = threadIdx.x; i < kPanel / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
  }
  fence_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(&kv_full, 1);
    mbar_init(&kv_empty, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&t_full[i], 1);
      mbar_init(&t_empty[i], kRows);
    }
    mbar_init(&done_bar, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  const Waiter wt{&abort_flag, gerr, p.wait_ns};

  if (warp == 0) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kRows, BS, E::is_f16, false, false);
      const uint64_t da0 = sdesc_kmajor(smem_u32(ring), 0);
      const uint64_t db0 = sdesc_kmajor(smem_u32(kv), 0);
      int g = 0, it = 0, kvn = 0;
      bool ok = true;
      for (int k = blockIdx.x; k < ngroups && ok; k += gridDim.x, ++kvn) {
        const int npk = (gbeg[k + 1] - gbeg[k] + TPK - 1) / TPK;
        ok = mbar_wait_poll(&kv_full, kvn & 1, wt);
        if (!ok) break;
        tc_fence_after();
        for (int j = 0; j < npk && ok; ++j, ++it) {
          const int set = it & 1;
          ok = mbar_wait_poll(&t_empty[set], ((it >> 1) & 1) ^ 1, wt);
          if (!ok) break;
          tc_fence_after();
          const uint32_t dS = tbase + set * (2 * BS), dP = dS + BS;
          for (int c = 0; c < nc && ok; ++c, ++g) {
            const int slot = g % kStages;
            ok = mbar_wait_poll(&a_full[slot], (g / kStages) & 1, wt);
            if (!ok) break;
            tc_fence_after();
            // stage c: pack panel c against key panel c (c < nS, kRope = 8), or
            // against value panel c - nS
            const int kvp = c < nS ? c : 9 + (c - nS);
            mma_ss_k64<2, 2>(c < nS ? dS : dP, da0 + desc_off(slot * kStageBytes), db0 + desc_off(kvp * kPanel), idesc,
                             (c == 0 || c == nS) ? 0u : 1u);
            mma_commit(&a_empty[slot]);
          }
          if (ok) mma_commit(&t_full[set]);
        }
        if (ok) mma_commit(&kv_empty);
      }
      mma_settle(&done_bar, gerr);   // no MMA still writing tensor memory at exit
    }
    __syncwarp();
  } else if (warp <= kStages) {
    // ---------------------------------------------------------------- TMA producers
    // Producer w (warps 1-3) fills ring slot w-1 for every third stage: the
    // pack's tokens' head rows of one 64-feature panel, one box of GK rows per
    // token (a missing token of the last pack reads rows below row 0: zeros).
    // Producer 0 also loads each group's key / value panels.
    if (lane == 0) {
      const int me = warp - 1;
      int g = 0, kvn = 0;
      bool ok = true;
      ArmLog alog, klog;
      for (int k = blockIdx.x; k < ngroups && ok; k += gridDim.x, ++kvn) {
        const int e0 = gbeg[k], e1 = gbeg[k + 1];
        const int npk = (e1 - e0 + TPK - 1) / TPK;
        if (me == 0) {
          if (kvn > 0) ok = mbar_wait(&kv_empty, (kvn - 1) & 1, wt);
          if (!ok) break;
          const int y0 = __ldg(groups + k) - BS;   // first key row (may be below 0: zeros)
          mbar_expect_tx(&kv_full, (uint32_t)(nS + 8) * kPanel);
          klog.arm(0, (uint32_t)kvn);
          for (int pn = 0; pn < 8; ++pn) tma_2d(smem_u32(kv + pn * kPanel), &maps.k, pn * 64, y0, &kv_full);
          if (p.has_rope) tma_2d(smem_u32(kv + 8 * kPanel), &maps.kr, 0, y0, &kv_full);
          for (int pn = 0; pn < 8; ++pn) tma_2d(smem_u32(kv + (9 + pn) * kPanel), &maps.v, pn * 64, y0, &kv_full);
        }
        for (int j = 0; j < npk && ok; ++j) {
          // the pack's first head rows, once per pack (a missing token of the
          // last pack: rows below row 0)
          int ys[TPK];
#pragma unroll
          for (int jt = 0; jt < TPK; ++jt) {
            const int e = e0 + j * TPK + jt;
            ys[jt] = e < e1 ? (p.tok0 + __ldg(entries + e) / p.Kidx) * p.G : -2 * GK;
          }
          for (int c = 0; c < nc && ok; ++c, ++g) {
            const int slot = g % kStages;
            if (slot != me) continue;
            ok = mbar_wait(&a_empty[slot], ((g / kStages) & 1) ^ 1, wt);
            if (!ok) break;
            mbar_expect_tx(&a_full[slot], (uint32_t)kStageBytes - (kRows - TPK * GK) * 128);
            alog.arm(slot, (uint32_t)(g / kStages));
            const CUtensorMap* mq = c < 8 ? &maps.qg : c < nS ? &maps.qrg : &maps.dOg;
            const int x = c < 8 ? c * 64 : c < nS ? 0 : (c - nS) * 64;
            const uint32_t dst = smem_u32(ring + slot * kStageBytes);
#pragma unroll
            for (int jt = 0; jt < TPK; ++jt) tma_2d(dst + jt * GK * 128, mq, x, ys[jt], &a_full[slot]);
          }
        }
      }
      // no copy still landing in shared memory at exit
      alog.settle(a_full, gerr);
      klog.settle(&kv_full, gerr);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue
    // Thread r = TMEM lane r = token-head row: token jt = r / GK of the pack,
    // head h = r % GK.  P and dS go to shared memory as [token][key][Gs
    // heads] (each pair's bs rows contiguous, as in the staging), then thread
    // jt < TPK copies token jt's two tiles with bulk copies.  Named barriers
    // run once per pack whatever happens, so their trip counts never depend
    // on the abort flag.
    const int r = threadIdx.x - 128;
    const int jt = r / GK, h = r - jt * GK;
    const float sl2 = p.scale * kLog2e;
    int it = 0;
    bool pending = false;   // this thread has bulk copies reading the tiles
    for (int k = blockIdx.x; k < ngroups; k += gridDim.x) {
      const int e0 = gbeg[k], e1 = gbeg[k + 1];
      const int npk = (e1 - e0 + TPK - 1) / TPK;
      for (int j = 0; j < npk; ++j, ++it) {
        const int set = it & 1;
        const int e = e0 + j * TPK + jt;
        const bool has = jt < TPK && e < e1;
        int tl = 0, ii = 0, ridx = 0, lim = -1;
        float m = 0.f, linv = 0.f, dsc = 0.f;
        if (has) {
          const int pr = __ldg(entries + e);
          tl = pr / p.Kidx;
          ii = pr - tl * p.Kidx;
          const int t = p.tok0 + tl;
          ridx = __ldg(p.idx + (size_t)t * p.Kidx + ii);
          lim = p.meta[t].limit;
          if (h < p.G) {
            const float l = __ldg(p.ssum + (size_t)t * p.G + h);
            m = l > 0.f ? __ldg(p.smax + (size_t)t * p.G + h) * kLog2e : 0.f;
            linv = l > 0.f ? 1.f / l : 0.f;
            dsc = __ldg(p.dsum + (size_t)t * p.G + h) * p.scale;
          }
        }
        const bool ok = __all_sync(0xffffffffu, !abort_flag && mbar_wait(&t_full[set], (it >> 1) & 1, wt));
        // the previous pack's copies must have read the tiles before they are rewritten
        if (pending) {
          bulk_wait_read();
          pending = false;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (ok) {
          tc_fence_after();
          const uint32_t td = tbase + set * (2 * BS) + ((uint32_t)((warp - 4) * 32) << 16);
          constexpr int CH = BS < 32 ? BS : 32;   // key columns per TMEM load
#pragma unroll 1
          for (int u0 = 0; u0 < BS; u0 += CH) {
            float s[CH], dp[CH];
            if constexpr (CH == 32) {
              tmem_ld32(td + u0, s);
              tmem_ld32(td + BS + u0, dp);
            } else {
              tmem_ld16(td + u0, s);
              tmem_ld16(td + BS + u0, dp);
            }
            if (jt < TPK && h < Gs) {
              T* op = epi_p + ((size_t)jt * BS + u0) * Gs + h;
              T* od = epi_ds + ((size_t)jt * BS + u0) * Gs + h;
#pragma unroll
              for (int u = 0; u < CH; ++u) {
                const int key = ridx + u0 + u;
                const bool valid = has && key >= 0 && key <= lim;
                const float pp = valid ? ex2(fmaf(s[u], sl2, -m)) * linv : 0.f;
                const float dd = pp != 0.f ? pp * fmaf(dp[u], p.scale, -dsc) : 0.f;
                op[u * Gs] = E::from_f(pp);
                od[u * Gs] = E::from_f(dd);
              }
            }
          }
          tc_fence_before();
        }
        mbar_arrive(&t_empty[set]);
        fence_async_smem();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        // thread r < TPK copies token r's tiles of the pack
        if (ok && r < TPK) {
          const int e2 = e0 + j * TPK + r;
          if (e2 < e1) {
            const int pr = __ldg(entries + e2);
            const int tl2 = pr / p.Kidx, ii2 = pr - tl2 * p.Kidx;
            const size_t row0 = ((size_t)tl2 * p.Kpad + (size_t)ii2 * BS) * Gs;
            const uint32_t bytes = (uint32_t)(BS * Gs * sizeof(T));
            bulk_store(pst + row0, smem_u32(epi_p + (size_t)r * BS * Gs), bytes);
            bulk_store(dsst + row0, smem_u32(epi_ds + (size_t)r * BS * Gs), bytes);
            bulk_commit();
            pending = true;
          }
        }
      }
    }
    if (pending) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 256);
  }
}

template <typename T, int BS, int GK>
cudaError_t launch_bg(const Maps& maps, const Prob& p, const int* groups, const int* gbeg, const int* ngroups,
                      const int* entries, void* pst, void* dsst, int* gerr, int nsm, cudaStream_t st) {
  auto kern = sdpb_kernel<T, BS, GK>;
  const int smem = smem_bytes(BS) > kOneCtaSmem ? smem_bytes(BS) : kOneCtaSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<nsm, kThreads, smem, st>>>(maps, p, groups, gbeg, ngroups, entries, static_cast<T*>(pst),
                                    static_cast<T*>(dsst), gerr);
  return cudaGetLastError();
}

template <typename T, int BS>
cudaError_t launch_b(const Maps& maps, const Prob& p, const int* groups, const int* gbeg, const int* ngroups,
                     const int* entries, void* pst, void* dsst, int* gerr, int nsm, cudaStream_t st) {
  const int gk = (p.G + 15) / 16 * 16;
  if (gk == 16) return launch_bg<T, BS, 16>(maps, p, groups, gbeg, ngroups, entries, pst, dsst, gerr, nsm, st);
  if (gk == 32) return launch_bg<T, BS, 32>(maps, p, groups, gbeg, ngroups, entries, pst, dsst, gerr, nsm, st);
  if (gk == 48) return launch_bg<T, BS, 48>(maps, p, groups, gbeg, ngroups, entries, pst, dsst, gerr, nsm, st);
  return launch_bg<T, BS, 64>(maps, p, groups, gbeg, ngroups, entries, pst, dsst, gerr, nsm, st);
}

}  // namespace

template <typename T>
cudaError_t launch_sdpb(const Maps& maps, const Prob& p, const int* groups, const int* gbeg, const int* ngroups,
                        const int* entries, void* pst, void* dsst, int* gerr, int nsm, cudaStream_t st) {
  if (p.ntok <= 0 || p.T2 <= 0) return cudaSuccess;
  if (p.bs == 16) return launch_b<T, 16>(maps, p, groups, gbeg, ngroups, entries, pst, dsst, gerr, nsm, st);
  if (p.bs == 32) return launch_b<T, 32>(maps, p, groups, gbeg, ngroups, entries, pst, dsst, gerr, nsm, st);
  return launch_b<T, 64>(maps, p, groups, gbeg, ngroups, entries, pst, dsst, gerr, nsm, st);
}

template cudaError_t launch_sdpb<__nv_bfloat16>(const Maps&, const Prob&, const int*, const int*, const int*,
                                                const int*, void*, void*, int*, int, cudaStream_t);
template cudaError_t launch_sdpb<__half>(const Maps&, const Prob&, const int*, const int*, const int*, const int*,
                                         void*, void*, int*, int, cudaStream_t);

}  // namespace sfa
