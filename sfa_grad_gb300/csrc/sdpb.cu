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
// rows of Gs heads).  The
// per-token score kernel (sdp.cu) instead loads a block's key and value rows
// once per selecting token; here they are loaded once per group.  The pack
// stream is bound by the bytes in flight, so the ring takes the shared
// memory the resident block leaves: five 16 KB stages, one producer warp
// each.
//
// The companion forward's score pass uses the same kernel without dP: MODE
// kModeFwdStats writes per pair and head the max of the raw scores over the
// block's valid keys and the sum of exp((s - max) * scale) (combined per
// token afterwards), and stages P~ = exp((s - max) * scale), which the P.V
// kernel (dqb.cu) rescales per pair to the final statistics.
//
// aclnnSparseFlashAttentionGrad doc, 功能说明 (selected blocks of
// sparseBlockSize keys) and 阶段1/阶段2 (dP, dS); MindSpore
// flash_attention_bwd.py, compute_Pij and compute_dSij.
#include "common.cuh"
#include "kernels.h"

namespace sfa {

namespace {

constexpr int kStages = 5;      // pack operand ring, one producer warp per stage slot
// warp 0: MMA issuer, warps 1-5: TMA producers, warps 6-9: epilogue
constexpr int kThreads = (1 + kStages + 4) * 32;
constexpr int kEpi0 = 1 + kStages;        // first epilogue warp
constexpr int kRows = 128;      // MMA M: token-head rows of a pack
constexpr int kStageBytes = kRows * 128;   // one 64-feature panel of the pack

// dynamic shared memory: KV panels (17 x bs rows), then the ring
__host__ __device__ constexpr int kv_bytes(int bs) { return 17 * bs * 128; }
__host__ __device__ constexpr int smem_bytes(int bs) { return kv_bytes(bs) + kStages * kStageBytes + 1024; }

template <typename T, int BS, int GK, int MODE>
__global__ void __launch_bounds__(kThreads, 1) sdpb_kernel(const __grid_constant__ Maps maps, Prob p, const int* groups,
                                                           const int* gbeg, const int* ngroups_p, const int* entries,
                                                           T* pst, T* dsst, float* tile_stats, int* gerr) {
  constexpr bool bwd = MODE == kModeBwd;
  using E = Elt<T>;
  constexpr int TPK = kRows / GK;          // tokens per pack
  constexpr int kPanel = BS * 128;         // one 64-feature panel of the block's rows
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* kv = smem;
  uint8_t* ring = smem + kv_bytes(BS);
  __shared__ uint64_t kv_full, kv_empty, a_full[kStages], a_empty[kStages], t_full[2], t_empty[2], done_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = *ngroups_p;
  const int nS = p.has_rope ? 9 : 8;       // stages of the score contraction
  const int nc = bwd ? nS + 8 : nS;        // + 8 of dP
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
    // Producer w (warps 1-5) fills ring slot w-1 for every fifth stage: the
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
          mbar_expect_tx(&kv_full, (uint32_t)(bwd ? nS + 8 : nS) * kPanel);
          klog.arm(0, (uint32_t)kvn);
          for (int pn = 0; pn < 8; ++pn) tma_2d(smem_u32(kv + pn * kPanel), &maps.k, pn * 64, y0, &kv_full);
          if (p.has_rope) tma_2d(smem_u32(kv + 8 * kPanel), &maps.kr, 0, y0, &kv_full);
          if (bwd)
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
  } else if (warp >= kEpi0) {
    // ---------------------------------------------------------------- epilogue
    // Warp w reads TMEM lane quadrant w % 4; thread r = TMEM lane = token-head
    // row: token jt = r / GK of the pack, head h = r % GK.  For each key u the
    // 16-bit P and dS values go straight to the pair's staged row (tl * Kpad
    // + index * bs + u, column h): a token's heads are contiguous, so a warp
    // store covers 32 contiguous bytes per token.  The pair data a pack needs
    // (entry -> index and token metadata -> statistics) is a chain of
    // dependent loads, so it is fetched two packs ahead: the entry of pack
    // n + 2 and the rest of pack n + 1 while pack n is processed.
    const int r = (warp & 3) * 32 + lane;
    const int jt = r / GK, h = r - jt * GK;
    const float sl2 = p.scale * kLog2e;
    // walk of this CTA's packs in order: group k (strided), pack j
    struct Pos {
      int k, j, e0, e1;
    };
    auto first = [&]() {
      Pos q{(int)blockIdx.x, 0, 0, 0};
      if (q.k < ngroups) {
        q.e0 = gbeg[q.k];
        q.e1 = gbeg[q.k + 1];
      }
      return q;
    };
    auto next = [&](Pos q) {
      if (q.k >= ngroups) return q;
      if ((++q.j) * TPK >= q.e1 - q.e0) {
        q.k += gridDim.x;
        q.j = 0;
        if (q.k < ngroups) {
          q.e0 = gbeg[q.k];
          q.e1 = gbeg[q.k + 1];
        }
      }
      return q;
    };
    // this thread's pair of a pack position, -1 if none
    auto pair_of = [&](const Pos& q) {
      const int e = q.e0 + q.j * TPK + jt;
      return (q.k < ngroups && jt < TPK && e < q.e1) ? __ldg(entries + e) : -1;
    };
    struct Meta {
      int ridx, lim;
      size_t row0, sidx;
      float m, linv, dsc;
    };
    auto meta_of = [&](int pr) {
      Meta d{0, -1, 0, 0, 0.f, 0.f, 0.f};
      if (pr < 0) return d;
      const int tl = pr / p.Kidx, ii = pr - tl * p.Kidx;
      const int t = p.tok0 + tl;
      d.ridx = __ldg(p.idx + (size_t)t * p.Kidx + ii);
      d.lim = p.meta[t].limit;
      d.row0 = (size_t)tl * p.Kpad + (size_t)ii * BS;
      d.sidx = (size_t)pr * p.G + h;
      if (MODE != kModeFwdStats && h < p.G) {
        const float l = __ldg(p.ssum + (size_t)t * p.G + h);
        d.m = l > 0.f ? __ldg(p.smax + (size_t)t * p.G + h) * kLog2e : 0.f;
        d.linv = l > 0.f ? 1.f / l : 0.f;
        if (bwd) d.dsc = __ldg(p.dsum + (size_t)t * p.G + h) * p.scale;
      }
      return d;
    };
    Pos cur = first();
    Pos nx1 = next(cur);
    int pr_cur = pair_of(cur), pr1 = pair_of(nx1);
    Meta mc = meta_of(pr_cur);
    int it = 0;
    for (; cur.k < ngroups && !abort_flag; ++it) {
      const int set = it & 1;
      const Pos nx2 = next(nx1);
      const int pr2 = pair_of(nx2);      // entry two packs ahead
      const Meta mn = meta_of(pr1);      // data one pack ahead
      const bool has = pr_cur >= 0;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&t_full[set], (it >> 1) & 1, wt));
      if (!ok) break;
      tc_fence_after();
      const uint32_t td = tbase + set * (2 * BS) + ((uint32_t)((warp & 3) * 32) << 16);
      constexpr int CH = BS < 32 ? BS : 32;   // key columns per TMEM load
      if constexpr (MODE == kModeFwdStats) {
        // the pair's partial statistics per (token, head) row: max of the raw
        // scores over the block's valid keys and the sum of exp((s - max) *
        // scale); P~ = exp((s - max) * scale) staged (0 for a masked key or a
        // padded head)
        float sv[BS];
#pragma unroll
        for (int u0 = 0; u0 < BS; u0 += CH) {
          if constexpr (CH == 32) tmem_ld32(td + u0, sv + u0);
          else tmem_ld16(td + u0, sv + u0);
        }
        float mx = -INFINITY;
        if (has && h < p.G) {
#pragma unroll
          for (int u = 0; u < BS; ++u) {
            const int key = mc.ridx + u;
            if (key >= 0 && key <= mc.lim) mx = fmaxf(mx, sv[u]);
          }
        }
        if (has && h < Gs) {
          T* op = pst + mc.row0 * Gs + h;
          float l = 0.f;
#pragma unroll
          for (int u = 0; u < BS; ++u) {
            const int key = mc.ridx + u;
            const float e = (mx != -INFINITY && key >= 0 && key <= mc.lim) ? ex2((sv[u] - mx) * sl2) : 0.f;
            l += e;
            op[(size_t)u * Gs] = E::from_f(e);
          }
          if (h < p.G) reinterpret_cast<float2*>(tile_stats)[mc.sidx] = make_float2(mx, l);
        }
      } else {
        const bool store = has && h < Gs;
        T* op = pst + mc.row0 * Gs + h;
        T* od = bwd ? dsst + mc.row0 * Gs + h : nullptr;
#pragma unroll 1
        for (int u0 = 0; u0 < BS; u0 += CH) {
          float s[CH], dp[CH];
          if constexpr (CH == 32) {
            tmem_ld32(td + u0, s);
            if (bwd) tmem_ld32(td + BS + u0, dp);
          } else {
            tmem_ld16(td + u0, s);
            if (bwd) tmem_ld16(td + BS + u0, dp);
          }
          if (store) {
#pragma unroll
            for (int u = 0; u < CH; ++u) {
              const int key = mc.ridx + u0 + u;
              const bool valid = key >= 0 && key <= mc.lim;
              const float pp = valid ? ex2(fmaf(s[u], sl2, -mc.m)) * mc.linv : 0.f;
              op[(size_t)(u0 + u) * Gs] = E::from_f(pp);
              if (bwd) {
                const float dd = pp != 0.f ? pp * fmaf(dp[u], p.scale, -mc.dsc) : 0.f;
                od[(size_t)(u0 + u) * Gs] = E::from_f(dd);
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&t_empty[set]);
      cur = nx1;
      nx1 = nx2;
      pr_cur = pr1;
      pr1 = pr2;
      mc = mn;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 256);
  }
}

template <typename T, int BS, int GK>
cudaError_t launch_bg(const Maps& maps, const Prob& p, int mode, const int* groups, const int* gbeg, const int* ngroups,
                      const int* entries, void* pst, void* dsst, float* tile_stats, int* gerr, int nsm,
                      cudaStream_t st) {
  if (mode != kModeFwdStats && mode != kModeBwd) return cudaErrorInvalidValue;
  auto kern = mode == kModeFwdStats ? sdpb_kernel<T, BS, GK, kModeFwdStats> : sdpb_kernel<T, BS, GK, kModeBwd>;
  const int smem = smem_bytes(BS) > kOneCtaSmem ? smem_bytes(BS) : kOneCtaSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<nsm, kThreads, smem, st>>>(maps, p, groups, gbeg, ngroups, entries, static_cast<T*>(pst),
                                    static_cast<T*>(dsst), tile_stats, gerr);
  return cudaGetLastError();
}

template <typename T, int BS>
cudaError_t launch_b(const Maps& maps, const Prob& p, int mode, const int* groups, const int* gbeg, const int* ngroups,
                     const int* entries, void* pst, void* dsst, float* tile_stats, int* gerr, int nsm,
                     cudaStream_t st) {
  const int gk = (p.G + 15) / 16 * 16;
  if (gk == 16)
    return launch_bg<T, BS, 16>(maps, p, mode, groups, gbeg, ngroups, entries, pst, dsst, tile_stats, gerr, nsm, st);
  if (gk == 32)
    return launch_bg<T, BS, 32>(maps, p, mode, groups, gbeg, ngroups, entries, pst, dsst, tile_stats, gerr, nsm, st);
  if (gk == 48)
    return launch_bg<T, BS, 48>(maps, p, mode, groups, gbeg, ngroups, entries, pst, dsst, tile_stats, gerr, nsm, st);
  return launch_bg<T, BS, 64>(maps, p, mode, groups, gbeg, ngroups, entries, pst, dsst, tile_stats, gerr, nsm, st);
}

}  // namespace

template <typename T>
cudaError_t launch_sdpb(const Maps& maps, const Prob& p, int mode, const int* groups, const int* gbeg,
                        const int* ngroups, const int* entries, void* pst, void* dsst, float* tile_stats, int* gerr,
                        int nsm, cudaStream_t st) {
  if (p.ntok <= 0 || p.T2 <= 0) return cudaSuccess;
  if (p.bs == 16)
    return launch_b<T, 16>(maps, p, mode, groups, gbeg, ngroups, entries, pst, dsst, tile_stats, gerr, nsm, st);
  if (p.bs == 32)
    return launch_b<T, 32>(maps, p, mode, groups, gbeg, ngroups, entries, pst, dsst, tile_stats, gerr, nsm, st);
  return launch_b<T, 64>(maps, p, mode, groups, gbeg, ngroups, entries, pst, dsst, tile_stats, gerr, nsm, st);
}

template cudaError_t launch_sdpb<__nv_bfloat16>(const Maps&, const Prob&, int, const int*, const int*, const int*,
                                                const int*, void*, void*, float*, int*, int, cudaStream_t);
template cudaError_t launch_sdpb<__half>(const Maps&, const Prob&, int, const int*, const int*, const int*,
                                         const int*, void*, void*, float*, int*, int, cudaStream_t);

}  // namespace sfa
