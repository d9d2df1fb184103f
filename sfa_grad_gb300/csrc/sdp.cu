// Score / softmax-gradient kernel: for one query token and a tile of 128 of its
// selected keys it recomputes
//     S^T = K_sel . [q || qRope]^T * scale        (tcgen05, keys on M, heads on N)
//     dP^T = V_sel . dO^T
// in tensor memory, then applies the saved softmax statistics:
//     P  = exp(S - softmaxMax) / softmaxSum                (masked keys -> 0)
//     dS = P * (dP - Dsum) * scale
// and writes P^T and dS^T (input dtype, heads contiguous) for the later
// contractions.  Forward modes reuse the score half: per-tile max/sum partials,
// or P from final statistics.
//
// aclnnSparseFlashAttentionGrad doc, 功能说明 (gather by topkIndices) and
// 阶段1/阶段2 (dP, dS); MindSpore flash_attention_bwd.py, compute_Pij
// (P from saved max and sum) and compute_dSij.
#include "common.cuh"
#include "kernels.h"

namespace sfa {

namespace {

constexpr int kKeys = 128;          // keys per work item (MMA M)
constexpr int kStages = 5;
constexpr int kProducerWarps = 3;
constexpr int kThreads = 256;       // warp 0 MMA, 1-3 producers, 4-7 epilogue

template <int GP>
struct SdpSmem {
  static constexpr int kA = kKeys * 128;   // one 64-wide panel of 128 key rows
  static constexpr int kB = GP * 128;      // one 64-wide panel of GP head rows
  static constexpr int kStage = kA + kB;
  static constexpr int kBytes = kStages * kStage + 1024;  // + alignment slack
};

template <typename T, int GP, int MODE>
__global__ void __launch_bounds__(kThreads, 1) sdp_kernel(Prob p, void* out_p, void* out_ds, float* tile_stats, int* gerr) {
  using E = Elt<T>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full_bar[kStages], empty_bar[kStages], tfull_bar[2], tempty_bar[2];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ float red_buf[4][GP][2];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool bwd = (MODE == kModeBwd);
  const int nS = p.has_rope ? 9 : 8;           // 64-wide chunks of the score contraction
  const int nchunks = bwd ? nS + 8 : nS;      // + 8 chunks of dP
  const int ntiles = p.Kpad / kKeys;
  const int nitems = p.ntok * ntiles;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], kProducerWarps * 32);
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      mbar_init(&tempty_bar[i], 128);
    }
    abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kKeys, GP, E::is_f16, false, false);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int item = blockIdx.x; item < nitems && !abort_flag; item += gridDim.x, ++it) {
        const int set = it & 1;
        const uint32_t tph = (it >> 1) & 1;
        if (!mbar_wait(&tempty_bar[set], tph ^ 1, &abort_flag, gerr)) break;
        tc_fence_after();
        const uint32_t tS = tbase + set * (2 * GP);
        const uint32_t tP = tS + GP;
        for (int c = 0; c < nchunks; ++c) {
          if (!mbar_wait(&full_bar[stage], phase, &abort_flag, gerr)) break;
          tc_fence_after();
          const uint32_t a = smem_u32(smem + stage * SdpSmem<GP>::kStage);
          const uint32_t b = a + SdpSmem<GP>::kA;
          const uint32_t d = c < nS ? tS : tP;
          const bool first = (c == 0 || c == nS);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ss(d, sdesc_kmajor(a, ks), sdesc_kmajor(b, ks), idesc, (first && ks == 0) ? 0u : 1u);
          mma_commit(&empty_bar[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        mma_commit(&tfull_bar[set]);
      }
    }
    __syncwarp();
  } else if (warp <= kProducerWarps) {
    // ---------------------------------------------------------------- producers (cp.async gathers)
    const int pt = threadIdx.x - 32;          // 0 .. 95
    constexpr int kNP = kProducerWarps * 32;
    constexpr int kRows = kKeys + GP;         // rows per stage
    constexpr int kMine = (kRows + kNP - 1) / kNP;
    const T* q = static_cast<const T*>(p.q);
    const T* qr = static_cast<const T*>(p.qr);
    const T* k = static_cast<const T*>(p.k);
    const T* kr = static_cast<const T*>(p.kr);
    const T* v = static_cast<const T*>(p.v);
    const T* dO = static_cast<const T*>(p.dO);
    int stage = 0;
    uint32_t phase = 0;
    int issued = 0, signalled = 0;
    int sig_stage = 0;
    constexpr int kLag = 2;
    for (int item = blockIdx.x; item < nitems && !abort_flag; item += gridDim.x) {
      const int tl = item / ntiles, kt = item % ntiles;
      const int t = p.tok0 + tl;
      const TokMeta m = p.meta[t];
      int rowid[kMine];   // >= 0: kv row (A) ; for B rows: head index ; -1: zero fill
#pragma unroll
      for (int i = 0; i < kMine; ++i) {
        const int r = pt + i * kNP;
        if (r < kKeys) rowid[i] = slot_row(p, m, t, kt * kKeys + r);
        else if (r < kRows) rowid[i] = (r - kKeys) < p.G ? (r - kKeys) : -1;
        else rowid[i] = -1;
      }
      for (int c = 0; c < nchunks; ++c) {
        if (!mbar_wait(&empty_bar[stage], phase ^ 1, &abort_flag, gerr)) break;
        const uint32_t a = smem_u32(smem + stage * SdpSmem<GP>::kStage);
        const uint32_t b = a + SdpSmem<GP>::kA;
#pragma unroll
        for (int i = 0; i < kMine; ++i) {
          const int r = pt + i * kNP;
          if (r >= kRows) continue;
          const T* src;
          uint32_t dst;
          const int id = rowid[i];
          if (r < kKeys) {
            dst = a;
            const int rr = id < 0 ? 0 : id;
            if (c < 8) src = k + (size_t)rr * 512 + c * 64;
            else if (c < nS) src = kr + (size_t)rr * 64;
            else src = v + (size_t)rr * 512 + (c - nS) * 64;
          } else {
            const int h = r - kKeys;
            dst = b;
            const size_t tok = (size_t)t * p.G + (id < 0 ? 0 : id);
            if (c < 8) src = q + tok * 512 + c * 64;
            else if (c < nS) src = qr + tok * 64;
            else src = dO + tok * 512 + (c - nS) * 64;
          }
          const uint32_t nb = id < 0 ? 0u : 16u;
          const uint32_t row = (r < kKeys) ? r : (r - kKeys);
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) cp_async16(dst + swz_chunk(row, cc), src + cc * 8, nb);
        }
        cp_async_commit();
        ++issued;
        if (issued - signalled > kLag) {
          cp_async_wait<kLag>();
          fence_async_smem();
          mbar_arrive(&full_bar[sig_stage]);
          if (++sig_stage == kStages) sig_stage = 0;
          ++signalled;
        }
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
    }
    cp_async_wait<0>();
    fence_async_smem();
    while (signalled < issued) {
      mbar_arrive(&full_bar[sig_stage]);
      if (++sig_stage == kStages) sig_stage = 0;
      ++signalled;
    }
  } else {
    // ---------------------------------------------------------------- epilogue (thread = key)
    const int ew = warp - 4;              // TMEM lane quadrant
    const int key = ew * 32 + lane;
    const float log2e = 1.4426950408889634f;
    const float sl2 = p.scale * log2e;
    int it = 0;
    // The forward-statistics path uses named barriers between the four
    // epilogue warps, so its trip count never depends on the abort flag: an
    // abandoned wait only skips the work of the item.
    for (int item = blockIdx.x; item < nitems && (MODE == kModeFwdStats || !abort_flag); item += gridDim.x, ++it) {
      const int set = it & 1;
      const uint32_t tph = (it >> 1) & 1;
      const int tl = item / ntiles, kt = item % ntiles;
      const int t = p.tok0 + tl;
      const int slot = kt * kKeys + key;
      const int row = slot_row(p, p.meta[t], t, slot);
      const bool valid = row >= 0;
      const bool ok = !abort_flag && mbar_wait(&tfull_bar[set], tph, &abort_flag, gerr);
      if (!ok && MODE != kModeFwdStats) break;
      tc_fence_after();
      const uint32_t tS = tbase + set * (2 * GP) + ((uint32_t)(ew * 32) << 16);
      const uint32_t tP = tS + GP;
      const float* smax = p.smax + (size_t)t * p.G;
      const float* ssum = p.ssum + (size_t)t * p.G;
      const float* dsum = p.dsum + (size_t)t * p.G;
      if (MODE == kModeFwdStats) {
        // per head over the tile's valid keys: max of the raw score s and
        // sum of exp((s - max) * scale)
#pragma unroll 1
        for (int hc = 0; hc < GP / 32; ++hc) {
          float s[32];
          if (ok) tmem_ld32(tS + hc * 32, s);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float x = (valid && ok) ? s[j] : -INFINITY;
            float mx = x;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            float e = (x == -INFINITY) ? 0.f : exp2f((x - mx) * sl2);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
            if (lane == 0) {
              red_buf[ew][hc * 32 + j][0] = mx;
              red_buf[ew][hc * 32 + j][1] = e;
            }
          }
        }
        tc_fence_before();
        if (ok) mbar_arrive(&tempty_bar[set]);
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (key < p.G) {
          float mx = -INFINITY;
          for (int w = 0; w < 4; ++w) mx = fmaxf(mx, red_buf[w][key][0]);
          float l = 0.f;
          if (mx != -INFINITY)
            for (int w = 0; w < 4; ++w)
              if (red_buf[w][key][0] != -INFINITY) l += red_buf[w][key][1] * exp2f((red_buf[w][key][0] - mx) * sl2);
          float* ts = tile_stats + (((size_t)tl * ntiles + kt) * p.G + key) * 2;
          ts[0] = mx;   // raw score (unscaled)
          ts[1] = l;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        continue;
      }
      T* prow = static_cast<T*>(out_p) + ((size_t)tl * p.Kpad + slot) * GP;
      T* dsrow = bwd ? static_cast<T*>(out_ds) + ((size_t)tl * p.Kpad + slot) * GP : nullptr;
#pragma unroll 1
      for (int hc = 0; hc < GP / 32; ++hc) {
        float s[32], dp[32];
        tmem_ld32(tS + hc * 32, s);
        if (bwd) tmem_ld32(tP + hc * 32, dp);
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          float pv[2], dv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int h = hc * 32 + j + u;
            float pp = 0.f, dd = 0.f;
            if (valid && h < p.G) {
              const float l = __ldg(ssum + h);
              if (l > 0.f) {
                const float mlog = __ldg(smax + h) * log2e;
                pp = exp2f(s[j + u] * sl2 - mlog) * (1.0f / l);
                if (bwd) dd = pp * (dp[j + u] - __ldg(dsum + h)) * p.scale;
              }
            }
            pv[u] = pp;
            dv[u] = dd;
          }
          pk[j / 2] = E::pack(pv[0], pv[1]);
          dk[j / 2] = E::pack(dv[0], dv[1]);
        }
        uint4* pd = reinterpret_cast<uint4*>(prow + hc * 32);
#pragma unroll
        for (int u = 0; u < 4; ++u) pd[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        if (bwd) {
          uint4* dd = reinterpret_cast<uint4*>(dsrow + hc * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u) dd[u] = make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty_bar[set]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <typename T, int GP, int MODE>
cudaError_t launch_one(const Prob& p, void* out_p, void* out_ds, float* tile_stats, int* gerr, int nsm,
                       cudaStream_t st) {
  auto kern = sdp_kernel<T, GP, MODE>;
  const int smem = SdpSmem<GP>::kBytes > kOneCtaSmem ? SdpSmem<GP>::kBytes : kOneCtaSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nitems = p.ntok * (p.Kpad / kKeys);
  const int grid = nitems < nsm ? nitems : nsm;
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, kThreads, smem, st>>>(p, out_p, out_ds, tile_stats, gerr);
  return cudaGetLastError();
}

}  // namespace

template <typename T>
cudaError_t launch_sdp(const Prob& p, int mode, void* out_p, void* out_ds, float* tile_stats, int* gerr, int nsm,
                       cudaStream_t st) {
  if (p.Gp == 64) {
    if (mode == kModeBwd) return launch_one<T, 64, kModeBwd>(p, out_p, out_ds, tile_stats, gerr, nsm, st);
    if (mode == kModeFwdStats) return launch_one<T, 64, kModeFwdStats>(p, out_p, out_ds, tile_stats, gerr, nsm, st);
    return launch_one<T, 64, kModeFwdP>(p, out_p, out_ds, tile_stats, gerr, nsm, st);
  }
  if (mode == kModeBwd) return launch_one<T, 128, kModeBwd>(p, out_p, out_ds, tile_stats, gerr, nsm, st);
  if (mode == kModeFwdStats) return launch_one<T, 128, kModeFwdStats>(p, out_p, out_ds, tile_stats, gerr, nsm, st);
  return launch_one<T, 128, kModeFwdP>(p, out_p, out_ds, tile_stats, gerr, nsm, st);
}

template cudaError_t launch_sdp<__nv_bfloat16>(const Prob&, int, void*, void*, float*, int*, int, cudaStream_t);
template cudaError_t launch_sdp<__half>(const Prob&, int, void*, void*, float*, int*, int, cudaStream_t);

}  // namespace sfa
