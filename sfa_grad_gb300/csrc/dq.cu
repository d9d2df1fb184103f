// Query-side contraction over a token's selected keys, on the tensor cores:
//   mode 0:  [dQ || dQRope](t) = dS(t) . [K || KRope]_sel   (3 chunks of 192 features;
//            the softmax scale is already folded into the stored dS)
//   mode 1:  O(t) = P(t) . V_sel                              (2 chunks of 256 features)
// Heads on M (padded to 128), features on N, keys (64 per pipeline stage) on K;
// the accumulator stays in tensor memory for the whole key loop and is written
// once, so dQ needs no atomics.
//
// aclnnSparseFlashAttentionGrad doc, 阶段3 (dQ = dS K[u] / sqrt(d)); MindSpore
// flash_attention_bwd.py, update_dQi.
#include "common.cuh"
#include "kernels.h"

namespace sfa {

namespace {

constexpr int kSlots = 64;         // keys per pipeline stage (MMA K extent)
constexpr int kStages = 4;
constexpr int kProducerWarps = 3;
constexpr int kThreads = 256;

template <int NCOL>
struct DqSmem {
  static constexpr int kA = 2 * kSlots * 128;            // two 64-head panels (heads 0-63, 64-127)
  static constexpr int kB = (NCOL / 64) * kSlots * 128;  // feature panels
  static constexpr int kStage = kA + kB;
  static constexpr int kBytes = kStages * kStage + 1024;
};

template <typename T, int GP, int MODE>
__global__ void __launch_bounds__(kThreads, 1) dq_kernel(Prob p, const T* Ast, T* out_main, T* out_rope, int* gerr) {
  using E = Elt<T>;
  constexpr int NCOL = MODE == 0 ? 192 : 256;
  constexpr int NPART = MODE == 0 ? 3 : 2;
  using S = DqSmem<NCOL>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full_bar[kStages], empty_bar[kStages], tfull_bar[2], tempty_bar[2];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunks = p.Kpad / kSlots;
  const int nitems = p.ntok * NPART;

  if (GP == 64) {
    // heads 64-127 do not exist: their A panel stays zero for the whole kernel
    for (int s = 0; s < kStages; ++s) {
      uint4* z = reinterpret_cast<uint4*>(smem + s * S::kStage + kSlots * 128);
      for (int i = threadIdx.x; i < kSlots * 128 / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
    }
    fence_async_smem();
  }
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
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, NCOL, E::is_f16, true, true);
      int stage = 0, it = 0;
      uint32_t phase = 0;
      for (int item = blockIdx.x; item < nitems && !abort_flag; item += gridDim.x, ++it) {
        const int set = it & 1;
        if (!mbar_wait(&tempty_bar[set], ((it >> 1) & 1) ^ 1, &abort_flag, gerr)) break;
        tc_fence_after();
        const uint32_t d = tbase + set * 256;
        for (int c = 0; c < nchunks; ++c) {
          if (!mbar_wait(&full_bar[stage], phase, &abort_flag, gerr)) break;
          tc_fence_after();
          const uint32_t a = smem_u32(smem + stage * S::kStage);
          const uint32_t b = a + S::kA;
#pragma unroll
          for (int ks = 0; ks < kSlots / 16; ++ks)
            mma_ss(d, sdesc_mnmajor(a, ks, kSlots), sdesc_mnmajor(b, ks, kSlots), idesc, (c == 0 && ks == 0) ? 0u : 1u);
          mma_commit(&empty_bar[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        mma_commit(&tfull_bar[set]);
      }
    }
    __syncwarp();
  } else if (warp <= kProducerWarps) {
    const int pt = threadIdx.x - 32;
    constexpr int kNP = kProducerWarps * 32;
    constexpr int kHP = GP / 64;
    constexpr int kFP = NCOL / 64;
    const T* k = static_cast<const T*>(MODE == 0 ? p.k : p.v);
    const T* kr = static_cast<const T*>(p.kr);
    int stage = 0, issued = 0, signalled = 0, sig_stage = 0;
    uint32_t phase = 0;
    constexpr int kLag = 2;
    for (int item = blockIdx.x; item < nitems && !abort_flag; item += gridDim.x) {
      const int tl = item / NPART, part = item % NPART;
      const int t = p.tok0 + tl;
      const TokMeta m = p.meta[t];
      const int f0 = part * NCOL;
      for (int c = 0; c < nchunks; ++c) {
        if (!mbar_wait(&empty_bar[stage], phase ^ 1, &abort_flag, gerr)) break;
        const uint32_t a = smem_u32(smem + stage * S::kStage);
        const uint32_t b = a + S::kA;
        const T* tile = Ast + ((size_t)tl * p.Kpad + (size_t)c * kSlots) * GP;
        // A: stored rows [slot][GP heads] -> MN-major head panels
        for (int r = pt; r < kSlots * kHP; r += kNP) {
          const int s = r % kSlots, hp = r / kSlots;
          const T* src = tile + (size_t)s * GP + hp * 64;
          const uint32_t dst = a + hp * (kSlots * 128);
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) cp_async16(dst + swz_chunk(s, cc), src + cc * 8, 16u);
        }
        // B: gathered key rows -> MN-major feature panels
        for (int r = pt; r < kSlots * kFP; r += kNP) {
          const int s = r % kSlots, fp = r / kSlots;
          const int row = slot_row(p, m, t, c * kSlots + s);
          const int f = f0 + fp * 64;
          const T* src;
          uint32_t nb = row >= 0 ? 16u : 0u;
          const int rr = row < 0 ? 0 : row;
          if (MODE == 1 || f < 512) src = k + (size_t)rr * 512 + f;
          else {
            src = p.has_rope ? kr + (size_t)rr * 64 + (f - 512) : k;
            if (!p.has_rope) nb = 0u;
          }
          const uint32_t dst = b + fp * (kSlots * 128);
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) cp_async16(dst + swz_chunk(s, cc), src + cc * 8, nb);
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
    // ---------------------------------------------------------------- epilogue (thread = head)
    const int ew = warp - 4;
    const int h = ew * 32 + lane;
    int it = 0;
    for (int item = blockIdx.x; item < nitems && !abort_flag; item += gridDim.x, ++it) {
      const int set = it & 1;
      const int tl = item / NPART, part = item % NPART;
      const int t = p.tok0 + tl;
      if (!mbar_wait(&tfull_bar[set], (it >> 1) & 1, &abort_flag, gerr)) break;
      tc_fence_after();
      const uint32_t td = tbase + set * 256 + ((uint32_t)(ew * 32) << 16);
      for (int c = 0; c < NCOL; c += 32) {
        float v[32];
        tmem_ld32(td + c, v);
        const int f = part * NCOL + c;
        T* dst = nullptr;
        if (h < p.G) {
          if (MODE == 1 || f < 512) dst = out_main + ((size_t)t * p.G + h) * 512 + f;
          else if (p.has_rope) dst = out_rope + ((size_t)t * p.G + h) * 64 + (f - 512);
        }
        if (dst) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = E::pack(v[2 * j], v[2 * j + 1]);
          uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
          for (int u = 0; u < 4; ++u) d4[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
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
cudaError_t launch_one(const Prob& p, const void* A, void* o1, void* o2, int* gerr, int nsm, cudaStream_t st) {
  constexpr int NCOL = MODE == 0 ? 192 : 256;
  constexpr int NPART = MODE == 0 ? 3 : 2;
  auto kern = dq_kernel<T, GP, MODE>;
  const int smem = DqSmem<NCOL>::kBytes > kOneCtaSmem ? DqSmem<NCOL>::kBytes : kOneCtaSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nitems = p.ntok * NPART;
  const int grid = nitems < nsm ? nitems : nsm;
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, kThreads, smem, st>>>(p, static_cast<const T*>(A), static_cast<T*>(o1), static_cast<T*>(o2), gerr);
  return cudaGetLastError();
}

}  // namespace

template <typename T>
cudaError_t launch_dq(const Prob& p, int mode, const void* A, void* out_main, void* out_rope, int* gerr, int nsm,
                      cudaStream_t st) {
  if (p.Gp == 64)
    return mode == 0 ? launch_one<T, 64, 0>(p, A, out_main, out_rope, gerr, nsm, st)
                     : launch_one<T, 64, 1>(p, A, out_main, out_rope, gerr, nsm, st);
  return mode == 0 ? launch_one<T, 128, 0>(p, A, out_main, out_rope, gerr, nsm, st)
                   : launch_one<T, 128, 1>(p, A, out_main, out_rope, gerr, nsm, st);
}

template cudaError_t launch_dq<__nv_bfloat16>(const Prob&, int, const void*, void*, void*, int*, int, cudaStream_t);
template cudaError_t launch_dq<__half>(const Prob&, int, const void*, void*, void*, int*, int, cudaStream_t);

}  // namespace sfa
