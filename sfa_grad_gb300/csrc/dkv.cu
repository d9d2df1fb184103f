// Key-side gradients.  For one query token and one 192/256-wide feature chunk
// of the key-side output row [dK (512) | dKRope (64) | dV (512)], it loops over
// the token's selected keys 128 at a time and forms, on the tensor cores,
//     dV_tile           = P^T  . dO            (keys x 256, contraction over heads)
//     [dK|dKRope]_tile  = dS^T . [q || qRope]  (keys x 192, scale already in dS)
// then scatters every valid key row into the fp32 accumulator with vector
// reductions (non-deterministic order), or writes it as a per-(token, slot)
// partial row for the fixed-order reduction.
//
// aclnnSparseFlashAttentionGrad doc, 阶段1 (dV = P^T dO) and 阶段3
// (dK = dS^T Q / sqrt(d)); MindSpore flash_attention_bwd.py, update_dVj and
// update_dKj (atomic accumulation into zero-initialised fp32 outputs).
#include "common.cuh"
#include "kernels.h"

namespace sfa {

namespace {

constexpr int kKeys = 128;
constexpr int kStages = 4;
constexpr int kProducerWarps = 3;
constexpr int kThreads = 256;
constexpr int kChunks = 5;        // dK 3 x 192, dV 2 x 256
constexpr int kAccRow = 1088;     // fp32 accumulator row: dK | dKRope | dV

__device__ __forceinline__ void chunk_geom(int ch, int& ncol, int& col0) {
  if (ch < 3) { ncol = 192; col0 = ch * 192; }
  else { ncol = 256; col0 = 576 + (ch - 3) * 256; }
}

template <int GP>
struct DkvSmem {
  static constexpr int kB = 4 * GP * 128;           // up to 4 feature panels of GP head rows
  static constexpr int kA = (GP / 64) * kKeys * 128;  // head panels of 128 slot rows
  static constexpr int kBytes = kB + kStages * kA + 1024;
};

__device__ __forceinline__ void red_add_v4(float* dst, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(dst), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

template <typename T, int GP, bool DET>
__global__ void __launch_bounds__(kThreads, 1) dkv_kernel(Prob p, const T* Pst, const T* dSst, float* acc,
                                                          float* partials, int* gerr) {
  using E = Elt<T>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = smem;
  uint8_t* sA = smem + DkvSmem<GP>::kB;
  __shared__ uint64_t full_bar[kStages], empty_bar[kStages], tfull_bar[2], tempty_bar[2], bempty_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = p.Kpad / kKeys;
  const int nitems = p.ntok * kChunks;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], kProducerWarps * 32);
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      mbar_init(&tempty_bar[i], 128);
    }
    mbar_init(&bempty_bar, 1);
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
      int stage = 0, tcount = 0, icount = 0;
      uint32_t phase = 0;
      for (int item = blockIdx.x; item < nitems && !abort_flag; item += gridDim.x, ++icount) {
        const int ch = item % kChunks;
        int ncol, col0;
        chunk_geom(ch, ncol, col0);
        const uint32_t idesc = idesc_f16(kKeys, ncol, E::is_f16, false, true);
        const uint32_t b = smem_u32(sB);
        for (int kt = 0; kt < ntiles; ++kt, ++tcount) {
          const int set = tcount & 1;
          if (!mbar_wait(&tempty_bar[set], ((tcount >> 1) & 1) ^ 1, &abort_flag, gerr)) break;
          if (!mbar_wait(&full_bar[stage], phase, &abort_flag, gerr)) break;
          tc_fence_after();
          const uint32_t a = smem_u32(sA + stage * DkvSmem<GP>::kA);
          const uint32_t d = tbase + set * 256;
#pragma unroll
          for (int ks = 0; ks < GP / 16; ++ks)
            mma_ss(d, sdesc_kmajor(a + (ks >> 2) * (kKeys * 128), ks & 3), sdesc_mnmajor(b, ks, GP), idesc,
                   ks > 0 ? 1u : 0u);
          mma_commit(&empty_bar[stage]);
          mma_commit(&tfull_bar[set]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        mma_commit(&bempty_bar);
      }
    }
    __syncwarp();
  } else if (warp <= kProducerWarps) {
    // ---------------------------------------------------------------- producers
    const int pt = threadIdx.x - 32;
    constexpr int kNP = kProducerWarps * 32;
    const T* q = static_cast<const T*>(p.q);
    const T* qr = static_cast<const T*>(p.qr);
    const T* dO = static_cast<const T*>(p.dO);
    int stage = 0, issued = 0, signalled = 0, sig_stage = 0, icount = 0;
    uint32_t phase = 0;
    constexpr int kLag = 2;
    constexpr int kHP = GP / 64;
    for (int item = blockIdx.x; item < nitems && !abort_flag; item += gridDim.x, ++icount) {
      const int tl = item / kChunks, ch = item % kChunks;
      const int t = p.tok0 + tl;
      int ncol, col0;
      chunk_geom(ch, ncol, col0);
      // flush: every issued tile must be signalled before waiting for the
      // previous item's MMAs to release the B panels
      cp_async_wait<0>();
      fence_async_smem();
      while (signalled < issued) {
        mbar_arrive(&full_bar[sig_stage]);
        if (++sig_stage == kStages) sig_stage = 0;
        ++signalled;
      }
      if (icount > 0 && !mbar_wait(&bempty_bar, (icount - 1) & 1, &abort_flag, gerr)) break;
      // B panels: GP head rows x ncol features, MN-major (feature panels)
      {
        const uint32_t b = smem_u32(sB);
        const int npan = ncol / 64;
        for (int r = pt; r < GP * npan; r += kNP) {
          const int h = r % GP, pb = r / GP;
          const int f = (ch < 3 ? col0 : col0 - 576) + pb * 64;   // feature in the source tensor
          const T* src;
          if (ch < 3) src = (f < 512 || !p.has_rope) ? q + ((size_t)t * p.G + (h < p.G ? h : 0)) * 512 + (f < 512 ? f : 0)
                                                     : qr + ((size_t)t * p.G + (h < p.G ? h : 0)) * 64 + (f - 512);
          else src = dO + ((size_t)t * p.G + (h < p.G ? h : 0)) * 512 + f;
          uint32_t nb = h < p.G ? 16u : 0u;
          if (ch < 3 && f >= 512 && !p.has_rope) { src = q; nb = 0u; }
          const uint32_t dst = b + pb * (GP * 128);
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) cp_async16(dst + swz_chunk(h, cc), src + cc * 8, nb);
        }
      }
      const T* Ast = ch < 3 ? dSst : Pst;
      for (int kt = 0; kt < ntiles; ++kt) {
        if (!mbar_wait(&empty_bar[stage], phase ^ 1, &abort_flag, gerr)) break;
        const uint32_t a = smem_u32(sA + stage * DkvSmem<GP>::kA);
        const T* tile = Ast + ((size_t)tl * p.Kpad + (size_t)kt * kKeys) * GP;
        for (int r = pt; r < kKeys * kHP; r += kNP) {
          const int s = r % kKeys, hp = r / kKeys;
          const T* src = tile + (size_t)s * GP + hp * 64;
          const uint32_t dst = a + hp * (kKeys * 128);
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) cp_async16(dst + swz_chunk(s, cc), src + cc * 8, 16u);
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
    // ---------------------------------------------------------------- drain (thread = slot)
    const int ew = warp - 4;
    const int key = ew * 32 + lane;
    int tcount = 0;
    for (int item = blockIdx.x; item < nitems && !abort_flag; item += gridDim.x) {
      const int tl = item / kChunks, ch = item % kChunks;
      const int t = p.tok0 + tl;
      const TokMeta m = p.meta[t];
      int ncol, col0;
      chunk_geom(ch, ncol, col0);
      for (int kt = 0; kt < ntiles; ++kt, ++tcount) {
        const int set = tcount & 1;
        const int slot = kt * kKeys + key;
        const int row = slot_row(p, m, t, slot);
        if (!mbar_wait(&tfull_bar[set], (tcount >> 1) & 1, &abort_flag, gerr)) break;
        tc_fence_after();
        const uint32_t td = tbase + set * 256 + ((uint32_t)(ew * 32) << 16);
        float* dst;
        if (DET) dst = partials + ((size_t)tl * p.Kpad + slot) * kAccRow + col0;
        else dst = acc + (size_t)(row < 0 ? 0 : row) * kAccRow + col0;
        for (int c = 0; c < ncol; c += 32) {
          float v[32];
          tmem_ld32(td + c, v);
          if (DET) {
            float4* d4 = reinterpret_cast<float4*>(dst + c);
#pragma unroll
            for (int u = 0; u < 8; ++u)
              d4[u] = row >= 0 ? make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3])
                               : make_float4(0.f, 0.f, 0.f, 0.f);
          } else if (row >= 0) {
#pragma unroll
            for (int u = 0; u < 8; ++u) red_add_v4(dst + c + 4 * u, v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty_bar[set]);
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

template <typename T, int GP>
cudaError_t launch_gp(const Prob& p, const void* P, const void* dS, float* acc, float* partials, int* gerr, int nsm,
                      cudaStream_t st) {
  const int smem = DkvSmem<GP>::kBytes > kOneCtaSmem ? DkvSmem<GP>::kBytes : kOneCtaSmem;
  const int nitems = p.ntok * kChunks;
  const int grid = nitems < nsm ? nitems : nsm;
  if (grid <= 0) return cudaSuccess;
  if (partials) {
    auto kern = dkv_kernel<T, GP, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, st>>>(p, static_cast<const T*>(P), static_cast<const T*>(dS), acc, partials, gerr);
  } else {
    auto kern = dkv_kernel<T, GP, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, st>>>(p, static_cast<const T*>(P), static_cast<const T*>(dS), acc, partials, gerr);
  }
  return cudaGetLastError();
}

}  // namespace

template <typename T>
cudaError_t launch_dkv(const Prob& p, const void* P, const void* dS, float* acc, float* partials, int* gerr, int nsm,
                       cudaStream_t st) {
  if (p.Gp == 64) return launch_gp<T, 64>(p, P, dS, acc, partials, gerr, nsm, st);
  return launch_gp<T, 128>(p, P, dS, acc, partials, gerr, nsm, st);
}

template cudaError_t launch_dkv<__nv_bfloat16>(const Prob&, const void*, const void*, float*, float*, int*, int,
                                               cudaStream_t);
template cudaError_t launch_dkv<__half>(const Prob&, const void*, const void*, float*, float*, int*, int, cudaStream_t);

}  // namespace sfa
