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
constexpr int kStages = 3;
constexpr int kDrainThreads = 256;           // warps 4-11
constexpr int kThreads = 128 + kDrainThreads;
constexpr int kStgRow = 36;                   // floats per staged row (32 + pad)
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
  static constexpr int kStg = (kDrainThreads / 32) * 32 * kStgRow * 4;  // per-warp transpose buffers
  static constexpr int kBytes = kB + kStages * kA + kStg + 1024;
};

__device__ __forceinline__ void red_add_v4(float* dst, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(dst), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

template <typename T, int GP, bool DET>
__global__ void __launch_bounds__(kThreads, 1) dkv_kernel(const __grid_constant__ Maps maps, Prob p, float* acc,
                                                          float* partials, int* gerr) {
  using E = Elt<T>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = smem;
  uint8_t* sA = smem + DkvSmem<GP>::kB;
  float* sStg = reinterpret_cast<float*>(sA + kStages * DkvSmem<GP>::kA);
  __shared__ uint64_t full_bar[kStages], empty_bar[kStages], tfull_bar[2], tempty_bar[2], bempty_bar, bfull_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = p.Kpad / kKeys;
  const int nitems = p.ntok * kChunks;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      mbar_init(&tempty_bar[i], kDrainThreads);
    }
    mbar_init(&bempty_bar, 1);
    mbar_init(&bfull_bar, 1);
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
        if (!mbar_wait_poll(&bfull_bar, icount & 1, &abort_flag, gerr)) break;
        for (int kt = 0; kt < ntiles; ++kt, ++tcount) {
          const int set = tcount & 1;
          if (!mbar_wait_poll(&tempty_bar[set], ((tcount >> 1) & 1) ^ 1, &abort_flag, gerr)) break;
          if (!mbar_wait_poll(&full_bar[stage], phase, &abort_flag, gerr)) break;
          tc_fence_after();
          const uint64_t da = sdesc_kmajor(smem_u32(sA + stage * DkvSmem<GP>::kA), 0);
          const uint64_t db = sdesc_mnmajor(b, 0, GP);
          const uint32_t d = tbase + set * 256;
          mma_ss_k64<2, 128>(d, da, db, idesc, 0u);
          if (GP == 128) mma_ss_k64<2, 128>(d, da + desc_off(kKeys * 128), db + 512, idesc, 1u);
          mma_commit(&empty_bar[stage]);
          mma_commit(&tfull_bar[set]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        mma_commit(&bempty_bar);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- producer (TMA, lane 0)
    // Per item: the token's head rows of q / qRope / dO for the chunk's
    // feature panels (B, kept for the whole item); per key tile: the staged
    // P^T or dS^T rows as 64x64 boxes (A).
    if (lane == 0) {
      int stage = 0, icount = 0;
      uint32_t phase = 0;
      constexpr int kHP = GP / 64;
      bool ok = true;
      for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x, ++icount) {
        const int tl = item / kChunks, ch = item % kChunks;
        const int t = p.tok0 + tl;
        int ncol, col0;
        chunk_geom(ch, ncol, col0);
        if (icount > 0) ok = mbar_wait(&bempty_bar, (icount - 1) & 1, &abort_flag, gerr);
        if (!ok) break;
        {
          const uint32_t b = smem_u32(sB);
          const int npan = ncol / 64;
          mbar_expect_tx(&bfull_bar, npan * GP * 128);
          for (int pb = 0; pb < npan; ++pb) {
            const CUtensorMap* mp;
            int x, y = t * p.G;
            if (ch >= 3) { mp = &maps.dO; x = col0 - 576 + pb * 64; }
            else {
              const int f = col0 + pb * 64;
              if (f < 512) { mp = &maps.q; x = f; }
              else if (p.has_rope) { mp = &maps.qr; x = f - 512; }
              else { mp = &maps.q; x = 0; y = -2 * GP; }   // no rope part: rows outside the map read as zeros
            }
            tma_2d(b + pb * (GP * 128), mp, x, y, &bfull_bar);
          }
        }
        const CUtensorMap* mA = ch < 3 ? &maps.dS : &maps.P;
        for (int kt = 0; kt < ntiles && ok; ++kt) {
          ok = mbar_wait(&empty_bar[stage], phase ^ 1, &abort_flag, gerr);
          if (!ok) break;
          const uint32_t a = smem_u32(sA + stage * DkvSmem<GP>::kA);
          mbar_expect_tx(&full_bar[stage], DkvSmem<GP>::kA);
          const int y0 = tl * p.Kpad + kt * kKeys;
#pragma unroll
          for (int hp = 0; hp < kHP; ++hp) {
            tma_2d(a + hp * (kKeys * 128), mA, hp * 64, y0, &full_bar[stage]);
            tma_2d(a + hp * (kKeys * 128) + 64 * 128, mA, hp * 64, y0 + 64, &full_bar[stage]);
          }
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- drain
    // Eight warps: warp w reads TMEM lanes (slots) 32*(w%4) .. +31 and one
    // half of the chunk's columns.  Each 32-column slice is transposed through
    // a per-warp shared buffer so that one reduction instruction covers four
    // key rows x 128 contiguous bytes.
    const int q = warp & 3;
    const int half = (warp - 4) >> 2;
    const int key = q * 32 + lane;
    float* stg = sStg + (warp - 4) * 32 * kStgRow;
    int tcount = 0;
    for (int item = blockIdx.x; item < nitems && !abort_flag; item += gridDim.x) {
      const int tl = item / kChunks, ch = item % kChunks;
      int ncol, col0;
      chunk_geom(ch, ncol, col0);
      const int cbeg = half * (ncol / 2), cend = cbeg + ncol / 2;
      for (int kt = 0; kt < ntiles; ++kt, ++tcount) {
        const int set = tcount & 1;
        const int slot = kt * kKeys + key;
        const int row = p.rowtab[(size_t)tl * p.Kpad + slot];
        const bool ok = mbar_wait(&tfull_bar[set], (tcount >> 1) & 1, &abort_flag, gerr);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        const uint32_t td = tbase + set * 256 + ((uint32_t)(q * 32) << 16);
        for (int c = cbeg; c < cend; c += 32) {
          float v[32];
          tmem_ld32(td + c, v);
          float4* mine = reinterpret_cast<float4*>(stg + lane * kStgRow);
#pragma unroll
          for (int u = 0; u < 8; ++u) mine[u] = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
          __syncwarp();
#pragma unroll
          for (int rr = 0; rr < 8; ++rr) {
            const int rl = rr * 4 + (lane >> 3), c4 = lane & 7;
            const float4 x = reinterpret_cast<const float4*>(stg + rl * kStgRow)[c4];
            const int grow = __shfl_sync(0xffffffffu, row, rl);
            if (DET) {
              float* dst = partials + ((size_t)tl * p.Kpad + kt * kKeys + q * 32 + rl) * kAccRow + col0 + c + c4 * 4;
              *reinterpret_cast<float4*>(dst) = grow >= 0 ? x : make_float4(0.f, 0.f, 0.f, 0.f);
            } else if (grow >= 0) {
              red_add_v4(acc + (size_t)grow * kAccRow + col0 + c + c4 * 4, x.x, x.y, x.z, x.w);
            }
          }
          __syncwarp();
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
cudaError_t launch_gp(const Maps& maps, const Prob& p, float* acc, float* partials, int* gerr, int nsm,
                      cudaStream_t st) {
  const int smem = DkvSmem<GP>::kBytes > kOneCtaSmem ? DkvSmem<GP>::kBytes : kOneCtaSmem;
  const int nitems = p.ntok * kChunks;
  const int grid = nitems < nsm ? nitems : nsm;
  if (grid <= 0) return cudaSuccess;
  if (partials) {
    auto kern = dkv_kernel<T, GP, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, st>>>(maps, p, acc, partials, gerr);
  } else {
    auto kern = dkv_kernel<T, GP, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, st>>>(maps, p, acc, partials, gerr);
  }
  return cudaGetLastError();
}

}  // namespace

template <typename T>
cudaError_t launch_dkv(const Maps& maps, const Prob& p, float* acc, float* partials, int* gerr, int nsm,
                       cudaStream_t st) {
  if (p.Gp == 64) return launch_gp<T, 64>(maps, p, acc, partials, gerr, nsm, st);
  return launch_gp<T, 128>(maps, p, acc, partials, gerr, nsm, st);
}

template cudaError_t launch_dkv<__nv_bfloat16>(const Maps&, const Prob&, float*, float*, int*, int, cudaStream_t);
template cudaError_t launch_dkv<__half>(const Maps&, const Prob&, float*, float*, int*, int, cudaStream_t);

}  // namespace sfa
