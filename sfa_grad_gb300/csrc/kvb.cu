// Key-major dK / dV for block-sparse indices (sparseBlockSize >= 16).
//
// An index r of token t selects the bs consecutive kv rows starting at
// g = kv_start(t) + r.  Every (token, index) pair with the same start g adds
// to the same bs key rows, so instead of reducing each pair's 1088-float rows
// into the accumulator (4352 B per key per pair), the pairs are grouped by g
// and each group's sums are formed in tensor memory:
//     [dK || dKRope]^T(g .. g+bs) = sum over the group's pairs of
//                                   [q || qRope](t)^T . dS^T(t, slots of r)
//     dV^T(g .. g+bs)             = sum of dO(t)^T . P^T(t, slots of r)
// with features on the MMA's M side (128 per accumulator), the block's keys
// on N and the token's heads on K; the finished tile is added to the
// accumulator once per group.
//
// Grouping (per token chunk): count pairs per start row, scan into offsets and
// a list of non-empty starts, scatter the pairs.  A start may lie up to bs-1
// rows below its segment (an index r > -bs still covers keys 0 .. r+bs-1), so
// start g is binned at g + bs.  Pairs whose block has no attendable key (all
// keys below 0, or the start past the causal / segment limit) are left out;
// keys of a block outside the segment or beyond the limit carry P = dS = 0
// from the score kernel and add nothing (rows below 0 are not written).
//
// aclnnSparseFlashAttentionGrad doc, 阶段1 (dV = P^T dO) and 阶段3 (dK);
// 参数说明 sparseBlockSize (a selected block of contiguous keys).
#include "common.cuh"
#include "kernels.h"

namespace sfa {

namespace {

constexpr int kThreads = 256;   // warp 0: MMA issuer, warps 1..nprod: TMA producers, warps 4-7: epilogue
constexpr int kAccRow = 1088;
constexpr int kMaxStages = 6;
constexpr int kStageCap = 200 * 1024;   // shared memory for the operand ring

// Pair (token, index) of the chunk and whether its block can contribute;
// bin = start row + bs, in [1, T2 + bs).
__device__ __forceinline__ bool pair_start(const Prob& p, long long i, int& bin) {
  const int tl = (int)(i / p.Kidx), ii = (int)(i - (long long)tl * p.Kidx);
  const int t = p.tok0 + tl;
  const int r = __ldg(p.idx + (size_t)t * p.Kidx + ii);
  const TokMeta m = p.meta[t];
  if ((long long)r + p.bs <= 0 || r > m.limit) return false;
  const long long g = (long long)m.kv_start + r;
  if (g >= p.T2) return false;
  bin = (int)(g + p.bs);
  return true;
}

// Counts the chunk's pairs per bin.  With staging buffers given, it also
// zeroes the staged P^T / dS^T rows that the key-major score kernel (sdpb.cu)
// does not write: those of pairs left out of every group and of the padding
// slots past K * bs, which the query-side contraction still reads.
__global__ void blk_count_kernel(Prob p, int* cnt, uint8_t* pst, uint8_t* dsst, float* ts, int rowbytes) {
  const int nb = p.Kpad / p.bs;   // index positions per token, padding included
  const long long n = (long long)p.ntok * nb;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int tl = (int)(i / nb), ii = (int)(i - (long long)tl * nb);
    int bin;
    if (ii < p.Kidx && pair_start(p, (long long)tl * p.Kidx + ii, bin)) {
      atomicAdd(cnt + bin, 1);
      continue;
    }
    const size_t off = ((size_t)tl * p.Kpad + (size_t)ii * p.bs) * rowbytes;
    for (int k = 0; k < p.bs * rowbytes / 16; ++k) {
      if (pst) reinterpret_cast<uint4*>(pst + off)[k] = make_uint4(0, 0, 0, 0);
      if (dsst) reinterpret_cast<uint4*>(dsst + off)[k] = make_uint4(0, 0, 0, 0);
    }
    if (ts && ii < p.Kidx) {
      float2* e = reinterpret_cast<float2*>(ts) + ((size_t)tl * p.Kidx + ii) * p.G;
      for (int h = 0; h < p.G; ++h) e[h] = make_float2(-INFINITY, 0.f);
    }
  }
}

// One block: exclusive scan of the per-bin counts (nbins entries) into
// cursor[] (the next free entry of each bin), and the compacted list of
// non-empty bins with their first entry: groups[k], gbeg[k];
// gbeg[ngroups] = total entries.  The block walks the bins 4096 at a time
// (four consecutive bins per thread, coalesced), scanning each tile with warp
// shuffles and carrying the running totals.
// With nres given (key-major blocks, bins = start + bs), also the number of
// non-empty bins per residue bin % bs (nres[0 .. bs)).
__global__ void __launch_bounds__(1024) blk_scan_kernel(const int* cnt, int nbins, int* cursor, int* groups, int* gbeg,
                                                        int* ngroups, int bs, int* nres) {
  __shared__ int ex_sum[32], ex_nz[32];
  __shared__ int carry[2];
  __shared__ int res_cnt[64];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry[0] = carry[1] = 0;
  if (tid < 64) res_cnt[tid] = 0;
  __syncthreads();
  for (int base = 0; base < nbins; base += 4096) {
    const int b0 = base + tid * 4;
    int c[4], sum = 0, nz = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      c[u] = b0 + u < nbins ? cnt[b0 + u] : 0;
      sum += c[u];
      nz += c[u] > 0;
    }
    int is = sum, in = nz;   // inclusive scans within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, is, o), b = __shfl_up_sync(0xffffffffu, in, o);
      if (lane >= o) {
        is += a;
        in += b;
      }
    }
    if (lane == 31) {
      ex_sum[warp] = is;
      ex_nz[warp] = in;
    }
    __syncthreads();
    if (warp == 0) {
      const int v = ex_sum[lane], w = ex_nz[lane];
      int a = v, b = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, a, o), y = __shfl_up_sync(0xffffffffu, b, o);
        if (lane >= o) {
          a += x;
          b += y;
        }
      }
      ex_sum[lane] = a - v;
      ex_nz[lane] = b - w;
    }
    __syncthreads();
    int off = carry[0] + ex_sum[warp] + is - sum, k = carry[1] + ex_nz[warp] + in - nz;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (b0 + u < nbins) {
        cursor[b0 + u] = off;
        if (c[u] > 0) {
          groups[k] = b0 + u;
          gbeg[k] = off;
          ++k;
          if (nres) atomicAdd(&res_cnt[(b0 + u) % bs], 1);
        }
        off += c[u];
      }
    }
    __syncthreads();
    if (tid == 1023) {   // the tile's last bins: running totals through the tile
      carry[0] = off;
      carry[1] = k;
    }
    __syncthreads();
  }
  if (tid == 0) {
    *ngroups = carry[1];
    gbeg[carry[1]] = carry[0];
  }
  if (nres && tid < bs) nres[tid] = res_cnt[tid];
}

__global__ void blk_scatter_kernel(Prob p, int* cursor, int* entries) {
  const long long n = (long long)p.ntok * p.Kidx;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    int bin;
    if (pair_start(p, i, bin)) entries[atomicAdd(cursor + bin, 1)] = (int)i;
  }
}

// Shared-memory stage: A = 9 (or 8) feature panels of GK head rows each
// (MN-major: 64 features x GK K-rows, 128-byte swizzle), then B = 64 slot rows
// x 64 heads of the staged dS^T or P^T (K-major).
__host__ __device__ constexpr int stage_bytes(int gk) { return 9 * gk * 128 + 64 * 128; }

// GK (the token's heads rounded up to 16) is a template parameter: the MMA
// issue path is one thread whose instruction latency is not hidden, and with
// compile-time K steps and panel offsets a pair's 4-5 MMAs issue back to back
// (runtime trip counts cost about four times the MMA time).
// res >= 0 (deterministic mode): only the groups whose start is congruent to
// res modulo bs.  Two such blocks never share a key row, so every key row
// receives at most one tile per launch, and the launches for res = 0 .. bs-1
// run in stream order: each row's sum has one fixed order.  res < 0: every
// group.
template <typename T, int GK>
__global__ void __launch_bounds__(kThreads, 1) kvb_kernel(const __grid_constant__ BlkMaps maps, Prob p, int bs,
                                                          int nstages, int nprod, const int* groups, const int* gbeg,
                                                          const int* ngroups_p, const int* entries, float* acc,
                                                          int res, const int* nres, int* gerr) {
  if (res >= 0 && nres[res] == 0) return;   // no group with this start residue
  using E = Elt<T>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages], tfull_bar, tempty_bar, done_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = *ngroups_p;
  const int nitems = 2 * ngroups;          // (group, dK | dV)
  constexpr int gk = GK;
  constexpr int sbytes = stage_bytes(GK);
  constexpr int panel = GK * 128;          // one 64-feature panel of GK head rows
  constexpr int nks = GK / 16;             // K steps per pair

  if (threadIdx.x == 0) {
    for (int i = 0; i < nstages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    mbar_init(&tfull_bar, 1);
    mbar_init(&tempty_bar, 128);
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

  // chunks of an item: dK = 4 panels pairs of q (+ 1 rope panel), dV = 4 of dO
  auto nchunks_of = [&](int kind) { return kind == 0 ? (p.has_rope ? 5 : 4) : 4; };
  // whether this launch takes group grp (bins are start + bs >= 1)
  auto taken = [&](int grp) { return res < 0 || __ldg(groups + grp) % bs == res; };

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, bs, E::is_f16, true, false);
      const uint64_t d0 = sdesc_mnmajor(smem_u32(smem), 0, gk);
      const uint64_t b0 = sdesc_kmajor(smem_u32(smem + 9 * panel), 0);
      const uint32_t dcol[5] = {tbase, tbase + bs, tbase + 2 * bs, tbase + 3 * bs, tbase + 4 * bs};
      int s = 0, it = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x) {
        const int grp = item >> 1, kind = item & 1;
        if (!taken(grp)) continue;
        const bool five = nchunks_of(kind) == 5;
        const int e0 = gbeg[grp], e1 = gbeg[grp + 1];
        ok = mbar_wait_poll(&tempty_bar, (it & 1) ^ 1, wt);
        if (!ok) break;
        tc_fence_after();
        for (int e = e0; e < e1 && ok; ++e) {
          ok = mbar_wait_poll(&full_bar[s], ph, wt);
          if (!ok) break;
          tc_fence_after();
          const uint64_t sa = d0 + desc_off(s * sbytes), sb = b0 + desc_off(s * sbytes);
          const uint32_t acc0 = e > e0 ? 1u : 0u;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int ks = 0; ks < nks; ++ks)
              mma_ss(dcol[c], sa + desc_off(2 * c * panel) + (uint64_t)(ks * 128), sb + (uint64_t)(ks * 2), idesc,
                     ks > 0 ? 1u : acc0);
          if (five) {
#pragma unroll
            for (int ks = 0; ks < nks; ++ks)
              mma_ss(dcol[4], sa + desc_off(8 * panel) + (uint64_t)(ks * 128), sb + (uint64_t)(ks * 2), idesc,
                     ks > 0 ? 1u : acc0);
          }
          mma_commit(&empty_bar[s]);
          if (++s == nstages) {
            s = 0;
            ph ^= 1;
          }
        }
        if (ok) mma_commit(&tfull_bar);
        ++it;
      }
      mma_settle(&done_bar, gerr);   // no MMA still writing tensor memory at exit
    }
    __syncwarp();
  } else if (warp <= nprod) {
    // One thread per producer warp issues two or three boxes per pair; nprod
    // producers take every nprod-th pair.  nstages is a multiple of nprod, so
    // each stage slot has one producer and is refilled in order.
    if (lane == 0) {
      const int me = warp - 1;
      int g = 0;
      bool ok = true;
      ArmLog alog;
      for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x) {
        const int grp = item >> 1, kind = item & 1;
        if (!taken(grp)) continue;
        const int nc = nchunks_of(kind);
        const int e0 = gbeg[grp], e1 = gbeg[grp + 1];
        const uint32_t abytes = (kind == 0 && p.has_rope ? 9 : 8) * panel;
        for (int e = e0; e < e1 && ok; ++e, ++g) {
          if (g % nprod != me) continue;
          const int s = g % nstages;
          ok = mbar_wait(&empty_bar[s], ((g / nstages) & 1) ^ 1, wt);
          if (!ok) break;
          const int pr = __ldg(entries + e);
          const int tl = pr / p.Kidx, ii = pr - tl * p.Kidx;
          const int hrow = (p.tok0 + tl) * p.G;
          uint64_t* fb = &full_bar[s];
          const uint32_t base = smem_u32(smem + s * sbytes);
          mbar_expect_tx(fb, abytes + 64 * 128);
          alog.arm(s, (uint32_t)(g / nstages));
          // all eight 64-feature panels of the token's head rows in one box,
          // plus the rope panel
          tma_3d(base, kind == 0 ? &maps.q : &maps.dO, 0, hrow, 0, fb);
          if (nc == 5) tma_2d(base + 8 * panel, &maps.qr, 0, hrow, fb);
          tma_2d(base + 9 * panel, kind == 0 ? &maps.dS : &maps.P, 0, tl * p.Kpad + ii * bs, fb);
        }
      }
      alog.settle(full_bar, gerr);   // no copy still landing in shared memory at exit
    }
    __syncwarp();
  } else if (warp >= 4) {
    // Epilogue: warp w reads TMEM lanes (features) 32*(w%4) .. +31.  For
    // each accumulator and each key of the block, the warp's 32 lanes add 32
    // consecutive floats of that key's accumulator row.
    const int qd = warp & 3;
    const int f = qd * 32 + lane;
    int it = 0;
    for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
      const int grp = item >> 1, kind = item & 1;
      if (!taken(grp)) continue;
      const int nc = nchunks_of(kind);
      const int g0 = groups[grp] - bs;   // first key row (may be below 0)
      const bool ok = __all_sync(0xffffffffu, !abort_flag && mbar_wait(&tfull_bar, it & 1, wt));
      if (ok) {
        tc_fence_after();
        for (int c = 0; c < nc; ++c) {
          const bool rope = kind == 0 && c == 4;
          const int col = kind == 0 ? (rope ? 512 : c * 128) : 576 + c * 128;
          const bool live = !rope || f < 64;
          for (int u0 = 0; u0 < bs; u0 += 32) {
            float v[32];
            tmem_ld32(tbase + c * bs + u0 + ((uint32_t)(qd * 32) << 16), v);
            const int nu = bs - u0 < 32 ? bs - u0 : 32;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int row = g0 + u0 + j;
              if (j < nu && live && row >= 0 && row < p.T2)
                atomicAdd(acc + (size_t)row * kAccRow + col + f, v[j]);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty_bar);
      ++it;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace

cudaError_t launch_blk_count(const Prob& p, int* cnt, void* pst, void* dsst, float* tile_stats, cudaStream_t st) {
  if (p.ntok <= 0 || p.T2 <= 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(cnt, 0, (size_t)(p.T2 + p.bs) * sizeof(int), st);
  if (e != cudaSuccess) return e;
  const long long n = (long long)p.ntok * (p.Kpad / p.bs);
  const int grid = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  blk_count_kernel<<<grid, 256, 0, st>>>(p, cnt, static_cast<uint8_t*>(pst), static_cast<uint8_t*>(dsst), tile_stats,
                                         p.Gs * 2);
  return cudaGetLastError();
}

cudaError_t launch_blk_scan(const int* cnt, int nbins, int* cursor, int* groups, int* gbeg, int* ngroups, int bs,
                            int* nres, cudaStream_t st) {
  if (nbins <= 0) return cudaSuccess;
  blk_scan_kernel<<<1, 1024, 0, st>>>(cnt, nbins, cursor, groups, gbeg, ngroups, bs, nres);
  return cudaGetLastError();
}

cudaError_t launch_blk_scatter(const Prob& p, int* cursor, int* entries, cudaStream_t st) {
  if (p.ntok <= 0 || p.T2 <= 0) return cudaSuccess;
  const long long n = (long long)p.ntok * p.Kidx;
  const int grid = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  blk_scatter_kernel<<<grid, 256, 0, st>>>(p, cursor, entries);
  return cudaGetLastError();
}

namespace {
int kvb_stages(int gk) {
  const int s = kStageCap / stage_bytes(gk);
  return s < kMaxStages ? s : kMaxStages;
}
}  // namespace

template <typename T>
cudaError_t launch_kvb(const BlkMaps& maps, const Prob& p, int bs, const int* groups, const int* gbeg,
                       const int* ngroups, const int* entries, float* acc, int res, const int* nres, int* gerr,
                       int nsm, cudaStream_t st) {
  if (p.ntok <= 0 || p.T2 <= 0) return cudaSuccess;
  const int gk = (p.G + 15) / 16 * 16;
  const int nst = kvb_stages(gk);
  const int nprod = nst % 3 == 0 ? 3 : nst % 2 == 0 ? 2 : 1;
  const int smem_b = nst * stage_bytes(gk) + 1024;
  const int smem = smem_b > kOneCtaSmem ? smem_b : kOneCtaSmem;
  auto kern = gk == 16 ? kvb_kernel<T, 16> : gk == 32 ? kvb_kernel<T, 32> : gk == 48 ? kvb_kernel<T, 48> : kvb_kernel<T, 64>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<nsm, kThreads, smem, st>>>(maps, p, bs, nst, nprod, groups, gbeg, ngroups, entries, acc, res, nres, gerr);
  return cudaGetLastError();
}

template cudaError_t launch_kvb<__nv_bfloat16>(const BlkMaps&, const Prob&, int, const int*, const int*, const int*,
                                               const int*, float*, int, const int*, int*, int, cudaStream_t);
template cudaError_t launch_kvb<__half>(const BlkMaps&, const Prob&, int, const int*, const int*, const int*,
                                        const int*, float*, int, const int*, int*, int, cudaStream_t);

}  // namespace sfa
