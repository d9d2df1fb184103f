// Deterministic key-side reduction (deterministic = 1; aclnnSparseFlashAttentionGrad
// doc, 约束说明 确定性计算).  The key-side kernel writes one partial row
// [dK | dKRope | dV] per (token, slot) of the chunk instead of using atomics,
// each element rounded once to bf16 (half the bytes of fp32 through HBM;
// the sums stay fp32); then, per chunk:
//  1. a stable counting sort of the chunk's (kv row, token, slot) entries:
//     count per kv row, scan into offsets and the list of rows that receive
//     anything, scatter the entry ids (token * Kpad + slot), then sort each
//     row's segment ascending, which fixes the (token, slot) order;
//  2. one block per receiving row adds the row's partial rows in that order
//     and adds the sum to the fp32 accumulator.
// Each key's sum therefore has one fixed order: chunk, token, slot.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace sfa {

namespace {

constexpr int kAccRow = 1088;
constexpr int kCols4 = kAccRow / 4;     // 272 float4 columns
// Segment sort: segments of up to kShortCap entries are sorted one per warp
// by a launch with many warps per SM; longer ones one per block by a second
// launch, in shared memory up to kLongCap entries and in global scratch
// beyond that.
constexpr int kSortWarps = 8;
constexpr int kShortCap = 1024;
constexpr int kLongCap = 4096;

__global__ void det_count_kernel(Prob p, int* cnt) {
  const long long n = (long long)p.ntok * p.Kpad;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int row = p.rowtab[i];
    if (row >= 0) atomicAdd(cnt + row, 1);
  }
}

__global__ void det_scatter_kernel(Prob p, int* cursor, int* ent) {
  const long long n = (long long)p.ntok * p.Kpad;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int row = p.rowtab[i];
    if (row >= 0) ent[atomicAdd(cursor + row, 1)] = (int)i;
  }
}

// Ascending bitonic sort of a[0 .. np) (np a power of two) by one warp.
__device__ __forceinline__ void warp_bitonic(int* a, int np, int lane) {
  for (int kk = 2; kk <= np; kk <<= 1) {
    for (int j = kk >> 1; j > 0; j >>= 1) {
      for (int i = lane; i < np; i += 32) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const int x = a[i], y = a[ixj];
          if ((x > y) == ((i & kk) == 0)) {
            a[i] = y;
            a[ixj] = x;
          }
        }
      }
      __syncwarp();
    }
  }
}

// One warp per receiving row sorts the row's entry ids ascending, for the
// segments of 2 .. kShortCap entries, in static shared memory.
__global__ void __launch_bounds__(256) det_segsort_kernel(const int* gbeg, const int* ngroups_p, int* ent) {
  __shared__ int buf[kSortWarps][kShortCap];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = *ngroups_p;
  for (int k = blockIdx.x * kSortWarps + warp; k < ngroups; k += gridDim.x * kSortWarps) {
    const int b = gbeg[k], n = gbeg[k + 1] - b;
    if (n <= 1 || n > kShortCap) continue;
    int np = 1;
    while (np < n) np <<= 1;
    int* a = buf[warp];
    for (int i = lane; i < np; i += 32) a[i] = i < n ? ent[b + i] : INT_MAX;
    __syncwarp();
    warp_bitonic(a, np, lane);
    for (int i = lane; i < n; i += 32) ent[b + i] = a[i];
    __syncwarp();
  }
}

// One block per longer segment (many occurrences of one key in the chunk):
// an ascending bitonic sort by 256 threads, in shared memory up to kLongCap
// entries, beyond that in a padded copy at scratch + 2 * begin, which never
// overlaps another segment's copy.
__global__ void __launch_bounds__(256) det_segsort_long_kernel(const int* gbeg, const int* ngroups_p, int* ent,
                                                               int* scratch) {
  __shared__ int buf[kLongCap];
  const int tid = threadIdx.x;
  const int ngroups = *ngroups_p;
  for (int k = blockIdx.x; k < ngroups; k += gridDim.x) {
    const int b = gbeg[k], n = gbeg[k + 1] - b;
    if (n <= kShortCap) continue;
    int np = 1;
    while (np < n) np <<= 1;
    int* a = np <= kLongCap ? buf : scratch + 2 * (size_t)b;
    for (int i = tid; i < np; i += 256) a[i] = i < n ? ent[b + i] : INT_MAX;
    __syncthreads();
    for (int kk = 2; kk <= np; kk <<= 1) {
      for (int j = kk >> 1; j > 0; j >>= 1) {
        for (int i = tid; i < np; i += 256) {
          const int ixj = i ^ j;
          if (ixj > i) {
            const int x = a[i], y = a[ixj];
            if ((x > y) == ((i & kk) == 0)) {
              a[i] = y;
              a[ixj] = x;
            }
          }
        }
        __syncthreads();
      }
    }
    for (int i = tid; i < n; i += 256) ent[b + i] = a[i];
    __syncthreads();
  }
}

// Four bf16 of a partial row (8 bytes) as fp32.
__device__ __forceinline__ float4 bf16x4(uint2 r) {
  return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xffff0000u), __uint_as_float(r.y << 16),
                     __uint_as_float(r.y & 0xffff0000u));
}

// One block (272 threads, four columns each) per receiving row k: adds the
// row's bf16 partial rows in sorted (token, slot) order in fp32, eight loads
// in flight.
__global__ void __launch_bounds__(kCols4) det_reduce_kernel(const int* groups, const int* gbeg, const int* ngroups_p,
                                                            const int* ent, const uint16_t* partials, float* acc) {
  const int ngroups = *ngroups_p;
  const int tid = threadIdx.x;
  for (int k = blockIdx.x; k < ngroups; k += gridDim.x) {
    const int row = groups[k];
    const int b = gbeg[k], e = gbeg[k + 1];
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    int i = b;
    for (; i + 8 <= e; i += 8) {
      uint2 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = __ldg(reinterpret_cast<const uint2*>(partials + (size_t)__ldg(ent + i + u) * kAccRow) + tid);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 f = bf16x4(v[u]);
        s.x += f.x; s.y += f.y; s.z += f.z; s.w += f.w;
      }
    }
    for (; i < e; ++i) {
      const float4 f =
          bf16x4(__ldg(reinterpret_cast<const uint2*>(partials + (size_t)__ldg(ent + i) * kAccRow) + tid));
      s.x += f.x; s.y += f.y; s.z += f.z; s.w += f.w;
    }
    float4* g = reinterpret_cast<float4*>(acc + (size_t)row * kAccRow) + tid;
    float4 x = *g;
    x.x += s.x; x.y += s.y; x.z += s.z; x.w += s.w;
    *g = x;
  }
}

int grid_for(long long n) { return (int)((n + 255) / 256 < 8192 ? (n + 255) / 256 : 8192); }

}  // namespace

cudaError_t launch_det_count(const Prob& p, int* cnt, cudaStream_t st) {
  if (p.ntok <= 0 || p.T2 <= 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(cnt, 0, (size_t)p.T2 * sizeof(int), st);
  if (e != cudaSuccess) return e;
  det_count_kernel<<<grid_for((long long)p.ntok * p.Kpad), 256, 0, st>>>(p, cnt);
  return cudaGetLastError();
}

cudaError_t launch_det_scatter(const Prob& p, int* cursor, int* ent, cudaStream_t st) {
  if (p.ntok <= 0 || p.T2 <= 0) return cudaSuccess;
  det_scatter_kernel<<<grid_for((long long)p.ntok * p.Kpad), 256, 0, st>>>(p, cursor, ent);
  return cudaGetLastError();
}

cudaError_t launch_det_sort(const Prob& p, const int* gbeg, const int* ngroups, int* ent, int* scratch, bool long_segs,
                            cudaStream_t st) {
  if (p.ntok <= 0 || p.T2 <= 0) return cudaSuccess;
  if (!long_segs) {
    const int grid = (p.T2 + 7) / 8 < 4096 ? (p.T2 + 7) / 8 : 4096;
    det_segsort_kernel<<<grid, 256, 0, st>>>(gbeg, ngroups, ent);
  } else {
    det_segsort_long_kernel<<<4 * 152, 256, 0, st>>>(gbeg, ngroups, ent, scratch);
  }
  return cudaGetLastError();
}

cudaError_t launch_det_reduce(const Prob& p, const int* groups, const int* gbeg, const int* ngroups, const int* ent,
                              const uint16_t* partials, float* acc, cudaStream_t st) {
  if (p.ntok <= 0 || p.T2 <= 0) return cudaSuccess;
  const int grid = p.T2 < 16384 ? p.T2 : 16384;
  det_reduce_kernel<<<grid, kCols4, 0, st>>>(groups, gbeg, ngroups, ent, partials, acc);
  return cudaGetLastError();
}

}  // namespace sfa
