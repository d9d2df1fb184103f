// Deterministic key-side reduction (deterministic = 1; aclnnSparseFlashAttentionGrad
// doc, 约束说明 确定性计算).  The key-side kernel writes one partial row
// [dK | dKRope | dV] per (token, slot) instead of using atomics; then
//  1. every token's (kv row, slot) pairs are sorted by (row, slot) in shared
//     memory (bitonic sort, a fixed network, so the result is unique), and
//  2. a block owning 4 consecutive kv rows walks the chunk's tokens in
//     ascending order, finds the rows it owns in each token's sorted list by
//     binary search, and adds the matching partial rows in (token, slot)
//     order into a shared-memory accumulator, which it finally adds to the
//     fp32 accumulator.  Each key's sum therefore has one fixed order: chunk,
//     token, slot.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace sfa {

namespace {

constexpr int kRowsPerBlock = 4;      // 17 KB of shared accumulator: several blocks per SM
constexpr int kAccRow = 1088;
constexpr int kCols4 = kAccRow / 4;     // 272 float4 columns
constexpr int kRedThreads = 288;
constexpr int kTokBatch = 256;
constexpr int kMaxMatch = 2048;

__global__ void __launch_bounds__(1024) sort_keys_kernel(Prob p, int npow2, int* skey, int* sslot) {
  extern __shared__ unsigned long long keys[];
  const int tl = blockIdx.x;
  const int t = p.tok0 + tl;
  const TokMeta m = p.meta[t];
  for (int s = threadIdx.x; s < npow2; s += blockDim.x) {
    unsigned long long key = ~0ull;
    if (s < p.Keff) {
      const int row = slot_row(p, m, t, s);
      if (row >= 0) key = ((unsigned long long)(unsigned)row << 32) | (unsigned)s;
    }
    keys[s] = key;
  }
  __syncthreads();
  for (int k = 2; k <= npow2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < npow2; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = keys[i], b = keys[ixj];
          const bool up = (i & k) == 0;
          if ((a > b) == up) {
            keys[i] = b;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  int* ko = skey + (size_t)tl * p.Kpad;
  int* so = sslot + (size_t)tl * p.Kpad;
  for (int r = threadIdx.x; r < p.Kpad; r += blockDim.x) {
    const unsigned long long key = keys[r];
    ko[r] = key == ~0ull ? INT_MAX : (int)(key >> 32);
    so[r] = (int)(key & 0xffffffffu);
  }
}

__device__ __forceinline__ int lower_bound(const int* a, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a + mid) < x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kRedThreads) det_reduce_kernel(Prob p, const int* skey, const int* sslot,
                                                                   const float* partials, float* acc) {
  extern __shared__ float4 acc_s[];                 // [kRowsPerBlock][kCols4]
  __shared__ int lo_s[kTokBatch], cnt_s[kTokBatch], off_s[kTokBatch + 1];
  __shared__ int m_slot[kMaxMatch], m_key[kMaxMatch], m_tok[kMaxMatch];
  const int j0 = blockIdx.x * kRowsPerBlock;
  const int tid = threadIdx.x;
  for (int i = tid; i < kRowsPerBlock * kCols4; i += kRedThreads) acc_s[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int tb = 0; tb < p.ntok; tb += kTokBatch) {
    const int nb = (p.ntok - tb) < kTokBatch ? (p.ntok - tb) : kTokBatch;
    __syncthreads();
    if (tid < nb) {
      const int* ks = skey + (size_t)(tb + tid) * p.Kpad;
      const int lo = lower_bound(ks, p.Kpad, j0);
      const int hi = lower_bound(ks, p.Kpad, j0 + kRowsPerBlock);
      lo_s[tid] = lo;
      cnt_s[tid] = hi - lo;
    }
    __syncthreads();
    if (tid == 0) {
      int o = 0;
      for (int i = 0; i < nb; ++i) {
        off_s[i] = o;
        o += cnt_s[i];
      }
      off_s[nb] = o;
    }
    __syncthreads();
    const int total = off_s[nb];
    for (int m0 = 0; m0 < total; m0 += kMaxMatch) {
      const int m1 = (total - m0) < kMaxMatch ? total : m0 + kMaxMatch;
      if (tid < nb) {
        const int a = off_s[tid], b = a + cnt_s[tid];
        const int e0 = a > m0 ? a : m0, e1 = b < m1 ? b : m1;
        const int* ks = skey + (size_t)(tb + tid) * p.Kpad;
        const int* ss = sslot + (size_t)(tb + tid) * p.Kpad;
        for (int e = e0; e < e1; ++e) {
          const int r = lo_s[tid] + (e - a);
          m_slot[e - m0] = __ldg(ss + r);
          m_key[e - m0] = __ldg(ks + r) - j0;
          m_tok[e - m0] = tb + tid;
        }
      }
      __syncthreads();
      if (tid < kCols4) {
        const int n = m1 - m0;
        int e = 0;
        for (; e + 8 <= n; e += 8) {
          float4 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            v[u] = __ldg(reinterpret_cast<const float4*>(partials + ((size_t)m_tok[e + u] * p.Kpad + m_slot[e + u]) * kAccRow) + tid);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            float4& a = acc_s[m_key[e + u] * kCols4 + tid];
            a.x += v[u].x; a.y += v[u].y; a.z += v[u].z; a.w += v[u].w;
          }
        }
        for (; e < n; ++e) {
          const float4 v = __ldg(reinterpret_cast<const float4*>(partials + ((size_t)m_tok[e] * p.Kpad + m_slot[e]) * kAccRow) + tid);
          float4& a = acc_s[m_key[e] * kCols4 + tid];
          a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
        }
      }
      __syncthreads();
    }
  }
  __syncthreads();
  for (int i = tid; i < kRowsPerBlock * kCols4; i += kRedThreads) {
    const int r = i / kCols4, c = i - r * kCols4;
    const int j = j0 + r;
    if (j >= p.T2) continue;
    float4* g = reinterpret_cast<float4*>(acc + (size_t)j * kAccRow) + c;
    float4 x = *g;
    const float4 a = acc_s[i];
    x.x += a.x; x.y += a.y; x.z += a.z; x.w += a.w;
    *g = x;
  }
}

}  // namespace

cudaError_t launch_sort_keys(const Prob& p, int* sorted_key, int* sorted_slot, cudaStream_t st) {
  if (p.ntok <= 0) return cudaSuccess;
  int n = 1;
  while (n < p.Kpad) n <<= 1;
  const int smem = n * 8;
  cudaError_t e = cudaFuncSetAttribute(sort_keys_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  sort_keys_kernel<<<p.ntok, 1024, smem, st>>>(p, n, sorted_key, sorted_slot);
  return cudaGetLastError();
}

cudaError_t launch_det_reduce(const Prob& p, const int* sorted_key, const int* sorted_slot, const float* partials,
                              float* acc, cudaStream_t st) {
  if (p.ntok <= 0 || p.T2 <= 0) return cudaSuccess;
  const int smem = kRowsPerBlock * kCols4 * 16;
  cudaError_t e = cudaFuncSetAttribute(det_reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  det_reduce_kernel<<<(p.T2 + kRowsPerBlock - 1) / kRowsPerBlock, kRedThreads, smem, st>>>(p, sorted_key, sorted_slot,
                                                                                         partials, acc);
  return cudaGetLastError();
}

}  // namespace sfa
