// Small bandwidth-bound kernels around the tensor-core stages:
//  * per-token metadata: KV segment start and the last attendable key
//    (sparseMode 0: kvlen - 1; sparseMode 3, rightDownCausal: kvlen - qlen + i),
//    with TND lengths prefix-summed and validated on the device;
//  * Dsum = rowsum(dO * O) over the 512 value features (FlashSoftmaxGrad);
//  * the fp32 key-side accumulator cast to the output dtype;
//  * the forward's per-tile (max, sum) partials combined into softmaxMax/Sum.
//
// aclnnSparseFlashAttentionGrad doc: 参数说明 (actualSeqLengths rows), Mask
// table (sparseMode 3), 阶段2 (FlashSoftmaxGrad); MindSpore
// flash_attention_bwd.py, compute_Di.
#include "common.cuh"
#include "kernels.h"

namespace sfa {

namespace {

// One thread: prefix sums of the per-batch lengths, validated against T1/T2.
// batch_ofs = [q starts (B+1) | kv starts (B+1)].
__global__ void batch_prefix_kernel(const int* act_q, const int* act_kv, int B, int T1, int T2, int* batch_ofs,
                                    int* gerr) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  long long sq = 0, sk = 0;
  bool bad = false;
  batch_ofs[0] = 0;
  batch_ofs[B + 1] = 0;
  for (int b = 0; b < B; ++b) {
    const int lq = act_q[b], lk = act_kv[b];
    if (lq < 0 || lk < 0) bad = true;
    sq += lq;
    sk += lk;
    batch_ofs[b + 1] = (int)(sq > 0x7fffffff ? 0x7fffffff : sq);
    batch_ofs[B + 2 + b] = (int)(sk > 0x7fffffff ? 0x7fffffff : sk);
  }
  if (sq != T1 || sk != T2) bad = true;
  if (bad) {
    atomicExch(gerr, kErrSeqLens);
    batch_ofs[B] = -1;  // marks the call invalid for the meta kernel
  }
}

__global__ void meta_kernel(int layout, int T1, int B, int S1, int S2, int mode, const int* batch_ofs,
                            const int* act_q, const int* act_kv, TokMeta* meta) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T1) return;
  int kv_start, qlen, kvlen, i;
  if (layout == 0) {
    const int b = t / S1;
    i = t - b * S1;
    kv_start = b * S2;
    qlen = S1;
    kvlen = S2;
  } else {
    if (batch_ofs[B] < 0) {  // invalid lengths: every key masked
      meta[t] = TokMeta{0, -1};
      return;
    }
    int lo = 0, hi = B - 1;  // last b with q_start[b] <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (batch_ofs[mid] <= t) lo = mid;
      else hi = mid - 1;
    }
    // skip empty batches that share the start offset
    int b = lo;
    while (b < B - 1 && batch_ofs[b + 1] <= t) ++b;
    i = t - batch_ofs[b];
    kv_start = batch_ofs[B + 1 + b];
    qlen = act_q[b];
    kvlen = act_kv[b];
  }
  long long lim = (long long)kvlen - 1;
  if (mode == 3) {
    const long long c = (long long)kvlen - qlen + i;
    if (c < lim) lim = c;
  }
  if (lim < -1) lim = -1;
  meta[t] = TokMeta{kv_start, (int)lim};
}

// Row table of a token chunk: the kv row each (token, slot) reads, -1 if the
// slot is masked (功能说明 gather with block expansion; Mask table).
__global__ void rowtab_kernel(Prob p) {
  const long long n = (long long)p.ntok * p.Kpad;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int tl = (int)(i / p.Kpad), s = (int)(i - (long long)tl * p.Kpad);
    const int t = p.tok0 + tl;
    p.rowtab[i] = slot_row(p, p.meta[t], t, s);
  }
}

// One warp per (token, head) row of 512 elements.
template <typename T>
__global__ void dsum_kernel(const T* dO, const T* out, int rows, float* dsum) {
  using E = Elt<T>;
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= rows) return;
  const uint4* a = reinterpret_cast<const uint4*>(dO + (size_t)w * 512);
  const uint4* b = reinterpret_cast<const uint4*>(out + (size_t)w * 512);
  float acc = 0.f;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const uint4 x = __ldg(a + lane + 32 * u), y = __ldg(b + lane + 32 * u);
    const T* xs = reinterpret_cast<const T*>(&x);
    const T* ys = reinterpret_cast<const T*>(&y);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc = fmaf(E::to_f(xs[j]), E::to_f(ys[j]), acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) dsum[w] = acc;
}

// acc row (1088 fp32) = [dK 512 | dKRope 64 | dV 512]; one thread per 4 floats.
template <typename T>
__global__ void cast_kernel(const float* acc, long long n4, T* dk, T* dkr, T* dv, int has_rope) {
  using E = Elt<T>;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / 272;
    const int c = (int)(i - row * 272) * 4;
    const float4 x = __ldg(reinterpret_cast<const float4*>(acc) + i);
    uint2 o;
    o.x = E::pack(x.x, x.y);
    o.y = E::pack(x.z, x.w);
    T* dst;
    if (c < 512) dst = dk + row * 512 + c;
    else if (c < 576) {
      if (!has_rope) continue;
      dst = dkr + row * 64 + (c - 512);
    } else dst = dv + row * 512 + (c - 576);
    *reinterpret_cast<uint2*>(dst) = o;
  }
}

// Per (token, head): combine the partial (max of raw score, sum of exp) pairs
// in one pass, rescaling the running sum whenever the running max grows.
__global__ void stats_combine_kernel(const float* ts, int ntok, int ntiles, int G, int tok0, float scale, float* smax,
                                     float* ssum) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= ntok * G) return;
  const int tl = i / G, h = i - tl * G;
  const float sl2 = scale * 1.4426950408889634f;
  const float2* e = reinterpret_cast<const float2*>(ts) + (size_t)tl * ntiles * G + h;
  float mx = -INFINITY, l = 0.f;
  for (int kt = 0; kt < ntiles; ++kt) {
    const float2 pr = e[(size_t)kt * G];
    if (pr.x == -INFINITY) continue;   // no valid key in the partial
    if (pr.x > mx) {
      l = l * exp2f((mx - pr.x) * sl2) + pr.y;
      mx = pr.x;
    } else {
      l += pr.y * exp2f((pr.x - mx) * sl2);
    }
  }
  const size_t o = (size_t)(tok0 + tl) * G + h;
  smax[o] = mx == -INFINITY ? -INFINITY : mx * scale;
  ssum[o] = l;
}

}  // namespace

cudaError_t launch_batch_prefix(const Prob& p, int B, const int* act_q, const int* act_kv, int* batch_ofs, int* gerr,
                                cudaStream_t st) {
  batch_prefix_kernel<<<1, 1, 0, st>>>(act_q, act_kv, B, p.T1, p.T2, batch_ofs, gerr);
  return cudaGetLastError();
}

cudaError_t launch_meta(const Prob& p, int layout, int B, int S1, int S2, int mode, const int* act_q, const int* act_kv,
                        int* batch_ofs, TokMeta* meta, int* gerr, cudaStream_t st) {
  (void)gerr;
  if (p.T1 > 0) meta_kernel<<<(p.T1 + 255) / 256, 256, 0, st>>>(layout, p.T1, B, S1, S2, mode, batch_ofs, act_q, act_kv, meta);
  return cudaGetLastError();
}

cudaError_t launch_rowtab(const Prob& p, cudaStream_t st) {
  const long long n = (long long)p.ntok * p.Kpad;
  if (n == 0) return cudaSuccess;
  long long blocks = (n + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  rowtab_kernel<<<(int)blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dsum(const Prob& p, int tok0, int ntok, float* dsum, cudaStream_t st) {
  const int rows = ntok * p.G;
  if (rows == 0) return cudaSuccess;
  const size_t r0 = (size_t)tok0 * p.G;
  dsum_kernel<T><<<(rows + 7) / 8, 256, 0, st>>>(static_cast<const T*>(p.dO) + r0 * 512,
                                                 static_cast<const T*>(p.out) + r0 * 512, rows, dsum + r0);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_cast(const float* acc, int T2, void* dk, void* dkr, void* dv, int has_rope, cudaStream_t st) {
  const long long n4 = (long long)T2 * 272;
  if (n4 == 0) return cudaSuccess;
  long long blocks = (n4 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  cast_kernel<T><<<(int)blocks, 256, 0, st>>>(acc, n4, static_cast<T*>(dk), static_cast<T*>(dkr), static_cast<T*>(dv),
                                              has_rope);
  return cudaGetLastError();
}

cudaError_t launch_stats_combine(const Prob& p, const float* tile_stats, int ntiles, float* smax, float* ssum,
                                 cudaStream_t st) {
  const int n = p.ntok * p.G;
  if (n == 0) return cudaSuccess;
  stats_combine_kernel<<<(n + 255) / 256, 256, 0, st>>>(tile_stats, p.ntok, ntiles, p.G, p.tok0, p.scale, smax, ssum);
  return cudaGetLastError();
}

template cudaError_t launch_dsum<__nv_bfloat16>(const Prob&, int, int, float*, cudaStream_t);
template cudaError_t launch_dsum<__half>(const Prob&, int, int, float*, cudaStream_t);
template cudaError_t launch_cast<__nv_bfloat16>(const float*, int, void*, void*, void*, int, cudaStream_t);
template cudaError_t launch_cast<__half>(const float*, int, void*, void*, void*, int, cudaStream_t);

}  // namespace sfa
