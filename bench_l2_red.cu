// Ceiling of L2-resident fp32 reductions on this GPU: the bound of the
// key-side scatter (kvq.cu), which adds 1088-float key rows into an
// accumulator that stays in L2.  Warps add into random 128-byte pieces of a
// 4096 x 1088 fp32 array (17.8 MB) with one of four instruction shapes:
//   v4x4:  red.global.add.v4.f32, 4 rows x 128 B per warp instruction
//   v2x2:  red.global.add.v2.f32, 2 rows x 128 B per warp instruction
//   f32x1: red.global.add.f32,    1 row  x 128 B per warp instruction
//   v2x8:  red.global.add.v2.f32, 8 rows x 32 B per warp instruction
// and prints one JSON line with the best rate of each (bytes added / time,
// CUDA events, 152 CTAs of 8 or 16 warps, second of two runs).
// Build and run: python bench.py --l2-red-ceiling
#include <cstdio>
#include <cuda_runtime.h>

namespace {

constexpr int kRows = 4096, kCols = 1088, kSegs = kCols / 32;

__device__ __forceinline__ unsigned mix(unsigned x) {
  x ^= x >> 16;
  x *= 0x7feb352dU;
  x ^= x >> 15;
  x *= 0x846ca68bU;
  x ^= x >> 16;
  return x;
}

template <int MODE>
__global__ void red_kernel(float* acc, int iters) {
  const int lane = threadIdx.x & 31;
  const unsigned wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const float v = 1.0f + lane;
  for (int it = 0; it < iters; ++it) {
    const unsigned h = mix(wid * 7919u + it);
    const int s = (h >> 12) % kSegs;   // 128-byte piece of the row
    if (MODE == 0) {
      const int r = (h + (lane >> 3) * 977u) % kRows;
      float* d = acc + (size_t)r * kCols + s * 32 + (lane & 7) * 4;
      asm volatile("red.global.add.v4.f32 [%0], {%1,%1,%1,%1};" ::"l"(d), "f"(v) : "memory");
    } else if (MODE == 1) {
      const int r = (h + (lane >> 4) * 977u) % kRows;
      float* d = acc + (size_t)r * kCols + s * 32 + (lane & 15) * 2;
      asm volatile("red.global.add.v2.f32 [%0], {%1,%1};" ::"l"(d), "f"(v) : "memory");
    } else if (MODE == 2) {
      const int r = h % kRows;
      float* d = acc + (size_t)r * kCols + s * 32 + lane;
      asm volatile("red.global.add.f32 [%0], %1;" ::"l"(d), "f"(v) : "memory");
    } else {
      const int r = (h + (lane >> 2) * 977u) % kRows;
      float* d = acc + (size_t)r * kCols + s * 32 + (lane & 3) * 2;
      asm volatile("red.global.add.v2.f32 [%0], {%1,%1};" ::"l"(d), "f"(v) : "memory");
    }
  }
}

template <int MODE>
float run(float* acc, int grid, int warps, int iters, cudaEvent_t a, cudaEvent_t b) {
  float ms = 0.f;
  for (int rep = 0; rep < 2; ++rep) {
    cudaEventRecord(a);
    red_kernel<MODE><<<grid, warps * 32>>>(acc, iters);
    cudaEventRecord(b);
    cudaEventSynchronize(b);
    cudaEventElapsedTime(&ms, a, b);
  }
  return ms;
}

}  // namespace

int main() {
  float* acc = nullptr;
  if (cudaMalloc(&acc, (size_t)kRows * kCols * 4) != cudaSuccess) return 1;
  cudaMemset(acc, 0, (size_t)kRows * kCols * 4);
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  int nsm = 0;
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0);
  const char* names[4] = {"v4x4", "v2x2", "f32x1", "v2x8"};
  const int bytes[4] = {512, 256, 128, 256};
  double best[4] = {0, 0, 0, 0};
  for (int mode = 0; mode < 4; ++mode)
    for (int warps : {8, 16}) {
      const int iters = 2000000 / bytes[mode];
      float ms = mode == 0 ? run<0>(acc, nsm, warps, iters, a, b)
               : mode == 1 ? run<1>(acc, nsm, warps, iters, a, b)
               : mode == 2 ? run<2>(acc, nsm, warps, iters, a, b)
                           : run<3>(acc, nsm, warps, iters, a, b);
      const double gbs = (double)nsm * warps * iters * bytes[mode] / (ms * 1e-3) / 1e9;
      if (gbs > best[mode]) best[mode] = gbs;
    }
  const cudaError_t e = cudaDeviceSynchronize();
  printf("{\"sms\": %d", nsm);
  for (int m = 0; m < 4; ++m) printf(", \"%s_gbs\": %.0f", names[m], best[m]);
  printf(", \"status\": \"%s\"}\n", cudaGetErrorString(e));
  cudaFree(acc);
  return e == cudaSuccess ? 0 : 1;
}
