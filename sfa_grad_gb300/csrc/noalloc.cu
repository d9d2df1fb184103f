// sfa_grad_noalloc: the backward for callers that cannot allocate device
// memory.  Some callers cannot call cudaMalloc: a plugin whose host
// framework owns every byte of the device through its own pool, code that runs
// while a stream is being captured into a CUDA graph, or a latency-critical
// path that must not risk the implicit device-wide synchronisation that
// cudaMalloc / cudaFree can cause.  This entry point takes the workspace from
// a fixed array compiled into the library instead of from the caller.
//
// The scratch is a file-scope __device__ array of kScratchBytes.  Every GPU
// that loads the library holds it until the process exits.  In host code the
// array's name is only a host-side stand-in, so the device address is looked
// up once per device (with that device current) by cudaGetSymbolAddress and
// passed to the kernels like any workspace.  The first call on a device does
// that lookup; make that first call before starting any stream capture.  The
// cached address belongs to the device's context: the library must not be
// used across cudaDeviceReset.  The kernels' device error word (a pipeline
// wait that gave up, invalid TND lengths) lives in the scratch too;
// sfa_noalloc_read_device_error reads and clears it.
//
// All calls share the one array and it keeps the previous call's contents:
// the backward clears everything it needs to start at zero (the fp32
// key-side accumulator and the error word) and overwrites the rest before
// reading it.  Calls whose work overlaps on the GPU (other streams, other
// threads) race on the array and must be serialised by the caller.
#include <cstdio>
#include <mutex>

#include "sfa_grad.h"
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = SFA_NOALLOC_SCRATCH_BYTES;   // 64 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};


// The static scratch's device address on the current device, looked up once
// per device (with that device current) and cached.  The cache assumes the
// device's primary context lives as long as the process: after
// cudaDeviceReset the module is loaded again and the cached address would be
// stale, so the library must not be used across a device reset.
sfa_status scratch_address(void** out) {
  int dev = 0;
  const cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    char msg[160];
    if (ge != cudaSuccess)
      snprintf(msg, sizeof(msg), "sfa_grad_noalloc: cudaGetDevice failed: %s", cudaGetErrorString(ge));
    else
      snprintf(msg, sizeof(msg), "sfa_grad_noalloc: device index %d is outside 0..%d", dev, kMaxDevices - 1);
    sfa::set_last_error(msg);
    return SFA_ERR_RUNTIME;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* a = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&a, g_scratch);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      char msg[160];
      snprintf(msg, sizeof(msg), "sfa_grad_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
      sfa::set_last_error(msg);
      return SFA_ERR_RUNTIME;
    }
    g_scratch_ptr[dev] = a;
  }
  *out = g_scratch_ptr[dev];
  return SFA_OK;
}

}  // namespace

extern "C" {

sfa_status sfa_grad_noalloc(const sfa_params* p, const void* q, const void* k, const void* v, const int32_t* indices,
                            const void* d_out, const void* out, const float* softmax_max, const float* softmax_sum,
                            const int32_t* act_seq_q, const int32_t* act_seq_kv, const void* q_rope,
                            const void* k_rope, void* dq, void* dk, void* dv, void* dq_rope, void* dk_rope,
                            void* stream) {
  if (!p) return SFA_ERR_NULLPTR;
  size_t need = 0;
  const sfa_status s = sfa_grad_workspace_size(p, &need);
  if (s != SFA_OK) return s;
  if (need > kScratchBytes) {
    char msg[160];
    snprintf(msg, sizeof(msg), "sfa_grad_noalloc: problem needs %zu bytes of workspace, the static scratch holds %zu",
             need, kScratchBytes);
    sfa::set_last_error(msg);
    return SFA_ERR_SHAPE;
  }
  void* ptr = nullptr;
  const sfa_status a = scratch_address(&ptr);
  if (a != SFA_OK) return a;
  return sfa_grad(p, q, k, v, indices, d_out, out, softmax_max, softmax_sum, act_seq_q, act_seq_kv, q_rope, k_rope, dq,
                  dk, dv, dq_rope, dk_rope, ptr, kScratchBytes, stream);
}

sfa_status sfa_noalloc_read_device_error(void* stream, int32_t* code) {
  if (!code) return SFA_ERR_NULLPTR;
  void* ptr = nullptr;
  const sfa_status a = scratch_address(&ptr);
  if (a != SFA_OK) return a;
  // the error word sits at the start of the workspace, as in sfa_grad's
  return sfa_read_device_error(ptr, stream, code);
}

}  // extern "C"
