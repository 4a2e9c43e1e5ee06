// pa_decode_static.cu -- pa_decode_run_static: plan + decode + reduce with the
// workspace taken from a fixed array in device memory instead of from the caller.
//
// Who needs it: callers that cannot call cudaMalloc -- code running inside another
// runtime's memory budget (an inference server or plugin host that owns all device
// memory and refuses allocations from outside its own allocator), and latency-critical
// loops where cudaMalloc / cudaFree may synchronise the device.  They still pass their
// own inputs and output; only the scratch (plan, task list, partial results, status
// word) lives in the array below.
//
// The array is a file-scope __device__ object: every GPU that loads this library holds
// kStaticWorkspaceBytes of it until the process exits.  All calls on a device share it
// and it keeps the previous call's contents, so calls that overlap on the GPU (two
// streams, two threads) race on it and must be serialised by the caller.  Its device
// address is looked up once per device, by the first call made with that device
// current; a device reset (cudaDeviceReset) invalidates that address, so the library
// must not be used on a device after it has been reset.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pa_decode.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = PA_DECODE_STATIC_WORKSPACE_BYTES;

static __device__ __align__(256) unsigned char g_static_ws[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;

// Device address of g_static_ws on the current device, which must also be the device of
// `stream` (PA_ERR_INVALID_ARG otherwise: the kernels would run on one device with another
// device's array).  In host code the name g_static_ws is only a host-side stand-in, never
// a device address, so the address is looked up once per device with that device current.
pa_status static_ws_address(void* stream, void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {nullptr};
  int dev = 0, sdev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  if (cudaStreamGetDevice(reinterpret_cast<cudaStream_t>(stream), &sdev) != cudaSuccess)
    return PA_ERR_INVALID_ARG;
  if (sdev != dev) return PA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return PA_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_run_static(const pa_decode_args* args, void* stream) {
  pa_status st = pa_decode_validate(args);
  if (st != PA_OK) return st;
  const size_t need = pa_decode_workspace_size(args);
  if (need == 0) return PA_ERR_CUDA;
  if (need > kStaticWorkspaceBytes) return PA_ERR_WORKSPACE;  // beyond the fixed maximum
  void* ws = nullptr;
  if ((st = static_ws_address(stream, &ws)) != PA_OK) return st;
  // The status word and task count are the only fields read before the plan rewrites
  // them; clear them so a stale value from the previous call can never be seen.
  if (cudaMemsetAsync(ws, 0, 256, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  return pa_decode_run(args, ws, kStaticWorkspaceBytes, stream);
}

// The status word is the first int32 of the workspace (see pa_decode_read_status).
extern "C" pa_status pa_decode_read_status_static(int32_t* host_status, void* stream) {
  if (!host_status) return PA_ERR_INVALID_ARG;
  void* ws = nullptr;
  pa_status st = static_ws_address(stream, &ws);
  if (st != PA_OK) return st;
  return pa_decode_read_status(ws, host_status, stream);
}
