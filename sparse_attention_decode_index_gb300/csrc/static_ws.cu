// csa2_layer_group_static: the layer-group entry point for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain a device workspace: a plugin living inside
// a host framework that owns every device allocation and hands out only the
// tensors it manages, or a latency-critical decode loop that must not call
// cudaMalloc (which can implicitly synchronise the device).  For them this
// entry point runs the same layer group as csa2_layer_group, but on scratch
// memory that the library itself holds: a file-scope __device__ array of
// kStaticWorkspaceBytes, which every GPU that loads this library keeps for
// the life of the process.  A __device__ array starts zeroed when the module
// is loaded, so its header (the sticky device error word) needs no clearing.
//
// Host code may not use the array's name as a device address (in host code it
// is only a stand-in symbol), so the device address is looked up with
// cudaGetSymbolAddress once per device, with that device current, on the
// first call made while it is the current device.  The lookup runs under a
// per-device std::call_once, so host threads making their first calls at the
// same time do not race on it.
#include <cstdint>
#include <mutex>

#include "../../include/csa2.h"
#include "internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(32) << 20;   // 32 MiB

__device__ __align__(256) unsigned char g_static_ws[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;

struct DeviceSlot {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
DeviceSlot g_slots[kMaxDevices];

}  // namespace

namespace csa2 {

int static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CSA2_ERR_CUDA;
  DeviceSlot& s = g_slots[dev];
  std::call_once(s.once, [&s] { s.err = cudaGetSymbolAddress(&s.ptr, g_static_ws); });
  if (s.err != cudaSuccess || s.ptr == nullptr) return CSA2_ERR_CUDA;
  *out = s.ptr;
  return CSA2_OK;
}

}  // namespace csa2

extern "C" {

int csa2_layer_group_static(const csa2_shape* shape, const csa2_layer* layers, int32_t n_layers,
                            const void* k_main, const void* v_main, const void* k_idx, const void* kb,
                            const int32_t* n_valid, const int32_t* n_swa, csa2_stream_t stream) {
  const size_t need = csa2_workspace_bytes(shape);
  if (need == 0) return CSA2_ERR_INVALID_ARG;
  if (need > kStaticWorkspaceBytes) return CSA2_ERR_WORKSPACE;
  void* ws = nullptr;
  const int st = csa2::static_scratch(&ws);
  if (st != CSA2_OK) return st;
  return csa2_layer_group(shape, layers, n_layers, k_main, v_main, k_idx, kb, n_valid, n_swa, ws,
                          kStaticWorkspaceBytes, stream);
}

int csa2_read_static_device_error(csa2_stream_t stream, int32_t* detail) {
  void* ws = nullptr;
  const int st = csa2::static_scratch(&ws);
  if (st != CSA2_OK) return st;
  return csa2_read_device_error(ws, stream, detail);
}

}  // extern "C"
