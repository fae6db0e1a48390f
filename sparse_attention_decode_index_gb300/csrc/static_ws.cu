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
// the life of the process.
//
// Host code may not use the array's name as a device address (in host code it
// is only a stand-in symbol), so the device address is looked up with
// cudaGetSymbolAddress once per device, with that device current, on the
// first call made while it is the current device; that first call also
// zeroes the array's header (the sticky device error word).
#include <cstdint>

#include "../../include/csa2.h"
#include "internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(32) << 20;   // 32 MiB

__device__ __align__(256) unsigned char g_static_ws[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
void* g_static_ptr[kMaxDevices];

// Device address of g_static_ws on the current device (set up on first use).
int static_workspace(void** out, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CSA2_ERR_CUDA;
  if (g_static_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || p == nullptr) return CSA2_ERR_CUDA;
    // the header holds the sticky device error word, which must start at zero
    if (cudaMemsetAsync(p, 0, 256, stream) != cudaSuccess) return CSA2_ERR_CUDA;
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return CSA2_OK;
}

}  // namespace

extern "C" {

int csa2_layer_group_static(const csa2_shape* shape, const csa2_layer* layers, int32_t n_layers,
                            const void* k_main, const void* v_main, const void* k_idx, const void* kb,
                            const int32_t* n_valid, const int32_t* n_swa, csa2_stream_t stream) {
  const size_t need = csa2_workspace_bytes(shape);
  if (need == 0) return CSA2_ERR_INVALID_ARG;
  if (need > kStaticWorkspaceBytes) return CSA2_ERR_WORKSPACE;
  void* ws = nullptr;
  const int st = static_workspace(&ws, stream);
  if (st != CSA2_OK) return st;
  return csa2_layer_group(shape, layers, n_layers, k_main, v_main, k_idx, kb, n_valid, n_swa, ws,
                          kStaticWorkspaceBytes, stream);
}

}  // extern "C"
