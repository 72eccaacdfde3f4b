// Allocation-free entry point.
//
// Some callers cannot allocate device memory at the moment they need the gradient
// accumulated: code running under a custom or fixed-pool allocator that must not grow,
// and runtimes that forbid cudaMalloc after start-up.  For them this file owns a fixed
// block of device memory, a file-scope __device__ array, and uses it as the workspace of
// ewg_accumulate.  The block is reserved on every device that loads the library and kept
// until the process exits (under CUDA's default lazy module loading, from the first
// call on the device, whose address lookup loads this module).  Calls are limited to
// sizes whose workspace fits in it.  The first call on a device looks up the block's
// device address (make it at start-up, outside any stream capture); calls that overlap
// on the GPU race on the block.
#include <mutex>

#include "ewg.h"
#include "ewg_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = EWG_STATIC_SCRATCH_BYTES;

// Device storage of the workspace.  In host code this name is only a stand-in for the
// device symbol: its device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

extern "C" int ewg_accumulate_static(const void* ids, int ids_dtype, int64_t num_tokens,
                                     const void* grad, int grad_dtype, int64_t grad_row_stride,
                                     void* main_grad, int main_grad_dtype, int64_t num_embeddings,
                                     int64_t hidden, int64_t main_grad_row_stride, void* stream,
                                     void** scratch_out) {
  const size_t need = ewg_workspace_bytes(num_tokens, hidden);
  if (need == 0 || need > kStaticScratchBytes) {
    ewg::set_last_error(
        "ewg_accumulate_static: the workspace for these sizes exceeds the static scratch "
        "(EWG_STATIC_SCRATCH_BYTES); use ewg_accumulate with a caller workspace");
    return EWG_ERR_UNSUPPORTED;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    ewg::set_last_error("ewg_accumulate_static: no usable current device");
    return EWG_ERR_CUDA;
  }
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {   // first call on this device
      e = cudaGetSymbolAddress(&g_scratch_addr[dev], g_scratch);
      if (e != cudaSuccess) {
        g_scratch_addr[dev] = nullptr;
        ewg::set_last_error("ewg_accumulate_static: cudaGetSymbolAddress failed");
        return EWG_ERR_CUDA;
      }
    }
    ws = g_scratch_addr[dev];
  }
  if (scratch_out) *scratch_out = ws;
  // The plan writes every workspace word it later reads (status, counters included),
  // so nothing left by an earlier call needs clearing.
  return ewg_accumulate(ids, ids_dtype, num_tokens, grad, grad_dtype, grad_row_stride, main_grad,
                        main_grad_dtype, num_embeddings, hidden, main_grad_row_stride, ws,
                        kStaticScratchBytes, stream);
}
