// csa_index_topk_static: block indexing and Top-K with no workspace from the caller.
//
// csa_index_topk needs scratch device memory for the block scores it ranks, and takes it from the
// caller. Some callers have no way to provide it at the point where they select blocks: code that runs
// under a host framework whose allocator already owns the device memory and forbids raw cudaMalloc,
// plug-ins that may only use buffers they were handed, or real-time serving loops that must not
// allocate (and so must not risk an allocator stall) once they are running. For them this entry point
// takes its scratch from an array that the library itself places in device memory when it is loaded.
// The caller still passes every input and output buffer.
//
// The array is fixed in size (CSA_STATIC_INDEX_SCRATCH_BYTES) and is held by every GPU that loads the
// library until the process exits. Its device address is looked up per device, by the first call that
// succeeds while that device is current; host code must not pass the array's own name to a kernel, since
// on the host that name is only a stand-in for the device copy.
#include <cstdio>
#include <mutex>

#include "csa_internal.cuh"

namespace {

static __device__ __align__(256) uint8_t g_index_scratch[CSA_STATIC_INDEX_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// The array's device address per device, looked up by the first call that succeeds with that device
// current. A failed lookup (for example inside a stream capture that forbids it) is not remembered: the
// next call tries again.
std::mutex g_addr_mu;
void* g_addr[kMaxDevices] = {};

}  // namespace

extern "C" csa_status csa_index_topk_static(int64_t batch, const csa_index_args* args, int32_t* status_out,
                                            cudaStream_t stream) {
  // the arguments first, then the size of the call's scratch against the array, then the device
  const csa_status valid = csa::validate_index_args(batch, args);
  if (valid != CSA_OK) return valid;
  const size_t need = csa_index_topk_workspace_size(batch, args);
  if (need > (size_t)CSA_STATIC_INDEX_SCRATCH_BYTES) {
    csa::set_last_error("csa_index_topk_static: this call needs %zu bytes of scratch, more than the %zu bytes "
                        "of the library's static array; use csa_index_topk with a workspace",
                        need, (size_t)CSA_STATIC_INDEX_SCRATCH_BYTES);
    return CSA_ERR_WORKSPACE_TOO_SMALL;
  }
  if (status_out != nullptr && (reinterpret_cast<uintptr_t>(status_out) % 4) != 0) return CSA_ERR_ALIGNMENT;
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return csa::cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return CSA_ERR_UNSUPPORTED_DEVICE;
  void* ptr = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_addr_mu);
    if (g_addr[dev] == nullptr) {
      void* found = nullptr;
      if (cudaError_t e = cudaGetSymbolAddress(&found, g_index_scratch)) {
        (void)cudaGetLastError();
        return csa::cuda_fail(e, "cudaGetSymbolAddress of the static index scratch");
      }
      g_addr[dev] = found;
    }
    ptr = g_addr[dev];
  }

  // The array keeps whatever the previous call left in it; only the status word must start at zero
  // (every score slot the kernels read is written by the same call first).
  if (cudaError_t e = cudaMemsetAsync(ptr, 0, CSA_WS_HEADER_BYTES, stream))
    return csa::cuda_fail(e, "static scratch status reset");
  const csa_status st = csa_index_topk(batch, args, ptr, (size_t)CSA_STATIC_INDEX_SCRATCH_BYTES, stream);
  if (st != CSA_OK) return st;
  if (status_out != nullptr) {
    if (cudaError_t e = cudaMemcpyAsync(status_out, ptr, sizeof(int32_t), cudaMemcpyDeviceToDevice, stream))
      return csa::cuda_fail(e, "static scratch status copy");
  }
  return CSA_OK;
}
