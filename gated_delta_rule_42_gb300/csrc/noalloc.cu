// kda_chunk_fwd_noalloc: the chunked forward for callers that cannot allocate
// device memory.
//
// Some callers have no way to hand the library a workspace: a host program
// linked against libkda alone, with no allocator of its own; a runtime that
// plans every device byte at start-up and forbids allocation afterwards; code
// running on a worker that may not call cudaMalloc because it would
// synchronise the device or fragment a pre-partitioned memory budget.  For
// them this entry point runs kda_chunk_fwd on a scratch buffer that lives in
// the library itself: a file-scope device array of kNoAllocScratchBytes
// (4 MiB), held by every GPU that loads the library until the process exits.
//
// Usage rules:
//  * The first call on each device looks the array's device address up
//    (cudaGetSymbolAddress, with that device current) and caches it for the
//    life of the process; make that first call before any CUDA-graph capture
//    on the device.  A device reset (cudaDeviceReset, or a reset of the
//    primary context) after that first call is not supported: the module is
//    reloaded and the cached address would no longer be the array's.
//  * Every call shares the one array.  Calls whose work may overlap on the GPU
//    (different streams, or different host threads, without ordering between
//    them) race on it; order them on one stream.
//  * Nothing in the array has to start at zero: every byte the forward reads
//    is written earlier in the same call.  The array keeps the last call's
//    contents.
//  * Problems whose workspace exceeds the array are rejected before anything
//    is launched (KDA_ERR_WORKSPACE, with the sizes in kda_last_error()).
#include <stdio.h>

#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

}  // namespace

extern "C" {

kda_status kda_chunk_fwd_noalloc(const kda_inputs *in, void *o, float *hT, void *stream) {
  char msg[256];
  const size_t need = kda_chunk_fwd_workspace_size(in);
  if (need == 0)  // invalid problem: let the regular entry point report why (nothing is launched)
    return kda_chunk_fwd(in, o, hT, nullptr, 0, stream);
  if (need > kNoAllocScratchBytes) {
    snprintf(msg, sizeof(msg), "kda_chunk_fwd_noalloc: problem needs %zu bytes of scratch; the static scratch holds %zu",
             need, kNoAllocScratchBytes);
    kda::set_last_error(msg);
    return KDA_ERR_WORKSPACE;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    snprintf(msg, sizeof(msg), "kda_chunk_fwd_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    kda::set_last_error(msg);
    return KDA_ERR_CUDA;
  }
  void *scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_addr[dev] == nullptr) {
      void *p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr) {
        snprintf(msg, sizeof(msg), "kda_chunk_fwd_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        kda::set_last_error(msg);
        return KDA_ERR_CUDA;
      }
      g_addr[dev] = p;
    }
    scratch = g_addr[dev];
  }
  return kda_chunk_fwd(in, o, hT, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
