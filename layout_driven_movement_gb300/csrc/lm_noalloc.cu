// lm_layout_copy_host_static: the host-buffer copy of lm_layout_copy_host
// for callers that cannot allocate device memory.
//
// lm_layout_copy_host needs two device staging buffers from its caller.
// Some callers cannot provide them: a library embedded in a program whose
// memory manager has reserved the device's memory for itself (a cudaMalloc
// from outside it fails, or goes behind its accounting), or code on a path
// that cannot afford cudaMalloc/cudaFree (cudaFree waits for the whole
// device).  This variant stages through one fixed area instead: a
// file-scope __device__ array of LM_HOST_COPY_STATIC_BYTES, which every GPU
// that loads this library holds from the module's load until the process
// exits.  Nothing here calls cudaMalloc, cudaFree or any other allocating
// routine.

#include <cuda_runtime.h>

#include <mutex>

#include "lm_internal.h"

// The staging area: the source at offset 0, the destination at the next
// 256-byte boundary after the source's capacity.
static __device__ __align__(256) unsigned char
    g_lm_host_copy_staging[LM_HOST_COPY_STATIC_BYTES];

namespace {

constexpr int kMaxDevices = 64;

// Device address of the area on each device, looked up once per device with
// that device current.  In host code the array's name is only a host-side
// stand-in, so the address must come from cudaGetSymbolAddress.
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

int staging_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    lm::set_cuda_error(int(e));
    return LM_E_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return LM_E_INVALID;
  std::lock_guard<std::mutex> g(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_lm_host_copy_staging);
    if (e != cudaSuccess || !p) {
      lm::set_cuda_error(int(e));
      return LM_E_CUDA;
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return LM_OK;
}

}  // namespace

extern "C" int lm_layout_copy_host_static(const lm_plan* plan,
                                          const void* src_host,
                                          int64_t src_capacity_elems,
                                          void* dst_host,
                                          int64_t dst_capacity_elems,
                                          void* cuda_stream) {
  try {
    if (!plan) return LM_E_INVALID;
    if (plan->size == 0) return LM_OK;
    if (!src_host || !dst_host) return LM_E_INVALID;
    if (src_capacity_elems < 0 || dst_capacity_elems < 0) return LM_E_INVALID;
    const int64_t eb = plan->eb;
    const int64_t src_bytes = lm::mul_chk(src_capacity_elems, eb);
    const int64_t dst_bytes = lm::mul_chk(dst_capacity_elems, eb);
    const int64_t dst_at = lm::add_chk(src_bytes, 255) / 256 * 256;
    // the copy must fit the fixed area: source, padding, destination
    if (lm::add_chk(dst_at, dst_bytes) > int64_t(LM_HOST_COPY_STATIC_BYTES))
      return LM_E_CAPACITY;
    void* base = nullptr;
    const int rc = staging_address(&base);
    if (rc != LM_OK) return rc;
    char* area = static_cast<char*>(base);
    // the same upload, copy and download as lm_layout_copy_host, with the
    // fixed area as its staging buffers
    return lm_layout_copy_host(plan, src_host, src_capacity_elems, dst_host,
                               dst_capacity_elems, area, area + dst_at,
                               cuda_stream);
  } catch (const lm::Error& e) {
    return e.status;
  } catch (...) {
    return LM_E_INVALID;
  }
}
