// mha_noalloc.cu - split-KV attention forward for callers that cannot
// allocate device memory.
//
// mha_fwd_kv needs a workspace for the per-split partial results, and it
// expects the caller to provide it.  Some callers have no way to obtain one:
// a plug-in handed only the raw pointers of tensors another runtime owns, a
// service that reserves all device memory at start-up and forbids
// allocation while serving requests, or a host program without access to
// the allocator that produced its buffers.  This entry point serves them
// with a fixed scratch buffer that lives in the library's own module memory:
// the caller passes inputs and outputs only.
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "mha_fwd.h"
#include "mha_internal.h"

namespace {

// The scratch buffer: 16 MiB of module memory, held by every GPU that loads
// the library until the process exits.  The host-side name is only a
// stand-in; the device address comes from cudaGetSymbolAddress below.
constexpr size_t kScratchBytes = static_cast<size_t>(16) << 20;
static __device__ __align__(256) unsigned char g_kv_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch buffer on the current device, looked up
// once per device (with that device current) and cached.  The library's
// device check runs first, so a GPU the kernels cannot run on is reported
// as MHA_ERR_NO_DEVICE, as mha_fwd_kv reports it, before any lookup.
int scratch_address(void** out) {
  int dev = 0;
  unsigned* status = nullptr;
  const int rc = mha_host::device_setup(&dev, &status);
  if (rc != MHA_OK) return rc;
  if (dev >= kMaxDevices) return MHA_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kv_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();  // leave no pending error behind for the caller
      return MHA_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MHA_OK;
}

}  // namespace

extern "C" int mha_fwd_kv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                  int B, int H, int Nq, int Nk, int d, float scale, int causal,
                                  int num_splits, void* stream) {
  const size_t need = mha_fwd_kv_workspace_size(B, H, Nq, Nk, d, num_splits);
  if (need > kScratchBytes) return MHA_ERR_SCRATCH_LIMIT;
  if (need == 0)  // empty problem or invalid arguments: reported without any CUDA call
    return mha_fwd_kv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, num_splits, nullptr, 0, stream);
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != MHA_OK) return rc;
  // Every element of the scratch that the merge step reads is written by the
  // partial step of the same call (when every device-side wait completes),
  // and the work-tile counter is zeroed by the call's first kernel, so
  // nothing needs clearing between calls.
  return mha_fwd_kv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, num_splits, scratch,
                    kScratchBytes, stream);
}
