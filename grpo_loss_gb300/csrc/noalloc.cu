// grpo_loss_fwd_noalloc: the forward pass for callers that cannot allocate
// device memory.
//
// Some callers have no way to hand the library a workspace: a plain C host
// without a caching allocator (where cudaMalloc would synchronise the device
// and stall every other stream), code running under a fixed memory budget
// that forbids new allocations once training has started, or code that runs
// where allocation is not allowed at all. This entry point takes only the
// inputs and outputs and keeps its scratch in a statically sized device array
// that lives for as long as the library is loaded.
#include <mutex>

#include "../../include/grpo.h"
#include "internal.h"

namespace {

// Scratch shared by every call on a device. Every GPU that loads the library
// holds these bytes until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GRPO_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
// Device address of the array, per device ordinal, looked up once. It
// belongs to the context that was current then: after cudaDeviceReset (or
// any teardown of the primary context) the module is loaded again and the
// array may live elsewhere, so the entry point must not be used across a
// reset.
void* g_scratch_dev[64] = {nullptr};

// After the forward has run: if a device-side check failed (a valid token
// with an id outside [0, V), or an expired pipeline wait), mark the loss and
// the KL mean NaN. This caller has no workspace through which to read the
// error word.
__global__ void k_mark_loss_on_error(const uint32_t* err, float* loss, float* kl_mean) {
  if (threadIdx.x == 0 && *err != 0u) {
    *loss = __int_as_float(0x7fc00000);
    if (kl_mean) *kl_mean = __int_as_float(0x7fc00000);
  }
}

// First call on a device: look up the array's device address with that
// device current. Host code may not use the array's name as an address: in
// host code it names a host-side stand-in, not device memory.
grpo_status scratch_for_current_device(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GRPO_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GRPO_ERR_CUDA;
    g_scratch_dev[dev] = p;
  }
  *ptr = g_scratch_dev[dev];
  return GRPO_OK;
}

}  // namespace

extern "C" grpo_status grpo_loss_fwd_noalloc(const grpo_problem* problem, const void* H_pol,
                                             const void* H_ref, const void* W,
                                             const int32_t* ids, const uint8_t* mask,
                                             const float* adv, float* logp_pol, float* logp_ref,
                                             float* lse_pol, float* loss, float* kl_mean,
                                             cudaStream_t stream) {
  if (!problem || !loss) return GRPO_ERR_INVALID_ARG;
  size_t need = 0;
  grpo_status st = grpo_workspace_size(problem, &need, nullptr);
  if (st != GRPO_OK) return st;
  if (need > GRPO_NOALLOC_SCRATCH_BYTES) return GRPO_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((st = scratch_for_current_device(&scratch)) != GRPO_OK) return st;
  // The regular forward clears the scratch's control word (error bits and
  // block count) itself; every other scratch region is written before it is
  // read, so stale contents from an earlier call do not matter.
  st = grpo_loss_fwd(problem, H_pol, H_ref, W, ids, mask, adv, logp_pol, logp_ref, lse_pol,
                     loss, kl_mean, scratch, GRPO_NOALLOC_SCRATCH_BYTES, stream);
  if (st != GRPO_OK) return st;
  k_mark_loss_on_error<<<1, 32, 0, stream>>>(static_cast<const uint32_t*>(scratch), loss,
                                              kl_mean);
  return cudaGetLastError() == cudaSuccess ? GRPO_OK : GRPO_ERR_CUDA;
}
