// Router + top-(T/K) selection for callers that cannot allocate device memory.
//
// Some callers have no way to obtain scratch memory: a plugin inside another
// runtime that is handed only its input and output buffers, a serving loop that
// must not allocate once it is running (an allocation can synchronise the device
// and stall every stream), or a process whose device memory is already held by
// another framework's caching allocator, so that cudaMalloc fails although the
// pool has room. This variant keeps its scratch -- the fp32 router logits and a
// device status word -- in a fixed array that is part of the library image, and
// calls no cudaMalloc, cudaFree or allocating library routine.
//
// The array is shared by every call in the process on a given device and keeps
// the last call's contents; the status word is cleared at the start of each call
// and the logits are fully rewritten, so nothing stale is read. Calls that
// overlap on the GPU (different streams, no ordering between them) race on the
// array. Every call that is not being captured into a CUDA graph looks up the
// array's device address afresh (a host-side query, with the call's device current)
// and remembers it per device; a call made during stream capture uses the remembered
// address, so make one call on the device before any capture -- and again after a
// device reset, which reloads the library's device image at a new address.

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "xmod.h"

namespace xmod {
namespace {

constexpr size_t kStatusBytes = 256;
constexpr size_t kScratchBytes = kStatusBytes + sizeof(float) * (size_t)XMOD_NOALLOC_MAX_TOKENS;

// Device-resident scratch: status word, then logits[XMOD_NOALLOC_MAX_TOKENS].
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device. In host code the
// array's name is only a host-side stand-in, so the address must come from the
// runtime. Outside stream capture it is looked up on every call (so a device reset,
// which moves the array, is picked up by the next call); during capture, where the
// lookup could load the module, the address remembered by the last uncaptured call on
// this device is used, and a device never called outside capture is an error.
void* scratch_on_current_device(cudaStream_t s, int* err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = XMOD_ERR_CUDA;
    return nullptr;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
    *err = XMOD_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      *err = XMOD_ERR_CUDA;
      return nullptr;
    }
    g_addr[dev] = p;
  }
  if (!g_addr[dev]) *err = XMOD_ERR_INVALID_ARG;   // first call on this device is captured
  return g_addr[dev];
}

inline bool al16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }
inline bool al16n(const void* p) { return !p || ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace xmod

using namespace xmod;

extern "C" int xmod_router_topk_noalloc(const xmod_dims* dm, int K, const void* x,
                                        const void* w_r, const float* bias, int32_t* idx,
                                        float* r_sel, int* status_out, void* stream) {
  if (!dm || (dm->dtype != XMOD_BF16 && dm->dtype != XMOD_FP32)) return XMOD_ERR_INVALID_ARG;
  if (dm->B <= 0 || dm->T <= 0 || dm->d <= 0 || dm->d % 8) return XMOD_ERR_INVALID_ARG;
  if (K <= 0 || K > dm->T) return XMOD_ERR_INVALID_ARG;
  if (!al16(x) || !al16(w_r) || !al16(idx) || !al16n(bias) || !al16n(r_sel) ||
      (status_out && ((uintptr_t)status_out & 3u)))
    return XMOD_ERR_INVALID_ARG;
  if ((int64_t)dm->B * dm->T > (int64_t)XMOD_NOALLOC_MAX_TOKENS) return XMOD_ERR_UNSUPPORTED;
  if (dm->T > topk_max_T()) return XMOD_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  int err = XMOD_OK;
  void* base = scratch_on_current_device(s, &err);
  if (!base) return err;
  int* status = reinterpret_cast<int*>(base);
  float* logits = reinterpret_cast<float*>(reinterpret_cast<char*>(base) + kStatusBytes);
  Ctx c{s, status};
  if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return XMOD_ERR_CUDA;
  cudaError_t e;
  {
    ProfScope p("router", s);
    e = launch_router(c, dm->dtype, (int64_t)dm->B * dm->T, dm->d, x, w_r, bias, logits, nullptr);
  }
  count_launch();
  if (e != cudaSuccess) return XMOD_ERR_CUDA;
  {
    ProfScope p("topk", s);
    e = launch_topk(c, dm->B, dm->T, dm->T / K, logits, idx, r_sel);
  }
  count_launch();
  if (e != cudaSuccess) return XMOD_ERR_CUDA;
  if (status_out &&
      cudaMemcpyAsync(status_out, status, sizeof(int), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return XMOD_ERR_CUDA;
  return XMOD_OK;
}
