// ds_vit_encode_noalloc: the single-image encode without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they encode:
// a host application that carves the whole device-memory budget into its own
// pool at start-up and forbids any other allocation, a latency-critical loop
// that must not pay cudaMalloc's implicit device synchronisation, or a plugin
// interface whose fixed signature passes only inputs and outputs.  For them
// this entry point runs the same encode with its scratch (activations,
// QKV, MLP hidden, merger input) in a fixed, file-scope device array that is
// part of the library image: every GPU that loads the library holds it until
// the process exits, and no call allocates or frees anything.
//
// Limits and sharing: images of at most DS_VIT_NOALLOC_MAX_PATCHES patches
// (the worst such grid needs about 20 MiB of scratch; the array holds
// DS_VIT_NOALLOC_SCRATCH_BYTES).  All calls on a device share the one array
// and it keeps the previous call's contents; nothing in it needs to start at
// zero (every buffer is written in full before it is read).  Calls whose
// kernels overlap on the GPU (different streams without ordering between them)
// race on the array.
#include "internal.h"

#include <mutex>
#include <vector>

namespace {

constexpr size_t kScratchBytes = DS_VIT_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Host code cannot use g_noalloc_scratch as a device address (on the host it
// names a stand-in object).  Its device address belongs to one CUDA context:
// after cudaDeviceReset, or in a context the caller created itself, the array
// lives at another address.  So the address is looked up (cudaGetSymbolAddress,
// with the device current) once per context, keyed by the context's unique ID,
// which the driver never reuses within a process (a context handle can be).
struct ScratchEntry {
  unsigned long long ctx_id;
  void* addr;
};
std::vector<ScratchEntry> g_scratch;
std::mutex g_scratch_mu;

using PfnCtxGetCurrent = CUresult (*)(CUcontext*);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name, int version) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &fn, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return reinterpret_cast<Fn>(fn);
}

// Unique ID of the context current on this thread (the device's primary
// context is made current first when the thread has none).
int current_context_id(int dev, unsigned long long* id) {
  static const PfnCtxGetCurrent get_current = driver_fn<PfnCtxGetCurrent>("cuCtxGetCurrent", 4000);
  static const PfnCtxGetId get_id = driver_fn<PfnCtxGetId>("cuCtxGetId", 12000);
  if (!get_current || !get_id) return DS_VIT_ECUDA;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return DS_VIT_ECUDA;
  if (!ctx) {
    if (cudaSetDevice(dev) != cudaSuccess) {   // binds (and creates) the primary context
      cudaGetLastError();
      return DS_VIT_ECUDA;
    }
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return DS_VIT_ECUDA;
  }
  return get_id(ctx, id) == CUDA_SUCCESS ? DS_VIT_OK : DS_VIT_ECUDA;
}

int scratch_address(int dev, void** out) {
  unsigned long long id = 0;
  const int rc = current_context_id(dev, &id);
  if (rc != DS_VIT_OK) return rc;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  for (const ScratchEntry& e : g_scratch) {
    if (e.ctx_id == id) {
      *out = e.addr;
      return DS_VIT_OK;
    }
  }
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
    cudaGetLastError();
    return DS_VIT_ECUDA;
  }
  g_scratch.push_back({id, ptr});
  *out = ptr;
  return DS_VIT_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" int ds_vit_encode_noalloc(const ds_vit_prepared* p, const uint8_t* pixels, int32_t H,
                                     int32_t W, void* out, void* stream) {
  // Argument checks in the order the header states: pointers and their
  // alignment, image size, device, then the patch limit of the scratch array.
  if (!p || !pixels || !out || !aligned(out, 16) || !aligned(pixels, 4)) return DS_VIT_EINVAL;
  int32_t h = H, w = W;
  size_t need = 0;
  const int rc = ds_vit_workspace_bytes(p, 1, &h, &w, &need);   // validates H and W
  if (rc != DS_VIT_OK) return rc;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return DS_VIT_ECUDA;
  }
  if (dev != dsvit::prepared_device(p)) return DS_VIT_EINVAL;
  if (static_cast<int64_t>(H / 14) * (W / 14) > DS_VIT_NOALLOC_MAX_PATCHES || need > kScratchBytes)
    return DS_VIT_ERANGE;
  void* scratch = nullptr;
  const int rs = scratch_address(dev, &scratch);
  if (rs != DS_VIT_OK) return rs;
  return ds_vit_encode(p, pixels, H, W, out, scratch, kScratchBytes, stream);
}
