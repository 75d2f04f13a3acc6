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

namespace {

constexpr size_t kScratchBytes = DS_VIT_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Host code cannot use g_noalloc_scratch as a device address (on the host it
// names a stand-in object).  The device address is looked up once per device,
// with that device current, on the first call made on it.
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return DS_VIT_ECUDA;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return DS_VIT_ECUDA;
    }
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return DS_VIT_OK;
}

}  // namespace

extern "C" int ds_vit_encode_noalloc(const ds_vit_prepared* p, const uint8_t* pixels, int32_t H,
                                     int32_t W, void* out, void* stream) {
  if (!p || !pixels || !out) return DS_VIT_EINVAL;
  int32_t h = H, w = W;
  size_t need = 0;
  const int rc = ds_vit_workspace_bytes(p, 1, &h, &w, &need);   // validates H and W
  if (rc != DS_VIT_OK) return rc;
  if (static_cast<int64_t>(H / 14) * (W / 14) > DS_VIT_NOALLOC_MAX_PATCHES || need > kScratchBytes)
    return DS_VIT_ERANGE;
  void* scratch = nullptr;
  const int rs = scratch_address(&scratch);
  if (rs != DS_VIT_OK) return rs;
  return ds_vit_encode(p, pixels, H, W, out, scratch, kScratchBytes, stream);
}
