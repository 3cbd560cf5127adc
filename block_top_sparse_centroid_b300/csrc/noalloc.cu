// Block top-k decode for callers that cannot allocate device memory.
//
// kin_blocktopk_decode takes its scratch from the caller, which is normally a buffer the
// caller allocated once.  Some callers cannot do even that: a serving process that
// hands every byte of the GPU to its KV-cache pool at start-up and forbids later
// allocations, a plug-in that runs inside a host framework which owns all device memory,
// or a latency-critical loop where cudaMalloc / cudaFree would synchronise the device.
// For them this file keeps one fixed scratch area in the library itself, as a
// file-scope device array that every GPU which loads the library holds until exit.
#include <mutex>

#include "kin.h"
#include "kin_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = 32u << 20;   // 32 MiB per GPU
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_mutex;
void *g_scratch_addr[kMaxDevices] = {};   // device address of the array, per device

}  // namespace

extern "C" kin_status kin_blocktopk_decode_static(const kin_kv_cache *cache,
                                                  const kin_decode_args *args,
                                                  kin_stream_t stream) {
  using kin::set_error;
  size_t need = 0;
  kin_status s = kin_workspace_size(cache, args, 0, &need);
  if (s != KIN_OK) return s;
  if (need > kStaticScratchBytes)
    return set_error(KIN_ERR_WORKSPACE,
                     "these shapes need %zu bytes of scratch; the library's static scratch "
                     "holds %zu (use kin_blocktopk_decode with a caller workspace)",
                     need, kStaticScratchBytes);
  if (cache->k_pages == nullptr) return set_error(KIN_ERR_INVALID_ARG, "k_pages is NULL");
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, cache->k_pages);
  if (e != cudaSuccess)
    return set_error(KIN_ERR_CUDA, "cudaPointerGetAttributes: %s", cudaGetErrorString(e));
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return set_error(KIN_ERR_INVALID_ARG, "cache pages are not device memory");
  const int dev = attr.device;
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(KIN_ERR_UNSUPPORTED, "device %d is beyond the %d supported", dev, kMaxDevices);
  int cur = -1;
  e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return set_error(KIN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (cur != dev) {
    e = cudaSetDevice(dev);
    if (e != cudaSuccess) return set_error(KIN_ERR_CUDA, "cudaSetDevice: %s", cudaGetErrorString(e));
  }
  // the caller's device is current again when this call returns, on every path
  struct Restore {
    int prev;
    bool switched;
    ~Restore() {
      if (switched) cudaSetDevice(prev);
    }
  } restore{cur, cur != dev};
  void *scratch = nullptr;
  {
    // First call on a device: resolve the array's device address with that device
    // current (the host-side name is only a stand-in, never a device address).
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_addr[dev] == nullptr) {
      void *p = nullptr;
      e = cudaGetSymbolAddress(&p, g_static_scratch);
      if (e != cudaSuccess)
        return set_error(KIN_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  kin_decode_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = kStaticScratchBytes;
  return kin_blocktopk_decode(cache, &a, stream);
}
