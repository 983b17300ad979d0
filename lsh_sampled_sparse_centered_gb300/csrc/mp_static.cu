// Decode entry point that needs no scratch buffer from the caller.
//
// Some callers cannot hand the library a scratch allocation: a plugin running
// inside a host application whose device memory is owned by that application's
// pool, a serving loop that has reserved all device memory up front, or a latency-
// critical path that must not call cudaMalloc because the call can block on the
// device. For them, mp_decode_attention_static runs the same decode step with its
// scratch in a fixed array compiled into this library.
//
// The array is a file-scope __device__ variable of MP_STATIC_SCRATCH_BYTES: every
// GPU that loads the library keeps it resident until the process exits. Host code
// cannot use the array's name as a device address, so the first call on each device
// asks the runtime for the address (cudaGetSymbolAddress, with that device current)
// and caches it for the life of the process. The cache assumes the device's primary
// context is never torn down: after cudaDeviceReset the module is loaded again and the
// array can sit at another address, so a process that resets a device must not call
// this entry point afterwards. All calls share the array and it keeps the previous call's
// contents; the only words that must start at zero, the split-K completion
// counters, are reset on the device by the first kernel of every call. Two calls
// whose kernels overlap on the GPU (different streams, or different host threads
// without ordering) race on the array.
#include <mutex>

#include "mp_internal.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[MP_STATIC_SCRATCH_BYTES];

std::mutex g_static_mu;
void* g_static_addr[kMaxDevices] = {};

}  // namespace

extern "C" int mp_decode_attention_static(const mp_config* cfg, void* tables, const void* keys,
                                          const void* values, int32_t n, const void* q, float* out, void* stream) {
  mp_decode_layout layout;
  const int rc = mp_decode_layout_get(cfg, &layout);
  if (rc != MP_OK) return rc;
  if (layout.total_bytes > MP_STATIC_SCRATCH_BYTES) return MP_ERR_SCRATCH;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MP_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return MP_ERR_CUDA;
      g_static_addr[dev] = p;
    }
    scratch = g_static_addr[dev];
  }
  return mp_decode_attention(cfg, tables, keys, values, n, q, out, scratch, MP_STATIC_SCRATCH_BYTES, stream);
}
