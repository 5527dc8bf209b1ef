// Newton-Schulz for callers that cannot allocate device memory.
//
// muon_ns_batched allocates its workspace with cudaMallocAsync, and
// muon_ns_batched_ws needs the caller to hand it memory.  Some callers can do
// neither: a host that owns all device memory through its own arena and
// forbids allocations by libraries it loads, a runtime with a fixed memory
// budget that must not allocate after start-up, or a C caller with no device
// allocator at all.  muon_ns_batched_static gives them the same computation
// on a scratch array that this file reserves statically on the device.
//
// The scratch is resident on every GPU that loads this library until the
// process exits.  Host code cannot use the array's name as a device address
// (it is a host-side stand-in), so the first call on each device looks the
// address up with cudaGetSymbolAddress, with that device current, and caches
// it.  All calls share the one array and the array keeps whatever the last
// call left there; no part of it has to start at zero, because every byte a
// call reads is written earlier in the same call.  Calls whose work overlaps on
// the GPU (other streams, other host threads) race on the array.
#include <mutex>

#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_ns_static_scratch[MUON_NS_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MUON_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ns_static_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return MUON_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MUON_OK;
}

}  // namespace

extern "C" int muon_ns_batched_static(void *X, int64_t batch, int64_t m, int64_t n, int steps, const float coeffs[3],
                                      float eps, muon_stream_t stream) {
  // the errors of muon_ns_batched first, in its order, then the size limit,
  // all before any CUDA call
  int st = muon::ns_precheck(X, batch, m, n, steps, coeffs, eps);
  if (st != MUON_OK || batch == 0) return st;
  if (muon_ns_workspace_bytes(batch, m, n) > MUON_NS_STATIC_SCRATCH_BYTES) return MUON_ERR_NO_MEMORY;
  void *scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != MUON_OK) return st;
  return muon_ns_batched_ws(X, batch, m, n, steps, coeffs, eps, scratch, MUON_NS_STATIC_SCRATCH_BYTES, stream);
}
