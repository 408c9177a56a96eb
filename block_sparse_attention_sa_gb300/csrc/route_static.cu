// route_static.cu -- sa_route_static: the router for callers that cannot
// allocate device memory.
//
// sa_route needs a scratch workspace (pooled blocks, pooled logits, masks,
// counts). Some callers cannot hand one over: a plugin running inside an
// inference engine that has already reserved all of HBM for its own pool,
// or code on a latency-critical path where a cudaMalloc would synchronise
// the device. For them this file owns a fixed scratch array in device memory
// and runs the unchanged sa_route on it.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds its SA_ROUTE_STATIC_WS_BYTES until the process exits. Host
// code cannot use the array's name as a device pointer, so the first call on
// each device (with that device current) asks the runtime for the array's
// device address and caches it; that first call should therefore come before
// any stream capture. All calls on a device share the one array and find in
// it whatever the previous call left: the router zeroes the few counters that
// must start at zero on every call, and two calls whose work overlaps on the
// GPU (different streams, no ordering between them) race on the array.
#include <mutex>

#include "sa_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_route_scratch[SA_ROUTE_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_route_scratch on the current device (looked up once).
sa_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // do not leave the lookup's error for the caller's next check
      return SA_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SA_OK;
}

}  // namespace

extern "C" sa_status sa_route_static(const sa_params* p, const void* q, const void* k,
                                     int32_t* row_ptr, int32_t* col_idx, int64_t col_cap,
                                     int32_t* dev_status, void* stream) {
  // Arguments first, in sa_route's order, then the capacity: a call that is
  // wrong in both ways reports the argument, as sa_route would.
  const size_t need = sa_route_workspace_bytes(p);
  if (need == 0)  // invalid parameters: let sa_route name the problem
    return sa_route(p, q, k, row_ptr, col_idx, col_cap, nullptr, 0, dev_status, stream);
  if (!q || !k || !row_ptr || !col_idx || col_cap < 0) return SA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) & 15u) != 0 || (reinterpret_cast<uintptr_t>(k) & 15u) != 0)
    return SA_ERR_INVALID_ARG;
  if (need > SA_ROUTE_STATIC_WS_BYTES) return SA_ERR_CAPACITY;
  void* ws = nullptr;
  const sa_status s = scratch_address(&ws);
  if (s != SA_OK) return s;
  return sa_route(p, q, k, row_ptr, col_idx, col_cap, ws, SA_ROUTE_STATIC_WS_BYTES, dev_status,
                  stream);
}
