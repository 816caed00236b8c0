// dit_static_scratch.cu -- dit_selfcheck_static: the runtime-key self-check
// for callers that cannot allocate device memory.
//
// dit_selfcheck needs a workspace from the caller.  Some callers cannot get
// one at the moment they want the check: a process whose device memory is
// entirely reserved by a framework's caching allocator (any extra cudaMalloc
// would fail or fragment it), or a latency-critical loop that must not call
// cudaMalloc/cudaFree, which may synchronise the whole device.  For them the
// workspace lives here, in a file-scope device array that every GPU loading
// the library holds (DIT_SELFCHECK_STATIC_BYTES, 4 MiB) until the process
// exits.  The caller still passes the output, the mismatch counter.
//
// The array's name in host code is only a stand-in for the device symbol, so
// the host asks the runtime for its device address (cudaGetSymbolAddress),
// once per device with that device current, and hands that address on.
// Nothing in the array needs to start at zero: each check writes every
// element it later reads.  Every call shares the array, so calls that
// overlap on the GPU (other streams, other host threads) race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "dit_elementwise.h"

namespace {

static __device__ __align__(256) unsigned char g_scratch[DIT_SELFCHECK_STATIC_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];  // device address of g_scratch, per device
std::mutex g_scratch_mu;

// The device address of g_scratch on the current device (set up on the
// first call per device); NULL if the runtime cannot provide it.
void* scratch_address(int device) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess) {
      (void)cudaGetLastError();  // not the caller's next error
      return nullptr;
    }
    g_scratch_addr[device] = p;
  }
  return g_scratch_addr[device];
}

}  // namespace

extern "C" {

dit_status dit_selfcheck_static(dit_op op, dit_dtype dtype, dit_layout gate_layout,
                                dit_layout mod_layout, int64_t D, unsigned int* mismatches,
                                dit_stream_t stream) {
  // every argument check of dit_selfcheck but the workspace's: with no
  // workspace it returns DIT_ERR_WORKSPACE exactly when the rest is valid,
  // and launches nothing
  const dit_status st =
      dit_selfcheck(op, dtype, gate_layout, mod_layout, D, nullptr, 0, mismatches, stream);
  if (st != DIT_ERR_WORKSPACE) return st;
  const int64_t need = dit_selfcheck_workspace_bytes(op, dtype, D);
  if (need < 0 || need > (int64_t)DIT_SELFCHECK_STATIC_BYTES) return DIT_ERR_WORKSPACE;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices) {
    (void)cudaGetLastError();
    return DIT_ERR_NO_DEVICE;
  }
  void* ws = scratch_address(device);
  if (!ws) return DIT_ERR_NO_DEVICE;
  return dit_selfcheck(op, dtype, gate_layout, mod_layout, D, ws,
                       (int64_t)DIT_SELFCHECK_STATIC_BYTES, mismatches, stream);
}

}  // extern "C"
