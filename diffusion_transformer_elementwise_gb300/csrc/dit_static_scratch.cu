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
// the host asks the runtime for its device address (cudaGetSymbolAddress) on
// every call, with the caller's device current, and hands that address on.
// It is not cached: after cudaDeviceReset the module is loaded again in a new
// context and the array may sit elsewhere.
// Nothing in the array needs to start at zero: each check writes every
// element it later reads.  Every call shares the array, so calls that
// overlap on the GPU (other streams, other host threads) race on it.
#include <cuda_runtime.h>

#include "dit_elementwise.h"

namespace {

static __device__ __align__(256) unsigned char g_scratch[DIT_SELFCHECK_STATIC_BYTES];

// The device address of g_scratch in the current context; NULL if the
// runtime cannot provide it.
void* scratch_address() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess) {
    (void)cudaGetLastError();  // not the caller's next error
    return nullptr;
  }
  return p;
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
  if (cudaGetDevice(&device) != cudaSuccess || device < 0) {
    (void)cudaGetLastError();
    return DIT_ERR_NO_DEVICE;
  }
  void* ws = scratch_address();
  if (!ws) return DIT_ERR_NO_DEVICE;
  return dit_selfcheck(op, dtype, gate_layout, mod_layout, D, ws,
                       (int64_t)DIT_SELFCHECK_STATIC_BYTES, mismatches, stream);
}

dit_status dit_selfcheck_static_workspace(void** workspace, int64_t* bytes) {
  if (!workspace || !bytes) return DIT_ERR_NULL_PTR;
  *workspace = nullptr;
  *bytes = 0;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0) {
    (void)cudaGetLastError();
    return DIT_ERR_NO_DEVICE;
  }
  void* ws = scratch_address();
  if (!ws) return DIT_ERR_NO_DEVICE;
  *workspace = ws;
  *bytes = (int64_t)DIT_SELFCHECK_STATIC_BYTES;
  return DIT_OK;
}

}  // extern "C"
