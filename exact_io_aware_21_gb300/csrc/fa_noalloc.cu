// Split-KV decode for callers that cannot allocate device memory.
//
// fa_decode needs a caller-provided workspace for its per-split partial results.
// Some callers have no way to provide one: an inference server that reserves
// all device memory for its own pool at start-up and forbids any later
// cudaMalloc (an allocation there synchronises the device and fragments the
// pool), or a plug-in whose host framework gives it only the tensors of the
// call.  fa_decode_noalloc serves them: it runs the same kernels with the
// partials kept in a fixed array compiled into this library.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds FA_DECODE_SCRATCH_BYTES of device memory until the process
// exits.  Its host-side name is only a stand-in for the symbol, not a device
// address: the device address is looked up with cudaGetSymbolAddress, once
// per device, on the first call made with that device current.
#include <mutex>

#include "../../include/fa.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[FA_DECODE_SCRATCH_BYTES];

std::mutex g_mu;
void* g_addr[64] = {};  // device address of g_decode_scratch, per device ordinal

int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_decode_noalloc_max_bytes(void) { return FA_DECODE_SCRATCH_BYTES; }

int fa_decode_noalloc(const fa_tensor_t* q, const fa_tensor_t* kcache, const fa_tensor_t* vcache,
                      const fa_tensor_t* o, float* lse, const fa_shape_t* shape, int num_splits, void* stream) {
  const size_t need = fa_decode_workspace_size(shape, num_splits);
  if (need == 0) return FA_ERR_INVALID;
  if (need > FA_DECODE_SCRATCH_BYTES) return FA_ERR_TOO_LARGE;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != FA_OK) return rc;
  // fa_decode clears the scratch's header on `stream` before its kernels run
  // and writes every partial it later reads, so nothing left by an earlier
  // call can leak into this one.
  return fa_decode(q, kcache, vcache, o, lse, shape, num_splits, scratch, FA_DECODE_SCRATCH_BYTES, stream);
}

int fa_decode_noalloc_status(void* stream, int* status) {
  if (!status) return FA_ERR_INVALID;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != FA_OK) return rc;
  // the array starts with the same header as a workspace, status word first
  return fa_get_device_status(scratch, stream, status);
}

}  // extern "C"
