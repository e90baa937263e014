// noalloc.cu -- nc_forward_static_scratch: the forward pass with its activation scratch
// taken from a fixed array compiled into the library instead of a caller buffer.
//
// Some callers cannot allocate device memory at the point where they run the model: code
// hosted by a framework that owns every device buffer through its own pool and forbids raw
// cudaMalloc, or a latency-bound serving loop where cudaMalloc / cudaFree would stall (they
// can synchronise the device).  Such callers already hold the model (created earlier), the
// token buffer and the logits buffer; this entry point needs nothing else.
//
// The scratch lives in one file-scope __device__ array of NC_STATIC_SCRATCH_BYTES.  Every
// GPU that loads this library keeps that much memory reserved until the process exits.
// Host code must not hand the array's name to a kernel (on the host it names a shadow
// variable, not device memory); the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on that device.
// Under CUDA's lazy module loading that lookup is also what loads this library's device code
// on the device and reserves the array, so the first call can fail with NC_ERR_CUDA when the
// device is short of memory; callers make it at set-up time.
#include <mutex>

#include "internal.h"
#include "nc.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[NC_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
nc_status scratch_for_current_device(void** out) {
  int dev = -1;
  const nc_status s = nc::cuda_status(cudaGetDevice(&dev));
  if (s != NC_OK) return s;
  if (dev < 0 || dev >= kMaxDevices) return NC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    const nc_status e = nc::cuda_status(cudaGetSymbolAddress(&p, g_static_scratch));
    if (e != NC_OK) return e;
    if (p == nullptr) return NC_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return NC_OK;
}

}  // namespace

extern "C" nc_status nc_forward_static_scratch(nc_model* m, const int32_t* tokens, int B, int T,
                                               void* logits, void* stream) {
  if (m == nullptr || tokens == nullptr || logits == nullptr) return NC_ERR_INVALID_ARG;
  size_t need = 0;
  nc_status s = nc_workspace_bytes(m, B, T, &need);
  if (s != NC_OK) return s;
  if (need > static_cast<size_t>(NC_STATIC_SCRATCH_BYTES)) return NC_ERR_WORKSPACE;
  void* scratch = nullptr;
  s = scratch_for_current_device(&scratch);
  if (s != NC_OK) return s;
  // Every region of the scratch is written before it is read within one forward, so the
  // previous call's leftovers need no clearing.
  return nc_forward(m, tokens, B, T, logits, scratch, static_cast<size_t>(NC_STATIC_SCRATCH_BYTES), stream);
}
