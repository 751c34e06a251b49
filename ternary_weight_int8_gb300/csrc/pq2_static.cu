// pq2_static.cu — pq2_linear with a static device workspace, for callers
// that cannot allocate device memory.  No step of the method lives here: the
// call hands a file-scope device array to pq2_linear as its workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "pq2.h"

namespace {

// The workspace of every pq2_linear_static call on a device (q, s_x and
// sum(q)); pq2_linear requires 256-byte alignment.
static __device__ __align__(256) unsigned char g_scratch[PQ2_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per
// device with that device current; nullptr on failure.
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int pq2_linear_static(const void* x, int x_dtype, int64_t ldx, int64_t M, int64_t N,
                                 int64_t K, const uint8_t* codes, const uint16_t* scales,
                                 void* y, int y_dtype, int32_t* dev_status, void* stream) {
  if (!x || !codes || !scales || !y) return PQ2_ERR_NULL;
  const size_t need = pq2_linear_workspace_bytes(M, K);
  if (need == 0 || need > PQ2_STATIC_SCRATCH_BYTES) return PQ2_ERR_SHAPE;
  void* ws = scratch_for_current_device();
  if (!ws) return PQ2_ERR_CUDA;
  return pq2_linear(x, x_dtype, ldx, M, N, K, codes, scales, y, y_dtype, ws,
                    PQ2_STATIC_SCRATCH_BYTES, dev_status, stream);
}
