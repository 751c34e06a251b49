// pq2_static.cu — pq2_linear with a static device workspace, for callers
// that cannot allocate device memory.  No step of the method lives here: the
// call hands a file-scope device array to pq2_linear as its workspace.
#include <cuda.h>
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
unsigned long long g_scratch_ctx[kMaxDevices] = {};  // context ID the address belongs to

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique ID of the current context (0 if it cannot be had).  A device reset
// replaces the primary context, and with it the ID and the module holding
// g_scratch, so the address is looked up again for a new ID.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    cudaGetLastError();
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_scratch in the current device's context.  It is looked
// up with that device current on the device's first call (the lookup also
// creates the device's primary context), and again whenever the current
// context is not the one the address was found in (a device reset replaces
// it), or on every call where the context ID cannot be read.  nullptr on
// failure.  No call here allocates or frees memory.
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  const unsigned long long ctx = current_context_id();
  if (g_scratch_ptr[dev] && ctx != 0 && ctx == g_scratch_ctx[dev]) return g_scratch_ptr[dev];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    g_scratch_ptr[dev] = nullptr;
    return nullptr;
  }
  g_scratch_ptr[dev] = p;
  g_scratch_ctx[dev] = current_context_id();
  return p;
}

// The stream must belong to the current device, whose scratch address is
// passed on (a kernel on another device would be handed a foreign address).
bool stream_on_current_device(void* stream) {
  if (!stream) return true;  // the legacy default stream of the current device
  int dev = -1, sdev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return dev == sdev;
}

}  // namespace

extern "C" int pq2_linear_static(const void* x, int x_dtype, int64_t ldx, int64_t M, int64_t N,
                                 int64_t K, const uint8_t* codes, const uint16_t* scales,
                                 void* y, int y_dtype, int32_t* dev_status, void* stream) {
  // Argument errors in pq2_linear's order (NULL, dtype, shape), the size of
  // the static scratch being a shape limit.
  if (!x || !codes || !scales || !y) return PQ2_ERR_NULL;
  if (x_dtype != PQ2_BF16 && x_dtype != PQ2_F16 && x_dtype != PQ2_F32) return PQ2_ERR_DTYPE;
  if (y_dtype != PQ2_F32 && y_dtype != PQ2_BF16) return PQ2_ERR_DTYPE;
  const size_t need = pq2_linear_workspace_bytes(M, K);
  if (need == 0 || need > PQ2_STATIC_SCRATCH_BYTES) return PQ2_ERR_SHAPE;
  if (!stream_on_current_device(stream)) return PQ2_ERR_CUDA;
  void* ws = scratch_for_current_device();
  if (!ws) return PQ2_ERR_CUDA;
  return pq2_linear(x, x_dtype, ldx, M, N, K, codes, scales, y, y_dtype, ws,
                    PQ2_STATIC_SCRATCH_BYTES, dev_status, stream);
}
