// pq2_api.cu — the C ABI of libpq2: argument validation, device checks and
// dispatch to the kernels.  Every argument error is reported before any CUDA
// call, so invalid calls never touch the device.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "pq2.h"
#include "pq2_internal.h"

namespace {

constexpr int kLayoutVersion = 1;  // code plane [N][K/4] then fp16 scales [N][K/128]
constexpr int64_t kMaxK = (int64_t)1 << 24;
constexpr int64_t kMaxN = (int64_t)1 << 30;
constexpr int64_t kMaxM = (int64_t)1 << 20;
constexpr int kMaxDevices = 64;

// Per-device cache: 0 = unknown, 1 = sm_103 (GB300), 2 = other architecture.
std::atomic<int> g_arch[kMaxDevices];
std::atomic<int> g_sms[kMaxDevices];

bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

bool valid_k(int64_t K) { return K >= 128 && K % 128 == 0 && K <= kMaxK; }
bool valid_n(int64_t N) { return N >= 1 && N <= kMaxN; }

// Compute capability 10.3 check and SM count of the current device.
int device_check(int* sm_count) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return PQ2_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return PQ2_ERR_CUDA;
  int arch = g_arch[dev].load(std::memory_order_acquire);
  if (arch == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return PQ2_ERR_CUDA;
    }
    g_sms[dev].store(sms, std::memory_order_relaxed);
    arch = (major == 10 && minor == 3) ? 1 : 2;
    g_arch[dev].store(arch, std::memory_order_release);
  }
  if (arch != 1) return PQ2_ERR_ARCH;
  *sm_count = g_sms[dev].load(std::memory_order_relaxed);
  return PQ2_OK;
}

int elem_bytes(int dtype) { return dtype == PQ2_F32 ? 4 : 2; }

bool valid_layout(int q_layout) {
  return q_layout == PQ2_Q_ROWS || q_layout == PQ2_Q_PLANES || q_layout == PQ2_Q_F16 ||
         q_layout == PQ2_Q_F8 || q_layout == PQ2_Q_MMV16;
}

int check_mmv_args(const int8_t* q, const float* sx, const int32_t* qsum,
                   const uint8_t* codes, const uint16_t* scales, const void* y,
                   int y_dtype, int64_t M, int64_t N, int64_t K, int decode) {
  if (!q || !sx || !qsum || !codes || !scales || !y) return PQ2_ERR_NULL;
  if (M < 1 || M > 8 || !valid_n(N) || !valid_k(K)) return PQ2_ERR_SHAPE;
  if (y_dtype != PQ2_F32 && y_dtype != PQ2_BF16) return PQ2_ERR_DTYPE;
  if (decode != PQ2_DECODE_ADDXOR && decode != PQ2_DECODE_PLANES) return PQ2_ERR_DTYPE;
  if (!aligned(q, 16) || !aligned(codes, 16) || !aligned(sx, 4) || !aligned(qsum, 4) ||
      !aligned(scales, 2) || !aligned(y, elem_bytes(y_dtype)))
    return PQ2_ERR_ALIGN;
  return PQ2_OK;
}

}  // namespace

extern "C" {

int pq2_layout_version(void) { return kLayoutVersion; }

const char* pq2_status_string(int status) {
  switch (status) {
    case PQ2_OK: return "ok";
    case PQ2_ERR_NULL: return "a required pointer is NULL";
    case PQ2_ERR_SHAPE: return "shape, stride or size out of range";
    case PQ2_ERR_ALIGN: return "pointer or stride misaligned";
    case PQ2_ERR_DTYPE: return "unknown dtype, layout or decoder";
    case PQ2_ERR_ARCH: return "device is not compute capability 10.3 (GB300)";
    case PQ2_ERR_LAUNCH: return "CUDA launch failed";
    case PQ2_ERR_TIMEOUT: return "a bounded device wait gave up";
    case PQ2_ERR_CUDA: return "CUDA runtime query failed";
    default: return "unknown status";
  }
}

size_t pq2_prepared_bytes(int64_t N, int64_t K) {
  if (!valid_n(N) || !valid_k(K)) return 0;
  return (size_t)N * (size_t)(K / 4) + (size_t)N * (size_t)(K / 128) * 2;
}

int pq2_prepare(const uint8_t* raw, int64_t raw_row_stride, int64_t N, int64_t K,
                uint8_t* codes, uint16_t* scales, void* stream) {
  if (!raw || !codes || !scales) return PQ2_ERR_NULL;
  if (!valid_n(N) || !valid_k(K) || raw_row_stride < K / 128 * 34) return PQ2_ERR_SHAPE;
  if (!aligned(codes, 16) || !aligned(scales, 2)) return PQ2_ERR_ALIGN;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  return pq2::launch_prepare(raw, raw_row_stride, N, K, codes, scales,
                             static_cast<cudaStream_t>(stream));
}

int pq2_quantize_act(const void* x, int x_dtype, int64_t ldx, int64_t M, int64_t K,
                     void* q, int q_layout, float* sx, int32_t* qsum, void* stream) {
  if (!x || !q || !sx) return PQ2_ERR_NULL;
  if (x_dtype != PQ2_BF16 && x_dtype != PQ2_F16 && x_dtype != PQ2_F32) return PQ2_ERR_DTYPE;
  if (!valid_layout(q_layout)) return PQ2_ERR_DTYPE;
  if (M < 1 || M > kMaxM || !valid_k(K) || ldx < K || ldx > ((int64_t)1 << 40))
    return PQ2_ERR_SHAPE;
  if (!aligned(x, elem_bytes(x_dtype)) || !aligned(q, 16) || !aligned(sx, 4) ||
      (qsum && !aligned(qsum, 4)))
    return PQ2_ERR_ALIGN;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  return pq2::launch_quantize(x, x_dtype, ldx, M, K, q, q_layout, sx, qsum,
                              static_cast<cudaStream_t>(stream));
}

// The masked-plane decoder needs one LOP3 per code byte where the add/XOR
// expansion needs about three, and on GB300 both share the half-rate integer
// pipe with dp4a; it is the faster decoder for every M.
int pq2_mmv_decoder(int64_t M) {
  (void)M;
  return PQ2_DECODE_PLANES;
}

int pq2_mmv_ex(const int8_t* q, const float* sx, const int32_t* qsum, const uint8_t* codes,
               const uint16_t* scales, void* y, int y_dtype, int64_t M, int64_t N,
               int64_t K, int decode, int flags, int32_t* dev_status, void* stream) {
  if (int st = check_mmv_args(q, sx, qsum, codes, scales, y, y_dtype, M, N, K, decode))
    return st;
  if (flags & ~(PQ2_MMV_OVERLAP_WEIGHTS | PQ2_MMV_INDEPENDENT)) return PQ2_ERR_DTYPE;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  const int overlap = (flags & PQ2_MMV_INDEPENDENT) ? 2 : (flags & PQ2_MMV_OVERLAP_WEIGHTS) ? 1 : 0;
  return pq2::launch_mmv(q, sx, qsum, codes, scales, y, y_dtype, nullptr, M, N, K, decode,
                         overlap, sms, dev_status, static_cast<cudaStream_t>(stream));
}

int pq2_mmv_tc(const uint16_t* q_mmv16, const float* sx, const int32_t* qcorr,
               const uint8_t* codes, const uint16_t* scales, void* y, int y_dtype, int64_t M,
               int64_t N, int64_t K, int flags, int32_t* dev_status, void* stream) {
  if (int st = check_mmv_args(reinterpret_cast<const int8_t*>(q_mmv16), sx, qcorr, codes, scales,
                              y, y_dtype, M, N, K, PQ2_DECODE_PLANES))
    return st;
  if (flags & ~(PQ2_MMV_OVERLAP_WEIGHTS | PQ2_MMV_INDEPENDENT)) return PQ2_ERR_DTYPE;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  const int overlap = (flags & PQ2_MMV_INDEPENDENT) ? 2 : (flags & PQ2_MMV_OVERLAP_WEIGHTS) ? 1 : 0;
  return pq2::launch_mmv(reinterpret_cast<const int8_t*>(q_mmv16), sx, qcorr, codes, scales, y,
                         y_dtype, nullptr, M, N, K, pq2::kDecodeTensor, overlap, sms, dev_status,
                         static_cast<cudaStream_t>(stream));
}

// pq2_linear's choice between the two GEMVs (same bits), from their measured
// cost in a chain of dependent calls on GB300: the dp4a kernel's cost grows
// with M, the tensor-core kernel's does not.  The tensor-core kernel wins
// from M = 6 on every layer shape, and at M = 5 where a CTA holds at most 72
// rows of at most 8 splits (attn_qkv, 5120 x 6144; not ffn_up's 115-row or
// ffn_down's 16-split slabs).
int pq2_linear_tensor_gemv(int64_t M, int64_t N, int64_t K, int sm_count) {
  if (M < 5 || M > 8) return 0;
  if (M >= 6) return 1;
  pq2::MmvGeometry g;
  if (!pq2::mmv_geometry(N, K, sm_count, &g)) return 0;
  return g.splits <= 8 && g.rows_max <= 72 ? 1 : 0;
}

int pq2_mmv(const int8_t* q, const float* sx, const int32_t* qsum, const uint8_t* codes,
            const uint16_t* scales, void* y, int y_dtype, int64_t M, int64_t N, int64_t K,
            int32_t* dev_status, void* stream) {
  return pq2_mmv_ex(q, sx, qsum, codes, scales, y, y_dtype, M, N, K,
                    pq2_mmv_decoder(M < 1 ? 1 : M), 0, dev_status, stream);
}

int pq2_quantize_act_grouped(const void* x, int x_dtype, int64_t ldx, int64_t M, int64_t K,
                             int act_group, void* q, int q_layout, float* sx, int32_t* qsum,
                             void* stream) {
  if (act_group != 128 && act_group != 64 && act_group != 32) return PQ2_ERR_SHAPE;
  if (q_layout == PQ2_Q_MMV16 && act_group != 128) return PQ2_ERR_SHAPE;
  if (!x || !q || !sx) return PQ2_ERR_NULL;
  if (x_dtype != PQ2_BF16 && x_dtype != PQ2_F16 && x_dtype != PQ2_F32) return PQ2_ERR_DTYPE;
  if (!valid_layout(q_layout)) return PQ2_ERR_DTYPE;
  if (M < 1 || M > kMaxM || !valid_k(K) || ldx < K || ldx > ((int64_t)1 << 40))
    return PQ2_ERR_SHAPE;
  if (!aligned(x, elem_bytes(x_dtype)) || !aligned(q, 16) || !aligned(sx, 4) ||
      (qsum && !aligned(qsum, 4)))
    return PQ2_ERR_ALIGN;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  return pq2::launch_quantize(x, x_dtype, ldx, M, K, q, q_layout, sx, qsum,
                              static_cast<cudaStream_t>(stream), act_group);
}

int pq2_mmv_grouped(const int8_t* q, const float* sx, const int32_t* qsum, const uint8_t* codes,
                    const uint16_t* scales, void* y, int y_dtype, int64_t M, int64_t N,
                    int64_t K, int act_group, int flags, int32_t* dev_status, void* stream) {
  if (int st = check_mmv_args(q, sx, qsum, codes, scales, y, y_dtype, M, N, K,
                              PQ2_DECODE_PLANES))
    return st;
  if (act_group != 128 && act_group != 64 && act_group != 32) return PQ2_ERR_SHAPE;
  if (flags & ~(PQ2_MMV_OVERLAP_WEIGHTS | PQ2_MMV_INDEPENDENT)) return PQ2_ERR_DTYPE;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  const int overlap = (flags & PQ2_MMV_INDEPENDENT) ? 2 : (flags & PQ2_MMV_OVERLAP_WEIGHTS) ? 1 : 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The kernel holds at most four columns' partial sums: columns 4..M-1 run
  // as a second pass over the weights.  A column's result does not depend on
  // the others, so the bits are those of one pass.
  const int64_t GA = K / act_group, first = M < 4 ? M : 4;
  if (int st = pq2::launch_mmv_grouped(q, sx, qsum, codes, scales, y, y_dtype, nullptr, first, N,
                                       K, act_group, overlap, sms, dev_status, s))
    return st;
  if (M == first) return PQ2_OK;
  return pq2::launch_mmv_grouped(q + 4 * K, sx + 4 * GA, qsum + 4 * GA, codes, scales,
                                 static_cast<uint8_t*>(y) + 4 * N * elem_bytes(y_dtype), y_dtype,
                                 nullptr, M - 4, N, K, act_group, overlap, sms, dev_status, s);
}

int pq2_debug_group_dots_grouped(const int8_t* q, const int32_t* qsum, const uint8_t* codes,
                                 int64_t M, int64_t N, int64_t K, int act_group, int32_t* dots,
                                 int32_t* dev_status, void* stream) {
  if (!q || !qsum || !codes || !dots) return PQ2_ERR_NULL;
  if (M < 1 || M > 8 || !valid_n(N) || !valid_k(K) ||
      (act_group != 128 && act_group != 64 && act_group != 32))
    return PQ2_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(codes, 16) || !aligned(dots, 4) || !aligned(qsum, 4))
    return PQ2_ERR_ALIGN;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t GA = K / act_group, first = M < 4 ? M : 4;
  if (int st = pq2::launch_mmv_grouped(q, nullptr, qsum, codes, nullptr, nullptr, PQ2_F32, dots,
                                       first, N, K, act_group, 0, sms, dev_status, s))
    return st;
  if (M == first) return PQ2_OK;
  return pq2::launch_mmv_grouped(q + 4 * K, nullptr, qsum + 4 * GA, codes, nullptr, nullptr,
                                 PQ2_F32, dots + 4 * N * GA, M - 4, N, K, act_group, 0, sms,
                                 dev_status, s);
}

int pq2_ptq_prepare(const uint8_t* raw, int64_t raw_row_stride, int64_t N, int64_t K,
                    uint8_t* qs, uint32_t* side, void* stream) {
  if (!raw || !qs || !side) return PQ2_ERR_NULL;
  if (!valid_n(N) || !valid_k(K) || K % 256 || raw_row_stride < K / 128 * 28)
    return PQ2_ERR_SHAPE;
  if (!aligned(qs, 16) || !aligned(side, 8)) return PQ2_ERR_ALIGN;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  return pq2::launch_ptq_prepare(raw, raw_row_stride, N, K, qs, side,
                                 static_cast<cudaStream_t>(stream));
}

namespace {
int check_ptq_args(const int8_t* q, const int32_t* qsum, const uint8_t* qs, const uint32_t* side,
                   int64_t M, int64_t N, int64_t K, int act_group) {
  if (!q || !qsum || !qs || !side) return PQ2_ERR_NULL;
  if (M < 1 || M > 4 || !valid_n(N) || !valid_k(K) || K % 256 ||
      (act_group != 128 && act_group != 64 && act_group != 32))
    return PQ2_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(qsum, 4) || !aligned(qs, 16) || !aligned(side, 8))
    return PQ2_ERR_ALIGN;
  return PQ2_OK;
}
}  // namespace

int pq2_ptq_mmv(const int8_t* q_rows, const float* sx, const int32_t* qsum, const uint8_t* qs,
                const uint32_t* side, void* y, int y_dtype, int64_t M, int64_t N, int64_t K,
                int act_group, int flags, void* stream) {
  if (int st = check_ptq_args(q_rows, qsum, qs, side, M, N, K, act_group)) return st;
  if (!sx || !y) return PQ2_ERR_NULL;
  if (y_dtype != PQ2_F32 && y_dtype != PQ2_BF16) return PQ2_ERR_DTYPE;
  if (flags & ~(PQ2_MMV_OVERLAP_WEIGHTS | PQ2_MMV_INDEPENDENT)) return PQ2_ERR_DTYPE;
  if (!aligned(sx, 4) || !aligned(y, elem_bytes(y_dtype))) return PQ2_ERR_ALIGN;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  const int overlap = (flags & PQ2_MMV_INDEPENDENT) ? 2 : (flags & PQ2_MMV_OVERLAP_WEIGHTS) ? 1 : 0;
  return pq2::launch_ptq_mmv(q_rows, sx, qsum, qs, side, y, y_dtype, nullptr, M, N, K, act_group,
                             overlap, sms, static_cast<cudaStream_t>(stream));
}

size_t pq2_ptq_linear_workspace_bytes(int64_t M, int64_t K, int act_group) {
  if (M < 1 || M > 4 || !valid_k(K) || K % 256 ||
      (act_group != 128 && act_group != 64 && act_group != 32))
    return 0;
  const size_t GA = (size_t)(K / act_group);
  const size_t q_bytes = (size_t)M * (size_t)K;
  const size_t sx_off = (q_bytes + 255) / 256 * 256;
  const size_t qs_off = (sx_off + (size_t)M * GA * 4 + 255) / 256 * 256;
  return qs_off + (size_t)M * GA * 4;
}

int pq2_ptq_linear(const void* x, int x_dtype, int64_t ldx, int64_t M, int64_t N, int64_t K,
                   const uint8_t* qs, const uint32_t* side, int act_group, void* y, int y_dtype,
                   void* workspace, size_t workspace_bytes, void* stream) {
  if (!x || !qs || !side || !y || !workspace) return PQ2_ERR_NULL;
  if (x_dtype != PQ2_BF16 && x_dtype != PQ2_F16 && x_dtype != PQ2_F32) return PQ2_ERR_DTYPE;
  if (y_dtype != PQ2_F32 && y_dtype != PQ2_BF16) return PQ2_ERR_DTYPE;
  const size_t need = pq2_ptq_linear_workspace_bytes(M, K, act_group);
  if (need == 0 || !valid_n(N) || ldx < K || ldx > ((int64_t)1 << 40)) return PQ2_ERR_SHAPE;
  if (workspace_bytes < need) return PQ2_ERR_SHAPE;
  if (!aligned(x, elem_bytes(x_dtype)) || !aligned(workspace, 256) || !aligned(qs, 16) ||
      !aligned(side, 8) || !aligned(y, elem_bytes(y_dtype)))
    return PQ2_ERR_ALIGN;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  const size_t GA = (size_t)(K / act_group);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t sx_off = ((size_t)M * (size_t)K + 255) / 256 * 256;
  const size_t qs_off = (sx_off + (size_t)M * GA * 4 + 255) / 256 * 256;
  float* sx = reinterpret_cast<float*>(ws + sx_off);
  int32_t* qsum = reinterpret_cast<int32_t*>(ws + qs_off);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (int st = pq2::launch_quantize(x, x_dtype, ldx, M, K, ws, PQ2_Q_ROWS, sx, qsum, s,
                                    act_group))
    return st;
  // The GEMV streams its weights while the quantisation runs.
  return pq2::launch_ptq_mmv(reinterpret_cast<const int8_t*>(ws), sx, qsum, qs, side, y, y_dtype,
                             nullptr, M, N, K, act_group, 1, sms, s);
}

int pq2_debug_ptq_dots(const int8_t* q_rows, const int32_t* qsum, const uint8_t* qs,
                       const uint32_t* side, int64_t M, int64_t N, int64_t K, int act_group,
                       int32_t* dots, void* stream) {
  if (int st = check_ptq_args(q_rows, qsum, qs, side, M, N, K, act_group)) return st;
  if (!dots) return PQ2_ERR_NULL;
  if (!aligned(dots, 4)) return PQ2_ERR_ALIGN;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  return pq2::launch_ptq_mmv(q_rows, nullptr, qsum, qs, side, nullptr, PQ2_F32, dots, M, N, K,
                             act_group, 0, sms, static_cast<cudaStream_t>(stream));
}

int pq2_mmv_gated(const int8_t* q, const float* sx, const int32_t* qsum, const uint8_t* codes,
                  const uint16_t* scales, void* out, int out_dtype, int64_t M, int64_t N,
                  int64_t K, int flags, int32_t* dev_status, void* stream) {
  if (int st = check_mmv_args(q, sx, qsum, codes, scales, out, out_dtype, M, N, K,
                              PQ2_DECODE_PLANES))
    return st;
  if (N % 2) return PQ2_ERR_SHAPE;
  if (flags & ~(PQ2_MMV_OVERLAP_WEIGHTS | PQ2_MMV_INDEPENDENT)) return PQ2_ERR_DTYPE;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  const int overlap = (flags & PQ2_MMV_INDEPENDENT) ? 2 : (flags & PQ2_MMV_OVERLAP_WEIGHTS) ? 1 : 0;
  return pq2::launch_mmv_gated(q, sx, qsum, codes, scales, out, out_dtype, M, N, K,
                               pq2::kDecodeMaskPlanes, overlap, sms, dev_status,
                               static_cast<cudaStream_t>(stream));
}

// q bytes per element in pq2_linear's workspace: int8 planes for the dp4a
// GEMV (M <= 4), fp16 where the tensor-core GEMV (PQ2_Q_MMV16, M = 5..8)
// or the prefill GEMM (M >= 9) may run.
static size_t linear_q_elem(int64_t M) { return M <= 4 ? 1 : 2; }

size_t pq2_linear_workspace_bytes(int64_t M, int64_t K) {
  if (M < 1 || M > kMaxM || !valid_k(K)) return 0;
  const size_t G = (size_t)(K / 128);
  const size_t q_bytes = (size_t)M * (size_t)K * linear_q_elem(M);
  const size_t sx_off = (q_bytes + 255) / 256 * 256;
  const size_t qs_off = (sx_off + (size_t)M * G * 4 + 255) / 256 * 256;
  return qs_off + (size_t)M * G * 4;
}

int pq2_linear(const void* x, int x_dtype, int64_t ldx, int64_t M, int64_t N, int64_t K,
               const uint8_t* codes, const uint16_t* scales, void* y, int y_dtype,
               void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (!x || !codes || !scales || !y || !workspace) return PQ2_ERR_NULL;
  if (x_dtype != PQ2_BF16 && x_dtype != PQ2_F16 && x_dtype != PQ2_F32) return PQ2_ERR_DTYPE;
  if (y_dtype != PQ2_F32 && y_dtype != PQ2_BF16) return PQ2_ERR_DTYPE;
  if (M < 1 || M > kMaxM || !valid_n(N) || !valid_k(K) || ldx < K ||
      ldx > ((int64_t)1 << 40))
    return PQ2_ERR_SHAPE;
  if (workspace_bytes < pq2_linear_workspace_bytes(M, K)) return PQ2_ERR_SHAPE;
  if (!aligned(x, elem_bytes(x_dtype)) || !aligned(workspace, 256) || !aligned(codes, 16) ||
      !aligned(scales, 2) || !aligned(y, elem_bytes(y_dtype)))
    return PQ2_ERR_ALIGN;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  const size_t G = (size_t)(K / 128);
  const bool small = M <= 8;
  const bool tensor = small && pq2_linear_tensor_gemv(M, N, K, sms);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t q_bytes = (size_t)M * (size_t)K * linear_q_elem(M);
  const size_t sx_off = (q_bytes + 255) / 256 * 256;
  const size_t qs_off = (sx_off + (size_t)M * G * 4 + 255) / 256 * 256;
  float* sx = reinterpret_cast<float*>(ws + sx_off);
  int32_t* qs = reinterpret_cast<int32_t*>(ws + qs_off);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int layout = !small ? PQ2_Q_F8 : tensor ? PQ2_Q_MMV16 : PQ2_Q_PLANES;
  if (int st = pq2::launch_quantize(x, x_dtype, ldx, M, K, ws, layout, sx, qs, s)) return st;
  // Prefill on the 8-bit tensor path: bit-identical to the fp16 one, faster.
  if (!small)
    return pq2::launch_mm(ws, true, sx, qs, codes, scales, y, y_dtype, nullptr, M, N, K, sms,
                          dev_status, s);
  return pq2::launch_mmv(reinterpret_cast<const int8_t*>(ws), sx, qs, codes, scales, y,
                         y_dtype, nullptr, M, N, K,
                         tensor ? pq2::kDecodeTensor : pq2_mmv_decoder(M), 1, sms, dev_status,
                         s);
}

int pq2_linear_gated(const void* x, int x_dtype, int64_t ldx, int64_t M, int64_t N, int64_t K,
                     const uint8_t* codes, const uint16_t* scales, void* out, int out_dtype,
                     void* workspace, size_t workspace_bytes, int32_t* dev_status,
                     void* stream) {
  if (!x || !codes || !scales || !out || !workspace) return PQ2_ERR_NULL;
  if (x_dtype != PQ2_BF16 && x_dtype != PQ2_F16 && x_dtype != PQ2_F32) return PQ2_ERR_DTYPE;
  if (out_dtype != PQ2_F32 && out_dtype != PQ2_BF16) return PQ2_ERR_DTYPE;
  if (M < 1 || M > 8 || !valid_n(N) || N % 2 || !valid_k(K) || ldx < K ||
      ldx > ((int64_t)1 << 40))
    return PQ2_ERR_SHAPE;
  if (workspace_bytes < pq2_linear_workspace_bytes(M, K)) return PQ2_ERR_SHAPE;
  if (!aligned(x, elem_bytes(x_dtype)) || !aligned(workspace, 256) || !aligned(codes, 16) ||
      !aligned(scales, 2) || !aligned(out, elem_bytes(out_dtype)))
    return PQ2_ERR_ALIGN;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  const size_t G = (size_t)(K / 128);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t q_bytes = (size_t)M * (size_t)K;
  const size_t sx_off = (q_bytes + 255) / 256 * 256;
  const size_t qs_off = (sx_off + (size_t)M * G * 4 + 255) / 256 * 256;
  float* sx = reinterpret_cast<float*>(ws + sx_off);
  int32_t* qs = reinterpret_cast<int32_t*>(ws + qs_off);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (int st = pq2::launch_quantize(x, x_dtype, ldx, M, K, ws, PQ2_Q_PLANES, sx, qs, s))
    return st;
  return pq2::launch_mmv_gated(reinterpret_cast<const int8_t*>(ws), sx, qs, codes, scales, out,
                               out_dtype, M, N, K, pq2::kDecodeMaskPlanes, 1, sms, dev_status,
                               s);
}

int pq2_norm_hadamard_quantize(const uint16_t* x, const uint16_t* residual,
                               uint16_t* residual_out, const uint16_t* w, const int8_t* sign,
                               float eps, int64_t M, int64_t K, uint16_t* norm_out, void* q,
                               int q_layout, float* sx, int32_t* qsum, void* stream) {
  if (!x || !w || !sign || !q || !sx) return PQ2_ERR_NULL;
  if (!valid_layout(q_layout)) return PQ2_ERR_DTYPE;
  if (M < 1 || M > kMaxM || K < 1024 || K > PQ2_PREP_MAX_K || K % 1024) return PQ2_ERR_SHAPE;
  if (!(eps >= 0.0f) || eps > 1.0f) return PQ2_ERR_SHAPE;
  if (!aligned(x, 2) || (residual && !aligned(residual, 2)) || (residual_out && !aligned(residual_out, 2)) ||
      !aligned(w, 2) || (norm_out && !aligned(norm_out, 2)) || !aligned(q, 16) ||
      !aligned(sx, 4) || (qsum && !aligned(qsum, 4)))
    return PQ2_ERR_ALIGN;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  return pq2::launch_norm_hadamard_quantize(x, residual, residual_out, w, sign, eps, M, K,
                                            norm_out, q, q_layout, sx, qsum,
                                            static_cast<cudaStream_t>(stream));
}

namespace {
int mm_call(const void* q, bool f8, const float* sx, const int32_t* qsum, const uint8_t* codes,
            const uint16_t* scales, void* y, int y_dtype, int64_t M, int64_t N, int64_t K,
            int act_group, int32_t* dev_status, void* stream) {
  if (!q || !sx || !qsum || !codes || !scales || !y) return PQ2_ERR_NULL;
  if (M < 1 || M > kMaxM || !valid_n(N) || !valid_k(K) ||
      (act_group != 128 && act_group != 64 && act_group != 32))
    return PQ2_ERR_SHAPE;
  if (y_dtype != PQ2_F32 && y_dtype != PQ2_BF16) return PQ2_ERR_DTYPE;
  if (!aligned(q, 16) || !aligned(codes, 16) || !aligned(sx, 4) || !aligned(qsum, 4) ||
      !aligned(scales, 2) || !aligned(y, elem_bytes(y_dtype)))
    return PQ2_ERR_ALIGN;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  return pq2::launch_mm(q, f8, sx, qsum, codes, scales, y, y_dtype, nullptr, M, N, K, sms,
                        dev_status, static_cast<cudaStream_t>(stream), act_group);
}
}  // namespace

int pq2_mm(const uint16_t* q_f16, const float* sx, const int32_t* qsum, const uint8_t* codes,
           const uint16_t* scales, void* y, int y_dtype, int64_t M, int64_t N, int64_t K,
           int32_t* dev_status, void* stream) {
  return mm_call(q_f16, false, sx, qsum, codes, scales, y, y_dtype, M, N, K, 128, dev_status,
                 stream);
}

int pq2_mm_f8(const uint8_t* q_f8, const float* sx, const int32_t* qsum, const uint8_t* codes,
              const uint16_t* scales, void* y, int y_dtype, int64_t M, int64_t N, int64_t K,
              int32_t* dev_status, void* stream) {
  return mm_call(q_f8, true, sx, qsum, codes, scales, y, y_dtype, M, N, K, 128, dev_status,
                 stream);
}

int pq2_mm_grouped(const uint16_t* q_f16, const float* sx, const int32_t* qsum,
                   const uint8_t* codes, const uint16_t* scales, void* y, int y_dtype, int64_t M,
                   int64_t N, int64_t K, int act_group, int32_t* dev_status, void* stream) {
  return mm_call(q_f16, false, sx, qsum, codes, scales, y, y_dtype, M, N, K, act_group,
                 dev_status, stream);
}

int pq2_mm_f8_grouped(const uint8_t* q_f8, const float* sx, const int32_t* qsum,
                      const uint8_t* codes, const uint16_t* scales, void* y, int y_dtype,
                      int64_t M, int64_t N, int64_t K, int act_group, int32_t* dev_status,
                      void* stream) {
  return mm_call(q_f8, true, sx, qsum, codes, scales, y, y_dtype, M, N, K, act_group,
                 dev_status, stream);
}

// q bytes per element in pq2_linear_grouped's workspace: int8 planes for
// the grouped GEMV (M <= 8), the two e4m3 planes for the prefill GEMM.
static size_t linear_grouped_q_elem(int64_t M) { return M <= 8 ? 1 : 2; }

size_t pq2_linear_grouped_workspace_bytes(int64_t M, int64_t K, int act_group) {
  if (M < 1 || M > kMaxM || !valid_k(K) ||
      (act_group != 128 && act_group != 64 && act_group != 32))
    return 0;
  const size_t GA = (size_t)(K / act_group);
  const size_t q_bytes = (size_t)M * (size_t)K * linear_grouped_q_elem(M);
  const size_t sx_off = (q_bytes + 255) / 256 * 256;
  const size_t qs_off = (sx_off + (size_t)M * GA * 4 + 255) / 256 * 256;
  return qs_off + (size_t)M * GA * 4;
}

int pq2_linear_grouped(const void* x, int x_dtype, int64_t ldx, int64_t M, int64_t N, int64_t K,
                       const uint8_t* codes, const uint16_t* scales, int act_group, void* y,
                       int y_dtype, void* workspace, size_t workspace_bytes,
                       int32_t* dev_status, void* stream) {
  if (!x || !codes || !scales || !y || !workspace) return PQ2_ERR_NULL;
  if (x_dtype != PQ2_BF16 && x_dtype != PQ2_F16 && x_dtype != PQ2_F32) return PQ2_ERR_DTYPE;
  if (y_dtype != PQ2_F32 && y_dtype != PQ2_BF16) return PQ2_ERR_DTYPE;
  const size_t need = pq2_linear_grouped_workspace_bytes(M, K, act_group);
  if (need == 0 || !valid_n(N) || ldx < K || ldx > ((int64_t)1 << 40)) return PQ2_ERR_SHAPE;
  if (workspace_bytes < need) return PQ2_ERR_SHAPE;
  if (!aligned(x, elem_bytes(x_dtype)) || !aligned(workspace, 256) || !aligned(codes, 16) ||
      !aligned(scales, 2) || !aligned(y, elem_bytes(y_dtype)))
    return PQ2_ERR_ALIGN;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  const size_t GA = (size_t)(K / act_group);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t q_bytes = (size_t)M * (size_t)K * linear_grouped_q_elem(M);
  const size_t sx_off = (q_bytes + 255) / 256 * 256;
  const size_t qs_off = (sx_off + (size_t)M * GA * 4 + 255) / 256 * 256;
  float* sx = reinterpret_cast<float*>(ws + sx_off);
  int32_t* qs = reinterpret_cast<int32_t*>(ws + qs_off);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool small = M <= 8;
  if (int st = pq2::launch_quantize(x, x_dtype, ldx, M, K, ws, small ? PQ2_Q_PLANES : PQ2_Q_F8,
                                    sx, qs, s, act_group))
    return st;
  if (!small)
    return pq2::launch_mm(ws, true, sx, qs, codes, scales, y, y_dtype, nullptr, M, N, K, sms,
                          dev_status, s, act_group);
  // The grouped GEMV holds four columns' partial sums: columns 4..M-1 run as
  // a second pass (same bits as one pass).  The first pass streams its
  // weights while the quantisation runs.
  const int8_t* q = reinterpret_cast<const int8_t*>(ws);
  const int64_t first = M < 4 ? M : 4;
  if (int st = pq2::launch_mmv_grouped(q, sx, qs, codes, scales, y, y_dtype, nullptr, first, N,
                                       K, act_group, 1, sms, dev_status, s))
    return st;
  if (M == first) return PQ2_OK;
  return pq2::launch_mmv_grouped(q + 4 * K, sx + 4 * GA, qs + 4 * GA, codes, scales,
                                 static_cast<uint8_t*>(y) + 4 * N * elem_bytes(y_dtype), y_dtype,
                                 nullptr, M - 4, N, K, act_group, 1, sms, dev_status, s);
}

int pq2_debug_group_dots(const void* q, const int32_t* qsum, const uint8_t* codes,
                         int64_t M, int64_t N, int64_t K, int path, int32_t* dots,
                         int32_t* dev_status, void* stream) {
  if (!q || !codes || !dots) return PQ2_ERR_NULL;
  if (path != PQ2_PATH_MMV_ADDXOR && path != PQ2_PATH_MM && path != PQ2_PATH_MMV_PLANES &&
      path != PQ2_PATH_MM_F8 && path != PQ2_PATH_MMV_TC)
    return PQ2_ERR_DTYPE;
  const bool mm = path == PQ2_PATH_MM || path == PQ2_PATH_MM_F8;
  if (path != PQ2_PATH_MMV_ADDXOR && !qsum) return PQ2_ERR_NULL;
  if (!valid_n(N) || !valid_k(K)) return PQ2_ERR_SHAPE;
  if (mm ? (M < 1 || M > kMaxM) : (M < 1 || M > 8)) return PQ2_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(codes, 16) || !aligned(dots, 4) ||
      (qsum && !aligned(qsum, 4)))
    return PQ2_ERR_ALIGN;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (mm)
    return pq2::launch_mm(q, path == PQ2_PATH_MM_F8, nullptr, qsum, codes, nullptr, nullptr,
                          PQ2_F32, dots, M, N, K, sms, dev_status, s);
  // The dot-only variant reads neither scales nor y; sx is unused as well.
  return pq2::launch_mmv(static_cast<const int8_t*>(q), nullptr, qsum, codes, nullptr, nullptr,
                         PQ2_F32, dots, M, N, K,
                         path == PQ2_PATH_MMV_PLANES ? pq2::kDecodeMaskPlanes
                         : path == PQ2_PATH_MMV_TC   ? pq2::kDecodeTensor
                                                     : pq2::kDecodeAddXor,
                         0, sms, dev_status, s);
}

int pq2_debug_mm_dots_grouped(const void* q, int path, const uint8_t* codes, int64_t M,
                              int64_t N, int64_t K, int act_group, int32_t* dots,
                              int32_t* dev_status, void* stream) {
  if (!q || !codes || !dots) return PQ2_ERR_NULL;
  if (path != PQ2_PATH_MM && path != PQ2_PATH_MM_F8) return PQ2_ERR_DTYPE;
  if (M < 1 || M > kMaxM || !valid_n(N) || !valid_k(K) ||
      (act_group != 128 && act_group != 64 && act_group != 32))
    return PQ2_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(codes, 16) || !aligned(dots, 4)) return PQ2_ERR_ALIGN;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  return pq2::launch_mm(q, path == PQ2_PATH_MM_F8, nullptr, nullptr, codes, nullptr, nullptr,
                        PQ2_F32, dots, M, N, K, sms, dev_status,
                        static_cast<cudaStream_t>(stream), act_group);
}

int pq2_debug_mmv_drop_arrival(const int8_t* q, const float* sx, const int32_t* qsum,
                               const uint8_t* codes, const uint16_t* scales, void* y,
                               int y_dtype, int64_t M, int64_t N, int64_t K,
                               int64_t wait_limit_cycles, int32_t* dev_status, void* stream) {
  if (int st = check_mmv_args(q, sx, qsum, codes, scales, y, y_dtype, M, N, K,
                              PQ2_DECODE_PLANES))
    return st;
  if (!dev_status) return PQ2_ERR_NULL;
  if (wait_limit_cycles < 1000 || wait_limit_cycles > (int64_t)1 << 32) return PQ2_ERR_SHAPE;
  if (!aligned(dev_status, 4)) return PQ2_ERR_ALIGN;
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  return pq2::launch_mmv_drop_arrival(q, sx, qsum, codes, scales, y, y_dtype, M, N, K,
                                      (long long)wait_limit_cycles, sms, dev_status,
                                      static_cast<cudaStream_t>(stream));
}

int pq2_mmv_geometry(int64_t N, int64_t K, int sm_count, int* ctas, int* threads,
                     int* splits, int* rows_max) {
  pq2::MmvGeometry g;
  if (!pq2::mmv_geometry(N, K, sm_count, &g)) return PQ2_ERR_SHAPE;
  if (ctas) *ctas = g.ctas;
  if (threads) *threads = g.threads;
  if (splits) *splits = g.splits;
  if (rows_max) *rows_max = g.rows_max;
  return PQ2_OK;
}

}  // extern "C"
