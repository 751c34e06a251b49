// pq2_quantize.cu — weight-plane preparation and per-group INT8 activation
// quantisation (sm_103a).
//
// Preparation: page "Kernel experiments: recorded evidence" (KE), Test 1
// (prepare_pq2, separate buffers) and Test 4 (shared prepared layout).
// Quantisation: KE Test 6 (_quantize) and page "Baseline and the integer
// breakthrough" (BIB), "Calculate with small integers", step 1; plane order
// and group sums: KE Test 21 (plane-order quantisation).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pq2_device.cuh"
#include "pq2_internal.h"
#include "pq2_quant.cuh"

namespace pq2 {
namespace {

// One thread per 34-byte block: bytes 0-1 are the little-endian fp16 scale,
// bytes 2..33 the 32 code bytes (weight k in bits 2(k%4) of byte k/4).
// Raw rows have an arbitrary byte stride, so the block is read bytewise; the
// code plane row is 16-byte aligned and written with two 16-byte stores.
__global__ void prepare_kernel(const uint8_t* __restrict__ raw,
                               int64_t raw_stride, int64_t N, int G,
                               uint8_t* __restrict__ codes,
                               uint16_t* __restrict__ scales) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= N * G) return;
  const int64_t n = idx / G;
  const int g = (int)(idx % G);
  const uint8_t* b = raw + n * raw_stride + (int64_t)g * 34;
  scales[idx] = (uint16_t)(b[0] | (b[1] << 8));
  uint32_t w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
    w[j] = (uint32_t)b[2 + 4 * j] | ((uint32_t)b[3 + 4 * j] << 8) |
           ((uint32_t)b[4 + 4 * j] << 16) | ((uint32_t)b[5 + 4 * j] << 24);
  uint4* dst = reinterpret_cast<uint4*>(codes + n * (int64_t)G * 32 +
                                        (int64_t)g * 32);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

template <int XT>
__device__ __forceinline__ float to_f32(const void* x, int64_t i);
template <>
__device__ __forceinline__ float to_f32<PQ2_BF16>(const void* x, int64_t i) {
  return __bfloat162float(static_cast<const __nv_bfloat16*>(x)[i]);
}
template <>
__device__ __forceinline__ float to_f32<PQ2_F16>(const void* x, int64_t i) {
  return __half2float(static_cast<const __half*>(x)[i]);
}
template <>
__device__ __forceinline__ float to_f32<PQ2_F32>(const void* x, int64_t i) {
  return static_cast<const float*>(x)[i];
}

// Four consecutive activations starting at element i (i % 4 == 0).  With
// `vec` the four are fetched with one 8-byte (16-bit types) or 16-byte (fp32)
// load; the host sets it only when base and row stride allow it.
template <int XT>
__device__ __forceinline__ void load4(const void* x, int64_t i, bool vec,
                                      float a[4]) {
  if (vec) {
    if (XT == PQ2_F32) {
      const float4 v = *reinterpret_cast<const float4*>(
          static_cast<const float*>(x) + i);
      a[0] = v.x; a[1] = v.y; a[2] = v.z; a[3] = v.w;
    } else {
      const uint2 v = *reinterpret_cast<const uint2*>(
          static_cast<const uint16_t*>(x) + i);
      const uint16_t h[4] = {(uint16_t)(v.x & 0xffff), (uint16_t)(v.x >> 16),
                             (uint16_t)(v.y & 0xffff), (uint16_t)(v.y >> 16)};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (XT == PQ2_BF16)
          a[j] = __uint_as_float((uint32_t)h[j] << 16);
        else
          a[j] = __half2float(__ushort_as_half(h[j]));
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) a[j] = to_f32<XT>(x, i + j);
  }
}

// One warp per (row m, 128-group g); lane L owns elements 4L..4L+3 of the
// group (quantize_group4 / store_group4), in activation groups of 4 * LANES
// elements: sx and qsum are [M][K / (4 * LANES)].
template <int XT, int LANES>
__global__ void __launch_bounds__(256) quantize_kernel(
    const void* __restrict__ x, int64_t ldx, int64_t M, int G, bool vec,
    void* __restrict__ q, int layout, float* __restrict__ sx,
    int32_t* __restrict__ qsum) {
  // Launched with programmatic dependent launch: let the next kernel start
  // its independent prologue now (it waits for this grid before it reads q,
  // s_x or sum(q)), and wait for the previous grid before touching memory.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= M * G) return;
  const int64_t m = warp / G;
  const int g = (int)(warp % G);
  const int64_t K = (int64_t)G * kGroup;

  float a[4];
  load4<XT>(x, m * ldx + (int64_t)g * kGroup + 4 * lane, vec, a);
  constexpr int NSUB = 32 / LANES;  // activation groups per 128-group
  int qi[4];
  const float s = quantize_group4<LANES>(a, qi);
  store_group4<LANES>(qi, lane, q, layout, m * K + (int64_t)g * kGroup,
                      qsum ? qsum + (m * G + g) * NSUB : nullptr);
  if (lane % LANES == 0) sx[(m * G + g) * NSUB + lane / LANES] = s;
}

// Many rows: eight lanes per (row m, 128-group g), four consecutive groups
// of the row-major group index per warp (quantize_group16 / store_group16);
// lane j = L % 8 loads its group's elements 16j..16j+15 with 16-byte loads
// (the host guarantees the alignment).  The same bytes as quantize_kernel, in
// about a quarter of its instructions per group.  Not for PQ2_Q_MMV16.
template <int XT, int LG>
__global__ void __launch_bounds__(256) quantize16_kernel(
    const void* __restrict__ x, int64_t ldx, int64_t M, int G, void* __restrict__ q, int layout,
    float* __restrict__ sx, int32_t* __restrict__ qsum) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31, j = lane & 7;
  const int64_t total = M * G;
  if (warp * 4 >= total) return;  // the whole warp leaves together
  const int64_t gi = warp * 4 + (lane >> 3);
  const bool valid = gi < total;  // a ragged last warp keeps its lanes for the shuffles
  const int64_t m = valid ? gi / G : 0;
  const int g = valid ? (int)(gi - m * G) : 0;
  const int64_t K = (int64_t)G * kGroup;
  constexpr int NSUB = 8 / LG;  // activation groups per 128-group
  float a[16];
  if (XT == PQ2_F32) {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(x) + m * ldx +
                                                        (int64_t)g * kGroup + 16 * j);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 v = valid ? src[k] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      a[4 * k] = v.x; a[4 * k + 1] = v.y; a[4 * k + 2] = v.z; a[4 * k + 3] = v.w;
    }
  } else {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + m * ldx +
                                                      (int64_t)g * kGroup + 16 * j);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint4 v = valid ? src[k] : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint16_t h = (uint16_t)(w[e >> 1] >> (16 * (e & 1)));
        a[8 * k + e] = XT == PQ2_BF16 ? __uint_as_float((uint32_t)h << 16)
                                      : __half2float(__ushort_as_half(h));
      }
    }
  }
  int qi[16];
  const float s = quantize_group16<LG>(a, qi);
  store_group16<LG>(qi, j, valid, q, layout, m * K + (int64_t)g * kGroup,
                    qsum ? qsum + gi * NSUB : nullptr);
  if (valid && j % LG == 0) sx[gi * NSUB + j / LG] = s;
}

}  // namespace

int launch_prepare(const uint8_t* raw, int64_t raw_stride, int64_t N,
                   int64_t K, uint8_t* codes, uint16_t* scales,
                   cudaStream_t stream) {
  const int G = (int)(K / kGroup);
  const int64_t blocks_needed = (N * G + 255) / 256;
  prepare_kernel<<<(unsigned)blocks_needed, 256, 0, stream>>>(
      raw, raw_stride, N, G, codes, scales);
  return cudaGetLastError() == cudaSuccess ? PQ2_OK : PQ2_ERR_LAUNCH;
}

namespace {

template <int XT>
cudaError_t launch_quantize_xt(const cudaLaunchConfig_t& cfg, int act_group, const void* x,
                               int64_t ldx, int64_t M, int G, bool vec, void* q, int q_layout,
                               float* sx, int32_t* qsum) {
  switch (act_group) {
    case 64:
      return cudaLaunchKernelEx(&cfg, quantize_kernel<XT, 16>, x, ldx, M, G, vec, q, q_layout, sx,
                                qsum);
    case 32:
      return cudaLaunchKernelEx(&cfg, quantize_kernel<XT, 8>, x, ldx, M, G, vec, q, q_layout, sx,
                                qsum);
    default:
      return cudaLaunchKernelEx(&cfg, quantize_kernel<XT, 32>, x, ldx, M, G, vec, q, q_layout, sx,
                                qsum);
  }
}

// Groups from which the eight-lanes-per-group kernel runs (M >= 410 at
// K = 5120): with fewer groups, one warp per group keeps more loads in
// flight (measured faster at M = 128 and 256), and the few-row (decode)
// calls keep that kernel.
constexpr int64_t kQuant16Groups = 16384;

template <int XT>
cudaError_t launch_quantize16_xt(const cudaLaunchConfig_t& cfg, int lg, const void* x,
                                 int64_t ldx, int64_t M, int G, void* q, int q_layout, float* sx,
                                 int32_t* qsum) {
  switch (lg) {
    case 4:
      return cudaLaunchKernelEx(&cfg, quantize16_kernel<XT, 4>, x, ldx, M, G, q, q_layout, sx,
                                qsum);
    case 2:
      return cudaLaunchKernelEx(&cfg, quantize16_kernel<XT, 2>, x, ldx, M, G, q, q_layout, sx,
                                qsum);
    default:
      return cudaLaunchKernelEx(&cfg, quantize16_kernel<XT, 8>, x, ldx, M, G, q, q_layout, sx,
                                qsum);
  }
}

}  // namespace

int launch_quantize(const void* x, int x_dtype, int64_t ldx, int64_t M,
                    int64_t K, void* q, int q_layout, float* sx, int32_t* qsum,
                    cudaStream_t stream, int act_group) {
  const int G = (int)(K / kGroup);
  const int elem = x_dtype == PQ2_F32 ? 4 : 2;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(x);
  const bool vec = (addr % (4 * elem) == 0) && (ldx % 4 == 0);
  // Many rows (at least kQuant16Groups groups): eight lanes per group, when
  // the layout allows it and every group's elements start on 16 bytes.
  const bool wide = M * G >= kQuant16Groups && q_layout != PQ2_Q_MMV16 && addr % 16 == 0 &&
                    (ldx * elem) % 16 == 0 && reinterpret_cast<uintptr_t>(q) % 16 == 0;
  if (wide) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((M * G + 31) / 32));  // 8 warps x 4 groups per block
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int lg = act_group / 16;
    cudaError_t e;
    switch (x_dtype) {
      case PQ2_BF16: e = launch_quantize16_xt<PQ2_BF16>(cfg, lg, x, ldx, M, G, q, q_layout, sx, qsum); break;
      case PQ2_F16: e = launch_quantize16_xt<PQ2_F16>(cfg, lg, x, ldx, M, G, q, q_layout, sx, qsum); break;
      default: e = launch_quantize16_xt<PQ2_F32>(cfg, lg, x, ldx, M, G, q, q_layout, sx, qsum); break;
    }
    if (e != cudaSuccess) {
      cudaGetLastError();
      return PQ2_ERR_LAUNCH;
    }
    return PQ2_OK;
  }
  const int64_t warps = M * G;
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  switch (x_dtype) {
    case PQ2_BF16:
      e = launch_quantize_xt<PQ2_BF16>(cfg, act_group, x, ldx, M, G, vec, q, q_layout, sx, qsum);
      break;
    case PQ2_F16:
      e = launch_quantize_xt<PQ2_F16>(cfg, act_group, x, ldx, M, G, vec, q, q_layout, sx, qsum);
      break;
    default:
      e = launch_quantize_xt<PQ2_F32>(cfg, act_group, x, ldx, M, G, vec, q, q_layout, sx, qsum);
      break;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PQ2_ERR_LAUNCH;
  }
  return PQ2_OK;
}

}  // namespace pq2
