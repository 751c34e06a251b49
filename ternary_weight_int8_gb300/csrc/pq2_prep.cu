// pq2_prep.cu — fused preparation of the activations (sm_103a): RMSNorm,
// random signs, the 1024-point Walsh-Hadamard transform and the group-128
// INT8 quantisation in one kernel, writing q, s_x and sum(q) for the GEMV or
// GEMM.
//
// Method: page "Kernel experiments: recorded evidence" (KE), Test 18
// ("RMSNorm + Hadamard + Q8 fusion"): h = x (+ residual) in fp32; the sum of
// h^2 is kept in 2048 strided partial sums and then summed; inv =
// 1/sqrt(mean + eps); the normalised row (h * inv) * (w + 1) is rounded to
// bf16, multiplied by the signs, transformed per 1024-element block, rounded
// to bf16 again and quantised per 128-group (KE Test 6).  The accepted
// variant of the page matches a fixed reduction structure so that the codes
// are exact; here that structure is: partial i sums h[j]^2 for j = i mod 2048
// in increasing j (fp32), then p[i] += p[i + len] for len = 1024, 512, .., 1.
// inv uses an IEEE square root and an IEEE division; the transform is the
// orthonormal one (butterfly passes of half-width 1, 2, .., 512, then the
// exact factor 1/32).
//
// One CTA (512 threads) per row: the row's h sits in shared memory between
// the two passes; each 1024-block is transformed in shared memory (ten
// butterfly passes) and quantised by eight warps, one 128-group each.
#include <cuda_bf16.h>

#include "pq2_device.cuh"
#include "pq2_internal.h"
#include "pq2_quant.cuh"

namespace pq2 {
namespace {

constexpr int kPrepThreads = 512;
constexpr int kLanes = 2048;  // strided partial sums of h^2
constexpr int kHad = 1024;    // transform block

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float((uint32_t)b << 16);
}
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__global__ void __launch_bounds__(kPrepThreads, 1)
    prep_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ res,
                uint16_t* __restrict__ res_out, const uint16_t* __restrict__ w,
                const int8_t* __restrict__ sign, float eps, int K,
                uint16_t* __restrict__ norm_out, void* __restrict__ q, int layout,
                float* __restrict__ sx, int32_t* __restrict__ qsum) {
  extern __shared__ float sh[];
  float* hs = sh;            // [K]     h = x (+ residual), fp32
  float* vb = sh + K;        // [1024]  the block being transformed
  float* tree = vb + kHad;   // [512]   cross-thread levels of the sum
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t m = blockIdx.x;
  const int G = K / kGroup;
  // Programmatic dependent launch, as the stand-alone quantiser.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // Pass 1: h, the optional residual output, and lanes t + 512k (k = 0..3)
  // of the 2048 strided partial sums of h^2, in increasing j.
  const uint16_t* xr = x + m * K;
  float p[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int base = 0; base < K; base += kLanes) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = base + t + kPrepThreads * k;
      if (j < K) {
        float a = bf16_bits_to_float(xr[j]);
        if (res) a = __fadd_rn(a, bf16_bits_to_float(res[m * K + j]));
        hs[j] = a;
        if (res_out) res_out[m * K + j] = float_to_bf16_bits(a);
        p[k] = __fadd_rn(p[k], __fmul_rn(a, a));
      }
    }
  }
  // p[i] += p[i + len]: len 1024 and 512 inside the thread (lanes t + 512k),
  // 256 .. 32 through shared memory, 16 .. 1 by shuffles in warp 0.
  p[0] = __fadd_rn(p[0], p[2]);
  p[1] = __fadd_rn(p[1], p[3]);
  p[0] = __fadd_rn(p[0], p[1]);
  tree[t] = p[0];
  __syncthreads();
  for (int len = 256; len >= 32; len >>= 1) {
    if (t < len) tree[t] = __fadd_rn(tree[t], tree[t + len]);
    __syncthreads();
  }
  if (warp == 0) {
    float v = tree[lane];
#pragma unroll
    for (int len = 16; len >= 1; len >>= 1) {
      const float o = __shfl_down_sync(0xffffffffu, v, len);
      if (lane < len) v = __fadd_rn(v, o);
    }
    if (lane == 0) tree[0] = v;
  }
  __syncthreads();
  const float mean = __fdiv_rn(tree[0], (float)K);
  const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));

  // Pass 2, block by block: normalise, round to bf16, apply the signs,
  // transform, round to bf16, quantise.
  for (int b = 0; b < K; b += kHad) {
#pragma unroll
    for (int e = t; e < kHad; e += kPrepThreads) {
      const int j = b + e;
      const float tn =
          __fmul_rn(__fmul_rn(hs[j], inv), __fadd_rn(bf16_bits_to_float(w[j]), 1.0f));
      const uint16_t nb = float_to_bf16_bits(tn);
      if (norm_out) norm_out[m * K + j] = nb;
      vb[e] = bf16_bits_to_float(nb) * (float)sign[j];  // exact: the sign is +-1
    }
    __syncthreads();
    for (int h = 1; h < kHad; h <<= 1) {
      const int j = (t / h) * 2 * h + (t % h);  // pair t of this pass
      const float a = vb[j], c = vb[j + h];
      vb[j] = __fadd_rn(a, c);
      vb[j + h] = __fsub_rn(a, c);
      __syncthreads();
    }
#pragma unroll
    for (int e = t; e < kHad; e += kPrepThreads)
      vb[e] = bf16_bits_to_float(float_to_bf16_bits(vb[e] * 0.03125f));  // 1/32: exact
    __syncthreads();
    if (warp < kHad / kGroup) {
      const int gi = b / kGroup + warp;
      float a[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = vb[warp * kGroup + 4 * lane + i];
      int qi[4];
      const float s = quantize_group4(a, qi);
      store_group4(qi, lane, q, layout, m * K + (int64_t)gi * kGroup,
                   qsum ? qsum + m * G + gi : nullptr);
      if (lane == 0) sx[m * G + gi] = s;
    }
    __syncthreads();
  }
}

}  // namespace

int launch_norm_hadamard_quantize(const uint16_t* x, const uint16_t* residual,
                                  uint16_t* residual_out, const uint16_t* w, const int8_t* sign,
                                  float eps, int64_t M, int64_t K, uint16_t* norm_out, void* q,
                                  int q_layout, float* sx, int32_t* qsum, cudaStream_t stream) {
  const int smem = (int)((K + kHad + kPrepThreads) * sizeof(float));
  static int configured = 0;
  if (smem > configured) {
    if (cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess) {
      cudaGetLastError();
      return PQ2_ERR_LAUNCH;
    }
    configured = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)M);
  cfg.blockDim = dim3(kPrepThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, prep_kernel, x, residual, residual_out, w, sign, eps, (int)K,
                         norm_out, q, q_layout, sx, qsum) != cudaSuccess) {
    cudaGetLastError();
    return PQ2_ERR_LAUNCH;
  }
  return PQ2_OK;
}

}  // namespace pq2
