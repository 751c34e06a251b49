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
// Rows of up to eight 1024-blocks: one cluster of CTAs per row (below).
// Longer rows: one CTA per row (256 threads, four per SM, for many rows; 1024
// threads for few rows, where one row's latency counts): the row's h sits in shared
// memory between the passes.  With 1024 threads, 64 threads form the sum of
// squares (levels 1024..64 of its tree inside a thread) and up to four warps
// share each 1024-block of the transform; otherwise each warp owns whole
// 1024-blocks: lane l holds elements 32i + l (i = 0..31) in registers, so
// the passes of half-width 1..16 are shuffles between lanes and those of
// 32..512 are butterflies inside a lane, with no block-wide barrier; the
// rounded block is written back over its h.  Then all the warps share the row's
// 128-groups (each a latency chain of shuffles), in the quantiser's lane
// layout (elements 4l..4l+3 of a group per lane).
#include <cuda_bf16.h>

#include "pq2_device.cuh"
#include "pq2_internal.h"
#include "pq2_quant.cuh"

namespace pq2 {
namespace {

constexpr int kLanes = 2048;  // strided partial sums of h^2
constexpr int kHad = 1024;    // transform block

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float((uint32_t)b << 16);
}
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
// Two roundings to bf16 in one conversion instruction (each half rounded to
// nearest even, as float_to_bf16_bits): a in the low half, b in the high.
__device__ __forceinline__ uint32_t float2_to_bf16x2_bits(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// The bf16 value with bits b times the sign +1 / -1 held in the int8 s:
// exact, so a flip of the sign bit.
__device__ __forceinline__ float bf16_signed(uint16_t b, int8_t s) {
  return __uint_as_float(((uint32_t)b << 16) ^ (((uint32_t)(uint8_t)s & 0x80u) << 24));
}
// One butterfly half: the lower lane of a pair keeps a + o, the upper o - a.
// With sgn = +1 / -1, fma(a, sgn, o) rounds a * sgn + o once and a * sgn is
// exact, so it equals __fadd_rn(a, o) / __fsub_rn(o, a), signed zeros
// included, in one instruction instead of a select between two.
__device__ __forceinline__ float butterfly(float a, float o, float sgn) {
  return __fmaf_rn(a, sgn, o);
}
// Packed pairs of fp32 (element 0 in the low half): one instruction, two
// IEEE round-to-nearest results, the same as two scalar operations.
__device__ __forceinline__ void add_sub_f32x2(float& a0, float& a1, float& c0, float& c1) {
  uint64_t a = ((uint64_t)__float_as_uint(a1) << 32) | __float_as_uint(a0);
  uint64_t c = ((uint64_t)__float_as_uint(c1) << 32) | __float_as_uint(c0);
  uint64_t sum, dif;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(sum) : "l"(a), "l"(c));
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(dif) : "l"(a), "l"(c));
  a0 = __uint_as_float((uint32_t)sum);
  a1 = __uint_as_float((uint32_t)(sum >> 32));
  c0 = __uint_as_float((uint32_t)dif);
  c1 = __uint_as_float((uint32_t)(dif >> 32));
}

// The transform of every 1024-block of a row by W warps per block (W = 2, 4
// or 8): warp u of block b holds the elements b + (1024/W) u + 32 i + l,
// i < 32/W, of lane l.  Passes of half-width 1..16 are shuffles, those up to
// 512/W pair registers of a lane, and the last log2(W) passes pair elements
// of two warps through shared memory (the block's h, already read), in the
// order 1, 2, .., 512 of the single-warp transform, so the bits are the
// same.  Every warp of the CTA reaches the same barriers.
// The norm weights (bf16 bits, two per word) and signs (bytes, four per
// word) of a lane's elements in the transform_shared layout for W = 2, 4, 8,
// loaded at kernel entry so that their latency overlaps the first pass.
struct TransformOperands {
  uint32_t wb[8];
  uint32_t sb[4];
};

template <int W>
__device__ __forceinline__ void load_transform_operands(const uint16_t* __restrict__ w,
                                                        const int8_t* __restrict__ sign, int nblk,
                                                        int warp, int lane, TransformOperands& o) {
  constexpr int E = 32 / W, kSpan = kHad / W;
  if (warp >= nblk * W) return;
  const int base = (warp / W) * kHad + kSpan * (warp % W);
#pragma unroll
  for (int i = 0; i < E; i += 2)
    o.wb[i / 2] = (uint32_t)w[base + 32 * i + lane] | ((uint32_t)w[base + 32 * (i + 1) + lane] << 16);
#pragma unroll
  for (int i = 0; i < E; i += 4) {
    uint32_t v = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) v |= (uint32_t)(uint8_t)sign[base + 32 * (i + e) + lane] << (8 * e);
    o.sb[i / 4] = v;
  }
}

template <int W, int kWarps>
__device__ __forceinline__ void transform_shared(float* hs, const TransformOperands& o,
                                                 float inv, uint16_t* __restrict__ norm_out,
                                                 int64_t m, int K, int nblk, int warp, int lane) {
  constexpr int E = 32 / W;           // registers per lane
  constexpr int kSpan = kHad / W;     // elements per warp
  const bool busy = warp < nblk * W;  // nblk * W <= kWarps
  const int b = (warp / W) * kHad, u = warp % W;
  const int base = b + kSpan * u;
  float r[E];
  if (busy) {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const int j = base + 32 * i + lane;
      const float w1 = __fadd_rn(bf16_bits_to_float((uint16_t)(o.wb[i / 2] >> (16 * (i & 1)))), 1.0f);
      const int8_t sg = (int8_t)(uint8_t)(o.sb[i / 4] >> (8 * (i & 3)));
      const float tn = __fmul_rn(__fmul_rn(hs[j], inv), w1);
      const uint16_t nb = float_to_bf16_bits(tn);
      if (norm_out) norm_out[m * K + j] = nb;
      r[i] = bf16_signed(nb, sg);  // exact: the sign is +-1
    }
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
      const float sgn = (lane & h) ? -1.0f : 1.0f;
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const float o = __shfl_xor_sync(0xffffffffu, r[i], h);
        r[i] = butterfly(r[i], o, sgn);
      }
    }
#pragma unroll
    for (int d = 1; d < E; d <<= 1) {
#pragma unroll
      for (int i = 0; i < E; ++i) {
        if (i & d) continue;
        const float a = r[i], c = r[i + d];
        r[i] = __fadd_rn(a, c);
        r[i + d] = __fsub_rn(a, c);
      }
    }
  }
  // half-widths kSpan .. 512: warp u pairs with warp u ^ (h / kSpan)
#pragma unroll
  for (int hw = 1; hw < W; hw <<= 1) {
    __syncthreads();  // every warp has read its h (first round) or its partner's values
    if (busy) {
#pragma unroll
      for (int i = 0; i < E; ++i) hs[base + 32 * i + lane] = r[i];
    }
    __syncthreads();
    if (busy) {
      const bool upper = (u & hw) != 0;
      const int pbase = b + kSpan * (u ^ hw);
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const float o = hs[pbase + 32 * i + lane];
        r[i] = upper ? __fsub_rn(o, r[i]) : __fadd_rn(r[i], o);
      }
    }
  }
  __syncthreads();  // partners have read the exchanged values
  if (busy) {
#pragma unroll
    for (int i = 0; i < E; ++i)  // 1/32 is exact
      hs[base + 32 * i + lane] = bf16_bits_to_float(float_to_bf16_bits(r[i] * 0.03125f));
  }
}

// kPrepThreads threads per row: 1024 when few rows run (the latency of one
// row: more warps share its 128-groups), 256 for many rows (four CTAs per
// SM).  The thread count changes which thread holds which of the 2048 lanes,
// never the order of an operation.
template <int kPrepThreads>
__global__ void __launch_bounds__(kPrepThreads, kPrepThreads == 256 ? 4 : 1)
    prep_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ res,
                uint16_t* __restrict__ res_out, const uint16_t* __restrict__ w,
                const int8_t* __restrict__ sign, float eps, int K, int vec, int fused_arg,
                uint16_t* __restrict__ norm_out, void* __restrict__ q, int layout,
                float* __restrict__ sx, int32_t* __restrict__ qsum) {
  extern __shared__ float sh[];
  // Many rows (256 threads): each warp transforms and quantises its 1024-blocks
  // in registers, 32 consecutive elements per lane (below), and h is stored
  // with its 4-element chunks swizzled so that those reads are free of bank
  // conflicts: element e sits at hpos(e).  The host sets fused_arg when the
  // layout and alignments allow it.
  const bool fused = kPrepThreads == 256 && fused_arg != 0;
  auto hpos = [&](int e) {
    return fused ? 32 * (e >> 5) + 4 * (((e >> 2) & 7) ^ ((e >> 5) & 7)) + (e & 3) : e;
  };
  float* hs = sh;          // [K]    h = x (+ residual), then the transformed row
  float* tree = sh + K;    // [512]  cross-thread levels of the sum
  constexpr int kPrepWarps = kPrepThreads / 32;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t m = blockIdx.x;
  const int G = K / kGroup;
  // Programmatic dependent launch, as the stand-alone quantiser.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // Latency variant: the transform's norm weights and signs go out first.
  const int nblk = K / kHad;
  const int W = kPrepThreads == 1024 ? (nblk <= 8 ? 4 : nblk <= 16 ? 2 : 1) : 1;
  TransformOperands ops;
  if (W == 4) load_transform_operands<4>(w, sign, nblk, warp, lane, ops);
  if (W == 2) load_transform_operands<2>(w, sign, nblk, warp, lane, ops);

  // Pass 1a: h = x (+ residual) into shared memory, and the optional
  // residual output.  With 16-byte aligned rows the loads (eight bf16 each)
  // go out four per thread at a time before any is used (all of them for
  // K <= 8192); else element by element.
  const uint16_t* xr = x + m * K;
  if (vec) {
    constexpr int kBatch = 4;
    const int chunks = K / 8;
    for (int c0 = 0; c0 < chunks; c0 += kBatch * kPrepThreads) {
      uint4 xv[kBatch], rv[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int c = c0 + t + kPrepThreads * u;
        if (c < chunks) {
          xv[u] = reinterpret_cast<const uint4*>(xr)[c];
          if (res) rv[u] = reinterpret_cast<const uint4*>(res + m * K)[c];
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int c = c0 + t + kPrepThreads * u;
        if (c < chunks) {
          const uint32_t xw[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
          const uint32_t rw[4] = {rv[u].x, rv[u].y, rv[u].z, rv[u].w};
          float h8[8];
          uint32_t ob[4];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint16_t xb = (uint16_t)(xw[e >> 1] >> (16 * (e & 1)));
            float a = bf16_bits_to_float(xb);
            if (res) a = __fadd_rn(a, bf16_bits_to_float((uint16_t)(rw[e >> 1] >> (16 * (e & 1)))));
            h8[e] = a;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) ob[e] = float2_to_bf16x2_bits(h8[2 * e], h8[2 * e + 1]);
          *reinterpret_cast<float4*>(hs + hpos(8 * c)) = make_float4(h8[0], h8[1], h8[2], h8[3]);
          *reinterpret_cast<float4*>(hs + hpos(8 * c + 4)) =
              make_float4(h8[4], h8[5], h8[6], h8[7]);
          if (res_out)
            reinterpret_cast<uint4*>(res_out + m * K)[c] = make_uint4(ob[0], ob[1], ob[2], ob[3]);
        }
      }
    }
  } else {
    for (int j = t; j < K; j += kPrepThreads) {
      float a = bf16_bits_to_float(xr[j]);
      if (res) a = __fadd_rn(a, bf16_bits_to_float(res[m * K + j]));
      hs[hpos(j)] = a;
      if (res_out) res_out[m * K + j] = float_to_bf16_bits(a);
    }
  }
  __syncthreads();
  if constexpr (kPrepThreads == 1024) {
    // Pass 1b, latency variant: 64 threads own the lanes i, i + 64, ..,
    // i + 1984 of the 2048 strided partial sums (i = t), so the levels
    // len = 1024 .. 64 of the tree pair two lanes of one thread; level 32
    // goes through shared memory and 16 .. 1 by shuffles in warp 0.
    if (t < 64) {
      float p[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) p[k] = 0.0f;
      for (int base = 0; base < K; base += kLanes) {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int j = base + t + 64 * k;
          if (j < K) p[k] = __fadd_rn(p[k], __fmul_rn(hs[j], hs[j]));
        }
      }
      // lane t + 64k pairs with lane t + 64(k + step) at level 64 * step
#pragma unroll
      for (int step = 16; step >= 1; step >>= 1)
#pragma unroll
        for (int k = 0; k < step; ++k) p[k] = __fadd_rn(p[k], p[k + step]);
      if (t >= 32) tree[t] = p[0];
      tree[64 + t] = p[0];
    }
    __syncthreads();
    if (warp == 0) {
      float v = __fadd_rn(tree[64 + lane], tree[lane + 32]);  // level 32
#pragma unroll
      for (int len = 16; len >= 1; len >>= 1) {
        const float o = __shfl_down_sync(0xffffffffu, v, len);
        if (lane < len) v = __fadd_rn(v, o);
      }
      if (lane == 0) tree[0] = v;
    }
    __syncthreads();
  } else {
    // Pass 1b: lanes t + kPrepThreads * k of the 2048 strided partial sums of
    // h^2, each in increasing j (slices of 2048 outside, the thread's lanes
    // inside, so a slice's loads go out together).
    constexpr int kPer = kLanes / kPrepThreads;
    float p[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) p[k] = 0.0f;
    // Every j this thread reads has the same chunk and row bits below 2^8,
    // so its swizzled position is j plus one offset.
    const int dj = hpos(t) - t;
    for (int base = 0; base < K; base += kLanes) {
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int j = base + t + kPrepThreads * k;
        if (j < K) {
          const float v = hs[j + dj];
          p[k] = __fadd_rn(p[k], __fmul_rn(v, v));
        }
      }
    }
    // p[i] += p[i + len]: len 1024 .. kPrepThreads inside the thread (lane
    // t + kPrepThreads * k pairs with k + kPer/2, then k + kPer/4, ..), the
    // levels below kPrepThreads down to 32 through shared memory, 16 .. 1 by
    // shuffles in warp 0.
#pragma unroll
    for (int step = kPer / 2; step >= 1; step >>= 1)
#pragma unroll
      for (int k = 0; k < step; ++k) p[k] = __fadd_rn(p[k], p[k + step]);
    tree[t] = p[0];
    __syncthreads();
    for (int len = kPrepThreads / 2; len >= 32; len >>= 1) {
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
  }
  const float mean = __fdiv_rn(tree[0], (float)K);
  const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));

  // Pass 2: normalise, round to bf16, apply the signs, transform, round to
  // bf16, and store the block back.
  // Warps per 1024-block (W, chosen at entry): up to four in the latency
  // variant (each lane then holds 8 of the block's values, and the passes of
  // half-width 256 and 512 exchange halves through shared memory), one
  // otherwise.
  if (W == 4) {
    transform_shared<4, kPrepWarps>(hs, ops, inv, norm_out, m, K, nblk, warp, lane);
    __syncthreads();
  } else if (W == 2) {
    transform_shared<2, kPrepWarps>(hs, ops, inv, norm_out, m, K, nblk, warp, lane);
    __syncthreads();
  } else if (fused) {
    // Passes 2 and 3 together, one 1024-block per warp at a time, with no
    // block-wide barrier: lane l holds the block's elements 32l + i
    // (i = 0..31), so the transform's passes of half-width 1..16 pair
    // registers of one lane.  A transpose through the block's own shared
    // memory gives lane l the elements 32i + l for the passes of half-width
    // 32..512 (again registers of one lane), and a second one brings the
    // rounded block back to 32 consecutive elements per lane: a quarter of a
    // 128-group, quantised by four lanes.  Every operation and its order are
    // those of the other paths.
    for (int b = warp * kHad; b < K; b += kPrepWarps * kHad) {
      float* blk = hs + b;
      const int sw = lane & 7;  // the lane's chunk swizzle (row 32 * lane)
      float r[32];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float4 v = *reinterpret_cast<const float4*>(blk + 32 * lane + 4 * (k ^ sw));
        r[4 * k] = v.x; r[4 * k + 1] = v.y; r[4 * k + 2] = v.z; r[4 * k + 3] = v.w;
      }
      // Normalise, round to bf16 and apply the signs, eight elements per
      // 16-byte load of norm weights (and 8-byte load of signs).
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 wq = __ldg(reinterpret_cast<const uint4*>(w + b + 32 * lane) + k);
        const uint2 sq = __ldg(reinterpret_cast<const uint2*>(sign + b + 32 * lane) + k);
        const uint32_t wv[4] = {wq.x, wq.y, wq.z, wq.w};
        const uint32_t sv[2] = {sq.x, sq.y};
        uint32_t nb2[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          const int i = 8 * k + 2 * e2;
          const uint32_t wp2 = wv[e2];  // norm weights of elements i, i + 1
          const float tn0 =
              __fmul_rn(__fmul_rn(r[i], inv), __fadd_rn(__uint_as_float(wp2 << 16), 1.0f));
          const float tn1 = __fmul_rn(__fmul_rn(r[i + 1], inv),
                                      __fadd_rn(__uint_as_float(wp2 & 0xffff0000u), 1.0f));
          nb2[e2] = float2_to_bf16x2_bits(tn0, tn1);
          // The signs of elements i and i + 1 (bytes 2 (e2 & 1), + 1 of a
          // sign word) flip bits 15 and 31 of the pair: exact.
          const uint32_t sw2 = sv[e2 >> 1] >> (16 * (e2 & 1));
          const uint32_t v = nb2[e2] ^ (((sw2 & 0x80u) << 8) | ((sw2 & 0x8000u) << 16));
          r[i] = __uint_as_float(v << 16);
          r[i + 1] = __uint_as_float(v & 0xffff0000u);
        }
        if (norm_out)
          reinterpret_cast<uint4*>(norm_out + m * K + b + 32 * lane)[k] =
              make_uint4(nb2[0], nb2[1], nb2[2], nb2[3]);
      }
      // Half-width 1 (registers i, i + 1), then 2..16 on packed pairs.
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float a = r[i], c = r[i + 1];
        r[i] = __fadd_rn(a, c);
        r[i + 1] = __fsub_rn(a, c);
      }
#pragma unroll
      for (int d = 2; d < 32; d <<= 1) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          if (i & d) continue;
          add_sub_f32x2(r[i], r[i + 1], r[i + d], r[i + d + 1]);
        }
      }
      // Transpose: element 32i + l to lane l, register i.  Element e sits at
      // hpos(e) - b: with row 32 * (e >> 5) and chunk (e >> 2) & 7, each
      // access below touches 32 different banks.
      __syncwarp();
#pragma unroll
      for (int k = 0; k < 8; ++k)
        *reinterpret_cast<float4*>(blk + 32 * lane + 4 * (k ^ sw)) =
            make_float4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = blk[32 * i + 4 * ((lane >> 2) ^ (i & 7)) + (lane & 3)];
      // Half-width 32 (registers i, i + 1), then 64..512 on packed pairs.
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float a = r[i], c = r[i + 1];
        r[i] = __fadd_rn(a, c);
        r[i + 1] = __fsub_rn(a, c);
      }
#pragma unroll
      for (int d = 2; d < 32; d <<= 1) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          if (i & d) continue;
          add_sub_f32x2(r[i], r[i + 1], r[i + d], r[i + d + 1]);
        }
      }
#pragma unroll
      for (int i = 0; i < 32; i += 2) {  // 1/32 is exact; two bf16 roundings at once
        const uint32_t v = float2_to_bf16x2_bits(r[i] * 0.03125f, r[i + 1] * 0.03125f);
        r[i] = __uint_as_float(v << 16);
        r[i + 1] = __uint_as_float(v & 0xffff0000u);
      }
      // Back to 32 consecutive elements per lane.
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 32; ++i) blk[32 * i + 4 * ((lane >> 2) ^ (i & 7)) + (lane & 3)] = r[i];
      __syncwarp();
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float4 v = *reinterpret_cast<const float4*>(blk + 32 * lane + 4 * (k ^ sw));
        r[4 * k] = v.x; r[4 * k + 1] = v.y; r[4 * k + 2] = v.z; r[4 * k + 3] = v.w;
      }
      // Lane j = l % 4 of group b / 128 + l / 4 holds its elements 32j..32j+31,
      // its chunks 2j and 2j + 1, quantised and stored one chunk at a time.
      const GroupScale z = quantize_scale32(r);
      const int gi = b / kGroup + (lane >> 2);
      const int64_t gbase = m * K + (int64_t)gi * kGroup;
      int tsum = 0;
      if (!z.exact) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          int qh[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            qh[e] = quantize_product(r[16 * hf + e], z.inv);
            tsum += qh[e];
          }
          store_chunk16(qh, 2 * (lane & 3) + hf, q, layout, gbase);
        }
      } else {
        // Some group of the warp has a near tie (rare, warp-uniform): the
        // IEEE divisions, on the values the block's shared memory still
        // holds (so the registers above need not live through this path).
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          int qh[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int i = 16 * hf + e;
            const float a = blk[32 * lane + 4 * ((i >> 2) ^ sw) + (i & 3)];
            qh[e] = quantize_clamp(rintf(__fdiv_rn(a, z.d)));
            tsum += qh[e];
          }
          store_chunk16(qh, 2 * (lane & 3) + hf, q, layout, gbase);
        }
      }
#pragma unroll
      for (int off = 2; off > 0; off >>= 1) tsum += __shfl_xor_sync(0xffffffffu, tsum, off);
      if ((lane & 3) == 0) {
        sx[m * G + gi] = z.s;
        if (qsum) qsum[m * G + gi] = tsum;
      }
    }
    return;
  } else {
    // Pass 2, one 1024-block per warp at a time: normalise, round to bf16,
    // apply the signs, transform, round to bf16, and store the block back.
    for (int b = warp * kHad; b < K; b += kPrepWarps * kHad) {
      float r[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int j = b + 32 * i + lane;
        const float tn =
            __fmul_rn(__fmul_rn(hs[j], inv), __fadd_rn(bf16_bits_to_float(w[j]), 1.0f));
        const uint16_t nb = float_to_bf16_bits(tn);
        if (norm_out) norm_out[m * K + j] = nb;
        r[i] = bf16_signed(nb, sign[j]);  // exact: the sign is +-1
      }
      // Passes of half-width 1..16 pair lanes l and l ^ h (the lower lane of a
      // pair keeps a + c, the upper a - c) ...
#pragma unroll
      for (int h = 1; h < 32; h <<= 1) {
        const float sgn = (lane & h) ? -1.0f : 1.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float o = __shfl_xor_sync(0xffffffffu, r[i], h);
          r[i] = butterfly(r[i], o, sgn);
        }
      }
      // ... those of 32..512 pair registers i and i + h/32 of one lane
      // (half-width 64 and up on packed pairs of registers).
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float a = r[i], c = r[i + 1];
        r[i] = __fadd_rn(a, c);
        r[i + 1] = __fsub_rn(a, c);
      }
#pragma unroll
      for (int d = 2; d < 32; d <<= 1) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          if (i & d) continue;
          add_sub_f32x2(r[i], r[i + 1], r[i + d], r[i + d + 1]);
        }
      }
#pragma unroll
      for (int i = 0; i < 32; ++i)  // 1/32 is exact; the warp has read all of its h
        hs[b + 32 * i + lane] = bf16_bits_to_float(float_to_bf16_bits(r[i] * 0.03125f));
    }
    __syncthreads();
  }
  // Pass 3: the row's 128-groups shared by all warps, four per warp with
  // eight lanes per group (lane j holds elements 16j..16j+15) where the
  // layout allows it: a quarter of the warp instructions per group of one
  // group per warp, which is kept for the tensor-core GEMV's layout.
  if (layout != PQ2_Q_MMV16 && (reinterpret_cast<uintptr_t>(q) & 15) == 0) {
    const int j = lane & 7;
    for (int g4 = 4 * warp; g4 < G; g4 += 4 * kPrepWarps) {
      const int gi = g4 + (lane >> 3);
      const bool valid = gi < G;  // lanes past the row keep the warp's shuffles
      const float4* src =
          reinterpret_cast<const float4*>(hs + (valid ? gi : 0) * kGroup + 16 * j);
      float a[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 v = src[k];
        a[4 * k] = v.x; a[4 * k + 1] = v.y; a[4 * k + 2] = v.z; a[4 * k + 3] = v.w;
      }
      int qi[16];
      const float s = quantize_group16<8>(a, qi);
      store_group16<8>(qi, j, valid, q, layout, m * K + (int64_t)gi * kGroup,
                       qsum ? qsum + m * G + gi : nullptr);
      if (valid && j == 0) sx[m * G + gi] = s;
    }
  } else {
    for (int gi = warp; gi < G; gi += kPrepWarps) {
      const float4 v4 = *reinterpret_cast<const float4*>(hs + gi * kGroup + 4 * lane);
      const float a[4] = {v4.x, v4.y, v4.z, v4.w};
      int qi[4];
      const float s = quantize_group4(a, qi);
      store_group4(qi, lane, q, layout, m * K + (int64_t)gi * kGroup,
                   qsum ? qsum + m * G + gi : nullptr);
      if (lane == 0) sx[m * G + gi] = s;
    }
  }
}

// ---------------------------------------------------------------- clusters
// A row of K = 1024 C elements (C <= 8) spread over a cluster of C CTAs, CTA
// c owning the transform block [1024c, 1024c + 1024): the load, the
// transform and the quantisation of a row then run on C SMs at once.  Every
// CTA writes h^2 of its block to its shared memory, and after one cluster
// barrier forms the whole 2048-lane reduction tree itself from the cluster's
// squares (distributed shared memory), in the order of the one-CTA kernel
// with 256 threads, so every CTA holds the same bits of inv.

constexpr int kClusterThreads = 256;  // 8 warps: one per group of a block
constexpr int64_t kClusterMaxRows = 64;

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The float at the same shared-memory offset as `local` in CTA `rank` of the
// cluster.
__device__ __forceinline__ float ld_cluster(const float* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"(smem_u32(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

__global__ void __launch_bounds__(kClusterThreads)
    prep_cluster_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ res,
                        uint16_t* __restrict__ res_out, const uint16_t* __restrict__ w,
                        const int8_t* __restrict__ sign, float eps, int K, int vec,
                        uint16_t* __restrict__ norm_out, void* __restrict__ q, int layout,
                        float* __restrict__ sx, int32_t* __restrict__ qsum) {
  __shared__ __align__(16) float hs[kHad];   // h, then the transformed block
  __shared__ __align__(16) float sq[kHad];   // h^2, read by the whole cluster
  __shared__ float tree[kClusterThreads];
  constexpr int kWarps = kClusterThreads / 32;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int C = K / kHad;
  const uint32_t c = cluster_ctarank();
  const int64_t m = blockIdx.x / C;
  const int G = K / kGroup;
  const int64_t row0 = m * K + (int64_t)c * kHad;  // first element of the block
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  TransformOperands ops;
  load_transform_operands<kWarps>(w + c * kHad, sign + c * kHad, 1, warp, lane, ops);

  // Pass 1a: h = x (+ residual) of the block, four elements per thread.
  {
    const int j = 4 * t;
    float h4[4];
    if (vec) {
      const uint2 xv = *reinterpret_cast<const uint2*>(x + row0 + j);
      uint2 rv = make_uint2(0u, 0u);
      if (res) rv = *reinterpret_cast<const uint2*>(res + row0 + j);
      const uint32_t xw[2] = {xv.x, xv.y}, rw[2] = {rv.x, rv.y};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float a = bf16_bits_to_float((uint16_t)(xw[e >> 1] >> (16 * (e & 1))));
        if (res) a = __fadd_rn(a, bf16_bits_to_float((uint16_t)(rw[e >> 1] >> (16 * (e & 1)))));
        h4[e] = a;
      }
      if (res_out)
        *reinterpret_cast<uint2*>(res_out + row0 + j) =
            make_uint2((uint32_t)float_to_bf16_bits(h4[0]) |
                           ((uint32_t)float_to_bf16_bits(h4[1]) << 16),
                       (uint32_t)float_to_bf16_bits(h4[2]) |
                           ((uint32_t)float_to_bf16_bits(h4[3]) << 16));
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float a = bf16_bits_to_float(x[row0 + j + e]);
        if (res) a = __fadd_rn(a, bf16_bits_to_float(res[row0 + j + e]));
        h4[e] = a;
        if (res_out) res_out[row0 + j + e] = float_to_bf16_bits(a);
      }
    }
    *reinterpret_cast<float4*>(hs + j) = make_float4(h4[0], h4[1], h4[2], h4[3]);
    *reinterpret_cast<float4*>(sq + j) =
        make_float4(__fmul_rn(h4[0], h4[0]), __fmul_rn(h4[1], h4[1]), __fmul_rn(h4[2], h4[2]),
                    __fmul_rn(h4[3], h4[3]));
  }
  cluster_arrive();  // the block's squares are visible to the cluster
  cluster_wait();

  // Pass 1b: lanes t + 256k (k < 8) of the 2048 strided partial sums, each
  // in increasing j, element j read from CTA j / 1024 of the cluster; then
  // the tree, as the 256-thread one-CTA kernel forms it.
  // Every remote load goes out before the first addition (K <= 8192: at
  // most four slices of 2048), then the sums are formed in increasing j.
  constexpr int kPer = kLanes / kClusterThreads;
  constexpr int kSlices = 8 * kHad / kLanes;
  float v[kSlices][kPer];
#pragma unroll
  for (int sl = 0; sl < kSlices; ++sl)
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int j = sl * kLanes + t + kClusterThreads * k;
      v[sl][k] = j < K ? ld_cluster(sq + (j & (kHad - 1)), (uint32_t)(j / kHad)) : 0.0f;
    }
  cluster_arrive();  // done reading the cluster's squares (waited for at exit)
  float p[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    p[k] = 0.0f;
#pragma unroll
    for (int sl = 0; sl < kSlices; ++sl)
      if (sl * kLanes + t + kClusterThreads * k < K) p[k] = __fadd_rn(p[k], v[sl][k]);
  }
#pragma unroll
  for (int step = kLanes / kClusterThreads / 2; step >= 1; step >>= 1)
#pragma unroll
    for (int k = 0; k < step; ++k) p[k] = __fadd_rn(p[k], p[k + step]);
  tree[t] = p[0];
  __syncthreads();
  if (warp == 0) {
    // Levels 128, 64, 32 in the registers of warp 0 (lane l holds lanes
    // l + 32k of the tree, so each pair i, i + len meets in one lane), then
    // 16 .. 1 by shuffles.
    float u[kWarps];
#pragma unroll
    for (int k = 0; k < kWarps; ++k) u[k] = tree[lane + 32 * k];
#pragma unroll
    for (int step = kWarps / 2; step >= 1; step >>= 1)
#pragma unroll
      for (int k = 0; k < step; ++k) u[k] = __fadd_rn(u[k], u[k + step]);
    float v = u[0];
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

  // Pass 2: the block's transform by all eight warps (four values a lane).
  transform_shared<kWarps, kWarps>(hs, ops, inv, norm_out ? norm_out + c * kHad : nullptr, m, K,
                                   1, warp, lane);
  __syncthreads();
  // Pass 3: the block's eight 128-groups, one per warp.
  {
    const int gi = warp;
    const int g = (int)c * (kHad / kGroup) + gi;
    const float4 v4 = *reinterpret_cast<const float4*>(hs + gi * kGroup + 4 * lane);
    const float a[4] = {v4.x, v4.y, v4.z, v4.w};
    int qi[4];
    const float s = quantize_group4(a, qi);
    store_group4(qi, lane, q, layout, m * K + (int64_t)g * kGroup,
                 qsum ? qsum + m * G + g : nullptr);
    if (lane == 0) sx[m * G + g] = s;
  }
  cluster_wait();  // no CTA leaves while another may still read its squares
}

template <int kPrepThreads>
int launch_prep(const uint16_t* x, const uint16_t* residual, uint16_t* residual_out,
                const uint16_t* w, const int8_t* sign, float eps, int64_t M, int64_t K,
                uint16_t* norm_out, void* q, int q_layout, float* sx, int32_t* qsum,
                cudaStream_t stream) {
  const int smem = (int)((K + kPrepThreads) * sizeof(float));
  static int configured = 0;
  if (smem > configured) {
    if (cudaFuncSetAttribute(prep_kernel<kPrepThreads>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
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
  auto a16 = [](const void* ptr) { return reinterpret_cast<uintptr_t>(ptr) % 16 == 0; };
  const int vec = a16(x) && (!residual || a16(residual)) && (!residual_out || a16(residual_out));
  // The register path of the many-row kernel: 16-byte loads of the norm
  // weights and signs, 16-byte stores of q (and of the normalised row).
  const int fused = q_layout != PQ2_Q_MMV16 && a16(q) && a16(w) && a16(sign) &&
                    (!norm_out || a16(norm_out));
  if (cudaLaunchKernelEx(&cfg, prep_kernel<kPrepThreads>, x, residual, residual_out, w, sign,
                         eps, (int)K, vec, fused,
                         norm_out, q, q_layout, sx, qsum) != cudaSuccess) {
    cudaGetLastError();
    return PQ2_ERR_LAUNCH;
  }
  return PQ2_OK;
}

int launch_prep_cluster(const uint16_t* x, const uint16_t* residual, uint16_t* residual_out,
                        const uint16_t* w, const int8_t* sign, float eps, int64_t M, int64_t K,
                        uint16_t* norm_out, void* q, int q_layout, float* sx, int32_t* qsum,
                        cudaStream_t stream) {
  const int C = (int)(K / kHad);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(M * C));
  cfg.blockDim = dim3(kClusterThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  auto a8 = [](const void* ptr) { return reinterpret_cast<uintptr_t>(ptr) % 8 == 0; };
  const int vec = a8(x) && (!residual || a8(residual)) && (!residual_out || a8(residual_out));
  if (cudaLaunchKernelEx(&cfg, prep_cluster_kernel, x, residual, residual_out, w, sign, eps,
                         (int)K, vec, norm_out, q, q_layout, sx, qsum) != cudaSuccess) {
    cudaGetLastError();
    return PQ2_ERR_LAUNCH;
  }
  return PQ2_OK;
}

}  // namespace

int launch_norm_hadamard_quantize(const uint16_t* x, const uint16_t* residual,
                                  uint16_t* residual_out, const uint16_t* w, const int8_t* sign,
                                  float eps, int64_t M, int64_t K, uint16_t* norm_out, void* q,
                                  int q_layout, float* sx, int32_t* qsum, cudaStream_t stream) {
  // Few rows of at most eight transform blocks: one cluster CTA per block
  // (the latency of a row, spread over K / 1024 SMs).
  if (K <= 8 * kHad && M <= kClusterMaxRows)
    return launch_prep_cluster(x, residual, residual_out, w, sign, eps, M, K, norm_out, q,
                               q_layout, sx, qsum, stream);
  // Rows resident at once with 256 threads: four per SM on 152 SMs.
  if (M < 4 * 152)
    return launch_prep<1024>(x, residual, residual_out, w, sign, eps, M, K, norm_out, q,
                             q_layout, sx, qsum, stream);
  return launch_prep<256>(x, residual, residual_out, w, sign, eps, M, K, norm_out, q, q_layout,
                          sx, qsum, stream);
}

}  // namespace pq2
