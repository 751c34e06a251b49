// pq2_quant.cuh — the per-group INT8 activation quantisation as warp-level
// device functions, shared by the stand-alone quantisation kernel and the
// fused norm / Hadamard / quantisation kernel, so both produce the same bytes
// by construction.
//
// Method: page "Kernel experiments: recorded evidence" (KE), Test 6
// (_quantize) and page "Baseline and the integer breakthrough" (BIB),
// "Calculate with small integers", step 1: per group of 128 activations
// s = max|a| / 127, q = clamp(round_half_even(a / s), -127, 127), with
// s = 0 (an all-zero group) dividing by 1.  Layouts: KE Test 21 (plane
// order) and the prefill MMA operand order (include/pq2.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "pq2.h"

namespace pq2 {

// One 128-group held by a full warp, lane L owning elements 4L..4L+3, in
// activation groups of 4 * LANES elements (LANES = 32: the whole 128-group;
// 16 or 8: groups of 64 or 32, KE Test 9).  Returns the scale s of the
// lane's activation group (the same in all its lanes) and the lane's four q,
// equal to
// clamp(rint(a / d)) with the IEEE round-to-nearest quotient a / d.
// The quotient is first formed as t = a * rcp(d) (rcp correctly rounded):
// t differs from the rounded quotient by at most |a / d| * 2^-23 + 2^-24
// relative, i.e. 2.3e-5 for |a / d| <= 127.01, so rint(t) is rint(a / d)
// unless t lies within 1e-4 of a half-integer (t - rint(t) is exact).  If any
// element of the group is that close (or d < 2^-120, where rcp(d) may
// overflow), the whole group takes the IEEE divisions: one uniform branch,
// rarely taken.
template <int LANES = 32>
__device__ __forceinline__ float quantize_group4(const float a[4], int qi[4]) {
  float amax = fmaxf(fmaxf(fabsf(a[0]), fabsf(a[1])), fmaxf(fabsf(a[2]), fabsf(a[3])));
#pragma unroll
  for (int off = LANES / 2; off > 0; off >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float s = __fdiv_rn(amax, 127.0f);
  const float d = s > 0.0f ? s : 1.0f;
  const float inv = __frcp_rn(d);
  bool near_tie = d < 7.52316385e-37f;  // 2^-120
  float r[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float t = __fmul_rn(a[j], inv);
    r[j] = rintf(t);
    near_tie |= fabsf(t - r[j]) > 0.4999f;
  }
  if (__any_sync(0xffffffffu, near_tie)) {
#pragma unroll
    for (int j = 0; j < 4; ++j) r[j] = rintf(__fdiv_rn(a[j], d));
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) qi[j] = (int)fminf(fmaxf(r[j], -127.0f), 127.0f);
  return s;
}

// Store one 128-group's q (lane L holding elements 4L..4L+3 of the group
// that starts at element `base` of q) in the requested layout, and the sum of
// q of each of its activation groups of 4 * LANES elements (to qsum[0 ..
// 32 / LANES - 1] when non-null).  Every lane of the warp must call it.
template <int LANES = 32>
__device__ __forceinline__ void store_group4(const int qi[4], int lane, void* q, int layout,
                                             int64_t base, int32_t* qsum) {
  const uint32_t packed = (uint32_t)(qi[0] & 0xff) | ((uint32_t)(qi[1] & 0xff) << 8) |
                          ((uint32_t)(qi[2] & 0xff) << 16) | ((uint32_t)(qi[3] & 0xff) << 24);
  if (layout == PQ2_Q_ROWS) {
    reinterpret_cast<uint32_t*>(static_cast<int8_t*>(q) + base)[lane] = packed;
  } else if (layout == PQ2_Q_PLANES) {
    // Plane word (s, w) = q[16w + 4b + s] for b = 0..3: byte s of the packed
    // words of lanes 4w..4w+3.  Lane L = 8s + w assembles it, so the warp
    // writes the group's 128 bytes as one coalesced line.
    const int s_out = lane >> 3, w_out = lane & 7;
    uint32_t out = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t v = __shfl_sync(0xffffffffu, packed, 4 * w_out + b);
      out |= ((v >> (8 * s_out)) & 0xffu) << (8 * b);
    }
    reinterpret_cast<uint32_t*>(static_cast<int8_t*>(q) + base)[lane] = out;
  } else if (layout == PQ2_Q_F8) {
    // Two e4m3 planes of the 8-bit prefill MMA, q = 16 a + b with
    // a = q >> 4 in [-8, 7] and b = q & 15 in [0, 15], both exact in e4m3:
    // bytes 0..127 of the group hold 16 a, bytes 128..255 hold b, each in the
    // operand K order.  Word W = 4i + c of a plane holds the elements
    // 16i + 8(c >> 1) + (c & 1) + 2e, e = 0..3: bytes (c & 1) and (c & 1) + 2
    // of lanes 4i + 2(c >> 1) and 4i + 2(c >> 1) + 1.
    uint32_t hi = 0, lo = 0;
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      const __nv_fp8x2_storage_t h2 = __nv_cvt_float2_to_fp8x2(
          make_float2((float)(16 * (qi[j] >> 4)), (float)(16 * (qi[j + 1] >> 4))),
          __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t l2 = __nv_cvt_float2_to_fp8x2(
          make_float2((float)(qi[j] & 15), (float)(qi[j + 1] & 15)), __NV_SATFINITE, __NV_E4M3);
      hi |= (uint32_t)h2 << (8 * j);
      lo |= (uint32_t)l2 << (8 * j);
    }
    const int src = 4 * (lane >> 2) + 2 * ((lane & 3) >> 1);
    const uint32_t sel = (lane & 1) ? 0x7531u : 0x6420u;
    const uint32_t ha = __shfl_sync(0xffffffffu, hi, src), hb = __shfl_sync(0xffffffffu, hi, src + 1);
    const uint32_t la = __shfl_sync(0xffffffffu, lo, src), lb = __shfl_sync(0xffffffffu, lo, src + 1);
    uint32_t* out = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(q) + 2 * base);
    out[lane] = __byte_perm(ha, hb, sel);
    out[32 + lane] = __byte_perm(la, lb, sel);
  } else if (layout == PQ2_Q_MMV16) {
    // Fragment order of the small-batch tensor-core GEMV (128-groups only):
    // position P = 32t + 4j + 2r + e of the group (lane L writes P = 4L..4L+3,
    // so t = L / 8, j = L % 8, (r, e) = the slot's two bits) holds element
    // i = 16(t + 4(j / 4)) + 8e + f, f = 2(j % 4) + r, divided by 4^f (f <= 4)
    // or 4^(f - 3) (f >= 5): the weight that meets it in the GEMV is then
    // 1024 + code * that power of 4, and the group's correction below
    // removes the 1024 and the code's -1 offset.
    const int t = lane >> 3, j = lane & 7;
    const int wbase = 16 * (t + 4 * (j >> 2)) + 2 * (j & 3);
    uint32_t out[2];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int i = wbase + 8 * (s & 1) + (s >> 1);
      const int f = 2 * (j & 3) + (s >> 1);
      const uint32_t v = __shfl_sync(0xffffffffu, packed, i >> 2);
      const int qv = (int)(int8_t)((v >> (8 * (i & 3))) & 0xffu);
      // 1 / 4^f or 1 / 4^(f-3): exact powers of two, so q / scale is exact
      const float inv = f <= 4 ? __int_as_float((127 - 2 * f) << 23)
                               : __int_as_float((127 - 2 * (f - 3)) << 23);
      const uint32_t h = (uint32_t)__half_as_ushort(__float2half_rn((float)qv * inv));
      if (s & 1)
        out[s >> 1] |= h << 16;
      else
        out[s >> 1] = h;
    }
    reinterpret_cast<uint2*>(static_cast<__half*>(q) + base)[lane] = make_uint2(out[0], out[1]);
    // Correction: sum over the group of q * (1 + 1024 / scale), the scale of
    // element i being that of its field f = i % 8 (weights 1025, 257, 65, 17,
    // 5, 65, 17, 5); |correction| <= 127 * 16 * 1456 < 2^22.
    int c = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int f = (4 * lane + k) & 7;
      const int wgt = f <= 4 ? 1 + (1024 >> (2 * f)) : 1 + (1024 >> (2 * (f - 3)));
      c += qi[k] * wgt;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
    if (qsum && lane == 0) qsum[0] = c;
    return;
  } else {
    // Operand order of the prefill MMA: inside each 16-element chunk (lanes
    // 4c..4c+3, element 4b + s held by lane 4c + b), element 4b + s goes to
    // position 4s + 2(b & 1) + (b >> 1).  Lane L = 4c + s' writes positions
    // 4s'..4s'+3, i.e. element s' of lanes 4c + 0, 2, 1, 3.
    const int c = lane >> 2, s_out = lane & 3;
    int o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int b = (j >> 1) | ((j & 1) << 1);  // 0, 2, 1, 3
      const uint32_t v = __shfl_sync(0xffffffffu, packed, 4 * c + b);
      o[j] = (int)(int8_t)((v >> (8 * s_out)) & 0xffu);
    }
    __half2 h01 = __halves2half2(__int2half_rn(o[0]), __int2half_rn(o[1]));
    __half2 h23 = __halves2half2(__int2half_rn(o[2]), __int2half_rn(o[3]));
    uint2 v;
    v.x = *reinterpret_cast<uint32_t*>(&h01);
    v.y = *reinterpret_cast<uint32_t*>(&h23);
    reinterpret_cast<uint2*>(static_cast<__half*>(q) + base)[lane] = v;
  }
  int t = qi[0] + qi[1] + qi[2] + qi[3];
#pragma unroll
  for (int off = LANES / 2; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
  if (qsum && lane % LANES == 0) qsum[lane / LANES] = t;
}

// ------------------------------------------------------------------------
// The same quantisation with eight lanes per 128-group: lane j = L % 8 of a
// group's eight lanes holds its elements 16j..16j+15, so a warp quantises
// four groups at once.  The per-element arithmetic is quantize_group4's; the
// reductions run over 8 lanes instead of 32 and the output layouts (except
// the tensor-core GEMV's PQ2_Q_MMV16) are assembled inside the lane, so a
// group costs about a quarter of the warp instructions.  Activation groups of
// 16 * LG elements (LG = 8, 4, 2 lanes: 128, 64, 32); groups of LG lanes are
// aligned.  Every lane of the warp must call it.
template <int LG = 8>
__device__ __forceinline__ float quantize_group16(const float (&a)[16], int (&qi)[16]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(a[i]));
#pragma unroll
  for (int off = LG / 2; off > 0; off >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float s = __fdiv_rn(amax, 127.0f);
  const float d = s > 0.0f ? s : 1.0f;
  const float inv = __frcp_rn(d);
  bool near_tie = d < 7.52316385e-37f;  // 2^-120
  float r[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float t = __fmul_rn(a[i], inv);
    r[i] = rintf(t);
    near_tie |= fabsf(t - r[i]) > 0.4999f;
  }
  // Any near tie in the warp sends all its groups through the IEEE
  // divisions, which give the same q wherever the product is not near a tie.
  if (__any_sync(0xffffffffu, near_tie)) {
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = rintf(__fdiv_rn(a[i], d));
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) qi[i] = (int)fminf(fmaxf(r[i], -127.0f), 127.0f);
  return s;
}

// Store the sixteen q of lane j (elements 16j..16j+15 of the 128-group that
// starts at element `base` of q) in the requested layout (not PQ2_Q_MMV16),
// and sum(q) of each activation group of 16 * LG elements (to qsum[0 ..
// 8 / LG - 1] when non-null, which `store` says for this lane's group).  The
// layouts are those of store_group4.  Every lane of the warp must call it.
template <int LG = 8>
__device__ __forceinline__ void store_group16(const int (&qi)[16], int j, bool store, void* q,
                                              int layout, int64_t base, int32_t* qsum) {
  auto byte = [&](int i) { return (uint32_t)(qi[i] & 0xff); };
  if (store) {
    if (layout == PQ2_Q_ROWS) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        w[k] = byte(4 * k) | (byte(4 * k + 1) << 8) | (byte(4 * k + 2) << 16) |
               (byte(4 * k + 3) << 24);
      reinterpret_cast<uint4*>(static_cast<int8_t*>(q) + base)[j] =
          make_uint4(w[0], w[1], w[2], w[3]);
    } else if (layout == PQ2_Q_PLANES) {
      // Plane word (s, w) = q[16w + 4b + s], b = 0..3, is word 8s + w of the
      // group: chunk w = j holds all four of its bytes.
      uint32_t* out = reinterpret_cast<uint32_t*>(static_cast<int8_t*>(q) + base);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        out[8 * s + j] =
            byte(s) | (byte(4 + s) << 8) | (byte(8 + s) << 16) | (byte(12 + s) << 24);
    } else if (layout == PQ2_Q_F8) {
      // Word c of chunk j in each plane holds the chunk's elements
      // 8(c >> 1) + (c & 1) + 2e, e = 0..3 (16a plane, then the b plane).
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        hi[c] = 0;
        lo[c] = 0;
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const int i0 = 8 * (c >> 1) + (c & 1) + 2 * e, i1 = i0 + 2;
          const __nv_fp8x2_storage_t h2 = __nv_cvt_float2_to_fp8x2(
              make_float2((float)(16 * (qi[i0] >> 4)), (float)(16 * (qi[i1] >> 4))),
              __NV_SATFINITE, __NV_E4M3);
          const __nv_fp8x2_storage_t l2 = __nv_cvt_float2_to_fp8x2(
              make_float2((float)(qi[i0] & 15), (float)(qi[i1] & 15)), __NV_SATFINITE,
              __NV_E4M3);
          hi[c] |= (uint32_t)h2 << (8 * e);
          lo[c] |= (uint32_t)l2 << (8 * e);
        }
      }
      uint4* out = reinterpret_cast<uint4*>(static_cast<uint8_t*>(q) + 2 * base);
      out[j] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      out[8 + j] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    } else {
      // Prefill MMA operand order: element 4b + s of the chunk goes to
      // position 4s + 2(b & 1) + (b >> 1).
      uint32_t h[8];
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const __half2 p01 = __halves2half2(__int2half_rn(qi[s]), __int2half_rn(qi[8 + s]));
        const __half2 p23 = __halves2half2(__int2half_rn(qi[4 + s]), __int2half_rn(qi[12 + s]));
        h[2 * s] = *reinterpret_cast<const uint32_t*>(&p01);
        h[2 * s + 1] = *reinterpret_cast<const uint32_t*>(&p23);
      }
      uint4* out = reinterpret_cast<uint4*>(static_cast<__half*>(q) + base);
      out[2 * j] = make_uint4(h[0], h[1], h[2], h[3]);
      out[2 * j + 1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
  }
  int t = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) t += qi[i];
#pragma unroll
  for (int off = LG / 2; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
  if (store && qsum && j % LG == 0) qsum[j / LG] = t;
}

// ------------------------------------------------------------------------
// The same quantisation with four lanes per 128-group: lane j = L % 4 of a
// group's four lanes holds its elements 32j..32j+31 (the fused
// preparation's layout after its transform), so a warp quantises eight
// groups at once with two shuffle levels per reduction.  The per-element
// arithmetic is quantize_group4's.  quantize_scale32 forms the group's
// scale and decides, warp-wide, between the product and the IEEE division
// (near ties); the caller then forms each q (the product or the division,
// rounded, then quantize_clamp), so the 32 rounded values never need
// registers beside the 32 inputs.  Every lane of the warp must call
// quantize_scale32.
struct GroupScale {
  float s, d, inv;
  bool exact;  // some group of the warp has a near tie: IEEE divisions
};
// Round to the nearest integer, ties to even, for |t| < 2^22: t + 1.5 * 2^23
// lies in [2^23, 2^24), where the float spacing is 1, so the addition rounds
// t's fraction exactly as rint does (1.5 * 2^23 is even), and the integer
// sits in the low mantissa bits.  Two full-rate instructions instead of a
// round and a conversion.  rint_magic_int is the integer, rint_magic_f the
// float (the subtraction is exact).
constexpr float kRintMagic = 12582912.0f;  // 1.5 * 2^23
__device__ __forceinline__ int rint_magic_int(float t) {
  return __float_as_int(__fadd_rn(t, kRintMagic)) - __float_as_int(kRintMagic);
}
__device__ __forceinline__ float rint_magic_f(float t) {
  return __fsub_rn(__fadd_rn(t, kRintMagic), kRintMagic);
}
__device__ __forceinline__ GroupScale quantize_scale32(const float (&a)[32]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(a[i]));
#pragma unroll
  for (int off = 2; off > 0; off >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  GroupScale z;
  z.s = __fdiv_rn(amax, 127.0f);
  z.d = z.s > 0.0f ? z.s : 1.0f;
  z.inv = __frcp_rn(z.d);
  bool near_tie = z.d < 7.52316385e-37f;  // 2^-120
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float t = __fmul_rn(a[i], z.inv);  // |t| <= 127 (1 + 2^-22)
    near_tie |= fabsf(t - rint_magic_f(t)) > 0.4999f;
  }
  z.exact = __any_sync(0xffffffffu, near_tie);
  return z;
}
// The clamp of a rounded quotient to the int8 range of q.
__device__ __forceinline__ int quantize_clamp(float r) {
  return (int)fminf(fmaxf(r, -127.0f), 127.0f);
}
// q of one element on the product path of quantize_scale32: |a * inv| is at
// most 127 (1 + 2^-22), so rint_magic_int applies and the clamp is on the
// integer.
__device__ __forceinline__ int quantize_product(float a, float inv) {
  return max(min(rint_magic_int(__fmul_rn(a, inv)), 127), -127);
}

// Store the sixteen q of one 16-element chunk c (0..7) of the 128-group that
// starts at element `base` of q, in the requested layout (not PQ2_Q_MMV16):
// the layouts of store_group16.
__device__ __forceinline__ void store_chunk16(const int (&qi)[16], int c, void* q, int layout,
                                              int64_t base) {
  auto byte = [&](int i) { return (uint32_t)(qi[i] & 0xff); };
  if (layout == PQ2_Q_ROWS) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      w[k] = byte(4 * k) | (byte(4 * k + 1) << 8) | (byte(4 * k + 2) << 16) |
             (byte(4 * k + 3) << 24);
    reinterpret_cast<uint4*>(static_cast<int8_t*>(q) + base)[c] =
        make_uint4(w[0], w[1], w[2], w[3]);
  } else if (layout == PQ2_Q_PLANES) {
    uint32_t* out = reinterpret_cast<uint32_t*>(static_cast<int8_t*>(q) + base);
#pragma unroll
    for (int s = 0; s < 4; ++s)
      out[8 * s + c] = byte(s) | (byte(4 + s) << 8) | (byte(8 + s) << 16) | (byte(12 + s) << 24);
  } else if (layout == PQ2_Q_F8) {
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int cw = 0; cw < 4; ++cw) {
      hi[cw] = 0;
      lo[cw] = 0;
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const int i0 = 8 * (cw >> 1) + (cw & 1) + 2 * e, i1 = i0 + 2;
        const __nv_fp8x2_storage_t h2 = __nv_cvt_float2_to_fp8x2(
            make_float2((float)(16 * (qi[i0] >> 4)), (float)(16 * (qi[i1] >> 4))),
            __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t l2 = __nv_cvt_float2_to_fp8x2(
            make_float2((float)(qi[i0] & 15), (float)(qi[i1] & 15)), __NV_SATFINITE, __NV_E4M3);
        hi[cw] |= (uint32_t)h2 << (8 * e);
        lo[cw] |= (uint32_t)l2 << (8 * e);
      }
    }
    uint4* out = reinterpret_cast<uint4*>(static_cast<uint8_t*>(q) + 2 * base);
    out[c] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    out[8 + c] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  } else {
    uint32_t h[8];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const __half2 p01 = __halves2half2(__int2half_rn(qi[s]), __int2half_rn(qi[8 + s]));
      const __half2 p23 = __halves2half2(__int2half_rn(qi[4 + s]), __int2half_rn(qi[12 + s]));
      h[2 * s] = *reinterpret_cast<const uint32_t*>(&p01);
      h[2 * s + 1] = *reinterpret_cast<const uint32_t*>(&p23);
    }
    uint4* out = reinterpret_cast<uint4*>(static_cast<__half*>(q) + base);
    out[2 * c] = make_uint4(h[0], h[1], h[2], h[3]);
    out[2 * c + 1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

}  // namespace pq2
