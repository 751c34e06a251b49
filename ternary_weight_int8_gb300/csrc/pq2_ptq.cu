// pq2_ptq.cu — PTQ1_0 weights (five trits per byte) x INT8 activations on
// sm_103a: the preparation byte move and the small-batch GEMV (M = 1..4).
//
// Format: page "KERNEL_REPORT: PTQ1_0 small-batch decoding on the PrismML
// fork, RTX 3060 12GB" (KR), "What the source said": a 28-byte block per 128
// weights; 24 qs bytes holding five trits each, unpacked by multiplying by 3
// in a 16-bit lane and taking the part above the low byte; qh, two bytes
// with the other 8 trits; the fp16 scale d in the last two bytes; a trit t
// means weight t - 1.  Which trit is which weight: trit n of qs byte j is
// weight 24n + j, trit n (n < 4) of qh byte j is weight 120 + 2n + j.
//
// Prepared layout (this library's own): a qs plane u8[N][24 G] (the qs bytes
// of each block, in order) and a side plane u32[N][G] holding qh in bits
// 0-15 and d's bits in 16-31: still 28 bytes per 128 weights.
//
// Activations: the grouped quantiser (pq2_quantize_act_grouped) in the row
// layout, activation groups of A = 128, 64 or 32 (KR's activations come in
// 32-element blocks with a scale each; A = 32 is that case).
//
// GEMV design:
//  * CTA c owns rows [N*c/P, N*(c+1)/P), P = min(N, #SM); thread t owns
//    split z = t % S and row r = t / S, and the block pairs p = z, z+S, ...
//    of its row (a pair is 48 qs bytes: three 16-byte pieces).  S is a power
//    of two chosen from (N, K, #SM) only.
//  * Every thread streams its own pairs into a private ring of shared-memory
//    slots with cp.async, several pairs ahead; there is no producer warp and
//    no barrier wait that could stall on another thread.  q, s_x and sum(q)
//    of all columns are copied once per CTA (q XOR-swizzled by pair so that
//    the splits of a warp read different banks).
//  * Trit decode of a qs word (bytes b0..b3): b0, b2 and b1, b3 in the 16-bit
//    lanes of two registers; P_n = lane * 3^(n+1) never leaves its lane
//    (255 * 243 < 2^16), and H_n, the byte above each lane's low byte, is
//    floor(b * 3^(n+1) / 256); the trits are T_n = H_n - 3 H_(n-1) bytewise
//    (no borrow: floor(3x) >= 3 floor(x)), the same digits as the repeated
//    x3-and-carry of the format, with independent products instead of a
//    chain.  T_n holds the trits of weights 24n + 4w .. +3, which meet the
//    q word 6n + w in one dp4a.u32.s32; the -1 offset is removed with
//    sum(q) once per activation group.  The decode runs level by level over
//    a block's six qs words, so a level's six trit words meet 24
//    consecutive q bytes (three 8-byte shared loads per column) and the
//    live state stays small enough for three CTAs per SM.
//  * y = sum over blocks g of d_g * (sum over activation groups h of
//    float(dot_gh) * s_x_gh), fp32, every operation rounded to nearest, h
//    ascending, the blocks of a split in order, then a fixed xor butterfly
//    over the S splits.  Nothing depends on M: column m is bit-identical for
//    every M.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "pq2_device.cuh"
#include "pq2_internal.h"

namespace pq2 {
namespace {

constexpr int kRawBlock = 28;
constexpr int kQsBytes = 24;
constexpr int kPairBytes = 48;
constexpr int kSlotChunks = 4;          // 3 x 16 qs bytes + 8 side bytes
// q of a block pair (256 bytes) sits at a pitch of 272 bytes: the splits of a
// warp read consecutive pairs, 17 16-byte units apart, in different banks.
constexpr int kQPitch = 272;
constexpr int kMaxThreads = 288;
constexpr int kSoloSmem = 120 * 1024;  // one CTA per SM
constexpr int kMaxSmem = 227 * 1024;

struct PtqParams {
  const int8_t* q;          // [M][K], natural order
  const float* sx;          // [M][K/A]
  const int32_t* qsum;      // [M][K/A]
  const uint8_t* qs;        // [N][24 G]
  const uint32_t* side;     // [N][G]: qh | d << 16
  void* y;                  // [M][N]
  int32_t* dots;            // [M][N][K/A] (dot-only variant)
  int N, K, G, G2;
  int ctas, splits, depth;  // depth: ring slots per thread (4 or 8)
  int threads;
  int ring_off, sx_off, qs_off;
  int y_bf16;
  int overlap;
};

__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Trits of the two qh bytes (bits 0-15 of side): weights 120..123 and
// 124..127 of the block, as two words in weight order.
__device__ __forceinline__ void decode_qh(uint32_t side, uint32_t& t01, uint32_t& t23) {
  const uint32_t x = __byte_perm(side, 0u, 0x4140);   // qh0, qh1 in 16-bit lanes
  const uint32_t h01 = __byte_perm(x * 3u, x * 9u, 0x7531);
  const uint32_t h23 = __byte_perm(x * 27u, x * 81u, 0x7531);
  t01 = h01 - 3u * (h01 << 16);
  t23 = h23 - 3u * __byte_perm(h01, h23, 0x5432);
}

template <int M, int NSUB, bool DOTS>
__global__ void __launch_bounds__(kMaxThreads, 3) ptq_mmv_kernel(const PtqParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  grid_dep_launch();
  constexpr int A = 128 / NSUB;
  const int tid = threadIdx.x, T = p.threads;
  const int S = p.splits, z = tid % S, r = tid / S;
  const int c = blockIdx.x;
  const int n0 = (int)((int64_t)p.N * c / p.ctas), n1 = (int)((int64_t)p.N * (c + 1) / p.ctas);
  const int n = n0 + r;
  const bool active = n < n1;
  const int K = p.K, G = p.G, GA = G * NSUB;
  const int n_it = active && z < p.G2 ? (p.G2 - z + S - 1) / S : 0;
  const int D = p.depth;

  const uint32_t ring = smem_u32(smem + p.ring_off);
  auto slot_addr = [&](int slot, int chunk) -> uint32_t {
    return ring + (uint32_t)(((slot * kSlotChunks + chunk) * T + tid) * 16);
  };
  const uint8_t* qs_row = p.qs + (size_t)n * (size_t)(kQsBytes * G);
  const uint32_t* side_row = p.side + (size_t)n * (size_t)G;
  auto load_pair = [&](int it) {
    const int pp = z + S * it;
    const uint8_t* src = qs_row + (size_t)pp * kPairBytes;
    const int slot = it & (D - 1);
    cp_async16(slot_addr(slot, 0), src);
    cp_async16(slot_addr(slot, 1), src + 16);
    cp_async16(slot_addr(slot, 2), src + 32);
    cp_async8(slot_addr(slot, 3), side_row + 2 * pp);
  };
  // q (pairs at a pitch of kQPitch bytes), s_x and sum(q): all threads.
  const int QP = p.G2 * kQPitch;  // bytes of one column's q in shared memory
  auto load_inputs = [&]() {
    const uint32_t qb = smem_u32(smem);
    const int chunks = M * (K / 16);
    for (int i = tid; i < chunks; i += T) {
      const int m = i / (K / 16), k16 = i % (K / 16);
      const uint32_t dst = qb + (uint32_t)(m * QP + (k16 >> 4) * kQPitch + 16 * (k16 & 15));
      cp_async16(dst, p.q + (size_t)m * K + 16 * k16);
    }
    const uint32_t sb = smem_u32(smem + p.sx_off), tb = smem_u32(smem + p.qs_off);
    for (int i = tid; i < M * GA; i += T) {
      if (!DOTS) cp_async4(sb + 4 * i, p.sx + i);
      cp_async4(tb + 4 * i, p.qsum + i);
    }
  };

  if (p.overlap == 0) grid_dep_wait();
  if (n_it > 0) load_pair(0);
  cp_commit();
  if (p.overlap == 1) grid_dep_wait();
  load_inputs();
  cp_commit();
  for (int s = 1; s < D - 1; ++s) {
    if (s < n_it) load_pair(s);
    cp_commit();
  }
  if (D == 8) cp_wait<6>(); else if (D == 4) cp_wait<2>(); else cp_wait<0>();
  __syncthreads();

  const int8_t* qsm = reinterpret_cast<const int8_t*>(smem);
  const float* sxs = reinterpret_cast<const float*>(smem + p.sx_off);
  const int32_t* tss = reinterpret_cast<const int32_t*>(smem + p.qs_off);
  float yacc[M];
#pragma unroll
  for (int m = 0; m < M; ++m) yacc[m] = 0.0f;

#pragma unroll 1
  for (int it = 0; it < n_it; ++it) {
    if (it + D - 1 < n_it) load_pair(it + D - 1);
    cp_commit();
    if (D == 8) cp_wait<7>(); else if (D == 4) cp_wait<3>(); else cp_wait<1>();
    const int slot = it & (D - 1);
    const int pp = z + S * it;
    const uint8_t* sl = smem + p.ring_off + (size_t)((slot * kSlotChunks) * T + tid) * 16;
    const uint4 w0 = *reinterpret_cast<const uint4*>(sl);
    const uint4 w1 = *reinterpret_cast<const uint4*>(sl + (size_t)T * 16);
    const uint4 w2 = *reinterpret_cast<const uint4*>(sl + (size_t)2 * T * 16);
    const uint2 sd = *reinterpret_cast<const uint2*>(sl + (size_t)3 * T * 16);
    const uint32_t words[12] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y,
                                w1.z, w1.w, w2.x, w2.y, w2.z, w2.w};
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int g = 2 * pp + b;
      const uint32_t side = b ? sd.y : sd.x;
      // Level-major: the trits of level lv of all six qs words meet the q
      // words 6 lv .. 6 lv + 5 (24 consecutive bytes), so the decode state
      // is the split bytes and the previous H of each word.
      uint32_t lo[6], hi[6], prev[6];
#pragma unroll
      for (int wi = 0; wi < 6; ++wi) {
        lo[wi] = __byte_perm(words[6 * b + wi], 0u, 0x4240);  // b0, b2 in 16-bit lanes
        hi[wi] = __byte_perm(words[6 * b + wi], 0u, 0x4341);  // b1, b3
        prev[wi] = 0u;
      }
      const int8_t* qblk = qsm + pp * kQPitch + 128 * b;
      int acc[M][NSUB];
#pragma unroll
      for (int m = 0; m < M; ++m)
#pragma unroll
        for (int h = 0; h < NSUB; ++h) acc[m][h] = 0;
      uint32_t f = 3;
#pragma unroll
      for (int lv = 0; lv < 5; ++lv) {
        uint32_t t[6];
#pragma unroll
        for (int wi = 0; wi < 6; ++wi) {
          const uint32_t hv = __byte_perm(lo[wi] * f, hi[wi] * f, 0x7351);
          t[wi] = hv - 3u * prev[wi];
          prev[wi] = hv;
        }
        f *= 3;
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const uint2* qv = reinterpret_cast<const uint2*>(qblk + m * QP + 24 * lv);
          const uint2 q0 = qv[0], q1 = qv[1], q2 = qv[2];
          const uint32_t qw[6] = {q0.x, q0.y, q1.x, q1.y, q2.x, q2.y};
#pragma unroll
          for (int wi = 0; wi < 6; ++wi) {
            const int h = (24 * lv + 4 * wi) / A;
            acc[m][h] = dp4a_us(t[wi], (int)qw[wi], acc[m][h]);
          }
        }
      }
      uint32_t th01, th23;
      decode_qh(side, th01, th23);
      const float d = __half2float(__ushort_as_half((unsigned short)(side >> 16)));
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const uint2 qh = *reinterpret_cast<const uint2*>(qblk + m * QP + 120);
        acc[m][NSUB - 1] = dp4a_us(th01, (int)qh.x, acc[m][NSUB - 1]);
        acc[m][NSUB - 1] = dp4a_us(th23, (int)qh.y, acc[m][NSUB - 1]);
        const int j0 = m * GA + g * NSUB;
        float xs[NSUB];
        int ts[NSUB];
        if constexpr (NSUB == 4) {
          const float4 v = *reinterpret_cast<const float4*>(sxs + j0);
          const int4 u = *reinterpret_cast<const int4*>(tss + j0);
          xs[0] = v.x; xs[1] = v.y; xs[2] = v.z; xs[3] = v.w;
          ts[0] = u.x; ts[1] = u.y; ts[2] = u.z; ts[3] = u.w;
        } else if constexpr (NSUB == 2) {
          const float2 v = *reinterpret_cast<const float2*>(sxs + j0);
          const int2 u = *reinterpret_cast<const int2*>(tss + j0);
          xs[0] = v.x; xs[1] = v.y;
          ts[0] = u.x; ts[1] = u.y;
        } else {
          xs[0] = sxs[j0];
          ts[0] = tss[j0];
        }
        float inner = 0.0f;
#pragma unroll
        for (int h = 0; h < NSUB; ++h) {
          const int dot = acc[m][h] - ts[h];
          if (DOTS) {
            p.dots[((size_t)m * p.N + n) * GA + g * NSUB + h] = dot;
          } else {
            const float x = __fmul_rn((float)dot, xs[h]);
            inner = h == 0 ? x : __fadd_rn(inner, x);
          }
        }
        if (!DOTS) yacc[m] = __fadd_rn(yacc[m], __fmul_rn(inner, d));
      }
    }
  }
  cp_wait<0>();
  if constexpr (!DOTS) {
    // fixed xor butterfly over the S splits of a row (adjacent lanes)
#pragma unroll
    for (int m = 0; m < M; ++m)
      for (int off = 1; off < S; off <<= 1)
        yacc[m] = __fadd_rn(yacc[m], __shfl_xor_sync(0xffffffffu, yacc[m], off));
    if (p.overlap == 2) grid_dep_wait();
    if (active && z == 0) {
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const size_t o = (size_t)m * p.N + n;
        if (p.y_bf16)
          static_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(yacc[m]);
        else
          static_cast<float*>(p.y)[o] = yacc[m];
      }
    }
  }
}

// One thread per block: 24 qs bytes to the qs plane, qh and d to the side
// plane.
__global__ void ptq_prepare_kernel(const uint8_t* raw, int64_t raw_stride, int N, int G,
                                   uint8_t* qs, uint32_t* side) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)N * G) return;
  const int64_t n = i / G, g = i % G;
  const uint8_t* b = raw + n * raw_stride + g * kRawBlock;
  uint32_t* dst = reinterpret_cast<uint32_t*>(qs + n * (int64_t)(kQsBytes * G) + g * kQsBytes);
#pragma unroll
  for (int w = 0; w < 6; ++w)
    dst[w] = (uint32_t)b[4 * w] | ((uint32_t)b[4 * w + 1] << 8) |
             ((uint32_t)b[4 * w + 2] << 16) | ((uint32_t)b[4 * w + 3] << 24);
  side[i] = (uint32_t)b[24] | ((uint32_t)b[25] << 8) | ((uint32_t)b[26] << 16) |
            ((uint32_t)b[27] << 24);
}

template <int M, int NSUB, bool DOTS>
int launch_ptq_one(const PtqParams& p, int smem, cudaStream_t stream) {
  auto kern = ptq_mmv_kernel<M, NSUB, DOTS>;
  static int configured = 0;
  if (smem > configured) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem) !=
        cudaSuccess)
      return PQ2_ERR_LAUNCH;
    configured = kMaxSmem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.ctas);
  cfg.blockDim = dim3(p.threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) {
    cudaGetLastError();
    return PQ2_ERR_LAUNCH;
  }
  return PQ2_OK;
}

template <int NSUB, bool DOTS>
int launch_ptq_m(int M, const PtqParams& p, int smem, cudaStream_t s) {
  switch (M) {
    case 1: return launch_ptq_one<1, NSUB, DOTS>(p, smem, s);
    case 2: return launch_ptq_one<2, NSUB, DOTS>(p, smem, s);
    case 3: return launch_ptq_one<3, NSUB, DOTS>(p, smem, s);
    case 4: return launch_ptq_one<4, NSUB, DOTS>(p, smem, s);
    default: return PQ2_ERR_SHAPE;
  }
}

template <bool DOTS>
int launch_ptq_sub(int nsub, int M, const PtqParams& p, int smem, cudaStream_t s) {
  switch (nsub) {
    case 1: return launch_ptq_m<1, DOTS>(M, p, smem, s);
    case 2: return launch_ptq_m<2, DOTS>(M, p, smem, s);
    case 4: return launch_ptq_m<4, DOTS>(M, p, smem, s);
    default: return PQ2_ERR_SHAPE;
  }
}

int align16(int v) { return (v + 15) & ~15; }

}  // namespace

// Geometry: P = min(N, #SM) CTAs (more when a CTA would exceed 288 rows),
// R = ceil(N / P) rows, S = the largest power of two <= 32 with R * S <= 288
// and S <= the number of block pairs.  A function of (N, K, #SM) only.
bool ptq_geometry(int64_t N, int64_t K, int sm_count, int* ctas, int* rows, int* splits) {
  if (N < 1 || K < 256 || K % 256 || sm_count < 1) return false;
  int64_t P = std::min<int64_t>(N, sm_count);
  if ((N + P - 1) / P > kMaxThreads) P = (N + kMaxThreads - 1) / kMaxThreads;
  const int R = (int)((N + P - 1) / P);
  const int G2 = (int)(K / 256);
  int S = 1;
  while (S < 32 && R * (2 * S) <= kMaxThreads && 2 * S <= G2) S *= 2;
  *ctas = (int)P;
  *rows = R;
  *splits = S;
  return true;
}

int launch_ptq_prepare(const uint8_t* raw, int64_t raw_stride, int64_t N, int64_t K, uint8_t* qs,
                       uint32_t* side, cudaStream_t stream) {
  const int64_t G = K / 128, total = N * G;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  ptq_prepare_kernel<<<(unsigned)blocks, threads, 0, stream>>>(raw, raw_stride, (int)N, (int)G,
                                                                qs, side);
  if (cudaGetLastError() != cudaSuccess) return PQ2_ERR_LAUNCH;
  return PQ2_OK;
}

int launch_ptq_mmv(const int8_t* q, const float* sx, const int32_t* qsum, const uint8_t* qs,
                   const uint32_t* side, void* y, int y_dtype, int32_t* dots, int64_t M,
                   int64_t N, int64_t K, int act_group, int overlap, int sm_count,
                   cudaStream_t stream) {
  if (act_group != 128 && act_group != 64 && act_group != 32) return PQ2_ERR_SHAPE;
  const int nsub = 128 / act_group;
  int ctas, R, S;
  if (M < 1 || M > 4 || !ptq_geometry(N, K, sm_count, &ctas, &R, &S)) return PQ2_ERR_SHAPE;
  PtqParams p{};
  p.q = q; p.sx = sx; p.qsum = qsum; p.qs = qs; p.side = side; p.y = y; p.dots = dots;
  p.N = (int)N; p.K = (int)K; p.G = (int)(K / 128); p.G2 = (int)(K / 256);
  p.ctas = ctas; p.splits = S;
  p.threads = (R * S + 31) / 32 * 32;
  p.y_bf16 = y_dtype == PQ2_BF16;
  p.overlap = overlap;
  const int GA = p.G * nsub;
  p.sx_off = align16((int)M * p.G2 * kQPitch);
  p.qs_off = align16(p.sx_off + (int)M * GA * 4);
  p.ring_off = align16(p.qs_off + (int)M * GA * 4);
  const int slot_bytes = p.threads * kSlotChunks * 16;
  // Ring depth: the deepest of 8, 4, 2 slots that keeps three CTAs (the
  // register budget of the kernel) within an SM's shared memory; a call that
  // waits for the kernel before it takes the whole SM.
  const int per_sm = 3;
  const int budget = overlap == 1 ? kMaxSmem : (228 * 1024) / per_sm - 1024;
  p.depth = 2;
  for (int d : {8, 4})
    if (p.ring_off + d * slot_bytes <= budget) {
      p.depth = d;
      break;
    }
  int smem = p.ring_off + p.depth * slot_bytes;
  if (smem > kMaxSmem) return PQ2_ERR_SHAPE;
  // A call that waits for the kernel before it takes a whole SM (more than
  // half the shared memory), so chained calls fill the SMs one CTA each.
  if (overlap == 1) smem = std::max(smem, kSoloSmem);
  return dots ? launch_ptq_sub<true>(nsub, (int)M, p, smem, stream)
              : launch_ptq_sub<false>(nsub, (int)M, p, smem, stream);
}

}  // namespace pq2
