// pq2_mmv.cu — small-batch (M = 1..8) ternary x INT8 GEMV for sm_103a.
//
// Method: page "Baseline and the integer breakthrough" (BIB), "Calculate with
// small integers" (steps 2-4) and "Unpack four weights with fewer
// instructions"; page "Kernel experiments: recorded evidence" (KE), Tests 1,
// 6, 14 (add/XOR decode, DP4A group dots, one weight tile reused for every
// token) and Test 21 (plane-order q, masked planes with the sum(q) offset).
//
// GB300 design (not the pages' Triton/sm_86 tiling):
//  * One CTA per SM, sized (<= 110 KB shared memory, <= 352 threads) so that
//    two CTAs fit on an SM: with programmatic dependent launch the next call's
//    CTA streams its weights while this one finishes.
//  * CTA c owns the contiguous rows [N*c/P, N*(c+1)/P); every weight byte is
//    read from HBM exactly once for all M columns.
//  * Weights arrive by 2-D tensor TMA: one box is 128 code bytes (4 groups)
//    of every row of the CTA, written with the 128-byte swizzle, so a stage is
//    a handful of large requests.  q for the stage's groups follows as one
//    swizzled box per column (a group of 128 q bytes per box row).  A
//    producer warp keeps a ring of stages full.
//  * Consumer thread t owns (split z = t % S, row r = t / S) and handles the
//    interleaved groups g = z, z+S, z+2S, ... of its row; S divides 32, so the
//    S partial sums of a row live in adjacent lanes of one warp.  The swizzle
//    keeps both the code reads and the q reads free of bank conflicts.
//  * The group dot is lane-local and exact (int32).  Scaling follows the
//    method's order, t = (float(dot) * s_x) * s_w, y_z += t, with explicit
//    round-to-nearest intrinsics, and the S partials of a row are combined by
//    a fixed warp-shuffle butterfly.  Nothing in that sequence depends on M or
//    on the decoder, so column m is bit-identical for every M (batch
//    invariance).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "pq2_device.cuh"
#include "pq2_internal.h"

namespace pq2 {
namespace {

constexpr int kMaxConsumerThreads = 352;
constexpr int kMaxBlock = kMaxConsumerThreads + 32;
constexpr int kMaxSplits = 64;
constexpr int kMaxBoxRows = 256;          // TMA box height limit
constexpr int kSmemBudget = 110 * 1024;   // two CTAs per SM
constexpr int kMaxStages = 48;
constexpr int kBoxBytes = 128;            // 4 groups of 32 code bytes

struct MmvParams {
  const int8_t* q;        // [M][K], plane order inside each group
  const float* sx;        // [M][G]
  const int32_t* qsum;    // [M][G]
  const uint16_t* scales; // [N][G] fp16 bits
  void* y;                // [M][N] fp32 or bf16
  int32_t* dots;          // [M][N][G] (dot-only variant)
  int32_t* status;
  int N, K, G;
  int ctas, splits, rows_max, stages_total, ring;
  int cons_threads;
  int stage_groups;       // Gs: groups per stage (a multiple of 4 and of S)
  int box_stride;         // bytes per box in shared memory (1024-aligned)
  int stage_bytes;        // boxes + q region
  int q_off;              // q region inside a stage
  int qbox_stride;        // bytes per column's q box inside a stage (1024-aligned)
  int sw_off, sx_off, qs_off, ring_off;
  int y_bf16;
  int overlap;            // 1: stream weights before the grid dependency
                          // resolves; 2: stream every input before it
  int sw_bulk;            // weight-scale slab arrives by one bulk copy (G % 8 == 0)
  int sx_bulk;            // s_x and sum(q) arrive by bulk copies with stage 0
};

// Batched global -> shared copy of `count` 16-bit values by `threads`
// threads: every thread issues its loads before its stores, so the copy
// costs one or two memory round trips instead of one per element.
__device__ __forceinline__ void preload_u16(uint16_t* dst, const uint16_t* src, int count,
                                            int tid, int threads) {
  constexpr int B = 16;
  for (int base = tid; base < count; base += B * threads) {
    uint16_t v[B];
#pragma unroll
    for (int j = 0; j < B; ++j) {
      const int i = base + j * threads;
      v[j] = i < count ? __ldg(src + i) : (uint16_t)0;
    }
#pragma unroll
    for (int j = 0; j < B; ++j) {
      const int i = base + j * threads;
      if (i < count) dst[i] = v[j];
    }
  }
}

__device__ __forceinline__ void preload_u32(uint32_t* dst, const uint32_t* src, int count,
                                            int tid, int threads) {
  constexpr int B = 8;
  for (int base = tid; base < count; base += B * threads) {
    uint32_t v[B];
#pragma unroll
    for (int j = 0; j < B; ++j) {
      const int i = base + j * threads;
      v[j] = i < count ? __ldg(src + i) : 0u;
    }
#pragma unroll
    for (int j = 0; j < B; ++j) {
      const int i = base + j * threads;
      if (i < count) dst[i] = v[j];
    }
  }
}

__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Exact int32 dot of one 128-group for every column.
//   c0, c1 : the group's two 16-byte halves of code bytes (swizzled smem)
// Plane s of code word w (bytes 4w..4w+3 of the group) holds the codes of
// weights 16w + 4b + s (b = 0..3); in plane order those activations are the
// 4 bytes at s*32 + 4w, so one 32-bit q word meets one 32-bit plane word.
//   qz     : the group's box row of q for column 0 (128 bytes, 128-byte
//            swizzled with key qsw); column m at qz + m * q_mstride
template <int M, int DEC>
__device__ __forceinline__ void group_dot(const uint8_t* c0, const uint8_t* c1,
                                          const int8_t* qz, int q_mstride, int qsw,
                                          const int32_t* qs, int qs_mstride, int dot[M]) {
  // Independent accumulator chains per column: one per plane for M <= 2
  // (instruction-level parallelism), two for larger M (registers).  Masked
  // planes: even planes accumulate code * q, odd planes 4 * code * q.
  constexpr int NA = M <= 2 ? 4 : 2;
  int acc[NA][M];
#pragma unroll
  for (int a = 0; a < NA; ++a)
#pragma unroll
    for (int m = 0; m < M; ++m) acc[a][m] = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 c = *reinterpret_cast<const uint4*>(h ? c1 : c0);
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    uint32_t cs[4];  // the words shifted down by 4 bits: planes 2, 3 in place of 0, 1
#pragma unroll
    for (int w = 0; w < 4; ++w) cs[w] = cw[w] >> 4;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      int4 qv[M];
#pragma unroll
      for (int m = 0; m < M; ++m)
        qv[m] = *reinterpret_cast<const int4*>(qz + m * q_mstride + ((s * 32 + 16 * h) ^ qsw));
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t wv;
        if (DEC == kDecodeAddXor) {
          // Spread: the four codes of plane s, one per byte (values 0..3).
          // +0x7F7F7F7F cannot carry between bytes; ^0x80808080 maps
          // 127/128/129/130 to the signed bytes -1/0/+1/+2.
          const uint32_t spread = (cw[w] >> (2 * s)) & 0x03030303u;
          wv = (spread + 0x7F7F7F7Fu) ^ 0x80808080u;
        } else {
          // Masked plane: bytes code (s even) or 4 * code (s odd), unsigned.
          wv = ((s < 2) ? cw[w] : cs[w]) & ((s & 1) ? 0x0C0C0C0Cu : 0x03030303u);
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const int qw = w == 0 ? qv[m].x : w == 1 ? qv[m].y : w == 2 ? qv[m].z : qv[m].w;
          int& a = acc[NA == 4 ? s : (s & 1)][m];
          a = (DEC == kDecodeAddXor) ? __dp4a((int)wv, qw, a) : dp4a_us(wv, qw, a);
        }
      }
    }
  }
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const int even = NA == 4 ? acc[0][m] + acc[2][m] : acc[0][m];
    const int odd = NA == 4 ? acc[1][m] + acc[3][m] : acc[1][m];
    if (DEC == kDecodeAddXor) {
      dot[m] = even + odd;
    } else {
      // `odd` is exactly 4 * sum(code * q) over planes 1 and 3: shift it
      // back, then remove the codes' -1 offset with the group sum of q.
      dot[m] = even + (odd >> 2) - qs[m * qs_mstride];
    }
  }
}

template <int M, int DEC, bool DOTS>
__global__ void __launch_bounds__(kMaxBlock, 2)
    mmv_kernel(const __grid_constant__ CUtensorMap map_hi,
               const __grid_constant__ CUtensorMap map_lo,
               const __grid_constant__ CUtensorMap map_q, const MmvParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // The 128-byte swizzle needs 1024-byte aligned boxes.
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + p.ring;
  uint64_t* swbar = empty + p.ring;
  __half* sw_s = reinterpret_cast<__half*>(smem + p.sw_off);    // [rows_max][G]
  float* sx_s = reinterpret_cast<float*>(smem + p.sx_off);      // [M][G]
  int32_t* qs_s = reinterpret_cast<int32_t*>(smem + p.qs_off);  // [M][G]
  uint8_t* ring = smem + p.ring_off;

  const int c = blockIdx.x;
  const int n0 = (int)((int64_t)p.N * c / p.ctas);
  const int R = (int)((int64_t)p.N * (c + 1) / p.ctas) - n0;
  const CUtensorMap* map = (R == p.rows_max) ? &map_hi : &map_lo;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cons_warps = p.cons_threads >> 5;
  const int S = p.splits, G = p.G, Gs = p.stage_groups;
  const bool independent = p.overlap >= 2;

  if (tid == 0) {
    for (int s = 0; s < p.ring; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], cons_warps);
    }
    mbar_init(swbar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Dependent grids are released only after this grid's own wait (every
  // thread waits, then triggers), so at most this grid and the one before it
  // run when the next call starts.

  if (warp == cons_warps) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&map_q) : "memory");
    }
    bool ok = true;
    const bool need_qs = DEC == kDecodeMaskPlanes;
    const uint32_t side_b = (uint32_t)(M * G * 4);
    if (!DOTS && p.sw_bulk && lane == 0) {
      if (!p.overlap) grid_dep_wait();
      const uint32_t bytes = (uint32_t)(R * G * 2);
      mbar_arrive_expect_tx(swbar, bytes);
      bulk_g2s(sw_s, p.scales + (size_t)n0 * G, bytes, swbar);
    }
    // Issue stage i: weights (unless already issued), q boxes, and with
    // stage 0 s_x and sum(q).  The arrival announces every byte of the stage
    // that has not been announced before, ahead of the copies it covers.
    auto issue = [&](int i, bool weights, bool inputs) {
      const int slot = i % p.ring;
      const int g0 = i * Gs, nb = min(Gs, G - g0), boxes = (nb + 3) / 4;
      uint8_t* st = ring + (size_t)slot * p.stage_bytes;
      if (lane != 0) return;
      const uint32_t wbytes = weights ? (uint32_t)(boxes * R * kBoxBytes) : 0u;
      if (!inputs) {
        mbar_expect_tx(&full[slot], wbytes);
      } else {
        const bool side = (i == 0) && p.sx_bulk;
        const uint32_t extra = side ? (DOTS ? 0u : side_b) + (need_qs ? side_b : 0u) : 0u;
        mbar_arrive_expect_tx(&full[slot], wbytes + (uint32_t)(M * Gs * kGroup) + extra);
        for (int m = 0; m < M; ++m)
          tma_load_2d(st + p.q_off + m * p.qbox_stride, &map_q, 0, m * G + g0, &full[slot]);
        if (side) {
          if (!DOTS) bulk_g2s(sx_s, p.sx, side_b, &full[slot]);
          if (need_qs) bulk_g2s(qs_s, p.qsum, side_b, &full[slot]);
        }
      }
      for (int b = 0; weights && b < boxes; ++b)
        tma_load_2d(st + b * p.box_stride, map, (g0 + 4 * b) * kGroupCodeBytes, n0, &full[slot]);
    };
    const int pre = p.overlap ? min(p.ring, p.stages_total) : 0;
    for (int i = 0; i < pre; ++i) issue(i, true, independent);
    grid_dep_wait();
    grid_dep_launch();
    for (int i = 0; i < p.stages_total; ++i) {
      const int slot = i % p.ring;
      if (i < pre) {
        if (!independent) issue(i, false, true);
        continue;
      }
      if (i >= p.ring) ok = ok && mbar_wait(&empty[slot], ((i / p.ring) - 1) & 1);
      issue(i, true, true);
    }
    if (!ok && lane == 0) report(p.status, PQ2_ERR_TIMEOUT);
    return;
  }

  // ------------------------------------------------------------ consumers
  // Reads before the grid dependency resolves: none by default, the weight
  // scales with the overlap flag, every input when the call is independent.
  if (!p.overlap) grid_dep_wait();
  if (!DOTS && !p.sw_bulk)
    preload_u16(reinterpret_cast<uint16_t*>(sw_s), p.scales + (size_t)n0 * G, R * G, tid,
                p.cons_threads);
  grid_dep_wait();
  grid_dep_launch();
  if (!p.sx_bulk) {
    if (!DOTS)
      preload_u32(reinterpret_cast<uint32_t*>(sx_s), reinterpret_cast<const uint32_t*>(p.sx),
                  M * G, tid, p.cons_threads);
    if (DEC == kDecodeMaskPlanes)
      preload_u32(reinterpret_cast<uint32_t*>(qs_s), reinterpret_cast<const uint32_t*>(p.qsum),
                  M * G, tid, p.cons_threads);
    named_bar_sync(1, p.cons_threads);
  }
  bool ok = true;
  if (!DOTS && p.sw_bulk) ok = ok && mbar_wait(swbar, 0);

  const int z = tid % S;
  const int r = tid / S;
  const bool active = r < R;
  const int sw_x = (r & 7) << 4;  // 128-byte swizzle of the code boxes: chunk ^= row % 8
  float yacc[M];
#pragma unroll
  for (int m = 0; m < M; ++m) yacc[m] = 0.0f;

  for (int i = 0; i < p.stages_total; ++i) {
    const int slot = i % p.ring;
    ok = ok && mbar_wait(&full[slot], (i / p.ring) & 1);
    const uint8_t* st = ring + (size_t)slot * p.stage_bytes;
    const int g0 = i * Gs;
    if (active && ok) {
      for (int l = z; l < Gs; l += S) {
        const int g = g0 + l;
        if (g >= G) break;
        const uint8_t* row = st + (l >> 2) * p.box_stride + r * kBoxBytes;
        const int lo = (l & 3) * 32;  // logical byte offset of the group in the box row
        int dot[M];
        group_dot<M, DEC>(row + (lo ^ sw_x), row + ((lo + 16) ^ sw_x),
                          reinterpret_cast<const int8_t*>(st + p.q_off) + l * kGroup,
                          p.qbox_stride, (l & 7) << 4, qs_s + g, G, dot);
        if (DOTS) {
#pragma unroll
          for (int m = 0; m < M; ++m) p.dots[((size_t)m * p.N + n0 + r) * G + g] = dot[m];
        } else {
          const float ws = __half2float(sw_s[r * G + g]);
#pragma unroll
          for (int m = 0; m < M; ++m) {
            float t = __fmul_rn(__int2float_rn(dot[m]), sx_s[m * G + g]);
            t = __fmul_rn(t, ws);
            yacc[m] = __fadd_rn(yacc[m], t);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
  if (!ok && lane == 0) report(p.status, PQ2_ERR_TIMEOUT);
  if constexpr (!DOTS) {
    // Combine the S split partials of each row (adjacent lanes) with a fixed
    // butterfly; lane z = 0 stores.  The order is a function of S alone.
#pragma unroll
    for (int m = 0; m < M; ++m)
      for (int off = S >> 1; off > 0; off >>= 1)
        yacc[m] = __fadd_rn(yacc[m], __shfl_xor_sync(0xffffffffu, yacc[m], off));
    if (active && z == 0) {
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const size_t o = (size_t)m * p.N + n0 + r;
        if (p.y_bf16)
          static_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(yacc[m]);
        else
          static_cast<float*>(p.y)[o] = yacc[m];
      }
    }
  }
}

// ------------------------------------------------------------------- host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// Tensor map over a row-major byte matrix [rows][row_bytes]; box = 128 bytes
// x box_rows, 128-byte swizzle.
bool encode_map(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes,
                int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)kBoxBytes, (cuuint32_t)std::max(box_rows, 1)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

int align_up(int v, int a) { return (v + a - 1) / a * a; }
int gcd(int a, int b) { return b ? gcd(b, a % b) : a; }

template <int M, int DEC, bool DOTS>
int launch_one(const CUtensorMap& hi, const CUtensorMap& lo, const CUtensorMap& qm,
               const MmvParams& p, int smem, cudaStream_t stream) {
  auto kern = mmv_kernel<M, DEC, DOTS>;
  static int configured = 0;  // largest dynamic smem size set so far
  if (smem > configured) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget + 1024) !=
        cudaSuccess)
      return PQ2_ERR_LAUNCH;
    configured = kSmemBudget + 1024;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.ctas);
  cfg.blockDim = dim3(p.cons_threads + 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, hi, lo, qm, p) != cudaSuccess) {
    cudaGetLastError();
    return PQ2_ERR_LAUNCH;
  }
  return PQ2_OK;
}

template <int DEC, bool DOTS>
int launch_m(int M, const CUtensorMap& hi, const CUtensorMap& lo, const CUtensorMap& qm,
             const MmvParams& p, int smem, cudaStream_t s) {
  switch (M) {
    case 1: return launch_one<1, DEC, DOTS>(hi, lo, qm, p, smem, s);
    case 2: return launch_one<2, DEC, DOTS>(hi, lo, qm, p, smem, s);
    case 3: return launch_one<3, DEC, DOTS>(hi, lo, qm, p, smem, s);
    case 4: return launch_one<4, DEC, DOTS>(hi, lo, qm, p, smem, s);
    case 5: return launch_one<5, DEC, DOTS>(hi, lo, qm, p, smem, s);
    case 6: return launch_one<6, DEC, DOTS>(hi, lo, qm, p, smem, s);
    case 7: return launch_one<7, DEC, DOTS>(hi, lo, qm, p, smem, s);
    case 8: return launch_one<8, DEC, DOTS>(hi, lo, qm, p, smem, s);
    default: return PQ2_ERR_SHAPE;
  }
}

}  // namespace

// Geometry: P = min(N, #SM) CTAs (more when a CTA would exceed 256 rows),
// R = ceil(N / P) rows for the largest CTA, and the split count S (a divisor
// of 32, so a row's splits share a warp) that best fills the consumer lanes
// (R*S of 32*ceil(R*S/32)) and the groups (G of S*ceil(G/S)) with at least
// ~6 warps.  A function of (N, K, SM count) only.
bool mmv_geometry(int64_t N, int64_t K, int sm_count, MmvGeometry* out) {
  if (N < 1 || K < kGroup || K % kGroup || sm_count < 1) return false;
  if (N > (int64_t)1 << 30 || K > (int64_t)1 << 24) return false;
  const int G = (int)(K / kGroup);
  int64_t ctas = std::min<int64_t>(N, sm_count);
  if ((N + ctas - 1) / ctas > kMaxBoxRows) ctas = (N + kMaxBoxRows - 1) / kMaxBoxRows;
  if (ctas > (1 << 30)) return false;
  const int R = (int)((N + ctas - 1) / ctas);
  int best_s = 1;
  double best = -1.0;
  for (int S = 1; S <= std::min(std::min(G, kMaxSplits), 16); S *= 2) {
    const int lanes = R * S;
    if (lanes > kMaxConsumerThreads) break;
    const int T = align_up(lanes, 32);
    const int steps = (G + S - 1) / S;
    const double eff = (double)lanes / T * ((double)G / ((double)S * steps));
    const double score = eff * std::min(1.0, T / 192.0);
    if (score > best + 1e-9) {
      best = score;
      best_s = S;
    }
  }
  out->ctas = (int)ctas;
  out->splits = best_s;
  out->rows_max = R;
  out->threads = align_up(R * best_s, 32);
  out->steps = (G + best_s - 1) / best_s;
  return true;
}

int launch_mmv(const int8_t* q, const float* sx, const int32_t* qsum, const uint8_t* codes,
               const uint16_t* scales, void* y, int y_dtype, int32_t* dots, int64_t M,
               int64_t N, int64_t K, int decode, int overlap, int sm_count, int32_t* status,
               cudaStream_t stream) {
  MmvGeometry geo;
  if (!mmv_geometry(N, K, sm_count, &geo)) return PQ2_ERR_SHAPE;
  MmvParams p{};
  p.q = q; p.sx = sx; p.qsum = qsum; p.scales = scales;
  p.y = y; p.dots = dots; p.status = status;
  p.N = (int)N; p.K = (int)K; p.G = (int)(K / kGroup);
  p.ctas = geo.ctas; p.splits = geo.splits; p.rows_max = geo.rows_max;
  p.cons_threads = geo.threads;
  p.overlap = overlap;
  p.y_bf16 = y_dtype == PQ2_BF16;
  p.sw_bulk = (K / kGroup) % 8 == 0 && reinterpret_cast<uintptr_t>(scales) % 16 == 0;
  {
    const bool a16 = (reinterpret_cast<uintptr_t>(sx) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(qsum) % 16 == 0);
    p.sx_bulk = a16 && ((M * (K / kGroup) * 4) % 16 == 0);
  }
  const int mi = (int)M, R = geo.rows_max, S = geo.splits, G = p.G;
  const int unit = 4 * S / gcd(4, S);
  p.box_stride = align_up(R * kBoxBytes, 1024);
  // fixed region: barriers, weight scales, s_x, sum(q)
  p.sw_off = align_up(2 * 8 * kMaxStages + 8, 128);
  p.sx_off = align_up(p.sw_off + G * R * 2, 16);
  p.qs_off = align_up(p.sx_off + mi * G * 4, 16);
  p.ring_off = align_up(p.qs_off + mi * G * 4, 1024);
  const int room = kSmemBudget - p.ring_off;
  // Stage: k units of lcm(4, S) groups, aiming at ~16-24 KB of codes.
  auto stage_bytes = [&](int gs) {
    return (gs / 4) * p.box_stride + mi * align_up(gs * kGroup, 1024);
  };
  int gs = unit;
  while (gs + unit <= std::max(unit, (G + 3) / 4 * 4) && stage_bytes(gs + unit) <= 24 * 1024 &&
         stage_bytes(gs + unit) * 3 <= room)
    gs += unit;
  p.stage_groups = gs;
  p.q_off = (gs / 4) * p.box_stride;
  p.qbox_stride = align_up(gs * kGroup, 1024);
  p.stage_bytes = stage_bytes(gs);
  p.stages_total = (G + gs - 1) / gs;
  if (room < p.stage_bytes) return PQ2_ERR_SHAPE;
  p.ring = std::min(std::min(p.stages_total, room / p.stage_bytes), kMaxStages);
  const int smem = 1024 + p.ring_off + p.ring * p.stage_bytes;  // + alignment slack

  CUtensorMap hi, lo, qm;
  const int rows_lo = (int)(N / geo.ctas);
  if (!encode_map(&hi, codes, N, K / 4, R) ||
      !encode_map(&lo, codes, N, K / 4, rows_lo > 0 ? rows_lo : R) ||
      !encode_map(&qm, q, M * (K / kGroup), kGroup, gs))
    return PQ2_ERR_LAUNCH;
  if (dots)
    return decode == kDecodeMaskPlanes
               ? launch_m<kDecodeMaskPlanes, true>(mi, hi, lo, qm, p, smem, stream)
               : launch_m<kDecodeAddXor, true>(mi, hi, lo, qm, p, smem, stream);
  return decode == kDecodeMaskPlanes
             ? launch_m<kDecodeMaskPlanes, false>(mi, hi, lo, qm, p, smem, stream)
             : launch_m<kDecodeAddXor, false>(mi, hi, lo, qm, p, smem, stream);
}

}  // namespace pq2
