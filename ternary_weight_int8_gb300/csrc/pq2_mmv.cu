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

constexpr int kMaxConsumerThreads = 288;
constexpr int kRowsPerThread = 2;         // rows sharing each q load
constexpr int kMaxBlock = kMaxConsumerThreads + 32;
constexpr int kMaxSplits = 64;
constexpr int kMaxBoxRows = 256;          // TMA box height limit
constexpr int kSmemBudget = 110 * 1024;   // two CTAs per SM
constexpr int kSoloSmem = 120 * 1024;     // one CTA per SM (dynamic request)
constexpr int kMaxDynSmem = 227 * 1024;   // opt-in dynamic shared memory per block
constexpr int kMaxStages = 48;
// Tensor-core consumer: 8 warps, each owning one split (two when S = 16) and
// its 16-row tiles (a share of them when S < 8): at most kTcTiles tiles of
// one split, or kTcTiles2 tiles of each of two.
constexpr int kTcWarps = 8;
constexpr int kTcTiles = 5;
constexpr int kTcTiles2 = 3;
constexpr int kTcUnits = 6;  // accumulators: max(kTcTiles, 2 * kTcTiles2)
constexpr int kTcBlock = (kTcWarps + 1) * 32;
constexpr int kBoxBytes = 128;            // 4 groups of 32 code bytes
// Shared-memory offset of the abort flag: after the largest barrier region
// (full[kMaxStages], empty[kMaxStages], the scale barrier), before sw_off.
constexpr int kAbortOff = 2 * 8 * kMaxStages + 8;

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
  int groups_per_thread;  // Gs / S when that is 1 or 2 (S >= 4), else 0
  int box_stride;         // bytes per box in shared memory (1024-aligned)
  int stage_bytes;        // boxes + q region
  int q_off;              // q region inside a stage
  int qbox_stride;        // bytes per column's q box inside a stage (1024-aligned)
  int sw_off, sx_off, qs_off, ring_off;
  int part_off;           // tensor-core path: split partials [S][R][M] fp32
  int y_bf16;
  int overlap;            // 1: stream weights before the grid dependency
                          // resolves; 2: stream every input before it
  int sw_bulk;            // weight-scale slab arrives by one bulk copy (G % 8 == 0)
  int side16;             // s_x and sum(q) copied in 16-byte pieces (aligned)
  // Gated output (gate/up): CTA rows n0.. are outputs; gate rows n0.. and up
  // rows up_row + n0.. of the weights, the up boxes up_smem rows after the
  // gate boxes (a multiple of 8, so both keep the 128-byte swizzle keys).
  int gated;
  int up_row;             // I = N / 2: first up row of the weights
  int up_smem;            // rows between a gate box and its up box in smem
  int y_ld;               // output row stride (N, or I when gated)
  // Test knobs of the bounded-wait path (pq2_debug_mmv_drop_arrival): consumer
  // warp 0 skips its release of stage drop_stage (-1: none), and the
  // producer's wait for a free ring slot gives up after empty_limit clocks.
  int drop_stage;
  long long empty_limit;
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

__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Gated output of the gate/up projection: silu(g) * u = g / (1 + e^-g) * u
// in fp32, each operation rounded to nearest (expf is CUDA's, 2 ulp).
__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the arrival is counted in advance, so the phase waits for it).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Shared-memory loads by 32-bit shared address.  The operands live at
// run-time offsets from the aligned dynamic shared base; explicit ld.shared
// keeps every read on the shared-memory path.
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// Tensor-core GEMV pieces (decoder kDecodeTensor).
//
// A code word holds 16 weights: bits 2f..2f+1 of its low half are weight
// 16w + f and of its high half weight 16w + 8 + f (f = 0..7).  OR-ed into
// fp16 1024 (0x6400), a field masked in place at bit 2f' is the exact value
// 1024 + c * 4^f'; fields f = 0..4 sit at f' = f, fields 5..7 at f' = f - 3
// after one shift of the word by 6.  h[f] is then a half pair (weight 16w + f,
// weight 16w + 8 + f), one LOP3 each.  The activations arrive divided by the
// same power of four (PQ2_Q_MMV16), so every product is 1024 q / 4^f' + c q,
// an integer, and the fp32 accumulator holds the exact sum (|sum| < 2^22).
__device__ __forceinline__ void decode_f16_fields(uint32_t w, uint32_t (&h)[8]) {
  constexpr uint32_t kMagic = 0x64006400u;
  h[0] = (w & 0x00030003u) | kMagic;
  h[1] = (w & 0x000C000Cu) | kMagic;
  h[2] = (w & 0x00300030u) | kMagic;
  h[3] = (w & 0x00C000C0u) | kMagic;
  h[4] = (w & 0x03000300u) | kMagic;
  const uint32_t s = w >> 6;
  h[5] = (s & 0x00300030u) | kMagic;
  h[6] = (s & 0x00C000C0u) | kMagic;
  h[7] = (s & 0x03000300u) | kMagic;
}

// d += A * B on a 16 x 8 x 16 tile, fp16 operands, fp32 accumulation.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16 bytes from global memory through the read-only path.
__device__ __forceinline__ uint4 ldg_nc16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Combine the S split partials of one output (S a power of two, at most 16)
// in the order of the dp4a consumer's xor butterfly, as lane 0 sees it: at
// each step v[z] += v[z + off] for z < off, off = S/2 .. 1.
template <int S>
__device__ __forceinline__ float split_tree(const float* part, int stride) {
  float v[S];
#pragma unroll
  for (int z = 0; z < S; ++z) v[z] = part[z * stride];
#pragma unroll
  for (int off = S >> 1; off > 0; off >>= 1)
#pragma unroll
    for (int z = 0; z < off; ++z) v[z] = __fadd_rn(v[z], v[z + off]);
  return v[0];
}

// Exact int32 dots of one 128-group for RP weight rows and columns
// m0 .. m0+MB-1.  Each 16-byte chunk of q is loaded once and used for all RP
// rows, which keeps shared-memory traffic (q is common to every row) low.
//   c0[r], c1[r] : shared addresses of row r's two 16-byte halves of the
//                  group's code bytes (swizzled)
// Plane s of code word w (bytes 4w..4w+3 of the group) holds the codes of
// weights 16w + 4b + s (b = 0..3); in plane order those activations are the
// 4 bytes at s*32 + 4w, so one 32-bit q word meets one 32-bit plane word.
//   qz     : shared address of the group's box row of q for column m0 (128
//            bytes, 128-byte swizzled with key qsw); column m0+m at
//            qz + m * q_mstride
//   qs     : shared address of sum(q) of the group for column m0; column
//            m0+m at qs + m * qs_mstride
template <int MB, int RP, int DEC>
__device__ __forceinline__ void group_dot(const uint32_t (&c0)[RP], const uint32_t (&c1)[RP],
                                          uint32_t qz, int q_mstride, int qsw, uint32_t qs,
                                          int qs_mstride, int (&dot)[RP][MB]) {
  // Independent accumulator chains: one per plane when few (instruction-level
  // parallelism), else one per plane parity (registers).  Masked planes:
  // even planes accumulate code * q, odd planes 4 * code * q.
  constexpr int NA = MB * RP <= 4 ? 4 : 2;
  int acc[RP][NA][MB];
#pragma unroll
  for (int r = 0; r < RP; ++r)
#pragma unroll
    for (int a = 0; a < NA; ++a)
#pragma unroll
      for (int m = 0; m < MB; ++m) acc[r][a][m] = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t cw[RP][4];
#pragma unroll
    for (int r = 0; r < RP; ++r) {
      const uint4 c = lds128(h ? c1[r] : c0[r]);
      cw[r][0] = c.x; cw[r][1] = c.y; cw[r][2] = c.z; cw[r][3] = c.w;
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      if (s == 2) {
        // Planes 2 and 3 sit where planes 0 and 1 were once the words are
        // shifted down by 4 bits.
#pragma unroll
        for (int r = 0; r < RP; ++r)
#pragma unroll
          for (int w = 0; w < 4; ++w) cw[r][w] >>= 4;
      }
      uint4 qv[MB];
#pragma unroll
      for (int m = 0; m < MB; ++m)
        qv[m] = lds128(qz + m * q_mstride + ((s * 32 + 16 * h) ^ qsw));
#pragma unroll
      for (int r = 0; r < RP; ++r)
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t wv;
          if (DEC == kDecodeAddXor) {
            // Spread: the four codes of plane s, one per byte (values 0..3).
            // +0x7F7F7F7F cannot carry between bytes; ^0x80808080 maps
            // 127/128/129/130 to the signed bytes -1/0/+1/+2.
            const uint32_t spread = (cw[r][w] >> (2 * (s & 1))) & 0x03030303u;
            wv = (spread + 0x7F7F7F7Fu) ^ 0x80808080u;
          } else {
            // Masked plane: bytes code (s even) or 4 * code (s odd), unsigned.
            wv = cw[r][w] & ((s & 1) ? 0x0C0C0C0Cu : 0x03030303u);
          }
#pragma unroll
          for (int m = 0; m < MB; ++m) {
            const int qw =
                (int)(w == 0 ? qv[m].x : w == 1 ? qv[m].y : w == 2 ? qv[m].z : qv[m].w);
            int& a = acc[r][NA == 4 ? s : (s & 1)][m];
            a = (DEC == kDecodeAddXor) ? __dp4a((int)wv, qw, a) : dp4a_us(wv, qw, a);
          }
        }
    }
  }
#pragma unroll
  for (int m = 0; m < MB; ++m) {
    // `odd` is exactly 4 * sum(code * q) over planes 1 and 3 (masked planes):
    // shift it back, then remove the codes' -1 offset with the group sum of q.
    const int qsm = DEC == kDecodeAddXor ? 0 : (int)lds32(qs + m * qs_mstride);
#pragma unroll
    for (int r = 0; r < RP; ++r) {
      const int even = NA == 4 ? acc[r][0][m] + acc[r][2][m] : acc[r][0][m];
      const int odd = NA == 4 ? acc[r][1][m] + acc[r][3][m] : acc[r][1][m];
      dot[r][m] = DEC == kDecodeAddXor ? even + odd : even + (odd >> 2) - qsm;
    }
  }
}

// Partial dots of one 128-group over its NSUB activation groups of
// A = 128 / NSUB elements (KE Test 9), masked-plane decoder: activation group
// u covers weights [uA, uA + A), i.e. half h = u / (NSUB / 2) of the group's
// code bytes and, for A = 32, code words 2v, 2v + 1 of that half
// (v = u % 2).  Each partial is finished as in group_dot with its own
// sum(q) and handed to emit(u, dot[RP][MB]) in increasing u.
//   qs : shared address of sum(q) of activation group 0 of this 128-group
//        for column 0; group u of column m at qs + (m * qs_mstride) + 4u
template <int MB, int RP, int NSUB, typename Emit>
__device__ __forceinline__ void group_dot_sub(const uint32_t (&c0)[RP], const uint32_t (&c1)[RP],
                                              uint32_t qz, int q_mstride, int qsw, uint32_t qs,
                                              int qs_mstride, Emit&& emit) {
  static_assert(NSUB == 2 || NSUB == 4, "activation groups of 64 or 32");
  constexpr int HS = NSUB / 2;  // activation groups per half
  constexpr int WPS = 4 / HS;   // code words of a half per activation group
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t cw[RP][4];
#pragma unroll
    for (int r = 0; r < RP; ++r) {
      const uint4 c = lds128(h ? c1[r] : c0[r]);
      cw[r][0] = c.x; cw[r][1] = c.y; cw[r][2] = c.z; cw[r][3] = c.w;
    }
    // even planes accumulate code * q, odd planes 4 * code * q
    int acc[HS][RP][2][MB];
#pragma unroll
    for (int v = 0; v < HS; ++v)
#pragma unroll
      for (int r = 0; r < RP; ++r)
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int m = 0; m < MB; ++m) acc[v][r][a][m] = 0;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      if (s == 2) {
#pragma unroll
        for (int r = 0; r < RP; ++r)
#pragma unroll
          for (int w = 0; w < 4; ++w) cw[r][w] >>= 4;
      }
      uint4 qv[MB];
#pragma unroll
      for (int m = 0; m < MB; ++m)
        qv[m] = lds128(qz + m * q_mstride + ((s * 32 + 16 * h) ^ qsw));
#pragma unroll
      for (int r = 0; r < RP; ++r)
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t wv = cw[r][w] & ((s & 1) ? 0x0C0C0C0Cu : 0x03030303u);
#pragma unroll
          for (int m = 0; m < MB; ++m) {
            const int qw =
                (int)(w == 0 ? qv[m].x : w == 1 ? qv[m].y : w == 2 ? qv[m].z : qv[m].w);
            int& a = acc[w / WPS][r][s & 1][m];
            a = dp4a_us(wv, qw, a);
          }
        }
    }
#pragma unroll
    for (int v = 0; v < HS; ++v) {
      const int u = h * HS + v;
      int dot[RP][MB];
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        const int qsm = (int)lds32(qs + m * qs_mstride + 4 * u);
#pragma unroll
        for (int r = 0; r < RP; ++r)
          dot[r][m] = acc[v][r][0][m] + (acc[v][r][1][m] >> 2) - qsm;
      }
      emit(u, dot);
    }
  }
}

// Up to four columns two CTAs fit on an SM (a call overlaps the next one);
// more columns need the registers of one CTA per SM.
template <int M, int DEC, bool DOTS, int NSUB = 1>
__global__ void __launch_bounds__(DEC == kDecodeTensor ? kTcBlock : kMaxBlock,
                                  (M <= 4 || DEC == kDecodeTensor) ? 2 : 1)
    mmv_kernel(const __grid_constant__ CUtensorMap map_hi,
               const __grid_constant__ CUtensorMap map_lo,
               const MmvParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // The 128-byte swizzle needs 1024-byte aligned boxes.
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + p.ring;
  uint64_t* swbar = empty + p.ring;
  // Set by the producer when it stops early (a wait gave up), once every
  // copy it issued has landed; the consumers' waits then give up too.
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
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
  // An independent call reads no output of earlier kernels: it waits for
  // them only before storing y.
  const bool independent = !DOTS && p.overlap >= 2;

  if (tid == 0) {
    for (int s = 0; s < p.ring; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], cons_warps);
    }
    mbar_init(swbar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // Release the next kernel on the stream now.  Its CTAs then take the SM
  // slots that this grid's predecessor frees, one by one, which keeps the
  // grids spread one CTA per SM; released later, a grid finds SMs with
  // uneven free slots and some SMs receive two of its CTAs.
  grid_dep_launch();

  if (warp == cons_warps) {
    // ---------------------------------------------------------- producer
    if (lane == 0) asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
    bool ok = true;
    const bool need_qs = DEC != kDecodeAddXor;  // sum(q), or the tensor path's corrections
    if (!DOTS && p.sw_bulk && lane == 0) {
      if (!p.overlap) grid_dep_wait();
      const uint32_t bytes = (uint32_t)(R * G * 2);
      mbar_arrive_expect_tx(swbar, p.gated ? 2 * bytes : bytes);
      bulk_g2s(sw_s, p.scales + (size_t)n0 * G, bytes, swbar);
      if (p.gated)
        bulk_g2s(sw_s + (size_t)p.up_smem * G, p.scales + (size_t)(p.up_row + n0) * G, bytes,
                 swbar);
    }
    // Weights of stage i: TMA boxes announced on the stage barrier without
    // arriving, so the stage completes only once its inputs are issued too.
    auto issue_weights = [&](int i) {
      if (lane != 0) return;
      const int slot = i % p.ring;
      const int g0 = i * Gs, boxes = (min(Gs, G - g0) + 3) / 4;
      uint8_t* st = ring + (size_t)slot * p.stage_bytes;
      mbar_expect_tx(&full[slot], (uint32_t)(boxes * R * kBoxBytes * (p.gated ? 2 : 1)));
      for (int b = 0; b < boxes; ++b) {
        tma_load_2d(st + b * p.box_stride, map, (g0 + 4 * b) * kGroupCodeBytes, n0, &full[slot]);
        if (p.gated)
          tma_load_2d(st + b * p.box_stride + p.up_smem * kBoxBytes, map,
                      (g0 + 4 * b) * kGroupCodeBytes, p.up_row + n0, &full[slot]);
      }
    };
    // Inputs of stage i (and with stage 0 s_x and sum(q)), copied by the
    // whole warp with cp.async rather than TMA: the SM's TMA unit serves its
    // requests in order, and these few small copies must not queue behind
    // the weights that the next call's CTA on this SM prefetches.  q rows
    // land in the same 128-byte swizzled layout the consumers read.
    auto issue_inputs = [&](int i) {
      const int slot = i % p.ring;
      const int g0 = i * Gs, nb = min(Gs, G - g0);
      const uint32_t dst0 = smem_u32(ring) + slot * p.stage_bytes + p.q_off;
      const int8_t* src0 = p.q + (size_t)g0 * kGroup;
      // Lane = 16-byte chunk c of row l of a block of four group rows; no
      // division in the address arithmetic.
      const int c = lane & 7;
      if (DEC != kDecodeTensor)  // the tensor-core consumers read q themselves
        for (int m = 0; m < M; ++m)
          for (int l = lane >> 3; l < nb; l += 4)
            cp_async16(dst0 + m * p.qbox_stride + l * kGroup + ((c ^ (l & 7)) << 4),
                       src0 + ((size_t)m * G + l) * kGroup + c * 16);
      if (i == 0) {
        if (p.side16) {
          for (int idx = 4 * lane; idx < M * G * NSUB; idx += 128) {
            if (!DOTS) cp_async16(smem_u32(sx_s + idx), p.sx + idx);
            if (need_qs) cp_async16(smem_u32(qs_s + idx), p.qsum + idx);
          }
        } else {
          for (int idx = lane; idx < M * G * NSUB; idx += 32) {
            if (!DOTS) cp_async4(sx_s + idx, p.sx + idx);
            if (need_qs) cp_async4(qs_s + idx, p.qsum + idx);
          }
        }
      }
      cp_async_mbar_arrive(&full[slot]);
      __syncwarp();
      warp_arrive(&full[slot]);
    };
    // Stages that fit the ring go out at once: each stage's weights and then
    // its inputs (an independent call), or every stage's weights now and the
    // inputs once the grid dependency resolves (weights-only overlap).
    const int pre = p.overlap ? min(p.ring, p.stages_total) : 0;
    for (int i = 0; i < pre; ++i) {
      issue_weights(i);
      if (independent) issue_inputs(i);
    }
    if (!independent) grid_dep_wait();
    for (int i = 0; i < p.stages_total; ++i) {
      if (i < pre) {
        if (!independent) issue_inputs(i);
        continue;
      }
      if (i >= p.ring) {
        bool freed = true;
        if (lane == 0)
          freed = mbar_wait_until(&empty[i % p.ring], ((i / p.ring) - 1) & 1, p.empty_limit,
                                  nullptr);
        freed = __shfl_sync(0xffffffffu, freed, 0);
        if (!freed) {
          // Stop issuing: the slot may still be read.  Copies of the last
          // `ring` issued stages may still be landing (earlier stages' slots
          // were released, so theirs have); wait for them before the
          // consumers are told to stop, so that no copy outlives the CTA.
          ok = false;
          if (lane == 0) {
            for (int j = max(0, i - p.ring); j < i; ++j)
              mbar_wait(&full[j % p.ring], (j / p.ring) & 1);
            *abort_flag = 1;
            __threadfence_block();
          }
          __syncwarp();
          break;
        }
      }
      issue_weights(i);
      issue_inputs(i);
    }
    if (!ok && lane == 0) report(p.status, PQ2_ERR_TIMEOUT);
    return;
  }

  // ------------------------------------------------------------ consumers
  // Reads before the grid dependency resolves: none by default, the weight
  // scales with the overlap flag; q, s_x and sum(q) arrive through the stage
  // barriers.
  if (!p.overlap) grid_dep_wait();
  if (!DOTS && !p.sw_bulk) {
    preload_u16(reinterpret_cast<uint16_t*>(sw_s), p.scales + (size_t)n0 * G, R * G, tid,
                p.cons_threads);
    if (p.gated)
      preload_u16(reinterpret_cast<uint16_t*>(sw_s) + (size_t)p.up_smem * G,
                  p.scales + (size_t)(p.up_row + n0) * G, R * G, tid, p.cons_threads);
    named_bar_sync(1, p.cons_threads);
  }
  bool ok = true;
  if (!DOTS && p.sw_bulk) ok = ok && mbar_wait(swbar, 0);

  if constexpr (DEC == kDecodeTensor) {
    // ---------------------------------------------- tensor-core consumers
    // Warp w owns the splits z = w % gstep + gstep * ss (ss < S / gstep; two
    // when S = 16) and, when S < 8, the 16-row tiles tfirst + tw * ts.  For
    // each of its groups, ascending (the split's order), it loads that
    // group's B fragments (lane 4c + t: column c, 32 fp16 values) straight
    // from global memory (every CTA reads the same q) and, per tile, decodes
    // four code words (rows g, g + 8; words t, t + 4), runs eight mma.sync and
    // adds the scaled exact dots to its split partials.
    const __half* qf = reinterpret_cast<const __half*>(p.q);
    if (p.overlap == 1) grid_dep_wait();  // q is read directly, not via the stages
    const int g8 = lane >> 2, t4 = lane & 3;
    const int gstep = S < kTcWarps ? S : kTcWarps;
    const int gfirst = warp % gstep;
    const int tw = S < kTcWarps ? kTcWarps / S : 1;
    const int tfirst = S < kTcWarps ? warp / S : 0;
    const int nt = (R + 15) >> 4;
    const int nts = tfirst < nt ? (nt - tfirst + tw - 1) / tw : 0;
    const int nss = S / gstep;
    const int c0 = 2 * t4, c1 = c0 + 1;
    const uint32_t ring_s = smem_u32(ring), sw_base = smem_u32(sw_s);
    // Split partials per unit: tile ts of the first split at [ts]; with two
    // splits (S = 16, where a CTA holds at most 36 rows: 3 tiles) tile ts of
    // the second at [kTcTiles2 + ts].
    float yacc[kTcUnits][4];
#pragma unroll
    for (int u = 0; u < kTcUnits; ++u)
#pragma unroll
      for (int k = 0; k < 4; ++k) yacc[u][k] = 0.0f;
    uint32_t b[16];
    const bool recycle = p.stages_total > p.ring;
    for (int i = 0; i < p.stages_total; ++i) {
      const int slot = i % p.ring;
      ok = ok && mbar_wait_until(&full[slot], (i / p.ring) & 1, kWaitLimitCycles, abort_flag);
      const uint32_t st_s = ring_s + slot * p.stage_bytes;
      const int g0 = i * Gs;
      if (ok) {
#pragma unroll 1
        for (int l = gfirst; l < Gs && g0 + l < G; l += gstep) {
          const int g = g0 + l;
          if (g8 < M) {
            const uint8_t* src =
                reinterpret_cast<const uint8_t*>(qf + ((size_t)g8 * G + g) * kGroup) + t4 * 64;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint4 v = ldg_nc16(src + 16 * c);
              b[4 * c] = v.x; b[4 * c + 1] = v.y; b[4 * c + 2] = v.z; b[4 * c + 3] = v.w;
            }
          } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) b[c] = 0u;
          }
          const int ss = (g % S) / gstep;
          const uint32_t box = st_s + (l >> 2) * p.box_stride;
          const int ch = (l & 3) * 2;
          float xs0 = 0.0f, xs1 = 0.0f, cr0 = 0.0f, cr1 = 0.0f;
          if (c0 < M) {
            xs0 = sx_s[c0 * G + g];
            cr0 = (float)qs_s[c0 * G + g];
          }
          if (c1 < M) {
            xs1 = sx_s[c1 * G + g];
            cr1 = (float)qs_s[c1 * G + g];
          }
#pragma unroll
          for (int ts = 0; ts < kTcTiles; ++ts) {
            if (ts >= nts) break;
            const int tau = tfirst + ts * tw;
            const int r0 = min(tau * 16 + g8, R - 1), r1 = min(tau * 16 + g8 + 8, R - 1);
            const uint32_t a0 = box + r0 * kBoxBytes + 4 * t4, a1 = box + r1 * kBoxBytes + 4 * t4;
            const uint32_t w00 = lds32(a0 + ((ch ^ (r0 & 7)) << 4));
            const uint32_t w01 = lds32(a0 + (((ch + 1) ^ (r0 & 7)) << 4));
            const uint32_t w10 = lds32(a1 + ((ch ^ (r1 & 7)) << 4));
            const uint32_t w11 = lds32(a1 + (((ch + 1) ^ (r1 & 7)) << 4));
            float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            {
              uint32_t ha[8], hb[8];
              decode_f16_fields(w00, ha);
              decode_f16_fields(w10, hb);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                mma_f16(d, ha[2 * j], hb[2 * j], ha[2 * j + 1], hb[2 * j + 1], b[2 * j],
                        b[2 * j + 1]);
            }
            {
              uint32_t ha[8], hb[8];
              decode_f16_fields(w01, ha);
              decode_f16_fields(w11, hb);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                mma_f16(d, ha[2 * j], hb[2 * j], ha[2 * j + 1], hb[2 * j + 1], b[8 + 2 * j],
                        b[8 + 2 * j + 1]);
            }
            // d: (row tau16 + g8, columns c0, c1), (row + 8, c0, c1); the
            // exact dot is d minus the column's correction (exact in fp32).
            if constexpr (DOTS) {
              const int rr[2] = {tau * 16 + g8, tau * 16 + g8 + 8};
              const float cr[2] = {cr0, cr1};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int row = rr[k >> 1], col = c0 + (k & 1);
                if (row < R && col < M)
                  p.dots[((size_t)col * p.N + n0 + row) * G + g] =
                      (int)__fsub_rn(d[k], cr[k & 1]);
              }
            } else {
              const float ws0 =
                  __half2float(__ushort_as_half((uint16_t)lds16(sw_base + (r0 * G + g) * 2)));
              const float ws1 =
                  __half2float(__ushort_as_half((uint16_t)lds16(sw_base + (r1 * G + g) * 2)));
              float tv[4];
              tv[0] = __fmul_rn(__fmul_rn(__fsub_rn(d[0], cr0), xs0), ws0);
              tv[1] = __fmul_rn(__fmul_rn(__fsub_rn(d[1], cr1), xs1), ws0);
              tv[2] = __fmul_rn(__fmul_rn(__fsub_rn(d[2], cr0), xs0), ws1);
              tv[3] = __fmul_rn(__fmul_rn(__fsub_rn(d[3], cr1), xs1), ws1);
              if (ss == 0) {
#pragma unroll
                for (int k = 0; k < 4; ++k) yacc[ts][k] = __fadd_rn(yacc[ts][k], tv[k]);
              } else if (ts < kTcTiles2) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  yacc[kTcTiles2 + ts][k] = __fadd_rn(yacc[kTcTiles2 + ts][k], tv[k]);
              }
            }
          }
        }
      }
      if (recycle) {
        __syncwarp();
        warp_arrive_if(!(i == p.drop_stage && warp == 0), &empty[slot]);
      }
    }
    if (!ok && lane == 0) report(p.status, PQ2_ERR_TIMEOUT);
    if constexpr (!DOTS) {
      // part[z][row][m]: every split's partial of every output of the CTA
      float* part = reinterpret_cast<float*>(smem + p.part_off);
#pragma unroll
      for (int u = 0; u < kTcUnits; ++u) {
        const int ss = nss == 1 ? 0 : u / kTcTiles2;
        const int ts = nss == 1 ? u : u - kTcTiles2 * ss;
        if (ts >= nts || (nss == 1 && u >= kTcTiles)) continue;
        const int z = gfirst + ss * gstep;
        const int tau = tfirst + ts * tw;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int row = tau * 16 + g8 + 8 * (k >> 1), col = c0 + (k & 1);
          if (row < R && col < M) part[((size_t)z * R + row) * M + col] = yacc[u][k];
        }
      }
      named_bar_sync(1, p.cons_threads);  // every partial is in place
      grid_dep_wait();  // earlier kernels may still read or write y
      for (int o = tid; o < R * M; o += p.cons_threads) {
        const int row = o / M, m = o - row * M;
        const float* src = part + (size_t)row * M + m;
        const int stride = R * M;
        float v;
        switch (S) {
          case 1: v = split_tree<1>(src, stride); break;
          case 2: v = split_tree<2>(src, stride); break;
          case 4: v = split_tree<4>(src, stride); break;
          case 8: v = split_tree<8>(src, stride); break;
          default: v = split_tree<16>(src, stride); break;
        }
        const size_t off = (size_t)m * p.y_ld + n0 + row;
        if (p.y_bf16)
          static_cast<__nv_bfloat16*>(p.y)[off] = __float2bfloat16_rn(v);
        else
          static_cast<float*>(p.y)[off] = v;
      }
    }
  } else {

  // Thread t owns split z = t % S and the RP rows rb, rb + H, rb + 2H ..
  // (rb = t / S, H = ceil(R / RP)).  A warp then reads code rows with
  // consecutive indices, whose 128-byte swizzle keys (row % 8) differ in the
  // low bit, so its 16-byte code loads spread over all eight chunk slots of
  // a 128-byte line (rows 2rb, 2rb + 1 would leave half the slots, and the
  // banks behind them, unused).  A row beyond R is a duplicate of row R-1,
  // computed but never stored.  Gated: the two rows are gate row rb and
  // up row rb (up_smem rows further in shared memory), for output rb.
  constexpr int RP = kRowsPerThread;
  static_assert(RP == 2, "the gated output pairs a thread's two rows");
  const int z = tid % S;
  const int rb = tid / S;
  const int H = p.gated ? p.up_smem : (R + RP - 1) / RP;
  const int Rv = p.gated ? H + R : R;  // rows beyond Rv - 1 do not exist
  int rows[RP];
  bool valid[RP];
#pragma unroll
  for (int r = 0; r < RP; ++r) {
    valid[r] = (p.gated ? rb < R : rb < H) && rb + r * H < Rv;
    rows[r] = min(rb + r * H, Rv - 1);
  }
  const bool active = valid[0];
  const uint32_t ring_s = smem_u32(ring), sw_base = smem_u32(sw_s);
  const uint32_t sx_base = smem_u32(sx_s), qs_base = smem_u32(qs_s);
  float yacc[RP][M];
#pragma unroll
  for (int r = 0; r < RP; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) yacc[r][m] = 0.0f;

  // Scale and accumulate the dots of columns m0 .. m0+MB-1 in the method's
  // order: t = (float(dot) * s_x) * s_w, y += t (activation group u of the
  // 128-group g when NSUB > 1).
  constexpr int GA_PER_G = NSUB;
  auto consume = [&](auto& dot, int m0, int g, int u) {
    constexpr int MB = sizeof(dot[0]) / sizeof(int);
    if constexpr (DOTS) {
#pragma unroll
      for (int r = 0; r < RP; ++r)
        if (valid[r])
#pragma unroll
          for (int m = 0; m < MB; ++m)
            p.dots[((size_t)(m0 + m) * p.N + n0 + rows[r]) * G * NSUB + g * NSUB + u] =
                dot[r][m];
    } else {
      float ws[RP];
#pragma unroll
      for (int r = 0; r < RP; ++r)
        ws[r] = __half2float(__ushort_as_half((uint16_t)lds16(sw_base + (rows[r] * G + g) * 2)));
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        const float xs =
            __uint_as_float(lds32(sx_base + (((m0 + m) * G + g) * GA_PER_G + u) * 4));
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          float t = __fmul_rn(__int2float_rn(dot[r][m]), xs);
          t = __fmul_rn(t, ws[r]);
          yacc[r][m0 + m] = __fadd_rn(yacc[r][m0 + m], t);
        }
      }
    }
  };

  // One group of the stage at shared address st_s: its dots for every
  // column, scaled and accumulated.
  auto do_group = [&](uint32_t st_s, int l, int g) {
    const int lo = (l & 3) * 32;  // logical byte offset of the group in the box row
    uint32_t c0[RP], c1[RP];
#pragma unroll
    for (int r = 0; r < RP; ++r) {
      // 128-byte swizzle of the code boxes: 16-byte chunk ^= row % 8
      const uint32_t rowa = st_s + (l >> 2) * p.box_stride + rows[r] * kBoxBytes;
      const int sw = (rows[r] & 7) << 4;
      c0[r] = rowa + (lo ^ sw);
      c1[r] = rowa + ((lo + 16) ^ sw);
    }
    const uint32_t qz = st_s + p.q_off + l * kGroup;
    const int qsw = (l & 7) << 4;
    // Columns in blocks of at most four keep the accumulators in registers.
    constexpr int MA = M <= 4 ? M : 4;
    if constexpr (NSUB > 1) {
      static_assert(M <= 4 && DEC == kDecodeMaskPlanes, "activation groups: M <= 4, planes");
      group_dot_sub<M, RP, NSUB>(c0, c1, qz, p.qbox_stride, qsw, qs_base + g * NSUB * 4,
                                 G * NSUB * 4,
                                 [&](int u, auto& dot) { consume(dot, 0, g, u); });
    } else {
      {
        int dot[RP][MA];
        group_dot<MA, RP, DEC>(c0, c1, qz, p.qbox_stride, qsw, qs_base + g * 4, G * 4, dot);
        consume(dot, 0, g, 0);
      }
      if constexpr (M > 4) {
        int dot[RP][M - 4];
        group_dot<M - 4, RP, DEC>(c0, c1, qz + 4 * p.qbox_stride, p.qbox_stride, qsw,
                                  qs_base + (4 * G + g) * 4, G * 4, dot);
        consume(dot, 4, g, 0);
      }
    }
  };

  // A thread's groups in a stage are z + j*S for j < Gs/S.  The geometry
  // makes that count 1 or 2 whenever S >= 4; up to two columns those cases
  // run as straight-line code (a run-time loop here measurably slows the
  // latency-bound stage); smaller S (tiny K) takes the general loop.
  const int gpt = p.groups_per_thread;
  const bool recycle = p.stages_total > p.ring;
  for (int i = 0; i < p.stages_total; ++i) {
    const int slot = i % p.ring;
    ok = ok && mbar_wait_until(&full[slot], (i / p.ring) & 1, kWaitLimitCycles, abort_flag);
    const uint32_t st_s = ring_s + slot * p.stage_bytes;
    const int g0 = i * Gs;
    if (active && ok) {
      if constexpr (M >= 3) {
        // One copy of the (large) group code: with three copies, instruction
        // fetch stalled these kernels, above all when calls of different M
        // alternate (measured 8-12 % per call).
#pragma unroll 1
        for (int l = z; l < Gs && g0 + l < G; l += S) do_group(st_s, l, g0 + l);
      } else if (gpt == 1) {
        if (g0 + z < G) do_group(st_s, z, g0 + z);
      } else if (gpt == 2) {
        if (g0 + z < G) do_group(st_s, z, g0 + z);
        if (g0 + z + S < G) do_group(st_s, z + S, g0 + z + S);
      } else {
        for (int l = z; l < Gs && g0 + l < G; l += S) do_group(st_s, l, g0 + l);
      }
    }
    if (recycle) {
      __syncwarp();
      warp_arrive_if(!(i == p.drop_stage && warp == 0), &empty[slot]);
    }
  }
  if (!ok && lane == 0) report(p.status, PQ2_ERR_TIMEOUT);
  if constexpr (!DOTS) {
    // Combine the S split partials of each row (adjacent lanes) with a fixed
    // butterfly; lane z = 0 stores.  The order is a function of S alone.
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
      for (int m = 0; m < M; ++m)
        for (int off = S >> 1; off > 0; off >>= 1)
          yacc[r][m] = __fadd_rn(yacc[r][m], __shfl_xor_sync(0xffffffffu, yacc[r][m], off));
    grid_dep_wait();  // earlier kernels may still read or write y
    if (z == 0 && p.gated) {
      if (valid[0]) {
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const size_t o = (size_t)m * p.y_ld + n0 + rb;
          const float v = silu_mul(yacc[0][m], yacc[1][m]);
          if (p.y_bf16)
            static_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(v);
          else
            static_cast<float*>(p.y)[o] = v;
        }
      }
    } else if (z == 0) {
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        if (!valid[r]) continue;
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const size_t o = (size_t)m * p.y_ld + n0 + rows[r];
          if (p.y_bf16)
            static_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(yacc[r][m]);
          else
            static_cast<float*>(p.y)[o] = yacc[r][m];
        }
      }
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

template <int M, int DEC, bool DOTS, int NSUB = 1>
int launch_one(const CUtensorMap& hi, const CUtensorMap& lo,
               const MmvParams& p, int smem, cudaStream_t stream) {
  auto kern = mmv_kernel<M, DEC, DOTS, NSUB>;
  static int configured = 0;  // largest dynamic smem size set so far
  if (smem > configured) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem) !=
        cudaSuccess)
      return PQ2_ERR_LAUNCH;
    configured = kMaxDynSmem;
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
  if (cudaLaunchKernelEx(&cfg, kern, hi, lo, p) != cudaSuccess) {
    cudaGetLastError();
    return PQ2_ERR_LAUNCH;
  }
  return PQ2_OK;
}

template <int DEC, bool DOTS>
int launch_m(int M, const CUtensorMap& hi, const CUtensorMap& lo,
             const MmvParams& p, int smem, cudaStream_t s) {
  switch (M) {
    case 1: return launch_one<1, DEC, DOTS>(hi, lo, p, smem, s);
    case 2: return launch_one<2, DEC, DOTS>(hi, lo, p, smem, s);
    case 3: return launch_one<3, DEC, DOTS>(hi, lo, p, smem, s);
    case 4: return launch_one<4, DEC, DOTS>(hi, lo, p, smem, s);
    case 5: return launch_one<5, DEC, DOTS>(hi, lo, p, smem, s);
    case 6: return launch_one<6, DEC, DOTS>(hi, lo, p, smem, s);
    case 7: return launch_one<7, DEC, DOTS>(hi, lo, p, smem, s);
    case 8: return launch_one<8, DEC, DOTS>(hi, lo, p, smem, s);
    default: return PQ2_ERR_SHAPE;
  }
}

// Activation groups of 128 / NSUB (NSUB = 2, 4), masked planes, M <= 4.
template <bool DOTS>
int launch_m_sub(int nsub, int M, const CUtensorMap& hi, const CUtensorMap& lo,
                 const MmvParams& p, int smem, cudaStream_t s) {
  constexpr int D = kDecodeMaskPlanes;
  if (nsub == 2) {
    switch (M) {
      case 1: return launch_one<1, D, DOTS, 2>(hi, lo, p, smem, s);
      case 2: return launch_one<2, D, DOTS, 2>(hi, lo, p, smem, s);
      case 3: return launch_one<3, D, DOTS, 2>(hi, lo, p, smem, s);
      case 4: return launch_one<4, D, DOTS, 2>(hi, lo, p, smem, s);
      default: return PQ2_ERR_SHAPE;
    }
  }
  switch (M) {
    case 1: return launch_one<1, D, DOTS, 4>(hi, lo, p, smem, s);
    case 2: return launch_one<2, D, DOTS, 4>(hi, lo, p, smem, s);
    case 3: return launch_one<3, D, DOTS, 4>(hi, lo, p, smem, s);
    case 4: return launch_one<4, D, DOTS, 4>(hi, lo, p, smem, s);
    default: return PQ2_ERR_SHAPE;
  }
}

}  // namespace

// Geometry: P = min(N, #SM) CTAs (more when a CTA would exceed 256 rows),
// R = ceil(N / P) rows for the largest CTA, and the split count S (a divisor
// of 32, so a row's splits share a warp) that best fills the consumer lanes
// (ceil(R/2)*S threads, two rows each, of 32*ceil(ceil(R/2)*S/32)) and the
// groups (G of S*ceil(G/S)) with at least ~6 warps.  A function of (N, K,
// SM count) only.
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
  const int pairs = (R + kRowsPerThread - 1) / kRowsPerThread;
  for (int S = 1; S <= std::min(std::min(G, kMaxSplits), 16); S *= 2) {
    const int lanes = pairs * S;
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
  out->threads = align_up(pairs * best_s, 32);
  out->steps = (G + best_s - 1) / best_s;
  return true;
}

namespace {

// pq2_mmv over N weight rows, or (gated) the gate/up form: outputs
// n < I = N / 2 from weight rows n and I + n.  The split count S comes from
// the geometry of all N rows either way, so a row's fp32 sum is the same.
int launch_mmv_impl(const int8_t* q, const float* sx, const int32_t* qsum,
                    const uint8_t* codes, const uint16_t* scales, void* y, int y_dtype,
                    int32_t* dots, int64_t M, int64_t N, int64_t K, int decode, int overlap,
                    bool gated, int sm_count, int32_t* status, cudaStream_t stream,
                    int nsub = 1, int drop_stage = -1, long long empty_limit = kWaitLimitCycles) {
  if (nsub != 1 && ((nsub != 2 && nsub != 4) || M > 4 || gated || decode != kDecodeMaskPlanes))
    return PQ2_ERR_SHAPE;
  const bool tensor = decode == kDecodeTensor;
  if (tensor && gated) return PQ2_ERR_SHAPE;
  MmvGeometry geo;
  if (!mmv_geometry(N, K, sm_count, &geo)) return PQ2_ERR_SHAPE;
  if (gated && (N % 2 || dots)) return PQ2_ERR_SHAPE;
  int64_t rows_out = N, ctas = geo.ctas;
  int rows_max = geo.rows_max, threads = geo.threads;
  if (gated) {
    // One output (a gate row and an up row) per thread and split: at most
    // 288 / S outputs and 256 box rows per CTA.
    const int64_t I = N / 2;
    const int64_t per = std::min<int64_t>(kMaxBoxRows, kMaxConsumerThreads / geo.splits);
    ctas = std::max<int64_t>(std::min<int64_t>(I, sm_count), (I + per - 1) / per);
    rows_max = (int)((I + ctas - 1) / ctas);
    threads = align_up(rows_max * geo.splits, 32);
    rows_out = I;
  }
  MmvParams p{};
  p.q = q; p.sx = sx; p.qsum = qsum; p.scales = scales;
  p.y = y; p.dots = dots; p.status = status;
  p.N = (int)rows_out; p.K = (int)K; p.G = (int)(K / kGroup);
  p.ctas = (int)ctas; p.splits = geo.splits; p.rows_max = rows_max;
  p.cons_threads = tensor ? kTcWarps * 32 : threads;
  p.gated = gated;
  p.up_row = gated ? (int)(N / 2) : 0;
  p.up_smem = gated ? align_up(rows_max, 8) : 0;
  p.y_ld = (int)rows_out;
  p.overlap = overlap;
  p.y_bf16 = y_dtype == PQ2_BF16;
  p.sw_bulk = (K / kGroup) % 8 == 0 && reinterpret_cast<uintptr_t>(scales) % 16 == 0;
  p.side16 = (M * (K / kGroup) * nsub) % 4 == 0 && reinterpret_cast<uintptr_t>(sx) % 16 == 0 &&
             reinterpret_cast<uintptr_t>(qsum) % 16 == 0;
  const int mi = (int)M, R = rows_max, S = geo.splits, G = p.G;
  const int unit = 4 * S / gcd(4, S);
  // rows of weights (and of their scales) a CTA keeps per 4-group box chunk
  const int slab = gated ? 2 * p.up_smem : R;
  p.box_stride = align_up(slab * kBoxBytes, 1024);
  // fixed region: barriers, weight scales, s_x, sum(q)
  p.sw_off = align_up(kAbortOff + 4, 128);
  p.sx_off = align_up(p.sw_off + G * slab * 2, 16);
  p.qs_off = align_up(p.sx_off + mi * G * nsub * 4, 16);
  p.part_off = align_up(p.qs_off + mi * G * nsub * 4, 16);
  p.ring_off = align_up(p.part_off + (tensor ? S * R * mi * 4 : 0), 1024);
  const int room = kSmemBudget - p.ring_off;
  // Stage: k units of lcm(4, S) groups, aiming at ~16-24 KB of codes.  The
  // tensor-core consumers read q from global memory: no q in the stages.
  const int q_cols = tensor ? 0 : mi;
  auto stage_bytes = [&](int gs) {
    return (gs / 4) * p.box_stride + q_cols * align_up(gs * kGroup, 1024);
  };
  // Stage: 2S groups when two such stages fit the ring, else S (S >= 8), or
  // 8 groups (S = 4), so that a thread meets one or two groups per stage.
  // Two independent groups between stage waits keep more loads and dp4a in
  // flight per warp (the warps of a CTA move through the stages together);
  // measured 4-13 % faster than one at M = 1-2.  Smaller S (tiny K) grows
  // the stage by units of lcm(4, S) groups towards ~16-24 KB of codes.
  int gs;
  if (S >= 4) {
    gs = S >= 8 ? S : 8;
    if (S >= 8 && G >= 2 * S && 2 * stage_bytes(2 * S) <= room) gs = 2 * S;
    if (stage_bytes(gs) * 3 > room && S == 4) gs = 4;
    p.groups_per_thread = gs / S;
  } else {
    gs = unit;
    while (gs + unit <= std::max(unit, (G + 3) / 4 * 4) && stage_bytes(gs + unit) <= 24 * 1024 &&
           stage_bytes(gs + unit) * 3 <= room)
      gs += unit;
    p.groups_per_thread = 0;
  }
  p.stage_groups = gs;
  p.q_off = (gs / 4) * p.box_stride;
  p.qbox_stride = align_up(gs * kGroup, 1024);
  p.stage_bytes = stage_bytes(gs);
  p.stages_total = (G + gs - 1) / gs;
  if (room < p.stage_bytes) return PQ2_ERR_SHAPE;
  // (A ring sized from the whole SM for calls that wait for the kernel
  // before them, so that the entire slab streams in during the wait, measured
  // slower in chains of dependent calls: 7.5 -> 8.2 us on ffn_up, 8.8 -> 9.5
  // us on ffn_down at M = 1.)
  p.ring = std::min(std::min(p.stages_total, room / p.stage_bytes), kMaxStages);
  p.drop_stage = drop_stage;
  p.empty_limit = empty_limit;
  if (tensor) {
    const int nt = (R + 15) / 16, tw = S < kTcWarps ? kTcWarps / S : 1;
    const int nts = (nt + tw - 1) / tw;
    if (S > 2 * kTcWarps || nts > kTcTiles || (S > kTcWarps && nts > kTcTiles2))
      return PQ2_ERR_SHAPE;
  }
  // A dropped release only matters where a slot is reused.
  if (drop_stage >= 0 && (p.stages_total <= p.ring || drop_stage + p.ring >= p.stages_total))
    return PQ2_ERR_SHAPE;
  int smem = 1024 + p.ring_off + p.ring * p.stage_bytes;  // + alignment slack
  // A call that waits for the kernel before it (weights-only overlap) takes
  // a whole SM: more than half the shared memory keeps a second CTA of any
  // grid off it.  Chained calls then fill each SM as its previous CTA
  // leaves, one per SM, and a call's weights still stream in while the
  // quantisation and the two grid hand-overs in front of it run.
  if (overlap == 1) smem = std::max(smem, kSoloSmem);

  CUtensorMap hi, lo;
  const int rows_lo = (int)(rows_out / ctas);
  if (!encode_map(&hi, codes, N, K / 4, R) ||
      !encode_map(&lo, codes, N, K / 4, rows_lo > 0 ? rows_lo : R))
    return PQ2_ERR_LAUNCH;
  if (nsub > 1)
    return dots ? launch_m_sub<true>(nsub, mi, hi, lo, p, smem, stream)
                : launch_m_sub<false>(nsub, mi, hi, lo, p, smem, stream);
  if (tensor)
    return dots ? launch_m<kDecodeTensor, true>(mi, hi, lo, p, smem, stream)
                : launch_m<kDecodeTensor, false>(mi, hi, lo, p, smem, stream);
  if (dots)
    return decode == kDecodeMaskPlanes
               ? launch_m<kDecodeMaskPlanes, true>(mi, hi, lo, p, smem, stream)
               : launch_m<kDecodeAddXor, true>(mi, hi, lo, p, smem, stream);
  return decode == kDecodeMaskPlanes
             ? launch_m<kDecodeMaskPlanes, false>(mi, hi, lo, p, smem, stream)
             : launch_m<kDecodeAddXor, false>(mi, hi, lo, p, smem, stream);
}

}  // namespace

int launch_mmv(const int8_t* q, const float* sx, const int32_t* qsum, const uint8_t* codes,
               const uint16_t* scales, void* y, int y_dtype, int32_t* dots, int64_t M,
               int64_t N, int64_t K, int decode, int overlap, int sm_count, int32_t* status,
               cudaStream_t stream) {
  return launch_mmv_impl(q, sx, qsum, codes, scales, y, y_dtype, dots, M, N, K, decode,
                         overlap, false, sm_count, status, stream);
}

int launch_mmv_grouped(const int8_t* q, const float* sx, const int32_t* qsum,
                       const uint8_t* codes, const uint16_t* scales, void* y, int y_dtype,
                       int32_t* dots, int64_t M, int64_t N, int64_t K, int act_group,
                       int overlap, int sm_count, int32_t* status, cudaStream_t stream) {
  if (act_group != 128 && act_group != 64 && act_group != 32) return PQ2_ERR_SHAPE;
  return launch_mmv_impl(q, sx, qsum, codes, scales, y, y_dtype, dots, M, N, K,
                         kDecodeMaskPlanes, overlap, false, sm_count, status, stream,
                         128 / act_group);
}

int launch_mmv_drop_arrival(const int8_t* q, const float* sx, const int32_t* qsum,
                            const uint8_t* codes, const uint16_t* scales, void* y, int y_dtype,
                            int64_t M, int64_t N, int64_t K, long long wait_limit, int sm_count,
                            int32_t* status, cudaStream_t stream) {
  return launch_mmv_impl(q, sx, qsum, codes, scales, y, y_dtype, nullptr, M, N, K,
                         kDecodeMaskPlanes, 0, false, sm_count, status, stream, 1, 0,
                         wait_limit);
}

int launch_mmv_gated(const int8_t* q, const float* sx, const int32_t* qsum,
                     const uint8_t* codes, const uint16_t* scales, void* out, int out_dtype,
                     int64_t M, int64_t N, int64_t K, int decode, int overlap, int sm_count,
                     int32_t* status, cudaStream_t stream) {
  return launch_mmv_impl(q, sx, qsum, codes, scales, out, out_dtype, nullptr, M, N, K, decode,
                         overlap, true, sm_count, status, stream);
}

}  // namespace pq2
