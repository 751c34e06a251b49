// pq2_mm.cu — prefill (M >= 16) ternary x INT8 matmul on tcgen05 tensor
// cores (sm_103a).
//
// Method: page "Kernel experiments: recorded evidence" (KE), Test 7 (INT8
// tensor-core MMQ prefill: per 128-group, an integer dot on the tensor cores,
// then the group's activation and weight scales) and Test 2 (load each packed
// byte once and expand its four codes); page "Baseline and the integer
// breakthrough", "Use matrix hardware for prefill".
//
// GB300 design.  sm_103a has no 8-bit integer tcgen05 MMA, so the contraction
// runs as kind::f16: A = q widened to fp16 (exact, |q| <= 127), B = the codes
// decoded to fp16 c-1 in {-1, 0, 1, 2} (exact).  Each 128-group is one
// accumulation of eight K=16 MMAs into a fresh fp32 TMEM tile: every partial
// sum is an integer of magnitude <= 32512 < 2^24, so the group dot is exact,
// exactly the int32 per-group partial of the method.  The epilogue then scales
// it by s_x * s_w and adds it into an fp32 accumulator.
//
// One CTA computes a tile of 128 tokens x 128 output rows:
//   warp 0      TMA producer: q tiles (two 64-column boxes per group, 128-byte
//               swizzle, the canonical K-major layout of the MMA) and code
//               tiles (32 bytes x 128 rows per group)
//   warp 1      TMEM allocation; lane 0 issues the MMAs and commits
//   warps 2-3   decoders: code bytes -> fp16 B tile in the same swizzled layout
//   warps 4-11  epilogue: one token row and half the columns per thread, reads
//               the group's fp32 D from TMEM (double-buffered), scales and
//               accumulates, stores y
// Every wait is bounded; a wait that gives up records PQ2_ERR_TIMEOUT and the
// protocol continues without the work so that no thread is left waiting.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "pq2_device.cuh"
#include "pq2_internal.h"

namespace pq2 {
namespace {

constexpr int BM = 128;          // tokens per tile (MMA M)
constexpr int BN = 128;          // output rows per tile (MMA N)
constexpr int kStagesA = 3;      // q tile stages
constexpr int kStagesC = 4;      // code tile stages
constexpr int kStagesB = 2;      // decoded weight tile stages
constexpr int kGC = 8;           // groups per weight-scale chunk
constexpr int kThreads = 384;
constexpr int kEpiThreads = 256;  // warps 4-11: two per TMEM lane quarter
constexpr int kEpiCols = BN / 2;  // columns per epilogue thread
constexpr int kABytes = BM * kGroup * 2;   // 32 KB: q tile of one group (fp16)
constexpr int kBBytes = BN * kGroup * 2;   // 32 KB: decoded weights of one group
constexpr int kCBytes = BN * kGroupCodeBytes;  // 4 KB: code bytes of one group
constexpr int kTmemCols = 2 * BN;          // two fp32 D buffers

struct MmParams {
  const float* sx;         // [M][G]
  const uint16_t* scales;  // [N][G]
  void* y;                 // [M][N]
  int32_t* dots;           // [M][N][G] (dot-only variant)
  int32_t* status;
  int M, N, K, G;
  int y_bf16;
};

// Shared-memory layout (offsets from a 1024-byte aligned base).
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStagesA * kABytes;
constexpr int kOffC = kOffB + kStagesB * kBBytes;
constexpr int kOffSW = kOffC + kStagesC * kCBytes;        // 2 chunks of [kGC][BN] fp16
constexpr int kOffBar = kOffSW + 2 * kGC * BN * 2;
constexpr int kNumBars = 2 * kStagesA + 2 * kStagesC + 2 * kStagesB + 4;
constexpr int kOffTmemAddr = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffTmemAddr + 16 + 1024;     // + alignment slack

// ------------------------------------------------------------ tcgen05 PTX
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, fp16 inputs, fp32 accumulation.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every MMA issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Generic-proxy shared-memory writes -> visible to the tensor core.
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int x, int y,
                                       uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle,
// 8-row core groups 1024 bytes apart (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B and 128-byte rows).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)(16 >> 4) << 16;           // leading byte offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                   // descriptor version
  d |= (uint64_t)2 << 61;                   // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16, D fp32, A and B fp16, both K-major.
__host__ __device__ constexpr uint32_t instr_desc_f16(int m, int n) {
  return (1u << 4)                      // D format: f32
         | (0u << 7) | (0u << 10)       // A, B format: f16
         | (0u << 15) | (0u << 16)      // A, B K-major
         | ((uint32_t)(n >> 3) << 17)   // N / 8
         | ((uint32_t)(m >> 4) << 24);  // M / 16
}

// Two codes (bits 0-1 and 2-3 of x) -> fp16x2 (c0 - 1, c1 - 1): the halves
// 0x6400 | c are 1024 + c exactly, and subtracting 1025 is exact.
__device__ __forceinline__ uint32_t decode_pair(uint32_t x) {
  const uint32_t u = (x & 3u) | ((x & 0xCu) << 14) | 0x64006400u;
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&u),
                            __halves2half2(__ushort_as_half(0x6401), __ushort_as_half(0x6401)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

template <bool DOTS>
__global__ void __launch_bounds__(kThreads, 1)
    mm_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_c,
              const MmParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* a_full = bars;
  uint64_t* a_empty = a_full + kStagesA;
  uint64_t* c_full = a_empty + kStagesA;
  uint64_t* c_empty = c_full + kStagesC;
  uint64_t* b_full = c_empty + kStagesC;
  uint64_t* b_empty = b_full + kStagesB;
  uint64_t* d_full = b_empty + kStagesB;
  uint64_t* d_empty = d_full + 2;
  uint32_t* tmem_addr_s = reinterpret_cast<uint32_t*>(smem + kOffTmemAddr);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
  const int G = p.G;

  if (tid == 0) {
    for (int i = 0; i < kStagesA; ++i) { mbar_init(&a_full[i], 1); mbar_init(&a_empty[i], 1); }
    for (int i = 0; i < kStagesC; ++i) { mbar_init(&c_full[i], 1); mbar_init(&c_empty[i], 2); }
    for (int i = 0; i < kStagesB; ++i) { mbar_init(&b_full[i], 2); mbar_init(&b_empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&d_full[i], 1); mbar_init(&d_empty[i], kEpiThreads / 32); }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_addr_s, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_addr_s;
  // Inputs may come from the previous kernel on the stream.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  bool ok = true;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&map_q) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&map_c) : "memory");
      for (int g = 0; g < G; ++g) {
        const int sa = g % kStagesA, sc = g % kStagesC;
        if (g >= kStagesA) ok = ok && mbar_wait(&a_empty[sa], ((g / kStagesA) - 1) & 1);
        uint8_t* a = smem + kOffA + sa * kABytes;
        mbar_arrive_expect_tx(&a_full[sa], kABytes);
        tma_2d(a, &map_q, g * kGroup, m0, &a_full[sa]);
        tma_2d(a + kABytes / 2, &map_q, g * kGroup + 64, m0, &a_full[sa]);
        if (g >= kStagesC) ok = ok && mbar_wait(&c_empty[sc], ((g / kStagesC) - 1) & 1);
        mbar_arrive_expect_tx(&c_full[sc], kCBytes);
        tma_2d(smem + kOffC + sc * kCBytes, &map_c, g * kGroupCodeBytes, n0, &c_full[sc]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = instr_desc_f16(BM, BN);
      for (int g = 0; g < G; ++g) {
        const int sa = g % kStagesA, sb = g % kStagesB, d = g & 1;
        ok = ok && mbar_wait(&a_full[sa], (g / kStagesA) & 1);
        ok = ok && mbar_wait(&b_full[sb], (g / kStagesB) & 1);
        if (g >= 2) ok = ok && mbar_wait(&d_empty[d], ((g >> 1) - 1) & 1);
        tc_fence_after();
        const uint32_t a_base = smem_u32(smem + kOffA + sa * kABytes);
        const uint32_t b_base = smem_u32(smem + kOffB + sb * kBBytes);
        const uint32_t d_tmem = tmem_base + d * BN;
        if (ok) {
#pragma unroll
          for (int k = 0; k < kGroup / 16; ++k) {
            // K step k: 64-column atom k/4, 32-byte offset (k%4) inside the
            // 128-byte swizzled row.
            const uint32_t off = (k >> 2) * (BM * 128) + (k & 3) * 32;
            const uint32_t boff = (k >> 2) * (BN * 128) + (k & 3) * 32;
            mma_f16(d_tmem, smem_desc_sw128(a_base + off), smem_desc_sw128(b_base + boff),
                    idesc, k > 0 ? 1u : 0u);
          }
        }
        mma_commit(&a_empty[sa]);
        mma_commit(&b_empty[sb]);
        mma_commit(&d_full[d]);
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ decoders
    const int dt = tid - 64;  // 0..63, two rows each
    for (int g = 0; g < G; ++g) {
      const int sc = g % kStagesC, sb = g % kStagesB;
      ok = ok && mbar_wait(&c_full[sc], (g / kStagesC) & 1);
      if (g >= kStagesB) ok = ok && mbar_wait(&b_empty[sb], ((g / kStagesB) - 1) & 1);
      const uint8_t* cs = smem + kOffC + sc * kCBytes;
      uint8_t* bs = smem + kOffB + sb * kBBytes;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int n = dt + 64 * rr;
        const uint4 c0 = *reinterpret_cast<const uint4*>(cs + n * kGroupCodeBytes);
        const uint4 c1 = *reinterpret_cast<const uint4*>(cs + n * kGroupCodeBytes + 16);
        const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        // 16 chunks of 16 bytes = 8 weights = 2 code bytes each.
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t two = (cw[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
          uint4 v;
          v.x = decode_pair(two & 0xF);
          v.y = decode_pair((two >> 4) & 0xF);
          v.z = decode_pair((two >> 8) & 0xF);
          v.w = decode_pair((two >> 12) & 0xF);
          const int atom = j >> 3, jj = j & 7;
          uint8_t* dst = bs + atom * (BN * 128) + (n >> 3) * 1024 + (n & 7) * 128 +
                         ((jj ^ (n & 7)) << 4);
          *reinterpret_cast<uint4*>(dst) = v;
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&c_empty[sc]);
        mbar_arrive(&b_full[sb]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int et = tid - 128;      // 0..255
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int half = (warp - 4) >> 2;
    const int col0 = half * kEpiCols;
    const int row = 32 * quarter + lane;
    const int m = m0 + row;
    __half* sw_s = reinterpret_cast<__half*>(smem + kOffSW);  // [2][kGC][BN]
    float acc[kEpiCols];
#pragma unroll
    for (int n = 0; n < kEpiCols; ++n) acc[n] = 0.0f;
    const int nchunks = (G + kGC - 1) / kGC;
    // Weight-scale chunk loader: kGC x BN fp16, 4 values per thread.
    constexpr int kSwPer = kGC * BN / kEpiThreads;
    uint16_t swv[kSwPer];
    float sxv[kGC], sxn[kGC];
    auto load_chunk = [&](int ch) {
#pragma unroll
      for (int j = 0; j < kSwPer; ++j) {
        const int idx = et + kEpiThreads * j;  // idx = gg * BN + n
        const int gg = idx / BN, n = idx % BN, g = ch * kGC + gg;
        swv[j] = (!DOTS && g < G && n0 + n < p.N) ? __ldg(p.scales + (size_t)(n0 + n) * G + g)
                                                  : (uint16_t)0;
      }
#pragma unroll
      for (int gg = 0; gg < kGC; ++gg) {
        const int g = ch * kGC + gg;
        sxn[gg] = (!DOTS && g < G && m < p.M) ? __ldg(p.sx + (size_t)m * G + g) : 0.0f;
      }
    };
    load_chunk(0);
    for (int ch = 0; ch < nchunks; ++ch) {
      uint16_t* dst = reinterpret_cast<uint16_t*>(sw_s) + (ch & 1) * kGC * BN;
#pragma unroll
      for (int j = 0; j < kSwPer; ++j) dst[et + kEpiThreads * j] = swv[j];
#pragma unroll
      for (int gg = 0; gg < kGC; ++gg) sxv[gg] = sxn[gg];
      named_bar_sync(1, kEpiThreads);
      if (ch + 1 < nchunks) load_chunk(ch + 1);
      const __half* swc = sw_s + (ch & 1) * kGC * BN + col0;
#pragma unroll 1
      for (int gg = 0; gg < kGC; ++gg) {
        const int g = ch * kGC + gg;
        if (g >= G) break;
        const int d = g & 1;
        ok = ok && mbar_wait(&d_full[d], (g >> 1) & 1);
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(32 * quarter) << 16) + d * BN + col0;
#pragma unroll
        for (int cb = 0; cb < kEpiCols / 16; ++cb) {
          uint32_t v[16];
          tmem_ld16(taddr + cb * 16, v);
          tmem_ld_wait();
          if (DOTS) {
            if (m < p.M) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int n = n0 + col0 + cb * 16 + j;
                if (n < p.N)
                  p.dots[((size_t)m * p.N + n) * G + g] = (int32_t)__uint_as_float(v[j]);
              }
            }
          } else {
            const float sx = sxv[gg];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float t = __fmul_rn(__uint_as_float(v[j]), sx);
              acc[cb * 16 + j] = __fmaf_rn(t, __half2float(swc[gg * BN + cb * 16 + j]),
                                           acc[cb * 16 + j]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&d_empty[d]);
      }
      named_bar_sync(1, kEpiThreads);  // the scale buffer of this chunk may be reused
    }
    if (!DOTS && m < p.M) {
      if (p.y_bf16) {
        __nv_bfloat16* yr = static_cast<__nv_bfloat16*>(p.y) + (size_t)m * p.N + n0 + col0;
        for (int n = 0; n < kEpiCols; ++n)
          if (n0 + col0 + n < p.N) yr[n] = __float2bfloat16_rn(acc[n]);
      } else {
        float* yr = static_cast<float*>(p.y) + (size_t)m * p.N + n0 + col0;
        for (int n = 0; n < kEpiCols; ++n)
          if (n0 + col0 + n < p.N) yr[n] = acc[n];
      }
    }
  }
  if (!ok) report(p.status, PQ2_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
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
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
    else
      cudaGetLastError();
  });
  return fn;
}

template <bool DOTS>
int launch_mm_t(const CUtensorMap& mq, const CUtensorMap& mc, const MmParams& p,
                cudaStream_t stream) {
  auto kern = mm_kernel<DOTS>;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess)
      return PQ2_ERR_LAUNCH;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.N + BN - 1) / BN, (p.M + BM - 1) / BM);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, mq, mc, p) != cudaSuccess) {
    cudaGetLastError();
    return PQ2_ERR_LAUNCH;
  }
  return PQ2_OK;
}

}  // namespace

int launch_mm(const uint16_t* q_f16, const float* sx, const uint8_t* codes,
              const uint16_t* scales, void* y, int y_dtype, int32_t* dots, int64_t M,
              int64_t N, int64_t K, int sm_count, int32_t* status, cudaStream_t stream) {
  (void)sm_count;
  if (M > (int64_t)1 << 20 || N > (int64_t)1 << 30) return PQ2_ERR_SHAPE;
  if ((N + BN - 1) / BN > 0x7fffffff || (M + BM - 1) / BM > 65535) return PQ2_ERR_SHAPE;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PQ2_ERR_LAUNCH;
  CUtensorMap mq, mc;
  {
    // q: fp16 [M][K], box 64 x 128 (128-byte rows), 128-byte swizzle.
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)BM};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&mq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(q_f16), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PQ2_ERR_LAUNCH;
  }
  {
    // codes: u8 [N][K/4], box 32 x 128 (one group of 128 rows), no swizzle.
    const cuuint64_t dims[2] = {(cuuint64_t)(K / 4), (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)(K / 4)};
    const cuuint32_t box[2] = {(cuuint32_t)kGroupCodeBytes, (cuuint32_t)BN};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PQ2_ERR_LAUNCH;
  }
  MmParams p{};
  p.sx = sx; p.scales = scales; p.y = y; p.dots = dots; p.status = status;
  p.M = (int)M; p.N = (int)N; p.K = (int)K; p.G = (int)(K / kGroup);
  p.y_bf16 = y_dtype == PQ2_BF16;
  return dots ? launch_mm_t<true>(mq, mc, p, stream) : launch_mm_t<false>(mq, mc, p, stream);
}

}  // namespace pq2
