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
// runs as kind::f16.  The weights are the MMA's A operand and live in tensor
// memory: decoder threads (one weight row each) turn a 4-byte code word into
// eight fp16x2 words of c - 1 (one shift, then a LOP3 and one exact HFMA2
// per word: field s masked in place and OR-ed with 0x6400 is the fp16 value
// 1024 + c * 4^s) and store them with tcgen05.st, so decoded weights never
// touch shared memory.  q (B operand, fp16, exact)
// streams into shared memory by TMA in the matching K order
// (pq2_quantize_act's PQ2_Q_F16 layout).  Each 128-group is one accumulation
// of eight K=16 MMAs into a fresh fp32 TMEM tile: every partial sum is an
// integer of magnitude <= 32512 < 2^24, so D is the exact int32 per-group
// partial of the method.  The epilogue scales it by s_x * s_w into fp32.
//
// An 8-bit variant (pq2_mm_f8) decodes the weights to e4m3 with one byte
// permute per four weights and takes q as two exact e4m3 planes (16a and b,
// q = 16a + b, PQ2_Q_F8); each K step is two kind::f8f6f4 MMAs into the same
// group tile, at twice the fp16 rate, so the tensor time is unchanged while
// the decode costs 11 instead of 17 instructions per 16 weights and A takes
// half the tensor memory, leaving room for a third D buffer.
//
// Activation groups of 64 or 32 (KE Test 9, "Smaller Q8 activation groups";
// pq2_mm_grouped, pq2_mm_f8_grouped): a weight group's K steps split into
// 128 / A accumulation units, each into its own fresh D buffer of the same
// ring and scaled by its own s_x (the kernel's NSUB template parameter).
//
// At most 16 tokens (activation groups of 128): the narrow kernel, NW = 16.
// The MMA's N is 16, a D buffer takes 16 columns (eight in flight), q
// arrives in 16-row boxes, and one epilogue warp per lane quarter reads D.
// The arithmetic of every output is that of the full tile.
//
// One CTA computes a tile of 128 output rows x 128 tokens:
//   warp 0      TMA producer: q tiles (two 64-column boxes per group, 128-byte
//               swizzle, the canonical K-major layout) and code tiles
//   warp 1      TMEM allocation; one elected lane issues the MMAs and commits
//   warps 2-5   decoders: one weight row per thread, codes -> TMEM A tile
//   warps 6-21  epilogue: one weight row and 32 tokens per thread, reads D
//               (two buffers in flight, three on the 8-bit path), scales it
//               and adds it into fp32 running sums in registers, finally
//               stores y
//   warp 22     scheduler: waits until a unit's A, q and D buffer are
//               ready, then releases the MMA warp (named barrier)
//   warp 23     scales: stages s_x and s_w chunk by chunk for the epilogue
// A warp may only reach the TMEM lanes 32*(warp % 4) .. +31, so each role
// spans four consecutive warps (one per lane quarter).
// Every wait is bounded and fails fast: a wait that gives up records
// PQ2_ERR_TIMEOUT and the protocol continues without the work.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "pq2_device.cuh"
#include "pq2_internal.h"

namespace pq2 {
namespace {

constexpr int BW = 128;          // weight rows per tile (MMA M, A in TMEM)
constexpr int BT = 128;          // tokens per tile (MMA N, B in shared memory)
constexpr int kGC = 4;           // accumulation units per scale chunk
constexpr int kEpiWarps = 16;     // warps 6-21: four per TMEM lane quarter
constexpr int kSchedWarp = 6 + kEpiWarps;  // warp 22: waits on the MMA's inputs
constexpr int kScaleWarp = 7 + kEpiWarps;  // warp 23: stages the scales
constexpr int kThreads = (8 + kEpiWarps) * 32;
constexpr int kEpiCols = BT / 4;  // tokens per epilogue thread
// Tensor-memory budget (512 columns): fp16 A takes 64 columns per group, so
// two D buffers (128 columns each) fit beside four A buffers; e4m3 A takes 32,
// which leaves room for a third D buffer.
template <bool F8> constexpr int kDBufT = F8 ? 3 : 2;  // D buffers in flight
template <bool F8> constexpr int kAColsT = F8 ? 32 : 64;  // A columns per group
// Few tokens (M <= kNarrowN): the MMA's N is kNarrowN, a D buffer takes
// kNarrowN columns and kNarrowDBuf of them fit beside the A buffers.
constexpr int kNarrowN = 16;
constexpr int kNarrowDBuf = 8;
constexpr int kDBufMax = 8;
constexpr int kABuf = 4;          // decoded weight (A) buffers in flight
// Unit-completion barriers: more than every distance by which the MMA can
// lead a waiter (5 groups of NSUB units for the q producer).
template <int NSUB> constexpr int kDoneT = 8 * NSUB;
constexpr int kDoneMax = 32;
static_assert(kNarrowDBuf * kNarrowN + kABuf * 64 <= 512, "tensor memory budget (narrow)");
constexpr int kCBytes = BW * kGroupCodeBytes;  // 4 KB: code bytes of one group
constexpr int kDCol = 0;                       // D buffers: columns [0, kDBuf*BT)
template <bool F8> constexpr int kAColT = kDBufT<F8> * BT;  // A buffers after them
constexpr int kTmemCols = 512;
static_assert(kAColT<false> + kABuf * kAColsT<false> <= kTmemCols, "tensor memory budget");
static_assert(kAColT<true> + kABuf * kAColsT<true> <= kTmemCols, "tensor memory budget");

struct MmParams {
  const float* sx;         // [M][G * NSUB]
  const uint16_t* scales;  // [N][G]
  void* y;                 // [M][N]
  int32_t* dots;           // [M][N][G * NSUB] (dot-only variant)
  int32_t* status;
  int M, N, K, G;
  int y_bf16;
  int vec_scales;  // whole chunks and s_x / s_w aligned for one vector load each
};

// Shared-memory layout (offsets from a 1024-byte aligned base) for MMA width
// NW (tokens per accumulation unit).  The q stage of a group holds two
// 64-column boxes of NW rows (32 KB for a 128-token tile, 4 KB for the
// narrow kernel).  (Deeper code rings, 12 stages beside 5 q stages and 32
// in the narrow kernel, measured the same at M = 16 .. 4096.)
// Scale ring: 2 chunks of {s_x [kGC][BT] fp32, s_w [BW][kGC / NSUB] fp16}
// (a chunk is kGC accumulation units, kGC / NSUB weight groups).
constexpr int kSxBytes = kGC * BT * 4;
constexpr int kSwBytes = BW * kGC * 2;
constexpr int kSBytes = kSxBytes + kSwBytes;
template <int NW>
struct Layout {
  static constexpr int stagesQ = 6;  // q tile stages
  static constexpr int stagesC = 4;  // code tile stages
  static constexpr int qBytes = NW * kGroup * 2;    // q tile of one group
  static constexpr int offQ = 0;
  static constexpr int offC = offQ + stagesQ * qBytes;
  static constexpr int offS = offC + stagesC * kCBytes;
  static constexpr int offBar = offS + 2 * kSBytes;
  static constexpr int numBars = stagesQ + 2 * stagesC + kABuf + kDoneMax + kDBufMax + 4;
  static constexpr int offTmemAddr = offBar + numBars * 8;
  static constexpr int smemBytes = offTmemAddr + 16 + 1024;  // + alignment slack
  static_assert(qBytes % 2048 == 0, "each 64-column q box starts on a 1024-byte swizzle atom");
  static_assert(smemBytes <= 227 * 1024, "shared memory per CTA");
};

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
// The MMA issue below is predicated, not branched: every lane of the MMA
// warp runs the same instructions and only the lane that elect.sync picks
// (`on` != 0) issues.  A branch around the issue (if lane == 0) made the
// warp diverge and reconverge once per group, which cost more clocks per
// group than the tensor pipe needs for the group's MMAs.
__device__ __forceinline__ uint32_t elect_one() {
  uint32_t r = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(r));
  return r;
}
// D[tmem] (+)= A[tmem] * B[smem]^T, fp16 inputs, fp32 accumulation; issued
// by the thread with on != 0.
__device__ __forceinline__ void mma_f16_ta(uint32_t on, uint32_t d_tmem, uint32_t a_tmem,
                                           uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(on)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, e4m3 inputs, fp32 accumulation; issued
// by the thread with on != 0.
__device__ __forceinline__ void mma_f8_ta(uint32_t on, uint32_t d_tmem, uint32_t a_tmem,
                                          uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(on)
      : "memory");
}
// Arrive once on `bar` when every MMA issued so far by the issuing thread
// (on != 0) is done.
__device__ __forceinline__ void mma_commit(uint32_t on, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %1, 0;\n\t"
      "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(on)
      : "memory");
}
// Packed pairs of fp32 (element 0 in the low half): one instruction, two
// IEEE round-to-nearest results, the same as two scalar operations.
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo, uint32_t hi) {
  return ((uint64_t)hi << 32) | lo;
}
// acc += (d * x) * sw for two tokens: (d0, d1) and (x0, x1) become 64-bit
// operands as register pairs inside the asm.  Built with shifts and ORs in
// C++ instead, the pairs cost about as many instructions as the arithmetic
// (measured: the epilogue took 5-9 % longer).
__device__ __forceinline__ void epi_fma2(uint64_t& acc, uint32_t d0, uint32_t d1, uint32_t x0,
                                         uint32_t x1, uint64_t sw2) {
  asm("{\n\t.reg .b64 d, x, t;\n\tmov.b64 d, {%1, %2};\n\tmov.b64 x, {%3, %4};\n\t"
      "mul.rn.f32x2 t, d, x;\n\tfma.rn.f32x2 %0, t, %5, %0;\n\t}"
      : "+l"(acc)
      : "r"(d0), "r"(d1), "r"(x0), "r"(x1), "l"(sw2));
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
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
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

// Instruction descriptor: D fp32, A and B format code 0 (fp16 under
// kind::f16, e4m3 under kind::f8f6f4), both K-major (A may come from tensor
// memory).
__host__ __device__ constexpr uint32_t instr_desc_f16(int m, int n) {
  return (1u << 4)                      // D format: f32
         | (0u << 7) | (0u << 10)       // A, B format: f16
         | (0u << 15) | (0u << 16)      // A, B K-major
         | ((uint32_t)(n >> 3) << 17)   // N / 8
         | ((uint32_t)(m >> 4) << 24);  // M / 16
}

// Eight fp16x2 words of one code word w, in the operand K order: word
// j = 2s + pb holds the weights c - 1 of (byte pb, field s) and (byte pb + 2,
// field s), i.e. weights 4pb + s and 4(pb + 2) + s.  Field s masked in place
// and OR-ed with 0x6400 gives the fp16 value 1024 + c * 4^s exactly (the
// field sits in the low mantissa bits); one HFMA2 by 4^-s with the bias
// -(1024 * 4^-s + 1), both exact in fp16, leaves exactly c - 1.  Bytes 1 and
// 3 come from one shift by 8, so a word costs 1 SHF + 8 LOP3 + 8 HFMA2.
__device__ __forceinline__ void decode_word(uint32_t w, uint32_t* out) {
  // fp16 bit patterns: 1, 1/4, 1/16, 1/64 and -1025, -257, -65, -17
  constexpr uint16_t kScale[4] = {0x3C00, 0x3400, 0x2C00, 0x2400};
  constexpr uint16_t kBias[4] = {0xE401, 0xDC04, 0xD410, 0xCC40};
  const uint32_t w8 = w >> 8;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const __half2 sc = __halves2half2(__ushort_as_half(kScale[s]), __ushort_as_half(kScale[s]));
    const __half2 bi = __halves2half2(__ushort_as_half(kBias[s]), __ushort_as_half(kBias[s]));
#pragma unroll
    for (int pb = 0; pb < 2; ++pb) {
      const uint32_t u = ((pb ? w8 : w) & (0x00030003u << (2 * s))) | 0x64006400u;
      const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&u), sc, bi);
      out[2 * s + pb] = *reinterpret_cast<const uint32_t*>(&r);
    }
  }
}

// Four e4m3 words of one code word w in the operand K order of PQ2_Q_F8:
// word 0 holds the weights 0, 2, 4, 6 of the code word (weight 4j + s is
// field s of byte j, bits 8j + 2s), word 1 the weights 1, 3, 5, 7, word 2
// 8, 10, 12, 14 and word 3 9, 11, 13, 15.  Masked with 0x3333, four fields
// sit in the four selector nibbles of a byte permute that picks from the
// table {-1, 0, +1, +2} in e4m3: 1 SHF + ... = 3 SHF + 4 LOP3 + 4 PRMT.
__device__ __forceinline__ void decode_word_f8(uint32_t w, uint32_t* out) {
  constexpr uint32_t kTable = 0x403800B8u;  // bytes: e4m3 -1, 0, +1, +2
  const uint32_t w2 = w >> 2;
  out[0] = __byte_perm(kTable, 0u, w & 0x3333u);
  out[1] = __byte_perm(kTable, 0u, w2 & 0x3333u);
  out[2] = __byte_perm(kTable, 0u, (w >> 16) & 0x3333u);
  out[3] = __byte_perm(kTable, 0u, (w2 >> 16) & 0x3333u);
}

// NSUB accumulation units per weight group: 1 for activation groups of 128,
// 2 for 64 and 4 for 32 (KE Test 9).  Unit u = g * NSUB + h is the partial
// dot of weight group g over activation group h: 8 / NSUB of the group's K
// steps accumulated into one fresh D buffer, scaled by s_x[m][u] and
// s_w[n][g].  The units of all groups share the ring of D buffers, so the
// tensor-memory layout and the 128-token tile are the same for every NSUB;
// a smaller activation group costs more D round trips and more epilogue
// arithmetic per weight group, not more decoding.
template <bool DOTS, bool F8, int NSUB, int NW>
__global__ void __launch_bounds__(kThreads, 1)
    mm_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_c,
              const MmParams p) {
  // NW: the MMA's N, tokens per accumulation unit.  BT for a full token tile;
  // kNarrowN when the call has at most that many tokens: the q copies are
  // NW rows, a D buffer is NW columns (kNarrowDBuf of them in flight, a
  // ring eight deep instead of two or three), and one epilogue warp per
  // lane quarter reads it.
  constexpr bool kNarrow = NW < BT;
  static_assert(NW == BT || (NW == kNarrowN && NSUB == 1), "token widths");
  constexpr int kDBuf = kNarrow ? kNarrowDBuf : kDBufT<F8>;
  constexpr int kACol = kDBuf * NW, kACols = kAColsT<F8>;
  constexpr int kDone = kNarrow ? 2 * kNarrowDBuf : kDoneT<NSUB>;
  constexpr int kEpiLive = kNarrow ? 4 : kEpiWarps;  // epilogue warps that take part
  constexpr int kCols = kNarrow ? NW : kEpiCols;      // tokens per epilogue thread
  constexpr int kQTx = NW * kGroup * 2;               // q bytes per group
  static_assert(kDBuf <= kDBufMax && kACol + kABuf * kACols <= kTmemCols, "buffers");
  using L = Layout<NW>;
  constexpr int kStagesQ = L::stagesQ, kStagesC = L::stagesC, kQBytes = L::qBytes;
  constexpr int kOffQ = L::offQ, kOffC = L::offC, kOffS = L::offS, kOffBar = L::offBar;
  constexpr int kOffTmemAddr = L::offTmemAddr;
  constexpr int kGW = kGC / NSUB;  // weight groups per scale chunk
  static_assert(NSUB == 1 || NSUB == 2 || NSUB == 4, "activation groups of 128, 64 or 32");
  static_assert(kDone <= kDoneMax, "completion barriers");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars;
  uint64_t* c_full = q_full + kStagesQ;
  uint64_t* c_empty = c_full + kStagesC;
  uint64_t* a_full = c_empty + kStagesC;
  uint64_t* g_done = a_full + kABuf;   // kDone: unit u's MMAs are complete
  uint64_t* d_empty = g_done + kDoneMax;
  uint64_t* s_full = d_empty + kDBufMax;
  uint64_t* s_empty = s_full + 2;
  uint32_t* tmem_addr_s = reinterpret_cast<uint32_t*>(smem + kOffTmemAddr);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Token tiles vary fastest: CTAs running together read different q tiles
  // (no L2 hot spot) and share a few weight tiles.
  const int m0 = blockIdx.x * BT, n0 = blockIdx.y * BW;
  const int G = p.G, GU = p.G * NSUB;
  // Wait until unit j's MMAs are complete (ring of kDone barriers, one
  // phase per kDone units; no waiter lags the MMA by kDone units).
  auto done_wait = [&](int j) { return mbar_wait(&g_done[j % kDone], (j / kDone) & 1); };

  if (tid == 0) {
    for (int i = 0; i < kStagesQ; ++i) mbar_init(&q_full[i], 1);
    for (int i = 0; i < kDone; ++i) mbar_init(&g_done[i], 1);
    for (int i = 0; i < kStagesC; ++i) { mbar_init(&c_full[i], 1); mbar_init(&c_empty[i], 4); }
    for (int i = 0; i < kABuf; ++i) mbar_init(&a_full[i], 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 32);
      mbar_init(&s_empty[i], kEpiLive);
    }
    for (int i = 0; i < kDBuf; ++i) mbar_init(&d_empty[i], kEpiLive);
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
    // Lane 0 issues the TMA copies of codes and q group by group.
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&map_q) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&map_c) : "memory");
      for (int g = 0; g < G; ++g) {
        const int sq = g % kStagesQ, sc = g % kStagesC;
        if (g >= kStagesC) ok = ok && mbar_wait(&c_empty[sc], ((g / kStagesC) - 1) & 1);
        mbar_arrive_expect_tx(&c_full[sc], kCBytes);
        tma_2d(smem + kOffC + sc * kCBytes, &map_c, g * kGroupCodeBytes, n0, &c_full[sc]);
        // The q stage is free once the last unit of its previous group is done.
        if (g >= kStagesQ) ok = ok && done_wait((g - kStagesQ) * NSUB + NSUB - 1);
        uint8_t* qs = smem + kOffQ + sq * kQBytes;
        mbar_arrive_expect_tx(&q_full[sq], kQTx);
        tma_2d(qs, &map_q, g * kGroup, m0, &q_full[sq]);
        tma_2d(qs + kQBytes / 2, &map_q, g * kGroup + 64, m0, &q_full[sq]);
      }
    }
    __syncwarp();
  } else if (warp == kScaleWarp) {
    // ------------------------------------------------------------- scales
    // All 32 lanes stage the scales of each chunk of kGC units (s_x of the
    // tile's tokens, s_w of its rows) into the two-slot scale ring, loading
    // chunk ch + 1 into registers while chunk ch waits for its slot.  A warp
    // of its own: the waits for a free slot (the epilogue's pace) never
    // delay the TMA issue of codes and q.
    const int nchunks = (GU + kGC - 1) / kGC;
    if (p.vec_scales) {
      // Lane l stages tokens l + 32u and weight rows l + 32u: the chunk's
      // kGC s_x of one token (and its kGW s_w of one row) are consecutive in
      // memory, so each is one vector load, against kGC strided loads.
      // Every chunk is full (GU % kGC == 0).
      using WVec = typename std::conditional<
          kGW == 4, uint2, typename std::conditional<kGW == 2, uint32_t, uint16_t>::type>::type;
      float4 xv[BT / 32];
      WVec wv[BW / 32];
      auto load_scales = [&](int ch) {
#pragma unroll
        for (int u = 0; u < BT / 32; ++u) {
          const int m = m0 + lane + 32 * u;
          xv[u] = (!DOTS && m < p.M)
                      ? __ldg(reinterpret_cast<const float4*>(p.sx + (size_t)m * GU + ch * kGC))
                      : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int u = 0; u < BW / 32; ++u) {
          const int n = n0 + lane + 32 * u;
          wv[u] = (!DOTS && n < p.N)
                      ? __ldg(reinterpret_cast<const WVec*>(p.scales + (size_t)n * G + ch * kGW))
                      : WVec{};
        }
      };
      load_scales(0);
      for (int ch = 0; ch < nchunks; ++ch) {
        const int slot = ch & 1;
        if (ch >= 2) ok = ok && mbar_wait(&s_empty[slot], ((ch >> 1) - 1) & 1);
        float* sxs = reinterpret_cast<float*>(smem + kOffS + slot * kSBytes);  // [kGC][BT]
        uint16_t* sws = reinterpret_cast<uint16_t*>(smem + kOffS + slot * kSBytes + kSxBytes);
#pragma unroll
        for (int u = 0; u < BT / 32; ++u) {
          const int t = lane + 32 * u;
          sxs[0 * BT + t] = xv[u].x;
          sxs[1 * BT + t] = xv[u].y;
          sxs[2 * BT + t] = xv[u].z;
          sxs[3 * BT + t] = xv[u].w;
        }
#pragma unroll
        for (int u = 0; u < BW / 32; ++u)
          *reinterpret_cast<WVec*>(sws + (lane + 32 * u) * kGW) = wv[u];  // [BW][kGW]
        mbar_arrive(&s_full[slot]);
        if (ch + 1 < nchunks) load_scales(ch + 1);
      }
    } else {
      constexpr int kPerX = kGC * BT / 32, kPerW = kGW * BW / 32;
      float xv[kPerX];
      uint16_t wv[kPerW];
      auto load_scales = [&](int ch) {
#pragma unroll
        for (int j = 0; j < kPerX; ++j) {
          const int idx = lane + 32 * j;  // idx = uu * BT + t
          const int uu = idx / BT, t = idx % BT, u = ch * kGC + uu, m = m0 + t;
          xv[j] = (!DOTS && u < GU && m < p.M) ? __ldg(p.sx + (size_t)m * GU + u) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < kPerW; ++j) {
          const int idx = lane + 32 * j;  // idx = r * kGW + gg
          const int r = idx / kGW, gw = ch * kGW + idx % kGW, n = n0 + r;
          wv[j] = (!DOTS && gw < G && n < p.N) ? __ldg(p.scales + (size_t)n * G + gw)
                                               : (uint16_t)0;
        }
      };
      load_scales(0);
      for (int ch = 0; ch < nchunks; ++ch) {
        const int slot = ch & 1;
        if (ch >= 2) ok = ok && mbar_wait(&s_empty[slot], ((ch >> 1) - 1) & 1);
        float* sxs = reinterpret_cast<float*>(smem + kOffS + slot * kSBytes);  // [kGC][BT]
        uint16_t* sws = reinterpret_cast<uint16_t*>(smem + kOffS + slot * kSBytes + kSxBytes);
#pragma unroll
        for (int j = 0; j < kPerX; ++j) sxs[lane + 32 * j] = xv[j];
#pragma unroll
        for (int j = 0; j < kPerW; ++j) sws[lane + 32 * j] = wv[j];
        mbar_arrive(&s_full[slot]);
        if (ch + 1 < nchunks) load_scales(ch + 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    // The issuing thread touches no shared memory and no mbarrier while its
    // MMAs run: such an access waits for the MMAs in flight, which left the
    // tensor pipe idle between groups.  The scheduler warp does the waiting;
    // the two warps meet once per unit at named barrier 1.
    constexpr uint32_t idesc = instr_desc_f16(BW, NW);
    // K steps per unit: fp16 has eight K = 16 steps per group, e4m3 four
    // K = 32 steps, each one MMA per q plane.
    constexpr int kSteps = (F8 ? 4 : 8) / NSUB;
    const uint32_t issuer = elect_one();
    for (int u = 0; u < GU; ++u) {
      named_bar_sync(1, 64);
      const int g = u / NSUB, h = u % NSUB;
      const int sq = g % kStagesQ, b = g % kABuf, db = u % kDBuf;
      tc_fence_after();
      // Between two MMAs of a unit only an add: the descriptor's start
      // address field is in 16-byte units.
      const uint64_t qd = smem_desc_sw128(smem_u32(smem + kOffQ + sq * kQBytes));
      const uint32_t d_tmem = tmem_base + kDCol + db * NW;
      const uint32_t a_tmem = tmem_base + kACol + b * kACols;  // b = g % kABuf
      if constexpr (F8) {
        // Plane 0 (16a) is B box 0 and plane 1 (b) box 1 (NW rows x 128
        // bytes each); K step k sits at 32-byte offset k in the swizzled row
        // and in A columns 8k..8k+7, for both planes.
#pragma unroll
        for (int pl = 0; pl < 2; ++pl)
#pragma unroll
          for (int i = 0; i < kSteps; ++i) {
            const int k = h * kSteps + i;
            const uint64_t boff16 = (uint64_t)((pl * (NW * 128) + k * 32) >> 4);
            mma_f8_ta(issuer, d_tmem, a_tmem + 8 * k, qd + boff16, idesc,
                      (pl > 0 || i > 0) ? 1u : 0u);
          }
      } else {
#pragma unroll
        for (int i = 0; i < kSteps; ++i) {
          // fp16 K step k: B box k/4 (NW rows x 128 bytes) at 32-byte offset
          // (k%4) inside the swizzled row, A columns 8k..8k+7.
          const int k = h * kSteps + i;
          const uint64_t boff16 = (uint64_t)(((k >> 2) * (NW * 128) + (k & 3) * 32) >> 4);
          mma_f16_ta(issuer, d_tmem, a_tmem + 8 * k, qd + boff16, idesc, i > 0 ? 1u : 0u);
        }
      }
      // One commit per unit tells the q producer, the decoders and the
      // epilogue alike.
      mma_commit(issuer, &g_done[u % kDone]);
    }
  } else if (warp == kSchedWarp) {
    // ------------------------------------------------------------ scheduler
    // Per unit: A decoded (lane 0) and q tile landed (lane 1) for the first
    // unit of a group, D buffer read by the epilogue (lane 2); then release
    // the MMA warp.  Both warps run exactly GU rounds of named barrier 1,
    // whatever the waits return, so a wait that gives up (reported below)
    // cannot leave the MMA warp stuck.
    for (int u = 0; u < GU; ++u) {
      const int g = u / NSUB, h = u % NSUB;
      const int sq = g % kStagesQ, b = g % kABuf, db = u % kDBuf;
      // Lanes 0-2 wait at the same time, in one code path: three waits in
      // three divergent branches cost several hundred clocks per group even
      // when every phase has already completed.
      uint64_t* bar = lane == 0 ? &a_full[b] : lane == 1 ? &q_full[sq] : &d_empty[db];
      const uint32_t parity = lane == 0   ? (uint32_t)(g / kABuf) & 1u
                              : lane == 1 ? (uint32_t)(g / kStagesQ) & 1u
                                          : (uint32_t)((u / kDBuf) - 1) & 1u;
      if ((lane < 2 && h == 0) || (lane == 2 && u >= kDBuf)) ok = ok && mbar_wait(bar, parity);
      tc_fence_before();
      __syncwarp();
      named_bar_sync(1, 64);
    }
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------ decoders
    const int quarter = warp & 3;
    const int row = 32 * quarter + lane;
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    for (int g = 0; g < G; ++g) {
      const int sc = g % kStagesC, b = g % kABuf;
      ok = ok && mbar_wait(&c_full[sc], (g / kStagesC) & 1);
      // The A buffer is free once the last unit of its previous group is done.
      if (g >= kABuf) ok = ok && done_wait((g - kABuf) * NSUB + NSUB - 1);
      tc_fence_after();
      const uint8_t* cs = smem + kOffC + sc * kCBytes + row * kGroupCodeBytes;
      const uint4 c0 = *reinterpret_cast<const uint4*>(cs);
      const uint4 c1 = *reinterpret_cast<const uint4*>(cs + 16);
      const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      const uint32_t taddr = tmem_base + lane_base + kACol + b * kACols;
      if constexpr (F8) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t v[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) decode_word_f8(cw[4 * h + i], v + 4 * i);
          tmem_st16(taddr + 16 * h, v);
        }
      } else {
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t v[16];
          decode_word(cw[2 * h], v);
          decode_word(cw[2 * h + 1], v + 8);
          tmem_st16(taddr + 16 * h, v);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      warp_arrive(&c_empty[sc]);
      warp_arrive(&a_full[b]);
    }
  } else if (warp >= 6 && warp < 6 + kEpiLive) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int col0 = ((warp - 6) >> 2) * kEpiCols;
    const int row = 32 * quarter + lane;
    const int n = n0 + row;
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    // Token pairs (2j, 2j+1) of the thread's columns, as packed fp32 pairs.
    uint64_t acc2[kCols / 2];
#pragma unroll
    for (int j = 0; j < kCols / 2; ++j) acc2[j] = 0ull;
    const int nchunks = (GU + kGC - 1) / kGC;
    const bool live = m0 + col0 < p.M;  // some token of the warp's columns is real
    for (int ch = 0; ch < nchunks; ++ch) {
      const int slot = ch & 1;
      ok = ok && mbar_wait(&s_full[slot], (ch >> 1) & 1);
      const float* sxs = reinterpret_cast<const float*>(smem + kOffS + slot * kSBytes);
      const __half* sws = reinterpret_cast<const __half*>(smem + kOffS + slot * kSBytes + kSxBytes);
#pragma unroll 1
      for (int uu = 0; uu < kGC; ++uu) {
        const int u = ch * kGC + uu;
        if (u >= GU) break;
        const int db = u % kDBuf;
        ok = ok && done_wait(u);
        tc_fence_after();
        if (!live) {
          // No valid token in this warp's columns (a partial last tile, as
          // for M = 16): release D without reading it.  The wait above keeps
          // the warp in step: its arrival for unit u + kDBuf cannot come
          // before every warp has released unit u's buffer.
          tc_fence_before();
          __syncwarp();
          warp_arrive(&d_empty[db]);
          continue;
        }
        const float* sxg = sxs + uu * BT + col0;
        const float sw = __half2float(sws[row * kGW + uu / NSUB]);
        const uint64_t sw2 = f2_pack(__float_as_uint(sw), __float_as_uint(sw));
        const uint32_t taddr = tmem_base + lane_base + kDCol + db * NW + col0;
#pragma unroll
        for (int hh = 0; hh < kCols / 16; ++hh) {
          uint32_t v[16];
          tmem_ld16(taddr + 16 * hh, v);
          tmem_ld_wait();
          if (hh == kCols / 16 - 1) {
            // D has been read: release the buffer to the MMA before the math.
            tc_fence_before();
            __syncwarp();
            warp_arrive(&d_empty[db]);
          }
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            // four tokens' s_x per 16-byte broadcast load
            const uint4 xv = *reinterpret_cast<const uint4*>(sxg + 16 * hh + 4 * j4);
            if (DOTS) {
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                const int m = m0 + col0 + 16 * hh + 4 * j4 + jj;
                const float dot = __uint_as_float(v[4 * j4 + jj]);  // exact integer unit dot
                if (m < p.M && n < p.N) p.dots[((size_t)m * p.N + n) * GU + u] = (int32_t)dot;
              }
            } else {
              // acc += (dot * s_x) * s_w for two tokens per instruction pair
              const int t2 = (16 * hh + 4 * j4) / 2;
              epi_fma2(acc2[t2], v[4 * j4], v[4 * j4 + 1], xv.x, xv.y, sw2);
              epi_fma2(acc2[t2 + 1], v[4 * j4 + 2], v[4 * j4 + 3], xv.z, xv.w, sw2);
            }
          }
        }
      }
      __syncwarp();
      warp_arrive(&s_empty[slot]);
    }
    if (!DOTS && n < p.N) {
#pragma unroll
      for (int t = 0; t < kCols; ++t) {
        const int m = m0 + col0 + t;
        const float a = __uint_as_float((uint32_t)(acc2[t / 2] >> (32 * (t & 1))));
        if (m < p.M) {
          const size_t o = (size_t)m * p.N + n;
          if (p.y_bf16)
            static_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(a);
          else
            static_cast<float*>(p.y)[o] = a;
        }
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

template <bool DOTS, bool F8, int NSUB, int NW>
int launch_mm_t(const CUtensorMap& mq, const CUtensorMap& mc, const MmParams& p,
                cudaStream_t stream) {
  auto kern = mm_kernel<DOTS, F8, NSUB, NW>;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Layout<NW>::smemBytes) !=
        cudaSuccess)
      return PQ2_ERR_LAUNCH;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.M + BT - 1) / BT, (p.N + BW - 1) / BW);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Layout<NW>::smemBytes;
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

template <int NSUB, int NW = BT>
int launch_mm_n(bool f8, bool dots, const CUtensorMap& mq, const CUtensorMap& mc,
                const MmParams& p, cudaStream_t stream) {
  if (f8)
    return dots ? launch_mm_t<true, true, NSUB, NW>(mq, mc, p, stream)
                : launch_mm_t<false, true, NSUB, NW>(mq, mc, p, stream);
  return dots ? launch_mm_t<true, false, NSUB, NW>(mq, mc, p, stream)
              : launch_mm_t<false, false, NSUB, NW>(mq, mc, p, stream);
}

}  // namespace

int launch_mm(const void* q_op, bool f8, const float* sx, const int32_t* qsum,
              const uint8_t* codes, const uint16_t* scales, void* y, int y_dtype, int32_t* dots,
              int64_t M, int64_t N, int64_t K, int sm_count, int32_t* status,
              cudaStream_t stream, int act_group) {
  (void)sm_count;
  if (act_group != 128 && act_group != 64 && act_group != 32) return PQ2_ERR_SHAPE;
  const int nsub = kGroup / act_group;
  if (M > (int64_t)1 << 20 || N > (int64_t)1 << 30) return PQ2_ERR_SHAPE;
  if ((M + BT - 1) / BT > 0x7fffffff || (N + BW - 1) / BW > 65535) return PQ2_ERR_SHAPE;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PQ2_ERR_LAUNCH;
  // At most kNarrowN tokens (activation groups of 128): the narrow kernel.
  const bool narrow = nsub == 1 && M <= kNarrowN;
  CUtensorMap mq, mc;
  {
    // q: fp16 [M][K] (or its e4m3 planes, the same 2 bytes per element),
    // box 64 x 128 (128-byte rows; kNarrowN rows for the narrow kernel),
    // 128-byte swizzle.
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)(narrow ? kNarrowN : BT)};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&mq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(q_op), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PQ2_ERR_LAUNCH;
  }
  {
    // codes: u8 [N][K/4], box 32 x 128 (one group of 128 rows), no swizzle.
    const cuuint64_t dims[2] = {(cuuint64_t)(K / 4), (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)(K / 4)};
    const cuuint32_t box[2] = {(cuuint32_t)kGroupCodeBytes, (cuuint32_t)BW};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PQ2_ERR_LAUNCH;
  }
  MmParams p{};
  (void)qsum;
  p.sx = sx; p.scales = scales; p.y = y; p.dots = dots; p.status = status;
  p.M = (int)M; p.N = (int)N; p.K = (int)K; p.G = (int)(K / kGroup);
  p.y_bf16 = y_dtype == PQ2_BF16;
  // One vector load per token (kGC s_x) and per row (kGC / nsub s_w) for
  // every chunk: whole chunks, and both start addresses aligned to the load.
  const int gw = kGC / nsub;
  p.vec_scales = (p.G % gw == 0) && reinterpret_cast<uintptr_t>(sx) % 16 == 0 &&
                 reinterpret_cast<uintptr_t>(scales) % (2 * gw) == 0;
  if (nsub == 2) return launch_mm_n<2>(f8, dots != nullptr, mq, mc, p, stream);
  if (nsub == 4) return launch_mm_n<4>(f8, dots != nullptr, mq, mc, p, stream);
  if (narrow) return launch_mm_n<1, kNarrowN>(f8, dots != nullptr, mq, mc, p, stream);
  return launch_mm_n<1>(f8, dots != nullptr, mq, mc, p, stream);
}

}  // namespace pq2
