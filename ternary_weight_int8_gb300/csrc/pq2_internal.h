// pq2_internal.h — host-side declarations shared by the libpq2 translation
// units (launchers called by the C ABI in pq2_api.cu).  Not installed.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "pq2.h"

namespace pq2 {

// Geometry of pq2_mmv, a pure function of (N, K, SM count): never of M.
struct MmvGeometry {
  int ctas;      // CTAs (one per SM, fewer when N is small)
  int threads;   // consumer threads per CTA (multiple of 32)
  int splits;    // S: interleaved K splits per row inside a CTA
  int rows_max;  // rows of the largest CTA
  int steps;     // ceil(G / S): pipeline steps (one group per thread each)
};

bool mmv_geometry(int64_t N, int64_t K, int sm_count, MmvGeometry* g);

// Decoders of the code bytes used by the small-batch kernel.
enum MmvDecode {
  kDecodeAddXor = 0,      // spread + 0x7F7F7F7F, ^ 0x80808080, signed dp4a
  kDecodeMaskPlanes = 1,  // masked planes, unsigned dp4a, minus sum(q)
  kDecodeTensor = 2       // fp16 fragments 1024 + c * 4^s, mma.sync, minus the
                          // PQ2_Q_MMV16 correction (q in that layout)
};

int launch_prepare(const uint8_t* raw, int64_t raw_stride, int64_t N,
                   int64_t K, uint8_t* codes, uint16_t* scales,
                   cudaStream_t stream);

// act_group: activation group of 128 (default), 64 or 32 elements; sx and
// qsum are [M][K / act_group].
int launch_quantize(const void* x, int x_dtype, int64_t ldx, int64_t M,
                    int64_t K, void* q, int q_layout, float* sx, int32_t* qsum,
                    cudaStream_t stream, int act_group = 128);

// overlap 1: the CTAs may stream the weight planes before the preceding
// kernels on the stream have completed (programmatic dependent launch);
// overlap 2: every input may be read early (see PQ2_MMV_INDEPENDENT).
int launch_mmv(const int8_t* q, const float* sx, const int32_t* qsum,
               const uint8_t* codes, const uint16_t* scales, void* y,
               int y_dtype, int32_t* dots, int64_t M, int64_t N, int64_t K,
               int decode, int overlap, int sm_count, int32_t* status,
               cudaStream_t stream);

// pq2_mmv with activation groups of act_group (128, 64, 32) elements: sx and
// qsum are [M][K/act_group]; dots (debug) [M][N][K/act_group].  M <= 4.
int launch_mmv_grouped(const int8_t* q, const float* sx, const int32_t* qsum,
                       const uint8_t* codes, const uint16_t* scales, void* y, int y_dtype,
                       int32_t* dots, int64_t M, int64_t N, int64_t K, int act_group,
                       int overlap, int sm_count, int32_t* status, cudaStream_t stream);

// pq2_mmv (masked planes, no overlap) with consumer warp 0 skipping its
// release of ring stage 0 and the producer's wait for a free slot limited to
// wait_limit SM clocks: the bounded-wait path, for tests.  PQ2_ERR_SHAPE when
// (N, K) gives no reused ring slot.
int launch_mmv_drop_arrival(const int8_t* q, const float* sx, const int32_t* qsum,
                            const uint8_t* codes, const uint16_t* scales, void* y, int y_dtype,
                            int64_t M, int64_t N, int64_t K, long long wait_limit, int sm_count,
                            int32_t* status, cudaStream_t stream);

// Gated gate/up output: out[m][n] = silu(y[m][n]) * y[m][n + N/2] for
// n < N/2, y as launch_mmv computes it (N even, dots not supported).
int launch_mmv_gated(const int8_t* q, const float* sx, const int32_t* qsum,
                     const uint8_t* codes, const uint16_t* scales, void* out, int out_dtype,
                     int64_t M, int64_t N, int64_t K, int decode, int overlap, int sm_count,
                     int32_t* status, cudaStream_t stream);

// Fused RMSNorm + signs + 1024-point Walsh-Hadamard + group-128 INT8
// quantisation of M rows of K bf16 activations (pq2_norm_hadamard_quantize).
int launch_norm_hadamard_quantize(const uint16_t* x, const uint16_t* residual,
                                  uint16_t* residual_out, const uint16_t* w, const int8_t* sign,
                                  float eps, int64_t M, int64_t K, uint16_t* norm_out, void* q,
                                  int q_layout, float* sx, int32_t* qsum, cudaStream_t stream);

// PTQ1_0: raw 28-byte blocks -> qs plane u8[N][24 K/128] + side plane
// u32[N][K/128] (qh | d << 16); GEMV on row-layout q with activation groups
// of act_group (128, 64, 32), M 1..4, K % 256 == 0.
int launch_ptq_prepare(const uint8_t* raw, int64_t raw_stride, int64_t N, int64_t K, uint8_t* qs,
                       uint32_t* side, cudaStream_t stream);
bool ptq_geometry(int64_t N, int64_t K, int sm_count, int* ctas, int* rows, int* splits);
int launch_ptq_mmv(const int8_t* q, const float* sx, const int32_t* qsum, const uint8_t* qs,
                   const uint32_t* side, void* y, int y_dtype, int32_t* dots, int64_t M,
                   int64_t N, int64_t K, int act_group, int overlap, int sm_count,
                   cudaStream_t stream);

// q_op: fp16 PQ2_Q_F16 (f8 false) or the e4m3 planes of PQ2_Q_F8 (f8 true).
int launch_mm(const void* q_op, bool f8, const float* sx, const int32_t* qsum,
              const uint8_t* codes, const uint16_t* scales, void* y, int y_dtype,
              int32_t* dots, int64_t M, int64_t N, int64_t K, int sm_count,
              int32_t* status, cudaStream_t stream, int act_group = 128);

}  // namespace pq2
