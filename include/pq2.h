/*
 * pq2.h — C ABI of libpq2, the GB300 (sm_103a) library for the small-batch
 * and prefill matrix multiply of a ternary-quantised LLM ("PQ2" weights).
 *
 * The method (pages "Kernel experiments: recorded evidence", abbreviated KE,
 * and "Baseline and the integer breakthrough", abbreviated BIB):
 *   * weights: each row of K weights is K/128 blocks of 34 bytes — an fp16
 *     scale s_w followed by 32 code bytes; weight k of a block is the 2-bit
 *     field k%4 of code byte k/4, and code c means weight c-1 (KE Test 1,
 *     Diagram 1; BIB "Unpack four weights with fewer instructions").
 *   * activations: each group of 128 consecutive activations of a row is
 *     quantised to INT8 with s_x = max|x|/127 (fp32), q = clamp(round half to
 *     even(x / s_x), -127, 127) (KE Test 6; BIB "Calculate with small
 *     integers", step 1).
 *   * output: y[m][n] = sum over groups g of dot_g * s_x[m][g] * s_w[n][g],
 *     dot_g the exact int32 dot of the group's weights and q (BIB steps 3-4),
 *     accumulated in fp32.
 *
 * Conventions shared by every entry point:
 *   * Pointers marked (device) are CUDA device pointers owned by the caller;
 *     the library never allocates, frees or keeps them.  Buffers passed to
 *     one call must not overlap unless stated.  The activations x and the
 *     output y of pq2_quantize_act, pq2_mmv and pq2_linear are read and
 *     written with plain loads and stores, so they may also be pinned host
 *     memory that the device addresses at its own address (unified
 *     addressing, e.g. over NVLink-C2C); weights and q must be device
 *     memory (tensor-memory-access copies).
 *   * `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     enqueued on it; no call synchronises the host with the device.
 *   * Shapes: K > 0 and K % 128 == 0, N >= 1, M in the entry point's range.
 *   * Argument errors are returned before anything is enqueued.  A launch
 *     failure returns PQ2_ERR_LAUNCH.  Device-side waits are bounded: a wait
 *     that gives up writes PQ2_ERR_TIMEOUT to *dev_status (when given) and
 *     the kernel returns early; results are then invalid.
 *   * The library only runs on compute capability 10.3 (GB300); any other
 *     device returns PQ2_ERR_ARCH.  Inputs must be finite (NaN/Inf in x
 *     give unspecified q).
 */
#ifndef PQ2_H
#define PQ2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point (and written to dev_status). */
enum {
  PQ2_OK = 0,
  PQ2_ERR_NULL = 1,      /* a required pointer is NULL                       */
  PQ2_ERR_SHAPE = 2,     /* M, N, K, a stride or a size is out of range      */
  PQ2_ERR_ALIGN = 3,     /* a pointer or stride breaks its alignment rule    */
  PQ2_ERR_DTYPE = 4,     /* unknown dtype or layout enum                     */
  PQ2_ERR_ARCH = 5,      /* current device is not compute capability 10.3   */
  PQ2_ERR_LAUNCH = 6,    /* the CUDA launch reported an error                */
  PQ2_ERR_TIMEOUT = 7,   /* a bounded device wait gave up (dev_status only)  */
  PQ2_ERR_CUDA = 8       /* a CUDA runtime query failed (no device, ...)     */
};

/* Element types of activations (x) and outputs (y). */
enum { PQ2_BF16 = 0, PQ2_F16 = 1, PQ2_F32 = 2 };

/* Layouts of the quantised activations written by pq2_quantize_act.
 *  PQ2_Q_ROWS   int8 q[M][K], row-major, natural order.
 *  PQ2_Q_PLANES int8, plane order inside every 128-group: element i of a
 *               group is stored at (i%4)*32 + i/4 (KE Test 21, plane-order
 *               quantisation), so that plane s of a 4-byte code word meets
 *               one contiguous 4-byte slice of q.  Operand of pq2_mmv.
 *  PQ2_Q_F16    fp16, the same integer values widened exactly (|q| <= 127),
 *               in the K order pq2_mm's weight decode produces: inside every
 *               16 consecutive elements (the 16 weights of one 4-byte code
 *               word), element 4b + s (code byte b, field s) is stored at
 *               position 4s + 2(b & 1) + (b >> 1).  Operand of pq2_mm: sm_103a
 *               has no 8-bit integer tcgen05 MMA, so the prefill contraction
 *               runs on the fp16 tensor path, whose fp32 sums of integer
 *               products below 2^24 are exact.
 *  PQ2_Q_F8     two e4m3 planes per 128-group (2 bytes per element, the size
 *               of PQ2_Q_F16): q = 16a + b with a = q >> 4 in [-8, 7] and
 *               b = q & 15 in [0, 15], both exact in e4m3; bytes 0..127 of a
 *               group hold e4m3(16a), bytes 128..255 hold e4m3(b), each in
 *               the K order of pq2_mm_f8's weight decode: inside every 16
 *               consecutive elements, element 8h + 2e + o (h, o in {0, 1},
 *               e = 0..3) is stored at position 4(2h + o) + e.  Operand of
 *               pq2_mm_f8 (the 8-bit tensor path, two MMAs per K step).
 *  PQ2_Q_MMV16  fp16 [M][K], the B operand of the small-batch tensor-core
 *               GEMV pq2_mmv_tc, 128-groups only: inside every group,
 *               position 32t + 4j + 2r + e (t, j, r, e = 0..3, 0..7, 0..1,
 *               0..1) holds element i = 16(t + 4(j/4)) + 8e + f with
 *               f = 2(j%4) + r, divided by 4^f for f <= 4 and by 4^(f-3) for
 *               f >= 5 (exact: powers of two).  With this layout qsum does
 *               not receive sum(q) but the group's offset correction
 *               sum_i q_i (1 + 1024 / scale_i), scale_i that element's
 *               divisor (an exact integer, |.| < 2^22). */
enum { PQ2_Q_ROWS = 0, PQ2_Q_PLANES = 1, PQ2_Q_F16 = 2, PQ2_Q_F8 = 3, PQ2_Q_MMV16 = 4 };

/* Version of the prepared plane layout; bump whenever what a kernel reads
 * changes, so callers can key caches on it (BIB: a layout switch must change
 * the compile identity). */
int pq2_layout_version(void);

/* Static, never-NULL description of a status code. */
const char *pq2_status_string(int status);

/* Bytes of a prepared matrix: codes N*K/4 plus scales N*(K/128)*2 — still
 * exactly 34 bytes per 128 weights (KE Test 4).  0 if the shape is invalid. */
size_t pq2_prepared_bytes(int64_t N, int64_t K);

/* pq2_prepare — split raw blocks into a code plane and a scale plane
 * (KE Test 1 prepare_pq2 with separate buffers; Test 4 shared prepared
 * layout).  A pure byte move: values are unchanged.
 *   raw            (device) u8, N rows of K/128 blocks of 34 bytes, rows
 *                  raw_row_stride bytes apart (>= K/128*34).
 *   codes          (device) u8[N][K/4]; 16-byte aligned.
 *   scales         (device) fp16 bit patterns [N][K/128]; 2-byte aligned.
 * raw must not overlap codes or scales. */
int pq2_prepare(const uint8_t *raw, int64_t raw_row_stride, int64_t N,
                int64_t K, uint8_t *codes, uint16_t *scales, void *stream);

/* pq2_quantize_act — per-128-group INT8 quantisation of activations
 * (KE Test 6 _quantize; BIB "Calculate with small integers", step 1):
 *   s = max|x| / 127 (fp32 IEEE division); d = s > 0 ? s : 1;
 *   q = clamp(round-half-even(x / d), -127, 127) (IEEE division).
 *   x        (device) x_dtype [M][ldx], ldx >= K elements.
 *   M        1 .. 1<<20.
 *   q        (device) written in q_layout: int8 [M][K] for ROWS/PLANES,
 *            fp16 [M][K] for F16 and MMV16, bytes [M][2K] for F8; 16-byte
 *            aligned.
 *   sx       (device) fp32 [M][K/128] activation scales; 4-byte aligned.
 *   qsum     (device, may be NULL) int32 [M][K/128], sum of q per group
 *            (KE Test 21, the correction for the codes' -1 offset). */
int pq2_quantize_act(const void *x, int x_dtype, int64_t ldx, int64_t M,
                     int64_t K, void *q, int q_layout, float *sx,
                     int32_t *qsum, void *stream);

/* Decoders of the 2-bit codes used by the small-batch kernel; both give the
 * same exact int32 group dots.
 *  PQ2_DECODE_ADDXOR  the pages' add/XOR expansion (KE Test 1 _expand_byte;
 *                     BIB "Unpack four weights with fewer instructions"):
 *                     four codes spread one per byte, + 0x7F7F7F7F,
 *                     ^ 0x80808080, giving signed bytes c-1 for a signed
 *                     dp4a.
 *  PQ2_DECODE_PLANES  masked planes (KE Test 21): byte & (3 << 2s) = c*4^s
 *                     for an unsigned x signed dp4a, each plane shifted back
 *                     and the -1 offset removed once per group with sum(q). */
enum { PQ2_DECODE_ADDXOR = 0, PQ2_DECODE_PLANES = 1 };

/* pq2_mmv — small-batch (M = 1..8) ternary x INT8 GEMV with weight reuse
 * (BIB "Calculate with small integers"; KE Tests 6, 12, 14): every packed
 * weight byte is read from HBM once and used for all M columns; codes are
 * decoded in registers and multiplied with dp4a 4-way int8 dot products,
 * 32 per 128-group, into an exact int32 group dot, which is then scaled as
 * (float(dot) * s_x) * s_w and added in fp32.  The decoder is chosen from M
 * only (see pq2_mmv_decoder); pq2_mmv_ex takes it explicitly.
 *   q_planes (device) int8 [M][K] in PQ2_Q_PLANES order; 16-byte aligned.
 *   sx       (device) fp32 [M][K/128]; 4-byte aligned.
 *   qsum     (device) int32 [M][K/128] group sums of q (from
 *            pq2_quantize_act); 4-byte aligned.
 *   codes    (device) u8 [N][K/4] from pq2_prepare; 16-byte aligned.
 *   scales   (device) fp16 [N][K/128] from pq2_prepare; 2-byte aligned.
 *   y        (device) y_dtype [M][N] (PQ2_F32 or PQ2_BF16, bf16 = round to
 *            nearest even of the fp32 result); aligned to its element.
 *   dev_status (device, may be NULL) int32; PQ2_ERR_TIMEOUT is stored there
 *            if a device wait gives up; never cleared by the library.
 * Batch invariance: the fp32 operation sequence of output column m depends
 * only on (N, K) and the device's SM count, never on M, and the group dots
 * are exact, so column m is bit-identical for every M that contains it. */
int pq2_mmv(const int8_t *q_planes, const float *sx, const int32_t *qsum,
            const uint8_t *codes, const uint16_t *scales, void *y,
            int y_dtype, int64_t M, int64_t N, int64_t K, int32_t *dev_status,
            void *stream);

/* Flags of pq2_mmv_ex.  Every libpq2 kernel is launched with programmatic
 * dependent launch: it may start before the kernel enqueued before it on the
 * stream completes, and waits for it before reading anything that kernel may
 * write.  pq2_quantize_act, pq2_mmv, pq2_mmv_ex and pq2_mmv_gated release
 * the next kernel as soon as they start; pq2_mm releases it only once the kernel before it
 * has completed.  So the kernels that may still run when a call starts are
 * those enqueued at or after the latest "ordering point" before it: a
 * pq2_mm call, a host synchronisation, an event wait, a copy, or a kernel
 * launched without programmatic dependent launch (pq2_prepare is one).
 * Without flags a call needs nothing of this.
 *  PQ2_MMV_OVERLAP_WEIGHTS  the call may stream codes and scales from HBM
 *      before earlier kernels complete.  Legal when no kernel that may still
 *      run writes codes or scales (e.g. the weights were prepared before the
 *      latest ordering point).
 *  PQ2_MMV_INDEPENDENT      the call reads every input early and computes
 *      before earlier kernels complete.  Legal when no kernel that may still run writes any input of this call
 *      (e.g. back-to-back projections of the same quantised activations).
 *      y is always written only after the kernel before the call has
 *      completed. */
enum { PQ2_MMV_OVERLAP_WEIGHTS = 1, PQ2_MMV_INDEPENDENT = 2 };

/* pq2_mmv with an explicit decoder (PQ2_DECODE_ADDXOR or PQ2_DECODE_PLANES)
 * and flags; results are bit-identical to pq2_mmv for every decoder. */
int pq2_mmv_ex(const int8_t *q_planes, const float *sx, const int32_t *qsum,
               const uint8_t *codes, const uint16_t *scales, void *y,
               int y_dtype, int64_t M, int64_t N, int64_t K, int decode,
               int flags, int32_t *dev_status, void *stream);

/* pq2_mmv_tc — the small-batch GEMV (M = 1..8) on the legacy tensor-core
 * path (mma.sync m16n8k16, fp16 operands, fp32 accumulation): the same
 * output as pq2_mmv, bit for bit, at an arithmetic cost that does not grow
 * with M.  Each code word is expanded in registers, one logic operation per
 * two weights, into the exact fp16 values 1024 + c * 4^f; the activations
 * come divided by the same powers of four (PQ2_Q_MMV16), so every product is
 * an integer and the fp32 sum of a group is exact; subtracting the group's
 * correction leaves the exact dot of BIB step 3.  The split of the groups,
 * the scaling (float(dot) * s_x) * s_w and the order of the fp32 additions
 * are pq2_mmv's (a function of N, K and the SM count only), hence the same
 * bits and the same batch invariance.
 *   q_mmv16  (device) fp16 [M][K] from pq2_quantize_act(PQ2_Q_MMV16);
 *            16-byte aligned.
 *   sx       (device) fp32 [M][K/128] from the same call.
 *   qcorr    (device) int32 [M][K/128], the corrections that call writes to
 *            its qsum argument.
 *   codes, scales, y, y_dtype, M, N, K, flags, dev_status as for pq2_mmv_ex
 *            (flags: the same stream contract).
 * Returns PQ2_ERR_SHAPE for shapes whose per-CTA tiling it does not cover
 * (none of the library's geometries), else as pq2_mmv_ex. */
int pq2_mmv_tc(const uint16_t *q_mmv16, const float *sx, const int32_t *qcorr,
               const uint8_t *codes, const uint16_t *scales, void *y, int y_dtype,
               int64_t M, int64_t N, int64_t K, int flags, int32_t *dev_status,
               void *stream);

/* 1 if pq2_linear runs the tensor-core GEMV (pq2_mmv_tc on PQ2_Q_MMV16) for
 * M columns of an N x K matrix on a device with sm_count SMs, 0 if it runs
 * pq2_mmv (host only, no CUDA call); the results are the same.  The choice
 * follows the two kernels' measured cost: the tensor-core GEMV from M = 6,
 * and at M = 5 where a CTA of pq2_mmv_geometry holds at most 72 rows in at
 * most 8 splits. */
int pq2_linear_tensor_gemv(int64_t M, int64_t N, int64_t K, int sm_count);

/* pq2_linear — the complete projection y = x W^T (quantise, then the GEMV),
 * as the pages time it ("complete call", KE Tests 3, 6): pq2_quantize_act
 * into the caller's workspace, then pq2_mmv (M = 1..8; pq2_mmv_tc on
 * PQ2_Q_MMV16 for the M where pq2_linear_tensor_gemv says so, with the same
 * bits) with PQ2_MMV_OVERLAP_WEIGHTS, so that it streams the weights while
 * the quantisation and the kernel before it finish, or pq2_mm_f8 on PQ2_Q_F8
 * (M >= 9; bit-identical to pq2_mm, faster).  Hence
 * codes and scales must not be written by a kernel that may still run when
 * the call starts (see the flags of pq2_mmv_ex).
 * Results are bit-identical to pq2_quantize_act + pq2_mmv / pq2_mm_f8.
 * The workspace holds q with one byte per element for M <= 4 and two
 * otherwise (the tensor-core GEMV and the prefill GEMM take 16-bit q).
 *   x         (device) x_dtype [M][ldx], ldx >= K; M 1 .. 1<<20 (M 9..15,
 *             between the pages' GEMV and prefill sizes, run as the prefill
 *             GEMM's one partial token tile).
 *   workspace (device) pq2_linear_workspace_bytes(M, K) bytes, 256-byte
 *             aligned, holding q, s_x and sum(q); contents are scratch.
 *   codes, scales, y, y_dtype, dev_status as for pq2_mmv. */
int pq2_linear(const void *x, int x_dtype, int64_t ldx, int64_t M, int64_t N,
               int64_t K, const uint8_t *codes, const uint16_t *scales,
               void *y, int y_dtype, void *workspace, size_t workspace_bytes,
               int32_t *dev_status, void *stream);

/* Workspace bytes pq2_linear needs for M columns of K inputs (0 if the
 * shape is invalid). */
size_t pq2_linear_workspace_bytes(int64_t M, int64_t K);

/* Activation groups of 64 or 32 (page "Kernel experiments: recorded
 * evidence", Test 9, "Smaller Q8 activation groups"): the activations get
 * one scale per act_group elements, the weights keep their 128-groups and
 * scales, and each 128-group's dot splits into 128 / act_group partial dots,
 * each scaled by its own activation scale:
 *   y[m][n] = sum_g sum_{h < 128/A} (float(dot_gh) * s_x[m][g*128/A + h])
 *             * s_w[n][g]        (fp32, each operation rounded to nearest)
 * act_group = 128 is exactly pq2_quantize_act / pq2_mmv.
 *
 * pq2_quantize_act_grouped — pq2_quantize_act with activation groups of
 * act_group (128, 64, 32) elements; sx and qsum are [M][K / act_group].
 * q keeps the layouts of pq2_quantize_act. */
int pq2_quantize_act_grouped(const void *x, int x_dtype, int64_t ldx,
                             int64_t M, int64_t K, int act_group, void *q,
                             int q_layout, float *sx, int32_t *qsum,
                             void *stream);

/* pq2_mmv_grouped — pq2_mmv_ex (masked-plane decoder, flags) on activations
 * quantised by pq2_quantize_act_grouped with the same act_group; M 1..8.
 * The kernel holds four columns' partial sums at most: M = 5..8 runs as two
 * passes over the weights (columns 0..3, then 4..M-1), with the same bits as
 * one pass (a column's result does not depend on the others).  Batch
 * invariant like pq2_mmv.  Returns PQ2_ERR_SHAPE for M > 8 or another
 * act_group, else as pq2_mmv_ex. */
int pq2_mmv_grouped(const int8_t *q_planes, const float *sx,
                    const int32_t *qsum, const uint8_t *codes,
                    const uint16_t *scales, void *y, int y_dtype, int64_t M,
                    int64_t N, int64_t K, int act_group, int flags,
                    int32_t *dev_status, void *stream);

/* The exact partial dots of pq2_mmv_grouped, dots[m][n][j] = sum over k in
 * [j*A, j*A + A) of (c_{n,k} - 1) q_{m,k}, from the same device code, for
 * parity checks (M 1..8, q in PQ2_Q_PLANES order, qsum from
 * pq2_quantize_act_grouped).  dots (device) int32 [M][N][K / A]. */
int pq2_debug_group_dots_grouped(const int8_t *q_planes, const int32_t *qsum,
                                 const uint8_t *codes, int64_t M, int64_t N,
                                 int64_t K, int act_group, int32_t *dots,
                                 int32_t *dev_status, void *stream);

/* PTQ1_0 weights (page "KERNEL_REPORT: PTQ1_0 small-batch decoding on the
 * PrismML fork, RTX 3060 12GB", "What the source said"): each row of K
 * weights is K/128 blocks of 28 bytes: qs (bytes 0-23, five trits per byte),
 * qh (bytes 24-25, four trits per byte), the fp16 scale d (bytes 26-27,
 * little-endian).  Trit n (0 first) of a byte b is floor(b * 3^(n+1) / 256)
 * mod 3, the digit left above the low byte after n + 1 multiplications by 3;
 * trit t means weight t - 1.  Weight order inside a block (the page does
 * not fix it; this library's reading): trit n of qs byte j is weight 24n + j,
 * trit n of qh byte j is weight 120 + 2n + j.
 *
 * pq2_ptq_prepare — raw blocks (device, N rows, row stride raw_row_stride
 * bytes >= 28 K/128) -> qs plane u8[N][24 K/128] (16-byte aligned) and side
 * plane u32[N][K/128] (8-byte aligned): bits 0-15 qh (byte 24 low), bits
 * 16-31 d.  A byte move; K % 256 == 0. */
int pq2_ptq_prepare(const uint8_t *raw, int64_t raw_row_stride, int64_t N,
                    int64_t K, uint8_t *qs, uint32_t *side, void *stream);

/* pq2_ptq_mmv — y[m][n] = sum_g d_g * sum_h float(dot_gh) * s_x[m][g*128/A+h]
 * for M = 1..4 columns of activations quantised by pq2_quantize_act_grouped
 * with the same act_group A (128, 64 or 32; PQ2_Q_ROWS layout, sum(q)
 * required), dot_gh the exact integer dot of activation group h of block g:
 * fp32, each operation rounded to nearest, a fixed order that depends on
 * (N, K, SM count) only, so column m is bit-identical for every M.
 * y fp32 or bf16 (RNE of the fp32 result) [M][N].  flags as pq2_mmv_ex
 * (PQ2_MMV_OVERLAP_WEIGHTS, PQ2_MMV_INDEPENDENT, same stream contract).
 * K % 256 == 0; the kernel has no waits that can time out. */
int pq2_ptq_mmv(const int8_t *q_rows, const float *sx, const int32_t *qsum,
                const uint8_t *qs, const uint32_t *side, void *y, int y_dtype,
                int64_t M, int64_t N, int64_t K, int act_group, int flags,
                void *stream);

/* pq2_ptq_linear — the complete PTQ1_0 projection: pq2_quantize_act_grouped
 * (PQ2_Q_ROWS, act_group) into the caller's workspace, then pq2_ptq_mmv with
 * PQ2_MMV_OVERLAP_WEIGHTS (the GEMV streams its weights while the
 * quantisation runs; qs and side must not be written by a kernel that may
 * still run).  Bit-identical to the two calls.
 *   x         (device or device-addressable host) x_dtype [M][ldx], M 1..4.
 *   workspace (device) pq2_ptq_linear_workspace_bytes(M, K, act_group)
 *             bytes, 256-byte aligned; contents are scratch.
 * Returns PQ2_ERR_SHAPE for a workspace that is too small, else as the two
 * calls. */
size_t pq2_ptq_linear_workspace_bytes(int64_t M, int64_t K, int act_group);
int pq2_ptq_linear(const void *x, int x_dtype, int64_t ldx, int64_t M,
                   int64_t N, int64_t K, const uint8_t *qs, const uint32_t *side,
                   int act_group, void *y, int y_dtype, void *workspace,
                   size_t workspace_bytes, void *stream);

/* The exact partial dots of pq2_ptq_mmv, dots[m][n][j] = sum over k in
 * [jA, jA + A) of (t_{n,k} - 1) q_{m,k}, from the same device code (parity
 * checks).  dots (device) int32 [M][N][K / A]. */
int pq2_debug_ptq_dots(const int8_t *q_rows, const int32_t *qsum,
                       const uint8_t *qs, const uint32_t *side, int64_t M,
                       int64_t N, int64_t K, int act_group, int32_t *dots,
                       void *stream);

/* pq2_mmv_gated — the gate/up projection with its gated activation in the
 * GEMV's epilogue (page "Kernel experiments: recorded evidence", Test 12,
 * "gated" fusion screen: the projection's output z = x W^T of width N is
 * split in halves, gate = z[:, :N/2], up = z[:, N/2:], and the result is
 * silu(gate) * up computed in fp32 and rounded to the output type):
 *   out[m][n] = silu(y[m][n]) * y[m][n + N/2],  n < N/2,
 *   silu(v)   = v / (1 + exp(-v)),
 * each operation in fp32 with round-to-nearest (exp: CUDA's expf, 2 ulp),
 * where y is the fp32 sum pq2_mmv forms for those rows, with the same
 * operation order (the split count comes from all N rows), so gate and up
 * are bit-identical to pq2_mmv's y.  Batch invariant like pq2_mmv.  Gate
 * row n and up row n + N/2 are streamed by the same CTA; the N/2 x M
 * intermediate never exists.
 *   q_planes, sx, qsum, codes, scales, M, K, flags, dev_status as for
 *            pq2_mmv_ex (masked-plane decoder).  codes/scales hold N rows:
 *            the gate rows, then the up rows.
 *   N        even, 2 .. 1<<30.
 *   out      (device) out_dtype [M][N/2] (PQ2_F32 or PQ2_BF16).
 * Returns PQ2_ERR_SHAPE for an odd N, else as pq2_mmv_ex. */
int pq2_mmv_gated(const int8_t *q_planes, const float *sx, const int32_t *qsum,
                  const uint8_t *codes, const uint16_t *scales, void *out,
                  int out_dtype, int64_t M, int64_t N, int64_t K, int flags,
                  int32_t *dev_status, void *stream);

/* pq2_linear_gated — the complete gated call for M = 1..8:
 * pq2_quantize_act into the workspace, then pq2_mmv_gated with
 * PQ2_MMV_OVERLAP_WEIGHTS (the stream contract of pq2_linear).  Results are
 * bit-identical to pq2_quantize_act + pq2_mmv_gated.
 *   x, x_dtype, ldx, workspace as for pq2_linear (M 1..8 only);
 *   N, codes, scales, out, out_dtype, dev_status as for pq2_mmv_gated. */
int pq2_linear_gated(const void *x, int x_dtype, int64_t ldx, int64_t M,
                     int64_t N, int64_t K, const uint8_t *codes,
                     const uint16_t *scales, void *out, int out_dtype,
                     void *workspace, size_t workspace_bytes,
                     int32_t *dev_status, void *stream);

/* Size of the static device scratch of pq2_linear_static (1 MiB). */
#define PQ2_STATIC_SCRATCH_BYTES ((size_t)1 << 20)

/* pq2_linear_static — pq2_linear for callers that cannot allocate device
 * memory (for example code running where cudaMalloc is not allowed, or
 * runtimes whose allocator owns all device memory).  The pages have no
 * counterpart: this is a deployment convenience, not a step of the method.
 * The call allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine): its workspace (q, s_x and sum(q), laid out as for pq2_linear) is
 * a file-scope static device array of PQ2_STATIC_SCRATCH_BYTES in every
 * device's context, which each device holds until the process exits.  Its
 * device address is looked up (cudaGetSymbolAddress) with the device current
 * on the first call on that device, which also creates the device's primary
 * context, and again whenever the current context differs from the one the
 * address was found in (after a device reset).  Make the first call on a
 * device before capturing any stream into a graph.
 *   Arguments, results and errors as for pq2_linear, without the workspace;
 *   errors in pq2_linear's order (NULL, dtype, shape).
 *   stream   must belong to the current device (NULL is the current
 *            device's legacy default stream): the scratch address is the
 *            current device's.  Another device's stream returns PQ2_ERR_CUDA.
 *   Returns PQ2_ERR_SHAPE, before any CUDA call, when
 *   pq2_linear_workspace_bytes(M, K) exceeds PQ2_STATIC_SCRATCH_BYTES (for
 *   example M = 4 with K above 246,656, M = 8 with K above 63,488, or
 *   M = 16 with K above 31,744);
 *   PQ2_ERR_CUDA if the scratch address cannot be obtained.
 * Every call on a device shares the one scratch array, which keeps the last
 * call's contents.  Nothing in it needs to start at zero: each call writes
 * all of it that it reads.  Calls that may run at the same time on the GPU
 * (for example on two streams) race on it; calls in order on one stream do
 * not. */
int pq2_linear_static(const void *x, int x_dtype, int64_t ldx, int64_t M,
                      int64_t N, int64_t K, const uint8_t *codes,
                      const uint16_t *scales, void *y, int y_dtype,
                      int32_t *dev_status, void *stream);

/* The decoder pq2_mmv uses for M columns (host only). */
int pq2_mmv_decoder(int64_t M);

/* Largest K pq2_norm_hadamard_quantize takes (a row's fp32 copy stays in
 * shared memory). */
#define PQ2_PREP_MAX_K 32768

/* pq2_norm_hadamard_quantize — the activations' preparation fused into one
 * kernel (page "Kernel experiments: recorded evidence", Test 18, "RMSNorm +
 * Hadamard + Q8 fusion"), per row m of K columns:
 *   h    = x (+ residual), fp32
 *   S    = sum of h^2: partial i (0..2047) sums h[j]^2 for j = i mod 2048 in
 *          increasing j, then p[i] += p[i + len] for len = 1024, 512, .., 1
 *          (fp32; S = p[0])
 *   inv  = 1 / sqrt(S / K + eps)            (IEEE square root and division)
 *   n    = bf16((h * inv) * (w + 1))         (norm weight w, applied as w + 1)
 *   v    = n * sign                          (sign +1 / -1 per column)
 *   v    = bf16(WHT(v)) per 1024-column block, WHT the orthonormal
 *          Walsh-Hadamard transform (butterfly passes of half-width 1, 2, ..,
 *          512 in fp32, then the exact factor 1/32)
 *   q, sx, qsum = pq2_quantize_act of v (group 128, same rounding)
 * Every fp32 operation rounds to nearest; the codes are therefore a function
 * of the inputs alone (bit-exact against the CPU oracle).
 *   x            (device) bf16 [M][K].
 *   residual     (device, may be NULL) bf16 [M][K], added to x first.
 *   residual_out (device, may be NULL) bf16 [M][K] <- bf16(h).
 *   w            (device) bf16 [K]; sign (device) int8 [K], each +1 or -1.
 *   eps          0 <= eps <= 1.
 *   M            1 .. 1<<20;  K a multiple of 1024, 1024 .. PQ2_PREP_MAX_K.
 *   norm_out     (device, may be NULL) bf16 [M][K] <- n.
 *   q, q_layout, sx, qsum as for pq2_quantize_act.
 * Returns PQ2_ERR_SHAPE for K or eps out of range, else as
 * pq2_quantize_act; launched with programmatic dependent launch like it. */
int pq2_norm_hadamard_quantize(const uint16_t *x, const uint16_t *residual,
                               uint16_t *residual_out, const uint16_t *w,
                               const int8_t *sign, float eps, int64_t M,
                               int64_t K, uint16_t *norm_out, void *q,
                               int q_layout, float *sx, int32_t *qsum,
                               void *stream);

/* pq2_mm — prefill (M >= 16; any M >= 1) ternary x INT8 matmul as a dense tensor-core
 * contraction (KE Test 7 "INT8 tensor-core MMQ prefill"; BIB "Use matrix
 * hardware for prefill"): per 128-group the exact dot of q and the decoded
 * codes is formed on tcgen05 tensor cores (fp16 operands holding integer
 * values, fp32 accumulation confined to one group, hence exact), then scaled
 * by s_x * s_w into an fp32 accumulator.
 *   q_f16    (device) fp16 [M][K] from pq2_quantize_act(PQ2_Q_F16);
 *            16-byte aligned.
 *   sx       (device) fp32 [M][K/128].
 *   qsum     (device) int32 [M][K/128] group sums of q.
 *   codes, scales as for pq2_mmv.
 *   y        (device) y_dtype [M][N] (PQ2_F32 or PQ2_BF16).
 *   M        1 .. 1<<20 (the prefill sizes are M >= 16; a smaller M is one
 *            partial 128-token tile).
 *   dev_status as for pq2_mmv. */
int pq2_mm(const uint16_t *q_f16, const float *sx, const int32_t *qsum,
           const uint8_t *codes, const uint16_t *scales, void *y, int y_dtype,
           int64_t M, int64_t N, int64_t K, int32_t *dev_status, void *stream);

/* pq2_mm_f8 — pq2_mm on the 8-bit tensor path: the weights decode to e4m3
 * (-1, 0, +1; code 3 gives +2) and q comes as the two exact e4m3 planes of
 * PQ2_Q_F8; each K step is two kind::f8f6f4 MMAs (16a and b) accumulating
 * into the same fp32 group tile, whose integer sums stay below 2^24, so the
 * group dot is exact and y is bit-identical to pq2_mm's.
 *   q_f8     (device) [M][2K] bytes from pq2_quantize_act(PQ2_Q_F8);
 *            16-byte aligned.  Other arguments as for pq2_mm. */
int pq2_mm_f8(const uint8_t *q_f8, const float *sx, const int32_t *qsum,
              const uint8_t *codes, const uint16_t *scales, void *y,
              int y_dtype, int64_t M, int64_t N, int64_t K,
              int32_t *dev_status, void *stream);

/* pq2_mm_grouped, pq2_mm_f8_grouped — pq2_mm and pq2_mm_f8 on activations
 * quantised by pq2_quantize_act_grouped with activation groups of act_group
 * A = 128, 64 or 32 elements (KE Test 9, "Smaller Q8 activation groups":
 * the weights and their 128-weight scales stay as they are, each weight
 * group's dot splits into 128 / A separately scaled partial dots):
 *   y[m][n] = sum over weight groups g, then over h = 0 .. 128/A - 1, of
 *             (dot_gh * s_x[m][g*128/A + h]) * s_w[n][g]
 * with dot_gh the exact integer dot of activation group h of block g, each
 * a separate tensor-core accumulation (exact, as for pq2_mm), scaled in fp32.
 *   q_f16 / q_f8 as for pq2_mm / pq2_mm_f8, from pq2_quantize_act_grouped
 *            (PQ2_Q_F16 / PQ2_Q_F8, the same act_group).
 *   sx, qsum (device) [M][K / act_group].
 * act_group 128 gives exactly pq2_mm / pq2_mm_f8.  Returns PQ2_ERR_SHAPE for
 * another act_group, else as pq2_mm. */
int pq2_mm_grouped(const uint16_t *q_f16, const float *sx, const int32_t *qsum,
                   const uint8_t *codes, const uint16_t *scales, void *y,
                   int y_dtype, int64_t M, int64_t N, int64_t K, int act_group,
                   int32_t *dev_status, void *stream);
int pq2_mm_f8_grouped(const uint8_t *q_f8, const float *sx, const int32_t *qsum,
                      const uint8_t *codes, const uint16_t *scales, void *y,
                      int y_dtype, int64_t M, int64_t N, int64_t K,
                      int act_group, int32_t *dev_status, void *stream);

/* pq2_linear_grouped — the complete projection with activation groups of
 * act_group elements (128, 64, 32; KE Test 9 times exactly this call at
 * M = 128 and 512): pq2_quantize_act_grouped into the caller's workspace,
 * then pq2_mmv_grouped (M = 1..8, masked-plane decoder, weights streamed
 * while the quantisation runs) or pq2_mm_f8_grouped (M >= 9).
 * Bit-identical to those calls.
 *   x, ldx, codes, scales, y, y_dtype, dev_status as for pq2_linear.
 *   workspace (device) pq2_linear_grouped_workspace_bytes(M, K, act_group)
 *             bytes, 256-byte aligned; contents are scratch.
 * pq2_linear_grouped_workspace_bytes returns 0 for invalid arguments.
 * Returns PQ2_ERR_SHAPE for a workspace that is too small or another
 * act_group, else as the calls it makes. */
size_t pq2_linear_grouped_workspace_bytes(int64_t M, int64_t K, int act_group);
int pq2_linear_grouped(const void *x, int x_dtype, int64_t ldx, int64_t M,
                       int64_t N, int64_t K, const uint8_t *codes,
                       const uint16_t *scales, int act_group, void *y,
                       int y_dtype, void *workspace, size_t workspace_bytes,
                       int32_t *dev_status, void *stream);

/* Paths of pq2_debug_group_dots. */
enum { PQ2_PATH_MMV_ADDXOR = 0, PQ2_PATH_MM = 1, PQ2_PATH_MMV_PLANES = 2,
       PQ2_PATH_MM_F8 = 3, PQ2_PATH_MMV_TC = 4 };

/* pq2_debug_group_dots — the exact per-group int32 dots
 * dots[m][n][g] = sum_{k in g} (c_{n,k} - 1) q_{m,k} computed by the SAME
 * device decode and dot code as pq2_mmv with either decoder (paths 0 and 2,
 * q int8 in PQ2_Q_PLANES order, qsum required for path 2, M 1..8) or as
 * pq2_mm (path 1, q fp16 PQ2_Q_F16 and qsum, M >= 1) or pq2_mm_f8 (path 3,
 * q PQ2_Q_F8 and qsum, M >= 1) or pq2_mmv_tc (path 4, q PQ2_Q_MMV16 and
 * its corrections in qsum, M 1..8), for parity checks.
 *   dots (device) int32 [M][N][K/128]. */
int pq2_debug_group_dots(const void *q, const int32_t *qsum,
                         const uint8_t *codes, int64_t M, int64_t N, int64_t K,
                         int path, int32_t *dots, int32_t *dev_status,
                         void *stream);

/* pq2_debug_mm_dots_grouped — the exact partial dots of pq2_mm_grouped
 * (path PQ2_PATH_MM, q PQ2_Q_F16) or pq2_mm_f8_grouped (PQ2_PATH_MM_F8,
 * q PQ2_Q_F8) from the same device code, for parity checks:
 * dots[m][n][j] = sum over k in [j*A, j*A + A) of (c_{n,k} - 1) q_{m,k}.
 *   q from pq2_quantize_act_grouped with the same act_group; M >= 1.
 *   dots (device) int32 [M][N][K / act_group]. */
int pq2_debug_mm_dots_grouped(const void *q, int path, const uint8_t *codes,
                              int64_t M, int64_t N, int64_t K, int act_group,
                              int32_t *dots, int32_t *dev_status,
                              void *stream);

/* pq2_debug_mmv_drop_arrival — a test of the bounded device waits (the
 * status convention above), not a step of the method: pq2_mmv (masked-plane
 * decoder, no flags) in which one consumer warp does not release the first
 * ring stage of its weight pipeline, so the producer's wait for that slot,
 * limited here to wait_limit_cycles SM clocks (1000 .. 2^32), gives up.  The
 * producer then issues no further copy, waits (bounded) until every copy it
 * issued has landed, and tells the consumers to stop; the kernel writes
 * PQ2_ERR_TIMEOUT to *dev_status (required here) and returns.  y is
 * unspecified afterwards; the device and its context stay usable.  Returns
 * PQ2_ERR_SHAPE when (N, K) gives a pipeline whose slots are never reused
 * (nothing to wait for), else as pq2_mmv. */
int pq2_debug_mmv_drop_arrival(const int8_t *q_planes, const float *sx,
                               const int32_t *qsum, const uint8_t *codes,
                               const uint16_t *scales, void *y, int y_dtype,
                               int64_t M, int64_t N, int64_t K,
                               int64_t wait_limit_cycles, int32_t *dev_status,
                               void *stream);

/* pq2_mmv_geometry — the launch geometry pq2_mmv uses for (N, K) on a device
 * with sm_count SMs (host only, no CUDA call): CTAs, threads per CTA,
 * interleaved K splits per row and row count of the largest CTA.  It does
 * not depend on M. Returns PQ2_ERR_SHAPE for invalid shapes. */
int pq2_mmv_geometry(int64_t N, int64_t K, int sm_count, int *ctas,
                     int *threads, int *splits, int *rows_max);

#ifdef __cplusplus
}
#endif
#endif /* PQ2_H */
