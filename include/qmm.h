/*
 * qmm.h -- C ABI of the GB300 (sm_103a) GGUF block-quantized matmul library.
 *
 * The operations follow the candle tutorial pages:
 *  - "同一个 GGUF，CPU 和 Metal 生成的文字不一样", section 出处: QMatMul has a CPU
 *    form that quantizes every activation row (Q8_0 activations for Q8_0
 *    weights, Q8K for K-quant weights) and takes integer block dot products,
 *    and a Metal form that multiplies f32 activations by weight blocks
 *    dequantized inside the kernel; CANDLE_DEQUANTIZE_ALL is the third form
 *    (dequantize every weight to f32, then a plain matmul).
 *  - "自己量化", section 3 (量化): QTensor::quantize(tensor, type) quantizes
 *    row-major weights along the last dimension and fails with a shape
 *    error when that dimension is not a multiple of the block size; section
 *    和下载的 Q8_0 逐字节比: a Q8_0 block's scale is max|x|/127; section
 *    动脑筋答案: activations are quantized row by row in groups of 32 (Q8_0)
 *    or 256 (Q8K).
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers owned by the caller unless stated.  The
 *    library allocates nothing.  It keeps two 4-byte device words per
 *    device: the error word (see qmm_last_device_error) and the spin limit
 *    of its bounded waits (see qmm_test_set_wait_limit).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Argument errors are returned synchronously, before
 *    anything is launched.  QMM_ERR_CUDA reports a launch error.
 *  - Stream order holds for every input and output.  The decode kernels
 *    are programmatic dependent launches: when the previous kernel in the
 *    stream is one of this library's, they may start while it finishes and
 *    read the quantized weights early, but they wait for it to complete
 *    before they read x, write y or touch the workspace.  A caller's kernel
 *    that does not itself trigger dependents early (griddepcontrol
 *    .launch_dependents) completes first, so it may write the weights.
 *  - Matrices are row-major.  W is [N, K] (N output rows, K input channels,
 *    the GGUF / Linear convention), x is [M, K], y = x . W^T is [M, N].
 *    Blocks run along K inside a row; a quantized matrix is N rows of
 *    K / block_values blocks, each block in the GGUF byte layout:
 *      Q8_0: { f16 d; int8 q[32]; }                                34 B / 32
 *      Q4_K: { f16 d; f16 dmin; u8 scales[12]; u8 q[128]; }      144 B / 256
 *      Q8_K: { f32 d; int8 q[256]; int16 bsums[16]; }             292 B / 256
 *    (Q4_K: 8 sub-blocks of 32 with 6-bit scale sc_j and min m_j packed in
 *    `scales`; byte 32c+l of q holds value l of sub-block 2c in its low
 *    nibble and value l of sub-block 2c+1 in its high nibble.)
 *  - Alignment: quantized buffers, x and workspace must start on a 16-byte
 *    boundary, float outputs on a 4-byte boundary (QMM_ERR_ALIGN).
 *  - M = 0 or N = 0 is a no-op returning QMM_OK.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* qmm_stream_t;   /* same type as cudaStream_t */

typedef enum {
    QMM_F32 = 0,    /* plain f32 (only as a dequantization target)          */
    QMM_Q8_0 = 1,   /* 32 values: f16 scale, int8 codes                      */
    QMM_Q4_K = 2,   /* 256 values: f16 d/dmin, 6-bit sub-block scales/mins   */
    QMM_Q8_K = 3,   /* 256 values: f32 scale, int8 codes, 16 int16 sums      */
    QMM_Q4_0 = 4,   /* 32 values: f16 scale, 4-bit codes offset by 8 (18 B)  */
    QMM_Q5_0 = 5,   /* 32 values: f16 scale, 5-bit codes offset by 16 (22 B) */
    QMM_Q6_K = 6    /* 256 values: 6-bit codes offset by 32, 16 int8 group scales, f16 d (210 B) */
} qmm_type;

typedef enum {
    QMM_INT8_ACT = 0,  /* CPU form: activations quantized per row, integer block dots */
    QMM_F32_ACT = 1    /* Metal form: f32 activations x in-kernel dequantized weights */
} qmm_act_mode;

typedef enum {
    QMM_OK = 0,
    QMM_ERR_NULL = 1,       /* a required pointer is NULL                        */
    QMM_ERR_SHAPE = 2,      /* negative size, or K not a multiple of the block   */
    QMM_ERR_TYPE = 3,       /* type not valid for this call / bad pairing        */
    QMM_ERR_ALIGN = 4,      /* pointer misaligned                                */
    QMM_ERR_WORKSPACE = 5,  /* workspace smaller than qmm_matmul_workspace()     */
    QMM_ERR_CUDA = 6,       /* a CUDA runtime call or launch failed              */
    QMM_ERR_TIMEOUT = 7     /* a device-side wait gave up (reported by qmm_last_device_error) */
} qmm_status;

/* Values per block: 32 (Q8_0, Q4_0, Q5_0), 256 (Q4_K, Q8_K, Q6_K), 1 (F32); 0
   for an unknown type. */
int64_t qmm_block_values(qmm_type t);

/* Bytes per block: 34 (Q8_0), 144 (Q4_K), 292 (Q8_K), 18 (Q4_0), 22 (Q5_0),
   210 (Q6_K); 4 for F32; 0 for an unknown type.  ("自己量化" section 大小和误差
   and the byte listings of section 和下载的 Q8_0 逐字节比: the printed sizes fix
   34 B per 32 values for Q8_0, 144 B per 256 for Q4K, 22 B per 32 for Q5_0,
   18 B per 32 for Q4_0, and the downloaded Q4_K_M closes with 210 B per 256
   for Q6K.) */
size_t qmm_block_bytes(qmm_type t);

/* Bytes of one quantized row of K values; 0 when K is not a multiple of the
   block size (the QTensor::quantize shape error) or K < 0. */
size_t qmm_row_bytes(qmm_type t, int64_t K);

/* Quantize weights w [N, K] (f32, device) into wq (N * qmm_row_bytes(wtype, K)
   bytes, device).  wtype: QMM_Q8_0, QMM_Q4_K, QMM_Q4_0, QMM_Q5_0 or QMM_Q6_K ("自己量化"
   section 3, QTensor::quantize).  Q8_0: per 32 values d = max|x|/127, codes
   round(x / d) with ties away from zero.  Q4_K: per sub-block of 32 a step
   (max - min(0, min))/15 and offset -min(0, min), super-block scales
   d = max step / 63 and dmin = max offset / 63, 6-bit factors and 4-bit
   codes by rounding (the pages do not give the K-quant algorithm; this is the
   closed-form min/max reading).  Q4_0 / Q5_0 (off = 8 / 16; the pages give
   only their sizes): the value m of largest magnitude (the first on ties,
   sign kept) sets d = m / -off, codes round(x / d) + off clamped to
   [0, 2 off - 1]; block = f16 d, (Q5_0) a little-endian 32-bit word whose
   bit i is bit 4 of code i, then 16 bytes with code j in the low nibble of
   byte j and code j + 16 in its high nibble (the public GGUF layout); the
   weight is f(d) (code - off).  Q6_K (the pages give only its size): per
   group of 16 the value m_j of largest magnitude (the first on ties, sign
   kept) gives s_j = m_j / -32; d = max |s_j| / 127; int8 group scales
   sc_j = round(s_j / d); codes round(x / (f(d) sc_j)) in [-32, 31], stored
   +32 as 4 low bits (ql[128]) and 2 high bits (qh[64]): value i = 128h +
   32q + l has its low bits in nibble q/2 of ql[64h + 32 (q % 2) + l] and its
   high bits in bits 2q..2q+1 of qh[32h + l]; then the 16 scales and f16 d
   (the public GGUF layout).  Errors: NULL, SHAPE (K % block), TYPE, ALIGN. */
qmm_status qmm_quantize_weights(qmm_type wtype, const float* w, int64_t N, int64_t K, void* wq,
                                qmm_stream_t stream);

/* Quantize activations x [M, K] row by row ("同一个 GGUF…" section 出处,
   from_float; "自己量化" 动脑筋答案: each row is quantized on its own).
   atype: QMM_Q8_0 (blocks of 32, f16 scale) or QMM_Q8_K (blocks of 256, f32
   scale, int16 sums of 16 codes).  Output xq: M * qmm_row_bytes(atype, K)
   bytes.  qmm_matmul(QMM_INT8_ACT) performs exactly this quantization inside
   its own launch; this call exports the codes.  Errors as above. */
qmm_status qmm_quantize_act(qmm_type atype, const float* x, int64_t M, int64_t K, void* xq,
                            qmm_stream_t stream);

/* Dequantize rows blocks -> out [rows, K] f32 (the CANDLE_DEQUANTIZE_ALL form,
   "同一个 GGUF…" section 出处).  Q8_0 and Q8_K: f(d) * q; Q4_K:
   (f(d) * sc_j) * q - f(dmin) * m_j, both products exact in f32, one rounding
   in the subtraction; Q4_0 / Q5_0: f(d) (code - off), exact; Q6_K:
   (f(d) sc_j) code, exact (bit-exact contract).  t: Q8_0, Q4_K, Q8_K, Q4_0,
   Q5_0 or Q6_K. */
qmm_status qmm_dequantize(qmm_type t, const void* q, int64_t rows, int64_t K, float* out,
                          qmm_stream_t stream);

/* Workspace bytes qmm_matmul needs for this shape (0 when none).  The
   workspace holds activations prepared once per call for large decode
   weight matrices, split-K partial sums and their arrival counters, and the
   prefill GEMM's activation operand. */
size_t qmm_matmul_workspace(qmm_type wtype, qmm_act_mode mode, int64_t M, int64_t N, int64_t K);

/* Number of kernel launches one qmm_matmul call makes for this shape on the
   current device (decode: an activation-preparing kernel for large weight
   matrices, the decode kernel, a K-split reduction; prefill: the activation
   operand, for Q6_K its weights repacked to 16-byte aligned slots, and the
   GEMM).  0 for an invalid shape or type.  Launches nothing.
   (A diagnostic of this library; the pages have no counterpart.) */
int qmm_matmul_launches(qmm_type wtype, qmm_act_mode mode, int64_t M, int64_t N, int64_t K);

/* y [M, N] f32 = x [M, K] f32 . W^T with W given as quantized blocks wq
   (wtype QMM_Q8_0, QMM_Q4_K, QMM_Q4_0, QMM_Q5_0 or QMM_Q6_K).
   mode QMM_INT8_ACT ("同一个 GGUF…" section 出处, the CPU form): each row of x
     is quantized in-kernel to Q8_0 (Q8_0, Q4_0 and Q5_0 weights) or Q8_K
     (Q4_K and Q6_K weights), per-block int32 dot products of signed codes are
     formed exactly and combined as
       Q8_0, Q4_0, Q5_0: y = sum_b f(d_w) f(d_a) isum_b
       Q4_K: y = sum_s d_a (f(d) S_sc - f(dmin) S_m),
             S_sc = sum_j sc_j isum_j, S_m = sum_j m_j (sum of the sub-block's codes)
       Q6_K: y = sum_s d_a f(d) S, S = sum_j sc_j isum_j over the 16 groups of 16.
   mode QMM_F32_ACT (the Metal form): y = sum_k x_k w_k with w the dequantized
     weights, x kept at f32 accuracy.
   Floats: |y - exact| <= 1e-5 * (sum of |scaled block terms|) + 1e-6.
   workspace: device memory of at least qmm_matmul_workspace(...) bytes (may
   be NULL when that is 0); its contents need no initialisation.
   Errors: NULL, SHAPE, TYPE, ALIGN, WORKSPACE, CUDA. */
qmm_status qmm_matmul(qmm_type wtype, qmm_act_mode mode, const void* wq, const float* x, float* y,
                      int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                      qmm_stream_t stream);

/* Test hook: the exact integer block sums of the CPU form, computed by the
   same kernel, fragment layout and in-kernel activation quantization as
   qmm_matmul(QMM_INT8_ACT), written out instead of being scaled.
   x is f32 [M, K].  out (int32, device):
     Q8_0, Q4_0, Q5_0: [M][N][K/32]  isum of each 32-block (signed codes);
     Q4_K: [M][N][K/256][2]      (S_sc, S_m) of each super-block;
     Q6_K: [M][N][K/256]         S of each super-block.
   Bit-exact contract.  Errors as for qmm_matmul (no workspace). */
qmm_status qmm_block_sums(qmm_type wtype, const void* wq, const float* x, int64_t M, int64_t N, int64_t K,
                          int32_t* out, qmm_stream_t stream);

/* One item of qmm_matmul_batch: y [M, N] = x [M, K] . W^T (all device memory). */
typedef struct {
    const void* wq;   /* weight blocks, N * qmm_row_bytes(wtype, K) bytes, 16-byte aligned */
    const float* x;   /* activations [M, K] f32, 16-byte aligned                         */
    float* y;         /* output [M, N] f32, 4-byte aligned                                */
    int64_t M, N, K;
} qmm_matmul_desc;

#define QMM_BATCH_MAX_M 8        /* activation rows per item, at most          */
#define QMM_BATCH_MAX_MK 16384   /* M * K per item, at most                     */

/* Many independent small matmuls in one launch (per 256 items): the linears
   of a decode step (q, k, v, o, gate, up, down and the output head), which
   issued one by one are bound by launch latency rather than by their weight
   bytes.  Each item computes exactly what qmm_matmul(wtype, mode, ...) computes
   for it ("同一个 GGUF…" section 出处: int8_act quantizes each activation row
   to Q8_0, or to Q8K for Q4_K and Q6_K weights, and forms exact int32 block
   dots; f32_act multiplies f32 activations by the dequantized weights in f32),
   within the same bound.
   wtype: any weight type (QMM_Q8_0, QMM_Q4_0, QMM_Q5_0, QMM_Q4_K, QMM_Q6_K),
   one type and one form for the whole batch (qmm_matmul_batch_typed mixes
   types).  items: host array of `count` descriptors, read during the call
   (the launch carries a copy), so the call can be captured in a CUDA graph.
   Items with M = 0 or N = 0 are skipped.  Items may share x; their y must not
   overlap.  Needs no workspace.
   Errors: TYPE; SHAPE (negative sizes, K not a multiple of the block size,
   M > QMM_BATCH_MAX_M or M * K > QMM_BATCH_MAX_MK); NULL; ALIGN; CUDA.
   Nothing is launched when any item is invalid. */
qmm_status qmm_matmul_batch(qmm_type wtype, qmm_act_mode mode, const qmm_matmul_desc* items, int64_t count,
                            qmm_stream_t stream);

/* One item of qmm_matmul_batch_typed: a qmm_matmul_desc with its own weight type. */
typedef struct {
    qmm_type wtype;   /* QMM_Q8_0, QMM_Q4_0, QMM_Q5_0, QMM_Q4_K or QMM_Q6_K        */
    const void* wq;   /* weight blocks, N * qmm_row_bytes(wtype, K) bytes, 16-byte aligned */
    const float* x;   /* activations [M, K] f32, 16-byte aligned                         */
    float* y;         /* output [M, N] f32, 4-byte aligned                                */
    int64_t M, N, K;
} qmm_matmul_typed_desc;

/* qmm_matmul_batch for items of different weight types in one launch: a whole
   decode step of a mixed-type file, such as the Q4_K_M files the "GGUF 文件"
   page describes (Q5_0 and Q8_0 matrices where the row length is not a
   multiple of 256, Q4_K and Q6_K elsewhere).  Each item computes exactly what
   qmm_matmul(item.wtype, mode, ...) computes for it, within the same bound;
   mode is one form for the whole batch.  Same contract and errors as
   qmm_matmul_batch (TYPE also for an item's invalid wtype). */
qmm_status qmm_matmul_batch_typed(qmm_act_mode mode, const qmm_matmul_typed_desc* items, int64_t count,
                                  qmm_stream_t stream);

/* qmm_matmul for callers that cannot allocate device memory.
   (The pages have no counterpart: this is an addition of this library.)
   Some callers never call cudaMalloc themselves: a host engine that owns all
   device allocations and hands a plugin only finished input/output buffers,
   or a latency-critical loop that must not hit the allocator.  This call
   computes exactly what qmm_matmul computes, but when the shape needs a
   workspace it uses one array of QMM_STATIC_WORKSPACE_BYTES that the library
   keeps in device memory (every GPU that loads the library holds it until
   the process exits); it calls no cudaMalloc, cudaFree or allocating routine.
   - Shapes whose workspace (qmm_matmul_workspace) exceeds
     QMM_STATIC_WORKSPACE_BYTES are refused with QMM_ERR_WORKSPACE before
     anything is launched.
   - The first call on a device looks up the array's device address (with
     that device current); make that first call before any stream capture.
   - Every call shares the one array and it keeps the last call's contents:
     each call clears on `stream` whatever part must start at zero (the
     K-split arrival counters of the streaming and tcgen05 kernels), but
     calls that overlap on the GPU (other streams, other host threads) race
     on it.
   Other arguments and errors as qmm_matmul. */
#define QMM_STATIC_WORKSPACE_BYTES (8u << 20)
qmm_status qmm_matmul_static_workspace(qmm_type wtype, qmm_act_mode mode, const void* wq, const float* x, float* y,
                                       int64_t M, int64_t N, int64_t K, qmm_stream_t stream);

/* Failure-test hooks.  (The pages have no counterpart: these exist so that
   the library's failure paths can be exercised without faulting a GPU.)
   qmm_test_inject arms an injected failure, consumed by the next `count`
   calls that reach it; QMM_INJECT_OFF disarms every kind.
   - QMM_INJECT_LAUNCH_FAILURE: qmm_matmul / qmm_block_sums return
     QMM_ERR_CUDA at once, as if the launch had failed, without any CUDA call
     (the outputs are not touched).
   - QMM_INJECT_STALL: the next decode-kernel launch (qmm_dmma_kernel, the
     M <= 16 warp-MMA path) issues no weight stage from stage `arg` on in its
     first block, so that block's consumers wait in vain: their bounded wait
     gives up, the block drains the copies it did issue and exits, and
     qmm_last_device_error then reports QMM_ERR_TIMEOUT.  The call's output
     is undefined; later calls are unaffected.
   qmm_test_set_wait_limit sets the bounded waits' spin limit on the current
   device to 2^log2_clocks SM clocks (16..31; 0 restores the default 2^31,
   about one second), so that an injected stall ends in milliseconds.  It
   writes device memory synchronously.  Errors: SHAPE (argument out of
   range), TYPE (unknown kind), CUDA. */
typedef enum { QMM_INJECT_OFF = 0, QMM_INJECT_LAUNCH_FAILURE = 1, QMM_INJECT_STALL = 2 } qmm_inject_kind;
qmm_status qmm_test_inject(qmm_inject_kind kind, int count, int arg);
qmm_status qmm_test_set_wait_limit(int log2_clocks);

/* Reads and clears the current device's error word (synchronizes that
   device).  QMM_ERR_TIMEOUT if a device-side wait of an earlier launch gave
   up after its bounded spin (its outputs are then undefined), QMM_OK
   otherwise, QMM_ERR_CUDA if the read itself failed. */
qmm_status qmm_last_device_error(void);

/* Static English text for a status code. */
const char* qmm_status_string(qmm_status s);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
