/*
 * qgemv.h - C ABI of the GB300 block-quantized matrix-vector product.
 *
 * y = W . x for W stored as byte-exact GGUF blocks (Q8_0, Q4_0, Q4_1, Q5_0,
 * Q2_K, Q3_K, Q4_K, Q5_K, Q6_K), x quantized once per call to the activation
 * blocks paired with the weight type (Q8_0, Q8_1 or Q8_K), exact int32 sums
 * inside every block and float only for the block scales.
 *
 * Citations name the reference pages by title and section:
 *   [rml]      "Quantization" (rayaq.ca/rml)
 *   [sipllm]   "Quantization" (sipllm docs)
 *   [lesson21] "Building Q8_0 and Q4_0 Like ggml" (codeloopback)
 *   [candle]   "量化格式" (quantized formats, candle)
 *
 * Conventions for every call below
 *   - Pointers named W, x, xq, y, out, isums, workspace are DEVICE pointers
 *     (cudaMalloc / torch CUDA tensors) owned by the caller. The library
 *     allocates nothing and keeps no reference after the call returns.
 *   - Every device pointer must be 16-byte aligned (QG_ERR_ALIGN otherwise).
 *   - W is [n_out][n_in] row-major: row o starts at byte o * qtype_nbytes(type,
 *     n_in), rows and blocks follow each other with no padding ([lesson21]
 *     Example 9). x is f32 [n_vec][n_in], y is f32 [n_vec][n_out]:
 *     y[v * n_out + o] = sum_i W[o, i] * x[v, i].
 *   - n_in must be a whole number of blocks (QG_ERR_SHAPE otherwise;
 *     [lesson21] Example 15 rejects a row of 100). 1 <= n_vec <= QG_MAX_NVEC.
 *   - All work is enqueued on `stream` (NULL = the legacy default stream);
 *     no call synchronizes. Argument errors are returned before anything is
 *     enqueued. A CUDA launch error is returned as QG_ERR_CUDA.
 *   - Kernels launched by these calls use programmatic dependent launch: a
 *     product may begin streaming W while the kernel enqueued before it on
 *     the same stream is still finishing. quantize_rows provides for this
 *     (its last kernel starts only after the weights are written), so a
 *     product may directly follow the quantize_rows call that writes its W.
 *     A kernel of the caller's own that writes W must not be the last work
 *     enqueued before the product on that stream; any other stream-ordered
 *     work in between (another library call, a copy, an ordinary kernel)
 *     restores full ordering. x, y and the workspace follow ordinary stream
 *     order.
 *   - Inputs with NaN or inf are outside the contract of the product; the
 *     quantizers map NaN to code 0 and let an infinite scale through, as
 *     [candle] "一些边界值" (special values) shows.
 */
#ifndef GB300_QGEMV_H
#define GB300_QGEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared opaquely so this header does not
 * need the CUDA headers. */
typedef struct CUstream_st *qg_stream_t;

/* ggml element-type ids, the numbers a GGUF tensor record stores
 * ([rml] The type table; [sipllm] On-disk block geometry). */
enum qg_type {
    QG_F32 = 0,
    QG_F16 = 1,
    QG_Q4_0 = 2,   /* 32 elements, 18 bytes: f16 d, 16 bytes of nibbles      */
    QG_Q4_1 = 3,   /* 32 elements, 20 bytes: f16 d, f16 m, 16 bytes of nibbles */
    QG_Q5_0 = 6,   /* 32 elements, 22 bytes: f16 d, u32 qh (fifth bits), 16 bytes of nibbles */
    QG_Q8_0 = 8,   /* 32 elements, 34 bytes: f16 d, 32 int8                  */
    QG_Q8_1 = 9,   /* 32 elements, 36 bytes: f16 d, f16 s, 32 int8 (activations only) */
    QG_Q2_K = 10,  /* 256 elements, 84 bytes: 16 B scales|mins, 64 B qs, f16 d, f16 dmin */
    QG_Q3_K = 11,  /* 256 elements, 110 bytes: 32 B hmask, 64 B qs, 12 B scales, f16 d */
    QG_Q4_K = 12,  /* 256 elements, 144 bytes: f16 d, f16 dmin, 12 B scales, 128 B qs */
    QG_Q5_K = 13,  /* 256 elements, 176 bytes: f16 d, f16 dmin, 12 B scales, 32 B qh, 128 B qs */
    QG_Q6_K = 14,  /* 256 elements, 210 bytes: 128 B ql, 64 B qh, 16 int8 scales, f16 d */
    QG_Q8_K = 15   /* 256 elements, 292 bytes: f32 d, 256 int8, 16 int16 bsums (activations only) */
};

enum qg_status {
    QG_OK = 0,
    QG_ERR_TYPE = -1,      /* unknown or unsupported type id                  */
    QG_ERR_SHAPE = -2,     /* n not whole blocks, a size out of range         */
    QG_ERR_ALIGN = -3,     /* a device pointer not 16-byte aligned            */
    QG_ERR_NULL = -4,      /* a required pointer is NULL                      */
    QG_ERR_PAIR = -5,      /* the weight type has no activation pairing       */
    QG_ERR_CUDA = -6,      /* a CUDA call failed (see qg_last_cuda_error)     */
    QG_ERR_WORKSPACE = -7  /* workspace NULL or smaller than required         */
};

#define QG_MAX_NVEC 8

/* ---- Type table ---------------------------------------------------------- */

/* Bytes taken by n elements of `type`: n / block_elems * block_bytes
 * ([rml] The type table; [sipllm] type_nbytes). Returns -1 for an unknown
 * type or when n is negative or not a whole number of blocks. */
int64_t qtype_nbytes(int type, int64_t n);

/* Block geometry of `type` ([candle] GgmlDType table). Writes the elements
 * and bytes of one block; returns QG_OK or QG_ERR_TYPE (outputs untouched).
 * elems/bytes are host pointers and may not be NULL. */
int qtype_block(int type, int *elems, int *bytes);

/* Activation type paired with a weight type ([rml] DotActivationType;
 * [candle] VecDotType table): Q4_0, Q5_0 and Q8_0 -> QG_Q8_0, Q4_1 ->
 * QG_Q8_1, the K-quants Q2_K..Q6_K -> QG_Q8_K. Returns QG_ERR_PAIR for any
 * other type. */
int qtype_act_type(int weight_type);

/* Static text for a status code. Never NULL. */
const char *qg_status_string(int status);

/* Text of the last CUDA error seen by this library on the calling thread
 * ("" if none). */
const char *qg_last_cuda_error(void);

/* ---- Quantizers ---------------------------------------------------------- */

/* Activation quantization, once per call ([rml] Quantization; [lesson21]
 * Example 2; [candle] BlockQ8_0::from_float):
 *   act_type QG_Q8_0: per 32 elements amax = max |x|, d = amax / 127 (f32),
 *     id = 1/d (0 if d == 0), stored d = f16(d), code = roundf(x * id)
 *     (halves away from zero, codes from the unrounded id).
 *   act_type QG_Q8_1: the Q8_0 rule, plus s = f16(sum of the codes * d)
 *     computed in f32 from the unrounded d, a NaN s (only a block holding
 *     inf gives one) stored as 0x7E00 (the pages pair Q8_1 with Q4_1 but
 *     print neither its layout nor this rule: the library's reading).
 *   act_type QG_Q8_K: the same rule per 256 elements with d stored as f32,
 *     codes clamped to [-127, 127], and bsums[k] = sum of codes 16k..16k+15
 *     ([candle] block table; the pages do not print the rule, this is the
 *     library's stated reading).
 * x: f32 [n_vec][n_in] (device). xq: n_vec * qtype_nbytes(act_type, n_in)
 * bytes of byte-exact GGUF blocks (device). n_vec may be any positive count
 * here. */
int quantize_act(int act_type, const float *x, void *xq, int64_t n_in, int64_t n_vec,
                 qg_stream_t stream);

/* Weight quantization with ggml's reference rules, the bytes llama.cpp
 * writes ([lesson21] Examples 2, 5, 7, 8 and 14):
 *   QG_Q8_0: as quantize_act(QG_Q8_0).
 *   QG_Q4_0: per 32 elements the first element of strictly largest |x| gives
 *     max, d = max / -8, id = 1/d (0 if d == 0), code = min(15, (int)(x*id +
 *     8.5f)) with the multiply and add rounded separately; byte j holds
 *     element j in its low nibble and element j+16 in its high nibble.
 *   QG_Q4_1: per 32 elements min and max, d = (max - min) / 15, id = 1/d (0
 *     if d == 0), stored f16(d) and f16(min), code = min(15, (int)((x - min)
 *     * id + 0.5f)) with each step rounded in f32 from the unrounded min;
 *     nibbles as Q4_0.
 *   QG_Q5_0: Q4_0's signed max, d = max / -16, code = min(31, (int)(x * id +
 *     16.5f)); the low 4 bits in nibbles as Q4_0, bit 4 of code j in bit j of
 *     the little-endian 32-bit word qh.
 *   (int) is the cast of the lesson's Java code: truncation toward zero, 0
 *   for NaN, the int range's end beyond it; a code below 0 (only from -inf,
 *   when 1/d overflows for a subnormal max) keeps its low bits, 0.
 * x: f32 [n_rows][n_in]; out: n_rows * qtype_nbytes(type, n_in) bytes.
 * Enqueues the quantizer and then one empty kernel launched without
 * programmatic dependent launch, so that a product enqueued next on the
 * stream, which starts streaming W early, sees the finished weights. */
int quantize_rows(int type, const float *x, void *out, int64_t n_rows, int64_t n_in,
                  qg_stream_t stream);

/* ---- Dequantization ------------------------------------------------------ */

/* Every element of n_rows rows to f32 ([sipllm] Per-format dequant; [candle]
 * block table; [rml] Unpacking the packed fields):
 *   Q8_0, Q8_1: q * d     Q4_0: (code - 8) * d     Q5_0: (code - 16) * d
 *   Q4_1: code * d + m (the product is exact; the sum rounds once)
 *   Q4_K: (d * sc_j) * q - dmin * m_j, j = e / 32, 6-bit sc/m unpacked as in
 *         [rml]'s element-200 trace
 *   Q6_K: (d * sc_j) * (q - 32), j = e / 16, q = 4 low bits from ql and 2
 *         high bits from qh (element mapping: the library's stated reading)
 *   Q5_K: as Q4_K with q = nibble | (bit j of qh[e % 32]) << 4
 *   Q2_K: (d * sc_j) * q - dmin * m_j, j = e / 16, sc/m the low/high nibble
 *         of scales[j], q = bits 2k..2k+1 of qs[32n + 16h + l] for
 *         e = 128n + 32k + 16h + l
 *   Q3_K: (d * (sc_j - 32)) * (q - 4 * (1 - hbit)), j = e / 16, q as Q2_K,
 *         hbit = bit 4n + k of hmask[16h + l], sc_j the 6-bit field whose
 *         low 4 bits are nibble j / 8 of byte j % 8 and high 2 bits are bits
 *         2(j / 4) of byte 8 + j % 4
 *   (the Q2_K, Q3_K and Q5_K layouts are ggml's, which the pages do not
 *   print: the library's stated reading)
 *   Q8_K: q * d
 * Every product is exact in f32, so results are unique (only the
 * subtraction of Q2_K, Q4_K and Q5_K and the addition of Q4_1 round, to
 * nearest even). W: n_rows * qtype_nbytes(type, n_in)
 * bytes; out: f32 [n_rows][n_in]. */
int dequantize_rows(int type, const void *W, float *out, int64_t n_rows, int64_t n_in,
                    qg_stream_t stream);

/* ---- Matrix-vector product ----------------------------------------------- */

/* Bytes of workspace qgemv needs: the quantized activations,
 * n_vec * qtype_nbytes(qtype_act_type(type), n_in). 0 on a bad argument. */
size_t qgemv_workspace_bytes(int type, int64_t n_in, int64_t n_vec);

/* y = W . x ([sipllm] The fused matmul; [rml] Quantized dot products;
 * [lesson21] Examples 10-11): quantizes x once into `workspace` with
 * quantize_act's rule for the paired activation type, then for every row
 * and block forms the exact int32 block sum and adds
 *   Q8_0, Q4_0, Q5_0, Q3_K, Q6_K: S * (d_w * d_x)
 *   Q4_1:                         S * (d_w * d_x) + m_w * s_x
 *   Q2_K, Q4_K, Q5_K:             d_x * (d_w * S_q - dmin_w * S_m)
 * in f32. The f32 order of these few float operations is not fixed by the
 * pages; results agree with an f64 accumulation to about 1e-5 relative.
 * For the K-quant weight types (Q2_K .. Q6_K) with n_vec >= 3 the sums are formed on the tensor cores
 * (mma.sync, f16 operands that hold the integer codes exactly, f32
 * accumulation per sub-block, which is exact) and the sub-block scales are
 * applied in f32 per sub-block -- the same tolerance holds. So are those of
 * the 32-element types (eight blocks at a time, n_in a multiple of 256) when
 * n_out * n_in * (n_vec - 3) >= 40 * 2^20, the size from which that kernel
 * measured faster; the block's float step is then the one above. The vector
 * count from which this path is taken can be changed with the environment
 * variable QG_MMA_MIN_NVEC, the size with QG_MMA_GROUP_MELEM (in 2^20
 * elements; both read once per process).
 * workspace: device buffer of at least qgemv_workspace_bytes(type, n_in,
 * n_vec) bytes (workspace_bytes gives its size). Limits: n_out <=
 * 2^31 - 1; n_vec * n_in must be small enough for the activations of one
 * call to fit in one SM's shared memory next to two weight stages
 * (QG_ERR_SHAPE otherwise; every shape with n_vec * n_in <= 65536 fits). */
int qgemv(int type, const void *W, const float *x, float *y, int64_t n_out, int64_t n_in,
          int64_t n_vec, void *workspace, size_t workspace_bytes, qg_stream_t stream);

/* The product on activations already quantized by quantize_act (byte-exact
 * blocks of the paired type, [rml] VecDot takes quantized activations).
 * Same limits and float step as qgemv. */
int qgemv_xq(int type, const void *W, const void *xq, float *y, int64_t n_out, int64_t n_in,
             int64_t n_vec, qg_stream_t stream);

/* Diagnostic: the exact per-block int32 sums that qgemv_xq forms, written to
 * isums[((v * n_out + o) * nb + b) * k + t], nb = n_in / block elements,
 * k = 2 for Q2_K, Q4_K and Q5_K (t = 0: S_q = sum_j sc_j sum_{i in j}
 * q_i a_i, t = 1: S_m = sum_j m_j (sum of a over sub-block j)) and k = 1
 * otherwise (Q3_K: sum_j sc_j sum_{i in j} q_i a_i with signed q; Q8_0:
 * sum qw qx; Q4_0: sum (code - 8) qx; Q5_0: sum (code - 16) qx; Q4_1:
 * sum code qx, its min term m_w s_x being float; Q6_K: sum_j sc_j
 * sum_{i in j} (q_i - 32) a_i) ([rml] Quantized dot products, Kernels and
 * references). Runs the __dp4a kernel that qgemv_xq runs for fewer than 3
 * vectors (the tensor-core kernel accumulates the same exact sums, some
 * scaled by 2^-24, but does not write them out). */
int qgemv_block_isums(int type, const void *W, const void *xq, int32_t *isums, int64_t n_out,
                      int64_t n_in, int64_t n_vec, qg_stream_t stream);

/* The product without a workspace, for callers that cannot allocate device
 * memory where they run it: a plugin whose host framework owns every device
 * buffer and passes it none, a decode loop that must not call cudaMalloc or
 * cudaFree (they can synchronize the whole device), or code recorded by CUDA
 * stream capture, where allocation is not allowed. The reference pages have
 * no counterpart; this is a property of this library's interface.
 *
 * Same arguments, result and limits as qgemv without workspace and
 * workspace_bytes. The quantized activations go to a fixed array of 256 KiB
 * (262144 bytes) inside the library's device memory, which every GPU that
 * loads the library holds until the process exits. Calls whose activations
 * need more (qgemv_workspace_bytes(type, n_in, n_vec) > 262144) return
 * QG_ERR_WORKSPACE and enqueue nothing. The call allocates nothing.
 *
 * Where qgemv would quantize x inside the product's own launch (small x,
 * see QG_FUSED_QUANT_KIB) this call does the same and does not touch the
 * array.
 *
 * All calls on a device share that array. Calls ordered on one stream are
 * safe. Calls that may run at the same time on the GPU (different streams,
 * or different host threads without ordering between them) race on it and
 * give wrong results. The array keeps the previous call's contents; every
 * byte a call reads is written earlier in the same call, so nothing needs
 * clearing.
 *
 * The first call on each device that uses the array, with that device
 * current, looks up the array's device address (cudaGetSymbolAddress) and
 * keeps it for the life of the process. Make that first call before any
 * stream capture that includes this function. A device reset
 * (cudaDeviceReset, or a reset of the primary context) frees the array and
 * leaves the kept address stale: do not call this function after one. */
int qgemv_noalloc(int type, const void *W, const float *x, float *y, int64_t n_out, int64_t n_in,
                  int64_t n_vec, qg_stream_t stream);

/* ---- Batches of independent products -------------------------------------- */

#define QG_MAX_BATCH 256

/* One matrix of a batched call (host struct; device pointers inside). */
typedef struct {
    const void *W;   /* weight blocks [n_out][n_in], 16-byte aligned */
    const float *x;  /* f32 activations [n_vec][n_in], 16-byte aligned */
    float *y;        /* f32 output [n_vec][n_out], 16-byte aligned */
    int64_t n_out;   /* rows of this matrix (0 allowed) */
} qg_gemv_mat;

/* Workspace bytes qgemv_batched needs for n_mats matrices: 16 when the
 * activations are small enough to be quantized inside the product (4 *
 * n_in * n_vec <= QG_FUSED_QUANT_KIB, 16 KiB by default, and not a
 * product that may take the tensor cores, n_vec >= 3), else the quantized
 * activations of every matrix,
 * n_mats * qgemv_workspace_bytes(type, n_in, n_vec). 0 on a bad argument. */
size_t qgemv_batched_workspace_bytes(int type, int64_t n_in, int64_t n_vec, int n_mats);

/* y_i = W_i . x_i for n_mats independent matrices of one type, row length
 * n_in and vector count n_vec, in one launch ([sipllm] The fused matmul,
 * applied to several matrices; [rml] Quantized dot products; [candle]
 * vec_dot_4 reuses one activation load across rows). Same arithmetic,
 * result and limits as qgemv for each matrix. The matrices must be
 * independent: no y_i may alias any W_j or x_j of the same call. The rows of
 * all matrices are spread over the GPU's SMs as one stream, so a batch of
 * small matrices runs at the bandwidth of one large one. mats is a host
 * array read during the call (1 <= n_mats <= QG_MAX_BATCH). */
int qgemv_batched(int type, const qg_gemv_mat *mats, int n_mats, int64_t n_in, int64_t n_vec, void *workspace,
                  size_t workspace_bytes, qg_stream_t stream);

/* ---- Prefill: many tokens ------------------------------------------------ */

/* Workspace bytes qgemm needs: the f16 copy of W (2 * n_out * n_in) and of x
 * (2 * n_tok * n_in), each rounded up to 256 bytes. 0 on a bad argument.
 * When qgemm expands Q4_K blocks inside the GEMM, the W part holds the
 * f32 partial products of a k split instead (never more than it has room
 * for: the split is chosen to fit). */
size_t qgemm_workspace_bytes(int type, int64_t n_out, int64_t n_in, int64_t n_tok);

/* The product for many tokens at once (prefill): y[t][o] = sum_i
 * W[o][i] * x[t][i] for t < n_tok, with W of any weight type above
 * ([sipllm] The fused matmul: matmul_quant dequantizes a row to f32 and dots
 * it with f32 x; here the whole product is one dense GEMM). Steps, all on
 * `stream`: dequantize W to f16 (round to nearest even) into the workspace,
 * round x to f16 into the workspace, then a tcgen05 tensor-core GEMM with
 * f32 accumulation. For Q4_K weights and up to 2048 tokens for 4096 rows (by
 * default; see the knob QG_FUSED_GEMM of qg_tune) W is instead dequantized inside the
 * GEMM (raw blocks are loaded into shared memory and expanded to the same
 * f16 values in tensor memory, where the mma reads them; no f16 copy of W is
 * written), with the same result bit for bit; when its 128 x 128 tiles are
 * fewer than the SMs it also splits each tile's k-range into parts (knob
 * QG_GEMM_KSPLIT), whose f32 partial products go to the workspace and are
 * added to y in part order by one more launch: deterministic, and within
 * n_in 2^-23 sum_i |W[o][i] x[t][i]| of the unsplit result. The result differs from the f32 product by the f16
 * rounding of each weight and activation (at most 2^-11 relative each) and
 * the f32 accumulation: |y - y_exact| <= (2^-10 + n_in 2^-24) sum_i
 * |W[o][i] x[t][i]| (values beyond f16's range, 65504, become inf).
 * Unlike qgemv, x is not quantized to Q8 blocks.
 * W: blocks [n_out][n_in] (device, 16-byte aligned); x: f32 [n_tok][n_in];
 * y: f32 [n_tok][n_out]; workspace: qgemm_workspace_bytes, 16-byte aligned.
 * n_in must be a multiple of the block size; 0 <= n_out, n_tok < 2^31.
 * n_in == 0 writes zeros. Returns QG_OK or an error before anything is
 * enqueued (QG_ERR_TYPE, QG_ERR_PAIR, QG_ERR_SHAPE, QG_ERR_NULL,
 * QG_ERR_ALIGN, QG_ERR_WORKSPACE), or QG_ERR_CUDA if a launch fails. */
int qgemm(int type, const void *W, const float *x, float *y, int64_t n_out, int64_t n_in, int64_t n_tok,
          void *workspace, size_t workspace_bytes, qg_stream_t stream);

/* The dense GEMM step of qgemm on its own, for callers that keep f16
 * operands (for instance weights dequantized once and reused across prefill
 * calls): y[t][o] = sum_k A[o][k] * B[t][k] with A f16 [n_out][K] and B f16
 * [n_tok][K] (row-major, device, 16-byte aligned; K a multiple of 8, 0 <= K,
 * n_out, n_tok < 2^31), y f32 [n_tok][n_out], f32 accumulation on the
 * tcgen05 tensor cores. qgemm's workspace holds its A (offset 0) and B
 * (offset 2 * n_out * K rounded up to 256 bytes) in this form. K == 0
 * writes zeros. Returns QG_OK, QG_ERR_SHAPE, QG_ERR_NULL, QG_ERR_ALIGN or
 * QG_ERR_CUDA. */
int qgemm_f16(const void *A, const void *B, float *y, int64_t n_out, int64_t n_tok, int64_t K, qg_stream_t stream);

/* ---- Introspection --------------------------------------------------------- */

/* Which kernel and launch plan a product over n_mats matrices with
 * total_rows rows in all (row length n_in, n_vec vectors) would use on the
 * current device, as one line of text for logs and benchmarks, e.g.
 * "gemv_mma_kernel<Q4_K,regs,8w> grid=152 stages=5 kb=16 smem=226240
 * partials=10" (mode, consumer warps, CTAs, ring stages, blocks per stage
 * row, shared memory, partial-output buffers). The string
 * belongs to the library (per host thread, overwritten by the next call).
 * Returns "" on a bad argument or when the shape has no plan; "cuda: ..." on
 * a CUDA error. Launches nothing. */
const char *qgemv_kernel_info(int type, int64_t total_rows, int64_t n_in, int64_t n_vec, int n_mats);

/* The same for qgemm on these sizes: the GEMM kernel with its token-tile
 * width, CTAs, k-split parts and the launches one call makes, e.g.
 * "gemm_q4k_tmem_kernel<256> grid=128 ksplit=2 launches=3" (x to f16, the
 * fused GEMM, the sum of the k-split parts) or "gemm_f16_tc_kernel<128>
 * grid=152 ksplit=1 launches=3" (W to f16, x to f16, the GEMM). Same
 * ownership and errors as qgemv_kernel_info; launches nothing. */
const char *qgemm_kernel_info(int type, int64_t n_out, int64_t n_in, int64_t n_tok);

/* Sets a tuning knob for the rest of the process (the pages have no
 * counterpart; the knobs choose between kernels that compute the same
 * product). name is one of the environment variables the library reads once
 * at first use: QG_CTAS_PER_SM, QG_RING_KIB, QG_MMA_MIN_NVEC (vectors from
 * which the K-quant types use the tensor cores), QG_MMA_GROUP_MELEM (the
 * 32-element types do from n_out * n_in * (n_vec - 3) >= this many 2^20
 * elements; 0: from QG_MMA_MIN_NVEC vectors), QG_MMA_PANEL (0 automatic, 1 a
 * shared-memory activation panel, 8 the int8 panel), QG_MMA_KB (longest
 * chunk of blocks a panel-mode stage takes; 0 no limit), QG_FUSED_QUANT_KIB (f32 x of at most this many KiB is quantized
 * inside the GEMV), QG_FUSED_MAX_MIB (... for a single matrix of at most this
 * many MiB of blocks; default: no limit), QG_TC (the tcgen05 Q4_K kernel for three or
 * more vectors, rows of 2048 or 4096 elements: 0 never, the default; 1
 * whenever it fits), QG_FUSED_GEMM (qgemm on Q4_K weights: 0 writes the f16
 * copy of W to the workspace first; 1 dequantizes inside the GEMM, into
 * tensor memory, instead; 2, the default, does so while that GEMM has at
 * most two 256-token tiles per SM: up to 2048 tokens for 4096 rows),
 * QG_GEMM_KSPLIT (that fused GEMM, when its 128 x 128 tiles are fewer than the
 * SMs, splits each tile's k-blocks into at most this many parts, 1 to 8, the
 * default 8, at least 4 k-blocks a part; the parts' f32 sums are added in part
 * order, so results stay deterministic). value is clamped to the knob's range; the old
 * value goes to *previous when that is not NULL. Returns QG_OK, QG_ERR_NULL
 * or QG_ERR_TYPE (unknown name). Host-only; affects launches planned after
 * it returns. */
int qg_tune(const char *name, int value, int *previous);

/* ---- Device-side status -------------------------------------------------- */

/* Every wait inside the kernels is bounded (about one second). A wait that
 * runs out records a nonzero code in a device word and the kernel returns
 * early. This call synchronizes the current device, writes the word to
 * *code (host pointer), clears it and returns QG_OK (or QG_ERR_CUDA). */
int qg_device_error(int32_t *code);

/* Self-test of that mechanism (the pages have no counterpart): enqueues on
 * `stream` one single-thread kernel that waits, with the same bounded wait
 * the product kernels use, on an mbarrier that nothing completes. After
 * about one second the wait gives up, the kernel records the code a
 * consumer wait records (2) and returns; no fault, no trap, and the context
 * stays usable. Read the code with qg_device_error. Returns QG_OK or
 * QG_ERR_CUDA. */
int qg_selftest_bounded_wait(qg_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_QGEMV_H */
