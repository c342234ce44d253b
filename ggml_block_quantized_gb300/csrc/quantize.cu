// quantize.cu - activation and weight quantizers (byte-exact GGUF blocks).
//
// Q8_0 ("Building Q8_0 and Q4_0 Like ggml", Example 2; "量化格式" (candle),
// BlockQ8_0::from_float): per 32 values amax = max |x| (NaN ignored),
// d = amax / 127 (f32), id = 1/d or 0, stored d = f16(d), code =
// roundf(x * id) with halves away from zero, from the unrounded id.
// Q8_K: the same rule per 256 values with d kept in f32, codes clamped to
// [-127, 127] and bsums[k] = sum of codes 16k..16k+15 (the library's reading;
// the pages give only the block layout and the role of bsums).
// Q4_0 ("Building Q8_0 and Q4_0 Like ggml", Example 5; "Quantization" (rml),
// A worked example: Q4_0): the first value of strictly largest magnitude is
// max, d = max / -8, id = 1/d or 0, code = min(15, (int)(x*id + 8.5f)) with
// the multiply and the add rounded separately; byte j = code j | code j+16 << 4.
// Q4_1 ("Building Q8_0 and Q4_0 Like ggml", Example 7): min and max of the
// block, d = (max - min) / 15, id = 1/d or 0, stored f16(d) and f16(min),
// code = min(15, (int)((x - min) * id + 0.5f)) with each step rounded in f32
// from the unrounded min; nibbles as Q4_0.
// Q5_0 (same page, Example 8): Q4_0's signed max, d = max / -16, code =
// min(31, (int)(x * id + 16.5f)); low 4 bits in nibbles as Q4_0, bit 4 of
// code j in bit j of the little-endian 32-bit word qh.
// Q8_1 (activations of Q4_1; the candle VecDotType table pairs them): the
// Q8_0 rule plus s = f16(sum of codes * d) from the f32 d, a NaN s (only
// from a block holding inf) stored as 0x7E00 (the library's reading: the
// pages give neither the layout nor the rule of s).
//
// One warp per block. The only float operations are the IEEE-rounded
// division, reciprocal, multiply and add written below (the library is built
// without fast-math, so '/' is correctly rounded), roundf and the f16
// conversion, so the bytes equal the scalar definition's.
#include "qg_common.cuh"

namespace qg {

// Float to int as the lesson's Java code casts it: truncation toward zero,
// 0 for NaN, the int range's end beyond it (a NaN element, or a scale so
// small that 1/d overflows, reaches those cases). Written out rather than
// left to the conversion instruction's own NaN and overflow rules.
__device__ __forceinline__ int java_f2i(float t) {
    if (t != t) return 0;
    if (t >= 2147483648.0f) return 2147483647;
    if (t <= -2147483648.0f) return -2147483647 - 1;
    return static_cast<int>(t);
}

// Two 4-bit codes into one byte: the low 4 bits of each (a code below 0
// comes only from -inf and keeps its low bits, 0).
__device__ __forceinline__ uint8_t pack_nibbles(int lo, int hi) {
    return static_cast<uint8_t>((static_cast<uint32_t>(lo) & 0xFu) | ((static_cast<uint32_t>(hi) & 0xFu) << 4));
}

__device__ __forceinline__ float warp_max_abs(float a) {
    // fmaxf ignores NaN, as the scalar rule's comparison does
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
    return a;
}

// ---------------------------------------------------------------- Q8_0
// One 32-value block, lane i owns value i. ob: 34 bytes.
__device__ __forceinline__ void q8_0_block(const float *xb, uint8_t *ob, int lane) {
    const float v = __ldg(xb + lane);
    const float amax = warp_max_abs(fabsf(v));
    const float d = amax / 127.0f;
    const float id = d != 0.0f ? 1.0f / d : 0.0f;
    const int q = code_from_rounded(roundf(__fmul_rn(v, id)), -128, 127);
    ob[2 + lane] = static_cast<uint8_t>(static_cast<int8_t>(q));
    // the f16 scale as one 16-bit store (blocks start 2-byte aligned)
    if (lane == 0) *reinterpret_cast<unsigned short *>(ob) = __half_as_ushort(__float2half_rn(d));
}

// ---------------------------------------------------------------- Q8_K
// One 256-value block, lane i owns values 8i..8i+7. ob: 292 bytes
// (f32 d | 256 int8 | 16 int16 bsums).
__device__ __forceinline__ void q8_k_block(const float *xb, uint8_t *ob, int lane) {
    const float4 *src = reinterpret_cast<const float4 *>(xb + 8 * lane);
    const float4 u = __ldg(src), w = __ldg(src + 1);
    const float v[8] = {u.x, u.y, u.z, u.w, w.x, w.y, w.z, w.w};
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
    const float amax = warp_max_abs(a);
    const float d = amax / 127.0f;
    const float id = d != 0.0f ? 1.0f / d : 0.0f;
    uint32_t packed[2] = {0u, 0u};
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int q = code_from_rounded(roundf(__fmul_rn(v[i], id)), -127, 127);
        sum += q;
        packed[i >> 2] |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * (i & 3));
    }
    // bsums[k] covers lanes 2k and 2k+1
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    uint32_t *qs = reinterpret_cast<uint32_t *>(ob + 4 + 8 * lane);
    qs[0] = packed[0];
    qs[1] = packed[1];
    if ((lane & 1) == 0) reinterpret_cast<int16_t *>(ob + 260)[lane >> 1] = static_cast<int16_t>(sum);
    if (lane == 0) *reinterpret_cast<float *>(ob) = d;
}

// ---------------------------------------------------------------- Q4_0
// One 32-value block, lane i owns value i. ob: 18 bytes.
__device__ __forceinline__ void q4_0_block(const float *xb, uint8_t *ob, int lane) {
    const float v = __ldg(xb + lane);
    // First index of strictly largest |x| in scan order: reduce (|x|, index)
    // keeping the larger magnitude and, on a tie, the smaller index. NaN
    // never wins (the scalar test amax < |x| is false for NaN).
    float best = (v != v) ? -1.0f : fabsf(v);
    int idx = lane;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        const float ob_ = __shfl_xor_sync(0xffffffffu, best, m);
        const int oi = __shfl_xor_sync(0xffffffffu, idx, m);
        if (ob_ > best || (ob_ == best && oi < idx)) {
            best = ob_;
            idx = oi;
        }
    }
    const float vmax = __shfl_sync(0xffffffffu, v, idx);
    // an all-zero block keeps max = +0 (no element replaces it)
    const float mx = best > 0.0f ? vmax : 0.0f;
    const float d = mx / -8.0f;
    const float id = d != 0.0f ? 1.0f / d : 0.0f;
    const float t = __fadd_rn(__fmul_rn(v, id), 8.5f);
    int code = java_f2i(t);
    code = code < 15 ? code : 15;
    const int hi = __shfl_down_sync(0xffffffffu, code, 16);
    if (lane < 16) ob[2 + lane] = pack_nibbles(code, hi);
    if (lane == 0) *reinterpret_cast<unsigned short *>(ob) = __half_as_ushort(__float2half_rn(d));
}

// ---------------------------------------------------------------- Q8_1
// One 32-value block, lane i owns value i. ob: 36 bytes (f16 d | f16 s | 32 int8).
__device__ __forceinline__ void q8_1_block(const float *xb, uint8_t *ob, int lane) {
    const float v = __ldg(xb + lane);
    const float amax = warp_max_abs(fabsf(v));
    const float d = amax / 127.0f;
    const float id = d != 0.0f ? 1.0f / d : 0.0f;
    const int q = code_from_rounded(roundf(__fmul_rn(v, id)), -128, 127);
    ob[4 + lane] = static_cast<uint8_t>(static_cast<int8_t>(q));
    int sum = q;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, m);
    if (lane == 0) {
        const uint32_t dbits = __half_as_ushort(__float2half_rn(d));
        // a block holding inf has d = inf and s = 0 * inf: one fixed quiet NaN
        const float sv = __fmul_rn(static_cast<float>(sum), d);
        const uint32_t sbits = sv != sv ? 0x7E00u : __half_as_ushort(__float2half_rn(sv));
        *reinterpret_cast<uint32_t *>(ob) = dbits | (sbits << 16);  // blocks start 4-byte aligned
    }
}

// ---------------------------------------------------------------- Q4_1
// One 32-value block, lane i owns value i. ob: 20 bytes.
__device__ __forceinline__ void q4_1_block(const float *xb, uint8_t *ob, int lane) {
    const float v = __ldg(xb + lane);
    // min and max over the block; fminf/fmaxf skip a NaN, as the scalar
    // comparisons (false for NaN) do
    float mn = v, mx = v;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, m));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
    }
    if (mn != mn) { mn = 3.4028234663852886e38f; mx = -3.4028234663852886e38f; }  // all NaN: untouched start values
    const float d = __fsub_rn(mx, mn) / 15.0f;
    const float id = d != 0.0f ? 1.0f / d : 0.0f;
    const float t = __fadd_rn(__fmul_rn(__fsub_rn(v, mn), id), 0.5f);
    int code = java_f2i(t);
    code = code < 15 ? code : 15;
    const int hi = __shfl_down_sync(0xffffffffu, code, 16);
    if (lane < 16) ob[4 + lane] = pack_nibbles(code, hi);
    if (lane == 0) {
        const uint32_t dbits = __half_as_ushort(__float2half_rn(d));
        const uint32_t mbits = __half_as_ushort(__float2half_rn(mn));
        *reinterpret_cast<uint32_t *>(ob) = dbits | (mbits << 16);  // blocks start 4-byte aligned
    }
}

// First index of strictly largest |x| in scan order, its value (0 for an
// all-zero block), as Q4_0 and Q5_0 take it.
__device__ __forceinline__ float signed_max(float v, int lane) {
    float best = (v != v) ? -1.0f : fabsf(v);
    int idx = lane;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        const float ob_ = __shfl_xor_sync(0xffffffffu, best, m);
        const int oi = __shfl_xor_sync(0xffffffffu, idx, m);
        if (ob_ > best || (ob_ == best && oi < idx)) {
            best = ob_;
            idx = oi;
        }
    }
    const float vmax = __shfl_sync(0xffffffffu, v, idx);
    return best > 0.0f ? vmax : 0.0f;
}

// ---------------------------------------------------------------- Q5_0
// One 32-value block, lane i owns value i. ob: 22 bytes (2-byte aligned).
__device__ __forceinline__ void q5_0_block(const float *xb, uint8_t *ob, int lane) {
    const float v = __ldg(xb + lane);
    const float d = signed_max(v, lane) / -16.0f;
    const float id = d != 0.0f ? 1.0f / d : 0.0f;
    const float t = __fadd_rn(__fmul_rn(v, id), 16.5f);
    int code = java_f2i(t);
    code = code < 31 ? code : 31;
    const uint32_t qh = __ballot_sync(0xffffffffu, (static_cast<uint32_t>(code) >> 4) & 1u);
    const int hi = __shfl_down_sync(0xffffffffu, code, 16);
    if (lane < 16) ob[6 + lane] = pack_nibbles(code, hi);
    if (lane == 0) {
        unsigned short *h = reinterpret_cast<unsigned short *>(ob);
        h[0] = __half_as_ushort(__float2half_rn(d));
        h[1] = static_cast<unsigned short>(qh & 0xFFFFu);
        h[2] = static_cast<unsigned short>(qh >> 16);
    }
}

template <int TYPE>
__device__ __forceinline__ void quantize_block(const float *xb, uint8_t *ob, int lane) {
    if (TYPE == QG_Q8_0) q8_0_block(xb, ob, lane);
    else if (TYPE == QG_Q8_K) q8_k_block(xb, ob, lane);
    else if (TYPE == QG_Q8_1) q8_1_block(xb, ob, lane);
    else if (TYPE == QG_Q4_1) q4_1_block(xb, ob, lane);
    else if (TYPE == QG_Q5_0) q5_0_block(xb, ob, lane);
    else q4_0_block(xb, ob, lane);
}

template <int TYPE>
__host__ __device__ constexpr int quant_block_bytes() {
    return TYPE == QG_Q8_K ? 292 : TYPE == QG_Q8_0 ? 34 : TYPE == QG_Q8_1 ? 36 : TYPE == QG_Q4_1 ? 20
                                                                                 : TYPE == QG_Q5_0 ? 22 : 18;
}

// One warp per block over n_blocks consecutive blocks.
template <int TYPE>
__global__ void quantize_kernel(const float *__restrict__ x, uint8_t *__restrict__ out, int64_t n_blocks) {
    pdl_allow_dependents();
    pdl_wait_prior_grids();
    constexpr int elems = TYPE == QG_Q8_K ? 256 : 32;
    constexpr int bytes = quant_block_bytes<TYPE>();
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t b = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); b < n_blocks;
         b += warps)
        quantize_block<TYPE>(x + b * elems, out + b * bytes, lane);
}

// Batches: the activations of matrix m (blocks_per_mat blocks, from t.x[m])
// go to out + m * blocks_per_mat * block bytes.
template <int TYPE>
__global__ void quantize_batched_kernel(const QuantTable t, uint8_t *__restrict__ out, int n_mats,
                                        int64_t blocks_per_mat) {
    pdl_allow_dependents();
    pdl_wait_prior_grids();
    constexpr int elems = TYPE == QG_Q8_K ? 256 : 32;
    constexpr int bytes = quant_block_bytes<TYPE>();
    const int lane = threadIdx.x & 31;
    const int64_t n_blocks = blocks_per_mat * n_mats;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t b = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); b < n_blocks;
         b += warps) {
        const int64_t m = b / blocks_per_mat, i = b % blocks_per_mat;
        quantize_block<TYPE>(t.x[m] + i * elems, out + b * bytes, lane);
    }
}

// Launches (kernels are launched from the translation unit that defines them).
cudaError_t launch_quantize_kernel(int type, int grid, int block, cudaStream_t s, const float *x, uint8_t *out,
                                   int64_t n_blocks) {
    switch (type) {
    case QG_Q8_0: return launch_pdl(quantize_kernel<QG_Q8_0>, grid, block, 0, s, x, out, n_blocks);
    case QG_Q8_K: return launch_pdl(quantize_kernel<QG_Q8_K>, grid, block, 0, s, x, out, n_blocks);
    case QG_Q4_0: return launch_pdl(quantize_kernel<QG_Q4_0>, grid, block, 0, s, x, out, n_blocks);
    case QG_Q8_1: return launch_pdl(quantize_kernel<QG_Q8_1>, grid, block, 0, s, x, out, n_blocks);
    case QG_Q4_1: return launch_pdl(quantize_kernel<QG_Q4_1>, grid, block, 0, s, x, out, n_blocks);
    case QG_Q5_0: return launch_pdl(quantize_kernel<QG_Q5_0>, grid, block, 0, s, x, out, n_blocks);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_quantize_batched_kernel(int type, int grid, int block, cudaStream_t s, const QuantTable &t,
                                           uint8_t *out, int n_mats, int64_t blocks_per_mat) {
    switch (type) {
    case QG_Q8_0: return launch_pdl(quantize_batched_kernel<QG_Q8_0>, grid, block, 0, s, t, out, n_mats, blocks_per_mat);
    case QG_Q8_K: return launch_pdl(quantize_batched_kernel<QG_Q8_K>, grid, block, 0, s, t, out, n_mats, blocks_per_mat);
    case QG_Q8_1: return launch_pdl(quantize_batched_kernel<QG_Q8_1>, grid, block, 0, s, t, out, n_mats, blocks_per_mat);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qg
