// dequant.cu - dequantize_rows: every element of a block-quantized matrix
// to f32 ("Quantization" (sipllm), Per-format dequant; "量化格式" (candle),
// block structure table; "Quantization" (rml), Unpacking the packed fields).
//
// Each thread writes 8 consecutive elements (two 16-byte streaming stores),
// consecutive threads consecutive groups, so the f32 output -- the bulk of
// the traffic, 4 bytes per element against 0.56..1.06 read -- is written
// fully coalesced. Every product below is exact in f32 (a f16 d has 11
// significant bits, the sub-block scales at most 7, the codes at most 6), so
// the values are unique and equal the scalar definition bit for bit; the
// explicit __fmul_rn/__fsub_rn only make the order visible.
#include "qg_common.cuh"

namespace qg {

__device__ __forceinline__ void store8(float *dst, const float (&v)[8]) {
    float4 *d4 = reinterpret_cast<float4 *>(dst);
    __stcs(d4, make_float4(v[0], v[1], v[2], v[3]));
    __stcs(d4 + 1, make_float4(v[4], v[5], v[6], v[7]));
}

// The same 8 values rounded to f16 (round to nearest even), one 16-byte
// store: the operand form of the prefill GEMM.
__device__ __forceinline__ void store8(__half *dst, const float (&v)[8]) {
    uint4 o;
    o.x = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v[0]))) |
          (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v[1]))) << 16);
    o.y = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v[2]))) |
          (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v[3]))) << 16);
    o.z = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v[4]))) |
          (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v[5]))) << 16);
    o.w = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v[6]))) |
          (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v[7]))) << 16);
    __stcs(reinterpret_cast<uint4 *>(dst), o);
}

__device__ __forceinline__ uint32_t ldg_u16(const uint8_t *p) {
    return static_cast<uint32_t>(__ldg(reinterpret_cast<const uint16_t *>(p)));
}

// groups: total 8-element groups = n_rows * n_in / 8; W is the flat block stream.
template <class O>
__global__ void dequant_q8_0_kernel(const uint8_t *__restrict__ W, O *__restrict__ out, int64_t groups) {
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint8_t *blk = W + (g >> 2) * 34;
        const float d = f16_bits_to_f32(ldg_u16(blk));
        const uint8_t *qs = blk + 2 + 8 * (g & 3);
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(static_cast<float>(static_cast<int8_t>(__ldg(qs + i))), d);
        store8(out + g * 8, v);
    }
}

template <class O>
__global__ void dequant_q4_0_kernel(const uint8_t *__restrict__ W, O *__restrict__ out, int64_t groups) {
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint8_t *blk = W + (g >> 2) * 18;
        const float d = f16_bits_to_f32(ldg_u16(blk));
        const int q = static_cast<int>(g & 3);       // elements 8q..8q+7 of the block
        const uint8_t *qs = blk + 2 + 8 * (q & 1);   // bytes (8q..8q+7) mod 16
        const int shift = q >= 2 ? 4 : 0;            // elements 16.. use the high nibble
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int code = (__ldg(qs + i) >> shift) & 0xF;
            v[i] = __fmul_rn(static_cast<float>(code - 8), d);
        }
        store8(out + g * 8, v);
    }
}

// Q4_1: code * d is exact (4 + 11 bits), so code * d + m rounds once.
template <class O>
__global__ void dequant_q4_1_kernel(const uint8_t *__restrict__ W, O *__restrict__ out, int64_t groups) {
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint8_t *blk = W + (g >> 2) * 20;
        const float d = f16_bits_to_f32(ldg_u16(blk));
        const float m = f16_bits_to_f32(ldg_u16(blk + 2));
        const int q = static_cast<int>(g & 3);
        const uint8_t *qs = blk + 4 + 8 * (q & 1);
        const int shift = q >= 2 ? 4 : 0;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int code = (__ldg(qs + i) >> shift) & 0xF;
            v[i] = __fadd_rn(__fmul_rn(static_cast<float>(code), d), m);
        }
        store8(out + g * 8, v);
    }
}

// Q5_0: 5-bit code = nibble | bit e of qh << 4, value (code - 16) * d.
template <class O>
__global__ void dequant_q5_0_kernel(const uint8_t *__restrict__ W, O *__restrict__ out, int64_t groups) {
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint8_t *blk = W + (g >> 2) * 22;
        const float d = f16_bits_to_f32(ldg_u16(blk));
        const uint32_t qh = ldg_u16(blk + 2) | (ldg_u16(blk + 4) << 16);
        const int q = static_cast<int>(g & 3);
        const uint8_t *qs = blk + 6 + 8 * (q & 1);
        const int shift = q >= 2 ? 4 : 0;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = 8 * q + i;
            const int code = ((__ldg(qs + i) >> shift) & 0xF) | (((qh >> e) & 1u) << 4);
            v[i] = __fmul_rn(static_cast<float>(code - 16), d);
        }
        store8(out + g * 8, v);
    }
}

// Q8_1: q * d (s is not part of the values).
template <class O>
__global__ void dequant_q8_1_kernel(const uint8_t *__restrict__ W, O *__restrict__ out, int64_t groups) {
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint8_t *blk = W + (g >> 2) * 36;
        const float d = f16_bits_to_f32(ldg_u16(blk));
        const uint8_t *qs = blk + 4 + 8 * (g & 3);
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(static_cast<float>(static_cast<int8_t>(__ldg(qs + i))), d);
        store8(out + g * 8, v);
    }
}

template <class O>
__global__ void dequant_q4_k_kernel(const uint8_t *__restrict__ W, O *__restrict__ out, int64_t groups) {
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        // the block's d, dmin and scales in two 8-byte loads, the group's 8
        // codes in one (the 144-byte blocks keep W's 16-byte alignment)
        const uint8_t *blk = W + (g >> 5) * 144;
        const int e0 = 8 * static_cast<int>(g & 31);
        const int j = e0 >> 5;                      // sub-block
        const uint2 h0 = __ldg(reinterpret_cast<const uint2 *>(blk));      // d | dmin | scales[0..3]
        const uint2 h1 = __ldg(reinterpret_cast<const uint2 *>(blk + 8));  // scales[4..11]
        const float d = f16_bits_to_f32(h0.x);
        const float dmin = f16_bits_to_f32(h0.x >> 16);
        const uint32_t sw[3] = {h0.y, h1.x, h1.y};
        auto s8 = [&](int k) { return static_cast<int>((sw[k >> 2] >> (8 * (k & 3))) & 0xFFu); };
        int sc, m;
        if (j < 4) {
            sc = s8(j) & 63;
            m = s8(j + 4) & 63;
        } else {
            sc = (s8(j + 4) & 0xF) | ((s8(j - 4) >> 6) << 4);
            m = (s8(j + 4) >> 4) | ((s8(j) >> 6) << 4);
        }
        const int p = e0 & 63;                       // position in the 64-element chunk
        const uint2 qw = __ldg(reinterpret_cast<const uint2 *>(blk + 16 + 32 * (e0 >> 6) + (p & 31)));
        const int shift = p >= 32 ? 4 : 0;
        const float dsc = __fmul_rn(d, static_cast<float>(sc));
        const float off = __fmul_rn(dmin, static_cast<float>(m));
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int q = ((i < 4 ? qw.x : qw.y) >> (8 * (i & 3) + shift)) & 0xF;
            v[i] = __fsub_rn(__fmul_rn(dsc, static_cast<float>(q)), off);
        }
        store8(out + g * 8, v);
    }
}

template <class O>
__global__ void dequant_q6_k_kernel(const uint8_t *__restrict__ W, O *__restrict__ out, int64_t groups) {
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint8_t *blk = W + (g >> 5) * 210;
        const int e0 = 8 * static_cast<int>(g & 31);
        const int h = e0 >> 7, k = (e0 >> 5) & 3, l0 = e0 & 31;
        const float d = f16_bits_to_f32(ldg_u16(blk + 208));
        const int sc = static_cast<int8_t>(__ldg(blk + 192 + (e0 >> 4)));
        const float dsc = __fmul_rn(d, static_cast<float>(sc));
        const uint8_t *ql = blk + 64 * h + 32 * (k & 1) + l0;
        const uint8_t *qh = blk + 128 + 32 * h + l0;
        const int lshift = k >= 2 ? 4 : 0;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int q = ((__ldg(ql + i) >> lshift) & 0xF) | (((__ldg(qh + i) >> (2 * k)) & 3) << 4);
            v[i] = __fmul_rn(dsc, static_cast<float>(q - 32));
        }
        store8(out + g * 8, v);
    }
}

// Q5_K: Q4_K's scales, mins and nibbles plus bit j of qh[e % 32] as bit 4
// of the code (sub-block j = e / 32).
template <class O>
__global__ void dequant_q5_k_kernel(const uint8_t *__restrict__ W, O *__restrict__ out, int64_t groups) {
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint8_t *blk = W + (g >> 5) * 176;
        const int e0 = 8 * static_cast<int>(g & 31);
        const int j = e0 >> 5;
        const float d = f16_bits_to_f32(ldg_u16(blk));
        const float dmin = f16_bits_to_f32(ldg_u16(blk + 2));
        const uint8_t *s = blk + 4;
        int sc, m;
        if (j < 4) {
            sc = __ldg(s + j) & 63;
            m = __ldg(s + j + 4) & 63;
        } else {
            sc = (__ldg(s + j + 4) & 0xF) | ((__ldg(s + j - 4) >> 6) << 4);
            m = (__ldg(s + j + 4) >> 4) | ((__ldg(s + j) >> 6) << 4);
        }
        const float dsc = __fmul_rn(d, static_cast<float>(sc));
        const float off = __fmul_rn(dmin, static_cast<float>(m));
        const uint8_t *qs = blk + 48 + 32 * (j >> 1) + (e0 & 31);
        const uint8_t *qh = blk + 16 + (e0 & 31);
        const int shift = (j & 1) ? 4 : 0;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int q = ((__ldg(qs + i) >> shift) & 0xF) | (((__ldg(qh + i) >> j) & 1) << 4);
            v[i] = __fsub_rn(__fmul_rn(dsc, static_cast<float>(q)), off);
        }
        store8(out + g * 8, v);
    }
}

// Q2_K: element e = 128n + 32j + 16h + l takes bits 2j of qs[32n + 16h + l];
// sub-block e / 16 has scale scales[e/16] & 15 and min scales[e/16] >> 4.
template <class O>
__global__ void dequant_q2_k_kernel(const uint8_t *__restrict__ W, O *__restrict__ out, int64_t groups) {
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint8_t *blk = W + (g >> 5) * 84;
        const int e0 = 8 * static_cast<int>(g & 31);
        const int n = e0 >> 7, j = (e0 >> 5) & 3, h = (e0 >> 4) & 1, l0 = e0 & 15;
        const int sm = __ldg(blk + (e0 >> 4));
        const float d = f16_bits_to_f32(ldg_u16(blk + 80));
        const float dmin = f16_bits_to_f32(ldg_u16(blk + 82));
        const float dsc = __fmul_rn(d, static_cast<float>(sm & 0xF));
        const float off = __fmul_rn(dmin, static_cast<float>(sm >> 4));
        const uint8_t *qs = blk + 16 + 32 * n + 16 * h + l0;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int q = (__ldg(qs + i) >> (2 * j)) & 3;
            v[i] = __fsub_rn(__fmul_rn(dsc, static_cast<float>(q)), off);
        }
        store8(out + g * 8, v);
    }
}

// Q3_K: the Q2_K 2-bit value less 4 when bit 4n + j of hmask[16h + l] is
// clear; scale = 6-bit field - 32 (low 4 bits in nibble (e/16) / 8 of byte
// (e/16) % 8, high 2 bits at bits 2((e/16) / 4) of byte 8 + (e/16) % 4).
template <class O>
__global__ void dequant_q3_k_kernel(const uint8_t *__restrict__ W, O *__restrict__ out, int64_t groups) {
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint8_t *blk = W + (g >> 5) * 110;
        const int e0 = 8 * static_cast<int>(g & 31);
        const int n = e0 >> 7, j = (e0 >> 5) & 3, h = (e0 >> 4) & 1, l0 = e0 & 15;
        const int sb = e0 >> 4;
        const int lo4 = (__ldg(blk + 96 + (sb & 7)) >> (4 * (sb >> 3))) & 0xF;
        const int hi2 = (__ldg(blk + 104 + (sb & 3)) >> (2 * (sb >> 2))) & 3;
        const float d = f16_bits_to_f32(ldg_u16(blk + 108));
        const float dsc = __fmul_rn(d, static_cast<float>((lo4 | (hi2 << 4)) - 32));
        const uint8_t *qs = blk + 32 + 32 * n + 16 * h + l0;
        const uint8_t *hm = blk + 16 * h + l0;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int q2 = (__ldg(qs + i) >> (2 * j)) & 3;
            const int hb = (__ldg(hm + i) >> (4 * n + j)) & 1;
            v[i] = __fmul_rn(dsc, static_cast<float>(q2 - (hb ? 0 : 4)));
        }
        store8(out + g * 8, v);
    }
}

template <class O>
__global__ void dequant_q8_k_kernel(const uint8_t *__restrict__ W, O *__restrict__ out, int64_t groups) {
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint8_t *blk = W + (g >> 5) * 292;
        const float d = __ldg(reinterpret_cast<const float *>(blk));
        const int8_t *qs = reinterpret_cast<const int8_t *>(blk + 4 + 8 * (g & 31));
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(static_cast<float>(__ldg(qs + i)), d);
        store8(out + g * 8, v);
    }
}


// One dequantization launch over `groups` 8-element groups (kernel
// templates are launched from the translation unit that defines them).
template <class O>
cudaError_t launch_dequant(int type, const uint8_t *w, O *out, int64_t groups, unsigned g, int threads,
                           cudaStream_t s) {
    switch (type) {
    case QG_Q8_0: dequant_q8_0_kernel<O><<<g, threads, 0, s>>>(w, out, groups); break;
    case QG_Q4_0: dequant_q4_0_kernel<O><<<g, threads, 0, s>>>(w, out, groups); break;
    case QG_Q4_1: dequant_q4_1_kernel<O><<<g, threads, 0, s>>>(w, out, groups); break;
    case QG_Q5_0: dequant_q5_0_kernel<O><<<g, threads, 0, s>>>(w, out, groups); break;
    case QG_Q8_1: dequant_q8_1_kernel<O><<<g, threads, 0, s>>>(w, out, groups); break;
    case QG_Q4_K: dequant_q4_k_kernel<O><<<g, threads, 0, s>>>(w, out, groups); break;
    case QG_Q6_K: dequant_q6_k_kernel<O><<<g, threads, 0, s>>>(w, out, groups); break;
    case QG_Q2_K: dequant_q2_k_kernel<O><<<g, threads, 0, s>>>(w, out, groups); break;
    case QG_Q3_K: dequant_q3_k_kernel<O><<<g, threads, 0, s>>>(w, out, groups); break;
    case QG_Q5_K: dequant_q5_k_kernel<O><<<g, threads, 0, s>>>(w, out, groups); break;
    case QG_Q8_K: dequant_q8_k_kernel<O><<<g, threads, 0, s>>>(w, out, groups); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}
template cudaError_t launch_dequant<float>(int, const uint8_t *, float *, int64_t, unsigned, int, cudaStream_t);
template cudaError_t launch_dequant<__half>(int, const uint8_t *, __half *, int64_t, unsigned, int, cudaStream_t);

}  // namespace qg
