// Index-key quantisation, one warp per row (device side).
//
// Low-precision lightning-indexer keys (pogovet.com DeepSeek-V4 article, details 4-5):
//   E4M3 + fp32 row scale : s = amax/448 (IEEE fp32 divide), code = RNE_e4m3_satfinite(x/s)
//   E2M1 + UE8M0 per 32   : e = min{e : amax <= 6*2^e}, code = RNE_e2m1(x * 2^-e)
// The decisions (scale, rounding) are made in float32 with exact scaling, so the codes are
// a deterministic function of the input values.
#pragma once
#include "common.cuh"

namespace csahca {

// E2M1 code of an already-scaled value (|y| <= 6 expected; saturates), round to nearest even.
__device__ __forceinline__ uint32_t e2m1_code(float y) {
    const float a = fabsf(y);
    const float ulp = (a < 2.0f) ? 0.5f : ((a < 4.0f) ? 1.0f : 2.0f);
    float q = rintf(a / ulp) * ulp;           // exact: division by a power of two
    q = fminf(q, 6.0f);
    const int h = (int)(q * 2.0f);            // 0,1,2,3,4,6,8,12
    uint32_t mag = (h <= 4) ? (uint32_t)h : (h == 6 ? 5u : (h == 8 ? 6u : 7u));
    return mag | (signbit(y) ? 8u : 0u);
}

// Smallest e with amax <= 6*2^e (0 for amax == 0), clamped to the UE8M0 range.
__device__ __forceinline__ int ue8m0_exponent(float amax) {
    if (!(amax > 0.0f)) return 0;
    int ex;
    frexpf(amax, &ex);
    int e = ex - 4;
    while (ldexpf(6.0f, e) < amax) ++e;
    return max(-127, min(127, e));
}

// Quantise one row of d_I values held by a warp (lane holds E = d_I/32 consecutive values,
// E <= 8) into `fmt`.  Writes codes_row / scale_row of that format.
__device__ __forceinline__ void quantize_row_warp(const float (&x)[8], int E, int d_I, int fmt,
                                                  void* codes_row, void* scale_row) {
    const int lane = threadIdx.x & 31;
    if (fmt == CSAHCA_F32) {
        float* o = static_cast<float*>(codes_row) + lane * E;
        #pragma unroll
        for (int e = 0; e < 8; ++e) if (e < E) o[e] = x[e];
    } else if (fmt == CSAHCA_BF16) {
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(codes_row) + lane * E;
        #pragma unroll
        for (int e = 0; e < 8; ++e) if (e < E) o[e] = __float2bfloat16_rn(x[e]);
    } else if (fmt == CSAHCA_E4M3_ROWSCALE) {
        float amax = 0.0f;
        #pragma unroll
        for (int e = 0; e < 8; ++e) if (e < E) amax = fmaxf(amax, fabsf(x[e]));
        amax = warp_max(amax);
        const float s = (amax > 0.0f) ? __fdiv_rn(amax, 448.0f) : 1.0f;
        uint8_t* o = static_cast<uint8_t*>(codes_row) + lane * E;
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (e < E) o[e] = (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(x[e], s), __NV_SATFINITE, __NV_E4M3);
        if (lane == 0) *static_cast<float*>(scale_row) = s;
    } else {  // CSAHCA_E2M1_UE8M0, E even
        float amax = 0.0f;
        #pragma unroll
        for (int e = 0; e < 8; ++e) if (e < E) amax = fmaxf(amax, fabsf(x[e]));
        // lanes sharing a 32-value block: 32/E consecutive lanes
        const int group = 32 / E;
        for (int o = group / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const int ex = ue8m0_exponent(amax);
        uint8_t* o = static_cast<uint8_t*>(codes_row) + lane * E / 2;
        #pragma unroll
        for (int e = 0; e < 8; e += 2) {
            if (e >= E) break;
            const uint32_t lo = e2m1_code(ldexpf(x[e], -ex));
            const uint32_t hi = e2m1_code(ldexpf(x[e + 1], -ex));
            o[e / 2] = (uint8_t)(lo | (hi << 4));
        }
        if ((lane % group) == 0) static_cast<uint8_t*>(scale_row)[(lane * E) / 32] = (uint8_t)(ex + 127);
    }
}

// Load lane's E consecutive input values of a row (F32 or BF16 input).
__device__ __forceinline__ void load_row_slice(const void* row, int in_dtype, int E, float (&x)[8]) {
    const int lane = threadIdx.x & 31;
    for (int e = 0; e < 8; ++e) x[e] = 0.0f;
    if (in_dtype == CSAHCA_F32) {
        const float* p = static_cast<const float*>(row) + lane * E;
        #pragma unroll
        for (int e = 0; e < 8; ++e) if (e < E) x[e] = p[e];
    } else {
        const __nv_bfloat16* p = static_cast<const __nv_bfloat16*>(row) + lane * E;
        #pragma unroll
        for (int e = 0; e < 8; ++e) if (e < E) x[e] = __bfloat162float(p[e]);
    }
}

// Bytes of one stored key row / its scale.
__host__ __device__ inline int64_t key_row_bytes(int fmt, int d_I) {
    return fmt == CSAHCA_F32 ? 4LL * d_I : fmt == CSAHCA_BF16 ? 2LL * d_I
         : fmt == CSAHCA_E4M3_ROWSCALE ? (int64_t)d_I : (int64_t)d_I / 2;
}
__host__ __device__ inline int64_t key_scale_bytes(int fmt, int d_I) {
    return fmt == CSAHCA_E4M3_ROWSCALE ? 4 : fmt == CSAHCA_E2M1_UE8M0 ? d_I / 32 : 0;
}


// ---------------------------------------------------------------- FP8 compressed K/V
// Storage of pooled K/V rows of d = 128 in the CSAHCA_KV_FP8 layout (pogovet.com article,
// detail 5: KV entries in FP8, the RoPE dims in BF16): per 64 values one power-of-two scale 2^e,
// e = the smallest integer with amax <= 448 * 2^e (amax = f 2^ex, f in [0.5, 1): e = ex - 9 when
// f <= 0.875 = 448 / 2^9, else ex - 8; 0 for a zero block; clamped to [-127, 127]), codes
// RNE_e4m3(x * 2^-e) (the scaling is exact); the last 64 dims of K in bfloat16.
// Rows start on 32-byte sectors: K row (224 bytes) = 64 codes | its scale byte | the V row's two
// scale bytes | 29 zero bytes | 64 bf16 RoPE dims at byte 96; V row (128 bytes) = 128 codes.
constexpr int kKv8KRow = 224;
constexpr int kKv8VRow = 128;
constexpr int kKv8Rope = 96;    // byte offset of the RoPE dims in a K row

__device__ __forceinline__ int kv8_block_exponent(float amax) {
    if (!(amax > 0.0f)) return 0;
    int ex;
    const float f = frexpf(amax, &ex);
    const int e = f <= 0.875f ? ex - 9 : ex - 8;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^k for k in [-127, 127] as a float (2^-127 is subnormal).
__device__ __forceinline__ float pow2f(int k) {
    return k >= -126 ? __int_as_float((127 + k) << 23) : __int_as_float(0x00400000);
}

// One warp stores one pooled entry: lane L holds 8 consecutive pooled values, lanes 0-15 the K
// row (dims 8L .. 8L+7), lanes 16-31 the V row (dims 8(L-16) ..).  krow / vrow: the entry's K
// (kKv8KRow bytes) and V (kKv8VRow bytes) rows, 16-byte aligned.  All 32 lanes take part.
__device__ __forceinline__ void store_kv8_warp(const float (&x)[8], unsigned char* krow, unsigned char* vrow,
                                               int lane) {
    float am = 0.0f;
#pragma unroll
    for (int c = 0; c < 8; ++c) am = fmaxf(am, fabsf(x[c]));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));   // the lane's block: 8 aligned lanes
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
    const int e = kv8_block_exponent(am);
    const int e_v1 = __shfl_sync(0xffffffffu, e, 24);
    if (lane >= 8 && lane < 16) {                           // K dims 64..127: bfloat16
        uint4 u;
        u.x = pack_bf16x2(x[0], x[1]);
        u.y = pack_bf16x2(x[2], x[3]);
        u.z = pack_bf16x2(x[4], x[5]);
        u.w = pack_bf16x2(x[6], x[7]);
        *reinterpret_cast<uint4*>(krow + kKv8Rope + (lane - 8) * 16) = u;
    } else {
        const float sc = pow2f(-e);
        uint32_t w[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t c0 = __nv_cvt_float2_to_fp8x2(make_float2(x[4 * h] * sc, x[4 * h + 1] * sc), __NV_SATFINITE,
                                                         __NV_E4M3);
            const uint32_t c1 = __nv_cvt_float2_to_fp8x2(make_float2(x[4 * h + 2] * sc, x[4 * h + 3] * sc),
                                                         __NV_SATFINITE, __NV_E4M3);
            w[h] = c0 | (c1 << 16);
        }
        unsigned char* dst = lane < 8 ? krow + lane * 8 : vrow + (lane - 16) * 8;
        *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    }
    const int e_v0 = __shfl_sync(0xffffffffu, e, 16);
    if (lane == 0) {
        *reinterpret_cast<uint4*>(krow + 64) =
            make_uint4((uint32_t)(e + 127) | ((uint32_t)(e_v0 + 127) << 8) | ((uint32_t)(e_v1 + 127) << 16), 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(krow + 80) = make_uint4(0u, 0u, 0u, 0u);
    }
}

}  // namespace csahca
