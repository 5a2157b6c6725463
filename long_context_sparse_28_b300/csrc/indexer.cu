// a5: lightning-indexer scores I(t,s) = sum_h w[t,h] * ReLU(q[t,h] . khat_s) and the
// csa_index_topk entry point (scores -> top-k).
//
// honbul.tistory.com/221 "CSA" (a small indexer finds the blocks related to the current
// token); pogovet.com DeepSeek-V4 article, detail 4 (FP4 lightning indexer, top-k blocks per
// query) and detail 5 (the indexer runs in FP4).
//
// Generic CUDA-core kernel: one thread per (query row, compressed entry).  The key codes are
// decoded exactly (e4m3 / e2m1 code values are small integers times powers of two) and the
// per-row (e4m3) or per-32 (e2m1) scale is applied to each 32-wide partial dot product, so
// the only rounding is the fp32 accumulation.
#include "common.cuh"
#include "quant.cuh"

namespace csahca {
namespace {

__device__ __forceinline__ float e2m1_value(uint32_t c) {
    const uint32_t mag = c & 7u, e = mag >> 1, mt = mag & 1u;
    const float v = (e == 0) ? 0.5f * (float)mt : ldexpf(1.0f + 0.5f * (float)mt, (int)e - 1);
    return (c & 8u) ? -v : v;
}

// 8 consecutive code values (unscaled) of key row `row` starting at channel c0.
__device__ __forceinline__ void key_codes8(const void* codes, int fmt, int d_I, int64_t row, int c0,
                                           float (&kv)[8]) {
    if (fmt == CSAHCA_F32) {
        load8(static_cast<const float*>(codes) + row * d_I + c0, kv);
    } else if (fmt == CSAHCA_BF16) {
        load8(static_cast<const __nv_bfloat16*>(codes) + row * d_I + c0, kv);
    } else if (fmt == CSAHCA_E4M3_ROWSCALE) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(codes) + row * d_I + c0));
        const uint32_t w[2] = {u.x, u.y};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t byte = (w[i >> 2] >> (8 * (i & 3))) & 0xFFu;
            const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)byte, __NV_E4M3);
            kv[i] = __half2float(__half(h));
        }
    } else {
        const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(codes) + row * (d_I / 2) + c0 / 2));
#pragma unroll
        for (int i = 0; i < 8; ++i) kv[i] = e2m1_value((u >> (4 * i)) & 0xFu);
    }
}

__device__ __forceinline__ float block_scale(const void* scales, int fmt, int d_I, int64_t row, int blk) {
    if (fmt == CSAHCA_E4M3_ROWSCALE) return __ldg(static_cast<const float*>(scales) + row);
    if (fmt == CSAHCA_E2M1_UE8M0) {
        const int e = (int)__ldg(static_cast<const uint8_t*>(scales) + row * (d_I / 32) + blk) - 127;
        return ldexpf(1.0f, e);
    }
    return 1.0f;
}

template <int MAXH>
__global__ void __launch_bounds__(256) index_score_kernel(
    const void* __restrict__ q_idx, int q_dtype, const float* __restrict__ w, const void* __restrict__ k_codes,
    const void* __restrict__ k_scale, int fmt, int T, int H_I, int d_I, const int64_t* __restrict__ q_pos,
    int64_t Ncap, int m, float* __restrict__ S) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ float sh[];                 // q [H_I][d_I], then w [H_I]
    float* qs = sh;
    float* ws = sh + H_I * d_I;
    const int r = blockIdx.y;
    const int b = r / T;
    const int64_t p = q_pos[r];
    int64_t n = (p >= 0) ? (p + 1) / m : 0;
    n = n < Ncap ? n : Ncap;
    const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if ((int64_t)blockIdx.x * blockDim.x >= n) return;   // CTA-uniform
    for (int i = threadIdx.x; i < H_I * d_I; i += blockDim.x) {
        const int64_t off = (int64_t)r * H_I * d_I + i;
        qs[i] = (q_dtype == CSAHCA_F32) ? static_cast<const float*>(q_idx)[off]
                                        : __bfloat162float(static_cast<const __nv_bfloat16*>(q_idx)[off]);
    }
    for (int i = threadIdx.x; i < H_I; i += blockDim.x) ws[i] = w[(int64_t)r * H_I + i];
    __syncthreads();
    if (s >= n) return;
    const int64_t row = (int64_t)b * Ncap + s;
    float acc[MAXH];
#pragma unroll
    for (int h = 0; h < MAXH; ++h) acc[h] = 0.0f;
    for (int blk = 0; blk < d_I / 32; ++blk) {
        float part[MAXH];
#pragma unroll
        for (int h = 0; h < MAXH; ++h) part[h] = 0.0f;
        for (int c0 = blk * 32; c0 < blk * 32 + 32; c0 += 8) {
            float kv[8];
            key_codes8(k_codes, fmt, d_I, row, c0, kv);
#pragma unroll
            for (int h = 0; h < MAXH; ++h) {
                if (h < H_I) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) part[h] = fmaf(qs[h * d_I + c0 + c], kv[c], part[h]);
                }
            }
        }
        const float sc = block_scale(k_scale, fmt, d_I, row, blk);
#pragma unroll
        for (int h = 0; h < MAXH; ++h) acc[h] = fmaf(sc, part[h], acc[h]);
    }
    float score = 0.0f;
#pragma unroll
    for (int h = 0; h < MAXH; ++h)
        if (h < H_I) score = fmaf(ws[h], fmaxf(acc[h], 0.0f), score);
    S[(int64_t)r * Ncap + s] = score;
}

}  // namespace
// OCP MX FP4 (E2M1 codes, UE8M0 per 32) rows of 64 values -> bf16, exactly: e2m1 values have at
// most two significant bits and the scale is a power of two, so every product is a bf16 value
// while the scale exponent stays within bf16's range (byte - 127 <= 125, i.e. inputs below ~1e38).
// One thread per 8 values (4 code bytes).
__global__ void __launch_bounds__(256) expand_e2m1_rows_kernel(const uint8_t* __restrict__ codes,
                                                               const uint8_t* __restrict__ scales, int64_t rows,
                                                               __nv_bfloat16* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= rows * 8) return;
    const int64_t row = t >> 3;
    const int part = (int)(t & 7);                       // values 8 part .. 8 part + 7
    const uint32_t c4 = *reinterpret_cast<const uint32_t*>(codes + row * 32 + part * 4);
    const float sc = ldexpf(1.0f, (int)scales[row * 2 + (part >> 2)] - 127);
    // E2M1 code s e1 e0 m: |x| = m / 2 for e = 0, (1 + m / 2) 2^(e - 1) otherwise
    auto e2m1 = [](uint32_t c) {
        const uint32_t e = (c >> 1) & 3u, mb = c & 1u;
        const float mag = e == 0 ? 0.5f * (float)mb : ldexpf(1.0f + 0.5f * (float)mb, (int)e - 1);
        return (c & 8u) ? -mag : mag;
    };
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t byte = (c4 >> (8 * j)) & 0xFFu;   // the even element in the low nibble
        o[j] = pack_bf16x2(e2m1(byte & 0xFu) * sc, e2m1(byte >> 4) * sc);
    }
    *reinterpret_cast<uint4*>(out + row * 64 + part * 8) = make_uint4(o[0], o[1], o[2], o[3]);
}

// FP4 queries with many rows (chunked prefill): the rows' keys and queries are expanded exactly to
// bf16 in the workspace and scored by the bf16 prefill indexer, whose tiles serve 128 / H_I query
// rows at once (the block-scaled decode indexer takes one query row per work item).
bool fp4_prefill_form(int B, int T, int H_I, int d_I, int64_t Ncap) {
    return (int64_t)B * T > 256 && d_I == 64 && (H_I == 16 || H_I == 32 || H_I == 64) && T % (128 / H_I) == 0 &&
           Ncap >= 1;
}
size_t fp4_prefill_scratch_bytes(int B, int T, int H_I, int64_t Ncap) {
    return align256((size_t)B * Ncap * 64 * 2) + align256((size_t)B * T * H_I * 64 * 2);
}

}  // namespace csahca

using namespace csahca;

extern "C" {

size_t csa_index_topk_fp4_workspace(int B, int T, int H_I, int64_t Ncap, int k) {
    const size_t base = csa_index_topk_workspace(B, T, Ncap, k);
    if (base == 0 || !fp4_prefill_form(B, T, H_I, 64, Ncap)) return base;
    return base + fp4_prefill_scratch_bytes(B, T, H_I, Ncap);
}

size_t csa_index_topk_workspace(int B, int T, int64_t Ncap, int k) {
    (void)k;
    if (B <= 0 || T <= 0 || Ncap < 0) return 0;
    const int64_t R = (int64_t)B * T;
    return align256((size_t)R * Ncap * 4) + topk_workspace_bytes(R, Ncap);
}

static csahca_status index_validate(const void* q_idx, csahca_dtype q_dtype, const float* w, const void* k_codes,
                                    const void* k_scale, csahca_dtype key_fmt, int B, int T, int H_I, int d_I,
                                    const int64_t* q_pos, int64_t Ncap, int m) {
    CSAHCA_REQUIRE(q_idx && w && k_codes && q_pos);
    CSAHCA_REQUIRE(q_dtype == CSAHCA_F32 || q_dtype == CSAHCA_BF16);
    CSAHCA_REQUIRE(key_fmt >= CSAHCA_F32 && key_fmt <= CSAHCA_E2M1_UE8M0);
    CSAHCA_REQUIRE(B >= 1 && T >= 1 && (int64_t)B * T <= 65535 && H_I >= 1 && H_I <= 64);
    CSAHCA_REQUIRE(d_I >= 32 && d_I <= 256 && d_I % 32 == 0 && H_I * d_I <= 4096);
    CSAHCA_REQUIRE(m >= 1 && Ncap >= 1);
    if (key_fmt >= CSAHCA_E4M3_ROWSCALE) CSAHCA_REQUIRE(k_scale != nullptr);
    if (key_fmt == CSAHCA_F32) CSAHCA_REQUIRE(aligned(k_codes, 32));
    else CSAHCA_REQUIRE(aligned(k_codes, 16));
    return CSAHCA_OK;
}

// Launches the scores kernel; with a non-null hist1 the decode tensor-core kernel also accumulates
// the top-k histogram (*hist_done = true); the prefill and generic kernels do not (the top-k then
// forms it in a pass of its own).
static csahca_status index_scores_launch(const void* q_idx, csahca_dtype q_dtype, const float* w,
                                         const void* k_codes, const void* k_scale, csahca_dtype key_fmt, int B,
                                         int T, int H_I, int d_I, const int64_t* q_pos, int64_t Ncap, int m,
                                         float* S, uint32_t* hist1, bool* hist_done, cudaStream_t st) {
    const int R = B * T;
    if (hist_done) *hist_done = false;
    if (index_tc_supported(q_dtype, key_fmt, H_I, d_I, Ncap, k_codes, k_scale, B, R)) {
        unsigned* err = err_word();
        if (!err) return CSAHCA_ERR_CUDA;
        const cudaError_t e = index_tc_launch(q_idx, w, k_codes, k_scale, key_fmt, B, T, H_I, q_pos, Ncap, m, S,
                                              hist1, err, st);
        if (e != cudaErrorNotSupported) {
            count_launch();
            if (hist_done) *hist_done = hist1 != nullptr;
            return e == cudaSuccess ? CSAHCA_OK : CSAHCA_ERR_CUDA;
        }
    }
    if (index_prefill_supported(q_dtype, key_fmt, H_I, d_I, Ncap, q_idx, k_codes, B, T)) {
        unsigned* err = err_word();
        if (!err) return CSAHCA_ERR_CUDA;
        const cudaError_t e = index_prefill_launch(q_idx, w, k_codes, B, T, H_I, q_pos, Ncap, m, S, err, st);
        if (e != cudaErrorNotSupported) {
            count_launch();
            return e == cudaSuccess ? CSAHCA_OK : CSAHCA_ERR_CUDA;
        }
    }
    dim3 grid((unsigned)cdiv(Ncap, 256), (unsigned)R);
    const size_t smem = (size_t)(H_I * d_I + H_I) * 4;
    if (H_I <= 16)
        (void)launch_pdl(index_score_kernel<16>, dim3(grid), dim3(256), smem, st, q_idx, q_dtype, w, k_codes, k_scale, key_fmt, T, H_I, d_I,
                                                        q_pos, Ncap, m, S);
    else
        (void)launch_pdl(index_score_kernel<64>, dim3(grid), dim3(256), smem, st, q_idx, q_dtype, w, k_codes, k_scale, key_fmt, T, H_I, d_I,
                                                        q_pos, Ncap, m, S);
    count_launch();
    CSAHCA_CHECK_LAUNCH();
    return CSAHCA_OK;
}

csahca_status csa_index_scores(const void* q_idx, csahca_dtype q_dtype, const float* w, const void* k_codes,
                               const void* k_scale, csahca_dtype key_fmt, int B, int T, int H_I, int d_I,
                               const int64_t* q_pos, int64_t Ncap, int m, float* scores, csahca_stream_t stream) {
    const csahca_status v = index_validate(q_idx, q_dtype, w, k_codes, k_scale, key_fmt, B, T, H_I, d_I, q_pos,
                                           Ncap, m);
    if (v != CSAHCA_OK) return v;
    CSAHCA_REQUIRE(scores != nullptr);
    return index_scores_launch(q_idx, q_dtype, w, k_codes, k_scale, key_fmt, B, T, H_I, d_I, q_pos, Ncap, m, scores,
                               nullptr, nullptr, (cudaStream_t)stream);
}

csahca_status csa_index_topk(const void* q_idx, csahca_dtype q_dtype, const float* w, const void* k_codes,
                             const void* k_scale, csahca_dtype key_fmt, int B, int T, int H_I, int d_I,
                             const int64_t* q_pos, int64_t Ncap, int m, int k, int32_t* idx_out, float* scores_out,
                             void* workspace, size_t ws_bytes, csahca_stream_t stream) {
    const csahca_status v = index_validate(q_idx, q_dtype, w, k_codes, k_scale, key_fmt, B, T, H_I, d_I, q_pos,
                                           Ncap, m);
    if (v != CSAHCA_OK) return v;
    CSAHCA_REQUIRE(idx_out != nullptr && k >= 1 && k <= 65536);
    const int R = B * T;
    if (!workspace || !aligned(workspace, 256) || ws_bytes < csa_index_topk_workspace(B, T, Ncap, k))
        return CSAHCA_ERR_WORKSPACE;
    // workspace: the top-k's histograms (zero between calls: the top-k clears each row's after
    // use) and bitmaps, then the scores
    char* ws = static_cast<char*>(workspace);
    TopkWorkspace tw = topk_carve(ws, R, Ncap);
    float* S = scores_out ? scores_out : reinterpret_cast<float*>(ws + topk_workspace_bytes(R, Ncap));
    cudaStream_t st = (cudaStream_t)stream;
    bool hist_done = false;
    const csahca_status e = index_scores_launch(q_idx, q_dtype, w, k_codes, k_scale, key_fmt, B, T, H_I, d_I, q_pos,
                                                Ncap, m, S, tw.hist1, &hist_done, st);
    if (e != CSAHCA_OK) return e;
    return topk_launch(S, Ncap, R, nullptr, q_pos, m, Ncap, k, idx_out, tw, hist_done, st);
}

csahca_status csa_index_topk_fp4(const void* q_codes, const void* q_scale, const float* w, const void* k_codes,
                                 const void* k_scale, int B, int T, int H_I, int d_I, const int64_t* q_pos,
                                 int64_t Ncap, int m, int k, int32_t* idx_out, float* scores_out, void* workspace,
                                 size_t ws_bytes, csahca_stream_t stream) {
    CSAHCA_REQUIRE(q_codes && q_scale && w && k_codes && k_scale && q_pos && idx_out);
    CSAHCA_REQUIRE(B >= 1 && T >= 1 && (int64_t)B * T <= 65535 && m >= 1 && Ncap >= 1 && k >= 1 && k <= 65536);
    CSAHCA_REQUIRE(H_I >= 1 && d_I >= 32 && d_I % 32 == 0);
    const int R = B * T;
    if (!(d_I == 64 && (H_I == 16 || H_I == 32 || H_I == 64)) ||
        !index_tc_supported(CSAHCA_BF16, CSAHCA_E2M1_UE8M0, H_I, d_I, Ncap, k_codes, k_scale, B, R) ||
        !aligned(q_codes, 16) || !aligned(q_scale, 2))
        return CSAHCA_ERR_UNSUPPORTED;
    if (!workspace || !aligned(workspace, 256) || ws_bytes < csa_index_topk_workspace(B, T, Ncap, k))
        return CSAHCA_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    TopkWorkspace tw = topk_carve(ws, R, Ncap);
    float* S = scores_out ? scores_out : reinterpret_cast<float*>(ws + topk_workspace_bytes(R, Ncap));
    cudaStream_t st = (cudaStream_t)stream;
    unsigned* err = err_word();
    if (!err) return CSAHCA_ERR_CUDA;
    const size_t base = csa_index_topk_workspace(B, T, Ncap, k);
    if (fp4_prefill_form(B, T, H_I, d_I, Ncap) && ws_bytes >= base + fp4_prefill_scratch_bytes(B, T, H_I, Ncap)) {
        __nv_bfloat16* kb = reinterpret_cast<__nv_bfloat16*>(ws + base);
        __nv_bfloat16* qb = reinterpret_cast<__nv_bfloat16*>(ws + base + align256((size_t)B * Ncap * 64 * 2));
        const int64_t krows = (int64_t)B * Ncap, qrows = (int64_t)R * H_I;
        if (index_prefill_supported(CSAHCA_BF16, CSAHCA_BF16, H_I, d_I, Ncap, qb, kb, B, T)) {
            (void)launch_pdl(expand_e2m1_rows_kernel, dim3((unsigned)cdiv(krows * 8, 256)), dim3(256), 0, st,
                             static_cast<const uint8_t*>(k_codes), static_cast<const uint8_t*>(k_scale), krows, kb);
            (void)launch_pdl(expand_e2m1_rows_kernel, dim3((unsigned)cdiv(qrows * 8, 256)), dim3(256), 0, st,
                             static_cast<const uint8_t*>(q_codes), static_cast<const uint8_t*>(q_scale), qrows, qb);
            count_launch(2);
            const cudaError_t ep = index_prefill_launch(qb, w, kb, B, T, H_I, q_pos, Ncap, m, S, err, st);
            if (ep == cudaSuccess) {
                count_launch();
                return topk_launch(S, Ncap, R, nullptr, q_pos, m, Ncap, k, idx_out, tw, false, st);
            }
            if (ep != cudaErrorNotSupported) return CSAHCA_ERR_CUDA;
        }
    }
    const cudaError_t e = index_tc_q4_launch(q_codes, q_scale, w, k_codes, k_scale, B, T, H_I, q_pos, Ncap, m, S,
                                             tw.hist1, err, st);
    count_launch();
    if (e == cudaErrorNotSupported) return CSAHCA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return CSAHCA_ERR_CUDA;
    return topk_launch(S, Ncap, R, nullptr, q_pos, m, Ncap, k, idx_out, tw, true, st);
}

}  // extern "C"
