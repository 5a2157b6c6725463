// a7 / a8: CSA sparse attention and HCA dense attention, split over key chunks with an exact
// log-sum-exp merge.
//
// CSA (honbul.tistory.com/221 "CSA"; pogovet.com detail 4): keys = the selected compressed
// entries followed by the raw window.  HCA (honbul.tistory.com/221 "HCA"; pogovet.com detail 4):
// keys = every visible compressed entry followed by the raw window.  Both: one joint softmax per
// head; the key range of a query is cut into `splits` chunks processed by separate CTAs, each
// writing (o_s normalised, lse_s); the merge computes lse = log sum exp(lse_s) and
// o = sum_s exp(lse_s - lse) o_s in the fixed order s = 0, 1, ...
//
// This file holds the generic CUDA-core kernel (any supported dtype/H/d); the tensor-core
// kernel for bf16, d = 128 lives in attend_tc.cu and shares the merge and the key-list rules.
#include "common.cuh"
#include "attend.cuh"

#include <algorithm>

namespace csahca {
namespace {

constexpr int kTile = 32;

template <typename T, int HPW, int DPL>
__global__ void __launch_bounds__(256) attend_split_kernel(AttendArgs a, int kps, float* __restrict__ o_part,
                                                           float* __restrict__ lse_part, unsigned* err) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ float smem[];
    const int H = a.H, d = a.d;
    float* Qs = smem;                              // [H][d]
    float* Ks = Qs + H * d;                        // [kTile][d+1]
    float* Vs = Ks + kTile * (d + 1);              // [kTile][d]
    __shared__ const T* kptr[kTile];
    __shared__ const T* vptr[kTile];

    const int r = blockIdx.y, split = blockIdx.x, S = gridDim.x;
    const int b = r / a.T;
    const int64_t p = a.q_pos[r];
    const KeyList kl = key_list(a, r, b, p);
    const int64_t k0 = (int64_t)split * kps;
    const int64_t k1 = kl.total < k0 + kps ? kl.total : k0 + kps;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const T* q = static_cast<const T*>(a.q) + (int64_t)r * H * d;
    for (int i = threadIdx.x; i < H * d; i += blockDim.x) Qs[i] = to_f32(q[i]);

    float mrun[HPW], lrun[HPW], o[HPW][DPL];
#pragma unroll
    for (int i = 0; i < HPW; ++i) {
        mrun[i] = -INFINITY;
        lrun[i] = 0.0f;
#pragma unroll
        for (int c = 0; c < DPL; ++c) o[i][c] = 0.0f;
    }

    for (int64_t t0 = k0; t0 < k1; t0 += kTile) {
        __syncthreads();
        if (threadIdx.x < kTile) {
            const int64_t key = t0 + threadIdx.x;
            const T* kp = nullptr;
            const T* vp = nullptr;
            if (key < k1) key_rows<T>(a, kl, r, b, p, key, &kp, &vp, err);
            kptr[threadIdx.x] = kp;
            vptr[threadIdx.x] = vp;
        }
        __syncthreads();
        const int vec = d / 8;
        for (int it = threadIdx.x; it < kTile * vec; it += blockDim.x) {
            const int j = it / vec, c = (it % vec) * 8;
            float x[8], y[8];
            if (kptr[j]) {
                load8(kptr[j] + c, x);
                load8(vptr[j] + c, y);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = y[e] = 0.0f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                Ks[j * (d + 1) + c + e] = x[e];
                Vs[j * d + c + e] = y[e];
            }
        }
        __syncthreads();
        const bool valid = kptr[lane] != nullptr;
#pragma unroll
        for (int i = 0; i < HPW; ++i) {
            const int h = warp + 8 * i;
            if (h >= H) break;
            float s = 0.0f;
            const float* qh = Qs + h * d;
            const float* kj = Ks + lane * (d + 1);
            for (int c = 0; c < d; ++c) s = fmaf(qh[c], kj[c], s);
            s = valid ? s * a.scale : -INFINITY;
            const float tmax = warp_max(s);
            const float mnew = fmaxf(mrun[i], tmax);
            if (mnew == -INFINITY) continue;                // nothing valid yet (warp-uniform)
            const float alpha = expf(mrun[i] - mnew);       // exp(-inf) = 0 on the first tile
            const float pj = valid ? expf(s - mnew) : 0.0f;
            lrun[i] = lrun[i] * alpha + warp_sum(pj);
#pragma unroll
            for (int c = 0; c < DPL; ++c) o[i][c] *= alpha;
            for (int j = 0; j < kTile; ++j) {
                const float pv = __shfl_sync(0xffffffffu, pj, j);
#pragma unroll
                for (int c = 0; c < DPL; ++c) {
                    const int col = lane + 32 * c;
                    if (col < d) o[i][c] = fmaf(pv, Vs[j * d + col], o[i][c]);
                }
            }
            mrun[i] = mnew;
        }
    }
    // partial result of this split
#pragma unroll
    for (int i = 0; i < HPW; ++i) {
        const int h = warp + 8 * i;
        if (h >= H) break;
        const int64_t base = ((int64_t)r * S + split) * H + h;
        const float inv = lrun[i] > 0.0f ? 1.0f / lrun[i] : 0.0f;
#pragma unroll
        for (int c = 0; c < DPL; ++c) {
            const int col = lane + 32 * c;
            if (col < d) o_part[base * d + col] = o[i][c] * inv;
        }
        if (lane == 0) lse_part[base] = lrun[i] > 0.0f ? mrun[i] + logf(lrun[i]) : -INFINITY;
    }
}

// One warp per (query, head): lanes first turn the S partial log-sum-exps into merge weights
// (max-subtracted, fixed order), then stream the S partial outputs with 16-byte loads, four
// splits in flight at a time.
constexpr int kMergeWarps = 8;

template <typename T>
__global__ void __launch_bounds__(32 * kMergeWarps) merge_kernel(int R, int S, int H, int d,
                                                                 const float* __restrict__ o_part,
                                                                 const float* __restrict__ lse_part,
                                                                 T* __restrict__ out, float* __restrict__ lse_out) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    if (gw >= (int64_t)R * H) return;
    const int r = (int)(gw / H), h = (int)(gw % H);
    const float* lp = lse_part + (int64_t)r * S * H + h;
    const float* op0 = o_part + ((int64_t)r * S * H + h) * d;
    float mx = -INFINITY, tot = 0.0f;
    if (S <= 32) {
        // split s's lse and weight live in lane s; slots without keys (lse = -inf) get weight 0
        // and their (unwritten) partial output is never used
        const float ls = lane < S ? __ldg(lp + (int64_t)lane * H) : -INFINITY;
        mx = warp_max(ls);
        const float e = (ls == -INFINITY || mx == -INFINITY) ? 0.0f : expf(ls - mx);
        tot = warp_sum(e);
        const float wl = tot > 0.0f ? e / tot : 0.0f;
        for (int c0 = lane * 4; c0 < d; c0 += 128) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int s0 = 0; s0 < S; s0 += 4) {
                float4 o[4];
                float ws[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    ws[u] = __shfl_sync(0xffffffffu, wl, (s0 + u) & 31);
                    ws[u] = s0 + u < S ? ws[u] : 0.0f;
                    o[u] = ws[u] != 0.0f ? __ldg(reinterpret_cast<const float4*>(op0 + (int64_t)(s0 + u) * H * d + c0))
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    acc.x = fmaf(ws[u], o[u].x, acc.x);
                    acc.y = fmaf(ws[u], o[u].y, acc.y);
                    acc.z = fmaf(ws[u], o[u].z, acc.z);
                    acc.w = fmaf(ws[u], o[u].w, acc.w);
                }
            }
            T* op = out + ((int64_t)r * H + h) * d + c0;
            from_f32(op[0], acc.x);
            from_f32(op[1], acc.y);
            from_f32(op[2], acc.z);
            from_f32(op[3], acc.w);
        }
    } else {
        for (int s = lane; s < S; s += 32) mx = fmaxf(mx, __ldg(lp + (int64_t)s * H));
        mx = warp_max(mx);
        for (int s = lane; s < S; s += 32) {
            const float ls = __ldg(lp + (int64_t)s * H);
            tot += (ls == -INFINITY || mx == -INFINITY) ? 0.0f : expf(ls - mx);
        }
        tot = warp_sum(tot);
        const float inv = tot > 0.0f ? 1.0f / tot : 0.0f;
        for (int c0 = lane * 4; c0 < d; c0 += 128) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int s = 0; s < S; ++s) {
                const float ls = __ldg(lp + (int64_t)s * H);
                if (ls == -INFINITY) continue;
                const float e = expf(ls - mx) * inv;
                const float4 o = __ldg(reinterpret_cast<const float4*>(op0 + (int64_t)s * H * d + c0));
                acc.x = fmaf(e, o.x, acc.x);
                acc.y = fmaf(e, o.y, acc.y);
                acc.z = fmaf(e, o.z, acc.z);
                acc.w = fmaf(e, o.w, acc.w);
            }
            T* op = out + ((int64_t)r * H + h) * d + c0;
            from_f32(op[0], acc.x);
            from_f32(op[1], acc.y);
            from_f32(op[2], acc.z);
            from_f32(op[3], acc.w);
        }
    }
    if (lane == 0 && lse_out) lse_out[(int64_t)r * H + h] = tot > 0.0f ? mx + logf(tot) : -INFINITY;
}

template <typename T, int HPW, int DPL>
cudaError_t launch_split(const AttendArgs& a, int S, int kps, float* o_part, float* lse_part, unsigned* err,
                         cudaStream_t st) {
    const size_t smem = (size_t)(a.H * a.d + kTile * (a.d + 1) + kTile * a.d) * 4;
    auto kern = attend_split_kernel<T, HPW, DPL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)S, (unsigned)(a.B * a.T));
    (void)launch_pdl(kern, dim3(grid), dim3(256), smem, st, a, kps, o_part, lse_part, err);
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_generic(const AttendArgs& a, int S, int kps, float* o_part, float* lse_part, unsigned* err,
                             cudaStream_t st) {
    const int hpw = (a.H + 7) / 8;
    if (a.d <= 64) {
        if (hpw <= 1) return launch_split<T, 1, 2>(a, S, kps, o_part, lse_part, err, st);
        if (hpw <= 2) return launch_split<T, 2, 2>(a, S, kps, o_part, lse_part, err, st);
        if (hpw <= 4) return launch_split<T, 4, 2>(a, S, kps, o_part, lse_part, err, st);
        return launch_split<T, 8, 2>(a, S, kps, o_part, lse_part, err, st);
    }
    if (hpw <= 1) return launch_split<T, 1, 4>(a, S, kps, o_part, lse_part, err, st);
    if (hpw <= 2) return launch_split<T, 2, 4>(a, S, kps, o_part, lse_part, err, st);
    if (hpw <= 4) return launch_split<T, 4, 4>(a, S, kps, o_part, lse_part, err, st);
    return launch_split<T, 8, 4>(a, S, kps, o_part, lse_part, err, st);
}

}  // namespace

SplitPlan plan_splits(int R, int64_t total_max, int splits_req) {
    // Keys per split are whole 128-key tiles.  Automatic plan: about two partial results per SM
    // over all query rows (at most 16 per row): the tensor-core kernel balances the tiles of few
    // rows over all SMs and needs spare partial slots for that; many rows get one split each.
    SplitPlan sp;
    total_max = std::max<int64_t>(total_max, 1);
    const int64_t tiles = cdiv(total_max, 128);
    int64_t s0 = splits_req > 0 ? splits_req
                                : std::min<int64_t>(16, std::max<int64_t>(1, cdiv(2 * (int64_t)num_sms(), std::max(R, 1))));
    s0 = std::min(s0, tiles);
    const int64_t kps = cdiv(tiles, s0) * 128;
    sp.kps = (int)kps;
    sp.S = (int)cdiv(total_max, kps);
    return sp;
}

size_t attend_workspace_bytes(int R, int H, int d, const SplitPlan& sp) {
    return kRowCounterBytes + align256((size_t)R * sp.S * H * d * 4) + align256((size_t)R * sp.S * H * 4);
}

csahca_status attend_run(const AttendArgs& a, int splits_req, void* workspace, size_t ws_bytes,
                         cudaStream_t st) {
    const int R = a.B * a.T;
    const SplitPlan sp = plan_splits(R, a.total_max, splits_req);
    if (!workspace || !aligned(workspace, 256) || ws_bytes < attend_workspace_bytes(R, a.H, a.d, sp))
        return CSAHCA_ERR_WORKSPACE;
    unsigned* row_cnt = static_cast<unsigned*>(workspace);
    float* o_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + kRowCounterBytes);
    float* lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + kRowCounterBytes +
                                               align256((size_t)R * sp.S * a.H * a.d * 4));
    unsigned* err = err_word();
    if (!err) return CSAHCA_ERR_CUDA;
    cudaError_t e;
    if (attend_tc_supported(a)) {
        e = attend_tc_launch(a, sp.S, sp.kps, o_part, lse_part, row_cnt, err, st);
        count_launch();
        if (e != cudaSuccess) return CSAHCA_ERR_CUDA;
        if (attend_tc_merges(a, sp.S)) {
            CSAHCA_CHECK_LAUNCH();
            return CSAHCA_OK;
        }
    } else {
        if (a.dtype == CSAHCA_F32) {
            e = dispatch_generic<float>(a, sp.S, sp.kps, o_part, lse_part, err, st);
        } else {
            e = dispatch_generic<__nv_bfloat16>(a, sp.S, sp.kps, o_part, lse_part, err, st);
        }
        count_launch();
        if (e != cudaSuccess) return CSAHCA_ERR_CUDA;
    }
    const unsigned mgrid = (unsigned)cdiv((int64_t)R * a.H, kMergeWarps);
    if (a.dtype == CSAHCA_F32)
        (void)launch_pdl(merge_kernel<float>, dim3(mgrid), dim3(32 * kMergeWarps), 0, st, R, sp.S, a.H, a.d, o_part, lse_part, (float*)a.out,
                                                                a.lse);
    else
        (void)launch_pdl(merge_kernel<__nv_bfloat16>, dim3(mgrid), dim3(32 * kMergeWarps), 0, st, R, sp.S, a.H, a.d, o_part, lse_part,
                                                                        (__nv_bfloat16*)a.out, a.lse);
    count_launch();
    CSAHCA_CHECK_LAUNCH();
    return CSAHCA_OK;
}

csahca_status attend_validate(const AttendArgs& a) {
    CSAHCA_REQUIRE(a.q && a.ck && a.cv && a.q_pos && a.out);
    CSAHCA_REQUIRE(a.dtype == CSAHCA_F32 || a.dtype == CSAHCA_BF16 || a.dtype == CSAHCA_KV_FP8);
    CSAHCA_REQUIRE(a.B >= 1 && a.T >= 1 && (int64_t)a.B * a.T <= 65535 && a.H >= 1 && a.d >= 8);
    CSAHCA_REQUIRE(a.d % 8 == 0 && a.Ncap >= 1 && a.W >= 0);
    if (a.W > 0) CSAHCA_REQUIRE(a.ring_k && a.ring_v && a.ring_cap >= 1);
    if (!a.chunk_k) CSAHCA_REQUIRE(a.W <= a.ring_cap || a.W == 0);
    else CSAHCA_REQUIRE(a.chunk_v && a.chunk_pos0 && a.chunk_stride >= 1);
    if (a.is_csa) CSAHCA_REQUIRE(a.k >= 0 && (a.idx || a.k == 0));   // k = 0: the window alone
    else CSAHCA_REQUIRE(a.m >= 1);
    const size_t al = (a.dtype == CSAHCA_F32) ? 32 : 16;
    CSAHCA_REQUIRE(aligned(a.q, al) && aligned(a.ck, al) && aligned(a.cv, al));
    if (a.ring_k) CSAHCA_REQUIRE(aligned(a.ring_k, al) && aligned(a.ring_v, al));
    if (a.chunk_k) CSAHCA_REQUIRE(aligned(a.chunk_k, al) && aligned(a.chunk_v, al));
    if (attend_tc_supported(a)) return CSAHCA_OK;
    if (a.dtype == CSAHCA_KV_FP8) return CSAHCA_ERR_UNSUPPORTED;      // FP8 caches: tensor-core path only
    if (!(a.d == 64 || a.d == 128) || a.H > 64) return CSAHCA_ERR_UNSUPPORTED;
    return CSAHCA_OK;
}

}  // namespace csahca

using namespace csahca;

extern "C" {

size_t csa_attend_workspace(int B, int T, int H, int d, int k, int W) {
    if (B <= 0 || T <= 0 || H <= 0 || d <= 0 || k < 0 || W < 0) return 0;
    const SplitPlan sp = plan_splits(B * T, tile_space_keys(k, W), 0);
    return attend_workspace_bytes(B * T, H, d, sp);
}

size_t hca_attend_workspace(int B, int T, int H, int d, int64_t Ncap, int W, int splits) {
    if (B <= 0 || T <= 0 || H <= 0 || d <= 0 || Ncap < 0 || W < 0) return 0;
    const SplitPlan sp = plan_splits(B * T, tile_space_keys(Ncap, W), splits);
    return attend_workspace_bytes(B * T, H, d, sp);
}

csahca_status csa_attend(const void* q, int B, int T, int H, int d, float scale, const void* ck, const void* cv,
                         int64_t Ncap, const int32_t* idx, int k, const void* ring_k, const void* ring_v, int ring_cap,
                         int W, const void* chunk_k, const void* chunk_v, const int64_t* chunk_pos0,
                         int64_t chunk_stride, const int64_t* q_pos, csahca_dtype dtype, void* out, float* lse,
                         void* workspace, size_t ws_bytes, csahca_stream_t stream) {
    AttendArgs a{};
    a.is_csa = true;
    a.q = q; a.B = B; a.T = T; a.H = H; a.d = d; a.scale = scale; a.ck = ck; a.cv = cv; a.Ncap = Ncap;
    a.idx = idx; a.k = k; a.m = 1; a.ring_k = ring_k; a.ring_v = ring_v; a.ring_cap = ring_cap; a.W = W;
    a.chunk_k = chunk_k; a.chunk_v = chunk_v; a.chunk_pos0 = chunk_pos0; a.chunk_stride = chunk_stride;
    a.q_pos = q_pos; a.dtype = dtype; a.out = out; a.lse = lse;
    a.total_max = tile_space_keys(k, W);
    const csahca_status v = attend_validate(a);
    if (v != CSAHCA_OK) return v;
    return attend_run(a, 0, workspace, ws_bytes, (cudaStream_t)stream);
}

csahca_status hca_attend(const void* q, int B, int T, int H, int d, float scale, const void* ck, const void* cv,
                         int64_t Ncap, int m, const void* ring_k, const void* ring_v, int ring_cap, int W,
                         const void* chunk_k, const void* chunk_v, const int64_t* chunk_pos0, int64_t chunk_stride,
                         const int64_t* q_pos, int splits, csahca_dtype dtype, void* out, float* lse,
                         void* workspace, size_t ws_bytes, csahca_stream_t stream) {
    AttendArgs a{};
    a.is_csa = false;
    a.q = q; a.B = B; a.T = T; a.H = H; a.d = d; a.scale = scale; a.ck = ck; a.cv = cv; a.Ncap = Ncap;
    a.idx = nullptr; a.k = 0; a.m = m; a.ring_k = ring_k; a.ring_v = ring_v; a.ring_cap = ring_cap; a.W = W;
    a.chunk_k = chunk_k; a.chunk_v = chunk_v; a.chunk_pos0 = chunk_pos0; a.chunk_stride = chunk_stride;
    a.q_pos = q_pos; a.dtype = dtype; a.out = out; a.lse = lse;
    a.total_max = tile_space_keys(Ncap, W);
    if (splits < 0) return CSAHCA_ERR_INVALID_ARG;
    const csahca_status v = attend_validate(a);
    if (v != CSAHCA_OK) return v;
    return attend_run(a, splits, workspace, ws_bytes, (cudaStream_t)stream);
}

}  // extern "C"
