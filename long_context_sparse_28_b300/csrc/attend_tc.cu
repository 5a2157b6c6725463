// Tensor-core split attention for bf16 and d = 128 (CSA: selected entries + window; HCA: every
// visible entry + window), sm_103a tcgen05 + TMEM.
//
// All H query heads of a query share one KV stream (honbul.tistory.com/221 "CSA"/"HCA";
// pogovet.com detail 4), so one tile of 128 keys against all heads is a dense contraction:
//   S^T[128 keys x H]  = K_tile[128 x 128] . Q^T          (A = K, K-major; B = Q, K-major)
//   O^T[128 dims x H] += V_tile^T[128 x 128] . P[128 x H]  (A = V, MN-major; B = P, MN-major)
// Keys are the M dimension, so every thread owns one key row of S^T (tcgen05.ld 32x32b) and
// the V tile is used exactly as loaded (no transpose).  Softmax per head runs over the
// columns: the per-tile column maximum is a warp transpose-reduction plus 4-way smem merge;
// the running maximum is raised lazily (only when it grows by more than 2^8), and only then is
// the O^T accumulator in TMEM rescaled.  Row sums are kept per thread and reduced once at the
// end.  Each CTA is persistent over (query, key-split) items; K/V tiles are gathered row by
// row with cp.async into 128-byte-swizzled shared memory, double-buffered, zero-filled for
// empty slots.  Partial results (o normalised, lse) go to the split workspace and are merged
// by the shared merge kernel.
#include "attend.cuh"
#include "tc_ptx.cuh"

namespace csahca {
namespace {

using namespace tc;

constexpr int kKeys = 128;           // keys per tile (MMA M)
constexpr int kD = 128;              // head dim
constexpr int kStages = 2;
constexpr uint32_t kHalf = kKeys * 128;   // one 64-column half of a [128][128] bf16 tile: 16 KB
constexpr float kRescaleThreshold = 8.0f; // log2 units

template <int H>
struct Smem {
    static constexpr uint32_t q = 0;                                  // 2 halves x [H][128 B]
    static constexpr uint32_t q_half = H * 128;
    static constexpr uint32_t p = 2 * q_half;                         // [128 keys][H bf16] (64-head regions)
    static constexpr uint32_t p_region = kKeys * 128;
    static constexpr uint32_t p_bytes = ((H + 63) / 64) * p_region;
    static constexpr uint32_t kv = (p + p_bytes + 1023) / 1024 * 1024;
    static constexpr uint32_t stage = 4 * kHalf;                      // K halves, then V halves
    static constexpr uint32_t total = kv + kStages * stage;
};

struct Misc {
    uint64_t bar_s, bar_o;
    uint32_t tmem_base;
    int flag;
    float red[4][128];
    float mrun[128];
    float alpha[128];
    float linv[128];
    const __nv_bfloat16* rowk[kStages][kKeys];
    const __nv_bfloat16* rowv[kStages][kKeys];
    unsigned char valid[kStages][kKeys];
};

// Column (head) reduction of NV = H values per thread across the 32 lanes of a warp: after the
// call lane l holds the result for heads [l*H/32, (l+1)*H/32) in v[0 .. H/32).
template <int H, bool MAX>
__device__ __forceinline__ void warp_col_reduce(float (&v)[H]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 16, n = H; off >= 1; off >>= 1) {
        const int half = n / 2;
        if (half < H / 32) break;
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int j = 0; j < H / 2; ++j) {
            if (j < half) {
                const float send = up ? v[j] : v[j + half];
                const float keep = up ? v[j + half] : v[j];
                const float recv = __shfl_xor_sync(0xffffffffu, send, off);
                v[j] = MAX ? fmaxf(keep, recv) : keep + recv;
            }
        }
        n = half;
    }
}

template <int H>
__global__ void __launch_bounds__(128, 1) attend_tc_kernel(AttendArgs a, int S, int kps, float* __restrict__ o_part,
                                                           float* __restrict__ lse_part, unsigned* err) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~uintptr_t(1023));
    __shared__ Misc ms;
    using L = Smem<H>;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    constexpr uint32_t kCols = (2 * H <= 32) ? 32 : (2 * H <= 64 ? 64 : (2 * H <= 128 ? 128 : 256));

    if (warp == 0) {
        tmem_alloc(&ms.tmem_base, kCols);
        tmem_relinquish();
    }
    if (t == 0) {
        mbar_init(&ms.bar_s, 1);
        mbar_init(&ms.bar_o, 1);
        fence_mbar_init();
        ms.flag = 0;
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = ms.tmem_base;
    const uint32_t t_s = tmem, t_o = tmem + H;
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    const uint32_t sbase = smem_u32(sm);
    uint32_t ph_s = 0, ph_o = 0;
    const float c_log2 = a.scale * 1.4426950408889634f;
    const uint64_t pol_stream = l2_policy_evict_first();     // K/V rows are read once per step
    const uint32_t id_qk = idesc_f16(128, H, 1, 0, 0);
    const uint32_t id_pv = idesc_f16(128, H, 1, 1, 1);

    const int R = a.B * a.T;
    const int items = R * S;
    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const int r = item / S, split = item % S;
        const int b = r / a.T;
        const int64_t p = a.q_pos[r];
        const KeyList kl = key_list(a, r, b, p);
        const int64_t k0 = (int64_t)split * kps;
        const int64_t k1 = kl.total < k0 + kps ? kl.total : k0 + kps;
        const int ntiles = k1 > k0 ? (int)((k1 - k0 + kKeys - 1) / kKeys) : 0;
        const int64_t obase = ((int64_t)r * S + split) * H;

        if (t < H) ms.mrun[t] = -INFINITY;
        // queue Q (row r) for this item, 16-byte chunks into the swizzled K-major layout
        const __nv_bfloat16* qr = static_cast<const __nv_bfloat16*>(a.q) + (int64_t)r * H * kD;
        for (int c = t; c < H * 16; c += 128) {
            const int h = c >> 4, cc = c & 15;
            cp_async16(sbase + L::q + (cc >> 3) * L::q_half + sw128(h, cc & 7), qr + h * kD + cc * 8, 16);
        }

        // gathers tile `tile` of this item into stage `st`
        auto issue_tile = [&](int tile, int st) {
            const int64_t key = k0 + (int64_t)tile * kKeys + t;
            const __nv_bfloat16* kp = nullptr;
            const __nv_bfloat16* vp = nullptr;
            if (key < k1) key_rows<__nv_bfloat16>(a, kl, r, b, p, key, &kp, &vp, err);
            ms.rowk[st][t] = kp;
            ms.rowv[st][t] = vp;
            ms.valid[st][t] = kp != nullptr;
            __syncthreads();
            const uint32_t stb = sbase + L::kv + st * L::stage;
            for (int row = warp; row < kKeys; row += 4) {
                const __nv_bfloat16* src = (lane < 16) ? ms.rowk[st][row] : ms.rowv[st][row];
                const int cc = lane & 15;
                const uint32_t dst = stb + (lane < 16 ? 0 : 2 * kHalf) + (cc >> 3) * kHalf + sw128(row, cc & 7);
                if (src) cp_async16_hint(dst, src + cc * 8, 16, pol_stream);
                else cp_async16(dst, qr, 0);                 // zero fill (no bytes read)
            }
        };

        float lsum[H];
#pragma unroll
        for (int h = 0; h < H; ++h) lsum[h] = 0.0f;

        if (ntiles > 0) issue_tile(0, 0);
        cp_async_commit();

        for (int i = 0; i < ntiles; ++i) {
            const int st = i % kStages;
            if (i > 0) {                                     // PV(i-1) done: frees P, O and stage st^1
                mbar_wait(&ms.bar_o, ph_o, err);
                ph_o ^= 1;
                fence_after_sync();
            }
            if (i + 1 < ntiles) issue_tile(i + 1, (i + 1) % kStages);
            cp_async_commit();
            cp_async_wait<1>();
            fence_proxy_async();
            __syncthreads();
            // ---- S^T = K . Q^T
            if (t == 0) {
                fence_after_sync();
                const uint32_t kb = sbase + L::kv + st * L::stage;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint64_t ad = smem_desc(kb + (j >> 2) * kHalf + (j & 3) * 32, 16, 1024);
                    const uint64_t bd = smem_desc(sbase + L::q + (j >> 2) * L::q_half + (j & 3) * 32, 16, 1024);
                    mma_ss(t_s, ad, bd, id_qk, j > 0);
                }
                mma_commit(&ms.bar_s);
            }
            mbar_wait(&ms.bar_s, ph_s, err);
            ph_s ^= 1;
            fence_after_sync();
            const bool valid = ms.valid[st][t] != 0;
            // ---- column maxima (the S tile stays in TMEM and is read again below)
            {
                float v[H];
#pragma unroll
                for (int c0 = 0; c0 < H; c0 += 16) {
                    uint32_t rr[16];
                    tmem_ld16(t_s + lane_off + c0, rr);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; ++k) v[c0 + k] = valid ? __uint_as_float(rr[k]) * c_log2 : -INFINITY;
                }
                warp_col_reduce<H, true>(v);
#pragma unroll
                for (int j = 0; j < H / 32; ++j) ms.red[warp][lane * (H / 32) + j] = v[j];
            }
            __syncthreads();
            if (t < H) {
                const float tmax = fmaxf(fmaxf(ms.red[0][t], ms.red[1][t]), fmaxf(ms.red[2][t], ms.red[3][t]));
                const float mo = ms.mrun[t];
                float al = 1.0f;
                if (tmax > mo + kRescaleThreshold || (mo == -INFINITY && tmax != -INFINITY)) {
                    al = (mo == -INFINITY) ? 0.0f : exp2f(mo - tmax);
                    ms.mrun[t] = tmax;
                    ms.flag = 1;
                }
                ms.alpha[t] = al;
            }
            __syncthreads();
            const bool rescale = ms.flag != 0;
            // ---- P = exp2(s - m), row sums, P tile (MN-major: [key][head]), 16 heads at a time
#pragma unroll
            for (int c0 = 0; c0 < H; c0 += 16) {
                uint32_t rr[16];
                tmem_ld16(t_s + lane_off + c0, rr);
                tmem_wait_ld();
                uint32_t pk[8];
#pragma unroll
                for (int k = 0; k < 16; k += 2) {
                    const int h = c0 + k;
                    const float s0 = valid ? __uint_as_float(rr[k]) * c_log2 : -INFINITY;
                    const float s1 = valid ? __uint_as_float(rr[k + 1]) * c_log2 : -INFINITY;
                    const float m0 = ms.mrun[h], m1 = ms.mrun[h + 1];
                    const float p0 = (m0 == -INFINITY) ? 0.0f : exp2f(s0 - m0);
                    const float p1 = (m1 == -INFINITY) ? 0.0f : exp2f(s1 - m1);
                    lsum[h] = lsum[h] * ms.alpha[h] + p0;
                    lsum[h + 1] = lsum[h + 1] * ms.alpha[h + 1] + p1;
                    pk[k / 2] = pack_bf16x2(p0, p1);
                }
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int chunk = c0 / 8 + c;
                    const uint32_t dst = sbase + L::p + (chunk >> 3) * L::p_region + sw128(t, chunk & 7);
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(pk[4 * c]),
                                 "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                                 : "memory");
                }
            }
            // ---- rescale the O^T accumulator (lane = dim) when some running maximum moved
            if (rescale && i > 0) {
#pragma unroll
                for (int c0 = 0; c0 < H; c0 += 16) {
                    uint32_t rr[16];
                    tmem_ld16(t_o + lane_off + c0, rr);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; ++k) rr[k] = __float_as_uint(__uint_as_float(rr[k]) * ms.alpha[c0 + k]);
                    tmem_st16(t_o + lane_off + c0, rr);
                }
                tmem_wait_st();
            }
            fence_proxy_async();
            fence_before_sync();
            __syncthreads();
            if (t == 0) ms.flag = 0;
            // ---- O^T += V^T . P
            if (t == 0) {
                fence_after_sync();
                const uint32_t vb = sbase + L::kv + st * L::stage + 2 * kHalf;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint64_t ad = smem_desc(vb + j * 2048, kHalf, 1024);
                    const uint64_t bd = smem_desc(sbase + L::p + j * 2048, L::p_region, 1024);
                    mma_ss(t_o, ad, bd, id_pv, (i > 0 || j > 0) ? 1u : 0u);
                }
                mma_commit(&ms.bar_o);
            }
        }
        if (ntiles > 0) {
            mbar_wait(&ms.bar_o, ph_o, err);
            ph_o ^= 1;
            fence_after_sync();
        }
        cp_async_wait<0>();
        // ---- row sums across the 128 keys, partial lse, normalised partial output
        warp_col_reduce<H, false>(lsum);
#pragma unroll
        for (int j = 0; j < H / 32; ++j) ms.red[warp][lane * (H / 32) + j] = lsum[j];
        __syncthreads();
        if (t < H) {
            const float l = ms.red[0][t] + ms.red[1][t] + ms.red[2][t] + ms.red[3][t];
            const float m = ms.mrun[t];
            const bool any = (l > 0.0f) && (m != -INFINITY);
            ms.linv[t] = any ? 1.0f / l : 0.0f;
            lse_part[obase + t] = any ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
        }
        __syncthreads();
        if (ntiles > 0) {
#pragma unroll
            for (int c0 = 0; c0 < H; c0 += 16) {
                uint32_t rr[16];
                tmem_ld16(t_o + lane_off + c0, rr);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    o_part[(obase + c0 + k) * kD + t] = __uint_as_float(rr[k]) * ms.linv[c0 + k];
            }
        } else {
            for (int h = 0; h < H; ++h) o_part[(obase + h) * kD + t] = 0.0f;
        }
        fence_before_sync();
        __syncthreads();
    }
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, kCols);
}

template <int H>
cudaError_t launch_tc(const AttendArgs& a, int S, int kps, float* o_part, float* lse_part, unsigned* err,
                      cudaStream_t st) {
    const size_t smem = Smem<H>::total + 1024;
    auto kern = attend_tc_kernel<H>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int items = a.B * a.T * S;
    const int grid = items < num_sms() ? items : num_sms();
    kern<<<grid, 128, smem, st>>>(a, S, kps, o_part, lse_part, err);
    return cudaGetLastError();
}

}  // namespace

bool attend_tc_supported(const AttendArgs& a) {
    return a.dtype == CSAHCA_BF16 && a.d == 128 && (a.H == 32 || a.H == 64);
}

cudaError_t attend_tc_launch(const AttendArgs& a, int S, int kps, float* o_part, float* lse_part, unsigned* err,
                             cudaStream_t st) {
    switch (a.H) {
        case 32: return launch_tc<32>(a, S, kps, o_part, lse_part, err, st);
        case 64: return launch_tc<64>(a, S, kps, o_part, lse_part, err, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace csahca
