// Tensor-core lightning-indexer scores for low-precision keys (e4m3 + row scale, e2m1 + UE8M0
// per 32 values), d_I = 64, one query row per item (decode).
//
// I(t,s) = sum_h w[t,h] * ReLU(q[t,h] . khat_s)  (honbul.tistory.com/221 "CSA"; pogovet.com
// DeepSeek-V4 article, detail 4 (FP4 lightning indexer) and detail 5).
//
// Per 128-key tile:  D[128 keys x H_I] = A[128 keys x 64] . Q^T  on tcgen05 (kind::f16):
//   * key codes stream through shared memory with 1-D bulk async copies (an NS-stage ring fed by
//     one producer thread, mbarrier transaction counts);
//   * each thread owns one key row: it decodes its 64 codes exactly to f16 with the hardware
//     e4m3/e2m1 -> f16x2 conversions (every code value is a small integer times a power of two)
//     and writes the row into TMEM, where it is the MMA's A operand (no shared-memory round trip);
//   * the query row is the B operand in shared memory (K-major, 128-byte swizzle): bf16 queries
//     are scaled per head by a power of two 2^e_h into f16 range, exactly; the factor 2^-e_h is
//     folded into the head weight w';
//   * the per-row (e4m3) or per-32 (e2m1, two accumulators) key scales are applied to the fp32
//     accumulators in the epilogue: score = sum_h w'_h ReLU(sum_blocks s_block D_block[h]).
// The MMA of tile g overlaps the epilogue of tile g-1 (two A and two D buffers in TMEM).
// CTAs are persistent over (row, chunk of 8 tiles) items and keep the copy ring running
// across items.  Only the rounding of the fp32 accumulation differs from exact arithmetic.
#include "common.cuh"
#include "tc_ptx.cuh"
#include "quant.cuh"

#include <algorithm>
#include <cstddef>

namespace csahca {
namespace {

using namespace tc;

constexpr int kKeys = 128;
constexpr int kDI = 64;
constexpr int kChunkTiles = 8;

template <int FMT, int HI>
struct IdxCfg {
    static constexpr int row_bytes = FMT == CSAHCA_E4M3_ROWSCALE ? 64 : 32;
    static constexpr int scale_bytes = FMT == CSAHCA_E4M3_ROWSCALE ? 4 : 2;
    static constexpr int tile_bytes = kKeys * row_bytes;
    static constexpr int stages = 4;
    static constexpr int nacc = FMT == CSAHCA_E2M1_UE8M0 ? 2 : 1;
    static constexpr uint32_t a_cols = 32;                 // 64 16-bit values per key row
    static constexpr uint32_t d_cols = nacc * HI;
    static constexpr uint32_t need_cols = a_cols + d_cols;
    static constexpr uint32_t tmem_cols = need_cols <= 32 ? 32 : need_cols <= 64 ? 64 : need_cols <= 128 ? 128
                                        : need_cols <= 256 ? 256 : 512;
    static constexpr int tmem_ctas = 512 / tmem_cols;
    // shared memory: code stages | scale stages | q buffers (2 x HI rows x 128 B)
    static constexpr uint32_t off_scale = stages * tile_bytes;
    static constexpr uint32_t off_q = (off_scale + stages * kKeys * scale_bytes + 1023) / 1024 * 1024;
    static constexpr uint32_t q_buf = HI * 128;
    static constexpr uint32_t total = off_q + 2 * q_buf;
};

struct IdxMisc {
    alignas(16) float wq[2][64];        // read as float4
    alignas(16) uint32_t hist[4096];    // top-12-bit histogram of the current item's scores (fused top-k pass)
    unsigned amax[2][64];
    uint64_t full[4];
    uint64_t mma_done;
    uint32_t tmem_base;
};
static_assert(offsetof(IdxMisc, wq) % 16 == 0, "wq is read with 16-byte loads");

struct Tile {          // one 128-key tile of one query row
    int item;
    int r;
    int64_t s0;        // first key of the tile
    int64_t n;         // visible keys of the row
};

// Walks this CTA's items (row r = item % R, chunk c = item / R) tile by tile, skipping empty ones.
struct Cursor {
    int item, items, stride, R;
    int64_t Ncap;
    int m;
    const int64_t* q_pos;
    Tile cur;
    int64_t s_end;
    bool valid;

    __device__ void start(int first, int nitems, int step, int rows, int64_t ncap, int mm, const int64_t* qp) {
        item = first - step;
        items = nitems;
        stride = step;
        R = rows;
        Ncap = ncap;
        m = mm;
        q_pos = qp;
        valid = true;
        next_item();
    }
    __device__ void next_item() {
        for (;;) {
            item += stride;
            if (item >= items) {
                valid = false;
                return;
            }
            const int r = item % R, c = item / R;
            const int64_t p = q_pos[r];
            int64_t n = (p >= 0) ? (p + 1) / m : 0;
            n = n < Ncap ? n : Ncap;
            const int64_t s0 = (int64_t)c * kChunkTiles * kKeys;
            if (s0 < n) {
                cur.item = item;
                cur.r = r;
                cur.s0 = s0;
                cur.n = n;
                const int64_t e = s0 + (int64_t)kChunkTiles * kKeys;
                s_end = e < n ? e : n;
                return;
            }
        }
    }
    __device__ void advance() {
        cur.s0 += kKeys;
        if (cur.s0 >= s_end) next_item();
    }
};

template <int FMT, int HI>
__global__ void __launch_bounds__(128) index_tc_kernel(const __nv_bfloat16* __restrict__ q_idx,
                                                       const float* __restrict__ w,
                                                       const uint8_t* __restrict__ k_codes,
                                                       const uint8_t* __restrict__ k_scale, int T,
                                                       const int64_t* __restrict__ q_pos, int64_t Ncap, int m,
                                                       int R, float* __restrict__ S, uint32_t* __restrict__ hist1,
                                                       unsigned* err) {
    using C = IdxCfg<FMT, HI>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~uintptr_t(1023));
    __shared__ IdxMisc ms;
    const int t = threadIdx.x, warp = t >> 5;
    const uint32_t sbase = smem_u32(sm);

    if (warp == 0) {
        tmem_alloc(&ms.tmem_base, C::tmem_cols);
        tmem_relinquish();
    }
    if (t == 0) {
        for (int s = 0; s < C::stages; ++s) mbar_init(&ms.full[s], 1);
        mbar_init(&ms.mma_done, 1);
        fence_mbar_init();
    }
    for (int i = t; i < 4096; i += 128) ms.hist[i] = 0u;
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = ms.tmem_base;
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    const int items = R * (int)cdiv(Ncap, (int64_t)kChunkTiles * kKeys);

    // key codes are read once per step: keep them from evicting the scores the top-k re-reads
    const uint64_t pol_stream = l2_policy_evict_first();
    const uint64_t pol_keep = l2_policy_evict_last();
    // producer (thread 0): issues the bulk copies of tile `pt` into stage pg % NS
    Cursor prod;
    int64_t pg = 0;
    auto produce = [&]() {
        const int st = (int)(pg % C::stages);
        const Tile& x = prod.cur;
        const int b = x.r / T;
        const int64_t rows = (x.n - x.s0) < kKeys ? (x.n - x.s0) : kKeys;
        const int64_t srows = ((rows + 7) / 8) * 8;                 // stays within Ncap (Ncap % 8 == 0)
        const int64_t row0 = (int64_t)b * Ncap + x.s0;
        const uint32_t cb = (uint32_t)(rows * C::row_bytes);
        const uint32_t sb = (uint32_t)(srows * C::scale_bytes);
        mbar_arrive_expect_tx(&ms.full[st], cb + sb);
        bulk_g2s_hint(sbase + st * C::tile_bytes, k_codes + row0 * C::row_bytes, cb, &ms.full[st], pol_stream);
        bulk_g2s_hint(sbase + C::off_scale + st * kKeys * C::scale_bytes, k_scale + row0 * C::scale_bytes, sb,
                      &ms.full[st], pol_stream);
        ++pg;
        prod.advance();
    };
    if (t == 0) {
        prod.start(blockIdx.x, items, gridDim.x, R, Ncap, m, q_pos);
        for (int i = 0; i < C::stages && prod.valid; ++i) produce();
    }

    Cursor cons;
    cons.start(blockIdx.x, items, gridDim.x, R, Ncap, m, q_pos);
    int64_t g = 0;
    int qrow = -1, qbuf = 1;
    int cur_item = -1, cur_r = 0;
    uint32_t ph_mma = 0;
    const uint32_t id = idesc_f16(128, HI, 0, 0, 0);
    const uint32_t abuf = tmem;
    const uint32_t dbuf = tmem + C::a_cols;

    // adds the item's smem histogram to the row's global one and clears it
    auto flush_hist = [&](int r) {
        __syncthreads();
        uint32_t* gh = hist1 + (int64_t)r * 4096;
        for (int i = t; i < 4096; i += 128) {
            const uint32_t v = ms.hist[i];
            if (v) {
                atomicAdd(&gh[i], v);
                ms.hist[i] = 0u;
            }
        }
        __syncthreads();
    };

    while (cons.valid) {
        const Tile x = cons.cur;
        const int st = (int)(g % C::stages);
        if (hist1 != nullptr && x.item != cur_item && cur_item >= 0) flush_hist(cur_r);
        cur_item = x.item;
        cur_r = x.r;
        // ---- query row for this tile (B operand, f16 scaled per head; w' = w * 2^-e)
        if (x.r != qrow) {
            qrow = x.r;
            qbuf ^= 1;
            if (t < HI) ms.amax[qbuf][t] = 0u;
            __syncthreads();
            const __nv_bfloat16* qr = q_idx + (int64_t)qrow * HI * kDI;
            for (int c = t; c < HI * 8; c += 128) {                 // 8 chunks of 8 values per head
                const uint4 u = __ldg(reinterpret_cast<const uint4*>(qr) + c);
                const uint32_t wds[4] = {u.x, u.y, u.z, u.w};
                float amax = 0.0f;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(wds[i] << 16)),
                                             fabsf(__uint_as_float(wds[i] & 0xFFFF0000u))));
                atomicMax(&ms.amax[qbuf][c >> 3], __float_as_uint(amax));
            }
            __syncthreads();
            for (int c = t; c < HI * 8; c += 128) {
                const int h = c >> 3;
                const float amax = __uint_as_float(ms.amax[qbuf][h]);
                int ex = 0;
                if (amax > 0.0f) {
                    frexpf(amax, &ex);                              // amax in [2^(ex-1), 2^ex)
                    ex = 15 - ex;                                   // amax * 2^e in [2^14, 2^15)
                }
                const uint4 u = __ldg(reinterpret_cast<const uint4*>(qr) + c);
                const uint32_t wds[4] = {u.x, u.y, u.z, u.w};
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float lo = ldexpf(__uint_as_float(wds[i] << 16), ex);
                    const float hi = ldexpf(__uint_as_float(wds[i] & 0xFFFF0000u), ex);
                    __half2 hh = __floats2half2_rn(lo, hi);
                    o[i] = *reinterpret_cast<uint32_t*>(&hh);
                }
                const uint32_t dst = sbase + C::off_q + qbuf * C::q_buf + sw128(h, c & 7);
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(o[0]), "r"(o[1]), "r"(o[2]),
                             "r"(o[3])
                             : "memory");
                if ((c & 7) == 0) ms.wq[qbuf][h] = ldexpf(w[(int64_t)qrow * HI + h], -ex);
            }
            fence_proxy_async();
        }
        // ---- this thread's key row -> f16 -> TMEM (A operand)
        mbar_wait(&ms.full[st], (uint32_t)((g / C::stages) & 1), err);
        uint32_t a[32];
        const unsigned char* row = sm + st * C::tile_bytes + t * C::row_bytes;
        float sc0, sc1 = 0.0f;
        if (FMT == CSAHCA_E2M1_UE8M0) {
            const uint4 u0 = *reinterpret_cast<const uint4*>(row);
            const uint4 u1 = *reinterpret_cast<const uint4*>(row + 16);
            const uint32_t wds[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t o[4];
                cvt_e2m1x8_f16(wds[i], o);
                a[4 * i] = o[0]; a[4 * i + 1] = o[1]; a[4 * i + 2] = o[2]; a[4 * i + 3] = o[3];
            }
            const uint32_t e2 = *reinterpret_cast<const uint16_t*>(sm + C::off_scale + st * kKeys * 2 + t * 2);
            sc0 = ue8m0_value(e2 & 0xFFu);
            sc1 = ue8m0_value(e2 >> 8);
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 u = *reinterpret_cast<const uint4*>(row + 16 * c);
                const uint32_t wds[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t o[2];
                    cvt_e4m3x4_f16(wds[i], o);
                    a[8 * c + 2 * i] = o[0];
                    a[8 * c + 2 * i + 1] = o[1];
                }
            }
            sc0 = *reinterpret_cast<const float*>(sm + C::off_scale + st * kKeys * 4 + t * 4);
        }
        tmem_st32(abuf + lane_off, a);
        tmem_wait_st();
        fence_before_sync();
        __syncthreads();                         // stage st consumed, A written, q ready, D read
        if (t == 0) {
            if (prod.valid) produce();           // refill stage st with the tile NS steps ahead
            fence_after_sync();
            const uint32_t qb = sbase + C::off_q + qbuf * C::q_buf;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint64_t bd = smem_desc(qb + j * 32, 16, 1024);
                const uint32_t dst = (C::nacc == 2 && j >= 2) ? dbuf + HI : dbuf;
                const uint32_t acc = (C::nacc == 2) ? (uint32_t)(j & 1) : (uint32_t)(j > 0);
                mma_ts(dst, abuf + j * 8, bd, id, acc);
            }
            mma_commit(&ms.mma_done);
        }
        // ---- epilogue: score = sum_h w'_h ReLU(scaled accumulators)
        mbar_wait(&ms.mma_done, ph_mma, err);
        ph_mma ^= 1;
        fence_after_sync();
        float score = 0.0f;
        const float4* wq4 = reinterpret_cast<const float4*>(ms.wq[qbuf]);
#pragma unroll
        for (int c0 = 0; c0 < HI; c0 += 16) {
            uint32_t r0[16];
            tmem_ld16(dbuf + lane_off + c0, r0);
            float wv[16];
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const float4 q4 = wq4[c0 / 4 + k4];
                wv[4 * k4] = q4.x; wv[4 * k4 + 1] = q4.y; wv[4 * k4 + 2] = q4.z; wv[4 * k4 + 3] = q4.w;
            }
            if (C::nacc == 2) {
                uint32_t r1[16];
                tmem_ld16(dbuf + lane_off + HI + c0, r1);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float v = fmaf(sc0, __uint_as_float(r0[k]), sc1 * __uint_as_float(r1[k]));
                    score = fmaf(wv[k], fmaxf(v, 0.0f), score);
                }
            } else {
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k) score = fmaf(wv[k], fmaxf(__uint_as_float(r0[k]), 0.0f), score);
            }
        }
        if (C::nacc == 1) score *= sc0;
        const int64_t s = x.s0 + t;
        if (s < x.n) st_global_hint(S + (int64_t)x.r * Ncap + s, score, pol_keep);
        if (hist1 != nullptr) {                        // warp-aggregated histogram update
            const uint32_t bin = (s < x.n) ? (ordered_key(score) >> 20) : 0xFFFFFFFFu;
            const uint32_t peers = __match_any_sync(0xffffffffu, bin);
            if (bin != 0xFFFFFFFFu && (t & 31) == __ffs(peers) - 1) atomicAdd(&ms.hist[bin], (uint32_t)__popc(peers));
        }
        fence_before_sync();
        ++g;
        cons.advance();
    }
    if (hist1 != nullptr && cur_item >= 0) flush_hist(cur_r);
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, C::tmem_cols);
}

template <int FMT, int HI>
cudaError_t launch_index_tc(const void* q_idx, const float* w, const void* k_codes, const void* k_scale, int B,
                            int T, const int64_t* q_pos, int64_t Ncap, int m, float* S, uint32_t* hist1, unsigned* err,
                            cudaStream_t st) {
    using C = IdxCfg<FMT, HI>;
    // shared memory sized so that no more CTAs fit on an SM than TMEM can hold
    const size_t per_cta = (size_t)(228 * 1024) / (C::tmem_ctas + 1) + 1024 - sizeof(IdxMisc);
    const size_t smem = std::max<size_t>((size_t)C::total + 1024, per_cta);
    // CTAs per SM: limited by shared memory (228 KB per SM, 1 KB reserved per CTA) and TMEM
    const size_t per_sm_cta = smem + sizeof(IdxMisc) + 1024;
    const int occ = std::max(1, std::min((int)((size_t)(228 * 1024) / per_sm_cta), C::tmem_ctas));
    auto kern = index_tc_kernel<FMT, HI>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int R = B * T;
    const int64_t items = (int64_t)R * cdiv(Ncap, (int64_t)kChunkTiles * kKeys);
    const int grid = (int)std::min<int64_t>(items, (int64_t)num_sms() * occ);
    kern<<<grid, 128, smem, st>>>(static_cast<const __nv_bfloat16*>(q_idx), w, static_cast<const uint8_t*>(k_codes),
                                  static_cast<const uint8_t*>(k_scale), T, q_pos, Ncap, m, R, S, hist1, err);
    return cudaGetLastError();
}

}  // namespace

bool index_tc_supported(int q_dtype, int key_fmt, int H_I, int d_I, int64_t Ncap, const void* k_codes,
                        const void* k_scale, int64_t R) {
    return q_dtype == CSAHCA_BF16 && (key_fmt == CSAHCA_E4M3_ROWSCALE || key_fmt == CSAHCA_E2M1_UE8M0) &&
           d_I == kDI && (H_I == 16 || H_I == 32 || H_I == 64) && Ncap % 8 == 0 && aligned(k_codes, 16) &&
           aligned(k_scale, 16) && R * cdiv(Ncap, (int64_t)kChunkTiles * kKeys) < (1LL << 31);
}

cudaError_t index_tc_launch(const void* q_idx, const float* w, const void* k_codes, const void* k_scale, int key_fmt,
                            int B, int T, int H_I, const int64_t* q_pos, int64_t Ncap, int m, float* S,
                            uint32_t* hist1, unsigned* err, cudaStream_t st) {
#define CSAHCA_IDX_CASE(F, HH)                                                                                  \
    if (key_fmt == F && H_I == HH)                                                                              \
        return launch_index_tc<F, HH>(q_idx, w, k_codes, k_scale, B, T, q_pos, Ncap, m, S, hist1, err, st);
    CSAHCA_IDX_CASE(CSAHCA_E2M1_UE8M0, 16)
    CSAHCA_IDX_CASE(CSAHCA_E2M1_UE8M0, 32)
    CSAHCA_IDX_CASE(CSAHCA_E2M1_UE8M0, 64)
    CSAHCA_IDX_CASE(CSAHCA_E4M3_ROWSCALE, 16)
    CSAHCA_IDX_CASE(CSAHCA_E4M3_ROWSCALE, 32)
    CSAHCA_IDX_CASE(CSAHCA_E4M3_ROWSCALE, 64)
#undef CSAHCA_IDX_CASE
    return cudaErrorNotSupported;
}

}  // namespace csahca
