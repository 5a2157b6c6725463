// Tensor-core lightning-indexer scores for chunked prefill: bf16 keys and bf16 queries, d_I = 64,
// H_I in {16, 32, 64}, many query rows.
//
// I(t,s) = sum_h w[t,h] * ReLU(q[t,h] . k_s)  (honbul.tistory.com/221 "CSA"; pogovet.com
// DeepSeek-V4 article, detail 4).  In prefill the rows are many and the keys are shared by all of
// them, so the scores are a dense contraction: one work item is a group of QR = 128 / H_I
// consecutive query rows (the B operand: N = QR * H_I = 128 rows of (query row, head), K = d_I)
// against a chunk of up to 64 key tiles of 128 keys (the A operand, M = 128), on the
// 5th-generation tensor core (tcgen05.mma kind::f16, bf16 x bf16 -> fp32 in TMEM).  Keys and the
// group's queries arrive by 2-D TMA (128-byte swizzle); the keys of a chunk are shared by the
// groups that run at the same time (items are ordered chunk-major), so they come from L2.
//
// Warp roles (persistent CTAs over (chunk, group) items):
//   warp 8     producer: per item the group's query tile, head weights and visible counts into one
//              of two query slots; per tile (one lane) the TMA box of 128 keys;
//   warp 9     one thread issues the 4 MMAs of a tile (K = 16 each) into one of two TMEM
//              accumulators;
//   warps 0-7  epilogue: warp e reads TMEM lanes 32 (e % 4) .. (the tile's keys) and the columns of
//              query rows [(e / 4) QR/2, (e / 4 + 1) QR/2): per key and row the score
//              sum_h w_h ReLU(D[row, h]), stored to S (consecutive lanes, consecutive keys).
// Scores of keys a row does not see (s >= its visible count) are not stored.  The top-k's first
// histogram is not formed here: with thousands of rows a separate histogram pass over the scores
// costs less than the epilogue's shared-memory atomics (one per key and row) did.
#include "common.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

#include <algorithm>
#include <cstddef>
#include <cstring>

namespace csahca {
namespace {

using namespace tc;

constexpr int kKeysT = 128;          // keys per tile (MMA M)
constexpr int kDI = 64;              // index dim (128 bytes of bf16: one swizzled row)
constexpr int kChunkTiles = 64;      // tiles per item: 8192 keys
constexpr int kNS = 4;               // key-tile stages (two CTAs per SM: 2 x 96 KB of shared memory)
constexpr int kEpiWarps = 8;
constexpr int kThreadsP = 32 * kEpiWarps + 64;
constexpr uint32_t kTileBytes = kKeysT * 128;   // 16 KB
constexpr uint32_t kQBytes = 128 * 128;         // 128 (row, head) rows x 128 B

template <int HI>
struct PCfg {
    static constexpr int QR = 128 / HI;                        // query rows per item
    static constexpr uint32_t off_q = kNS * kTileBytes;        // two query slots
    static constexpr uint32_t smem = off_q + 2 * kQBytes;
    static_assert(HI == 16 || HI == 32 || HI == 64, "heads");
};

struct alignas(16) PMisc {
    uint64_t full[kNS], empty[kNS], qfull[2], qfree[2], dfull[2], dfree[2];
    uint32_t tmem_base;
    alignas(16) float w[2][128];     // head weights of the slot's (row, head) columns (read as float2)
    alignas(16) int nvis[2][8];      // visible entries of the slot's rows
    alignas(16) int4 item[2];        // per slot: first row, key0 of the chunk, tiles, flags
};
static_assert(offsetof(PMisc, w) % 16 == 0 && offsetof(PMisc, item) % 16 == 0, "PMisc vector fields");

// Item i (chunk-major): chunk c = i / G, group g = i % G; its tiles cover keys
// [c * 8192, c * 8192 + 128 * tiles) of the group's sequence, tiles limited by the group's largest
// visible count.
template <int HI>
__global__ void __launch_bounds__(kThreadsP, 2) index_prefill_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap, const float* __restrict__ w,
    int T, const int64_t* __restrict__ q_pos, int64_t Ncap, int m, int R, float* __restrict__ S,
    unsigned* err) {
    using C = PCfg<HI>;
    constexpr int QR = C::QR;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~uintptr_t(1023));
    __shared__ PMisc ms;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = smem_u32(sm);

    if (warp == 0) {
        tmem_alloc(&ms.tmem_base, 256);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&ms.full[s], 1);
            mbar_init(&ms.empty[s], 1);
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(&ms.qfull[d], 1);
            mbar_init(&ms.qfree[d], 1 + kEpiWarps);   // MMA commit + the epilogue warps
            mbar_init(&ms.dfull[d], 1);
            mbar_init(&ms.dfree[d], kEpiWarps);
        }
        fence_mbar_init();
    }
    pdl_wait();
    pdl_trigger();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = ms.tmem_base;
    const int G = R / QR;
    const int chunks = (int)cdiv(Ncap, (int64_t)kChunkTiles * kKeysT);
    const int items = G * chunks;

    if (warp == kEpiWarps) {
        // ======================================================================== producer
        if (lane == 0) {
            const uint64_t pol_keys = l2_policy_evict_last();     // shared by the groups of a chunk
            const uint64_t pol_q = l2_policy_evict_first();
            uint32_t u = 0, it = 0;
            for (int item = blockIdx.x; item < items; item += gridDim.x) {
                const int c = item / G, g = item % G;
                const int r0 = g * QR, b = r0 / T;
                int nmax = 0;
                int nv[QR];
#pragma unroll
                for (int j = 0; j < QR; ++j) {
                    const int64_t p = q_pos[r0 + j];
                    int64_t n = (p >= 0) ? (p + 1) / m : 0;
                    n = n < Ncap ? n : Ncap;
                    nv[j] = (int)n;
                    nmax = max(nmax, (int)n);
                }
                const int64_t key0 = (int64_t)c * kChunkTiles * kKeysT;
                if (key0 >= nmax) continue;
                const int64_t tl = cdiv(nmax - key0, (int64_t)kKeysT);
                const int tiles = (int)(tl < kChunkTiles ? tl : kChunkTiles);
                const uint32_t qs = it & 1;
                if (it >= 2) mbar_wait(&ms.qfree[qs], ((it >> 1) + 1) & 1, err);
#pragma unroll
                for (int j = 0; j < QR; ++j) ms.nvis[qs][j] = nv[j];
                for (int j = 0; j < QR * HI; ++j) ms.w[qs][j] = w[(int64_t)r0 * HI + j];
                ms.item[qs] = make_int4(r0, (int)key0, tiles, 0);
                mbar_arrive_expect_tx(&ms.qfull[qs], kQBytes);
                tma_load_2d(sbase + C::off_q + qs * kQBytes, &qmap, 0, r0 * HI, &ms.qfull[qs], pol_q);
                for (int t = 0; t < tiles; ++t, ++u) {
                    const uint32_t s = u % kNS;
                    if (u >= (uint32_t)kNS) mbar_wait(&ms.empty[s], ((u / kNS) + 1) & 1, err);
                    mbar_arrive_expect_tx(&ms.full[s], kTileBytes);
                    tma_load_2d(sbase + s * kTileBytes, &kmap, 0, (int)((int64_t)b * Ncap + key0 + (int64_t)t * kKeysT),
                                &ms.full[s], pol_keys);
                }
                ++it;
            }
            // end of work: an item record with no tiles
            const uint32_t qs = it & 1;
            if (it >= 2) mbar_wait(&ms.qfree[qs], ((it >> 1) + 1) & 1, err);
            ms.item[qs] = make_int4(0, 0, 0, 1);
            mbar_arrive(&ms.qfull[qs]);
        }
        __syncwarp();
    } else if (warp == kEpiWarps + 1) {
        // ============================================================================= MMA
        if (lane == 0) {
            const uint32_t id = idesc_f16(128, 128, 1, 0, 0);
            const uint64_t a0 = smem_desc(sbase, 16, 1024);
            const uint64_t b0 = smem_desc(sbase + C::off_q, 16, 1024);
            uint32_t u = 0, dn = 0;
            for (uint32_t it = 0;; ++it) {
                const uint32_t qs = it & 1;
                mbar_wait(&ms.qfull[qs], (it >> 1) & 1, err);
                const int4 itm = ms.item[qs];
                if (itm.w) break;
                const uint64_t bq = b0 + ((qs * kQBytes) >> 4);
                for (int t = 0; t < itm.z; ++t, ++u, ++dn) {
                    const uint32_t s = u % kNS, d = dn & 1;
                    mbar_wait(&ms.full[s], (u / kNS) & 1, err);
                    if (dn >= 2) mbar_wait(&ms.dfree[d], ((dn >> 1) + 1) & 1, err);
                    fence_after_sync();
                    const uint64_t a = a0 + ((s * kTileBytes) >> 4);
#pragma unroll
                    for (int k = 0; k < 4; ++k)                   // K = 16 per MMA: 32 bytes
                        mma_ss(tmem + d * 128, a + (uint64_t)(2 * k), bq + (uint64_t)(2 * k), id, (uint32_t)(k > 0));
                    mma_commit(&ms.dfull[d]);
                    mma_commit(&ms.empty[s]);
                }
                mma_commit(&ms.qfree[qs]);
            }
        }
        __syncwarp();
    } else {
        // ======================================================================== epilogue
        const int qd = warp & 3, hh = warp >> 2;          // TMEM lane quarter, half of the rows
        const int key_l = 32 * qd + lane;                 // key of the tile this thread scores
        const uint32_t lane_off = (uint32_t)(32 * qd) << 16;
        uint32_t dn = 0;
        for (uint32_t it = 0;; ++it) {
            const uint32_t qs = it & 1;
            mbar_wait(&ms.qfull[qs], (it >> 1) & 1, err);
            const int4 itm = ms.item[qs];
            if (itm.w) break;
            const int r0 = itm.x, key0 = itm.y;
            // this thread's rows hh QR/2 + j, j < QR/2, own the 64 consecutive accumulator columns
            // [64 hh, 64 hh + 64) of a tile (QR/2 rows x H_I heads); their head weights are read
            // from shared memory (broadcast) so that two CTAs' registers fit an SM
            constexpr int kCols = (QR / 2) * HI;
            static_assert(kCols == 64, "64 columns per epilogue thread");
            int nv[QR / 2];
#pragma unroll
            for (int j = 0; j < QR / 2; ++j) nv[j] = ms.nvis[qs][hh * (QR / 2) + j];
            const float2* wsm = reinterpret_cast<const float2*>(&ms.w[qs][hh * kCols]);
            for (int t = 0; t < itm.z; ++t, ++dn) {
                const uint32_t d = dn & 1;
                mbar_wait(&ms.dfull[d], (dn >> 1) & 1, err);
                fence_after_sync();
                const int key = key0 + t * kKeysT + key_l;
                // all 64 columns in one round trip, then the accumulator goes back to the MMA warp
                uint32_t v[kCols];
#pragma unroll
                for (int c = 0; c < kCols; c += 16) {
                    uint32_t t16[16];
                    tmem_ld16(tmem + d * 128 + lane_off + hh * kCols + c, t16);
#pragma unroll
                    for (int k = 0; k < 16; ++k) v[c + k] = t16[k];
                }
                tmem_wait_ld();
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ms.dfree[d]);
                float sc[QR / 2];
#pragma unroll
                for (int j = 0; j < QR / 2; ++j) {
                    uint64_t acc = f2_pack(0.0f, 0.0f);
#pragma unroll
                    for (int k = 0; k < HI; k += 2) {
                        const int c = j * HI + k;
                        acc = f2_fma(f2_pack(wsm[c / 2].x, wsm[c / 2].y),
                                     f2_pack(fmaxf(__uint_as_float(v[c]), 0.0f), fmaxf(__uint_as_float(v[c + 1]), 0.0f)),
                                     acc);
                    }
                    float a0, a1;
                    f2_unpack(acc, a0, a1);
                    sc[j] = a0 + a1;
                }
#pragma unroll
                for (int j = 0; j < QR / 2; ++j) {
                    const int row = hh * (QR / 2) + j;
                    if (key < nv[j]) S[(int64_t)(r0 + row) * Ncap + key] = sc[j];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.qfree[qs]);
        }
    }
    __syncwarp();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

template <int HI>
cudaError_t launch_prefill(const void* q_idx, const float* w, const void* k_codes, int B, int T, const int64_t* q_pos,
                           int64_t Ncap, int m, float* S, unsigned* err, cudaStream_t st) {
    using C = PCfg<HI>;
    CUtensorMap kmap, qmap;
    std::memset(&kmap, 0, sizeof kmap);
    std::memset(&qmap, 0, sizeof qmap);
    const int R = B * T;
    if (!encode_tmap_2d(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k_codes, kDI, (uint64_t)B * Ncap, kDI * 2, kDI, kKeysT) ||
        !encode_tmap_2d(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q_idx, kDI, (uint64_t)R * HI, kDI * 2, kDI, 128))
        return cudaErrorNotSupported;
    const size_t smem = (size_t)C::smem + 1024;
    auto kern = index_prefill_kernel<HI>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t items = (int64_t)(R / C::QR) * cdiv(Ncap, (int64_t)kChunkTiles * kKeysT);
    const int grid = (int)std::min<int64_t>(items, 2 * num_sms());   // two CTAs per SM
    (void)launch_pdl(kern, dim3(grid), dim3(kThreadsP), smem, st, kmap, qmap, w, T, q_pos, Ncap, m, R, S, err);
    return cudaGetLastError();
}

}  // namespace

bool index_prefill_supported(int q_dtype, int key_fmt, int H_I, int d_I, int64_t Ncap, const void* q_idx,
                             const void* k_codes, int B, int T) {
    if (!(q_dtype == CSAHCA_BF16 && key_fmt == CSAHCA_BF16 && d_I == kDI && (H_I == 16 || H_I == 32 || H_I == 64)))
        return false;
    const int QR = 128 / H_I;
    const int64_t R = (int64_t)B * T;
    return T % QR == 0 && R >= QR && R * H_I >= 128 && aligned(q_idx, 32) && aligned(k_codes, 32) &&
           (int64_t)B * Ncap >= kKeysT && (int64_t)B * Ncap < (1LL << 31) && R * H_I < (1LL << 31);
}

cudaError_t index_prefill_launch(const void* q_idx, const float* w, const void* k_codes, int B, int T, int H_I,
                                 const int64_t* q_pos, int64_t Ncap, int m, float* S, unsigned* err,
                                 cudaStream_t st) {
    switch (H_I) {
        case 16: return launch_prefill<16>(q_idx, w, k_codes, B, T, q_pos, Ncap, m, S, err, st);
        case 32: return launch_prefill<32>(q_idx, w, k_codes, B, T, q_pos, Ncap, m, S, err, st);
        case 64: return launch_prefill<64>(q_idx, w, k_codes, B, T, q_pos, Ncap, m, S, err, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace csahca
