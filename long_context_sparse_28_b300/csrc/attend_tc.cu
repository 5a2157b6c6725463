// Tensor-core split attention for bf16 and d = 128 (CSA: selected entries + window; HCA: every
// visible entry + window), sm_103a tcgen05 + TMEM + TMA.
//
// All H query heads of a query share one KV stream (honbul.tistory.com/221 "CSA"/"HCA";
// pogovet.com detail 4), so one tile of 128 keys against all heads is a dense contraction:
//   S^T[128 keys x H]  = K_tile[128 x 128] . Q^T          (A = K, K-major; B = Q, K-major)
//   O^T[128 dims x H] += V_tile^T[128 x 128] . P[128 x H]  (A = V, MN-major; B = P, MN-major)
// Keys are the M dimension: a thread owns one key row of S^T (tcgen05.ld 32x32b) and the V tile
// is used as loaded.  One warpgroup per 16 heads forms P; one more warp only issues the MMAs
// (16 per tile) and hands over through mbarriers, so no softmax barrier waits on MMA issue.  The
// softmax makes one pass over S with the running maxima; only when some score exceeds its
// head's running maximum by more than 2^8 (always on an item's first tile) are the tile maxima
// formed, the maxima raised, P formed again and the O^T accumulator in TMEM rescaled; row sums
// stay per thread until the end of the work item.
//
// Keys are addressed in tile space: the compressed keys of a query fill tiles [0, nt_c), the
// window fills tiles [nt_c, nt_c + nt_w).  A tile whose rows are contiguous in memory (HCA
// entries; the decode window ring when it holds exactly 128 tokens) is fetched as two 2-D TMA
// boxes (128-byte swizzle) by one thread; selected CSA entries and chunked-prefill windows are
// gathered row by row with cp.async.  K and V tiles have their own two-slot rings: K(i+2) is
// requested once MMA1(i) is done, V(i+1) once PV(i-1) is done, and the MMA warp issues MMA1(i+2)
// right after PV(i), so loads, both MMAs and the softmax of the next tile overlap.  With few
// query rows each CTA takes one near-equal piece of one row's tiles (pieces sized from the rows'
// actual lengths); otherwise CTAs are persistent over (row, key-split) items.  Partial results
// (o normalised, lse) go to the split workspace; each item then counts its arrival at its row
// (an atomic on a per-row counter of the workspace), and the row's last item merges the row's
// partials exactly and resets the counter, so no second launch is needed and nothing waits.
#include "attend.cuh"
#include "quant.cuh"
#include "tc_ptx.cuh"

#include "tmap.cuh"

#include <algorithm>
#include <cstddef>
#include <cstring>

namespace csahca {
namespace {

using namespace tc;

constexpr int kKeys = 128;                 // keys per tile (MMA M)
constexpr int kD = 128;                    // head dim
constexpr int kHG = 16;                    // heads per softmax warpgroup (one tcgen05.ld of 16 columns)
constexpr uint32_t kHalf = kKeys * 128;    // [128 rows][64 bf16] swizzled half tile: 16 KB
constexpr uint32_t kTile = 2 * kHalf;      // one K or V tile: 32 KB
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kSchedRows = 256;            // piece schedule for up to this many query rows
constexpr int kMergeSlots = 16;            // partial slots merged per pass

// Softmax / load threads: one warpgroup (128 threads, one per key row) per 16 heads; then the
// MMA warp.
template <int H, bool F8 = false>
struct Thr {
    static_assert(H % kHG == 0, "heads in groups of 16");
    static constexpr int kSoft = (H / kHG) * kKeys;
    static constexpr int kThreads = kSoft + 32;
};

template <int H>
struct Smem {
    static constexpr uint32_t q = 0;                                  // 2 halves x [H][128 B]
    static constexpr uint32_t q_half = H * 128;
    static constexpr uint32_t p = 2 * q_half;                         // two P buffers [128 keys][H] bf16
    static constexpr uint32_t p_region = kKeys * 128;
    static constexpr uint32_t p_bytes = ((H + 63) / 64) * p_region;
    static constexpr uint32_t p_lo = p + 2 * p_bytes;                 // their low parts P - bf16(P)
    static constexpr uint32_t k = (p_lo + 2 * p_bytes + 1023) / 1024 * 1024;  // two K slots
    static constexpr uint32_t v = k + 2 * kTile;                      // two V slots
    static constexpr uint32_t total = v + 2 * kTile;
};

struct alignas(16) Misc {
    uint64_t kfull[2], vfull[2], sdone[2], odone, pready;
    uint64_t k8full[2], v8full[2];   // FP8 caches: a tile's codes have landed (before conversion)
    uint64_t mfull;                  // the row merge's partials have landed in shared memory
    uint32_t tmem_base;
    int flag[4][2];                  // per warpgroup and tile (ring of 2): one of its maxima moved
    alignas(16) float red[16][32];
    alignas(16) float mrun[64];      // read as float4
    alignas(16) float mold[64];      // running maxima before the tile's update (float4)
    alignas(16) float alpha[64];     // read as float4
    float linv[64];
    unsigned char valid[4][kKeys];   // per tile (ring of 4): row holds a key of this query
    int32_t eidx[4][kKeys];          // per tile (ring of 4), CSA: the row's selected entry (-1: none)
    int snt[kSchedRows];             // piece schedule: tiles of each query row
    int my_row, my_piece, my_t0, my_nt;  // piece schedule: this CTA's piece (row -1: none), its
    int my_empty_row;                // row's slots [my_slots_from, S) it marks empty, a row
    int my_slots_from;               // without tiles whose slots it marks empty (or -1), and
    int64_t my_p;                    // the query position of its row
    int my_np;                       // pieces (= partial slots) of its row
    int merge_now;                   // this CTA arrived last at its row: it merges the row
    alignas(16) float mw[kMergeSlots * 64];   // the merge's per-(slot, head) log-sum-exps, then weights
};
static_assert(offsetof(Misc, mrun) % 16 == 0 && offsetof(Misc, mold) % 16 == 0 && offsetof(Misc, alpha) % 16 == 0,
              "float4 fields");

struct ItemTiles {
    int r, b, nt_c, t0, nt, slot;
    int expect;                      // partial slots of the row, written by as many items
    int64_t p;
    KeyList kl;
};

struct Maps {
    CUtensorMap ck, cv, rk, rv;
    CUtensorMap k8, kr, v8;          // FP8 caches: K codes + scale bytes, K RoPE dims (bf16), V codes
};

// Piece schedule, computed by one warp (no more query rows than CTAs, S >= 2 partial slots per
// row): every row is cut into ceil(tiles / L) pieces of near-equal length, L the smallest length
// >= the average tiles per CTA for which all pieces fit the grid and no row has more than S
// pieces; CTA c takes the c-th piece (row by row), whose partial result goes to slot = piece
// index.  The general form is kept out of line (it runs once per CTA and its code should not crowd
// the tile loop); its inputs come by value: the kernel's parameters, read through a reference in
// an out-of-line call, take a generic load each (about 0.5 us for the schedule's few fields).
struct SchedIn {
    const int64_t* q_pos;
    int64_t Ncap;
    int R, m, k, is_csa;
};

__device__ __forceinline__ int compressed_tiles(const SchedIn& si, int64_t p) {
    int64_t n;
    if (si.is_csa) {
        n = si.k;
    } else {
        n = (p < 0) ? 0 : ((si.m & (si.m - 1)) == 0 ? (p + 1) >> (__ffs(si.m) - 1) : (p + 1) / si.m);
        n = n < si.Ncap ? n : si.Ncap;
    }
    return (int)cdiv(n, kKeys);
}

// Up to 32 rows (the decode batches), one row per lane: the same schedule in registers and
// shuffles, inlined (the out-of-line call's first instruction fetch costs about 0.4 us).
__device__ __forceinline__ void piece_schedule_rows32(const SchedIn& si, int S, int nt_w, Misc& ms, int lane) {
    const int R = si.R;
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    {
        const bool in = lane < R;
        const int64_t pq = in ? si.q_pos[lane] : 0;
        const int nt = in ? compressed_tiles(si, pq) + nt_w : 0;
        int total = nt, ntmax = nt;
        for (int o = 16; o > 0; o >>= 1) {
            total += __shfl_xor_sync(0xffffffffu, total, o);
            ntmax = max(ntmax, __shfl_xor_sync(0xffffffffu, ntmax, o));
        }
        int len = max(max((int)cdiv(total, G), (int)cdiv(ntmax, S)), 1);
        for (;;) {
            int cnt = (nt + len - 1) / len;
            for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
            if (cnt <= G) break;
            ++len;
        }
        const int np = (nt + len - 1) / len;
        int x = np;
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        const int first = x - np;
        if (lane == 0) {
            ms.my_row = -1;
            ms.my_slots_from = S;
            ms.my_empty_row = -1;
        }
        __syncwarp();
        if (in && np > 0 && c >= first && c < first + np) {
            const int piece = c - first;
            const int t0 = piece * nt / np;
            ms.my_row = lane;
            ms.my_piece = piece;
            ms.my_t0 = t0;
            ms.my_nt = (piece + 1) * nt / np - t0;
            ms.my_p = pq;
            ms.my_np = np;
            if (piece == 0) ms.my_slots_from = np;
        }
        if (in && np == 0 && lane == c) ms.my_empty_row = lane;   // R <= gridDim.x
    }
}

// (out of line where inlining it would push the tile loop's registers into spills)
__device__ __noinline__ void piece_schedule_rows32_ool(const SchedIn si, int S, int nt_w, Misc& ms, int lane) {
    piece_schedule_rows32(si, S, nt_w, ms, lane);
}

__device__ __noinline__ void piece_schedule(const SchedIn si, int S, int nt_w, Misc& ms, int lane) {
    const int R = si.R;
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    int total = 0, ntmax = 0;
#pragma unroll 1
    for (int q = lane; q < R; q += 32) {
        const int n = compressed_tiles(si, si.q_pos[q]) + nt_w;
        ms.snt[q] = n;
        total += n;
        ntmax = max(ntmax, n);
    }
    for (int o = 16; o > 0; o >>= 1) {
        total += __shfl_xor_sync(0xffffffffu, total, o);
        ntmax = max(ntmax, __shfl_xor_sync(0xffffffffu, ntmax, o));
    }
    __syncwarp();
    int len = max(max((int)cdiv(total, G), (int)cdiv(ntmax, S)), 1);
    for (;;) {                                      // usually one or two rounds
        int cnt = 0;
#pragma unroll 1
        for (int q = lane; q < R; q += 32) cnt += (ms.snt[q] + len - 1) / len;
        for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        if (cnt <= G) break;
        ++len;
    }
    if (lane == 0) {
        ms.my_row = -1;
        ms.my_slots_from = S;
        ms.my_empty_row = -1;
    }
    __syncwarp();
    // first CTA of each row: exclusive prefix of the piece counts, rows in order
    int carry = 0;
#pragma unroll 1
    for (int q0 = 0; q0 < R; q0 += 32) {
        const int q = q0 + lane;
        const int nt = q < R ? ms.snt[q] : 0;
        const int np = (nt + len - 1) / len;
        int x = np;
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        const int first = carry + x - np;
        carry += __shfl_sync(0xffffffffu, x, 31);
        if (q < R && np > 0 && c >= first && c < first + np) {
            const int piece = c - first;
            const int t0 = piece * nt / np;
            ms.my_row = q;
            ms.my_piece = piece;
            ms.my_t0 = t0;
            ms.my_nt = (piece + 1) * nt / np - t0;
            ms.my_p = si.q_pos[q];
            ms.my_np = np;
            if (piece == 0) ms.my_slots_from = np;
        }
        if (q < R && np == 0 && q == c) ms.my_empty_row = q;   // R <= gridDim.x
    }
}

// One K (is_v = false) or V tile -- keys [ti * 128, ti * 128 + 128) of query row r's tile space --
// into shared memory at `dst`; completion on `bar` counts kSoft arrivals plus the TMA bytes.
// Called by all kSoft loading threads.  For a K tile, valid[row] records whether the row holds a
// key of the query.  A tile of contiguous rows with a tensor map is two 2-D TMA boxes issued by
// thread 0; otherwise the rows are gathered with cp.async (kSoft / 128 threads per row).  With
// `track_cp` every thread's arrival waits for all its earlier cp.async copies (the query tile
// loaded just before), else a TMA tile's arrivals are made at once by thread 0.
// CSA selected entries: a K tile records each row's entry in e_dst[row]; a V tile reads them from
// e_src (its K tile's record) instead of the index list, and a K tile takes the thread's row's
// entry from e_pre when the caller loaded it ahead (else kNoEntry: read here).
constexpr int32_t kNoEntry = INT32_MIN;

template <int kSoft>
__device__ __forceinline__ void load_tile(const AttendArgs& a, const Maps& maps, int use_tma_c, int use_tma_w, int r,
                                       int b, int64_t p, int64_t n_c, int64_t total, int nt_c, int ti, bool is_v,
                                       uint32_t dst, uint64_t* bar, unsigned char* valid, const void* zsrc,
                                       uint64_t pol, bool track_cp, unsigned* err, int32_t* e_dst = nullptr,
                                       const int32_t* e_src = nullptr, int32_t e_pre = kNoEntry) {
    const int tid = threadIdx.x;
    const bool comp = ti < nt_c;
    if (comp ? use_tma_c : use_tma_w) {
        if (!is_v && tid < kKeys) {
            // ring slot `tid` of the decode window holds token t = tid (mod 128) of the last 128
            valid[tid] = comp ? ((int64_t)ti * kKeys + tid < n_c) : (p - ((p - tid) & (kKeys - 1)) >= 0);
        }
        if (tid == 0) {
            mbar_expect_tx(bar, kTile);
            const CUtensorMap* mp = comp ? (is_v ? &maps.cv : &maps.ck) : (is_v ? &maps.rv : &maps.rk);
            const int y = comp ? (int)((int64_t)b * a.Ncap + (int64_t)ti * kKeys) : b * a.ring_cap;
            tma_load_2d(dst, mp, 0, y, bar, pol);
            tma_load_2d(dst + kHalf, mp, 64, y, bar, pol);
            if (!track_cp) mbar_arrive_cnt(bar, kSoft);     // the arrivals of all loading threads
        }
        if (track_cp) cp_async_arrive_noinc(bar);
        return;
    }
    constexpr int kTpr = kSoft / kKeys;
    constexpr int kCpt = 16 / kTpr;
    const int rr = tid / kTpr, part = tid % kTpr;
    const int64_t key = comp ? (int64_t)ti * kKeys + rr : n_c + (int64_t)(ti - nt_c) * kKeys + rr;
    const bool in = key < (comp ? n_c : total);
    const __nv_bfloat16* kp = nullptr;
    const __nv_bfloat16* vp = nullptr;
    int32_t e = -1;
    if (in && comp && a.is_csa) {
        // (the selected-entry path of key_rows, with the entry possibly known already)
        e = e_src ? e_src[rr] : (e_pre != kNoEntry ? e_pre : a.idx[(int64_t)r * a.k + key]);
        if (e >= a.Ncap) {
            flag_error(err, ERRBIT_BOUNDS);
            e = -1;
        }
        if (e >= 0) {
            const int64_t off = ((int64_t)b * a.Ncap + e) * a.d;
            kp = static_cast<const __nv_bfloat16*>(a.ck) + off;
            vp = static_cast<const __nv_bfloat16*>(a.cv) + off;
        }
    } else if (in) {
        KeyList kl;
        kl.n_c = n_c;
        kl.total = total;
        key_rows<__nv_bfloat16>(a, kl, r, b, p, key, &kp, &vp, err);
    }
    if (!is_v && part == 0) {
        valid[rr] = kp != nullptr;
        if (e_dst) e_dst[rr] = e < 0 ? -1 : e;
    }
    const __nv_bfloat16* src = is_v ? vp : kp;
#pragma unroll
    for (int c = 0; c < kCpt; ++c) {
        const int cc = part * kCpt + c;              // 16-byte chunk of the row: half cc / 8
        const uint32_t d = dst + (cc >> 3) * kHalf + sw128(rr, cc & 7);
        if (src) cp_async16_hint(d, src + cc * 8, 16, pol);
        else cp_async16(d, zsrc, 0);                 // zero fill (no bytes read)
    }
    cp_async_arrive_noinc(bar);
}

// FP8 caches (CSAHCA_KV_FP8).  A compressed K tile lands as 128 dense rows of 128 bytes (the row's
// 64 codes, the scale bytes of the K and V rows and the bytes after them) in the slot's first half
// and its RoPE dims (bf16) in the second half with the 128-byte swizzle of a bf16 tile; a V tile's
// codes land as 128 dense rows of 128 bytes in the slot's second half.  The V scale bytes reach
// a side buffer when the K tile is expanded.  The threads of a tile row then turn it into bf16
// within the row's own 128-byte rows.  Contiguous tiles come by TMA (issued by thread 0),
// selected entries are gathered with cp.async; completion is counted on `bar` as in load_tile.
constexpr uint32_t kVScale = kKeys * 16;                // V scale rows of one slot: 2 KB

template <int kSoft>
__device__ __forceinline__ void load_tile_f8(const AttendArgs& a, const Maps& maps, int use_tma, int r, int b,
                                             int64_t n_c, int ti, bool is_v, uint32_t dst, uint32_t vsc,
                                             uint64_t* bar, unsigned char* valid, const void* zsrc, uint64_t pol,
                                             bool track_cp, unsigned* err) {
    const int tid = threadIdx.x;
    if (use_tma) {
        if (!is_v && tid < kKeys) valid[tid] = (int64_t)ti * kKeys + tid < n_c;
        if (tid == 0) {
            const int y = (int)((int64_t)b * a.Ncap + (int64_t)ti * kKeys);
            mbar_expect_tx(bar, is_v ? kHalf : 2 * kHalf);
            if (is_v) {
                tma_load_2d(dst + kHalf, &maps.v8, 0, y, bar, pol);
            } else {
                tma_load_2d(dst, &maps.k8, 0, y, bar, pol);
                tma_load_2d(dst + kHalf, &maps.kr, 0, y, bar, pol);
            }
            if (!track_cp) mbar_arrive_cnt(bar, kSoft);
        }
        if (track_cp) cp_async_arrive_noinc(bar);
        return;
    }
    constexpr int kTpr = kSoft / kKeys;                 // threads per row
    const int rr = tid / kTpr, part = tid % kTpr;
    const int64_t key = (int64_t)ti * kKeys + rr;
    const unsigned char* src = nullptr;
    if (key < n_c) {
        int64_t e = key;
        if (a.is_csa) {
            e = a.idx[(int64_t)r * a.k + key];
            if (e >= a.Ncap) {
                flag_error(err, ERRBIT_BOUNDS);
                e = -1;
            }
        }
        if (e >= 0)
            src = static_cast<const unsigned char*>(is_v ? a.cv : a.ck) +
                  ((int64_t)b * a.Ncap + e) * (is_v ? kKv8VRow : kKv8KRow);
    }
    if (!is_v && part == 0) valid[rr] = src != nullptr;
    // K: 6 chunks of codes, scale bytes and zeros (dense row rr of the first half), 8 of RoPE dims
    // (swizzled second half); V: 8 chunks of codes (dense row rr of the second half)
    (void)vsc;
    const int nch = is_v ? 8 : 14;
    for (int c = part; c < nch; c += kTpr) {
        uint32_t d;
        if (is_v) d = dst + kHalf + rr * 128 + c * 16;
        else d = c < 6 ? dst + rr * 128 + c * 16 : dst + kHalf + sw128(rr, c - 6);
        if (src) cp_async16_hint(d, src + c * 16, 16, pol);
        else cp_async16(d, zsrc, 0);                    // zero fill (no bytes read)
    }
    cp_async_arrive_noinc(bar);
}

// 8 E4M3 codes (two 32-bit words) times 2^e -> 8 bf16 (exact: the product has at most 4
// significant bits).
__device__ __forceinline__ uint4 e4m3x8_to_bf16x8(uint32_t w0, uint32_t w1, float sc) {
    uint32_t o[4];
    const uint32_t w[2] = {w0, w1};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[h >> 1] >> (16 * (h & 1))), __NV_E4M3);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
        o[h] = pack_bf16x2(f.x * sc, f.y * sc);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// 2^(byte - 127) for a UE8M0 scale byte (2^-127 is subnormal; 255 is not produced by the pooling).
__device__ __forceinline__ float ue8m0_to_f32(uint32_t byte) {
    return byte ? __uint_as_float(byte << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 c;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(c.x), "=r"(c.y), "=r"(c.z), "=r"(c.w) : "r"(addr));
    return c;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 u) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(u.x), "r"(u.y), "r"(u.z), "r"(u.w) : "memory");
}

// Part `pt` (of kTpr) of row r of a K tile: its codes (the staged dense row r of the first half)
// -> bf16 in place.  The kTpr threads of a row sit in one warp: every one reads its codes and the
// scale byte, then (after __syncwarp) writes its chunks of the row.
template <int kTpr>
__device__ __forceinline__ void convert_k_part(uint32_t slot, uint32_t vsc, int r, int pt) {
    constexpr int kU = 64 / 16 / kTpr;                  // 16-code pieces per part
    uint4 c[kU];
#pragma unroll
    for (int i = 0; i < kU; ++i) c[i] = lds128(slot + r * 128 + (pt * kU + i) * 16);
    uint32_t sb;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(sb) : "r"(slot + r * 128 + 64));
    __syncwarp();
    if (pt == 0) asm volatile("st.shared.u32 [%0], %1;" ::"r"(vsc + r * 16), "r"(sb >> 8) : "memory");   // V's two
    const float sc = ue8m0_to_f32(sb & 0xFFu);
#pragma unroll
    for (int i = 0; i < kU; ++i) {
        const int j = 2 * (pt * kU + i);                // output chunks j, j + 1 (8 dims each)
        sts128(slot + sw128(r, j), e4m3x8_to_bf16x8(c[i].x, c[i].y, sc));
        sts128(slot + sw128(r, j + 1), e4m3x8_to_bf16x8(c[i].z, c[i].w, sc));
    }
}

// Part `pt` of row r of a V tile: codes (the staged dense row r of the second half) and scales ->
// bf16 dims 0..63 (first half) and 64..127 (second half), or zeros for a row that holds no key.
template <int kTpr>
__device__ __forceinline__ void convert_v_part(uint32_t slot, uint32_t vsc, int r, int pt, bool zero) {
    constexpr int kU = 128 / 16 / kTpr;
    uint4 c[kU];
#pragma unroll
    for (int i = 0; i < kU; ++i) c[i] = lds128(slot + kHalf + r * 128 + (pt * kU + i) * 16);
    uint32_t sb;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(sb) : "r"(vsc + r * 16));
    __syncwarp();
    const float sc0 = ue8m0_to_f32(sb & 0xFFu), sc1 = ue8m0_to_f32((sb >> 8) & 0xFFu);
#pragma unroll
    for (int i = 0; i < kU; ++i) {
        const int j = 2 * (pt * kU + i);                // output chunks j, j + 1 of the row's 16
        const float sc = j < 8 ? sc0 : sc1;
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        sts128(slot + (j >> 3) * kHalf + sw128(r, j & 7), zero ? z : e4m3x8_to_bf16x8(c[i].x, c[i].y, sc));
        sts128(slot + ((j + 1) >> 3) * kHalf + sw128(r, (j + 1) & 7), zero ? z : e4m3x8_to_bf16x8(c[i].z, c[i].w, sc));
    }
}

// Part `pt` of row r of a bf16 V tile: zeros (a row that holds no key of the query).
template <int kTpr>
__device__ __forceinline__ void zero_v_part(uint32_t slot, int r, int pt) {
    constexpr int kC = 16 / kTpr;
#pragma unroll
    for (int i = 0; i < kC; ++i) {
        const int j = pt * kC + i;
        sts128(slot + (j >> 3) * kHalf + sw128(r, j & 7), make_uint4(0u, 0u, 0u, 0u));
    }
}

// The row's last item merges the row's partial results (see arrive_and_merge in the kernel): up to
// kMergeStage slots at a time, one thread bulk-copies the slots' partial outputs (32 KB each,
// contiguous) and log-sum-exps into shared memory -- the tile buffers, idle once the item's MMAs
// are complete -- so a pass costs one round trip; one thread per head then forms the maxima,
// sums (rescaled across passes) and weights, and every thread adds its units (4 dims of one head)
// over the slots.  Out of line: it runs once per row and keeps its registers out of the tile
// loop's allocation.
constexpr int kMergeStage = 6;   // 6 x 32 KB of partial outputs in [L::p, L::total)

template <int H>
__device__ __noinline__ void merge_row(int r, int ns, int S, const float* __restrict__ lse_part,
                                       const float* __restrict__ o_part, __nv_bfloat16* __restrict__ out,
                                       float* __restrict__ lse_out, Misc& ms, int tid, uint32_t stage,
                                       uint32_t& mpass, unsigned* err) {
    constexpr int kSoft = Thr<H>::kSoft;
    constexpr uint32_t kSlotBytes = H * kD * 4;
    static_assert(kMergeStage * kSlotBytes <= Smem<H>::total - Smem<H>::p, "merge staging fits the tile buffers");
    static_assert(kMergeStage <= kMergeSlots, "lse staging");
    constexpr int kUnits = H * (kD / 4) / kSoft;   // units per thread (4)
    const float* lrow = lse_part + (int64_t)r * S * H;
    const float* orow = o_part + (int64_t)r * S * H * kD;
    float4 acc[kUnits];
#pragma unroll
    for (int u = 0; u < kUnits; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    static_assert(kSoft == 8 * H && kMergeStage <= 8, "eight merging threads per head, one slot each");
    const int wh = tid >> 3, wq = tid & 7;         // head wh, slot wq of a pass (kMergeStage <= 8)
    float mx = -INFINITY, tot = 0.0f;              // per head (its eight threads hold the same values)
    for (int s0 = 0; s0 < ns; s0 += kMergeStage) {
        const int nsl = min(kMergeStage, ns - s0);
        if (tid == 0) {
            fence_proxy_async();                       // the partials, for the bulk copies
            mbar_arrive_expect_tx(&ms.mfull, (uint32_t)nsl * (kSlotBytes + H * 4));
            for (int q = 0; q < nsl; ++q)
                bulk_g2s(stage + q * kSlotBytes, orow + (int64_t)(s0 + q) * H * kD, kSlotBytes, &ms.mfull);
            bulk_g2s(smem_u32(ms.mw), lrow + (int64_t)s0 * H, (uint32_t)nsl * H * 4, &ms.mfull);
        }
        mbar_wait(&ms.mfull, mpass & 1, err);
        ++mpass;
        {
            // a head's slots over its eight threads: the maximum by shuffles, one exponential per
            // thread, then the sum in slot order (as one thread would add them)
            const float ls = wq < nsl ? ms.mw[wq * H + wh] : -INFINITY;
            float m2 = fmaxf(mx, ls);
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) m2 = fmaxf(m2, __shfl_xor_sync(0xffffffffu, m2, o));
            const float rs = (m2 == -INFINITY) ? 0.0f : expf(mx - m2);   // 0 on the first pass
            const float e = ls == -INFINITY ? 0.0f : expf(ls - m2);
            tot *= rs;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float eq = __shfl_sync(0xffffffffu, e, (tid & ~7) | q);
                if (q < nsl) tot += eq;
            }
            mx = m2;
            if (wq < nsl) ms.mw[wq * H + wh] = e;
            if (wq == 0) ms.alpha[wh] = rs;
        }
        named_barrier_sync(1, kSoft);
#pragma unroll
        for (int u = 0; u < kUnits; ++u) {
            const int unit = tid + u * kSoft, hh = unit / (kD / 4), c4 = unit % (kD / 4);
            const float rs = ms.alpha[hh];
            float4 a4 = make_float4(acc[u].x * rs, acc[u].y * rs, acc[u].z * rs, acc[u].w * rs);
            for (int q = 0; q < nsl; ++q) {
                const float wgt = ms.mw[q * H + hh];
                float4 v;
                asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                             : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                             : "r"(stage + q * kSlotBytes + (uint32_t)(hh * kD + c4 * 4) * 4));
                a4.x = fmaf(wgt, v.x, a4.x);
                a4.y = fmaf(wgt, v.y, a4.y);
                a4.z = fmaf(wgt, v.z, a4.z);
                a4.w = fmaf(wgt, v.w, a4.w);
            }
            acc[u] = a4;
        }
        named_barrier_sync(1, kSoft);                  // the staging is reused by the next pass
    }
    if (wq == 0) {
        ms.linv[wh] = tot > 0.0f ? 1.0f / tot : 0.0f;
        if (lse_out) lse_out[(int64_t)r * H + wh] = tot > 0.0f ? mx + logf(tot) : -INFINITY;
    }
    named_barrier_sync(1, kSoft);
    fence_proxy_async();              // the staging reads, before the next item's copies into the buffers
    __nv_bfloat16* orow_out = out + (int64_t)r * H * kD;
#pragma unroll
    for (int u = 0; u < kUnits; ++u) {
        const int unit = tid + u * kSoft;
        const float li = ms.linv[unit / (kD / 4)];
        reinterpret_cast<uint2*>(orow_out)[unit] =
            make_uint2(pack_bf16x2(acc[u].x * li, acc[u].y * li), pack_bf16x2(acc[u].z * li, acc[u].w * li));
    }
}

template <int H, bool F8>
__global__ void __launch_bounds__(Thr<H, F8>::kThreads, 1)
    attend_tc_kernel(const __grid_constant__ AttendArgs a, int S, int kps, const __grid_constant__ Maps maps, int use_tma_c, int use_tma_w,
                     int fixed_np, float* __restrict__ o_part, float* __restrict__ lse_part,
                     unsigned* __restrict__ row_cnt, unsigned* err) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~uintptr_t(1023));
    __shared__ Misc ms;
    using L = Smem<H>;
    constexpr int kSoft = Thr<H>::kSoft;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr uint32_t kCols = (3 * H <= 128) ? 128 : 256;   // S[2] + O

    // TMEM and barriers touch no global memory: set up while the preceding kernel finishes
    if (warp == 0) {
        tmem_alloc(&ms.tmem_base, kCols);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int i = 0; i < 2; ++i) {
            // FP8 caches: the loads complete on k8full / v8full; the softmax warps expand the codes
            // and release each tile (one arrival per warp)
            mbar_init(&ms.kfull[i], F8 ? kSoft / 32 : kSoft);
            mbar_init(&ms.vfull[i], F8 ? kSoft / 32 : kSoft);
            mbar_init(&ms.k8full[i], kSoft);
            mbar_init(&ms.v8full[i], kSoft);
            mbar_init(&ms.sdone[i], 1);
            for (int w4 = 0; w4 < 4; ++w4) ms.flag[w4][i] = 0;
        }
        mbar_init(&ms.odone, 1);
        mbar_init(&ms.pready, kSoft / 32);
        mbar_init(&ms.mfull, 1);
        fence_mbar_init();
    }
    pdl_wait();
    pdl_trigger();
    const int R = a.B * a.T;
    const int items = R * S;
    const int tps = kps / kKeys;
    const int nt_w = (int)cdiv(a.W, kKeys);
    // With few query rows each CTA takes one piece of one row (piece_schedule); otherwise items
    // are (row, split) pairs, split s holding tiles [s kps, (s+1) kps).
    const bool pieces = R <= kSchedRows && R <= (int)gridDim.x && S >= 2;
    // one split per row (many rows): each item is a whole row, written as the final output (bf16,
    // and the lse) with no merge
    const bool direct = !pieces && S == 1;
    if (pieces && warp == 0) {
        if (fixed_np > 0) {
            // every row has the same tiles (CSA: k selected entries + the window); the host cut
            // them into fixed_np pieces per row, so CTA c takes piece c % fixed_np of row c / fixed_np
            if (lane == 0) {
                const int c = (int)blockIdx.x, q = c / fixed_np, piece = c % fixed_np;
                const int nt = (int)cdiv(a.k, kKeys) + nt_w;
                ms.my_row = q < R ? q : -1;
                ms.my_empty_row = -1;
                ms.my_slots_from = piece == 0 ? fixed_np : S;
                ms.my_piece = piece;
                ms.my_t0 = piece * nt / fixed_np;
                ms.my_nt = (piece + 1) * nt / fixed_np - ms.my_t0;
                ms.my_p = q < R ? a.q_pos[q] : 0;
                ms.my_np = fixed_np;
            }
        } else {
            const SchedIn si{a.q_pos, a.Ncap, R, a.m, a.k, a.is_csa};
            if (R <= 32) {
                if constexpr (F8) piece_schedule_rows32_ool(si, S, nt_w, ms, lane);
                else piece_schedule_rows32(si, S, nt_w, ms, lane);
            } else {
                piece_schedule(si, S, nt_w, ms, lane);
            }
        }
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = ms.tmem_base;
    const uint32_t t_o = tmem + 2 * H;
    const uint32_t sbase = smem_u32(sm);
    // next work item of this CTA (cursor `cur`: an item index; with the piece schedule 0 before
    // and 1 after the CTA's piece); tile range [t0, t0 + nt) of the row's tile space:
    // compressed tiles first, then the window
    auto next_item = [&](int& cur, ItemTiles& it) -> bool {
        if (pieces) {
            if (cur != 0 || ms.my_row < 0) return false;
            cur = 1;
            it.r = ms.my_row;
            it.t0 = ms.my_t0;
            it.nt = ms.my_nt;
            it.slot = ms.my_piece;
            it.p = ms.my_p;
            it.expect = ms.my_np;
        } else {
            if (cur >= items) return false;
            it.r = cur / S;
            it.slot = cur % S;
            it.t0 = it.slot * tps;
            it.expect = S;
            cur += gridDim.x;
            it.p = a.q_pos[it.r];
        }
        it.b = it.r / a.T;
        it.kl = key_list(a, it.r, it.b, it.p);
        it.nt_c = (int)cdiv(it.kl.n_c, kKeys);
        if (!pieces) {
            const int t1 = min(it.nt_c + nt_w, it.t0 + tps);
            it.nt = t1 > it.t0 ? t1 - it.t0 : 0;
        }
        return true;
    };
    const int cur0 = pieces ? 0 : (int)blockIdx.x;

    if (warp == kSoft / 32) {
        // ========================================================================= MMA warp
        // Order per item: MMA1(0), MMA1(1), then PV(i), MMA1(i+2) for each tile i.  MMA1(i+2)
        // overwrites the S buffer of tile i, which the softmax has read once P(i) is ready.
        if (lane == 0) {
            const uint32_t id_qk = idesc_f16(128, H, 1, 0, 0);
            const uint32_t id_pv = idesc_f16(128, H, 1, 1, 1);
            const uint64_t q_desc = smem_desc(sbase + L::q, 16, 1024);
            const uint64_t p_desc = smem_desc(sbase + L::p, L::p_region, 1024);
            uint32_t g = 0;
            ItemTiles it;
            for (int cur = cur0; next_item(cur, it);) {
                const int nt = it.nt;
                if (nt == 0) continue;
                // step s: PV(s - 2) (s >= 2), then MMA1(s) (s < nt)
#pragma unroll 1
                for (int st = 0; st < nt + 2; ++st) {
                    if (st >= 2) {              // O^T += V^T . P(i)
                        const int i = st - 2;
                        const uint32_t seq = g + (uint32_t)i;
                        mbar_wait(&ms.pready, seq & 1, err);
                        mbar_wait(&ms.vfull[seq & 1], (seq >> 1) & 1, err);
                        fence_proxy_async();
                        fence_after_sync();
                        const uint64_t v_desc = smem_desc(sbase + L::v + (seq & 1) * kTile, kHalf, 1024);
                        const uint64_t pb_desc = p_desc + (uint64_t)(((seq & 1) * L::p_bytes) >> 4);
                        constexpr uint64_t lo_off = (uint64_t)((L::p_lo - L::p) >> 4);
#pragma unroll
                        for (int j = 0; j < 16; ++j)      // P = P_hi + P_lo: 8 K steps each
                            mma_ss(t_o, v_desc + (uint64_t)(((j & 7) * 2048) >> 4),
                                   pb_desc + (j >= 8 ? lo_off : 0) + (uint64_t)(((j & 7) * 2048) >> 4), id_pv,
                                   (i > 0 || j > 0) ? 1u : 0u);
                        mma_commit(&ms.odone);
                    }
                    if (st < nt) {              // S^T(st) = K(st) . Q^T into S buffer (g + st) & 1
                        const uint32_t seq = g + (uint32_t)st;
                        mbar_wait(&ms.kfull[seq & 1], (seq >> 1) & 1, err);
                        fence_proxy_async();
                        fence_after_sync();
                        const uint64_t k_desc = smem_desc(sbase + L::k + (seq & 1) * kTile, 16, 1024);
                        const uint32_t sb = tmem + (seq & 1) * H;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            mma_ss(sb, k_desc + (uint64_t)(((j >> 2) * kHalf + (j & 3) * 32) >> 4),
                                   q_desc + (uint64_t)(((j >> 2) * L::q_half + (j & 3) * 32) >> 4), id_qk, j > 0);
                        mma_commit(&ms.sdone[seq & 1]);
                    }
                }
                g += (uint32_t)nt;
            }
        }
        __syncwarp();
    } else {
        // ==================================================================== softmax warps
        constexpr int HG = kHG;                     // heads per warpgroup
        const int wg = warp >> 2;                   // warpgroup: heads [wg*HG, wg*HG + HG)
        const int row = tid & (kKeys - 1);          // key row of S^T / dim row of O^T = TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        const float c_log2 = a.scale * 1.4426950408889634f;      // scale > 0 (checked on the host)
        const uint64_t pol_stream = l2_policy_evict_first();     // K/V rows are read once per step
        uint32_t g = 0;                                          // tiles processed so far by this CTA

        if (pieces && ms.my_empty_row >= 0) {      // a row without keys: o = 0, lse = -inf
            const int64_t er = ms.my_empty_row;
            uint4* orow = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + er * H * kD);
            for (int i = tid; i < H * kD / 8; i += kSoft) orow[i] = make_uint4(0u, 0u, 0u, 0u);
            if (a.lse && tid < H) a.lse[er * H + tid] = -INFINITY;
        }
        // After an item's partial is written: count the arrival at its row (one acquire-release
        // atomic, cumulative over the barrier); the row's last item merges the row's partial results
        // exactly, slots s = 0, 1, ... in that order (slots with lse = -inf hold no keys):
        //     lse = log sum_s exp(lse_s),  o = sum_s exp(lse_s - lse) o_s,
        // and resets the counter (merge_row).
        uint32_t mpass = 0;                         // merge passes so far (the mfull barrier's phase)
        auto arrive_and_merge = [&](const ItemTiles& itm) {
            named_barrier_sync(1, kSoft);
            if (tid == 0) {
                // acq_rel: releases this CTA's partial (the barrier above orders every thread's
                // stores before it) and, for the last arrival, acquires the other items' partials
                unsigned before;
                asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                             : "=r"(before) : "l"(&row_cnt[itm.r]) : "memory");
                ms.merge_now = before + 1u == (unsigned)itm.expect;
            }
            named_barrier_sync(1, kSoft);
            if (!ms.merge_now) return;
            merge_row<H>(itm.r, itm.expect, S, lse_part, o_part, static_cast<__nv_bfloat16*>(a.out), a.lse, ms,
                         tid, sbase + L::p, mpass, err);
            if (tid == 0) row_cnt[itm.r] = 0u;             // ready for the next call
        };
        ItemTiles it;
        for (int cur = cur0; next_item(cur, it);) {
            const int r = it.r, b = it.b, nt_c = it.nt_c, t0 = it.t0, nt = it.nt;
            const int64_t p = it.p;
            const KeyList kl = it.kl;
            const int64_t obase = ((int64_t)r * S + it.slot) * H;
            const __nv_bfloat16* qr = static_cast<const __nv_bfloat16*>(a.q) + (int64_t)r * H * kD;

            if (nt == 0) {                       // a slot without keys: o = 0 (finite), lse = -inf
                if (direct) {
                    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) + obase * kD;
                    for (int i = tid; i < H * kD; i += kSoft) orow[i] = __float2bfloat16(0.0f);
                    if (a.lse && tid < H) a.lse[obase + tid] = -INFINITY;
                } else {
                    for (int i = tid; i < H * kD; i += kSoft) o_part[obase * kD + i] = 0.0f;
                    if (tid < H) lse_part[obase + tid] = -INFINITY;
                }
                if (pieces) arrive_and_merge(it);
                continue;
            }
            if (tid < H) ms.mrun[tid] = -INFINITY;

            // Tile i's loads are the (g + i)-th of each ring, so slot = (g + i) & 1.
            // (FP8 caches: every load completes on k8full / v8full, the converters pass it on)
            int32_t e_next = kNoEntry;               // (CSA) this thread's row's entry of the next K gather
            auto load = [&](int i, bool is_v) {
                const uint32_t seq = g + (uint32_t)i;
                const uint32_t dst = sbase + (is_v ? L::v : L::k) + (seq & 1) * kTile;
                uint64_t* bar = F8 ? (is_v ? &ms.v8full[seq & 1] : &ms.k8full[seq & 1])
                                   : (is_v ? &ms.vfull[seq & 1] : &ms.kfull[seq & 1]);
                if (F8 && t0 + i < nt_c)
                    load_tile_f8<kSoft>(a, maps, use_tma_c, r, b, kl.n_c, t0 + i, is_v, dst,
                                        sbase + L::total + (seq & 1) * kVScale, bar, ms.valid[seq & 3], qr, pol_stream,
                                        i == 0 && !is_v, err);
                else
                    load_tile<kSoft>(a, maps, use_tma_c, use_tma_w, r, b, p, kl.n_c, kl.total, nt_c, t0 + i, is_v,
                                     dst, bar, ms.valid[seq & 3], qr, pol_stream, i == 0 && !is_v, err,
                                     is_v ? nullptr : ms.eidx[seq & 3],
                                     (is_v && i > 0) ? ms.eidx[seq & 3] : nullptr,   // (V(0): its K record is
                                     is_v ? kNoEntry : e_next);                       //  not visible yet)
            };
            // CSA gathers: the entry of this thread's row in the tile after next, loaded one tile
            // ahead (the K gather then issues without waiting on the index list)
            const int kTprL = kSoft / kKeys;
            auto entry_ahead = [&](int i) -> int32_t {
                const int64_t key = (int64_t)(t0 + i) * kKeys + tid / kTprL;
                if (F8 || !a.is_csa || i >= nt || t0 + i >= nt_c || key >= kl.n_c) return kNoEntry;
                return a.idx[(int64_t)r * a.k + key];
            };

            // FP8 caches: tile i's codes -> bf16 in place by the softmax warps, then the tile is
            // released to the MMA warp (K: before MMA1 needs it; V: with the tile's zeroing of rows
            // that hold no key, before PV)
            constexpr int kTpr = kSoft / kKeys;
            auto conv = [&](int i, bool is_v, bool zero_invalid) {
                const uint32_t seq = g + (uint32_t)i;
                mbar_wait(is_v ? &ms.v8full[seq & 1] : &ms.k8full[seq & 1], (seq >> 1) & 1, err);
                const uint32_t slot = sbase + (is_v ? L::v : L::k) + (seq & 1) * kTile;
                const int cr = tid / kTpr, cp = tid % kTpr;
                const bool zr = zero_invalid && ms.valid[seq & 3][cr] == 0;
                if (t0 + i < nt_c) {
                    if (is_v) convert_v_part<kTpr>(slot, sbase + L::total + (seq & 1) * kVScale, cr, cp, zr);
                    else convert_k_part<kTpr>(slot, sbase + L::total + (seq & 1) * kVScale, cr, cp);
                } else if (is_v && zr) {
                    zero_v_part<kTpr>(slot, cr, cp);
                }
                fence_proxy_async();
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(is_v ? &ms.vfull[seq & 1] : &ms.kfull[seq & 1]);
            };

            // ---- prologue: Q, K(0), K(1), V(0) in flight (K(0) completes only once Q has landed)
            for (int c = tid; c < H * 16; c += kSoft) {
                const int h = c >> 4, cc = c & 15;
                cp_async16(sbase + L::q + (cc >> 3) * L::q_half + sw128(h, cc & 7), qr + h * kD + cc * 8, 16);
            }
            e_next = kNoEntry;
            load(0, false);
            if (nt > 1) load(1, false);
            load(0, true);
            e_next = entry_ahead(2);
            named_barrier_sync(1, kSoft);                  // valid[] of tiles 0 and 1
            if constexpr (F8) conv(0, false, false);

            float lsum[HG];
#pragma unroll
            for (int h = 0; h < HG; ++h) lsum[h] = 0.0f;

#pragma unroll 1
            for (int i = 0; i < nt; ++i) {
                const uint32_t seq = g + (uint32_t)i;
                const int ti = t0 + i;
                if constexpr (F8)
                    if (i + 1 < nt) conv(i + 1, false, false);   // K(i+1): loaded one tile ago
                mbar_wait(&ms.sdone[seq & 1], (seq >> 1) & 1, err);
                fence_after_sync();
                // Each thread holds one key row of this warpgroup's 16 heads (raw scores; rows that
                // are not keys of the query give p = 0).
                const bool valid = ms.valid[seq & 3][row] != 0;
                const uint32_t scol = tmem + (seq & 1) * H + wg * HG + lane_off;
                // P buffer (i & 1): its last reader PV(i-2) precedes MMA1(i) and is complete
                const uint32_t prow = sbase + L::p + (seq & 1) * L::p_bytes + ((wg * HG / 8) >> 3) * L::p_region;
                const int pchunk = (wg * HG / 8) & 7;                 // 8 heads per 16-byte chunk
                // P goes to the MMA as two bf16 parts, P_hi = bf16(P) and P_lo = bf16(P - P_hi), so the
                // products P V keep about 16 significant bits of P
                auto store_p = [&](const float* pp16) {
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        hi[k] = pack_bf16x2(pp16[2 * k], pp16[2 * k + 1]);
                        lo[k] = pack_bf16x2(pp16[2 * k] - __uint_as_float(hi[k] << 16),
                                            pp16[2 * k + 1] - __uint_as_float(hi[k] & 0xFFFF0000u));
                    }
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(prow + sw128(row, pchunk + c)),
                                     "r"(hi[4 * c]), "r"(hi[4 * c + 1]), "r"(hi[4 * c + 2]), "r"(hi[4 * c + 3])
                                     : "memory");
                        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};"
                                     ::"r"(prow + (L::p_lo - L::p) + sw128(row, pchunk + c)),
                                     "r"(lo[4 * c]), "r"(lo[4 * c + 1]), "r"(lo[4 * c + 2]), "r"(lo[4 * c + 3])
                                     : "memory");
                    }
                };
                // K slot of tile i is free (MMA1(i) complete)
                if (i + 2 < nt) load(i + 2, false);
                e_next = entry_ahead(i + 3);
                // ---- P = 2^(s c - m) with the running maxima m, exponents capped at the threshold.
                // When some score exceeds its head's running maximum by more than the threshold
                // (always on an item's first tile, which skips this pass) the maxima are raised
                // and P is formed again below.
                bool grow = true;
                if (i > 0) {
                    uint32_t rr[16];
                    float pp[16];
                    tmem_ld16(scol, rr);
                    tmem_wait_ld();
                    bool need = false;
#pragma unroll
                    for (int k = 0; k < 16; k += 4) {
                        const float4 m4 = *reinterpret_cast<const float4*>(&ms.mrun[wg * HG + k]);
                        const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float x = __uint_as_float(rr[k + u]) * c_log2;
                            need |= x > mm[u] + kRescaleThreshold;
                            pp[k + u] = (mm[u] == -INFINITY || !valid) ? 0.0f
                                                                       : ex2_approx(fminf(x - mm[u], kRescaleThreshold));
                            lsum[k + u] += pp[k + u];
                        }
                    }
                    store_p(pp);
                    grow = named_barrier_or(2 + wg, 128, need && valid);   // this warpgroup's heads
                }
                // everyone is done with tile i-1's flag (the barrier above, or on an item's first
                // tile the previous item's closing barriers)
                if ((tid & 127) == 0) ms.flag[wg][(seq + 1) & 1] = 0;
                bool rescale = false;
                if (grow) {
                    // tile maxima per head: a warp reduction, then a 4-way merge over the warpgroup
                    float mine = -INFINITY;
                    {
                        uint32_t rr[16];
                        tmem_ld16(scol, rr);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            const float mx = redux_max_f32(valid ? __uint_as_float(rr[k]) : -INFINITY);
                            mine = (lane == k) ? mx : mine;
                        }
                    }
                    ms.red[warp][lane] = mine;
                    // (the warpgroup owns its heads' maxima: its own barriers suffice)
                    named_barrier_sync(2 + wg, 128);
                    if ((tid & 127) < HG) {
                        const int hh = tid & 127, hd = wg * HG + hh;
                        const float traw = fmaxf(fmaxf(ms.red[4 * wg][hh], ms.red[4 * wg + 1][hh]),
                                                 fmaxf(ms.red[4 * wg + 2][hh], ms.red[4 * wg + 3][hh]));
                        const float tmax = traw * c_log2;
                        const float mo = ms.mrun[hd];
                        float al = 1.0f;
                        if (tmax > mo + kRescaleThreshold || (mo == -INFINITY && tmax != -INFINITY)) {
                            al = (mo == -INFINITY) ? 0.0f : ex2_approx(mo - tmax);
                            ms.mrun[hd] = tmax;
                            ms.flag[wg][seq & 1] = 1;
                        }
                        ms.mold[hd] = mo;
                        ms.alpha[hd] = al;
                    }
                    named_barrier_sync(2 + wg, 128);
                    rescale = ms.flag[wg][seq & 1] != 0;
                    // P again with the new maxima; the row sums drop the first pass's term
                    // (recomputed exactly as it was added) and are rescaled
                    uint32_t rr[16];
                    float pp[16];
                    tmem_ld16(scol, rr);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; k += 4) {
                        const int h = wg * HG + k;
                        const float4 m4 = *reinterpret_cast<const float4*>(&ms.mrun[h]);
                        const float4 o4 = *reinterpret_cast<const float4*>(&ms.mold[h]);
                        const float4 a4 = *reinterpret_cast<const float4*>(&ms.alpha[h]);
                        const float mn[4] = {m4.x, m4.y, m4.z, m4.w};
                        const float mo[4] = {o4.x, o4.y, o4.z, o4.w};
                        const float al[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float x = __uint_as_float(rr[k + u]) * c_log2;
                            const float pold = (i == 0 || mo[u] == -INFINITY || !valid)
                                                   ? 0.0f
                                                   : ex2_approx(fminf(x - mo[u], kRescaleThreshold));
                            pp[k + u] = (mn[u] == -INFINITY || !valid) ? 0.0f : ex2_approx(x - mn[u]);
                            lsum[k + u] = fmaf(lsum[k + u] - pold, al[u], pp[k + u]);
                        }
                    }
                    store_p(pp);
                }
                // ---- PV(i-1) done: O and the V slot of tile i-1 are free
                if (i > 0) {
                    mbar_wait(&ms.odone, (seq - 1) & 1, err);
                    fence_after_sync();
                }
                if (i + 1 < nt) load(i + 1, true);
                // ---- rescale the O^T accumulator (lane = dim) when some running maximum moved
                if (rescale && i > 0) {
#pragma unroll
                    for (int c0 = 0; c0 < HG; c0 += 16) {
                        uint32_t rr[16];
                        const uint32_t oa = t_o + wg * HG + c0 + lane_off;
                        tmem_ld16(oa, rr);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            rr[k] = __float_as_uint(__uint_as_float(rr[k]) * ms.alpha[wg * HG + c0 + k]);
                        tmem_st16(oa, rr);
                    }
                    tmem_wait_st();
                }
                // ---- a TMA tile may hold rows that are not keys of this query (entries not yet
                // visible, the next sequence, ring slots before token 0): zero their V rows, since
                // P = 0 does not cancel a non-finite value.
                const bool comp = ti < nt_c;
                const bool vzero = comp ? (use_tma_c && (int64_t)(ti + 1) * kKeys > kl.n_c)
                                        : (use_tma_w && p < kKeys - 1);
                if constexpr (F8) {
                    conv(i, true, vzero);
                } else if (vzero) {
                    mbar_wait(&ms.vfull[seq & 1], (seq >> 1) & 1, err);
                    if (tid < kKeys && !valid) {
                        const uint32_t vrow = sbase + L::v + (seq & 1) * kTile + row * 128;
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(vrow + c * 16), "r"(0u)
                                         : "memory");
                            asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(vrow + kHalf + c * 16),
                                         "r"(0u)
                                         : "memory");
                        }
                    }
                }
                // ---- P(i) and O ready for PV(i)
                fence_proxy_async();
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ms.pready);
            }
            // ---- row sums across the 128 keys and the partial lse (while the last PV runs), then
            // the normalised partial output
            float mine = 0.0f;
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                const float sum = warp_sum(lsum[h]);
                mine = (lane == h) ? sum : mine;
            }
            ms.red[warp][lane] = mine;
            named_barrier_sync(1, kSoft);
            if (tid < H) {
                const int gq = tid / HG, hh = tid % HG;
                const float l = ms.red[4 * gq][hh] + ms.red[4 * gq + 1][hh] + ms.red[4 * gq + 2][hh] +
                                ms.red[4 * gq + 3][hh];
                const float m = ms.mrun[tid];
                const bool any = (l > 0.0f) && (m != -INFINITY);
                ms.linv[tid] = any ? 1.0f / l : 0.0f;
                const float lse = any ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
                if (!direct) lse_part[obase + tid] = lse;
                else if (a.lse) a.lse[obase + tid] = lse;
            }
            named_barrier_sync(1, kSoft);
            mbar_wait(&ms.odone, (g + (uint32_t)nt - 1) & 1, err);
            fence_after_sync();
            g += (uint32_t)nt;
#pragma unroll
            for (int c0 = 0; c0 < HG; c0 += 16) {
                uint32_t rr[16];
                tmem_ld16(t_o + wg * HG + c0 + lane_off, rr);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int h = wg * HG + c0 + k;
                    const float o = __uint_as_float(rr[k]) * ms.linv[h];
                    if (direct) static_cast<__nv_bfloat16*>(a.out)[(obase + h) * kD + row] = __float2bfloat16(o);
                    else o_part[(obase + h) * kD + row] = o;
                }
            }
            fence_before_sync();
            if (pieces) arrive_and_merge(it);
            else named_barrier_sync(1, kSoft);
        }
    }
    __syncwarp();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, kCols);
}

// --------------------------------------------------------------------------- host side
// Map over `rows` rows of 128 bf16 (256-byte pitch), boxes of 64 columns x 128 rows (the layout of
// the MMA operands).  False when the map cannot be made; the caller then gathers rows instead.
bool encode_rows(CUtensorMap* m, const void* base, int64_t rows) {
    return rows > 0 && encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, kD, (uint64_t)rows, kD * 2, 64, kKeys);
}

template <int H, bool F8>
cudaError_t launch_tc(const AttendArgs& a, int S, int kps, float* o_part, float* lse_part, unsigned* row_cnt,
                      unsigned* err, cudaStream_t st) {
    Maps maps;
    std::memset(&maps, 0, sizeof maps);
    int use_c = 0, use_w = 0;
    // HCA entries of a sequence are contiguous; CSA entries are gathered through the index list.
    const uint64_t crows = (uint64_t)a.B * (uint64_t)a.Ncap;
    if (!a.is_csa && !F8 && encode_rows(&maps.ck, a.ck, (int64_t)crows) && encode_rows(&maps.cv, a.cv, (int64_t)crows))
        use_c = 1;
    if (!a.is_csa && F8 &&
        encode_tmap_2d_sw(&maps.k8, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.ck, 128, crows, kKv8KRow, 128, kKeys,
                          CU_TENSOR_MAP_SWIZZLE_NONE) &&
        encode_tmap_2d_sw(&maps.kr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<const char*>(a.ck) + kKv8Rope, 64,
                          crows, kKv8KRow, 64, kKeys, CU_TENSOR_MAP_SWIZZLE_128B) &&
        encode_tmap_2d_sw(&maps.v8, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.cv, 128, crows, kKv8VRow, 128, kKeys,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
        use_c = 1;
    // The decode window is the whole ring when it holds exactly one tile of tokens.
    if (a.chunk_k == nullptr && a.W == kKeys && a.ring_cap == kKeys && a.ring_k != nullptr &&
        encode_rows(&maps.rk, a.ring_k, (int64_t)a.B * a.ring_cap) &&
        encode_rows(&maps.rv, a.ring_v, (int64_t)a.B * a.ring_cap))
        use_w = 1;
    const size_t smem = Smem<H>::total + (F8 ? 2 * kVScale : 0) + 1024;
    auto kern = attend_tc_kernel<H, F8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int R = a.B * a.T;
    const int items = R * S;
    const int grid = items < num_sms() ? items : num_sms();
    // CSA rows all hold k + W keys: the piece schedule is the same for every row and is made here
    // (the kernel's own schedule, with all rows' tile counts equal)
    int fixed_np = 0;
    if (a.is_csa && R <= kSchedRows && R <= grid && S >= 2) {
        const int nt = (int)(cdiv(a.k, kKeys) + cdiv(a.W, kKeys));
        if (nt > 0) {
            int len = std::max(std::max((int)cdiv((int64_t)R * nt, grid), (int)cdiv(nt, S)), 1);
            while ((int64_t)R * cdiv(nt, len) > grid) ++len;
            fixed_np = (int)cdiv(nt, len);
        }
    }
    (void)launch_pdl(kern, dim3(grid), dim3(Thr<H, F8>::kThreads), smem, st, a, S, kps, maps, use_c, use_w, fixed_np,
                     o_part, lse_part, row_cnt, err);
    return cudaGetLastError();
}

}  // namespace

bool attend_tc_merges(const AttendArgs& a, int S) {
    // the kernel's piece schedule (few rows) merges in the row's last CTA; with many rows every
    // CTA takes (row, split) items and the shared merge kernel follows (it spreads the merges of
    // many rows over the whole GPU), unless a row is one split, written out directly
    const int R = a.B * a.T;
    const int items = R * S;
    const int grid = items < num_sms() ? items : num_sms();
    return S == 1 || (R <= kSchedRows && R <= grid && S >= 2);
}

bool attend_tc_supported(const AttendArgs& a) {
    return (a.dtype == CSAHCA_BF16 || a.dtype == CSAHCA_KV_FP8) && a.d == 128 && (a.H == 32 || a.H == 64) &&
           a.scale > 0.0f && aligned(a.out, 16);
}

cudaError_t attend_tc_launch(const AttendArgs& a, int S, int kps, float* o_part, float* lse_part, unsigned* row_cnt,
                             unsigned* err, cudaStream_t st) {
    switch (a.H) {
        case 32:
            return a.dtype == CSAHCA_KV_FP8 ? launch_tc<32, true>(a, S, kps, o_part, lse_part, row_cnt, err, st)
                                            : launch_tc<32, false>(a, S, kps, o_part, lse_part, row_cnt, err, st);
        case 64:
            return a.dtype == CSAHCA_KV_FP8 ? launch_tc<64, true>(a, S, kps, o_part, lse_part, row_cnt, err, st)
                                            : launch_tc<64, false>(a, S, kps, o_part, lse_part, row_cnt, err, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace csahca
