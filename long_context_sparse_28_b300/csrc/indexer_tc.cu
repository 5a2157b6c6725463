// Tensor-core lightning-indexer scores for low-precision keys (e2m1 + UE8M0 per 32 values,
// e4m3 + fp32 row scale), d_I = 64, any number of query rows.
//
// I(t,s) = sum_h w[t,h] * ReLU(q[t,h] . khat_s)  (honbul.tistory.com/221 "CSA"; pogovet.com
// DeepSeek-V4 article, detail 4 (FP4 lightning indexer) and detail 5).
//
// The key codes are never decoded on the CUDA cores: the 5th-generation tensor core multiplies
// them as they are stored (tcgen05.mma kind::f8f6f4, A = e2m1 or e4m3 codes).  A stage holds 256
// keys of one query row: one 2-D TMA box of 128 rows x 128 codes, each row two consecutive keys
// (packed e2m1 codes are expanded by the TMA into the 16-byte-per-16-codes shared-memory form the
// MMA reads; e4m3 codes are copied as bytes), 128-byte swizzle.  With M = 128 rows, the MMA over
// code columns [0, 64) gives the even keys and over [64, 128) the odd keys.
//
// The query must be an 8-bit operand too.  Each bf16 head vector is scaled by a power of two 2^e_h
// (largest element into [2^7, 2^8)) and split exactly as q' = hi + 2^-5 lo with hi = e4m3(q') and
// lo = 32 (q' - hi): the remainder has at most 3 significant bits, so lo is an e4m3 value.  The
// B operand stacks the hi rows over the lo rows (N = 2 H_I), so one MMA per 32-code block gives
// both parts.  (Elements below 2^-13 of their head's largest element are the exception: lo is
// then rounded, an error below 2^-20 of that largest element; so are heads whose largest element
// is below 2^-114, whose exponent is capped.)
//   e2m1 keys (UE8M0 per 32 codes): the MMA applies every scale (kind::mxf8f6f4 block_scale): a
//     key's factor for its code block is the A scale of its row; the hi rows' blocks multiply with
//     the B factor 2^-e_h and the lo rows' blocks -- issued as further MMAs into the same
//     accumulator columns -- with 2^-(e_h+5) (bytes 0-1 / 2-3 of the head's factor word), so the
//     accumulator of a key holds q . khat per head directly (one column per head) and the epilogue
//     forms score = sum_h w_h ReLU(D[h]).  The scale
//     factors reach TMEM with tcgen05.cp, which wants an M = 128 operand's factors as 32 lines of
//     16 bytes (row r's four bytes -- even key blocks 0/1, odd key blocks 0/1 -- in word r / 32 of
//     line r % 32).  The codes are therefore loaded with a 4-D TMA map that puts TMA row 4 l + j
//     of a stage into MMA row 32 j + l: the stage's 512 scale bytes, bulk-copied as they are
//     stored, are then already that image (keys need Ncap % 256 == 0).  The producer writes the
//     query's factors with its image.
//   e4m3 keys (fp32 row scale): kind::f8f6f4; 2^-e_h is folded into the head weight w' and the
//     row scale applied in the epilogue: score = s_key sum_h w'_h ReLU(D_hi[h] + 2^-5 D_lo[h]).
// The epilogue works on pairs of heads with f32x2 arithmetic.  Apart from the exceptions above the
// result differs from exact arithmetic only by the rounding of the fp32 accumulation.
//
// Warp roles (persistent CTAs over (row, chunk of 8 stages) work items):
//   warp 4     producer: per work item, the q image and folded head weights of its row into one of
//              two query slots (the next item's row is loaded one item ahead); per stage (one lane)
//              the stage's (row, first key, visible count, flags) record, the TMA box of codes and
//              a bulk copy of the scales;
//   warps 5-6  MMA warps, taking alternate stages (their per-stage waits and issue overlap): hand the
//              stage's record to the epilogue through the accumulator buffer's slot, then one thread
//              copies the stage's scale factors (and a new query's) into TMEM and issues the MMAs
//              into the buffer (up to four buffers, as TMEM allows);
//   warps 0-3  epilogue: thread j owns TMEM lane j (two consecutive keys of the stage): scores to
//              global memory, and the top-12-bit histogram of the scores (the top-k's first pass),
//              accumulated per piece in shared memory (16-bit counts; a piece has at most 128
//              stages) and added to the row's global histogram.
#include "common.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

#include <algorithm>
#include <cstddef>
#include <cstring>

namespace csahca {
namespace {

using namespace tc;

constexpr int kPair = 256;            // keys per stage (128 TMA rows of two keys)
constexpr int kDI = 64;
constexpr int kChunkStages = 8;       // stages per work item: 2048 keys of one query row
constexpr int kMaxNS = 6;             // shared-memory stages (at most)
constexpr int kEpi = 128;             // epilogue threads (warps 0-3)
constexpr int kMaxMmaWarps = 5;       // MMA-issuing warps (at most), taking the stages in turn
// stage flags: no more work (kFirstTerm: the record the epilogue receives) / last stage of a piece
constexpr int kTerm = 1, kLast = 2, kFirstTerm = 4;
// Longest piece: its keys' histogram is kept in 16-bit shared-memory counts until the piece ends
constexpr int kMaxPieceStages = 128;  // 32768 keys
enum : uint32_t { kE4M3 = 0, kE2M1 = 5 };   // kind::f8f6f4 operand formats
constexpr float kLoScale = 0.03125f;         // lo rows of the query operand carry 32 x the remainder

constexpr int kSchedRows = 256;       // balanced piece schedule for up to this many query rows
constexpr int kMaxBuf = 5;            // TMEM accumulator buffers (at most)

struct alignas(16) IdxMisc {
    alignas(16) uint32_t hist[2048];      // top-12-bit histogram of the scores since the last flush:
                                          // bin b is the 16-bit half (b & 1) of word b >> 1 (at most
                                          // kMaxPieceStages x 256 keys); read and cleared as uint4
    alignas(16) int4 dmeta[kMaxBuf];      // record of the stage in each accumulator buffer
    uint64_t full[kMaxNS], empty[kMaxNS], dfull[kMaxBuf], dfree[kMaxBuf], qfree[2];
    uint32_t tmem_base;
    int soff[kSchedRows + 1];             // piece schedule: first stage of each row (producer only)
    int nvis[kSchedRows];                 // and its visible entries
};
static_assert(offsetof(IdxMisc, hist) % 16 == 0 && offsetof(IdxMisc, full) % 8 == 0, "IdxMisc alignment");

template <int FMT, int HI, bool Q4 = false>
struct Cfg {
    static constexpr bool fp4 = FMT == CSAHCA_E2M1_UE8M0;            // block scales applied by the MMA
    static constexpr int NQ = Q4 ? HI : 2 * HI;                      // B rows: FP4 queries, or hi + lo rows
    static constexpr uint32_t code_tx = fp4 ? kPair * 32 : kPair * 64;  // global code bytes per stage
    static constexpr int scale_bytes = fp4 ? 2 : 4;                  // per key
    // stage: codes (128 rows x 128 B, swizzled) | scales (e4m3: 1 KB; fp4: the 512-byte factor
    // image at off_sfa) | record
    static constexpr uint32_t off_scale = 16384;
    static constexpr uint32_t off_sfa = off_scale + 512;
    static constexpr uint32_t off_meta = off_scale + kPair * 4;
    static constexpr uint32_t stage = (off_meta + 16 + 1023) / 1024 * 1024;
    // query slot (one per work item, two in flight): q image (2 HI rows x 128 B: hi rows, then
    // lo rows, codes in the first 64 bytes) | head weights | (fp4) the B scale-factor image
    static constexpr uint32_t q_img = NQ * 128;
    static constexpr uint32_t off_sfb = (q_img + HI * 4 + 15) / 16 * 16;
    static constexpr uint32_t q_slot = ((fp4 ? off_sfb + 512 : q_img + HI * 4) + 1023) / 1024 * 1024;
    // as many stages as leave room for two CTAs per SM (228 KB, 1 KB reserved per CTA, 1 KB
    // alignment slack, the static shared memory)
    static constexpr int ns_fit = (int)((114 * 1024 - 1024 - 1024 - sizeof(IdxMisc) - 2 * q_slot -
                                         (fp4 ? 0 : kMaxBuf * kPair * 4)) / stage);
    static constexpr int ns_cap = ns_fit < 3 ? 3 : (ns_fit > kMaxNS ? kMaxNS : ns_fit);
    // e2m1 keys with bf16 queries: the MMA adds the lo part into the hi part's accumulator (its own
    // B scale factor 2^-(e_h+5) in bytes 2-3 of the head's factor word), one column per head
    static constexpr bool fused = fp4 && !Q4;
    static constexpr bool one_part = fused || Q4;                    // one accumulator column per head
    static constexpr uint32_t acc_cols = one_part ? HI : NQ;         // hi | lo columns (e4m3 keys)
    static constexpr uint32_t d_cols = 2 * acc_cols;                 // even + odd keys
    // fp4: scale factors of A (4 columns per stage slot) and B (4 per query slot)
    static constexpr uint32_t sf_cols = fp4 ? 4 * kMaxNS + 8 : 0;
    // accumulator buffers: the MMA of a stage waits for the epilogue to have read the buffer of the
    // stage nbuf earlier, so more buffers keep more stages between the two in flight; as many as
    // fit in 256 columns (two CTAs per SM), else in 512
    static constexpr int fit256 = (int)((256 - sf_cols) / d_cols), fit512 = (int)((512 - sf_cols) / d_cols);
    static constexpr int nbuf_fit = fit256 >= 2 ? (fit256 < kMaxBuf ? fit256 : kMaxBuf)
                                                : (fit512 < kMaxBuf ? (fit512 < 1 ? 1 : fit512) : kMaxBuf);
    // NMW MMA warps take the stages in turn (warp u % NMW issues stage u).  An mbarrier wait on a
    // phase parity is only sound when its waiter consumes the barrier's phases one after another,
    // so each warp must own its own stage slots and accumulator buffers: both counts multiples of
    // NMW (stage u: slot u % NS and buffer u % nbuf are congruent to u mod NMW).  Five warps with
    // one slot and one buffer each where five of both fit (a slot count two warps cannot share
    // evenly) and the queries are bf16 (two operand parts per stage; with FP4 queries a stage is
    // half the MMA work and five warps measured slower), else two warps, or one with a single buffer.
    static constexpr int NMW = (!Q4 && ns_cap >= 5 && nbuf_fit >= 5) ? 5 : nbuf_fit >= 2 ? 2 : 1;
    static constexpr int nbuf = nbuf_fit / NMW * NMW;
    static constexpr int NS = ns_cap / NMW * NMW;
    static_assert(NMW <= kMaxMmaWarps && NS >= NMW && nbuf >= NMW && NS % NMW == 0 && nbuf % NMW == 0,
                  "stage slots and buffers per MMA warp");
    static constexpr int threads = kEpi + 32 + 32 * NMW;   // + producer warp + MMA warps
    static constexpr uint32_t off_qslots = NS * stage;
    // e4m3: the row scales of the stage in each accumulator buffer (copied by the MMA warp)
    static constexpr uint32_t off_dscale = off_qslots + 2 * q_slot;
    static constexpr uint32_t smem = off_dscale + (fp4 ? 0 : kMaxBuf * kPair * 4);
    static constexpr uint32_t sfa_col = nbuf * d_cols, sfb_col = sfa_col + 4 * kMaxNS;
    static constexpr uint32_t used_cols = nbuf * d_cols + sf_cols;
    static constexpr uint32_t tmem_cols = used_cols <= 32 ? 32 : used_cols <= 64 ? 64 : used_cols <= 128 ? 128
                                          : used_cols <= 256 ? 256 : 512;
    static_assert(used_cols <= 512, "TMEM columns");
    static_assert(HI % 16 == 0 && HI <= 64, "heads");
    static_assert(!fp4 || off_sfa + 512 <= off_meta, "fp4 stage layout");
    static_assert(!Q4 || fp4, "FP4 queries go with FP4 keys");
    // the next item's query row is loaded one item ahead when its share fits in a few registers
    static constexpr bool prefetch_q = HI <= 16;
};

// One lane's share of the q image of a row: unit (head h, half hf) = lane + 32 j covers 32
// elements of head h and yields two 16-byte chunks of hi codes and two of lo codes (lo = 32 x the
// remainder, e4m3); returns the head's exponent e_h in exq[j] and its weight in wq[j] (with FOLD,
// the folded weight w_h 2^-e_h).  `raw` holds the unit's 32 values.
template <int HI, bool FOLD>
__device__ __forceinline__ void make_q_image(const uint4 (&raw)[2 * HI / 32][4], const float* __restrict__ w_row,
                                             int lane, uint4 (&img)[2 * HI / 32][4], float (&wq)[2 * HI / 32],
                                             int (&exq)[2 * HI / 32]) {
    constexpr int kUnits = 2 * HI / 32;
#pragma unroll
    for (int j = 0; j < kUnits; ++j) {
        const int h = (lane + 32 * j) >> 1;
        float x[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t wd[4] = {raw[j][c].x, raw[j][c].y, raw[j][c].z, raw[j][c].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                x[8 * c + 2 * i] = __uint_as_float(wd[i] << 16);
                x[8 * c + 2 * i + 1] = __uint_as_float(wd[i] & 0xFFFF0000u);
            }
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));   // other half of head h
        int ex = 0;
        if (amax > 0.0f) {
            frexpf(amax, &ex);                  // amax in [2^(ex-1), 2^ex)
            ex = min(8 - ex, 122);              // amax * 2^ex in [2^7, 2^8) (capped: UE8M0 range)
        }
        uint32_t hw[8], lw[8];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
            float y[4], hv[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) y[k] = ldexpf(x[i + k], ex);
            const uint32_t h01 = cvt_e4m3x2(y[0], y[1]), h23 = cvt_e4m3x2(y[2], y[3]);
            e4m3x2_to_f32(h01, hv[0], hv[1]);
            e4m3x2_to_f32(h23, hv[2], hv[3]);
            const uint32_t l01 = cvt_e4m3x2(32.0f * (y[0] - hv[0]), 32.0f * (y[1] - hv[1]));
            const uint32_t l23 = cvt_e4m3x2(32.0f * (y[2] - hv[2]), 32.0f * (y[3] - hv[3]));
            hw[i / 4] = h01 | (h23 << 16);
            lw[i / 4] = l01 | (l23 << 16);
        }
        img[j][0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        img[j][1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
        img[j][2] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        img[j][3] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
        wq[j] = FOLD ? ldexpf(w_row[h], -ex) : w_row[h];
        exq[j] = ex;
    }
}

template <int HI>
__device__ __forceinline__ void load_q_raw(const __nv_bfloat16* __restrict__ q_row, int lane,
                                           uint4 (&raw)[2 * HI / 32][4]) {
#pragma unroll
    for (int j = 0; j < 2 * HI / 32; ++j) {
        const int unit = lane + 32 * j;
        const uint4* src = reinterpret_cast<const uint4*>(q_row + (unit >> 1) * kDI + (unit & 1) * 32);
#pragma unroll
        for (int c = 0; c < 4; ++c) raw[j][c] = __ldg(src + c);
    }
}

template <int FMT, int HI, bool Q4>
__global__ void __launch_bounds__(Cfg<FMT, HI, Q4>::threads) index_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                                                            const __nv_bfloat16* __restrict__ q_idx,
                                                            const uint8_t* __restrict__ q_scale,
                                                            const float* __restrict__ w,
                                                            const uint8_t* __restrict__ k_scale, int T,
                                                            const int64_t* __restrict__ q_pos, int64_t Ncap, int m,
                                                            int R, float* __restrict__ S,
                                                            uint32_t* __restrict__ hist1, unsigned* err) {
    using C = Cfg<FMT, HI, Q4>;
    constexpr int kUnits = 2 * HI / 32;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~uintptr_t(1023));
    __shared__ IdxMisc ms;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = smem_u32(sm);

    if (warp == 0) {
        tmem_alloc(&ms.tmem_base, C::tmem_cols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(&ms.full[s], 1);
            mbar_init(&ms.empty[s], 1);       // the MMA commit: the epilogue never reads a stage
        }
        for (int d = 0; d < kMaxBuf; ++d) {
            mbar_init(&ms.dfull[d], 2);       // the MMA commit + the MMA warp's record of the stage
            mbar_init(&ms.dfree[d], 4);
        }
        // 4 epilogue warps, once per item: the epilogue takes the stages in order after their MMAs
        // completed, so its arrivals at a piece's end imply that every MMA of the piece is done
        for (int d = 0; d < 2; ++d) mbar_init(&ms.qfree[d], 4);
        fence_mbar_init();
    }
    if (tid < kEpi)
        for (int i = tid; i < 2048; i += kEpi) ms.hist[i] = 0u;
    // TMEM, barriers and shared memory touch no global memory: set up while the preceding kernel
    // finishes
    pdl_wait();
    pdl_trigger();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = ms.tmem_base;
    const int items = R * (int)cdiv(Ncap, (int64_t)kChunkStages * kPair);

    if (warp == 4) {
        // ======================================================================== producer
        const uint64_t pol_stream = l2_policy_evict_first();     // codes are read once per step
        // Work pieces (row r, its visible count n, stage range [s0, s_end) of 256 keys each),
        // produced one ahead.  Few rows: the rows' stages, concatenated, are cut into gridDim.x
        // equal ranges and a CTA streams its range (a piece per row it overlaps, split into
        // pieces of at most kMaxPieceStages stages).  Otherwise: (row, chunk of kChunkStages
        // stages) items, round-robin over the CTAs.
        const bool balanced = R <= kSchedRows;
        int lo = 0, hi = 0, brow = 0;
        int64_t bnext = 0;                      // balanced: next key of row brow to stream
        if (balanced) {
            int carry = 0;
            for (int base = 0; base < R; base += 32) {
                const int q = base + lane;
                int ns = 0;
                if (q < R) {
                    const int64_t p = q_pos[q];
                    int64_t nn = (p >= 0) ? (p + 1) / m : 0;
                    nn = nn < Ncap ? nn : Ncap;
                    ms.nvis[q] = (int)nn;
                    ns = (int)((nn + kPair - 1) / kPair);
                }
                int x = ns;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                if (q < R) ms.soff[q + 1] = carry + x;
                carry += __shfl_sync(0xffffffffu, x, 31);
            }
            if (lane == 0) ms.soff[0] = 0;
            __syncwarp();
            const int len = (carry + (int)gridDim.x - 1) / (int)gridDim.x;
            lo = (int)blockIdx.x * len;
            hi = min(carry, lo + len);
        }
        int c_item = (int)blockIdx.x;          // round-robin cursor
        bool c_ok = false;                      // candidate next piece
        int c_r = 0;
        int64_t c_n = 0, c_s0 = 0, c_send = 0, c_p = 0;
        uint4 c_raw[kUnits][4];
        auto fetch_next = [&]() {               // fills the candidate; blocking only when round-robin
            c_ok = false;
            if (balanced) {
                for (; brow < R; ++brow, bnext = 0) {
                    const int st0 = ms.soff[brow], st1 = ms.soff[brow + 1];
                    if (st0 >= hi) break;
                    if (st1 <= lo || st1 == st0) continue;
                    c_r = brow;
                    c_n = ms.nvis[brow];
                    const int64_t b0 = (int64_t)(max(lo, st0) - st0) * kPair;
                    const int64_t e = (int64_t)(min(hi, st1) - st0) * kPair;
                    const int64_t end = e < c_n ? e : c_n;
                    c_s0 = bnext > b0 ? bnext : b0;
                    const int64_t cap = c_s0 + (int64_t)kMaxPieceStages * kPair;
                    c_send = end < cap ? end : cap;
                    c_ok = true;
                    if (c_send < end) {
                        bnext = c_send;                 // the rest of this row's range follows
                    } else {
                        ++brow;
                        bnext = 0;
                    }
                    break;
                }
            } else {
                for (; c_item < items; c_item += gridDim.x) {
                    const int rr = c_item % R;
                    const int64_t p = (c_item == (int)blockIdx.x) ? q_pos[rr] : c_p;
                    int64_t nn = (p >= 0) ? (p + 1) / m : 0;
                    nn = nn < Ncap ? nn : Ncap;
                    const int64_t s0 = (int64_t)(c_item / R) * kChunkStages * kPair;
                    const int nxt = c_item + (int)gridDim.x;
                    c_p = nxt < items ? q_pos[nxt % R] : 0;          // the next candidate's position
                    if (s0 >= nn) continue;
                    const int64_t e = s0 + (int64_t)kChunkStages * kPair;
                    c_r = rr;
                    c_n = nn;
                    c_s0 = s0;
                    c_send = e < nn ? e : nn;
                    c_ok = true;
                    c_item = nxt;
                    break;
                }
            }
            if (c_ok && C::prefetch_q && !Q4) load_q_raw<HI>(q_idx + (int64_t)c_r * HI * kDI, lane, c_raw);
        };
        fetch_next();
        uint32_t u = 0;                       // stages issued
        for (uint32_t it = 0; c_ok; ++it) {
            const int r = c_r;
            const int64_t n = c_n, s_end = c_send;
            int64_t s0 = c_s0;
            uint4 raw[kUnits][4];
            if (C::prefetch_q) {
#pragma unroll
                for (int j = 0; j < kUnits; ++j)
#pragma unroll
                    for (int c = 0; c < 4; ++c) raw[j][c] = c_raw[j][c];
            }
            fetch_next();
            // query slot of this piece: free once the MMAs and epilogue of piece it-2 are done
            const uint32_t qs = it & 1;
            if (it >= 2) mbar_wait(&ms.qfree[qs], ((it >> 1) + 1) & 1, err);
            unsigned char* qsl = sm + C::off_qslots + qs * C::q_slot;
            if constexpr (Q4) {
                // FP4 queries (E2M1 codes, two per byte, and a UE8M0 byte per 32): unit (head h, half
                // hf) = lane + 32 j holds 32 codes = two groups of 16, each stored as the MMA reads a
                // 4-bit operand (the 8 packed bytes, then 8 bytes of padding); the B scale factors are
                // the query's own scale bytes (byte k of column h: block k)
                const uint8_t* qc = reinterpret_cast<const uint8_t*>(q_idx) + (int64_t)r * HI * (kDI / 2);
#pragma unroll
                for (int j = 0; j < kUnits; ++j) {
                    const int unit = lane + 32 * j, h = unit >> 1, hf = unit & 1;
                    const uint4 pk = __ldg(reinterpret_cast<const uint4*>(qc + h * (kDI / 2) + hf * 16));
                    *reinterpret_cast<uint4*>(qsl + sw128(h, 2 * hf)) = make_uint4(pk.x, pk.y, 0u, 0u);
                    *reinterpret_cast<uint4*>(qsl + sw128(h, 2 * hf + 1)) = make_uint4(pk.z, pk.w, 0u, 0u);
                    if (hf == 0) {
                        reinterpret_cast<float*>(qsl + C::q_img)[h] = w[(int64_t)r * HI + h];
                        const uint32_t sc = __ldg(reinterpret_cast<const uint16_t*>(q_scale) + (int64_t)r * HI + h);
                        reinterpret_cast<uint32_t*>(qsl + C::off_sfb)[(h & 31) * 4 + (h >> 5)] = sc | (sc << 16);
                    }
                }
            } else {
            if (!C::prefetch_q) load_q_raw<HI>(q_idx + (int64_t)r * HI * kDI, lane, raw);
            uint4 img[kUnits][4];
            float wq[kUnits];
            int exq[kUnits];
            make_q_image<HI, !C::fp4>(raw, w + (int64_t)r * HI, lane, img, wq, exq);
#pragma unroll
            for (int j = 0; j < kUnits; ++j) {
                const int unit = lane + 32 * j, h = unit >> 1, hf = unit & 1;
#pragma unroll
                for (int c = 0; c < 4; ++c)                       // hi: row h, lo: row HI + h
                    *reinterpret_cast<uint4*>(qsl + sw128(h + (c >> 1) * HI, 2 * hf + (c & 1))) = img[j][c];
                if (hf == 0) {
                    reinterpret_cast<float*>(qsl + C::q_img)[h] = wq[j];
                    if (C::fp4) {
                        // B scale factors (every K block alike): column n's byte in word n / 32 of
                        // line n % 32; hi column h: 2^-e_h, lo column HI + h: 2^-(e_h + 5)
                        uint32_t* sfb = reinterpret_cast<uint32_t*>(qsl + C::off_sfb);
                        // (the MMA adds the lo rows into the hi rows' columns: their factor is
                        // byte 2 + block of column h's word)
                        sfb[(h & 31) * 4 + (h >> 5)] = (uint32_t)(127 - exq[j]) * 0x0101u | (uint32_t)(122 - exq[j]) * 0x01010000u;
                    }
                }
            }
            }
            fence_proxy_async();
            __syncwarp();
            // stages of the piece (one lane)
            if (lane == 0) {
                const int b = r / T;
                for (; s0 < s_end; s0 += kPair, ++u) {
                    const uint32_t s = u % C::NS;
                    if (u >= (uint32_t)C::NS) mbar_wait(&ms.empty[s], ((u / C::NS) + 1) & 1, err);
                    unsigned char* st = sm + s * C::stage;
                    const uint32_t sb = sbase + s * C::stage;
                    const int flags = ((s0 + kPair >= s_end) ? kLast : 0) | (int)(qs << 8) | (int)((it & 0x7FFFu) << 16);
                    *reinterpret_cast<int4*>(st + C::off_meta) = make_int4(r, (int)s0, (int)n, flags);
                    const int64_t key0 = (int64_t)b * Ncap + s0;
                    const int64_t nk = (Ncap - s0) < kPair ? (Ncap - s0) : kPair;   // Ncap % 8 == 0
                    const uint32_t sbytes = (uint32_t)nk * C::scale_bytes;
                    mbar_arrive_expect_tx(&ms.full[s], C::code_tx + sbytes);
                    if (C::fp4) {
                        // MMA row R = 32 j + l holds TMA row 4 l + j of the 128 (keys 2(4l+j), +1), so the
                        // stage's scale bytes, copied as they are stored, form the factor image
                        tma_load_4d(sb, &kmap, 0, 0, 0, (int)(key0 / kPair), &ms.full[s], pol_stream);
                    } else {
                        tma_load_2d(sb, &kmap, 0, (int)(key0 / 2), &ms.full[s], pol_stream);
                    }
                    bulk_g2s_hint(sb + (C::fp4 ? C::off_sfa : C::off_scale), k_scale + key0 * C::scale_bytes, sbytes, &ms.full[s],
                                  pol_stream);
                }
            }
            u = __shfl_sync(0xffffffffu, u, 0);
        }
        if (lane == 0) {                      // end of work: one record for each MMA warp
            for (int j = 0; j < C::NMW; ++j, ++u) {
                const uint32_t s = u % C::NS;
                if (u >= (uint32_t)C::NS) mbar_wait(&ms.empty[s], ((u / C::NS) + 1) & 1, err);
                *reinterpret_cast<int4*>(sm + s * C::stage + C::off_meta) = make_int4(0, 0, 0, kTerm | (j ? 0 : kFirstTerm));
                mbar_arrive(&ms.full[s]);
            }
        }
        __syncwarp();
    } else if (warp >= 5 && warp < 5 + C::NMW) {
        // ============================================================================= MMA
        constexpr uint32_t af = C::fp4 ? kE2M1 : kE4M3;
        // descriptors of stage 0 and query slot 0; other addresses add (offset >> 4)
        const uint64_t a_desc0 = smem_desc(sbase, 16, 1024);
        const uint64_t b_desc0 = smem_desc(sbase + C::off_qslots, 16, 1024);
        // stages u = mw, mw + NMW, ...: the warps' per-stage waits and issue overlap; each
        // stage's MMAs and commits come from one thread, so the commits track exactly that stage
        const uint32_t mw = (uint32_t)(warp - 5);
        int prev_piece = -1;                      // piece (low 15 bits) of this warp's previous stage
        for (uint32_t u = mw; mw < (uint32_t)C::NMW; u += C::NMW) {
            const uint32_t s = u % C::NS;
            mbar_wait(&ms.full[s], (u / C::NS) & 1, err);
            const int4 meta = *reinterpret_cast<const int4*>(sm + s * C::stage + C::off_meta);
            const uint32_t d = u % C::nbuf, qs = (uint32_t)(meta.w >> 8) & 1u;
            if (meta.w & kTerm) {
                if (!(meta.w & kFirstTerm)) break;
                // end of work: hand the record to the epilogue through the next buffer
                if (u >= (uint32_t)C::nbuf) mbar_wait(&ms.dfree[d], ((u / C::nbuf) + 1) & 1, err);
                if (lane == 0) {
                    ms.dmeta[d] = meta;
                    mbar_arrive_cnt(&ms.dfull[d], 2);
                }
                break;
            }
            __syncwarp();
            // the accumulator buffer (with its record slot) is free once the epilogue has read it
            if (u >= (uint32_t)C::nbuf) mbar_wait(&ms.dfree[d], ((u / C::nbuf) + 1) & 1, err);
            if (!C::fp4) {
                const float4* src = reinterpret_cast<const float4*>(sm + s * C::stage + C::off_scale);
                float4* dst = reinterpret_cast<float4*>(sm + C::off_dscale + d * kPair * 4);
                dst[lane] = src[lane];
                dst[lane + 32] = src[lane + 32];
            }
            if (lane == 0) ms.dmeta[d] = meta;
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&ms.dfull[d]);            // the record (the MMA commit is the other arrival)
                fence_after_sync();
                const uint64_t ad0 = a_desc0 + ((s * C::stage) >> 4);
                const uint64_t bd0 = b_desc0 + ((qs * C::q_slot) >> 4);
                const uint32_t dbuf = tmem + d * C::d_cols;
                if (C::fp4) {
                    // factors reach TMEM before the MMAs that read them (issued in order by this thread)
                    const uint32_t sfa = tmem + C::sfa_col + 4 * s, sfb = tmem + C::sfb_col + 4 * qs;
                    if ((meta.w >> 16) != prev_piece)     // a new piece: its query's B factors
                        tmem_cp_32x128b_x4(sfb, smem_desc(sbase + C::off_qslots + qs * C::q_slot + C::off_sfb, 16, 128, 0));
                    tmem_cp_32x128b_x4(sfa, smem_desc(sbase + s * C::stage + C::off_sfa, 16, 128, 0));
#pragma unroll
                    for (int e = 0; e < 2; ++e)              // even keys: code columns [0,64); odd: [64,128)
#pragma unroll
                        for (int blk = 0; blk < 2; ++blk)    // 32-code blocks (one MMA K step each)
                        {
                            mma_mxf8f6f4_bs(dbuf + e * C::acc_cols, ad0 + (uint64_t)(e * 4 + blk * 2),
                                            bd0 + (uint64_t)(blk * 2),
                                            idesc_mxf8f6f4_bs(128, C::acc_cols, af, Q4 ? kE2M1 : kE4M3, 2 * e + blk, blk),
                                            sfa, sfb,
                                            (uint32_t)(blk > 0));
                            if constexpr (C::fused)       // the lo rows (row HI on), factor byte 2 + blk
                                mma_mxf8f6f4_bs(dbuf + e * C::acc_cols, ad0 + (uint64_t)(e * 4 + blk * 2),
                                                bd0 + (uint64_t)((HI * 128) >> 4) + (uint64_t)(blk * 2),
                                                idesc_mxf8f6f4_bs(128, C::acc_cols, af, kE4M3, 2 * e + blk, 2 + blk),
                                                sfa, sfb, 1u);
                        }
                } else {
                    const uint32_t id = idesc_f8f6f4(128, 2 * HI, af, kE4M3);
#pragma unroll
                    for (int e = 0; e < 2; ++e)
#pragma unroll
                        for (int blk = 0; blk < 2; ++blk)
                            mma_f8f6f4(dbuf + e * C::acc_cols, ad0 + (uint64_t)(e * 4 + blk * 2), bd0 + (uint64_t)(blk * 2),
                                       id, (uint32_t)(blk > 0));
                }
                mma_commit(&ms.dfull[d]);
                mma_commit(&ms.empty[s]);
            }
            prev_piece = meta.w >> 16;
            __syncwarp();
        }
    } else {
        // ======================================================================== epilogue
        const uint64_t pol_keep = l2_policy_evict_last();       // the top-k re-reads the scores
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        for (uint32_t u = 0;; ++u) {
            const uint32_t d = u % C::nbuf;
            mbar_wait(&ms.dfull[d], (u / C::nbuf) & 1, err);
            fence_after_sync();
            const int4 meta = ms.dmeta[d];
            if (meta.w & kTerm) break;
            const uint32_t qs = (uint32_t)(meta.w >> 8) & 1u;
            float se = 1.0f, so = 1.0f;                      // e4m3: row scales of keys 2j (e), 2j+1 (o)
            if (!C::fp4) {
                const float2 f2 = reinterpret_cast<const float2*>(sm + C::off_dscale + d * kPair * 4)[tid];
                se = f2.x;
                so = f2.y;
            }
            const float4* wq4 = reinterpret_cast<const float4*>(sm + C::off_qslots + qs * C::q_slot + C::q_img);
            const uint32_t dbuf = tmem + d * C::d_cols + lane_off;
            // per key: pairs of heads (h, h+1) in f32x2 lanes, v = D_hi + D_lo (fp4: scaled by the
            // MMA) or D_hi + 2^-5 D_lo (e4m3).  When the stage's accumulators fit in registers they
            // are all loaded first and the TMEM buffer is handed back to the MMA warp before the
            // arithmetic.
            const uint64_t Ll = f2_pack(kLoScale, kLoScale);
            auto head_pairs = [&](uint64_t& acc, const uint32_t* hv, const uint32_t* lv, const uint64_t* wv) {
#pragma unroll
                for (int k = 0; k < 16; k += 2) {
                    const uint64_t hp = f2_pack(__uint_as_float(hv[k]), __uint_as_float(hv[k + 1]));
                    uint64_t v = hp;                          // one part (fused hi + lo, or FP4 queries)
                    if constexpr (!C::one_part) {
                        const uint64_t lp = f2_pack(__uint_as_float(lv[k]), __uint_as_float(lv[k + 1]));
                        v = C::fp4 ? f2_add(hp, lp) : f2_fma(Ll, lp, hp);
                    }
                    float a0, a1;
                    f2_unpack(v, a0, a1);
                    acc = f2_fma(wv[k / 2], f2_pack(fmaxf(a0, 0.0f), fmaxf(a1, 0.0f)), acc);
                }
            };
            auto weights16 = [&](int c0, uint64_t (&wv)[8]) {
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    const float4 q4 = wq4[c0 / 4 + k4];
                    wv[2 * k4] = f2_pack(q4.x, q4.y);
                    wv[2 * k4 + 1] = f2_pack(q4.z, q4.w);
                }
            };
            uint64_t acc2[2] = {f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f)};
            if constexpr (C::d_cols <= 128) {
                uint32_t dv[C::d_cols];
#pragma unroll
                for (int c = 0; c < (int)C::d_cols; c += 16) {
                    uint32_t t16[16];
                    tmem_ld16(dbuf + c, t16);
#pragma unroll
                    for (int k = 0; k < 16; ++k) dv[c + k] = t16[k];
                }
                tmem_wait_ld();
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ms.dfree[d]);
#pragma unroll
                for (int key = 0; key < 2; ++key)
#pragma unroll
                    for (int c0 = 0; c0 < HI; c0 += 16) {
                        uint64_t wv[8];
                        weights16(c0, wv);
                        const int h = key * (int)C::acc_cols + c0;
                        head_pairs(acc2[key], dv + h, dv + h + (C::one_part ? 0 : HI), wv);
                    }
            } else {
#pragma unroll
                for (int key = 0; key < 2; ++key) {
                    const uint32_t abase = dbuf + key * C::acc_cols;
#pragma unroll
                    for (int c0 = 0; c0 < HI; c0 += 16) {
                        uint64_t wv[8];
                        weights16(c0, wv);
                        uint32_t h0[16], l0[16];
                        tmem_ld16(abase + c0, h0);
                        if (!C::one_part) tmem_ld16(abase + HI + c0, l0);
                        tmem_wait_ld();
                        head_pairs(acc2[key], h0, l0, wv);
                    }
                }
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ms.dfree[d]);
            }
            float acc_e, acc_o;
            {
                float x0, x1;
                f2_unpack(acc2[0], x0, x1);
                acc_e = (x0 + x1) * se;
                f2_unpack(acc2[1], x0, x1);
                acc_o = (x0 + x1) * so;
            }
            // (at the piece's end) query slot consumed
            __syncwarp();
            if (lane == 0 && (meta.w & kLast)) mbar_arrive(&ms.qfree[qs]);
            // keys of TMEM lane tid: e2m1 tiles are loaded permuted (MMA row 32 j + l = TMA row 4 l + j)
            const int64_t key = (int64_t)meta.y + 2 * (C::fp4 ? 4 * (tid & 31) + (tid >> 5) : tid);
            const bool v0 = key < meta.z, v1 = key + 1 < meta.z;
            float* dst = S + (int64_t)meta.x * Ncap + key;
            if (v1) st_global_v2_hint(dst, acc_e, acc_o, pol_keep);
            else if (v0) st_global_hint(dst, acc_e, pol_keep);
            if (hist1 != nullptr) {
                if (v0) {
                    const uint32_t bin = ordered_key(acc_e) >> 20;
                    atomicAdd(&ms.hist[bin >> 1], 1u << ((bin & 1) * 16));
                }
                if (v1) {
                    const uint32_t bin = ordered_key(acc_o) >> 20;
                    atomicAdd(&ms.hist[bin >> 1], 1u << ((bin & 1) * 16));
                }
                if (meta.w & kLast) {                     // piece done: add to the row's histogram
                    named_barrier_sync(1, kEpi);
                    uint32_t* gh = hist1 + (int64_t)meta.x * 4096;
                    for (int i = 4 * tid; i < 2048; i += 4 * kEpi) {   // words of two 16-bit counts
                        const uint4 v = *reinterpret_cast<const uint4*>(&ms.hist[i]);
                        if (v.x | v.y | v.z | v.w) {
                            const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                if (wd[k] & 0xFFFFu) atomicAdd(&gh[2 * (i + k)], wd[k] & 0xFFFFu);
                                if (wd[k] >> 16) atomicAdd(&gh[2 * (i + k) + 1], wd[k] >> 16);
                            }
                            *reinterpret_cast<uint4*>(&ms.hist[i]) = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    named_barrier_sync(1, kEpi);
                }
            }
        }
    }
    __syncwarp();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, C::tmem_cols);
}

template <int FMT, int HI, bool Q4 = false>
cudaError_t launch_index_tc(const void* q_idx, const void* q_scale, const float* w, const void* k_codes,
                            const void* k_scale, int B, int T, const int64_t* q_pos, int64_t Ncap, int m, float* S,
                            uint32_t* hist1, unsigned* err, cudaStream_t st) {
    using C = Cfg<FMT, HI, Q4>;
    CUtensorMap kmap;
    std::memset(&kmap, 0, sizeof kmap);
    const uint64_t rows = (uint64_t)B * (uint64_t)Ncap / 2;          // two keys per row of 128 codes
    bool ok;
    if (C::fp4) {
        // tiles of 128 TMA rows (256 keys) read as [l 32][j 4] with row 4 l + j landing in smem row 32 j + l
        const uint64_t dims[4] = {128, 32, 4, rows / 128};
        const uint64_t strides[3] = {4 * 64, 64, 128 * 64};
        const uint32_t box[4] = {128, 32, 4, 1};
        ok = rows % 128 == 0 && encode_tmap_nd(&kmap, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4, k_codes, dims, strides, box);
    } else {
        ok = encode_tmap_2d(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, k_codes, 128, rows, 128, 128, 128);
    }
    if (!ok) return cudaErrorNotSupported;
    const size_t smem = (size_t)C::smem + 1024;
    // CTAs per SM: shared memory (228 KB per SM, 1 KB reserved per CTA) and TMEM (512 columns)
    const size_t per_cta = smem + sizeof(IdxMisc) + 1024;
    const int occ = std::max(1, std::min((int)((size_t)(228 * 1024) / per_cta), (int)(512 / C::tmem_cols)));
    auto kern = index_tc_kernel<FMT, HI, Q4>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int R = B * T;
    const int64_t items = (int64_t)R * cdiv(Ncap, (int64_t)kChunkStages * kPair);
    const int grid = (int)std::min<int64_t>(items, (int64_t)num_sms() * occ);
    (void)launch_pdl(kern, dim3(grid), dim3(C::threads), smem, st, kmap, static_cast<const __nv_bfloat16*>(q_idx),
                     static_cast<const uint8_t*>(q_scale), w,
                                       static_cast<const uint8_t*>(k_scale), T, q_pos, Ncap, m, R, S, hist1, err);
    return cudaGetLastError();
}

}  // namespace

bool index_tc_supported(int q_dtype, int key_fmt, int H_I, int d_I, int64_t Ncap, const void* k_codes,
                        const void* k_scale, int B, int64_t R) {
    return q_dtype == CSAHCA_BF16 && (key_fmt == CSAHCA_E4M3_ROWSCALE || key_fmt == CSAHCA_E2M1_UE8M0) &&
           d_I == kDI && (H_I == 16 || H_I == 32 || H_I == 64) &&
           Ncap % (key_fmt == CSAHCA_E2M1_UE8M0 ? kPair : 8) == 0 && aligned(k_codes, 32) &&
           aligned(k_scale, 16) && (int64_t)B * Ncap / 2 >= 128 && (int64_t)B * Ncap < (1LL << 31) &&
           R * cdiv(Ncap, (int64_t)kChunkStages * kPair) < (1LL << 31);
}

cudaError_t index_tc_launch(const void* q_idx, const float* w, const void* k_codes, const void* k_scale, int key_fmt,
                            int B, int T, int H_I, const int64_t* q_pos, int64_t Ncap, int m, float* S,
                            uint32_t* hist1, unsigned* err, cudaStream_t st) {
#define CSAHCA_IDX_CASE(F, HH)                                                                                  \
    if (key_fmt == F && H_I == HH)                                                                              \
        return launch_index_tc<F, HH>(q_idx, nullptr, w, k_codes, k_scale, B, T, q_pos, Ncap, m, S, hist1, err, st);
    CSAHCA_IDX_CASE(CSAHCA_E2M1_UE8M0, 16)
    CSAHCA_IDX_CASE(CSAHCA_E2M1_UE8M0, 32)
    CSAHCA_IDX_CASE(CSAHCA_E2M1_UE8M0, 64)
    CSAHCA_IDX_CASE(CSAHCA_E4M3_ROWSCALE, 16)
    CSAHCA_IDX_CASE(CSAHCA_E4M3_ROWSCALE, 32)
    CSAHCA_IDX_CASE(CSAHCA_E4M3_ROWSCALE, 64)
#undef CSAHCA_IDX_CASE
    return cudaErrorNotSupported;
}

cudaError_t index_tc_q4_launch(const void* q_codes, const void* q_scale, const float* w, const void* k_codes,
                               const void* k_scale, int B, int T, int H_I, const int64_t* q_pos, int64_t Ncap, int m,
                               float* S, uint32_t* hist1, unsigned* err, cudaStream_t st) {
    switch (H_I) {
        case 16: return launch_index_tc<CSAHCA_E2M1_UE8M0, 16, true>(q_codes, q_scale, w, k_codes, k_scale, B, T, q_pos, Ncap, m, S, hist1, err, st);
        case 32: return launch_index_tc<CSAHCA_E2M1_UE8M0, 32, true>(q_codes, q_scale, w, k_codes, k_scale, B, T, q_pos, Ncap, m, S, hist1, err, st);
        case 64: return launch_index_tc<CSAHCA_E2M1_UE8M0, 64, true>(q_codes, q_scale, w, k_codes, k_scale, B, T, q_pos, Ncap, m, S, hist1, err, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace csahca
