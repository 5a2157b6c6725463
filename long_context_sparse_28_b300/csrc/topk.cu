// a6: per-query top-k over float32 indexer scores (honbul.tistory.com/221 "CSA": the Top-k
// Selector keeps only part of the compressed entries; pogovet.com detail 4: the indexer picks
// the top-k compressed blocks of every query).
//
// Exact radix select on the order-preserving 32-bit image of each score (12 + 12 + 8 bits):
//   hist   : 4096-bin histogram of the top 12 bits per row -- fused into the indexer's
//            tensor-core epilogue, or a separate pass over the scores;
//   select : one launch; a row is handled by a cluster of P CTAs, CTA p owning the p-th slice of
//            the row's entries (whole 32-entry words).  Every CTA finds the boundary bin b1 where
//            the running count from the top reaches k; when the elements of bins >= b1 number at
//            most kCap, each CTA gathers those of its slice, (key, index), into shared memory
//            (otherwise it re-reads its slice for every pass).  The next 12 and 8 bits are
//            resolved with histograms of the CTAs' candidates summed over the cluster through
//            distributed shared memory; each CTA then marks its "above the threshold" and "equal
//            to the threshold" entries in two bitmaps of its slice, learns from the others' counts
//            how many of the lowest-index "equal" entries are its to take and where its output
//            starts, and writes its selected indices in ascending order.
// Output: indices ascending, -1 padded.  Ties go to the lower index; the result is exact and
// deterministic for any non-NaN scores (-0 == +0).
#include "common.cuh"

#include <cooperative_groups.h>

namespace csahca {
namespace {

constexpr int kBins12 = 4096;
constexpr int kBins8 = 256;
constexpr int kSlice = 32768;      // scores per histogram CTA
constexpr int kCap = 8192;         // candidate-list capacity per row
constexpr int kThreads = 256;      // histogram pass
constexpr int kSelThreads = 1024;  // select pass

__device__ __forceinline__ int64_t row_nvis(int r, const int64_t* n_vis_arr, const int64_t* q_pos, int m,
                                            int64_t Ncap) {
    if (n_vis_arr) return n_vis_arr[r];
    const int64_t p = q_pos[r];
    int64_t v = (p >= 0) ? (p + 1) / m : 0;
    return v < Ncap ? v : Ncap;
}

// Finds the bin b (counting from the top) where the running count reaches `need`:
// above(b) < need <= above(b) + hist[b], above(b) = sum of the bins above b.  nb must be a
// multiple of blockDim.x.  Results broadcast through shared memory.
__device__ void find_bin(const uint32_t* hist, int nb, uint32_t need, int* sh_scan, int* sh_res, int* bin_out,
                         uint32_t* above_out) {
    const int per = nb / blockDim.x;
    const int chunk = blockDim.x - 1 - threadIdx.x;      // thread 0 owns the highest bins
    const int lo = chunk * per;
    int local = 0;
    for (int i = 0; i < per; ++i) local += (int)hist[lo + i];
    int total;
    const int above = block_exclusive_scan(local, sh_scan, &total);
    if (threadIdx.x == 0) {
        sh_res[0] = 0;
        sh_res[1] = 0;
    }
    __syncthreads();
    if ((uint32_t)above < need && need <= (uint32_t)(above + local)) {
        uint32_t acc = (uint32_t)above;
        for (int b = lo + per - 1; b >= lo; --b) {
            const uint32_t h = hist[b];
            if (acc + h >= need) {
                sh_res[0] = b;
                sh_res[1] = (int)acc;
                break;
            }
            acc += h;
        }
    }
    __syncthreads();
    *bin_out = sh_res[0];
    *above_out = (uint32_t)sh_res[1];
    __syncthreads();
}

// Histogram of the top 12 bits (used when the scores were not produced by the fused indexer).
__global__ void __launch_bounds__(kThreads) topk_hist_kernel(const float* __restrict__ scores, int64_t stride,
                                                             const int64_t* __restrict__ n_vis_arr,
                                                             const int64_t* __restrict__ q_pos, int m, int64_t Ncap,
                                                             uint32_t* __restrict__ hist1) {
    pdl_wait();
    pdl_trigger();
    __shared__ uint32_t sh[kBins12];
    const int r = blockIdx.y;
    const int64_t n = min(row_nvis(r, n_vis_arr, q_pos, m, Ncap), stride);
    const int64_t s0 = (int64_t)blockIdx.x * kSlice;
    if (s0 >= n) return;
    const int64_t s1 = min(n, s0 + kSlice);
    for (int i = threadIdx.x; i < kBins12; i += blockDim.x) sh[i] = 0;
    __syncthreads();
    const float* row = scores + (int64_t)r * stride;
    int64_t s = s0;
    if ((reinterpret_cast<uintptr_t>(row + s0) & 15) == 0) {      // 16-byte loads
        const float4* r4 = reinterpret_cast<const float4*>(row + s0);
        const int64_t n4 = (s1 - s0) / 4;
        for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
            const float4 x = __ldg(r4 + i);
            atomicAdd(&sh[ordered_key(x.x) >> 20], 1u);
            atomicAdd(&sh[ordered_key(x.y) >> 20], 1u);
            atomicAdd(&sh[ordered_key(x.z) >> 20], 1u);
            atomicAdd(&sh[ordered_key(x.w) >> 20], 1u);
        }
        s = s0 + n4 * 4;
    }
    for (s += threadIdx.x; s < s1; s += blockDim.x) atomicAdd(&sh[ordered_key(row[s]) >> 20], 1u);
    __syncthreads();
    uint32_t* gh = hist1 + (int64_t)r * kBins12;
    for (int i = threadIdx.x; i < kBins12; i += blockDim.x)
        if (sh[i]) atomicAdd(&gh[i], sh[i]);
}

// Smallest float32 whose ordered key has top-12-bit bin b (inverse of ordered_key on b << 20).
__device__ __forceinline__ float bin_floor_value(int b) {
    const uint32_t key = (uint32_t)b << 20;
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

constexpr int kWarpSpan = 1024;    // scores per warp and step of the collect pass (32 per lane)
constexpr int kSmemWords = 8192;   // bitmap words of a slice kept in shared memory (262144 entries)
constexpr int kMaxCluster = 8;
// shared memory: candidates | the cluster's candidates | two histograms | two bitmaps
constexpr size_t kSelSmem = 2 * (size_t)kCap * 8 + 2 * (size_t)kBins12 * 4 + 2 * (size_t)kSmemWords * 4;

// The warp's span [w0, w0 + cnt_n) of `row` into registers: lane element e is entry
// ((e >> 2) * 32 + lane) * 4 + (e & 3) (16-byte loads when aligned and full; -inf past the end).
__device__ __forceinline__ void load_span(const float* __restrict__ row, int64_t w0, int cnt_n, int lane,
                                          float (&v)[32]) {
    const float* src = row + w0;
    const bool vec = ((reinterpret_cast<uintptr_t>(src) & 15) == 0) && cnt_n == kWarpSpan;
    if (vec) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 x = __ldg(reinterpret_cast<const float4*>(src) + j * 32 + lane);
            v[4 * j] = x.x; v[4 * j + 1] = x.y; v[4 * j + 2] = x.z; v[4 * j + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int i = (j * 32 + lane) * 4 + c;
                v[4 * j + c] = i < cnt_n ? __ldg(src + i) : -INFINITY;
            }
    }
}

// Appends the elements >= tv of a loaded span to the shared candidate list (one shared atomic per
// warp).  Candidates are few (about k per row), so their values are read again from the row.
__device__ __forceinline__ void collect_loaded(const float* __restrict__ row, int64_t w0, int cnt_n, float tv,
                                               const float (&v)[32], uint2* cs, int* sh_nc, int lane, int cap) {
    uint32_t bits = 0;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        const int i = ((e >> 2) * 32 + lane) * 4 + (e & 3);
        if (i < cnt_n && v[e] >= tv) bits |= 1u << e;
    }
    const int mine = __popc(bits);
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (total == 0) return;
    int base = 0;
    if (lane == 0) base = atomicAdd(sh_nc, total);
    base = __shfl_sync(0xffffffffu, base, 0) + incl - mine;
    while (bits) {
        const int e = __ffs(bits) - 1;
        bits &= bits - 1;
        const int i = ((e >> 2) * 32 + lane) * 4 + (e & 3);
        if (base < cap) cs[base] = make_uint2(ordered_key(__ldg(row + w0 + i)), (uint32_t)(w0 + i));
        ++base;
    }
}

// Exclusive block-wide prefix sums of two counts at once (one pass of barriers).
__device__ __forceinline__ int2 block_exclusive_scan2(int a, int b, int2* sh) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = a, y = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int xa = __shfl_up_sync(0xffffffffu, x, o), ya = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) {
            x += xa;
            y += ya;
        }
    }
    if (lane == 31) sh[wid] = make_int2(x, y);
    __syncthreads();
    if (wid == 0) {
        int2 t = (lane < nw) ? sh[lane] : make_int2(0, 0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int xa = __shfl_up_sync(0xffffffffu, t.x, o), ya = __shfl_up_sync(0xffffffffu, t.y, o);
            if (lane >= o) {
                t.x += xa;
                t.y += ya;
            }
        }
        if (lane < nw) sh[lane] = t;
    }
    __syncthreads();
    const int2 base = (wid > 0) ? sh[wid - 1] : make_int2(0, 0);
    const int2 res = make_int2(base.x + x - a, base.y + y - b);
    __syncthreads();
    return res;
}

__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Sums bins [0, nb) of `hist` over the CTAs of the cluster (distributed shared memory) into `out`.
__device__ __forceinline__ void cluster_sum(cooperative_groups::cluster_group& cl, uint32_t* hist, uint32_t* out,
                                            int nb) {
    const int P = (int)cl.num_blocks();
    for (int i = threadIdx.x; i < nb; i += blockDim.x) {
        uint32_t s = 0;
        for (int q = 0; q < P; ++q) s += cl.map_shared_rank(hist, q)[i];
        out[i] = s;
    }
}

// Grid (P, rows), clusters of (P, 1, 1): the CTAs of a cluster share one row.
__global__ void __launch_bounds__(kSelThreads, 1) topk_select_kernel(
    const float* __restrict__ scores, int64_t stride, const int64_t* __restrict__ n_vis_arr,
    const int64_t* __restrict__ q_pos, int m, int64_t Ncap, int k, uint32_t* __restrict__ hist1,
    uint32_t* __restrict__ win, uint32_t* __restrict__ tie, int64_t words, int32_t* __restrict__ idx_out,
    int cap, int smem_words, int self_hist) {
    pdl_wait();
    pdl_trigger();
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    extern __shared__ __align__(16) unsigned char fsm[];
    uint2* cs = reinterpret_cast<uint2*>(fsm);
    // shared memory (sizes from the launch): candidates [cap] | (clusters) the row's candidates [cap] |
    // two histograms | two bitmaps [smem_words]
    const bool clustered = cooperative_groups::this_cluster().num_blocks() > 1;
    uint2* ga = clustered ? cs + cap : cs;             // the whole row's candidates (fast path)
    uint32_t* hmine = reinterpret_cast<uint32_t*>(fsm + (clustered ? 2 : 1) * (size_t)cap * 8);
    uint32_t* hsum = hmine + kBins12;
    uint32_t* swin = hsum + kBins12;
    uint32_t* stie = swin + smem_words;
    __shared__ int sh_scan[33];
    __shared__ int sh_res[2];
    __shared__ int sh_nc;
    __shared__ int sh_cnt[2];                          // this CTA's "above" and "equal" counts
    __shared__ int2 sh_scan2[32];
    const int r = blockIdx.y, P = (int)cl.num_blocks(), p = (int)cl.block_rank();
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nthr >> 5;
    // the row's first histogram into shared memory, loaded together with the row's length; or
    // (self_hist: one CTA per row and no histogram from the indexer) formed here from the row's
    // scores, which the collect pass below then reads again from L2
    const int64_t n = min(row_nvis(r, n_vis_arr, q_pos, m, Ncap), min(stride, words * 32));
    if (self_hist) {
        for (int i = tid; i < kBins12; i += nthr) hsum[i] = 0u;
        __syncthreads();
        const float* srow = scores + (int64_t)r * stride;
        int64_t s = 0;
        if ((reinterpret_cast<uintptr_t>(srow) & 15) == 0) {
            const float4* r4 = reinterpret_cast<const float4*>(srow);
            const int64_t n4 = n / 4;
            for (int64_t i = tid; i < n4; i += nthr) {
                const float4 x = __ldg(r4 + i);
                atomicAdd(&hsum[ordered_key(x.x) >> 20], 1u);
                atomicAdd(&hsum[ordered_key(x.y) >> 20], 1u);
                atomicAdd(&hsum[ordered_key(x.z) >> 20], 1u);
                atomicAdd(&hsum[ordered_key(x.w) >> 20], 1u);
            }
            s = n4 * 4;
        }
        for (s += tid; s < n; s += nthr) atomicAdd(&hsum[ordered_key(srow[s]) >> 20], 1u);
    } else {
        for (int i = tid; i < kBins12 / 4; i += nthr)
            reinterpret_cast<uint4*>(hsum)[i] = reinterpret_cast<const uint4*>(hist1 + (int64_t)r * kBins12)[i];
    }
    int32_t* out = idx_out + (int64_t)r * k;
    uint32_t* hrow = hist1 + (int64_t)r * kBins12;
    if (n <= k) {                                   // every visible entry is selected, in order
        if (p == 0) {
            for (int j = tid; j < k; j += nthr) out[j] = j < n ? j : -1;
            for (int i = tid; i < kBins12; i += nthr) hrow[i] = 0u;   // the histogram, cleared for the next call
        }
        return;                                     // (the whole cluster takes this branch)
    }
    const float* row = scores + (int64_t)r * stride;
    // this CTA's slice: bitmap words [w_lo, w_hi), entries [s_lo, s_hi)
    const int64_t nwords = (n + 31) / 32;
    const int64_t w_lo = nwords * p / P, w_hi = nwords * (p + 1) / P;
    const int64_t s_lo = w_lo * 32, s_hi = min(n, w_hi * 32);
    const int64_t sw = w_hi - w_lo;
    const bool smem_bits = sw <= smem_words;
    uint32_t* wr = smem_bits ? swin : win + (int64_t)r * words + w_lo;
    uint32_t* tr = smem_bits ? stie : tie + (int64_t)r * words + w_lo;
    // ---- boundary bin of the top 12 bits (every CTA, from the row's histogram)
    const uint32_t* h = hsum;
    // the warp's first span is loaded while the boundary bin is found
    float vf[32];
    const int64_t w00 = s_lo + (int64_t)warp * kWarpSpan;
    const int n00 = (int)max((int64_t)0, min((int64_t)kWarpSpan, s_hi - w00));
    if (n00 > 0) load_span(row, w00, n00, lane, vf);
    int b1;
    uint32_t above1;
    __syncthreads();                                  // the histogram copy
    find_bin(h, kBins12, (uint32_t)k, sh_scan, sh_res, &b1, &above1);
    const bool fast = above1 + h[b1] <= (uint32_t)cap;
    if (tid == 0) sh_nc = 0;
    for (int i = tid; i < kBins12; i += nthr) hmine[i] = 0;
    __syncthreads();
    // ---- candidates of the slice (spans of 1024 entries)
    if (fast) {
        const float tv = bin_floor_value(b1);
        if (n00 > 0) collect_loaded(row, w00, n00, tv, vf, cs, &sh_nc, lane, cap);
        for (int64_t w0 = w00 + (int64_t)nw * kWarpSpan; w0 < s_hi; w0 += (int64_t)nw * kWarpSpan) {
            const int cnt = (int)min((int64_t)kWarpSpan, s_hi - w0);
            float v[32];
            load_span(row, w0, cnt, lane, v);
            collect_loaded(row, w0, cnt, tv, v, cs, &sh_nc, lane, cap);
        }
    }
    __syncthreads();
    const int nc = fast ? min(sh_nc, cap) : 0;
    if (fast) {
        // ---- every CTA gathers the row's candidates from the cluster and resolves the row alone
        cl.sync();                                  // every candidate list is complete
        if (p == 0)                                 // every CTA has its copy: clear the row's histogram
            for (int i = tid; i < kBins12; i += nthr) hrow[i] = 0u;
        // list sizes of all CTAs (one remote read each), then one pass over the concatenation in
        // which a thread's remote loads are independent (two in flight per iteration)
        int off[kMaxCluster + 1];
        off[0] = 0;
#pragma unroll
        for (int q = 0; q < kMaxCluster; ++q)
            off[q + 1] = q < P ? min(off[q] + *cl.map_shared_rank(&sh_nc, q), cap) : off[q];   // the row holds <= cap
        const int tot = off[kMaxCluster];
        auto src_of = [&](int i) -> const uint2* {
            int q = 0, start = 0;
#pragma unroll
            for (int j = 1; j < kMaxCluster; ++j)
                if (i >= off[j]) {
                    q = j;
                    start = off[j];
                }
            const uint2* base = q == p ? cs : cl.map_shared_rank(cs, q);
            return base + (i - start);
        };
        for (int i = tid; clustered && i < tot; i += 2 * nthr) {   // (one CTA: its list is the row's)
            const int i2 = i + nthr;
            const uint2 x = *src_of(i);
            const uint2 y = i2 < tot ? *src_of(i2) : make_uint2(0u, 0u);
            ga[i] = x;
            if (i2 < tot) ga[i2] = y;
        }
        __syncthreads();
        cluster_arrive_release();                   // done with the other CTAs' lists (waited at the end)
        // bits 19..8 and 7..0 of the boundary bin's members
        for (int i = tid; i < tot; i += nthr) {
            const uint32_t key = ga[i].x;
            if ((int)(key >> 20) == b1) atomicAdd(&hmine[(key >> 8) & 0xFFFu], 1u);
        }
        __syncthreads();
        int b2;
        uint32_t above2;
        find_bin(hmine, kBins12, (uint32_t)k - above1, sh_scan, sh_res, &b2, &above2);
        const uint32_t pre = ((uint32_t)b1 << 12) | (uint32_t)b2;
        for (int i = tid; i < kBins12; i += nthr) hsum[i] = 0;
        __syncthreads();
        for (int i = tid; i < tot; i += nthr) {
            const uint32_t key = ga[i].x;
            if ((key >> 8) == pre) atomicAdd(&hsum[key & 0xFFu], 1u);
        }
        __syncthreads();
        int b3;
        uint32_t above3;
        find_bin(hsum, kBins8 < nthr ? nthr : kBins8, (uint32_t)k - above1 - above2, sh_scan, sh_res, &b3, &above3);
        const uint32_t thr = (pre << 8) | (uint32_t)b3;
        const int ties_needed = (int)((uint32_t)k - above1 - above2 - above3);
        // selected entries before this CTA's slice: its output offset, and the ties already taken
        if (tid == 0) {
            sh_cnt[0] = 0;
            sh_cnt[1] = 0;
        }
        for (int64_t w = tid; w < sw; w += nthr) {
            wr[w] = 0u;
            tr[w] = 0u;
        }
        __syncthreads();
        int a_before = 0, t_before = 0;
        for (int i = tid; i < tot; i += nthr) {
            const uint2 e = ga[i];
            if ((int64_t)e.y < s_lo) {
                a_before += e.x > thr;
                t_before += e.x == thr;
            }
        }
        a_before = __reduce_add_sync(0xffffffffu, a_before);
        t_before = __reduce_add_sync(0xffffffffu, t_before);
        if (lane == 0) {
            atomicAdd(&sh_cnt[0], a_before);
            atomicAdd(&sh_cnt[1], t_before);
        }
        // this slice's bitmaps, from its own candidates
        for (int i = tid; i < nc; i += nthr) {
            const uint2 e = cs[i];
            const uint32_t li = e.y - (uint32_t)s_lo;
            if (e.x > thr) atomicOr(&wr[li >> 5], 1u << (li & 31));
            else if (e.x == thr) atomicOr(&tr[li >> 5], 1u << (li & 31));
        }
        __threadfence_block();
        __syncthreads();
        const int out_off = sh_cnt[0] + min(ties_needed, sh_cnt[1]);
        const int my_ties = max(0, ties_needed - sh_cnt[1]);
        const int64_t per = (sw + nthr - 1) / nthr;
        const int64_t v0 = min(sw, (int64_t)tid * per), v1 = min(sw, v0 + per);
        int nwin = 0, ntie = 0;
        for (int64_t w = v0; w < v1; ++w) {
            nwin += __popc(wr[w]);
            ntie += __popc(tr[w]);
        }
        // the first my_ties ties of the slice in index order are taken: the takes before a thread
        // add up to min(my_ties, ties before it)
        const int2 before = block_exclusive_scan2(nwin, ntie, sh_scan2);
        const int take = max(0, min(my_ties - before.y, ntie));
        int pos = out_off + before.x + min(my_ties, before.y), rem = take;
        for (int64_t w = v0; w < v1; ++w) {
            uint32_t t = tr[w];
            uint32_t tsel = 0;
            while (t && rem > 0) {
                const uint32_t low = t & (~t + 1u);
                tsel |= low;
                t ^= low;
                --rem;
            }
            uint32_t bits = wr[w] | tsel;
            while (bits) {
                const int b = __ffs(bits) - 1;
                if (pos < k) out[pos] = (int32_t)(s_lo + (w * 32 + b));
                ++pos;
                bits &= bits - 1;
            }
        }
        cluster_wait_acquire();                     // the others have finished reading this CTA's list
        return;
    }
    // ---- the slow path: the boundary bin holds too many entries for the candidate lists; every
    // pass re-reads the slice and the histograms are summed over the cluster
    // visits (key, index) of this CTA's part: its candidates, or its whole slice
    auto for_each = [&](auto&& f) {
        if (fast) {
            for (int i = tid; i < nc; i += nthr) f(cs[i].x, (int64_t)cs[i].y);
        } else {
            for (int64_t s = s_lo + tid; s < s_hi; s += nthr) f(ordered_key(row[s]), s);
        }
    };
    // ---- bits 19..8 inside the boundary bin, summed over the cluster
    for_each([&](uint32_t key, int64_t) {
        if ((int)(key >> 20) == b1) atomicAdd(&hmine[(key >> 8) & 0xFFFu], 1u);
    });
    cl.sync();
    cluster_sum(cl, hmine, hsum, kBins12);
    cl.sync();                                      // every CTA has read the others' histograms
    int b2;
    uint32_t above2;
    find_bin(hsum, kBins12, (uint32_t)k - above1, sh_scan, sh_res, &b2, &above2);
    // ---- bits 7..0 inside the 24-bit prefix
    const uint32_t pre = ((uint32_t)b1 << 12) | (uint32_t)b2;
    for (int i = tid; i < kBins12; i += nthr) hmine[i] = 0;
    __syncthreads();
    for_each([&](uint32_t key, int64_t) {
        if ((key >> 8) == pre) atomicAdd(&hmine[key & 0xFFu], 1u);
    });
    cl.sync();
    const int nb3 = kBins8 < nthr ? nthr : kBins8;
    cluster_sum(cl, hmine, hsum, nb3);
    __syncthreads();
    int b3;
    uint32_t above3;
    find_bin(hsum, nb3, (uint32_t)k - above1 - above2, sh_scan, sh_res, &b3, &above3);
    const uint32_t thr = (pre << 8) | (uint32_t)b3;
    const int ties_needed = (int)((uint32_t)k - above1 - above2 - above3);
    // ---- bitmaps of the slice
    for (int64_t w = tid; w < sw; w += nthr) {
        wr[w] = 0u;
        tr[w] = 0u;
    }
    __syncthreads();
    if (fast) {
        for (int i = tid; i < nc; i += nthr) {
            const uint2 e = cs[i];
            const uint32_t li = e.y - (uint32_t)s_lo;
            if (e.x > thr) atomicOr(&wr[li >> 5], 1u << (li & 31));
            else if (e.x == thr) atomicOr(&tr[li >> 5], 1u << (li & 31));
        }
    } else {
        for (int64_t g = s_lo + (int64_t)warp * 32; g < s_hi; g += (int64_t)nw * 32) {
            const int64_t s = g + lane;
            const uint32_t key = s < s_hi ? ordered_key(row[s]) : 0u;
            const uint32_t wb = __ballot_sync(0xffffffffu, s < s_hi && key > thr);
            const uint32_t tb = __ballot_sync(0xffffffffu, s < s_hi && key == thr);
            if (lane == 0) {
                wr[(g - s_lo) / 32] = wb;
                tr[(g - s_lo) / 32] = tb;
            }
        }
    }
    __threadfence_block();
    __syncthreads();
    // ---- per-thread word ranges; this CTA's counts, shared with the cluster
    const int64_t per = (sw + nthr - 1) / nthr;
    const int64_t v0 = min(sw, (int64_t)tid * per), v1 = min(sw, v0 + per);
    int nwin = 0, ntie = 0;
    for (int64_t w = v0; w < v1; ++w) {
        nwin += __popc(wr[w]);
        ntie += __popc(tr[w]);
    }
    int tot_win, tot_tie;
    const int tie_before_local = block_exclusive_scan(ntie, sh_scan, &tot_tie);
    (void)block_exclusive_scan(nwin, sh_scan, &tot_win);
    if (tid == 0) {
        sh_cnt[0] = tot_win;
        sh_cnt[1] = tot_tie;
    }
    cl.sync();
    // ties go to the lowest indices: the CTAs before this one take theirs first
    int ties_before = 0, out_off = 0;
    for (int q = 0; q < p; ++q) {
        const int* c = cl.map_shared_rank(sh_cnt, q);
        const int aq = c[0], tq = c[1];
        const int take_q = max(0, min(ties_needed - ties_before, tq));
        out_off += aq + take_q;
        ties_before += tq;
    }
    cl.sync();                                      // the last reads of another CTA's shared memory
    if (p == 0)                                     // every CTA has read the histogram: clear it
        for (int i = tid; i < kBins12; i += nthr) hrow[i] = 0u;
    const int my_ties = max(0, min(ties_needed - ties_before, tot_tie));
    const int take = max(0, min(my_ties - tie_before_local, ntie));
    int tot;
    const int pos0 = block_exclusive_scan(nwin + take, sh_scan, &tot);
    int pos = out_off + pos0, rem = take;
    for (int64_t w = v0; w < v1; ++w) {
        uint32_t t = tr[w];
        uint32_t tsel = 0;
        while (t && rem > 0) {
            const uint32_t low = t & (~t + 1u);
            tsel |= low;
            t ^= low;
            --rem;
        }
        uint32_t bits = wr[w] | tsel;
        while (bits) {
            const int b = __ffs(bits) - 1;
            if (pos < k) out[pos] = (int32_t)(s_lo + (w * 32 + b));
            ++pos;
            bits &= bits - 1;
        }
    }
}

}  // namespace

size_t topk_workspace_bytes(int64_t R, int64_t stride) {
    const int64_t words = (stride + 31) / 32;
    return align256((size_t)R * kBins12 * 4) + align256((size_t)R * words * 4) * 2;
}

TopkWorkspace topk_carve(void* ws, int64_t R, int64_t stride) {
    TopkWorkspace t;
    t.words = (stride + 31) / 32;
    char* p = static_cast<char*>(ws);
    t.hist1 = reinterpret_cast<uint32_t*>(p); p += align256((size_t)R * kBins12 * 4);
    t.win = reinterpret_cast<uint32_t*>(p); p += align256((size_t)R * t.words * 4);
    t.tie = reinterpret_cast<uint32_t*>(p);
    return t;
}


csahca_status topk_launch(const float* scores, int64_t stride, int R, const int64_t* n_vis_arr,
                          const int64_t* q_pos, int m, int64_t Ncap, int k, int32_t* idx_out,
                          const TopkWorkspace& tw, bool hist_ready, cudaStream_t stream) {
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSelSmem) !=
                cudaSuccess ||
            cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) != cudaSuccess)
            return CSAHCA_ERR_CUDA;
        attr_set[dev] = true;
    }
    // CTAs per row (one cluster per row): spread few rows over the SMs, one CTA per row otherwise
    const int64_t spans = std::max<int64_t>(1, cdiv(stride, (int64_t)kWarpSpan * (kSelThreads / 32)));
    int P = (int)std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(num_sms() / R, kMaxCluster), spans));
    while (P & (P - 1)) --P;                         // a power of two
    // One CTA per row (many rows, short rows): a lean form -- 512 threads, 4096 candidates, bitmaps
    // sized to the row, no gathered copy -- so that two CTAs share an SM.
    const bool lean = P == 1 && tw.words <= 4096;
    // Without the indexer's histogram: one CTA per row forms its row's histogram itself; several
    // CTAs per row need the row's histogram first (a pass of its own).  (The histograms are zero
    // on entry: the workspace starts zero-filled and every select pass clears the rows it used.)
    const int self_hist = (!hist_ready && P == 1) ? 1 : 0;
    if (!hist_ready && !self_hist) {
        const int64_t HP = std::max<int64_t>(1, cdiv(stride, kSlice));
        (void)launch_pdl(topk_hist_kernel, dim3((unsigned)HP, (unsigned)R), dim3(kThreads), 0, stream, scores, stride,
                         n_vis_arr, q_pos, m, Ncap, tw.hist1);
        count_launch();
        CSAHCA_CHECK_LAUNCH();
    }
    const int threads = lean ? 512 : kSelThreads;
    const int cap = lean ? 4096 : kCap;
    const int smem_words = lean ? (int)tw.words : kSmemWords;
    const size_t smem = (size_t)(P > 1 ? 2 : 1) * cap * 8 + 2 * (size_t)kBins12 * 4 + 2 * (size_t)smem_words * 4;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)P, (unsigned)R);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)P;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    (void)cudaLaunchKernelEx(&cfg, topk_select_kernel, scores, stride, n_vis_arr, q_pos, m, Ncap, k,
                             tw.hist1, tw.win, tw.tie, tw.words, idx_out, cap, smem_words, self_hist);
    count_launch();
    CSAHCA_CHECK_LAUNCH();
    return CSAHCA_OK;
}

}  // namespace csahca

using namespace csahca;

extern "C" {

size_t csa_topk_workspace(int R, int64_t row_stride, int k) {
    (void)k;
    if (R <= 0 || row_stride < 0) return 0;
    return topk_workspace_bytes(R, row_stride);
}

csahca_status csa_topk_from_scores(const float* scores, int64_t row_stride, int R, const int64_t* n_vis, int k,
                                   int32_t* idx_out, void* workspace, size_t ws_bytes, csahca_stream_t stream) {
    CSAHCA_REQUIRE(scores && n_vis && idx_out && R >= 1 && row_stride >= 1 && k >= 1 && k <= 65536);
    CSAHCA_REQUIRE(R <= 65535);
    if (!workspace || !aligned(workspace, 256) || ws_bytes < topk_workspace_bytes(R, row_stride))
        return CSAHCA_ERR_WORKSPACE;
    TopkWorkspace tw = topk_carve(workspace, R, row_stride);
    return topk_launch(scores, row_stride, R, n_vis, nullptr, 1, row_stride, k, idx_out, tw, false,
                       (cudaStream_t)stream);
}

}  // extern "C"
