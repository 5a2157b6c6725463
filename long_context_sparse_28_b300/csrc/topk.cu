// a6: per-query top-k over float32 indexer scores (honbul.tistory.com/221 "CSA": the Top-k
// Selector keeps only part of the compressed entries; pogovet.com detail 4: the indexer picks
// the top-k compressed blocks of every query).
//
// Exact radix select on the order-preserving 32-bit image of each score (12 + 12 + 8 bits):
//   hist  : 4096-bin histogram of the top 12 bits per row -- fused into the indexer's
//           tensor-core epilogue, or a separate pass over the scores;
//   collect (slices x rows CTAs): every CTA finds the boundary bin b1 from the histogram; when
//           the elements in bins >= b1 number at most kCap, they are appended (key, index) to a
//           per-row candidate list;
//   finish (one CTA per row): resolves the remaining 20 bits on the candidates (or, for rows
//           whose boundary bin is too full, on the whole row), marks "above the threshold" and
//           "equal to the threshold" entries in two bitmaps, then scans the bitmaps in index
//           order: every "above" bit plus the lowest-index "equal" bits needed to reach k.
// Output: indices ascending, -1 padded.  Ties go to the lower index; the result is exact and
// deterministic for any non-NaN scores (-0 == +0).
#include "common.cuh"

namespace csahca {
namespace {

constexpr int kBins12 = 4096;
constexpr int kBins8 = 256;
constexpr int kSlice = 8192;       // candidates per collect CTA (multiple of 32)
constexpr int kCap = 8192;         // candidate-list capacity per row
constexpr int kThreads = 256;
constexpr int kFinishThreads = 1024;

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
    __shared__ uint32_t sh[kBins12];
    const int r = blockIdx.y;
    const int64_t n = min(row_nvis(r, n_vis_arr, q_pos, m, Ncap), stride);
    const int64_t s0 = (int64_t)blockIdx.x * kSlice;
    if (s0 >= n) return;
    const int64_t s1 = min(n, s0 + kSlice);
    for (int i = threadIdx.x; i < kBins12; i += blockDim.x) sh[i] = 0;
    __syncthreads();
    const float* row = scores + (int64_t)r * stride;
    for (int64_t s = s0 + threadIdx.x; s < s1; s += blockDim.x) atomicAdd(&sh[ordered_key(row[s]) >> 20], 1u);
    __syncthreads();
    uint32_t* gh = hist1 + (int64_t)r * kBins12;
    for (int i = threadIdx.x; i < kBins12; i += blockDim.x)
        if (sh[i]) atomicAdd(&gh[i], sh[i]);
}

// Appends every element of bins >= b1 to the row's candidate list when they fit.
__global__ void __launch_bounds__(kThreads) topk_collect_kernel(const float* __restrict__ scores, int64_t stride,
                                                                const int64_t* __restrict__ n_vis_arr,
                                                                const int64_t* __restrict__ q_pos, int m,
                                                                int64_t Ncap, int k, const uint32_t* __restrict__ hist1,
                                                                uint2* __restrict__ cand, int* __restrict__ cand_n) {
    __shared__ int sh_scan[33];
    __shared__ int sh_res[2];
    const int r = blockIdx.y;
    const int64_t n = min(row_nvis(r, n_vis_arr, q_pos, m, Ncap), stride);
    const int64_t s0 = (int64_t)blockIdx.x * kSlice;
    if (s0 >= n || n <= k) return;                       // CTA-uniform
    int b1;
    uint32_t above1;
    const uint32_t* h = hist1 + (int64_t)r * kBins12;
    find_bin(h, kBins12, (uint32_t)k, sh_scan, sh_res, &b1, &above1);
    if (above1 + h[b1] > (uint32_t)kCap) return;        // the finish kernel scans the whole row
    const int64_t s1 = min(n, s0 + kSlice);
    const float* row = scores + (int64_t)r * stride;
    const int lane = threadIdx.x & 31;
    for (int64_t base = s0 + (threadIdx.x & ~31); base < s1; base += blockDim.x) {
        const int64_t s = base + lane;
        uint32_t key = 0;
        bool take = false;
        if (s < s1) {
            key = ordered_key(row[s]);
            take = (int)(key >> 20) >= b1;
        }
        const uint32_t bal = __ballot_sync(0xffffffffu, take);
        if (bal) {
            int off = 0;
            if (lane == 0) off = atomicAdd(&cand_n[r], __popc(bal));
            off = __shfl_sync(0xffffffffu, off, 0);
            if (take) cand[(int64_t)r * kCap + off + __popc(bal & ((1u << lane) - 1u))] = make_uint2(key, (uint32_t)s);
        }
    }
}

// One CTA per row: exact threshold, bitmaps, ascending compaction.
__global__ void __launch_bounds__(kFinishThreads) topk_finish_kernel(
    const float* __restrict__ scores, int64_t stride, const int64_t* __restrict__ n_vis_arr,
    const int64_t* __restrict__ q_pos, int m, int64_t Ncap, int k, const uint32_t* __restrict__ hist1,
    const uint2* __restrict__ cand, const int* __restrict__ cand_n, uint32_t* __restrict__ win,
    uint32_t* __restrict__ tie, int64_t words, int32_t* __restrict__ idx_out) {
    __shared__ uint32_t sh_hist[kBins12];
    __shared__ int sh_scan[33];
    __shared__ int sh_res[2];
    const int r = blockIdx.x;
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nthr >> 5;
    const int64_t n = min(row_nvis(r, n_vis_arr, q_pos, m, Ncap), min(stride, words * 32));
    const int64_t nwords = (n + 31) / 32;
    uint32_t* wr = win + (int64_t)r * words;
    uint32_t* tr = tie + (int64_t)r * words;
    const float* row = scores + (int64_t)r * stride;
    int ties_needed = 0;

    if (n <= k) {                                         // every visible entry is selected
        for (int64_t w = tid; w < nwords; w += nthr) {
            const int64_t rem = n - w * 32;
            wr[w] = rem >= 32 ? 0xffffffffu : ((1u << rem) - 1u);
            tr[w] = 0u;
        }
    } else {
        int b1;
        uint32_t above1;
        const uint32_t* h1 = hist1 + (int64_t)r * kBins12;
        find_bin(h1, kBins12, (uint32_t)k, sh_scan, sh_res, &b1, &above1);
        const bool fast = above1 + h1[b1] <= (uint32_t)kCap;
        const int nc = fast ? cand_n[r] : 0;
        const uint2* cr = cand + (int64_t)r * kCap;
        // visits (key, index) of the source: the candidate list, or the whole row
        auto for_each = [&](auto&& f) {
            if (fast) {
                for (int i = tid; i < nc; i += nthr) {
                    const uint2 e = cr[i];
                    f(e.x, (int64_t)e.y);
                }
            } else {
                for (int64_t s = tid; s < n; s += nthr) f(ordered_key(row[s]), s);
            }
        };
        // bits 19..8 inside the boundary bin
        for (int i = tid; i < kBins12; i += nthr) sh_hist[i] = 0;
        __syncthreads();
        for_each([&](uint32_t key, int64_t) {
            if ((int)(key >> 20) == b1) atomicAdd(&sh_hist[(key >> 8) & 0xFFFu], 1u);
        });
        __syncthreads();
        int b2;
        uint32_t above2;
        find_bin(sh_hist, kBins12, (uint32_t)k - above1, sh_scan, sh_res, &b2, &above2);
        // bits 7..0 inside the 24-bit prefix
        const uint32_t pre = ((uint32_t)b1 << 12) | (uint32_t)b2;
        for (int i = tid; i < kBins12; i += nthr) sh_hist[i] = 0;
        __syncthreads();
        for_each([&](uint32_t key, int64_t) {
            if ((key >> 8) == pre) atomicAdd(&sh_hist[key & 0xFFu], 1u);
        });
        __syncthreads();
        int b3;
        uint32_t above3;
        find_bin(sh_hist, kBins8 < nthr ? nthr : kBins8, (uint32_t)k - above1 - above2, sh_scan, sh_res, &b3,
                 &above3);
        const uint32_t thr = (pre << 8) | (uint32_t)b3;
        ties_needed = (int)((uint32_t)k - above1 - above2 - above3);
        // bitmaps
        if (fast) {
            for (int64_t w = tid; w < nwords; w += nthr) {
                wr[w] = 0u;
                tr[w] = 0u;
            }
            __syncthreads();
            for (int i = tid; i < nc; i += nthr) {
                const uint2 e = cr[i];
                if (e.x > thr) atomicOr(&wr[e.y >> 5], 1u << (e.y & 31));
                else if (e.x == thr) atomicOr(&tr[e.y >> 5], 1u << (e.y & 31));
            }
        } else {
            for (int64_t g = (int64_t)warp * 32; g < n; g += (int64_t)nw * 32) {
                const int64_t s = g + lane;
                const uint32_t key = s < n ? ordered_key(row[s]) : 0u;
                const uint32_t wb = __ballot_sync(0xffffffffu, s < n && key > thr);
                const uint32_t tb = __ballot_sync(0xffffffffu, s < n && key == thr);
                if (lane == 0) {
                    wr[g / 32] = wb;
                    tr[g / 32] = tb;
                }
            }
        }
    }
    __threadfence_block();
    __syncthreads();
    // ascending compaction: all "above" bits, then the lowest-index "equal" bits
    const int64_t per = (nwords + nthr - 1) / nthr;
    const int64_t w0 = min(nwords, (int64_t)tid * per), w1 = min(nwords, w0 + per);
    int nwin = 0, ntie = 0;
    for (int64_t w = w0; w < w1; ++w) {
        nwin += __popc(wr[w]);
        ntie += __popc(tr[w]);
    }
    int tot;
    const int tie_before = block_exclusive_scan(ntie, sh_scan, &tot);
    const int take = max(0, min(ties_needed - tie_before, ntie));
    const int pos0 = block_exclusive_scan(nwin + take, sh_scan, &tot);
    int32_t* out = idx_out + (int64_t)r * k;
    int pos = pos0, rem = take;
    for (int64_t w = w0; w < w1; ++w) {
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
            if (pos < k) out[pos] = (int32_t)(w * 32 + b);
            ++pos;
            bits &= bits - 1;
        }
    }
    const int total = (int)min((int64_t)k, n);
    for (int j = total + tid; j < k; j += nthr) out[j] = -1;
}

}  // namespace

size_t topk_workspace_bytes(int64_t R, int64_t stride) {
    const int64_t words = (stride + 31) / 32;
    return align256((size_t)R * kBins12 * 4) + align256((size_t)R * 4) + align256((size_t)R * kCap * 8) +
           align256((size_t)R * words * 4) * 2;
}

TopkWorkspace topk_carve(void* ws, int64_t R, int64_t stride) {
    TopkWorkspace t;
    t.words = (stride + 31) / 32;
    char* p = static_cast<char*>(ws);
    t.hist1 = reinterpret_cast<uint32_t*>(p); p += align256((size_t)R * kBins12 * 4);
    t.cand_n = reinterpret_cast<int*>(p); p += align256((size_t)R * 4);
    t.cand = reinterpret_cast<uint2*>(p); p += align256((size_t)R * kCap * 8);
    t.win = reinterpret_cast<uint32_t*>(p); p += align256((size_t)R * t.words * 4);
    t.tie = reinterpret_cast<uint32_t*>(p);
    return t;
}

size_t topk_zero_bytes(int64_t R) { return align256((size_t)R * kBins12 * 4) + align256((size_t)R * 4); }

csahca_status topk_launch(const float* scores, int64_t stride, int R, const int64_t* n_vis_arr,
                          const int64_t* q_pos, int m, int64_t Ncap, int k, int32_t* idx_out,
                          const TopkWorkspace& tw, bool hist_ready, cudaStream_t stream) {
    const int64_t P = std::max<int64_t>(1, cdiv(stride, kSlice));
    dim3 grid((unsigned)P, (unsigned)R);
    if (!hist_ready) {
        if (cudaMemsetAsync(tw.hist1, 0, topk_zero_bytes(R), stream) != cudaSuccess) return CSAHCA_ERR_CUDA;
        topk_hist_kernel<<<grid, kThreads, 0, stream>>>(scores, stride, n_vis_arr, q_pos, m, Ncap, tw.hist1);
        count_launch();
        CSAHCA_CHECK_LAUNCH();
    }
    topk_collect_kernel<<<grid, kThreads, 0, stream>>>(scores, stride, n_vis_arr, q_pos, m, Ncap, k, tw.hist1,
                                                       tw.cand, tw.cand_n);
    count_launch();
    CSAHCA_CHECK_LAUNCH();
    topk_finish_kernel<<<R, kFinishThreads, 0, stream>>>(scores, stride, n_vis_arr, q_pos, m, Ncap, k, tw.hist1,
                                                         tw.cand, tw.cand_n, tw.win, tw.tie, tw.words, idx_out);
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
