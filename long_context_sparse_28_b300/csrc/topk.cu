// a6: per-query top-k over float32 indexer scores (honbul.tistory.com/221 "CSA": the Top-k
// Selector keeps only part of the compressed entries; pogovet.com detail 4: the indexer picks
// the top-k compressed blocks of every query).
//
// Exact radix select on the order-preserving 32-bit image of each score, split 12 + 12 + 8
// bits.  Every pass runs over (slice, row) CTAs so that long rows (262144 candidates) spread
// over the whole GPU; the per-row histograms live in global memory (L2), and each CTA
// re-derives the running threshold from them, so no CTA waits on another.
//   pass 1 : histogram of the top 12 bits
//   pass 2 : histogram of the next 12 bits among elements in the boundary bin
//   pass 3 : histogram of the low 8 bits among elements matching the 24-bit prefix
//   pass 4 : threshold known exactly -> bitmaps of "above" and "equal" candidates
//   compact: per row, ascending scan of the bitmaps; all "above" bits and the lowest-index
//            "equal" bits needed to reach k -> indices in ascending order, -1 padded.
// Ties are therefore broken by lower index, and the result is bit-exact for any scores.
#include "common.cuh"

namespace csahca {
namespace {

constexpr int kBins12 = 4096;
constexpr int kBins8 = 256;
constexpr int kSlice = 8192;       // candidates per CTA per pass (multiple of 32)
constexpr int kPassThreads = 256;

__device__ __forceinline__ int64_t row_nvis(int r, const int64_t* n_vis_arr, const int64_t* q_pos, int m,
                                            int64_t Ncap) {
    if (n_vis_arr) return n_vis_arr[r];
    const int64_t p = q_pos[r];
    int64_t v = (p >= 0) ? (p + 1) / m : 0;
    return v < Ncap ? v : Ncap;
}

// Finds the bin b (counting from the top) where the running count reaches `need`:
// above(b) < need <= above(b) + hist[b], above(b) = sum of the bins above b.
// nb must be a multiple of blockDim.x.  Results broadcast through shared memory.
__device__ void find_bin(const uint32_t* __restrict__ hist, int nb, uint32_t need, int* sh_scan, int* sh_res,
                         int* bin_out, uint32_t* above_out) {
    const int per = nb / blockDim.x;
    const int chunk = blockDim.x - 1 - threadIdx.x;      // thread 0 owns the highest bins
    const int lo = chunk * per;
    int local = 0;
    for (int i = 0; i < per; ++i) local += (int)hist[lo + i];
    int total;
    const int above = block_exclusive_scan(local, sh_scan, &total);
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

struct RowSel {
    int b1, b2, b3;
    uint32_t above1, above2, above3;
};

__global__ void __launch_bounds__(kPassThreads) topk_pass_kernel(
    int pass, const float* __restrict__ scores, int64_t stride, const int64_t* __restrict__ n_vis_arr,
    const int64_t* __restrict__ q_pos, int m, int64_t Ncap, int k, uint32_t* hist1, uint32_t* hist2,
    uint32_t* hist3, uint32_t* win, uint32_t* tie, int32_t* ties_needed, int64_t words) {
    __shared__ uint32_t sh_hist[kBins12];
    __shared__ int sh_scan[33];
    __shared__ int sh_res[2];
    const int r = blockIdx.y;
    const int64_t n = min(row_nvis(r, n_vis_arr, q_pos, m, Ncap), stride);   // never read past the row
    const int64_t s0 = (int64_t)blockIdx.x * kSlice;
    if (s0 >= n && !(pass == 4 && blockIdx.x == 0)) return;       // CTA-uniform
    const bool all_selected = n <= k;
    if (all_selected && pass != 4) return;
    const float* row = scores + (int64_t)r * stride;
    const int64_t s1 = min(n, s0 + kSlice);

    RowSel sel{0, 0, 0, 0, 0, 0};
    if (pass >= 2 && !all_selected) {
        find_bin(hist1 + (int64_t)r * kBins12, kBins12, (uint32_t)k, sh_scan, sh_res, &sel.b1, &sel.above1);
    }
    if (pass >= 3 && !all_selected) {
        find_bin(hist2 + (int64_t)r * kBins12, kBins12, (uint32_t)k - sel.above1, sh_scan, sh_res, &sel.b2,
                 &sel.above2);
    }
    if (pass >= 4 && !all_selected) {
        find_bin(hist3 + (int64_t)r * kBins8, kBins8, (uint32_t)k - sel.above1 - sel.above2, sh_scan, sh_res,
                 &sel.b3, &sel.above3);
    }

    if (pass <= 3) {
        const int nb = (pass == 3) ? kBins8 : kBins12;
        for (int i = threadIdx.x; i < nb; i += blockDim.x) sh_hist[i] = 0;
        __syncthreads();
        const uint32_t pre24 = ((uint32_t)sel.b1 << 12) | (uint32_t)sel.b2;
        for (int64_t s = s0 + threadIdx.x; s < s1; s += blockDim.x) {
            const uint32_t key = ordered_key(row[s]);
            if (pass == 1) {
                atomicAdd(&sh_hist[key >> 20], 1u);
            } else if (pass == 2) {
                if ((int)(key >> 20) == sel.b1) atomicAdd(&sh_hist[(key >> 8) & 0xFFFu], 1u);
            } else {
                if ((key >> 8) == pre24) atomicAdd(&sh_hist[key & 0xFFu], 1u);
            }
        }
        __syncthreads();
        uint32_t* gh = (pass == 1 ? hist1 : pass == 2 ? hist2 : hist3) + (int64_t)r * nb;
        for (int i = threadIdx.x; i < nb; i += blockDim.x)
            if (sh_hist[i]) atomicAdd(&gh[i], sh_hist[i]);
        return;
    }

    // pass 4: exact threshold -> bitmaps
    const uint32_t thr = all_selected ? 0u
                                      : (((uint32_t)sel.b1 << 20) | ((uint32_t)sel.b2 << 8) | (uint32_t)sel.b3);
    if (blockIdx.x == 0 && threadIdx.x == 0)
        ties_needed[r] = all_selected ? 0 : (int32_t)((uint32_t)k - sel.above1 - sel.above2 - sel.above3);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int64_t g = s0 + (int64_t)warp * 32; g < s1; g += (int64_t)nw * 32) {
        const int64_t s = g + lane;
        const bool valid = s < s1;
        uint32_t key = 0;
        if (valid) key = ordered_key(row[s]);
        const uint32_t wb = __ballot_sync(0xffffffffu, valid && (all_selected || key > thr));
        const uint32_t tb = __ballot_sync(0xffffffffu, valid && !all_selected && key == thr);
        if (lane == 0) {
            win[(int64_t)r * words + g / 32] = wb;
            tie[(int64_t)r * words + g / 32] = tb;
        }
    }
}

__global__ void __launch_bounds__(1024) topk_compact_kernel(const int64_t* __restrict__ n_vis_arr,
                                                            const int64_t* __restrict__ q_pos, int m, int64_t Ncap,
                                                            int k, const uint32_t* __restrict__ win,
                                                            const uint32_t* __restrict__ tie,
                                                            const int32_t* __restrict__ ties_needed, int64_t words,
                                                            int32_t* __restrict__ idx_out) {
    __shared__ int sh_scan[33];
    const int r = blockIdx.x;
    const int64_t n = min(row_nvis(r, n_vis_arr, q_pos, m, Ncap), words * 32);
    const int64_t nwords = (n + 31) / 32;
    const int64_t per = (nwords + blockDim.x - 1) / blockDim.x;
    const int64_t w0 = min(nwords, (int64_t)threadIdx.x * per), w1 = min(nwords, w0 + per);
    const uint32_t* wr = win + (int64_t)r * words;
    const uint32_t* tr = tie + (int64_t)r * words;
    int nwin = 0, ntie = 0;
    for (int64_t w = w0; w < w1; ++w) {
        nwin += __popc(wr[w]);
        ntie += __popc(tr[w]);
    }
    int tot;
    const int tie_before = block_exclusive_scan(ntie, sh_scan, &tot);
    const int need = (n > 0) ? ties_needed[r] : 0;
    const int take = max(0, min(need - tie_before, ntie));
    const int pos0 = block_exclusive_scan(nwin + take, sh_scan, &tot);
    int32_t* out = idx_out + (int64_t)r * k;
    int pos = pos0, rem = take;
    for (int64_t w = w0; w < w1; ++w) {
        uint32_t t = tr[w];
        uint32_t tsel = 0;
        while (t && rem > 0) {                 // lowest-index ties first
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
    const int total = min((int64_t)k, n) > 0 ? (int)min((int64_t)k, n) : 0;
    for (int j = total + threadIdx.x; j < k; j += blockDim.x) out[j] = -1;
}

}  // namespace

size_t topk_workspace_bytes(int64_t R, int64_t stride) {
    const int64_t words = (stride + 31) / 32;
    return align256((size_t)R * kBins12 * 4) * 2 + align256((size_t)R * kBins8 * 4) +
           align256((size_t)R * words * 4) * 2 + align256((size_t)R * 4);
}

TopkWorkspace topk_carve(void* ws, int64_t R, int64_t stride) {
    TopkWorkspace t;
    t.words = (stride + 31) / 32;
    char* p = static_cast<char*>(ws);
    t.hist1 = reinterpret_cast<uint32_t*>(p); p += align256((size_t)R * kBins12 * 4);
    t.hist2 = reinterpret_cast<uint32_t*>(p); p += align256((size_t)R * kBins12 * 4);
    t.hist3 = reinterpret_cast<uint32_t*>(p); p += align256((size_t)R * kBins8 * 4);
    t.win = reinterpret_cast<uint32_t*>(p); p += align256((size_t)R * t.words * 4);
    t.tie = reinterpret_cast<uint32_t*>(p); p += align256((size_t)R * t.words * 4);
    t.ties_needed = reinterpret_cast<int32_t*>(p);
    return t;
}

csahca_status topk_launch(const float* scores, int64_t stride, int R, const int64_t* n_vis_arr,
                          const int64_t* q_pos, int m, int64_t Ncap, int k, int32_t* idx_out,
                          const TopkWorkspace& tw, cudaStream_t stream) {
    const size_t hist_bytes = reinterpret_cast<char*>(tw.win) - reinterpret_cast<char*>(tw.hist1);
    if (cudaMemsetAsync(tw.hist1, 0, hist_bytes, stream) != cudaSuccess) return CSAHCA_ERR_CUDA;
    const int64_t P = std::max<int64_t>(1, cdiv(stride, kSlice));
    dim3 grid((unsigned)P, (unsigned)R);
    for (int pass = 1; pass <= 4; ++pass) {
        topk_pass_kernel<<<grid, kPassThreads, 0, stream>>>(pass, scores, stride, n_vis_arr, q_pos, m, Ncap, k,
                                                            tw.hist1, tw.hist2, tw.hist3, tw.win, tw.tie,
                                                            tw.ties_needed, tw.words);
        count_launch();
        CSAHCA_CHECK_LAUNCH();
    }
    topk_compact_kernel<<<R, 1024, 0, stream>>>(n_vis_arr, q_pos, m, Ncap, k, tw.win, tw.tie, tw.ties_needed,
                                                tw.words, idx_out);
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
    return topk_launch(scores, row_stride, R, n_vis, nullptr, 1, row_stride, k, idx_out, tw, (cudaStream_t)stream);
}

}  // extern "C"
