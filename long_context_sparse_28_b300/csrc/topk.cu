// a6: per-query top-k over float32 indexer scores (honbul.tistory.com/221 "CSA": the Top-k
// Selector keeps only part of the compressed entries; pogovet.com detail 4: the indexer picks
// the top-k compressed blocks of every query).
//
// Exact radix select on the order-preserving 32-bit image of each score (12 + 12 + 8 bits):
//   hist   : 4096-bin histogram of the top 12 bits per row -- fused into the indexer's
//            tensor-core epilogue, or a separate pass over the scores;
//   select : one launch, P CTAs per row.  Every CTA of a row finds the boundary bin b1 where the
//            running count from the top reaches k; when the elements of bins >= b1 number at
//            most kCap, each CTA appends those of its slice of the row, (key, index), to the
//            row's candidate list.  The last CTA of the row to finish (an arrival counter; no
//            CTA waits for another) resolves the remaining 20 bits on the candidates (or, when
//            the boundary bin is too full, on the whole row), marks "above the threshold" and
//            "equal to the threshold" entries in two bitmaps, then scans the bitmaps in index
//            order: every "above" bit plus the lowest-index "equal" bits needed to reach k.
// Output: indices ascending, -1 padded.  Ties go to the lower index; the result is exact and
// deterministic for any non-NaN scores (-0 == +0).
#include "common.cuh"

namespace csahca {
namespace {

constexpr int kBins12 = 4096;
constexpr int kBins8 = 256;
constexpr int kSlice = 8192;       // scores per histogram CTA
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
    for (int64_t s = s0 + threadIdx.x; s < s1; s += blockDim.x) atomicAdd(&sh[ordered_key(row[s]) >> 20], 1u);
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
constexpr int kSmemWords = 8192;   // bitmaps in shared memory for rows of up to 262144 entries
constexpr size_t kSelSmem = (size_t)kCap * 8 + 2 * (size_t)kSmemWords * 4 + (size_t)kBins12 * 4;

// Appends the elements >= tv of the warp's span [w0, w0 + cnt_n) of `row` to the candidate list
// (16-byte loads when aligned and full, one atomic per warp).
__device__ __forceinline__ void collect_span(const float* __restrict__ row, int64_t w0, int cnt_n, float tv,
                                             uint2* cand_row, int* cand_cnt, int lane) {
    const float* src = row + w0;
    const bool vec = ((reinterpret_cast<uintptr_t>(src) & 15) == 0) && cnt_n == kWarpSpan;
    float v[32];
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
    if (lane == 0) base = atomicAdd(cand_cnt, total);
    base = __shfl_sync(0xffffffffu, base, 0) + incl - mine;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        if (bits & (1u << e)) {
            const int i = ((e >> 2) * 32 + lane) * 4 + (e & 3);
            if (base < kCap) cand_row[base] = make_uint2(ordered_key(v[e]), (uint32_t)(w0 + i));
            ++base;
        }
    }
}

// Grid (P, rows).  Threshold, collect and (last CTA of each row) exact finish; see the file
// comment.  Candidates and, for rows of up to kSmemWords * 32 entries, both bitmaps live in
// shared memory.
__global__ void __launch_bounds__(kSelThreads, 1) topk_select_kernel(
    const float* __restrict__ scores, int64_t stride, const int64_t* __restrict__ n_vis_arr,
    const int64_t* __restrict__ q_pos, int m, int64_t Ncap, int k, const uint32_t* __restrict__ hist1,
    uint2* cand, int* cand_n, int* done, uint32_t* __restrict__ win, uint32_t* __restrict__ tie, int64_t words,
    int32_t* __restrict__ idx_out) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) unsigned char fsm[];
    uint2* cs = reinterpret_cast<uint2*>(fsm);
    uint32_t* swin = reinterpret_cast<uint32_t*>(fsm + (size_t)kCap * 8);
    uint32_t* stie = swin + kSmemWords;
    uint32_t* sh_hist = stie + kSmemWords;
    __shared__ int sh_scan[33];
    __shared__ int sh_res[2];
    __shared__ int sh_last;
    const int r = blockIdx.y, P = gridDim.x;
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nthr >> 5;
    const int64_t n = min(row_nvis(r, n_vis_arr, q_pos, m, Ncap), min(stride, words * 32));
    const int64_t nwords = (n + 31) / 32;
    int32_t* out = idx_out + (int64_t)r * k;
    if (n <= k) {                                   // every visible entry is selected, in order
        if (blockIdx.x == 0)
            for (int j = tid; j < k; j += nthr) out[j] = j < n ? j : -1;
        return;
    }
    const float* row = scores + (int64_t)r * stride;
    // ---- boundary bin of the top 12 bits (every CTA of the row, from the same histogram)
    const uint32_t* h = hist1 + (int64_t)r * kBins12;
    int b1;
    uint32_t above1;
    find_bin(h, kBins12, (uint32_t)k, sh_scan, sh_res, &b1, &above1);
    const bool fast = above1 + h[b1] <= (uint32_t)kCap;
    // ---- collect: this CTA's spans of the row (span g of the row goes to CTA g % P)
    uint2* cand_row = cand + (int64_t)r * kCap;
    if (fast) {
        const float tv = bin_floor_value(b1);
        for (int64_t g = (int64_t)blockIdx.x + (int64_t)P * warp; g * kWarpSpan < n; g += (int64_t)P * nw) {
            const int64_t w0 = g * kWarpSpan;
            collect_span(row, w0, (int)min((int64_t)kWarpSpan, n - w0), tv, cand_row, &cand_n[r], lane);
        }
    }
    // ---- the last CTA of the row to get here resolves it
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        sh_last = atomicAdd(&done[r], 1) == P - 1;
    }
    __syncthreads();
    if (!sh_last) return;
    __threadfence();
    const bool smem_bits = nwords <= kSmemWords;
    uint32_t* wr = smem_bits ? swin : win + (int64_t)r * words;
    uint32_t* tr = smem_bits ? stie : tie + (int64_t)r * words;
    const int nc = fast ? min(__ldcg(&cand_n[r]), kCap) : 0;
    for (int i = tid; i < nc; i += nthr) cs[i] = __ldcg(&cand_row[i]);
    for (int64_t w = tid; w < nwords; w += nthr) {
        wr[w] = 0u;
        tr[w] = 0u;
    }
    for (int i = tid; i < kBins12; i += nthr) sh_hist[i] = 0;
    __syncthreads();
    // visits (key, index) of the source: the candidate list, or the whole row
    auto for_each = [&](auto&& f) {
        if (fast) {
            for (int i = tid; i < nc; i += nthr) f(cs[i].x, (int64_t)cs[i].y);
        } else {
            for (int64_t s = tid; s < n; s += nthr) f(ordered_key(row[s]), s);
        }
    };
    // bits 19..8 inside the boundary bin
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
    find_bin(sh_hist, kBins8 < nthr ? nthr : kBins8, (uint32_t)k - above1 - above2, sh_scan, sh_res, &b3, &above3);
    const uint32_t thr = (pre << 8) | (uint32_t)b3;
    const int ties_needed = (int)((uint32_t)k - above1 - above2 - above3);
    // bitmaps
    if (fast) {
        for (int i = tid; i < nc; i += nthr) {
            const uint2 e = cs[i];
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
}

}  // namespace

size_t topk_workspace_bytes(int64_t R, int64_t stride) {
    const int64_t words = (stride + 31) / 32;
    return align256((size_t)R * kBins12 * 4) + align256((size_t)R * 8) + align256((size_t)R * kCap * 8) +
           align256((size_t)R * words * 4) * 2;
}

TopkWorkspace topk_carve(void* ws, int64_t R, int64_t stride) {
    TopkWorkspace t;
    t.words = (stride + 31) / 32;
    char* p = static_cast<char*>(ws);
    t.hist1 = reinterpret_cast<uint32_t*>(p); p += align256((size_t)R * kBins12 * 4);
    t.cand_n = reinterpret_cast<int*>(p);
    t.done = t.cand_n + R;                      p += align256((size_t)R * 8);
    t.cand = reinterpret_cast<uint2*>(p); p += align256((size_t)R * kCap * 8);
    t.win = reinterpret_cast<uint32_t*>(p); p += align256((size_t)R * t.words * 4);
    t.tie = reinterpret_cast<uint32_t*>(p);
    return t;
}

size_t topk_zero_bytes(int64_t R) { return align256((size_t)R * kBins12 * 4) + align256((size_t)R * 8); }

csahca_status topk_launch(const float* scores, int64_t stride, int R, const int64_t* n_vis_arr,
                          const int64_t* q_pos, int m, int64_t Ncap, int k, int32_t* idx_out,
                          const TopkWorkspace& tw, bool hist_ready, cudaStream_t stream) {
    if (!hist_ready) {
        const int64_t P = std::max<int64_t>(1, cdiv(stride, kSlice));
        if (zero_words(tw.hist1, topk_zero_bytes(R) / 4, stream) != cudaSuccess) return CSAHCA_ERR_CUDA;
        (void)launch_pdl(topk_hist_kernel, dim3((unsigned)P, (unsigned)R), dim3(kThreads), 0, stream, scores, stride,
                         n_vis_arr, q_pos, m, Ncap, tw.hist1);
        count_launch();
        CSAHCA_CHECK_LAUNCH();
    }
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSelSmem) !=
            cudaSuccess)
            return CSAHCA_ERR_CUDA;
        attr_set[dev] = true;
    }
    // CTAs per row: one wave over the SMs for few rows (each row is collected by P CTAs and
    // finished by the last of them), one per row otherwise
    const int64_t spans = std::max<int64_t>(1, cdiv(stride, (int64_t)kWarpSpan * (kSelThreads / 32)));
    const int P = (int)std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(num_sms() / R, 8), spans));
    (void)launch_pdl(topk_select_kernel, dim3((unsigned)P, (unsigned)R), dim3(kSelThreads), kSelSmem, stream, scores,
                     stride, n_vis_arr, q_pos, m, Ncap, k, tw.hist1, tw.cand, tw.cand_n, tw.done, tw.win, tw.tie,
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
    return topk_launch(scores, row_stride, R, n_vis, nullptr, 1, row_stride, k, idx_out, tw, false,
                       (cudaStream_t)stream);
}

}  // extern "C"
