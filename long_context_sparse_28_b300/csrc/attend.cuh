// Shared definitions of the attention kernels: argument block, key-list rules, split plan.
#pragma once
#include "common.cuh"

namespace csahca {

struct AttendArgs {
    bool is_csa;
    const void* q;
    int B, T, H, d;
    float scale;
    const void* ck;
    const void* cv;
    int64_t Ncap;
    const int32_t* idx;   // CSA: [B*T][k]
    int k;                // CSA: selected entries per query
    int m;                // HCA: block size (visibility)
    const void* ring_k;
    const void* ring_v;
    int ring_cap, W;
    const void* chunk_k;
    const void* chunk_v;
    const int64_t* chunk_pos0;
    int64_t chunk_stride;
    const int64_t* q_pos;
    csahca_dtype dtype;
    void* out;
    float* lse;
    int64_t total_max;    // upper bound of keys per query (sizes the split plan)
};

// Keys of one query, in order: n_c compressed keys (CSA: the k selected slots, HCA: every
// visible entry), then the W window slots (token p-W+1+i; slots before token 0 are empty).
struct KeyList {
    int64_t n_c;
    int64_t total;
};

__device__ __forceinline__ KeyList key_list(const AttendArgs& a, int r, int b, int64_t p) {
    (void)r; (void)b;
    KeyList kl;
    if (a.is_csa) {
        kl.n_c = a.k;
    } else {
        // (integer division is slow on the GPU: shift when the block size is a power of two)
        const int64_t n = (p < 0) ? 0 : ((a.m & (a.m - 1)) == 0 ? (p + 1) >> (__ffs(a.m) - 1) : (p + 1) / a.m);
        kl.n_c = n < a.Ncap ? n : a.Ncap;
    }
    kl.total = kl.n_c + a.W;
    return kl;
}

// Row pointers of key `key` of query row r (nullptr/nullptr for an empty slot).
template <typename T>
__device__ __forceinline__ void key_rows(const AttendArgs& a, const KeyList& kl, int r, int b, int64_t p,
                                         int64_t key, const T** kp, const T** vp, unsigned* err) {
    *kp = nullptr;
    *vp = nullptr;
    const int d = a.d;
    if (key < kl.n_c) {
        int64_t e = key;
        if (a.is_csa) {
            e = a.idx[(int64_t)r * a.k + key];
            if (e < 0) return;
            if (e >= a.Ncap) {
                flag_error(err, ERRBIT_BOUNDS);
                return;
            }
        }
        const int64_t off = ((int64_t)b * a.Ncap + e) * d;
        *kp = static_cast<const T*>(a.ck) + off;
        *vp = static_cast<const T*>(a.cv) + off;
        return;
    }
    const int64_t t = p - a.W + 1 + (key - kl.n_c);
    if (t < 0) return;
    if (a.chunk_k != nullptr && t >= a.chunk_pos0[b]) {
        const int64_t i = t - a.chunk_pos0[b];
        if (i >= a.chunk_stride) {
            flag_error(err, ERRBIT_BOUNDS);
            return;
        }
        const int64_t off = ((int64_t)b * a.chunk_stride + i) * d;
        *kp = static_cast<const T*>(a.chunk_k) + off;
        *vp = static_cast<const T*>(a.chunk_v) + off;
        return;
    }
    const int64_t off = ((int64_t)b * a.ring_cap + (t % a.ring_cap)) * d;
    *kp = static_cast<const T*>(a.ring_k) + off;
    *vp = static_cast<const T*>(a.ring_v) + off;
}

// Upper bound of a query's keys in tile space (both attention paths size their split plan with
// it): the compressed keys rounded up to whole 128-key tiles, then the window likewise.
inline int64_t tile_space_keys(int64_t n_c_max, int64_t W) { return cdiv(n_c_max, 128) * 128 + cdiv(W, 128) * 128; }

struct SplitPlan {
    int S;     // splits per query
    int kps;   // keys per split (multiple of 128)
};
SplitPlan plan_splits(int R, int64_t total_max, int splits_req);
// Workspace: per-row arrival counters (kRowCounterBytes, zero between calls: the tensor-core path's
// last CTA of a row merges the row's partials and resets its counter), then the partials.
constexpr size_t kRowCounterBytes = 65536 * 4;
size_t attend_workspace_bytes(int R, int H, int d, const SplitPlan& sp);
// Host-side argument checks and the split + merge launch sequence shared by the entry points.
csahca_status attend_validate(const AttendArgs& a);
csahca_status attend_run(const AttendArgs& a, int splits_req, void* workspace, size_t ws_bytes, cudaStream_t st);

// Tensor-core path (bf16, d = 128): availability and launch of the split kernel.
bool attend_tc_supported(const AttendArgs& a);
// True when the tensor-core kernel merges the rows' partials itself (few query rows).
bool attend_tc_merges(const AttendArgs& a, int S);
// The kernel also merges each row's partials into a.out / a.lse (the row's last CTA, counted in
// row_cnt), so no merge launch follows it.
cudaError_t attend_tc_launch(const AttendArgs& a, int S, int kps, float* o_part, float* lse_part, unsigned* row_cnt,
                             unsigned* err,
                             cudaStream_t st);

}  // namespace csahca
