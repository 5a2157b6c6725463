// Shared device/host helpers of the CSA + HCA CUDA library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/csa_hca.h"

namespace csahca {

// ------------------------------------------------------------------ error word / bookkeeping
enum : unsigned { ERRBIT_BOUNDS = 1u, ERRBIT_TIMEOUT = 2u };

// Device address of the error word on the current device (cached per device).
unsigned* err_word();
// Counts kernel launches enqueued by this library (per host thread).
void count_launch(int n = 1);

__device__ __forceinline__ void flag_error(unsigned* err, unsigned bit) { atomicOr(err, bit); }

#define CSAHCA_CHECK_LAUNCH()                                        \
    do {                                                             \
        cudaError_t e_ = cudaGetLastError();                         \
        if (e_ != cudaSuccess) return CSAHCA_ERR_CUDA;               \
    } while (0)

#define CSAHCA_REQUIRE(cond)                                         \
    do {                                                             \
        if (!(cond)) return CSAHCA_ERR_INVALID_ARG;                  \
    } while (0)

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
__host__ __device__ inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int num_sms();

// ------------------------------------------------------------- programmatic dependent launch
// Every kernel of the library is launched with programmatic stream serialization: its CTAs may
// be scheduled while the previous kernel in the stream is still running.  Each kernel therefore
// starts with pdl_wait() (returns once the previous grid has completed and its memory is
// visible; immediately when there is none) before it reads any global memory, then calls
// pdl_trigger() so that the next kernel may be scheduled in turn.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ------------------------------------------------------------------------- vector I/O
// 8 consecutive elements <-> float[8]; p must be 16-byte (bf16) / 32-byte (f32) aligned.
__device__ __forceinline__ void load8(const float* p, float (&o)[8]) {
    float4 a = __ldg(reinterpret_cast<const float4*>(p));
    float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&o)[8]) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[2 * i] = __uint_as_float(w[i] << 16);
        o[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}
// plain (non-__ldg) variant for buffers written earlier in the same kernel
__device__ __forceinline__ void load8_rw(const float* p, float (&o)[8]) {
    float4 a = *reinterpret_cast<const float4*>(p);
    float4 b = *(reinterpret_cast<const float4*>(p) + 1);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void load8_rw(const __nv_bfloat16* p, float (&o)[8]) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[2 * i] = __uint_as_float(w[i] << 16);
        o[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}
__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
    uint4 u;
    u.x = pack_bf16x2(v[0], v[1]);
    u.y = pack_bf16x2(v[2], v[3]);
    u.z = pack_bf16x2(v[4], v[5]);
    u.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8], int) { store8(p, v); }

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f32(float& d, float x) { d = x; }
__device__ __forceinline__ void from_f32(__nv_bfloat16& d, float x) { d = __float2bfloat16_rn(x); }

// --------------------------------------------------------------------------- warp utils
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Block-wide exclusive prefix sum of one value per thread (blockDim.x a multiple of 32,
// <= 1024).  `sh` must hold 33 ints.  Returns the exclusive prefix; *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* sh, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int s = (lane < nw) ? sh[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < nw) sh[lane] = s;          // inclusive per-warp totals
        if (lane == 31) sh[32] = s;
    }
    __syncthreads();
    int warp_base = (wid > 0) ? sh[wid - 1] : 0;
    int res = warp_base + x - v;
    *total = sh[32];
    __syncthreads();
    return res;
}

// Monotone map float32 -> uint32 (larger float -> larger key); -0 and +0 map to the same key.
__device__ __forceinline__ uint32_t ordered_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (f == 0.0f) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// --------------------------------------------------------------- internal launchers
// Tensor-core indexer scores (low-precision keys, bf16 queries, d_I = 64, Ncap % 8 == 0).
bool index_tc_supported(int q_dtype, int key_fmt, int H_I, int d_I, int64_t Ncap, const void* k_codes,
                        const void* k_scale, int B, int64_t R);
// cudaErrorNotSupported when the key tensor map cannot be built (the caller takes the generic path).
// hist1 (nullable): [B*T][4096] histogram of the top 12 bits of each visible score's ordered key.
cudaError_t index_tc_launch(const void* q_idx, const float* w, const void* k_codes, const void* k_scale, int key_fmt,
                            int B, int T, int H_I, const int64_t* q_pos, int64_t Ncap, int m, float* S,
                            uint32_t* hist1, unsigned* err, cudaStream_t st);

// Tensor-core indexer with FP4 queries (E2M1 codes + UE8M0 per 32, the keys' form) and e2m1 keys.
cudaError_t index_tc_q4_launch(const void* q_codes, const void* q_scale, const float* w, const void* k_codes,
                               const void* k_scale, int B, int T, int H_I, const int64_t* q_pos, int64_t Ncap, int m,
                               float* S, uint32_t* hist1, unsigned* err, cudaStream_t st);
// Tensor-core indexer scores for chunked prefill (bf16 keys and queries, d_I = 64, T a multiple of
// 128 / H_I); scores only (the top-k forms its first histogram in a pass of its own).
bool index_prefill_supported(int q_dtype, int key_fmt, int H_I, int d_I, int64_t Ncap, const void* q_idx,
                             const void* k_codes, int B, int T);
cudaError_t index_prefill_launch(const void* q_idx, const float* w, const void* k_codes, int B, int T, int H_I,
                                 const int64_t* q_pos, int64_t Ncap, int m, float* S, unsigned* err, cudaStream_t st);

// Top-k over float32 scores (rows of `stride`, n_vis per row from q_pos or n_vis arrays).
struct TopkWorkspace {
    uint32_t* hist1;   // [R][4096] histogram of the top 12 bits (zeroed before it is accumulated)
    uint32_t* win;     // [R][words] bitmap of entries above the threshold (rows too long for
    uint32_t* tie;     // [R][words] bitmap of entries equal to it          shared memory)
    int64_t words;
};
size_t topk_workspace_bytes(int64_t R, int64_t stride);
TopkWorkspace topk_carve(void* ws, int64_t R, int64_t stride);
// n_vis for row r is either n_vis_arr[r] (if non-NULL) or min(Ncap, (q_pos[r]+1)/m).
// hist_ready: hist1 was filled by the caller (the fused indexer); else a histogram pass fills it
// (hist1 is zero on entry either way: the workspace starts zero-filled and every call clears
// the rows it used).
csahca_status topk_launch(const float* scores, int64_t stride, int R, const int64_t* n_vis_arr,
                          const int64_t* q_pos, int m, int64_t Ncap, int k, int32_t* idx_out,
                          const TopkWorkspace& tw, bool hist_ready, cudaStream_t stream);

}  // namespace csahca
