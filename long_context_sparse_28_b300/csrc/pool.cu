// a1/a2 softmax-gated pooling (bulk compress) and a3 cache append / ring write.
//
// Pooling (pogovet.com DeepSeek-V4 article, detail 4; honbul.tistory.com/221 "CSA", "HCA"):
//   alpha_i = softmax_i(gate[j*m+i] + bias[i]);  C[j] = sum_i alpha_i X[j*m+i]  (X = K and V).
// One warp pools one block: lanes compute the m softmax weights cooperatively, then each lane
// owns 8 consecutive channels of K or V (16-byte loads for bf16) and walks the m tokens in
// order, accumulating in fp32.  HBM-bound: the raw K/V are read once, the entries written once.
//
// Cache append (honbul.tistory.com/221 "KV cache를 줄이는 방식"): recent raw tokens live in a
// ring (the window cache), which also holds the tail of the block being filled; a block is
// pooled into the compressed cache the moment its last token arrives.
#include "common.cuh"
#include "quant.cuh"

namespace csahca {
namespace {

constexpr int kMaxM = 256;

// Stores that ask L2 to keep the line (evict-last): the window ring is small and read again by the
// attention of every step and by the pooling of the next block, while a step streams hundreds of
// megabytes of caches through L2.
__device__ __forceinline__ uint64_t keep_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void st_keep(void* ptr, uint4 u, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(ptr), "r"(u.x), "r"(u.y), "r"(u.z),
                 "r"(u.w), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void store8_keep(__nv_bfloat16* p, const float (&v)[8], uint64_t pol) {
    st_keep(p, make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                          pack_bf16x2(v[6], v[7])),
            pol);
}
__device__ __forceinline__ void store8_keep(float* p, const float (&v)[8], uint64_t pol) {
    st_keep(p, make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3])),
            pol);
    st_keep(p + 4, make_uint4(__float_as_uint(v[4]), __float_as_uint(v[5]), __float_as_uint(v[6]), __float_as_uint(v[7])),
            pol);
}
__device__ __forceinline__ void st_keep_f32(float* ptr, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(ptr), "r"(__float_as_uint(v)), "l"(pol) : "memory");
}

// Softmax weights of one block, distributed over the warp: lane holds alpha of slots
// lane + 32*r (r < 8).  `zsrc(i)` returns gate_i + bias_i.
template <typename Z>
__device__ __forceinline__ void block_weights(int m, Z zsrc, float (&a)[8]) {
    const int lane = threadIdx.x & 31;
    float zmax = -INFINITY;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int i = lane + 32 * r;
        a[r] = (i < m) ? zsrc(i) : -INFINITY;
        zmax = fmaxf(zmax, a[r]);
    }
    zmax = warp_max(zmax);
    float zs = 0.0f;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int i = lane + 32 * r;
        a[r] = (i < m) ? expf(a[r] - zmax) : 0.0f;
        zs += a[r];
    }
    zs = warp_sum(zs);
#pragma unroll
    for (int r = 0; r < 8; ++r) a[r] = a[r] / zs;
}

__device__ __forceinline__ float alpha_of(const float (&a)[8], int i) {
    float v = 0.0f;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const float t = __shfl_sync(0xffffffffu, a[r], i & 31);
        if ((i >> 5) == r) v = t;
    }
    return v;
}

// Pool one block with one warp.  rowptr(which, i) -> pointer to token i's row of K (which=0)
// or V (which=1).  Writes ck_row / cv_row: rows of T, or (kKv8, d = 128: one pass, every lane
// active) the entry's FP8 K and V rows.
template <typename T, bool kKv8, typename RowPtr>
__device__ __forceinline__ void pool_block_warp(int m, int d, const float (&a)[8], RowPtr rowptr,
                                                void* ck_row, void* cv_row) {
    const int lane = threadIdx.x & 31;
    const int groups = d / 8;                 // 8-channel groups per tensor
    for (int g0 = 0; g0 < 2 * groups; g0 += 32) {
        const int g = g0 + lane;
        const bool active = g < 2 * groups;
        const int which = (g < groups) ? 0 : 1;
        const int col = (g % groups) * 8;
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int i = 0; i < m; ++i) {
            // warp-uniform loop: all lanes shuffle (one shuffle when every weight is in a[0])
            const float al = m <= 32 ? __shfl_sync(0xffffffffu, a[0], i) : alpha_of(a, i);
            if (active) {
                float x[8];
                load8_rw(rowptr(which, i) + col, x);
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[c] = fmaf(al, x[c], acc[c]);
            }
        }
        if constexpr (kKv8)
            store_kv8_warp(acc, static_cast<unsigned char*>(ck_row), static_cast<unsigned char*>(cv_row), lane);
        else if (active)
            store8(static_cast<T*>(which ? cv_row : ck_row) + col, acc);
    }
}

template <typename T, bool kKv8>
__global__ void compress_kernel(const T* __restrict__ k_raw, const T* __restrict__ v_raw,
                                const float* __restrict__ gate, int64_t raw_stride,
                                const int64_t* __restrict__ raw_pos0, const int64_t* __restrict__ n_raw,
                                const float* __restrict__ bias, int m, int B, int d, void* ck, void* cv,
                                int64_t Ncap, int64_t max_blocks, unsigned* err) {
    pdl_wait();
    pdl_trigger();
    const int wpc = blockDim.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t total = (int64_t)B * max_blocks;
    for (int64_t wid = (int64_t)blockIdx.x * wpc + (threadIdx.x >> 5); wid < total;
         wid += (int64_t)gridDim.x * wpc) {
        const int b = (int)(wid / max_blocks);
        const int64_t jl = wid % max_blocks;
        const int64_t p0 = raw_pos0[b], n = n_raw[b];
        const int64_t j = (p0 + m - 1) / m + jl;          // first block fully inside + jl
        if ((j + 1) * m > p0 + n) continue;
        if (j >= Ncap || (j + 1) * m - p0 > raw_stride || p0 < 0) {
            if (lane == 0) flag_error(err, ERRBIT_BOUNDS);
            continue;
        }
        const int64_t row0 = (int64_t)b * raw_stride + (j * m - p0);
        const float* g = gate + row0;
        float a[8];
        block_weights(m, [&](int i) { return g[i] + bias[i]; }, a);
        auto rowptr = [&](int which, int i) -> const T* {
            return (which ? v_raw : k_raw) + (row0 + i) * (int64_t)d;
        };
        const int64_t e = (int64_t)b * Ncap + j;
        if constexpr (kKv8)
            pool_block_warp<T, true>(m, d, a, rowptr, static_cast<unsigned char*>(ck) + e * kKv8KRow,
                                     static_cast<unsigned char*>(cv) + e * kKv8VRow);
        else
            pool_block_warp<T, false>(m, d, a, rowptr, static_cast<T*>(ck) + e * d, static_cast<T*>(cv) + e * d);
    }
}

// Large blocks (m >= 64) with one CTA of four warps per block: warp q sums tokens
// [q m / 4, (q + 1) m / 4) of every channel group (the same per-token weights), the partial sums
// meet in shared memory and warp 0 adds them in quarter order and stores the entry.  Four times
// the loads in flight of the one-warp form, for the few large blocks of a prefill chunk.
template <typename T, bool kKv8>
__global__ void __launch_bounds__(128) compress_split_kernel(
    const T* __restrict__ k_raw, const T* __restrict__ v_raw, const float* __restrict__ gate, int64_t raw_stride,
    const int64_t* __restrict__ raw_pos0, const int64_t* __restrict__ n_raw, const float* __restrict__ bias, int m,
    int B, int d, void* ck, void* cv, int64_t Ncap, int64_t max_blocks, unsigned* err) {
    pdl_wait();
    pdl_trigger();
    __shared__ float part[4][4][32][8];       // [quarter][channel-group pass (d <= 512)][lane][channel]
    const int q = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int groups = d / 8;                 // 8-channel groups per tensor
    const int64_t total = (int64_t)B * max_blocks;
    for (int64_t bid = blockIdx.x; bid < total; bid += gridDim.x) {
        const int b = (int)(bid / max_blocks);
        const int64_t jl = bid % max_blocks;
        const int64_t p0 = raw_pos0[b], n = n_raw[b];
        const int64_t j = (p0 + m - 1) / m + jl;          // first block fully inside + jl
        if ((j + 1) * m > p0 + n) continue;
        if (j >= Ncap || (j + 1) * m - p0 > raw_stride || p0 < 0) {
            if (threadIdx.x == 0) flag_error(err, ERRBIT_BOUNDS);
            continue;
        }
        const int64_t row0 = (int64_t)b * raw_stride + (j * m - p0);
        const float* g = gate + row0;
        float a[8];
        block_weights(m, [&](int i) { return g[i] + bias[i]; }, a);
        const int i0 = q * m / 4, i1 = (q + 1) * m / 4;
        for (int g0 = 0, it = 0; g0 < 2 * groups; g0 += 32, ++it) {
            const int gi = g0 + lane;
            const bool active = gi < 2 * groups;
            const T* base = (gi < groups ? k_raw : v_raw) + (gi % groups) * 8;
            float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            for (int i = i0; i < i1; ++i) {
                const float al = alpha_of(a, i);  // warp-uniform loop: all lanes shuffle
                if (active) {
                    float x[8];
                    load8_rw(base + (row0 + i) * (int64_t)d, x);
#pragma unroll
                    for (int c = 0; c < 8; ++c) acc[c] = fmaf(al, x[c], acc[c]);
                }
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) part[q][it][lane][c] = acc[c];
        }
        __syncthreads();
        if (q == 0) {
            const int64_t e = (int64_t)b * Ncap + j;
            for (int g0 = 0, it = 0; g0 < 2 * groups; g0 += 32, ++it) {
                const int gi = g0 + lane;
                float acc[8];
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    acc[c] = ((part[0][it][lane][c] + part[1][it][lane][c]) + part[2][it][lane][c]) +
                             part[3][it][lane][c];
                if constexpr (kKv8) {
                    store_kv8_warp(acc, static_cast<unsigned char*>(ck) + e * kKv8KRow,
                                   static_cast<unsigned char*>(cv) + e * kKv8VRow, lane);
                } else if (gi < 2 * groups) {
                    T* dst = static_cast<T*>(gi < groups ? ck : cv) + e * d + (gi % groups) * 8;
                    store8(dst, acc);
                }
            }
        }
        __syncthreads();                      // the partial sums are reused by the next block
    }
}

// One CTA per sequence: pool completed blocks (reading old tokens from the ring), then write
// the new tokens into the ring.  A completed block is pooled by the whole CTA: warp 0 computes
// the m softmax weights into shared memory, then every thread sums a subset of the m tokens for
// 8 channels of K or V, and the partial sums are added in a fixed order.  Loads that do not need
// the weights -- a thread's tokens when its subset has at most 4, the block's index-key row
// (warp 1) -- are issued before the weights' barrier, so a decode step's block costs about one
// memory round trip after the position is known.  Ring slots are computed with 32-bit arithmetic
// from one 64-bit remainder per block (ring_cap >= m - 1, so one conditional subtraction).
constexpr int kAppendThreads = 256;

template <typename T, bool kKv8>
__global__ void __launch_bounds__(kAppendThreads) append_kernel(
    const T* __restrict__ k_new, const T* __restrict__ v_new, const float* __restrict__ gate_new,
    const void* kidx_new, int kidx_dtype, int kidx_rows, const int64_t* __restrict__ pos, int n_new, int d,
    const float* __restrict__ bias, int m, T* ring_k, T* ring_v, float* ring_gate, int ring_cap, void* ck, void* cv,
    int64_t Ncap, void* k_codes, void* k_scale, int key_fmt, int d_I, unsigned* err) {
    pdl_wait();
    pdl_trigger();
    __shared__ float alpha[kMaxM];
    __shared__ float part[kAppendThreads * 8];
    const int b = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // the new tokens bound for the ring: loaded first (they do not depend on the position) when
    // one pass of the block covers them (a decode step's token), stored at the end
    const int first = n_new > ring_cap ? n_new - ring_cap : 0;
    const int vec = d / 8;
    const int items = (n_new - first) * vec;
    const bool pre = items <= kAppendThreads;
    float yk[8], yv[8], yg = 0.0f;
    if (pre && tid < items) {
        const int i = first + tid / vec, c = (tid % vec) * 8;
        load8_rw(k_new + ((int64_t)b * n_new + i) * d + c, yk);
        load8_rw(v_new + ((int64_t)b * n_new + i) * d + c, yv);
        if (c == 0) yg = gate_new[(int64_t)b * n_new + i];
    }
    // warp 0, for blocks of m <= 32 tokens: the sequence's ring gates (4 slots per lane) and the slot
    // biases, also loaded before the position is known
    const bool small_m = m <= 32 && ring_cap <= 128;
    float rg4[4] = {0.f, 0.f, 0.f, 0.f}, bz = 0.0f;
    if (warp == 0 && small_m) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (lane * 4 + c < ring_cap) rg4[c] = ring_gate[(int64_t)b * ring_cap + lane * 4 + c];
        if (lane < m) bz = bias[lane];
    }
    const int64_t p = pos[b];
    if (p < 0) {
        if (tid == 0) flag_error(err, ERRBIT_BOUNDS);
        return;
    }
    // completed blocks: [j_lo, j_hi) (shifts when m is a power of two)
    const bool pow2 = (m & (m - 1)) == 0;
    const int msh = __ffs(m) - 1;
    const int64_t j_lo = pow2 ? (p >> msh) : p / m, j_hi = pow2 ? ((p + n_new) >> msh) : (p + n_new) / m;
    const T* kn = k_new + (int64_t)b * n_new * d;
    const T* vn = v_new + (int64_t)b * n_new * d;
    const float* gn = gate_new + (int64_t)b * n_new;
    const T* rk = ring_k + (int64_t)b * ring_cap * d;
    const T* rv = ring_v + (int64_t)b * ring_cap * d;
    const float* rg = ring_gate + (int64_t)b * ring_cap;
    const int G = 2 * d / 8;                               // 8-channel groups of K then V
    const int NS = G >= kAppendThreads ? 1 : kAppendThreads / G;   // token subsets
    const int per = (m + NS - 1) / NS;
    const int g = tid % G, ts = tid / G;
    const int which = (g < G / 2) ? 0 : 1;
    const int col = (g % (G / 2)) * 8;
    const int i0 = ts * per, i1 = min(m, i0 + per);
    for (int64_t j = j_lo; j < j_hi; ++j) {
        if (j >= Ncap) {
            if (tid == 0) flag_error(err, ERRBIT_BOUNDS);
            continue;
        }
        const int64_t t0 = j * m;
        const int t0r = (int)(t0 % ring_cap);
        // row of token t0 + i of K (which = 0) or V: new tokens from the input, older ones from the ring
        auto tok = [&](int i, int wh) -> const T* {
            const int64_t t = t0 + i;
            if (t >= p) return (wh ? vn : kn) + (t - p) * d;
            int sl = t0r + i;
            if (sl >= ring_cap) sl -= ring_cap;
            return (wh ? rv : rk) + (int64_t)sl * d;
        };
        // loads independent of the weights first
        float x[4][8];
        const int nx = (ts < NS && per <= 4) ? i1 - i0 : 0;
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (u < nx) load8_rw(tok(i0 + u, which) + col, x[u]);
        float kx[8];
        const bool quant = k_codes != nullptr && warp == 1;
        if (quant) {
            const int r = (int)(j - j_lo);
            const int64_t in_bytes = (kidx_dtype == CSAHCA_F32 ? 4 : 2);
            const char* row = static_cast<const char*>(kidx_new) + (((int64_t)b * kidx_rows + r) * d_I) * in_bytes;
            load_row_slice(row, kidx_dtype, d_I / 32, kx);
        }
        if (warp == 0 && small_m) {
            // lane i < m: slot i's logit, the ring's gate taken from the preloaded registers
            const int64_t t = t0 + lane;
            int sl = t0r + (lane < m ? lane : 0);
            if (sl >= ring_cap) sl -= ring_cap;
            float g = 0.0f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float x = __shfl_sync(0xffffffffu, rg4[c], sl >> 2);
                if ((sl & 3) == c) g = x;
            }
            if (lane < m && t >= p) g = gn[t - p];
            const float z = lane < m ? g + bz : -INFINITY;
            const float zmax = warp_max(z);
            const float e = lane < m ? expf(z - zmax) : 0.0f;
            const float zs = warp_sum(e);
            if (lane < m) alpha[lane] = e / zs;
        } else if (warp == 0) {
            float a[8];
            block_weights(m, [&](int i) {
                const int64_t t = t0 + i;
                int sl = t0r + i;
                if (sl >= ring_cap) sl -= ring_cap;
                return ((t >= p) ? gn[t - p] : rg[sl]) + bias[i];
            }, a);
#pragma unroll
            for (int r = 0; r < 8; ++r)
                if (lane + 32 * r < m) alpha[lane + 32 * r] = a[r];
        }
        __syncthreads();
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (ts < NS) {
            if (per <= 4) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (u < nx)
#pragma unroll
                        for (int c = 0; c < 8; ++c) acc[c] = fmaf(alpha[i0 + u], x[u][c], acc[c]);
            } else {
                int i = i0;
                for (; i + 4 <= i1; i += 4) {
                    float y[4][8];
#pragma unroll
                    for (int u = 0; u < 4; ++u) load8_rw(tok(i + u, which) + col, y[u]);
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int c = 0; c < 8; ++c) acc[c] = fmaf(alpha[i + u], y[u][c], acc[c]);
                }
                for (; i < i1; ++i) {
                    float y[8];
                    load8_rw(tok(i, which) + col, y);
#pragma unroll
                    for (int c = 0; c < 8; ++c) acc[c] = fmaf(alpha[i], y[c], acc[c]);
                }
            }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) part[tid * 8 + c] = acc[c];
        __syncthreads();
        if (tid < G) {                                      // subsets added in order 0..NS-1
            float o[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            for (int q = 0; q < NS; ++q)
#pragma unroll
                for (int c = 0; c < 8; ++c) o[c] += part[(q * G + tid) * 8 + c];
            const int64_t e = (int64_t)b * Ncap + j;
            if constexpr (kKv8) {                           // d = 128: G = 32, warp 0
                store_kv8_warp(o, static_cast<unsigned char*>(ck) + e * kKv8KRow,
                               static_cast<unsigned char*>(cv) + e * kKv8VRow, lane);
            } else {
                const int wh = (tid < G / 2) ? 0 : 1;
                const int cl = (tid % (G / 2)) * 8;
                store8(static_cast<T*>(wh ? cv : ck) + e * d + cl, o);
            }
        }
        if (quant) {
            const int E = d_I / 32;
            const int64_t er = (int64_t)b * Ncap + j;
            quantize_row_warp(kx, E, d_I, key_fmt, static_cast<char*>(k_codes) + er * key_row_bytes(key_fmt, d_I),
                              k_scale ? static_cast<char*>(k_scale) + er * key_scale_bytes(key_fmt, d_I) : nullptr);
        }
        __syncthreads();
    }
    // write the last min(n_new, ring_cap) tokens into the ring (32-bit indices: the host checks
    // that n_new * d / 8 fits)
    T* wk = ring_k + (int64_t)b * ring_cap * d;
    T* wv = ring_v + (int64_t)b * ring_cap * d;
    const int base = (int)(p % ring_cap);
    if (pre) {
        if (tid < items) {
            const uint64_t pol = keep_policy();
            const int i = first + tid / vec, c = (tid % vec) * 8;
            const int64_t slot = (base + i) % ring_cap;
            store8_keep(wk + slot * d + c, yk, pol);
            store8_keep(wv + slot * d + c, yv, pol);
            if (c == 0) st_keep_f32(ring_gate + (int64_t)b * ring_cap + slot, yg, pol);
        }
        return;
    }
    for (int it = tid; it < items; it += blockDim.x) {
        const int i = first + it / vec;
        const int c = (it % vec) * 8;
        const int64_t slot = (base + i) % ring_cap;
        float y[8];
        load8_rw(kn + (int64_t)i * d + c, y);
        store8(wk + slot * d + c, y);
        load8_rw(vn + (int64_t)i * d + c, y);
        store8(wv + slot * d + c, y);
    }
    for (int i = first + tid; i < n_new; i += blockDim.x)
        ring_gate[(int64_t)b * ring_cap + (base + i) % ring_cap] = gn[i];
}

template <typename T>
__global__ void ring_write_kernel(const T* __restrict__ k_new, const T* __restrict__ v_new,
                                  const float* __restrict__ gate_new, int64_t new_stride,
                                  const int64_t* __restrict__ pos, int n_new, int d, T* ring_k,
                                  T* ring_v, float* ring_gate, int ring_cap) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.y;
    const int64_t p = pos[b];
    if (p < 0) return;                     // no valid slot for a negative position
    const int first = n_new > ring_cap ? n_new - ring_cap : 0;
    const int vec = d / 8;
    const int64_t items = (int64_t)(n_new - first) * vec;
    for (int64_t it = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; it < items;
         it += (int64_t)gridDim.x * blockDim.x) {
        const int i = first + (int)(it / vec);
        const int c = (int)(it % vec) * 8;
        const int64_t slot = (p + i) % ring_cap;
        float x[8];
        load8(k_new + ((int64_t)b * new_stride + i) * d + c, x);
        store8(ring_k + ((int64_t)b * ring_cap + slot) * d + c, x);
        load8(v_new + ((int64_t)b * new_stride + i) * d + c, x);
        store8(ring_v + ((int64_t)b * ring_cap + slot) * d + c, x);
        if (c == 0) ring_gate[(int64_t)b * ring_cap + slot] = gate_new[(int64_t)b * new_stride + i];
    }
}

bool kv_dtype_ok(csahca_dtype t) { return t == CSAHCA_F32 || t == CSAHCA_BF16 || t == CSAHCA_KV_FP8; }

csahca_status compress_impl(const void* k_raw, const void* v_raw, const float* gate, int64_t raw_stride,
                            const int64_t* raw_pos0, const int64_t* n_raw, const float* bias, int m,
                            int B, int d, csahca_dtype kv, void* ck, void* cv, int64_t Ncap,
                            cudaStream_t stream) {
    CSAHCA_REQUIRE(k_raw && v_raw && gate && raw_pos0 && n_raw && bias && ck && cv);
    CSAHCA_REQUIRE(m >= 1 && m <= kMaxM && B >= 1 && d >= 8 && d <= 512 && d % 8 == 0);
    CSAHCA_REQUIRE(raw_stride >= 0 && Ncap >= 0);
    CSAHCA_REQUIRE(kv_dtype_ok(kv));
    if (kv == CSAHCA_KV_FP8) CSAHCA_REQUIRE(d == 128);
    const size_t al = (kv == CSAHCA_F32) ? 32 : 16;
    CSAHCA_REQUIRE(aligned(k_raw, al) && aligned(v_raw, al) && aligned(ck, al) && aligned(cv, al));
    const int64_t max_blocks = raw_stride / m + 1;
    const int64_t warps = (int64_t)B * max_blocks;
    if (warps == 0 || Ncap == 0 || raw_stride == 0) return CSAHCA_OK;
    unsigned* err = err_word();
    if (!err) return CSAHCA_ERR_CUDA;
    if (m >= 64) {                            // four warps per block
        const int grid = (int)std::min<int64_t>(warps, (int64_t)num_sms() * 16);
        if (kv == CSAHCA_F32)
            (void)launch_pdl(compress_split_kernel<float, false>, dim3(grid), dim3(128), 0, stream,
                (const float*)k_raw, (const float*)v_raw, gate, raw_stride, raw_pos0, n_raw, bias, m, B, d,
                ck, cv, Ncap, max_blocks, err);
        else if (kv == CSAHCA_BF16)
            (void)launch_pdl(compress_split_kernel<__nv_bfloat16, false>, dim3(grid), dim3(128), 0, stream,
                (const __nv_bfloat16*)k_raw, (const __nv_bfloat16*)v_raw, gate, raw_stride, raw_pos0, n_raw,
                bias, m, B, d, ck, cv, Ncap, max_blocks, err);
        else
            (void)launch_pdl(compress_split_kernel<__nv_bfloat16, true>, dim3(grid), dim3(128), 0, stream,
                (const __nv_bfloat16*)k_raw, (const __nv_bfloat16*)v_raw, gate, raw_stride, raw_pos0, n_raw,
                bias, m, B, d, ck, cv, Ncap, max_blocks, err);
        count_launch();
        CSAHCA_CHECK_LAUNCH();
        return CSAHCA_OK;
    }
    const int threads = 256;
    const int64_t want = cdiv(warps, threads / 32);
    const int grid = (int)std::min<int64_t>(want, (int64_t)num_sms() * 16);
    if (kv == CSAHCA_F32)
        (void)launch_pdl(compress_kernel<float, false>, dim3(grid), dim3(threads), 0, stream,
            (const float*)k_raw, (const float*)v_raw, gate, raw_stride, raw_pos0, n_raw, bias, m, B, d,
            ck, cv, Ncap, max_blocks, err);
    else if (kv == CSAHCA_BF16)
        (void)launch_pdl(compress_kernel<__nv_bfloat16, false>, dim3(grid), dim3(threads), 0, stream,
            (const __nv_bfloat16*)k_raw, (const __nv_bfloat16*)v_raw, gate, raw_stride, raw_pos0, n_raw,
            bias, m, B, d, ck, cv, Ncap, max_blocks, err);
    else
        (void)launch_pdl(compress_kernel<__nv_bfloat16, true>, dim3(grid), dim3(threads), 0, stream,
            (const __nv_bfloat16*)k_raw, (const __nv_bfloat16*)v_raw, gate, raw_stride, raw_pos0, n_raw,
            bias, m, B, d, ck, cv, Ncap, max_blocks, err);
    count_launch();
    CSAHCA_CHECK_LAUNCH();
    return CSAHCA_OK;
}

csahca_status append_impl(const void* k_new, const void* v_new, const float* gate_new, const void* kidx_new,
                          csahca_dtype kidx_dtype, const int64_t* pos, int B, int n_new, int d,
                          csahca_dtype kv, const float* bias, int m, void* ring_k, void* ring_v,
                          float* ring_gate, int ring_cap, void* ck, void* cv, int64_t Ncap, void* k_codes,
                          void* k_scale, csahca_dtype key_fmt, int d_I, cudaStream_t stream) {
    CSAHCA_REQUIRE(k_new && v_new && gate_new && pos && bias && ring_k && ring_v && ring_gate && ck && cv);
    CSAHCA_REQUIRE(m >= 1 && m <= kMaxM && B >= 1 && n_new >= 0 && d >= 8 && d <= 512 && d % 8 == 0);
    CSAHCA_REQUIRE((int64_t)n_new * (d / 8) < (1LL << 30) && (int64_t)n_new + ring_cap < (1LL << 30));
    CSAHCA_REQUIRE(ring_cap >= 1 && ring_cap >= m - 1 && Ncap >= 0);
    CSAHCA_REQUIRE(kv_dtype_ok(kv));
    if (kv == CSAHCA_KV_FP8) CSAHCA_REQUIRE(d == 128);
    const size_t al = (kv == CSAHCA_F32) ? 32 : 16;
    CSAHCA_REQUIRE(aligned(k_new, al) && aligned(v_new, al) && aligned(ring_k, al) && aligned(ring_v, al) &&
                   aligned(ck, al) && aligned(cv, al));
    if (k_codes) {
        CSAHCA_REQUIRE(kidx_new && (kidx_dtype == CSAHCA_F32 || kidx_dtype == CSAHCA_BF16));
        CSAHCA_REQUIRE(d_I >= 32 && d_I <= 256 && d_I % 32 == 0);
        CSAHCA_REQUIRE(key_fmt >= CSAHCA_F32 && key_fmt <= CSAHCA_E2M1_UE8M0);
        if (key_fmt == CSAHCA_E2M1_UE8M0) CSAHCA_REQUIRE(d_I % 64 == 0);
        if (key_fmt >= CSAHCA_E4M3_ROWSCALE) CSAHCA_REQUIRE(k_scale != nullptr);
    }
    if (n_new == 0) return CSAHCA_OK;
    unsigned* err = err_word();
    if (!err) return CSAHCA_ERR_CUDA;
    const int kidx_rows = n_new / m + 1;
    if (kv == CSAHCA_F32)
        (void)launch_pdl(append_kernel<float, false>, dim3(B), dim3(kAppendThreads), 0, stream,
            (const float*)k_new, (const float*)v_new, gate_new, kidx_new, kidx_dtype, kidx_rows, pos, n_new, d,
            bias, m, (float*)ring_k, (float*)ring_v, ring_gate, ring_cap, ck, cv, Ncap, k_codes,
            k_scale, key_fmt, d_I, err);
    else if (kv == CSAHCA_BF16)
        (void)launch_pdl(append_kernel<__nv_bfloat16, false>, dim3(B), dim3(kAppendThreads), 0, stream,
            (const __nv_bfloat16*)k_new, (const __nv_bfloat16*)v_new, gate_new, kidx_new, kidx_dtype, kidx_rows,
            pos, n_new, d, bias, m, (__nv_bfloat16*)ring_k, (__nv_bfloat16*)ring_v, ring_gate, ring_cap,
            ck, cv, Ncap, k_codes, k_scale, key_fmt, d_I, err);
    else
        (void)launch_pdl(append_kernel<__nv_bfloat16, true>, dim3(B), dim3(kAppendThreads), 0, stream,
            (const __nv_bfloat16*)k_new, (const __nv_bfloat16*)v_new, gate_new, kidx_new, kidx_dtype, kidx_rows,
            pos, n_new, d, bias, m, (__nv_bfloat16*)ring_k, (__nv_bfloat16*)ring_v, ring_gate, ring_cap,
            ck, cv, Ncap, k_codes, k_scale, key_fmt, d_I, err);
    count_launch();
    CSAHCA_CHECK_LAUNCH();
    return CSAHCA_OK;
}

}  // namespace
}  // namespace csahca

using namespace csahca;

extern "C" {

csahca_status csa_compress(const void* k_raw, const void* v_raw, const float* gate, int64_t raw_stride,
                           const int64_t* raw_pos0, const int64_t* n_raw, const float* slot_bias, int m,
                           int B, int d, csahca_dtype kv_dtype, void* ck, void* cv, int64_t Ncap,
                           csahca_stream_t stream) {
    return compress_impl(k_raw, v_raw, gate, raw_stride, raw_pos0, n_raw, slot_bias, m, B, d, kv_dtype, ck, cv,
                         Ncap, (cudaStream_t)stream);
}

csahca_status hca_compress(const void* k_raw, const void* v_raw, const float* gate, int64_t raw_stride,
                           const int64_t* raw_pos0, const int64_t* n_raw, const float* slot_bias, int m,
                           int B, int d, csahca_dtype kv_dtype, void* ck, void* cv, int64_t Ncap,
                           csahca_stream_t stream) {
    return compress_impl(k_raw, v_raw, gate, raw_stride, raw_pos0, n_raw, slot_bias, m, B, d, kv_dtype, ck, cv,
                         Ncap, (cudaStream_t)stream);
}

csahca_status csa_cache_append(const void* k_new, const void* v_new, const float* gate_new, const void* kidx_new,
                               csahca_dtype kidx_dtype, const int64_t* pos, int B, int n_new, int d,
                               csahca_dtype kv_dtype, const float* slot_bias, int m, void* ring_k, void* ring_v,
                               float* ring_gate, int ring_cap, void* ck, void* cv, int64_t Ncap, void* k_codes,
                               void* k_scale, csahca_dtype key_fmt, int d_I, csahca_stream_t stream) {
    if (!k_codes) return CSAHCA_ERR_INVALID_ARG;
    return append_impl(k_new, v_new, gate_new, kidx_new, kidx_dtype, pos, B, n_new, d, kv_dtype, slot_bias, m,
                       ring_k, ring_v, ring_gate, ring_cap, ck, cv, Ncap, k_codes, k_scale, key_fmt, d_I,
                       (cudaStream_t)stream);
}

csahca_status hca_cache_append(const void* k_new, const void* v_new, const float* gate_new, const int64_t* pos,
                               int B, int n_new, int d, csahca_dtype kv_dtype, const float* slot_bias, int m,
                               void* ring_k, void* ring_v, float* ring_gate, int ring_cap, void* ck, void* cv,
                               int64_t Ncap, csahca_stream_t stream) {
    return append_impl(k_new, v_new, gate_new, nullptr, CSAHCA_BF16, pos, B, n_new, d, kv_dtype, slot_bias, m,
                       ring_k, ring_v, ring_gate, ring_cap, ck, cv, Ncap, nullptr, nullptr, CSAHCA_BF16, 0,
                       (cudaStream_t)stream);
}

csahca_status swa_ring_write(const void* k_new, const void* v_new, const float* gate_new, int64_t new_stride,
                             const int64_t* pos, int B, int n_new, int d, csahca_dtype kv_dtype, void* ring_k,
                             void* ring_v, float* ring_gate, int ring_cap, csahca_stream_t stream) {
    CSAHCA_REQUIRE(k_new && v_new && gate_new && pos && ring_k && ring_v && ring_gate);
    CSAHCA_REQUIRE(B >= 1 && n_new >= 0 && new_stride >= n_new && d >= 8 && d <= 512 && d % 8 == 0 && ring_cap >= 1);
    CSAHCA_REQUIRE(kv_dtype_ok(kv_dtype));
    const size_t al = (kv_dtype == CSAHCA_F32) ? 32 : 16;
    CSAHCA_REQUIRE(aligned(k_new, al) && aligned(v_new, al) && aligned(ring_k, al) && aligned(ring_v, al));
    if (n_new == 0) return CSAHCA_OK;
    const int first = n_new > ring_cap ? n_new - ring_cap : 0;
    const int64_t items = (int64_t)(n_new - first) * (d / 8);
    dim3 grid((unsigned)std::max<int64_t>(1, std::min<int64_t>(cdiv(items, 256), 64)), B);
    if (kv_dtype == CSAHCA_F32)
        (void)launch_pdl(ring_write_kernel<float>, dim3(grid), dim3(256), 0, (cudaStream_t)stream, 
            (const float*)k_new, (const float*)v_new, gate_new, new_stride, pos, n_new, d, (float*)ring_k,
            (float*)ring_v, ring_gate, ring_cap);
    else
        (void)launch_pdl(ring_write_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, (cudaStream_t)stream, 
            (const __nv_bfloat16*)k_new, (const __nv_bfloat16*)v_new, gate_new, new_stride, pos, n_new, d,
            (__nv_bfloat16*)ring_k, (__nv_bfloat16*)ring_v, ring_gate, ring_cap);
    count_launch();
    CSAHCA_CHECK_LAUNCH();
    return CSAHCA_OK;
}

}  // extern "C"
