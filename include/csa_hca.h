/*
 * csa_hca.h -- C ABI of the B300 (sm_103a) hybrid compressed attention library
 * (libcsahca.so): CSA (compressed sparse attention, m = 4) and HCA (heavily compressed
 * attention, m = 128), decode and chunked prefill.
 *
 * The method (DeepSeek-V4 summary pages):
 *   honbul.tistory.com/221, section "CSA: 압축한 뒤, 필요한 기억만 골라서 보기" -- several tokens
 *     are compressed into one KV entry, a small indexer finds the blocks related to the
 *     current token, only the top candidates enter attention, and recent tokens are kept
 *     in a separate sliding window;
 *   same page, section "HCA: 더 강하게 압축하고, 압축된 전체를 보기" -- stronger compression,
 *     no sparse selection, attention over every compressed entry;
 *   same page, section "KV cache를 줄이는 방식" -- a compressed KV cache, a cache of recent
 *     tokens for the window, and the tail state of tokens that do not yet fill a block,
 *     kept apart (not a paged layout);
 *   pogovet.com "DeepSeek-V4: a million-token context that agents can actually use",
 *     detail 4 -- CSA pools 4 KV entries into one with softmax-gated pooling that has a
 *     learned position bias, an FP4 lightning indexer picks the top-k compressed blocks
 *     per query, plus a sliding-window branch; HCA pools 128 entries and attends densely
 *     over all compressed blocks; detail 5 -- the indexer runs in FP4.
 *
 * Conventions (all entry points):
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless stated.  The
 *     library never frees, retains or allocates memory; scratch space is a caller-provided
 *     workspace sized by the matching *_workspace() function (256-byte aligned).  The one
 *     exception is hca_attend_noalloc, whose scratch is a fixed array inside the library.
 *   - The workspaces of csa_index_topk, csa_index_topk_fp4, csa_attend and hca_attend carry
 *     state between calls: zero-fill a workspace once after allocating it.  Every call leaves
 *     its state area zero again (per-row histograms that the top-k clears after reading them,
 *     per-row arrival counters that the row's last CTA resets), so no call spends a launch on
 *     clearing it.  Zero it again after a call that recorded a device error, and (top-k only)
 *     before a call with more query rows B*T than the calls it served so far.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = legacy default),
 *     in stream order.  Kernels are launched with programmatic dependent launch: a kernel may
 *     start while the previous kernel on the stream finishes, but it reads and writes global
 *     memory only after that kernel has completed.
 *   - Arguments are validated on the host before any launch; a rejected call returns
 *     CSAHCA_ERR_INVALID_ARG / _UNSUPPORTED / _WORKSPACE and enqueues nothing.
 *   - A failed launch returns CSAHCA_ERR_CUDA.  Errors found on the device (index out of
 *     range, a bounded wait that gave up) are recorded in a device error word and reported
 *     by csahca_device_status().
 *   - Layouts are row-major, batch-major and contiguous; the last index is fastest.
 *   - Positions are 0-based.  A query at position p sees compressed entry j iff the entry's
 *     last token is <= p, i.e. j < (p+1)/m (integer division), capped at Ncap, and the raw
 *     window of the W tokens max(0,p-W+1) .. p (its own token included).  Window rows and
 *     compressed rows enter ONE joint softmax; they are not de-duplicated.
 *   - All H query heads share one KV stream (K and V rows of width d) and one top-k set.
 *   - Raw tokens of the window live in a ring of `ring_cap` slots per sequence: token t is
 *     in slot t % ring_cap.  During chunked prefill, window tokens at positions >= the
 *     chunk's first position are read from the chunk instead.
 *   - No entry point is thread-safe with respect to concurrent calls that share a workspace.
 */
#ifndef CSA_HCA_H
#define CSA_HCA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* csahca_stream_t; /* identical to cudaStream_t */

typedef enum {
    CSAHCA_OK = 0,
    CSAHCA_ERR_INVALID_ARG = 1, /* bad pointer / size / value; nothing enqueued          */
    CSAHCA_ERR_UNSUPPORTED = 2, /* valid, but this dtype/shape combination is not built   */
    CSAHCA_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed                 */
    CSAHCA_ERR_TIMEOUT = 4,     /* (device) a bounded wait gave up                        */
    CSAHCA_ERR_BOUNDS = 5,      /* (device) an index was out of range; access skipped     */
    CSAHCA_ERR_WORKSPACE = 6    /* workspace NULL, too small or not 256-byte aligned      */
} csahca_status;

typedef enum {
    CSAHCA_F32 = 0,          /* float32                                                  */
    CSAHCA_BF16 = 1,         /* bfloat16                                                 */
    CSAHCA_E4M3_ROWSCALE = 2,/* index keys: OCP FP8 E4M3 codes [rows][d_I] (uint8) plus one
                                float32 scale per row, s = amax/448 (1 for a zero row);
                                key = s * code                                           */
    CSAHCA_E2M1_UE8M0 = 3,   /* index keys: OCP MX FP4 E2M1 codes, two per byte, the even
                                element in the low nibble: [rows][d_I/2] (uint8), plus one
                                UE8M0 scale byte (2^(byte-127)) per 32 values:
                                [rows][d_I/32] (uint8); key = 2^(byte-127) * code        */
    CSAHCA_KV_FP8 = 4        /* kv_dtype of pooling, appends and attention: compressed K/V
                                in FP8 with the RoPE dims of K in BF16 (layout below); raw
                                tokens, ring, queries and outputs stay bfloat16          */
} csahca_dtype;

/* Compressed K/V in FP8 (pogovet.com article, detail 5: most KV entries are stored in FP8, only
 * the RoPE dimensions in BF16).  d = 128.  The pages fix neither the RoPE width nor the scale;
 * the layout takes the last 64 dims of a K row as its RoPE dims and one power-of-two scale per
 * 64 FP8 values:
 *   ck: [B][Ncap][224] bytes per K row -- bytes 0..63 the E4M3 codes of dims 0..63, byte 64
 *       their scale byte, bytes 65 / 66 the scale bytes of the entry's V dims 0..63 / 64..127,
 *       bytes 67..95 zero, bytes 96..223 dims 64..127 as bfloat16;
 *   cv: [B][Ncap][128] bytes per V row -- the E4M3 codes of dims 0..127.
 * (Rows start on 32-byte boundaries; the V row's scales travel with the K row.)
 * A block of 64 pooled float32 values with largest magnitude amax gets e = the smallest integer
 * with amax <= 448 * 2^e (0 for an all-zero block; clamped to [-127, 127]), the byte e + 127,
 * and codes RNE_e4m3(x * 2^-e); a value reads back as code * 2^e (exactly a bfloat16 number).
 * The bfloat16 dims are the pooled values rounded to nearest even. */
#define CSAHCA_KV_FP8_K_ROW 224
#define CSAHCA_KV_FP8_V_ROW 128

/* ------------------------------------------------------------------ a1 / a2: pooling
 * Softmax-gated pooling (pogovet.com article, detail 4; honbul.tistory.com/221 "CSA" and
 * "HCA"): block j of sequence b covers tokens j*m .. j*m+m-1;
 *     alpha_i = softmax_i(gate[j*m+i] + slot_bias[i]),  i < m;
 *     ck[b][j] = sum_i alpha_i K[j*m+i],   cv[b][j] = sum_i alpha_i V[j*m+i]
 * (one scalar gate per token, K and V share alpha; fp32 arithmetic, one rounding to the
 * storage dtype).  csa_compress is the CSA compressor (m = 4), hca_compress the HCA one
 * (m = 128); both accept any 1 <= m <= 256.
 *   k_raw, v_raw : [B][raw_stride][d] kv_dtype; row i of sequence b is token raw_pos0[b]+i
 *   gate         : [B][raw_stride] float32 gate logits of the same tokens
 *   raw_pos0     : [B] int64 (device) position of row 0;  n_raw: [B] int64 (device) rows used
 *   slot_bias    : [m] float32
 *   ck, cv       : [B][Ncap][d] kv_dtype; every block lying entirely inside
 *                  [raw_pos0[b], raw_pos0[b]+n_raw[b]) is written at entry j; blocks with
 *                  j >= Ncap are skipped and flag CSAHCA_ERR_BOUNDS on the device.
 *   kv_dtype     : CSAHCA_F32 or CSAHCA_BF16.  d: 1..512, d % 8 == 0.  Or CSAHCA_KV_FP8: raw
 *                  tokens bfloat16, ck/cv in the FP8 layout above (the pooled float32 values
 *                  quantised once), d = 128.  With m = 1 this quantises given rows.
 */
csahca_status csa_compress(const void* k_raw, const void* v_raw, const float* gate,
                           int64_t raw_stride, const int64_t* raw_pos0, const int64_t* n_raw,
                           const float* slot_bias, int m, int B, int d, csahca_dtype kv_dtype,
                           void* ck, void* cv, int64_t Ncap, csahca_stream_t stream);
csahca_status hca_compress(const void* k_raw, const void* v_raw, const float* gate,
                           int64_t raw_stride, const int64_t* raw_pos0, const int64_t* n_raw,
                           const float* slot_bias, int m, int B, int d, csahca_dtype kv_dtype,
                           void* ck, void* cv, int64_t Ncap, csahca_stream_t stream);

/* ------------------------------------------------------------- a4: index-key quantise
 * Low-precision lightning-indexer keys (pogovet.com article, details 4-5; honbul.tistory.com
 * /221 FP4 QAT of the CSA indexer's query-key path).  Converts `rows` input rows
 * [rows][d_I] (in_dtype F32 or BF16) into key_fmt storage (see csahca_dtype):
 *   F32 / BF16 : copy/convert (k_scale unused, may be NULL);
 *   E4M3_ROWSCALE : s = amax/448 in fp32, code = RNE_e4m3_satfinite(x / s) (fp32 divide);
 *   E2M1_UE8M0 : per 32 values, e = smallest integer with amax <= 6*2^e (0 for a zero
 *                block), code = RNE_e2m1(x * 2^-e), stored exponent byte e + 127.
 * d_I % 32 == 0 for E2M1, d_I <= 256.
 */
csahca_status csa_index_key_quantize(const void* k_in, csahca_dtype in_dtype, int64_t rows,
                                     int d_I, csahca_dtype key_fmt, void* k_codes,
                                     void* k_scale, csahca_stream_t stream);

/* ----------------------------------------------------------- a5 + a6: indexer + top-k
 * Lightning indexer (honbul.tistory.com/221 "CSA"; pogovet.com detail 4) with the score
 *     I(t,s) = sum_{h < H_I} w[t][h] * max(0, q_idx[t][h][:] . khat_s)
 * over the visible entries s < n_vis(t) = min(Ncap, (q_pos[t]+1)/m), followed by top-k:
 * order by score descending, equal scores by lower index; the chosen indices are written in
 * ascending order, padded with -1 when n_vis < k.  Deterministic.
 *   q_idx     : [B][T][H_I][d_I] q_dtype (F32 or BF16)
 *   w         : [B][T][H_I] float32
 *   k_codes, k_scale : index keys of sequence b at rows b*Ncap .. (key_fmt layout)
 *   q_pos     : [B*T] int64 (device) query positions
 *   idx_out   : [B][T][k] int32
 *   scores_out: NULL, or [B][T][Ncap] float32 receiving the scores of the visible entries
 *               (entries >= n_vis are left untouched)
 *   workspace : csa_index_topk_workspace(B, T, Ncap, k) bytes, zero-filled before first use
 *               (see Conventions)
 * Supported: 1 <= H_I <= 64; 32 <= d_I <= 256, d_I % 32 == 0; H_I*d_I <= 4096; B*T <= 65535;
 * 1 <= k <= 65536 (k larger than the visible entries pads with -1).
 */
csahca_status csa_index_topk(const void* q_idx, csahca_dtype q_dtype, const float* w,
                             const void* k_codes, const void* k_scale, csahca_dtype key_fmt,
                             int B, int T, int H_I, int d_I, const int64_t* q_pos, int64_t Ncap,
                             int m, int k, int32_t* idx_out, float* scores_out, void* workspace,
                             size_t ws_bytes, csahca_stream_t stream);
size_t csa_index_topk_workspace(int B, int T, int64_t Ncap, int k);
/* Workspace bytes of csa_index_topk_fp4 that allow its prefill form (see there): the bytes of
 * csa_index_topk_workspace, plus B*Ncap*128 + B*T*H_I*128 (rounded to 256) when the form applies. */
size_t csa_index_topk_fp4_workspace(int B, int T, int H_I, int64_t Ncap, int k);

/* The lightning indexer with FP4 queries as well as FP4 keys (pogovet.com detail 5: the indexer runs
 * in FP4; honbul.tistory.com/221: FP4 QAT of the CSA indexer's query-key path).  The queries come in
 * the keys' OCP MX E2M1 form -- q_codes [B][T][H_I][d_I/2] (two codes per byte, the even element in
 * the low nibble) and q_scale [B][T][H_I][d_I/32] UE8M0 bytes, as csa_index_key_quantize produces
 * from bf16 queries with key_fmt CSAHCA_E2M1_UE8M0 -- and the score is
 *     I(t,s) = sum_{h < H_I} w[t][h] * max(0, qhat[t][h][:] . khat_s),  qhat = 2^(byte-127) * code,
 * exact up to the fp32 accumulation.  Keys are CSAHCA_E2M1_UE8M0.  Top-k and outputs as
 * csa_index_topk.  Workspace: csa_index_topk_workspace(B, T, Ncap, k) bytes at least; with
 * csa_index_topk_fp4_workspace(B, T, H_I, Ncap, k) bytes and more than 256 query rows (chunked
 * prefill, T a multiple of 128 / H_I) the keys and queries are first expanded to bf16 in the
 * workspace -- exactly, for block scales up to 2^125 -- and scored 128 / H_I query rows per tensor-
 * core tile; otherwise one query row per work item on the block-scaled MMA.  Supported: d_I = 64,
 * H_I in {16, 32, 64}, Ncap % 256 == 0, k_codes 32-byte, k_scale and q_codes 16-byte, q_scale
 * 2-byte aligned; otherwise CSAHCA_ERR_UNSUPPORTED and nothing is enqueued. */
csahca_status csa_index_topk_fp4(const void* q_codes, const void* q_scale, const float* w,
                                 const void* k_codes, const void* k_scale, int B, int T, int H_I,
                                 int d_I, const int64_t* q_pos, int64_t Ncap, int m, int k,
                                 int32_t* idx_out, float* scores_out, void* workspace,
                                 size_t ws_bytes, csahca_stream_t stream);

/* The indexer scores alone (same arguments and rule as csa_index_topk): writes
 * scores[(b*T+t)*Ncap + s] for the visible entries s < n_vis(t); other entries are untouched. */
csahca_status csa_index_scores(const void* q_idx, csahca_dtype q_dtype, const float* w,
                               const void* k_codes, const void* k_scale, csahca_dtype key_fmt,
                               int B, int T, int H_I, int d_I, const int64_t* q_pos, int64_t Ncap,
                               int m, float* scores, csahca_stream_t stream);

/* Top-k alone over caller-given float32 scores (same order rule and output as above):
 * row r uses scores[r*row_stride + s] for s < n_vis[r] (int64, device).  Scores must not be
 * NaN; -0 and +0 are equal.  Bit-exact with any correct implementation of the rule. */
csahca_status csa_topk_from_scores(const float* scores, int64_t row_stride, int R,
                                   const int64_t* n_vis, int k, int32_t* idx_out,
                                   void* workspace, size_t ws_bytes, csahca_stream_t stream);
size_t csa_topk_workspace(int R, int64_t row_stride, int k);

/* ------------------------------------------------------------------ a7: CSA attention
 * Attention of each query over its selected compressed entries plus the raw window, one
 * joint softmax (honbul.tistory.com/221 "CSA": compressed long-term memory used together
 * with recent raw memory; pogovet.com detail 4: top-k blocks plus a sliding-window branch):
 *     s_i = scale * q[h] . key_i;  out[h] = sum_i softmax(s)_i value_i;  lse[h] = logsumexp(s)
 *   q       : [B][T][H][d] dtype;  out: [B][T][H][d] dtype;  lse: NULL or [B][T][H] float32
 *   ck, cv  : [B][Ncap][d] dtype;  idx: [B][T][k] int32 (-1 entries are skipped; an entry
 *             outside [0, Ncap) is skipped and flags CSAHCA_ERR_BOUNDS on the device);
 *             k = 0 (idx may then be NULL) attends over the raw window alone
 *   ring_k, ring_v : [B][ring_cap][d] dtype (token t in slot t % ring_cap)
 *   chunk_k, chunk_v : NULL (decode) or [B][chunk_stride][d] raw tokens starting at position
 *             chunk_pos0[b] (int64, device); window tokens >= chunk_pos0[b] come from here
 *   W       : window length, 0 <= W <= ring_cap (W <= ring_cap + chunk length for prefill)
 *   q_pos   : [B*T] int64 (device)
 *   dtype   : CSAHCA_F32 or CSAHCA_BF16 (q, caches, ring, chunk and out share it), or
 *             CSAHCA_KV_FP8 (ck/cv in the FP8 layout above; q, ring, chunk and out bfloat16;
 *             d = 128, H in {32, 64}, else CSAHCA_ERR_UNSUPPORTED)
 *   workspace : csa_attend_workspace(B, T, H, d, k, W) bytes, zero-filled before first use
 *               (see Conventions)
 * An empty key set (no selected entry, W = 0) gives out = 0 and lse = -inf.
 */
csahca_status csa_attend(const void* q, int B, int T, int H, int d, float scale, const void* ck,
                         const void* cv, int64_t Ncap, const int32_t* idx, int k,
                         const void* ring_k, const void* ring_v, int ring_cap, int W,
                         const void* chunk_k, const void* chunk_v, const int64_t* chunk_pos0,
                         int64_t chunk_stride, const int64_t* q_pos, csahca_dtype dtype,
                         void* out, float* lse, void* workspace, size_t ws_bytes,
                         csahca_stream_t stream);
size_t csa_attend_workspace(int B, int T, int H, int d, int k, int W);

/* ------------------------------------------------------------------ a8: HCA attention
 * Dense attention over every visible compressed entry (j < min(Ncap, (p+1)/m)) plus the raw
 * window, one joint softmax (honbul.tistory.com/221 "HCA"; pogovet.com detail 4: no sparse
 * selection, dense over all compressed blocks).  The key range is split into chunks that
 * run in parallel; partial results (o_s, lse_s) are merged exactly,
 *     lse = log sum_s exp(lse_s),  o = sum_s exp(lse_s - lse) o_s,
 * in the fixed order s = 0, 1, ... (deterministic).
 * Arguments as csa_attend; `m` is the HCA block size; `splits` = 0 picks the split count.
 * workspace : hca_attend_workspace(B, T, H, d, Ncap, W, splits) bytes, zero-filled before first
 *             use (see Conventions).
 */
csahca_status hca_attend(const void* q, int B, int T, int H, int d, float scale, const void* ck,
                         const void* cv, int64_t Ncap, int m, const void* ring_k,
                         const void* ring_v, int ring_cap, int W, const void* chunk_k,
                         const void* chunk_v, const int64_t* chunk_pos0, int64_t chunk_stride,
                         const int64_t* q_pos, int splits, csahca_dtype dtype, void* out,
                         float* lse, void* workspace, size_t ws_bytes, csahca_stream_t stream);
size_t hca_attend_workspace(int B, int T, int H, int d, int64_t Ncap, int W, int splits);

/* HCA dense attention without any caller workspace and without allocating.  (The method's
 * pages have no counterpart: this serves callers that cannot allocate device memory when they
 * run attention -- e.g. a runtime with a fixed memory budget or an embedding that only hands
 * over its input/output buffers.)  Same arguments and results as hca_attend, minus the
 * workspace: the split-K partial results live in one fixed device array of
 * hca_attend_noalloc_scratch_bytes() bytes (16 MiB) inside the library, which every GPU that
 * loads the library keeps until the process exits.  The split count is lowered until the
 * partials fit; if one split per query (B*T*H*(d+1)*4 bytes plus alignment, plus the 256 KiB
 * of per-row arrival counters) does not fit, the call returns CSAHCA_ERR_WORKSPACE and
 * enqueues nothing.  The array starts zeroed when the library loads, and every call leaves its
 * counters zero again (after a call that recorded a device error, later results of this entry
 * point are not guaranteed in that process).  All calls on a device share the
 * array, so calls that may overlap on the GPU (different streams without ordering) race and
 * must be serialised by the caller.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current); make that first call before any
 * stream capture.  Calls no cudaMalloc/cudaFree or allocating library routine. */
csahca_status hca_attend_noalloc(const void* q, int B, int T, int H, int d, float scale,
                                 const void* ck, const void* cv, int64_t Ncap, int m,
                                 const void* ring_k, const void* ring_v, int ring_cap, int W,
                                 const void* chunk_k, const void* chunk_v,
                                 const int64_t* chunk_pos0, int64_t chunk_stride,
                                 const int64_t* q_pos, int splits, csahca_dtype dtype, void* out,
                                 float* lse, csahca_stream_t stream);
size_t hca_attend_noalloc_scratch_bytes(void);

/* --------------------------------------------------------- a3: compressed-KV cache append
 * Appends n_new raw tokens per sequence (positions pos[b] .. pos[b]+n_new-1, int64 device)
 * to the split cache of honbul.tistory.com/221 "KV cache를 줄이는 방식": the raw tokens go
 * to the window ring (which also holds the tail of an incomplete block, so ring_cap must be
 * >= m-1 and >= 1); every block completed by these tokens is pooled (tokens before pos[b]
 * are read from the ring, the others from the input) and written to ck/cv at its entry
 * index; for CSA the index key of each completed block (kidx_new row r = the r-th block
 * completed in this call: [B][kidx_rows][d_I], kidx_rows = n_new/m + 1) is quantised into
 * k_codes/k_scale (key_fmt) at the same entry index.
 *   k_new, v_new : [B][n_new][d] kv_dtype (bfloat16 for CSAHCA_KV_FP8, whose ck/cv take the
 *                  FP8 layout above while the ring stays bfloat16);  gate_new: [B][n_new] float32
 *   ring_k, ring_v : [B][ring_cap][d];  ring_gate: [B][ring_cap] float32
 * Pooling reads the ring before the new tokens are written to it.
 */
csahca_status csa_cache_append(const void* k_new, const void* v_new, const float* gate_new,
                               const void* kidx_new, csahca_dtype kidx_dtype,
                               const int64_t* pos, int B, int n_new, int d,
                               csahca_dtype kv_dtype, const float* slot_bias, int m,
                               void* ring_k, void* ring_v, float* ring_gate, int ring_cap,
                               void* ck, void* cv, int64_t Ncap, void* k_codes, void* k_scale,
                               csahca_dtype key_fmt, int d_I, csahca_stream_t stream);
csahca_status hca_cache_append(const void* k_new, const void* v_new, const float* gate_new,
                               const int64_t* pos, int B, int n_new, int d,
                               csahca_dtype kv_dtype, const float* slot_bias, int m,
                               void* ring_k, void* ring_v, float* ring_gate, int ring_cap,
                               void* ck, void* cv, int64_t Ncap, csahca_stream_t stream);

/* Writes raw tokens into the window ring only (no pooling): the last step of a chunked
 * prefill, after the chunk's attention has read the old ring.  k_new/v_new:
 * [B][new_stride][d], gate_new: [B][new_stride]; tokens pos[b] .. pos[b]+n_new-1. */
csahca_status swa_ring_write(const void* k_new, const void* v_new, const float* gate_new,
                             int64_t new_stride, const int64_t* pos, int B, int n_new, int d,
                             csahca_dtype kv_dtype, void* ring_k, void* ring_v,
                             float* ring_gate, int ring_cap, csahca_stream_t stream);

/* --------------------------------------------------------------------------- status */
/* Synchronises `stream`, then returns and clears the device error word of the current
 * device (CSAHCA_OK, CSAHCA_ERR_BOUNDS or CSAHCA_ERR_TIMEOUT), or CSAHCA_ERR_CUDA. */
csahca_status csahca_device_status(csahca_stream_t stream);
const char* csahca_status_string(csahca_status s);
/* Self-test of the bounded device waits (no counterpart on the method's pages): launches one warp
 * that waits on a device barrier nothing ever completes, through the same wait routine the
 * tensor-core kernels use.  After ~limit_ns (1 .. 1e9 ns) the wait gives up, records
 * CSAHCA_ERR_TIMEOUT in the device error word and the kernel ends normally, so the context stays
 * usable; csahca_device_status() then reports CSAHCA_ERR_TIMEOUT.  Returns INVALID_ARG for a
 * limit outside the range, CUDA if the launch fails. */
csahca_status csahca_selftest_bounded_wait(uint64_t limit_ns, csahca_stream_t stream);
/* Number of kernel launches this library has enqueued on the calling host thread. */
uint64_t csahca_launch_count(void);
int csahca_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CSA_HCA_H */
