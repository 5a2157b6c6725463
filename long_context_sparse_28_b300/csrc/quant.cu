// a4: bulk index-key quantisation (one warp per row).
#include "common.cuh"
#include "quant.cuh"

namespace csahca {
namespace {

__global__ void quantize_rows_kernel(const void* __restrict__ in, int in_dtype, int64_t rows, int d_I,
                                     int fmt, void* codes, void* scales) {
    pdl_wait();
    pdl_trigger();
    const int wpc = blockDim.x >> 5;
    const int E = d_I / 32;
    const int64_t in_row_bytes = (int64_t)d_I * (in_dtype == CSAHCA_F32 ? 4 : 2);
    const int64_t crb = key_row_bytes(fmt, d_I), srb = key_scale_bytes(fmt, d_I);
    for (int64_t r = (int64_t)blockIdx.x * wpc + (threadIdx.x >> 5); r < rows; r += (int64_t)gridDim.x * wpc) {
        float x[8];
        load_row_slice(static_cast<const char*>(in) + r * in_row_bytes, in_dtype, E, x);
        quantize_row_warp(x, E, d_I, fmt, static_cast<char*>(codes) + r * crb,
                          scales ? static_cast<char*>(scales) + r * srb : nullptr);
    }
}

}  // namespace
}  // namespace csahca

using namespace csahca;

extern "C" csahca_status csa_index_key_quantize(const void* k_in, csahca_dtype in_dtype, int64_t rows, int d_I,
                                                csahca_dtype key_fmt, void* k_codes, void* k_scale,
                                                csahca_stream_t stream) {
    CSAHCA_REQUIRE(k_in && k_codes && rows >= 0);
    CSAHCA_REQUIRE(in_dtype == CSAHCA_F32 || in_dtype == CSAHCA_BF16);
    CSAHCA_REQUIRE(key_fmt >= CSAHCA_F32 && key_fmt <= CSAHCA_E2M1_UE8M0);
    CSAHCA_REQUIRE(d_I >= 32 && d_I <= 256 && d_I % 32 == 0);
    if (key_fmt == CSAHCA_E2M1_UE8M0) CSAHCA_REQUIRE(d_I % 64 == 0);
    if (key_fmt >= CSAHCA_E4M3_ROWSCALE) CSAHCA_REQUIRE(k_scale != nullptr);
    if (rows == 0) return CSAHCA_OK;
    const int threads = 256;
    const int64_t want = cdiv(rows, threads / 32);
    const int grid = (int)std::min<int64_t>(want, (int64_t)num_sms() * 16);
    (void)launch_pdl(quantize_rows_kernel, dim3(grid), dim3(threads), 0, (cudaStream_t)stream, k_in, in_dtype, rows, d_I, key_fmt, k_codes,
                                                                    k_scale);
    count_launch();
    CSAHCA_CHECK_LAUNCH();
    return CSAHCA_OK;
}
