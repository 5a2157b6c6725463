// Library runtime: the device error word, launch bookkeeping and status reporting.
#include "common.cuh"
#include "tc_ptx.cuh"

#include <atomic>
#include <mutex>

namespace csahca {

// One error word per device that loads the library; kernels OR error bits into it.
__device__ unsigned g_error_word;

namespace {
constexpr int kMaxDevices = 64;
unsigned* g_err_ptr[kMaxDevices] = {nullptr};
int g_sms[kMaxDevices] = {0};
std::mutex g_mu;
thread_local uint64_t g_launches = 0;
}  // namespace

unsigned* err_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    if (g_err_ptr[dev]) return g_err_ptr[dev];
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<unsigned*>(p);
    }
    return g_err_ptr[dev];
}

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    if (!g_sms[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sms[dev] = n > 0 ? n : 148;
    }
    return g_sms[dev];
}

void count_launch(int n) { g_launches += (uint64_t)n; }

namespace {
// One warp waits on an mbarrier that nothing ever arrives on, through the same bounded wait the
// tensor-core kernels use; the wait gives up after limit_ns, flags CSAHCA_ERR_TIMEOUT in the
// error word and the kernel returns normally.
__global__ void bounded_wait_kernel(uint64_t limit_ns, unsigned* err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();
    (void)tc::mbar_wait(&bar, 0, err, limit_ns);
}
}  // namespace

}  // namespace csahca

extern "C" {

csahca_status csahca_device_status(csahca_stream_t stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return CSAHCA_ERR_CUDA;
    unsigned* p = csahca::err_word();
    if (!p) return CSAHCA_ERR_CUDA;
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, csahca::g_error_word, sizeof v) != cudaSuccess) return CSAHCA_ERR_CUDA;
    if (cudaMemcpyToSymbol(csahca::g_error_word, &zero, sizeof zero) != cudaSuccess) return CSAHCA_ERR_CUDA;
    if (v & csahca::ERRBIT_TIMEOUT) return CSAHCA_ERR_TIMEOUT;
    if (v & csahca::ERRBIT_BOUNDS) return CSAHCA_ERR_BOUNDS;
    return CSAHCA_OK;
}

const char* csahca_status_string(csahca_status s) {
    switch (s) {
        case CSAHCA_OK: return "ok";
        case CSAHCA_ERR_INVALID_ARG: return "invalid argument";
        case CSAHCA_ERR_UNSUPPORTED: return "unsupported dtype/shape combination";
        case CSAHCA_ERR_CUDA: return "CUDA error";
        case CSAHCA_ERR_TIMEOUT: return "bounded device wait timed out";
        case CSAHCA_ERR_BOUNDS: return "device-side index out of range";
        case CSAHCA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    }
    return "unknown status";
}

uint64_t csahca_launch_count(void) { return csahca::g_launches; }

csahca_status csahca_selftest_bounded_wait(uint64_t limit_ns, csahca_stream_t stream) {
    if (limit_ns == 0 || limit_ns > 1000000000ull) return CSAHCA_ERR_INVALID_ARG;
    unsigned* err = csahca::err_word();
    if (!err) return CSAHCA_ERR_CUDA;
    csahca::bounded_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(limit_ns, err);
    csahca::count_launch();
    return cudaGetLastError() == cudaSuccess ? CSAHCA_OK : CSAHCA_ERR_CUDA;
}

int csahca_version(void) { return 1; }

}  // extern "C"
