// hca_attend_noalloc: HCA dense attention for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point where they run
// attention: a host runtime with its own fixed memory budget that forbids allocation after
// start-up, an embedding that hands out only the input/output buffers it owns, or code that
// must not touch an allocator at all.  hca_attend needs a caller-provided workspace for its
// split-K partial results; this variant instead keeps those partials in one fixed-size
// device array owned by this library (kScratchBytes below), so the caller passes only the
// inputs and outputs.
//
// Cost of this choice: every GPU that loads the library holds the array until the process
// exits, and all calls on a device share it.
#include "attend.cuh"

#include <mutex>

namespace csahca {
namespace {

// Upper bound of the split-K scratch: partial outputs [R][S][H][d] fp32 plus their
// log-sum-exps [R][S][H] fp32 (two 256-byte-aligned parts).
constexpr size_t kScratchBytes = size_t(16) << 20;   // 16 MiB

static __device__ __align__(256) unsigned char g_hca_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_dev_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of g_hca_scratch on the current device.  Host code cannot use the symbol
// itself (on the host it names a stand-in, not GPU memory), so the address is looked up once
// per device, with that device current, and cached.
csahca_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CSAHCA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_dev_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_hca_scratch) != cudaSuccess || p == nullptr) return CSAHCA_ERR_CUDA;
        g_scratch_dev_ptr[dev] = p;
    }
    *out = g_scratch_dev_ptr[dev];
    return CSAHCA_OK;
}

}  // namespace
}  // namespace csahca

using namespace csahca;

extern "C" {

size_t hca_attend_noalloc_scratch_bytes(void) { return kScratchBytes; }

csahca_status hca_attend_noalloc(const void* q, int B, int T, int H, int d, float scale, const void* ck,
                                 const void* cv, int64_t Ncap, int m, const void* ring_k, const void* ring_v,
                                 int ring_cap, int W, const void* chunk_k, const void* chunk_v,
                                 const int64_t* chunk_pos0, int64_t chunk_stride, const int64_t* q_pos, int splits,
                                 csahca_dtype dtype, void* out, float* lse, csahca_stream_t stream) {
    AttendArgs a{};
    a.is_csa = false;
    a.q = q; a.B = B; a.T = T; a.H = H; a.d = d; a.scale = scale; a.ck = ck; a.cv = cv; a.Ncap = Ncap;
    a.idx = nullptr; a.k = 0; a.m = m; a.ring_k = ring_k; a.ring_v = ring_v; a.ring_cap = ring_cap; a.W = W;
    a.chunk_k = chunk_k; a.chunk_v = chunk_v; a.chunk_pos0 = chunk_pos0; a.chunk_stride = chunk_stride;
    a.q_pos = q_pos; a.dtype = dtype; a.out = out; a.lse = lse;
    a.total_max = tile_space_keys(Ncap, W);
    if (splits < 0) return CSAHCA_ERR_INVALID_ARG;
    const csahca_status v = attend_validate(a);
    if (v != CSAHCA_OK) return v;
    // Pick the split count as hca_attend would, then lower it until the partials fit the
    // fixed scratch; if even one split per query does not fit, refuse the call.
    const int R = B * T;
    int s_req = splits > 0 ? splits : plan_splits(R, a.total_max, 0).S;
    while (s_req > 1 && attend_workspace_bytes(R, H, d, plan_splits(R, a.total_max, s_req)) > kScratchBytes)
        s_req = (s_req + 1) / 2 < s_req ? (s_req + 1) / 2 : s_req - 1;
    if (attend_workspace_bytes(R, H, d, plan_splits(R, a.total_max, s_req)) > kScratchBytes)
        return CSAHCA_ERR_WORKSPACE;
    void* scratch = nullptr;
    const csahca_status sa = scratch_address(&scratch);
    if (sa != CSAHCA_OK) return sa;
    return attend_run(a, s_req, scratch, kScratchBytes, (cudaStream_t)stream);
}

}  // extern "C"
