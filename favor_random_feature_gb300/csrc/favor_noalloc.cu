// favor_noalloc.cu -- favor_attn_forward_noalloc: the tensor-core forward pass
// run on a fixed scratch array that the library owns from load time, for
// callers that must not allocate device memory on the call path.
//
// Who cannot allocate: a process whose framework reserves the GPU's memory
// up front in its own caching pool (so a further cudaMalloc fails or evicts
// the framework's cache), and serving loops that cannot afford the implicit
// device-wide synchronisation of cudaMalloc / cudaFree in the middle of a
// request.  favor_attn_forward grows a workspace with cudaMalloc the first
// time it meets a larger shape; this entry point never calls cudaMalloc,
// cudaFree or any allocating routine.
//
// The scratch is one file-scope __device__ array of kNoAllocScratchBytes.
// Every GPU that loads the library holds it until the process exits.  All
// calls share it and each call leaves its contents behind: two calls whose
// kernels overlap on the GPU (different streams, or different host threads
// without ordering) race on it.  Nothing in it needs to start at zero: within
// a call every scratch word is written by one kernel before another kernel
// reads it.
#include <mutex>

#include "favor_internal.h"

namespace favor {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB
constexpr int kMaxDev = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_addr[kMaxDev];   // device address of the array, per device

// The array's host-side name is only a stand-in: the kernels need its device
// address, looked up once per device with that device current.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FAVOR_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDev) return FAVOR_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return FAVOR_ERR_CUDA;
        }
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return FAVOR_OK;
}

}  // namespace
}  // namespace favor

using namespace favor;

extern "C" int favor_attn_forward_noalloc(const void *q, const void *k, const void *v,
                                          const float *omega, float *out, int B, int H, int L,
                                          int d, int dv, int m, int causal, int feature_map,
                                          cudaStream_t stream) {
    Problem p;
    int rc = make_problem(B, H, L, d, dv, m, causal, feature_map, &p);
    if (rc) return rc;
    if ((rc = validate_args(q, k, v, omega, out, 2, p))) return rc;
    // the size check first: it needs no device and touches no pointer
    const Problem pw = tc_widen(p);
    if (tc_scratch_bytes(pw) > kNoAllocScratchBytes) return FAVOR_ERR_UNSUPPORTED;
    if (!tc_supported(pw)) return FAVOR_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    if ((rc = scratch_address(&scratch))) return rc;
    return tc_run(q, k, v, omega, out, pw, stream, scratch, kNoAllocScratchBytes);
}
