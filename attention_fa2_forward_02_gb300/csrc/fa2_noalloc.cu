// fa2_noalloc.cu - fa2_backward for callers that cannot allocate device memory.
//
// fa2_backward needs a device workspace (the row sums D, a base-2 copy of the
// LSE and a float32 dQ accumulator).  Some callers cannot hand one over: code whose device memory is
// owned by a host framework's pool or arena (a raw cudaMalloc there would
// bypass the pool's accounting), and services that fix their memory budget at
// start-up and must not allocate - or risk running out of memory - while
// serving.  fa2_backward_noalloc serves them: it takes the workspace from a
// fixed array in this file instead of from the caller.
//
// The array is kNoallocScratchBytes per device, reserved on every GPU that
// loads this library until the process exits.  Its device address is looked
// up once per device (cudaGetSymbolAddress) on the first call made with that
// device current; make that first call before capturing any stream.  All calls
// share the one array: calls whose GPU work overlaps (different streams, or
// different host threads, on one device) race on it and must be serialised by
// the caller.  Nothing in the array has to start at zero: every call rewrites
// all of the part it reads.
#include <mutex>

#include "fa2.h"
#include "internal.h"

namespace fa2 {

// 8 MiB: the two-pass backward needs 8 bytes of workspace per query row (rounded
// up to 128 rows per head), so this covers BH * ceil(n_q / 128) * 128 <= 1,048,576;
// the one-pass backward (4 * head size bytes more per row, the dQ accumulator)
// runs when it fits too.
constexpr size_t kNoallocScratchBytes = size_t(8) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once per
// device).  In host code the symbol itself is only a host-side stand-in, not a
// device address, so it is never passed to a kernel directly.
fa2_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA2_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA2_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FA2_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return FA2_OK;
}

}  // namespace
}  // namespace fa2

extern "C" fa2_status fa2_backward_noalloc(const void* q, const void* k, const void* v, const void* o, const void* d_o,
                                           const float* lse, void* dq, void* dk, void* dv, int64_t bh, int64_t n_q,
                                           int64_t n_k, int32_t head_dim, fa2_dtype dtype, float softmax_scale,
                                           void* stream) {
    const size_t need = fa2::two_pass_workspace_size(bh, n_q, n_k, head_dim, dtype);
    if (need == 0)  // invalid sizes: the regular entry point names the offending argument, launching nothing
        return fa2_backward(q, k, v, o, d_o, lse, dq, dk, dv, nullptr, 0, bh, n_q, n_k, head_dim, dtype,
                            softmax_scale, stream);
    if (need > fa2::kNoallocScratchBytes) return FA2_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    const fa2_status st = fa2::scratch_address(&scratch);
    if (st != FA2_OK) return st;
    // the one-pass backward when its dQ accumulator fits as well, else the two-pass one
    if (fa2_backward_workspace_size(bh, n_q, n_k, head_dim, dtype) <= fa2::kNoallocScratchBytes)
        return fa2_backward(q, k, v, o, d_o, lse, dq, dk, dv, scratch, fa2::kNoallocScratchBytes, bh, n_q, n_k,
                            head_dim, dtype, softmax_scale, stream);
    return fa2::backward_two_pass(q, k, v, o, d_o, lse, dq, dk, dv, scratch, fa2::kNoallocScratchBytes, bh, n_q, n_k,
                                  head_dim, dtype, softmax_scale, stream);
}
