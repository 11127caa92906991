// api.cu - the C ABI declared in include/fa2.h: argument validation, dispatch
// to the kernel translation units, tensor-map encoding and the watchdog word.
#include <math.h>

#include <atomic>
#include <mutex>

#include "fa2.h"
#include "internal.h"

namespace fa2 {

// Watchdog word: kernels OR kStatusTimeout into it when a bounded wait gives up.
__device__ unsigned int g_watchdog_word;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn encode_fn() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode;
}

constexpr int kMaxDevices = 64;
constexpr int kMaxSlots = 64;
std::mutex g_mu;
unsigned int* g_status_ptr[kMaxDevices] = {};
std::atomic<uint64_t> g_smem_done[kMaxSlots];

bool status_word(unsigned int** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_watchdog_word) != cudaSuccess) return false;
        g_status_ptr[dev] = static_cast<unsigned int*>(p);
    }
    *out = g_status_ptr[dev];
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dtype(fa2_dtype d) { return d == FA2_DTYPE_F32 || d == FA2_DTYPE_F16 || d == FA2_DTYPE_BF16; }

// 16-bit types: any multiple of 8 up to 128 (rows of whole 16-byte units, as the
// tensor-memory copies need): the kernels run at the next of 32, 64, 128 with the
// extra columns read as zeros (TMA fills past the tensor edge) and never stored.
// float32 (plain loads and stores): any head dimension up to 128.
bool supported_head_dim(int32_t d, fa2_dtype dtype) {
    if (dtype == FA2_DTYPE_F32) return d >= 1 && d <= 128;
    return d >= 8 && d <= 128 && d % 8 == 0;
}

constexpr int64_t kMaxGridY = 65535;
constexpr int64_t kMaxSeq = (int64_t)1 << 30;

// Shared size checks of the attention calls.
fa2_status check_attention_sizes(int64_t bh, int64_t n_q, int64_t n_k, int32_t head_dim, fa2_dtype dtype, float scale) {
    if (bh <= 0 || n_q <= 0 || n_k <= 0 || head_dim <= 0) return FA2_ERR_INVALID_ARG;
    if (!valid_dtype(dtype)) return FA2_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return FA2_ERR_INVALID_ARG;
    if (!supported_head_dim(head_dim, dtype)) return FA2_ERR_UNSUPPORTED;
    if (bh > kMaxGridY || n_q > kMaxSeq || n_k > kMaxSeq) return FA2_ERR_UNSUPPORTED;
    return FA2_OK;
}

}  // namespace

bool encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* base, uint64_t d0, uint64_t d1,
                    uint64_t d2, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0 * (uint64_t)elem_bytes, d0 * d1 * (uint64_t)elem_bytes};
    const cuuint32_t box[3] = {box0, box1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    auto encode = [&] {
        return fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    };
    CUresult r = encode();
    if (r == CUDA_ERROR_INVALID_CONTEXT) {
        // A host thread with no current context yet (the runtime makes one current only at
        // its first launch or allocation there): the driver call needs one, so make the
        // primary context of the thread's device current, as the launch would, and retry.
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return false;
        r = encode();
    }
    return r == CUDA_SUCCESS;
}

bool watchdog_word(unsigned int** out) { return status_word(out); }

int sm_count() {
    static std::atomic<int> counts[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    int n = counts[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
        counts[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

cudaError_t ensure_smem_limit(const void* func, int bytes, int slot) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (slot < 0 || slot >= kMaxSlots || dev >= 64) return cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    const uint64_t bit = 1ull << dev;
    if (g_smem_done[slot].load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) g_smem_done[slot].fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Whether a thread-block cluster of `size` (2, 4, 8 or 16) CTAs of `func` (`threads` threads,
// `smem` dynamic shared-memory bytes, its limit already raised) can be resident at once on
// the current device; asked of the runtime once per (slot, size, device). A cluster of 16
// needs the kernel's non-portable-cluster-size attribute, set here first.
std::atomic<uint64_t> g_cluster_asked[kMaxSlots][4], g_cluster_fits[kMaxSlots][4];

bool cluster_fits(const void* func, int threads, int smem, int size, int slot) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const int li = size == 2 ? 0 : (size == 4 ? 1 : (size == 8 ? 2 : 3));
    const bool cached = dev >= 0 && dev < 64 && slot >= 0 && slot < kMaxSlots;
    const uint64_t bit = cached ? 1ull << dev : 0;
    if (cached && (g_cluster_asked[slot][li].load(std::memory_order_acquire) & bit))
        return g_cluster_fits[slot][li].load(std::memory_order_acquire) & bit;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)size, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)size;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const bool allowed =
        size <= 8 || cudaFuncSetAttribute(func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    const bool fits = allowed && cudaOccupancyMaxActiveClusters(&n, func, &cfg) == cudaSuccess && n > 0;
    if (!fits) (void)cudaGetLastError();  // a refused query leaves no error behind
    if (cached) {
        if (fits) g_cluster_fits[slot][li].fetch_or(bit, std::memory_order_acq_rel);
        g_cluster_asked[slot][li].fetch_or(bit, std::memory_order_acq_rel);
    }
    return fits;
}

// fa2_backward runs the one-pass kernel (dQ through float32 reductions) for kernel head
// sizes up to 64 with enough key tiles (below) and the two-pass kernels otherwise.  Measured on GB300
// at BH = 32, N = 8192 (preprocess included): head size 32 / 64: 1.51 / 1.65 ms
// one-pass against 1.58 / 1.75 ms for the two passes in one grid; head size 128:
// 2.99 ms against 2.27 ms, where the reductions (4 bytes per query row, key tile
// and head column) reach the L2's reduction throughput.
// The one-pass kernel runs one CTA per key tile of each head; with fewer than half of a
// 148-SM part's worth of them (bh * ceil(n_k / 128) <= 74) the two passes in one grid,
// whose dQ CTAs and key-range and query-range splits add parallelism, are faster (GB300,
// bf16, d = 64: B*H = 2, N = 4096: 0.068 -> 0.050 ms; B*H = 1, N = 8192: 0.117 -> 0.086 ms;
// at 128 and 256 key-tile CTAs the one-pass kernel stays ahead: 0.070 / 0.076 against
// 0.089 / 0.086 ms). Those shapes take the two passes at every head size.
fa2_launch_info& launch_record() {
    thread_local fa2_launch_info record{};
    return record;
}

static bool use_one_pass(int64_t bh, int64_t n_q, int64_t n_k, int32_t head_dim) {
    (void)n_q;
    return pad_head_dim(head_dim) <= 64 && 2 * bh * ((n_k + 127) / 128) > 148;
}

// Workspace of the two-pass backward (the stage entry points, the PSA backward):
// D and LSE2, float32, padded to a multiple of 128 rows per head.
size_t two_pass_workspace_size(int64_t bh, int64_t n_q, int64_t n_k, int32_t head_dim, fa2_dtype dtype) {
    if (check_attention_sizes(bh, n_q, n_k, head_dim, dtype, 1.0f) != FA2_OK) return 0;
    const int64_t n_q_pad = (n_q + 127) / 128 * 128;
    return 2 * (size_t)(bh * n_q_pad) * sizeof(float);
}

namespace {

// stages = kBwdAll with one_pass, for a head size the one-pass kernel serves: the one-pass
// backward (fa2_backward_workspace_size bytes); otherwise the given stages of the two-pass
// backward (two_pass_workspace_size bytes).
fa2_status backward_common(const void* q, const void* k, const void* v, const void* o, const void* d_o, const float* lse,
                           void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int64_t bh,
                           int64_t n_q, int64_t n_k, int32_t head_dim, fa2_dtype dtype, float softmax_scale,
                           void* stream, int stages, bool one_pass) {
    // pointers each stage reads or writes; the others may be null
    const bool pre = stages & kBwdPreprocess, dkdv = stages & kBwdDkDv, dqs = stages & kBwdDq;
    if ((pre && (!o || !d_o || !lse)) || ((dkdv || dqs) && (!q || !k || !v || !d_o)) || (dkdv && (!dk || !dv)) ||
        (dqs && !dq))
        return FA2_ERR_INVALID_ARG;
    fa2_status st = check_attention_sizes(bh, n_q, n_k, head_dim, dtype, softmax_scale);
    if (st != FA2_OK) return st;
    if (dtype == FA2_DTYPE_F32) return FA2_ERR_UNSUPPORTED;
    const void* ptrs[] = {q, k, v, o, d_o, lse, dq, dk, dv};
    for (const void* ptr : ptrs)
        if (ptr && !aligned16(ptr)) return FA2_ERR_MISALIGNED;
    one_pass = one_pass && stages == kBwdAll && use_one_pass(bh, n_q, n_k, head_dim);
    const size_t need = one_pass ? fa2_backward_workspace_size(bh, n_q, n_k, head_dim, dtype)
                                 : two_pass_workspace_size(bh, n_q, n_k, head_dim, dtype);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) return FA2_ERR_WORKSPACE;
    BwdParams p{};
    p.q = q; p.k = k; p.v = v; p.o = o; p.d_o = d_o; p.lse = lse;
    p.dq = dq; p.dk = dk; p.dv = dv;
    p.n_q_pad = (n_q + 127) / 128 * 128;
    p.delta = static_cast<float*>(workspace);
    p.lse2 = p.delta + bh * p.n_q_pad;
    if (one_pass) p.dq_acc = p.lse2 + bh * p.n_q_pad;  // 16-byte aligned: n_q_pad is a multiple of 128
    // the split dQ pass of the two-pass kernels, when the workspace also holds its partial sums
    const size_t part = (!one_pass && (stages & kBwdDq)) ? dq_partial_bytes(bh, n_q, n_k, head_dim) : 0;
    if (part && workspace_bytes >= two_pass_workspace_size(bh, n_q, n_k, head_dim, dtype) + part) {
        p.dq_part = p.lse2 + bh * p.n_q_pad;
        p.dq_splits = dq_key_splits(bh, n_q, n_k);
    }
    p.bh = bh; p.n_q = n_q; p.n_k = n_k; p.d = head_dim; p.dtype = (int)dtype; p.scale = softmax_scale;
    if (!status_word(&p.status)) return FA2_ERR_CUDA;
    fa2_launch_info& rec = launch_record();  // the launch code fills in the splits it takes
    rec.bwd_one_pass = one_pass ? 1 : 0;
    rec.bwd_dkv_query_ranges = 1;
    rec.bwd_dq_key_ranges = 1;
    rec.bwd_key_tiles_per_cta = 0;
    const cudaError_t e = one_pass ? launch_bwd_fused(p, static_cast<cudaStream_t>(stream))
                                   : launch_bwd_tc(p, static_cast<cudaStream_t>(stream), stages);
    return e == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

}  // namespace

fa2_status backward_two_pass(const void* q, const void* k, const void* v, const void* o, const void* d_o,
                             const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                             int64_t bh, int64_t n_q, int64_t n_k, int32_t head_dim, fa2_dtype dtype,
                             float softmax_scale, void* stream) {
    if (!q || !k || !v || !o || !d_o || !lse || !dq || !dk || !dv) return FA2_ERR_INVALID_ARG;
    return backward_common(q, k, v, o, d_o, lse, dq, dk, dv, workspace, workspace_bytes, bh, n_q, n_k, head_dim, dtype,
                           softmax_scale, stream, kBwdAll, false);
}

}  // namespace fa2

using namespace fa2;

extern "C" {

fa2_status fa2_forward(const void* q, const void* k, const void* v, void* o, float* lse, int64_t bh, int64_t n_q,
                       int64_t n_k, int32_t head_dim, fa2_dtype dtype, float softmax_scale, void* stream) {
    if (!q || !k || !v || !o || !lse) return FA2_ERR_INVALID_ARG;
    fa2_status st = check_attention_sizes(bh, n_q, n_k, head_dim, dtype, softmax_scale);
    if (st != FA2_OK) return st;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA2_ERR_MISALIGNED;
    FwdParams p{q, k, v, o, lse, bh, n_q, n_k, head_dim, (int)dtype, softmax_scale, nullptr};
    if (!status_word(&p.status)) return FA2_ERR_CUDA;
    launch_record().fwd_key_ranges = 1;  // the tensor-core launch records its split
    const cudaError_t e = dtype == FA2_DTYPE_F32 ? launch_fwd_f32(p, static_cast<cudaStream_t>(stream))
                                                 : launch_fwd_tc(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

fa2_status psa_fa2_forward(const void* packed, void* o_lo, void* o_hi, float* lse, int64_t bh, int64_t n,
                           int32_t key_dim, fa2_dtype dtype, float softmax_scale, void* stream) {
    if (!packed || !o_lo || !o_hi || !lse) return FA2_ERR_INVALID_ARG;
    fa2_status st = check_attention_sizes(bh, n, n, key_dim, dtype, softmax_scale);
    if (st != FA2_OK) return st;
    if (dtype == FA2_DTYPE_F32 || key_dim > 64) return FA2_ERR_UNSUPPORTED;
    if (!aligned16(packed) || !aligned16(o_lo) || !aligned16(o_hi) || !aligned16(lse)) return FA2_ERR_MISALIGNED;
    // sections of the packed buffer, as FlashAttn2PsaRuntimeOp addresses them: base + s * BH * N * KEY_DIM
    const size_t section = (size_t)bh * (size_t)n * (size_t)key_dim * 2;
    const char* base = static_cast<const char*>(packed);
    FwdParams p{base, base + section, base + 2 * section, o_lo, lse, bh, n, n, key_dim, (int)dtype, softmax_scale, nullptr};
    p.v2 = base + 3 * section;
    p.o2 = o_hi;
    if (!status_word(&p.status)) return FA2_ERR_CUDA;
    return launch_fwd_tc_dual_v(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

// The one-pass backward adds the float32 dQ accumulator, [bh, n_q_pad, pad_head_dim(head_dim)].
size_t fa2_backward_workspace_size(int64_t bh, int64_t n_q, int64_t n_k, int32_t head_dim, fa2_dtype dtype) {
    const size_t two_pass = two_pass_workspace_size(bh, n_q, n_k, head_dim, dtype);
    if (two_pass == 0) return 0;
    if (!use_one_pass(bh, n_q, n_k, head_dim)) return two_pass + dq_partial_bytes(bh, n_q, n_k, head_dim);
    const int64_t n_q_pad = (n_q + 127) / 128 * 128;
    return two_pass + (size_t)(bh * n_q_pad) * (size_t)pad_head_dim(head_dim) * sizeof(float);
}

fa2_status fa2_backward(const void* q, const void* k, const void* v, const void* o, const void* d_o, const float* lse,
                        void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int64_t bh, int64_t n_q,
                        int64_t n_k, int32_t head_dim, fa2_dtype dtype, float softmax_scale, void* stream) {
    if (!q || !k || !v || !o || !d_o || !lse || !dq || !dk || !dv) return FA2_ERR_INVALID_ARG;
    return backward_common(q, k, v, o, d_o, lse, dq, dk, dv, workspace, workspace_bytes, bh, n_q, n_k, head_dim, dtype,
                           softmax_scale, stream, kBwdAll, true);
}

fa2_status fa2_backward_preprocess(const void* o, const void* d_o, const float* lse, void* workspace,
                                   size_t workspace_bytes, int64_t bh, int64_t n_q, int64_t n_k, int32_t head_dim,
                                   fa2_dtype dtype, void* stream) {
    if (!o || !d_o || !lse) return FA2_ERR_INVALID_ARG;
    return backward_common(nullptr, nullptr, nullptr, o, d_o, lse, nullptr, nullptr, nullptr, workspace,
                           workspace_bytes, bh, n_q, n_k, head_dim, dtype, 1.0f, stream, kBwdPreprocess, false);
}

fa2_status fa2_backward_dkdv(const void* q, const void* k, const void* v, const void* d_o, const void* workspace,
                             size_t workspace_bytes, void* dk, void* dv, int64_t bh, int64_t n_q, int64_t n_k,
                             int32_t head_dim, fa2_dtype dtype, float softmax_scale, void* stream) {
    if (!q || !k || !v || !d_o || !dk || !dv) return FA2_ERR_INVALID_ARG;
    return backward_common(q, k, v, nullptr, d_o, nullptr, nullptr, dk, dv, const_cast<void*>(workspace),
                           workspace_bytes, bh, n_q, n_k, head_dim, dtype, softmax_scale, stream, kBwdDkDv, false);
}

fa2_status fa2_backward_dq(const void* q, const void* k, const void* v, const void* d_o, const void* workspace,
                           size_t workspace_bytes, void* dq, int64_t bh, int64_t n_q, int64_t n_k, int32_t head_dim,
                           fa2_dtype dtype, float softmax_scale, void* stream) {
    if (!q || !k || !v || !d_o || !dq) return FA2_ERR_INVALID_ARG;
    return backward_common(q, k, v, nullptr, d_o, nullptr, dq, nullptr, nullptr, const_cast<void*>(workspace),
                           workspace_bytes, bh, n_q, n_k, head_dim, dtype, softmax_scale, stream, kBwdDq, false);
}

fa2_status fa2_backward_passes(const void* q, const void* k, const void* v, const void* d_o, const void* workspace,
                               size_t workspace_bytes, void* dq, void* dk, void* dv, int64_t bh, int64_t n_q,
                               int64_t n_k, int32_t head_dim, fa2_dtype dtype, float softmax_scale, void* stream) {
    if (!q || !k || !v || !d_o || !dq || !dk || !dv) return FA2_ERR_INVALID_ARG;
    return backward_common(q, k, v, nullptr, d_o, nullptr, dq, dk, dv, const_cast<void*>(workspace), workspace_bytes,
                           bh, n_q, n_k, head_dim, dtype, softmax_scale, stream, kBwdDkDv | kBwdDq, false);
}

fa2_status psa_fa2_backward(const void* packed, const void* o_lo, const void* o_hi, const void* d_o_lo,
                            const void* d_o_hi, const float* lse, void* d_packed, void* workspace,
                            size_t workspace_bytes, int64_t bh, int64_t n, int32_t key_dim, fa2_dtype dtype,
                            float softmax_scale, void* stream) {
    if (!packed || !o_lo || !o_hi || !d_o_lo || !d_o_hi || !lse || !d_packed) return FA2_ERR_INVALID_ARG;
    fa2_status st = check_attention_sizes(bh, n, n, key_dim, dtype, softmax_scale);
    if (st != FA2_OK) return st;
    if (dtype == FA2_DTYPE_F32 || key_dim > 64) return FA2_ERR_UNSUPPORTED;
    const void* ptrs[] = {packed, o_lo, o_hi, d_o_lo, d_o_hi, lse, d_packed};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return FA2_ERR_MISALIGNED;
    const size_t need = two_pass_workspace_size(bh, n, n, key_dim, dtype);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) return FA2_ERR_WORKSPACE;
    // sections of the packed buffers: base + s * BH * N * KEY_DIM (FlashAttn2PsaRuntimeOp's pointer arithmetic)
    const size_t section = (size_t)bh * (size_t)n * (size_t)key_dim * 2;
    const char* in = static_cast<const char*>(packed);
    char* out = static_cast<char*>(d_packed);
    BwdParams p{};
    p.q = in; p.k = in + section; p.v = in + 2 * section; p.v2 = in + 3 * section;
    p.o = o_lo; p.o2 = o_hi; p.d_o = d_o_lo; p.d_o2 = d_o_hi; p.lse = lse;
    p.dq = out; p.dk = out + section; p.dv = out + 2 * section; p.dv2 = out + 3 * section;
    p.n_q_pad = (n + 127) / 128 * 128;
    p.delta = static_cast<float*>(workspace);
    p.lse2 = p.delta + bh * p.n_q_pad;
    p.bh = bh; p.n_q = n; p.n_k = n; p.d = key_dim; p.dtype = (int)dtype; p.scale = softmax_scale;
    if (!status_word(&p.status)) return FA2_ERR_CUDA;
    return launch_bwd_tc_dual_v(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

static fa2_status psa_common(int32_t H, int32_t W, int32_t B, int32_t num_heads, fa2_dtype dtype, int* elem_bytes) {
    if (H <= 0 || W <= 0 || B <= 0 || num_heads <= 0) return FA2_ERR_INVALID_ARG;
    if (!valid_dtype(dtype)) return FA2_ERR_INVALID_ARG;
    *elem_bytes = dtype == FA2_DTYPE_F32 ? 4 : 2;
    if ((int64_t)H * W > kMaxSeq) return FA2_ERR_UNSUPPORTED;
    return FA2_OK;
}

fa2_status psa_pack_qkv(const void* qkv, void* packed, int32_t qkv_h, int32_t H, int32_t W, int32_t B, int32_t num_heads,
                        fa2_dtype dtype, void* stream) {
    if (!qkv || !packed) return FA2_ERR_INVALID_ARG;
    int eb = 0;
    fa2_status st = psa_common(H, W, B, num_heads, dtype, &eb);
    if (st != FA2_OK) return st;
    if (qkv_h <= 0 || qkv_h % (4 * num_heads) != 0) return FA2_ERR_INVALID_ARG;
    if (!aligned16(qkv) || !aligned16(packed)) return FA2_ERR_MISALIGNED;
    if (4LL * B * num_heads > kMaxGridY) return FA2_ERR_UNSUPPORTED;
    PsaParams p{qkv, nullptr, packed, 0, eb, B, num_heads, qkv_h / (4 * num_heads), (int64_t)H * W, qkv_h, 0};
    return launch_psa(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

fa2_status psa_merge_attn_nchw(const void* lo, const void* hi, void* out, int32_t c, int32_t H, int32_t W, int32_t B,
                               int32_t num_heads, fa2_dtype dtype, void* stream) {
    if (!lo || !hi || !out) return FA2_ERR_INVALID_ARG;
    int eb = 0;
    fa2_status st = psa_common(H, W, B, num_heads, dtype, &eb);
    if (st != FA2_OK) return st;
    if (c <= 0 || c % (2 * num_heads) != 0) return FA2_ERR_INVALID_ARG;
    if (!aligned16(lo) || !aligned16(hi) || !aligned16(out)) return FA2_ERR_MISALIGNED;
    if (2LL * B * num_heads > kMaxGridY) return FA2_ERR_UNSUPPORTED;
    PsaParams p{lo, hi, out, 1, eb, B, num_heads, c / (2 * num_heads), (int64_t)H * W, 0, c};
    return launch_psa(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

// Shared checks of the V extraction and the adjoints: sizes, channel counts
// (qkv_h = num_heads * 4 * KD, c = num_heads * 2 * KD), alignment, grid limits.
static fa2_status psa_checks(const void* const* ptrs, int nptrs, int32_t qkv_h, int32_t c, int32_t H, int32_t W,
                             int32_t B, int32_t num_heads, fa2_dtype dtype, int* eb, int sections) {
    for (int i = 0; i < nptrs; ++i)
        if (!ptrs[i]) return FA2_ERR_INVALID_ARG;
    fa2_status st = psa_common(H, W, B, num_heads, dtype, eb);
    if (st != FA2_OK) return st;
    if (qkv_h <= 0 || qkv_h % (4 * num_heads) != 0) return FA2_ERR_INVALID_ARG;
    if (c >= 0 && c != qkv_h / 2) return FA2_ERR_INVALID_ARG;
    for (int i = 0; i < nptrs; ++i)
        if (!aligned16(ptrs[i])) return FA2_ERR_MISALIGNED;
    if ((int64_t)sections * B * num_heads > kMaxGridY) return FA2_ERR_UNSUPPORTED;
    return FA2_OK;
}

fa2_status psa_extract_v_nchw(const void* qkv, void* v, int32_t qkv_h, int32_t c, int32_t H, int32_t W, int32_t B,
                              int32_t num_heads, fa2_dtype dtype, void* stream) {
    const void* ptrs[] = {qkv, v};
    int eb = 0;
    fa2_status st = psa_checks(ptrs, 2, qkv_h, c, H, W, B, num_heads, dtype, &eb, 1);
    if (st != FA2_OK) return st;
    PsaParams p{qkv, nullptr, v, kPsaExtractV, eb, B, num_heads, qkv_h / (4 * num_heads), (int64_t)H * W, qkv_h, c};
    return launch_psa(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

fa2_status psa_pack_qkv_backward(const void* d_packed, void* d_qkv, int32_t qkv_h, int32_t H, int32_t W, int32_t B,
                                 int32_t num_heads, fa2_dtype dtype, void* stream) {
    const void* ptrs[] = {d_packed, d_qkv};
    int eb = 0;
    fa2_status st = psa_checks(ptrs, 2, qkv_h, -1, H, W, B, num_heads, dtype, &eb, 4);
    if (st != FA2_OK) return st;
    PsaParams p{d_packed, nullptr, d_qkv, kPsaPackBwd, eb, B, num_heads, qkv_h / (4 * num_heads), (int64_t)H * W, qkv_h, 0};
    return launch_psa(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

fa2_status psa_merge_attn_backward(const void* d_merged, void* d_lo, void* d_hi, int32_t c, int32_t H, int32_t W,
                                   int32_t B, int32_t num_heads, fa2_dtype dtype, void* stream) {
    const void* ptrs[] = {d_merged, d_lo, d_hi};
    int eb = 0;
    if (c <= 0) return FA2_ERR_INVALID_ARG;
    fa2_status st = psa_checks(ptrs, 3, 2 * c, c, H, W, B, num_heads, dtype, &eb, 2);
    if (st != FA2_OK) return st;
    PsaParams p{d_merged, nullptr, d_lo, kPsaMergeBwd, eb, B, num_heads, c / (2 * num_heads), (int64_t)H * W, 2 * c, c};
    p.dst1 = d_hi;
    return launch_psa(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

fa2_status psa_extract_v_backward(const void* d_v, void* d_qkv, int32_t qkv_h, int32_t c, int32_t H, int32_t W,
                                  int32_t B, int32_t num_heads, fa2_dtype dtype, void* stream) {
    const void* ptrs[] = {d_v, d_qkv};
    int eb = 0;
    fa2_status st = psa_checks(ptrs, 2, qkv_h, c, H, W, B, num_heads, dtype, &eb, 1);
    if (st != FA2_OK) return st;
    PsaParams p{d_v, nullptr, d_qkv, kPsaExtractVBwd, eb, B, num_heads, qkv_h / (4 * num_heads), (int64_t)H * W, qkv_h, c};
    p.dtype = (int)dtype;
    return launch_psa(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

fa2_status fa2_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA2_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_watchdog_word, sizeof(word)) != cudaSuccess) return FA2_ERR_CUDA;
    if (word == 0) return FA2_OK;
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_watchdog_word, &zero, sizeof(zero)) != cudaSuccess) return FA2_ERR_CUDA;
    return FA2_ERR_DEVICE_TIMEOUT;
}

fa2_status fa2_last_launch_info(fa2_launch_info* info) {
    if (!info) return FA2_ERR_INVALID_ARG;
    *info = launch_record();
    return FA2_OK;
}

const char* fa2_status_string(fa2_status s) {
    switch (s) {
        case FA2_OK: return "ok";
        case FA2_ERR_INVALID_ARG: return "invalid argument (null pointer, size <= 0, inconsistent shape or bad scale)";
        case FA2_ERR_UNSUPPORTED: return "unsupported (head_dim not a multiple of 8 in [8, 128], dtype, or a size beyond the kernels' limits)";
        case FA2_ERR_MISALIGNED: return "a tensor base pointer is not 16-byte aligned";
        case FA2_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
        case FA2_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait (watchdog)";
        case FA2_ERR_WORKSPACE: return "workspace missing, misaligned or smaller than fa2_backward_workspace_size";
        case FA2_ERR_SCRATCH_LIMIT: return "problem too large for fa2_backward_noalloc's fixed 8 MiB scratch";
        default: return "unknown status";
    }
}

}  // extern "C"
