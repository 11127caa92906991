// internal.h - host-side interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "fa2.h"

namespace fa2 {

enum Dtype : int { kF32 = 0, kF16 = 1, kBf16 = 2 };

// The kernel size a head dimension runs at (head_dim is a multiple of 8, <= 128).
inline int pad_head_dim(int d) { return d <= 32 ? 32 : (d <= 64 ? 64 : 128); }

// Key ranges the dQ pass of the two-pass backward divides each query tile's keys into when
// the unsplit dQ CTAs (one per query tile, each looping over all key tiles of its head)
// would not fill one wave of a 148-SM part: enough ranges for about one dQ CTA per SM, at
// least 8 key tiles per range, at most 8 ranges. Each range's CTA writes a float32 partial
// sum and a last kernel adds them in range order (bit-reproducible). With a wave of dQ
// CTAs or more the split only adds the partial sums' traffic (measured on GB300 at
// B=1 H=32 N_q=1024 N_k=32768: 1.249 ms unsplit, 1.259 ms in two ranges). A function of the
// sizes alone, so that the results do not depend on the device.
inline int dq_key_splits(int64_t bh, int64_t n_q, int64_t n_k) {
    const int64_t n_qt = (n_q + 127) / 128, n_kt = (n_k + 127) / 128;
    const int64_t dq_ctas = bh * n_qt;
    int64_t s = (148 + dq_ctas - 1) / dq_ctas;
    if (s > n_kt / 8) s = n_kt / 8;
    if (s > 8) s = 8;
    return s < 2 ? 1 : (int)s;
}

// Largest cluster of the key- and query-range splits over n_tiles tiles: 16 CTAs (a
// non-portable cluster size) where each CTA's share of a row, kernel head size / 16 columns,
// is still a whole 16-byte group of float32 (64 and 128) and each range keeps at least 16
// tiles, else 8. With fewer tiles per range the 16-way exchange of the combine costs more
// than the shorter loops save (GB300, d = 128: B*H = 4, N_q = 16384, N_k = 256, dK/dV query
// ranges 8 -> 16: 0.099 -> 0.123 ms; with 16 tiles per range, B*H = 2, N_q = 32768,
// N_k = 128: 0.117 -> 0.094 ms, and the forward at B*H = 2, N_q = 128, N_k = 32768: 0.074 ->
// 0.054 ms).
inline int max_range_splits(int kernel_head_dim, int64_t n_tiles) {
    return kernel_head_dim >= 64 && n_tiles >= 16 * 16 ? 16 : 8;
}

// Key ranges of the forward's cluster split (one CTA per range, the ranges of a query-tile
// pair in one thread-block cluster): when the forward's CTAs (query-tile pairs x heads) would
// fill at most half of a 148-SM part, the largest power of two up to max_range_splits that
// keeps at most 148 CTAs and at least 8 key tiles per range; else 1. A function of the sizes alone, so
// that the results do not depend on the device.
inline int fwd_key_splits(int64_t ctas, int64_t n_kt, int kernel_head_dim) {
    const int max_splits = max_range_splits(kernel_head_dim, n_kt);
    if (ctas < 1 || 2 * ctas > 148) return 1;
    int64_t cap = 148 / ctas;
    if (cap > n_kt / 8) cap = n_kt / 8;
    if (cap > max_splits) cap = max_splits;
    int s = 1;
    while (2 * s <= cap) s *= 2;
    return s;
}

// Query ranges the dK/dV pass divides each key tile's queries into (one CTA per range, the
// ranges of a key tile in one thread-block cluster that adds their dK and dV in distributed
// shared memory): for queries far outnumbering the keys (at least 16 query tiles per key
// tile) of few heads (the dK/dV CTAs, key tiles x heads, filling at most half of a 148-SM
// part), the largest power of two up to max_range_splits that keeps at most 148 CTAs and at
// least 8 query tiles per range; else 1. The split pass runs apart from the dQ pass, so it pays only
// where unsplit dK/dV CTAs would each walk far more query tiles than the dQ CTAs walk key
// tiles (measured on GB300, d = 128: 16 query tiles per key tile 1.2x faster, 8 and fewer
// slower than the one-grid passes). A function of the sizes alone.
inline int dkv_query_splits(int64_t bh, int64_t n_q, int64_t n_k, int kernel_head_dim) {
    const int64_t n_kt = (n_k + 127) / 128, ctas = bh * n_kt, n_qt = (n_q + 127) / 128;
    const int max_splits = max_range_splits(kernel_head_dim, n_qt);
    if (ctas < 1 || 2 * ctas > 148 || n_qt < 16 * n_kt) return 1;
    int64_t cap = 148 / ctas;
    if (cap > n_qt / 8) cap = n_qt / 8;
    if (cap > max_splits) cap = max_splits;
    int s = 1;
    while (2 * s <= cap) s *= 2;
    return s;
}

// Bytes of the float32 dQ partial sums of a split dQ pass ([splits, bh, n_q_pad, kernel
// head size]); 0 when the pass is not split.
inline size_t dq_partial_bytes(int64_t bh, int64_t n_q, int64_t n_k, int d) {
    const int s = dq_key_splits(bh, n_q, n_k);
    if (s < 2) return 0;
    return (size_t)s * (size_t)bh * (size_t)((n_q + 127) / 128 * 128) * (size_t)pad_head_dim(d) * sizeof(float);
}

struct FwdParams {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;
    int64_t bh, n_q, n_k;
    int d;
    int dtype;
    float scale;
    unsigned int* status;  // device watchdog word
    const void* v2 = nullptr;  // second value tensor (PSA V_hi) for launch_fwd_tc_dual_v
    void* o2 = nullptr;        // its output
};

struct BwdParams {
    const void* q;
    const void* k;
    const void* v;
    const void* o;
    const void* d_o;
    const float* lse;
    void* dq;
    void* dk;
    void* dv;
    float* delta;  // [bh, n_q_pad] minus the row sums D (0 in the padding rows), inside the workspace
    float* lse2;   // [bh, n_q_pad] -LSE * log2(e) (-inf in the padding rows), inside the workspace
    int64_t n_q_pad;
    int64_t bh, n_q, n_k;
    int d;
    int dtype;
    float scale;
    unsigned int* status;
    // second (V, O, dO) triple sharing the probabilities, for launch_bwd_tc_dual_v
    const void* v2 = nullptr;
    const void* o2 = nullptr;
    const void* d_o2 = nullptr;
    void* dv2 = nullptr;
    // float32 dQ accumulator of the one-pass backward, [bh, n_q_pad, pad_head_dim(d)],
    // inside the workspace; zeroed by the preprocess stage when set
    float* dq_acc = nullptr;
    // float32 dQ partial sums of a split dQ pass, [dq_splits, bh, n_q_pad,
    // pad_head_dim(d)], inside the workspace (null: the dQ pass is not split)
    float* dq_part = nullptr;
    int dq_splits = 1;
};

// The PSA rearrangements.  Pack / merge and their adjoints are batched 2-D
// transposes (dst block z, [cols, rows] row-major, is the transpose of src block
// z, [rows, cols] row-major) whose block offsets come from the map `kind`
// selects; the V extraction and its adjoint copy / accumulate contiguous runs.
enum PsaKind : int { kPsaPack = 0, kPsaMerge = 1, kPsaExtractV = 2, kPsaPackBwd = 3, kPsaMergeBwd = 4, kPsaExtractVBwd = 5 };

struct PsaParams {
    const void* src0;
    const void* src1;  // merge: hi (src0 = lo); otherwise unused
    void* dst;
    int kind;          // PsaKind
    int elem_bytes;    // 2 or 4
    int64_t B, nh, kd, n, qkv_h, c;
    void* dst1 = nullptr;  // merge backward: d_hi (dst = d_lo)
    int dtype = 0;         // Dtype, for the accumulating adjoint
};

cudaError_t launch_fwd_tc(const FwdParams& p, cudaStream_t stream);
cudaError_t launch_fwd_f32(const FwdParams& p, cudaStream_t stream);
// One pass over the scores applied to two value tensors (v, v2) with outputs (o, o2).
cudaError_t launch_fwd_tc_dual_v(const FwdParams& p, cudaStream_t stream);
// Backward stages, combinable as a bit mask.
enum BwdStage : int { kBwdPreprocess = 1, kBwdDkDv = 2, kBwdDq = 4, kBwdAll = 7 };
cudaError_t launch_bwd_tc(const BwdParams& p, cudaStream_t stream, int stages);
// All three stages for two (V, O, dO) triples sharing Q, K and the probabilities:
// dQ, dK from the summed dS; dV and dV2 per triple.
cudaError_t launch_bwd_tc_dual_v(const BwdParams& p, cudaStream_t stream);
// The whole backward in three launches: preprocess (also zeroing p.dq_acc), one
// pass over key tiles producing dK, dV and the dQ sums, and the dQ rounding pass.
cudaError_t launch_bwd_fused(const BwdParams& p, cudaStream_t stream);
cudaError_t launch_psa(const PsaParams& p, cudaStream_t stream);

// Workspace bytes of the two-pass backward (D and LSE2 only); 0 for invalid sizes.
size_t two_pass_workspace_size(int64_t bh, int64_t n_q, int64_t n_k, int32_t head_dim, fa2_dtype dtype);
// fa2_backward through the two-pass kernels (preprocess, dK/dV pass, dQ pass):
// needs only two_pass_workspace_size bytes of workspace.
fa2_status backward_two_pass(const void* q, const void* k, const void* v, const void* o, const void* d_o,
                             const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                             int64_t bh, int64_t n_q, int64_t n_k, int32_t head_dim, fa2_dtype dtype,
                             float softmax_scale, void* stream);

// Encodes a 3-D tiled tensor map over a contiguous [d2, d1, d0] tensor of
// `elem_bytes` elements (d0 innermost), box {box0, box1, 1}.  Returns false on failure.
bool encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* base, uint64_t d0, uint64_t d1,
                    uint64_t d2, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle);

// Device address of the watchdog word on the current device (looked up once per device).
bool watchdog_word(unsigned int** out);

// Number of SMs of the current device (looked up once per device; 148 if the query fails).
int sm_count();
// Whether a cluster of `size` (2, 4, 8 or 16) CTAs of `func` can be resident at once on the
// current device (its dynamic shared-memory limit already raised to `smem`; for 16, the
// non-portable cluster size is allowed for it first); cached per slot and size.
bool cluster_fits(const void* func, int threads, int smem, int size, int slot);

// The calling host thread's record of what its most recent calls launched (returned by
// fa2_last_launch_info); the launch code writes the choices it made.
fa2_launch_info& launch_record();

// Raises the dynamic shared-memory limit of `func` on the current device once.
cudaError_t ensure_smem_limit(const void* func, int bytes, int slot);

}  // namespace fa2
