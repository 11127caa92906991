/*
 * fa2.h - C ABI of the GB300 (sm_103a) FlashAttention-2 + PSA library.
 *
 * Every entry point enqueues its work on `stream` (a cudaStream_t passed as a
 * plain pointer; NULL means the legacy default stream) and returns at once.  No
 * entry point allocates device memory, synchronises, or throws; each returns an
 * fa2_status.  Arguments are validated on the host before anything is launched:
 * a call that returns anything but FA2_OK has launched nothing, except
 * FA2_ERR_CUDA, which reports a failed launch.  FA2_OK means "enqueued": a kernel
 * that later gives up a bounded wait on the device is reported only by
 * fa2_device_status (see there), and leaves that call's outputs partly written.
 * Device pointers must be memory of the calling thread's current device, where the
 * kernels run (memory of another device is not checked for and is not valid).
 * Any host thread may call the library.  A thread with no current CUDA context gets the
 * primary context of its current device made current (as a kernel launch would) before
 * the library's first driver call there.
 *
 * Common conventions
 *  - All tensor pointers are caller-owned DEVICE memory, contiguous, row-major,
 *    in the layouts given per call.  The library keeps no pointer after the call
 *    returns; the caller keeps the buffers alive until the stream work is done.
 *  - Outputs must not alias inputs or each other.
 *  - Base pointers must be 16-byte aligned (FA2_ERR_MISALIGNED otherwise).
 *  - Sizes are 64-bit where a product can pass 2^31; every size must be > 0
 *    (FA2_ERR_INVALID_ARG), following the pages' rule that an empty sequence or
 *    head dimension is an error ("vyre-libs 0.7.2 flash_attention_2.rs",
 *    flash_attention_2: a trap program for seq_len, head_dim or tile_size 0).
 *  - Layout of attention tensors: [BH, N, HEAD_DIM] with BH = BATCH * N_HEADS
 *    ("vision-rs 0.1.1 flash_attn2.rs", module comment: all tensors stored as
 *    [BATCH * N_HEADS, N_CTX, HEAD_DIM] row-major, contiguous).
 *  - HEAD_DIM: for BF16 / F16 any multiple of 8 from 8 to 128 (rows must be
 *    whole 16-byte units for the tensor-memory copies); for F32 any value from 1
 *    to 128, as the pages' builders allow (e.g. 7).  The kernels run at the next
 *    of 32, 64, 128; the columns beyond HEAD_DIM are read as zeros and never
 *    written.  A 16-bit head dimension that is not a multiple of 8 returns
 *    FA2_ERR_UNSUPPORTED.
 */
#ifndef FA2_GB300_H
#define FA2_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA2_OK = 0,
    FA2_ERR_INVALID_ARG = 1,     /* a size <= 0, a null pointer, inconsistent shapes, bad scale */
    FA2_ERR_UNSUPPORTED = 2,     /* valid arguments this build has no kernel for (head_dim, dtype) */
    FA2_ERR_MISALIGNED = 3,      /* a base pointer not 16-byte aligned */
    FA2_ERR_CUDA = 4,            /* a CUDA runtime call or kernel launch failed */
    FA2_ERR_DEVICE_TIMEOUT = 5,  /* a kernel gave up a bounded wait (reported by fa2_device_status) */
    FA2_ERR_WORKSPACE = 6,       /* workspace pointer null/misaligned or smaller than required */
    FA2_ERR_SCRATCH_LIMIT = 7    /* the problem needs more than fa2_backward_noalloc's fixed scratch */
} fa2_status;

typedef enum {
    FA2_DTYPE_F32 = 0,   /* IEEE binary32 */
    FA2_DTYPE_F16 = 1,   /* IEEE binary16 */
    FA2_DTYPE_BF16 = 2   /* bfloat16 */
} fa2_dtype;

/*
 * fa2_forward - attention forward with the saved row log-sum-exp.
 *
 * Defined by "vision-rs 0.1.1 flash_attn2.rs", kernel flash_attention2_forward:
 * for each (bh, i): s_ij = softmax_scale * sum_d q[bh,i,d] k[bh,j,d];
 * O[bh,i,:] = sum_j softmax_j(s_i.) v[bh,j,:]; LSE[bh,i] = m_i + ln l_i with
 * m_i = max_j s_ij and l_i = sum_j exp(s_ij - m_i) (the online-softmax
 * recurrence of that kernel reaches this up to rounding).  No masking.
 *
 *   q    [bh, n_q, head_dim]   dtype, device, read
 *   k, v [bh, n_k, head_dim]   dtype, device, read
 *   o    [bh, n_q, head_dim]   dtype, device, written (rounded to nearest even)
 *   lse  [bh, n_q]             float32, device, written, natural log of the
 *                              scaled scores (the page stores it in the input
 *                              dtype; this library always stores float32)
 *   softmax_scale              > 0 and finite; callers normally pass 1/sqrt(head_dim)
 *
 * dtype BF16 / F16: head_dim a multiple of 8 in [8, 128]; tensor-core kernel, float32
 * accumulation, the probabilities rounded to dtype before the P.V product.
 * dtype F32: any head_dim in [1, 128]; a float32 CUDA-core kernel (meant for
 * small problems; float32 products and sums throughout).
 * Few query tiles, many keys (bh * ceil(n_q / 256) CTAs filling at most half of 148 SMs,
 * at least 16 key tiles): the keys of each 256-row query block are split over a
 * thread-block cluster of 2, 4, 8 or 16 CTAs (16 only for head_dim > 32 and at least 256
 * key tiles; at least 8 key tiles per CTA) whose (O, max, sum) are combined in
 * distributed shared memory, in a fixed order (the result depends on the sizes only, on
 * any device that can hold such a cluster at once; one that cannot takes fewer ranges).
 * Precision over long key ranges: each row's O and l are summed one 128-key tile at a
 * time in float32 over a CTA's key range, so the error can grow like (key tiles per
 * CTA) * 2^-24 times sum_j P_ij |v_j| (about 1.5e-5 at 256 key tiles; 0.8 % at 131,079,
 * which one head of 16.8M keys would give a single CTA, 0.05 % as the cluster's 16 ranges).
 * n_q and n_k are limited to 2^30 and bh to 65535 (FA2_ERR_UNSUPPORTED past them).
 * Errors: FA2_ERR_INVALID_ARG, FA2_ERR_UNSUPPORTED, FA2_ERR_MISALIGNED, FA2_ERR_CUDA.
 */
fa2_status fa2_forward(const void* q, const void* k, const void* v, void* o, float* lse,
                       int64_t bh, int64_t n_q, int64_t n_k, int32_t head_dim,
                       fa2_dtype dtype, float softmax_scale, void* stream);

/*
 * fa2_backward_workspace_size - bytes of device workspace fa2_backward needs
 * for these sizes (0 if the sizes are invalid).  With n_q_pad = ceil(n_q / 128) * 128
 * and hd = head_dim rounded up to 32, 64 or 128, the workspace holds
 *   the row sums D = rowsum(O * dO), float32 [bh, n_q_pad]      (4 * bh * n_q_pad bytes),
 *   a base-2 copy of the LSE, float32 [bh, n_q_pad]             (4 * bh * n_q_pad bytes),
 *   for the one-pass backward (head_dim <= 64, bh * ceil(n_k / 128) > 74), the float32 dQ accumulator
 *   [bh, n_q_pad, hd]                                           (4 * bh * n_q_pad * hd bytes),
 *   for head_dim > 64 when the dQ pass is split, its float32 partial sums
 *   [splits, bh, n_q_pad, hd]                          (4 * splits * bh * n_q_pad * hd bytes).
 * A dK/dV pass split over query ranges (see fa2_backward) adds its shares in shared
 * memory and takes no workspace.
 * The dQ pass (one CTA per 128-row query tile, looping over all key tiles) is split when
 * its CTAs, ceil(n_q / 128) * bh of them, would be fewer than about 148 (one wave): each
 * query tile's keys are divided into splits = min(ceil(148 / (bh * ceil(n_q / 128))),
 * floor(ceil(n_k / 128) / 8), 8) ranges (no split if that is below 2), each range's CTA
 * writes a float32 partial sum and a last kernel adds them in range order, so dq stays
 * bit-reproducible (it can differ in the last bits from the unsplit pass's sum).
 * The three stage entry points below need only the first two parts
 * (8 * bh * n_q_pad bytes); a buffer of this size serves them as well (the dQ pass then
 * runs unsplit); given the partial sums' room too, they split the dQ pass as fa2_backward
 * does, and their results equal fa2_backward's bit for bit for head_dim > 64.
 */
size_t fa2_backward_workspace_size(int64_t bh, int64_t n_q, int64_t n_k, int32_t head_dim, fa2_dtype dtype);

/*
 * fa2_backward - dQ, dK and dV of attention from dO, O and the saved LSE.
 *
 * Defined by "vision-rs 0.1.1 flash_attn2.rs", kernels
 * flash_attention2_backward_dq and flash_attention2_backward_dkv:
 * D_i = sum_d O_id dO_id;  P_ij = exp(s_ij - LSE_i);  dV_j = sum_i P_ij dO_i;
 * dS_ij = P_ij (dO_i . v_j - D_i);  dQ_i = scale sum_j dS_ij k_j;
 * dK_j = scale sum_i dS_ij q_i.
 *  - head_dim > 64: the page's structure, a pass over key tiles (dK, dV) and a
 *    pass over query tiles (dQ), after the row sums D: two launches (the stage
 *    entry points fa2_backward_preprocess and fa2_backward_passes below);
 *  - head_dim <= 64 with more than 74 key tiles in all (bh * ceil(n_k / 128) > 74;
 *    fewer run the two launches above): the row sums D (and a reset of the dQ
 *    accumulator), one pass over key tiles that also adds each tile's share of dQ
 *    into a float32 accumulator in the workspace with reductions, and a rounding
 *    pass for dq.
 *    The page's dQ pass recomputes S and dP; at these head sizes that costs more
 *    than the reductions.  The reductions land in any order, so dq is not
 *    bit-reproducible from run to run here (dk and dv are).
 *  - many more queries than keys in few heads (bh * ceil(n_k / 128) key tiles filling
 *    at most half of 148 SMs, at least 16 query tiles per key tile): the dK/dV pass
 *    splits each key tile's queries over a thread-block cluster of 2, 4, 8 or 16 CTAs
 *    (16 only for head_dim > 32 and at least 256 query tiles; at least 8 query tiles
 *    per CTA) that add their shares in distributed shared memory, in a fixed order
 *    (bit-reproducible; a device that cannot hold such a cluster at once takes fewer
 *    ranges), and the dQ pass follows as its own launch.
 *  - few query tiles, many keys: the dQ pass splits each query tile's keys into
 *    ranges whose float32 partial sums the workspace holds, added in a fixed order.
 *
 *   q, o, d_o   [bh, n_q, head_dim]  dtype, device, read (o and lse as written by fa2_forward)
 *   k, v        [bh, n_k, head_dim]  dtype, device, read
 *   lse         [bh, n_q]            float32, device, read
 *   dq          [bh, n_q, head_dim]  dtype, device, written
 *   dk, dv      [bh, n_k, head_dim]  dtype, device, written
 *   workspace   caller-owned device scratch of at least
 *               fa2_backward_workspace_size(...) bytes, 16-byte aligned; its
 *               contents on entry do not matter; the call overwrites it.
 *
 * dtype BF16 / F16 with head_dim a multiple of 8 in [8, 128]; float32 accumulation.
 * dtype F32 returns FA2_ERR_UNSUPPORTED.
 * Errors: FA2_ERR_INVALID_ARG, FA2_ERR_UNSUPPORTED, FA2_ERR_MISALIGNED,
 *         FA2_ERR_WORKSPACE, FA2_ERR_CUDA.
 */
fa2_status fa2_backward(const void* q, const void* k, const void* v, const void* o, const void* d_o,
                        const float* lse, void* dq, void* dk, void* dv,
                        void* workspace, size_t workspace_bytes,
                        int64_t bh, int64_t n_q, int64_t n_k, int32_t head_dim,
                        fa2_dtype dtype, float softmax_scale, void* stream);

/*
 * The two-pass backward as three stages, callable one by one: the structure of
 * the pages, whose two main passes are separate kernels ("vision-rs 0.1.1
 * flash_attn2.rs", flash_attention2_backward_dq and flash_attention2_backward_dkv).
 * fa2_backward_preprocess followed by fa2_backward_passes (or by _dkdv and _dq, in
 * either order) on one stream gives, bit for bit, what fa2_backward gives for
 * head_dim > 64; for head_dim <= 64 the same gradients without the one-pass
 * kernel's reductions (dq bit-reproducible).  The stages need a workspace of
 * 8 * bh * ceil(n_q / 128) * 128 bytes; fa2_backward_workspace_size bytes also
 * do.  Arguments mean what they mean for fa2_backward; the workspace must be the
 * same buffer across the calls.
 *
 * fa2_backward_preprocess - fills the workspace from o, d_o and lse
 *   (D_i = sum_d O_id dO_id, the row sum both passes subtract).
 * fa2_backward_dkdv - dk and dv from q, k, v, d_o and a filled workspace
 *   (the pass over key tiles).
 * fa2_backward_dq - dq from q, k, v, d_o and a filled workspace (the pass over
 *   query tiles).
 * fa2_backward_passes - dq, dk and dv from a filled workspace: both passes in
 *   one launch, whose CTAs for the two passes share the GPU (what fa2_backward
 *   runs after the preprocess for head_dim > 64).
 * Errors as for fa2_backward.
 */
fa2_status fa2_backward_preprocess(const void* o, const void* d_o, const float* lse, void* workspace,
                                   size_t workspace_bytes, int64_t bh, int64_t n_q, int64_t n_k, int32_t head_dim,
                                   fa2_dtype dtype, void* stream);
fa2_status fa2_backward_dkdv(const void* q, const void* k, const void* v, const void* d_o, const void* workspace,
                             size_t workspace_bytes, void* dk, void* dv, int64_t bh, int64_t n_q, int64_t n_k,
                             int32_t head_dim, fa2_dtype dtype, float softmax_scale, void* stream);
fa2_status fa2_backward_dq(const void* q, const void* k, const void* v, const void* d_o, const void* workspace,
                           size_t workspace_bytes, void* dq, int64_t bh, int64_t n_q, int64_t n_k, int32_t head_dim,
                           fa2_dtype dtype, float softmax_scale, void* stream);
fa2_status fa2_backward_passes(const void* q, const void* k, const void* v, const void* d_o, const void* workspace,
                               size_t workspace_bytes, void* dq, void* dk, void* dv, int64_t bh, int64_t n_q,
                               int64_t n_k, int32_t head_dim, fa2_dtype dtype, float softmax_scale, void* stream);

/*
 * fa2_backward_noalloc - fa2_backward without a caller-supplied workspace and
 * without allocating any device memory.
 *
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory at call time - code whose device memory belongs
 * to a host framework's pool (a raw cudaMalloc would bypass its accounting) and
 * services that fix their memory budget at start-up and must not allocate, or
 * risk running out of memory, while serving.  Arguments and results are those
 * of fa2_backward minus the workspace; the caller still passes every input and
 * output.  The workspace comes from one fixed 8 MiB device array inside the
 * library (reserved on each GPU that loads the library until the process
 * exits).  Problems whose fa2_backward_workspace_size fits in it run as
 * fa2_backward runs them; others run the two-pass stages, which need 8 bytes
 * per padded query row and so cover bh * ceil(n_q / 128) * 128 <= 1,048,576
 * query rows; larger problems return FA2_ERR_SCRATCH_LIMIT and launch nothing.
 * The first call on a device looks up that array's device address, with the
 * device current; make that first call before any stream capture.  All calls
 * share the array, so calls whose GPU work overlaps (several streams or host
 * threads on one device) race on it: serialise them.  Nothing in it needs to
 * start at zero; each call rewrites what it reads.
 * Errors: those of fa2_backward (except FA2_ERR_WORKSPACE), FA2_ERR_SCRATCH_LIMIT.
 */
fa2_status fa2_backward_noalloc(const void* q, const void* k, const void* v, const void* o, const void* d_o,
                                const float* lse, void* dq, void* dk, void* dv,
                                int64_t bh, int64_t n_q, int64_t n_k, int32_t head_dim,
                                fa2_dtype dtype, float softmax_scale, void* stream);

/*
 * psa_pack_qkv - NCHW QKV to the packed [4, B*num_heads, H*W, KEY_DIM] buffer.
 *
 * Defined by "vision_rs/models/yolo/kernels/attention/psa.rs", kernel
 * psa_pack_qkv (same argument order): KEY_DIM = qkv_h / (4 * num_heads) and
 * packed[s, b*num_heads + h, n, dd] = qkv[b, h*4*KEY_DIM + s*KEY_DIM + dd, n]
 * for section s (0 Q, 1 K, 2 V_lo, 3 V_hi) and n = y*W + x.  The memory order
 * is section-major, as in that kernel's store and in FlashAttn2PsaRuntimeOp's
 * pointer arithmetic.
 *
 *   qkv     [B, qkv_h, H, W]              dtype, device, read
 *   packed  [4, B*num_heads, H*W, KEY_DIM] dtype, device, written
 *
 * A pure copy of 2- or 4-byte words: the result is bit-exact for any bit
 * pattern.  qkv_h must be a multiple of 4*num_heads (FA2_ERR_INVALID_ARG).
 */
fa2_status psa_pack_qkv(const void* qkv, void* packed, int32_t qkv_h, int32_t H, int32_t W,
                        int32_t B, int32_t num_heads, fa2_dtype dtype, void* stream);

/*
 * psa_merge_attn_nchw - the two attention outputs (V_lo and V_hi) back to NCHW.
 *
 * Defined by "vision_rs/models/yolo/kernels/attention/psa.rs", kernel
 * psa_merge_attn_nchw: with KEY_DIM = c / (2 * num_heads),
 * out[b, h*2*KEY_DIM + dd, n] = lo[b*num_heads + h, n, dd] and
 * out[b, h*2*KEY_DIM + KEY_DIM + dd, n] = hi[b*num_heads + h, n, dd].
 * The page's kernel takes no B (it comes from its grid); here B is explicit.
 *
 *   lo, hi  [B*num_heads, H*W, KEY_DIM]  dtype, device, read
 *   out     [B, c, H, W]                 dtype, device, written
 *
 * Bit-exact copy.  c must be a multiple of 2*num_heads (FA2_ERR_INVALID_ARG).
 */
fa2_status psa_merge_attn_nchw(const void* lo, const void* hi, void* out, int32_t c, int32_t H,
                               int32_t W, int32_t B, int32_t num_heads, fa2_dtype dtype, void* stream);

/*
 * psa_fa2_forward - both PSA attention calls (V_lo and V_hi) in one pass.
 *
 * Defined by "vision_rs/models/yolo/kernels/attention/psa.rs",
 * FlashAttn2PsaRuntimeOp::new_lo / new_hi: attention with HEAD_DIM = KEY_DIM on
 * Q = section 0, K = section 1 of the packed buffer and V = section 2 (V_lo) or
 * section 3 (V_hi), softmax_scale = 1/sqrt(KEY_DIM) as that op passes it.  The
 * two calls share Q and K, hence their scores, probabilities and LSE; this call
 * computes them once and applies them to both value sections, writing exactly
 * what two fa2_forward calls on (Q, K, V_lo) and (Q, K, V_hi) would write up to
 * rounding order (the module comment's "V split trick", without the second pass).
 *
 *   packed      [4, bh, n, key_dim]   dtype, device, read (as written by psa_pack_qkv)
 *   o_lo, o_hi  [bh, n, key_dim]      dtype, device, written
 *   lse         [bh, n]               float32, device, written (shared by both)
 *
 * dtype F16 / BF16, key_dim a multiple of 8 in [8, 64]; FA2_ERR_UNSUPPORTED otherwise.
 * Errors: FA2_ERR_INVALID_ARG, FA2_ERR_UNSUPPORTED, FA2_ERR_MISALIGNED, FA2_ERR_CUDA.
 */
fa2_status psa_fa2_forward(const void* packed, void* o_lo, void* o_hi, float* lse, int64_t bh, int64_t n,
                           int32_t key_dim, fa2_dtype dtype, float softmax_scale, void* stream);

/*
 * psa_fa2_backward - the backward of both PSA attention calls into d_packed.
 *
 * Defined by "vision_rs/models/yolo/kernels/attention/psa.rs", kernel
 * psa_fa2_backward as FlashAttn2PsaRuntimeOp wires it for the V_lo and V_hi
 * calls: section 0 of d_packed receives dQ_lo + dQ_hi, section 1 dK_lo + dK_hi
 * (the page adds them with atomics), section 2 dV_lo and section 3 dV_hi.
 * The two calls share Q, K, the scores and the probabilities P, so
 * dS = P * (dO_lo V_lo^T + dO_hi V_hi^T - D_lo - D_hi) gives both sums at once;
 * one pass over key tiles (dK, dV_lo, dV_hi) and one over query tiles (dQ),
 * with plain stores: deterministic, no zeroing of d_packed needed.
 *
 *   packed          [4, bh, n, key_dim]  dtype, device, read (Q, K, V_lo, V_hi)
 *   o_lo, o_hi      [bh, n, key_dim]     dtype, device, read (as written by psa_fa2_forward)
 *   d_o_lo, d_o_hi  [bh, n, key_dim]     dtype, device, read (gradients of o_lo, o_hi)
 *   lse             [bh, n]              float32, device, read (from psa_fa2_forward)
 *   d_packed        [4, bh, n, key_dim]  dtype, device, written (every element)
 *   workspace       16-byte aligned, at least 8 * bh * ceil(n / 128) * 128 bytes (D and the
 *                   base-2 LSE of the two-pass stages; fa2_backward_workspace_size bytes also do)
 *
 * dtype F16 / BF16, key_dim a multiple of 8 in [8, 64].  Errors as for fa2_backward.
 */
fa2_status psa_fa2_backward(const void* packed, const void* o_lo, const void* o_hi, const void* d_o_lo,
                            const void* d_o_hi, const float* lse, void* d_packed, void* workspace,
                            size_t workspace_bytes, int64_t bh, int64_t n, int32_t key_dim, fa2_dtype dtype,
                            float softmax_scale, void* stream);

/*
 * psa_extract_v_nchw - the V_lo / V_hi channels of QKV as an NCHW tensor.
 *
 * Defined by "vision_rs/models/yolo/kernels/attention/psa.rs", kernel
 * psa_extract_v_nchw (same argument order, B explicit): with
 * KEY_DIM = qkv_h / (4 * num_heads), v[b, h*2*KEY_DIM + t, n] =
 * qkv[b, h*4*KEY_DIM + 2*KEY_DIM + t, n] for t < 2*KEY_DIM.
 *
 *   qkv  [B, qkv_h, H, W]  dtype, device, read
 *   v    [B, c, H, W]      dtype, device, written; c must equal qkv_h / 2
 *
 * Bit-exact copy.  Errors: FA2_ERR_INVALID_ARG, FA2_ERR_MISALIGNED, FA2_ERR_UNSUPPORTED, FA2_ERR_CUDA.
 */
fa2_status psa_extract_v_nchw(const void* qkv, void* v, int32_t qkv_h, int32_t c, int32_t H, int32_t W,
                              int32_t B, int32_t num_heads, fa2_dtype dtype, void* stream);

/*
 * psa_pack_qkv_backward - the adjoint of psa_pack_qkv: d_packed back to NCHW.
 *
 * "vision_rs/models/yolo/kernels/attention/psa.rs", kernel psa_pack_qkv_backward
 * (same argument order): d_qkv[b, h*4*KEY_DIM + s*KEY_DIM + dd, n] =
 * d_packed[s, b*num_heads + h, n, dd].  The page accumulates with atomics into
 * a zeroed d_qkv because psa_extract_v_backward also adds into the V channels;
 * here this call WRITES every element of d_qkv (no zeroing needed, bit-exact,
 * deterministic) and psa_extract_v_backward, called after it on the same
 * stream, adds its part.
 *
 *   d_packed [4, B*num_heads, H*W, KEY_DIM]  dtype, device, read
 *   d_qkv    [B, qkv_h, H, W]                dtype, device, written
 */
fa2_status psa_pack_qkv_backward(const void* d_packed, void* d_qkv, int32_t qkv_h, int32_t H, int32_t W,
                                 int32_t B, int32_t num_heads, fa2_dtype dtype, void* stream);

/*
 * psa_merge_attn_backward - the adjoint of psa_merge_attn_nchw.
 *
 * "vision_rs/models/yolo/kernels/attention/psa.rs", kernel psa_merge_attn_backward
 * (same argument order, B explicit): d_lo[b*num_heads + h, n, dd] =
 * d_merged[b, h*2*KEY_DIM + dd, n], d_hi[...] = d_merged[b, h*2*KEY_DIM + KEY_DIM + dd, n]
 * with KEY_DIM = c / (2 * num_heads).  Plain stores, bit-exact.
 *
 *   d_merged   [B, c, H, W]                   dtype, device, read
 *   d_lo, d_hi [B*num_heads, H*W, KEY_DIM]    dtype, device, written
 */
fa2_status psa_merge_attn_backward(const void* d_merged, void* d_lo, void* d_hi, int32_t c, int32_t H, int32_t W,
                                   int32_t B, int32_t num_heads, fa2_dtype dtype, void* stream);

/*
 * psa_extract_v_backward - the adjoint of psa_extract_v_nchw, accumulated.
 *
 * "vision_rs/models/yolo/kernels/attention/psa.rs", kernel psa_extract_v_backward
 * (same argument order, B explicit): d_qkv[b, h*4*KEY_DIM + 2*KEY_DIM + t, n] +=
 * d_v[b, h*2*KEY_DIM + t, n] for t < 2*KEY_DIM.  The page uses atomic_add; here
 * each element is read, added in float32 and rounded once (RNE) to dtype, in a
 * single deterministic pass.  Call it after psa_pack_qkv_backward on the same
 * stream.  Other channels of d_qkv are left as they are.
 *
 *   d_v    [B, c, H, W]      dtype, device, read; c must equal qkv_h / 2
 *   d_qkv  [B, qkv_h, H, W]  dtype, device, read and written
 */
fa2_status psa_extract_v_backward(const void* d_v, void* d_qkv, int32_t qkv_h, int32_t c, int32_t H, int32_t W,
                                  int32_t B, int32_t num_heads, fa2_dtype dtype, void* stream);

/*
 * fa2_device_status - the watchdog word of the library's kernels.
 *
 * Every wait of a kernel's threads on an mbarrier (a TMA copy landing, a tensor-core
 * product completing, another warp's signal) is bounded in time: about one second of
 * %globaltimer without progress.  A thread that gives up records it in a device-side
 * word, raises its CTA's abort flag, drains the copies it has in flight and returns;
 * the CTA frees its tensor memory and exits.  This call synchronises `stream`, reads
 * that word on the current device, clears it and returns FA2_OK or
 * FA2_ERR_DEVICE_TIMEOUT (FA2_ERR_CUDA if the synchronisation failed).
 *
 * What this does NOT cover, stated plainly:
 *  - A launch call (fa2_forward, fa2_backward, ...) returns FA2_OK once its kernels
 *    are enqueued.  If a wait later gives up on the device, the outputs of that call
 *    are left partly written (the CTAs that gave up skip their remaining work) while
 *    the launch status stayed FA2_OK: only fa2_device_status reports it.  Callers that
 *    need to know must call it (it synchronises) before trusting the outputs.
 *  - The warp that issues the tensor-core products waits on named barriers
 *    (barrier.sync), which have no time limit.  They complete because every producer
 *    arrives exactly once per event even after a failed wait of its own (the failure
 *    skips work, not arrivals); the bound on the whole kernel therefore rests on the
 *    producers' bounded waits, not on a limit of the issuer's own.
 *  - The limit counts wall-clock time, including time the context spends descheduled
 *    on a shared or time-sliced GPU; a long preemption can trip it with no fault in
 *    the kernel.
 */
fa2_status fa2_device_status(void* stream);

/*
 * fa2_watchdog_selftest - drives the bounded-wait path on purpose.
 *
 * Launches one thread on `stream` that waits on a shared-memory barrier no one
 * will complete, with the same time-bounded wait the pipeline kernels use.  The
 * wait gives up after about one second, records the timeout in the watchdog
 * word and returns; nothing faults or hangs.  A following fa2_device_status()
 * returns FA2_ERR_DEVICE_TIMEOUT (and clears the word).  For tests of the
 * failure-detection path; the pages have no counterpart (their invalid-size
 * path is a trap program, which this library never emits on a device).
 * Errors: FA2_ERR_CUDA if the launch fails.
 */
fa2_status fa2_watchdog_selftest(void* stream);

/*
 * fa2_last_launch_info - which kernels the calling host thread's most recent calls
 * launched, as the sizes and this device decided (cluster sizes after the residency
 * check included).  Each field is written by the calls named beside it, when their
 * arguments were valid, and keeps its value otherwise; all are 0 before any such call.
 *   fwd_key_ranges         fa2_forward, psa_fa2_forward: CTAs of a thread-block cluster
 *                          splitting each 256-row query block's keys (1: no split)
 *   bwd_one_pass           fa2_backward (and _noalloc, and the stage entry points, which
 *                          set 0): 1 if the one-pass kernel ran
 *   bwd_dkv_query_ranges   the same calls: CTAs of a cluster splitting each key tile's
 *                          queries in the dK/dV pass (1: no split, or no dK/dV stage)
 *   bwd_dq_key_ranges      the same calls: key ranges of the dQ pass's float32 partial
 *                          sums (1: no split, or no dQ stage)
 *   bwd_key_tiles_per_cta  the same calls: key tiles per dK/dV CTA of the kernel running
 *                          both passes in one grid (0: that kernel did not run)
 * The record is per host thread and describes enqueued work, not completed work.
 * Errors: FA2_ERR_INVALID_ARG (info is NULL).
 */
typedef struct fa2_launch_info {
    int32_t fwd_key_ranges;
    int32_t bwd_one_pass;
    int32_t bwd_dkv_query_ranges;
    int32_t bwd_dq_key_ranges;
    int32_t bwd_key_tiles_per_cta;
} fa2_launch_info;
fa2_status fa2_last_launch_info(fa2_launch_info* info);

/* fa2_status_string - a static, human-readable message for a status code. */
const char* fa2_status_string(fa2_status s);

#ifdef __cplusplus
}
#endif

#endif /* FA2_GB300_H */
