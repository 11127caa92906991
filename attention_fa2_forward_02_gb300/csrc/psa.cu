// psa.cu - the PSA (YOLO C2PSA) rearrangement passes and their adjoints.
//
// "vision_rs/models/yolo/kernels/attention/psa.rs":
//   psa_pack_qkv:           packed[s, b*nh + h, n, dd] = qkv[b, h*4*KD + s*KD + dd, n]
//   psa_merge_attn_nchw:    out[b, h*2*KD + dd, n] = lo[b*nh + h, n, dd],
//                           out[b, h*2*KD + KD + dd, n] = hi[b*nh + h, n, dd]
//   psa_extract_v_nchw:     v[b, h*2*KD + t, n] = qkv[b, h*4*KD + 2*KD + t, n], t < 2*KD
//   psa_merge_attn_backward, psa_pack_qkv_backward: the same index maps read the
//                           other way round (plain stores: no two writes overlap)
//   psa_extract_v_backward: d_qkv[b, h*4*KD + 2*KD + t, n] += d_v[b, h*2*KD + t, n]
// pack / merge and their adjoints are batches of 2-D transposes between a
// channel-major block [KD, N] (NCHW, positions contiguous) and a token-major
// block [N, KD].  The page's kernels read or write with a stride of H*W
// elements; here each CTA stages a tile in shared memory so that both the
// global reads and the global writes are contiguous 16-byte vectors.  The V
// extraction and its adjoint move contiguous runs of 2*KD*N elements per head.
// Copies move words without interpreting them (any bit pattern survives); the
// accumulating adjoint adds in float32 and rounds once to the storage type.
#include <atomic>
#include "common.cuh"
#include "internal.h"

namespace fa2 {
namespace {

constexpr int kThreads = 256;

// Block z of a transpose: which source / destination buffer and the element
// offsets of the block in them.
struct BlockRef {
    int64_t src_off, dst_off;
    int src_sel, dst_sel;
};

// channel-major [KD, N] -> token-major [N, KD]
struct PackMap {  // qkv -> packed, z = (s, bh)
    int64_t bnh, nh, kd, n, qkv_h;
    __device__ BlockRef operator()(int64_t z) const {
        const int64_t s = z / bnh, bh = z % bnh, b = bh / nh, h = bh % nh;
        return {(b * qkv_h + h * 4 * kd + s * kd) * n, (s * bnh + bh) * n * kd, 0, 0};
    }
};
struct MergeBwdMap {  // d_merged -> d_lo / d_hi, z = (half, bh)
    int64_t bnh, nh, kd, n, c;
    __device__ BlockRef operator()(int64_t z) const {
        const int64_t half = z / bnh, bh = z % bnh, b = bh / nh, h = bh % nh;
        return {(b * c + h * 2 * kd + half * kd) * n, bh * n * kd, 0, (int)half};
    }
};
// token-major [N, KD] -> channel-major [KD, N]
struct MergeMap {  // lo / hi -> out, z = (half, bh)
    int64_t bnh, nh, kd, n, c;
    __device__ BlockRef operator()(int64_t z) const {
        const int64_t half = z / bnh, bh = z % bnh, b = bh / nh, h = bh % nh;
        return {bh * n * kd, (b * c + h * 2 * kd + half * kd) * n, (int)half, 0};
    }
};
struct PackBwdMap {  // d_packed -> d_qkv, z = (s, bh)
    int64_t bnh, nh, kd, n, qkv_h;
    __device__ BlockRef operator()(int64_t z) const {
        const int64_t s = z / bnh, bh = z % bnh, b = bh / nh, h = bh % nh;
        return {(s * bnh + bh) * n * kd, (b * qkv_h + h * 4 * kd + s * kd) * n, 0, 0};
    }
};

template <typename W>
struct Vec16 {
    static constexpr int N = 16 / sizeof(W);
};

// Transposes block z: src [R, C] row-major -> dst [C, R] row-major, tile TR x TC.
// kVec: R and C are multiples of the 16-byte vector width and block offsets
// are aligned to it.
template <typename W, int TR, int TC, bool kVec, typename Map>
__global__ void __launch_bounds__(kThreads)
    psa_transpose_kernel(const W* __restrict__ src0, const W* __restrict__ src1, W* __restrict__ dst0,
                         W* __restrict__ dst1, int64_t R, int64_t C, Map map) {
    constexpr int V = kVec ? Vec16<W>::N : 1;
    __shared__ __align__(16) W tile[TR][TC + Vec16<W>::N];
    const BlockRef blk = map((int64_t)blockIdx.z);
    const W* src = (blk.src_sel ? src1 : src0) + blk.src_off;
    W* out = (blk.dst_sel ? dst1 : dst0) + blk.dst_off;
    const int64_t r0 = (int64_t)blockIdx.y * TR;
    const int64_t c0 = (int64_t)blockIdx.x * TC;

    // load: rows r0.., contiguous along C
    for (int idx = threadIdx.x; idx < TR * TC / V; idx += kThreads) {
        const int r = idx / (TC / V);
        const int cv = (idx % (TC / V)) * V;
        const int64_t gr = r0 + r, gc = c0 + cv;
        if constexpr (kVec) {
            if (gr < R && gc < C)
                *reinterpret_cast<uint4*>(&tile[r][cv]) = *reinterpret_cast<const uint4*>(src + gr * C + gc);
        } else {
            if (gr < R && gc < C) tile[r][cv] = src[gr * C + gc];
        }
    }
    __syncthreads();
    // store: rows c0.. of dst, contiguous along R
    for (int idx = threadIdx.x; idx < TC * TR / V; idx += kThreads) {
        const int c = idx / (TR / V);
        const int rv = (idx % (TR / V)) * V;
        const int64_t gc = c0 + c, gr = r0 + rv;
        if (gc >= C || gr >= R) continue;
        if constexpr (kVec) {
            union {
                uint4 u;
                W w[Vec16<W>::N];
            } pk;
#pragma unroll
            for (int i = 0; i < V; ++i) pk.w[i] = tile[rv + i][c];
            *reinterpret_cast<uint4*>(out + gc * R + gr) = pk.u;
        } else {
            out[gc * R + gr] = tile[rv][c];
        }
    }
}

// 16-bit data with R and C multiples of 8: each thread moves one 8 x 8 block of
// block z.  It loads the block's 8 rows as 16-byte vectors, transposes it in
// registers - word m of output row j pairs elements (2m, j) and (2m + 1, j), one
// byte permute per word - and stores 8 vectors along R.  No shared memory, no bank
// conflicts, 8 loads in flight.  Neighbouring lanes take neighbouring blocks along
// the dimension with fewer blocks (kRowFast: along R), so that both sides are
// contiguous runs: the loads of a row, and the stores of a destination row.
template <typename Map, bool kRowFast>
__global__ void __launch_bounds__(kThreads)
    psa_transpose8_kernel(const uint16_t* __restrict__ src0, const uint16_t* __restrict__ src1,
                          uint16_t* __restrict__ dst0, uint16_t* __restrict__ dst1, int64_t R, int64_t C,
                          int64_t batches, Map map) {
    const int64_t rb_n = R / 8, cb_n = C / 8, blocks = rb_n * cb_n;
    const int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (t >= batches * blocks) return;
    const int64_t z = t / blocks, rem = t % blocks;
    const int64_t rb = kRowFast ? rem % rb_n : rem / cb_n, cb = kRowFast ? rem / rb_n : rem % cb_n;
    const BlockRef blk = map(z);
    const uint16_t* src = (blk.src_sel ? src1 : src0) + blk.src_off + (rb * 8) * C + cb * 8;
    uint16_t* out = (blk.dst_sel ? dst1 : dst0) + blk.dst_off + (cb * 8) * R + rb * 8;
    uint32_t w[8][4];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + k * C);
        w[k][0] = v.x;
        w[k][1] = v.y;
        w[k][2] = v.z;
        w[k][3] = v.w;
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t lo[4], hi[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            lo[m] = __byte_perm(w[2 * m][p], w[2 * m + 1][p], 0x5410);  // elements (2m, 2p), (2m+1, 2p)
            hi[m] = __byte_perm(w[2 * m][p], w[2 * m + 1][p], 0x7632);  // elements (2m, 2p+1), (2m+1, 2p+1)
        }
        *reinterpret_cast<uint4*>(out + (2 * p) * R) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        *reinterpret_cast<uint4*>(out + (2 * p + 1) * R) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    }
}

// SMs of the current device, looked up once per device (0 if the query fails).
inline int sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int sms = cache[dev].load(std::memory_order_relaxed);
    if (sms == 0 && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
        cache[dev].store(sms, std::memory_order_relaxed);
    return sms;
}

template <typename W, int TR, int TC, typename Map>
cudaError_t launch_t(const PsaParams& p, int64_t R, int64_t C, int64_t batches, Map map, bool vec, cudaStream_t stream) {
    const dim3 grid((unsigned)((C + TC - 1) / TC), (unsigned)((R + TR - 1) / TR), (unsigned)batches);
    const W* s0 = static_cast<const W*>(p.src0);
    const W* s1 = static_cast<const W*>(p.src1 ? p.src1 : p.src0);
    W* d0 = static_cast<W*>(p.dst);
    W* d1 = static_cast<W*>(p.dst1 ? p.dst1 : p.dst);
    if constexpr (sizeof(W) == 2) {
        // One thread per 64 elements: worth it only while the grid still gives every SM
        // several blocks; smaller tensors keep the tiled kernel's finer grid.
        const bool fills = batches * (R / 8) * (C / 8) >= (int64_t)4 * sm_count() * kThreads;
        if (vec && R % 8 == 0 && C % 8 == 0 && fills) {
            const int64_t threads = batches * (R / 8) * (C / 8);
            const unsigned grid = (unsigned)((threads + kThreads - 1) / kThreads);
            if (R < C)
                psa_transpose8_kernel<Map, true><<<grid, kThreads, 0, stream>>>(s0, s1, d0, d1, R, C, batches, map);
            else
                psa_transpose8_kernel<Map, false><<<grid, kThreads, 0, stream>>>(s0, s1, d0, d1, R, C, batches, map);
            return cudaGetLastError();
        }
    }
    if (vec)
        psa_transpose_kernel<W, TR, TC, true, Map><<<grid, kThreads, 0, stream>>>(s0, s1, d0, d1, R, C, map);
    else
        psa_transpose_kernel<W, TR, TC, false, Map><<<grid, kThreads, 0, stream>>>(s0, s1, d0, d1, R, C, map);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- V extraction and its adjoint
//
// Per head the V_lo and V_hi channels of QKV (channels h*4*KD + 2*KD .. h*4*KD + 4*KD)
// and of V (h*2*KD .. h*2*KD + 2*KD) are contiguous runs of len = 2*KD*N elements.

template <typename W>
__device__ __forceinline__ float widen(W x, int dtype) {
    if constexpr (sizeof(W) == 4) {
        return __uint_as_float(x);
    } else {
        if (dtype == kBf16) return __uint_as_float(((uint32_t)x) << 16);
        return __half2float(__ushort_as_half(x));
    }
}

template <typename W>
__device__ __forceinline__ W narrow(float x, int dtype) {
    if constexpr (sizeof(W) == 4) {
        return __float_as_uint(x);
    } else {
        if (dtype == kBf16) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
        return __half_as_ushort(__float2half_rn(x));
    }
}

// kAdd = false: qkv (src) -> v (dst) copy.  kAdd = true: d_qkv (dst) += d_v (src).
template <typename W, bool kAdd, bool kVec>
__global__ void __launch_bounds__(kThreads)
    psa_v_runs_kernel(const W* __restrict__ src, W* __restrict__ dst, int64_t len, int64_t nh, int64_t kd, int64_t n,
                      int64_t qkv_h, int64_t c, int dtype) {
    constexpr int V = kVec ? Vec16<W>::N : 1;
    const int64_t bh = blockIdx.y, b = bh / nh, h = bh % nh;
    const int64_t qkv_off = (b * qkv_h + h * 4 * kd + 2 * kd) * n;
    const int64_t v_off = (b * c + h * 2 * kd) * n;
    const W* s = src + (kAdd ? v_off : qkv_off);
    W* d = dst + (kAdd ? qkv_off : v_off);
    for (int64_t i = ((int64_t)blockIdx.x * kThreads + threadIdx.x) * V; i < len; i += (int64_t)gridDim.x * kThreads * V) {
        if constexpr (kVec) {
            union {
                uint4 u;
                W w[Vec16<W>::N];
            } a;
            a.u = *reinterpret_cast<const uint4*>(s + i);
            if constexpr (kAdd) {
                union {
                    uint4 u;
                    W w[Vec16<W>::N];
                } o;
                o.u = *reinterpret_cast<const uint4*>(d + i);
#pragma unroll
                for (int t = 0; t < V; ++t) o.w[t] = narrow<W>(widen<W>(o.w[t], dtype) + widen<W>(a.w[t], dtype), dtype);
                *reinterpret_cast<uint4*>(d + i) = o.u;
            } else {
                *reinterpret_cast<uint4*>(d + i) = a.u;
            }
        } else {
            if constexpr (kAdd)
                d[i] = narrow<W>(widen<W>(d[i], dtype) + widen<W>(s[i], dtype), dtype);
            else
                d[i] = s[i];
        }
    }
}

template <typename W>
cudaError_t launch_v_runs(const PsaParams& p, bool add, cudaStream_t stream) {
    constexpr int V = Vec16<W>::N;
    const int64_t len = 2 * p.kd * p.n;
    const bool vec = (p.kd % V == 0) || (p.n % V == 0);
    const int64_t per_block = (int64_t)kThreads * (vec ? V : 1);
    const unsigned gx = (unsigned)std::min<int64_t>((len + per_block - 1) / per_block, 1024);
    const dim3 grid(gx, (unsigned)(p.B * p.nh), 1);
    const W* s = static_cast<const W*>(p.src0);
    W* d = static_cast<W*>(p.dst);
#define FA2_V_RUNS(ADD, VEC) \
    psa_v_runs_kernel<W, ADD, VEC><<<grid, kThreads, 0, stream>>>(s, d, len, p.nh, p.kd, p.n, p.qkv_h, p.c, p.dtype)
    if (add) {
        if (vec) FA2_V_RUNS(true, true); else FA2_V_RUNS(true, false);
    } else {
        if (vec) FA2_V_RUNS(false, true); else FA2_V_RUNS(false, false);
    }
#undef FA2_V_RUNS
    return cudaGetLastError();
}

template <typename W>
cudaError_t launch_w(const PsaParams& p, cudaStream_t stream) {
    constexpr int V = Vec16<W>::N;
    const bool vec = (p.kd % V == 0) && (p.n % V == 0);
    const int64_t bnh = p.B * p.nh;
    switch (p.kind) {
        case kPsaPack:  // block [KD channels, N positions] -> [N, KD]
            return launch_t<W, 32, 64>(p, p.kd, p.n, 4 * bnh, PackMap{bnh, p.nh, p.kd, p.n, p.qkv_h}, vec, stream);
        case kPsaMergeBwd:
            return launch_t<W, 32, 64>(p, p.kd, p.n, 2 * bnh, MergeBwdMap{bnh, p.nh, p.kd, p.n, p.c}, vec, stream);
        case kPsaMerge:  // block [N positions, KD] -> [KD channels, N]
            return launch_t<W, 64, 32>(p, p.n, p.kd, 2 * bnh, MergeMap{bnh, p.nh, p.kd, p.n, p.c}, vec, stream);
        case kPsaPackBwd:
            return launch_t<W, 64, 32>(p, p.n, p.kd, 4 * bnh, PackBwdMap{bnh, p.nh, p.kd, p.n, p.qkv_h}, vec, stream);
        case kPsaExtractV:
            return launch_v_runs<W>(p, false, stream);
        case kPsaExtractVBwd:
            return launch_v_runs<W>(p, true, stream);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_psa(const PsaParams& p, cudaStream_t stream) {
    if (p.elem_bytes == 2) return launch_w<uint16_t>(p, stream);
    if (p.elem_bytes == 4) return launch_w<uint32_t>(p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa2
