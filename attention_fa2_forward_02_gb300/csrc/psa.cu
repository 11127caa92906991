// psa.cu - the PSA (YOLO C2PSA) rearrangement passes as coalesced tiled transposes.
//
// "vision_rs/models/yolo/kernels/attention/psa.rs":
//   psa_pack_qkv:        packed[s, b*nh + h, n, dd] = qkv[b, h*4*KD + s*KD + dd, n]
//   psa_merge_attn_nchw: out[b, h*2*KD + dd, n] = lo[b*nh + h, n, dd],
//                        out[b, h*2*KD + KD + dd, n] = hi[b*nh + h, n, dd]
// Both are batches of 2-D transposes between a channel-major block [KD, N]
// (NCHW, spatial positions contiguous) and a token-major block [N, KD].  The
// page's kernels read (pack) or write (merge) with a stride of H*W elements;
// here each CTA stages a tile in shared memory so that both the global reads
// and the global writes are contiguous 16-byte vectors.  Words are moved, never
// interpreted, so any bit pattern (NaN payloads included) survives unchanged.
#include "common.cuh"
#include "internal.h"

namespace fa2 {
namespace {

constexpr int kThreads = 256;

// Element offsets of block z for the two maps.
struct PackMap {
    int64_t bnh, nh, kd, n, qkv_h;
    __device__ void operator()(int64_t z, int64_t& src_off, int64_t& dst_off, int& which) const {
        const int64_t s = z / bnh, bh = z % bnh, b = bh / nh, h = bh % nh;
        src_off = (b * qkv_h + h * 4 * kd + s * kd) * n;
        dst_off = (s * bnh + bh) * n * kd;
        which = 0;
    }
};
struct MergeMap {
    int64_t bnh, nh, kd, n, c;
    __device__ void operator()(int64_t z, int64_t& src_off, int64_t& dst_off, int& which) const {
        const int64_t half = z / bnh, bh = z % bnh, b = bh / nh, h = bh % nh;
        src_off = bh * n * kd;
        dst_off = (b * c + h * 2 * kd + half * kd) * n;
        which = (int)half;
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
    psa_transpose_kernel(const W* __restrict__ src0, const W* __restrict__ src1, W* __restrict__ dst, int64_t R,
                         int64_t C, Map map) {
    constexpr int V = kVec ? Vec16<W>::N : 1;
    __shared__ __align__(16) W tile[TR][TC + Vec16<W>::N];
    int64_t src_off, dst_off;
    int which;
    map((int64_t)blockIdx.z, src_off, dst_off, which);
    const W* src = (which ? src1 : src0) + src_off;
    W* out = dst + dst_off;
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

template <typename W, int TR, int TC, typename Map>
cudaError_t launch_t(const PsaParams& p, int64_t R, int64_t C, int64_t batches, Map map, bool vec, cudaStream_t stream) {
    const dim3 grid((unsigned)((C + TC - 1) / TC), (unsigned)((R + TR - 1) / TR), (unsigned)batches);
    const W* s0 = static_cast<const W*>(p.src0);
    const W* s1 = static_cast<const W*>(p.src1 ? p.src1 : p.src0);
    W* d = static_cast<W*>(p.dst);
    if (vec)
        psa_transpose_kernel<W, TR, TC, true, Map><<<grid, kThreads, 0, stream>>>(s0, s1, d, R, C, map);
    else
        psa_transpose_kernel<W, TR, TC, false, Map><<<grid, kThreads, 0, stream>>>(s0, s1, d, R, C, map);
    return cudaGetLastError();
}

template <typename W>
cudaError_t launch_w(const PsaParams& p, cudaStream_t stream) {
    constexpr int V = Vec16<W>::N;
    const bool vec = (p.kd % V == 0) && (p.n % V == 0);
    const int64_t bnh = p.B * p.nh;
    if (p.kind == 0) {
        // block [KD channels, N positions] -> [N, KD]
        const PackMap m{bnh, p.nh, p.kd, p.n, p.qkv_h};
        return launch_t<W, 32, 64>(p, p.kd, p.n, 4 * bnh, m, vec, stream);
    }
    // block [N positions, KD] -> [KD channels, N]
    const MergeMap m{bnh, p.nh, p.kd, p.n, p.c};
    return launch_t<W, 64, 32>(p, p.n, p.kd, 2 * bnh, m, vec, stream);
}

}  // namespace

cudaError_t launch_psa(const PsaParams& p, cudaStream_t stream) {
    if (p.elem_bytes == 2) return launch_w<uint16_t>(p, stream);
    if (p.elem_bytes == 4) return launch_w<uint32_t>(p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa2
