// fa2_fwd_f32.cu - float32 attention forward on the CUDA cores.
//
// "vision-rs 0.1.1 flash_attn2.rs", flash_attention2_forward, in float32: the
// per-key online-softmax recurrence m' = max(m, s), alpha = exp(m - m'),
// p = exp(s - m'), l = alpha*l + p, acc = alpha*acc + p*v, then O = acc / l and
// LSE = m + ln l.  One warp per query row (lane i holds head-dim elements
// i, i+32, ...); the CTA's eight rows share K/V tiles staged in shared memory.
// Tensor cores are not used: their float32 path (tf32) would not meet a 1e-4
// error bound.  Meant for small problems.
#include "common.cuh"
#include "internal.h"

namespace fa2 {
namespace {

constexpr int kRows = 8;      // query rows (warps) per CTA
constexpr int kKeyTile = 32;  // keys per shared-memory tile

template <int D>
__global__ void __launch_bounds__(kRows * 32)
    fa2_fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
                       float* __restrict__ o, float* __restrict__ lse, int n_q, int n_k, int d_act, float scale) {
    constexpr int E = D / 32;  // elements per lane
    __shared__ float ks[kKeyTile][D];
    __shared__ float vs[kKeyTile][D];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int bh = blockIdx.y;
    const int row = blockIdx.x * kRows + warp;
    const bool active = row < n_q;

    float qr[E], acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        // elements past the true head dimension d_act <= D are zero
        const bool in = active && lane + 32 * e < d_act;
        qr[e] = in ? q[((size_t)bh * n_q + row) * d_act + lane + 32 * e] : 0.f;
        acc[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const float* kb = k + (size_t)bh * n_k * d_act;
    const float* vb = v + (size_t)bh * n_k * d_act;
    for (int j0 = 0; j0 < n_k; j0 += kKeyTile) {
        const int nt = min(kKeyTile, n_k - j0);
        __syncthreads();
        for (int i = threadIdx.x; i < nt * D; i += blockDim.x) {
            const int r = i / D, cidx = i % D;
            const bool in = cidx < d_act;
            ks[r][cidx] = in ? kb[(size_t)(j0 + r) * d_act + cidx] : 0.f;
            vs[r][cidx] = in ? vb[(size_t)(j0 + r) * d_act + cidx] : 0.f;
        }
        __syncthreads();
        for (int j = 0; j < nt; ++j) {
            float dot = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) dot = fmaf(qr[e], ks[j][lane + 32 * e], dot);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
            const float s = dot * scale;
            const float m_new = fmaxf(m, s);
            const float alpha = expf(m - m_new);
            const float p = expf(s - m_new);
            l = alpha * l + p;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = fmaf(p, vs[j][lane + 32 * e], alpha * acc[e]);
            m = m_new;
        }
    }
    if (active) {
#pragma unroll
        for (int e = 0; e < E; ++e)
            if (lane + 32 * e < d_act) o[((size_t)bh * n_q + row) * d_act + lane + 32 * e] = acc[e] / l;
        if (lane == 0) lse[(size_t)bh * n_q + row] = m + logf(l);
    }
}

template <int D>
cudaError_t launch_impl(const FwdParams& p, cudaStream_t stream) {
    const dim3 grid((unsigned)((p.n_q + kRows - 1) / kRows), (unsigned)p.bh, 1);
    fa2_fwd_f32_kernel<D><<<grid, kRows * 32, 0, stream>>>(static_cast<const float*>(p.q), static_cast<const float*>(p.k),
                                                          static_cast<const float*>(p.v), static_cast<float*>(p.o), p.lse,
                                                          (int)p.n_q, (int)p.n_k, p.d, p.scale);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_f32(const FwdParams& p, cudaStream_t stream) {
    switch (pad_head_dim(p.d)) {
        case 32: return launch_impl<32>(p, stream);
        case 64: return launch_impl<64>(p, stream);
        case 128: return launch_impl<128>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa2
