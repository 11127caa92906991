// fa2_bwd_tc.cu - attention backward on the sm_103a tensor cores.
//
// What it computes: "vision-rs 0.1.1 flash_attn2.rs", kernels
// flash_attention2_backward_dq and flash_attention2_backward_dkv:
//   D_i = sum_d O_id dO_id,  P_ij = exp(s_ij - LSE_i),  dV_j = sum_i P_ij dO_i,
//   dS_ij = P_ij (dO_i . v_j - D_i),  dQ_i = scale sum_j dS_ij k_j,
//   dK_j = scale sum_i dS_ij q_i.
// Structure as on that page - a pass over key rows for dK/dV and a pass over
// query rows for dQ - at tile granularity, in three launches:
//   1. preprocess: D (float32) and LSE * log2(e), padded per head to a multiple
//      of 128 rows (+inf / 0 in the padding, which makes those rows' P zero);
//   2. dK/dV: one CTA per 128-key tile (keys = TMEM lanes), looping over
//      128-query tiles:  S^T = K Q^T, dP^T = V dO^T, P^T and dS^T elementwise,
//      dV += P^T dO, dK += dS^T Q;
//   3. dQ: one CTA per 128-query tile, looping over 128-key tiles:
//      S = Q K^T, dP = dO V^T, dS elementwise, dQ += dS K.
// In both passes the elementwise work is split in two steps with their own
// barriers so that it overlaps the tensor core (see the MMA orders below).
// The 16-bit P^T / dS^T / dS are written back into tensor memory over the
// score columns they came from and consumed from there by the next MMA.
// Warp roles (320 threads): warp 0 TMA, warp 1 TMEM allocation + MMA issue,
// warps 2-9 elementwise (two warps per TMEM lane quarter).
#include "bwd_common.cuh"
#include "internal.h"

namespace fa2 {
namespace {

// ------------------------------------------------------------------------------ preprocess

// D_i = sum_d O_id dO_id (summed over the (O, dO) pairs when o2 / d_o2 are given).
// With dq_acc given, also zeroes the float32 dQ accumulator of the one-pass
// backward ([bh, n_q_pad, D] floats, D the kernel head size): each thread clears
// the 8 floats of its own row and part, so the grid clears all of it.
template <int D, bool kBf16>
__global__ void __launch_bounds__(256)
    bwd_preprocess_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ d_o,
                          const uint16_t* __restrict__ o2, const uint16_t* __restrict__ d_o2, const float* __restrict__ lse,
                          float* __restrict__ delta, float* __restrict__ lse2, float* __restrict__ dq_acc, int n_q,
                          int n_q_pad, int d_act) {
    constexpr int TPR = D / 8;             // threads per row, 8 elements (16 bytes) each
    constexpr int RPC = 256 / TPR;         // rows per CTA
    const int bh = blockIdx.y;
    const int r = blockIdx.x * RPC + threadIdx.x / TPR;
    const int part = threadIdx.x % TPR;
    if (dq_acc && r < n_q_pad) {
        float4* z = reinterpret_cast<float4*>(dq_acc + ((size_t)bh * n_q_pad + r) * D + part * 8);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float acc = 0.f;
    if (r < n_q && part * 8 < d_act) {  // rows of d_act <= D elements
        const size_t off = ((size_t)bh * n_q + r) * d_act + part * 8;
        for (int pair = 0; pair < (o2 ? 2 : 1); ++pair) {
            const uint4 a = *reinterpret_cast<const uint4*>((pair ? o2 : o) + off);
            const uint4 b = *reinterpret_cast<const uint4*>((pair ? d_o2 : d_o) + off);
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
            const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float2 fa, fb;
                if constexpr (kBf16) {
                    fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[i]));
                    fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bw[i]));
                } else {
                    fa = __half22float2(*reinterpret_cast<const __half2*>(&aw[i]));
                    fb = __half22float2(*reinterpret_cast<const __half2*>(&bw[i]));
                }
                acc = fmaf(fa.x, fb.x, acc);
                acc = fmaf(fa.y, fb.y, acc);
            }
        }
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, TPR);
    if (part == 0 && r < n_q_pad) {
        const size_t w = (size_t)bh * n_q_pad + r;
        // stored negated: the passes add them (-inf in the padding rows makes their P zero)
        delta[w] = r < n_q ? -acc : 0.f;
        lse2[w] = r < n_q ? -lse[(size_t)bh * n_q + r] * kLog2e : -INFINITY;
    }
}

// ------------------------------------------------------------------------------ shared pieces

// kNV = number of (V, dO) pairs sharing the probabilities: 1 (plain attention) or
// 2 (the PSA V_lo / V_hi pair: dP = dO_lo V_lo^T + dO_hi V_hi^T, one dV per pair).
template <int D, int kNV>
struct BwdCfg : Tile16<D> {
    static constexpr int kStages = D == 128 ? 2 : (D == 64 ? 3 : 4);
    static constexpr int kTile = BT * D * 2;
    static_assert(256 + (kNV + 1) * D <= (int)kBwdTmemCols, "tensor memory budget");
    // dK/dV kernel: K, V (and V2) resident; per stage Q_i, dO_i (and dO2_i), lse2_i, delta_i
    static constexpr int kStageDkv = (1 + kNV) * kTile + 2 * BT * 4;
    static constexpr int kDkvOut = (1 + kNV) * kTile + kStages * kStageDkv;  // the warps' output slabs
    static constexpr int kDkvBar = kDkvOut + kOutStageBytes;
    // dQ kernel: Q, dO (and dO2) live in tensor memory (copied once per CTA); per
    // stage K_j, V_j (and V2_j) in shared memory
    static constexpr int kStagesDq = D == 128 ? 3 : 4;
    static constexpr int kStageDq = (1 + kNV) * kTile;
    static constexpr int kDqOut = kStagesDq * kStageDq;  // the warps' output slabs
    static constexpr int kDqBar = kDqOut + kOutStageBytes;
    static constexpr int kQCol = 256 + D;                              // Q as 16-bit pairs: D/2 columns
    static constexpr int kDoCol = 256 + D + D / 2;                     // dO (then dO2): D/2 columns each
    static_assert(kDoCol + kNV * D / 2 <= (int)kBwdTmemCols, "tensor memory budget of the dQ pass");
    static constexpr int kNumBars = 2 * (kStagesDq > kStages ? kStagesDq : kStages) + kBwdBars;
    static constexpr int kSmemDkv = kDkvBar + kNumBars * 8 + 16 + 1024;
    static constexpr int kSmemDq = kDqBar + kNumBars * 8 + 16 + 1024;
    static_assert(kSmemDkv <= 227 * 1024 && kSmemDq <= 227 * 1024, "shared memory budget");
    static_assert(kStageDkv % 1024 == 0 && kDkvOut % 1024 == 0 && kDqOut % 1024 == 0, "stage alignment");
    // One value tensor: the MMA issuer waits only on named barriers, fed by the
    // elementwise warps and by a relay warp (warp 10) that waits for the TMA stages; a
    // shared-memory access (an mbarrier test included) by the issuing warp between MMA
    // groups costs a few hundred clocks of tensor-pipe time. The two-value PSA form
    // keeps lane 0 of the issuer waiting on the mbarriers itself.
    static constexpr bool kNamed = kNV == 1;
    static constexpr int kThreads = kNamed ? kBwdThreads + 32 : kBwdThreads;
};

// Named barriers of the issuer (one value tensor): kNbE1 "P^T ready" (dK/dV) / "S read"
// (dQ; first "Q, dO in tensor memory"), kNbE2 "dS ready", 3 + s "stage s loaded" (relay).
__host__ __device__ constexpr uint32_t nb_stage(int s) { return 3 + (uint32_t)s; }

// ------------------------------------------------------------------------------ dK / dV
//
// MMA order per query tile i (one thread issues, the tensor core executes in order):
//   S^T(i) -> s_full, dP^T(i) -> dp_full, [e1(i)] dV += P^T(i) dO(i),
//   S^T(i+1) -> s_full, [e2(i)] dK += dS^T(i) Q(i) -> empty, dP^T(i+1) -> dp_full, ...
// so P^T(i) is computed while dP^T(i) runs, dS^T(i) while dV(i) and S^T(i+1) run.
// S^T(i+1) overwrites the columns holding P^T(i) only after dV(i), which reads
// them, was issued; dP^T(i+1) likewise follows dK(i).

// One CTA of the dK/dV pass: key tiles kt, kt + 1, ..., kt + n_items - 1 of head bh,
// one after another (n_items > 1 with one value tensor only). Steps run over
// g = u * n_qt + i (key tile u of the CTA, query tile i), so the stage ring and its
// barriers carry on from one key tile to the next; the next tile's K and V load as soon
// as the products reading the current ones have completed (kv_free, during the
// current tile's last query tiles), and its first S^T and dP^T are issued while the
// elementwise warps write the current tile's dK and dV. The tensor maps are the
// kernel's own __grid_constant__ parameters (TMA reads them from parameter space).
//
// kSplitQ: one key tile (n_items = 1) over one of `splits` query ranges, the CTAs of the
// ranges in one thread-block cluster (consecutive blockIdx.x, blockIdx.x mod splits the
// rank; range r = query tiles [floor(r n_qt / splits), floor((r + 1) n_qt / splits)), never
// empty while n_qt >= splits, which the launch ensures with at least 8 per range). Each
// ends with its range's share of dK and dV in tensor memory; every CTA then sends each
// CTA the columns that CTA writes, through distributed shared memory in the buffers its
// loops no longer use, and each adds the shares of its columns in rank order and stores
// them.
template <int D, bool kBf16, int kNV, bool kSplitQ = false>
__device__ __forceinline__ void dkdv_cta(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                         const CUtensorMap& tm_do, const CUtensorMap& tm_v2, const CUtensorMap& tm_do2,
                                         const CUtensorMap& tm_dk, const CUtensorMap& tm_dv, const float* __restrict__ lse2, const float* __restrict__ delta,
                                         void* __restrict__ dk, void* __restrict__ dv, void* __restrict__ dv2, int n_q,
                                         int n_k, int n_q_pad, int d_act, float scale, float scale_log2,
                                         unsigned int* status, int kt, int n_items, int bh, int splits = 1) {
    using C = BwdCfg<D, kNV>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_addr);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int n_qt = (n_q + BT - 1) / BT, q_lo = 0, rank = 0;  // query tiles [q_lo, q_lo + n_qt)
    if constexpr (kSplitQ) {
        static_assert(kNV == 1, "split query ranges with one value tensor");
        rank = (int)(blockIdx.x % (unsigned)splits);
        const int all = n_qt;  // balanced ranges: none empty while all >= splits (the launch takes >= 8 per range)
        q_lo = (int)((int64_t)rank * all / splits);
        n_qt = (int)((int64_t)(rank + 1) * all / splits) - q_lo;
        n_items = n_qt > 0 ? 1 : 0;  // an empty range would only meet the cluster's barriers
    }
    if constexpr (!C::kNamed) n_items = 1;
    bool elem_ok = false;  // an elementwise thread's state at the end, for the split's combine

    const Bars bars{base + C::kDkvBar, S};
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kDkvBar + C::kNumBars * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kDkvBar + C::kNumBars * 8 + 4);
    const Watchdog wd{abort_flag, status};
    const uint32_t k_smem = base;
    auto v_smem = [&](int v) { return base + (1 + v) * C::kTile; };  // V, V2 resident after K
    auto stage_q = [&](int s) { return base + (1 + kNV) * C::kTile + s * C::kStageDkv; };
    auto stage_do = [&](int s, int v) { return stage_q(s) + (1 + v) * C::kTile; };
    auto stage_l2 = [&](int s) { return stage_q(s) + (1 + kNV) * C::kTile; };
    auto stage_dl = [&](int s) { return stage_l2(s) + BT * 4; };

    if (threadIdx.x == 0) init_bars(bars, abort_flag, 1);
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), kBwdTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_do);
            int issued = 0, armed = 0;  // stage fills issued (steps), K / V fills armed (key tiles)
            bool ok = true;
            for (int u = 0; ok && u < n_items; ++u) {
                // K and V of key tile u, once the products reading the previous ones have completed
                if (u > 0 && !(ok = mbar_wait(bars.kv_free(), (u - 1) & 1, wd))) break;
                const int k0 = (kt + u) * BT;
                mbar_arrive_expect_tx(bars.resident(), (1 + kNV) * C::kTile);
                for (int a = 0; a < C::kAtoms; ++a) {
                    tma_load_3d(k_smem + a * BT * C::kAtomRowBytes, &tm_k, bars.resident(), a * C::kAtomCols, k0, bh);
                    for (int v = 0; v < kNV; ++v)
                        tma_load_3d(v_smem(v) + a * BT * C::kAtomRowBytes, v ? &tm_v2 : &tm_v, bars.resident(),
                                    a * C::kAtomCols, k0, bh);
                }
                armed = u + 1;
                for (int i = 0; i < n_qt; ++i) {
                    const int g = u * n_qt + i, s = g % S;
                    if (g >= S && !(ok = mbar_wait(bars.empty(s), ((g / S) & 1) ^ 1, wd))) break;
                    mbar_arrive_expect_tx(bars.full(s), (1 + kNV) * C::kTile + 2 * BT * 4);
                    for (int a = 0; a < C::kAtoms; ++a) {
                        tma_load_3d(stage_q(s) + a * BT * C::kAtomRowBytes, &tm_q, bars.full(s), a * C::kAtomCols,
                                    (q_lo + i) * BT, bh);
                        for (int v = 0; v < kNV; ++v)
                            tma_load_3d(stage_do(s, v) + a * BT * C::kAtomRowBytes, v ? &tm_do2 : &tm_do, bars.full(s),
                                        a * C::kAtomCols, (q_lo + i) * BT, bh);
                    }
                    const size_t w = (size_t)bh * n_q_pad + (size_t)(q_lo + i) * BT;
                    bulk_load(stage_l2(s), lse2 + w, BT * 4, bars.full(s));
                    bulk_load(stage_dl(s), delta + w, BT * 4, bars.full(s));
                    issued = g + 1;
                }
            }
            if (!ok) {
                if (armed > 0) drain_wait(bars.resident(), (armed - 1) & 1);
                for (int g = (issued > S ? issued - S : 0); g < issued; ++g) drain_wait(bars.full(g % S), (g / S) & 1);
            }
        }
    } else if (warp == 1) {
        if constexpr (C::kNamed) {
            const uint32_t idesc_s = idesc_f16_f32acc(BT, BT, kBf16, false, false);
            const uint32_t idesc_g = idesc_f16_f32acc(BT, D, kBf16, false, true);
            // Descriptors built once (stage 0, k-step 0); every other operand adds a
            // constant to the start-address field (16-byte units; shared addresses stay
            // below 256 KB). Fewer instructions per MMA keep the issuer, which shares its
            // sub-partition with two elementwise warps, ahead of the tensor pipe.
            const uint64_t dk0 = C::kmajor(k_smem, 0, BT), dv0 = C::kmajor(v_smem(0), 0, BT);
            const uint64_t dq0 = C::kmajor(stage_q(0), 0, BT), ddo0 = C::kmajor(stage_do(0, 0), 0, BT);
            const uint64_t mq0 = C::mnmajor(stage_q(0), 0, BT), mdo0 = C::mnmajor(stage_do(0, 0), 0, BT);
            auto st_off = [&](int s) { return (uint64_t)((s * C::kStageDkv) >> 4); };
            auto issue_st = [&](int s) {  // S^T = K Q^T
                const uint64_t b = dq0 + st_off(s);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t o = (uint64_t)(C::koff(kk, BT) >> 4);
                    mma_ss(tmem, dk0 + o, b + o, idesc_s, kk > 0);
                }
            };
            auto issue_dpt = [&](int s) {  // dP^T = V dO^T
                const uint64_t b = ddo0 + st_off(s);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t o = (uint64_t)(C::koff(kk, BT) >> 4);
                    mma_ss(tmem + 128u, dv0 + o, b + o, idesc_s, kk > 0);
                }
            };
            static_assert(nb_stage(S - 1) < 16, "named barriers");
            for (int u = 0; u < n_items; ++u) {
                const int g0 = u * n_qt;
                const bool next_tile = u + 1 < n_items;
                // S^T(0) overwrites the columns of the previous tile's last P^T only after its
                // dV was issued, dP^T(0) those of its last dS^T after its dK (issue order);
                // dV and dK of this tile restart their accumulators only after the
                // elementwise warps, which read the previous tile's out first, meet at e1.
                nb_sync(nb_stage(g0 % S), 64);  // K, V of key tile u and its first Q / dO stage
                if (lane == 0) {
                    tc_fence_after();
                    issue_st(g0 % S);
                    mma_commit(bars.s_full());
                    issue_dpt(g0 % S);
                    mma_commit(bars.dp_full());
                    if (n_qt == 1 && next_tile) mma_commit(bars.kv_free());  // last readers of K, V issued
                }
                __syncwarp();
                for (int i = 0; i < n_qt; ++i) {
                    const int g = g0 + i;
                    const int s = g % S;
                    const int sn = (g + 1) % S;
                    const bool more = i + 1 < n_qt;
                    nb_sync(kNbE1, kNbElem);  // P^T(i) in tensor memory
                    if (lane == 0) {
                        tc_fence_after();
                        const uint64_t b = mdo0 + st_off(s);
#pragma unroll
                        for (int kk = 0; kk < BT / 16; ++kk)  // dV += P^T dO
                            mma_ts(tmem + 256u, tmem + kPackedCol + (uint32_t)(kk * 8), b + (uint64_t)(kk * C::kAtomRowBytes),
                                   idesc_g, (i > 0 || kk > 0));
                        if (!kSplitQ && !more) mma_commit(bars.dv_done());  // dV of key tile u complete
                    }
                    __syncwarp();
                    if (more) {
                        nb_sync(nb_stage(sn), 64);  // Q, dO of tile i + 1
                        if (lane == 0) {
                            tc_fence_after();
                            issue_st(sn);
                            mma_commit(bars.s_full());
                        }
                        __syncwarp();
                    }
                    nb_sync(kNbE2, kNbElem);  // dS^T(i) in tensor memory
                    if (lane == 0) {
                        tc_fence_after();
                        const uint64_t b = mq0 + st_off(s);
#pragma unroll
                        for (int kk = 0; kk < BT / 16; ++kk)  // dK += dS^T Q
                            mma_ts(tmem + 256u + (uint32_t)D, tmem + 128u + kPackedCol + (uint32_t)(kk * 8),
                                   b + (uint64_t)(kk * C::kAtomRowBytes), idesc_g, (i > 0 || kk > 0));
                        mma_commit(bars.empty(s));
                        if (more) {
                            issue_dpt(sn);
                            mma_commit(bars.dp_full());
                            if (i + 2 == n_qt && next_tile) mma_commit(bars.kv_free());  // last readers of K, V issued
                        }
                    }
                    __syncwarp();
                }
                if (lane == 0) mma_commit(bars.done());  // dV, dK of key tile u complete
                __syncwarp();
            }
            if (lane == 0 && n_items > 0) drain_wait(bars.done(), (uint32_t)((n_items - 1) & 1));
            __syncwarp();
        } else {
            if (lane == 0) {
                const uint32_t idesc_s = idesc_f16_f32acc(BT, BT, kBf16, false, false);
                const uint32_t idesc_g = idesc_f16_f32acc(BT, D, kBf16, false, true);
                auto issue_st = [&](int s) {  // S^T = K Q^T
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(tmem, C::kmajor(k_smem, kk, BT), C::kmajor(stage_q(s), kk, BT), idesc_s, kk > 0);
                };
                auto issue_dpt = [&](int s) {  // dP^T = sum over pairs of V dO^T
#pragma unroll
                    for (int v = 0; v < kNV; ++v)
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_ss(tmem + 128u, C::kmajor(v_smem(v), kk, BT), C::kmajor(stage_do(s, v), kk, BT), idesc_s,
                                   (v > 0 || kk > 0));
                };
                bool ok = mbar_wait(bars.resident(), 0, wd) && mbar_wait(bars.full(0), 0, wd);
                if (ok) {
                    tc_fence_after();
                    issue_st(0);
                    mma_commit(bars.s_full());
                    issue_dpt(0);
                    mma_commit(bars.dp_full());
                }
                for (int i = 0; ok && i < n_qt; ++i) {
                    const int s = i % S;
                    const int sn = (i + 1) % S;
                    const bool more = i + 1 < n_qt;
                    if (!(ok = mbar_wait(bars.e1(), i & 1, wd))) break;
                    tc_fence_after();
#pragma unroll
                    for (int v = 0; v < kNV; ++v)
#pragma unroll
                        for (int kk = 0; kk < BT / 16; ++kk)  // dV += P^T dO (one accumulator per pair)
                            mma_ts(tmem + 256u + (uint32_t)(v * D), tmem + kPackedCol + (uint32_t)(kk * 8),
                                   C::mnmajor(stage_do(s, v), kk, BT), idesc_g, (i > 0 || kk > 0));
                    if (more) {
                        if (!(ok = mbar_wait(bars.full(sn), ((i + 1) / S) & 1, wd))) break;
                        tc_fence_after();
                        issue_st(sn);
                        mma_commit(bars.s_full());
                    }
                    if (!(ok = mbar_wait(bars.e2(), i & 1, wd))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < BT / 16; ++kk)  // dK += dS^T Q
                        mma_ts(tmem + 256u + (uint32_t)(kNV * D), tmem + 128u + kPackedCol + (uint32_t)(kk * 8),
                               C::mnmajor(stage_q(s), kk, BT), idesc_g, (i > 0 || kk > 0));
                    mma_commit(bars.empty(s));
                    if (more) {
                        issue_dpt(sn);
                        mma_commit(bars.dp_full());
                    }
                }
                mma_commit(bars.done());
                drain_wait(bars.done(), 0);
            }
        }
    } else if (C::kNamed && warp == kBwdRelayWarp) {
        // TMA relay: signals each Q / dO stage (each key tile's first with its K and V) to
        // the issuer
        bool ok = true;
        for (int u = 0; u < n_items; ++u)
            for (int i = 0; i < n_qt; ++i) {
                const int g = u * n_qt + i, s = g % S;
                if (i == 0) ok = ok && warp_wait(bars.resident(), u & 1, wd);
                ok = ok && warp_wait(bars.full(s), (g / S) & 1, wd);
                nb_arrive(nb_stage(s), 64);
            }
    } else {
        // Two warps per TMEM lane quarter; warp `half` owns query columns [64*half, 64*half + 64).
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t t_s = tmem + lane_off, t_dp = tmem + lane_off + 128u;
        const uint32_t out_slab = base + C::kDkvOut + (uint32_t)((warp - 2) * kOutSlabBytes);
        const float2 scale2 = make_float2(scale_log2, scale_log2);
        bool ok = true;
        // a failed wait skips the work of this and later tiles, not the signals
        auto signal = [&](uint32_t nb, uint32_t mbar) {
            if constexpr (C::kNamed) nb_arrive(nb, kNbElem);
            else mbar_arrive(mbar);
        };
        // One value tensor, no query split: each accumulator leaves as soon as the products
        // that write it have completed, and before the products that restart it are issued.
        // dV of key tile u (dv_done) right after the tile's last e2, while its last dK
        // product and the next tile's first S^T and dP^T run; dK of key tile u (done) with
        // the next tile's first dS^T, while its first dV and second S^T run. Every warp writes
        // its 32 key rows of the 32-column chunks half, half + 2, ... of each, by TMA stores.
        constexpr bool kOutInLoop = C::kNamed && !kSplitQ;
        auto write_acc = [&](int acc, int tile) {  // acc 0: dV, 1: dK (times scale)
            if (!(ok = ok && warp_wait(acc ? bars.done() : bars.dv_done(), (uint32_t)(tile & 1), wd))) return;
            tc_fence_after();
            const uint32_t src = tmem + lane_off + 256u + (uint32_t)(acc * D);
#pragma unroll
            for (int c = half; c < D / 32; c += 2) {
                uint32_t r[32];
                tmem_ld32(src + 32u * (uint32_t)c, r);
                tmem_ld_wait();
                reg_fence(r);
                store_chunk_tma<kBf16>(acc ? &tm_dk : &tm_dv, out_slab, 32 * c, (kt + tile) * BT + quarter * 32, n_k, d_act,
                                       bh, r, acc ? scale : 1.f);
            }
        };
        for (int u = 0; u < n_items; ++u) {
        for (int i = 0; i < n_qt; ++i) {
            const int g = u * n_qt + i;
            const int s = g % S;
            if (!(ok = ok && warp_wait(bars.s_full(), g & 1, wd) && warp_wait(bars.full(s), (g / S) & 1, wd))) {
                signal(kNbE1, bars.e1());
                signal(kNbE2, bars.e2());
                continue;
            }
            tc_fence_after();
            const float* l2 = reinterpret_cast<const float*>(smem + (stage_l2(s) - base));
            const float* dl = reinterpret_cast<const float*>(smem + (stage_dl(s) - base));
            // step 1: P^T = 2^(S^T * scale * log2e - LSE2) for both owned chunks
            float2 p[2][16];
            {
                uint32_t ra[32], rb[32];
                tmem_ld32(t_s + 32u * owned_chunk(half, 0), ra);
                tmem_ld32(t_s + 32u * owned_chunk(half, 1), rb);
                tmem_ld_wait();
                reg_fence(ra);
                reg_fence(rb);
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int c = owned_chunk(half, cc);
                    const uint32_t* r = cc == 0 ? ra : rb;
                    uint32_t pk[16];
#pragma unroll
                    for (int x = 0; x < 16; x += 2) {
                        const float4 nl = *reinterpret_cast<const float4*>(l2 + 32 * c + 2 * x);  // -LSE2, 4 queries
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            float2 v = __ffma2_rn(make_float2(__uint_as_float(r[2 * (x + u)]), __uint_as_float(r[2 * (x + u) + 1])),
                                                  scale2, u ? make_float2(nl.z, nl.w) : make_float2(nl.x, nl.y));
                            v.x = ex2_approx(v.x);
                            v.y = ex2_approx(v.y);
                            p[cc][x + u] = v;
                            pk[x + u] = pack2<kBf16>(v.x, v.y);
                        }
                    }
                    tmem_st16(t_s + kPackedCol + 16u * c, pk);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            signal(kNbE1, bars.e1());
            // step 2: dS^T = P^T * (dP^T - D), chunk by chunk in write-safe order
            if (!(ok = ok && warp_wait(bars.dp_full(), g & 1, wd))) {
                signal(kNbE2, bars.e2());
                continue;
            }
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c = owned_chunk(half, cc);
                uint32_t rp[32];
                tmem_ld32(t_dp + 32u * c, rp);
                tmem_ld_wait();
                reg_fence(rp);
                uint32_t pk[16];
#pragma unroll
                for (int x = 0; x < 16; x += 2) {
                    const float4 nd = *reinterpret_cast<const float4*>(dl + 32 * c + 2 * x);  // -D, 4 queries
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float2 ds = __fmul2_rn(
                            p[cc][x + u], __fadd2_rn(make_float2(__uint_as_float(rp[2 * (x + u)]), __uint_as_float(rp[2 * (x + u) + 1])),
                                                     u ? make_float2(nd.z, nd.w) : make_float2(nd.x, nd.y)));
                        pk[x + u] = pack2<kBf16>(ds.x, ds.y);
                    }
                }
                tmem_st16(t_dp + kPackedCol + 16u * c, pk);
            }
            tmem_st_wait();
            if constexpr (kOutInLoop)
                if (i == 0 && u > 0) write_acc(1, u - 1);  // read before e2 lets dK(u, 0) restart it
            tc_fence_before();
            signal(kNbE2, bars.e2());
        }
        if constexpr (kOutInLoop) {
            write_acc(0, u);
        } else {
            // the split's share stays in tensor memory for the cluster's combine below; the
            // two-value form stores dK, dV row by row once all its products have completed
            if (ok) ok = warp_wait(bars.done(), (uint32_t)(u & 1), wd);
            if constexpr (kSplitQ) elem_ok = ok;
            else if (ok) {
                tc_fence_after();
                const int key = (kt + u) * BT + quarter * 32 + lane;
                const size_t row = (size_t)bh * n_k + key;
                // half 0 writes dV (each pair's), half 1 writes dK (scaled)
#pragma unroll
                for (int v = 0; v < (half ? 1 : kNV); ++v) {
                    const uint32_t src = tmem + lane_off + 256u + (uint32_t)((half ? kNV : v) * D);
                    void* dst = half ? dk : (v ? dv2 : dv);
                    const float mul = half ? scale : 1.f;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(src + 32u * c, r);
                        tmem_ld_wait();
                        reg_fence(r);
                        store_row_chunk<kBf16>(dst, row, d_act, c, r, mul, key < n_k);
                    }
                }
            }
        }
        }  // key tiles
        if constexpr (kOutInLoop)
            if (n_items > 0) write_acc(1, n_items - 1);
        if (lane == 0) bulk_wait_group0();  // this warp's stores complete before the CTA exits
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (kSplitQ) {
        // Every thread of every CTA of the cluster meets at each of the two barriers. The
        // shares land in [splits][128 rows][dV, dK][w columns] float32 from shared address 0
        // (the K, V and stage buffers, idle once every CTA's loops are over).
        static_assert(128 * 2 * D * 4 <= C::kDkvBar, "split combine buffer");
        const bool elem = warp >= 2 && warp < 10;
        const int quarter = warp & 3, half = (warp - 2) >> 2;  // half 0: dV, half 1: dK
        const int row = quarter * 32 + lane;                   // key row within the tile
        const int w = D / splits;                               // columns this CTA writes: [rank w, rank w + w)
        cluster_sync_all();
        if (elem) {
            tc_fence_after();
            const uint32_t src = tmem + ((uint32_t)(quarter * 32) << 16) + 256u + (uint32_t)(half * D);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(src + 32u * c, r);
                tmem_ld_wait();
                reg_fence(r);
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const int col = 32 * c + 4 * g, owner = col / w;
                    const uint32_t dst = base + (uint32_t)((((rank * 128 + row) * 2 + half) * w + col - owner * w) * 4);
                    // a CTA whose waits failed sends exact zeros (its tensor memory may hold anything)
                    st_cluster_v4(cluster_map(dst, (uint32_t)owner), elem_ok ? __uint_as_float(r[4 * g]) : 0.f,
                                  elem_ok ? __uint_as_float(r[4 * g + 1]) : 0.f, elem_ok ? __uint_as_float(r[4 * g + 2]) : 0.f,
                                  elem_ok ? __uint_as_float(r[4 * g + 3]) : 0.f);
                }
            }
        }
        cluster_sync_all();
        if (elem) {
            const float* part = reinterpret_cast<const float*>(smem);
            const int key = kt * BT + row;
            const float mul = half ? scale : 1.f;
            uint16_t* grow = static_cast<uint16_t*>(half ? dk : dv) + ((size_t)bh * n_k + key) * d_act;
            for (int g = 0; g < w; g += 4) {
                float a[4] = {0.f, 0.f, 0.f, 0.f};
                for (int r = 0; r < splits; ++r)  // in rank order
#pragma unroll
                    for (int i = 0; i < 4; ++i) a[i] += part[((r * 128 + row) * 2 + half) * w + g + i];
                const int col = rank * w + g;  // d_act is a multiple of 8: a 4-column group is all in or all out
                if (key < n_k && col < d_act)
                    *reinterpret_cast<uint2*>(grow + col) =
                        make_uint2(pack2<kBf16>(a[0] * mul, a[1] * mul), pack2<kBf16>(a[2] * mul, a[3] * mul));
            }
        }
        tc_fence_before();
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kBwdTmemCols);
    }
}

// ------------------------------------------------------------------------------ dQ
//
// MMA order per key tile j:
//   S(j) -> s_full, dP(j) -> dp_full, [e1(j): S(j) read] S(j+1) -> s_full,
//   [e2(j)] dQ += dS(j) K(j) -> empty, dP(j+1) -> dp_full, ...
// dS lives in the dP columns, so dP(j+1) follows dQ(j); the S columns hold only
// scores, so S(j+1) needs nothing but the elementwise warps having read S(j).
// Q and dO are the same for every key tile: the elementwise warps copy them once
// into tensor memory (16-bit pairs, the layout an MMA reads its A operand in), so
// S and dP read only K and V from shared memory.

// One CTA of the dQ pass: query tile qt of head bh, over key tiles [j0, j1). With plane < 0
// the CTA covers all key tiles and writes dq; otherwise it writes its float32 partial sum
// (unscaled) to plane `plane` of the split dQ pass's partial sums, through tm_dqp.
template <int D, bool kBf16, int kNV>
__device__ __forceinline__ void dq_cta(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const CUtensorMap& tm_v2,
                                       const CUtensorMap& tm_dq, const uint16_t* __restrict__ q_ptr, const uint16_t* __restrict__ do_ptr,
                                       const uint16_t* __restrict__ do2_ptr, const float* __restrict__ lse2,
                                       const float* __restrict__ delta, void* __restrict__ dq, int n_q, int n_k,
                                       int n_q_pad, int d_act, float scale, float scale_log2, unsigned int* status,
                                       int qt, int bh, const CUtensorMap& tm_dqp, int j0, int j1, int plane) {
    using C = BwdCfg<D, kNV>;
    constexpr int S = C::kStagesDq;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_addr);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q0 = qt * BT;
    const int nj = j1 - j0;  // key tiles of this CTA

    const Bars bars{base + C::kDqBar, S};
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kDqBar + C::kNumBars * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kDqBar + C::kNumBars * 8 + 4);
    const Watchdog wd{abort_flag, status};
    auto stage_k = [&](int s) { return base + s * C::kStageDq; };
    auto stage_v = [&](int s, int v) { return stage_k(s) + (1 + v) * C::kTile; };

    if (threadIdx.x == 0) init_bars(bars, abort_flag, kElemThreads);
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), kBwdTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            if (kNV == 2) prefetch_tmap(&tm_v2);
            int issued = 0;
            bool ok = true;
            for (int j = 0; j < nj; ++j) {
                const int s = j % S;
                if (j >= S && !(ok = mbar_wait(bars.empty(s), ((j / S) & 1) ^ 1, wd))) break;
                mbar_arrive_expect_tx(bars.full(s), (1 + kNV) * C::kTile);
                for (int a = 0; a < C::kAtoms; ++a) {
                    tma_load_3d(stage_k(s) + a * BT * C::kAtomRowBytes, &tm_k, bars.full(s), a * C::kAtomCols, (j0 + j) * BT, bh);
                    for (int v = 0; v < kNV; ++v)
                        tma_load_3d(stage_v(s, v) + a * BT * C::kAtomRowBytes, v ? &tm_v2 : &tm_v, bars.full(s),
                                    a * C::kAtomCols, (j0 + j) * BT, bh);
                }
                issued = j + 1;
            }
            if (!ok) {
                for (int j = (issued > S ? issued - S : 0); j < issued; ++j) drain_wait(bars.full(j % S), (j / S) & 1);
            }
        }
    } else if (warp == 1) {
        if constexpr (C::kNamed) {
            const uint32_t idesc_s = idesc_f16_f32acc(BT, BT, kBf16, false, false);
            const uint32_t idesc_g = idesc_f16_f32acc(BT, D, kBf16, false, true);
            // descriptors built once (stage 0, k-step 0), as in the dK/dV pass
            const uint64_t dk0 = C::kmajor(stage_k(0), 0, BT), dv0 = C::kmajor(stage_v(0, 0), 0, BT);
            const uint64_t mk0 = C::mnmajor(stage_k(0), 0, BT);
            auto st_off = [&](int s) { return (uint64_t)((s * C::kStageDq) >> 4); };
            auto issue_s = [&](int s) {  // S = Q K^T, Q from tensor memory
                const uint64_t b = dk0 + st_off(s);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ts(tmem, tmem + (uint32_t)(C::kQCol + kk * 8), b + (uint64_t)(C::koff(kk, BT) >> 4), idesc_s, kk > 0);
            };
            auto issue_dp = [&](int s) {  // dP = dO V^T, dO from tensor memory
                const uint64_t b = dv0 + st_off(s);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ts(tmem + 128u, tmem + (uint32_t)(C::kDoCol + kk * 8), b + (uint64_t)(C::koff(kk, BT) >> 4), idesc_s,
                           kk > 0);
            };
            static_assert(nb_stage(S - 1) < 16, "named barriers");
            nb_sync(kNbE1, kNbElem);   // Q and dO copied into tensor memory
            nb_sync(nb_stage(0), 64);  // the first K / V stage
            if (lane == 0) {
                tc_fence_after();
                issue_s(0);
                mma_commit(bars.s_full());
                issue_dp(0);
                mma_commit(bars.dp_full());
            }
            __syncwarp();
            for (int j = 0; j < nj; ++j) {
                const int s = j % S;
                const int sn = (j + 1) % S;
                const bool more = j + 1 < nj;
                nb_sync(kNbE1, kNbElem);  // S(j) read: its columns may be overwritten
                if (more) {
                    nb_sync(nb_stage(sn), 64);  // K, V of tile j + 1
                    if (lane == 0) {
                        tc_fence_after();
                        issue_s(sn);
                        mma_commit(bars.s_full());
                    }
                    __syncwarp();
                }
                nb_sync(kNbE2, kNbElem);  // dS(j) in tensor memory
                if (lane == 0) {
                    tc_fence_after();
                    const uint64_t b = mk0 + st_off(s);
#pragma unroll
                    for (int kk = 0; kk < BT / 16; ++kk)  // dQ += dS K
                        mma_ts(tmem + 256u, tmem + 128u + kPackedCol + (uint32_t)(kk * 8), b + (uint64_t)(kk * C::kAtomRowBytes),
                               idesc_g, (j > 0 || kk > 0));
                    mma_commit(bars.empty(s));
                    if (more) {
                        issue_dp(sn);
                        mma_commit(bars.dp_full());
                    }
                }
                __syncwarp();
            }
            if (lane == 0) {
                mma_commit(bars.done());
                drain_wait(bars.done(), 0);
            }
            __syncwarp();
        } else {
            if (lane == 0) {
                const uint32_t idesc_s = idesc_f16_f32acc(BT, BT, kBf16, false, false);
                const uint32_t idesc_g = idesc_f16_f32acc(BT, D, kBf16, false, true);
                auto issue_s = [&](int s) {  // S = Q K^T, Q from tensor memory
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ts(tmem, tmem + (uint32_t)(C::kQCol + kk * 8), C::kmajor(stage_k(s), kk, BT), idesc_s, kk > 0);
                };
                auto issue_dp = [&](int s) {  // dP = sum over pairs of dO V^T, dO from tensor memory
#pragma unroll
                    for (int v = 0; v < kNV; ++v)
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_ts(tmem + 128u, tmem + (uint32_t)(C::kDoCol + v * D / 2 + kk * 8),
                                   C::kmajor(stage_v(s, v), kk, BT), idesc_s, (v > 0 || kk > 0));
                };
                bool ok = mbar_wait(bars.resident(), 0, wd) && mbar_wait(bars.full(0), 0, wd);
                if (ok) {
                    tc_fence_after();
                    issue_s(0);
                    mma_commit(bars.s_full());
                    issue_dp(0);
                    mma_commit(bars.dp_full());
                }
                for (int j = 0; ok && j < nj; ++j) {
                    const int s = j % S;
                    const int sn = (j + 1) % S;
                    const bool more = j + 1 < nj;
                    if (more) {
                        if (!(ok = mbar_wait(bars.e1(), j & 1, wd) && mbar_wait(bars.full(sn), ((j + 1) / S) & 1, wd))) break;
                        tc_fence_after();
                        issue_s(sn);
                        mma_commit(bars.s_full());
                    }
                    if (!(ok = mbar_wait(bars.e2(), j & 1, wd))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < BT / 16; ++kk)  // dQ += dS K
                        mma_ts(tmem + 256u, tmem + 128u + kPackedCol + (uint32_t)(kk * 8), C::mnmajor(stage_k(s), kk, BT),
                               idesc_g, (j > 0 || kk > 0));
                    mma_commit(bars.empty(s));
                    if (more) {
                        issue_dp(sn);
                        mma_commit(bars.dp_full());
                    }
                }
                mma_commit(bars.done());
                drain_wait(bars.done(), 0);
            }
        }
    } else if (C::kNamed && warp == kBwdRelayWarp) {
        // TMA relay: signals each K / V stage to the issuer
        bool ok = warp_wait(bars.full(0), 0, wd);
        nb_arrive(nb_stage(0), 64);
        for (int j = 1; j < nj; ++j) {
            const int s = j % S;
            ok = ok && warp_wait(bars.full(s), (j / S) & 1, wd);
            nb_arrive(nb_stage(s), 64);
        }
    } else {
        // Two warps per TMEM lane quarter; warp `half` owns key columns [64*half, 64*half + 64).
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t t_s = tmem + lane_off, t_dp = tmem + lane_off + 128u;
        const int row = q0 + quarter * 32 + lane;
        const size_t w = (size_t)bh * n_q_pad + row;  // row < n_q_pad always
        const float my_nl2 = lse2[w];  // -LSE * log2(e)
        const float my_nd = delta[w];   // -D
        // This thread's row of Q (half 0) or of dO / dO2 (half 1) into tensor memory,
        // zeros past the last query; pairs of 16-bit elements per 32-bit column.
        {
            const bool valid = row < n_q;
            for (int t = 0; t < (half ? kNV : 1); ++t) {
                const uint16_t* src = half ? (t ? do2_ptr : do_ptr) : q_ptr;
                const uint32_t col = half ? (uint32_t)(C::kDoCol + t * D / 2) : (uint32_t)C::kQCol;
                const uint4* rowp = reinterpret_cast<const uint4*>(src + ((size_t)bh * n_q + (valid ? row : 0)) * d_act);
                if constexpr (D >= 64) {
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {
                        uint32_t wv[32];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const uint4 x = (valid && (c * 8 + u) * 8 < d_act) ? rowp[c * 8 + u] : make_uint4(0u, 0u, 0u, 0u);
                            wv[4 * u] = x.x;
                            wv[4 * u + 1] = x.y;
                            wv[4 * u + 2] = x.z;
                            wv[4 * u + 3] = x.w;
                        }
                        tmem_st32(tmem + lane_off + col + 32u * c, wv);
                    }
                } else {
                    uint32_t wv[16];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint4 x = (valid && u * 8 < d_act) ? rowp[u] : make_uint4(0u, 0u, 0u, 0u);
                        wv[4 * u] = x.x;
                        wv[4 * u + 1] = x.y;
                        wv[4 * u + 2] = x.z;
                        wv[4 * u + 3] = x.w;
                    }
                    tmem_st16(tmem + lane_off + col, wv);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            if constexpr (C::kNamed) nb_arrive(kNbE1, kNbElem);
            else mbar_arrive(bars.resident());
        }
        const float2 scale2 = make_float2(scale_log2, scale_log2);
        const float2 neg_l2 = make_float2(my_nl2, my_nl2), neg_d = make_float2(my_nd, my_nd);
        bool ok = true;
        // a failed wait skips the work of this and later tiles, not the signals
        auto signal = [&](uint32_t nb, uint32_t mbar) {
            if constexpr (C::kNamed) nb_arrive(nb, kNbElem);
            else mbar_arrive(mbar);
        };
        for (int j = 0; j < nj; ++j) {
            if (!(ok = ok && warp_wait(bars.s_full(), j & 1, wd))) {
                signal(kNbE1, bars.e1());
                signal(kNbE2, bars.e2());
                continue;
            }
            tc_fence_after();
            const int valid = n_k - (j0 + j) * BT;
            // step 1: P = 2^(S * scale * log2e - LSE2) in registers; then S may be overwritten
            float2 p[2][16];
            {
                uint32_t ra[32], rb[32];
                tmem_ld32(t_s + 32u * owned_chunk(half, 0), ra);
                tmem_ld32(t_s + 32u * owned_chunk(half, 1), rb);
                tmem_ld_wait();
                reg_fence(ra);
                reg_fence(rb);
                tc_fence_before();
                signal(kNbE1, bars.e1());
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const uint32_t* r = cc == 0 ? ra : rb;
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        float2 v = __ffma2_rn(make_float2(__uint_as_float(r[2 * x]), __uint_as_float(r[2 * x + 1])), scale2,
                                              neg_l2);
                        v.x = ex2_approx(v.x);
                        v.y = ex2_approx(v.y);
                        p[cc][x] = v;
                    }
                }
            }
            // step 2: dS = P * (dP - D), zero past the last key (where P may even overflow);
            // both owned chunks read before either is overwritten by its 16-bit result
            if (!(ok = warp_wait(bars.dp_full(), j & 1, wd))) {
                signal(kNbE2, bars.e2());
                continue;
            }
            tc_fence_after();
            uint32_t rp[2][32];
            tmem_ld32(t_dp + 32u * owned_chunk(half, 0), rp[0]);
            tmem_ld32(t_dp + 32u * owned_chunk(half, 1), rp[1]);
            tmem_ld_wait();
            reg_fence(rp[0]);
            reg_fence(rp[1]);
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c = owned_chunk(half, cc);
                uint32_t pk[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const float2 ds = __fmul2_rn(
                        p[cc][x], __fadd2_rn(make_float2(__uint_as_float(rp[cc][2 * x]), __uint_as_float(rp[cc][2 * x + 1])), neg_d));
                    pk[x] = pack2<kBf16>(ds.x, ds.y);
                }
                if (valid < BT) {
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const int col = 32 * c + 2 * x;
                        if (col >= valid) pk[x] &= 0xFFFF0000u;
                        if (col + 1 >= valid) pk[x] &= 0x0000FFFFu;
                    }
                }
                tmem_st16(t_dp + kPackedCol + 16u * c, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            signal(kNbE2, bars.e2());
        }
        if (ok) ok = warp_wait(bars.done(), 0, wd);
        if (ok) {
            tc_fence_after();
            const uint32_t out_slab = base + C::kDqOut + (uint32_t)((warp - 2) * kOutSlabBytes);
            // the two warps of a quarter split the dQ columns: 32-column chunks alternate
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                if ((c & 1) != half) continue;
                uint32_t r[32];
                tmem_ld32(tmem + lane_off + 256u + 32u * c, r);
                tmem_ld_wait();
                reg_fence(r);
                if constexpr (C::kNamed) {
                    if (plane < 0) {
                        store_chunk_tma<kBf16>(&tm_dq, out_slab, 32 * c, q0 + quarter * 32, n_q, d_act, bh, r, scale);
                    } else {  // two 16-column float32 boxes of the partial sum
                        store_chunk_tma_f32(&tm_dqp, out_slab, 32 * c, q0 + quarter * 32, plane, r, 0);
                        store_chunk_tma_f32(&tm_dqp, out_slab, 32 * c + 16, q0 + quarter * 32, plane, r, 16);
                    }
                } else {
                    store_row_chunk<kBf16>(dq, (size_t)bh * n_q + row, d_act, c, r, scale, row < n_q);
                }
            }
            if (lane == 0) bulk_wait_group0();  // this warp's stores complete before the CTA exits
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kBwdTmemCols);
    }
}

// ------------------------------------------------------------------------------ kernels

// The work of the x-th dQ CTA of head bh when the pass divides each query tile's keys into
// `splits` ranges: range r = x / n_qt, query tile x mod n_qt (the query tiles of one key
// range next to each other, so that they share its K and V tiles in L2), key tiles
// [r L, min(n_kt, r L + L)) with L = ceil(n_kt / splits), partial-sum plane r * heads + bh.
struct DqWork {
    int qt, j0, j1, plane;
};
__device__ __forceinline__ DqWork dq_work(int x, int bh, int n_qt, int n_kt, int splits, int heads) {
    if (splits <= 1) return DqWork{x, 0, n_kt, -1};
    const int r = x / n_qt, len = (n_kt + splits - 1) / splits;
    const int j0 = r * len, j1 = j0 + len < n_kt ? j0 + len : n_kt;
    return DqWork{x % n_qt, j0, j1, r * heads + bh};
}

// dq = scale * (the split dQ pass's float32 partial sums added in key-range order), rounded to
// the 16-bit type: one thread per 4 columns of a row, a warp's loads 512 contiguous bytes.
template <bool kBf16>
__global__ void __launch_bounds__(256)
    bwd_dq_combine_kernel(const float4* __restrict__ part, void* __restrict__ dq, int heads, int n_q, int n_q_pad,
                          int hd, int d_act, int splits, float scale) {
    const int groups = d_act / 4;
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (i >= (int64_t)heads * n_q * groups) return;
    const int g = (int)(i % groups);
    const int64_t rowi = i / groups;  // head * n_q + row
    const int row = (int)(rowi % n_q), b = (int)(rowi / n_q);
    const int64_t plane = (int64_t)heads * n_q_pad * (hd / 4);
    const float4* src = part + ((int64_t)b * n_q_pad + row) * (hd / 4) + g;
    float4 acc = src[0];
    for (int r = 1; r < splits; ++r) {
        const float4 x = src[r * plane];
        acc.x += x.x;
        acc.y += x.y;
        acc.z += x.z;
        acc.w += x.w;
    }
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(dq) + rowi * d_act + 4 * g) =
        make_uint2(pack2<kBf16>(acc.x * scale, acc.y * scale), pack2<kBf16>(acc.z * scale, acc.w * scale));
}

template <int D, bool kBf16, int kNV>
__global__ void __launch_bounds__(BwdCfg<D, kNV>::kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_v2, const __grid_constant__ CUtensorMap tm_do2,
                    const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                    const float* __restrict__ lse2, const float* __restrict__ delta, void* __restrict__ dk,
                    void* __restrict__ dv, void* __restrict__ dv2, int n_q, int n_k, int n_q_pad, int d_act, float scale,
                    float scale_log2, unsigned int* status) {
    dkdv_cta<D, kBf16, kNV>(tm_q, tm_k, tm_v, tm_do, tm_v2, tm_do2, tm_dk, tm_dv, lse2, delta, dk, dv, dv2, n_q, n_k,
                            n_q_pad, d_act, scale, scale_log2, status, blockIdx.x, 1, blockIdx.y);
}

// The dK/dV pass with each key tile's queries split over a cluster of `splits` CTAs
// (grid x = key tiles x splits, cluster splits x 1 x 1).
template <int D, bool kBf16>
__global__ void __launch_bounds__(BwdCfg<D, 1>::kThreads, 1)
    bwd_dkdv_split_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                          const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                          const float* __restrict__ lse2, const float* __restrict__ delta, void* __restrict__ dk,
                          void* __restrict__ dv, int n_q, int n_k, int n_q_pad, int d_act, float scale, float scale_log2,
                          unsigned int* status, int splits) {
    dkdv_cta<D, kBf16, 1, true>(tm_q, tm_k, tm_v, tm_do, tm_v, tm_do, tm_dk, tm_dv, lse2, delta, dk, dv, nullptr, n_q,
                                n_k, n_q_pad, d_act, scale, scale_log2, status, (int)(blockIdx.x / (unsigned)splits), 1,
                                blockIdx.y, splits);
}

template <int D, bool kBf16, int kNV>
__global__ void __launch_bounds__(BwdCfg<D, kNV>::kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_v2, const __grid_constant__ CUtensorMap tm_dq,
                  const __grid_constant__ CUtensorMap tm_dqp, const uint16_t* __restrict__ q_ptr,
                  const uint16_t* __restrict__ do_ptr, const uint16_t* __restrict__ do2_ptr,
                  const float* __restrict__ lse2, const float* __restrict__ delta, void* __restrict__ dq, int n_q,
                  int n_k, int n_q_pad, int d_act, float scale, float scale_log2, unsigned int* status, int splits) {
    const int n_qt = (n_q + BT - 1) / BT;
    const DqWork w = dq_work((int)blockIdx.x, (int)blockIdx.y, n_qt, (n_k + BT - 1) / BT, splits, (int)gridDim.y);
    dq_cta<D, kBf16, kNV>(tm_k, tm_v, tm_v2, tm_dq, q_ptr, do_ptr, do2_ptr, lse2, delta, dq, n_q, n_k, n_q_pad, d_act,
                          scale, scale_log2, status, w.qt, (int)blockIdx.y, tm_dqp, w.j0, w.j1, w.plane);
}

// Both passes in one launch.  The passes are independent once D and LSE2 are in
// the workspace; one grid lets the CTAs of one fill the SMs the other leaves idle
// in its last wave.  A dK/dV CTA takes kt_per_cta consecutive key tiles (the last
// of a head fewer), n_kc = ceil(n_kt / kt_per_cta) of them per head.  Order of the
// CTAs (x fastest, then the head y), the dQ CTAs of a head numbered as dq_work takes them:
//   dq_first == 0: per head, x < n_kc runs the dK/dV pass for key tiles from
//     x * kt_per_cta and the rest the dQ pass for query tile x - n_kc, so that a
//     head's two sets of CTAs run together and share its Q, K, V, dO in L2;
//   dq_first == 1: the dQ CTAs of all heads first, then all dK/dV CTAs - for
//     shapes whose dQ CTAs (n_kt key tiles each) are much longer than the dK/dV
//     CTAs: started first, they do not end in a tail.
template <int D, bool kBf16, int kNV>
__global__ void __launch_bounds__(BwdCfg<D, kNV>::kThreads, 1)
    bwd_passes_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_v2, const __grid_constant__ CUtensorMap tm_do2,
                      const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                      const __grid_constant__ CUtensorMap tm_dv, const __grid_constant__ CUtensorMap tm_dqp,
                      const uint16_t* __restrict__ q_ptr, const uint16_t* __restrict__ do_ptr,
                      const uint16_t* __restrict__ do2_ptr, const float* __restrict__ lse2,
                      const float* __restrict__ delta, void* __restrict__ dq, void* __restrict__ dk, void* __restrict__ dv,
                      void* __restrict__ dv2, int n_q, int n_k, int n_q_pad, int d_act, float scale, float scale_log2,
                      unsigned int* status, int dq_first, int kt_per_cta, int splits) {
    const int n_kt = (n_k + BT - 1) / BT, n_qt = (n_q + BT - 1) / BT;
    const int n_kc = (n_kt + kt_per_cta - 1) / kt_per_cta;
    const int n_dqc = n_qt * (splits > 1 ? splits : 1);  // dQ CTAs per head
    int dkdv_cta_x = -1, dq_x = -1, bh;
    if (!dq_first) {
        bh = blockIdx.y;
        if ((int)blockIdx.x < n_kc) dkdv_cta_x = blockIdx.x;
        else dq_x = blockIdx.x - n_kc;
    } else {
        const int lin = blockIdx.y * gridDim.x + blockIdx.x, n_dq = (int)gridDim.y * n_dqc;
        if (lin < n_dq) {
            bh = lin / n_dqc;
            dq_x = lin % n_dqc;
        } else {
            bh = (lin - n_dq) / n_kc;
            dkdv_cta_x = (lin - n_dq) % n_kc;
        }
    }
    if (dkdv_cta_x >= 0) {
        const int kt = dkdv_cta_x * kt_per_cta;
        const int items = n_kt - kt < kt_per_cta ? n_kt - kt : kt_per_cta;
        dkdv_cta<D, kBf16, kNV>(tm_q, tm_k, tm_v, tm_do, tm_v2, tm_do2, tm_dk, tm_dv, lse2, delta, dk, dv, dv2, n_q, n_k,
                                n_q_pad, d_act, scale, scale_log2, status, kt, items, bh);
    }
    else {
        const DqWork w = dq_work(dq_x, bh, n_qt, n_kt, splits, (int)gridDim.y);
        dq_cta<D, kBf16, kNV>(tm_k, tm_v, tm_v2, tm_dq, q_ptr, do_ptr, do2_ptr, lse2, delta, dq, n_q, n_k, n_q_pad, d_act,
                              scale, scale_log2, status, w.qt, bh, tm_dqp, w.j0, w.j1, w.plane);
    }
}

// ------------------------------------------------------------------------------ launch

// Key tiles per dK/dV CTA of the one-grid launch: at least 32 query tiles per CTA, so
// that the fixed cost of a key tile (K and V load, pipeline fill, dK / dV write-out,
// about 5.6 us on GB300) is partly hidden behind the next tile's work. Measured on
// GB300 (bf16, head size 128, BH = 32): N_q = 1024, N_k = 32768 1.353 -> 1.270 ms with
// 4 key tiles per CTA (1.301 with 8); N_q = N_k = 8192 keeps 1 (2 read 2.345 against
// 2.303 ms). Fewer key tiles per CTA where that would leave fewer dK/dV CTAs than SMs
// (few heads): there the grid's parallelism matters more than the hidden fixed cost.
static int dkdv_tiles_per_cta(int n_qt, int n_kt, int64_t bh, int sms) {
    int m = (32 + n_qt - 1) / n_qt;
    m = m < 1 ? 1 : (m > 8 ? 8 : m);
    while (m > 1 && bh * (int64_t)((n_kt + m - 1) / m) < sms) --m;
    return m;
}

template <int D, bool kBf16, int kNV>
cudaError_t launch_impl(const BwdParams& p, cudaStream_t stream, int slot, int stages) {
    using C = BwdCfg<D, kNV>;
    if (stages & kBwdPreprocess) {
        constexpr int RPC = 256 / (D / 8);
        const dim3 grid((unsigned)((p.n_q_pad + RPC - 1) / RPC), (unsigned)p.bh, 1);
        bwd_preprocess_kernel<D, kBf16><<<grid, 256, 0, stream>>>(
            static_cast<const uint16_t*>(p.o), static_cast<const uint16_t*>(p.d_o),
            kNV == 2 ? static_cast<const uint16_t*>(p.o2) : nullptr, kNV == 2 ? static_cast<const uint16_t*>(p.d_o2) : nullptr,
            p.lse, p.delta, p.lse2, p.dq_acc, (int)p.n_q, (int)p.n_q_pad, p.d);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (!(stages & (kBwdDkDv | kBwdDq))) return cudaSuccess;
    const CUtensorMapDataType dt = kBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUtensorMapSwizzle sw = D >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    CUtensorMap tq, tk, tv, tdo, tv2, tdo2, tdq, tdk, tdv, tdqp;
    const void* v2 = kNV == 2 ? p.v2 : p.v;
    const void* do2 = kNV == 2 ? p.d_o2 : p.d_o;
    // maps over the true head dimension p.d <= D: TMA fills the box columns past it with zeros
    const uint64_t d = (uint64_t)p.d;
    if (!encode_tmap_3d(&tq, dt, 2, p.q, d, (uint64_t)p.n_q, (uint64_t)p.bh, C::kAtomCols, BT, sw) ||
        !encode_tmap_3d(&tdo, dt, 2, p.d_o, d, (uint64_t)p.n_q, (uint64_t)p.bh, C::kAtomCols, BT, sw) ||
        !encode_tmap_3d(&tdo2, dt, 2, do2, d, (uint64_t)p.n_q, (uint64_t)p.bh, C::kAtomCols, BT, sw) ||
        !encode_tmap_3d(&tk, dt, 2, p.k, d, (uint64_t)p.n_k, (uint64_t)p.bh, C::kAtomCols, BT, sw) ||
        !encode_tmap_3d(&tv, dt, 2, p.v, d, (uint64_t)p.n_k, (uint64_t)p.bh, C::kAtomCols, BT, sw) ||
        !encode_tmap_3d(&tv2, dt, 2, v2, d, (uint64_t)p.n_k, (uint64_t)p.bh, C::kAtomCols, BT, sw))
        return cudaErrorInvalidValue;
    // the gradients, stored by TMA in boxes of 32 columns x 32 rows (one warp's slab); the
    // two-value PSA form writes its gradients with plain stores and passes these unused
    const bool named = C::kNamed;
    const void* out_dq = named && p.dq ? p.dq : p.q;
    const void* out_dk = named && p.dk ? p.dk : p.k;
    const void* out_dv = named && p.dv ? p.dv : p.v;
    if (!encode_tmap_3d(&tdq, dt, 2, out_dq, d, (uint64_t)p.n_q, (uint64_t)p.bh, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tmap_3d(&tdk, dt, 2, out_dk, d, (uint64_t)p.n_k, (uint64_t)p.bh, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tmap_3d(&tdv, dt, 2, out_dv, d, (uint64_t)p.n_k, (uint64_t)p.bh, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    // the split dQ pass's float32 partial sums: [splits * bh, n_q_pad, D], boxes of 16 x 32
    // (without a split the map is encoded over q and never used)
    const int splits = C::kNamed && p.dq_part ? p.dq_splits : 1;
    const bool split = splits > 1;
    if (C::kNamed && (stages & kBwdDq)) launch_record().bwd_dq_key_ranges = splits;  // plain attention only
    if (!encode_tmap_3d(&tdqp, split ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : dt, split ? 4 : 2,
                        split ? static_cast<const void*>(p.dq_part) : p.q, split ? (uint64_t)D : d,
                        split ? (uint64_t)p.n_q_pad : (uint64_t)p.n_q, (uint64_t)(split ? splits * p.bh : p.bh),
                        split ? 16 : 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    const float scale_log2 = p.scale * kLog2e;
    // the combine of a split dQ pass, after the kernel that wrote the partial sums
    auto combine = [&]() -> cudaError_t {
        if (!split) return cudaSuccess;
        const int64_t threads = p.bh * p.n_q * (p.d / 4);
        bwd_dq_combine_kernel<kBf16><<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(
            reinterpret_cast<const float4*>(p.dq_part), p.dq, (int)p.bh, (int)p.n_q, (int)p.n_q_pad, D, p.d, splits,
            p.scale);
        return cudaGetLastError();
    };
    cudaError_t e = cudaSuccess;
    const int n_kt = (int)((p.n_k + BT - 1) / BT), n_qt = (int)((p.n_q + BT - 1) / BT);
    // many queries, few key tiles: the dK/dV pass over query ranges in clusters, then the dQ pass
    int qsplits = C::kNamed ? dkv_query_splits(p.bh, p.n_q, p.n_k, D) : 1;
    auto split_kern = bwd_dkdv_split_kernel<D, kBf16>;
    if (qsplits > 1 && (stages & kBwdDkDv)) {
        const int split_slot = 52 + (slot - 16) / 2;  // slots 52..61
        e = ensure_smem_limit(reinterpret_cast<const void*>(split_kern), C::kSmemDkv, split_slot);
        if (e != cudaSuccess) return e;
        // a device that cannot hold the whole cluster at once takes fewer ranges
        while (qsplits > 1 &&
               !cluster_fits(reinterpret_cast<const void*>(split_kern), C::kThreads, C::kSmemDkv, qsplits, split_slot))
            qsplits /= 2;
    }
    if (qsplits > 1 && (stages & kBwdDkDv)) {
        launch_record().bwd_dkv_query_ranges = qsplits;
        auto kern = split_kern;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(n_kt * qsplits), (unsigned)p.bh, 1);
        cfg.blockDim = dim3(C::kThreads, 1, 1);
        cfg.dynamicSmemBytes = C::kSmemDkv;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)qsplits;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tdo, tdk, tdv, p.lse2, p.delta, p.dk, p.dv, (int)p.n_q, (int)p.n_k,
                               (int)p.n_q_pad, p.d, p.scale, scale_log2, p.status, qsplits);
        if (e != cudaSuccess) return e;
        stages &= ~kBwdDkDv;  // the dQ pass follows on its own
    }
    if ((stages & (kBwdDkDv | kBwdDq)) == (kBwdDkDv | kBwdDq)) {
        auto both = bwd_passes_kernel<D, kBf16, kNV>;
        constexpr int smem = C::kSmemDkv > C::kSmemDq ? C::kSmemDkv : C::kSmemDq;
        e = ensure_smem_limit(reinterpret_cast<const void*>(both), smem, 42 + (slot - 16) / 2);  // slots 42..51
        if (e != cudaSuccess) return e;
        const int m = C::kNamed ? dkdv_tiles_per_cta(n_qt, n_kt, p.bh, sm_count()) : 1;
        if (C::kNamed) launch_record().bwd_key_tiles_per_cta = m;
        const int n_kc = (n_kt + m - 1) / m;
        const int dq_len = (n_kt + splits - 1) / splits;  // key tiles per dQ CTA
        both<<<dim3((unsigned)(n_kc + n_qt * splits), (unsigned)p.bh, 1), C::kThreads, smem, stream>>>(
            tq, tk, tv, tdo, tv2, tdo2, tdq, tdk, tdv, tdqp, static_cast<const uint16_t*>(p.q), static_cast<const uint16_t*>(p.d_o),
            static_cast<const uint16_t*>(kNV == 2 ? p.d_o2 : p.d_o), p.lse2, p.delta, p.dq, p.dk, p.dv, p.dv2, (int)p.n_q,
            (int)p.n_k, (int)p.n_q_pad, p.d, p.scale, scale_log2, p.status, dq_len >= 4 * m * n_qt ? 1 : 0, m, splits);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        return combine();
    }
    if (stages & kBwdDkDv) {
        auto dkdv = bwd_dkdv_kernel<D, kBf16, kNV>;
        e = ensure_smem_limit(reinterpret_cast<const void*>(dkdv), C::kSmemDkv, slot);
        if (e != cudaSuccess) return e;
        dkdv<<<dim3((unsigned)n_kt, (unsigned)p.bh, 1), C::kThreads, C::kSmemDkv, stream>>>(
            tq, tk, tv, tdo, tv2, tdo2, tdk, tdv, p.lse2, p.delta, p.dk, p.dv, p.dv2, (int)p.n_q, (int)p.n_k, (int)p.n_q_pad,
            p.d, p.scale, scale_log2, p.status);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (!(stages & kBwdDq)) return cudaSuccess;
    auto dqk = bwd_dq_kernel<D, kBf16, kNV>;
    e = ensure_smem_limit(reinterpret_cast<const void*>(dqk), C::kSmemDq, slot + 1);
    if (e != cudaSuccess) return e;
    dqk<<<dim3((unsigned)(n_qt * splits), (unsigned)p.bh, 1), C::kThreads, C::kSmemDq, stream>>>(
        tk, tv, tv2, tdq, tdqp, static_cast<const uint16_t*>(p.q), static_cast<const uint16_t*>(p.d_o),
        static_cast<const uint16_t*>(kNV == 2 ? p.d_o2 : p.d_o), p.lse2, p.delta, p.dq, (int)p.n_q, (int)p.n_k,
        (int)p.n_q_pad, p.d, p.scale, scale_log2, p.status, splits);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return combine();
}

}  // namespace

cudaError_t launch_bwd_tc(const BwdParams& p, cudaStream_t stream, int stages) {
    const bool bf = p.dtype == kBf16;
    switch (pad_head_dim(p.d)) {
        case 32: return bf ? launch_impl<32, true, 1>(p, stream, 16, stages) : launch_impl<32, false, 1>(p, stream, 18, stages);
        case 64: return bf ? launch_impl<64, true, 1>(p, stream, 20, stages) : launch_impl<64, false, 1>(p, stream, 22, stages);
        case 128:
            return bf ? launch_impl<128, true, 1>(p, stream, 24, stages) : launch_impl<128, false, 1>(p, stream, 26, stages);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bwd_tc_dual_v(const BwdParams& p, cudaStream_t stream) {
    const bool bf = p.dtype == kBf16;
    switch (pad_head_dim(p.d)) {
        case 32: return bf ? launch_impl<32, true, 2>(p, stream, 28, kBwdAll) : launch_impl<32, false, 2>(p, stream, 30, kBwdAll);
        case 64: return bf ? launch_impl<64, true, 2>(p, stream, 32, kBwdAll) : launch_impl<64, false, 2>(p, stream, 34, kBwdAll);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa2
