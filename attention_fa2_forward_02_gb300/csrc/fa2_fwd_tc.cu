// fa2_fwd_tc.cu - attention forward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes: "vision-rs 0.1.1 flash_attn2.rs", flash_attention2_forward
// (scores scaled by softmax_scale, the online-softmax recurrence over key rows,
// O = acc / l, LSE = m + ln l), over the flat [BH, N, HEAD_DIM] layout.  The
// page runs one key row at a time per query row; here the recurrence runs one
// 128-key tile at a time per 128-row query tile, the tile form of the update
// that "vyre-libs 0.7.2 flash_attention_2.rs" describes for flash_attention_2
// (all scores of a tile first, then one (m, l, o_acc) update per tile).
//
// CTA shape: two 128-row query tiles (Q0, Q1) sharing every K/V tile.
//   warp 0      TMA producer: Q0/Q1 once, then a K ring and a V ring
//   warp 1      allocates tensor memory; lane 0 issues every tcgen05.mma
//   warps 2-5   softmax for Q0 (one thread per query row / TMEM lane)
//   warps 6-9   softmax for Q1
//   warp 10     (one value tensor) waits for the TMA copies on behalf of the issuer
// With one value tensor the issuer never waits on an mbarrier: a shared-memory access (an
// mbarrier test included) by the warp that issues tcgen05.mma costs a few hundred
// clocks of tensor-pipe time each. Warp 10 and the softmax groups signal it through
// named barriers instead (barrier.arrive; the issuer's barrier.sync is not a memory
// access): one barrier per query tile for "P ready", one per ring stage for "V
// loaded" and "K loaded". A producer cannot arrive twice on one barrier before the
// issuer has synced on it (its next arrival needs a tile the issuer has not yet
// released or issued), and every producer arrives exactly once per event whatever
// happens: a failed bounded wait skips the work, not the arrival, and raises the
// watchdog status. The issuer itself never gives up; a failure elsewhere only makes
// it multiply stale tiles until its loop ends. The two-value PSA form keeps lane 0 of
// the issuer waiting on the mbarriers itself.
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,128) S0 = Q0 K^T   [128,256) S1 = Q1 K^T   [256,256+D) O0   [256+D,256+2D) O1
// The probabilities P (16-bit) are written back over the first 64 columns of
// their S tile and consumed from tensor memory by the P.V MMA.  MMA order per
// key tile j:  PV0(j), S0(j+1), PV1(j), S1(j+1): while one softmax group works
// on its scores the tensor core runs the other group's products.
//
// Running maximum: exact except that the O / l rescale is skipped while the
// new tile maximum exceeds the reference maximum by at most 8 (base-2 units);
// the reference then lags the true maximum by at most 8, so every exponent is
// <= 2^8 and the final O = acc / l is the same quotient up to rounding.
//
// Few CTAs, many keys (fewer query-tile pairs than SMs): a thread-block cluster of
// `splits` CTAs (2, 4, 8, or 16 at head sizes 64 and 128) shares a query-tile pair, CTA r taking key tiles
// [floor(r n_kv / splits), floor((r + 1) n_kv / splits)), never empty (n_kv >= 8 splits). Each ends with its own (O_r, m_r,
// l_r) per row; the cluster then combines them through distributed shared memory in the
// Q/K/V buffers its loops no longer use: every CTA sends each row's (m_r, l_r) to all,
// scales its O_r by 2^(m_r - M) / L (M the largest m_r, L the sum of l_r 2^(m_r - M)) and
// sends each CTA the columns that CTA stores; each adds the parts in rank order (so the
// result does not depend on timing) and writes its columns of O, rank 0 the LSE, M + log2 L.
#include "common.cuh"
#include "internal.h"

namespace fa2 {
namespace {

constexpr int BM = 128;            // query rows per tile = TMEM lanes
constexpr int BN = 128;            // keys per K/V tile
constexpr int kQTiles = 2;         // query tiles per CTA
constexpr int kRelayWarp = 10;
// Named barriers (0 is __syncthreads): 1 + t: P of query tile t ready (softmax group
// t + issuer, 160 threads); then per ring stage s: V loaded, K loaded (relay + issuer,
// 64 threads).
constexpr uint32_t kNbP = 1;
__host__ __device__ constexpr uint32_t nb_v(int s) { return 1 + 2 + (uint32_t)s; }
__host__ __device__ constexpr uint32_t nb_k(int S, int s) { return 1 + 2 + (uint32_t)(S + s); }

constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.693147180559945309f;

// kNV = number of value tensors sharing the scores: 1 (plain attention) or 2
// (the PSA V_lo / V_hi pair, whose probabilities are identical).
template <int D, int kNV>
struct FwdCfg : Tile16<D> {
    static constexpr int kStages = D == 128 ? 2 : (D == 64 ? 3 : 4);
    // One value tensor: the issuer is fed through named barriers and a TMA relay warp
    // (11 warps). The two-value PSA form keeps the issuer's own mbarrier waits.
    static constexpr bool kNamed = kNV == 1;
    static constexpr int kThreads = kNamed ? 352 : 320;
    static constexpr int kQTileBytes = BM * D * 2;
    static constexpr int kKVTileBytes = BN * D * 2;
    static constexpr int kVStageBytes = kNV * kKVTileBytes;
    static constexpr int kSmemQ = 0;
    static constexpr int kSmemK = kSmemQ + kQTiles * kQTileBytes;
    static constexpr int kSmemV = kSmemK + kStages * kKVTileBytes;
    static constexpr int kSmemBar = kSmemV + kStages * kVStageBytes;
    static constexpr int kNumBars = 1 + 4 * kStages + 2 + 2 + 1;
    static constexpr int kSmemMisc = kSmemBar + kNumBars * 8;
    static constexpr int kSmemBytes = kSmemMisc + 16 + 1024;  // + slack to align the base to 1024
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(256 + 2 * kNV * D <= (int)kTmemCols, "tensor memory budget");
    // cluster combine: (m, l) of every CTA's 256 rows, then every CTA's share of each row
    static constexpr int kExchMl = 0;
    static constexpr int kExchRecv = 16 * 256 * 8;  // up to 16 CTAs' (m, l) of 256 rows
    static_assert(kExchRecv + 256 * D * 4 <= kSmemBar, "cluster combine buffers");
};

template <int D, bool kBf16, int kNV>
__global__ void __launch_bounds__(FwdCfg<D, kNV>::kThreads, 1)
    fa2_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_v2,
                      void* __restrict__ o_ptr, void* __restrict__ o2_ptr, float* __restrict__ lse_ptr, int n_q, int n_k,
                      int d_act, float scale_log2, unsigned int* status, int splits) {
    using C = FwdCfg<D, kNV>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_addr);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int bh = blockIdx.y;
    // splits > 1: the CTAs of a cluster (consecutive blockIdx.x; the cluster is splits x 1 x 1,
    // so blockIdx.x mod splits is the CTA's rank in it) share a query-tile pair
    const int rank = (int)(blockIdx.x % (unsigned)splits);
    const int q0 = (blockIdx.x / splits) * (BM * kQTiles);
    const int n_kv_all = (n_k + BN - 1) / BN;
    // this CTA's key tiles: [j0, j0 + n_kv), the rank-th of `splits` balanced ranges (none
    // empty: the launch takes at least 8 key tiles per range)
    const int j0 = (int)((int64_t)rank * n_kv_all / splits);
    const int n_kv = (int)((int64_t)(rank + 1) * n_kv_all / splits) - j0;
    float ep_m2 = 0.f, ep_l = 0.f;  // a softmax thread's row state, kept for the cluster combine
    bool ep_ok = false;

    const uint32_t bars = base + C::kSmemBar;
    const uint32_t B_Q = bars;
    auto B_KF = [&](int s) { return bars + 8u * (1 + s); };
    auto B_KE = [&](int s) { return bars + 8u * (1 + S + s); };
    auto B_VF = [&](int s) { return bars + 8u * (1 + 2 * S + s); };
    auto B_VE = [&](int s) { return bars + 8u * (1 + 3 * S + s); };
    auto B_SF = [&](int t) { return bars + 8u * (1 + 4 * S + t); };
    auto B_PF = [&](int t) { return bars + 8u * (3 + 4 * S + t); };
    const uint32_t B_OD = bars + 8u * (5 + 4 * S);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kSmemMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kSmemMisc + 4);
    const Watchdog wd{abort_flag, status};

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(B_Q, 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(B_KF(s), 1);
            mbar_init(B_KE(s), 1);
            mbar_init(B_VF(s), 1);
            mbar_init(B_VE(s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(B_SF(t), 1);
            mbar_init(B_PF(t), BM);
        }
        mbar_init(B_OD, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    const uint32_t q_smem = base + C::kSmemQ;
    const uint32_t k_smem = base + C::kSmemK;
    const uint32_t v_smem = base + C::kSmemV;

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            if (kNV == 2) prefetch_tmap(&tm_v2);
            mbar_arrive_expect_tx(B_Q, kQTiles * C::kQTileBytes);
            for (int t = 0; t < kQTiles; ++t)
                for (int a = 0; a < C::kAtoms; ++a)
                    tma_load_3d(q_smem + t * C::kQTileBytes + a * BM * C::kAtomRowBytes, &tm_q, B_Q, a * C::kAtomCols,
                                q0 + t * BM, bh);
            int issued = 0;
            bool ok = true;
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % S;
                const uint32_t release_parity = ((j / S) & 1) ^ 1;
                if (j >= S && !(ok = mbar_wait(B_KE(s), release_parity, wd))) break;
                mbar_arrive_expect_tx(B_KF(s), C::kKVTileBytes);
                for (int a = 0; a < C::kAtoms; ++a)
                    tma_load_3d(k_smem + s * C::kKVTileBytes + a * BN * C::kAtomRowBytes, &tm_k, B_KF(s),
                                a * C::kAtomCols, (j0 + j) * BN, bh);
                if (j >= S && !(ok = mbar_wait(B_VE(s), release_parity, wd))) {
                    issued = 2 * j + 1;
                    break;
                }
                mbar_arrive_expect_tx(B_VF(s), C::kVStageBytes);
                for (int v = 0; v < kNV; ++v)
                    for (int a = 0; a < C::kAtoms; ++a)
                        tma_load_3d(v_smem + s * C::kVStageBytes + v * C::kKVTileBytes + a * BN * C::kAtomRowBytes,
                                    v ? &tm_v2 : &tm_v, B_VF(s), a * C::kAtomCols, (j0 + j) * BN, bh);
                issued = 2 * j + 2;
            }
            if (!ok) {
                // Drain the copies still in flight before the CTA's shared memory is released.
                drain_wait(B_Q, 0);
                for (int i = (issued > 2 * S ? issued - 2 * S : 0); i < issued; ++i) {
                    const int j = i >> 1, s = j % S;
                    drain_wait((i & 1) ? B_VF(s) : B_KF(s), (j / S) & 1);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if constexpr (C::kNamed) {
            const uint32_t idesc_s = idesc_f16_f32acc(BM, BN, kBf16, false, false);
            const uint32_t idesc_o = idesc_f16_f32acc(BM, D, kBf16, false, true);
            // Descriptors of query tile / ring stage 0 at k-step 0, built once; every other
            // operand adds a constant to the start-address field (16-byte units; shared
            // addresses stay below 256 KB, so nothing carries out of the field). The
            // issuer shares its sub-partition with two busy softmax warps: the fewer
            // instructions it needs per MMA, the fuller it keeps the tensor pipe.
            const uint64_t dq0 = C::kmajor(q_smem, 0, BM);
            const uint64_t dk0 = C::kmajor(k_smem, 0, BN);
            const uint64_t dv0 = C::mnmajor(v_smem, 0, BN);
            auto issue_s = [&](int t, int s) {
                const uint32_t d_tmem = tmem + (uint32_t)(t * BN);
                const uint64_t qa = dq0 + (uint64_t)((t * C::kQTileBytes) >> 4);
                const uint64_t kb = dk0 + (uint64_t)((s * C::kKVTileBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(d_tmem, qa + (uint64_t)(C::koff(kk, BM) >> 4), kb + (uint64_t)(C::koff(kk, BN) >> 4), idesc_s,
                           kk > 0 ? 1u : 0u);
            };
            auto issue_pv = [&](int t, int s, bool acc) {
                const uint32_t d_tmem = tmem + 256u + (uint32_t)(t * D);
                const uint64_t vb = dv0 + (uint64_t)((s * C::kVStageBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ts(d_tmem, tmem + (uint32_t)(t * BN + kk * 8), vb + (uint64_t)(kk * C::kAtomRowBytes), idesc_o,
                           (acc || kk > 0) ? 1u : 0u);
            };
            static_assert(1 + 2 + 2 * S <= 16, "named barriers");
            nb_sync(nb_k(S, 0), 64);  // Q and the first K tile
            if (lane == 0) {
                tc_fence_after();
                issue_s(0, 0);
                mma_commit(B_SF(0));
                issue_s(1, 0);
                mma_commit(B_SF(1));
                mma_commit(B_KE(0));
            }
            __syncwarp();
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % S;
                const int jn = j + 1;
                const int sn = jn % S;
                nb_sync(nb_v(s), 64);  // V tile j
                for (int t = 0; t < kQTiles; ++t) {
                    nb_sync(kNbP + t, BM + 32);  // P of query tile t
                    if (lane == 0) {
                        tc_fence_after();
                        issue_pv(t, s, j > 0);
                        if (t == kQTiles - 1) mma_commit(B_VE(s));
                    }
                    if (jn < n_kv) {
                        if (t == 0) nb_sync(nb_k(S, sn), 64);  // K tile j + 1
                        if (lane == 0) {
                            tc_fence_after();
                            issue_s(t, sn);
                            mma_commit(B_SF(t));
                            if (t == kQTiles - 1) mma_commit(B_KE(sn));
                        }
                    }
                    __syncwarp();
                }
            }
            // Completion of everything issued: the softmax groups read O after it,
            // and tensor memory is released only after it.
            if (lane == 0) {
                mma_commit(B_OD);
                drain_wait(B_OD, 0);
            }
            __syncwarp();
        } else {
            // lane 0 waits on the mbarriers itself
            if (lane == 0) {
                const uint32_t idesc_s = idesc_f16_f32acc(BM, BN, kBf16, false, false);
                const uint32_t idesc_o = idesc_f16_f32acc(BM, D, kBf16, false, true);
                // descriptors built once, as in the named-barrier issuer above
                const uint64_t dq0 = C::kmajor(q_smem, 0, BM);
                const uint64_t dk0 = C::kmajor(k_smem, 0, BN);
                const uint64_t dv0 = C::mnmajor(v_smem, 0, BN);
                auto issue_s = [&](int t, int s) {
                    const uint32_t d_tmem = tmem + (uint32_t)(t * BN);
                    const uint64_t qa = dq0 + (uint64_t)((t * C::kQTileBytes) >> 4);
                    const uint64_t kb = dk0 + (uint64_t)((s * C::kKVTileBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(d_tmem, qa + (uint64_t)(C::koff(kk, BM) >> 4), kb + (uint64_t)(C::koff(kk, BN) >> 4), idesc_s,
                               kk > 0 ? 1u : 0u);
                };
                auto issue_pv = [&](int t, int s, bool acc) {
#pragma unroll
                    for (int v = 0; v < kNV; ++v) {
                        const uint32_t d_tmem = tmem + 256u + (uint32_t)((t * kNV + v) * D);
                        const uint64_t vb = dv0 + (uint64_t)((s * C::kVStageBytes + v * C::kKVTileBytes) >> 4);
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk)
                            mma_ts(d_tmem, tmem + (uint32_t)(t * BN + kk * 8), vb + (uint64_t)(kk * C::kAtomRowBytes), idesc_o,
                                   (acc || kk > 0) ? 1u : 0u);
                    }
                };
                bool ok = mbar_wait(B_Q, 0, wd) && mbar_wait(B_KF(0), 0, wd);
                if (ok) {
                    tc_fence_after();
                    issue_s(0, 0);
                    mma_commit(B_SF(0));
                    issue_s(1, 0);
                    mma_commit(B_SF(1));
                    mma_commit(B_KE(0));
                }
                for (int j = 0; ok && j < n_kv; ++j) {
                    const int s = j % S;
                    const int jn = j + 1;
                    const int sn = jn % S;
                    if (!(ok = mbar_wait(B_VF(s), (j / S) & 1, wd))) break;
                    for (int t = 0; t < kQTiles; ++t) {
                        if (!(ok = mbar_wait(B_PF(t), j & 1, wd))) break;
                        tc_fence_after();
                        issue_pv(t, s, j > 0);
                        if (t == kQTiles - 1) mma_commit(B_VE(s));
                        if (jn < n_kv) {
                            if (t == 0) {
                                if (!(ok = mbar_wait(B_KF(sn), (jn / S) & 1, wd))) break;
                                tc_fence_after();
                            }
                            issue_s(t, sn);
                            mma_commit(B_SF(t));
                            if (t == kQTiles - 1) mma_commit(B_KE(sn));
                        }
                    }
                }
                // Completion of everything issued: the softmax groups read O after it,
                // and tensor memory is released only after it.
                mma_commit(B_OD);
                drain_wait(B_OD, 0);
            }
        }
    } else if (C::kNamed && warp == kRelayWarp) {
        // ------------------------------------------------------------------ TMA relay
        // Waits for the copies the issuer needs, in the order it needs them.
        bool ok = warp_wait(B_Q, 0, wd) && warp_wait(B_KF(0), 0, wd);
        nb_arrive(nb_k(S, 0), 64);
        for (int j = 0; j < n_kv; ++j) {
            const int s = j % S;
            const int jn = j + 1;
            const int sn = jn % S;
            ok = ok && warp_wait(B_VF(s), (j / S) & 1, wd);
            nb_arrive(nb_v(s), 64);
            if (jn < n_kv) {
                ok = ok && warp_wait(B_KF(sn), (jn / S) & 1, wd);
                nb_arrive(nb_k(S, sn), 64);
            }
        }
    } else {
        // ------------------------------------------------------------------ softmax groups
        const int t = (warp - 2) >> 2;
        const int quarter = warp & 3;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t s_addr = tmem + lane_off + (uint32_t)(t * BN);
        const uint32_t o_addr = tmem + lane_off + 256u + (uint32_t)(t * kNV * D);  // kNV accumulators of D columns
        float m2 = -INFINITY;  // reference maximum, base-2 units (score * scale * log2 e)
        float l = 0.f;
        bool ok = true;
        const float2 scale2 = make_float2(scale_log2, scale_log2);
        for (int j = 0; j < n_kv; ++j) {
            // a failed wait skips the work of this and later tiles, not the meeting
            ok = ok && warp_wait(B_SF(t), j & 1, wd);
            if (ok) {
                tc_fence_after();
                // The score row (128 columns) into registers: one read of the S tile per key tile.
                uint32_t sr[BN / 32][32];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) tmem_ld32(s_addr + 32u * c, sr[c]);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) reg_fence(sr[c]);
                // Only the last key tile can be partial: its columns past the last key become
                // -inf, which drops them from the maximum and gives them probability 0.
                const int valid = n_k - (j0 + j) * BN;
                if (valid < BN) {
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (32 * c + i >= valid) sr[c][i] = __float_as_uint(-INFINITY);
                }
                // The row maximum: 8 independent chains of three-input maxima.
                float mx;
                {
                    float m8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) m8[i] = -INFINITY;
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c)
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            m8[i & 7] = fmax3(m8[i & 7], __uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1]));
                    mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                }
                const float m_new = mx * scale_log2;
                float alpha = 1.f;   // factor for O and l when the reference maximum moves
                bool rescale = false;
                if (j == 0) {
                    m2 = m_new;
                } else {
                    const bool need = m_new > m2 + kRescaleThreshold;
                    rescale = __any_sync(0xffffffffu, need);
                    if (need) {
                        alpha = ex2_approx(m2 - m_new);
                        l *= alpha;
                        m2 = m_new;
                    }
                }
                // p = 2^(s*scale*log2e - m2) from the registers, row sum in two packed partial
                // sums, P packed to 16 bits and stored over the score columns (all already read).
                {
                    const float2 negm2 = make_float2(-m2, -m2);
                    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float2 x = make_float2(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1]));
                            float2 y = __ffma2_rn(x, scale2, negm2);
                            y.x = ex2_approx(y.x);
                            y.y = ex2_approx(y.y);
                            if (i & 1) acc1 = __fadd2_rn(acc1, y);
                            else acc0 = __fadd2_rn(acc0, y);
                            pk[i] = pack2<kBf16>(y.x, y.y);
                        }
                        tmem_st16(s_addr + 16u * c, pk);
                    }
                    l += (acc0.x + acc1.x) + (acc0.y + acc1.y);
                }
                // The O rescale, when some row's reference maximum moved: before P is released
                // to the P.V product (which is issued only after the arrival below), and after
                // the previous P.V product (whose completion preceded this S tile's).
                if (rescale) {
#pragma unroll
                    for (int c = 0; c < kNV * D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(o_addr + 32u * c, o);
                        tmem_ld_wait();
                        reg_fence(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(o_addr + 32u * c, o);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
            }
            // P of this tile ready for the issuer
            if constexpr (C::kNamed) nb_arrive(kNbP + t, BM + 32);
            else mbar_arrive(B_PF(t));
        }
        if (ok) ok = warp_wait(B_OD, 0, wd);
        if (C::kNamed && splits > 1) {
            ep_m2 = m2;
            ep_l = l;
            ep_ok = ok;
        } else if (ok) {
            tc_fence_after();
            const int row = q0 + t * BM + quarter * 32 + lane;
            const float inv_l = 1.f / l;
#pragma unroll
            for (int v = 0; v < kNV; ++v) {
                // rows of d_act <= D elements: the columns past d_act (zeros from the padded
                // tiles) are never stored
                uint16_t* orow = reinterpret_cast<uint16_t*>(v ? o2_ptr : o_ptr) + ((size_t)bh * n_q + row) * d_act;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(o_addr + (uint32_t)(v * D) + 32u * c, r);
                    tmem_ld_wait();
                    reg_fence(r);
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack2<kBf16>(__uint_as_float(r[2 * i]) * inv_l, __uint_as_float(r[2 * i + 1]) * inv_l);
                    if (row < n_q) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
                        for (int w = 0; w < 4; ++w)
                            if (32 * c + 8 * w < d_act)
                                dst[w] = make_uint4(pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
                    }
                }
            }
            if (row < n_q) lse_ptr[(size_t)bh * n_q + row] = (m2 + lg2_approx(l)) * kLn2;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (C::kNamed && splits > 1) {  // (the two-value form never splits)
        // Every thread of every CTA of the cluster meets at each of the three barriers.
        const bool row_thread = warp >= 2 && warp < 10;  // the softmax threads: one query row each
        const int t = (warp - 2) >> 2, quarter = warp & 3;
        const int row_l = t * BM + quarter * 32 + lane;  // row within the pair, 0..255
        const int w = D / splits;                         // columns this CTA stores: [rank w, rank w + w)
        const uint32_t ml = base + C::kExchMl, recv = base + C::kExchRecv;
        cluster_sync_all();  // every CTA has left its key loop: its Q/K/V buffers are free
        if (row_thread)
            for (int r = 0; r < splits; ++r)
                st_cluster_v2(cluster_map(ml + (uint32_t)((rank * 256 + row_l) * 8), (uint32_t)r), ep_m2, ep_l);
        cluster_sync_all();
        float big_m = -INFINITY, big_l = 0.f;
        if (row_thread) {
            const float2* mlp = reinterpret_cast<const float2*>(smem + C::kExchMl);
            for (int r = 0; r < splits; ++r) big_m = fmaxf(big_m, mlp[r * 256 + row_l].x);
            for (int r = 0; r < splits; ++r) big_l += mlp[r * 256 + row_l].y * ex2_approx(mlp[r * 256 + row_l].x - big_m);
            const float f = ep_ok ? ex2_approx(ep_m2 - big_m) / big_l : 0.f;
            tc_fence_after();
            const uint32_t o_addr = tmem + ((uint32_t)(quarter * 32) << 16) + 256u + (uint32_t)(t * D);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(o_addr + 32u * c, r);
                tmem_ld_wait();
                reg_fence(r);
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const int col = 32 * c + 4 * g, owner = col / w;
                    const uint32_t dst = recv + (uint32_t)(((rank * 256 + row_l) * w + col - owner * w) * 4);
                    // a row whose waits failed sends exact zeros (its tensor memory may hold anything)
                    st_cluster_v4(cluster_map(dst, (uint32_t)owner), ep_ok ? __uint_as_float(r[4 * g]) * f : 0.f,
                                  ep_ok ? __uint_as_float(r[4 * g + 1]) * f : 0.f,
                                  ep_ok ? __uint_as_float(r[4 * g + 2]) * f : 0.f,
                                  ep_ok ? __uint_as_float(r[4 * g + 3]) * f : 0.f);
                }
            }
        }
        cluster_sync_all();
        if (row_thread) {
            const float* part = reinterpret_cast<const float*>(smem + C::kExchRecv);
            const int row = q0 + row_l;
            uint16_t* orow = reinterpret_cast<uint16_t*>(o_ptr) + ((size_t)bh * n_q + row) * d_act;
            for (int g = 0; g < w; g += 4) {
                float a[4] = {0.f, 0.f, 0.f, 0.f};
                for (int r = 0; r < splits; ++r)  // in rank order
#pragma unroll
                    for (int i = 0; i < 4; ++i) a[i] += part[(r * 256 + row_l) * w + g + i];
                const int col = rank * w + g;  // d_act is a multiple of 8: a 4-column group is all in or all out
                if (row < n_q && col < d_act)
                    *reinterpret_cast<uint2*>(orow + col) = make_uint2(pack2<kBf16>(a[0], a[1]), pack2<kBf16>(a[2], a[3]));
            }
            if (rank == 0 && row < n_q) lse_ptr[(size_t)bh * n_q + row] = (big_m + lg2_approx(big_l)) * kLn2;
        }
        tc_fence_before();
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, bool kBf16, int kNV>
cudaError_t launch_impl(const FwdParams& p, cudaStream_t stream, int slot) {
    using C = FwdCfg<D, kNV>;
    const CUtensorMapDataType dt = kBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUtensorMapSwizzle sw = D >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    CUtensorMap tq, tk, tv, tv2;
    // maps over the true head dimension p.d <= D: TMA fills the box columns past it with zeros
    const uint64_t d = (uint64_t)p.d;
    if (!encode_tmap_3d(&tq, dt, 2, p.q, d, (uint64_t)p.n_q, (uint64_t)p.bh, C::kAtomCols, BM, sw) ||
        !encode_tmap_3d(&tk, dt, 2, p.k, d, (uint64_t)p.n_k, (uint64_t)p.bh, C::kAtomCols, BN, sw) ||
        !encode_tmap_3d(&tv, dt, 2, p.v, d, (uint64_t)p.n_k, (uint64_t)p.bh, C::kAtomCols, BN, sw) ||
        !encode_tmap_3d(&tv2, dt, 2, kNV == 2 ? p.v2 : p.v, d, (uint64_t)p.n_k, (uint64_t)p.bh, C::kAtomCols, BN, sw))
        return cudaErrorInvalidValue;
    auto kern = fa2_fwd_tc_kernel<D, kBf16, kNV>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), C::kSmemBytes, slot);
    if (e != cudaSuccess) return e;
    const int64_t pairs = (p.n_q + BM * kQTiles - 1) / (BM * kQTiles);
    const float scale_log2 = p.scale * 1.4426950408889634f;
    int splits = kNV == 1 ? fwd_key_splits(pairs * p.bh, (p.n_k + BN - 1) / BN, D) : 1;
    // a device that cannot hold the whole cluster at once takes fewer ranges
    while (splits > 1 && !cluster_fits(reinterpret_cast<const void*>(kern), C::kThreads, C::kSmemBytes, splits, slot))
        splits /= 2;
    launch_record().fwd_key_ranges = splits;
    if (splits == 1) {
        const dim3 grid((unsigned)pairs, (unsigned)p.bh, 1);
        kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, tv2, p.o, p.o2, p.lse, (int)p.n_q, (int)p.n_k,
                                                        p.d, scale_log2, p.status, 1);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(pairs * splits), (unsigned)p.bh, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tv2, p.o, p.o2, p.lse, (int)p.n_q, (int)p.n_k, p.d, scale_log2,
                              p.status, splits);
}

}  // namespace

cudaError_t launch_fwd_tc(const FwdParams& p, cudaStream_t stream) {
    const bool bf = p.dtype == kBf16;
    switch (pad_head_dim(p.d)) {
        case 32: return bf ? launch_impl<32, true, 1>(p, stream, 0) : launch_impl<32, false, 1>(p, stream, 1);
        case 64: return bf ? launch_impl<64, true, 1>(p, stream, 2) : launch_impl<64, false, 1>(p, stream, 3);
        case 128: return bf ? launch_impl<128, true, 1>(p, stream, 4) : launch_impl<128, false, 1>(p, stream, 5);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_fwd_tc_dual_v(const FwdParams& p, cudaStream_t stream) {
    const bool bf = p.dtype == kBf16;
    switch (pad_head_dim(p.d)) {
        case 32: return bf ? launch_impl<32, true, 2>(p, stream, 6) : launch_impl<32, false, 2>(p, stream, 7);
        case 64: return bf ? launch_impl<64, true, 2>(p, stream, 8) : launch_impl<64, false, 2>(p, stream, 9);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa2
