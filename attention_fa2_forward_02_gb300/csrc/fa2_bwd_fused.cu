// fa2_bwd_fused.cu - attention backward in one pass over key tiles, on the
// sm_103a tensor cores (tcgen05 + TMEM + TMA), for kernel head sizes 32 and 64.
//
// What it computes: the gradients of "vision-rs 0.1.1 flash_attn2.rs", kernels
// flash_attention2_backward_dq and flash_attention2_backward_dkv:
//   P_ij = exp(s_ij - LSE_i),  dV_j = sum_i P_ij dO_i,  dS_ij = P_ij (dO_i . v_j - D_i),
//   dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j.
// That page computes dQ in a pass of its own over query rows, which forms S and
// dP a second time.  Here the pass over key tiles also forms the product
// dS_(i,j) K_j of the query tile i it is visiting and adds it into a float32 dQ
// accumulator in the workspace; a last small kernel scales the sums and rounds
// them into dq.  Each dQ element is then a float32 sum of per-key-tile float32
// partial sums, added in whatever order the CTAs reach it (not bit-reproducible
// from run to run).
//
// Per CTA: one 128-key tile (K, V resident in shared memory), looping over the
// query tiles of its head starting at tile (key tile index mod n_qt), so that the
// CTAs of a head add into different query tiles at any one time.
// Tensor memory (512 columns x 128 lanes):
//   [0, 128)      S^T = K Q^T; then P^T, 16-bit, in columns [32, 96)
//   [128, 256)    dP^T = V dO^T; then dS^T, 16-bit, in [160, 224)
//   [256, 256+D) dV    [256+D, 256+2D) dK    [256+2D+b*D, 256+3D+b*D) dQ of query
//   tiles with i % 2 == b: two buffers, so that the next dP^T need not wait for the
//   current dQ to be read out.
// dS itself (queries x keys, the A operand of the dQ product) is written by the
// elementwise warps into a shared-memory buffer of its own.
//
// The dQ additions leave the elementwise warps' path: each warp copies its 32 rows x
// D/2 columns of a finished dQ tile out of tensor memory into a 4 KB (D = 64) block of
// shared memory and one of its lanes hands that block to the TMA engine as one bulk
// float32 reduction into the accumulator (cp.reduce.async.bulk ... add.f32); the engine
// performs the additions in L2 while the warps go on.  Before the warp rewrites its
// block for the next tile, that lane waits until the engine has read the previous one.
// The accumulator is laid out per (head, query tile) as [4 quarters][2 halves][D/8]
// [32 rows][4 floats] (quarter = row / 32, half = column / (D/2)), so that each warp's
// block is one contiguous run and the rounding kernel still reads 512 contiguous bytes
// per warp.  At the end the CTA's dK and dV leave by TMA stores, each warp staging its
// 32-row chunks in the same block.
//
// MMA order per query tile i (one thread issues, the tensor core runs in order; S^T(0)
// and dP^T(0) first):
//   [e1(i)] dV += P^T(i) dO(i);  [stage i+1] S^T(i+1) -> s_full;
//   [e2(i)] dK += dS^T(i) Q(i);  dQ_i = dS(i) K -> dq_full, empty;  dP^T(i+1) -> dp_full
// The bracketed events reach the issuing warp as named barriers: e1, e2 from the
// elementwise warps, "stage loaded" from a relay warp (warp 10) that waits on the
// TMA barriers.  dQ_i goes to buffer i % 2, last written by dQ_(i-2), which the warps
// read out before their e2(i-1) arrival: no barrier of its own.
// Elementwise warps per query tile i:
//   [s_full] P^T(i) -> e1;  [dq_full(i-1)] dQ_(i-1) to shared memory, bulk reduction;
//   [dp_full] dS^T(i) into TMEM, dS(i) into shared memory -> e2
// so the warps compute P under dK, dQ and dP^T, stage dQ under dV and compute dS under
// S^T, while the tensor core runs dV, S^T, dK, dQ, dP^T back to back; dP^T(i) is
// complete by the time the warps turn to dS(i).
// In-order execution of the tensor core is what makes the column reuse safe: an
// MMA that overwrites columns another reads (S^T(i+1) over P^T(i), dP^T(i+1) over
// dS^T(i)) is always issued after the MMA that reads them.
#include "bwd_common.cuh"
#include "internal.h"

namespace fa2 {
namespace {

template <int D>
struct FusedCfg : Tile16<D> {
    static_assert(D == 32 || D == 64, "the one-pass kernel serves head sizes up to 64");
    static constexpr int kStages = D == 64 ? 3 : 4;
    static constexpr int kTile = BT * D * 2;
    static constexpr int kDsBytes = BT * BT * 2;
    // per elementwise warp: 32 rows x D/2 float32 of a dQ tile, staged for the bulk reduction
    static constexpr int kDqBlockBytes = 32 * (D / 2) * 4;
    // K, V resident; per stage Q_i, dO_i, lse2_i, delta_i; the dS buffer; the dQ blocks; barriers
    static constexpr int kStage = 2 * kTile + 2 * BT * 4;
    static constexpr int kSmemStages = 2 * kTile;
    static constexpr int kSmemDs = kSmemStages + kStages * kStage;
    static constexpr int kSmemDq = kSmemDs + kDsBytes;
    static constexpr int kSmemBar = kSmemDq + 8 * kDqBlockBytes;
    static constexpr int kNumBars = 2 * kStages + kBwdBars;
    static constexpr int kSmemBytes = kSmemBar + kNumBars * 8 + 16 + 1024;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(kStage % 1024 == 0 && kSmemDs % 1024 == 0, "operand alignment");
    static constexpr uint32_t kDqCol = 256 + 2 * D;  // the two dQ buffers
    static_assert(kDqCol + 2 * D <= kBwdTmemCols, "tensor memory budget");
    static constexpr int kThreads = kBwdThreads + 32;  // + the TMA relay warp
};

// Named barriers of this kernel besides kNbE1 / kNbE2: stage s loaded.
__host__ __device__ constexpr uint32_t nb_fstage(int s) { return 3 + (uint32_t)s; }

template <int D, bool kBf16>
__global__ void __launch_bounds__(FusedCfg<D>::kThreads, 1)
    bwd_fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                     const float* __restrict__ lse2, const float* __restrict__ delta, float* __restrict__ dq_acc,
                     void* __restrict__ dk, void* __restrict__ dv, int n_q, int n_k, int n_q_pad, int d_act, float scale,
                     float scale_log2, unsigned int* status) {
    using C = FusedCfg<D>;
    using DsTile = Tile16<BT>;  // dS as a [keys, queries] tile: MN-major A operand of the dQ product
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_addr);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y;
    const int k0 = blockIdx.x * BT;
    const int n_qt = (n_q + BT - 1) / BT;
    const int qt_first = blockIdx.x % n_qt;
    auto qtile = [&](int i) { return (i + qt_first) % n_qt; };

    const Bars bars{base + C::kSmemBar, S};
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kSmemBar + C::kNumBars * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kSmemBar + C::kNumBars * 8 + 4);
    const Watchdog wd{abort_flag, status};
    const uint32_t k_smem = base;
    const uint32_t v_smem = base + C::kTile;
    auto stage_q = [&](int s) { return base + C::kSmemStages + s * C::kStage; };
    auto stage_do = [&](int s) { return stage_q(s) + C::kTile; };
    auto stage_l2 = [&](int s) { return stage_q(s) + 2 * C::kTile; };
    auto stage_dl = [&](int s) { return stage_l2(s) + BT * 4; };
    const uint32_t ds_smem = base + C::kSmemDs;

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
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_do);
            mbar_arrive_expect_tx(bars.resident(), 2 * C::kTile);
            for (int a = 0; a < C::kAtoms; ++a) {
                tma_load_3d(k_smem + a * BT * C::kAtomRowBytes, &tm_k, bars.resident(), a * C::kAtomCols, k0, bh);
                tma_load_3d(v_smem + a * BT * C::kAtomRowBytes, &tm_v, bars.resident(), a * C::kAtomCols, k0, bh);
            }
            int issued = 0;
            bool ok = true;
            for (int i = 0; i < n_qt; ++i) {
                const int s = i % S;
                const int qt = qtile(i);
                if (i >= S && !(ok = mbar_wait(bars.empty(s), ((i / S) & 1) ^ 1, wd))) break;
                mbar_arrive_expect_tx(bars.full(s), 2 * C::kTile + 2 * BT * 4);
                for (int a = 0; a < C::kAtoms; ++a) {
                    tma_load_3d(stage_q(s) + a * BT * C::kAtomRowBytes, &tm_q, bars.full(s), a * C::kAtomCols, qt * BT, bh);
                    tma_load_3d(stage_do(s) + a * BT * C::kAtomRowBytes, &tm_do, bars.full(s), a * C::kAtomCols, qt * BT,
                                bh);
                }
                const size_t w = (size_t)bh * n_q_pad + (size_t)qt * BT;
                bulk_load(stage_l2(s), lse2 + w, BT * 4, bars.full(s));
                bulk_load(stage_dl(s), delta + w, BT * 4, bars.full(s));
                issued = i + 1;
            }
            if (!ok) {
                drain_wait(bars.resident(), 0);
                for (int i = (issued > S ? issued - S : 0); i < issued; ++i) drain_wait(bars.full(i % S), (i / S) & 1);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        // The whole warp syncs on the named barriers; lane 0 issues.
        const uint32_t idesc_s = idesc_f16_f32acc(BT, BT, kBf16, false, false);  // S^T, dP^T
        const uint32_t idesc_g = idesc_f16_f32acc(BT, D, kBf16, false, true);    // dV, dK: A from TMEM
        const uint32_t idesc_q = idesc_f16_f32acc(BT, D, kBf16, true, true);     // dQ: both MN-major
        // Descriptors built once (stage 0, k-step 0); every other operand adds a constant
        // to the start-address field (16-byte units; shared addresses stay below 256 KB).
        const uint64_t dk0 = C::kmajor(k_smem, 0, BT), dv0 = C::kmajor(v_smem, 0, BT);
        const uint64_t dq0 = C::kmajor(stage_q(0), 0, BT), ddo0 = C::kmajor(stage_do(0), 0, BT);
        const uint64_t mq0 = C::mnmajor(stage_q(0), 0, BT), mdo0 = C::mnmajor(stage_do(0), 0, BT);
        const uint64_t mk0 = C::mnmajor(k_smem, 0, BT), mds0 = DsTile::mnmajor(ds_smem, 0, BT);
        auto st_off = [&](int s) { return (uint64_t)((s * C::kStage) >> 4); };
        auto issue_st = [&](int s) {  // S^T = K Q^T
            const uint64_t b = dq0 + st_off(s);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t o = (uint64_t)(C::koff(kk, BT) >> 4);
                mma_ss(tmem, dk0 + o, b + o, idesc_s, kk > 0);
            }
        };
        static_assert(nb_fstage(S - 1) < 16, "named barriers");
        auto issue_dpt = [&](int s) {  // dP^T = V dO^T
            const uint64_t bd = ddo0 + st_off(s);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t o = (uint64_t)(C::koff(kk, BT) >> 4);
                mma_ss(tmem + 128u, dv0 + o, bd + o, idesc_s, kk > 0);
            }
            mma_commit(bars.dp_full());
        };
        nb_sync(nb_fstage(0), 64);  // K, V and the first Q / dO stage
        if (lane == 0) {
            tc_fence_after();
            issue_st(0);
            mma_commit(bars.s_full());
            issue_dpt(0);
        }
        __syncwarp();
        for (int i = 0; i < n_qt; ++i) {
            const int s = i % S;
            const int sn = (i + 1) % S;
            const bool more = i + 1 < n_qt;
            nb_sync(kNbE1, kNbElem);  // P^T(i) in tensor memory
            if (lane == 0) {
                tc_fence_after();
                const uint64_t b = mdo0 + st_off(s);
#pragma unroll
                for (int kk = 0; kk < BT / 16; ++kk)  // dV += P^T dO
                    mma_ts(tmem + 256u, tmem + kPackedCol + (uint32_t)(kk * 8), b + (uint64_t)(kk * C::kAtomRowBytes),
                           idesc_g, (i > 0 || kk > 0));
            }
            __syncwarp();
            if (more) {
                nb_sync(nb_fstage(sn), 64);  // Q, dO of tile i + 1
                if (lane == 0) {
                    tc_fence_after();
                    issue_st(sn);
                    mma_commit(bars.s_full());
                }
                __syncwarp();
            }
            nb_sync(kNbE2, kNbElem);  // dS^T(i) in tensor memory, dS(i) in shared memory
            if (lane == 0) {
                tc_fence_after();
                const uint64_t b = mq0 + st_off(s);
#pragma unroll
                for (int kk = 0; kk < BT / 16; ++kk)  // dK += dS^T Q
                    mma_ts(tmem + 256u + (uint32_t)D, tmem + 128u + kPackedCol + (uint32_t)(kk * 8),
                           b + (uint64_t)(kk * C::kAtomRowBytes), idesc_g, (i > 0 || kk > 0));
#pragma unroll
                for (int kk = 0; kk < BT / 16; ++kk)  // dQ_i = dS K (keys are the reduction dimension)
                    mma_ss(tmem + C::kDqCol + (uint32_t)((i & 1) * D), mds0 + (uint64_t)(kk * DsTile::kAtomRowBytes),
                           mk0 + (uint64_t)(kk * C::kAtomRowBytes), idesc_q, kk > 0);
                mma_commit(bars.dq_full());
                mma_commit(bars.empty(s));
                if (more) issue_dpt(sn);  // over dS^T(i), which dK(i) has been issued to read
            }
            __syncwarp();
        }
        if (lane == 0) {
            mma_commit(bars.done());
            drain_wait(bars.done(), 0);
        }
        __syncwarp();
    } else if (warp == kBwdRelayWarp) {
        // ------------------------------------------------------------------ TMA relay
        bool ok = warp_wait(bars.resident(), 0, wd) && warp_wait(bars.full(0), 0, wd);
        nb_arrive(nb_fstage(0), 64);
        for (int i = 1; i < n_qt; ++i) {
            const int s = i % S;
            ok = ok && warp_wait(bars.full(s), (i / S) & 1, wd);
            nb_arrive(nb_fstage(s), 64);
        }
    } else {
        // ------------------------------------------------------------------ elementwise warps
        // Two warps per TMEM lane quarter; warp `half` owns query columns [64*half, 64*half + 64)
        // of the score tiles and dQ columns [half*D/2, half*D/2 + D/2).
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t t_s = tmem + lane_off, t_dp = tmem + lane_off + 128u;
        const int r = quarter * 32 + lane;  // key row (score tiles) and query row (dQ tile) of this thread
        const uint32_t t_dq0 = tmem + lane_off + C::kDqCol + (uint32_t)(half * (D / 2));
        const bool key_valid = k0 + r < n_k;
        const float2 scale2 = make_float2(scale_log2, scale_log2);
        // dQ of the i-th visited query tile: this warp's 32 rows x D/2 columns out of TMEM
        // into its block of shared memory, then one bulk float32 reduction of the block into
        // the accumulator by lane 0 (see the layout above). A failed wait skips the work.
        const uint32_t dq_block = base + C::kSmemDq + (uint32_t)((warp - 2) * C::kDqBlockBytes);
        auto reduce_dq = [&](int i, bool ok) -> bool {
            if (!(ok && warp_wait(bars.dq_full(), i & 1, wd))) return false;
            tc_fence_after();
            uint32_t v[D / 2];
            if constexpr (D == 64) tmem_ld32(t_dq0 + (uint32_t)((i & 1) * D), v);
            else tmem_ld16(t_dq0 + (uint32_t)((i & 1) * D), v);
            if (lane == 0) bulk_wait_group_read0();  // the engine has read this block's previous contents
            tmem_ld_wait();
            reg_fence(v);
            __syncwarp();
#pragma unroll
            for (int g = 0; g < D / 8; ++g)  // [D/8][32 rows][4 floats]
                st_shared_v4(dq_block + (uint32_t)((g * 32 + lane) * 16), v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                float* tile = dq_acc + ((size_t)bh * n_qt + qtile(i)) * (size_t)(BT * D) +
                              (size_t)(quarter * 2 + half) * (C::kDqBlockBytes / 4);
                bulk_reduce_add_f32(tile, dq_block, C::kDqBlockBytes);
                bulk_commit_group();
            }
            return true;
        };
        bool ok = true;
        for (int i = 0; i < n_qt; ++i) {
            const int s = i % S;
            if (!(ok = ok && warp_wait(bars.s_full(), i & 1, wd) && warp_wait(bars.full(s), (i / S) & 1, wd))) {
                nb_arrive(kNbE1, kNbElem);
                nb_arrive(kNbE2, kNbElem);
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
                    const uint32_t* rr = cc == 0 ? ra : rb;
                    uint32_t pk[16];
#pragma unroll
                    for (int x = 0; x < 16; x += 2) {
                        const float4 nl = *reinterpret_cast<const float4*>(l2 + 32 * c + 2 * x);  // -LSE2, 4 queries
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            float2 v = __ffma2_rn(make_float2(__uint_as_float(rr[2 * (x + u)]), __uint_as_float(rr[2 * (x + u) + 1])),
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
            nb_arrive(kNbE1, kNbElem);
            // the previous query tile's dQ, while dV(i) and dP^T(i) run
            if (i > 0) ok = reduce_dq(i - 1, ok);
            // step 2: dS^T = P^T * (dP^T - D) into TMEM (for dK) and as dS into shared memory
            // (for dQ); both owned chunks read before either is overwritten.  Rows of keys
            // past the last one (zero K rows, where P may even overflow) get dS = 0.
            if (!(ok = ok && warp_wait(bars.dp_full(), i & 1, wd))) {
                nb_arrive(kNbE2, kNbElem);
                continue;
            }
            tc_fence_after();
            const uint32_t ds_row = ds_smem + (uint32_t)r * 128u;  // row r of the [keys, queries] tile
            const uint32_t swz = (uint32_t)(r & 7);                   // 128-byte swizzle of that row
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
                for (int x = 0; x < 16; x += 2) {
                    const float4 nd = *reinterpret_cast<const float4*>(dl + 32 * c + 2 * x);  // -D, 4 queries
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float2 ds = __fmul2_rn(
                            p[cc][x + u], __fadd2_rn(make_float2(__uint_as_float(rp[cc][2 * (x + u)]), __uint_as_float(rp[cc][2 * (x + u) + 1])),
                                                     u ? make_float2(nd.z, nd.w) : make_float2(nd.x, nd.y)));
                        pk[x + u] = key_valid ? pack2<kBf16>(ds.x, ds.y) : 0u;
                    }
                }
                tmem_st16(t_dp + kPackedCol + 16u * c, pk);
                // queries [32c, 32c + 32): 64-column atom c / 2, 16-byte chunks 4 (c % 2) .. + 3
                const uint32_t atom = ds_row + (uint32_t)(c >> 1) * (uint32_t)(BT * 128);
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    st_shared_v4(atom + (((uint32_t)((c & 1) * 4 + w) ^ swz) << 4), pk[4 * w], pk[4 * w + 1],
                                 pk[4 * w + 2], pk[4 * w + 3]);
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            nb_arrive(kNbE2, kNbElem);
        }
        if (n_qt > 0) ok = reduce_dq(n_qt - 1, ok);
        if (lane == 0) bulk_wait_group0();  // this warp's reductions complete before the CTA exits
        __syncwarp();
        if (ok) ok = warp_wait(bars.done(), 0, wd);
        if (ok) {
            tc_fence_after();
            // half 0 writes dV, half 1 writes dK (scaled); the warp's dQ block (its bulk
            // reductions complete) serves as the slab of the TMA stores
            const uint32_t src = tmem + lane_off + 256u + (uint32_t)(half * D);
            const float mul = half ? scale : 1.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(src + 32u * c, v);
                tmem_ld_wait();
                reg_fence(v);
                store_chunk_tma<kBf16>(half ? &tm_dk : &tm_dv, dq_block, 32 * c, k0 + quarter * 32, n_k, d_act, bh, v, mul);
            }
            if (lane == 0) bulk_wait_group0();  // the stores complete before the CTA exits
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

// dq[bh, row, :d_act] = scale * the accumulated sums, rounded to the 16-bit dtype.
// One thread per query row; for each 4-column group a warp's loads cover 512
// contiguous bytes of the [quarter][half][D/8][32 rows][4] tile layout.
template <int D, bool kBf16>
__global__ void __launch_bounds__(BT)
    bwd_dq_round_kernel(const float4* __restrict__ dq_acc, void* __restrict__ dq, int n_q, int d_act, float scale) {
    const int qt = blockIdx.x, bh = blockIdx.y, r = threadIdx.x;
    const int row = qt * BT + r;
    if (row >= n_q) return;
    const int n_qt = gridDim.x;
    const float4* tile = dq_acc + ((size_t)bh * n_qt + qt) * (size_t)(D / 4) * BT;
    uint4* out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(dq) + ((size_t)bh * n_q + row) * d_act);
    const int quarter = r >> 5, lane = r & 31;
#pragma unroll
    for (int g = 0; g < D / 8; ++g) {  // output columns [8g, 8g + 8): float4 groups 2g and 2g + 1
        if (8 * g >= d_act) break;
        float4 ab[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int c4 = 2 * g + u;                          // 4-column group of the row
            const int half = c4 / (D / 8), gi = c4 % (D / 8);  // its half and group within the half
            ab[u] = tile[(size_t)((quarter * 2 + half) * (D / 8) + gi) * 32 + lane];
        }
        const float4 a = ab[0], b = ab[1];
        out[g] = make_uint4(pack2<kBf16>(a.x * scale, a.y * scale), pack2<kBf16>(a.z * scale, a.w * scale),
                            pack2<kBf16>(b.x * scale, b.y * scale), pack2<kBf16>(b.z * scale, b.w * scale));
    }
}

template <int D, bool kBf16>
cudaError_t fused_impl(const BwdParams& p, cudaStream_t stream, int slot) {
    using C = FusedCfg<D>;
    if (!p.dq_acc) return cudaErrorInvalidValue;
    cudaError_t e = launch_bwd_tc(p, stream, kBwdPreprocess);  // D, LSE2, zeroed accumulator
    if (e != cudaSuccess) return e;
    const CUtensorMapDataType dt = kBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUtensorMapSwizzle sw = D >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    CUtensorMap tq, tk, tv, tdo, tdk, tdv;
    // maps over the true head dimension p.d <= D: TMA fills the box columns past it with zeros
    const uint64_t d = (uint64_t)p.d;
    if (!encode_tmap_3d(&tq, dt, 2, p.q, d, (uint64_t)p.n_q, (uint64_t)p.bh, C::kAtomCols, BT, sw) ||
        !encode_tmap_3d(&tdo, dt, 2, p.d_o, d, (uint64_t)p.n_q, (uint64_t)p.bh, C::kAtomCols, BT, sw) ||
        !encode_tmap_3d(&tk, dt, 2, p.k, d, (uint64_t)p.n_k, (uint64_t)p.bh, C::kAtomCols, BT, sw) ||
        !encode_tmap_3d(&tv, dt, 2, p.v, d, (uint64_t)p.n_k, (uint64_t)p.bh, C::kAtomCols, BT, sw) ||
        !encode_tmap_3d(&tdk, dt, 2, p.dk, d, (uint64_t)p.n_k, (uint64_t)p.bh, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tmap_3d(&tdv, dt, 2, p.dv, d, (uint64_t)p.n_k, (uint64_t)p.bh, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    auto kern = bwd_fused_kernel<D, kBf16>;
    e = ensure_smem_limit(reinterpret_cast<const void*>(kern), C::kSmemBytes, slot);
    if (e != cudaSuccess) return e;
    const int n_qt = (int)((p.n_q + BT - 1) / BT);
    kern<<<dim3((unsigned)((p.n_k + BT - 1) / BT), (unsigned)p.bh, 1), C::kThreads, C::kSmemBytes, stream>>>(
        tq, tk, tv, tdo, tdk, tdv, p.lse2, p.delta, p.dq_acc, p.dk, p.dv, (int)p.n_q, (int)p.n_k, (int)p.n_q_pad, p.d, p.scale,
        p.scale * kLog2e, p.status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bwd_dq_round_kernel<D, kBf16><<<dim3((unsigned)n_qt, (unsigned)p.bh, 1), BT, 0, stream>>>(
        reinterpret_cast<const float4*>(p.dq_acc), p.dq, (int)p.n_q, p.d, p.scale);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_fused(const BwdParams& p, cudaStream_t stream) {
    const bool bf = p.dtype == kBf16;
    switch (pad_head_dim(p.d)) {
        case 32: return bf ? fused_impl<32, true>(p, stream, 36) : fused_impl<32, false>(p, stream, 37);
        case 64: return bf ? fused_impl<64, true>(p, stream, 38) : fused_impl<64, false>(p, stream, 39);
        default: return cudaErrorInvalidValue;  // head sizes above 64 run the two-pass kernels
    }
}

}  // namespace fa2
