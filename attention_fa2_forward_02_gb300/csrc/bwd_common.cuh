// bwd_common.cuh - constants, barriers and store helpers shared by the backward
// kernels (the two-pass kernels in fa2_bwd_tc.cu, the one-pass kernel in
// fa2_bwd_fused.cu).
#pragma once

#include "common.cuh"

namespace fa2 {

constexpr int BT = 128;         // rows of every tile (keys or queries)
constexpr int kBwdThreads = 320;   // warp 0 TMA, warp 1 MMA, warps 2-9 elementwise
constexpr int kElemThreads = 256;
// The 16-bit probabilities / dS of a 128-column fp32 score tile occupy 64 columns
// starting at column 32 of that tile: the warp owning score columns [0, 64)
// writes [32, 64) and the one owning [64, 128) writes [64, 96), so each warp only
// overwrites columns it has itself already read.
constexpr uint32_t kPackedCol = 32;
constexpr uint32_t kBwdTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBwdBars = 9;  // barriers besides the per-stage full / empty pairs

// Named barriers (bar.arrive by the producers, bar.sync by the whole issuing warp) in
// place of mbarrier waits in the MMA issuer: a shared-memory access by the issuing warp
// between MMA groups, an mbarrier test included, costs a few hundred clocks of
// tensor-pipe time. Warp kBwdRelayWarp waits for the TMA stages and relays them. A
// producer cannot arrive twice on one barrier before the issuer has synced on it, and
// arrives once per event whatever happens (a failed bounded wait skips its work, not its
// arrival, and raises the watchdog status); the issuer never gives up.
constexpr int kBwdRelayWarp = 10;
constexpr uint32_t kNbE1 = 1, kNbE2 = 2;
constexpr uint32_t kNbElem = kElemThreads + 32;  // elementwise warps + issuer

// Barriers of the backward kernels:
//   resident  K, V loaded once per CTA (TMA transaction count); in the dQ pass,
//             Q and dO copied into tensor memory (256 arrivals)
//   full[s]   stage s loaded                         (TMA transaction count)
//   empty[s]  stage s no longer read by any MMA      (tcgen05.commit)
//   s_full    the first score tile (S^T or S) is in TMEM   (tcgen05.commit)
//   dp_full   the second score tile (dP^T or dP) is in TMEM (tcgen05.commit)
//   e1        elementwise step 1 done: P^T is in TMEM (dK/dV passes); S has
//             been read (dQ pass)                    (256 arrivals)
//   e2        elementwise step 2 done: dS^T / dS is in place (256 arrivals)
//   dq_full   one-pass kernel: the dQ product of a query tile is in TMEM (tcgen05.commit);
//             as dv_done in the dK/dV pass: every dV product of the current key tile has
//             completed                              (tcgen05.commit)
//   dq_read   one-pass kernel: that product has been read out (256 arrivals)
//   done      every MMA issued has completed; the dK/dV pass: every MMA of the
//             current key tile                       (tcgen05.commit)
//   kv_free   dK/dV pass over several key tiles: the last products reading the
//             current tile's K and V have completed  (tcgen05.commit)
struct Bars {
    uint32_t base;
    int S;
    __device__ uint32_t resident() const { return base; }
    __device__ uint32_t full(int s) const { return base + 8u * (1 + s); }
    __device__ uint32_t empty(int s) const { return base + 8u * (1 + S + s); }
    __device__ uint32_t s_full() const { return base + 8u * (1 + 2 * S); }
    __device__ uint32_t dp_full() const { return base + 8u * (2 + 2 * S); }
    __device__ uint32_t e1() const { return base + 8u * (3 + 2 * S); }
    __device__ uint32_t e2() const { return base + 8u * (4 + 2 * S); }
    __device__ uint32_t done() const { return base + 8u * (5 + 2 * S); }
    __device__ uint32_t dq_full() const { return base + 8u * (6 + 2 * S); }
    __device__ uint32_t dv_done() const { return dq_full(); }
    __device__ uint32_t dq_read() const { return base + 8u * (7 + 2 * S); }
    __device__ uint32_t kv_free() const { return base + 8u * (8 + 2 * S); }
};

__device__ __forceinline__ void init_bars(const Bars& b, volatile int* abort_flag, uint32_t resident_count) {
    *abort_flag = 0;
    mbar_init(b.resident(), resident_count);
    for (int s = 0; s < b.S; ++s) {
        mbar_init(b.full(s), 1);
        mbar_init(b.empty(s), 1);
    }
    mbar_init(b.s_full(), 1);
    mbar_init(b.dp_full(), 1);
    mbar_init(b.e1(), kElemThreads);
    mbar_init(b.e2(), kElemThreads);
    mbar_init(b.done(), 1);
    mbar_init(b.dq_full(), 1);
    mbar_init(b.dq_read(), kElemThreads);
    mbar_init(b.kv_free(), 1);
    fence_barrier_init();
}

// Stores columns [32c, 32c + 32) of a row of d_act elements (16-byte pieces past
// d_act, zeros of the padded tile, are skipped).
template <bool kBf16>
__device__ __forceinline__ void store_row_chunk(void* base, size_t row, int d_act, int c, const uint32_t (&r)[32],
                                                float mul, bool valid) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = pack2<kBf16>(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
    if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(base) + row * d_act + 32 * c);
#pragma unroll
        for (int v = 0; v < 4; ++v)
            if (32 * c + 8 * v < d_act) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
    }
}

// Gradient tiles written by TMA stores. Each elementwise warp owns 32 rows (its TMEM lane
// quarter) of a 128-row tile; per 32-column chunk it packs its rows into its own 2 KB slab
// of shared memory (32 rows x 64 bytes, the box of the output's tensor map) and one lane
// stores the box. Plain per-thread stores would write a 16-byte piece of a different row
// (a different cache line) per lane and instruction; the TMA writes whole rows. The map's
// bounds clip the rows past the last one and the columns past the head size.
constexpr int kOutSlabBytes = 32 * 32 * 2;
constexpr int kOutStageBytes = 8 * kOutSlabBytes;  // one slab per elementwise warp

template <bool kBf16>
__device__ __forceinline__ void store_chunk_tma(const CUtensorMap* map, uint32_t slab, int col0, int row0, int n_rows,
                                                int d_act, int bh, const uint32_t (&r)[32], float mul) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = pack2<kBf16>(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
    if (lane_id() == 0) bulk_wait_group_read0();  // the previous store has read the slab
    __syncwarp();
    const uint32_t row = slab + lane_id() * 64u;
#pragma unroll
    for (int w = 0; w < 4; ++w) st_shared_v4(row + 16u * w, pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane_id() == 0 && row0 < n_rows && col0 < d_act) {
        tma_store_3d(map, slab, col0, row0, bh);
        bulk_commit_group();
    }
}

// The float32 form: 16 of the 32 columns in r (from `first`) as one box of 32 rows x 64
// bytes, stored unscaled into plane `plane` (the boxes always lie inside that tensor).
__device__ __forceinline__ void store_chunk_tma_f32(const CUtensorMap* map, uint32_t slab, int col0, int row0, int plane,
                                                    const uint32_t (&r)[32], int first) {
    if (lane_id() == 0) bulk_wait_group_read0();  // the previous store has read the slab
    __syncwarp();
    const uint32_t row = slab + lane_id() * 64u;
#pragma unroll
    for (int w = 0; w < 4; ++w)
        st_shared_v4(row + 16u * w, r[first + 4 * w], r[first + 4 * w + 1], r[first + 4 * w + 2], r[first + 4 * w + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane_id() == 0) {
        tma_store_3d(map, slab, col0, row0, plane);
        bulk_commit_group();
    }
}

// The two 32-column chunks an elementwise warp owns, in the order that lets it
// write 16-bit results at kPackedCol without overwriting a column it has not read.
__device__ __forceinline__ int owned_chunk(int half, int cc) { return 2 * half + (half == 0 ? 1 - cc : cc); }

}  // namespace fa2
