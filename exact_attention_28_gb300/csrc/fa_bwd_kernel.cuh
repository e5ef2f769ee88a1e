// Attention backward for sm_103a: recomputation of P from the forward's LSE
// and five gradient GEMMs on the tensor cores (tcgen05, accumulators in TMEM).
//
// Gradients, per (batch, head) ("6. FlashAttention 分块逻辑" section 7.1,
// "9.4 FlashAttention 与 FlashMLA" sections 9.4.3 and 9.4.5):
//   P  = exp(scale * Q K^T - LSE)           (recomputed, never stored in HBM)
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  D = rowsum(dO * O)
//   dQ = scale * dS K,  dK = scale * dS^T Q
// The dQ and the dK/dV accumulations run in different directions, so, as
// section 9.4.5 lays out, there are two kernels after a preprocessing pass:
//   fa_bwd_dot_kernel   D_i = sum_c dO_ic O_ic (one warp per row)
//   fa_bwd_dkdv_kernel  one CTA per 128-key tile, looping over query tiles
//                       (KV-outer): S^T = K Q^T, dP^T = V dO^T in TMEM, then
//                       P^T and dS^T (thread = key) back into TMEM as bf16,
//                       dV += P^T dO, dK += dS^T Q
//   fa_bwd_dq_kernel    one CTA per 128-query tile, looping over key tiles
//                       (Q-outer): S = Q K^T, dP = dO V^T, dS, dQ += dS K
// Each CTA has 6 warps: thread t < 128 owns TMEM lane t (a key in the first
// kernel, a query in the second) and does the elementwise work; thread 128
// issues the MMAs, so that the elementwise phases of one step overlap the
// GEMMs of the neighbouring ones; thread 160 issues the TMA loads, refilling
// each tile of a double-buffered stage as soon as its last GEMM has read it.
// Every wait is bounded like the forward's.
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {

constexpr int kBwdThreads = 192;   // warps 0-3: elementwise (thread = TMEM lane), warp 4: MMAs, warp 5: loads

struct BwdParams {
    CUtensorMap tmQ, tmK, tmV, tmdO;   // [BH][N][D] bf16, box {64, 128, 1}, 128-byte swizzle
    const float *LSE;                  // [BH][Nq] from the forward (natural log)
    const float *Dsum;                 // [BH][Nq] rowsum(dO * O)
    __nv_bfloat16 *dQ, *dK, *dV;       // outputs
    int BH, Nq, Nk, Tr, Tc, causal;
    float c2;                          // scale * log2(e)
    float scale;
};

// Streamed tiles: A (Q in dK/dV, K in dQ) has three slots, B (dO, V) two.
// A is read last by the step's final GEMM, so with two slots its refill
// could start only about one step before it is needed again.
constexpr int kSlotsA = 3, kSlotsB = 2;

template <int D>
struct BwdConfig {
    static constexpr int kTile = 128 * D * 2;            // one [128][D] bf16 tile
    // dK/dV kernel: K_j, V_j resident; Q_i in 3 slots, dO_i in 2
    // dQ kernel:    Q_i, dO_i resident; K_j in 3 slots, V_j in 2
    static constexpr int kTileBytes = (2 + kSlotsA + kSlotsB) * kTile;
    static constexpr int kStatOffset = kTileBytes;       // 2 stages x (lse2[128], d[128]) fp32
    static constexpr int kBarOffset = kStatOffset + 2 * 2 * 128 * 4;
    static constexpr int kBarBytes = 160;
    static constexpr int kUsed = kBarOffset + kBarBytes;
    // room to align the dynamic shared memory to 1024 bytes (the kernel checks
    // the base it gets against this slack)
    static constexpr int kSmemBytes = kUsed + 1024 <= 232448 ? kUsed + 1024 : 232448;
    static constexpr int kSlack = kSmemBytes - kUsed;
    static_assert(kSlack >= 512, "shared memory");
    static constexpr uint32_t kTmemCols = 512;
};

// ------------------------------------------------------------ preprocessing

// D = rowsum(dO * O) in fp32, one warp per row.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_dot_kernel(const __nv_bfloat16 *__restrict__ O,
                                                         const __nv_bfloat16 *__restrict__ dO,
                                                         float *__restrict__ Dsum, long long rows) {
    const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    float acc = 0.f;
    #pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        const long long idx = row * D + lane + 32 * c;
        acc = fmaf(__bfloat162float(O[idx]), __bfloat162float(dO[idx]), acc);
    }
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) Dsum[row] = acc;
}

// ------------------------------------------------------------------ shared

// Barriers of both kernels (one arrival unless noted).
// Streamed tiles A and B: Q and dO in the dK/dV kernel, K and V in the dQ
// kernel; step n uses A slot n % 3 and B slot n % 2.
struct BwdShared {
    uint32_t loadA0, loadB0;   // + 8 * slot: the tile landed
    uint32_t freeA0, freeB0;   // + 8 * slot: the last GEMM reading the tile completed
    uint32_t first;     // the resident pair of tiles landed
    uint32_t sfull;     // the score GEMM of the current step completed
    uint32_t dpfull;    // the dP GEMM of the current step completed
    uint32_t pready;    // (128) phase A done: P stored (dK/dV) or S read into registers (dQ)
    uint32_t dsready;   // (128) phase B done: dS stored
    uint32_t done;
    volatile int *abort_flag;
};

// One tile (D/64 boxes) into `dst`, completing on `bar`.
__device__ __forceinline__ void bwd_load_tile(const CUtensorMap *map, uint32_t dst, uint32_t bar, int row, int bh,
                                              int chunks, int tile_bytes) {
    ptx::mbar_arrive_expect_tx(bar, tile_bytes);
    const uint64_t pol = ptx::l2_policy_evict_last();
    for (int c = 0; c < chunks; ++c) ptx::tma_load_3d(dst + c * kChunkBytes, map, bar, c * 64, row, bh, pol);
}

__device__ __forceinline__ void bwd_load_pair(const CUtensorMap *a, const CUtensorMap *b, uint32_t dst_a,
                                              uint32_t dst_b, uint32_t bar, int row, int bh, int chunks,
                                              int tile_bytes) {
    ptx::mbar_arrive_expect_tx(bar, 2 * tile_bytes);
    const uint64_t pol = ptx::l2_policy_evict_last();
    for (int c = 0; c < chunks; ++c) {
        ptx::tma_load_3d(dst_a + c * kChunkBytes, a, bar, c * 64, row, bh, pol);
        ptx::tma_load_3d(dst_b + c * kChunkBytes, b, bar, c * 64, row, bh, pol);
    }
}

// This thread's TMEM stores are complete and ordered before its arrival on
// `bar`, which the MMA warp waits for before reading them.
__device__ __forceinline__ void tmem_stores_then_arrive(uint32_t bar) {
    ptx::tmem_wait_store();
    ptx::tc_fence_before_sync();
    ptx::mbar_arrive(bar);
}

// Writes this thread's TMEM row (row `row` of the [n_rows][D] matrix at
// `rows`) of D fp32 columns, times `mul`, as bf16; rows >= n_rows are not
// written.  The lanes of a warp hold consecutive rows, and each group of 8
// lanes exchanges 16-byte pieces so that every store writes whole 128-byte
// lines (64 columns of one row per group).
template <int D>
__device__ __forceinline__ void store_row_bf16(uint32_t taddr, float mul, __nv_bfloat16 *rows, int row, int n_rows) {
    const uint32_t j8 = threadIdx.x & 7u;
    #pragma unroll 1
    for (int c = 0; c < D / 64; ++c) {
        uint32_t x[32];
        #pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            uint32_t o[32];
            ptx::tmem_load_32cols(taddr + c * 64 + hh * 32, o);
            #pragma unroll
            for (int i = 0; i < 16; ++i)
                x[16 * hh + i] = ptx::pack_bf16x2(__uint_as_float(o[2 * i]) * mul, __uint_as_float(o[2 * i + 1]) * mul);
        }
        transpose_8x8_pieces(x);
        #pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int r = row - static_cast<int>(j8) + e;
            if (r < n_rows)
                *reinterpret_cast<uint4 *>(rows + static_cast<size_t>(r) * D + 64 * c + 8 * j8) =
                    make_uint4(x[4 * e], x[4 * e + 1], x[4 * e + 2], x[4 * e + 3]);
        }
    }
}

// Phase A of one TMEM row of 128 score columns: P = 2^(c*s - lse2) for the
// visible columns col_lo <= c < col_hi, 0 elsewhere (column c's lse2 is
// col_lse2[c] when kPerColumn -- the dK/dV kernel, one query per column --
// else the row's own).  P stays in registers (fp32) for phase B; with
// kStoreP it is also written as bf16 pairs over the score region's first 64
// columns (the A operand of dV += P^T dO).
template <bool kPerColumn, bool kStoreP>
__device__ __forceinline__ void bwd_phase_a(const uint32_t (&sv)[128], float (&pv)[128], uint32_t tS, float c2,
                                            const float *col_lse2, float row_lse2, int col_lo, int col_hi) {
    // the statistics as float4 reads of shared memory (one per 4 columns)
    const bool full = __all_sync(0xffffffffu, col_lo <= 0 && col_hi >= 128);   // warp-uniform
    #pragma unroll
    for (int c = 0; c < 128; c += 4) {
        float4 l4 = make_float4(row_lse2, row_lse2, row_lse2, row_lse2);
        if constexpr (kPerColumn) l4 = *reinterpret_cast<const float4 *>(col_lse2 + c);
        const float l[4] = {l4.x, l4.y, l4.z, l4.w};
        #pragma unroll
        for (int e = 0; e < 4; ++e) pv[c + e] = ptx::ex2(fmaf(__uint_as_float(sv[c + e]), c2, -l[e]));
    }
    if (!full) {
        #pragma unroll
        for (int c = 0; c < 128; ++c) pv[c] = (c >= col_lo && c < col_hi) ? pv[c] : 0.f;
    }
    if constexpr (kStoreP) {
        #pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t pk[16];
            #pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = ptx::pack_bf16x2(pv[32 * q + 2 * i], pv[32 * q + 2 * i + 1]);
            ptx::tmem_store_16cols(tS + 16 * q, pk);
        }
    }
}

// Phase B: dS = P * (dP - D) over the 128 columns, in quarters of 32 (each
// quarter's dS goes to columns 16q.., already read), as bf16 pairs over the
// dP region's first 64 columns (the A operand of the dK or dQ GEMM).
template <bool kPerColumn>
__device__ __forceinline__ void bwd_phase_b(const float (&pv)[128], uint32_t tdP, const float *col_d, float row_d) {
    #pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t dp[32];
        ptx::tmem_load_32cols(tdP + 32 * q, dp);
        uint32_t dk[16];
        #pragma unroll
        for (int i = 0; i < 16; i += 2) {
            const int c = 32 * q + 2 * i;
            float4 d4 = make_float4(row_d, row_d, row_d, row_d);
            if constexpr (kPerColumn) d4 = *reinterpret_cast<const float4 *>(col_d + c);
            dk[i] = ptx::pack_bf16x2(pv[c] * (__uint_as_float(dp[2 * i]) - d4.x),
                                     pv[c + 1] * (__uint_as_float(dp[2 * i + 1]) - d4.y));
            dk[i + 1] = ptx::pack_bf16x2(pv[c + 2] * (__uint_as_float(dp[2 * i + 2]) - d4.z),
                                         pv[c + 3] * (__uint_as_float(dp[2 * i + 3]) - d4.w));
        }
        ptx::tmem_store_16cols(tdP + 16 * q, dk);
    }
}

// Set-up of both kernels: smem carve-up, barriers, TMEM allocation by warp 4.
// Returns false (on every thread, before anything else) when the dynamic
// shared memory base leaves less than the configured slack for 1024-byte
// alignment; the status word then gets bit 2 and the CTA does nothing.
template <int D>
__device__ __forceinline__ bool bwd_setup(uint8_t *smem_raw, uint32_t &base, uint8_t *&base_ptr, BwdShared &sh,
                                          uint32_t &tmem) {
    using C = BwdConfig<D>;
    const uint32_t raw = ptx::smem_addr(smem_raw);
    base = (raw + 1023u) & ~1023u;
    if (base - raw > static_cast<uint32_t>(C::kSlack)) {
        if (threadIdx.x == 0) atomicOr(&g_fa_status, 4u);
        return false;
    }
    base_ptr = smem_raw + (base - raw);
    const uint32_t bars = base + C::kBarOffset;
    sh.loadA0 = bars + 0;     // kSlotsA
    sh.loadB0 = bars + 24;    // kSlotsB
    sh.freeA0 = bars + 40;    // kSlotsA
    sh.freeB0 = bars + 64;    // kSlotsB
    sh.first = bars + 80;
    sh.sfull = bars + 88;
    sh.dpfull = bars + 96;
    sh.pready = bars + 104;
    sh.dsready = bars + 112;
    sh.done = bars + 120;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(base_ptr + C::kBarOffset + 128);
    sh.abort_flag = reinterpret_cast<volatile int *>(base_ptr + C::kBarOffset + 132);
    static_assert(136 <= C::kBarBytes, "barrier block");
    if (threadIdx.x == 0) {
        for (int i = 0; i < kSlotsA; ++i) {
            ptx::mbar_init(sh.loadA0 + 8 * i, 1);
            ptx::mbar_init(sh.freeA0 + 8 * i, 1);
        }
        for (int i = 0; i < kSlotsB; ++i) {
            ptx::mbar_init(sh.loadB0 + 8 * i, 1);
            ptx::mbar_init(sh.freeB0 + 8 * i, 1);
        }
        ptx::mbar_init(sh.first, 1);
        ptx::mbar_init(sh.sfull, 1);
        ptx::mbar_init(sh.dpfull, 1);
        ptx::mbar_init(sh.pready, 128);
        ptx::mbar_init(sh.dsready, 128);
        ptx::mbar_init(sh.done, 1);
        *sh.abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if ((threadIdx.x >> 5) == 4) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_holder), C::kTmemCols);
        ptx::tmem_relinquish_alloc_permit();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    tmem = *tmem_holder;
    return true;
}

// Loads the producer thread has issued, for the drain at the end.
struct BwdLoads {
    int a[kSlotsA] = {0, 0, 0}, b[kSlotsB] = {0, 0};
    bool first = false;
};

// Teardown: the MMA thread (128) waits for all its MMAs, the load thread
// (160) for the copies it issued; then warp 4 frees TMEM.
template <int D>
__device__ __forceinline__ void bwd_teardown(uint32_t tmem, const BwdShared &sh, const BwdLoads &ld) {
    if (threadIdx.x == 128) {
        ptx::mma_commit(sh.done);
        wait_drain(sh.done, 0);
    }
    if (threadIdx.x == 160) {
        for (int s = 0; s < kSlotsA; ++s)
            if (ld.a[s] > 0) wait_drain(sh.loadA0 + 8 * s, (ld.a[s] - 1) & 1);
        for (int s = 0; s < kSlotsB; ++s)
            if (ld.b[s] > 0) wait_drain(sh.loadB0 + 8 * s, (ld.b[s] - 1) & 1);
        if (ld.first) wait_drain(sh.first, 0);
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    if ((threadIdx.x >> 5) == 4) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, BwdConfig<D>::kTmemCols);
    }
}

// ------------------------------------------------------------ dK, dV kernel
//
// TMEM: S^T [0,128) (P^T as bf16 pairs in [0,64)), dP^T [128,256) (dS^T in
// [128,192)), dV [256, 256+D), dK [256+D, 256+2D).  Lane = key.
// Warps 0-3: thread t = key j*128 + t, elementwise.  Warp 4 (converged,
// lane 0 issues) runs the MMAs, warp 5's lane 0 the loads; per query tile n:
//   wait P^T(n) -> dV += P^T dO_n;  S^T(n+1) = K Q_{n+1}^T     (S^T free once P^T is read)
//   wait dS^T(n) -> dK += dS^T Q_n; dP^T(n+1) = V dO_{n+1}^T
// so phase A of step n+1 runs while dK(n) and dP^T(n+1) execute, and phase
// B of step n while dV(n) and S^T(n+1) do.

// Loads of the dK/dV kernel: K_j, V_j once; Q_i (tile A, slot n % 3) and
// dO_i (tile B, slot n % 2) of query tile i_begin + n, each refilled as soon
// as the GEMMs reading it are done (dO after dV, Q after dK).
template <int D>
__device__ void dkdv_load_role(const BwdParams &p, const BwdShared &sh, uint32_t base, int j, int bh, int i_begin,
                               int n_i, BwdLoads &ld) {
    using C = BwdConfig<D>;
    const uint32_t sK = base, sV = base + C::kTile;
    const uint32_t sQ0 = base + 2 * C::kTile, sdO0 = base + (2 + kSlotsA) * C::kTile;
    constexpr int kChunks = D / 64;
    ptx::mbar_arrive_expect_tx(sh.first, 2 * C::kTile);
    ld.first = true;
    {
        const uint64_t pol = ptx::l2_policy_evict_first();
        for (int c = 0; c < kChunks; ++c) {
            ptx::tma_load_3d(sK + c * kChunkBytes, &p.tmK, sh.first, c * 64, j * kBC, bh, pol);
            ptx::tma_load_3d(sV + c * kChunkBytes, &p.tmV, sh.first, c * 64, j * kBC, bh, pol);
        }
    }
    for (int n = 0; n < kSlotsA && n < n_i; ++n) {
        bwd_load_tile(&p.tmQ, sQ0 + n * C::kTile, sh.loadA0 + 8 * n, (i_begin + n) * kBR, bh, kChunks, C::kTile);
        ++ld.a[n];
    }
    for (int n = 0; n < kSlotsB && n < n_i; ++n) {
        bwd_load_tile(&p.tmdO, sdO0 + n * C::kTile, sh.loadB0 + 8 * n, (i_begin + n) * kBR, bh, kChunks, C::kTile);
        ++ld.b[n];
    }
    for (int n = 0; n + kSlotsB < n_i; ++n) {
        const int a = n % kSlotsA, b = n % kSlotsB;
        if (!wait_bar(sh.freeB0 + 8 * b, (n / kSlotsB) & 1, sh.abort_flag, 18, blockIdx.x, n)) return;
        bwd_load_tile(&p.tmdO, sdO0 + b * C::kTile, sh.loadB0 + 8 * b, (i_begin + n + kSlotsB) * kBR, bh, kChunks,
                      C::kTile);
        ++ld.b[b];
        if (n + kSlotsA < n_i) {
            if (!wait_bar(sh.freeA0 + 8 * a, (n / kSlotsA) & 1, sh.abort_flag, 18, blockIdx.x, n)) return;
            bwd_load_tile(&p.tmQ, sQ0 + a * C::kTile, sh.loadA0 + 8 * a, (i_begin + n + kSlotsA) * kBR, bh, kChunks,
                          C::kTile);
            ++ld.a[a];
        }
    }
}

template <int D>
__device__ void dkdv_mma_role(const BwdParams &p, const BwdShared &sh, uint32_t tmem, uint32_t base, int n_i) {
    using C = BwdConfig<D>;
    const uint32_t sK = base, sV = base + C::kTile;
    const uint32_t sQ0 = base + 2 * C::kTile, sdO0 = base + (2 + kSlotsA) * C::kTile;
    const uint32_t tST = tmem + 0, tdPT = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;
    if (!wait_bar_warp(sh.first, 0, sh.abort_flag, 10, blockIdx.x, -1)) return;
    if (!wait_bar_warp(sh.loadA0, 0, sh.abort_flag, 10, blockIdx.x, 0)) return;
    ptx::tc_fence_after_sync();
    issue_s<D, kBC>(tST, sK, sQ0);        // S^T(0) = K Q_0^T
    ptx::mma_commit(sh.sfull);
    if (!wait_bar_warp(sh.loadB0, 0, sh.abort_flag, 10, blockIdx.x, 0)) return;
    ptx::tc_fence_after_sync();
    issue_s<D, kBC>(tdPT, sV, sdO0);      // dP^T(0) = V dO_0^T
    ptx::mma_commit(sh.dpfull);
    for (int n = 0; n < n_i; ++n) {
        const int a = n % kSlotsA, b = n % kSlotsB;
        const int an = (n + 1) % kSlotsA, bn = (n + 1) % kSlotsB;
        if (!wait_bar_warp(sh.pready, n & 1, sh.abort_flag, 11, blockIdx.x, n)) return;
        ptx::tc_fence_after_sync();
        issue_pv<D, kBC>(tdV, tST, sdO0 + b * C::kTile, n > 0);    // dV += P^T dO_n
        ptx::mma_commit(sh.freeB0 + 8 * b);                   // dO_n read for the last time
        if (n + 1 < n_i) {
            if (!wait_bar_warp(sh.loadA0 + 8 * an, ((n + 1) / kSlotsA) & 1, sh.abort_flag, 12, blockIdx.x, n + 1)) return;
            ptx::tc_fence_after_sync();
            issue_s<D, kBC>(tST, sK, sQ0 + an * C::kTile);         // S^T(n+1)
            ptx::mma_commit(sh.sfull);
        }
        if (!wait_bar_warp(sh.dsready, n & 1, sh.abort_flag, 13, blockIdx.x, n)) return;
        ptx::tc_fence_after_sync();
        issue_pv<D, kBC>(tdK, tdPT, sQ0 + a * C::kTile, n > 0);    // dK += dS^T Q_n
        ptx::mma_commit(sh.freeA0 + 8 * a);                   // Q_n read for the last time
        if (n + 1 < n_i) {
            if (!wait_bar_warp(sh.loadB0 + 8 * bn, ((n + 1) / kSlotsB) & 1, sh.abort_flag, 14, blockIdx.x, n + 1)) return;
            ptx::tc_fence_after_sync();
            issue_s<D, kBC>(tdPT, sV, sdO0 + bn * C::kTile);       // dP^T(n+1)
            ptx::mma_commit(sh.dpfull);
        }
    }
}

template <int D>
__device__ void dkdv_elementwise_role(const BwdParams &p, const BwdShared &sh, uint32_t tmem, float *stat, int j,
                                      int bh, int i_begin, int n_i) {
    const int t = threadIdx.x;
    const uint32_t lane_off = static_cast<uint32_t>((t >> 5) * 32) << 16;
    const uint32_t tST = tmem + lane_off, tdPT = tmem + lane_off + 128;
    const uint32_t tdV = tmem + lane_off + 256, tdK = tmem + lane_off + 256 + D;
    const int key = j * kBC + t;
    const size_t out_row = (static_cast<size_t>(bh) * p.Nk + key) * D;
    if (n_i <= 0) {   // no query sees this key
        if (key < p.Nk)
            for (int c = 0; c < D; ++c) p.dV[out_row + c] = p.dK[out_row + c] = __float2bfloat16_rn(0.f);
        return;
    }
    bool ok = true;
    for (int n = 0; n < n_i; ++n) {
        const int i = i_begin + n;
        const int s = n & 1;
        {   // per-query statistics of this tile, in log2 units; padding rows masked
            const int q = i * kBR + t;
            const bool live = q < p.Nq;
            stat[(s * 2 + 0) * 128 + t] = live ? p.LSE[static_cast<size_t>(bh) * p.Nq + q] * 1.4426950408889634f
                                               : INFINITY;
            stat[(s * 2 + 1) * 128 + t] = live ? p.Dsum[static_cast<size_t>(bh) * p.Nq + q] : 0.f;
        }
        // publishes the statistics; every thread leaves the loop together
        if (!ptx::named_barrier_and(1, 128, ok)) { ok = false; break; }
        if (!wait_bar(sh.sfull, n & 1, sh.abort_flag, 15, blockIdx.x, n)) { ok = false; continue; }
        ptx::tc_fence_after_sync();
        // visible query columns for this key: all, or those at or after the key
        // on the diagonal tile; a key past Nk has none
        const int col_lo = key >= p.Nk ? kBR : (p.causal && i == j ? t : 0);
        float pv[128];
        {
            uint32_t sv[128];
            ptx::tmem_load_128cols(tST, sv);
            bwd_phase_a<true, true>(sv, pv, tST, p.c2, stat + (s * 2 + 0) * 128, 0.f, col_lo, kBR);
        }
        tmem_stores_then_arrive(sh.pready);
        if (!wait_bar(sh.dpfull, n & 1, sh.abort_flag, 16, blockIdx.x, n)) { ok = false; continue; }
        ptx::tc_fence_after_sync();
        bwd_phase_b<true>(pv, tdPT, stat + (s * 2 + 1) * 128, 0.f);
        tmem_stores_then_arrive(sh.dsready);
    }
    if (!ptx::named_barrier_and(1, 128, ok)) return;
    // the last accumulation done: dV and scale * dK for this key
    const int a_last = (n_i - 1) % kSlotsA;
    if (!wait_bar(sh.freeA0 + 8 * a_last, ((n_i - 1) / kSlotsA) & 1, sh.abort_flag, 17, blockIdx.x, n_i)) return;
    ptx::tc_fence_after_sync();
    const size_t head = static_cast<size_t>(bh) * p.Nk * D;
    store_row_bf16<D>(tdV, 1.f, p.dV + head, key, p.Nk);
    store_row_bf16<D>(tdK, p.scale, p.dK + head, key, p.Nk);
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) fa_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
    using C = BwdConfig<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint32_t base;
    uint8_t *base_ptr;
    BwdShared sh;
    uint32_t tmem;
    if (!bwd_setup<D>(smem_raw, base, base_ptr, sh, tmem)) return;
    // heavy tiles (small j under the causal mask) get the low block indices
    const int j = blockIdx.x / p.BH;
    const int bh = blockIdx.x % p.BH;
    const int i_begin = p.causal ? j : 0;      // query tiles that can see key tile j
    const int n_i = p.Tr - i_begin;
    BwdLoads ld;
    if (threadIdx.x < 128) {
        dkdv_elementwise_role<D>(p, sh, tmem, reinterpret_cast<float *>(base_ptr + C::kStatOffset), j, bh, i_begin,
                                 n_i);
    } else if ((threadIdx.x >> 5) == 4 && n_i > 0) {   // the whole warp, converged; lane 0 issues
        dkdv_mma_role<D>(p, sh, tmem, base, n_i);
    } else if (threadIdx.x == 160 && n_i > 0) {
        dkdv_load_role<D>(p, sh, base, j, bh, i_begin, n_i, ld);
    }
    __syncwarp();
    bwd_teardown<D>(tmem, sh, ld);
}

// --------------------------------------------------------------- dQ kernel
//
// TMEM: S [0,128), dP [128,256) (dS as bf16 pairs in [128,192)), dQ [256, 256+D).
// Lane = query.  Warp 4 (converged, lane 0 issues), per key tile n:
//   wait S(n) read -> S(n+1) = Q K_{n+1}^T   (S(n) is in the threads' registers)
//   wait dS(n)     -> dQ += dS K_n;  dP(n+1) = dO V_{n+1}^T

// Loads of the dQ kernel: Q_i, dO_i once; K_j (tile A, slot n % 3) and V_j
// (tile B, slot n % 2) of key tile n, each refilled once its GEMMs are done
// (V after dP, K after dQ).
template <int D>
__device__ void dq_load_role(const BwdParams &p, const BwdShared &sh, uint32_t base, int i, int bh, int n_j,
                             BwdLoads &ld) {
    using C = BwdConfig<D>;
    const uint32_t sQ = base, sdO = base + C::kTile;
    const uint32_t sK0 = base + 2 * C::kTile, sV0 = base + (2 + kSlotsA) * C::kTile;
    constexpr int kChunks = D / 64;
    bwd_load_pair(&p.tmQ, &p.tmdO, sQ, sdO, sh.first, i * kBR, bh, kChunks, C::kTile);
    ld.first = true;
    for (int n = 0; n < kSlotsA && n < n_j; ++n) {
        bwd_load_tile(&p.tmK, sK0 + n * C::kTile, sh.loadA0 + 8 * n, n * kBC, bh, kChunks, C::kTile);
        ++ld.a[n];
    }
    for (int n = 0; n < kSlotsB && n < n_j; ++n) {
        bwd_load_tile(&p.tmV, sV0 + n * C::kTile, sh.loadB0 + 8 * n, n * kBC, bh, kChunks, C::kTile);
        ++ld.b[n];
    }
    for (int n = 0; n + kSlotsB < n_j; ++n) {
        const int a = n % kSlotsA, b = n % kSlotsB;
        if (!wait_bar(sh.freeB0 + 8 * b, (n / kSlotsB) & 1, sh.abort_flag, 28, blockIdx.x, n)) return;
        bwd_load_tile(&p.tmV, sV0 + b * C::kTile, sh.loadB0 + 8 * b, (n + kSlotsB) * kBC, bh, kChunks, C::kTile);
        ++ld.b[b];
        if (n + kSlotsA < n_j) {
            if (!wait_bar(sh.freeA0 + 8 * a, (n / kSlotsA) & 1, sh.abort_flag, 28, blockIdx.x, n)) return;
            bwd_load_tile(&p.tmK, sK0 + a * C::kTile, sh.loadA0 + 8 * a, (n + kSlotsA) * kBC, bh, kChunks, C::kTile);
            ++ld.a[a];
        }
    }
}

template <int D>
__device__ void dq_mma_role(const BwdParams &p, const BwdShared &sh, uint32_t tmem, uint32_t base, int n_j) {
    using C = BwdConfig<D>;
    const uint32_t sQ = base, sdO = base + C::kTile;
    const uint32_t sK0 = base + 2 * C::kTile, sV0 = base + (2 + kSlotsA) * C::kTile;
    const uint32_t tS = tmem + 0, tdP = tmem + 128, tdQ = tmem + 256;
    if (!wait_bar_warp(sh.first, 0, sh.abort_flag, 20, blockIdx.x, -1)) return;
    if (!wait_bar_warp(sh.loadA0, 0, sh.abort_flag, 20, blockIdx.x, 0)) return;
    ptx::tc_fence_after_sync();
    issue_s<D, kBC>(tS, sQ, sK0);        // S(0) = Q K_0^T
    ptx::mma_commit(sh.sfull);
    if (!wait_bar_warp(sh.loadB0, 0, sh.abort_flag, 20, blockIdx.x, 0)) return;
    ptx::tc_fence_after_sync();
    issue_s<D, kBC>(tdP, sdO, sV0);      // dP(0) = dO V_0^T
    ptx::mma_commit(sh.dpfull);
    ptx::mma_commit(sh.freeB0);     // V_0 read for the last time
    for (int n = 0; n < n_j; ++n) {
        const int a = n % kSlotsA;
        const int an = (n + 1) % kSlotsA, bn = (n + 1) % kSlotsB;
        if (!wait_bar_warp(sh.pready, n & 1, sh.abort_flag, 21, blockIdx.x, n)) return;
        if (n + 1 < n_j) {
            if (!wait_bar_warp(sh.loadA0 + 8 * an, ((n + 1) / kSlotsA) & 1, sh.abort_flag, 22, blockIdx.x, n + 1)) return;
            ptx::tc_fence_after_sync();
            issue_s<D, kBC>(tS, sQ, sK0 + an * C::kTile);          // S(n+1)
            ptx::mma_commit(sh.sfull);
        }
        if (!wait_bar_warp(sh.dsready, n & 1, sh.abort_flag, 23, blockIdx.x, n)) return;
        ptx::tc_fence_after_sync();
        issue_pv<D, kBC>(tdQ, tdP, sK0 + a * C::kTile, n > 0);     // dQ += dS K_n
        ptx::mma_commit(sh.freeA0 + 8 * a);                   // K_n read for the last time
        if (n + 1 < n_j) {
            if (!wait_bar_warp(sh.loadB0 + 8 * bn, ((n + 1) / kSlotsB) & 1, sh.abort_flag, 24, blockIdx.x, n + 1)) return;
            ptx::tc_fence_after_sync();
            issue_s<D, kBC>(tdP, sdO, sV0 + bn * C::kTile);        // dP(n+1)
            ptx::mma_commit(sh.dpfull);
            ptx::mma_commit(sh.freeB0 + 8 * bn);              // V_{n+1} read for the last time
        }
    }
}

template <int D>
__device__ void dq_elementwise_role(const BwdParams &p, const BwdShared &sh, uint32_t tmem, int i, int bh, int n_j) {
    const int t = threadIdx.x;
    const uint32_t lane_off = static_cast<uint32_t>((t >> 5) * 32) << 16;
    const uint32_t tS = tmem + lane_off, tdP = tmem + lane_off + 128, tdQ = tmem + lane_off + 256;
    const int q = i * kBR + t;
    const bool qlive = q < p.Nq;
    const float row_lse2 = qlive ? p.LSE[static_cast<size_t>(bh) * p.Nq + q] * 1.4426950408889634f : INFINITY;
    const float row_d = qlive ? p.Dsum[static_cast<size_t>(bh) * p.Nq + q] : 0.f;
    for (int n = 0; n < n_j; ++n) {
        if (!wait_bar(sh.sfull, n & 1, sh.abort_flag, 25, blockIdx.x, n)) return;
        ptx::tc_fence_after_sync();
        // visible key columns: below Nk, and at or before the query on the diagonal
        int col_hi = min(kBC, p.Nk - n * kBC);
        if (p.causal && n == i) col_hi = min(col_hi, t + 1);
        if (!qlive) col_hi = 0;
        float pv[128];
        {
            uint32_t sv[128];
            ptx::tmem_load_128cols(tS, sv);
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(sh.pready);   // S(n) is in registers: its columns may be overwritten
            bwd_phase_a<false, false>(sv, pv, tS, p.c2, nullptr, row_lse2, 0, col_hi);
        }
        if (!wait_bar(sh.dpfull, n & 1, sh.abort_flag, 26, blockIdx.x, n)) return;
        ptx::tc_fence_after_sync();
        bwd_phase_b<false>(pv, tdP, nullptr, row_d);
        tmem_stores_then_arrive(sh.dsready);
    }
    const int a_last = (n_j - 1) % kSlotsA;
    if (!wait_bar(sh.freeA0 + 8 * a_last, ((n_j - 1) / kSlotsA) & 1, sh.abort_flag, 27, blockIdx.x, n_j)) return;
    ptx::tc_fence_after_sync();
    store_row_bf16<D>(tdQ, p.scale, p.dQ + static_cast<size_t>(bh) * p.Nq * D, q, p.Nq);
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) fa_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint32_t base;
    uint8_t *base_ptr;
    BwdShared sh;
    uint32_t tmem;
    if (!bwd_setup<D>(smem_raw, base, base_ptr, sh, tmem)) return;
    // heavy tiles (large i under the causal mask) get the low block indices
    const int i = p.causal ? (p.Tr - 1 - blockIdx.x / p.BH) : blockIdx.x / p.BH;
    const int bh = blockIdx.x % p.BH;
    int n_j = p.Tc;
    if (p.causal) {
        const int q_end = min(p.Nq, (i + 1) * kBR);
        n_j = min(p.Tc, (q_end - 1) / kBC + 1);
    }
    BwdLoads ld;
    if (threadIdx.x < 128) dq_elementwise_role<D>(p, sh, tmem, i, bh, n_j);
    else if ((threadIdx.x >> 5) == 4) dq_mma_role<D>(p, sh, tmem, base, n_j);   // whole warp; lane 0 issues
    else if (threadIdx.x == 160) dq_load_role<D>(p, sh, base, i, bh, n_j, ld);
    __syncwarp();
    bwd_teardown<D>(tmem, sh, ld);
}

}  // namespace fa
