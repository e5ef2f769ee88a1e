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
// Each CTA is one warpgroup: thread t owns TMEM lane t (a key in the first
// kernel, a query in the second); thread 0 issues the TMA loads and MMAs.
// Loads are double-buffered; every wait is bounded like the forward's.
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {

constexpr int kBwdThreads = 128;

struct BwdParams {
    CUtensorMap tmQ, tmK, tmV, tmdO;   // [BH][N][D] bf16, box {64, 128, 1}, 128-byte swizzle
    const float *LSE;                  // [BH][Nq] from the forward (natural log)
    const float *Dsum;                 // [BH][Nq] rowsum(dO * O)
    __nv_bfloat16 *dQ, *dK, *dV;       // outputs
    int BH, Nq, Nk, Tr, Tc, causal;
    float c2;                          // scale * log2(e)
    float scale;
};

template <int D>
struct BwdConfig {
    static constexpr int kTile = 128 * D * 2;            // one [128][D] bf16 tile
    // dK/dV kernel: K_j, V_j resident; Q_i, dO_i double-buffered
    // dQ kernel:    Q_i, dO_i resident; K_j, V_j double-buffered
    static constexpr int kTileBytes = 6 * kTile;
    static constexpr int kStatOffset = kTileBytes;       // 2 stages x (lse2[128], d[128]) fp32
    static constexpr int kBarOffset = kStatOffset + 2 * 2 * 128 * 4;
    static constexpr int kSmemBytes = kBarOffset + 128 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory");
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

struct BwdShared {
    uint32_t load0;     // + 8 * stage: TMA tiles of a stage landed
    uint32_t first;     // the resident pair of tiles landed
    uint32_t mma_s;     // the two score-side GEMMs of an iteration completed
    uint32_t mma_acc0;  // + 8 * stage: the accumulating GEMMs that read a stage completed
    uint32_t done;
    volatile int *abort_flag;
};

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

// Thread-block barrier for the elementwise -> MMA hand-off: every thread's
// TMEM stores are complete and visible to the MMA issued next.
__device__ __forceinline__ void tmem_stores_to_mma() {
    ptx::tmem_wait_store();
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
}

// Writes one TMEM row of D fp32 columns, times `mul`, as bf16 to global.
template <int D>
__device__ __forceinline__ void store_row_bf16(uint32_t taddr, float mul, __nv_bfloat16 *dst, bool live) {
    #pragma unroll 1
    for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        ptx::tmem_load_32cols(taddr + ch * 32, o);
        uint32_t h[16];
        #pragma unroll
        for (int i = 0; i < 16; ++i)
            h[i] = ptx::pack_bf16x2(__uint_as_float(o[2 * i]) * mul, __uint_as_float(o[2 * i + 1]) * mul);
        if (live) {
            uint4 *p = reinterpret_cast<uint4 *>(dst + ch * 32);
            #pragma unroll
            for (int i = 0; i < 4; ++i) p[i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
        }
    }
}

// The elementwise step shared by both kernels, for one TMEM row of 128
// score columns: P = 2^(c*s - lse2), dS = P * (dP - D), with masked columns
// giving P = dS = 0.  Column q's lse2 and D come from `col_lse2`/`col_d`
// (the first kernel: per query column) or are the row's own (the second).
// P (if wanted) and dS are packed to bf16 pairs and written over the first 64
// columns of the score region and of the dP region respectively.
template <bool kWantP, bool kPerColumnStats>
__device__ __forceinline__ void bwd_elementwise(uint32_t tS, uint32_t tdP, float c2, const float *col_lse2,
                                                const float *col_d, float row_lse2, float row_d, int col_lo,
                                                int col_hi) {
    // columns c with col_lo <= c < col_hi are visible (others: P = 0)
    #pragma unroll 1
    for (int half = 0; half < 2; ++half) {
        uint32_t s[64], dp[64];
        ptx::tmem_load_32cols(tS + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        ptx::tmem_load_32cols(tS + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        ptx::tmem_load_32cols(tdP + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
        ptx::tmem_load_32cols(tdP + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
        uint32_t pk[32], dk[32];
        #pragma unroll
        for (int i = 0; i < 32; ++i) {
            float pv[2], dv[2];
            #pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int c = 64 * half + 2 * i + e;
                const float lse2 = kPerColumnStats ? col_lse2[c] : row_lse2;
                const float dd = kPerColumnStats ? col_d[c] : row_d;
                float p = ptx::ex2(fmaf(__uint_as_float(s[2 * i + e]), c2, -lse2));
                p = (c >= col_lo && c < col_hi) ? p : 0.f;
                pv[e] = p;
                dv[e] = p * (__uint_as_float(dp[2 * i + e]) - dd);
            }
            pk[i] = ptx::pack_bf16x2(pv[0], pv[1]);
            dk[i] = ptx::pack_bf16x2(dv[0], dv[1]);
        }
        if (kWantP) {
            ptx::tmem_store_16cols(tS + 32 * half, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
            ptx::tmem_store_16cols(tS + 32 * half + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]));
        }
        ptx::tmem_store_16cols(tdP + 32 * half, *reinterpret_cast<const uint32_t(*)[16]>(&dk[0]));
        ptx::tmem_store_16cols(tdP + 32 * half + 16, *reinterpret_cast<const uint32_t(*)[16]>(&dk[16]));
    }
}

// Shared set-up of both kernels: smem carve-up, barriers, TMEM allocation.
template <int D>
__device__ __forceinline__ uint32_t bwd_setup(uint8_t *smem_raw, uint32_t &base, uint8_t *&base_ptr, BwdShared &sh) {
    using C = BwdConfig<D>;
    const uint32_t raw = ptx::smem_addr(smem_raw);
    base = (raw + 1023u) & ~1023u;
    base_ptr = smem_raw + (base - raw);
    const uint32_t bars = base + C::kBarOffset;
    sh.load0 = bars + 0;      // 2
    sh.first = bars + 16;
    sh.mma_s = bars + 24;
    sh.mma_acc0 = bars + 32;  // 2
    sh.done = bars + 48;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(base_ptr + C::kBarOffset + 64);
    sh.abort_flag = reinterpret_cast<volatile int *>(base_ptr + C::kBarOffset + 68);
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(sh.load0 + 8 * i, 1);
            ptx::mbar_init(sh.mma_acc0 + 8 * i, 1);
        }
        ptx::mbar_init(sh.first, 1);
        ptx::mbar_init(sh.mma_s, 1);
        ptx::mbar_init(sh.done, 1);
        *sh.abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (threadIdx.x < 32) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_holder), C::kTmemCols);
        ptx::tmem_relinquish_alloc_permit();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    return *tmem_holder;
}

template <int D>
__device__ __forceinline__ void bwd_teardown(uint32_t tmem, const BwdShared &sh) {
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) {
            ptx::mma_commit(sh.done);
            wait_drain(sh.done, 0);
        }
        __syncwarp();
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, BwdConfig<D>::kTmemCols);
    }
}

// ------------------------------------------------------------ dK, dV kernel

// TMEM: S^T [0,128) (P^T as bf16 pairs in [0,64)), dP^T [128,256) (dS^T in
// [128,192)), dV [256, 256+D), dK [256+D, 256+2D).  Lane = key.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) fa_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
    using C = BwdConfig<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint32_t base;
    uint8_t *base_ptr;
    BwdShared sh;
    const uint32_t tmem = bwd_setup<D>(smem_raw, base, base_ptr, sh);
    const int t = threadIdx.x;
    const int warp = t >> 5;

    // heavy tiles (small j under the causal mask) get the low block indices
    const int j = blockIdx.x / p.BH;
    const int bh = blockIdx.x % p.BH;
    const int i_begin = p.causal ? j : 0;      // query tiles that can see key tile j
    const int n_i = p.Tr - i_begin;
    const uint32_t sK = base, sV = base + C::kTile;
    const uint32_t sQ[2] = {base + 2 * C::kTile, base + 3 * C::kTile};
    const uint32_t sdO[2] = {base + 4 * C::kTile, base + 5 * C::kTile};
    float *stat = reinterpret_cast<float *>(base_ptr + C::kStatOffset);   // [2][2][128]: lse2, D
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tST = tmem + 0, tdPT = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;
    constexpr int kChunks = D / 64;
    bool ok = true;

    if (t == 0 && n_i > 0) {
        ptx::mbar_arrive_expect_tx(sh.first, 2 * C::kTile);
        const uint64_t pol = ptx::l2_policy_evict_first();
        for (int c = 0; c < kChunks; ++c) {
            ptx::tma_load_3d(sK + c * kChunkBytes, &p.tmK, sh.first, c * 64, j * kBC, bh, pol);
            ptx::tma_load_3d(sV + c * kChunkBytes, &p.tmV, sh.first, c * 64, j * kBC, bh, pol);
        }
        for (int s = 0; s < 2 && s < n_i; ++s)
            bwd_load_pair(&p.tmQ, &p.tmdO, sQ[s], sdO[s], sh.load0 + 8 * s, (i_begin + s) * kBR, bh, kChunks,
                          C::kTile);
    }
    const int key = j * kBC + t;
    // every failure decision below is made block-wide (__syncthreads_and), so
    // all threads leave the loop together and meet at the same barriers
    for (int n = 0; n < n_i; ++n) {
        const int i = i_begin + n;
        const int s = n & 1;
        const uint32_t use = n >> 1;
        // per-query statistics of this tile, in log2 units, padding rows masked
        {
            const int q = i * kBR + t;
            const bool live = q < p.Nq;
            stat[(s * 2 + 0) * 128 + t] = live ? p.LSE[static_cast<size_t>(bh) * p.Nq + q] * 1.4426950408889634f
                                               : INFINITY;
            stat[(s * 2 + 1) * 128 + t] = live ? p.Dsum[static_cast<size_t>(bh) * p.Nq + q] : 0.f;
        }
        bool step_ok = true;
        if (t == 0) {
            if (n == 0) step_ok = wait_bar(sh.first, 0, sh.abort_flag, 10, blockIdx.x, -1);
            step_ok = step_ok && wait_bar(sh.load0 + 8 * s, use & 1, sh.abort_flag, 10, blockIdx.x, n);
            if (step_ok) {
                ptx::tc_fence_after_sync();
                issue_s<D>(tmem + tST, sK, sQ[s]);      // S^T = K_j Q_i^T
                issue_s<D>(tmem + tdPT, sV, sdO[s]);    // dP^T = V_j dO_i^T
                ptx::mma_commit(sh.mma_s);
            }
        }
        if (!__syncthreads_and(step_ok)) { ok = false; break; }   // also publishes the statistics
        if (!__syncthreads_and(wait_bar(sh.mma_s, n & 1, sh.abort_flag, 11, blockIdx.x, n))) { ok = false; break; }
        ptx::tc_fence_after_sync();
        // visible query columns for this key: all, or those at or after the key
        // on the diagonal tile; a key past Nk has none
        const int col_lo = key >= p.Nk ? kBR : (p.causal && i == j ? t : 0);
        bwd_elementwise<true, true>(tmem + lane_off + tST, tmem + lane_off + tdPT, p.c2, stat + (s * 2 + 0) * 128,
                                    stat + (s * 2 + 1) * 128, 0.f, 0.f, col_lo, kBR);
        tmem_stores_to_mma();
        step_ok = true;
        if (t == 0) {
            issue_pv<D>(tmem + tdV, tmem + tST, sdO[s], n > 0);   // dV += P^T dO_i
            issue_pv<D>(tmem + tdK, tmem + tdPT, sQ[s], n > 0);   // dK += dS^T Q_i
            ptx::mma_commit(sh.mma_acc0 + 8 * s);
            if (n + 2 < n_i) {   // refill this stage once its readers are done
                step_ok = wait_bar(sh.mma_acc0 + 8 * s, use & 1, sh.abort_flag, 12, blockIdx.x, n);
                if (step_ok)
                    bwd_load_pair(&p.tmQ, &p.tmdO, sQ[s], sdO[s], sh.load0 + 8 * s, (i + 2) * kBR, bh, kChunks,
                                  C::kTile);
            }
        }
        // the stage's statistics may be rewritten two iterations later
        if (!__syncthreads_and(step_ok)) { ok = false; break; }
    }
    // wait for the last accumulation, then write dV and scale * dK for this key
    if (n_i > 0 && ok) {
        const int s = (n_i - 1) & 1;
        const uint32_t use = (n_i - 1) >> 1;
        if (wait_bar(sh.mma_acc0 + 8 * s, use & 1, sh.abort_flag, 13, blockIdx.x, n_i)) {
            ptx::tc_fence_after_sync();
            const bool live = key < p.Nk;
            const size_t row = (static_cast<size_t>(bh) * p.Nk + key) * D;
            store_row_bf16<D>(tmem + lane_off + tdV, 1.f, p.dV + row, live);
            store_row_bf16<D>(tmem + lane_off + tdK, p.scale, p.dK + row, live);
        }
    } else if (n_i <= 0 && key < p.Nk) {   // no query sees this key
        const size_t row = (static_cast<size_t>(bh) * p.Nk + key) * D;
        for (int c = 0; c < D; ++c) p.dV[row + c] = p.dK[row + c] = __float2bfloat16_rn(0.f);
    }
    // drain outstanding loads before the CTA's shared memory is released
    if (t == 0)
        for (int s = 0; s < 2 && s < n_i; ++s) {
            const int last = (n_i - 1 - s) >= 0 ? ((n_i - 1 - s) / 2) * 2 + s : -1;
            if (last >= 0) wait_drain(sh.load0 + 8 * s, (last >> 1) & 1);
        }
    bwd_teardown<D>(tmem, sh);
}

// --------------------------------------------------------------- dQ kernel

// TMEM: S [0,128), dP [128,256) (dS as bf16 pairs in [128,192)), dQ [256, 256+D).
// Lane = query.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) fa_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
    using C = BwdConfig<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint32_t base;
    uint8_t *base_ptr;
    BwdShared sh;
    const uint32_t tmem = bwd_setup<D>(smem_raw, base, base_ptr, sh);
    const int t = threadIdx.x;
    const int warp = t >> 5;

    // heavy tiles (large i under the causal mask) get the low block indices
    const int i = p.causal ? (p.Tr - 1 - blockIdx.x / p.BH) : blockIdx.x / p.BH;
    const int bh = blockIdx.x % p.BH;
    int n_j = p.Tc;
    if (p.causal) {
        const int q_end = min(p.Nq, (i + 1) * kBR);
        n_j = min(p.Tc, (q_end - 1) / kBC + 1);
    }
    const uint32_t sQ = base, sdO = base + C::kTile;
    const uint32_t sK[2] = {base + 2 * C::kTile, base + 3 * C::kTile};
    const uint32_t sV[2] = {base + 4 * C::kTile, base + 5 * C::kTile};
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + 0, tdP = tmem + 128, tdQ = tmem + 256;
    constexpr int kChunks = D / 64;
    const int q = i * kBR + t;
    const bool qlive = q < p.Nq;
    const float row_lse2 = qlive ? p.LSE[static_cast<size_t>(bh) * p.Nq + q] * 1.4426950408889634f : INFINITY;
    const float row_d = qlive ? p.Dsum[static_cast<size_t>(bh) * p.Nq + q] : 0.f;
    bool ok = true;

    if (t == 0) {
        bwd_load_pair(&p.tmQ, &p.tmdO, sQ, sdO, sh.first, i * kBR, bh, kChunks, C::kTile);
        for (int s = 0; s < 2 && s < n_j; ++s)
            bwd_load_pair(&p.tmK, &p.tmV, sK[s], sV[s], sh.load0 + 8 * s, s * kBC, bh, kChunks, C::kTile);
    }
    for (int n = 0; n < n_j; ++n) {
        const int jj = n;
        const int s = n & 1;
        const uint32_t use = n >> 1;
        bool step_ok = true;
        if (t == 0) {
            if (n == 0) step_ok = wait_bar(sh.first, 0, sh.abort_flag, 14, blockIdx.x, -1);
            step_ok = step_ok && wait_bar(sh.load0 + 8 * s, use & 1, sh.abort_flag, 14, blockIdx.x, n);
            if (step_ok) {
                ptx::tc_fence_after_sync();
                issue_s<D>(tmem + tS, sQ, sK[s]);     // S = Q_i K_j^T
                issue_s<D>(tmem + tdP, sdO, sV[s]);   // dP = dO_i V_j^T
                ptx::mma_commit(sh.mma_s);
            }
        }
        if (!__syncthreads_and(step_ok)) { ok = false; break; }
        if (!__syncthreads_and(wait_bar(sh.mma_s, n & 1, sh.abort_flag, 15, blockIdx.x, n))) { ok = false; break; }
        ptx::tc_fence_after_sync();
        // visible key columns: below Nk, and at or before the query on the diagonal
        int col_hi = min(kBC, p.Nk - jj * kBC);
        if (p.causal && jj == i) col_hi = min(col_hi, t + 1);
        if (!qlive) col_hi = 0;
        bwd_elementwise<false, false>(tmem + lane_off + tS, tmem + lane_off + tdP, p.c2, nullptr, nullptr,
                                      row_lse2, row_d, 0, col_hi);
        tmem_stores_to_mma();
        step_ok = true;
        if (t == 0) {
            issue_pv<D>(tmem + tdQ, tmem + tdP, sK[s], n > 0);   // dQ += dS K_j
            ptx::mma_commit(sh.mma_acc0 + 8 * s);
            if (n + 2 < n_j) {
                step_ok = wait_bar(sh.mma_acc0 + 8 * s, use & 1, sh.abort_flag, 16, blockIdx.x, n);
                if (step_ok)
                    bwd_load_pair(&p.tmK, &p.tmV, sK[s], sV[s], sh.load0 + 8 * s, (jj + 2) * kBC, bh, kChunks,
                                  C::kTile);
            }
        }
        if (!__syncthreads_and(step_ok)) { ok = false; break; }
    }
    if (ok) {
        const int s = (n_j - 1) & 1;
        const uint32_t use = (n_j - 1) >> 1;
        if (wait_bar(sh.mma_acc0 + 8 * s, use & 1, sh.abort_flag, 17, blockIdx.x, n_j)) {
            ptx::tc_fence_after_sync();
            store_row_bf16<D>(tmem + lane_off + tdQ, p.scale, p.dQ + (static_cast<size_t>(bh) * p.Nq + q) * D, qlive);
        }
    }
    if (t == 0)
        for (int s = 0; s < 2 && s < n_j; ++s) {
            const int last = ((n_j - 1 - s) / 2) * 2 + s;
            wait_drain(sh.load0 + 8 * s, (last >> 1) & 1);
        }
    bwd_teardown<D>(tmem, sh);
}

}  // namespace fa
