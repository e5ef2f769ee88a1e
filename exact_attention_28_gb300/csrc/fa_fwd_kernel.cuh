// FlashAttention forward for sm_103a: TMA loads, tcgen05 MMAs into tensor
// memory (TMEM), online softmax by dedicated warpgroups, persistent CTAs.
//
// What is computed (per (batch, head), per query row i):
//   S_ij = scale * q_i . k_j over the visible keys j (j < Nk; j <= i if causal)
//   O_i  = sum_j exp(S_ij - m_i) v_j / l_i,  LSE_i = m_i + ln l_i
// following "9.4 FlashAttention 与 FlashMLA" 9.4.2 (online softmax recurrence,
// online update of O, O_final = O / l) and 9.4.3 (fused forward, Q-block outer
// loop, KV-block inner loop), "6. FlashAttention 分块逻辑" 3.1-5.2 (blocked
// loops with causal block classes), and 9.4.5 (store lse = m + log l).
//
// Work decomposition.  A work item is one (batch*head, Q-tile pair): two Q
// tiles of BR = 128 rows that share every K/V tile they stream, or a single
// Q tile for load balancing at the end of the list.  CTAs are persistent: the
// grid is at most one CTA per SM and each CTA walks the item list with a
// static stride, reversing direction every round ("snake") so heavy and light
// items (causal) even out.  Items come in groups of heads whose K/V fit in
// L2 together, heaviest first inside a group.
//
// Roles inside a CTA (head dimension 128: 384 threads, 3 warpgroups; head
// dimension 64: 320 threads, two CTAs per SM):
//   warps 0-3   softmax for Q tile 0 (TMEM lanes 0-127: thread = query row)
//   warps 4-7   softmax for Q tile 1
//   warp  8     TMA producer: Q tiles once per item, then K_j, V_j into a ring
//   warp  9     MMA issuer (one thread) and TMEM owner
//   warps 10-11 idle at head dimension 128 (they complete the third warpgroup)
// At head dimension 128 the softmax warpgroups raise their register limit to
// 208 (128 scores per thread plus room for many exponentials in flight); the
// third warpgroup lowers its own to 88.
//
// Tensor memory (BC = keys per K/V tile: 128 at d = 128, 64 at d = 64; fp32 cells):
//   [0, BC)          S_0 = Q_0 K_j^T (fp32);  P_0 (bf16 pairs) overwrites its first BC/2 columns
//   [BC, 2BC)        S_1 / P_1
//   [2BC, 2BC+D)     O_0 accumulator
//   [2BC+D, 2BC+2D)  O_1 accumulator
// (512 columns at d = 128; 256 at d = 64, so that two CTAs fit an SM.)
//
// MMA order per KV step j (tile t = 0, 1):  PV_0(j), S_0(j+1), PV_1(j), S_1(j+1).
// While the tensor core runs the other tile's two MMAs, the softmax warps of
// tile t turn S_t(j+1) into P_t(j+1).  Because every tcgen05.commit tracks all
// earlier MMAs of the issuing thread, "S_t(j+1) is ready" also means PV_t(j)
// has finished, so the softmax warps may rescale O_t in place at that point.
//
// Online softmax in base 2: with c = scale*log2(e), t_ij = c*S_ij and
// p = 2^(t - m).  The reference maximum m is only raised when a tile's row
// maximum exceeds it by more than TAU = 8 (so p <= 2^8); otherwise the O
// rescale is skipped (alpha == 1 exactly).  The recurrence of 9.4.2 holds for
// any reference value, so the result is unchanged; LSE = ln2 * (m + log2 l).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx_sm103.cuh"

namespace fa {

constexpr int kBR = 128;          // query rows per Q tile (= TMEM lanes)
constexpr int kBC = 128;          // keys per K/V tile of the backward (the forward's is Config::kBC)
constexpr int kSoftmaxWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
// d = 128 (384 threads, one CTA per SM, 168 registers per thread at launch):
constexpr uint32_t kSoftmaxRegs = 208;  // after setmaxnreg
constexpr uint32_t kOtherRegs = 88;     // producer / MMA warpgroup
static_assert(kSoftmaxRegs * 256 + kOtherRegs * 128 <= 168 * 384, "register split exceeds the launch allocation");
constexpr int kChunkBytes = 128 * 128;  // one [128 rows x 64 bf16] swizzled TMA box (backward)
constexpr float kTau = 8.0f;            // log2-domain slack before the max is raised
// E4M3 P: a smaller slack and a headroom, p = 2^(c*s - m + 4) in (0, 2^8]:
// the row maximum's weight lands in [2^4, 2^8] (E4M3 reaches 448), so keys
// up to 14 log2 units below it stay above E4M3's smallest subnormal 2^-9
// instead of 10 (with p <= 1 they would underflow and their mass be lost).
constexpr float kTauF8 = 4.0f;
constexpr float kHeadroomF8 = 4.0f;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait, then abort

// Kernel variants, fixed at compile time so that the dense forward carries
// none of the others' per-tile work.  Independent bits:
//   kSplit -- items cut into key-range slices, fp32 partials (merged afterwards);
//   kPaged -- K/V gathered from a block table, per-sequence key counts;
//   kFp8   -- E4M3 Q, K and transposed V with per-head scales, P in E4M3.
// kDense (none) reads contiguous bf16 K/V and writes bf16 O directly.
enum Mode : int { kDense = 0, kSplit = 1, kPaged = 2, kPagedSplit = 3, kFp8 = 4 };

// Device status word: bit 0 = a pipeline wait expired, bit 1 = a shutdown
// wait expired.  Read and cleared by the host.
__device__ unsigned int g_fa_status;
// First failure: {block, role, item, step}.
__device__ int g_fa_diag[4];

// Tile geometry.  bf16: a [rows][D] tile is D/64 boxes of [rows][64].
// E4M3 (D = 128 only): a Q or K tile is one box of [128 rows][128 bytes] and
// a V tile is V^T's [D channel rows][128 keys], also one box.
//
// Head dimension 128: K/V tiles of BC = 128 keys, one CTA of 384 threads per
// SM holding 512 TMEM columns (S_0, S_1 of 128 columns, O_0, O_1 of 128).
// Head dimension 64: K/V tiles of BC = 64 keys, so one CTA needs only 256
// TMEM columns (S 64 + 64, O 64 + 64) and about 100 KB of shared memory, and
// two CTAs share each SM: four query tiles' softmax warps per SM instead of
// two, which hides the latency of each tile's softmax step behind the other
// tiles' work (at d = 64 a tile's GEMMs are too short to hide it alone).
template <int D, bool F8 = false>
struct Config {
    static_assert(D == 64 || D == 128, "head dimension");
    static_assert(!F8 || D == 128, "the E4M3 path has D = 128 (one 128-byte row per tile row)");
    static constexpr int kElem = F8 ? 1 : 2;
    static constexpr int kBC = D == 64 ? 64 : 128;          // keys per K/V tile
    static constexpr int kCtasPerSm = D == 64 ? 2 : 1;
    static constexpr int kThreads = D == 64 ? 320 : 384;    // d = 64: no idle warps, no register split
    static constexpr bool kRegSplit = D == 128;             // setmaxnreg between the warpgroups
    static constexpr int kChunks = D * kElem / 128;         // 128-byte swizzle chunks per row
    static constexpr int kQChunkBytes = kBR * 128;          // one [128 rows][128 B] box
    static constexpr int kKVChunkBytes = kBC * 128;         // one [BC rows][128 B] box
    static constexpr int kQTileBytes = kBR * D * kElem;
    static constexpr int kKVTileBytes = kBC * D * kElem;
    static constexpr int kSlots = F8 ? 10 : (D == 128 ? 5 : 8);   // K/V ring depth (tiles)
    // Head dimension 64: K(j) and V(j) (ring indices 2i, 2i+1) share one
    // full and one empty barrier, those of the K slot.  The MMA thread then
    // waits once per key step instead of twice and commits one release instead
    // of two (each costs it about as much as issuing an MMA; at d = 64 that
    // thread paces the step).
    static constexpr bool kPairedSlots = D == 64 && !F8;
    static_assert(!kPairedSlots || kSlots % 2 == 0, "paired K/V slots need an even ring");
    static constexpr int kQBytes = 2 * kQTileBytes;
    static constexpr int kRingBytes = kSlots * kKVTileBytes;
    static constexpr int kBarOffset = kQBytes + kRingBytes;
    static constexpr int kSmemBytes = kBarOffset + 256 + 1024;  // + barriers, + alignment slack
    static_assert(kSmemBytes * kCtasPerSm + 1024 * kCtasPerSm <= 233472,
                  "the CTAs of one SM exceed its 228 KB of shared memory");
    static_assert(kSmemBytes <= 232448, "exceeds the 227 KB of shared memory a CTA may use");
    // TMEM columns: S_t at t * BC (P_t, bf16 pairs, over its first BC / 2
    // columns), O_t at 2 * BC + t * D
    static constexpr uint32_t kTmemCols = 2 * kBC + 2 * D;
    static constexpr uint32_t kTmemS = 0, kTmemO = 2 * kBC;
    static_assert(kTmemCols == 256 || kTmemCols == 512, "TMEM allocation is a power of two");
};

// Keys per K/V tile for head dimension d (the host's view of Config::kBC).
__host__ __device__ constexpr int kv_tile_keys(int d) { return d == 64 ? Config<64>::kBC : Config<128>::kBC; }

// Division of a 32-bit unsigned integer by an invariant divisor d >= 1 by a
// multiplication (Granlund and Montgomery, "Division by invariant integers
// using multiplication", PLDI 1994, section 4): with l = ceil(log2 d),
// m = floor(2^32 (2^l - d) / d) + 1 and t = floor(m n / 2^32),
// n / d = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0), exact for every n.
// The work-item decode divides by the head count, the heads per group and
// the key slices; hardware integer division by a runtime value takes tens of
// dependent instructions, which every role paid at every item.
struct FastDiv {
    uint32_t d, m, sh1, sh2;
};
__host__ inline FastDiv make_fastdiv(uint32_t d) {
    uint32_t l = 0;
    while ((uint64_t{1} << l) < d) ++l;   // d < 2^31 here, so l <= 31 and nothing overflows
    const uint64_t m = ((uint64_t{1} << 32) * ((uint64_t{1} << l) - d)) / d + 1;
    return FastDiv{d, static_cast<uint32_t>(m), l < 1 ? l : 1u, l > 1 ? l - 1 : 0u};
}
__host__ __device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f) {
#ifdef __CUDA_ARCH__
    const uint32_t t = __umulhi(f.m, n);
#else
    const uint32_t t = static_cast<uint32_t>((static_cast<uint64_t>(f.m) * n) >> 32);
#endif
    return (t + ((n - t) >> f.sh1)) >> f.sh2;
}

struct FwdParams {
    CUtensorMap tmQ;   // [BH][Nq][D] bf16, box {64, 128, 1}, 128-byte swizzle
    CUtensorMap tmK;   // [BH][Nk][D]
    CUtensorMap tmV;   // [BH][Nk][D]
    __nv_bfloat16 *O;  // [BH][Nq][D]
    float *LSE;        // [BH][Nq]
    int BH, Nq, Nk;
    int Tr;            // Q tiles per head = ceil(Nq / 128)
    int bc;            // keys per K/V tile (Config<D>::kBC)
    int Tc;            // K/V tiles per head = ceil(Nk / bc)
    int P;             // Q-tile pairs per head = ceil(Tr / 2)
    int n_pair_items;  // items [0, n_pair_items) are whole pairs
    int n_items;       // the rest are single tiles of the last pairs in order
    int heads_per_group;  // items are ordered by groups of heads (L2 locality)
    int kv_splits;     // > 1: each item covers 1/kv_splits of its key range and writes partials
    float *O_part;     // [kv_splits][BH][Nq][D] fp32 partial outputs (normalised by their own sum)
    float *LSE_part;   // [kv_splits][BH][Nq] fp32 partial log-sum-exp (-inf: no visible key)
    // paged key/value cache (kPaged kernels): tmK/tmV are 4-D maps over
    // [num_blocks][H][block_size][D]; key position k of sequence b lives in
    // row k % block_size of physical block block_table[b][k / block_size]
    int H, block_size, max_blocks;
    const int *block_table;   // [B][max_blocks]; < 0: unallocated (its keys are skipped)
    const int *seq_lens;      // [B] keys per sequence
    // E4M3 inputs (kFp8 kernels): the value of a code is code * descale[bh];
    // tmV maps V^T [BH][D][ceil16(Nk)]
    const float *descale_q, *descale_k, *descale_v;
    int causal;
    float c2;          // scale * log2(e)
    // test hook (fa_fwd_test_missing_load): the first K tile of this work
    // item is never loaded, so a bounded wait expires; -1 in every other call
    int drop_load_item;
    // invariant divisors of the work-item decode (set with the sizes above)
    FastDiv fd_splits, fd_per_group, fd_hg, fd_last_gsize, fd_bh, fd_2bh, fd_h;
    int bc_shift;          // log2(bc)
    int block_shift;       // paged: log2(block_size)
};

struct Item {
    int bh;
    int q0;        // first query row of tile 0 of this item
    int ntiles;    // 1 or 2
    int kv0;       // first K/V tile of the item's key range
    int nk[2];     // one past the last K/V tile each query tile visits; a tile with
                   // nk <= kv0 has nothing to do in this item
    int split;     // index of the key-range slice (0 without splitting)
    int seq_len;   // keys of this item's sequence (Nk unless paged)
    int q_shift;   // causal: query row i sees keys k <= i + q_shift
};

// Item w of the list.  Heads are taken in groups of heads_per_group whose
// K/V fit in L2 together; inside a group, pairs go by descending pair index
// (for causal the heaviest first), heads inner.  Without key splitting the
// last pairs of the list (the lightest) are split into single-tile items;
// with it, each pair appears kv_splits times in a row, once per slice of the
// keys its tiles can see ("6. FlashAttention 分块逻辑" section 11: the key
// blocks are processed independently and merged afterwards).
__host__ __device__ __forceinline__ Item decode_item(const FwdParams &p, int w, bool splitting) {
    int r, first, single, split = 0;
    if (splitting) {
        r = static_cast<int>(fdiv(w, p.fd_splits)); split = w - r * p.kv_splits; first = 0; single = 0;
    } else if (w < p.n_pair_items) {
        r = w; first = 0; single = 0;
    } else if (!p.causal) {
        const int s = w - p.n_pair_items;   // all tiles cost the same: both tiles of a pair in turn
        r = p.n_pair_items + (s >> 1); first = s & 1; single = 1;
    } else {
        // causal: singles by decreasing cost, i.e. per pair index (heads in
        // chunks of BH) first the upper tile 2p+1 of every head, then the
        // lower tile 2p, so the snake's second round pairs heavy with light
        const int s = w - p.n_pair_items;
        const int r0 = p.n_pair_items;
        // split pairs in the first, partial chunk (the split pairs run to the
        // end of the list, which is a whole number of chunks)
        const int r0_mod = r0 - static_cast<int>(fdiv(r0, p.fd_bh)) * p.BH;
        const int m0 = r0_mod ? p.BH - r0_mod : 0;
        if (s < 2 * m0) {
            first = s < m0 ? 1 : 0;
            r = r0 + (s < m0 ? s : s - m0);
        } else {
            const int s2 = s - 2 * m0, c = static_cast<int>(fdiv(s2, p.fd_2bh)), rem = s2 - c * 2 * p.BH;
            first = rem < p.BH ? 1 : 0;
            r = r0 + m0 + c * p.BH + (rem < p.BH ? rem : rem - p.BH);
        }
        single = 1;
    }
    const int per_group = p.heads_per_group * p.P;
    const int g = static_cast<int>(fdiv(r, p.fd_per_group));
    const int rr = r - g * per_group;
    const int rest = p.BH - g * p.heads_per_group;
    const bool full_group = p.heads_per_group <= rest;
    const int gsize = full_group ? p.heads_per_group : rest;
    const int pq = static_cast<int>(fdiv(rr, full_group ? p.fd_hg : p.fd_last_gsize));
    const int pair = p.P - 1 - pq;
    Item it;
    it.bh = g * p.heads_per_group + (rr - pq * gsize);
    it.q0 = (2 * pair + first) * kBR;
    const int left = p.Tr - (2 * pair + first);
    it.ntiles = single ? 1 : (left >= 2 ? 2 : 1);
    int vis[2];
    #pragma unroll
    for (int t = 0; t < 2; ++t) {
        int nk = 0;
        if (t < it.ntiles) {
            nk = p.Tc;
            if (p.causal) {
                const int q_end_raw = it.q0 + (t + 1) * kBR;
                const int q_end = q_end_raw < p.Nq ? q_end_raw : p.Nq;   // rows >= Nq are padding
                const int need = ((q_end - 1) >> p.bc_shift) + 1;
                nk = need < p.Tc ? need : p.Tc;
            }
        }
        vis[t] = nk;
    }
    it.split = split;
    it.seq_len = p.Nk;
    it.q_shift = 0;
    if (splitting) {
        const int nkv = vis[0] > vis[1] ? vis[0] : vis[1];
        const int kb = static_cast<int>(fdiv(split * nkv, p.fd_splits));
        const int ke = static_cast<int>(fdiv((split + 1) * nkv, p.fd_splits));
        it.kv0 = kb;
        #pragma unroll
        for (int t = 0; t < 2; ++t) it.nk[t] = vis[t] < ke ? vis[t] : ke;
    } else {
        it.kv0 = 0;
        it.nk[0] = vis[0];
        it.nk[1] = vis[1];
    }
    return it;
}

// Device-side completion of an item for the paged cache: the sequence's own
// key count (read from device memory) bounds every tile's key range, and the
// Nq queries are the last Nq positions of the sequence, so under the causal
// mask row i sees keys k <= i + (seq_len - Nq).  With key splitting the
// slices divide this per-sequence range.  A tile left with no visible key
// gets nk <= kv0 (its rows are written as empty).
template <int MODE>
__device__ __forceinline__ Item resolve_item(const FwdParams &p, int w) {
    Item it = decode_item(p, w, (MODE & kSplit) != 0);
    if constexpr ((MODE & kPaged) == 0) {
        return it;
    } else {
        const int cap = p.max_blocks * p.block_size;
        int seq = __ldg(p.seq_lens + fdiv(it.bh, p.fd_h));
        seq = seq < 0 ? 0 : (seq > cap ? cap : seq);
        it.seq_len = seq;
        it.q_shift = seq - p.Nq;
        int vis[2];
        #pragma unroll
        for (int t = 0; t < 2; ++t) {
            int keys = t < it.ntiles ? seq : 0;
            if (p.causal && t < it.ntiles) {
                const int q_end = min(p.Nq, it.q0 + (t + 1) * kBR);
                keys = min(seq, q_end + it.q_shift);
            }
            vis[t] = keys > 0 ? ((keys + p.bc - 1) >> p.bc_shift) : 0;
        }
        if constexpr ((MODE & kSplit) != 0) {
            const int nkv = max(vis[0], vis[1]);
            const int kb = static_cast<int>(fdiv(it.split * nkv, p.fd_splits));
            const int ke = static_cast<int>(fdiv((it.split + 1) * nkv, p.fd_splits));
            it.kv0 = kb;
            #pragma unroll
            for (int t = 0; t < 2; ++t) it.nk[t] = min(vis[t], ke);
        } else {
            it.kv0 = 0;
            it.nk[0] = vis[0];
            it.nk[1] = vis[1];
        }
        return it;
    }
}

// Paged cache: a BC-key tile is read as BC / rows boxes of rows =
// min(block_size, BC) keys, box s from one page.  page_of_box gives that
// page for tile j of sequence b, or -1 when it is unallocated or past the
// table (keys past the table lie beyond the sequence and are masked anyway).
template <int BC>
__device__ __forceinline__ int page_of_box(const FwdParams &p, int b, int j, int s, int rows) {
    const int lp = (j * BC + s * rows) >> p.block_shift;
    return lp < p.max_blocks ? __ldg(p.block_table + static_cast<size_t>(b) * p.max_blocks + lp) : -1;
}

// The pages of all boxes of tile j (at most 8: block_size >= 16).
template <int BC>
__device__ __forceinline__ void pages_of_tile(const FwdParams &p, int b, int j, int rows, int (&pg)[8]) {
    #pragma unroll
    for (int s = 0; s < 8; ++s) pg[s] = s * rows < BC ? page_of_box<BC>(p, b, j, s, rows) : 0;
}

// Loads one BC-key tile of the paged cache from the pages pg (chunks of
// BC rows x 128 bytes).  An unallocated page is read from block 0 (its keys
// are masked by the softmax).
template <int BC>
__device__ __forceinline__ void tma_load_paged_tile(const FwdParams &p, const CUtensorMap *map, uint32_t dst,
                                                    uint32_t bar, int h, int j, int rows, const int (&pg)[8],
                                                    int chunks, uint64_t pol) {
    #pragma unroll
    for (int s = 0; s < 8; ++s) {
        if (s * rows >= BC) break;
        const int phy = pg[s] < 0 ? 0 : pg[s];
        const int row0 = (j * BC + s * rows) & (p.block_size - 1);
        for (int c = 0; c < chunks; ++c)
            ptx::tma_load_4d(dst + c * BC * 128 + s * rows * 128, map, bar, c * 64, row0, h, phy, pol);
    }
}

// Item index of round k for CTA b of G (snake order), or -1 when done.
__host__ __device__ __forceinline__ int item_of_round(const FwdParams &p, int k, int b, int G) {
    const int w = k * G + ((k & 1) ? (G - 1 - b) : b);
    return w < p.n_items ? w : -1;
}
__device__ __forceinline__ int item_of_round(const FwdParams &p, int k) {
    return item_of_round(p, k, blockIdx.x, gridDim.x);
}

struct Shared {
    uint32_t q_full, q_empty;
    uint32_t kv_full0, kv_empty0;  // + 8 * slot
    uint32_t s_full0, p_full0, o_full0;  // + 8 * tile
    // single-tile items: S alternates between the two tiles' S regions;
    // s_alt marks S ready in the second one, pv_done each P V but the last
    uint32_t s_alt, pv_done;
    uint32_t done;
    volatile int *abort_flag;
};

// Bounded wait: true when the phase completed; false after the time limit
// or when another warp of this CTA has aborted.
__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                       int role, int item, int step) {
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((n & 63u) == 0) {
            if (*abort_flag) return false;
            if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                if (atomicOr(&g_fa_status, 1u) == 0u) {
                    g_fa_diag[0] = blockIdx.x; g_fa_diag[1] = role;
                    g_fa_diag[2] = item; g_fa_diag[3] = step;
                }
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         int role, int item, int step) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, abort_flag, role, item, step);
}

// Warp-uniform bounded wait: every lane polls and all leave together, with
// the same result (the MMA warp runs its loop converged).
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                              int role, int item, int step) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, role, item, step));
}

// Bounded wait used while shutting down: ignores the abort flag (copies and
// MMAs already started must still be waited for), gives up after the limit.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((n & 63u) == 0 && ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(&g_fa_status, 2u);
            return false;
        }
    }
}

// ------------------------------------------------------------ producer warp

template <int D, int MODE>
__device__ void producer_role(const FwdParams &p, const Shared &sh, uint32_t smem_q,
                              uint32_t smem_ring, uint32_t &loads_issued, uint32_t &q_arms) {
    using C = Config<D, (MODE & kFp8) != 0>;
    const uint64_t pol_q = ptx::l2_policy_evict_first();
    const uint64_t pol_kv = ptx::l2_policy_evict_last();
    uint32_t it = 0;
    for (int k = 0;; ++k) {
        const int w = item_of_round(p, k);
        if (w < 0) break;
        const Item item = resolve_item<MODE>(p, w);
        if (k > 0 && !wait_bar(sh.q_empty, (k - 1) & 1, sh.abort_flag, 0, w, -1)) break;
        ptx::mbar_arrive_expect_tx(sh.q_full, item.ntiles * C::kQTileBytes);
        ++q_arms;
        for (int t = 0; t < item.ntiles; ++t)
            #pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
                ptx::tma_load_3d(smem_q + t * C::kQTileBytes + c * C::kQChunkBytes, &p.tmQ, sh.q_full,
                                 c * 64, item.q0 + t * kBR, item.bh, pol_q);
        const int nkv = max(item.nk[0], item.nk[1]);
        // paged: the pages of tile j (pg) and of tile j + 1 (pg_next, fetched
        // one tile ahead so the table lookups do not delay the copies)
        [[maybe_unused]] int pg[8], pg_next[8];
        [[maybe_unused]] const int rows = p.block_size < C::kBC ? p.block_size : C::kBC;
        if constexpr ((MODE & kPaged) != 0)
            if (item.kv0 < nkv) pages_of_tile<C::kBC>(p, fdiv(item.bh, p.fd_h), item.kv0, rows, pg_next);
        bool ok = true;
        for (int j = item.kv0; j < nkv && ok; ++j) {
            if constexpr ((MODE & kPaged) != 0) {
                #pragma unroll
                for (int s = 0; s < 8; ++s) pg[s] = pg_next[s];
                if (j + 1 < nkv) pages_of_tile<C::kBC>(p, fdiv(item.bh, p.fd_h), j + 1, rows, pg_next);
            }
            const bool drop = w == p.drop_load_item && j == item.kv0;   // test hook: K(j) never arrives
            #pragma unroll 1
            for (int which = 0; which < 2; ++which, ++it) {
                const uint32_t slot = it % C::kSlots;
                const uint32_t use = it / C::kSlots;
                // paired slots: V(j) lands on K(j)'s barrier, armed for both tiles
                const uint32_t full = sh.kv_full0 + 8 * (C::kPairedSlots ? slot & ~1u : slot);
                if (!C::kPairedSlots || which == 0) {
                    if (!wait_bar(sh.kv_empty0 + 8 * slot, (use & 1) ^ 1, sh.abort_flag, 0, w, j)) {
                        ok = false;
                        break;
                    }
                    if (drop && (C::kPairedSlots || which == 0)) continue;
                    ptx::mbar_arrive_expect_tx(full, (C::kPairedSlots ? 2 : 1) * C::kKVTileBytes);
                } else if (drop) {
                    continue;
                }
                const CUtensorMap *map = which ? &p.tmV : &p.tmK;
                if constexpr ((MODE & kPaged) != 0) {
                    tma_load_paged_tile<C::kBC>(p, map, smem_ring + slot * C::kKVTileBytes, full,
                                                item.bh - static_cast<int>(fdiv(item.bh, p.fd_h)) * p.H, j, rows, pg,
                                        C::kChunks, pol_kv);
                } else if constexpr ((MODE & kFp8) != 0) {
                    // K: rows j*128.. of [Nk][128 B]; V^T: columns j*128.. of [D][ldn]
                    ptx::tma_load_3d(smem_ring + slot * C::kKVTileBytes, map, full, which ? j * C::kBC : 0,
                                     which ? 0 : j * C::kBC, item.bh, pol_kv);
                } else {
                    #pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        ptx::tma_load_3d(smem_ring + slot * C::kKVTileBytes + c * C::kKVChunkBytes, map, full,
                                         c * 64, j * C::kBC, item.bh, pol_kv);
                }
                loads_issued = it + 1;
            }
        }
        if (!ok) break;
    }
}

// Paged cache: the whole producer warp runs this loop.  Lane 0 waits for free
// ring slots and arms the barriers; lane c + chunks * s copies box s (keys
// s * rows .. of the tile, one page) of column chunk c, so the up to 16 boxes
// of a tile of 16-key pages leave in one warp instruction instead of one
// after another, and each lane looks up the page of its own box, one tile
// ahead.
template <int D, int MODE>
__device__ void producer_role_paged(const FwdParams &p, const Shared &sh, uint32_t smem_q, uint32_t smem_ring,
                                    uint32_t &loads_issued, uint32_t &q_arms, int lane) {
    using C = Config<D, false>;
    const uint64_t pol_q = ptx::l2_policy_evict_first();
    const uint64_t pol_kv = ptx::l2_policy_evict_last();
    const int rows = p.block_size < C::kBC ? p.block_size : C::kBC;
    const int copies = (C::kBC / rows) * C::kChunks;   // <= 16
    const int box = lane / C::kChunks, chunk = lane % C::kChunks;
    const bool mine = lane < copies;
    uint32_t it = 0;
    for (int k = 0;; ++k) {
        const int w = item_of_round(p, k);
        if (w < 0) break;
        const Item item = resolve_item<MODE>(p, w);
        bool ok = true;
        if (lane == 0) {
            if (k > 0 && !wait_bar(sh.q_empty, (k - 1) & 1, sh.abort_flag, 0, w, -1)) {
                ok = false;
            } else {
                ptx::mbar_arrive_expect_tx(sh.q_full, item.ntiles * C::kQTileBytes);
                ++q_arms;
                for (int t = 0; t < item.ntiles; ++t)
                    #pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        ptx::tma_load_3d(smem_q + t * C::kQTileBytes + c * C::kQChunkBytes, &p.tmQ, sh.q_full,
                                         c * 64, item.q0 + t * kBR, item.bh, pol_q);
            }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        const int nkv = max(item.nk[0], item.nk[1]);
        const int b = static_cast<int>(fdiv(item.bh, p.fd_h)), h = item.bh - b * p.H;
        int page_next = (mine && item.kv0 < nkv) ? page_of_box<C::kBC>(p, b, item.kv0, box, rows) : 0;
        for (int j = item.kv0; j < nkv && ok; ++j) {
            const int page = page_next;
            if (mine && j + 1 < nkv) page_next = page_of_box<C::kBC>(p, b, j + 1, box, rows);
            #pragma unroll 1
            for (int which = 0; which < 2; ++which, ++it) {
                const uint32_t slot = it % C::kSlots;
                const uint32_t use = it / C::kSlots;
                // paired slots: V(j) lands on K(j)'s barrier, armed for both tiles
                const uint32_t full = sh.kv_full0 + 8 * (C::kPairedSlots ? slot & ~1u : slot);
                const bool skip = w == p.drop_load_item && j == item.kv0 && (C::kPairedSlots || which == 0);   // test hook
                bool armed = true;
                if (lane == 0 && (!C::kPairedSlots || which == 0)) {
                    armed = wait_bar(sh.kv_empty0 + 8 * slot, (use & 1) ^ 1, sh.abort_flag, 0, w, j);
                    if (armed && !skip)
                        ptx::mbar_arrive_expect_tx(full, (C::kPairedSlots ? 2 : 1) * C::kKVTileBytes);
                }
                if (!__shfl_sync(0xffffffffu, armed, 0)) {
                    ok = false;
                    break;
                }
                __syncwarp();   // lane 0's expect_tx is ordered before the copies (the count may also go below zero)
                if (!skip && mine) {
                    // an unallocated page is read from block 0 (its keys are masked by the softmax)
                    const int phy = page < 0 ? 0 : page;
                    const int row0 = (j * C::kBC + box * rows) & (p.block_size - 1);
                    ptx::tma_load_4d(smem_ring + slot * C::kKVTileBytes + chunk * C::kKVChunkBytes + box * rows * 128,
                                     which ? &p.tmV : &p.tmK, full, chunk * 64, row0, h, phy, pol_kv);
                }
                loads_issued = it + 1;
            }
        }
        if (!ok) break;
    }
}

// ----------------------------------------------------------------- MMA warp

// S_t = Q_t K_j^T: D/16 MMAs of K = 16, N = BC.  Q and K tiles are D/64
// boxes of [128 or BC rows][64 cols], 128-byte swizzled; step kk reads
// columns 16kk..16kk+15, i.e. box kk/4 at byte offset 32*(kk%4) inside each
// 128-byte row.
// E4M3: D/32 MMAs of K = 32, the same 32-byte steps inside the one chunk.
// (The backward calls it with BC = 128 for its transposed products.)
template <int D, int BC, bool F8 = false>
__device__ __forceinline__ void issue_s(uint32_t tmem_s, uint32_t q_tile, uint32_t k_tile) {
    constexpr int kElem = F8 ? 1 : 2;
    constexpr uint32_t kIdesc =
        F8 ? ptx::instr_desc_e4m3_f32(kBR, BC) : ptx::instr_desc_bf16_f32(kBR, BC, false, false);
    constexpr uint32_t hi = ptx::sdesc_sw128_hi(1024);
    const uint32_t a0 = ptx::sdesc_sw128_lo(q_tile, 16);
    const uint32_t b0 = ptx::sdesc_sw128_lo(k_tile, 16);
    constexpr int kSteps = D * kElem / 32;
    #pragma unroll
    for (int kk = 0; kk < kSteps; ++kk) {
        const uint32_t offa = ((kk >> 2) * (kBR * 128) + (kk & 3) * 32) >> 4;
        const uint32_t offb = ((kk >> 2) * (BC * 128) + (kk & 3) * 32) >> 4;
        if constexpr (F8)
            ptx::mma_f8_ss(tmem_s, a0 + offa, hi, b0 + offb, hi, kIdesc, kk > 0 ? 1u : 0u);
        else
            ptx::mma_bf16_ss(tmem_s, a0 + offa, hi, b0 + offb, hi, kIdesc, kk > 0 ? 1u : 0u);
    }
}

// O_t (+)= P_t V_j: BC/16 MMAs of K = 16 keys; P_t is read from TMEM (16
// keys = 8 columns of bf16 pairs per step).  V tile: [BC keys][D] as D/64
// boxes of [BC][64]; the B operand is MN-major (D contiguous): 8-key groups
// SBO = 1024 B apart, 64-column groups LBO = one box (BC * 128 B) apart.
//
// E4M3: 4 MMAs of K = 32 keys; P is 4 keys per TMEM column (8 columns per
// step) and V^T [D rows][128 keys] is a K-major operand like K in S: 8-row
// groups 1024 B apart, 32-byte steps along the keys.
template <int D, int BC, bool F8 = false>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint32_t v_tile,
                                         bool accumulate) {
    // bf16: V [keys][D] is an MN-major B operand; E4M3: V^T [D][keys] is K-major
    constexpr uint32_t kIdesc =
        F8 ? ptx::instr_desc_e4m3_f32(kBR, D) : ptx::instr_desc_bf16_f32(kBR, D, false, true);
    constexpr uint32_t hi = ptx::sdesc_sw128_hi(1024);
    if constexpr (F8) {
        const uint32_t b0 = ptx::sdesc_sw128_lo(v_tile, 16);
        #pragma unroll
        for (int kk = 0; kk < BC / 32; ++kk)
            ptx::mma_f8_ts(tmem_o, tmem_p + kk * 8, b0 + ((kk * 32) >> 4), hi, kIdesc,
                           (accumulate || kk > 0) ? 1u : 0u);
    } else {
        const uint32_t b0 = ptx::sdesc_sw128_lo(v_tile, BC * 128);
        #pragma unroll
        for (int kk = 0; kk < BC / 16; ++kk)
            ptx::mma_bf16_ts(tmem_o, tmem_p + kk * 8, b0 + ((kk * 16 * 128) >> 4), hi, kIdesc,
                             (accumulate || kk > 0) ? 1u : 0u);
    }
}

template <int D, int MODE>
__device__ void mma_role(const FwdParams &p, const Shared &sh, uint32_t tmem, uint32_t smem_q,
                         uint32_t smem_ring) {
    constexpr bool F8 = (MODE & kFp8) != 0;
    using C = Config<D, F8>;
    uint32_t it = 0;
    uint32_t p_phase[2] = {0u, 0u};
    const uint32_t tS[2] = {tmem + C::kTmemS, tmem + C::kTmemS + C::kBC};
    const uint32_t tO[2] = {tmem + C::kTmemO, tmem + C::kTmemO + D};
    const uint32_t sQ[2] = {smem_q, smem_q + C::kQTileBytes};
    for (int k = 0;; ++k) {
        const int w = item_of_round(p, k);
        if (w < 0) break;
        const Item item = resolve_item<MODE>(p, w);
        const int kv0 = item.kv0;
        const int nk0 = item.nk[0], nk1 = item.nk[1];   // tile t is active for kv0 <= j < nk_t
        const int nkv = max(nk0, nk1);
        if (!wait_bar_warp(sh.q_full, k & 1, sh.abort_flag, 1, w, -1)) return;
        ptx::tc_fence_after_sync();
        if (nkv <= kv0) {   // an empty key slice: release Q and move on
            ptx::mma_commit(sh.q_empty);
            continue;
        }

        if (item.ntiles == 1) {
            // One query tile: S alternates between the two S regions, so S(j+1)
            // is computed while the softmax works on S(j), and only P(j) V_j
            // lies between two softmax steps.  Ring index of K(j) is
            // b0 + 2 (j - kv0), of V(j) one more.
            const uint32_t b0 = it;
            auto ring_bar = [&](uint32_t idx) { return sh.kv_full0 + 8 * (idx % C::kSlots); };
            auto ring_tile = [&](uint32_t idx) { return smem_ring + (idx % C::kSlots) * C::kKVTileBytes; };
            auto issue_s_buf = [&](int jj) -> bool {   // S(jj) into buffer (jj - kv0) & 1
                const uint32_t ki = b0 + 2 * (jj - kv0);
                if (!wait_bar_warp(ring_bar(ki), (ki / C::kSlots) & 1, sh.abort_flag, 1, w, jj)) return false;
                ptx::tc_fence_after_sync();
                const int buf = (jj - kv0) & 1;
                issue_s<D, C::kBC, F8>(tS[buf], sQ[0], ring_tile(ki));
                ptx::mma_commit(buf ? sh.s_alt : sh.s_full0);
                if (!C::kPairedSlots) ptx::mma_commit(sh.kv_empty0 + 8 * (ki % C::kSlots));
                return true;
            };
            if (!issue_s_buf(kv0)) return;
            if (kv0 + 1 < nk0 && !issue_s_buf(kv0 + 1)) return;
            if (nk0 <= kv0 + 2) ptx::mma_commit(sh.q_empty);   // every S of the item issued
            for (int j = kv0; j < nk0; ++j) {
                const uint32_t vi = b0 + 2 * (j - kv0) + 1;
                // paired slots: V(j) arrived with K(j), before S(j) was issued
                if (!C::kPairedSlots && !wait_bar_warp(ring_bar(vi), (vi / C::kSlots) & 1, sh.abort_flag, 1, w, j)) return;
                if (!wait_bar_warp(sh.p_full0, p_phase[0], sh.abort_flag, 1, w, j)) return;
                p_phase[0] ^= 1u;
                ptx::tc_fence_after_sync();
                issue_pv<D, C::kBC, F8>(tO[0], tS[(j - kv0) & 1], ring_tile(vi), j > kv0);
                ptx::mma_commit(j == nk0 - 1 ? sh.o_full0 : sh.pv_done);
                ptx::mma_commit(sh.kv_empty0 + 8 * ((C::kPairedSlots ? vi - 1 : vi) % C::kSlots));
                if (j + 2 < nk0) {
                    if (!issue_s_buf(j + 2)) return;
                    if (j + 3 == nk0) ptx::mma_commit(sh.q_empty);
                }
            }
            it = b0 + 2 * (nk0 - kv0);
            continue;
        }

        // S_t(kv0) for both tiles from the first K tile.
        uint32_t ks = it % C::kSlots;
        if (!wait_bar_warp(sh.kv_full0 + 8 * ks, (it / C::kSlots) & 1, sh.abort_flag, 1, w, kv0)) return;
        ptx::tc_fence_after_sync();
        for (int t = 0; t < 2; ++t) {
            if (item.nk[t] > kv0) {
                issue_s<D, C::kBC, F8>(tS[t], sQ[t], smem_ring + ks * C::kKVTileBytes);
                ptx::mma_commit(sh.s_full0 + 8 * t);
            }
        }
        if (!C::kPairedSlots) ptx::mma_commit(sh.kv_empty0 + 8 * ks);
        if (nkv == kv0 + 1) ptx::mma_commit(sh.q_empty);
        ++it;

        for (int j = kv0; j < nkv; ++j) {
            const uint32_t vs = it % C::kSlots;
            // paired slots: V(j) arrived with K(j), before S(j) was issued
            if (!C::kPairedSlots) {
                if (!wait_bar_warp(sh.kv_full0 + 8 * vs, (it / C::kSlots) & 1, sh.abort_flag, 1, w, j)) return;
                ptx::tc_fence_after_sync();
            }
            ++it;
            const uint32_t v_tile = smem_ring + vs * C::kKVTileBytes;
            const bool more = j + 1 < nkv;
            const uint32_t ks2 = it % C::kSlots;

            // Each tile's step is a cycle: softmax_t(j) -> P_t(j) V_j -> S_t(j+1)
            // -> softmax_t(j+1).  Only MMA issues sit in it: K(j+1) is awaited
            // before P_0(j) (this thread is idle until then anyway) and V_j's
            // slot is released after S_1(j+1).
            if (more) {
                if (!wait_bar_warp(sh.kv_full0 + 8 * ks2, (it / C::kSlots) & 1, sh.abort_flag, 1, w, j + 1))
                    return;
            }
            if (j < nk0) {
                if (!wait_bar_warp(sh.p_full0, p_phase[0], sh.abort_flag, 1, w, j)) return;
                p_phase[0] ^= 1u;
                ptx::tc_fence_after_sync();
                issue_pv<D, C::kBC, F8>(tO[0], tS[0], v_tile, j > kv0);
                if (j == nk0 - 1) ptx::mma_commit(sh.o_full0);
            }
            ptx::tc_fence_after_sync();
            if (more && j + 1 < nk0) {
                issue_s<D, C::kBC, F8>(tS[0], sQ[0], smem_ring + ks2 * C::kKVTileBytes);
                ptx::mma_commit(sh.s_full0);
            }
            if (j < nk1) {
                if (!wait_bar_warp(sh.p_full0 + 8, p_phase[1], sh.abort_flag, 1, w, j)) return;
                p_phase[1] ^= 1u;
                ptx::tc_fence_after_sync();
                issue_pv<D, C::kBC, F8>(tO[1], tS[1], v_tile, j > kv0);
                if (j == nk1 - 1) ptx::mma_commit(sh.o_full0 + 8);
            }
            if (more && j + 1 < nk1) {
                issue_s<D, C::kBC, F8>(tS[1], sQ[1], smem_ring + ks2 * C::kKVTileBytes);
                ptx::mma_commit(sh.s_full0 + 8);
            }
            ptx::mma_commit(sh.kv_empty0 + 8 * (C::kPairedSlots ? vs - 1 : vs));   // paired: the K/V pair
            if (more) {
                if (!C::kPairedSlots) ptx::mma_commit(sh.kv_empty0 + 8 * ks2);
                if (j + 2 == nkv) ptx::mma_commit(sh.q_empty);
                ++it;
            }
        }
    }
}

// ------------------------------------------------------------ softmax warps
//
// One softmax warpgroup per Q tile; thread = query row = TMEM lane (warp w
// reads lanes 32*(w%4)..+31).  Each thread holds its row's 128 scores in
// registers (the warpgroup runs with 208 registers, see the kernel), so the
// row maximum is an in-register reduction and many exponentials of
// independent pairs can be in flight together.

// Row extreme (max for a positive scale, min for a negative one) of N = 64
// or 128 scores: eight independent three-input chains, then a short tree.
template <int N>
__device__ __forceinline__ float row_extreme(const uint32_t (&s)[N], bool pos) {
    static_assert(N == 64 || N == 128, "row length");
    float a[8];
    #pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = __uint_as_float(s[i]);
    if (pos) {
        #pragma unroll
        for (int c = 8; c + 16 <= N - 8; c += 16)
            #pragma unroll
            for (int i = 0; i < 8; ++i)
                a[i] = ptx::max3(a[i], __uint_as_float(s[c + 2 * i]), __uint_as_float(s[c + 2 * i + 1]));
        #pragma unroll
        for (int i = 0; i < 4; ++i)
            a[i] = ptx::max3(a[i], __uint_as_float(s[N - 8 + 2 * i]), __uint_as_float(s[N - 7 + 2 * i]));
        return fmaxf(ptx::max3(a[0], a[1], a[2]), ptx::max3(a[3], ptx::max3(a[4], a[5], a[6]), a[7]));
    }
    #pragma unroll
    for (int c = 8; c + 16 <= N - 8; c += 16)
        #pragma unroll
        for (int i = 0; i < 8; ++i)
            a[i] = ptx::min3(a[i], __uint_as_float(s[c + 2 * i]), __uint_as_float(s[c + 2 * i + 1]));
    #pragma unroll
    for (int i = 0; i < 4; ++i)
        a[i] = ptx::min3(a[i], __uint_as_float(s[N - 8 + 2 * i]), __uint_as_float(s[N - 7 + 2 * i]));
    return fminf(ptx::min3(a[0], a[1], a[2]), ptx::min3(a[3], ptx::min3(a[4], a[5], a[6]), a[7]));
}

// P for the row's N scores: p = 2^(c*s - m), packed to bf16 pairs (round
// to nearest even) and stored over the first N/2 TMEM columns of the S tile;
// returns the row sum of the fp32 p.  Masked keys hold -inf*sign(c) and come
// out as p = 0.  (The sum that normalises O adds the bf16 rounding of each
// tile's largest weight, see max_weight_rounding.)
template <int N>
__device__ __forceinline__ void exp_pack_store(const uint32_t (&s)[N], float c2, float neg_m, uint32_t tP,
                                               float &sum_exact) {
    const uint64_t c2x2 = ptx::f2_pack(c2, c2), mx2 = ptx::f2_pack(neg_m, neg_m);
    uint64_t acc_e[4];
    #pragma unroll
    for (int i = 0; i < 4; ++i) acc_e[i] = ptx::f2_pack(0.f, 0.f);
    uint32_t pk[N / 2];
    #pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        const uint64_t t = ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])),
                                       c2x2, mx2);
        float t0, t1;
        ptx::f2_unpack(t, t0, t1);
        const float p0 = ptx::ex2(t0), p1 = ptx::ex2(t1);
        acc_e[i & 3] = ptx::f2_add(acc_e[i & 3], ptx::f2_pack(p0, p1));
        pk[i] = ptx::pack_bf16x2(p0, p1);
    }
    #pragma unroll
    for (int q = 0; q < N / 32; ++q)
        ptx::tmem_store_16cols(tP + 16 * q, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16 * q]));
    float e0, e1;
    ptx::f2_unpack(ptx::f2_add(ptx::f2_add(acc_e[0], acc_e[1]), ptx::f2_add(acc_e[2], acc_e[3])), e0, e1);
    sum_exact = e0 + e1;
}

// Transpose, within each group of 8 lanes, the 8 x 8 matrix whose row j is
// lane j's eight 16-byte pieces x[4e .. 4e+3], e = 0..7: afterwards lane j
// holds piece j of lane e's row in x[4e .. 4e+3].  Three butterfly exchanges
// (lane distance 4, 2, 1), each swapping the off-diagonal blocks of that size.
__device__ __forceinline__ void transpose_8x8_pieces(uint32_t (&x)[32]) {
    const uint32_t lane = threadIdx.x & 31u;
    #pragma unroll
    for (int m = 4; m >= 1; m >>= 1) {
        const bool upper = (lane & static_cast<uint32_t>(m)) != 0;
        #pragma unroll
        for (int e = 0; e < 8; ++e) {
            if (e & m) continue;
            #pragma unroll
            for (int w = 0; w < 4; ++w) {
                // the lower lane gives away its piece e|m and takes the partner's piece e
                const uint32_t give = upper ? x[4 * e + w] : x[4 * (e | m) + w];
                const uint32_t take = __shfl_xor_sync(0xffffffffu, give, m);
                if (upper) x[4 * e + w] = take;
                else x[4 * (e | m) + w] = take;
            }
        }
    }
}

// bf16(p) - p for the weight p of the tile's extreme score mx, computed with
// the arithmetic exp_pack_store applies to that key, so the result is the
// exact rounding error P V sees on the row's largest weight of the tile.
// O is normalised by the fp32 sum plus these errors: a row dominated by one
// key then carries no 2^-9 relative bias into O (the weights of the other
// keys are small, and their rounding errors average out).
__device__ __forceinline__ float max_weight_rounding(float mx, float c2, float neg_m) {
    float t, t1;
    ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(mx, mx), ptx::f2_pack(c2, c2), ptx::f2_pack(neg_m, neg_m)), t, t1);
    const float pmax = ptx::ex2(t);
    const uint32_t pk = ptx::pack_bf16x2(pmax, pmax);
    return __uint_as_float(pk << 16) - pmax;
}

// E4M3 P: the same exponentials, packed four keys to a TMEM column (32
// columns over the start of the S tile); the rounded sum adds the E4M3 values
// (widened exactly) that P V uses.
__device__ __forceinline__ void exp_pack_store128_e4m3(const uint32_t (&s)[128], float c2, float neg_m, uint32_t tP,
                                                       float &sum_exact, float &sum_rounded) {
    const uint64_t c2x2 = ptx::f2_pack(c2, c2), mx2 = ptx::f2_pack(neg_m, neg_m);
    uint64_t acc_e[4];
    #pragma unroll
    for (int i = 0; i < 4; ++i) acc_e[i] = ptx::f2_pack(0.f, 0.f);
    float r[8];
    #pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = 0.f;
    uint32_t pk[32];
    #pragma unroll
    for (int i = 0; i < 32; ++i) {
        float p[4];
        #pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint64_t t = ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[4 * i + 2 * h]),
                                                        __uint_as_float(s[4 * i + 2 * h + 1])), c2x2, mx2);
            float t0, t1;
            ptx::f2_unpack(t, t0, t1);
            p[2 * h] = ptx::ex2(t0);
            p[2 * h + 1] = ptx::ex2(t1);
            acc_e[(2 * i + h) & 3] = ptx::f2_add(acc_e[(2 * i + h) & 3], ptx::f2_pack(p[2 * h], p[2 * h + 1]));
        }
        pk[i] = ptx::pack_e4m3x4(p[0], p[1], p[2], p[3]);
        ptx::add_e4m3x4_to_f32(r[4 * (i & 1)], r[4 * (i & 1) + 1], r[4 * (i & 1) + 2], r[4 * (i & 1) + 3], pk[i]);
    }
    ptx::tmem_store_32cols(tP, pk);
    float e0, e1;
    ptx::f2_unpack(ptx::f2_add(ptx::f2_add(acc_e[0], acc_e[1]), ptx::f2_add(acc_e[2], acc_e[3])), e0, e1);
    sum_exact = e0 + e1;
    sum_rounded = ((r[0] + r[1]) + (r[2] + r[3])) + ((r[4] + r[5]) + (r[6] + r[7]));
}

template <int D, int MODE>
__device__ void softmax_role(const FwdParams &p, const Shared &sh, uint32_t tmem, int tile, int quad, int lane) {
    constexpr bool F8 = (MODE & kFp8) != 0;
    using C = Config<D, F8>;
    constexpr int BC = C::kBC;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::kTmemS + tile * BC;
    const uint32_t tO = tmem + lane_off + C::kTmemO + tile * D;
    float c2 = p.c2;
    const bool pos = c2 > 0.f;   // the descales are positive: the sign is the scale's
    // A masked key must never win the row extreme and must give p = 0:
    // -inf for a positive scale, +inf for a negative one (the host never
    // passes c2 == 0, see fa_fwd).
    const float mask_val = pos ? -INFINITY : INFINITY;
    // paged: keys per box (min(block_size, BC)) and its log2
    [[maybe_unused]] const int page_rows = p.block_size < BC ? p.block_size : BC;
    [[maybe_unused]] const int page_shift = (MODE & kPaged) != 0 ? 31 - __clz(page_rows) : 0;
    uint32_t s_phase = 0, o_phase = 0;
    uint32_t sa_phase = 0, pv_phase = 0;   // single-tile items (tile 0 only)

    for (int k = 0;; ++k) {
        const int w = item_of_round(p, k);
        if (w < 0) break;
        const Item item = resolve_item<MODE>(p, w);
        if (tile >= item.ntiles) continue;
        const int nk = item.nk[tile];
        const int qg = item.q0 + tile * kBR + row;   // this thread's query row
        const size_t prow = (static_cast<size_t>(item.split) * p.BH + item.bh) * p.Nq + qg;   // partial row
        // no visible key for this tile (in this slice): empty rows.  Every
        // dense tile sees key 0, so only the other variants test for it.
        if (MODE != kDense && nk <= item.kv0) {
            if (qg < p.Nq) {
                if ((MODE & kSplit) != 0) {
                    p.LSE_part[prow] = -INFINITY;
                } else {
                    __nv_bfloat16 *orow = p.O + (static_cast<size_t>(item.bh) * p.Nq + qg) * D;
                    for (int c = 0; c < D; c += 8) __stcs(reinterpret_cast<uint4 *>(orow + c), make_uint4(0, 0, 0, 0));
                    p.LSE[static_cast<size_t>(item.bh) * p.Nq + qg] = -INFINITY;
                }
            }
            continue;
        }
        const int key_lim = p.causal ? min(item.seq_len, qg + 1 + item.q_shift) : item.seq_len;
        const bool single = item.ntiles == 1;
        [[maybe_unused]] float out_scale = 1.f;   // E4M3: V's descale
        if constexpr (F8) {
            // scores of the codes times descale_q * descale_k; kept a normal
            // number (at least the smallest), like the host does for a zero
            // scale: the flush-to-zero arithmetic below would read a subnormal
            // as 0, and a masked key's -inf times 0 is NaN
            c2 = p.c2 * __ldg(p.descale_q + item.bh) * __ldg(p.descale_k + item.bh);
            if (fabsf(c2) < 1.17549435e-38f) c2 = pos ? 1.17549435e-38f : -1.17549435e-38f;
            out_scale = __ldg(p.descale_v + item.bh);
        }
        float m_ref = -INFINITY;   // log2-domain reference maximum
        float l = 0.f;             // sum of p (fp32), for LSE
        float l_rounded = 0.f;     // the sum that normalises O (E4M3: of the rounded p;
                                   // bf16: the rounding of each tile's largest weight, added to l)

        for (int j = item.kv0; j < nk; ++j) {
            // paged: lane s looks up the page of box s of this tile before the
            // wait, so the load overlaps it
            [[maybe_unused]] int box_page = 0;
            if constexpr ((MODE & kPaged) != 0)
                if (lane * page_rows < BC) box_page = page_of_box<BC>(p, fdiv(item.bh, p.fd_h), j, lane, page_rows);
            // single-tile items alternate S buffers (the second is tile 1's region)
            const bool alt = single && ((j - item.kv0) & 1);
            const uint32_t tSj = tS + (alt ? static_cast<uint32_t>(BC) : 0u);
            if (alt) {
                if (!wait_bar(sh.s_alt, sa_phase, sh.abort_flag, 2, w, j)) return;
                sa_phase ^= 1u;
            } else {
                if (!wait_bar(sh.s_full0 + 8 * tile, s_phase, sh.abort_flag, 2 + tile, w, j)) return;
                s_phase ^= 1u;
            }
            ptx::tc_fence_after_sync();
            // S; at head dimension 64 the load's own max reduction gives the row
            // maximum for a positive scale (a negative scale needs the minimum:
            // software).  At 128 it measured no faster than the software maximum.
            constexpr bool kHwMax = BC == 64;
            uint32_t s[BC];
            float mparts[BC / 32];
            if (kHwMax && pos) {
                if constexpr (BC == 128)
                    ptx::tmem_load_128cols_max(tSj, s, mparts);
                else
                    ptx::tmem_load_64cols_max(tSj, s, mparts);
            } else {
                if constexpr (BC == 128)
                    ptx::tmem_load_128cols(tSj, s);
                else
                    ptx::tmem_load_64cols(tSj, s);
            }
            const int kvalid = key_lim - j * BC;
            bool masked;   // warp-uniform: some key of this tile is invisible to some row of the warp
            if constexpr ((MODE & kPaged) != 0) {
                // bit s: box s lies in an unallocated page (warp-uniform)
                const uint32_t holes = __ballot_sync(0xffffffffu, box_page < 0);
                masked = __any_sync(0xffffffffu, kvalid < BC) || holes;
                if (masked) {
                    // column mask, bit c % 32 of word c / 32 (a box holds >= 16 columns)
                    uint32_t cm[BC / 32];
                    #pragma unroll
                    for (int q = 0; q < BC / 32; ++q) {
                        cm[q] = ((holes >> ((32 * q) >> page_shift)) & 1u) ? 0x0000FFFFu : 0u;
                        cm[q] |= ((holes >> ((32 * q + 16) >> page_shift)) & 1u) ? 0xFFFF0000u : 0u;
                    }
                    #pragma unroll
                    for (int c = 0; c < BC; ++c)
                        if (c >= kvalid || ((cm[c >> 5] >> (c & 31)) & 1u)) s[c] = __float_as_uint(mask_val);
                }
            } else {
                masked = __any_sync(0xffffffffu, kvalid < BC);
                if (masked) {
                    #pragma unroll
                    for (int c = 0; c < BC; ++c)
                        if (c >= kvalid) s[c] = __float_as_uint(mask_val);
                }
            }
            float mx;
            if (kHwMax && pos && !masked) {
                if constexpr (BC == 128)
                    mx = fmaxf(ptx::max3(mparts[0], mparts[1], mparts[2]), mparts[3]);
                else
                    mx = fmaxf(mparts[0], mparts[1]);
            } else {
                mx = row_extreme<BC>(s, pos);   // over the masked scores
            }
            const float m_tile = kvalid > 0 ? mx * c2 : -INFINITY;
            float alpha = 1.f;
            if (m_tile > m_ref + (F8 ? kTauF8 : kTau)) {
                alpha = ptx::ex2(m_ref - m_tile);   // 0 on the first visible tile
                m_ref = m_tile;
            }
            l *= alpha;
            l_rounded *= alpha;

            // m_ref is finite once a row has seen a key (every row sees key 0
            // in its first tile); the guard keeps a fully masked row at p = 0.
            if constexpr (F8) {
                float se, sr;
                exp_pack_store128_e4m3(s, c2, m_ref == -INFINITY ? 0.f : kHeadroomF8 - m_ref, tSj, se, sr);
                l += se;
                l_rounded += sr;
            } else {
                const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
                float se;
                exp_pack_store<BC>(s, c2, neg_m, tSj, se);
                l += se;
                if (m_tile != -INFINITY) l_rounded += max_weight_rounding(mx, c2, neg_m);
            }
            // single-tile items: S(j) ready no longer implies P(j-1) V done;
            // wait for it before O may be rescaled (it is normally done by now)
            if (single && j > item.kv0) {
                if (!wait_bar(sh.pv_done, pv_phase, sh.abort_flag, 2, w, j)) return;
                pv_phase ^= 1u;
                ptx::tc_fence_after_sync();
            }
            // Rescale O_t in TMEM when this warp's reference maximum moved
            // (PV_t(j-1) has completed, see the header; PV_t(j) waits for us).
            if (__any_sync(0xffffffffu, j > item.kv0 && alpha != 1.f)) {
                #pragma unroll 1
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t o[32];
                    ptx::tmem_load_32cols(tO + ch * 32, o);
                    #pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    ptx::tmem_store_32cols(tO + ch * 32, o);
                }
            }
            ptx::tmem_wait_store();
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(sh.p_full0 + 8 * tile);
        }

        // Epilogue: O = O / l in bf16, LSE = ln2 * (m + log2 l).
        if (!wait_bar(sh.o_full0 + 8 * tile, o_phase, sh.abort_flag, 2 + tile, w, nk)) return;
        o_phase ^= 1u;
        ptx::tc_fence_after_sync();
        // a row that saw no key at all (possible only with the paged cache) is empty: O = 0, LSE = -inf
        if constexpr (!F8) l_rounded += l;
        float inv_l = l_rounded > 0.f ? 1.f / l_rounded : 0.f;
        if constexpr (F8) inv_l *= out_scale;
        const bool live = qg < p.Nq;
        // (the E4M3 weights carry the headroom factor 2^4: l does too, O not)
        const float lse = l > 0.f ? (m_ref - (F8 ? kHeadroomF8 : 0.f) + ptx::lg2(l)) * 0.69314718055994531f
                                  : -INFINITY;
        if constexpr ((MODE & kSplit) != 0) {
            // partial of this key slice: O / l in fp32 and its LSE
            // whole 128-byte lines, as below: 32 fp32 columns are eight 16-byte pieces
            const uint32_t j8 = threadIdx.x & 7u;
            #pragma unroll 1
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t o[32];
                ptx::tmem_load_32cols(tO + ch * 32, o);
                #pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * inv_l);
                transpose_8x8_pieces(o);
                #pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int r = qg - static_cast<int>(j8) + e;
                    if (r < p.Nq)
                        __stcs(reinterpret_cast<uint4 *>(p.O_part + (prow - j8 + e) * D + 32 * ch + 4 * j8),
                               make_uint4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]));
                }
            }
            if (live) p.LSE_part[prow] = lse;
        } else {
            // O leaves as whole 128-byte lines: 64 columns at a time, each group of
            // 8 lanes (8 consecutive rows) exchanges its 8 x 8 block of 16-byte
            // pieces, so that in store e the group writes all of row e's 128 bytes.
            const uint32_t j8 = threadIdx.x & 7u;
            #pragma unroll 1
            for (int c = 0; c < D / 64; ++c) {
                uint32_t o[64];
                ptx::tmem_load_64cols(tO + c * 64, o);
                uint32_t x[32];
                #pragma unroll
                for (int i = 0; i < 32; ++i)
                    x[i] = ptx::pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
                transpose_8x8_pieces(x);
                #pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int r = qg - static_cast<int>(j8) + e;
                    if (r < p.Nq) {
                        // streaming stores: O is written once, keep L2 for K/V
                        uint4 *dst = reinterpret_cast<uint4 *>(p.O + (static_cast<size_t>(item.bh) * p.Nq + r) * D + 64 * c + 8 * j8);
                        __stcs(dst, make_uint4(x[4 * e], x[4 * e + 1], x[4 * e + 2], x[4 * e + 3]));
                    }
                }
            }
            if (live) p.LSE[static_cast<size_t>(item.bh) * p.Nq + qg] = lse;
        }
        ptx::tc_fence_before_sync();
    }
}

// ------------------------------------------------------------------- kernel

template <int D, int MODE>
__global__ void __launch_bounds__(Config<D>::kThreads, Config<D>::kCtasPerSm)
    fa_fwd_kernel(const __grid_constant__ FwdParams p) {
    using C = Config<D, (MODE & kFp8) != 0>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte-swizzled operand tiles.
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t smem_q = base;
    const uint32_t smem_ring = base + C::kQBytes;
    const uint32_t bars = base + C::kBarOffset;
    // barrier block: 11 fixed barriers, 2 * kSlots ring barriers, then the
    // TMEM address holder and the abort flag
    constexpr int kHolder = 88 + 16 * C::kSlots;
    static_assert(kHolder + 8 <= 256, "barrier block overflows its 256 bytes");
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(base_ptr + C::kBarOffset + kHolder);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base_ptr + C::kBarOffset + kHolder + 4);

    Shared sh;
    sh.q_full = bars + 0;
    sh.q_empty = bars + 8;
    sh.s_full0 = bars + 16;       // 2 barriers
    sh.p_full0 = bars + 32;       // 2
    sh.o_full0 = bars + 48;       // 2
    sh.done = bars + 64;
    sh.s_alt = bars + 72;
    sh.pv_done = bars + 80;
    sh.kv_full0 = bars + 88;      // kSlots
    sh.kv_empty0 = bars + 88 + 8 * C::kSlots;
    sh.abort_flag = abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        ptx::mbar_init(sh.q_full, 1);
        ptx::mbar_init(sh.q_empty, 1);
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(sh.s_full0 + 8 * t, 1);
            ptx::mbar_init(sh.p_full0 + 8 * t, 128);
            ptx::mbar_init(sh.o_full0 + 8 * t, 1);
        }
        ptx::mbar_init(sh.done, 1);
        ptx::mbar_init(sh.s_alt, 1);
        ptx::mbar_init(sh.pv_done, 1);
        for (int s = 0; s < C::kSlots; ++s) {
            ptx::mbar_init(sh.kv_full0 + 8 * s, 1);
            ptx::mbar_init(sh.kv_empty0 + 8 * s, 1);
        }
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == kProducerWarp && lane == 0) {
        ptx::prefetch_tensormap(&p.tmQ);
        ptx::prefetch_tensormap(&p.tmK);
        ptx::prefetch_tensormap(&p.tmV);
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_holder), C::kTmemCols);
        ptx::tmem_relinquish_alloc_permit();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_holder;
    // The launch lets this grid start while the previous kernel of the stream
    // drains (programmatic dependent launch).  Nothing above touched global
    // memory; below, every access comes after the previous kernel completed:
    // one warp waits for it, the others at the barrier, where they issue
    // nothing.  The grid does not release its own dependents early (a
    // dependent grid resident beside this one's last CTAs slowed them).
    if (threadIdx.x < 32) ptx::griddep_wait();
    __syncthreads();

    uint32_t loads_issued = 0, q_arms = 0;
    if (warp < kSoftmaxWarps) {
        if constexpr (C::kRegSplit) ptx::setmaxnreg_inc<kSoftmaxRegs>();
        softmax_role<D, MODE>(p, sh, tmem, warp >> 2, warp & 3, lane);
    } else if (warp == kProducerWarp) {
        if constexpr (C::kRegSplit) ptx::setmaxnreg_dec<kOtherRegs>();
        if constexpr ((MODE & kPaged) != 0)
            producer_role_paged<D, MODE>(p, sh, smem_q, smem_ring, loads_issued, q_arms, lane);
        if (lane == 0) {
            if constexpr ((MODE & kPaged) == 0)
                producer_role<D, MODE>(p, sh, smem_q, smem_ring, loads_issued, q_arms);
            // Drain: every copy this CTA started must land before it exits.
            const uint32_t first = loads_issued > (uint32_t)C::kSlots ? loads_issued - C::kSlots : 0u;
            for (uint32_t x = first; x < loads_issued; ++x)
                if (!C::kPairedSlots || (x & 1u) == 0)   // paired: one barrier per K/V pair
                    wait_drain(sh.kv_full0 + 8 * (x % C::kSlots), (x / C::kSlots) & 1);
            if (q_arms > 0) wait_drain(sh.q_full, (q_arms - 1) & 1);
        }
        __syncwarp();
    } else {
        if constexpr (C::kRegSplit) ptx::setmaxnreg_dec<kOtherRegs>();
        // the whole warp, converged: uniform descriptor arithmetic; lane 0 issues
        if (warp == kMmaWarp) mma_role<D, MODE>(p, sh, tmem, smem_q, smem_ring);
        __syncwarp();
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        if (lane == 0) {
            // All MMAs this thread issued must finish before TMEM is released.
            ptx::mma_commit(sh.done);
            wait_drain(sh.done, 0);
        }
        __syncwarp();
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ---------------------------------------------------------- split-KV merge
//
// Combines the kv_splits partial results of each query row with the
// online-softmax merge of "6. FlashAttention 分块逻辑" sections 11.3 and 13.2:
// with partial outputs O_s (already divided by their own sums) and
// LSE_s = m_s + ln l_s, the merged row is
//   m = max_s LSE_s,  w_s = exp(LSE_s - m),  O = sum_s w_s O_s / sum_s w_s,
//   LSE = m + ln sum_s w_s.
// One warp per row; lane c holds columns c, c+32, ...  Empty partials
// (LSE_s = -inf) carry no weight and are not read.
template <int D>
__global__ void __launch_bounds__(256) fa_merge_kernel(const float *__restrict__ O_part,
                                                       const float *__restrict__ LSE_part,
                                                       __nv_bfloat16 *__restrict__ O, float *__restrict__ LSE,
                                                       long long rows, int splits) {
    const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    float m = -INFINITY;
    for (int s = 0; s < splits; ++s) m = fmaxf(m, LSE_part[s * rows + row]);
    float acc[D / 32];
    #pragma unroll
    for (int c = 0; c < D / 32; ++c) acc[c] = 0.f;
    float wsum = 0.f;
    for (int s = 0; s < splits; ++s) {
        const float lse = LSE_part[s * rows + row];
        if (lse == -INFINITY) continue;
        const float w = expf(lse - m);
        wsum += w;
        const float *src = O_part + (s * rows + row) * D;
        #pragma unroll
        for (int c = 0; c < D / 32; ++c) acc[c] = fmaf(w, src[lane + 32 * c], acc[c]);
    }
    // a row no slice saw a key of (possible only with the paged cache): O = 0, LSE = -inf
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    __nv_bfloat16 *dst = O + row * D;
    #pragma unroll
    for (int c = 0; c < D / 32; ++c) dst[lane + 32 * c] = __float2bfloat16_rn(acc[c] * inv);
    if (lane == 0) LSE[row] = m + logf(wsum);
}

}  // namespace fa
