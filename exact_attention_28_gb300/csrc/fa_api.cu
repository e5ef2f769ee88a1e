// Host side of libfa_gb300.so: argument validation, TMA tensor maps, the
// persistent schedule, and the launch.  Implements the C ABI of include/fa.h.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "fa_bwd_kernel.cuh"
#include "fa_fp8_quant.cuh"
#include "fa_fwd_kernel.cuh"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// so the library needs no link-time dependency on libcuda.
EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Every map of this library: 128-byte swizzle, 256-byte L2 promotion, no
// interleave, zero fill, unit element strides.  Encoded maps are kept in a
// small per-thread cache keyed by everything that goes into the encoding
// (element type, rank, address, sizes, strides, box), so a repeated call on
// the same buffers and shapes skips the driver call; a hit returns exactly the
// map the driver would encode again, whatever else changed in between.
bool encode_cached(CUtensorMap *map, CUtensorMapDataType type, int rank, const void *ptr, const cuuint64_t *dims,
                   const cuuint64_t *strides, const cuuint32_t *box) {
    struct Entry {
        bool used;
        CUtensorMapDataType type;
        int rank;
        const void *ptr;
        cuuint64_t dims[4], strides[3];
        cuuint32_t box[4];
        CUtensorMap map;
    };
    constexpr int kEntries = 32;
    thread_local Entry cache[kEntries] = {};
    thread_local int next = 0;
    for (Entry &e : cache) {
        if (!e.used || e.type != type || e.rank != rank || e.ptr != ptr) continue;
        bool same = true;
        for (int i = 0; i < rank; ++i) same = same && e.dims[i] == dims[i] && e.box[i] == box[i];
        for (int i = 0; i + 1 < rank; ++i) same = same && e.strides[i] == strides[i];
        if (same) {
            *map = e.map;
            return true;
        }
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (fn(map, type, static_cast<cuuint32_t>(rank), const_cast<void *>(ptr), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    Entry &e = cache[next];
    next = (next + 1) % kEntries;
    e = Entry{};
    e.used = true;
    e.type = type;
    e.rank = rank;
    e.ptr = ptr;
    for (int i = 0; i < rank; ++i) {
        e.dims[i] = dims[i];
        e.box[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i) e.strides[i] = strides[i];
    e.map = *map;
    return true;
}

// [BH][N][d] bf16, boxes of 64 columns x box_rows rows x 1 head, 128-byte
// swizzle.  Rows past N inside a head read as zero (the map is 3-D, so a box
// never spills into the next head).
bool make_map(CUtensorMap *map, const void *ptr, int64_t BH, int64_t N, int d, int box_rows = fa::kBR) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
    return encode_cached(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box);
}

// Paged cache [num_blocks][H][block_size][d] bf16, boxes of 64 columns x
// min(block_size, keys per K/V tile) rows of one head of one block, 128-byte
// swizzle.
bool make_map_paged(CUtensorMap *map, const void *ptr, int num_blocks, int H, int block_size, int d) {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(block_size),
                                static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(block_size) * d * 2,
                                   static_cast<cuuint64_t>(H) * block_size * d * 2};
    const int bc = fa::kv_tile_keys(d);
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(block_size < bc ? block_size : bc), 1, 1};
    return encode_cached(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, ptr, dims, strides, box);
}

// 8-bit [BH][rows][inner] (inner bytes per row, a multiple of 16), boxes of
// 128 bytes x box_rows rows x 1 head, 128-byte swizzle: E4M3 Q and K
// ([BH][N][128], box 128 x 128) and V^T ([BH][128][ldn], box 128 keys x 128
// channels).
bool make_map_u8(CUtensorMap *map, const void *ptr, int64_t BH, int64_t rows, int64_t inner, int box_rows) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows) * inner};
    const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(box_rows), 1};
    return encode_cached(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, ptr, dims, strides, box);
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

fa_status validate(const void *Q, const void *K, const void *V, const void *O, const float *LSE, int B,
                   int H, int Nq, int Nk, int d, float scale) {
    if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    // B*H heads and B*H*N*d elements must fit the kernel's index arithmetic
    // (int heads and tiles, 64-bit element offsets) and the TMA map (< 2^32
    // per dimension, strides < 2^40 bytes).
    const int64_t BH = static_cast<int64_t>(B) * H;
    if (BH > (int64_t{1} << 30)) return FA_ERR_INVALID_ARG;
    const int64_t tiles = BH * ((static_cast<int64_t>(Nq) + 255) / 256) * 2;
    if (tiles > (int64_t{1} << 30)) return FA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(Nq > Nk ? Nq : Nk) * d * 2 >= (int64_t{1} << 40)) return FA_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(LSE, 4))
        return FA_ERR_MISALIGNED;
    return FA_OK;
}

// The work list: per head, P = ceil(Tr/2) Q-tile pairs; all pairs of all
// heads are whole items except the last n_split (the lightest), which are
// split into single-tile items so the last round of the persistent grid is
// evenly filled.  Only pairs holding two tiles are split.
void plan_schedule(fa::FwdParams &p, int grid_ctas) {
    const int64_t BH = p.BH;
    const int64_t NP = BH * p.P;
    const int64_t units = BH * p.Tr;                        // Q tiles in total
    const int64_t two_tile_pairs = BH * (p.Tr / 2);         // pairs with both tiles present
    int64_t keep = static_cast<int64_t>(grid_ctas) * (units / (2 * static_cast<int64_t>(grid_ctas)));
    if (keep > NP) keep = NP;
    int64_t split = NP - keep;
    if (split > two_tile_pairs) split = two_tile_pairs;
    p.n_pair_items = static_cast<int>(NP - split);
    p.n_items = static_cast<int>(NP + split);
}

// Heads per group of the item order.  Non-causal items all cost the same,
// so heads are grouped to keep their K and V within 48 MB (well inside the
// 126 MB L2, leaving room for the streamed Q and O).  Causal items differ in
// cost; one group over all heads keeps the list heaviest-first, which the
// snake assignment needs to balance the CTAs.
int heads_per_group(int64_t BH, int64_t Nk, int d, int causal) {
    if (causal) return static_cast<int>(BH);
    const int64_t kv_bytes = Nk * d * 2 * 2;
    int64_t hg = (int64_t{48} << 20) / (kv_bytes > 0 ? kv_bytes : 1);
    if (hg < 1) hg = 1;
    if (hg > BH) hg = BH;
    return static_cast<int>(hg);
}

// Persistent CTAs per SM of the forward for head dimension d.
int ctas_per_sm(int d) { return d == 64 ? fa::Config<64>::kCtasPerSm : fa::Config<128>::kCtasPerSm; }

// Shapes, scale and schedule of one call (everything but pointers and maps);
// returns the grid size (at most ctas_per_sm(d) CTAs per SM).  kv_splits > 1
// cuts every item's key range into that many slices, each a work item of its
// own.
int setup_params(fa::FwdParams &p, int B, int H, int Nq, int Nk, int d, float scale, int causal, int sms,
                 int kv_splits = 1) {
    std::memset(&p, 0, sizeof p);
    const int64_t BH = static_cast<int64_t>(B) * H;
    p.BH = static_cast<int>(BH);
    p.Nq = Nq;
    p.Nk = Nk;
    p.Tr = (Nq + fa::kBR - 1) / fa::kBR;
    p.bc = fa::kv_tile_keys(d);
    p.Tc = (Nk + p.bc - 1) / p.bc;
    p.P = (p.Tr + 1) / 2;
    p.causal = causal != 0;
    // c2 = scale * log2(e).  A zero scale is run as the smallest normal float:
    // every score then changes by at most |S| * 2^-126, far below fp32
    // resolution of the outputs, and masked keys keep an exact p = 0.
    double c2 = static_cast<double>(scale) * 1.4426950408889634;
    if (scale == 0.0f) c2 = 1.1754943508222875e-38 * 1.4426950408889634;
    p.c2 = static_cast<float>(c2);
    p.heads_per_group = heads_per_group(BH, Nk, d, causal);
    p.kv_splits = kv_splits > 1 ? kv_splits : 1;
    p.drop_load_item = -1;
    // the decode's invariant divisors (all >= 1; every dividend is < 2^31)
    const int64_t groups = (BH + p.heads_per_group - 1) / p.heads_per_group;
    p.fd_splits = fa::make_fastdiv(static_cast<uint32_t>(p.kv_splits));
    p.fd_per_group = fa::make_fastdiv(static_cast<uint32_t>(p.heads_per_group) * static_cast<uint32_t>(p.P));
    p.fd_hg = fa::make_fastdiv(static_cast<uint32_t>(p.heads_per_group));
    p.fd_last_gsize = fa::make_fastdiv(static_cast<uint32_t>(BH - (groups - 1) * p.heads_per_group));
    p.fd_bh = fa::make_fastdiv(static_cast<uint32_t>(BH));
    p.fd_2bh = fa::make_fastdiv(static_cast<uint32_t>(2 * BH));
    p.H = H;
    p.fd_h = fa::make_fastdiv(static_cast<uint32_t>(H));
    p.bc_shift = p.bc == 64 ? 6 : 7;
    p.block_shift = 0;
    if (p.kv_splits > 1) {
        const int64_t NP = static_cast<int64_t>(p.BH) * p.P;
        p.n_pair_items = static_cast<int>(NP);
        p.n_items = static_cast<int>(NP * p.kv_splits);
    } else {
        plan_schedule(p, ctas_per_sm(d) * sms);
    }
    const int ctas = ctas_per_sm(d) * sms;
    return p.n_items < ctas ? p.n_items : ctas;
}

// Key-range slices for the split path.  Splitting costs a partial write, a
// merge and a re-read per slice, so it pays only when the unsplit work list
// leaves most SMs idle (at most half of them busy); then as many slices as
// keep all items in one round (items <= SMs: a second, partial round would
// double the time), never more slices than K/V tiles, at most 64.
int choose_splits(int64_t BH, int Nq, int Nk, int d, int sms) {
    const int64_t ctas = static_cast<int64_t>(ctas_per_sm(d)) * sms;
    const int64_t pairs = BH * ((Nq + 2 * fa::kBR - 1) / (2 * fa::kBR));
    if (2 * pairs > ctas) return 1;
    const int bc = fa::kv_tile_keys(d);
    const int64_t tc = (Nk + bc - 1) / bc;
    int64_t s = ctas / pairs;
    if (s > tc) s = tc;
    if (s > 64) s = 64;
    return s < 1 ? 1 : static_cast<int>(s);
}

// Workspace of the split path: [splits][BH][Nq][d] fp32 partial outputs, then
// [splits][BH][Nq] fp32 partial LSE at a 256-byte boundary.
size_t splitkv_o_bytes(int64_t BH, int Nq, int d, int splits) {
    return ((static_cast<size_t>(splits) * BH * Nq * d * 4) + 255) & ~static_cast<size_t>(255);
}
size_t splitkv_bytes(int64_t BH, int Nq, int d, int splits) {
    return splitkv_o_bytes(BH, Nq, d, splits) + static_cast<size_t>(splits) * BH * Nq * 4;
}

struct DeviceInfo {
    int sms = 0;
    bool attr[2][4] = {};   // forward kernel [d == 128][mode] has its shared-memory limit set
    bool attr_fp8 = false;  // the E4M3 forward (d = 128)
    bool bwd_attr64 = false, bwd_attr128 = false;
};
std::mutex g_dev_mu;
DeviceInfo g_dev[64];

template <int D, int MODE>
fa_status launch(const fa::FwdParams &p, int grid, cudaStream_t stream, bool &attr_done) {
    using C = fa::Config<D, (MODE & fa::kFp8) != 0>;
    if (!attr_done) {
        // the whole shared memory as carveout, so that kCtasPerSm CTAs fit an SM
        if (cudaFuncSetAttribute(fa::fa_fwd_kernel<D, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(fa::fa_fwd_kernel<D, MODE>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 100) != cudaSuccess)
            return FA_ERR_CUDA;
        attr_done = true;
    }
    // Programmatic stream serialisation: the CTAs may be launched and set up
    // (barriers, tensor memory) while the previous kernel of the stream
    // drains; the kernel waits for it before its first global access.
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, fa::fa_fwd_kernel<D, MODE>, p) != cudaSuccess) return FA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Launches the forward variant for head dimension d and the given mode.
// Caller holds g_dev_mu (attr points into g_dev).
template <int MODE>
fa_status launch_mode(const fa::FwdParams &p, int d, int grid, cudaStream_t stream, bool (&attr)[2][4]) {
    return d == 64 ? launch<64, MODE>(p, grid, stream, attr[0][MODE])
                   : launch<128, MODE>(p, grid, stream, attr[1][MODE]);
}

}  // namespace

namespace {

fa_status device_info(int &sms, DeviceInfo *&out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo &info = g_dev[dev];
    if (info.sms == 0 && cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return FA_ERR_CUDA;
    sms = info.sms;
    out = &info;
    return FA_OK;
}

// Encodes the maps and launches the attention kernel (partials when
// kv_splits > 1, into O_part / LSE_part).
fa_status run_forward(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H, int Nq,
                      int Nk, int d, float scale, int causal, int kv_splits, float *O_part, float *LSE_part,
                      cudaStream_t stream, int drop_load_item = -1) {
    int sms;
    DeviceInfo *info;
    fa_status st = device_info(sms, info);
    if (st != FA_OK) return st;
    fa::FwdParams p;
    const int grid = setup_params(p, B, H, Nq, Nk, d, scale, causal, sms, kv_splits);
    const int64_t BH = static_cast<int64_t>(B) * H;
    if (!make_map(&p.tmQ, Q, BH, Nq, d) || !make_map(&p.tmK, K, BH, Nk, d, p.bc) ||
        !make_map(&p.tmV, V, BH, Nk, d, p.bc))
        return FA_ERR_CUDA;
    p.O = static_cast<__nv_bfloat16 *>(O);
    p.LSE = LSE;
    p.O_part = O_part;
    p.LSE_part = LSE_part;
    p.drop_load_item = drop_load_item;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    return kv_splits > 1 ? launch_mode<fa::kSplit>(p, d, grid, stream, info->attr)
                         : launch_mode<fa::kDense>(p, d, grid, stream, info->attr);
}

fa_status run_merge(const float *O_part, const float *LSE_part, void *O, float *LSE, int64_t rows, int d, int splits,
                    cudaStream_t stream) {
    const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
    if (d == 64)
        fa::fa_merge_kernel<64><<<blocks, 256, 0, stream>>>(O_part, LSE_part, static_cast<__nv_bfloat16 *>(O), LSE,
                                                           rows, splits);
    else
        fa::fa_merge_kernel<128><<<blocks, 256, 0, stream>>>(O_part, LSE_part, static_cast<__nv_bfloat16 *>(O), LSE,
                                                            rows, splits);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" fa_status fa_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                            int Nq, int Nk, int d, float scale, int causal, fa_stream_t stream) {
    fa_status st = validate(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale);
    if (st != FA_OK) return st;
    return run_forward(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale, causal, 1, nullptr, nullptr,
                       reinterpret_cast<cudaStream_t>(stream));
}

// The forward with one K tile deliberately left unloaded: exercises the
// bounded waits and the clean shutdown of the kernel (see the header).
extern "C" fa_status fa_fwd_test_missing_load(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                                              int H, int Nq, int Nk, int d, float scale, int causal, int item,
                                              fa_stream_t stream) {
    fa_status st = validate(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale);
    if (st != FA_OK) return st;
    if (item < 0) return FA_ERR_INVALID_ARG;
    return run_forward(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale, causal, 1, nullptr, nullptr,
                       reinterpret_cast<cudaStream_t>(stream), item);
}

namespace {

// Arguments of the paged entry points (before anything is enqueued).
fa_status validate_paged(const void *Q, const void *K_cache, const void *V_cache, const int *block_table,
                         const int *seq_lens, const void *O, const float *LSE, int B, int H, int Nq, int max_blocks,
                         int num_blocks, int block_size, int d, float scale) {
    if (!block_table || !seq_lens) return FA_ERR_INVALID_ARG;
    if (max_blocks < 1 || num_blocks < 1) return FA_ERR_INVALID_ARG;
    if (block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128 && block_size != 256)
        return FA_ERR_UNSUPPORTED;
    const int64_t cap = static_cast<int64_t>(max_blocks) * block_size;
    if (cap > (int64_t{1} << 30) || static_cast<int64_t>(num_blocks) * H * block_size * d * 2 >= (int64_t{1} << 40))
        return FA_ERR_INVALID_ARG;
    fa_status st = validate(Q, K_cache, V_cache, O, LSE, B, H, Nq, static_cast<int>(cap), d, scale);
    if (st != FA_OK) return st;
    if (!aligned(block_table, 4) || !aligned(seq_lens, 4)) return FA_ERR_MISALIGNED;
    return FA_OK;
}

// Encodes the maps and launches the paged kernel (partials when kv_splits > 1).
fa_status run_paged(const void *Q, const void *K_cache, const void *V_cache, const int *block_table,
                    const int *seq_lens, void *O, float *LSE, int B, int H, int Nq, int max_blocks, int num_blocks,
                    int block_size, int d, float scale, int causal, int kv_splits, float *O_part, float *LSE_part,
                    cudaStream_t stream) {
    const int64_t cap = static_cast<int64_t>(max_blocks) * block_size;
    int sms;
    DeviceInfo *info;
    fa_status st = device_info(sms, info);
    if (st != FA_OK) return st;
    fa::FwdParams p;
    const int grid = setup_params(p, B, H, Nq, static_cast<int>(cap), d, scale, causal, sms, kv_splits);
    const int64_t BH = static_cast<int64_t>(B) * H;
    if (!make_map(&p.tmQ, Q, BH, Nq, d) || !make_map_paged(&p.tmK, K_cache, num_blocks, H, block_size, d) ||
        !make_map_paged(&p.tmV, V_cache, num_blocks, H, block_size, d))
        return FA_ERR_CUDA;
    p.O = static_cast<__nv_bfloat16 *>(O);
    p.LSE = LSE;
    p.O_part = O_part;
    p.LSE_part = LSE_part;
    p.H = H;
    p.block_size = block_size;
    p.block_shift = 31 - __builtin_clz(static_cast<unsigned>(block_size));   // a power of two, 16..256
    p.max_blocks = max_blocks;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    return kv_splits > 1 ? launch_mode<fa::kPagedSplit>(p, d, grid, stream, info->attr)
                         : launch_mode<fa::kPaged>(p, d, grid, stream, info->attr);
}

}  // namespace

extern "C" fa_status fa_fwd_paged(const void *Q, const void *K_cache, const void *V_cache, const int *block_table,
                                  const int *seq_lens, void *O, float *LSE, int B, int H, int Nq, int max_blocks,
                                  int num_blocks, int block_size, int d, float scale, int causal,
                                  fa_stream_t stream) {
    fa_status st = validate_paged(Q, K_cache, V_cache, block_table, seq_lens, O, LSE, B, H, Nq, max_blocks,
                                  num_blocks, block_size, d, scale);
    if (st != FA_OK) return st;
    return run_paged(Q, K_cache, V_cache, block_table, seq_lens, O, LSE, B, H, Nq, max_blocks, num_blocks,
                     block_size, d, scale, causal, 1, nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" fa_status fa_splitkv_workspace(int B, int H, int Nq, int Nk, int d, int causal, int *num_splits,
                                          size_t *bytes) {
    (void)causal;
    if (!num_splits || !bytes || *num_splits < 0) return FA_ERR_INVALID_ARG;
    char dummy[16] __attribute__((aligned(16)));
    fa_status st = validate(dummy, dummy, dummy, dummy, reinterpret_cast<float *>(dummy), B, H, Nq, Nk, d, 1.0f);
    if (st != FA_OK) return st;
    const int64_t BH = static_cast<int64_t>(B) * H;
    if (*num_splits == 0) {
        int sms;
        DeviceInfo *info;
        st = device_info(sms, info);
        if (st != FA_OK) return st;
        *num_splits = choose_splits(BH, Nq, Nk, d, sms);
    }
    if (*num_splits > 256) return FA_ERR_INVALID_ARG;
    *bytes = splitkv_bytes(BH, Nq, d, *num_splits);
    return FA_OK;
}

extern "C" fa_status fa_fwd_splitkv(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                                    int Nq, int Nk, int d, float scale, int causal, int num_splits,
                                    void *workspace, size_t workspace_bytes, fa_stream_t stream) {
    fa_status st = validate(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale);
    if (st != FA_OK) return st;
    if (num_splits < 1 || num_splits > 256 || !workspace) return FA_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return FA_ERR_MISALIGNED;
    const int64_t BH = static_cast<int64_t>(B) * H;
    if (workspace_bytes < splitkv_bytes(BH, Nq, d, num_splits)) return FA_ERR_INVALID_ARG;
    float *O_part = static_cast<float *>(workspace);
    float *LSE_part = reinterpret_cast<float *>(static_cast<char *>(workspace) + splitkv_o_bytes(BH, Nq, d, num_splits));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (num_splits == 1)   // one slice: the plain forward writes O and LSE itself
        return run_forward(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale, causal, 1, nullptr, nullptr, s);
    st = run_forward(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale, causal, num_splits, O_part, LSE_part, s);
    if (st != FA_OK) return st;
    return run_merge(O_part, LSE_part, O, LSE, BH * Nq, d, num_splits, s);
}

extern "C" fa_status fa_fwd_paged_splitkv(const void *Q, const void *K_cache, const void *V_cache,
                                          const int *block_table, const int *seq_lens, void *O, float *LSE, int B,
                                          int H, int Nq, int max_blocks, int num_blocks, int block_size, int d,
                                          float scale, int causal, int num_splits, void *workspace,
                                          size_t workspace_bytes, fa_stream_t stream) {
    fa_status st = validate_paged(Q, K_cache, V_cache, block_table, seq_lens, O, LSE, B, H, Nq, max_blocks,
                                  num_blocks, block_size, d, scale);
    if (st != FA_OK) return st;
    if (num_splits < 1 || num_splits > 256 || !workspace) return FA_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return FA_ERR_MISALIGNED;
    const int64_t BH = static_cast<int64_t>(B) * H;
    if (workspace_bytes < splitkv_bytes(BH, Nq, d, num_splits)) return FA_ERR_INVALID_ARG;
    float *O_part = static_cast<float *>(workspace);
    float *LSE_part = reinterpret_cast<float *>(static_cast<char *>(workspace) + splitkv_o_bytes(BH, Nq, d, num_splits));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (num_splits == 1)
        return run_paged(Q, K_cache, V_cache, block_table, seq_lens, O, LSE, B, H, Nq, max_blocks, num_blocks,
                         block_size, d, scale, causal, 1, nullptr, nullptr, s);
    st = run_paged(Q, K_cache, V_cache, block_table, seq_lens, O, LSE, B, H, Nq, max_blocks, num_blocks, block_size,
                   d, scale, causal, num_splits, O_part, LSE_part, s);
    if (st != FA_OK) return st;
    return run_merge(O_part, LSE_part, O, LSE, BH * Nq, d, num_splits, s);
}

// ------------------------------------------------------------------- E4M3

extern "C" fa_status fa_fwd_fp8(const void *Q8, const void *K8, const void *Vt8, const float *descale_q,
                                const float *descale_k, const float *descale_v, void *O, float *LSE, int B, int H,
                                int Nq, int Nk, int d, float scale, int causal, fa_stream_t stream) {
    fa_status st = validate(Q8, K8, Vt8, O, LSE, B, H, Nq, Nk, d, scale);
    if (st != FA_OK) return st;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    if (!descale_q || !descale_k || !descale_v) return FA_ERR_INVALID_ARG;
    if (!aligned(descale_q, 4) || !aligned(descale_k, 4) || !aligned(descale_v, 4)) return FA_ERR_MISALIGNED;
    int sms;
    DeviceInfo *info;
    st = device_info(sms, info);
    if (st != FA_OK) return st;
    fa::FwdParams p;
    const int grid = setup_params(p, B, H, Nq, Nk, d, scale, causal, sms, 1);
    const int64_t BH = static_cast<int64_t>(B) * H;
    const int64_t ldn = (static_cast<int64_t>(Nk) + 15) / 16 * 16;
    if (!make_map_u8(&p.tmQ, Q8, BH, Nq, d, fa::kBR) || !make_map_u8(&p.tmK, K8, BH, Nk, d, fa::kBC) ||
        !make_map_u8(&p.tmV, Vt8, BH, d, ldn, d))
        return FA_ERR_CUDA;
    p.O = static_cast<__nv_bfloat16 *>(O);
    p.LSE = LSE;
    p.descale_q = descale_q;
    p.descale_k = descale_k;
    p.descale_v = descale_v;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    return launch<128, fa::kFp8>(p, grid, reinterpret_cast<cudaStream_t>(stream), info->attr_fp8);
}

extern "C" fa_status fa_quantize_fp8(const void *X, void *X8, float *descale, int B, int H, int N, int d,
                                     const float *signs, int transpose, fa_stream_t stream) {
    if (!X || !X8 || !descale) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    const int64_t BH = static_cast<int64_t>(B) * H;
    const int64_t blocks = (static_cast<int64_t>(N) + fa::kQuantRows - 1) / fa::kQuantRows;
    if (BH > (int64_t{1} << 30) || blocks > 65535) return FA_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(X8, 16) || !aligned(descale, 4) || (signs && !aligned(signs, 4)))
        return FA_ERR_MISALIGNED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int ldn = (N + 15) / 16 * 16;
    const dim3 grid(static_cast<unsigned>(BH), static_cast<unsigned>(blocks));
    const __nv_bfloat16 *x = static_cast<const __nv_bfloat16 *>(X);
    uint8_t *x8 = static_cast<uint8_t *>(X8);
    unsigned *amax = reinterpret_cast<unsigned *>(descale);
    if (cudaMemsetAsync(descale, 0, static_cast<size_t>(BH) * 4, s) != cudaSuccess) return FA_ERR_CUDA;
    if (d == 64) {
        fa::fa_amax_kernel<64><<<grid, fa::kQuantThreads, 0, s>>>(x, signs, amax, N);
        if (transpose) fa::fa_quant_kernel<64, true><<<grid, fa::kQuantThreads, 0, s>>>(x, signs, amax, x8, N, ldn);
        else fa::fa_quant_kernel<64, false><<<grid, fa::kQuantThreads, 0, s>>>(x, signs, amax, x8, N, ldn);
    } else {
        fa::fa_amax_kernel<128><<<grid, fa::kQuantThreads, 0, s>>>(x, signs, amax, N);
        if (transpose) fa::fa_quant_kernel<128, true><<<grid, fa::kQuantThreads, 0, s>>>(x, signs, amax, x8, N, ldn);
        else fa::fa_quant_kernel<128, false><<<grid, fa::kQuantThreads, 0, s>>>(x, signs, amax, x8, N, ldn);
    }
    const float rs = signs ? static_cast<float>(1.0 / std::sqrt(static_cast<double>(d))) : 1.0f;
    fa::fa_descale_kernel<<<static_cast<unsigned>((BH + 255) / 256), 256, 0, s>>>(descale, static_cast<int>(BH), rs);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

extern "C" fa_status fa_schedule(int B, int H, int Nq, int Nk, int d, int causal, int num_sms, int num_splits,
                                 int32_t *items, int64_t capacity, int64_t *n_items) {
    if (!n_items || num_sms < 1 || num_splits < 1 || num_splits > 256) return FA_ERR_INVALID_ARG;
    const float scale = 1.0f;
    char dummy[16] __attribute__((aligned(16)));
    fa_status st = validate(dummy, dummy, dummy, dummy, reinterpret_cast<float *>(dummy), B, H, Nq, Nk, d, scale);
    if (st != FA_OK) return st;
    fa::FwdParams p;
    const int grid = setup_params(p, B, H, Nq, Nk, d, scale, causal, num_sms, num_splits);
    *n_items = p.n_items;
    if (!items) return FA_OK;
    if (capacity < p.n_items) return FA_ERR_INVALID_ARG;
    int64_t n = 0;
    for (int b = 0; b < grid; ++b) {
        for (int k = 0;; ++k) {
            const int w = fa::item_of_round(p, k, b, grid);
            if (w < 0) break;
            const fa::Item it = fa::decode_item(p, w, p.kv_splits > 1);
            int32_t *out = items + 8 * n++;
            out[0] = b; out[1] = k; out[2] = it.bh; out[3] = it.q0; out[4] = it.kv0;
            out[5] = it.nk[0]; out[6] = it.ntiles > 1 ? it.nk[1] : -1; out[7] = it.split;
        }
    }
    return n == p.n_items ? FA_OK : FA_ERR_INVALID_ARG;
}

// ------------------------------------------------------------ host buffers
//
// fa_fwd_host moves the inputs in and the outputs out around the forward.  A
// large call is cut into up to kHostChunksMax groups of heads that flow
// through three internal streams (copy in, compute, copy out): while group c
// is being computed, group c+1 is copied in and group c-1 is copied out, so
// the two copy directions and the tensor cores work at the same time.  The streams and events are created
// once per device and shared by all calls (enqueueing is serialised).

namespace {

constexpr int kHostChunksMax = 8;
constexpr size_t kHostChunkMinBytes = size_t{8} << 20;   // input bytes per group, at least

struct HostPipe {
    bool ready = false;
    cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t in_done[kHostChunksMax] = {}, out_ready[kHostChunksMax] = {};
};
HostPipe g_pipe[64];
std::mutex g_pipe_mu;   // held while a call enqueues (the streams and events are shared)

// The current device's streams and events (created on first use).  Caller
// holds g_pipe_mu.
fa_status host_pipe(HostPipe *&out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FA_ERR_CUDA;
    HostPipe &hp = g_pipe[dev];
    if (!hp.ready) {
        bool ok = true;
        for (cudaStream_t *st : {&hp.h2d, &hp.comp, &hp.d2h})
            ok = ok && cudaStreamCreateWithFlags(st, cudaStreamNonBlocking) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&hp.end, cudaEventDisableTiming) == cudaSuccess;
        for (int c = 0; c < kHostChunksMax && ok; ++c)
            ok = cudaEventCreateWithFlags(&hp.in_done[c], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&hp.out_ready[c], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) return FA_ERR_CUDA;
        hp.ready = true;
    }
    out = &hp;
    return FA_OK;
}

// Number of head groups for a call: enough input bytes per group that each
// copy runs at full speed.  The host link (about 200 GB/s each way) is slower
// than the forward for every shape with at least one such group, so more
// groups mean more overlap even where a group fills only part of the GPU
// (measured on the 2 x 16 x 4096 x 128 forward: 3 groups 0.734 ms, 8 groups
// 0.684 ms per call).
int host_chunks(int64_t BH, int Nq, int Nk, int d, int sms) {
    (void)sms;
    const size_t in_bytes = static_cast<size_t>(BH) * (static_cast<size_t>(Nq) + 2 * static_cast<size_t>(Nk)) * d * 2;
    int64_t c = static_cast<int64_t>(in_bytes / kHostChunkMinBytes);
    c = std::min<int64_t>(c, kHostChunksMax);
    c = std::min<int64_t>(c, BH);
    return static_cast<int>(std::max<int64_t>(c, 1));
}

}  // namespace

extern "C" int fa_host_groups(int B, int H, int Nq, int Nk, int d, int num_sms) {
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || (d != 64 && d != 128) || num_sms < 1) return 0;
    return host_chunks(static_cast<int64_t>(B) * H, Nq, Nk, d, num_sms);
}

extern "C" fa_status fa_fwd_host(const void *hQ, const void *hK, const void *hV, void *hO, float *hLSE,
                                 void *dQ, void *dK, void *dV, void *dO, float *dLSE, int B, int H, int Nq,
                                 int Nk, int d, float scale, int causal, fa_stream_t stream) {
    if (!hQ || !hK || !hV || !hO || !hLSE) return FA_ERR_INVALID_ARG;
    fa_status st = validate(dQ, dK, dV, dO, dLSE, B, H, Nq, Nk, d, scale);
    if (st != FA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t BH = static_cast<int64_t>(B) * H;
    const size_t q_head = static_cast<size_t>(Nq) * d * 2, kv_head = static_cast<size_t>(Nk) * d * 2;
    const size_t lse_head = static_cast<size_t>(Nq) * 4;
    int sms;
    DeviceInfo *info;
    st = device_info(sms, info);
    if (st != FA_OK) return st;
    const int chunks = host_chunks(BH, Nq, Nk, d, sms);
    auto cp = [](void *dst, const void *src, size_t n, cudaMemcpyKind k, cudaStream_t on) {
        return cudaMemcpyAsync(dst, src, n, k, on) == cudaSuccess;
    };
    auto at = [](const void *base, size_t off) { return static_cast<const char *>(base) + off; };
    auto at_mut = [](void *base, size_t off) { return static_cast<char *>(base) + off; };
    if (chunks == 1) {
        if (!cp(dQ, hQ, BH * q_head, cudaMemcpyHostToDevice, s) || !cp(dK, hK, BH * kv_head, cudaMemcpyHostToDevice, s) ||
            !cp(dV, hV, BH * kv_head, cudaMemcpyHostToDevice, s))
            return FA_ERR_CUDA;
        st = fa_fwd(dQ, dK, dV, dO, dLSE, B, H, Nq, Nk, d, scale, causal, stream);
        if (st != FA_OK) return st;
        if (!cp(hO, dO, BH * q_head, cudaMemcpyDeviceToHost, s) || !cp(hLSE, dLSE, BH * lse_head, cudaMemcpyDeviceToHost, s))
            return FA_ERR_CUDA;
        return FA_OK;
    }

    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe *hp;
    st = host_pipe(hp);
    if (st != FA_OK) return st;
    // fork: the internal streams start after the caller's earlier work on `s`
    if (cudaEventRecord(hp->start, s) != cudaSuccess) return FA_ERR_CUDA;
    for (cudaStream_t x : {hp->h2d, hp->comp, hp->d2h})
        if (cudaStreamWaitEvent(x, hp->start, 0) != cudaSuccess) return FA_ERR_CUDA;
    bool ok = true;
    for (int c = 0; c < chunks && ok; ++c) {
        const int64_t h0 = BH * c / chunks, h1 = BH * (c + 1) / chunks;
        const size_t n = static_cast<size_t>(h1 - h0);
        // one copy stream: each group's inputs land as early as they can (two
        // streams shared the link between groups and delayed every compute;
        // measured on the 16K causal forward: 3.17 ms per call with two,
        // 2.45 ms with one)
        cudaStream_t in = hp->h2d;
        ok = cp(at_mut(dQ, h0 * q_head), at(hQ, h0 * q_head), n * q_head, cudaMemcpyHostToDevice, in) &&
             cp(at_mut(dK, h0 * kv_head), at(hK, h0 * kv_head), n * kv_head, cudaMemcpyHostToDevice, in) &&
             cp(at_mut(dV, h0 * kv_head), at(hV, h0 * kv_head), n * kv_head, cudaMemcpyHostToDevice, in) &&
             cudaEventRecord(hp->in_done[c], in) == cudaSuccess &&
             cudaStreamWaitEvent(hp->comp, hp->in_done[c], 0) == cudaSuccess;
        if (ok)   // the group's heads are a contiguous [1, n, N, d] block of each tensor
            ok = run_forward(at(dQ, h0 * q_head), at(dK, h0 * kv_head), at(dV, h0 * kv_head), at_mut(dO, h0 * q_head),
                             reinterpret_cast<float *>(at_mut(dLSE, h0 * lse_head)), 1, static_cast<int>(n), Nq, Nk,
                             d, scale, causal, 1, nullptr, nullptr, hp->comp) == FA_OK;
        ok = ok && cudaEventRecord(hp->out_ready[c], hp->comp) == cudaSuccess &&
             cudaStreamWaitEvent(hp->d2h, hp->out_ready[c], 0) == cudaSuccess &&
             cp(at_mut(hO, h0 * q_head), at(dO, h0 * q_head), n * q_head, cudaMemcpyDeviceToHost, hp->d2h) &&
             cp(at_mut(hLSE, h0 * lse_head), at(dLSE, h0 * lse_head), n * lse_head, cudaMemcpyDeviceToHost, hp->d2h);
    }
    if (!ok) {
        // leave nothing of this call running unordered with the caller's stream
        for (cudaStream_t x : {hp->h2d, hp->comp, hp->d2h}) cudaStreamSynchronize(x);
        return FA_ERR_CUDA;
    }
    // join: the last copy out follows every compute, and each compute its copies in
    if (cudaEventRecord(hp->end, hp->d2h) != cudaSuccess || cudaStreamWaitEvent(s, hp->end, 0) != cudaSuccess)
        return FA_ERR_CUDA;
    return FA_OK;
}

// ------------------------------------------------- split keys without allocating
//
// Some callers cannot allocate device memory where they call attention: serving
// loops with a latency budget that rules out the allocator (cudaMalloc may
// synchronise the device), frameworks whose allocator owns all memory up front,
// and plugins that an inference runtime hands only the tensors they read and
// write and forbids to allocate while they execute.  For them the
// split-key forward can put its partial results in a scratch area that lives in
// this file: a fixed array in device global memory, which every GPU that loads
// the library holds until the process exits.  Its host-side name is only a
// stand-in; the device address is looked up once per device.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t{16} << 20;   // 16 MiB on each GPU
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
void *g_noalloc_addr[64];   // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device (looked up on the
// first call on that device).
fa_status noalloc_scratch(void *&addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!g_noalloc_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return FA_ERR_CUDA;
        g_noalloc_addr[dev] = ptr;
    }
    addr = g_noalloc_addr[dev];
    return FA_OK;
}

}  // namespace

extern "C" fa_status fa_fwd_splitkv_noalloc(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                                            int H, int Nq, int Nk, int d, float scale, int causal, int num_splits,
                                            fa_stream_t stream) {
    fa_status st = validate(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale);
    if (st != FA_OK) return st;
    if (num_splits < 0 || num_splits > 256) return FA_ERR_INVALID_ARG;
    const int64_t BH = static_cast<int64_t>(B) * H;
    if (num_splits == 0) {
        int sms;
        DeviceInfo *info;
        st = device_info(sms, info);
        if (st != FA_OK) return st;
        num_splits = choose_splits(BH, Nq, Nk, d, sms);
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (num_splits == 1)   // one slice: no partials, no scratch
        return run_forward(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale, causal, 1, nullptr, nullptr, s);
    if (splitkv_bytes(BH, Nq, d, num_splits) > kNoAllocScratchBytes) return FA_ERR_TOO_LARGE;
    void *scratch = nullptr;
    st = noalloc_scratch(scratch);
    if (st != FA_OK) return st;
    // Nothing needs clearing: the forward writes every partial the merge reads.
    float *O_part = static_cast<float *>(scratch);
    float *LSE_part = reinterpret_cast<float *>(static_cast<char *>(scratch) + splitkv_o_bytes(BH, Nq, d, num_splits));
    st = run_forward(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale, causal, num_splits, O_part, LSE_part, s);
    if (st != FA_OK) return st;
    return run_merge(O_part, LSE_part, O, LSE, BH * Nq, d, num_splits, s);
}

// ------------------------------------------------------------------ backward

namespace {

template <int D>
fa_status launch_bwd(const fa::BwdParams &p, const void *O, const void *dO, float *Dsum, cudaStream_t stream,
                     bool &attr_done) {
    using C = fa::BwdConfig<D>;
    if (!attr_done) {
        if (cudaFuncSetAttribute(fa::fa_bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(fa::fa_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes) != cudaSuccess)
            return FA_ERR_CUDA;
        attr_done = true;
    }
    const long long rows = static_cast<long long>(p.BH) * p.Nq;
    fa::fa_bwd_dot_kernel<D><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(O), static_cast<const __nv_bfloat16 *>(dO), Dsum, rows);
    fa::fa_bwd_dkdv_kernel<D><<<static_cast<unsigned>(p.BH) * p.Tc, fa::kBwdThreads, C::kSmemBytes, stream>>>(p);
    fa::fa_bwd_dq_kernel<D><<<static_cast<unsigned>(p.BH) * p.Tr, fa::kBwdThreads, C::kSmemBytes, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" fa_status fa_bwd_workspace(int B, int H, int Nq, int Nk, int d, size_t *bytes) {
    if (!bytes) return FA_ERR_INVALID_ARG;
    char dummy[16] __attribute__((aligned(16)));
    fa_status st = validate(dummy, dummy, dummy, dummy, reinterpret_cast<float *>(dummy), B, H, Nq, Nk, d, 1.0f);
    if (st != FA_OK) return st;
    *bytes = static_cast<size_t>(B) * H * Nq * 4;
    return FA_OK;
}

extern "C" fa_status fa_bwd(const void *Q, const void *K, const void *V, const void *O, const float *LSE,
                            const void *dO, void *dQ, void *dK, void *dV, int B, int H, int Nq, int Nk, int d,
                            float scale, int causal, void *workspace, size_t workspace_bytes, fa_stream_t stream) {
    fa_status st = validate(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale);
    if (st != FA_OK) return st;
    if (!dO || !dQ || !dK || !dV || !workspace) return FA_ERR_INVALID_ARG;
    if (!aligned(dO, 16) || !aligned(dQ, 16) || !aligned(dK, 16) || !aligned(dV, 16) || !aligned(workspace, 16))
        return FA_ERR_MISALIGNED;
    const int64_t BH = static_cast<int64_t>(B) * H;
    if (workspace_bytes < static_cast<size_t>(BH) * Nq * 4) return FA_ERR_INVALID_ARG;
    int sms;
    DeviceInfo *info;
    st = device_info(sms, info);
    if (st != FA_OK) return st;
    fa::BwdParams p;
    std::memset(&p, 0, sizeof p);
    if (!make_map(&p.tmQ, Q, BH, Nq, d) || !make_map(&p.tmK, K, BH, Nk, d) || !make_map(&p.tmV, V, BH, Nk, d) ||
        !make_map(&p.tmdO, dO, BH, Nq, d))
        return FA_ERR_CUDA;
    p.LSE = LSE;
    p.Dsum = static_cast<float *>(workspace);
    p.dQ = static_cast<__nv_bfloat16 *>(dQ);
    p.dK = static_cast<__nv_bfloat16 *>(dK);
    p.dV = static_cast<__nv_bfloat16 *>(dV);
    p.BH = static_cast<int>(BH);
    p.Nq = Nq;
    p.Nk = Nk;
    p.Tr = (Nq + fa::kBR - 1) / fa::kBR;
    p.Tc = (Nk + fa::kBC - 1) / fa::kBC;
    p.causal = causal != 0;
    p.scale = scale;
    double c2 = static_cast<double>(scale) * 1.4426950408889634;
    if (scale == 0.0f) c2 = 1.1754943508222875e-38 * 1.4426950408889634;
    p.c2 = static_cast<float>(c2);
    std::lock_guard<std::mutex> lock(g_dev_mu);
    bool &attr = d == 64 ? info->bwd_attr64 : info->bwd_attr128;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return d == 64 ? launch_bwd<64>(p, O, dO, static_cast<float *>(workspace), s, attr)
                   : launch_bwd<128>(p, O, dO, static_cast<float *>(workspace), s, attr);
}

extern "C" fa_status fa_check_device_status(fa_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
    unsigned int status = 0;
    if (cudaMemcpyFromSymbol(&status, fa::g_fa_status, sizeof status) != cudaSuccess) return FA_ERR_CUDA;
    if (status == 0) return FA_OK;
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(fa::g_fa_status, &zero, sizeof zero) != cudaSuccess) return FA_ERR_CUDA;
    // bit 2: a backward kernel got a shared-memory base it could not align and did nothing
    return (status & 4u) ? FA_ERR_CUDA : FA_ERR_TIMEOUT;
}

extern "C" const char *fa_status_string(fa_status s) {
    switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: null pointer, size < 1, non-finite scale or size overflow";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: head dimension must be 64 or 128";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED: Q, K, V, O need 16-byte alignment, LSE 4-byte";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel wait expired; outputs are undefined";
    case FA_ERR_TOO_LARGE:
        return "FA_ERR_TOO_LARGE: the partial results need more than the library's fixed 16 MiB scratch area";
    }
    return "unknown fa_status";
}
