/*
 * fa.h -- C ABI of the GB300 (sm_103a) FlashAttention forward library
 * (libfa_gb300.so).
 *
 * The operation is exact softmax attention computed tile by tile with the
 * online-softmax running maximum and running sum, so the N x N score matrix
 * never reaches HBM:
 *
 *   S = scale * Q K^T,   P = softmax(S) row-wise (over the visible keys),
 *   O = P V,             LSE_i = m_i + ln(l_i)  (log-sum-exp of row i of S)
 *
 * Definitions followed:
 *   - "9.4 FlashAttention 与 FlashMLA", sections 9.4.2 (online softmax
 *     recurrence and the online update of O) and 9.4.3 (the fused forward
 *     pass), 9.4.5 (the forward also stores lse = m + log(l));
 *   - "6. FlashAttention 分块逻辑", sections 3.1 (Q-block / KV-block loops,
 *     S = Q K^T * scale), 3.3 and 9 ([B,H,N,d] handled as B*H independent
 *     sequences), 4.1-4.2 (causal mask: key j visible to query i iff j <= i);
 *   - "08. Triton Flash Attention", Step 4 (the wrapper that takes q, k, v and
 *     sm_scale and returns the attention output).
 *
 * All entry points are plain C: pointers, sizes, a stream handle.  Nothing is
 * thrown across the ABI and no error state is kept between calls, except the
 * device-side status word described at fa_check_device_status().
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream); NULL is the legacy default stream. */
typedef struct CUstream_st *fa_stream_t;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,  /* null pointer, a size < 1, non-finite scale, size overflow */
    FA_ERR_UNSUPPORTED = 2,  /* head dimension d other than 64 or 128 */
    FA_ERR_MISALIGNED = 3,   /* Q, K, V or O not 16-byte aligned, or LSE not 4-byte aligned */
    FA_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed (launch, copy, encode) */
    FA_ERR_TIMEOUT = 5,      /* a kernel wait ran past its limit (see fa_check_device_status) */
    FA_ERR_TOO_LARGE = 6     /* more scratch than fa_fwd_splitkv_noalloc's fixed area holds */
} fa_status;

/*
 * fa_fwd -- attention forward on device buffers.
 *
 *   Q    bf16 [B, H, Nq, d]   contiguous row-major, device memory, read only
 *   K    bf16 [B, H, Nk, d]   contiguous row-major, device memory, read only
 *   V    bf16 [B, H, Nk, d]   contiguous row-major, device memory, read only
 *   O    bf16 [B, H, Nq, d]   output, device memory, fully overwritten
 *   LSE  fp32 [B, H, Nq]      output, device memory: ln sum_j exp(S_ij) per row
 *   B, H, Nq, Nk >= 1;  d in {64, 128};  scale finite (1/sqrt(d) is usual)
 *   causal != 0: key j is visible to query i iff j <= i, with absolute indices
 *                (top-left alignment; every row sees key 0, so none is empty)
 *   stream: the work is enqueued on this stream and the call returns at once.
 *
 * Ownership: every pointer is caller-owned; the library allocates nothing and
 * keeps no pointer after returning.  Q, K, V must not overlap O or LSE.
 * Inputs are assumed finite; NaN or Inf in Q, K or V gives undefined output.
 *
 * Errors are reported before anything is enqueued, except FA_ERR_CUDA from the
 * launch itself.  A wait inside the kernel that runs past its limit does not
 * hang the GPU: the kernel stops, records the fact in a device status word and
 * the outputs are undefined; fa_check_device_status() reports it.
 *
 * Launch: the forward kernels (fa_fwd and every entry point below that runs
 * them) are launched with programmatic stream serialisation, so their CTAs
 * may be set up while the previous kernel of the stream drains; each waits
 * for that kernel to complete before its first global-memory access, so
 * ordering on the stream is unchanged.
 */
fa_status fa_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
                 int B, int H, int Nq, int Nk, int d, float scale, int causal,
                 fa_stream_t stream);

/*
 * fa_fwd_host -- the same operation end to end from host memory: copies hQ,
 * hK, hV to the caller's device buffers dQ, dK, dV, runs the forward, and
 * copies dO, dLSE back to hO, hLSE.  Host buffers should be pinned
 * (page-locked) for the copies to be asynchronous.  Shapes, layouts,
 * alignment and errors are those of fa_fwd; the call does not wait for
 * completion (synchronise `stream` before reading hO, hLSE).
 *
 * A large call is split into groups of whole heads (fa_host_groups says how
 * many) that are pipelined: group c is computed while group c+1 is copied in
 * and group c-1 copied out, on streams internal to the library that fork
 * from `stream` (after the work already enqueued on it) and join back into it
 * (later work on `stream` sees every output).  The result is bit-identical to
 * fa_fwd on the same device buffers.  The internal streams are created on the
 * first pipelined call on a device and kept until the process exits.
 */
fa_status fa_fwd_host(const void *hQ, const void *hK, const void *hV, void *hO, float *hLSE,
                      void *dQ, void *dK, void *dV, void *dO, float *dLSE,
                      int B, int H, int Nq, int Nk, int d, float scale, int causal,
                      fa_stream_t stream);

/*
 * fa_host_groups -- how many head groups fa_fwd_host pipelines for these
 * shapes on a GPU with num_sms SMs (host only; no GPU needed): at least
 * 8 MiB of inputs per group, at most 8 groups and one head per group (the
 * SM count does not change the answer at present).  1 means no pipelining.
 * Returns 0 for invalid sizes.
 */
int fa_host_groups(int B, int H, int Nq, int Nk, int d, int num_sms);

/*
 * fa_fwd_test_missing_load -- fa_fwd with one deliberate failure, for testing
 * the library's failure detection: the first K tile of work item `item` (an
 * index into the list fa_schedule returns, 0 is always valid) is never
 * loaded.  The kernel's wait for it gives up after its one-second limit, the
 * kernel stops every role, waits (again with a limit) for the copies and
 * MMAs it started, releases its tensor memory and exits; the GPU context
 * stays usable.  fa_check_device_status then returns FA_ERR_TIMEOUT and O,
 * LSE are undefined.  The pages have no counterpart; this is a property of
 * the library.  Arguments as fa_fwd; item < 0 gives FA_ERR_INVALID_ARG.
 */
fa_status fa_fwd_test_missing_load(const void *Q, const void *K, const void *V, void *O, float *LSE,
                                   int B, int H, int Nq, int Nk, int d, float scale, int causal,
                                   int item, fa_stream_t stream);

/*
 * fa_check_device_status -- synchronises `stream`, then reads and clears the
 * device status word that kernels of this library set when one of their
 * bounded waits expires.  Returns FA_OK, FA_ERR_TIMEOUT, or FA_ERR_CUDA if the
 * synchronisation itself failed or a backward kernel was given a shared-memory
 * base it could not align (it then computes nothing).
 *
 * Scope: there is one status word per device per process, shared by every
 * stream and every host thread that runs this library's kernels on that
 * device.  A timeout in any of them is reported to the first caller that
 * checks after it (whatever stream that caller names; only that stream is
 * synchronised, so a kernel still running elsewhere may set the word after
 * the check) and the check clears it for everyone.  A caller that runs
 * several streams or threads and must know which call failed should check
 * after each call with the other streams idle, or treat FA_ERR_TIMEOUT as
 * "some call since the last check on this device failed".
 */
fa_status fa_check_device_status(fa_stream_t stream);

/*
 * fa_fwd_splitkv -- the same operation with each query tile's key range cut
 * into num_splits slices that run as independent work items, followed by a
 * merge ("6. FlashAttention 分块逻辑", section 11: FlashDecoding -- key/value
 * blocks processed in parallel, each keeping its own max and sum, then
 * reduced; section 13.2: the correct merge of (m, l, o) triples).  It gives
 * short-query / long-key shapes (decoding) enough parallel work to fill the
 * GPU.
 *
 *   Q, K, V, O, LSE, B, H, Nq, Nk, d, scale, causal: as fa_fwd
 *   num_splits   1..256 slices (fa_splitkv_workspace picks one when asked)
 *   workspace    caller-owned device memory, 256-byte aligned, at least the
 *                size fa_splitkv_workspace returns; holds the fp32 partial
 *                outputs [num_splits][B*H][Nq][d] and partial LSE
 *                [num_splits][B*H][Nq]; contents on entry are ignored and are
 *                undefined afterwards
 *   stream       both kernels (partials, merge) are enqueued on it
 *
 * Errors: as fa_fwd; FA_ERR_INVALID_ARG also for num_splits out of range, a
 * NULL or too small workspace; FA_ERR_MISALIGNED for a workspace not 256-byte
 * aligned.  Two calls sharing a workspace must not overlap in time.
 */
fa_status fa_fwd_splitkv(const void *Q, const void *K, const void *V, void *O, float *LSE,
                         int B, int H, int Nq, int Nk, int d, float scale, int causal, int num_splits,
                         void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * fa_splitkv_workspace -- workspace bytes fa_fwd_splitkv needs.  *num_splits
 * = 0 asks for the library's choice for the current device: 1 (no
 * splitting) unless the unsplit work list would keep at most half of the SMs
 * busy, else the most slices that keep every work item in one round (items
 * <= SMs), at most one slice per 128-key tile and at most 64 (this reads the
 * device's SM count); any other value is used
 * as given.  No allocation and no GPU work; with *num_splits > 0 no GPU is
 * needed at all.  With one slice fa_fwd_splitkv is fa_fwd and does not touch
 * the workspace.
 */
fa_status fa_splitkv_workspace(int B, int H, int Nq, int Nk, int d, int causal, int *num_splits,
                               size_t *bytes);

/*
 * fa_fwd_paged -- attention forward over a paged key/value cache ("6.
 * FlashAttention 分块逻辑", section 12: the block table maps each logical
 * block of a sequence to a physical block of the cache, unallocated blocks
 * are skipped, and the tiles are gathered inside the kernel instead of first
 * copying a contiguous K/V).
 *
 *   Q        bf16 [B, H, Nq, d]: the queries of each sequence; they are the
 *            LAST Nq positions of the sequence (prefill: Nq = seq_len;
 *            decoding: Nq = 1)
 *   K_cache, V_cache  bf16 [num_blocks, H, block_size, d], device memory
 *   block_table  int32 [B, max_blocks], device memory: physical block of
 *            logical block l of sequence b; a negative entry is unallocated
 *            and its keys take no part
 *   seq_lens int32 [B], device memory: keys of sequence b (key position k is
 *            row k % block_size of block block_table[b][k / block_size]);
 *            values are clamped to [0, max_blocks * block_size]
 *   O, LSE   as fa_fwd.  causal != 0: query i of sequence b sees keys
 *            k <= i + seq_len[b] - Nq.  A row that sees no key at all
 *            (seq_len < Nq under causal, or only unallocated blocks) gets
 *            O = 0 and LSE = -inf.
 *   block_size in {16, 32, 64, 128, 256}; d in {64, 128}.
 * Errors as fa_fwd; FA_ERR_INVALID_ARG also for NULL block_table/seq_lens or
 * max_blocks, num_blocks < 1; FA_ERR_UNSUPPORTED for another block_size;
 * FA_ERR_MISALIGNED for block_table or seq_lens not 4-byte aligned.
 * Block-table entries >= num_blocks read as zero keys (the copy engine fills
 * out-of-range rows with zeros); keep them in range.
 */
fa_status fa_fwd_paged(const void *Q, const void *K_cache, const void *V_cache, const int *block_table,
                       const int *seq_lens, void *O, float *LSE, int B, int H, int Nq, int max_blocks,
                       int num_blocks, int block_size, int d, float scale, int causal, fa_stream_t stream);

/*
 * fa_fwd_paged_splitkv -- fa_fwd_paged with each query tile's key range cut
 * into num_splits slices run as independent work items and merged afterwards
 * (the decoding case of "6. FlashAttention 分块逻辑": section 12's paged
 * cache read in parallel slices as in section 11, merged as in section 13.2).
 * The slices divide each sequence's own visible key range, so short
 * sequences get short slices; a slice with no key contributes nothing.
 *
 *   Q .. causal  as fa_fwd_paged
 *   num_splits, workspace, workspace_bytes  as fa_fwd_splitkv, with the size
 *                from fa_splitkv_workspace(B, H, Nq, max_blocks * block_size,
 *                d, causal, ...)
 *
 * Errors: those of fa_fwd_paged and of fa_fwd_splitkv.
 */
fa_status fa_fwd_paged_splitkv(const void *Q, const void *K_cache, const void *V_cache, const int *block_table,
                               const int *seq_lens, void *O, float *LSE, int B, int H, int Nq, int max_blocks,
                               int num_blocks, int block_size, int d, float scale, int causal, int num_splits,
                               void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * fa_quantize_fp8 -- per-(batch, head) E4M3 quantisation of a bf16 tensor for
 * fa_fwd_fp8 ("9.4 FlashAttention 与 FlashMLA", section 9.4.4: FlashAttention-3
 * computes attention in FP8 and, before quantising, multiplies Q and K by a
 * random orthogonal matrix -- "incoherent processing" -- which leaves Q K^T
 * unchanged and spreads outlier channels over all channels).
 *
 *   X        bf16 [B, H, N, d], device memory, 16-byte aligned
 *   signs    NULL, or device fp32 [d] of +1/-1: rotate each row by
 *            M = diag(signs) H / sqrt(d) (H the Sylvester-Hadamard matrix,
 *            applied as a fast Walsh-Hadamard transform).  Pass the same
 *            signs for Q and K, and NULL for V.
 *   transpose 0: X8 is E4M3 [B, H, N, d];  1: X8 is E4M3 [B, H, d, ldn] with
 *            ldn = N rounded up to a multiple of 16 and zero padding (the V
 *            layout fa_fwd_fp8 takes)
 *   X8       output, device memory, 16-byte aligned
 *   descale  output, device fp32 [B, H]: code * descale approximates the
 *            (rotated) value; amax / 448 per head (/ sqrt(d) when rotated), 1
 *            for a head of zeros
 * Codes: round to nearest even of (rotated x) * (448 / amax), saturating;
 * every step is one fp32 operation in a fixed order, so the result is the
 * same on any launch.  Four stream operations (a clear of descale, then
 * three kernels).
 * Errors: FA_ERR_INVALID_ARG for NULL pointers, B, H, N < 1 or N above
 * 4,194,240; FA_ERR_UNSUPPORTED for d not 64 or 128; FA_ERR_MISALIGNED.
 */
fa_status fa_quantize_fp8(const void *X, void *X8, float *descale, int B, int H, int N, int d,
                          const float *signs, int transpose, fa_stream_t stream);

/*
 * fa_fwd_fp8 -- the attention forward on E4M3 inputs (FlashAttention-3's FP8
 * mode, "9.4 FlashAttention 与 FlashMLA" section 9.4.4): S = Q K^T on the
 * codes in one tcgen05 MMA kind (fp32 accumulation), scaled by
 * scale * descale_q * descale_k; P rounded to E4M3 for P V (P in V's type,
 * as the bf16 path rounds P to bf16); O = (P V) * descale_v / l in bf16.
 *
 *   Q8       E4M3 [B, H, Nq, d]      (fa_quantize_fp8, transpose = 0)
 *   K8       E4M3 [B, H, Nk, d]      (transpose = 0; same signs as Q8)
 *   Vt8      E4M3 [B, H, d, ldn]     (transpose = 1), ldn = Nk rounded up to
 *            16; the padding columns must hold finite codes (0 does)
 *   descale_q, descale_k, descale_v  device fp32 [B, H], positive
 *   O, LSE, B, H, Nq, Nk, scale, causal, stream: as fa_fwd
 *   d        128 only
 * Errors: as fa_fwd (FA_ERR_UNSUPPORTED for d != 128); FA_ERR_INVALID_ARG
 * for a NULL descale; FA_ERR_MISALIGNED for a descale not 4-byte aligned.
 */
fa_status fa_fwd_fp8(const void *Q8, const void *K8, const void *Vt8, const float *descale_q,
                     const float *descale_k, const float *descale_v, void *O, float *LSE, int B, int H,
                     int Nq, int Nk, int d, float scale, int causal, fa_stream_t stream);

/*
 * fa_bwd -- gradients of the attention forward ("6. FlashAttention 分块逻辑"
 * section 7; "9.4 FlashAttention 与 FlashMLA" sections 9.4.3 and 9.4.5): P is
 * recomputed tile by tile from Q, K and the forward's LSE, never stored, and
 *   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - rowsum(dO * O)),
 *   dQ = scale dS K,  dK = scale dS^T Q.
 * Three kernels run on `stream`: rowsum(dO * O) into the workspace, dK/dV
 * (one CTA per 128-key tile, looping over query tiles) and dQ (one CTA per
 * 128-query tile, looping over key tiles).
 *
 *   Q, K, V, O, LSE  the forward's inputs and outputs (fa_fwd layouts)
 *   dO    bf16 [B, H, Nq, d]  gradient of the loss with respect to O
 *   dQ    bf16 [B, H, Nq, d]  output;  dK, dV  bf16 [B, H, Nk, d]  outputs
 *   workspace  caller-owned device memory, 16-byte aligned, at least
 *              fa_bwd_workspace bytes (fp32 [B, H, Nq]); contents ignored
 *   B, H, Nq, Nk, d, scale, causal: exactly those of the forward call
 * Errors as fa_fwd; FA_ERR_INVALID_ARG also for a NULL dO, dQ, dK, dV or
 * workspace or a too small workspace.  Outputs must not overlap inputs.
 */
fa_status fa_bwd(const void *Q, const void *K, const void *V, const void *O, const float *LSE,
                 const void *dO, void *dQ, void *dK, void *dV,
                 int B, int H, int Nq, int Nk, int d, float scale, int causal,
                 void *workspace, size_t workspace_bytes, fa_stream_t stream);

/* fa_bwd_workspace -- bytes of workspace fa_bwd needs (B * H * Nq * 4). No GPU needed. */
fa_status fa_bwd_workspace(int B, int H, int Nq, int Nk, int d, size_t *bytes);

/*
 * fa_fwd_splitkv_noalloc -- fa_fwd_splitkv for callers that cannot allocate
 * device memory: serving loops whose latency budget rules out the allocator
 * (cudaMalloc may synchronise the device), frameworks whose allocator owns all
 * memory up front, plugins that an inference runtime hands only their input
 * and output tensors and forbids to allocate while they execute.  The
 * pages have no counterpart; this is a property of the library, not of the
 * method.
 *
 * The partial results go to a scratch area inside the library: a fixed
 * 16 MiB array in device memory that every GPU loading the library holds
 * until the process exits.  The call allocates nothing (no cudaMalloc, no
 * cudaFree, no allocating library routine).  The caller still passes Q, K, V,
 * O and LSE, with the meaning, layout and errors of fa_fwd_splitkv;
 * num_splits = 0 lets the library choose, as fa_splitkv_workspace does.
 *
 *   - Limit: num_splits * B * H * Nq * (d + 1) * 4 bytes (plus alignment) must
 *     fit in 16 MiB, else FA_ERR_TOO_LARGE and nothing is enqueued.  One slice
 *     needs no scratch at all.
 *   - The first call on a device looks up the device address of the scratch
 *     array (cudaGetSymbolAddress, with that device current); make that first
 *     call before any stream capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; nothing needs clearing, since each call writes every partial it
 *     reads.  Calls whose kernels overlap on the GPU (different streams without
 *     ordering between them) race on the array and give undefined results.
 */
fa_status fa_fwd_splitkv_noalloc(const void *Q, const void *K, const void *V, void *O, float *LSE,
                                 int B, int H, int Nq, int Nk, int d, float scale, int causal,
                                 int num_splits, fa_stream_t stream);

/*
 * fa_schedule -- the work list fa_fwd (num_splits = 1) or fa_fwd_splitkv
 * would run for these shapes on a GPU with num_sms SMs (host only; no GPU
 * needed).  The kernel's persistent CTAs each walk this list; a work item is
 * one (batch*head, pair of 128-row query tiles) or a single tile, over all
 * the key/value tiles it can see or one slice of them -- the parallelisation
 * over batch x heads x query blocks that "9.4 FlashAttention 与 FlashMLA"
 * section 9.4.4 describes for FA2.  Key/value tiles hold 128 keys at d = 128
 * and 64 keys at d = 64, where two CTAs run on each SM (up to 2 * num_sms
 * CTAs).
 *
 *   items     int32 [capacity][8], caller-owned, may be NULL to only count:
 *             {cta, round, batch*head, first query row, first KV tile,
 *              end KV tile of query tile 0, end KV tile of query tile 1 (-1 if
 *              the item holds one tile), key slice index}
 *   n_items   out: number of items
 * Returns FA_ERR_INVALID_ARG for bad sizes or capacity < *n_items (after
 * setting *n_items), FA_ERR_UNSUPPORTED for d not in {64, 128}.
 */
fa_status fa_schedule(int B, int H, int Nq, int Nk, int d, int causal, int num_sms, int num_splits,
                      int32_t *items, int64_t capacity, int64_t *n_items);

/* A static, human-readable name for a status code (never NULL). */
const char *fa_status_string(fa_status s);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
