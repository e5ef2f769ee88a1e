// Per-(batch, head) E4M3 quantisation of bf16 Q, K, V for the FP8 forward,
// with the optional random Hadamard rotation of "incoherent processing"
// ("9.4 FlashAttention 与 FlashMLA", section 9.4.4: FlashAttention-3 runs
// attention in FP8 and multiplies Q and K by a random orthogonal matrix first,
// which leaves Q K^T unchanged and spreads channel outliers).
//
// For each head: u = x (or x D H, D = diag(signs), H the Sylvester-Hadamard
// matrix, by the fast Walsh-Hadamard transform), amax = max |u|,
// code = E4M3(u * (448 / amax)) with round-to-nearest-even and saturation,
// descale = amax / 448 (times 1/sqrt(d) when rotated, so that
// code * descale approximates x M with M = D H / sqrt(d) orthogonal).  Every
// step is a single fp32 operation in a fixed order, so the codes do not
// depend on the launch shape.
//
// Grids are (heads, row blocks of 64).  Three kernels after the host clears `descale`: the per-head maximum (an
// atomic max on the fp32 bits, which order like the values for
// non-negative numbers), the codes, and the conversion of the maximum in
// `descale` into the scale.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "ptx_sm103.cuh"

namespace fa {

constexpr int kQuantRows = 64;       // token rows per CTA
constexpr int kQuantThreads = 256;   // 8 warps x 8 rows

// Row `row` as this lane's D/32 consecutive channels (lane * D/32 + t), in
// fp32; rotated when signs != nullptr.  Butterfly stage h pairs channels i
// and i + h (bit h of i clear): (a, b) -> (a + b, a - b); stages h < D/32 stay
// inside a lane, the others pair lanes lane ^ (h / (D/32)).
template <int D>
__device__ __forceinline__ void load_row(const __nv_bfloat16 *row, const float *signs, int lane,
                                         float (&u)[D / 32]) {
    constexpr int PER = D / 32;
    if constexpr (PER == 4) {
        const uint2 w = *reinterpret_cast<const uint2 *>(row + lane * 4);
        u[0] = __uint_as_float(w.x << 16);
        u[1] = __uint_as_float(w.x & 0xFFFF0000u);
        u[2] = __uint_as_float(w.y << 16);
        u[3] = __uint_as_float(w.y & 0xFFFF0000u);
    } else {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(row + lane * 2);
        u[0] = __uint_as_float(w << 16);
        u[1] = __uint_as_float(w & 0xFFFF0000u);
    }
    if (signs == nullptr) return;
    #pragma unroll
    for (int t = 0; t < PER; ++t) u[t] *= signs[lane * PER + t];   // +-1: exact
    #pragma unroll
    for (int h = 1; h < PER; h <<= 1) {
        #pragma unroll
        for (int t = 0; t < PER; ++t) {
            if (t & h) continue;
            const float a = u[t], b = u[t + h];
            u[t] = __fadd_rn(a, b);
            u[t + h] = __fsub_rn(a, b);
        }
    }
    #pragma unroll
    for (int h = PER; h < D; h <<= 1) {
        const int lm = h / PER;
        #pragma unroll
        for (int t = 0; t < PER; ++t) {
            const float o = __shfl_xor_sync(0xffffffffu, u[t], lm);
            u[t] = (lane & lm) ? __fsub_rn(o, u[t]) : __fadd_rn(u[t], o);
        }
    }
}

// amax_bits[bh] = max(amax_bits[bh], bits of max |u| over this CTA's rows).
template <int D>
__global__ void __launch_bounds__(kQuantThreads) fa_amax_kernel(const __nv_bfloat16 *__restrict__ X,
                                                                const float *__restrict__ signs,
                                                                unsigned *__restrict__ amax_bits, int N) {
    const int bh = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float m = 0.f;
    for (int i = 0; i < kQuantRows / 8; ++i) {
        const int r = blockIdx.y * kQuantRows + warp * 8 + i;   // warp-uniform
        if (r >= N) break;
        float u[D / 32];
        load_row<D>(X + (static_cast<size_t>(bh) * N + r) * D, signs, lane, u);
        #pragma unroll
        for (int t = 0; t < D / 32; ++t) m = fmaxf(m, fabsf(u[t]));
    }
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0 && m > 0.f) atomicMax(amax_bits + bh, __float_as_uint(m));
}

// Codes of this CTA's rows: [bh][N][D], or transposed [bh][D][ldn] (rows
// N..ldn-1 written as zero) through a shared-memory tile.
template <int D, bool TRANSPOSE>
__global__ void __launch_bounds__(kQuantThreads) fa_quant_kernel(const __nv_bfloat16 *__restrict__ X,
                                                                 const float *__restrict__ signs,
                                                                 const unsigned *__restrict__ amax_bits,
                                                                 uint8_t *__restrict__ X8, int N, int ldn) {
    constexpr int PER = D / 32;
    // [channel][row], rows padded to 68 bytes so that the lanes' byte stores
    // and the 4-byte reads below spread over the banks
    constexpr int kPitch = kQuantRows + 4;
    __shared__ __align__(16) uint8_t tile[TRANSPOSE ? D * kPitch : 16];
    const int bh = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.y * kQuantRows;
    const float a = __uint_as_float(amax_bits[bh]);
    const float inv = a > 0.f ? __fdiv_rn(448.f, a) : 0.f;
    for (int i = 0; i < kQuantRows / 8; ++i) {
        const int rl = warp * 8 + i, r = n0 + rl;               // warp-uniform
        uint32_t w = 0;
        if (r < N) {
            float u[PER];
            load_row<D>(X + (static_cast<size_t>(bh) * N + r) * D, signs, lane, u);
            if constexpr (PER == 4)
                w = ptx::pack_e4m3x4(__fmul_rn(u[0], inv), __fmul_rn(u[1], inv), __fmul_rn(u[2], inv),
                                     __fmul_rn(u[3], inv));
            else
                w = ptx::pack_e4m3x4(__fmul_rn(u[0], inv), __fmul_rn(u[1], inv), 0.f, 0.f) & 0xFFFFu;
        }
        if constexpr (!TRANSPOSE) {
            if (r < N) {
                uint8_t *dst = X8 + (static_cast<size_t>(bh) * N + r) * D + lane * PER;
                if constexpr (PER == 4) *reinterpret_cast<uint32_t *>(dst) = w;
                else *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(w);
            }
        } else {
            #pragma unroll
            for (int t = 0; t < PER; ++t) tile[(lane * PER + t) * kPitch + rl] = (w >> (8 * t)) & 0xFFu;
        }
    }
    if constexpr (TRANSPOSE) {
        __syncthreads();
        // D channels x 64 rows = D * 4 pieces of 16 bytes
        for (int c = threadIdx.x; c < D * (kQuantRows / 16); c += kQuantThreads) {
            const int ch = c / (kQuantRows / 16), part = c % (kQuantRows / 16);
            const int k0 = n0 + part * 16;
            if (k0 < ldn) {
                const uint32_t *src = reinterpret_cast<const uint32_t *>(tile + ch * kPitch + part * 16);
                *reinterpret_cast<uint4 *>(X8 + (static_cast<size_t>(bh) * D + ch) * ldn + k0) =
                    make_uint4(src[0], src[1], src[2], src[3]);
            }
        }
    }
}

// descale[bh]: the maximum left there by fa_amax_kernel -> amax / 448 * rs
// (rs = 1/sqrt(d) when rotated, else 1); 1 for a head of zeros.
__global__ void fa_descale_kernel(float *descale, int BH, float rs) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= BH) return;
    const float a = descale[i];
    descale[i] = a > 0.f ? __fmul_rn(__fdiv_rn(a, 448.f), rs) : 1.f;
}

}  // namespace fa
