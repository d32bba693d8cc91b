// rotate_quant.cu -- incoherent processing before fp8 attention.
//
// marketmaker.cc "Flash Attention and sequence length", FA3 (item 3): Q and
// K are multiplied by the same random orthogonal matrix before the
// block-wise FP8 quantisation, which spreads a few large entries over all d
// components so that the block scales (amax / 448) no longer have to cover
// them.  The matrix here is diag(s) H_d, s = +-1 random signs, H_d the
// Sylvester Hadamard matrix (entries +-1, H H^T = d I), applied
// unnormalised: (Q R)(K R)^T = d Q K^T, so attention on the rotated codes
// uses scale / d.  Without signs the rows are quantised as they are (the
// naive arm).  A block is `rpb` consecutive rows of one head.
//
// One warp per row: lane l holds elements l*E .. l*E+E-1 (E = d / 32); the
// fast Walsh-Hadamard transform pairs element e with e + h for h = 1, 2,
// ..., d/2 -- inside a lane while h < E, across lanes (shfl.xor by h / E)
// after.  Pass 1 takes each block's amax of the (rotated) rows (atomic max on
// the float bits, non-negative), pass 2 recomputes the transform and writes
// codes rn_satfinite(y / scale), scale = amax / 448, division in fp32.
#include "common.cuh"
#include "launch.h"

namespace attn {

namespace rq {

template <int D, bool BF16, bool ROT>
__device__ __forceinline__ void rotate_row(const uint16_t *row, const int8_t *signs, int lane,
                                           float (&y)[D / 32]) {
    constexpr int E = D / 32;
#pragma unroll
    for (int k = 0; k < E; ++k) {
        const uint16_t v = row[lane * E + k];
        const float x = BF16 ? __uint_as_float(static_cast<uint32_t>(v) << 16)
                             : __half2float(__ushort_as_half(v));
        y[k] = (ROT && signs[lane * E + k] < 0) ? -x : x;
    }
    if constexpr (ROT) {
#pragma unroll
        for (int h = 1; h < D; h <<= 1) {
            if (h < E) {
#pragma unroll
                for (int k = 0; k < E; ++k)
                    if ((k & h) == 0) {
                        const float a = y[k], b = y[k + h];
                        y[k] = a + b;
                        y[k + h] = a - b;
                    }
            } else {
                const int m = h / E;
                const bool upper = (lane & m) != 0;
#pragma unroll
                for (int k = 0; k < E; ++k) {
                    const float p = __shfl_xor_sync(0xffffffffu, y[k], m);
                    y[k] = upper ? p - y[k] : y[k] + p;
                }
            }
        }
    }
}

// Block index of row r: head r / rows_per_head, block (r % rows_per_head) / rpb
// of that head's nb blocks.
__device__ __forceinline__ long long block_of(long long r, int rows_per_head, int rpb, int nb) {
    return (r / rows_per_head) * nb + (r % rows_per_head) / rpb;
}

template <int D, bool BF16, bool ROT>
__global__ void __launch_bounds__(256)
    rotq_amax_kernel(const uint16_t *__restrict__ X, const int8_t *__restrict__ signs,
                     unsigned *__restrict__ amax_bits, long long rows, int rows_per_head, int rpb,
                     int nb) {
    const long long r = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows)
        return;
    float y[D / 32];
    rotate_row<D, BF16, ROT>(X + r * D, signs, lane, y);
    float a = 0.f;
#pragma unroll
    for (int k = 0; k < D / 32; ++k)
        a = fmaxf(a, fabsf(y[k]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    if (lane == 0 && a > 0.f)
        atomicMax(amax_bits + block_of(r, rows_per_head, rpb, nb), __float_as_uint(a));
}

template <int D, bool BF16, bool ROT>
__global__ void __launch_bounds__(256)
    rotq_quant_kernel(const uint16_t *__restrict__ X, const int8_t *__restrict__ signs,
                      const unsigned *__restrict__ amax_bits, uint8_t *__restrict__ codes,
                      float *__restrict__ scales, long long rows, int rows_per_head, int rpb,
                      int nb) {
    constexpr int E = D / 32;
    const long long r = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows)
        return;
    const long long blk = block_of(r, rows_per_head, rpb, nb);
    const float amax = __uint_as_float(amax_bits[blk]);
    const float scale = (amax > 0.f && isfinite(amax)) ? amax / 448.0f : 1.0f;
    if (lane == 0 && (r % rows_per_head) % rpb == 0)
        scales[blk] = scale;
    float y[E];
    rotate_row<D, BF16, ROT>(X + r * D, signs, lane, y);
    uint8_t q[E];
#pragma unroll
    for (int k = 0; k < E; k += 2) {
        unsigned short w;
        // cvt packs its first source into the upper byte
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
            : "=h"(w)
            : "f"(__fdiv_rn(y[k + 1], scale)), "f"(__fdiv_rn(y[k], scale)));
        q[k] = static_cast<uint8_t>(w & 0xFF);
        q[k + 1] = static_cast<uint8_t>(w >> 8);
    }
    uint8_t *dst = codes + r * D + lane * E;
    if constexpr (E == 2) {
        *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(q[0] | (q[1] << 8));
    } else if constexpr (E == 4) {
        *reinterpret_cast<uint32_t *>(dst) =
            q[0] | (q[1] << 8) | (q[2] << 16) | (static_cast<uint32_t>(q[3]) << 24);
    } else {
        uint2 v;
        v.x = q[0] | (q[1] << 8) | (q[2] << 16) | (static_cast<uint32_t>(q[3]) << 24);
        v.y = q[4] | (q[5] << 8) | (q[6] << 16) | (static_cast<uint32_t>(q[7]) << 24);
        *reinterpret_cast<uint2 *>(dst) = v;
    }
}

} // namespace rq

template <int D, bool BF16, bool ROT>
static cudaError_t rotq_t(const RotQArgs &a, cudaStream_t st) {
    const long long rows = static_cast<long long>(a.heads) * a.rows_per_head;
    const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
    const int rpb = a.rows_per_block;
    const int nb = (a.rows_per_head + rpb - 1) / rpb;
    cudaError_t e =
        cudaMemsetAsync(a.amax_ws, 0, static_cast<size_t>(a.heads) * nb * 4, st);
    if (e != cudaSuccess)
        return e;
    rq::rotq_amax_kernel<D, BF16, ROT><<<grid, 256, 0, st>>>(
        static_cast<const uint16_t *>(a.X), a.signs, a.amax_ws, rows, a.rows_per_head, rpb, nb);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    rq::rotq_quant_kernel<D, BF16, ROT><<<grid, 256, 0, st>>>(
        static_cast<const uint16_t *>(a.X), a.signs, a.amax_ws, a.codes, a.scales, rows,
        a.rows_per_head, rpb, nb);
    return cudaGetLastError();
}

template <int D>
static cudaError_t rotq_d(const RotQArgs &a, cudaStream_t st) {
    if (a.signs != nullptr)
        return a.bf16 ? rotq_t<D, true, true>(a, st) : rotq_t<D, false, true>(a, st);
    return a.bf16 ? rotq_t<D, true, false>(a, st) : rotq_t<D, false, false>(a, st);
}

cudaError_t rotate_quantize_launch(const RotQArgs &a, cudaStream_t st) {
    switch (a.d) {
    case 64: return rotq_d<64>(a, st);
    case 128: return rotq_d<128>(a, st);
    case 256: return rotq_d<256>(a, st);
    }
    return cudaErrorInvalidValue;
}

} // namespace attn
