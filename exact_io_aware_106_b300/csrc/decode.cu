// decode.cu -- single-token attention over a block-paged KV cache.
//
// Split-KV: every CTA owns (sequence s, KV head hk, a chunk of heads of that
// group, a range of `tps` tokens).  It streams the range in 16-token units
// (one unit = a contiguous 16 x d slice of a cache block) through a ring of
// shared-memory stages filled by 1-D bulk copies, and folds them into the
// per-row online-softmax state (m, l, u) of auturnal.com "From attention to
// IO-aware execution" §8: running max m, denominator l, un-normalised sum u,
// both rescaled by 2^(m - m') when a unit raises the max.  The CTA writes
// its partial (m, l, u) per query head; a second kernel merges the partials
// of a sequence with the same alignment rule and emits O = u / l and the
// log-sum-exp.  Decode is bound by HBM bandwidth (code-journey.com,
// "Attention co-design", prefill vs decode), so the kernel is built around
// keeping many bulk copies in flight and uses CUDA-core FMAs.
//
// Scores are kept in the log2 domain: q is pre-multiplied by
// scale * log2(e) (* k_scale for an E4M3 cache) so that p = 2^(s - m).
// The running max is only moved when a unit's max exceeds it by more than
// 2^8 (p stays <= 256); any reference value not below the visible scores
// gives the same u / l, by the max-subtraction invariance of §8.
#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace attn {

namespace dec {

constexpr int kUnit = 16;     // tokens per streamed unit
constexpr int kCW = 4;        // consumer warps per CTA
constexpr int kThreads = (kCW + 1) * 32;
constexpr int kMaxUnits = 256; // units per CTA (tps <= 4096)
constexpr float kRescaleThreshold = 8.0f;

template <int D, bool KV8>
struct Layout {
    static constexpr int ESZ = KV8 ? 1 : 2;
    static constexpr int ROW_BYTES = D * ESZ;
    static constexpr int UNIT_BYTES = kUnit * ROW_BYTES;
    static constexpr int CH_BYTES = ROW_BYTES >= 128 ? 16 : 8; // bytes a lane reads per chunk
    static constexpr int CH = CH_BYTES / ESZ;                   // elements per chunk
    static constexpr int NCHUNK = ROW_BYTES / (8 * CH_BYTES);   // chunks per row per lane
    static constexpr int EPL = D / 8;                           // elements per lane
    static constexpr int NST0 = 65536 / (2 * UNIT_BYTES);
    static constexpr int NST = NST0 < 4 ? 4 : (NST0 > 16 ? 16 : NST0);
    static_assert(NCHUNK * CH == EPL, "lane element split");
    // block groups (1, 2 or 4) take units round-robin: a stage must always
    // belong to the same group for the parity waits to be exact
    static_assert(NST % kCW == 0, "each stage must belong to one block group");
};

// Element index of chunk c, element i of lane column dc.
template <int D, bool KV8>
__device__ __forceinline__ int elem_index(int c, int dc, int i) {
    using Ly = Layout<D, KV8>;
    return c * 8 * Ly::CH + dc * Ly::CH + i;
}

__device__ __forceinline__ void e4m3x2_to_f32(unsigned short v, float &lo, float &hi) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
    lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
    hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
}

// Read this lane's EPL elements of one cache row from shared memory.
template <int D, bool KV8, bool BF16>
__device__ __forceinline__ void load_row(const uint8_t *row, int dc, float (&x)[D / 8]) {
    using Ly = Layout<D, KV8>;
#pragma unroll
    for (int c = 0; c < Ly::NCHUNK; ++c) {
        const uint8_t *p = row + c * 8 * Ly::CH_BYTES + dc * Ly::CH_BYTES;
        uint32_t w[4];
        if constexpr (Ly::CH_BYTES == 16) {
            uint4 v = *reinterpret_cast<const uint4 *>(p);
            w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
        } else {
            uint2 v = *reinterpret_cast<const uint2 *>(p);
            w[0] = v.x, w[1] = v.y, w[2] = 0, w[3] = 0;
        }
        constexpr int NW = Ly::CH_BYTES / 4;
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            if constexpr (KV8) {
                float a, b, cc, dd;
                e4m3x2_to_f32(static_cast<unsigned short>(w[k] & 0xFFFFu), a, b);
                e4m3x2_to_f32(static_cast<unsigned short>(w[k] >> 16), cc, dd);
                x[c * Ly::CH + 4 * k + 0] = a;
                x[c * Ly::CH + 4 * k + 1] = b;
                x[c * Ly::CH + 4 * k + 2] = cc;
                x[c * Ly::CH + 4 * k + 3] = dd;
            } else {
                x[c * Ly::CH + 2 * k + 0] = lo16<BF16>(w[k]);
                x[c * Ly::CH + 2 * k + 1] = hi16<BF16>(w[k]);
            }
        }
    }
}

__host__ __device__ constexpr int ilog2c(int x) { return x <= 1 ? 0 : 1 + ilog2c(x / 2); }

// After the transposed reduction over the 8 lanes of a token group, lane
// bits 2,1,0 (shuffle offsets 4,2,1) select halves of the value index
// j = g * 4 + t (head g, token t of the lane's token group).  Step k
// (offset 4 >> k) halves the list while it has more than one entry and then
// fixes j bit (L - 1 - k), L = log2(4 * HPW).
template <int HPW>
struct Red {
    static constexpr int NV = 4 * HPW;             // partial values per lane
    static constexpr int L = ilog2c(NV);
    static constexpr int NF = NV >= 8 ? NV / 8 : 1; // values left per lane
    __host__ __device__ static constexpr bool halving(int k) { return (NV >> (k + 1)) >= 1; }
    __host__ __device__ static constexpr int jbit(int k) { return L - 1 - k; }
    // lane-bit mask (within bits 0..2) whose j bit is a token bit
    __host__ __device__ static constexpr int tokmask() {
        int m = 0;
        for (int k = 0; k < 3; ++k)
            if (halving(k) && jbit(k) <= 1)
                m |= (4 >> k);
        return m;
    }
};

template <int HPW>
__device__ __forceinline__ int red_jindex(int i, int lane) {
    using R = Red<HPW>;
    int j = i;
#pragma unroll
    for (int k = 0; k < 3; ++k)
        if (R::halving(k))
            j += ((lane >> (2 - k)) & 1) << R::jbit(k);
    return j;
}

template <int D, int HPW, bool BF16, bool KV8>
__global__ void __launch_bounds__(kThreads)
    decode_split_kernel(const void *__restrict__ q_, const uint8_t *__restrict__ Kc,
                        const uint8_t *__restrict__ Vc, const int32_t *__restrict__ block_table,
                        const int32_t *__restrict__ seq_lens, const float *__restrict__ k_scale,
                        const float *__restrict__ v_scale, float2 *__restrict__ ws_ml,
                        float *__restrict__ ws_u, int Hq, int Hkv, int G, int nhg, int hg_cta,
                        int n_hg_chunks, int block_size, int max_blocks, int num_blocks,
                        int max_seq_len, int tps, int max_splits, float qk_scale_log2,
                        unsigned *err) {
    using Ly = Layout<D, KV8>;
    using R = Red<HPW>;
    constexpr int EPL = Ly::EPL;
    constexpr int NST = Ly::NST;

    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *stages = smem;                                  // NST x (K unit, V unit)
    float *scratch = reinterpret_cast<float *>(smem + NST * 2 * Ly::UNIT_BYTES);
    constexpr int SCR_PER_WARP = HPW * kUnit + 4 * HPW;      // p[g][16], alpha[g], bsum[g]
    int32_t *blk_ids = reinterpret_cast<int32_t *>(scratch + kCW * SCR_PER_WARP);
    uint64_t *bars = reinterpret_cast<uint64_t *>(blk_ids + kMaxUnits);
    __shared__ int s_flag;      // 1 = bad index / length, 2 = aborted
    __shared__ int s_abort;

    const int split = blockIdx.x;
    const int hk = blockIdx.y / n_hg_chunks;
    const int hg0 = (blockIdx.y % n_hg_chunks) * hg_cta; // first head group of this CTA
    const int s = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int len = seq_lens[s];
    const int t0 = split * tps;
    const bool len_ok = len >= 0 && len <= max_seq_len &&
                        (len + block_size - 1) / block_size <= max_blocks;
    const int hg_here = min(hg_cta, nhg - hg0); // head groups this CTA serves
    const int n_heads_cta = hg_here * HPW;
    const int head0 = hk * G + hg0 * HPW;

    auto write_invalid = [&]() {
        for (int i = threadIdx.x; i < n_heads_cta; i += blockDim.x) {
            size_t o = (static_cast<size_t>(s) * Hq + head0 + i) * max_splits + split;
            ws_ml[o] = make_float2(0.f, -1.f); // l < 0 marks an unusable partial
        }
    };

    if (!len_ok) { // the combine kernel zeroes this sequence's output
        if (split == 0 && threadIdx.x == 0 && blockIdx.y == 0)
            atomicOr(err, DERR_INDEX);
        return;
    }
    if (t0 >= len)
        return; // past the end of this sequence: no partial for this split
    const int t1 = min(len, t0 + tps);
    const int nunits = (t1 - t0 + kUnit - 1) / kUnit;

    // ---- validate and stage the block indices of this range
    if (threadIdx.x == 0) {
        s_flag = 0;
        s_abort = 0;
    }
    __syncthreads();
    for (int u = threadIdx.x; u < nunits; u += blockDim.x) {
        int blk = (t0 + u * kUnit) / block_size;
        int phys = block_table[static_cast<size_t>(s) * max_blocks + blk];
        if (phys < 0 || phys >= num_blocks)
            s_flag = 1;
        blk_ids[u] = phys;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(smem_u32(&bars[i]), 1);         // full: producer arrive + tx bytes
            mbar_init(smem_u32(&bars[NST + i]), hg_here); // empty: one arrive per consumer warp
        }
        fence_barrier_init();
    }
    __syncthreads();
    if (s_flag) {
        if (threadIdx.x == 0)
            atomicOr(err, DERR_INDEX);
        write_invalid();
        return;
    }
    volatile int *abort_flag = &s_abort;
    const int nbg = kCW / hg_here; // block groups

    if (warp == kCW) {
        // ------------------------------------------------ producer warp
        if (lane == 0) {
            int issued = 0;
            for (int u = 0; u < nunits; ++u) {
                const int st = u % NST;
                if (u >= NST &&
                    !mbar_wait(smem_u32(&bars[NST + st]), ((u / NST) - 1) & 1, abort_flag, err))
                    break;
                const int pos = t0 + u * kUnit;
                const int sub = (pos % block_size) / kUnit;
                const size_t off =
                    ((static_cast<size_t>(blk_ids[u]) * Hkv + hk) * block_size + sub * kUnit) *
                    Ly::ROW_BYTES;
                uint8_t *dst = stages + st * 2 * Ly::UNIT_BYTES;
                const uint32_t fb = smem_u32(&bars[st]);
                mbar_arrive_expect_tx(fb, 2 * Ly::UNIT_BYTES);
                bulk_g2s(smem_u32(dst), Kc + off, Ly::UNIT_BYTES, fb);
                bulk_g2s(smem_u32(dst + Ly::UNIT_BYTES), Vc + off, Ly::UNIT_BYTES, fb);
                issued = u + 1;
            }
            if (*abort_flag) {
                // let copies already in flight land before the CTA exits
                for (int u = max(0, issued - NST); u < issued; ++u)
                    mbar_wait_drain(smem_u32(&bars[u % NST]), (u / NST) & 1);
            }
        }
    } else {
        // ------------------------------------------------ consumer warps
        const int hgl = warp % hg_here; // head group within the CTA
        const int bg = warp / hg_here;  // block group
        const bool active = warp < hg_here * nbg;
        const int tg = lane >> 3, dc = lane & 7;
        const int hbase = head0 + hgl * HPW;
        const float csc = qk_scale_log2 * (KV8 ? k_scale[hk] : 1.0f);

        float q[HPW][EPL];
#pragma unroll
        for (int g = 0; g < HPW; ++g) {
            const size_t qoff = (static_cast<size_t>(s) * Hq + hbase + g) * D;
#pragma unroll
            for (int c = 0; c < Ly::NCHUNK; ++c)
#pragma unroll
                for (int i = 0; i < Ly::CH; ++i) {
                    const int e = elem_index<D, KV8>(c, dc, i);
                    float x;
                    if constexpr (BF16)
                        x = __bfloat162float(static_cast<const __nv_bfloat16 *>(q_)[qoff + e]);
                    else
                        x = __half2float(static_cast<const __half *>(q_)[qoff + e]);
                    q[g][c * Ly::CH + i] = x * csc;
                }
        }
        float o[HPW][EPL];
#pragma unroll
        for (int g = 0; g < HPW; ++g)
#pragma unroll
            for (int e = 0; e < EPL; ++e)
                o[g][e] = 0.f;
        float m_own = -INFINITY, l_own = 0.f;
        const int g_lane = red_jindex<HPW>(0, lane) >> 2;
        float *ps = scratch + warp * SCR_PER_WARP; // [HPW][16]
        float *hs = ps + HPW * kUnit;              // [HPW][4]: alpha, bsum
        bool ok = true;

        for (int u = bg; active && u < nunits; u += nbg) {
            const int st = u % NST;
            if (!mbar_wait(smem_u32(&bars[st]), (u / NST) & 1, abort_flag, err)) {
                ok = false;
                break;
            }
            const uint8_t *Ks = stages + st * 2 * Ly::UNIT_BYTES;
            const uint8_t *Vs = Ks + Ly::UNIT_BYTES;
            const int upos = t0 + u * kUnit;

            // scores: partial dot products over this lane's elements
            float part[R::NV];
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                float k[EPL];
                load_row<D, KV8, BF16>(Ks + (tg * 4 + it) * Ly::ROW_BYTES, dc, k);
#pragma unroll
                for (int g = 0; g < HPW; ++g) {
                    float acc = 0.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e)
                        acc = fmaf(q[g][e], k[e], acc);
                    part[g * 4 + it] = acc;
                }
            }
            // transposed reduction across the 8 lanes of the token group
            {
                int n = R::NV;
#pragma unroll
                for (int k = 0; k < 3; ++k) {
                    const int off = 4 >> k;
                    if (R::halving(k)) {
                        const int h = n / 2;
                        const bool upper = (lane & off) != 0;
#pragma unroll
                        for (int i = 0; i < R::NV / 2; ++i) {
                            if (i < h) {
                                const float send = upper ? part[i] : part[i + h];
                                const float keep = upper ? part[i + h] : part[i];
                                part[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                            }
                        }
                        n = h;
                    } else {
                        part[0] += __shfl_xor_sync(0xffffffffu, part[0], off);
                    }
                }
            }
            // mask, head max, probabilities, head sums
            float sv[R::NF];
            float bmax = -INFINITY;
#pragma unroll
            for (int i = 0; i < R::NF; ++i) {
                const int t = red_jindex<HPW>(i, lane) & 3;
                const bool valid = upos + tg * 4 + t < t1;
                sv[i] = valid ? part[i] : -INFINITY;
                bmax = fmaxf(bmax, sv[i]);
            }
#pragma unroll
            for (int b = 0; b < 3; ++b)
                if (R::tokmask() & (1 << b))
                    bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 1 << b));
            bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 8));
            bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 16));
            float m_use = m_own;
            if (bmax > m_own + kRescaleThreshold || m_own == -INFINITY)
                m_use = fmaxf(bmax, m_own);
            const float alpha =
                (m_use == m_own) ? 1.0f : ((m_own == -INFINITY) ? 0.f : ex2(m_own - m_use));
            float bsum = 0.f;
            __syncwarp();
#pragma unroll
            for (int i = 0; i < R::NF; ++i) {
                const int t = red_jindex<HPW>(i, lane) & 3;
                const float p = ex2(sv[i] - m_use);
                bsum += p;
                ps[g_lane * kUnit + tg * 4 + t] = p;
            }
#pragma unroll
            for (int b = 0; b < 3; ++b)
                if (R::tokmask() & (1 << b))
                    bsum += __shfl_xor_sync(0xffffffffu, bsum, 1 << b);
            bsum += __shfl_xor_sync(0xffffffffu, bsum, 8);
            bsum += __shfl_xor_sync(0xffffffffu, bsum, 16);
            if ((lane & R::tokmask()) == 0 && tg == 0) {
                hs[g_lane * 4 + 0] = alpha;
                hs[g_lane * 4 + 1] = bsum;
            }
            l_own = l_own * alpha + bsum;
            m_own = m_use;
            __syncwarp();

            // rescale u when any head's reference moved
            float al[HPW];
            bool any = false;
#pragma unroll
            for (int g = 0; g < HPW; ++g) {
                al[g] = hs[g * 4 + 0];
                any |= (al[g] != 1.0f);
            }
            if (any) {
#pragma unroll
                for (int g = 0; g < HPW; ++g)
#pragma unroll
                    for (int e = 0; e < EPL; ++e)
                        o[g][e] *= al[g];
            }
            // u += p V over this lane's tokens
            float pv[HPW][4];
#pragma unroll
            for (int g = 0; g < HPW; ++g) {
                const float4 t4 = *reinterpret_cast<const float4 *>(ps + g * kUnit + tg * 4);
                pv[g][0] = t4.x, pv[g][1] = t4.y, pv[g][2] = t4.z, pv[g][3] = t4.w;
            }
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                if (upos + tg * 4 + it < t1) {
                    float v[EPL];
                    load_row<D, KV8, BF16>(Vs + (tg * 4 + it) * Ly::ROW_BYTES, dc, v);
#pragma unroll
                    for (int g = 0; g < HPW; ++g)
#pragma unroll
                        for (int e = 0; e < EPL; ++e)
                            o[g][e] = fmaf(pv[g][it], v[e], o[g][e]);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bars[NST + st]));
        }

        // sum u over the four token groups
#pragma unroll
        for (int g = 0; g < HPW; ++g)
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], 8);
                o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], 16);
            }
        if (!ok)
            s_flag = 2;

        // ---- merge the block-group warps of each head group (consumers only)
        asm volatile("bar.sync 1, %0;" ::"r"(kCW * 32) : "memory");
        float *mrg = reinterpret_cast<float *>(stages); // stages are drained now
        float *mrg_ml = mrg;                            // [kCW][HPW][2]
        float *mrg_u = mrg + kCW * HPW * 2;             // [kCW][HPW][D]
        if (active && (lane & R::tokmask()) == 0 && tg == 0) {
            mrg_ml[(warp * HPW + g_lane) * 2 + 0] = m_own;
            mrg_ml[(warp * HPW + g_lane) * 2 + 1] = l_own;
        }
        if (active && tg == 0) {
#pragma unroll
            for (int g = 0; g < HPW; ++g)
#pragma unroll
                for (int c = 0; c < Ly::NCHUNK; ++c)
#pragma unroll
                    for (int i = 0; i < Ly::CH; ++i)
                        mrg_u[(warp * HPW + g) * D + elem_index<D, KV8>(c, dc, i)] =
                            o[g][c * Ly::CH + i];
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kCW * 32) : "memory");
        const bool bad = s_flag != 0;
        const float vsc = KV8 ? v_scale[hk] : 1.0f;
        for (int idx = threadIdx.x; idx < n_heads_cta * D; idx += kCW * 32) {
            const int lh = idx / D, e = idx % D;
            const int hgl2 = lh / HPW, g = lh % HPW;
            float M = -INFINITY;
            for (int b2 = 0; b2 < nbg; ++b2)
                M = fmaxf(M, mrg_ml[((b2 * hg_here + hgl2) * HPW + g) * 2]);
            float Lsum = 0.f, U = 0.f;
            for (int b2 = 0; b2 < nbg; ++b2) {
                const int w = b2 * hg_here + hgl2;
                const float mw = mrg_ml[(w * HPW + g) * 2];
                const float sc = (mw == -INFINITY) ? 0.f : ex2(mw - M);
                Lsum += sc * mrg_ml[(w * HPW + g) * 2 + 1];
                U += sc * mrg_u[(w * HPW + g) * D + e];
            }
            const size_t o_idx = (static_cast<size_t>(s) * Hq + head0 + lh) * max_splits + split;
            ws_u[o_idx * D + e] = U * vsc;
            if (e == 0)
                ws_ml[o_idx] = bad ? make_float2(0.f, -1.f) : make_float2(M, Lsum);
        }
    }
}

template <int D, typename OutT>
__global__ void __launch_bounds__(D)
    decode_combine_kernel(const float2 *__restrict__ ws_ml, const float *__restrict__ ws_u,
                          const int32_t *__restrict__ seq_lens, OutT *__restrict__ O,
                          float *__restrict__ lse, int Hq, int block_size, int max_blocks,
                          int max_seq_len, int tps, int max_splits) {
    const int sh = blockIdx.x;
    const int s = sh / Hq;
    const int e = threadIdx.x;
    const int len = seq_lens[s];
    const bool len_ok = len >= 0 && len <= max_seq_len &&
                        (len + block_size - 1) / block_size <= max_blocks;
    const int nsplit = len_ok ? (len + tps - 1) / tps : 0;
    const float2 *ml = ws_ml + static_cast<size_t>(sh) * max_splits;
    float M = -INFINITY;
    bool bad = !len_ok;
    for (int k = 0; k < nsplit; ++k) {
        const float2 v = ml[k];
        bad |= v.y < 0.f;
        M = fmaxf(M, v.x);
    }
    float L = 0.f, U = 0.f;
    if (!bad) {
        for (int k = 0; k < nsplit; ++k) {
            const float2 v = ml[k];
            const float w = ex2(v.x - M);
            L += w * v.y;
            U += w * ws_u[(static_cast<size_t>(sh) * max_splits + k) * D + e];
        }
    }
    float out = 0.f, l_out;
    if (bad) {
        l_out = __int_as_float(0x7fc00000); // NaN marks an invalid row
    } else if (nsplit == 0) {
        l_out = -INFINITY; // empty sequence
    } else {
        out = U / L;
        l_out = M * 0.69314718055994530942f + logf(L);
    }
    if constexpr (sizeof(OutT) == 4)
        O[static_cast<size_t>(sh) * D + e] = out;
    else if constexpr (std::is_same<OutT, __nv_bfloat16>::value)
        O[static_cast<size_t>(sh) * D + e] = __float2bfloat16_rn(out);
    else
        O[static_cast<size_t>(sh) * D + e] = __float2half_rn(out);
    if (lse != nullptr && e == 0)
        lse[sh] = l_out;
}

} // namespace dec

// ---------------------------------------------------------------------------
// 16-bit cache: the two small products on the warp-level tensor cores.
//
// Per CTA: (split, KV head hk, sequence s).  The G <= 16 query heads of the
// group are the rows of one 16-row MMA tile (rows G..15 are zero), so a
// 16-token unit costs D/8 MMAs for S = q K^T and D/8 (2 D/8 with the P
// residual) for u += P V, instead of ~G * 16 * D * 2 scalar FMAs.  K and V
// units arrive by TMA into 128-byte-swizzled shared memory (one 3-D tensor
// map per cache, box 64 x 16), which makes the ldmatrix reads of both the
// K operand and the transposed V operand free of bank conflicts.  A producer
// warp keeps NST units in flight; consumer warp w takes units w, w + 4, ...
// with its own (m, l, u) per row, and the four states are merged at the end.
// The online-softmax statistics follow the same rules as the scalar path:
// log2-domain scores, a reference max moved only when a unit's max exceeds
// it by more than 8, alpha = 2^(m - m') applied to l and u.
namespace dm {

constexpr int kUnit = 16;     // tokens per unit (one TMA box row count)
constexpr int kNC = 4;        // consumer warps
constexpr int kThreads = (kNC + 1) * 32;
constexpr int kMaxUnits = 256; // units per CTA (tps <= 4096)
constexpr int kSplitKeys = 512; // sequences shorter than this carry the P residual
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct Lay {
    static constexpr int PANELS = D / 64;               // 128-byte column panels
    static constexpr int PANEL_BYTES = kUnit * 128;     // one TMA box
    static constexpr int HALF = PANELS * PANEL_BYTES;   // K (or V) of one unit
    static constexpr int STAGE = 2 * HALF;
    // Unit u lives in stage u % NST and is consumed by warp u % kNC.  With
    // NST a multiple of kNC a stage is only ever consumed by one warp, so
    // that warp has itself waited for the stage's previous phase before it
    // waits (by parity) for the next one; otherwise a warp could wait on a
    // stage whose previous fill, for another warp, has not landed yet, and
    // the parity test would pass one phase early.
    static constexpr int NST = D == 64 ? 12 : (D == 128 ? 8 : 4);
    static_assert(NST % kNC == 0, "each stage must belong to one consumer warp");
    static constexpr int MIN_CTAS = D == 64 ? 4 : (D == 128 ? 3 : 2);
    static constexpr int QROW = 2 * D + 16;             // padded q row (conflict-free ldmatrix)
    static constexpr int RING = NST * STAGE;
    static constexpr int MERGE_U = kNC * 16 * D * 4;
    static constexpr int MERGE = MERGE_U + kNC * 16 * 8;
    static constexpr int OFF_Q = RING > MERGE ? RING : MERGE;
    static constexpr int OFF_BLK = OFF_Q + 16 * QROW;
    static constexpr int OFF_BAR = OFF_BLK + kMaxUnits * 4;
    static constexpr int SMEM = OFF_BAR + 2 * NST * 8 + 16 + 1024; // + alignment slack
};

__device__ __forceinline__ float max4(float a, float b, float c, float d) {
    return fmaxf(fmaxf(a, b), fmaxf(c, d));
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, Lay<D>::MIN_CTAS)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const void *__restrict__ q_,
                      const int32_t *__restrict__ block_table,
                      const int32_t *__restrict__ seq_lens, float2 *__restrict__ ws_ml,
                      float *__restrict__ ws_u, int Hq, int G, int block_size, int max_blocks,
                      int num_blocks, int max_seq_len, int tps, int max_splits, float c,
                      unsigned *err) {
    using Ly = Lay<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u; // swizzle atoms repeat every 1 KB
    uint8_t *base = smem_raw + (base_s - raw_s);
    int32_t *blk_ids = reinterpret_cast<int32_t *>(base + Ly::OFF_BLK);
    const uint32_t sQ = base_s + Ly::OFF_Q;
    const uint32_t bar0 = base_s + Ly::OFF_BAR;
    auto b_full = [&](int i) { return bar0 + 8u * i; };
    auto b_empty = [&](int i) { return bar0 + 8u * (Ly::NST + i); };
    __shared__ int s_flag; // 1 = bad index, 2 = aborted
    __shared__ int s_abort;

    const int split = blockIdx.x, hk = blockIdx.y, s = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int len = seq_lens[s];
    const bool len_ok = len >= 0 && len <= max_seq_len &&
                        (len + block_size - 1) / block_size <= max_blocks;
    if (!len_ok) { // the combine kernel zeroes this sequence's output
        if (split == 0 && hk == 0 && threadIdx.x == 0)
            atomicOr(err, DERR_INDEX);
        return;
    }
    const int t0 = split * tps;
    if (t0 >= len)
        return; // past the end of this sequence: no partial for this split
    const int t1 = min(len, t0 + tps);
    const int nunits = (t1 - t0 + kUnit - 1) / kUnit;
    const int head0 = hk * G;

    if (threadIdx.x == 0) {
        s_flag = 0;
        s_abort = 0;
    }
    __syncthreads();
    for (int u = threadIdx.x; u < nunits; u += kThreads) {
        const int phys =
            block_table[static_cast<size_t>(s) * max_blocks + (t0 + u * kUnit) / block_size];
        if (phys < 0 || phys >= num_blocks)
            s_flag = 1;
        blk_ids[u] = phys;
    }
    // the group's query rows, zero rows up to 16
    for (int i = threadIdx.x; i < 16 * (D / 8); i += kThreads) {
        const int r = i / (D / 8), c8 = i % (D / 8);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < G)
            v = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(q_) +
                                                 (static_cast<size_t>(s) * Hq + head0 + r) * D +
                                                 c8 * 8);
        *reinterpret_cast<uint4 *>(base + Ly::OFF_Q + r * Ly::QROW + c8 * 16) = v;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < Ly::NST; ++i) {
            mbar_init(b_full(i), 1);  // producer arrive + tx bytes
            mbar_init(b_empty(i), 1); // the consuming warp
        }
        fence_barrier_init();
    }
    __syncthreads();
    if (s_flag) {
        if (threadIdx.x == 0)
            atomicOr(err, DERR_INDEX);
        for (int r = threadIdx.x; r < G; r += kThreads)
            ws_ml[(static_cast<size_t>(s) * Hq + head0 + r) * max_splits + split] =
                make_float2(0.f, -1.f); // l < 0 marks an unusable partial
        return;
    }
    volatile int *abort_flag = &s_abort;

    if (warp == kNC) {
        // ------------------------------------------------ producer warp
        if (lane == 0) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            int issued = 0;
            for (int u = 0; u < nunits; ++u) {
                const int st = u % Ly::NST;
                if (u >= Ly::NST &&
                    !mbar_wait(b_empty(st), ((u / Ly::NST) - 1) & 1, abort_flag, err))
                    break;
                const int y = hk * block_size + (t0 + u * kUnit) % block_size;
                const uint32_t dst = base_s + st * Ly::STAGE;
                mbar_arrive_expect_tx(b_full(st), Ly::STAGE);
#pragma unroll
                for (int p = 0; p < Ly::PANELS; ++p) {
                    tma_load_3d(dst + p * Ly::PANEL_BYTES, &tm_k, b_full(st), p * 64, y,
                                blk_ids[u]);
                    tma_load_3d(dst + Ly::HALF + p * Ly::PANEL_BYTES, &tm_v, b_full(st), p * 64,
                                y, blk_ids[u]);
                }
                issued = u + 1;
            }
            if (*abort_flag) {
                // let copies already in flight land before the CTA exits
                for (int u = max(0, issued - Ly::NST); u < issued; ++u)
                    mbar_wait_drain(b_full(u % Ly::NST), (u / Ly::NST) & 1);
            }
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    const int g = lane >> 2, t = lane & 3;
    const int mj = lane >> 3, mr = lane & 7; // ldmatrix: matrix index, row
    const uint32_t q_lane = sQ + (mr + (mj & 1) * 8) * Ly::QROW + (mj >> 1) * 16;
    const int k_tok = mr + (mj >> 1) * 8; // K rows: matrices {t0-7,d0-7},{t0-7,d8-15},{t8-15,..}
    const int v_tok = mr + (mj & 1) * 8;  // V rows: matrices {t0-7,d0-7},{t8-15,d0-7},{t0-7,d8-15},..
    const bool split_p = len < kSplitKeys;

    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
        o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    bool ok = true;

    for (int u = warp; u < nunits; u += kNC) {
        const int st = u % Ly::NST;
        if (!mbar_wait(b_full(st), (u / Ly::NST) & 1, abort_flag, err)) {
            ok = false;
            break;
        }
        const uint32_t Ks = base_s + st * Ly::STAGE;
        const uint32_t Vs = Ks + Ly::HALF;
        const int nvalid = min(kUnit, t1 - (t0 + u * kUnit));
        if (nvalid < kUnit) {
            // V rows past the sequence end get p = 0; zero them so that stale
            // non-finite cache contents cannot reach u through 0 * x
            uint8_t *vg = base + (Vs - base_s);
            const int nz = (kUnit - nvalid) * 8; // 16-byte chunks per panel
            for (int i = lane; i < Ly::PANELS * nz; i += 32) {
                const int p = i / nz, r = nvalid + (i % nz) / 8, ch = i % 8;
                *reinterpret_cast<uint4 *>(vg + p * Ly::PANEL_BYTES + r * 128 + ch * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
        }

        // S = q K^T: 16 rows x 16 tokens as two 8-token column tiles
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kc = 0; kc < D / 16; ++kc) {
            uint32_t a[4], b[4];
            ldsm_x4(a, q_lane + kc * 32);
            const int dcol = kc * 16 + (mj & 1) * 8;
            ldsm_x4(b, Ks + (dcol >> 6) * Ly::PANEL_BYTES + k_tok * 128 +
                           ((((dcol & 63) >> 3) ^ (k_tok & 7)) << 4));
            mma16816<BF16>(s0, a, b[0], b[1]);
            mma16816<BF16>(s1, a, b[2], b[3]);
        }
        // log2-domain scores; row g: tokens 2t, 2t+1, 8+2t, 9+2t; row g+8 the same
        float sc[8] = {s0[0] * c, s0[1] * c, s1[0] * c, s1[1] * c,
                       s0[2] * c, s0[3] * c, s1[2] * c, s1[3] * c};
        if (nvalid < kUnit) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tok = (i >> 1) * 8 + 2 * t + (i & 1);
                if (tok >= nvalid)
                    sc[i] = sc[4 + i] = -INFINITY;
            }
        }
        float mx[2] = {max4(sc[0], sc[1], sc[2], sc[3]), max4(sc[4], sc[5], sc[6], sc[7])};
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        }
        float alpha[2], neg[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            float mu = m[r];
            if (mx[r] > m[r] + kRescaleThreshold || m[r] == -INFINITY)
                mu = fmaxf(mx[r], m[r]);
            alpha[r] = (mu == m[r]) ? 1.0f : ((m[r] == -INFINITY) ? 0.f : ex2(m[r] - mu));
            neg[r] = (mu == -INFINITY) ? 0.f : -mu;
            m[r] = mu;
        }
        float p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            p[i] = ex2(sc[i] + neg[i >> 2]);
        l[0] = l[0] * alpha[0] + ((p[0] + p[1]) + (p[2] + p[3]));
        l[1] = l[1] * alpha[1] + ((p[4] + p[5]) + (p[6] + p[7]));
        if (__any_sync(0xffffffffu, alpha[0] != 1.0f || alpha[1] != 1.0f)) {
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
                o[n][0] *= alpha[0];
                o[n][1] *= alpha[0];
                o[n][2] *= alpha[1];
                o[n][3] *= alpha[1];
            }
        }
        // P as the A operand: {(g, 2t..), (g+8, 2t..), (g, 8+2t..), (g+8, 8+2t..)}
        uint32_t pa[4] = {pack2<BF16>(p[0], p[1]), pack2<BF16>(p[4], p[5]),
                          pack2<BF16>(p[2], p[3]), pack2<BF16>(p[6], p[7])};
        uint32_t pl[4];
        if (split_p) {
            // rounding residual of the 16-bit P, multiplied in as a second
            // product so that short sequences do not see P's rounding
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int lo_i = (i & 1) * 4 + (i >> 1) * 2;
                pl[i] = pack2<BF16>(p[lo_i] - lo16<BF16>(pa[i]), p[lo_i + 1] - hi16<BF16>(pa[i]));
            }
        }
        // u += P V: V^T fragments by transposed ldmatrix, two d-tiles per load
#pragma unroll
        for (int np = 0; np < D / 16; ++np) {
            uint32_t b[4];
            const int dcol = np * 16 + (mj >> 1) * 8;
            ldsm_x4_t(b, Vs + (dcol >> 6) * Ly::PANEL_BYTES + v_tok * 128 +
                             ((((dcol & 63) >> 3) ^ (v_tok & 7)) << 4));
            mma16816<BF16>(o[2 * np], pa, b[0], b[1]);
            mma16816<BF16>(o[2 * np + 1], pa, b[2], b[3]);
            if (split_p) {
                mma16816<BF16>(o[2 * np], pl, b[0], b[1]);
                mma16816<BF16>(o[2 * np + 1], pl, b[2], b[3]);
            }
        }
        __syncwarp();
        if (nvalid < kUnit)
            fence_proxy_async_smem(); // the zeroing stores precede the next copy into this stage
        if (lane == 0)
            mbar_arrive(b_empty(st));
    }
    // the four lanes of a quad hold partial row sums of the same rows
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
        l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
    }
    if (!ok)
        s_flag = 2;

    // ---- merge the consumer warps' states (the ring is drained: every
    // issued unit was consumed before its consumer reached this barrier)
    asm volatile("bar.sync 1, %0;" ::"r"(kNC * 32) : "memory");
    float *mrg_u = reinterpret_cast<float *>(base);                      // [kNC][16][D]
    float2 *mrg_ml = reinterpret_cast<float2 *>(base + Ly::MERGE_U);     // [kNC][16]
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
        const int col = n * 8 + 2 * t;
        if (g < G)
            *reinterpret_cast<float2 *>(mrg_u + (warp * 16 + g) * D + col) =
                make_float2(o[n][0], o[n][1]);
        if (g + 8 < G)
            *reinterpret_cast<float2 *>(mrg_u + (warp * 16 + g + 8) * D + col) =
                make_float2(o[n][2], o[n][3]);
    }
    if (t == 0) {
        mrg_ml[warp * 16 + g] = make_float2(m[0], l[0]);
        mrg_ml[warp * 16 + g + 8] = make_float2(m[1], l[1]);
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kNC * 32) : "memory");
    const bool bad = s_flag != 0;
    for (int idx = threadIdx.x; idx < G * D; idx += kNC * 32) {
        const int r = idx / D, e = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kNC; ++w)
            M = fmaxf(M, mrg_ml[w * 16 + r].x);
        float Lsum = 0.f, U = 0.f;
#pragma unroll
        for (int w = 0; w < kNC; ++w) {
            const float2 ml = mrg_ml[w * 16 + r];
            const float sc = (ml.x == -INFINITY) ? 0.f : ex2(ml.x - M);
            Lsum += sc * ml.y;
            U += sc * mrg_u[(w * 16 + r) * D + e];
        }
        const size_t o_idx = (static_cast<size_t>(s) * Hq + head0 + r) * max_splits + split;
        ws_u[o_idx * D + e] = U;
        if (e == 0)
            ws_ml[o_idx] = bad ? make_float2(0.f, -1.f) : make_float2(M, Lsum);
    }
}

} // namespace dm

// ------------------------------------------------------------------ host

// Tokens per split: a function of max_seq_len only, so that the workspace
// size can be computed without the other arguments.
int decode_tokens_per_split(int max_seq_len) {
    int t = 256;
    while (t < 2048 && t * 32 < max_seq_len)
        t *= 2;
    return t;
}

int decode_max_splits(int max_seq_len) {
    const int tps = decode_tokens_per_split(max_seq_len);
    return max(1, (max_seq_len + tps - 1) / tps);
}

size_t decode_workspace_bytes(int num_seqs, int Hq, int d, int max_seq_len) {
    const size_t n = static_cast<size_t>(num_seqs) * Hq * decode_max_splits(max_seq_len);
    size_t ml = n * sizeof(float2);
    ml = (ml + 255) & ~static_cast<size_t>(255);
    return ml + n * d * sizeof(float);
}

template <int D, int HPW, bool BF16, bool KV8>
static cudaError_t launch_split(const DecodeArgs &a, float2 *ws_ml, float *ws_u, int tps,
                                int max_splits, cudaStream_t st) {
    using Ly = dec::Layout<D, KV8>;
    const int G = a.Hq / a.Hkv;
    const int nhg = G / HPW;
    const int hg_cta = nhg < dec::kCW ? nhg : dec::kCW;
    const int n_chunks = (nhg + hg_cta - 1) / hg_cta;
    const size_t smem = Ly::NST * 2 * Ly::UNIT_BYTES +
                        dec::kCW * (HPW * dec::kUnit + 4 * HPW) * sizeof(float) +
                        dec::kMaxUnits * sizeof(int32_t) + 2 * Ly::NST * sizeof(uint64_t) + 64;
    const size_t merge = dec::kCW * HPW * (2 + D) * sizeof(float);
    const size_t smem_total = smem > merge + 64 ? smem : merge + 64;
    auto kern = dec::decode_split_kernel<D, HPW, BF16, KV8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_total));
    if (e != cudaSuccess)
        return e;
    dim3 grid(max_splits, a.Hkv * n_chunks, a.num_seqs);
    kern<<<grid, dec::kThreads, smem_total, st>>>(
        a.q, static_cast<const uint8_t *>(a.Kc), static_cast<const uint8_t *>(a.Vc),
        a.block_table, a.seq_lens, a.k_scale, a.v_scale, ws_ml, ws_u, a.Hq, a.Hkv, G, nhg, hg_cta,
        n_chunks, a.block_size, a.max_blocks, a.num_blocks, a.max_seq_len, tps, max_splits,
        a.scale * 1.4426950408889634f, a.err);
    return cudaGetLastError();
}

template <int D, bool BF16, bool KV8>
static cudaError_t dispatch_hpw(const DecodeArgs &a, float2 *ws_ml, float *ws_u, int tps,
                                int max_splits, cudaStream_t st) {
    const int G = a.Hq / a.Hkv;
    constexpr int HMAX = 512 / D;
    int hpw = 1;
    while (hpw * 2 <= HMAX && G % (hpw * 2) == 0)
        hpw *= 2;
    switch (hpw) {
    case 1: return launch_split<D, 1, BF16, KV8>(a, ws_ml, ws_u, tps, max_splits, st);
    case 2: return launch_split<D, 2, BF16, KV8>(a, ws_ml, ws_u, tps, max_splits, st);
    case 4:
        if constexpr (HMAX >= 4)
            return launch_split<D, 4, BF16, KV8>(a, ws_ml, ws_u, tps, max_splits, st);
        break;
    case 8:
        if constexpr (HMAX >= 8)
            return launch_split<D, 8, BF16, KV8>(a, ws_ml, ws_u, tps, max_splits, st);
        break;
    }
    return cudaErrorInvalidValue;
}

template <int D, typename OutT>
static cudaError_t launch_combine(const DecodeArgs &a, const float2 *ws_ml, const float *ws_u,
                                  int tps, int max_splits, cudaStream_t st) {
    dec::decode_combine_kernel<D, OutT><<<a.num_seqs * a.Hq, D, 0, st>>>(
        ws_ml, ws_u, a.seq_lens, static_cast<OutT *>(a.O), a.lse, a.Hq, a.block_size,
        a.max_blocks, a.max_seq_len, tps, max_splits);
    return cudaGetLastError();
}

template <int D, bool BF16>
static cudaError_t launch_mma(const DecodeArgs &a, float2 *ws_ml, float *ws_u, int tps,
                              int max_splits, cudaStream_t st) {
    using Ly = dm::Lay<D>;
    // cache [num_blocks, Hkv, block_size, D] viewed as {D, Hkv * block_size, num_blocks}
    const uint64_t dims[3] = {static_cast<uint64_t>(D),
                              static_cast<uint64_t>(a.Hkv) * a.block_size,
                              static_cast<uint64_t>(a.num_blocks)};
    const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2,
                                 static_cast<uint64_t>(a.Hkv) * a.block_size * D * 2};
    const uint32_t box[3] = {64, static_cast<uint32_t>(dm::kUnit), 1};
    CUtensorMap mk, mv;
    if (!make_tmap_3d_16bit(&mk, a.Kc, BF16, dims, strides, box) ||
        !make_tmap_3d_16bit(&mv, a.Vc, BF16, dims, strides, box))
        return cudaErrorInvalidValue;
    auto kern = dm::decode_mma_kernel<D, BF16>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::SMEM);
    if (e != cudaSuccess)
        return e;
    dim3 grid(max_splits, a.Hkv, a.num_seqs);
    kern<<<grid, dm::kThreads, Ly::SMEM, st>>>(
        mk, mv, a.q, a.block_table, a.seq_lens, ws_ml, ws_u, a.Hq, a.Hq / a.Hkv, a.block_size,
        a.max_blocks, a.num_blocks, a.max_seq_len, tps, max_splits,
        a.scale * 1.4426950408889634f, a.err);
    return cudaGetLastError();
}

template <int D>
static cudaError_t decode_d(const DecodeArgs &a, cudaStream_t st) {
    const int tps = decode_tokens_per_split(a.max_seq_len);
    const int max_splits = decode_max_splits(a.max_seq_len);
    const size_t n = static_cast<size_t>(a.num_seqs) * a.Hq * max_splits;
    size_t ml_bytes = (n * sizeof(float2) + 255) & ~static_cast<size_t>(255);
    float2 *ws_ml = static_cast<float2 *>(a.workspace);
    float *ws_u = reinterpret_cast<float *>(static_cast<uint8_t *>(a.workspace) + ml_bytes);
    cudaError_t e;
    if (a.kv_e4m3)
        e = dispatch_hpw<D, true, true>(a, ws_ml, ws_u, tps, max_splits, st);
    else if (a.q_bf16)
        e = launch_mma<D, true>(a, ws_ml, ws_u, tps, max_splits, st);
    else
        e = launch_mma<D, false>(a, ws_ml, ws_u, tps, max_splits, st);
    if (e != cudaSuccess)
        return e;
    switch (a.out_dtype) {
    case 0: return launch_combine<D, __half>(a, ws_ml, ws_u, tps, max_splits, st);
    case 1: return launch_combine<D, __nv_bfloat16>(a, ws_ml, ws_u, tps, max_splits, st);
    default: return launch_combine<D, float>(a, ws_ml, ws_u, tps, max_splits, st);
    }
}

cudaError_t decode_launch(const DecodeArgs &a, cudaStream_t st) {
    switch (a.d) {
    case 64: return decode_d<64>(a, st);
    case 128: return decode_d<128>(a, st);
    case 256: return decode_d<256>(a, st);
    }
    return cudaErrorInvalidValue;
}

} // namespace attn
