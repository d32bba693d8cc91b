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
        e = dispatch_hpw<D, true, false>(a, ws_ml, ws_u, tps, max_splits, st);
    else
        e = dispatch_hpw<D, false, false>(a, ws_ml, ws_u, tps, max_splits, st);
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
