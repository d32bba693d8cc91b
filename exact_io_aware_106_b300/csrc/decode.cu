// decode.cu -- single-token attention over a block-paged KV cache.
//
// The method (auturnal.com "From attention to IO-aware execution" §8): one
// query row per head against every cached key, with the running max m,
// denominator l and un-normalised sum u of the online softmax, rescaled by
// 2^(m - m') when a block raises the max.  Decode is bound by HBM bandwidth
// (code-journey.com, "Attention co-design", prefill vs decode: GEMM-M is the
// group size G), so the kernel is built to stream every K/V byte once at
// full bandwidth.  The cache is block-paged (papanda925.com, block-wise KV
// cache): token t of sequence s sits in slot t % block_size of physical
// block block_table[s][t / block_size], layout [num_blocks, Hkv, block, d].
//
// Split-KV: one CTA per (split of tps tokens, KV head hk, sequence s).  The
// G <= 16 query heads of the group are the rows of one 16-row warp-level
// MMA tile (mma.sync m16n8k16, rows G..15 zero; with several new tokens per
// sequence the G x n_new rows fill as many 16-row tiles as needed, one CTA
// each), so a 16-token unit costs
// D/8 MMAs for S = q K^T and D/8 (2 D/8 with the P residual) for u += P V
// instead of ~2 G 16 D scalar FMAs: the consumer warps stay far ahead of
// HBM.  A producer warp streams 16-token units of K and V by TMA into a
// ring of swizzled shared-memory stages; consumer warp w takes units w,
// w + 4, ... with its own (m, l, u), and the four states are merged at the
// end of the split.  A second kernel merges the splits of a sequence with
// the same alignment rule and writes O = u / l and the log-sum-exp.
//
// 16-bit caches: the MMA runs in the cache's format; K fragments by
// ldmatrix, V^T fragments by transposed ldmatrix, both from 128-byte-swizzled
// stages.  E4M3 caches: K and V stay 8-bit in shared memory and are widened
// to f16 in registers (cvt.rn.f16x2.e4m3x2).  For q K^T each lane's ldmatrix
// word holds 4 consecutive d of one token, so the MMA's k index is permuted
// within each 16-element chunk (k = 2t, 2t+1, 2t+8, 2t+9 <-> d = 4t .. 4t+3)
// and q is laid out in shared memory in the same permuted fragment order,
// converted to f16 with one power-of-two scale per CTA.  For P V a transposed
// ldmatrix of byte pairs gives tokens (2t, 2t+1) x d (2g, 2g+1); a byte
// permute splits it into an even-d and an odd-d fragment, so each lane ends
// up owning 4 consecutive output columns.  The per-head scales fold into the
// score scale (k) and the partial (v).
//
// Scores are in the log2 domain (c = scale * log2 e).  u / l does not depend
// on the reference max subtracted (the max-subtraction invariance of §8), so
// it is kept stale: it moves only when a unit's max exceeds it by more than
// 8.  With E4M3 caches a unit's p is first taken against it and kept while
// no lane's partial row sum exceeds 2^15 (so no p does), and the row max is
// formed only for a row's first unit and when that test fails.
#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace attn {

namespace dec {

template <int D, typename OutT>
__global__ void __launch_bounds__(D)
    decode_combine_kernel(const float2 *__restrict__ ws_ml, const float *__restrict__ ws_u,
                          const int32_t *__restrict__ seq_lens, OutT *__restrict__ O,
                          float *__restrict__ lse, int Hq, int T, int block_size,
                          int max_blocks, int max_seq_len, int tps, int max_splits) {
    // the split kernel's partials are complete and visible past this point
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int sh = blockIdx.x; // (sequence, query head, new token)
    const int s = sh / (Hq * T);
    const int e = threadIdx.x;
    const int len = seq_lens[s];
    const bool len_ok = len >= (T > 1 ? T : 0) && len <= max_seq_len &&
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

namespace dm {

constexpr int kUnit = 16;       // tokens per unit (one TMA box row count)
constexpr int kNC = 4;          // consumer warps
constexpr int kThreads = (kNC + 1) * 32;
constexpr int kMaxUnits = 256;  // units per CTA (tps <= 4096)
constexpr int kSplitKeys = 512; // sequences shorter than this carry the P residual
constexpr float kRescaleThreshold = 8.0f;
constexpr float kSumLimit = 32768.0f; // keeps every kept p inside the f16 range

// resident CTAs per SM.  A CTA serves NRT x NG 16-row tiles: its kNC
// consumer warps form NG groups of kNC / NG, each group takes NRT tiles and
// every warp keeps NRT tiles' accumulators (NRT = 2 at head size 64 only,
// where they fit; NG = 2 at head sizes 128 and 256, where the two groups
// share each K/V copy instead)
template <int D, int NRT = 1, int NG = 1>
constexpr int min_ctas() {
    static_assert(NRT == 1 || D == 64, "two row tiles per warp at head size 64 only");
    static_assert(NG == 1 || (D >= 128 && NRT == 1), "two consumer groups at head size >= 128");
    return NRT == 1 ? (D == 64 ? 4 : (D == 128 ? 3 : 2)) : 3;
}

template <int D, bool KV8, int NRT = 1, int NG = 1>
struct Lay {
    static constexpr int GW = kNC / NG;  // consumer warps per group
    static constexpr int NTC = NRT * NG; // row tiles per CTA
    static constexpr int ROWB = KV8 ? D : 2 * D;          // bytes of one cache row
    static constexpr int PW = ROWB < 128 ? ROWB : 128;     // row bytes per panel = swizzle span
    static constexpr int PANELS = ROWB / PW;
    static constexpr int PANEL_BYTES = kUnit * PW;         // one TMA box
    static constexpr int HALF = PANELS * PANEL_BYTES;      // K (or V) of one unit
    static constexpr int STAGE = 2 * HALF;
    // Unit u lives in stage u % NST and is consumed by warp u % GW of every
    // group.  With NST a multiple of GW a stage is only ever consumed by the
    // same warp of each group, so that warp has itself waited for the
    // stage's previous phase before it waits (by parity) for the next one;
    // otherwise a warp could wait on a stage whose previous fill, for another
    // warp, has not landed yet, and the parity test would pass one phase
    // early.
    static constexpr int NST = KV8 ? (D == 64 ? 24 : (D == 128 ? 16 : 8))
                                   : (D == 64 ? 12 : (D == 128 ? 8 : 4));
    static_assert(NST % GW == 0, "each stage must belong to one consumer warp per group");
    // producer lanes issuing copies side by side: four for units up to 8 KB,
    // one for 16 KB units (16-bit caches at d = 256), which one lane keeps
    // up with and which four lanes slowed down
    static constexpr int ISSUE_LANES = STAGE >= 16384 ? 1 : 4;
    static_assert(NST % ISSUE_LANES == 0, "each stage must belong to one producer lane");
    static constexpr int MIN_CTAS = min_ctas<D, NRT, NG>();
    static constexpr int QROW = 2 * D + 16;                // padded q row (16-bit caches)
    static constexpr int QBYTES1 = KV8 ? (D / 16) * 32 * 16 : 16 * QROW; // one row tile
    static constexpr int QBYTES = NTC * QBYTES1;
    static constexpr int RING = NST * STAGE;
    static constexpr int MERGE_U = GW * 16 * D * 4;
    static constexpr int MERGE = MERGE_U + GW * 16 * 8; // one group's merge area
    static constexpr int OFF_Q = RING > NG * MERGE ? RING : NG * MERGE;
    static constexpr int OFF_BLK = OFF_Q + QBYTES;
    static constexpr int OFF_BAR = OFF_BLK + kMaxUnits * 4;
    static constexpr int SMEM = OFF_BAR + 2 * NST * 8 + 16 + 1024; // + alignment slack
};

// Byte offset of 16-byte chunk `ch` of row `row` inside a TMA-swizzled panel
// whose rows are PW bytes (128: chunk ^= row mod 8; 64: chunk ^= row/2 mod 4).
template <int PW>
__device__ __forceinline__ uint32_t swz(int row, int ch) {
    if constexpr (PW == 128)
        return static_cast<uint32_t>(row * 128 + ((ch ^ (row & 7)) << 4));
    else
        return static_cast<uint32_t>(row * 64 + ((ch ^ ((row >> 1) & 3)) << 4));
}

// Shared address of logical byte column `col` (a multiple of 16) of token
// `row` in the K (or V) half of a stage.
template <int D, bool KV8>
__device__ __forceinline__ uint32_t kv_addr(uint32_t half, int row, int col) {
    using Ly = Lay<D, KV8>;
    return half + (col / Ly::PW) * Ly::PANEL_BYTES + swz<Ly::PW>(row, (col % Ly::PW) >> 4);
}

__device__ __forceinline__ float max4(float a, float b, float c, float d) {
    return fmaxf(fmaxf(a, b), fmaxf(c, d));
}

// Two E4M3 codes (low byte first) widened to f16x2, exactly.
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t v) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<unsigned short>(v & 0xFFFFu)));
    return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %1, %2;" : "=r"(r) : "r"(a), "r"(sel));
    return r;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

template <int D, bool QBF16, bool KV8, int NRT, int NG>
__global__ void __launch_bounds__(kThreads, Lay<D, KV8, NRT, NG>::MIN_CTAS)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const void *__restrict__ q_,
                      const int32_t *__restrict__ block_table,
                      const int32_t *__restrict__ seq_lens, const float *__restrict__ k_scale,
                      const float *__restrict__ v_scale, float2 *__restrict__ ws_ml,
                      float *__restrict__ ws_u, int Hq, int G, int T, int ngrp, int block_size,
                      int max_blocks,
                      int num_blocks, int max_seq_len, int tps, int max_splits, float c,
                      unsigned *err) {
    using Ly = Lay<D, KV8, NRT, NG>;
    constexpr int NTC = Ly::NTC, GW = Ly::GW;
    constexpr bool MB = KV8 ? false : QBF16; // operand format of the MMAs (bf16 or f16)
    // the combine kernel may start launching once every CTA of this grid has
    // started; it waits for this grid's completion before it reads anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
    __shared__ int s_amax[NTC]; // max |q| of each row tile as float bits (E4M3 caches)

    // x = (split, group of NTC row tiles): the groups of one split are
    // adjacent, so the K/V they all stream is read from DRAM about once
    const int split = blockIdx.x / ngrp, grp = blockIdx.x % ngrp;
    const int hk = blockIdx.y, s = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int len = seq_lens[s];
    const bool len_ok = len >= (T > 1 ? T : 0) && len <= max_seq_len &&
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
    // rows of the group: r = g * T + i for head head0 + g and new token i
    // (q [num_seqs, Hq, T, d], so a group's rows are contiguous); this CTA
    // takes the NTC 16-row tiles [row0 + 16 rt, row0 + 16 rt + 16) of them
    const int row0 = 16 * NTC * grp;
    int R[NTC]; // real rows of each tile
#pragma unroll
    for (int rt = 0; rt < NTC; ++rt)
        R[rt] = max(0, min(16, G * T - row0 - 16 * rt));
    const uint16_t *qg = static_cast<const uint16_t *>(q_) +
                         ((static_cast<size_t>(s) * Hq + head0) * T + row0) * D;

    if (threadIdx.x == 0) {
        s_flag = 0;
        s_abort = 0;
#pragma unroll
        for (int rt = 0; rt < NTC; ++rt)
            s_amax[rt] = 0;
    }
    __syncthreads();
    for (int u = threadIdx.x; u < nunits; u += kThreads) {
        const int phys =
            block_table[static_cast<size_t>(s) * max_blocks + (t0 + u * kUnit) / block_size];
        if (phys < 0 || phys >= num_blocks)
            s_flag = 1;
        blk_ids[u] = phys;
    }
    if constexpr (!KV8) {
        // the tiles' query rows, zero rows up to 16 per tile, padded rows
        for (int i = threadIdx.x; i < NTC * 16 * (D / 8); i += kThreads) {
            const int r = i / (D / 8), c8 = i % (D / 8); // r = 16 rt + row in tile
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if ((r & 15) < R[r >> 4])
                v = *reinterpret_cast<const uint4 *>(qg + static_cast<size_t>(r) * D + c8 * 8);
            *reinterpret_cast<uint4 *>(base + Ly::OFF_Q + r * Ly::QROW + c8 * 16) = v;
        }
    } else {
#pragma unroll
        for (int rt = 0; rt < NTC; ++rt) {
            float amax = 0.f;
            for (int i = threadIdx.x; i < R[rt] * D; i += kThreads) {
                const uint16_t x16 = qg[static_cast<size_t>(16 * rt) * D + i];
                const float x = QBF16 ? __uint_as_float(static_cast<uint32_t>(x16) << 16)
                                      : __half2float(__ushort_as_half(x16));
                amax = fmaxf(amax, fabsf(x));
            }
            if (amax > 0.f)
                atomicMax(&s_amax[rt], __float_as_int(amax)); // non-negative floats order as ints
        }
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < Ly::NST; ++i) {
            mbar_init(b_full(i), 1);    // producer arrive + tx bytes
            mbar_init(b_empty(i), NG);  // one consuming warp per group
        }
        fence_barrier_init();
    }
    __syncthreads();
    // power-of-two scale that keeps the f16 copy of each tile's q in range
    float qs[NTC];
#pragma unroll
    for (int rt = 0; rt < NTC; ++rt)
        qs[rt] = 1.0f;
    if constexpr (KV8) {
#pragma unroll
        for (int rt = 0; rt < NTC; ++rt) {
            const float amax = __int_as_float(s_amax[rt]);
            if (amax > 0.f && isfinite(amax))
                qs[rt] = exp2f(14.0f - floorf(log2f(amax)));
        }
        // q as f16 in the permuted fragment order: chunk ch, lane (g, t) gets
        // {(g, 4t..4t+1), (g+8, 4t..4t+1), (g, 4t+2..4t+3), (g+8, 4t+2..4t+3)}
        for (int i = threadIdx.x; i < NTC * (D / 16) * 32; i += kThreads) {
            const int rt = i / ((D / 16) * 32), ii = i % ((D / 16) * 32);
            const int ch = ii >> 5, ln = ii & 31, gg = ln >> 2, tt = ln & 3;
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {   // row gg + 8 h
#pragma unroll
                for (int k = 0; k < 2; ++k) { // elements 4t + 2k, 4t + 2k + 1
                    const int row = gg + 8 * h;
                    float x0 = 0.f, x1 = 0.f;
                    if (row < R[rt]) {
                        const int e = ch * 16 + 4 * tt + 2 * k;
                        const uint16_t *src = qg + static_cast<size_t>(16 * rt + row) * D + e;
                        x0 = QBF16 ? __uint_as_float(static_cast<uint32_t>(src[0]) << 16)
                                   : __half2float(__ushort_as_half(src[0]));
                        x1 = QBF16 ? __uint_as_float(static_cast<uint32_t>(src[1]) << 16)
                                   : __half2float(__ushort_as_half(src[1]));
                    }
                    w[2 * k + h] = pack2<false>(x0 * qs[rt], x1 * qs[rt]);
                }
            }
            *reinterpret_cast<uint4 *>(base + Ly::OFF_Q + rt * Ly::QBYTES1 + ii * 16) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
        __syncthreads();
    }
    if (s_flag) {
        if (threadIdx.x == 0)
            atomicOr(err, DERR_INDEX);
        for (int r = threadIdx.x; r < NTC * 16; r += kThreads)
            if ((r & 15) < R[r >> 4])
                ws_ml[((static_cast<size_t>(s) * Hq + head0) * T + row0 + r) * max_splits +
                      split] = make_float2(0.f, -1.f); // l < 0 marks an unusable partial
        return;
    }
    volatile int *abort_flag = &s_abort;

    if (warp == kNC) {
        // ------------------------------------------------ producer warp
        // IL lanes issue at once, lane i the units i, i + IL, ...: each unit
        // costs its lane a stage wait and an expect-tx arrival of a few hundred
        // cycles besides the copies, so with one issuing lane the cells with
        // small units (16 tokens x 64 bytes of K and of V) could not keep HBM
        // busy.  The lanes divide the stages among them (NST is a multiple of
        // IL), so each stage is refilled, waited on and drained by one lane.
        // test hook: no copies at all, so the consumers' first wait expires
        // (and they unwind: this warp has nothing in flight to drain)
        if ((*reinterpret_cast<const volatile unsigned *>(err + CTL_HOOKS) & HOOK_WITHHOLD_KV) !=
            0u)
            return;
        constexpr int IL = Ly::ISSUE_LANES;
        if (lane < IL) {
            if (lane == 0) {
                prefetch_tmap(&tm_k);
                prefetch_tmap(&tm_v);
            }
            int last = -1; // last unit this lane issued
            for (int u = lane; u < nunits; u += IL) {
                const int st = u % Ly::NST;
                if (u >= Ly::NST &&
                    !mbar_wait(b_empty(st), ((u / Ly::NST) - 1) & 1, abort_flag, err))
                    break;
                const int y = hk * block_size + (t0 + u * kUnit) % block_size;
                const uint32_t dst = base_s + st * Ly::STAGE;
                mbar_arrive_expect_tx(b_full(st), Ly::STAGE);
#pragma unroll
                for (int p = 0; p < Ly::PANELS; ++p) {
                    const int x = p * (KV8 ? Ly::PW : Ly::PW / 2); // elements
                    tma_load_3d(dst + p * Ly::PANEL_BYTES, &tm_k, b_full(st), x, y, blk_ids[u]);
                    tma_load_3d(dst + Ly::HALF + p * Ly::PANEL_BYTES, &tm_v, b_full(st), x, y,
                                blk_ids[u]);
                }
                last = u;
            }
            if (*abort_flag) {
                // let this lane's copies in flight land before the CTA exits
                for (int u = last; u >= 0 && u > last - Ly::NST; u -= IL)
                    mbar_wait_drain(b_full(u % Ly::NST), (u / Ly::NST) & 1);
            }
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    // group gi (warps GW gi .. GW gi + GW - 1) takes the row tiles
    // [NRT gi, NRT gi + NRT) of the CTA; warp wl of a group the units
    // wl, wl + GW, ...  (every group streams every unit)
    const int gi = warp / GW, wl = warp % GW, rt0 = gi * NRT;
    const int g = lane >> 2, t = lane & 3;
    const int mj = lane >> 3, mr = lane & 7; // ldmatrix: matrix index, row
    const bool split_p = len < kSplitKeys;
    float cq[NRT];
#pragma unroll
    for (int rt = 0; rt < NRT; ++rt)
        cq[rt] = KV8 ? c * k_scale[hk] / qs[rt0 + rt] : c;

    float o[NRT][D / 8][4];
    float m[NRT][2], l[NRT][2];
#pragma unroll
    for (int rt = 0; rt < NRT; ++rt) {
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
            o[rt][n][0] = o[rt][n][1] = o[rt][n][2] = o[rt][n][3] = 0.f;
        m[rt][0] = m[rt][1] = -INFINITY;
        l[rt][0] = l[rt][1] = 0.f;
    }
    bool ok = true, ref_all = false;

    for (int u = wl; u < nunits; u += GW) {
        const int st = u % Ly::NST;
        if (!mbar_wait_warp(b_full(st), (u / Ly::NST) & 1, abort_flag, err)) {
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
            constexpr int CPR = Ly::PW / 16; // 16-byte chunks per panel row
            const int nz = (kUnit - nvalid) * CPR;
            for (int i = lane; i < Ly::PANELS * nz; i += 32) {
                const int p = i / nz, r = nvalid + (i % nz) / CPR, ch = i % CPR;
                *reinterpret_cast<uint4 *>(vg + p * Ly::PANEL_BYTES + r * Ly::PW + ch * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
        }

        // S = q K^T: 16 rows x 16 tokens per tile as two 8-token column tiles;
        // every K fragment serves all NRT row tiles
        float s0[NRT][4], s1[NRT][4];
#pragma unroll
        for (int rt = 0; rt < NRT; ++rt)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                s0[rt][i] = s1[rt][i] = 0.f;
        if constexpr (!KV8) {
            // matrices {t0-7,d0-7}, {t0-7,d8-15}, {t8-15,d0-7}, {t8-15,d8-15}
            const int k_tok = mr + (mj >> 1) * 8;
            const uint32_t q_lane = sQ + (mr + (mj & 1) * 8) * Ly::QROW + (mj >> 1) * 16;
#pragma unroll
            for (int kc = 0; kc < D / 16; ++kc) {
                uint32_t b[4];
                ldsm_x4(b, kv_addr<D, KV8>(Ks, k_tok, (kc * 16 + (mj & 1) * 8) * 2));
#pragma unroll
                for (int rt = 0; rt < NRT; ++rt) {
                    uint32_t a[4];
                    ldsm_x4(a, q_lane + (rt0 + rt) * 16 * Ly::QROW + kc * 32);
                    mma16816<MB>(s0[rt], a, b[0], b[1]);
                    mma16816<MB>(s1[rt], a, b[2], b[3]);
                }
            }
        } else {
            // matrices {t0-7,c}, {t8-15,c}, {t0-7,c+1}, {t8-15,c+1} of 16-byte chunks
            const int k_tok = mr + (mj & 1) * 8;
#pragma unroll
            for (int cp = 0; cp < D / 32; ++cp) {
                uint32_t b[4];
                ldsm_x4(b, kv_addr<D, KV8>(Ks, k_tok, (2 * cp + (mj >> 1)) * 16));
                const uint32_t kb00 = e4m3x2_f16x2(b[0]), kb01 = e4m3x2_f16x2(b[0] >> 16);
                const uint32_t kb10 = e4m3x2_f16x2(b[1]), kb11 = e4m3x2_f16x2(b[1] >> 16);
                const uint32_t kb20 = e4m3x2_f16x2(b[2]), kb21 = e4m3x2_f16x2(b[2] >> 16);
                const uint32_t kb30 = e4m3x2_f16x2(b[3]), kb31 = e4m3x2_f16x2(b[3] >> 16);
#pragma unroll
                for (int rt = 0; rt < NRT; ++rt) {
                    const uint32_t qt = sQ + (rt0 + rt) * Ly::QBYTES1;
                    const uint4 q0 = lds128(qt + ((2 * cp) * 32 + lane) * 16);
                    const uint4 q1 = lds128(qt + ((2 * cp + 1) * 32 + lane) * 16);
                    const uint32_t a0[4] = {q0.x, q0.y, q0.z, q0.w};
                    const uint32_t a1[4] = {q1.x, q1.y, q1.z, q1.w};
                    mma16816<false>(s0[rt], a0, kb00, kb01);
                    mma16816<false>(s1[rt], a0, kb10, kb11);
                    mma16816<false>(s0[rt], a1, kb20, kb21);
                    mma16816<false>(s1[rt], a1, kb30, kb31);
                }
            }
        }
        uint32_t pa[NRT][4], pl[NRT][4];
#pragma unroll
        for (int rt = 0; rt < NRT; ++rt) {
            // log2-domain scores; row g: tokens 2t, 2t+1, 8+2t, 9+2t; row g+8 the same
            float sc[8] = {s0[rt][0] * cq[rt], s0[rt][1] * cq[rt], s1[rt][0] * cq[rt],
                           s1[rt][1] * cq[rt], s0[rt][2] * cq[rt], s0[rt][3] * cq[rt],
                           s1[rt][2] * cq[rt], s1[rt][3] * cq[rt]};
            if (nvalid < kUnit) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int tok = (i >> 1) * 8 + 2 * t + (i & 1);
                    if (tok >= nvalid)
                        sc[i] = sc[4 + i] = -INFINITY;
                }
            }
            if (T > 1 && t0 + u * kUnit + kUnit - 1 > len - T) {
                // new token i sees cached token p iff p <= len - T + i (bottom-right)
                const int rb = row0 + 16 * (rt0 + rt);
                const int lim0 = len - T + ((rb + g) % T), lim1 = len - T + ((rb + g + 8) % T);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int p = t0 + u * kUnit + (i >> 1) * 8 + 2 * t + (i & 1);
                    if (p > lim0)
                        sc[i] = -INFINITY;
                    if (p > lim1)
                        sc[4 + i] = -INFINITY;
                }
            }
            // E4M3 caches (bound by the consumers' instruction issue): once
            // every row of the warp has a reference max, p is taken against
            // it at once and kept while no lane's partial row sum exceeds
            // kSumLimit (each p is at most its lane's partial sum);
            // otherwise the unit is redone from the row max.  (16-bit caches,
            // near the copy bandwidth, measured no gain from it.)
            float p[8];
            float alpha[2] = {1.0f, 1.0f};
            bool kept = false;
            if (KV8 && ref_all) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    p[i] = ex2(sc[i] - m[rt][i >> 2]);
                const float ps0 = (p[0] + p[1]) + (p[2] + p[3]);
                const float ps1 = (p[4] + p[5]) + (p[6] + p[7]);
                kept = __all_sync(0xffffffffu, ps0 <= kSumLimit && ps1 <= kSumLimit);
                if (kept) {
                    l[rt][0] += ps0;
                    l[rt][1] += ps1;
                }
            }
            if (!kept) {
                float mx[2] = {max4(sc[0], sc[1], sc[2], sc[3]),
                               max4(sc[4], sc[5], sc[6], sc[7])};
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                }
                float neg[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    float mu = m[rt][r];
                    if (mx[r] > m[rt][r] + kRescaleThreshold || m[rt][r] == -INFINITY)
                        mu = fmaxf(mx[r], m[rt][r]);
                    alpha[r] = (mu == m[rt][r])
                                   ? 1.0f
                                   : ((m[rt][r] == -INFINITY) ? 0.f : ex2(m[rt][r] - mu));
                    neg[r] = (mu == -INFINITY) ? 0.f : -mu;
                    m[rt][r] = mu;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    p[i] = ex2(sc[i] + neg[i >> 2]);
                l[rt][0] = l[rt][0] * alpha[0] + ((p[0] + p[1]) + (p[2] + p[3]));
                l[rt][1] = l[rt][1] * alpha[1] + ((p[4] + p[5]) + (p[6] + p[7]));
            }
            if (!kept && __any_sync(0xffffffffu, alpha[0] != 1.0f || alpha[1] != 1.0f)) {
#pragma unroll
                for (int n = 0; n < D / 8; ++n) {
                    o[rt][n][0] *= alpha[0];
                    o[rt][n][1] *= alpha[0];
                    o[rt][n][2] *= alpha[1];
                    o[rt][n][3] *= alpha[1];
                }
            }
            // P as the A operand: {(g, 2t..), (g+8, 2t..), (g, 8+2t..), (g+8, 8+2t..)}
            pa[rt][0] = pack2<MB>(p[0], p[1]);
            pa[rt][1] = pack2<MB>(p[4], p[5]);
            pa[rt][2] = pack2<MB>(p[2], p[3]);
            pa[rt][3] = pack2<MB>(p[6], p[7]);
            if (split_p) {
                // rounding residual of the 16-bit P, multiplied in as a second
                // product so that short sequences do not see P's rounding
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int lo_i = (i & 1) * 4 + (i >> 1) * 2;
                    pl[rt][i] = pack2<MB>(p[lo_i] - lo16<MB>(pa[rt][i]),
                                          p[lo_i + 1] - hi16<MB>(pa[rt][i]));
                }
            }
        }
        // u += P V; every V fragment serves all NRT row tiles
        if constexpr (!KV8) {
            // V^T fragments by transposed ldmatrix, two d-tiles per load:
            // matrices {t0-7,d0-7}, {t8-15,d0-7}, {t0-7,d8-15}, {t8-15,d8-15}
            const int v_tok = mr + (mj & 1) * 8;
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
                uint32_t b[4];
                ldsm_x4_t(b, kv_addr<D, KV8>(Vs, v_tok, (np * 16 + (mj >> 1) * 8) * 2));
#pragma unroll
                for (int rt = 0; rt < NRT; ++rt) {
                    mma16816<MB>(o[rt][2 * np], pa[rt], b[0], b[1]);
                    mma16816<MB>(o[rt][2 * np + 1], pa[rt], b[2], b[3]);
                    if (split_p) {
                        mma16816<MB>(o[rt][2 * np], pl[rt], b[0], b[1]);
                        mma16816<MB>(o[rt][2 * np + 1], pl[rt], b[2], b[3]);
                    }
                }
            }
        } else {
            // transposed ldmatrix of byte pairs: lane (g, t) receives, per
            // 16-byte chunk c, tokens 2t, 2t+1 at d = 16c + 2g, 16c + 2g + 1;
            // byte permutes split it into the even-d and odd-d fragments
            const int v_tok = mr + (mj & 1) * 8;
#pragma unroll
            for (int cp = 0; cp < D / 32; ++cp) {
                uint32_t b[4];
                ldsm_x4_t(b, kv_addr<D, KV8>(Vs, v_tok, (2 * cp + (mj >> 1)) * 16));
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int ch = 2 * cp + h;
                    const uint32_t lo = b[2 * h], hi = b[2 * h + 1]; // tokens 0-7, 8-15
                    const uint32_t ev0 = e4m3x2_f16x2(prmt(lo, 0x0020u));
                    const uint32_t ev1 = e4m3x2_f16x2(prmt(hi, 0x0020u));
                    const uint32_t od0 = e4m3x2_f16x2(prmt(lo, 0x0031u));
                    const uint32_t od1 = e4m3x2_f16x2(prmt(hi, 0x0031u));
#pragma unroll
                    for (int rt = 0; rt < NRT; ++rt) {
                        mma16816<false>(o[rt][2 * ch], pa[rt], ev0, ev1);
                        mma16816<false>(o[rt][2 * ch + 1], pa[rt], od0, od1);
                        if (split_p) {
                            mma16816<false>(o[rt][2 * ch], pl[rt], ev0, ev1);
                            mma16816<false>(o[rt][2 * ch + 1], pl[rt], od0, od1);
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (nvalid < kUnit)
            fence_proxy_async_smem(); // the zeroing stores precede the next copy into this stage
        if (lane == 0)
            mbar_arrive(b_empty(st));
        if constexpr (KV8) {
            bool fin = true;
#pragma unroll
            for (int rt = 0; rt < NRT; ++rt)
                fin = fin && m[rt][0] != -INFINITY && m[rt][1] != -INFINITY;
            ref_all = __all_sync(0xffffffffu, fin);
        }
    }
    // the four lanes of a quad hold partial row sums of the same rows
#pragma unroll
    for (int rt = 0; rt < NRT; ++rt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            l[rt][r] += __shfl_xor_sync(0xffffffffu, l[rt][r], 1);
            l[rt][r] += __shfl_xor_sync(0xffffffffu, l[rt][r], 2);
        }
    if (!ok)
        s_flag = 2;

    // ---- merge each group's warp states, one row tile at a time, in the
    // group's own area over the ring.  The ring is drained once every
    // consumer warp of every group has reached the first barrier (every
    // issued unit was consumed before its consumers got there).
    asm volatile("bar.sync 1, %0;" ::"r"(kNC * 32) : "memory");
    float *mrg_u = reinterpret_cast<float *>(base + gi * Ly::MERGE);                  // [GW][16][D]
    float2 *mrg_ml = reinterpret_cast<float2 *>(base + gi * Ly::MERGE + Ly::MERGE_U); // [GW][16]
    const float vsc = KV8 ? v_scale[hk] : 1.0f;
    const int gtid = threadIdx.x - gi * GW * 32; // thread within the group
#pragma unroll
    for (int rt = 0; rt < NRT; ++rt) {
        if (rt > 0) // the previous tile's merge reads are done
            asm volatile("bar.sync %0, %1;" ::"r"(2 + gi), "r"(GW * 32) : "memory");
        const int Rt = R[rt0 + rt];
        if constexpr (!KV8) {
            // n-tile n, column 2t + e  <->  d = 8 n + 2 t + e
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
                const int col = n * 8 + 2 * t;
                if (g < Rt)
                    *reinterpret_cast<float2 *>(mrg_u + (wl * 16 + g) * D + col) =
                        make_float2(o[rt][n][0], o[rt][n][1]);
                if (g + 8 < Rt)
                    *reinterpret_cast<float2 *>(mrg_u + (wl * 16 + g + 8) * D + col) =
                        make_float2(o[rt][n][2], o[rt][n][3]);
            }
        } else {
            // chunk ch: even tile 2 ch holds d = 16 ch + 4t + {0, 2}, odd tile
            // 2 ch + 1 holds d = 16 ch + 4t + {1, 3}
#pragma unroll
            for (int ch = 0; ch < D / 16; ++ch) {
                const int col = ch * 16 + 4 * t;
                if (g < Rt)
                    *reinterpret_cast<float4 *>(mrg_u + (wl * 16 + g) * D + col) =
                        make_float4(o[rt][2 * ch][0], o[rt][2 * ch + 1][0], o[rt][2 * ch][1],
                                    o[rt][2 * ch + 1][1]);
                if (g + 8 < Rt)
                    *reinterpret_cast<float4 *>(mrg_u + (wl * 16 + g + 8) * D + col) =
                        make_float4(o[rt][2 * ch][2], o[rt][2 * ch + 1][2], o[rt][2 * ch][3],
                                    o[rt][2 * ch + 1][3]);
            }
        }
        if (t == 0) {
            mrg_ml[wl * 16 + g] = make_float2(m[rt][0], l[rt][0]);
            mrg_ml[wl * 16 + g + 8] = make_float2(m[rt][1], l[rt][1]);
        }
        asm volatile("bar.sync %0, %1;" ::"r"(2 + gi), "r"(GW * 32) : "memory");
        const bool bad = s_flag != 0;
        for (int idx = gtid; idx < Rt * D; idx += GW * 32) {
            const int r = idx / D, e = idx % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < GW; ++w)
                M = fmaxf(M, mrg_ml[w * 16 + r].x);
            float Lsum = 0.f, U = 0.f;
#pragma unroll
            for (int w = 0; w < GW; ++w) {
                const float2 ml = mrg_ml[w * 16 + r];
                const float sc = (ml.x == -INFINITY) ? 0.f : ex2(ml.x - M);
                Lsum += sc * ml.y;
                U += sc * mrg_u[(w * 16 + r) * D + e];
            }
            const size_t o_idx =
                ((static_cast<size_t>(s) * Hq + head0) * T + row0 + 16 * (rt0 + rt) + r) * max_splits +
                split;
            ws_u[o_idx * D + e] = U * vsc;
            if (e == 0)
                ws_ml[o_idx] = bad ? make_float2(0.f, -1.f) : make_float2(M, Lsum);
        }
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

template <int D, typename OutT>
// The combine kernel is launched as a programmatic dependent of the split
// kernel: its launch and CTA set-up overlap the split kernel's last CTAs,
// and each of its CTAs waits (griddepcontrol.wait) until the split kernel
// has finished and its partials are visible.
static cudaError_t launch_combine(const DecodeArgs &a, const float2 *ws_ml, const float *ws_u,
                                  int tps, int max_splits, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.num_seqs * a.Hq * a.T), 1, 1);
    cfg.blockDim = dim3(D, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(
        &cfg, dec::decode_combine_kernel<D, OutT>, ws_ml, ws_u, a.seq_lens,
        static_cast<OutT *>(a.O), a.lse, a.Hq, a.T, a.block_size, a.max_blocks, a.max_seq_len, tps,
        max_splits);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

// 16-row tiles of a KV head's query rows (G x n_new of them)
static int decode_row_tiles(const DecodeArgs &a) { return (a.Hq / a.Hkv * a.T + 15) / 16; }

// Row tiles per CTA: two when they pair up, so that each K/V copy serves
// both.  At head size 64 one warp takes both tiles (each K/V fragment serves
// both; MQA G = 32: 0.125 -> 0.096 ms); at 128 and 256 the doubled
// accumulators would leave room for one CTA per SM (measured slower at
// 128), so the consumer warps split into two groups of two, one per tile,
// sharing the copy (spec-decode-8 at 128: 1.127 -> 0.757 ms).
template <int D>
static int decode_tiles_per_cta(const DecodeArgs &a) {
    return decode_row_tiles(a) % 2 == 0 ? 2 : 1;
}

template <int D, bool QBF16, bool KV8, int NRT, int NG>
static cudaError_t launch_mma(const DecodeArgs &a, float2 *ws_ml, float *ws_u, int tps,
                              int max_splits, cudaStream_t st) {
    using Ly = dm::Lay<D, KV8, NRT, NG>;
    // cache [num_blocks, Hkv, block_size, D] viewed as {D, Hkv * block_size, num_blocks}
    const uint64_t esz = KV8 ? 1 : 2;
    const uint64_t dims[3] = {static_cast<uint64_t>(D),
                              static_cast<uint64_t>(a.Hkv) * a.block_size,
                              static_cast<uint64_t>(a.num_blocks)};
    const uint64_t strides[2] = {D * esz, static_cast<uint64_t>(a.Hkv) * a.block_size * D * esz};
    const uint32_t box[3] = {static_cast<uint32_t>(Ly::PW / esz),
                             static_cast<uint32_t>(dm::kUnit), 1};
    const TmapElem el = KV8 ? TmapElem::U8 : (QBF16 ? TmapElem::BF16 : TmapElem::F16);
    CUtensorMap mk, mv;
    if (!make_tmap_3d(&mk, a.Kc, el, dims, strides, box, Ly::PW) ||
        !make_tmap_3d(&mv, a.Vc, el, dims, strides, box, Ly::PW))
        return cudaErrorInvalidValue;
    auto kern = dm::decode_mma_kernel<D, QBF16, KV8, NRT, NG>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::SMEM);
    if (e != cudaSuccess)
        return e;
    const int ngrp = decode_row_tiles(a) / Ly::NTC; // CTAs per (split, KV head, sequence)
    dim3 grid(max_splits * ngrp, a.Hkv, a.num_seqs);
    kern<<<grid, dm::kThreads, Ly::SMEM, st>>>(
        mk, mv, a.q, a.block_table, a.seq_lens, a.k_scale, a.v_scale, ws_ml, ws_u, a.Hq,
        a.Hq / a.Hkv, a.T, ngrp, a.block_size, a.max_blocks, a.num_blocks, a.max_seq_len, tps,
        max_splits, a.scale * 1.4426950408889634f, a.err);
    return cudaGetLastError();
}

// Tokens per split for one call: at least the workspace's split length (so
// the partials fit), doubled while the grid still has at least `waves` waves
// of CTAs -- longer splits amortise each CTA's set-up and merge.
static int choose_tps(const DecodeArgs &a, int resident_per_sm, int tiles_per_cta, int waves) {
    int tps = decode_tokens_per_split(a.max_seq_len);
    const long long pairs = static_cast<long long>(a.num_seqs) * a.Hkv *
                            (decode_row_tiles(a) / tiles_per_cta); // CTAs per split
    const long long slots = static_cast<long long>(sm_count()) * resident_per_sm;
    while (tps < 2048) {
        const long long splits = (a.max_seq_len + 2LL * tps - 1) / (2LL * tps);
        if (pairs * splits < waves * slots)
            break;
        tps *= 2;
    }
    return tps;
}

template <int D>
static cudaError_t decode_d(const DecodeArgs &a, cudaStream_t st) {
    const int ntc = decode_tiles_per_cta<D>(a);
    int resident = dm::min_ctas<D, 1>();
    if constexpr (D == 64)
        resident = ntc == 2 ? dm::min_ctas<D, 2, 1>() : resident;
    if constexpr (D >= 128)
        resident = ntc == 2 ? dm::min_ctas<D, 1, 2>() : resident;
    // Wave target: the calls with the fewest bytes per CTA (head size 64,
    // E4M3 at 256) gain from longer splits -- one wave: d = 64 cells 6-22%
    // faster, d = 256 E4M3 up to 8% -- where 16-bit d = 128 loses 5-7%.
    const int waves = (D == 64 || (D == 256 && a.kv_e4m3)) ? 1 : 4;
    const int tps = choose_tps(a, resident, ntc, waves);
    const int max_splits = max(1, (a.max_seq_len + tps - 1) / tps);
    const size_t n = static_cast<size_t>(a.num_seqs) * a.Hq * a.T * max_splits;
    size_t ml_bytes = (n * sizeof(float2) + 255) & ~static_cast<size_t>(255);
    float2 *ws_ml = static_cast<float2 *>(a.workspace);
    float *ws_u = reinterpret_cast<float *>(static_cast<uint8_t *>(a.workspace) + ml_bytes);
    cudaError_t e;
    auto run = [&](auto nrt_c, auto ng_c) -> cudaError_t {
        constexpr int NRT = decltype(nrt_c)::value, NG = decltype(ng_c)::value;
        if (a.kv_e4m3)
            return a.q_bf16
                       ? launch_mma<D, true, true, NRT, NG>(a, ws_ml, ws_u, tps, max_splits, st)
                       : launch_mma<D, false, true, NRT, NG>(a, ws_ml, ws_u, tps, max_splits, st);
        return a.q_bf16
                   ? launch_mma<D, true, false, NRT, NG>(a, ws_ml, ws_u, tps, max_splits, st)
                   : launch_mma<D, false, false, NRT, NG>(a, ws_ml, ws_u, tps, max_splits, st);
    };
    using I1 = std::integral_constant<int, 1>;
    using I2 = std::integral_constant<int, 2>;
    if constexpr (D == 64)
        e = ntc == 2 ? run(I2{}, I1{}) : run(I1{}, I1{});
    else
        e = ntc == 2 ? run(I1{}, I2{}) : run(I1{}, I1{});
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
