// backward_sm103.cu -- gradients of exact attention on sm_103a tensor cores.
//
// The method (marketmaker.cc "Flash Attention and sequence length",
// "Rückwärtsdurchlauf"): nothing n x n is kept from the forward pass; the
// probabilities are recomputed block by block from Q, K and the stored row
// statistic lse = ln sum_j exp(s_ij):  P = exp(s - lse).  With dO the
// upstream gradient,
//   dV = P^T dO,   dP = dO V^T,   D_i = sum_c dO_ic O_ic  (= sum_j P_ij dP_ij),
//   dS = P * (dP - D),   dQ = scale dS K,   dK = scale dS^T Q,
// and dK, dV of a KV head summed over the G query heads that read it
// (code-journey.com "Attention co-design", Group Size).
//
// Three kernels, no atomics (every gradient element has one writer):
//   bwd_prep_kernel   D = rowsum(dO * O), one warp per row.
//   bwd_kv_kernel     one CTA per (b, KV head, 128-key block): K and V stay
//                     in shared memory; for every query head of the group
//                     and every query block that sees the keys,
//                       S^T = K Q^T, dP^T = V dO^T        (tcgen05, TMEM)
//                       P^T, dS^T                          (8 warps, two per key row)
//                       dV += P^T dO, dK += dS^T Q         (tcgen05, A = TMEM)
//   bwd_q_kernel      one CTA per (b, head, 128-row query block): for every
//                     key block it sees, S = Q K^T, dP = dO V^T, dS, and
//                     dQ += dS K.
// Every score product is a full 128 x 128 block (N = 128: a tcgen05.mma with
// N = 64 runs at two thirds of the tensor core's rate).  Per step t the
// tensor core runs, in order: dP(t), S(t+1), the second products of
// softmax half 0 of step t, those of half 1, then dP(t+1).  The softmax
// warps load S(t+1) into registers as soon as it lands (freeing its columns
// for S(t+2)) and take its exponentials while prod1(t) and dP(t+1) run;
// they form half 0's dS while S(t+2) runs and half 1's while half 0's
// products run, so the tensor core does not wait on them.
// P and dS enter the second products in the inputs' 16-bit format; the
// accumulators are fp32 in tensor memory.  Scores are in the log2 domain:
// p = 2^(s c - lse log2 e), c = scale log2 e.
#include "common.cuh"
#include "launch.h"

namespace attn {

namespace bw {

constexpr int BT = 128; // rows of a key block and of a query block
constexpr int HS = 64;  // columns of a softmax half (queries for dK/dV, keys for dQ)
constexpr int kSoftmaxWarps = 8; // two per TMEM lane quarter
constexpr int kThreads = 32 * kSoftmaxWarps + 64;
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kMmaWarp = kSoftmaxWarps + 1;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct Cfg {
    static constexpr int TILE = BT * D * 2;          // one 128-row 16-bit tile
    static constexpr int PANELS = D / 64;
    // Two streamed tiles per step, each in its own ring: X feeds the step's
    // score product (Q for dK/dV, K for dQ), Y the second product (dO, V).
    // S(t+1) is issued right after dP(t), so X is the ring that needs depth.
    static constexpr int NX = D == 128 ? 3 : 4;
    static constexpr int NY = D == 128 ? 2 : 4;
    static constexpr int OFF_A = 0;                  // resident tile pair (K,V or Q,dO)
    static constexpr int OFF_X = OFF_A + 2 * TILE;
    static constexpr int OFF_Y = OFF_X + NX * TILE;
    static constexpr int OFF_ROW = OFF_Y + NY * TILE; // -lse2 / -D of 128 rows, 2 buffers
    static constexpr int OFF_BAR = OFF_ROW + 2 * 2 * BT * 4;
    // the dK/dV kernel releases a step's X and Y stages together, on one
    // barrier per step modulo NU (a common multiple of the ring depths)
    static constexpr int NU = D == 128 ? 6 : 4;
    static_assert(NU % NX == 0 && NU % NY == 0, "NU must be a multiple of both ring depths");
    // afull, xfull/xempty[NX], yfull/yempty[NY], sready, dpready, sfree,
    // pready[2], done, drain, used[NU]
    static constexpr int NBAR = 1 + 2 * NX + 2 * NY + 3 + 2 + 2 + NU;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_USED = OFF_MISC + 64;  // from the 1024-aligned base
    // room to align the base; at d = 128 the rings leave less than 1024
    // bytes, and a kernel whose base needs more padding reports DERR_INDEX
    static constexpr int SMEM = SMEM_USED + 1024 < 227 * 1024 ? SMEM_USED + 1024 : 227 * 1024;
    // a step's 128 x 128 scores at S_COL, the second product at DP_COL.
    // The softmax warps load all their score columns at once (which frees
    // them for the next step's scores) and write their 16-bit results (two
    // per column) over the dP columns they have read.
    static constexpr int S_COL = 0, DP_COL = BT;
    static constexpr int ACC0 = 2 * BT, ACC1 = 2 * BT + D;
    static_assert(2 * BT + 2 * D <= 512, "tensor memory budget");
    static_assert(SMEM_USED + 128 <= SMEM, "shared memory budget");
};

struct Shape {
    int B, Hq, Hkv, G, n_q, n_kv, causal, nqb, nkb;
    float c, scale;
};

// D_i = sum_c dO_ic O_ic (fp32); O in the inputs' 16-bit format or in fp32
// (OF32).  Each thread takes 8 elements of a row with 16-byte loads (D / 8
// lanes per row), and each warp PREP_UNROLL groups of 32 / (D / 8) rows, all
// loads issued before the arithmetic so that several are in flight.
constexpr int PREP_UNROLL = 4;
template <int D>
constexpr long long prep_rows_per_block() {
    return 8LL * (32 / (D / 8)) * PREP_UNROLL; // 8 warps per 256-thread block
}
template <int D, bool BF16, bool OF32>
__global__ void __launch_bounds__(256)
    bwd_prep_kernel(const void *__restrict__ O_, const uint16_t *__restrict__ dO,
                    float *__restrict__ Drow, long long rows) {
    constexpr int LPR = D / 8;   // lanes per row
    constexpr int RPW = 32 / LPR; // rows per warp and group
    const int lane = threadIdx.x & 31, sub = lane / LPR, c = lane % LPR;
    const long long r0 = (static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * RPW *
                         PREP_UNROLL;
    uint4 g[PREP_UNROLL], o[PREP_UNROLL][OF32 ? 2 : 1];
#pragma unroll
    for (int u = 0; u < PREP_UNROLL; ++u) {
        const long long r = r0 + u * RPW + sub;
        g[u] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int h = 0; h < (OF32 ? 2 : 1); ++h)
            o[u][h] = make_uint4(0u, 0u, 0u, 0u);
        if (r < rows) {
            g[u] = *reinterpret_cast<const uint4 *>(dO + r * D + c * 8);
            if constexpr (OF32) {
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    static_cast<const float *>(O_) + r * D + c * 8);
                o[u][0] = src[0];
                o[u][1] = src[1];
            } else {
                o[u][0] = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(O_) +
                                                          r * D + c * 8);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < PREP_UNROLL; ++u) {
        const uint32_t gw[4] = {g[u].x, g[u].y, g[u].z, g[u].w};
        float ov[8];
        if constexpr (OF32) {
            const uint32_t w[8] = {o[u][0].x, o[u][0].y, o[u][0].z, o[u][0].w,
                                   o[u][1].x, o[u][1].y, o[u][1].z, o[u][1].w};
#pragma unroll
            for (int e = 0; e < 8; ++e)
                ov[e] = __uint_as_float(w[e]);
        } else {
            const uint32_t w[4] = {o[u][0].x, o[u][0].y, o[u][0].z, o[u][0].w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                ov[2 * e] = lo16<BF16>(w[e]), ov[2 * e + 1] = hi16<BF16>(w[e]);
        }
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc = fmaf(lo16<BF16>(gw[e]), ov[2 * e], acc);
            acc = fmaf(hi16<BF16>(gw[e]), ov[2 * e + 1], acc);
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, off);
        const long long r = r0 + u * RPW + sub;
        if (c == 0 && r < rows)
            Drow[r] = acc;
    }
}

// Loads one 128-row tile of a [d, n, bh] tensor map (all d/64 panels).
template <int D>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                          int row, int bh) {
#pragma unroll
    for (int p = 0; p < D / 64; ++p)
        tma_load_3d(dst + p * BT * 128, map, bar, p * 64, row, bh);
}

// Issues acc += A(tmem, 128 rows x 64 in 16-bit) * B(rows [64 e, 64 e + 64)
// of a 128-row smem tile, MN-major: K = tile rows, N = D): the second
// product of one softmax half.  A holds two per column, written by the two
// warps of a row quarter: elements [0, 32) at columns [0, 16) of a_half,
// elements [32, 64) at columns [32, 48).
template <int D>
__device__ __forceinline__ void mma_tmem_a_half(uint32_t acc, uint32_t a_half, uint32_t b_tile,
                                                int e, uint32_t idesc, bool first) {
    // one descriptor low word, stepped by offset >> 4 (the start-address
    // field is the low 14 bits of address >> 4 and shared addresses stay
    // below 2^18, so the add never carries out of it) under the layout's
    // constant high word: no descriptor is rebuilt between the issuing
    // thread's MMAs
    const uint32_t b0 = sdesc_lo(b_tile, BT * 128);
#pragma unroll
    for (int k = 0; k < HS / 16; ++k) {
        const uint64_t bd =
            sdesc(b0 + static_cast<uint32_t>(((e * (HS / 16) + k) * 16 * 128) >> 4),
                  sdesc_sw128_hi(1024));
        mma_ts(acc, a_half + (k >> 1) * 32 + (k & 1) * 8, bd, idesc, (first && k == 0) ? 0u : 1u);
    }
}

// Issues acc = A(smem tile, K-major, 128 rows) * B(smem tile, K-major, 128
// rows)^T over K = D: a 128 x 128 score block.
template <int D>
__device__ __forceinline__ void mma_ss_block(uint32_t acc, uint32_t a_tile, uint32_t b_tile,
                                             uint32_t idesc) {
    const uint32_t a0 = sdesc_lo(a_tile, 16), b0 = sdesc_lo(b_tile, 16);
    constexpr uint32_t hi = sdesc_sw128_hi(1024);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k / 4) * (BT * 128) + (k % 4) * 32;
        mma_ss(acc, sdesc(a0 + (off >> 4), hi), sdesc(b0 + (off >> 4), hi), idesc,
               k > 0 ? 1u : 0u);
    }
}

// Writes 32 accumulator columns of this thread's row to global memory.
template <int OUT>
__device__ __forceinline__ void store32(void *dst_base, size_t elem_off, const float (&o)[32]) {
    if constexpr (OUT == 2) {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(dst_base) + elem_off);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
    } else {
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(dst_base) + elem_off);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pack2<OUT == 1>(o[8 * i], o[8 * i + 1]),
                                pack2<OUT == 1>(o[8 * i + 2], o[8 * i + 3]),
                                pack2<OUT == 1>(o[8 * i + 4], o[8 * i + 5]),
                                pack2<OUT == 1>(o[8 * i + 6], o[8 * i + 7]));
    }
}

// First query block that sees key block kb (bottom-right causal), else 0.
__device__ __forceinline__ int first_qblock(const Shape &sh, int kb) {
    if (!sh.causal)
        return 0;
    const int off = sh.n_kv - sh.n_q;
    const int need = kb * BT - off; // smallest query row that sees key kb*BT
    return need <= 0 ? 0 : need / BT;
}

// Number of key blocks query block qb sees.
__device__ __forceinline__ int key_blocks(const Shape &sh, int qb) {
    if (!sh.causal)
        return sh.nkb;
    const int r_last = min(qb * BT + BT - 1, sh.n_q - 1);
    return min(sh.nkb, (r_last + sh.n_kv - sh.n_q) / BT + 1);
}

// ========================================================================
// dK, dV: one CTA per (b, KV head, key block).  Step t = (query head of the
// group, query block): S^T, dP^T of the step's 128 queries, then dV, dK fed
// half by half as the softmax warps finish each 64 queries (P^T of queries
// [64 e + 32 c, +32) at dP^T columns [64 e + 32 c, +16), dS^T at the next 16).
template <int D, bool BF16, int OUT>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_do, const float *__restrict__ lse,
                  const float *__restrict__ Drow, void *__restrict__ dK, void *__restrict__ dV,
                  const Shape sh, unsigned *err) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);
    const uint32_t sK = base_s + C::OFF_A, sV = sK + C::TILE;
    auto sQ = [&](int st) { return base_s + C::OFF_X + st * C::TILE; };  // ring X
    auto sDO = [&](int st) { return base_s + C::OFF_Y + st * C::TILE; }; // ring Y
    // per step: -lse * log2(e) and -D of its 128 queries, double-buffered
    float *s_row = reinterpret_cast<float *>(base + C::OFF_ROW);
    const uint32_t bar0 = base_s + C::OFF_BAR;
    const uint32_t b_afull = bar0;
    // (the slots of the per-ring empty barriers, which the dQ kernel uses,
    // stay unused here: b_used below releases both rings)
    auto b_xfull = [&](int i) { return bar0 + 8u * (1 + i); };
    auto b_yfull = [&](int i) { return bar0 + 8u * (1 + 2 * C::NX + i); };
    const uint32_t b_s = bar0 + 8u * (1 + 2 * C::NX + 2 * C::NY); // scores ready
    const uint32_t b_dp = b_s + 8u;                   // second product ready
    const uint32_t b_sfree = b_s + 16u;               // scores loaded by the softmax warps
    auto b_pready = [&](int e) { return b_s + 8u * (3 + e); }; // half e packed
    const uint32_t b_done = b_s + 40u;
    const uint32_t b_drain = b_done + 8u;
    // step u's Q and dO stages consumed (one commit releases both rings)
    auto b_used = [&](int u) { return b_drain + 8u * (1 + u % C::NU); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + C::OFF_MISC + 8);

    if (base_s - raw_s + C::SMEM_USED > static_cast<uint32_t>(C::SMEM)) {
        if (threadIdx.x == 0)
            atomicOr(err, DERR_INDEX); // the base needed more alignment padding than reserved
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // heaviest key blocks first (causal: early keys are seen by more queries)
    const int kb = static_cast<int>(blockIdx.x) / (sh.B * sh.Hkv);
    const int bkv = static_cast<int>(blockIdx.x) % (sh.B * sh.Hkv);
    const int b = bkv / sh.Hkv, hk = bkv % sh.Hkv;
    const int qb0 = first_qblock(sh, kb);
    const int nq_steps = sh.nqb - qb0;     // query blocks per query head
    const int nsteps = sh.G * nq_steps;    // (head, query block) steps

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(b_afull, 1);
        for (int i = 0; i < C::NX; ++i)
            mbar_init(b_xfull(i), 1);
        for (int i = 0; i < C::NY; ++i)
            mbar_init(b_yfull(i), 1);
        mbar_init(b_s, 1);
        mbar_init(b_dp, 1);
        mbar_init(b_sfree, kSoftmaxWarps);
        for (int e = 0; e < 2; ++e)
            mbar_init(b_pready(e), kSoftmaxWarps);
        mbar_init(b_done, 1);
        mbar_init(b_drain, 1);
        for (int i = 0; i < C::NU; ++i)
            mbar_init(b_used(i), 1);
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // lane 0: K, V, then the Q ring; lane 1: the dO ring (each ring runs
        // at its own pace)
        if (lane < 2) {
            const bool is_x = lane == 0;
            const int n = is_x ? C::NX : C::NY;
            if (is_x) {
                mbar_arrive_expect_tx(b_afull, 2 * C::TILE);
                load_tile<D>(sK, &tm_k, b_afull, kb * BT, bkv);
                load_tile<D>(sV, &tm_v, b_afull, kb * BT, bkv);
            }
            int issued = 0;
            for (int t = 0; t < nsteps; ++t) {
                const int st = t % n;
                // stage st was last read by step t - n.  A waiter is never
                // two phases behind on b_used: step t - n + NU cannot be
                // consumed before this ring has refilled its stage, which
                // needs this very wait
                if (t >= n && !mbar_wait(b_used(t - n), ((t - n) / C::NU) & 1, abort_flag, err))
                    break;
                const int h = hk * sh.G + t / nq_steps;
                const int qb = qb0 + t % nq_steps;
                const int bh = b * sh.Hq + h;
                const uint32_t full = is_x ? b_xfull(st) : b_yfull(st);
                mbar_arrive_expect_tx(full, C::TILE);
                load_tile<D>(is_x ? sQ(st) : sDO(st), is_x ? &tm_q : &tm_do, full, qb * BT, bh);
                issued = t + 1;
            }
            if (*abort_flag) {
                if (is_x)
                    mbar_wait_drain(b_afull, 0);
                for (int u = max(0, issued - n); u < issued; ++u)
                    mbar_wait_drain(is_x ? b_xfull(u % n) : b_yfull(u % n), (u / n) & 1);
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16(BT, BT, BF16, false, false);
            constexpr uint32_t idesc_acc = idesc_f16(BT, D, BF16, false, true);
            bool ok = mbar_wait(b_afull, 0, abort_flag, err);
            if (ok && nsteps > 0)
                ok = mbar_wait(b_xfull(0), 0, abort_flag, err) &&
                     mbar_wait(b_yfull(0), 0, abort_flag, err);
            if (ok && nsteps > 0) {
                tc_fence_after();
                mma_ss_block<D>(tmem + C::S_COL, sK, sQ(0), idesc_s);
                tc_commit(b_s);
                mma_ss_block<D>(tmem + C::DP_COL, sV, sDO(0), idesc_s);
                tc_commit(b_dp);
            }
            for (int t = 0; ok && t < nsteps; ++t) {
                const int xt = t % C::NX, yt = t % C::NY;
                const int xn = (t + 1) % C::NX, yn = (t + 1) % C::NY;
                const bool next = t + 1 < nsteps;
                if (next) {
                    // both usually complete by now: one fused wait (the two
                    // try_waits back to back) instead of two in a row
                    if (!mbar_wait3(b_xfull(xn), ((t + 1) / C::NX) & 1, true, b_sfree, t & 1,
                                    true, 0u, 0u, false, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // the softmax warps hold step t's scores in registers
                    mma_ss_block<D>(tmem + C::S_COL, sK, sQ(xn), idesc_s);
                    tc_commit(b_s);
                }
                if (!mbar_wait(b_pready(0), t & 1, abort_flag, err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // dV += P^T dO, dK += dS^T Q over queries 0-63
                mma_tmem_a_half<D>(tmem + C::ACC0, tmem + C::DP_COL, sDO(yt), 0, idesc_acc,
                                   t == 0);
                mma_tmem_a_half<D>(tmem + C::ACC1, tmem + C::DP_COL + 16, sQ(xt), 0, idesc_acc,
                                   t == 0);
                // step t+1's first operand tile has usually landed long
                // before: tested together with P ready (the later wait for
                // it below is then satisfied at once)
                if (!mbar_wait3(b_pready(1), t & 1, true, b_yfull(yn), ((t + 1) / C::NY) & 1, next,
                                0u, 0u, false, abort_flag, err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the same over queries 64-127
                mma_tmem_a_half<D>(tmem + C::ACC0, tmem + C::DP_COL + 64, sDO(yt), 1, idesc_acc,
                                   false);
                mma_tmem_a_half<D>(tmem + C::ACC1, tmem + C::DP_COL + 80, sQ(xt), 1, idesc_acc,
                                   false);
                tc_commit(b_used(t)); // step t's Q and dO consumed
                if (next) {
                    tc_fence_after();
                    // after half 1's products, which read these columns (the
                    // tensor core runs in issue order)
                    mma_ss_block<D>(tmem + C::DP_COL, sV, sDO(yn), idesc_s);
                    tc_commit(b_dp);
                }
            }
            if (ok)
                tc_commit(b_done);
            tc_commit(b_drain);
            mbar_wait_drain(b_drain, 0);
        }
    } else {
        // ---- warps 0-7: one key row each, two warps per TMEM lane quarter;
        // warp half c takes queries [32 c, 32 c + 32) of each softmax half
        const int quarter = warp & 3, cpart = warp >> 2;
        const int j = quarter * 32 + lane; // key within the block
        const int key = kb * BT + j;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const int off = sh.n_kv - sh.n_q;
        const bool key_ok = key < sh.n_kv;
        // a statistic of query j of step t, fetched one step ahead so the
        // global loads are off the critical path: -lse log2(e) by warps 0-3,
        // -D by warps 4-7 (queries past n_q: p = 2^-inf = 0)
        auto fetch = [&](int t) {
            float v = cpart ? 0.f : -INFINITY;
            if (t < nsteps) {
                const size_t bh = static_cast<size_t>(b) * sh.Hq + hk * sh.G + t / nq_steps;
                const int q = (qb0 + t % nq_steps) * BT + j;
                if (q < sh.n_q)
                    v = cpart ? -Drow[bh * sh.n_q + q] : -lse[bh * sh.n_q + q] * kLog2e;
            }
            return v;
        };
        float nv = fetch(0);
        bool ok = true;
        const uint32_t tS = tmem + lane_off + C::S_COL;
        const uint32_t tP = tmem + lane_off + C::DP_COL;
        const float2 c2 = make_float2(sh.c, sh.c);
        for (int t = 0; t < nsteps; ++t) {
            const int qb = qb0 + t % nq_steps;
            float *rl = s_row + (t & 1) * 2 * BT; // -lse2 of the step's 128 queries
            float *rd = rl + BT;                  // -D
            // buffer t&1 was last read in step t-2; every warp has passed
            // step t-1's barrier since, so it is free
            (cpart ? rd : rl)[j] = nv;
            asm volatile("bar.sync 1, %0;" ::"n"(32 * kSoftmaxWarps) : "memory");
            nv = fetch(t + 1);
            // after a failed wait the warp keeps looping (and meeting the
            // named barrier above) without touching tensor memory, so that
            // its sibling warps never wait on it there
            if (!ok || !mbar_wait_warp(b_s, t & 1, abort_flag, err)) {
                ok = false;
                continue;
            }
            tc_fence_after();
            // query i (of the step's block) sees this key iff key <= qb*BT + i + off
            const int i_min = key - off - qb * BT; // first visible query (causal)
            // p of queries [i0, i0 + 32) from their 32 score columns
            auto probs = [&](const uint32_t(&us)[32], int i0, float2(&p)[16]) {
                const float4 *l4 = reinterpret_cast<const float4 *>(rl + i0);
#pragma unroll
                for (int w = 0; w < 16; ++w) {
                    const float4 l = l4[w / 2];
                    const float2 x = __ffma2_rn(
                        make_float2(__uint_as_float(us[2 * w]), __uint_as_float(us[2 * w + 1])),
                        c2, (w & 1) ? make_float2(l.z, l.w) : make_float2(l.x, l.y));
                    p[w] = make_float2(ex2(x.x), ex2(x.y));
                }
                if (!key_ok || (sh.causal && i_min > i0)) {
#pragma unroll
                    for (int w = 0; w < 16; ++w) {
                        if (!key_ok || i0 + 2 * w < i_min)
                            p[w].x = 0.f;
                        if (!key_ok || i0 + 2 * w + 1 < i_min)
                            p[w].y = 0.f;
                    }
                }
            };
            // dS = P (dP - D); P packed over dP columns [i0, i0 + 16), dS over
            // [i0 + 16, i0 + 32): the columns this warp has just read
            auto grads = [&](const float2(&p)[16], const uint32_t(&ud)[32], int i0) {
                const float4 *d4 = reinterpret_cast<const float4 *>(rd + i0);
                uint32_t pw[16], dw[16];
#pragma unroll
                for (int w = 0; w < 16; ++w) {
                    const float4 d = d4[w / 2];
                    const float2 g = __fadd2_rn(
                        make_float2(__uint_as_float(ud[2 * w]), __uint_as_float(ud[2 * w + 1])),
                        (w & 1) ? make_float2(d.z, d.w) : make_float2(d.x, d.y));
                    const float2 ds = __fmul2_rn(p[w], g);
                    pw[w] = pack2<BF16>(p[w].x, p[w].y);
                    dw[w] = pack2<BF16>(ds.x, ds.y);
                }
                tmem_st16(tP + i0, pw);
                tmem_st16(tP + i0 + 16, dw);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
            };
            // this warp's queries of the two halves: [32 c, +32) and [64 + 32 c, +32)
            const int i0 = 32 * cpart, i1 = HS + 32 * cpart;
            float2 p0[16], p1[16];
            {
                uint32_t us0[32], us1[32];
                tmem_ld32x2(tS + i0, us0, tS + i1, us1);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(b_sfree); // the next step's S^T may overwrite them
                probs(us0, i0, p0);
                probs(us1, i1, p1);
            }
            if (!mbar_wait_warp(b_dp, t & 1, abort_flag, err)) {
                ok = false;
                continue;
            }
            tc_fence_after();
            {
                uint32_t ud[32];
                tmem_ld32(tP + i0, ud);
                grads(p0, ud, i0);
                if (lane == 0)
                    mbar_arrive(b_pready(0));
            }
            {
                uint32_t ud[32];
                tmem_ld32(tP + i1, ud);
                grads(p1, ud, i1);
                if (lane == 0)
                    mbar_arrive(b_pready(1));
            }
        }
        if (ok && nsteps > 0)
            ok = mbar_wait_warp(b_done, 0, abort_flag, err);
        tc_fence_after();
        // the tensor-memory loads are warp-wide (.sync.aligned): every lane
        // executes them; only the stores depend on the row being real
        const size_t orow = (static_cast<size_t>(bkv) * sh.n_kv + key) * D;
#pragma unroll 1
        for (int c = cpart; c < 2 * (D / 32); c += 2) {
            // chunks [0, D/32) of dV, then of dK (scaled)
            const bool is_k = c >= D / 32;
            const int ch = is_k ? c - D / 32 : c;
            uint32_t u[32];
            tmem_ld32(tmem + lane_off + (is_k ? C::ACC1 : C::ACC0) + ch * 32, u);
            if (key_ok) {
                const float f = is_k ? sh.scale : 1.f;
                float o[32];
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    o[i] = (ok && nsteps > 0) ? __uint_as_float(u[i]) * f : 0.f;
                store32<OUT>(is_k ? dK : dV, orow + ch * 32, o);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ========================================================================
// dQ: one CTA per (b, query head, query block).  Step t = key block: S, dP
// of its 128 keys, then dQ fed half by half as the softmax warps finish each
// 64 keys (dS of keys [64 e + 32 c, +32) at dP columns [64 e + 32 c, +16)).
// Key blocks past the last visible key are not computed.
template <int D, bool BF16, int OUT>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_q_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_do, const float *__restrict__ lse,
                 const float *__restrict__ Drow, void *__restrict__ dQ, const Shape sh,
                 unsigned *err) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);
    const uint32_t sQ = base_s + C::OFF_A, sDO = sQ + C::TILE;
    auto sK = [&](int st) { return base_s + C::OFF_X + st * C::TILE; }; // ring X
    auto sV = [&](int st) { return base_s + C::OFF_Y + st * C::TILE; }; // ring Y
    const uint32_t bar0 = base_s + C::OFF_BAR;
    const uint32_t b_afull = bar0;
    auto b_xfull = [&](int i) { return bar0 + 8u * (1 + i); };
    auto b_xempty = [&](int i) { return bar0 + 8u * (1 + C::NX + i); };
    auto b_yfull = [&](int i) { return bar0 + 8u * (1 + 2 * C::NX + i); };
    auto b_yempty = [&](int i) { return bar0 + 8u * (1 + 2 * C::NX + C::NY + i); };
    const uint32_t b_s = bar0 + 8u * (1 + 2 * C::NX + 2 * C::NY); // scores ready
    const uint32_t b_dp = b_s + 8u;                   // second product ready
    const uint32_t b_sfree = b_s + 16u;               // scores loaded by the softmax warps
    auto b_pready = [&](int e) { return b_s + 8u * (3 + e); }; // half e packed
    const uint32_t b_done = b_s + 40u;
    const uint32_t b_drain = b_done + 8u;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + C::OFF_MISC + 8);

    if (base_s - raw_s + C::SMEM_USED > static_cast<uint32_t>(C::SMEM)) {
        if (threadIdx.x == 0)
            atomicOr(err, DERR_INDEX); // the base needed more alignment padding than reserved
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nbh = sh.B * sh.Hq;
    const int qb = sh.nqb - 1 - static_cast<int>(blockIdx.x) / nbh; // heaviest first
    const int bh = static_cast<int>(blockIdx.x) % nbh;
    const int b = bh / sh.Hq, h = bh % sh.Hq;
    const int bkv = b * sh.Hkv + h / sh.G;
    // key blocks up to the query block's last visible key
    int keys = sh.n_kv;
    if (sh.causal)
        keys = min(keys, min(qb * BT + BT - 1, sh.n_q - 1) + (sh.n_kv - sh.n_q) + 1);
    const int nsteps = (keys + BT - 1) / BT;

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(b_afull, 1);
        for (int i = 0; i < C::NX; ++i) {
            mbar_init(b_xfull(i), 1);
            mbar_init(b_xempty(i), 1);
        }
        for (int i = 0; i < C::NY; ++i) {
            mbar_init(b_yfull(i), 1);
            mbar_init(b_yempty(i), 1);
        }
        mbar_init(b_s, 1);
        mbar_init(b_dp, 1);
        mbar_init(b_sfree, kSoftmaxWarps);
        for (int e = 0; e < 2; ++e)
            mbar_init(b_pready(e), kSoftmaxWarps);
        mbar_init(b_done, 1);
        mbar_init(b_drain, 1);
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // lane 0: Q, dO, then the K ring; lane 1: the V ring
        if (lane < 2) {
            const bool is_x = lane == 0;
            const int n = is_x ? C::NX : C::NY;
            if (is_x) {
                mbar_arrive_expect_tx(b_afull, 2 * C::TILE);
                load_tile<D>(sQ, &tm_q, b_afull, qb * BT, bh);
                load_tile<D>(sDO, &tm_do, b_afull, qb * BT, bh);
            }
            int issued = 0;
            for (int t = 0; t < nsteps; ++t) {
                const int st = t % n;
                if (t >= n && !mbar_wait(is_x ? b_xempty(st) : b_yempty(st), ((t / n) - 1) & 1,
                                         abort_flag, err))
                    break;
                const uint32_t full = is_x ? b_xfull(st) : b_yfull(st);
                mbar_arrive_expect_tx(full, C::TILE);
                load_tile<D>(is_x ? sK(st) : sV(st), is_x ? &tm_k : &tm_v, full, t * BT, bkv);
                issued = t + 1;
            }
            if (*abort_flag) {
                if (is_x)
                    mbar_wait_drain(b_afull, 0);
                for (int u = max(0, issued - n); u < issued; ++u)
                    mbar_wait_drain(is_x ? b_xfull(u % n) : b_yfull(u % n), (u / n) & 1);
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16(BT, BT, BF16, false, false);
            constexpr uint32_t idesc_acc = idesc_f16(BT, D, BF16, false, true);
            bool ok = mbar_wait(b_afull, 0, abort_flag, err);
            if (ok && nsteps > 0)
                ok = mbar_wait(b_xfull(0), 0, abort_flag, err) &&
                     mbar_wait(b_yfull(0), 0, abort_flag, err);
            if (ok && nsteps > 0) {
                tc_fence_after();
                mma_ss_block<D>(tmem + C::S_COL, sQ, sK(0), idesc_s);
                tc_commit(b_s);
                mma_ss_block<D>(tmem + C::DP_COL, sDO, sV(0), idesc_s);
                tc_commit(b_dp);
                tc_commit(b_yempty(0)); // V is read by dP alone
            }
            for (int t = 0; ok && t < nsteps; ++t) {
                const int xt = t % C::NX, yt = t % C::NY;
                const int xn = (t + 1) % C::NX, yn = (t + 1) % C::NY;
                const bool next = t + 1 < nsteps;
                if (next) {
                    // both usually complete by now: one fused wait (the two
                    // try_waits back to back) instead of two in a row
                    if (!mbar_wait3(b_xfull(xn), ((t + 1) / C::NX) & 1, true, b_sfree, t & 1,
                                    true, 0u, 0u, false, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // the softmax warps hold step t's scores in registers
                    mma_ss_block<D>(tmem + C::S_COL, sQ, sK(xn), idesc_s);
                    tc_commit(b_s);
                }
                if (!mbar_wait(b_pready(0), t & 1, abort_flag, err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // dQ += dS K over keys 0-63 of the block
                mma_tmem_a_half<D>(tmem + C::ACC0, tmem + C::DP_COL, sK(xt), 0, idesc_acc,
                                   t == 0);
                // step t+1's first operand tile has usually landed long
                // before: tested together with P ready (the later wait for
                // it below is then satisfied at once)
                if (!mbar_wait3(b_pready(1), t & 1, true, b_yfull(yn), ((t + 1) / C::NY) & 1, next,
                                0u, 0u, false, abort_flag, err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the same over keys 64-127
                mma_tmem_a_half<D>(tmem + C::ACC0, tmem + C::DP_COL + 64, sK(xt), 1, idesc_acc,
                                   false);
                tc_commit(b_xempty(xt)); // step t's K consumed
                if (next) {
                    tc_fence_after();
                    // after half 1's products, which read these columns (the
                    // tensor core runs in issue order)
                    mma_ss_block<D>(tmem + C::DP_COL, sDO, sV(yn), idesc_s);
                    tc_commit(b_dp);
                    tc_commit(b_yempty(yn)); // V is read by dP alone
                }
            }
            if (ok)
                tc_commit(b_done);
            tc_commit(b_drain);
            mbar_wait_drain(b_drain, 0);
        }
    } else {
        // ---- warps 0-7: one query row each, two warps per TMEM lane
        // quarter; warp half c takes keys [32 c, 32 c + 32) of each softmax half
        const int quarter = warp & 3, cpart = warp >> 2;
        const int i = quarter * 32 + lane;
        const int row = qb * BT + i;
        const bool row_ok = row < sh.n_q;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const float nl =
            row_ok ? -lse[static_cast<size_t>(bh) * sh.n_q + row] * kLog2e : -INFINITY;
        const float nd = row_ok ? -Drow[static_cast<size_t>(bh) * sh.n_q + row] : 0.f;
        const int lim = sh.causal ? row + (sh.n_kv - sh.n_q) : sh.n_kv - 1; // last visible key
        const int klim = min(lim, sh.n_kv - 1);
        const float2 c2 = make_float2(sh.c, sh.c), l2 = make_float2(nl, nl),
                     d2 = make_float2(nd, nd);
        bool ok = true;
        const uint32_t tS = tmem + lane_off + C::S_COL;
        const uint32_t tP = tmem + lane_off + C::DP_COL;
        // p of keys [k0, k0 + 32) of step t from their 32 score columns
        auto probs = [&](const uint32_t(&us)[32], int t, int k0, float2(&p)[16]) {
#pragma unroll
            for (int w = 0; w < 16; ++w) {
                const float2 x = __ffma2_rn(
                    make_float2(__uint_as_float(us[2 * w]), __uint_as_float(us[2 * w + 1])), c2,
                    l2);
                p[w] = make_float2(ex2(x.x), ex2(x.y));
            }
            const int kl = klim - (t * BT + k0); // last visible key among the 32
            if (kl < 31) {
#pragma unroll
                for (int w = 0; w < 16; ++w) {
                    if (2 * w > kl)
                        p[w].x = 0.f;
                    if (2 * w + 1 > kl)
                        p[w].y = 0.f;
                }
            }
        };
        // dS = P (dP - D), packed over dP columns [k0, k0 + 16): columns this
        // warp has just read
        auto grads = [&](const float2(&p)[16], const uint32_t(&ud)[32], int k0) {
            uint32_t dw[16];
#pragma unroll
            for (int w = 0; w < 16; ++w) {
                const float2 g = __fadd2_rn(
                    make_float2(__uint_as_float(ud[2 * w]), __uint_as_float(ud[2 * w + 1])), d2);
                const float2 ds = __fmul2_rn(p[w], g);
                dw[w] = pack2<BF16>(ds.x, ds.y);
            }
            tmem_st16(tP + k0, dw);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
        };
        for (int t = 0; t < nsteps; ++t) {
            if (!mbar_wait_warp(b_s, t & 1, abort_flag, err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // this warp's keys of the two halves: [32 c, +32) and [64 + 32 c, +32)
            const int k0 = 32 * cpart, k1 = HS + 32 * cpart;
            float2 p0[16], p1[16];
            {
                uint32_t us0[32], us1[32];
                tmem_ld32x2(tS + k0, us0, tS + k1, us1);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(b_sfree); // the next step's S may overwrite them
                probs(us0, t, k0, p0);
                probs(us1, t, k1, p1);
            }
            if (!mbar_wait_warp(b_dp, t & 1, abort_flag, err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            {
                uint32_t ud[32];
                tmem_ld32(tP + k0, ud);
                grads(p0, ud, k0);
                if (lane == 0)
                    mbar_arrive(b_pready(0));
            }
            {
                uint32_t ud[32];
                tmem_ld32(tP + k1, ud);
                grads(p1, ud, k1);
                if (lane == 0)
                    mbar_arrive(b_pready(1));
            }
        }
        if (ok && nsteps > 0)
            ok = mbar_wait_warp(b_done, 0, abort_flag, err);
        tc_fence_after();
        const size_t orow = (static_cast<size_t>(bh) * sh.n_q + row) * D;
#pragma unroll 1
        for (int ch = cpart; ch < D / 32; ch += 2) {
            uint32_t u[32];
            tmem_ld32(tmem + lane_off + C::ACC0 + ch * 32, u); // warp-wide
            if (row_ok) {
                float o[32];
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    o[k] = (ok && nsteps > 0) ? __uint_as_float(u[k]) * sh.scale : 0.f;
                store32<OUT>(dQ, orow + ch * 32, o);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

} // namespace bw

// ------------------------------------------------------------------ host

// [d, n, bh] 16-bit tensor map, box {64, 128, 1}, 128-byte swizzle.
static bool bw_map(CUtensorMap *m, const void *ptr, int d, int n, int bh, bool bf16) {
    const uint64_t dims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(n),
                              static_cast<uint64_t>(bh)};
    const uint64_t strides[2] = {static_cast<uint64_t>(d) * 2,
                                 static_cast<uint64_t>(d) * 2 * static_cast<uint64_t>(n)};
    const uint32_t box[3] = {64, static_cast<uint32_t>(bw::BT), 1};
    return make_tmap_3d_16bit(m, ptr, bf16, dims, strides, box);
}

size_t backward_workspace_bytes(int B, int Hq, int n_q) {
    const size_t n = static_cast<size_t>(B) * Hq * n_q * sizeof(float);
    return (n + 255) & ~static_cast<size_t>(255);
}

template <int D, bool BF16, int OUT>
static cudaError_t backward_t(const BackwardArgs &a, cudaStream_t st) {
    using C = bw::Cfg<D>;
    CUtensorMap mq, mk, mv, mdo;
    if (!bw_map(&mq, a.Q, D, a.n_q, a.B * a.Hq, BF16) ||
        !bw_map(&mk, a.K, D, a.n_kv, a.B * a.Hkv, BF16) ||
        !bw_map(&mv, a.V, D, a.n_kv, a.B * a.Hkv, BF16) ||
        !bw_map(&mdo, a.dO, D, a.n_q, a.B * a.Hq, BF16))
        return cudaErrorInvalidValue;
    bw::Shape sh;
    sh.B = a.B;
    sh.Hq = a.Hq;
    sh.Hkv = a.Hkv;
    sh.G = a.Hq / a.Hkv;
    sh.n_q = a.n_q;
    sh.n_kv = a.n_kv;
    sh.causal = a.causal;
    sh.nqb = (a.n_q + bw::BT - 1) / bw::BT;
    sh.nkb = (a.n_kv + bw::BT - 1) / bw::BT;
    sh.c = a.scale * bw::kLog2e;
    sh.scale = a.scale;
    float *Drow = static_cast<float *>(a.workspace);
    const long long rows = static_cast<long long>(a.B) * a.Hq * a.n_q;
    const unsigned prep_grid = static_cast<unsigned>((rows + bw::prep_rows_per_block<D>() - 1) /
                                                     bw::prep_rows_per_block<D>());
    if (a.o_f32)
        bw::bwd_prep_kernel<D, BF16, true><<<prep_grid, 256, 0, st>>>(
            a.O, static_cast<const uint16_t *>(a.dO), Drow, rows);
    else
        bw::bwd_prep_kernel<D, BF16, false><<<prep_grid, 256, 0, st>>>(
            a.O, static_cast<const uint16_t *>(a.dO), Drow, rows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    auto kkv = bw::bwd_kv_kernel<D, BF16, OUT>;
    e = cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess)
        return e;
    kkv<<<static_cast<unsigned>(sh.nkb * a.B * a.Hkv), bw::kThreads, C::SMEM, st>>>(
        mq, mk, mv, mdo, a.lse, Drow, a.dK, a.dV, sh, a.err);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    auto kq = bw::bwd_q_kernel<D, BF16, OUT>;
    e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess)
        return e;
    kq<<<static_cast<unsigned>(sh.nqb * a.B * a.Hq), bw::kThreads, C::SMEM, st>>>(
        mq, mk, mv, mdo, a.lse, Drow, a.dQ, sh, a.err);
    return cudaGetLastError();
}

template <int D, bool BF16>
static cudaError_t backward_out(const BackwardArgs &a, cudaStream_t st) {
    switch (a.out_dtype) {
    case 0: return backward_t<D, BF16, 0>(a, st);
    case 1: return backward_t<D, BF16, 1>(a, st);
    default: return backward_t<D, BF16, 2>(a, st);
    }
}

cudaError_t backward_launch(const BackwardArgs &a, cudaStream_t st) {
    if (a.d == 64)
        return a.bf16 ? backward_out<64, true>(a, st) : backward_out<64, false>(a, st);
    if (a.d == 128)
        return a.bf16 ? backward_out<128, true>(a, st) : backward_out<128, false>(a, st);
    return cudaErrorInvalidValue;
}

} // namespace attn
