// prefill_sm103.cu -- exact attention forward on sm_103a tensor cores.
//
// The method (auturnal.com "From attention to IO-aware execution" §8;
// marketmaker.cc "Flash Attention and sequence length", "The Flash Attention
// algorithm" and "The online softmax recurrence"): Q is cut into row blocks
// and K, V into column blocks; for every (row block, column block) the score
// tile S = Q K^T is formed on chip, the running row max m, denominator l and
// un-normalised output u are rescaled by exp(m - m') when the block raises
// the max, u += P V, and u / l is written once at the end.  The full score
// matrix never leaves the SM.  Normalisation is deferred to the end of the
// loop (the FA2 scheduling on the same page), causal tiles entirely in the
// future are skipped (the same page's section on causal masking), and query
// head h reads KV head h / G (code-journey.com "Attention co-design", Group
// Size).
//
// B300 mapping (one CTA = 2 query tiles of 128 rows = 256 rows of one head):
//   warp 8      TMA producer: Q tiles once, then K_j / V_j through rings of
//               shared-memory stages (swizzled, one 3-D tensor map per
//               operand so tails read zeros).
//   warp 9      MMA issuer (one thread): S_t = Q_t K_j^T into tensor memory
//               (tcgen05.mma, A and B from shared memory), then
//               O_t += P_t V_j with P_t read from tensor memory.
//   warps 0-7   softmax, one warpgroup per query tile, one thread per row:
//               tcgen05.ld the 128 scores of its row, row max, p = 2^(s*c-m)
//               on the SFU, row sum, P packed to 16-bit back into tensor
//               memory over the consumed scores, O rescaled in tensor memory
//               when the reference max moves, final O / l and lse.
//   warps 10-11 (E4M3 inputs only) widen each V tile to f16 on chip.
// The two tiles ping-pong: while warpgroup 0 turns S_0 into P_0, the tensor
// core computes O_1 += P_1 V_j and S_1 for the next block, and vice versa.
//
// Tensor memory (512 columns x 128 lanes): S_0 [0,128), S_1 [128,256),
// O_0 [256, 256+D), O_1 [256+D, 256+2D).  P_t (16-bit, two per column)
// overwrites the first 64 columns of S_t; for rows with few visible keys
// the rounding residual P - P_hi is stored in the next 64 columns and
// multiplied in as a second MMA, so that the 16-bit rounding of P does not
// reach the output where too few terms average it out.
//
// E4M3 inputs (one fp32 scale per head of Q, K and V): S = Q K^T runs on the
// 8-bit tensor cores (kind::f8f6f4, both operands K-major as TMA lands them);
// P V runs in f16 -- the converter warp widens the E4M3 V tile exactly into
// the same swizzled f16 layout that 16-bit inputs arrive in.  The scales
// fold into the score factor (q_scale * k_scale) and the epilogue (v_scale).
//
// Scores are in the log2 domain (c = scale * log2 e).  u / l does not depend
// on which reference value is subtracted (the max-subtraction invariance of
// §8), so the reference max m is kept stale: a block's P is computed
// against it at once and kept while no row's sum of p exceeds 2^15 (then no
// p does, and P stays inside the f16 range) -- the row max is formed only
// for a row's first block and when that test fails, and then m moves only
// if the block's max exceeds it by more than 8.  This spares the row max on
// almost every block and most O rescales.
#include <atomic>

#include "common.cuh"
#include "launch.h"

namespace attn {

namespace pf {

constexpr int BM = 128;      // query rows per tile
constexpr int NT = 2;        // query tiles per CTA
constexpr int BN = 128;      // keys per block
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kConvWarp = 10;
constexpr int kSplitKeys = 512; // rows seeing fewer keys carry the P residual

constexpr float kRescaleThreshold = 8.0f;
// a block computed against the reference max is kept while no row's sum of
// p exceeds this (so no p does: every p is at most its row's sum), which
// keeps each p inside the f16 range of the P operand
constexpr float kSumLimit = 32768.0f;
// Registers per thread: 384 threads launch with 168 each (the most that three
// warps per SM sub-partition allow); the producer / MMA / converter
// warpgroup (warps 8-11) hands most of its share to the two softmax
// warpgroups, whose 128-score rows would otherwise spill:
// 256 x 208 + 128 x 88 = 384 x 168, and per SM sub-partition (warps k, k+4,
// k+8) 208 + 208 + 88 = 3 x 168.
constexpr int kThreadsAll = 384;
constexpr int kLaunchRegs = 168;
constexpr int kRegsSoftmax = 208;
constexpr int kRegsOther = 88;
static_assert(256 * kRegsSoftmax + 128 * kRegsOther == kThreadsAll * kLaunchRegs,
              "register split must add up to the launch allocation");

template <int D, bool F8>
struct Cfg {
    static constexpr int EB = F8 ? 1 : 2;                   // bytes per Q/K element
    static constexpr int PW = D * EB < 128 ? D * EB : 128;  // Q/K row bytes per panel = swizzle span
    static constexpr int QK_PANELS = D * EB / PW;
    static constexpr int Q_TILE_BYTES = BM * D * EB;
    static constexpr int K_BYTES = BN * D * EB;
    static constexpr int V_BYTES = BN * D * 2;              // 16-bit V operand stage
    static constexpr int VS_BYTES = BN * D;                 // E4M3 V staging
    static constexpr int NK = (F8 || D == 64) ? 3 : 2;      // K stages
    static constexpr int NV = (D == 64 || !F8) ? 3 : 2;     // V stages
    // 16-bit inputs: V stages are released by the softmax warps (below)
    // instead of a commit of the MMA-issuing thread, one block later; the
    // third V stage covers the delay (E4M3 V is released by the widening
    // warps)
    static constexpr bool SOFTMAX_FREES_V = !F8;
    static constexpr int NVS = F8 ? 2 : 0;                  // E4M3 V staging buffers
    static constexpr int NCONV = F8 ? 2 : 0;                // V widening warps
    static constexpr int THREADS = kThreadsAll; // warps 10-11 idle for 16-bit inputs
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + NT * Q_TILE_BYTES;
    static constexpr int OFF_V = OFF_K + NK * K_BYTES;
    static constexpr int OFF_VS = OFF_V + NV * V_BYTES;
    static constexpr int OFF_BAR = OFF_VS + NVS * VS_BYTES;
    static constexpr int NBAR = 1 + 2 * NK + 2 * NV + 2 * NVS + 2 * NT + 2;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 64 + 1024; // + alignment slack
    __host__ __device__ static constexpr int S_COL(int t) { return t * BN; }
    __host__ __device__ static constexpr int O_COL(int t) { return NT * BN + t * D; }
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(NT * BN + NT * D <= 512, "tensor memory budget");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

struct Shape {
    int B, Hq, Hkv, G, n_q, n_kv, causal, nqb;
    int kvg;     // (batch, KV head) pairs per group of the CTA order (work_item)
    float c;     // scale * log2(e)
    float scale; // for reference only
};

// Scales of E4M3 inputs (null for 16-bit inputs).  Q and K carry one scale
// per head or one per block of 128 rows of a head: query tile t (rows
// 128t .. 128t+127) of head bh uses q[bh * qh + t * qb], keys 128j .. 128j+127
// of KV head bkv use k[bkv * kh + j * kb] (qb = kb = 0 and qh = kh = 1 for
// per-head scales).  V has one scale per KV head.
struct Scales {
    const float *q;
    const float *k;
    const float *v;
    int qh, qb, kh, kb;
};

// Block-paged K/V (prefill over a cache): per sequence b, seq_lens[b]
// tokens, token t in slot t % bs of block table[b][t / bs], layout
// [num_blocks, Hkv, bs, d].  Unused (null) for dense K/V.
struct Paged {
    const int32_t *table;
    const int32_t *lens;
    const uint8_t *vcache;
    int bs, max_blocks, num_blocks, max_len;
    int v4; // V by one 4-D box per cache block into unit-major stages (d = 256, bs = 16)
};

// Paged V stages can be unit-major at d = 256 only (see paged_kv_producer);
// the call takes that form when its cache blocks are 16 tokens (Paged::v4).
template <int D>
constexpr bool kPagedV4 = D == 256;

// Shared-memory descriptor of the V operand (B, MN-major, 128-byte swizzle)
// for the P.V product over keys [16 k, 16 k + 16) of a V stage at vb: dense
// stages are [panel][key] (panel stride BN rows), unit-major paged ones
// [unit][panel][token] (16-token units: panel stride 16 rows).
// (The unit-major form is taken with 16-token blocks only, so the 16 keys
// of step k are exactly unit k: a constant stride, nothing computed per MMA
// in the issuing thread.)
//
// Descriptors are built once per operand region and stepped by adding the
// byte offset >> 4 to their low word: the start-address field is the low 14
// bits of the address >> 4, and no shared-memory address reaches 2^18, so
// the add never carries out of the field; the high word is a constant of
// the layout.  (Rebuilding them per MMA put integer work between the
// issuing thread's MMAs, and 64-bit bases cost that thread's small register
// budget spills.)  lv / lv4: the stage's low word for the [panel][key] /
// unit-major layout.
template <bool PAGED, int D, int BN>
__device__ __forceinline__ uint64_t pv_desc(uint32_t lv, uint32_t lv4, int k, int v4) {
    constexpr uint32_t hi = sdesc_sw128_hi(1024);
    if constexpr (PAGED && kPagedV4<D>)
        if (v4)
            return sdesc(lv4 + static_cast<uint32_t>((k * ((D / 64) * 16 * 128)) >> 4), hi);
    return sdesc(lv + static_cast<uint32_t>((k * 16 * 128) >> 4), hi);
}

// Low descriptor words of a V stage (see pv_desc).
template <int BN>
__device__ __forceinline__ uint32_t pv_base(uint32_t vb) {
    return sdesc_lo(vb, BN * 128);
}
__device__ __forceinline__ uint32_t pv_base4(uint32_t vb) { return sdesc_lo(vb, 16 * 128); }

// Whole-warp producer of the K and V blocks (BN keys, 16-bit, D) of one
// (sequence, KV head) from a block-paged cache, one cache block ("unit") of
// block_size tokens per lane.  K: one TMA box (block_size tokens x 64
// elements) per unit and 128-byte panel, into the swizzled stage layout
// dense tiles have ([panel][key]).  V at d = 256 with 16-token blocks
// (Paged::v4): one 4-D box per unit holding its four panels, so the V stage
// is unit-major ([unit][panel][token], each panel a swizzled block of
// block_size rows; pv_desc steps the P.V operand through it).  Such a box
// costs the TMA unit more than a plain one and pays only where it replaces
// four 2 KB boxes: d = 256 with 32- or 64-token blocks measured 3-14%
// slower with it, d = 128 1447 -> 917 TFLOP/s, d = 64 787 -> 695; there V
// keeps one box per panel.  Units past the sequence end read a block
// coordinate past the tensor, which TMA fills with zeros.  The one V unit
// that holds the sequence end is copied with plain loads and its rows past
// the end zeroed: their p is 0, and 0 * (stale non-finite cache contents)
// must not reach u.  K rows past the end need no care -- their scores are
// replaced by -inf.  Block ids are fetched one key block ahead, one lane per
// unit; lane u issues unit u's boxes.  [KP0, KP1) and [VP0, VP1) are the
// 128-byte panels of each K and V row this warp copies (an empty range: not
// that tensor): a warp's TMA instructions are taken one at a time, so with
// warps to spare the boxes are spread over several warps.  Each warp
// arrives once per stage on the full barriers it feeds, announcing its own
// bytes (the barriers count the warps that feed them).
template <int D, int BN, int NK, int NV, int KP0, int KP1, int VP0, int VP1>
__device__ __forceinline__ void paged_kv_producer(
    const Paged &pg, int b, int hkv, int Hkv, int n_kv, int nb_max, const CUtensorMap *tm_k,
    const CUtensorMap *tm_v, uint32_t sK, uint32_t sV, uint32_t kfull0, uint32_t kempty0,
    uint32_t vfull0, uint32_t vempty0, volatile int *abort_flag, unsigned *err, int lane) {
    const int U = pg.bs;                        // tokens per unit: one cache block
    const int UPB = BN / U;                     // units per key block (BN % U == 0)
    constexpr bool DO_K = KP1 > KP0, DO_V = VP1 > VP0;
    static_assert(0 <= KP0 && KP0 <= KP1 && KP1 <= D / 64, "K panel range");
    static_assert(0 <= VP0 && VP0 <= VP1 && VP1 <= D / 64, "V panel range");
    static_assert(DO_K || DO_V, "a producer feeds at least one tensor");
    constexpr bool V4_OK = kPagedV4<D>;
    static_assert(!V4_OK || !DO_V || (VP0 == 0 && VP1 == D / 64),
                  "one V box holds every panel of a unit");
    const bool v4 = V4_OK && pg.v4 != 0;
    constexpr int VNP = VP1 - VP0;
    constexpr int VCH = VNP > 0 ? VNP * 8 : 1;      // 16-byte chunks of a V row it copies
    constexpr int K_STAGE = BN * (KP1 - KP0) * 128; // this warp's bytes of a K stage
    const int v_unit = U * 128 * VNP;               // this warp's bytes of one V unit
    constexpr int STAGE = BN * D * 2;               // bytes of a whole stage
    const unsigned full = 0xffffffffu;
    const int32_t *trow = pg.table + static_cast<size_t>(b) * pg.max_blocks;
    auto unit_blk = [&](int j) -> int {
        const int tok = j * BN + U * lane;
        if (lane >= UPB || tok >= n_kv)
            return -1;
        const int phys = trow[tok / pg.bs];
        return (phys >= 0 && phys < pg.num_blocks) ? phys : -2;
    };
    int nxt = nb_max > 0 ? unit_blk(0) : -1;
    bool bad = false;
    int k_issued = 0, v_issued = 0;
    for (int j = 0; j < nb_max; ++j) {
        const int cur = nxt;
        if (j + 1 < nb_max)
            nxt = unit_blk(j + 1);
        bad |= cur == -2;
        const int z = cur >= 0 ? cur : pg.num_blocks;
        const int y = hkv * pg.bs; // a unit is a whole cache block
        int ok = 1;
        if constexpr (DO_K) {
            const int ks = j % NK;
            if (j >= NK) {
                if (lane == 0)
                    ok = mbar_wait(kempty0 + 8u * ks, ((j / NK) - 1) & 1, abort_flag, err);
                ok = __shfl_sync(full, ok, 0);
            }
            if (!ok)
                break;
            if (lane == 0)
                mbar_arrive_expect_tx(kfull0 + 8u * ks, K_STAGE);
            __syncwarp();
            // lane u issues unit u's boxes: one instruction starts every unit's copy
            if (lane < UPB) {
#pragma unroll
                for (int p = KP0; p < KP1; ++p)
                    tma_load_3d(sK + ks * STAGE + p * BN * 128 + lane * U * 128, tm_k,
                                kfull0 + 8u * ks, p * 64, y, z);
            }
            k_issued = j + 1;
        }
        if constexpr (!DO_V)
            continue;
        const int vs = j % NV;
        if (j >= NV) {
            if (lane == 0)
                ok = mbar_wait(vempty0 + 8u * vs, ((j / NV) - 1) & 1, abort_flag, err);
            ok = __shfl_sync(full, ok, 0);
        }
        if (!ok)
            break;
        const int rem = n_kv - j * BN; // keys of this block inside the sequence
        const int up = (rem > 0 && rem < BN && rem % U != 0) ? rem / U : -1;
        if (up >= 0) {
            const int blk = __shfl_sync(full, cur, up);
            const int nval = rem % U;
            const size_t row0 = (static_cast<size_t>(blk >= 0 ? blk : 0) * Hkv + hkv) * pg.bs;
            for (int i = lane; i < U * VNP * 8; i += 32) { // U rows x this warp's chunks
                const int r = i / VCH, c = VP0 * 8 + i % VCH;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (r < nval && blk >= 0)
                    v = *reinterpret_cast<const uint4 *>(pg.vcache + (row0 + r) * (D * 2) + c * 16);
                const uint32_t dst =
                    v4 ? sV + vs * STAGE + up * ((D / 64) * U * 128) + (c / 8) * (U * 128) +
                             swz_offset<128>(r, c % 8)
                       : sV + vs * STAGE + (c / 8) * (BN * 128) + swz_offset<128>(up * U + r, c % 8);
                sts_v4(dst, v.x, v.y, v.z, v.w);
            }
            fence_proxy_async_smem(); // generic writes -> tensor-core reads
            __syncwarp();
        }
        if (lane == 0)
            mbar_arrive_expect_tx(vfull0 + 8u * vs, (UPB - (up >= 0 ? 1 : 0)) * v_unit);
        __syncwarp();
        if (lane < UPB && lane != up) {
            if (v4) {
                tma_load_4d(sV + vs * STAGE + lane * ((D / 64) * U * 128), tm_v, vfull0 + 8u * vs,
                            0, y, 0, z);
            } else {
#pragma unroll
                for (int p = VP0; p < VP1; ++p)
                    tma_load_3d(sV + vs * STAGE + p * BN * 128 + lane * U * 128, tm_v,
                                vfull0 + 8u * vs, p * 64, y, z);
            }
        }
        v_issued = j + 1;
    }
    if (__any_sync(full, bad) && lane == 0)
        atomicOr(err, DERR_INDEX);
    if (lane == 0 && *abort_flag) { // let in-flight copies land before the CTA exits
        if constexpr (DO_K)
            for (int u = max(0, k_issued - NK); u < k_issued; ++u)
                mbar_wait_drain(kfull0 + 8u * (u % NK), (u / NK) & 1);
        if constexpr (DO_V)
            for (int u = max(0, v_issued - NV); u < v_issued; ++u)
                mbar_wait_drain(vfull0 + 8u * (u % NV), (u / NV) & 1);
    }
}

// A paged sequence whose length the table cannot hold (or that is shorter
// than its causal query rows): the CTA writes O = 0, lse = NaN and records
// the error.  Returns the sequence length, or -1 after handling an invalid one.
template <int D, int OUT>
__device__ __forceinline__ int paged_len_or_reject(const Paged &pg, const Shape &sh, int b, int bh,
                                                   int row0, int rows, void *O, float *lse,
                                                   unsigned *err) {
    const int len = pg.lens[b];
    const bool ok = len >= (sh.causal ? sh.n_q : 1) && len <= pg.max_len &&
                    (len + pg.bs - 1) / pg.bs <= pg.max_blocks;
    if (ok)
        return len;
    if (threadIdx.x == 0)
        atomicOr(err, DERR_INDEX);
    const int r_hi = min(row0 + rows, sh.n_q);
    for (int i = threadIdx.x; i < (r_hi - row0) * D; i += blockDim.x) {
        const size_t o = (static_cast<size_t>(bh) * sh.n_q + row0) * D + i;
        if constexpr (OUT == 2)
            static_cast<float *>(O)[o] = 0.f;
        else
            static_cast<uint16_t *>(O)[o] = 0;
    }
    if (lse != nullptr)
        for (int i = threadIdx.x; i < r_hi - row0; i += blockDim.x)
            lse[static_cast<size_t>(bh) * sh.n_q + row0 + i] = __int_as_float(0x7fc00000);
    return -1;
}

// CTA index -> (query block, batch, head).  The (batch, KV head) pairs are
// taken in groups of kvg; within a group the query blocks run in descending
// order (heaviest causal work first), then the group's pairs and the G query
// heads of each.  The host sizes a group so that its K / V fit in L2 with
// room to spare: the CTAs resident at one time then stream K / V that stay in
// L2 while all the group's query heads and query blocks read them (at
// n = 32768, d = 128, one KV head's K / V are 16.8 MB, and with every head
// resident at once they outgrow L2 and are re-read from DRAM about 23
// times), while the readers of any one line stay spread over the group's
// pairs and query blocks.  When all K / V fit, the whole grid is one group:
// heaviest query blocks of every head first.
__device__ __forceinline__ void work_item(const Shape &sh, int idx, int &qb, int &b, int &h) {
    const int per_group = sh.nqb * sh.kvg * sh.G;
    const int grp = idx / per_group, rem = idx % per_group;
    const int kvg = min(sh.kvg, sh.B * sh.Hkv - grp * sh.kvg); // the last group may be smaller
    const int width = kvg * sh.G;
    qb = sh.nqb - 1 - rem / width;
    const int inner = rem % width;
    const int pair = grp * sh.kvg + inner / sh.G;
    b = pair / sh.Hkv;
    h = (pair % sh.Hkv) * sh.G + inner % sh.G;
}

// Paged calls: the sequence at position pos of the CTA order when the
// sequences are taken longest first (ties by index), so that the long ones
// do not make the last wave's tail.  Each warp ranks the seq_lens entries
// itself with shuffles (rank of c = the entries ordered before it; a total
// order, so any lengths give a permutation).  Calls with more than
// kLongestFirstMaxB sequences keep the given order.
constexpr int kLongestFirstMaxB = 64;

__device__ __forceinline__ int longest_first(const int32_t *lens, int B, int pos) {
    if (B > kLongestFirstMaxB)
        return pos;
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    int found = pos;
    for (int c0 = 0; c0 < B; c0 += 32) {
        const int c = c0 + lane;
        const int mine = c < B ? lens[c] : 0;
        int rank = 0;
        for (int k0 = 0; k0 < B; k0 += 32) {
            const int other = k0 + lane < B ? lens[k0 + lane] : 0;
#pragma unroll 8
            for (int i = 0; i < 32; ++i) {
                const int o = __shfl_sync(full, other, i);
                const int k = k0 + i;
                rank += (k < B && (o > mine || (o == mine && k < c))) ? 1 : 0;
            }
        }
        const unsigned hit = __ballot_sync(full, c < B && rank == pos);
        if (hit)
            found = c0 + __ffs(hit) - 1;
    }
    return found;
}

__device__ __forceinline__ int tile_blocks(const Shape &sh, int q0, int t) {
    const int r0 = q0 + t * BM;
    if (r0 >= sh.n_q)
        return 0;
    const int nkb = (sh.n_kv + BN - 1) / BN;
    if (!sh.causal)
        return nkb;
    const int r_last = min(r0 + BM - 1, sh.n_q - 1);
    const int k_last = r_last + (sh.n_kv - sh.n_q);
    return min(nkb, k_last / BN + 1);
}

__device__ __forceinline__ bool tile_split(const Shape &sh, int q0, int t) {
    const int r0 = q0 + t * BM;
    const int keys = sh.causal ? (r0 + (sh.n_kv - sh.n_q) + 1) : sh.n_kv;
    return keys < kSplitKeys;
}

// p = 2^(s*c - m) for the NB scores of this thread's row, packed to 16 bits
// and stored over the consumed scores (P_hi in columns [0, NB/2) of the S
// tile; with SPLIT, the rounding residual p - P_hi in columns [NB/2, NB)).
// Returns the row sum of p (fp32, eight independent partial sums).  The
// score scaling and the sums run as packed pairs (fma/add .f32x2: one
// instruction per two elements, each lane rounded as the scalar form).
template <int NB, bool BF16, bool SPLIT>
__device__ __forceinline__ float exp_pack_store(const float (&s)[NB], float c, float neg,
                                                uint32_t tS) {
    float2 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        acc[i] = make_float2(0.f, 0.f);
    const float2 c2 = make_float2(c, c), n2 = make_float2(neg, neg);
#pragma unroll
    for (int ch = 0; ch < NB / 32; ++ch) {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float2 x =
                __ffma2_rn(make_float2(s[ch * 32 + 2 * i], s[ch * 32 + 2 * i + 1]), c2, n2);
            const float2 p = make_float2(ex2(x.x), ex2(x.y));
            acc[i & 3] = __fadd2_rn(acc[i & 3], p);
            hi[i] = pack2<BF16>(p.x, p.y);
            if constexpr (SPLIT)
                lo[i] = pack2<BF16>(p.x - lo16<BF16>(hi[i]), p.y - hi16<BF16>(hi[i]));
        }
        tmem_st16(tS + ch * 16, hi);
        if constexpr (SPLIT)
            tmem_st16(tS + NB / 2 + ch * 16, lo);
    }
    return ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) +
           ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
}

// Widen one E4M3 V tile [ROWS][D] (panels of PW-byte rows, PW-byte swizzle)
// into the f16 operand layout (panels of 64 elements = 128-byte rows,
// 128-byte swizzle) -- the layout 16-bit V tiles arrive in by TMA.  Warp
// `part` of `nparts` converts every nparts-th group of 32 chunks.
template <int D, int ROWS, int PW>
__device__ __forceinline__ void widen_v_tile(uint32_t src, uint32_t dst, int lane, int part,
                                             int nparts) {
    constexpr int CPR = D / 16; // 16-byte source chunks per row
#pragma unroll 4
    for (int i = part * 32 + lane; i < ROWS * CPR; i += 32 * nparts) {
        const int r = i / CPR, c = i % CPR;
        const uint4 v = lds_v4(src + (c * 16 / PW) * (ROWS * PW) +
                               swz_offset<PW>(r, (c * 16 % PW) >> 4));
        const uint32_t pb = dst + (c / 4) * (ROWS * 128);
        sts_v4(pb + swz_offset<128>(r, 2 * (c % 4)), e4m3x2_to_f16x2(v.x),
               e4m3x2_to_f16x2(v.x >> 16), e4m3x2_to_f16x2(v.y), e4m3x2_to_f16x2(v.y >> 16));
        sts_v4(pb + swz_offset<128>(r, 2 * (c % 4) + 1), e4m3x2_to_f16x2(v.z),
               e4m3x2_to_f16x2(v.z >> 16), e4m3x2_to_f16x2(v.w), e4m3x2_to_f16x2(v.w >> 16));
    }
}

template <int D, bool BF16, bool F8, bool PAGED, int OUT>
__global__ void __launch_bounds__(Cfg<D, F8>::THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_o, void *__restrict__ O,
                   float *__restrict__ lse, const Shape sh_in, const Scales sc, const Paged pg,
                   unsigned *err) {
    using C = Cfg<D, F8>;
    static_assert(!(PAGED && F8), "paged prefill reads 16-bit caches");
    Shape sh = sh_in;
    constexpr bool PB = F8 ? false : BF16; // format of P and of the V operand
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base (128-byte swizzle atoms repeat every 1 KB)
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);

    const uint32_t sQ = base_s + C::OFF_Q;
    const uint32_t sK = base_s + C::OFF_K;
    const uint32_t sV = base_s + C::OFF_V;
    const uint32_t sVS = base_s + C::OFF_VS;
    const uint32_t bar0 = base_s + C::OFF_BAR;
    const uint32_t b_qfull = bar0;
    auto b_kfull = [&](int i) { return bar0 + 8u * (1 + i); };
    auto b_kempty = [&](int i) { return bar0 + 8u * (1 + C::NK + i); };
    auto b_vfull = [&](int i) { return bar0 + 8u * (1 + 2 * C::NK + i); };
    auto b_vempty = [&](int i) { return bar0 + 8u * (1 + 2 * C::NK + C::NV + i); };
    auto b_vsfull = [&](int i) { return bar0 + 8u * (1 + 2 * C::NK + 2 * C::NV + i); };
    auto b_vsempty = [&](int i) {
        return bar0 + 8u * (1 + 2 * C::NK + 2 * C::NV + C::NVS + i);
    };
    constexpr int SB = 1 + 2 * C::NK + 2 * C::NV + 2 * C::NVS;
    auto b_sfull = [&](int t) { return bar0 + 8u * (SB + t); };
    auto b_pfull = [&](int t) { return bar0 + 8u * (SB + NT + t); };
    const uint32_t b_ofull = bar0 + 8u * (SB + 2 * NT);
    const uint32_t b_drain = b_ofull + 8u;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + C::OFF_MISC + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- work item: query blocks heaviest first within groups of (sequence,
    // KV head) pairs sized for L2, so that the K/V read by the group's CTAs
    // stream from DRAM about once; paged sequences longest first.
    int qb, b, h;
    work_item(sh, static_cast<int>(blockIdx.x), qb, b, h);
    if constexpr (PAGED)
        b = longest_first(pg.lens, sh.B, b);
    const int bh = b * sh.Hq + h;
    const int bkv = b * sh.Hkv + h / sh.G;
    const int q0 = qb * (NT * BM);
    if constexpr (PAGED) {
        const int len = paged_len_or_reject<D, OUT>(pg, sh, b, bh, q0, NT * BM, O, lse, err);
        if (len < 0)
            return;
        sh.n_kv = len;
    }
    int nb[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t)
        nb[t] = tile_blocks(sh, q0, t);
    const int nb_max = max(nb[0], nb[1]);

    // ---- set-up: barriers, tensor memory
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(b_qfull, 1);
        for (int i = 0; i < C::NK; ++i) {
            mbar_init(b_kfull(i), 1);
            mbar_init(b_kempty(i), 1);
        }
        for (int i = 0; i < C::NV; ++i) {
            mbar_init(b_vfull(i), F8 ? C::NCONV : 1);
            mbar_init(b_vempty(i), 1);
        }
        for (int i = 0; i < C::NVS; ++i) {
            mbar_init(b_vsfull(i), 1);
            mbar_init(b_vsempty(i), C::NCONV);
        }
        for (int t = 0; t < NT; ++t) {
            mbar_init(b_sfull(t), 1);
            mbar_init(b_pfull(t), 4);
        }
        mbar_init(b_ofull, 1);
        mbar_init(b_drain, 1);
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the roles of warps 8-11 run with few registers, the softmax
    // warpgroups with many; each side finishes on its own (no code is shared
    // across the two register budgets)
    if (warp >= kProducerWarp) {
        setmaxnreg_dec<kRegsOther>();
        if (warp == kProducerWarp && PAGED) {
            // ================================================= paged producer
            if (lane == 0) {
                int ntiles = 0;
                for (int t = 0; t < NT; ++t)
                    ntiles += nb[t] > 0;
                mbar_arrive_expect_tx(b_qfull, ntiles * C::Q_TILE_BYTES);
                for (int t = 0; t < NT; ++t)
                    if (nb[t] > 0)
                        for (int p = 0; p < C::QK_PANELS; ++p)
                            tma_load_3d(sQ + t * C::Q_TILE_BYTES + p * BM * C::PW, &tm_q, b_qfull,
                                        p * 64, q0 + t * BM, bh);
            }
            paged_kv_producer<D, BN, C::NK, C::NV, 0, D / 64, 0, 0>(
                pg, b, h / sh.G, sh.Hkv, sh.n_kv, nb_max, &tm_k, &tm_v, sK, sV, b_kfull(0),
                b_kempty(0), b_vfull(0), b_vempty(0), abort_flag, err, lane);
            if (lane == 0 && *abort_flag)
                mbar_wait_drain(b_qfull, 0);
        } else if (warp == kConvWarp && PAGED) {
            // ================================================= paged V producer
            // (paged inputs are 16-bit: the widening warps are free)
            static_assert(!PAGED || !F8, "paged inputs are 16-bit");
            paged_kv_producer<D, BN, C::NK, C::NV, 0, 0, 0, D / 64>(
                pg, b, h / sh.G, sh.Hkv, sh.n_kv, nb_max, &tm_k, &tm_v, sK, sV, b_kfull(0),
                b_kempty(0), b_vfull(0), b_vempty(0), abort_flag, err, lane);
        } else if (warp == kProducerWarp) {
            // ================================================= TMA producer
            if (lane == 0) {
                constexpr int XP = C::PW / C::EB; // elements per Q/K panel row
                // test hook: without the Q copy the MMA issuer's first wait
                // expires, which exercises the unwinding below
                const bool withhold_q =
                    (*reinterpret_cast<const volatile unsigned *>(err + CTL_HOOKS) &
                     HOOK_WITHHOLD_Q) != 0u;
                int ntiles = 0;
                for (int t = 0; t < NT; ++t)
                    ntiles += nb[t] > 0;
                if (!withhold_q) {
                    mbar_arrive_expect_tx(b_qfull, ntiles * C::Q_TILE_BYTES);
                    for (int t = 0; t < NT; ++t)
                        if (nb[t] > 0)
                            for (int p = 0; p < C::QK_PANELS; ++p)
                                tma_load_3d(sQ + t * C::Q_TILE_BYTES + p * BM * C::PW, &tm_q,
                                            b_qfull, p * XP, q0 + t * BM, bh);
                }
                int k_issued = 0, v_issued = 0;
                for (int j = 0; j < nb_max; ++j) {
                    const int ks = j % C::NK;
                    if (j >= C::NK &&
                        !mbar_wait(b_kempty(ks), ((j / C::NK) - 1) & 1, abort_flag, err))
                        break;
                    mbar_arrive_expect_tx(b_kfull(ks), C::K_BYTES);
                    for (int p = 0; p < C::QK_PANELS; ++p)
                        tma_load_3d(sK + ks * C::K_BYTES + p * BN * C::PW, &tm_k, b_kfull(ks),
                                    p * XP, j * BN, bkv);
                    k_issued = j + 1;
                    if constexpr (F8) {
                        // E4M3 V into staging; the converter warp fills the V stage
                        const int vs = j % C::NVS;
                        if (j >= C::NVS &&
                            !mbar_wait(b_vsempty(vs), ((j / C::NVS) - 1) & 1, abort_flag, err))
                            break;
                        mbar_arrive_expect_tx(b_vsfull(vs), C::VS_BYTES);
                        for (int p = 0; p < C::QK_PANELS; ++p)
                            tma_load_3d(sVS + vs * C::VS_BYTES + p * BN * C::PW, &tm_v,
                                        b_vsfull(vs), p * XP, j * BN, bkv);
                    } else {
                        const int vs = j % C::NV;
                        if (j >= C::NV &&
                            !mbar_wait(b_vempty(vs), ((j / C::NV) - 1) & 1, abort_flag, err))
                            break;
                        mbar_arrive_expect_tx(b_vfull(vs), C::V_BYTES);
                        for (int p = 0; p < D / 64; ++p)
                            tma_load_3d(sV + vs * C::V_BYTES + p * BN * 128, &tm_v, b_vfull(vs),
                                        p * 64, j * BN, bkv);
                    }
                    v_issued = j + 1;
                }
                if (*abort_flag) { // let in-flight copies land before the CTA exits
                    if (!withhold_q)
                        mbar_wait_drain(b_qfull, 0);
                    for (int u = max(0, k_issued - C::NK); u < k_issued; ++u)
                        mbar_wait_drain(b_kfull(u % C::NK), (u / C::NK) & 1);
                    if constexpr (F8) {
                        for (int u = max(0, v_issued - C::NVS); u < v_issued; ++u)
                            mbar_wait_drain(b_vsfull(u % C::NVS), (u / C::NVS) & 1);
                    } else {
                        for (int u = max(0, v_issued - C::NV); u < v_issued; ++u)
                            mbar_wait_drain(b_vfull(u % C::NV), (u / C::NV) & 1);
                    }
                }
            }
        } else if (warp >= kConvWarp) {
            // ================================================= V widening (E4M3)
            if constexpr (F8) {
                for (int j = 0; j < nb_max; ++j) {
                    const int ss = j % C::NVS, vs = j % C::NV;
                    if (!mbar_wait_warp(b_vsfull(ss), (j / C::NVS) & 1, abort_flag, err))
                        break;
                    if (j >= C::NV &&
                        !mbar_wait_warp(b_vempty(vs), ((j / C::NV) - 1) & 1, abort_flag, err))
                        break;
                    widen_v_tile<D, BN, C::PW>(sVS + ss * C::VS_BYTES, sV + vs * C::V_BYTES, lane,
                                               warp - kConvWarp, C::NCONV);
                    fence_proxy_async_smem(); // generic writes -> tensor-core reads
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(b_vsempty(ss));
                        mbar_arrive(b_vfull(vs));
                    }
                }
            }
        } else if (warp == kMmaWarp) {
            // ================================================= MMA issuer
            if (lane == 0) {
                constexpr uint32_t idesc_qk = idesc_f16(BM, BN, F8 ? false : BF16, false, false);
                constexpr uint32_t idesc_pv = idesc_f16(BM, D, PB, false, true);
                bool split[NT];
    #pragma unroll
                for (int t = 0; t < NT; ++t)
                    split[t] = tile_split(sh, q0, t);

                // low descriptor words of the operand regions (stepped, see pv_desc)
                constexpr uint32_t hqk = sdesc_kmajor_hi(C::PW);
                const uint32_t lq0 = sdesc_lo(sQ, 16u), lk0 = sdesc_lo(sK, 16u);
                const uint32_t lv0 = pv_base<BN>(sV), lv40 = pv_base4(sV);
                auto issue_qk = [&](int t, int ks) {
                    const uint32_t qa = lq0 + static_cast<uint32_t>((t * C::Q_TILE_BYTES) >> 4);
                    const uint32_t kb = lk0 + static_cast<uint32_t>((ks * C::K_BYTES) >> 4);
    #pragma unroll
                    for (int k = 0; k < D * C::EB / 32; ++k) { // 32-byte K steps
                        const uint32_t byte = k * 32;
                        const uint32_t offa = (byte / C::PW) * (BM * C::PW) + byte % C::PW;
                        const uint32_t offb = (byte / C::PW) * (BN * C::PW) + byte % C::PW;
                        const uint64_t ad = sdesc(qa + (offa >> 4), hqk);
                        const uint64_t bd = sdesc(kb + (offb >> 4), hqk);
                        if constexpr (F8)
                            mma_ss_f8(tmem + C::S_COL(t), ad, bd, idesc_qk, k > 0 ? 1u : 0u);
                        else
                            mma_ss(tmem + C::S_COL(t), ad, bd, idesc_qk, k > 0 ? 1u : 0u);
                    }
                };
                auto issue_pv = [&](int t, int vs, bool first) {
                    const uint32_t voff = static_cast<uint32_t>((vs * C::V_BYTES) >> 4);
                    const uint32_t dv = lv0 + voff, dv4 = lv40 + voff;
    #pragma unroll
                    for (int k = 0; k < BN / 16; ++k) {
                        const uint64_t bd = pv_desc<PAGED, D, BN>(dv, dv4, k, pg.v4);
                        mma_ts(tmem + C::O_COL(t), tmem + C::S_COL(t) + k * 8, bd, idesc_pv,
                               (first && k == 0) ? 0u : 1u);
                    }
                    if (split[t]) {
    #pragma unroll
                        for (int k = 0; k < BN / 16; ++k) {
                            const uint64_t bd = pv_desc<PAGED, D, BN>(dv, dv4, k, pg.v4);
                            mma_ts(tmem + C::O_COL(t), tmem + C::S_COL(t) + 64 + k * 8, bd, idesc_pv,
                                   1u);
                        }
                    }
                };

                bool ok = mbar_wait(b_qfull, 0, abort_flag, err);
                if (ok && nb_max > 0) {
                    ok = mbar_wait(b_kfull(0), 0, abort_flag, err);
                    if (ok) {
                        tc_fence_after();
                        for (int t = 0; t < NT; ++t)
                            if (nb[t] > 0) {
                                issue_qk(t, 0);
                                tc_commit(b_sfull(t));
                            }
                    }
                }
                for (int j = 0; ok && j < nb_max; ++j) {
                    const int vs = j % C::NV;
                    const int kn = j + 1, ks = kn % C::NK;
                    const bool need_k = kn < nb_max;
                    // At d = 128, V(j), K(j+1) and tile 0's P(j) are usually
                    // all there by now: one fused wait instead of three in a
                    // row (each satisfied wait costs the issuing thread ~100
                    // cycles while the tensor core drains its short queue; a
                    // clock64 trace: 305 -> 120-170 cycles, block period
                    // 3070 -> 2930).  At d = 64 the softmax is the bound and
                    // the fused form measured slower, so it waits in turn.
                    constexpr bool kFused = D == 128;
                    // E4M3 inputs (softmax-bound) wait for K(j+1) only where
                    // tile 0's next S product needs it, behind its P.V issue
                    constexpr bool kLateK = kFused && F8;
                    const bool waited =
                        kFused ? mbar_wait3(b_vfull(vs), (j / C::NV) & 1, true, b_kfull(ks),
                                            (kn / C::NK) & 1, need_k && !kLateK, b_pfull(0),
                                            j & 1, j < nb[0], abort_flag, err)
                               : (mbar_wait(b_vfull(vs), (j / C::NV) & 1, abort_flag, err) &&
                                  (!need_k || mbar_wait(b_kfull(ks), (kn / C::NK) & 1,
                                                        abort_flag, err)));
                    if (!waited) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (j < nb[0]) {
                        if (!kFused) {
                            if (!mbar_wait(b_pfull(0), j & 1, abort_flag, err)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        issue_pv(0, vs, j == 0);
                        if constexpr (kLateK) {
                            if (need_k &&
                                !mbar_wait(b_kfull(ks), (kn / C::NK) & 1, abort_flag, err)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        if (kn < nb[0]) {
                            issue_qk(0, ks);
                            tc_commit(b_sfull(0));
                        }
                    } else if constexpr (kLateK) {
                        if (need_k &&
                            !mbar_wait(b_kfull(ks), (kn / C::NK) & 1, abort_flag, err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    if (j < nb[1]) {
                        if (!mbar_wait(b_pfull(1), j & 1, abort_flag, err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_pv(1, vs, j == 0);
                    }
                    if constexpr (!C::SOFTMAX_FREES_V)
                        tc_commit(b_vempty(vs));
                    if (j < nb[1] && kn < nb[1]) {
                        issue_qk(1, ks);
                        tc_commit(b_sfull(1));
                    }
                    // K(j+1) is released by the softmax warps that wait for
                    // the last S product reading it (below)
                }
                if (ok)
                    tc_commit(b_ofull);
                // every MMA this thread issued must finish before tensor memory
                // is released
                tc_commit(b_drain);
                mbar_wait_drain(b_drain, 0);
            }
        }
        // ---- teardown: every tensor-memory access is done before release
        tc_fence_before();
        __syncthreads();
        if (warp == kMmaWarp) {
            tc_fence_after();
            tmem_dealloc(tmem, C::TMEM_COLS);
        }
        return;
    }
    setmaxnreg_inc<kRegsSoftmax>();
    {
        // ================================================= softmax warps
        const int t = warp >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int row_g = q0 + t * BM + r;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + C::S_COL(t);
        const uint32_t tO = tmem + lane_off + C::O_COL(t);
        const int off = sh.n_kv - sh.n_q;
        const bool split = tile_split(sh, q0, t);
        const int r0 = q0 + t * BM;
        // score factor c = scale * log2(e) [* q_scale * k_scale of this
        // (query tile, key block) pair for E4M3 inputs; the next block's k
        // scale is fetched one block ahead]
        // (a tile past the last query row has no blocks and reads no scale)
        const bool live = nb[t] > 0;
        const float cq =
            (F8 && live) ? sh.c * sc.q[static_cast<size_t>(bh) * sc.qh + (r0 / BM) * sc.qb]
                         : sh.c;
        const float *ksc = F8 ? sc.k + static_cast<size_t>(bkv) * sc.kh : nullptr;
        float k_next = (F8 && live) ? ksc[0] : 1.0f;
        float m = -INFINITY, l = 0.f;
        bool ok = true, ref_all = false;

        // The tile whose S product is the last to read each K stage (tile
        // 1, which has at least tile 0's blocks, unless it lies past n_q)
        // releases the stage once its S-full phase has passed: the commit
        // behind it tracks every earlier product of the issuing thread, so
        // no product still reads K(j) -- nor V(j-1), whose P.V products were
        // issued before S(j).  An arrive from this side replaces a commit in
        // the MMA-issuing thread, whose barrier work is what keeps the
        // tensor core idle between products.  (The last V stage of the
        // sequence is never released: nothing waits for it.)
        const bool frees_k = (t == 1 || nb[1] == 0) && quarter == 0 && lane == 0;
        for (int j = 0; j < nb[t]; ++j) {
            const float c = F8 ? cq * k_next : cq;
            if constexpr (F8)
                if (j + 1 < nb[t])
                    k_next = ksc[(j + 1) * sc.kb];
            if (!mbar_wait_warp(b_sfull(t), j & 1, abort_flag, err)) {
                ok = false;
                break;
            }
            if (frees_k) {
                mbar_arrive(b_kempty(j % C::NK));
                if (C::SOFTMAX_FREES_V && j > 0)
                    mbar_arrive(b_vempty((j - 1) % C::NV));
            }
            tc_fence_after();
            float s[BN];
            {
                uint32_t u[BN];
                tmem_ld128(tS, u);
#pragma unroll
                for (int i = 0; i < BN; ++i)
                    s[i] = __uint_as_float(u[i]);
            }
            const int kbase = j * BN;
            const bool need_mask =
                (sh.causal && kbase + BN - 1 > r0 + off) || (kbase + BN > sh.n_kv);
            if (need_mask) {
                int lim = sh.causal ? row_g + off : sh.n_kv - 1;
                lim = min(lim, sh.n_kv - 1) - kbase;
#pragma unroll
                for (int k = 0; k < BN; ++k)
                    if (k > lim)
                        s[k] = -INFINITY;
            }
            // Once every row of the warp has a reference max, P is computed
            // against it straight away: p >= 0, so the block's sum bounds
            // every p, and while no row's sum exceeds kSumLimit the
            // reference stands and the row max is never formed.  Otherwise
            // (a score far above the reference, or a non-finite one) the
            // block is redone from its row max, as for the first block.
            float sum = 0.f, alpha = 1.0f, m_use = m;
            bool kept = false;
            if (ref_all && !split) {
                sum = exp_pack_store<BN, PB, false>(s, c, -m, tS);
                kept = __all_sync(0xffffffffu, sum <= kSumLimit);
            }
            if (!kept) {
                // row max as a tree of three-input maxima: eight independent
                // chains taking two scores per step, then 8 -> 1
                float mx8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    mx8[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
                for (int k = 16; k < BN; k += 2)
                    mx8[(k >> 1) & 7] = max3(mx8[(k >> 1) & 7], s[k], s[k + 1]);
                const float mx = fmaxf(max3(mx8[0], mx8[1], mx8[2]),
                                       fmaxf(max3(mx8[3], mx8[4], mx8[5]),
                                             fmaxf(mx8[6], mx8[7])));
                const float m_blk = mx * c;
                if (m_blk > m + kRescaleThreshold || m == -INFINITY)
                    m_use = fmaxf(m_blk, m);
                alpha = (m_use == m) ? 1.0f : ((m == -INFINITY) ? 0.f : ex2(m - m_use));
                const float neg = (m_use == -INFINITY) ? 0.f : -m_use;
                sum = split ? exp_pack_store<BN, PB, true>(s, c, neg, tS)
                            : exp_pack_store<BN, PB, false>(s, c, neg, tS);
            }
            // O_t holds the sum over earlier blocks (their MMAs completed
            // before S_t of this block was produced); rescale it in place.
            if (!kept && __any_sync(0xffffffffu, alpha != 1.0f) && j > 0) {
#pragma unroll 1
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t u[32];
                    tmem_ld32(tO + ch * 32, u);
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float2 v = __fmul2_rn(
                            make_float2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1])),
                            a2);
                        u[2 * i] = __float_as_uint(v.x);
                        u[2 * i + 1] = __float_as_uint(v.y);
                    }
                    tmem_st32(tO + ch * 32, u);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(b_pfull(t));
            l = l * alpha + sum;
            m = m_use;
            ref_all = __all_sync(0xffffffffu, m != -INFINITY);
        }
        if (ok && nb[t] > 0)
            ok = mbar_wait_warp(b_ofull, 0, abort_flag, err);
        tc_fence_after();
        // 16-bit O of 16-bit inputs leaves through TMA: each warp stages its
        // 32 rows in the tile's Q buffer (free once the O-full barrier has
        // passed: every product has completed) in the Q tile's own swizzled
        // layout and stores them with one tensor copy per 64-column panel, so
        // O reaches L2 as whole lines instead of 16-byte pieces of 32 rows.
        // After an abort the plain stores below write the zero rows (a Q copy
        // might still be landing in that buffer).
        constexpr bool TMA_O = !F8 && OUT != 2;
        if (TMA_O && nb[t] > 0 && ok) {
            const float inv = l > 0.f ? 1.0f / l : 0.f;
            const uint32_t sO = sQ + t * C::Q_TILE_BYTES + quarter * 32 * 128;
#pragma unroll 1
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t u[32];
                tmem_ld32(tO + ch * 32, u);
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[i] = pack2<OUT == 1>(__uint_as_float(u[2 * i]) * inv,
                                           __uint_as_float(u[2 * i + 1]) * inv);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int c = ch * 4 + k; // 16-byte chunk of the row
                    sts_v4(sO + (c / 8) * (BM * 128) + swz_offset<128>(lane, c % 8), w[4 * k],
                           w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
                }
            }
            fence_proxy_async_smem(); // generic writes -> TMA reads
            __syncwarp();
            if (lane == 0) {
#pragma unroll
                for (int p = 0; p < D / 64; ++p)
                    tma_store_3d(&tm_o, sO + p * (BM * 128), p * 64, r0 + quarter * 32, bh);
                bulk_commit_group();
                bulk_wait_group_read0(); // the buffer outlives the copy's reads
            }
            __syncwarp();
            if (lse != nullptr && row_g < sh.n_q)
                lse[static_cast<size_t>(bh) * sh.n_q + row_g] =
                    (m + __log2f(l)) * 0.69314718055994530942f;
        } else if (nb[t] > 0) {
            // ---- epilogue: O = u / l, lse = ln(sum exp(scale * s))
            const bool row_ok = row_g < sh.n_q;
            const float vsc = F8 ? sc.v[bkv] : 1.0f;
            const float inv = (ok && l > 0.f) ? vsc / l : 0.f;
            const size_t orow = (static_cast<size_t>(bh) * sh.n_q + row_g) * D;
#pragma unroll 1
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t u[32];
                tmem_ld32(tO + ch * 32, u);
                if (row_ok) {
                    float o[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        o[i] = ok ? __uint_as_float(u[i]) * inv : 0.f;
                    if constexpr (OUT == 2) {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(O) + orow +
                                                                 ch * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2],
                                                 o[4 * i + 3]);
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(O) + orow +
                                                               ch * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(pack2<OUT == 1>(o[8 * i], o[8 * i + 1]),
                                                pack2<OUT == 1>(o[8 * i + 2], o[8 * i + 3]),
                                                pack2<OUT == 1>(o[8 * i + 4], o[8 * i + 5]),
                                                pack2<OUT == 1>(o[8 * i + 6], o[8 * i + 7]));
                    }
                }
            }
            if (lse != nullptr && row_ok)
                lse[static_cast<size_t>(bh) * sh.n_q + row_g] =
                    ok ? (m + __log2f(l)) * 0.69314718055994530942f
                       : __int_as_float(0x7fc00000);
        }
    }

    // ---- teardown of the softmax warps (tensor memory is released by the
    // MMA warp once every warp has passed this barrier)
    tc_fence_before();
    __syncthreads();
}

} // namespace pf

// ---------------------------------------------------------------------------
// Head size 256.  Two 128-row tiles would need 2 x (128 + 256) tensor-memory
// columns, more than the 512 an SM has, so one CTA owns one query tile and
// the overlap comes from double-buffering S over consecutive key blocks:
// while the softmax warpgroup turns S_(j mod 2) into P, the tensor core
// computes O += P_(j-1) V_(j-1) and S_(j+1).  16-bit inputs use 128-key
// blocks (S buffers of 128 columns, O at 256: 512 in all) with one K and one
// V stage next to Q: 64-key blocks made every score MMA (M = 128, N = 64)
// read 6 KB of shared-memory operands per 131k multiply-adds, more than the
// SM's shared memory delivers, while N = 128 halves that per flop.  E4M3
// inputs keep 64-key blocks (with ten warps a 128-score row would not fit
// the registers) and two stages.
//   warp 4      TMA producer: lane 0 Q once and the K stages, lane 1 the V
//               stages, each waiting only for its own stage (paged calls:
//               Q and K panels 0-1)
//   warp 5      MMA issuer (one thread)
//   warps 6-9   (E4M3 inputs only) widen each V tile to f16, a quarter each
//   warps 6-7   (paged calls only) K panels 2-3; V
//   warps 0-3   softmax, one thread per row; the epilogue
// Tensor memory: S_0 [0,BN), S_1 [BN,2BN), O [2BN, 2BN+256).  A block that moves
// the reference max rescales O only after the previous block's P V product
// has completed (barrier o_done, one phase per product).
namespace pfw {

constexpr int D = 256;
constexpr int BM = 128;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kConvWarp = 6;
// Paged calls: the K and V boxes of a 128-key block (8 units x 4 panels
// each, 2 KB per box) come from three warps -- the producer warp and warps
// 6-7, present only then -- since one warp takes its TMA instructions one
// at a time, and 64 boxes per block from one warp left the tensor core idle
// about two thirds of the time.  (A ninth warp would cap every thread at
// 168 registers, three warps per SM sub-partition, and spill the softmax.)
constexpr int kPagedExtraWarps = 2;

template <bool F8>
struct Cfg {
    // 16-bit: 128-key blocks (N = 128 keeps the score products within the
    // shared-memory operand bandwidth), one K and one V stage next to Q
    static constexpr int BN = F8 ? 64 : 128;
    static constexpr int NK = F8 ? 2 : 1, NV = F8 ? 2 : 1;
    static constexpr int EB = F8 ? 1 : 2;
    static constexpr int PW = 128;
    static constexpr int QK_PANELS = D * EB / PW;
    static constexpr int Q_BYTES = BM * D * EB;
    static constexpr int K_BYTES = BN * D * EB;
    static constexpr int V_BYTES = BN * D * 2;
    static constexpr int VS_BYTES = BN * D;
    static constexpr int NVS = F8 ? 2 : 0;
    static constexpr int NCONV = F8 ? 4 : 0; // V widening warps
    static constexpr int THREADS = 192 + 32 * NCONV;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + NK * K_BYTES;
    static constexpr int OFF_VS = OFF_V + NV * V_BYTES;
    static constexpr int OFF_BAR = OFF_VS + NVS * VS_BYTES;
    // qfull, kfull/kempty, vfull/vempty, vsfull/vsempty, sfull[2], pfull[2],
    // odone, ofull, drain
    static constexpr int NBAR = 1 + 2 * NK + 2 * NV + 2 * NVS + 4 + 3;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 64 + 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};
constexpr int S_COL0 = 0;
constexpr uint32_t TMEM_COLS = 512;

template <int BN>
__device__ __forceinline__ int tile_blocks(const pf::Shape &sh, int r0) {
    const int nkb = (sh.n_kv + BN - 1) / BN;
    if (!sh.causal)
        return nkb;
    const int r_last = min(r0 + BM - 1, sh.n_q - 1);
    return min(nkb, (r_last + (sh.n_kv - sh.n_q)) / BN + 1);
}

template <bool F8, bool PAGED>
constexpr int threads() { return Cfg<F8>::THREADS + (PAGED ? 32 * kPagedExtraWarps : 0); }

template <bool BF16, bool F8, bool PAGED, int OUT>
__global__ void __launch_bounds__(threads<F8, PAGED>(), 1)
    prefill_wide_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_o, void *__restrict__ O,
                        float *__restrict__ lse, const pf::Shape sh_in, const pf::Scales sc,
                        const pf::Paged pg, unsigned *err) {
    using C = Cfg<F8>;
    constexpr int BN = C::BN, NK = C::NK, NV = C::NV, O_COL = 2 * BN;
    static_assert(O_COL + D <= 512, "tensor memory budget");
    static_assert(!(PAGED && F8), "paged prefill reads 16-bit caches");
    pf::Shape sh = sh_in;
    constexpr bool PB = F8 ? false : BF16;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);
    const uint32_t sQ = base_s + C::OFF_Q, sK = base_s + C::OFF_K, sV = base_s + C::OFF_V;
    const uint32_t sVS = base_s + C::OFF_VS;
    const uint32_t bar0 = base_s + C::OFF_BAR;
    const uint32_t b_qfull = bar0;
    auto b_kfull = [&](int i) { return bar0 + 8u * (1 + i); };
    auto b_kempty = [&](int i) { return bar0 + 8u * (1 + NK + i); };
    auto b_vfull = [&](int i) { return bar0 + 8u * (1 + 2 * NK + i); };
    auto b_vempty = [&](int i) { return bar0 + 8u * (1 + 2 * NK + NV + i); };
    auto b_vsfull = [&](int i) { return bar0 + 8u * (1 + 2 * NK + 2 * NV + i); };
    auto b_vsempty = [&](int i) { return bar0 + 8u * (1 + 2 * NK + 2 * NV + C::NVS + i); };
    constexpr int SB = 1 + 2 * NK + 2 * NV + 2 * C::NVS;
    auto b_sfull = [&](int b) { return bar0 + 8u * (SB + b); };
    auto b_pfull = [&](int b) { return bar0 + 8u * (SB + 2 + b); };
    const uint32_t b_odone = bar0 + 8u * (SB + 4);
    const uint32_t b_ofull = b_odone + 8u;
    const uint32_t b_drain = b_ofull + 8u;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + C::OFF_MISC + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int qb, b, h;
    pf::work_item(sh, static_cast<int>(blockIdx.x), qb, b, h);
    if constexpr (PAGED)
        b = pf::longest_first(pg.lens, sh.B, b);
    const int bh = b * sh.Hq + h;
    const int bkv = b * sh.Hkv + h / sh.G;
    const int r0 = qb * BM;
    if constexpr (PAGED) {
        const int len = pf::paged_len_or_reject<D, OUT>(pg, sh, b, bh, r0, BM, O, lse, err);
        if (len < 0)
            return;
        sh.n_kv = len;
    }
    const int nb = tile_blocks<BN>(sh, r0);

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(b_qfull, 1);
        for (int i = 0; i < NK; ++i) {
            mbar_init(b_kfull(i), PAGED ? 2 : 1); // paged: two warps copy K
            mbar_init(b_kempty(i), 1);
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(b_vfull(i), F8 ? C::NCONV : 1);
            mbar_init(b_vempty(i), 1);
        }
        for (int i = 0; i < C::NVS; ++i) {
            mbar_init(b_vsfull(i), 1);
            mbar_init(b_vsempty(i), C::NCONV);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(b_sfull(i), 1);
            mbar_init(b_pfull(i), 4);
        }
        mbar_init(b_odone, 1);
        mbar_init(b_ofull, 1);
        mbar_init(b_drain, 1);
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (PAGED && (warp == kProducerWarp || warp >= kConvWarp)) {
        // ================================================= paged producers
        // (panels of each 512-byte row) warp 4: Q, K 0-1; warp 6: K 2-3;
        // warp 7: V 0-3.  No warp copies both tensors: with one K and one V
        // stage, a K copy queued behind a V-empty wait would hold the next
        // block's scores back until the previous block's P V had finished.
        static_assert(!PAGED || C::NCONV == 0, "paged inputs are 16-bit");
        if (warp == kProducerWarp) {
            if (lane == 0) {
                mbar_arrive_expect_tx(b_qfull, C::Q_BYTES);
                for (int p = 0; p < C::QK_PANELS; ++p)
                    tma_load_3d(sQ + p * BM * C::PW, &tm_q, b_qfull, p * 64, r0, bh);
            }
            pf::paged_kv_producer<D, BN, NK, NV, 0, 2, 0, 0>(
                pg, b, h / sh.G, sh.Hkv, sh.n_kv, nb, &tm_k, &tm_v, sK, sV, b_kfull(0),
                b_kempty(0), b_vfull(0), b_vempty(0), abort_flag, err, lane);
            if (lane == 0 && *abort_flag)
                mbar_wait_drain(b_qfull, 0);
        } else if (warp == kConvWarp) {
            pf::paged_kv_producer<D, BN, NK, NV, 2, 4, 0, 0>(
                pg, b, h / sh.G, sh.Hkv, sh.n_kv, nb, &tm_k, &tm_v, sK, sV, b_kfull(0),
                b_kempty(0), b_vfull(0), b_vempty(0), abort_flag, err, lane);
        } else {
            pf::paged_kv_producer<D, BN, NK, NV, 0, 0, 0, 4>(
                pg, b, h / sh.G, sh.Hkv, sh.n_kv, nb, &tm_k, &tm_v, sK, sV, b_kfull(0),
                b_kempty(0), b_vfull(0), b_vempty(0), abort_flag, err, lane);
        }
    } else if (warp == kProducerWarp) {
        // ================================================= TMA producer
        // lane 0 streams Q and K, lane 1 streams V: each waits only for its
        // own stage, so a single-stage K never queues behind a V wait
        constexpr int XP = C::PW / C::EB;
        if (lane == 0) {
            // test hook, as in the d <= 128 kernel: without the Q copy the MMA
            // issuer's first wait expires and every role unwinds
            const bool withhold_q =
                (*reinterpret_cast<const volatile unsigned *>(err + CTL_HOOKS) &
                 HOOK_WITHHOLD_Q) != 0u;
            if (!withhold_q) {
                mbar_arrive_expect_tx(b_qfull, C::Q_BYTES);
                for (int p = 0; p < C::QK_PANELS; ++p)
                    tma_load_3d(sQ + p * BM * C::PW, &tm_q, b_qfull, p * XP, r0, bh);
            }
            int k_issued = 0;
            for (int j = 0; j < nb; ++j) {
                const int ks = j % NK;
                if (j >= NK && !mbar_wait(b_kempty(ks), ((j / NK) - 1) & 1, abort_flag, err))
                    break;
                mbar_arrive_expect_tx(b_kfull(ks), C::K_BYTES);
                for (int p = 0; p < C::QK_PANELS; ++p)
                    tma_load_3d(sK + ks * C::K_BYTES + p * BN * C::PW, &tm_k, b_kfull(ks),
                                p * XP, j * BN, bkv);
                k_issued = j + 1;
            }
            if (*abort_flag) { // let in-flight copies land before the CTA exits
                if (!withhold_q)
                    mbar_wait_drain(b_qfull, 0);
                for (int u = max(0, k_issued - NK); u < k_issued; ++u)
                    mbar_wait_drain(b_kfull(u % NK), (u / NK) & 1);
            }
        } else if (lane == 1) {
            int v_issued = 0;
            for (int j = 0; j < nb; ++j) {
                if constexpr (F8) {
                    const int vs = j % C::NVS;
                    if (j >= C::NVS &&
                        !mbar_wait(b_vsempty(vs), ((j / C::NVS) - 1) & 1, abort_flag, err))
                        break;
                    mbar_arrive_expect_tx(b_vsfull(vs), C::VS_BYTES);
                    for (int p = 0; p < C::QK_PANELS; ++p)
                        tma_load_3d(sVS + vs * C::VS_BYTES + p * BN * C::PW, &tm_v,
                                    b_vsfull(vs), p * XP, j * BN, bkv);
                } else {
                    const int vs = j % NV;
                    if (j >= NV && !mbar_wait(b_vempty(vs), ((j / NV) - 1) & 1, abort_flag, err))
                        break;
                    mbar_arrive_expect_tx(b_vfull(vs), C::V_BYTES);
                    for (int p = 0; p < D / 64; ++p)
                        tma_load_3d(sV + vs * C::V_BYTES + p * BN * 128, &tm_v, b_vfull(vs),
                                    p * 64, j * BN, bkv);
                }
                v_issued = j + 1;
            }
            if (*abort_flag) {
                if constexpr (F8) {
                    for (int u = max(0, v_issued - C::NVS); u < v_issued; ++u)
                        mbar_wait_drain(b_vsfull(u % C::NVS), (u / C::NVS) & 1);
                } else {
                    for (int u = max(0, v_issued - NV); u < v_issued; ++u)
                        mbar_wait_drain(b_vfull(u % NV), (u / NV) & 1);
                }
            }
        }
    } else if (warp >= kConvWarp) {
        // ================================================= V widening (E4M3)
        if constexpr (F8) {
            for (int j = 0; j < nb; ++j) {
                const int ss = j % C::NVS, vs = j % NV;
                if (!mbar_wait_warp(b_vsfull(ss), (j / C::NVS) & 1, abort_flag, err))
                    break;
                if (j >= NV && !mbar_wait_warp(b_vempty(vs), ((j / NV) - 1) & 1, abort_flag, err))
                    break;
                pf::widen_v_tile<D, BN, C::PW>(sVS + ss * C::VS_BYTES, sV + vs * C::V_BYTES,
                                               lane, warp - kConvWarp, C::NCONV);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(b_vsempty(ss));
                    mbar_arrive(b_vfull(vs));
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ================================================= MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_f16(BM, BN, F8 ? false : BF16, false, false);
            constexpr uint32_t idesc_pv = idesc_f16(BM, D, PB, false, true);
            const bool split = (sh.causal ? (r0 + (sh.n_kv - sh.n_q) + 1) : sh.n_kv) <
                               pf::kSplitKeys;
            // low descriptor words of the operand regions (stepped, see pf::pv_desc)
            constexpr uint32_t hqk = sdesc_kmajor_hi(C::PW);
            const uint32_t lq0 = sdesc_lo(sQ, 16u), lk0 = sdesc_lo(sK, 16u);
            const uint32_t lv0 = pf::pv_base<BN>(sV), lv40 = pf::pv_base4(sV);
            auto issue_qk = [&](int buf, int ks) {
                const uint32_t kb = lk0 + static_cast<uint32_t>((ks * C::K_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < D * C::EB / 32; ++k) {
                    const uint32_t byte = k * 32;
                    const uint32_t offa = (byte / C::PW) * (BM * C::PW) + byte % C::PW;
                    const uint32_t offb = (byte / C::PW) * (BN * C::PW) + byte % C::PW;
                    const uint64_t ad = sdesc(lq0 + (offa >> 4), hqk);
                    const uint64_t bd = sdesc(kb + (offb >> 4), hqk);
                    if constexpr (F8)
                        mma_ss_f8(tmem + S_COL0 + buf * BN, ad, bd, idesc_qk, k > 0 ? 1u : 0u);
                    else
                        mma_ss(tmem + S_COL0 + buf * BN, ad, bd, idesc_qk, k > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int buf, int vs, bool first) {
                const uint32_t voff = static_cast<uint32_t>((vs * C::V_BYTES) >> 4);
                const uint32_t dv = lv0 + voff, dv4 = lv40 + voff;
#pragma unroll
                for (int k = 0; k < BN / 16; ++k) {
                    const uint64_t bd = pf::pv_desc<PAGED, D, BN>(dv, dv4, k, pg.v4);
                    mma_ts(tmem + O_COL, tmem + S_COL0 + buf * BN + k * 8, bd, idesc_pv,
                           (first && k == 0) ? 0u : 1u);
                }
                if (split) {
#pragma unroll
                    for (int k = 0; k < BN / 16; ++k) {
                        const uint64_t bd = pf::pv_desc<PAGED, D, BN>(dv, dv4, k, pg.v4);
                        mma_ts(tmem + O_COL, tmem + S_COL0 + buf * BN + BN / 2 + k * 8, bd,
                               idesc_pv, 1u);
                    }
                }
            };
            bool ok = mbar_wait(b_qfull, 0, abort_flag, err);
            // S for the first two blocks
            for (int j = 0; ok && j < min(2, nb); ++j) {
                ok = mbar_wait(b_kfull(j % NK), (j / NK) & 1, abort_flag, err);
                if (!ok)
                    break;
                tc_fence_after();
                issue_qk(j & 1, j % NK);
                tc_commit(b_sfull(j & 1));
                tc_commit(b_kempty(j % NK));
            }
            for (int j = 0; ok && j < nb; ++j) {
                const int buf = j & 1, vs = j % NV;
                if (!mbar_wait(b_vfull(vs), (j / NV) & 1, abort_flag, err) ||
                    !mbar_wait(b_pfull(buf), (j >> 1) & 1, abort_flag, err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_pv(buf, vs, j == 0);
                tc_commit(b_vempty(vs));
                tc_commit(b_odone);
                const int jn = j + 2;
                if (jn < nb) {
                    if (!mbar_wait(b_kfull(jn % NK), (jn / NK) & 1, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_qk(buf, jn % NK);
                    tc_commit(b_sfull(buf));
                    tc_commit(b_kempty(jn % NK));
                }
            }
            if (ok)
                tc_commit(b_ofull);
            tc_commit(b_drain);
            mbar_wait_drain(b_drain, 0);
        }
    } else {
        // ================================================= softmax warps
        const int r = warp * 32 + lane;
        const int row_g = r0 + r;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t tO = tmem + lane_off + O_COL;
        const int off = sh.n_kv - sh.n_q;
        const bool split = (sh.causal ? (r0 + off + 1) : sh.n_kv) < pf::kSplitKeys;
        // per (query tile, key block) score factor, as in the d <= 128 kernel;
        // a 128-key scale block spans 128 / BN of this kernel's key blocks
        const float cq =
            F8 ? sh.c * sc.q[static_cast<size_t>(bh) * sc.qh + (r0 / BM) * sc.qb] : sh.c;
        const float *ksc = F8 ? sc.k + static_cast<size_t>(bkv) * sc.kh : nullptr;
        float k_next = (F8 && nb > 0) ? ksc[0] : 1.0f;
        float m = -INFINITY, l = 0.f;
        bool ok = true, ref_all = false;
        for (int j = 0; j < nb; ++j) {
            const float c = F8 ? cq * k_next : cq;
            if constexpr (F8)
                if (j + 1 < nb)
                    k_next = ksc[((j + 1) * BN / 128) * sc.kb];
            const int buf = j & 1;
            const uint32_t tS = tmem + lane_off + S_COL0 + buf * BN;
            if (!mbar_wait_warp(b_sfull(buf), (j >> 1) & 1, abort_flag, err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[BN];
            {
                uint32_t u[BN];
                if constexpr (BN == 128)
                    tmem_ld128(tS, u);
                else
                    tmem_ld64(tS, u);
#pragma unroll
                for (int i = 0; i < BN; ++i)
                    s[i] = __uint_as_float(u[i]);
            }
            const int kbase = j * BN;
            if ((sh.causal && kbase + BN - 1 > r0 + off) || (kbase + BN > sh.n_kv)) {
                int lim = sh.causal ? row_g + off : sh.n_kv - 1;
                lim = min(lim, sh.n_kv - 1) - kbase;
#pragma unroll
                for (int k = 0; k < BN; ++k)
                    if (k > lim)
                        s[k] = -INFINITY;
            }
            // P against the reference max first, kept while no row's sum
            // exceeds the limit; else redone from the row max, as in the
            // d <= 128 kernel
            float sum = 0.f, alpha = 1.0f, m_use = m;
            bool kept = false;
            if (ref_all && !split) {
                sum = pf::exp_pack_store<BN, PB, false>(s, c, -m, tS);
                kept = __all_sync(0xffffffffu, sum <= pf::kSumLimit);
            }
            if (!kept) {
                float mx8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    mx8[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
                for (int k = 16; k < BN; k += 2)
                    mx8[(k >> 1) & 7] = max3(mx8[(k >> 1) & 7], s[k], s[k + 1]);
                const float mx = fmaxf(max3(mx8[0], mx8[1], mx8[2]),
                                       fmaxf(max3(mx8[3], mx8[4], mx8[5]),
                                             fmaxf(mx8[6], mx8[7])));
                const float m_blk = mx * c;
                if (m_blk > m + pf::kRescaleThreshold || m == -INFINITY)
                    m_use = fmaxf(m_blk, m);
                alpha = (m_use == m) ? 1.0f : ((m == -INFINITY) ? 0.f : ex2(m - m_use));
                const float neg = (m_use == -INFINITY) ? 0.f : -m_use;
                if (__any_sync(0xffffffffu, alpha != 1.0f) && j > 0) {
                    // O must hold exactly the blocks before j: wait for P_(j-1) V_(j-1)
                    if (!mbar_wait_warp(b_odone, (j - 1) & 1, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int ch = 0; ch < D / 32; ++ch) {
                        uint32_t u[32];
                        tmem_ld32(tO + ch * 32, u);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
                        tmem_st32(tO + ch * 32, u);
                    }
                }
                sum = split ? pf::exp_pack_store<BN, PB, true>(s, c, neg, tS)
                            : pf::exp_pack_store<BN, PB, false>(s, c, neg, tS);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(b_pfull(buf));
            l = l * alpha + sum;
            m = m_use;
            ref_all = __all_sync(0xffffffffu, m != -INFINITY);
        }
        if (ok && nb > 0)
            ok = mbar_wait_warp(b_ofull, 0, abort_flag, err);
        tc_fence_after();
        // 16-bit O of 16-bit inputs: each warp stages its 32 rows in the Q
        // buffer (free once O-full has passed) and stores them by TMA, as in
        // pf::prefill_kernel; after an abort the plain stores write zeros
        constexpr bool TMA_O = !F8 && OUT != 2;
        if (TMA_O && ok && nb > 0) {
            const float inv = l > 0.f ? 1.0f / l : 0.f;
            const uint32_t sO = sQ + warp * 32 * 128;
#pragma unroll 1
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t u[32];
                tmem_ld32(tO + ch * 32, u);
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[i] = pack2<OUT == 1>(__uint_as_float(u[2 * i]) * inv,
                                           __uint_as_float(u[2 * i + 1]) * inv);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int c = ch * 4 + k; // 16-byte chunk of the row
                    sts_v4(sO + (c / 8) * (BM * 128) + swz_offset<128>(lane, c % 8), w[4 * k],
                           w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
                }
            }
            fence_proxy_async_smem(); // generic writes -> TMA reads
            __syncwarp();
            if (lane == 0) {
#pragma unroll
                for (int p = 0; p < D / 64; ++p)
                    tma_store_3d(&tm_o, sO + p * (BM * 128), p * 64, r0 + warp * 32, bh);
                bulk_commit_group();
                bulk_wait_group_read0(); // the buffer outlives the copy's reads
            }
            __syncwarp();
            if (lse != nullptr && row_g < sh.n_q)
                lse[static_cast<size_t>(bh) * sh.n_q + row_g] =
                    (m + __log2f(l)) * 0.69314718055994530942f;
        } else {
            const bool row_ok = row_g < sh.n_q;
            const float vsc = F8 ? sc.v[bkv] : 1.0f;
            const float inv = (ok && l > 0.f) ? vsc / l : 0.f;
            const size_t orow = (static_cast<size_t>(bh) * sh.n_q + row_g) * D;
#pragma unroll 1
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t u[32];
                tmem_ld32(tO + ch * 32, u);
                if (row_ok) {
                    float o[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        o[i] = ok ? __uint_as_float(u[i]) * inv : 0.f;
                    if constexpr (OUT == 2) {
                        float4 *dst =
                            reinterpret_cast<float4 *>(static_cast<float *>(O) + orow + ch * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                    } else {
                        uint4 *dst =
                            reinterpret_cast<uint4 *>(static_cast<uint16_t *>(O) + orow + ch * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(pack2<OUT == 1>(o[8 * i], o[8 * i + 1]),
                                                pack2<OUT == 1>(o[8 * i + 2], o[8 * i + 3]),
                                                pack2<OUT == 1>(o[8 * i + 4], o[8 * i + 5]),
                                                pack2<OUT == 1>(o[8 * i + 6], o[8 * i + 7]));
                    }
                }
            }
            if (lse != nullptr && row_ok)
                lse[static_cast<size_t>(bh) * sh.n_q + row_g] =
                    ok ? (m + __log2f(l)) * 0.69314718055994530942f : __int_as_float(0x7fc00000);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

} // namespace pfw

// ------------------------------------------------------------------ host

// [d, n, bh] tensor map: 16-bit elements in 128-byte (64-element) panel
// rows, or E4M3 bytes in min(d, 128)-byte panel rows; `rows` per box, the
// panel width as swizzle span, zero fill past n.
static bool make_map(CUtensorMap *m, const void *ptr, int d, int n, int bh, bool bf16, bool f8,
                     int rows) {
    const uint64_t esz = f8 ? 1 : 2;
    const int pw = f8 ? (d < 128 ? d : 128) : 128;
    const uint64_t dims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(n),
                              static_cast<uint64_t>(bh)};
    const uint64_t strides[2] = {static_cast<uint64_t>(d) * esz,
                                 static_cast<uint64_t>(d) * esz * static_cast<uint64_t>(n)};
    const uint32_t box[3] = {static_cast<uint32_t>(pw / esz), static_cast<uint32_t>(rows), 1};
    const TmapElem el = f8 ? TmapElem::U8 : (bf16 ? TmapElem::BF16 : TmapElem::F16);
    return make_tmap_3d(m, ptr, el, dims, strides, box, pw);
}

// K / V bytes the CTAs of one group of the grid order may share through L2
// (a third of its 126 MB).
#ifndef ATTN_KV_GROUP_BYTES
#define ATTN_KV_GROUP_BYTES (40ll << 20)
#endif

// (batch, KV head) pairs per group of the CTA order (pf::work_item): as many
// as keep the group's K / V within ATTN_KV_GROUP_BYTES, at least one (for a
// paged cache, sized by the longest sequence the call allows).
static int kv_group(const PrefillArgs &a) {
    const long long pairs = static_cast<long long>(a.B) * a.Hkv;
    const long long esz = a.e4m3 ? 1 : 2;
    const long long per_pair = 2ll * (a.paged ? a.max_seq_len : a.n_kv) * a.d * esz;
    const long long g = ATTN_KV_GROUP_BYTES / (per_pair > 0 ? per_pair : 1);
    return static_cast<int>(g < 1 ? 1 : (g > pairs ? pairs : g));
}

static pf::Shape make_shape(const PrefillArgs &a, int rows_per_cta) {
    pf::Shape sh;
    sh.kvg = kv_group(a);
    sh.B = a.B;
    sh.Hq = a.Hq;
    sh.Hkv = a.Hkv;
    sh.G = a.Hq / a.Hkv;
    sh.n_q = a.n_q;
    sh.n_kv = a.n_kv;
    sh.causal = a.causal;
    sh.nqb = (a.n_q + rows_per_cta - 1) / rows_per_cta;
    sh.c = a.scale * 1.4426950408889634f;
    sh.scale = a.scale;
    return sh;
}

// E4M3 scale indexing: per head (stride 1, no block step) or per 128-row
// block (one row of ceil(n / 128) scales per head).
static pf::Scales make_scales(const PrefillArgs &a) {
    pf::Scales sc{a.q_scale, a.k_scale, a.v_scale, 1, 0, 1, 0};
    if (a.e4m3_blocks) {
        sc.qh = (a.n_q + 127) / 128;
        sc.qb = 1;
        sc.kh = (a.n_kv + 127) / 128;
        sc.kb = 1;
    }
    return sc;
}

// Cache [num_blocks, Hkv, bs, d] (16-bit) viewed as {d, Hkv * bs, num_blocks},
// box 64 x bs x 1 (one panel of one head's cache block), 128-byte swizzle.
static bool make_cache_map(CUtensorMap *m, const void *ptr, const PrefillArgs &a) {
    const uint64_t dims[3] = {static_cast<uint64_t>(a.d),
                              static_cast<uint64_t>(a.Hkv) * a.block_size,
                              static_cast<uint64_t>(a.num_blocks)};
    const uint64_t strides[2] = {static_cast<uint64_t>(a.d) * 2,
                                 static_cast<uint64_t>(a.Hkv) * a.block_size * a.d * 2};
    const uint32_t box[3] = {64, static_cast<uint32_t>(a.block_size), 1};
    return make_tmap_3d(m, ptr, a.bf16 ? TmapElem::BF16 : TmapElem::F16, dims, strides, box, 128);
}

// Paged V by one 4-D box per cache block: d = 256 with 16-token blocks.
static bool paged_v4(const PrefillArgs &a) {
    return a.paged && a.d == 256 && a.block_size == 16;
}

// The V cache viewed as {64, Hkv * bs, d / 64, num_blocks}: the third
// dimension steps through a row's 128-byte panels, so that one box
// {64, bs, d / 64, 1} lands a cache block as [panel][token] swizzled blocks.
static bool make_cache_map_v(CUtensorMap *m, const void *ptr, const PrefillArgs &a) {
    const uint64_t dims[4] = {64, static_cast<uint64_t>(a.Hkv) * a.block_size,
                              static_cast<uint64_t>(a.d / 64), static_cast<uint64_t>(a.num_blocks)};
    const uint64_t strides[3] = {static_cast<uint64_t>(a.d) * 2, 128,
                                 static_cast<uint64_t>(a.Hkv) * a.block_size * a.d * 2};
    const uint32_t box[4] = {64, static_cast<uint32_t>(a.block_size),
                             static_cast<uint32_t>(a.d / 64), 1};
    return make_tmap_4d(m, ptr, a.bf16 ? TmapElem::BF16 : TmapElem::F16, dims, strides, box, 128);
}

static bool make_kv_maps(CUtensorMap *mk, CUtensorMap *mv, const PrefillArgs &a, int D, bool bf16,
                         bool f8, int rows) {
    if (a.paged) // V: one box per cache block at d = 256 with 16-token blocks (Paged::v4)
        return make_cache_map(mk, a.K, a) &&
               (paged_v4(a) ? make_cache_map_v(mv, a.V, a) : make_cache_map(mv, a.V, a));
    return make_map(mk, a.K, D, a.n_kv, a.B * a.Hkv, bf16, f8, rows) &&
           make_map(mv, a.V, D, a.n_kv, a.B * a.Hkv, bf16, f8, rows);
}

static pf::Paged make_paged(const PrefillArgs &a) {
    pf::Paged pg{};
    if (a.paged) {
        pg.table = a.block_table;
        pg.lens = a.seq_lens;
        pg.vcache = static_cast<const uint8_t *>(a.V);
        pg.bs = a.block_size;
        pg.max_blocks = a.max_blocks;
        pg.num_blocks = a.num_blocks;
        pg.max_len = a.max_seq_len;
        pg.v4 = paged_v4(a) ? 1 : 0;
    }
    return pg;
}

template <int D, bool BF16, bool F8, bool PAGED, int OUT>
static cudaError_t launch_prefill_t(const PrefillArgs &a, cudaStream_t st) {
    using C = pf::Cfg<D, F8>;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, a.Q, D, a.n_q, a.B * a.Hq, BF16, F8, pf::BM) ||
        !make_kv_maps(&mk, &mv, a, D, BF16, F8, pf::BN))
        return cudaErrorInvalidValue;
    // O [B * Hq, n_q, D] in its 16-bit format, 32-row boxes (one warp's rows)
    // for the TMA-stored epilogue; fp32 and E4M3-input calls store directly
    // and never read this map
    if (!F8 && OUT != 2) {
        if (!make_map(&mo, a.O, D, a.n_q, a.B * a.Hq, OUT == 1, false, 32))
            return cudaErrorInvalidValue;
    } else {
        mo = mq;
    }
    const pf::Shape sh = make_shape(a, pf::NT * pf::BM);
    const pf::Scales sc = make_scales(a);
    auto kern = pf::prefill_kernel<D, BF16, F8, PAGED, OUT>;
    // the in-kernel register split adds up only if the kernel launches with
    // exactly kLaunchRegs registers per thread; never launch it otherwise.
    // The count is looked up once per instance; concurrent callers may race
    // to store the same value, which the atomic makes well defined.
    static std::atomic<int> regs_cache{-1};
    int regs = regs_cache.load(std::memory_order_relaxed);
    if (regs < 0) {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess)
            return cudaErrorInvalidDeviceFunction;
        regs = fa.numRegs;
        regs_cache.store(regs, std::memory_order_relaxed);
    }
    if (regs != pf::kLaunchRegs)
        return cudaErrorInvalidConfiguration;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess)
        return e;
    const long long grid = static_cast<long long>(sh.nqb) * a.B * a.Hq;
    if (grid > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, st>>>(mq, mk, mv, mo, a.O, a.lse, sh,
                                                                  sc, make_paged(a), a.err);
    return cudaGetLastError();
}

template <bool BF16, bool F8, bool PAGED, int OUT>
static cudaError_t launch_prefill_wide(const PrefillArgs &a, cudaStream_t st) {
    using C = pfw::Cfg<F8>;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, a.Q, pfw::D, a.n_q, a.B * a.Hq, BF16, F8, pfw::BM) ||
        !make_kv_maps(&mk, &mv, a, pfw::D, BF16, F8, pfw::Cfg<F8>::BN))
        return cudaErrorInvalidValue;
    if (!F8 && OUT != 2) { // 32-row boxes of O for the TMA-stored epilogue
        if (!make_map(&mo, a.O, pfw::D, a.n_q, a.B * a.Hq, OUT == 1, false, 32))
            return cudaErrorInvalidValue;
    } else {
        mo = mq;
    }
    const pf::Shape sh = make_shape(a, pfw::BM);
    const pf::Scales sc = make_scales(a);
    auto kern = pfw::prefill_wide_kernel<BF16, F8, PAGED, OUT>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess)
        return e;
    const long long grid = static_cast<long long>(sh.nqb) * a.B * a.Hq;
    if (grid > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    kern<<<static_cast<unsigned>(grid), pfw::threads<F8, PAGED>(), C::SMEM, st>>>(
        mq, mk, mv, mo, a.O, a.lse, sh, sc, make_paged(a), a.err);
    return cudaGetLastError();
}

template <int D, bool BF16, bool F8, bool PAGED>
static cudaError_t launch_out(const PrefillArgs &a, cudaStream_t st) {
    if constexpr (D == 256) {
        switch (a.out_dtype) {
        case 0: return launch_prefill_wide<BF16, F8, PAGED, 0>(a, st);
        case 1: return launch_prefill_wide<BF16, F8, PAGED, 1>(a, st);
        default: return launch_prefill_wide<BF16, F8, PAGED, 2>(a, st);
        }
    } else {
        switch (a.out_dtype) {
        case 0: return launch_prefill_t<D, BF16, F8, PAGED, 0>(a, st);
        case 1: return launch_prefill_t<D, BF16, F8, PAGED, 1>(a, st);
        default: return launch_prefill_t<D, BF16, F8, PAGED, 2>(a, st);
        }
    }
}

template <int D>
static cudaError_t launch_d(const PrefillArgs &a, cudaStream_t st) {
    if (a.paged)
        return a.bf16 ? launch_out<D, true, false, true>(a, st)
                      : launch_out<D, false, false, true>(a, st);
    if (a.e4m3)
        return launch_out<D, false, true, false>(a, st);
    return a.bf16 ? launch_out<D, true, false, false>(a, st)
                  : launch_out<D, false, false, false>(a, st);
}

cudaError_t prefill_launch(const PrefillArgs &a, cudaStream_t st) {
    switch (a.d) {
    case 64: return launch_d<64>(a, st);
    case 128: return launch_d<128>(a, st);
    case 256: return launch_d<256>(a, st);
    }
    return cudaErrorInvalidValue;
}

} // namespace attn
