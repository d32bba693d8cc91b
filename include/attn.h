/*
 * attn.h -- C ABI of libattn.so: exact IO-aware attention on B300 (sm_103a).
 *
 * What is computed (all entry points): scaled dot-product attention
 *     O = softmax(scale * Q K^T [masked]) V
 * (auturnal.com, "From attention to IO-aware execution", §2; papanda925.com,
 * "Transformer complexity strategies", standard-attention pseudocode),
 * evaluated tile by tile with the online-softmax statistics of §8 of the
 * first page: a running max m, denominator l and un-normalised sum u per
 * query row, rescaled by exp(m - m') whenever a block raises the max, u / l
 * emitted at the end.  The n_q x n_kv score matrix never reaches device
 * memory.
 *
 * Conventions shared by every call
 *  - Every pointer argument is a DEVICE pointer unless stated otherwise; the
 *    caller owns every buffer.  The library keeps no allocation of its own
 *    beyond one 4-byte device error word per device (plus the scratch array
 *    of attn_decode_static_ws, and the three streams and event set that
 *    attn_prefill_from_host creates per device on first use).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls are asynchronous on that stream; results are valid once
 *    the stream has reached the call.
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns ATTN_ERR_INVALID (or ATTN_ERR_UNSUPPORTED for a valid
 *    but unimplemented combination) and launches nothing.  A launch failure
 *    returns ATTN_ERR_CUDA.
 *  - Errors that only the device can see (a block-table entry out of range,
 *    a sequence longer than the table, a bounded wait that expired) are
 *    recorded in the device error word and the affected output is written
 *    as zeros; attn_last_error() reports and clears them.
 *  - Tensors are contiguous, innermost dimension last, 16-byte aligned.
 *  - GQA: query head h reads KV head h / (Hq / Hkv)
 *    (code-journey.com, "Attention co-design", Group Size: G query heads
 *    share one KV head; G = 1 is MHA).
 *  - Causal masks are aligned bottom-right: query i sees key j iff
 *    j <= i + (n_kv - n_q) (marketmaker.cc, "Flash Attention and sequence
 *    length", causal masking; the pages do not fix the alignment for
 *    n_q != n_kv, this reading makes a decode query see the whole cache).
 *  - lse, when requested, is the natural log-sum-exp of the row's scaled
 *    scores, ln sum_j exp(scale * q.k_j), in fp32.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID = 1,     /* bad argument (host check) or bad index (device) */
    ATTN_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. head size) */
    ATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
    ATTN_ERR_TIMEOUT = 4      /* a bounded device-side wait expired */
} attn_status;

typedef enum {
    ATTN_F16 = 0,
    ATTN_BF16 = 1,
    ATTN_F32 = 2,
    ATTN_E4M3 = 3 /* OCP FP8 E4M3 ("fn"), one fp32 scale per KV head */
} attn_dtype;

/* Prefill / full attention.
 *   Q   [B, Hq,  n_q,  d]   in_dtype (F16, BF16 or E4M3)
 *   K,V [B, Hkv, n_kv, d]   in_dtype
 *   O   [B, Hq,  n_q,  d]   out_dtype (F16, BF16 or F32)
 *   lse [B, Hq,  n_q]       fp32, or NULL
 *   q_scale [B * Hq], k_scale, v_scale [B * Hkv]: fp32 per-head scales of
 *           an E4M3 input (dequantised value = code * scale); NULL for
 *           16-bit inputs.  With E4M3 inputs q K^T runs on the 8-bit tensor
 *           cores and P V in f16 (V widened on chip, exactly).
 * d in {64, 128, 256}; Hq % Hkv == 0; causal requires n_q <= n_kv.
 * scale is the factor applied to q.k (1/sqrt(d) for the textbook form).
 * Host-side errors: ATTN_ERR_INVALID for null pointers (scales included for
 * E4M3), non-positive sizes, misalignment, Hq % Hkv != 0, causal with
 * n_q > n_kv; ATTN_ERR_UNSUPPORTED for other d or dtype combinations.  One
 * kernel launch. */
ATTN_API attn_status attn_prefill(const void *Q, const void *K, const void *V, void *O,
                         float *lse, int B, int Hq, int Hkv, int n_q, int n_kv,
                         int d, int causal, float scale, attn_dtype in_dtype,
                         attn_dtype out_dtype, const float *q_scale,
                         const float *k_scale, const float *v_scale, void *stream);

/* Size of the row blocks that carry one E4M3 scale in
 * attn_prefill_e4m3_blocks and attn_rotate_quantize_e4m3 (the prefill's
 * query tile and key block). */
#define ATTN_E4M3_SCALE_BLOCK 128

/* attn_prefill for E4M3 Q, K, V with block-wise scales on Q and K
 * (marketmaker.cc, "Flash Attention and sequence length", FA3 item 3:
 * block-wise fp8 quantisation, after the rotation of
 * attn_rotate_quantize_e4m3 or without it).  Rows 128 b .. 128 b + 127 of
 * a head of Q (of K) share one scale:
 *   q_scale [B * Hq,  ceil(n_q  / 128)] fp32: q_scale[bh][b] for query rows of
 *           block b of head bh (bh = batch * Hq + head);
 *   k_scale [B * Hkv, ceil(n_kv / 128)] fp32, likewise for keys;
 *   v_scale [B * Hkv] fp32: one scale per KV head (V is not rotated).
 * Dequantised value = code * scale.  The score of query i and key j is
 * formed as scale * q_scale[bh][i/128] * k_scale[bkv][j/128] * (codes q_i .
 * k_j), so each (query tile, key block) pair of score tiles carries one
 * scale product.  Q [B, Hq, n_q, d], K, V [B, Hkv, n_kv, d] E4M3; O, lse,
 * sizes, checks and errors as attn_prefill (the scale arrays' sizes are the
 * caller's responsibility).  One kernel launch. */
ATTN_API attn_status attn_prefill_e4m3_blocks(const void *Q, const void *K, const void *V,
                                              void *O, float *lse, int B, int Hq, int Hkv,
                                              int n_q, int n_kv, int d, int causal, float scale,
                                              attn_dtype out_dtype, const float *q_scale,
                                              const float *k_scale, const float *v_scale,
                                              void *stream);

/* attn_prefill with Q, K, V starting in host memory and O (and lse) ending
 * there, the host<->device copies overlapped with the attention kernels
 * (auturnal.com, "From attention to IO-aware execution" §10: the slowest
 * memory level sets the pace -- here the host link).  The B*Hq heads are
 * split into chunks of consecutive (batch, head) pairs, whole KV-head groups
 * or an exact part of one; chunk c's Q (and the K, V of KV heads that begin
 * in it) is copied in on a library-owned stream, its attention runs once the
 * copy has landed, and its O / lse are copied out on a second library-owned
 * stream once it is done, so that copy-in, attention and copy-out of
 * neighbouring chunks run at the same time.
 *   Q_host, K_host, V_host, O_host, lse_host: host buffers with the layouts
 *     of attn_prefill's device buffers.  They should be page-locked
 *     (cudaHostAlloc / cudaHostRegister); pageable memory gives the same
 *     results but the copies then do not overlap.  lse_host and lse are both
 *     NULL or both non-NULL.
 *   Q, K, V, O, lse: caller-owned device buffers of the full sizes; on
 *     completion they hold the inputs and outputs too.
 *   chunks: wanted number of chunks (0: about 32, each >= 1 wave of CTAs;
 *     rounded to what the head grouping allows, at most 64).
 *   other arguments, checks and errors as attn_prefill.
 * The work is ordered after everything already on `stream`, and work
 * enqueued on `stream` after the call runs after the last copy-out: O_host
 * is complete once `stream` has been synchronised.  Calls on one device are
 * serialised by a lock while they enqueue.  One kernel launch per chunk. */
ATTN_API attn_status attn_prefill_from_host(const void *Q_host, const void *K_host,
                                            const void *V_host, void *O_host, float *lse_host,
                                            void *Q, void *K, void *V, void *O, float *lse,
                                            int B, int Hq, int Hkv, int n_q, int n_kv, int d,
                                            int causal, float scale, attn_dtype in_dtype,
                                            attn_dtype out_dtype, const float *q_scale,
                                            const float *k_scale, const float *v_scale,
                                            int chunks, void *stream);

/* Heads per chunk attn_prefill_from_host uses for these sizes on a GPU with
 * `sms` SMs (pure host arithmetic; the chunk count is ceil(B*Hq / result)).
 * Returns 0 for invalid sizes. */
ATTN_API int attn_prefill_from_host_heads_per_chunk(int B, int Hq, int Hkv, int n_q, int d,
                                                    int chunks, int sms);

/* Prefill over a block-paged KV cache: prefix caching / chunked prefill
 * (code-journey.com, "Attention co-design", short ISL over a long cached
 * prefix; papanda925.com, block-wise KV cache).  The n_q new tokens of each
 * sequence are its last n_q; their K/V must already be in the cache
 * (attn_kv_append).
 *   Q        [B, Hq, n_q, d]                    in_dtype (F16 / BF16)
 *   Kcache,
 *   Vcache   [num_blocks, Hkv, block_size, d]    in_dtype
 *   block_table [B, max_blocks_per_seq] int32, seq_lens [B] int32: token t
 *            of sequence b is slot t % block_size of block
 *            block_table[b][t / block_size]; seq_lens[b] is the sequence's
 *            total length (prefix + n_q), in [n_q, max_seq_len] when causal
 *   O        [B, Hq, n_q, d] out_dtype;  lse [B, Hq, n_q] fp32 or NULL
 * Causal rows are aligned bottom-right: new token i of sequence b sees
 * cached token j iff j <= i + seq_lens[b] - n_q.  d in {64, 128, 256};
 * block_size in {16, 32, 64}.  A sequence whose length or block entries the
 * table cannot hold gets O = 0, lse = NaN, and the device error word
 * records ATTN_ERR_INVALID.  One kernel launch. */
ATTN_API attn_status attn_prefill_paged(const void *Q, const void *Kcache, const void *Vcache,
                                        const int32_t *block_table, const int32_t *seq_lens,
                                        void *O, float *lse, int B, int Hq, int Hkv, int n_q,
                                        int d, int block_size, int max_blocks_per_seq,
                                        int num_blocks, int max_seq_len, int causal,
                                        float scale, attn_dtype in_dtype,
                                        attn_dtype out_dtype, void *stream);

/* Bytes of caller-provided device workspace attn_decode needs for these
 * sizes (split-KV partial states).  max_seq_len bounds every seq_lens[s]. */
ATTN_API size_t attn_decode_workspace_bytes(int num_seqs, int Hq, int d,
                                   int max_seq_len);

/* Single-token decode over a block-paged KV cache
 * (papanda925.com, block-wise KV cache; code-journey.com, prefill vs
 * decode: one query token against the whole cache).
 *   q        [num_seqs, Hq, d]                        q_dtype (F16 / BF16)
 *   Kcache,
 *   Vcache   [num_blocks, Hkv, block_size, d]          kv_dtype: same as
 *            q_dtype, or E4M3 with k_scale/v_scale [Hkv] fp32 (dequantised
 *            value = code * scale; q may then be F16 or BF16)
 *   block_table [num_seqs, max_blocks_per_seq] int32: token t of sequence s
 *            is slot t % block_size of block block_table[s][t / block_size]
 *   seq_lens [num_seqs] int32, each in [0, max_seq_len]
 *   O        [num_seqs, Hq, d] out_dtype;  lse [num_seqs, Hq] fp32 or NULL
 *   workspace: >= attn_decode_workspace_bytes(...) bytes, 256-byte aligned;
 *            its contents on entry do not matter and are overwritten.
 * block_size in {16, 32, 64}; d in {64, 128, 256}; Hq / Hkv <= 64 (each 16
 * query heads of a group are one CTA per split; the K/V of a split is read
 * from DRAM once and by the other 16-row tiles from L2); q, the caches and
 * the workspace 16-byte aligned (the workspace 256-byte).
 * A sequence of length 0 yields O = 0 and lse = -inf.  Two kernel launches
 * (split kernel, then combine).  The workspace must not be shared by
 * overlapping calls. */
ATTN_API attn_status attn_decode(const void *q, const void *Kcache, const void *Vcache,
                        const int32_t *block_table, const int32_t *seq_lens,
                        void *O, float *lse, int num_seqs, int Hq, int Hkv,
                        int d, int block_size, int max_blocks_per_seq,
                        int num_blocks, int max_seq_len, float scale,
                        attn_dtype q_dtype, attn_dtype kv_dtype,
                        attn_dtype out_dtype, const float *k_scale,
                        const float *v_scale, void *workspace,
                        size_t workspace_bytes, void *stream);

/* Multi-token decode (speculative / draft verification: several new tokens
 * per sequence, code-journey.com "Attention co-design" -- more query rows
 * per KV head raise decode's GEMM-M).  The n_new new tokens of sequence s
 * are its last n_new; their K/V must already be in the cache.  New token i
 * sees cached token p iff p <= seq_lens[s] - n_new + i (bottom-right).
 *   q   [num_seqs, Hq, n_new, d];  O [num_seqs, Hq, n_new, d];
 *   lse [num_seqs, Hq, n_new] or NULL
 * Everything else as attn_decode, with (Hq / Hkv) * n_new <= 64, every
 * seq_lens[s] >= n_new, and a workspace of at least
 * attn_decode_workspace_bytes(num_seqs * n_new, Hq, d, max_seq_len) bytes.
 * n_new = 1 is attn_decode.  Two kernel launches. */
ATTN_API attn_status attn_decode_tokens(const void *q, const void *Kcache, const void *Vcache,
                                        const int32_t *block_table, const int32_t *seq_lens,
                                        void *O, float *lse, int num_seqs, int n_new, int Hq,
                                        int Hkv, int d, int block_size,
                                        int max_blocks_per_seq, int num_blocks,
                                        int max_seq_len, float scale, attn_dtype q_dtype,
                                        attn_dtype kv_dtype, attn_dtype out_dtype,
                                        const float *k_scale, const float *v_scale,
                                        void *workspace, size_t workspace_bytes, void *stream);

/* KV-cache append (papanda925.com, KV-cache management concept: the K/V of
 * each new token is added to the cache).
 *   k_new, v_new [T, Hkv, d] src_dtype (F16 / BF16)
 *   token r goes to sequence seq_ids[r], position positions[r]: block
 *   block_table[seq][pos / block_size], slot pos % block_size.
 * kv_dtype == src_dtype copies the bits; kv_dtype == E4M3 stores
 * e4m3_rn_satfinite(x / scale[h]) with the division in fp32.
 * seq_lens are NOT updated: the caller owns them.  Out-of-range ids,
 * positions or block entries are skipped and recorded in the device error
 * word.  One kernel launch (none when T == 0). */
ATTN_API attn_status attn_kv_append(const void *k_new, const void *v_new, void *Kcache,
                           void *Vcache, const int32_t *block_table,
                           const int32_t *seq_ids, const int32_t *positions,
                           int T, int num_seqs, int Hkv, int d, int block_size,
                           int max_blocks_per_seq, int num_blocks,
                           attn_dtype src_dtype, attn_dtype kv_dtype,
                           const float *k_scale, const float *v_scale,
                           void *stream);

/* Bytes of caller-provided device workspace attn_backward needs (one fp32
 * per query row). */
ATTN_API size_t attn_backward_workspace_bytes(int B, int Hq, int n_q);

/* Backward pass (marketmaker.cc, "Flash Attention and sequence length",
 * backward pass: probabilities recomputed from Q, K and the stored row
 * statistic, O(n) extra memory).  For the forward O = softmax(scale Q K^T
 * [causal]) V and upstream gradient dO:
 *   dV = P^T dO, dP = dO V^T, D_i = sum_c dO_ic O_ic, dS = P * (dP - D),
 *   dQ = scale dS K, dK = scale dS^T Q,
 * dK and dV of a KV head summed over its G query heads.
 *   Q, dO [B, Hq, n_q, d] in_dtype (F16 / BF16);  K, V [B, Hkv, n_kv, d]
 *   O   [B, Hq, n_q, d] o_dtype: in_dtype or F32 -- the forward's output; D_i
 *       is formed from it, so a 16-bit O moves D_i by its rounding error
 *       (in a row that averages few keys this shows in dQ, dK at the
 *       rounding level of O; an fp32 O removes it)
 *   lse [B, Hq, n_q] fp32: the forward's log-sum-exp (attn_prefill)
 *   dQ [B, Hq, n_q, d], dK, dV [B, Hkv, n_kv, d] out_dtype (F16/BF16/F32)
 *   workspace >= attn_backward_workspace_bytes(B, Hq, n_q), 256-aligned.
 * d in {64, 128}; causal requires n_q <= n_kv (bottom-right).  Three kernel
 * launches (D, then dK/dV, then dQ); every gradient element is written by
 * exactly one thread (no atomics). */
ATTN_API attn_status attn_backward(const void *Q, const void *K, const void *V, const void *O,
                                   const void *dO, const float *lse, void *dQ, void *dK,
                                   void *dV, int B, int Hq, int Hkv, int n_q, int n_kv, int d,
                                   int causal, float scale, attn_dtype in_dtype,
                                   attn_dtype o_dtype, attn_dtype out_dtype, void *workspace,
                                   size_t workspace_bytes, void *stream);

/* Incoherent processing for fp8 attention (marketmaker.cc, "Flash Attention
 * and sequence length", FA3 item 3: a random orthogonal rotation of Q and K
 * before the block-wise FP8 quantisation spreads outliers over all
 * components).  Each row x of X becomes y = x diag(signs) H_d (H_d the
 * Sylvester Hadamard matrix, entries +-1, unnormalised), quantised per block
 * of rows_per_block consecutive rows of a head: scale = amax / 448 over the
 * block's rotated values, codes = e4m3_rn_satfinite(y / scale) with the
 * division in fp32.  Rotating Q and K with the same signs gives
 * (Q R)(K R)^T = d Q K^T: pass scale / d to the prefill with the codes (V is
 * quantised without rotation).  signs == NULL quantises the rows as they are
 * (naive fp8).
 *   X [heads, rows_per_head, d] in_dtype (F16 / BF16); signs [d] int8, +-1
 *     (host-chosen, e.g. seeded random), or NULL
 *   rows_per_block: 0 (or >= rows_per_head) for one scale per head;
 *     ATTN_E4M3_SCALE_BLOCK for the scales attn_prefill_e4m3_blocks takes
 *   codes [heads, rows_per_head, d] E4M3;
 *   scales [heads, nb] fp32, nb = ceil(rows_per_head / rows_per_block)
 *   amax_ws: device scratch of heads * nb * 4 bytes
 * d in {64, 128, 256}.  One memset and two kernel launches. */
ATTN_API attn_status attn_rotate_quantize_e4m3(const void *X, const int8_t *signs, void *codes,
                                               float *scales, void *amax_ws, int heads,
                                               int rows_per_head, int d, int rows_per_block,
                                               attn_dtype in_dtype, void *stream);

/* Synchronises `stream`, then returns and clears the current device's error
 * word: ATTN_ERR_TIMEOUT if a bounded wait expired, ATTN_ERR_INVALID if a
 * device-side index check failed, ATTN_ERR_CUDA if the stream reports a
 * CUDA error, else ATTN_OK. */
ATTN_API attn_status attn_last_error(void *stream);

/* Test entry point for the bounded waits (a failure-path check; the method
 * has no counterpart of it).  Every wait inside the kernels of these
 * libraries gives up after a limit (2 s by default), records
 * ATTN_ERR_TIMEOUT, and the CTA unwinds: copies in flight land, tensor
 * memory is freed, the CTA's output rows are written as O = 0 and
 * lse = NaN.  This call runs attn_prefill (16-bit inputs, d in {64, 128, 256})
 * with the limit set to wait_limit_us and with the producer of the dense
 * prefill kernel withholding its Q copy, so that the first wait on Q
 * expires in every CTA.  The limit and the hook are set and cleared in
 * stream order around the one kernel launch, and the call synchronises
 * `stream` before it returns; it must not overlap any other call on the
 * device (their waits would see the short limit).  Returns ATTN_OK when
 * the launch went through; attn_last_error() then reports
 * ATTN_ERR_TIMEOUT.  wait_limit_us in [1, 1000000]. */
ATTN_API attn_status attn_debug_prefill_timeout(const void *Q, const void *K, const void *V,
                                                void *O, float *lse, int B, int Hq, int Hkv,
                                                int n_q, int n_kv, int d, int causal,
                                                float scale, attn_dtype in_dtype,
                                                attn_dtype out_dtype, unsigned wait_limit_us,
                                                void *stream);

/* Test entry point for the bounded waits of every kernel (a failure-path
 * check; the method has no counterpart of it): synchronises `stream`, then
 * sets the wait limit to wait_limit_us (0: the 2 s default) and the test
 * hooks to `hooks`, bits of:
 *   ATTN_HOOK_WITHHOLD_Q   the dense prefill's producer withholds its Q copy
 *   ATTN_HOOK_WITHHOLD_KV  the decode split kernel's producer issues no K/V
 *                          copy
 * so that a wait expires, the kernel records ATTN_ERR_TIMEOUT, and the
 * affected output rows are written as O = 0 and lse = NaN.  They stay set
 * for every later call on the device until cleared with (0, 0); nothing
 * else may run on the device meanwhile.  wait_limit_us <= 1000000 and no
 * other hook bits, else ATTN_ERR_INVALID. */
#define ATTN_HOOK_WITHHOLD_Q 1u
#define ATTN_HOOK_WITHHOLD_KV 2u
ATTN_API attn_status attn_debug_set_hooks(unsigned wait_limit_us, unsigned hooks, void *stream);

/* Static string naming a status code (never NULL). *//* Static string naming a status code (never NULL). */
ATTN_API const char *attn_status_str(attn_status s);

/* Number of kernel launches the most recent successful call of each entry
 * point made on this host thread (0 after a host-side error). */
ATTN_API int attn_last_launch_count(void);

/* Largest scratch attn_decode_static_ws can use: 16 MiB per device. */
#define ATTN_DECODE_STATIC_WS_BYTES (16u << 20)

/* attn_decode without a caller-provided workspace, for callers that may not
 * allocate device memory themselves: code running inside a host framework
 * that owns every device allocation, or latency-critical threads that cannot
 * afford cudaMalloc (it may synchronise the whole device).  There is no
 * counterpart of this call on the source pages; it only changes where the
 * split-KV scratch lives.
 *
 * Arguments, results and errors are those of attn_decode, minus the
 * workspace.  The scratch is a 16 MiB array compiled into the library
 * (ATTN_DECODE_STATIC_WS_BYTES), held by every GPU that loads the library
 * until the process exits.  Sizes whose scratch need
 * (attn_decode_workspace_bytes) exceeds it return ATTN_ERR_UNSUPPORTED before
 * anything runs.  Nothing is allocated: no cudaMalloc, no cudaFree.
 *
 * The first call on a device looks up the array's device address on that
 * device (current device at call time); make that first call before any
 * stream capture.  Every call on a device shares the one array: calls whose
 * kernels may overlap on the GPU (other streams, other host threads) race on
 * it and must be serialised by the caller.  The kernels write every scratch
 * entry before reading it, so the contents a previous call left behind do
 * not matter and nothing needs clearing. */
ATTN_API attn_status attn_decode_static_ws(
    const void *q, const void *Kcache, const void *Vcache,
    const int32_t *block_table, const int32_t *seq_lens, void *O, float *lse,
    int num_seqs, int Hq, int Hkv, int d, int block_size,
    int max_blocks_per_seq, int num_blocks, int max_seq_len, float scale,
    attn_dtype q_dtype, attn_dtype kv_dtype, attn_dtype out_dtype,
    const float *k_scale, const float *v_scale, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
