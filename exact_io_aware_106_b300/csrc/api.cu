// api.cu -- the extern "C" boundary of libattn.so (declared in attn.h):
// host-side argument validation, the per-device error word, dispatch to the
// prefill, decode and KV-append launchers.
#include <math.h>
#include <mutex>

#include "attn.h"
#include "common.cuh"
#include "launch.h"


// The per-device control words every kernel receives (common.cuh): [0] is
// the error word (bits DERR_TIMEOUT / DERR_INDEX, set by kernels with
// atomicOr, read and cleared by attn_last_error()); [1] and [2] are the wait
// limit and test hooks that only attn_debug_prefill_timeout sets.
__device__ unsigned int g_attn_err_word[attn::CTL_WORDS];

namespace {

thread_local int t_last_launches = 0;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned *g_err_ptr[kMaxDevices] = {nullptr};

// Device address of the error word on the current device (looked up once
// per device with that device current).
unsigned *err_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_err_word) != cudaSuccess)
            return nullptr;
        g_err_ptr[dev] = static_cast<unsigned *>(p);
    }
    return g_err_ptr[dev];
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool is16(attn_dtype t) { return t == ATTN_F16 || t == ATTN_BF16; }
bool is_out(attn_dtype t) { return t == ATTN_F16 || t == ATTN_BF16 || t == ATTN_F32; }
int out_code(attn_dtype t) { return t == ATTN_F16 ? 0 : (t == ATTN_BF16 ? 1 : 2); }

} // namespace

extern "C" {

const char *attn_status_str(attn_status s) {
    switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID: return "ATTN_ERR_INVALID";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    }
    return "ATTN_UNKNOWN_STATUS";
}

int attn_last_launch_count(void) { return t_last_launches; }

} // extern "C"

namespace {

// Host-side checks shared by attn_prefill and attn_prefill_from_host; fills
// `a` on success.
attn_status prefill_args(const void *Q, const void *K, const void *V, void *O, float *lse,
                         int B, int Hq, int Hkv, int n_q, int n_kv, int d, int causal,
                         float scale, attn_dtype in_dtype, attn_dtype out_dtype,
                         const float *q_scale, const float *k_scale, const float *v_scale,
                         attn::PrefillArgs *a) {
    if (!Q || !K || !V || !O)
        return ATTN_ERR_INVALID;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || n_q <= 0 || n_kv <= 0 || d <= 0 || Hq % Hkv != 0)
        return ATTN_ERR_INVALID;
    if (causal && n_q > n_kv)
        return ATTN_ERR_INVALID;
    if (!isfinite(scale))
        return ATTN_ERR_INVALID;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) ||
        (lse && !aligned(lse, 4)))
        return ATTN_ERR_INVALID;
    const bool e4 = in_dtype == ATTN_E4M3;
    if ((!is16(in_dtype) && !e4) || !is_out(out_dtype) || (d != 64 && d != 128 && d != 256))
        return ATTN_ERR_UNSUPPORTED;
    if (e4 && (!q_scale || !k_scale || !v_scale || !aligned(q_scale, 4) ||
               !aligned(k_scale, 4) || !aligned(v_scale, 4)))
        return ATTN_ERR_INVALID;
    const long long nqb = (n_q + 127) / 128;
    if (nqb * B * Hq > 0x7fffffffLL)
        return ATTN_ERR_UNSUPPORTED;
    unsigned *err = err_word();
    if (!err)
        return ATTN_ERR_CUDA;
    *a = attn::PrefillArgs{Q, K, V, O, lse, B, Hq, Hkv, n_q, n_kv, d, causal ? 1 : 0, scale,
                           in_dtype == ATTN_BF16, e4, out_code(out_dtype),
                           e4 ? q_scale : nullptr, e4 ? k_scale : nullptr,
                           e4 ? v_scale : nullptr, err};
    return ATTN_OK;
}

} // namespace

extern "C" {

attn_status attn_prefill(const void *Q, const void *K, const void *V, void *O, float *lse, int B,
                         int Hq, int Hkv, int n_q, int n_kv, int d, int causal, float scale,
                         attn_dtype in_dtype, attn_dtype out_dtype, const float *q_scale,
                         const float *k_scale, const float *v_scale, void *stream) {
    t_last_launches = 0;
    attn::PrefillArgs a;
    const attn_status s = prefill_args(Q, K, V, O, lse, B, Hq, Hkv, n_q, n_kv, d, causal, scale,
                                       in_dtype, out_dtype, q_scale, k_scale, v_scale, &a);
    if (s != ATTN_OK)
        return s;
    if (attn::prefill_launch(a, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    t_last_launches = 1;
    return ATTN_OK;
}

attn_status attn_prefill_e4m3_blocks(const void *Q, const void *K, const void *V, void *O,
                                     float *lse, int B, int Hq, int Hkv, int n_q, int n_kv,
                                     int d, int causal, float scale, attn_dtype out_dtype,
                                     const float *q_scale, const float *k_scale,
                                     const float *v_scale, void *stream) {
    t_last_launches = 0;
    attn::PrefillArgs a;
    const attn_status s = prefill_args(Q, K, V, O, lse, B, Hq, Hkv, n_q, n_kv, d, causal, scale,
                                       ATTN_E4M3, out_dtype, q_scale, k_scale, v_scale, &a);
    if (s != ATTN_OK)
        return s;
    a.e4m3_blocks = true;
    if (attn::prefill_launch(a, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    t_last_launches = 1;
    return ATTN_OK;
}

int attn_prefill_from_host_heads_per_chunk(int B, int Hq, int Hkv, int n_q, int d, int chunks,
                                           int sms) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || n_q <= 0 || d <= 0 || chunks < 0 ||
        sms <= 0)
        return 0;
    return attn::pipeline_heads_per_chunk(B, Hq, Hkv, n_q, d, chunks, sms);
}

attn_status attn_prefill_from_host(const void *Q_host, const void *K_host, const void *V_host,
                                   void *O_host, float *lse_host, void *Q, void *K, void *V,
                                   void *O, float *lse, int B, int Hq, int Hkv, int n_q,
                                   int n_kv, int d, int causal, float scale,
                                   attn_dtype in_dtype, attn_dtype out_dtype,
                                   const float *q_scale, const float *k_scale,
                                   const float *v_scale, int chunks, void *stream) {
    t_last_launches = 0;
    if (!Q_host || !K_host || !V_host || !O_host || (lse_host != nullptr) != (lse != nullptr))
        return ATTN_ERR_INVALID;
    if (chunks < 0)
        return ATTN_ERR_INVALID;
    attn::PrefillArgs a;
    const attn_status s = prefill_args(Q, K, V, O, lse, B, Hq, Hkv, n_q, n_kv, d, causal, scale,
                                       in_dtype, out_dtype, q_scale, k_scale, v_scale, &a);
    if (s != ATTN_OK)
        return s;
    const attn::HostIO h{Q_host, K_host, V_host, O_host, lse_host};
    int launches = 0;
    if (attn::prefill_pipelined(a, h, chunks, static_cast<cudaStream_t>(stream), &launches) !=
        cudaSuccess)
        return ATTN_ERR_CUDA;
    t_last_launches = launches;
    return ATTN_OK;
}

attn_status attn_prefill_paged(const void *Q, const void *Kcache, const void *Vcache,
                               const int32_t *block_table, const int32_t *seq_lens, void *O,
                               float *lse, int B, int Hq, int Hkv, int n_q, int d,
                               int block_size, int max_blocks_per_seq, int num_blocks,
                               int max_seq_len, int causal, float scale, attn_dtype in_dtype,
                               attn_dtype out_dtype, void *stream) {
    t_last_launches = 0;
    if (!Q || !Kcache || !Vcache || !block_table || !seq_lens || !O)
        return ATTN_ERR_INVALID;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || n_q <= 0 || d <= 0 || Hq % Hkv != 0 ||
        block_size <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || max_seq_len <= 0)
        return ATTN_ERR_INVALID;
    if (static_cast<long long>(max_seq_len) >
        static_cast<long long>(max_blocks_per_seq) * block_size)
        return ATTN_ERR_INVALID;
    if (causal && n_q > max_seq_len)
        return ATTN_ERR_INVALID;
    if (!isfinite(scale))
        return ATTN_ERR_INVALID;
    if (!aligned(Q, 16) || !aligned(Kcache, 16) || !aligned(Vcache, 16) || !aligned(O, 16) ||
        !aligned(block_table, 4) || !aligned(seq_lens, 4) || (lse && !aligned(lse, 4)))
        return ATTN_ERR_INVALID;
    if (!is16(in_dtype) || !is_out(out_dtype) || (d != 64 && d != 128 && d != 256) ||
        (block_size != 16 && block_size != 32 && block_size != 64))
        return ATTN_ERR_UNSUPPORTED;
    const long long nqb = (n_q + 127) / 128;
    if (nqb * B * Hq > 0x7fffffffLL)
        return ATTN_ERR_UNSUPPORTED;
    unsigned *err = err_word();
    if (!err)
        return ATTN_ERR_CUDA;
    attn::PrefillArgs a{Q, Kcache, Vcache, O, lse, B, Hq, Hkv, n_q, max_seq_len, d,
                        causal ? 1 : 0, scale, in_dtype == ATTN_BF16, false,
                        out_code(out_dtype), nullptr, nullptr, nullptr, err};
    a.paged = true;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.block_size = block_size;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.max_seq_len = max_seq_len;
    if (attn::prefill_launch(a, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    t_last_launches = 1;
    return ATTN_OK;
}

size_t attn_decode_workspace_bytes(int num_seqs, int Hq, int d, int max_seq_len) {
    if (num_seqs <= 0 || Hq <= 0 || d <= 0 || max_seq_len < 0)
        return 0;
    return attn::decode_workspace_bytes(num_seqs, Hq, d, max_seq_len);
}

} // extern "C"

namespace {

// Shared by attn_decode (T = 1) and attn_decode_tokens.
attn_status decode_impl(const void *q, const void *Kcache, const void *Vcache,
                        const int32_t *block_table, const int32_t *seq_lens, void *O, float *lse,
                        int num_seqs, int T, int Hq, int Hkv, int d, int block_size,
                        int max_blocks_per_seq, int num_blocks, int max_seq_len, float scale,
                        attn_dtype q_dtype, attn_dtype kv_dtype, attn_dtype out_dtype,
                        const float *k_scale, const float *v_scale, void *workspace,
                        size_t workspace_bytes, void *stream) {
    t_last_launches = 0;
    if (!q || !Kcache || !Vcache || !block_table || !seq_lens || !O || !workspace)
        return ATTN_ERR_INVALID;
    if (num_seqs <= 0 || num_seqs > 65535 || T <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 ||
        block_size <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || max_seq_len < 0)
        return ATTN_ERR_INVALID;
    if (static_cast<long long>(max_seq_len) >
        static_cast<long long>(max_blocks_per_seq) * block_size)
        return ATTN_ERR_INVALID;
    if (T > 1 && max_seq_len < T)
        return ATTN_ERR_INVALID;
    if (!isfinite(scale))
        return ATTN_ERR_INVALID;
    if (!is16(q_dtype) || !is_out(out_dtype))
        return ATTN_ERR_UNSUPPORTED;
    const bool e4 = kv_dtype == ATTN_E4M3;
    if (!(kv_dtype == q_dtype || e4))
        return ATTN_ERR_UNSUPPORTED;
    if (e4 && (!k_scale || !v_scale))
        return ATTN_ERR_INVALID;
    if ((d != 64 && d != 128 && d != 256) ||
        (block_size != 16 && block_size != 32 && block_size != 64) ||
        static_cast<long long>(Hq / Hkv) * T > 64)
        return ATTN_ERR_UNSUPPORTED;
    if (static_cast<long long>(num_seqs) * Hq * T > 0x7fffffffLL)
        return ATTN_ERR_UNSUPPORTED;
    if (!aligned(Kcache, 16) || !aligned(Vcache, 16) || !aligned(q, 16) || !aligned(O, 4) ||
        !aligned(workspace, 256) || !aligned(block_table, 4) || !aligned(seq_lens, 4))
        return ATTN_ERR_INVALID;
    if (workspace_bytes < attn::decode_workspace_bytes(num_seqs * T, Hq, d, max_seq_len))
        return ATTN_ERR_INVALID;
    unsigned *err = err_word();
    if (!err)
        return ATTN_ERR_CUDA;
    attn::DecodeArgs a{q, Kcache, Vcache, block_table, seq_lens, O, lse, num_seqs, Hq, Hkv, d,
                       block_size, max_blocks_per_seq, num_blocks, max_seq_len, scale,
                       q_dtype == ATTN_BF16, e4, out_code(out_dtype), k_scale, v_scale,
                       workspace, err};
    a.T = T;
    if (attn::decode_launch(a, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    t_last_launches = 2;
    return ATTN_OK;
}

} // namespace

extern "C" {

attn_status attn_decode(const void *q, const void *Kcache, const void *Vcache,
                        const int32_t *block_table, const int32_t *seq_lens, void *O, float *lse,
                        int num_seqs, int Hq, int Hkv, int d, int block_size,
                        int max_blocks_per_seq, int num_blocks, int max_seq_len, float scale,
                        attn_dtype q_dtype, attn_dtype kv_dtype, attn_dtype out_dtype,
                        const float *k_scale, const float *v_scale, void *workspace,
                        size_t workspace_bytes, void *stream) {
    return decode_impl(q, Kcache, Vcache, block_table, seq_lens, O, lse, num_seqs, 1, Hq, Hkv,
                       d, block_size, max_blocks_per_seq, num_blocks, max_seq_len, scale, q_dtype,
                       kv_dtype, out_dtype, k_scale, v_scale, workspace, workspace_bytes, stream);
}

attn_status attn_decode_tokens(const void *q, const void *Kcache, const void *Vcache,
                               const int32_t *block_table, const int32_t *seq_lens, void *O,
                               float *lse, int num_seqs, int n_new, int Hq, int Hkv, int d,
                               int block_size, int max_blocks_per_seq, int num_blocks,
                               int max_seq_len, float scale, attn_dtype q_dtype,
                               attn_dtype kv_dtype, attn_dtype out_dtype, const float *k_scale,
                               const float *v_scale, void *workspace, size_t workspace_bytes,
                               void *stream) {
    return decode_impl(q, Kcache, Vcache, block_table, seq_lens, O, lse, num_seqs, n_new, Hq,
                       Hkv, d, block_size, max_blocks_per_seq, num_blocks, max_seq_len, scale,
                       q_dtype, kv_dtype, out_dtype, k_scale, v_scale, workspace,
                       workspace_bytes, stream);
}

attn_status attn_kv_append(const void *k_new, const void *v_new, void *Kcache, void *Vcache,
                           const int32_t *block_table, const int32_t *seq_ids,
                           const int32_t *positions, int T, int num_seqs, int Hkv, int d,
                           int block_size, int max_blocks_per_seq, int num_blocks,
                           attn_dtype src_dtype, attn_dtype kv_dtype, const float *k_scale,
                           const float *v_scale, void *stream) {
    t_last_launches = 0;
    if (T < 0 || num_seqs <= 0 || Hkv <= 0 || block_size <= 0 || max_blocks_per_seq <= 0 ||
        num_blocks <= 0)
        return ATTN_ERR_INVALID;
    if (T == 0)
        return ATTN_OK;
    if (!k_new || !v_new || !Kcache || !Vcache || !block_table || !seq_ids || !positions)
        return ATTN_ERR_INVALID;
    if (!is16(src_dtype))
        return ATTN_ERR_UNSUPPORTED;
    const bool e4 = kv_dtype == ATTN_E4M3;
    if (!(kv_dtype == src_dtype || e4))
        return ATTN_ERR_UNSUPPORTED;
    if (e4 && (!k_scale || !v_scale))
        return ATTN_ERR_INVALID;
    if (d != 64 && d != 128 && d != 256)
        return ATTN_ERR_UNSUPPORTED;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(Kcache, 16) ||
        !aligned(Vcache, 16))
        return ATTN_ERR_INVALID;
    if (static_cast<long long>(T) * Hkv > 0x7fffffffLL)
        return ATTN_ERR_UNSUPPORTED;
    unsigned *err = err_word();
    if (!err)
        return ATTN_ERR_CUDA;
    attn::AppendArgs a{k_new, v_new, Kcache, Vcache, block_table, seq_ids, positions, T,
                       num_seqs, Hkv, d, block_size, max_blocks_per_seq, num_blocks,
                       src_dtype == ATTN_BF16, e4, k_scale, v_scale, err};
    if (attn::kv_append_launch(a, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    t_last_launches = 1;
    return ATTN_OK;
}

size_t attn_backward_workspace_bytes(int B, int Hq, int n_q) {
    if (B <= 0 || Hq <= 0 || n_q <= 0)
        return 0;
    return attn::backward_workspace_bytes(B, Hq, n_q);
}

attn_status attn_backward(const void *Q, const void *K, const void *V, const void *O,
                          const void *dO, const float *lse, void *dQ, void *dK, void *dV, int B,
                          int Hq, int Hkv, int n_q, int n_kv, int d, int causal, float scale,
                          attn_dtype in_dtype, attn_dtype o_dtype, attn_dtype out_dtype,
                          void *workspace, size_t workspace_bytes, void *stream) {
    t_last_launches = 0;
    if (!Q || !K || !V || !O || !dO || !lse || !dQ || !dK || !dV || !workspace)
        return ATTN_ERR_INVALID;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || n_q <= 0 || n_kv <= 0 || d <= 0 || Hq % Hkv != 0)
        return ATTN_ERR_INVALID;
    if (causal && n_q > n_kv)
        return ATTN_ERR_INVALID;
    if (!isfinite(scale))
        return ATTN_ERR_INVALID;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) ||
        !aligned(dO, 16) || !aligned(dQ, 16) || !aligned(dK, 16) || !aligned(dV, 16) ||
        !aligned(lse, 4) || !aligned(workspace, 256))
        return ATTN_ERR_INVALID;
    if (!is16(in_dtype) || !is_out(out_dtype) || (d != 64 && d != 128) ||
        !(o_dtype == in_dtype || o_dtype == ATTN_F32))
        return ATTN_ERR_UNSUPPORTED;
    const long long nqb = (n_q + 127) / 128, nkb = (n_kv + 127) / 128;
    if (nqb * B * Hq > 0x7fffffffLL || nkb * B * Hkv > 0x7fffffffLL)
        return ATTN_ERR_UNSUPPORTED;
    if (workspace_bytes < attn::backward_workspace_bytes(B, Hq, n_q))
        return ATTN_ERR_INVALID;
    unsigned *err = err_word();
    if (!err)
        return ATTN_ERR_CUDA;
    attn::BackwardArgs a{Q, K, V, O, dO, lse, dQ, dK, dV, B, Hq, Hkv, n_q, n_kv, d,
                         causal ? 1 : 0, scale, in_dtype == ATTN_BF16, o_dtype == ATTN_F32,
                         out_code(out_dtype), workspace, err};
    if (attn::backward_launch(a, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    t_last_launches = 3;
    return ATTN_OK;
}

attn_status attn_rotate_quantize_e4m3(const void *X, const int8_t *signs, void *codes,
                                      float *scales, void *amax_ws, int heads,
                                      int rows_per_head, int d, int rows_per_block,
                                      attn_dtype in_dtype, void *stream) {
    t_last_launches = 0;
    if (!X || !codes || !scales || !amax_ws || heads <= 0 || rows_per_head <= 0 ||
        rows_per_block < 0)
        return ATTN_ERR_INVALID;
    if (!is16(in_dtype) || (d != 64 && d != 128 && d != 256))
        return ATTN_ERR_UNSUPPORTED;
    if (!aligned(X, 16) || !aligned(codes, 16) || !aligned(scales, 4) || !aligned(amax_ws, 4))
        return ATTN_ERR_INVALID;
    if (static_cast<long long>(heads) * rows_per_head > (1LL << 40))
        return ATTN_ERR_UNSUPPORTED;
    const int rpb = (rows_per_block == 0 || rows_per_block > rows_per_head) ? rows_per_head
                                                                            : rows_per_block;
    attn::RotQArgs a{X, signs, static_cast<uint8_t *>(codes), scales,
                     static_cast<unsigned *>(amax_ws), heads, rows_per_head, d, rpb,
                     in_dtype == ATTN_BF16};
    if (attn::rotate_quantize_launch(a, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    t_last_launches = 2;
    return ATTN_OK;
}

attn_status attn_debug_prefill_timeout(const void *Q, const void *K, const void *V, void *O,
                                       float *lse, int B, int Hq, int Hkv, int n_q, int n_kv,
                                       int d, int causal, float scale, attn_dtype in_dtype,
                                       attn_dtype out_dtype, unsigned wait_limit_us,
                                       void *stream) {
    t_last_launches = 0;
    if (wait_limit_us == 0 || wait_limit_us > 1000000u)
        return ATTN_ERR_INVALID;
    if (!is16(in_dtype) || (d != 64 && d != 128 && d != 256))
        return ATTN_ERR_UNSUPPORTED; // the hook lives in the dense kernels' producers
    attn::PrefillArgs a;
    const attn_status s = prefill_args(Q, K, V, O, lse, B, Hq, Hkv, n_q, n_kv, d, causal, scale,
                                       in_dtype, out_dtype, nullptr, nullptr, nullptr, &a);
    if (s != ATTN_OK)
        return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // set the limit and the hook, run the prefill, clear both: all in stream
    // order; the stream is synchronised before the host words go out of scope
    const unsigned set_words[2] = {wait_limit_us, attn::HOOK_WITHHOLD_Q};
    static const unsigned clear_words[2] = {0u, 0u};
    if (cudaMemcpyToSymbolAsync(g_attn_err_word, set_words, sizeof set_words,
                                attn::CTL_WAIT_US * sizeof(unsigned), cudaMemcpyHostToDevice,
                                st) != cudaSuccess)
        return ATTN_ERR_CUDA;
    const cudaError_t e = attn::prefill_launch(a, st);
    if (cudaMemcpyToSymbolAsync(g_attn_err_word, clear_words, sizeof clear_words,
                                attn::CTL_WAIT_US * sizeof(unsigned), cudaMemcpyHostToDevice,
                                st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess || e != cudaSuccess)
        return ATTN_ERR_CUDA;
    t_last_launches = 1;
    return ATTN_OK;
}

static_assert(ATTN_HOOK_WITHHOLD_Q == attn::HOOK_WITHHOLD_Q &&
                  ATTN_HOOK_WITHHOLD_KV == attn::HOOK_WITHHOLD_KV,
              "hook bits of the header and the kernels agree");

attn_status attn_debug_set_hooks(unsigned wait_limit_us, unsigned hooks, void *stream) {
    t_last_launches = 0;
    if (wait_limit_us > 1000000u || (hooks & ~attn::HOOK_ALL) != 0u)
        return ATTN_ERR_INVALID;
    if (!err_word())
        return ATTN_ERR_CUDA;
    // after the work already queued on `stream`, before anything queued later
    const unsigned words[2] = {wait_limit_us, hooks};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess ||
        cudaMemcpyToSymbol(g_attn_err_word, words, sizeof words,
                           attn::CTL_WAIT_US * sizeof(unsigned), cudaMemcpyHostToDevice) !=
            cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

attn_status attn_last_error(void *stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return ATTN_ERR_CUDA;
    unsigned w = 0;
    if (cudaMemcpyFromSymbol(&w, g_attn_err_word, sizeof w, attn::CTL_ERR * sizeof w) !=
        cudaSuccess)
        return ATTN_ERR_CUDA;
    if (w != 0) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_attn_err_word, &zero, sizeof zero, attn::CTL_ERR * sizeof w) !=
            cudaSuccess)
            return ATTN_ERR_CUDA;
    }
    if (w & attn::DERR_TIMEOUT)
        return ATTN_ERR_TIMEOUT;
    if (w & attn::DERR_INDEX)
        return ATTN_ERR_INVALID;
    return ATTN_OK;
}

} // extern "C"

// ------------------------------------------------ decode without allocation

// Split-KV scratch for attn_decode_static_ws, compiled into the library so
// that callers who may not allocate device memory can still decode.  In
// host code this name is only a stand-in for the symbol: the device address
// comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_decode_scratch[ATTN_DECODE_STATIC_WS_BYTES];

namespace {

std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_decode_scratch on the current device, looked up once
// per device with that device current; nullptr if the lookup fails.
void *decode_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
            return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

} // namespace

extern "C" attn_status attn_decode_static_ws(
    const void *q, const void *Kcache, const void *Vcache, const int32_t *block_table,
    const int32_t *seq_lens, void *O, float *lse, int num_seqs, int Hq, int Hkv, int d,
    int block_size, int max_blocks_per_seq, int num_blocks, int max_seq_len, float scale,
    attn_dtype q_dtype, attn_dtype kv_dtype, attn_dtype out_dtype, const float *k_scale,
    const float *v_scale, void *stream) {
    t_last_launches = 0;
    if (num_seqs <= 0 || Hq <= 0 || d <= 0 || max_seq_len < 0)
        return ATTN_ERR_INVALID;
    // the scratch must hold every split's partial state for these sizes
    if (attn::decode_workspace_bytes(num_seqs, Hq, d, max_seq_len) >
        static_cast<size_t>(ATTN_DECODE_STATIC_WS_BYTES))
        return ATTN_ERR_UNSUPPORTED;
    void *ws = decode_scratch();
    if (!ws)
        return ATTN_ERR_CUDA;
    return attn_decode(q, Kcache, Vcache, block_table, seq_lens, O, lse, num_seqs, Hq, Hkv, d,
                       block_size, max_blocks_per_seq, num_blocks, max_seq_len, scale, q_dtype,
                       kv_dtype, out_dtype, k_scale, v_scale, ws, ATTN_DECODE_STATIC_WS_BYTES,
                       stream);
}
