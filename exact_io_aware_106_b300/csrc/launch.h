// launch.h -- host-side launcher interfaces shared by api.cu and the kernel
// translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace attn {

struct PrefillArgs {
    const void *Q;
    const void *K;
    const void *V;
    void *O;
    float *lse;
    int B, Hq, Hkv, n_q, n_kv, d, causal;
    float scale;
    bool bf16;
    bool e4m3;     // E4M3 inputs with per-head scales
    int out_dtype; // 0 f16, 1 bf16, 2 f32
    const float *q_scale;
    const float *k_scale;
    const float *v_scale;
    unsigned *err;
    // E4M3 Q / K scales per 128-row block of a head instead of per head
    bool e4m3_blocks = false;
    // prefill over a block-paged cache (K, V are then the caches)
    bool paged = false;
    const int32_t *block_table = nullptr;
    const int32_t *seq_lens = nullptr;
    int block_size = 0, max_blocks = 0, num_blocks = 0, max_seq_len = 0;
};

struct DecodeArgs {
    const void *q;
    const void *Kc;
    const void *Vc;
    const int32_t *block_table;
    const int32_t *seq_lens;
    void *O;
    float *lse;
    int num_seqs, Hq, Hkv, d, block_size, max_blocks, num_blocks, max_seq_len;
    float scale;
    bool q_bf16, kv_e4m3;
    int out_dtype; // 0 f16, 1 bf16, 2 f32
    const float *k_scale;
    const float *v_scale;
    void *workspace;
    unsigned *err;
    int T = 1; // new query tokens per sequence (multi-token decode)
};

struct AppendArgs {
    const void *k_new;
    const void *v_new;
    void *Kc;
    void *Vc;
    const int32_t *block_table;
    const int32_t *seq_ids;
    const int32_t *positions;
    int T, num_seqs, Hkv, d, block_size, max_blocks, num_blocks;
    bool bf16, to_e4m3;
    const float *k_scale;
    const float *v_scale;
    unsigned *err;
};

enum class TmapElem { BF16, F16, U8 };

// 3-D tensor map (dims innermost first, strides in bytes for dims 1, 2) with
// the given swizzle span (128, 64 or 0 bytes) and zero fill outside bounds.
bool make_tmap_3d(CUtensorMap *m, const void *ptr, TmapElem elem, const uint64_t dims[3],
                  const uint64_t strides_bytes[2], const uint32_t box[3], int swizzle_bytes);

// 4-D form.  The strides need not grow with the dimension: a dimension may
// step through a row in smaller strides than the one before it (the paged
// V cache's panels, 128 bytes apart, taken as the box's outer dimension so
// that each panel lands as its own swizzled block of rows).
bool make_tmap_4d(CUtensorMap *m, const void *ptr, TmapElem elem, const uint64_t dims[4],
                  const uint64_t strides_bytes[3], const uint32_t box[4], int swizzle_bytes);

// Number of SMs of the current device (cached per device).
int sm_count();

// Host-resident buffers of a pipelined prefill (same layouts as the device
// ones in PrefillArgs).
struct HostIO {
    const void *Q;
    const void *K;
    const void *V;
    void *O;
    float *lse; // null: lse is not copied back
};

// Heads per chunk of the pipelined prefill (see pipeline.cu).
int pipeline_heads_per_chunk(int B, int Hq, int Hkv, int n_q, int d, int want, int sms);

// Prefill of `a` (device buffers) with inputs copied from and outputs copied
// to `h` chunk by chunk, copies overlapped with compute; ordered after
// earlier work on `st`, and later work on `st` waits for the last copy.
cudaError_t prefill_pipelined(const PrefillArgs &a, const HostIO &h, int want_chunks,
                              cudaStream_t st, int *launches);

struct BackwardArgs {
    const void *Q, *K, *V, *O, *dO;
    const float *lse;
    void *dQ, *dK, *dV;
    int B, Hq, Hkv, n_q, n_kv, d, causal;
    float scale;
    bool bf16;
    bool o_f32;    // O given in fp32 (else in the inputs' 16-bit format)
    int out_dtype; // 0 f16, 1 bf16, 2 f32
    void *workspace;
    unsigned *err;
};

cudaError_t backward_launch(const BackwardArgs &a, cudaStream_t st);

struct RotQArgs {
    const void *X;       // [heads, rows_per_head, d] 16-bit
    const int8_t *signs; // [d], +-1; null: no rotation
    uint8_t *codes;      // [heads, rows_per_head, d] E4M3
    float *scales;       // [heads, nb], nb = ceil(rows_per_head / rows_per_block)
    unsigned *amax_ws;   // [heads, nb] scratch
    int heads, rows_per_head, d, rows_per_block;
    bool bf16;
};

cudaError_t rotate_quantize_launch(const RotQArgs &a, cudaStream_t st);
size_t backward_workspace_bytes(int B, int Hq, int n_q);

// 3-D tensor map over a 16-bit tensor with 128-byte swizzle and zero fill
// outside the bounds (dims innermost first, strides in bytes for dims 1, 2).
bool make_tmap_3d_16bit(CUtensorMap *m, const void *ptr, bool bf16, const uint64_t dims[3],
                        const uint64_t strides_bytes[2], const uint32_t box[3]);

cudaError_t prefill_launch(const PrefillArgs &a, cudaStream_t st);
cudaError_t decode_launch(const DecodeArgs &a, cudaStream_t st);
cudaError_t kv_append_launch(const AppendArgs &a, cudaStream_t st);
size_t decode_workspace_bytes(int num_seqs, int Hq, int d, int max_seq_len);
int decode_tokens_per_split(int max_seq_len);
int decode_max_splits(int max_seq_len);

} // namespace attn
