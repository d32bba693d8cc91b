// pipeline.cu -- prefill with host-resident inputs and outputs, the PCIe
// copies overlapped with the attention kernels.
//
// The IO-aware argument (auturnal.com "From attention to IO-aware execution"
// §10: the slowest level of the memory hierarchy sets the pace) applied one
// level further out: when Q, K, V start in host memory and O must end there,
// the host link, not HBM, is the slowest level, and copying everything before
// computing anything leaves the GPU idle for the whole transfer.  So the
// heads are cut into chunks of consecutive (batch, head) pairs, and three
// queues run side by side:
//   copy-in  : Q of chunk c (+ K, V of the KV heads chunk c begins)
//   compute  : attention of chunk c once its copy-in has landed
//   copy-out : O (and lse) of chunk c once its attention is done
// Chunk c+1's copy-in, chunk c's attention and chunk c-1's copy-out overlap.
// Attention of consecutive chunks alternates between two compute streams so
// that the next chunk's CTAs fill the SMs that the previous chunk's tail
// leaves idle.  Each chunk is an ordinary prefill launch on offset pointers:
// heads of one chunk are contiguous in every [B, H, n, d] tensor.
#include <mutex>

#include "launch.h"

namespace attn {

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 64;

struct PipeCtx {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr, comp2 = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t landed[kMaxChunks] = {};
    cudaEvent_t done[kMaxChunks] = {};
};

std::mutex g_pipe_mu[kMaxDevices];
PipeCtx g_pipe[kMaxDevices];

cudaError_t init_ctx(PipeCtx &c) {
    if (c.ready)
        return cudaSuccess;
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&c.in, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&c.out, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&c.comp2, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&c.start, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&c.end, cudaEventDisableTiming)) != cudaSuccess)
        return e;
    for (int i = 0; i < kMaxChunks; ++i)
        if ((e = cudaEventCreateWithFlags(&c.landed[i], cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&c.done[i], cudaEventDisableTiming)) != cudaSuccess)
            return e;
    c.ready = true;
    return cudaSuccess;
}

} // namespace

// Heads per chunk for F = B*Hq flattened heads in groups of G (one KV head
// each): a whole number of groups, or an exact divisor of G, so that every
// chunk is a valid prefill on its own (B' = 1, Hq' = heads, Hkv' = heads/G or
// 1).  `want` = 0 picks about 32 chunks, each at least one wave of CTAs:
// the first chunk's copy-in and the last chunk's copy-out are the only
// copies nothing hides, so smaller chunks shorten them, while the two
// alternating compute streams hide the tails of small launches.
int pipeline_heads_per_chunk(int B, int Hq, int Hkv, int n_q, int d, int want, int sms) {
    const long long F = static_cast<long long>(B) * Hq;
    const int G = Hq / Hkv;
    const long long groups = static_cast<long long>(B) * Hkv;
    if (want <= 0) {
        const long long rows_per_cta = d > 128 ? 128 : 256;
        const long long ctas_per_head = (n_q + rows_per_cta - 1) / rows_per_cta;
        const long long min_heads = (sms + ctas_per_head - 1) / ctas_per_head;
        long long w = F / (min_heads > 0 ? min_heads : 1);
        want = static_cast<int>(w < 1 ? 1 : (w > 32 ? 32 : w));
    }
    if (want > kMaxChunks)
        want = kMaxChunks;
    if (want <= groups) {
        const long long gpc = (groups + want - 1) / want; // groups per chunk
        return static_cast<int>(gpc * G);
    }
    // more chunks than groups: split each group into m equal parts, m | G
    for (int m = 2; m <= G && groups * m <= kMaxChunks; ++m)
        if (G % m == 0 && groups * m >= want)
            return G / m;
    return G;
}

cudaError_t prefill_pipelined(const PrefillArgs &a, const HostIO &h, int want_chunks,
                              cudaStream_t st, int *launches) {
    *launches = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_pipe_mu[dev]);
    PipeCtx &c = g_pipe[dev];
    if ((e = init_ctx(c)) != cudaSuccess)
        return e;

    const int G = a.Hq / a.Hkv;
    const long long F = static_cast<long long>(a.B) * a.Hq;
    const int hpc = pipeline_heads_per_chunk(a.B, a.Hq, a.Hkv, a.n_q, a.d, want_chunks,
                                             sm_count());
    const size_t ein = a.e4m3 ? 1 : 2;
    const size_t eout = a.out_dtype == 2 ? 4 : 2;
    const size_t q_head = static_cast<size_t>(a.n_q) * a.d * ein;
    const size_t kv_head = static_cast<size_t>(a.n_kv) * a.d * ein;
    const size_t o_head = static_cast<size_t>(a.n_q) * a.d * eout;
    const size_t l_head = static_cast<size_t>(a.n_q) * 4;
    auto cb = [](const void *p, size_t off) { return static_cast<const char *>(p) + off; };
    auto mb = [](void *p, size_t off) { return static_cast<char *>(p) + off; };

    // everything already on `st` (earlier users of these buffers) first
    if ((e = cudaEventRecord(c.start, st)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(c.in, c.start, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(c.out, c.start, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(c.comp2, c.start, 0)) != cudaSuccess)
        return e;
    int k = 0;
    for (long long f0 = 0; f0 < F; f0 += hpc, ++k) {
        const int heads = static_cast<int>(F - f0 < hpc ? F - f0 : hpc);
        // copy-in: Q of the chunk, K and V of every KV head that starts in it
        if ((e = cudaMemcpyAsync(mb(const_cast<void *>(a.Q), f0 * q_head), cb(h.Q, f0 * q_head),
                                 heads * q_head, cudaMemcpyHostToDevice, c.in)) != cudaSuccess)
            return e;
        const long long g0 = (f0 + G - 1) / G, g1 = (f0 + heads + G - 1) / G;
        if (g1 > g0) {
            const size_t off = g0 * kv_head, bytes = (g1 - g0) * kv_head;
            if ((e = cudaMemcpyAsync(mb(const_cast<void *>(a.K), off), cb(h.K, off), bytes,
                                     cudaMemcpyHostToDevice, c.in)) != cudaSuccess ||
                (e = cudaMemcpyAsync(mb(const_cast<void *>(a.V), off), cb(h.V, off), bytes,
                                     cudaMemcpyHostToDevice, c.in)) != cudaSuccess)
                return e;
        }
        if ((e = cudaEventRecord(c.landed[k], c.in)) != cudaSuccess)
            return e;
        // attention of the chunk on offset pointers
        cudaStream_t cs = (k & 1) ? c.comp2 : st;
        if ((e = cudaStreamWaitEvent(cs, c.landed[k], 0)) != cudaSuccess)
            return e;
        PrefillArgs p = a;
        const long long kv0 = f0 / G;
        p.Q = cb(a.Q, f0 * q_head);
        p.K = cb(a.K, kv0 * kv_head);
        p.V = cb(a.V, kv0 * kv_head);
        p.O = mb(a.O, f0 * o_head);
        p.lse = a.lse ? reinterpret_cast<float *>(mb(a.lse, f0 * l_head)) : nullptr;
        p.B = 1;
        p.Hq = heads;
        p.Hkv = heads >= G ? heads / G : 1;
        if (a.e4m3) {
            p.q_scale = a.q_scale + f0;
            p.k_scale = a.k_scale + kv0;
            p.v_scale = a.v_scale + kv0;
        }
        if ((e = prefill_launch(p, cs)) != cudaSuccess)
            return e;
        ++*launches;
        if ((e = cudaEventRecord(c.done[k], cs)) != cudaSuccess)
            return e;
        // copy-out of the chunk's results
        if ((e = cudaStreamWaitEvent(c.out, c.done[k], 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(mb(h.O, f0 * o_head), cb(a.O, f0 * o_head), heads * o_head,
                                 cudaMemcpyDeviceToHost, c.out)) != cudaSuccess)
            return e;
        if (h.lse && (e = cudaMemcpyAsync(mb(h.lse, f0 * l_head), cb(a.lse, f0 * l_head),
                                          heads * l_head, cudaMemcpyDeviceToHost,
                                          c.out)) != cudaSuccess)
            return e;
    }
    // later work on `st` sees the results in host memory
    if ((e = cudaEventRecord(c.end, c.out)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(st, c.end, 0)) != cudaSuccess)
        return e;
    return cudaSuccess;
}

} // namespace attn
