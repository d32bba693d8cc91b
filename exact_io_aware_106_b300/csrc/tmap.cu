// tmap.cu -- host-side construction of TMA tensor maps (cuTensorMapEncodeTiled
// reached through the runtime's driver entry-point query, so the library
// needs no libcuda at link time).
#include <atomic>

#include "common.cuh"
#include "launch.h"

namespace attn {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

static bool make_tmap(CUtensorMap *m, const void *ptr, TmapElem elem, int rank,
                      const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                      int swizzle_bytes) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc)
        return false;
    cuuint64_t d[4], s[3];
    cuuint32_t b[4], estr[4];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        estr[i] = 1;
        if (i + 1 < rank)
            s[i] = strides_bytes[i];
    }
    const CUtensorMapDataType dt = elem == TmapElem::BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : elem == TmapElem::F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const CUtensorMapSwizzle sw = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                        : CU_TENSOR_MAP_SWIZZLE_NONE;
    CUresult r = enc(m, dt, static_cast<cuuint32_t>(rank), const_cast<void *>(ptr), d, s, b, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_3d(CUtensorMap *m, const void *ptr, TmapElem elem, const uint64_t dims[3],
                  const uint64_t strides_bytes[2], const uint32_t box[3], int swizzle_bytes) {
    return make_tmap(m, ptr, elem, 3, dims, strides_bytes, box, swizzle_bytes);
}

bool make_tmap_4d(CUtensorMap *m, const void *ptr, TmapElem elem, const uint64_t dims[4],
                  const uint64_t strides_bytes[3], const uint32_t box[4], int swizzle_bytes) {
    return make_tmap(m, ptr, elem, 4, dims, strides_bytes, box, swizzle_bytes);
}

bool make_tmap_3d_16bit(CUtensorMap *m, const void *ptr, bool bf16, const uint64_t dims[3],
                        const uint64_t strides_bytes[2], const uint32_t box[3]) {
    return make_tmap_3d(m, ptr, bf16 ? TmapElem::BF16 : TmapElem::F16, dims, strides_bytes, box,
                        128);
}

int sm_count() {
    // per-device cache; threads that race store the same value
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 148;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n <= 0)
            n = 148;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

} // namespace attn
