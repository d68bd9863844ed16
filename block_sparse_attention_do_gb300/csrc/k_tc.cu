// k_tc.cu -- host helpers of the tensor-core kernels: which problems they
// take, the device's SM count and TMA tensor-map construction.
#include <mutex>

#include "tc_common.cuh"

namespace nsa {

bool tc_supported(const Geo &g, int dtype)
{
    if (!(dtype == NSA_DTYPE_BF16 && g.D == kHead && g.bs == kKeys && g.G >= 1 && g.G <= kRows))
        return false;
    // the row-gather maps (G % 8 == 0) fold the batch index into the head or
    // the token index: strides where neither folds go to the other-shapes
    // kernels (k_gtc.cu)
    int bt;
    return g.G % 8 != 0 || (rows_map_form(g, g.Hq, g.sq, bt) && rows_map_form(g, g.Hq, g.so, bt));
}

int num_sms()
{
    static int cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 148;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
    });
    return fn;
}

}  // namespace

bool make_tmap(CUtensorMap *map, const void *base, const Geo &g, int H, int box_tok, int box_heads, const Strides &s,
               bool keys)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
    cuuint32_t rank;
    const cuuint64_t es = 2;  // bf16
    if (g.thd) {
        rank = 3;
        dims[0] = g.D;
        dims[1] = H;
        dims[2] = keys ? g.ntok_k : g.ntok;
        strides[0] = (cuuint64_t)s.h * es;
        strides[1] = (cuuint64_t)s.t * es;
        box[0] = 64;
        box[1] = box_heads;
        box[2] = box_tok;
    } else {
        rank = 4;
        dims[0] = g.D;
        dims[1] = keys ? g.Tk : g.T;
        dims[2] = H;
        dims[3] = g.B;
        strides[0] = (cuuint64_t)s.t * es;
        strides[1] = (cuuint64_t)s.h * es;
        strides[2] = (cuuint64_t)s.b * es;
        box[0] = 64;
        box[1] = box_tok;
        box[2] = box_heads;
        box[3] = 1;
    }
    if (dims[rank - 1] == 0)
        return false;
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_rows(CUtensorMap *map, const void *base, const Geo &g, int H, int G, const Strides &s, int bt)
{
    auto fn = encode_fn();
    if (!fn || G % 8 != 0 || H % 8 != 0 || G / 8 > 256)
        return false;
    const cuuint64_t es = 2;  // bf16
    cuuint64_t dims[5], strides[4];
    cuuint32_t box[5] = {64, 8, 2, (cuuint32_t)(G / 8), 1}, estr[5] = {1, 1, 1, 1, 1};
    dims[0] = 64;
    dims[1] = 8;
    dims[2] = 2;
    strides[0] = (cuuint64_t)s.h * es;      // the next head
    strides[1] = 64 * es;                   // the second 64-column half of a row
    strides[2] = 8 * (cuuint64_t)s.h * es;  // the next head octet
    strides[3] = (cuuint64_t)s.t * es;      // the next token
    if (g.thd) {
        dims[3] = H / 8;
        dims[4] = g.ntok;
    } else if (bt) {
        // (b, t) folded: token index b*T + t (needs s.b = T * s.t)
        if (g.B > 1 && s.b != (int64_t)g.T * s.t)
            return false;
        dims[3] = H / 8;
        dims[4] = (cuuint64_t)g.B * g.T;
    } else {
        // (b, head) folded into one octet index (needs s.b = H * s.h unless B = 1)
        if (g.B > 1 && s.b != (int64_t)H * s.h)
            return false;
        dims[3] = (cuuint64_t)g.B * H / 8;
        dims[4] = g.T;
    }
    if (dims[3] == 0 || dims[4] == 0)
        return false;
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_3d(CUtensorMap *map, const void *base, const uint64_t dims[3], const uint64_t strides_bytes[2],
                  const uint32_t box[3])
{
    auto fn = encode_fn();
    if (!fn || dims[0] == 0 || dims[1] == 0 || dims[2] == 0)
        return false;
    cuuint64_t d[3] = {dims[0], dims[1], dims[2]}, st[2] = {strides_bytes[0], strides_bytes[1]};
    cuuint32_t bx[3] = {box[0], box[1], box[2]}, estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), d, st, bx, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace nsa
