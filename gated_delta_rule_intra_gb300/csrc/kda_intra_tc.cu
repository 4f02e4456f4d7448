// Host side of the tensor-core kernel: tensor maps, the SM count, and the dispatch
// to the instantiations per q/k element type, sequence layout and diagonal-block
// form (kda_intra_tc_{bf16,fp16}[_varlen][_fd].cu).
#include "kda_intra_tc.cuh"

namespace kda {

cudaError_t launch_tc_bf16(const BwdArgs &a, cudaStream_t stream);
cudaError_t launch_tc_fp16(const BwdArgs &a, cudaStream_t stream);
cudaError_t launch_tc_bf16_varlen(const BwdArgs &a, cudaStream_t stream);
cudaError_t launch_tc_fp16_varlen(const BwdArgs &a, cudaStream_t stream);
cudaError_t launch_tc_bf16_fd(const BwdArgs &a, cudaStream_t stream);
cudaError_t launch_tc_fp16_fd(const BwdArgs &a, cudaStream_t stream);
cudaError_t launch_tc_bf16_varlen_fd(const BwdArgs &a, cudaStream_t stream);
cudaError_t launch_tc_fp16_varlen_fd(const BwdArgs &a, cudaStream_t stream);
cudaError_t launch_tc_bf16_split(const BwdArgs &a, cudaStream_t stream);
cudaError_t launch_tc_fp16_split(const BwdArgs &a, cudaStream_t stream);

namespace tcimpl {
namespace {
int g_num_sms[kMaxDev];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t get_encoder() {
    if (g_encode) return cudaSuccess;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return cudaSuccess;
}

cudaError_t encode(CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *base,
                   const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box,
                   CUtensorMapL2promotion l2 = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(m, dt, (cuuint32_t)rank, const_cast<void *>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, l2,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

namespace {

// What a set of tensor maps depends on.  A map is a pure function of these, so a set
// encoded once serves every later call with the same key (the host's per-call cost).
struct MapKey {
    const void *q, *k, *g, *dAqk, *dAkk;
    int B, T, H, HV;
    bool fp16, varlen;
    bool operator==(const MapKey &o) const {
        return q == o.q && k == o.k && g == o.g && dAqk == o.dAqk && dAkk == o.dAkk &&
               B == o.B && T == o.T && H == o.H && HV == o.HV && fp16 == o.fp16 &&
               varlen == o.varlen;
    }
};
thread_local MapKey t_key;
thread_local TmaMaps t_maps;
thread_local bool t_valid = false;

cudaError_t encode_maps(const BwdArgs &a, TmaMaps *tm);

}  // namespace

cudaError_t make_maps(const BwdArgs &a, TmaMaps *tm) {
    const MapKey key = {a.q, a.k, a.g, a.dAqk, a.dAkk, a.B, a.T, a.H,
                        a.HV > 0 ? a.HV : a.H, a.fp16, a.cu_seqlens != nullptr};
    if (t_valid && key == t_key) {
        *tm = t_maps;
        return cudaSuccess;
    }
    const cudaError_t e = encode_maps(a, tm);
    if (e != cudaSuccess) return e;
    t_key = key;
    t_maps = *tm;
    t_valid = true;
    return cudaSuccess;
}

namespace {

cudaError_t encode_maps(const BwdArgs &a, TmaMaps *tm) {
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    const cuuint64_t rows = (cuuint64_t)a.B * a.T, HQ = (cuuint64_t)a.H;
    const cuuint64_t H = (cuuint64_t)(a.HV > 0 ? a.HV : a.H);
    const CUtensorMapDataType io =
        a.fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    {  // q, k: (channel, head, token row); one unit = box (128, 1, 64)
        const cuuint64_t dims[3] = {KD, HQ, rows};
        const cuuint64_t str[2] = {KD * 2, HQ * KD * 2};
        const cuuint32_t box[3] = {KD, 1, BT};
        if ((e = encode(&tm->q, io, 3, a.q, dims, str, box)) != cudaSuccess) return e;
        if ((e = encode(&tm->k, io, 3, a.k, dims, str, box)) != cudaSuccess) return e;
    }
    {  // g
        const cuuint64_t dims[3] = {KD, H, rows};
        const cuuint64_t str[2] = {KD * 4, H * KD * 4};
        const cuuint32_t box[3] = {KD, 1, BT};
        if ((e = encode(&tm->g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.g, dims, str, box)) !=
            cudaSuccess)
            return e;
        const cuuint32_t box16[3] = {KD, 1, BC};
        if ((e = encode(&tm->g16, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.g, dims, str, box16)) !=
            cudaSuccess)
            return e;
    }
    {
        const cuuint64_t dims[3] = {KD, HQ, rows};
        const cuuint64_t str[2] = {KD * 2, HQ * KD * 2};
        const cuuint32_t box16[3] = {KD, 1, BC};
        if ((e = encode(&tm->q16, io, 3, a.q, dims, str, box16)) != cudaSuccess) return e;
        if ((e = encode(&tm->k16, io, 3, a.k, dims, str, box16)) != cudaSuccess) return e;
    }
    // no L2 promotion for dA: a promoted fetch would also pull the rows' unused upper part
    const CUtensorMapL2promotion l2 = CU_TENSOR_MAP_L2_PROMOTION_NONE;
    if (!a.cu_seqlens) {
        // dA: (col%4, row%8, row/8, col/4, head); the box of row-block t covers its blocks
        // (t, 0..t) and lands them as tensor-core operands (4 floats, 8 rows, 2 row groups,
        // then column chunks: block j at j KB)
        const cuuint64_t dims[5] = {4, 8, rows / 8, BT / 4, H};
        const cuuint64_t str[4] = {H * BT * 4, 8 * H * BT * 4, 16, BT * 4};
        for (int t = 0; t < NBLK; ++t) {
            const cuuint32_t box[5] = {4, 8, 2, (cuuint32_t)(4 * (t + 1)), 1};
            if ((e = encode(&tm->daqk[t], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, a.dAqk, dims, str,
                            box, l2)) != cudaSuccess)
                return e;
            if ((e = encode(&tm->dakk[t], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, a.dAkk, dims, str,
                            box, l2)) != cudaSuccess)
                return e;
        }
    } else {
        // variable-length units start at any row: (col%4, row, col/4, head), box
        // (4, 16, 4(t+1), 1) -- the same bytes in the same operand layout (row n of a
        // block at n*16 bytes inside each 256-byte column chunk)
        const cuuint64_t dims[4] = {4, rows, BT / 4, H};
        const cuuint64_t str[3] = {H * BT * 4, 16, BT * 4};
        for (int t = 0; t < NBLK; ++t) {
            const cuuint32_t box[4] = {4, BC, (cuuint32_t)(4 * (t + 1)), 1};
            if ((e = encode(&tm->daqk[t], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.dAqk, dims, str,
                            box, l2)) != cudaSuccess)
                return e;
            if ((e = encode(&tm->dakk[t], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.dAkk, dims, str,
                            box, l2)) != cudaSuccess)
                return e;
        }
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t num_sms(int *n, int *devp) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int v = (dev >= 0 && dev < kMaxDev) ? g_num_sms[dev] : 0;
    if (v == 0) {
        if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        if (dev >= 0 && dev < kMaxDev) g_num_sms[dev] = v;
    }
    *n = v;
    *devp = dev;
    return cudaSuccess;
}

}  // namespace tcimpl

cudaError_t launch_intra_tc(const BwdArgs &a, cudaStream_t stream) {
    if (a.split) return a.fp16 ? launch_tc_fp16_split(a, stream) : launch_tc_bf16_split(a, stream);
    if (a.factor_diag) {
        if (a.cu_seqlens)
            return a.fp16 ? launch_tc_fp16_varlen_fd(a, stream)
                          : launch_tc_bf16_varlen_fd(a, stream);
        return a.fp16 ? launch_tc_fp16_fd(a, stream) : launch_tc_bf16_fd(a, stream);
    }
    if (a.cu_seqlens)
        return a.fp16 ? launch_tc_fp16_varlen(a, stream) : launch_tc_bf16_varlen(a, stream);
    return a.fp16 ? launch_tc_fp16(a, stream) : launch_tc_bf16(a, stream);
}

}  // namespace kda
