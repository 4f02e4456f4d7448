// C ABI of libkda: argument validation and dispatch (see include/kda.h).
#include <stdint.h>
#include <string.h>

#include <mutex>

#include <cuda_runtime.h>

#include "kda_launch.h"

// The library is built with hidden visibility; the C ABI declared in kda.h is exported.
#pragma GCC visibility push(default)
#include "kda.h"
#pragma GCC visibility pop

namespace {

constexpr int kMaxDevices = 64;
// 0 = unknown, 1 = supported (cc 10.3), 2 = unsupported.  Written once per device;
// a benign race writes the same value twice.
volatile int g_device_ok[kMaxDevices];

struct Range {
    uintptr_t lo, hi;
};

bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

kda_status_t check_shape(int B, int T, int H, bool varlen = false) {
    if (B <= 0 || T <= 0 || H <= 0 || H > KDA_MAX_H) return KDA_ERR_SHAPE;
    if (!varlen && T % KDA_BT != 0) return KDA_ERR_SHAPE;
    const long long rows = (long long)B * T * H;
    const long long units = rows / KDA_BT;
    if (units > 0x7fffffffLL) return KDA_ERR_SHAPE;     // grid limit
    if ((long long)B * T > 0x7fffffffLL) return KDA_ERR_SHAPE;  // 32-bit TMA row coordinate
    if (rows > (1LL << 52) / KDA_K) return KDA_ERR_SHAPE; // index arithmetic headroom
    return KDA_OK;
}

kda_status_t check_args(const void *q, const void *k, const float *g, const float *beta,
                        const float *dAqk, const float *dAkk, float *dq, float *dk,
                        float *db, float *dg, int B, int T, int H, kda_dtype_t dt,
                        bool device_alignment) {
    if (!q || !k || !g || !beta || !dAqk || !dAkk || !dq || !dk || !db || !dg)
        return KDA_ERR_NULL;
    kda_status_t st = check_shape(B, T, H);
    if (st != KDA_OK) return st;
    if (dt != KDA_BF16 && dt != KDA_FP16) return KDA_ERR_DTYPE;
    if (device_alignment) {
        const void *a16[] = {q, k, g, dAqk, dAkk, dq, dk, dg};
        for (const void *p : a16)
            if ((uintptr_t)p % 16u) return KDA_ERR_ALIGN;
        if ((uintptr_t)beta % 4u || (uintptr_t)db % 4u) return KDA_ERR_ALIGN;
    }
    const size_t rows = (size_t)B * T * H;
    const Range in[] = {
        {(uintptr_t)q, (uintptr_t)q + rows * KDA_K * 2},
        {(uintptr_t)k, (uintptr_t)k + rows * KDA_K * 2},
        {(uintptr_t)g, (uintptr_t)g + rows * KDA_K * 4},
        {(uintptr_t)beta, (uintptr_t)beta + rows * 4},
        {(uintptr_t)dAqk, (uintptr_t)dAqk + rows * KDA_BT * 4},
        {(uintptr_t)dAkk, (uintptr_t)dAkk + rows * KDA_BT * 4},
    };
    const Range out[] = {
        {(uintptr_t)dq, (uintptr_t)dq + rows * KDA_K * 4},
        {(uintptr_t)dk, (uintptr_t)dk + rows * KDA_K * 4},
        {(uintptr_t)db, (uintptr_t)db + rows * 4},
        {(uintptr_t)dg, (uintptr_t)dg + rows * KDA_K * 4},
    };
    for (int o = 0; o < 4; ++o) {
        for (const Range &r : in)
            if (overlaps(out[o], r)) return KDA_ERR_OVERLAP;
        for (int p = o + 1; p < 4; ++p)
            if (overlaps(out[o], out[p])) return KDA_ERR_OVERLAP;
    }
    return KDA_OK;
}

kda_status_t check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices && g_device_ok[dev] != 0)
        return g_device_ok[dev] == 1 ? KDA_OK : KDA_ERR_UNSUPPORTED_DEVICE;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return KDA_ERR_CUDA;
    const bool ok = (major == 10 && minor == 3);
    if (dev >= 0 && dev < kMaxDevices) g_device_ok[dev] = ok ? 1 : 2;
    return ok ? KDA_OK : KDA_ERR_UNSUPPORTED_DEVICE;
}

// Validation of the extended entry point: q/k have H heads, everything else HV.
kda_status_t check_ex(const void *q, const void *k, const float *g, const float *beta,
                      const float *dAqk, const float *dAkk, void *dq, void *dk, float *db,
                      float *dg, int B, int T, int H, kda_dtype_t dt,
                      const kda_intra_bwd_opts_t &o) {
    if (!q || !k || !g || !beta || !dAqk || !dAkk || !dq || !dk || !db || !dg)
        return KDA_ERR_NULL;
    const int HV = o.HV ? o.HV : H;
    if (H <= 0 || HV <= 0 || HV % H != 0) return KDA_ERR_SHAPE;
    const bool varlen = o.cu_seqlens || o.chunk_indices;
    if (varlen) {
        if (!o.cu_seqlens || (!o.chunk_indices && o.num_chunks > 0)) return KDA_ERR_NULL;
        if (B != 1 || o.num_seqs <= 0 || o.num_chunks < 0) return KDA_ERR_SHAPE;
        if ((long long)o.num_chunks * HV > 0x7fffffffLL) return KDA_ERR_SHAPE;
        if ((uintptr_t)o.cu_seqlens % 4u || (uintptr_t)o.chunk_indices % 4u)
            return KDA_ERR_ALIGN;
    }
    kda_status_t st = check_shape(B, T, HV, varlen);
    if (st != KDA_OK) return st;
    if (dt != KDA_BF16 && dt != KDA_FP16) return KDA_ERR_DTYPE;
    if (o.fold_dg != 0 && o.fold_dg != 1) return KDA_ERR_OPTION;
    if (o.dqdk_io_dtype != 0 && o.dqdk_io_dtype != 1) return KDA_ERR_OPTION;
    if (o.dqdk_io_dtype && HV != H) return KDA_ERR_OPTION;
    if (o.factor_diag != 0 && o.factor_diag != 1) return KDA_ERR_OPTION;
    if (o.split_tf32 != 0 && o.split_tf32 != 1) return KDA_ERR_OPTION;
    if (o.split_tf32 && (varlen || o.fold_dg || o.dqdk_io_dtype || o.factor_diag || o.dq_in ||
                         o.dk_in || o.dg_in || o.db_in))
        return KDA_ERR_OPTION;
    const void *a16[] = {q, k, g, dAqk, dAkk, dq, dk, dg};
    for (const void *p : a16)
        if ((uintptr_t)p % 16u) return KDA_ERR_ALIGN;
    const void *a4[] = {beta, db, o.dq_in, o.dk_in, o.dg_in, o.db_in};
    for (const void *p : a4)
        if ((uintptr_t)p % 4u) return KDA_ERR_ALIGN;
    const size_t rq = (size_t)B * T * H, rv = (size_t)B * T * HV;
    const size_t odq = o.dqdk_io_dtype ? 2 : 4;
    const Range in[] = {
        {(uintptr_t)q, (uintptr_t)q + rq * KDA_K * 2},
        {(uintptr_t)k, (uintptr_t)k + rq * KDA_K * 2},
        {(uintptr_t)g, (uintptr_t)g + rv * KDA_K * 4},
        {(uintptr_t)beta, (uintptr_t)beta + rv * 4},
        {(uintptr_t)dAqk, (uintptr_t)dAqk + rv * KDA_BT * 4},
        {(uintptr_t)dAkk, (uintptr_t)dAkk + rv * KDA_BT * 4},
        {(uintptr_t)o.cu_seqlens,
         varlen ? (uintptr_t)o.cu_seqlens + ((size_t)o.num_seqs + 1) * 4 : 0},
        {(uintptr_t)o.chunk_indices,
         varlen ? (uintptr_t)o.chunk_indices + (size_t)o.num_chunks * 8 : 0},
    };
    const Range opt_in[] = {
        {(uintptr_t)o.dq_in, o.dq_in ? (uintptr_t)o.dq_in + rv * KDA_K * 4 : 0},
        {(uintptr_t)o.dk_in, o.dk_in ? (uintptr_t)o.dk_in + rv * KDA_K * 4 : 0},
        {(uintptr_t)o.db_in, o.db_in ? (uintptr_t)o.db_in + rv * 4 : 0},
        {(uintptr_t)o.dg_in, o.dg_in ? (uintptr_t)o.dg_in + rv * KDA_K * 4 : 0},
    };
    const Range out[] = {
        {(uintptr_t)dq, (uintptr_t)dq + rv * KDA_K * odq},
        {(uintptr_t)dk, (uintptr_t)dk + rv * KDA_K * odq},
        {(uintptr_t)db, (uintptr_t)db + rv * 4},
        {(uintptr_t)dg, (uintptr_t)dg + rv * KDA_K * 4},
    };
    for (int a = 0; a < 4; ++a) {
        for (const Range &r : in)
            if (overlaps(out[a], r)) return KDA_ERR_OVERLAP;
        for (int b = a + 1; b < 4; ++b)
            if (overlaps(out[a], out[b])) return KDA_ERR_OVERLAP;
        for (int b = 0; b < 4; ++b) {
            if (!opt_in[b].lo) continue;
            // an incoming gradient may be its own output exactly (in place), nothing else
            const bool same = (a == b) && opt_in[b].lo == out[a].lo && opt_in[b].hi == out[a].hi;
            if (!same && overlaps(out[a], opt_in[b])) return KDA_ERR_OVERLAP;
        }
    }
    return KDA_OK;
}

// Bounds-checked debug build: the caller's device flag word (kda_debug_set_flags),
// passed to every launch.  Always null in the normal build.
unsigned *g_debug_flags = nullptr;

kda::BwdArgs pack(const void *q, const void *k, const float *g, const float *beta,
                  const float *dAqk, const float *dAkk, float *dq, float *dk, float *db,
                  float *dg, int B, int T, int H, kda_dtype_t dt) {
    kda::BwdArgs a;
    a.q = q; a.k = k; a.g = g; a.beta = beta; a.dAqk = dAqk; a.dAkk = dAkk;
    a.dq = dq; a.dk = dk; a.db = db; a.dg = dg;
    a.B = B; a.T = T; a.H = H;
    a.fp16 = (dt == KDA_FP16);
    a.dbg = g_debug_flags;
    return a;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// kda_intra_bwd_host's internal streams and events, made once per device.
constexpr int kMaxPieces = 64;
struct HostPipe {
    std::mutex mu;  // held while one call enqueues its work
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev[2 * kMaxPieces + 5] = {};
};
std::mutex g_pipe_mu;
HostPipe *g_pipe[kMaxDevices];

kda_status_t host_pipe(HostPipe **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    if (!g_pipe[dev]) {
        HostPipe *hp = new HostPipe;
        bool ok = cudaStreamCreateWithFlags(&hp->s_in, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&hp->s_out, cudaStreamNonBlocking) == cudaSuccess;
        for (cudaEvent_t &e : hp->ev)
            ok = ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            for (cudaEvent_t e : hp->ev)
                if (e) cudaEventDestroy(e);
            if (hp->s_in) cudaStreamDestroy(hp->s_in);
            if (hp->s_out) cudaStreamDestroy(hp->s_out);
            delete hp;
            return KDA_ERR_CUDA;
        }
        g_pipe[dev] = hp;
    }
    *out = g_pipe[dev];
    return KDA_OK;
}

}  // namespace

extern "C" {

kda_status_t kda_intra_bwd_fp32(const void *q, const void *k, const float *g,
                                const float *beta, const float *dAqk, const float *dAkk,
                                float *dq, float *dk, float *db, float *dg, int B, int T,
                                int H, kda_dtype_t qk_dtype, kda_stream_t stream) {
    kda_status_t st = check_args(q, k, g, beta, dAqk, dAkk, dq, dk, db, dg, B, T, H,
                                 qk_dtype, true);
    if (st != KDA_OK) return st;
    if ((st = check_device()) != KDA_OK) return st;
    (void)cudaGetLastError();  // launch errors below must be this call's own
    const kda::BwdArgs a = pack(q, k, g, beta, dAqk, dAkk, dq, dk, db, dg, B, T, H, qk_dtype);
    return kda::launch_intra_fp32(a, (cudaStream_t)stream) == cudaSuccess ? KDA_OK
                                                                          : KDA_ERR_CUDA;
}

kda_status_t kda_intra_bwd_ex(const void *q, const void *k, const float *g,
                              const float *beta, const float *dAqk, const float *dAkk,
                              void *dq, void *dk, float *db, float *dg, int B, int T, int H,
                              kda_dtype_t qk_dtype, const kda_intra_bwd_opts_t *opts,
                              kda_stream_t stream) {
    kda_intra_bwd_opts_t o;
    memset(&o, 0, sizeof(o));
    if (opts) o = *opts;
    kda_status_t st = check_ex(q, k, g, beta, dAqk, dAkk, dq, dk, db, dg, B, T, H, qk_dtype, o);
    if (st != KDA_OK) return st;
    if ((st = check_device()) != KDA_OK) return st;
    (void)cudaGetLastError();
    kda::BwdArgs a = pack(q, k, g, beta, dAqk, dAkk, (float *)dq, (float *)dk, db, dg, B, T,
                          H, qk_dtype);
    a.HV = o.HV ? o.HV : H;
    a.dq_in = o.dq_in;
    a.dk_in = o.dk_in;
    a.dg_in = o.dg_in;
    a.db_in = o.db_in;
    a.fold_dg = o.fold_dg != 0;
    a.emit_io = o.dqdk_io_dtype != 0;
    a.factor_diag = o.factor_diag != 0;
    a.split = o.split_tf32 != 0;
    a.cu_seqlens = o.cu_seqlens;
    a.chunk_indices = o.chunk_indices;
    a.num_seqs = o.num_seqs;
    a.num_chunks = o.num_chunks;
    return kda::launch_intra_tc(a, (cudaStream_t)stream) == cudaSuccess ? KDA_OK
                                                                        : KDA_ERR_CUDA;
}

kda_status_t kda_intra_bwd(const void *q, const void *k, const float *g, const float *beta,
                           const float *dAqk, const float *dAkk, float *dq, float *dk,
                           float *db, float *dg, int B, int T, int H, kda_dtype_t qk_dtype,
                           kda_stream_t stream) {
    kda_status_t st = check_args(q, k, g, beta, dAqk, dAkk, dq, dk, db, dg, B, T, H,
                                 qk_dtype, true);
    if (st != KDA_OK) return st;
    if ((st = check_device()) != KDA_OK) return st;
    (void)cudaGetLastError();
    const kda::BwdArgs a = pack(q, k, g, beta, dAqk, dAkk, dq, dk, db, dg, B, T, H, qk_dtype);
    return kda::launch_intra_tc(a, (cudaStream_t)stream) == cudaSuccess ? KDA_OK
                                                                        : KDA_ERR_CUDA;
}

kda_status_t kda_intra_fwd_ex(const void *q, const void *k, const float *g, const float *beta,
                              float *Aqk, float *Akk, int B, int T, int H,
                              kda_dtype_t qk_dtype, const kda_intra_fwd_opts_t *opts,
                              kda_stream_t stream) {
    kda_intra_fwd_opts_t o;
    memset(&o, 0, sizeof(o));
    if (opts) o = *opts;
    if (!q || !k || !g || !beta || !Aqk || !Akk) return KDA_ERR_NULL;
    const int HV = o.HV ? o.HV : H;
    if (H <= 0 || HV <= 0 || HV % H != 0) return KDA_ERR_SHAPE;
    const bool varlen = o.cu_seqlens || o.chunk_indices;
    if (varlen) {
        if (!o.cu_seqlens || (!o.chunk_indices && o.num_chunks > 0)) return KDA_ERR_NULL;
        if (B != 1 || o.num_seqs <= 0 || o.num_chunks < 0) return KDA_ERR_SHAPE;
        if ((long long)o.num_chunks * HV > 0x7fffffffLL) return KDA_ERR_SHAPE;
        if ((uintptr_t)o.cu_seqlens % 4u || (uintptr_t)o.chunk_indices % 4u)
            return KDA_ERR_ALIGN;
    }
    kda_status_t st = check_shape(B, T, HV, varlen);
    if (st != KDA_OK) return st;
    if (qk_dtype != KDA_BF16 && qk_dtype != KDA_FP16) return KDA_ERR_DTYPE;
    const void *a16[] = {q, k, g, Aqk, Akk};
    for (const void *p : a16)
        if ((uintptr_t)p % 16u) return KDA_ERR_ALIGN;
    if ((uintptr_t)beta % 4u) return KDA_ERR_ALIGN;
    const size_t rq = (size_t)B * T * H, rv = (size_t)B * T * HV;
    const Range in[] = {
        {(uintptr_t)q, (uintptr_t)q + rq * KDA_K * 2},
        {(uintptr_t)k, (uintptr_t)k + rq * KDA_K * 2},
        {(uintptr_t)g, (uintptr_t)g + rv * KDA_K * 4},
        {(uintptr_t)beta, (uintptr_t)beta + rv * 4},
        {(uintptr_t)o.cu_seqlens,
         varlen ? (uintptr_t)o.cu_seqlens + ((size_t)o.num_seqs + 1) * 4 : 0},
        {(uintptr_t)o.chunk_indices,
         varlen ? (uintptr_t)o.chunk_indices + (size_t)o.num_chunks * 8 : 0},
    };
    const Range out[] = {
        {(uintptr_t)Aqk, (uintptr_t)Aqk + rv * KDA_BT * 4},
        {(uintptr_t)Akk, (uintptr_t)Akk + rv * KDA_BT * 4},
    };
    for (const Range &ob : out)
        for (const Range &r : in)
            if (overlaps(ob, r)) return KDA_ERR_OVERLAP;
    if (overlaps(out[0], out[1])) return KDA_ERR_OVERLAP;
    if ((st = check_device()) != KDA_OK) return st;
    (void)cudaGetLastError();
    kda::FwdArgs a;
    a.q = q; a.k = k; a.g = g; a.beta = beta; a.Aqk = Aqk; a.Akk = Akk;
    a.B = B; a.T = T; a.H = H;
    a.fp16 = (qk_dtype == KDA_FP16);
    a.HV = HV;
    a.cu_seqlens = o.cu_seqlens;
    a.chunk_indices = o.chunk_indices;
    a.num_seqs = o.num_seqs;
    a.num_chunks = o.num_chunks;
    a.dbg = g_debug_flags;
    return kda::launch_intra_fwd(a, (cudaStream_t)stream) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_intra_fwd(const void *q, const void *k, const float *g, const float *beta,
                           float *Aqk, float *Akk, int B, int T, int H, kda_dtype_t qk_dtype,
                           kda_stream_t stream) {
    return kda_intra_fwd_ex(q, k, g, beta, Aqk, Akk, B, T, H, qk_dtype, nullptr, stream);
}

size_t kda_intra_bwd_host_workspace_bytes(int B, int T, int H, kda_dtype_t qk_dtype) {
    if (check_shape(B, T, H) != KDA_OK) return 0;
    if (qk_dtype != KDA_BF16 && qk_dtype != KDA_FP16) return 0;
    const size_t rows = (size_t)B * T * H;
    return 2 * align256(rows * KDA_K * 2)        /* q, k */
           + 4 * align256(rows * KDA_K * 4)      /* g, dq, dk, dg */
           + 2 * align256(rows * 4)              /* beta, db */
           + 2 * align256(rows * KDA_BT * 4);    /* dAqk, dAkk */
}

kda_status_t kda_intra_bwd_host(const void *q, const void *k, const float *g,
                                const float *beta, const float *dAqk, const float *dAkk,
                                float *dq, float *dk, float *db, float *dg, int B, int T,
                                int H, kda_dtype_t qk_dtype, void *workspace,
                                size_t workspace_bytes, kda_stream_t stream) {
    kda_status_t st = check_args(q, k, g, beta, dAqk, dAkk, dq, dk, db, dg, B, T, H,
                                 qk_dtype, false);
    if (st != KDA_OK) return st;
    const size_t need = kda_intra_bwd_host_workspace_bytes(B, T, H, qk_dtype);
    if (!workspace || workspace_bytes < need) return KDA_ERR_WORKSPACE;
    if ((uintptr_t)workspace % 256u) return KDA_ERR_ALIGN;
    if ((st = check_device()) != KDA_OK) return st;
    (void)cudaGetLastError();

    const size_t rows = (size_t)B * T * H;
    const size_t nqk = rows * KDA_K * 2, nk4 = rows * KDA_K * 4, nrow = rows * 4,
                 nda = rows * KDA_BT * 4;
    char *w = (char *)workspace;
    char *dq_d = w;                 w += align256(nk4);
    char *dk_d = w;                 w += align256(nk4);
    char *dg_d = w;                 w += align256(nk4);
    char *db_d = w;                 w += align256(nrow);
    char *q_d = w;                  w += align256(nqk);
    char *k_d = w;                  w += align256(nqk);
    char *g_d = w;                  w += align256(nk4);
    char *beta_d = w;               w += align256(nrow);
    char *aqk_d = w;                w += align256(nda);
    char *akk_d = w;

    // Pipeline over pieces: contiguous runs of 64-token chunks of the flattened
    // [1, B*T] token axis (chunks never straddle a sequence since T % 64 == 0).  Inputs
    // of piece p+1 go up on one internal stream while piece p computes on the caller's
    // stream and piece p-1 comes down on another, so both copy directions and the
    // kernel overlap.  Events order everything after earlier work on the caller's
    // stream, and the caller's stream waits for the last copy of each direction.  Every
    // copy carries a fixed cost of a few microseconds, so pieces are large (about 96 MB
    // of input: fewer copies, against a longer pipeline fill and drain), and beta and
    // db, 1/128 of the rows' bytes, move whole: beta before the first piece, db after
    // the last.  A second copy stream per direction measured slower (the copies contend).
    const long long chunks = (long long)B * T / KDA_BT;
    const size_t in_bytes = 2 * nqk + nk4 + nrow + 2 * nda;
    long long P = (long long)(in_bytes / ((size_t)96 << 20));
    if (P < 1) P = 1;
    if (P > kMaxPieces) P = kMaxPieces;
    if (P > chunks) P = chunks;

    // The internal streams and events of this device, made on its first call and kept.
    // The lock makes each call's enqueue sequence contiguous, so an event is recorded
    // again only after every wait on its previous record has been issued (a wait binds
    // to the record current when it is issued).  Calls from several threads therefore
    // queue their copies one call after another on the shared internal streams.
    HostPipe *hp = nullptr;
    if ((st = host_pipe(&hp)) != KDA_OK) return st;
    std::lock_guard<std::mutex> lock(hp->mu);
    cudaStream_t s = (cudaStream_t)stream, s_in = hp->s_in, s_out = hp->s_out;
    cudaEvent_t *ev = hp->ev;
    kda_status_t result = KDA_OK;
    auto fail = [&](kda_status_t code) {
        if (result == KDA_OK) result = code;
    };
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
    cudaEvent_t e_start = ev[0], e_done = ev[1], e_beta = ev[2 * P + 2],
                e_last = ev[2 * P + 3], e_in_done = ev[2 * P + 4];
    if (cudaEventRecord(e_start, s) != cudaSuccess ||
        cudaStreamWaitEvent(s_in, e_start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(s_out, e_start, 0) != cudaSuccess) {
        fail(KDA_ERR_CUDA);
        return result;  // nothing is queued on the internal streams
    }
    if (cudaMemcpyAsync(beta_d, beta, nrow, h2d, s_in) != cudaSuccess ||
        cudaEventRecord(e_beta, s_in) != cudaSuccess ||
        cudaStreamWaitEvent(s, e_beta, 0) != cudaSuccess)
        fail(KDA_ERR_CUDA);
    for (long long p = 0; p < P && result == KDA_OK; ++p) {
        const long long c0 = p * chunks / P, c1 = (p + 1) * chunks / P;
        const size_t r0 = (size_t)c0 * KDA_BT * H, nr = (size_t)(c1 - c0) * KDA_BT * H;
        const int Tp = (int)((c1 - c0) * KDA_BT);
        cudaEvent_t e_in = ev[2 + 2 * p], e_k = ev[3 + 2 * p];
        const size_t oqk = r0 * KDA_K * 2, o4 = r0 * KDA_K * 4, orow = r0 * 4,
                     oda = r0 * KDA_BT * 4;
        const size_t lqk = nr * KDA_K * 2, l4 = nr * KDA_K * 4, lda = nr * KDA_BT * 4;
        if (cudaMemcpyAsync(q_d + oqk, (const char *)q + oqk, lqk, h2d, s_in) != cudaSuccess ||
            cudaMemcpyAsync(k_d + oqk, (const char *)k + oqk, lqk, h2d, s_in) != cudaSuccess ||
            cudaMemcpyAsync(g_d + o4, (const char *)g + o4, l4, h2d, s_in) != cudaSuccess ||
            cudaMemcpyAsync(aqk_d + oda, (const char *)dAqk + oda, lda, h2d, s_in) !=
                cudaSuccess ||
            cudaMemcpyAsync(akk_d + oda, (const char *)dAkk + oda, lda, h2d, s_in) !=
                cudaSuccess ||
            cudaEventRecord(e_in, s_in) != cudaSuccess ||
            cudaStreamWaitEvent(s, e_in, 0) != cudaSuccess) {
            fail(KDA_ERR_CUDA);
            break;
        }
        const kda_status_t st2 = kda_intra_bwd(
            q_d + oqk, k_d + oqk, (const float *)(g_d + o4), (const float *)(beta_d + orow),
            (const float *)(aqk_d + oda), (const float *)(akk_d + oda),
            (float *)(dq_d + o4), (float *)(dk_d + o4), (float *)(db_d + orow),
            (float *)(dg_d + o4), 1, Tp, H, qk_dtype, stream);
        if (st2 != KDA_OK) {
            fail(st2);
            break;
        }
        if (cudaEventRecord(e_k, s) != cudaSuccess ||
            cudaStreamWaitEvent(s_out, e_k, 0) != cudaSuccess ||
            cudaMemcpyAsync((char *)dq + o4, dq_d + o4, l4, d2h, s_out) != cudaSuccess ||
            cudaMemcpyAsync((char *)dk + o4, dk_d + o4, l4, d2h, s_out) != cudaSuccess ||
            cudaMemcpyAsync((char *)dg + o4, dg_d + o4, l4, d2h, s_out) != cudaSuccess) {
            fail(KDA_ERR_CUDA);
            break;
        }
    }
    // db of every piece, once the last kernel is done
    if (result == KDA_OK &&
        (cudaEventRecord(e_last, s) != cudaSuccess ||
         cudaStreamWaitEvent(s_out, e_last, 0) != cudaSuccess ||
         cudaMemcpyAsync(db, db_d, nrow, d2h, s_out) != cudaSuccess))
        fail(KDA_ERR_CUDA);
    // The caller's stream waits for the last copy of both directions, also after a
    // failure midway: no upload still reading the caller's host inputs, and no
    // download still writing its outputs, outlives the caller's stream.
    if (cudaEventRecord(e_done, s_out) != cudaSuccess ||
        cudaEventRecord(e_in_done, s_in) != cudaSuccess ||
        cudaStreamWaitEvent(s, e_done, 0) != cudaSuccess ||
        cudaStreamWaitEvent(s, e_in_done, 0) != cudaSuccess)
        fail(KDA_ERR_CUDA);
    return result;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// kda_intra_bwd_host_static: the host entry point with its device staging in a fixed
// array of this library, for callers that may not allocate device memory.

// The staging buffers.  Every GPU on which this module is loaded holds it until the
// process exits.  Host code must not pass this name to a kernel: on the host it is a
// stand-in, not a device address; scratch_base() looks the address up.
static __device__ __align__(256) unsigned char g_host_scratch[KDA_HOST_STATIC_MAX_BYTES];

namespace {

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices];  // device address of g_host_scratch, per device

// The array's device address on the current device, looked up on the first call there.
kda_status_t scratch_base(char **base) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_host_scratch) != cudaSuccess || !p)
            return KDA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *base = (char *)g_scratch_addr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" {

kda_status_t kda_intra_bwd_host_static(const void *q, const void *k, const float *g,
                                       const float *beta, const float *dAqk,
                                       const float *dAkk, float *dq, float *dk, float *db,
                                       float *dg, int B, int T, int H, kda_dtype_t qk_dtype,
                                       kda_stream_t stream) {
    kda_status_t st = check_args(q, k, g, beta, dAqk, dAkk, dq, dk, db, dg, B, T, H,
                                 qk_dtype, false);
    if (st != KDA_OK) return st;
    if (kda_intra_bwd_host_workspace_bytes(B, T, H, qk_dtype) > KDA_HOST_STATIC_MAX_BYTES)
        return KDA_ERR_TOO_LARGE;
    if ((st = check_device()) != KDA_OK) return st;
    char *w = nullptr;
    if ((st = scratch_base(&w)) != KDA_OK) return st;
    (void)cudaGetLastError();

    // Same carving as kda_intra_bwd_host.  The uploads overwrite every input byte and
    // the kernel every output byte, so the previous call's contents never leak in.
    const size_t rows = (size_t)B * T * H;
    const size_t nqk = rows * KDA_K * 2, nk4 = rows * KDA_K * 4, nrow = rows * 4,
                 nda = rows * KDA_BT * 4;
    char *dq_d = w;                 w += align256(nk4);
    char *dk_d = w;                 w += align256(nk4);
    char *dg_d = w;                 w += align256(nk4);
    char *db_d = w;                 w += align256(nrow);
    char *q_d = w;                  w += align256(nqk);
    char *k_d = w;                  w += align256(nqk);
    char *g_d = w;                  w += align256(nk4);
    char *beta_d = w;               w += align256(nrow);
    char *aqk_d = w;                w += align256(nda);
    char *akk_d = w;

    // One stream, in order: uploads, the kernel, downloads.  At these sizes there is
    // nothing to gain from the pipelined pieces of kda_intra_bwd_host.
    const cudaStream_t s = (cudaStream_t)stream;
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
    if (cudaMemcpyAsync(q_d, q, nqk, h2d, s) != cudaSuccess ||
        cudaMemcpyAsync(k_d, k, nqk, h2d, s) != cudaSuccess ||
        cudaMemcpyAsync(g_d, g, nk4, h2d, s) != cudaSuccess ||
        cudaMemcpyAsync(beta_d, beta, nrow, h2d, s) != cudaSuccess ||
        cudaMemcpyAsync(aqk_d, dAqk, nda, h2d, s) != cudaSuccess ||
        cudaMemcpyAsync(akk_d, dAkk, nda, h2d, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    st = kda_intra_bwd(q_d, k_d, (const float *)g_d, (const float *)beta_d,
                       (const float *)aqk_d, (const float *)akk_d, (float *)dq_d,
                       (float *)dk_d, (float *)db_d, (float *)dg_d, B, T, H, qk_dtype,
                       stream);
    if (st != KDA_OK) return st;
    if (cudaMemcpyAsync(dq, dq_d, nk4, d2h, s) != cudaSuccess ||
        cudaMemcpyAsync(dk, dk_d, nk4, d2h, s) != cudaSuccess ||
        cudaMemcpyAsync(dg, dg_d, nk4, d2h, s) != cudaSuccess ||
        cudaMemcpyAsync(db, db_d, nrow, d2h, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    return KDA_OK;
}

const char *kda_status_str(kda_status_t status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_NULL: return "KDA_ERR_NULL: a required pointer is NULL";
        case KDA_ERR_SHAPE:
            return "KDA_ERR_SHAPE: need B,T > 0, 0 < H <= 65536 and T % 64 == 0 "
                   "(varlen: B == 1, num_seqs > 0, num_chunks >= 0)";
        case KDA_ERR_DTYPE: return "KDA_ERR_DTYPE: qk_dtype must be KDA_BF16 or KDA_FP16";
        case KDA_ERR_ALIGN: return "KDA_ERR_ALIGN: a pointer is misaligned";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: a CUDA call or kernel launch failed";
        case KDA_ERR_UNSUPPORTED_DEVICE:
            return "KDA_ERR_UNSUPPORTED_DEVICE: needs compute capability 10.3 (sm_103a)";
        case KDA_ERR_OVERLAP: return "KDA_ERR_OVERLAP: argument buffers overlap";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE: workspace missing or too small";
        case KDA_ERR_OPTION: return "KDA_ERR_OPTION: unsupported option combination";
        case KDA_ERR_TOO_LARGE:
            return "KDA_ERR_TOO_LARGE: the problem needs more than the library's fixed "
                   "32 MiB of staging (KDA_HOST_STATIC_MAX_BYTES); use kda_intra_bwd_host "
                   "with a workspace";
    }
    return "KDA_ERR_UNKNOWN";
}

int kda_abi_version(void) { return KDA_ABI_VERSION; }

#ifdef KDA_DEBUG_CHECKS
int kda_debug_checks(void) { return 1; }

kda_status_t kda_debug_set_flags(unsigned int *device_word) {
    if ((uintptr_t)device_word % 4u) return KDA_ERR_ALIGN;
    g_debug_flags = device_word;
    return KDA_OK;
}
#else
int kda_debug_checks(void) { return 0; }

kda_status_t kda_debug_set_flags(unsigned int *) { return KDA_ERR_OPTION; }
#endif

}  // extern "C"
