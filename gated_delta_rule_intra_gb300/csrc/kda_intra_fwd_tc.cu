// Tensor-core kernel for the KDA intra-chunk forward (sm_103a, tcgen05 + TMEM + TMA):
// the two score matrices of every unit (b, h, 64-token chunk),
//     Aqk[r,s] = sum_d q[r,d] k[s,d] 2^(g[r,d] - g[s,d])            (s <= r)
//     Akk[r,s] = beta[r] sum_d k[r,d] k[s,d] 2^(g[r,d] - g[s,d])    (s <  r)
// (bwd_intra page, module docstring: the forward whose gradient the backward takes),
// written as [B,T,H,64] fp32 rows with zeros outside the support.
//
// Persistent grid, one 512-thread CTA per SM, two TMA input stages.  Per unit:
//  * cross-sub-block blocks (r in block t, s in block j < t) through the target
//    block's first row: 2^(g_r - g_s) = 2^(g_r - g_16t) * 2^(g_16t - g_s), both
//    exponents <= 0 (the gate-magnitude law).  A[m, d] = q_r 2^(g_r - g_16t) for
//    TMEM lane m = r and beta_r k_r 2^(g_r - g_16t) for lane m = 64 + r (written by
//    tcgen05.st from the thread owning the lane); B_t[s, d] = k_s 2^(g_16t - g_s)
//    for s < 16t in shared memory.  Three TF32 MMA chains (N = 16t, K = 128) give
//    every cross entry of Aqk (lanes 0..63) and Akk (lanes 64..127) at once.
//  * diagonal 16x16 blocks on the FP32 pipes with one exp2 per (r, s, d): thread
//    (row pair {a, 15-a} of block i, 8 channels) sums over its channels, then a
//    transposed shuffle reduction over the 16 lanes of its half-warp finishes the
//    sum over d.
//  * both tiles are assembled in a 128B-swizzled staging buffer whose entries
//    outside the support stay zero, and leave through four TMA stores.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kda_common.cuh"
#include "kda_launch.h"
#include "tc_ptx.cuh"

namespace kda {
namespace fwdimpl {
namespace {

constexpr int FW_THREADS = 512;
constexpr uint32_t SPIN_LIMIT = 1u << 22;

// ---- shared memory (offsets from a 1024-byte aligned base) ----
// Input stage: q, k as two 8 KB boxes each (64 rows x 64 elements = 128 B rows), g as
// four 8 KB boxes (64 rows x 32 floats); every box is 128B-swizzled: the 16-byte chunk
// c of row r sits at chunk position c ^ (r % 8) of the row's 128 bytes.
constexpr int FS_Q = 0;
constexpr int FS_K = 16384;
constexpr int FS_G = 32768;
constexpr int FSTAGE = 65536;
constexpr int FM_STG = 2 * FSTAGE;              // Aqk, Akk tiles: 2 x 2 swizzled 8 KB boxes
constexpr int FM_B = FM_STG + 32768;            // B_1, B_2, B_3: [16t][128] tf32, K-major
constexpr int FM_BETA = FM_B + 49152;           // f32 [2][64]
constexpr int FM_DIAG = FM_BETA + 512;          // f32 [2][512]: diagonal sums until the epilogue
constexpr int FM_BAR = FM_DIAG + 2 * 512 * 4;   // full[2], mma, staging free, operands
constexpr int FM_TSLOT = FM_BAR + 40;
constexpr int FM_META = FM_TSLOT + 8;           // varlen: per stage {first token row, valid rows}
constexpr int FM_LUT = FM_META + 16;            // varlen: the same for this CTA's units,
constexpr int LUT_BATCH = 32;                   // two batches of 32
constexpr int FM_TOTAL = FM_LUT + 2 * LUT_BATCH * 8;
constexpr int FM_ALLOC = FM_TOTAL + 1024;       // slack for aligning the base
static_assert(FM_STG % 1024 == 0, "swizzled staging needs 1024-byte alignment");
static_assert(FM_ALLOC <= 232448, "shared memory");

constexpr uint32_t FSTAGE_TX_BYTES = 2 * BT * KD * 2 + BT * KD * 4;
constexpr uint32_t FULL_ARRIVALS = 1 + 32;

// B_t at FM_B + boff(t): element (n, k) at (k/4)*256t + (n/8)*128 + (n%8)*16 + (k%4)*4
__host__ __device__ constexpr int boff(int t) { return 4096 * t * (t - 1); }
// TMEM: A in columns 0..127, D_t (16t columns) at tm_d(t)
__device__ __forceinline__ uint32_t tm_d(int t) { return 128u + 8u * (uint32_t)(t * (t - 1)); }
constexpr uint32_t TM_COLS = 256;

// byte offset of element (r, c) of a swizzled tile made of 128-byte-row boxes
template <int ESIZE>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    constexpr int PER_ROW = 128 / ESIZE;  // elements per box row
    const int box = c / PER_ROW, cc = c % PER_ROW;
    const int chunk = (cc * ESIZE) >> 4, within = (cc * ESIZE) & 15;
    return (uint32_t)(box * 8192 + r * 128 + ((chunk ^ (r & 7)) << 4) + within);
}
// staging: tensor 0 = Aqk, 1 = Akk; column s in box s / 32
__device__ __forceinline__ uint32_t stg_off(int tensor, int r, int s) {
    return (uint32_t)(tensor * 16384) + swz<4>(r, s);
}

struct FwdMaps {
    CUtensorMap q, k, g, aqk, akk;
};

// Options: H in the kernel is the number of heads of g, beta and the outputs (HV); q
// and k have HV / G heads.  Variable-length launches: unit u is head u % H of chunk
// chunk_indices[2c+1] of sequence chunk_indices[2c], c = u / H, sequence n being
// tokens [cu_seqlens[n], cu_seqlens[n+1]).
struct FwdExtras {
    int G;
    const int *cu_seqlens, *chunk_indices;
    int num_seqs;
    // bounds-checked debug build: the flag word and the extents checked against
    unsigned *dbg;
    size_t nrows;    // token rows x heads of g, beta and the outputs
    int num_chunks;  // entries of chunk_indices (variable-length launches)
};

// First token row and valid rows (1..64) of a variable-length unit; {0, 0} for an
// entry that names no chunk of cu_seqlens (the unit is then skipped).
__device__ __forceinline__ void varlen_rows(long long u, int H, int T, const FwdExtras &ex,
                                            int &start, int &len) {
    const size_t c = (size_t)((unsigned)u / (unsigned)H);
    start = 0;
    len = 0;
    if (!dbg_ok(ex.dbg, 2 * c + 1, 2 * (size_t)ex.num_chunks, DBG_LOAD)) return;
    const int n = __ldg(ex.chunk_indices + 2 * c), j = __ldg(ex.chunk_indices + 2 * c + 1);
    if (n >= 0 && n < ex.num_seqs && j >= 0) {
        const long long bos = __ldg(ex.cu_seqlens + n), eos = __ldg(ex.cu_seqlens + n + 1);
        const long long st = bos + (long long)BT * j;
        if (bos >= 0 && st < eos && eos <= T) {
            start = (int)st;
            len = (int)(eos - st < BT ? eos - st : BT);
        }
    }
}

// One warp queues a unit's copies: 8 swizzled TMA boxes from lane 0 (rows past the
// tensor's end are zero-filled), beta as 64 four-byte cp.async copies from all lanes
// (zero-filled past the unit's valid rows).  A variable-length unit's row range is
// recorded in `meta` by lane 0 before its arrival on the stage barrier; it comes from
// `known` ({first row, valid rows}) when given, else from the chunk table.
template <typename io_t, bool VARLEN>
__device__ __forceinline__ void load_unit(unsigned char *st, float *sbeta, uint64_t *full,
                                          int *meta, const FwdMaps &tm,
                                          const float *__restrict__ beta, long long u, int T,
                                          int H, const FwdExtras &ex, int lane,
                                          const int *known = nullptr) {
    int row, h, len = BT;
    if constexpr (VARLEN) {
        if (known) {
            row = known[0];
            len = known[1];
        } else {
            varlen_rows(u, H, T, ex, row, len);
        }
        h = (int)((unsigned)u % (unsigned)H);
        if (lane == 0) {
            meta[0] = row;
            meta[1] = len;
        }
    } else {
        const Unit x = decode_unit(u, H, T / BT);
        row = x.b * T + x.c * BT;
        h = x.h;
    }
    if (lane == 0) {
        tc::mbar_arrive_expect_tx(full, FSTAGE_TX_BYTES);
        for (int b = 0; b < 2; ++b) {
            tc::tma_load_3d(st + FS_Q + b * 8192, &tm.q, 64 * b, h / ex.G, row, full);
            tc::tma_load_3d(st + FS_K + b * 8192, &tm.k, 64 * b, h / ex.G, row, full);
        }
        for (int b = 0; b < 4; ++b) tc::tma_load_3d(st + FS_G + b * 8192, &tm.g, 32 * b, h, row, full);
    }
    const float *b0 = beta + ((size_t)row * H + h);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int r = lane + 32 * e;
        const uint32_t s = tc::smem_u32(sbeta + r);
        const bool take = r < len && dbg_ok(ex.dbg, (size_t)(row + r) * H + h, ex.nrows, DBG_LOAD);
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(s),
                     "l"(take ? b0 + (size_t)r * H : beta), "r"(take ? 4 : 0)
                     : "memory");
    }
    tc::cp_async_mbar_arrive_noinc(full);
}

// The same copies spread over warps 0..8 (part = warp): warp 0 arms the barrier and
// issues the first q box, warps 1..7 one box each, warp 8 the beta copies; every warp
// of the CTA leaves the unit's barrier together, so no warp carries all of them.
template <typename io_t, bool VARLEN>
__device__ __forceinline__ void load_unit_part(int part, unsigned char *st, float *sbeta,
                                               uint64_t *full, int *meta, const FwdMaps &tm,
                                               const float *__restrict__ beta, long long u,
                                               int T, int H, const FwdExtras &ex, int lane,
                                               const int *known) {
    int row, h, len = BT;
    if constexpr (VARLEN) {
        row = known[0];
        len = known[1];
        h = (int)((unsigned)u % (unsigned)H);
    } else {
        const Unit x = decode_unit(u, H, T / BT);
        row = x.b * T + x.c * BT;
        h = x.h;
    }
    if (part < 8) {
        if (lane == 0) {
            if (part == 0) {
                if constexpr (VARLEN) {
                    meta[0] = row;
                    meta[1] = len;
                }
                tc::mbar_arrive_expect_tx(full, FSTAGE_TX_BYTES);
            }
            if (part < 2)
                tc::tma_load_3d(st + FS_Q + part * 8192, &tm.q, 64 * part, h / ex.G, row, full);
            else if (part < 4)
                tc::tma_load_3d(st + FS_K + (part - 2) * 8192, &tm.k, 64 * (part - 2), h / ex.G,
                                row, full);
            else
                tc::tma_load_3d(st + FS_G + (part - 4) * 8192, &tm.g, 32 * (part - 4), h, row,
                                full);
        }
        return;
    }
    const float *b0 = beta + ((size_t)row * H + h);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int r = lane + 32 * e;
        const uint32_t s = tc::smem_u32(sbeta + r);
        const bool take = r < len && dbg_ok(ex.dbg, (size_t)(row + r) * H + h, ex.nrows, DBG_LOAD);
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(s),
                     "l"(take ? b0 + (size_t)r * H : beta), "r"(take ? 4 : 0)
                     : "memory");
    }
    tc::cp_async_mbar_arrive_noinc(full);
}

// Sum of v[0..15] over the 16 lanes of a half-warp, transposed: lane (lane & 15) = j
// ends with the total of index j in v[0].  15 shuffles.
__device__ __forceinline__ float reduce16(float (&v)[16], int lane) {
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1) {
        const bool hi = (lane & w) != 0;
#pragma unroll
        for (int j = 0; j < w; ++j) {
            const float send = hi ? v[j] : v[j + w];
            const float keep = hi ? v[j + w] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
    }
    return v[0];
}

// Eight channels {4c..4c+3, 64+4c..64+4c+3} of one row of a swizzled stage tile.
template <typename io_t>
__device__ __forceinline__ void ld8_io(const unsigned char *tile, int r, int c, float2 (&x)[4]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint2 w = *reinterpret_cast<const uint2 *>(tile + swz<2>(r, 64 * h + 4 * c));
        const io_t *e = reinterpret_cast<const io_t *>(&w);
        x[2 * h] = make_float2(to_f32(e[0]), to_f32(e[1]));
        x[2 * h + 1] = make_float2(to_f32(e[2]), to_f32(e[3]));
    }
}
__device__ __forceinline__ void ld8_f32(const unsigned char *tile, int r, int c, float2 (&x)[4]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float4 w = *reinterpret_cast<const float4 *>(tile + swz<4>(r, 64 * h + 4 * c));
        x[2 * h] = make_float2(w.x, w.y);
        x[2 * h + 1] = make_float2(w.z, w.w);
    }
}

// VARLEN: units from cu_seqlens / chunk_indices.  A unit's rows past its sequence's
// end never reach a valid output (row r only meets sources s <= r), so nothing is
// masked on the way in; a short chunk's valid rows leave through plain stores.
template <typename io_t, bool VARLEN>
__global__ void __launch_bounds__(FW_THREADS, 1)
kda_intra_fwd_tc_kernel(const __grid_constant__ FwdMaps tm, const float *__restrict__ beta,
                        float *Aqk, float *Akk, int T, int H, long long units,
                        const FwdExtras ex) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem =
        smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);  // 1024-aligned
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + FM_BAR);
    uint64_t *mbar = full + 2;
    uint64_t *stg_free = full + 3;  // completes once per unit: the last tiles have left
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + FM_TSLOT);
    int *meta = reinterpret_cast<int *>(smem + FM_META);
    unsigned char *stg = smem + FM_STG;
    const long long stride = gridDim.x;

    if (warp == 0) tc::tmem_alloc(tslot, TM_COLS);
    if (tid == 0) {
        tc::mbar_init(&full[0], FULL_ARRIVALS);
        tc::mbar_init(&full[1], FULL_ARRIVALS);
        tc::mbar_init(mbar, 3);                 // one commit per MMA chain
        tc::mbar_init(stg_free, 1);
        tc::mbar_init(stg_free + 1, 16);        // operands written, one arrival per warp
        tc::prefetch_tmap(&tm.q);
        tc::prefetch_tmap(&tm.k);
        tc::prefetch_tmap(&tm.g);
        tc::prefetch_tmap(&tm.aqk);
        tc::prefetch_tmap(&tm.akk);
    }
    // the staging entries outside the support are never written again: zero them once
    for (int x = tid; x < 32768 / 16; x += FW_THREADS)
        reinterpret_cast<uint4 *>(stg)[x] = make_uint4(0u, 0u, 0u, 0u);
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tslot;

    // VARLEN: lane j of warp 0 looks up the row range of this CTA's unit k0 + j, for the
    // refills of a whole batch of units at once (warps 0..8 share every refill)
    int *lut = reinterpret_cast<int *>(smem + FM_LUT);
    auto lookup_batch = [&](const int k0) {
        const long long uk = blockIdx.x + (long long)(k0 + lane) * stride;
        if (uk < units) {
            int start, len;
            varlen_rows(uk, H, T, ex, start, len);
            int *e = lut + ((k0 / LUT_BATCH) & 1) * 2 * LUT_BATCH + 2 * lane;
            e[0] = start;
            e[1] = len;
        }
        __syncwarp();
    };
    if (warp == 0) {
        const long long u0 = blockIdx.x;
        float *sb = reinterpret_cast<float *>(smem + FM_BETA);
        if (u0 < units)
            load_unit<io_t, VARLEN>(smem, sb, &full[0], meta, tm, beta, u0, T, H, ex, lane);
        if (u0 + stride < units)
            load_unit<io_t, VARLEN>(smem + FSTAGE, sb + 64, &full[1], meta + 2, tm, beta,
                                    u0 + stride, T, H, ex, lane);
        if constexpr (VARLEN) {
            lookup_batch(0);
            lookup_batch(LUT_BATCH);
        }
    }

    const float nan = __int_as_float(0x7fc00000);
    bool ok = true;
    int it = 0;
    for (long long u = blockIdx.x; u < units; u += stride, ++it) {
        const int sidx = it & 1;
        unsigned char *st = smem + sidx * FSTAGE;
        const unsigned char *sq = st + FS_Q, *sk = st + FS_K, *sg = st + FS_G;
        const float *sbeta = reinterpret_cast<const float *>(smem + FM_BETA) + 64 * sidx;
        ok &= tc::mbar_wait(&full[sidx], (uint32_t)(it >> 1) & 1u, SPIN_LIMIT);
        // the unit's first token row, head and valid rows (read now: the stage's meta
        // is rewritten by the refill that follows this unit's last barrier)
        int row, h, len = BT;
        if constexpr (VARLEN) {
            row = meta[2 * sidx];
            len = meta[2 * sidx + 1];
            h = (int)((unsigned)u % (unsigned)H);
        } else {
            const Unit x = decode_unit(u, H, T / BT);
            row = x.b * T + x.c * BT;
            h = x.h;
        }

        // ---- prescale: thread = (TMEM lane m, 32 channels).  Lane m < 64 holds the q
        // row m, lane m >= 64 the beta*k row m - 64 (A operand). ----
        {
            const int Lq = warp & 3, d0 = 32 * (warp >> 2);
            const bool isk = Lq >= 2;
            const int r = 32 * (Lq & 1) + lane, t = r >> 4;
            const unsigned char *sx = isk ? sk : sq;
            const float scale = isk ? sbeta[r] : 1.f;
            const uint32_t tl = tbase + ((uint32_t)(32 * Lq) << 16);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v[16];
#pragma unroll
                for (int c = 0; c < 2; ++c) {  // 8 channels per 16-byte chunk of x
                    const int ch = d0 + 16 * h + 8 * c;
                    const uint4 w = *reinterpret_cast<const uint4 *>(sx + swz<2>(r, ch));
                    const io_t *e = reinterpret_cast<const io_t *>(&w);
#pragma unroll
                    for (int q4 = 0; q4 < 2; ++q4) {
                        const float4 gr = *reinterpret_cast<const float4 *>(sg + swz<4>(r, ch + 4 * q4));
                        const float4 gb =
                            *reinterpret_cast<const float4 *>(sg + swz<4>(16 * t, ch + 4 * q4));
                        const int o = 8 * c + 4 * q4;
                        const float2 s2 = make_float2(scale, scale);
                        const float2 d01 = __ffma2_rn(make_float2(gb.x, gb.y), make_float2(-1.f, -1.f), make_float2(gr.x, gr.y));
                        const float2 d23 = __ffma2_rn(make_float2(gb.z, gb.w), make_float2(-1.f, -1.f), make_float2(gr.z, gr.w));
                        const float2 x01 = __fmul2_rn(
                            __fmul2_rn(make_float2(to_f32(e[4 * q4 + 0]), to_f32(e[4 * q4 + 1])), s2),
                            make_float2(ex2(d01.x), ex2(d01.y)));
                        const float2 x23 = __fmul2_rn(
                            __fmul2_rn(make_float2(to_f32(e[4 * q4 + 2]), to_f32(e[4 * q4 + 3])), s2),
                            make_float2(ex2(d23.x), ex2(d23.y)));
                        v[o + 0] = x01.x;
                        v[o + 1] = x01.y;
                        v[o + 2] = x23.x;
                        v[o + 3] = x23.y;
                    }
                }
                tc::tmem_st16(tl + (uint32_t)(d0 + 16 * h), v);
            }
        }
        {
            // B_tt[s, d] = k_s 2^(g_16tt - g_s) for s < 16tt (exponent <= 0): 96 rows of
            // 32 four-channel chunks, six per thread; a warp covers consecutive rows of
            // one chunk, so its loads and stores are bank-conflict free.
#pragma unroll
            for (int j = 0; j < 6; ++j) {
                const int item = tid + FW_THREADS * j;
                const int brow = item % 96, ch = 4 * (item / 96);
                const int tt = brow < 16 ? 1 : brow < 48 ? 2 : 3;
                const int sr = brow - 8 * tt * (tt - 1);  // source row s
                const uint2 w = *reinterpret_cast<const uint2 *>(sk + swz<2>(sr, ch));
                const io_t *kk = reinterpret_cast<const io_t *>(&w);
                const float4 gs = *reinterpret_cast<const float4 *>(sg + swz<4>(sr, ch));
                const float4 gt = *reinterpret_cast<const float4 *>(sg + swz<4>(BC * tt, ch));
                const float2 d01 = __ffma2_rn(make_float2(gs.x, gs.y), make_float2(-1.f, -1.f), make_float2(gt.x, gt.y));
                const float2 d23 = __ffma2_rn(make_float2(gs.z, gs.w), make_float2(-1.f, -1.f), make_float2(gt.z, gt.w));
                const float2 o01 = __fmul2_rn(make_float2(to_f32(kk[0]), to_f32(kk[1])),
                                              make_float2(ex2(d01.x), ex2(d01.y)));
                const float2 o23 = __fmul2_rn(make_float2(to_f32(kk[2]), to_f32(kk[3])),
                                              make_float2(ex2(d23.x), ex2(d23.y)));
                const float4 o = make_float4(o01.x, o01.y, o23.x, o23.y);
                *reinterpret_cast<float4 *>(smem + FM_B + boff(tt) + (ch >> 2) * 256 * tt +
                                            (sr >> 3) * 128 + (sr & 7) * 16) = o;
            }
        }
        // operands complete: every warp arrives on the operands barrier; warps 13, 14
        // and 15 each wait for it and issue one of the three MMA chains, so none of the
        // warps that refilled the stage (0..8, last at this point) issues them.  Thread 0
        // also releases the staging once the previous unit's tiles have left it.
        tc::tmem_wait_st();
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        if (tid == 0) {
            tc::bulk_wait_read_all();
            tc::mbar_arrive(stg_free);
        }
        __syncwarp();
        {
            if (lane == 0) tc::mbar_arrive(stg_free + 1);
            // warps 13, 14, 15 each issue one MMA chain (target block t = warp - 12) once
            // every warp's operands are written
            if (warp >= 13) {
                ok &= tc::mbar_wait(stg_free + 1, (uint32_t)it & 1u, SPIN_LIMIT);
                tc::fence_after_sync();
                if (tc::elect_one()) {
                    const int t = warp - 12;
                    const uint64_t b0 =
                        tc::smem_desc(tc::smem_u32(smem + FM_B + boff(t)), 256 * t, 128);
                    const uint32_t id = tc::idesc_tf32(128, 16 * t);
#pragma unroll
                    for (int kk = 0; kk < KD / 8; ++kk)
                        tc::mma_tf32_ts(tbase + tm_d(t), tbase + 8 * kk,
                                        b0 + (uint64_t)((512 * t * kk) >> 4), id, kk > 0);
                    tc::mma_commit(mbar);
                }
            }
            __syncwarp();
        }

        // ---- diagonal blocks: thread = (block i, rows rb = 16i+15-a and ra = 16i+a,
        // channel group c).  Two 16-slot transposed reductions over the half-warp's 16
        // channel groups: the first holds rb against sources 16i..16i+7 (Aqk, Akk),
        // the second packs rb against 16i+8..rb and ra against 16i..ra into the 16
        // slots exactly (7-a + a+1 Aqk, 7-a + a Akk, and rb's own Aqk diagonal in the
        // one Akk slot left free).  Lane c keeps slot c for the epilogue. ----
        float *dval = reinterpret_cast<float *>(smem + FM_DIAG) + tid;
        {
            const int i = warp >> 2;
            const int a = 2 * (warp & 3) + (lane >> 4);
            const int c = lane & 15;
            const int rb = BC * i + BC - 1 - a, ra = BC * i + a;
            const float2 neg1 = make_float2(-1.f, -1.f);
            // sums over this lane's 8 channels of q_r k_s E and k_r k_s E
            auto src = [&](const float2(&qv)[4], const float2(&kv)[4], const float2(&gv)[4],
                           const int srow, float &oq, float &ok_) {
                float2 ks[4], gs[4];
                ld8_io<io_t>(sk, srow, c, ks);
                ld8_f32(sg, srow, c, gs);
                float2 pq = make_float2(0.f, 0.f), pk = make_float2(0.f, 0.f);
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const float2 df = __ffma2_rn(gs[x], neg1, gv[x]);
                    const float2 tq = __fmul2_rn(ks[x], make_float2(ex2(df.x), ex2(df.y)));
                    pq = __ffma2_rn(qv[x], tq, pq);
                    pk = __ffma2_rn(kv[x], tq, pk);
                }
                oq = pq.x + pq.y;
                ok_ = pk.x + pk.y;
            };
            float v[16];
            {
                float2 qv[4], kv[4], gv[4];
                ld8_io<io_t>(sq, rb, c, qv);
                ld8_io<io_t>(sk, rb, c, kv);
                ld8_f32(sg, rb, c, gv);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if ((j & 1) == 0) asm volatile("" ::: "memory");
                    src(qv, kv, gv, BC * i + j, v[j], v[8 + j]);
                }
                dval[0] = reduce16(v, lane);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    v[j] = v[8 + j] = 0.f;
                    if ((j & 1) == 0) asm volatile("" ::: "memory");
                    if (j <= 7 - a) {
                        float oq, ok_;
                        src(qv, kv, gv, BC * i + 8 + j, oq, ok_);
                        if (j == 7 - a) {
                            v[8 + j] = oq;  // Aqk[rb][rb]
                        } else {
                            v[j] = oq;
                            v[8 + j] = ok_;
                        }
                    }
                }
            }
            {
                float2 qv[4], kv[4], gv[4];
                ld8_io<io_t>(sq, ra, c, qv);
                ld8_io<io_t>(sk, ra, c, kv);
                ld8_f32(sg, ra, c, gv);
#pragma unroll
                for (int sl = 0; sl < 8; ++sl) {
                    if ((sl & 1) == 0) asm volatile("" ::: "memory");
                    if (sl <= a) {
                        float oq, ok_;
                        src(qv, kv, gv, BC * i + sl, oq, ok_);
                        v[7 - sl] = oq;
                        if (sl < a) v[15 - sl] = ok_;
                    }
                }
            }
            dval[512] = reduce16(v, lane);
        }

        // ---- cross blocks: TMEM lane m -> row r of Aqk (m < 64) or Akk (m >= 64),
        // warp (Lq, Dq) takes the 16 source columns 16Dq.. of its lanes' target block ----
        ok &= tc::mbar_wait(mbar, (uint32_t)it & 1u, SPIN_LIMIT);
        tc::fence_after_sync();
        ok &= tc::mbar_wait(stg_free, (uint32_t)it & 1u, SPIN_LIMIT);
        {  // the diagonal entries kept above
            const int i = warp >> 2;
            const int a = 2 * (warp & 3) + (lane >> 4);
            const int c = lane & 15;
            const int rb = BC * i + BC - 1 - a, ra = BC * i + a;
            // first reduction: Aqk[rb][16i + c] (c < 8), Akk[rb][16i + c - 8]
            {
                const float val = c < 8 ? dval[0] : dval[0] * sbeta[rb];
                *reinterpret_cast<float *>(stg + stg_off(c >> 3, rb, BC * i + (c & 7))) =
                    ok ? val : nan;
            }
            // second reduction: the packed slots
            {
                int tensor, r, col;
                float scale = 1.f;
                if (c <= 6 - a) {
                    tensor = 0, r = rb, col = 8 + c;
                } else if (c <= 7) {
                    tensor = 0, r = ra, col = 7 - c;
                } else if (c <= 14 - a) {
                    tensor = 1, r = rb, col = c, scale = sbeta[rb];
                } else if (c == 15 - a) {
                    tensor = 0, r = rb, col = 15 - a;
                } else {
                    tensor = 1, r = ra, col = 15 - c, scale = sbeta[ra];
                }
                *reinterpret_cast<float *>(stg + stg_off(tensor, r, BC * i + col)) =
                    ok ? dval[512] * scale : nan;
            }
        }
        {
            const int Lq = warp & 3, Dq = warp >> 2;
            const int r = 32 * (Lq & 1) + lane, tensor = Lq >> 1;
            const int t_lo = 2 * (Lq & 1), t_hi = t_lo + 1;  // blocks of lanes 0-15, 16-31
            const uint32_t tl = tbase + ((uint32_t)(32 * Lq) << 16);
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                const int t = part ? t_lo : t_hi;
                if (Dq < t) {  // warp-uniform
                    float v[16];
                    tc::tmem_ld16(tl + tm_d(t) + 16 * Dq, v);
                    tc::tmem_wait_ld();
                    if ((lane >> 4) == (part ? 0 : 1)) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            float4 o = make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2],
                                                   v[4 * q4 + 3]);
                            if (!ok) o = make_float4(nan, nan, nan, nan);
                            *reinterpret_cast<float4 *>(stg + stg_off(tensor, r, 16 * Dq + 4 * q4)) = o;
                        }
                    }
                }
            }
        }

        // ---- unit done: tiles out through TMA, stage refilled ----
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (tid == 0 && len == BT) {
            tc::tma_store_3d(&tm.aqk, stg, 0, h, row);
            tc::tma_store_3d(&tm.aqk, stg + 8192, 32, h, row);
            tc::tma_store_3d(&tm.akk, stg + 16384, 0, h, row);
            tc::tma_store_3d(&tm.akk, stg + 24576, 32, h, row);
            tc::bulk_commit_group();
        }
        if (VARLEN && len < BT) {  // a short chunk: its valid rows only, by plain stores
            const int per = len * (BT / 4);
            for (int x = tid; x < 2 * per; x += FW_THREADS) {
                const int tensor = x >= per, rem = x - tensor * per;
                const int r = rem / (BT / 4), c4 = rem % (BT / 4);
                const float4 v = *reinterpret_cast<const float4 *>(stg + stg_off(tensor, r, 4 * c4));
                const size_t di = ((size_t)(row + r) * H + h) * BT + 4 * c4;
                if (dbg_ok(ex.dbg, di + 3, ex.nrows * BT, DBG_STORE))
                    *reinterpret_cast<float4 *>((tensor ? Akk : Aqk) + di) = v;
            }
            __syncthreads();  // the staging is read before the next unit may write it
        }
        if constexpr (VARLEN) {
            if (warp == 0 && ((it + 2) % LUT_BATCH) == 0) lookup_batch(it + 2 + LUT_BATCH);
        }
        if (warp <= 8 && u + 2 * stride < units)
            load_unit_part<io_t, VARLEN>(warp, st,
                                         reinterpret_cast<float *>(smem + FM_BETA) + 64 * sidx,
                                         &full[sidx], meta + 2 * sidx, tm, beta, u + 2 * stride,
                                         T, H, ex, lane,
                                         lut + (((it + 2) / LUT_BATCH) & 1) * 2 * LUT_BATCH +
                                             2 * ((it + 2) % LUT_BATCH));
    }

    dbg_flag(ex.dbg, !ok, DBG_WAIT);
    if (tid == 0) tc::bulk_wait_all();
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tbase, TM_COLS);
    }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
int g_num_sms[kMaxDev];

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

// 3-d map (element, head, token row) with a 64-row box of 128-byte rows, 128B swizzle
cudaError_t encode_rows(CUtensorMap *m, CUtensorMapDataType dt, int esize, const void *base,
                        cuuint64_t width, cuuint64_t heads, cuuint64_t rows) {
    const cuuint64_t dims[3] = {width, heads, rows};
    const cuuint64_t str[2] = {width * esize, heads * width * esize};
    const cuuint32_t box[3] = {(cuuint32_t)(128 / esize), 1, BT};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, dt, 3, const_cast<void *>(base), dims, str, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// What a set of forward tensor maps depends on (a map is a pure function of these):
// the maps of a thread's previous call are reused when the key is the same.
struct FwdKey {
    const void *q, *k, *g, *Aqk, *Akk;
    int B, T, H, HV;
    bool fp16;
    bool operator==(const FwdKey &o) const {
        return q == o.q && k == o.k && g == o.g && Aqk == o.Aqk && Akk == o.Akk && B == o.B &&
               T == o.T && H == o.H && HV == o.HV && fp16 == o.fp16;
    }
};
thread_local FwdKey t_key;
thread_local FwdMaps t_maps;
thread_local bool t_valid = false;

cudaError_t fwd_maps(const FwdArgs &a, int HV, FwdMaps *tm) {
    const FwdKey key = {a.q, a.k, a.g, a.Aqk, a.Akk, a.B, a.T, a.H, HV, a.fp16};
    if (t_valid && key == t_key) {
        *tm = t_maps;
        return cudaSuccess;
    }
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    const cuuint64_t rows = (cuuint64_t)a.B * a.T, HQ = (cuuint64_t)a.H, H = (cuuint64_t)HV;
    const CUtensorMapDataType io =
        a.fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapDataType f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    if ((e = encode_rows(&tm->q, io, 2, a.q, KD, HQ, rows)) != cudaSuccess ||
        (e = encode_rows(&tm->k, io, 2, a.k, KD, HQ, rows)) != cudaSuccess ||
        (e = encode_rows(&tm->g, f32, 4, a.g, KD, H, rows)) != cudaSuccess ||
        (e = encode_rows(&tm->aqk, f32, 4, a.Aqk, BT, H, rows)) != cudaSuccess ||
        (e = encode_rows(&tm->akk, f32, 4, a.Akk, BT, H, rows)) != cudaSuccess)
        return e;
    t_key = key;
    t_maps = *tm;
    t_valid = true;
    return cudaSuccess;
}

template <typename io_t, bool VARLEN>
cudaError_t launch_typed(const FwdArgs &a, cudaStream_t stream) {
    auto kern = kda_intra_fwd_tc_kernel<io_t, VARLEN>;
    static volatile int smem_set[kMaxDev];  // this instantiation's attribute, per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = smem_limit_once(kern, FM_ALLOC, dev, smem_set)) != cudaSuccess) return e;
    int nsm = (dev >= 0 && dev < kMaxDev) ? g_num_sms[dev] : 0;
    if (nsm == 0) {
        if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        if (dev >= 0 && dev < kMaxDev) g_num_sms[dev] = nsm;
    }
    const int HV = a.HV > 0 ? a.HV : a.H;
    FwdMaps tm;
    if ((e = fwd_maps(a, HV, &tm)) != cudaSuccess) return e;
    FwdExtras ex;
    ex.G = HV / a.H;
    ex.cu_seqlens = a.cu_seqlens;
    ex.chunk_indices = a.chunk_indices;
    ex.num_seqs = a.num_seqs;
    ex.dbg = a.dbg;
    ex.nrows = (size_t)a.B * a.T * HV;
    ex.num_chunks = a.num_chunks;
    const long long units =
        VARLEN ? (long long)a.num_chunks * HV : (long long)a.B * HV * (a.T / BT);
    if (units == 0) return cudaSuccess;
    const unsigned grid = (unsigned)(units < nsm ? units : nsm);
    kern<<<grid, FW_THREADS, FM_ALLOC, stream>>>(tm, a.beta, a.Aqk, a.Akk, a.T, HV, units, ex);
    return cudaGetLastError();
}

}  // namespace
}  // namespace fwdimpl

cudaError_t launch_intra_fwd(const FwdArgs &a, cudaStream_t stream) {
    if (a.cu_seqlens)
        return a.fp16 ? fwdimpl::launch_typed<__half, true>(a, stream)
                      : fwdimpl::launch_typed<__nv_bfloat16, true>(a, stream);
    return a.fp16 ? fwdimpl::launch_typed<__half, false>(a, stream)
                  : fwdimpl::launch_typed<__nv_bfloat16, false>(a, stream);
}

}  // namespace kda
