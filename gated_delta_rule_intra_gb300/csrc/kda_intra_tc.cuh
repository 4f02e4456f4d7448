// Tensor-core kernel for the KDA intra-chunk backward (sm_103a, tcgen05 + TMEM + TMA).
//
// Persistent grid, one 512-thread CTA per SM, units (b, h, 64-token chunk) dealt
// round-robin.  Two shared-memory stages hold the inputs of consecutive units; the
// tensor memory accelerator fills a stage while the other one is being computed.
// There is no CTA-wide barrier inside the unit loop: warps hand work to each other
// through mbarriers and a shared counter, so fast warps run ahead into the next unit
// instead of idling:
//   * the stage-full mbarrier completes when a unit's TMA tiles and beta have landed;
//   * every warp arrives on an operands mbarrier once its tensor-core operands are
//     written and goes on to its diagonal block; warps 13, 14 and 15 wait for it and
//     issue the unit's 36 MMAs, 12 each, in parallel;
//   * the last warp to finish a unit (the shared counter) releases its stage and loads
//     the unit after next into it (SPLIT: each sub-block loads its own rows);
//   * the per-row sum for dbeta meets across the four warps of a sub-block at a
//     128-thread named barrier.
//
// Thread (i, d) owns sub-block i (rows 16i..16i+15) at channel d; its TMEM lane is d
// (warp w reaches lanes 32(w%4)..32(w%4)+31, and d = 32(w%4) + lane).
//
// Cross-sub-block terms (bwd_intra page, module docstring): for r in block t and
// s in block j < t,
//     2^(g_r - g_s) = 2^(g_r - g_b0(t)) * 2^(g_b0(t) - g_e(j)) * 2^(g_e(j) - g_s)
// with b0(t) = 16t and e(j) = 16(j+1); every exponent is <= 0.  The last two
// factors are folded into a TF32 operand per target block t,
//     A_t[d, s] = k[s,d] 2^(g_16t - g_s)   (s < 16t),
// kept in TMEM and multiplied on the tensor core by the dA rows of block t:
//     Xq_t[d, n] = sum_s A_t[d, s] dAqk[16t+n, s]   (same for Xk_t with dAkk)
// and the first factor is applied on the TMEM->register path.  The column side
// uses the mirrored split through the source block's end boundary:
//     P_j[d, s] = sum_{r in blk j} q[r,d] 2^(g_r - g_16j) dAqk[r,s]
//               + beta_r k[r,d] 2^(g_r - g_16j) dAkk[r,s]        (s < 16j)
//     dkt_cross[s,d] = 2^(g_e(i) - g_s) * sum_{j>i} 2^(g_16j - g_e(i)) P_j[d, s].
// The 16x16 diagonal blocks run on the FP32 pipes, two source rows at a time in
// packed FP32x2 arithmetic, with one exp2 per (r, s, d).  Optionally (FACTOR) their
// lower-left 8x8 quadrant (rows 8..15 against sources 0..7) is factorized through
// row 8 of the block,
//     2^(g_r - g_s) = 2^(g_r - g_8) * 2^(g_8 - g_s),  both exponents <= 0,
// so it costs four FMAs per (r, s, d); the two 8x8 triangles keep one exp2 per
// (r, s, d).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "kda_common.cuh"
#include "kda_launch.h"
#include "tc_ptx.cuh"

namespace kda {
namespace tcimpl {

constexpr int TC_THREADS = 512;
constexpr int TC_WARPS = TC_THREADS / 32;
constexpr int MMA_WARPS = 3;  // warps 13..15 issue the MMAs

// ---- shared memory: two input stages + single-buffered derived operands ----
// dA tiles: the ten lower 16x16 blocks (t, j <= t) of a unit, block (t, j) at
// dablk(t, j) KB, each in the K-major core-matrix layout of a tensor-core operand:
// element (n, k) (n = row in block t, k = column in block j) at byte
//     (k/4)*256 + (n/8)*128 + (n%8)*16 + (k%4)*4.
// Blocks (t, 0..t-1) are contiguous, so they form the B operand of target t
// (N = 16 rows, K = 16t, core matrices 256 B apart along K and 128 B along N).
constexpr int ST_Q = 0;                      // io_t [64][128]
constexpr int ST_K = ST_Q + BT * KD * 2;     // io_t [64][128]
constexpr int ST_G = ST_K + BT * KD * 2;     // f32  [64][128]
constexpr int ST_DQ = ST_G + BT * KD * 4;    // dAqk: 10 blocks x 1 KB
constexpr int ST_DK = ST_DQ + 10 * 1024;     // dAkk
constexpr int ST_BETA = ST_DK + 10 * 1024;   // f32 [64]
constexpr int STAGE_BYTES = ST_BETA + 256;   // 86272
constexpr int SM_BCQ = 2 * STAGE_BYTES;      // dAqk blocks of target j transposed (K-major)
constexpr int SM_BCK = SM_BCQ + 6144;
constexpr int SM_DBP = SM_BCK + 6144;        // db partials f32 [4][64]
constexpr int SM_FULL = SM_DBP + 1024;       // 2 stage-full mbarriers
constexpr int SM_MMA = SM_FULL + 16;         // MMAs-done mbarrier, operands-written mbarrier
constexpr int SM_CNT = SM_MMA + 16;          // (unused), unit-done counter
constexpr int SM_TSLOT = SM_CNT + 8;
constexpr int SM_META = SM_TSLOT + 8;        // varlen: per stage {first token row, valid rows}
constexpr int SM_LUT = SM_META + 16;         // varlen: {first row, valid rows} of this
                                             // CTA's units, two batches of 32
constexpr int LUT_BATCH = 32;
constexpr int SM_TRTAB = SM_LUT + 2 * LUT_BATCH * 8;  // per-thread transpose indices
                                                      // (option instantiations)
constexpr int SM_TOTAL = SM_TRTAB + 3 * TC_THREADS * 4;
// extra shared memory of the split-TF32 variant: the low parts of the dA operands, as
// tensor-core operands in the layouts of their high parts -- the six off-diagonal blocks
// of each tensor (row-block t's blocks (t, 0..t-1) at block t(t-1)/2 + j, so each target's
// run is contiguous), then the transposed column-side blocks -- and the barrier and
// counter of the second MMA pass.
constexpr int SM_SPLIT_Q = (SM_TOTAL + 1023) / 1024 * 1024;
constexpr int SM_SPLIT_K = SM_SPLIT_Q + 6144;
constexpr int SM_SPLIT_CQ = SM_SPLIT_K + 6144;
constexpr int SM_SPLIT_CK = SM_SPLIT_CQ + 6144;
constexpr int SM_SPLIT_BAR = SM_SPLIT_CK + 6144;  // pass-2 MMAs-done and operands mbarriers
constexpr int SM_TOTAL_SPLIT = SM_SPLIT_BAR + 16;
// extra shared memory of the fold_dg variant: the per-row dg bank [64][128] and the
// per-(sub-block, channel) totals, double-buffered by unit parity
constexpr int SM_FOLD_BANK = (SM_TOTAL + 127) / 128 * 128;
constexpr int SM_FOLD_TOT = SM_FOLD_BANK + BT * KD * 4;
constexpr int SM_TOTAL_FOLD = SM_FOLD_TOT + 2 * NBLK * KD * 4;
static_assert(STAGE_BYTES % 128 == 0, "TMA destinations need 128-byte alignment");
static_assert(SM_TOTAL_SPLIT <= 232448 && SM_TOTAL_FOLD <= 232448, "shared memory per CTA");
static_assert(ST_DQ % 1024 == 0 && ST_DK % 1024 == 0, "dA tiles alignment");

constexpr uint32_t STAGE_TX_BYTES = 2 * BT * KD * 2 + BT * KD * 4 + 2 * 10 * 1024;
constexpr uint32_t FULL_ARRIVALS = 1 + 32;  // expect_tx by lane 0 + beta copies by 32 lanes
constexpr uint32_t SLICE_TX_BYTES = 2 * BC * KD * 2 + BC * KD * 4;  // q, k, g rows of a sub-block
constexpr uint32_t FULL_ARRIVALS_SLICED = NBLK * (1 + 32);

__host__ __device__ constexpr int dablk(int t, int j) { return t * (t + 1) / 2 + j; }

// byte offset of target j's transposed operand inside a 6 KB region: 1, 2, 3 KB
__device__ __forceinline__ uint32_t bcol_off(int j) { return 512u * (uint32_t)((j - 1) * j); }

// ---- TMEM column map (512 columns, fp32) ----
__device__ __forceinline__ uint32_t tm_arow(int t) { return 8u * (uint32_t)(t * (t - 1)); }  // A_t: 16t cols
constexpr uint32_t TM_AQB = 96;    // q_r 2^(g_r - g_16j), column r-16  (48 cols)
constexpr uint32_t TM_AKBB = 144;  // beta_r k_r 2^(g_r - g_16j)          (48 cols)
constexpr uint32_t TM_XQ = 192;    // Xq_t at +16(t-1)                     (48 cols)
constexpr uint32_t TM_XK = 240;    // Xk_t                                   (48 cols)
__device__ __forceinline__ uint32_t tm_p(int j) { return 288u + 8u * (uint32_t)(j * (j - 1)); }
constexpr uint32_t TM_FB = 384;    // 2^(g_r - g_16i) for block i >= 1 at +16(i-1)
constexpr uint32_t TM_FA = 432;    // 2^(g_16(i+1) - g_s) for block i <= 2 at +16i
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t SPIN_LIMIT = 1u << 22;

// q, k, g: one unit's [64 x 128] tile.  daqk[t], dakk[t]: row-block t's lower blocks
// (t, 0..t) in one box of 16 rows x 16(t+1) columns, landing in the operand layout.
struct TmaMaps {
    CUtensorMap q, k, g, daqk[NBLK], dakk[NBLK];
    CUtensorMap q16, k16, g16;  // 16-row boxes: one sub-block's rows (fixed length)
};

// Options of the extended entry point.  H in the kernel is the number of heads of g,
// beta, dA and the outputs (HV); q and k have HV / G heads.
struct Extras {
    const float *dq_in, *dk_in, *dg_in, *db_in;  // added in-kernel when non-null
    int G;  // value heads per q/k head
    // variable-length launches: sequence n is tokens [cu_seqlens[n], cu_seqlens[n+1])
    // of the packed T axis; unit u is head u % H of chunk chunk_indices[2c+1] of
    // sequence chunk_indices[2c], c = u / H
    const int *cu_seqlens, *chunk_indices;
    int num_seqs;
    // bounds-checked debug build: the flag word and the extents checked against
    unsigned *dbg;
    size_t nrows;    // token rows x heads of g, beta, dA and the outputs
    int num_chunks;  // entries of chunk_indices (variable-length launches)
};

// Where a variable-length unit lives: first token row, valid rows (1..64; 0 for an
// entry of chunk_indices that names no chunk of cu_seqlens, which is then skipped)
// and head.
struct VarUnit {
    int start, len, h;
};

__device__ __forceinline__ VarUnit varlen_unit(long long u, int H, int T, const Extras ex) {
    const unsigned uu = (unsigned)u, c = uu / (unsigned)H;
    VarUnit x;
    x.h = (int)(uu - c * (unsigned)H);
    x.start = 0;
    x.len = 0;
    if (!dbg_ok(ex.dbg, 2 * (size_t)c + 1, 2 * (size_t)ex.num_chunks, DBG_LOAD)) return x;
    const int n = __ldg(ex.chunk_indices + 2 * (size_t)c);
    const int ci = __ldg(ex.chunk_indices + 2 * (size_t)c + 1);
    if (n >= 0 && n < ex.num_seqs && ci >= 0) {
        const long long bos = __ldg(ex.cu_seqlens + n), eos = __ldg(ex.cu_seqlens + n + 1);
        const long long st = bos + (long long)BT * ci;
        if (bos >= 0 && st < eos && eos <= T) {
            x.start = (int)st;
            x.len = (int)(eos - st < BT ? eos - st : BT);
        }
    }
    return x;
}

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}
template <> __device__ __forceinline__ __half from_f32<__half>(float x) {
    return __float2half_rn(x);
}

__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(gmem) : "memory");
}
// Same, or four zero bytes (nothing read) when !take.
__device__ __forceinline__ void cp_async4_zfill(void *smem, const void *gmem, bool take) {
    uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(s), "l"(gmem),
                 "r"(take ? 4 : 0)
                 : "memory");
}

// x rounded to TF32 (10 explicit mantissa bits, round to nearest, ties away), as FP32.
__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t y;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(y) : "f"(x));
    return __uint_as_float(y);
}

// 16 TMEM columns of a TF32 operand: the values themselves, or (SPLIT) their high
// (LO = false) or low (LO = true) parts.
template <bool SPLIT, bool LO>
__device__ __forceinline__ void tmem_st_part(uint32_t taddr, const float (&v)[16]) {
    if constexpr (SPLIT) {
        float w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = LO ? v[e] - tf32_rna(v[e]) : tf32_rna(v[e]);
        tc::tmem_st16(taddr, w);
    } else {
        tc::tmem_st16(taddr, v);
    }
}

// *p += v in L2 (round to nearest; subnormal inputs and results flush to zero).
__device__ __forceinline__ void red_add(float *p, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// One warp queues every copy of one unit into a stage: 11 TMA tiles from lane 0,
// beta as 64 four-byte copies from all lanes (its rows are H floats apart, so no
// tensor map can describe it when H is not a multiple of 4).  A variable-length unit
// may start at any token row: its dA tiles come through the 4-d map (any row start),
// rows past the sequence's end are loaded as they are (or zero-filled past the
// tensor's end) and masked by the consumer, and their beta is zero-filled.  Its row
// range comes from `known` ({first row, valid rows}, read by lane 0 and broadcast)
// when given, else from the chunk table.  Lane 0 records it in `meta` before its
// arrival on the stage barrier, which publishes it with the data.
template <bool VARLEN>
__device__ __forceinline__ void load_unit(unsigned char *st, uint64_t *full, int *meta,
                                          const TmaMaps &tm, const float *__restrict__ beta,
                                          long long u, int T, int H, const Extras ex,
                                          int lane, const int *known = nullptr) {
    int row, h, len = BT;  // first token row of the unit, head, valid rows
    if constexpr (VARLEN) {
        if (known) {
            int a = 0, b = 0;
            if (lane == 0) {
                a = known[0];
                b = known[1];
            }
            row = __shfl_sync(0xffffffffu, a, 0);
            len = __shfl_sync(0xffffffffu, b, 0);
            h = (int)((unsigned)u % (unsigned)H);
        } else {
            const VarUnit x = varlen_unit(u, H, T, ex);
            row = x.start;
            len = x.len;
            h = x.h;
        }
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
        tc::mbar_arrive_expect_tx(full, STAGE_TX_BYTES);
        tc::tma_load_3d(st + ST_Q, &tm.q, 0, h / ex.G, row, full);
        tc::tma_load_3d(st + ST_K, &tm.k, 0, h / ex.G, row, full);
        tc::tma_load_3d(st + ST_G, &tm.g, 0, h, row, full);
        // row-block t's blocks (t, 0..t) are contiguous in the stage: one box each
#pragma unroll
        for (int t = 0; t < NBLK; ++t) {
            if constexpr (VARLEN) {
                tc::tma_load_4d(st + ST_DQ + dablk(t, 0) * 1024, &tm.daqk[t], 0, row + BC * t, 0,
                                h, full);
                tc::tma_load_4d(st + ST_DK + dablk(t, 0) * 1024, &tm.dakk[t], 0, row + BC * t, 0,
                                h, full);
            } else {
                const int rg = (row + BC * t) >> 3;
                tc::tma_load_5d(st + ST_DQ + dablk(t, 0) * 1024, &tm.daqk[t], 0, 0, rg, 0, h, full);
                tc::tma_load_5d(st + ST_DK + dablk(t, 0) * 1024, &tm.dakk[t], 0, 0, rg, 0, h, full);
            }
        }
    }
    const float *b0 = beta + (size_t)row * H + h;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int r = lane + 32 * e;
        const size_t bi = (size_t)(row + r) * H + h;
        if constexpr (VARLEN) {
            const bool take = r < len && dbg_ok(ex.dbg, bi, ex.nrows, DBG_LOAD);
            cp_async4_zfill(st + ST_BETA + r * 4, take ? b0 + (size_t)r * H : beta, take);
        } else {
            if (dbg_ok(ex.dbg, bi, ex.nrows, DBG_LOAD))
                cp_async4(st + ST_BETA + r * 4, b0 + (size_t)r * H);
            else
                cp_async4_zfill(st + ST_BETA + r * 4, beta, false);
        }
    }
    tc::cp_async_mbar_arrive_noinc(full);
}

// Fixed-length units, one sub-block's share of the copies into a stage: rows
// 16i..16i+15 of q, k and g and row-block i's dA blocks (five TMA tiles from lane 0),
// and those rows' beta (16 four-byte copies).  Per sub-block the stage barrier counts
// one arrival carrying the share's bytes and 32 copy arrivals.
__device__ __forceinline__ void load_slice(unsigned char *st, uint64_t *full, const TmaMaps &tm,
                                           const float *__restrict__ beta, long long u, int H,
                                           const Extras ex, int lane, int i) {
    const unsigned qq = (unsigned)u / (unsigned)H;
    const int h = (int)((unsigned)u - qq * (unsigned)H);
    const int row = BT * (int)qq + BC * i;  // first token row of the share
    if (lane == 0) {
        tc::mbar_arrive_expect_tx(full, SLICE_TX_BYTES + 2048u * (uint32_t)(i + 1));
        tc::tma_load_3d(st + ST_Q + i * BC * KD * 2, &tm.q16, 0, h / ex.G, row, full);
        tc::tma_load_3d(st + ST_K + i * BC * KD * 2, &tm.k16, 0, h / ex.G, row, full);
        tc::tma_load_3d(st + ST_G + i * BC * KD * 4, &tm.g16, 0, h, row, full);
        tc::tma_load_5d(st + ST_DQ + dablk(i, 0) * 1024, &tm.daqk[i], 0, 0, row >> 3, 0, h, full);
        tc::tma_load_5d(st + ST_DK + dablk(i, 0) * 1024, &tm.dakk[i], 0, 0, row >> 3, 0, h, full);
    }
    if (lane < BC) {
        const size_t bi = (size_t)(row + lane) * H + h;
        unsigned char *dst = st + ST_BETA + (BC * i + lane) * 4;
        if (dbg_ok(ex.dbg, bi, ex.nrows, DBG_LOAD))
            cp_async4(dst, beta + bi);
        else
            cp_async4_zfill(dst, beta, false);
    }
    tc::cp_async_mbar_arrive_noinc(full);
}

// ACCUM: add the optional incoming gradients of Extras (1: loaded and added; 2: dq_in,
// dk_in and, without FOLD, dg_in are the outputs themselves, and the stores add to them
// in L2 with red.global.add instead: nothing to load); FOLD: return dg as its
// inclusive reverse cumsum inside each chunk; EMIT: store dq and dk as io_t;
// FACTOR: the diagonal blocks' lower-left quadrant through row 8 (see above);
// VARLEN: units come from cu_seqlens / chunk_indices, and a unit's rows past its
// sequence's end (row >= len, "foreign" rows) are masked: their q, k, beta and
// diagonal-block dA rows read as 0, their gate as the last valid row's (so every
// exponent stays <= 0), their off-diagonal dA rows are zeroed in the column-side
// operands, and nothing is stored for them.
// SPLIT: the cross-sub-block sums in split TF32 for FP32-level accuracy.  Every operand
// x is cut into hi = tf32(x) (round to nearest) and lo = x - hi (exact in FP32); the
// tensor core accumulates A_hi B_hi + A_hi B_lo (pass 1) and A_lo B_hi (pass 2, after
// A_lo replaces A_hi in TMEM), leaving out A_lo B_lo (about 2^-22 of the product).
template <typename io_t, int ACCUM, bool FOLD, bool EMIT, bool VARLEN, bool FACTOR,
          bool SPLIT = false>
__global__ void __launch_bounds__(TC_THREADS, 1)
kda_intra_bwd_tc_kernel(const __grid_constant__ TmaMaps tm, const float *__restrict__ beta,
                        void *dq_out, void *dk_out, float *db, float *dg, int T, int H,
                        long long units, const Extras ex) {
    float *dq = reinterpret_cast<float *>(dq_out);
    float *dk = reinterpret_cast<float *>(dk_out);
    extern __shared__ __align__(1024) unsigned char smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int i = tid >> 7;  // sub-block, warp-uniform
    const int d = tid & 127;
    const int r0 = i * BC;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + SM_FULL);
    uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + SM_MMA);
    uint32_t *done_count = reinterpret_cast<uint32_t *>(smem + SM_CNT) + 1;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + SM_TSLOT);
    float *sdbp = reinterpret_cast<float *>(smem + SM_DBP);
    const long long stride = gridDim.x;

    uint64_t *mbar2 = reinterpret_cast<uint64_t *>(smem + SM_SPLIT_BAR);  // SPLIT only
    if (warp == 0) tc::tmem_alloc(tslot, TM_COLS);
    // SPLIT: each sub-block refills its own rows of a stage as soon as its four warps
    // are done with them (measured faster there; slower on the other paths)
    constexpr bool SLICED = SPLIT && !VARLEN;
    if (tid == 0) {
        tc::mbar_init(&full[0], SLICED ? FULL_ARRIVALS_SLICED : FULL_ARRIVALS);
        tc::mbar_init(&full[1], SLICED ? FULL_ARRIVALS_SLICED : FULL_ARRIVALS);
        tc::mbar_init(mbar, MMA_WARPS);        // one commit per issuing warp
        tc::mbar_init(mbar + 1, TC_WARPS);     // operands written, one arrival per warp
        if constexpr (SPLIT) {
            tc::mbar_init(mbar2, MMA_WARPS);
            tc::mbar_init(mbar2 + 1, TC_WARPS);
        }
        done_count[0] = 0u;
        tc::prefetch_tmap(&tm.q);
        tc::prefetch_tmap(&tm.k);
        tc::prefetch_tmap(&tm.g);
        if constexpr (SLICED) {
            tc::prefetch_tmap(&tm.q16);
            tc::prefetch_tmap(&tm.k16);
            tc::prefetch_tmap(&tm.g16);
        }
#pragma unroll
        for (int t = 0; t < NBLK; ++t) {
            tc::prefetch_tmap(&tm.daqk[t]);
            tc::prefetch_tmap(&tm.dakk[t]);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tslot;
    const uint32_t tlane = tbase + ((uint32_t)(32 * (warp & 3)) << 16);

    int *meta = reinterpret_cast<int *>(smem + SM_META);
    int *lut = reinterpret_cast<int *>(smem + SM_LUT);
    // The column-side transposes move the same three elements for this thread in every
    // unit: element x's (source float, destination float, in-chunk row).  The option
    // instantiations, whose registers are fuller, pack them once into a table read each
    // unit; the plain ones and those with both incoming gradients and the fold recompute
    // them (measured faster each way).
    constexpr bool TRTAB = (ACCUM || FOLD || VARLEN) && !(ACCUM && FOLD);
    uint32_t *trtab = reinterpret_cast<uint32_t *>(smem + SM_TRTAB);
    auto tr_index = [&](const int x, int &src, int &dst, int &row) {
        const int idx = tid + x * TC_THREADS;  // < 1536
        const int j = idx >= 768 ? 3 : idx >= 256 ? 2 : 1;
        const int e = idx - 128 * j * (j - 1);
        // e enumerates the destination floats in order (n/8, k/4, n%8, k%4)
        const int n = (e >> 7) * 8 + ((e >> 2) & 7);  // s
        const int kk = ((e >> 5) & 3) * 4 + (e & 3);  // r - 16j
        src = dablk(j, n >> 4) * 256 + ((n & 15) >> 2) * 64 + (kk >> 3) * 32 + (kk & 7) * 4 +
              (n & 3);
        dst = (int)bcol_off(j) / 4 + e;
        row = BC * j + kk;
    };
    if constexpr (TRTAB) {
#pragma unroll
        for (int x = 0; x < 3; ++x) {
            int src, dst, row;
            tr_index(x, src, dst, row);  // src < 2304, dst < 1536, row < 64
            trtab[x * TC_THREADS + tid] =
                ((uint32_t)src << 17) | ((uint32_t)dst << 6) | (uint32_t)row;
        }
    }
    // VARLEN: lane j of warp 0 looks up the row range of this CTA's unit k0 + j (two
    // dependent table reads), for the refills of a whole batch of units at once
    auto lookup_batch = [&](const int k0) {
        const long long uk = blockIdx.x + (long long)(k0 + lane) * stride;
        if (uk < units) {
            const VarUnit x = varlen_unit(uk, H, T, ex);
            int *e = lut + ((k0 / LUT_BATCH) & 1) * 2 * LUT_BATCH + 2 * lane;
            e[0] = x.start;
            e[1] = x.len;
        }
    };
    if (SLICED && warp == 0) {  // the first two units of this CTA
        for (int s = 0; s < 2; ++s) {
            const long long us = blockIdx.x + s * stride;
            if (us < units)
                for (int j = 0; j < NBLK; ++j)
                    load_slice(smem + s * STAGE_BYTES, &full[s], tm, beta, us, H, ex, lane, j);
        }
    } else if (warp == 0) {  // the first two units of this CTA
        const long long u0 = blockIdx.x;
        if (u0 < units) load_unit<VARLEN>(smem, &full[0], meta, tm, beta, u0, T, H, ex, lane);
        if (u0 + stride < units)
            load_unit<VARLEN>(smem + STAGE_BYTES, &full[1], meta + 2, tm, beta, u0 + stride, T,
                              H, ex, lane);
        if constexpr (VARLEN) lookup_batch(0);
    }

    bool ok = true;
    int it = 0;
    // Head of the current unit, advanced by stride mod H each iteration.  With u = q H + h
    // the unit's first [token * H + head] row is 64 u - 63 h, so no unit needs a division.
    // (The instantiations that load incoming gradients keep the decode: their registers are
    // fuller.  Measured each way.)
    constexpr bool DECODE = ACCUM == 1 || (ACCUM == 2 && FOLD);
    const unsigned dhh = (unsigned)stride % (unsigned)H;
    unsigned hh = (unsigned)blockIdx.x % (unsigned)H;
    auto unit_row = [&](const long long u, const int r) -> size_t {  // fixed-length: row r
        if constexpr (DECODE) return grow(decode_unit(u, H, T / BT), r, T, H);
        else return (size_t)64 * (size_t)u - (size_t)63 * hh + (size_t)r * H;
    };
    auto unit_head = [&](const long long u) -> unsigned {
        if constexpr (DECODE) return (unsigned)u % (unsigned)H;
        else return hh;
    };
    for (long long u = blockIdx.x; u < units;
         u += stride, ++it, hh = hh + dhh >= (unsigned)H ? hh + dhh - (unsigned)H : hh + dhh) {
        const int sidx = it & 1;
        unsigned char *st = smem + sidx * STAGE_BYTES;
        ok &= tc::mbar_wait(&full[sidx], (uint32_t)(it >> 1) & 1u, SPIN_LIMIT);

        const float *sg = reinterpret_cast<const float *>(st + ST_G);
        const io_t *sq = reinterpret_cast<const io_t *>(st + ST_Q);
        const io_t *sk = reinterpret_cast<const io_t *>(st + ST_K);
        const float *sbeta = reinterpret_cast<const float *>(st + ST_BETA);
        // valid rows of this unit and the last of them (rows past it take its gate)
        int ulen = BT;
        if constexpr (VARLEN) ulen = meta[2 * sidx + 1];
        const bool partial = VARLEN && ulen < BT;
        // rows past the end take the last valid row's gate
        const float glastv = partial ? sg[(ulen > 0 ? ulen - 1 : 0) * KD + d] : 0.f;
        auto gsel = [&](const int r, const float v) { return (partial && r >= ulen) ? glastv : v; };

        // VARLEN, chunk shorter than 64 rows: each sub-block group zeroes its foreign
        // rows (row >= len) of q and of its diagonal dA blocks, the only stage data its
        // rows read without a register-side mask, so the diagonal and epilogue rows run
        // unguarded and foreign rows contribute exact zeros.  k, beta and g are masked
        // in registers / at load (below).
        if (partial) {
            {
                const int f = (d & 63) * 4;  // float4 of the diagonal block, row n
                const int n = ((f >> 5) & 1) * 8 + ((f >> 2) & 7);
                float *blk = reinterpret_cast<float *>(st + ((d >> 6) ? ST_DK : ST_DQ)) +
                             dablk(i, i) * 256 + f;
                if (r0 + n >= ulen) *reinterpret_cast<float4 *>(blk) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            {
                const int n = d >> 3;  // row n of the block, 32-byte part d & 7
                if (r0 + n >= ulen) {
                    uint4 *p = reinterpret_cast<uint4 *>(st + ST_Q + (r0 + n) * KD * 2 + (d & 7) * 32);
                    p[0] = make_uint4(0u, 0u, 0u, 0u);
                    p[1] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            tc::fence_proxy_async_smem();  // generic writes into a stage TMA refills later
            tc::named_bar_sync(9 + i, 128);
        }

        // ACCUM: the unit's incoming-gradient rows (3 tensors x 64 rows of 512 bytes) are
        // requested into L2 now; the epilogue reads them a few microseconds later
        if constexpr (ACCUM) {
            if (tid < 3 * BT) {
                const int tsel = tid / BT, r = tid % BT;
                const float *src = tsel == 0 ? ex.dq_in : tsel == 1 ? ex.dk_in : ex.dg_in;
                size_t grow0;
                if constexpr (VARLEN) {
                    grow0 = (size_t)meta[2 * sidx] * H + unit_head(u);
                } else {
                    grow0 = unit_row(u, 0);
                }
                const size_t gi = (grow0 + (size_t)r * H) * KD;
                if (src && r < ulen && dbg_ok(ex.dbg, gi + KD - 1, ex.nrows * KD, DBG_LOAD))
                    tc::prefetch_l2(src + gi, KD * 4);
            }
        }

        // VARLEN: once every 32 units, warp 0 looks up the next batch; the refills read
        // the batch table (published by warp 0's unit-done arrivals)
        if constexpr (VARLEN) {
            if (warp == 0 && (it % LUT_BATCH) == 0) lookup_batch(it + LUT_BATCH);
        }

        // ---- column-side B operands: dA blocks (j, 0..j-1) transposed.  The loads go
        // out first so their latency overlaps the column loads and the prescale. ----
        float trq[3], trk[3];
        int trdst[3];
        {
            const float *aq = reinterpret_cast<const float *>(st + ST_DQ);
            const float *ak = reinterpret_cast<const float *>(st + ST_DK);
#pragma unroll
            for (int x = 0; x < 3; ++x) {
                int src, row;
                if constexpr (TRTAB) {
                    const uint32_t w = trtab[x * TC_THREADS + tid];
                    src = (int)(w >> 17);
                    trdst[x] = (int)((w >> 6) & 2047u);
                    row = (int)(w & 63u);
                } else {
                    tr_index(x, src, trdst[x], row);
                }
                trq[x] = aq[src];
                trk[x] = ak[src];
                if (VARLEN && row >= ulen) trq[x] = trk[x] = 0.f;
            }
        }

        // this thread's column of its block, as (even row, odd row) pairs
        float2 g2[BC / 2], k2[BC / 2];
#pragma unroll
        for (int m = 0; m < BC / 2; ++m) {
            const int ra = r0 + 2 * m, rb = ra + 1;
            g2[m] = make_float2(sg[ra * KD + d], sg[rb * KD + d]);
            k2[m] = make_float2(to_f32(sk[ra * KD + d]), to_f32(sk[rb * KD + d]));
        }
        if (partial) {
#pragma unroll
            for (int m = 0; m < BC / 2; ++m) {
                const int ra = r0 + 2 * m, rb = ra + 1;
                if (ra >= ulen) g2[m].x = glastv, k2[m].x = 0.f;
                if (rb >= ulen) g2[m].y = glastv, k2[m].y = 0.f;
            }
        }
#define KDA_EL(arr, r) (((r) & 1) ? arr[(r) >> 1].y : arr[(r) >> 1].x)

        // ---- prescaled TF32 operands and post-factors into TMEM ----
        float c2 = 0.f, c3 = 0.f;  // 2^(g_16(i+2) - g_e(i)), 2^(g_16(i+3) - g_e(i))
        if (i < NBLK - 1) {
            const float ge = gsel(r0 + BC, sg[(r0 + BC) * KD + d]);
            const float2 ge2 = make_float2(ge, ge), m1 = make_float2(-1.f, -1.f);
            float a[BC], v[BC];
#pragma unroll
            for (int m = 0; m < BC / 2; ++m) {
                const float2 df = __ffma2_rn(g2[m], m1, ge2);
                a[2 * m] = ex2(df.x);
                a[2 * m + 1] = ex2(df.y);
                const float2 vv = __fmul2_rn(k2[m], make_float2(a[2 * m], a[2 * m + 1]));
                v[2 * m] = vv.x;
                v[2 * m + 1] = vv.y;
            }
            tc::tmem_st16(tlane + TM_FA + 16 * i, a);
            tmem_st_part<SPLIT, false>(tlane + tm_arow(i + 1) + 16 * i, v);
            if (i + 2 < NBLK) {
                c2 = ex2(gsel(r0 + 2 * BC, sg[(r0 + 2 * BC) * KD + d]) - ge);
#pragma unroll
                for (int m = 0; m < BC / 2; ++m) {
                    const float2 t = __fmul2_rn(make_float2(v[2 * m], v[2 * m + 1]), make_float2(c2, c2));
                    a[2 * m] = t.x;
                    a[2 * m + 1] = t.y;
                }
                tmem_st_part<SPLIT, false>(tlane + tm_arow(i + 2) + 16 * i, a);
            }
            if (i + 3 < NBLK) {
                c3 = ex2(gsel(r0 + 3 * BC, sg[(r0 + 3 * BC) * KD + d]) - ge);
#pragma unroll
                for (int m = 0; m < BC / 2; ++m) {
                    const float2 t = __fmul2_rn(make_float2(v[2 * m], v[2 * m + 1]), make_float2(c3, c3));
                    a[2 * m] = t.x;
                    a[2 * m + 1] = t.y;
                }
                tmem_st_part<SPLIT, false>(tlane + tm_arow(i + 3) + 16 * i, a);
            }
        }
        if (i > 0) {
            float b[BC], v[BC];
            const float2 g0 = make_float2(-g2[0].x, -g2[0].x), p1 = make_float2(1.f, 1.f);
#pragma unroll
            for (int m = 0; m < BC / 2; ++m) {
                const float2 df = __ffma2_rn(g2[m], p1, g0);
                b[2 * m] = m == 0 ? 1.f : ex2(df.x);
                b[2 * m + 1] = ex2(df.y);
            }
            tc::tmem_st16(tlane + TM_FB + 16 * (i - 1), b);
#pragma unroll
            for (int m = 0; m < BC / 2; ++m) {
                const float2 t = __fmul2_rn(make_float2(to_f32(sq[(r0 + 2 * m) * KD + d]),
                                                        to_f32(sq[(r0 + 2 * m + 1) * KD + d])),
                                            make_float2(b[2 * m], b[2 * m + 1]));
                v[2 * m] = t.x;
                v[2 * m + 1] = t.y;
            }
            tmem_st_part<SPLIT, false>(tlane + TM_AQB + 16 * (i - 1), v);
#pragma unroll
            for (int m = 0; m < BC / 2; ++m) {
                const float2 bk = __fmul2_rn(*reinterpret_cast<const float2 *>(sbeta + r0 + 2 * m), k2[m]);
                const float2 t = __fmul2_rn(bk, make_float2(b[2 * m], b[2 * m + 1]));
                v[2 * m] = t.x;
                v[2 * m + 1] = t.y;
            }
            tmem_st_part<SPLIT, false>(tlane + TM_AKBB + 16 * (i - 1), v);
        }

        {
            float *cq = reinterpret_cast<float *>(smem + SM_BCQ);
            float *ck = reinterpret_cast<float *>(smem + SM_BCK);
            if constexpr (SPLIT) {
                // this thread is the only one that reads or writes its three elements of
                // each tensor's off-diagonal blocks: the high parts replace them in the
                // stage (row-side B operands) and go transposed to the column-side
                // operands; the low parts go to the same places of the low-part copies
                float *aq = reinterpret_cast<float *>(st + ST_DQ);
                float *ak = reinterpret_cast<float *>(st + ST_DK);
                float *ql = reinterpret_cast<float *>(smem + SM_SPLIT_Q);
                float *kl = reinterpret_cast<float *>(smem + SM_SPLIT_K);
                float *cql = reinterpret_cast<float *>(smem + SM_SPLIT_CQ);
                float *ckl = reinterpret_cast<float *>(smem + SM_SPLIT_CK);
#pragma unroll
                for (int x = 0; x < 3; ++x) {
                    int src, dst, row;
                    tr_index(x, src, dst, row);
                    const int blk = src >> 8;  // dablk(t, j), j < t
                    const int t = blk >= 6 ? 3 : blk >= 3 ? 2 : 1;
                    const int lsrc = ((t * (t - 1) / 2) + (blk - t * (t + 1) / 2)) * 256 + (src & 255);
                    const float hq = tf32_rna(trq[x]), hk = tf32_rna(trk[x]);
                    const float lq = trq[x] - hq, lk = trk[x] - hk;
                    cq[dst] = hq;
                    ck[dst] = hk;
                    cql[dst] = lq;
                    ckl[dst] = lk;
                    aq[src] = hq;
                    ak[src] = hk;
                    ql[lsrc] = lq;
                    kl[lsrc] = lk;
                }
            } else {
#pragma unroll
                for (int x = 0; x < 3; ++x) {
                    cq[trdst[x]] = trq[x];
                    ck[trdst[x]] = trk[x];
                }
            }
        }

        // operands complete: TMEM stores landed, smem stores visible to the tensor core.
        // Every warp arrives on the operands barrier and goes on to its diagonal block;
        // warps 13, 14 and 15 (sub-block 3, the lightest prescale) wait for it and issue
        // the MMAs, each a third of the accumulator chains.  No warp issues on its way
        // from its own operands to its diagonal, and the three issue in parallel.
        tc::tmem_wait_st();
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncwarp();
        uint32_t prev = 0;
        if (lane == 0) tc::mbar_arrive(mbar + 1);
        // The unit's MMAs of one pass, the chains of warp w (each accumulator chain stays
        // on one thread: Xq_t, Xk_t over K = 16t, P_j over the q and beta*k sides):
        //   w = 13: Xq_3, Xk_3;  w = 14: Xq_2, Xk_2, P_1;  w = 15: Xq_1, Xk_1, P_2, P_3
        // (12 MMAs each).  pass 1: A (SPLIT: A_hi) times the dA blocks (SPLIT: then times
        // their low parts); pass 2 (SPLIT): A_lo times the dA blocks.
        auto issue_chains = [&](const int pass) {
            const uint64_t dq0 = tc::smem_desc(tc::smem_u32(st + ST_DQ), 256, 128);
            const uint64_t dk0 = tc::smem_desc(tc::smem_u32(st + ST_DK), 256, 128);
            const uint64_t cq0 = tc::smem_desc(tc::smem_u32(smem + SM_BCQ), 128, 512);
            const uint64_t ck0 = tc::smem_desc(tc::smem_u32(smem + SM_BCK), 128, 512);
            const uint64_t ql0 = tc::smem_desc(tc::smem_u32(smem + SM_SPLIT_Q), 256, 128);
            const uint64_t kl0 = tc::smem_desc(tc::smem_u32(smem + SM_SPLIT_K), 256, 128);
            const uint64_t cql0 = tc::smem_desc(tc::smem_u32(smem + SM_SPLIT_CQ), 128, 512);
            const uint64_t ckl0 = tc::smem_desc(tc::smem_u32(smem + SM_SPLIT_CK), 128, 512);
            const uint32_t id16 = tc::idesc_tf32(128, 16);
            const bool lo_b = SPLIT && pass == 1;  // also the low parts of B
            const bool first = pass == 1;          // the chain's first MMA overwrites D
            auto xchain = [&](const int t, const bool kside) {
                const uint64_t bhi = kside ? dk0 : dq0, blo = kside ? kl0 : ql0;
                const uint32_t d = tbase + (kside ? TM_XK : TM_XQ) + 16 * (t - 1);
                for (int kk = 0; kk < 2 * t; ++kk)
                    tc::mma_tf32_ts(d, tbase + tm_arow(t) + 8 * kk,
                                    bhi + (uint64_t)((dablk(t, 0) * 1024 + 512 * kk) >> 4), id16,
                                    !first || kk > 0);
                if (lo_b)
                    for (int kk = 0; kk < 2 * t; ++kk)
                        tc::mma_tf32_ts(d, tbase + tm_arow(t) + 8 * kk,
                                        blo + (uint64_t)(((t * (t - 1) / 2) * 1024 + 512 * kk) >> 4),
                                        id16, true);
            };
            auto pchain = [&](const int j) {
                const uint32_t idj = tc::idesc_tf32(128, 16 * j);
                for (int kk = 0; kk < 2; ++kk)
                    tc::mma_tf32_ts(tbase + tm_p(j), tbase + TM_AQB + 16 * (j - 1) + 8 * kk,
                                    cq0 + ((bcol_off(j) + 256 * kk) >> 4), idj, !first || kk > 0);
                for (int kk = 0; kk < 2; ++kk)
                    tc::mma_tf32_ts(tbase + tm_p(j), tbase + TM_AKBB + 16 * (j - 1) + 8 * kk,
                                    ck0 + ((bcol_off(j) + 256 * kk) >> 4), idj, true);
                if (lo_b)
                    for (int kk = 0; kk < 2; ++kk) {
                        const uint64_t off = (bcol_off(j) + 256 * kk) >> 4;
                        tc::mma_tf32_ts(tbase + tm_p(j), tbase + TM_AQB + 16 * (j - 1) + 8 * kk,
                                        cql0 + off, idj, true);
                        tc::mma_tf32_ts(tbase + tm_p(j), tbase + TM_AKBB + 16 * (j - 1) + 8 * kk,
                                        ckl0 + off, idj, true);
                    }
            };
            if (tc::elect_one()) {
                if (warp == 13) {
                    xchain(3, false);
                    xchain(3, true);
                } else if (warp == 14) {
                    xchain(2, false);
                    xchain(2, true);
                    pchain(1);
                } else {
                    xchain(1, false);
                    xchain(1, true);
                    pchain(2);
                    pchain(3);
                }
                tc::mma_commit(pass == 1 ? mbar : mbar2);
            }
            __syncwarp();
        };
        if (warp >= TC_WARPS - MMA_WARPS) {
            ok &= tc::mbar_wait(mbar + 1, (uint32_t)it & 1u, SPIN_LIMIT);
            tc::fence_after_sync();
            issue_chains(1);
        }

        // ---- diagonal block, two source rows at a time in packed FP32x2: one exp2 per
        // (r, s, d), shared by both sides (FACTOR: in the two 8x8 triangles, with the
        // factorized quadrant in between).  Rows run in descending order: once row r is
        // processed, its row sums and its column sum dkt[r] are complete, so each row is
        // written out right away.  Rows 15..8 (92 of the 120 pairs) run before the MMA
        // result is needed; rows 7..0 after it. ----
        float accq[BC], acck[BC], dbv[BC];
        float2 dkt2[BC / 2];
#pragma unroll
        for (int m = 0; m < BC / 2; ++m) dkt2[m] = make_float2(0.f, 0.f);
        const float *dgq = reinterpret_cast<const float *>(st + ST_DQ) + dablk(i, i) * 256;
        const float *dgk = reinterpret_cast<const float *>(st + ST_DK) + dablk(i, i) * 256;
        const float2 neg1 = make_float2(-1.f, -1.f);
        size_t orow0;  // output row (token * H + head) of row r0
        if constexpr (VARLEN) {
            orow0 = (size_t)(meta[2 * sidx] + r0) * H + unit_head(u);
        } else {
            orow0 = unit_row(u, r0);
        }
        const size_t obase = orow0 * KD + d;
        const uint32_t hk = (uint32_t)H * KD;

        // FACTOR: the lower-left quadrant (rows 8..15 against sources 0..7) through
        // row 8, 2^(g_r - g_s) = 2^(g_r - g_8) 2^(g_8 - g_s), both exponents <= 0.
        // kbq[m] holds k_s 2^(g_8 - g_s) for the source pair m; dktq[m] the column
        // sums still to be scaled by 2^(g_8 - g_s).
        const float g8 = KDA_EL(g2, BC / 2);
        float2 kbq[BC / 4], dktq[BC / 4];
        if constexpr (FACTOR) {
#pragma unroll
            for (int m = 0; m < BC / 4; ++m) {
                const float2 df = __ffma2_rn(g2[m], neg1, make_float2(g8, g8));
                kbq[m] = __fmul2_rn(k2[m], make_float2(ex2(df.x), ex2(df.y)));
                dktq[m] = make_float2(0.f, 0.f);
            }
        }

        auto diag_row = [&](const int r) {
            const float gv = KDA_EL(g2, r), kv = KDA_EL(k2, r);
            const float qv = to_f32(sq[(r0 + r) * KD + d]);
            const float kbr = sbeta[r0 + r] * kv;
            const float2 grr = make_float2(gv, gv);
            const float2 qq = make_float2(qv, qv);
            const float2 kb2 = make_float2(kbr, kbr);
            float2 aacc = make_float2(0.f, 0.f), kacc = make_float2(0.f, 0.f);
            // row r's 16-byte chunk c of the diagonal block sits at c*64 + roff floats
            const int roff = (r >> 3) * 32 + (r & 7) * 4;
            int cfirst = 0;
            if (FACTOR && r >= BC / 2) {  // the factorized quadrant: sources 0..7
                const float ar = r == BC / 2 ? 1.f : ex2(gv - g8);
                const float2 qa = make_float2(ar * qv, ar * qv);
                const float2 kba = make_float2(ar * kbr, ar * kbr);
                float2 sq2 = make_float2(0.f, 0.f), sk2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const float4 aq4 = *reinterpret_cast<const float4 *>(dgq + c * 64 + roff);
                    const float4 ak4 = *reinterpret_cast<const float4 *>(dgk + c * 64 + roff);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int m = 2 * c + h;
                        const float2 aq = h ? make_float2(aq4.z, aq4.w) : make_float2(aq4.x, aq4.y);
                        const float2 ak = h ? make_float2(ak4.z, ak4.w) : make_float2(ak4.x, ak4.y);
                        sq2 = __ffma2_rn(aq, kbq[m], sq2);
                        sk2 = __ffma2_rn(ak, kbq[m], sk2);
                        dktq[m] = __ffma2_rn(ak, kba, __ffma2_rn(aq, qa, dktq[m]));
                    }
                }
                accq[r] = ar * (sq2.x + sq2.y);
                acck[r] = ar * (sk2.x + sk2.y);
                cfirst = 2;
            }
            // pairs (2m, 2m+1) cover s < r; for odd r the last pair is (r-1, r) and
            // carries the diagonal term (E = 1, dAkk[r][r] outside the support -> 0)
#pragma unroll
            for (int c = cfirst; c < (r + 3) / 4; ++c) {
                const float4 aq4 = *reinterpret_cast<const float4 *>(dgq + c * 64 + roff);
                const float4 ak4 = *reinterpret_cast<const float4 *>(dgk + c * 64 + roff);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int m = 2 * c + h;
                    if (2 * m < r) {
                        const float2 aq = h ? make_float2(aq4.z, aq4.w) : make_float2(aq4.x, aq4.y);
                        float2 ak = h ? make_float2(ak4.z, ak4.w) : make_float2(ak4.x, ak4.y);
                        if (2 * m + 1 == r) ak.y = 0.f;
                        const float2 df = __ffma2_rn(g2[m], neg1, grr);
                        const float2 ev = make_float2(ex2(df.x), ex2(df.y));
                        const float2 tq = __fmul2_rn(k2[m], ev);
                        aacc = __ffma2_rn(aq, tq, aacc);
                        kacc = __ffma2_rn(ak, tq, kacc);
                        const float2 uu = __ffma2_rn(aq, qq, __fmul2_rn(ak, kb2));
                        dkt2[m] = __ffma2_rn(uu, ev, dkt2[m]);
                    }
                }
            }
            accq[r] += aacc.x + aacc.y;
            acck[r] += kacc.x + kacc.y;
            if ((r & 1) == 0) {  // even r: the diagonal term on its own
                const float aqd = dgq[(r >> 2) * 64 + roff + (r & 3)];
                accq[r] = fmaf(aqd, kv, accq[r]);
                dkt2[r >> 1].x = fmaf(aqd, qv, dkt2[r >> 1].x);
            }
        };
        // incoming gradients (ACCUM): fetched two output rows ahead of their use (three
        // measured 5% slower, five 13% slower); in place (ACCUM == 2) only dg_in under the
        // fold is loaded, the stores add the others
        constexpr bool INPLACE = ACCUM == 2;
        constexpr int AHEAD = 2;
        float inq[BC], ink[BC], ing[BC];
        auto fetch_in = [&](const int r) {
            if constexpr (ACCUM) {
                const bool live = !VARLEN || r0 + r < ulen;
                const size_t off = obase + (size_t)((uint32_t)r * hk);
                const bool rd = live && dbg_ok(ex.dbg, off, ex.nrows * KD, DBG_LOAD);
                inq[r] = (!INPLACE && rd && ex.dq_in) ? __ldg(ex.dq_in + off) : 0.f;
                ink[r] = (!INPLACE && rd && ex.dk_in) ? __ldg(ex.dk_in + off) : 0.f;
                ing[r] = ((!INPLACE || FOLD) && rd && ex.dg_in) ? __ldg(ex.dg_in + off) : 0.f;
            }
        };
        float fold_run = 0.f;  // FOLD: running suffix sum of dg inside the sub-block
        float *bank = reinterpret_cast<float *>(smem + SM_FOLD_BANK);
        auto out_row = [&](const int r) {
            const int row = r0 + r;
            const size_t off = obase + (size_t)((uint32_t)r * hk);
            if (r >= AHEAD) fetch_in(r - AHEAD);
            // foreign rows: nothing is stored
            const bool live = (!VARLEN || row < ulen) && dbg_ok(ex.dbg, off, ex.nrows * KD, DBG_STORE);
            const float qv = to_f32(sq[row * KD + d]);
            const float kv = KDA_EL(k2, r), dkv = KDA_EL(dkt2, r);
            // every rounding spelled out (no compiler-chosen contraction), so all
            // instantiations give bitwise the same values
            const float pk = __fmul_rn(sbeta[row], acck[r]);
            float vq = accq[r], vk = fmaf(sbeta[row], acck[r], dkv);
            float vg = __fmul_rn(LN2, fmaf(qv, accq[r], __fmul_rn(__fsub_rn(pk, dkv), kv)));
            if constexpr (ACCUM) {
                vq += inq[r];
                vk += ink[r];
                vg += ing[r];
            }
            if (live) {
                if constexpr (EMIT) {
                    reinterpret_cast<io_t *>(dq_out)[off] = from_f32<io_t>(vq);
                    reinterpret_cast<io_t *>(dk_out)[off] = from_f32<io_t>(vk);
                } else if constexpr (INPLACE) {
                    red_add(dq + off, vq);
                    red_add(dk + off, vk);
                } else {
                    dq[off] = vq;
                    dk[off] = vk;
                }
            }
            if constexpr (FOLD) {
                fold_run += live ? vg : 0.f;
                bank[row * KD + d] = fold_run;
            } else if constexpr (INPLACE) {
                if (live) red_add(dg + off, vg);
            } else {
                if (live) dg[off] = vg;
            }
            dbv[r] = acck[r] * kv;  // kv = 0 on foreign rows; their db is never stored
        };
        // db[r] = sum over d of 8 rows at a time: transpose-reduce across the warp's lanes
        // (lane l ends with row (l>>2)&7), then a fixed-order sum over the block's 4 warps.
        auto db_rows = [&](const int rbase) {
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = dbv[rbase + j];
#pragma unroll
            for (int w = 4, m = 16; w >= 1; w >>= 1, m >>= 1) {
                const bool hi = (lane & m) != 0;
#pragma unroll
                for (int j = 0; j < w; ++j) {
                    const float send = hi ? v[j] : v[j + w];
                    const float keep = hi ? v[j + w] : v[j];
                    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                }
            }
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
            if ((lane & 3) == 0) sdbp[(warp & 3) * BT + r0 + rbase + (lane >> 2)] = v[0];
        };

        // the first rows' incoming gradients: fetched here, or, with the fold (the fullest
        // registers), only after the post-factors, just before the first output row
        // (measured faster each way)
        if constexpr (!FOLD) {
#pragma unroll
            for (int r = BC - 1; r >= BC - AHEAD; --r) fetch_in(r);
        }
        // SPLIT: rows 15..12, then the second MMA pass is prepared, then rows 11..8
        constexpr int RMID = SPLIT ? 3 * BC / 4 : BC / 2;
#pragma unroll
        for (int r = BC - 1; r >= RMID; --r) {
            if constexpr (!FACTOR) accq[r] = acck[r] = 0.f;
            diag_row(r);
        }
        if constexpr (SPLIT) {
            // pass 1 done: the A operands it read are replaced by their low parts
            // (recomputed exactly as in the prescale), then warps 13..15 issue pass 2
            ok &= tc::mbar_wait(mbar, (uint32_t)it & 1u, SPIN_LIMIT);
            tc::fence_after_sync();
            if (i < NBLK - 1) {
                float a[BC], v[BC];
                tc::tmem_ld16(tlane + TM_FA + 16 * i, a);
                tc::tmem_wait_ld();
#pragma unroll
                for (int m = 0; m < BC / 2; ++m) {
                    const float2 vv = __fmul2_rn(k2[m], make_float2(a[2 * m], a[2 * m + 1]));
                    v[2 * m] = vv.x;
                    v[2 * m + 1] = vv.y;
                }
                tmem_st_part<true, true>(tlane + tm_arow(i + 1) + 16 * i, v);
                if (i + 2 < NBLK) {
#pragma unroll
                    for (int m = 0; m < BC / 2; ++m) {
                        const float2 t = __fmul2_rn(make_float2(v[2 * m], v[2 * m + 1]), make_float2(c2, c2));
                        a[2 * m] = t.x;
                        a[2 * m + 1] = t.y;
                    }
                    tmem_st_part<true, true>(tlane + tm_arow(i + 2) + 16 * i, a);
                }
                if (i + 3 < NBLK) {
#pragma unroll
                    for (int m = 0; m < BC / 2; ++m) {
                        const float2 t = __fmul2_rn(make_float2(v[2 * m], v[2 * m + 1]), make_float2(c3, c3));
                        a[2 * m] = t.x;
                        a[2 * m + 1] = t.y;
                    }
                    tmem_st_part<true, true>(tlane + tm_arow(i + 3) + 16 * i, a);
                }
            }
            if (i > 0) {
                float b[BC], v[BC];
                tc::tmem_ld16(tlane + TM_FB + 16 * (i - 1), b);
                tc::tmem_wait_ld();
#pragma unroll
                for (int m = 0; m < BC / 2; ++m) {
                    const float2 t = __fmul2_rn(make_float2(to_f32(sq[(r0 + 2 * m) * KD + d]),
                                                            to_f32(sq[(r0 + 2 * m + 1) * KD + d])),
                                                make_float2(b[2 * m], b[2 * m + 1]));
                    v[2 * m] = t.x;
                    v[2 * m + 1] = t.y;
                }
                tmem_st_part<true, true>(tlane + TM_AQB + 16 * (i - 1), v);
#pragma unroll
                for (int m = 0; m < BC / 2; ++m) {
                    const float2 bk = __fmul2_rn(*reinterpret_cast<const float2 *>(sbeta + r0 + 2 * m), k2[m]);
                    const float2 t = __fmul2_rn(bk, make_float2(b[2 * m], b[2 * m + 1]));
                    v[2 * m] = t.x;
                    v[2 * m + 1] = t.y;
                }
                tmem_st_part<true, true>(tlane + TM_AKBB + 16 * (i - 1), v);
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(mbar2 + 1);
            if (warp >= TC_WARPS - MMA_WARPS) {
                ok &= tc::mbar_wait(mbar2 + 1, (uint32_t)it & 1u, SPIN_LIMIT);
                tc::fence_after_sync();
                issue_chains(2);
            }
            __syncwarp();
#pragma unroll
            for (int r = RMID - 1; r >= BC / 2; --r) {
                if constexpr (!FACTOR) accq[r] = acck[r] = 0.f;
                diag_row(r);
            }
        }
        if constexpr (FACTOR) {
#pragma unroll
            for (int m = 0; m < BC / 4; ++m) {
                const float2 df = __ffma2_rn(g2[m], neg1, make_float2(g8, g8));
                dkt2[m] = __ffma2_rn(make_float2(ex2(df.x), ex2(df.y)), dktq[m], dkt2[m]);
            }
        }

        // ---- cross terms: wait for the MMAs, apply the post-factors ----
        ok &= tc::mbar_wait(SPLIT ? mbar2 : mbar, (uint32_t)it & 1u, SPIN_LIMIT);
        tc::fence_after_sync();
        if (i > 0) {
            float f[BC], x[BC];
            tc::tmem_ld16(tlane + TM_FB + 16 * (i - 1), f);
            tc::tmem_ld16(tlane + TM_XQ + 16 * (i - 1), x);
            tc::tmem_wait_ld();
#pragma unroll
            for (int r = 0; r < BC; ++r) accq[r] = fmaf(f[r], x[r], r >= BC / 2 ? accq[r] : 0.f);
            tc::tmem_ld16(tlane + TM_XK + 16 * (i - 1), x);
            tc::tmem_wait_ld();
#pragma unroll
            for (int r = 0; r < BC; ++r) acck[r] = fmaf(f[r], x[r], r >= BC / 2 ? acck[r] : 0.f);
        } else {
#pragma unroll
            for (int r = 0; r < BC / 2; ++r) accq[r] = acck[r] = 0.f;
        }
        if (i < NBLK - 1) {
            float y[BC], p[BC];
            tc::tmem_ld16(tlane + tm_p(i + 1) + 16 * i, y);
            tc::tmem_wait_ld();
            if (i + 2 < NBLK) {
                tc::tmem_ld16(tlane + tm_p(i + 2) + 16 * i, p);
                tc::tmem_wait_ld();
#pragma unroll
                for (int s = 0; s < BC; ++s) y[s] = fmaf(c2, p[s], y[s]);
            }
            if (i + 3 < NBLK) {
                tc::tmem_ld16(tlane + tm_p(i + 3) + 16 * i, p);
                tc::tmem_wait_ld();
#pragma unroll
                for (int s = 0; s < BC; ++s) y[s] = fmaf(c3, p[s], y[s]);
            }
            tc::tmem_ld16(tlane + TM_FA + 16 * i, p);
            tc::tmem_wait_ld();
#pragma unroll
            for (int m = 0; m < BC / 2; ++m)
                dkt2[m] = __ffma2_rn(make_float2(p[2 * m], p[2 * m + 1]),
                                     make_float2(y[2 * m], y[2 * m + 1]), dkt2[m]);
        }
        if (!ok) {  // a wait gave up: poison this unit instead of hanging
            const float nan = __int_as_float(0x7fc00000);
#pragma unroll
            for (int r = 0; r < BC; ++r) accq[r] = acck[r] = nan;
#pragma unroll
            for (int m = 0; m < BC / 2; ++m) dkt2[m] = make_float2(nan, nan);
        }

        // ---- rows 15..8 are complete: write them; then rows 7..0 ----
        if constexpr (FOLD) {
#pragma unroll
            for (int r = BC - 1; r >= BC - AHEAD; --r) fetch_in(r);
        }
#pragma unroll
        for (int r = BC - 1; r >= BC / 2; --r) out_row(r);
        db_rows(BC / 2);
#pragma unroll
        for (int r = BC / 2 - 1; r >= 0; --r) {
            diag_row(r);
            out_row(r);
        }
        db_rows(0);
#undef KDA_EL
        tc::named_bar_sync(1 + i, 128);
        if constexpr (SLICED) {
            // the sub-block's rows of the stage are read no more in this unit (every
            // other sub-block's reads of them came before this unit's MMAs completed)
            if ((warp & 3) == 1 && u + 2 * stride < units) {
                tc::fence_proxy_async_smem();
                load_slice(st, &full[sidx], tm, beta, u + 2 * stride, H, ex, lane, i);
            }
        }
        if ((warp & 3) == 0 && lane < BC && (!VARLEN || r0 + lane < ulen)) {
            const int row = r0 + lane;
            // recomputed here rather than kept live across the unit (register budget)
            const size_t brow =
                VARLEN ? (size_t)(meta[2 * sidx] + row) * H + unit_head(u) : unit_row(u, row);
            float v = (sdbp[row] + sdbp[BT + row]) + (sdbp[2 * BT + row] + sdbp[3 * BT + row]);
            if (dbg_ok(ex.dbg, brow, ex.nrows, DBG_STORE)) {
                if constexpr (ACCUM) {
                    if (ex.db_in) v += ex.db_in[brow];
                }
                db[brow] = v;
            }
        }
        if constexpr (FOLD) {
            // the four threads of channel d (one per sub-block, in warps c, c+4, c+8,
            // c+12) exchange their sub-block totals; each adds the totals of the later
            // sub-blocks to its banked in-block suffix sums
            float *tot = reinterpret_cast<float *>(smem + SM_FOLD_TOT) + (it & 1) * NBLK * KD;
            tot[i * KD + d] = fold_run;
            tc::named_bar_sync(5 + (warp & 3), 128);
            float later = 0.f;
#pragma unroll
            for (int j = NBLK - 1; j > 0; --j)
                if (j > i) later += tot[j * KD + d];
#pragma unroll
            for (int r = 0; r < BC; ++r) {
                const size_t off = obase + (size_t)((uint32_t)r * hk);
                if ((!VARLEN || r0 + r < ulen) && dbg_ok(ex.dbg, off, ex.nrows * KD, DBG_STORE))
                    dg[off] = bank[(r0 + r) * KD + d] + later;
            }
        }

        // ---- unit done: the last warp releases the stage and refills it (SLICED: the
        // sub-blocks have refilled their rows above) ----
        if constexpr (!SLICED) {
            tc::fence_before_sync();
            __syncwarp();
            prev = 0;
            if (lane == 0) prev = tc::atomic_add_acq_rel_smem(done_count, 1u);
            prev = __shfl_sync(0xffffffffu, prev, 0);
            if ((prev % TC_WARPS) == TC_WARPS - 1 && u + 2 * stride < units) {
                tc::fence_proxy_async_smem();
                load_unit<VARLEN>(st, &full[sidx], meta + 2 * sidx, tm, beta, u + 2 * stride,
                                  T, H, ex, lane,
                                  lut + (((it + 2) / LUT_BATCH) & 1) * 2 * LUT_BATCH +
                                      2 * ((it + 2) % LUT_BATCH));
            }
        }
    }

    dbg_flag(ex.dbg, !ok, DBG_WAIT);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tbase, TM_COLS);
    }
}

// ---------------------------------------------------------------- host side

// Defined once in kda_intra_tc.cu.  make_maps reuses the maps of its thread's previous
// call when the pointers and shapes are the same; num_sms also returns the device.
cudaError_t make_maps(const BwdArgs &a, TmaMaps *tm);
cudaError_t num_sms(int *n, int *dev);

template <typename io_t, int ACCUM, bool FOLD, bool EMIT, bool VARLEN, bool FACTOR,
          bool SPLIT = false>
cudaError_t launch_typed(const BwdArgs &a, cudaStream_t stream) {
    auto kern = kda_intra_bwd_tc_kernel<io_t, ACCUM, FOLD, EMIT, VARLEN, FACTOR, SPLIT>;
    static_assert(!(FOLD && SPLIT), "no shared-memory layout for both");
    const int smem_bytes = FOLD ? SM_TOTAL_FOLD : SPLIT ? SM_TOTAL_SPLIT : SM_TOTAL;
    static volatile int smem_set[kMaxDev];  // this instantiation's attribute, per device
    int nsm = 0, dev = 0;
    cudaError_t e = num_sms(&nsm, &dev);
    if (e != cudaSuccess) return e;
    if ((e = smem_limit_once(kern, smem_bytes, dev, smem_set)) != cudaSuccess) return e;
    TmaMaps tm;
    if ((e = make_maps(a, &tm)) != cudaSuccess) return e;
    const int HV = a.HV > 0 ? a.HV : a.H;
    Extras ex;
    ex.dq_in = a.dq_in;
    ex.dk_in = a.dk_in;
    ex.dg_in = a.dg_in;
    ex.db_in = a.db_in;
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
    kern<<<grid, TC_THREADS, smem_bytes, stream>>>(tm, a.beta, a.dq, a.dk, a.db, a.dg, a.T, HV,
                                                   units, ex);
    return cudaGetLastError();
}

template <typename io_t, bool EMIT, bool VARLEN, bool FACTOR>
cudaError_t launch_opts(const BwdArgs &a, cudaStream_t stream) {
    const bool accum = a.dq_in || a.dk_in || a.dg_in || a.db_in;
    // in place: dq_in, dk_in (and dg_in unless folded) are the outputs themselves
    const bool in_place = !EMIT && a.dq_in == a.dq && a.dk_in == a.dk &&
                          (a.fold_dg || a.dg_in == a.dg);
    if (accum && in_place && !EMIT)
        return a.fold_dg ? launch_typed<io_t, 2, true, false, VARLEN, FACTOR>(a, stream)
                         : launch_typed<io_t, 2, false, false, VARLEN, FACTOR>(a, stream);
    if (accum)
        return a.fold_dg ? launch_typed<io_t, 1, true, EMIT, VARLEN, FACTOR>(a, stream)
                         : launch_typed<io_t, 1, false, EMIT, VARLEN, FACTOR>(a, stream);
    return a.fold_dg ? launch_typed<io_t, 0, true, EMIT, VARLEN, FACTOR>(a, stream)
                     : launch_typed<io_t, 0, false, EMIT, VARLEN, FACTOR>(a, stream);
}

// The split-TF32 cross sums: fixed-length units, no other option but grouped value
// heads.
template <typename io_t>
cudaError_t launch_split(const BwdArgs &a, cudaStream_t stream) {
    return launch_typed<io_t, 0, false, false, false, false, true>(a, stream);
}

// Every option combination of one q/k element type, one sequence layout and one
// diagonal-block form.
template <typename io_t, bool VARLEN, bool FACTOR>
cudaError_t launch_io(const BwdArgs &a, cudaStream_t stream) {
    return a.emit_io ? launch_opts<io_t, true, VARLEN, FACTOR>(a, stream)
                     : launch_opts<io_t, false, VARLEN, FACTOR>(a, stream);
}

}  // namespace tcimpl
}  // namespace kda
