// Tensor-core kernel for the KDA intra-chunk backward (sm_103a, tcgen05 + TMEM).
//
// Persistent grid (one 512-thread CTA per SM), units (b, h, 64-token chunk) dealt
// round-robin.  Each unit's inputs are staged with 16-byte cp.async into one of two
// shared-memory stages while the previous unit is being computed.
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
// 36 MMAs (M=128 channels, N=16..48, K=8) per unit, issued by one thread, run while
// all warps compute the 16x16 diagonal blocks with one exp2 per (r, s, d).
#include "kda_common.cuh"
#include "kda_launch.h"
#include "tc_ptx.cuh"

namespace kda {
namespace {

constexpr int TC_THREADS = 512;

// ---- shared memory: two input stages + single-buffered derived operands ----
constexpr int ST_Q = 0;                        // io_t [64][128]
constexpr int ST_K = ST_Q + BT * KD * 2;       // io_t [64][128]
constexpr int ST_G = ST_K + BT * KD * 2;       // f32  [64][128]
constexpr int ST_BQ = ST_G + BT * KD * 4;      // dAqk rows of block t, cols < 16t (K-major core layout)
constexpr int ST_BK = ST_BQ + 6144;            // same for dAkk
constexpr int ST_DQ = ST_BK + 6144;            // dAqk diagonal blocks f32 [4][16][16]
constexpr int ST_DK = ST_DQ + 4096;            // dAkk diagonal blocks
constexpr int ST_BETA = ST_DK + 4096;          // f32 [64]
constexpr int STAGE_BYTES = ST_BETA + 256;     // 86272
constexpr int SM_BCQ = 2 * STAGE_BYTES;        // dAqk blocks of target j transposed (K-major)
constexpr int SM_BCK = SM_BCQ + 6144;
constexpr int SM_DBP = SM_BCK + 6144;          // db partials f32 [4][64]
constexpr int SM_MBAR = SM_DBP + 1024;
constexpr int SM_TSLOT = SM_MBAR + 16;
constexpr int SM_TOTAL = SM_TSLOT + 8;
static_assert(STAGE_BYTES % 128 == 0, "stage alignment");

// byte offset of block t's operand inside a 6 KB B region: sizes 1, 2, 3 KB
__device__ __forceinline__ uint32_t blk_off(int t) { return 512u * (uint32_t)((t - 1) * t); }

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

constexpr uint32_t MBAR_SPIN_LIMIT = 1u << 20;

__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(gmem) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Queue this thread's share of one unit's input copies into a stage.  Row r of
// the unit sits at global row `row0 + r*H` of every [B, T, H, *] tensor.
template <typename io_t>
__device__ __forceinline__ void issue_unit_loads(unsigned char *st, const io_t *__restrict__ q,
                                                 const io_t *__restrict__ k,
                                                 const float *__restrict__ g,
                                                 const float *__restrict__ beta,
                                                 const float *__restrict__ dAqk,
                                                 const float *__restrict__ dAkk,
                                                 size_t row0, int H, int tid) {
    const size_t e128 = row0 * KD, e64 = row0 * BT;
    const uint32_t hk = (uint32_t)H * KD;
#pragma unroll
    for (int x = 0; x < 2; ++x) {  // q, k: 64 rows x 16 chunks
        const int r = (tid >> 4) + 32 * x, c = tid & 15;
        const size_t off = e128 + (size_t)((uint32_t)r * hk + c * 8);
        cp_async16(st + ST_Q + r * 256 + c * 16, q + off);
        cp_async16(st + ST_K + r * 256 + c * 16, k + off);
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {  // g: 64 rows x 32 chunks
        const int r = (tid >> 5) + 16 * x, c = tid & 31;
        cp_async16(st + ST_G + r * 512 + c * 16, g + e128 + (size_t)((uint32_t)r * hk + c * 4));
    }
    // dA: 64 rows x 16 chunks, of which row r of block t needs the first 4(t+1):
    // 4t off-diagonal chunks for the tensor-core operand of block t, then the
    // 4 chunks of the diagonal block.
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        const int r = (tid >> 4) + 32 * x, c = tid & 15;
        const int t = r >> 4, n = r & 15;
        if (c < 4 * (t + 1)) {
            const size_t src = e64 + (size_t)((uint32_t)r * H * BT + c * 4);
            const bool off_diag = c < 4 * t;
            const uint32_t dst =
                off_diag ? blk_off(t) + (uint32_t)((n >> 3) * (512 * t) + c * 128 + (n & 7) * 16)
                         : (uint32_t)(t * 1024 + n * 64 + (c - 4 * t) * 16);
            cp_async16(st + (off_diag ? ST_BQ : ST_DQ) + dst, dAqk + src);
            cp_async16(st + (off_diag ? ST_BK : ST_DK) + dst, dAkk + src);
        }
    }
    if (tid < BT) cp_async4(st + ST_BETA + tid * 4, beta + row0 + (size_t)tid * H);
}

template <typename io_t>
__global__ void __launch_bounds__(TC_THREADS, 1)
kda_intra_bwd_tc_kernel(const io_t *__restrict__ q, const io_t *__restrict__ k,
                        const float *__restrict__ g, const float *__restrict__ beta,
                        const float *__restrict__ dAqk, const float *__restrict__ dAkk,
                        float *__restrict__ dq, float *__restrict__ dk,
                        float *__restrict__ db, float *__restrict__ dg, int T, int H,
                        long long units) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int i = tid >> 7;  // sub-block, warp-uniform
    const int d = tid & 127;
    const int r0 = i * BC;
    const int NT = T / BT;
    uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + SM_MBAR);          // MMAs done
    uint32_t *ops_count = reinterpret_cast<uint32_t *>(smem + SM_MBAR + 8);  // warps done
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + SM_TSLOT);
    float *sdbp = reinterpret_cast<float *>(smem + SM_DBP);

    if (warp == 0) tc::tmem_alloc(tslot, TM_COLS);
    if (tid == 0) {
        tc::mbar_init(mbar, 1);
        *ops_count = 0u;
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tslot;
    const uint32_t tlane = tbase + ((uint32_t)(32 * (warp & 3)) << 16);

    long long u = blockIdx.x;
    if (u < units)
        issue_unit_loads(smem, q, k, g, beta, dAqk, dAkk, grow(decode_unit(u, H, NT), 0, T, H), H,
                         tid);
    cp_async_commit();

    uint32_t phase = 0;
    for (int it = 0; u < units; ++it, u += gridDim.x) {
        unsigned char *st = smem + (it & 1) * STAGE_BYTES;
        const Unit un = decode_unit(u, H, NT);
        if (u + gridDim.x < units)
            issue_unit_loads(smem + ((it + 1) & 1) * STAGE_BYTES, q, k, g, beta, dAqk, dAkk,
                             grow(decode_unit(u + gridDim.x, H, NT), 0, T, H), H, tid);
        cp_async_commit();
        cp_async_wait_group<1>();
        __syncthreads();

        const float *sg = reinterpret_cast<const float *>(st + ST_G);
        const io_t *sq = reinterpret_cast<const io_t *>(st + ST_Q);
        const io_t *sk = reinterpret_cast<const io_t *>(st + ST_K);
        const float *sbeta = reinterpret_cast<const float *>(st + ST_BETA);

        // this thread's column of its block, as (even row, odd row) pairs
        float2 g2[BC / 2], k2[BC / 2];
#pragma unroll
        for (int m = 0; m < BC / 2; ++m) {
            g2[m] = make_float2(sg[(r0 + 2 * m) * KD + d], sg[(r0 + 2 * m + 1) * KD + d]);
            k2[m] = make_float2(to_f32(sk[(r0 + 2 * m) * KD + d]),
                                to_f32(sk[(r0 + 2 * m + 1) * KD + d]));
        }
#define KDA_EL(arr, r) (((r) & 1) ? arr[(r) >> 1].y : arr[(r) >> 1].x)

        // ---- prescaled TF32 operands and post-factors into TMEM ----
        float c2 = 0.f, c3 = 0.f;  // 2^(g_16(i+2) - g_e(i)), 2^(g_16(i+3) - g_e(i))
        if (i < NBLK - 1) {
            const float ge = sg[(r0 + BC) * KD + d];
            float a[BC], v[BC];
#pragma unroll
            for (int s = 0; s < BC; ++s) {
                a[s] = ex2(ge - KDA_EL(g2, s));
                v[s] = KDA_EL(k2, s) * a[s];
            }
            tc::tmem_st16(tlane + TM_FA + 16 * i, a);
            tc::tmem_st16(tlane + tm_arow(i + 1) + 16 * i, v);
            if (i + 2 < NBLK) {
                c2 = ex2(sg[(r0 + 2 * BC) * KD + d] - ge);
#pragma unroll
                for (int s = 0; s < BC; ++s) a[s] = v[s] * c2;
                tc::tmem_st16(tlane + tm_arow(i + 2) + 16 * i, a);
            }
            if (i + 3 < NBLK) {
                c3 = ex2(sg[(r0 + 3 * BC) * KD + d] - ge);
#pragma unroll
                for (int s = 0; s < BC; ++s) a[s] = v[s] * c3;
                tc::tmem_st16(tlane + tm_arow(i + 3) + 16 * i, a);
            }
        }
        if (i > 0) {
            float b[BC], v[BC];
            b[0] = 1.f;
#pragma unroll
            for (int r = 1; r < BC; ++r) b[r] = ex2(KDA_EL(g2, r) - g2[0].x);
            tc::tmem_st16(tlane + TM_FB + 16 * (i - 1), b);
#pragma unroll
            for (int r = 0; r < BC; ++r) v[r] = to_f32(sq[(r0 + r) * KD + d]) * b[r];
            tc::tmem_st16(tlane + TM_AQB + 16 * (i - 1), v);
#pragma unroll
            for (int r = 0; r < BC; ++r) v[r] = sbeta[r0 + r] * KDA_EL(k2, r) * b[r];
            tc::tmem_st16(tlane + TM_AKBB + 16 * (i - 1), v);
        }

        // ---- column-side B operands: dA blocks of target j transposed ----
        {
            const float *bq = reinterpret_cast<const float *>(st + ST_BQ);
            const float *bk = reinterpret_cast<const float *>(st + ST_BK);
            float *cq = reinterpret_cast<float *>(smem + SM_BCQ);
            float *ck = reinterpret_cast<float *>(smem + SM_BCK);
#pragma unroll
            for (int x = 0; x < 3; ++x) {
                const int idx = tid + x * TC_THREADS;  // < 1536
                const int j = idx >= 768 ? 3 : idx >= 256 ? 2 : 1;
                const int e = idx - 128 * j * (j - 1);
                // e enumerates the destination bytes/4 in order: (n/8, k/4, n%8, k%4)
                const int n = (e >> 7) * 8 + ((e >> 2) & 7);  // s
                const int kk = ((e >> 5) & 3) * 4 + (e & 3);  // r - 16j
                const int src = (int)blk_off(j) / 4 + (kk >> 3) * (128 * j) + (n >> 2) * 32 +
                                (kk & 7) * 4 + (n & 3);
                const int dst = (int)blk_off(j) / 4 + e;
                cq[dst] = bq[src];
                ck[dst] = bk[src];
            }
        }
        // operands complete: TMEM stores landed, smem stores visible to the tensor core;
        // the last warp to finish issues the 36 MMAs (no thread waits for the others)
        tc::tmem_wait_st();
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncwarp();
        uint32_t prev = 0;
        if (lane == 0) prev = tc::atomic_add_acq_rel_smem(ops_count, 1u);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if ((prev & 15u) == 15u && lane == 0) {
            tc::fence_after_sync();
            const uint32_t bq = tc::smem_u32(st + ST_BQ), bk = tc::smem_u32(st + ST_BK);
            const uint32_t id16 = tc::idesc_tf32(128, 16);
#pragma unroll
            for (int t = 1; t < NBLK; ++t) {
#pragma unroll
                for (int kk = 0; kk < 2 * t; ++kk) {
                    const uint32_t a = tbase + tm_arow(t) + 8 * kk;
                    const uint32_t boff = blk_off(t) + 256 * kk;
                    tc::mma_tf32_ts(tbase + TM_XQ + 16 * (t - 1), a,
                                    tc::smem_desc(bq + boff, 128, 512 * t), id16, kk > 0);
                    tc::mma_tf32_ts(tbase + TM_XK + 16 * (t - 1), a,
                                    tc::smem_desc(bk + boff, 128, 512 * t), id16, kk > 0);
                }
            }
            const uint32_t cq = tc::smem_u32(smem + SM_BCQ), ck = tc::smem_u32(smem + SM_BCK);
#pragma unroll
            for (int j = 1; j < NBLK; ++j) {
                const uint32_t idj = tc::idesc_tf32(128, 16 * j);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    tc::mma_tf32_ts(tbase + tm_p(j), tbase + TM_AQB + 16 * (j - 1) + 8 * kk,
                                    tc::smem_desc(cq + blk_off(j) + 256 * kk, 128, 512), idj,
                                    kk > 0);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    tc::mma_tf32_ts(tbase + tm_p(j), tbase + TM_AKBB + 16 * (j - 1) + 8 * kk,
                                    tc::smem_desc(ck + blk_off(j) + 256 * kk, 128, 512), idj,
                                    true);
            }
            tc::mma_commit(mbar);
        }
        __syncwarp();

        // ---- diagonal block: one exp2 per (r, s, d), shared by both sides, computed
        // two source rows at a time with packed FP32x2 arithmetic ----
        float accq[BC], acck[BC];
        float2 dkt2[BC / 2];
#pragma unroll
        for (int m = 0; m < BC / 2; ++m) dkt2[m] = make_float2(0.f, 0.f);
        {
            const float *dgq = reinterpret_cast<const float *>(st + ST_DQ) + i * 256;
            const float *dgk = reinterpret_cast<const float *>(st + ST_DK) + i * 256;
            const float2 neg1 = make_float2(-1.f, -1.f);
#pragma unroll
            for (int r = 0; r < BC; ++r) {
                const float gv = KDA_EL(g2, r), kv = KDA_EL(k2, r);
                const float qv = to_f32(sq[(r0 + r) * KD + d]);
                const float kbr = sbeta[r0 + r] * kv;
                const float2 grr = make_float2(gv, gv);
                const float2 qq = make_float2(qv, qv);
                const float2 kb2 = make_float2(kbr, kbr);
                float2 aacc = make_float2(0.f, 0.f), kacc = make_float2(0.f, 0.f);
                // pairs (2m, 2m+1) cover s < r; for odd r the last pair is (r-1, r) and
                // carries the diagonal term (E = 1, dAkk[r][r] outside the support -> 0)
#pragma unroll
                for (int c = 0; c < (r + 3) / 4; ++c) {
                    const float4 aq4 = *reinterpret_cast<const float4 *>(dgq + r * 16 + 4 * c);
                    const float4 ak4 = *reinterpret_cast<const float4 *>(dgk + r * 16 + 4 * c);
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
                accq[r] = aacc.x + aacc.y;
                acck[r] = kacc.x + kacc.y;
                if ((r & 1) == 0) {  // even r: the diagonal term on its own
                    const float aqd = dgq[r * 16 + r];
                    accq[r] = fmaf(aqd, kv, accq[r]);
                    dkt2[r >> 1].x = fmaf(aqd, qv, dkt2[r >> 1].x);
                }
            }
        }

        // ---- cross terms: wait for the MMAs, apply the post-factors ----
        const bool ok = tc::mbar_wait(mbar, phase, MBAR_SPIN_LIMIT);
        phase ^= 1u;
        tc::fence_after_sync();
        if (i > 0) {
            float f[BC], x[BC];
            tc::tmem_ld16(tlane + TM_FB + 16 * (i - 1), f);
            tc::tmem_ld16(tlane + TM_XQ + 16 * (i - 1), x);
            tc::tmem_wait_ld();
#pragma unroll
            for (int r = 0; r < BC; ++r) accq[r] = fmaf(f[r], x[r], accq[r]);
            tc::tmem_ld16(tlane + TM_XK + 16 * (i - 1), x);
            tc::tmem_wait_ld();
#pragma unroll
            for (int r = 0; r < BC; ++r) acck[r] = fmaf(f[r], x[r], acck[r]);
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
        if (!ok) {  // the MMAs never signalled: poison this unit instead of hanging
            const float nan = __int_as_float(0x7fc00000);
#pragma unroll
            for (int r = 0; r < BC; ++r) accq[r] = acck[r] = nan;
#pragma unroll
            for (int m = 0; m < BC / 2; ++m) dkt2[m] = make_float2(nan, nan);
        }

        // ---- epilogue ----
        float dbv[BC];
        {
            const size_t base = grow(un, r0, T, H) * KD + d;
            const uint32_t hk = (uint32_t)H * KD;
#pragma unroll
            for (int r = 0; r < BC; ++r) {
                const int row = r0 + r;
                const size_t off = base + (size_t)((uint32_t)r * hk);
                const float qv = to_f32(sq[row * KD + d]);
                const float kv = KDA_EL(k2, r), dkv = KDA_EL(dkt2, r);
                const float pk = sbeta[row] * acck[r];
                dq[off] = accq[r];
                dk[off] = pk + dkv;
                dg[off] = LN2 * fmaf(qv, accq[r], (pk - dkv) * kv);
                dbv[r] = acck[r] * kv;
            }
        }
#undef KDA_EL
        // db[r] = sum over d: transpose-reduce the 16 row sums across the warp's lanes,
        // lane l ends with row l>>1; then a fixed-order sum over the block's 4 warps.
#pragma unroll
        for (int w = 8, m = 16; w >= 1; w >>= 1, m >>= 1) {
            const bool hi = (lane & m) != 0;
#pragma unroll
            for (int j = 0; j < w; ++j) {
                const float send = hi ? dbv[j] : dbv[j + w];
                const float keep = hi ? dbv[j + w] : dbv[j];
                dbv[j] = keep + __shfl_xor_sync(0xffffffffu, send, m);
            }
        }
        dbv[0] += __shfl_xor_sync(0xffffffffu, dbv[0], 1);
        if ((lane & 1) == 0) sdbp[(warp & 3) * BT + r0 + (lane >> 1)] = dbv[0];
        tc::fence_before_sync();
        __syncthreads();
        if (tid < BT)
            db[grow(un, tid, T, H)] = (sdbp[tid] + sdbp[BT + tid]) +
                                      (sdbp[2 * BT + tid] + sdbp[3 * BT + tid]);
        tc::fence_after_sync();
    }

    cp_async_wait_group<0>();
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tbase, TM_COLS);
    }
}

int g_num_sms[64];

template <typename io_t>
cudaError_t launch_typed(const BwdArgs &a, cudaStream_t stream) {
    auto kern = kda_intra_bwd_tc_kernel<io_t>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM_TOTAL);
    if (e != cudaSuccess) return e;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    int nsm = (dev >= 0 && dev < 64) ? g_num_sms[dev] : 0;
    if (nsm == 0) {
        if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64) g_num_sms[dev] = nsm;
    }
    const long long units = (long long)a.B * a.H * (a.T / BT);
    const unsigned grid = (unsigned)(units < nsm ? units : nsm);
    kern<<<grid, TC_THREADS, SM_TOTAL, stream>>>((const io_t *)a.q, (const io_t *)a.k, a.g,
                                                 a.beta, a.dAqk, a.dAkk, a.dq, a.dk, a.db,
                                                 a.dg, a.T, a.H, units);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_intra_tc(const BwdArgs &a, cudaStream_t stream) {
    return a.fp16 ? launch_typed<__half>(a, stream) : launch_typed<__nv_bfloat16>(a, stream);
}

}  // namespace kda
