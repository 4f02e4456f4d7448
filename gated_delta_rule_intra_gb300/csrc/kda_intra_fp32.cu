// All-FP32 kernel for the KDA intra-chunk backward.
//
// The persistent pipeline of the tensor-core kernel (one 512-thread CTA per SM, two
// TMA input stages, no CTA-wide barrier inside the unit loop, the last warp to finish
// a unit refills its stage), with every product and sum in FP32 on the SIMT pipes.
// Thread (i, d) owns sub-block i (rows 16i..16i+15) at channel d:
//
//  * cross-sub-block terms first, through the per-boundary factorization of the
//    bwd_intra page's module docstring: for r in block i and s in block j < i,
//        2^(g_r - g_s) = 2^(g_r - g_16i) * 2^(g_16i - g_e(j)) * 2^(g_e(j) - g_s),
//    e(j) = 16(j+1), every exponent <= 0 (the gate-magnitude law).  The row side
//    prescales the thread's own source column k[s,d] 2^(g_e(j) - g_s) on the fly and
//    reads the dA rows of the target block four columns per 16-byte load; the column
//    side does the mirror through the source block's end boundary.
//  * then the diagonal 16x16 blocks with one exp2 per (r, s, d), two source rows at a
//    time in packed FP32x2, rows in descending order so each row is final (and
//    written) as soon as it is processed.
//  * db[r] = sum_d acck[r,d] k[r,d]: a transposed warp reduction of 8 rows at a time,
//    then a fixed-order sum over the four warps of the sub-block (deterministic).
#include "kda_intra_tc.cuh"

namespace kda {
namespace fp32impl {
namespace {

using namespace tcimpl;

// Unlike the tensor-core kernel, no per-unit MMA couples the warps here, so the four
// sub-block groups may drift up to a unit apart: the unit-done counters are per stage
// and the db partials are double-buffered by unit parity.
constexpr int F_DBP = 2 * STAGE_BYTES;  // db partials f32 [2][4][64]
constexpr int F_FULL = F_DBP + 2048;    // 2 stage-full mbarriers
constexpr int F_CNT = F_FULL + 16;      // unit-done counter per stage
constexpr int F_TOTAL = F_CNT + 16;

template <typename io_t>
__global__ void __launch_bounds__(TC_THREADS, 1)
kda_intra_bwd_fp32_kernel(const __grid_constant__ TmaMaps tm, const float *__restrict__ beta,
                          float *dq, float *dk, float *db, float *dg, int T, int H,
                          long long units, const Extras ex) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int i = tid >> 7;  // sub-block, warp-uniform
    const int d = tid & 127;
    const int r0 = i * BC;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + F_FULL);
    uint32_t *done_count = reinterpret_cast<uint32_t *>(smem + F_CNT);
    float *sdbp = reinterpret_cast<float *>(smem + F_DBP);
    const long long stride = gridDim.x;

    if (tid == 0) {
        tc::mbar_init(&full[0], FULL_ARRIVALS);
        tc::mbar_init(&full[1], FULL_ARRIVALS);
        done_count[0] = done_count[1] = 0u;
        tc::prefetch_tmap(&tm.q);
        tc::prefetch_tmap(&tm.k);
        tc::prefetch_tmap(&tm.g);
#pragma unroll
        for (int t = 0; t < NBLK; ++t) {
            tc::prefetch_tmap(&tm.daqk[t]);
            tc::prefetch_tmap(&tm.dakk[t]);
        }
    }
    __syncthreads();
    if (warp == 0) {  // the first two units of this CTA
        const long long u0 = blockIdx.x;
        if (u0 < units) load_unit<false>(smem, &full[0], nullptr, tm, beta, u0, T, H, ex, lane);
        if (u0 + stride < units)
            load_unit<false>(smem + STAGE_BYTES, &full[1], nullptr, tm, beta, u0 + stride, T, H,
                             ex, lane);
    }

    bool ok = true;
    int it = 0;
    // head of the current unit, advanced by stride mod H; u = q H + h makes the unit's
    // first [token * H + head] row 64 u - 63 h, with no division per unit
    const unsigned dhh = (unsigned)stride % (unsigned)H;
    unsigned hh = (unsigned)blockIdx.x % (unsigned)H;
    for (long long u = blockIdx.x; u < units;
         u += stride, ++it, hh = hh + dhh >= (unsigned)H ? hh + dhh - (unsigned)H : hh + dhh) {
        const int sidx = it & 1;
        unsigned char *st = smem + sidx * STAGE_BYTES;
        ok &= tc::mbar_wait(&full[sidx], (uint32_t)(it >> 1) & 1u, SPIN_LIMIT);

        const float *sg = reinterpret_cast<const float *>(st + ST_G);
        const io_t *sq = reinterpret_cast<const io_t *>(st + ST_Q);
        const io_t *sk = reinterpret_cast<const io_t *>(st + ST_K);
        const float *sbeta = reinterpret_cast<const float *>(st + ST_BETA);
        const float *daq = reinterpret_cast<const float *>(st + ST_DQ);
        const float *dak = reinterpret_cast<const float *>(st + ST_DK);
        // element (n, k) of a 16x16 dA block sits at (k/4)*64 + (n/8)*32 + (n%8)*4 + k%4
        auto rowoff = [](const int n) { return (n >> 3) * 32 + (n & 7) * 4; };

        float2 g2[BC / 2], k2[BC / 2];  // this thread's column of its block, row pairs
#pragma unroll
        for (int m = 0; m < BC / 2; ++m) {
            g2[m] = make_float2(sg[(r0 + 2 * m) * KD + d], sg[(r0 + 2 * m + 1) * KD + d]);
            k2[m] = make_float2(to_f32(sk[(r0 + 2 * m) * KD + d]),
                                to_f32(sk[(r0 + 2 * m + 1) * KD + d]));
        }
#define KDA_EL(arr, r) (((r) & 1) ? arr[(r) >> 1].y : arr[(r) >> 1].x)

        // ---- row side: target block i, source blocks j < i ----
        float accq[BC], acck[BC];
#pragma unroll
        for (int r = 0; r < BC; ++r) accq[r] = acck[r] = 0.f;
        if (i > 0) {
            // packed FP32x2 partial sums over even / odd source columns
            float2 pq[BC], pk[BC];
#pragma unroll
            for (int r = 0; r < BC; ++r) pq[r] = pk[r] = make_float2(0.f, 0.f);
            for (int j = 0; j < i; ++j) {
                const float ge = sg[BC * (j + 1) * KD + d];
                const float cj = (j == i - 1) ? 1.f : ex2(g2[0].x - ge);  // 2^(g_16i - g_e(j))
                const float *bq = daq + dablk(i, j) * 256;
                const float *bk = dak + dablk(i, j) * 256;
#pragma unroll 2
                for (int c4 = 0; c4 < 4; ++c4) {
                    float kv[4];
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const int s = BC * j + 4 * c4 + x;
                        kv[x] = to_f32(sk[s * KD + d]) * ex2(ge - sg[s * KD + d]) * cj;
                    }
                    const float2 k01 = make_float2(kv[0], kv[1]), k23 = make_float2(kv[2], kv[3]);
#pragma unroll
                    for (int r = 0; r < BC; ++r) {
                        const float4 aq = *reinterpret_cast<const float4 *>(bq + c4 * 64 + rowoff(r));
                        const float4 ak = *reinterpret_cast<const float4 *>(bk + c4 * 64 + rowoff(r));
                        pq[r] = __ffma2_rn(make_float2(aq.z, aq.w), k23, __ffma2_rn(make_float2(aq.x, aq.y), k01, pq[r]));
                        pk[r] = __ffma2_rn(make_float2(ak.z, ak.w), k23, __ffma2_rn(make_float2(ak.x, ak.y), k01, pk[r]));
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < BC; ++r) {
                accq[r] = pq[r].x + pq[r].y;
                acck[r] = pk[r].x + pk[r].y;
            }
#pragma unroll
            for (int r = 1; r < BC; ++r) {  // 2^(g_r - g_16i); 1 for r = 0
                const float b = ex2(KDA_EL(g2, r) - g2[0].x);
                accq[r] *= b;
                acck[r] *= b;
            }
        }

        // ---- column side: source block i, target blocks j > i ----
        float2 dkt2[BC / 2];
#pragma unroll
        for (int m = 0; m < BC / 2; ++m) dkt2[m] = make_float2(0.f, 0.f);
        if (i < NBLK - 1) {
            const float ge = sg[(r0 + BC) * KD + d];
            for (int j = i + 1; j < NBLK; ++j) {
                const float gb = sg[BC * j * KD + d];
                const float cj = (j == i + 1) ? 1.f : ex2(gb - ge);  // 2^(g_16j - g_e(i))
                const float *bq = daq + dablk(j, i) * 256;
                const float *bk = dak + dablk(j, i) * 256;
#pragma unroll 4
                for (int r = 0; r < BC; ++r) {
                    const int rr = BC * j + r;
                    const float f = ex2(sg[rr * KD + d] - gb) * cj;
                    const float qb = to_f32(sq[rr * KD + d]) * f;
                    const float kbb = sbeta[rr] * to_f32(sk[rr * KD + d]) * f;
                    const float2 qb2 = make_float2(qb, qb), kb2 = make_float2(kbb, kbb);
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const float4 aq = *reinterpret_cast<const float4 *>(bq + c4 * 64 + rowoff(r));
                        const float4 ak = *reinterpret_cast<const float4 *>(bk + c4 * 64 + rowoff(r));
                        dkt2[2 * c4] = __ffma2_rn(make_float2(aq.x, aq.y), qb2,
                                                  __ffma2_rn(make_float2(ak.x, ak.y), kb2, dkt2[2 * c4]));
                        dkt2[2 * c4 + 1] = __ffma2_rn(make_float2(aq.z, aq.w), qb2,
                                                      __ffma2_rn(make_float2(ak.z, ak.w), kb2, dkt2[2 * c4 + 1]));
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < BC / 2; ++m)  // 2^(g_e(i) - g_s)
                dkt2[m] = __fmul2_rn(dkt2[m], make_float2(ex2(ge - g2[m].x), ex2(ge - g2[m].y)));
        }

        float *dbp = sdbp + (it & 1) * NBLK * BT;
        // ---- diagonal block, rows in descending order; each row is final once done ----
        const float *dgq = daq + dablk(i, i) * 256;
        const float *dgk = dak + dablk(i, i) * 256;
        const float2 neg1 = make_float2(-1.f, -1.f);
        const size_t urow0 = (size_t)64 * (size_t)u - (size_t)63 * hh;
        const size_t obase = (urow0 + (size_t)r0 * H) * KD + d;
        const uint32_t hk = (uint32_t)H * KD;
        float dbv[BC];
        auto diag_row = [&](const int r) {
            const float gv = KDA_EL(g2, r), kv = KDA_EL(k2, r);
            const float qv = to_f32(sq[(r0 + r) * KD + d]);
            const float kbr = sbeta[r0 + r] * kv;
            const float2 grr = make_float2(gv, gv), qq = make_float2(qv, qv),
                         kb2 = make_float2(kbr, kbr);
            float2 aacc = make_float2(0.f, 0.f), kacc = make_float2(0.f, 0.f);
            const int roff = rowoff(r);
            // pairs (2m, 2m+1) cover s < r; for odd r the last pair is (r-1, r) and
            // carries the diagonal term (E = 1, dAkk[r][r] outside the support -> 0)
#pragma unroll
            for (int c = 0; c < (r + 3) / 4; ++c) {
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
        auto out_row = [&](const int r) {  // row r is final: dq, dk, dg
            const int row = r0 + r;
            const float qv = to_f32(sq[row * KD + d]);
            const float kv = KDA_EL(k2, r), dkv = KDA_EL(dkt2, r);
            const float pk = __fmul_rn(sbeta[row], acck[r]);
            const size_t off = obase + (size_t)((uint32_t)r * hk);
            float vq = accq[r], vk = fmaf(sbeta[row], acck[r], dkv);
            float vg = __fmul_rn(LN2, fmaf(qv, accq[r], __fmul_rn(__fsub_rn(pk, dkv), kv)));
            if (!ok) vq = vk = vg = __int_as_float(0x7fc00000);
            if (dbg_ok(ex.dbg, off, ex.nrows * KD, DBG_STORE)) {
                dq[off] = vq;
                dk[off] = vk;
                dg[off] = vg;
            }
            dbv[r] = ok ? acck[r] * kv : __int_as_float(0x7fc00000);
        };
        // db over 8 rows: transpose-reduce across the warp's lanes (lane l ends with
        // row (l>>2)&7), then a fixed-order sum over the sub-block's 4 warps
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
            if ((lane & 3) == 0) dbp[(warp & 3) * BT + r0 + rbase + (lane >> 2)] = v[0];
        };
        // rows 15..8: the diagonal first, then their outputs; then rows 7..0 one by one
#pragma unroll
        for (int r = BC - 1; r >= BC / 2; --r) diag_row(r);
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
        if ((warp & 3) == 0 && lane < BC) {
            const int row = r0 + lane;
            const size_t bi = urow0 + (size_t)row * H;
            if (dbg_ok(ex.dbg, bi, ex.nrows, DBG_STORE))
                db[bi] = (dbp[row] + dbp[BT + row]) + (dbp[2 * BT + row] + dbp[3 * BT + row]);
        }

        // ---- unit done: the last warp releases the stage and refills it ----
        __syncwarp();
        uint32_t prev = 0;
        if (lane == 0) prev = tc::atomic_add_acq_rel_smem(done_count + sidx, 1u);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if ((prev % TC_WARPS) == TC_WARPS - 1 && u + 2 * stride < units) {
            tc::fence_proxy_async_smem();
            load_unit<false>(st, &full[sidx], nullptr, tm, beta, u + 2 * stride, T, H, ex, lane);
        }
    }
    dbg_flag(ex.dbg, !ok, DBG_WAIT);
}

template <typename io_t>
cudaError_t launch_typed(const BwdArgs &a, cudaStream_t stream) {
    auto kern = kda_intra_bwd_fp32_kernel<io_t>;
    static volatile int smem_set[kMaxDev];
    int nsm = 0, dev = 0;
    cudaError_t e = num_sms(&nsm, &dev);
    if (e != cudaSuccess) return e;
    if ((e = smem_limit_once(kern, F_TOTAL, dev, smem_set)) != cudaSuccess) return e;
    TmaMaps tm;
    if ((e = make_maps(a, &tm)) != cudaSuccess) return e;
    Extras ex = {};
    ex.G = 1;
    ex.dbg = a.dbg;
    ex.nrows = (size_t)a.B * a.T * a.H;
    const long long units = (long long)a.B * a.H * (a.T / BT);
    const unsigned grid = (unsigned)(units < nsm ? units : nsm);
    kern<<<grid, TC_THREADS, F_TOTAL, stream>>>(tm, a.beta, (float *)a.dq, (float *)a.dk, a.db,
                                                a.dg, a.T, a.H, units, ex);
    return cudaGetLastError();
}

}  // namespace
}  // namespace fp32impl

cudaError_t launch_intra_fp32(const BwdArgs &a, cudaStream_t stream) {
    return a.fp16 ? fp32impl::launch_typed<__half>(a, stream)
                  : fp32impl::launch_typed<__nv_bfloat16>(a, stream);
}

}  // namespace kda
