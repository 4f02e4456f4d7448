// All-FP32 SIMT kernel for the KDA intra-chunk backward.
//
// One CTA of 512 threads per unit (b, h, 64-token chunk).  Thread (i, d) owns
// sub-block i (rows 16i..16i+15) at channel d for the whole computation:
//
//  * cross-sub-block terms through the per-boundary factorization of the
//    bwd_intra page's module docstring: for r in block i and s in block j < i,
//        2^(g_r - g_s) = 2^(g_r - g_b0(i)) * 2^(g_b0(i) - g_e(j)) * 2^(g_e(j) - g_s)
//    where b0(i) = 16i is block i's first row and e(j) = 16(j+1) the row after
//    block j.  Every factor has a non-positive exponent (the gate-magnitude law),
//    so nothing overflows at any gate magnitude.  k is prescaled by the last
//    factor (kb), q and beta*k by the first (qb, kbb); the middle factor is one
//    value per (i, j, d); the contractions over the 16 rows of a source/target
//    block run on the FP32 pipes here.
//  * diagonal 16x16 blocks computed directly with exactly one exp2 per (r, s, d)
//    (nothing factorized inside a diagonal block); each E[r,s,d] feeds both the
//    row-side sums (dq, the dAkk row sum) and the column-side sum of source row s.
//  * epilogue: dq = accq; dk = beta*acck + dkt; dg = ln2 (q accq + (beta acck - dkt) k);
//    db[r] = sum_d acck[r,d] k[r,d] via a warp butterfly + a fixed-order sum of the
//    four warps covering the row (deterministic).
#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

constexpr int FP32_THREADS = 512;

template <typename io_t>
struct Fp32Smem {
    float g[BT][KD];
    float daqk[BT][BT];   // only the lower 16x16 blocks are loaded and read
    float dakk[BT][BT];
    float kb[3 * BC][KD];   // kb[s][d]       = k[s,d] 2^(g[e(s),d] - g[s,d]),  s < 48
    float qb[3 * BC][KD];   // qb[r-16][d]    = q[r,d] 2^(g[r,d] - g[b0(r),d]), r >= 16
    float kbb[3 * BC][KD];  // kbb[r-16][d]   = beta[r] k[r,d] 2^(same)
    io_t q[BT][KD];
    io_t k[BT][KD];
    float beta[BT];
    float dbpart[4][BT];
};

template <typename io_t>
__global__ void __launch_bounds__(FP32_THREADS, 1)
kda_intra_bwd_fp32_kernel(const io_t *__restrict__ q, const io_t *__restrict__ k,
                          const float *__restrict__ g, const float *__restrict__ beta,
                          const float *__restrict__ dAqk, const float *__restrict__ dAkk,
                          float *__restrict__ dq, float *__restrict__ dk,
                          float *__restrict__ db, float *__restrict__ dg, int T, int H) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Fp32Smem<io_t> &s = *reinterpret_cast<Fp32Smem<io_t> *>(smem_raw);
    const int tid = threadIdx.x;
    const Unit u = decode_unit(blockIdx.x, H, T / BT);

    // ---- load the unit: q, k, g rows and the lower-block part of each dA row ----
    for (int idx = tid; idx < BT * (KD / 8); idx += FP32_THREADS) {
        const int r = idx >> 4, c = idx & 15;
        const size_t off = grow(u, r, T, H) * KD + c * 8;
        cp_async16(&s.q[r][c * 8], q + off);
        cp_async16(&s.k[r][c * 8], k + off);
    }
    for (int idx = tid; idx < BT * (KD / 4); idx += FP32_THREADS) {
        const int r = idx >> 5, c = idx & 31;
        cp_async16(&s.g[r][c * 4], g + grow(u, r, T, H) * KD + c * 4);
    }
    for (int idx = tid; idx < BT * (BT / 4); idx += FP32_THREADS) {
        const int r = idx >> 4, c = idx & 15;
        if (c < ((r >> 4) + 1) * 4) {  // columns up to the end of row r's block
            const size_t off = grow(u, r, T, H) * BT + c * 4;
            cp_async16(&s.daqk[r][c * 4], dAqk + off);
            cp_async16(&s.dakk[r][c * 4], dAkk + off);
        }
    }
    cp_async_commit();
    if (tid < BT) s.beta[tid] = beta[grow(u, tid, T, H)];
    cp_async_wait_all();
    __syncthreads();

    // ---- this thread's column of its own block ----
    const int i = tid >> 7;  // warp-uniform
    const int d = tid & 127;
    const int r0 = i * BC;
    float gr[BC], kr[BC], qr[BC];
#pragma unroll
    for (int r = 0; r < BC; ++r) {
        gr[r] = s.g[r0 + r][d];
        kr[r] = to_f32(s.k[r0 + r][d]);
        qr[r] = to_f32(s.q[r0 + r][d]);
    }

    // ---- prescale (both exponents <= 0) ----
    if (i < NBLK - 1) {
        const float ge = s.g[r0 + BC][d];
#pragma unroll
        for (int r = 0; r < BC; ++r) s.kb[r0 + r][d] = kr[r] * ex2(ge - gr[r]);
    }
    if (i > 0) {
#pragma unroll
        for (int r = 0; r < BC; ++r) {
            const float f = ex2(gr[r] - gr[0]);
            s.qb[r0 - BC + r][d] = qr[r] * f;
            s.kbb[r0 - BC + r][d] = s.beta[r0 + r] * kr[r] * f;
        }
    }
    __syncthreads();

    float accq[BC], acck[BC], dkt[BC];
#pragma unroll
    for (int r = 0; r < BC; ++r) accq[r] = acck[r] = dkt[r] = 0.f;

    // ---- row side: target block i, source blocks j < i; four source columns per
    // 16-byte load of each dA row ----
    for (int j = 0; j < i; ++j) {
        const float cj = (j == i - 1) ? 1.f : ex2(gr[0] - s.g[BC * (j + 1)][d]);
#pragma unroll 1
        for (int s4 = 0; s4 < BC; s4 += 4) {
            const int sc = BC * j + s4;
            float kv[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) kv[x] = s.kb[sc + x][d] * cj;
#pragma unroll
            for (int r = 0; r < BC; ++r) {
                const float4 aq = *reinterpret_cast<const float4 *>(&s.daqk[r0 + r][sc]);
                const float4 ak = *reinterpret_cast<const float4 *>(&s.dakk[r0 + r][sc]);
                accq[r] = fmaf(aq.x, kv[0], fmaf(aq.y, kv[1], fmaf(aq.z, kv[2], fmaf(aq.w, kv[3], accq[r]))));
                acck[r] = fmaf(ak.x, kv[0], fmaf(ak.y, kv[1], fmaf(ak.z, kv[2], fmaf(ak.w, kv[3], acck[r]))));
            }
        }
    }
    if (i > 0) {
#pragma unroll
        for (int r = 0; r < BC; ++r) {
            const float f = ex2(gr[r] - gr[0]);
            accq[r] *= f;
            acck[r] *= f;
        }
    }

    // ---- column side: source block i, target blocks j > i; each dA row segment of
    // the source block read as four 16-byte loads ----
    for (int j = i + 1; j < NBLK; ++j) {
        const float cj = (j == i + 1) ? 1.f : ex2(s.g[BC * j][d] - s.g[r0 + BC][d]);
#pragma unroll 2
        for (int rl = 0; rl < BC; ++rl) {
            const int rr = BC * j + rl;
            const float qv = s.qb[rr - BC][d] * cj;
            const float kv = s.kbb[rr - BC][d] * cj;
#pragma unroll
            for (int s4 = 0; s4 < BC; s4 += 4) {
                const float4 aq = *reinterpret_cast<const float4 *>(&s.daqk[rr][r0 + s4]);
                const float4 ak = *reinterpret_cast<const float4 *>(&s.dakk[rr][r0 + s4]);
                dkt[s4 + 0] = fmaf(aq.x, qv, fmaf(ak.x, kv, dkt[s4 + 0]));
                dkt[s4 + 1] = fmaf(aq.y, qv, fmaf(ak.y, kv, dkt[s4 + 1]));
                dkt[s4 + 2] = fmaf(aq.z, qv, fmaf(ak.z, kv, dkt[s4 + 2]));
                dkt[s4 + 3] = fmaf(aq.w, qv, fmaf(ak.w, kv, dkt[s4 + 3]));
            }
        }
    }
    if (i < NBLK - 1) {
        const float ge = s.g[r0 + BC][d];
#pragma unroll
        for (int sl = 0; sl < BC; ++sl) dkt[sl] *= ex2(ge - gr[sl]);
    }

    // ---- diagonal block: one exp2 per (r, s, d), shared by both sides ----
#pragma unroll
    for (int r = 0; r < BC; ++r) {
        const float aqd = s.daqk[r0 + r][r0 + r];  // s = r: E = 1
        accq[r] = fmaf(aqd, kr[r], accq[r]);
        dkt[r] = fmaf(aqd, qr[r], dkt[r]);
        const float kbr = s.beta[r0 + r] * kr[r];
#pragma unroll
        for (int sl = 0; sl < r; ++sl) {
            const float e = ex2(gr[r] - gr[sl]);
            const float aq = s.daqk[r0 + r][r0 + sl];
            const float ak = s.dakk[r0 + r][r0 + sl];
            const float t = kr[sl] * e;
            accq[r] = fmaf(aq, t, accq[r]);
            acck[r] = fmaf(ak, t, acck[r]);
            dkt[sl] = fmaf(fmaf(aq, qr[r], ak * kbr), e, dkt[sl]);
        }
    }

    // ---- epilogue ----
    const int lane = tid & 31;
    const int wq = (tid >> 5) & 3;
#pragma unroll
    for (int r = 0; r < BC; ++r) {
        const int row = r0 + r;
        const size_t off = grow(u, row, T, H) * KD + d;
        const float pk = s.beta[row] * acck[r];
        dq[off] = accq[r];
        dk[off] = pk + dkt[r];
        dg[off] = LN2 * fmaf(qr[r], accq[r], (pk - dkt[r]) * kr[r]);
        float v = acck[r] * kr[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) s.dbpart[wq][row] = v;
    }
    __syncthreads();
    if (tid < BT)
        db[grow(u, tid, T, H)] =
            (s.dbpart[0][tid] + s.dbpart[1][tid]) + (s.dbpart[2][tid] + s.dbpart[3][tid]);
}

template <typename io_t>
cudaError_t launch_typed(const BwdArgs &a, cudaStream_t stream) {
    const size_t smem = sizeof(Fp32Smem<io_t>);
    auto kern = kda_intra_bwd_fp32_kernel<io_t>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long units = (long long)a.B * a.H * (a.T / BT);
    kern<<<(unsigned)units, FP32_THREADS, smem, stream>>>(
        (const io_t *)a.q, (const io_t *)a.k, a.g, a.beta, a.dAqk, a.dAkk, (float *)a.dq,
        (float *)a.dk, a.db, a.dg, a.T, a.H);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_intra_fp32(const BwdArgs &a, cudaStream_t stream) {
    return a.fp16 ? launch_typed<__half>(a, stream) : launch_typed<__nv_bfloat16>(a, stream);
}

}  // namespace kda
