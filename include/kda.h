/*
 * libkda -- intra-chunk backward of chunked KDA (Kimi Delta Attention, the gated
 * delta rule with a per-channel gate) on sm_103a.
 *
 * What it computes (bwd_intra page: the module docstring of kernel_fun/kda/_kernels/
 * bwd_intra.py, its diagonal and epilogue loops, and the host wrapper's tensor
 * contract).  Tokens are cut into chunks of KDA_BT = 64; a "unit" is one
 * (batch b, head h, chunk c).  Inside a unit, with rows r, s in [0, 64), channels
 * d in [0, 128) and E[r,s,d] = 2^(g[r,d] - g[s,d]):
 *
 *   Aqk[r,s] = sum_d q[r,d] k[s,d] E[r,s,d]             (s <= r)
 *   Akk[r,s] = beta[r] * sum_d k[r,d] k[s,d] E[r,s,d]   (s <  r)
 *
 * Given the upstream gradients dAqk and dAkk, the library returns the gradients
 * of L = sum dAqk*Aqk + sum dAkk*Akk with respect to q, k, beta and g:
 *
 *   dq[r]   = sum_{s<=r} dAqk[r,s] k[s] E[r,s]
 *   dk[t]   = beta[t] sum_{s<t} dAkk[t,s] k[s] E[t,s]
 *             + sum_{r>=t} (dAqk[r,t] q[r] + [r>t] dAkk[r,t] beta[r] k[r]) E[r,t]
 *   db[r]   = sum_{s<r} dAkk[r,s] sum_d k[r,d] k[s,d] E[r,s,d]
 *   dg[t]   = ln2 * ( q[t] (dq[t]) + (beta[t] acck[t] - dkt[t]) k[t] )
 *             where acck[t] = sum_{s<t} dAkk[t,s] k[s] E[t,s] and dkt[t] is the
 *             second line of dk[t]  (all products per channel d)
 *
 * dg is the gradient with respect to g exactly as passed (a log2 cumulative gate):
 * it is the bwd_intra page's epilogue value times ln2.  A caller whose gate lives
 * in natural-log units (g_nat = g * ln2) gets dL/dg_nat as dg / ln2.
 *
 * Supported shapes: K = 128 (head dimension), chunk 64; fixed-length sequences with
 * T a multiple of 64, or (kda_intra_bwd_ex only) variable-length sequences packed
 * along T and described by cu_seqlens.  g must be the inclusive chunk-local
 * cumulative sum of per-step log2 gates that are <= 0 (non-increasing inside each
 * chunk): every exponent the kernels evaluate is then <= 0.
 *
 * Memory: every pointer is caller-owned DEVICE memory (except the *_host entry
 * point), contiguous row-major, 16-byte aligned, and must not overlap another
 * argument:
 *   q, k        [B, T, H, 128]  bf16 or fp16 (qk_dtype)
 *   g           [B, T, H, 128]  fp32
 *   beta        [B, T, H]       fp32
 *   dAqk, dAkk  [B, T, H, 64]   fp32; row = token, column = source index inside the
 *                               token's chunk.  Entries outside the support (dAqk
 *                               above the diagonal, dAkk on or above it) are ignored.
 *   dq, dk, dg  [B, T, H, 128]  fp32 outputs, fully overwritten
 *   db          [B, T, H]       fp32 output, fully overwritten
 *
 * Calls are asynchronous on `stream` (0 = the legacy default stream): no host
 * synchronisation and no device allocation happens inside.  Inputs are not modified.
 * Argument errors are reported before anything is launched; no call aborts the
 * process.
 *
 * Stalled pipelines: every wait of a kernel on its own copies or tensor-core work is
 * bounded (about 4M polls).  A wait that gives up does not hang or trap: the kernel
 * writes NaN into the outputs of the unit it was working on and carries on.  The call
 * has already returned KDA_OK when this happens (the status only covers the arguments
 * and the launch), so in the normal build a stalled pipeline is seen only as NaN
 * outputs, which NaN or Inf inputs can also produce.  The bounds-checked debug build
 * (kda_debug_set_flags below) also sets KDA_DBG_WAIT in its flag word, which tells the
 * two apart.  No valid input makes a wait give up on a healthy GPU.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * ABI versions (kda_abi_version() returns the loaded library's):
 *   9  kda_intra_bwd_opts_t gains split_tf32 (appended; the struct grew)
 *   8  kda_intra_bwd_host_static, KDA_HOST_STATIC_MAX_BYTES, KDA_ERR_TOO_LARGE
 *   7  kda_debug_checks, kda_debug_set_flags (the bounds-checked debug build)
 *   6  kda_intra_bwd_opts_t gains factor_diag (appended; the struct grew)
 *   5  kda_intra_fwd_ex and kda_intra_fwd_opts_t
 *   4  kda_intra_fwd
 *   3  variable-length fields of kda_intra_bwd_opts_t (cu_seqlens .. num_chunks)
 *   2  kda_intra_bwd_ex and kda_intra_bwd_opts_t
 *   1  kda_intra_bwd, kda_intra_bwd_fp32, the host entry point, status helpers
 * Option structs only grow at their end, and the library reads sizeof(its own struct)
 * from the pointer it is given.  A caller compiled against an older header would have
 * the library read past the end of its struct, so a caller that passes an option struct
 * must check at start-up that kda_abi_version() equals the KDA_ABI_VERSION it was
 * compiled with (the Python binding refuses to load any other version).
 */
#define KDA_ABI_VERSION 9
#define KDA_BT 64  /* chunk length */
#define KDA_BC 16  /* sub-block length inside a chunk */
#define KDA_K 128  /* head dimension */
#define KDA_MAX_H 65536 /* largest supported head count */

/* Same type as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_NULL = 1,               /* a required pointer is NULL */
    KDA_ERR_SHAPE = 2,              /* B,T,H <= 0, H > KDA_MAX_H, T % 64 != 0, too large;
                                       varlen: B != 1, num_seqs <= 0, num_chunks < 0 */
    KDA_ERR_DTYPE = 3,              /* qk_dtype not KDA_BF16 / KDA_FP16 */
    KDA_ERR_ALIGN = 4,              /* a pointer is not 16-byte aligned */
    KDA_ERR_CUDA = 5,               /* a CUDA runtime call or the launch failed */
    KDA_ERR_UNSUPPORTED_DEVICE = 6, /* current device is not compute capability 10.3 */
    KDA_ERR_OVERLAP = 7,            /* two argument buffers overlap */
    KDA_ERR_WORKSPACE = 8,          /* workspace missing or too small (*_host only) */
    KDA_ERR_OPTION = 9,             /* unsupported option combination (*_ex), or debug
                                       reporting asked of a build without checks */
    KDA_ERR_TOO_LARGE = 10          /* the call needs more scratch than the library's
                                       fixed KDA_HOST_STATIC_MAX_BYTES
                                       (kda_intra_bwd_host_static only) */
} kda_status_t;

typedef enum { KDA_BF16 = 0, KDA_FP16 = 1 } kda_dtype_t;

/*
 * The intra-chunk backward, fast path: 16x16 diagonal sub-blocks on the FP32 pipes
 * with one exp2 per (r, s, d); the cross-sub-block sums factorized through each
 * sub-block's boundary gate (every exp2 argument <= 0) and contracted on the
 * tensor cores in TF32 with FP32 accumulation.  Accuracy: max|err| / max|ref|
 * <= 2e-3 per output tensor against the fp64 definition.
 */
kda_status_t kda_intra_bwd(const void *q, const void *k, const float *g,
                           const float *beta, const float *dAqk, const float *dAkk,
                           float *dq, float *dk, float *db, float *dg,
                           int B, int T, int H, kda_dtype_t qk_dtype,
                           kda_stream_t stream);

/*
 * Same contract, every product and sum in FP32 (the cross-sub-block sums on the
 * FP32 pipes through the same boundary factorization).  Slower; accuracy
 * max|err| / max|ref| <= 1e-4 per output tensor.
 */
kda_status_t kda_intra_bwd_fp32(const void *q, const void *k, const float *g,
                                const float *beta, const float *dAqk, const float *dAkk,
                                float *dq, float *dk, float *db, float *dg,
                                int B, int T, int H, kda_dtype_t qk_dtype,
                                kda_stream_t stream);

/*
 * End-to-end convenience for callers holding HOST buffers: copies the six inputs
 * into `workspace` (device memory of at least kda_intra_bwd_host_workspace_bytes()
 * bytes, caller-owned, 256-byte aligned), runs kda_intra_bwd, and copies the four
 * outputs back into the host buffers.  The work is pipelined over pieces of about
 * 96 MB of input (whole 64-token chunks; beta goes up whole before the first piece
 * and db comes down whole after the last): uploads run on one internal stream,
 * downloads on another and the kernels on `stream`, so both copy directions and the
 * compute overlap; events order it all after earlier work on `stream`, and `stream`
 * waits for the last copy of each direction (also when a call fails midway).  The two
 * internal streams and their events are made by the first call on each device and
 * kept until the process exits; calls from several threads queue their work one call
 * after another on them.  Copies are truly asynchronous only when the host buffers
 * are page-locked.  The call returns once everything is queued: synchronise
 * `stream` before reading the outputs or reusing the inputs.  Host pointers need no
 * particular alignment.
 */
size_t kda_intra_bwd_host_workspace_bytes(int B, int T, int H, kda_dtype_t qk_dtype);

kda_status_t kda_intra_bwd_host(const void *q, const void *k, const float *g,
                                const float *beta, const float *dAqk, const float *dAkk,
                                float *dq, float *dk, float *db, float *dg,
                                int B, int T, int H, kda_dtype_t qk_dtype,
                                void *workspace, size_t workspace_bytes,
                                kda_stream_t stream);

/*
 * kda_intra_bwd_host without a workspace argument, for callers that hold only host
 * buffers and may not allocate device memory: a plugin or FFI caller inside a host
 * application whose device memory is owned by another allocator (a framework's
 * caching pool that has reserved it, a fixed per-process budget), or code on a
 * latency-critical path where cudaMalloc's implicit device synchronisation is not
 * acceptable.  The paper has no counterpart for this entry point; it is a deployment
 * convenience around the same kernel.
 *
 * The device staging buffers live in one array of this library, KDA_HOST_STATIC_MAX_BYTES
 * (32 MiB) of global memory that every GPU on which the library's device code is loaded
 * holds until the process exits.  A call whose staging need,
 * kda_intra_bwd_host_workspace_bytes(B, T, H, qk_dtype), exceeds it returns
 * KDA_ERR_TOO_LARGE before anything is queued.  The need is 3080 bytes per token-head
 * row, so up to B*T*H = 10,880 rows fit (for instance B = 2, T = 1024, H = 4); larger
 * problems take kda_intra_bwd_host with a caller-owned workspace.  The call allocates
 * nothing (no cudaMalloc, no cudaFree, no stream, no event): it queues the six uploads,
 * the kernel and the four downloads, in that order, on `stream` and returns.
 * Synchronise `stream` before reading the outputs or reusing the inputs.
 *
 * The first call on each device looks up the array's device address (with that device
 * current); make that first call before any stream capture on that device.  Every call,
 * on every stream and thread, shares the one array: calls whose work overlaps on the GPU
 * race on it, so order them on one stream (or synchronise between them).  The array keeps
 * the last call's contents; nothing in it needs to start at zero, since each call
 * overwrites every byte it reads.  Same arguments, status codes and accuracy as
 * kda_intra_bwd_host otherwise.
 */
#define KDA_HOST_STATIC_MAX_BYTES 33554432u /* 32 MiB */

kda_status_t kda_intra_bwd_host_static(const void *q, const void *k, const float *g,
                                       const float *beta, const float *dAqk,
                                       const float *dAkk, float *dq, float *dk,
                                       float *db, float *dg, int B, int T, int H,
                                       kda_dtype_t qk_dtype, kda_stream_t stream);

/*
 * Options of kda_intra_bwd_ex.  Zero-initialise, then set what you need; a zeroed
 * struct (or a NULL pointer) gives exactly kda_intra_bwd.  These follow the bwd_intra
 * page's host wrapper and kernel options (its incoming-gradient tensors, fold_dg,
 * emit_bf16 and gva group size).
 *
 *   HV             heads of g, beta, dAqk, dAkk and of every output and *_in tensor;
 *                  q and k keep H heads and value head hv reads q/k head hv / (HV / H)
 *                  (grouped value attention).  0 means HV = H.  Must be a multiple of H.
 *   dq_in, dk_in,  optional [B,T,HV,128] fp32 gradients added in-kernel to dq, dk, dg
 *   dg_in          (NULL = none).  May be the same pointer as the matching output
 *                  (in-place accumulation); any other overlap is rejected.  When dq_in,
 *                  dk_in and (without fold_dg) dg_in are all their outputs, the kernel
 *                  reads none of them: its stores add to them in L2 (red.global.add, one
 *                  rounding as otherwise, but subnormal sums flush to zero), the fastest
 *                  way to accumulate.
 *   db_in          optional [B,T,HV] fp32 added to db; may equal db.
 *   fold_dg        1: dg comes back as its inclusive reverse cumsum inside each
 *                  64-token chunk, out[t] = sum_{t' >= t in t's chunk} dg[t'] (the
 *                  per-step gate's gradient; dg_in is added before the fold).
 *   dqdk_io_dtype  1: dq and dk are written in qk_dtype (round to nearest) instead of
 *                  fp32 -- bitwise the cast of the fp32 result.  Not allowed with HV > H
 *                  (the grouped-head reduction that follows must see fp32 values).
 *   cu_seqlens     variable-length sequences (the host wrapper's cu_seqlens /
 *   chunk_indices  chunk_indices pair).  B must be 1 and T is the packed token count
 *   num_seqs       (any T >= 1).  cu_seqlens: device int32 [num_seqs + 1], sequence n
 *   num_chunks     is tokens [cu_seqlens[n], cu_seqlens[n+1]), 0 = cu_seqlens[0] <=
 *                  ... <= cu_seqlens[num_seqs] <= T.  chunk_indices: device int32
 *                  [num_chunks][2], entry c = (n, j) names chunk j of sequence n, i.e.
 *                  tokens cu_seqlens[n] + 64j ... min(+64, cu_seqlens[n+1]) - 1; chunks
 *                  restart at every sequence start, and a sequence's last chunk may be
 *                  short.  Each unit is then (chunk entry, head); all per-chunk
 *                  definitions above apply to the chunk's valid rows only (g is the
 *                  cumsum restarted at each chunk start, dA rows are indexed from the
 *                  chunk start, fold_dg folds over the valid rows).  Both pointers are
 *                  NULL for fixed-length calls (chunk_indices may also be NULL when
 *                  num_chunks == 0: nothing is launched); the rows of tokens that no entry names
 *                  are left untouched.  The values are read on the device only: an
 *                  entry that names no chunk of cu_seqlens (n out of range, j past the
 *                  sequence's end, a sequence past T) is skipped, so no input value can
 *                  make the kernel access memory outside the argument buffers.
 *   factor_diag    0: every pair of a 16x16 diagonal block takes its own exp2, one per
 *                  (r, s, d), as in kda_intra_bwd.  1: the lower-left 8x8 quadrant of
 *                  each diagonal block (rows 8..15 against sources 0..7 of the block) is
 *                  factorized through the block's row 8, 2^(g_r - g_s) =
 *                  2^(g_r - g_8) * 2^(g_8 - g_s); both exponents are <= 0 (g is
 *                  non-increasing inside a chunk), so nothing can overflow, and the
 *                  quadrant costs four FMAs per (r, s, d) instead of an exp2 and seven
 *                  FP32 operations (about 4% less kernel time).  The result differs
 *                  from the exact form by rounding only; same accuracy contract.
 *   split_tf32     1: the cross-sub-block sums in split TF32 for FP32-level accuracy:
 *                  every tensor-core operand x is cut into hi = tf32(x) and lo = x - hi
 *                  and each product is taken as A_hi B_hi + A_hi B_lo + A_lo B_hi on the
 *                  tensor cores with FP32 accumulation (the dropped A_lo B_lo is about
 *                  2^-22 of the product); the diagonal blocks stay on the FP32 pipes.
 *                  Accuracy max|err| / max|ref| <= 1e-4 per output tensor, as
 *                  kda_intra_bwd_fp32, at about half its time.  Fixed-length sequences
 *                  only, and no other option but HV; anything else is KDA_ERR_OPTION.
 *
 * Runs on the tensor-core path (the same accuracy contract as kda_intra_bwd, except
 * with split_tf32).
 */
typedef struct {
    int HV;
    const float *dq_in;
    const float *dk_in;
    const float *dg_in;
    const float *db_in;
    int fold_dg;
    int dqdk_io_dtype;
    const int *cu_seqlens;
    const int *chunk_indices;
    int num_seqs;
    int num_chunks;
    int factor_diag;
    int split_tf32;
} kda_intra_bwd_opts_t;

kda_status_t kda_intra_bwd_ex(const void *q, const void *k, const float *g,
                              const float *beta, const float *dAqk, const float *dAkk,
                              void *dq, void *dk, float *db, float *dg,
                              int B, int T, int H, kda_dtype_t qk_dtype,
                              const kda_intra_bwd_opts_t *opts, kda_stream_t stream);

/*
 * The intra-chunk forward: the two score matrices whose gradients kda_intra_bwd
 * takes, for every unit (b, h, 64-token chunk) and rows r, s of the chunk,
 *
 *   Aqk[r,s] = sum_d q[r,d] k[s,d] E[r,s,d]             (s <= r, else 0)
 *   Akk[r,s] = beta[r] * sum_d k[r,d] k[s,d] E[r,s,d]   (s <  r, else 0)
 *
 * (same definitions as above).  q, k, g, beta as for kda_intra_bwd; Aqk and Akk are
 * [B, T, H, 64] fp32 device outputs, fully overwritten (zeros outside the support),
 * 16-byte aligned, not overlapping anything else.  Cross-sub-block entries come from
 * TF32 tensor-core products through the boundary factorization (every exp2 argument
 * <= 0), the diagonal 16x16 blocks from FP32 with one exp2 per (r, s, d).
 * Accuracy: max|err| / max|ref| <= 2e-3 per output tensor.  Same shape rules, status
 * codes and asynchrony as kda_intra_bwd.
 */
kda_status_t kda_intra_fwd(const void *q, const void *k, const float *g,
                           const float *beta, float *Aqk, float *Akk,
                           int B, int T, int H, kda_dtype_t qk_dtype,
                           kda_stream_t stream);

/*
 * Options of kda_intra_fwd_ex (zero-initialise; a zeroed struct or NULL gives exactly
 * kda_intra_fwd), with the meanings of kda_intra_bwd_opts_t:
 *   HV             heads of g, beta, Aqk and Akk; q and k keep H heads, and value head
 *                  hv reads q/k head hv / (HV / H).  0 means HV = H.
 *   cu_seqlens,    variable-length sequences packed along T (B == 1, any T >= 1):
 *   chunk_indices, the same tables and the same checks as for the backward.  Rows of
 *   num_seqs,      a chunk past its sequence's end take no part in any valid entry and
 *   num_chunks     are not written; tokens no entry names are left untouched.
 */
typedef struct {
    int HV;
    const int *cu_seqlens;
    const int *chunk_indices;
    int num_seqs;
    int num_chunks;
} kda_intra_fwd_opts_t;

kda_status_t kda_intra_fwd_ex(const void *q, const void *k, const float *g,
                              const float *beta, float *Aqk, float *Akk,
                              int B, int T, int H, kda_dtype_t qk_dtype,
                              const kda_intra_fwd_opts_t *opts, kda_stream_t stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char *kda_status_str(kda_status_t status);

/*
 * Bounds-checked debug build.  The same sources compiled with -DKDA_DEBUG_CHECKS (the
 * build script's libkda_debug.so) check every global index their kernels compute
 * (output stores, incoming-gradient and beta reads, chunk-table reads) against the
 * extent of its buffer.  An index out of range sets KDA_DBG_STORE or KDA_DBG_LOAD in a
 * caller-owned device word and the access is skipped; a bounded wait that gives up sets
 * KDA_DBG_WAIT.  Nothing traps or asserts.  TMA tiles need no check: the tensor maps
 * clip them.
 *
 * kda_debug_checks() is 1 in such a build, 0 otherwise.  kda_debug_set_flags(word)
 * makes every later launch of this library report into `word` (device memory, 4 bytes,
 * caller-owned; NULL stops reporting); the library never clears or reads it.  Set it
 * before launching, from one thread.  Returns KDA_ERR_OPTION in a build without checks
 * and KDA_ERR_ALIGN for a word that is not 4-byte aligned.
 */
#define KDA_DBG_STORE 1u
#define KDA_DBG_LOAD 2u
#define KDA_DBG_WAIT 4u
int kda_debug_checks(void);
kda_status_t kda_debug_set_flags(unsigned int *device_word);

/* KDA_ABI_VERSION of the loaded library. */
int kda_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
