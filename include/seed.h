/*
 * seed.h — C-ABI of the sink + low-rank recurrent-state decode library (libseed.so).
 *
 * Method: "Shallow Encoding Emits Deep Memories" (SEED).  Each linear-attention
 * or state-space head keeps its d_k x d_v recurrent state as a state sink plus
 * low-rank factors,
 *
 *     S = a vbar^T + U_eff W^T                      (picx.dev summary, Methodology >
 *                                                    SEED Architecture, decode paragraph)
 *
 * where vbar (d_v) is a fixed unit direction per (layer, head), shared by all
 * requests (thelatestinai.com list view, appendix accounting table), a (d_k) is
 * the sink coefficient, and U (d_k x m), W (d_v x m) are the content factors.
 * The page calls the value-side factor V; it is W here.
 *
 * Every decode step reads out and updates each state (list view, Table 1,
 * decode column) with the exact factored update of Lemma 2 (summary, Methodology
 * > Exact Update (Lemma 2)), which appends columns; every T steps the factors are
 * compressed back to rank r (Table 1: "compressed to rank R every W steps"; the
 * pages' R and W are r and T here).
 *
 * Conventions for every call:
 *  - All array pointers are DEVICE pointers owned by the caller; the library
 *    allocates nothing and keeps no state between calls, with one exception:
 *    the fixed 64 MiB device scratch of seed_recompress_noalloc (one array per
 *    device that loads the library, held until the process exits).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream).  Arguments are validated on the host before any launch; on a
 *    validation error nothing is launched and a seed_status code is returned.
 *  - Conditions found on the device (non-finite values, a Jacobi SVD that did
 *    not converge) are written per head to `status[h]` when `status` is not
 *    NULL; read it after synchronising.  0 = OK, otherwise a seed_status code.
 *  - Floating-point vectors (q, k, v, o, a, S, scales, the per-channel gate)
 *    are fp32, contiguous per head, with 16-byte aligned base pointers.
 *    Factors U and W are fp32, bf16 or fp16, rounded on store as
 *    seed_state.rounding says; arithmetic is fp32.  fp16 factors must stay
 *    within its range (|x| < 65504): the library does not rescale them.
 *  - d_k must be 128; d_v must be 128 or 64.  The largest number of factor
 *    columns a head may hold is SEED_MAX_COLUMNS.
 */
#ifndef SEED_H_
#define SEED_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *seed_stream_t;

typedef enum {
  SEED_OK = 0,
  SEED_ERR_INVALID_ARG = 1,      /* NULL pointer, negative size, unknown enum value        */
  SEED_ERR_UNSUPPORTED_SHAPE = 2,/* d_k != 128, d_v not in {64,128}, r > min(d_k,d_v),
                                    r_max + growth*T > SEED_MAX_COLUMNS                    */
  SEED_ERR_CAPACITY = 3,         /* a decode step would exceed r + growth*T columns        */
  SEED_ERR_ALIGNMENT = 4,        /* a pointer is not 16-byte aligned                       */
  SEED_ERR_CUDA = 5,             /* a CUDA launch failed                                    */
  SEED_ERR_NOT_CONVERGED = 6,    /* device, per head: Jacobi SVD hit its sweep limit        */
  SEED_ERR_NONFINITE = 7,        /* device, per head: a non-finite value was produced       */
  SEED_ERR_TIMEOUT = 8           /* device, per head: a bounded wait for a copy gave up     */
} seed_status;

typedef enum {
  SEED_GDN = 0,    /* Gated DeltaNet:       S' = alpha (I - beta k k^T) S + beta k v^T          */
  SEED_KDA = 1,    /* Kimi Delta Attention: S' = diag(alpha) (I - beta k k^T) S + beta k v^T    */
  SEED_MAMBA2 = 2  /* Mamba-2:              S' = exp(dt A) S + dt B x^T  (N = d_k, P = d_v)      */
} seed_variant;

typedef enum { SEED_F32 = 0, SEED_BF16 = 1, SEED_F16 = 2 } seed_dtype;

/* How a factor element is rounded when it is stored in a 16-bit factor dtype
 * (picx.dev summary, Practical implications: 16-bit factors; list view, the
 * drift table by storage format and rounding).  32-bit factors ignore it. */
typedef enum {
  SEED_ROUND_NEAREST = 0,    /* round to nearest even                                 */
  SEED_ROUND_STOCHASTIC = 1  /* up with probability (x - lo) / (hi - lo), so that the
                                stored value is x on average; the random bits come
                                from Philox4x32-10 keyed by seed_state.sr_seed, with
                                the pool column and element as counter               */
} seed_rounding;

#define SEED_MAX_COLUMNS 64

/*
 * The factored state of n_heads heads.  Plain struct, filled by the caller.
 *
 * Column layout: head h owns columns [col0(h), col0(h) + cap(h)) of the column
 * pools U, W (and of `scale` for GDN/Mamba-2), where
 *     cap(h)  = rank(h) + growth * T,   growth = 2 for KDA, 1 otherwise,
 *     col0(h) = col_offset[h]           if col_offset != NULL (ragged ranks),
 *             = h * (r_max + growth * T) otherwise (r_max = r when rank == NULL).
 * Column j of head h is contiguous: U + (col0(h) + j) * d_k elements, W +
 * (col0(h) + j) * d_v elements.  The head currently holds
 *     m(h) = rank(h) + growth * steps_since_compress
 * columns.
 *
 * The effective key factor is U_eff = U diag(scale[col0 .. col0+m)) for GDN and
 * Mamba-2 (the gate products of the existing columns are kept as column scales,
 * so columns are never rewritten), and U_eff = diag(D_h) U for KDA with
 * D_h = scale + h * d_k (a per-head row scale that carries the per-channel gate).
 */
typedef struct {
  int32_t variant;               /* seed_variant                                          */
  int32_t factor_dtype;          /* seed_dtype of U and W                                 */
  int32_t n_heads;               /* >= 0; 0 makes every call a no-op                      */
  int32_t d_k;                   /* 128 (Mamba-2: state size N)                           */
  int32_t d_v;                   /* 128 or 64 (Mamba-2: head dimension P)                 */
  int32_t T;                     /* steps between compressions, >= 1                      */
  int32_t r;                     /* rank kept by compressions when rank == NULL            */
  int32_t r_max;                 /* an upper bound of rank[] (== r when rank == NULL)     */
  int32_t steps_since_compress;  /* s: advanced by seed_decode_step on success, reset to 0
                                    by seed_compress_dense and seed_recompress            */
  int32_t rounding;              /* seed_rounding of stored 16-bit factor elements         */
  const int32_t *rank;           /* [n_heads] per-head rank, or NULL                       */
  const int64_t *col_offset;     /* [n_heads] first column of each head, or NULL           */
  float *a;                      /* [n_heads][d_k] sink coefficients                       */
  void *U;                       /* [columns][d_k] key-side factor, factor_dtype           */
  void *W;                       /* [columns][d_v] value-side factor, factor_dtype         */
  float *scale;                  /* GDN, Mamba-2: [columns] column scales;
                                    KDA: [n_heads][d_k] row scales D                       */
  const float *vbar;             /* [n_dir][d_v] unit sink directions                      */
  const int32_t *vbar_index;     /* [n_heads] direction of each head, or NULL (= h)        */
  int32_t *status;               /* [n_heads] per-head device status, or NULL              */
  uint64_t sr_seed;              /* key of the stochastic-rounding bits: change it from call
                                    to call (e.g. the global step number) for fresh bits; the
                                    same seed and inputs give the same bits                */
  const int32_t *head_order;     /* [n_heads] every head once, grouped by column class, or
                                    NULL (see below)                                       */
  int32_t class_end[4];          /* with head_order: where each column class ends in it    */
} seed_state;

/*
 * Column classes (optional, for ragged ranks).  Head h belongs to class c when
 * its capacity r(h) + growth * T lies in (16c, 16c + 16] (class 0 also takes 0).
 * With head_order != NULL, positions [class_end[c-1], class_end[c]) of
 * head_order (class_end[-1] = 0) list the heads of class c, and class_end[3] =
 * n_heads.  seed_decode_step and the 16-bit paths of seed_recompress_ws /
 * seed_recompress_noalloc then launch once per class, each launch sized for its
 * class (shared-memory stages of 16(c+1) columns) and covering exactly its heads;
 * the results are the same as without the order, head for head.  The host checks
 * that class_end is nondecreasing and ends at n_heads; head_order must list every
 * head once (not checked).  A listed head whose columns exceed its class's size
 * is left untouched by the call that finds it so, with status
 * SEED_ERR_INVALID_ARG.  32-bit factors ignore the order.
 */

/* Columns one head needs: r + growth * T. */
int32_t seed_columns_per_head(int32_t variant, int32_t r, int32_t T);

/*
 * seed_compress_dense — dense states -> sink + rank-r factors.
 * (list view, Table 1: the states that leave the prefill are compressed to the
 * sink plus rank-R factors; summary, Lemma 1: the sink split a = S vbar/|vbar|^2,
 * C = S - a vbar^T.)
 *   S          [n_heads][d_k][d_v] fp32, row-major per head (read only).
 *   st         writes a, the first rank(h) columns of U and W (U = X_r Sigma_r,
 *              W = Y_r from the SVD C = X Sigma Y^T, largest singular values
 *              first; computed as U = C y_k, W = y_k), scales (or D) = 1; sets
 *              st->steps_since_compress = 0.
 *   trunc_err  [n_heads] |C - U W^T|_F, or NULL.
 * Householder QR with column pivoting C P = Q R, then one-sided Jacobi on R^T
 * (R^T J = V Sigma, y = P v), fp32; per-head status 6 if the sweep limit is
 * reached (the factors are still written).
 */
int seed_compress_dense(const float *S, seed_state *st, float *trunc_err, seed_stream_t stream);

/*
 * seed_decode_step — one read-out + exact factored update for every head.
 * (summary, Exact Update (Lemma 2); list view, Table 1: read-out and update of
 * each recurrent state.)  With omega = v.vbar/|vbar|^2 and eps = v - omega vbar:
 *   GDN:     a' = g a + beta (omega - g k.a) k,  U' = [U, k] (scales *= g, new 1),
 *            W' = [W, beta (eps - g W U_eff^T k)],           g = alpha
 *   KDA:     a' = alpha*(a - beta k (k.a)) + beta omega k,  D' = alpha*D,
 *            U' = [U, k/D, k/D'],  W' = [W, -beta W U_eff^T k, beta eps]
 *   Mamba-2: a' = g a + dt omega B,  U' = [U, dt B] (scales *= g),  W' = [W, eps],
 *            g = exp(dt A)
 * and the read-out of the updated state o = S'^T q = vbar (a'.q) + W' U_eff'^T q.
 * The read-out uses the stored (rounded) new columns, so o is exactly the
 * read-out of the state that the factors now hold.
 *   q, k    [n_heads][d_k]  (Mamba-2: C and B)
 *   v       [n_heads][d_v]  (Mamba-2: x)
 *   gate    GDN: alpha [n_heads];  KDA: alpha [n_heads][d_k];  Mamba-2: dt [n_heads]
 *   beta    [n_heads] (GDN, KDA); ignored for Mamba-2 (may be NULL)
 *   A       Mamba-2: [n_dir] indexed like vbar; NULL otherwise
 *   o       [n_heads][d_v] output
 * Returns SEED_ERR_CAPACITY without launching when steps_since_compress >= T.
 * On success increments st->steps_since_compress.
 */
int seed_decode_step(seed_state *st, const float *q, const float *k, const float *v,
                     const float *gate, const float *beta, const float *A, float *o,
                     seed_stream_t stream);

/*
 * seed_recompress — factors back to rank r (list view, Table 1, every T steps;
 * error bound: summary, Open-Loop Error Bound (Corollary 4)).
 * A = U_eff, B = W (m columns each); Householder QR A = Q_a R_a, B = Q_b R_b;
 * core K = R_a R_b^T = X Sigma Y^T, found as K P = Q R (column pivoting) and a
 * one-sided Jacobi on R^T (R^T J = V Sigma, Y = P V); keep the rank(h) largest:
 * U = Q_a K Y_r (= Q_a X_r Sigma_r), W = Q_b Y_r; scales (or D) = 1; a unchanged.
 *   trunc_err  [n_heads] sqrt(sum of the discarded sigma^2), or NULL.
 * Sets st->steps_since_compress = 0.  Per-head status 6 if the sweep limit is hit.
 */
int seed_recompress(seed_state *st, float *trunc_err, seed_stream_t stream);

/*
 * seed_recompress_ex — seed_recompress that also reports, per head, the number
 * of Jacobi sweeps it ran (sweeps [n_heads] int32, or NULL; -1 where the sweep
 * limit was reached).  Used to count the work of a recompression.
 */
int seed_recompress_ex(seed_state *st, float *trunc_err, int32_t *sweeps, seed_stream_t stream);

/*
 * seed_recompress_workspace_bytes — size of the device workspace that
 * seed_recompress_ws needs to recompress `heads` heads per group, at the
 * state's full capacity (r_max + growth*T columns per head), so that one
 * allocation serves every call on this state (it depends on the factor dtype:
 * about 24 KB a head at 48 columns for 16-bit factors, 49 KB for 32-bit).
 * Written to *bytes.
 * Returns a seed_status code (SEED_ERR_INVALID_ARG for heads < 1 or bytes NULL).
 */
int seed_recompress_workspace_bytes(const seed_state *st, int32_t heads, int64_t *bytes);

/*
 * seed_recompress_ws — the recompression of seed_recompress_ex in three phases
 * that pass their intermediates through a caller-provided workspace; the same
 * truncation (the rank(h) largest singular values of U_eff W^T kept, U = X_r
 * Sigma_r, W orthonormal, scales reset), agreeing with seed_recompress_ex to
 * rounding, not bit for bit.  The route depends on the factor dtype:
 *   32-bit factors: (1) per head, Householder QR of U_eff and of W (W's
 *     reflectors kept) and the core K = R_a R_b^T; (2) per head, the Jacobi
 *     SVD of K; (3) per head and factor, U = U_eff (R_b^T Y_r) (= Q_a K Y_r) and
 *     W = Q_b Y_r by W's reflectors applied to [Y_r; 0]; no Q is formed.
 *   16-bit factors: (1) per head, the Gram matrix W^T W on the tensor cores, its
 *     Cholesky R_b^T R_b, B = U_eff R_b^T (tensor cores) and M = B^T B; (2) per
 *     head, the eigenvectors Y of M (pivoted Cholesky, then one-sided Jacobi);
 *     (3) per head and factor, U = U_eff R_b^T Y_r and W = W R_b^{-1} Y_r on the
 *     tensor cores.  Its resolution of nearly dependent columns of W, about
 *     1e-3 of their norm, is finer than the rounding of a stored 16-bit column.
 * Each phase has its own layout, so more heads are resident per SM than in the
 * single kernel of seed_recompress.
 *   workspace        DEVICE memory owned by the caller, 16-byte aligned
 *   workspace_bytes  its size; heads are processed in groups of as many as it
 *                    holds (SEED_ERR_INVALID_ARG if not even one); groups of at
 *                    least 8 x the SM count keep every SM busy
 * The workspace may not be used by any other call until this one has finished
 * on `stream`.  Sets st->steps_since_compress = 0.
 */
int seed_recompress_ws(seed_state *st, float *trunc_err, int32_t *sweeps, void *workspace,
                       int64_t workspace_bytes, seed_stream_t stream);

/*
 * seed_recompress_noalloc — seed_recompress_ws on a scratch array that the
 * library holds in device memory, for callers that cannot call cudaMalloc to
 * provide a workspace: a host runtime that owns no CUDA allocator of its own,
 * or a serving loop that must not allocate (allocation can synchronise the
 * device and fragment a pool sized in advance) on the decode path.  The pages
 * have no counterpart of this call: it is plumbing of this library.
 *   The scratch is a fixed 64 MiB per device, reserved when the library's
 *   kernels are loaded on that device; all heads are recompressed in one group,
 *   so a state whose heads need more than that is rejected with
 *   SEED_ERR_UNSUPPORTED_SHAPE before any CUDA call; use seed_recompress_ws for
 *   such states.  The need is n_heads x the per-head workspace at the current
 *   column count m = r_max + growth * steps_since_compress;
 *   seed_recompress_workspace_bytes(st, 1) reports the per-head size at full
 *   capacity (steps_since_compress = T), an upper bound of it.
 *   All calls on a device share the one scratch: two calls that may overlap
 *   (on different streams or host threads) race on it and must be ordered by
 *   the caller.
 *   Every call looks the scratch's device address up on the host
 *   (cudaGetSymbolAddress, no allocation) and sets kernel attributes; the first
 *   call on a device also loads the library's kernels there, so make it before
 *   any stream capture.
 * Results are bit-identical to seed_recompress_ws.  SEED_ERR_CUDA if the
 * scratch cannot be found.  Sets st->steps_since_compress = 0.
 */
int seed_recompress_noalloc(seed_state *st, float *trunc_err, int32_t *sweeps, seed_stream_t stream);

/*
 * seed_materialize — S = a vbar^T + U_eff W^T for every head (tests, export).
 *   S_out  [n_heads][d_k][d_v] fp32, row-major per head.
 */
int seed_materialize(const seed_state *st, float *S_out, seed_stream_t stream);

/*
 * seed_dense_decode_step — the original model's dense-state step, used as the
 * in-run comparison (list view, abstract: every decode step loads and stores
 * whole recurrent states).  Same recurrences and read-out as above, on a dense
 * fp32 state that is read and written once:
 *   S          [n_heads][d_k][d_v] fp32, updated in place
 *   q,k,v,gate,beta,A,o   as in seed_decode_step
 *   dir_index  [n_heads] index into A (Mamba-2), or NULL (= h)
 */
int seed_dense_decode_step(int32_t variant, int32_t n_heads, int32_t d_k, int32_t d_v, float *S,
                           const float *q, const float *k, const float *v, const float *gate,
                           const float *beta, const float *A, const int32_t *dir_index, float *o,
                           seed_stream_t stream);

/* Text of a seed_status code. */
const char *seed_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SEED_H_ */
