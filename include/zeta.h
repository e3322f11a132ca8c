/*
 * zeta.h -- C ABI of the ZETA hot path on one GB300 (sm_103a).
 *
 * Method: "ZETA: Leveraging Z-order Curves for Efficient Top-k Attention"
 * (arXiv 2501.14577).  Queries and keys live in a low-dimensional space
 * (d_K = 3 by default), are quantised and bit-interleaved into one-dimensional
 * Z-order (Morton) codes, keys are sorted for every chunk-aligned causal prefix,
 * each query takes the k keys around its insertion rank in that order, and the
 * selected keys plus the query's own-chunk causal keys are combined with the
 * Adaptive Cauchy-softmax into a weighted sum of values.
 *
 * Conventions shared by every call
 *   - Every tensor is a contiguous row-major device array with the batch and
 *     head dimensions leading: [B, H, N, ...].  One (b, h) pair is a "slice";
 *     slices are independent except that the gamma gradient sums over b.
 *   - The caller owns and allocates every buffer, workspaces included (sizes
 *     come from the *_bytes / *_entries queries).  The library never allocates,
 *     never synchronises the stream and keeps no global state.
 *   - Work is enqueued on the given stream (0 = legacy default stream).  A
 *     returned ZETA_OK means the arguments were valid and the launches were
 *     enqueued; device-side findings are written to *dev_status when a status
 *     word is given (read it after synchronising).
 *   - Arguments are checked before anything is launched.  An empty problem
 *     (B*H*N == 0) is valid and launches nothing.
 *   - Code width: codes are uint32 when d_K*bits <= 32, else uint64.
 *   - Limits: 1 <= d_K <= 8, 1 <= bits <= 24, d_K*bits <= 64, C >= 1, C | N,
 *     1 <= k <= C, 1 <= d_V <= 256, N < 2^31; zeta_sort_chunks also needs
 *     N / C <= 1024.
 */
#ifndef ZETA_H
#define ZETA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ZETA_OK = 0,
    ZETA_ERR_INVALID_ARG = 1,     /* null pointer, bad size, C not dividing N, ...  */
    ZETA_ERR_UNSUPPORTED = 2,     /* valid request outside the implemented limits   */
    ZETA_ERR_WORKSPACE = 3,       /* workspace missing or smaller than required      */
    ZETA_ERR_CUDA = 4,            /* a launch failed (cudaGetLastError was not 0)    */
    ZETA_ERR_DEVICE_TIMEOUT = 5,  /* a bounded device wait gave up (status word)     */
    ZETA_ERR_BOUNDS = 6           /* an index outside its legal range (status word)  */
} zeta_status_t;

typedef enum { ZETA_F32 = 0, ZETA_BF16 = 1 } zeta_dtype_t;

/* Weight kernel of the attended set, in the low two bits of
 * zeta_problem_t.flags (d2 = |q_i - k_j|^2, a_ij = w_ij / s_i, s_i = sum_j w_ij):
 *   ZETA_W_CAUCHY      w = 1 / (1 + d2 / gamma^2): the method's Adaptive
 *                      Cauchy softmax (OpenReview reply A2 "Discussion on its
 *                      robustness").
 *   ZETA_W_SOFTMAX     w = exp(-(d2 - m_i) / gamma^2), m_i the smallest d2 of
 *                      query i's attended set: the usual softmax of
 *                      -d2 / gamma^2 ("negative Euclidean with traditional
 *                      softmax", reply A3 "Justification for Euclidean
 *                      Distance Claim"); rowsum_i is s_i with that shift.
 *   ZETA_W_INV_EUCLID  w = 1 / sqrt(d2 + 1e-12): inverse Euclidean distance
 *                      (same reply); gamma does not enter, dgamma is 0.
 * The squared distance inside the softmax and the 1e-12 guard are readings:
 * the pages name the kernels without formulas. */
typedef enum { ZETA_W_CAUCHY = 0, ZETA_W_SOFTMAX = 1, ZETA_W_INV_EUCLID = 2 } zeta_weight_t;

/* Problem statement: B batch, H heads, N tokens, d_K query/key width, d_V value
 * width, k window length, C chunk length, bits grid bits per coordinate,
 * v_dtype element type of v / out / dout / dv, flags: bits 0-1 the weight
 * kernel (zeta_weight_t), other bits reserved (pass 0).
 * These are the quantities the pages use to state the method: the 12-bit grid
 * and d_K = 3 (OpenReview reply A2 "Clarification of Binary Expansion and
 * Precision"), the chunk count and d_K = d_Q = 3 (reply A2 "Details about
 * experiments"), k and the trainable gamma (reply A2 "Discussion on its
 * robustness"). */
typedef struct {
    int32_t B, H, N, d_K, d_V, k, C, bits;
    int32_t v_dtype;
    uint32_t flags;
} zeta_problem_t;

/* Bytes per Z-order code (4 or 8); 0 when the problem is invalid. */
size_t zeta_code_bytes(const zeta_problem_t *p);

/* Entries T of the prefix table of one slice: C * n * (n - 1) / 2 with
 * n = N / C.  Prefix c (c = 1..n-1) occupies entries [C*c*(c-1)/2, +c*C).
 * Returns -1 when the problem is invalid. */
int64_t zeta_prefix_entries(const zeta_problem_t *p);

/* Workspace bytes needed by zeta_sort_chunks / zeta_attend_bwd (0 if invalid). */
size_t zeta_sort_workspace_bytes(const zeta_problem_t *p);
size_t zeta_bwd_workspace_bytes(const zeta_problem_t *p);

/* Human-readable name of a status code (static storage). */
const char *zeta_status_string(zeta_status_t s);

/*
 * zeta_encode -- Z-order code of every token.
 * Passage: OpenReview reply A2 "Clarification of Binary Expansion and
 * Precision" (normalise each coordinate to [0, 1], discretise to a grid of
 * 2^bits cells, interleave the bits of the d_K cell indices), and the reply on
 * dimension-ordering asymmetry (coordinate order K^1, K^2, K^3).
 * Reading: the normalisation is the fixed map [-1, 1) -> [0, 1); in float32,
 * t = (x + 1) * 2^(bits-1), u = min(max(floor(t), 0), 2^bits - 1) (NaN -> 0);
 * bit j of coordinate d goes to code bit j*d_K + (d_K - 1 - d).
 *   x      in : float  [B, H, N, d_K]
 *   codes  out: uint32 or uint64 (see zeta_code_bytes) [B, H, N]
 * Errors: ZETA_ERR_INVALID_ARG on null pointers or invalid sizes.
 */
zeta_status_t zeta_encode(const zeta_problem_t *p, const float *x, void *codes,
                          cudaStream_t stream);

/*
 * zeta_sort_chunks -- sorted key order of every chunk-aligned causal prefix.
 * Passage: OpenReview reply A3 "Chunking ... & Where efficiency is coming from"
 * (radix sort of the Z-order codes) and the atlas.scime.ai summary, "Approach"
 * (keys are sorted and split into chunks, so that all queries search their
 * causal past at the same time).
 * Prefix c holds the keys of chunks 0..c-1 ordered by (code, token index).
 *   key_codes     in : codes of the keys [B, H, N]
 *   prefix_codes  out: same code type [B, H, T]      (T = zeta_prefix_entries)
 *   prefix_idx    out: int32 token indices [B, H, T]
 *   workspace     scratch of at least zeta_sort_workspace_bytes, 256-B aligned
 * Errors: ZETA_ERR_INVALID_ARG, ZETA_ERR_UNSUPPORTED (N / C > 1024),
 *         ZETA_ERR_WORKSPACE (missing or too small).
 */
zeta_status_t zeta_sort_chunks(const zeta_problem_t *p, const void *key_codes,
                               void *prefix_codes, int32_t *prefix_idx,
                               void *workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * zeta_sort_chunks_noalloc -- zeta_sort_chunks without a workspace argument,
 * for callers that cannot allocate device memory when they need the sorted
 * prefixes (code running inside an allocator or memory-pool callback, plug-ins
 * whose host framework owns every device allocation, processes whose device
 * footprint must stay fixed after start-up).  The pages have no counterpart:
 * this is an interface convenience, not part of the method.
 * Scratch: one file-scope device array of 32 MiB, which every GPU that loads
 * this library holds until the process exits.
 * Checks, in order, before anything is launched: every check of
 * zeta_sort_chunks (the same errors; a problem with nothing to sort, empty or
 * with fewer than two chunks, returns ZETA_OK and touches no scratch), then
 * the scratch size: a problem whose zeta_sort_workspace_bytes exceeds 32 MiB
 * is rejected with ZETA_ERR_WORKSPACE.
 * Set-up: the first call on a device (with that device current) looks up the
 * array's device address with cudaGetSymbolAddress and caches it; make that
 * first call before any stream capture on that device.
 * Sharing: every call uses the same array, which keeps the previous call's
 * contents (nothing in it needs to start at zero).  Calls whose work overlaps
 * on the GPU (different streams, or different host threads on one device)
 * race on the array; order them on one stream.
 * Arguments and results are those of zeta_sort_chunks.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
zeta_status_t zeta_sort_chunks_noalloc(const zeta_problem_t *p, const void *key_codes,
                                       void *prefix_codes, int32_t *prefix_idx,
                                       cudaStream_t stream);

/*
 * zeta_select_topk -- the k keys around each query's insertion rank.
 * Passage: OpenReview reply A3 (binary search of the insertion position) and
 * reply A2 "Clarification" (the window centred at the insertion position).
 * For query i in chunk c >= 1, with M = c*C: r = number of prefix-c keys whose
 * code is <= the query's code; start = min(max(r - ceil(k/2), 0), M - k); the
 * row is prefix_idx[prefix c][start .. start + k).  Chunk-0 rows are all -1.
 *   q_codes       in : codes of the queries [B, H, N]
 *   prefix_codes  in : from zeta_sort_chunks
 *   prefix_idx    in : from zeta_sort_chunks
 *   idx           out: int32 [B, H, N, k]
 * Errors: ZETA_ERR_INVALID_ARG.
 */
zeta_status_t zeta_select_topk(const zeta_problem_t *p, const void *q_codes,
                               const void *prefix_codes, const int32_t *prefix_idx,
                               int32_t *idx, cudaStream_t stream);

/*
 * zeta_encode_curves -- codes of every token along several Z-order curves.
 * Passage: OpenReview discussion, follow-up reply on interleaving the bits of
 * different dimensions (several curves)
 * (the key coordinates are interleaved in several orders: the three cyclic
 * shifts of (K^1, K^2, K^3), or all six orderings).
 * Curve m reads coordinate axes[m][s] into slot s, slot 0 being the most
 * significant bit of each level; with axes[m] = (0, 1, ..., d_K - 1) the code
 * is the one zeta_encode writes.  Quantisation as for zeta_encode.
 *   x       in : float [B, H, N, d_K]
 *   curves  in : 1..8
 *   axes    in : HOST int32 [curves][d_K], every row a permutation of 0..d_K-1
 *                (read during the call only)
 *   codes   out: code type of the problem [curves][B, H, N]
 * Errors: ZETA_ERR_INVALID_ARG (null pointers, curves out of range, a row of
 *         axes that is not a permutation).
 */
zeta_status_t zeta_encode_curves(const zeta_problem_t *p, const float *x, int32_t curves,
                                 const int32_t *axes, void *codes, cudaStream_t stream);

/*
 * zeta_select_topk_curves -- the union of one window per curve.
 * Passage: OpenReview discussion, follow-up reply on interleaving the bits of
 * different dimensions (several curves)
 * (every curve collects k // curves of the k tokens).
 * Reading of the union: with km = k // curves, curve m gives the km keys that
 * zeta_select_topk would give with km in place of k (its own prefix table);
 * the windows are listed in curve order, a key already listed is dropped, and
 * the row is padded to k with -1.  Chunk-0 rows are all -1.
 *   q_codes       in : [curves][B, H, N]  (zeta_encode_curves)
 *   prefix_codes  in : [curves][B, H, T]  (curve m's key codes sorted by
 *   prefix_idx    in : [curves][B, H, T]   zeta_sort_chunks; one call on the
 *                      problem with B replaced by curves*B sorts every curve,
 *                      as the two layouts coincide)
 *   idx           out: int32 [B, H, N, k], for zeta_attend_fwd / _bwd
 * Limits: 1 <= curves <= 8, k // curves >= 1, k <= 256.
 * Errors: ZETA_ERR_INVALID_ARG, ZETA_ERR_UNSUPPORTED (k > 256).
 */
zeta_status_t zeta_select_topk_curves(const zeta_problem_t *p, int32_t curves,
                                      const void *q_codes, const void *prefix_codes,
                                      const int32_t *prefix_idx, int32_t *idx,
                                      cudaStream_t stream);

/* Widths of the projection front end: D input features per token, F hidden
 * units per head. */
typedef struct {
    int32_t D, F;
} zeta_proj_t;

/*
 * zeta_project_encode -- queries and keys from token features, with their codes.
 * Passage: OpenReview reply A "LLMs impact the selection of d_K" (a two-layer
 * neural network projects the input into the keys) and reply A2
 * "Clarification of Binary Expansion and Precision" (the codes).
 * Reading: per head hd, and separately for queries (projection 0) and keys
 * (projection 1):
 *   h_f = max(0, W1[hd*F + f] . x_t + b1[hd*F + f]),  y_c = tanh(W2[hd][c] . h + b2[hd][c])
 * (tanh puts the coordinates in (-1, 1), the quantiser's range); y is written
 * out and encoded exactly as zeta_encode would encode it.
 *   x        in : bf16 [B, N, D]           (16-B aligned)
 *   w1       in : bf16 [2, H*F, D]         (16-B aligned; rows are hidden units)
 *   b1       in : float [2, H*F]
 *   w2       in : float [2, H, d_K, F]
 *   b2       in : float [2, H, d_K]
 *   q, k     out: float [B, H, N, d_K]
 *   q_codes, k_codes  out: code type of the problem [B, H, N]
 *   dev_status  optional int32 device word (ZETA_ERR_DEVICE_TIMEOUT if a
 *               bounded wait of the kernel gave up)
 * Limits: F = 64, D a multiple of 64, H = 4 or 8, d_K <= 4, B*N < 2^31.
 * The first layer runs on the tensor cores with bf16 inputs and float32
 * accumulation; the rest in float32.
 * Errors: ZETA_ERR_INVALID_ARG, ZETA_ERR_UNSUPPORTED (outside the limits).
 */
zeta_status_t zeta_project_encode(const zeta_problem_t *p, const zeta_proj_t *pj,
                                  const void *x, const void *w1, const float *b1,
                                  const float *w2, const float *b2, float *q, float *k,
                                  void *q_codes, void *k_codes, int32_t *dev_status,
                                  cudaStream_t stream);

/*
 * zeta_attend_fwd -- Adaptive Cauchy-softmax over the selected keys.
 * Passage: OpenReview reply A2 "Discussion on its robustness" (trainable gamma,
 * Cauchy softmax), reply A3 "Justification for Euclidean Distance Claim", and
 * the atlas.scime.ai summary, "Approach".
 * The attended set of query i in chunk c is its window (non-negative entries
 * of idx row i) plus every key j of its own chunk with cC <= j <= i.  With
 * w_ij = 1 / (1 + |q_i - k_j|^2 / gamma_h^2) (or the kernel that flags
 * selects, see zeta_weight_t) and s_i = sum_j w_ij:
 * out_i = sum_j w_ij v_j / s_i, rowsum_i = s_i.
 *   q, k    in : float [B, H, N, d_K]
 *   v       in : v_dtype [B, H, N, d_V]  (16-B aligned; the tensor-core kernel
 *                (bf16, d_V = 64, d_K <= 4) reads value rows 32 bytes at a time
 *                and runs only where v is 32-B aligned, the general kernel
 *                otherwise)
 *   gamma   in : float [H]
 *   idx     in : int32 [B, H, N, k]; entries must be -1 or in [0, cC)
 *   out     out: v_dtype [B, H, N, d_V]  (16-B aligned)
 *   rowsum  out: float [B, H, N]
 *   dev_status  optional int32 device word; an idx entry outside its range is
 *               skipped and ZETA_ERR_BOUNDS is recorded there.
 * Errors: ZETA_ERR_INVALID_ARG, ZETA_ERR_UNSUPPORTED.
 */
zeta_status_t zeta_attend_fwd(const zeta_problem_t *p, const float *q, const float *k,
                              const void *v, const float *gamma, const int32_t *idx,
                              void *out, float *rowsum, int32_t *dev_status,
                              cudaStream_t stream);

/*
 * zeta_select_attend_fwd -- zeta_select_topk and zeta_attend_fwd in one call.
 * Passage: as for those two calls (OpenReview reply A3 "Chunking ... & Where
 * efficiency is coming from": binary search of the insertion position; the
 * attended set and weights of zeta_attend_fwd).
 * On the tensor-core shapes (bf16 values, d_V = 64, d_K <= 4, v 32-B aligned)
 * one kernel finds each query's window by binary search in its sorted prefix,
 * reads the window as a contiguous run of prefix_idx, attends, and writes the
 * run to idx for zeta_attend_bwd; otherwise the two calls run one after the
 * other.
 * Results are those of zeta_select_topk followed by zeta_attend_fwd.
 *   q, k, v, gamma   in : as for zeta_attend_fwd
 *   q_codes          in : codes of the queries [B, H, N]
 *   prefix_codes, prefix_idx  in : from zeta_sort_chunks
 *   idx              out: int32 [B, H, N, k] (as zeta_select_topk writes it)
 *   out, rowsum      out: as for zeta_attend_fwd
 *   dev_status       optional int32 device word (as for zeta_attend_fwd)
 * Errors: ZETA_ERR_INVALID_ARG, ZETA_ERR_UNSUPPORTED.
 */
zeta_status_t zeta_select_attend_fwd(const zeta_problem_t *p, const float *q, const float *k,
                                     const void *v, const float *gamma, const void *q_codes,
                                     const void *prefix_codes, const int32_t *prefix_idx,
                                     int32_t *idx, void *out, float *rowsum,
                                     int32_t *dev_status, cudaStream_t stream);

/*
 * zeta_attend_bwd -- gradients through the weights, selection fixed.
 * Passage: the forward/backward timings of the OpenReview replies A3/A4 (the
 * method is trained end to end) and the forward definition above.
 * With a_ij = w_ij / s_i, g_ij = dO_i . v_j and gbar_i = sum_j a_ij g_ij
 * (= dO_i . out_i for the exact output):
 *   dL/dw_ij = (g_ij - gbar_i) / s_i
 *   dq_i     = sum_j dL/dw_ij * 2 (dw/dd2)_ij (q_i - k_j)
 *   dk_j     = -sum_i dL/dw_ij * 2 (dw/dd2)_ij (q_i - k_j)
 *   dv_j     = sum_i a_ij dO_i
 *   dgamma_h = sum_{b,i,j} dL/dw_ij * (dw/dgamma)_ij
 * with, per weight kernel, dw/dd2 = -w^2/gamma^2 and dw/dgamma =
 * 2 w (1 - w) / gamma (Cauchy); -w/gamma^2 and 2 w (d2 - m_i) / gamma^3
 * (softmax); -w^3/2 and 0 (inverse Euclidean).
 * s_i and gbar_i are recomputed from q, k, v and idx (one pass over each
 * query's set), so the forward's rounded output is not needed.
 *   q, k, v, gamma, idx  in : as for zeta_attend_fwd
 *   dout         in : v_dtype [B, H, N, d_V]  (16-B aligned)
 *   dq, dk       out: float [B, H, N, d_K]
 *   dv           out: v_dtype [B, H, N, d_V]  (16-B aligned)
 *   dgamma       out: float [H]
 *   workspace    scratch of at least zeta_bwd_workspace_bytes, 256-B aligned
 *   dev_status   optional int32 device word (ZETA_ERR_BOUNDS as for the forward;
 *                ZETA_ERR_DEVICE_TIMEOUT if a bounded wait of the tensor-core
 *                own-chunk kernel gave up)
 * Every output is overwritten.  Reductions run in a fixed order, so results
 * are bit-reproducible run to run.
 * Errors: ZETA_ERR_INVALID_ARG, ZETA_ERR_UNSUPPORTED, ZETA_ERR_WORKSPACE.
 */
zeta_status_t zeta_attend_bwd(const zeta_problem_t *p, const float *q, const float *k,
                              const void *v, const float *gamma, const int32_t *idx,
                              const void *dout, float *dq, float *dk, void *dv, float *dgamma,
                              void *workspace, size_t ws_bytes, int32_t *dev_status,
                              cudaStream_t stream);

/*
 * zeta_check_bounded_wait -- diagnostic of the device-side failure detection.
 * The pages have no counterpart: every wait of the TMA-fed and tensor-core
 * kernels (zeta_project_encode, the own-chunk block of zeta_attend_bwd) on an
 * mbarrier polls a bounded number of times
 * and, when it gives up, records ZETA_ERR_DEVICE_TIMEOUT in the status word and
 * lets the kernel return.  This call runs that wait on one barrier, completed
 * beforehand when arrive != 0 and never completed otherwise, polling at most
 * `iterations` times.
 *   dev_status  int32 device word (required); ZETA_ERR_DEVICE_TIMEOUT is written
 *               there when the wait gave up, nothing otherwise.
 * Errors: ZETA_ERR_INVALID_ARG (null dev_status, zero iterations).
 */
zeta_status_t zeta_check_bounded_wait(uint32_t iterations, int32_t arrive, int32_t *dev_status,
                                      cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ZETA_H */
