/*
 * fadkv.h -- C ABI of the FAD-KV per-token KV encoding library (sm_103a).
 *
 * What it computes comes from "FAD-KV: Adaptive Dictionary KV Caching for
 * Efficient Reasoning Decoding" (thelatestinai.com/papers/2610.37921):
 *   - abstract: each token's key or value head-vector is represented as a
 *     sparse combination of dictionary atoms; a screening-based sparse coder
 *     makes a one-shot Top-n selection of a small candidate pool and then
 *     refines coefficients; a fixed-size adaptation reuses inactive atoms
 *     instead of growing the dictionary;
 *   - Fig. 2 caption: if the reconstruction error of an incoming vector is
 *     high, an inactive atom is replaced by a context-relevant atom, keeping
 *     the dictionary size fixed throughout decoding;
 *   - Table 5: ridge parameter 1e-4 + 0.20 diag(G), thresholds 0.50 (key) /
 *     0.70 (value), N = 4096 / 8192, s = 8 / 16, n = 256 / 512.
 * Conventions the pages leave open, fixed by this library:
 *   - the s atoms are chosen greedily inside the pool: at step k the atom of
 *     the pool (not yet chosen) with the largest |<d_j, e_k>| is added, the
 *     coefficients are refit by the ridge solve, e_{k+1} = x - D_S c;
 *   - every tie (Top-n cut, greedy choice) goes to the lower atom index;
 *   - replacement order: the m-th flagged vector of a call (ascending vector
 *     index, relres > delta strictly) takes the m-th inactive atom (ascending
 *     atom index, usage == 0 after the call's usage increments);
 *   - the replacement atom is the normalised ridge residual e/||e||; the
 *     vector gets it as an extra term with coefficient ||e||.
 *
 * Memory and threading model
 *   - Every array argument is a DEVICE pointer unless stated otherwise.  The
 *     caller owns all device memory (dictionary, usage counts, workspace,
 *     inputs, outputs); the library never allocates or frees device memory.
 *   - A handle covers G = num_dicts independent dictionaries of the same
 *     shape, stored back to back, so one call encodes a whole decode step
 *     (all layers, keys and values) in one launch per kernel.
 *     Layouts (row-major, dictionary-major):
 *       atoms     [G][N][d]   binary16 or binary32 (params.dtype)
 *       usage     [G][N]      int32
 *       x         [G][V][d]   same type as atoms
 *       idx       [G][V][s]   int32, pick order; -1 for a non-finite input
 *       coef      [G][V][s]   float32
 *       relres    [G][V]      float32, ||x - D_S c|| / ||x||  (0 if x = 0)
 *       repl_id   [G][V]      int32, replacement atom or -1
 *       repl_coef [G][V]      float32
 *       xhat      [G][V][d]   float32
 *   - All calls are asynchronous on the given CUDA stream (a cudaStream_t
 *     passed as void*; NULL = legacy default stream).  A handle is not
 *     thread-safe: issue its calls from one thread, in stream order.
 *   - Every encode batch must be passed to fadkv_adapt before the next
 *     encode or adapt on the same handle (otherwise the usage counts would
 *     miss that batch and an atom in use could be overwritten).  The host
 *     enforces this and returns FADKV_ERR_SEQUENCE.
 *
 * Errors
 *   - Functions return a fadkv_status; nothing is thrown across the ABI.
 *   - Argument errors are detected on the host before any launch, and leave
 *     the handle's state unchanged.
 *   - Conditions found on the device (non-finite input, a refit matrix that
 *     is not positive definite) set bits in the per-dictionary device status
 *     word, read back by fadkv_dict_stats after a stream sync.
 */
#ifndef FADKV_H
#define FADKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FADKV_ABI_VERSION 1
#define FADKV_MAX_DICTS 256   /* dictionaries per handle */
#define FADKV_MAX_S 32        /* largest sparsity s */
#define FADKV_MAX_POOL 1024   /* largest pool size n */

typedef enum {
    FADKV_OK = 0,
    FADKV_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer */
    FADKV_ERR_UNSUPPORTED = 2,   /* shape outside what the kernels implement */
    FADKV_ERR_SEQUENCE = 3,      /* encode/adapt called out of order */
    FADKV_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    FADKV_ERR_WORKSPACE = 5      /* workspace too small */
} fadkv_status;

typedef enum { FADKV_F16 = 0, FADKV_F32 = 1 } fadkv_dtype;

/* Device status word bits (per dictionary, see fadkv_dict_stats). */
#define FADKV_DEV_NONFINITE_INPUT 0x1   /* an input held a NaN or infinity */
#define FADKV_DEV_NOT_SPD 0x2           /* a refit matrix lost positive definiteness */
#define FADKV_DEV_TIMEOUT 0x4           /* a kernel gave up waiting on its own pipeline */

typedef struct {
    int32_t num_dicts;   /* G, 1 .. FADKV_MAX_DICTS */
    int32_t N;           /* atoms per dictionary, multiple of 64 */
    int32_t d;           /* head dimension: 64 or 128 */
    int32_t n;           /* Top-n pool size, s <= n <= min(N, FADKV_MAX_POOL) */
    int32_t s;           /* atoms per vector, 1 .. FADKV_MAX_S */
    float lambda_abs;    /* ridge, absolute part (Table 5: 1e-4) */
    float lambda_rel;    /* ridge, part relative to diag(G) (Table 5: 0.20) */
    int32_t dtype;       /* fadkv_dtype of atoms and inputs */
    int32_t max_batch;   /* largest V (vectors per dictionary) of one call */
} fadkv_params;

typedef struct fadkv_dict_s* fadkv_dict;

/* Version of this ABI (FADKV_ABI_VERSION of the built library). */
int32_t fadkv_abi_version(void);

/* Human-readable name of a status code (static string). */
const char* fadkv_status_string(fadkv_status status);

/* Message of the last CUDA error seen by a call on this host thread
   (static thread-local buffer; "" if none). */
const char* fadkv_last_error(void);

/* Bytes of device workspace a handle with these parameters needs.
   Host-only; writes *bytes.  Errors: INVALID_ARG, UNSUPPORTED. */
fadkv_status fadkv_workspace_bytes(const fadkv_params* params, size_t* bytes);

/* Create a handle over caller-owned device memory.
     atoms      [G][N][d] dictionary (mutated by fadkv_adapt), 16-byte aligned
     usage      [G][N] usage counts (mutated by fadkv_adapt); an atom is
                inactive while its count is 0; a negative count marks a
                free slot, a row that holds no atom yet (keep its row zero:
                screening still reads it, and a zero row scores 0), which
                only fadkv_adapt_append fills
     delta      HOST array [G] of adaptation thresholds (Table 5: 0.50 for a
                key dictionary, 0.70 for a value dictionary); copied
     workspace  device buffer of at least fadkv_workspace_bytes bytes,
                256-byte aligned, ZERO-FILLED before this call (it holds the
                per-dictionary counters); owned by the caller, used by the
                handle until fadkv_dict_destroy
   Host-only: makes no CUDA call.  Errors: INVALID_ARG, UNSUPPORTED,
   WORKSPACE. */
fadkv_status fadkv_dict_create(const fadkv_params* params, void* atoms, int32_t* usage,
                               const float* delta, void* workspace, size_t workspace_bytes,
                               fadkv_dict* out);

/* Rebuild the handle's Gram matrices from the atoms as they stand.  For
   binary16 dictionaries screened on the tensor cores (N a multiple of 128,
   n <= 512, s <= 16) the greedy coder reads the inner products of the atoms
   from a Gram matrix per dictionary kept in the workspace (G * N * N * 4
   bytes of fadkv_workspace_bytes).  It is built by the first fadkv_encode
   and kept up to date by fadkv_adapt / fadkv_adapt_append, which rewrite its
   rows and columns of the atoms they write.  A caller that changes atoms in
   any other way (its own copies, fadkv_adapt_noalloc on the same buffer)
   calls this before the next fadkv_encode.  Asynchronous on `stream`; a
   no-op for handles without Gram matrices.  Errors: INVALID_ARG, CUDA. */
fadkv_status fadkv_dict_refresh(fadkv_dict dict, void* stream);

/* Free the host-side handle.  Device memory stays with the caller.
   The caller must make sure no work of this handle is still running. */
fadkv_status fadkv_dict_destroy(fadkv_dict dict);

/* Encode V vectors per dictionary (abstract; Fig. 2 caption: screening-based
   sparse coding).  For every x: scores r = D x; pool P = the n atoms with the
   largest |r_j| (ties to the lower j); s greedy picks inside P with the ridge
   refit (G + diag(lambda_abs + lambda_rel G_ii)) c = D_S x after each pick;
   relres = ||x - D_S c|| / ||x||.
     x [G][V][d]; outputs idx [G][V][s], coef [G][V][s], relres [G][V].
   0 <= V <= max_batch.  Every vector is encoded against the dictionary as it
   stands at the start of the call.  A vector holding a NaN or infinity gets
   idx = -1, coef = 0, relres = NaN and sets FADKV_DEV_NONFINITE_INPUT.
   Errors: INVALID_ARG, SEQUENCE (previous encode not adapted yet), CUDA. */
fadkv_status fadkv_encode(fadkv_dict dict, const void* x, int32_t V, int32_t* idx, float* coef,
                          float* relres, void* stream);

/* PL encode: the cheaper coder of the "PL (ours)" rows of Tables 1-4 (Table 4:
   Cost 0.13 of OMP, against 0.19 for the greedy coder).  The pages name it
   without spelling it out; this library reads it as screening plus a single
   ridge fit, the reading that cost supports: for every x, scores r = D x;
   S = the s atoms with the largest |r_j| (ties to the lower j); one solve
   (G + diag(lambda_abs + lambda_rel G_ii)) c = D_S x with G = D_S D_S^T;
   relres = ||x - D_S c|| / ||x|| (0 if x = 0).
     x [G][V][d]; outputs idx [G][V][s] in ASCENDING atom order (not a pick
     order), coef [G][V][s] aligned with idx, relres [G][V].
   Arguments, ordering and errors as for fadkv_encode: the batch counts as
   an encode and must be passed to fadkv_adapt (which works the same on
   either coder's output) before the next encode; a non-finite x gets
   idx = -1, coef = 0, relres = NaN.  The handle's n is not used.
   Errors: INVALID_ARG, SEQUENCE, CUDA. */
fadkv_status fadkv_encode_pl(fadkv_dict dict, const void* x, int32_t V, int32_t* idx, float* coef,
                             float* relres, void* stream);

/* Fixed-size adaptation of the batch just encoded (abstract; Fig. 2 caption).
   usage[idx] += 1 for every selected atom; then the m-th vector with
   relres > delta[g] (ascending v) takes the m-th atom with usage == 0
   (ascending id): that atom becomes e/||e|| with e = x - D_S c (rounded to
   the dictionary type), its usage becomes 1, repl_id[v] = its id and
   repl_coef[v] = ||e||.  Other vectors get repl_id = -1, repl_coef = 0.
   Flagged vectors left without an inactive atom keep their s-term code and
   are counted as overflow.  The dictionary keeps N atoms; free slots
   (usage < 0) are never taken.
   Arguments are the same x, V, idx, coef, relres as the encode call.
   Errors: INVALID_ARG, SEQUENCE (no encode pending, or a different V), CUDA. */
fadkv_status fadkv_adapt(fadkv_dict dict, const void* x, int32_t V, const int32_t* idx,
                         const float* coef, const float* relres, int32_t* repl_id,
                         float* repl_coef, void* stream);

/* Append-only growth: the strategy the pages contrast FAD-KV with (abstract:
   naive append-only updates grow the dictionary during generation; Fig. 2
   caption: FAD-KV replaces an inactive atom instead of appending a new one),
   for side-by-side runs.  The same as fadkv_adapt except for the rows the
   flagged vectors take: the m-th flagged vector (ascending v, relres >
   delta[g]) takes the m-th FREE SLOT (usage < 0, ascending id) instead of an
   inactive atom, so the dictionary grows by one atom per flagged vector
   into the capacity the caller reserved, and no atom, inactive or not, is
   ever rewritten.  Flagged vectors beyond the free slots are counted as
   overflow; "atoms replaced" in fadkv_dict_stats counts appended atoms.
   The dictionary's size is the number of rows with usage >= 0.  Arguments,
   sequence contract and errors as for fadkv_adapt. */
fadkv_status fadkv_adapt_append(fadkv_dict dict, const void* x, int32_t V, const int32_t* idx,
                                const float* coef, const float* relres, int32_t* repl_id,
                                float* repl_coef, void* stream);

/* Fixed-size adaptation without a handle and without caller scratch.  The
   pages have no counterpart to this call: it runs the same adaptation as
   fadkv_adapt (same kernel, same results) for callers that cannot give the
   library any device memory of its own, e.g. a plain C runtime with a fixed
   memory plan and no allocator, or a decode loop that must not call
   cudaMalloc / cudaFree since either can synchronise the whole device.
     params     shape and dtype (max_batch is not used; V is limited by the
                scratch instead); the same checks as fadkv_workspace_bytes
     atoms      [G][N][d] dictionary, 16-byte aligned (mutated)
     usage      [G][N] int32 usage counts (mutated)
     delta      HOST array [G] of thresholds, each >= 0
     x, V, idx, coef, relres, repl_id, repl_coef: as for fadkv_adapt
     stream     cudaStream_t as void*; NULL = legacy default stream
   Scratch: one statically sized device array inside the library (4 MiB per
   device) holds the inactive-atom list, the flagged-vector list and the
   counters.  A call needs 256-rounded 4*G*N + 4*G*V bytes plus 64*G; more
   than 4 MiB returns FADKV_ERR_WORKSPACE with the sizes in
   fadkv_last_error(), before any CUDA call.  Nothing in the scratch has to
   start at zero, and the library allocates and frees nothing.
   The first call on a device looks up the scratch's address there
   (cudaGetSymbolAddress, with that device current) and keeps it for the CUDA
   context current at the time; a call made in another context of that device
   (a non-primary context made current, or the primary context re-created
   after cudaDeviceReset) looks it up again.  A caller that records its calls
   under stream capture should make one call on each device, in the context
   it captures in, before capture begins.  All calls on one device share the
   one scratch array:
   calls that may run concurrently (different streams or host threads) race,
   so issue them in order on one stream.  There is no sequence check and no
   per-dictionary statistics: the caller keeps encode/adapt order itself.
   Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA. */
fadkv_status fadkv_adapt_noalloc(const fadkv_params* params, void* atoms, int32_t* usage,
                                 const float* delta, const void* x, int32_t V, const int32_t* idx,
                                 const float* coef, const float* relres, int32_t* repl_id,
                                 float* repl_coef, void* stream);

/* Sparse reconstruction (abstract: a sparse combination of atoms):
   xhat_v = sum_k coef[v][k] d_{idx[v][k]} + repl_coef[v] d_{repl_id[v]}.
   repl_id / repl_coef may both be NULL (no replacement terms); entries with
   idx or repl_id = -1 are skipped.  Valid for any code produced earlier by
   encode + adapt: atoms in use are never overwritten.
   Errors: INVALID_ARG, CUDA. */
fadkv_status fadkv_reconstruct(fadkv_dict dict, int32_t V, const int32_t* idx, const float* coef,
                               const int32_t* repl_id, const float* repl_coef, float* xhat,
                               void* stream);

/* Per-dictionary counters, copied to HOST memory host_out[G][FADKV_STATS_FIELDS];
   synchronises the stream.  Fields, in order: vectors encoded (adapted),
   atoms replaced, flagged vectors, overflow (flagged without an inactive
   atom), non-finite inputs, Top-n slow-path uses, device status word, 0.
   Errors: INVALID_ARG, CUDA. */
#define FADKV_STATS_FIELDS 8
fadkv_status fadkv_dict_stats(fadkv_dict dict, int64_t* host_out, void* stream);

/* Test hook: the Top-n pool of each x without changing any state.
   pool [G][V][n] int32, the pool's atom ids in no particular order (-1 for
   a non-finite input); pool_r (may be NULL) [G][V][n] float32 |r| of those
   atoms, in the same order.  Errors: INVALID_ARG, CUDA. */
fadkv_status fadkv_debug_pool(fadkv_dict dict, const void* x, int32_t V, int32_t* pool,
                              float* pool_r, void* stream);

/* Test hook: screening scores [G][V][N] float32 of each x, from the same
   screening kernel encode uses (tensor cores for binary16 dictionaries).
   No state changes.  V must not exceed the handle's internal pass size
   (at least min(max_batch, 128)).  Errors: INVALID_ARG, CUDA. */
fadkv_status fadkv_debug_scores(fadkv_dict dict, const void* x, int32_t V, float* scores, void* stream);

/* Test hook: the wall-clock limit, in nanoseconds, of the waits inside the
   tensor-core screening pipeline of this handle (0 = the default, 200 ms).
   A wait that runs out sets FADKV_DEV_TIMEOUT in the status word and the
   kernel stops early: that pass's candidates are then incomplete (codes stay
   valid atom ids, but are not the exact encode).  The kernel still waits for
   every copy and MMA it issued, with the default limit, before it returns.
   Host-only.  Errors: INVALID_ARG. */
fadkv_status fadkv_debug_wait_limit(fadkv_dict dict, uint64_t limit_ns);

/* Test hook: launches one thread that waits, with a limit of limit_ns
   (1 .. 10^10), on a barrier nothing ever arrives on, so the wait runs out
   and sets FADKV_DEV_TIMEOUT in dictionary 0's status word (read it with
   fadkv_dict_stats).  Nothing else is touched.  Asynchronous on `stream`.
   Errors: INVALID_ARG, CUDA. */
fadkv_status fadkv_debug_wait_probe(fadkv_dict dict, uint64_t limit_ns, void* stream);

/* ---------------------------------------------------------------------------
   The compressed KV store and decode attention over it.  Handle-free: both
   calls work on caller-owned buffers only.

   What the cache keeps instead of K and V is the codes (Table 4: the
   per-sequence KV memory of the dictionary methods against full KV).  The
   pages give no storage format; this library packs every nonzero into one
   32-bit word:
     bits 31..13  the coefficient rounded to 11 significant bits (round to
                  nearest, ties to even) in the layout of binary32's top 19
                  bits (sign, 8-bit exponent, 10 fraction bits); magnitudes
                  below 2^-126 are stored as 0;
     bits 12..0   the atom id (so N <= 8192).
   A token's code is s + 1 words: its s terms, then its replacement term
   from the adaptation (word 0 when it has none).  A skipped term (id -1, a
   zero or non-finite coefficient) is word 0: coefficient 0, atom 0.
   --------------------------------------------------------------------------- */
#define FADKV_PACK_ID_BITS 13

/* Store one step's codes in the per-sequence caches.
     G dictionaries, each with V = B * H vectors ordered v = b * H + h
     (sequence b, KV head h); idx / coef [G][V][s] and repl_id / repl_coef
     [G][V] (both NULL: no replacement words) as fadkv_encode / fadkv_adapt
     wrote them; pos [B] device int32: the token position of this step in
     each sequence's cache; cache [G][B][H][Tmax][s+1] uint32, written at
     [g][b][h][pos[b]][0..s] only (positions outside [0, Tmax) are skipped).
   All pointers are device pointers, 4-byte aligned.  Asynchronous on
   `stream`.  Errors: INVALID_ARG, UNSUPPORTED (N > 8192, s > FADKV_MAX_S),
   CUDA. */
fadkv_status fadkv_store_codes(int32_t G, int32_t B, int32_t H, int32_t s, int32_t N, const int32_t* idx,
                               const float* coef, const int32_t* repl_id, const float* repl_coef,
                               const int32_t* pos, uint32_t* cache, int32_t Tmax, void* stream);

typedef struct {
    int32_t layers;     /* L */
    int32_t B;          /* sequences */
    int32_t Hq;         /* query heads (a multiple of Hkv) */
    int32_t Hkv;        /* KV heads; query head h reads KV head h / (Hq / Hkv) */
    int32_t d;          /* head dimension: 64 or 128 */
    int32_t N;          /* atoms per dictionary, <= 8192 */
    int32_t s;          /* terms per code (s + 1 words per token) */
    int32_t Tmax;       /* cache capacity in tokens */
    int32_t dtype;      /* fadkv_dtype of the dictionaries */
    float scale;        /* score scale, 1/sqrt(d) for standard attention */
    int64_t dict_stride;   /* elements from layer l's key (value) dictionary to layer l+1's; a multiple of 8 */
    int64_t cache_stride;  /* words from layer l's key (value) cache to layer l+1's */
} fadkv_attn_params;

/* Decode attention over the compressed store, for every layer, sequence and
   query head in one call (three kernel launches for binary16 dictionaries,
   one for binary32):
     out[l][b][h] = sum_t p_t v_t,  p = softmax_t(scale <q[l][b][h], k_t>),
   over the tokens t < lengths[b] of KV head h / (Hq / Hkv) of sequence b,
   where k_t and v_t are the sparse combinations their packed codes name:
   k_t = sum_i c_ti dict_k[j_ti].  Neither K nor V is rebuilt: with
   u = dict_k q the scores are s + 1 gathers from u per token, and the output
   is dict_v^T w with w the attention-weighted sum of the value codes.
     dict_k, dict_v  device, layer l's [N][d] dictionaries at + l*dict_stride
                     (with one handle's atoms [2L][N][d], keys at even g:
                     dict_k = atoms, dict_v = atoms + N*d, dict_stride = 2*N*d),
                     16-byte aligned
     cache_k, cache_v device, layer l's [B][Hkv][Tmax][s+1] packed codes at
                     + l*cache_stride (fadkv_store_codes with G = 2L: cache_k
                     = cache, cache_v = cache + B*Hkv*Tmax*(s+1), cache_stride
                     = 2*B*Hkv*Tmax*(s+1))
     lengths         device [B] int32, clamped to [0, Tmax]; an empty
                     sequence gives 0
     q, out          device [L][B][Hq][d] float32 (q 16-byte aligned: its rows
                     are read as vectors)
     workspace       device, >= fadkv_attend_workspace_bytes bytes, 256-byte
                     aligned, caller-owned (contents need no initialisation)
   With binary16 dictionaries the two dictionary products run as per-layer
   tensor-core GEMMs over all sequences and heads (q and w enter as two
   binary16 terms each, about 22 significant bits; FP32 sums); the token
   pass is FP32.  Binary32 dictionaries: FP32 throughout.  Asynchronous on
   `stream`.  Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA. */
fadkv_status fadkv_attend(const fadkv_attn_params* params, const void* dict_k, const void* dict_v,
                          const uint32_t* cache_k, const uint32_t* cache_v, const int32_t* lengths,
                          const float* q, float* out, void* workspace, size_t workspace_bytes,
                          void* stream);

/* Device workspace fadkv_attend needs for these parameters (host-only;
   writes *bytes).  Binary16 dictionaries: the per-layer products U = scale
   Q D_K^T and the token pass's weights W, 8 * layers * B * Hq *
   round_up(N, 16) bytes and a little more; binary32 dictionaries: 0 (the
   workspace may then be NULL).  Errors: INVALID_ARG, UNSUPPORTED. */
fadkv_status fadkv_attend_workspace_bytes(const fadkv_attn_params* params, size_t* bytes);

/* Kernel classes reported by fadkv_profile_read. */
#define FADKV_PROFILE_KERNELS 8
#define FADKV_K_SCREEN 0       /* screening (tensor cores + candidate filter, or FP32 scores) */
#define FADKV_K_TOPN 1         /* Top-n: the selection from the screening records and the exact
                                  pool fixup, or the radix Top-n over FP32 scores (binary32) */
#define FADKV_K_GREEDY 2       /* in-pool greedy selection + ridge refit (the PL fit for
                                  fadkv_encode_pl) */
#define FADKV_K_ADAPT 3        /* fixed-size adaptation */
#define FADKV_K_RECONSTRUCT 4  /* sparse reconstruction */
#define FADKV_K_GRAM 5         /* the dictionaries' Gram matrices: the build at the first encode
                                  (or fadkv_dict_refresh) and the update after each adaptation */

/* Tracing.  The library always counts its kernel launches per class.  With
   profiling enabled it also brackets every launch with a pair of CUDA events
   recorded on the launch stream and accumulates the device time between
   them.  Not for use inside CUDA-graph capture.  Errors: INVALID_ARG. */
fadkv_status fadkv_profile_enable(fadkv_dict dict, int32_t enable);

/* The kernel classes that profiling brackets with events: bit k of
   class_mask stands for class k (FADKV_K_*); all classes by default.  Launch
   counts are kept for every class regardless.  Bracketing fewer launches
   leaves the others back to back on the stream, so a timed step is
   perturbed less.  Errors: INVALID_ARG. */
fadkv_status fadkv_profile_select(fadkv_dict dict, uint32_t class_mask);

/* Launch counts and device milliseconds per kernel class since the last
   reset, written to HOST arrays launches[FADKV_PROFILE_KERNELS] and
   ms[FADKV_PROFILE_KERNELS] (either may be NULL).  Waits for the recorded
   events.  reset != 0 clears the accumulators afterwards.
   Errors: INVALID_ARG, CUDA. */
fadkv_status fadkv_profile_read(fadkv_dict dict, int64_t* launches, double* ms, int32_t reset);

#ifdef __cplusplus
}
#endif

#endif /* FADKV_H */
