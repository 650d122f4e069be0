// Internal declarations shared by the CUDA sources of the FAD-KV library.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fadkv.h"

namespace fadkv {

constexpr int kMaxDicts = FADKV_MAX_DICTS;
constexpr int kMaxS = FADKV_MAX_S;
constexpr int kMaxPool = FADKV_MAX_POOL;

// Per-dictionary device counters, in the order fadkv_dict_stats reports them.
enum Counter : int {
    kCntEncoded = 0,
    kCntReplaced = 1,
    kCntFlagged = 2,
    kCntOverflow = 3,
    kCntNonfinite = 4,
    kCntFallback = 5,
    kCntStatus = 6,
    kCntFields = FADKV_STATS_FIELDS
};

// Adaptation thresholds, passed by value to the adapt kernel.
struct DeltaTable {
    float v[kMaxDicts];
};

// Shape of one handle, as the kernels see it.
struct Shape {
    int G, N, d, n, s, dtype;
    float lambda_abs, lambda_rel;
};

// Message for fadkv_last_error on the calling host thread.
void set_last_error(const char* msg);

// Programmatic dependent launch between the kernels of a step: a kernel may
// be scheduled while its predecessor on the stream drains.  pdl_begin()
// waits until the predecessor's results are in global memory (a no-op when
// the kernel was launched normally) and lets the successor be scheduled; every
// kernel launched with launch_pdl calls it before its first global access.
// FADKV_PDL=0 launches normally.
__device__ __forceinline__ void pdl_begin()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
bool pdl_enabled();
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k, static_cast<Args&&>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Element access for the two storage types.
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }

// ---------------------------------------------------------------------------
// Launchers (one translation unit each).  All return the launch error.
// ---------------------------------------------------------------------------

// Candidate capacity per vector: four times the pool size (the screening
// threshold aims at about 1.5n candidates).  On the FP32 path a vector's list
// is made of up to kCountSlots regions, each described by one slot word in
// cand_count[.][kCountSlots]:
//   bit 31      the region overflowed (the consumer redoes the vector exactly)
//   bits 30..16 offset of the region in the vector's list (entries)
//   bits 15..0  keys in the region
// A zero word is an empty slot; consumers reset every word to zero.
__host__ __device__ inline int cand_cap(int n) { return 4 * n; }
constexpr int kCountSlots = 32;
constexpr uint32_t kSlotOverflow = 0x80000000u;
__host__ __device__ inline uint32_t slot_word(bool over, int offset, int count)
{
    return (over ? kSlotOverflow : 0u) | ((uint32_t)offset << 16) | (uint32_t)(count > 0xffff ? 0xffff : count);
}
__host__ __device__ inline int slot_count(uint32_t w) { return (int)(w & 0xffffu); }
__host__ __device__ inline int slot_offset(uint32_t w) { return (int)((w >> 16) & 0x7fffu); }
__host__ __device__ inline bool slot_over(uint32_t w) { return (w & kSlotOverflow) != 0u; }

// Candidate keys: (bits(|r_j|) << 32) | (0xffffffff - j).  The larger key is
// the larger |r|, then the lower atom index: the Top-n pool is the n largest
// keys of a vector.

// Screening scores r[g][v][j] = <x_gv, d_gj> for vectors [v0, v0+Vc) of
// every dictionary on the FP32 pipe; scores is [G][Vc][N] fp32.
cudaError_t launch_screen_ffma(const Shape& sh, const void* atoms, const void* x, int64_t x_gstride,
                               int v0, int Vc, float* scores, cudaStream_t st);

// Exact Top-n of materialised scores: writes the n pool keys of every vector
// to the start of its candidate list, slot 0 = n keys at offset 0 (0 keys for
// non-finite scores).
cudaError_t launch_topn_radix(const Shape& sh, const float* scores, int Vc, unsigned long long* cand,
                              int* cand_count, int cap, cudaStream_t st);

// Tensor-core screening with the fused |r| >= tau filter (binary16 only).
// One CTA per SM; CTA b takes units [b*T/B, (b+1)*T/B) of the T = G * tiles *
// (N/128) (dictionary, 128-vector tile, 128-atom chunk) units, chunk fastest.
//
// Output: per vector and 128-atom chunk c, one record of kRecBytes at
// rec + ((g * Vc + v) * (N/128) + c) * kRecBytes, in 32-bit words:
//   word 0      header: overflow << 31 | count
//   words 1..4  masks: bit t of word 1 + k set when atom c*128 + 32k + t
//               was kept
//   words 5..   the count kept scores r_j (binary32, exact, with their
//               sign), in ascending atom order
// A record with more than kRecVals kept scores is flagged: the consumer
// redoes such a vector exactly.
constexpr int kRecWords = 32;
constexpr int kRecBytes = kRecWords * 4;
constexpr int kRecVals = kRecWords - 5;
__host__ __device__ inline uint32_t rec_header(bool over, int count)
{
    return (over ? 0x80000000u : 0u) | (uint32_t)count;
}
struct ScreenTCArgs {
    int G, N, V, v0, Vc;      // V: vectors per dictionary of the whole call
    const void* x;            // [G][V][d] binary16 (read for ||x||)
    float alpha;              // tau = alpha * ||x|| / sqrt(d)
    unsigned char* rec;       // [G][Vc][N/128] records of kRecBytes
    float* dump;              // test hook: if set, write all scores [G][Vc][N] instead
    long long* counters;      // [G][kCntFields] (status word)
    unsigned long long wait_ns;   // limit of the pipeline's waits (0: the default; a test hook shortens it)
};
// Host-side state a handle keeps between launches: the encoded tensor maps of
// the dictionaries and of the last inputs (by base address and row count)
// and whether the kernel's shared-memory limit was raised.
struct ScreenTCCache {
    alignas(64) unsigned char map_d[128];
    alignas(64) unsigned char map_x[128];
    const void* d_base = nullptr;
    long long d_rows = -1;
    const void* x_base = nullptr;
    long long x_rows = -1;
    bool attr_done[2] = {false, false};
};
bool screen_tc_supported(const Shape& sh);
int screen_tc_grid(const Shape& sh, int Vc, int sms);
cudaError_t launch_screen_tc(const Shape& sh, const void* atoms, const ScreenTCArgs& a, int sms, ScreenTCCache* cache,
                             cudaStream_t st);

// Exact Top-n pool from the screening records, one warp per vector; pool
// [G][Vc][n] atom ids and pool_r [G][Vc][n] their scores r_j (signed).  A
// record that overflowed still lists every kept atom in its masks: the warp
// recomputes those scores on the FP32 pipe.  pool[0] = -2 where the exact
// slow path must redo the vector (fewer than n candidates, or more than
// cap).
struct SelectArgs {
    int G, Vc, N, n, cap;     // cap: the most candidates taken (else the slow path)
    int d, V, v0;             // head dimension; the call's vectors per dictionary and this pass's first
    const __half* x;          // [G][V][d] (for records whose scores must be recomputed)
    const __half* atoms;      // [G][N][d]
    const unsigned char* rec; // [G][Vc][N/128] screening records
    int32_t* pool;            // [G][Vc][n]
    float* pool_r;            // [G][Vc][n]
    uint32_t* slow_seq;       // set to `seq` when some vector of the pass needs the slow path
    uint32_t seq;             // number of this screening pass (never 0)
};
cudaError_t launch_select(const SelectArgs& a, cudaStream_t st);
size_t select_smem_bytes(int cap);
// Keys a selection warp holds: the screening threshold aims at 1.5n
// candidates, so 2n leaves room for the spread; more take the slow path.
__host__ __device__ inline int select_cap(int n) { return 2 * n; }

// Exact Top-n from the candidate lists (slow exact path for lists shorter
// than n or longer than cap), then greedy selection inside the pool plus
// ridge refit; writes idx/coef/relres for vectors [v0, v0+Vc) (outputs are
// [G][V][...]).  With pool_out set it only writes the pool ids (debug hook).
struct GreedyArgs {
    const void* atoms;
    const void* x;
    unsigned long long* cand; // [G][Vc][cap]
    int* cand_count;          // [G][Vc][kCountSlots] slot words; reset to 0 once consumed
    int cap;
    int32_t* idx;
    float* coef;
    float* relres;
    const int32_t* pool_in;   // optional [G][Vc][n] pool from launch_select (then cand* unused)
    int32_t* pool_out;        // optional [G][V][n]
    float* pool_r_out;        // optional [G][V][n] (with pool_out)
    long long* counters;      // [G][kCntFields]
    int V;                    // vectors per dictionary in the whole call
    int v0, Vc;
};
cudaError_t launch_greedy(const Shape& sh, const GreedyArgs& a, cudaStream_t st);
size_t greedy_smem_bytes(const Shape& sh);

// Gram matrices of the dictionaries (binary16): gram [G][N][N] fp32 and its
// diagonal gdiag [G][N].  Build: every entry.  Update: the rows and columns
// of the nrows[g] atoms listed at rows + g * row_stride (the atoms an
// adaptation just wrote).
bool greedy_gram_supported(const Shape& sh);
size_t gram_bytes(const Shape& sh);
cudaError_t launch_gram_build(const Shape& sh, const void* atoms, float* gram, float* gdiag, int sms,
                              cudaStream_t st);
cudaError_t launch_gram_update(const Shape& sh, const void* atoms, const int32_t* rows, const int32_t* nrows,
                               int row_stride, float* gram, float* gdiag, int sms, cudaStream_t st);

// Greedy selection + ridge refit over the Gram matrix, in the correlation
// domain (binary16, n <= 512, s <= 16): the pool's ids and signed scores
// come from the selection (or the pool fixup), the pick's Gram row from
// gram; writes idx/coef/relres for vectors [v0, v0+Vc).
struct GramGreedyArgs {
    const __half* atoms;      // [G][N][d]
    const __half* x;          // [G][V][d]
    const int32_t* pool;      // [G][Vc][n]
    const float* pool_r;      // [G][Vc][n]
    const float* gram;        // [G][N][N]
    const float* gdiag;       // [G][N]
    int32_t* idx;             // [G][V][s]
    float* coef;              // [G][V][s]
    float* relres;            // [G][V]
    long long* counters;      // [G][kCntFields]
    int V, v0, Vc;
};
cudaError_t launch_greedy_gram(const Shape& sh, const GramGreedyArgs& a, cudaStream_t st);

// Exact pool (ids and signed scores) of the vectors the selection kernel
// left to the slow path (pool[0] == -2): all N scores on the FP32 pipe,
// exact Top-n.
cudaError_t launch_pool_fixup(const Shape& sh, const GreedyArgs& a, int32_t* pool, float* pool_r,
                              const uint32_t* slow_seq, uint32_t seq, int sms, cudaStream_t st);

// PL encode's fit: the s atoms of the Top-s set in ascending order and one
// ridge fit over them, one warp per vector.  The set comes from `pool`
// ([G][Vc][s] ids in any order; the selection + pool fixup with n = s) or,
// when pool is null, from the FP32 path's candidate keys (cand, cand_count,
// cap; the radix Top-n with n = s writes them in ascending atom order).
struct PlArgs {
    const void* atoms;
    const void* x;
    const int32_t* pool;
    const unsigned long long* cand;
    const int* cand_count;
    int cap;
    int32_t* idx;
    float* coef;
    float* relres;
    long long* counters;      // [G][kCntFields]
    int V;                    // vectors per dictionary in the whole call
    int v0, Vc;
};
cudaError_t launch_pl_fit(const Shape& sh, const PlArgs& a, cudaStream_t st);

// The compressed store: packed words of a step's codes written into the
// per-sequence caches [G][B][H][Tmax][s+1] at each sequence's position.
struct StoreArgs {
    int G, B, H, s, N, Tmax;
    const int32_t* idx;       // [G][B*H][s]
    const float* coef;
    const int32_t* repl_id;   // [G][B*H] or null
    const float* repl_coef;
    const int32_t* pos;       // [B]
    uint32_t* cache;
};
cudaError_t launch_store_codes(const StoreArgs& a, cudaStream_t st);

// Decode attention over packed K/V codes, one CTA per (layer, sequence, KV head).
struct AttendArgs {
    const void* dict_k;       // layer l's key dictionary at dict_k + l * dict_stride (elements)
    const void* dict_v;
    long long dict_stride;
    const uint32_t* cache_k;  // [B][Hkv][Tmax][s+1] per layer, layers cache_stride words apart
    const uint32_t* cache_v;
    long long cache_stride;
    const int32_t* lengths;   // [B]
    const float* q;           // [L][B][Hq][d]
    float* out;               // [L][B][Hq][d]
    int L, B, Hq, Hkv, d, N, s, Tmax, dtype;
    float scale;
    // binary16 dictionaries: workspace of the per-layer GEMMs (attend_bind_workspace)
    int Npad;                 // N rounded up to 16
    float* U;                 // [L][B*Hq][Npad] scale q D_K^T
    __half* Whi;              // [L][B*Hq][Npad] w / S, scaled per row, two binary16 terms
    __half* Wlo;
    float* wunscale;          // [L][B*Hq] the per-row scale's inverse (0 for an empty sequence)
};
inline int attend_npad(int N) { return (N + 15) / 16 * 16; }
bool attend_supported(int d, int N, int s);
size_t attend_workspace_bytes(int L, int B, int Hq, int N, int dtype);
void attend_bind_workspace(AttendArgs& a, void* ws);
cudaError_t launch_attend(const AttendArgs& a, cudaStream_t st);

// Fixed-size adaptation, one CTA per dictionary.
struct AdaptArgs {
    void* atoms;
    int32_t* usage;
    const void* x;
    const int32_t* idx;
    const float* coef;
    const float* relres;
    int32_t* repl_id;
    float* repl_coef;
    int32_t* inactive;        // [G][N] scratch
    int32_t* flagged;         // [G][max_batch] scratch
    int32_t* nrep;            // optional [G]: atoms written by this call (their ids: inactive[g][0..nrep))
    long long* counters;      // [G][kCntFields]
    int V;
    int append;               // 0: reuse inactive atoms (usage == 0); 1: fill free slots (usage < 0)
};
cudaError_t launch_adapt(const Shape& sh, const AdaptArgs& a, const DeltaTable& delta, cudaStream_t st);
// Kernels launch_adapt launches for V vectors per dictionary (the usage
// increments run over the whole grid first when the batch is large).
int adapt_launches(const Shape& sh, int V);

// Test hook: one thread waits, with a limit of limit_ns, on an mbarrier that
// nothing arrives on, so the wait runs out and sets FADKV_DEV_TIMEOUT in
// *status.
cudaError_t launch_wait_probe(unsigned long long* status, unsigned long long limit_ns, cudaStream_t st);

// xhat = D_S c (+ repl term).
cudaError_t launch_reconstruct(const Shape& sh, const void* atoms, int V, const int32_t* idx,
                               const float* coef, const int32_t* repl_id, const float* repl_coef,
                               float* xhat, cudaStream_t st);

}  // namespace fadkv
