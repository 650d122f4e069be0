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

// Element access for the two storage types.
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }

// ---------------------------------------------------------------------------
// Launchers (one translation unit each).  All return the launch error.
// ---------------------------------------------------------------------------

// Screening scores r[g][v][j] = <x_gv, d_gj> for vectors [v0, v0+Vc) of
// every dictionary; scores is [G][Vc][N] fp32.
cudaError_t launch_screen_ffma(const Shape& sh, const void* atoms, const void* x, int64_t x_gstride,
                               int v0, int Vc, float* scores, cudaStream_t st);

// Exact Top-n of |scores| per vector (ties to the lower atom index), pools
// written in ascending atom order: pool_id/pool_r [G][Vc][n].  A vector whose
// scores hold a NaN or infinity gets pool ids -1.
cudaError_t launch_topn_radix(const Shape& sh, const float* scores, int Vc, int32_t* pool_id,
                              float* pool_r, cudaStream_t st);

// Greedy selection inside the pool plus ridge refit; writes idx/coef/relres
// for vectors [v0, v0+Vc) (output arrays are [G][V][...] with per-dictionary
// stride V).
struct GreedyArgs {
    const void* atoms;
    const void* x;
    const int32_t* pool_id;   // [G][Vc][n], ascending atom order
    const float* pool_r;      // [G][Vc][n]
    int32_t* idx;
    float* coef;
    float* relres;
    long long* counters;      // [G][kCntFields]
    int V;                    // vectors per dictionary in the whole call
    int v0, Vc;
};
cudaError_t launch_greedy(const Shape& sh, const GreedyArgs& a, cudaStream_t st);
size_t greedy_smem_bytes(const Shape& sh);

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
    long long* counters;      // [G][kCntFields]
    int V;
};
cudaError_t launch_adapt(const Shape& sh, const AdaptArgs& a, const DeltaTable& delta, cudaStream_t st);

// xhat = D_S c (+ repl term).
cudaError_t launch_reconstruct(const Shape& sh, const void* atoms, int V, const int32_t* idx,
                               const float* coef, const int32_t* repl_id, const float* repl_coef,
                               float* xhat, cudaStream_t st);

}  // namespace fadkv
