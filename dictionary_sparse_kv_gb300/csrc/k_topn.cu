// Exact Top-n candidate pool from materialised screening scores.
//
// "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding",
// abstract ("a one-shot Top-n selection identifies a small candidate pool")
// and Fig. 1 caption (a small Top-n screened pool recalls most full-OMP
// atoms).  Ties at the cut go to the lower atom index.
//
// One CTA per vector.  The keys are the bit patterns of |r_j| (for
// non-negative floats the unsigned order of the bits is the numeric order),
// so an MSD radix select over 4 x 8 bits finds the n-th largest key T
// exactly.  The pool is then every atom with key > T plus the lowest-index
// atoms with key == T, written in ascending atom order by an ordered block
// compaction.  The result is unique, so it is deterministic.  The pool is
// handed on as candidate keys (bits(|r_j|) << 32 | (0xffffffff - j)) with a
// count of exactly n, the form the greedy kernel consumes.
#include "fadkv_internal.cuh"

namespace fadkv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Block-wide exclusive scan of one 32-bit value (kThreads threads); also
// returns the block total.  `ws` is kWarps words of shared memory.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* ws, uint32_t& total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) ws[warp] = incl;
    __syncthreads();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t t = ws[w];
        if (w < warp) before += t;
        all += t;
    }
    __syncthreads();
    total = all;
    return before + incl - v;
}

__global__ void __launch_bounds__(kThreads)
topn_radix_kernel(const float* __restrict__ scores, int N, int n, int Vc, unsigned long long* __restrict__ cand,
                  int* __restrict__ cand_count, int cap)
{
    extern __shared__ uint32_t keys[];   // [N]
    __shared__ uint32_t hist[256];
    __shared__ uint32_t scan_ws[kWarps];
    __shared__ uint32_t s_prefix, s_remaining;

    const int v = blockIdx.x, g = blockIdx.y, tid = threadIdx.x;
    const float* r = scores + ((size_t)g * Vc + v) * N;
    unsigned long long* out = cand + ((size_t)g * Vc + v) * cap;

    int bad = 0;
    for (int j = tid; j < N; j += kThreads) {
        const uint32_t k = __float_as_uint(r[j]) & 0x7fffffffu;
        bad |= (k >= 0x7f800000u);
        keys[j] = k;
    }
    if (__syncthreads_or(bad)) {
        // non-finite scores come only from a non-finite input, which the
        // consumer detects on its own; an empty list sends it there
        if (tid == 0) cand_count[((size_t)g * Vc + v) * kCountSlots] = 0;
        return;
    }

    uint32_t prefix = 0, mask = 0, remaining = (uint32_t)n;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kThreads) hist[i] = 0;
        __syncthreads();
        for (int j = tid; j < N; j += kThreads) {
            const uint32_t k = keys[j];
            if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 0xffu], 1u);
        }
        __syncthreads();
        if (tid < 32) {
            // lane l covers bins 255-8l down to 248-8l (lane 0 holds the top)
            const int hi = 255 - 8 * tid;
            uint32_t local = 0;
#pragma unroll
            for (int b = 0; b < 8; ++b) local += hist[hi - b];
            uint32_t incl = local;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o) incl += t;
            }
            const uint32_t above = incl - local;
            if (above < remaining && remaining <= incl) {
                uint32_t acc = above;
                for (int b = 0; b < 8; ++b) {
                    const uint32_t c = hist[hi - b];
                    if (acc + c >= remaining) {
                        s_prefix = prefix | ((uint32_t)(hi - b) << shift);
                        s_remaining = remaining - acc;
                        break;
                    }
                    acc += c;
                }
            }
        }
        __syncthreads();
        prefix = s_prefix;
        remaining = s_remaining;
        mask |= 0xffu << shift;
        __syncthreads();
    }

    // prefix = the n-th largest key; take every key above it and the first
    // `remaining` keys equal to it, in ascending atom order.
    const uint32_t T = prefix;
    uint32_t base_out = 0, base_eq = 0;
    for (int j0 = 0; j0 < N; j0 += kThreads) {
        const int j = j0 + tid;
        const uint32_t k = (j < N) ? keys[j] : 0u;
        const uint32_t gt = (j < N && k > T) ? 1u : 0u;
        const uint32_t eq = (j < N && k == T) ? 1u : 0u;
        uint32_t tot;
        const uint32_t ex = block_exclusive_scan(gt << 16 | eq, scan_ws, tot);
        const uint32_t rank_eq = ex & 0xffffu, rank_gt = ex >> 16;
        const uint32_t eq_left = (remaining > base_eq) ? remaining - base_eq : 0u;
        const bool take = gt || (eq && rank_eq < eq_left);
        if (take) {
            const uint32_t pos = base_out + rank_gt + min(rank_eq, eq_left);
            out[pos] = ((unsigned long long)k << 32) | (unsigned long long)(0xffffffffu - (uint32_t)j);
        }
        const uint32_t tot_eq = tot & 0xffffu, tot_gt = tot >> 16;
        base_out += tot_gt + min(tot_eq, eq_left);
        base_eq += tot_eq;
    }
    if (tid == 0) cand_count[((size_t)g * Vc + v) * kCountSlots] = n;
}

}  // namespace

cudaError_t launch_topn_radix(const Shape& sh, const float* scores, int Vc, unsigned long long* cand,
                              int* cand_count, int cap, cudaStream_t st)
{
    if (Vc <= 0) return cudaSuccess;
    const size_t smem = sizeof(uint32_t) * (size_t)sh.N;
    cudaError_t e = cudaFuncSetAttribute(topn_radix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(Vc, sh.G);
    topn_radix_kernel<<<grid, kThreads, smem, st>>>(scores, sh.N, sh.n, Vc, cand, cand_count, cap);
    return cudaGetLastError();
}

}  // namespace fadkv
