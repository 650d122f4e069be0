// Exact Top-n pool of one vector from its screening candidates, for the
// greedy kernels (one CTA per vector, any multiple of 32 threads up to 1024).
//
// "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding",
// abstract: a one-shot Top-n selection gives the candidate pool; ties go to
// the lower atom index (a convention of this library).
//
// Candidate keys are (bits(|r_j|) << 32) | (0xffffffff - j): the n largest
// keys are the pool.  The list arrives split into regions with one count
// each; if a region overflowed, or fewer than n atoms passed the screening
// threshold, every score is recomputed on the FP32 pipe and all N atoms are
// candidates (exact slow path).  The n-th largest key is found by an MSD
// radix select over the 64-bit keys, stopping as soon as the boundary bin is
// taken whole; an ordered compaction then lists the pool.
#pragma once

#include "fadkv_internal.cuh"

namespace fadkv {
namespace sel {

__device__ __forceinline__ unsigned long long screen_key(float r, int atom)
{
    return ((unsigned long long)(__float_as_uint(r) & 0x7fffffffu) << 32) |
           (unsigned long long)(0xffffffffu - (unsigned)atom);
}

// fp32 dot product of a 16-byte aligned row of D elements with e.
template <typename T, int D>
__device__ __forceinline__ float row_dot_f32(const T* row, const float* e);

template <>
__device__ __forceinline__ float row_dot_f32<__half, 128>(const __half* row, const float* e)
{
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        const uint4 q = reinterpret_cast<const uint4*>(row)[c];
        const __half2* h = reinterpret_cast<const __half2*>(&q);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(h[i]);
            acc[c & 3] = fmaf(f.x, e[c * 8 + 2 * i], acc[c & 3]);
            acc[c & 3] = fmaf(f.y, e[c * 8 + 2 * i + 1], acc[c & 3]);
        }
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}
template <>
__device__ __forceinline__ float row_dot_f32<__half, 64>(const __half* row, const float* e)
{
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 q = reinterpret_cast<const uint4*>(row)[c];
        const __half2* h = reinterpret_cast<const __half2*>(&q);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(h[i]);
            acc[c & 3] = fmaf(f.x, e[c * 8 + 2 * i], acc[c & 3]);
            acc[c & 3] = fmaf(f.y, e[c * 8 + 2 * i + 1], acc[c & 3]);
        }
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}
template <>
__device__ __forceinline__ float row_dot_f32<float, 128>(const float* row, const float* e)
{
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        const float4 q = reinterpret_cast<const float4*>(row)[c];
        acc[c & 3] = fmaf(q.x, e[c * 4], acc[c & 3]);
        acc[c & 3] = fmaf(q.y, e[c * 4 + 1], acc[c & 3]);
        acc[c & 3] = fmaf(q.z, e[c * 4 + 2], acc[c & 3]);
        acc[c & 3] = fmaf(q.w, e[c * 4 + 3], acc[c & 3]);
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}
template <>
__device__ __forceinline__ float row_dot_f32<float, 64>(const float* row, const float* e)
{
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        const float4 q = reinterpret_cast<const float4*>(row)[c];
        acc[c & 3] = fmaf(q.x, e[c * 4], acc[c & 3]);
        acc[c & 3] = fmaf(q.y, e[c * 4 + 1], acc[c & 3]);
        acc[c & 3] = fmaf(q.z, e[c * 4 + 2], acc[c & 3]);
        acc[c & 3] = fmaf(q.w, e[c * 4 + 3], acc[c & 3]);
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// Shared scratch of the selection (besides the key buffer).
struct Scratch {
    uint32_t* hist;             // [256]
    uint32_t* scan;             // [nwarps]
    uint32_t* misc;             // [4 + 2 * kCountSlots]
    unsigned long long* pref;   // [1]
};

// Reads the slot words of this vector's candidate list and resets them.
// Returns the total count (also left in misc[0]), or -1 if a region
// overflowed.  The regions' offsets in the gathered key array are left in
// misc[4 ..] and their offsets in the list in misc[4 + kCountSlots ..].
// Whole block calls it; ends with a barrier.
__device__ __forceinline__ int intake_counts(const GreedyArgs& a, size_t gv, Scratch sc)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int* counts = a.cand_count + gv * kCountSlots;
    if (warp == 0) {
        const uint32_t wd = (uint32_t)counts[lane];
        const int c = slot_count(wd);
        const int over = __any_sync(0xffffffffu, slot_over(wd));
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        sc.misc[4 + lane] = (uint32_t)(incl - c);
        sc.misc[4 + kCountSlots + lane] = (uint32_t)slot_offset(wd);
        if (lane == 31) sc.misc[0] = over ? 0xffffffffu : (uint32_t)incl;
        counts[lane] = 0;   // consumed: ready for the next call
    }
    __syncthreads();
    return (int)sc.misc[0];
}

// Fills keys[] with the candidates (or, on the slow path, every atom's key
// computed against xs) and returns how many.  Ends with a barrier.
template <typename T, int D>
__device__ __forceinline__ int intake_keys(const GreedyArgs& a, size_t gv, int count, int n, int N, const T* A,
                                           const float* xs, unsigned long long* keys, Scratch sc,
                                           long long* cnt)
{
    const int tid = threadIdx.x, nt = blockDim.x;
    int K;
    if (count >= n) {
        K = count;
        const unsigned long long* src = a.cand + gv * a.cap;
        for (int r = 0; r < kCountSlots; ++r) {
            const int off = (int)sc.misc[4 + r];
            const int len = (r + 1 < kCountSlots ? (int)sc.misc[5 + r] : K) - off;
            const int so = (int)sc.misc[4 + kCountSlots + r];
            for (int i = tid; i < len; i += nt) keys[off + i] = src[so + i];
        }
    } else {
        K = N;
        for (int j = tid; j < N; j += nt) keys[j] = screen_key(row_dot_f32<T, D>(A + (size_t)j * D, xs), j);
        if (tid == 0) atomicAdd((unsigned long long*)&cnt[kCntFallback], 1ull);
    }
    __syncthreads();
    return K;
}

// The n largest of K unique keys: writes pid[0..n) (atom ids, candidate
// order) and mag[0..n) (|r|).  Whole block calls it; ends with a barrier.
__device__ __forceinline__ void top_n(const unsigned long long* keys, int K, int n, int* pid, float* mag,
                                      Scratch sc)
{
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const int nw = nt >> 5;
    unsigned long long prefix = 0ull, mask = 0ull;
    uint32_t remaining = (uint32_t)n;
    int shift = 56;
    for (;; shift -= 8) {
        for (int i = tid; i < 256; i += nt) sc.hist[i] = 0;
        __syncthreads();
        for (int i0 = 0; i0 < K; i0 += nt) {
            // one shared-memory atomic per distinct bin per warp: keys crowd
            // into few bins in the first passes
            const int i = i0 + tid;
            const unsigned long long k = (i < K) ? keys[i] : 0ull;
            const bool in = (i < K) && (k & mask) == prefix;
            const uint32_t bin = in ? ((uint32_t)(k >> shift) & 0xffu) : 0x100u;
            const unsigned peers = __match_any_sync(0xffffffffu, bin);
            if (in && (__ffs(peers) - 1) == lane) atomicAdd(&sc.hist[bin], (uint32_t)__popc(peers));
        }
        __syncthreads();
        if (warp == 0) {
            const int hi = 255 - 8 * lane;
            uint32_t local = 0;
#pragma unroll
            for (int b = 0; b < 8; ++b) local += sc.hist[hi - b];
            uint32_t incl = local;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            const uint32_t above = incl - local;
            if (above < remaining && remaining <= incl) {
                uint32_t acc = above;
                for (int b = 0; b < 8; ++b) {
                    const uint32_t c = sc.hist[hi - b];
                    if (acc + c >= remaining) {
                        sc.pref[0] = prefix | ((unsigned long long)(hi - b) << shift);
                        sc.misc[1] = remaining - acc;
                        sc.misc[2] = (c == remaining - acc) ? 1u : 0u;   // boundary bin taken whole
                        break;
                    }
                    acc += c;
                }
            }
        }
        __syncthreads();
        prefix = sc.pref[0];
        remaining = sc.misc[1];
        mask |= 0xffull << shift;
        if (sc.misc[2] || shift == 0) break;
    }
    // selected: keys whose bits from `shift` up are >= prefix's
    uint32_t base = 0;
    const unsigned long long lim = prefix >> shift;
    for (int i0 = 0; i0 < K; i0 += nt) {
        const int i = i0 + tid;
        const unsigned long long k = (i < K) ? keys[i] : 0ull;
        const uint32_t f = (i < K && (k >> shift) >= lim) ? 1u : 0u;
        const unsigned bal = __ballot_sync(0xffffffffu, f);
        if (lane == 0) sc.scan[warp] = __popc(bal);
        __syncthreads();
        uint32_t before = 0, total = 0;
        for (int w = 0; w < nw; ++w) {
            const uint32_t c = sc.scan[w];
            before += (w < warp) ? c : 0u;
            total += c;
        }
        if (f) {
            const uint32_t pos = base + before + __popc(bal & ((1u << lane) - 1u));
            if (pos < (uint32_t)n) {
                pid[pos] = (int)(0xffffffffu - (uint32_t)(k & 0xffffffffull));
                mag[pos] = __uint_as_float((uint32_t)(k >> 32));
            }
        }
        base += total;
        __syncthreads();
    }
}

}  // namespace sel
}  // namespace fadkv
