// Exact Top-n pool, then in-pool greedy selection with a ridge refit after
// every pick.
//
// "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding":
// abstract (screening-based sparse coding: a one-shot Top-n pool followed by
// lightweight coefficient refinement) and Table 5 (ridge parameter
// lambda = 1e-4 + 0.20 diag(G)).  Greedy selection inside the pool and the
// lower-index tie rule are conventions of this library.
//
// Per vector x:
//   pool P = the n largest candidate keys (bits(|r_j|) << 32 | ~j), i.e. the
//            n largest |r_j|, ties to the lower j.  The candidates are the
//            atoms that passed the screening filter; if there are fewer than
//            n of them (or the list overflowed) every score is recomputed
//            here on the FP32 pipe and all N atoms are candidates;
//   e_0 = x;  for k = 0..s-1:
//     j* = argmax_{j in P \ S} |<d_j, e_k>|   (ties: lower atom index)
//     S <- S + j*
//     A = G_SS + diag(lambda_abs + lambda_rel G_ii),  A c = D_S x
//     e_{k+1} = x - D_S c
//   relres = ||e_s|| / ||x||
// At k = 0 the correlations are <d_j, x> recomputed over the gathered pool.
// The Cholesky factor of A grows by one row per pick (the factor of a
// leading block is the leading block of the factor), so a refit costs O(k^2).
//
// This is the FP32-pipe kernel, used for binary32 dictionaries, for binary16
// dictionaries whose atom count is not a multiple of 128 (screened on the
// FP32 pipe) and for the pool test hook: one CTA
// (256 threads) per vector; the pool (exact Top-n from select.cuh) is
// gathered once into shared memory (rows padded by 16 bytes: eight threads
// reading eight consecutive rows hit distinct banks); thread t owns pool
// slots t, t+256, ...
#include <stdlib.h>
#include <string.h>

#include "select.cuh"

namespace fadkv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxPerThread = kMaxPool / kThreads;   // 4

struct GreedyLayout {
    size_t uni, xs, es, sa, lm, z, c, gram, fred, a0, kred, pid, sslot, hist, scan, misc, total;
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline GreedyLayout greedy_layout(int n, int d, int elem, int N, int cap)
{
    GreedyLayout L;
    size_t o = 0;
    const size_t pool = (size_t)n * (d * elem + 16);
    const size_t keys = (size_t)(N > cap ? N : cap) * 8;
    L.uni = o;   o += align_up(pool > keys ? pool : keys, 16);
    L.xs = o;    o += sizeof(float) * d;
    L.es = o;    o += sizeof(float) * d;
    L.sa = o;    o += sizeof(float) * kMaxS * d;
    L.lm = o;    o += sizeof(float) * kMaxS * kMaxS;
    L.z = o;     o += sizeof(float) * kMaxS;
    L.c = o;     o += sizeof(float) * kMaxS;
    L.gram = o;  o += sizeof(float) * (kMaxS + 4);
    L.fred = o;  o += sizeof(float) * kWarps * 2;
    L.a0 = o;    o += sizeof(float) * n;
    o = align_up(o, 8);
    L.kred = o;  o += sizeof(unsigned long long) * (kWarps + 2);
    L.pid = o;   o += sizeof(int) * n;
    L.sslot = o; o += sizeof(int) * kMaxS;
    L.hist = o;  o += sizeof(uint32_t) * 256;
    L.scan = o;  o += sizeof(uint32_t) * kWarps;
    L.misc = o;  o += sizeof(uint32_t) * (4 + 2 * kCountSlots);
    L.total = align_up(o, 16);
    return L;
}

// 16-byte chunk of a pool row converted to fp32 and dotted with e.
__device__ __forceinline__ float chunk_dot(const uint4& q, const float* e, const __half*)
{
    const __half2* h = reinterpret_cast<const __half2*>(&q);
    const float4 e0 = *reinterpret_cast<const float4*>(e);
    const float4 e1 = *reinterpret_cast<const float4*>(e + 4);
    const float2 a = __half22float2(h[0]), b = __half22float2(h[1]);
    const float2 c = __half22float2(h[2]), d = __half22float2(h[3]);
    float acc = a.x * e0.x;
    acc = fmaf(a.y, e0.y, acc);
    acc = fmaf(b.x, e0.z, acc);
    acc = fmaf(b.y, e0.w, acc);
    acc = fmaf(c.x, e1.x, acc);
    acc = fmaf(c.y, e1.y, acc);
    acc = fmaf(d.x, e1.z, acc);
    acc = fmaf(d.y, e1.w, acc);
    return acc;
}
__device__ __forceinline__ float chunk_dot(const uint4& q, const float* e, const float*)
{
    const float4 a = *reinterpret_cast<const float4*>(&q);
    const float4 e0 = *reinterpret_cast<const float4*>(e);
    float acc = a.x * e0.x;
    acc = fmaf(a.y, e0.y, acc);
    acc = fmaf(a.z, e0.z, acc);
    acc = fmaf(a.w, e0.w, acc);
    return acc;
}

// <row, e> over D elements; `row` is 16-byte aligned (shared or global).
template <typename T, int D>
__device__ __forceinline__ float row_dot(const T* row, const float* e)  // pool rows in shared memory
{
    constexpr int EPC = 16 / sizeof(T);   // elements per 16-byte chunk
    constexpr int CPR = D / EPC;          // chunks per row
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < CPR; ++c) {
        const uint4 q = reinterpret_cast<const uint4*>(row)[c];
        acc[c & 3] += chunk_dot(q, e + c * EPC, (const T*)nullptr);
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long t = __shfl_xor_sync(0xffffffffu, v, o);
        v = t > v ? t : v;
    }
    return v;
}

// Greedy key: larger |a| first, then the lower atom index (atom < 2^23);
// the low 10 bits carry the pool slot, which never decides the order since
// (|a|, atom) is unique.
__device__ __forceinline__ unsigned long long pick_key(float a, int atom, int slot)
{
    return ((unsigned long long)(__float_as_uint(a) & 0x7fffffffu) << 33) |
           ((unsigned long long)(0x7fffffu - (unsigned)atom) << 10) | (unsigned long long)slot;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
greedy_kernel(Shape sh, GreedyArgs a)
{
    const int vc = blockIdx.x, g = blockIdx.y;
    const int v = a.v0 + vc;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = sh.n, s = sh.s, N = sh.N;
    constexpr int RSB = D * (int)sizeof(T) + 16;   // padded pool row, bytes

    const GreedyLayout L = greedy_layout(n, D, sizeof(T), N, a.cap);
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char* P = smem + L.uni;
    unsigned long long* keys = (unsigned long long*)(smem + L.uni);
    float* xs = (float*)(smem + L.xs);
    float* es = (float*)(smem + L.es);
    float* SA = (float*)(smem + L.sa);
    float* Lm = (float*)(smem + L.lm);
    float* zz = (float*)(smem + L.z);
    float* cc = (float*)(smem + L.c);
    float* gram = (float*)(smem + L.gram);
    float* fred = (float*)(smem + L.fred);
    float* a0 = (float*)(smem + L.a0);
    unsigned long long* kred = (unsigned long long*)(smem + L.kred);
    int* pid = (int*)(smem + L.pid);
    int* sslot = (int*)(smem + L.sslot);
    uint32_t* hist = (uint32_t*)(smem + L.hist);
    uint32_t* scan_ws = (uint32_t*)(smem + L.scan);
    uint32_t* misc = (uint32_t*)(smem + L.misc);

    const size_t gv = (size_t)g * a.Vc + vc;
    const T* X = (const T*)a.x + ((size_t)g * a.V + v) * D;
    const T* A = (const T*)a.atoms + (size_t)g * N * D;
    long long* cnt = a.counters + (size_t)g * kCntFields;

    // ---- x, its norm and finiteness; the candidate count ----
    float xsq = 0.f;
    int bad = 0;
    for (int t = tid; t < D; t += kThreads) {
        const float xv = to_f32(X[t]);
        xs[t] = xv;
        es[t] = xv;
        bad |= !isfinite(xv);
        xsq = fmaf(xv, xv, xsq);
    }
    xsq = warp_sum(xsq);
    if (lane == 0) fred[warp] = xsq;
    sel::Scratch sc{hist, scan_ws, misc, kred + kWarps};
    int count = -1;                               // < n: exact slow path
    if (a.pool_in) {
        if (tid == 0) misc[0] = (uint32_t)a.pool_in[gv * n];
    } else {
        count = sel::intake_counts(a, gv, sc);
    }
    bad = __syncthreads_or(bad);
    const bool have_pool = a.pool_in && (int)misc[0] != -2;
    if (bad) {
        if (a.pool_out) {
            for (int i = tid; i < n; i += kThreads) a.pool_out[((size_t)g * a.V + v) * n + i] = -1;
            return;
        }
        for (int k = tid; k < s; k += kThreads) {
            a.idx[((size_t)g * a.V + v) * s + k] = -1;
            a.coef[((size_t)g * a.V + v) * s + k] = 0.f;
        }
        if (tid == 0) {
            a.relres[(size_t)g * a.V + v] = __int_as_float(0x7fc00000);
            atomicAdd((unsigned long long*)&cnt[kCntNonfinite], 1ull);
            atomicOr((unsigned long long*)&cnt[kCntStatus], (unsigned long long)FADKV_DEV_NONFINITE_INPUT);
        }
        return;
    }
    float xnorm2 = 0.f;
    for (int w = 0; w < kWarps; ++w) xnorm2 += fred[w];

    // ---- the pool ----
    if (have_pool) {
        for (int i = tid; i < n; i += kThreads) pid[i] = a.pool_in[gv * n + i];
    } else {
        const int K = sel::intake_keys<T, D>(a, gv, count, n, N, A, xs, keys, sc, cnt);
        sel::top_n(keys, K, n, pid, a0, sc);
    }
    __syncthreads();

    // ---- the pool's atoms into shared memory (over the keys) ----
    {
        constexpr int CPR = D * (int)sizeof(T) / 16;
        for (int c = tid; c < n * CPR; c += kThreads) {
            const int i = c / CPR, part = c % CPR;
            const uint4 q = reinterpret_cast<const uint4*>(A + (size_t)pid[i] * D)[part];
            *reinterpret_cast<uint4*>(P + (size_t)i * RSB + part * 16) = q;
        }
    }
    __syncthreads();
    // step-0 correlations <d_j, x> of the pool on the FP32 pipe
    float av[kMaxPerThread];
    int aid[kMaxPerThread];
    unsigned picked = 0;
#pragma unroll
    for (int m = 0; m < kMaxPerThread; ++m) {
        const int i = tid + m * kThreads;
        av[m] = (i < n) ? row_dot<T, D>((const T*)(P + (size_t)i * RSB), xs) : 0.f;
        aid[m] = (i < n) ? pid[i] : 0;
        if (i < n) a0[i] = fabsf(av[m]);
    }
    if (a.pool_out) {
        __syncthreads();
        for (int i = tid; i < n; i += kThreads) {
            a.pool_out[((size_t)g * a.V + v) * n + i] = pid[i];
            if (a.pool_r_out) a.pool_r_out[((size_t)g * a.V + v) * n + i] = a0[i];
        }
        return;
    }

    const float la = sh.lambda_abs, lr = sh.lambda_rel;
    for (int k = 0; k < s; ++k) {
        // ---- argmax over the unpicked pool atoms ----
        unsigned long long best = 0ull;
#pragma unroll
        for (int m = 0; m < kMaxPerThread; ++m) {
            const int i = tid + m * kThreads;
            if (i < n && !((picked >> m) & 1u)) {
                const unsigned long long key = pick_key(av[m], aid[m], i);
                best = key > best ? key : best;
            }
        }
        best = warp_max_u64(best);
        if (lane == 0) kred[warp] = best;
        __syncthreads();
        unsigned long long win = 0ull;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) win = kred[w] > win ? kred[w] : win;
        const int slot = (int)(win & 0x3ffull);
        if ((slot % kThreads) == tid) picked |= 1u << (slot / kThreads);
        if (tid == 0) sslot[k] = slot;
        // the picked atom -> SA[k] (fp32)
        {
            const T* row = (const T*)(P + (size_t)slot * RSB);
            for (int t = tid; t < D; t += kThreads) SA[k * D + t] = to_f32(row[t]);
        }
        __syncthreads();

        // ---- Gram row of the new atom and its right-hand side ----
        // gram[i] = <a_i, a_k> for i <= k; gram[k+1] = <a_k, x>
        for (int i = warp; i <= k + 1; i += kWarps) {
            const float* u = (i <= k) ? SA + i * D : xs;
            const float* w = SA + k * D;
            float acc = 0.f;
            for (int t = lane; t < D; t += 32) acc = fmaf(u[t], w[t], acc);
            acc = warp_sum(acc);
            if (lane == 0) gram[i] = acc;
        }
        __syncthreads();

        // ---- Cholesky row k, forward and back substitution (one thread) ----
        if (tid == 0) {
            float* Lk = Lm + k * kMaxS;
            for (int i = 0; i < k; ++i) {
                float val = gram[i];
                const float* Li = Lm + i * kMaxS;
                for (int m = 0; m < i; ++m) val = fmaf(-Li[m], Lk[m], val);
                Lk[i] = val / Li[i];
            }
            float dk = fmaf(gram[k], lr, gram[k]) + la;
            for (int m = 0; m < k; ++m) dk = fmaf(-Lk[m], Lk[m], dk);
            if (!(dk > 0.f)) {
                atomicOr((unsigned long long*)&cnt[kCntStatus], (unsigned long long)FADKV_DEV_NOT_SPD);
                dk = 1e-30f;
            }
            const float lkk = sqrtf(dk);
            Lk[k] = lkk;
            float zk = gram[k + 1];
            for (int m = 0; m < k; ++m) zk = fmaf(-Lk[m], zz[m], zk);
            zz[k] = zk / lkk;
            for (int i = k; i >= 0; --i) {
                float val = zz[i];
                for (int m = i + 1; m <= k; ++m) val = fmaf(-Lm[m * kMaxS + i], cc[m], val);
                cc[i] = val / Lm[i * kMaxS + i];
            }
        }
        __syncthreads();

        // ---- residual e = x - D_S c ----
        for (int t = tid; t < D; t += kThreads) {
            float val = xs[t];
            for (int i = 0; i <= k; ++i) val = fmaf(-cc[i], SA[i * D + t], val);
            es[t] = val;
        }
        __syncthreads();

        // ---- correlations with the new residual ----
        if (k + 1 < s) {
#pragma unroll
            for (int m = 0; m < kMaxPerThread; ++m) {
                const int i = tid + m * kThreads;
                if (i < n) av[m] = row_dot<T, D>((const T*)(P + (size_t)i * RSB), es);
            }
        }
    }

    // ---- outputs ----
    float esq = 0.f;
    for (int t = tid; t < D; t += kThreads) esq = fmaf(es[t], es[t], esq);
    esq = warp_sum(esq);
    if (lane == 0) fred[kWarps + warp] = esq;
    __syncthreads();
    if (tid == 0) {
        float e2 = 0.f;
        for (int w = 0; w < kWarps; ++w) e2 += fred[kWarps + w];
        a.relres[(size_t)g * a.V + v] = (xnorm2 > 0.f) ? sqrtf(e2) / sqrtf(xnorm2) : 0.f;
    }
    for (int k = tid; k < s; k += kThreads) {
        a.idx[((size_t)g * a.V + v) * s + k] = pid[sslot[k]];
        a.coef[((size_t)g * a.V + v) * s + k] = cc[k];
    }
}

template <typename T, int D>
cudaError_t launch_t(const Shape& sh, const GreedyArgs& a, cudaStream_t st)
{
    const size_t smem = greedy_layout(sh.n, D, sizeof(T), sh.N, a.cap).total;
    auto k = greedy_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.Vc, sh.G);
    k<<<grid, kThreads, smem, st>>>(sh, a);
    return cudaGetLastError();
}

}  // namespace

size_t greedy_smem_bytes(const Shape& sh)
{
    return greedy_layout(sh.n, sh.d, sh.dtype == FADKV_F16 ? 2 : 4, sh.N, cand_cap(sh.n)).total;
}

cudaError_t launch_greedy(const Shape& sh, const GreedyArgs& a, cudaStream_t st)
{
    if (a.Vc <= 0) return cudaSuccess;
    if (sh.dtype == FADKV_F16) {
        if (sh.d == 128) return launch_t<__half, 128>(sh, a, st);
        return launch_t<__half, 64>(sh, a, st);
    }
    if (sh.d == 128) return launch_t<float, 128>(sh, a, st);
    return launch_t<float, 64>(sh, a, st);
}

}  // namespace fadkv
