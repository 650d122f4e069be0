// PL encode: one ridge fit over the Top-s atoms, no greedy iterations.
//
// "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding",
// Tables 1-4, the "PL (ours)" rows: the cheaper of the two coders, Cost 0.13
// of OMP in Table 4 against 0.19 for the greedy coder.  The pages do not
// spell it out; the reading this library takes is the one that cost
// supports -- screening (N d) plus a single fit over s atoms:
//   S = the s atoms of largest |r_j| (ties to the lower j), in ascending
//       atom order;
//   (G + diag(lambda_abs + lambda_rel G_ii)) c = D_S x, G = D_S D_S^T
//       (Table 5's ridge, the same as every greedy refit);
//   relres = ||x - D_S c|| / ||x||  (0 for x = 0).
//
// The Top-s set comes from the same screening and selection kernels as the
// greedy coder's pool (with n = s).  This kernel takes it per vector, either
// as atom ids in any order (the selection's pool) or as the FP32 path's
// candidate keys (already in ascending atom order), and does the fit.
//
// One warp per vector, everything in registers: lane l holds elements
// [E l, E l + E) of x and of each of the s atom rows (E = D / 32); the Gram
// entries and right-hand sides come from one mma.sync tile per 16 columns
// (binary16, s <= 8) or else from warp reductions; lane i holds row i of
// the fit matrix, and the Cholesky factorisation and both triangular solves
// run column by column with shuffles.  FP32 throughout.
#include <type_traits>

#include "fadkv_internal.cuh"

namespace fadkv {
namespace {

constexpr int kPlWarps = 8;

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// E consecutive elements of a row, widened to float (8- or 16-byte loads).
template <typename T, int E> struct Part;
template <> struct Part<__half, 4> {
    static __device__ __forceinline__ void load(const __half* p, float (&o)[4])
    {
        const uint2 q = *reinterpret_cast<const uint2*>(p);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&q.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&q.y));
        o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
    }
};
template <> struct Part<__half, 2> {
    static __device__ __forceinline__ void load(const __half* p, float (&o)[2])
    {
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(p));
        o[0] = a.x; o[1] = a.y;
    }
};
template <> struct Part<float, 4> {
    static __device__ __forceinline__ void load(const float* p, float (&o)[4])
    {
        const float4 a = *reinterpret_cast<const float4*>(p);
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    }
};
template <> struct Part<float, 2> {
    static __device__ __forceinline__ void load(const float* p, float (&o)[2])
    {
        const float2 a = *reinterpret_cast<const float2*>(p);
        o[0] = a.x; o[1] = a.y;
    }
};

template <typename T, int D, int SMAX>
__global__ void __launch_bounds__(kPlWarps * 32)
pl_fit_kernel(Shape sh, PlArgs a)
{
    pdl_begin();
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const long long gv = (long long)blockIdx.x * kPlWarps + (threadIdx.x >> 5);
    if (gv >= (long long)sh.G * a.Vc) return;
    const int g = (int)(gv / a.Vc), v = a.v0 + (int)(gv % a.Vc);
    const int s = sh.s, N = sh.N;
    const size_t out = ((size_t)g * a.V + v) * s;
    long long* cnt = a.counters + (size_t)g * kCntFields;

    // x, its norm, finiteness
    float xr[E];
    Part<T, E>::load((const T*)a.x + ((size_t)g * a.V + v) * D + E * lane, xr);
    bool bad = false;
    float xsq = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        bad |= !isfinite(xr[e]);
        xsq = fmaf(xr[e], xr[e], xsq);
    }
    xsq = warp_sum(xsq);

    // the Top-s ids: lane k < s holds one; a valid set is s distinct ids in [0, N)
    int id = 0x7fffffff;
    bool ok = true;
    if (lane < s) {
        if (a.pool) {
            id = a.pool[gv * s + lane];
        } else {
            id = (int)(0xffffffffu - (uint32_t)(a.cand[gv * a.cap + lane] & 0xffffffffull));
            ok = a.cand_count[gv * kCountSlots] == s;
        }
        ok = ok && id >= 0 && id < N;
    }
    if (__any_sync(0xffffffffu, bad)) {
        if (lane < s) {
            a.idx[out + lane] = -1;
            a.coef[out + lane] = 0.f;
        }
        if (lane == 0) {
            a.relres[(size_t)g * a.V + v] = __int_as_float(0x7fc00000);
            atomicAdd((unsigned long long*)&cnt[kCntNonfinite], 1ull);
            atomicOr((unsigned long long*)&cnt[kCntStatus], (unsigned long long)FADKV_DEV_NONFINITE_INPUT);
        }
        return;
    }
    if (!__all_sync(0xffffffffu, ok)) {
        // cannot come from the selection kernels; keeps every load in bounds
        if (lane < s) {
            a.idx[out + lane] = -1;
            a.coef[out + lane] = 0.f;
        }
        if (lane == 0) a.relres[(size_t)g * a.V + v] = __int_as_float(0x7fc00000);
        return;
    }

    // ascending order: sid[k] = the id of rank k (ranks of distinct ids)
    int rank = 0;
#pragma unroll
    for (int j = 0; j < SMAX; ++j) {
        const int o = __shfl_sync(0xffffffffu, id, j);
        rank += (j < s && o < id) ? 1 : 0;
    }
    int sid[SMAX];
#pragma unroll
    for (int k = 0; k < SMAX; ++k) {
        const unsigned who = __ballot_sync(0xffffffffu, lane < s && rank == k);
        sid[k] = who ? __shfl_sync(0xffffffffu, id, __ffs(who) - 1) : 0;
    }

    // the rows D_S, lane's E elements of each
    const T* A = (const T*)a.atoms + (size_t)g * N * D + E * lane;
    float rw[SMAX][E];
#pragma unroll
    for (int k = 0; k < SMAX; ++k) {
        if (k < s) {
            Part<T, E>::load(A + (size_t)sid[k] * D, rw[k]);
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) rw[k][e] = 0.f;
        }
    }

    // lane i: row i of the fit matrix (ar) and the right-hand side b_i
    const float la = sh.lambda_abs, lr = sh.lambda_rel;
    float ar[SMAX];
    float bi = 0.f;
    if constexpr (SMAX == 8 && std::is_same<T, __half>::value) {
        // binary16, s <= 8: G = D_S D_S^T and b = D_S x from one m16n8k16
        // tile per 16 columns -- A rows 0..7 the picked atoms, row 8 x (rows
        // 9..15 zero), B columns the same atoms (exact products, FP32 sums);
        // lane (g8, t4) ends with G[g8][2t4, 2t4+1] and, for g8 = 0,
        // b[2t4, 2t4+1]
        const int g8 = lane >> 2, t4 = lane & 3;
        int myrow = 0;
#pragma unroll
        for (int k = 0; k < SMAX; ++k)
            if (g8 == k) myrow = sid[k];
        const bool rowok = g8 < s;
        const __half* arow = (const __half*)a.atoms + ((size_t)g * N + myrow) * D + 2 * t4;
        const __half* xrow = (const __half*)a.x + ((size_t)g * a.V + v) * D + 2 * t4;
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kt = 0; kt < D / 16; ++kt) {
            uint32_t f[4];
            f[0] = rowok ? __ldg(reinterpret_cast<const uint32_t*>(arow + kt * 16)) : 0u;
            f[1] = g8 == 0 ? __ldg(reinterpret_cast<const uint32_t*>(xrow + kt * 16)) : 0u;
            f[2] = rowok ? __ldg(reinterpret_cast<const uint32_t*>(arow + kt * 16 + 8)) : 0u;
            f[3] = g8 == 0 ? __ldg(reinterpret_cast<const uint32_t*>(xrow + kt * 16 + 8)) : 0u;
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                "{%0,%1,%2,%3};\n"
                : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                : "r"(f[0]), "r"(f[1]), "r"(f[2]), "r"(f[3]), "r"(f[0]), "r"(f[2]));
        }
        // lane i gathers row i of G (from lanes 4i + j/2) and b_i (lane i/2)
#pragma unroll
        for (int j = 0; j < SMAX; ++j) {
            const float gij = __shfl_sync(0xffffffffu, (j & 1) ? c[1] : c[0], (4 * lane + (j >> 1)) & 31);
            ar[j] = (j < s && lane < s) ? (j == lane ? fmaf(gij, lr, gij) + la : gij) : 0.f;
        }
        const float be = __shfl_sync(0xffffffffu, c[2], (lane >> 1) & 31);
        const float bo = __shfl_sync(0xffffffffu, c[3], (lane >> 1) & 31);
        bi = lane < s ? ((lane & 1) ? bo : be) : 0.f;
    } else {
#pragma unroll
    for (int i = 0; i < SMAX; ++i) {
        ar[i] = 0.f;
        if (i < s) {
            float p = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) p = fmaf(rw[i][e], xr[e], p);
            p = warp_sum(p);
            if (lane == i) bi = p;
        }
    }
#pragma unroll
    for (int i = 0; i < SMAX; ++i) {
#pragma unroll
        for (int j = 0; j <= i; ++j) {
            if (i < s) {
                float p = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) p = fmaf(rw[i][e], rw[j][e], p);
                p = warp_sum(p);
                if (i == j) p = fmaf(p, lr, p) + la;
                if (lane == i) ar[j] = p;
                if (lane == j) ar[i] = p;
            }
        }
    }
    }

    // Cholesky A = L L^T in place: lane i's ar[k] becomes L_ik (k <= i)
    unsigned long long* status = (unsigned long long*)&cnt[kCntStatus];
#pragma unroll
    for (int k = 0; k < SMAX; ++k) {
        if (k < s) {
            float dk = __shfl_sync(0xffffffffu, ar[k], k);
            if (!(dk > 0.f)) {
                if (lane == 0) atomicOr(status, (unsigned long long)FADKV_DEV_NOT_SPD);
                dk = 1e-30f;
            }
            const float lkk = sqrtf(dk);
            const float lik = (lane == k) ? lkk : ar[k] / lkk;
            ar[k] = lik;
#pragma unroll
            for (int j = k + 1; j < SMAX; ++j) {
                const float ljk = __shfl_sync(0xffffffffu, lik, j);
                if (j < s && lane > k) ar[j] = fmaf(-lik, ljk, ar[j]);
            }
        }
    }
    // forward L y = b, y replicated in every lane (yv)
    float yv[SMAX];
#pragma unroll
    for (int k = 0; k < SMAX; ++k) {
        yv[k] = 0.f;
        if (k < s) {
            const float lkk = __shfl_sync(0xffffffffu, ar[k], k);
            const float yk = __shfl_sync(0xffffffffu, bi, k) / lkk;
            yv[k] = yk;
            if (lane > k) bi = fmaf(-ar[k], yk, bi);
        }
    }
    // backward L^T c = y (L_ki from lane k)
#pragma unroll
    for (int k = SMAX - 1; k >= 0; --k) {
        if (k < s) {
            const float lkk = __shfl_sync(0xffffffffu, ar[k], k);
            const float ck = yv[k] / lkk;
            yv[k] = ck;
#pragma unroll
            for (int i = 0; i < k; ++i) yv[i] = fmaf(-__shfl_sync(0xffffffffu, ar[i], k), ck, yv[i]);
        }
    }

    // residual and outputs
    float esq = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        float r = xr[e];
#pragma unroll
        for (int k = 0; k < SMAX; ++k)
            if (k < s) r = fmaf(-yv[k], rw[k][e], r);
        esq = fmaf(r, r, esq);
    }
    esq = warp_sum(esq);
    int my_id = 0;
    float my_c = 0.f;
#pragma unroll
    for (int k = 0; k < SMAX; ++k)
        if (lane == k) {
            my_id = sid[k];
            my_c = yv[k];
        }
    if (lane < s) {
        a.idx[out + lane] = my_id;
        a.coef[out + lane] = my_c;
    }
    if (lane == 0) a.relres[(size_t)g * a.V + v] = xsq > 0.f ? sqrtf(esq) / sqrtf(xsq) : 0.f;
}

template <typename T, int D>
cudaError_t launch_d(const Shape& sh, const PlArgs& a, cudaStream_t st)
{
    const long long warps = (long long)sh.G * a.Vc;
    const dim3 grid((unsigned)((warps + kPlWarps - 1) / kPlWarps));
    if (sh.s <= 8) return launch_pdl(pl_fit_kernel<T, D, 8>, grid, dim3(kPlWarps * 32), 0, st, sh, a);
    if (sh.s <= 16) return launch_pdl(pl_fit_kernel<T, D, 16>, grid, dim3(kPlWarps * 32), 0, st, sh, a);
    return launch_pdl(pl_fit_kernel<T, D, 32>, grid, dim3(kPlWarps * 32), 0, st, sh, a);
}

}  // namespace

cudaError_t launch_pl_fit(const Shape& sh, const PlArgs& a, cudaStream_t st)
{
    if (a.Vc <= 0) return cudaSuccess;
    if (sh.s < 1 || sh.s > 32 || (sh.d != 64 && sh.d != 128)) return cudaErrorInvalidValue;
    if (sh.dtype == FADKV_F16)
        return sh.d == 128 ? launch_d<__half, 128>(sh, a, st) : launch_d<__half, 64>(sh, a, st);
    return sh.d == 128 ? launch_d<float, 128>(sh, a, st) : launch_d<float, 64>(sh, a, st);
}

}  // namespace fadkv
