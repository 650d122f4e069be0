// In-pool greedy selection with a ridge refit after every pick -- binary16
// dictionaries, pool correlations on the tensor cores.
//
// "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding":
// abstract (screening-based sparse coding: a one-shot Top-n pool followed by
// lightweight coefficient refinement) and Table 5 (ridge parameter
// lambda = 1e-4 + 0.20 diag(G)).  Greedy selection inside the pool and the
// lower-index tie rule are conventions of this library.
//
// Per vector x with pool P (exact Top-n from select.cuh):
//   e_0 = x;  for k = 0..s-1:
//     j* = argmax_{j in P \ S} |<d_j, e_k>|   (ties: lower atom index)
//     S <- S + j*
//     A = G_SS + diag(lambda_abs + lambda_rel G_ii),  A c = D_S x
//     e_{k+1} = x - D_S c
//   relres = ||e_s|| / ||x||
//
// One CTA of NW warps per vector; warp w owns pool slots SPW*w .. SPW*w+SPW-1
// (SPW = 16 * m16-tiles per warp).  The
// pool's binary16 atoms stay in registers for the whole greedy loop, as the
// A fragments of mma.sync.m16n8k16 (rows = atoms).  Every pass multiplies
// them by an 8-column B operand (fp32 accumulation):
//   columns 0, 1: the residual split in two binary16 terms, e 2^p = hi + lo
//                 (p from ||x||, so no term overflows; the split leaves a
//                 relative error near 2^-22): <d_j, e> = (acc_0 + acc_1) 2^-p;
//   column 2:     the atom picked last (exact in binary16): its Gram column
//                 <d_j, d_pick> over the pool, kept in shared memory, so the
//                 next refit reads its Gram row instead of computing it.
// The first pass takes x instead of e: the signed scores r_j of the pool
// (step-0 correlations and the refit's right-hand sides).  Inside each
// 32-element block of the head dimension, thread t of a fragment row holds
// the 8 consecutive elements 8t..8t+7 (one 16-byte load) -- a permutation of
// the contraction index, applied identically to A and B, so the products are
// unchanged.  The refit updates the inverse Cholesky factor of A by one row
// per pick on one warp (see refit_warp), overlapped with the copy of the
// picked atom.  Three barriers per step.
#include <stdlib.h>
#include <string.h>

#include "select.cuh"

namespace fadkv {
namespace {

template <int D>
struct MmaLayout {
    size_t keys, xs, es, sa, bsm, lm, z, c, gram, gcol, rsl, nrm, fred, kred, pid, mag, sslot, hist, scan, misc, pref,
        total;
};

__host__ __device__ inline size_t al(size_t v, size_t a) { return (v + a - 1) / a * a; }

template <int D>
__host__ __device__ inline MmaLayout<D> mma_layout(int n_pad, int N, int cap, int nw)
{
    MmaLayout<D> L;
    size_t o = 0;
    L.keys = o;  o += al((size_t)(N > cap ? N : cap) * 8, 16);
    L.xs = o;    o += 4 * D;
    L.es = o;    o += 4 * D;
    L.sa = o;    o += 4 * (size_t)kMaxS * D;
    L.bsm = o;   o += 2 * 8 * D;                 // B operand: 8 columns x D binary16
    L.lm = o;    o += 4 * kMaxS * (kMaxS + 1);    // inverse Cholesky factor, padded rows
    L.z = o;     o += 4 * kMaxS;
    L.c = o;     o += 4 * kMaxS;
    L.gram = o;  o += 4 * kMaxS;                 // l of the current refit
    L.gcol = o;  o += 4 * (size_t)n_pad * kMaxS; // Gram columns of the picks: [slot][i]
    L.rsl = o;   o += 4 * (size_t)n_pad;         // signed scores of the pool
    L.nrm = o;   o += 4 * (size_t)n_pad;         // squared norms of the pool atoms
    L.fred = o;  o += 4 * 2 * nw;
    o = al(o, 8);
    L.kred = o;  o += 8 * (nw + 1);
    L.pref = o;  o += 8;
    L.pid = o;   o += 4 * (size_t)n_pad;
    L.mag = o;   o += 4 * (size_t)n_pad;
    L.sslot = o; o += 4 * kMaxS;
    L.hist = o;  o += 4 * 256;
    L.scan = o;  o += 4 * nw;
    L.misc = o;  o += 4 * (4 + 2 * kCountSlots);
    L.total = al(o, 16);
    return L;
}

__device__ __forceinline__ void hmma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}


// Larger |a| first, then the lower atom index (atom < 2^23); the low 10
// bits carry the pool slot, which never decides the order.
__device__ __forceinline__ unsigned long long pick_key(float a, int atom, int slot)
{
    return ((unsigned long long)(__float_as_uint(a) & 0x7fffffffu) << 33) |
           ((unsigned long long)(0x7fffffu - (unsigned)atom) << 10) | (unsigned long long)slot;
}

__device__ __forceinline__ void put8(float* dst, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3)
{
    const uint32_t w[4] = {w0, w1, w2, w3};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        dst[2 * i] = f.x;
        dst[2 * i + 1] = f.y;
    }
}

// One pick of the ridge refit, by one warp.  With A = G_SS + diag(lambda_abs
// + lambda_rel G_ii) = L L^T, the warp keeps M = L^-1 (lower triangular,
// rows padded to kMaxS + 1 floats), z = M b and c = M^T z = A^-1 b.  Adding
// pick k with Gram row g = <d_i, d_new> (i < k), gkk = ||d_new||^2 and
// bk = <d_new, x>:
//   l = M g,  L_kk = sqrt(gkk (1 + lambda_rel) + lambda_abs - l.l),
//   z_k = (bk - l.z) / L_kk,  w = -(l^T M) / L_kk  (the new row of M),
//   c <- c + z_k w,  c_k = z_k / L_kk.
// Lane i owns row i (for l) and column i (for w and c): O(k) work per lane.
constexpr int kMS = kMaxS + 1;   // padded row stride of M (conflict-free rows and columns)

template <int SMAX>
__device__ __forceinline__ void refit_warp(int k, int lane, const float* grow, float gkk, float bk, float la, float lr,
                                           float* M, float* lbuf, float* zz, float* cc,
                                           unsigned long long* status)
{
    float li = 0.f;
#pragma unroll
    for (int m = 0; m < SMAX; ++m)
        if (m <= lane && lane < k) li = fmaf(M[lane * kMS + m], grow[m], li);
    if (lane < k) lbuf[lane] = li;
    float ll = li * li;
    float lz = (lane < k) ? li * zz[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ll += __shfl_xor_sync(0xffffffffu, ll, o);
        lz += __shfl_xor_sync(0xffffffffu, lz, o);
    }
    float dk = fmaf(gkk, lr, gkk) + la - ll;
    if (!(dk > 0.f)) {
        if (lane == 0) atomicOr(status, (unsigned long long)FADKV_DEV_NOT_SPD);
        dk = 1e-30f;
    }
    const float inv = __frcp_rn(sqrtf(dk));
    const float zk = (bk - lz) * inv;
    __syncwarp();
    if (lane < k) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < SMAX; ++i)
            if (i >= lane && i < k) acc = fmaf(lbuf[i], M[i * kMS + lane], acc);
        const float w = -acc * inv;
        M[k * kMS + lane] = w;
        cc[lane] = fmaf(zk, w, cc[lane]);
    } else if (lane == k) {
        M[k * kMS + k] = inv;
        zz[k] = zk;
        cc[k] = zk * inv;
    }
    __syncwarp();
}

// NW warps per vector, MT m16 tiles (16 pool slots each) per warp; with
// MT <= 2 the head dimension is split across two accumulator sets (KS = 2)
// so each warp runs 2*MT independent chains of KP/KS*2 dependent MMAs.
template <int NW, int MT>
struct MinBlocks {
    static constexpr int value = (NW * 32 <= 128) ? 3 : ((NW * 32 <= 256 && MT <= 2) ? 2 : 1);
};

template <int D, int NW, int MT, int SMAX>
__global__ void __launch_bounds__(NW * 32, MinBlocks<NW, MT>::value)
greedy_mma_kernel(Shape sh, GreedyArgs a)
{
    constexpr int KT = D / 16, KP = D / 32, NT = NW * 32;
    constexpr int SPW = MT * 16;                 // pool slots per warp
    constexpr int KS = (MT <= 2) ? 2 : 1;        // accumulator sets along the head dimension
    const int vc = blockIdx.x, g = blockIdx.y;
    const int v = a.v0 + vc;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int n = sh.n, s = sh.s, N = sh.N;
    const int n_pad = NW * SPW;

    const MmaLayout<D> L = mma_layout<D>(n_pad, N, a.cap, NW);
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned long long* keys = (unsigned long long*)(smem + L.keys);
    float* xs = (float*)(smem + L.xs);
    float* es = (float*)(smem + L.es);
    float* SA = (float*)(smem + L.sa);
    __half* Bsm = (__half*)(smem + L.bsm);
    float* Lm = (float*)(smem + L.lm);
    float* zz = (float*)(smem + L.z);
    float* cc = (float*)(smem + L.c);
    float* gram = (float*)(smem + L.gram);
    float* fred = (float*)(smem + L.fred);
    unsigned long long* kred = (unsigned long long*)(smem + L.kred);
    int* pid = (int*)(smem + L.pid);
    float* mag = (float*)(smem + L.mag);
    int* sslot = (int*)(smem + L.sslot);
    sel::Scratch sc{(uint32_t*)(smem + L.hist), (uint32_t*)(smem + L.scan), (uint32_t*)(smem + L.misc),
                    (unsigned long long*)(smem + L.pref)};

    const size_t gv = (size_t)g * a.Vc + vc;
    const __half* X = (const __half*)a.x + ((size_t)g * a.V + v) * D;
    const __half* Aglob = (const __half*)a.atoms + (size_t)g * N * D;
    long long* cnt = a.counters + (size_t)g * kCntFields;

    // ---- x, its norm and finiteness ----
    float xsq = 0.f;
    int bad = 0;
    for (int t = tid; t < D; t += NT) {
        const float xv = __half2float(X[t]);
        xs[t] = xv;
        bad |= !isfinite(xv);
        xsq = fmaf(xv, xv, xsq);
    }
    xsq = warp_sum(xsq);
    if (lane == 0) fred[warp] = xsq;
    int count = -1;                               // < n: exact slow path
    if (a.pool_in) {
        if (tid == 0) sc.misc[0] = (uint32_t)a.pool_in[gv * n];
    } else {
        count = sel::intake_counts(a, gv, sc);
    }
    bad = __syncthreads_or(bad);
    const bool have_pool = a.pool_in && (int)sc.misc[0] != -2;
    if (bad) {
        if (a.pool_out) {
            for (int i = tid; i < n; i += NT) a.pool_out[((size_t)g * a.V + v) * n + i] = -1;
            return;
        }
        for (int k = tid; k < s; k += NT) {
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
    for (int w = 0; w < NW; ++w) xnorm2 += fred[w];

    // ---- the pool ----
    if (have_pool) {
        for (int i = tid; i < n; i += NT) pid[i] = a.pool_in[gv * n + i];
        __syncthreads();
    } else {
        const int K = sel::intake_keys<__half, D>(a, gv, count, n, N, Aglob, xs, keys, sc, cnt);
        sel::top_n(keys, K, n, pid, mag, sc);
    }
    if (a.pool_out) {
        // |r| of the pool members comes from the first MMA pass below
        for (int i = tid; i < n; i += NT) a.pool_out[((size_t)g * a.V + v) * n + i] = pid[i];
        if (!a.pool_r_out) return;
    }

    // ---- pool atoms -> A fragments (registers), squared norms ----
    float* gcol = (float*)(smem + L.gcol);
    float* rsl = (float*)(smem + L.rsl);
    float* nrm = (float*)(smem + L.nrm);
    uint32_t Af[MT][KT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const int s0 = warp * SPW + mt * 16 + g8;
        const int r0 = (s0 < n) ? pid[s0] : -1;
        const int r1 = (s0 + 8 < n) ? pid[s0 + 8] : -1;
        float n0 = 0.f, n1 = 0.f;
#pragma unroll
        for (int kp = 0; kp < KP; ++kp) {
            uint4 q0 = make_uint4(0, 0, 0, 0), q1 = make_uint4(0, 0, 0, 0);
            if (r0 >= 0) q0 = *reinterpret_cast<const uint4*>(Aglob + (size_t)r0 * D + 32 * kp + 8 * t4);
            if (r1 >= 0) q1 = *reinterpret_cast<const uint4*>(Aglob + (size_t)r1 * D + 32 * kp + 8 * t4);
            Af[mt][2 * kp][0] = q0.x;
            Af[mt][2 * kp][2] = q0.y;
            Af[mt][2 * kp + 1][0] = q0.z;
            Af[mt][2 * kp + 1][2] = q0.w;
            Af[mt][2 * kp][1] = q1.x;
            Af[mt][2 * kp][3] = q1.y;
            Af[mt][2 * kp + 1][1] = q1.z;
            Af[mt][2 * kp + 1][3] = q1.w;
            const __half2* h0 = reinterpret_cast<const __half2*>(&q0);
            const __half2* h1 = reinterpret_cast<const __half2*>(&q1);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f0 = __half22float2(h0[i]), f1 = __half22float2(h1[i]);
                n0 = fmaf(f0.x, f0.x, fmaf(f0.y, f0.y, n0));
                n1 = fmaf(f1.x, f1.x, fmaf(f1.y, f1.y, n1));
            }
        }
        n0 += __shfl_xor_sync(0xffffffffu, n0, 1);
        n0 += __shfl_xor_sync(0xffffffffu, n0, 2);
        n1 += __shfl_xor_sync(0xffffffffu, n1, 1);
        n1 += __shfl_xor_sync(0xffffffffu, n1, 2);
        if (t4 == 0) {
            nrm[s0] = n0;
            nrm[s0 + 8] = n1;
        }
    }

    // scale 2^p with ||e|| <= ||x|| < 2^ex: |e_t| 2^p < 2^14 (no binary16 overflow)
    int ex = 0;
    frexpf(sqrtf(xnorm2), &ex);
    const float scale = (xnorm2 > 0.f) ? ldexpf(1.f, 14 - ex) : 1.f;
    const float inv_scale = (xnorm2 > 0.f) ? ldexpf(1.f, ex - 14) : 1.f;

    // B operand of the first pass: x split into columns 0, 1; the rest 0
    for (int i = tid; i < 8 * D; i += NT) {
        __half val = __float2half_rn(0.f);
        if (i < 2 * D) {
            const float sv = xs[i % D] * scale;
            const __half hi = __float2half_rn(sv);
            val = (i < D) ? hi : __float2half_rn(sv - __half2float(hi));
        }
        Bsm[i] = val;
    }
    __syncthreads();

    float acc[MT][4];
    auto mma_pass = [&]() {
        float part[MT][KS][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int r = 0; r < 4; ++r) part[mt][ks][r] = 0.f;
#pragma unroll
        for (int kp = 0; kp < KP; ++kp) {
            const uint4 qb = *reinterpret_cast<const uint4*>(Bsm + g8 * D + 32 * kp + 8 * t4);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                hmma(part[mt][kp % KS], Af[mt][2 * kp], qb.x, qb.y);
                hmma(part[mt][kp % KS], Af[mt][2 * kp + 1], qb.z, qb.w);
            }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                float t = part[mt][0][r];
#pragma unroll
                for (int ks = 1; ks < KS; ++ks) t += part[mt][ks][r];
                acc[mt][r] = t;
            }
    };

    // ---- first pass: signed scores of the pool, step-0 correlations ----
    // lanes with t4 == 0 own slots m = 2*mt + h -> SPW*warp + 16*mt + 8*h + g8
    mma_pass();
    float av[2 * MT];
    unsigned live = 0;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const float r0 = (acc[mt][0] + acc[mt][1]) * inv_scale;
        const float r1 = (acc[mt][2] + acc[mt][3]) * inv_scale;
        av[2 * mt] = r0;
        av[2 * mt + 1] = r1;
        const int s0 = warp * SPW + mt * 16 + g8;
        if (t4 == 0) {
            rsl[s0] = r0;
            rsl[s0 + 8] = r1;
            if (s0 < n) live |= 1u << (2 * mt);
            if (s0 + 8 < n) live |= 1u << (2 * mt + 1);
        }
    }
    if (a.pool_out) {
        __syncthreads();
        for (int i = tid; i < n; i += NT) a.pool_r_out[((size_t)g * a.V + v) * n + i] = fabsf(rsl[i]);
        return;
    }
    // the first argmax: best live slot of this warp -> kred[warp]
    auto warp_best = [&]() {
        unsigned long long best = 0ull;
        if (t4 == 0) {
#pragma unroll
            for (int m = 0; m < 2 * MT; ++m) {
                if ((live >> m) & 1u) {
                    const int sl = warp * SPW + (m >> 1) * 16 + (m & 1) * 8 + g8;
                    const unsigned long long key = pick_key(av[m], pid[sl], sl);
                    best = key > best ? key : best;
                }
            }
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            const unsigned long long t = __shfl_xor_sync(0xffffffffu, best, o);
            best = t > best ? t : best;
        }
        if (lane == 0) kred[warp] = best;
    };
    warp_best();
    __syncthreads();

    const float la = sh.lambda_abs, lr = sh.lambda_rel;
    unsigned long long* status = (unsigned long long*)&cnt[kCntStatus];
    for (int k = 0; k < s; ++k) {
        // ---- the pick: best of the warps' bests ----
        unsigned long long win = 0ull;
#pragma unroll
        for (int w = 0; w < NW; ++w) win = kred[w] > win ? kred[w] : win;
        const int slot = (int)(win & 0x3ffull);
        const int w_o = slot / SPW, mt_o = (slot % SPW) >> 4, h_o = (slot >> 3) & 1, g_o = slot & 7;

        // ---- the picked atom: fp32 copy SA[k] and B column 2 (owner lanes) ----
        if (warp == w_o && g8 == g_o) {
            if (t4 == 0) live &= ~(1u << (2 * mt_o + h_o));
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                if (mt == mt_o) {
#pragma unroll
                    for (int kp = 0; kp < KP; ++kp) {
                        const uint32_t w0 = h_o ? Af[mt][2 * kp][1] : Af[mt][2 * kp][0];
                        const uint32_t w1 = h_o ? Af[mt][2 * kp][3] : Af[mt][2 * kp][2];
                        const uint32_t w2 = h_o ? Af[mt][2 * kp + 1][1] : Af[mt][2 * kp + 1][0];
                        const uint32_t w3 = h_o ? Af[mt][2 * kp + 1][3] : Af[mt][2 * kp + 1][2];
                        put8(SA + k * D + 32 * kp + 8 * t4, w0, w1, w2, w3);
                        *reinterpret_cast<uint4*>(Bsm + 2 * D + 32 * kp + 8 * t4) = make_uint4(w0, w1, w2, w3);
                    }
                }
            }
        }
        // ---- ridge refit, by the warp after the owner warp ----
        if (warp == (w_o + 1) % NW) {
            if (lane == 0) sslot[k] = slot;
            refit_warp<SMAX>(k, lane, gcol + (size_t)slot * kMaxS, nrm[slot], rsl[slot], la, lr, Lm, gram, zz, cc,
                             status);
        }
        __syncthreads();

        // ---- residual e = x - D_S c, split into B columns 0, 1 ----
        for (int t = tid; t < D; t += NT) {
            float val = xs[t];
#pragma unroll
            for (int i = 0; i < SMAX; ++i)
                if (i <= k) val = fmaf(-cc[i], SA[i * D + t], val);
            es[t] = val;
            const float sv = val * scale;
            const __half hi = __float2half_rn(sv);
            Bsm[t] = hi;
            Bsm[D + t] = __float2half_rn(sv - __half2float(hi));
        }
        if (k + 1 == s) break;
        __syncthreads();

        // ---- correlations with the new residual; Gram column of the pick ----
        mma_pass();
        if (t4 == 0) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                av[2 * mt] = (acc[mt][0] + acc[mt][1]) * inv_scale;
                av[2 * mt + 1] = (acc[mt][2] + acc[mt][3]) * inv_scale;
            }
        } else if (t4 == 1) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const int s0 = warp * SPW + mt * 16 + g8;
                gcol[(size_t)s0 * kMaxS + k] = acc[mt][0];
                gcol[(size_t)(s0 + 8) * kMaxS + k] = acc[mt][2];
            }
        }
        warp_best();
        __syncthreads();
    }
    __syncthreads();

    // ---- outputs ----
    float esq = 0.f;
    for (int t = tid; t < D; t += NT) esq = fmaf(es[t], es[t], esq);
    esq = warp_sum(esq);
    if (lane == 0) fred[NW + warp] = esq;
    __syncthreads();
    if (tid == 0) {
        float e2 = 0.f;
        for (int w = 0; w < NW; ++w) e2 += fred[NW + w];
        a.relres[(size_t)g * a.V + v] = (xnorm2 > 0.f) ? sqrtf(e2) / sqrtf(xnorm2) : 0.f;
    }
    for (int k = tid; k < s; k += NT) {
        a.idx[((size_t)g * a.V + v) * s + k] = pid[sslot[k]];
        a.coef[((size_t)g * a.V + v) * s + k] = cc[k];
    }
}

template <int D, int NW, int MT, int SMAX>
cudaError_t launch_t(const Shape& sh, const GreedyArgs& a, cudaStream_t st)
{
    const size_t smem = mma_layout<D>(NW * MT * 16, sh.N, a.cap, NW).total;
    auto k = greedy_mma_kernel<D, NW, MT, SMAX>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.Vc, sh.G);
    k<<<grid, NW * 32, smem, st>>>(sh, a);
    return cudaGetLastError();
}

template <int D, int NW, int MT>
cudaError_t launch_s(const Shape& sh, const GreedyArgs& a, cudaStream_t st)
{
    if (sh.s <= 8) return launch_t<D, NW, MT, 8>(sh, a, st);
    if (sh.s <= 16) return launch_t<D, NW, MT, 16>(sh, a, st);
    return launch_t<D, NW, MT, 32>(sh, a, st);
}

// Warps per vector: 2 m16 tiles (32 pool slots) per warp by default;
// FADKV_GREEDY_TILES=4 selects 4 tiles per warp (fewer, register-heavier warps).
int tiles_per_warp()
{
    const char* f = getenv("FADKV_GREEDY_TILES");
    return (f && strcmp(f, "4") == 0) ? 4 : 2;
}

template <int D>
cudaError_t launch_d(const Shape& sh, const GreedyArgs& a, cudaStream_t st)
{
    if (tiles_per_warp() == 4) {
        if (sh.n <= 256) return launch_s<D, 4, 4>(sh, a, st);
        if (sh.n <= 512) return launch_s<D, 8, 4>(sh, a, st);
        return launch_s<D, 16, 4>(sh, a, st);
    }
    if (sh.n <= 256) return launch_s<D, 8, 2>(sh, a, st);
    if (sh.n <= 512) return launch_s<D, 16, 2>(sh, a, st);
    return launch_s<D, 16, 4>(sh, a, st);
}

}  // namespace

size_t greedy_mma_smem_bytes(const Shape& sh)
{
    // the largest of the layouts the launcher may pick
    const int npad = sh.n <= 256 ? 256 : (sh.n <= 512 ? 512 : 1024);
    const int nw = 16;
    return sh.d == 128 ? mma_layout<128>(npad, sh.N, cand_cap(sh.n), nw).total
                       : mma_layout<64>(npad, sh.N, cand_cap(sh.n), nw).total;
}

cudaError_t launch_greedy_mma(const Shape& sh, const GreedyArgs& a, cudaStream_t st)
{
    if (a.Vc <= 0) return cudaSuccess;
    return sh.d == 128 ? launch_d<128>(sh, a, st) : launch_d<64>(sh, a, st);
}

}  // namespace fadkv
