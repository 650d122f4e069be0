// In-pool greedy selection with a ridge refit after every pick, the pool
// correlations computed on the 5th-generation tensor cores.
//
// "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding":
// abstract (screening-based sparse coding: a one-shot Top-n pool, then
// lightweight coefficient refinement) and Table 5 (ridge parameter
// lambda = 1e-4 + 0.20 diag(G)).  Greedy selection inside the pool and the
// lower-index tie rule are conventions of this library; a step is the same
// arithmetic as in the other greedy kernels:
//   j_k = argmax_{j in P \ S} |<d_j, e_k>|,  S <- S + j_k,
//   (G_SS + diag(lambda_abs + lambda_rel G_ii)) c = D_S x,  e_{k+1} = x - D_S c.
//
// Instead of keeping each vector's pool resident (latency-bound: a few
// vectors per SM), every pick is one dense GEMM over a tile of 128 vectors
// of one dictionary and a slice of its atoms:
//   A = e_k 2^p of every vector split in two binary16 terms (hi, lo; the
//       split leaves a relative error near 2^-22), written by the vector's
//       own thread into its TMEM lane -- columns [0, d/2) hi, [d/2, d) lo,
//       two elements per column;
//   B = 64-atom chunks of the dictionary, streamed by TMA (128-byte
//       swizzle, 3 stages);
//   D = A_hi B^T + A_lo B^T in TMEM (fp32), two 64-column buffers;
//   the vector's thread scans its accumulator row for the largest |.| over
//   the atoms of its pool not yet picked (a bitmask per vector in shared
//   memory), ties to the lower atom index.  The scale 2^p is the same along
//   the row, so raw accumulators are compared.
// This does N/n times the multiply-adds of a pool-restricted product, on a
// unit several times faster and without the per-vector dependency chain.
// The C slices of a tile form a thread-block cluster; their CTAs swap the
// per-vector winners through distributed shared memory (one remote store and
// one release-arrive per peer), so all hold the same pick.  Each CTA then
// refits every vector of the tile (inverse Cholesky factor M = L^-1, per
// vector in shared memory, one thread per vector), forms e_{k+1} and writes
// the next A operand; cluster rank 0 writes the outputs.
//
// Warp roles (256 threads): warp 0 issues TMA loads, warp 1 issues MMAs (one
// thread each), warp 2 owns the TMEM allocation, warps 4..7 own one vector
// each per thread (TMEM lane = tile row).  Every wait is bounded: on expiry
// the kernel flags FADKV_DEV_TIMEOUT in the status word and winds down.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "select.cuh"
#include "tc_common.cuh"

namespace fadkv {
namespace {

using namespace tc;

constexpr int kThreadsG = 256;
constexpr int kTileG = 128;     // vectors per tile (MMA M)
constexpr int kChunkG = 64;     // atoms per MMA (MMA N)
constexpr int kStagesG = 3;     // atom-chunk pipeline depth
constexpr int kTmemColsG = 256;
constexpr int kMaxClusterG = 8;

struct GtcLayout {
    uint32_t b, mask, st, xch, bar, taddr, total, alloc;
};

// ns: atoms of the largest slice; C: CTAs per cluster.
__host__ __device__ inline GtcLayout gtc_layout(int d, int smax, int ns, int C)
{
    GtcLayout L;
    uint32_t o = 0;
    L.b = o;     o += (uint32_t)(kStagesG * (d / 64) * kChunkG * 128);          // 1024-byte multiples
    L.mask = o;  o += (uint32_t)((ns / 32) * kTileG * 4);                        // [word][row]
    L.st = o;    o += (uint32_t)((smax * (smax + 1) / 2 + 3 * smax) * kTileG * 4);  // M, z, c, picks: [entry][row]
    L.xch = o;   o += (uint32_t)(2 * C * kTileG * 8);                            // [parity][rank][row]
    o = (o + 7u) & ~7u;
    L.bar = o;   o += (uint32_t)((2 * kStagesG + 2 + 2 + 1 + 2) * 8);
    L.taddr = o; o += 16;
    L.total = o;
    L.alloc = o + 1024;                                                          // 1024-byte alignment slack
    return L;
}

__device__ __forceinline__ void load8(const __half* p, float (&f)[8])
{
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    const __half2* h = reinterpret_cast<const __half2*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __half22float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ int tri(int i, int j) { return i * (i + 1) / 2 + j; }

template <int D, int SMAX>
__global__ void __launch_bounds__(kThreadsG, 2)
greedy_tc_kernel(const __grid_constant__ CUtensorMap map_d, Shape sh, GreedyTCArgs a, int C)
{
    constexpr int KH = D / 64, KT = D / 16, ACOLS = D / 2;
    constexpr uint32_t kStageBytes = (uint32_t)(KH * kChunkG * 128);
    constexpr uint32_t kIdescG = idesc_f16(kTileG, kChunkG);
    constexpr int TRI = SMAX * (SMAX + 1) / 2;

    const int N = sh.N, n = sh.n, s = sh.s;
    const int nchunks_all = N / kChunkG;
    const int cps = (nchunks_all + C - 1) / C;
    const GtcLayout L = gtc_layout(D, SMAX, cps * kChunkG, C);
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sB = sbase + L.b;
    uint32_t* mask = (uint32_t*)(smem + L.mask);
    float* stf = (float*)(smem + L.st);
    const uint32_t bar0 = sbase + L.bar;
    auto full_bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    auto empty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(kStagesG + i); };
    auto accf_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * kStagesG + i); };
    auto acce_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * kStagesG + 2 + i); };
    const uint32_t afull_bar = bar0 + 8u * (uint32_t)(2 * kStagesG + 4);
    auto xfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * kStagesG + 5 + i); };
    uint32_t* taddr_slot = (uint32_t*)(smem + L.taddr);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.y;
    const int rank = (C > 1) ? (int)cluster_rank() : 0;
    const int tile = blockIdx.x / C;
    const int c0 = rank * cps;
    const int nch = max(0, min(cps, nchunks_all - c0));
    const int atom0 = c0 * kChunkG;
    unsigned long long* status = (unsigned long long*)&a.counters[(size_t)g * kCntFields + kCntStatus];

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStagesG; ++i) {
            mbar_init(full_bar(i), 1);
            mbar_init(empty_bar(i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(accf_bar(i), 1);
            mbar_init(acce_bar(i), kTileG);
        }
        mbar_init(afull_bar, kTileG);
        for (int i = 0; i < 2; ++i) mbar_init(xfull_bar(i), C > 1 ? (uint32_t)((C - 1) * kTileG) : 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(taddr_slot)),
                     "r"(kTmemColsG));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tbase = *taddr_slot;
    if (C > 1) cluster_sync();   // every CTA's barriers exist before any remote arrive

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_d)) : "memory");
            int cc = 0;
            bool ok = true;
            for (int k = 0; k < s && ok; ++k) {
                for (int c = 0; c < nch; ++c) {
                    const int st = cc % kStagesG;
                    const uint32_t ph = (uint32_t)(cc / kStagesG) & 1u;
                    ok = mbar_wait(empty_bar(st), ph ^ 1u, status);
                    if (!ok) break;
                    mbar_expect_tx(full_bar(st), kStageBytes);
                    const int arow = g * N + atom0 + c * kChunkG;
#pragma unroll
                    for (int h = 0; h < KH; ++h)
                        tma_load_2d(sB + (uint32_t)st * kStageBytes + (uint32_t)(h * kChunkG * 128), &map_d, h * 64,
                                    arow, full_bar(st));
                    ++cc;
                }
            }
            // drain: every issued load must have landed before the CTA exits
            for (int i = max(0, cc - kStagesG); i < cc; ++i)
                mbar_wait(full_bar(i % kStagesG), (uint32_t)(i / kStagesG) & 1u, status);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int cc = 0;
            bool ok = true;
            for (int k = 0; k < s && ok; ++k) {
                ok = mbar_wait(afull_bar, (uint32_t)k & 1u, status);
                if (!ok) break;
                fence_after();
                for (int c = 0; c < nch; ++c) {
                    const int st = cc % kStagesG;
                    const uint32_t ph = (uint32_t)(cc / kStagesG) & 1u;
                    const int buf = cc & 1;
                    const uint32_t bph = (uint32_t)(cc >> 1) & 1u;
                    ok = mbar_wait(acce_bar(buf), bph ^ 1u, status);
                    if (ok) ok = mbar_wait(full_bar(st), ph, status);
                    if (!ok) break;
                    fence_after();
                    const uint32_t dt = tbase + (uint32_t)(D + buf * kChunkG);
                    const uint32_t bst = sB + (uint32_t)st * kStageBytes;
#pragma unroll
                    for (int kk = 0; kk < KT; ++kk) {
                        const uint32_t koff = (uint32_t)((kk >> 2) * kChunkG * 128 + (kk & 3) * 32);
                        mma_ts(dt, tbase + (uint32_t)(kk * 8), sdesc(bst + koff), kIdescG, kk > 0 ? 1u : 0u);
                    }
#pragma unroll
                    for (int kk = 0; kk < KT; ++kk) {
                        const uint32_t koff = (uint32_t)((kk >> 2) * kChunkG * 128 + (kk & 3) * 32);
                        mma_ts(dt, tbase + (uint32_t)(ACOLS + kk * 8), sdesc(bst + koff), kIdescG, 1u);
                    }
                    mma_commit(empty_bar(st));
                    mma_commit(accf_bar(buf));
                    ++cc;
                }
            }
            // drain: the last accumulator must be complete before TMEM is freed
            if (cc > 0) mbar_wait(accf_bar((cc - 1) & 1), (uint32_t)((cc - 1) >> 1) & 1u, status);
        }
    } else if (warp >= 4) {
        // ---------------- one vector per thread ----------------
        const int q = warp - 4;
        const int r = q * 32 + lane;                       // tile row = TMEM lane
        const int vloc = tile * kTileG + r;                // vector inside this pass
        const bool valid = vloc < a.Vc;
        const int v = a.v0 + (valid ? vloc : 0);
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const __half* Ag = (const __half*)a.atoms + (size_t)g * N * D;
        const __half* xrow = (const __half*)a.x + ((size_t)g * a.V + v) * D;
        float* Mst = stf;                                  // [TRI][row]
        float* zst = stf + TRI * kTileG;                   // [SMAX][row]
        float* cst = zst + SMAX * kTileG;                  // [SMAX][row]
        int* pst = (int*)(cst + SMAX * kTileG);            // [SMAX][row]
        const float la = sh.lambda_abs, lr = sh.lambda_rel;

        // x: finiteness, norm, scale 2^p with |e_t| 2^p < 2^14
        float xn2 = 0.f;
        bool bad = false;
        if (valid) {
            for (int t0 = 0; t0 < D; t0 += 8) {
                float f[8];
                load8(xrow + t0, f);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    bad |= !isfinite(f[u]);
                    xn2 = fmaf(f[u], f[u], xn2);
                }
            }
        }
        bool active = valid && !bad;
        int ex = 0;
        frexpf(sqrtf(xn2), &ex);
        const float scale = (xn2 > 0.f) ? ldexpf(1.f, 14 - ex) : 1.f;

        // pool membership of this slice's atoms
        for (int w = 0; w < 2 * nch; ++w) mask[w * kTileG + r] = 0u;
        if (active) {
            const int32_t* pl = a.pool + ((size_t)g * a.Vc + vloc) * n;
            const unsigned span = (unsigned)(nch * kChunkG);
#pragma unroll 4
            for (int i = 0; i < n; ++i) {
                const int j = __ldg(pl + i) - atom0;
                if ((unsigned)j < span) mask[(j >> 5) * kTileG + r] |= 1u << (j & 31);
            }
        }

        // e -> A operand (hi, lo) of this lane, 32 elements at a time
        auto write_a = [&](int cb, const float (&e)[32]) {
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const float s0 = e[2 * u] * scale, s1 = e[2 * u + 1] * scale;
                const __half h0 = __float2half_rn(s0), h1 = __float2half_rn(s1);
                const __half l0 = __float2half_rn(s0 - __half2float(h0));
                const __half l1 = __float2half_rn(s1 - __half2float(h1));
                const __half2 hh = __halves2half2(h0, h1), ll = __halves2half2(l0, l1);
                hi[u] = *reinterpret_cast<const uint32_t*>(&hh);
                lo[u] = *reinterpret_cast<const uint32_t*>(&ll);
            }
            tmem_st16(tbase + lane_off + (uint32_t)(cb * 16), hi);
            tmem_st16(tbase + lane_off + (uint32_t)(ACOLS + cb * 16), lo);
        };
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
            float e[32];
#pragma unroll
            for (int u8 = 0; u8 < 4; ++u8) {
                float f[8];
                if (active) load8(xrow + cb * 32 + u8 * 8, f);
#pragma unroll
                for (int u = 0; u < 8; ++u) e[u8 * 8 + u] = active ? f[u] : 0.f;
            }
            write_a(cb, e);
        }
        tmem_st_wait();

        int cc = 0;
        bool ok = true;
        float esq = 0.f;
        for (int k = 0; k < s; ++k) {
            fence_before();
            mbar_arrive(afull_bar);                        // A_k is in TMEM

            // ---- sweep: masked argmax over this slice ----
            uint32_t best = 0u;                            // (|acc| bits) + 1 for pool atoms, 0 otherwise
            int bj = -1;
            for (int c = 0; c < nch; ++c) {
                const int buf = cc & 1;
                const uint32_t bph = (uint32_t)(cc >> 1) & 1u;
                if (ok) ok = mbar_wait(accf_bar(buf), bph, status);
                ok = __all_sync(0xffffffffu, ok);
                if (ok) {
                    fence_after();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t acc[32];
                        tmem_ld32(tbase + lane_off + (uint32_t)(D + buf * kChunkG + h * 32), acc);
                        const uint32_t mw = mask[(c * 2 + h) * kTileG + r];
                        const int j0 = atom0 + c * kChunkG + h * 32;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const uint32_t key = ((mw >> i) & 1u) ? (acc[i] & 0x7fffffffu) + 1u : 0u;
                            const bool take = key > best;
                            best = take ? key : best;
                            bj = take ? j0 + i : bj;
                        }
                    }
                }
                fence_before();
                mbar_arrive(acce_bar(buf));
                ++cc;
            }

            // ---- the cluster's winner: larger key, then the lower atom ----
            if (C > 1) {
                const int par = k & 1;
                const uint32_t mine = sbase + L.xch + (uint32_t)(((par * C + rank) * kTileG + r) * 8);
                for (int p = 0; p < C; ++p)
                    if (p != rank) st_peer_u2(map_peer(mine, (uint32_t)p), best, (uint32_t)bj);
                for (int p = 0; p < C; ++p)
                    if (p != rank) mbar_arrive_peer(map_peer(xfull_bar(par), (uint32_t)p));
                const bool got = ok && mbar_wait<true>(xfull_bar(par), (uint32_t)(k >> 1) & 1u, status);
                if (got) {
                    for (int p = 0; p < C; ++p) {
                        if (p == rank) continue;
                        const uint2 o = *reinterpret_cast<const uint2*>(smem + L.xch + ((par * C + p) * kTileG + r) * 8);
                        if (o.x > best || (o.x == best && o.y < (uint32_t)bj)) {
                            best = o.x;
                            bj = (int)o.y;
                        }
                    }
                } else {
                    ok = false;
                }
            }
            if (!(best > 0u) || bj < 0 || bj >= N) active = false;   // no pool atom left (not reached for n >= s)
            const int jk = bj;
            if (active) {
                const int jj = jk - atom0;
                if ((unsigned)jj < (unsigned)(nch * kChunkG)) mask[(jj >> 5) * kTileG + r] &= ~(1u << (jj & 31));
                pst[k * kTileG + r] = jk;

                // ---- Gram row of the pick, its norm and <d, x> ----
                int pk[SMAX];
#pragma unroll
                for (int i = 0; i < SMAX; ++i) pk[i] = (i < k) ? pst[i * kTileG + r] : 0;
                float bk = 0.f, gkk = 0.f, gr[SMAX];
#pragma unroll
                for (int i = 0; i < SMAX; ++i) gr[i] = 0.f;
                const __half* dn = Ag + (size_t)jk * D;
#pragma unroll 1
                for (int t0 = 0; t0 < D; t0 += 8) {
                    float fn[8], fx[8];
                    load8(dn + t0, fn);
                    load8(xrow + t0, fx);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        bk = fmaf(fn[u], fx[u], bk);
                        gkk = fmaf(fn[u], fn[u], gkk);
                    }
#pragma unroll
                    for (int i = 0; i < SMAX; ++i) {
                        if (i < k) {
                            float fi[8];
                            load8(Ag + (size_t)pk[i] * D + t0, fi);
#pragma unroll
                            for (int u = 0; u < 8; ++u) gr[i] = fmaf(fn[u], fi[u], gr[i]);
                        }
                    }
                }

                // ---- ridge refit: one row more of M = L^-1 ----
                // A = G_SS + diag(lambda_abs + lambda_rel G_ii) = L L^T,
                // z = M b, c = M^T z.  l = M g, L_kk = sqrt(gkk (1 + lr) + la - l.l),
                // z_k = (b_k - l.z) / L_kk, new row w = -(l^T M) / L_kk,
                // c <- c + z_k w, c_k = z_k / L_kk.
                float l[SMAX];
                float ll = 0.f, lz = 0.f;
#pragma unroll
                for (int i = 0; i < SMAX; ++i) {
                    float li = 0.f;
                    if (i < k) {
#pragma unroll
                        for (int m = 0; m <= i; ++m) li = fmaf(Mst[tri(i, m) * kTileG + r], gr[m], li);
                        ll = fmaf(li, li, ll);
                        lz = fmaf(li, zst[i * kTileG + r], lz);
                    }
                    l[i] = li;
                }
                float dk = fmaf(gkk, lr, gkk) + la - ll;
                if (!(dk > 0.f)) {
                    atomicOr(status, (unsigned long long)FADKV_DEV_NOT_SPD);
                    dk = 1e-30f;
                }
                const float inv = __frcp_rn(sqrtf(dk));
                const float zk = (bk - lz) * inv;
#pragma unroll
                for (int j = 0; j < SMAX; ++j) {
                    if (j < k) {
                        float acc = 0.f;
#pragma unroll
                        for (int i = j; i < SMAX; ++i)
                            if (i < k) acc = fmaf(l[i], Mst[tri(i, j) * kTileG + r], acc);
                        const float w = -acc * inv;
                        Mst[tri(k, j) * kTileG + r] = w;
                        cst[j * kTileG + r] = fmaf(zk, w, cst[j * kTileG + r]);
                    }
                }
                Mst[tri(k, k) * kTileG + r] = inv;
                zst[k * kTileG + r] = zk;
                cst[k * kTileG + r] = zk * inv;
            }

            // ---- residual e_{k+1} = x - D_S c: the next A operand, or relres ----
            const bool last = (k + 1 == s);
            float cr[SMAX];
            int pr[SMAX];
#pragma unroll
            for (int i = 0; i < SMAX; ++i) {
                cr[i] = (active && i <= k) ? cst[i * kTileG + r] : 0.f;
                pr[i] = (active && i <= k) ? pst[i * kTileG + r] : 0;
            }
#pragma unroll 1
            for (int cb = 0; cb < D / 32; ++cb) {
                float e[32];
#pragma unroll
                for (int u8 = 0; u8 < 4; ++u8) {
                    float f[8];
                    if (active) load8(xrow + cb * 32 + u8 * 8, f);
#pragma unroll
                    for (int u = 0; u < 8; ++u) e[u8 * 8 + u] = active ? f[u] : 0.f;
                }
                if (active) {
#pragma unroll
                    for (int i = 0; i < SMAX; ++i) {
                        if (i <= k) {
                            const __half* di = Ag + (size_t)pr[i] * D + cb * 32;
#pragma unroll
                            for (int u8 = 0; u8 < 4; ++u8) {
                                float f[8];
                                load8(di + u8 * 8, f);
#pragma unroll
                                for (int u = 0; u < 8; ++u) e[u8 * 8 + u] = fmaf(-cr[i], f[u], e[u8 * 8 + u]);
                            }
                        }
                    }
                }
                if (!last) {
                    write_a(cb, e);
                } else {
#pragma unroll
                    for (int u = 0; u < 32; ++u) esq = fmaf(e[u], e[u], esq);
                }
            }
            if (!last) tmem_st_wait();
        }

        // ---- outputs (cluster rank 0) ----
        if (rank == 0 && valid) {
            const size_t o = (size_t)g * a.V + v;
            long long* cnt = a.counters + (size_t)g * kCntFields;
            if (bad) {
                for (int k = 0; k < s; ++k) {
                    a.idx[o * s + k] = -1;
                    a.coef[o * s + k] = 0.f;
                }
                a.relres[o] = __int_as_float(0x7fc00000);
                atomicAdd((unsigned long long*)&cnt[kCntNonfinite], 1ull);
                atomicOr((unsigned long long*)&cnt[kCntStatus], (unsigned long long)FADKV_DEV_NONFINITE_INPUT);
            } else {
                for (int k = 0; k < s; ++k) {
                    a.idx[o * s + k] = active ? pst[k * kTileG + r] : -1;
                    a.coef[o * s + k] = active ? cst[k * kTileG + r] : 0.f;
                }
                a.relres[o] = (xn2 > 0.f) ? sqrtf(esq) / sqrtf(xn2) : 0.f;
            }
        }
    }

    fence_before();
    __syncthreads();
    if (warp == 2) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kTmemColsG));
    }
    if (C > 1) cluster_sync();   // no CTA leaves while a peer may still write to it
}

// ---------------------------------------------------------------------------
// Exact pool of the vectors the selection kernel left to the slow path.
// ---------------------------------------------------------------------------
template <int D>
struct FixupLayout {
    size_t keys, xs, pid, mag, hist, scan, misc, pref, total;
};

template <int D>
__host__ __device__ inline FixupLayout<D> fixup_layout(int N, int n, int nw)
{
    FixupLayout<D> L;
    size_t o = 0;
    L.keys = o; o += (size_t)N * 8;
    L.xs = o;   o += 4 * D;
    L.pid = o;  o += 4 * (size_t)n;
    L.mag = o;  o += 4 * (size_t)n;
    L.hist = o; o += 4 * 256;
    L.scan = o; o += 4 * (size_t)nw;
    L.misc = o; o += 4 * (4 + kCountSlots);
    o = (o + 7) & ~(size_t)7;
    L.pref = o; o += 8;
    L.total = o;
    return L;
}

constexpr int kFixThreads = 256;

template <int D>
__global__ void __launch_bounds__(kFixThreads)
pool_fixup_kernel(Shape sh, GreedyArgs a, int32_t* pool)
{
    const FixupLayout<D> L = fixup_layout<D>(sh.N, sh.n, kFixThreads / 32);
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned long long* keys = (unsigned long long*)(smem + L.keys);
    float* xs = (float*)(smem + L.xs);
    int* pid = (int*)(smem + L.pid);
    float* mag = (float*)(smem + L.mag);
    sel::Scratch sc{(uint32_t*)(smem + L.hist), (uint32_t*)(smem + L.scan), (uint32_t*)(smem + L.misc),
                    (unsigned long long*)(smem + L.pref)};
    __shared__ int flagged[kFixThreads];
    __shared__ int nflagged;
    const int n = sh.n, N = sh.N;
    const long long total = (long long)sh.G * a.Vc;
    for (long long base = (long long)blockIdx.x * kFixThreads; base < total;
         base += (long long)gridDim.x * kFixThreads) {
      // the flags of kFixThreads vectors at once, then the flagged ones in turn
      if (threadIdx.x == 0) nflagged = 0;
      __syncthreads();
      const long long mine = base + threadIdx.x;
      if (mine < total && pool[mine * n] == -2) flagged[atomicAdd(&nflagged, 1)] = (int)threadIdx.x;
      __syncthreads();
      const int nf = nflagged;
      for (int f = 0; f < nf; ++f) {
        const long long gv = base + flagged[f];
        const int g = (int)(gv / a.Vc), vc = (int)(gv % a.Vc);
        const __half* X = (const __half*)a.x + ((size_t)g * a.V + a.v0 + vc) * D;
        int bad = 0;
        for (int t = threadIdx.x; t < D; t += kFixThreads) {
            xs[t] = __half2float(X[t]);
            bad |= !isfinite(xs[t]);
        }
        bad = __syncthreads_or(bad);
        if (bad) {
            // the greedy kernel reports a non-finite input itself; any valid pool will do
            for (int i = threadIdx.x; i < n; i += kFixThreads) pool[gv * n + i] = i;
            __syncthreads();
            continue;
        }
        const __half* A = (const __half*)a.atoms + (size_t)g * N * D;
        long long* cnt = a.counters + (size_t)g * kCntFields;
        const int K = sel::intake_keys<__half, D>(a, (size_t)gv, -1, n, N, A, xs, keys, sc, cnt);
        sel::top_n(keys, K, n, pid, mag, sc);
        for (int i = threadIdx.x; i < n; i += kFixThreads) pool[gv * n + i] = pid[i];
        __syncthreads();
      }
      __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
constexpr double kTailChunks = 6.0;   // per-pick tail of a CTA, in chunk-MMA units (cluster choice)
constexpr size_t kSmemPerSm = 228 * 1024;
constexpr size_t kSmemPerCta = 227 * 1024;
constexpr size_t kSmemFloor = 80 * 1024;

int smax_for(int s) { return s <= 8 ? 8 : 16; }

template <int D, int SMAX>
cudaError_t launch_tc(const Shape& sh, const GreedyTCArgs& a, int C, cudaStream_t st)
{
    CUtensorMap md;
    if (!make_tma_map_f16(&md, a.atoms, (long long)sh.G * sh.N, D, kChunkG)) return cudaErrorInvalidValue;
    const int nchunks_all = sh.N / kChunkG;
    const int cps = (nchunks_all + C - 1) / C;
    // at least 80 KB: never more than two CTAs (2 x 256 TMEM columns) per SM
    size_t smem = gtc_layout(D, SMAX, cps * kChunkG, C).alloc;
    if (smem < kSmemFloor) smem = kSmemFloor;
    auto k = greedy_tc_kernel<D, SMAX>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int tiles = (a.Vc + kTileG - 1) / kTileG;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles * C), (unsigned)sh.G, 1);
    cfg.blockDim = dim3(kThreadsG, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (C > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    e = cudaLaunchKernelEx(&cfg, k, md, sh, a, C);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// CTAs per cluster: balances the chunks the busiest SM streams (CTAs of one
// SM share its tensor core) against the per-pick tail of each CTA, within
// the shared-memory budget.  FADKV_GREEDY_CLUSTER=c forces c.
int choose_cluster(const Shape& sh, int tiles, int sms)
{
    const int T = sh.N / kChunkG;
    const int smax = smax_for(sh.s);
    const char* f = getenv("FADKV_GREEDY_CLUSTER");
    if (f) {
        const int c = atoi(f);
        if (c >= 1 && c <= kMaxClusterG && c <= T) {
            const int cps = (T + c - 1) / c;
            if ((c - 1) * cps < T && gtc_layout(sh.d, smax, cps * kChunkG, c).alloc <= kSmemPerCta) return c;
        }
    }
    int bestC = 1;
    double bestCost = 1e300;
    for (int C = 1; C <= kMaxClusterG && C <= T; ++C) {
        const int cps = (T + C - 1) / C;
        if ((C - 1) * cps >= T) continue;                   // a rank without atoms
        size_t smem = gtc_layout(sh.d, smax, cps * kChunkG, C).alloc;
        if (smem > kSmemPerCta) continue;
        if (smem < kSmemFloor) smem = kSmemFloor;
        const int res = (2 * (smem + 1024) <= kSmemPerSm) ? 2 : 1;
        const double total = (double)sh.G * tiles * C;
        const double cost = ceil(total / sms) * cps + ceil(total / ((double)sms * res)) * kTailChunks * sh.s / 8.0;
        if (cost < bestCost - 1e-9) {
            bestCost = cost;
            bestC = C;
        }
    }
    return bestC;
}

template <int D>
cudaError_t launch_fixup_t(const Shape& sh, const GreedyArgs& a, int32_t* pool, int sms, cudaStream_t st)
{
    const size_t smem = fixup_layout<D>(sh.N, sh.n, kFixThreads / 32).total;
    auto k = pool_fixup_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long total = (long long)sh.G * a.Vc;
    const long long blocks = (total + kFixThreads - 1) / kFixThreads;
    const long long want = 2LL * sms;
    const unsigned grid = (unsigned)(blocks < want ? blocks : want);
    k<<<grid, kFixThreads, smem, st>>>(sh, a, pool);
    return cudaGetLastError();
}

}  // namespace

bool greedy_tc_supported(const Shape& sh)
{
    if (sh.dtype != FADKV_F16 || (sh.d != 64 && sh.d != 128) || sh.N % kChunkG != 0 || sh.s > 16) return false;
    // the smallest layout (8-CTA clusters) must fit
    const int T = sh.N / kChunkG;
    const int C = T < kMaxClusterG ? T : kMaxClusterG;
    const int cps = (T + C - 1) / C;
    return gtc_layout(sh.d, smax_for(sh.s), cps * kChunkG, C).alloc <= kSmemPerCta;
}

cudaError_t launch_greedy_tc(const Shape& sh, const GreedyTCArgs& a, int sms, cudaStream_t st)
{
    if (a.Vc <= 0) return cudaSuccess;
    const int tiles = (a.Vc + kTileG - 1) / kTileG;
    const int C = choose_cluster(sh, tiles, sms);
    if (sh.d == 128) return sh.s <= 8 ? launch_tc<128, 8>(sh, a, C, st) : launch_tc<128, 16>(sh, a, C, st);
    return sh.s <= 8 ? launch_tc<64, 8>(sh, a, C, st) : launch_tc<64, 16>(sh, a, C, st);
}

cudaError_t launch_pool_fixup(const Shape& sh, const GreedyArgs& a, int32_t* pool, int sms, cudaStream_t st)
{
    if (a.Vc <= 0) return cudaSuccess;
    return sh.d == 128 ? launch_fixup_t<128>(sh, a, pool, sms, st) : launch_fixup_t<64>(sh, a, pool, sms, st);
}

}  // namespace fadkv
