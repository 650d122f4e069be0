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
constexpr int kStagesG = 2;     // atom-chunk pipeline depth
constexpr int kTmemColsG = 256;
constexpr int kMaxClusterG = 8;

struct GtcLayout {
    uint32_t b, mask, st, gbuf, vec, stage, xch, bar, taddr, total, alloc;
};

// ns: atoms of the largest slice; C: CTAs per cluster.
__host__ __device__ inline GtcLayout gtc_layout(int d, int smax, int ns, int C)
{
    GtcLayout L;
    uint32_t o = 0;
    L.b = o;     o += (uint32_t)(kStagesG * (d / 64) * kChunkG * 128);          // 1024-byte multiples
    L.mask = o;  o += (uint32_t)((ns / 32) * kTileG * 4);                        // [word][row]
    L.st = o;    o += (uint32_t)((smax * (smax + 1) / 2 + 3 * smax) * kTileG * 4);  // M, z, c, picks: [entry][row]
    L.gbuf = o;  o += (uint32_t)((smax + 2) * kTileG * 4);                       // Gram row, ||d||^2, <d,x>: [entry][row]
    L.vec = o;   o += (uint32_t)(3 * kTileG * 4);                                // scale, ||x||^2, state: [row]
    L.stage = o; o += (uint32_t)(4 * 2 * 32 * 32 * 2);                           // per warp: hi, lo [32 rows][32] binary16
    L.xch = o;   o += (uint32_t)(2 * C * kTileG * 8);                            // [parity][rank][row]
    o = (o + 7u) & ~7u;
    L.bar = o;   o += (uint32_t)((2 * kStagesG + 2 + 2 + 1 + 2) * 8);
    L.taddr = o; o += 16;
    L.total = o;
    L.alloc = o + 1024;                                                          // 1024-byte alignment slack
    return L;
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
        // ---------------- the vectors: warps 4..7, one TMEM lane quadrant each ----------------
        // Thread-per-vector work (row r = TMEM lane): the sweep, the cluster
        // exchange and the refit.  Warp-cooperative work (8 lanes per vector,
        // 4 vectors at a time, each lane 4 consecutive elements of every
        // 32-element quarter, so a row quarter is one 64-byte segment): the
        // statistics of x, the pool masks, the Gram row of the pick and the
        // residual, which is staged per quarter and written to TMEM by the
        // lane owners.
        const int q = warp - 4;
        const int r = q * 32 + lane;                       // tile row = TMEM lane
        const int gs = lane >> 3, l8 = lane & 7;           // vector slot of the group, lane in the group
        const int rows = min(kTileG, a.Vc - tile * kTileG);
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const __half* Ag = (const __half*)a.atoms + (size_t)g * N * D;
        const __half* Xt = (const __half*)a.x + ((size_t)g * a.V + a.v0 + (size_t)tile * kTileG) * D;   // row R at Xt + R D
        float* Mst = stf;                                  // [TRI][row]
        float* zst = stf + TRI * kTileG;                   // [SMAX][row]
        float* cst = zst + SMAX * kTileG;                  // [SMAX][row]
        int* pst = (int*)(cst + SMAX * kTileG);            // [SMAX][row]
        float* gbuf = (float*)(smem + L.gbuf);             // [SMAX + 2][row]
        float* vscale = (float*)(smem + L.vec);            // [row]
        float* vxn2 = vscale + kTileG;                     // [row]
        int* vstate = (int*)(vxn2 + kTileG);               // [row]: 0 none, 1 active, 2 non-finite
        __half* stg_hi = (__half*)(smem + L.stage) + q * (2 * 32 * 32);
        __half* stg_lo = stg_hi + 32 * 32;
        const float la = sh.lambda_abs, lr = sh.lambda_rel;

        // 4 elements of a binary16 row at element e (8-byte load)
        auto ld4 = [](const __half* p, float (&f)[4]) {
            const uint2 u = *reinterpret_cast<const uint2*>(p);
            const float2 a0 = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
            const float2 a1 = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
            f[0] = a0.x; f[1] = a0.y; f[2] = a1.x; f[3] = a1.y;
        };

        // ---- x: finiteness, norm, scale 2^p with |e_t| 2^p < 2^14 ----
#pragma unroll 1
        for (int it = 0; it < 8; ++it) {
            const int R = q * 32 + it * 4 + gs;
            float sq = 0.f;
            int bad = 0;
            if (R < rows) {
#pragma unroll
                for (int cq = 0; cq < D / 32; ++cq) {
                    float f[4];
                    ld4(Xt + (size_t)R * D + cq * 32 + 4 * l8, f);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        bad |= !isfinite(f[u]);
                        sq = fmaf(f[u], f[u], sq);
                    }
                }
            }
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                bad |= __shfl_xor_sync(0xffffffffu, bad, o);
            }
            if (l8 == 0) {
                int ex = 0;
                frexpf(sqrtf(sq), &ex);
                vscale[R] = (sq > 0.f) ? ldexpf(1.f, 14 - ex) : 1.f;
                vxn2[R] = sq;
                vstate[R] = (R < rows) ? (bad ? 2 : 1) : 0;
            }
        }

        // ---- pool membership of this slice's atoms (bitmask per row) ----
        for (int w = 0; w < 2 * nch; ++w) mask[w * kTileG + r] = 0u;
        __syncwarp();
        {
            const unsigned span = (unsigned)(nch * kChunkG);
#pragma unroll 1
            for (int v = 0; v < 32; ++v) {
                const int R = q * 32 + v;
                if (R >= rows) break;
                const int32_t* pl = a.pool + ((size_t)g * a.Vc + (size_t)tile * kTileG + R) * n;
#pragma unroll 4
                for (int i = lane; i < n; i += 32) {
                    const int j = __ldg(pl + i) - atom0;
                    if ((unsigned)j < span) atomicOr(&mask[(j >> 5) * kTileG + R], 1u << (j & 31));
                }
            }
        }
        __syncwarp();

        // ---- residual with the first kk+1 picks -> A operand (or ||e||^2) ----
        // kk = -1: e = x.  Row order: row 32q + 4 it + gs at staging row 4 it + gs.
        float esq[8];
#pragma unroll
        for (int it = 0; it < 8; ++it) esq[it] = 0.f;
        auto residual_pass = [&](int kk, bool to_tmem) {
#pragma unroll 1
            for (int cq = 0; cq < D / 32; ++cq) {
#pragma unroll 2
                for (int it = 0; it < 8; ++it) {
                    const int lr_ = it * 4 + gs;
                    const int R = q * 32 + lr_;
                    const bool act = vstate[R] == 1;
                    float e[4] = {0.f, 0.f, 0.f, 0.f};
                    if (act) {
                        ld4(Xt + (size_t)R * D + cq * 32 + 4 * l8, e);
#pragma unroll
                        for (int i = 0; i < SMAX; ++i) {
                            if (i <= kk) {
                                const float ci = cst[i * kTileG + R];
                                float f[4];
                                ld4(Ag + (size_t)pst[i * kTileG + R] * D + cq * 32 + 4 * l8, f);
#pragma unroll
                                for (int u = 0; u < 4; ++u) e[u] = fmaf(-ci, f[u], e[u]);
                            }
                        }
                    }
                    if (to_tmem) {
                        const float sc = vscale[R];
                        __half h[4], l[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float sv = e[u] * sc;
                            h[u] = __float2half_rn(sv);
                            l[u] = __float2half_rn(sv - __half2float(h[u]));
                        }
                        const __half2 h01 = __halves2half2(h[0], h[1]), h23 = __halves2half2(h[2], h[3]);
                        const __half2 l01 = __halves2half2(l[0], l[1]), l23 = __halves2half2(l[2], l[3]);
                        uint2 uh, ul;
                        uh.x = *reinterpret_cast<const uint32_t*>(&h01);
                        uh.y = *reinterpret_cast<const uint32_t*>(&h23);
                        ul.x = *reinterpret_cast<const uint32_t*>(&l01);
                        ul.y = *reinterpret_cast<const uint32_t*>(&l23);
                        *reinterpret_cast<uint2*>(stg_hi + lr_ * 32 + 4 * l8) = uh;
                        *reinterpret_cast<uint2*>(stg_lo + lr_ * 32 + 4 * l8) = ul;
                    } else {
#pragma unroll
                        for (int u = 0; u < 4; ++u) esq[it] = fmaf(e[u], e[u], esq[it]);
                    }
                }
                if (to_tmem) {
                    __syncwarp();
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int w4 = 0; w4 < 4; ++w4) {
                        const uint4 th = *reinterpret_cast<const uint4*>(stg_hi + lane * 32 + w4 * 8);
                        const uint4 tl = *reinterpret_cast<const uint4*>(stg_lo + lane * 32 + w4 * 8);
                        hi[w4 * 4 + 0] = th.x; hi[w4 * 4 + 1] = th.y; hi[w4 * 4 + 2] = th.z; hi[w4 * 4 + 3] = th.w;
                        lo[w4 * 4 + 0] = tl.x; lo[w4 * 4 + 1] = tl.y; lo[w4 * 4 + 2] = tl.z; lo[w4 * 4 + 3] = tl.w;
                    }
                    tmem_st16(tbase + lane_off + (uint32_t)(cq * 16), hi);
                    tmem_st16(tbase + lane_off + (uint32_t)(ACOLS + cq * 16), lo);
                    __syncwarp();
                }
            }
            if (to_tmem) tmem_st_wait();
        };
        residual_pass(-1, true);

        int cc = 0;
        bool ok = true;
        for (int k = 0; k < s; ++k) {
            fence_before();
            mbar_arrive(afull_bar);                        // A_k is in TMEM

            // ---- sweep: masked argmax over this slice (thread per vector) ----
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
            if (vstate[r] == 1) {
                if (!(best > 0u) || bj < 0 || bj >= N) {
                    vstate[r] = 0;                          // no pool atom left (not reached for n >= s)
                } else {
                    const int jj = bj - atom0;
                    if ((unsigned)jj < (unsigned)(nch * kChunkG)) mask[(jj >> 5) * kTileG + r] &= ~(1u << (jj & 31));
                    pst[k * kTileG + r] = bj;
                }
            }
            __syncwarp();

            // ---- Gram row of the pick, its norm and <d, x> (8 lanes per vector) ----
#pragma unroll 1
            for (int it = 0; it < 8; ++it) {
                const int R = q * 32 + it * 4 + gs;
                const bool act = vstate[R] == 1;
                float gp[SMAX];
#pragma unroll
                for (int i = 0; i < SMAX; ++i) gp[i] = 0.f;
                float bp = 0.f, np = 0.f;
                if (act) {
                    const __half* dn = Ag + (size_t)pst[k * kTileG + R] * D;
                    int pk[SMAX];
#pragma unroll
                    for (int i = 0; i < SMAX; ++i) pk[i] = (i < k) ? pst[i * kTileG + R] : 0;
#pragma unroll
                    for (int cq = 0; cq < D / 32; ++cq) {
                        const int e0 = cq * 32 + 4 * l8;
                        float fn[4], fx[4];
                        ld4(dn + e0, fn);
                        ld4(Xt + (size_t)R * D + e0, fx);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            bp = fmaf(fn[u], fx[u], bp);
                            np = fmaf(fn[u], fn[u], np);
                        }
#pragma unroll
                        for (int i = 0; i < SMAX; ++i) {
                            if (i < k) {
                                float fi[4];
                                ld4(Ag + (size_t)pk[i] * D + e0, fi);
#pragma unroll
                                for (int u = 0; u < 4; ++u) gp[i] = fmaf(fn[u], fi[u], gp[i]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    bp += __shfl_xor_sync(0xffffffffu, bp, o);
                    np += __shfl_xor_sync(0xffffffffu, np, o);
#pragma unroll
                    for (int i = 0; i < SMAX; ++i)
                        if (i < k) gp[i] += __shfl_xor_sync(0xffffffffu, gp[i], o);
                }
                if (l8 == 0 && act) {
#pragma unroll
                    for (int i = 0; i < SMAX; ++i)
                        if (i < k) gbuf[i * kTileG + R] = gp[i];
                    gbuf[SMAX * kTileG + R] = np;
                    gbuf[(SMAX + 1) * kTileG + R] = bp;
                }
            }
            __syncwarp();

            // ---- ridge refit: one row more of M = L^-1 (thread per vector) ----
            // A = G_SS + diag(lambda_abs + lambda_rel G_ii) = L L^T,
            // z = M b, c = M^T z.  l = M g, L_kk = sqrt(gkk (1 + lr) + la - l.l),
            // z_k = (b_k - l.z) / L_kk, new row w = -(l^T M) / L_kk,
            // c <- c + z_k w, c_k = z_k / L_kk.
            if (vstate[r] == 1) {
                const float gkk = gbuf[SMAX * kTileG + r], bk = gbuf[(SMAX + 1) * kTileG + r];
                float gr[SMAX], l[SMAX];
#pragma unroll
                for (int i = 0; i < SMAX; ++i) gr[i] = (i < k) ? gbuf[i * kTileG + r] : 0.f;
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
            __syncwarp();

            // ---- residual e_{k+1} = x - D_S c: the next A operand, or ||e_s||^2 ----
            residual_pass(k, k + 1 < s);
        }

        // ---- outputs (cluster rank 0) ----
        if (rank == 0) {
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                float e2 = esq[it];
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) e2 += __shfl_xor_sync(0xffffffffu, e2, o);
                const int R = q * 32 + it * 4 + gs;
                if (l8 == 0 && R < rows && vstate[R] != 2) {
                    const float xn2 = vxn2[R];
                    a.relres[(size_t)g * a.V + a.v0 + (size_t)tile * kTileG + R] =
                        (xn2 > 0.f) ? sqrtf(e2) / sqrtf(xn2) : 0.f;
                }
            }
            if (r < rows) {
                const size_t o = (size_t)g * a.V + a.v0 + (size_t)tile * kTileG + r;
                long long* cnt = a.counters + (size_t)g * kCntFields;
                const int stt = vstate[r];
                if (stt == 2) {
                    for (int k = 0; k < s; ++k) {
                        a.idx[o * s + k] = -1;
                        a.coef[o * s + k] = 0.f;
                    }
                    a.relres[o] = __int_as_float(0x7fc00000);
                    atomicAdd((unsigned long long*)&cnt[kCntNonfinite], 1ull);
                    atomicOr((unsigned long long*)&cnt[kCntStatus], (unsigned long long)FADKV_DEV_NONFINITE_INPUT);
                } else {
                    for (int k = 0; k < s; ++k) {
                        a.idx[o * s + k] = stt == 1 ? pst[k * kTileG + r] : -1;
                        a.coef[o * s + k] = stt == 1 ? cst[k * kTileG + r] : 0.f;
                    }
                }
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
    L.misc = o; o += 4 * (4 + 2 * kCountSlots);
    o = (o + 7) & ~(size_t)7;
    L.pref = o; o += 8;
    L.total = o;
    return L;
}

constexpr int kFixThreads = 256;

template <int D>
__global__ void __launch_bounds__(kFixThreads)
pool_fixup_kernel(Shape sh, GreedyArgs a, int32_t* pool, const uint32_t* slow_seq, uint32_t seq)
{
    pdl_begin();
    if (*slow_seq != seq) return;                      // no vector of this pass was flagged
    const FixupLayout<D> L = fixup_layout<D>(sh.N, sh.n, kFixThreads / 32);
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned long long* keys = (unsigned long long*)(smem + L.keys);
    float* xs = (float*)(smem + L.xs);
    int* pid = (int*)(smem + L.pid);
    float* mag = (float*)(smem + L.mag);
    sel::Scratch sc{(uint32_t*)(smem + L.hist), (uint32_t*)(smem + L.scan), (uint32_t*)(smem + L.misc),
                    (unsigned long long*)(smem + L.pref)};
    __shared__ long long flagged[kFixThreads];
    __shared__ int nflagged;
    const int n = sh.n, N = sh.N;
    const long long total = (long long)sh.G * a.Vc;
    // vector gv belongs to CTA gv mod gridDim: flagged vectors, which come in
    // runs of neighbours, spread over the CTAs.  The flags of a CTA's next
    // kFixThreads vectors are read at once, then the flagged ones in turn.
    const long long stride = (long long)gridDim.x * kFixThreads;
    for (long long base = blockIdx.x; base < total; base += stride) {
      if (threadIdx.x == 0) nflagged = 0;
      __syncthreads();
      const long long mine = base + (long long)threadIdx.x * gridDim.x;
      if (mine < total && pool[mine * n] == -2) flagged[atomicAdd(&nflagged, 1)] = mine;
      __syncthreads();
      const int nf = nflagged;
      for (int f = 0; f < nf; ++f) {
        const long long gv = flagged[f];
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
cudaError_t launch_fixup_t(const Shape& sh, const GreedyArgs& a, int32_t* pool, const uint32_t* slow_seq,
                           uint32_t seq, int sms, cudaStream_t st)
{
    const size_t smem = fixup_layout<D>(sh.N, sh.n, kFixThreads / 32).total;
    auto k = pool_fixup_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long total = (long long)sh.G * a.Vc;
    const long long want = 2LL * sms;
    const unsigned grid = (unsigned)(total < want ? total : want);
    return launch_pdl(k, dim3(grid), dim3(kFixThreads), smem, st, sh, a, pool, slow_seq, seq);
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

cudaError_t launch_pool_fixup(const Shape& sh, const GreedyArgs& a, int32_t* pool, const uint32_t* slow_seq,
                              uint32_t seq, int sms, cudaStream_t st)
{
    if (a.Vc <= 0) return cudaSuccess;
    return sh.d == 128 ? launch_fixup_t<128>(sh, a, pool, slow_seq, seq, sms, st)
                       : launch_fixup_t<64>(sh, a, pool, slow_seq, seq, sms, st);
}

}  // namespace fadkv
