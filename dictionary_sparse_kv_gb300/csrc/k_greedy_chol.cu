// In-pool greedy selection with the ridge refit carried as an incremental
// Cholesky factor in the correlation domain -- binary16 dictionaries, the
// pool resident in registers as mma.sync operands.
//
// "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding":
// abstract (screening-based sparse coding: a one-shot Top-n pool followed by
// lightweight coefficient refinement) and Table 5 (ridge lambda = 1e-4 +
// 0.20 diag(G)).  Greedy selection inside the pool and the lower-index tie
// rule are conventions of this library.
//
// The step the method defines -- pick j* = argmax |<d_j, e_k>| over the
// pool, refit (G_SS + diag(la + lr G_ii)) c = D_S x, e = x - D_S c -- is
// carried without forming e (the way batch OMP carries plain OMP):
// with A_SS = L L^T, z = L^-1 D_S^T x and l_j = L^-1 G_{S,j} for every pool
// atom j,
//   <d_j, e> = r_j - l_j . z                       (r = D x: the screening scores)
//   picking j*:  L_kk = sqrt(G_j*j* (1 + lr) + la - |l_j*|^2),
//                z_k  = <d_j*, e> / L_kk,
//   every j:     l_j[k] = (G_{j,j*} - l_j* . l_j) / L_kk,
//                <d_j, e> -= z_k l_j[k],
//   at the end   c = L^-T z (back substitution), e = x - D_S c.
// Per step the only contraction is the pick's Gram column G_{P,j*}: one
// mma.sync pass of the register-resident pool against the pick's binary16
// row (exact products, fp32 sums).
//
// One CTA of NW warps per vector; warp w holds pool slots 32w .. 32w+31 as
// two m16 tiles of A fragments (loaded from a copy of the pool's rows in
// shared memory, which also serves the pick's row as the B column); lane
// (g8, t4) keeps the Cholesky state of slot t4 of its row group (tile t4>>1,
// row g8 + 8 (t4&1)).  Each warp ends a step by publishing its best slot
// (key, l vector, correlation, |l|^2, G_jj), so one barrier per step
// suffices.
#include <stdlib.h>
#include <string.h>

#include "fadkv_internal.cuh"

namespace fadkv {
namespace {

constexpr int kMT = 2;   // m16 tiles per warp

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

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid)
{
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(valid ? 16 : 0) : "memory");
}

// The pool's copy in shared memory: row r (D binary16) holds its 16-byte
// chunk c at position c ^ (r & 7), so the fragment loads of a warp (rows
// g8 = 0..7, chunks t4 + 4 kp) spread over all banks.
__device__ __forceinline__ const uint4* prow_chunk(const __half* prow, int D, int r, int c)
{
    return reinterpret_cast<const uint4*>(prow + (size_t)r * D + ((c ^ (r & 7)) << 3));
}

// RT: m16 tiles per warp whose A fragments stay in registers (2: all; 1:
// the second tile is read from the shared copy at every pass, which frees
// the registers for three CTAs per SM).  FIXED: s == SMAX, known at compile
// time, so the pick loop unrolls and every index into the per-slot factor
// row is a constant.
template <int D, int NW, int SMAX, int RT, bool FIXED>
__global__ void __launch_bounds__(NW * 32, NW <= 8 ? (RT == 2 ? 2 : 3) : 1)
greedy_chol_kernel(Shape sh, GreedyArgs a)
{
    pdl_begin();
    constexpr int KT = D / 16, KP = D / 32, NT = NW * 32;
    constexpr int SPW = kMT * 16, NPAD = NW * SPW;
    constexpr int PL = SMAX + 4;                 // published floats: l[SMAX], corr, |l|^2, G_jj, slot
    const int vc = blockIdx.x, g = blockIdx.y;
    const int v = a.v0 + vc;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int n = sh.n, s = FIXED ? SMAX : sh.s, N = sh.N;

    __shared__ float xs[D];
    __shared__ int pid[NPAD];
    __shared__ __align__(16) __half bx[2 * D];         // first pass: x 2^p split in two binary16 terms
    __shared__ __align__(16) float publ[2][NW][PL];    // each warp's best: l, corr, |l|^2, G_jj, slot
    __shared__ unsigned long long kred[2][NW];
    extern __shared__ __align__(16) unsigned char dsm[];
    __half* prow = (__half*)dsm;                       // the pool's rows [NPAD][D], chunk-swizzled
    __shared__ float zrec[SMAX], irec[SMAX], lrow[SMAX][SMAX + 1];
    __shared__ int sslot[SMAX];
    __shared__ float fred[NW];

    const size_t gv = (size_t)g * a.Vc + vc;
    const __half* X = (const __half*)a.x + ((size_t)g * a.V + v) * D;
    const __half* Aglob = (const __half*)a.atoms + (size_t)g * N * D;
    long long* cnt = a.counters + (size_t)g * kCntFields;
    unsigned long long* status = (unsigned long long*)&cnt[kCntStatus];
    const size_t out = (size_t)g * a.V + v;

    // ---- x, its norm and finiteness; the pool ----
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
    for (int i = tid; i < NPAD; i += NT) pid[i] = (i < n) ? a.pool_in[gv * n + i] : -1;
    bad = __syncthreads_or(bad);
    if (!bad) {
        // the pool's rows into shared memory (coalesced 16-byte copies; a
        // thread keeps one 16-byte column of the rows)
        static_assert(NT % (D / 8) == 0, "whole rows per pass");
        const int part = tid % (D / 8);
        const __half* src0 = Aglob + 8 * part;
        for (int row = tid / (D / 8); row < NPAD; row += NT / (D / 8)) {
            const int id = pid[row];
            cp_async16(prow + (size_t)row * D + ((part ^ (row & 7)) << 3), src0 + (size_t)(id >= 0 ? id : 0) * D,
                       id >= 0);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();
    }
    if (bad) {
        for (int k = tid; k < s; k += NT) {
            a.idx[out * s + k] = -1;
            a.coef[out * s + k] = 0.f;
        }
        if (tid == 0) {
            a.relres[out] = __int_as_float(0x7fc00000);
            atomicAdd((unsigned long long*)&cnt[kCntNonfinite], 1ull);
            atomicOr(status, (unsigned long long)FADKV_DEV_NONFINITE_INPUT);
        }
        return;
    }
    float xnorm2 = 0.f;
    for (int w = 0; w < NW; ++w) xnorm2 += fred[w];

    // ---- pool atoms -> A fragments; G_jj of this lane's slot ----
    // Inside each 32-element block of the head dimension, thread t4 of a row
    // holds elements 8 t4 .. 8 t4 + 7 (one 16-byte load): a permutation of the
    // contraction index applied alike to A and B.
    uint32_t Af[RT][KT][4];
    float dlo[kMT], dhi[kMT];         // diag(A A^T) of rows g8 and g8 + 8 (lanes with t4 = g8 / 2)
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
        const int s0 = warp * SPW + mt * 16 + g8;
        uint32_t fr[KT][4];
#pragma unroll
        for (int kp = 0; kp < KP; ++kp) {
            const uint4 q0 = *prow_chunk(prow, D, s0, 4 * kp + t4);
            const uint4 q1 = *prow_chunk(prow, D, s0 + 8, 4 * kp + t4);
            fr[2 * kp][0] = q0.x;
            fr[2 * kp][2] = q0.y;
            fr[2 * kp + 1][0] = q0.z;
            fr[2 * kp + 1][2] = q0.w;
            fr[2 * kp][1] = q1.x;
            fr[2 * kp][3] = q1.y;
            fr[2 * kp + 1][1] = q1.z;
            fr[2 * kp + 1][3] = q1.w;
        }
        // A A^T on the tensor pipe: the B fragment of "columns = rows 0..7 of
        // the tile" is (a0, a2) of the same lane, of "rows 8..15" (a1, a3);
        // the diagonal lands in the lanes with 2 t4 = g8 or 2 t4 + 1 = g8
        float plo[2][4] = {}, phi[2][4] = {};
#pragma unroll
        for (int kt = 0; kt < KT; ++kt) {
            hmma(plo[kt & 1], fr[kt], fr[kt][0], fr[kt][2]);
            hmma(phi[kt & 1], fr[kt], fr[kt][1], fr[kt][3]);
        }
        dlo[mt] = (g8 & 1) ? plo[0][1] + plo[1][1] : plo[0][0] + plo[1][0];
        dhi[mt] = (g8 & 1) ? phi[0][3] + phi[1][3] : phi[0][2] + phi[1][2];
        if (mt < RT) {
#pragma unroll
            for (int kt = 0; kt < KT; ++kt)
#pragma unroll
                for (int r = 0; r < 4; ++r) Af[mt < RT ? mt : 0][kt][r] = fr[kt][r];
        }
    }
    // this lane's slot is row (t4 & 1) * 8 + g8 of tile t4 >> 1; its G_jj is
    // held by lane (g8, t4 = g8 / 2)
    float gjj;
    {
        const int src = 4 * g8 + (g8 >> 1);
        const float l0 = __shfl_sync(0xffffffffu, dlo[0], src), l1 = __shfl_sync(0xffffffffu, dlo[1], src);
        const float h0 = __shfl_sync(0xffffffffu, dhi[0], src), h1 = __shfl_sync(0xffffffffu, dhi[1], src);
        gjj = (t4 >> 1) ? ((t4 & 1) ? h1 : l1) : ((t4 & 1) ? h0 : l0);
    }
    const int myslot = warp * SPW + (t4 >> 1) * 16 + (t4 & 1) * 8 + g8;
    const int myatom = pid[myslot];
    bool live = myatom >= 0;

    // scale 2^p with ||x|| < 2^ex: |x_t| 2^p < 2^14 (no binary16 overflow)
    int ex = 0;
    frexpf(sqrtf(xnorm2), &ex);
    const float scale = (xnorm2 > 0.f) ? ldexpf(1.f, 14 - ex) : 1.f;
    const float inv_scale = (xnorm2 > 0.f) ? ldexpf(1.f, ex - 14) : 1.f;
    for (int t = tid; t < D; t += NT) {
        const float sv = xs[t] * scale;
        const __half hi = __float2half_rn(sv);
        bx[t] = hi;
        bx[D + t] = __float2half_rn(sv - __half2float(hi));
    }
    __syncthreads();

    // pool rows x B -> acc.  B column n of this lane (n = g8): `beven(kp)`
    // for even n, `bodd(kp)` for odd n.  With the same data in columns 0, 2,
    // 4, 6 (and 1, 3, 5, 7), lane (g8, t4) finds its slot's results in its
    // own accumulators: column 2 t4 (+ 1) of row g8 / g8 + 8 of each tile.
    float acc[kMT][4];
    auto mma_pass = [&](auto beven, auto bodd) {
        float part[kMT][2][4];
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
            for (int ks = 0; ks < 2; ++ks)
#pragma unroll
                for (int r = 0; r < 4; ++r) part[mt][ks][r] = 0.f;
#pragma unroll
        for (int kp = 0; kp < KP; ++kp) {
            const uint4 qb = (g8 & 1) ? bodd(kp) : beven(kp);
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt) {
                if (mt < RT) {
                    hmma(part[mt][kp & 1], Af[mt < RT ? mt : 0][2 * kp], qb.x, qb.y);
                    hmma(part[mt][kp & 1], Af[mt < RT ? mt : 0][2 * kp + 1], qb.z, qb.w);
                } else {
                    const int s0 = warp * SPW + mt * 16 + g8;
                    const uint4 q0 = *prow_chunk(prow, D, s0, 4 * kp + t4);
                    const uint4 q1 = *prow_chunk(prow, D, s0 + 8, 4 * kp + t4);
                    const uint32_t f0[4] = {q0.x, q1.x, q0.y, q1.y};
                    const uint32_t f1[4] = {q0.z, q1.z, q0.w, q1.w};
                    hmma(part[mt][kp & 1], f0, qb.x, qb.y);
                    hmma(part[mt][kp & 1], f1, qb.z, qb.w);
                }
            }
        }
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[mt][r] = part[mt][0][r] + part[mt][1][r];
    };
    // this lane's slot (t4: tile t4 >> 1, row g8 + 8 (t4 & 1)): even column,
    // plus the odd one when `two`
    auto mine = [&](bool two) -> float {
        const int h = t4 & 1;
        const float* am = (t4 >> 1) ? acc[1] : acc[0];
        const float e = h ? am[2] : am[0];
        const float o = h ? am[3] : am[1];
        return two ? e + o : e;
    };
    const auto zero16 = [](int) { return make_uint4(0u, 0u, 0u, 0u); };

    // ---- first pass: r_j for the pool ----
    mma_pass([&](int kp) { return *reinterpret_cast<const uint4*>(bx + 32 * kp + 8 * t4); },
             [&](int kp) { return *reinterpret_cast<const uint4*>(bx + D + 32 * kp + 8 * t4); });
    float corr = mine(true) * inv_scale;
    float ll = 0.f;
    float l[SMAX];
#pragma unroll
    for (int i = 0; i < SMAX; ++i) l[i] = 0.f;

    // this warp's best live slot (larger |corr|, then the lower atom) -> publish
    auto best_publish = [&](int par, int k) {
        const uint32_t key = live ? (__float_as_uint(corr) & 0x7fffffffu) + 1u : 0u;
        const uint32_t m = __reduce_max_sync(0xffffffffu, key);
        const uint32_t cand = (live && key == m) ? (uint32_t)myatom : 0xffffffffu;
        const uint32_t amin = __reduce_min_sync(0xffffffffu, cand);
        const bool win = m != 0u && live && key == m && (uint32_t)myatom == amin;
        const unsigned wb = __ballot_sync(0xffffffffu, win);
        if (lane == 0) kred[par][warp] = (m == 0u) ? 0ull : (((unsigned long long)m << 32) | (0xffffffffu - amin));
        if (wb != 0u && lane == __ffs(wb) - 1) {
            float* pl = publ[par][warp];
#pragma unroll
            for (int i = 0; i < SMAX; ++i)
                if (i < k) pl[i] = l[i];
            pl[SMAX] = corr;
            pl[SMAX + 1] = ll;
            pl[SMAX + 2] = gjj;
            pl[SMAX + 3] = __int_as_float(myslot);
        }
    };
    best_publish(0, 0);
    __syncthreads();

    const float la = sh.lambda_abs, lr = sh.lambda_rel;
#pragma unroll (FIXED ? SMAX : 1)
    for (int k = 0; k < s; ++k) {
        // ---- the pick: best of the warps' bests (lane w reads warp w's key) ----
        const int par = k & 1;
        const unsigned long long kv = (lane < NW) ? kred[par][lane] : 0ull;
        const uint32_t khi = (uint32_t)(kv >> 32), klo = (uint32_t)kv;
        const uint32_t mhi = __reduce_max_sync(0xffffffffu, khi);
        const uint32_t mlo = __reduce_max_sync(0xffffffffu, khi == mhi ? klo : 0u);
        const int w_o = __ffs(__ballot_sync(0xffffffffu, lane < NW && khi == mhi && klo == mlo)) - 1;
        const float* pl = publ[par][w_o];
        const float4 pq = *reinterpret_cast<const float4*>(pl + SMAX);
        const float cstar = pq.x, llstar = pq.y, gstar = pq.z;
        const int slot_o = __float_as_int(pq.w);
        float dk = fmaf(gstar, lr, gstar) + la - llstar;
        if (!(dk > 0.f)) {
            if (tid == 0) atomicOr(status, (unsigned long long)FADKV_DEV_NOT_SPD);
            dk = 1e-30f;
        }
        const float inv = rsqrtf(dk);                  // 1 / L_kk
        const float zk = cstar * inv;
        if (live && myslot == slot_o) live = false;
        if (warp == 0) {
            // the factor's row k and z_k for the end
            if (lane < k) lrow[k][lane] = pl[lane];
            if (lane == 0) {
                sslot[k] = slot_o;
                zrec[k] = zk;
                irec[k] = inv;
            }
        }
        if (k + 1 == s) break;

        // ---- Gram column of the pick; every slot's update ----
        mma_pass([&](int kp) { return *prow_chunk(prow, D, slot_o, 4 * kp + t4); }, zero16);
        const float gj = mine(false);
        float dot = 0.f;
#pragma unroll
        for (int i4 = 0; i4 < SMAX; i4 += 4) {
            if (i4 < k) {
                const float4 q = *reinterpret_cast<const float4*>(pl + i4);
                if (i4 + 0 < k) dot = fmaf(q.x, l[i4 + 0], dot);
                if (i4 + 1 < k) dot = fmaf(q.y, l[i4 + 1], dot);
                if (i4 + 2 < k) dot = fmaf(q.z, l[i4 + 2], dot);
                if (i4 + 3 < k) dot = fmaf(q.w, l[i4 + 3], dot);
            }
        }
        const float t = (gj - dot) * inv;
#pragma unroll
        for (int i = 0; i < SMAX; ++i)
            if (i == k) l[i] = t;
        ll = fmaf(t, t, ll);
        corr = fmaf(-zk, t, corr);
        best_publish(par ^ 1, k + 1);
        __syncthreads();
    }

    // ---- coefficients c = L^-T z, residual and outputs (warp 0) ----
    if (warp != 0) return;
    __syncwarp();
    // lane j holds c_j: for k = s-1 .. 0, c_k = acc_k / L_kk, then every
    // lane j < k removes L[k][j] c_k from its acc_j
    float accj = (lane < s) ? zrec[lane] : 0.f;
    const float invj = (lane < s) ? irec[lane] : 0.f;
    float cj = 0.f;
#pragma unroll
    for (int k = SMAX - 1; k >= 0; --k) {
        if (k < s) {
            const float ck = __shfl_sync(0xffffffffu, accj * invj, k);
            if (lane == k) cj = ck;
            if (lane < k) accj = fmaf(-lrow[k][lane], ck, accj);
        }
    }
    // e = x - D_S c on D/32 consecutive elements per lane
    constexpr int EPL = D / 32;
    float e[EPL];
#pragma unroll
    for (int u = 0; u < EPL; ++u) e[u] = xs[lane * EPL + u];
#pragma unroll
    for (int i = 0; i < SMAX; ++i) {
        const float ci = __shfl_sync(0xffffffffu, cj, i);
        if (i < s) {
#pragma unroll
            for (int u = 0; u < EPL; u += 2) {
                const int r = sslot[i], e0 = lane * EPL + u;
                const float2 d2 = __half22float2(*reinterpret_cast<const __half2*>(
                    reinterpret_cast<const __half*>(prow_chunk(prow, D, r, e0 >> 3)) + (e0 & 7)));
                e[u] = fmaf(-ci, d2.x, e[u]);
                e[u + 1] = fmaf(-ci, d2.y, e[u + 1]);
            }
        }
    }
    float esq = 0.f;
#pragma unroll
    for (int u = 0; u < EPL; ++u) esq = fmaf(e[u], e[u], esq);
    esq = warp_sum(esq);
    if (lane == 0) a.relres[out] = (xnorm2 > 0.f) ? sqrtf(esq) / sqrtf(xnorm2) : 0.f;
    if (lane < s) {
        a.idx[out * s + lane] = pid[sslot[lane]];
        a.coef[out * s + lane] = cj;
    }
}

// Both tiles in registers (two CTAs per SM) by default: measured faster on
// decode shapes than FADKV_CHOL_RT=1 (three CTAs per SM, second tile read
// from shared memory at every pass), also with the unrolled pick loop
// (3B decode step: 227 us against 283 us per launch).
int resident_tiles()
{
    const char* f = getenv("FADKV_CHOL_RT");
    return (f && strcmp(f, "1") == 0) ? 1 : 2;
}

template <int D, int NW, int SMAX, int RT>
cudaError_t launch_rt(const Shape& sh, const GreedyArgs& a, cudaStream_t st)
{
    const size_t smem = (size_t)NW * kMT * 16 * D * 2;
    auto k = sh.s == SMAX ? greedy_chol_kernel<D, NW, SMAX, RT, true> : greedy_chol_kernel<D, NW, SMAX, RT, false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.Vc, sh.G);
    return launch_pdl(k, grid, dim3(NW * 32), smem, st, sh, a);
}

template <int D, int NW, int SMAX>
cudaError_t launch_t(const Shape& sh, const GreedyArgs& a, cudaStream_t st)
{
    return resident_tiles() == 2 ? launch_rt<D, NW, SMAX, 2>(sh, a, st) : launch_rt<D, NW, SMAX, 1>(sh, a, st);
}

template <int D, int NW>
cudaError_t launch_s(const Shape& sh, const GreedyArgs& a, cudaStream_t st)
{
    return sh.s <= 8 ? launch_t<D, NW, 8>(sh, a, st) : launch_t<D, NW, 16>(sh, a, st);
}

template <int D>
cudaError_t launch_d(const Shape& sh, const GreedyArgs& a, cudaStream_t st)
{
    return sh.n <= 256 ? launch_s<D, 8>(sh, a, st) : launch_s<D, 16>(sh, a, st);
}

}  // namespace

bool greedy_chol_supported(const Shape& sh)
{
    return sh.dtype == FADKV_F16 && (sh.d == 64 || sh.d == 128) && sh.n <= 512 && sh.s <= 16;
}

cudaError_t launch_greedy_chol(const Shape& sh, const GreedyArgs& a, cudaStream_t st)
{
    if (a.Vc <= 0) return cudaSuccess;
    if (!a.pool_in) return cudaErrorInvalidValue;
    return sh.d == 128 ? launch_d<128>(sh, a, st) : launch_d<64>(sh, a, st);
}

}  // namespace fadkv
