// The dictionaries' Gram matrices and the in-pool greedy selection over them.
//
// "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding":
// abstract (screening-based sparse coding: a one-shot Top-n pool followed by
// lightweight coefficient refinement) and Table 5 (ridge lambda = 1e-4 +
// 0.20 diag(G)).  Greedy selection inside the pool and the lower-index tie
// rule are conventions of this library.
//
// A greedy step -- pick j* = argmax |<d_j, e_k>| over the pool, refit
// (G_SS + diag(la + lr G_ii)) c = D_S x, e = x - D_S c -- touches the atoms
// only through inner products: <d_j, x> (the screening scores, carried with
// the pool) and <d_j, d_j*> (the Gram matrix).  With every dictionary's Gram
// matrix kept up to date next to it, the refit is carried in the
// correlation domain without forming e (batch OMP, Rubinstein, Zibulevsky
// and Elad 2008): with A_SS = L L^T, z = L^-1 D_S^T x and l_j = L^-1 G_{S,j}
// for every pool atom j,
//   <d_j, e> = r_j - l_j . z
//   picking j*:  L_kk = sqrt(G_j*j* (1 + lr) + la - |l_j*|^2),
//                z_k  = <d_j*, e> / L_kk,
//   every j:     l_j[k] = (G_{j,j*} - l_j* . l_j) / L_kk,
//                <d_j, e> -= z_k l_j[k],
//   at the end   c = L^-T z (back substitution), e = x - D_S c.
// A pick then costs one gather of n Gram entries (row j* at the pool's atom
// ids) and O(k) flops per pool atom; nothing of the pool's atoms is read.
//
// Gram matrix: gram [G][N][N] fp32, gram[g][i][j] = <d_i, d_j> summed in
// ascending element order by fused multiply-adds of the binary16 elements
// widened to fp32, so the entry is the same whichever of the two atoms is
// taken first: the matrix is exactly symmetric.  gdiag [G][N] is its
// diagonal.  It is built once (gram_kernel over every row) and after each
// adaptation only the rows and columns of the atoms just written are
// recomputed.
#include "fadkv_internal.cuh"

namespace fadkv {
namespace {

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------------------
// Gram build and update
// ---------------------------------------------------------------------------
constexpr int kGT = 64;                 // rows and columns of a tile
constexpr int kGThreads = 256;          // 16 x 16 threads, 4 x 4 entries each

// Loads atoms ids[0..count) (ids null: first + i) of dictionary A into
// S[t][i] as fp32 (element-major, so a thread's four rows are one float4).
template <int D>
__device__ __forceinline__ void load_tile(float (*S)[kGT], const __half* A, const int32_t* ids, int first,
                                          int count)
{
    constexpr int CPR = D / 8;                         // 16-byte chunks per atom
    for (int c = threadIdx.x; c < kGT * CPR; c += kGThreads) {
        const int i = c % kGT, part = c / kGT;
        uint4 q = make_uint4(0u, 0u, 0u, 0u);
        if (i < count) {
            const int j = ids ? ids[i] : first + i;
            q = __ldg(reinterpret_cast<const uint4*>(A + (size_t)j * D) + part);
        }
        const __half2* h = reinterpret_cast<const __half2*>(&q);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 f = __half22float2(h[u]);
            S[part * 8 + 2 * u][i] = f.x;
            S[part * 8 + 2 * u + 1][i] = f.y;
        }
    }
}

// gram[g][r][c] = <d_r, d_c> for the rows r of a list and every column c,
// in 64 x 64 tiles handed out over the grid: tile t of dictionary g is row
// tile t / ctiles (of its row list) and column tile t % ctiles.  Build
// (rows == null): every atom is a row.  Update: the rows are the nrows[g]
// ids at rows + g * row_stride, and every entry is also written at [c][r]
// (both orders give the same bits); a dictionary with no rows has no tiles,
// so an update after a step that replaced nothing costs one pass over the
// counts.
template <int D>
__global__ void __launch_bounds__(kGThreads)
gram_kernel(const __half* __restrict__ atoms, int G, int N, const int32_t* __restrict__ rows,
            const int32_t* __restrict__ nrows, int row_stride, float* __restrict__ gram, float* __restrict__ gdiag)
{
    pdl_begin();
    extern __shared__ __align__(16) float gsm[];
    float (*As)[kGT] = reinterpret_cast<float (*)[kGT]>(gsm);
    float (*Bs)[kGT] = reinterpret_cast<float (*)[kGT]>(gsm + D * kGT);
    const bool update = rows != nullptr;
    const int ctiles = (N + kGT - 1) / kGT;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    // the tiles of dictionaries [0, g) come before those of g; the total
    // over every dictionary by each warp (lanes over dictionaries): an
    // update after a step without replacements leaves at once
    long long total = 0;
    for (int g = (int)(threadIdx.x & 31); g < G; g += 32) {
        const int nr = update ? nrows[g] : N;
        total += (long long)((nr + kGT - 1) / kGT) * ctiles;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    if (total == 0) return;
    // tiles [gbase, gend) belong to dictionary g; t only grows, so g only
    // advances, and t < total keeps it below G
    int g = -1;
    long long gbase = 0, gend = 0;
    for (long long t = blockIdx.x; t < total; t += gridDim.x) {
        while (t >= gend) {
            ++g;
            gbase = gend;
            const int ng = update ? nrows[g] : N;
            gend += (long long)((ng + kGT - 1) / kGT) * ctiles;
        }
        const int nr = update ? nrows[g] : N;
        const long long lt = t - gbase;
        const int r0 = (int)(lt / ctiles) * kGT, c0 = (int)(lt % ctiles) * kGT;
        const int rcount = min(kGT, nr - r0), ccount = min(kGT, N - c0);
        const int32_t* rl = update ? rows + (size_t)g * row_stride : nullptr;
        const __half* A = atoms + (size_t)g * N * D;
        float* Gg = gram + (size_t)g * N * N;
        __syncthreads();
        load_tile<D>(Bs, A, nullptr, c0, ccount);
        load_tile<D>(As, A, rl ? rl + r0 : nullptr, r0, rcount);
        __syncthreads();
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 8
        for (int k = 0; k < D; ++k) {
            const float4 av = *reinterpret_cast<const float4*>(&As[k][ty * 4]);
            const float4 bv = *reinterpret_cast<const float4*>(&Bs[k][tx * 4]);
            const float ar[4] = {av.x, av.y, av.z, av.w}, br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int ri = ty * 4 + i;
            if (ri >= rcount) continue;
            const int r = rl ? rl[r0 + ri] : r0 + ri;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int cj = tx * 4 + j;
                if (cj >= ccount) continue;
                const int c = c0 + cj;
                Gg[(size_t)r * N + c] = acc[i][j];
                if (update) Gg[(size_t)c * N + r] = acc[i][j];
                if (r == c) gdiag[(size_t)g * N + r] = acc[i][j];
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Greedy selection + ridge refit over the Gram matrix
// ---------------------------------------------------------------------------
// WPV warps per vector; each lane keeps SP pool slots (slot i = sp * 32 WPV
// + 32 w + lane of warp w): the atom id, the running correlation <d_j, e>
// and l_j itself (SMAX - 1 entries: the last pick needs no update); G_jj of
// the slots sits in shared memory and |l_j|^2 is summed by the lane that
// publishes a pick, in the order of l_j's entries.  A CTA of four warps serves 4 / WPV vectors, in the order of
// (dictionary, vector), so consecutive CTAs read the same dictionary's Gram
// matrix.  FIXED: s == SMAX, known at compile time, so the pick loop unrolls
// and every index into a slot's l is a constant.
constexpr int kGreedyWarps = 4;

template <int D, int WPV, int SP, int SMAX, bool FIXED>
__global__ void __launch_bounds__(kGreedyWarps * 32, 4)
greedy_gram_kernel(Shape sh, GramGreedyArgs a)
{
    pdl_begin();
    constexpr int VPC = kGreedyWarps / WPV;
    constexpr int GS = 32 * WPV;
    constexpr int LW = SMAX - 1;
    constexpr int PL = SMAX + 4;                  // published: l[SMAX], corr, |l|^2, G_jj, id
    constexpr int EPL = D / 32;
    static_assert(SMAX % 4 == 0, "published rows are read as float4");
    __shared__ __align__(16) float publ[VPC][2][WPV][PL];
    __shared__ float gjj_s[VPC][GS * SP];           // G_jj of every pool slot (read by the pick's lane)
    __shared__ unsigned long long kred[VPC][2][WPV];
    __shared__ float lrow[VPC][SMAX][SMAX];
    __shared__ float zrec[VPC][SMAX], irec[VPC][SMAX];
    __shared__ int sid[VPC][SMAX];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int grp = warp / WPV, w = warp - grp * WPV;
    const long long gv = (long long)blockIdx.x * VPC + grp;
    if (gv >= (long long)sh.G * a.Vc) return;     // the whole group leaves together
    const int g = (int)(gv / a.Vc), vc = (int)(gv - (long long)g * a.Vc);
    const int v = a.v0 + vc;
    const int n = sh.n, s = FIXED ? SMAX : sh.s, N = sh.N;
    long long* cnt = a.counters + (size_t)g * kCntFields;
    unsigned long long* status = (unsigned long long*)&cnt[kCntStatus];
    const size_t out = (size_t)g * a.V + v;

    auto group_sync = [&]() {
        if constexpr (WPV == 1)
            __syncwarp();
        else
            asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "n"(WPV * 32) : "memory");
    };

    // ---- x: this lane's D/32 consecutive elements, its norm, finiteness ----
    const __half* X = a.x + ((size_t)g * a.V + v) * D;
    float xv[EPL];
    if constexpr (EPL == 4) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(X) + lane);
        const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
        const float2 q = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
        xv[0] = p.x; xv[1] = p.y; xv[2] = q.x; xv[3] = q.y;
    } else {
        const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(X) + lane);
        const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&u));
        xv[0] = p.x; xv[1] = p.y;
    }
    float xsq = 0.f;
    bool finite = true;
#pragma unroll
    for (int u = 0; u < EPL; ++u) {
        finite = finite && isfinite(xv[u]);
        xsq = fmaf(xv[u], xv[u], xsq);
    }
    const float xnorm2 = warp_sum(xsq);
    if (!__all_sync(0xffffffffu, finite)) {
        if (w == 0) {
            if (lane < s) {
                a.idx[out * s + lane] = -1;
                a.coef[out * s + lane] = 0.f;
            }
            if (lane == 0) {
                a.relres[out] = __int_as_float(0x7fc00000);
                atomicAdd((unsigned long long*)&cnt[kCntNonfinite], 1ull);
                atomicOr(status, (unsigned long long)FADKV_DEV_NONFINITE_INPUT);
            }
        }
        return;
    }

    // ---- the pool: ids, scores r_j, G_jj ----
    const size_t pb = ((size_t)g * a.Vc + vc) * n;
    int id[SP];
    float corr[SP], l[SP][LW];
    uint32_t live = 0u;
#pragma unroll
    for (int sp = 0; sp < SP; ++sp) {
        const int i = sp * GS + w * 32 + lane;
        id[sp] = (i < n) ? a.pool[pb + i] : -1;
        corr[sp] = (i < n) ? a.pool_r[pb + i] : 0.f;
        live |= (i < n) ? (1u << sp) : 0u;
    }
#pragma unroll
    for (int sp = 0; sp < SP; ++sp) {
        gjj_s[grp][sp * GS + w * 32 + lane] = id[sp] >= 0 ? __ldg(a.gdiag + (size_t)g * N + id[sp]) : 0.f;
#pragma unroll
        for (int i = 0; i < LW; ++i) l[sp][i] = 0.f;
    }

    const float* Gg = a.gram + (size_t)g * N * N;
    const float la = sh.lambda_abs, lr = sh.lambda_rel;
#pragma unroll(FIXED ? SMAX : 1)
    for (int k = 0; k < s; ++k) {
        const int par = k & 1;
        // ---- this lane's best live slot: larger |corr|, then the lower atom ----
        uint32_t bk = 0u, bid = 0xffffffffu;
        int bsp = 0;
#pragma unroll
        for (int sp = 0; sp < SP; ++sp) {
            const uint32_t key = ((live >> sp) & 1u) ? (__float_as_uint(corr[sp]) & 0x7fffffffu) + 1u : 0u;
            if (key > bk || (key == bk && key != 0u && (uint32_t)id[sp] < bid)) {
                bk = key;
                bid = (uint32_t)id[sp];
                bsp = sp;
            }
        }
        // ---- the warp's best; its lane publishes the slot ----
        const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t amin = __reduce_min_sync(0xffffffffu, (bk == m) ? bid : 0xffffffffu);
        float* pw = publ[grp][par][w];
        if (m != 0u && bk == m && bid == amin) {
            // the winning slot's l (and |l|^2, summed in the order its
            // entries were made), correlation, G_jj and atom
            float llw = 0.f, cw = corr[0];
#pragma unroll
            for (int sp = 1; sp < SP; ++sp) cw = (bsp == sp) ? corr[sp] : cw;
#pragma unroll
            for (int i = 0; i < LW; ++i) {
                if (i < k) {
                    float r = l[0][i];
#pragma unroll
                    for (int sp = 1; sp < SP; ++sp) r = (bsp == sp) ? l[sp][i] : r;
                    pw[i] = r;
                    llw = fmaf(r, r, llw);
                }
            }
            pw[SMAX] = cw;
            pw[SMAX + 1] = llw;
            pw[SMAX + 2] = gjj_s[grp][bsp * GS + w * 32 + lane];
            pw[SMAX + 3] = __int_as_float((int)bid);
        }
        if (WPV > 1 && lane == 0)
            kred[grp][par][w] = (m == 0u) ? 0ull : (((unsigned long long)m << 32) | (0xffffffffu - amin));
        group_sync();
        int wo = 0;
        if constexpr (WPV > 1) {
            const unsigned long long kv = (lane < WPV) ? kred[grp][par][lane] : 0ull;
            const uint32_t khi = (uint32_t)(kv >> 32), klo = (uint32_t)kv;
            const uint32_t mhi = __reduce_max_sync(0xffffffffu, khi);
            const uint32_t mlo = __reduce_max_sync(0xffffffffu, khi == mhi ? klo : 0u);
            wo = __ffs(__ballot_sync(0xffffffffu, lane < WPV && khi == mhi && klo == mlo)) - 1;
        }
        const float* pl = publ[grp][par][wo];
        const float4 pq = *reinterpret_cast<const float4*>(pl + SMAX);
        const float cstar = pq.x, llstar = pq.y, gstar = pq.z;
        const int idstar = __float_as_int(pq.w);
        float dk = fmaf(gstar, lr, gstar) + la - llstar;
        if (!(dk > 0.f)) {
            if (w == 0 && lane == 0) atomicOr(status, (unsigned long long)FADKV_DEV_NOT_SPD);
            dk = 1e-30f;
        }
        const float inv = rsqrtf(dk);                  // 1 / L_kk
        const float zk = cstar * inv;
#pragma unroll
        for (int sp = 0; sp < SP; ++sp)
            if (id[sp] == idstar) live &= ~(1u << sp);
        if (w == 0) {
            // the factor's row k and z_k, for the back substitution
            if (lane < k) lrow[grp][k][lane] = pl[lane];
            if (lane == 0) {
                sid[grp][k] = idstar;
                zrec[grp][k] = zk;
                irec[grp][k] = inv;
            }
        }
        if (k + 1 == s) break;

        // ---- Gram row of the pick at the pool's atoms; every slot's update ----
        const float* grow = Gg + (size_t)idstar * N;
        float gcol[SP];
#pragma unroll
        for (int sp = 0; sp < SP; ++sp) gcol[sp] = __ldg(grow + (id[sp] >= 0 ? id[sp] : 0));
        float lst[LW];
#pragma unroll
        for (int i4 = 0; i4 < LW; i4 += 4) {
            if (i4 < k) {
                const float4 q = *reinterpret_cast<const float4*>(pl + i4);
                lst[i4] = q.x;
                if (i4 + 1 < LW) lst[i4 + 1] = q.y;
                if (i4 + 2 < LW) lst[i4 + 2] = q.z;
                if (i4 + 3 < LW) lst[i4 + 3] = q.w;
            }
        }
#pragma unroll
        for (int sp = 0; sp < SP; ++sp) {
            float dot = 0.f;
#pragma unroll
            for (int i = 0; i < LW; ++i)
                if (i < k) dot = fmaf(lst[i], l[sp][i], dot);
            const float t = (gcol[sp] - dot) * inv;
#pragma unroll
            for (int i = 0; i < LW; ++i)
                if (i == k) l[sp][i] = t;
            corr[sp] = fmaf(-zk, t, corr[sp]);
        }
    }

    // ---- c = L^-T z, the residual and the outputs (warp 0 of the group) ----
    if (w != 0) return;
    __syncwarp();
    // lane j holds c_j: for k = s-1 .. 0, c_k = acc_k / L_kk, then every
    // lane j < k removes L[k][j] c_k from its acc_j
    float accj = (lane < s) ? zrec[grp][lane] : 0.f;
    const float invj = (lane < s) ? irec[grp][lane] : 0.f;
    float cj = 0.f;
#pragma unroll
    for (int k = SMAX - 1; k >= 0; --k) {
        if (k < s) {
            const float ck = __shfl_sync(0xffffffffu, accj * invj, k);
            if (lane == k) cj = ck;
            if (lane < k) accj = fmaf(-lrow[grp][k][lane], ck, accj);
        }
    }
    // e = x - D_S c, this lane's D/32 consecutive elements
    const __half* Ag = a.atoms + (size_t)g * N * D;
    float e[EPL];
#pragma unroll
    for (int u = 0; u < EPL; ++u) e[u] = xv[u];
#pragma unroll
    for (int i = 0; i < SMAX; ++i) {
        const float ci = __shfl_sync(0xffffffffu, cj, i);
        if (i < s) {
            const __half* row = Ag + (size_t)sid[grp][i] * D + lane * EPL;
            float dr[EPL];
            if constexpr (EPL == 4) {
                const uint2 u = __ldg(reinterpret_cast<const uint2*>(row));
                const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
                const float2 q = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
                dr[0] = p.x; dr[1] = p.y; dr[2] = q.x; dr[3] = q.y;
            } else {
                const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(row));
                const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&u));
                dr[0] = p.x; dr[1] = p.y;
            }
#pragma unroll
            for (int u = 0; u < EPL; ++u) e[u] = fmaf(-ci, dr[u], e[u]);
        }
    }
    float esq = 0.f;
#pragma unroll
    for (int u = 0; u < EPL; ++u) esq = fmaf(e[u], e[u], esq);
    esq = warp_sum(esq);
    if (lane == 0) a.relres[out] = (xnorm2 > 0.f) ? sqrtf(esq) / sqrtf(xnorm2) : 0.f;
    if (lane < s) {
        a.idx[out * s + lane] = sid[grp][lane];
        a.coef[out * s + lane] = cj;
    }
}

template <int D, int WPV, int SP, int SMAX>
cudaError_t launch_cfg(const Shape& sh, const GramGreedyArgs& a, cudaStream_t st)
{
    constexpr int VPC = kGreedyWarps / WPV;
    const long long total = (long long)sh.G * a.Vc;
    const unsigned grid = (unsigned)((total + VPC - 1) / VPC);
    auto k = sh.s == SMAX ? greedy_gram_kernel<D, WPV, SP, SMAX, true> : greedy_gram_kernel<D, WPV, SP, SMAX, false>;
    return launch_pdl(k, dim3(grid), dim3(kGreedyWarps * 32), 0, st, sh, a);
}

template <int D>
cudaError_t launch_d(const Shape& sh, const GramGreedyArgs& a, cudaStream_t st)
{
    if (sh.s <= 8) {
        if (sh.n <= 128) return launch_cfg<D, 1, 4, 8>(sh, a, st);
        if (sh.n <= 256) return launch_cfg<D, 1, 8, 8>(sh, a, st);
        return launch_cfg<D, 2, 8, 8>(sh, a, st);
    }
    if (sh.n <= 128) return launch_cfg<D, 1, 4, 16>(sh, a, st);
    if (sh.n <= 256) return launch_cfg<D, 2, 4, 16>(sh, a, st);
    return launch_cfg<D, 4, 4, 16>(sh, a, st);
}

template <int D>
cudaError_t launch_gram_t(const Shape& sh, const void* atoms, const int32_t* rows, const int32_t* nrows,
                          int row_stride, float* gram, float* gdiag, int sms, cudaStream_t st)
{
    const size_t smem = 2 * (size_t)D * kGT * sizeof(float);
    auto k = gram_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // the build: three CTAs per SM (64 KB of shared memory each); an update
    // (usually a few tiles, often none): one per SM
    const unsigned grid = (unsigned)(rows ? sms : 3 * sms);
    return launch_pdl(k, dim3(grid), dim3(kGThreads), smem, st, (const __half*)atoms, sh.G, sh.N, rows, nrows,
                      row_stride, gram, gdiag);
}

}  // namespace

bool greedy_gram_supported(const Shape& sh)
{
    return sh.dtype == FADKV_F16 && (sh.d == 64 || sh.d == 128) && sh.n <= 512 && sh.s <= 16;
}

size_t gram_bytes(const Shape& sh) { return (size_t)sh.G * sh.N * sh.N * sizeof(float); }

cudaError_t launch_gram_build(const Shape& sh, const void* atoms, float* gram, float* gdiag, int sms, cudaStream_t st)
{
    return sh.d == 128 ? launch_gram_t<128>(sh, atoms, nullptr, nullptr, 0, gram, gdiag, sms, st)
                       : launch_gram_t<64>(sh, atoms, nullptr, nullptr, 0, gram, gdiag, sms, st);
}

cudaError_t launch_gram_update(const Shape& sh, const void* atoms, const int32_t* rows, const int32_t* nrows,
                               int row_stride, float* gram, float* gdiag, int sms, cudaStream_t st)
{
    return sh.d == 128 ? launch_gram_t<128>(sh, atoms, rows, nrows, row_stride, gram, gdiag, sms, st)
                       : launch_gram_t<64>(sh, atoms, rows, nrows, row_stride, gram, gdiag, sms, st);
}

cudaError_t launch_greedy_gram(const Shape& sh, const GramGreedyArgs& a, cudaStream_t st)
{
    if (a.Vc <= 0) return cudaSuccess;
    return sh.d == 128 ? launch_d<128>(sh, a, st) : launch_d<64>(sh, a, st);
}

}  // namespace fadkv
