// Fixed-size dictionary adaptation and sparse reconstruction.
//
// "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning
// Decoding": abstract (a fixed-size dictionary adaptation mechanism reuses
// inactive atoms instead of expanding the dictionary; each token's KV state
// is a sparse combination of atoms), Fig. 2 caption (if the reconstruction
// error is high, an inactive atom is replaced by a context-relevant atom and
// the dictionary size stays fixed) and Table 5 (delta = 0.50 key / 0.70
// value).  The replacement order is a convention of this library: the m-th
// flagged vector (ascending index) takes the m-th inactive atom (ascending
// index), which block-wide ordered compactions produce deterministically --
// never the order in which atomics happen to land.
#include "fadkv_internal.cuh"

namespace fadkv {
namespace {

constexpr int kAdaptThreads = 1024;
constexpr int kAdaptWarps = kAdaptThreads / 32;

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Ordered compaction over [0, count): out[pos] = i for every i with pred(i),
// in ascending i.  Returns the number kept.  Whole block must call it.
template <typename Pred>
__device__ int block_compact(int count, Pred pred, int32_t* out, int* ws)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int base = 0;
    for (int i0 = 0; i0 < count; i0 += kAdaptThreads) {
        const int i = i0 + tid;
        const int f = (i < count && pred(i)) ? 1 : 0;
        const unsigned bal = __ballot_sync(0xffffffffu, f);
        if (lane == 0) ws[warp] = __popc(bal);
        __syncthreads();
        int before = 0, total = 0;
        for (int w = 0; w < kAdaptWarps; ++w) {
            const int c = ws[w];
            before += (w < warp) ? c : 0;
            total += c;
        }
        if (f) out[base + before + __popc(bal & ((1u << lane) - 1u))] = i;
        base += total;
        __syncthreads();
    }
    return base;
}

// Step 1 of the adaptation for large batches, over the whole grid: usage +=
// 1 for every selected atom and "no replacement" for every vector, so that
// the per-dictionary kernel below is left with the ordered compactions.
__global__ void __launch_bounds__(256)
usage_kernel(int G, int N, int s, int V, const int32_t* __restrict__ idx, int32_t* usage, int32_t* repl_id,
             float* repl_coef)
{
    pdl_begin();
    const long long total = (long long)G * V * s;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int j = idx[i];
        const long long g = i / ((long long)V * s);
        if (j >= 0 && j < N) atomicAdd(&usage[g * N + j], 1);
        if (i % s == 0) {
            repl_id[i / s] = -1;
            repl_coef[i / s] = 0.f;
        }
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kAdaptThreads)
adapt_kernel(Shape sh, AdaptArgs a, DeltaTable delta, int max_batch, int usage_done)
{
    pdl_begin();
    __shared__ int ws[kAdaptWarps];
    const int g = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = sh.N, s = sh.s, V = a.V;
    T* atoms = (T*)a.atoms + (size_t)g * N * D;
    int32_t* usage = a.usage + (size_t)g * N;
    const int32_t* idx = a.idx + (size_t)g * V * s;
    const float* coef = a.coef + (size_t)g * V * s;
    const float* relres = a.relres + (size_t)g * V;
    const T* X = (const T*)a.x + (size_t)g * V * D;
    int32_t* repl_id = a.repl_id + (size_t)g * V;
    float* repl_coef = a.repl_coef + (size_t)g * V;
    int32_t* inactive = a.inactive + (size_t)g * N;
    int32_t* flagged = a.flagged + (size_t)g * max_batch;
    long long* cnt = a.counters + (size_t)g * kCntFields;
    const float dg = delta.v[g];

    // 1. usage += 1 for every selected atom; default "no replacement" (done
    //    by usage_kernel over the whole grid for large batches)
    if (!usage_done) {
        for (int i = tid; i < V * s; i += kAdaptThreads) {
            const int j = idx[i];
            if (j >= 0 && j < N) atomicAdd(&usage[j], 1);
        }
        for (int v = tid; v < V; v += kAdaptThreads) {
            repl_id[v] = -1;
            repl_coef[v] = 0.f;
        }
    }
    __syncthreads();

    // 2. flagged vectors in ascending v; 3. the rows they may take, in
    //    ascending id: inactive atoms (usage == 0) for the fixed-size
    //    adaptation, free slots (usage < 0) for append-only growth (only
    //    needed when some vector is flagged: the N-wide scan is skipped in
    //    the common step with no replacement)
    const int nF = block_compact(V, [&](int v) { return relres[v] > dg; }, flagged, ws);
    const bool app = a.append != 0;
    const int nL = nF > 0 ? block_compact(N, [&](int j) { return app ? usage[j] < 0 : usage[j] == 0; }, inactive, ws)
                          : 0;
    const int m = min(nL, nF);

    // 4. the r-th flagged vector takes the r-th inactive atom (one warp each).
    //    The residual reads only atoms selected in this batch (usage >= 1
    //    after step 1), never a row being overwritten (usage <= 0).
    constexpr int PL = D / 32;
    for (int r = warp; r < m; r += kAdaptWarps) {
        const int v = flagged[r], j = inactive[r];
        float e[PL];
#pragma unroll
        for (int q = 0; q < PL; ++q) e[q] = to_f32(X[(size_t)v * D + lane + 32 * q]);
        for (int k = 0; k < s; ++k) {
            const int sj = idx[(size_t)v * s + k];
            if (sj < 0 || sj >= N) continue;
            const float c = coef[(size_t)v * s + k];
#pragma unroll
            for (int q = 0; q < PL; ++q)
                e[q] = fmaf(-c, to_f32(atoms[(size_t)sj * D + lane + 32 * q]), e[q]);
        }
        float sq = 0.f;
#pragma unroll
        for (int q = 0; q < PL; ++q) sq = fmaf(e[q], e[q], sq);
        const float nrm = sqrtf(warp_sum(sq));
#pragma unroll
        for (int q = 0; q < PL; ++q)
            atoms[(size_t)j * D + lane + 32 * q] = from_f32<T>(nrm > 0.f ? e[q] / nrm : 0.f);
        if (lane == 0) {
            usage[j] = 1;
            repl_id[v] = j;
            repl_coef[v] = nrm;
        }
    }
    if (tid == 0) {
        if (a.nrep) a.nrep[g] = m;
        cnt[kCntEncoded] += V;
        cnt[kCntReplaced] += m;
        cnt[kCntFlagged] += nF;
        cnt[kCntOverflow] += nF - m;
    }
}

// PL consecutive elements of a row as fp32, one vector load (rows are
// 16-byte aligned: atoms are, and a row is 128 or 256 bytes).
template <int PL>
__device__ __forceinline__ void load_row(const __half* p, float (&r)[PL])
{
    static_assert(PL == 2 || PL == 4, "64 or 128 elements per row");
    if constexpr (PL == 4) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
        r[0] = a.x; r[1] = a.y; r[2] = b.x; r[3] = b.y;
    } else {
        const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(p));
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u));
        r[0] = a.x; r[1] = a.y;
    }
}
template <int PL>
__device__ __forceinline__ void load_row(const float* p, float (&r)[PL])
{
    if constexpr (PL == 4) {
        const float4 u = __ldg(reinterpret_cast<const float4*>(p));
        r[0] = u.x; r[1] = u.y; r[2] = u.z; r[3] = u.w;
    } else {
        const float2 u = __ldg(reinterpret_cast<const float2*>(p));
        r[0] = u.x; r[1] = u.y;
    }
}

// x_hat = D_S c (+ repl_coef d_repl), one warp per vector: lane k reads
// term k's atom id and coefficient and every lane the replacement's, then
// every term's row is loaded at once, each lane taking D/32 consecutive
// elements.
template <typename T, int D>
__global__ void __launch_bounds__(256)
reconstruct_kernel(const T* __restrict__ atoms, int G, int N, int s, int V, const int32_t* __restrict__ idx,
                   const float* __restrict__ coef, const int32_t* __restrict__ repl_id,
                   const float* __restrict__ repl_coef, float* __restrict__ xhat)
{
    pdl_begin();
    constexpr int PL = D / 32;
    static_assert(kMaxS <= 32, "one term per lane");
    const int lane = threadIdx.x & 31;
    const long long gv = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (gv >= (long long)G * V) return;
    const int g = (int)(gv / V);
    const T* A = atoms + (size_t)g * N * D;
    int jt = -1, jr = -1;
    float ct = 0.f, cr = 0.f;
    if (lane < s) {
        jt = idx[gv * s + lane];
        ct = coef[gv * s + lane];
    }
    if (repl_id) {
        jr = repl_id[gv];
        cr = repl_coef[gv];
    }
    // skipped terms: a valid row weighted by zero
    if (jt < 0 || jt >= N) {
        jt = 0;
        ct = 0.f;
    }
    if (jr < 0 || jr >= N) {
        jr = 0;
        cr = 0.f;
    }
    float acc[PL];
    {
        float r[PL];
        load_row(A + (size_t)jr * D + lane * PL, r);
#pragma unroll
        for (int q = 0; q < PL; ++q) acc[q] = cr * r[q];
    }
    // terms in batches of 8: all eight rows are loaded before any is used
    // (terms past s read row 0 with weight 0)
    for (int k0 = 0; k0 < s; k0 += 8) {
        float r[8][PL];
        float c8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int j = __shfl_sync(0xffffffffu, jt, (k0 + u) & 31);
            c8[u] = __shfl_sync(0xffffffffu, ct, (k0 + u) & 31);
            load_row(A + (size_t)(k0 + u < s ? j : 0) * D + lane * PL, r[u]);
            if (k0 + u >= s) c8[u] = 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int q = 0; q < PL; ++q) acc[q] = fmaf(c8[u], r[u][q], acc[q]);
    }
    float* out = xhat + gv * D + lane * PL;
#pragma unroll
    for (int q = 0; q < PL; ++q) out[q] = acc[q];
}

// Selected atoms per dictionary above which step 1 runs over the whole grid
// (one CTA per dictionary would take its atomics one after another).
constexpr long long kUsageSplit = 16384;

template <typename T, int D>
cudaError_t adapt_t(const Shape& sh, const AdaptArgs& a, const DeltaTable& delta, int max_batch,
                    cudaStream_t st)
{
    const bool split = (long long)a.V * sh.s > kUsageSplit;
    if (split) {
        const long long total = (long long)sh.G * a.V * sh.s;
        const long long want = (total + 255) / 256;
        const unsigned blocks = (unsigned)(want < 4096 ? want : 4096);
        const cudaError_t e = launch_pdl(usage_kernel, dim3(blocks), dim3(256), 0, st, sh.G, sh.N, sh.s, a.V, a.idx,
                                         a.usage, a.repl_id, a.repl_coef);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(adapt_kernel<T, D>, dim3(sh.G), dim3(kAdaptThreads), 0, st, sh, a, delta, max_batch,
                      split ? 1 : 0);
}

template <typename T, int D>
cudaError_t reconstruct_t(const Shape& sh, const void* atoms, int V, const int32_t* idx, const float* coef,
                          const int32_t* repl_id, const float* repl_coef, float* xhat, cudaStream_t st)
{
    const long long warps = (long long)sh.G * V;
    const unsigned blocks = (unsigned)((warps + 7) / 8);
    return launch_pdl(reconstruct_kernel<T, D>, dim3(blocks), dim3(256), 0, st, (const T*)atoms, sh.G, sh.N, sh.s, V,
                      idx, coef, repl_id, repl_coef, xhat);
}

}  // namespace

int adapt_launches(const Shape& sh, int V) { return (long long)V * sh.s > kUsageSplit ? 2 : 1; }

cudaError_t launch_adapt(const Shape& sh, const AdaptArgs& a, const DeltaTable& delta, cudaStream_t st)
{
    // flagged scratch holds max_batch entries per dictionary; V <= max_batch
    // is checked on the host, so the stride V is a valid lower bound here.
    const int stride = a.V > 0 ? a.V : 1;
    if (sh.dtype == FADKV_F16) {
        if (sh.d == 128) return adapt_t<__half, 128>(sh, a, delta, stride, st);
        return adapt_t<__half, 64>(sh, a, delta, stride, st);
    }
    if (sh.d == 128) return adapt_t<float, 128>(sh, a, delta, stride, st);
    return adapt_t<float, 64>(sh, a, delta, stride, st);
}

cudaError_t launch_reconstruct(const Shape& sh, const void* atoms, int V, const int32_t* idx,
                               const float* coef, const int32_t* repl_id, const float* repl_coef,
                               float* xhat, cudaStream_t st)
{
    if (V <= 0) return cudaSuccess;
    if (sh.dtype == FADKV_F16) {
        if (sh.d == 128) return reconstruct_t<__half, 128>(sh, atoms, V, idx, coef, repl_id, repl_coef, xhat, st);
        return reconstruct_t<__half, 64>(sh, atoms, V, idx, coef, repl_id, repl_coef, xhat, st);
    }
    if (sh.d == 128) return reconstruct_t<float, 128>(sh, atoms, V, idx, coef, repl_id, repl_coef, xhat, st);
    return reconstruct_t<float, 64>(sh, atoms, V, idx, coef, repl_id, repl_coef, xhat, st);
}

}  // namespace fadkv
