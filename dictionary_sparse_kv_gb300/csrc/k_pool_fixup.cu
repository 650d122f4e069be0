// Exact Top-n pool of the vectors the selection kernel left to the slow path.
//
// "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding",
// abstract: a one-shot Top-n selection gives the candidate pool; ties go to
// the lower atom index (a convention of this library).
//
// The selection kernel marks a vector with pool[0] = -2 when its screening
// records cannot give the pool exactly (a record overflowed, or the list
// holds fewer than n or more than the selection's capacity).  This kernel recomputes all N scores
// of such a vector on the FP32 pipe, takes the exact Top-n keys and writes
// the pool ids with their signed scores r_j.  It returns at once when the
// pass flagged nothing (the selection records the pass number in slow_seq).
#include "select.cuh"

namespace fadkv {
namespace {

struct FixupLayout {
    size_t keys, xs, pid, mag, hist, scan, misc, pref, total;
};

template <int D>
__host__ __device__ inline FixupLayout fixup_layout(int N, int n, int nw)
{
    FixupLayout L;
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
pool_fixup_kernel(Shape sh, GreedyArgs a, int32_t* pool, float* pool_r, const uint32_t* slow_seq, uint32_t seq)
{
    pdl_begin();
    if (*slow_seq != seq) return;                      // no vector of this pass was flagged
    const FixupLayout L = fixup_layout<D>(sh.N, sh.n, kFixThreads / 32);
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
            for (int i = threadIdx.x; i < n; i += kFixThreads) {
                pool[gv * n + i] = i;
                pool_r[gv * n + i] = 0.f;
            }
            __syncthreads();
            continue;
        }
        const __half* A = (const __half*)a.atoms + (size_t)g * N * D;
        long long* cnt = a.counters + (size_t)g * kCntFields;
        const int K = sel::intake_keys<__half, D>(a, (size_t)gv, -1, n, N, A, xs, keys, sc, cnt);
        sel::top_n(keys, K, n, pid, mag, sc);
        // the keys hold |r|: the signed score is the same FP32 dot again
        for (int i = threadIdx.x; i < n; i += kFixThreads) {
            pool[gv * n + i] = pid[i];
            pool_r[gv * n + i] = sel::row_dot_f32<__half, D>(A + (size_t)pid[i] * D, xs);
        }
        __syncthreads();
      }
      __syncthreads();
    }
}

template <int D>
cudaError_t launch_fixup_t(const Shape& sh, const GreedyArgs& a, int32_t* pool, float* pool_r,
                           const uint32_t* slow_seq, uint32_t seq, int sms, cudaStream_t st)
{
    const size_t smem = fixup_layout<D>(sh.N, sh.n, kFixThreads / 32).total;
    auto k = pool_fixup_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long total = (long long)sh.G * a.Vc;
    const long long want = 2LL * sms;
    const unsigned grid = (unsigned)(total < want ? total : want);
    return launch_pdl(k, dim3(grid), dim3(kFixThreads), smem, st, sh, a, pool, pool_r, slow_seq, seq);
}

}  // namespace

cudaError_t launch_pool_fixup(const Shape& sh, const GreedyArgs& a, int32_t* pool, float* pool_r,
                              const uint32_t* slow_seq, uint32_t seq, int sms, cudaStream_t st)
{
    if (a.Vc <= 0) return cudaSuccess;
    return sh.d == 128 ? launch_fixup_t<128>(sh, a, pool, pool_r, slow_seq, seq, sms, st)
                       : launch_fixup_t<64>(sh, a, pool, pool_r, slow_seq, seq, sms, st);
}

}  // namespace fadkv
