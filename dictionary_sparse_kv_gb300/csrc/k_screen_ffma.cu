// Screening scores on the FP32 pipe: r[g][v][j] = <x_gv, d_gj>.
//
// "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding",
// abstract: screening-based sparse coding starts from the correlations of the
// incoming vector with every atom of the dictionary.
//
// This is the general path: binary32 dictionaries (no TF32: the products must
// stay exact to IEEE fp32 rounding), and the reference for the tensor-core
// path.  One CTA computes a 64-vector x 64-atom tile with the whole head
// dimension staged in shared memory as fp32; each thread owns a 4 x 4 block
// of outputs.  Products are exact in fp32 for binary16 inputs; sums are in
// index order t = 0..d-1 (fmaf).
#include "fadkv_internal.cuh"

namespace fadkv {
namespace {

constexpr int kTileV = 64;
constexpr int kTileA = 64;
constexpr int kThreads = 256;

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
screen_ffma_kernel(const T* __restrict__ atoms, const T* __restrict__ x, long long x_gstride,
                   int N, int v0, int Vc, float* __restrict__ scores)
{
    constexpr int KP = D + 1;   // padded row: conflict-free column reads
    extern __shared__ float sm[];
    float* xs = sm;                    // [kTileV][KP]
    float* ds = sm + kTileV * KP;      // [kTileA][KP]

    const int g = blockIdx.z;
    const int j0 = blockIdx.x * kTileA;
    const int vt = blockIdx.y * kTileV;   // tile start inside the chunk
    const T* A = atoms + (size_t)g * N * D;
    const T* X = x + (size_t)g * x_gstride + (size_t)v0 * D;

    for (int i = threadIdx.x; i < kTileV * D; i += kThreads) {
        const int r = i / D, c = i % D;
        xs[r * KP + c] = (vt + r < Vc) ? to_f32(X[(size_t)(vt + r) * D + c]) : 0.f;
    }
    for (int i = threadIdx.x; i < kTileA * D; i += kThreads) {
        const int r = i / D, c = i % D;
        ds[r * KP + c] = (j0 + r < N) ? to_f32(A[(size_t)(j0 + r) * D + c]) : 0.f;
    }
    __syncthreads();

    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

#pragma unroll 4
    for (int k = 0; k < D; ++k) {
        float xv[4], dv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) xv[i] = xs[(ty * 4 + i) * KP + k];
#pragma unroll
        for (int j = 0; j < 4; ++j) dv[j] = ds[(tx + 16 * j) * KP + k];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], dv[j], acc[i][j]);
    }

    float* out = scores + (size_t)g * Vc * N;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int v = vt + ty * 4 + i;
        if (v >= Vc) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int a = j0 + tx + 16 * j;
            if (a < N) out[(size_t)v * N + a] = acc[i][j];
        }
    }
}

template <typename T, int D>
cudaError_t launch_t(const Shape& sh, const void* atoms, const void* x, int64_t x_gstride, int v0,
                     int Vc, float* scores, cudaStream_t st)
{
    const size_t smem = sizeof(float) * (size_t)(kTileV + kTileA) * (D + 1);
    auto k = screen_ffma_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((sh.N + kTileA - 1) / kTileA, (Vc + kTileV - 1) / kTileV, sh.G);
    k<<<grid, kThreads, smem, st>>>((const T*)atoms, (const T*)x, (long long)x_gstride, sh.N, v0, Vc,
                                    scores);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_screen_ffma(const Shape& sh, const void* atoms, const void* x, int64_t x_gstride,
                               int v0, int Vc, float* scores, cudaStream_t st)
{
    if (Vc <= 0) return cudaSuccess;
    if (sh.dtype == FADKV_F16) {
        if (sh.d == 128) return launch_t<__half, 128>(sh, atoms, x, x_gstride, v0, Vc, scores, st);
        return launch_t<__half, 64>(sh, atoms, x, x_gstride, v0, Vc, scores, st);
    }
    if (sh.d == 128) return launch_t<float, 128>(sh, atoms, x, x_gstride, v0, Vc, scores, st);
    return launch_t<float, 64>(sh, atoms, x, x_gstride, v0, Vc, scores, st);
}

}  // namespace fadkv
