// The compressed KV store and decode attention that reads it.
//
// "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding",
// Table 4 (per-sequence KV memory and decode latency of the dictionary
// methods against full KV) and the abstract (each token's KV state is a
// sparse combination of atoms).  The pages give neither a storage format
// nor an attention kernel; this library's choices:
//
// Packed words.  One 32-bit word per nonzero: bits 31..13 hold the
// coefficient rounded to 11 significant bits (round to nearest, ties to
// even) in the layout of binary32's top 19 bits; bits 12..0 the atom id
// (N <= 8192).  A token's code is s + 1 words (its s terms and the
// replacement term, word 0 when absent).
//
// Attention.  For a query q and cached tokens with k_t = sum_i c_ti d_(j_ti):
//   <q, k_t> = sum_i c_ti u_(j_ti),  u = D_K q      (one N x d product per query)
//   sum_t p_t v_t = D_V^T w,  w_j = sum_t p_t sum_i c'_ti [j'_ti = j]
// so neither K nor V is rebuilt: the token loop is s + 1 gathers from u and
// s + 1 scatters into w per token.  One CTA per (layer, sequence, KV head)
// handles the query heads that share the KV head, `hp` of them per pass:
//   1. u = scale D_K q for the pass's heads (FP32 pipe, rows read once,
//      a half-warp per row);
//   2. tokens in chunks (1024 with s + 1 <= 9 words): every thread loads all
//      words of its tokens at once, keeps their scores in registers, the
//      block forms the chunk's maximum; when the running maximum grows, w
//      and the partial sums are rescaled (online softmax at chunk
//      granularity); then p = exp(score - max) and the value codes scatter
//      p c' into w;
//   3. o = D_V^T w / sum p.
// With binary16 dictionaries steps 1 and 3 run instead as two per-layer
// tensor-core GEMMs over all sequences and heads (attend_u_kernel before
// the token pass, attend_o_kernel after it), so each dictionary is read
// once per layer rather than once per (sequence, KV head); binary32
// dictionaries keep the fused kernel.
#include <type_traits>

#include "fadkv_internal.cuh"

namespace fadkv {
namespace {

constexpr int kAttThreads = 512;
constexpr int kAttWarps = kAttThreads / 32;
constexpr uint32_t kIdMask = (1u << FADKV_PACK_ID_BITS) - 1u;

__device__ __forceinline__ uint32_t pack_word(float c, int id, int N)
{
    if (id < 0 || id >= N || !(c != 0.f) || !isfinite(c)) return 0u;
    uint32_t u = __float_as_uint(c);
    if ((u & 0x7f800000u) == 0u) return (uint32_t)id;          // below 2^-126: no coefficient
    u += 0x0fffu + ((u >> 13) & 1u);                          // round to nearest even at bit 13
    if ((u & 0x7f800000u) == 0x7f800000u) u = (u & 0x80000000u) | 0x7f7fe000u;   // saturate
    return (u & 0xffffe000u) | (uint32_t)id;
}

__device__ __forceinline__ float word_coef(uint32_t w) { return __uint_as_float(w & 0xffffe000u); }

__global__ void __launch_bounds__(256)
store_codes_kernel(StoreArgs a)
{
    const int W = a.s + 1;
    const long long total = (long long)a.G * a.B * a.H * W;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int k = (int)(i % W);
    const long long gv = i / W;                    // (g, b, h) flattened: v = b H + h
    const int h = (int)(gv % a.H);
    const int b = (int)((gv / a.H) % a.B);
    const int g = (int)(gv / ((long long)a.H * a.B));
    const int pos = a.pos[b];
    if (pos < 0 || pos >= a.Tmax) return;
    uint32_t w = 0u;
    if (k < a.s) {
        w = pack_word(a.coef[gv * a.s + k], a.idx[gv * a.s + k], a.N);
    } else if (a.repl_id) {
        w = pack_word(a.repl_coef[gv], a.repl_id[gv], a.N);
    }
    a.cache[((((size_t)g * a.B + b) * a.H + h) * a.Tmax + pos) * W + k] = w;
}

// ---------------------------------------------------------------------------
// attention
// ---------------------------------------------------------------------------

template <typename T, int D> struct Rows;
template <int D> struct Rows<__half, D> {
    // EL (4 or 8) consecutive elements of a row as floats
    template <int EL>
    static __device__ __forceinline__ void load(const __half* p, float (&o)[EL])
    {
        if constexpr (EL == 8) {
            load8(p, o);
        } else {
            const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&q.x));
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&q.y));
            o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
        }
    }
    // 8 consecutive elements of a row as floats
    static __device__ __forceinline__ void load8(const __half* p, float (&o)[8])
    {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
        const __half2* h = reinterpret_cast<const __half2*>(&q);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(h[i]);
            o[2 * i] = f.x;
            o[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ float2 load2(const __half* p)
    {
        return __half22float2(*reinterpret_cast<const __half2*>(p));
    }
};
template <int D> struct Rows<float, D> {
    template <int EL>
    static __device__ __forceinline__ void load(const float* p, float (&o)[EL])
    {
        if constexpr (EL == 8) {
            load8(p, o);
        } else {
            const float4 a = __ldg(reinterpret_cast<const float4*>(p));
            o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
        }
    }
    static __device__ __forceinline__ void load8(const float* p, float (&o)[8])
    {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p));
        const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
        o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
    }
    static __device__ __forceinline__ float2 load2(const float* p)
    {
        return *reinterpret_cast<const float2*>(p);
    }
};

// Block-wide maximum / sum of HP values per thread at once (one barrier
// pair); `red` holds kAttWarps * HP floats.
template <int HP>
__device__ __forceinline__ void block_max_n(float (&v)[HP], float* red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int h = 0; h < HP; ++h)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v[h] = fmaxf(v[h], __shfl_xor_sync(0xffffffffu, v[h], o));
    __syncthreads();
    if (lane == 0)
#pragma unroll
        for (int h = 0; h < HP; ++h) red[warp * HP + h] = v[h];
    __syncthreads();
#pragma unroll
    for (int h = 0; h < HP; ++h) {
        float m = red[h];
#pragma unroll
        for (int w = 1; w < kAttWarps; ++w) m = fmaxf(m, red[w * HP + h]);
        v[h] = m;
    }
}

template <int HP>
__device__ __forceinline__ void block_sum_n(float (&v)[HP], float* red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int h = 0; h < HP; ++h)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v[h] += __shfl_xor_sync(0xffffffffu, v[h], o);
    __syncthreads();
    if (lane == 0)
#pragma unroll
        for (int h = 0; h < HP; ++h) red[warp * HP + h] = v[h];
    __syncthreads();
#pragma unroll
    for (int h = 0; h < HP; ++h) {
        float m = 0.f;
#pragma unroll
        for (int w = 0; w < kAttWarps; ++w) m += red[w * HP + h];
        v[h] = m;
    }
}

// Tokens per thread per softmax chunk: a thread holds every word of its
// tokens in registers before using them (WM words per token at most).
template <int WM> __host__ __device__ constexpr int tokens_per_thread() { return WM <= 9 ? 2 : 1; }

template <typename T, int D, int HP, int WM, bool FUSED>
__global__ void __launch_bounds__(kAttThreads, 2)
attend_kernel(AttendArgs a)
{
    constexpr int TPT = tokens_per_thread<WM>();
    constexpr int CH = TPT * kAttThreads;           // tokens per chunk
    extern __shared__ __align__(16) float sm[];
    const int N = a.N, W = a.s + 1, grp = a.Hq / a.Hkv;
    const int l = blockIdx.y;
    const int b = blockIdx.x / a.Hkv, hk = blockIdx.x % a.Hkv;
    float* u = sm;                                  // [HP][N]
    float* w = u + (size_t)HP * N;                  // [HP][N]
    float* qs = w + (size_t)HP * N;                 // [HP][D]
    float* part = qs + HP * D;                      // [atom groups][HP][D] partial outputs
    __shared__ float red[kAttWarps * HP];
    __shared__ float fac_s[HP];

    const T* Dk = (const T*)a.dict_k + (size_t)l * a.dict_stride;
    const T* Dv = (const T*)a.dict_v + (size_t)l * a.dict_stride;
    const size_t cbase = (size_t)l * a.cache_stride + ((size_t)b * a.Hkv + hk) * a.Tmax * W;
    const uint32_t* ck = a.cache_k + cbase;
    const uint32_t* cv = a.cache_v + cbase;
    int T_len = a.lengths[b];
    T_len = T_len < 0 ? 0 : (T_len > a.Tmax ? a.Tmax : T_len);
    const int tid = threadIdx.x;

    for (int h0 = 0; h0 < grp; h0 += HP) {
        const int hn = min(HP, grp - h0);
        const float* q = a.q + (((size_t)l * a.B + b) * a.Hq + hk * grp + h0) * D;
        float* out = a.out + (((size_t)l * a.B + b) * a.Hq + hk * grp + h0) * D;
        for (int i = tid; i < HP * D; i += kAttThreads) qs[i] = (i / D < hn) ? q[i] : 0.f;
        __syncthreads();

        if constexpr (!FUSED) {
            // 1'. u from the per-layer GEMM's output U (scale already applied)
            const size_t row0 = (size_t)l * a.B * a.Hq + (size_t)b * a.Hq + hk * grp + h0;
            for (int i = tid; i < HP * N; i += kAttThreads) {
                const int h = i / N, j = i % N;
                u[i] = h < hn ? __ldg(a.U + (row0 + h) * a.Npad + j) : 0.f;
            }
            for (int i = tid; i < HP * N; i += kAttThreads) w[i] = 0.f;
        } else
        // 1. u = scale D_K q: half-warps read whole rows (coalesced), every
        //    lane takes D/16 consecutive elements against its slice of q held
        //    in registers, and the half-warp sums by shuffles
        {
            constexpr int EL = D / 16;                  // elements per lane
            const int lane = tid & 31, hl = lane & 15, half = lane >> 4;
            float qr[HP][EL];
#pragma unroll
            for (int h = 0; h < HP; ++h)
#pragma unroll
                for (int e = 0; e < EL; ++e) qr[h][e] = qs[h * D + hl * EL + e] * a.scale;
            for (int j0 = (tid >> 5) * 2; j0 < N; j0 += kAttWarps * 2) {
                const int j = j0 + half;
                float r[EL];
                if (j < N) {
                    Rows<T, D>::template load<EL>(Dk + (size_t)j * D + hl * EL, r);
                } else {
#pragma unroll
                    for (int e = 0; e < EL; ++e) r[e] = 0.f;
                }
                float acc[HP];
#pragma unroll
                for (int h = 0; h < HP; ++h) {
                    acc[h] = 0.f;
#pragma unroll
                    for (int e = 0; e < EL; ++e) acc[h] = fmaf(r[e], qr[h][e], acc[h]);
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1) acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], o);
                }
                if (hl < HP && j < N) {
                    float mine = acc[0];
#pragma unroll
                    for (int h = 1; h < HP; ++h)
                        if (hl == h) mine = acc[h];
                    u[(size_t)hl * N + j] = mine;
                }
            }
            for (int i = tid; i < HP * N; i += kAttThreads) w[i] = 0.f;
        }
        __syncthreads();

        // 2. tokens, chunk by chunk, with the running maximum and sums; a
        //    thread's tokens of a chunk are c0 + tid + k * kAttThreads
        float M[HP], psum[HP];
#pragma unroll
        for (int h = 0; h < HP; ++h) {
            M[h] = -INFINITY;
            psum[h] = 0.f;
        }
        for (int c0 = 0; c0 < T_len; c0 += CH) {
            uint32_t wd[TPT][WM];
#pragma unroll
            for (int k = 0; k < TPT; ++k) {
                const int t = c0 + tid + k * kAttThreads;
                const uint32_t* src = ck + (size_t)t * W;
#pragma unroll
                for (int i = 0; i < WM; ++i) wd[k][i] = (t < T_len && i < W) ? __ldg(src + i) : 0u;
            }
            float sc[TPT][HP], mx[HP];
#pragma unroll
            for (int h = 0; h < HP; ++h) mx[h] = -INFINITY;
#pragma unroll
            for (int k = 0; k < TPT; ++k) {
#pragma unroll
                for (int h = 0; h < HP; ++h) sc[k][h] = 0.f;
#pragma unroll
                for (int i = 0; i < WM; ++i) {
                    const float c = word_coef(wd[k][i]);
                    const uint32_t j = min(wd[k][i] & kIdMask, (uint32_t)(N - 1));
#pragma unroll
                    for (int h = 0; h < HP; ++h) sc[k][h] = fmaf(c, u[(size_t)h * N + j], sc[k][h]);
                }
                if (c0 + tid + k * kAttThreads < T_len)
#pragma unroll
                    for (int h = 0; h < HP; ++h) mx[h] = fmaxf(mx[h], sc[k][h]);
            }
            // the value words of the same tokens, loaded while the maximum is formed
#pragma unroll
            for (int k = 0; k < TPT; ++k) {
                const int t = c0 + tid + k * kAttThreads;
                const uint32_t* src = cv + (size_t)t * W;
#pragma unroll
                for (int i = 0; i < WM; ++i) wd[k][i] = (t < T_len && i < W) ? __ldg(src + i) : 0u;
            }
            block_max_n<HP>(mx, red);
            // rescale w and the partial sums where the running maximum grew
            bool grew = false;
#pragma unroll
            for (int h = 0; h < HP; ++h) {
                const float Mn = fmaxf(M[h], mx[h]);
                const bool g = Mn > M[h] && M[h] > -INFINITY;
                const float f = g ? __expf(M[h] - Mn) : 1.f;
                grew |= g;
                psum[h] *= f;
                if (tid == 0) fac_s[h] = f;
                M[h] = Mn;
            }
            if (grew) {
                __syncthreads();
                for (int i = tid; i < HP * N; i += kAttThreads) w[i] *= fac_s[i / N];
                __syncthreads();
            }
#pragma unroll
            for (int k = 0; k < TPT; ++k) {
                if (c0 + tid + k * kAttThreads >= T_len) continue;
                float p[HP];
#pragma unroll
                for (int h = 0; h < HP; ++h) {
                    p[h] = __expf(sc[k][h] - M[h]);
                    psum[h] += p[h];
                }
#pragma unroll
                for (int i = 0; i < WM; ++i) {
                    const float c = word_coef(wd[k][i]);
                    if (c == 0.f) continue;
                    const uint32_t j = min(wd[k][i] & kIdMask, (uint32_t)(N - 1));
#pragma unroll
                    for (int h = 0; h < HP; ++h) atomicAdd(&w[(size_t)h * N + j], p[h] * c);
                }
            }
        }
        block_sum_n<HP>(psum, red);
        if (tid < HP) fac_s[tid] = 0.f;
#pragma unroll
        for (int h = 0; h < HP; ++h)
            if (tid == 0) fac_s[h] = psum[h];           // the sums, read back below
        __syncthreads();

        if constexpr (!FUSED) {
            // 3'. hand w / S to the second GEMM as two binary16 terms, scaled
            //     per row by a power of two so the largest lands in [2^14, 2^15)
            float mw[HP];
#pragma unroll
            for (int h = 0; h < HP; ++h) mw[h] = 0.f;
            for (int i = tid; i < HP * N; i += kAttThreads) {
                const float v = fabsf(w[i]);
#pragma unroll
                for (int h = 0; h < HP; ++h)
                    if (i / N == h) mw[h] = fmaxf(mw[h], v);
            }
            block_max_n<HP>(mw, red);
            const int Np = a.Npad;
            const size_t row0 = (size_t)l * a.B * a.Hq + (size_t)b * a.Hq + hk * grp + h0;
            for (int h = 0; h < hn; ++h) {
                const float S = fac_s[h];
                const float m = S > 0.f ? mw[h] / S : 0.f;
                const int e = m > 0.f ? 14 - ilogbf(m) : 0;
                const int ec = e > 126 ? 126 : (e < -126 ? -126 : e);
                const float sc = __int_as_float((127 + ec) << 23);     // 2^ec, exact
                const float f = S > 0.f ? sc / S : 0.f;
                __half2* hi = reinterpret_cast<__half2*>(a.Whi + (row0 + h) * Np);
                __half2* lo = reinterpret_cast<__half2*>(a.Wlo + (row0 + h) * Np);
                for (int j2 = tid; j2 < Np / 2; j2 += kAttThreads) {
                    const int j = 2 * j2;
                    const float v0 = j < N ? w[(size_t)h * N + j] * f : 0.f;
                    const float v1 = j + 1 < N ? w[(size_t)h * N + j + 1] * f : 0.f;
                    const __half2 h2 = __floats2half2_rn(v0, v1);
                    hi[j2] = h2;
                    lo[j2] = __floats2half2_rn(v0 - __low2float(h2), v1 - __high2float(h2));
                }
                if (tid == 0) a.wunscale[row0 + h] = (S > 0.f && m > 0.f) ? 1.f / sc : 0.f;
            }
            __syncthreads();
            continue;
        }
        // 3. o = D_V^T w / S: thread = (atom group, column pair)
        constexpr int CP = D / 2;                       // column pairs
        constexpr int AG = kAttThreads / CP;            // atom groups
        const int cp = tid % CP, ag = tid / CP;
        float o[HP][2];
#pragma unroll
        for (int h = 0; h < HP; ++h) o[h][0] = o[h][1] = 0.f;
#pragma unroll 8
        for (int j = ag; j < N; j += AG) {
            const float2 v = Rows<T, D>::load2(Dv + (size_t)j * D + 2 * cp);
#pragma unroll
            for (int h = 0; h < HP; ++h) {
                const float wj = w[(size_t)h * N + j];
                o[h][0] = fmaf(wj, v.x, o[h][0]);
                o[h][1] = fmaf(wj, v.y, o[h][1]);
            }
        }
#pragma unroll
        for (int h = 0; h < HP; ++h) {
            part[((size_t)ag * HP + h) * D + 2 * cp] = o[h][0];
            part[((size_t)ag * HP + h) * D + 2 * cp + 1] = o[h][1];
        }
        __syncthreads();
        for (int i = tid; i < hn * D; i += kAttThreads) {
            const int h = i / D;
            float acc = 0.f;
            for (int g2 = 0; g2 < AG; ++g2) acc += part[((size_t)g2 * HP + h) * D + (i % D)];
            const float S = fac_s[h];
            out[i] = S > 0.f ? acc / S : 0.f;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// binary16 dictionaries: the two dictionary products as per-layer GEMMs
// (mma.sync m16n8k16 from shared-memory tiles, binary16 operands, FP32
// sums), so a layer's dictionaries are read once per tile of query rows, not
// once per (sequence, KV head):
//   U = scale Q D_K^T   [B Hq][N]   before the token pass,
//   O = W D_V           [B Hq][d]   after it (W = the token pass's w / S).
// The FP32 operands (queries, w) enter as two binary16 terms, hi + lo, after
// a per-row power-of-two scale that puts the row's largest entry in
// [2^14, 2^15): about 22 significant bits, no overflow.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void hmma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// 2^k for the row maximum m: k = 14 - floor(log2 m), clamped to binary32's
// normal exponents; 1 for m = 0.
__device__ __forceinline__ float row_scale(float m)
{
    const int e = m > 0.f ? 14 - ilogbf(m) : 0;
    const int ec = e > 126 ? 126 : (e < -126 ? -126 : e);
    return __int_as_float((127 + ec) << 23);
}

// Shared-memory fragments: four 8x8 binary16 matrices (row addresses given by
// lanes 8j..8j+7 for matrix j); .trans delivers them transposed.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ uint32_t saddr(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}
// 16 bytes global -> shared, asynchronous; zero-filled when `valid` is false
// (no byte is read then).
__device__ __forceinline__ void cp16(uint32_t dst, const void* src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// U: a CTA takes 64 query rows x 128 atoms of one layer.  The rows enter
// shared memory as two binary16 terms after their power-of-two scale, the
// atoms as stored (rows padded by 16 bytes, so the eight rows an ldmatrix
// reads sit in different banks); 8 warps, 2 (rows) x 4 (atoms), 32 x 32
// outputs each, every fragment from shared memory.
constexpr int kUBM = 64, kUBN = 128, kUThreads = 256;

template <int D>
struct USmem {
    static constexpr int LD = D + 8;
    __half qh[kUBM][LD], ql[kUBM][LD], dk[kUBN][LD];
    float rs[kUBM];
};

template <int D>
__global__ void __launch_bounds__(kUThreads)
attend_u_kernel(AttendArgs a)
{
    extern __shared__ __align__(16) unsigned char u_raw[];
    USmem<D>& sm = *reinterpret_cast<USmem<D>*>(u_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int M = a.B * a.Hq, N = a.N, l = blockIdx.z;
    const int row0 = blockIdx.y * kUBM, atom0 = blockIdx.x * kUBN;
    const float* Q = a.q + (size_t)l * M * D;
    const __half* Dk = (const __half*)a.dict_k + (size_t)l * a.dict_stride;

    // the atom tile (zeros past N) is on its way while the rows are scaled
    for (int i = tid; i < kUBN * (D / 8); i += kUThreads) {
        const int r = i / (D / 8), c = (i % (D / 8)) * 8;
        const bool ok = atom0 + r < N;
        cp16(saddr(&sm.dk[r][c]), Dk + (size_t)(ok ? atom0 + r : 0) * D + c, ok);
    }
    cp_commit();
    // per-row scale: four lanes on a row
    {
        const int r = tid >> 2, part = tid & 3;
        float mx = 0.f;
        if (row0 + r < M) {
            const float4* qr = reinterpret_cast<const float4*>(Q + (size_t)(row0 + r) * D + part * (D / 4));
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
                const float4 v = __ldg(qr + i);
                mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
            }
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        if (part == 0) sm.rs[r] = row_scale(mx);
    }
    __syncthreads();
    for (int i = tid; i < kUBM * (D / 2); i += kUThreads) {
        const int r = i / (D / 2), c = (i % (D / 2)) * 2;
        float2 v = make_float2(0.f, 0.f);
        if (row0 + r < M) v = __ldg(reinterpret_cast<const float2*>(Q + (size_t)(row0 + r) * D + c));
        const float sc = sm.rs[r];
        v.x *= sc;
        v.y *= sc;
        const __half2 h = __floats2half2_rn(v.x, v.y);
        *reinterpret_cast<__half2*>(&sm.qh[r][c]) = h;
        *reinterpret_cast<__half2*>(&sm.ql[r][c]) = __floats2half2_rn(v.x - __low2float(h), v.y - __high2float(h));
    }
    cp_wait<0>();
    __syncthreads();

    const int wm = warp >> 2, wn = warp & 3;
    float acc[2][4][4];
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) acc[mi][ni][0] = acc[mi][ni][1] = acc[mi][ni][2] = acc[mi][ni][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D; kk += 16) {
        uint32_t ah[2][4], al[2][4], b[4][2];
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
            const int r = wm * 32 + mi * 16 + (lane & 15), c = kk + (lane >> 4) * 8;
            ldsm_x4(ah[mi], saddr(&sm.qh[r][c]));
            ldsm_x4(al[mi], saddr(&sm.ql[r][c]));
        }
#pragma unroll
        for (int ni = 0; ni < 4; ni += 2) {
            const int n = wn * 32 + ni * 8 + (lane & 7) + ((lane >> 4) << 3), c = kk + ((lane >> 3) & 1) * 8;
            uint32_t t[4];
            ldsm_x4(t, saddr(&sm.dk[n][c]));
            b[ni][0] = t[0];
            b[ni][1] = t[1];
            b[ni + 1][0] = t[2];
            b[ni + 1][1] = t[3];
        }
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                hmma16816(acc[mi][ni], ah[mi], b[ni][0], b[ni][1]);
                hmma16816(acc[mi][ni], al[mi], b[ni][0], b[ni][1]);
            }
    }
    float* U = a.U + (size_t)l * M * a.Npad;
    const int g8 = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int rl = wm * 32 + mi * 16 + g8 + hr * 8, row = row0 + rl;
            if (row >= M) continue;
            const float f = a.scale / sm.rs[rl];
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int col = atom0 + wn * 32 + ni * 8 + 2 * t4;
                const float v0 = acc[mi][ni][2 * hr] * f, v1 = acc[mi][ni][2 * hr + 1] * f;
                float* dst = U + (size_t)row * a.Npad + col;
                if (col + 1 < N)
                    *reinterpret_cast<float2*>(dst) = make_float2(v0, v1);
                else if (col < N)
                    *dst = v0;
            }
        }
}

// O: a CTA takes 32 rows of W and all D columns of one layer and runs over
// the atoms in chunks of 64, two chunks in flight (cp.async): W's two
// binary16 terms and D_V's rows in shared memory, D_V's fragments by
// transposing ldmatrix; 4 warps, each the 32 rows x D/4 columns.
constexpr int kOBM = 32, kOBK = 64, kOThreads = 128;

template <int D>
struct OSmem {
    static constexpr int LDW = kOBK + 8, LDV = D + 8;
    __half wh[2][kOBM][LDW], wl[2][kOBM][LDW], dv[2][kOBK][LDV];
};

template <int D>
__global__ void __launch_bounds__(kOThreads)
attend_o_kernel(AttendArgs a)
{
    constexpr int NT = D / 32;                          // n8 tiles per warp
    extern __shared__ __align__(16) unsigned char o_raw[];
    OSmem<D>& sm = *reinterpret_cast<OSmem<D>*>(o_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int M = a.B * a.Hq, N = a.N, Np = a.Npad, l = blockIdx.y;
    const int row0 = blockIdx.x * kOBM;
    const __half* Dv = (const __half*)a.dict_v + (size_t)l * a.dict_stride;
    const __half* Whi = a.Whi + (size_t)l * M * Np;
    const __half* Wlo = a.Wlo + (size_t)l * M * Np;
    const int nchunks = (Np + kOBK - 1) / kOBK;

    auto load = [&](int ch, int buf) {
        const int k0 = ch * kOBK;
        for (int i = tid; i < kOBM * (kOBK / 8); i += kOThreads) {
            const int r = i / (kOBK / 8), c = (i % (kOBK / 8)) * 8;
            const bool ok = row0 + r < M && k0 + c < Np;
            const size_t off = ok ? (size_t)(row0 + r) * Np + k0 + c : 0;
            cp16(saddr(&sm.wh[buf][r][c]), Whi + off, ok);
            cp16(saddr(&sm.wl[buf][r][c]), Wlo + off, ok);
        }
        for (int i = tid; i < kOBK * (D / 8); i += kOThreads) {
            const int r = i / (D / 8), c = (i % (D / 8)) * 8;
            const bool ok = k0 + r < N;
            cp16(saddr(&sm.dv[buf][r][c]), Dv + (size_t)(ok ? k0 + r : 0) * D + c, ok);
        }
        cp_commit();
    };

    float acc[2][NT][4];
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < NT; ++ni) acc[mi][ni][0] = acc[mi][ni][1] = acc[mi][ni][2] = acc[mi][ni][3] = 0.f;
    load(0, 0);
    for (int ch = 0; ch < nchunks; ++ch) {
        const int buf = ch & 1;
        if (ch + 1 < nchunks) {
            load(ch + 1, buf ^ 1);
            cp_wait<1>();
        } else {
            cp_wait<0>();
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kOBK; kk += 16) {
            uint32_t ah[2][4], al[2][4], b[NT][2];
#pragma unroll
            for (int mi = 0; mi < 2; ++mi) {
                const int r = mi * 16 + (lane & 15), c = kk + (lane >> 4) * 8;
                ldsm_x4(ah[mi], saddr(&sm.wh[buf][r][c]));
                ldsm_x4(al[mi], saddr(&sm.wl[buf][r][c]));
            }
#pragma unroll
            for (int ni = 0; ni < NT; ni += 2) {
                // matrices: (atoms kk..+7, cols n0..+7), (kk+8.., n0..), (kk.., n0+8..), (kk+8.., n0+8..)
                const int k = kk + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int n = warp * (D / 4) + ni * 8 + (lane >> 4) * 8;
                uint32_t t[4];
                ldsm_x4_trans(t, saddr(&sm.dv[buf][k][n]));
                b[ni][0] = t[0];
                b[ni][1] = t[1];
                b[ni + 1][0] = t[2];
                b[ni + 1][1] = t[3];
            }
#pragma unroll
            for (int mi = 0; mi < 2; ++mi)
#pragma unroll
                for (int ni = 0; ni < NT; ++ni) {
                    hmma16816(acc[mi][ni], ah[mi], b[ni][0], b[ni][1]);
                    hmma16816(acc[mi][ni], al[mi], b[ni][0], b[ni][1]);
                }
        }
        __syncthreads();                                // the buffer is loaded again two chunks on
    }
    const int g8 = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int row = row0 + mi * 16 + g8 + hr * 8;
            if (row >= M) continue;
            const size_t orow = (size_t)l * M + row;
            const float f = a.wunscale[orow];
#pragma unroll
            for (int ni = 0; ni < NT; ++ni) {
                const int col = warp * (D / 4) + ni * 8 + 2 * t4;
                *reinterpret_cast<float2*>(a.out + orow * D + col) =
                    make_float2(acc[mi][ni][2 * hr] * f, acc[mi][ni][2 * hr + 1] * f);
            }
        }
}

template <int D, int HP>
size_t attend_smem(int N)
{
    const int AG = kAttThreads / (D / 2);
    return sizeof(float) * ((size_t)2 * HP * N + (size_t)HP * D + (size_t)AG * HP * D);
}

template <typename T, int D, int HP, int WM>
cudaError_t launch_hpw(const AttendArgs& a, cudaStream_t st)
{
    const size_t smem = attend_smem<D, HP>(a.N);
    auto k = attend_kernel<T, D, HP, WM, !std::is_same<T, __half>::value>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<dim3(a.B * a.Hkv, a.L), kAttThreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <typename T, int D, int HP>
cudaError_t launch_hp(const AttendArgs& a, cudaStream_t st)
{
    const int W = a.s + 1;
    if (W <= 9) return launch_hpw<T, D, HP, 9>(a, st);
    if (W <= 17) return launch_hpw<T, D, HP, 17>(a, st);
    return launch_hpw<T, D, HP, 33>(a, st);
}

constexpr size_t kAttSmemMax = 200 * 1024;

template <typename T, int D>
cudaError_t launch_d(const AttendArgs& a, cudaStream_t st)
{
    const int grp = a.Hq / a.Hkv;
    if (grp >= 4 && attend_smem<D, 4>(a.N) <= kAttSmemMax) return launch_hp<T, D, 4>(a, st);
    if (grp >= 3 && attend_smem<D, 3>(a.N) <= kAttSmemMax) return launch_hp<T, D, 3>(a, st);
    if (grp >= 2 && attend_smem<D, 2>(a.N) <= kAttSmemMax) return launch_hp<T, D, 2>(a, st);
    return launch_hp<T, D, 1>(a, st);
}

template <int D>
cudaError_t launch_u(const AttendArgs& a, cudaStream_t st)
{
    const int M = a.B * a.Hq;
    const size_t smem = sizeof(USmem<D>);
    cudaError_t e = cudaFuncSetAttribute(attend_u_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((a.N + kUBN - 1) / kUBN), (unsigned)((M + kUBM - 1) / kUBM), (unsigned)a.L);
    attend_u_kernel<D><<<grid, kUThreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_o(const AttendArgs& a, cudaStream_t st)
{
    const int M = a.B * a.Hq;
    const size_t smem = sizeof(OSmem<D>);
    cudaError_t e = cudaFuncSetAttribute(attend_o_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attend_o_kernel<D><<<dim3((unsigned)((M + kOBM - 1) / kOBM), (unsigned)a.L), kOThreads, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

bool attend_supported(int d, int N, int s)
{
    if (d != 64 && d != 128) return false;
    if (N < 1 || N > (1 << FADKV_PACK_ID_BITS) || s < 0 || s > FADKV_MAX_S) return false;
    return d == 128 ? attend_smem<128, 1>(N) <= kAttSmemMax : attend_smem<64, 1>(N) <= kAttSmemMax;
}

cudaError_t launch_store_codes(const StoreArgs& a, cudaStream_t st)
{
    const long long total = (long long)a.G * a.B * a.H * (a.s + 1);
    if (total <= 0) return cudaSuccess;
    store_codes_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(a);
    return cudaGetLastError();
}

size_t attend_workspace_bytes(int L, int B, int Hq, int N, int dtype)
{
    if (dtype != FADKV_F16) return 0;
    const size_t rows = (size_t)L * B * Hq, Np = (size_t)attend_npad(N);
    const auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    return up(rows * Np * sizeof(float)) + 2 * up(rows * Np * sizeof(__half)) + up(rows * sizeof(float));
}

void attend_bind_workspace(AttendArgs& a, void* ws)
{
    const size_t rows = (size_t)a.L * a.B * a.Hq, Np = (size_t)a.Npad;
    const auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    unsigned char* p = (unsigned char*)ws;
    a.U = (float*)p;
    p += up(rows * Np * sizeof(float));
    a.Whi = (__half*)p;
    p += up(rows * Np * sizeof(__half));
    a.Wlo = (__half*)p;
    p += up(rows * Np * sizeof(__half));
    a.wunscale = (float*)p;
}

cudaError_t launch_attend(const AttendArgs& a, cudaStream_t st)
{
    if (a.L <= 0 || a.B <= 0) return cudaSuccess;
    if (a.dtype != FADKV_F16) return a.d == 128 ? launch_d<float, 128>(a, st) : launch_d<float, 64>(a, st);
    cudaError_t e = a.d == 128 ? launch_u<128>(a, st) : launch_u<64>(a, st);
    if (e != cudaSuccess) return e;
    e = a.d == 128 ? launch_d<__half, 128>(a, st) : launch_d<__half, 64>(a, st);
    if (e != cudaSuccess) return e;
    return a.d == 128 ? launch_o<128>(a, st) : launch_o<64>(a, st);
}

}  // namespace fadkv
