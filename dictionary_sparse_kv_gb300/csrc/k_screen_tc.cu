// Screening on the 5th-generation tensor cores with a fused candidate filter.
//
// "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding",
// abstract: screening-based sparse coding correlates each incoming vector
// with every atom, then a one-shot Top-n selection keeps a small pool.
//
// Per CTA: one dictionary g, a tile of 128 vectors (the MMA's M = TMEM
// lanes) and a slice of the atoms, streamed in chunks of 128 atoms (N = 128
// TMEM columns).  S[v][j] = sum_t X[v][t] D[j][t] is a K-major x K-major
// product: A = the vector tile, B = the atom chunk, both binary16 in shared
// memory with the 128-byte swizzle written by TMA; fp32 accumulation in TMEM,
// two accumulator buffers so the epilogue of chunk c overlaps the MMAs of
// chunk c+1.  Scores never reach HBM: the epilogue thread of vector v keeps
// atom j only if |S[v][j]| >= tau_v and appends the 64-bit key
// (bits(|S|) << 32) | (0xffffffff - j) to its own region of the vector's
// candidate list -- one region per (atom slice, accumulator buffer), so
// appends are plain stores, with no atomics and nothing to wait for; the
// exact Top-n (ties to the lower index) is taken from the regions by the
// consumer.  tau_v = alpha * ||x_v|| / sqrt(d), with alpha set on the host so
// that an atom uncorrelated with x_v passes with probability ~1.5n/N; lists
// that end shorter than n or overflow a region are redone exactly by the
// consumer.
//
// Warp roles (384 threads): warp 0 issues TMA loads, warp 1 issues MMAs
// (one thread), warp 2 owns the TMEM allocation, warps 4..11 are the
// epilogue (warp 4+e reads TMEM lanes 32(e%4).. and handles the chunks
// whose accumulator buffer is e/4).  About 97 KB of shared memory and 256
// TMEM columns per CTA: two CTAs share an SM.  Every wait is bounded by a
// wall-clock limit; on expiry the CTA sets FADKV_DEV_TIMEOUT in the status
// word, drains its own copies and MMAs (bounded), frees TMEM and returns.
#include "tc_common.cuh"

namespace fadkv {
namespace {

constexpr int kThreads = 384;
constexpr int kTileV = 128;        // vectors per CTA (MMA M)
constexpr int kChunk = 128;        // atoms per MMA chunk (MMA N)
constexpr int kStages = 2;         // B (atom chunk) pipeline depth
constexpr int kTmemCols = 2 * kChunk;

using namespace tc;

// Instruction descriptor: M = 128 vectors, N = 128 atoms.
constexpr uint32_t kIdesc = idesc_f16(kTileV, kChunk);

__device__ __forceinline__ void mma_f16(uint32_t dtmem, uint64_t a, uint64_t b, uint32_t acc)
{
    mma_ss(dtmem, a, b, kIdesc, acc);
}
__device__ __forceinline__ void tc_fence_before() { fence_before(); }
__device__ __forceinline__ void tc_fence_after() { fence_after(); }

template <int D>
struct SmemLayout {
    static constexpr int KH = D / 64;                          // 64-element (128-byte) K halves
    static constexpr int kTileBytes = KH * kChunk * 128;       // one 128-row operand tile
    static constexpr int a_off = 0;
    static constexpr int b_off = kTileBytes;
    static constexpr int bar_off = b_off + kStages * kTileBytes;
    static constexpr int n_bars = 2 * kStages + 4 + 1;
    static constexpr int taddr_off = bar_off + n_bars * 8;
    static constexpr int total = taddr_off + 16;
    static constexpr int alloc = total + 1024;                 // slack for 1024-byte alignment
};

template <int D, bool kDump>
__global__ void __launch_bounds__(kThreads, 2)
screen_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_d,
                 ScreenTCArgs a)
{
    using L = SmemLayout<D>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sA = sbase + L::a_off, sB = sbase + L::b_off;
    const uint32_t bar0 = sbase + L::bar_off;
    auto full_bar = [&](int i) { return bar0 + 8u * i; };
    auto empty_bar = [&](int i) { return bar0 + 8u * (kStages + i); };
    auto tfull_bar = [&](int i) { return bar0 + 8u * (2 * kStages + i); };
    auto tempty_bar = [&](int i) { return bar0 + 8u * (2 * kStages + 2 + i); };
    const uint32_t afull_bar = bar0 + 8u * (2 * kStages + 4);
    uint32_t* taddr_slot = (uint32_t*)(smem + L::taddr_off);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.y;
    const int tile = blockIdx.x / a.slices, slice = blockIdx.x % a.slices;
    const int nchunks_all = a.N / kChunk;
    const int cps = (nchunks_all + a.slices - 1) / a.slices;
    const int c0 = slice * cps;
    const int nch = max(0, min(cps, nchunks_all - c0));
    unsigned long long* status = (unsigned long long*)&a.counters[(size_t)g * kCntFields + kCntStatus];

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(full_bar(i), 1);
            mbar_init(empty_bar(i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull_bar(i), 1);
            mbar_init(tempty_bar(i), 128);
        }
        mbar_init(afull_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(taddr_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *taddr_slot;

    const int row0 = g * a.V + a.v0 + tile * kTileV;   // first row of this tile in x viewed as [G*V][D]
    constexpr uint32_t kTileBytes = (uint32_t)L::kTileBytes;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_x)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_d)) : "memory");
            mbar_expect_tx(afull_bar, kTileBytes);
            for (int h = 0; h < L::KH; ++h) tma_load_2d(sA + h * kChunk * 128, &map_x, h * 64, row0, afull_bar);
            int issued = 0;
            bool ok = true;
            for (int c = 0; c < nch && ok; ++c) {
                const int st = c % kStages;
                const uint32_t ph = (uint32_t)(c / kStages) & 1u;
                ok = mbar_wait(empty_bar(st), ph ^ 1u, status);
                if (!ok) break;
                mbar_expect_tx(full_bar(st), kTileBytes);
                const int arow = g * a.N + (c0 + c) * kChunk;
                for (int h = 0; h < L::KH; ++h)
                    tma_load_2d(sB + st * kTileBytes + h * kChunk * 128, &map_d, h * 64, arow, full_bar(st));
                ++issued;
            }
            // drain: every issued load must have landed before the CTA exits
            mbar_wait(afull_bar, 0, status);
            for (int c = max(0, issued - kStages); c < issued; ++c)
                mbar_wait(full_bar(c % kStages), (uint32_t)(c / kStages) & 1u, status);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            bool ok = mbar_wait(afull_bar, 0, status);
            int issued = 0;
            for (int c = 0; c < nch && ok; ++c) {
                const int st = c % kStages;
                const uint32_t ph = (uint32_t)(c / kStages) & 1u;
                const int buf = c & 1;
                const uint32_t bph = (uint32_t)(c >> 1) & 1u;
                ok = mbar_wait(tempty_bar(buf), bph ^ 1u, status);
                if (!ok) break;
                ok = mbar_wait(full_bar(st), ph, status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t dt = tbase + (uint32_t)(buf * kChunk);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (uint32_t)((kk >> 2) * kChunk * 128 + (kk & 3) * 32);
                    mma_f16(dt, sdesc(sA + koff), sdesc(sB + st * kTileBytes + koff), kk > 0 ? 1u : 0u);
                }
                mma_commit(empty_bar(st));
                mma_commit(tfull_bar(buf));
                ++issued;
            }
            // drain: the last accumulator must be complete before TMEM is freed
            if (issued > 0) mbar_wait(tfull_bar((issued - 1) & 1), (uint32_t)((issued - 1) >> 1) & 1u, status);
        }
    } else if (warp >= 4) {
        // ---------------- epilogue ----------------
        const int e = warp - 4;
        const int q = e & 3;                                // TMEM lane group
        const int hb = e >> 2;                              // accumulator buffer handled
        const int r = q * 32 + lane;                        // TMEM lane = row of the vector tile
        const int vloc = tile * kTileV + r;                 // vector index inside the chunk
        const bool valid = vloc < a.Vc;
        const int region = slice * 2 + hb;
        const int cs = a.cap / (2 * a.slices);              // entries per region
        unsigned long long* list =
            a.cand + ((size_t)g * a.Vc + (valid ? vloc : 0)) * a.cap + (size_t)region * cs;
        uint32_t tau_bits = 0u;
        int cnt = 0;
        bool ok = mbar_wait(afull_bar, 0, status);
        if (ok && !kDump) {
            // ||x||^2 from this row of the swizzled A tile (all 16-byte chunks
            // of the row, whatever their swizzled order)
            float sq = 0.f;
#pragma unroll
            for (int h = 0; h < L::KH; ++h) {
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint4 w = *reinterpret_cast<const uint4*>(
                        smem + L::a_off + h * kChunk * 128 + r * 128 + ((ch ^ (r & 7)) * 16));
                    const __half2* hv = reinterpret_cast<const __half2*>(&w);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = __half22float2(hv[i]);
                        sq = fmaf(f.x, f.x, sq);
                        sq = fmaf(f.y, f.y, sq);
                    }
                }
            }
            // rows past the batch never pass (|S| bits are below 0xffffffff)
            tau_bits = valid ? __float_as_uint(a.alpha * sqrtf(sq * (1.0f / (float)D))) : 0xffffffffu;
        }
        for (int c = hb; c < nch && ok; c += 2) {
            const uint32_t bph = (uint32_t)(c >> 1) & 1u;
            ok = mbar_wait(tfull_bar(hb), bph, status);
            if (!ok) break;
            tc_fence_after();
            const int atom0 = (c0 + c) * kChunk;
#pragma unroll
            for (int qq = 0; qq < kChunk / 32; ++qq) {
                uint32_t v[32];
                tmem_ld32(tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)(hb * kChunk + qq * 32), v);
                if (kDump) {
                    if (valid) {
                        float* out = a.dump + ((size_t)g * a.Vc + vloc) * a.N + atom0 + qq * 32;
#pragma unroll
                        for (int i = 0; i < 32; ++i) out[i] = __uint_as_float(v[i]);
                    }
                } else {
                    const uint32_t lo0 = 0xffffffffu - (uint32_t)(atom0 + qq * 32);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        // branch-free: a predicated store, then the count.  Past
                        // the region's end the last slot is reused: the count
                        // then exceeds the region and the consumer redoes the
                        // vector exactly.
                        const uint32_t mag = v[i] & 0x7fffffffu;
                        unsigned long long* slot = list + min(cnt, cs - 1);
                        asm volatile(
                            "{\n\t.reg .pred p;\n\t"
                            "setp.ge.u32 p, %0, %1;\n\t"
                            "@p st.global.v2.u32 [%2], {%3, %0};\n\t}"
                            ::"r"(mag), "r"(tau_bits), "l"(slot), "r"(lo0 - (uint32_t)i)
                            : "memory");
                        cnt += (mag >= tau_bits) ? 1 : 0;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(tempty_bar(hb));
        }
        if (valid && !kDump)
            a.cand_count[((size_t)g * a.Vc + vloc) * kCountSlots + region] = cnt;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kTmemCols));
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

template <int D, bool kDump>
cudaError_t launch_t(const Shape& sh, const void* atoms, const void* x, int V, const ScreenTCArgs& a, int sms,
                     cudaStream_t st)
{
    CUtensorMap mx, md;
    if (!make_tma_map_f16(&mx, x, (long long)sh.G * V, D, 128) ||
        !make_tma_map_f16(&md, atoms, (long long)sh.G * sh.N, D, 128))
        return cudaErrorInvalidValue;
    auto k = screen_tc_kernel<D, kDump>;
    const int smem = SmemLayout<D>::alloc;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int tiles = (a.Vc + kTileV - 1) / kTileV;
    dim3 grid(tiles * a.slices, sh.G);
    k<<<grid, kThreads, smem, st>>>(mx, md, a);
    return cudaGetLastError();
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tma_encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

bool make_tma_map_f16(CUtensorMap* m, const void* base, long long rows, int d, int box_rows)
{
    auto fn = tma_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int screen_tc_slices(const Shape& sh, int Vc, int sms)
{
    // two CTAs per SM; at least 64 entries per candidate region
    const int tiles = (Vc + kTileV - 1) / kTileV;
    const int nchunks = sh.N / kChunk;
    int s = 2 * sms / (sh.G * tiles);
    const int by_cap = cand_cap(sh.n) / 128;
    if (s > by_cap) s = by_cap;
    if (s > kMaxSlices) s = kMaxSlices;
    if (s > nchunks) s = nchunks;
    if (s < 1) s = 1;
    return s;
}

bool screen_tc_supported(const Shape& sh)
{
    return sh.dtype == FADKV_F16 && (sh.d == 64 || sh.d == 128) && sh.N % kChunk == 0;
}

cudaError_t launch_screen_tc(const Shape& sh, const void* atoms, const void* x, int V, const ScreenTCArgs& a,
                             int sms, cudaStream_t st)
{
    if (a.Vc <= 0) return cudaSuccess;
    const bool dump = a.dump != nullptr;
    if (sh.d == 128)
        return dump ? launch_t<128, true>(sh, atoms, x, V, a, sms, st) : launch_t<128, false>(sh, atoms, x, V, a, sms, st);
    return dump ? launch_t<64, true>(sh, atoms, x, V, a, sms, st) : launch_t<64, false>(sh, atoms, x, V, a, sms, st);
}

}  // namespace fadkv
