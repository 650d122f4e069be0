// Screening on the 5th-generation tensor cores with a fused candidate filter.
//
// "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding",
// abstract: screening-based sparse coding correlates each incoming vector
// with every atom, then a one-shot Top-n selection keeps a small pool.
//
// Work: the (dictionary g, tile of 128 vectors, chunk of 128 atoms) units,
// chunk fastest, split evenly over one persistent CTA per SM: CTA b takes the
// contiguous units [b*T/B, (b+1)*T/B), so every SM streams the same number
// of atom chunks whatever G and the batch are.  A run of units of one
// (g, tile) is a segment; its vector tile is the MMA's A operand (two
// buffers, so the next segment's tile loads under the current one).
//
// S[v][j] = sum_t X[v][t] D[j][t] per unit: A = the vector tile (M = 128 TMEM
// lanes), B = the atom chunk (N = 128 columns), both binary16 K-major with the
// 128-byte swizzle written by TMA; fp32 accumulation in TMEM, two accumulator
// buffers.  Scores never reach HBM.  The epilogue thread of vector v keeps
// atom j if |S[v][j]| >= tau_v, tau_v = alpha * ||x_v|| / sqrt(d) with alpha
// set on the host so that an atom uncorrelated with x_v passes with
// probability ~1.5n/N.  Each kept score becomes a 32-bit packed key (|S|
// exactly, relative to the exponent of tau_v, its sign and the atom's
// column; see ScreenTCArgs) appended to the vector's record of the unit in shared
// memory: one predicated 4-byte store per score.  After each unit the warp
// copies its 32 records out with 16-byte loads and stores, eight lanes on a
// record: the candidate output lands as whole sectors.  A row with more than kRecKeys kept scores in a unit makes
// the consumer redo the vector.
//
// Warp roles (384 threads): warp 0 issues TMA loads, warp 1 issues MMAs (one
// thread), warp 2 owns the TMEM allocation, warps 4..11 are the epilogue
// (warp 4+e reads TMEM lanes 32(e%4).. and handles the units whose
// accumulator buffer is e/4).  Every wait is bounded by a wall-clock limit;
// on expiry the CTA sets FADKV_DEV_TIMEOUT in the status word, drains its own
// copies and MMAs (the producer waits for every atom chunk it issued, the MMA
// issuer for its last commit, each with the full limit), frees TMEM and
// returns.
#include "tc_common.cuh"

namespace fadkv {
namespace {

constexpr int kThreads = 512;
constexpr int kTileV = 128;        // vectors per tile (MMA M)
constexpr int kChunk = 128;        // atoms per chunk (MMA N)
constexpr int kStagesFor(int D) { return D == 64 ? 10 : 5; }  // atom chunk pipeline depth
constexpr int kTmemCols = 512;     // two accumulator buffers (128 columns each), two vector tiles
constexpr int kAcol = 2 * kChunk;  // first TMEM column of the vector tiles
constexpr int kEpiWarps = 8;
// A row's record in shared memory sits in a slot of kRecWords + 4 words
// (144 bytes): consecutive rows start 4 banks apart, so the rows' appends,
// which advance at similar rates, rarely hit the same bank.
constexpr int kSlotWords = kRecWords + 4;
constexpr int kWarpStageWords = 32 * kSlotWords + 32;      // a warp's 32 slots + a guard of 32 words
static_assert(kRecWords >= 32 && kSlotWords - kRecWords <= 32,
              "a row spills at most 32 words past its record: into the next slot or the guard");
static_assert(kSlotWords * 4 % 16 == 0 && kRecBytes % 16 == 0, "records are copied in 16-byte pieces");

using namespace tc;

// Instruction descriptor: M = 128 vectors, N = 128 atoms.
constexpr uint32_t kIdesc = idesc_f16(kTileV, kChunk);

template <int D>
struct SmemLayout {
    static constexpr int kStages = kStagesFor(D);
    static constexpr int KH = D / 64;                          // 64-element (128-byte) K halves
    static constexpr int kTileBytes = KH * kChunk * 128;       // one 128-row operand tile
    static constexpr int b_off = 0;                            // kStages atom chunks
    static constexpr int s_off = b_off + kStages * kTileBytes; // the epilogue warps' records
    static constexpr int bar_off = s_off + kEpiWarps * kWarpStageWords * 4;
    static constexpr int n_bars = 2 * kStages + 8;
    static constexpr int taddr_off = bar_off + n_bars * 8;
    static constexpr int total = taddr_off + 16;
    static constexpr int alloc = total + 1024;                 // slack for 1024-byte alignment
};

// Walks a CTA's units in order without divisions: the unit's chunk c and its
// (dictionary g, tile); pair = g * tiles + tile.
struct UnitCursor {
    int pair, c, g, tile, nch, tiles;
    __device__ __forceinline__ void init(long long u, int nch_, int tiles_)
    {
        nch = nch_;
        tiles = tiles_;
        const long long p = u / nch;
        pair = (int)p;
        c = (int)(u - p * nch);
        g = pair / tiles;
        tile = pair - g * tiles;
    }
    __device__ __forceinline__ void advance(int k)
    {
        c += k;
        while (c >= nch) {
            c -= nch;
            ++pair;
            if (++tile == tiles) {
                tile = 0;
                ++g;
            }
        }
    }
};

template <int D, bool kDump>
__global__ void __launch_bounds__(kThreads, 1)
screen_tc_kernel(const __grid_constant__ CUtensorMap map_d, ScreenTCArgs a)
{
    using L = SmemLayout<D>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sB = sbase + L::b_off;
    const uint32_t bar0 = sbase + L::bar_off;
    auto full_bar = [&](int i) { return bar0 + 8u * i; };
    auto empty_bar = [&](int i) { return bar0 + 8u * (L::kStages + i); };
    auto tfull_bar = [&](int i) { return bar0 + 8u * (2 * L::kStages + i); };
    auto tempty_bar = [&](int i) { return bar0 + 8u * (2 * L::kStages + 2 + i); };
    auto afull_bar = [&](int i) { return bar0 + 8u * (2 * L::kStages + 4 + i); };
    auto aempty_bar = [&](int i) { return bar0 + 8u * (2 * L::kStages + 6 + i); };
    uint32_t* taddr_slot = (uint32_t*)(smem + L::taddr_off);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nch = a.N / kChunk;
    const int tiles = (a.Vc + kTileV - 1) / kTileV;
    const long long T = (long long)a.G * tiles * nch;
    const int B = (int)gridDim.x, b = (int)blockIdx.x;
    const long long u0 = (long long)b * T / B, u1 = (long long)(b + 1) * T / B;
    const int nu = (int)(u1 - u0);
    const int g_first = (int)(u0 / nch / tiles);
    unsigned long long* status = (unsigned long long*)&a.counters[(size_t)g_first * kCntFields + kCntStatus];
    const unsigned long long wait_ns = a.wait_ns ? a.wait_ns : kWaitNs;   // pipeline waits (drains: kWaitNs)

    if (threadIdx.x == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_d)) : "memory");
        for (int i = 0; i < L::kStages; ++i) {
            mbar_init(full_bar(i), 1);
            mbar_init(empty_bar(i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull_bar(i), 1);
            mbar_init(tempty_bar(i), 128);
            mbar_init(afull_bar(i), 128);
            mbar_init(aempty_bar(i), 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_begin();                      // the predecessor's writes (x, atoms) are visible from here
    // The TMEM allocation is published to the MMA and epilogue warps (and
    // warp 2) by a named barrier: the producer starts streaming at once.
    constexpr int kTmemSyncThreads = 32 * (2 + kEpiWarps + 4);
    uint32_t tbase = 0;
    if (warp != 0 && warp != 3) {
        if (warp == 2) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(taddr_slot)),
                         "r"(kTmemCols));
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        }
        fence_before();
        asm volatile("bar.sync 1, %0;" ::"n"(kTmemSyncThreads) : "memory");
        fence_after();
        tbase = *taddr_slot;
    }
    constexpr uint32_t kTileBytes = (uint32_t)L::kTileBytes;

    if (warp == 0) {
        // ---------------- TMA producer (atom chunks) ----------------
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            UnitCursor uc;
            uc.init(u0, nch, tiles);
            for (int i = 0; i < nu && ok; ++i, uc.advance(1)) {
                const int st = i % L::kStages;
                ok = mbar_wait(empty_bar(st), ((uint32_t)(i / L::kStages) & 1u) ^ 1u, status, wait_ns);
                if (!ok) break;
                mbar_expect_tx(full_bar(st), kTileBytes);
                const int arow = uc.g * a.N + uc.c * kChunk;
                for (int h = 0; h < L::KH; ++h)
                    tma_load_2d(sB + st * kTileBytes + h * kChunk * 128, &map_d, h * 64, arow, full_bar(st));
                ++issued;
            }
            // drain: every issued load must have landed before the CTA exits
            for (int i = max(0, issued - L::kStages); i < issued; ++i)
                mbar_wait(full_bar(i % L::kStages), (uint32_t)(i / L::kStages) & 1u, status);
        }
    } else if (warp >= 4 + kEpiWarps) {
        // ---------------- vector tiles into TMEM ----------------
        // Warp 12+q writes rows 32q.. of each segment's tile (binary16 pairs,
        // K-major: column k holds elements 2k, 2k+1) into its TMEM buffer,
        // the MMAs' A operand; rows past the batch are zeros.
        const int q = warp - 4 - kEpiWarps;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        int prev = -1, seg = -1;
        bool ok = true;
        UnitCursor uc;
        uc.init(u0, nch, tiles);
        for (int i = 0; i < nu && ok; ++i, uc.advance(1)) {
            if (uc.pair == prev) continue;
            prev = uc.pair;
            ++seg;
            const int ab = seg & 1;
            // the buffer's previous tile (segment seg-2) must be done with
            if (seg >= 2) ok = mbar_wait(aempty_bar(ab), (uint32_t)((seg >> 1) - 1) & 1u, status, wait_ns);
            if (!ok) break;
            fence_after();
            const int vloc = uc.tile * kTileV + q * 32 + lane;
            const uint4* xr = reinterpret_cast<const uint4*>((const __half*)a.x +
                                                             ((size_t)uc.g * a.V + a.v0 + (vloc < a.Vc ? vloc : 0)) * D);
#pragma unroll
            for (int h = 0; h < D / 32; ++h) {
                uint32_t w[16];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint4 t = vloc < a.Vc ? __ldg(xr + h * 4 + k) : make_uint4(0u, 0u, 0u, 0u);
                    w[4 * k + 0] = t.x;
                    w[4 * k + 1] = t.y;
                    w[4 * k + 2] = t.z;
                    w[4 * k + 3] = t.w;
                }
                tmem_st16(tbase + lane_off + (uint32_t)(kAcol + ab * (D / 2) + h * 16), w);
            }
            tmem_st_wait();
            fence_before();
            mbar_arrive(afull_bar(ab));
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int prev = -1, seg = -1, issued = 0;
            bool ok = true;
            UnitCursor uc;
            uc.init(u0, nch, tiles);
            for (int i = 0; i < nu && ok; ++i, uc.advance(1)) {
                if (uc.pair != prev) {
                    // the previous segment's tile is free once its MMAs complete
                    if (seg >= 0) mma_commit(aempty_bar(seg & 1));
                    prev = uc.pair;
                    ++seg;
                    ok = mbar_wait(afull_bar(seg & 1), (uint32_t)(seg >> 1) & 1u, status, wait_ns);
                    if (!ok) break;
                }
                const int buf = i & 1;
                ok = mbar_wait(tempty_bar(buf), ((uint32_t)(i >> 1) & 1u) ^ 1u, status, wait_ns);
                if (!ok) break;
                const int st = i % L::kStages;
                ok = mbar_wait(full_bar(st), (uint32_t)(i / L::kStages) & 1u, status, wait_ns);
                if (!ok) break;
                fence_after();
                const uint32_t dt = tbase + (uint32_t)(buf * kChunk);
                const uint32_t at = tbase + (uint32_t)(kAcol + (seg & 1) * (D / 2));
                const uint32_t aB = sB + (uint32_t)st * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (uint32_t)((kk >> 2) * kChunk * 128 + (kk & 3) * 32);
                    mma_ts(dt, at + (uint32_t)(kk * 8), sdesc(aB + koff), kIdesc, kk > 0 ? 1u : 0u);
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
        uint32_t* const recs = reinterpret_cast<uint32_t*>(smem + L::s_off) + e * kWarpStageWords;
        uint32_t* const myrec = recs + lane * kSlotWords;    // word 0 header, then the keys
        int cur = -1, g = 0, vloc = 0;
        bool valid = false, ok = true;
        float tau = __int_as_float(0x7fffffff), top = 0.f;
        uint32_t eb = 0, nbase = 0;
        UnitCursor uc;
        uc.init(u0 + hb, nch, tiles);
        for (int i = hb; i < nu && ok; i += 2, uc.advance(2)) {
            const int c = uc.c;
            if (uc.pair != cur) {
                cur = uc.pair;
                g = uc.g;
                vloc = uc.tile * kTileV + r;
                valid = vloc < a.Vc;
                // tau from ||x||^2 (rows past the batch: NaN, never passes)
                tau = __int_as_float(0x7fffffff);
                if (valid && !kDump) {
                    const uint4* xr =
                        reinterpret_cast<const uint4*>((const __half*)a.x + ((size_t)g * a.V + a.v0 + vloc) * D);
                    float sq = 0.f;
#pragma unroll
                    for (int k = 0; k < D / 8; ++k) {
                        const uint4 w = __ldg(xr + k);
                        const __half2* hv = reinterpret_cast<const __half2*>(&w);
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const float2 f = __half22float2(hv[t]);
                            sq = fmaf(f.x, f.x, sq);
                            sq = fmaf(f.y, f.y, sq);
                        }
                    }
                    tau = a.alpha * sqrtf(sq * (1.0f / (float)D));
                }
                // the key window: tau's exponent field, the largest value kept exactly
                const uint32_t base_bits = __float_as_uint(tau) & 0x7f800000u;
                eb = base_bits >> 23;
                nbase = 0u - base_bits;
                top = __uint_as_float(base_bits + kRecValueMask);
            }
            const int buf = i & 1;
            ok = mbar_wait(tfull_bar(buf), (uint32_t)(i >> 1) & 1u, status, wait_ns);
            if (!ok) break;
            fence_after();
            const uint32_t tcol = tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kChunk);
            int k = 1;                                      // next word of this row's record
            int k0 = 0;                                     // keys of atoms c*128 + [0, 64)
            bool ovf = false;
            // one 32-column group: append the packed keys of the kept scores
            auto stage = [&](const uint32_t (&v)[32], int qq) {
                if constexpr (kDump) {
                    if (valid) {
                        float* out = a.dump + ((size_t)g * a.Vc + vloc) * a.N + c * kChunk + qq * 32;
#pragma unroll
                        for (int t = 0; t < 32; ++t) out[t] = __uint_as_float(v[t]);
                    }
                    return;
                } else {
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        const float f = fabsf(__uint_as_float(v[t]));
                        if (f >= tau) {
                            myrec[k] = __float_as_uint(fminf(f, top)) + nbase + ((v[t] >> 31) << kRecSignShift) +
                                       ((uint32_t)((qq & 1) * 32 + t) << 26);
                            ++k;
                        }
                    }
                    // a row may run past its record by at most 32 words (into
                    // the next row's slot, or the warp's guard after row 31):
                    // flagged below
                    ovf |= k > kRecWords;
                    k = min(k, kRecWords);
                    if (qq == 1) k0 = k - 1;
                }
            };
            // TMEM loads double-buffered in registers: group g+1 is in flight
            // while group g is filtered
            static_assert(kChunk == 128, "four 32-column groups per unit");
            uint32_t va[32], vb[32];
            tmem_ld32_async(tcol, va);
            tmem_wait32(va);
            tmem_ld32_async(tcol + 32, vb);
            stage(va, 0);
            tmem_wait32(vb);
            tmem_ld32_async(tcol + 64, va);
            stage(vb, 1);
            tmem_wait32(va);
            tmem_ld32_async(tcol + 96, vb);
            stage(va, 2);
            tmem_wait32(vb);
            // every column of this buffer is in registers: hand it back
            fence_before();
            mbar_arrive(tempty_bar(buf));
            stage(vb, 3);
            if (kDump) continue;
            // a row that ran past its record spilled into the next row's record
            // only (the group clamp bounds the spill to one record): both are
            // flagged
            const int prev_ovf = __shfl_up_sync(0xffffffffu, ovf ? 1 : 0, 1);   // every lane takes part
            const bool over = ovf || (lane > 0 && prev_ovf != 0);
            const int cnt = k - 1;
            myrec[0] = rec_header(over, eb, k0, cnt);
            __syncwarp();
            // copy the 32 records out: eight lanes on a record (16 bytes each),
            // four records at a time, only the pieces holding words
            const int part = lane & 7, rsub = lane >> 3;
            const int pieces = valid ? (cnt + 4) / 4 : 0;
            unsigned char* const out = a.rec + ((size_t)g * a.Vc + (size_t)(vloc - lane)) * nch * kRecBytes +
                                       (size_t)c * kRecBytes;
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int j = it * 4 + rsub;
                const int pj = __shfl_sync(0xffffffffu, pieces, j);
                if (part < pj) {
                    const uint4 w = reinterpret_cast<const uint4*>(recs + j * kSlotWords)[part];
                    *reinterpret_cast<uint4*>(out + (size_t)j * nch * kRecBytes + part * 16) = w;
                }
            }
            __syncwarp();
        }
    }

    fence_before();
    __syncthreads();
    if (warp == 2) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kTmemCols));
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

template <int D, bool kDump>
cudaError_t launch_t(const Shape& sh, const void* atoms, const ScreenTCArgs& a, int sms, ScreenTCCache* cache,
                     cudaStream_t st)
{
    static_assert(sizeof(CUtensorMap) <= sizeof(cache->map_d), "tensor map size");
    CUtensorMap* md = reinterpret_cast<CUtensorMap*>(cache->map_d);
    const long long drows = (long long)sh.G * sh.N;
    if (cache->d_base != atoms || cache->d_rows != drows) {
        cache->d_base = nullptr;
        if (!make_tma_map_f16(md, atoms, drows, D, 128)) return cudaErrorInvalidValue;
        cache->d_base = atoms;
        cache->d_rows = drows;
    }
    auto k = screen_tc_kernel<D, kDump>;
    const int smem = SmemLayout<D>::alloc;
    if (!cache->attr_done[kDump ? 1 : 0]) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        cache->attr_done[kDump ? 1 : 0] = true;
    }
    return launch_pdl(k, dim3(screen_tc_grid(sh, a.Vc, sms)), dim3(kThreads), smem, st, *md, a);
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

int screen_tc_grid(const Shape& sh, int Vc, int sms)
{
    // one CTA per SM (fewer if there are fewer units than SMs)
    const int tiles = (Vc + kTileV - 1) / kTileV;
    const long long T = (long long)sh.G * tiles * (sh.N / kChunk);
    return (int)(T < sms ? (T > 0 ? T : 1) : sms);
}

// One thread waits on an mbarrier that expects one arrival and gets none:
// the bounded wait runs out after limit_ns and flags the status word.  No
// copy or MMA is issued, so nothing is left in flight when it returns.
__global__ void wait_probe_kernel(unsigned long long* status, unsigned long long limit_ns)
{
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_wait(b, 0u, status, limit_ns);
}

cudaError_t launch_wait_probe(unsigned long long* status, unsigned long long limit_ns, cudaStream_t st)
{
    wait_probe_kernel<<<1, 1, 0, st>>>(status, limit_ns);
    return cudaGetLastError();
}

bool screen_tc_supported(const Shape& sh)
{
    return sh.dtype == FADKV_F16 && (sh.d == 64 || sh.d == 128) && sh.N % kChunk == 0;
}

cudaError_t launch_screen_tc(const Shape& sh, const void* atoms, const ScreenTCArgs& a, int sms, ScreenTCCache* cache,
                             cudaStream_t st)
{
    if (a.Vc <= 0) return cudaSuccess;
    const bool dump = a.dump != nullptr;
    if (sh.d == 128)
        return dump ? launch_t<128, true>(sh, atoms, a, sms, cache, st)
                    : launch_t<128, false>(sh, atoms, a, sms, cache, st);
    return dump ? launch_t<64, true>(sh, atoms, a, sms, cache, st) : launch_t<64, false>(sh, atoms, a, sms, cache, st);
}

}  // namespace fadkv
