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
// (g, tile) is a segment; its vector tile is the MMA's A operand.
//
// S[v][j] = sum_t X[v][t] D[j][t] per unit: A = the vector tile (M = 128
// rows), B = the atom chunk (N = 128 columns), both binary16 K-major with the
// 128-byte swizzle, both brought into shared memory by TMA (the vector tile
// in two buffers, so the next segment's tile loads under the current one;
// the atom chunks through kStages stages); fp32 accumulation in TMEM, three
// accumulator buffers.  Scores never reach HBM.  The epilogue thread of
// vector v keeps atom j if |S[v][j]| >= tau_v, tau_v = alpha * ||x_v|| /
// sqrt(d), with alpha set on the host so that an atom uncorrelated with x_v
// passes with probability ~1.3n/N.  A unit's kept scores go to the vector's
// record (see ScreenTCArgs): four 32-bit masks of the columns kept and the
// scores themselves, exact binary32, in column order -- per score one
// compare, and for a kept one a shared-memory store, a pointer bump and a
// mask bit.  After each unit the warp copies its 32 records out with 16-byte
// loads and stores, eight lanes on a record: the candidate output lands as
// whole sectors.  A row with more than kRecVals kept scores in a unit makes
// the consumer redo the vector.
//
// Warp roles (512 threads): warp 0 issues TMA loads (vector tiles and atom
// chunks), warp 1 issues MMAs (one thread), warp 2 owns the TMEM allocation,
// warp 3 has no role (asking for chunks ahead into L2 was measured: it only
// slowed the stream), warps 4..15 are the epilogue: three groups of four,
// group k takes the units i with i mod 3 = k (accumulator buffer k), warp w
// reads TMEM lanes 32 (w mod 4)...  Each group computes the thresholds of its rows at each
// new segment from the vectors in global memory (coalesced: sixteen lanes
// on a row).  Every wait is bounded by a wall-clock limit; on expiry the CTA
// sets FADKV_DEV_TIMEOUT in the status word, drains its own copies and MMAs
// (the producer waits for every copy it issued, the MMA issuer for its last
// commit, each with the full limit), frees TMEM and returns.
#include "tc_common.cuh"

namespace fadkv {
namespace {

constexpr int kThreads = 512;
constexpr int kTileV = 128;        // vectors per tile (MMA M)
constexpr int kChunk = 128;        // atoms per chunk (MMA N)
constexpr int kAcc = 3;            // accumulator buffers (and epilogue groups)
constexpr int kTmemCols = 512;     // kAcc x 128 columns, allocated as a power of two
constexpr int kEpiWarps = 4 * kAcc;
constexpr int kStagesFor(int D) { return D == 64 ? 6 : 3; }  // atom chunk pipeline depth
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
    static constexpr int kTileBytes = KH * 128 * 128;          // one 128-row operand tile
    static constexpr int b_off = 0;                            // kStages atom chunks
    static constexpr int a_off = b_off + kStages * kTileBytes; // two vector tiles
    static constexpr int s_off = a_off + 2 * kTileBytes;       // the epilogue warps' records
    static constexpr int bar_off = s_off + kEpiWarps * kWarpStageWords * 4;
    static constexpr int n_bars = 2 * kStages + 2 * kAcc + 4;
    static constexpr int taddr_off = bar_off + n_bars * 8;
    static constexpr int total = taddr_off + 16;
    static constexpr int alloc = total + 1024;                 // slack for 1024-byte alignment
    static_assert(alloc <= 227 * 1024, "shared memory");
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
screen_tc_kernel(const __grid_constant__ CUtensorMap map_d, const __grid_constant__ CUtensorMap map_x,
                 ScreenTCArgs a)
{
    using L = SmemLayout<D>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sB = sbase + L::b_off;
    const uint32_t sA = sbase + L::a_off;
    const uint32_t bar0 = sbase + L::bar_off;
    auto full_bar = [&](int i) { return bar0 + 8u * i; };
    auto empty_bar = [&](int i) { return bar0 + 8u * (L::kStages + i); };
    auto tfull_bar = [&](int i) { return bar0 + 8u * (2 * L::kStages + i); };
    auto tempty_bar = [&](int i) { return bar0 + 8u * (2 * L::kStages + kAcc + i); };
    auto afull_bar = [&](int i) { return bar0 + 8u * (2 * L::kStages + 2 * kAcc + i); };
    auto aempty_bar = [&](int i) { return bar0 + 8u * (2 * L::kStages + 2 * kAcc + 2 + i); };
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
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_x)) : "memory");
        for (int i = 0; i < L::kStages; ++i) {
            mbar_init(full_bar(i), 1);
            mbar_init(empty_bar(i), 1);
        }
        for (int i = 0; i < kAcc; ++i) {
            mbar_init(tfull_bar(i), 1);
            mbar_init(tempty_bar(i), 128);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(afull_bar(i), 1);
            mbar_init(aempty_bar(i), 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_begin();                      // the predecessor's writes (x, atoms) are visible from here
    // The TMEM allocation is published to the MMA and epilogue warps (and
    // warp 2) by a named barrier: the producer starts streaming at once.
    constexpr int kTmemSyncThreads = 32 * (2 + kEpiWarps);
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
        // ---------------- TMA producer: vector tiles and atom chunks ----------------
        if (lane == 0) {
            int issued = 0, seg = -1, prev = -1;
            int a_loads[2] = {0, 0};
            bool ok = true;
            UnitCursor uc;
            uc.init(u0, nch, tiles);
            for (int i = 0; i < nu && ok; ++i, uc.advance(1)) {
                if (uc.pair != prev) {
                    // a new segment: its vector tile into buffer seg & 1 once
                    // the MMAs of segment seg - 2 are done with it
                    prev = uc.pair;
                    ++seg;
                    const int ab = seg & 1;
                    if (seg >= 2) ok = mbar_wait(aempty_bar(ab), (uint32_t)((seg >> 1) - 1) & 1u, status, wait_ns);
                    if (!ok) break;
                    mbar_expect_tx(afull_bar(ab), kTileBytes);
                    const int xrow = uc.g * a.V + a.v0 + uc.tile * kTileV;
                    for (int h = 0; h < L::KH; ++h)
                        tma_load_2d(sA + ab * kTileBytes + h * 128 * 128, &map_x, h * 64, xrow, afull_bar(ab));
                    ++a_loads[ab];
                }
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
            for (int ab = 0; ab < 2; ++ab)
                if (a_loads[ab] > 0) mbar_wait(afull_bar(ab), (uint32_t)(a_loads[ab] - 1) & 1u, status);
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
                const int buf = i % kAcc;
                ok = mbar_wait(tempty_bar(buf), ((uint32_t)(i / kAcc) & 1u) ^ 1u, status, wait_ns);
                if (!ok) break;
                const int st = i % L::kStages;
                ok = mbar_wait(full_bar(st), (uint32_t)(i / L::kStages) & 1u, status, wait_ns);
                if (!ok) break;
                fence_after();
                const uint32_t dt = tbase + (uint32_t)(buf * kChunk);
                const uint32_t aA = sA + (uint32_t)(seg & 1) * kTileBytes;
                const uint32_t aB = sB + (uint32_t)st * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (uint32_t)((kk >> 2) * 128 * 128 + (kk & 3) * 32);
                    mma_ss(dt, sdesc(aA + koff), sdesc(aB + koff), kIdesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(empty_bar(st));
                mma_commit(tfull_bar(buf));
                ++issued;
            }
            // drain: the last accumulator must be complete before TMEM is freed
            if (issued > 0)
                mbar_wait(tfull_bar((issued - 1) % kAcc), (uint32_t)((issued - 1) / kAcc) & 1u, status);
        }
    } else if (warp >= 4) {
        // ---------------- epilogue ----------------
        const int e = warp - 4;
        const int grp = e >> 2;                             // accumulator buffer handled
        const int q = warp & 3;                             // TMEM lane group
        const int r = q * 32 + lane;                        // TMEM lane = row of the vector tile
        uint32_t* const recs = reinterpret_cast<uint32_t*>(smem + L::s_off) + e * kWarpStageWords;
        uint32_t* const myrec = recs + lane * kSlotWords;   // header, four masks, then the scores
        const uint32_t myrec_s = smem_u32(myrec);
        int cur = -1, g = 0, vloc = 0;
        bool valid = false, wlive = false, ok = true;
        float tau = __int_as_float(0x7fffffff);
        UnitCursor uc;
        uc.init(u0 + grp, nch, tiles);
        for (int i = grp; i < nu && ok; i += kAcc, uc.advance(kAcc)) {
            const int c = uc.c;
            if (uc.pair != cur) {
                cur = uc.pair;
                g = uc.g;
                vloc = uc.tile * kTileV + r;
                valid = vloc < a.Vc;
                wlive = __any_sync(0xffffffffu, valid);     // a small or ragged batch leaves whole warps idle
                // tau from ||x||^2 of this lane's row (rows past the batch:
                // NaN, never passes).  The warp's 32 rows are read whole,
                // sixteen lanes (eight for d = 64) on a row.
                tau = __int_as_float(0x7fffffff);
                if constexpr (!kDump) {
                    constexpr int LPR = D / 8;                  // lanes per row, 16 bytes each
                    constexpr int RPI = 32 / LPR;               // rows per load
                    const int wrow0 = uc.tile * kTileV + q * 32;
                    const __half* xw = (const __half*)a.x + ((size_t)g * a.V + a.v0) * D;
                    float mine = 0.f;
                    constexpr int NIT = 32 / RPI;
                    uint4 xw4[NIT];                             // every load in flight at once
#pragma unroll
                    for (int it = 0; it < NIT; ++it) {
                        const int rr = it * RPI + lane / LPR;   // row within the warp's 32
                        xw4[it] = (wrow0 + rr < a.Vc)
                                      ? __ldg(reinterpret_cast<const uint4*>(xw + (size_t)(wrow0 + rr) * D) + (lane % LPR))
                                      : make_uint4(0u, 0u, 0u, 0u);
                    }
#pragma unroll
                    for (int it = 0; it < NIT; ++it) {
                        float s = 0.f;
                        {
                            const __half2* hv = reinterpret_cast<const __half2*>(&xw4[it]);
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const float2 f = __half22float2(hv[t]);
                                s = fmaf(f.x, f.x, s);
                                s = fmaf(f.y, f.y, s);
                            }
                        }
#pragma unroll
                        for (int o = LPR / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                        // row it*RPI + k sits in lanes k*LPR .. ; lane `lane` owns row `lane`
#pragma unroll
                        for (int k = 0; k < RPI; ++k) {
                            const float v = __shfl_sync(0xffffffffu, s, k * LPR);
                            if (lane == it * RPI + k) mine = v;
                        }
                    }
                    if (valid) tau = a.alpha * sqrtf(mine * (1.0f / (float)D));
                }
            }
            const int buf = i % kAcc;
            ok = mbar_wait(tfull_bar(buf), (uint32_t)(i / kAcc) & 1u, status, wait_ns);
            if (!ok) break;
            fence_after();
            if (!wlive) {
                // none of this warp's 32 rows is in the batch: nothing to read
                // or write; the buffer is released as soon as it is full, so
                // the warp never runs ahead of the group
                fence_before();
                mbar_arrive(tempty_bar(buf));
                continue;
            }
            const uint32_t tcol = tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kChunk);
            // shared-memory address of this row's next score slot
            uint32_t wp = myrec_s + 5u * 4u;
            const uint32_t wend = myrec_s + (uint32_t)kRecWords * 4u;
            bool ovf = false;
            uint32_t mask[4];
            // one 32-column group: the kept scores and their mask bits
            auto stage = [&](const uint32_t (&v)[32], int qq) {
                if constexpr (kDump) {
                    if (valid) {
                        float* out = a.dump + ((size_t)g * a.Vc + vloc) * a.N + c * kChunk + qq * 32;
#pragma unroll
                        for (int t = 0; t < 32; ++t) out[t] = __uint_as_float(v[t]);
                    }
                    mask[qq] = 0u;
                    return;
                } else {
                    uint32_t m = 0u;
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        if (fabsf(__uint_as_float(v[t])) >= tau) {
                            asm volatile("st.shared.b32 [%0], %1;" ::"r"(wp), "r"(v[t]) : "memory");
                            wp += 4u;
                            m |= 1u << t;
                        }
                    }
                    mask[qq] = m;
                    // a row may run past its record by at most 32 words (into
                    // the next row's slot, or the warp's guard after row 31):
                    // flagged below
                    ovf |= wp > wend;
                    wp = wp > wend ? wend : wp;
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
            const int cnt = (int)((wp - myrec_s) >> 2) - 5;
            myrec[0] = rec_header(over, cnt);
            myrec[1] = mask[0];
            myrec[2] = mask[1];
            myrec[3] = mask[2];
            myrec[4] = mask[3];
            __syncwarp();
            // copy the 32 records out: eight lanes on a record (16 bytes each),
            // four records at a time, only the pieces holding words
            const int part = lane & 7, rsub = lane >> 3;
            const int pieces = valid ? (cnt + 5 + 3) / 4 : 0;
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
    // the inputs [G][V][d]: one map over all G * V rows (a tile past a
    // dictionary's batch reads the next rows, whose scores are never kept;
    // past the last row TMA fills zeros)
    CUtensorMap* mx = reinterpret_cast<CUtensorMap*>(cache->map_x);
    const long long xrows = (long long)sh.G * a.V;
    if (cache->x_base != a.x || cache->x_rows != xrows) {
        cache->x_base = nullptr;
        if (!make_tma_map_f16(mx, a.x, xrows, D, 128)) return cudaErrorInvalidValue;
        cache->x_base = a.x;
        cache->x_rows = xrows;
    }
    auto k = screen_tc_kernel<D, kDump>;
    const int smem = SmemLayout<D>::alloc;
    if (!cache->attr_done[kDump ? 1 : 0]) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        cache->attr_done[kDump ? 1 : 0] = true;
    }
    return launch_pdl(k, dim3(screen_tc_grid(sh, a.Vc, sms)), dim3(kThreads), smem, st, *md, *mx, a);
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
