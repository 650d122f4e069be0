// Exact Top-n pool from the screening candidates, one warp per vector.
//
// "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding",
// abstract: a one-shot Top-n selection identifies a small candidate pool;
// ties go to the lower atom index (a convention of this library).
//
// The candidates of a vector arrive as the screening kernel's records: per
// 128-atom chunk a header, the mask of the atoms kept and their scores.  A
// warp decodes
// them into 64-bit keys (bits(|r_j|) << 32) | ((0x7fffffff - j) << 1) |
// sign(r_j) in its slice of shared memory (the larger key is the larger |r|,
// then the lower atom index; the sign bit never decides, atoms being
// distinct), then:
//   1. buckets the keys by |r| on a grid of 256 buckets over the binary32
//      bit patterns between the smallest and largest |r| of the list (the
//      range is tracked while decoding; the grid is monotone in |r|, so every
//      key of a higher bucket beats every key of a lower one);
//   2. finds the bucket B holding the n-th largest key from the histogram;
//   3. in one pass takes all keys above B and compacts B's keys, then the
//      best `rem` keys of B by full 64-bit key (|r|, then the lower index) --
//      by rank within the warp when B holds at most 32 keys, else by an MSD
//      radix select restricted to B.
// Only warp-level synchronisation, so many warps share an SM and hide each
// other's latency.  A vector whose list overflowed or holds fewer than n
// keys gets pool[0] = -2 and is left to the exact slow path of the greedy
// kernel.
#include "fadkv_internal.cuh"

namespace fadkv {
namespace {

constexpr int kWarpsPerCta = 4;

__device__ __forceinline__ unsigned long long sel_key(uint32_t absbits, uint32_t atom, uint32_t sign)
{
    return ((unsigned long long)absbits << 32) | (((0x7fffffffu - atom) << 1) | sign);
}
__device__ __forceinline__ int key_atom(unsigned long long k) { return (int)(0x7fffffffu - ((uint32_t)k >> 1)); }
__device__ __forceinline__ float key_r(unsigned long long k)
{
    return __uint_as_float((uint32_t)(k >> 32) | ((uint32_t)k << 31));
}

// KPL: keys per lane held in registers after the decode (cap <= 32 KPL)
template <int KPL>
__global__ void __launch_bounds__(kWarpsPerCta * 32, 5)
select_kernel(SelectArgs a)
{
    pdl_begin();
    extern __shared__ unsigned long long kbuf_all[];   // [kWarpsPerCta][cap]
    __shared__ uint32_t hist_all[kWarpsPerCta][256];
    // 32 records of a warp, one 36-word row each (16-byte aligned rows; a
    // record's reads by its lane hit banks four apart from the next lane's)
    constexpr int kStageRow = 36;
    __shared__ __align__(16) uint32_t stage_all[kWarpsPerCta][32 * kStageRow];
    const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
    const long long gw = (long long)blockIdx.x * kWarpsPerCta + wl;   // (g, vc) flattened
    if (gw >= (long long)a.G * a.Vc) return;
    uint32_t* hist = hist_all[wl];
    unsigned long long* keys = kbuf_all + (size_t)wl * a.cap;
    const int n = a.n;
    int32_t* pool = a.pool + gw * n;
    float* pool_r = a.pool_r + gw * n;
    auto put = [&](int pos, unsigned long long k) {
        pool[pos] = key_atom(k);
        pool_r[pos] = key_r(k);
    };

    // the screening records of this vector, 32 at a time: every record's
    // 16-byte pieces in one batch of loads (eight lanes on a record, four
    // records per load) into the warp's staging rows; then lane l decodes
    // record l: its scores go to the sum of the counts of the records before
    // it, the v-th score with the atom of the (v+1)-th set bit of the
    // record's 128-bit mask (128 c + the bit's position)
    const int nch = a.N / 128;
    const unsigned char* rec = a.rec + (size_t)gw * nch * kRecBytes;
    uint32_t* const stage = stage_all[wl];
    const int part = lane & 7, rsub = lane >> 3;
    constexpr int kIt = 8;                  // loads per lane: 32 records x 8 pieces over 32 lanes
    static_assert(kRecBytes / 16 == 8, "eight lanes cover a record");
    int gbase = 0;
    uint32_t lo = 0xffffffffu, hi = 0u;      // range of |r| bits over the keys this lane writes
    for (int cg = 0; cg < nch; cg += 32) {
        const int cc = cg + lane;
        uint4 w[kIt];
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int j = cg + it * 4 + rsub;
            w[it] = j < nch ? __ldg(reinterpret_cast<const uint4*>(rec + (size_t)j * kRecBytes) + part)
                            : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int it = 0; it < kIt; ++it)
            reinterpret_cast<uint4*>(stage + (it * 4 + rsub) * kStageRow)[part] = w[it];
        __syncwarp();
        const uint32_t* const mine = stage + lane * kStageRow;
        const bool live = cc < nch;
        const uint32_t h = live ? mine[0] : 0u;
        const uint32_t mk[4] = {live ? mine[1] : 0u, live ? mine[2] : 0u, live ? mine[3] : 0u, live ? mine[4] : 0u};
        // every kept atom is in the masks, also past the record's room
        const int cnt = __popc(mk[0]) + __popc(mk[1]) + __popc(mk[2]) + __popc(mk[3]);
        const bool over = (h >> 31) != 0u;
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        const int off = gbase + incl - cnt;
        if (live && !over) {
            int vi = 0;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                uint32_t m = mk[qq];
                while (m != 0u && vi < cnt) {
                    const uint32_t t = (uint32_t)(__ffs(m) - 1);
                    m &= m - 1u;
                    if (off + vi < a.cap) {
                        const uint32_t val = mine[5 + vi];
                        const uint32_t ab = val & 0x7fffffffu;
                        keys[off + vi] = sel_key(ab, (uint32_t)cc * 128u + 32u * qq + t, val >> 31);
                        lo = min(lo, ab);
                        hi = max(hi, ab);
                    }
                    ++vi;
                }
            }
        }
        // a record that overflowed (or that a neighbour's overflow wrote
        // into) has its masks but not all its scores: the warp recomputes
        // the scores of its kept atoms on the FP32 pipe, lane l the l-th
        // kept atom of each 32-atom group
        unsigned ob = __ballot_sync(0xffffffffu, live && over);
        while (ob != 0u) {
            const int j = __ffs(ob) - 1;
            ob &= ob - 1u;
            const int offj = __shfl_sync(0xffffffffu, off, j);
            const int cj = cg + j;
            const int g = (int)(gw / a.Vc), vc = (int)(gw - (long long)g * a.Vc);
            const __half* xr = a.x + ((size_t)g * a.V + a.v0 + vc) * a.d;
            int base = 0;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                const uint32_t mq = __shfl_sync(0xffffffffu, mk[qq], j);
                const int pq = __popc(mq);
                if (lane < pq) {
                    uint32_t mm = mq;
                    for (int r = 0; r < lane; ++r) mm &= mm - 1u;
                    const uint32_t atom = (uint32_t)cj * 128u + 32u * qq + (uint32_t)(__ffs(mm) - 1);
                    const __half* ar = a.atoms + ((size_t)g * a.N + atom) * a.d;
                    // every 16-byte piece of both rows in flight at once (d <= 128)
                    uint4 xa[16], aa[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const bool in = c < a.d / 8;
                        xa[c] = in ? __ldg(reinterpret_cast<const uint4*>(xr) + c) : make_uint4(0u, 0u, 0u, 0u);
                        aa[c] = in ? __ldg(reinterpret_cast<const uint4*>(ar) + c) : make_uint4(0u, 0u, 0u, 0u);
                    }
                    float acc = 0.f;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const __half2* xh = reinterpret_cast<const __half2*>(&xa[c]);
                        const __half2* ah = reinterpret_cast<const __half2*>(&aa[c]);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float2 xf = __half22float2(xh[u]), af = __half22float2(ah[u]);
                            acc = fmaf(xf.x, af.x, acc);
                            acc = fmaf(xf.y, af.y, acc);
                        }
                    }
                    const uint32_t bits = __float_as_uint(acc);
                    if (offj + base + lane < a.cap) {
                        keys[offj + base + lane] = sel_key(bits & 0x7fffffffu, atom, bits >> 31);
                        lo = min(lo, bits & 0x7fffffffu);
                        hi = max(hi, bits & 0x7fffffffu);
                    }
                }
                base += pq;
            }
        }
        gbase = __shfl_sync(0xffffffffu, off + cnt, 31);
        __syncwarp();
    }
    const int K = gbase;
    auto slow = [&]() {
        if (lane == 0) {
            pool[0] = -2;                              // exact slow path (pool fixup, or the greedy kernel)
            *a.slow_seq = a.seq;                       // every writer stores the same value
        }
    };
    // too few or too many keys: the slow path
    if (K < n || K > a.cap) {
        slow();
        return;
    }
    __syncwarp();

    // 1. the bucket grid: 256 buckets over the bit patterns of |r| between
    //    the smallest and largest kept (non-negative binary32 values order
    //    like their bits, so the buckets are monotone in |r|; the grid is
    //    near logarithmic, which spreads the many scores just above the
    //    screening threshold over many buckets)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    const uint32_t span = hi - lo;
    const int bsh = span > 255u ? (32 - __clz(span)) - 8 : 0;   // (span >> bsh) <= 255
    auto bucket = [&](unsigned long long k) -> uint32_t {
        return min(255u, ((uint32_t)(k >> 32) - lo) >> bsh);
    };

    // the keys into registers, key i in lane i % 32 at slot i / 32: the
    // passes below read no shared memory
    const int nk = (K + 31) >> 5;
    unsigned long long kr[KPL];
#pragma unroll
    for (int j = 0; j < KPL; ++j) kr[j] = (j * 32 + lane < K) ? keys[j * 32 + lane] : 0ull;

    // 2. histogram and the boundary bucket (lane l scans buckets 255-8l .. 248-8l)
#pragma unroll
    for (int b = 0; b < 8; ++b) hist[lane * 8 + b] = 0;
    __syncwarp();
#pragma unroll
    for (int j = 0; j < KPL; ++j)
        if (j * 32 + lane < K) atomicAdd(&hist[bucket(kr[j])], 1u);
    __syncwarp();
    const int top = 255 - 8 * lane;
    uint32_t local = 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) local += hist[top - b];
    uint32_t inc = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    const uint32_t above0 = inc - local;
    const bool mine = above0 < (uint32_t)n && (uint32_t)n <= inc;
    uint32_t bsel = 0, rem = 0, nb = 0;
    if (mine) {
        uint32_t acc = above0;
        for (int b = 0; b < 8; ++b) {
            const uint32_t h = hist[top - b];
            if (acc + h >= (uint32_t)n) {
                bsel = (uint32_t)(top - b);
                rem = (uint32_t)n - acc;
                nb = h;
                break;
            }
            acc += h;
        }
    }
    const int sl = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
    bsel = __shfl_sync(0xffffffffu, bsel, sl);
    rem = __shfl_sync(0xffffffffu, rem, sl);
    nb = __shfl_sync(0xffffffffu, nb, sl);

    // 3. one pass: keys above the boundary bucket go to the pool (with the
    //    bucket's own when all of it is taken); otherwise the bucket's keys
    //    are compacted to the front of the shared buffer
    const bool whole_b = rem == nb;
    unsigned long long* bkeys = keys;
    int base = 0, mb = 0;
#pragma unroll
    for (int j = 0; j < KPL; ++j) {
        if (j >= nk) break;
        const int i = j * 32 + lane;
        const unsigned long long k = kr[j];
        const uint32_t b = (i < K) ? bucket(k) : 0u;
        const bool fp = (i < K) && (b > bsel || (whole_b && b == bsel));
        const bool fc = (i < K) && !whole_b && b == bsel;
        const unsigned balp = __ballot_sync(0xffffffffu, fp);
        const unsigned balc = __ballot_sync(0xffffffffu, fc);
        if (fp) put(base + __popc(balp & ((1u << lane) - 1u)), k);
        if (fc) bkeys[mb + __popc(balc & ((1u << lane) - 1u))] = k;
        base += __popc(balp);
        mb += __popc(balc);
    }
    if (whole_b) return;
    __syncwarp();
    if (mb <= 32) {
        const unsigned long long mk = (lane < mb) ? bkeys[lane] : 0ull;
        uint32_t rank = 0;   // keys of the bucket larger than mine (keys are unique)
        for (int j = 0; j < mb; ++j) rank += (__shfl_sync(0xffffffffu, mk, j) > mk) ? 1u : 0u;
        const bool f = lane < mb && rank < rem;
        const unsigned bal = __ballot_sync(0xffffffffu, f);
        if (f) put(base + __popc(bal & ((1u << lane) - 1u)), mk);
        return;
    }
    // rare: a crowded bucket -- MSD radix select over the bucket's keys
    unsigned long long prefix = 0ull, mask = 0ull;
    uint32_t remaining = rem;
    int shift = 56;
    for (;; shift -= 8) {
#pragma unroll
        for (int b = 0; b < 8; ++b) hist[lane * 8 + b] = 0;
        __syncwarp();
        for (int i = lane; i < mb; i += 32) {
            const unsigned long long k = bkeys[i];
            if ((k & mask) == prefix) atomicAdd(&hist[(uint32_t)(k >> shift) & 0xffu], 1u);
        }
        __syncwarp();
        uint32_t loc = 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) loc += hist[top - b];
        uint32_t in2 = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, in2, o);
            if (lane >= o) in2 += t;
        }
        const uint32_t ab = in2 - loc;
        const bool mn = ab < remaining && remaining <= in2;
        uint32_t bs = 0, rn = 0, whole = 0;
        if (mn) {
            uint32_t acc = ab;
            for (int b = 0; b < 8; ++b) {
                const uint32_t h = hist[top - b];
                if (acc + h >= remaining) {
                    bs = (uint32_t)(top - b);
                    rn = remaining - acc;
                    whole = (h == rn) ? 1u : 0u;
                    break;
                }
                acc += h;
            }
        }
        const int s2 = __ffs(__ballot_sync(0xffffffffu, mn)) - 1;
        bs = __shfl_sync(0xffffffffu, bs, s2);
        rn = __shfl_sync(0xffffffffu, rn, s2);
        whole = __shfl_sync(0xffffffffu, whole, s2);
        prefix |= (unsigned long long)bs << shift;
        remaining = rn;
        mask |= 0xffull << shift;
        __syncwarp();
        if (whole || shift == 0) break;
    }
    const unsigned long long lim = prefix >> shift;
    for (int i0 = 0; i0 < mb; i0 += 32) {
        const int i = i0 + lane;
        const unsigned long long k = (i < mb) ? bkeys[i] : 0ull;
        const bool f = (i < mb) && (k >> shift) >= lim;
        const unsigned bal = __ballot_sync(0xffffffffu, f);
        if (f) put(base + __popc(bal & ((1u << lane) - 1u)), k);
        base += __popc(bal);
    }
}

}  // namespace

size_t select_smem_bytes(int cap) { return (size_t)kWarpsPerCta * cap * sizeof(unsigned long long); }

cudaError_t launch_select(const SelectArgs& a, cudaStream_t st)
{
    const long long warps = (long long)a.G * a.Vc;
    if (warps <= 0) return cudaSuccess;
    if (a.cap > 32 * 32) return cudaErrorInvalidValue;
    const size_t smem = select_smem_bytes(a.cap);
    auto k = a.cap <= 32 * 16 ? select_kernel<16> : select_kernel<32>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned blocks = (unsigned)((warps + kWarpsPerCta - 1) / kWarpsPerCta);
    return launch_pdl(k, dim3(blocks), dim3(kWarpsPerCta * 32), smem, st, a);
}

}  // namespace fadkv
