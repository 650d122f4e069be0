// Exact Top-n pool from the screening candidates, one warp per vector.
//
// "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding",
// abstract: a one-shot Top-n selection identifies a small candidate pool;
// ties go to the lower atom index (a convention of this library).
//
// The candidates of a vector arrive as 64-bit keys (bits(|r_j|) << 32) |
// (0xffffffff - j) split into regions with one count each.  A warp gathers
// them into its own slice of shared memory, finds the n-th largest by an MSD
// radix select over bytes -- a 256-bin histogram per warp, one shared atomic
// per distinct bin per 32 keys -- and writes the pool's atom ids (in no
// particular order) with ballots.  Only warp-level synchronisation: many
// warps share an SM and hide each other's latency, and the register-heavy
// greedy kernel starts from the finished pool.  A vector whose list
// overflowed or holds fewer than n keys gets pool[0] = -2 and is left to the
// exact slow path of the greedy kernel.
#include "fadkv_internal.cuh"

namespace fadkv {
namespace {

constexpr int kWarpsPerCta = 4;

__global__ void __launch_bounds__(kWarpsPerCta * 32)
select_kernel(SelectArgs a)
{
    extern __shared__ unsigned long long kbuf_all[];   // [kWarpsPerCta][cap]
    __shared__ uint32_t hist_all[kWarpsPerCta][256];
    __shared__ int offs_all[kWarpsPerCta][kCountSlots + 1];
    const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
    const long long gw = (long long)blockIdx.x * kWarpsPerCta + wl;   // (g, vc) flattened
    if (gw >= (long long)a.G * a.Vc) return;
    uint32_t* hist = hist_all[wl];
    int* offs = offs_all[wl];
    unsigned long long* keys = kbuf_all + (size_t)wl * a.cap;
    const int n = a.n;
    int32_t* pool = a.pool + gw * n;

    // region counts -> total and region offsets
    const int nreg = 2 * a.slices;
    const int cs = a.cap / nreg;
    int* counts = a.cand_count + gw * kCountSlots;
    const int c = (lane < nreg) ? counts[lane] : 0;
    const int over = __any_sync(0xffffffffu, c > cs);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    const int K = __shfl_sync(0xffffffffu, incl, 31);
    if (lane < nreg) {
        offs[lane] = incl - c;
        counts[lane] = 0;                              // consumed: ready for the next call
    }
    if (over || K < n) {
        if (lane == 0) pool[0] = -2;                   // exact slow path in the greedy kernel
        return;
    }
    __syncwarp();

    // gather the regions back to back
    const unsigned long long* src = a.cand + gw * a.cap;
    for (int r = 0; r < nreg; ++r) {
        const int o0 = offs[r];
        const int len = (r + 1 < nreg ? offs[r + 1] : K) - o0;
        for (int i = lane; i < len; i += 32) keys[o0 + i] = src[(size_t)r * cs + i];
    }
    __syncwarp();

    // MSD radix select of the n-th largest key
    unsigned long long prefix = 0ull, mask = 0ull;
    uint32_t remaining = (uint32_t)n;
    int shift = 56;
    for (;; shift -= 8) {
#pragma unroll
        for (int b = 0; b < 8; ++b) hist[lane * 8 + b] = 0;
        __syncwarp();
        for (int i0 = 0; i0 < K; i0 += 32) {
            const int i = i0 + lane;
            const unsigned long long k = (i < K) ? keys[i] : 0ull;
            const bool in = (i < K) && (k & mask) == prefix;
            const uint32_t bin = in ? ((uint32_t)(k >> shift) & 0xffu) : 0x100u;
            const unsigned peers = __match_any_sync(0xffffffffu, bin);
            if (in && (__ffs(peers) - 1) == lane) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
        }
        __syncwarp();
        // lane l covers bins 255-8l .. 248-8l (lane 0 holds the top)
        const int hi = 255 - 8 * lane;
        uint32_t local = 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) local += hist[hi - b];
        uint32_t inc = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += t;
        }
        const uint32_t above = inc - local;
        const bool mine = above < remaining && remaining <= inc;
        uint32_t bin_sel = 0, rem_new = 0, whole = 0;
        if (mine) {
            uint32_t acc = above;
            for (int b = 0; b < 8; ++b) {
                const uint32_t h = hist[hi - b];
                if (acc + h >= remaining) {
                    bin_sel = (uint32_t)(hi - b);
                    rem_new = remaining - acc;
                    whole = (h == rem_new) ? 1u : 0u;
                    break;
                }
                acc += h;
            }
        }
        const int src_lane = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
        bin_sel = __shfl_sync(0xffffffffu, bin_sel, src_lane);
        rem_new = __shfl_sync(0xffffffffu, rem_new, src_lane);
        whole = __shfl_sync(0xffffffffu, whole, src_lane);
        prefix |= (unsigned long long)bin_sel << shift;
        remaining = rem_new;
        mask |= 0xffull << shift;
        __syncwarp();
        if (whole || shift == 0) break;
    }

    // selected: keys whose bits from `shift` up are >= prefix's
    const unsigned long long lim = prefix >> shift;
    int base = 0;
    for (int i0 = 0; i0 < K; i0 += 32) {
        const int i = i0 + lane;
        const unsigned long long k = (i < K) ? keys[i] : 0ull;
        const bool f = (i < K) && (k >> shift) >= lim;
        const unsigned bal = __ballot_sync(0xffffffffu, f);
        if (f) {
            const int pos = base + __popc(bal & ((1u << lane) - 1u));
            if (pos < n) pool[pos] = (int)(0xffffffffu - (uint32_t)(k & 0xffffffffull));
        }
        base += __popc(bal);
    }
}

}  // namespace

size_t select_smem_bytes(int cap) { return (size_t)kWarpsPerCta * cap * sizeof(unsigned long long); }

cudaError_t launch_select(const SelectArgs& a, cudaStream_t st)
{
    const long long warps = (long long)a.G * a.Vc;
    if (warps <= 0) return cudaSuccess;
    const size_t smem = select_smem_bytes(a.cap);
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned blocks = (unsigned)((warps + kWarpsPerCta - 1) / kWarpsPerCta);
    select_kernel<<<blocks, kWarpsPerCta * 32, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace fadkv
