// fadkv_adapt_noalloc: the fixed-size adaptation (the same kernel as
// fadkv_adapt) run without a handle and without any memory from the caller
// beyond the arrays it already owns.
//
// Who needs it: a caller that cannot hand the library device memory for
// scratch.  Examples are a plain C runtime that drives a fixed memory plan
// and has no allocator to call, and a decode loop that must not call
// cudaMalloc or cudaFree because both can synchronise the whole device and
// stall the streams of other work.  Such a caller still owns the dictionary,
// the usage counts, the inputs and the outputs; the adaptation's own scratch
// (inactive-atom list, flagged-vector list, counters) lives here, in one
// statically sized device array of this library.
//
// Nothing in the scratch has to start at zero: the two lists are written in
// full before they are read inside the same launch, and the counters are
// only accumulated, never read back.  Every call on one device uses the same
// array, so calls that can run at the same time (different streams, or
// different host threads) race on it: issue them in order on one stream.
#include <cuda.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "fadkv_internal.cuh"

namespace fadkv {
namespace {

// 4 MiB: int32 inactive [G][N], int32 flagged [G][V], int64 counters
// [G][kCntFields], each part 256-byte aligned.
constexpr size_t kNoallocScratchBytes = size_t(4) << 20;
static __device__ __align__(256) unsigned char g_adapt_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
// Per device: the scratch's address and the CUDA context it was looked up in.
struct ScratchAddr {
    void* ctx;
    unsigned char* addr;
};
ScratchAddr g_scratch[kMaxDevices];

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

// The calling thread's current CUDA context (the driver's cuCtxGetCurrent,
// reached through the runtime's entry-point query), or null if unknown.
void* current_context()
{
    using Fn = CUresult (*)(CUcontext*);
    static Fn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (Fn) nullptr;
        return (Fn)f;
    }();
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return (void*)c;
}

// Device address of this device's copy of the scratch array, valid in the
// context current on the calling thread.  The first call on a device (which
// must be current) looks it up; later calls in the same context reuse it.
// A different context on that device (a non-primary context made current,
// or the primary context re-created after cudaDeviceReset) gets its own
// lookup, so no call ever writes through an address from a context that
// may be gone.
cudaError_t scratch_for_device(int dev, unsigned char** out)
{
    std::lock_guard<std::mutex> lock(g_setup_mu);
    void* ctx = current_context();
    ScratchAddr& s = g_scratch[dev];
    if (!s.addr || !ctx || s.ctx != ctx) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_adapt_scratch);
        if (e != cudaSuccess) return e;
        // the runtime may have made the device's primary context current
        // during the lookup: key the cache on the context as it is now
        s.ctx = current_context();
        s.addr = (unsigned char*)p;
    }
    *out = s.addr;
    return cudaSuccess;
}

fadkv_status fail(const char* what, cudaError_t e)
{
    char msg[256];
    snprintf(msg, sizeof(msg), "fadkv_adapt_noalloc: %s: %s (%d)", what, cudaGetErrorString(e), (int)e);
    set_last_error(msg);
    return FADKV_ERR_CUDA;
}

bool aligned_to(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace
}  // namespace fadkv

using namespace fadkv;

extern "C" fadkv_status fadkv_adapt_noalloc(const fadkv_params* p, void* atoms, int32_t* usage,
                                            const float* delta, const void* x, int32_t V, const int32_t* idx,
                                            const float* coef, const float* relres, int32_t* repl_id,
                                            float* repl_coef, void* stream)
{
    size_t ws = 0;
    const fadkv_status pst = fadkv_workspace_bytes(p, &ws);   // shape checks only
    if (pst != FADKV_OK) return pst;
    if (V < 0) return FADKV_ERR_INVALID_ARG;
    if (!atoms || !usage || !delta) return FADKV_ERR_INVALID_ARG;
    if (!aligned_to(atoms, 16) || !aligned_to(usage, 4)) return FADKV_ERR_INVALID_ARG;
    if (V > 0 && (!x || !idx || !coef || !relres || !repl_id || !repl_coef)) return FADKV_ERR_INVALID_ARG;
    if (V > 0 && (!aligned_to(x, 16) || !aligned_to(idx, 4) || !aligned_to(coef, 4) ||
                  !aligned_to(relres, 4) || !aligned_to(repl_id, 4) || !aligned_to(repl_coef, 4)))
        return FADKV_ERR_INVALID_ARG;
    const int G = p->num_dicts;
    for (int g = 0; g < G; ++g)
        if (!(delta[g] >= 0.f)) return FADKV_ERR_INVALID_ARG;

    const size_t off_flagged = round256((size_t)G * p->N * sizeof(int32_t));
    const size_t off_counters = off_flagged + round256((size_t)G * (size_t)(V > 0 ? V : 1) * sizeof(int32_t));
    const size_t need = off_counters + (size_t)G * kCntFields * sizeof(long long);
    if (need > kNoallocScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "fadkv_adapt_noalloc: G=%d N=%d V=%d needs %zu bytes of scratch, the static scratch holds %zu",
                 G, (int)p->N, (int)V, need, kNoallocScratchBytes);
        set_last_error(msg);
        return FADKV_ERR_WORKSPACE;
    }
    if (V == 0) return FADKV_OK;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail("cudaGetDevice", e);
    if (dev < 0 || dev >= kMaxDevices) {
        set_last_error("fadkv_adapt_noalloc: device ordinal beyond the 64 this library tracks");
        return FADKV_ERR_UNSUPPORTED;
    }
    unsigned char* base = nullptr;
    e = scratch_for_device(dev, &base);
    if (e != cudaSuccess) return fail("cudaGetSymbolAddress", e);

    const Shape sh{G, p->N, p->d, p->n, p->s, p->dtype, p->lambda_abs, p->lambda_rel};
    DeltaTable dt;
    memset(&dt, 0, sizeof(dt));
    for (int g = 0; g < G; ++g) dt.v[g] = delta[g];
    AdaptArgs a;
    a.atoms = atoms;
    a.usage = usage;
    a.x = x;
    a.idx = idx;
    a.coef = coef;
    a.relres = relres;
    a.repl_id = repl_id;
    a.repl_coef = repl_coef;
    a.inactive = (int32_t*)base;
    a.flagged = (int32_t*)(base + off_flagged);
    a.nrep = nullptr;
    a.counters = (long long*)(base + off_counters);
    a.V = V;
    a.append = 0;
    e = launch_adapt(sh, a, dt, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail("launch", e);
    return FADKV_OK;
}
