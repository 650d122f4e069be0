// Host side of the C ABI declared in include/fadkv.h: argument checks, the
// encode/adapt sequence contract, workspace carving and kernel launches.
// The library never allocates device memory: the caller passes the
// dictionary, the usage counts and one zero-filled workspace.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <new>
#include <vector>

#include "fadkv_internal.cuh"

using namespace fadkv;

namespace {

thread_local char g_last_error[256] = "";

void set_error(const char* where, cudaError_t e)
{
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(e), (int)e);
}

// Host-side fault injection for tests: FADKV_FAULT=cuda makes every call
// that would launch work fail with FADKV_ERR_CUDA before launching anything.
bool fault_injected()
{
    const char* f = getenv("FADKV_FAULT");
    return f && strcmp(f, "cuda") == 0;
}

constexpr size_t kAlign = 256;
constexpr size_t kScoreBudget = size_t(1) << 30;   // FP32 path: materialised scores per chunk
constexpr size_t kCandBudget = size_t(512) << 20;  // candidate lists per chunk

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Screening path: tensor cores for binary16 dictionaries (FADKV_SCREEN=ffma
// forces the FP32 path, used to cross-check the two).
bool use_tc(const fadkv_params& p)
{
    const char* f = getenv("FADKV_SCREEN");
    if (f && strcmp(f, "ffma") == 0) return false;
    Shape sh{p.num_dicts, p.N, p.d, p.n, p.s, p.dtype, p.lambda_abs, p.lambda_rel};
    return screen_tc_supported(sh);
}

struct Layout {
    bool tc;     // screening on tensor cores with candidate filtering
    bool gram;   // greedy over the dictionaries' Gram matrices (binary16, tensor-core screening)
    int chunk;   // vectors per dictionary per encode pass
    int cap;     // candidate capacity per vector
    size_t counters, scores, cand, cand_count, pool, pool_r, inactive, flagged, slow, nrep, gdiag, gram_off, total;
};

Layout make_layout(const fadkv_params& p)
{
    Layout L;
    L.tc = use_tc(p);
    const Shape sh{p.num_dicts, p.N, p.d, p.n, p.s, p.dtype, p.lambda_abs, p.lambda_rel};
    L.gram = L.tc && greedy_gram_supported(sh);
    L.cap = cand_cap(p.n);
    const size_t G = (size_t)p.num_dicts;
    const size_t mb = (size_t)(p.max_batch > 0 ? p.max_batch : 1);
    // candidate bytes per vector: the FP32 path's lists, or the tensor-core
    // path's screening records (kRecBytes per 128 atoms)
    const size_t cand_bytes = L.tc ? (size_t)(p.N / 128) * kRecBytes : (size_t)L.cap * 8;
    size_t chunk = L.tc ? kCandBudget / (G * cand_bytes) : kScoreBudget / (G * (size_t)p.N * sizeof(float));
    if (chunk >= mb) chunk = mb;
    else if (chunk >= 256) chunk = chunk / 128 * 128;   // whole MMA tiles
    if (chunk < 1) chunk = 1;
    L.chunk = (int)chunk;
    size_t o = 0;
    L.counters = o;   o = align_up(o + G * kCntFields * sizeof(long long), kAlign);
    L.scores = o;     o = align_up(o + (L.tc ? 0 : G * chunk * (size_t)p.N * sizeof(float)), kAlign);
    L.cand = o;       o = align_up(o + G * chunk * cand_bytes, kAlign);
    L.cand_count = o; o = align_up(o + G * chunk * kCountSlots * sizeof(int), kAlign);
    L.pool = o;       o = align_up(o + (L.tc ? G * chunk * (size_t)p.n * sizeof(int32_t) : 0), kAlign);
    L.pool_r = o;     o = align_up(o + (L.tc ? G * chunk * (size_t)p.n * sizeof(float) : 0), kAlign);
    L.inactive = o;   o = align_up(o + G * (size_t)p.N * sizeof(int32_t), kAlign);
    L.flagged = o;    o = align_up(o + G * mb * sizeof(int32_t), kAlign);
    L.slow = o;       o = align_up(o + sizeof(uint32_t), kAlign);
    L.nrep = o;       o = align_up(o + G * sizeof(int32_t), kAlign);
    L.gdiag = o;      o = align_up(o + (L.gram ? G * (size_t)p.N * sizeof(float) : 0), kAlign);
    L.gram_off = o;   o = align_up(o + (L.gram ? gram_bytes(sh) : 0), kAlign);
    L.total = o;
    return L;
}

// alpha with P(|Z| >= alpha) = min(1, 1.3n/N) for a standard normal Z, by
// bisection on erfc: an atom uncorrelated with x has |<d, x>| ~ ||x||/sqrt(d)
// |Z|, so tau = alpha ||x|| / sqrt(d) keeps about 1.3n candidates per vector
// (the count sits four standard deviations above n at the decode shapes; a
// list that ends short is redone exactly).
float screen_alpha(int n, int N)
{
    double f = 1.3 * n / (double)N;
    if (f >= 1.0) return 0.f;
    double lo = 0.0, hi = 40.0;
    for (int i = 0; i < 200; ++i) {
        const double mid = 0.5 * (lo + hi);
        if (erfc(mid / sqrt(2.0)) > f) lo = mid;
        else hi = mid;
    }
    return (float)lo;
}

fadkv_status check_params(const fadkv_params* p)
{
    if (!p) return FADKV_ERR_INVALID_ARG;
    if (p->num_dicts < 1 || p->N < 1 || p->d < 1 || p->n < 1 || p->s < 1 || p->max_batch < 0)
        return FADKV_ERR_INVALID_ARG;
    if (p->s > p->n || p->n > p->N) return FADKV_ERR_INVALID_ARG;
    if (!(p->lambda_abs >= 0.f) || !(p->lambda_rel >= 0.f)) return FADKV_ERR_INVALID_ARG;
    if (p->dtype != FADKV_F16 && p->dtype != FADKV_F32) return FADKV_ERR_INVALID_ARG;
    if (p->num_dicts > FADKV_MAX_DICTS || p->s > FADKV_MAX_S || p->n > FADKV_MAX_POOL)
        return FADKV_ERR_UNSUPPORTED;
    if (p->d != 64 && p->d != 128) return FADKV_ERR_UNSUPPORTED;
    if (p->N % 64 != 0) return FADKV_ERR_UNSUPPORTED;
    if ((size_t)p->N * sizeof(uint32_t) > 200 * 1024) return FADKV_ERR_UNSUPPORTED;   // Top-n keys in smem
    if (p->lambda_abs == 0.f && p->lambda_rel == 0.f) {
        // plain least squares is allowed; positive definiteness then rests on
        // the selected atoms being linearly independent (status bit if not)
    }
    Shape sh{p->num_dicts, p->N, p->d, p->n, p->s, p->dtype, p->lambda_abs, p->lambda_rel};
    if (greedy_smem_bytes(sh) > 227 * 1024) return FADKV_ERR_UNSUPPORTED;
    return FADKV_OK;
}

bool aligned(const void* ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

}  // namespace

// Records a message for fadkv_last_error on this host thread (used by entry
// points defined in other translation units).
bool fadkv::pdl_enabled()
{
    static const bool on = [] {
        const char* f = getenv("FADKV_PDL");
        return !(f && strcmp(f, "0") == 0);
    }();
    return on;
}

void fadkv::set_last_error(const char* msg)
{
    snprintf(g_last_error, sizeof(g_last_error), "%s", msg);
}

struct ProfRec {
    int cls;
    cudaEvent_t start, stop;
};

struct fadkv_dict_s {
    fadkv_params p;
    Shape sh;
    Layout L;
    void* atoms;
    int32_t* usage;
    unsigned char* ws;
    size_t ws_bytes;
    DeltaTable delta;
    bool pending;      // an encode batch waits for its adapt
    int32_t pending_V;
    int sms;           // multiprocessors of the device (queried at first use)
    uint32_t seq;      // screening passes issued (the slow-path flag names the pass)
    bool gram_ready;   // the Gram matrices hold the current atoms
    unsigned long long wait_ns;   // screening pipeline's wait limit (0: the kernel's default)
    float alpha;       // screening threshold factor
    ScreenTCCache tc_cache;   // tensor maps of the screening kernel
    // tracing
    bool prof_on;
    uint32_t prof_mask;    // kernel classes bracketed while profiling
    int64_t launches[FADKV_PROFILE_KERNELS];
    double ms[FADKV_PROFILE_KERNELS];
    std::vector<ProfRec> prof_pending;
    std::vector<cudaEvent_t> prof_free;
};

namespace {

long long* counters(fadkv_dict h) { return (long long*)(h->ws + h->L.counters); }

cudaEvent_t prof_event(fadkv_dict h)
{
    if (!h->prof_free.empty()) {
        cudaEvent_t e = h->prof_free.back();
        h->prof_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Brackets one kernel launch for tracing; `launch` returns its cudaError_t.
template <typename F>
cudaError_t traced(fadkv_dict h, int cls, cudaStream_t st, F&& launch)
{
    cudaEvent_t a = nullptr, b = nullptr;
    if (h->prof_on && ((h->prof_mask >> cls) & 1u)) {
        a = prof_event(h);
        b = prof_event(h);
        if (a && b) cudaEventRecord(a, st);
    }
    const cudaError_t e = launch();
    if (e == cudaSuccess) h->launches[cls] += 1;
    if (a && b) {
        cudaEventRecord(b, st);
        h->prof_pending.push_back(ProfRec{cls, a, b});
    } else {
        if (a) h->prof_free.push_back(a);
        if (b) h->prof_free.push_back(b);
    }
    return e;
}

cudaError_t ensure_device_info(fadkv_dict h)
{
    if (h->sms > 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) h->sms = sms > 0 ? sms : 1;
    return e;
}

unsigned long long* cand_buf(fadkv_dict h) { return (unsigned long long*)(h->ws + h->L.cand); }
int* cand_count_buf(fadkv_dict h) { return (int*)(h->ws + h->L.cand_count); }

// Screening of vectors [v0, v0+Vc) of every dictionary: candidate lists
// (tensor-core path) or the exact Top-n keys (FP32 path).  With `dump` set,
// writes all scores [G][Vc][N] instead (test hook).

// n_sel: the pool size to select (the handle's n for the greedy coder, s
// for the PL fit).
cudaError_t run_screen(fadkv_dict h, const void* x, int32_t V, int v0, int Vc, float* dump, cudaStream_t st,
                       int n_sel)
{
    cudaError_t e = ensure_device_info(h);
    if (e != cudaSuccess) return e;
    if (h->L.tc) {
        ScreenTCArgs a;
        a.G = h->p.num_dicts;
        a.N = h->p.N;
        a.V = V;
        a.v0 = v0;
        a.Vc = Vc;
        a.x = x;
        a.alpha = h->alpha;
        a.rec = h->ws + h->L.cand;
        a.dump = dump;
        a.counters = counters(h);
        a.wait_ns = h->wait_ns;
        e = traced(h, FADKV_K_SCREEN, st, [&] { return launch_screen_tc(h->sh, h->atoms, a, h->sms, &h->tc_cache, st); });
        if (e != cudaSuccess || dump) return e;
        SelectArgs sa;
        sa.G = h->p.num_dicts;
        sa.Vc = Vc;
        sa.N = h->p.N;
        sa.n = n_sel;
        sa.cap = select_cap(h->p.n);
        sa.d = h->p.d;
        sa.V = V;
        sa.v0 = v0;
        sa.x = (const __half*)x;
        sa.atoms = (const __half*)h->atoms;
        sa.rec = h->ws + h->L.cand;
        sa.pool = (int32_t*)(h->ws + h->L.pool);
        sa.pool_r = (float*)(h->ws + h->L.pool_r);
        if (++h->seq == 0) h->seq = 1;                 // 0 is the workspace's initial value
        sa.slow_seq = (uint32_t*)(h->ws + h->L.slow);
        sa.seq = h->seq;
        return traced(h, FADKV_K_TOPN, st, [&] { return launch_select(sa, st); });
    }
    float* scores = dump ? dump : (float*)(h->ws + h->L.scores);
    e = traced(h, FADKV_K_SCREEN, st, [&] {
        return launch_screen_ffma(h->sh, h->atoms, x, (int64_t)V * h->p.d, v0, Vc, scores, st);
    });
    if (e != cudaSuccess || dump) return e;
    Shape sh = h->sh;
    sh.n = n_sel;
    return traced(h, FADKV_K_TOPN, st, [&] {
        return launch_topn_radix(sh, scores, Vc, cand_buf(h), cand_count_buf(h), h->L.cap, st);
    });
}

float* gram_ptr(fadkv_dict h) { return (float*)(h->ws + h->L.gram_off); }
float* gdiag_ptr(fadkv_dict h) { return (float*)(h->ws + h->L.gdiag); }

// The Gram matrices of every dictionary, from the atoms as they stand.
cudaError_t build_gram(fadkv_dict h, cudaStream_t st)
{
    cudaError_t e = ensure_device_info(h);
    if (e != cudaSuccess) return e;
    e = traced(h, FADKV_K_GRAM, st, [&] {
        return launch_gram_build(h->sh, h->atoms, gram_ptr(h), gdiag_ptr(h), h->sms, st);
    });
    if (e == cudaSuccess) h->gram_ready = true;
    return e;
}

GreedyArgs greedy_args(fadkv_dict h, const void* x, int32_t V, int v0, int Vc)
{
    GreedyArgs a;
    a.atoms = h->atoms;
    a.x = x;
    a.cand = cand_buf(h);
    a.cand_count = cand_count_buf(h);
    a.cap = h->L.cap;
    a.pool_in = h->L.tc ? (const int32_t*)(h->ws + h->L.pool) : nullptr;
    a.idx = nullptr;
    a.coef = nullptr;
    a.relres = nullptr;
    a.pool_out = nullptr;
    a.pool_r_out = nullptr;
    a.counters = counters(h);
    a.V = V;
    a.v0 = v0;
    a.Vc = Vc;
    return a;
}

}  // namespace

extern "C" {

int32_t fadkv_abi_version(void) { return FADKV_ABI_VERSION; }

const char* fadkv_status_string(fadkv_status s)
{
    switch (s) {
    case FADKV_OK: return "ok";
    case FADKV_ERR_INVALID_ARG: return "invalid argument";
    case FADKV_ERR_UNSUPPORTED: return "unsupported shape";
    case FADKV_ERR_SEQUENCE: return "encode/adapt called out of order";
    case FADKV_ERR_CUDA: return "CUDA error";
    case FADKV_ERR_WORKSPACE: return "workspace too small";
    }
    return "unknown status";
}

const char* fadkv_last_error(void) { return g_last_error; }

fadkv_status fadkv_workspace_bytes(const fadkv_params* p, size_t* bytes)
{
    if (!bytes) return FADKV_ERR_INVALID_ARG;
    const fadkv_status st = check_params(p);
    if (st != FADKV_OK) return st;
    *bytes = make_layout(*p).total;
    return FADKV_OK;
}

fadkv_status fadkv_dict_create(const fadkv_params* p, void* atoms, int32_t* usage, const float* delta,
                               void* workspace, size_t workspace_bytes, fadkv_dict* out)
{
    if (!out) return FADKV_ERR_INVALID_ARG;
    *out = nullptr;
    const fadkv_status st = check_params(p);
    if (st != FADKV_OK) return st;
    if (!atoms || !usage || !delta || !workspace) return FADKV_ERR_INVALID_ARG;
    if (!aligned(atoms, 16) || !aligned(usage, 4) || !aligned(workspace, kAlign)) return FADKV_ERR_INVALID_ARG;
    for (int g = 0; g < p->num_dicts; ++g)
        if (!(delta[g] >= 0.f)) return FADKV_ERR_INVALID_ARG;
    const Layout L = make_layout(*p);
    if (workspace_bytes < L.total) return FADKV_ERR_WORKSPACE;
    fadkv_dict h = new (std::nothrow) fadkv_dict_s();
    if (!h) return FADKV_ERR_INVALID_ARG;
    h->p = *p;
    h->sh = Shape{p->num_dicts, p->N, p->d, p->n, p->s, p->dtype, p->lambda_abs, p->lambda_rel};
    h->L = L;
    h->atoms = atoms;
    h->usage = usage;
    h->ws = (unsigned char*)workspace;
    h->ws_bytes = workspace_bytes;
    memset(&h->delta, 0, sizeof(h->delta));
    for (int g = 0; g < p->num_dicts; ++g) h->delta.v[g] = delta[g];
    h->pending = false;
    h->pending_V = 0;
    h->sms = 0;
    h->seq = 0;
    h->gram_ready = false;
    h->wait_ns = 0;
    h->alpha = screen_alpha(p->n, p->N);
    h->prof_on = false;
    h->prof_mask = 0xffffffffu;
    for (int i = 0; i < FADKV_PROFILE_KERNELS; ++i) {
        h->launches[i] = 0;
        h->ms[i] = 0.0;
    }
    *out = h;
    return FADKV_OK;
}

fadkv_status fadkv_dict_destroy(fadkv_dict h)
{
    if (!h) return FADKV_ERR_INVALID_ARG;
    for (auto& r : h->prof_pending) {
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    for (auto e : h->prof_free) cudaEventDestroy(e);
    delete h;
    return FADKV_OK;
}

fadkv_status fadkv_dict_refresh(fadkv_dict h, void* stream)
{
    if (!h) return FADKV_ERR_INVALID_ARG;
    if (fault_injected()) {
        set_error("fadkv_dict_refresh", cudaErrorLaunchFailure);
        return FADKV_ERR_CUDA;
    }
    if (!h->L.gram) return FADKV_OK;
    const cudaError_t e = build_gram(h, (cudaStream_t)stream);
    if (e != cudaSuccess) {
        set_error("fadkv_dict_refresh", e);
        return FADKV_ERR_CUDA;
    }
    return FADKV_OK;
}

fadkv_status fadkv_profile_enable(fadkv_dict h, int32_t enable)
{
    if (!h) return FADKV_ERR_INVALID_ARG;
    h->prof_on = enable != 0;
    return FADKV_OK;
}

fadkv_status fadkv_profile_select(fadkv_dict h, uint32_t class_mask)
{
    if (!h) return FADKV_ERR_INVALID_ARG;
    h->prof_mask = class_mask;
    return FADKV_OK;
}

fadkv_status fadkv_profile_read(fadkv_dict h, int64_t* launches, double* ms, int32_t reset)
{
    if (!h) return FADKV_ERR_INVALID_ARG;
    cudaError_t err = cudaSuccess;
    for (auto& r : h->prof_pending) {
        float t = 0.f;
        cudaError_t e = cudaEventSynchronize(r.stop);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&t, r.start, r.stop);
        if (e == cudaSuccess) h->ms[r.cls] += (double)t;
        else if (err == cudaSuccess) err = e;
        h->prof_free.push_back(r.start);
        h->prof_free.push_back(r.stop);
    }
    h->prof_pending.clear();
    for (int i = 0; i < FADKV_PROFILE_KERNELS; ++i) {
        if (launches) launches[i] = h->launches[i];
        if (ms) ms[i] = h->ms[i];
        if (reset) {
            h->launches[i] = 0;
            h->ms[i] = 0.0;
        }
    }
    if (err != cudaSuccess) {
        set_error("fadkv_profile_read", err);
        return FADKV_ERR_CUDA;
    }
    return FADKV_OK;
}

fadkv_status fadkv_encode(fadkv_dict h, const void* x, int32_t V, int32_t* idx, float* coef, float* relres,
                          void* stream)
{
    if (!h) return FADKV_ERR_INVALID_ARG;
    if (V < 0 || V > h->p.max_batch) return FADKV_ERR_INVALID_ARG;
    if (V > 0 && (!x || !idx || !coef || !relres)) return FADKV_ERR_INVALID_ARG;
    if (V > 0 && (!aligned(x, 16) || !aligned(idx, 4) || !aligned(coef, 4) || !aligned(relres, 4)))
        return FADKV_ERR_INVALID_ARG;
    if (h->pending) return FADKV_ERR_SEQUENCE;
    if (fault_injected()) {
        set_error("fadkv_encode", cudaErrorLaunchFailure);
        return FADKV_ERR_CUDA;
    }
    cudaStream_t st = (cudaStream_t)stream;
    if (V > 0 && h->L.gram && !h->gram_ready) {
        const cudaError_t e = build_gram(h, st);
        if (e != cudaSuccess) {
            set_error("fadkv_encode", e);
            return FADKV_ERR_CUDA;
        }
    }
    const int chunk = h->L.chunk;
    for (int v0 = 0; v0 < V; v0 += chunk) {
        const int Vc = (V - v0 < chunk) ? V - v0 : chunk;
        cudaError_t e = run_screen(h, x, V, v0, Vc, nullptr, st, h->p.n);
        if (e == cudaSuccess && h->L.gram) {
            int32_t* pool = (int32_t*)(h->ws + h->L.pool);
            float* pool_r = (float*)(h->ws + h->L.pool_r);
            GreedyArgs fa = greedy_args(h, x, V, v0, Vc);
            e = traced(h, FADKV_K_TOPN, st, [&] {
                return launch_pool_fixup(h->sh, fa, pool, pool_r, (const uint32_t*)(h->ws + h->L.slow), h->seq,
                                         h->sms, st);
            });
            if (e == cudaSuccess) {
                GramGreedyArgs ga;
                ga.atoms = (const __half*)h->atoms;
                ga.x = (const __half*)x;
                ga.pool = pool;
                ga.pool_r = pool_r;
                ga.gram = gram_ptr(h);
                ga.gdiag = gdiag_ptr(h);
                ga.idx = idx;
                ga.coef = coef;
                ga.relres = relres;
                ga.counters = counters(h);
                ga.V = V;
                ga.v0 = v0;
                ga.Vc = Vc;
                e = traced(h, FADKV_K_GREEDY, st, [&] { return launch_greedy_gram(h->sh, ga, st); });
            }
        } else if (e == cudaSuccess) {
            // FP32-pipe greedy: binary32 dictionaries, atoms not screened on
            // the tensor cores, or shapes beyond the Gram kernel's (n > 512
            // or s > 16); it takes the selection's pool where there is one
            GreedyArgs a = greedy_args(h, x, V, v0, Vc);
            a.idx = idx;
            a.coef = coef;
            a.relres = relres;
            e = traced(h, FADKV_K_GREEDY, st, [&] { return launch_greedy(h->sh, a, st); });
        }
        if (e != cudaSuccess) {
            set_error("fadkv_encode", e);
            return FADKV_ERR_CUDA;
        }
    }
    h->pending = true;
    h->pending_V = V;
    return FADKV_OK;
}

fadkv_status fadkv_encode_pl(fadkv_dict h, const void* x, int32_t V, int32_t* idx, float* coef,
                             float* relres, void* stream)
{
    if (!h) return FADKV_ERR_INVALID_ARG;
    if (V < 0 || V > h->p.max_batch) return FADKV_ERR_INVALID_ARG;
    if (V > 0 && (!x || !idx || !coef || !relres)) return FADKV_ERR_INVALID_ARG;
    if (V > 0 && (!aligned(x, 16) || !aligned(idx, 4) || !aligned(coef, 4) || !aligned(relres, 4)))
        return FADKV_ERR_INVALID_ARG;
    if (h->pending) return FADKV_ERR_SEQUENCE;
    if (fault_injected()) {
        set_error("fadkv_encode_pl", cudaErrorLaunchFailure);
        return FADKV_ERR_CUDA;
    }
    cudaStream_t st = (cudaStream_t)stream;
    Shape sh = h->sh;
    sh.n = h->p.s;                                     // the Top-s set
    const int chunk = h->L.chunk;
    for (int v0 = 0; v0 < V; v0 += chunk) {
        const int Vc = (V - v0 < chunk) ? V - v0 : chunk;
        cudaError_t e = run_screen(h, x, V, v0, Vc, nullptr, st, h->p.s);
        PlArgs pa;
        pa.atoms = h->atoms;
        pa.x = x;
        pa.pool = nullptr;
        pa.cand = cand_buf(h);
        pa.cand_count = cand_count_buf(h);
        pa.cap = h->L.cap;
        pa.idx = idx;
        pa.coef = coef;
        pa.relres = relres;
        pa.counters = counters(h);
        pa.V = V;
        pa.v0 = v0;
        pa.Vc = Vc;
        if (e == cudaSuccess && h->L.tc) {
            int32_t* pool = (int32_t*)(h->ws + h->L.pool);
            float* pool_r = (float*)(h->ws + h->L.pool_r);
            GreedyArgs fa = greedy_args(h, x, V, v0, Vc);
            e = traced(h, FADKV_K_TOPN, st, [&] {
                return launch_pool_fixup(sh, fa, pool, pool_r, (const uint32_t*)(h->ws + h->L.slow), h->seq, h->sms,
                                         st);
            });
            pa.pool = pool;
        }
        if (e == cudaSuccess) e = traced(h, FADKV_K_GREEDY, st, [&] { return launch_pl_fit(h->sh, pa, st); });
        if (e != cudaSuccess) {
            set_error("fadkv_encode_pl", e);
            return FADKV_ERR_CUDA;
        }
    }
    h->pending = true;
    h->pending_V = V;
    return FADKV_OK;
}

namespace {

fadkv_status adapt_call(const char* name, fadkv_dict h, const void* x, int32_t V, const int32_t* idx,
                        const float* coef, const float* relres, int32_t* repl_id, float* repl_coef, void* stream,
                        int append)
{
    if (!h) return FADKV_ERR_INVALID_ARG;
    if (V < 0 || V > h->p.max_batch) return FADKV_ERR_INVALID_ARG;
    if (V > 0 && (!x || !idx || !coef || !relres || !repl_id || !repl_coef)) return FADKV_ERR_INVALID_ARG;
    if (V > 0 && (!aligned(x, 16) || !aligned(repl_id, 4) || !aligned(repl_coef, 4)))
        return FADKV_ERR_INVALID_ARG;
    if (!h->pending || h->pending_V != V) return FADKV_ERR_SEQUENCE;
    if (fault_injected()) {
        set_error(name, cudaErrorLaunchFailure);
        return FADKV_ERR_CUDA;
    }
    AdaptArgs a;
    a.atoms = h->atoms;
    a.usage = h->usage;
    a.x = x;
    a.idx = idx;
    a.coef = coef;
    a.relres = relres;
    a.repl_id = repl_id;
    a.repl_coef = repl_coef;
    a.inactive = (int32_t*)(h->ws + h->L.inactive);
    a.flagged = (int32_t*)(h->ws + h->L.flagged);
    a.nrep = (int32_t*)(h->ws + h->L.nrep);
    a.counters = counters(h);
    a.V = V;
    a.append = append;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = traced(h, FADKV_K_ADAPT, st, [&] { return launch_adapt(h->sh, a, h->delta, st); });
    if (e == cudaSuccess) h->launches[FADKV_K_ADAPT] += adapt_launches(h->sh, V) - 1;
    // the rows and columns of the atoms just written (none, if the Gram
    // matrices are not built yet: the build reads the atoms as they stand)
    if (e == cudaSuccess && h->L.gram && h->gram_ready)
        e = traced(h, FADKV_K_GRAM, st, [&] {
            return launch_gram_update(h->sh, h->atoms, a.inactive, a.nrep, h->p.N, gram_ptr(h), gdiag_ptr(h), h->sms,
                                      st);
        });
    if (e != cudaSuccess) {
        set_error(name, e);
        return FADKV_ERR_CUDA;
    }
    h->pending = false;
    h->pending_V = 0;
    return FADKV_OK;
}

}  // namespace

fadkv_status fadkv_adapt(fadkv_dict h, const void* x, int32_t V, const int32_t* idx, const float* coef,
                         const float* relres, int32_t* repl_id, float* repl_coef, void* stream)
{
    return adapt_call("fadkv_adapt", h, x, V, idx, coef, relres, repl_id, repl_coef, stream, 0);
}

fadkv_status fadkv_adapt_append(fadkv_dict h, const void* x, int32_t V, const int32_t* idx, const float* coef,
                                const float* relres, int32_t* repl_id, float* repl_coef, void* stream)
{
    return adapt_call("fadkv_adapt_append", h, x, V, idx, coef, relres, repl_id, repl_coef, stream, 1);
}

fadkv_status fadkv_reconstruct(fadkv_dict h, int32_t V, const int32_t* idx, const float* coef,
                               const int32_t* repl_id, const float* repl_coef, float* xhat, void* stream)
{
    if (!h) return FADKV_ERR_INVALID_ARG;
    if (V < 0 || V > h->p.max_batch) return FADKV_ERR_INVALID_ARG;
    if (V > 0 && (!idx || !coef || !xhat)) return FADKV_ERR_INVALID_ARG;
    if ((repl_id == nullptr) != (repl_coef == nullptr)) return FADKV_ERR_INVALID_ARG;
    if (fault_injected()) {
        set_error("fadkv_reconstruct", cudaErrorLaunchFailure);
        return FADKV_ERR_CUDA;
    }
    cudaStream_t st = (cudaStream_t)stream;
    const cudaError_t e = traced(h, FADKV_K_RECONSTRUCT, st, [&] {
        return launch_reconstruct(h->sh, h->atoms, V, idx, coef, repl_id, repl_coef, xhat, st);
    });
    if (e != cudaSuccess) {
        set_error("fadkv_reconstruct", e);
        return FADKV_ERR_CUDA;
    }
    return FADKV_OK;
}

fadkv_status fadkv_dict_stats(fadkv_dict h, int64_t* host_out, void* stream)
{
    if (!h || !host_out) return FADKV_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(host_out, counters(h),
                                    sizeof(long long) * kCntFields * (size_t)h->p.num_dicts,
                                    cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        set_error("fadkv_dict_stats", e);
        return FADKV_ERR_CUDA;
    }
    return FADKV_OK;
}

fadkv_status fadkv_debug_pool(fadkv_dict h, const void* x, int32_t V, int32_t* pool, float* pool_r,
                              void* stream)
{
    if (!h) return FADKV_ERR_INVALID_ARG;
    if (V < 0 || V > h->p.max_batch) return FADKV_ERR_INVALID_ARG;
    if (V > 0 && (!x || !pool || !aligned(x, 16))) return FADKV_ERR_INVALID_ARG;
    if (fault_injected()) {
        set_error("fadkv_debug_pool", cudaErrorLaunchFailure);
        return FADKV_ERR_CUDA;
    }
    cudaStream_t st = (cudaStream_t)stream;
    const int chunk = h->L.chunk;
    for (int v0 = 0; v0 < V; v0 += chunk) {
        const int Vc = (V - v0 < chunk) ? V - v0 : chunk;
        cudaError_t e = run_screen(h, x, V, v0, Vc, nullptr, st, h->p.n);
        if (e == cudaSuccess) {
            GreedyArgs a = greedy_args(h, x, V, v0, Vc);
            a.pool_out = pool;
            a.pool_r_out = pool_r;
            e = launch_greedy(h->sh, a, st);
        }
        if (e != cudaSuccess) {
            set_error("fadkv_debug_pool", e);
            return FADKV_ERR_CUDA;
        }
    }
    return FADKV_OK;
}

fadkv_status fadkv_debug_wait_limit(fadkv_dict h, uint64_t limit_ns)
{
    if (!h) return FADKV_ERR_INVALID_ARG;
    h->wait_ns = (unsigned long long)limit_ns;
    return FADKV_OK;
}

fadkv_status fadkv_debug_wait_probe(fadkv_dict h, uint64_t limit_ns, void* stream)
{
    if (!h || limit_ns == 0 || limit_ns > 10ull * 1000 * 1000 * 1000) return FADKV_ERR_INVALID_ARG;
    if (fault_injected()) {
        set_error("fadkv_debug_wait_probe", cudaErrorLaunchFailure);
        return FADKV_ERR_CUDA;
    }
    unsigned long long* status = (unsigned long long*)&counters(h)[kCntStatus];
    const cudaError_t e = launch_wait_probe(status, (unsigned long long)limit_ns, (cudaStream_t)stream);
    if (e != cudaSuccess) {
        set_error("fadkv_debug_wait_probe", e);
        return FADKV_ERR_CUDA;
    }
    return FADKV_OK;
}

fadkv_status fadkv_debug_scores(fadkv_dict h, const void* x, int32_t V, float* scores, void* stream)
{
    if (!h) return FADKV_ERR_INVALID_ARG;
    if (V < 0 || V > h->p.max_batch) return FADKV_ERR_INVALID_ARG;
    if (V > 0 && (!x || !scores || !aligned(x, 16))) return FADKV_ERR_INVALID_ARG;
    if (V > h->L.chunk) return FADKV_ERR_INVALID_ARG;   // one pass: [G][V][N] output
    if (fault_injected()) {
        set_error("fadkv_debug_scores", cudaErrorLaunchFailure);
        return FADKV_ERR_CUDA;
    }
    if (V == 0) return FADKV_OK;
    const cudaError_t e = run_screen(h, x, V, 0, V, scores, (cudaStream_t)stream, h->p.n);
    if (e != cudaSuccess) {
        set_error("fadkv_debug_scores", e);
        return FADKV_ERR_CUDA;
    }
    return FADKV_OK;
}

}  // extern "C"

fadkv_status fadkv_store_codes(int32_t G, int32_t B, int32_t H, int32_t s, int32_t N, const int32_t* idx,
                               const float* coef, const int32_t* repl_id, const float* repl_coef,
                               const int32_t* pos, uint32_t* cache, int32_t Tmax, void* stream)
{
    if (G < 0 || B < 0 || H < 1 || s < 0 || N < 1 || Tmax < 1) return FADKV_ERR_INVALID_ARG;
    if (N > (1 << FADKV_PACK_ID_BITS) || s > FADKV_MAX_S) return FADKV_ERR_UNSUPPORTED;
    if ((repl_id == nullptr) != (repl_coef == nullptr)) return FADKV_ERR_INVALID_ARG;
    const long long work = (long long)G * B * H;
    if (work > 0 && (!idx || !coef || !pos || !cache)) return FADKV_ERR_INVALID_ARG;
    if (work > 0 && (!aligned(idx, 4) || !aligned(coef, 4) || !aligned(pos, 4) || !aligned(cache, 4) ||
                     (repl_id && (!aligned(repl_id, 4) || !aligned(repl_coef, 4)))))
        return FADKV_ERR_INVALID_ARG;
    if (fault_injected()) {
        set_error("fadkv_store_codes", cudaErrorLaunchFailure);
        return FADKV_ERR_CUDA;
    }
    StoreArgs a;
    a.G = G;
    a.B = B;
    a.H = H;
    a.s = s;
    a.N = N;
    a.Tmax = Tmax;
    a.idx = idx;
    a.coef = coef;
    a.repl_id = repl_id;
    a.repl_coef = repl_coef;
    a.pos = pos;
    a.cache = cache;
    const cudaError_t e = launch_store_codes(a, (cudaStream_t)stream);
    if (e != cudaSuccess) {
        set_error("fadkv_store_codes", e);
        return FADKV_ERR_CUDA;
    }
    return FADKV_OK;
}

namespace {

fadkv_status attend_check(const fadkv_attn_params* p)
{
    if (!p) return FADKV_ERR_INVALID_ARG;
    if (p->layers < 0 || p->B < 0 || p->Hq < 1 || p->Hkv < 1 || p->Hq % p->Hkv != 0 || p->s < 0 ||
        p->N < 1 || p->Tmax < 0 || !(p->scale == p->scale) || p->dict_stride < 0 || p->cache_stride < 0)
        return FADKV_ERR_INVALID_ARG;
    if (p->dtype != FADKV_F16 && p->dtype != FADKV_F32) return FADKV_ERR_INVALID_ARG;
    if (!attend_supported(p->d, p->N, p->s)) return FADKV_ERR_UNSUPPORTED;
    return FADKV_OK;
}

}  // namespace

fadkv_status fadkv_attend_workspace_bytes(const fadkv_attn_params* p, size_t* bytes)
{
    const fadkv_status st = attend_check(p);
    if (st != FADKV_OK) return st;
    if (!bytes) return FADKV_ERR_INVALID_ARG;
    *bytes = attend_workspace_bytes(p->layers, p->B, p->Hq, p->N, p->dtype);
    return FADKV_OK;
}

fadkv_status fadkv_attend(const fadkv_attn_params* p, const void* dict_k, const void* dict_v,
                          const uint32_t* cache_k, const uint32_t* cache_v, const int32_t* lengths,
                          const float* q, float* out, void* workspace, size_t workspace_bytes, void* stream)
{
    const fadkv_status st = attend_check(p);
    if (st != FADKV_OK) return st;
    const size_t need = attend_workspace_bytes(p->layers, p->B, p->Hq, p->N, p->dtype);
    if (workspace_bytes < need || (need > 0 && !workspace)) return FADKV_ERR_WORKSPACE;
    if (need > 0 && !aligned(workspace, 256)) return FADKV_ERR_INVALID_ARG;
    const long long work = (long long)p->layers * p->B;
    if (work > 0 && (!dict_k || !dict_v || !cache_k || !cache_v || !lengths || !q || !out))
        return FADKV_ERR_INVALID_ARG;
    if (work > 0 && (!aligned(dict_k, 16) || !aligned(dict_v, 16) || p->dict_stride % 8 != 0 ||
                     !aligned(cache_k, 4) || !aligned(cache_v, 4) || !aligned(lengths, 4) || !aligned(q, 16) ||
                     !aligned(out, 4)))
        return FADKV_ERR_INVALID_ARG;
    if (fault_injected()) {
        set_error("fadkv_attend", cudaErrorLaunchFailure);
        return FADKV_ERR_CUDA;
    }
    AttendArgs a;
    a.dict_k = dict_k;
    a.dict_v = dict_v;
    a.dict_stride = p->dict_stride;
    a.cache_k = cache_k;
    a.cache_v = cache_v;
    a.cache_stride = p->cache_stride;
    a.lengths = lengths;
    a.q = q;
    a.out = out;
    a.L = p->layers;
    a.B = p->B;
    a.Hq = p->Hq;
    a.Hkv = p->Hkv;
    a.d = p->d;
    a.N = p->N;
    a.s = p->s;
    a.Tmax = p->Tmax;
    a.dtype = p->dtype;
    a.scale = p->scale;
    a.Npad = attend_npad(p->N);
    a.U = nullptr;
    a.Whi = a.Wlo = nullptr;
    a.wunscale = nullptr;
    if (need > 0) attend_bind_workspace(a, workspace);
    const cudaError_t e = launch_attend(a, (cudaStream_t)stream);
    if (e != cudaSuccess) {
        set_error("fadkv_attend", e);
        return FADKV_ERR_CUDA;
    }
    return FADKV_OK;
}
