// Host runtime behind the C ABI declared in include/tkv.h: context, device
// pools, pinned host stores, page tables, the step protocol, the per-layer T1
// prefetch pipeline (copy stream) and the re-tier driver.
//
// Method: "Not All Thoughts Need HBM: Semantics-Aware Memory Hierarchy for
// LLM Reasoning" (gist.science summary; fugumt.com abstract).  The per-layer
// T1 fetch before each attention step follows "Zero-approximation-error
// offloading"; the re-tier every Delta steps and the delta prefetch of newly
// promoted rows follow "System implementation"; the tier counts and the
// protected set follow "Four-tier classification".
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include <sys/mman.h>
#include <sys/syscall.h>
#include <unistd.h>

#include "../../include/tkv.h"
#include "tkv_internal.cuh"

using namespace tkv;

// A large pinned host store (T1 rows, T2 masters, host T2 records): either a registered
// anonymous mapping backed by transparent huge pages, or a cudaHostAlloc block.
struct HostStore {
    void* ptr = nullptr;      // what the library uses
    void* map = nullptr;      // the mapping (huge-page arena), else null
    size_t map_len = 0;
    size_t huge_bytes = 0;    // bytes of the store backed by huge pages (from /proc/self/smaps)
};

struct tkv_ctx {
    tkv_config cfg{};
    int L = 0, B = 0, Hq = 0, Hkv = 0, G = 0, d = 0, Nmax = 0, S0 = 0, S1 = 0, S2 = 0;
    int64_t ppm[4] = {0, 0, 0, 0};
    int device = 0;
    cudaStream_t compute = nullptr, copy = nullptr, copy2 = nullptr;
    bool own_compute = false, own_copy = false;
    cudaEvent_t ev_split = nullptr;
    static constexpr int kCopyLanes = 4;                  // streams of the multi-engine T1 transport
    cudaStream_t copyx[kCopyLanes - 1] = {nullptr, nullptr, nullptr};
    cudaEvent_t ev_join[kCopyLanes - 1] = {nullptr, nullptr, nullptr};

    // device
    __nv_bfloat16* k0v0 = nullptr;
    __nv_bfloat16* stage = nullptr;
    uint8_t* t2 = nullptr;                   // T2 pool (HBM), or the device view of the host pool
    uint8_t* t2_host = nullptr;              // TKV_T2_HOST: the pinned host pool
    uint8_t* stage2 = nullptr;               // TKV_T2_HOST: T2 staging ring [2][2][B][Hkv][S2][d+16]
    uint8_t *tier = nullptr, *new_tier = nullptr, *forced = nullptr;
    int32_t *slot = nullptr, *new_slot = nullptr, *free_scratch = nullptr;
    float* s = nullptr;
    uint32_t* rl_loc = nullptr;
    int32_t *rl_pos = nullptr, *rl_count = nullptr;
    float* g = nullptr;
    float *part = nullptr, *zs = nullptr;    // attention scratch: item partials, logits
    int32_t *t0_free = nullptr, *t0_top = nullptr;
    int4 *moves_now = nullptr, *moves_delta = nullptr;
    RetierOut* outp = nullptr;
    RetierParams* params = nullptr;
    int32_t* err = nullptr;
    int32_t* pos_n = nullptr;                // [B] committed positions (device copy of N)

    // pinned host
    HostStore hs_h1, hs_h2m, hs_t2;                   // the large stores
    int host_numa = -1;                               // NUMA node the large stores are bound to, or -1
    __nv_bfloat16 *h1 = nullptr, *h2m = nullptr;      // host pointers
    __nv_bfloat16 *d_h1 = nullptr, *d_h2m = nullptr;  // device views
    RetierOut* h_outp = nullptr;
    RetierParams* h_params = nullptr;
    int32_t* h_err = nullptr;

    cudaEvent_t ev_t1[2] = {nullptr, nullptr}, ev_attn[2] = {nullptr, nullptr}, ev_retier = nullptr;

    // host mirrors (identical to the device values after every call)
    int N = 0;                         // committed positions
    std::vector<int> count[4];         // tokens per tier, per sequence
    std::vector<int> R;                // retained positions, per sequence
    int hw1 = 0;                       // T1 slots streamed per layer
    int hw2 = 0;                       // T2 slots streamed per layer (TKV_T2_HOST)
    int64_t step = 0, retiers = 0;

    // protocol state
    int open_n = 0, appended = 0, decoded = 0;
    std::vector<char> prefetched;
    // decode-token rows appended but not yet written (the layer's attention kernel writes them)
    std::vector<const void*> pend_k, pend_v;

    // CUDA-graph decode steps
    bool capturing = false;
    cudaStream_t cap_stream = nullptr, cap_saved_compute = nullptr;
    cudaEvent_t ev_fork = nullptr;        // recorded on the capture stream when the capture opens
    bool copy_joined = false;             // the copy stream has joined the capture
    bool copyx_joined[3] = {false, false, false};   // and so have the helper copy streams
    bool attn_in_capture[2] = {false, false};
    int cap_rows = 0;                     // rows per group the captured launch geometry covers
    struct Saved {
        int N;
        std::vector<int> count0, R;
        int64_t step, launches;
        tkv_stats st;
    } cap_saved;
    cudaGraphExec_t graph_exec = nullptr;
    int graph_steps_left = 0;
    int64_t graph_launches = 0, graph_t1_bytes = 0, graph_t2_bytes = 0;
    int delta_max = 0;                 // pending delta moves (max over sequences), 0 = none
    int delta_chunk = 1;               // layers per delta launch (about 1 MB of rows per launch)
    std::vector<char> delta_done;      // per layer: its delta is enqueued (valid while delta_max > 0)

    int resident = 1;                  // attention CTAs resident on the device at once
    int last_splits = 0;

    // timing (tkv_profile_begin / tkv_profile_end): kinds 0 attention main kernel, 1 T1 copy,
    // 2 delta, 3 attention combine kernel
    static constexpr int kProfKinds = 4;
    static constexpr int kProfPairs = 16384;
    std::vector<cudaEvent_t> prof_ev[kProfKinds];   // 2 per pair, created on first use
    int prof_used[kProfKinds] = {0, 0, 0, 0};
    double prof_bytes[kProfKinds] = {0, 0, 0, 0};
    bool profiling = false;
    int64_t launches = 0;
    tkv_status status = TKV_OK;
    int cuda_error = 0, cuda_error_line = 0;   // the first failing CUDA call (diagnostics)
    // host-side fault injection (TKV_FAULT_INJECT, read at creation; a test hook)
    bool inject_hostalloc = false;
    int64_t inject_at = 0, inject_count = 0;
    tkv_stats st{};
    size_t hbm_alloc = 0, host_alloc = 0;
};

namespace {

struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) cudaSetDevice(dev);
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

tkv_status fail(tkv_ctx* c, tkv_status s) {
    if (c && c->status == TKV_OK) c->status = s;
    return s;
}

// The first failing CUDA call: its error code and the source line of the call.
tkv_status fail_cuda(tkv_ctx* c, cudaError_t e, int line) {
    if (c && c->status == TKV_OK) {
        c->cuda_error = (int)e;
        c->cuda_error_line = line;
    }
    return fail(c, TKV_ECUDA);
}

// A checked CUDA call made on behalf of a context: the first failure poisons the context.
// With fault injection on, the inject_at-th checked call is reported as failed
// (cudaErrorUnknown) after it ran, so no device work goes wrong.
#define CK(x)                                                                              \
    do {                                                                                   \
        cudaError_t e_ = (x);                                                              \
        if (e_ == cudaSuccess && ctx->inject_at > 0 && ++ctx->inject_count == ctx->inject_at) \
            e_ = cudaErrorUnknown;                                                         \
        if (e_ != cudaSuccess) {                                                           \
            (void)cudaGetLastError();                                                      \
            return fail_cuda(ctx, e_, __LINE__);                                           \
        }                                                                                  \
    } while (0)

#define CHECK_CTX()                                        \
    do {                                                   \
        if (!ctx) return TKV_EINVAL;                       \
        if (ctx->status != TKV_OK) return TKV_ESTATE;      \
    } while (0)

int64_t to_ppm(float r) { return (int64_t)std::llround((double)r * 1000000.0); }
int64_t count_of(int64_t ppm, int64_t n) { return ppm * n / 1000000; }

template <typename T>
cudaError_t dalloc(tkv_ctx* c, T** p, size_t n) {
    if (n == 0) {
        *p = nullptr;
        return cudaSuccess;
    }
    cudaError_t e = cudaMalloc((void**)p, n * sizeof(T));
    if (e == cudaSuccess) c->hbm_alloc += n * sizeof(T);
    return e;
}

template <typename T>
cudaError_t halloc(tkv_ctx* c, T** p, size_t n) {
    if (n == 0 || c->inject_hostalloc) {
        *p = nullptr;
        return n == 0 ? cudaSuccess : cudaErrorMemoryAllocation;
    }
    cudaError_t e = cudaHostAlloc((void**)p, n * sizeof(T), cudaHostAllocMapped | cudaHostAllocPortable);
    if (e == cudaSuccess) c->host_alloc += n * sizeof(T);
    return e;
}

// ------------------------------------------------------------ host arenas
// The T1 store of a large configuration is tens of GB of pinned host memory that the copy
// engine reads once per decode step, so the rate at which the copy engine reads it sets the
// step time.  Backed by base pages (what cudaHostAlloc returns), a store of tens of GB needs
// more DMA translations than the host link keeps mapped, and the rate can drop well below the
// link's (measured on GB300 guests: a 43 GB store read per layer at 211 GB/s fresh, falling
// to 15-110 GB/s once host memory had been freed and reused; with huge pages it held).  So a
// store of 1 GiB or more is an anonymous mapping aligned to the transparent-huge-page size,
// advised MADV_HUGEPAGE, bound to the host NUMA node closest to the GPU when the host has
// several, populated, and registered with CUDA (mapped, portable).  If a step fails, the store
// falls back to cudaHostAlloc.

size_t thp_size() {
    size_t v = 0;
    if (FILE* f = std::fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
        unsigned long long x = 0;
        if (std::fscanf(f, "%llu", &x) == 1) v = (size_t)x;
        std::fclose(f);
    }
    return v >= 4096 && (v & (v - 1)) == 0 ? v : (size_t)2 << 20;
}

// Online NUMA nodes of the host (1 when unknown).
int online_nodes() {
    int n = 1;
    if (FILE* f = std::fopen("/sys/devices/system/node/online", "r")) {
        char buf[256] = {0};
        if (std::fgets(buf, sizeof(buf), f)) {
            // "0", "0-1", "0,2-3": count the ids
            n = 0;
            const char* p = buf;
            while (*p) {
                char* e = nullptr;
                const long a = std::strtol(p, &e, 10);
                if (e == p) break;
                long b = a;
                p = e;
                if (*p == '-') {
                    b = std::strtol(p + 1, &e, 10);
                    p = e;
                }
                n += (int)(b - a + 1);
                if (*p == ',') ++p;
                else break;
            }
            if (n < 1) n = 1;
        }
        std::fclose(f);
    }
    return n;
}

// Sum of AnonHugePages over the mappings inside [addr, addr + len), in bytes (0 when unknown).
size_t huge_bytes_of(const void* addr, size_t len) {
    FILE* f = std::fopen("/proc/self/smaps", "r");
    if (!f) return 0;
    char line[512];
    bool in = false;
    size_t out = 0;
    const unsigned long long a = (unsigned long long)(uintptr_t)addr, b = a + len;
    while (std::fgets(line, sizeof(line), f)) {
        unsigned long long lo = 0, hi = 0;
        if (std::sscanf(line, "%llx-%llx ", &lo, &hi) == 2 && std::strchr(line, '-') < std::strchr(line, ' ')) {
            in = lo >= a && hi <= b;
            continue;
        }
        unsigned long long kb = 0;
        if (in && std::sscanf(line, "AnonHugePages: %llu kB", &kb) == 1) out += (size_t)kb * 1024;
    }
    std::fclose(f);
    return out;
}

// Maps `len` bytes (a multiple of `align`) aligned to `align` and populates them with huge
// pages (bound to NUMA node `numa` if >= 0).  Returns null on failure.
char* map_unit(size_t len, size_t align, int numa) {
    const size_t unit = len;
    void* m = mmap(nullptr, len + align, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
    if (m == MAP_FAILED) return nullptr;
    char* p = (char*)(((uintptr_t)m + align - 1) / align * align);
    if (p > (char*)m) munmap(m, (size_t)(p - (char*)m));
    char* end = (char*)m + len + align;
    if (p + unit < end) munmap(p + unit, (size_t)(end - (p + unit)));
    if (numa >= 0 && numa < 1024) {
        unsigned long mask[16] = {0};
        mask[numa / 64] = 1ul << (numa % 64);
        (void)syscall(SYS_mbind, p, unit, 2 /* MPOL_BIND */, mask, 1024ul, 0u);   // a refusal keeps the default
    }
    madvise(p, unit, MADV_HUGEPAGE);
    if (madvise(p, unit, 23 /* MADV_POPULATE_WRITE */) != 0) {
        const long pg = sysconf(_SC_PAGESIZE) > 0 ? sysconf(_SC_PAGESIZE) : 4096;
        for (size_t o = 0; o < unit; o += (size_t)pg) ((volatile char*)p)[o] = 0;
    }
    return p;
}

cudaError_t harena_alloc(tkv_ctx* c, HostStore& hs, size_t bytes) {
    hs = HostStore();
    if (bytes == 0) return cudaSuccess;
    if (c->inject_hostalloc) return cudaErrorMemoryAllocation;
    const bool arena = c->cfg.host_alloc == TKV_HOST_HUGE_ARENA ||
                       (c->cfg.host_alloc == TKV_HOST_AUTO && bytes >= ((size_t)1 << 30));
    if (arena) {
        const size_t huge = thp_size();
        const size_t body = (bytes + huge - 1) / huge * huge;
        char* p = map_unit(body, huge, c->host_numa);
        if (p && cudaHostRegister(p, body, cudaHostRegisterMapped | cudaHostRegisterPortable) == cudaSuccess) {
            hs.ptr = p;
            hs.map = p;
            hs.map_len = body;
            hs.huge_bytes = std::min(huge_bytes_of(p, body), body);
            c->host_alloc += body;
            return cudaSuccess;
        }
        (void)cudaGetLastError();
        if (p) munmap(p, body);
    }
    cudaError_t e = cudaHostAlloc(&hs.ptr, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e == cudaSuccess) c->host_alloc += bytes;
    else hs.ptr = nullptr;
    return e;
}

void harena_free(HostStore& hs) {
    if (!hs.ptr) return;
    if (hs.map) {
        cudaHostUnregister(hs.ptr);
        munmap(hs.map, hs.map_len);
    } else {
        cudaFreeHost(hs.ptr);
    }
    hs = HostStore();
}

int protected_count(int N, int prompt, int sinks, int W) {
    const int a = std::min(N, std::max(prompt, sinks));
    const int w0 = std::max(0, N - W);
    return a + (N - std::max(a, w0));
}

size_t row_bytes_bf16(const tkv_ctx* c) { return (size_t)2 * c->Hkv * c->d * 2; }   // K+V, one layer

void free_all(tkv_ctx* c) {
    cudaFree(c->k0v0); cudaFree(c->stage); cudaFree(c->stage2);
    if (c->t2_host) harena_free(c->hs_t2);
    else cudaFree(c->t2);
    cudaFree(c->tier); cudaFree(c->new_tier); cudaFree(c->forced);
    cudaFree(c->slot); cudaFree(c->new_slot); cudaFree(c->free_scratch);
    cudaFree(c->s); cudaFree(c->rl_loc); cudaFree(c->rl_pos); cudaFree(c->rl_count);
    cudaFree(c->g); cudaFree(c->part); cudaFree(c->zs); cudaFree(c->t0_free); cudaFree(c->t0_top);
    cudaFree(c->moves_now); cudaFree(c->moves_delta); cudaFree(c->outp); cudaFree(c->params);
    cudaFree(c->err); cudaFree(c->pos_n);
    harena_free(c->hs_h1); harena_free(c->hs_h2m); cudaFreeHost(c->h_outp); cudaFreeHost(c->h_params);
    cudaFreeHost(c->h_err);
    for (int i = 0; i < 2; ++i) {
        if (c->ev_t1[i]) cudaEventDestroy(c->ev_t1[i]);
        if (c->ev_attn[i]) cudaEventDestroy(c->ev_attn[i]);
    }
    if (c->ev_retier) cudaEventDestroy(c->ev_retier);
    if (c->graph_exec) cudaGraphExecDestroy(c->graph_exec);
    if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
    if (c->ev_fork) cudaEventDestroy(c->ev_fork);
    for (auto& v : c->prof_ev)
        for (cudaEvent_t e : v) cudaEventDestroy(e);
    if (c->own_compute && c->compute) cudaStreamDestroy(c->compute);
    if (c->own_copy && c->copy) cudaStreamDestroy(c->copy);
    if (c->copy2) cudaStreamDestroy(c->copy2);
    if (c->ev_split) cudaEventDestroy(c->ev_split);
    for (int i = 0; i < tkv_ctx::kCopyLanes - 1; ++i) {
        if (c->copyx[i]) cudaStreamDestroy(c->copyx[i]);
        if (c->ev_join[i]) cudaEventDestroy(c->ev_join[i]);
    }
    (void)cudaGetLastError();
}

// Brackets of timed work: prof_open before, prof_close after (no-ops unless profiling).
bool prof_open(tkv_ctx* c, int kind, cudaStream_t st) {
    if (!c->profiling || c->prof_used[kind] >= tkv_ctx::kProfPairs) return false;
    return cudaEventRecord(c->prof_ev[kind][2 * c->prof_used[kind]], st) == cudaSuccess;
}
void prof_close(tkv_ctx* c, int kind, cudaStream_t st, double bytes) {
    cudaEventRecord(c->prof_ev[kind][2 * c->prof_used[kind] + 1], st);
    c->prof_used[kind]++;
    c->prof_bytes[kind] += bytes;
}

// Reads the device status word; returns it (0 if clear).
tkv_status read_device_status(tkv_ctx* ctx) {
    if (cudaMemcpy(ctx->h_err, ctx->err, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess) {
        (void)cudaGetLastError();
        return fail(ctx, TKV_ECUDA);
    }
    if (*ctx->h_err) return fail(ctx, (tkv_status)*ctx->h_err);
    return TKV_OK;
}

// Enqueues the delta moves left by the last re-tier for layers [l0, l1).
// Events recorded inside a capture only mark points of that capture, and a replay does
// not record them.  After a capture and after every replay they are recorded again on
// the compute stream, behind everything the replay did (copy-stream work included), so
// the eager calls that follow wait on the right work.
cudaError_t rerecord_events(tkv_ctx* ctx) {
    for (int i = 0; i < 2; ++i) {
        cudaError_t e = cudaEventRecord(ctx->ev_attn[i], ctx->compute);
        if (e == cudaSuccess) e = cudaEventRecord(ctx->ev_t1[i], ctx->compute);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

void drop_graph(tkv_ctx* ctx) {
    if (ctx->graph_exec) cudaGraphExecDestroy(ctx->graph_exec);
    ctx->graph_exec = nullptr;
    ctx->graph_steps_left = 0;
}

tkv_status enqueue_delta(tkv_ctx* ctx, int l0, int l1, cudaStream_t st) {
    if (ctx->delta_max <= 0) return TKV_OK;
    MoveArgs m{};
    m.moves = ctx->moves_delta;
    m.counts = &ctx->outp[0].n_delta;
    m.count_stride = (int)(sizeof(RetierOut) / sizeof(int32_t));
    m.k0v0 = ctx->k0v0; m.t2 = ctx->t2; m.h1 = ctx->d_h1; m.h2m = ctx->d_h2m;
    m.t1_res = ctx->cfg.t1_transport == TKV_T1_RESIDENT ? ctx->stage : nullptr;
    m.layer_begin = l0; m.layer_end = l1;
    m.L = ctx->L; m.B = ctx->B; m.Hkv = ctx->Hkv; m.d = ctx->d; m.Nmax = ctx->Nmax;
    m.S0 = ctx->S0; m.S1 = ctx->S1; m.S2 = ctx->S2;
    m.max_count = ctx->delta_max;
    int64_t n = 0;
    for (int b = 0; b < ctx->B; ++b) n += ctx->h_outp[b].n_delta;
    const int64_t bytes = n * (int64_t)(l1 - l0) * (int64_t)row_bytes_bf16(ctx);
    const bool timed = prof_open(ctx, 2, st);
    CK(launch_moves(m, st));
    if (timed) prof_close(ctx, 2, st, (double)bytes);
    ctx->launches++;
    ctx->st.h2d_bytes_delta += bytes;
    return TKV_OK;
}

// Enqueues the delta of every layer in [l0, l1) not enqueued yet, as launches over runs of
// consecutive such layers of at most `chunk` layers, and marks those layers done.
tkv_status enqueue_delta_range(tkv_ctx* ctx, int l0, int l1, int chunk, cudaStream_t st) {
    int l = l0;
    while (l < l1) {
        if (ctx->delta_done[l]) {
            ++l;
            continue;
        }
        int e = l;
        while (e < l1 && e - l < chunk && !ctx->delta_done[e]) ++e;
        tkv_status r = enqueue_delta(ctx, l, e, st);
        if (r != TKV_OK) return r;
        for (int k = l; k < e; ++k) ctx->delta_done[k] = 1;
        l = e;
    }
    return TKV_OK;
}

// Re-tier core shared by tkv_retier (ranked) and tkv_set_tiers (forced).
tkv_status run_retier(tkv_ctx* ctx, bool forced) {
    const int N = ctx->N, B = ctx->B;
    drop_graph(ctx);
    // a delta left by an earlier re-tier that no decode step has consumed yet
    if (ctx->delta_max > 0) {
        tkv_status r = enqueue_delta_range(ctx, 0, ctx->L, ctx->L, ctx->compute);
        if (r != TKV_OK) return r;
        ctx->delta_max = 0;
    }
    const int P = protected_count(N, ctx->cfg.prompt_len, ctx->cfg.num_sinks, ctx->cfg.recent_window);
    const int64_t n0 = std::max<int64_t>(P, count_of(ctx->ppm[0], N));
    const int64_t n2 = count_of(ctx->ppm[2], N);
    const int64_t n3 = count_of(ctx->ppm[3], N);
    for (int b = 0; b < B; ++b) {
        RetierParams& p = ctx->h_params[b];
        std::memset(&p, 0, sizeof(p));
        p.forced = forced ? 1 : 0;
        const int64_t t3 = ctx->count[3][b];
        const int64_t n_cand = N - P - t3;
        const int64_t e = std::min(std::max<int64_t>(n3 - t3, 0), n_cand);
        const int64_t m = n_cand - e;
        const int64_t c0 = std::min(n0 - P, m);
        const int64_t c2 = std::min(n2, m - c0);
        p.c0 = (int)c0;
        p.c2 = (int)c2;
        p.c1 = (int)(m - c0 - c2);
        p.n_cand = (int)n_cand;
    }
    CK(cudaMemcpyAsync(ctx->params, ctx->h_params, B * sizeof(RetierParams), cudaMemcpyHostToDevice,
                       ctx->compute));
    RetierArgs a{};
    a.s = ctx->s; a.tier = ctx->tier; a.slot = ctx->slot; a.forced = ctx->forced;
    a.params = ctx->params; a.new_tier = ctx->new_tier; a.new_slot = ctx->new_slot;
    a.free_scratch = ctx->free_scratch; a.rl_loc = ctx->rl_loc; a.rl_pos = ctx->rl_pos;
    a.rl_count = ctx->rl_count; a.t0_free = ctx->t0_free; a.t0_top = ctx->t0_top;
    a.moves_now = ctx->moves_now; a.moves_delta = ctx->moves_delta; a.outp = ctx->outp;
    a.B = B; a.N = N; a.Nmax = ctx->Nmax; a.S0 = ctx->S0; a.S1 = ctx->S1; a.S2 = ctx->S2;
    a.prompt_len = ctx->cfg.prompt_len; a.num_sinks = ctx->cfg.num_sinks;
    a.window = ctx->cfg.recent_window;
    CK(launch_retier(a, ctx->compute));
    ctx->launches++;
    CK(cudaMemcpyAsync(ctx->h_outp, ctx->outp, B * sizeof(RetierOut), cudaMemcpyDeviceToHost,
                       ctx->compute));
    CK(cudaStreamSynchronize(ctx->compute));
    tkv_status ds = read_device_status(ctx);
    if (ds != TKV_OK) return ds;

    int hw = 0, hw2 = 0, max_now = 0, max_delta = 0;
    int64_t k[8] = {0};
    for (int b = 0; b < B; ++b) {
        const RetierOut& o = ctx->h_outp[b];
        if (o.error) return fail(ctx, (tkv_status)o.error);
        for (int t = 0; t < 4; ++t) ctx->count[t][b] = o.count[t];
        ctx->R[b] = N - o.count[3];
        hw = std::max(hw, o.hw1);
        hw2 = std::max(hw2, o.hw2);
        max_now = std::max(max_now, o.n_now);
        max_delta = std::max(max_delta, o.n_delta);
        for (int q = 0; q < 7; ++q) k[q] += o.kinds[q];
    }
    ctx->hw1 = hw;
    ctx->hw2 = hw2;
    // rows leaving T0 / entering T2 or T1 from the host side: now, all layers
    MoveArgs m{};
    m.moves = ctx->moves_now;
    m.counts = &ctx->outp[0].n_now;
    m.count_stride = (int)(sizeof(RetierOut) / sizeof(int32_t));
    m.k0v0 = ctx->k0v0; m.t2 = ctx->t2; m.h1 = ctx->d_h1; m.h2m = ctx->d_h2m;
    m.t1_res = ctx->cfg.t1_transport == TKV_T1_RESIDENT ? ctx->stage : nullptr;
    m.layer_begin = 0; m.layer_end = ctx->L;
    m.L = ctx->L; m.B = B; m.Hkv = ctx->Hkv; m.d = ctx->d; m.Nmax = ctx->Nmax;
    m.S0 = ctx->S0; m.S1 = ctx->S1; m.S2 = ctx->S2;
    m.max_count = max_now;
    CK(launch_moves(m, ctx->compute));
    if (max_now > 0) ctx->launches++;
    CK(cudaEventRecord(ctx->ev_retier, ctx->compute));
    ctx->delta_max = max_delta;
    // small deltas are gathered several layers per launch: each launch costs a host-link
    // round trip and a launch, whatever it moves
    {
        int64_t rows = 0;
        for (int b = 0; b < B; ++b) rows += ctx->h_outp[b].n_delta;
        const int64_t per_layer = rows * (int64_t)row_bytes_bf16(ctx);
        const int64_t want = int64_t(1) << 20;
        ctx->delta_chunk = (int)std::min<int64_t>(ctx->L, std::max<int64_t>(1, per_layer > 0 ? (want + per_layer - 1) / per_layer : 1));
        std::fill(ctx->delta_done.begin(), ctx->delta_done.end(), 0);
    }

    const int64_t rb = (int64_t)row_bytes_bf16(ctx) * ctx->L;
    ctx->st.last_promoted = k[MV_T1_T0] + k[MV_T2_T0];
    ctx->st.last_demoted_t1 = k[MV_T0_T1];
    ctx->st.last_quantised = k[MV_T0_T2] + k[MV_T1_T2];
    ctx->st.last_evicted = k[0];
    ctx->st.last_t2_to_t1 = k[MV_T2_T1];
    ctx->st.d2h_bytes_writeback += (k[MV_T0_T1] + k[MV_T0_T2] + k[MV_T1_T2] + k[MV_T2_T1]) * rb;
    ctx->retiers++;
    return TKV_OK;
}

tkv_status issue_prefetch(tkv_ctx* ctx, int layer) {
    const int slotr = layer & 1;
    if (ctx->capturing) {
        // Inside a captured step only events recorded in the capture order the copy
        // stream; a replay as a whole follows everything enqueued before it.
        if (!ctx->copy_joined) {
            CK(cudaStreamWaitEvent(ctx->copy, ctx->ev_fork, 0));
            ctx->copy_joined = true;
        }
        if (ctx->attn_in_capture[slotr]) CK(cudaStreamWaitEvent(ctx->copy, ctx->ev_attn[slotr], 0));
    } else {
        CK(cudaStreamWaitEvent(ctx->copy, ctx->ev_attn[slotr], 0));
        CK(cudaStreamWaitEvent(ctx->copy, ctx->ev_retier, 0));
    }
    if (ctx->hw1 > 0 && ctx->cfg.t1_transport != TKV_T1_RESIDENT) {
        const size_t pitch = (size_t)ctx->S1 * ctx->d * sizeof(__nv_bfloat16);
        const size_t layer_elems = (size_t)2 * ctx->B * ctx->Hkv * ctx->S1 * ctx->d;
        const __nv_bfloat16* src = ctx->h1 + (size_t)layer * layer_elems;
        const __nv_bfloat16* dsrc = ctx->d_h1 + (size_t)layer * layer_elems;
        __nv_bfloat16* dst = ctx->stage + (size_t)slotr * layer_elems;
        const size_t width = (size_t)ctx->hw1 * ctx->d * sizeof(__nv_bfloat16);
        const int height = 2 * ctx->B * ctx->Hkv;
        const int mode = ctx->cfg.t1_transport;
        const bool timed = prof_open(ctx, 1, ctx->copy);
        if (mode == TKV_T1_MULTI_CE) {
            // rows split over the copy stream and kCopyLanes - 1 helper streams
            const int parts = tkv_ctx::kCopyLanes;
            for (int k = 1; k < parts; ++k) {
                const int r0 = height * k / parts, r1 = height * (k + 1) / parts;
                if (r1 <= r0) continue;
                cudaStream_t hs = ctx->copyx[k - 1];
                if (ctx->capturing) {
                    // helper streams join the capture like the copy stream
                    if (!ctx->copyx_joined[k - 1]) {
                        CK(cudaStreamWaitEvent(hs, ctx->ev_fork, 0));
                        ctx->copyx_joined[k - 1] = true;
                    }
                    if (ctx->attn_in_capture[slotr]) CK(cudaStreamWaitEvent(hs, ctx->ev_attn[slotr], 0));
                } else {
                    CK(cudaStreamWaitEvent(hs, ctx->ev_attn[slotr], 0));
                    CK(cudaStreamWaitEvent(hs, ctx->ev_retier, 0));
                }
                CK(cudaMemcpy2DAsync((uint8_t*)dst + (size_t)r0 * pitch, pitch, (const uint8_t*)src + (size_t)r0 * pitch,
                                     pitch, width, r1 - r0, cudaMemcpyHostToDevice, hs));
                CK(cudaEventRecord(ctx->ev_join[k - 1], hs));
            }
            const int r1 = height / parts;
            if (r1 > 0)
                CK(cudaMemcpy2DAsync(dst, pitch, src, pitch, width, r1, cudaMemcpyHostToDevice, ctx->copy));
            for (int k = 1; k < parts; ++k)
                if (height * (k + 1) / parts > height * k / parts)
                    CK(cudaStreamWaitEvent(ctx->copy, ctx->ev_join[k - 1], 0));
            if (timed) prof_close(ctx, 1, ctx->copy, (double)(width * height));
            ctx->st.h2d_bytes_t1_stream += (int64_t)(width * height);
            goto t1_done;
        }
        {
        // rows [0, h_ce) by the copy engine, [h_ce, height) by the copy kernel
        const int h_ce = mode == TKV_T1_COPY_ENGINE ? height : mode == TKV_T1_SM_COPY ? 0 : height / 2;
        if (h_ce < height) {
            cudaStream_t ks = ctx->copy;
            if (h_ce > 0) {
                ks = ctx->copy2;
                CK(cudaStreamWaitEvent(ks, ctx->ev_attn[slotr], 0));
                CK(cudaStreamWaitEvent(ks, ctx->ev_retier, 0));
            }
            CK(launch_t1_copy(dsrc, dst, pitch / 16, width / 16, h_ce, height, ks));
            ctx->launches++;
            if (h_ce > 0) CK(cudaEventRecord(ctx->ev_split, ks));
        }
        if (h_ce > 0)
            CK(cudaMemcpy2DAsync(dst, pitch, src, pitch, width, h_ce, cudaMemcpyHostToDevice, ctx->copy));
        if (h_ce > 0 && h_ce < height) CK(cudaStreamWaitEvent(ctx->copy, ctx->ev_split, 0));
        if (timed) prof_close(ctx, 1, ctx->copy, (double)(width * height));
        ctx->st.h2d_bytes_t1_stream += (int64_t)(width * height);
        }
    }
t1_done:
    if (ctx->t2_host && ctx->hw2 > 0) {
        // T2 records of the layer, rows [0, hw2) of every (K/V, sequence, head), into staging slot layer % 2
        const size_t rec = (size_t)ctx->d + 16;
        const size_t pitch = (size_t)ctx->S2 * rec;
        const size_t layer_bytes = (size_t)2 * ctx->B * ctx->Hkv * pitch;
        const size_t width = (size_t)ctx->hw2 * rec;
        const int height = 2 * ctx->B * ctx->Hkv;
        const bool timed = prof_open(ctx, 1, ctx->copy);
        CK(cudaMemcpy2DAsync(ctx->stage2 + (size_t)slotr * layer_bytes, pitch,
                             ctx->t2_host + (size_t)layer * layer_bytes, pitch, width, height,
                             cudaMemcpyHostToDevice, ctx->copy));
        if (timed) prof_close(ctx, 1, ctx->copy, (double)(width * height));
        ctx->st.h2d_bytes_t2_stream += (int64_t)(width * height);
    }
    if (ctx->delta_max > 0 && !ctx->delta_done[layer]) {
        // this layer's delta and that of the following layers of its chunk whose delta is
        // not enqueued yet, before this layer's T1 event (layers may be prefetched in any order)
        tkv_status r = enqueue_delta_range(ctx, layer, std::min(ctx->L, layer + ctx->delta_chunk),
                                           ctx->delta_chunk, ctx->copy);
        if (r != TKV_OK) return r;
    }
    CK(cudaEventRecord(ctx->ev_t1[slotr], ctx->copy));
    ctx->prefetched[layer] = 1;
    return TKV_OK;
}

}  // namespace

extern "C" {

const char* tkv_status_string(tkv_status s) {
    switch (s) {
        case TKV_OK: return "ok";
        case TKV_EINVAL: return "invalid argument or call order";
        case TKV_ENOMEM: return "out of memory";
        case TKV_ECUDA: return "CUDA error";
        case TKV_ECAPACITY: return "tier store or position capacity exceeded";
        case TKV_ETIMEOUT: return "bounded device wait timed out";
        case TKV_ESTATE: return "context poisoned by an earlier error";
    }
    return "unknown status";
}

tkv_status tkv_create(const tkv_config* cfg, tkv_ctx** out) {
    if (!cfg || !out) return TKV_EINVAL;
    *out = nullptr;
    const tkv_config& c = *cfg;
    if (c.num_layers < 1 || c.num_kv_heads < 1 || c.num_q_heads < 1 || c.batch < 1) return TKV_EINVAL;
    if (c.num_q_heads % c.num_kv_heads) return TKV_EINVAL;
    const int G = c.num_q_heads / c.num_kv_heads;
    if (G > 8 || (c.head_dim != 64 && c.head_dim != 128)) return TKV_EINVAL;
    if (c.max_tokens < 1 || c.max_tokens > 65536) return TKV_EINVAL;
    if (c.prompt_len < 0 || c.num_sinks < 0 || c.recent_window < 0) return TKV_EINVAL;
    if (c.t0_capacity < 0 || c.t1_capacity < 0 || c.t2_capacity < 0) return TKV_EINVAL;
    if (c.t1_transport < TKV_T1_COPY_ENGINE || c.t1_transport > TKV_T1_RESIDENT) return TKV_EINVAL;
    if (c.t2_placement != TKV_T2_HBM && c.t2_placement != TKV_T2_HOST) return TKV_EINVAL;
    if (c.host_alloc < TKV_HOST_AUTO || c.host_alloc > TKV_HOST_HUGE_ARENA) return TKV_EINVAL;
    const float r[4] = {c.ratio_t0, c.ratio_t1, c.ratio_t2, c.ratio_t3};
    int64_t ppm[4], sum = 0;
    for (int i = 0; i < 4; ++i) {
        if (!(r[i] >= 0.f && r[i] <= 1.f)) return TKV_EINVAL;
        ppm[i] = to_ppm(r[i]);
        sum += ppm[i];
    }
    if (std::llabs(sum - 1000000) > 8) return TKV_EINVAL;

    tkv_ctx* ctx = new (std::nothrow) tkv_ctx();
    if (!ctx) return TKV_ENOMEM;
    ctx->cfg = c;
    ctx->L = c.num_layers; ctx->B = c.batch; ctx->Hq = c.num_q_heads; ctx->Hkv = c.num_kv_heads;
    ctx->G = G; ctx->d = c.head_dim; ctx->Nmax = c.max_tokens;
    ctx->S0 = c.t0_capacity ? c.t0_capacity : c.max_tokens;
    ctx->S1 = c.t1_capacity ? c.t1_capacity : c.max_tokens;
    ctx->S2 = c.t2_capacity ? c.t2_capacity : (ppm[2] > 0 ? c.max_tokens : 0);
    for (int i = 0; i < 4; ++i) ctx->ppm[i] = ppm[i];
    ctx->device = c.device;
    if (const char* fi = std::getenv("TKV_FAULT_INJECT")) {
        if (std::strcmp(fi, "hostalloc") == 0) ctx->inject_hostalloc = true;
        else if (std::strncmp(fi, "call:", 5) == 0) ctx->inject_at = std::max(0LL, std::atoll(fi + 5));
    }
    DeviceGuard guard(c.device);

    auto bail = [&](tkv_status s) {
        free_all(ctx);
        delete ctx;
        return s;
    };
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || c.device < 0 || c.device >= ndev) {
        (void)cudaGetLastError();
        return bail(TKV_ECUDA);
    }
    if (cudaSetDevice(c.device) != cudaSuccess) return bail(TKV_ECUDA);

    if (c.compute_stream) ctx->compute = (cudaStream_t)c.compute_stream;
    else {
        if (cudaStreamCreateWithFlags(&ctx->compute, cudaStreamNonBlocking) != cudaSuccess) return bail(TKV_ECUDA);
        ctx->own_compute = true;
    }
    if (c.copy_stream) ctx->copy = (cudaStream_t)c.copy_stream;
    else {
        if (cudaStreamCreateWithFlags(&ctx->copy, cudaStreamNonBlocking) != cudaSuccess) return bail(TKV_ECUDA);
        ctx->own_copy = true;
    }

    const size_t L = ctx->L, B = ctx->B, Hkv = ctx->Hkv, d = ctx->d, Nmax = ctx->Nmax;
    const size_t S0 = ctx->S0, S1 = ctx->S1, S2 = ctx->S2;
    bool ok = true;
    auto A = [&](cudaError_t e) {
        if (e != cudaSuccess) ok = false;
    };
    A(dalloc(ctx, &ctx->k0v0, L * 2 * B * Hkv * S0 * d));
    // T1 staging: a two-slot ring, or (TKV_T1_RESIDENT) a resident copy of every layer's T1 rows
    A(dalloc(ctx, &ctx->stage, (c.t1_transport == TKV_T1_RESIDENT ? L : 2) * 2 * B * Hkv * S1 * d));
    const bool t2_host = c.t2_placement == TKV_T2_HOST;
    if (!t2_host) A(dalloc(ctx, &ctx->t2, L * 2 * B * Hkv * S2 * (d + 16)));
    else A(dalloc(ctx, &ctx->stage2, 2 * 2 * B * Hkv * S2 * (d + 16)));
    A(dalloc(ctx, &ctx->tier, B * Nmax));
    A(dalloc(ctx, &ctx->new_tier, B * Nmax));
    A(dalloc(ctx, &ctx->forced, B * Nmax));
    A(dalloc(ctx, &ctx->slot, B * Nmax));
    A(dalloc(ctx, &ctx->new_slot, B * Nmax));
    A(dalloc(ctx, &ctx->free_scratch, B * std::max(S0, std::max(S1, S2))));
    A(dalloc(ctx, &ctx->s, B * Nmax));
    A(dalloc(ctx, &ctx->rl_loc, B * Nmax));
    A(dalloc(ctx, &ctx->rl_pos, B * Nmax));
    A(dalloc(ctx, &ctx->rl_count, B));
    A(dalloc(ctx, &ctx->g, B * Hkv * Nmax));
    A(dalloc(ctx, &ctx->zs, attention_zs_floats(G, (int)B, (int)Hkv, (int)Nmax)));
    A(dalloc(ctx, &ctx->t0_free, B * S0));
    A(dalloc(ctx, &ctx->t0_top, B));
    A(dalloc(ctx, &ctx->moves_now, B * Nmax));
    A(dalloc(ctx, &ctx->moves_delta, B * Nmax));
    A(dalloc(ctx, &ctx->outp, B));
    A(dalloc(ctx, &ctx->params, B));
    A(dalloc(ctx, &ctx->err, 1));
    A(dalloc(ctx, &ctx->pos_n, B));
    if (!ok) {
        (void)cudaGetLastError();
        return bail(TKV_ENOMEM);
    }
    {
        int numa = -1;
        if (online_nodes() > 1 && cudaDeviceGetAttribute(&numa, cudaDevAttrHostNumaId, c.device) == cudaSuccess)
            ctx->host_numa = numa;
        (void)cudaGetLastError();
    }
    A(harena_alloc(ctx, ctx->hs_h1, L * 2 * B * Hkv * S1 * d * sizeof(__nv_bfloat16)));
    A(harena_alloc(ctx, ctx->hs_h2m, L * 2 * B * Hkv * S2 * d * sizeof(__nv_bfloat16)));
    if (t2_host) A(harena_alloc(ctx, ctx->hs_t2, L * 2 * B * Hkv * S2 * (d + 16)));
    ctx->h1 = (__nv_bfloat16*)ctx->hs_h1.ptr;
    ctx->h2m = (__nv_bfloat16*)ctx->hs_h2m.ptr;
    ctx->t2_host = (uint8_t*)ctx->hs_t2.ptr;
    A(halloc(ctx, &ctx->h_outp, B));
    A(halloc(ctx, &ctx->h_params, B));
    A(halloc(ctx, &ctx->h_err, 1));
    if (!ok) {
        (void)cudaGetLastError();
        return bail(TKV_ENOMEM);
    }
    if (ctx->h1 && cudaHostGetDevicePointer((void**)&ctx->d_h1, ctx->h1, 0) != cudaSuccess) return bail(TKV_ECUDA);
    if (ctx->h2m && cudaHostGetDevicePointer((void**)&ctx->d_h2m, ctx->h2m, 0) != cudaSuccess) return bail(TKV_ECUDA);
    if (ctx->t2_host && cudaHostGetDevicePointer((void**)&ctx->t2, ctx->t2_host, 0) != cudaSuccess) return bail(TKV_ECUDA);
    std::memset(ctx->h_outp, 0, B * sizeof(RetierOut));

    // page tables: empty; T0 free stack holds every slot, lowest on top
    std::vector<int32_t> fr(B * S0);
    for (size_t b = 0; b < B; ++b)
        for (size_t j = 0; j < S0; ++j) fr[b * S0 + j] = (int32_t)(S0 - 1 - j);
    std::vector<int32_t> top(B, (int32_t)S0);
    bool e = true;
    auto E = [&](cudaError_t x) {
        if (x != cudaSuccess) e = false;
    };
    E(cudaMemcpy(ctx->t0_free, fr.data(), fr.size() * 4, cudaMemcpyHostToDevice));
    E(cudaMemcpy(ctx->t0_top, top.data(), B * 4, cudaMemcpyHostToDevice));
    E(cudaMemset(ctx->rl_count, 0, B * 4));
    E(cudaMemset(ctx->tier, 0, B * Nmax));
    E(cudaMemset(ctx->s, 0, B * Nmax * 4));
    E(cudaMemset(ctx->outp, 0, B * sizeof(RetierOut)));
    E(cudaMemset(ctx->err, 0, 4));
    E(cudaMemset(ctx->pos_n, 0, B * 4));
    for (int i = 0; i < 2; ++i) {
        E(cudaEventCreateWithFlags(&ctx->ev_t1[i], cudaEventDisableTiming));
        E(cudaEventCreateWithFlags(&ctx->ev_attn[i], cudaEventDisableTiming));
    }
    E(cudaEventCreateWithFlags(&ctx->ev_retier, cudaEventDisableTiming));
    E(cudaEventCreateWithFlags(&ctx->ev_fork, cudaEventDisableTiming));
    E(cudaStreamCreateWithFlags(&ctx->cap_stream, cudaStreamNonBlocking));
    E(cudaEventCreateWithFlags(&ctx->ev_split, cudaEventDisableTiming));
    E(cudaStreamCreateWithFlags(&ctx->copy2, cudaStreamNonBlocking));
    for (int i = 0; i < tkv_ctx::kCopyLanes - 1; ++i) {
        E(cudaStreamCreateWithFlags(&ctx->copyx[i], cudaStreamNonBlocking));
        E(cudaEventCreateWithFlags(&ctx->ev_join[i], cudaEventDisableTiming));
    }
    if (!e) {
        (void)cudaGetLastError();
        return bail(TKV_ECUDA);
    }

    // kernel set-up: the largest attention launch stages a full retained-list window per CTA
    {
        const size_t smem = attention_smem_bytes(G, ctx->d, attention_max_window_rows());
        if (attention_prepare(G, ctx->d, smem) != cudaSuccess) return bail(TKV_ECUDA);
        ctx->resident = attention_resident_ctas(G, ctx->d, smem);
        if (ctx->resident < 1) return bail(TKV_ECUDA);
        if (dalloc(ctx, &ctx->part, attention_part_floats(G, ctx->d, ctx->B, ctx->Hkv, ctx->Nmax, ctx->resident)) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            return bail(TKV_ENOMEM);
        }
    }
    if (retier_prepare(retier_smem_bytes(ctx->S0, ctx->S1, ctx->S2)) != cudaSuccess) return bail(TKV_ECUDA);

    for (int t = 0; t < 4; ++t) ctx->count[t].assign(B, 0);
    ctx->R.assign(B, 0);
    ctx->prefetched.assign(L, 0);
    ctx->delta_done.assign(L, 0);
    ctx->pend_k.assign(L, nullptr);
    ctx->pend_v.assign(L, nullptr);
    *out = ctx;
    return TKV_OK;
}

void tkv_destroy(tkv_ctx* ctx) {
    if (!ctx) return;
    DeviceGuard guard(ctx->device);
    if (ctx->capturing) {
        cudaGraph_t g = nullptr;
        cudaStreamEndCapture(ctx->cap_stream, &g);
        if (g) cudaGraphDestroy(g);
        ctx->compute = ctx->cap_saved_compute;
        ctx->capturing = false;
        (void)cudaGetLastError();
    }
    if (ctx->compute) cudaStreamSynchronize(ctx->compute);
    if (ctx->copy) cudaStreamSynchronize(ctx->copy);
    free_all(ctx);
    delete ctx;
}

tkv_status tkv_append(tkv_ctx* ctx, int32_t layer, const void* k, const void* v, int32_t n_tokens) {
    CHECK_CTX();
    if (!k || !v || n_tokens < 1 || layer < 0 || layer >= ctx->L) return TKV_EINVAL;
    // rows are copied in 16-byte units
    if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15u) return TKV_EINVAL;
    if (n_tokens > 1 && ctx->capturing) return TKV_EINVAL;
    DeviceGuard guard(ctx->device);
    if (n_tokens > 1) drop_graph(ctx);
    const int B = ctx->B;
    if (ctx->open_n == 0) {
        if (layer != 0) return TKV_EINVAL;
        if (ctx->N + n_tokens > ctx->Nmax) return TKV_ECAPACITY;
        for (int b = 0; b < B; ++b)
            if (ctx->count[0][b] + n_tokens > ctx->S0) return TKV_ECAPACITY;
        int nl = 0;
        CK(launch_open(ctx->t0_free, ctx->t0_top, ctx->tier, ctx->slot, ctx->s, ctx->rl_loc, ctx->rl_pos,
                       ctx->rl_count, ctx->pos_n, B, ctx->Nmax, ctx->S0, n_tokens, ctx->compute, &nl));
        ctx->launches += nl;
        for (int b = 0; b < B; ++b) {
            ctx->count[0][b] += n_tokens;
            ctx->R[b] += n_tokens;
        }
        ctx->open_n = n_tokens;
        ctx->appended = 0;
        ctx->decoded = 0;
        std::fill(ctx->prefetched.begin(), ctx->prefetched.end(), 0);
    } else {
        if (n_tokens != ctx->open_n || layer != ctx->appended) return TKV_EINVAL;
    }
    if (n_tokens == 1) {
        // written by this layer's attention kernel
        ctx->pend_k[layer] = k;
        ctx->pend_v[layer] = v;
    } else {
        CK(launch_append_rows((const __nv_bfloat16*)k, (const __nv_bfloat16*)v, ctx->k0v0, ctx->slot, layer,
                              B, ctx->Hkv, ctx->d, ctx->Nmax, ctx->S0, ctx->N, n_tokens, ctx->compute));
        ctx->launches++;
    }
    ctx->appended++;
    if (ctx->open_n > 1 && ctx->appended == ctx->L) {
        ctx->N += ctx->open_n;
        ctx->open_n = 0;
    }
    return TKV_OK;
}

tkv_status tkv_prefetch(tkv_ctx* ctx, int32_t layer) {
    CHECK_CTX();
    if (layer < 0 || layer >= ctx->L) return TKV_EINVAL;
    if (ctx->open_n != 1 || ctx->prefetched[layer]) return TKV_EINVAL;
    // staging slot layer % 2 is still read by layer - 2's attention until it is issued
    if (layer >= 2 && ctx->decoded < layer - 1) return TKV_EINVAL;
    DeviceGuard guard(ctx->device);
    return issue_prefetch(ctx, layer);
}

tkv_status tkv_decode_step(tkv_ctx* ctx, int32_t layer, const void* q, float* out) {
    CHECK_CTX();
    if (!q || !out || layer < 0 || layer >= ctx->L) return TKV_EINVAL;
    if (ctx->open_n != 1 || layer != ctx->decoded || layer >= ctx->appended) return TKV_EINVAL;
    DeviceGuard guard(ctx->device);
    if (!ctx->prefetched[layer]) {
        tkv_status r = issue_prefetch(ctx, layer);
        if (r != TKV_OK) return r;
    }
    const int slotr = layer & 1;
    CK(cudaStreamWaitEvent(ctx->compute, ctx->ev_t1[slotr], 0));

    int rmax = 0;
    for (int b = 0; b < ctx->B; ++b) rmax = std::max(rmax, ctx->R[b]);
    const AttnPlan plan = attention_plan(ctx->G, ctx->d, ctx->B, ctx->Hkv, rmax, ctx->resident);
    AttnArgs a{};
    a.q = (const __nv_bfloat16*)q;
    a.out = out;
    a.k0v0 = ctx->k0v0;
    a.stage = ctx->stage + (size_t)(ctx->cfg.t1_transport == TKV_T1_RESIDENT ? layer : slotr) * 2 * ctx->B *
                               ctx->Hkv * ctx->S1 * ctx->d;
    if (ctx->t2_host) {
        a.t2 = ctx->stage2 + (size_t)slotr * 2 * ctx->B * ctx->Hkv * ctx->S2 * (ctx->d + 16);
        a.t2_layer = 0;
    } else {
        a.t2 = ctx->t2;
        a.t2_layer = layer;
    }
    a.new_k = (const __nv_bfloat16*)ctx->pend_k[layer];
    a.new_v = (const __nv_bfloat16*)ctx->pend_v[layer];
    ctx->pend_k[layer] = ctx->pend_v[layer] = nullptr;
    a.rl_loc = ctx->rl_loc;
    a.rl_count = ctx->rl_count;
    a.g = ctx->g;
    a.part = ctx->part;
    a.zs = ctx->zs;
    a.err = ctx->err;
    a.layer = layer; a.L = ctx->L; a.B = ctx->B; a.Hq = ctx->Hq; a.Hkv = ctx->Hkv; a.d = ctx->d;
    a.Nmax = ctx->Nmax; a.S0 = ctx->S0; a.S1 = ctx->S1; a.S2 = ctx->S2;
    a.item_rows = plan.item_rows;
    a.items_per_group = plan.items_per_group;
    a.items_per_cta = plan.items_per_cta;
    a.grid = plan.grid;
    a.part_per_group = plan.part_per_group;
    a.qscale = (float)(1.4426950408889634 / std::sqrt((double)ctx->d));
    const bool timed = prof_open(ctx, 0, ctx->compute);
    // when timed, the main kernel and the combine kernel are bracketed separately
    cudaEvent_t mid0 = nullptr, mid1 = nullptr;
    if (timed) {
        mid0 = ctx->prof_ev[0][2 * ctx->prof_used[0] + 1];
        mid1 = ctx->prof_used[3] < tkv_ctx::kProfPairs ? ctx->prof_ev[3][2 * ctx->prof_used[3]] : nullptr;
    }
    CK(launch_attention(a, ctx->compute, mid0, mid1));
    ctx->launches += 2;
    if (timed) {
        // main kernel: the K/V rows it reads (bf16 rows of T0 / T1, T2 codes + scales) and q
        double bytes = (double)ctx->B * ctx->Hq * ctx->d * 2;
        for (int b = 0; b < ctx->B; ++b)
            bytes += (double)(ctx->count[0][b] + ctx->count[1][b]) * 4.0 * ctx->Hkv * ctx->d +
                     (double)ctx->count[2][b] * (2.0 * ctx->Hkv * ctx->d + 8.0 * ctx->Hkv);
        ctx->prof_used[0]++;
        ctx->prof_bytes[0] += bytes;
        if (mid1) {
            // combine: out (fp32) written, the logits and alpha sums of the retained rows
            double cb = (double)ctx->B * ctx->Hq * ctx->d * 4;
            const int GP = ctx->G <= 4 ? 4 : 8;
            for (int b = 0; b < ctx->B; ++b) cb += (double)ctx->R[b] * ctx->Hkv * (GP * 4.0 + 8.0);
            prof_close(ctx, 3, ctx->compute, cb);
        }
    }
    CK(cudaEventRecord(ctx->ev_attn[slotr], ctx->compute));
    if (ctx->capturing) {
        ctx->attn_in_capture[slotr] = true;
        // the launch plan is a function of ceil(rmax / 64): replays stay within this 64-row bucket
        // so that they run the geometry an eager step would
        ctx->cap_rows = std::min(plan.items_per_group * plan.item_rows, (rmax + 63) / 64 * 64);
    }
    ctx->last_splits = plan.grid;
    ctx->decoded++;
    if (ctx->decoded == ctx->L) {
        const float inv = (float)(1.0 / ((double)ctx->L * (double)ctx->Hq));
        // a captured fold covers every retained count its replays can meet
        CK(launch_fold(ctx->g, ctx->rl_pos, ctx->rl_count, ctx->s, ctx->B, ctx->Hkv, ctx->Nmax,
                       ctx->capturing ? ctx->cap_rows : rmax,
                       inv, ctx->compute));
        ctx->launches++;
        ctx->N += 1;
        ctx->open_n = 0;
        ctx->step++;
        ctx->delta_max = 0;   // this step's prefetches applied the delta for every layer
    }
    return TKV_OK;
}

tkv_status tkv_retier(tkv_ctx* ctx) {
    CHECK_CTX();
    if (ctx->open_n != 0 || ctx->capturing) return TKV_EINVAL;
    DeviceGuard guard(ctx->device);
    return run_retier(ctx, false);
}

tkv_status tkv_get_scores(tkv_ctx* ctx, float* dst) {
    CHECK_CTX();
    if (ctx->capturing) return TKV_EINVAL;   // synchronous: not inside a capture
    if (!dst) return TKV_EINVAL;
    DeviceGuard guard(ctx->device);
    CK(cudaStreamSynchronize(ctx->copy));
    CK(cudaStreamSynchronize(ctx->compute));
    if (ctx->N > 0)
        CK(cudaMemcpy2D(dst, ctx->N * sizeof(float), ctx->s, ctx->Nmax * sizeof(float), ctx->N * sizeof(float),
                        ctx->B, cudaMemcpyDeviceToHost));
    return read_device_status(ctx);
}

tkv_status tkv_set_scores(tkv_ctx* ctx, const float* src) {
    CHECK_CTX();
    if (ctx->capturing) return TKV_EINVAL;   // synchronous: not inside a capture
    if (!src || ctx->open_n != 0) return TKV_EINVAL;
    DeviceGuard guard(ctx->device);
    CK(cudaStreamSynchronize(ctx->compute));
    if (ctx->N > 0)
        CK(cudaMemcpy2D(ctx->s, ctx->Nmax * sizeof(float), src, ctx->N * sizeof(float), ctx->N * sizeof(float),
                        ctx->B, cudaMemcpyHostToDevice));
    return TKV_OK;
}

tkv_status tkv_get_tiers(tkv_ctx* ctx, uint8_t* dst) {
    CHECK_CTX();
    if (ctx->capturing) return TKV_EINVAL;   // synchronous: not inside a capture
    if (!dst) return TKV_EINVAL;
    DeviceGuard guard(ctx->device);
    CK(cudaStreamSynchronize(ctx->copy));
    CK(cudaStreamSynchronize(ctx->compute));
    if (ctx->N > 0)
        CK(cudaMemcpy2D(dst, ctx->N, ctx->tier, ctx->Nmax, ctx->N, ctx->B, cudaMemcpyDeviceToHost));
    return read_device_status(ctx);
}

tkv_status tkv_set_tiers(tkv_ctx* ctx, const uint8_t* src) {
    CHECK_CTX();
    if (ctx->capturing) return TKV_EINVAL;   // synchronous: not inside a capture
    if (!src || ctx->open_n != 0) return TKV_EINVAL;
    DeviceGuard guard(ctx->device);
    const int N = ctx->N, B = ctx->B;
    std::vector<uint8_t> cur((size_t)B * N);
    tkv_status r = tkv_get_tiers(ctx, cur.data());
    if (r != TKV_OK) return r;
    for (size_t i = 0; i < cur.size(); ++i) {
        if (src[i] > 3) return TKV_EINVAL;
        if (cur[i] == 3 && src[i] != 3) return TKV_EINVAL;
        // protected positions (sinks, prompt, recent window at the current N) are never evicted
        const int pos = (int)(i % (size_t)N);
        if (src[i] == 3 && (pos < ctx->cfg.num_sinks || pos < ctx->cfg.prompt_len ||
                            pos >= N - ctx->cfg.recent_window))
            return TKV_EINVAL;
    }
    if (N > 0)
        CK(cudaMemcpy2D(ctx->forced, ctx->Nmax, src, N, N, B, cudaMemcpyHostToDevice));
    return run_retier(ctx, true);
}

tkv_status tkv_get_row(tkv_ctx* ctx, int32_t layer, int32_t seq, int32_t pos, void* dst,
                       float* scales, int32_t* tier_out) {
    CHECK_CTX();
    if (ctx->capturing) return TKV_EINVAL;   // synchronous: not inside a capture
    if (!dst || !tier_out || layer < 0 || layer >= ctx->L || seq < 0 || seq >= ctx->B || pos < 0 ||
        pos >= ctx->N)
        return TKV_EINVAL;
    DeviceGuard guard(ctx->device);
    CK(cudaStreamSynchronize(ctx->copy));
    CK(cudaStreamSynchronize(ctx->compute));
    uint8_t t = 0;
    int32_t sl = 0;
    const size_t p = (size_t)seq * ctx->Nmax + pos;
    CK(cudaMemcpy(&t, ctx->tier + p, 1, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(&sl, ctx->slot + p, 4, cudaMemcpyDeviceToHost));
    *tier_out = t;
    const int d = ctx->d;
    for (int kv = 0; kv < 2; ++kv) {
        for (int h = 0; h < ctx->Hkv; ++h) {
            const size_t o = (size_t)kv * ctx->Hkv + h;
            if (t == 0) {
                CK(cudaMemcpy((uint16_t*)dst + o * d,
                              ctx->k0v0 + row_index(layer, kv, seq, h, sl, ctx->B, ctx->Hkv, ctx->S0) * d,
                              (size_t)d * 2, cudaMemcpyDeviceToHost));
            } else if (t == 1) {
                std::memcpy((uint16_t*)dst + o * d,
                            ctx->h1 + row_index(layer, kv, seq, h, sl, ctx->B, ctx->Hkv, ctx->S1) * d,
                            (size_t)d * 2);
            } else if (t == 2) {
                const size_t ri = row_index(layer, kv, seq, h, sl, ctx->B, ctx->Hkv, ctx->S2) * (d + 16);
                if (ctx->t2_host) {
                    std::memcpy((uint8_t*)dst + o * d, ctx->t2_host + ri, (size_t)d);
                    if (scales) std::memcpy(scales + o, ctx->t2_host + ri + d, 4);
                } else {
                    CK(cudaMemcpy((uint8_t*)dst + o * d, ctx->t2 + ri, (size_t)d, cudaMemcpyDeviceToHost));
                    if (scales) CK(cudaMemcpy(scales + o, ctx->t2 + ri + d, 4, cudaMemcpyDeviceToHost));
                }
            }
        }
    }
    return read_device_status(ctx);
}

tkv_status tkv_profile_begin(tkv_ctx* ctx) {
    CHECK_CTX();
    if (ctx->capturing) return TKV_EINVAL;   // synchronous: not inside a capture
    DeviceGuard guard(ctx->device);
    for (int k = 0; k < tkv_ctx::kProfKinds; ++k) {
        if (ctx->prof_ev[k].empty()) {
            ctx->prof_ev[k].resize(2 * tkv_ctx::kProfPairs, nullptr);
            for (auto& e : ctx->prof_ev[k]) CK(cudaEventCreate(&e));
        }
        ctx->prof_used[k] = 0;
        ctx->prof_bytes[k] = 0.0;
    }
    ctx->profiling = true;
    return TKV_OK;
}

tkv_status tkv_profile_end(tkv_ctx* ctx, tkv_prof_entry* attn, tkv_prof_entry* combine, tkv_prof_entry* t1,
                           tkv_prof_entry* delta) {
    CHECK_CTX();
    if (ctx->capturing) return TKV_EINVAL;   // synchronous: not inside a capture
    DeviceGuard guard(ctx->device);
    ctx->profiling = false;
    CK(cudaStreamSynchronize(ctx->copy));
    CK(cudaStreamSynchronize(ctx->compute));
    tkv_prof_entry* outs[tkv_ctx::kProfKinds] = {attn, t1, delta, combine};
    for (int k = 0; k < tkv_ctx::kProfKinds; ++k) {
        double ms = 0.0;
        for (int i = 0; i < ctx->prof_used[k]; ++i) {
            float t = 0.f;
            CK(cudaEventElapsedTime(&t, ctx->prof_ev[k][2 * i], ctx->prof_ev[k][2 * i + 1]));
            ms += t;
        }
        if (outs[k]) {
            outs[k]->ms = ms;
            outs[k]->count = ctx->prof_used[k];
            outs[k]->bytes = ctx->prof_bytes[k];
        }
    }
    return read_device_status(ctx);
}

tkv_status tkv_capture_begin(tkv_ctx* ctx) {
    CHECK_CTX();
    if (ctx->capturing || ctx->open_n != 0 || ctx->delta_max > 0 || ctx->profiling) return TKV_EINVAL;
    if (ctx->cfg.t1_transport == TKV_T1_SPLIT) return TKV_EINVAL;
    DeviceGuard guard(ctx->device);
    drop_graph(ctx);
    ctx->cap_saved.N = ctx->N;
    ctx->cap_saved.count0 = ctx->count[0];
    ctx->cap_saved.R = ctx->R;
    ctx->cap_saved.step = ctx->step;
    ctx->cap_saved.launches = ctx->launches;
    ctx->cap_saved.st = ctx->st;
    CK(cudaStreamBeginCapture(ctx->cap_stream, cudaStreamCaptureModeThreadLocal));
    if (cudaEventRecord(ctx->ev_fork, ctx->cap_stream) != cudaSuccess) {
        cudaGraph_t g = nullptr;
        cudaStreamEndCapture(ctx->cap_stream, &g);
        if (g) cudaGraphDestroy(g);
        (void)cudaGetLastError();
        return fail(ctx, TKV_ECUDA);
    }
    ctx->cap_saved_compute = ctx->compute;
    ctx->compute = ctx->cap_stream;
    ctx->capturing = true;
    ctx->copy_joined = false;
    for (bool& j : ctx->copyx_joined) j = false;
    ctx->attn_in_capture[0] = ctx->attn_in_capture[1] = false;
    ctx->cap_rows = 0;
    return TKV_OK;
}

tkv_status tkv_capture_end(tkv_ctx* ctx, int32_t* steps_valid) {
    if (!ctx || !ctx->capturing) return TKV_EINVAL;
    DeviceGuard guard(ctx->device);
    cudaGraph_t graph = nullptr;
    const cudaError_t ce = cudaStreamEndCapture(ctx->cap_stream, &graph);
    ctx->capturing = false;
    ctx->compute = ctx->cap_saved_compute;
    const bool one_step = ctx->open_n == 0 && ctx->step == ctx->cap_saved.step + 1;
    const int64_t launches = ctx->launches - ctx->cap_saved.launches;
    const int64_t t1 = ctx->st.h2d_bytes_t1_stream - ctx->cap_saved.st.h2d_bytes_t1_stream;
    const int64_t t2b = ctx->st.h2d_bytes_t2_stream - ctx->cap_saved.st.h2d_bytes_t2_stream;
    // nothing of the captured step has run: back to the state before it
    ctx->N = ctx->cap_saved.N;
    ctx->count[0] = ctx->cap_saved.count0;
    ctx->R = ctx->cap_saved.R;
    ctx->step = ctx->cap_saved.step;
    ctx->launches = ctx->cap_saved.launches;
    ctx->st = ctx->cap_saved.st;
    ctx->open_n = 0;
    ctx->appended = ctx->decoded = 0;
    std::fill(ctx->pend_k.begin(), ctx->pend_k.end(), nullptr);
    std::fill(ctx->pend_v.begin(), ctx->pend_v.end(), nullptr);
    if (rerecord_events(ctx) != cudaSuccess) {
        if (graph) cudaGraphDestroy(graph);
        (void)cudaGetLastError();
        return fail(ctx, TKV_ECUDA);
    }
    if (ce != cudaSuccess || !graph) {
        (void)cudaGetLastError();
        return fail(ctx, TKV_ECUDA);
    }
    if (!one_step) {
        cudaGraphDestroy(graph);
        return TKV_EINVAL;
    }
    const cudaError_t ie = cudaGraphInstantiate(&ctx->graph_exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ie != cudaSuccess) {
        ctx->graph_exec = nullptr;
        (void)cudaGetLastError();
        return fail(ctx, TKV_ECUDA);
    }
    // replay k (from 1) decodes with R_b + k retained rows and N + k positions
    int rmax = 0, c0max = 0;
    for (int b = 0; b < ctx->B; ++b) {
        rmax = std::max(rmax, ctx->R[b]);
        c0max = std::max(c0max, ctx->count[0][b]);
    }
    int valid = std::min(ctx->cap_rows - rmax, ctx->Nmax - ctx->N);
    valid = std::max(0, std::min(valid, ctx->S0 - c0max));
    ctx->graph_steps_left = valid;
    ctx->graph_launches = launches;
    ctx->graph_t1_bytes = t1;
    ctx->graph_t2_bytes = t2b;
    if (steps_valid) *steps_valid = valid;
    return TKV_OK;
}

tkv_status tkv_replay(tkv_ctx* ctx) {
    CHECK_CTX();
    if (ctx->capturing || !ctx->graph_exec || ctx->graph_steps_left <= 0 || ctx->open_n != 0 ||
        ctx->delta_max > 0)
        return TKV_EINVAL;
    DeviceGuard guard(ctx->device);
    CK(cudaGraphLaunch(ctx->graph_exec, ctx->compute));
    CK(rerecord_events(ctx));
    ctx->N += 1;
    for (int b = 0; b < ctx->B; ++b) {
        ctx->count[0][b] += 1;
        ctx->R[b] += 1;
    }
    ctx->step++;
    ctx->launches += ctx->graph_launches;
    ctx->st.h2d_bytes_t1_stream += ctx->graph_t1_bytes;
    ctx->st.h2d_bytes_t2_stream += ctx->graph_t2_bytes;
    ctx->graph_steps_left--;
    return TKV_OK;
}

tkv_status tkv_sync(tkv_ctx* ctx) {
    CHECK_CTX();
    if (ctx->capturing) return TKV_EINVAL;   // synchronous: not inside a capture
    DeviceGuard guard(ctx->device);
    CK(cudaStreamSynchronize(ctx->copy));
    CK(cudaStreamSynchronize(ctx->compute));
    return read_device_status(ctx);
}

tkv_status tkv_measure_host_link(int32_t device, int64_t bytes, double* h2d_ce_gbs, double* h2d_sm_gbs,
                                 double* d2h_ce_gbs) {
    if (bytes < (1 << 20) || (bytes & 15) || device < 0) return TKV_EINVAL;
    DeviceGuard guard(device);
    if (cudaSetDevice(device) != cudaSuccess) {
        (void)cudaGetLastError();
        return TKV_ECUDA;
    }
    const size_t n = (size_t)bytes;
    void *h = nullptr, *dh = nullptr, *dbuf = nullptr;
    cudaStream_t st = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    tkv_status rc = TKV_OK;
    double best[3] = {0.0, 0.0, 0.0};   // GB/s: H2D copy engine, H2D SM loads, D2H copy engine
    if (cudaHostAlloc(&h, n, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess ||
        cudaMalloc(&dbuf, n) != cudaSuccess) {
        rc = TKV_ENOMEM;
    } else if (cudaHostGetDevicePointer(&dh, h, 0) != cudaSuccess ||
               cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess ||
               cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        rc = TKV_ECUDA;
    } else {
        std::memset(h, 0x5a, n);
        // one untimed pass of each kind, then the best of three timed passes
        for (int rep = 0; rep < 4 && rc == TKV_OK; ++rep) {
            for (int kind = 0; kind < 3; ++kind) {
                cudaError_t e = cudaEventRecord(e0, st);
                if (e == cudaSuccess) {
                    if (kind == 0) e = cudaMemcpyAsync(dbuf, h, n, cudaMemcpyHostToDevice, st);
                    else if (kind == 1) e = launch_t1_copy(dh, dbuf, n / 16, n / 16, 0, 1, st);
                    else e = cudaMemcpyAsync(h, dbuf, n, cudaMemcpyDeviceToHost, st);
                }
                if (e == cudaSuccess) e = cudaEventRecord(e1, st);
                if (e == cudaSuccess) e = cudaEventSynchronize(e1);
                float ms = 0.f;
                if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
                if (e != cudaSuccess) {
                    rc = TKV_ECUDA;
                    break;
                }
                if (rep > 0 && ms > 0.f) best[kind] = std::max(best[kind], (double)n / (ms * 1e-3) / 1e9);
            }
        }
    }
    if (st) cudaStreamSynchronize(st);
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (st) cudaStreamDestroy(st);
    if (dbuf) cudaFree(dbuf);
    if (h) cudaFreeHost(h);
    (void)cudaGetLastError();
    if (rc != TKV_OK) return rc;
    if (h2d_ce_gbs) *h2d_ce_gbs = best[0];
    if (h2d_sm_gbs) *h2d_sm_gbs = best[1];
    if (d2h_ce_gbs) *d2h_ce_gbs = best[2];
    return TKV_OK;
}

tkv_status tkv_get_stats(tkv_ctx* ctx, tkv_stats* out) {
    if (!ctx || !out) return TKV_EINVAL;
    tkv_stats s = ctx->st;
    s.num_tokens = ctx->N;
    s.step = ctx->step;
    s.retiers = ctx->retiers;
    for (int t = 0; t < 4; ++t) {
        s.tier_count[t] = 0;
        for (int b = 0; b < ctx->B; ++b) s.tier_count[t] += ctx->count[t][b];
    }
    s.t1_rows_streamed = ctx->hw1;
    s.hbm_bytes_allocated = (int64_t)ctx->hbm_alloc;
    s.host_bytes_allocated = (int64_t)ctx->host_alloc;
    const int64_t rb = (int64_t)row_bytes_bf16(ctx) * ctx->L;
    const int64_t r2 = (int64_t)2 * ctx->Hkv * (ctx->d + 16) * ctx->L;
    // T0 rows, T2 records in HBM (or their two staged layers), and the two staged layers of T1
    const int64_t t2_in_hbm = ctx->t2_host ? (int64_t)2 * ctx->B * ctx->hw2 * 2 * ctx->Hkv * (ctx->d + 16)
                                           : s.tier_count[2] * r2;
    const int64_t t1_layers = ctx->cfg.t1_transport == TKV_T1_RESIDENT ? ctx->L : 2;
    s.hbm_bytes_kv_resident = s.tier_count[0] * rb + t2_in_hbm +
                              t1_layers * ctx->B * ctx->hw1 * (int64_t)row_bytes_bf16(ctx);
    s.kv_bytes_full_cache = (int64_t)ctx->N * ctx->B * rb;
    s.kernel_launches = ctx->launches;
    s.status = ctx->status;
    s.attn_splits = ctx->last_splits;
    s.host_huge_bytes = (int64_t)(ctx->hs_h1.huge_bytes + ctx->hs_h2m.huge_bytes + ctx->hs_t2.huge_bytes);
    s.host_numa_node = ctx->host_numa;
    s.cuda_error = ctx->cuda_error;
    s.cuda_error_line = ctx->cuda_error_line;
    *out = s;
    return TKV_OK;
}

}  // extern "C"
