/*
 * tkv.h -- tiered KV-cache decode attention for one GB300 GPU (sm_103a).
 *
 * The method ("Not All Thoughts Need HBM: Semantics-Aware Memory Hierarchy
 * for LLM Reasoning"; gist.science summary and fugumt.com abstract) keeps
 * every token of a reasoning chain in one of four tiers:
 *
 *   T0  HBM, full precision (bf16)          -- protected tokens and the most
 *                                              important reasoning tokens
 *   T1  pinned host DDR, full precision     -- fetched back into HBM before
 *                                              each attention step (or read
 *                                              from an HBM copy the re-tier
 *                                              keeps: TKV_T1_RESIDENT)
 *   T2  8-bit (FP8-E4M3, one fp32 scale per token, layer and KV head, for K
 *       and for V), kept in HBM or in pinned host memory (TKV_T2_HOST) and
 *       dequantised inside the attention load
 *   T3  evicted (dropped from every store)
 *
 * ranked by the cumulative attention score
 *     s_i(t) = s_i(t-1) + (1/|L|) sum_l (1/H) sum_h alpha_{l,h}(t)[i]
 * ("Importance scoring") and re-tiered every Delta decode steps ("System
 * implementation", Delta = 64).  The prompt, the first `num_sinks` tokens and
 * the last `recent_window` tokens are protected and always in T0
 * ("Four-tier classification").
 *
 * Conventions for every call:
 *   - Device pointers are caller-owned CUDA device memory (e.g. a torch
 *     tensor's data_ptr()) and must stay valid until the work enqueued on the
 *     context's compute stream has completed.  Host pointers are caller-owned
 *     and are only read or written during the call.
 *   - All GPU work is enqueued asynchronously on the context's streams; calls
 *     return without waiting unless their comment says they synchronise.
 *   - No call aborts or traps.  Argument errors return TKV_EINVAL and change
 *     nothing.  The first CUDA error (or a device-side status word set by a
 *     kernel) poisons the context: that call returns TKV_ECUDA / TKV_ETIMEOUT /
 *     TKV_ECAPACITY and every later call except tkv_destroy, tkv_get_stats and
 *     tkv_status_string returns TKV_ESTATE.
 *   - One context is used from one host thread at a time.
 *   - Fault injection (a test hook for the error paths, host side only): if
 *     the environment variable TKV_FAULT_INJECT is set when tkv_create runs,
 *       "hostalloc"  makes that context's pinned host allocations fail
 *                    (tkv_create returns TKV_ENOMEM and frees what it took);
 *       "call:N"     makes the N-th checked CUDA call of that context (counted
 *                    from 1 after creation) report failure after it ran:
 *                    the call returns TKV_ECUDA, the context is poisoned
 *                    (tkv_stats.cuda_error = cudaErrorUnknown) and no device
 *                    work goes wrong.
 *
 * Shapes: L layers, B sequences, Hq query heads, Hkv KV heads, G = Hq / Hkv,
 * d = head_dim (64 or 128).  Query head h reads KV head h / G (GQA).
 * All sequences of a batch advance together: they hold the same number N of
 * positions.
 */
#ifndef TKV_H
#define TKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TKV_OK = 0,
    TKV_EINVAL = 1,     /* bad argument or call out of order; nothing changed */
    TKV_ENOMEM = 2,     /* device or pinned host allocation failed */
    TKV_ECUDA = 3,      /* a CUDA runtime call failed; context poisoned */
    TKV_ECAPACITY = 4,  /* a tier store or the position capacity is full */
    TKV_ETIMEOUT = 5,   /* a bounded device-side wait ran out; context poisoned */
    TKV_ESTATE = 6      /* context poisoned by an earlier error */
} tkv_status;

typedef struct tkv_ctx tkv_ctx;

/* T1 transports (tkv_config.t1_transport): the same bytes land in the same
 * staging rows either way, so results do not depend on the choice.
 *   TKV_T1_COPY_ENGINE  one cudaMemcpy2DAsync per layer on the copy stream
 *   TKV_T1_SM_COPY      a copy kernel on the copy stream whose threads load
 *                       the pinned host rows directly (zero-copy) and store
 *                       them to staging
 *   TKV_T1_SPLIT        half the rows by the copy engine, half by the copy
 *                       kernel on a second stream, concurrently
 *   TKV_T1_MULTI_CE     the rows split four ways over four copy streams, so
 *                       that several copy engines run at once
 *   TKV_T1_RESIDENT     the other reading of "System implementation": an HBM
 *                       copy of every layer's T1 rows is kept next to the host
 *                       store and updated by the re-tier's moves, so only the
 *                       delta crosses the host link (no per-step T1 stream;
 *                       T1 then occupies HBM like T0) */
enum { TKV_T1_COPY_ENGINE = 0, TKV_T1_SM_COPY = 1, TKV_T1_SPLIT = 2, TKV_T1_MULTI_CE = 3,
       TKV_T1_RESIDENT = 4 };

/* Where the T2 rows (E4M3 codes + fp32 scales) live (tkv_config.t2_placement):
 *   TKV_T2_HBM   in an HBM pool that the attention kernel reads in place
 *   TKV_T2_HOST  in pinned host memory, the placement "Four-tier
 *                classification" gives T2: each layer's T2 records are copied
 *                with its T1 rows into an HBM staging ring before its attention.
 * The same bytes reach the kernel either way, so the results are identical. */
enum { TKV_T2_HBM = 0, TKV_T2_HOST = 1 };

/* How the pinned host stores (T1 rows, full-precision copies of T2 rows, host
 * T2 records) are allocated (tkv_config.host_alloc):
 *   TKV_HOST_HUGE_ARENA    an anonymous mapping aligned to and populated with
 *                          transparent huge pages, bound to the host NUMA node
 *                          closest to the device when the host has several,
 *                          registered with cudaHostRegister (mapped, portable);
 *                          falls back to cudaHostAlloc if a step fails.  Huge
 *                          pages keep the host link's DMA translations few, so
 *                          the per-step copy of a store of tens of GB keeps to
 *                          the link's rate.
 *   TKV_HOST_PINNED_ALLOC  cudaHostAlloc (mapped, portable).
 *   TKV_HOST_AUTO          the huge-page arena for stores of 1 GiB or more,
 *                          cudaHostAlloc below (default).
 * The bytes stored are the same either way. */
enum { TKV_HOST_AUTO = 0, TKV_HOST_PINNED_ALLOC = 1, TKV_HOST_HUGE_ARENA = 2 };

typedef struct {
    int32_t num_layers;       /* L >= 1 */
    int32_t num_q_heads;      /* Hq, a multiple of num_kv_heads, Hq / Hkv <= 8 */
    int32_t num_kv_heads;     /* Hkv >= 1 */
    int32_t head_dim;         /* d: 64 or 128 */
    int32_t batch;            /* B >= 1 */
    int32_t max_tokens;       /* capacity of positions per sequence, <= 65536 */
    int32_t prompt_len;       /* protected prompt [0, prompt_len) */
    int32_t num_sinks;        /* protected attention sinks [0, num_sinks) */
    int32_t recent_window;    /* protected recent window [N - W, N) */
    int32_t retier_interval;  /* Delta; informational for callers (tkv_retier is explicit) */
    float ratio_t0;           /* tier shares of N; held internally as parts per million */
    float ratio_t1;
    float ratio_t2;
    float ratio_t3;
    int32_t t0_capacity;      /* HBM T0 slots per sequence; 0 = max_tokens */
    int32_t t1_capacity;      /* pinned-host T1 slots per sequence (and HBM staging rows); 0 = max_tokens */
    int32_t t2_capacity;      /* T2 slots per sequence; 0 = max_tokens if ratio_t2 > 0, else 0 */
    int32_t t1_transport;     /* how T1 rows reach the attention kernel: TKV_T1_COPY_ENGINE,
                                 TKV_T1_SM_COPY, TKV_T1_SPLIT, TKV_T1_MULTI_CE or TKV_T1_RESIDENT
                                 (see above) */
    int32_t device;           /* CUDA device ordinal */
    void* compute_stream;     /* cudaStream_t for attention, append, fold, re-tier; NULL = create a
                                 non-blocking one (then order the caller's work with tkv_sync);
                                 cudaStreamLegacy / cudaStreamPerThread are accepted */
    void* copy_stream;        /* cudaStream_t for T1 prefetch and delta prefetch; NULL = create one */
    int32_t t2_placement;     /* where T2 rows live: TKV_T2_HBM (0, default) or TKV_T2_HOST */
    int32_t host_alloc;       /* host stores: TKV_HOST_AUTO (0, default), TKV_HOST_PINNED_ALLOC or
                                 TKV_HOST_HUGE_ARENA (see above) */
} tkv_config;

typedef struct {
    int64_t num_tokens;            /* N: positions per sequence so far */
    int64_t step;                  /* decode steps completed */
    int64_t retiers;               /* re-tiers completed */
    int64_t tier_count[4];         /* tokens per tier, summed over the batch */
    int64_t t1_rows_streamed;      /* T1 slots copied per layer per sequence per step (high-water mark) */
    int64_t last_promoted;         /* last re-tier: tokens moved into T0 from T1/T2 (summed over batch) */
    int64_t last_demoted_t1;       /* last re-tier: tokens moved T0 -> T1 */
    int64_t last_quantised;        /* last re-tier: tokens moved into T2 */
    int64_t last_evicted;          /* last re-tier: tokens newly evicted */
    int64_t last_t2_to_t1;         /* last re-tier: tokens moved T2 -> T1 */
    int64_t h2d_bytes_t1_stream;   /* cumulative bytes of the per-layer T1 stream */
    int64_t h2d_bytes_delta;       /* cumulative bytes of delta prefetch (promotions) */
    int64_t d2h_bytes_writeback;   /* cumulative bytes written back to the host stores */
    int64_t hbm_bytes_allocated;   /* device bytes held by the context */
    int64_t host_bytes_allocated;  /* pinned host bytes held by the context */
    int64_t hbm_bytes_kv_resident; /* KV bytes in HBM now: T0 rows + T2 rows (or their two staged layers)
                                      + T1 staging (or the resident T1 copy) */
    int64_t kv_bytes_full_cache;   /* bf16 KV bytes of all N positions (no tiering) */
    int64_t kernel_launches;       /* kernels this context has launched (all kinds) */
    int32_t status;                /* tkv_status of the context */
    int32_t attn_splits;           /* CTAs of the last attention launch */
    int64_t h2d_bytes_t2_stream;   /* cumulative bytes of the per-layer T2 stream (TKV_T2_HOST) */
    int64_t host_huge_bytes;       /* bytes of the host stores backed by huge pages */
    int32_t host_numa_node;        /* NUMA node the host stores are bound to, -1 = none */
    int32_t cuda_error;            /* cudaError_t of the CUDA call that poisoned the context, 0 = none */
    int32_t cuda_error_line;       /* source line of that call in the library (diagnostics) */
    int32_t pad0;
} tkv_stats;

/* Creates a context: device pools for T0 (bf16), T2 (fp8 + scales) and the
 * two-deep T1 staging ring, pinned mapped host stores for T1 and for the
 * full-precision copy of T2 rows, page tables and the score vector s.
 * Every position starts in T0.  Ownership of *out passes to the caller.
 * Errors: TKV_EINVAL (shape/ratio checks), TKV_ENOMEM, TKV_ECUDA. */
tkv_status tkv_create(const tkv_config* cfg, tkv_ctx** out);

/* Frees everything the context holds (after synchronising its streams). */
void tkv_destroy(tkv_ctx* ctx);

/* Appends n_tokens new positions for one layer ("Four-tier classification":
 * new tokens fall in the recent window, so they enter T0).
 * k, v: device bf16 [B][n_tokens][Hkv][d].
 * k and v must be 16-byte aligned (TKV_EINVAL otherwise).
 * Protocol: a group of n tokens opens with layer 0 and every layer is
 * appended in order 0..L-1.  With n_tokens == 1 the group is a decode step:
 * tkv_decode_step(layer) follows tkv_append(layer), and the step closes after
 * tkv_decode_step(L-1).  A decode token's rows are written into T0 by the
 * attention kernel of that tkv_decode_step (no launch of their own), so k and v
 * must stay valid and unchanged until that call's work has run on the compute
 * stream.  With n_tokens > 1 (prefill) the rows are copied on the compute
 * stream at once and the positions are committed when layer L-1 is appended;
 * pre-filled positions start with s = 0 and are not scored.
 * Errors: TKV_EINVAL (layer out of order, NULL pointers, n_tokens < 1),
 * TKV_ECAPACITY (max_tokens or T0 capacity would be exceeded; nothing changes). */
tkv_status tkv_append(tkv_ctx* ctx, int32_t layer, const void* k, const void* v,
                      int32_t n_tokens);

/* Enqueues, on the copy stream, the fetch of `layer`'s T1 rows (full
 * precision, pinned host -> HBM staging slot layer % 2) and, on the first step
 * after a re-tier, the delta prefetch of the rows newly promoted into T0 for
 * that layer ("Zero-approximation-error offloading": T1 rows are fetched
 * before each attention step; "System implementation": asynchronous delta
 * prefetch of newly promoted tokens only).  Call it for layer l+1 before
 * tkv_decode_step(l) so the copy overlaps layer l's attention; if it was not
 * called, tkv_decode_step(layer) issues it itself.  Layers may be prefetched
 * in any order (at most two layers ahead of the attention): each layer's
 * delta is enqueued, once, before that layer's fetch completes.
 * Errors: TKV_EINVAL (layer out of range, or called twice for one layer in
 * one step). */
tkv_status tkv_prefetch(tkv_ctx* ctx, int32_t layer);

/* Decode attention of one layer for the open decode step, over all retained
 * positions (T0, T1, T2; T3 excluded) in logical order, with the softmax
 * scale 1/sqrt(d).  Also emits, per retained position, the sum over this
 * layer's query heads of the attention weights, and on the last layer folds
 * them into s ("Importance scoring").  The result does not depend on which of
 * T0 / T1 a token sits in (Proposition 1): the work split and the order of
 * every sum depend only on the retained set.
 * q: device bf16 [B][Hq][d].  out: device fp32 [B][Hq][d].
 * Errors: TKV_EINVAL (no open decode step, layer not yet appended, or out of
 * order), TKV_ECUDA. */
tkv_status tkv_decode_step(tkv_ctx* ctx, int32_t layer, const void* q, float* out);

/* Re-tiers every sequence by its current scores ("System implementation":
 * every Delta = 64 decode steps; the caller calls it when step % Delta == 0,
 * after tkv_decode_step(L-1)).  Ranking key: s descending, lower position
 * first on exact ties.  Counts: n_k = floor(ratio_k * N) with ratios held in
 * parts per million; T0's count includes the protected set; T3 is cumulative
 * and never gives a token back; after evictions T0, then T2, take their
 * targets from the ranked list and T1 takes the remainder (T1 shrinks first,
 * then T2, if the protected set is too large).
 * Rows leaving T0 are written back to the host store or quantised here; rows
 * entering T0 are fetched by the next step's tkv_prefetch.  Synchronises the
 * compute stream once (reads back the move counts).
 * Errors: TKV_EINVAL (a decode step or prefill group is open),
 * TKV_ECAPACITY (a tier store is full; context poisoned), TKV_ECUDA. */
tkv_status tkv_retier(tkv_ctx* ctx);

/* Copies s to the host: dst [B][N] fp32.  Synchronises. */
tkv_status tkv_get_scores(tkv_ctx* ctx, float* dst_host);

/* Replaces s from the host: src [B][N] fp32 (test hook: feed given scores to
 * the re-tier).  Synchronises. */
tkv_status tkv_set_scores(tkv_ctx* ctx, const float* src_host);

/* Copies the tier of every position to the host: dst [B][N] uint8 (0..3).
 * Synchronises. */
tkv_status tkv_get_tiers(tkv_ctx* ctx, uint8_t* dst_host);

/* Moves every position to the given tier (test hook, e.g. for Proposition 1:
 * same T3 set, different T0/T1 splits): src [B][N] uint8.  Data moves exactly
 * as in tkv_retier.  An evicted position cannot be given back a tier, and a
 * protected position (sinks, prompt, recent window at the current N) cannot be
 * evicted (TKV_EINVAL, nothing changes).  Synchronises. */
tkv_status tkv_set_tiers(tkv_ctx* ctx, const uint8_t* src_host);

/* Inspection hook: copies the stored K and V rows of one position of one
 * layer and sequence, from wherever its tier keeps them, to the host, and
 * returns its tier in *tier_out.
 *   T0 / T1: dst_host receives bf16 [2][Hkv][d] (K rows, then V rows) from
 *            the HBM T0 pool or the pinned host T1 store; scales untouched.
 *   T2:      dst_host receives the E4M3 codes uint8 [2][Hkv][d] and
 *            scales_host the fp32 scales [2][Hkv] from the HBM T2 pool.
 *   T3:      nothing is copied.
 * dst_host must hold 2*Hkv*d*2 bytes; scales_host 2*Hkv floats (may be NULL
 * when the caller knows the position is not in T2).  Synchronises.
 * Errors: TKV_EINVAL (indices out of range). */
tkv_status tkv_get_row(tkv_ctx* ctx, int32_t layer, int32_t seq, int32_t pos, void* dst_host,
                       float* scales_host, int32_t* tier_out);

/* Time and bytes of one kind of work between tkv_profile_begin and _end. */
typedef struct {
    double ms;          /* summed CUDA-event time of the timed launches or copies */
    int64_t count;      /* launches or copies timed */
    double bytes;       /* algorithmic bytes they moved */
} tkv_prof_entry;

/* Kernel and copy timing.  tkv_profile_begin clears the counters and, until
 * tkv_profile_end, brackets with CUDA events (at most 16384 of each kind):
 *   attn   -- every launch of the attention main kernel, on the compute
 *             stream, right around the kernel (after its wait for the T1
 *             fetch).  Bytes per launch and sequence: 4*Hkv*d per T0/T1 row,
 *             2*Hkv*d + 8*Hkv per T2 row (codes + two fp32 scales), plus q
 *             (bf16);
 *   combine -- every launch of the attention combine kernel that follows it
 *             (the bracket between the two kernels keeps them from
 *             overlapping while timed); bytes: out (fp32) plus, per retained
 *             row and KV head, its logits and its alpha running sum;
 *   t1     -- every per-layer T1 copy (pinned host -> HBM staging) on the
 *             copy stream; bytes = rows copied * 4*Hkv*d;
 *   delta  -- every delta-prefetch gather of promoted rows on the copy stream;
 *             bytes = rows gathered * 4*Hkv*d.
 * tkv_profile_end synchronises, stops recording and fills the entries (any
 * pointer may be NULL). */
tkv_status tkv_profile_begin(tkv_ctx* ctx);
tkv_status tkv_profile_end(tkv_ctx* ctx, tkv_prof_entry* attn, tkv_prof_entry* combine,
                           tkv_prof_entry* t1, tkv_prof_entry* delta);

/* Allocation-free decode step for callers that cannot let a library allocate
 * device memory: runtimes whose caching allocator owns the whole memory
 * budget, and decode loops that cannot afford the device-wide stalls that
 * cudaMalloc / cudaFree may cause.  The paper has no counterpart: this is a
 * packaging of the same attention kernel and score fold as tkv_decode_step,
 * over a dense cache in which every position is retained and resident.
 *   q:   device bf16 [L][B][Hq][d]
 *   kv:  device bf16 [L][2][B][Hkv][R][d]   (K rows, then V rows; positions
 *        0..R-1 in logical order, the decoded token included), 16-byte aligned
 *   out: device fp32 [L][B][Hq][d]
 *   s:   device fp32 [B][R], read and updated in place: s += the step's mean
 *        over layers and query heads of the attention weights
 *   stream: cudaStream_t to enqueue on (NULL = the legacy default stream)
 * Scratch lives in fixed file-scope device arrays (about 34 MiB), held by
 * every GPU that loads the library until exit: B*Hkv*R <= 131,072,
 * B*R <= 131,072, B <= 256; larger sizes return TKV_ECAPACITY before anything
 * is enqueued.
 * It calls no cudaMalloc, cudaFree or other allocating routine.  The first
 * call on a device (with that device current) resolves the scratch addresses
 * and should come before any stream capture.  All calls share the scratch and
 * leave their contents in it, so calls that overlap on the GPU race.  The call
 * enqueues work and returns without waiting.
 * Errors: TKV_EINVAL (NULL pointers, a misaligned kv, shapes), TKV_ECAPACITY
 * (beyond the limits above), TKV_ECUDA. */
tkv_status tkv_decode_dense_noalloc(const void* q, const void* kv, float* out, float* s,
                                    int32_t num_layers, int32_t batch, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t num_positions,
                                    void* stream);

/* CUDA-graph decode steps.  The pages have no counterpart: this is how a
 * serving loop takes the host-side cost of the per-layer calls (and the gaps
 * between launches) off a decode step.
 * tkv_capture_begin: between decode steps, with no delta prefetch pending
 * (i.e. not on the first step after a re-tier), profiling off and any T1
 * transport but TKV_T1_SPLIT.  The caller then makes one
 * decode step's calls (tkv_append / tkv_prefetch / tkv_decode_step for every
 * layer) as usual: they are recorded into a graph, on an internal stream, and
 * nothing runs.  tkv_capture_end instantiates the graph, puts the context back
 * to its state before the step and sets *steps_valid to the number of
 * replays the graph stays valid for (the launch geometry covers the retained
 * counts; capacity).  tkv_replay launches the graph on the compute stream: one
 * decode step, with the pointers given at capture (the caller refills those
 * buffers before each replay).  Any re-tier, tkv_set_tiers or prefill append
 * discards the graph.
 * Errors: TKV_EINVAL (call order, conditions above, no valid graph, the
 * captured calls were not exactly one decode step), TKV_ECUDA. */
tkv_status tkv_capture_begin(tkv_ctx* ctx);
tkv_status tkv_capture_end(tkv_ctx* ctx, int32_t* steps_valid);
tkv_status tkv_replay(tkv_ctx* ctx);

/* Measurement hook (no counterpart on the pages, which quote PCIe Gen5 x16 for
 * their prototype's host link): the bandwidth of this device's host link as
 * seen by the two ways the library moves host rows.  Allocates `bytes` of
 * pinned mapped host memory and of device memory, times the best of three
 * passes of each kind with CUDA events on a stream of its own, frees both and
 * synchronises:
 *   h2d_ce_gbs  one cudaMemcpyAsync, pinned host -> device (the copy engine
 *               that carries the per-layer T1 stream);
 *   h2d_sm_gbs  the library's copy kernel loading the mapped host buffer
 *               (zero-copy; the path the delta prefetch and TKV_T1_SM_COPY use);
 *   d2h_ce_gbs  one cudaMemcpyAsync, device -> pinned host.
 * GB/s = 1e9 bytes per second.  Any output pointer may be NULL.
 * Errors: TKV_EINVAL (bytes < 1 MiB or not a multiple of 16, device < 0),
 * TKV_ENOMEM, TKV_ECUDA. */
tkv_status tkv_measure_host_link(int32_t device, int64_t bytes, double* h2d_ce_gbs, double* h2d_sm_gbs,
                                 double* d2h_ce_gbs);

/* Waits for all enqueued work and reports any device-side status word. */
tkv_status tkv_sync(tkv_ctx* ctx);

/* Counters and sizes; valid on a poisoned context too. */
tkv_status tkv_get_stats(tkv_ctx* ctx, tkv_stats* out);

/* Static string for a status code. */
const char* tkv_status_string(tkv_status s);

#ifdef __cplusplus
}
#endif

#endif /* TKV_H */
