// Internal definitions shared by the tkv CUDA sources (not part of the C ABI).
//
// Device-memory layout (all row-major, innermost last):
//   T0 pool      k0v0  [L][2][B][Hkv][S0][d]        bf16   (2 = K, V)
//   T1 staging   stage [2][2][B][Hkv][S1][d]        bf16   (ring of 2 layers)
//   T2 pool      t2    [L][2][B][Hkv][S2][d + 16]   bytes: d E4M3 codes, then the
//                                                   fp32 scale and 12 bytes of padding
//   host T1      h1    [L][2][B][Hkv][S1][d]        bf16, pinned + mapped
//   host master  h2m   [L][2][B][Hkv][S2][d]        bf16, pinned + mapped: full-precision
//                                                   copy of every T2 row
//   page tables  tier [B][Nmax] u8, slot [B][Nmax] i32, s [B][Nmax] f32
//   retained     rl_loc [B][Nmax] u32 = tier << 30 | slot, rl_pos [B][Nmax] i32,
//                rl_count [B]  -- non-evicted positions in logical order
//   alpha sums   g [L][B][Hkv][Nmax] f32 (per retained index, this step)
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace tkv {

// Move kinds produced by a re-tier.
enum MoveKind : int {
    MV_T0_T1 = 1,   // write back a T0 row to the host T1 store      (at re-tier)
    MV_T0_T2 = 2,   // quantise a T0 row into T2, keep bf16 on host   (at re-tier)
    MV_T1_T2 = 3,   // quantise a host T1 row into T2, keep bf16      (at re-tier)
    MV_T2_T1 = 4,   // host master row -> host T1 store               (at re-tier)
    MV_T1_T0 = 5,   // host T1 row -> T0                              (delta prefetch)
    MV_T2_T0 = 6,   // host master row -> T0                          (delta prefetch)
};

// Per-sequence counters written by the re-tier kernel and read back once.
struct RetierOut {
    int32_t n_now;        // moves applied at re-tier time
    int32_t n_delta;      // moves left for the delta prefetch
    int32_t hw1;          // highest referenced T1 slot + 1
    int32_t hw2;          // highest referenced T2 slot + 1
    int32_t count[4];     // tokens per tier after the re-tier
    int32_t kinds[8];     // moves per kind
    int32_t error;        // 0 or a tkv_status
    int32_t pad[2];
};

// Per-sequence parameters of a re-tier (computed on the host).
struct RetierParams {
    int32_t forced;       // 1: take tiers from `forced_tiers`, 0: rank by s
    int32_t c0, c1, c2;   // ranked mode: candidates that go to T0 / T1 / T2
    int32_t n_cand;       // unprotected, not yet evicted positions
    int32_t pad[3];
};

__host__ __device__ constexpr inline uint32_t make_loc(int tier, int slot) {
    return ((uint32_t)tier << 30) | (uint32_t)slot;
}
__host__ __device__ inline int loc_tier(uint32_t loc) { return (int)(loc >> 30); }
__host__ __device__ inline int loc_slot(uint32_t loc) { return (int)(loc & 0x3FFFFFFFu); }

// Row index of (layer, kv, b, head, slot) in a [L][2][B][Hkv][S] store.
__host__ __device__ inline size_t row_index(int layer, int kv, int b, int h, int slot, int B,
                                            int Hkv, int S) {
    return ((((size_t)layer * 2 + kv) * B + b) * Hkv + h) * (size_t)S + slot;
}

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// bf16 pair packed in a 32-bit word -> two floats (exact).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Two E4M3 codes (low byte first) -> two floats (exact).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t w) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)w, __NV_E4M3);
    return __half22float2(*reinterpret_cast<__half2*>(&h));
}

}  // namespace tkv

// Launchers (defined in the .cu files, called by the host runtime).
namespace tkv {

struct AttnArgs {
    const __nv_bfloat16* q;      // [B][Hq][d]
    float* out;                  // [B][Hq][d]
    const __nv_bfloat16* k0v0;   // T0 pool (all layers)
    const __nv_bfloat16* stage;  // staging ring slot for this layer: [2][B][Hkv][S1][d]
    const uint8_t* t2;           // T2 records: the pool (all layers) or this layer's staging slot
    int t2_layer;                // layer index into t2: `layer` for the pool, 0 for a staging slot
    const __nv_bfloat16* new_k;  // [B][Hkv][d] this layer's decode-token K, written to its T0 slot
    const __nv_bfloat16* new_v;  //   by the CTA that owns the row (null: nothing to write)
    const uint32_t* rl_loc;      // [B][Nmax]
    const int32_t* rl_count;     // [B]
    float* g;                    // [B][Hkv][Nmax] per-position alpha sums, running over the step's layers
    float* part;                 // [B*Hkv][part_per_group][16 + G*d] softmax partials per (group, CTA of the group) (scratch)
    float* zs;                   // [B][Hkv][Nmax][GP] logits, log2-scaled (scratch)
    int32_t* err;                // status word (unused by kernels without device waits)
    int layer, L, B, Hq, Hkv, d, Nmax, S0, S1, S2;
    int items_per_group;         // ceil(max_b R_b / item_rows)
    int item_rows;               // rows per item: 64, 128 or 256
    int items_per_cta;           // contiguous items per CTA
    int grid;                    // CTAs of the main kernel
    int part_per_group;          // partial records per group (CTAs whose ranges can touch a group)
    float qscale;                // log2(e) / sqrt(d)
};

// Launch geometry shared by the context path and the allocation-free path.
struct AttnPlan {
    int item_rows, items_per_group, items_per_cta, grid, part_per_group;
    size_t smem;
};
// Plans a launch for B sequences x Hkv heads with at most rmax retained rows.
// `resident` = CTAs of the main kernel that fit on the device at once.
AttnPlan attention_plan(int G, int d, int B, int Hkv, int rmax, int resident);
size_t attention_part_floats(int G, int d, int B, int Hkv, int Nmax, int resident);   // scratch sizes
size_t attention_zs_floats(int G, int B, int Hkv, int Nmax);

// Launches the main kernel and the combine kernel.  If given, `after_main` is recorded between
// the two launches and `before_combine` right after it (event timing of each kernel).
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t st, cudaEvent_t after_main = nullptr,
                             cudaEvent_t before_combine = nullptr);
size_t attention_smem_bytes(int G, int d, int rl_rows);
int attention_max_window_rows();                                // retained rows a CTA can stage
cudaError_t attention_prepare(int G, int d, size_t smem);
int attention_resident_ctas(int G, int d, size_t smem);                  // CTAs per device
cudaError_t attention_ensure_smem(int G, int d, size_t smem);   // raises the cap, never lowers it

cudaError_t launch_fold(const float* g, const int32_t* rl_pos, const int32_t* rl_count, float* s,
                        int B, int Hkv, int Nmax, int rmax, float inv_lh, cudaStream_t st);

cudaError_t launch_open(int32_t* t0_free, int32_t* t0_top, uint8_t* tier, int32_t* slot, float* s,
                        uint32_t* rl_loc, int32_t* rl_pos, int32_t* rl_count, int32_t* pos_n, int B, int Nmax,
                        int S0, int n, cudaStream_t st, int* launches);

cudaError_t launch_append_rows(const __nv_bfloat16* k, const __nv_bfloat16* v,
                               __nv_bfloat16* k0v0, const int32_t* slot, int layer, int B,
                               int Hkv, int d, int Nmax, int S0, int N, int n, cudaStream_t st);

struct RetierArgs {
    const float* s;
    uint8_t* tier;
    int32_t* slot;
    const uint8_t* forced;       // [B][Nmax] or null
    const RetierParams* params;  // [B]
    uint8_t* new_tier;           // scratch [B][Nmax]
    int32_t* new_slot;           // scratch [B][Nmax]
    int32_t* free_scratch;       // scratch [B][max(S0,S1,S2)]
    uint32_t* rl_loc;
    int32_t* rl_pos;
    int32_t* rl_count;
    int32_t* t0_free;            // [B][S0]
    int32_t* t0_top;             // [B]
    uint32_t* resv1;             // [B][S1 words]
    uint32_t* resv2;             // [B][S2 words]
    int4* moves_now;             // [B][Nmax]
    int4* moves_delta;           // [B][Nmax]
    RetierOut* outp;             // [B]
    int B, N, Nmax, S0, S1, S2, prompt_len, num_sinks, window;
};

cudaError_t launch_retier(const RetierArgs& a, cudaStream_t st);
size_t retier_smem_bytes(int S0, int S1, int S2);
cudaError_t retier_prepare(size_t smem);

struct MoveArgs {
    const int4* moves;           // [B][Nmax]
    const int32_t* counts;       // per b: number of entries (stride count_stride ints)
    int count_stride;
    __nv_bfloat16* k0v0;
    uint8_t* t2;
    __nv_bfloat16* h1;           // device view of the host T1 store
    __nv_bfloat16* h2m;          // device view of the host master store
    __nv_bfloat16* t1_res;       // TKV_T1_RESIDENT: HBM copy of the T1 store [L][2][B][Hkv][S1][d], else null
    int layer_begin, layer_end;  // layers handled by this launch
    int L, B, Hkv, d, Nmax, S0, S1, S2;
    int max_count;
};

cudaError_t launch_moves(const MoveArgs& a, cudaStream_t st);

// Copies rows [row_begin, row_end) of a pitched 2-D region (16-byte units):
// dst[r * pitch16 + c] = src[r * pitch16 + c] for c < width16.
cudaError_t launch_t1_copy(const void* src, void* dst, size_t pitch16, size_t width16, int row_begin,
                           int row_end, cudaStream_t st);

}  // namespace tkv
