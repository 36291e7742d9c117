// Allocation-free decode step: tkv_decode_dense_noalloc.
//
// Some callers cannot let a library call cudaMalloc: a serving runtime whose
// caching allocator owns the whole device-memory budget (memory the library
// takes behind its back is not in that budget and can make the runtime's own
// allocations fail), and latency-critical decode loops, because cudaMalloc and
// cudaFree can synchronise the device and stall every stream on it.  This
// entry point serves them: it runs the same attention kernel and score fold
// as the context path, but its scratch -- the per-layer sums of attention
// weights, the retained-index table and the per-sequence counts -- lives in
// file-scope __device__ arrays of fixed size that every GPU which loads the
// library holds until the process exits.
//
// Set-up: the first call on a device (with that device current) resolves the
// arrays' device addresses with cudaGetSymbolAddress and sets the attention
// kernel's shared-memory limit; that first call should therefore come before
// any stream capture.
// Every call shares the arrays and leaves its contents in them; calls that
// overlap on the GPU (for example on two streams) race on them.
#include <cmath>
#include <mutex>

#include "../../include/tkv.h"
#include "tkv_internal.cuh"

using namespace tkv;

namespace {

constexpr size_t kMaxGroupRows = size_t(1) << 17;     // B*Hkv*R    <= 131,072
constexpr size_t kMaxAlphaFloats = kMaxGroupRows;     // per-row alpha sums over layers (0.5 MiB)
constexpr size_t kMaxTable = size_t(1) << 17;         // B*R        <= 131,072    (0.5 MiB)
constexpr int kMaxBatch = 256;
constexpr size_t kMaxZsFloats = kMaxGroupRows * 8;    // logits, 8 per row      (4 MiB)
// softmax partials: B*Hkv*part_per_group records of (16 + G*d) floats; this bound covers
// B*Hkv*R <= 131,072 at the usual shapes, larger plans return TKV_ECAPACITY (checked per call)
constexpr size_t kMaxPartFloats = (kMaxGroupRows / 128 + 2048 + 4096 + 64) * (16 + 8 * 128);   // ~29 MiB

static __device__ __align__(256) float g_alpha_scratch[kMaxAlphaFloats];
static __device__ __align__(256) float g_zs_scratch[kMaxZsFloats];
static __device__ __align__(256) float g_part_scratch[kMaxPartFloats];
static __device__ __align__(256) uint32_t g_index_scratch[kMaxTable];
static __device__ __align__(256) int32_t g_count_scratch[kMaxBatch];
static __device__ __align__(256) int32_t g_status_scratch[1];

struct DevScratch {
    bool ready = false;
    float* alpha = nullptr;
    float* zs = nullptr;
    float* part = nullptr;
    uint32_t* index = nullptr;
    int32_t* count = nullptr;
    int32_t* status = nullptr;
};

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
DevScratch g_dev[kMaxDevices];

// Retained index j of sequence b at [b * R + j] (all rows live in T0 slot j),
// count R per sequence, status word cleared.
__global__ void noalloc_fill_kernel(uint32_t* index, int32_t* count, int32_t* status, int B, int R) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < B * R) index[i] = make_loc(0, i % R);
    if (i < B) count[i] = R;
    if (i == 0) status[0] = 0;
}

tkv_status setup(int dev, DevScratch** out) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    DevScratch& s = g_dev[dev];
    if (!s.ready) {
        if (cudaGetSymbolAddress((void**)&s.alpha, g_alpha_scratch) != cudaSuccess ||
            cudaGetSymbolAddress((void**)&s.zs, g_zs_scratch) != cudaSuccess ||
            cudaGetSymbolAddress((void**)&s.part, g_part_scratch) != cudaSuccess ||
            cudaGetSymbolAddress((void**)&s.index, g_index_scratch) != cudaSuccess ||
            cudaGetSymbolAddress((void**)&s.count, g_count_scratch) != cudaSuccess ||
            cudaGetSymbolAddress((void**)&s.status, g_status_scratch) != cudaSuccess) {
            (void)cudaGetLastError();
            return TKV_ECUDA;
        }
        s.ready = true;
    }
    *out = &s;
    return TKV_OK;
}

}  // namespace

extern "C" tkv_status tkv_decode_dense_noalloc(const void* q, const void* kv, float* out, float* s,
                                               int32_t num_layers, int32_t batch, int32_t num_q_heads,
                                               int32_t num_kv_heads, int32_t head_dim,
                                               int32_t num_positions, void* stream) {
    const int L = num_layers, B = batch, Hq = num_q_heads, Hkv = num_kv_heads, d = head_dim;
    const int R = num_positions;
    if (!q || !kv || !out || !s) return TKV_EINVAL;
    if (reinterpret_cast<uintptr_t>(kv) & 15u) return TKV_EINVAL;   // rows are copied in 16-byte units
    if (L < 1 || B < 1 || Hkv < 1 || Hq < 1 || R < 1 || Hq % Hkv || Hq / Hkv > 8 || (d != 64 && d != 128))
        return TKV_EINVAL;
    // size limits of the fixed scratch
    if (B > kMaxBatch || (size_t)B * R > kMaxTable || (size_t)B * Hkv * R > kMaxGroupRows)
        return TKV_ECAPACITY;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return TKV_ECUDA;
    }
    DevScratch* sc = nullptr;
    tkv_status st0 = setup(dev, &sc);
    if (st0 != TKV_OK) return st0;
    cudaStream_t st = (cudaStream_t)stream;
    const int G = Hq / Hkv;

    // same launch plan as the context path
    const size_t smem_max = attention_smem_bytes(G, d, attention_max_window_rows());
    if (attention_ensure_smem(G, d, smem_max) != cudaSuccess) {
        (void)cudaGetLastError();
        return TKV_ECUDA;
    }
    const int resident = attention_resident_ctas(G, d, smem_max);
    if (resident < 1) return TKV_ECUDA;
    const AttnPlan plan = attention_plan(G, d, B, Hkv, R, resident);
    if (attention_part_floats(G, d, B, Hkv, R, resident) > kMaxPartFloats) return TKV_ECAPACITY;

    noalloc_fill_kernel<<<(B * R + 255) / 256, 256, 0, st>>>(sc->index, sc->count, sc->status, B, R);
    if (cudaGetLastError() != cudaSuccess) return TKV_ECUDA;
    AttnArgs a{};
    a.out = out;
    a.k0v0 = (const __nv_bfloat16*)kv;
    a.stage = nullptr;
    a.t2 = nullptr;
    a.rl_loc = sc->index;
    a.rl_count = sc->count;
    a.g = sc->alpha;
    a.part = sc->part;
    a.zs = sc->zs;
    a.err = sc->status;
    a.L = L; a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.d = d;
    a.Nmax = R; a.S0 = R; a.S1 = 0; a.S2 = 0;
    a.item_rows = plan.item_rows;
    a.items_per_group = plan.items_per_group;
    a.items_per_cta = plan.items_per_cta;
    a.grid = plan.grid;
    a.part_per_group = plan.part_per_group;
    a.qscale = (float)(1.4426950408889634 / std::sqrt((double)d));
    for (int l = 0; l < L; ++l) {
        a.layer = l;
        a.q = (const __nv_bfloat16*)q + (size_t)l * B * Hq * d;
        a.out = out + (size_t)l * B * Hq * d;
        if (launch_attention(a, st) != cudaSuccess) {
            (void)cudaGetLastError();
            return TKV_ECUDA;
        }
    }
    const float inv = (float)(1.0 / ((double)L * (double)Hq));
    // The fold maps retained index j to its position through an int32 table.  Here every
    // entry of the retained-index table is make_loc(0, j): tier bits 0 and slot j, which is
    // the integer j itself, so the same words serve as that position table.
    static_assert(sizeof(uint32_t) == sizeof(int32_t) && make_loc(0, 1) == 1u &&
                      make_loc(0, (int)(kMaxTable - 1)) == (uint32_t)(kMaxTable - 1),
                  "a T0 location word equals its slot, so the index table doubles as positions");
    if (launch_fold(sc->alpha, (const int32_t*)sc->index, sc->count, s, B, Hkv, R, R, inv, st) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return TKV_ECUDA;
    }
    return TKV_OK;
}
