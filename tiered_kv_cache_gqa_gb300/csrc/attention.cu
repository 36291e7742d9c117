// Decode attention over the tiered KV cache, with the per-position sums of
// the attention weights that feed the score update, and the score fold.
//
// Method: "Not All Thoughts Need HBM" (gist.science summary), sections
// "Zero-approximation-error offloading" (T1 rows take part at full precision;
// Proposition 1: the result depends on the evicted set only) and "Importance
// scoring" (s_i += mean over layers and heads of alpha[i]); ARKV summary,
// "Tri-state cache assignment" (8-bit rows are dequantised on the fly and taken
// in their original order).
//
// Work split.  The retained list of every (sequence b, KV head) group is cut
// into items of `item_rows` consecutive positions.  The main kernel runs
// persistent CTAs of four warps; CTA c owns a contiguous range of items in
// (b, KV head, item) order.  Within an item, warp w owns the tiles w, w + 4,
// ... of 16 rows (32 in the compact instantiation).  Each warp streams, item
// after item, the K rows and then the V rows of its tiles through its own
// shared-memory ring (4 slots of 16-row tiles, or 2 of 32) with 16-byte
// cp.async (16 lanes per 256-byte row, every row fetched from its home: T0
// pool, T1 staging or T2 records; the group's decode token from the caller's
// k/v, stored into its T0 slot from the ring), so the next tiles -- possibly
// of the next item -- are in flight while the current one is computed.  The
// only waits are cp.async.wait_group and CTA barriers; there are no spin loops.
//   K tile:  tensor cores (mma.m16n8k16, bf16 operands, fp32 accumulators):
//            S^T = K q^T for the tile's rows and the group's query heads,
//            K from the ring by ldmatrix, q^T in registers; z = S^T *
//            log2(e)/sqrt(d) (times the record's scale for a T2 row, whose
//            E4M3 codes are first widened in place to bf16, exactly).
//   stats:   per warp and group, online over its tiles: m_h = max z,
//            p = 2^(z - m_h), l_h = sum p; z goes to a global scratch for the
//            alpha sums.
//   V tile:  O^T += V^T p^T on the tensor cores, V^T by a transposing
//            ldmatrix, p^T from the score fragment by movmatrix; p enters as
//            two bf16 parts p = hi + lo (about 16 significant bits), each with
//            its own product into the same fp32 accumulators.  Absent rows of
//            a partial tile are zero-filled by the copy.
//   group end: the four warps' (m, l, O) are merged in shared memory (fixed
//            order) into the CTA's partial for the group, stored at (group,
//            the CTA's rank among the CTAs that touch the group).
// The combine kernel then merges a group's partials in CTA order into `out`,
// and adds per position g = sum_h 2^(z_h - M_h) / L_h (the sum over the group's
// query heads of alpha) to a running sum over the step's layers.  Item
// boundaries, the CTA ranges and every reduction order depend only on the
// retained counts, never on which tier a row sits in, so a row read from T0 or
// from T1 staging gives bit-identical results.  No atomics touch `out` or `g`.
// Launches in which a CTA streams at most 256 rows use a compact instantiation
// (32-row tiles in two ring slots, partly unrolled issue loops); the launch plan,
// and with it the instantiation, depends on the retained counts only.
#include <algorithm>
#include <cmath>

#include "tkv_internal.cuh"

namespace tkv {

constexpr int kAttnWarps = 4;
constexpr int kRingRows = 64;             // rows of a warp's ring: 4 slots of 16-row tiles (three in
                                          // flight while one is used), or, in the compact instantiation,
                                          // 2 slots of 32-row tiles (fewer serial steps per warp)
constexpr int kMaxSlots = 4;
constexpr int kCompactRows = 256;         // CTA windows up to this many rows use the compact instantiation
constexpr int kMinItemRows = 128;         // item sizes: 128 or 256 rows
constexpr int kMaxWindowRows = 3584;       // retained-list rows a CTA stages in shared memory
                                           // (two CTAs of the largest instantiation fit an SM)
constexpr int kCombineThreads = 256;       // combine block size (one out element per thread)
constexpr int kCombineRowsPerThread = 4;   // alpha rows per combine thread
constexpr int kCombineRows = kCombineThreads * kCombineRowsPerThread;

template <int G, int D>
struct AttnCfg {
    static constexpr int GP = (G <= 4) ? 4 : 8;      // z row stride (floats)
    static constexpr int ROWB = 2 * D + 16;          // ring row stride (bytes): 8 consecutive rows
                                                     // hit 8 different 16-byte bank groups
    static_assert(D == 64 || D == 128, "head_dim must be 64 or 128");
    static_assert(G >= 1 && G <= 8, "group size must be 1..8");

    static constexpr size_t sz_warp_ring = (size_t)kRingRows * ROWB;
    static constexpr int PS = 16 + G * D;            // floats of one (m[8], l[8], O[G][D]) record
    static constexpr size_t off_ring = 0;
    static constexpr size_t off_comb = kAttnWarps * sz_warp_ring;
    static constexpr size_t off_n = off_comb + (size_t)PS * 4;   // rows of each item
    // per item: rows, decode-token flag, (sequence << 16 | KV head)
    static constexpr size_t off_mask = off_n + (size_t)(kMaxWindowRows / kMinItemRows) * 3 * 4;   // T2 rows per ring slot
    static constexpr size_t off_rl = off_mask + (size_t)kAttnWarps * kMaxSlots * 4;

    static size_t smem(int rl_rows) { return off_rl + (size_t)rl_rows * 4; }
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// 4 bytes global -> shared
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
// 16 zero bytes into shared memory (a source size of 0: nothing is read from `src`)
__device__ __forceinline__ void cp_async16_zero(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(0) : "memory");
}
// four 8 x 8 bf16 matrices from shared memory (lanes 8i..8i+7 address the rows of matrix i)
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}
// the same, each matrix transposed on the way
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}
// transpose of an 8 x 8 bf16 matrix held one (row, column pair) per lane
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
// c += A (16 x 16, bf16) * B (16 x 8, bf16), fp32 accumulators
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Widens every T2 record of a ring stage (`mask`: its rows) in place to a row of D bf16
// values (every E4M3 value is exact in bf16), the whole warp on one record at a time, D / 32
// codes a lane; a record is D E4M3 codes followed by its fp32 scale.  `sc[i]` of the lanes
// that hold tile row gq + 8 i in the product fragments is multiplied by that row's scale.
template <int D, int ROWB, int NR>
__device__ __forceinline__ void widen_t2_rows(uint8_t* stage, uint32_t mask, int lane, int gq, float (&sc)[NR]) {
    while (mask != 0u) {
        const int r = __ffs(mask) - 1;
        mask &= mask - 1u;
        uint8_t* row = stage + (size_t)r * ROWB;
        const float scale = *reinterpret_cast<const float*>(row + D);
        if constexpr (D == 128) {
            const uint32_t w = reinterpret_cast<const uint32_t*>(row)[lane];
            const float2 lo = e4m3x2_to_float2((uint16_t)(w & 0xFFFFu));
            const float2 hi = e4m3x2_to_float2((uint16_t)(w >> 16));
            const __nv_bfloat162 blo = __floats2bfloat162_rn(lo.x, lo.y);
            const __nv_bfloat162 bhi = __floats2bfloat162_rn(hi.x, hi.y);
            __syncwarp();   // every lane has read its codes before any bf16 word lands on them
            reinterpret_cast<uint2*>(row)[lane] =
                make_uint2(*reinterpret_cast<const uint32_t*>(&blo), *reinterpret_cast<const uint32_t*>(&bhi));
        } else {
            const uint16_t w = reinterpret_cast<const uint16_t*>(row)[lane];
            const float2 f = e4m3x2_to_float2(w);
            const __nv_bfloat162 bf = __floats2bfloat162_rn(f.x, f.y);
            __syncwarp();
            reinterpret_cast<uint32_t*>(row)[lane] = *reinterpret_cast<const uint32_t*>(&bf);
        }
#pragma unroll
        for (int i = 0; i < NR; ++i)
            if (r == gq + 8 * i) sc[i] *= scale;
    }
    __syncwarp();
}

// COMPACT: 32-row tiles in two ring slots and partly unrolled issue loops, for launches in
// which a CTA streams at most 256 rows: there every warp runs one or two tiles, so fewer serial
// steps per warp pay, and the code runs about once per launch, so the instruction cache, not
// the arithmetic, sets its pace.
template <int G, int D, bool COMPACT>
__global__ void __launch_bounds__(kAttnWarps * 32, 3) attn_kernel(const AttnArgs a) {
    using C = AttnCfg<G, D>;
    constexpr int GP = C::GP, ROWB = C::ROWB, PS = C::PS;
    constexpr int kIssueUnroll = COMPACT ? 4 : 8;
    constexpr int kTileRows = COMPACT ? 32 : 16;        // rows per pipeline tile
    constexpr int kWarpStages = kRingRows / kTileRows;  // ring slots
    constexpr size_t kStageBytes = (size_t)kTileRows * ROWB;
    constexpr int MT = kTileRows / 16;                  // 16-row blocks of a tile
    constexpr int NT = kAttnWarps * 32;
    extern __shared__ __align__(128) uint8_t smem[];
    float* comb = reinterpret_cast<float*>(smem + C::off_comb);
    uint32_t* rl_s = reinterpret_cast<uint32_t*>(smem + C::off_rl);
    int* n_s = reinterpret_cast<int*>(smem + C::off_n);
    int* own_s = n_s + kMaxWindowRows / kMinItemRows;
    int* bk_s = n_s + 2 * (kMaxWindowRows / kMinItemRows);

    // the combine kernel may be scheduled once every CTA of this grid has started
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int IT = a.item_rows, IPG = a.items_per_group;
    const int total_items = a.B * a.Hkv * IPG;
    const int it0 = blockIdx.x * a.items_per_cta;
    const int it1 = min(total_items, it0 + a.items_per_cta);
    if (it0 >= it1) return;
    uint8_t* ring = smem + C::off_ring + (size_t)warp * C::sz_warp_ring;

    // Prologue in one round trip: the rows of every item, and the retained-list slices copied
    // straight into shared memory by 4-byte cp.async, all in flight at once (read up to the
    // item size, clamped to the capacity; entries past the count are never used).
    for (int item = it0 + tid; item < it1; item += NT) {
        const int g = item / IPG, b = g / a.Hkv, j0 = (item % IPG) * IT;
        const int R = a.rl_count[b];
        n_s[item - it0] = max(0, min(IT, R - j0));
        // the group's decode token (its last retained row) falls in this item
        own_s[item - it0] = (a.new_k != nullptr && R - 1 >= j0 && R - 1 < j0 + IT) ? 1 : 0;
        bk_s[item - it0] = (b << 16) | (g % a.Hkv);
    }
    for (int i = tid; i < (it1 - it0) * IT; i += NT) {
        const int item = it0 + i / IT, j = (item % IPG) * IT + i % IT;
        const int b = item / IPG / a.Hkv;
        if (j < a.Nmax) cp_async4(smem_u32(rl_s + i), a.rl_loc + (size_t)b * a.Nmax + j);
    }
    cp_async_commit();
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    // tiles of this warp in an item: warp, warp + 4, ... below ceil(n / kTileRows)
    auto warp_tiles = [&](int n) {
        const int nt = (n + kTileRows - 1) / kTileRows;
        return warp < nt ? (nt - warp + kAttnWarps - 1) / kAttnWarps : 0;
    };

    // row (within tile `tile` of item) of the group's decode token, or -1
    auto new_row_in = [&](int item, int tile) {
        const int n = n_s[item - it0];
        const int r = n - 1 - tile * kTileRows;
        return (own_s[item - it0] && r >= 0 && r < kTileRows) ? r : -1;
    };

    // ------------------------------------------------------------ issue side
    // Sequence per warp: for every item, for every tile of this warp: K tile, V tile.
    int ci_item = it0, ci_k = 0, ci_kv = 0, issued = 0;
    auto settle = [&]() {
        while (ci_item < it1 && warp_tiles(n_s[ci_item - it0]) == 0) ++ci_item;
    };
    settle();
    const uint8_t* k0v0 = reinterpret_cast<const uint8_t*>(a.k0v0);
    const uint8_t* stg = reinterpret_cast<const uint8_t*>(a.stage);
    const uint8_t* row_v = nullptr;    // the lane's V row of the tile whose K was issued last
    int row_bytes = 0;
    bool all_bf16_issue = false;       // the tile last issued as K has kTileRows bf16 rows (its K and V
                                       // copies take the fast path)
    uint32_t* mask_s = reinterpret_cast<uint32_t*>(smem + C::off_mask) + warp * kWarpStages;
    // Copies the next tile of this warp's sequence: 16 lanes per 256-byte row, 16 bytes
    // a lane; a row's source pointer travels by shuffle with its kind in the low bits
    // (bit 0: T2 record of D + 16 bytes, bit 1: no row).
    auto issue_next = [&]() {
        if (ci_item >= it1) return;
        const int item = ci_item, kv = ci_kv;
        const int n = n_s[item - it0];
        const int tile = warp + kAttnWarps * ci_k;
        const int jl = tile * kTileRows + lane;
        const uint8_t* src = nullptr;
        if (kv == 0) {
            const int bk = bk_s[item - it0], b = bk >> 16, kvh = bk & 0xFFFF;
            row_bytes = 0;
            bool fp8 = false;
            if (lane < kTileRows && jl < n) {
                const uint32_t loc = rl_s[(size_t)(item - it0) * IT + jl];
                const int tier = loc_tier(loc), slot = loc_slot(loc);
                if (tier == 0) {
                    src = k0v0 + row_index(a.layer, 0, b, kvh, slot, a.B, a.Hkv, a.S0) * (2 * D);
                    row_v = k0v0 + row_index(a.layer, 1, b, kvh, slot, a.B, a.Hkv, a.S0) * (2 * D);
                    row_bytes = 2 * D;
                } else if (tier == 1) {
                    src = stg + row_index(0, 0, b, kvh, slot, a.B, a.Hkv, a.S1) * (2 * D);
                    row_v = stg + row_index(0, 1, b, kvh, slot, a.B, a.Hkv, a.S1) * (2 * D);
                    row_bytes = 2 * D;
                } else {
                    src = a.t2 + row_index(a.t2_layer, 0, b, kvh, slot, a.B, a.Hkv, a.S2) * (D + 16);
                    row_v = a.t2 + row_index(a.t2_layer, 1, b, kvh, slot, a.B, a.Hkv, a.S2) * (D + 16);
                    row_bytes = D + 16;
                    fp8 = true;
                }
                if (lane == new_row_in(item, tile)) {
                    // not in its T0 slot yet: stream it from the caller's rows
                    src = reinterpret_cast<const uint8_t*>(a.new_k + ((size_t)b * a.Hkv + kvh) * D);
                    row_v = reinterpret_cast<const uint8_t*>(a.new_v + ((size_t)b * a.Hkv + kvh) * D);
                }
            }
            // the T2 rows of this K tile, for the consumer of its slot (and of the V slot after it)
            const uint32_t fm = __ballot_sync(0xffffffffu, fp8);
            if (lane == 0) mask_s[issued % kWarpStages] = fm;
        } else {
            src = row_v;
        }
        if (kv == 0) all_bf16_issue = __all_sync(0xffffffffu, lane >= kTileRows || row_bytes == 2 * D);
        const uint32_t dst0 = smem_u32(ring + (size_t)(issued % kWarpStages) * kStageBytes);
        const int col = lane & 15, half = lane >> 4;
        if (all_bf16_issue) {
            // kTileRows bf16 rows: no per-row kinds to decode
#pragma unroll kIssueUnroll
            for (int rr = 0; rr < kTileRows / 2; ++rr) {
                const int r = 2 * rr + half;
                const uint8_t* rsrc = reinterpret_cast<const uint8_t*>(
                    __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(src), r));
                if (col * 16 < 2 * D) cp_async16(dst0 + r * ROWB + col * 16, rsrc + col * 16);
            }
        } else {
            const unsigned long long tagged = (unsigned long long)src | (row_bytes == D + 16 ? 1ull : 0ull) |
                                              (row_bytes ? 0ull : 2ull);
#pragma unroll 4
            for (int rr = 0; rr < kTileRows / 2; ++rr) {
                const int r = 2 * rr + half;
                const unsigned long long t = __shfl_sync(0xffffffffu, tagged, r);
                const uint8_t* rsrc = (const uint8_t*)(t & ~15ull);
                const int nb = (t & 2ull) ? 0 : ((t & 1ull) ? D + 16 : 2 * D);
                if (col * 16 < nb)
                    cp_async16(dst0 + r * ROWB + col * 16, rsrc + col * 16);
                else if (nb == 0 && col * 16 < 2 * D)
                    cp_async16_zero(dst0 + r * ROWB + col * 16, k0v0);   // absent row: zeros, so that
                                                                         // p = 0 meets no NaN in the product
            }
        }
        ++issued;
        if (ci_kv == 0) {
            ci_kv = 1;
        } else {
            ci_kv = 0;
            if (++ci_k >= warp_tiles(n)) {
                ci_k = 0;
                ++ci_item;
                settle();
            }
        }
    };

    int consumed = 0;
    // the copy of `consumed` has landed once at most kWarpStages - 1 later groups are pending
    auto wait_slot = [&]() {
        cp_async_commit();
        cp_async_wait_group<kWarpStages - 1>();
    };
    // the first kWarpStages - 1 copies (empty groups past the end of the sequence)
#pragma unroll
    for (int i = 0; i < kWarpStages - 1; ++i) {
        issue_next();
        cp_async_commit();
    }

    // ---------------------------------------------------- per-warp segment state
    // Tensor-core fragments (mma.m16n8k16, bf16 in, fp32 accumulate).  A lane holds, of a
    // 16 x 8 accumulator, rows gq and gq + 8 and columns 2 cq, 2 cq + 1:
    //   scores  S^T[row][head] = k_row . q_head  (A: K rows from the ring, B: q^T);
    //   output  O^T[d][head]  += v_row[d] * p    (A: V^T from the ring, B: p^T).
    // Both put this lane's values on the query heads h0 = 2 cq and h1 = 2 cq + 1, so the
    // softmax rescale of O needs no exchange.  Heads past G are zero columns of q^T.
    const int gq = lane >> 2, cq = lane & 3;
    const int h0 = 2 * cq, h1 = 2 * cq + 1;
    uint32_t qf[D / 16][2];                          // q^T B fragments of the current group
    float m_r[2], l_r[2];                            // running max (warp-uniform) and this lane's share of l
    float o[D / 16][4];
    auto load_q = [&](int g) {
        const int b = g / a.Hkv, kvh = g % a.Hkv;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t lo = 0u, hi = 0u;
            if (gq < G) {
                const unsigned short* qh = reinterpret_cast<const unsigned short*>(
                    a.q + ((size_t)b * a.Hq + (size_t)kvh * G + gq) * D + ks * 16 + 2 * cq);
                lo = (uint32_t)qh[0] | ((uint32_t)qh[1] << 16);
                hi = (uint32_t)qh[8] | ((uint32_t)qh[9] << 16);
            }
            qf[ks][0] = lo;
            qf[ks][1] = hi;
        }
    };
    auto reset_segment = [&]() {
        m_r[0] = m_r[1] = -INFINITY;
        l_r[0] = l_r[1] = 0.f;
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
    };
    // merges the four warps' (m, l, O) of group g into this CTA's partial record for g and
    // stores it at (g, this CTA's rank among the CTAs that touch g).  At the end of the CTA's
    // run (`last`) every copy has been consumed, so each warp parks its record in its own idle
    // ring and the four records merge in one pass (fixed warp order); earlier, while later
    // tiles may be in flight in the rings, the warps fold their values into one shared record
    // in warp order.
    auto flush_segment = [&](int g, bool last) {
        float l0 = l_r[0], l1 = l_r[1];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        const int c_lo = (g * IPG) / a.items_per_cta;
        float* pout = a.part + ((size_t)g * a.part_per_group + (blockIdx.x - c_lo)) * PS;
        if (last) {
            float* cw = reinterpret_cast<float*>(ring);
            if (gq == 0) {
                if (h0 < G) {
                    cw[h0] = m_r[0];
                    cw[8 + h0] = l0;
                }
                if (h1 < G) {
                    cw[h1] = m_r[1];
                    cw[8 + h1] = l1;
                }
            }
#pragma unroll
            for (int dt = 0; dt < D / 16; ++dt) {
                const int d = dt * 16 + gq;
                if (h0 < G) {
                    cw[16 + h0 * D + d] = o[dt][0];
                    cw[16 + h0 * D + d + 8] = o[dt][2];
                }
                if (h1 < G) {
                    cw[16 + h1 * D + d] = o[dt][1];
                    cw[16 + h1 * D + d + 8] = o[dt][3];
                }
            }
            __syncthreads();
            const float* rec0 = reinterpret_cast<const float*>(smem + C::off_ring);
            constexpr size_t kRecStride = C::sz_warp_ring / sizeof(float);
            for (int i = tid; i < G * D + G; i += NT) {
                const int h = i < G * D ? i / D : i - G * D;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, rec0[w * kRecStride + h]);
                float acc = 0.f;
#pragma unroll
                for (int w = 0; w < kAttnWarps; ++w) {
                    const float mw = rec0[w * kRecStride + h];
                    const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
                    acc += f * (i < G * D ? rec0[w * kRecStride + 16 + i] : rec0[w * kRecStride + 8 + h]);
                }
                if (i < G * D) {
                    pout[16 + i] = acc;
                } else {
                    pout[h] = M;
                    pout[8 + h] = acc;
                }
            }
            return;
        }
        for (int w = 0; w < kAttnWarps; ++w) {
            if (warp == w) {
                // factors for the record so far (f_old) and this warp's values (f_new), per head
                float f_old0 = 0.f, f_old1 = 0.f, f_new0 = 1.f, f_new1 = 1.f, M0 = m_r[0], M1 = m_r[1];
                if (w > 0) {
                    const float c0 = comb[h0 < G ? h0 : 0], c1 = comb[h1 < G ? h1 : 0];
                    M0 = fmaxf(c0, m_r[0]);
                    M1 = fmaxf(c1, m_r[1]);
                    f_old0 = (c0 == -INFINITY) ? 0.f : exp2f(c0 - M0);
                    f_old1 = (c1 == -INFINITY) ? 0.f : exp2f(c1 - M1);
                    f_new0 = (m_r[0] == -INFINITY) ? 0.f : exp2f(m_r[0] - M0);
                    f_new1 = (m_r[1] == -INFINITY) ? 0.f : exp2f(m_r[1] - M1);
                }
#pragma unroll
                for (int dt = 0; dt < D / 16; ++dt) {
                    const int d = dt * 16 + gq;
                    float* c0p = comb + 16 + h0 * D + d;
                    float* c1p = comb + 16 + h1 * D + d;
                    if (h0 < G) {
                        c0p[0] = w ? c0p[0] * f_old0 + o[dt][0] * f_new0 : o[dt][0];
                        c0p[8] = w ? c0p[8] * f_old0 + o[dt][2] * f_new0 : o[dt][2];
                    }
                    if (h1 < G) {
                        c1p[0] = w ? c1p[0] * f_old1 + o[dt][1] * f_new1 : o[dt][1];
                        c1p[8] = w ? c1p[8] * f_old1 + o[dt][3] * f_new1 : o[dt][3];
                    }
                }
                __syncwarp();
                if (gq == 0) {
                    if (h0 < G) {
                        comb[8 + h0] = w ? comb[8 + h0] * f_old0 + l0 * f_new0 : l0;
                        comb[h0] = M0;
                    }
                    if (h1 < G) {
                        comb[8 + h1] = w ? comb[8 + h1] * f_old1 + l1 * f_new1 : l1;
                        comb[h1] = M1;
                    }
                }
            }
            __syncthreads();
        }
        for (int i = tid; i < G * D; i += NT) pout[16 + i] = comb[16 + i];
        if (tid < G) {
            pout[tid] = comb[tid];
            pout[8 + tid] = comb[8 + tid];
        }
        __syncthreads();
    };
    // ldmatrix lane offsets within a stage: K rows as the A operand (row-major 16 x 16 blocks)
    // and V rows as the transposed A operand of the output product
    const uint32_t k_lane = (uint32_t)(((lane & 7) + ((lane >> 3) & 1) * 8) * ROWB + (lane >> 4) * 16);
    const uint32_t v_lane = (uint32_t)(((lane & 7) + ((lane >> 4) & 1) * 8) * ROWB + ((lane >> 3) & 1) * 16);

    int cur_group = -1;
    for (int item = it0; item < it1; ++item) {
        const int g = item / IPG, b = g / a.Hkv, kvh = g % a.Hkv;
        const int j0 = (item % IPG) * IT;
        const int n = n_s[item - it0];
        if (g != cur_group) {
            if (cur_group >= 0) flush_segment(cur_group, false);
            load_q(g);
            reset_segment();
            cur_group = g;
        }
        const int nt = warp_tiles(n);
        float* zg = a.zs + (((size_t)b * a.Hkv + kvh) * a.Nmax + j0) * GP;
        for (int k = 0; k < nt; ++k) {
            const int tile = warp + kAttnWarps * k;
            const int nrows = min(kTileRows, n - tile * kTileRows);

            // ---------------------------------------------------------- K tile
            issue_next();                       // the copy kWarpStages - 1 ahead in this warp's sequence
            wait_slot();
            __syncwarp();
            const uint32_t tmask = mask_s[consumed % kWarpStages];
            // the decode token's rows go from the ring into their T0 slot (K now, V below)
            const int newr = new_row_in(item, tile);
            auto store_new_row = [&](int kv) {
                if (lane < 2 * D / 16) {
                    const int slot = loc_slot(rl_s[(size_t)(item - it0) * IT + tile * kTileRows + newr]);
                    const uint8_t* srow = ring + (size_t)(consumed % kWarpStages) * kStageBytes + (size_t)newr * ROWB;
                    uint8_t* drow = reinterpret_cast<uint8_t*>(const_cast<__nv_bfloat16*>(a.k0v0)) +
                                    row_index(a.layer, kv, b, kvh, slot, a.B, a.Hkv, a.S0) * (2 * D);
                    reinterpret_cast<uint4*>(drow)[lane] = reinterpret_cast<const uint4*>(srow)[lane];
                }
            };
            if (newr >= 0) store_new_row(0);
            uint8_t* stage_k = ring + (size_t)(consumed % kWarpStages) * kStageBytes;
            // row scales of this lane's score rows (tile rows gq + 8 i): log2(e)/sqrt(d), times
            // the record's scale for a T2 row
            float rs[2 * MT];
#pragma unroll
            for (int i = 0; i < 2 * MT; ++i) rs[i] = a.qscale;
            // T2 records of the stage become bf16 rows in place; their scales join rs
            if (tmask != 0u) widen_t2_rows<D, ROWB>(stage_k, tmask, lane, gq, rs);
            // two accumulator chains (even and odd 16-column steps of d), added at the end
            float s[MT][4], s2[MT][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) s[mt][i] = s2[mt][i] = 0.f;
            {
                const uint32_t kb = smem_u32(stage_k) + k_lane;
#pragma unroll
                for (int ks = 0; ks < D / 16; ks += 2)
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
                        ldsm_x4(kb + (uint32_t)(mt * 16 * ROWB + ks * 32), a0, a1, a2, a3);
                        ldsm_x4(kb + (uint32_t)(mt * 16 * ROWB + ks * 32 + 32), c0, c1, c2, c3);
                        mma_bf16(s[mt], a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
                        mma_bf16(s2[mt], c0, c1, c2, c3, qf[ks + 1][0], qf[ks + 1][1]);
                    }
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) s[mt][i] += s2[mt][i];
            }
            __syncwarp();
            ++consumed;

            // ------------------------------ online softmax update (warp-uniform max)
            // z[mt][i]: tile row mt * 16 + gq + 8 (i >> 1), head h0 + (i & 1); absent rows and
            // heads past G are -inf
            float z[MT][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = mt * 16 + gq + 8 * (i >> 1);
                    const bool live = r < nrows && h0 + (i & 1) < G;
                    z[mt][i] = live ? s[mt][i] * rs[2 * mt + (i >> 1)] : -INFINITY;
                }
            float tm0 = fmaxf(z[0][0], z[0][2]), tm1 = fmaxf(z[0][1], z[0][3]);
#pragma unroll
            for (int mt = 1; mt < MT; ++mt) {
                tm0 = fmaxf(tm0, fmaxf(z[mt][0], z[mt][2]));
                tm1 = fmaxf(tm1, fmaxf(z[mt][1], z[mt][3]));
            }
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                tm0 = fmaxf(tm0, __shfl_xor_sync(0xffffffffu, tm0, off));
                tm1 = fmaxf(tm1, __shfl_xor_sync(0xffffffffu, tm1, off));
            }
            const float mn0 = fmaxf(m_r[0], tm0), mn1 = fmaxf(m_r[1], tm1);
            const float sc0 = (m_r[0] == -INFINITY) ? 0.f : exp2f(m_r[0] - mn0);
            const float sc1 = (m_r[1] == -INFINITY) ? 0.f : exp2f(m_r[1] - mn1);
            m_r[0] = mn0;
            m_r[1] = mn1;
            // an unchanged maximum gives a factor of exactly 1: O is rescaled only when some
            // head's maximum moved
            if (__any_sync(0xffffffffu, sc0 != 1.f || sc1 != 1.f)) {
#pragma unroll
                for (int dt = 0; dt < D / 16; ++dt) {
                    o[dt][0] *= sc0;
                    o[dt][1] *= sc1;
                    o[dt][2] *= sc0;
                    o[dt][3] *= sc1;
                }
            }
            float p[MT][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    p[mt][i] = z[mt][i] == -INFINITY ? 0.f : exp2f(z[mt][i] - ((i & 1) ? mn1 : mn0));
            float ps0 = p[0][0] + p[0][2], ps1 = p[0][1] + p[0][3];
#pragma unroll
            for (int mt = 1; mt < MT; ++mt) {
                ps0 += p[mt][0] + p[mt][2];
                ps1 += p[mt][1] + p[mt][3];
            }
            l_r[0] = l_r[0] * sc0 + ps0;
            l_r[1] = l_r[1] * sc1 + ps1;
            // logits of this lane's heads for the alpha sums (slots of heads past G are never read)
            if (h0 < GP) {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int r = mt * 16 + gq + 8 * hh;
                        if (r < nrows)
                            *reinterpret_cast<float2*>(zg + (size_t)(tile * kTileRows + r) * GP + h0) =
                                make_float2(z[mt][2 * hh], z[mt][2 * hh + 1]);
                    }
            }

            // ---------------------------------------------------------- V tile
            issue_next();                       // and the one after it
            wait_slot();
            __syncwarp();
            if (newr >= 0) store_new_row(1);
            {
                uint8_t* stage_v = ring + (size_t)(consumed % kWarpStages) * kStageBytes;
                if (tmask != 0u) {
                    // T2 rows: widened in place as on the K side; p of such a row carries its scale
                    float vs[2 * MT];
#pragma unroll
                    for (int i = 0; i < 2 * MT; ++i) vs[i] = 1.0f;
                    widen_t2_rows<D, ROWB>(stage_v, tmask, lane, gq, vs);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            p[mt][2 * hh] *= vs[2 * mt + hh];
                            p[mt][2 * hh + 1] *= vs[2 * mt + hh];
                        }
                }
                const uint32_t vb = smem_u32(stage_v) + v_lane;
#pragma unroll
                for (int kk = 0; kk < MT; ++kk) {
                    // p^T as B operands, split p = hi + lo into two bf16 parts (about 16
                    // significant bits together); rows gq and gq + 8 of this 16-row step
                    uint32_t bh[2], bl[2];
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const float x = p[kk][2 * hh], y = p[kk][2 * hh + 1];
                        const __nv_bfloat162 hi2 = __floats2bfloat162_rn(x, y);
                        const uint32_t hw = *reinterpret_cast<const uint32_t*>(&hi2);
                        const float2 hf = bf16x2_to_float2(hw);
                        const __nv_bfloat162 lo2 = __floats2bfloat162_rn(x - hf.x, y - hf.y);
                        bh[hh] = movmatrix_t(hw);
                        bl[hh] = movmatrix_t(*reinterpret_cast<const uint32_t*>(&lo2));
                    }
#pragma unroll
                    for (int dt = 0; dt < D / 16; ++dt) {
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4_t(vb + (uint32_t)(kk * 16 * ROWB + dt * 32), a0, a1, a2, a3);
                        mma_bf16(o[dt], a0, a1, a2, a3, bh[0], bh[1]);
                        mma_bf16(o[dt], a0, a1, a2, a3, bl[0], bl[1]);
                    }
                }
            }
            __syncwarp();
            ++consumed;
        }
    }
    flush_segment(cur_group, true);
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Merges a group's partials (one per CTA whose range touches the group, in CTA
// order) into `out`, and writes the per-position sum over the group's query
// heads of alpha = 2^(z - M) / L.  Every load of the block is issued before the
// first barrier (the segment statistics, the block's share of the partial
// outputs, the logits of its rows), so the kernel costs about one memory round
// trip after the main kernel ends.  SEG partial outputs are loaded per thread before
// the barrier: 32 for launches whose groups have many partials (small batches, where
// latency rules), 8 otherwise (fewer registers: four blocks per SM instead of two).
template <int G, int D, int SEG>
__global__ void __launch_bounds__(256, SEG <= 8 ? 4 : 1) attn_combine_kernel(const AttnArgs a) {
    using C = AttnCfg<G, D>;
    constexpr int GP = C::GP, PS = C::PS;
    constexpr int kSegBatch = SEG;                   // partial outputs loaded per thread at once
    extern __shared__ __align__(16) float fsm[];     // m[seg][8], l[seg][8], then f[seg][8]
    __shared__ float Ms[8], Linv[8];
    // launched as a programmatic dependent of the main kernel: wait for its results
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int g = blockIdx.y, b = g / a.Hkv, kvh = g % a.Hkv;
    const int IPG = a.items_per_group, ipc = a.items_per_cta;
    const int c_lo = (g * IPG) / ipc, c_hi = ((g + 1) * IPG - 1) / ipc;
    const int ns = c_hi - c_lo + 1;
    float* m_s = fsm;
    float* l_s = fsm + ns * 8;
    float* f_s = fsm + 2 * ns * 8;
    const float* grec = a.part + (size_t)g * a.part_per_group * PS;
    auto rec = [&](int sg) { return grec + (size_t)sg * PS; };
    // (1) loads: segment statistics, this thread's first batch of partial outputs, its logits
    for (int t = threadIdx.x; t < ns * 8; t += blockDim.x) {
        const int sg = t >> 3, h = t & 7;
        const float* r = rec(sg);
        m_s[t] = h < G ? r[h] : -INFINITY;
        l_s[t] = h < G ? r[8 + h] : 0.f;
    }
    const int per = (G * D + gridDim.x - 1) / gridDim.x;
    const int i0 = blockIdx.x * per, i1 = min(G * D, i0 + per);
    const int idx = i0 + threadIdx.x;                // blockDim.x >= per: one element per thread
    const bool has_out = idx < i1;
    // only the warps that hold out elements load partial outputs (a warp-uniform branch); the
    // values are used in step (3) by the same threads only
    float v[kSegBatch];
    if (i0 + (int)(threadIdx.x & ~31u) < i1) {
#pragma unroll
        for (int k = 0; k < kSegBatch; ++k) v[k] = (has_out && k < ns) ? rec(k)[16 + idx] : 0.f;
    }
    // this thread's rows: j0 + k * kCombineThreads, k < kCombineRowsPerThread
    const int j0 = blockIdx.x * kCombineRows + threadIdx.x;
    const int R = a.rl_count[b];
    float zz[kCombineRowsPerThread][GP];
    float g_prev[kCombineRowsPerThread];
    float* gg = a.g + ((size_t)b * a.Hkv + kvh) * a.Nmax;
#pragma unroll
    for (int k = 0; k < kCombineRowsPerThread; ++k) {
        const int j = j0 + k * kCombineThreads;
        if (j < R) {
            const float* zg = a.zs + (((size_t)b * a.Hkv + kvh) * a.Nmax + j) * GP;
#pragma unroll
            for (int h = 0; h < GP; h += 4) {
                const float4 t = *reinterpret_cast<const float4*>(zg + h);
                zz[k][h] = t.x; zz[k][h + 1] = t.y; zz[k][h + 2] = t.z; zz[k][h + 3] = t.w;
            }
        }
        // running sum over layers of this row's alpha (layer 0 starts it)
        g_prev[k] = (j < R && a.layer > 0) ? gg[j] : 0.f;
    }
    __syncthreads();
    // (2) the group's M and L per head (one warp per head, segments across lanes, fixed
    // shuffle order), and every segment's factor 2^(m - M) / L
    {
        const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
        if (w < G) {
            const int h = w;
            float M = -INFINITY;
            for (int sg = lane; sg < ns; sg += 32) M = fmaxf(M, m_s[sg * 8 + h]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            float L = 0.f;
            for (int sg = lane; sg < ns; sg += 32) {
                const float ms = m_s[sg * 8 + h];
                const float f = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
                f_s[sg * 8 + h] = f;
                L += f * l_s[sg * 8 + h];
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
            const float inv = 1.0f / L;
            for (int sg = lane; sg < ns; sg += 32) f_s[sg * 8 + h] *= inv;
            if (lane == 0) {
                Ms[h] = M;
                Linv[h] = inv;
            }
        }
    }
    __syncthreads();
    // (3) out, summed in segment order; groups with more than kSegBatch segments load the rest now
    if (has_out) {
        const int h = idx / D;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < kSegBatch; ++k)
            if (k < ns) acc += v[k] * f_s[k * 8 + h];
        for (int s0 = kSegBatch; s0 < ns; s0 += kSegBatch) {
#pragma unroll
            for (int k = 0; k < kSegBatch; ++k) v[k] = (s0 + k < ns) ? rec(s0 + k)[16 + idx] : 0.f;
#pragma unroll
            for (int k = 0; k < kSegBatch; ++k)
                if (s0 + k < ns) acc += v[k] * f_s[(s0 + k) * 8 + h];
        }
        a.out[((size_t)b * a.Hq + (size_t)kvh * G) * D + idx] = acc;
    }
    // (4) alpha sums of this block's rows
#pragma unroll
    for (int k = 0; k < kCombineRowsPerThread; ++k) {
        const int j = j0 + k * kCombineThreads;
        if (j < R) {
            float acc = 0.f;
#pragma unroll
            for (int h = 0; h < G; ++h) acc += exp2f(zz[k][h] - Ms[h]) * Linv[h];
            gg[j] = g_prev[k] + acc;
        }
    }
}

// ------------------------------------------------------------------ dispatch
template <int G, int D>
static cudaError_t launch_gd(const AttnArgs& a, cudaStream_t st, cudaEvent_t after_main, cudaEvent_t before_combine) {
    using C = AttnCfg<G, D>;
    const size_t smem = C::smem(a.items_per_cta * a.item_rows);
    // at most two tiles per warp: the compact instantiation
    if (a.items_per_cta * a.item_rows <= kCompactRows)
        attn_kernel<G, D, true><<<a.grid, kAttnWarps * 32, smem, st>>>(a);
    else
        attn_kernel<G, D, false><<<a.grid, kAttnWarps * 32, smem, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (after_main && (e = cudaEventRecord(after_main, st)) != cudaSuccess) return e;
    if (before_combine && (e = cudaEventRecord(before_combine, st)) != cudaSuccess) return e;
    // one alpha row per thread; enough blocks that every block holds at most 256 out elements
    const int rows = a.items_per_group * a.item_rows;
    const int blocks = std::max((rows + kCombineRows - 1) / kCombineRows, (G * D + kCombineThreads - 1) / kCombineThreads);
    const int max_segs = a.part_per_group;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks, a.B * a.Hkv);
    cfg.blockDim = dim3(kCombineThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)max_segs * 3 * 8 * 4;
    auto kernel = max_segs <= 8 ? attn_combine_kernel<G, D, 8> : attn_combine_kernel<G, D, 32>;
    if (cfg.dynamicSmemBytes > 48 * 1024) {
        // raise the limit if needed, never lower it (other contexts may need more)
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kernel);
        if (e == cudaSuccess && (size_t)fa.maxDynamicSharedSizeBytes < cfg.dynamicSmemBytes)
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cfg.dynamicSmemBytes);
        if (e != cudaSuccess) return e;
    }
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <int G, int D>
static cudaError_t prepare_gd(size_t smem) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<G, D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_kernel<G, D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // the combine kernel asks for the same shared-memory carve-out as the main kernel, so that
    // an SM need not be reconfigured between the two
    e = cudaFuncSetAttribute(attn_combine_kernel<G, D, 8>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(attn_combine_kernel<G, D, 32>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                (int)cudaSharedmemCarveoutMaxShared);
}

template <int G, int D>
static size_t smem_gd(int rl_rows) {
    return AttnCfg<G, D>::smem(rl_rows);
}

template <int G, int D>
static int resident_gd(size_t smem) {
    int per_sm = 0, dev = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_kernel<G, D, false>, kAttnWarps * 32, smem) != cudaSuccess ||
        cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return per_sm * sms;
}

template <int G, int D>
static cudaError_t ensure_smem_gd(size_t smem) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, attn_kernel<G, D, false>);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fc;
    e = cudaFuncGetAttributes(&fc, attn_kernel<G, D, true>);
    if (e != cudaSuccess) return e;
    if ((size_t)fa.maxDynamicSharedSizeBytes >= smem && (size_t)fc.maxDynamicSharedSizeBytes >= smem)
        return cudaSuccess;
    return prepare_gd<G, D>(smem);
}

#define TKV_DISPATCH_G(D, FN, ...)                      \
    switch (G) {                                        \
        case 1: return FN<1, D>(__VA_ARGS__);           \
        case 2: return FN<2, D>(__VA_ARGS__);           \
        case 3: return FN<3, D>(__VA_ARGS__);           \
        case 4: return FN<4, D>(__VA_ARGS__);           \
        case 5: return FN<5, D>(__VA_ARGS__);           \
        case 6: return FN<6, D>(__VA_ARGS__);           \
        case 7: return FN<7, D>(__VA_ARGS__);           \
        case 8: return FN<8, D>(__VA_ARGS__);           \
        default: break;                                 \
    }

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t st, cudaEvent_t after_main, cudaEvent_t before_combine) {
    const int G = a.Hq / a.Hkv;
    if (a.d == 128) { TKV_DISPATCH_G(128, launch_gd, a, st, after_main, before_combine) }
    if (a.d == 64) { TKV_DISPATCH_G(64, launch_gd, a, st, after_main, before_combine) }
    return cudaErrorInvalidValue;
}

int attention_max_window_rows() { return kMaxWindowRows; }

size_t attention_smem_bytes(int G, int d, int rl_rows) {
    if (d == 128) { TKV_DISPATCH_G(128, smem_gd, rl_rows) }
    if (d == 64) { TKV_DISPATCH_G(64, smem_gd, rl_rows) }
    return 0;
}

cudaError_t attention_prepare(int G, int d, size_t smem) {
    if (d == 128) { TKV_DISPATCH_G(128, prepare_gd, smem) }
    if (d == 64) { TKV_DISPATCH_G(64, prepare_gd, smem) }
    return cudaErrorInvalidValue;
}

int attention_resident_ctas(int G, int d, size_t smem) {
    if (d == 128) { TKV_DISPATCH_G(128, resident_gd, smem) }
    if (d == 64) { TKV_DISPATCH_G(64, resident_gd, smem) }
    return 0;
}

cudaError_t attention_ensure_smem(int G, int d, size_t smem) {
    if (d == 128) { TKV_DISPATCH_G(128, ensure_smem_gd, smem) }
    if (d == 64) { TKV_DISPATCH_G(64, ensure_smem_gd, smem) }
    return cudaErrorInvalidValue;
}

AttnPlan attention_plan(int G, int d, int B, int Hkv, int rmax, int resident) {
    const int groups = B * Hkv;
    rmax = std::max(rmax, 1);
    resident = std::max(resident, 1);
    // Items of 256, 128 or 64 rows: the size whose heaviest CTA streams the fewest rows (waves
    // of resident CTAs times items per CTA times rows), the larger items on a tie.  The choice
    // depends on rmax only through ceil(rmax / 64).
    AttnPlan best{};
    long best_load = -1;
    for (int rows = 256; rows >= kMinItemRows; rows /= 2) {
        AttnPlan p{};
        p.item_rows = rows;
        p.items_per_group = (rmax + rows - 1) / rows;
        const int total = groups * p.items_per_group;
        p.grid = std::min(total, resident);
        p.items_per_cta = (total + p.grid - 1) / p.grid;
        const int max_items = kMaxWindowRows / rows;
        if (p.items_per_cta > max_items) {
            p.items_per_cta = max_items;
            p.grid = (total + max_items - 1) / max_items;
        }
        const long load = (long)((p.grid + resident - 1) / resident) * p.items_per_cta * rows;
        if (best_load < 0 || load < best_load) {
            best = p;
            best_load = load;
        }
    }
    best.part_per_group = (best.items_per_group + best.items_per_cta - 1) / best.items_per_cta + 1;
    best.smem = attention_smem_bytes(G, d, best.items_per_cta * best.item_rows);
    return best;
}

size_t attention_part_floats(int G, int d, int B, int Hkv, int Nmax, int resident) {
    // B * Hkv * part_per_group records, the largest over every retained count up to Nmax
    // (the plan is constant over each 64-row bucket of counts)
    size_t per_group = 0;
    for (int r = 64; r < Nmax + 64; r += 64)
        per_group = std::max(per_group, (size_t)attention_plan(G, d, B, Hkv, std::min(r, Nmax), resident).part_per_group);
    return (size_t)B * Hkv * per_group * (16 + (size_t)G * d);
}

size_t attention_zs_floats(int G, int B, int Hkv, int Nmax) {
    const int GP = (G <= 4) ? 4 : 8;
    return (size_t)B * Hkv * Nmax * GP;
}

// ---------------------------------------------------------------- score fold
// s[b][pos(j)] += (sum_kvh g[b][kvh][j]) / (L * Hq), g holding each (KV head,
// row)'s sum over layers and that head's query heads of alpha; fixed order.
__global__ void fold_kernel(const float* __restrict__ g, const int32_t* __restrict__ rl_pos,
                            const int32_t* __restrict__ rl_count, float* __restrict__ s, int Hkv,
                            int Nmax, float inv_lh) {
    const int b = blockIdx.y;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= rl_count[b]) return;
    const int pos = rl_pos[(size_t)b * Nmax + j];
    float acc = 0.f;
    for (int h = 0; h < Hkv; ++h) acc += g[((size_t)b * Hkv + h) * Nmax + j];
    s[(size_t)b * Nmax + pos] += acc * inv_lh;
}

cudaError_t launch_fold(const float* g, const int32_t* rl_pos, const int32_t* rl_count, float* s,
                        int B, int Hkv, int Nmax, int rmax, float inv_lh, cudaStream_t st) {
    if (rmax <= 0) return cudaSuccess;
    dim3 grid((rmax + 255) / 256, B);
    fold_kernel<<<grid, 256, 0, st>>>(g, rl_pos, rl_count, s, Hkv, Nmax, inv_lh);
    return cudaGetLastError();
}

}  // namespace tkv
