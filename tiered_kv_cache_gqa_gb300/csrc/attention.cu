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
// (b, KV head, item) order.  Within an item, warp w owns the 32-row tiles w and
// w + 4.  Each warp streams, item after item, the K rows and then the V rows
// of its tiles through its own two-stage shared-memory ring with 16-byte
// cp.async (16 lanes per 256-byte row, every row fetched from its home: T0
// pool, T1 staging or T2 records; the group's decode token from the caller's
// k/v, stored into its T0 slot from the ring), so the next tile -- possibly
// of the next item -- is in flight while the current one is computed.  The
// only waits are cp.async.wait_group and CTA barriers; there are no spin loops.
//   K tile:  lane = row; z_h = q'_h . k for the G query heads of the group,
//            q' = q * log2(e)/sqrt(d) in shared memory (broadcast reads),
//            packed f32x2 FMAs; T2 rows: z = scale * (q' . code values).
//   stats:   per warp and group, online over its tiles: m_h = max z,
//            p = 2^(z - m_h), l_h = sum p; z goes to a global scratch for the
//            alpha sums.
//   V tile:  the warp walks the tile's rows, lane = 4 (or 2) columns,
//            O_h += p * v.
//   group end: the four warps' (m, l, O) are merged in shared memory (fixed
//            order) into the CTA's partial for the group, stored at (group,
//            the CTA's rank among the CTAs that touch the group).
// The combine kernel then merges a group's partials in CTA order into `out`,
// and adds per position g = sum_h 2^(z_h - M_h) / L_h (the sum over the group's
// query heads of alpha) to a running sum over the step's layers.  Item
// boundaries, the CTA ranges and every reduction order depend only on the
// retained counts, never on which tier a row sits in, so a row read from T0 or
// from T1 staging gives bit-identical results.  No atomics touch `out` or `g`.
// Launches in which every warp streams at most two tiles use a compact
// instantiation (partly unrolled loops, same arithmetic in the same order).
#include <algorithm>
#include <cmath>

#include "tkv_internal.cuh"

namespace tkv {

constexpr int kAttnWarps = 4;
constexpr int kWarpStages = 2;
constexpr int kMaxWindowRows = 3584;       // retained-list rows a CTA stages in shared memory
                                           // (two CTAs of the largest instantiation fit an SM)
constexpr int kCombineRows = 256;          // alpha rows per combine block (one per thread)

template <int G, int D>
struct AttnCfg {
    static constexpr int GP = (G <= 4) ? 4 : 8;      // z / p row stride (floats)
    static constexpr int ROWB = 2 * D + 16;          // ring row stride (bytes), bank-skewed
    static constexpr int CPL = D / 32;               // V columns per lane
    static_assert(D == 64 || D == 128, "head_dim must be 64 or 128");
    static_assert(G >= 1 && G <= 8, "group size must be 1..8");

    static constexpr size_t sz_stage = (size_t)kRows * ROWB;
    static constexpr size_t sz_warp_ring = kWarpStages * sz_stage;
    static constexpr int PS = 16 + G * D;            // floats of one (m[8], l[8], O[G][D]) record
    static constexpr size_t off_ring = 0;
    static constexpr size_t off_q = kAttnWarps * sz_warp_ring;
    // p as (p, p) pairs, one row of PSTR floats per tile row: PSTR * 4 bytes is an odd multiple
    // of 16, so the lanes that write different rows hit different banks
    static constexpr int PSTR = 2 * GP + 4;
    static constexpr size_t off_p = off_q + (size_t)G * D * 4;
    static constexpr size_t off_comb = off_p + (size_t)kAttnWarps * kRows * PSTR * 4;
    static constexpr size_t off_n = off_comb + (size_t)kAttnWarps * PS * 4;   // rows of each item
    // per item: rows, decode-token flag, (sequence << 16 | KV head)
    static constexpr size_t off_rl = off_n + (size_t)(kMaxWindowRows / 128) * 3 * 4;

    static size_t smem(int rl_rows) { return off_rl + (size_t)rl_rows * 4; }
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_prev() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kWarpStages - 1) : "memory");
}

// COMPACT: partly unrolled loops, for launches in which every warp streams one or two
// tiles: the code then runs about once per launch and the instruction cache, not the
// arithmetic, sets its pace.
template <int G, int D, bool COMPACT>
__global__ void __launch_bounds__(kAttnWarps * 32, 2) attn_kernel(const AttnArgs a) {
    using C = AttnCfg<G, D>;
    constexpr int GP = C::GP, ROWB = C::ROWB, CPL = C::CPL, PS = C::PS, PSTR = C::PSTR;
    // QK lane map: a lane takes rows (lane & 15) and (lane & 15) + 16 of a tile and the query
    // heads of its half-warp: heads [0, GH) for lanes 0-15, [GH, G) for lanes 16-31.  Each q
    // element read from shared memory then feeds two rows.
    constexpr int GH = (G + 1) / 2;
    constexpr int kQKUnroll = COMPACT ? 4 : 8;          // chunks of 8 elements of a K row (half a row:
                                                        // a smaller loop body, fewer instruction-cache misses)
    constexpr int kPVUnroll = COMPACT ? 4 : kRows;      // rows of a V tile
    constexpr int kIssueUnroll = COMPACT ? 4 : 8;
    constexpr int NT = kAttnWarps * 32;
    extern __shared__ __align__(128) uint8_t smem[];
    float* q_s = reinterpret_cast<float*>(smem + C::off_q);
    float* comb = reinterpret_cast<float*>(smem + C::off_comb);
    uint32_t* rl_s = reinterpret_cast<uint32_t*>(smem + C::off_rl);
    int* n_s = reinterpret_cast<int*>(smem + C::off_n);
    int* own_s = n_s + kMaxWindowRows / 128;
    int* bk_s = n_s + 2 * (kMaxWindowRows / 128);

    // the combine kernel may be scheduled once every CTA of this grid has started
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int IT = a.item_rows, IPG = a.items_per_group;
    const int total_items = a.B * a.Hkv * IPG;
    const int it0 = blockIdx.x * a.items_per_cta;
    const int it1 = min(total_items, it0 + a.items_per_cta);
    if (it0 >= it1) return;
    uint8_t* ring = smem + C::off_ring + (size_t)warp * C::sz_warp_ring;
    float* p_s = reinterpret_cast<float*>(smem + C::off_p) + (size_t)warp * kRows * C::PSTR;

    // Prologue in one round trip: the rows of every item, the retained-list slices
    // (read up to the item size, clamped to the capacity; entries past the count
    // are never used) and the first group's q.
    for (int item = it0 + tid; item < it1; item += NT) {
        const int g = item / IPG, b = g / a.Hkv, j0 = (item % IPG) * IT;
        const int R = a.rl_count[b];
        n_s[item - it0] = max(0, min(IT, R - j0));
        // the group's decode token (its last retained row) falls in this item
        own_s[item - it0] = (a.new_k != nullptr && R - 1 >= j0 && R - 1 < j0 + IT) ? 1 : 0;
        bk_s[item - it0] = (b << 16) | (g % a.Hkv);
    }
    for (int item = it0; item < it1; ++item) {
        const int g = item / IPG, b = g / a.Hkv, j0 = (item % IPG) * IT;
        const int cap = min(IT, a.Nmax - j0);
        const uint32_t* src = a.rl_loc + (size_t)b * a.Nmax + j0;
        uint32_t* dst = rl_s + (size_t)(item - it0) * IT;
        for (int r = tid; r < cap; r += NT) dst[r] = src[r];
    }
    // q of group g, scaled, into shared memory: 8 elements per 16-byte load when q is aligned
    auto load_q = [&](int g) {
        const int b = g / a.Hkv, kvh = g % a.Hkv;
        const __nv_bfloat16* qg = a.q + ((size_t)b * a.Hq + (size_t)kvh * G) * D;
        if ((reinterpret_cast<uintptr_t>(qg) & 15u) == 0) {
            for (int i = tid; i < G * D / 8; i += NT) {
                const uint4 w = reinterpret_cast<const uint4*>(qg)[i];
                const float2 f0 = bf16x2_to_float2(w.x), f1 = bf16x2_to_float2(w.y);
                const float2 f2 = bf16x2_to_float2(w.z), f3 = bf16x2_to_float2(w.w);
                float4* dst = reinterpret_cast<float4*>(q_s + 8 * i);
                dst[0] = make_float4(f0.x * a.qscale, f0.y * a.qscale, f1.x * a.qscale, f1.y * a.qscale);
                dst[1] = make_float4(f2.x * a.qscale, f2.y * a.qscale, f3.x * a.qscale, f3.y * a.qscale);
            }
        } else {
            for (int i = tid; i < G * D; i += NT) q_s[i] = __bfloat162float(qg[i]) * a.qscale;
        }
    };
    load_q(it0 / IPG);
    __syncthreads();
    // tiles of this warp in an item: warp, warp + 4, ... below ceil(n / 32)
    auto warp_tiles = [&](int n) {
        const int nt = (n + kRows - 1) / kRows;
        return warp < nt ? (nt - warp + kAttnWarps - 1) / kAttnWarps : 0;
    };

    // row (within tile `tile` of item) of the group's decode token, or -1
    auto new_row_in = [&](int item, int tile) {
        const int n = n_s[item - it0];
        const int r = n - 1 - tile * kRows;
        return (own_s[item - it0] && r >= 0 && r < kRows) ? r : -1;
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
    uint32_t fp8_mask_issue = 0;       // T2 rows of the tile last issued as K
    bool all_bf16_issue = false;       // that tile has 32 bf16 rows (its K and V copies take the fast path)
    // Copies the next tile of this warp's sequence: 16 lanes per 256-byte row, 16 bytes
    // a lane; a row's source pointer travels by shuffle with its kind in the low bits
    // (bit 0: T2 record of D + 16 bytes, bit 1: no row).
    auto issue_next = [&]() {
        if (ci_item >= it1) return;
        const int item = ci_item, kv = ci_kv;
        const int n = n_s[item - it0];
        const int tile = warp + kAttnWarps * ci_k;
        const int jl = tile * kRows + lane;
        const uint8_t* src = nullptr;
        if (kv == 0) {
            const int bk = bk_s[item - it0], b = bk >> 16, kvh = bk & 0xFFFF;
            row_bytes = 0;
            bool fp8 = false;
            if (jl < n) {
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
            fp8_mask_issue = __ballot_sync(0xffffffffu, fp8);
        } else {
            src = row_v;
        }
        if (kv == 0) all_bf16_issue = __all_sync(0xffffffffu, row_bytes == 2 * D);
        const uint32_t dst0 = smem_u32(ring + (size_t)(issued % kWarpStages) * C::sz_stage);
        const int col = lane & 15, half = lane >> 4;
        if (all_bf16_issue) {
            // 32 bf16 rows: no per-row kinds to decode
#pragma unroll kIssueUnroll
            for (int rr = 0; rr < kRows / 2; ++rr) {
                const int r = 2 * rr + half;
                const uint8_t* rsrc = reinterpret_cast<const uint8_t*>(
                    __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(src), r));
                if (col * 16 < 2 * D) cp_async16(dst0 + r * ROWB + col * 16, rsrc + col * 16);
            }
        } else {
            const unsigned long long tagged = (unsigned long long)src | (row_bytes == D + 16 ? 1ull : 0ull) |
                                              (row_bytes ? 0ull : 2ull);
#pragma unroll 4
            for (int rr = 0; rr < kRows / 2; ++rr) {
                const int r = 2 * rr + half;
                const unsigned long long t = __shfl_sync(0xffffffffu, tagged, r);
                const uint8_t* rsrc = (const uint8_t*)(t & ~15ull);
                const int nb = (t & 2ull) ? 0 : ((t & 1ull) ? D + 16 : 2 * D);
                if (col * 16 < nb) cp_async16(dst0 + r * ROWB + col * 16, rsrc + col * 16);
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

    issue_next();
    cp_async_commit();
    int consumed = 0;

    // ---------------------------------------------------- per-warp segment state
    const int rp = lane & 15, hg = lane >> 4;
    const int hbase = hg * GH;                       // first head of this lane's half-warp
    const int nh = hg ? G - GH : GH;                 // heads of this lane's half-warp
    float m_w[G], l_g[GH];                           // running max (all heads); sum of p (own heads)
    float2 o[G][CPL / 2];
    auto reset_segment = [&]() {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m_w[h] = -INFINITY;
#pragma unroll
            for (int c = 0; c < CPL / 2; ++c) o[h][c] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int h = 0; h < GH; ++h) l_g[h] = 0.f;
    };
    // merges the four warps' (m, l, O) of group g into this CTA's partial record for g
    auto flush_segment = [&](int g) {
        float* cw = comb + (size_t)warp * PS;
#pragma unroll
        for (int h = 0; h < GH; ++h) {
            // sum over the half-warp that owns head hbase + h
            float l = l_g[h];
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
            if (rp == 0 && h < nh) cw[8 + hbase + h] = l;
        }
        if (lane < G) {
            float m = m_w[0];
#pragma unroll
            for (int h = 1; h < G; ++h) m = lane == h ? m_w[h] : m;
            cw[lane] = m;
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int c = 0; c < CPL / 2; ++c)
                *reinterpret_cast<float2*>(cw + 16 + h * D + lane * CPL + 2 * c) = o[h][c];
        __syncthreads();
        // record (g, this CTA's rank among the CTAs that touch g)
        const int c_lo = (g * IPG) / a.items_per_cta;
        float* pout = a.part + ((size_t)g * a.part_per_group + (blockIdx.x - c_lo)) * PS;
        for (int i = tid; i < G * D + G; i += NT) {
            const int h = i < G * D ? i / D : i - G * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, comb[w * PS + h]);
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < kAttnWarps; ++w) {
                const float mw = comb[w * PS + h];
                const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
                acc += f * (i < G * D ? comb[w * PS + 16 + i] : comb[w * PS + 8 + h]);
            }
            if (i < G * D) {
                pout[16 + i] = acc;
            } else {
                pout[h] = M;
                pout[8 + h] = acc;
            }
        }
        __syncthreads();
    };

    int cur_group = -1;
    for (int item = it0; item < it1; ++item) {
        const int g = item / IPG, b = g / a.Hkv, kvh = g % a.Hkv;
        const int j0 = (item % IPG) * IT;
        const int n = n_s[item - it0];
        if (g != cur_group) {
            if (cur_group >= 0) {
                flush_segment(cur_group);
                load_q(g);
                __syncthreads();
            }
            reset_segment();
            cur_group = g;
        }
        const int nt = warp_tiles(n);
        float* zg = a.zs + (((size_t)b * a.Hkv + kvh) * a.Nmax + j0) * GP;
        for (int k = 0; k < nt; ++k) {
            const int tile = warp + kAttnWarps * k;
            const int ra = rp, rb = rp + 16;           // this lane's rows in the tile
            const int ja = tile * kRows + ra, jb = tile * kRows + rb;
            const bool valid_a = ja < n, valid_b = jb < n;

            // ---------------------------------------------------------- K tile
            issue_next();                       // the V tile of this tile
            cp_async_commit();
            const uint32_t tmask = fp8_mask_issue;
            cp_async_wait_prev();
            __syncwarp();
            // the decode token's rows go from the ring into their T0 slot (K now, V below)
            const int newr = new_row_in(item, tile);
            auto store_new_row = [&](int kv) {
                if (lane < 2 * D / 16) {
                    const int slot = loc_slot(rl_s[(size_t)(item - it0) * IT + tile * kRows + newr]);
                    const uint8_t* srow = ring + (size_t)(consumed % kWarpStages) * C::sz_stage + (size_t)newr * ROWB;
                    uint8_t* drow = reinterpret_cast<uint8_t*>(const_cast<__nv_bfloat16*>(a.k0v0)) +
                                    row_index(a.layer, kv, b, kvh, slot, a.B, a.Hkv, a.S0) * (2 * D);
                    reinterpret_cast<uint4*>(drow)[lane] = reinterpret_cast<const uint4*>(srow)[lane];
                }
            };
            if (newr >= 0) store_new_row(0);
            float za[GH], zb[GH];
            {
                const uint8_t* stage_k = ring + (size_t)(consumed % kWarpStages) * C::sz_stage;
                const uint8_t* row_a = stage_k + (size_t)ra * ROWB;
                const uint8_t* row_b = stage_k + (size_t)rb * ROWB;
                // two independent accumulator pairs per (row, head): (k0, k2) and (k1, k3) of each chunk
                float2 acca[GH], acca2[GH], accb[GH], accb2[GH];
#pragma unroll
                for (int h = 0; h < GH; ++h) acca[h] = acca2[h] = accb[h] = accb2[h] = make_float2(0.f, 0.f);
                // eight elements of a row from its chunk c: bf16, or E4M3 codes of a T2 record
                auto load8 = [&](const uint8_t* row, bool f8, int c, float2& k0, float2& k1, float2& k2, float2& k3) {
                    if (!f8) {
                        const uint4 w = *reinterpret_cast<const uint4*>(row + c * 16);
                        k0 = bf16x2_to_float2(w.x);
                        k1 = bf16x2_to_float2(w.y);
                        k2 = bf16x2_to_float2(w.z);
                        k3 = bf16x2_to_float2(w.w);
                    } else {
                        const uint2 w = *reinterpret_cast<const uint2*>(row + c * 8);
                        k0 = e4m3x2_to_float2((uint16_t)(w.x & 0xFFFF));
                        k1 = e4m3x2_to_float2((uint16_t)(w.x >> 16));
                        k2 = e4m3x2_to_float2((uint16_t)(w.y & 0xFFFF));
                        k3 = e4m3x2_to_float2((uint16_t)(w.y >> 16));
                    }
                };
                auto qk_chunk = [&](int c, bool fa, bool fb) {
                    float2 a0, a1, a2, a3, b0, b1, b2, b3;
                    load8(row_a, fa, c, a0, a1, a2, a3);
                    load8(row_b, fb, c, b0, b1, b2, b3);
#pragma unroll
                    for (int h = 0; h < GH; ++h) {
                        // heads past G (the short half-warp of an odd G) read head G - 1; discarded
                        const float* qh = q_s + (size_t)min(hbase + h, G - 1) * D + c * 8;
                        const float4 qa = *reinterpret_cast<const float4*>(qh);
                        const float4 qb = *reinterpret_cast<const float4*>(qh + 4);
                        acca[h] = __ffma2_rn(make_float2(qa.x, qa.y), a0, acca[h]);
                        accb[h] = __ffma2_rn(make_float2(qa.x, qa.y), b0, accb[h]);
                        acca2[h] = __ffma2_rn(make_float2(qa.z, qa.w), a1, acca2[h]);
                        accb2[h] = __ffma2_rn(make_float2(qa.z, qa.w), b1, accb2[h]);
                        acca[h] = __ffma2_rn(make_float2(qb.x, qb.y), a2, acca[h]);
                        accb[h] = __ffma2_rn(make_float2(qb.x, qb.y), b2, accb[h]);
                        acca2[h] = __ffma2_rn(make_float2(qb.z, qb.w), a3, acca2[h]);
                        accb2[h] = __ffma2_rn(make_float2(qb.z, qb.w), b3, accb2[h]);
                    }
                };
                float sca = 1.0f, scb = 1.0f;
                if (tmask != 0u) {
                    // A tile with T2 rows: every T2 record of the stage is widened in place to a
                    // bf16 row (E4M3 values are exact in bf16), one row per lane -- row ra by
                    // the lanes 0-15, row rb by the lanes 16-31 -- and its scale kept aside; the
                    // dot products then run the bf16 loop and are scaled after it.
                    uint8_t* mine = const_cast<uint8_t*>(hg ? row_b : row_a);
                    float my_sc = 1.0f;
                    if ((tmask >> (hg ? rb : ra)) & 1u) {
                        my_sc = *reinterpret_cast<const float*>(mine + D);
                        uint4 codes[D / 16];
#pragma unroll
                        for (int c = 0; c < D / 16; ++c) codes[c] = reinterpret_cast<const uint4*>(mine)[c];
#pragma unroll
                        for (int c = 0; c < D / 16; ++c) {
                            const uint32_t w[4] = {codes[c].x, codes[c].y, codes[c].z, codes[c].w};
                            uint32_t outw[8];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float2 lo = e4m3x2_to_float2((uint16_t)(w[i] & 0xFFFF));
                                const float2 hi = e4m3x2_to_float2((uint16_t)(w[i] >> 16));
                                const __nv_bfloat162 blo = __floats2bfloat162_rn(lo.x, lo.y);
                                const __nv_bfloat162 bhi = __floats2bfloat162_rn(hi.x, hi.y);
                                outw[2 * i] = *reinterpret_cast<const uint32_t*>(&blo);
                                outw[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&bhi);
                            }
                            reinterpret_cast<uint4*>(mine)[2 * c] = make_uint4(outw[0], outw[1], outw[2], outw[3]);
                            reinterpret_cast<uint4*>(mine)[2 * c + 1] = make_uint4(outw[4], outw[5], outw[6], outw[7]);
                        }
                    }
                    __syncwarp();
                    // the scale of row ra sits with lane ra, that of row rb with lane 16 + rb - 16
                    sca = __shfl_sync(0xffffffffu, my_sc, rp);
                    scb = __shfl_sync(0xffffffffu, my_sc, 16 + rp);
                }
#pragma unroll kQKUnroll
                for (int c = 0; c < D / 8; ++c) qk_chunk(c, false, false);
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    const bool live = h < nh;
                    za[h] = (valid_a && live) ? ((acca[h].x + acca[h].y) + (acca2[h].x + acca2[h].y)) * sca : -INFINITY;
                    zb[h] = (valid_b && live) ? ((accb[h].x + accb[h].y) + (accb2[h].x + accb2[h].y)) * scb : -INFINITY;
                }
            }
            __syncwarp();
            ++consumed;

            // ------------------------------ online softmax update (warp-uniform max)
            // tile maxima of this half-warp's heads, then the other half-warp's by one exchange
            float tmax[G];
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                float tm = fmaxf(za[h], zb[h]);
#pragma unroll
                for (int off = 8; off > 0; off >>= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, off));
                const float other = __shfl_xor_sync(0xffffffffu, tm, 16);
                tmax[h] = hg ? other : tm;
                if (GH + h < G) tmax[GH + h] = hg ? tm : other;
            }
            float sc_all[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float m_new = fmaxf(m_w[h], tmax[h]);
                sc_all[h] = (m_w[h] == -INFINITY) ? 0.f : exp2f(m_w[h] - m_new);
                m_w[h] = m_new;
#pragma unroll
                for (int c = 0; c < CPL / 2; ++c) o[h][c] = __fmul2_rn(o[h][c], make_float2(sc_all[h], sc_all[h]));
            }
            float pa[GH], pb[GH];
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                // this lane's head hbase + h: its scale and new max, selected without indexing
                const float sc = (hg && GH + h < G) ? sc_all[GH + h < G ? GH + h : 0] : sc_all[h];
                const float mh = (hg && GH + h < G) ? m_w[GH + h < G ? GH + h : 0] : m_w[h];
                l_g[h] *= sc;
                pa[h] = za[h] == -INFINITY ? 0.f : exp2f(za[h] - mh);
                pb[h] = zb[h] == -INFINITY ? 0.f : exp2f(zb[h] - mh);
                l_g[h] += pa[h];
                l_g[h] += pb[h];
            }
            // p as (p, p) pairs of this lane's heads, rows ra and rb
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                if (h < nh) {
                    *reinterpret_cast<float2*>(p_s + (size_t)ra * PSTR + 2 * (hbase + h)) = make_float2(pa[h], pa[h]);
                    *reinterpret_cast<float2*>(p_s + (size_t)rb * PSTR + 2 * (hbase + h)) = make_float2(pb[h], pb[h]);
                }
            }
            // logits of this lane's heads for the alpha sums (slots of heads past G are never read)
            auto store_z = [&](float* dst, const float* z) {
                if constexpr (GH == 4) {
                    *reinterpret_cast<float4*>(dst) = make_float4(z[0], z[1], z[2], z[3]);
                } else if constexpr (GH == 2) {
                    *reinterpret_cast<float2*>(dst) = make_float2(z[0], z[1]);
                } else {
#pragma unroll
                    for (int h = 0; h < GH; ++h)
                        if (h < nh) dst[h] = z[h];
                }
            };
            if (valid_a) store_z(zg + (size_t)ja * GP + hbase, za);
            if (valid_b) store_z(zg + (size_t)jb * GP + hbase, zb);
            __syncwarp();

            // ---------------------------------------------------------- V tile
            issue_next();                       // the next K tile
            cp_async_commit();
            cp_async_wait_prev();
            __syncwarp();
            if (newr >= 0) store_new_row(1);
            {
                const int nrows = min(kRows, n - tile * kRows);
                const uint8_t* stage = ring + (size_t)(consumed % kWarpStages) * C::sz_stage;
                // o[h] += p[h] * v for one row; p read as (p, p) pairs
                auto pv_row = [&](int r, bool fp8) {
                    const uint8_t* row = stage + (size_t)r * ROWB;
                    float2 pp[G];
#pragma unroll
                    for (int h = 0; h < G; h += 2) {
                        const float4 t = *reinterpret_cast<const float4*>(p_s + (size_t)r * PSTR + 2 * h);
                        pp[h] = make_float2(t.x, t.y);
                        if (h + 1 < G) pp[h + 1] = make_float2(t.z, t.w);
                    }
                    float2 v[CPL / 2];
                    if (!fp8) {
                        if (CPL == 4) {
                            const uint2 w = *reinterpret_cast<const uint2*>(row + lane * 8);
                            v[0] = bf16x2_to_float2(w.x);
                            v[CPL / 2 - 1] = bf16x2_to_float2(w.y);
                        } else {
                            v[0] = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(row + lane * 4));
                        }
                    } else {
                        const float sc = *reinterpret_cast<const float*>(row + D);
#pragma unroll
                        for (int h = 0; h < G; ++h) pp[h] = __fmul2_rn(pp[h], make_float2(sc, sc));
                        if (CPL == 4) {
                            const uint32_t w = *reinterpret_cast<const uint32_t*>(row + lane * 4);
                            v[0] = e4m3x2_to_float2((uint16_t)(w & 0xFFFF));
                            v[CPL / 2 - 1] = e4m3x2_to_float2((uint16_t)(w >> 16));
                        } else {
                            v[0] = e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(row + lane * 2));
                        }
                    }
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int c = 0; c < CPL / 2; ++c) o[h][c] = __ffma2_rn(pp[h], v[c], o[h][c]);
                };
                if (nrows == kRows && tmask == 0u) {
#pragma unroll kPVUnroll
                    for (int r = 0; r < kRows; ++r) pv_row(r, false);
                } else {
#pragma unroll 4
                    for (int r = 0; r < nrows; ++r) pv_row(r, (tmask >> r) & 1u);
                }
            }
            __syncwarp();
            ++consumed;
        }
    }
    flush_segment(cur_group);
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Merges a group's partials (one per CTA whose range touches the group, in CTA
// order) into `out`, and writes the per-position sum over the group's query
// heads of alpha = 2^(z - M) / L.  Every load of the block is issued before the
// first barrier (the segment statistics, the block's share of the partial
// outputs, the logits of its rows), so the kernel costs about one memory round
// trip after the main kernel ends.
template <int G, int D>
__global__ void __launch_bounds__(256, 1) attn_combine_kernel(const AttnArgs a) {
    using C = AttnCfg<G, D>;
    constexpr int GP = C::GP, PS = C::PS;
    constexpr int kSegBatch = 32;                    // partial outputs loaded per thread at once
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
    const int j = blockIdx.x * kCombineRows + threadIdx.x;
    const bool has_row = j < a.Nmax;
    float zz[GP];
    if (has_row) {
        const float* zg = a.zs + (((size_t)b * a.Hkv + kvh) * a.Nmax + j) * GP;
#pragma unroll
        for (int h = 0; h < GP; h += 4) {
            const float4 t = *reinterpret_cast<const float4*>(zg + h);
            zz[h] = t.x; zz[h + 1] = t.y; zz[h + 2] = t.z; zz[h + 3] = t.w;
        }
    }
    const int R = a.rl_count[b];
    // running sum over layers of this row's alpha (layer 0 starts it)
    float* gj = a.g + ((size_t)b * a.Hkv + kvh) * a.Nmax + j;
    const float g_prev = (has_row && a.layer > 0) ? *gj : 0.f;
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
    if (has_row && j < R) {
        float acc = 0.f;
#pragma unroll
        for (int h = 0; h < G; ++h) acc += exp2f(zz[h] - Ms[h]) * Linv[h];
        *gj = g_prev + acc;
    }
}

// ------------------------------------------------------------------ dispatch
template <int G, int D>
static cudaError_t launch_gd(const AttnArgs& a, cudaStream_t st, cudaEvent_t after_main, cudaEvent_t before_combine) {
    using C = AttnCfg<G, D>;
    const size_t smem = C::smem(a.items_per_cta * a.item_rows);
    // at most two tiles per warp: the compact instantiation
    if (a.items_per_cta * a.item_rows <= 2 * kRows * kAttnWarps)
        attn_kernel<G, D, true><<<a.grid, kAttnWarps * 32, smem, st>>>(a);
    else
        attn_kernel<G, D, false><<<a.grid, kAttnWarps * 32, smem, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (after_main && (e = cudaEventRecord(after_main, st)) != cudaSuccess) return e;
    if (before_combine && (e = cudaEventRecord(before_combine, st)) != cudaSuccess) return e;
    // one alpha row per thread; enough blocks that every block holds at most 256 out elements
    const int rows = a.items_per_group * a.item_rows;
    const int blocks = std::max((rows + kCombineRows - 1) / kCombineRows, (G * D + kCombineRows - 1) / kCombineRows);
    const int max_segs = a.part_per_group;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks, a.B * a.Hkv);
    cfg.blockDim = dim3(kCombineRows, 1, 1);
    cfg.dynamicSmemBytes = (size_t)max_segs * 3 * 8 * 4;
    if (cfg.dynamicSmemBytes > 48 * 1024) {
        // raise the limit if needed, never lower it (other contexts may need more)
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, attn_combine_kernel<G, D>);
        if (e == cudaSuccess && (size_t)fa.maxDynamicSharedSizeBytes < cfg.dynamicSmemBytes)
            e = cudaFuncSetAttribute(attn_combine_kernel<G, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)cfg.dynamicSmemBytes);
        if (e != cudaSuccess) return e;
    }
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_combine_kernel<G, D>, a);
}

template <int G, int D>
static cudaError_t prepare_gd(size_t smem) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<G, D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(attn_kernel<G, D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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
    AttnPlan p{};
    const int groups = B * Hkv;
    rmax = std::max(rmax, 1);
    resident = std::max(resident, 1);
    // 256-row items, or 128-row items when that is needed to give every resident CTA work
    p.item_rows = (groups * ((rmax + 255) / 256) >= resident) ? 256 : 128;
    p.items_per_group = (rmax + p.item_rows - 1) / p.item_rows;
    const int total = groups * p.items_per_group;
    p.grid = std::min(total, resident);
    p.items_per_cta = (total + p.grid - 1) / p.grid;
    const int max_items = kMaxWindowRows / p.item_rows;
    if (p.items_per_cta > max_items) {
        p.items_per_cta = max_items;
        p.grid = (total + max_items - 1) / max_items;
    }
    p.part_per_group = (p.items_per_group + p.items_per_cta - 1) / p.items_per_cta + 1;
    p.smem = attention_smem_bytes(G, d, p.items_per_cta * p.item_rows);
    return p;
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
