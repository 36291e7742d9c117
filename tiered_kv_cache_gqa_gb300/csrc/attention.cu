// Decode attention over the tiered KV cache, with fused emission of the
// per-position attention-weight sums, and the score fold.
//
// Method: "Not All Thoughts Need HBM" (gist.science summary), sections
// "Zero-approximation-error offloading" (T1 rows take part at full precision;
// Proposition 1: the result depends on the evicted set only) and "Importance
// scoring" (s_i += mean over layers and heads of alpha[i]); ARKV summary,
// "Tri-state cache assignment" (8-bit rows are dequantised on the fly and taken
// in their original order).
//
// One thread-block cluster per (sequence b, KV head); its `splits` CTAs each
// own a contiguous run of the retained list (positions in logical order).  The
// run length depends only on the number of retained positions, never on which
// tier a row sits in, and every sum below has a fixed order, so a row read
// from T0 or from the T1 staging ring gives bit-identical results.
//
// Per CTA, four warps.  A warp owns the tiles w, w+4, ... (32 rows each) of the
// CTA's run; it streams the K rows of its tiles, then their V rows, through its
// own two-stage shared-memory ring with cp.async (16 bytes per lane, 16 lanes
// per 256-byte row, each row fetched from its home: T0 pool, T1 staging or T2
// pool), so loads for the next tile are in flight while the current one is
// computed.  The only waits are cp.async.wait_group and hardware barriers.
//   pass 1 (K): lane = row; z[h] = q'_h . k for the G query heads of the
//              group, with q' = q * log2(e)/sqrt(d) in shared memory
//              (broadcast reads) and packed f32x2 FMAs; z is kept in shared
//              memory; T2 rows: z = scale * (q' . code values).
//   softmax:   per-CTA max m_h over the run, p = 2^(z - m_h) in place,
//              l_h = sum p (fixed-order reduction).
//   pass 2 (V): the warp walks its tiles' rows; lane = 4 (or 2) columns;
//              O_h += p * v.
// Cluster merge (distributed shared memory): every CTA gathers all peers'
// (m, l) -> M_h, L_h, per-peer factors f_r = 2^(m_r - M)/L; it writes, for its
// own rows, g[j] = sum_h p_h[j] * f_self,h (the sum over the group's query
// heads of alpha), and reduces its share of O over the peers in rank order.
// No atomics touch `out` or `g`.
#include <cmath>

#include "tkv_internal.cuh"

namespace tkv {

#ifndef TKV_ATTN_WARPS
#define TKV_ATTN_WARPS 4
#endif
#ifndef TKV_WARP_STAGES
#define TKV_WARP_STAGES 2
#endif
constexpr int kAttnWarps = TKV_ATTN_WARPS;     // warps per CTA
constexpr int kWarpStages = TKV_WARP_STAGES;   // ring stages per warp

template <int G, int D>
struct AttnCfg {
    static constexpr int GP = (G <= 4) ? 4 : 8;      // z / p row stride (floats)
    static constexpr int ROWB = 2 * D + 16;          // ring row stride (bytes), bank-skewed
    static constexpr int CPL = D / 32;               // pass-2 columns per lane
    static_assert(D == 64 || D == 128, "head_dim must be 64 or 128");
    static_assert(G >= 1 && G <= 8, "group size must be 1..8");

    static constexpr size_t sz_stage = (size_t)kRows * ROWB;
    static constexpr size_t sz_warp_ring = kWarpStages * sz_stage;
    static constexpr size_t off_ring = 0;
    static constexpr size_t off_q = kAttnWarps * sz_warp_ring;
    static constexpr size_t off_o = off_q;   // O is written after q's last use
    static constexpr size_t off_m = off_q + (size_t)G * D * 4;
    static constexpr size_t off_l = off_m + 32;
    static constexpr size_t off_f = off_l + 32;
    static constexpr size_t off_mall = off_f + (size_t)kMaxSplits * 8 * 4;
    static constexpr size_t off_lall = off_mall + (size_t)kMaxSplits * 8 * 4;
    static constexpr size_t off_red = off_lall + (size_t)kMaxSplits * 8 * 4;
    static constexpr size_t off_wm = off_red + kAttnWarps * 32 * 4;
    static constexpr size_t off_zp = off_wm + kAttnWarps * 8 * 4;
    static_assert((size_t)G * D * 4 <= sz_warp_ring, "a warp's partial O reuses its ring");

    // then z/p (chunk x GP floats) and the CTA's slice of the retained list (chunk u32)
    static size_t smem(int chunk) { return off_zp + (size_t)chunk * GP * 4 + (size_t)chunk * 4; }
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_prev() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kWarpStages - 1) : "memory");
}

template <int G, int D>
__global__ void __launch_bounds__(kAttnWarps * 32) attn_kernel(const AttnArgs a) {
    using C = AttnCfg<G, D>;
    constexpr int GP = C::GP, ROWB = C::ROWB, CPL = C::CPL;
    constexpr int NT = kAttnWarps * 32;
    extern __shared__ __align__(128) uint8_t smem[];
    float* q_s = reinterpret_cast<float*>(smem + C::off_q);
    float* o_s = reinterpret_cast<float*>(smem + C::off_o);
    float* m_s = reinterpret_cast<float*>(smem + C::off_m);
    float* l_s = reinterpret_cast<float*>(smem + C::off_l);
    float* f_s = reinterpret_cast<float*>(smem + C::off_f);
    float* mall = reinterpret_cast<float*>(smem + C::off_mall);
    float* lall = reinterpret_cast<float*>(smem + C::off_lall);
    float* red = reinterpret_cast<float*>(smem + C::off_red);
    float* wm = reinterpret_cast<float*>(smem + C::off_wm);
    float* zp = reinterpret_cast<float*>(smem + C::off_zp);
    uint32_t* rl_s = reinterpret_cast<uint32_t*>(smem + C::off_zp + (size_t)a.chunk * GP * 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = (int)cluster_rank();
    const int kvh = blockIdx.y, b = blockIdx.z;
    const int S = a.splits;
    const int R = a.rl_count[b];
    const int j0 = rank * a.chunk;
    const int n = max(0, min(R, j0 + a.chunk) - j0);
    const int nst = (n + kRows - 1) / kRows;
    uint8_t* ring = smem + C::off_ring + (size_t)warp * C::sz_warp_ring;

    for (int i = tid; i < G * D; i += NT)
        q_s[i] = __bfloat162float(a.q[((size_t)b * a.Hq + (size_t)kvh * G) * D + i]) * a.qscale;
    {
        const uint32_t* rl_g = a.rl_loc + (size_t)b * a.Nmax + j0;
        for (int i = tid; i < n; i += NT) rl_s[i] = rl_g[i];
    }
    __syncthreads();

    // this warp's tiles: warp, warp + 4, ...; iterations 0..ntw-1 are K, ntw..2ntw-1 are V
    const int ntw = warp < nst ? (nst - warp + kAttnWarps - 1) / kAttnWarps : 0;
    const int total = 2 * ntw;
    const uint8_t* k0v0 = reinterpret_cast<const uint8_t*>(a.k0v0);
    const uint8_t* stg = reinterpret_cast<const uint8_t*>(a.stage);
    auto issue = [&](int i) {
        const int kv = i < ntw ? 0 : 1;
        const int tile = warp + kAttnWarps * (i < ntw ? i : i - ntw);
        const uint32_t dst0 = smem_u32(ring + (size_t)(i % kWarpStages) * C::sz_stage);
        const int col = lane & 15;
#pragma unroll 4
        for (int rr = 0; rr < kRows / 2; ++rr) {
            const int r = 2 * rr + (lane >> 4);
            const int jl = tile * kRows + r;
            if (jl >= n) break;
            const uint32_t loc = rl_s[jl];
            const int tier = loc_tier(loc), slot = loc_slot(loc);
            const uint8_t* src;
            int nbytes;
            if (tier == 0) {
                src = k0v0 + row_index(a.layer, kv, b, kvh, slot, a.B, a.Hkv, a.S0) * (2 * D);
                nbytes = 2 * D;
            } else if (tier == 1) {
                src = stg + row_index(0, kv, b, kvh, slot, a.B, a.Hkv, a.S1) * (2 * D);
                nbytes = 2 * D;
            } else {
                src = a.t2 + row_index(a.layer, kv, b, kvh, slot, a.B, a.Hkv, a.S2) * (D + 16);
                nbytes = D + 16;
            }
            if (col * 16 < nbytes) cp_async16(dst0 + r * ROWB + col * 16, src + col * 16);
        }
    };

#pragma unroll
    for (int i = 0; i < kWarpStages - 1; ++i) {
        if (i < total) issue(i);
        cp_async_commit();
    }

    // ------------------------------------------------------------ pass 1: logits
    float m_run[G];
#pragma unroll
    for (int h = 0; h < G; ++h) m_run[h] = -INFINITY;
    for (int i = 0; i < ntw; ++i) {
        if (i + kWarpStages - 1 < total) issue(i + kWarpStages - 1);
        cp_async_commit();
        cp_async_wait_prev();
        __syncwarp();
        const int tile = warp + kAttnWarps * i;
        const int jl = tile * kRows + lane;
        if (jl < n) {
            const uint8_t* row = ring + (size_t)(i % kWarpStages) * C::sz_stage + (size_t)lane * ROWB;
            const bool fp8 = loc_tier(rl_s[jl]) == 2;
            // two independent accumulator pairs per head: (k0, k2) and (k1, k3) lanes of each chunk
            float2 acc[G], acc2[G];
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h] = acc2[h] = make_float2(0.f, 0.f);
            float zscale = 1.0f;
            if (!fp8) {
#pragma unroll 4
                for (int c = 0; c < D / 8; ++c) {
                    const uint4 w = *reinterpret_cast<const uint4*>(row + c * 16);
                    const float2 k0 = bf16x2_to_float2(w.x), k1 = bf16x2_to_float2(w.y);
                    const float2 k2 = bf16x2_to_float2(w.z), k3 = bf16x2_to_float2(w.w);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float4 qa = *reinterpret_cast<const float4*>(q_s + h * D + c * 8);
                        const float4 qb = *reinterpret_cast<const float4*>(q_s + h * D + c * 8 + 4);
                        acc[h] = __ffma2_rn(make_float2(qa.x, qa.y), k0, acc[h]);
                        acc2[h] = __ffma2_rn(make_float2(qa.z, qa.w), k1, acc2[h]);
                        acc[h] = __ffma2_rn(make_float2(qb.x, qb.y), k2, acc[h]);
                        acc2[h] = __ffma2_rn(make_float2(qb.z, qb.w), k3, acc2[h]);
                    }
                }
            } else {
                zscale = *reinterpret_cast<const float*>(row + D);
#pragma unroll 4
                for (int c = 0; c < D / 8; ++c) {
                    const uint2 w = *reinterpret_cast<const uint2*>(row + c * 8);
                    const float2 k0 = e4m3x2_to_float2((uint16_t)(w.x & 0xFFFF));
                    const float2 k1 = e4m3x2_to_float2((uint16_t)(w.x >> 16));
                    const float2 k2 = e4m3x2_to_float2((uint16_t)(w.y & 0xFFFF));
                    const float2 k3 = e4m3x2_to_float2((uint16_t)(w.y >> 16));
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float4 qa = *reinterpret_cast<const float4*>(q_s + h * D + c * 8);
                        const float4 qb = *reinterpret_cast<const float4*>(q_s + h * D + c * 8 + 4);
                        acc[h] = __ffma2_rn(make_float2(qa.x, qa.y), k0, acc[h]);
                        acc2[h] = __ffma2_rn(make_float2(qa.z, qa.w), k1, acc2[h]);
                        acc[h] = __ffma2_rn(make_float2(qb.x, qb.y), k2, acc[h]);
                        acc2[h] = __ffma2_rn(make_float2(qb.z, qb.w), k3, acc2[h]);
                    }
                }
            }
            float z[GP];
#pragma unroll
            for (int h = 0; h < GP; ++h) z[h] = 0.f;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                z[h] = ((acc[h].x + acc[h].y) + (acc2[h].x + acc2[h].y)) * zscale;
                m_run[h] = fmaxf(m_run[h], z[h]);
            }
#pragma unroll
            for (int h = 0; h < GP; h += 4)
                *reinterpret_cast<float4*>(zp + (size_t)jl * GP + h) =
                    make_float4(z[h], z[h + 1], z[h + 2], z[h + 3]);
        }
        __syncwarp();
    }

    // ------------------------------------------ softmax statistics of the run
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float m = m_run[h];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0) wm[warp * 8 + h] = m;
    }
    __syncthreads();
    if (tid < G) {
        float m = wm[tid];
        for (int w = 1; w < kAttnWarps; ++w) m = fmaxf(m, wm[w * 8 + tid]);
        m_s[tid] = m;
    }
    __syncthreads();
    {
        const int h = tid % GP;
        float lsum = 0.f;
        if (h < G) {
            const float mh = m_s[h];
            for (int idx = tid; idx < n * GP; idx += NT) {
                const float p = exp2f(zp[idx] - mh);
                zp[idx] = p;
                lsum += p;
            }
        }
        red[tid] = lsum;
    }
    __syncthreads();
    if (tid < G) {
        float l = 0.f;
        for (int k = tid; k < NT; k += GP) l += red[k];
        l_s[tid] = l;
    }

    // ------------------------------------------------------------ pass 2: values
    float2 o[G][CPL / 2];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int c = 0; c < CPL / 2; ++c) o[h][c] = make_float2(0.f, 0.f);
    for (int i = ntw; i < total; ++i) {
        if (i + kWarpStages - 1 < total) issue(i + kWarpStages - 1);
        cp_async_commit();
        cp_async_wait_prev();
        __syncwarp();
        const int tile = warp + kAttnWarps * (i - ntw);
        const int nrows = min(kRows, n - tile * kRows);
        const uint8_t* stage = ring + (size_t)(i % kWarpStages) * C::sz_stage;
        for (int r = 0; r < nrows; ++r) {
            const int jl = tile * kRows + r;
            const uint8_t* row = stage + (size_t)r * ROWB;
            float p[GP];
#pragma unroll
            for (int h = 0; h < GP; h += 4) {
                const float4 t = *reinterpret_cast<const float4*>(zp + (size_t)jl * GP + h);
                p[h] = t.x; p[h + 1] = t.y; p[h + 2] = t.z; p[h + 3] = t.w;
            }
            float2 v[CPL / 2];
            if (loc_tier(rl_s[jl]) != 2) {
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
                for (int h = 0; h < G; ++h) p[h] *= sc;
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
                for (int c = 0; c < CPL / 2; ++c)
                    o[h][c] = __ffma2_rn(make_float2(p[h], p[h]), v[c], o[h][c]);
        }
        __syncwarp();
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();

    // combine the warps' partial O (fixed order); each warp's ring is free now
    {
        float* ored = reinterpret_cast<float*>(ring);
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int c = 0; c < CPL / 2; ++c)
                *reinterpret_cast<float2*>(ored + (size_t)h * D + lane * CPL + 2 * c) = o[h][c];
    }
    __syncthreads();
    for (int i = tid; i < G * D; i += NT) {
        float acc = 0.f;
        for (int w = 0; w < kAttnWarps; ++w)
            acc += reinterpret_cast<const float*>(smem + C::off_ring + (size_t)w * C::sz_warp_ring)[i];
        o_s[i] = acc;
    }

    // ------------------------------------------------------------ cluster merge
    cluster_sync_all();
    if (tid < kMaxSplits * 8) {
        const int r = tid >> 3, h = tid & 7;
        if (r < S && h < G) {
            mall[tid] = dsmem_ld_f32(dsmem_addr(smem_u32(m_s + h), r));
            lall[tid] = dsmem_ld_f32(dsmem_addr(smem_u32(l_s + h), r));
        }
    }
    __syncthreads();
    if (tid < G) {
        const int h = tid;
        float M = -INFINITY;
        for (int r = 0; r < S; ++r) M = fmaxf(M, mall[r * 8 + h]);
        float Lsum = 0.f;
        for (int r = 0; r < S; ++r) {
            const float mr = mall[r * 8 + h];
            const float e = (mr == -INFINITY) ? 0.f : exp2f(mr - M);
            f_s[r * 8 + h] = e;
            Lsum += lall[r * 8 + h] * e;
        }
        const float inv = 1.0f / Lsum;
        for (int r = 0; r < S; ++r) f_s[r * 8 + h] *= inv;
    }
    __syncthreads();

    // alpha sums over the group's query heads, for this CTA's rows
    {
        float f_self[G];
#pragma unroll
        for (int h = 0; h < G; ++h) f_self[h] = f_s[rank * 8 + h];
        float* gdst = a.g + (((size_t)a.layer * a.B + b) * a.Hkv + kvh) * a.Nmax + j0;
        for (int jl = tid; jl < n; jl += NT) {
            float acc = 0.f;
#pragma unroll
            for (int h = 0; h < G; ++h) acc += zp[(size_t)jl * GP + h] * f_self[h];
            gdst[jl] = acc;
        }
    }

    // this CTA's share of the output, reduced over the peers in rank order
    {
        const int per = (G * D + S - 1) / S;
        const int i0 = rank * per, i1 = min(G * D, i0 + per);
        const uint32_t ao = smem_u32(o_s);
        for (int i = i0 + tid; i < i1; i += NT) {
            const int h = i / D, c = i % D;
            float v[kMaxSplits];
#pragma unroll
            for (int r = 0; r < kMaxSplits; ++r)
                v[r] = (r < S) ? dsmem_ld_f32(dsmem_addr(ao + 4u * i, r)) : 0.f;
            float acc = 0.f;
#pragma unroll
            for (int r = 0; r < kMaxSplits; ++r)
                if (r < S) acc += v[r] * f_s[r * 8 + h];
            a.out[((size_t)b * a.Hq + (size_t)kvh * G + h) * D + c] = acc;
        }
    }
    cluster_sync_all();
}

// ------------------------------------------------------------------ dispatch
template <int G, int D>
static cudaError_t launch_gd(const AttnArgs& a, cudaStream_t st) {
    const size_t smem = AttnCfg<G, D>::smem(a.chunk);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.splits, a.Hkv, a.B);
    cfg.blockDim = dim3(kAttnWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_kernel<G, D>, a);
}

template <int G, int D>
static cudaError_t prepare_gd(size_t smem) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<G, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(attn_kernel<G, D>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <int G, int D>
static bool cluster_fits_gd(size_t smem, int s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(s, 1, 1);
    cfg.blockDim = dim3(kAttnWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = s;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attn_kernel<G, D>, &cfg) == cudaSuccess && n > 0) return true;
    (void)cudaGetLastError();
    return false;
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

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t st) {
    const int G = a.Hq / a.Hkv;
    if (a.d == 128) { TKV_DISPATCH_G(128, launch_gd, a, st) }
    if (a.d == 64) { TKV_DISPATCH_G(64, launch_gd, a, st) }
    return cudaErrorInvalidValue;
}

template <int G, int D>
static size_t smem_gd(int chunk) {
    return AttnCfg<G, D>::smem(chunk);
}

size_t attention_smem_bytes(int G, int d, int chunk) {
    if (d == 128) { TKV_DISPATCH_G(128, smem_gd, chunk) }
    if (d == 64) { TKV_DISPATCH_G(64, smem_gd, chunk) }
    return 0;
}

cudaError_t attention_prepare(int G, int d, size_t smem) {
    if (d == 128) { TKV_DISPATCH_G(128, prepare_gd, smem) }
    if (d == 64) { TKV_DISPATCH_G(64, prepare_gd, smem) }
    return cudaErrorInvalidValue;
}

template <int G, int D>
static cudaError_t ensure_smem_gd(size_t smem) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, attn_kernel<G, D>);
    if (e != cudaSuccess) return e;
    if ((size_t)fa.maxDynamicSharedSizeBytes >= smem) return cudaSuccess;
    return prepare_gd<G, D>(smem);
}

cudaError_t attention_ensure_smem(int G, int d, size_t smem) {
    if (d == 128) { TKV_DISPATCH_G(128, ensure_smem_gd, smem) }
    if (d == 64) { TKV_DISPATCH_G(64, ensure_smem_gd, smem) }
    return cudaErrorInvalidValue;
}

bool attention_cluster_fits(int G, int d, size_t smem, int splits) {
    if (d == 128) { TKV_DISPATCH_G(128, cluster_fits_gd, smem, splits) }
    if (d == 64) { TKV_DISPATCH_G(64, cluster_fits_gd, smem, splits) }
    return false;
}

// ---------------------------------------------------------------- score fold
// s[b][pos(j)] += (sum_l sum_kvh g[l][b][kvh][j]) / (L * Hq), fixed order.
__global__ void fold_kernel(const float* __restrict__ g, const int32_t* __restrict__ rl_pos,
                            const int32_t* __restrict__ rl_count, float* __restrict__ s, int L,
                            int B, int Hkv, int Nmax, float inv_lh) {
    const int b = blockIdx.y;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= rl_count[b]) return;
    float acc = 0.f;
    for (int l = 0; l < L; ++l)
        for (int h = 0; h < Hkv; ++h) acc += g[(((size_t)l * B + b) * Hkv + h) * Nmax + j];
    const int pos = rl_pos[(size_t)b * Nmax + j];
    s[(size_t)b * Nmax + pos] += acc * inv_lh;
}

cudaError_t launch_fold(const float* g, const int32_t* rl_pos, const int32_t* rl_count, float* s,
                        int L, int B, int Hkv, int Nmax, int rmax, float inv_lh, cudaStream_t st) {
    if (rmax <= 0) return cudaSuccess;
    dim3 grid((rmax + 255) / 256, B);
    fold_kernel<<<grid, 256, 0, st>>>(g, rl_pos, rl_count, s, L, B, Hkv, Nmax, inv_lh);
    return cudaGetLastError();
}

}  // namespace tkv
