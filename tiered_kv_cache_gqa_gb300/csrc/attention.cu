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
// Per CTA: warp 4 is the producer; it walks the run in tiles of 32 rows and,
// per row, issues one 1-D bulk copy (cp.async.bulk) from the row's home --
// T0 pool, T1 staging or T2 pool -- into a shared-memory ring whose stages
// complete on mbarriers.  It streams the K rows of the whole run, then the V
// rows.  Warps 0-3 consume:
//   pass 1 (K): lane = row; z[h] = q'_h . k for the G query heads of the
//              group, with q' = q * log2(e)/sqrt(d) held in shared memory
//              (broadcast reads) and packed f32x2 FMAs; z is kept in shared
//              memory; T2 rows: z = scale * (q' . code values).
//   softmax:   per-CTA max m_h over the run, p = 2^(z - m_h) in place,
//              l_h = sum p (fixed-order reduction).
//   pass 2 (V): the warp walks a tile's rows; lane = 4 (or 2) columns;
//              O_h += p * v.
// Cluster merge (distributed shared memory): every CTA reads all peers'
// (m, l) in rank order -> M_h, L_h, per-peer factors f_r = 2^(m_r - M)/L; it
// writes, for its own rows, g[j] = sum_h p_h[j] * f_self,h (the sum over the
// group's query heads of alpha), and reduces its share of O over the peers in
// rank order.  No atomics touch `out` or `g`.
#include "tkv_internal.cuh"

namespace tkv {

template <int G, int D>
struct AttnCfg {
    static constexpr int GP = (G <= 4) ? 4 : 8;      // z / p row stride (floats)
    static constexpr int ROWB = 2 * D + 16;          // ring row stride (bytes), bank-skewed
    static constexpr int NST = 6;                    // ring stages
    static constexpr int CPL = D / 32;               // pass-2 columns per lane
    static_assert(D == 64 || D == 128, "head_dim must be 64 or 128");
    static_assert(G >= 1 && G <= 8, "group size must be 1..8");

    static constexpr size_t off_ring = 0;
    static constexpr size_t sz_ring = (size_t)NST * kRows * ROWB;
    static constexpr size_t off_info = sz_ring;
    static constexpr size_t off_bars = off_info + 16 * NST;
    static constexpr size_t off_q = off_bars + 16 * NST;
    static constexpr size_t off_o = off_q + (size_t)G * D * 4;
    static constexpr size_t off_m = off_o + (size_t)G * D * 4;
    static constexpr size_t off_l = off_m + 32;
    static constexpr size_t off_f = off_l + 32;
    static constexpr size_t off_red = off_f + (size_t)kMaxSplits * 8 * 4;
    static constexpr size_t off_wm = off_red + 128 * 4;
    static constexpr size_t off_flag = off_wm + kConsumerWarps * 8 * 4;
    static constexpr size_t off_zp = off_flag + 16;
    static_assert((size_t)kConsumerWarps * G * D * 4 <= sz_ring, "warp partials reuse the ring");

    // the CTA's slice of the retained list follows zp: chunk u32
    static size_t smem(int chunk) { return off_zp + (size_t)chunk * GP * 4 + (size_t)chunk * 4; }
};

template <int G, int D>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(const AttnArgs a) {
    using C = AttnCfg<G, D>;
    constexpr int GP = C::GP, ROWB = C::ROWB, NST = C::NST, CPL = C::CPL;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ring = smem + C::off_ring;
    uint32_t* info = reinterpret_cast<uint32_t*>(smem + C::off_info);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::off_bars);
    float* q_s = reinterpret_cast<float*>(smem + C::off_q);
    float* o_s = reinterpret_cast<float*>(smem + C::off_o);
    float* m_s = reinterpret_cast<float*>(smem + C::off_m);
    float* l_s = reinterpret_cast<float*>(smem + C::off_l);
    float* f_s = reinterpret_cast<float*>(smem + C::off_f);
    float* red = reinterpret_cast<float*>(smem + C::off_red);
    float* wm = reinterpret_cast<float*>(smem + C::off_wm);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::off_flag);
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
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + NST);

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    for (int i = tid; i < G * D; i += kAttnThreads)
        q_s[i] = __bfloat162float(a.q[((size_t)b * a.Hq + (size_t)kvh * G) * D + i]) * a.qscale;
    {
        const uint32_t* rl_g = a.rl_loc + (size_t)b * a.Nmax + j0;
        for (int i = tid; i < n; i += kAttnThreads) rl_s[i] = rl_g[i];
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        int issued = 0;
        const uint32_t* rl = rl_s;
        for (int it = 0; it < 2 * nst; ++it) {
            if (*abort_flag) break;
            const int stage = it % NST, round = it / NST;
            if (round > 0) {
                bool ok = mbar_wait_bounded(empty0 + 8 * stage, (round - 1) & 1);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    *abort_flag = 1;
                    atomicExch(a.err, 5 /* TKV_ETIMEOUT */);
                    break;
                }
            }
            const int kv = it < nst ? 0 : 1;
            const int tile = it < nst ? it : it - nst;
            const int jl = tile * kRows + lane;
            uint32_t bytes = 0;
            const void* src = nullptr;
            bool fp8 = false;
            if (jl < n) {
                const uint32_t loc = rl[jl];
                const int tier = loc_tier(loc), slot = loc_slot(loc);
                if (tier == 0) {
                    src = a.k0v0 + row_index(a.layer, kv, b, kvh, slot, a.B, a.Hkv, a.S0) * D;
                    bytes = 2 * D;
                } else if (tier == 1) {
                    src = a.stage + row_index(0, kv, b, kvh, slot, a.B, a.Hkv, a.S1) * D;
                    bytes = 2 * D;
                } else {
                    src = a.t2 + row_index(a.layer, kv, b, kvh, slot, a.B, a.Hkv, a.S2) * (D + 16);
                    bytes = D + 16;
                    fp8 = true;
                }
            }
            const uint32_t mask = __ballot_sync(0xffffffffu, fp8);
            const uint32_t total = __reduce_add_sync(0xffffffffu, bytes);
            if (lane == 0) {
                info[4 * stage] = mask;
                info[4 * stage + 1] = (uint32_t)min(kRows, n - tile * kRows);
                mbar_arrive_expect_tx(full0 + 8 * stage, total);
            }
            __syncwarp();
            if (bytes) bulk_g2s(smem_u32(ring + (size_t)(stage * kRows + lane) * ROWB), src, bytes,
                                full0 + 8 * stage);
            issued = it + 1;
        }
        // Leave no bulk copy in flight into this CTA's shared memory.
        for (int it = max(0, issued - NST); it < issued; ++it)
            (void)mbar_wait_bounded(full0 + 8 * (it % NST), (it / NST) & 1);
        __syncwarp();
    } else {
        // ----------------------------------------------------------- consumers
        float m_run[G];
#pragma unroll
        for (int h = 0; h < G; ++h) m_run[h] = -INFINITY;

        // pass 1: logits
        for (int tile = warp; tile < nst; tile += kConsumerWarps) {
            if (*abort_flag) break;
            const int stage = tile % NST;
            bool ok = mbar_wait_bounded(full0 + 8 * stage, (tile / NST) & 1);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                *abort_flag = 1;
                atomicExch(a.err, 5);
                break;
            }
            const uint32_t mask = info[4 * stage];
            const int jl = tile * kRows + lane;
            if (jl < n) {
                const uint8_t* row = ring + (size_t)(stage * kRows + lane) * ROWB;
                float2 acc[G];
#pragma unroll
                for (int h = 0; h < G; ++h) acc[h] = make_float2(0.f, 0.f);
                float zscale = 1.0f;
                if (!((mask >> lane) & 1u)) {
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
                            acc[h] = __ffma2_rn(make_float2(qa.z, qa.w), k1, acc[h]);
                            acc[h] = __ffma2_rn(make_float2(qb.x, qb.y), k2, acc[h]);
                            acc[h] = __ffma2_rn(make_float2(qb.z, qb.w), k3, acc[h]);
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
                            acc[h] = __ffma2_rn(make_float2(qa.z, qa.w), k1, acc[h]);
                            acc[h] = __ffma2_rn(make_float2(qb.x, qb.y), k2, acc[h]);
                            acc[h] = __ffma2_rn(make_float2(qb.z, qb.w), k3, acc[h]);
                        }
                    }
                }
                float z[GP];
#pragma unroll
                for (int h = 0; h < GP; ++h) z[h] = 0.f;
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    z[h] = (acc[h].x + acc[h].y) * zscale;
                    m_run[h] = fmaxf(m_run[h], z[h]);
                }
#pragma unroll
                for (int h = 0; h < GP; h += 4)
                    *reinterpret_cast<float4*>(zp + (size_t)jl * GP + h) =
                        make_float4(z[h], z[h + 1], z[h + 2], z[h + 3]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * stage);
        }

        // softmax statistics of this CTA's run
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float m = m_run[h];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            if (lane == 0) wm[warp * 8 + h] = m;
        }
        named_bar_sync(1, kConsumerWarps * 32);
        if (tid < G) {
            float m = wm[tid];
            for (int w = 1; w < kConsumerWarps; ++w) m = fmaxf(m, wm[w * 8 + tid]);
            m_s[tid] = m;
        }
        named_bar_sync(1, kConsumerWarps * 32);
        {
            const int h = tid % GP;
            float lsum = 0.f;
            if (h < G) {
                const float mh = m_s[h];
                for (int idx = tid; idx < n * GP; idx += kConsumerWarps * 32) {
                    const float p = exp2f(zp[idx] - mh);
                    zp[idx] = p;
                    lsum += p;
                }
            }
            red[tid] = lsum;
        }
        named_bar_sync(1, kConsumerWarps * 32);
        if (tid < G) {
            float l = 0.f;
            for (int k = tid; k < kConsumerWarps * 32; k += GP) l += red[k];
            l_s[tid] = l;
        }

        // pass 2: values
        float2 o[G][CPL / 2];
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int c = 0; c < CPL / 2; ++c) o[h][c] = make_float2(0.f, 0.f);

        for (int tile = warp; tile < nst; tile += kConsumerWarps) {
            if (*abort_flag) break;
            const int it = nst + tile;
            const int stage = it % NST;
            bool ok = mbar_wait_bounded(full0 + 8 * stage, (it / NST) & 1);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                *abort_flag = 1;
                atomicExch(a.err, 5);
                break;
            }
            const uint32_t mask = info[4 * stage];
            const int nrows = (int)info[4 * stage + 1];
            for (int r = 0; r < nrows; ++r) {
                const int jl = tile * kRows + r;
                const uint8_t* row = ring + (size_t)(stage * kRows + r) * ROWB;
                float p[GP];
#pragma unroll
                for (int h = 0; h < GP; h += 4) {
                    const float4 t = *reinterpret_cast<const float4*>(zp + (size_t)jl * GP + h);
                    p[h] = t.x; p[h + 1] = t.y; p[h + 2] = t.z; p[h + 3] = t.w;
                }
                float2 v[CPL / 2];
                if (!((mask >> r) & 1u)) {
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
            if (lane == 0) mbar_arrive(empty0 + 8 * stage);
        }

        // combine the four warps' partial O (fixed order); the ring is free now
        named_bar_sync(1, kConsumerWarps * 32);
        float* ored = reinterpret_cast<float*>(ring);
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int c = 0; c < CPL / 2; ++c)
                *reinterpret_cast<float2*>(ored + ((size_t)warp * G + h) * D + lane * CPL + 2 * c) =
                    o[h][c];
        named_bar_sync(1, kConsumerWarps * 32);
        for (int i = tid; i < G * D; i += kConsumerWarps * 32) {
            float acc = ored[i];
            for (int w = 1; w < kConsumerWarps; ++w) acc += ored[(size_t)w * G * D + i];
            o_s[i] = acc;
        }
    }

    // ------------------------------------------------------------ cluster merge
    cluster_sync_all();
    if (tid < G) {
        const int h = tid;
        const uint32_t am = smem_u32(m_s + h), al = smem_u32(l_s + h);
        float M = -INFINITY;
        for (int r = 0; r < S; ++r) M = fmaxf(M, dsmem_ld_f32(dsmem_addr(am, r)));
        float Lsum = 0.f;
        for (int r = 0; r < S; ++r) {
            const float mr = dsmem_ld_f32(dsmem_addr(am, r));
            const float e = (mr == -INFINITY) ? 0.f : exp2f(mr - M);
            f_s[r * 8 + h] = e;
            Lsum += dsmem_ld_f32(dsmem_addr(al, r)) * e;
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
        for (int jl = tid; jl < n; jl += kAttnThreads) {
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
        for (int i = i0 + tid; i < i1; i += kAttnThreads) {
            const int h = i / D, c = i % D;
            float acc = 0.f;
            for (int r = 0; r < S; ++r) acc += dsmem_ld_f32(dsmem_addr(ao + 4u * i, r)) * f_s[r * 8 + h];
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
    cfg.blockDim = dim3(kAttnThreads, 1, 1);
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
    cfg.blockDim = dim3(kAttnThreads, 1, 1);
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
