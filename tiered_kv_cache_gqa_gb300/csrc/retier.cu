// Re-tiering, slot management, data movement between tiers, and appends.
//
// Method: "Not All Thoughts Need HBM" (gist.science summary): "Four-tier
// classification" (protected prompt / sinks / recent window in T0; most
// important reasoning tokens T0, medium T1 at full precision in host DDR, low
// T2 at 8 bits, the least important tail evicted for good) and "System
// implementation" (tiers re-assigned every Delta = 64 steps; asynchronous
// delta prefetch moves only the tokens newly promoted towards the GPU).
// FP8-E4M3 quantisation of T2 rows follows the ARKV summary's tri-state
// assignment (quantise, dequantise on the fly before attention).
#include "tkv_internal.cuh"

namespace tkv {

// --------------------------------------------------------------- block helpers
// Exclusive scan of one int per thread over a 1024-thread block.
__device__ int block_excl_scan(int v, int* tmp, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) tmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int y = tmp[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int z = __shfl_up_sync(0xffffffffu, y, off);
            if (lane >= off) y += z;
        }
        tmp[lane] = y;
    }
    __syncthreads();
    const int base = warp ? tmp[warp - 1] : 0;
    total = tmp[31];
    __syncthreads();
    return base + x - v;
}

__device__ int block_max(int v, int* tmp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
    if (lane == 0) tmp[warp] = v;
    __syncthreads();
    int r = tmp[0];
    for (int w = 1; w < 32; ++w) r = max(r, tmp[w]);
    __syncthreads();
    return r;
}

// Order-preserving map of a float to u32 (ascending floats -> ascending ints).
__device__ __forceinline__ uint32_t float_order(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Rank key: ascending key = higher s first, then lower position first.
__device__ __forceinline__ uint64_t rank_key(float s, int pos) {
    return ((uint64_t)(~float_order(s)) << 32) | (uint32_t)pos;
}

// ------------------------------------------------------------- re-tier kernel
// One 1024-thread CTA per sequence.
constexpr int kRetierThreads = 1024;

size_t retier_smem_bytes(int S0, int S1, int S2) {
    const size_t words = (size_t)(S0 + 31) / 32 + (S1 + 31) / 32 + (S2 + 31) / 32;
    return words * 4 + 3 * 256 * 4 + 64 * 4;
}

__global__ void __launch_bounds__(kRetierThreads) retier_kernel(const RetierArgs a) {
    extern __shared__ __align__(16) uint32_t sm[];
    const int b = blockIdx.x, tid = threadIdx.x;
    const int N = a.N;
    const int W0 = (a.S0 + 31) / 32, W1 = (a.S1 + 31) / 32, W2 = (a.S2 + 31) / 32;
    uint32_t* used[3] = {sm, sm + W0, sm + W0 + W1};
    const int Wx[3] = {W0, W1, W2};
    const int Sx[3] = {a.S0, a.S1, a.S2};
    int* hist = reinterpret_cast<int*>(sm + W0 + W1 + W2);   // [3][256]
    int* tmp = hist + 3 * 256;                                // 64 ints
    __shared__ uint64_t prefix[3];
    __shared__ int kk[3], active[3];
    __shared__ int err;
    __shared__ int tier_count[4];

    const size_t base = (size_t)b * a.Nmax;
    const float* s = a.s + base;
    const uint8_t* old_t = a.tier + base;
    const int32_t* old_s = a.slot + base;
    uint8_t* new_t = a.new_tier + base;
    int32_t* new_s = a.new_slot + base;
    const RetierParams P = a.params[b];

    const int seg = (N + kRetierThreads - 1) / kRetierThreads;
    const int i_beg = min(N, tid * seg), i_end = min(N, i_beg + seg);

    if (tid == 0) {
        err = 0;
        for (int t = 0; t < 4; ++t) tier_count[t] = 0;
    }
    for (int w = tid; w < W0 + W1 + W2; w += kRetierThreads) sm[w] = 0;
    __syncthreads();

    auto is_protected = [&](int i) {
        return i < a.num_sinks || i < a.prompt_len || i >= N - a.window;
    };

    // ---- phase A: new tier of every position
    if (P.forced) {
        for (int i = i_beg; i < i_end; ++i) new_t[i] = a.forced[base + i];
    } else {
        // radix-select the keys of ranks c0, c0+c1, c0+c1+c2 among the candidates
        const int ks[3] = {P.c0, P.c0 + P.c1, P.c0 + P.c1 + P.c2};
        if (tid < 3) {
            prefix[tid] = 0;
            kk[tid] = ks[tid];
            active[tid] = ks[tid] < P.n_cand;
        }
        __syncthreads();
        for (int shift = 56; shift >= 0; shift -= 8) {
            for (int k = tid; k < 3 * 256; k += kRetierThreads) hist[k] = 0;
            __syncthreads();
            const uint64_t hi_mask = (shift == 56) ? 0ull : (~0ull << (shift + 8));
            for (int i = i_beg; i < i_end; ++i) {
                if (is_protected(i) || old_t[i] == 3) continue;
                const uint64_t key = rank_key(s[i], i);
                const int digit = (int)((key >> shift) & 0xFF);
#pragma unroll
                for (int q = 0; q < 3; ++q)
                    if (active[q] && (key & hi_mask) == prefix[q]) atomicAdd(&hist[q * 256 + digit], 1);
            }
            __syncthreads();
            if (tid < 3 && active[tid]) {
                int cum = 0;
                for (int dgt = 0; dgt < 256; ++dgt) {
                    const int c = hist[tid * 256 + dgt];
                    if (cum + c > kk[tid]) {
                        kk[tid] -= cum;
                        prefix[tid] |= (uint64_t)dgt << shift;
                        break;
                    }
                    cum += c;
                }
            }
            __syncthreads();
        }
        uint64_t tau[3];
#pragma unroll
        for (int q = 0; q < 3; ++q) tau[q] = active[q] ? prefix[q] : ~0ull;
        for (int i = i_beg; i < i_end; ++i) {
            uint8_t t;
            if (is_protected(i)) t = 0;
            else if (old_t[i] == 3) t = 3;
            else {
                const uint64_t key = rank_key(s[i], i);
                t = key < tau[0] ? 0 : key < tau[1] ? 1 : key < tau[2] ? 2 : 3;
            }
            new_t[i] = t;
        }
    }
    __syncthreads();

    // ---- phase B: slots.  A slot stays taken if its token keeps the tier, or
    // (T1/T2 only) if its token moves to another live tier: that row is still
    // read after this re-tier (delta prefetch, quantise, copy), so the slot
    // becomes free at the next re-tier.  T0 leavers are copied out before any
    // row is written into their slots, so their slots free up at once.
    for (int i = i_beg; i < i_end; ++i) {
        const int o = old_t[i], n = new_t[i];
        if (o == 3) continue;
        const bool keep = (n == o) || (o != 0 && n != 3);
        if (keep) {
            const int sl = old_s[i];
            atomicOr(&used[o][sl >> 5], 1u << (sl & 31));
        }
    }
    __syncthreads();

    for (int X = 0; X < 3; ++X) {
        // free slots of tier X in ascending order -> free_scratch
        int32_t* fs = a.free_scratch + (size_t)b * max(a.S0, max(a.S1, a.S2));
        const int wseg = (Wx[X] + kRetierThreads - 1) / kRetierThreads;
        const int w_beg = min(Wx[X], tid * wseg), w_end = min(Wx[X], w_beg + wseg);
        auto free_bits = [&](int w) {
            uint32_t f = ~used[X][w];
            const int hi = Sx[X] - w * 32;
            if (hi < 32) f &= (hi <= 0) ? 0u : ((1u << hi) - 1u);
            return f;
        };
        int cnt = 0;
        for (int w = w_beg; w < w_end; ++w) cnt += __popc(free_bits(w));
        int F;
        int off = block_excl_scan(cnt, tmp, F);
        for (int w = w_beg; w < w_end; ++w) {
            uint32_t f = free_bits(w);
            while (f) {
                const int bit = __ffs(f) - 1;
                f &= f - 1;
                fs[off++] = w * 32 + bit;
            }
        }
        __syncthreads();
        // enterers of tier X, in position order, take fs[0], fs[1], ...
        int e = 0;
        for (int i = i_beg; i < i_end; ++i) e += (new_t[i] == X && old_t[i] != X);
        int E;
        int k = block_excl_scan(e, tmp, E);
        for (int i = i_beg; i < i_end; ++i) {
            if (new_t[i] != X) continue;
            if (old_t[i] == X) {
                new_s[i] = old_s[i];
            } else {
                if (k < F) new_s[i] = fs[k];
                else { new_s[i] = -1; err = 4; /* TKV_ECAPACITY */ }
                ++k;
            }
        }
        if (X == 0) {
            // remaining free T0 slots as a stack: popping from the top yields the lowest slot
            const int rem = max(0, F - E);
            for (int j = tid; j < rem; j += kRetierThreads)
                a.t0_free[(size_t)b * a.S0 + j] = fs[F - 1 - j];
            if (tid == 0) a.t0_top[b] = rem;
        }
        __syncthreads();
    }

    for (int i = i_beg; i < i_end; ++i)
        if (new_t[i] == 3) new_s[i] = -1;
    __syncthreads();

    // ---- phase C/D: retained list, move lists, counters
    int hw = 0, hw2 = 0, r = 0, mn = 0, md = 0;
    int kind_cnt[7] = {0, 0, 0, 0, 0, 0, 0};
    int cnt_t[4] = {0, 0, 0, 0};
    auto kind_of = [](int o, int n) {
        if (o == n || n == 3 || o == 3) return 0;
        if (o == 0) return n == 1 ? (int)MV_T0_T1 : (int)MV_T0_T2;
        if (o == 1) return n == 2 ? (int)MV_T1_T2 : (int)MV_T1_T0;
        return n == 1 ? (int)MV_T2_T1 : (int)MV_T2_T0;
    };
    for (int i = i_beg; i < i_end; ++i) {
        const int o = old_t[i], n = new_t[i];
        cnt_t[n]++;
        if (n == 3) continue;
        ++r;
        if (n == 1) hw = max(hw, new_s[i] + 1);
        if (n == 2) hw2 = max(hw2, new_s[i] + 1);
        const int kd = kind_of(o, n);
        if (kd) {
            kind_cnt[kd]++;
            if (kd <= MV_T2_T1) ++mn; else ++md;
        }
    }
    for (int i = i_beg; i < i_end; ++i)
        if (old_t[i] != 3 && new_t[i] == 3) kind_cnt[0]++;
    int R, MN, MD;
    int jr = block_excl_scan(r, tmp, R);
    int jn = block_excl_scan(mn, tmp, MN);
    int jd = block_excl_scan(md, tmp, MD);
    for (int i = i_beg; i < i_end; ++i) {
        const int o = old_t[i], n = new_t[i];
        if (n == 3) continue;
        a.rl_loc[base + jr] = make_loc(n, new_s[i]);
        a.rl_pos[base + jr] = i;
        ++jr;
        const int kd = kind_of(o, n);
        if (kd) {
            const int4 mv = make_int4(kd, old_s[i], new_s[i], i);
            if (kd <= MV_T2_T1) a.moves_now[base + jn++] = mv;
            else a.moves_delta[base + jd++] = mv;
        }
    }
    const int HW = block_max(hw, tmp);
    const int HW2 = block_max(hw2, tmp);
    for (int t = 0; t < 4; ++t) atomicAdd(&tier_count[t], cnt_t[t]);
    for (int kd = 0; kd < 7; ++kd) {
        int tot;
        block_excl_scan(kind_cnt[kd], tmp, tot);
        if (tid == 0) a.outp[b].kinds[kd] = tot;
    }
    __syncthreads();
    // commit the new tiers and slots
    for (int i = i_beg; i < i_end; ++i) {
        a.tier[base + i] = new_t[i];
        a.slot[base + i] = new_s[i];
    }
    if (tid == 0) {
        a.rl_count[b] = R;
        a.outp[b].n_now = MN;
        a.outp[b].n_delta = MD;
        a.outp[b].hw1 = HW;
        a.outp[b].hw2 = HW2;
        for (int t = 0; t < 4; ++t) a.outp[b].count[t] = tier_count[t];
        a.outp[b].error = err;
    }
}

// Raises the kernel's dynamic shared-memory limit to `smem` if it is lower; never lowers it
// (contexts of different capacities share the kernel, and a lower limit set by one would make
// another's launches fail).
cudaError_t retier_prepare(size_t smem) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, retier_kernel);
    if (e != cudaSuccess) return e;
    if ((size_t)fa.maxDynamicSharedSizeBytes >= smem) return cudaSuccess;
    return cudaFuncSetAttribute(retier_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_retier(const RetierArgs& a, cudaStream_t st) {
    const size_t smem = retier_smem_bytes(a.S0, a.S1, a.S2);
    cudaError_t e = retier_prepare(smem);
    if (e != cudaSuccess) return e;
    retier_kernel<<<a.B, kRetierThreads, smem, st>>>(a);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- row moves
// One warp per (move entry, layer); the warp handles the 2 * Hkv rows (K and V
// of every KV head) of that token and layer, D/8 lanes per row, 16 bytes a lane.
// T2 quantisation per row: amax over the row (fp32, exact), scale = amax / 448
// (IEEE division; 1 if amax = 0), code = E4M3(x / scale) rounded to nearest
// even with saturation.
template <int D>
__global__ void __launch_bounds__(128) moves_kernel(const MoveArgs a) {
    constexpr int LPR = D / 8;          // lanes per row
    constexpr int RPW = 32 / LPR;       // rows per warp pass
    constexpr int MAXIT = 2 * 8 / RPW;  // passes for 2 * Hkv rows, Hkv <= 8 per pass group
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z;
    const int layer = a.layer_begin + blockIdx.y;
    const int e = blockIdx.x * 4 + warp;
    if (e >= a.counts[(size_t)b * a.count_stride]) return;
    const int4 mv = a.moves[(size_t)b * a.Nmax + e];
    const int kind = mv.x, src = mv.y, dst = mv.z;
    const int sub = lane % LPR;
    for (int base = 0; base < 2 * a.Hkv; base += MAXIT * RPW) {
        // issue every load of this group before any store: one round trip to the source
        uint4 w[MAXIT];
#pragma unroll
        for (int it = 0; it < MAXIT; ++it) {
            const int row = base + it * RPW + lane / LPR;
            if (row >= 2 * a.Hkv) continue;
            const int kv = row / a.Hkv, h = row % a.Hkv;
            const __nv_bfloat16* sp;
            if (kind == MV_T0_T1 || kind == MV_T0_T2)
                sp = a.k0v0 + row_index(layer, kv, b, h, src, a.B, a.Hkv, a.S0) * D;
            else if (kind == MV_T1_T2 || kind == MV_T1_T0)   // the resident HBM copy when there is one
                sp = (a.t1_res ? a.t1_res : a.h1) + row_index(layer, kv, b, h, src, a.B, a.Hkv, a.S1) * D;
            else
                sp = a.h2m + row_index(layer, kv, b, h, src, a.B, a.Hkv, a.S2) * D;
            w[it] = *reinterpret_cast<const uint4*>(sp + sub * 8);
        }
#pragma unroll
        for (int it = 0; it < MAXIT; ++it) {
            const int row = base + it * RPW + lane / LPR;
            const bool live = row < 2 * a.Hkv;   // uniform within a row group
            const int kv = live ? row / a.Hkv : 0, h = live ? row % a.Hkv : 0;
            if (kind == MV_T0_T1 || kind == MV_T2_T1) {
                if (live) {
                    const size_t ri = row_index(layer, kv, b, h, dst, a.B, a.Hkv, a.S1) * D + sub * 8;
                    *reinterpret_cast<uint4*>(a.h1 + ri) = w[it];
                    if (a.t1_res) *reinterpret_cast<uint4*>(a.t1_res + ri) = w[it];   // the resident copy too
                }
            } else if (kind == MV_T1_T0 || kind == MV_T2_T0) {
                if (live)
                    *reinterpret_cast<uint4*>(a.k0v0 + row_index(layer, kv, b, h, dst, a.B, a.Hkv, a.S0) * D +
                                              sub * 8) = w[it];
            } else {
                // into T2: keep the bf16 row on the host, quantise into the T2 pool
                if (live)
                    *reinterpret_cast<uint4*>(a.h2m + row_index(layer, kv, b, h, dst, a.B, a.Hkv, a.S2) * D +
                                              sub * 8) = w[it];
                float x[8];
                const float2 p0 = bf16x2_to_float2(w[it].x), p1 = bf16x2_to_float2(w[it].y);
                const float2 p2 = bf16x2_to_float2(w[it].z), p3 = bf16x2_to_float2(w[it].w);
                x[0] = p0.x; x[1] = p0.y; x[2] = p1.x; x[3] = p1.y;
                x[4] = p2.x; x[5] = p2.y; x[6] = p3.x; x[7] = p3.y;
                float amax = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) amax = live ? fmaxf(amax, fabsf(x[j])) : 0.f;
#pragma unroll
                for (int off = LPR / 2; off > 0; off >>= 1)
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
                if (live) {
                    const float scale = (amax == 0.f) ? 1.0f : __fdiv_rn(amax, 448.0f);
                    uint32_t lo = 0, hi = 0;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t c = (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(x[j], scale),
                                                                           __NV_SATFINITE, __NV_E4M3);
                        if (j < 4) lo |= c << (8 * j);
                        else hi |= c << (8 * (j - 4));
                    }
                    uint8_t* rec = a.t2 + row_index(layer, kv, b, h, dst, a.B, a.Hkv, a.S2) * (D + 16);
                    *reinterpret_cast<uint2*>(rec + sub * 8) = make_uint2(lo, hi);
                    if (sub == 0) *reinterpret_cast<float4*>(rec + D) = make_float4(scale, 0.f, 0.f, 0.f);
                }
            }
        }
    }
}

cudaError_t launch_moves(const MoveArgs& a, cudaStream_t st) {
    if (a.max_count <= 0 || a.layer_end <= a.layer_begin) return cudaSuccess;
    dim3 grid((a.max_count + 3) / 4, a.layer_end - a.layer_begin, a.B);
    if (a.d == 128) moves_kernel<128><<<grid, 128, 0, st>>>(a);
    else if (a.d == 64) moves_kernel<64><<<grid, 128, 0, st>>>(a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

// ------------------------------------------------------------ T1 copy kernel
// SM-driven copy of the per-layer T1 rows from pinned host memory (zero-copy
// loads over the host link) into HBM staging; four independent 16-byte loads
// in flight per thread.
__global__ void __launch_bounds__(256) t1_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                      size_t pitch16, size_t width16, int row_begin,
                                                      int row_end) {
    const size_t total = (size_t)(row_end - row_begin) * width16;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; e + 3 * stride < total; e += 4 * stride) {
        uint4 w[4];
        size_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const size_t x = e + k * stride;
            o[k] = (size_t)(row_begin + x / width16) * pitch16 + x % width16;
            w[k] = src[o[k]];
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[o[k]] = w[k];
    }
    for (; e < total; e += stride) {
        const size_t o = (size_t)(row_begin + e / width16) * pitch16 + e % width16;
        dst[o] = src[o];
    }
}

cudaError_t launch_t1_copy(const void* src, void* dst, size_t pitch16, size_t width16, int row_begin,
                           int row_end, cudaStream_t st) {
    if (row_end <= row_begin || width16 == 0) return cudaSuccess;
    const size_t total = (size_t)(row_end - row_begin) * width16;
    const int blocks = (int)std::min<size_t>((total + 255) / 256, 152 * 8);
    t1_copy_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst),
                                           pitch16, width16, row_begin, row_end);
    return cudaGetLastError();
}

// ------------------------------------------------------------ open / append
// Opens n new positions [N, N+n) of every sequence in T0: pops T0 slots from
// the free stack, resets s, appends to the retained list.
// Opens n new positions of every sequence: T0 slots from the free stack, tier
// 0, s = 0, appended to the retained list.  The position counter lives on the
// device (pos_n[b], equal for every b), so a captured decode step replays with
// the right positions.  With n <= blockDim.x one block per sequence also
// commits (pops the slots, grows the retained count, advances pos_n);
// otherwise open_commit_kernel does, after every block has read the counters.
__global__ void open_kernel(const int32_t* __restrict__ t0_free, int32_t* t0_top, uint8_t* tier, int32_t* slot,
                            float* s, uint32_t* rl_loc, int32_t* rl_pos, int32_t* rl_count, int32_t* pos_n,
                            int Nmax, int S0, int n, int commit) {
    const int b = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int top = t0_top[b], cnt = rl_count[b], N = pos_n[b];
    if (i < n) {
        const int sl = t0_free[(size_t)b * S0 + top - 1 - i];
        const size_t p = (size_t)b * Nmax + N + i;
        tier[p] = 0;
        slot[p] = sl;
        s[p] = 0.f;
        const size_t j = (size_t)b * Nmax + cnt + i;
        rl_loc[j] = make_loc(0, sl);
        rl_pos[j] = N + i;
    }
    if (commit) {
        __syncthreads();
        if (threadIdx.x == 0) {
            t0_top[b] = top - n;
            rl_count[b] = cnt + n;
            pos_n[b] = N + n;
        }
    }
}

__global__ void open_commit_kernel(int32_t* t0_top, int32_t* rl_count, int32_t* pos_n, int B, int n) {
    const int b = threadIdx.x;
    if (b < B) {
        t0_top[b] -= n;
        rl_count[b] += n;
        pos_n[b] += n;
    }
}

cudaError_t launch_open(int32_t* t0_free, int32_t* t0_top, uint8_t* tier, int32_t* slot, float* s,
                        uint32_t* rl_loc, int32_t* rl_pos, int32_t* rl_count, int32_t* pos_n, int B, int Nmax,
                        int S0, int n, cudaStream_t st, int* launches) {
    dim3 grid((n + 255) / 256, B);
    const int fused = n <= 256;
    open_kernel<<<grid, 256, 0, st>>>(t0_free, t0_top, tier, slot, s, rl_loc, rl_pos, rl_count, pos_n, Nmax,
                                      S0, n, fused);
    *launches = 1;
    if (!fused) {
        open_commit_kernel<<<1, 32 * ((B + 31) / 32), 0, st>>>(t0_top, rl_count, pos_n, B, n);
        *launches = 2;
    }
    return cudaGetLastError();
}

// Copies the rows of n new positions of one layer into their T0 slots.
// k, v: [B][n][Hkv][d].  One thread per 16 bytes.
__global__ void append_rows_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                   __nv_bfloat16* k0v0, const int32_t* __restrict__ slot, int layer,
                                   int B, int Hkv, int d, int Nmax, int S0, int N, int n) {
    const int cpr = d / 8;   // 16-byte chunks per row
    const long long total = (long long)B * n * 2 * Hkv * cpr;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(e % cpr);
        long long row = e / cpr;
        const int h = (int)(row % Hkv);
        row /= Hkv;
        const int kv = (int)(row % 2);
        row /= 2;
        const int i = (int)(row % n);
        const int b = (int)(row / n);
        const size_t src = (((size_t)b * n + i) * Hkv + h) * cpr + c;
        const int sl = slot[(size_t)b * Nmax + N + i];
        const uint4 w = kv ? v[src] : k[src];
        *reinterpret_cast<uint4*>(k0v0 + row_index(layer, kv, b, h, sl, B, Hkv, S0) * d + c * 8) = w;
    }
}

cudaError_t launch_append_rows(const __nv_bfloat16* k, const __nv_bfloat16* v,
                               __nv_bfloat16* k0v0, const int32_t* slot, int layer, int B,
                               int Hkv, int d, int Nmax, int S0, int N, int n, cudaStream_t st) {
    const long long total = (long long)B * n * 2 * Hkv * (d / 8);
    const int blocks = (int)std::min<long long>((total + 255) / 256, 152LL * 16);
    append_rows_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const uint4*>(k),
                                               reinterpret_cast<const uint4*>(v), k0v0, slot, layer, B,
                                               Hkv, d, Nmax, S0, N, n);
    return cudaGetLastError();
}

}  // namespace tkv
