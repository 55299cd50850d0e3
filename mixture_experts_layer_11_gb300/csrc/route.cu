// route.cu -- router logits, softmax top-k gate, stable dispatch by expert,
// and the router backward (steps A1, A2, A3, A10 of the layer).
//
// The gating network's output decides each token's experts; tokens are then
// assigned to their target experts in token order, so that each expert sees
// one contiguous segment and no dispatch mask is built ("ES-MoE: Scaling
// Beyond the GPU Memory Limit for Large Mixture-of-Experts Model Training",
// review, section 3 "expert-wise offloading and processing"; "FastMoE",
// review, "proposed method": scatter/gather layout batching inputs by expert).
//
// Dispatch design: each block of 64 tokens records, per expert, a 64-bit
// mask of the tokens routed there (2 words of 32 bits).  Popcounts of those
// masks give the block's histogram; one single-block scan over the
// expert-major (expert, block) table gives every block's base row per expert;
// a token's rank inside its block is a popcount of the mask bits below it.
// Positions are therefore a pure function of idx: deterministic and stable.
#include <float.h>
#include <limits.h>
#include <stdlib.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float warp_max(float v) {
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// ---- vector load / store of 8 (bf16) or 4 (fp32) elements as fp32 ----------------

template <typename T> struct Vec;
template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* v) {
        uint4 u = *reinterpret_cast<const uint4*>(p);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
        #pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(h[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void unpack(const uint4& u, float* v) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
        #pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(h[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float* v) {
        uint4 u;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
        #pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        *reinterpret_cast<uint4*>(p) = u;
    }
};
template <> struct Vec<float> {
    static constexpr int N = 4;
    static __device__ __forceinline__ void load(const float* p, float* v) {
        float4 u = *reinterpret_cast<const float4*>(p);
        v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
    }
    static __device__ __forceinline__ void unpack(const uint4& u, float* v) {
        v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
        v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
    }
    static __device__ __forceinline__ void store(float* p, const float* v) {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};

// ---- A1: router logits for many experts: register-tiled SIMT GEMM ------------------
//
// logits[t][e] = sum_c x[t][c] Wg[e][c] + beta[e] with fp32 accumulation on the
// CUDA cores.  Tile 128 tokens x 32*NG experts (NG = 4, or 2 when E <= 64) per
// block of 128 threads; each thread owns 8 rows x 4*NG columns (rows ty*4+i
// and 64+ty*4+i, columns g*32+tx*4+w), accumulated as packed fp32 pairs
// (fma.rn.f32x2: one issue slot for two FMAs, each rounded as the scalar FMA).  K in steps of 16 through
// double-buffered shared memory (fp32, K-major, so that a thread reads its 4
// consecutive rows or columns as one 16-byte load).
//
// Work split ("stream-K"): the grid holds as many blocks as are co-resident,
// and the (tile, K step) iterations of the whole problem are cut into equal
// contiguous ranges, one per block, so every SM gets the same work whatever
// the tile count.  A block whose range holds a whole tile writes its logits;
// the pieces of a tile split between consecutive blocks go to scratch as fp32
// partial tiles, and a fix-up kernel adds them in block order (= K order) and
// adds beta: deterministic.  Without scratch (part == nullptr) every block
// takes whole tiles.

constexpr int kRtM = 128, kRtK = 16, kRtThreads = 128;

__device__ __forceinline__ uint64_t rt_pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void rt_unpack(uint64_t r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t rt_fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

struct RouterSplit {
    int G;              // blocks
    int64_t iters;      // tiles * ksteps
    int ksteps;         // K steps of 16 per tile
    int ntn;            // expert tiles
    int maxp;           // pieces per block (scratch slots)
    int bn;             // experts per tile (32 * NG)
};

// first iteration of block b
__device__ __forceinline__ int64_t rt_it0(const RouterSplit& sp, int b) {
    return (int64_t)b * sp.iters / sp.G;
}

template <typename TIn, int NG>
__global__ void __launch_bounds__(kRtThreads, 2) router_logits_tiled_kernel(
    int64_t T, int d, int E, const TIn* __restrict__ x, const TIn* __restrict__ Wg,
    const float* __restrict__ beta, float* __restrict__ logits, float* __restrict__ part,
    RouterSplit sp) {
    constexpr int VN = Vec<TIn>::N;            // elements per 16-byte load
    constexpr int LPR = kRtK / VN;             // 16-byte loads per row per K step
    constexpr int BNT = 32 * NG;               // experts per tile
    __shared__ __align__(16) float As[2][kRtK][kRtM];
    __shared__ __align__(16) float Bs[2][kRtK][BNT];
    const int tid = threadIdx.x;
    const int ty = tid >> 3, tx = tid & 7;
    const int b = blockIdx.x;
    int64_t it = rt_it0(sp, b);
    const int64_t it_end = rt_it0(sp, b + 1);
    int piece = 0;
    while (it < it_end) {
        const int64_t tile = it / sp.ksteps;
        const int ks0 = (int)(it % sp.ksteps);
        const int64_t rem = it_end - it;
        const int ks1 = (int)((int64_t)sp.ksteps < ks0 + rem ? (int64_t)sp.ksteps : ks0 + rem);
        const int64_t m0 = (tile / sp.ntn) * kRtM;
        const int n0 = (int)(tile % sp.ntn) * BNT;
        // this thread's row of the A tile (token m0 + tid) and of the B tile
        // (expert n0 + tid), K columns [k, k + 16), kept packed until stored
        uint4 ra[LPR], rb[LPR];
        auto load = [&](int ks) {
            const int k = ks * kRtK;
            const int64_t gm = m0 + tid;
            const int gn = n0 + tid;
            #pragma unroll
            for (int l = 0; l < LPR; ++l) {
                const int c = k + l * VN;
                ra[l] = (gm < T && c < d) ? *reinterpret_cast<const uint4*>(x + gm * d + c)
                                          : make_uint4(0, 0, 0, 0);
                rb[l] = (tid < BNT && gn < E && c < d)
                            ? *reinterpret_cast<const uint4*>(Wg + (int64_t)gn * d + c)
                            : make_uint4(0, 0, 0, 0);
            }
        };
        auto store = [&](int buf) {
            #pragma unroll
            for (int l = 0; l < LPR; ++l) {
                float va[VN], vb[VN];
                Vec<TIn>::unpack(ra[l], va);
                Vec<TIn>::unpack(rb[l], vb);
                #pragma unroll
                for (int u = 0; u < VN; ++u) {
                    As[buf][l * VN + u][tid] = va[u];
                    if (tid < BNT) Bs[buf][l * VN + u][tid] = vb[u];
                }
            }
        };
        uint64_t acc[8][2 * NG];
        #pragma unroll
        for (int i = 0; i < 8; ++i)
            #pragma unroll
            for (int j = 0; j < 2 * NG; ++j) acc[i][j] = 0;
        __syncthreads();   // the previous piece's last reads of the buffers are done
        load(ks0);
        store(0);
        __syncthreads();
        int buf = 0;
        for (int ks = ks0; ks < ks1; ++ks) {
            const bool more = ks + 1 < ks1;
            if (more) load(ks + 1);
            #pragma unroll
            for (int kk = 0; kk < kRtK; ++kk) {
                const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
                const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
                uint64_t bp[2 * NG];
                #pragma unroll
                for (int g = 0; g < NG; ++g) {
                    const ulonglong2 v =
                        *reinterpret_cast<const ulonglong2*>(&Bs[buf][kk][g * 32 + tx * 4]);
                    bp[2 * g] = v.x;
                    bp[2 * g + 1] = v.y;
                }
                const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                #pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint64_t sa = rt_pack(a[i], a[i]);
                    #pragma unroll
                    for (int j = 0; j < 2 * NG; ++j) acc[i][j] = rt_fma2(sa, bp[j], acc[i][j]);
                }
            }
            if (more) {
                store(buf ^ 1);
                __syncthreads();
                buf ^= 1;
            }
        }
        const bool whole = ks0 == 0 && ks1 == sp.ksteps;
        float* pt = whole ? nullptr : part + ((int64_t)b * sp.maxp + piece) * (kRtM * BNT);
        #pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4);
            const int64_t t = m0 + r;
            #pragma unroll
            for (int g = 0; g < NG; ++g) {
                const int cl = g * 32 + tx * 4;   // column inside the tile
                float o[4];
                rt_unpack(acc[i][2 * g], o[0], o[1]);
                rt_unpack(acc[i][2 * g + 1], o[2], o[3]);
                if (!whole) {
                    *reinterpret_cast<float4*>(pt + r * BNT + cl) = make_float4(o[0], o[1], o[2], o[3]);
                    continue;
                }
                if (t >= T) continue;
                const int e0 = n0 + cl;
                #pragma unroll
                for (int j = 0; j < 4; ++j) o[j] += (beta && e0 + j < E) ? beta[e0 + j] : 0.f;
                if ((E & 3) == 0 && e0 + 3 < E) {
                    *reinterpret_cast<float4*>(logits + t * E + e0) = make_float4(o[0], o[1], o[2], o[3]);
                } else {
                    #pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (e0 + j < E) logits[t * E + e0 + j] = o[j];
                }
            }
        }
        it += ks1 - ks0;
        ++piece;
    }
}

// Tiles split between blocks: logits = the pieces in block order + beta.  One
// block per tile; tiles held whole by one block were written by it.  The
// tile's pieces (block, piece index) are listed once in shared memory.
__global__ void __launch_bounds__(256) router_logits_fixup_kernel(
    int64_t T, int E, const float* __restrict__ beta, float* __restrict__ logits,
    const float* __restrict__ part, RouterSplit sp) {
    constexpr int kMaxPieces = 32;   // > the 16 blocks a tile is shared by, plus its ends
    __shared__ int npc;
    __shared__ int64_t pslot[kMaxPieces];
    const int64_t tile = blockIdx.x;
    if (threadIdx.x == 0) {
        const int64_t first = tile * sp.ksteps, last = first + sp.ksteps;   // iterations
        // the block holding iteration `first`: the last b with it0(b) <= first
        int b = (int)(first * sp.G / sp.iters);
        while (b + 1 < sp.G && rt_it0(sp, b + 1) <= first) ++b;
        while (b > 0 && rt_it0(sp, b) > first) --b;
        int n = 0;
        if (!(rt_it0(sp, b) <= first && rt_it0(sp, b + 1) >= last)) {   // not whole
            for (int bb = b; bb < sp.G && n < kMaxPieces; ++bb) {
                const int64_t it0 = rt_it0(sp, bb);
                if (it0 >= last) break;
                if (rt_it0(sp, bb + 1) <= it0) continue;   // an empty block
                // the piece of block bb holding this tile: tiles counted from its first
                pslot[n++] = ((int64_t)bb * sp.maxp + (tile - it0 / sp.ksteps)) *
                             ((int64_t)kRtM * sp.bn);
            }
        }
        npc = n;
    }
    __syncthreads();
    const int n = npc;
    if (n == 0) return;
    const int64_t m0 = (tile / sp.ntn) * kRtM;
    const int n0 = (int)(tile % sp.ntn) * sp.bn;
    const int vpr = sp.bn / 4;   // float4 per tile row
    for (int i = threadIdx.x; i < kRtM * vpr; i += blockDim.x) {
        const int r = i / vpr, c = (i % vpr) * 4;
        const int64_t t = m0 + r;
        if (t >= T) continue;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q = 0; q < n; ++q) {
            const float4 v = *reinterpret_cast<const float4*>(part + pslot[q] + r * sp.bn + c);
            a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
        }
        const int e0 = n0 + c;
        float o[4] = {a.x, a.y, a.z, a.w};
        #pragma unroll
        for (int j = 0; j < 4; ++j) o[j] += (beta && e0 + j < E) ? beta[e0 + j] : 0.f;
        if ((E & 3) == 0 && e0 + 3 < E) {
            *reinterpret_cast<float4*>(logits + t * E + e0) = make_float4(o[0], o[1], o[2], o[3]);
        } else {
            #pragma unroll
            for (int j = 0; j < 4; ++j)
                if (e0 + j < E) logits[t * E + e0 + j] = o[j];
        }
    }
}

// Blocks of the router logits kernel (64- or 128-expert tiles) that fit on the
// device at once.
int router_logits_slots(bool narrow) {
    static int cache[64][2] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return device_sm_count() * 2;
    int& c = cache[dev][narrow ? 1 : 0];
    if (c == 0) {
        int n = 0;
        if (narrow)
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &n, router_logits_tiled_kernel<__nv_bfloat16, 2>, kRtThreads, 0);
        else
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &n, router_logits_tiled_kernel<__nv_bfloat16, 4>, kRtThreads, 0);
        c = device_sm_count() * (n > 0 ? n : 1);
    }
    return c;
}

template <typename TIn>
cudaError_t router_logits_dispatch(const moe_shape& s, const TIn* x, const TIn* Wg,
                                   const float* beta, float* logits, float* part,
                                   size_t part_bytes, cudaStream_t st) {
    RouterSplit sp;
    const bool narrow = s.E <= 64;   // 64-expert tiles
    sp.bn = narrow ? 64 : 128;
    const int64_t mt = (s.T + kRtM - 1) / kRtM;
    sp.ntn = (s.E + sp.bn - 1) / sp.bn;
    sp.ksteps = (s.d + kRtK - 1) / kRtK;
    const int64_t tiles = mt * sp.ntn;
    sp.iters = tiles * sp.ksteps;
    const int64_t slots = router_logits_slots(narrow);
    const size_t tile_bytes = (size_t)kRtM * sp.bn * sizeof(float);
    bool split = part != nullptr && tiles % slots != 0;
    if (split) {
        // at most 16 blocks share a tile (the fix-up lists a tile's pieces)
        int64_t g = slots < sp.iters ? slots : sp.iters;
        if (g > 16 * tiles) g = 16 * tiles;
        sp.G = (int)g;
        const int64_t per = (sp.iters + sp.G - 1) / sp.G;
        sp.maxp = (int)(per / sp.ksteps + 2);
        if ((size_t)sp.G * sp.maxp * tile_bytes > part_bytes) split = false;
    }
    if (!split) {   // whole tiles, one per block
        sp.G = (int)tiles;
        sp.maxp = 1;
        part = nullptr;
    }
    if (sp.G <= 0) return cudaSuccess;
    if (narrow)
        router_logits_tiled_kernel<TIn, 2><<<sp.G, kRtThreads, 0, st>>>(s.T, s.d, s.E, x, Wg,
                                                                       beta, logits, part, sp);
    else
        router_logits_tiled_kernel<TIn, 4><<<sp.G, kRtThreads, 0, st>>>(s.T, s.d, s.E, x, Wg,
                                                                       beta, logits, part, sp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !split) return e;
    router_logits_fixup_kernel<<<(unsigned)tiles, 256, 0, st>>>(s.T, s.E, beta, logits, part, sp);
    return cudaGetLastError();
}

// ---- A2: softmax top-k gate + per-block expert bitmask histogram ----------------
//
// One warp per token; lane l holds logits of experts l, l+32, ...  Top-k by k
// rounds of a warp arg-max on (logit desc, expert index asc).  A NaN logit is
// ranked below every number (so k distinct valid experts are always chosen)
// and, like an infinite one, raises MOE_ERR_NONFINITE.  Blocks hold 64 tokens
// (the bitmask histogram) and 8 warps, 8 tokens per warp.

template <int EPL>
__device__ __forceinline__ void gate_token(int64_t t, int E, int k, int renorm, float (&L)[EPL],
                                           int lane, int tok, uint32_t (*bits)[kRouteWords],
                                           int32_t* __restrict__ idx, float* __restrict__ w,
                                           int32_t* status) {
    bool bad = false;
    #pragma unroll
    for (int q = 0; q < EPL; ++q) {
        const int e = lane + 32 * q;
        if (e < E) {
            if (!isfinite(L[q])) bad = true;
            if (isnan(L[q])) L[q] = -INFINITY;
        } else {
            L[q] = -INFINITY;
        }
    }
    if (__any_sync(kFull, bad) && lane == 0) report(status, MOE_ERR_NONFINITE);
    float m = L[0];
    #pragma unroll
    for (int q = 1; q < EPL; ++q) m = fmaxf(m, L[q]);
    m = warp_max(m);
    float z = 0.f;
    #pragma unroll
    for (int q = 0; q < EPL; ++q)
        if (lane + 32 * q < E) z += expf(L[q] - m);
    z = warp_sum(z);

    uint32_t taken = 0u;
    int my_e = 0;
    float my_p = 0.f, psum = 0.f;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int be = INT_MAX;
        #pragma unroll
        for (int q = 0; q < EPL; ++q) {
            const int e = lane + 32 * q;
            if (e < E && !((taken >> q) & 1u) && (be == INT_MAX || L[q] > bv)) {
                bv = L[q];
                be = e;
            }
        }
        #pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(kFull, bv, o);
            const int oe = __shfl_xor_sync(kFull, be, o);
            if (oe != INT_MAX && (be == INT_MAX || ov > bv || (ov == bv && oe < be))) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        const float p = expf(bv - m) / z;
        if (lane == j) { my_e = be; my_p = p; }
        psum += p;
        if (lane == 0) atomicOr(&bits[be][tok >> 5], 1u << (tok & 31));
    }
    if (lane < k) {
        idx[t * k + lane] = my_e;
        w[t * k + lane] = renorm ? my_p / psum : my_p;
    }
}

__device__ __forceinline__ void zero_bits(uint32_t (*bits)[kRouteWords], int E) {
    for (int i = threadIdx.x; i < E * kRouteWords; i += blockDim.x)
        bits[i / kRouteWords][i % kRouteWords] = 0u;
}

__device__ __forceinline__ void write_block_counts(uint32_t (*bits)[kRouteWords], int E, int nblk,
                                                   int32_t* block_counts) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int c = 0;
        #pragma unroll
        for (int q = 0; q < kRouteWords; ++q) c += __popc(bits[e][q]);
        block_counts[(int64_t)e * nblk + blockIdx.x] = c;
    }
}

// Gate on logits already in memory (given, or from a logits GEMM).  WARPS
// warps per 64-token block, 64 / WARPS tokens each: the per-token work is a
// chain of dependent shuffles, so many warps are kept in flight.
template <int EPL, int WARPS>
__global__ void __launch_bounds__(WARPS * 32) gate_hist_kernel(
    int64_t T, int E, int k, int renorm, int nblk, const float* __restrict__ logits,
    int32_t* __restrict__ idx, float* __restrict__ w, int32_t* __restrict__ block_counts,
    int32_t* status) {
    constexpr int TOK = kRouteBlockTokens / WARPS;
    __shared__ uint32_t bits[256][kRouteWords];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    zero_bits(bits, E);
    __syncthreads();
    for (int tt = 0; tt < TOK; ++tt) {
        const int tok = warp * TOK + tt;
        const int64_t t = (int64_t)blockIdx.x * kRouteBlockTokens + tok;
        if (t >= T) break;
        float L[EPL];
        #pragma unroll
        for (int q = 0; q < EPL; ++q) {
            const int e = lane + 32 * q;
            L[q] = (e < E) ? logits[t * E + e] : -INFINITY;
        }
        gate_token<EPL>(t, E, k, renorm, L, lane, tok, bits, idx, w, status);
    }
    __syncthreads();
    write_block_counts(bits, E, nblk, block_counts);
}

// Few experts (E <= 32): router logits, gate and histogram fused, one warp per
// token.  Each lane accumulates EP (= E rounded up to a power of two) partial
// dot products over its share of the row (16-byte loads of x and Wg, Wg
// staying in L1), then a reduce-scatter across the warp leaves expert e's sum
// in lanes e*32/EP ... e*32/EP + 32/EP - 1.
template <int EP>
__device__ __forceinline__ float reduce_scatter(float (&v)[EP], int lane) {
    #pragma unroll
    for (int half = EP / 2, off = 16; half >= 1; half >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
        #pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(kFull, send, off);
        }
    }
    float r = v[0];
    #pragma unroll
    for (int o = 16 / EP; o >= 1; o >>= 1) r += __shfl_xor_sync(kFull, r, o);
    return r;
}

// Router logits + gate for E <= 32, one launch.  A block owns one 64-token
// dispatch block; its WARPS warps own 64 / WARPS tokens each and take TPW of
// them at a time (their Wg loads shared).  Many warps per block keep enough
// loads in flight: the work per token is small and latency-bound.
template <typename TIn, int EP, int WARPS, int TPW>
__global__ void __launch_bounds__(WARPS * 32) router_gate_small_kernel(
    int64_t T, int d, int E, int k, int renorm, int nblk, const TIn* __restrict__ x,
    const TIn* __restrict__ Wg, const float* __restrict__ beta, float* __restrict__ logits,
    int32_t* __restrict__ idx, float* __restrict__ w, int32_t* __restrict__ block_counts,
    int32_t* status) {
    using V = Vec<TIn>;
    constexpr int TOK = kRouteBlockTokens / WARPS;   // tokens per warp
    __shared__ uint32_t bits[256][kRouteWords];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    zero_bits(bits, E);
    __syncthreads();
    const int nv = d / V::N;
    for (int tt0 = 0; tt0 < TOK; tt0 += TPW) {
        const int64_t t0 = (int64_t)blockIdx.x * kRouteBlockTokens + warp * TOK + tt0;
        if (t0 >= T) break;
        float acc[TPW][EP];
        #pragma unroll
        for (int i = 0; i < TPW; ++i)
            #pragma unroll
            for (int e = 0; e < EP; ++e) acc[i][e] = 0.f;
        #pragma unroll 2
        for (int c = lane; c < nv; c += 32) {
            float xv[TPW][V::N], wv[V::N];
            #pragma unroll
            for (int i = 0; i < TPW; ++i) {
                if (t0 + i < T) V::load(x + (t0 + i) * d + (int64_t)c * V::N, xv[i]);
                else
                    #pragma unroll
                    for (int u = 0; u < V::N; ++u) xv[i][u] = 0.f;
            }
            #pragma unroll
            for (int e = 0; e < EP; ++e) {
                if (e < E) {
                    V::load(Wg + (int64_t)e * d + (int64_t)c * V::N, wv);
                    #pragma unroll
                    for (int i = 0; i < TPW; ++i)
                        #pragma unroll
                        for (int u = 0; u < V::N; ++u) acc[i][e] = fmaf(xv[i][u], wv[u], acc[i][e]);
                }
            }
        }
        #pragma unroll
        for (int i = 0; i < TPW; ++i) {
            const int64_t t = t0 + i;
            const float r = reduce_scatter<EP>(acc[i], lane);
            if (t >= T) continue;   // warp-uniform
            // lane e (< E) takes expert e's sum
            const float le = __shfl_sync(kFull, r, (lane % EP) * (32 / EP));
            float L[1];
            L[0] = -INFINITY;
            if (lane < E) {
                L[0] = le + (beta ? beta[lane] : 0.f);
                logits[t * E + lane] = L[0];
            }
            gate_token<1>(t, E, k, renorm, L, lane, warp * TOK + tt0 + i, bits, idx, w, status);
        }
    }
    __syncthreads();
    write_block_counts(bits, E, nblk, block_counts);
}

template <typename TIn>
cudaError_t router_gate_small(const moe_shape& s, const TIn* x, const TIn* Wg, const float* beta,
                              float* logits, int32_t* idx, float* w, int32_t* block_counts,
                              int32_t* status, cudaStream_t st) {
    const int nblk = (int)route_blocks(s.T);
#define MOE_SMALL(EPV, WV, TV)                                                             \
    router_gate_small_kernel<TIn, EPV, WV, TV><<<nblk, (WV) * 32, 0, st>>>(                \
        s.T, s.d, s.E, s.k, s.renorm, nblk, x, Wg, beta, logits, idx, w, block_counts, status)
    if (s.E <= 1) MOE_SMALL(1, 32, 2);
    else if (s.E <= 2) MOE_SMALL(2, 32, 2);
    else if (s.E <= 4) MOE_SMALL(4, 32, 2);
    else if (s.E <= 8) MOE_SMALL(8, 32, 2);
    else if (s.E <= 16) MOE_SMALL(16, 16, 2);
    else MOE_SMALL(32, 16, 1);
#undef MOE_SMALL
    return cudaGetLastError();
}

// ---- A3: scan of the expert-major (expert, block) histogram ---------------------

__global__ void __launch_bounds__(1024) dispatch_scan_kernel(int E, int nblk, int32_t* data,
                                                            int32_t* counts,
                                                            int32_t* offsets) {
    // data: the expert-major table [E][nblk] of per-block counts, replaced by its
    // exclusive prefix sums in that order.  A warp takes whole experts and reads
    // their rows 32 consecutive entries at a time (coalesced): their totals,
    // then one scan of the E totals, then each row's prefixes from its base.
    __shared__ int base_s[kMaxExperts];
    __shared__ int grand;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    constexpr int U = 8;   // 32-entry loads in flight per lane
    for (int e = wid; e < E; e += 32) {
        const int32_t* row = data + (int64_t)e * nblk;
        int s = 0;
        for (int j0 = 0; j0 < nblk; j0 += 32 * U) {
            int v[U];
            #pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = j0 + 32 * u + lane;
                v[u] = j < nblk ? row[j] : 0;
            }
            #pragma unroll
            for (int u = 0; u < U; ++u) s += v[u];
        }
        #pragma unroll
        for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
        if (lane == 0) base_s[e] = s;
    }
    __syncthreads();
    if (wid == 0) {
        // exclusive scan of the E <= kMaxExperts (256) totals: 8 consecutive per lane
        int t[8], sum = 0;
        #pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane * 8 + i;
            t[i] = e < E ? base_s[e] : 0;
            sum += t[i];
        }
        int incl = sum;
        #pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
        __syncwarp();
        #pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane * 8 + i;
            if (e < E) base_s[e] = run;
            run += t[i];
        }
        if (lane == 31) grand = incl;
    }
    __syncthreads();
    for (int e = wid; e < E; e += 32) {
        int32_t* row = data + (int64_t)e * nblk;
        int run = base_s[e];
        for (int j0 = 0; j0 < nblk; j0 += 32 * U) {
            int v[U];
            #pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = j0 + 32 * u + lane;
                v[u] = j < nblk ? row[j] : 0;
            }
            #pragma unroll
            for (int u = 0; u < U; ++u) {
                int incl = v[u];
                #pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int x = __shfl_up_sync(kFull, incl, o);
                    if (lane >= o) incl += x;
                }
                const int j = j0 + 32 * u + lane;
                if (j < nblk) row[j] = run + incl - v[u];
                run += __shfl_sync(kFull, incl, 31);
            }
        }
        if (lane == 0) {
            offsets[e] = base_s[e];
            counts[e] = (e + 1 < E ? base_s[e + 1] : grand) - base_s[e];
        }
    }
    if (threadIdx.x == 0) offsets[E] = grand;
}

// ---- A3: stable rank inside each block -> pos, perm ------------------------------

__global__ void __launch_bounds__(kRouteBlockTokens) dispatch_rank_kernel(
    int64_t T, int E, int k, int nblk, const int32_t* __restrict__ idx,
    const int32_t* __restrict__ block_base, int32_t* __restrict__ pos,
    int32_t* __restrict__ perm) {
    __shared__ uint32_t bits[256][kRouteWords];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < E * kRouteWords; i += blockDim.x)
        bits[i / kRouteWords][i % kRouteWords] = 0u;
    __syncthreads();
    const int64_t t = (int64_t)blockIdx.x * kRouteBlockTokens + threadIdx.x;
    if (t < T)
        for (int j = 0; j < k; ++j) atomicOr(&bits[idx[t * k + j]][warp], 1u << lane);
    __syncthreads();
    if (t >= T) return;
    const uint32_t below = (1u << lane) - 1u;
    for (int j = 0; j < k; ++j) {
        const int e = idx[t * k + j];
        int r = __popc(bits[e][warp] & below);
        for (int q = 0; q < warp; ++q) r += __popc(bits[e][q]);
        const int32_t p = block_base[(int64_t)e * nblk + blockIdx.x] + r;
        pos[t * k + j] = p;
        perm[p] = (int32_t)(t * k + j);
    }
}

// ---- A10: router backward ----------------------------------------------------------
//
// Warp per token.  renorm: dL_j = w_j (dw_j - sum_i w_i dw_i) on the k selected
// experts (stored [T][k]).  Otherwise the full softmax Jacobian (stored
// [T][E]).  dx[t] += sum_e dL[t][e] Wg[e] (read-modify-write in the storage
// dtype, fp32 arithmetic).

template <typename TIn, int EPL, int KMAX>
__global__ void __launch_bounds__(256, KMAX <= 4 ? 3 : (KMAX <= 8 ? 2 : 1)) route_bwd_dx_kernel(
    int64_t T, int d, int E, int k, int renorm, const float* __restrict__ dw,
    const float* __restrict__ logits, const int32_t* __restrict__ idx,
    const float* __restrict__ w, const TIn* __restrict__ Wg,
    const TIn* __restrict__ dx_perm, const int32_t* __restrict__ pos, TIn* __restrict__ dx,
    float* __restrict__ dL, int dl_only) {
    __shared__ float g_s[8][256];
    __shared__ int e_s[8][256];
    using V = Vec<TIn>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * 8 + warp;
    if (t >= T) return;
    constexpr int VN = V::N;
    // vectors per lane in flight: U * KMAX row loads before any use
    constexpr int U = KMAX >= 4 ? 1 : (KMAX == 2 ? 2 : 4);
    // The gather of the permute backward (rows pos[t, j] of dx_perm) does not
    // depend on dL: its first loads are issued before dL is computed.
    int32_t p[KMAX];
    #pragma unroll
    for (int j = 0; j < KMAX; ++j) p[j] = (dx_perm && j < k) ? pos[t * k + j] : 0;
    uint4 raw[U][KMAX];
    auto gather = [&](int c0) {
        #pragma unroll
        for (int u = 0; u < U; ++u)
            #pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (j < k && c0 + 32 * VN * u < d)
                    raw[u][j] = __ldg(reinterpret_cast<const uint4*>(
                        dx_perm + (int64_t)p[j] * d + c0 + 32 * VN * u));
    };
    if (dx_perm) gather(lane * VN);
    int ng;  // number of (expert, dL) terms for this token
    if (renorm) {
        float wj = 0.f, dwj = 0.f;
        int ej = 0;
        if (lane < k) {
            wj = w[t * k + lane];
            dwj = dw[t * k + lane];
            ej = idx[t * k + lane];
        }
        const float sdot = warp_sum(wj * dwj);
        if (lane < k) {
            const float g = wj * (dwj - sdot);
            dL[t * k + lane] = g;
            g_s[warp][lane] = g;
            e_s[warp][lane] = ej;
        }
        ng = k;
    } else {
        float L[EPL], p[EPL];
        #pragma unroll
        for (int q = 0; q < EPL; ++q) {
            const int e = lane + 32 * q;
            L[q] = (e < E) ? logits[t * E + e] : -INFINITY;
        }
        float m = L[0];
        #pragma unroll
        for (int q = 1; q < EPL; ++q) m = fmaxf(m, L[q]);
        m = warp_max(m);
        float z = 0.f;
        #pragma unroll
        for (int q = 0; q < EPL; ++q) {
            p[q] = (lane + 32 * q < E) ? expf(L[q] - m) : 0.f;
            z += p[q];
        }
        z = warp_sum(z);
        #pragma unroll
        for (int q = 0; q < EPL; ++q) p[q] /= z;
        // c_j = dw_j * p[idx_j];  dL_e = -p_e * sum_j c_j + sum_j c_j [e == idx_j]
        float add[EPL];
        #pragma unroll
        for (int q = 0; q < EPL; ++q) add[q] = 0.f;
        float csum = 0.f;
        for (int j = 0; j < k; ++j) {
            const int a = idx[t * k + j];
            float pa_l = 0.f;
            #pragma unroll
            for (int q = 0; q < EPL; ++q)
                if (q == (a >> 5)) pa_l = p[q];
            const float pa = __shfl_sync(kFull, pa_l, a & 31);
            const float c = dw[t * k + j] * pa;
            csum += c;
            #pragma unroll
            for (int q = 0; q < EPL; ++q)
                if (lane + 32 * q == a) add[q] += c;
        }
        #pragma unroll
        for (int q = 0; q < EPL; ++q) {
            const int e = lane + 32 * q;
            if (e < E) {
                const float g = add[q] - p[q] * csum;
                dL[t * E + e] = g;
                g_s[warp][e] = g;
                e_s[warp][e] = e;
            }
        }
        ng = E;
    }
    if (dl_only) return;   // dx by the tiled dense kernel
    __syncwarp();
    for (int c0 = lane * VN; c0 < d; c0 += 32 * VN * U) {
        float acc[U][VN], wv[VN];
        if (dx_perm) {
            // permute backward fused in: dx = sum_j dx_perm[pos[t,j]] + router term
            // (the rows of this step were gathered one step ahead)
            #pragma unroll
            for (int u = 0; u < U; ++u) {
                #pragma unroll
                for (int e = 0; e < VN; ++e) acc[u][e] = 0.f;
                #pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    if (j >= k || c0 + 32 * VN * u >= d) break;
                    float xr[VN];
                    V::unpack(raw[u][j], xr);
                    #pragma unroll
                    for (int e = 0; e < VN; ++e) acc[u][e] += xr[e];
                }
            }
            if (c0 + 32 * VN * U < d) gather(c0 + 32 * VN * U);
        } else {
            #pragma unroll
            for (int u = 0; u < U; ++u)
                if (c0 + 32 * VN * u < d) V::load(dx + t * d + c0 + 32 * VN * u, acc[u]);
        }
        if (KMAX > 1 && ng <= KMAX) {
            // the gate rows of all terms are requested before the first is used
            uint4 wr[KMAX][U];
            #pragma unroll
            for (int i = 0; i < KMAX; ++i)
                #pragma unroll
                for (int u = 0; u < U; ++u)
                    if (i < ng && c0 + 32 * VN * u < d)
                        wr[i][u] = __ldg(reinterpret_cast<const uint4*>(
                            Wg + (int64_t)e_s[warp][i] * d + c0 + 32 * VN * u));
            #pragma unroll
            for (int i = 0; i < KMAX; ++i) {
                if (i >= ng) break;
                const float g = g_s[warp][i];
                #pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (c0 + 32 * VN * u >= d) break;
                    V::unpack(wr[i][u], wv);
                    #pragma unroll
                    for (int e = 0; e < VN; ++e) acc[u][e] = fmaf(g, wv[e], acc[u][e]);
                }
            }
        } else {
            for (int i = 0; i < ng; ++i) {
                const float g = g_s[warp][i];
                const TIn* wrow = Wg + (int64_t)e_s[warp][i] * d;
                #pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (c0 + 32 * VN * u >= d) break;
                    V::load(wrow + c0 + 32 * VN * u, wv);
                    #pragma unroll
                    for (int e = 0; e < VN; ++e) acc[u][e] = fmaf(g, wv[e], acc[u][e]);
                }
            }
        }
        #pragma unroll
        for (int u = 0; u < U; ++u)
            if (c0 + 32 * VN * u < d) V::store(dx + t * d + c0 + 32 * VN * u, acc[u]);
    }
}

// ---- A10, dense gate Jacobian (renorm off): two tiled products ------------------
// With renorm off every expert's logit gets a gradient, so dx's router term
// is the product dL [T, E] x Wg [E, d] and dWg = dL^T x: fp32 CUDA-core
// products tiled through shared memory (64 x 128 outputs per block, 8 x 4 per
// thread), with the reduction dimension in order.

template <typename T> struct Four;   // four consecutive elements
template <> struct Four<__nv_bfloat16> {
    static __device__ __forceinline__ float4 load(const __nv_bfloat16* p) {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, float4 v) {
        uint2 u;
        *reinterpret_cast<__nv_bfloat162*>(&u.x) = __floats2bfloat162_rn(v.x, v.y);
        *reinterpret_cast<__nv_bfloat162*>(&u.y) = __floats2bfloat162_rn(v.z, v.w);
        *reinterpret_cast<uint2*>(p) = u;
    }
};
template <> struct Four<float> {
    static __device__ __forceinline__ float4 load(const float* p) {
        return *reinterpret_cast<const float4*>(p);
    }
    static __device__ __forceinline__ void store(float* p, float4 v) {
        *reinterpret_cast<float4*>(p) = v;
    }
};

// dx[t, :] = sum_j dx_perm[pos[t, j], :] (or dx[t, :] as given when dx_perm is
// null) + sum_e dL[t, e] Wg[e, :]; experts in steps of 32.
template <typename TIn>
__global__ void __launch_bounds__(256) route_bwd_dx_dense_kernel(
    int64_t T, int d, int E, int k, const float* __restrict__ dL, const TIn* __restrict__ Wg,
    const TIn* __restrict__ dx_perm, const int32_t* __restrict__ pos, TIn* __restrict__ dx) {
    __shared__ float dl_s[64][33];
    __shared__ __align__(16) float wg_s[32][128];
    const int tid = threadIdx.x, lane = tid & 31, ty = tid >> 5;
    const int64_t t0 = (int64_t)blockIdx.x * 64;
    const int c0 = blockIdx.y * 128;
    float acc[8][4];
    #pragma unroll
    for (int i = 0; i < 8; ++i)
        #pragma unroll
        for (int u = 0; u < 4; ++u) acc[i][u] = 0.f;
    for (int e0 = 0; e0 < E; e0 += 32) {
        for (int i = tid; i < 64 * 32; i += 256) {
            const int r = i >> 5, q = i & 31;
            const int64_t t = t0 + r;
            dl_s[r][q] = (t < T && e0 + q < E) ? dL[t * E + e0 + q] : 0.f;
        }
        for (int i = tid; i < 32 * 32; i += 256) {
            const int q = i >> 5, cc = (i & 31) * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e0 + q < E && c0 + cc < d) v = Four<TIn>::load(Wg + (int64_t)(e0 + q) * d + c0 + cc);
            *reinterpret_cast<float4*>(&wg_s[q][cc]) = v;
        }
        __syncthreads();
        #pragma unroll 8
        for (int q = 0; q < 32; ++q) {
            const float4 b = *reinterpret_cast<const float4*>(&wg_s[q][lane * 4]);
            #pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float a = dl_s[ty * 8 + i][q];
                acc[i][0] = fmaf(a, b.x, acc[i][0]);
                acc[i][1] = fmaf(a, b.y, acc[i][1]);
                acc[i][2] = fmaf(a, b.z, acc[i][2]);
                acc[i][3] = fmaf(a, b.w, acc[i][3]);
            }
        }
        __syncthreads();
    }
    const int c = c0 + lane * 4;
    if (c >= d) return;
    #pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t t = t0 + ty * 8 + i;
        if (t >= T) break;
        float4 base = make_float4(0.f, 0.f, 0.f, 0.f);
        if (dx_perm) {
            for (int j = 0; j < k; ++j) {
                const float4 v = Four<TIn>::load(dx_perm + (int64_t)pos[t * k + j] * d + c);
                base.x += v.x; base.y += v.y; base.z += v.z; base.w += v.w;
            }
        } else {
            base = Four<TIn>::load(dx + t * d + c);
        }
        base.x += acc[i][0]; base.y += acc[i][1]; base.z += acc[i][2]; base.w += acc[i][3];
        Four<TIn>::store(dx + t * d + c, base);
    }
}

constexpr int kDwgDenseTokens = 256;   // tokens per dWg partial

// partial[tc][e][c] = sum over the tokens t of chunk tc of dL[t, e] x[t, c];
// block tile 64 experts x 128 columns, tokens in steps of 32.
template <typename TIn>
__global__ void __launch_bounds__(256) dwg_dense_partial_kernel(
    int64_t T, int d, int E, const float* __restrict__ dL, const TIn* __restrict__ x,
    float* __restrict__ partial) {
    __shared__ float dl_s[32][65];
    __shared__ __align__(16) float x_s[32][128];
    const int tid = threadIdx.x, lane = tid & 31, ty = tid >> 5;
    const int64_t tbase = (int64_t)blockIdx.x * kDwgDenseTokens;
    const int c0 = blockIdx.y * 128, e0 = blockIdx.z * 64;
    float acc[8][4];
    #pragma unroll
    for (int i = 0; i < 8; ++i)
        #pragma unroll
        for (int u = 0; u < 4; ++u) acc[i][u] = 0.f;
    for (int ts = 0; ts < kDwgDenseTokens; ts += 32) {
        for (int i = tid; i < 32 * 64; i += 256) {
            const int r = i >> 6, q = i & 63;
            const int64_t t = tbase + ts + r;
            dl_s[r][q] = (t < T && e0 + q < E) ? dL[t * E + e0 + q] : 0.f;
        }
        for (int i = tid; i < 32 * 32; i += 256) {
            const int r = i >> 5, cc = (i & 31) * 4;
            const int64_t t = tbase + ts + r;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < T && c0 + cc < d) v = Four<TIn>::load(x + t * d + c0 + cc);
            *reinterpret_cast<float4*>(&x_s[r][cc]) = v;
        }
        __syncthreads();
        #pragma unroll 8
        for (int r = 0; r < 32; ++r) {
            const float4 b = *reinterpret_cast<const float4*>(&x_s[r][lane * 4]);
            #pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float a = dl_s[r][ty * 8 + i];
                acc[i][0] = fmaf(a, b.x, acc[i][0]);
                acc[i][1] = fmaf(a, b.y, acc[i][1]);
                acc[i][2] = fmaf(a, b.z, acc[i][2]);
                acc[i][3] = fmaf(a, b.w, acc[i][3]);
            }
        }
        __syncthreads();
    }
    const int c = c0 + lane * 4;
    if (c >= d) return;
    #pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = e0 + ty * 8 + i;
        if (e >= E) break;
        *reinterpret_cast<float4*>(partial + ((int64_t)blockIdx.x * E + e) * d + c) =
            make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
}

// dWg[e][c] (+)= sum over chunks of partial[tc][e][c]: a block takes one expert
// and 32 columns, its 8 warps every 8th chunk, added in warp order.
__global__ void __launch_bounds__(256) dwg_dense_reduce_kernel(int d, int E, int ntc,
                                                               const float* __restrict__ partial,
                                                               float* __restrict__ dWg,
                                                               int accumulate) {
    __shared__ float red[8][32];
    const int e = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.y * 32 + lane;
    float sum = 0.f;
    if (c < d)
        for (int i = warp; i < ntc; i += 8) sum += partial[((int64_t)i * E + e) * d + c];
    red[warp][lane] = sum;
    __syncthreads();
    if (warp == 0 && c < d) {
        float s = 0.f;
        #pragma unroll
        for (int w = 0; w < 8; ++w) s += red[w][lane];
        float* o = dWg + (int64_t)e * d + c;
        *o = accumulate ? *o + s : s;
    }
}

template <typename TIn>
cudaError_t route_bwd_typed(const moe_shape& s, const float* dw, const float* logits,
                            const int32_t* idx, const float* w, const int32_t* perm,
                            const int32_t* offsets, const TIn* x, const TIn* Wg,
                            const TIn* dx_perm, const int32_t* pos, TIn* dx, float* dWg,
                            int accumulate, float* dL, float* partial, cudaStream_t st) {
    const int64_t T = s.T;
    const int d = s.d, E = s.E, k = s.k;
    const unsigned gx = (unsigned)((T + 7) / 8);
    // KMAX: compile-time bound on k for the fused permute backward (1 when not fused)
    const int kb = (dx_perm == nullptr || !s.renorm)
                       ? 1 : (k <= 1 ? 1 : k <= 2 ? 2 : k <= 4 ? 4 : k <= 8 ? 8 : 16);
    // renorm off: dL is dense; dx's router term and dWg are tiled products
    const bool dense = !s.renorm;
#define MOE_RBWD(EPLV, KMV)                                                                    \
    route_bwd_dx_kernel<TIn, EPLV, KMV><<<gx, 256, 0, st>>>(T, d, E, k, s.renorm, dw, logits, \
                                                           idx, w, Wg, dense ? nullptr : dx_perm, \
                                                           pos, dx, dL, (int)dense)
#define MOE_RBWD_K(EPLV)                                                                       \
    switch (kb) {                                                                              \
        case 1: MOE_RBWD(EPLV, 1); break;                                                      \
        case 2: MOE_RBWD(EPLV, 2); break;                                                      \
        case 4: MOE_RBWD(EPLV, 4); break;                                                      \
        case 8: MOE_RBWD(EPLV, 8); break;                                                      \
        default: MOE_RBWD(EPLV, 16); break;                                                    \
    }
    if (E <= 32) { MOE_RBWD_K(1) }
    else if (E <= 64) { MOE_RBWD_K(2) }
    else if (E <= 128) { MOE_RBWD_K(4) }
    else { MOE_RBWD_K(8) }
#undef MOE_RBWD_K
#undef MOE_RBWD
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    if (s.renorm) {
        // dWg[e] = sum over e's selected slots of dL(slot) x[token(slot)]
        return launch_segment_rowsum(s, x, d, offsets, perm, dL, dWg, accumulate, partial, st);
    }
    const unsigned gc = (unsigned)((d + 127) / 128);
    route_bwd_dx_dense_kernel<TIn><<<dim3((unsigned)((T + 63) / 64), gc), 256, 0, st>>>(
        T, d, E, k, dL, Wg, dx_perm, pos, dx);
    const int ntc = (int)((T + kDwgDenseTokens - 1) / kDwgDenseTokens);
    dwg_dense_partial_kernel<TIn><<<dim3((unsigned)ntc, gc, (unsigned)((E + 63) / 64)), 256, 0,
                                    st>>>(T, d, E, dL, x, partial);
    dwg_dense_reduce_kernel<<<dim3((unsigned)E, (unsigned)((d + 31) / 32)), 256, 0, st>>>(
        d, E, ntc, partial, dWg, accumulate);
    return cudaGetLastError();
}

__global__ void bounded_wait_kernel(uint64_t limit_ns, int32_t* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);  // nothing ever arrives on it
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!mbar_wait_bounded(smem_u32(&bar), 0, limit_ns, &abort_flag))
            report(status, MOE_ERR_TIMEOUT);
    }
}

// GELU and its derivative, exact (CUDA erff / expf) or fast (the bf16
// epilogue's approximation), for checking the latter against its error bound.
__global__ void debug_gelu_kernel(int64_t n, const float* __restrict__ x, float* __restrict__ g,
                                  float* __restrict__ gd, int fast) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float v = x[i];
    g[i] = fast ? gelu_fast(v) : gelu_f(v);
    gd[i] = fast ? gelu_grad_fast(v) : gelu_grad_f(v);
}

}  // namespace

cudaError_t launch_debug_gelu(int64_t n, const float* x, float* g, float* gd, int fast,
                              cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    debug_gelu_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(n, x, g, gd, fast);
    return cudaGetLastError();
}

// ---- launchers -----------------------------------------------------------------------

// The router runs on CUDA cores (fp32 FMA): the tensor cores are kept for the
// expert GEMMs.  MOE_ROUTER_TENSOR_CORES=1 (read at every call) opts into
// computing bf16 logits as one more segment of the tcgen05 grouped GEMM with
// an fp32 epilogue (d % 64 == 0), which costs little more than the read of x.
static bool router_on_tensor_cores() {
    const char* v = getenv("MOE_ROUTER_TENSOR_CORES");
    return v && v[0] == '1';
}

size_t router_logits_workspace(const moe_shape& s) {
    if (s.E <= 32) return 0;   // the fused small-E kernel
    const int bn = s.E <= 64 ? 64 : 128;
    const int64_t tiles = ((s.T + kRtM - 1) / kRtM) * ((s.E + bn - 1) / bn);
    // at most (tiles / G + 2) pieces per block, G <= 4 blocks per SM
    return (size_t)(tiles + 8 * (int64_t)device_sm_count()) * kRtM * bn * sizeof(float);
}

cudaError_t launch_route_gate(const moe_shape& s, const void* x, const void* Wg,
                             const float* beta, float* logits, int compute_logits, int32_t* idx,
                             float* w, int32_t* block_counts, float* part, size_t part_bytes,
                             int32_t* status, cudaStream_t st) {
    const bool bf = s.dtype == MOE_BF16;
    if (compute_logits && bf && s.d % 64 == 0 && router_on_tensor_cores()) {
        // bf16 logits on the tensor cores (fp32 accumulation), then the gate
        GemmVarM g{1, s.E, s.d, s.T, nullptr, x, Wg, true, Epi::Logits, beta, nullptr, logits,
                   nullptr};
        const cudaError_t e = launch_gemm_varm_tc(g, status, st);
        if (e != cudaSuccess) return e;
        compute_logits = 0;
    }
    if (compute_logits && s.E <= 32) {
        if (bf)
            return router_gate_small(s, (const __nv_bfloat16*)x, (const __nv_bfloat16*)Wg, beta,
                                     logits, idx, w, block_counts, status, st);
        return router_gate_small(s, (const float*)x, (const float*)Wg, beta, logits, idx, w,
                                 block_counts, status, st);
    }
    if (compute_logits) {
        cudaError_t e = bf ? router_logits_dispatch(s, (const __nv_bfloat16*)x,
                                                    (const __nv_bfloat16*)Wg, beta, logits, part,
                                                    part_bytes, st)
                           : router_logits_dispatch(s, (const float*)x, (const float*)Wg, beta,
                                                    logits, part, part_bytes, st);
        if (e != cudaSuccess) return e;
    }
    const int nblk = (int)route_blocks(s.T);
    const int E = s.E;
#define MOE_GATE(EPLV, WV)                                                                  \
    gate_hist_kernel<EPLV, WV><<<nblk, (WV) * 32, 0, st>>>(s.T, E, s.k, s.renorm, nblk, logits, \
                                                           idx, w, block_counts, status)
    if (E <= 32) MOE_GATE(1, 32);
    else if (E <= 64) MOE_GATE(2, 32);
    else if (E <= 128) MOE_GATE(4, 16);
    else MOE_GATE(8, 16);
#undef MOE_GATE
    return cudaGetLastError();
}

cudaError_t launch_dispatch_scan(const moe_shape& s, int32_t* block_counts, int32_t* counts,
                                 int32_t* offsets, cudaStream_t st) {
    dispatch_scan_kernel<<<1, 1024, 0, st>>>(s.E, (int)route_blocks(s.T), block_counts, counts,
                                             offsets);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_rank(const moe_shape& s, const int32_t* idx,
                                 const int32_t* block_base, int32_t* pos, int32_t* perm,
                                 cudaStream_t st) {
    const int nblk = (int)route_blocks(s.T);
    dispatch_rank_kernel<<<nblk, kRouteBlockTokens, 0, st>>>(s.T, s.E, s.k, nblk, idx, block_base, pos, perm);
    return cudaGetLastError();
}

size_t route_bwd_workspace(const moe_shape& s) {
    const int64_t T = s.T;
    const size_t dl = (size_t)T * (size_t)(s.renorm ? s.k : s.E) * sizeof(float);
    size_t part;
    if (s.renorm)
        part = (size_t)((T * s.k + kDwgChunk - 1) / kDwgChunk + s.E) * s.d * sizeof(float);
    else
        part = (size_t)((T + kDwgChunk - 1) / kDwgChunk) * s.E * s.d * sizeof(float);
    return ((dl + 255) & ~(size_t)255) + part;
}

cudaError_t launch_route_bwd(const moe_shape& s, const float* dw, const float* logits,
                             const int32_t* idx, const float* w, const int32_t* perm,
                             const int32_t* offsets, const void* x, const void* Wg,
                             const void* dx_perm, const int32_t* pos, void* dx, float* dWg,
                             int accumulate, float* dL, float* partial, cudaStream_t st) {
    if (s.dtype == MOE_BF16)
        return route_bwd_typed(s, dw, logits, idx, w, perm, offsets, (const __nv_bfloat16*)x,
                               (const __nv_bfloat16*)Wg, (const __nv_bfloat16*)dx_perm, pos,
                               (__nv_bfloat16*)dx, dWg, accumulate, dL, partial, st);
    return route_bwd_typed(s, dw, logits, idx, w, perm, offsets, (const float*)x,
                           (const float*)Wg, (const float*)dx_perm, pos, (float*)dx, dWg,
                           accumulate, dL, partial, st);
}

cudaError_t launch_bounded_wait(uint64_t limit_ns, int32_t* status, cudaStream_t st) {
    bounded_wait_kernel<<<1, 32, 0, st>>>(limit_ns, status);
    return cudaGetLastError();
}

}  // namespace moe
