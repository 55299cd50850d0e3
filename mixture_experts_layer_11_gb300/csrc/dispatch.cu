// dispatch.cu -- permute (scatter into expert-sorted rows), weighted combine
// back to token order, their backward, and per-expert column sums (bias
// gradients).  Steps A4, A6, A7, A9 of the layer and the bias part of A8.
//
// The expert-sorted layout is FastMoE's scatter/gather-by-expert layout
// ("FastMoE: A Fast Mixture-of-Expert Training System", review, "proposed
// method"); the permutation stage precedes the per-expert processing in
// ES-MoE (review, section 3 "expert-wise offloading and processing").
//
// All of these are bandwidth-bound row copies / reductions: one warp per
// token row, 16-byte vector accesses, every row read or written once.  The
// combine is a gather (no atomics), so results are deterministic.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

template <typename T> struct V16;  // 16 bytes of T as fp32 lanes
template <> struct V16<__nv_bfloat16> {
    static constexpr int N = 8;
    static __device__ __forceinline__ void unpack(const uint4& u, float* v) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
        #pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ uint4 pack(const float* v) {
        uint4 u;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
        #pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        return u;
    }
};
template <> struct V16<float> {
    static constexpr int N = 4;
    static __device__ __forceinline__ void unpack(const uint4& u, float* v) {
        v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
        v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
    }
    static __device__ __forceinline__ uint4 pack(const float* v) {
        return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                          __float_as_uint(v[3]));
    }
};

__device__ __forceinline__ uint4 ldg16(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void stg16(void* p, const uint4& v) {
    *reinterpret_cast<uint4*>(p) = v;
}

inline unsigned grid_for_rows(int64_t rows) {
    // 8 warps per block, one row per warp per iteration; enough blocks to
    // fill every SM several times over, grid-striding beyond that.
    const int64_t want = (rows + 7) / 8;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    return (unsigned)(want < cap ? (want > 0 ? want : 1) : cap);
}

// Vectors per lane kept in flight: U * KMAX 16-byte loads before any use.
template <int KMAX> struct Unroll { static constexpr int U = KMAX >= 8 ? 1 : 8 / KMAX; };

// ---- A4: X_perm[pos[t,j]] = x[t] ------------------------------------------------
// nv = row length in 16-byte vectors.  One warp per token row: read once,
// written to its k positions.
template <int KMAX>
__global__ void __launch_bounds__(256) permute_kernel(int64_t T, int nv, int k,
                                                      const uint4* __restrict__ x,
                                                      const int32_t* __restrict__ pos,
                                                      uint4* __restrict__ xp) {
    constexpr int U = KMAX >= 8 ? 2 : 4;
    const int lane = threadIdx.x & 31;
    const int64_t wstride = (int64_t)gridDim.x * 8;
    for (int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); t < T; t += wstride) {
        int32_t p[KMAX];
        #pragma unroll
        for (int j = 0; j < KMAX; ++j) p[j] = (j < k) ? __ldg(pos + t * k + j) : 0;
        const uint4* src = x + t * nv;
        for (int c0 = lane; c0 < nv; c0 += 32 * U) {
            uint4 v[U];
            #pragma unroll
            for (int u = 0; u < U; ++u)
                if (c0 + 32 * u < nv) v[u] = ldg16(src + c0 + 32 * u);
            #pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (j >= k) break;
                uint4* dst = xp + (int64_t)p[j] * nv + c0;
                #pragma unroll
                for (int u = 0; u < U; ++u)
                    if (c0 + 32 * u < nv) dst[32 * u] = v[u];
            }
        }
    }
}

// ---- A6 / A9: y[t] = sum_j w[t,j] Y[pos[t,j]] (w == null: weights 1) -------------
template <typename T, int KMAX>
__global__ void __launch_bounds__(256) combine_kernel(int64_t Tn, int nv, int k,
                                                      const uint4* __restrict__ Y,
                                                      const int32_t* __restrict__ pos,
                                                      const float* __restrict__ w,
                                                      uint4* __restrict__ y) {
    using V = V16<T>;
    constexpr int U = Unroll<KMAX>::U;
    const int lane = threadIdx.x & 31;
    const int64_t wstride = (int64_t)gridDim.x * 8;
    for (int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); t < Tn; t += wstride) {
        int32_t p[KMAX];
        float wj[KMAX];
        #pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            p[j] = (j < k) ? __ldg(pos + t * k + j) : 0;
            wj[j] = (j < k) ? (w ? __ldg(w + t * k + j) : 1.f) : 0.f;
        }
        for (int c0 = lane; c0 < nv; c0 += 32 * U) {
            uint4 r[U][KMAX];
            #pragma unroll
            for (int u = 0; u < U; ++u)
                #pragma unroll
                for (int j = 0; j < KMAX; ++j)
                    if (j < k && c0 + 32 * u < nv) r[u][j] = ldg16(Y + (int64_t)p[j] * nv + c0 + 32 * u);
            #pragma unroll
            for (int u = 0; u < U; ++u) {
                if (c0 + 32 * u >= nv) break;
                float acc[V::N], v[V::N];
                #pragma unroll
                for (int e = 0; e < V::N; ++e) acc[e] = 0.f;
                #pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    if (j >= k) break;
                    V::unpack(r[u][j], v);
                    #pragma unroll
                    for (int e = 0; e < V::N; ++e) acc[e] = fmaf(wj[j], v[e], acc[e]);
                }
                stg16(y + t * nv + c0 + 32 * u, V::pack(acc));
            }
        }
    }
}

// ---- A7: dY[pos[t,j]] = w[t,j] dy[t];  dw[t,j] = <dy[t], Y[pos[t,j]]> -------------
template <typename T, int KMAX>
__global__ void __launch_bounds__(256) combine_bwd_kernel(int64_t Tn, int nv, int k,
                                                          const uint4* __restrict__ dy,
                                                          const uint4* __restrict__ Y,
                                                          const int32_t* __restrict__ pos,
                                                          const float* __restrict__ w,
                                                          uint4* __restrict__ dY,
                                                          float* __restrict__ dw) {
    using V = V16<T>;
    constexpr int U = Unroll<KMAX>::U;
    const int lane = threadIdx.x & 31;
    const int64_t wstride = (int64_t)gridDim.x * 8;
    for (int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); t < Tn; t += wstride) {
        int32_t p[KMAX];
        float wj[KMAX], part[KMAX];
        #pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            p[j] = (j < k) ? __ldg(pos + t * k + j) : 0;
            wj[j] = (j < k) ? __ldg(w + t * k + j) : 0.f;
            part[j] = 0.f;
        }
        for (int c0 = lane; c0 < nv; c0 += 32 * U) {
            uint4 gr[U], r[U][KMAX];
            #pragma unroll
            for (int u = 0; u < U; ++u) {
                if (c0 + 32 * u < nv) gr[u] = ldg16(dy + t * nv + c0 + 32 * u);
                #pragma unroll
                for (int j = 0; j < KMAX; ++j)
                    if (j < k && c0 + 32 * u < nv) r[u][j] = ldg16(Y + (int64_t)p[j] * nv + c0 + 32 * u);
            }
            #pragma unroll
            for (int u = 0; u < U; ++u) {
                if (c0 + 32 * u >= nv) break;
                float g[V::N], v[V::N], o[V::N];
                V::unpack(gr[u], g);
                #pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    if (j >= k) break;
                    V::unpack(r[u][j], v);
                    #pragma unroll
                    for (int e = 0; e < V::N; ++e) {
                        part[j] = fmaf(g[e], v[e], part[j]);
                        o[e] = wj[j] * g[e];
                    }
                    stg16(dY + (int64_t)p[j] * nv + c0 + 32 * u, V::pack(o));
                }
            }
        }
        #pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (j >= k) break;
            float s = part[j];
            #pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
            if (lane == 0) dw[t * k + j] = s;
        }
    }
}

// ---- per-expert weighted row sums over segments ------------------------------------
// out[e][c] (+)= sum over the rows p of expert e's segment of wgt(p) * src[row(p)][c]:
// wgt = 1, row = p for the column sums of a permuted matrix (bias gradients);
// with perm given, slot s = perm[p], wgt = wsel[s], row = s / k (the router
// weight gradient of the selected experts, summed over their tokens).
// Phase 1: one partial per (expert, run of segment rows) and column tile; the
// block walks its rows kDwgChunk at a time, its 8 warps taking every 8th row,
// lanes consecutive 16-byte column vectors, and the warps' sums are added in
// warp order through shared memory.  A run is either a chunk of kDwgChunk rows
// (blocks in expert order), or, when the rows are gathered from a source larger
// than kSegPieceMinBytes, piece q of `pieces` equal pieces of the segment, with
// the blocks in piece-major order: pieces x E partials instead of one per
// kDwgChunk rows (a quarter of the partial bytes on a 32768-token, top-8 chunk
// of 128 experts), and, as a segment lists its slots in token order, the blocks
// that run together read the rows of one window of tokens for every expert, so
// a token's row, read once per selected expert, mostly comes from L2.  Phase 2:
// per expert and 32 or 128 columns (1 or 4 per lane), 8 warps take every 8th
// partial, added in warp order.  Deterministic.
constexpr int kSegCPL = 4;   // 16-byte vectors per lane in a column tile
constexpr int kSegPieces = 16;
constexpr int64_t kSegPieceMinBytes = 64ll << 20;

template <typename T>
__global__ void __launch_bounds__(256) seg_partial_kernel(int n, int E, int k, int pieces,
                                                          const int32_t* __restrict__ offsets,
                                                          const int32_t* __restrict__ perm,
                                                          const float* __restrict__ wsel,
                                                          const T* __restrict__ src,
                                                          float* __restrict__ partial) {
    using V = V16<T>;
    constexpr int TILE = 32 * kSegCPL * V::N;      // columns of one tile
    __shared__ __align__(16) float red[8][TILE];
    __shared__ int off_s[257];
    // the segment bounds, loaded in one step (not a chain of dependent loads)
    for (int i = threadIdx.x; i <= E; i += 256) off_s[i] = offsets[i];
    __syncthreads();
    int p0, p1;   // the block's rows
    if (pieces > 0) {
        // block x = q * E + e: piece q of expert e's segment (empty pieces
        // still write their zero partial, which phase 2 adds)
        const int e = blockIdx.x % E, q = blockIdx.x / E;
        const int cnt = off_s[e + 1] - off_s[e];
        const int len = (cnt + pieces - 1) / pieces;
        p0 = off_s[e] + min(cnt, q * len);
        p1 = off_s[e] + min(cnt, (q + 1) * len);
    } else {
        int e = 0, acc = 0, sub = -1;
        for (; e < E; ++e) {
            const int cnt = off_s[e + 1] - off_s[e];
            const int nc = (cnt + kDwgChunk - 1) / kDwgChunk;
            if ((int)blockIdx.x < acc + nc) { sub = blockIdx.x - acc; break; }
            acc += nc;
        }
        if (sub < 0) return;   // block-uniform
        p0 = off_s[e] + sub * kDwgChunk;
        p1 = min(off_s[e + 1], p0 + kDwgChunk);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ct0 = blockIdx.y * TILE;
    float a[kSegCPL][V::N];
    #pragma unroll
    for (int i = 0; i < kSegCPL; ++i)
        #pragma unroll
        for (int u = 0; u < V::N; ++u) a[i][u] = 0.f;
    constexpr int RPW = kDwgChunk / 8;   // rows per warp and step
    static_assert(RPW <= 32, "one lane per row");
    for (int pb = p0; pb < p1; pb += kDwgChunk) {
        const int pe = min(p1, pb + kDwgChunk);
        // The warp's rows pb + warp + 8 j (j < RPW): their slot, weight and
        // source row are fetched by lane j in one step, then every row's
        // vectors are requested before the first is used.
        int my_row = 0;
        float my_g = 1.f;
        {
            const int r = pb + warp + 8 * lane;
            if (lane < RPW && r < pe) {
                my_row = r;
                if (perm) {
                    const int sl = __ldg(perm + r);
                    my_g = __ldg(wsel + sl);
                    my_row = sl / k;
                }
            }
        }
        uint4 raw[RPW][kSegCPL];
        #pragma unroll
        for (int j = 0; j < RPW; ++j) {
            const int64_t row = __shfl_sync(0xffffffffu, my_row, j);
            const bool in = pb + warp + 8 * j < pe;
            #pragma unroll
            for (int i = 0; i < kSegCPL; ++i) {
                const int c = ct0 + (lane + 32 * i) * V::N;
                raw[j][i] = (in && c < n) ? ldg16(src + row * n + c) : make_uint4(0, 0, 0, 0);
            }
        }
        #pragma unroll
        for (int j = 0; j < RPW; ++j) {
            const float g = __shfl_sync(0xffffffffu, my_g, j);
            if (pb + warp + 8 * j >= pe) break;   // warp-uniform
            #pragma unroll
            for (int i = 0; i < kSegCPL; ++i) {
                float v[V::N];
                V::unpack(raw[j][i], v);
                #pragma unroll
                for (int u = 0; u < V::N; ++u) a[i][u] = fmaf(g, v[u], a[i][u]);
            }
        }
    }
    #pragma unroll
    for (int i = 0; i < kSegCPL; ++i)
        #pragma unroll
        for (int u = 0; u < V::N; u += 4)
            *reinterpret_cast<float4*>(&red[warp][(lane + 32 * i) * V::N + u]) =
                make_float4(a[i][u], a[i][u + 1], a[i][u + 2], a[i][u + 3]);
    __syncthreads();
    for (int j = threadIdx.x; j < TILE; j += 256) {
        const int c = ct0 + j;
        if (c >= n) break;
        float sum = 0.f;
        #pragma unroll
        for (int w = 0; w < 8; ++w) sum += red[w][j];
        partial[(int64_t)blockIdx.x * n + c] = sum;
    }
}

// VL consecutive columns per lane (1, or 4 when n % 4 == 0), 32 * VL per block
template <int VL>
__global__ void __launch_bounds__(256) seg_reduce_kernel(int n, int E, int pieces,
                                                         const int32_t* __restrict__ offsets,
                                                         const float* __restrict__ partial,
                                                         float* __restrict__ out, int accumulate) {
    __shared__ float red[8][32 * VL];
    __shared__ int off_s[257];
    const int e = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = (blockIdx.y * 32 + lane) * VL;
    for (int i = threadIdx.x; i <= e + 1; i += 256) off_s[i] = offsets[i];
    __syncthreads();
    // expert e's partials: start, start + stride, ... (nc of them)
    int start = 0, nc, stride = 1;
    if (pieces > 0) {
        start = e;
        nc = pieces;
        stride = E;
    } else {
        for (int q = 0; q < e; ++q) {
            const int cnt = off_s[q + 1] - off_s[q];
            start += (cnt + kDwgChunk - 1) / kDwgChunk;
        }
        const int cnt = off_s[e + 1] - off_s[e];
        nc = (cnt + kDwgChunk - 1) / kDwgChunk;
    }
    float sum[VL];
    #pragma unroll
    for (int x = 0; x < VL; ++x) sum[x] = 0.f;
    if (c < n) {
        // the warp's partials warp, warp + 8, ...: UN loads in flight, added in order
        constexpr int UN = VL == 1 ? 16 : 8;
        for (int i0 = warp; i0 < nc; i0 += 8 * UN) {
            float v[UN][VL];
            #pragma unroll
            for (int u = 0; u < UN; ++u) {
                const int i = i0 + 8 * u;
                const float* src = partial + ((int64_t)start + (int64_t)i * stride) * n + c;
                if (VL == 4) {
                    const float4 f = i < nc ? *reinterpret_cast<const float4*>(src)
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
                    v[u][0] = f.x; v[u][1 % VL] = f.y; v[u][2 % VL] = f.z; v[u][3 % VL] = f.w;
                } else {
                    v[u][0] = i < nc ? *src : 0.f;
                }
            }
            #pragma unroll
            for (int u = 0; u < UN; ++u)   // past the end: + 0
                #pragma unroll
                for (int x = 0; x < VL; ++x) sum[x] += v[u][x];
        }
    }
    #pragma unroll
    for (int x = 0; x < VL; ++x) red[warp][lane * VL + x] = sum[x];
    __syncthreads();
    if (warp == 0 && c < n) {
        #pragma unroll
        for (int x = 0; x < VL; ++x) {
            float t = 0.f;
            #pragma unroll
            for (int w = 0; w < 8; ++w) t += red[w][lane * VL + x];
            float* o = out + (int64_t)e * n + c + x;
            *o = accumulate ? *o + t : t;
        }
    }
}

template <template <int> class F, typename... Args>
cudaError_t by_k(int k, Args... args) {
    if (k <= 1) return F<1>::run(args...);
    if (k <= 2) return F<2>::run(args...);
    if (k <= 4) return F<4>::run(args...);
    if (k <= 8) return F<8>::run(args...);
    return F<16>::run(args...);
}

template <int KM> struct PermuteL {
    static cudaError_t run(const moe_shape& s, const void* x, const int32_t* pos, void* xp,
                           cudaStream_t st) {
        const int esz = s.dtype == MOE_BF16 ? 2 : 4;
        permute_kernel<KM><<<grid_for_rows(s.T), 256, 0, st>>>(s.T, s.d * esz / 16, s.k,
                                                               (const uint4*)x, pos, (uint4*)xp);
        return cudaGetLastError();
    }
};
template <int KM> struct CombineL {
    static cudaError_t run(const moe_shape& s, const void* Y, const int32_t* pos, const float* w,
                           void* y, cudaStream_t st) {
        const unsigned g = grid_for_rows(s.T);
        if (s.dtype == MOE_BF16)
            combine_kernel<__nv_bfloat16, KM><<<g, 256, 0, st>>>(s.T, s.d / 8, s.k, (const uint4*)Y,
                                                                 pos, w, (uint4*)y);
        else
            combine_kernel<float, KM><<<g, 256, 0, st>>>(s.T, s.d / 4, s.k, (const uint4*)Y, pos,
                                                         w, (uint4*)y);
        return cudaGetLastError();
    }
};
template <int KM> struct CombineBwdL {
    static cudaError_t run(const moe_shape& s, const void* dy, const void* Y, const int32_t* pos,
                           const float* w, void* dY, float* dw, cudaStream_t st) {
        const unsigned g = grid_for_rows(s.T);
        if (s.dtype == MOE_BF16)
            combine_bwd_kernel<__nv_bfloat16, KM><<<g, 256, 0, st>>>(
                s.T, s.d / 8, s.k, (const uint4*)dy, (const uint4*)Y, pos, w, (uint4*)dY, dw);
        else
            combine_bwd_kernel<float, KM><<<g, 256, 0, st>>>(
                s.T, s.d / 4, s.k, (const uint4*)dy, (const uint4*)Y, pos, w, (uint4*)dY, dw);
        return cudaGetLastError();
    }
};

}  // namespace

cudaError_t launch_permute(const moe_shape& s, const void* x, const int32_t* pos, void* x_perm,
                           cudaStream_t st) {
    return by_k<PermuteL>(s.k, s, x, pos, x_perm, st);
}

cudaError_t launch_combine(const moe_shape& s, const void* y_perm, const int32_t* pos,
                           const float* w, void* y, cudaStream_t st) {
    return by_k<CombineL>(s.k, s, y_perm, pos, w, y, st);
}

cudaError_t launch_combine_bwd(const moe_shape& s, const void* dy, const void* y_perm,
                               const int32_t* pos, const float* w, void* dy_perm, float* dw,
                               cudaStream_t st) {
    return by_k<CombineBwdL>(s.k, s, dy, y_perm, pos, w, dy_perm, dw, st);
}

size_t segment_colsum_workspace(const moe_shape& s, int n) {
    return (size_t)((s.T * s.k + kDwgChunk - 1) / kDwgChunk + s.E) * (size_t)n * sizeof(float);
}

cudaError_t launch_segment_rowsum(const moe_shape& s, const void* src, int n,
                                  const int32_t* offsets, const int32_t* perm,
                                  const float* wsel, float* out, int accumulate, float* partial,
                                  cudaStream_t st) {
    const int64_t nchunks = (s.T * s.k + kDwgChunk - 1) / kDwgChunk + s.E;
    const int esz = s.dtype == MOE_BF16 ? 2 : 4;
    const int tile = 32 * kSegCPL * (16 / esz);
    // pieces: rows gathered from a source well beyond what L2 keeps; no more
    // partials than the chunked runs' (the workspace holds nchunks of them)
    int pieces = 0;
    if (perm != nullptr && (int64_t)s.T * n * esz >= kSegPieceMinBytes)
        pieces = (int)std::min<int64_t>(kSegPieces, nchunks / s.E);
    const dim3 grid((unsigned)(pieces > 0 ? (int64_t)pieces * s.E : nchunks),
                    (unsigned)((n + tile - 1) / tile));
    if (s.dtype == MOE_BF16)
        seg_partial_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
            n, s.E, s.k, pieces, offsets, perm, wsel, (const __nv_bfloat16*)src, partial);
    else
        seg_partial_kernel<float><<<grid, 256, 0, st>>>(n, s.E, s.k, pieces, offsets, perm, wsel,
                                                        (const float*)src, partial);
    // 4 columns per lane when that still leaves two blocks per SM (wide
    // outputs, many experts), else 1 (more blocks for small problems)
    if (n % 4 == 0 && (int64_t)s.E * ((n + 127) / 128) >= 2 * (int64_t)device_sm_count())
        seg_reduce_kernel<4><<<dim3(s.E, (unsigned)((n + 127) / 128)), 256, 0, st>>>(
            n, s.E, pieces, offsets, partial, out, accumulate);
    else
        seg_reduce_kernel<1><<<dim3(s.E, (unsigned)((n + 31) / 32)), 256, 0, st>>>(
            n, s.E, pieces, offsets, partial, out, accumulate);
    return cudaGetLastError();
}

cudaError_t launch_segment_colsum(const moe_shape& s, const void* g, int n,
                                  const int32_t* offsets, float* out, int accumulate,
                                  float* partial, cudaStream_t st) {
    return launch_segment_rowsum(s, g, n, offsets, nullptr, nullptr, out, accumulate, partial,
                                 st);
}

}  // namespace moe
