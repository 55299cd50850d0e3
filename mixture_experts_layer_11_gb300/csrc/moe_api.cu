// moe_api.cu -- the C ABI of include/moe.h: argument validation, workspace
// carving, and the launch sequence of each step on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include <mutex>

#include "../../include/moe.h"
#include "kernels.h"

namespace moe {

uint64_t wait_limit_ns() {
    static uint64_t v = [] {
        const char* s = getenv("MOE_WAIT_TIMEOUT_NS");
        if (s && *s) {
            const unsigned long long x = strtoull(s, nullptr, 10);
            if (x > 0) return (uint64_t)x;
        }
        return (uint64_t)1000000000ull;  // 1 s
    }();
    return v;
}

int device_sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 132;
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 132;
    }
    return cache[dev];
}

}  // namespace moe

using namespace moe;

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }
inline bool ok_opt(const void* p) { return p == nullptr || aligned16(p); }
// the status word is one int32: 4-byte alignment suffices
inline bool ok_status(const int32_t* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

inline size_t esize(const moe_shape& s) { return s.dtype == MOE_BF16 ? 2 : 4; }

moe_status check_shape(const moe_shape* s) {
    if (!s) return MOE_ERR_INVALID;
    if (s->T < 0 || s->d <= 0 || s->f <= 0 || s->E < 1 || s->E > 256 || s->k < 1 ||
        s->k > 16 || s->k > s->E)
        return MOE_ERR_INVALID;
    if (s->dtype != MOE_F32 && s->dtype != MOE_BF16) return MOE_ERR_INVALID;
    if (s->renorm != 0 && s->renorm != 1) return MOE_ERR_INVALID;
    if (s->T * (int64_t)s->k >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if (s->d % 8 || s->f % 8) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

moe_status check_gemm_shape(const moe_shape* s) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (s->dtype == MOE_BF16 && (s->d % 64 || s->f % 64)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

inline moe_status cuda_status(cudaError_t e) {
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// block histograms, then the router logits' split tiles
size_t route_counts_ws(const moe_shape& s) {
    return align_up((size_t)s.E * (size_t)route_blocks(s.T) * sizeof(int32_t));
}
size_t route_ws(const moe_shape& s) {
    return route_counts_ws(s) + align_up(router_logits_workspace(s));
}

// column-sum partial rows of the bias gradients (either path)
size_t ffn_partial_bytes(const moe_shape& s) {
    const int n = s.d > s.f ? s.d : s.f;
    size_t part = segment_colsum_workspace(s, n);
    const size_t fused = gemm_colsum_workspace(s.T * s.k, s.E, s.f);   // db1 in the dH GEMM
    return align_up(fused > part ? fused : part);
}

// scratch of the split weight-gradient reductions over `rows` rows (bf16)
size_t split_bytes(const moe_shape& s, int64_t rows) {
    if (s.dtype != MOE_BF16) return 0;
    const size_t a = vark_split_workspace(rows, s.E, s.d, s.f);
    const size_t b = vark_split_workspace(rows, s.E, s.f, s.d);
    return align_up(a > b ? a : b);
}

size_t ffn_bwd_ws(const moe_shape& s) {
    const size_t dh = align_up((size_t)s.T * s.k * s.f * esize(s));
    return dh + ffn_partial_bytes(s) + split_bytes(s, s.T * s.k);
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID: return "MOE_ERR_INVALID: bad argument";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: unsupported shape or dtype";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: CUDA call or launch failed";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a bounded device wait ran out";
        case MOE_ERR_NONFINITE: return "MOE_ERR_NONFINITE: non-finite router logit";
    }
    return "unknown moe_status";
}

size_t moe_workspace_size(const moe_shape* s) {
    if (check_shape(s) != MOE_OK) return 0;
    size_t m = route_ws(*s);
    const size_t b = ffn_bwd_ws(*s);
    if (b > m) m = b;
    const size_t r = align_up(route_bwd_workspace(*s));
    if (r > m) m = r;
    return m;
}

moe_status moe_route(const moe_shape* s, const void* x, const void* Wg, const float* logit_bias,
                     float* logits, int compute_logits, int32_t* idx, float* w, int32_t* counts,
                     int32_t* offsets, int32_t* pos, int32_t* perm, void* ws,
                     int32_t* dev_status, moe_stream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (!ok_ptr(counts) || !ok_ptr(offsets)) return MOE_ERR_INVALID;
    if (s->T > 0) {
        if (!ok_ptr(logits) || !ok_ptr(idx) || !ok_ptr(w) || !ok_ptr(pos) || !ok_ptr(perm) ||
            !ok_ptr(ws) || !ok_status(dev_status))
            return MOE_ERR_INVALID;
        if (compute_logits && (!ok_ptr(x) || !ok_ptr(Wg) || !ok_opt(logit_bias)))
            return MOE_ERR_INVALID;
    }
    cudaStream_t st = (cudaStream_t)stream;
    int32_t* block_counts = (int32_t*)ws;
    float* part = (float*)((uint8_t*)ws + route_counts_ws(*s));
    cudaError_t e = cudaSuccess;
    if (s->T > 0)
        e = launch_route_gate(*s, x, Wg, logit_bias, logits, compute_logits, idx, w, block_counts,
                              part, router_logits_workspace(*s), dev_status, st);
    if (e == cudaSuccess) e = launch_dispatch_scan(*s, block_counts, counts, offsets, st);
    if (e == cudaSuccess && s->T > 0) e = launch_dispatch_rank(*s, idx, block_counts, pos, perm, st);
    return cuda_status(e);
}

moe_status moe_permute(const moe_shape* s, const void* x, const int32_t* pos, void* x_perm,
                       moe_stream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (s->T == 0) return MOE_OK;
    if (!ok_ptr(x) || !ok_ptr(pos) || !ok_ptr(x_perm)) return MOE_ERR_INVALID;
    return cuda_status(launch_permute(*s, x, pos, x_perm, (cudaStream_t)stream));
}

}  // extern "C"

namespace {

// A5 (perm == nullptr: act is X_perm) or A4 + A5 with the permute fused into
// the first GEMM's loads (act is x, row r of X_perm read as x[perm[r] / k]).
moe_status ffn_fwd(const moe_shape* s, const void* act, const int32_t* perm,
                   const int32_t* offsets, const void* W1, const void* b1, const void* W2,
                   const void* b2, void* G, void* A, void* y_perm, int32_t* dev_status,
                   moe_stream_t stream) {
    moe_status r = check_gemm_shape(s);
    if (r != MOE_OK) return r;
    if (s->T == 0) return MOE_OK;
    if (!ok_ptr(act) || !ok_ptr(offsets) || !ok_ptr(W1) || !ok_ptr(W2) || !ok_opt(b1) ||
        !ok_opt(b2) || !ok_ptr(G) || !ok_ptr(A) || !ok_ptr(y_perm) || !ok_status(dev_status) ||
        !ok_opt(perm))
        return MOE_ERR_INVALID;
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t P = s->T * s->k;
    GemmVarM g1{s->E, s->f, s->d, P, offsets, act, W1, true, Epi::BiasGelu, b1, nullptr, G, A};
    GemmVarM g2{s->E, s->d, s->f, P, offsets, A, W2, true, Epi::Bias, b2, nullptr, y_perm, nullptr};
    if (perm) {
        g1.gather = perm;
        g1.gather_k = s->k;
        g1.gather_rows = s->T;
    }
    cudaError_t e;
    if (s->dtype == MOE_BF16) {
        e = launch_gemm_varm_tc(g1, dev_status, st);
        if (e == cudaSuccess) e = launch_gemm_varm_tc(g2, dev_status, st);
    } else {
        e = launch_gemm_varm_simt(g1, st);
        if (e == cudaSuccess) e = launch_gemm_varm_simt(g2, st);
    }
    return cuda_status(e);
}

}  // namespace

extern "C" {

moe_status moe_expert_ffn_fwd(const moe_shape* s, const void* x_perm, const int32_t* offsets,
                              const void* W1, const void* b1, const void* W2, const void* b2,
                              void* G, void* A, void* y_perm, void* ws, int32_t* dev_status,
                              moe_stream_t stream) {
    (void)ws;
    return ffn_fwd(s, x_perm, nullptr, offsets, W1, b1, W2, b2, G, A, y_perm, dev_status, stream);
}

moe_status moe_expert_ffn_fwd_gather(const moe_shape* s, const void* x, const int32_t* perm,
                                     const int32_t* offsets, const void* W1, const void* b1,
                                     const void* W2, const void* b2, void* G, void* A,
                                     void* y_perm, void* ws, int32_t* dev_status,
                                     moe_stream_t stream) {
    (void)ws;
    if (s && s->T > 0 && !ok_ptr(perm)) return MOE_ERR_INVALID;
    return ffn_fwd(s, x, perm, offsets, W1, b1, W2, b2, G, A, y_perm, dev_status, stream);
}

moe_status moe_combine_fwd(const moe_shape* s, const void* y_perm, const int32_t* pos,
                           const float* w, void* y, moe_stream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (s->T == 0) return MOE_OK;
    if (!ok_ptr(y_perm) || !ok_ptr(pos) || !ok_opt(w) || !ok_ptr(y)) return MOE_ERR_INVALID;
    return cuda_status(launch_combine(*s, y_perm, pos, w, y, (cudaStream_t)stream));
}

moe_status moe_combine_bwd(const moe_shape* s, const void* dy, const void* y_perm,
                           const int32_t* pos, const float* w, void* dy_perm, float* dw,
                           moe_stream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (s->T == 0) return MOE_OK;
    if (!ok_ptr(dy) || !ok_ptr(y_perm) || !ok_ptr(pos) || !ok_ptr(w) || !ok_ptr(dy_perm) ||
        !ok_ptr(dw))
        return MOE_ERR_INVALID;
    return cuda_status(launch_combine_bwd(*s, dy, y_perm, pos, w, dy_perm, dw,
                                          (cudaStream_t)stream));
}

}  // extern "C"

namespace {

// A8, data half: dH = (dY W2[e]) * G, db1 (+)= sum_rows dH, dX = dH W1[e].
// `partial` holds the column-sum partial rows (ffn_partial_bytes).
cudaError_t ffn_bwd_data(const moe_shape& s, const void* dy_perm, const void* G,
                         const int32_t* offsets, const void* W1, const void* W2, void* dH,
                         void* dx_perm, float* db1, int accumulate, float* partial,
                         int32_t* status, cudaStream_t st) {
    const int E = s.E, d = s.d, f = s.f;
    const int64_t P = s.T * s.k;
    const bool tc = s.dtype == MOE_BF16;
    // dA = dY W2[e] (W2 stored [E,d,f] = [E,K,N]); dH = dA * G, G = GELU'(h)
    GemmVarM g_dh{E, f, d, P, offsets, dy_perm, W2, false, Epi::ScaleAux, nullptr, G, dH, nullptr};
    if (tc) {   // db1 = column sums of dH, taken in the dH GEMM's epilogue
        g_dh.colsum = db1;
        g_dh.colsum_partial = partial;
        g_dh.colsum_accumulate = accumulate;
    }
    // dX = dH W1[e] (W1 stored [E,f,d] = [E,K,N])
    GemmVarM g_dx{E, d, f, P, offsets, dH, W1, false, Epi::Plain, nullptr, nullptr, dx_perm, nullptr};
    cudaError_t e = tc ? launch_gemm_varm_tc(g_dh, status, st) : launch_gemm_varm_simt(g_dh, st);
    if (e == cudaSuccess)
        e = tc ? launch_gemm_varm_tc(g_dx, status, st) : launch_gemm_varm_simt(g_dx, st);
    if (e == cudaSuccess && !tc)
        e = launch_segment_colsum(s, dH, f, offsets, db1, accumulate, partial, st);
    return e;
}

// A8, weight half over nchunks dispatch chunks whose rows follow one another in
// dy_perm, x_perm, dH and A (chunk c holds chunk_T[c] * k rows, its expert
// offsets at offsets + c * ostride):
//   dW2[e] (+)= dY^T A,  db2[e] (+)= sum_rows dY,  dW1[e] (+)= dH^T X
// summed over every chunk's rows of expert e.  Chunks beyond what one launch
// walks go to further launches that accumulate.  `partial`: column-sum
// partial rows of the fp32 path (ffn_partial_bytes of the largest chunk).
// perm != nullptr: x_perm is the unpermuted x of all chunks (chunk c's tokens
// after those of chunks < c) and chunk c's rows of X_perm are read through its
// perm (at perm + c * perm_stride): row r is x[token base + perm[r] / k].
cudaError_t ffn_bwd_weights(const moe_shape& s, int nchunks, const int64_t* chunk_T,
                            const int32_t* offsets, int ostride, const void* dy_perm,
                            const void* x_perm, const void* dH, const void* A, float* dW1,
                            float* dW2, float* db2, int accumulate, float* partial,
                            void* split, size_t split_size, int32_t* status, cudaStream_t st,
                            const int32_t* perm = nullptr, int64_t perm_stride = 0) {
    const int E = s.E, d = s.d, f = s.f, k = s.k;
    const bool tc = s.dtype == MOE_BF16;
    int64_t P = 0, Ttot = 0;
    for (int c = 0; c < nchunks; ++c) {
        P += chunk_T[c] * k;
        Ttot += chunk_T[c];
    }
    int64_t base = 0, tbase = 0;
    for (int c0 = 0; c0 < nchunks; c0 += kMaxWgradChunks) {
        const int n = nchunks - c0 < kMaxWgradChunks ? nchunks - c0 : kMaxWgradChunks;
        const int acc = accumulate || c0 > 0;
        // dW2[e] = dY^T A  ([d, f]);  dW1[e] = dH^T X  ([f, d])
        GemmVarK g_w2{E, d, f, P, offsets + (int64_t)c0 * ostride, dy_perm, A, dW2, acc};
        if (tc) g_w2.bsum = db2;   // db2 = column sums of dY_perm, by the dW2 GEMM
        GemmVarK g_w1{E, f, d, P, offsets + (int64_t)c0 * ostride, dH, x_perm, dW1, acc};
        int64_t b = base, tb = tbase;
        for (int i = 0; i < n; ++i) {
            g_w2.seg_base[i] = g_w1.seg_base[i] = b;
            g_w1.gather_base[i] = tb;
            b += chunk_T[c0 + i] * k;
            tb += chunk_T[c0 + i];
        }
        if (perm) {
            g_w1.gather_b = perm + (int64_t)c0 * perm_stride;
            g_w1.gather_k = k;
            g_w1.gather_stride = perm_stride;
            g_w1.gather_rows = Ttot;
        }
        g_w2.nseg = g_w1.nseg = n;
        g_w2.ostride = g_w1.ostride = ostride;
        g_w2.part = g_w1.part = (float*)split;   // used by one launch after the other
        g_w2.part_bytes = g_w1.part_bytes = split ? split_size : 0;
        cudaError_t e = tc ? launch_gemm_vark_tc(g_w2, status, st) : launch_gemm_vark_simt(g_w2, st);
        if (e == cudaSuccess)
            e = tc ? launch_gemm_vark_tc(g_w1, status, st) : launch_gemm_vark_simt(g_w1, st);
        if (e != cudaSuccess) return e;
        if (!tc) {
            // db2 per chunk, in chunk order
            for (int i = 0; i < n; ++i) {
                moe_shape sc = s;
                sc.T = chunk_T[c0 + i];
                const int64_t rb = g_w2.seg_base[i];
                e = launch_segment_colsum(sc, (const float*)dy_perm + rb * d, d,
                                          offsets + (int64_t)(c0 + i) * ostride, db2,
                                          acc || i > 0, partial, st);
                if (e != cudaSuccess) return e;
            }
        }
        base = b;
        tbase = tb;
    }
    return cudaSuccess;
}

// zero the weight / bias gradients of an empty call (accumulate == 0)
cudaError_t zero_grads(const moe_shape& s, float* a, size_t na, float* b, size_t nb,
                       cudaStream_t st) {
    cudaError_t e = a ? cudaMemsetAsync(a, 0, sizeof(float) * na, st) : cudaSuccess;
    if (e == cudaSuccess && b) e = cudaMemsetAsync(b, 0, sizeof(float) * nb, st);
    (void)s;
    return e;
}

}  // namespace

extern "C" {

moe_status moe_expert_ffn_bwd(const moe_shape* s, const void* dy_perm, const void* x_perm,
                              const void* G, const void* A, const int32_t* offsets,
                              const void* W1, const void* W2, void* dx_perm, float* dW1,
                              float* db1, float* dW2, float* db2, int accumulate, void* ws,
                              int32_t* dev_status, moe_stream_t stream) {
    moe_status r = check_gemm_shape(s);
    if (r != MOE_OK) return r;
    if (!ok_ptr(dW1) || !ok_ptr(db1) || !ok_ptr(dW2) || !ok_ptr(db2)) return MOE_ERR_INVALID;
    cudaStream_t st = (cudaStream_t)stream;
    const int E = s->E, d = s->d, f = s->f;
    if (s->T == 0) {
        if (accumulate) return MOE_OK;
        cudaError_t e = zero_grads(*s, dW1, (size_t)E * f * d, db1, (size_t)E * f, st);
        if (e == cudaSuccess) e = zero_grads(*s, dW2, (size_t)E * d * f, db2, (size_t)E * d, st);
        return cuda_status(e);
    }
    if (!ok_ptr(dy_perm) || !ok_ptr(x_perm) || !ok_ptr(G) || !ok_ptr(A) || !ok_ptr(offsets) ||
        !ok_ptr(W1) || !ok_ptr(W2) || !ok_ptr(dx_perm) || !ok_ptr(ws) || !ok_status(dev_status))
        return MOE_ERR_INVALID;
    const int64_t P = s->T * s->k;
    // workspace: dH | column-sum partials | split scratch
    uint8_t* wsb = (uint8_t*)ws;
    void* dH = wsb;
    const size_t dh_bytes = align_up((size_t)P * f * esize(*s));
    float* partial = (float*)(wsb + dh_bytes);
    uint8_t* split = wsb + dh_bytes + ffn_partial_bytes(*s);
    cudaError_t e = ffn_bwd_data(*s, dy_perm, G, offsets, W1, W2, dH, dx_perm, db1, accumulate,
                                 partial, dev_status, st);
    const int64_t T = s->T;
    if (e == cudaSuccess)
        e = ffn_bwd_weights(*s, 1, &T, offsets, E + 1, dy_perm, x_perm, dH, A, dW1, dW2, db2,
                            accumulate, partial, split, split_bytes(*s, P), dev_status, st);
    return cuda_status(e);
}

moe_status moe_expert_ffn_bwd_data(const moe_shape* s, const void* dy_perm, const void* G,
                                   const int32_t* offsets, const void* W1, const void* W2,
                                   void* dH, void* dx_perm, float* db1, int accumulate, void* ws,
                                   int32_t* dev_status, moe_stream_t stream) {
    moe_status r = check_gemm_shape(s);
    if (r != MOE_OK) return r;
    if (!ok_ptr(db1)) return MOE_ERR_INVALID;
    cudaStream_t st = (cudaStream_t)stream;
    if (s->T == 0)
        return accumulate ? MOE_OK
                          : cuda_status(zero_grads(*s, db1, (size_t)s->E * s->f, nullptr, 0, st));
    if (!ok_ptr(dy_perm) || !ok_ptr(G) || !ok_ptr(offsets) || !ok_ptr(W1) || !ok_ptr(W2) ||
        !ok_ptr(dH) || !ok_ptr(dx_perm) || !ok_ptr(ws) || !ok_status(dev_status))
        return MOE_ERR_INVALID;
    return cuda_status(ffn_bwd_data(*s, dy_perm, G, offsets, W1, W2, dH, dx_perm, db1,
                                    accumulate, (float*)ws, dev_status, st));
}

size_t moe_expert_ffn_bwd_weights_workspace_size(const moe_shape* s, int nchunks,
                                                 const int64_t* chunk_T) {
    if (check_gemm_shape(s) != MOE_OK || nchunks < 1 || chunk_T == nullptr) return 0;
    int64_t T = 0, Tmax = 0;
    for (int c = 0; c < nchunks; ++c) {
        if (chunk_T[c] < 0) return 0;
        T += chunk_T[c];
        Tmax = chunk_T[c] > Tmax ? chunk_T[c] : Tmax;
    }
    moe_shape big = *s;
    big.T = Tmax;
    const size_t part = s->dtype == MOE_BF16 ? 0 : ffn_partial_bytes(big);
    const size_t split = split_bytes(*s, T * s->k);
    const size_t n = part + split;
    return n > 0 ? n : 256;
}

}  // extern "C"

namespace {

// The weight half's checks and dispatch; perm != nullptr: X rows gathered (see
// ffn_bwd_weights).
moe_status bwd_weights_entry(const moe_shape* s, int nchunks, const int64_t* chunk_T,
                             const int32_t* offsets, int offsets_stride, const void* dy_perm,
                             const void* xs, const int32_t* perm, int64_t perm_stride,
                             const void* dH, const void* A, float* dW1, float* dW2, float* db2,
                             int accumulate, void* ws, size_t ws_bytes, int32_t* dev_status,
                             moe_stream_t stream) {
    moe_status r = check_gemm_shape(s);
    if (r != MOE_OK) return r;
    if (nchunks < 1 || chunk_T == nullptr || offsets_stride < s->E + 1 || offsets_stride % 4)
        return MOE_ERR_INVALID;
    if (!ok_ptr(dW1) || !ok_ptr(dW2) || !ok_ptr(db2)) return MOE_ERR_INVALID;
    int64_t T = 0, Tmax = 0;
    for (int c = 0; c < nchunks; ++c) {
        if (chunk_T[c] < 0) return MOE_ERR_INVALID;
        T += chunk_T[c];
        if (chunk_T[c] > Tmax) Tmax = chunk_T[c];
    }
    if (T * (int64_t)s->k >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    const int E = s->E, d = s->d, f = s->f;
    if (T == 0) {
        if (accumulate) return MOE_OK;
        cudaError_t e = zero_grads(*s, dW1, (size_t)E * f * d, dW2, (size_t)E * d * f, st);
        if (e == cudaSuccess) e = zero_grads(*s, db2, (size_t)E * d, nullptr, 0, st);
        return cuda_status(e);
    }
    if (!ok_ptr(dy_perm) || !ok_ptr(xs) || !ok_ptr(dH) || !ok_ptr(A) || !ok_ptr(offsets) ||
        !ok_status(dev_status) || !ok_opt(ws) || (ws == nullptr && ws_bytes != 0))
        return MOE_ERR_INVALID;
    // a gather reads chunk c's perm entries [c * perm_stride, + chunk_T[c] * k)
    if (perm && (!ok_ptr(perm) || perm_stride < Tmax * s->k))
        return MOE_ERR_INVALID;
    moe_shape big = *s;
    big.T = Tmax;
    if (s->dtype != MOE_BF16) {
        // fp32: the column-sum partials of db2 (no split)
        if (ws == nullptr || ws_bytes < ffn_partial_bytes(big)) return MOE_ERR_INVALID;
        return cuda_status(ffn_bwd_weights(*s, nchunks, chunk_T, offsets, offsets_stride, dy_perm,
                                           xs, dH, A, dW1, dW2, db2, accumulate, (float*)ws,
                                           nullptr, 0, dev_status, st, perm, perm_stride));
    }
    return cuda_status(ffn_bwd_weights(*s, nchunks, chunk_T, offsets, offsets_stride, dy_perm,
                                       xs, dH, A, dW1, dW2, db2, accumulate, nullptr, ws,
                                       ws_bytes, dev_status, st, perm, perm_stride));
}

}  // namespace

extern "C" {

moe_status moe_expert_ffn_bwd_weights(const moe_shape* s, int nchunks, const int64_t* chunk_T,
                                      const int32_t* offsets, int offsets_stride,
                                      const void* dy_perm, const void* x_perm, const void* dH,
                                      const void* A, float* dW1, float* dW2, float* db2,
                                      int accumulate, void* ws, size_t ws_bytes,
                                      int32_t* dev_status, moe_stream_t stream) {
    return bwd_weights_entry(s, nchunks, chunk_T, offsets, offsets_stride, dy_perm, x_perm,
                             nullptr, 0, dH, A, dW1, dW2, db2, accumulate, ws, ws_bytes,
                             dev_status, stream);
}

moe_status moe_expert_ffn_bwd_weights_gather(const moe_shape* s, int nchunks,
                                             const int64_t* chunk_T, const int32_t* offsets,
                                             int offsets_stride, const void* dy_perm,
                                             const void* x, const int32_t* perm,
                                             int64_t perm_stride, const void* dH, const void* A,
                                             float* dW1, float* dW2, float* db2, int accumulate,
                                             void* ws, size_t ws_bytes, int32_t* dev_status,
                                             moe_stream_t stream) {
    if (perm == nullptr) return MOE_ERR_INVALID;
    return bwd_weights_entry(s, nchunks, chunk_T, offsets, offsets_stride, dy_perm, x, perm,
                             perm_stride, dH, A, dW1, dW2, db2, accumulate, ws, ws_bytes,
                             dev_status, stream);
}

moe_status moe_route_bwd(const moe_shape* s, const float* dw, const float* logits,
                         const int32_t* idx, const float* w, const int32_t* perm,
                         const int32_t* offsets, const void* x, const void* Wg,
                         const void* dx_perm, const int32_t* pos, void* dx, float* dWg,
                         int accumulate, void* ws, int32_t* dev_status, moe_stream_t stream) {
    (void)dev_status;
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (!ok_ptr(dWg)) return MOE_ERR_INVALID;
    cudaStream_t st = (cudaStream_t)stream;
    if (s->T == 0) {
        if (accumulate) return MOE_OK;
        return cuda_status(cudaMemsetAsync(dWg, 0, sizeof(float) * (size_t)s->E * s->d, st));
    }
    if (!ok_ptr(dw) || !ok_ptr(logits) || !ok_ptr(idx) || !ok_ptr(w) || !ok_ptr(perm) ||
        !ok_ptr(offsets) || !ok_ptr(x) || !ok_ptr(Wg) || !ok_ptr(dx) || !ok_ptr(ws))
        return MOE_ERR_INVALID;
    if (dx_perm != nullptr && !(aligned16(dx_perm) && ok_ptr(pos))) return MOE_ERR_INVALID;
    float* dL = (float*)ws;
    const size_t dl_bytes = (size_t)s->T * (size_t)(s->renorm ? s->k : s->E) * sizeof(float);
    float* partial = (float*)((uint8_t*)ws + align_up(dl_bytes));
    return cuda_status(launch_route_bwd(*s, dw, logits, idx, w, perm, offsets, x, Wg, dx_perm,
                                        pos, dx, dWg, accumulate, dL, partial, st));
}

}  // extern "C"

// ---- routing without a caller workspace ----------------------------------------
// The histogram scratch of moe_route_noalloc: a fixed device array inside the
// library (1 MiB on every GPU that loads it).  In host code the symbol names a
// host-side stand-in, never a device address: the device address is looked up
// once per device and passed to the kernels.
static __device__ __align__(256) int32_t g_route_noalloc_scratch[MOE_ROUTE_NOALLOC_MAX_SCRATCH];

namespace {

// Unique id of the calling thread's current CUDA context (0 if none or if the
// driver cannot tell), through the driver entry points the runtime exposes.
unsigned long long current_context_id() {
    typedef CUresult (*GetCurrent)(CUcontext*);
    typedef CUresult (*GetId)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(f);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(f);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array in the current device's context.  It is
// looked up (cudaGetSymbolAddress, with that device current) on the first call
// for the device, and again when the context has changed since (after a
// cudaDeviceReset the old address would be stale).  nullptr if the lookup
// fails.
int32_t* route_noalloc_scratch() {
    static std::mutex mu;
    static int32_t* addr[64] = {};
    static unsigned long long ctx_of[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long ctx = current_context_id();
    if (addr[dev] == nullptr || ctx == 0 || ctx != ctx_of[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_noalloc_scratch) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<int32_t*>(p);
        ctx_of[dev] = current_context_id();   // the lookup made the context current
    }
    return addr[dev];
}

}  // namespace

extern "C" {

moe_status moe_route_noalloc(const moe_shape* s, const void* x, const void* Wg,
                             const float* logit_bias, float* logits, int compute_logits,
                             int32_t* idx, float* w, int32_t* counts, int32_t* offsets,
                             int32_t* pos, int32_t* perm, int32_t* dev_status,
                             moe_stream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (!ok_ptr(counts) || !ok_ptr(offsets)) return MOE_ERR_INVALID;
    if (s->T > 0) {
        if (!ok_ptr(logits) || !ok_ptr(idx) || !ok_ptr(w) || !ok_ptr(pos) || !ok_ptr(perm) ||
            !ok_status(dev_status))
            return MOE_ERR_INVALID;
        if (compute_logits && (!ok_ptr(x) || !ok_ptr(Wg) || !ok_opt(logit_bias)))
            return MOE_ERR_INVALID;
    }
    if ((int64_t)s->E * route_blocks(s->T) > (int64_t)MOE_ROUTE_NOALLOC_MAX_SCRATCH)
        return MOE_ERR_UNSUPPORTED;
    int32_t* block_counts = route_noalloc_scratch();
    if (block_counts == nullptr) return MOE_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaSuccess;
    if (s->T > 0)   // no scratch for split logits tiles here: whole tiles
        e = launch_route_gate(*s, x, Wg, logit_bias, logits, compute_logits, idx, w, block_counts,
                              nullptr, 0, dev_status, st);
    if (e == cudaSuccess) e = launch_dispatch_scan(*s, block_counts, counts, offsets, st);
    if (e == cudaSuccess && s->T > 0) e = launch_dispatch_rank(*s, idx, block_counts, pos, perm, st);
    return cuda_status(e);
}

moe_status moe_debug_bounded_wait(uint64_t limit_ns, int32_t* dev_status, moe_stream_t stream) {
    if (dev_status == nullptr || !ok_status(dev_status)) return MOE_ERR_INVALID;
    return cuda_status(launch_bounded_wait(limit_ns, dev_status, (cudaStream_t)stream));
}

moe_status moe_set_gemm_max_units(int units) {
    if (units < 0) return MOE_ERR_INVALID;
    set_gemm_units_cap(units);
    return MOE_OK;
}

moe_status moe_debug_gelu(int64_t n, const float* x, float* gelu, float* gelu_grad, int fast,
                          moe_stream_t stream) {
    if (n < 0) return MOE_ERR_INVALID;
    if (n == 0) return MOE_OK;
    if (!ok_ptr(x) || !ok_ptr(gelu) || !ok_ptr(gelu_grad)) return MOE_ERR_INVALID;
    return cuda_status(launch_debug_gelu(n, x, gelu, gelu_grad, fast, (cudaStream_t)stream));
}

}  // extern "C"
