// kernels.h -- host-side launchers of the layer's kernels (internal to
// libmoe.so; the public interface is include/moe.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Tokens handled by one block of the gate / rank kernels: the per-block
// histogram is a bitmask of 64 tokens (two 32-bit words) per expert.
constexpr int kMaxExperts = 256;   // largest moe_shape::E the entry points accept
constexpr int kRouteBlockTokens = 64;
constexpr int kRouteWords = kRouteBlockTokens / 32;
// Rows summed per partial of the router weight gradient and of the bias
// gradients (column sums).
constexpr int kDwgChunk = 32;
// Dispatch chunks one weight-gradient GEMM launch walks (more are split over
// several launches that accumulate).
constexpr int kMaxWgradChunks = 16;

inline int64_t route_blocks(int64_t T) { return (T + kRouteBlockTokens - 1) / kRouteBlockTokens; }

// Default bound on every device-side wait (ns); MOE_WAIT_TIMEOUT_NS overrides.
uint64_t wait_limit_ns();
int device_sm_count();

// A1 (when compute_logits) + A2 + per-block histogram (block_counts laid out
// [E][nblk]).  E <= 32 fuses all three in one kernel.
// `part` (optional, part_bytes): scratch for the CUDA-core logits' split tiles
cudaError_t launch_route_gate(const moe_shape& s, const void* x, const void* Wg,
                             const float* beta, float* logits, int compute_logits, int32_t* idx,
                             float* w, int32_t* block_counts, float* part, size_t part_bytes,
                             int32_t* status, cudaStream_t st);
// scratch bytes of the CUDA-core router logits' split tiles
size_t router_logits_workspace(const moe_shape& s);
// A3 scan: block_counts -> block_base in place, counts, offsets
cudaError_t launch_dispatch_scan(const moe_shape& s, int32_t* block_counts,
                                 int32_t* counts, int32_t* offsets, cudaStream_t st);
// A3 stable rank: pos, perm
cudaError_t launch_dispatch_rank(const moe_shape& s, const int32_t* idx,
                                 const int32_t* block_base, int32_t* pos, int32_t* perm,
                                 cudaStream_t st);
// A10
cudaError_t launch_route_bwd(const moe_shape& s, const float* dw, const float* logits,
                             const int32_t* idx, const float* w, const int32_t* perm,
                             const int32_t* offsets, const void* x, const void* Wg,
                             const void* dx_perm, const int32_t* pos, void* dx, float* dWg,
                             int accumulate, float* dL, float* partial, cudaStream_t st);
size_t route_bwd_workspace(const moe_shape& s);  // dL + partials, bytes

// A4, A6/A9, A7
cudaError_t launch_permute(const moe_shape& s, const void* x, const int32_t* pos,
                           void* x_perm, cudaStream_t st);
cudaError_t launch_combine(const moe_shape& s, const void* y_perm, const int32_t* pos,
                           const float* w, void* y, cudaStream_t st);
cudaError_t launch_combine_bwd(const moe_shape& s, const void* dy, const void* y_perm,
                               const int32_t* pos, const float* w, void* dy_perm,
                               float* dw, cudaStream_t st);
// per-expert column sums of a [T*k, n] activation: out[e][c] (+)= sum rows
cudaError_t launch_segment_colsum(const moe_shape& s, const void* g, int n,
                                  const int32_t* offsets, float* out, int accumulate,
                                  float* partial, cudaStream_t st);
// per-expert weighted, gathered row sums: for the rows p of expert e's segment,
// slot = perm[p], out[e][c] (+)= sum wsel[slot] src[slot / k][c]
cudaError_t launch_segment_rowsum(const moe_shape& s, const void* src, int n,
                                  const int32_t* offsets, const int32_t* perm,
                                  const float* wsel, float* out, int accumulate, float* partial,
                                  cudaStream_t st);
size_t segment_colsum_workspace(const moe_shape& s, int n);

// Grouped expert GEMMs.  Operand layouts (row-major):
//   VarM ("fwd"/"dgrad"): for each expert e, rows [off_e, off_e+n_e) of act
//   [P, K] times the expert's weight, giving out rows [P, N].  The weight is
//   [E, N, K] (b_kmajor) or [E, K, N].
//   VarK ("wgrad"): C_e [M, N] (+)= act_a[seg_e, M]^T act_b[seg_e, N], fp32.
// BiasGelu: h = acc + bias; out0 = GELU'(h), out1 = GELU(h).
// Bias: out0 = acc + bias.  ScaleAux: out0 = acc * aux.  Plain: out0 = acc.
// Logits: fp32 out0 [P,N] = act W^T + bias (fp32 [N], optional), any N >= 1;
// the router logits, one segment (offsets may be null: rows [0, P)).
enum class Epi : int { BiasGelu = 0, Bias = 1, ScaleAux = 2, Plain = 3, Logits = 4 };

struct GemmVarM {
    int E, N, K;
    int64_t P;              // rows of act / out
    const int32_t* offsets; // [E+1]
    const void* act;        // [P, K]
    const void* weight;     // [E,N,K] or [E,K,N]
    bool weight_kmajor;     // true: [E,N,K]
    Epi epi;
    const void* bias;       // [E,N] or null
    const void* aux;        // ScaleAux: G = GELU'(h) [P,N]
    void* out0;             // [P,N]
    void* out1;             // BiasGelu: A = GELU(h) [P,N]
    // ScaleAux, tensor-core path: when non-null, also the per-expert column
    // sums of the stored out0 into colsum [E,N] (added to it when
    // colsum_accumulate), through colsum_partial (gemm_colsum_workspace bytes).
    float* colsum = nullptr;
    float* colsum_partial = nullptr;
    int colsum_accumulate = 0;
    // Row gather (the permute fused into the loads): when non-null, act is the
    // unpermuted source [gather_rows, K] and row r of the operand is
    // act[gather[r] / gather_k] (gather = the dispatch's perm, gather_k = k).
    const int32_t* gather = nullptr;
    int gather_k = 1;
    int64_t gather_rows = 0;
};
// Bytes of GemmVarM::colsum_partial for P rows, E experts, N columns.
size_t gemm_colsum_workspace(int64_t P, int E, int N);
struct GemmVarK {
    int E, M, N;
    int64_t P;              // rows of act_a / act_b (all segments)
    const int32_t* offsets; // [nseg][ostride]: each chunk's expert offsets (E+1 used)
    const void* act_a;      // [P, M]
    const void* act_b;      // [P, N]
    float* out;             // [E, M, N]
    int accumulate;
    // tensor-core path: when non-null, also bsum[e][m] (+)= sum over expert e's
    // rows of act_a[row][m] (a bias gradient), from one extra tile per
    // (expert, m-tile) whose B operand is a constant all-ones block
    float* bsum = nullptr;
    // expert e's rows are, in each dispatch chunk s < nseg,
    // [seg_base[s] + offsets[s*ostride + e], seg_base[s] + offsets[s*ostride + e + 1])
    int nseg = 1;
    int ostride = 0;
    int64_t seg_base[kMaxWgradChunks] = {};
    // tensor-core path: scratch for the partial tiles of long reductions split
    // into parts (none when null or too small for one tile)
    float* part = nullptr;
    size_t part_bytes = 0;
    // Row gather of act_b: when non-null, act_b is the unpermuted source
    // [gather_rows, N] and row r of chunk s's rows (r counted from seg_base[s])
    // is act_b[gather_base[s] + gather_b[s * gather_stride + r] / gather_k].
    const int32_t* gather_b = nullptr;
    int gather_k = 1;
    int64_t gather_stride = 0;
    int64_t gather_base[kMaxWgradChunks] = {};
    int64_t gather_rows = 0;
};
// Scratch bytes that let the weight-gradient GEMMs over `rows` rows split their
// long reductions as finely as they would (parts of >= 256 K blocks of 64 rows).
size_t vark_split_workspace(int64_t rows, int E, int M, int N);

// Cap on the tensor-core GEMMs' CTA pairs (single CTAs) per launch for the
// calling host thread; 0 = the co-resident maximum.
void set_gemm_units_cap(int64_t units);
cudaError_t launch_gemm_varm_tc(const GemmVarM& g, int32_t* status, cudaStream_t st);
cudaError_t launch_gemm_vark_tc(const GemmVarK& g, int32_t* status, cudaStream_t st);
cudaError_t launch_gemm_varm_simt(const GemmVarM& g, cudaStream_t st);
cudaError_t launch_gemm_vark_simt(const GemmVarK& g, cudaStream_t st);

// Diagnostics
cudaError_t launch_bounded_wait(uint64_t limit_ns, int32_t* status, cudaStream_t st);
cudaError_t launch_debug_gelu(int64_t n, const float* x, float* g, float* gd, int fast,
                              cudaStream_t st);

}  // namespace moe
