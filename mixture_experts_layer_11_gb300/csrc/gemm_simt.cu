// gemm_simt.cu -- grouped per-expert GEMMs in fp32 on CUDA cores (the fp32
// layer: tensor-core TF32 would not meet fp32 accuracy).
//
// The experts run over their own contiguous row segments only, with no
// padding ("ES-MoE", review, section 3 and section 4 table row "sequential
// processing"; "FastMoE", review, per-expert FMoELinear).  Same operand
// conventions and epilogues as the tensor-core path (kernels.h).
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int SB = 64;   // tile rows and columns
constexpr int SK = 16;   // K step

// Locate (expert, m-tile) of linear tile id `tid_lin` over experts' segments.
__device__ __forceinline__ bool find_mtile(int E, const int32_t* offsets, int tid_lin,
                                           int& e, int& mt) {
    int acc = 0;
    for (e = 0; e < E; ++e) {
        const int n = offsets[e + 1] - offsets[e];
        const int nt = (n + SB - 1) / SB;
        if (tid_lin < acc + nt) { mt = tid_lin - acc; return true; }
        acc += nt;
    }
    return false;
}

__global__ void __launch_bounds__(256) gemm_varm_f32_kernel(GemmVarM g) {
    __shared__ float As[SK][SB + 1];
    __shared__ float Bs[SK][SB + 1];
    int e, mt;
    if (!find_mtile(g.E, g.offsets, blockIdx.x, e, mt)) return;
    const int row0 = g.offsets[e] + mt * SB;
    const int rows = min(SB, g.offsets[e + 1] - row0);
    const int n0 = blockIdx.y * SB;
    const float* act = (const float*)g.act;
    const float* W = (const float*)g.weight + (int64_t)e * g.N * g.K;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < g.K; k0 += SK) {
        for (int i = threadIdx.x; i < SB * SK; i += 256) {
            const int r = i / SK, c = i % SK;
            float v = 0.f;
            if (r < rows && k0 + c < g.K) {
                const int64_t src = g.gather ? (int64_t)(g.gather[row0 + r] / g.gather_k)
                                             : (int64_t)(row0 + r);
                v = act[src * g.K + k0 + c];
            }
            As[c][r] = v;
        }
        for (int i = threadIdx.x; i < SB * SK; i += 256) {
            int n, c;
            float v = 0.f;
            if (g.weight_kmajor) {
                n = i / SK; c = i % SK;
                if (n0 + n < g.N && k0 + c < g.K) v = W[(int64_t)(n0 + n) * g.K + k0 + c];
            } else {
                c = i / SB; n = i % SB;
                if (n0 + n < g.N && k0 + c < g.K) v = W[(int64_t)(k0 + c) * g.N + n0 + n];
            }
            Bs[c][n] = v;
        }
        __syncthreads();
        #pragma unroll
        for (int kk = 0; kk < SK; ++kk) {
            float a[4], b[4];
            #pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
            #pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
            #pragma unroll
            for (int i = 0; i < 4; ++i)
                #pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    const float* bias = (const float*)g.bias;
    #pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = ty + 16 * i;
        if (r >= rows) continue;
        const int64_t row = row0 + r;
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx + 16 * j;
            if (n >= g.N) continue;
            float v = acc[i][j];
            const int64_t o = row * g.N + n;
            switch (g.epi) {
                case Epi::BiasGelu:
                    v += bias ? bias[(int64_t)e * g.N + n] : 0.f;
                    ((float*)g.out0)[o] = gelu_grad_f(v);
                    ((float*)g.out1)[o] = gelu_f(v);
                    break;
                case Epi::Bias:
                    v += bias ? bias[(int64_t)e * g.N + n] : 0.f;
                    ((float*)g.out0)[o] = v;
                    break;
                case Epi::ScaleAux:
                    ((float*)g.out0)[o] = v * ((const float*)g.aux)[o];
                    break;
                case Epi::Plain:
                    ((float*)g.out0)[o] = v;
                    break;
            }
        }
    }
}

__global__ void __launch_bounds__(256) gemm_vark_f32_kernel(GemmVarK g) {
    __shared__ float As[SK][SB + 1];
    __shared__ float Bs[SK][SB + 1];
    const int e = blockIdx.z;
    const int m0 = blockIdx.x * SB, n0 = blockIdx.y * SB;
    const int p0 = g.offsets[e], p1 = g.offsets[e + 1];
    const float* a = (const float*)g.act_a;
    const float* b = (const float*)g.act_b;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4] = {};
    for (int k0 = p0; k0 < p1; k0 += SK) {
        for (int i = threadIdx.x; i < SB * SK; i += 256) {
            const int c = i / SB, r = i % SB;  // c: row of the segment, r: column
            const bool kin = k0 + c < p1;
            As[c][r] = (kin && m0 + r < g.M) ? a[(int64_t)(k0 + c) * g.M + m0 + r] : 0.f;
            float bv = 0.f;
            if (kin && n0 + r < g.N) {
                const int64_t src = g.gather_b ? g.gather_base[0] + g.gather_b[k0 + c] / g.gather_k
                                               : (int64_t)(k0 + c);
                bv = b[src * g.N + n0 + r];
            }
            Bs[c][r] = bv;
        }
        __syncthreads();
        #pragma unroll
        for (int kk = 0; kk < SK; ++kk) {
            float av[4], bv[4];
            #pragma unroll
            for (int i = 0; i < 4; ++i) av[i] = As[kk][ty + 16 * i];
            #pragma unroll
            for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx + 16 * j];
            #pragma unroll
            for (int i = 0; i < 4; ++i)
                #pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
    #pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty + 16 * i;
        if (m >= g.M) continue;
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx + 16 * j;
            if (n >= g.N) continue;
            float* o = g.out + ((int64_t)e * g.M + m) * g.N + n;
            *o = g.accumulate ? *o + acc[i][j] : acc[i][j];
        }
    }
}

}  // namespace

cudaError_t launch_gemm_varm_simt(const GemmVarM& g, cudaStream_t st) {
    const int64_t mtiles = (g.P + SB - 1) / SB + g.E;  // upper bound over experts
    dim3 grid((unsigned)mtiles, (unsigned)((g.N + SB - 1) / SB));
    gemm_varm_f32_kernel<<<grid, 256, 0, st>>>(g);
    return cudaGetLastError();
}

cudaError_t launch_gemm_vark_simt(const GemmVarK& g, cudaStream_t st) {
    dim3 grid((unsigned)((g.M + SB - 1) / SB), (unsigned)((g.N + SB - 1) / SB), (unsigned)g.E);
    // one launch per dispatch chunk, each adding to the previous ones
    for (int s = 0; s < g.nseg; ++s) {
        GemmVarK c = g;
        c.nseg = 1;
        c.offsets = g.offsets + (int64_t)s * g.ostride;
        c.act_a = (const float*)g.act_a + g.seg_base[s] * g.M;
        if (g.gather_b) {   // rows of the unpermuted source, through chunk s's perm
            c.gather_b = g.gather_b + (int64_t)s * g.gather_stride;
            c.gather_base[0] = g.gather_base[s];
        } else {
            c.act_b = (const float*)g.act_b + g.seg_base[s] * g.N;
        }
        c.accumulate = g.accumulate || s > 0;
        gemm_vark_f32_kernel<<<grid, 256, 0, st>>>(c);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace moe
