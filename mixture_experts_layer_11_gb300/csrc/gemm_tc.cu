// gemm_tc.cu -- grouped per-expert GEMMs on the 5th-generation tensor cores
// (tcgen05.mma, fp32 accumulators in TMEM, operands staged by TMA).
//
// Each expert runs only over its own contiguous row segment of the
// expert-sorted activations, with no dispatch mask and no padding to a
// capacity ("ES-MoE", review, section 3 "expert-wise offloading and
// processing", section 4 table row "sequential processing"; the per-expert
// linear FMoELinear of "FastMoE", review, "proposed method").  Instead of
// running the experts one after another, all (expert, tile) work items of a
// call form one list that a persistent grid walks; segment boundaries are read
// from device memory, so no host synchronisation is needed.
//
// Two problem shapes:
//   VarM (forward, data gradient): out[seg_e, N] = act[seg_e, K] W_e^T with
//     the weight stored [E,N,K] (K-major) or [E,K,N] (MN-major); the segment
//     length varies per expert.  Rows past the segment are computed from
//     whatever TMA loads there and never stored.
//   VarK (weight gradient): C_e[M, N] (+)= act_a[seg_e, M]^T act_b[seg_e, N];
//     the reduction runs over the segment's rows, so rows past the segment in
//     the last K block are zeroed in shared memory before the MMA reads them.
//
// CTA = 10 warps: warp 0 issues TMA loads into a 4-stage ring, warp 1 issues
// tcgen05.mma (M=128, N=256, K=16 per instruction) into one of two TMEM
// accumulators (2 x 256 fp32 columns), warps 2-9 drain the other accumulator
// (tcgen05.ld), apply the fused epilogue (bias, GELU, GELU', fp32 accumulate)
// and write through a swizzled shared staging buffer with coalesced stores.
// Every wait is bounded; on expiry the CTA records MOE_ERR_TIMEOUT, waits for
// its own copies and MMAs in flight, frees TMEM and exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int BM = 128;            // tile rows (MMA M)
constexpr int BN = 256;            // tile columns (MMA N)
constexpr int BK = 64;             // K per stage: one 128-byte swizzle row of bf16
constexpr int STAGES = 4;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 32 * (2 + EPI_WARPS);
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SLAB_BYTES = 64 * BK * 2;    // one 64-wide MN slab of BK rows
constexpr int STAGING_BYTES = 32 * 64;     // per epilogue warp: 32 rows x 64 B
constexpr int TMEM_COLS = 2 * BN;
constexpr int MAX_E = 256;

struct TcParams {
    int E, M, N, K;          // VarM: N, K (M unused); VarK: M, N (K = segment)
    int64_t P;
    const int32_t* offsets;
    const void* bias;
    const void* aux;
    void* out0;
    void* out1;
    float* outf;
    int accumulate;
    int32_t* status;
    uint64_t limit_ns;
};

struct Ctrl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int nactive;
    int off[MAX_E + 1];
    int tile_start[MAX_E + 1];   // VarM: first tile of each expert
    int order[MAX_E];            // VarK: experts by descending row count
};

constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES +
                              (size_t)EPI_WARPS * STAGING_BYTES + sizeof(Ctrl);

struct Tile {
    int e, mt, nt, num_kb;
    int row0;     // VarM: first row of the tile; VarK: first row of the segment
    int rows;     // VarM: valid rows in the tile; VarK: rows of the segment
};

template <bool VAR_K>
__device__ __forceinline__ Tile get_tile(const Ctrl& c, const TcParams& p, int t, int& ecur) {
    Tile ti;
    const int NT = (p.N + BN - 1) / BN;
    if (!VAR_K) {
        while (c.tile_start[ecur + 1] <= t) ++ecur;
        const int local = t - c.tile_start[ecur];
        ti.e = ecur;
        ti.mt = local / NT;
        ti.nt = local % NT;
        ti.row0 = c.off[ecur] + ti.mt * BM;
        ti.rows = min(BM, c.off[ecur + 1] - ti.row0);
        ti.num_kb = p.K / BK;
    } else {
        const int MT = (p.M + BM - 1) / BM;
        const int per = MT * NT;
        ti.e = c.order[t / per];
        const int local = t % per;
        ti.mt = local / NT;
        ti.nt = local % NT;
        ti.row0 = c.off[ti.e];
        ti.rows = c.off[ti.e + 1] - ti.row0;
        ti.num_kb = (ti.rows + BK - 1) / BK;
    }
    return ti;
}

__device__ __forceinline__ void raise_abort(Ctrl& c, const TcParams& p) {
    *(volatile int*)&c.abort_flag = 1;
    report(p.status, MOE_ERR_TIMEOUT);
}

// ---- epilogue helpers: 32 rows x 64 bytes staging, 16-byte chunks XOR-swizzled
// so that both the per-row writes and the coalesced reads are conflict-free.
__device__ __forceinline__ uint32_t stg_off(int row, int ch) {
    return (uint32_t)(row * 64 + ((ch ^ ((row >> 1) & 3)) << 4));
}

__device__ __forceinline__ uint4 pack8_bf16(const float* v) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
    #pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    return u;
}

// this thread's row (lane) of 32 bf16 values -> staging
__device__ __forceinline__ void stage_row_bf16(uint8_t* stg, int lane, const float* v) {
    #pragma unroll
    for (int ch = 0; ch < 4; ++ch)
        *reinterpret_cast<uint4*>(stg + stg_off(lane, ch)) = pack8_bf16(v + 8 * ch);
}

// staging (32 rows x 32 bf16) -> global rows row0.., columns col0.., ld = N
__device__ __forceinline__ void store_tile_bf16(const uint8_t* stg, int lane, __nv_bfloat16* out,
                                                int64_t row0, int valid_rows, int64_t ld,
                                                int col0) {
    #pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int rr = it * 8 + (lane >> 2), ch = lane & 3;
        if (rr < valid_rows) {
            const uint4 v = *reinterpret_cast<const uint4*>(stg + stg_off(rr, ch));
            *reinterpret_cast<uint4*>(out + (row0 + rr) * ld + col0 + ch * 8) = v;
        }
    }
}

template <bool VAR_K, bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mapA,
                   const __grid_constant__ CUtensorMap mapB, const TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* staging_base = base + (size_t)STAGES * STAGE_BYTES;
    Ctrl& c = *reinterpret_cast<Ctrl*>(staging_base + (size_t)EPI_WARPS * STAGING_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;
    const int NT = (p.N + BN - 1) / BN;

    // ---- set-up: barriers, TMEM, tile list ------------------------------------
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&c.full[s]), 1);
            mbar_init(smem_u32(&c.empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&c.tfull[b]), 1);
            mbar_init(smem_u32(&c.tempty[b]), EPI_WARPS);
        }
        mbar_init(smem_u32(&c.drain), 1);
        c.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&c.tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    for (int i = threadIdx.x; i <= E; i += THREADS) c.off[i] = p.offsets[i];
    __syncthreads();
    if (!VAR_K) {
        if (threadIdx.x == 0) {
            int acc = 0;
            for (int e = 0; e < E; ++e) {
                c.tile_start[e] = acc;
                acc += ((c.off[e + 1] - c.off[e] + BM - 1) / BM) * NT;
            }
            c.tile_start[E] = acc;
            c.nactive = acc;   // number of tiles
        }
    } else {
        for (int e = threadIdx.x; e < E; e += THREADS) {
            const int n = c.off[e + 1] - c.off[e];
            int r = 0;
            for (int q = 0; q < E; ++q) {
                const int m = c.off[q + 1] - c.off[q];
                r += (m > n) || (m == n && q < e);
            }
            c.order[r] = e;
        }
        if (threadIdx.x == 0) {
            int act = 0;
            for (int e = 0; e < E; ++e) act += (c.off[e + 1] - c.off[e]) > 0;
            const int MT = (p.M + BM - 1) / BM;
            c.nactive = (p.accumulate ? act : E) * MT * NT;  // number of tiles
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = c.tmem_base;
    const int num_tiles = c.nactive;

    if (warp == 0) {
        // ---- TMA producer ---------------------------------------------------------
        if (lane == 0) {
            tma_prefetch_map(&mapA);
            tma_prefetch_map(&mapB);
            int stage = 0, ecur = 0;
            uint32_t phase = 0;
            int issued_parity[STAGES];
            for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const Tile ti = get_tile<VAR_K>(c, p, t, ecur);
                for (int kb = 0; kb < ti.num_kb; ++kb) {
                    if (!mbar_wait_bounded(smem_u32(&c.empty[stage]), phase ^ 1, p.limit_ns,
                                           &c.abort_flag)) {
                        raise_abort(c, p);
                        ok = false;
                        break;
                    }
                    const uint32_t sA = smem_u32(base + (size_t)stage * STAGE_BYTES);
                    const uint32_t sB = sA + A_BYTES;
                    const uint32_t fb = smem_u32(&c.full[stage]);
                    // bytes: full boxes, except MN slabs lying wholly past the edge
                    uint32_t bytes = 0;
                    if (!VAR_K) {
                        bytes += A_BYTES;
                        if (!B_MN) bytes += B_BYTES;
                        else
                            for (int i = 0; i < BN / 64; ++i)
                                if (ti.nt * BN + 64 * i < p.N) bytes += SLAB_BYTES;
                    } else {
                        for (int i = 0; i < BM / 64; ++i)
                            if (ti.mt * BM + 64 * i < p.M) bytes += SLAB_BYTES;
                        for (int i = 0; i < BN / 64; ++i)
                            if (ti.nt * BN + 64 * i < p.N) bytes += SLAB_BYTES;
                    }
                    mbar_arrive_expect_tx(fb, bytes);
                    if (!VAR_K) {
                        tma_load_2d(sA, &mapA, fb, kb * BK, ti.row0);
                        if (!B_MN) {
                            tma_load_3d(sB, &mapB, fb, kb * BK, ti.nt * BN, ti.e);
                        } else {
                            for (int i = 0; i < BN / 64; ++i)
                                if (ti.nt * BN + 64 * i < p.N)
                                    tma_load_3d(sB + i * SLAB_BYTES, &mapB, fb,
                                                ti.nt * BN + 64 * i, kb * BK, ti.e);
                        }
                    } else {
                        const int r = ti.row0 + kb * BK;
                        for (int i = 0; i < BM / 64; ++i)
                            if (ti.mt * BM + 64 * i < p.M)
                                tma_load_2d(sA + i * SLAB_BYTES, &mapA, fb, ti.mt * BM + 64 * i, r);
                        for (int i = 0; i < BN / 64; ++i)
                            if (ti.nt * BN + 64 * i < p.N)
                                tma_load_2d(sB + i * SLAB_BYTES, &mapB, fb, ti.nt * BN + 64 * i, r);
                    }
                    issued_parity[stage] = (int)phase;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) {
                // wait (bounded) for every copy this thread started
                for (int s = 0; s < STAGES; ++s)
                    if (issued_parity[s] >= 0)
                        mbar_wait_bounded(smem_u32(&c.full[s]), (uint32_t)issued_parity[s],
                                          p.limit_ns, nullptr);
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer -------------------------------------------------------------
        constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, A_MN, B_MN);
        int stage = 0, acc = 0, ecur = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            const Tile ti = get_tile<VAR_K>(c, p, t, ecur);
            if (ti.num_kb == 0) continue;
            if (!mbar_wait_warp(smem_u32(&c.tempty[acc]), acc_phase ^ 1, p.limit_ns,
                                &c.abort_flag)) {
                raise_abort(c, p);
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int kb = 0; kb < ti.num_kb; ++kb) {
                if (!mbar_wait_warp(smem_u32(&c.full[stage]), phase, p.limit_ns,
                                    &c.abort_flag)) {
                    raise_abort(c, p);
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint8_t* gA = base + (size_t)stage * STAGE_BYTES;
                uint8_t* gB = gA + A_BYTES;
                if (VAR_K) {
                    const int valid = ti.rows - kb * BK;
                    if (valid < BK) {
                        // zero K rows past the segment in all 6 MN slabs
                        const int nz = (BK - valid) * 8;  // 16-byte chunks per slab
                        for (int sl = 0; sl < (BM + BN) / 64; ++sl) {
                            uint8_t* slab = (sl < BM / 64) ? gA + sl * SLAB_BYTES
                                                           : gB + (sl - BM / 64) * SLAB_BYTES;
                            for (int i = lane; i < nz; i += 32)
                                *reinterpret_cast<uint4*>(slab + (valid + (i >> 3)) * 128 +
                                                          ((i & 7) << 4)) = make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                }
                if (lane == 0) {
                    const uint32_t sA = smem_u32(gA), sB = smem_u32(gB);
                    #pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t ad =
                            A_MN ? smem_desc_sw128(sA + kk * 2048, SLAB_BYTES, 1024)
                                 : smem_desc_sw128(sA + kk * 32, 16, 1024);
                        const uint64_t bd =
                            B_MN ? smem_desc_sw128(sB + kk * 2048, SLAB_BYTES, 1024)
                                 : smem_desc_sw128(sB + kk * 32, 16, 1024);
                        tc_mma_bf16(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit(smem_u32(&c.empty[stage]));
                }
                __syncwarp();
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
            if (lane == 0) tc_commit(smem_u32(&c.tfull[acc]));
            __syncwarp();
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
        // drain: every MMA this warp issued has completed before TMEM is freed
        if (lane == 0) tc_commit(smem_u32(&c.drain));
        __syncwarp();
        mbar_wait_bounded(smem_u32(&c.drain), 0, p.limit_ns, nullptr);
    } else {
        // ---- epilogue warps ----------------------------------------------------------
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int half = (warp - 2) >> 2;       // which 128 columns of the 256
        uint8_t* stg = staging_base + (warp - 2) * STAGING_BYTES;
        int acc = 0, ecur = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
            const Tile ti = get_tile<VAR_K>(c, p, t, ecur);
            if (ti.num_kb == 0) {
                // VarK expert without rows and accumulate == 0: gradient is zero
                if (VAR_K && !p.accumulate) {
                    const int col0 = ti.nt * BN + half * 128;
                    for (int rr = 0; rr < 32; ++rr) {
                        const int m = ti.mt * BM + q * 32 + rr;
                        const int col = col0 + lane * 4;
                        if (m < p.M && col < p.N)
                            *reinterpret_cast<float4*>(p.outf + ((int64_t)ti.e * p.M + m) * p.N + col) =
                                make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                continue;
            }
            // GELU' epilogue: the saved pre-activation H of this thread's row is
            // fetched ahead (chunk 0 before the accumulator is ready, chunk c+1
            // while chunk c is processed), so its latency overlaps other work.
            uint4 hnext[4];
            const int64_t grow_lane = (int64_t)ti.row0 + q * 32 + lane;
            const bool row_ok = (q * 32 + lane) < ti.rows;
            if (EPI == (int)Epi::GeluGrad && !VAR_K) {
                const int col0 = ti.nt * BN + half * 128;
                #pragma unroll
                for (int u = 0; u < 4; ++u)
                    hnext[u] = row_ok ? __ldg(reinterpret_cast<const uint4*>(
                                            (const __nv_bfloat16*)p.aux + grow_lane * p.N + col0 + u * 8))
                                      : make_uint4(0, 0, 0, 0);
            }
            if (!mbar_wait_warp(smem_u32(&c.tfull[acc]), acc_phase, p.limit_ns,
                                &c.abort_flag)) {
                raise_abort(c, p);
                break;
            }
            tc_fence_after();
            const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            #pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                const int cl = half * 128 + ch * 32;          // column inside the tile
                const int col0 = ti.nt * BN + cl;             // global column
                if (col0 >= p.N) break;                       // N % 64 == 0: whole chunks
                float v[32];
                tmem_ld32(trow + (uint32_t)cl, v);
                if (!VAR_K) {
                    const int64_t grow0 = (int64_t)ti.row0 + q * 32;   // global row of lane 0
                    const int valid = ti.rows - q * 32;
                    const int64_t N = p.N;
                    if (EPI == (int)Epi::BiasGelu || EPI == (int)Epi::Bias) {
                        if (p.bias) {
                            const __nv_bfloat16* bp =
                                (const __nv_bfloat16*)p.bias + (int64_t)ti.e * N + col0;
                            #pragma unroll
                            for (int u = 0; u < 32; u += 8) {
                                const uint4 bv = *reinterpret_cast<const uint4*>(bp + u);
                                const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&bv);
                                #pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const float2 f = __bfloat1622float2(h[i]);
                                    v[u + 2 * i] += f.x;
                                    v[u + 2 * i + 1] += f.y;
                                }
                            }
                        }
                        stage_row_bf16(stg, lane, v);
                        __syncwarp();
                        store_tile_bf16(stg, lane, (__nv_bfloat16*)p.out0, grow0, valid, N, col0);
                        __syncwarp();
                        if (EPI == (int)Epi::BiasGelu) {
                            #pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = gelu_fast(v[i]);
                            stage_row_bf16(stg, lane, v);
                            __syncwarp();
                            store_tile_bf16(stg, lane, (__nv_bfloat16*)p.out1, grow0, valid, N, col0);
                            __syncwarp();
                        }
                    } else if (EPI == (int)Epi::GeluGrad) {
                        uint4 hcur[4];
                        #pragma unroll
                        for (int u = 0; u < 4; ++u) hcur[u] = hnext[u];
                        if (ch < 3 && col0 + 32 < p.N) {
                            #pragma unroll
                            for (int u = 0; u < 4; ++u)
                                hnext[u] = row_ok ? __ldg(reinterpret_cast<const uint4*>(
                                                        (const __nv_bfloat16*)p.aux + grow_lane * N +
                                                        col0 + 32 + u * 8))
                                                  : make_uint4(0, 0, 0, 0);
                        }
                        #pragma unroll
                        for (int cc = 0; cc < 4; ++cc) {
                            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&hcur[cc]);
                            #pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float2 f = __bfloat1622float2(h[i]);
                                v[cc * 8 + 2 * i] *= gelu_grad_fast(f.x);
                                v[cc * 8 + 2 * i + 1] *= gelu_grad_fast(f.y);
                            }
                        }
                        stage_row_bf16(stg, lane, v);
                        __syncwarp();
                        store_tile_bf16(stg, lane, (__nv_bfloat16*)p.out0, grow0, valid, N, col0);
                        __syncwarp();
                    } else {  // Plain
                        stage_row_bf16(stg, lane, v);
                        __syncwarp();
                        store_tile_bf16(stg, lane, (__nv_bfloat16*)p.out0, grow0, valid, N, col0);
                        __syncwarp();
                    }
                } else {
                    // fp32 weight gradient, 16 columns (64 B per row) at a time
                    const int m0 = ti.mt * BM + q * 32;
                    const int valid = p.M - m0;
                    #pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        #pragma unroll
                        for (int cc = 0; cc < 4; ++cc)
                            *reinterpret_cast<float4*>(stg + stg_off(lane, cc)) =
                                make_float4(v[hh * 16 + cc * 4], v[hh * 16 + cc * 4 + 1],
                                            v[hh * 16 + cc * 4 + 2], v[hh * 16 + cc * 4 + 3]);
                        __syncwarp();
                        #pragma unroll
                        for (int it = 0; it < 4; ++it) {
                            const int rr = it * 8 + (lane >> 2), cc = lane & 3;
                            if (rr < valid) {
                                float4 o = *reinterpret_cast<const float4*>(stg + stg_off(rr, cc));
                                float4* dst = reinterpret_cast<float4*>(
                                    p.outf + ((int64_t)ti.e * p.M + m0 + rr) * p.N + col0 +
                                    hh * 16 + cc * 4);
                                if (p.accumulate) {
                                    const float4 old = *dst;
                                    o.x += old.x; o.y += old.y; o.z += old.z; o.w += old.w;
                                }
                                *dst = o;
                            }
                        }
                        __syncwarp();
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&c.tempty[acc]));
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
    }

    // ---- teardown ------------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---- host side ---------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// bf16 tensor map, 128-byte swizzle, zero fill outside the tensor.
// dims/box innermost first; strides in bytes for dims 1.. .
bool make_map(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gd[3], gs[2];
    cuuint32_t bx[3], es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) { gd[i] = dims[i]; bx[i] = box[i]; }
    for (int i = 0; i < rank - 1; ++i) gs[i] = strides[i];
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(ptr),
                    gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <bool VAR_K, bool A_MN, bool B_MN, int EPI>
cudaError_t launch_tc(const CUtensorMap& a, const CUtensorMap& b, const TcParams& p,
                      int64_t tiles_upper, cudaStream_t st) {
    auto kern = gemm_tc_kernel<VAR_K, A_MN, B_MN, EPI>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int64_t sms = device_sm_count();
    const unsigned grid = (unsigned)(tiles_upper < sms ? (tiles_upper > 0 ? tiles_upper : 1) : sms);
    kern<<<grid, THREADS, SMEM_BYTES, st>>>(a, b, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_varm_tc(const GemmVarM& g, int32_t* status, cudaStream_t st) {
    if (g.E > MAX_E || g.N % 64 || g.K % 64) return cudaErrorInvalidValue;
    CUtensorMap ma, mb;
    {
        const uint64_t dims[2] = {(uint64_t)g.K, (uint64_t)g.P};
        const uint64_t strides[1] = {(uint64_t)g.K * 2};
        const uint32_t box[2] = {BK, BM};
        if (!make_map(&ma, g.act, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    if (g.weight_kmajor) {
        const uint64_t dims[3] = {(uint64_t)g.K, (uint64_t)g.N, (uint64_t)g.E};
        const uint64_t strides[2] = {(uint64_t)g.K * 2, (uint64_t)g.N * g.K * 2};
        const uint32_t box[3] = {BK, BN, 1};
        if (!make_map(&mb, g.weight, 3, dims, strides, box)) return cudaErrorInvalidValue;
    } else {
        const uint64_t dims[3] = {(uint64_t)g.N, (uint64_t)g.K, (uint64_t)g.E};
        const uint64_t strides[2] = {(uint64_t)g.N * 2, (uint64_t)g.K * g.N * 2};
        const uint32_t box[3] = {64, BK, 1};
        if (!make_map(&mb, g.weight, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    TcParams p{};
    p.E = g.E; p.N = g.N; p.K = g.K; p.M = 0; p.P = g.P;
    p.offsets = g.offsets; p.bias = g.bias; p.aux = g.aux; p.out0 = g.out0; p.out1 = g.out1;
    p.outf = nullptr; p.accumulate = 0; p.status = status; p.limit_ns = wait_limit_ns();
    const int64_t NT = (g.N + BN - 1) / BN;
    const int64_t upper = ((g.P + BM - 1) / BM + g.E) * NT;
    switch (g.epi) {
        case Epi::BiasGelu:
            if (!g.weight_kmajor) return cudaErrorInvalidValue;
            return launch_tc<false, false, false, (int)Epi::BiasGelu>(ma, mb, p, upper, st);
        case Epi::Bias:
            if (!g.weight_kmajor) return cudaErrorInvalidValue;
            return launch_tc<false, false, false, (int)Epi::Bias>(ma, mb, p, upper, st);
        case Epi::GeluGrad:
            if (g.weight_kmajor) return cudaErrorInvalidValue;
            return launch_tc<false, false, true, (int)Epi::GeluGrad>(ma, mb, p, upper, st);
        case Epi::Plain:
            if (g.weight_kmajor) return cudaErrorInvalidValue;
            return launch_tc<false, false, true, (int)Epi::Plain>(ma, mb, p, upper, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_vark_tc(const GemmVarK& g, int32_t* status, cudaStream_t st) {
    if (g.E > MAX_E || g.M % 64 || g.N % 64) return cudaErrorInvalidValue;
    CUtensorMap ma, mb;
    {
        const uint64_t dims[2] = {(uint64_t)g.M, (uint64_t)g.P};
        const uint64_t strides[1] = {(uint64_t)g.M * 2};
        const uint32_t box[2] = {64, BK};
        if (!make_map(&ma, g.act_a, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[2] = {(uint64_t)g.N, (uint64_t)g.P};
        const uint64_t strides[1] = {(uint64_t)g.N * 2};
        const uint32_t box[2] = {64, BK};
        if (!make_map(&mb, g.act_b, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    TcParams p{};
    p.E = g.E; p.M = g.M; p.N = g.N; p.K = 0; p.P = g.P;
    p.offsets = g.offsets; p.outf = g.out; p.accumulate = g.accumulate;
    p.status = status; p.limit_ns = wait_limit_ns();
    const int64_t upper = (int64_t)g.E * ((g.M + BM - 1) / BM) * ((g.N + BN - 1) / BN);
    return launch_tc<true, true, true, (int)Epi::Plain>(ma, mb, p, upper, st);
}

}  // namespace moe
