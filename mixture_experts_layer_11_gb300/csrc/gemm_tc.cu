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
//   VarK (weight gradient): C_e[M, N] (+)= act_a[rows_e, M]^T act_b[rows_e, N];
//     the reduction runs over the expert's rows, which are its segments in one
//     or more dispatch chunks (chunk s holds the rows seg_base[s] + offsets of
//     that chunk), walked segment after segment.  Rows past a segment's end
//     in its last K block are zeroed in shared memory before the MMA reads them.
//     On a CTA pair each CTA zeroes its own operands: for a segment's last K
//     block the odd CTA's loads complete on its own stage barrier, its
//     otherwise idle MMA warp zeroes the tail and then arrives on the even
//     CTA's stage barrier (every other stage goes straight to the even CTA).
//
// Two CTA shapes (template PAIR):
//   1 CTA: tile 128 x 256, tcgen05.mma.cta_group::1 (M 128, N 256, K 16);
//     stages of 48 KB (A 128x64, B 256x64).
//   CTA pair (cluster of 2): tile 256 x 256, tcgen05.mma.cta_group::2 (M 256,
//     N 256, K 16) issued by the even CTA; each CTA holds its 128 rows of A
//     and 128 columns of B, so a stage is 32 KB.  Both CTAs' TMA loads
//     complete on the even CTA's stage barrier; MMA completion is multicast to
//     both CTAs' barriers; each CTA drains its own TMEM rows.
//
// CTA = 2 + 8 or 16 warps: warp 0 issues TMA loads, warp 1 issues the MMAs
// into one of two TMEM accumulators (2 x 256 fp32 columns), the other warps
// drain the other accumulator (tcgen05.ld) and apply the fused epilogue (bias,
// GELU, GELU', fp32 accumulate).  bf16 results go through a swizzled shared
// staging buffer and out by TMA tensor stores; fp32 weight gradients by
// coalesced stores.  Every wait is bounded; on expiry the CTA records
// MOE_ERR_TIMEOUT, waits for its own copies and MMAs in flight, frees TMEM
// and exits.
#include <cudaTypedefs.h>
#include <limits.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int BM = 128;            // rows per CTA (TMEM lanes)
constexpr int BN = 256;            // tile columns (MMA N)
constexpr int BK = 64;             // K per stage: one 128-byte swizzle row of bf16
constexpr int SLAB_BYTES = 64 * BK * 2;    // one 64-wide MN slab of BK rows
constexpr int TMEM_COLS = 2 * BN;
constexpr int MAX_E = 256;
// Weight-gradient split: a (m-tile, n-tile) of an expert whose reduction spans
// many K blocks is cut into parts of at most kb_part K blocks, so that a few
// long tiles do not leave most CTA pairs idle at the end of the launch.  The
// parts aim at kSplitUnitsPerPair work units per pair and have at least
// kKbPartMin K blocks (about 0.07 ms of MMAs per pair), so that the partial
// tiles' extra traffic stays small beside their MMA time.  Short parts also
// keep the pairs that read the same rows of an expert (its tiles of one part)
// close together in K, so that those rows are reused in L2: on the
// long-context weight gradients, parts of 256 K blocks instead of 1024 read
// less from DRAM and took 4% less time.
constexpr int kKbPartMin = 256;
constexpr int kSplitUnitsPerPair = 128;
// One-segment weight-gradient calls over at most this many rows take the lean
// kernel (no segment walk, no split).
constexpr int64_t kLeanMaxRows = 512 * 64;

template <bool PAIR> struct Shape {
    static constexpr int CTAS = PAIR ? 2 : 1;
    static constexpr int TILE_M = BM * CTAS;          // rows of one (pair) tile
    static constexpr int BN_CTA = BN / CTAS;          // B columns this CTA holds
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN_CTA * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
};

// Operand pipeline depth and epilogue staging, under the 227 KB per-CTA limit.
// The operand loads mostly come from L2 or DRAM with a latency of a few
// microseconds under load, so the stages take whatever the epilogue leaves:
// - bias + GELU stages G and A (one 32-row chunk each per warp, 32 KB) and
//   holds the fp32 bias (4 KB): 5 pair stages;
// - the one-output bf16 epilogues stage one chunk per warp (16 KB; the TMA
//   store of a chunk has read it long before the next chunk is written):
//   6 pair stages, or 5 for the GELU' scaling epilogue, which also receives
//   its saved GELU'(h) by TMA into a two-chunk ring per warp (32 KB);
// - the fp32 weight-gradient epilogue stages one chunk per warp (16 KB), next
//   to the all-ones slab (8 KB): 6 pair stages;
// - the router-logit epilogue stages 32 x 32 fp32 per warp (32 KB): 5.
// Single CTAs (48 KB stages) get 3, or 4 for the weight gradients.
template <bool PAIR, bool VAR_K, int EPI> struct Pipe {
    static constexpr bool AUX = !VAR_K && EPI == (int)Epi::ScaleAux;
    static constexpr bool GELU = !VAR_K && EPI == (int)Epi::BiasGelu;
    static constexpr bool HAS_BIAS = !VAR_K && (EPI == (int)Epi::BiasGelu || EPI == (int)Epi::Bias);
    static constexpr bool LOGITS = !VAR_K && EPI == (int)Epi::Logits;
    static constexpr int STAGING = (GELU || LOGITS) ? 32 * 1024 : 16 * 1024;
    static constexpr int BIAS = HAS_BIAS ? 4 * 1024 : 0;  // fp32 bias of each warp's columns
    static constexpr int AUXBUF = AUX ? 32 * 1024 : 0;    // GELU'(h) ring, 2 x 1 KB per warp
    static constexpr int ONES = VAR_K ? 64 * BK * 2 : 0;  // all-ones MN-major B slab (row sums)
    static constexpr int STAGES = PAIR ? ((GELU || AUX || LOGITS) ? 5 : 6) : (VAR_K ? 4 : 3);
};

// Epilogue shape.  The epilogue warps drain a 128 x 256 accumulator, each
// warp the TMEM lane quarter it may access (warp % 4) and a range of columns.
// The GELU epilogues (instruction-heavy: a short-K tile's drain takes longer
// than its MMAs) get 16 warps, 64 columns each, in 16-column chunks (register
// budget of 576 threads); the others 8 warps, 128 columns each, in 32-column
// chunks.
template <int EPI, bool VAR_K> struct EpiShape {
    static constexpr bool WIDE = !VAR_K && (EPI == (int)Epi::BiasGelu || EPI == (int)Epi::ScaleAux);
    static constexpr int WARPS = WIDE ? 16 : 8;
    static constexpr int CW = WIDE ? 16 : 32;              // columns per chunk
    static constexpr int COLS = BN / (WARPS / 4);          // columns per warp
    static constexpr int NCH = COLS / CW;                  // chunks per warp
    static constexpr int CHUNK_BYTES = 32 * CW * 2;        // one staged bf16 chunk
    // + the tail-relay warp of the weight gradients (see the kernel)
    static constexpr int THREADS = 32 * (2 + WARPS + (VAR_K ? 1 : 0));
};

template <int N> struct U4s { uint4 u[N]; };
template <bool B> struct BoolTag { static constexpr bool value = B; };

struct TcParams {
    int E, M, N, K;          // VarM: N, K (M unused); VarK: M, N (K = segment)
    int64_t P;
    const int32_t* offsets;
    const void* bias;
    const void* aux;
    void* out0;
    void* out1;
    float* outf;
    float* cpart;            // ScaleAux: column-sum partial rows [rows][N], or null
    float* bsum;             // VarK: per-expert row sums of act_a [E][M], or null
    int accumulate;
    int32_t* status;
    uint64_t limit_ns;
    // Test hook (MOE_DEBUG_GEMM_WITHHOLD): the even CTA's producer stops before
    // issuing K block withhold_kb of work unit withhold_unit (neither its
    // expect_tx nor its loads), so the MMA warp's bounded wait on that stage
    // runs out and the CTA takes its timeout teardown.  -1: off.
    int withhold_unit, withhold_kb;
    // VarK: expert e's rows in dispatch chunk s are
    // [seg_base[s] + offsets[s*ostride + e], seg_base[s] + offsets[s*ostride + e + 1]).
    int nseg, ostride;
    int64_t seg_base[kMaxWgradChunks];
    // VarK split: slots for partial tiles in the scratch map (0: no split),
    // and the number of CTA pairs of the launch (the split's unit target)
    int64_t part_cap;
    int split_units;
    float* bpart;            // VarK split: row sums of all-ones tiles of parts > 0
    // Row gather (the permute fused into the operand loads), or null: row r of
    // the expert-sorted operand (VarM: A; VarK: B) is row
    // gbase[s] + gather[s * gstride + r - seg_base[s]] / gk of the tensor map's
    // source (s = 0 for VarM), loaded four rows at a time by tile::gather4.
    const int32_t* gather;
    int gk;
    int64_t gstride;
    int64_t gbase[kMaxWgradChunks];
};

// K blocks per part of the split weight-gradient tiles (INT_MAX: no split):
// the smallest power of two >= kKbPartMin giving about kSplitUnitsPerPair
// units per pair, doubled until the partial tiles fit in `cap` slots.  kbs[e]
// is expert e's K-block count; MT x NT real tiles per expert.  Every kernel
// that needs the split computes it with this same function.
__device__ __forceinline__ int vark_kb_part(const int* kbs, int E, int MT, int NT, int nunits,
                                            int64_t cap) {
    if (cap <= 0) return INT_MAX;
    int64_t tot = 0;
    int kmax = 0;
    for (int e = 0; e < E; ++e) {
        tot += kbs[e];
        kmax = kbs[e] > kmax ? kbs[e] : kmax;
    }
    tot *= (int64_t)MT * NT;
    const int64_t want = tot / ((int64_t)kSplitUnitsPerPair * (nunits > 0 ? nunits : 1));
    int kp = kKbPartMin;
    while (kp < want && kp < kmax) kp *= 2;
    while (kp < kmax) {
        int64_t slots = 0;
        for (int e = 0; e < E; ++e)
            if (kbs[e] > kp) slots += (int64_t)((kbs[e] + kp - 1) / kp - 1) * MT * NT;
        if (slots <= cap) break;
        kp *= 2;
    }
    return kp >= kmax ? INT_MAX : kp;
}
__device__ __forceinline__ int vark_nsplit(int kb, int kp) {
    return kb > kp ? (kb + kp - 1) / kp : 1;
}

template <int STAGES> struct Ctrl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tail[STAGES];       // VarK, even / single CTA: a segment's last K block lands here
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint64_t gbar[16][2];        // ScaleAux: GELU'(h) ring, per epilogue warp
    uint32_t tmem_base;
    int abort_flag;
    int nactive;
    int off[MAX_E + 1];
    int tile_start[MAX_E + 1];   // VarM: first tile of each expert; VarK: K blocks of each
    int order[MAX_E];            // VarK: experts by descending row count
    int ustart[MAX_E + 1];       // VarK: first unit of each position of `order`
    int sbase[MAX_E];            // VarK: first scratch slot of each expert's split parts
    int kb_part;                 // VarK: K blocks per split part (INT_MAX: none)
};

template <bool PAIR, bool VAR_K, int EPI>
constexpr size_t smem_bytes() {
    using S = Shape<PAIR>;
    using PP = Pipe<PAIR, VAR_K, EPI>;
    return 1024 + (size_t)PP::STAGES * S::STAGE_BYTES + (size_t)PP::STAGING + (size_t)PP::BIAS +
           (size_t)PP::AUXBUF + (size_t)PP::ONES + sizeof(Ctrl<PP::STAGES>);
}

struct Tile {
    int e, mt, nt, num_kb;
    int row0;     // VarM: first row of this CTA's part; VarK: unused
    int rows;     // VarM: valid rows of this CTA's part (may be <= 0); VarK: the expert's rows
    bool ones;    // VarK: the extra tile against the all-ones B (row sums of act_a)
    int kb0;      // VarK: first K block of this part
    int slot;     // VarK: scratch slot of a split part > 0, else -1 (written to the output)
    int bslot;    // VarK: scratch row-sum slot of an all-ones tile of a part > 0, else -1
};

// VarK: walks an expert's K blocks segment after segment (dispatch chunks with
// rows for the expert), one BK-row block at a time.
struct SegCursor {
    int seg, kl, rows;   // current segment, K block inside it, the segment's rows
    int row0;            // first row of the segment (global row coordinate)
    const int* soff;     // one segment: its offsets in shared memory (else null)
    __device__ __forceinline__ void next_segment(const TcParams& p, int e) {
        for (++seg; seg < p.nseg; ++seg) {
            int a, b;
            if (soff) {
                a = soff[e];
                b = soff[e + 1];
            } else {
                const int32_t* o = p.offsets + (int64_t)seg * p.ostride;
                a = __ldg(o + e);
                b = __ldg(o + e + 1);
            }
            if (b > a) {
                rows = b - a;
                row0 = (int)(p.seg_base[seg] + a);
                kl = 0;
                return;
            }
        }
        rows = 0;
        row0 = 0;
        kl = 0;
    }
    // position at K block kb0 of the expert's blocks, counted over its segments;
    // off: the per-expert row prefix in shared memory, which for one segment
    // (seg_base 0) is that segment's offsets
    __device__ __forceinline__ void start(const TcParams& p, int e, int kb0, const int* off) {
        soff = p.nseg == 1 && p.seg_base[0] == 0 ? off : nullptr;
        seg = -1;
        next_segment(p, e);
        while (seg < p.nseg) {
            const int nkb = (rows + BK - 1) / BK;
            if (kb0 < nkb) {
                kl = kb0;
                return;
            }
            kb0 -= nkb;
            next_segment(p, e);
        }
    }
    __device__ __forceinline__ void advance(const TcParams& p, int e) {
        if (++kl * BK >= rows) next_segment(p, e);
    }
    __device__ __forceinline__ int row() const { return row0 + kl * BK; }
    __device__ __forceinline__ int valid() const { return rows - kl * BK; }   // rows of this block
};

template <bool VAR_K, bool PAIR, bool MULTI, typename C>
__device__ __forceinline__ Tile get_tile(const C& c, const TcParams& p, int t, int& ecur,
                                         int rank) {
    using S = Shape<PAIR>;
    Tile ti;
    const int NT = (p.N + BN - 1) / BN;
    if (!VAR_K) {
        while (c.tile_start[ecur + 1] <= t) ++ecur;
        const int local = t - c.tile_start[ecur];
        ti.e = ecur;
        ti.mt = local / NT;
        ti.nt = local % NT;
        ti.row0 = c.off[ecur] + ti.mt * S::TILE_M + rank * BM;
        ti.rows = min(BM, c.off[ecur + 1] - ti.row0);
        ti.num_kb = p.K / BK;
        ti.ones = false;
        ti.kb0 = 0;
        ti.slot = -1;
        ti.bslot = -1;
    } else if (!MULTI) {
        // one segment, no split: an expert's MT x (NT + all-ones) units, m-tile
        // groups each followed by its all-ones tile
        const int NTX = NT + (p.bsum ? 1 : 0);
        const int MT = (p.M + S::TILE_M - 1) / S::TILE_M;
        const int per = MT * NTX;
        ti.e = c.order[t / per];
        const int local = t % per;
        ti.mt = local / NTX;
        ti.nt = local % NTX;
        ti.ones = ti.nt == NT;
        ti.row0 = c.off[ti.e];
        ti.rows = c.off[ti.e + 1] - ti.row0;
        ti.num_kb = (ti.rows + BK - 1) / BK;
        ti.kb0 = 0;
        ti.slot = -1;
        ti.bslot = -1;
    } else {
        // An expert's units, part after part of its split K range (the units of
        // one part run at about the same time and share operand rows in L2):
        // its MT x NT tiles, ordered so that neighbouring units share the
        // operand with more slabs (m-tile groups when MT >= NT, each followed by
        // its all-ones tile; else n-tile groups, the all-ones tiles last), plus
        // an all-ones tile per m-tile when row sums are wanted.  ecur: position
        // in c.order.
        const int MT = (p.M + S::TILE_M - 1) / S::TILE_M;
        const int NTX = NT + (p.bsum ? 1 : 0);
        while (c.ustart[ecur + 1] <= t) ++ecur;
        ti.e = c.order[ecur];
        const int local = t - c.ustart[ecur];
        const int kb = c.tile_start[ti.e];   // K blocks over all of the expert's segments
        const int nparts = vark_nsplit(kb, c.kb_part);
        const int part = local / (MT * NTX);
        const int rem = local - part * MT * NTX;
        if (MT >= NT) {
            ti.mt = rem / NTX;
            ti.nt = rem % NTX;
        } else if (rem < MT * NT) {
            ti.nt = rem / MT;
            ti.mt = rem % MT;
        } else {
            ti.mt = rem - MT * NT;
            ti.nt = NT;
        }
        ti.ones = ti.nt == NT;
        const int ks = nparts > 1 ? (kb + nparts - 1) / nparts : kb;
        ti.kb0 = part * ks;
        ti.num_kb = min(ks, kb - ti.kb0);
        ti.slot = (part > 0 && !ti.ones)
                      ? c.sbase[ti.e] + (part - 1) * MT * NT + ti.mt * NT + ti.nt : -1;
        ti.bslot = (part > 0 && ti.ones) ? c.sbase[ti.e] / NT + (part - 1) * MT + ti.mt : -1;
        ti.row0 = 0;
        ti.rows = c.off[ti.e + 1] - c.off[ti.e];
    }
    return ti;
}

template <typename C>
__device__ __forceinline__ void raise_abort(C& c, const TcParams& p) {
    *(volatile int*)&c.abort_flag = 1;
    report(p.status, MOE_ERR_TIMEOUT);
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Shared::cluster address of the variable at shared address `a` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_rank(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// Arrivals on a barrier addressed through the cluster window (possibly in the
// peer CTA).  Default (CTA-scope) semantics: what they publish is ordered by
// other means (TMA completion bytes, tcgen05 fences), and a cluster-scope
// release here would wait on the thread's outstanding copies every stage.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cl_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cl_addr) : "memory");
}
// Arrive with release semantics at cluster scope: this thread's earlier
// shared-memory writes are visible to the peer CTA once the phase completes.
__device__ __forceinline__ void mbar_arrive_cluster_release(uint32_t cl_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cl_addr)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t cl_addr, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cluster.b64 _, [%0], %1;" ::"r"(cl_addr),
                 "r"(bytes)
                 : "memory");
}
// TMA loads whose completion is signalled on the pair's even CTA (cl_bar is a
// shared::cluster address).
__device__ __forceinline__ void tma2_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t cl_bar,
                                             int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(map), "r"(cl_bar), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void tma2_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t cl_bar,
                                             int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(map), "r"(cl_bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
// Four rows (row0..row3, one-row boxes of the map) at column c0, written to
// shared memory one after the other as a four-row box (the map's swizzle
// applies by shared address, as for a tiled box).
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, const int (&rows)[4]) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
        "l"(map), "r"(bar), "r"(c0), "r"(rows[0]), "r"(rows[1]), "r"(rows[2]), "r"(rows[3])
        : "memory");
}
// The same, completing on the pair's even CTA (cl_bar: shared::cluster address).
__device__ __forceinline__ void tma2_gather4(uint32_t dst, const CUtensorMap* map,
                                             uint32_t cl_bar, int32_t c0, const int (&rows)[4]) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile::gather4"
        ".mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
        "l"(map), "r"(cl_bar), "r"(c0), "r"(rows[0]), "r"(rows[1]), "r"(rows[2]), "r"(rows[3])
        : "memory");
}
__device__ __forceinline__ void tma2_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t cl_bar,
                                             int32_t c0, int32_t c1, int32_t c2, int32_t c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(map), "r"(cl_bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc2(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_mma2_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on the barrier at this shared offset in both CTAs of the pair once
// every tcgen05 op issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit2_both(uint32_t bar) {
    const uint16_t mask = 3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}
__device__ __forceinline__ void tc_commit2_local(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

// ---- epilogue helpers: staging of 32 rows x CW bf16 (CW*2 bytes per row),
// 16-byte chunks XOR-swizzled so that the per-row writes (one row per
// thread) and the coalesced reads are both free of bank conflicts.  The
// pattern is the TMA's: chunk index XOR address bit 7 for 32-byte rows
// (SWIZZLE_32B), XOR address bits 8:7 for 64-byte rows (SWIZZLE_64B).
template <int CW>
__device__ __forceinline__ uint32_t stg_off(int row, int ch) {
    if (CW == 32) return (uint32_t)(row * 64 + ((ch ^ ((row >> 1) & 3)) << 4));
    return (uint32_t)(row * 32 + ((ch ^ ((row >> 2) & 1)) << 4));
}

__device__ __forceinline__ uint4 pack8_bf16(const float* v) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
    #pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    return u;
}

// this thread's row (lane) of CW bf16 values, packed -> staging
template <int CW>
__device__ __forceinline__ void stage_row_packed(uint8_t* stg, int lane, const uint4* pk) {
    #pragma unroll
    for (int ch = 0; ch < CW / 8; ++ch)
        *reinterpret_cast<uint4*>(stg + stg_off<CW>(lane, ch)) = pk[ch];
}

// staging (32 rows x CW bf16) -> global rows row0.., columns col0.., ld = N
template <int CW>
__device__ __forceinline__ void store_tile_bf16(const uint8_t* stg, int lane, __nv_bfloat16* out,
                                                int64_t row0, int valid_rows, int64_t ld,
                                                int col0) {
    constexpr int CPR = CW / 8;                 // 16-byte chunks per row
    #pragma unroll
    for (int it = 0; it < CPR; ++it) {
        const int rr = it * (32 / CPR) + lane / CPR, ch = lane % CPR;
        if (rr < valid_rows) {
            const uint4 v = *reinterpret_cast<const uint4*>(stg + stg_off<CW>(rr, ch));
            *reinterpret_cast<uint4*>(out + (row0 + rr) * ld + col0 + ch * 8) = v;
        }
    }
}

// TMA tensor store of a staged box (shared -> global), tracked by this
// thread's bulk async-groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t c0,
                                             int32_t c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(map), "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}
// The same for a 3-D box, stored as is or added element by element to what
// global memory holds (fp32 weight gradients).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int32_t c0,
                                             int32_t c1, int32_t c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
                 ::"l"(map), "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int32_t c0,
                                                  int32_t c1, int32_t c2) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
        " [%0, {%2, %3, %4}], [%1];" ::"l"(map), "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// until at most N committed groups still read their shared-memory source
template <int N> __device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// until every committed group has completed its writes
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

template <int CW>
__device__ __forceinline__ void tmem_ld_cw(uint32_t taddr, float (&v)[CW]) {
    if constexpr (CW == 32) tmem_ld32(taddr, v);
    else tmem_ld16(taddr, v);
}

template <bool VAR_K, bool A_MN, bool B_MN, int EPI, bool PAIR, bool MULTI>
__global__ void __launch_bounds__(EpiShape<EPI, VAR_K>::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mapA,
                   const __grid_constant__ CUtensorMap mapB,
                   const __grid_constant__ CUtensorMap mapO0,
                   const __grid_constant__ CUtensorMap mapO1, const TcParams p) {
    using S = Shape<PAIR>;
    using ES = EpiShape<EPI, VAR_K>;
    using PP = Pipe<PAIR, VAR_K, EPI>;
    constexpr int THREADS = ES::THREADS;
    constexpr int CW = ES::CW;
    constexpr int STAGES = PP::STAGES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* staging_base = base + (size_t)STAGES * S::STAGE_BYTES;
    using CtrlT = Ctrl<STAGES>;
    float* bias_base = reinterpret_cast<float*>(staging_base + (size_t)PP::STAGING);
    uint8_t* aux_base = staging_base + (size_t)PP::STAGING + (size_t)PP::BIAS;
    uint8_t* ones_base = aux_base + (size_t)PP::AUXBUF;
    CtrlT& c = *reinterpret_cast<CtrlT*>(ones_base + (size_t)PP::ONES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;
    const int NT = (p.N + BN - 1) / BN;
    const int rank = PAIR ? (int)cluster_rank() : 0;
    const bool leader = rank == 0;
    const int unit0 = blockIdx.x / S::CTAS;          // this (pair of) CTA's first work unit
    const int nunits = gridDim.x / S::CTAS;

    // ---- set-up: barriers, TMEM, tile list ------------------------------------
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // even CTA: its own producer + the odd CTA (remote expect_tx, or the
            // weight-gradient relay); odd CTA of a weight-gradient pair: its producer
            mbar_init(smem_u32(&c.full[s]), leader ? S::CTAS : 1);
            mbar_init(smem_u32(&c.empty[s]), 1);
            mbar_init(smem_u32(&c.tail[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&c.tfull[b]), 1);
            mbar_init(smem_u32(&c.tempty[b]), ES::WARPS * S::CTAS);
        }
        mbar_init(smem_u32(&c.drain), 1);
        if (PP::AUX)
            for (int w = 0; w < ES::WARPS; ++w) {
                mbar_init(smem_u32(&c.gbar[w][0]), 1);
                mbar_init(smem_u32(&c.gbar[w][1]), 1);
            }
        c.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc2(smem_u32(&c.tmem_base), TMEM_COLS);
            tmem_relinquish2();
        } else {
            tmem_alloc(smem_u32(&c.tmem_base), TMEM_COLS);
            tmem_relinquish();
        }
    }
    if (!VAR_K || !MULTI) {
        for (int i = threadIdx.x; i <= E; i += THREADS)
            c.off[i] = p.offsets ? p.offsets[i] : (i == 0 ? 0 : (int)p.P);   // null: rows [0, P)
    } else {
        // per expert: rows and K blocks summed over its segments; c.off becomes
        // the prefix sum of the rows (so that off[e+1] - off[e] is expert e's
        // total), c.tile_start[e] its K-block count
        for (int e = threadIdx.x; e < E; e += THREADS) {
            int tot = 0, kbs = 0;
            for (int sg = 0; sg < p.nseg; ++sg) {
                const int32_t* o = p.offsets + (int64_t)sg * p.ostride;
                const int n = o[e + 1] - o[e];
                tot += n;
                kbs += (n + BK - 1) / BK;
            }
            c.off[e + 1] = tot;
            c.tile_start[e] = kbs;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            c.off[0] = 0;
            for (int e = 0; e < E; ++e) c.off[e + 1] += c.off[e];
        }
    }
    if (VAR_K && p.bsum) {
        // bf16 ones for the row-sum tile's B operand, read by the tensor core
        for (int i = threadIdx.x; i < PP::ONES / 16; i += THREADS)
            reinterpret_cast<uint4*>(ones_base)[i] =
                make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        fence_proxy_async_smem();
    }
    __syncthreads();
    if (!VAR_K) {
        if (threadIdx.x == 0) {
            int acc = 0;
            for (int e = 0; e < E; ++e) {
                c.tile_start[e] = acc;
                acc += ((c.off[e + 1] - c.off[e] + S::TILE_M - 1) / S::TILE_M) * NT;
            }
            c.tile_start[E] = acc;
            c.nactive = acc;   // number of work units
        }
    } else {
        // Unit order: without accumulation the experts without tokens come first
        // (their units only write zero tiles: the MMA warp skips them and the
        // epilogue writes them while the first real tiles are computed), then
        // the others by descending row count (longest processing time first).
        for (int e = threadIdx.x; e < E; e += THREADS) {
            const int n = c.off[e + 1] - c.off[e];
            const int kn = (n == 0 && !p.accumulate) ? INT_MAX : n;
            int r = 0;
            for (int q = 0; q < E; ++q) {
                const int m = c.off[q + 1] - c.off[q];
                const int km = (m == 0 && !p.accumulate) ? INT_MAX : m;
                r += (km > kn) || (km == kn && q < e);
            }
            c.order[r] = e;
        }
        if (!MULTI && threadIdx.x == 0) {
            int act = 0;
            for (int e = 0; e < E; ++e) act += (c.off[e + 1] - c.off[e]) > 0;
            const int MT = (p.M + S::TILE_M - 1) / S::TILE_M;
            const int NTX = NT + (p.bsum ? 1 : 0);
            c.nactive = (p.accumulate ? act : E) * MT * NTX;  // number of work units
        }
        if (MULTI) __syncthreads();
        if (MULTI && threadIdx.x == 0) {
            int act = 0;
            for (int e = 0; e < E; ++e) act += (c.off[e + 1] - c.off[e]) > 0;
            const int MT = (p.M + S::TILE_M - 1) / S::TILE_M;
            const int ONES = p.bsum ? 1 : 0;
            const int kp = vark_kb_part(c.tile_start, E, MT, NT, p.split_units, p.part_cap);
            c.kb_part = kp;
            int slots = 0;
            for (int e = 0; e < E; ++e) {
                c.sbase[e] = slots;
                slots += (vark_nsplit(c.tile_start[e], kp) - 1) * MT * NT;
            }
            int u = 0;
            for (int r = 0; r < E; ++r) {
                c.ustart[r] = u;
                u += MT * (NT + ONES) * vark_nsplit(c.tile_start[c.order[r]], kp);
            }
            c.ustart[E] = u;
            // number of work units: without accumulation every expert (the empty
            // ones write zeros), else the experts with rows (first in the order)
            c.nactive = p.accumulate ? c.ustart[act] : u;
        }
    }
    tc_fence_before();
    if (PAIR) cluster_sync(); else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = c.tmem_base;
    const int num_units = c.nactive;

    if (warp == 0) {
        // ---- TMA producer ---------------------------------------------------------
        // Lane 0 waits for free stages, arms the barriers and issues the box
        // loads.  With a row gather (the permute fused into the loads; GAT) the
        // whole warp walks the tiles and every lane also issues tile::gather4
        // loads of four source rows each: VarM, the CTA's 128 A rows per K block
        // (the rows are the tile's, fetched once per tile); VarK, the BK rows of
        // every B slab of a K block (fetched one K block ahead).
        if (lane == 0) {
            tma_prefetch_map(&mapA);
            tma_prefetch_map(&mapB);
        }
        auto producer = [&](auto gather_tag) {
            constexpr bool gat = decltype(gather_tag)::value;
            // VarK gather: (slab, four-row group) assignments per lane
            constexpr int kGatherJ = (S::B_BYTES / SLAB_BYTES) * (BK / 4) / 32;
            int stage = 0, ecur = 0;
            uint32_t phase = 0;
            // per stage, the parity of the last phase this CTA's copies count on
            // (of full[], or of tail[] for a segment's last K block), else -1
            int issued_parity[STAGES], issued_tail[STAGES];
            for (int s = 0; s < STAGES; ++s) issued_parity[s] = issued_tail[s] = -1;
            uint32_t tail_phase = 0;   // bit s: parity of tail[s]'s next phase
            bool ok = true;
            // source row of gathered operand row r of segment seg (r clamped to the
            // segment's last row: rows past it are never used, or zeroed by the relay)
            auto gsrc = [&](int seg, int r, int rlast) -> int {
                const int rr = r < rlast ? r : rlast;
                const int32_t v =
                    __ldg(p.gather + (int64_t)seg * p.gstride + (rr - p.seg_base[seg]));
                return (int)(p.gbase[seg] + v / p.gk);
            };
            for (int t = unit0; t < num_units && ok; t += nunits) {
                const Tile ti = get_tile<VAR_K, PAIR, MULTI>(c, p, t, ecur, rank);
                SegCursor cur;
                if (VAR_K && MULTI) cur.start(p, ti.e, ti.kb0, c.off);
                int arow[4];                 // VarM gather: this lane's four A rows
                int brow[kGatherJ][4];       // VarK gather: this lane's B rows, next K block
                if (gat && !VAR_K) {
                    // the CTA's part may start past the expert's rows (then no row is used)
                    const int rlast = c.off[ti.e + 1] - 1;
                    #pragma unroll
                    for (int q = 0; q < 4; ++q) arow[q] = gsrc(0, ti.row0 + 4 * lane + q, rlast);
                }
                // VarK gather: the rows of the K block the cursor is at
                auto fetch_b = [&](int kb) {
                    const int seg = MULTI ? cur.seg : 0;
                    const int r0 = MULTI ? cur.row() : ti.row0 + kb * BK;
                    const int rlast = MULTI ? cur.row0 + cur.rows - 1 : ti.row0 + ti.rows - 1;
                    #pragma unroll
                    for (int j = 0; j < kGatherJ; ++j) {
                        const int g = (lane + 32 * j) & (BK / 4 - 1);
                        #pragma unroll
                        for (int q = 0; q < 4; ++q) brow[j][q] = gsrc(seg, r0 + 4 * g + q, rlast);
                    }
                };
                if (gat && VAR_K && !ti.ones && ti.num_kb > 0) fetch_b(0);
                for (int kb = 0; kb < ti.num_kb; ++kb) {
                    if (leader && t == p.withhold_unit && kb == p.withhold_kb) {
                        // test hook: issue nothing more (no copy is left in
                        // flight for this stage); the copies already issued are
                        // waited for below
                        ok = false;
                        break;
                    }
                    bool got = true;
                    if (!gat || lane == 0)
                        got = mbar_wait_bounded(smem_u32(&c.empty[stage]), phase ^ 1, p.limit_ns,
                                                &c.abort_flag);
                    if (gat) got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
                    if (!got) {
                        if (!gat || lane == 0) raise_abort(c, p);
                        ok = false;
                        break;
                    }
                    const uint32_t sA = smem_u32(base + (size_t)stage * S::STAGE_BYTES);
                    const uint32_t sB = sA + S::A_BYTES;
                    const uint32_t fb = smem_u32(&c.full[stage]);
                    const uint32_t fbc = PAIR ? mapa_rank(fb, 0) : fb;   // even CTA's barrier
                    const int nB = ti.nt * BN + rank * S::BN_CTA;      // first B column held here
                    // bytes: full boxes, except MN slabs lying wholly past the edge
                    uint32_t bytes = 0;
                    if (!VAR_K) {
                        bytes += S::A_BYTES;
                        bytes += S::B_BYTES;   // whole box (columns past N zero-filled)
                    } else {
                        // whole boxes (slabs past the M / N edge are zero-filled); the
                        // row-sum tile reads only A
                        bytes = S::A_BYTES + (ti.ones ? 0 : S::B_BYTES);
                    }
                    // A segment's last K block (weight gradients) lands on a barrier
                    // of this CTA's own, for its relay warp to zero the rows past
                    // the segment before the MMAs read the stage: the odd CTA's
                    // stage barrier (which nothing else completes), the even or
                    // single CTA's tail barrier.
                    const int kvalid = VAR_K ? (MULTI ? cur.valid() : ti.rows - kb * BK) : BK;
                    const bool relay = VAR_K && kvalid < BK;
                    const uint32_t rb = (PAIR && !leader) ? fb : smem_u32(&c.tail[stage]);
                    if (!gat || lane == 0) {
                        if (relay) mbar_arrive_expect_tx(rb, bytes);
                        else if (PAIR && !leader) mbar_arrive_expect_tx_cluster(fbc, bytes);
                        else mbar_arrive_expect_tx(fb, bytes);
                    }
                    if (gat) __syncwarp();
                    const uint32_t lb = relay ? rb : fb;   // barrier of a CTA-local copy
                    auto load2 = [&](uint32_t dst, const CUtensorMap* m, int c0, int c1) {
                        if (PAIR && !relay) tma2_load_2d(dst, m, fbc, c0, c1);
                        else tma_load_2d(dst, m, lb, c0, c1);
                    };
                    auto load3 = [&](uint32_t dst, const CUtensorMap* m, int c0, int c1, int c2) {
                        if (PAIR && !relay) tma2_load_3d(dst, m, fbc, c0, c1, c2);
                        else tma_load_3d(dst, m, lb, c0, c1, c2);
                    };
                    auto gather4 = [&](uint32_t dst, const CUtensorMap* m, int c0, const int (&rows)[4]) {
                        if (PAIR && !relay) tma2_gather4(dst, m, fbc, c0, rows);
                        else tma_gather4(dst, m, lb, c0, rows);
                    };
                    if (!VAR_K) {
                        if (gat) gather4(sA + (uint32_t)lane * 512u, &mapA, kb * BK, arow);
                        else if (lane == 0) load2(sA, &mapA, kb * BK, ti.row0);
                        if (lane == 0) {
                            if (!B_MN) {
                                load3(sB, &mapB, kb * BK, nB, ti.e);
                            } else {
                                // this CTA's 64-column slabs of BK rows in one box
                                // (map: {column in slab, K row, slab, expert})
                                if (PAIR && !relay) tma2_load_4d(sB, &mapB, fbc, 0, kb * BK, nB / 64, ti.e);
                                else tma_load_4d(sB, &mapB, lb, 0, kb * BK, nB / 64, ti.e);
                            }
                        }
                    } else {
                        // one box per operand: this CTA's 64-column slabs of BK rows
                        // (maps: {column in slab, row, slab}); gathered B: BK / 4
                        // four-row loads per slab
                        const int r = MULTI ? cur.row() : ti.row0 + kb * BK;
                        const int mA = ti.mt * S::TILE_M + rank * BM;
                        if (lane == 0) load3(sA, &mapA, 0, r, mA / 64);
                        if (!ti.ones) {
                            if (!gat) {
                                if (lane == 0) load3(sB, &mapB, 0, r, nB / 64);
                            } else {
                                #pragma unroll
                                for (int j = 0; j < kGatherJ; ++j) {
                                    const int jj = lane + 32 * j;
                                    const int slab = jj / (BK / 4), g = jj % (BK / 4);
                                    // a slab past N (its columns are never stored)
                                    // reads the last real slab instead
                                    const int col = nB + slab * 64 < p.N ? nB + slab * 64 : p.N - 64;
                                    gather4(sB + (uint32_t)(slab * SLAB_BYTES + g * 512), &mapB, col,
                                            brow[j]);
                                }
                            }
                        }
                        if (MULTI) cur.advance(p, ti.e);
                        if (gat && !ti.ones && kb + 1 < ti.num_kb) fetch_b(kb + 1);
                    }
                    if (relay && (!PAIR || leader)) {
                        issued_tail[stage] = (int)((tail_phase >> stage) & 1u);
                        issued_parity[stage] = -1;
                        tail_phase ^= 1u << stage;
                    } else {
                        issued_parity[stage] = (int)phase;
                        issued_tail[stage] = -1;
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok && (!PAIR || leader) && (!gat || lane == 0)) {
                // wait (bounded) for every copy this CTA's barriers are counting
                for (int s = 0; s < STAGES; ++s) {
                    if (issued_parity[s] >= 0)
                        mbar_wait_bounded(smem_u32(&c.full[s]), (uint32_t)issued_parity[s],
                                          p.limit_ns, nullptr);
                    if (issued_tail[s] >= 0)
                        mbar_wait_bounded(smem_u32(&c.tail[s]), (uint32_t)issued_tail[s],
                                          p.limit_ns, nullptr);
                }
            }
        };
        if (p.gather == nullptr) {
            if (lane == 0) producer(BoolTag<false>{});
        } else {
            producer(BoolTag<true>{});
        }
        __syncwarp();
    } else if (warp == 1 || (VAR_K && warp == 2 + ES::WARPS)) {
        // ---- weight gradients: tail relay ---------------------------------------------
        // A segment's last K block holds rows of the next segment (or past the
        // end): this warp waits for such a stage on the CTA's own barrier (the
        // odd CTA's stage barrier, the even / single CTA's tail barrier), zeroes
        // the CTA's K rows past the segment in every MN slab (whole 128-byte
        // rows: the swizzle only permutes chunks inside a row), makes the writes
        // visible to the tensor core's reads and then counts the stage as loaded
        // on the even CTA's stage barrier.  The barriers it waits on complete only
        // for such blocks, so their phases are tracked per stage.  The odd CTA's
        // warp 1 (it issues no MMAs) and the even / single CTA's extra warp relay.
        const bool relay_warp = VAR_K && (PAIR && !leader ? warp == 1 : warp == 2 + ES::WARPS);
        if (relay_warp) {
            const bool odd = PAIR && !leader;
            int stage = 0, ecur = 0;
            uint32_t local_phase = 0;   // bit s: parity of the own barrier's next phase
            bool ok = true;
            for (int t = unit0; t < num_units && ok; t += nunits) {
                const Tile ti = get_tile<VAR_K, PAIR, MULTI>(c, p, t, ecur, rank);
                SegCursor cur;
                if (MULTI) cur.start(p, ti.e, ti.kb0, c.off);
                for (int kb = 0; kb < ti.num_kb; ++kb) {
                    const int valid = MULTI ? cur.valid() : ti.rows - kb * BK;
                    if (MULTI) cur.advance(p, ti.e);
                    if (valid < BK) {
                        const uint32_t own = odd ? smem_u32(&c.full[stage]) : smem_u32(&c.tail[stage]);
                        if (!mbar_wait_warp(own, (local_phase >> stage) & 1u, p.limit_ns,
                                            &c.abort_flag)) {
                            raise_abort(c, p);
                            ok = false;
                            break;
                        }
                        local_phase ^= 1u << stage;
                        uint8_t* gA = base + (size_t)stage * S::STAGE_BYTES;
                        const int nz = (BK - valid) * 8;  // 16-byte chunks per slab
                        for (int sl = 0; sl < S::STAGE_BYTES / SLAB_BYTES; ++sl) {
                            uint8_t* slab = gA + sl * SLAB_BYTES;
                            for (int i = lane; i < nz; i += 32)
                                *reinterpret_cast<uint4*>(slab + (valid + (i >> 3)) * 128 +
                                                          ((i & 7) << 4)) = make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            if (odd) mbar_arrive_cluster_release(mapa_rank(smem_u32(&c.full[stage]), 0));
                            else mbar_arrive(smem_u32(&c.full[stage]));
                        }
                    }
                    if (++stage == STAGES) stage = 0;
                }
            }
        }
        // ---- MMA issuer (the even CTA of a pair issues for both) ---------------------
        // One thread issues: it waits for a stage, issues its MMAs and their
        // commit and goes on to the next stage with nothing else in between
        // (the tensor core queues only a few MMAs, so every cycle spent between
        // two stages beyond that queue is an idle tensor core).
        if (leader && warp == 1) {
            constexpr uint32_t IDESC = idesc_bf16_f32(S::TILE_M, BN, A_MN, B_MN);
            // row-sum tile: N = 32 against the all-ones slab (the same slab for every
            // stage and K block)
            constexpr uint32_t IDESC_ONES = idesc_bf16_f32(S::TILE_M, 32, A_MN, B_MN);
            const uint64_t ones_desc =
                smem_desc_sw128(smem_u32(ones_base), B_MN ? SLAB_BYTES : 16, 1024);
            const uint32_t o_lo0 = (uint32_t)ones_desc;
            // Descriptors of stage 0's A and B; a stage or K step only moves the
            // start address (bits 0-13, in 16-byte units; shared addresses stay
            // below 256 KB, so the field never carries into the next one).
            const uint32_t smem0 = smem_u32(base);
            const uint64_t a_desc0 = smem_desc_sw128(smem0, A_MN ? SLAB_BYTES : 16, 1024);
            const uint64_t b_desc0 =
                smem_desc_sw128(smem0 + S::A_BYTES, B_MN ? SLAB_BYTES : 16, 1024);
            const uint32_t a_lo0 = (uint32_t)a_desc0, a_hi = (uint32_t)(a_desc0 >> 32);
            const uint32_t b_lo0 = (uint32_t)b_desc0, b_hi = (uint32_t)(b_desc0 >> 32);
            constexpr uint32_t A_KSTEP = (A_MN ? 2048u : 32u) >> 4;   // one K step of 16
            constexpr uint32_t B_KSTEP = (B_MN ? 2048u : 32u) >> 4;
            if (lane == 0) {
                int stage = 0, acc = 0, ecur = 0;
                uint32_t phase = 0, acc_phase = 0;
                bool ok = true;
                for (int t = unit0; t < num_units && ok; t += nunits) {
                    const Tile ti = get_tile<VAR_K, PAIR, MULTI>(c, p, t, ecur, rank);
                    if (ti.num_kb == 0) continue;
                    if (!mbar_wait_bounded(smem_u32(&c.tempty[acc]), acc_phase ^ 1, p.limit_ns,
                                           &c.abort_flag)) {
                        raise_abort(c, p);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                    const uint32_t idesc = ti.ones ? IDESC_ONES : IDESC;
                    for (int kb = 0; kb < ti.num_kb; ++kb) {
                        if (!mbar_wait_bounded(smem_u32(&c.full[stage]), phase, p.limit_ns,
                                               &c.abort_flag)) {
                            raise_abort(c, p);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t so = (uint32_t)stage * (uint32_t)(S::STAGE_BYTES >> 4);
                        #pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            const uint64_t ad =
                                ((uint64_t)a_hi << 32) | (uint64_t)(a_lo0 + so + kk * A_KSTEP);
                            const uint32_t blo = ti.ones ? o_lo0 + kk * B_KSTEP
                                                         : b_lo0 + so + kk * B_KSTEP;
                            const uint64_t bd = ((uint64_t)b_hi << 32) | (uint64_t)blo;
                            const uint32_t accum = (kk != 0 || kb != 0) ? 1u : 0u;
                            if (PAIR) tc_mma2_bf16(d_tmem, ad, bd, idesc, accum);
                            else tc_mma_bf16(d_tmem, ad, bd, idesc, accum);
                        }
                        if (PAIR) tc_commit2_both(smem_u32(&c.empty[stage]));
                        else tc_commit(smem_u32(&c.empty[stage]));
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                    if (!ok) break;
                    if (PAIR) tc_commit2_both(smem_u32(&c.tfull[acc]));
                    else tc_commit(smem_u32(&c.tfull[acc]));
                    if (++acc == 2) { acc = 0; acc_phase ^= 1; }
                }
            }
            __syncwarp();
            // drain: every MMA this warp issued has completed before TMEM is freed
            if (lane == 0) {
                if (PAIR) tc_commit2_local(smem_u32(&c.drain));
                else tc_commit(smem_u32(&c.drain));
            }
            __syncwarp();
            mbar_wait_bounded(smem_u32(&c.drain), 0, p.limit_ns, nullptr);
        }
    } else {
        // ---- epilogue warps ----------------------------------------------------------
        const int ew = warp - 2;
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int cq = ew >> 2;                 // which ES::COLS columns of the 256
        uint8_t* stg = staging_base + ew * (PP::STAGING / ES::WARPS);
        const uint32_t tempty_local0 = smem_u32(&c.tempty[0]);
        const uint32_t tempty_local1 = smem_u32(&c.tempty[1]);
        if (EPI != (int)Epi::Logits && lane == 0) {
            tma_prefetch_map(&mapO0);
            // second output (BiasGelu) or the saved GELU'(h) input (ScaleAux)
            if (EPI == (int)Epi::BiasGelu || EPI == (int)Epi::ScaleAux) tma_prefetch_map(&mapO1);
        }
        int acc = 0, ecur = 0;
        uint32_t acc_phase = 0;
        // Operands of the epilogue read from global memory stream ahead of the
        // accumulators, across tile boundaries (the next tile of this CTA is
        // known).  The saved GELU'(h) (ScaleAux): TMA boxes of the warp's 32
        // rows x 16 columns (the staging box's shape and swizzle) into a
        // two-chunk ring, issued two chunks ahead by lane 0 (gi chunks issued,
        // gc consumed).  The bias of the warp's columns: one tile ahead, held in
        // registers and written to shared memory as fp32 when its tile starts.
        constexpr bool kAux = PP::AUX;
        constexpr bool kBias = (EPI == (int)Epi::BiasGelu || EPI == (int)Epi::Bias) && !VAR_K;
        constexpr int BW = ES::COLS / 32;   // bias values per lane
        uint8_t* gring = aux_base + ew * 2 * ES::CHUNK_BYTES;
        int gi = 0, gc = 0;
        auto aux_col = [&](const Tile& tt, int ch) { return tt.nt * BN + cq * ES::COLS + ch * CW; };
        auto issue_aux = [&](const Tile& tt, int ch) {   // every lane; lane 0 issues
            if (aux_col(tt, ch) >= p.N) return;           // no such chunk: never consumed
            const int slot = gi & 1;
            if (lane == 0) {
                const uint32_t bar = smem_u32(&c.gbar[ew][slot]);
                mbar_arrive_expect_tx(bar, ES::CHUNK_BYTES);
                tma_load_2d(smem_u32(gring + slot * ES::CHUNK_BYTES), &mapO1, bar,
                            aux_col(tt, ch), tt.row0 + q * 32);
            }
            ++gi;
        };
        auto load_bias = [&](const Tile& tt, float (&b)[BW]) {
            const int cw = tt.nt * BN + cq * ES::COLS;
            const __nv_bfloat16* bp = (const __nv_bfloat16*)p.bias + (int64_t)tt.e * p.N;
            #pragma unroll
            for (int i = 0; i < BW; ++i) {
                const int col = cw + lane * BW + i;
                b[i] = (p.bias && col < p.N) ? __bfloat162float(bp[col]) : 0.f;
            }
        };
        Tile tcur;
        if (unit0 < num_units) tcur = get_tile<VAR_K, PAIR, MULTI>(c, p, unit0, ecur, rank);
        float bnext[BW];
        bool aborted = false;
        if (kAux && unit0 < num_units) {
            issue_aux(tcur, 0);
            if (ES::NCH > 1) issue_aux(tcur, 1);
        }
        if (kBias && unit0 < num_units) load_bias(tcur, bnext);
        for (int t = unit0; t < num_units; t += nunits) {
            const Tile ti = tcur;
            const bool has_next = t + nunits < num_units;
            if (has_next) tcur = get_tile<VAR_K, PAIR, MULTI>(c, p, t + nunits, ecur, rank);
            const bool mma_tile = ti.num_kb > 0;
            const int gc_tile = gc;   // GELU' chunks consumed before this tile
            float* bias_s = bias_base + ew * ES::COLS;
            if (kBias) {
                #pragma unroll
                for (int i = 0; i < BW; ++i) bias_s[lane * BW + i] = bnext[i];
                __syncwarp();
                if (has_next) load_bias(tcur, bnext);
            }
            if (mma_tile) {
                if (!mbar_wait_warp(smem_u32(&c.tfull[acc]), acc_phase, p.limit_ns,
                                    &c.abort_flag)) {
                    raise_abort(c, p);
                    break;
                }
                tc_fence_after();
            }
            const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            const int64_t grow0 = (int64_t)ti.row0 + q * 32;   // global row of lane 0
            const int valid = ti.rows - q * 32;                 // rows of this warp's box
            // One bf16 output chunk: the staged box goes out by TMA when all its
            // 32 rows belong to the segment, else row by row (segment end).
            auto emit = [&](uint8_t* buf, const uint4* pk, const CUtensorMap* map, void* out,
                            int col0) {
                stage_row_packed<CW>(buf, lane, pk);
                if (valid >= 32) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) tma_store_2d(map, smem_u32(buf), col0, (int32_t)grow0);
                } else {
                    __syncwarp();
                    store_tile_bf16<CW>(buf, lane, (__nv_bfloat16*)out, grow0, valid, p.N, col0);
                }
            };
            if (VAR_K && ti.ones && cq == 0) {
                // row sums of act_a: column 0 of the all-ones tile's accumulator
                float v[32];
                if (mma_tile) tmem_ld32(trow, v);
                else v[0] = 0.f;
                const int m = ti.mt * S::TILE_M + rank * BM + q * 32 + lane;
                if (MULTI && ti.bslot >= 0) {   // a split part > 0: its scratch row
                    p.bpart[(int64_t)ti.bslot * S::TILE_M + rank * BM + q * 32 + lane] = v[0];
                } else if (m < p.M) {
                    float* o = p.bsum + (int64_t)ti.e * p.M + m;
                    *o = p.accumulate ? *o + v[0] : v[0];
                }
            }
            #pragma unroll 1
            for (int ch = 0; ch < ES::NCH; ++ch) {
                const int cl = cq * ES::COLS + ch * CW;       // column inside the tile
                const int col0 = ti.nt * BN + cl;             // global column
                if (col0 >= p.N) break;                       // N % 64 == 0: whole chunks
                float v[CW];
                if (mma_tile) {
                    tmem_ld_cw<CW>(trow + (uint32_t)cl, v);
                } else {
                    #pragma unroll
                    for (int i = 0; i < CW; ++i) v[i] = 0.f;
                }
                if (EPI == (int)Epi::Logits) {
                    // fp32 logits [P, N], N any: + bias, staged as 32 x 32 fp32
                    // (word j of row r at r*32 + (j ^ r): conflict-free both
                    // ways), then stored row by row, columns < N only.
                    const float* beta = (const float*)p.bias;
                    float* sf = reinterpret_cast<float*>(stg);
                    #pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float b = (beta && col0 + j < p.N) ? __ldg(beta + col0 + j) : 0.f;
                        sf[lane * 32 + (j ^ lane)] = v[j] + b;
                    }
                    __syncwarp();
                    float* out = (float*)p.out0;
                    const bool col_ok = col0 + lane < p.N;
                    const int64_t grow0 = (int64_t)ti.row0 + q * 32;
                    const int valid = ti.rows - q * 32;
                    #pragma unroll 4
                    for (int r = 0; r < 32; ++r)
                        if (r < valid && col_ok)
                            out[(grow0 + r) * p.N + col0 + lane] = sf[r * 32 + (lane ^ r)];
                    __syncwarp();
                } else if (!VAR_K) {
                    if (kBias) {
                        const float4* b4 = reinterpret_cast<const float4*>(bias_s + ch * CW);
                        #pragma unroll
                        for (int u = 0; u < CW / 4; ++u) {
                            const float4 b = b4[u];
                            f2_unpack(f2_add(f2_pack(v[4 * u], v[4 * u + 1]), f2_pack(b.x, b.y)),
                                      v[4 * u], v[4 * u + 1]);
                            f2_unpack(f2_add(f2_pack(v[4 * u + 2], v[4 * u + 3]), f2_pack(b.z, b.w)),
                                      v[4 * u + 2], v[4 * u + 3]);
                        }
                    }
                    if (kAux) {
                        const int slot = gc & 1;
                        if (!mbar_wait_warp(smem_u32(&c.gbar[ew][slot]), (uint32_t)(gc >> 1) & 1u,
                                            p.limit_ns, &c.abort_flag)) {
                            raise_abort(c, p);
                            aborted = true;
                            break;
                        }
                        U4s<CW / 8> hcur;
                        #pragma unroll
                        for (int u = 0; u < CW / 8; ++u)
                            hcur.u[u] = *reinterpret_cast<const uint4*>(
                                gring + slot * ES::CHUNK_BYTES + stg_off<CW>(lane, u));
                        ++gc;
                        // the slot is refilled (async proxy) after every lane has read it
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (ch + 2 < ES::NCH) issue_aux(ti, ch + 2);
                        else if (has_next) issue_aux(tcur, ch + 2 - ES::NCH);
                        // bf16 pair word -> fp32 pair (low half first), packed multiply
                        #pragma unroll
                        for (int cc = 0; cc < CW / 8; ++cc) {
                            const uint32_t* wd = reinterpret_cast<const uint32_t*>(&hcur.u[cc]);
                            #pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int j = cc * 8 + 2 * i;
                                f2_unpack(f2_mul(f2_pack(v[j], v[j + 1]),
                                                 f2_pack(__uint_as_float(wd[i] << 16),
                                                         __uint_as_float(wd[i] & 0xffff0000u))),
                                          v[j], v[j + 1]);
                            }
                        }
                    }
                    // The staging written below was last read by the TMA stores
                    // of the previous chunk.
                    if (lane == 0) bulk_wait_read<0>();
                    __syncwarp();
                    if (EPI == (int)Epi::BiasGelu) {
                        // one Phi / exp evaluation gives both GELU(h) (kept in v)
                        // and GELU'(h) (stored for the backward)
                        float gd[CW];
                        #pragma unroll
                        for (int i = 0; i < CW; i += 2) {
                            const GeluParts2 r = gelu_parts_fast2(v[i], v[i + 1]);
                            f2_unpack(f2_add(r.Phi, r.xphi), gd[i], gd[i + 1]);
                            f2_unpack(f2_mul(f2_pack(v[i], v[i + 1]), r.Phi), v[i], v[i + 1]);
                        }
                        uint4 pg[CW / 8], pa[CW / 8];
                        #pragma unroll
                        for (int u = 0; u < CW / 8; ++u) {
                            pg[u] = pack8_bf16(gd + 8 * u);
                            pa[u] = pack8_bf16(v + 8 * u);
                        }
                        emit(stg, pg, &mapO0, p.out0, col0);
                        emit(stg + ES::CHUNK_BYTES, pa, &mapO1, p.out1, col0);
                    } else {
                        uint4 pk[CW / 8];
                        #pragma unroll
                        for (int u = 0; u < CW / 8; ++u) pk[u] = pack8_bf16(v + 8 * u);
                        emit(stg, pk, &mapO0, p.out0, col0);
                        if (EPI == (int)Epi::ScaleAux && CW == 16 && p.cpart) {
                            // column sums of this warp's rows inside the segment (rows
                            // past its end are masked), one partial row per (m-tile,
                            // CTA, lane quarter): a halving butterfly over the lanes,
                            // after which the even lanes hold one column each
                            float a[16];
                            const bool row_in = lane < valid;
                            #pragma unroll
                            for (int i = 0; i < 16; ++i) a[i] = (valid >= 32 || row_in) ? v[i] : 0.f;
                            #pragma unroll
                            for (int h = 8; h >= 1; h >>= 1) {
                                const bool up = (lane & (2 * h)) != 0;   // keeps the upper half
                                #pragma unroll
                                for (int j = 0; j < h; ++j) {
                                    const float send = up ? a[j] : a[j + h];
                                    const float keep = up ? a[j + h] : a[j];
                                    a[j] = keep + __shfl_xor_sync(0xffffffffu, send, 2 * h);
                                }
                            }
                            const float cs = a[0] + __shfl_xor_sync(0xffffffffu, a[0], 1);
                            // lane bits 4..1 select the column: 8, 4, 2, 1
                            const int c = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 +
                                          ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
                            const int64_t prow = ((int64_t)(t / NT) * S::CTAS + rank) * 4 + q;
                            if ((lane & 1) == 0) p.cpart[prow * p.N + col0 + c] = cs;
                        }
                    }
                    if (lane == 0) bulk_commit();
                    __syncwarp();
                } else {
                    // fp32 weight gradient, 32 rows x 16 columns (64-byte rows) at a
                    // time: staged like the bf16 boxes (64-byte swizzle) and sent
                    // by one TMA store, or, when accumulating, by one TMA
                    // reduction that adds it to what global memory holds.  The
                    // tensor map clips the rows past M.
                    static_assert(!VAR_K || CW == 32, "fp32 epilogue drains 32-column chunks");
                    const int m0 = ti.mt * S::TILE_M + rank * BM + q * 32;
                    if (m0 < p.M) {
                        #pragma unroll
                        for (int hh = 0; hh < CW / 16; ++hh) {
                            // the staging's previous box has been read by its TMA op
                            if (lane == 0) bulk_wait_read<0>();
                            __syncwarp();
                            #pragma unroll
                            for (int cc = 0; cc < 4; ++cc)
                                *reinterpret_cast<float4*>(stg + stg_off<32>(lane, cc)) =
                                    make_float4(v[hh * 16 + cc * 4], v[hh * 16 + cc * 4 + 1],
                                                v[hh * 16 + cc * 4 + 2], v[hh * 16 + cc * 4 + 3]);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                if (MULTI && ti.slot >= 0)   // a split part > 0: its scratch slot
                                    tma_store_3d(&mapO1, smem_u32(stg), cl + hh * 16,
                                                 rank * BM + q * 32, ti.slot);
                                else if (p.accumulate)
                                    tma_reduce_add_3d(&mapO0, smem_u32(stg), col0 + hh * 16, m0,
                                                      ti.e);
                                else
                                    tma_store_3d(&mapO0, smem_u32(stg), col0 + hh * 16, m0, ti.e);
                                bulk_commit();
                            }
                        }
                    }
                }
            }
            if (aborted) break;
            // a warp whose columns all lie past N consumed no GELU' chunk of this
            // tile, so the next tile's first chunks are not in flight yet
            if (kAux && has_next && gc == gc_tile) {
                issue_aux(tcur, 0);
                if (ES::NCH > 1) issue_aux(tcur, 1);
            }
            if (!mma_tile) continue;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                const uint32_t tb = acc ? tempty_local1 : tempty_local0;
                if (PAIR && !leader) mbar_arrive_cluster(mapa_rank(tb, 0));  // even CTA's barrier
                else mbar_arrive(tb);
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
        // every TMA store has written global memory (and read its staging), and
        // every GELU' load issued has landed, before the CTA exits
        if (lane == 0) bulk_wait_all();
        for (; kAux && gc < gi; ++gc)
            mbar_wait_warp(smem_u32(&c.gbar[ew][gc & 1]), (uint32_t)(gc >> 1) & 1u, p.limit_ns,
                           nullptr);
        __syncwarp();
    }

    // ---- teardown ------------------------------------------------------------------
    tc_fence_before();
    if (PAIR) cluster_sync(); else __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if (PAIR) tmem_dealloc2(tmem_base, TMEM_COLS);
        else tmem_dealloc(tmem_base, TMEM_COLS);
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

// bf16 tensor map (128-byte swizzle unless given), zero fill outside the tensor.
// dims/box innermost first; strides in bytes for dims 1.. .
bool make_map(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B,
              CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    auto fn = encode_fn();
    if (!fn) return false;
    if (rank < 1 || rank > 5) return false;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5] = {1, 1, 1, 1, 1};
    for (int i = 0; i < rank; ++i) { gd[i] = dims[i]; bx[i] = box[i]; }
    for (int i = 0; i < rank - 1; ++i) gs[i] = strides[i];
    CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void*>(ptr),
                    gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Launch options read from the environment at every launch (so that a test
// can change them between calls):
//   MOE_GEMM_PAIR=0        single CTAs (128 x 256 tiles) instead of CTA pairs;
//   MOE_GEMM_MAX_UNITS=n   at most n CTAs (or pairs) per launch, so that each
//                          walks more tiles of the static tile list;
//   MOE_DEBUG_GEMM_WITHHOLD=u:kb  test hook, see TcParams::withhold_unit.
bool use_pairs() {
    const char* s = getenv("MOE_GEMM_PAIR");
    return !(s && s[0] == '0');
}

// The caller's cap (moe_set_gemm_max_units), per host thread; 0: none.
thread_local int64_t t_units_cap = 0;

int64_t max_units_override() {
    const char* s = getenv("MOE_GEMM_MAX_UNITS");
    if (!s || !*s) return t_units_cap;
    const long long v = strtoll(s, nullptr, 10);
    return v > 0 ? (int64_t)v : t_units_cap;
}

void withhold_hook(TcParams& p) {
    p.withhold_unit = -1;
    p.withhold_kb = -1;
    const char* s = getenv("MOE_DEBUG_GEMM_WITHHOLD");
    if (!s || !*s) return;
    char* end = nullptr;
    const long u = strtol(s, &end, 10);
    if (end == s || *end != ':') return;
    const long kb = strtol(end + 1, nullptr, 10);
    if (u < 0 || kb < 0) return;
    p.withhold_unit = (int)u;
    p.withhold_kb = (int)kb;
}

template <bool VAR_K, bool A_MN, bool B_MN, int EPI, bool PAIR, bool MULTI>
cudaError_t launch_tc(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o0,
                      const CUtensorMap& o1, const TcParams& p_in, int64_t units_upper,
                      cudaStream_t st, int* units_out) {
    auto kern = gemm_tc_kernel<VAR_K, A_MN, B_MN, EPI, PAIR, MULTI>;
    constexpr size_t SMEM = smem_bytes<PAIR, VAR_K, EPI>();
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
    constexpr int THREADS = EpiShape<EPI, VAR_K>::THREADS;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    static int max_units = 0;   // co-resident CTAs (or pairs)
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)SMEM);
        if (attr_err != cudaSuccess) return;
        if (PAIR) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 2;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(2 * device_sm_count());
            cfg.blockDim = dim3(THREADS);
            cfg.dynamicSmemBytes = SMEM;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            int n = 0;
            attr_err = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
            max_units = n > 0 ? n : device_sm_count() / 2;
        } else {
            max_units = device_sm_count();
        }
    });
    if (attr_err != cudaSuccess) return attr_err;
    int64_t cap = max_units;
    const int64_t ov = max_units_override();
    if (ov > 0 && ov < cap) cap = ov;
    const int64_t units = units_upper < cap ? (units_upper > 0 ? units_upper : 1) : cap;
    TcParams p = p_in;
    p.split_units = (int)units;
    if (units_out) *units_out = (int)units;
    if (!PAIR) {
        kern<<<(unsigned)units, THREADS, SMEM, st>>>(a, b, o0, o1, p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(2 * units));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a, b, o0, o1, p);
}

template <bool VAR_K, bool A_MN, bool B_MN, int EPI, bool MULTI = false>
cudaError_t launch_either(bool pair, const CUtensorMap& a, const CUtensorMap& b,
                          const CUtensorMap& o0, const CUtensorMap& o1, const TcParams& p,
                          int64_t units1, int64_t units2, cudaStream_t st,
                          int* units_out = nullptr) {
    if (pair)
        return launch_tc<VAR_K, A_MN, B_MN, EPI, true, MULTI>(a, b, o0, o1, p, units2, st,
                                                              units_out);
    return launch_tc<VAR_K, A_MN, B_MN, EPI, false, MULTI>(a, b, o0, o1, p, units1, st,
                                                           units_out);
}

// Adds the split parts > 0 of the weight-gradient tiles (scratch slots, fp32
// [slot][tile_m][BN]) to the output [E, M, N] in part order, so that the result
// is out + part 0 (written by the GEMM) + part 1 + part 2 + ... whatever the
// order the GEMM's CTAs finished in.  Recomputes the GEMM's split from the same
// inputs.  A block takes one expert (blockIdx.y) and strides over its elements,
// four columns per thread.
__global__ void __launch_bounds__(256) vark_split_reduce_kernel(
    int E, int M, int N, int tile_m, int nseg, int ostride, const int32_t* __restrict__ offsets,
    int split_units, int64_t cap, const float* __restrict__ part, float* __restrict__ out,
    const float* __restrict__ bpart, float* __restrict__ bsum) {
    __shared__ int kbs[MAX_E];
    __shared__ int sb[MAX_E];
    __shared__ int kp_s;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int kb = 0;
        for (int sg = 0; sg < nseg; ++sg) {
            const int32_t* o = offsets + (int64_t)sg * ostride;
            kb += (o[e + 1] - o[e] + BK - 1) / BK;
        }
        kbs[e] = kb;
    }
    __syncthreads();
    const int MT = (M + tile_m - 1) / tile_m, NT = (N + BN - 1) / BN;
    if (threadIdx.x == 0) {
        const int kp = vark_kb_part(kbs, E, MT, NT, split_units, cap);
        kp_s = kp;
        int slots = 0;
        for (int e = 0; e < E; ++e) {
            sb[e] = slots;
            slots += (vark_nsplit(kbs[e], kp) - 1) * MT * NT;
        }
    }
    __syncthreads();
    const int e = blockIdx.y;
    const int S = vark_nsplit(kbs[e], kp_s);
    if (S <= 1) return;
    const int64_t n4 = (int64_t)M * N / 4;
    float4* o4 = reinterpret_cast<float4*>(out + (int64_t)e * M * N);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int m = (int)(i * 4 / N), n = (int)(i * 4 % N);
        const int mt = m / tile_m, nt = n / BN;
        float4 a = o4[i];
        for (int q = 1; q < S; ++q) {
            const int64_t slot = sb[e] + (int64_t)(q - 1) * MT * NT + mt * NT + nt;
            const float4 b = *reinterpret_cast<const float4*>(
                part + (slot * tile_m + (m % tile_m)) * BN + (n % BN));
            a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
        }
        o4[i] = a;
    }
    if (bsum && blockIdx.x == 0) {
        // row sums: bsum[e][m] + part 1 + part 2 + ... (block 0 of the expert)
        for (int m = threadIdx.x; m < M; m += blockDim.x) {
            const int mt = m / tile_m;
            float a = bsum[(int64_t)e * M + m];
            for (int q = 1; q < S; ++q)
                a += bpart[((int64_t)sb[e] / NT + (int64_t)(q - 1) * MT + mt) * tile_m + m % tile_m];
            bsum[(int64_t)e * M + m] = a;
        }
    }
}

// Column sums from the ScaleAux epilogue's partial rows: expert e owns the
// rows of its ceil(n_e / tile_m) m-tiles (rows_per_mtile each, experts in
// order).  A block takes one expert and 32 columns; its 8 warps take every
// 8th row and are added in warp order.  Deterministic.
__global__ void __launch_bounds__(256) colsum_mtile_reduce_kernel(
    int N, int E, const int32_t* __restrict__ offsets, int tile_m, int rows_per_mtile,
    const float* __restrict__ part, float* __restrict__ out, int accumulate) {
    __shared__ float red[8][32];
    __shared__ int off_s[MAX_E + 1];
    const int e = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.y * 32 + lane;
    // the segment bounds, loaded in one step (not a chain of dependent loads)
    for (int i = threadIdx.x; i <= e + 1; i += 256) off_s[i] = offsets[i];
    __syncthreads();
    int64_t m0 = 0;
    for (int q = 0; q < e; ++q) m0 += (off_s[q + 1] - off_s[q] + tile_m - 1) / tile_m;
    const int R = ((off_s[e + 1] - off_s[e] + tile_m - 1) / tile_m) * rows_per_mtile;
    const float* src = part + m0 * rows_per_mtile * N + c;
    float s = 0.f;
    if (c < N) {
        // the warp's rows warp, warp + 8, ...: 16 loads in flight, added in row order
        constexpr int UN = 16;
        for (int i0 = warp; i0 < R; i0 += 8 * UN) {
            float v[UN];
            #pragma unroll
            for (int u = 0; u < UN; ++u) {
                const int i = i0 + 8 * u;
                v[u] = i < R ? src[(int64_t)i * N] : 0.f;
            }
            #pragma unroll
            for (int u = 0; u < UN; ++u) s += v[u];   // past the end: + 0
        }
    }
    red[warp][lane] = s;
    __syncthreads();
    if (warp == 0 && c < N) {
        float t = 0.f;
        #pragma unroll
        for (int w = 0; w < 8; ++w) t += red[w][lane];
        float* o = out + (int64_t)e * N + c;
        *o = accumulate ? *o + t : t;
    }
}

// Map of a bf16 [P, N] output for the epilogue's TMA stores: boxes of 32 rows
// x CW columns, swizzled like the staging buffers.
bool make_out_map(CUtensorMap* m, void* ptr, int64_t P, int N, int CW) {
    const uint64_t dims[2] = {(uint64_t)N, (uint64_t)P};
    const uint64_t strides[1] = {(uint64_t)N * 2};
    const uint32_t box[2] = {(uint32_t)CW, 32};
    return make_map(m, ptr, 2, dims, strides, box,
                    CW == 16 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B);
}

}  // namespace

void set_gemm_units_cap(int64_t units) { t_units_cap = units > 0 ? units : 0; }

cudaError_t launch_gemm_varm_tc(const GemmVarM& g, int32_t* status, cudaStream_t st) {
    const bool logits = g.epi == Epi::Logits;
    if (g.E > MAX_E || g.K % 64 || g.N < 1) return cudaErrorInvalidValue;
    if (logits ? (g.E != 1 || g.N > BN) : (g.N % 64 != 0)) return cudaErrorInvalidValue;
    const bool pair = use_pairs();
    const uint32_t bn_cta = pair ? BN / 2 : BN;
    CUtensorMap ma, mb;
    if (g.gather) {
        // the unpermuted rows, one-row boxes for tile::gather4
        if (logits || g.gather_k < 1 || g.gather_rows < 1 || g.gather_rows >= ((int64_t)1 << 31))
            return cudaErrorInvalidValue;
        const uint64_t dims[2] = {(uint64_t)g.K, (uint64_t)g.gather_rows};
        const uint64_t strides[1] = {(uint64_t)g.K * 2};
        const uint32_t box[2] = {BK, 1};
        if (!make_map(&ma, g.act, 2, dims, strides, box)) return cudaErrorInvalidValue;
    } else {
        const uint64_t dims[2] = {(uint64_t)g.K, (uint64_t)g.P};
        const uint64_t strides[1] = {(uint64_t)g.K * 2};
        const uint32_t box[2] = {BK, BM};
        if (!make_map(&ma, g.act, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    if (g.weight_kmajor) {
        const uint64_t dims[3] = {(uint64_t)g.K, (uint64_t)g.N, (uint64_t)g.E};
        const uint64_t strides[2] = {(uint64_t)g.K * 2, (uint64_t)g.N * g.K * 2};
        const uint32_t box[3] = {BK, bn_cta, 1};
        if (!make_map(&mb, g.weight, 3, dims, strides, box)) return cudaErrorInvalidValue;
    } else {
        // [E, K, N] seen as {column in 64-wide slab, K row, slab, expert}: one box
        // fills a CTA's MN-major slabs of BK rows, slab after slab
        const uint64_t dims[4] = {64, (uint64_t)g.K, (uint64_t)g.N / 64, (uint64_t)g.E};
        const uint64_t strides[3] = {(uint64_t)g.N * 2, 128, (uint64_t)g.K * g.N * 2};
        const uint32_t box[4] = {64, BK, bn_cta / 64, 1};
        if (!make_map(&mb, g.weight, 4, dims, strides, box)) return cudaErrorInvalidValue;
    }
    TcParams p{};
    p.E = g.E; p.N = g.N; p.K = g.K; p.M = 0; p.P = g.P;
    p.offsets = g.offsets; p.bias = g.bias; p.aux = g.aux; p.out0 = g.out0; p.out1 = g.out1;
    p.outf = nullptr; p.accumulate = 0; p.status = status; p.limit_ns = wait_limit_ns();
    withhold_hook(p);
    p.gather = g.gather;
    p.gk = g.gather_k;
    const bool colsum = g.epi == Epi::ScaleAux && g.colsum != nullptr;
    if (colsum && !g.colsum_partial) return cudaErrorInvalidValue;
    p.cpart = colsum ? g.colsum_partial : nullptr;
    const int64_t NT = (g.N + BN - 1) / BN;
    const int64_t u1 = ((g.P + BM - 1) / BM + g.E) * NT;
    const int64_t u2 = ((g.P + 2 * BM - 1) / (2 * BM) + g.E) * NT;
    if (g.P >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;   // TMA row coordinate
    const bool wide = g.epi == Epi::BiasGelu || g.epi == Epi::ScaleAux;
    const int cw = wide ? EpiShape<(int)Epi::BiasGelu, false>::CW
                        : EpiShape<(int)Epi::Bias, false>::CW;
    CUtensorMap mo0, mo1;
    if (logits) {   // fp32 output, stored by the epilogue warps
        memset(&mo0, 0, sizeof(mo0));
        return launch_either<false, false, false, (int)Epi::Logits>(pair, ma, mb, mo0, mo0, p, u1, u2,
                                                                    st);
    }
    if (!make_out_map(&mo0, g.out0, g.P, g.N, cw)) return cudaErrorInvalidValue;
    if (g.epi == Epi::BiasGelu) {
        if (!make_out_map(&mo1, g.out1, g.P, g.N, cw)) return cudaErrorInvalidValue;
    } else if (g.epi == Epi::ScaleAux) {   // the saved GELU'(h), read in the same boxes
        if (!make_out_map(&mo1, const_cast<void*>(g.aux), g.P, g.N, cw)) return cudaErrorInvalidValue;
    } else {
        mo1 = mo0;
    }
    switch (g.epi) {
        case Epi::BiasGelu:
            if (!g.weight_kmajor) return cudaErrorInvalidValue;
            return launch_either<false, false, false, (int)Epi::BiasGelu>(pair, ma, mb, mo0, mo1, p, u1,
                                                                          u2, st);
        case Epi::Bias:
            if (!g.weight_kmajor) return cudaErrorInvalidValue;
            return launch_either<false, false, false, (int)Epi::Bias>(pair, ma, mb, mo0, mo1, p, u1, u2,
                                                                      st);
        case Epi::ScaleAux: {
            if (g.weight_kmajor) return cudaErrorInvalidValue;
            cudaError_t e = launch_either<false, false, true, (int)Epi::ScaleAux>(
                pair, ma, mb, mo0, mo1, p, u1, u2, st);
            if (e != cudaSuccess || !colsum) return e;
            colsum_mtile_reduce_kernel<<<dim3((unsigned)g.E, (unsigned)((g.N + 31) / 32)), 256,
                                         0, st>>>(g.N, g.E, g.offsets, pair ? 2 * BM : BM,
                                                  (pair ? 2 : 1) * 4, g.colsum_partial, g.colsum,
                                                  g.colsum_accumulate);
            return cudaGetLastError();
        }
        case Epi::Plain:
            if (g.weight_kmajor) return cudaErrorInvalidValue;
            return launch_either<false, false, true, (int)Epi::Plain>(pair, ma, mb, mo0, mo1, p, u1, u2,
                                                                      st);
    }
    return cudaErrorInvalidValue;
}

size_t vark_split_workspace(int64_t rows, int E, int M, int N) {
    // parts of >= kKbPartMin K blocks: at most (rows / 64 + E) / kKbPartMin parts
    // beyond the first over all experts, each needing MT x NT slots of 256 x 256
    // fp32 (+ a row-sum row); one more for rounding
    const int64_t parts = (rows / BK + E) / kKbPartMin + 1;
    const int64_t MT = (M + 2 * BM - 1) / (2 * BM), NT = (N + BN - 1) / BN;
    return (size_t)(parts * MT * NT) * (size_t)(2 * BM * BN * 4 + 2 * BM * 4);
}

size_t gemm_colsum_workspace(int64_t P, int E, int N) {
    // 4 partial rows per 128-row CTA tile.  Single CTAs: at most ceil(P/128) + E
    // tiles; pairs: 2 (ceil(P/256) + E) <= ceil(P/128) + 1 + 2E.
    return (size_t)((P + BM - 1) / BM + 2 * (int64_t)E + 1) * 4 * (size_t)N * sizeof(float);
}

cudaError_t launch_gemm_vark_tc(const GemmVarK& g, int32_t* status, cudaStream_t st) {
    if (g.E > MAX_E || g.M % 64 || g.N % 64) return cudaErrorInvalidValue;
    // Activations [P, M] and [P, N] seen as {column in 64-wide slab, row, slab}
    // (the slab stride, 128 bytes, is below the row stride): one TMA box fills a
    // CTA's MN-major slabs of BK rows, slab after slab.
    const bool pair = use_pairs();
    CUtensorMap ma, mb;
    {
        const uint64_t dims[3] = {64, (uint64_t)g.P, (uint64_t)g.M / 64};
        const uint64_t strides[2] = {(uint64_t)g.M * 2, 128};
        const uint32_t box[3] = {64, BK, BM / 64};
        if (!make_map(&ma, g.act_a, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    if (g.gather_b) {
        // the unpermuted rows, one-row boxes of one 64-column slab for tile::gather4
        if (g.gather_k < 1 || g.gather_rows < 1 || g.gather_rows >= ((int64_t)1 << 31))
            return cudaErrorInvalidValue;
        const uint64_t dims[2] = {(uint64_t)g.N, (uint64_t)g.gather_rows};
        const uint64_t strides[1] = {(uint64_t)g.N * 2};
        const uint32_t box[2] = {64, 1};
        if (!make_map(&mb, g.act_b, 2, dims, strides, box)) return cudaErrorInvalidValue;
    } else {
        const uint64_t dims[3] = {64, (uint64_t)g.P, (uint64_t)g.N / 64};
        const uint64_t strides[2] = {(uint64_t)g.N * 2, 128};
        const uint32_t box[3] = {64, BK, (uint32_t)(pair ? BN / 2 : BN) / 64};
        if (!make_map(&mb, g.act_b, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    if (g.nseg < 1 || g.nseg > kMaxWgradChunks) return cudaErrorInvalidValue;
    if (g.P >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;   // TMA row coordinate
    TcParams p{};
    p.E = g.E; p.M = g.M; p.N = g.N; p.K = 0; p.P = g.P;
    p.offsets = g.offsets; p.outf = g.out; p.accumulate = g.accumulate;
    p.nseg = g.nseg; p.ostride = g.ostride;
    for (int i = 0; i < g.nseg; ++i) p.seg_base[i] = g.seg_base[i];
    p.gather = g.gather_b;
    p.gk = g.gather_k;
    p.gstride = g.gather_stride;
    for (int i = 0; i < g.nseg; ++i) p.gbase[i] = g.gather_base[i];
    p.status = status; p.limit_ns = wait_limit_ns();
    withhold_hook(p);
    p.bsum = g.bsum;
    const int64_t NT = (g.N + BN - 1) / BN + (g.bsum ? 1 : 0);
    // without a split; the grid is capped at the co-resident CTAs (pairs) anyway
    const int64_t u1 = (int64_t)g.E * ((g.M + BM - 1) / BM) * NT;
    const int64_t u2 = (int64_t)g.E * ((g.M + 2 * BM - 1) / (2 * BM)) * NT;
    // scratch for the split parts: fp32 tiles [slot][tile_m][BN], stored by TMA
    // in the epilogue's 32 x 16 boxes
    const int tile_m = pair ? 2 * BM : BM;
    const int64_t slot_bytes = (int64_t)tile_m * BN * 4;
    // The segment walk and the split are compiled into a kernel of their own
    // (MULTI): a one-segment call over at most kLeanMaxRows rows takes the lean
    // kernel, without their code and set-up.
    // (The lean kernel reads the rows at the chunk's own offsets: a group of
    // chunks that does not start at row 0 takes the segment walk too.)
    const bool multi = g.nseg > 1 || g.seg_base[0] != 0 || g.P > kLeanMaxRows;
    // each partial tile's slot also reserves one row-sum row (tile_m floats)
    // after the tiles; the row sums of a split need at most one per N tiles
    int64_t cap = (multi && g.part) ? (int64_t)(g.part_bytes / (size_t)(slot_bytes + tile_m * 4))
                                    : 0;
    if (cap > ((int64_t)1 << 30)) cap = (int64_t)1 << 30;
    float* bpart = g.part ? g.part + cap * tile_m * BN : nullptr;
    CUtensorMap mpart;
    if (cap > 0) {
        const uint64_t dims[3] = {(uint64_t)BN, (uint64_t)tile_m, (uint64_t)cap};
        const uint64_t strides[2] = {(uint64_t)BN * 4, (uint64_t)slot_bytes};
        const uint32_t box[3] = {16, 32, 1};
        if (!make_map(&mpart, g.part, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B,
                      CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
            return cudaErrorInvalidValue;
    }
    p.part_cap = cap;
    p.bpart = bpart;
    // fp32 output [E, M, N]: boxes of 32 rows x 16 columns, 64-byte swizzle
    CUtensorMap mo;
    {
        const uint64_t dims[3] = {(uint64_t)g.N, (uint64_t)g.M, (uint64_t)g.E};
        const uint64_t strides[2] = {(uint64_t)g.N * 4, (uint64_t)g.M * g.N * 4};
        const uint32_t box[3] = {16, 32, 1};
        if (!make_map(&mo, g.out, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B,
                      CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
            return cudaErrorInvalidValue;
    }
    if (cap == 0) mpart = mo;
    // u1 / u2 bound the grid only; with a split there are more units than that
    const int64_t big = (int64_t)1 << 30;
    int units = 0;
    cudaError_t e =
        multi ? launch_either<true, true, true, (int)Epi::Plain, true>(
                    pair, ma, mb, mo, mpart, p, cap > 0 ? big : u1, cap > 0 ? big : u2, st, &units)
              : launch_either<true, true, true, (int)Epi::Plain, false>(pair, ma, mb, mo, mo, p,
                                                                        u1, u2, st, &units);
    if (e != cudaSuccess || cap == 0) return e;
    const int64_t n4 = (int64_t)g.M * g.N / 4;
    const unsigned gx = (unsigned)(n4 / 256 < 64 ? (n4 + 255) / 256 : 64);
    vark_split_reduce_kernel<<<dim3(gx, (unsigned)g.E), 256, 0, st>>>(
        g.E, g.M, g.N, tile_m, g.nseg, g.ostride, g.offsets, units, cap, g.part, g.out, bpart,
        g.bsum);
    return cudaGetLastError();
}

}  // namespace moe
