// attn_bwd.cu -- attention backward for GB300 (sm_103a): dQ, dK, dV of
// O = softmax(Q K^T / sqrt(d)) V, d = 128 or 64, on tcgen05 tensor cores, and its C ABI.
//
// Source pages: "HipKittens: Fast and Furious AMD Kernels (MLSys 2026)", "Key observations"
// (observation 3) and "Attention backward": the attention backward is the next kernel after
// the forward; "MoonMath AI open-sources a HIP attention kernel for AMD MI300X that beats
// AITER", opening section: the forward being differentiated.  With c = 1/sqrt(d),
// P = softmax(c Q K^T) recomputed from the forward's row log-sum-exp, and the upstream
// gradient dO:
//   dV = P^T dO,   dP = dO V^T,   D_i = dO_i . O_i,   dS = P * (dP - D),
//   dQ = c dS K,   dK = c dS^T Q.
// GB300 design:
//   * a preprocessing kernel forms D_i (fp32) and the base-2 log-sum-exp per query row and
//     zeroes the fp32 dQ accumulator;
//   * the main kernel gives each work unit one (b, K/V head) and one 128-key tile: K_j and
//     V_j stay in shared memory while the unit walks every query tile of every query head
//     that reads that K/V head.  Per query tile i it runs five tcgen05 GEMMs with the key
//     tile on the M side, so the recomputed probabilities come out transposed (one TMEM lane
//     per key) and feed the dV and dK products straight from tensor memory:
//       S^T  = K_j Q_i^T          (both operands K-major in shared memory)
//       dP^T = V_j dO_i^T
//       dV  += P^T dO_i           (P^T read from TMEM, dO_i an MN-major operand)
//       dK  += dS^T Q_i           (dS^T read from TMEM)
//       dQ_i = dS K_j             (dS^T also written to shared memory, read as an MN-major
//                                  A operand; K_j as an MN-major B operand)
//     dV and dK accumulate in TMEM for the whole unit and go out as TMA tile stores; dQ_i is
//     added into an fp32 accumulator in global memory by TMA tensor reductions (many key
//     tiles contribute, in no fixed order), or, in the deterministic mode, stored into an fp32
//     slice of its own key tile.  Causal units (which shrink with their key tile) run on a paired
//     schedule, and otherwise the units of a last, partial round run as query-range parts
//     whose fp32 dK/dV partials are added at the end;
//   * a last kernel rounds the dQ accumulator to bf16 (round to nearest even), or first adds
//     each row's key-tile slices in key-tile order (deterministic mode), and adds the split
//     units' dK/dV partials in part order.
// Variable-length batches (attn_bwd_varlen, the backward of attn_fwd_varlen) add a one-CTA
// planning kernel in front (per-sequence tensor maps narrowed with tensormap.replace, padded
// statistics offsets, the units heaviest first) and run varlen instances of the other three
// ("varlen" below).
// Each kernel is a programmatic dependent of the one before it in the stream.
// Roles: warp 8 TMA producer, warp 9 (one thread) MMA issuer; warpgroups 0 and 1 recompute P
// and form dS for query columns 0..63 and 64..127 of each step, then each drains half of dQ's
// columns; at the end of a unit warpgroup 0 writes dV and warpgroup 1 dK.  Every wait is
// bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <string.h>

#include <cmath>
#include <mutex>

#include "../../include/bf16_attn.h"
#include "ptx.cuh"

namespace {

constexpr int kBM = 128;                      // query rows per query tile
constexpr int kBN = 128;                      // keys per key tile (one unit)
constexpr int kChunkBytes = kBM * 64 * 2;     // 16 KB: one 64-column TMA box of 128 rows
constexpr int kThreads = 384;
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
constexpr uint32_t kTmemCols = 512;           // S^T/P^T/dQ | dP^T/dS^T | dV | dK

// Q_i and dO_i go through a two-stage ring (stage s % 2 for step s) so the next query
// tile loads while the current one is in use; each stage is Q then dO.
constexpr int kStages = 2;
constexpr int kDSBytes = kBM * kBN * 2;       // dS^T: 128 keys x 128 queries, bf16

// Head-dimension dependent geometry (D = 128 or 64); shared memory offsets are from a
// 1024-byte aligned base.
template <int D>
struct BGeo {
    static_assert(D == 64 || D == 128, "head dimension 64 or 128");
    static constexpr int kChunks = D / 64;                    // 64-column TMA boxes per row
    static constexpr int kTileBytes = kBM * D * 2;            // one 128-row tile of Q, K, V or dO
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kSmemK = 0;
    static constexpr int kSmemV = kSmemK + kTileBytes;
    static constexpr int kSmemStage0 = kSmemV + kTileBytes;
    static constexpr int kSmemDS = kSmemStage0 + kStages * kStageBytes;
    static constexpr int kSmemStats = kSmemDS + kDSBytes;     // base-2 LSE [128] then D [128]
    static constexpr int kSmemBars = kSmemStats + 2 * kBM * 4;
};
enum {
    kBarKV = 0,      // K_j, V_j loaded
    kBarKVEmpty,     // the unit's last GEMM reading K_j, V_j is done
    kBarQFull,       // [2] Q_i, dO_i of stage s % 2 loaded
    kBarQEmpty = kBarQFull + kStages,   // [2] the GEMMs reading that stage are done
    kBarStaged = kBarQEmpty + kStages,   // [2] the step's dQ staged in that stage (8 arrivals)
    kBarStats = kBarStaged + kStages,    // the step's row statistics loaded
    kBarSFull,       // S^T in TMEM
    kBarDPFull,      // dP^T in TMEM
    kBarPFull,       // P^T, dS^T in TMEM and dS^T in shared memory (256 arrivals)
    kBarRead,        // both warpgroups have read S^T and dP^T out of TMEM (256 arrivals)
    kBarDQFull,      // dQ_i in TMEM
    kBarDQEmpty,     // dQ_i read out of TMEM (256 arrivals: each warpgroup reads half its columns)
    kBarDKVFull,     // the unit's dK, dV final in TMEM
    kBarDKVEmpty,    // dK, dV read out of TMEM (256 arrivals)
    kBarOutStaged,   // [2] warpgroup h's 64 columns of dV (h = 0) or dK (h = 1) staged in box h (128 arrivals)
    kBarBoxFree = kBarOutStaged + 2,   // [2] warpgroup h's box store has read box h
    kBarDrain = kBarBoxFree + 2,
    kNumBars
};
template <int D>
__host__ __device__ constexpr int smem_misc() { return BGeo<D>::kSmemBars + kNumBars * 8; }
template <int D>
__host__ __device__ constexpr int smem_alloc() { return smem_misc<D>() + 16 + 1024; }
static_assert(smem_alloc<128>() <= 232448, "shared memory over the 227 KB limit");

enum : uint32_t {
    kSiteKV = 1, kSiteKVEmpty, kSiteQFull, kSiteQEmpty, kSiteSFull, kSitePFull, kSiteDQFull,
    kSiteDQEmpty, kSiteDKVFull, kSiteDKVEmpty, kSiteStats, kSiteDPFull, kSiteRead, kSiteOutStaged,
    kSiteOutFree, kSiteSeqlens
};
static_assert(kSiteDKVFull == ATTN_BWD_SITE_DKV_READY, "the dK/dV-ready wait site is part of the ABI");
static_assert(kSiteSeqlens == ATTN_BWD_SITE_SEQLENS, "the sequence-length check site is part of the ABI");

__device__ uint32_t g_bwd_status[2];   // [0] status code, [1] wait site

struct BwdParams {
    int B, H, Hkv, Sq, Skv, group;
    int nq, nkv, nq_pad_rows;    // query tiles, key tiles, rows per (b, h) in the stat arrays
    int n_units;
    int n_items, n_full;         // work items; items >= n_full are query-range parts of tail units
    int nsplit;                  // parts per split unit (1: nothing split)
    int paired;                  // 1: the paired schedule of causal units (sched_pos, unit_at)
    int causal, causal_off;      // key j visible to query i iff j <= i + causal_off
    int bshd;
    float scale;                 // 1/sqrt(d)
    float scale_log2;            // log2(e)/sqrt(d)
    const float* lse2;           // [B*H][nq_pad_rows] base-2 log-sum-exp
    const float* delta;          // [B*H][nq_pad_rows] D_i
    float* dq_acc;               // [B][H][Sq][d] fp32, or the deterministic mode's key-tile slices
    float* ws_dkv;               // [split items][2: dV, dK][128][d] fp32 partials
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    long long kv_sb, kv_ss, kv_sh;   // element strides of dK/dV for b, s, h
    unsigned long long wait_limit_ns;
    int test_hooks;              // ATTN_TEST_WITHHOLD_O_READY: CTA 0 skips its first unit's dK/dV-ready signal
    // variable-length batches (the kVarlen instance): per sequence b the tensor maps
    // vl_maps[7 b + 0..6] = Q, dO, K, V, dK, dV (bf16, the sequence's rows) and the dQ
    // accumulator (fp32 [H][total_q][d], the sequence's rows); the work units (b, K/V head, key
    // tile), heaviest first, and their count; the sequences' padded statistics row offsets
    const CUtensorMap* vl_maps;
    const int4* vl_units;
    const int* vl_n_units;
    const int* vl_pad;           // [B + 1], multiples of 128; statistics rows h * stat_stride + ...
    const int* cu_q;
    const int* cu_k;
    long long stat_stride;
};

struct Unit {
    int b, kvh, jt;          // batch, K/V head, key tile
    int it_lo;               // first query tile with a visible key
    int nsteps;              // query tiles x query heads of the group
    int st0, st1;            // the steps this work item runs, [st0, st1): all of them unless split
    int slot;                // split item: the row of its dV/dK partials in the workspace; else -1
    int sq, coff, pad;       // variable-length batches: the sequence's query count, causal
                             // offset (Skv - Sq) and first padded statistics row
};

__device__ __forceinline__ Unit decode_unit(const BwdParams& p, int k) {
    Unit u;
    u.jt = k % p.nkv;
    const int bk = k / p.nkv;
    u.kvh = bk % p.Hkv;
    u.b = bk / p.Hkv;
    u.it_lo = 0;
    if (p.causal) {
        // the first query that sees key jt*128 is jt*128 - causal_off
        const int first_q = u.jt * kBN - p.causal_off;
        u.it_lo = first_q <= 0 ? 0 : first_q / kBM;
    }
    const int nt = u.it_lo < p.nq ? p.nq - u.it_lo : 0;
    u.nsteps = nt * p.group;
    return u;
}

// The schedule: a CTA's n-th unit sits at position sched_pos(n) of the unit order, and
// unit_at() maps a position to a unit.  Without the mask every unit has the same length and
// positions go round-robin.  Causal units shrink with their key tile (fewer query tiles see
// later keys), and round-robin left CTAs up to 1.3-1.7x the mean load (a model of per-CTA
// query steps on the causal prefill and square shapes); so positions within each (b, K/V
// head) take key tiles 0, n-1, 1, n-2, ... and each CTA takes two consecutive positions per
// round, a pair whose lengths add up to about the same total.  A round still covers
// consecutive (b, K/V head) groups, so the Q and dO those units read stay shared in L2.
// Pairs are used (p.paired) for causal launches with at least two units per CTA.
template <bool kVarlen = false>
__device__ __forceinline__ int sched_pos(const BwdParams& p, int n) {
    // a variable-length batch's units come heaviest first: rounds alternate direction
    if constexpr (kVarlen)
        return n * (int)gridDim.x + ((n & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x);
    if (!p.paired) return n * (int)gridDim.x + (int)blockIdx.x;
    return (n >> 1) * 2 * (int)gridDim.x + 2 * (int)blockIdx.x + (n & 1);
}
__device__ __forceinline__ int unit_at(const BwdParams& p, int pos) {
    if (!p.paired) return pos;
    const int g = pos / p.nkv, i = pos % p.nkv;
    const int jt = (i & 1) ? p.nkv - 1 - (i >> 1) : (i >> 1);
    return g * p.nkv + jt;
}

// Work item at schedule position pos.  Items below n_full are whole units (the paired causal
// schedule maps positions to units first); the rest split the last, partial round's units into
// nsplit ranges of query steps each, whose dK/dV partials a final kernel adds in part order.
__device__ __forceinline__ Unit decode_varlen_unit(const BwdParams& p, int pos) {
    Unit u;
    const int4 e = __ldg(p.vl_units + pos);
    u.b = e.x;
    u.kvh = e.y;
    u.jt = e.z;
    const int q0 = __ldg(p.cu_q + u.b);
    u.sq = __ldg(p.cu_q + u.b + 1) - q0;
    u.coff = (__ldg(p.cu_k + u.b + 1) - __ldg(p.cu_k + u.b)) - u.sq;
    u.pad = __ldg(p.vl_pad + u.b);
    u.it_lo = 0;
    if (p.causal) {
        const int first_q = u.jt * kBN - u.coff;
        u.it_lo = first_q <= 0 ? 0 : first_q / kBM;
    }
    const int nq = (u.sq + kBM - 1) / kBM;
    u.nsteps = (u.it_lo < nq ? nq - u.it_lo : 0) * p.group;
    u.st0 = 0;
    u.st1 = u.nsteps;
    u.slot = -1;
    return u;
}

template <bool kVarlen = false>
__device__ __forceinline__ Unit decode_item(const BwdParams& p, int pos) {
    if constexpr (kVarlen) return decode_varlen_unit(p, pos);
    Unit u;
    if (pos < p.n_full) {
        u = decode_unit(p, unit_at(p, pos));
        u.st0 = 0;
        u.st1 = u.nsteps;
        u.slot = -1;
    } else {
        const int r = pos - p.n_full, t = r / p.nsplit, part = r % p.nsplit;
        u = decode_unit(p, p.n_full + t);
        const int base = u.nsteps / p.nsplit, rem = u.nsteps % p.nsplit;
        u.st0 = part * base + (part < rem ? part : rem);
        u.st1 = u.st0 + base + (part < rem ? 1 : 0);
        u.slot = r;
    }
    return u;
}

__device__ __forceinline__ bool bwd_wait(uint32_t bar, uint32_t parity, uint32_t site,
                                         volatile uint32_t* abort_flag, unsigned long long limit_ns) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer_ns() - t0 > limit_ns) {
            if (atomicCAS(&g_bwd_status[0], 0u, (uint32_t)ATTN_ERR_DEVICE_TIMEOUT) == 0u)
                atomicExch(&g_bwd_status[1], site);
            *abort_flag = 1u;
            return false;
        }
    }
}

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;              // 128-byte swizzle
    return d;
}

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// fp32 -> bf16 bits, round to nearest even (the conversion instruction), NaN stays NaN
__device__ __forceinline__ uint32_t pack2(float lo, float hi) { return ptx::pack_bf16x2(lo, hi); }

// global[tile at (c0, c1, c2)] += shared (fp32 add, done by the TMA unit; out-of-range
// elements of the box are skipped)
__device__ __forceinline__ void tma_reduce_add_3d(const void* tmap, uint32_t src, int c0, int c1, int c2) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(tmap)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// four floats from shared memory (an explicit shared-space load: through a generic pointer
// the loads went down the generic path, whose latency every element's chain then waited on)
__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}


// kDet: the deterministic mode (dQ terms stored to per-key-tile slices, not added); kVarlen: a
// variable-length batch (units, tensor maps and statistics offsets from its planning kernel).
// Separate instances, so the default one carries none of either.
template <int D, bool kDet, bool kVarlen = false>
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap domap,
                const __grid_constant__ CUtensorMap dqmap, const __grid_constant__ CUtensorMap dkmap,
                const __grid_constant__ CUtensorMap dvmap, const BwdParams p) {
    using G = BGeo<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bars = sbase + G::kSmemBars;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint32_t* tmem_holder = (uint32_t*)(smem + smem_misc<D>());
    volatile uint32_t* abort_flag = (volatile uint32_t*)(smem + smem_misc<D>() + 4);
    const uint32_t s_lse2 = ptx::smem_u32(smem + G::kSmemStats);   // base-2 LSE [128], then D [128]
    const uint32_t s_delta = s_lse2 + kBM * 4;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(kBarKV), 1);
        ptx::mbar_init(bar(kBarKVEmpty), 1);
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(bar(kBarQFull + i), 1);
            ptx::mbar_init(bar(kBarQEmpty + i), 1);
            ptx::mbar_init(bar(kBarStaged + i), 8);
        }
        ptx::mbar_init(bar(kBarStats), 1);
        ptx::mbar_init(bar(kBarSFull), 1);
        ptx::mbar_init(bar(kBarDPFull), 1);
        ptx::mbar_init(bar(kBarPFull), 2 * kBN);
        ptx::mbar_init(bar(kBarRead), 2 * kBN);
        ptx::mbar_init(bar(kBarDQFull), 1);
        ptx::mbar_init(bar(kBarDQEmpty), 2 * kBM);
        ptx::mbar_init(bar(kBarDKVFull), 1);
        ptx::mbar_init(bar(kBarDKVEmpty), 2 * kBN);
        ptx::mbar_init(bar(kBarOutStaged), kBN);
        ptx::mbar_init(bar(kBarOutStaged + 1), kBN);
        ptx::mbar_init(bar(kBarBoxFree), 1);
        ptx::mbar_init(bar(kBarBoxFree + 1), 1);
        ptx::mbar_init(bar(kBarDrain), 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == kWarpMma) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_holder), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const unsigned long long lim = p.wait_limit_ns;
    // the dQ rounding kernel may be scheduled as CTAs retire; it waits for this grid's memory
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // a variable-length batch's units and maps come from the kernels before this one: every
    // thread waits for their memory first
    if constexpr (kVarlen) asm volatile("griddepcontrol.wait;" ::: "memory");
    const int n_items = kVarlen ? __ldg(p.vl_n_units) : p.n_items;
    // TMEM: S^T then P^T | dP^T then dS^T, later dQ_i | dV | dK.  dQ_i goes where dP^T was, so
    // the next step's S^T GEMM does not wait for dQ_i to be read out.
    const uint32_t tS = tmem, tDP = tmem + 128u, tDV = tmem + 256u, tDK = tmem + 256u + (uint32_t)D, tDQ = tDP;

    // P^T = 2^(S^T log2(e)/sqrt(d) - LSE2) and dS^T = P^T (dP^T - D) for this thread's key row
    // and query columns 64*half .. 64*half + 63 of step s (warpgroup `half` runs it).  The
    // bf16 results go to TMEM over S^T and dP^T, where they take half the columns: column c of
    // P^T holds queries 2c and 2c+1, so warpgroup 1's results land on columns warpgroup 0
    // still reads.  Both warpgroups therefore read and compute first, meet on a barrier, and
    // only then store to TMEM.  dS^T also goes to shared memory (its own region) for dQ.
    auto pds_step = [&](const Unit& un, int it, uint32_t s, int half) -> bool {
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;                     // key row of the tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const int kj = un.jt * kBN + row;
        bool ok = bwd_wait(bar(kBarStats), s & 1u, kSiteStats, abort_flag, lim) &&
                  bwd_wait(bar(kBarSFull), s & 1u, kSiteSFull, abort_flag, lim) &&
                  bwd_wait(bar(kBarDPFull), s & 1u, kSiteDPFull, abort_flag, lim);
        if (!__all_sync(0xFFFFFFFFu, ok)) return false;
        ptx::tc_fence_after();
        const float cl = p.scale_log2;
        uint32_t pw[2][16], dw[2][16];
#pragma unroll
        for (int ci = 0; ci < 2; ++ci) {
            const int c = 2 * half + ci;
            uint32_t sv[32], dp[32];
            ptx::tmem_ld32(tS + lane_off + 32u * c, sv);
            ptx::tmem_ld32(tDP + lane_off + 32u * c, dp);
            const int q0 = it * kBM + 32 * c;
            // every column of this chunk visible to this key: no per-element test
            const int sq = kVarlen ? un.sq : p.Sq, coff = kVarlen ? un.coff : p.causal_off;
            const bool all_vis = q0 + 31 < sq && (!p.causal || kj <= q0 + coff);
            const float2 c2 = make_float2(cl, cl);
            if (all_vis) {
                // the packed arithmetic below without the mask
#pragma unroll
                for (int g4 = 0; g4 < 8; ++g4) {
                    const float4 l4 = ld_shared_f4(s_lse2 + (uint32_t)(4 * (32 * c + 4 * g4)));
                    const float4 d4 = ld_shared_f4(s_delta + (uint32_t)(4 * (32 * c + 4 * g4)));
                    const int col = 4 * g4;
                    const float2 x01 = __ffma2_rn(make_float2(__uint_as_float(sv[col]), __uint_as_float(sv[col + 1])), c2,
                                                  make_float2(-l4.x, -l4.y));
                    const float2 x23 = __ffma2_rn(make_float2(__uint_as_float(sv[col + 2]), __uint_as_float(sv[col + 3])), c2,
                                                  make_float2(-l4.z, -l4.w));
                    const float2 p01 = make_float2(ptx::ex2_approx(x01.x), ptx::ex2_approx(x01.y));
                    const float2 p23 = make_float2(ptx::ex2_approx(x23.x), ptx::ex2_approx(x23.y));
                    const float2 s01 = __fmul2_rn(p01, __fadd2_rn(make_float2(__uint_as_float(dp[col]), __uint_as_float(dp[col + 1])),
                                                                   make_float2(-d4.x, -d4.y)));
                    const float2 s23 = __fmul2_rn(p23, __fadd2_rn(make_float2(__uint_as_float(dp[col + 2]), __uint_as_float(dp[col + 3])),
                                                                   make_float2(-d4.z, -d4.w)));
                    pw[ci][2 * g4] = pack2(p01.x, p01.y);
                    pw[ci][2 * g4 + 1] = pack2(p23.x, p23.y);
                    dw[ci][2 * g4] = pack2(s01.x, s01.y);
                    dw[ci][2 * g4 + 1] = pack2(s23.x, s23.y);
                }
                continue;
            }
            // pair (this key, query q0 + col) is visible iff lo <= col < hi: hi from Sq, lo from
            // the causal diagonal (key kj <= q + causal_off)
            const int hi = sq - q0;
            const long long lo64 = p.causal ? (long long)kj - coff - q0 : 0ll;
            const int lo = lo64 < -1 ? -1 : (lo64 > 33 ? 33 : (int)lo64);
#pragma unroll
            for (int g4 = 0; g4 < 8; ++g4) {
                const float4 l4 = ld_shared_f4(s_lse2 + (uint32_t)(4 * (32 * c + 4 * g4)));
                const float4 d4 = ld_shared_f4(s_delta + (uint32_t)(4 * (32 * c + 4 * g4)));
                const int col = 4 * g4;
                const float2 x01 = __ffma2_rn(make_float2(__uint_as_float(sv[col]), __uint_as_float(sv[col + 1])), c2,
                                              make_float2(-l4.x, -l4.y));
                const float2 x23 = __ffma2_rn(make_float2(__uint_as_float(sv[col + 2]), __uint_as_float(sv[col + 3])), c2,
                                              make_float2(-l4.z, -l4.w));
                float2 p01 = make_float2(ptx::ex2_approx(x01.x), ptx::ex2_approx(x01.y));
                float2 p23 = make_float2(ptx::ex2_approx(x23.x), ptx::ex2_approx(x23.y));
                float2 s01 = __fmul2_rn(p01, __fadd2_rn(make_float2(__uint_as_float(dp[col]), __uint_as_float(dp[col + 1])),
                                                         make_float2(-d4.x, -d4.y)));
                float2 s23 = __fmul2_rn(p23, __fadd2_rn(make_float2(__uint_as_float(dp[col + 2]), __uint_as_float(dp[col + 3])),
                                                         make_float2(-d4.z, -d4.w)));
                // a masked pair takes no part: both zero, even where D is NaN (a query with no
                // visible key has a NaN output row); selects, no branches
                const bool v0 = (col >= lo) & (col < hi), v1 = (col + 1 >= lo) & (col + 1 < hi);
                const bool v2 = (col + 2 >= lo) & (col + 2 < hi), v3 = (col + 3 >= lo) & (col + 3 < hi);
                p01.x = v0 ? p01.x : 0.0f; s01.x = v0 ? s01.x : 0.0f;
                p01.y = v1 ? p01.y : 0.0f; s01.y = v1 ? s01.y : 0.0f;
                p23.x = v2 ? p23.x : 0.0f; s23.x = v2 ? s23.x : 0.0f;
                p23.y = v3 ? p23.y : 0.0f; s23.y = v3 ? s23.y : 0.0f;
                pw[ci][2 * g4] = pack2(p01.x, p01.y);
                pw[ci][2 * g4 + 1] = pack2(p23.x, p23.y);
                dw[ci][2 * g4] = pack2(s01.x, s01.y);
                dw[ci][2 * g4 + 1] = pack2(s23.x, s23.y);
            }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(kBarRead));
        ok = bwd_wait(bar(kBarRead), s & 1u, kSiteRead, abort_flag, lim);
        if (!__all_sync(0xFFFFFFFFu, ok)) return false;
        ptx::tc_fence_after();
#pragma unroll
        for (int ci = 0; ci < 2; ++ci) {
            const int c = 2 * half + ci;
            ptx::tmem_st16(tS + lane_off + 16u * c, pw[ci]);
            ptx::tmem_st16(tDP + lane_off + 16u * c, dw[ci]);
            // dS^T row `row`, queries 32c..32c+31: 16-byte pieces (c & 1)*4 + v of the 64-query
            // chunk c >> 1, at piece ^ (row & 7) (128-byte swizzle)
            const uint32_t rowaddr = sbase + G::kSmemDS + (uint32_t)((c >> 1) * kChunkBytes) + (uint32_t)row * 128u;
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
                const uint32_t pc = (uint32_t)((c & 1) * 4 + v4);
                ptx::st_shared_v4(rowaddr + ((pc ^ (uint32_t)(row & 7)) << 4), dw[ci][4 * v4], dw[ci][4 * v4 + 1],
                                  dw[ci][4 * v4 + 2], dw[ci][4 * v4 + 3]);
            }
        }
        ptx::tmem_wait_st();
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(kBarPFull));
        return true;
    };

    if (warp == kWarpTma && lane == 0) {
        // -------------------------------------------------------------------- TMA producer
        const uint64_t pol_kv = ptx::policy_evict_last();
        const uint64_t pol_q = ptx::policy_evict_last();
        uint32_t s = 0, u = 0, q_issued = 0;
        bool ok = true;
        // dQ of step t is staged in stage t % 2 by the P/dS warps; this thread adds it into the
        // fp32 accumulator with 8 * (D/64) TMA reductions (one 32 x 32 box per warp and 32
        // columns) just before it refills the stage, and waits for them to have read it.  Doing
        // this here rather than in the staging warps keeps the TMA unit's queue (a step's 64 KB
        // of reductions) off their path.  In the deterministic mode the same boxes are stored,
        // not added, into the slice of the unit's key tile ([key tile][B*H][Sq][d]); each
        // (key tile, query row) is written by one step only, and the final kernel adds the
        // slices in key-tile order.
        int hist_it[kStages] = {0, 0}, hist_bh[kStages] = {0, 0}, hist_jt[kStages] = {0, 0};
        int hist_b[kStages] = {0, 0};      // (variable-length batches) the sequence, for its dQ map
        // the preprocessing kernel's D, LSE and zeroed accumulator are waited for once, before
        // the first statistics load (every reduction comes after it), and in any case before
        // exit, so this grid's completion implies that kernel's
        bool dep_done = false;
        auto dep_wait = [&]() {
            if (!dep_done) asm volatile("griddepcontrol.wait;" ::: "memory");
            dep_done = true;
        };
        auto reduce_step = [&](uint32_t t) -> bool {
            const uint32_t tg = t % kStages;
            if (!bwd_wait(bar(kBarStaged + tg), (t / kStages) & 1u, kSiteDQEmpty, abort_flag, lim)) return false;
            const uint32_t stage = sbase + G::kSmemStage0 + tg * G::kStageBytes;
            constexpr int kHC = D / 2;
#pragma unroll
            for (int w = 0; w < 8; ++w)
#pragma unroll
                for (int cc = 0; cc < kHC / 32; ++cc) {
                    const uint32_t src = stage + (uint32_t)((w * (kHC / 32) + cc) * 4096);
                    const int x = kHC * (w >> 2) + 32 * cc, y = hist_it[tg] * kBM + 32 * (w & 3);
                    if constexpr (kDet) ptx::tma_store_4d(&dqmap, src, x, y, hist_bh[tg], hist_jt[tg]);
                    else if constexpr (kVarlen) tma_reduce_add_3d(p.vl_maps + 7 * hist_b[tg] + 6, src, x, y, hist_bh[tg]);
                    else tma_reduce_add_3d(&dqmap, src, x, y, hist_bh[tg]);
                }
            ptx::bulk_commit();
            return true;
        };
        // Q_i and dO_i of step s into its ring stage, once the stage's previous occupant (step
        // s - 2) has had its last GEMM and its dQ, staged there afterwards, has gone out and
        // been read
        auto load_q = [&](const Unit& un, int st, uint32_t s) -> bool {
            const int h = un.kvh * p.group + st % p.group;
            const int it = un.it_lo + st / p.group;
            const uint32_t sg = s % kStages;
            if (s >= (uint32_t)kStages) {
                if (!(bwd_wait(bar(kBarQEmpty + sg), ((s / kStages) - 1u) & 1u, kSiteQEmpty, abort_flag, lim) &&
                      reduce_step(s - kStages)))
                    return false;
                ptx::bulk_wait_read0();
            }
            ptx::mbar_arrive_expect_tx(bar(kBarQFull + sg), 2 * G::kTileBytes);
            const uint32_t qd = sbase + G::kSmemStage0 + sg * G::kStageBytes;
            for (int c = 0; c < G::kChunks; ++c) {
                const uint32_t dq = qd + c * kChunkBytes, dd = qd + G::kTileBytes + c * kChunkBytes;
                if constexpr (kVarlen) {
                    // the sequence's own maps, token-major, batch coordinate 0
                    ptx::tma_load_4d(dq, p.vl_maps + 7 * un.b + 0, bar(kBarQFull + sg), c * 64, h, it * kBM, 0, pol_q);
                    ptx::tma_load_4d(dd, p.vl_maps + 7 * un.b + 1, bar(kBarQFull + sg), c * 64, h, it * kBM, 0, pol_q);
                } else if (p.bshd) {
                    ptx::tma_load_4d(dq, &qmap, bar(kBarQFull + sg), c * 64, h, it * kBM, un.b, pol_q);
                    ptx::tma_load_4d(dd, &domap, bar(kBarQFull + sg), c * 64, h, it * kBM, un.b, pol_q);
                } else {
                    ptx::tma_load_4d(dq, &qmap, bar(kBarQFull + sg), c * 64, it * kBM, h, un.b, pol_q);
                    ptx::tma_load_4d(dd, &domap, bar(kBarQFull + sg), c * 64, it * kBM, h, un.b, pol_q);
                }
            }
            hist_it[sg] = it;
            hist_bh[sg] = kVarlen ? h : un.b * p.H + h;
            hist_jt[sg] = un.jt;
            hist_b[sg] = un.b;
            ++q_issued;
            return true;
        };
        // coordinates 1 and 2 of a unit's K_j, V_j boxes (the layout's order)
        auto kv_coords = [&](const Unit& un, int& c1, int& c2) {
            c1 = p.bshd ? un.kvh : un.jt * kBN;
            c2 = p.bshd ? un.jt * kBN : un.kvh;
        };
        for (int n = 0, k = sched_pos<kVarlen>(p, 0); k < n_items && ok; k = sched_pos<kVarlen>(p, ++n), ++u) {
            const Unit un = decode_item<kVarlen>(p, k);
            if constexpr (kVarlen) {
                // the sequence's maps (written by the planning kernel) before their first use;
                // a sequence without queries has no Q, dO or dQ maps and its units no steps
                const CUtensorMap* m = p.vl_maps + 7 * un.b;
                ptx::tensormap_acquire(m + 2);
                ptx::tensormap_acquire(m + 3);
                if (un.st1 > un.st0) {
                    ptx::tensormap_acquire(m + 0);
                    ptx::tensormap_acquire(m + 1);
                    ptx::tensormap_acquire(m + 6);
                }
            }
            // the unit's first Q/dO goes in before the wait for the previous unit's K/V to be
            // released, so that it does not wait behind that unit's last GEMMs
            if (un.st1 > un.st0 && !(ok = load_q(un, un.st0, s))) break;
            if (u > 0 && !(ok = bwd_wait(bar(kBarKVEmpty), (u - 1) & 1u, kSiteKVEmpty, abort_flag, lim))) break;
            ptx::mbar_arrive_expect_tx(bar(kBarKV), 2 * G::kTileBytes);
            for (int c = 0; c < G::kChunks; ++c) {
                const uint32_t dk = sbase + G::kSmemK + c * kChunkBytes, dv = sbase + G::kSmemV + c * kChunkBytes;
                if constexpr (kVarlen) {
                    ptx::tma_load_4d(dk, p.vl_maps + 7 * un.b + 2, bar(kBarKV), c * 64, un.kvh, un.jt * kBN, 0, pol_kv);
                    ptx::tma_load_4d(dv, p.vl_maps + 7 * un.b + 3, bar(kBarKV), c * 64, un.kvh, un.jt * kBN, 0, pol_kv);
                } else {
                    int c1, c2;
                    kv_coords(un, c1, c2);
                    ptx::tma_load_4d(dk, &kmap, bar(kBarKV), c * 64, c1, c2, un.b, pol_kv);
                    ptx::tma_load_4d(dv, &vmap, bar(kBarKV), c * 64, c1, c2, un.b, pol_kv);
                }
            }
            for (int st = un.st0; st < un.st1 && ok; ++st, ++s) {
                const int h = un.kvh * p.group + st % p.group;
                const int it = un.it_lo + st / p.group;
                if (st > un.st0 && !(ok = load_q(un, st, s))) break;
                // the statistics buffer is free once the previous step's P^T/dS^T are done
                if (s > 0 && !(ok = bwd_wait(bar(kBarPFull), (s - 1) & 1u, kSitePFull, abort_flag, lim))) break;
                dep_wait();
                ptx::mbar_arrive_expect_tx(bar(kBarStats), 2 * kBM * 4);
                const long long srow = kVarlen ? (long long)h * p.stat_stride + un.pad + (long long)it * kBM
                                               : ((long long)un.b * p.H + h) * p.nq_pad_rows + (long long)it * kBM;
                ptx::bulk_load_1d(sbase + G::kSmemStats, p.lse2 + srow, kBM * 4, bar(kBarStats));
                ptx::bulk_load_1d(sbase + G::kSmemStats + kBM * 4, p.delta + srow, kBM * 4, bar(kBarStats));
            }
        }
        // the last steps' dQ (at most two stages' worth) goes out after the loop
        for (uint32_t t = (s > (uint32_t)kStages ? s - kStages : 0u); t < s && ok; ++t) ok = reduce_step(t);
        ptx::bulk_wait0();
        // every issued load has landed before the CTA may exit
        if (u > 0) {
            const uint64_t t0 = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(bar(kBarKV), (u - 1) & 1u) && ptx::globaltimer_ns() - t0 < lim) {
            }
        }
        for (uint32_t n = (q_issued > (uint32_t)kStages ? q_issued - kStages : 0u); n < q_issued; ++n) {
            const uint64_t t0 = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(bar(kBarQFull + n % kStages), (n / kStages) & 1u) &&
                   ptx::globaltimer_ns() - t0 < lim) {
            }
        }
        if (q_issued > 0) {
            const uint64_t t0 = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(bar(kBarStats), (s - 1) & 1u) && ptx::globaltimer_ns() - t0 < lim) {
            }
        }
        dep_wait();
    } else if (warp == kWarpMma && lane == 0) {
        // -------------------------------------------------------------------- MMA issuer
        constexpr uint32_t idesc_s = idesc_bf16(kBN, kBM, false, false);  // K-major x K-major
        constexpr uint32_t idesc_o = idesc_bf16(kBN, D, false, true);     // TMEM A x MN-major B
        constexpr uint32_t idesc_q = idesc_bf16(kBM, D, true, true);      // MN-major A x MN-major B
        const uint64_t dK_k = sdesc(sbase + G::kSmemK, 16, 1024), dV_k = sdesc(sbase + G::kSmemV, 16, 1024);
        // stage 0's Q and dO; stage 1 is G::kStageBytes further (added to the address field)
        const uint64_t dQ_k = sdesc(sbase + G::kSmemStage0, 16, 1024);
        const uint64_t dDO_k = sdesc(sbase + G::kSmemStage0 + G::kTileBytes, 16, 1024);
        const uint64_t dQ_mn = sdesc(sbase + G::kSmemStage0, kChunkBytes, 1024);
        const uint64_t dDO_mn = sdesc(sbase + G::kSmemStage0 + G::kTileBytes, kChunkBytes, 1024);
        const uint64_t dDS_mn = sdesc(sbase + G::kSmemDS, kChunkBytes, 1024);
        const uint64_t dK_mn = sdesc(sbase + G::kSmemK, kChunkBytes, 1024);
        // D = A B^T over d: 8 K-steps of 16 (32 B inside a 64-column half, then the other half)
        auto gemm_kk = [&](uint32_t d, uint64_t a, uint64_t b) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t off = (uint64_t)(((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4);
                ptx::mma_ss(d, a + off, b + off, idesc_s, kk > 0 ? 1u : 0u);
            }
        };
        // D (+)= A[TMEM] B over 128 queries: 8 K-steps of 16 (8 TMEM columns of bf16 pairs; 2 KB of B)
        auto gemm_tm = [&](uint32_t d, uint32_t a, uint64_t b, bool acc) {
#pragma unroll
            for (int kk = 0; kk < kBM / 16; ++kk)
                ptx::mma_ts(d, a + (uint32_t)kk * 8u, b + (uint64_t)((kk * 2048) >> 4), idesc_o,
                            (kk > 0 || acc) ? 1u : 0u);
        };
        // dQ = dS K over 128 keys: both operands MN-major, 8 K-steps of 16 rows (2 KB each)
        auto gemm_mm = [&](uint32_t d, uint64_t a, uint64_t b) {
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
                ptx::mma_ss(d, a + (uint64_t)((kk * 2048) >> 4), b + (uint64_t)((kk * 2048) >> 4), idesc_q,
                            kk > 0 ? 1u : 0u);
        };
        uint32_t s = 0, u = 0;
        bool ok = true;
        for (int n = 0, k = sched_pos<kVarlen>(p, 0); k < n_items && ok; k = sched_pos<kVarlen>(p, ++n), ++u) {
            const Unit un = decode_item<kVarlen>(p, k);
            if (!(ok = bwd_wait(bar(kBarKV), u & 1u, kSiteKV, abort_flag, lim))) break;
            for (int st = un.st0; st < un.st1 && ok; ++st, ++s) {
                const uint32_t sg = s % kStages;
                const uint64_t so = (uint64_t)((sg * G::kStageBytes) >> 4);
                if (!(ok = bwd_wait(bar(kBarQFull + sg), (s / kStages) & 1u, kSiteQFull, abort_flag, lim))) break;
                ptx::tc_fence_after();
                gemm_kk(tS, dK_k, dQ_k + so);        // S^T = K_j Q_i^T
                ptx::mma_commit(bar(kBarSFull));
                // TMEM columns 128..255 hold the previous dQ until it has been read out
                if (s > 0 && !(ok = bwd_wait(bar(kBarDQEmpty), (s - 1) & 1u, kSiteDQEmpty, abort_flag, lim))) break;
                ptx::tc_fence_after();
                gemm_kk(tDP, dV_k, dDO_k + so);      // dP^T = V_j dO_i^T
                ptx::mma_commit(bar(kBarDPFull));
                if (!(ok = bwd_wait(bar(kBarPFull), s & 1u, kSitePFull, abort_flag, lim))) break;
                // the previous unit's dK, dV have been read before the first step overwrites them
                if (st == un.st0 && u > 0 && !(ok = bwd_wait(bar(kBarDKVEmpty), (u - 1) & 1u, kSiteDKVEmpty, abort_flag, lim)))
                    break;
                ptx::tc_fence_after();
                gemm_tm(tDV, tS, dDO_mn + so, st > un.st0);    // dV += P^T dO_i
                gemm_tm(tDK, tDP, dQ_mn + so, st > un.st0);    // dK += dS^T Q_i
                ptx::mma_commit(bar(kBarQEmpty + sg));
                gemm_mm(tDQ, dDS_mn, dK_mn);              // dQ_i = dS K_j
                ptx::mma_commit(bar(kBarDQFull));
            }
            if (!ok) break;
            if (un.st1 == un.st0 && u > 0 &&
                !(ok = bwd_wait(bar(kBarDKVEmpty), (u - 1) & 1u, kSiteDKVEmpty, abort_flag, lim)))
                break;
            // (test hook: CTA 0 withholds its first unit's dK/dV-ready signal, so that the
            // writer's bounded wait expires)
            if (!(p.test_hooks && u == 0 && blockIdx.x == 0)) ptx::mma_commit(bar(kBarDKVFull));
            ptx::mma_commit(bar(kBarKVEmpty));
        }
        ptx::mma_commit(bar(kBarDrain));
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(bar(kBarDrain), 0) && ptx::globaltimer_ns() - t0 < lim) {
        }
    } else if (warp < 8) {
        // -------------------------------------------------------------------- P^T, dS^T and dQ; dK, dV out
        // Warpgroup `half` forms P^T and dS^T for query columns 64*half .. 64*half + 63 of each
        // step, then drains its half of dQ_i's columns; at the end of a unit warpgroup 0 writes
        // dV and warpgroup 1 dK.  Splitting this work keeps both warpgroups equally loaded: with
        // one warpgroup draining all of dQ it reached the next step ~1200 cycles after the
        // other, which waited for it where the two meet.
        const int half = warp >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        constexpr int kHC = D / 2;              // dQ columns per warpgroup
        // staging for dQ_i: the step's own Q/dO stage, which its last GEMMs have read by the time
        // dQ_i is ready and which is not refilled before these reductions have read it; one 4 KB
        // box (32 rows x 32 fp32) per warp and 32 columns
        static_assert(8 * (kHC / 32) * 4096 == G::kStageBytes, "the dQ boxes fill one Q/dO stage");
        uint32_t s = 0, u = 0;
        bool ok = true;
        for (int n = 0, k = sched_pos<kVarlen>(p, 0); k < n_items && ok; k = sched_pos<kVarlen>(p, ++n), ++u) {
            const Unit un = decode_item<kVarlen>(p, k);
            for (int st = un.st0; st < un.st1 && ok; ++st, ++s) {
                if (!(ok = pds_step(un, un.it_lo + st / p.group, s, half))) break;
                ok = bwd_wait(bar(kBarDQFull), s & 1u, kSiteDQFull, abort_flag, lim);
                if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                ptx::tc_fence_after();
                // this warpgroup's half of dQ_i into registers, then release TMEM; per 32 columns,
                // this warp's 32 rows (times 1/sqrt(d)) into its staging box in the 128-byte
                // swizzle; the producer thread then adds the boxes into the fp32 dQ accumulator
                // with TMA reductions.  The TMA unit does the additions: per-thread atomics here
                // stalled the MMA thread's issue.
                uint32_t v[kHC];
                if constexpr (kHC == 64) ptx::tmem_ld64(tDQ + lane_off + 64u * half, v);
                else ptx::tmem_ld32(tDQ + lane_off + 32u * half, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(kBarDQEmpty));
#pragma unroll
                for (int cc = 0; cc < kHC / 32; ++cc) {
                    const uint32_t box = sbase + G::kSmemStage0 + (s % kStages) * G::kStageBytes +
                                         (uint32_t)(((half * 4 + quarter) * (kHC / 32) + cc) * 4096);
                    const uint32_t rowaddr = box + (uint32_t)lane * 128u;
#pragma unroll
                    for (int pc = 0; pc < 8; ++pc) {
                        const int e = 32 * cc + 4 * pc;
                        ptx::st_shared_v4(rowaddr + (((uint32_t)pc ^ (uint32_t)(lane & 7)) << 4),
                                          __float_as_uint(__uint_as_float(v[e]) * p.scale),
                                          __float_as_uint(__uint_as_float(v[e + 1]) * p.scale),
                                          __float_as_uint(__uint_as_float(v[e + 2]) * p.scale),
                                          __float_as_uint(__uint_as_float(v[e + 3]) * p.scale));
                    }
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(kBarStaged + (int)(s % kStages)));
            }
            if (!ok) continue;
            // warpgroup h writes its tensor (0: dV, 1: dK times 1/sqrt(d)) through box h of the
            // dS^T region (16 KB, 128 rows x 64 columns; the region is free from the unit's last
            // GEMMs to the next unit's first dS^T), 64 columns at a time: it reads them out of
            // TMEM and stages them in the box, and one thread stores the box with TMA (rows past
            // Skv are clipped) and waits for the store to have read it before the box is
            // refilled.  The two warpgroups work on their own boxes at the same time.  (One
            // warpgroup writing all of dK and dV row by row took ~5000-8000 cycles per unit;
            // the two tiles staged one after the other through the whole region, ~7000.)
            ok = bwd_wait(bar(kBarDKVFull), u & 1u, kSiteDKVFull, abort_flag, lim);
            if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
            ptx::tc_fence_after();
            // a split item's dV/dK are partial sums: they go, unscaled and in fp32, to the item's
            // row of the workspace (plain stores; one split item per CTA at most), and the final
            // kernel adds the parts in order.  The barrier steps below run the same either way.
            const bool split = un.slot >= 0;
            const float sc = half ? p.scale : 1.0f;
            const uint32_t box = sbase + G::kSmemDS + (uint32_t)(half * kChunkBytes);
#pragma unroll 1
            for (int cc = 0; cc < D / 64 && ok; ++cc) {
                const uint32_t rnd = u * (uint32_t)(D / 64) + (uint32_t)cc;   // this warpgroup's round
                // the box's previous store (this warpgroup's last round) has read it
                if (rnd > 0) {
                    ok = bwd_wait(bar(kBarBoxFree + half), (rnd - 1u) & 1u, kSiteOutFree, abort_flag, lim);
                    if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                }
#pragma unroll 1
                for (int c2 = 0; c2 < 2; ++c2) {
                    const int c = 2 * cc + c2;              // 32-column chunk of the row
                    uint32_t v[32];
                    if (un.st1 > un.st0) {
                        ptx::tmem_ld32((half ? tDK : tDV) + lane_off + 32u * c, v);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = 0u;
                    }
                    if (split) {
                        float4* dst = reinterpret_cast<float4*>(
                            p.ws_dkv + ((size_t)(un.slot * 2 + half) * kBN + (size_t)row) * D + 32 * c);
#pragma unroll
                        for (int v4 = 0; v4 < 8; ++v4)
                            dst[v4] = make_float4(__uint_as_float(v[4 * v4]), __uint_as_float(v[4 * v4 + 1]),
                                                  __uint_as_float(v[4 * v4 + 2]), __uint_as_float(v[4 * v4 + 3]));
                        continue;
                    }
                    // row `row` of the box, columns 32*c2 .. +31: 16-byte pieces c2*4 + v4 at
                    // piece ^ (row & 7) (the tensor map's 128-byte swizzle)
                    const uint32_t rowaddr = box + (uint32_t)row * 128u;
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        const uint32_t pc = (uint32_t)(c2 * 4 + v4);
                        const int e = 8 * v4;
                        ptx::st_shared_v4(rowaddr + ((pc ^ (uint32_t)(row & 7)) << 4),
                                          pack2(__uint_as_float(v[e]) * sc, __uint_as_float(v[e + 1]) * sc),
                                          pack2(__uint_as_float(v[e + 2]) * sc, __uint_as_float(v[e + 3]) * sc),
                                          pack2(__uint_as_float(v[e + 4]) * sc, __uint_as_float(v[e + 5]) * sc),
                                          pack2(__uint_as_float(v[e + 6]) * sc, __uint_as_float(v[e + 7]) * sc));
                    }
                }
                if (cc == D / 64 - 1) {                       // TMEM read out: the next unit may start
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar(kBarDKVEmpty));
                }
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive(bar(kBarOutStaged + half));
                if (quarter == 0) {
                    if (lane == 0) {
                        ok = bwd_wait(bar(kBarOutStaged + half), rnd & 1u, kSiteOutStaged, abort_flag, lim);
                        if (ok) {
                            if (!split) {
                                if constexpr (kVarlen) {
                                    const CUtensorMap* om = p.vl_maps + 7 * un.b + (half ? 4 : 5);
                                    if (cc == 0) ptx::tensormap_acquire(om);
                                    ptx::tma_store_4d(om, box, cc * 64, un.kvh, un.jt * kBN, 0);
                                } else {
                                    const int y1 = p.bshd ? un.kvh : un.jt * kBN;
                                    const int y2 = p.bshd ? un.jt * kBN : un.kvh;
                                    ptx::tma_store_4d(half ? (const void*)&dkmap : (const void*)&dvmap, box, cc * 64,
                                                      y1, y2, un.b);
                                }
                                ptx::bulk_commit();
                                ptx::bulk_wait_read0();
                            }
                            ptx::mbar_arrive(bar(kBarBoxFree + half));
                        }
                    }
                    ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
                }
            }
            if (!ok) break;
        }
        // the dK, dV stores complete before the CTA exits
        if (quarter == 0 && lane == 0) ptx::bulk_wait0();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// Preprocessing, one pass over O and dO: D_i = dO_i . O_i in fp32, the base-2 log-sum-exp,
// and zeros into query row i of the fp32 dQ accumulator (when there is one: the deterministic
// mode stores every slice row it reads and needs no zeros).  D / 8 lanes per padded query row,
// 8 columns (16-byte loads) per lane, grid-stride over rows; padded rows (q >= Sq) get D_i = 0
// and LSE 0 and have no accumulator row.  The row count is a multiple of 128, so every warp's
// rows are all in range or all out and its shuffles see all 32 lanes.  This kernel is itself a
// programmatic dependent of the stream's previous kernel (which may have written O, dO or the
// LSE, or still read the accumulator) and waits for its memory first.  The main kernel is this
// kernel's programmatic dependent: it may launch once every CTA here is past that wait, and
// its producer waits for this kernel's memory before the first statistics load or reduction.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const __nv_bfloat16* o, const __nv_bfloat16* dout,
                                                            const float* lse, float* lse2, float* delta,
                                                            float* dq_acc, int H, int Sq, int nq_pad_rows,
                                                            long long rows, long long o_sb, long long o_ss,
                                                            long long o_sh) {
    constexpr int kL = D / 8;                  // lanes per row: 16 or 8
    constexpr int kRows = 256 / kL;            // rows per block and pass
    // wait before letting the main kernel launch: it loads Q, K, V and dO before it waits for
    // this kernel, so it must not start before the previous kernel is done
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int sub = threadIdx.x / kL, c = (threadIdx.x % kL) * 8;
    for (long long r = (long long)blockIdx.x * kRows + sub; r < rows; r += (long long)gridDim.x * kRows) {
        const long long bh = r / nq_pad_rows;
        const int q = (int)(r % nq_pad_rows);
        const int b = (int)(bh / H), h = (int)(bh % H);
        float acc = 0.0f;
        if (q < Sq) {
            const long long off = (long long)b * o_sb + (long long)q * o_ss + (long long)h * o_sh + c;
            const uint4 ov = *reinterpret_cast<const uint4*>(o + off);
            const uint4 gv = *reinterpret_cast<const uint4*>(dout + off);
            const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[e]));
                const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
                acc = fmaf(of.x, gf.x, acc);
                acc = fmaf(of.y, gf.y, acc);
            }
            if (dq_acc) {
                float4* z = reinterpret_cast<float4*>(dq_acc + (bh * Sq + q) * D + c);
                z[0] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                z[1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
        }
#pragma unroll
        for (int s = kL / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, s);
        if (c == 0) {
            delta[r] = acc;
            lse2[r] = q < Sq ? lse[bh * Sq + q] * 1.4426950408889634f : 0.0f;
        }
    }
}

// The split units' dK, dV: the sum of their parts' fp32 partials, in part order (a fixed
// order, so results are deterministic), dK times 1/sqrt(d), rounded to nearest even.
struct DkvCombine {
    const float* ws;             // [T * P items][2: dV, dK][128][d]
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    int T, P, n_full, nkv, Hkv, Skv;
    long long kv_sb, kv_ss, kv_sh;
    float scale;
};

// The deterministic mode's dQ terms: nkv slices [key tile][B*H][Sq][d] of `slice` elements
// each; key tile j holds a row's terms if the row sees a key of that tile (j * 128 <= q +
// causal_off under the mask), and only those slices are read.  nkv = 0: a plain accumulator.
struct DqSlices {
    int nkv, causal, causal_off;
    long long slice;
};

// The backward's last kernel.  Blocks [0, dq_blocks): dq (bf16, the caller's layout) = dq_acc
// (fp32 [B][H][Sq][d]; in the deterministic mode the sum of the row's key-tile slices, added
// in key-tile order from +0), round to nearest even, 8 columns per thread (16-byte loads, one
// 16-byte store), grid-stride.  Blocks from dq_blocks on: the split units' dK/dV, one warp per
// (unit, tensor, key row), D/32 columns per lane.  Launched as a programmatic dependent of the
// main kernel: it waits for that kernel's memory first.  kDet: the deterministic mode's
// instance (ds.nkv slices), kept apart so that the default one stays as lean as before.
template <int D, bool kDet>
__global__ void __launch_bounds__(256) attn_bwd_dq_kernel(const float* dq_acc, __nv_bfloat16* dq, int H, int Sq,
                                                          long long n8, long long o_sb, long long o_ss,
                                                          long long o_sh, int dq_blocks, const DkvCombine cb,
                                                          const DqSlices ds) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if ((int)blockIdx.x < dq_blocks) {
        for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
             i += (long long)dq_blocks * blockDim.x) {
            const long long row = i / (D / 8);
            const int x = (int)(i % (D / 8)) * 8;
            const int q = (int)(row % Sq);
            const long long bh = row / Sq;
            const int h = (int)(bh % H), b = (int)(bh / H);
            float4 v0, v1;
            if constexpr (!kDet) {
                const float4* src = reinterpret_cast<const float4*>(dq_acc + row * D + x);
                v0 = src[0];
                v1 = src[1];
            } else {
                // key tiles 0..n-1 hold this row's terms
                long long last = ds.nkv - 1;
                if (ds.causal) {
                    const long long lim = (long long)q + ds.causal_off;
                    last = lim < 0 ? -1 : (lim / kBN < last ? lim / kBN : last);
                }
                v0 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                v1 = v0;
                const float* src = dq_acc + row * D + x;
                long long j = 0;
                // four slices' loads in flight, then their adds in order
                for (; j + 3 <= last; j += 4) {
                    float4 t[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float4* s4 = reinterpret_cast<const float4*>(src + (j + e) * ds.slice);
                        t[2 * e] = s4[0];
                        t[2 * e + 1] = s4[1];
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        v0.x += t[2 * e].x; v0.y += t[2 * e].y; v0.z += t[2 * e].z; v0.w += t[2 * e].w;
                        v1.x += t[2 * e + 1].x; v1.y += t[2 * e + 1].y; v1.z += t[2 * e + 1].z; v1.w += t[2 * e + 1].w;
                    }
                }
                for (; j <= last; ++j) {
                    const float4* s4 = reinterpret_cast<const float4*>(src + j * ds.slice);
                    const float4 a = s4[0], c = s4[1];
                    v0.x += a.x; v0.y += a.y; v0.z += a.z; v0.w += a.w;
                    v1.x += c.x; v1.y += c.y; v1.z += c.z; v1.w += c.w;
                }
            }
            __nv_bfloat16* dst = dq + (long long)b * o_sb + (long long)q * o_ss + (long long)h * o_sh + x;
            *reinterpret_cast<uint4*>(dst) = make_uint4(pack2(v0.x, v0.y), pack2(v0.z, v0.w), pack2(v1.x, v1.y),
                                                        pack2(v1.z, v1.w));
        }
        return;
    }
    const long long w = (long long)((int)blockIdx.x - dq_blocks) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= (long long)cb.T * 2 * kBN) return;
    const int r = (int)(w % kBN);
    const int which = (int)((w / kBN) % 2);            // 0: dV, 1: dK
    const int t = (int)(w / (2 * kBN));
    const int unit = cb.n_full + t;
    const int jt = unit % cb.nkv, bk = unit / cb.nkv;
    const int kvh = bk % cb.Hkv, b = bk / cb.Hkv;
    const int kj = jt * kBN + r;
    if (kj >= cb.Skv) return;
    constexpr int kC = D / 32;                         // columns per lane: 4 or 2
    float acc[kC];
#pragma unroll
    for (int e = 0; e < kC; ++e) acc[e] = 0.0f;
    for (int part = 0; part < cb.P; ++part) {
        const float* src = cb.ws + ((size_t)((t * cb.P + part) * 2 + which) * kBN + (size_t)r) * D + lane * kC;
#pragma unroll
        for (int e = 0; e < kC; ++e) acc[e] += src[e];
    }
    const float sc = which ? cb.scale : 1.0f;
    __nv_bfloat16* out = (which ? cb.dk : cb.dv) + (long long)b * cb.kv_sb + (long long)kj * cb.kv_ss +
                         (long long)kvh * cb.kv_sh + lane * kC;
    if constexpr (kC == 4)
        *reinterpret_cast<uint2*>(out) = make_uint2(pack2(acc[0] * sc, acc[1] * sc), pack2(acc[2] * sc, acc[3] * sc));
    else
        *reinterpret_cast<uint32_t*>(out) = pack2(acc[0] * sc, acc[1] * sc);
}

// ------------------------------------------------------------------------------ varlen
// Planning kernel of a variable-length backward, one CTA, first of the four kernels:
//   * checks the offsets (cu_q, cu_k start at >= 0, never decrease, end within the packed
//     tensors); otherwise it records ATTN_ERR_INVALID_ARG at the sequence-length site and
//     schedules no unit, and the later kernels write nothing;
//   * pad[b]: the first padded statistics row of sequence b (its rows rounded up to 128);
//   * per sequence, tensor maps narrowed to its rows (tensormap.replace on copies of the
//     whole-tensor maps, then a release fence for the tensor-map proxy): K, V, dK, dV when it
//     has keys, Q, dO and the dQ accumulator when it also has queries.  Loads past its end read
//     zeros and stores and reductions past its end are dropped, as at a dense tensor's end;
//   * the units (sequence, K/V head, key tile) ordered by their query steps, most first (a
//     counting sort capped at kCostBuckets - 1; equal counts in any order, which moves work
//     between CTAs but changes no result).
constexpr int kCostBuckets = 4096;

struct BwdVarlenPlan {
    const int* cu_q;
    const int* cu_k;
    int B, H, Hkv, group, causal;
    long long total_q, total_k;
    long long q_row_bytes, kv_row_bytes, acc_row_bytes;   // bytes per token row (acc: per head)
    const char* q;
    const char* dout;
    const char* k;
    const char* v;
    char* dk;
    char* dv;
    char* dq_acc;
    CUtensorMap* maps;           // [B][7]: Q, dO, K, V, dK, dV, dQ accumulator
    int4* units;
    int* n_units;
    int* pad;                    // [B + 1]
};

__device__ __forceinline__ void bwd_copy_map(CUtensorMap* dst, const CUtensorMap* src) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(CUtensorMap) / 16); ++i) d4[i] = s4[i];
}

// the map at dst (a copy of a whole-tensor map) moved to `base`, with `rows` rows on axis `ord`
__device__ __forceinline__ void bwd_narrow_map(CUtensorMap* dst, const void* base, int ord, int rows) {
    asm volatile("tensormap.replace.tile.global_address.global.b1024.b64 [%0], %1;" ::"l"(dst),
                 "l"(reinterpret_cast<uint64_t>(base))
                 : "memory");
    if (ord == 1)
        asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(dst), "r"(rows) : "memory");
    else
        asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 2, %1;" ::"l"(dst), "r"(rows) : "memory");
}

// query steps of unit (key tile jt) of a sequence with sq queries and skv keys, per K/V head
__device__ __forceinline__ int unit_steps(int jt, int sq, int skv, int causal, int group) {
    int it_lo = 0;
    if (causal) {
        const int first_q = jt * kBN - (skv - sq);
        it_lo = first_q <= 0 ? 0 : first_q / kBM;
    }
    const int nq = (sq + kBM - 1) / kBM;
    return (it_lo < nq ? nq - it_lo : 0) * group;
}

__global__ void __launch_bounds__(1024) attn_bwd_varlen_plan_kernel(
    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap domap,
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
    const __grid_constant__ CUtensorMap dkmap, const __grid_constant__ CUtensorMap dvmap,
    const __grid_constant__ CUtensorMap accmap, const BwdVarlenPlan a) {
    __shared__ int bad;
    __shared__ int bucket[kCostBuckets];
    __shared__ int warp_sums[32];
    __shared__ int carry;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nthreads = blockDim.x;
    if (tid == 0) {
        bad = (a.cu_q[0] < 0 || a.cu_k[0] < 0 || a.cu_q[a.B] > a.total_q || a.cu_k[a.B] > a.total_k) ? 1 : 0;
        carry = 0;
    }
    for (int i = tid; i < kCostBuckets; i += nthreads) bucket[i] = 0;
    __syncthreads();
    for (int b = tid; b < a.B; b += nthreads)
        if (a.cu_q[b + 1] < a.cu_q[b] || a.cu_k[b + 1] < a.cu_k[b]) bad = 1;
    __syncthreads();
    if (bad) {
        // -1 units: the attention kernel runs nothing and the last kernel writes nothing
        if (tid == 0) {
            *a.n_units = -1;
            if (atomicCAS(&g_bwd_status[0], 0u, (uint32_t)ATTN_ERR_INVALID_ARG) == 0u)
                atomicExch(&g_bwd_status[1], kSiteSeqlens);
        }
        for (int b = tid; b <= a.B; b += nthreads) a.pad[b] = 0;
        return;
    }
    for (int base = 0; base < a.B; base += nthreads) {
        const int b = base + tid;
        int sq = 0, skv = 0, rows = 0;
        if (b < a.B) {
            sq = a.cu_q[b + 1] - a.cu_q[b];
            skv = a.cu_k[b + 1] - a.cu_k[b];
            rows = (sq + kBM - 1) / kBM * kBM;
        }
        // exclusive prefix of the padded statistics rows
        int incl = rows;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) warp_sums[wid] = incl;
        __syncthreads();
        if (wid == 0) {
            int w = lane < (nthreads >> 5) ? warp_sums[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, w, off);
                if (lane >= off) w += y;
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        const int before = carry + (wid > 0 ? warp_sums[wid - 1] : 0) + incl - rows;
        if (b < a.B) {
            a.pad[b] = before;
            CUtensorMap* m = a.maps + 7 * (long long)b;
            const long long q0 = a.cu_q[b], k0 = a.cu_k[b];
            if (skv > 0) {
                bwd_copy_map(m + 2, &kmap);
                bwd_copy_map(m + 3, &vmap);
                bwd_copy_map(m + 4, &dkmap);
                bwd_copy_map(m + 5, &dvmap);
                bwd_narrow_map(m + 2, a.k + k0 * a.kv_row_bytes, 2, skv);
                bwd_narrow_map(m + 3, a.v + k0 * a.kv_row_bytes, 2, skv);
                bwd_narrow_map(m + 4, a.dk + k0 * a.kv_row_bytes, 2, skv);
                bwd_narrow_map(m + 5, a.dv + k0 * a.kv_row_bytes, 2, skv);
                if (sq > 0) {
                    bwd_copy_map(m + 0, &qmap);
                    bwd_copy_map(m + 1, &domap);
                    bwd_copy_map(m + 6, &accmap);
                    bwd_narrow_map(m + 0, a.q + q0 * a.q_row_bytes, 2, sq);
                    bwd_narrow_map(m + 1, a.dout + q0 * a.q_row_bytes, 2, sq);
                    bwd_narrow_map(m + 6, a.dq_acc + q0 * a.acc_row_bytes, 1, sq);
                }
                const int nkv = (skv + kBN - 1) / kBN;
                for (int jt = 0; jt < nkv; ++jt) {
                    const int c = unit_steps(jt, sq, skv, a.causal, a.group);
                    atomicAdd(&bucket[c < kCostBuckets - 1 ? c : kCostBuckets - 1], a.Hkv);
                }
            }
        }
        __syncthreads();
        if (tid == nthreads - 1) carry = before + rows;
        __syncthreads();
    }
    if (tid == 0) a.pad[a.B] = carry;
    // start of each bucket, most steps first: thread t owns buckets kCostBuckets - 4t - 1 down
    // to kCostBuckets - 4t - 4; an exclusive scan of the threads' sums over t
    constexpr int kPer = kCostBuckets / 1024;
    int local = 0;
    for (int i = 0; i < kPer; ++i) local += bucket[kCostBuckets - 1 - kPer * tid - i];
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += y;
    }
    __syncthreads();
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int w = lane < (nthreads >> 5) ? warp_sums[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, w, off);
            if (lane >= off) w += y;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    int start = (wid > 0 ? warp_sums[wid - 1] : 0) + incl - local;
    if (tid == nthreads - 1) *a.n_units = start + local;
    __syncthreads();
    for (int i = 0; i < kPer; ++i) {
        const int key = kCostBuckets - 1 - kPer * tid - i;
        const int c = bucket[key];
        bucket[key] = start;
        start += c;
    }
    __syncthreads();
    for (int b = tid; b < a.B; b += nthreads) {
        const int sq = a.cu_q[b + 1] - a.cu_q[b], skv = a.cu_k[b + 1] - a.cu_k[b];
        const int nkv = (skv + kBN - 1) / kBN;
        for (int jt = 0; jt < nkv; ++jt) {
            const int c = unit_steps(jt, sq, skv, a.causal, a.group);
            const int pos = atomicAdd(&bucket[c < kCostBuckets - 1 ? c : kCostBuckets - 1], a.Hkv);
            for (int h = 0; h < a.Hkv; ++h) a.units[pos + h] = make_int4(b, h, jt, 0);
        }
    }
    asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
}

// Statistics of a variable-length backward, second kernel: per head h and padded row, D = dO . O
// in fp32 and the base-2 LSE at h * stat_stride + pad[b] + i for query i of sequence b (0 in
// the padding rows, as in the dense preprocessing), and zeros into the sequence rows of the
// fp32 dQ accumulator [H][total_q][d].  D / 8 lanes per row, grid-stride; rows past pad[B]
// are not read by anyone.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_varlen_prep_kernel(const __nv_bfloat16* o, const __nv_bfloat16* dout,
                                                                   const float* lse, float* lse2, float* delta,
                                                                   float* dq_acc, const int* cu_q, const int* pad,
                                                                   int B, int H, long long total_q,
                                                                   long long stat_stride) {
    constexpr int kL = D / 8;
    constexpr int kRows = 256 / kL;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int sub = threadIdx.x / kL, c = (threadIdx.x % kL) * 8;
    const long long used = pad[B];
    const long long rows = (long long)H * stat_stride;
    for (long long r = (long long)blockIdx.x * kRows + sub; r < rows; r += (long long)gridDim.x * kRows) {
        const int h = (int)(r / stat_stride);
        const long long pr = r % stat_stride;
        if (pr >= used) continue;             // whole warps: stat_stride and used are multiples of 128
        int lo = 0, hi = B - 1;               // the last b with pad[b] <= pr
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pad[mid] <= pr) lo = mid;
            else hi = mid - 1;
        }
        const long long i = pr - pad[lo];
        const long long q0 = cu_q[lo], sq = cu_q[lo + 1] - q0;
        float acc = 0.0f;
        if (i < sq) {
            const long long off = ((q0 + i) * H + h) * D + c;
            const uint4 ov = *reinterpret_cast<const uint4*>(o + off);
            const uint4 gv = *reinterpret_cast<const uint4*>(dout + off);
            const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[e]));
                const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
                acc = fmaf(of.x, gf.x, acc);
                acc = fmaf(of.y, gf.y, acc);
            }
            float4* z = reinterpret_cast<float4*>(dq_acc + ((long long)h * total_q + q0 + i) * D + c);
            z[0] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            z[1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int sft = kL / 2; sft > 0; sft >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, sft);
        if (c == 0) {
            delta[r] = acc;
            lse2[r] = i < sq ? lse[(long long)h * total_q + q0 + i] * 1.4426950408889634f : 0.0f;
        }
    }
}

// Last kernel of a variable-length backward: dq (bf16, packed [total_q][H][d]) = the fp32
// accumulator [H][total_q][d], round to nearest even, for the query rows of a sequence with
// keys (rows of key-less sequences get zeros, rows outside every sequence are not written).
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_varlen_dq_kernel(const float* dq_acc, __nv_bfloat16* dq,
                                                                 const int* cu_q, const int* cu_k, int B, int H,
                                                                 long long total_q, const int* n_units) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (*n_units < 0) return;                        // offsets rejected: nothing is written
    const long long n8 = total_q * H * (D / 8);
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
        const long long tr = i / (D / 8);             // token row * H + head
        const int x = (int)(i % (D / 8)) * 8;
        const long long r = tr / H;
        const int h = (int)(tr % H);
        int lo = 0, hi = B - 1;                       // the last b with cu_q[b] <= r
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (cu_q[mid] <= r) lo = mid;
            else hi = mid - 1;
        }
        if (r < cu_q[lo] || r >= cu_q[lo + 1]) continue;
        uint4 out = make_uint4(0u, 0u, 0u, 0u);
        if (cu_k[lo + 1] > cu_k[lo]) {
            const float4* src = reinterpret_cast<const float4*>(dq_acc + ((long long)h * total_q + r) * D + x);
            const float4 v0 = src[0], v1 = src[1];
            out = make_uint4(pack2(v0.x, v0.y), pack2(v0.z, v0.w), pack2(v1.x, v1.y), pack2(v1.z, v1.w));
        }
        *reinterpret_cast<uint4*>(dq + tr * D + x) = out;
    }
}

// ------------------------------------------------------------------------------ host side
std::mutex g_bwd_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_bwd_encode = nullptr;
bool g_bwd_attr[64] = {};

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The fp32 dQ accumulator [B*H][Sq][d] for TMA reductions: box 32 columns x 32 rows, 128-byte
// swizzle (32 fp32 = 128 bytes per row); rows past Sq are out of range and skipped.
bool encode_dq(CUtensorMap* m, float* ptr, int64_t BH, int64_t Sq, int64_t d) {
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)Sq, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)(d * 4), (cuuint64_t)(Sq * d * 4)};
    cuuint32_t box[3] = {32, 32, 1}, estr[3] = {1, 1, 1};
    return g_bwd_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The deterministic mode's dQ slices [nkv][B*H][Sq][d] fp32 for TMA tile stores: the same
// 32 x 32 boxes and swizzle, one more coordinate for the key tile.
bool encode_dq_slices(CUtensorMap* m, float* ptr, int64_t nkv, int64_t BH, int64_t Sq, int64_t d) {
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)Sq, (cuuint64_t)BH, (cuuint64_t)nkv};
    cuuint64_t strides[3] = {(cuuint64_t)(d * 4), (cuuint64_t)(Sq * d * 4), (cuuint64_t)(BH * Sq * d * 4)};
    cuuint32_t box[4] = {32, 32, 1, 1}, estr[4] = {1, 1, 1, 1};
    return g_bwd_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ptr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode(CUtensorMap* m, const void* ptr, int64_t B, int64_t H, int64_t S, int64_t d, bool bshd) {
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
    dims[0] = (cuuint64_t)d;
    if (bshd) {
        dims[1] = H; dims[2] = S; dims[3] = B;
        strides[0] = d * 2; strides[1] = H * d * 2; strides[2] = S * H * d * 2;
        box[0] = 64; box[1] = 1; box[2] = kBM; box[3] = 1;
    } else {
        dims[1] = S; dims[2] = H; dims[3] = B;
        strides[0] = d * 2; strides[1] = S * d * 2; strides[2] = H * S * d * 2;
        box[0] = 64; box[1] = kBM; box[2] = 1; box[3] = 1;
    }
    return g_bwd_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int check_shape(const attn_bwd_args_t& a) {
    if (a.B < 1 || a.H < 1 || a.Hkv < 1 || a.Sq < 1 || a.Skv < 1 || a.d < 1) return ATTN_ERR_INVALID_ARG;
    if (a.H % a.Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (a.layout != ATTN_LAYOUT_BSHD && a.layout != ATTN_LAYOUT_BHSD) return ATTN_ERR_INVALID_ARG;
    if ((a.causal != 0 && a.causal != 1) || a.wait_limit_ms < 0) return ATTN_ERR_INVALID_ARG;
    if (a.test_hooks != 0 && a.test_hooks != ATTN_TEST_WITHHOLD_O_READY) return ATTN_ERR_INVALID_ARG;
    if (a.deterministic != 0 && a.deterministic != 1) return ATTN_ERR_INVALID_ARG;
    if (a.d != 128 && a.d != 64) return ATTN_ERR_UNSUPPORTED;
    const int64_t lim = (int64_t)1 << 30;
    if (a.Sq > lim || a.Skv > lim || a.B * a.H > lim || a.B * a.Hkv * cdiv(a.Skv, kBN) > lim ||
        a.B * a.H * cdiv(a.Sq, kBM) * kBM > lim)
        return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

// dQ elements held in the workspace: the accumulator, or one slice per key tile
int64_t dq_elems(const attn_bwd_args_t& a) {
    return (a.deterministic ? cdiv(a.Skv, kBN) : 1) * a.B * a.H * a.Sq * a.d;
}

size_t ws_bytes(const attn_bwd_args_t& a) {
    const int64_t rows_pad = a.B * a.H * cdiv(a.Sq, kBM) * kBM;
    return (size_t)dq_elems(a) * 4u + (size_t)(2 * rows_pad * 4);
}

// Query-range split of the units of the last, partial round (none for causal launches, whose
// units run on the paired schedule).  With T = units mod G left over (or all units when there
// are fewer than G), each is cut into P parts of at least kMinSplitSteps query steps, P chosen
// to minimise the longest CTA's load in the tail, ceil(T P / G) * (ceil(steps / P) + 3) (a
// part costs about three steps more than its steps: its K/V load, its pipeline fill and its
// partials' write; with one step of overhead the square backward split its 112 tail units 4
// ways and lost 5 %), the fewest parts among equals, with T P at most 4 G.  P = 1: nothing
// split.
constexpr int64_t kMinSplitSteps = 4;
struct BwdSplit {
    int64_t T, P;
};
BwdSplit bwd_split(const attn_bwd_args_t& a, int64_t G) {
    if (a.causal || G < 1) return {0, 1};
    const int64_t n_units = a.B * a.Hkv * cdiv(a.Skv, kBN);
    const int64_t steps = (a.H / a.Hkv) * cdiv(a.Sq, kBM);
    const int64_t T = n_units % G;
    if (T == 0) return {0, 1};
    int64_t bestP = 1, best = steps + 3;
    for (int64_t P = 2; P * kMinSplitSteps <= steps && T * P <= 4 * G; ++P) {
        const int64_t cost = cdiv(T * P, G) * (cdiv(steps, P) + 3);
        if (cost < best) {
            best = cost;
            bestP = P;
        }
    }
    return bestP > 1 ? BwdSplit{T, bestP} : BwdSplit{0, 1};
}

// the split partials' bytes: [T * P][2][128][d] fp32
size_t split_bytes(const attn_bwd_args_t& a, const BwdSplit& sp) {
    return (size_t)(sp.T * sp.P * 2 * kBN * a.d * 4);
}

// SM count of the current device (0 if there is none): the split depends on it
int64_t current_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return sms;
}

// The tensor-map encoder and, once per device, the kernels' shared-memory limits.
int bwd_setup(int dev) {
    std::lock_guard<std::mutex> g(g_bwd_mutex);
    if (!g_bwd_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) !=
                cudaSuccess ||
            qr != cudaDriverEntryPointSuccess || !fn)
            return ATTN_ERR_CUDA;
        g_bwd_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    if (!g_bwd_attr[dev]) {
        const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
        if (cudaFuncSetAttribute(attn_bwd_kernel<128, false>, attr, smem_alloc<128>()) != cudaSuccess ||
            cudaFuncSetAttribute(attn_bwd_kernel<64, false>, attr, smem_alloc<64>()) != cudaSuccess ||
            cudaFuncSetAttribute(attn_bwd_kernel<128, true>, attr, smem_alloc<128>()) != cudaSuccess ||
            cudaFuncSetAttribute(attn_bwd_kernel<64, true>, attr, smem_alloc<64>()) != cudaSuccess ||
            cudaFuncSetAttribute(attn_bwd_kernel<128, false, true>, attr, smem_alloc<128>()) != cudaSuccess ||
            cudaFuncSetAttribute(attn_bwd_kernel<64, false, true>, attr, smem_alloc<64>()) != cudaSuccess)
            return ATTN_ERR_CUDA;
        g_bwd_attr[dev] = true;
    }
    return ATTN_OK;
}

int check_varlen(const attn_bwd_varlen_args_t& a) {
    if (a.B < 1 || a.H < 1 || a.Hkv < 1 || a.total_q < 0 || a.total_k < 0 || a.d < 1) return ATTN_ERR_INVALID_ARG;
    if (a.H % a.Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if ((a.causal != 0 && a.causal != 1) || a.wait_limit_ms < 0 || a.reserved != 0 || a.reserved2 != 0)
        return ATTN_ERR_INVALID_ARG;
    if (a.d != 128 && a.d != 64) return ATTN_ERR_UNSUPPORTED;
    const int64_t lim = (int64_t)1 << 30;
    if (a.total_q > lim || a.total_k > lim || a.B > lim || a.H > lim || a.total_q + 127 * a.B > lim ||
        a.Hkv * (a.total_k / kBN + a.B) > lim)
        return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

// padded statistics rows per head: each sequence's queries rounded up to 128
int64_t varlen_stat_stride(const attn_bwd_varlen_args_t& a) { return cdiv(a.total_q + 127 * a.B, kBM) * kBM; }

// workspace: dQ accumulator | base-2 LSE | D | tensor maps (128-byte aligned) | item count and
// padded offsets | units
struct VarlenWs {
    size_t acc, stats, maps, misc, units, total;
};
VarlenWs varlen_ws(const attn_bwd_varlen_args_t& a) {
    VarlenWs w;
    w.acc = 0;
    w.stats = w.acc + (size_t)(a.H * a.total_q * a.d * 4);
    w.maps = (w.stats + (size_t)(2 * a.H * varlen_stat_stride(a) * 4) + 127) / 128 * 128;
    w.misc = w.maps + (size_t)(7 * a.B) * sizeof(CUtensorMap);
    w.units = w.misc + (size_t)((a.B + 2 + 3) / 4 * 16);
    w.total = w.units + (size_t)(a.Hkv * (a.total_k / kBN + a.B)) * 16;
    return w;
}

}  // namespace

extern "C" {

size_t attn_bwd_varlen_workspace_size(const attn_bwd_varlen_args_t* args) {
    if (!args || check_varlen(*args) != ATTN_OK) return 0;
    return varlen_ws(*args).total;
}

int attn_bwd_varlen(const attn_bwd_varlen_args_t* args, void* workspace, size_t workspace_bytes,
                    attn_stream_t stream_) {
    if (!args) return ATTN_ERR_INVALID_ARG;
    const attn_bwd_varlen_args_t& a = *args;
    if (!a.q || !a.k || !a.v || !a.o || !a.dout || !a.lse || !a.dq || !a.dk || !a.dv || !a.cu_seqlens_q ||
        !a.cu_seqlens_k)
        return ATTN_ERR_INVALID_ARG;
    int st = check_varlen(a);
    if (st != ATTN_OK) return st;
    const uintptr_t al = (uintptr_t)a.q | (uintptr_t)a.k | (uintptr_t)a.v | (uintptr_t)a.o | (uintptr_t)a.dout |
                         (uintptr_t)a.dq | (uintptr_t)a.dk | (uintptr_t)a.dv | (uintptr_t)workspace;
    if ((al & 15u) || (((uintptr_t)a.lse | (uintptr_t)a.cu_seqlens_q | (uintptr_t)a.cu_seqlens_k) & 3u))
        return ATTN_ERR_MISALIGNED;
    const VarlenWs w = varlen_ws(a);
    if (!workspace || workspace_bytes < w.total) return ATTN_ERR_WORKSPACE;
    const int64_t d = a.d;
    const uintptr_t qb = (uintptr_t)(a.total_q * a.H * d * 2), kb = (uintptr_t)(a.total_k * a.Hkv * d * 2);
    const uintptr_t outs[3][2] = {{(uintptr_t)a.dq, qb}, {(uintptr_t)a.dk, kb}, {(uintptr_t)a.dv, kb}};
    const uintptr_t ins[6][2] = {{(uintptr_t)a.q, qb}, {(uintptr_t)a.k, kb}, {(uintptr_t)a.v, kb},
                                 {(uintptr_t)a.o, qb}, {(uintptr_t)a.dout, qb}, {(uintptr_t)workspace, w.total}};
    for (int i = 0; i < 3; ++i) {
        if (outs[i][1] == 0) continue;
        for (int j = 0; j < 6; ++j)
            if (outs[i][0] < ins[j][0] + ins[j][1] && ins[j][0] < outs[i][0] + outs[i][1]) return ATTN_ERR_ALIAS;
        for (int j = 0; j < i; ++j)
            if (outs[i][0] < outs[j][0] + outs[j][1] && outs[j][0] < outs[i][0] + outs[i][1]) return ATTN_ERR_ALIAS;
    }
    cudaStream_t stream = (cudaStream_t)stream_;
    int dev = 0, sms = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_NO_DEVICE;
    }
    if (major != 10 || minor != 3) return ATTN_ERR_NO_DEVICE;
    if ((st = bwd_setup(dev)) != ATTN_OK) return st;
    char* ws = reinterpret_cast<char*>(workspace);
    float* dq_acc = reinterpret_cast<float*>(ws + w.acc);
    const int64_t SP = varlen_stat_stride(a);
    float* lse2 = reinterpret_cast<float*>(ws + w.stats);
    float* delta = lse2 + a.H * SP;
    CUtensorMap* maps = reinterpret_cast<CUtensorMap*>(ws + w.maps);
    int* n_units = reinterpret_cast<int*>(ws + w.misc);
    int* pad = n_units + 1;
    int4* units = reinterpret_cast<int4*>(ws + w.units);
    // whole-tensor maps, token-major with one batch; the planning kernel narrows copies of them
    // to each sequence (a tensor without rows gets a one-row map that nothing uses)
    const int64_t tq = a.total_q > 0 ? a.total_q : 1, tk = a.total_k > 0 ? a.total_k : 1;
    CUtensorMap qm, dom, km, vm, dkm, dvm, accm;
    if (!encode(&qm, a.q, 1, a.H, tq, d, true) || !encode(&dom, a.dout, 1, a.H, tq, d, true) ||
        !encode(&km, a.k, 1, a.Hkv, tk, d, true) || !encode(&vm, a.v, 1, a.Hkv, tk, d, true) ||
        !encode(&dkm, a.dk, 1, a.Hkv, tk, d, true) || !encode(&dvm, a.dv, 1, a.Hkv, tk, d, true) ||
        !encode_dq(&accm, dq_acc, a.H, tq, d))
        return ATTN_ERR_CUDA;
    BwdVarlenPlan pl;
    memset(&pl, 0, sizeof pl);
    pl.cu_q = a.cu_seqlens_q;
    pl.cu_k = a.cu_seqlens_k;
    pl.B = (int)a.B;
    pl.H = (int)a.H;
    pl.Hkv = (int)a.Hkv;
    pl.group = (int)(a.H / a.Hkv);
    pl.causal = a.causal;
    pl.total_q = a.total_q;
    pl.total_k = a.total_k;
    pl.q_row_bytes = a.H * d * 2;
    pl.kv_row_bytes = a.Hkv * d * 2;
    pl.acc_row_bytes = d * 4;
    pl.q = reinterpret_cast<const char*>(a.q);
    pl.dout = reinterpret_cast<const char*>(a.dout);
    pl.k = reinterpret_cast<const char*>(a.k);
    pl.v = reinterpret_cast<const char*>(a.v);
    pl.dk = reinterpret_cast<char*>(a.dk);
    pl.dv = reinterpret_cast<char*>(a.dv);
    pl.dq_acc = reinterpret_cast<char*>(dq_acc);
    pl.maps = maps;
    pl.units = units;
    pl.n_units = n_units;
    pl.pad = pad;

    BwdParams p;
    memset(&p, 0, sizeof p);
    p.B = (int)a.B;
    p.H = (int)a.H;
    p.Hkv = (int)a.Hkv;
    p.group = (int)(a.H / a.Hkv);
    p.nsplit = 1;
    p.causal = a.causal;
    p.bshd = 1;
    p.scale = (float)(1.0 / std::sqrt((double)d));
    p.scale_log2 = (float)((1.0 / std::sqrt((double)d)) * 1.4426950408889634);
    p.lse2 = lse2;
    p.delta = delta;
    p.dq_acc = dq_acc;
    p.wait_limit_ns = (unsigned long long)(a.wait_limit_ms > 0 ? a.wait_limit_ms : 2000) * 1000000ull;
    p.vl_maps = maps;
    p.vl_units = units;
    p.vl_n_units = n_units;
    p.vl_pad = pad;
    p.cu_q = a.cu_seqlens_q;
    p.cu_k = a.cu_seqlens_k;
    p.stat_stride = SP;

    // planning -> statistics (and dQ zeroing) -> main kernel -> dQ rounding, each a
    // programmatic dependent of the kernel before it in the stream
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t c;
    memset(&c, 0, sizeof c);
    c.gridDim = dim3(1);
    c.blockDim = dim3(1024);
    c.stream = stream;
    c.attrs = attr;
    c.numAttrs = 1;
    if (cudaLaunchKernelEx(&c, attn_bwd_varlen_plan_kernel, qm, dom, km, vm, dkm, dvm, accm, pl) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    const long long fill = (long long)sms * 8;
    const long long prows = a.H * SP;
    const long long prep_blocks = cdiv(prows, 256 / (d / 8));
    c.gridDim = dim3((unsigned)(prep_blocks < fill ? (prep_blocks > 0 ? prep_blocks : 1) : fill));
    c.blockDim = dim3(256);
    cudaError_t ce = d == 128
        ? cudaLaunchKernelEx(&c, attn_bwd_varlen_prep_kernel<128>, reinterpret_cast<const __nv_bfloat16*>(a.o),
                             reinterpret_cast<const __nv_bfloat16*>(a.dout), a.lse, lse2, delta, dq_acc,
                             (const int*)a.cu_seqlens_q, (const int*)pad, (int)a.B, (int)a.H, (long long)a.total_q,
                             (long long)SP)
        : cudaLaunchKernelEx(&c, attn_bwd_varlen_prep_kernel<64>, reinterpret_cast<const __nv_bfloat16*>(a.o),
                             reinterpret_cast<const __nv_bfloat16*>(a.dout), a.lse, lse2, delta, dq_acc,
                             (const int*)a.cu_seqlens_q, (const int*)pad, (int)a.B, (int)a.H, (long long)a.total_q,
                             (long long)SP);
    if (ce != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    c.gridDim = dim3((unsigned)sms);
    c.blockDim = dim3(kThreads);
    c.dynamicSmemBytes = d == 128 ? smem_alloc<128>() : smem_alloc<64>();
    ce = cudaLaunchKernelEx(&c, d == 128 ? attn_bwd_kernel<128, false, true> : attn_bwd_kernel<64, false, true>, qm, km,
                            vm, dom, accm, dkm, dvm, p);
    if (ce != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    const long long n8 = a.total_q * a.H * (d / 8);
    const long long blocks = cdiv(n8, 256);
    c.gridDim = dim3((unsigned)(blocks < fill ? (blocks > 0 ? blocks : 1) : fill));
    c.blockDim = dim3(256);
    c.dynamicSmemBytes = 0;
    ce = d == 128 ? cudaLaunchKernelEx(&c, attn_bwd_varlen_dq_kernel<128>, (const float*)dq_acc,
                                       reinterpret_cast<__nv_bfloat16*>(a.dq), (const int*)a.cu_seqlens_q,
                                       (const int*)a.cu_seqlens_k, (int)a.B, (int)a.H, (long long)a.total_q,
                                       (const int*)n_units)
                  : cudaLaunchKernelEx(&c, attn_bwd_varlen_dq_kernel<64>, (const float*)dq_acc,
                                       reinterpret_cast<__nv_bfloat16*>(a.dq), (const int*)a.cu_seqlens_q,
                                       (const int*)a.cu_seqlens_k, (int)a.B, (int)a.H, (long long)a.total_q,
                                       (const int*)n_units);
    if (ce != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

size_t attn_bwd_workspace_size(const attn_bwd_args_t* args) {
    if (!args || check_shape(*args) != ATTN_OK) return 0;
    return ws_bytes(*args) + split_bytes(*args, bwd_split(*args, current_sms()));
}

int attn_bwd(const attn_bwd_args_t* args, void* workspace, size_t workspace_bytes, attn_stream_t stream_) {
    if (!args) return ATTN_ERR_INVALID_ARG;
    const attn_bwd_args_t& a = *args;
    if (!a.q || !a.k || !a.v || !a.o || !a.dout || !a.lse || !a.dq || !a.dk || !a.dv) return ATTN_ERR_INVALID_ARG;
    int st = check_shape(a);
    if (st != ATTN_OK) return st;
    const uintptr_t al = (uintptr_t)a.q | (uintptr_t)a.k | (uintptr_t)a.v | (uintptr_t)a.o | (uintptr_t)a.dout |
                         (uintptr_t)a.dq | (uintptr_t)a.dk | (uintptr_t)a.dv | (uintptr_t)workspace;
    if ((al & 15u) || ((uintptr_t)a.lse & 3u)) return ATTN_ERR_MISALIGNED;
    const size_t need_min = ws_bytes(a);
    if (!workspace || workspace_bytes < need_min) return ATTN_ERR_WORKSPACE;
    // the tail split needs room for its partials; a workspace sized without it (another GPU
    // model, an older size query) just runs unsplit
    BwdSplit sp = bwd_split(a, current_sms());
    if (workspace_bytes < need_min + split_bytes(a, sp)) sp = BwdSplit{0, 1};
    const size_t need = need_min + split_bytes(a, sp);
    // the gradients must not overlap the inputs or each other
    const uintptr_t qb = (uintptr_t)(a.B * a.H * a.Sq * a.d * 2), kb = (uintptr_t)(a.B * a.Hkv * a.Skv * a.d * 2);
    const uintptr_t outs[3][2] = {{(uintptr_t)a.dq, qb}, {(uintptr_t)a.dk, kb}, {(uintptr_t)a.dv, kb}};
    const uintptr_t ins[6][2] = {{(uintptr_t)a.q, qb}, {(uintptr_t)a.k, kb}, {(uintptr_t)a.v, kb},
                                 {(uintptr_t)a.o, qb}, {(uintptr_t)a.dout, qb}, {(uintptr_t)workspace, need}};
    for (int i = 0; i < 3; ++i) {
        for (int j = 0; j < 6; ++j)
            if (outs[i][0] < ins[j][0] + ins[j][1] && ins[j][0] < outs[i][0] + outs[i][1]) return ATTN_ERR_ALIAS;
        for (int j = 0; j < i; ++j)
            if (outs[i][0] < outs[j][0] + outs[j][1] && outs[j][0] < outs[i][0] + outs[i][1]) return ATTN_ERR_ALIAS;
    }
    cudaStream_t stream = (cudaStream_t)stream_;
    int dev = 0, sms = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_NO_DEVICE;
    }
    if (major != 10 || minor != 3) return ATTN_ERR_NO_DEVICE;
    if ((st = bwd_setup(dev)) != ATTN_OK) return st;
    const bool bshd = a.layout == ATTN_LAYOUT_BSHD;
    CUtensorMap qm, km, vm, dom;
    const int64_t d = a.d;
    if (!encode(&qm, a.q, a.B, a.H, a.Sq, d, bshd) || !encode(&km, a.k, a.B, a.Hkv, a.Skv, d, bshd) ||
        !encode(&vm, a.v, a.B, a.Hkv, a.Skv, d, bshd) || !encode(&dom, a.dout, a.B, a.H, a.Sq, d, bshd))
        return ATTN_ERR_CUDA;

    BwdParams p;
    memset(&p, 0, sizeof p);
    p.B = (int)a.B; p.H = (int)a.H; p.Hkv = (int)a.Hkv; p.Sq = (int)a.Sq; p.Skv = (int)a.Skv;
    p.group = (int)(a.H / a.Hkv);
    p.nq = (int)cdiv(a.Sq, kBM);
    p.nkv = (int)cdiv(a.Skv, kBN);
    p.nq_pad_rows = p.nq * kBM;
    p.n_units = (int)(a.B * a.Hkv * p.nkv);
    p.nsplit = (int)sp.P;
    p.n_full = (int)(p.n_units - sp.T);
    p.n_items = (int)(p.n_full + sp.T * sp.P);
    p.causal = a.causal;
    p.causal_off = (int)(a.Skv - a.Sq);
    p.paired = (a.causal && p.n_units >= 2 * sms) ? 1 : 0;
    p.bshd = bshd ? 1 : 0;
    p.scale = (float)(1.0 / std::sqrt((double)d));
    p.scale_log2 = (float)((1.0 / std::sqrt((double)d)) * 1.4426950408889634);
    float* dq_acc = reinterpret_cast<float*>(workspace);
    float* lse2 = dq_acc + dq_elems(a);
    float* delta = lse2 + a.B * a.H * p.nq_pad_rows;
    p.ws_dkv = delta + a.B * a.H * p.nq_pad_rows;      // split partials (16-byte aligned)
    p.lse2 = lse2;
    p.delta = delta;
    p.dq_acc = dq_acc;
    CUtensorMap dqm, dkm, dvm;
    const bool dq_ok = a.deterministic ? encode_dq_slices(&dqm, dq_acc, p.nkv, a.B * a.H, a.Sq, d)
                                       : encode_dq(&dqm, dq_acc, a.B * a.H, a.Sq, d);
    if (!dq_ok || !encode(&dkm, a.dk, a.B, a.Hkv, a.Skv, d, bshd) ||
        !encode(&dvm, a.dv, a.B, a.Hkv, a.Skv, d, bshd))
        return ATTN_ERR_CUDA;
    p.dk = reinterpret_cast<__nv_bfloat16*>(a.dk);
    p.dv = reinterpret_cast<__nv_bfloat16*>(a.dv);
    long long q_sb, q_ss, q_sh;
    if (bshd) {
        p.kv_sb = a.Skv * a.Hkv * d; p.kv_ss = a.Hkv * d; p.kv_sh = d;
        q_sb = a.Sq * a.H * d; q_ss = a.H * d; q_sh = d;
    } else {
        p.kv_sb = a.Hkv * a.Skv * d; p.kv_ss = d; p.kv_sh = a.Skv * d;
        q_sb = a.H * a.Sq * d; q_ss = d; q_sh = a.Sq * d;
    }
    p.wait_limit_ns = (unsigned long long)(a.wait_limit_ms > 0 ? a.wait_limit_ms : 2000) * 1000000ull;
    p.test_hooks = a.test_hooks;

    // preprocessing (also zeroes the dQ accumulator, if any) -> main kernel -> dQ rounding, each a
    // programmatic dependent of the kernel before it in the stream
    const long long prows = a.B * a.H * (long long)p.nq_pad_rows;
    const long long fill = (long long)sms * 8;             // resident 256-thread blocks
    auto prep = d == 128 ? attn_bwd_prep_kernel<128> : attn_bwd_prep_kernel<64>;
    const long long prep_blocks = cdiv(prows, 256 / (d / 8));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t pc;
    memset(&pc, 0, sizeof pc);
    pc.gridDim = dim3((unsigned)(prep_blocks < fill ? prep_blocks : fill));
    pc.blockDim = dim3(256);
    pc.stream = stream;
    pc.attrs = attr;
    pc.numAttrs = 1;
    if (cudaLaunchKernelEx(&pc, prep, reinterpret_cast<const __nv_bfloat16*>(a.o),
                           reinterpret_cast<const __nv_bfloat16*>(a.dout), a.lse, lse2, delta,
                           a.deterministic ? nullptr : dq_acc, p.H, p.Sq,
                           p.nq_pad_rows, prows, q_sb, q_ss, q_sh) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)(p.n_items < sms ? p.n_items : sms));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = d == 128 ? smem_alloc<128>() : smem_alloc<64>();
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    auto kern = d == 128 ? (a.deterministic ? attn_bwd_kernel<128, true> : attn_bwd_kernel<128, false>)
                         : (a.deterministic ? attn_bwd_kernel<64, true> : attn_bwd_kernel<64, false>);
    cudaError_t ce = cudaLaunchKernelEx(&cfg, kern, qm, km, vm, dom, dqm, dkm, dvm, p);
    if (ce != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    const long long n8 = a.B * a.H * a.Sq * (d / 8);
    const long long conv_blocks = cdiv(n8, 256);
    const int dq_blocks = (int)(conv_blocks < fill ? conv_blocks : fill);
    DkvCombine cb;
    memset(&cb, 0, sizeof cb);
    cb.ws = p.ws_dkv;
    cb.dk = p.dk;
    cb.dv = p.dv;
    cb.T = (int)sp.T;
    cb.P = (int)sp.P;
    cb.n_full = p.n_full;
    cb.nkv = p.nkv;
    cb.Hkv = p.Hkv;
    cb.Skv = p.Skv;
    cb.kv_sb = p.kv_sb;
    cb.kv_ss = p.kv_ss;
    cb.kv_sh = p.kv_sh;
    cb.scale = p.scale;
    const long long comb_blocks = sp.T * 2 * kBN / 8;   // one warp per (unit, tensor, key row)
    DqSlices ds;
    ds.nkv = a.deterministic ? p.nkv : 0;
    ds.causal = p.causal;
    ds.causal_off = p.causal_off;
    ds.slice = a.B * a.H * a.Sq * d;
    cfg.gridDim = dim3((unsigned)(dq_blocks + comb_blocks));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    __nv_bfloat16* dqo = reinterpret_cast<__nv_bfloat16*>(a.dq);
    auto fin = d == 128 ? (a.deterministic ? attn_bwd_dq_kernel<128, true> : attn_bwd_dq_kernel<128, false>)
                        : (a.deterministic ? attn_bwd_dq_kernel<64, true> : attn_bwd_dq_kernel<64, false>);
    ce = cudaLaunchKernelEx(&cfg, fin, (const float*)dq_acc, dqo, p.H, p.Sq, n8, q_sb, q_ss, q_sh, dq_blocks, cb, ds);
    if (ce != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

int attn_bwd_get_device_status(attn_stream_t stream, int32_t* site) {
    if (site) *site = 0;
    uint32_t h[2] = {0u, 0u};
    const uint32_t zero[2] = {0u, 0u};
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess ||
        cudaMemcpyFromSymbol(h, g_bwd_status, sizeof h) != cudaSuccess ||
        cudaMemcpyToSymbol(g_bwd_status, zero, sizeof zero) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    if (site) *site = (int32_t)h[1];
    return (int)h[0];
}

}  // extern "C"
