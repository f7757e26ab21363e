// attn_fwd.cu -- bf16 attention forward for GB300 (sm_103a): kernels and the C ABI.
//
// O = softmax(Q K^T / sqrt(d)) V, d = 128 (or 64), BSHD or BHSD, any Sq/Skv, output rounded
// RTNE/RTNA/RTZ; optionally causal, with grouped K/V heads, and with the row log-sum-exp.
// Source page: "MoonMath AI open-sources a HIP attention kernel for AMD
// MI300X that beats AITER" (news.chathome.org), cited below as [MoonMath]:
//   opening section        -- the operation, layouts, d = 128, arbitrary lengths;
//   limitations paragraph  -- rounding modes, NaN/Inf bit-identical, determinism;
//   "Architecture: 8 waves, 2 groups, 2 barriers" -- two groups run the same
//                             QK^T / softmax / PV sequence out of phase so the matrix units
//                             never idle;
//   "Data placement and the 16x16x16 choice" -- K streamed through a double-buffered
//                             on-chip ring shared by all groups, extra Q tiles for K/V reuse,
//                             Flash-Decoding-style tail KV split over the compute units;
//   "Real use cases"       -- simple API launched on the caller's stream.
// The MI300X design is prior art.  The GB300 design here:
//   * one persistent CTA per SM, static round-robin over work items (deterministic);
//   * a work unit = one (b, h) and two 128-row query tiles (256 rows), so each K/V tile
//     feeds two query tiles;
//   * warp 8 streams Q and a K,V,K,V,... ring (128 KB: 4 x 32 KB stages at d = 128, 8 x 16 KB
//     at d = 64) with TMA + mbarriers;
//   * warp 9 (one thread) issues tcgen05.mma: S_i = Q_i K_j^T into tensor memory (TMEM) and
//     O_i += P_i V_j with P_i read from TMEM (it overwrites S_i, so P never goes through
//     shared memory) and V used as stored (MN-major operand, no transpose);
//   * warpgroups 0 and 1 each own one query tile: online softmax with exp2 and the scale
//     folded into one FMA, lazy O rescale (only when the running max grows by more than
//     2^tau), the epilogue (O / l, rounding mode, canonical NaN) and the store;
//   * the MMA order S0(j+1), S1(j+1) interleaved with PV0(j), PV1(j) keeps one query tile's
//     softmax running while the tensor core works on the other (the two-groups-out-of-phase
//     idea on tcgen05);
//   * tail units that would leave SMs idle in the last round are split along the keys;
//     each split writes fp32 O/l and a base-2 log-sum-exp, and a combine kernel merges them;
//   * for Sq <= 128 (one query tile per (b, h)) a second kernel, attn_fwd_short_kernel, runs
//     the same work items without the empty second tile (see "short queries" below);
//   * the kernels are templates on the head dimension and on the causal mask.  The causal
//     mask and grouped K/V heads are the features the [MoonMath] limitations paragraph lists
//     as missing; d = 64 is the second tile configuration of "HipKittens: Fast and Furious
//     AMD Kernels (MLSys 2026)", "Experiments and results";
//   * variable-length batches (the third missing feature of that paragraph) and a paged K/V
//     cache ("AMD zverejnilo postup pre custom diffusion attention kernel vo FlyDSL na ROCm",
//     the section on what AMD describes) run on a third template flag of the main kernel,
//     after a one-CTA kernel that narrows tensor maps to each sequence with tensormap.replace
//     and lays out the work list ("variable-length batches" below).
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

constexpr int kBM = 128;           // query rows per tile (one TMEM lane per row)
constexpr int kBN = 128;           // keys per KV tile
constexpr int kQTiles = 2;         // query tiles per work unit
constexpr int kUnitRows = kBM * kQTiles;
constexpr int kChunkBytes = kBM * 64 * 2;     // 16 KB: 128 rows x 64 bf16 (one TMA box)
constexpr int kThreads = 384;      // WG0, WG1 softmax; warp 8 TMA; warp 9 MMA; 10-11 spare
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
constexpr int kMinTilesPerSplit = 4;
// Register split (launch: 384 threads x 168 = 64512).  Softmax warpgroups 0-1 grow to 200,
// warpgroup 2 (TMA, MMA, two spare warps) shrinks to 104: 256*200 + 128*104 = 64512.
constexpr uint32_t kRegsSoftmax = 200;
constexpr uint32_t kRegsOther = 104;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsOther <= 65536 / kThreads * kThreads,
              "register split exceeds the launch budget");
constexpr uint32_t kTmemCols = 512;   // S0 | S1 | O0 | O1, 128 fp32 columns each

// Output staging: one 4 KB region per softmax warp (its 32 rows x 64 bf16 columns in the
// 128-byte swizzle TMA expects), filled once per 64 columns of the head dimension.  Only the
// warp's own TMA stores read it, so the warp's lane 0 waits for its previous store's read
// before refilling, and nothing else orders it.
constexpr int kStageRowsPerWarp = 32;
constexpr int kStageBytes = kStageRowsPerWarp * 64 * 2;

// Head-dimension dependent geometry (D = 128 or 64).  Shared memory offsets are from a
// 1024-byte aligned base.
template <int D>
struct Geo {
    static_assert(D == 64 || D == 128, "head dimension 64 or 128");
    static constexpr int kChunks = D / 64;                    // 64-column TMA boxes per row
    static constexpr int kTileBytes = kBM * D * 2;            // one 128-row tile of Q, K or V
    static constexpr int kStages = 4 * 128 / D;               // K/V ring: 128 KB in flight
    static constexpr int kSmemQ = 0;
    static constexpr int kSmemRing = kSmemQ + kQTiles * kTileBytes;
    static constexpr int kSmemStage = kSmemRing + kStages * kTileBytes;
    static constexpr int kSmemBars = kSmemStage + 8 * kStageBytes;
    // barrier indices
    static constexpr int kBarFull = 0;                // [kStages] ring slot loaded
    static constexpr int kBarEmpty = kStages;         // [kStages] ring slot released by the MMAs
    static constexpr int kBarQFull = 2 * kStages;
    static constexpr int kBarQEmpty = kBarQFull + 1;
    static constexpr int kBarSFull = kBarQEmpty + 1;  // [2] S_i ready in TMEM
    static constexpr int kBarPFull = kBarSFull + 2;   // [2] P_i written (and O_i rescaled)
    static constexpr int kBarOFull = kBarPFull + 2;   // [2] last PV of the unit done
    static constexpr int kBarDrain = kBarOFull + 2;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kSmemMisc = kSmemBars + kNumBars * 8;
    static constexpr int kSmemUsed = kSmemMisc + 16;
    static constexpr int kSmemAlloc = kSmemUsed + 1024;
    static_assert(kSmemAlloc <= 232448, "shared memory over the 227 KB limit");
};

// wait sites reported through the status word
enum : uint32_t {
    kSiteQEmpty = 1, kSiteRingEmpty, kSiteQFull, kSiteRingFull, kSitePFull, kSiteSFull,
    kSiteOFull, kSiteDrain, kSiteTeardown, kSitePVDone, kSiteOEmpty, kSiteStats, kSiteSeqlens
};
static_assert(kSiteOFull == ATTN_SITE_O_READY, "the O-ready wait site is part of the ABI");
static_assert(kSiteSeqlens == ATTN_SITE_SEQLENS, "the sequence-length check site is part of the ABI");

__device__ uint32_t g_status[2];   // [0] status code, [1] wait site

struct FwdParams {
    int B, H, Sq, Skv;
    int group;             // query heads per K/V head (H / Hkv)
    int causal;            // 1: key j visible to query i iff j <= i + causal_off
    int causal_off;        // Skv - Sq
    int nq, nkv;           // 256-row query blocks per (b, h); 128-key tiles
    int n_items, n_full;   // work items; items >= n_full are key splits of tail units
    int nsplit;
    int bshd;              // layout flag (coordinate order of the tensor maps)
    int round_mode;
    float scale_log2;      // (1/sqrt(d)) * log2(e)
    float tau;             // lazy-rescale threshold, log2 units
    __nv_bfloat16* o;
    float* ws_o;           // [split items][256][128] fp32
    float* ws_lse;         // [split items][256] fp32, base-2 log-sum-exp
    long long o_sb, o_ss, o_sh;   // element strides of O for b, s, h
    float* lse;            // optional [B][H][Sq] natural-log log-sum-exp, or null
    unsigned long long wait_limit_ns;
    int test_hooks;        // ATTN_TEST_WITHHOLD_O_READY: CTA 0 skips its first unit's O-ready signal
    // variable-length batches (the kVarlen instance only): B sequences packed along the token
    // axis; per sequence b a tensor map each for Q, K, V and O (vl_maps[4 b + 0..3]) that
    // covers only its rows; the work list, heaviest first (vl_blocks: sequence, query block,
    // key part, parts), each entry standing for H >> pack_shift items (one per query head or
    // packed head group), and the item count
    const CUtensorMap* vl_maps;
    const int4* vl_blocks;
    const int* vl_n_items;
    const int* cu_q;       // [B + 1] query row offsets
    const int* cu_k;       // [B + 1] key row offsets (unpaged)
    long long total_q;     // LSE row stride ([H][total_q])
    // paged K/V (a variable-length batch whose keys sit in cache pages): key j of sequence b
    // is slot j % page_size of page block_table[b * max_pages + j / page_size]; full pages
    // load through the whole-cache maps (kmap, vmap), the last page through the sequence's
    // own maps (vl_maps[4 b + 1, 2], narrowed to its used slots)
    int paged;
    const int* seqlens_k;  // [B]
    const int* block_table;
    int page_size, max_pages;
    // head packing (variable-length batches): the 2^pack_shift query heads that share a K/V
    // head are the rows of one tile, row r = token (r >> pack_shift), head h + (r & mask), so a
    // 256-row block holds 256 >> pack_shift tokens; 0: one head per tile
    int pack_shift;
};

struct Item {
    int b, h, hk, qb, kv_begin, kv_end, split_slot;   // hk: the K/V head query head h reads
    int sq, skv, causal_off;   // the sequence's lengths (variable-length batches only)
    int q0;                    // its first query row in the packed tensors (< 2^30)
};

// The item a CTA runs in its r-th round: round-robin, and for causal launches and
// variable-length batches in alternating direction (CTA c takes position c of even rounds and
// G - 1 - c of odd ones).  Their items run heaviest first and shrink from round to round, so
// plain round-robin gives the low CTAs the heavier item of every round (a trace on the causal
// prefill had the first CTA done 13 % before the last); alternating cancels that.  Within a
// CTA, items still increase with r.
template <bool kAlternate>
__device__ __forceinline__ int round_item(int r) {
    const int c = (kAlternate && (r & 1)) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x;
    return r * (int)gridDim.x + c;
}

// Work item k of a variable-length batch: query head (or packed head group) k % per_block of
// the entry vl_blocks[k / per_block], which the preprocessing kernel ordered by the key tiles
// they run, most first.  Lengths and offsets come from the sequence.  An entry (b, qb, part,
// parts) with parts > 1 runs the part-th of `parts` near-equal contiguous ranges of the block's
// key tiles into split slot k, and the variable-length combine kernel merges the parts.
template <bool kCausal>
__device__ __forceinline__ Item decode_varlen_item(const FwdParams& p, int k) {
    Item it;
    const int per_block = p.H >> p.pack_shift;        // items per entry
    const int4 e = __ldg(p.vl_blocks + k / per_block);
    it.b = e.x;
    it.qb = e.y;
    it.h = (k % per_block) << p.pack_shift;          // the first of the tile's heads
    const int q0 = __ldg(p.cu_q + it.b);
    it.sq = __ldg(p.cu_q + it.b + 1) - q0;
    it.skv = p.paged ? __ldg(p.seqlens_k + it.b) : __ldg(p.cu_k + it.b + 1) - __ldg(p.cu_k + it.b);
    it.q0 = q0;
    it.causal_off = it.skv - it.sq;
    int tiles = (it.skv + kBN - 1) / kBN;
    if constexpr (kCausal) {
        const int last = ((it.qb + 1) * kUnitRows >> p.pack_shift) - 1 + it.causal_off;   // last visible key
        const int need = last < 0 ? 1 : last / kBN + 1;
        tiles = need < tiles ? need : tiles;
    }
    if (e.w > 1) {
        const int base = tiles / e.w, rem = tiles % e.w;
        it.kv_begin = e.z * base + (e.z < rem ? e.z : rem);
        it.kv_end = it.kv_begin + base + (e.z < rem ? 1 : 0);
        it.split_slot = k;
    } else {
        it.kv_begin = 0;
        it.kv_end = tiles;
        it.split_slot = -1;
    }
    it.hk = p.group == 1 ? it.h : it.h / p.group;
    return it;
}

// Work item k of the static schedule.  kCausal is a template parameter so that the
// unmasked kernel carries none of the causal code.
template <bool kCausal, bool kVarlen = false>
__device__ __forceinline__ Item decode_item(const FwdParams& p, int k) {
    if constexpr (kVarlen) return decode_varlen_item<kCausal>(p, k);
    Item it;
    int unit;
    if (k < p.n_full) {
        unit = k;
        it.kv_begin = 0;
        it.kv_end = p.nkv;
        it.split_slot = -1;
    } else {
        const int r = k - p.n_full;
        const int t = r / p.nsplit, s = r % p.nsplit;
        unit = p.n_full + t;
        const int base = p.nkv / p.nsplit, rem = p.nkv % p.nsplit;
        it.kv_begin = s * base + (s < rem ? s : rem);
        it.kv_end = it.kv_begin + base + (s < rem ? 1 : 0);
        it.split_slot = r;
    }
    if constexpr (kCausal) {
        // heaviest first: query blocks nearest the end see the most keys; each block runs
        // only the key tiles up to its diagonal (at least one, which the mask then empties)
        const int bhn = p.B * p.H;
        it.qb = p.nq - 1 - unit / bhn;
        const int bh = unit % bhn;
        it.h = bh % p.H;
        it.b = bh / p.H;
        const int last = it.qb * kUnitRows + kUnitRows - 1 + p.causal_off;   // last visible key
        const int need = last < 0 ? 1 : last / kBN + 1;
        it.kv_end = need < it.kv_end ? need : it.kv_end;
    } else {
        it.qb = unit % p.nq;
        const int bh = unit / p.nq;
        it.h = bh % p.H;
        it.b = bh / p.H;
    }
    it.hk = p.group == 1 ? it.h : it.h / p.group;
    return it;
}

// Bounded mbarrier wait.  On expiry it records the site in the status word, raises the
// CTA's abort flag and returns false; every other wait then gives up at once.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, uint32_t site,
                                      volatile uint32_t* abort_flag,
                                      unsigned long long limit_ns) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer_ns() - t0 > limit_ns) {
            if (atomicCAS(&g_status[0], 0u, (uint32_t)ATTN_ERR_DEVICE_TIMEOUT) == 0u)
                atomicExch(&g_status[1], site);
            *abort_flag = 1u;
            return false;
        }
    }
}

// UMMA shared-memory descriptor, 128-byte swizzle, tcgen05 version bits.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;            // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;            // SWIZZLE_128B
    return d;
}

// Instruction descriptor for kind::f16: bf16 x bf16 -> fp32, dense.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4)                                   // D format: f32
           | (1u << 7)                                 // A format: bf16
           | (1u << 10)                                // B format: bf16
           | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16)
           | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// fp32 -> bf16 bits in the selected mode; NaN -> 0x7FC0.  [MoonMath] limitations paragraph.
__device__ __forceinline__ uint32_t round_bf16_bits(float f, int mode) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;
    if (mode == ATTN_ROUND_RTNE) u += 0x7FFFu + ((u >> 16) & 1u);
    else if (mode == ATTN_ROUND_RTNA) u += 0x8000u;
    return u >> 16;
}

// Scale 2*N fp32 accumulator columns (bit patterns in o) by inv and round each pair to one
// packed bf16x2 word in `mode`: the conversion instruction for RTNE and RTZ, and for RTNA the
// carry of half an ulp into the kept bits (magnitude rounds up at the tie, overflow carries
// into the exponent and gives inf).  These agree with round_bf16_bits on every non-NaN value;
// a NaN anywhere among the scaled values sends the whole group to round_bf16_bits, which
// gives NaN the pattern 0x7FC0.
template <int N>
__device__ __forceinline__ void scale_round_pairs(const uint32_t* o, float inv, int mode, uint32_t* w) {
    const float2 iv = make_float2(inv, inv);
    float2 x[N];
    float probe = 0.0f;
#pragma unroll
    for (int e = 0; e < N; ++e) {
        x[e] = __fmul2_rn(make_float2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), iv);
        probe = ptx::fmax3_nan(probe, x[e].x, x[e].y);
    }
    if (probe != probe) {
#pragma unroll
        for (int e = 0; e < N; ++e)
            w[e] = round_bf16_bits(x[e].x, mode) | (round_bf16_bits(x[e].y, mode) << 16);
    } else if (mode == ATTN_ROUND_RTNE) {
#pragma unroll
        for (int e = 0; e < N; ++e) w[e] = ptx::pack_bf16x2(x[e].x, x[e].y);
    } else if (mode == ATTN_ROUND_RTZ) {
#pragma unroll
        for (int e = 0; e < N; ++e) w[e] = ptx::pack_bf16x2_rz(x[e].x, x[e].y);
    } else {
#pragma unroll
        for (int e = 0; e < N; ++e)
            w[e] = __byte_perm(__float_as_uint(x[e].x) + 0x8000u, __float_as_uint(x[e].y) + 0x8000u, 0x7632);
    }
}

// softmax weight exponent for logit s relative to the reference m: x = (s - m) * c, which is
// exactly 0 for the key that set m (so a lone key gets weight 1 and O = its V row), kept
// >= -125.02 when s is finite so that a finite logit always has a positive (normal) weight;
// -inf stays -inf (weight exactly 0) and NaN stays NaN.  For x >= -124 the fma returns x
// unchanged (x * 2^-126 is far below half an ulp of x); for finite x < -124 it gives
// -124 - |x| * 2^-126 >= -125.02 since |x| < 2^127.
constexpr float kMinExponent = -124.0f;
constexpr float kLn2 = 0.693147180559945309f;
__device__ __forceinline__ float weight_exponent(float s, float c, float m) {
    const float x = (s - m) * c;
    return fmaf(x, 0x1p-126f, ptx::fmax_nan(x, kMinExponent));
}

// kVarlen: a variable-length batch or a paged K/V cache (per-sequence tensor maps from
// p.vl_maps, the work list from p.vl_blocks, both written by attn_varlen_prep_kernel); a
// separate instance.
template <int D, bool kCausal, bool kVarlen = false>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
                const FwdParams p) {
    using G = Geo<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bars = sbase + G::kSmemBars;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint32_t* tmem_holder = (uint32_t*)(smem + G::kSmemMisc);
    volatile uint32_t* abort_flag = (volatile uint32_t*)(smem + G::kSmemMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < G::kStages; ++s) {
            ptx::mbar_init(bar(G::kBarFull + s), 1);
            ptx::mbar_init(bar(G::kBarEmpty + s), 1);
        }
        ptx::mbar_init(bar(G::kBarQFull), 1);
        ptx::mbar_init(bar(G::kBarQEmpty), 1);
        for (int i = 0; i < kQTiles; ++i) {
            ptx::mbar_init(bar(G::kBarSFull + i), 1);
            ptx::mbar_init(bar(G::kBarPFull + i), kBM);
            ptx::mbar_init(bar(G::kBarOFull + i), 1);
        }
        ptx::mbar_init(bar(G::kBarDrain), 1);
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
    // launched as a programmatic dependent of the stream's previous kernel, whose output Q, K
    // and V may be and whose input O may be: only the prologue above overlaps its tail, and
    // every thread waits for its memory here before touching global memory
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the split-combine kernel may be scheduled as CTAs retire; it waits for this grid's memory
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // a variable-length batch's item count comes from its preprocessing kernel
    const int n_items = kVarlen ? __ldg(p.vl_n_items) : p.n_items;

    if (warp >= 8) {
        ptx::reg_dealloc<kRegsOther>();
        if (warp == kWarpTma && lane == 0) {
            // -------------------------------------------------------------- TMA producer
            const uint64_t pol_kv = ptx::policy_evict_last();
            const uint64_t pol_q = ptx::policy_evict_first();
            uint32_t pos = 0;             // ring position (monotonic)
            int u = 0;
            bool ok = true;
            for (int r = 0, k = round_item<kCausal || kVarlen>(0); k < n_items && ok; k = round_item<kCausal || kVarlen>(++r), ++u) {
                const Item it = decode_item<kCausal, kVarlen>(p, k);
                if (u > 0 && !(ok = wait_bar(bar(G::kBarQEmpty), (u - 1) & 1, kSiteQEmpty, abort_flag, lim)))
                    break;
                // tensor maps and batch coordinate: a variable-length batch's sequence has maps of
                // its own (token-major like BSHD, one "batch"), acquired before first use
                const void* qmp = &qmap;
                const void* kmp = &kmap;
                const void* vmp = &vmap;
                int bc = it.b;
                if constexpr (kVarlen) {
                    qmp = p.vl_maps + 4 * it.b;
                    kmp = p.vl_maps + 4 * it.b + 1;
                    vmp = p.vl_maps + 4 * it.b + 2;
                    ptx::tensormap_acquire(qmp);
                    ptx::tensormap_acquire(kmp);
                    ptx::tensormap_acquire(vmp);
                    bc = 0;
                }
                ptx::mbar_arrive_expect_tx(bar(G::kBarQFull), kQTiles * G::kTileBytes);
                for (int t = 0; t < kQTiles; ++t) {
                    // first token of the tile (with head packing, 128 >> pack_shift tokens
                    // of 2^pack_shift heads each: the Q map's box is (64, 2^shift, 128 >> shift))
                    const int row = kVarlen ? (it.qb * kUnitRows + t * kBM) >> p.pack_shift : it.qb * kUnitRows + t * kBM;
                    for (int c = 0; c < G::kChunks; ++c) {
                        const uint32_t dst = sbase + G::kSmemQ + t * G::kTileBytes + c * kChunkBytes;
                        if (kVarlen || p.bshd)
                            ptx::tma_load_4d(dst, qmp, bar(G::kBarQFull), c * 64, it.h, row, bc, pol_q);
                        else
                            ptx::tma_load_4d(dst, qmp, bar(G::kBarQFull), c * 64, row, it.h, bc, pol_q);
                    }
                }
                for (int j = it.kv_begin; j < it.kv_end && ok; ++j) {
                    for (int kv = 0; kv < 2; ++kv, ++pos) {
                        const uint32_t slot = pos % G::kStages;
                        const uint32_t ph = (pos / G::kStages) & 1u;
                        if (!(ok = wait_bar(bar(G::kBarEmpty + slot), ph ^ 1u, kSiteRingEmpty, abort_flag, lim)))
                            break;
                        ptx::mbar_arrive_expect_tx(bar(G::kBarFull + slot), G::kTileBytes);
                        const void* map = kv ? vmp : kmp;
                        int krow = j * kBN;
                        if constexpr (kVarlen) {
                            if (p.paged) {
                                // the tile lies in one page: the last one through the sequence's
                                // narrowed map, the others through the whole-cache map
                                const int pg = krow / p.page_size, slot0 = krow - pg * p.page_size;
                                if (pg == (it.skv - 1) / p.page_size) {
                                    krow = slot0;
                                } else {
                                    map = kv ? (const void*)&vmap : (const void*)&kmap;
                                    krow = __ldg(p.block_table + (long long)it.b * p.max_pages + pg) * p.page_size + slot0;
                                }
                            }
                        }
                        for (int c = 0; c < G::kChunks; ++c) {
                            const uint32_t dst = sbase + G::kSmemRing + slot * G::kTileBytes + c * kChunkBytes;
                            if (kVarlen || p.bshd)
                                ptx::tma_load_4d(dst, map, bar(G::kBarFull + slot), c * 64, it.hk, krow, bc, pol_kv);
                            else
                                ptx::tma_load_4d(dst, map, bar(G::kBarFull + slot), c * 64, krow, it.hk, bc, pol_kv);
                        }
                    }
                }
            }
            // every load issued has landed before the CTA may exit: the last G::kStages
            // positions cover each slot's most recent load
            for (uint32_t q = (pos > G::kStages ? pos - G::kStages : 0); q < pos; ++q) {
                const uint32_t ph = (q / G::kStages) & 1u;
                const uint64_t t0 = ptx::globaltimer_ns();
                while (!ptx::mbar_try_wait(bar(G::kBarFull + q % G::kStages), ph) && ptx::globaltimer_ns() - t0 < lim) {
                }
            }
        } else if (warp == kWarpMma && lane == 0) {
            // -------------------------------------------------------------- MMA issuer
            constexpr uint32_t idesc_s = idesc_bf16(kBM, kBN, false, false);
            constexpr uint32_t idesc_o = idesc_bf16(kBM, D, false, true);
            // TMEM columns: S_t at 128*t, O_t at 256 + 128*t
            // Q_i / K_j: K-major, 128 B rows, 8-row swizzle atoms 1024 B apart; the k-th
            // 16-element step sits 32 B further inside the atom, the second 64-column half
            // 16 KB further.  V_j: MN-major (d contiguous), the two 64-column halves 16 KB
            // apart (leading offset), 8-key groups 1024 B apart (stride offset); the k-th
            // 16-key step is 2 KB further.
            // Base descriptors; the address field counts 16-byte units, so moving the start
            // address by b bytes adds b >> 4 to the descriptor (no carry out of the field:
            // every address stays below 256 KB).
            const uint64_t dq0 = sdesc(sbase + G::kSmemQ, 16, 1024);
            const uint64_t dring = sdesc(sbase + G::kSmemRing, 16, 1024);
            const uint64_t dvring = sdesc(sbase + G::kSmemRing, kChunkBytes, 1024);
            // S_t = Q_t K^T: 8 steps of 16 along d (32 B inside a 64-column half, then the
            // other half 16 KB on).  Fully unrolled with constant offsets from one base
            // descriptor per operand: a rolled loop that recomputes descriptors costs ~200
            // cycles per MMA in issue, three times the 64-cycle MMA itself.
            auto issue_s = [&](int t, uint32_t kslot) {
                const uint64_t a0 = dq0 + (uint64_t)((t * G::kTileBytes) >> 4);
                const uint64_t b0 = dring + (uint64_t)((kslot * G::kTileBytes) >> 4);
                const uint32_t d = tmem + 128u * t;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4);
                    ptx::mma_ss(d, a0 + off, b0 + off, idesc_s, kk > 0 ? 1u : 0u);
                }
            };
            // O_t += P_t V: 8 steps of 16 keys (P: 8 TMEM columns each; V: 2 KB each)
            auto issue_o = [&](int t, uint32_t vslot, bool first) {
                const uint64_t b0 = dvring + (uint64_t)((vslot * G::kTileBytes) >> 4);
                const uint32_t d = tmem + 256u + (uint32_t)D * t, a = tmem + 128u * t;
                const uint32_t acc0 = first ? 0u : 1u;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    ptx::mma_ts(d, a + (uint32_t)kk * 8u, b0 + (uint64_t)((kk * 2048) >> 4), idesc_o,
                                kk > 0 ? 1u : acc0);
            };
            uint32_t pos = 0;
            uint32_t pcount = 0;   // P_t phases consumed (same count for both tiles)
            int u = 0;
            bool ok = true;
            for (int r = 0, k = round_item<kCausal || kVarlen>(0); k < n_items && ok; k = round_item<kCausal || kVarlen>(++r), ++u) {
                const Item it = decode_item<kCausal, kVarlen>(p, k);
                const int nk = it.kv_end - it.kv_begin;
                if (!(ok = wait_bar(bar(G::kBarQFull), u & 1, kSiteQFull, abort_flag, lim))) break;
                uint32_t kslot = pos % G::kStages;
                if (!(ok = wait_bar(bar(G::kBarFull + kslot), (pos / G::kStages) & 1u, kSiteRingFull, abort_flag, lim)))
                    break;
                ptx::tc_fence_after();
                for (int t = 0; t < kQTiles; ++t) {
                    issue_s(t, kslot);
                    ptx::mma_commit(bar(G::kBarSFull + t));
                }
                ptx::mma_commit(bar(G::kBarEmpty + kslot));
                if (nk == 1) ptx::mma_commit(bar(G::kBarQEmpty));
                ++pos;
                for (int jj = 0; jj < nk && ok; ++jj) {
                    const uint32_t vpos = pos;
                    const uint32_t vslot = vpos % G::kStages;
                    const bool more = jj + 1 < nk;
                    if (!(ok = wait_bar(bar(G::kBarFull + vslot), (vpos / G::kStages) & 1u, kSiteRingFull, abort_flag, lim)))
                        break;
                    const uint32_t kpos = vpos + 1;
                    kslot = kpos % G::kStages;
                    for (int t = 0; t < kQTiles; ++t) {
                        if (!(ok = wait_bar(bar(G::kBarPFull + t), pcount & 1u, kSitePFull, abort_flag, lim)))
                            break;
                        ptx::tc_fence_after();
                        issue_o(t, vslot, jj == 0);
                        // (test hook: CTA 0 withholds its first unit's O-ready signal for tile 0,
                        // so that the epilogue's bounded wait expires)
                        if (!more && !(p.test_hooks && u == 0 && t == 0 && blockIdx.x == 0))
                            ptx::mma_commit(bar(G::kBarOFull + t));
                        if (t == kQTiles - 1) ptx::mma_commit(bar(G::kBarEmpty + vslot));
                        if (more) {
                            if (t == 0) {
                                if (!(ok = wait_bar(bar(G::kBarFull + kslot), (kpos / G::kStages) & 1u, kSiteRingFull,
                                                    abort_flag, lim)))
                                    break;
                                ptx::tc_fence_after();
                            }
                            issue_s(t, kslot);
                            ptx::mma_commit(bar(G::kBarSFull + t));
                            if (t == kQTiles - 1) {
                                ptx::mma_commit(bar(G::kBarEmpty + kslot));
                                if (jj + 2 == nk) ptx::mma_commit(bar(G::kBarQEmpty));
                            }
                        }
                    }
                    ++pcount;
                    pos += more ? 2 : 1;
                }
            }
            // drain: every MMA this thread issued has finished before TMEM is released
            ptx::mma_commit(bar(G::kBarDrain));
            const uint64_t t0 = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(bar(G::kBarDrain), 0) && ptx::globaltimer_ns() - t0 < lim) {
            }
        }
    } else {
        ptx::reg_alloc<kRegsSoftmax>();
        // ------------------------------------------------------------------ softmax + epilogue
        const int t = warp >> 2;                    // query tile owned by this warpgroup
        const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
        const int row = quarter * 32 + lane;        // row within the tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + (uint32_t)(t * 128);
        const uint32_t tO = tmem + lane_off + 256u + (uint32_t)(t * D);
        const float c = p.scale_log2;
        uint32_t scount = 0;
        int u = 0;
        bool ok = true;
        for (int r = 0, k = round_item<kCausal || kVarlen>(0); k < n_items && ok; k = round_item<kCausal || kVarlen>(++r), ++u) {
            const Item it = decode_item<kCausal, kVarlen>(p, k);
            float m_ref = -INFINITY;      // running max of raw logits at the last rescale
            float l = 0.0f;               // running sum of weights relative to m_ref
            // A warp whose 32 rows all lie past the queries (the tail of a block; all but the
            // first few rows of a decoding step) keeps every wait and arrival but skips its
            // softmax and epilogue work: a row's S, P and O are its own TMEM lane, and these
            // rows are never stored.  The softmax warps sharing its scheduler run faster.  A
            // loop of its own, so that the live loop below compiles as it would alone.
            const int first_row = kVarlen ? (it.qb * kUnitRows + t * kBM + quarter * 32) >> p.pack_shift
                                          : it.qb * kUnitRows + t * kBM + quarter * 32;
            const bool live = first_row < (kVarlen ? it.sq : p.Sq);
            if (!live) {
                for (int j = it.kv_begin; j < it.kv_end; ++j) {
                    ok = wait_bar(bar(G::kBarSFull + t), scount & 1u, kSiteSFull, abort_flag, lim);
                    if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                    ++scount;
                    ptx::tc_fence_after();
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar(G::kBarPFull + t));
                }
            } else {
                for (int j = it.kv_begin; j < it.kv_end; ++j) {
                    ok = wait_bar(bar(G::kBarSFull + t), scount & 1u, kSiteSFull, abort_flag, lim);
                    if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                    ++scount;
                    ptx::tc_fence_after();
                    uint32_t s[128];
                    ptx::tmem_ld128(tS, s);
                    // keys of this tile past `limit` are absent: beyond Skv, or (causal) past this
                    // row's diagonal; they get -inf logits and so weight 0
                    int limit = kBN - 1;
                    const int skv = kVarlen ? it.skv : p.Skv;
                    if constexpr (kCausal) {
                        limit = skv - j * kBN - 1;
                        const int qpos = kVarlen ? (it.qb * kUnitRows + t * kBM + row) >> p.pack_shift
                                                 : it.qb * kUnitRows + t * kBM + row;   // the row's query
                        const int diag = qpos + (kVarlen ? it.causal_off : p.causal_off) - j * kBN;
                        limit = diag < limit ? diag : limit;
                    } else {
                        const int valid = skv - j * kBN;   // the same for every row of the tile
                        limit = valid < kBN ? valid - 1 : kBN - 1;
                    }
                    float mx, mn;
                    const bool any_masked = __any_sync(0xFFFFFFFFu, limit < kBN - 1);
                    if (D == 64 && any_masked) {
                        // at d = 64 (MMA-issue-bound) the split form below measured 4 % slower:
                        // mask first, then the fused max/min
    #pragma unroll
                        for (int e = 0; e < 128; ++e)
                            if (e > limit) s[e] = __float_as_uint(-INFINITY);
                    }
                    if (D == 128 && any_masked) {
                        // the row min (which only decides whether the exponent clamp below can be
                        // skipped) over the raw logits, before the mask: a masked key's weight is
                        // exactly 0 from its -inf and needs no clamp, and counting masked keys' raw
                        // logits (zero past Skv, where K is zero-filled) only makes the test stricter
                        float mna[4], mxa[4];
    #pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) mna[q4] = __uint_as_float(s[q4]);
    #pragma unroll
                        for (int e = 4; e < 124; e += 8) {
    #pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4)
                                mna[q4] = ptx::fmin3(mna[q4], __uint_as_float(s[e + q4]), __uint_as_float(s[e + 4 + q4]));
                        }
    #pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) mna[q4] = fminf(mna[q4], __uint_as_float(s[124 + q4]));
                        mn = ptx::fmin3(mna[0], mna[1], fminf(mna[2], mna[3]));
    #pragma unroll
                        for (int e = 0; e < 128; ++e)
                            if (e > limit) s[e] = __float_as_uint(-INFINITY);
    #pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) mxa[q4] = __uint_as_float(s[q4]);
    #pragma unroll
                        for (int e = 4; e < 124; e += 8) {
    #pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4)
                                mxa[q4] = ptx::fmax3(mxa[q4], __uint_as_float(s[e + q4]), __uint_as_float(s[e + 4 + q4]));
                        }
    #pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) mxa[q4] = fmaxf(mxa[q4], __uint_as_float(s[124 + q4]));
                        mx = ptx::fmax3(mxa[0], mxa[1], fmaxf(mxa[2], mxa[3]));
                    } else {
                        // row max and min: 3-input trees over 4 independent chains each
                        float mxa[4], mna[4];
    #pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) mxa[q4] = mna[q4] = __uint_as_float(s[q4]);
    #pragma unroll
                        for (int e = 4; e < 124; e += 8) {
    #pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                const float a = __uint_as_float(s[e + q4]), b = __uint_as_float(s[e + 4 + q4]);
                                mxa[q4] = ptx::fmax3(mxa[q4], a, b);
                                mna[q4] = ptx::fmin3(mna[q4], a, b);
                            }
                        }
    #pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            mxa[q4] = fmaxf(mxa[q4], __uint_as_float(s[124 + q4]));
                            mna[q4] = fminf(mna[q4], __uint_as_float(s[124 + q4]));
                        }
                        mx = ptx::fmax3(mxa[0], mxa[1], fmaxf(mxa[2], mxa[3]));
                        mn = ptx::fmin3(mna[0], mna[1], fminf(mna[2], mna[3]));
                    }
                    const float m_new = fmaxf(m_ref, mx);
                    bool rescale_o = false;
                    float alpha = 1.0f;
                    if (m_new > m_ref && (m_new - m_ref) * c > p.tau) {
                        if (m_ref == -INFINITY) {
                            alpha = 0.0f;      // nothing accumulated yet but 0*v terms
                        } else {
                            alpha = ptx::ex2_approx(fmaxf((m_ref - m_new) * c, -125.0f));
                            rescale_o = j > it.kv_begin;
                        }
                        l *= alpha;
                        m_ref = m_new;
                    }
                    const float m_use = (m_ref == -INFINITY) ? 0.0f : m_ref;
                    // Every exponent of this row is >= -124 and no logit is -inf: the clamp that
                    // keeps underflowing finite weights positive cannot fire, so skip it.
                    const bool plain = mn > -INFINITY && (mn - m_use) * c >= kMinExponent;
                    const float2 c2 = make_float2(c, c), nm2 = make_float2(-m_use, -m_use);
                    float2 lsum[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                      make_float2(0.f, 0.f)};
                    uint32_t pk[64];
                    if (__all_sync(0xFFFFFFFFu, plain)) {
    #pragma unroll
                        for (int e = 0; e < 64; ++e) {
                            const float2 x = __fmul2_rn(
                                __fadd2_rn(make_float2(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1])), nm2), c2);
                            const float2 pp = make_float2(ptx::ex2_approx(x.x), ptx::ex2_approx(x.y));
                            lsum[e & 3] = __fadd2_rn(lsum[e & 3], pp);
                            pk[e] = ptx::pack_bf16x2(pp.x, pp.y);
                        }
                    } else {
    #pragma unroll
                        for (int e = 0; e < 64; ++e) {
                            const float p0 = ptx::ex2_approx(weight_exponent(__uint_as_float(s[2 * e]), c, m_use));
                            const float p1 = ptx::ex2_approx(weight_exponent(__uint_as_float(s[2 * e + 1]), c, m_use));
                            lsum[e & 3] = __fadd2_rn(lsum[e & 3], make_float2(p0, p1));
                            pk[e] = ptx::pack_bf16x2(p0, p1);
                        }
                    }
                    ptx::tmem_st32(tS, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
                    ptx::tmem_st32(tS + 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
                    const float2 ls = __fadd2_rn(__fadd2_rn(lsum[0], lsum[1]), __fadd2_rn(lsum[2], lsum[3]));
                    l += ls.x + ls.y;
                    if (__any_sync(0xFFFFFFFFu, rescale_o)) {
                        const float a = rescale_o ? alpha : 1.0f;
                        const float2 a2 = make_float2(a, a);
    #pragma unroll 1
                        for (int ch = 0; ch < D / 32; ++ch) {
                            uint32_t o[32];
                            ptx::tmem_ld32(tO + ch * 32, o);
    #pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), a2);
                                o[2 * e] = __float_as_uint(v.x);
                                o[2 * e + 1] = __float_as_uint(v.y);
                            }
                            ptx::tmem_st32(tO + ch * 32, o);
                        }
                    }
                    ptx::tmem_wait_st();
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar(G::kBarPFull + t));
                }
            }
            if (!ok) break;
            // epilogue: O / l, rounding, store
            ok = wait_bar(bar(G::kBarOFull + t), u & 1, kSiteOFull, abort_flag, lim);
            if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
            ptx::tc_fence_after();
            if (!live) continue;
            const int qrow = kVarlen ? (it.qb * kUnitRows + t * kBM + row) >> p.pack_shift
                                     : it.qb * kUnitRows + t * kBM + row;
            const bool valid_row = qrow < (kVarlen ? it.sq : p.Sq);
            // the whole O_t row in registers with one TMEM wait
            uint32_t o[D];
            if constexpr (D == 128) ptx::tmem_ld128(tO, o);
            else ptx::tmem_ld64(tO, o);
            if (it.split_slot < 0) {
                const float inv = 1.0f / l;
                // natural-log log-sum-exp of the scaled logits: (m_ref*c + log2 l) * ln 2
                if (p.lse && valid_row) {
                    const int hrow = kVarlen ? it.h + (row & ((1 << p.pack_shift) - 1)) : it.h;
                    const long long li = kVarlen ? (long long)hrow * p.total_q + it.q0 + qrow
                                                 : ((long long)it.b * p.H + it.h) * p.Sq + qrow;
                    p.lse[li] = (m_ref * c + log2f(l)) * kLn2;
                }
                const uint32_t region = sbase + G::kSmemStage + (uint32_t)(warp * kStageBytes);
                // the warp's first token (with head packing its 32 rows are 32 >> pack_shift
                // tokens of 2^pack_shift heads: the O map's box is (64, 2^shift, 32 >> shift))
                const int r0 = kVarlen ? (it.qb * kUnitRows + t * kBM + quarter * kStageRowsPerWarp) >> p.pack_shift
                                       : it.qb * kUnitRows + t * kBM + quarter * kStageRowsPerWarp;
#pragma unroll
                for (int hc = 0; hc < D / 64; ++hc) {
                    uint32_t w[32];
                    scale_round_pairs<32>(o + 64 * hc, inv, p.round_mode, w);
                    // the region's previous TMA store (if any) has finished reading it
                    if (lane == 0) ptx::bulk_wait_read0();
                    __syncwarp();
                    // row `lane` of the region; 16-byte piece pc is stored at pc ^ (lane & 7)
                    // (128-byte swizzle)
                    const uint32_t rowaddr = region + (uint32_t)lane * 128u;
#pragma unroll
                    for (int pc = 0; pc < 8; ++pc)
                        ptx::st_shared_v4(rowaddr + (((uint32_t)pc ^ (uint32_t)(lane & 7)) << 4), w[4 * pc],
                                          w[4 * pc + 1], w[4 * pc + 2], w[4 * pc + 3]);
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (kVarlen) {
                            const CUtensorMap* om = p.vl_maps + 4 * it.b + 3;
                            if (hc == 0) ptx::tensormap_acquire(om);
                            ptx::tma_store_4d(om, region, hc * 64, it.h, r0, 0);
                        } else if (p.bshd) {
                            ptx::tma_store_4d(&omap, region, hc * 64, it.h, r0, it.b);
                        } else {
                            ptx::tma_store_4d(&omap, region, hc * 64, r0, it.h, it.b);
                        }
                        ptx::bulk_commit();
                    }
                }
            } else {
                // split partial: O/l in fp32 (the raw sum when l == 0) and LSE in log2 units
                const float inv = (l > 0.0f) ? 1.0f / l : 1.0f;
                const long long wrow = (long long)it.split_slot * kUnitRows + t * kBM + row;
                if (valid_row) {
                    float4* d4 = reinterpret_cast<float4*>(p.ws_o + wrow * D);
#pragma unroll
                    for (int v4 = 0; v4 < D / 4; ++v4)
                        d4[v4] = make_float4(__uint_as_float(o[4 * v4]) * inv, __uint_as_float(o[4 * v4 + 1]) * inv,
                                             __uint_as_float(o[4 * v4 + 2]) * inv, __uint_as_float(o[4 * v4 + 3]) * inv);
                    p.ws_lse[wrow] = m_ref * c + log2f(l);
                }
            }
        }
    }

    // ---------------------------------------------------------------------- teardown
    if (warp < 8 && lane == 0) ptx::bulk_wait0();   // this warp's output stores are complete
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------------- short queries
// For Sq <= 128 every (b, h) has a single 128-row query tile, which the kernel above would run
// beside an empty second tile.  attn_fwd_short_kernel takes that one tile as its unit (same
// work items, planner, key splits and workspace rows as above; the unit's rows 128..255 do
// not exist) and keeps the tensor core busy without a second tile:
//   * two S buffers in TMEM, so S_{g+1} = Q K_{g+1}^T is computed while the softmax of step g
//     runs (P_g overwrites S_g in place);
//   * warpgroups 0 and 1 each own one 64-key half of every key tile: an online softmax of its
//     own (running max m_h, sum l_h) into its own accumulator O_h;
//   * warpgroup 2 merges the halves, O = (w_a O_a + w_b O_b) / (w_a l_a + w_b l_b) with
//     w_h = 2^((m_h - m) c) (the combine kernel's clamped rule), and runs the epilogue;
//   * warp 12 streams Q and K_g, V_g into step slot g & 1; warp 14 issues the S GEMMs and
//     warp 13 the PV GEMMs, two issuing threads on different sub-partitions (a single
//     thread's tcgen05.mma issue rate is what bounds these pipelines).
// TMEM: S buffer 0 | S buffer 1 | O_a | O_b.
namespace sq {
constexpr int kHalfN = kBN / 2;    // keys of a tile that one softmax warpgroup owns
constexpr int kThreads = 512;      // 128 registers per thread
constexpr int kWarpEpi = 8;        // warps 8-11: merge and epilogue
constexpr int kWarpTma = 12;
constexpr int kWarpMma = 13;       // PV GEMMs (and TMEM allocation)
constexpr int kWarpMmaS = 14;      // S GEMMs
constexpr uint32_t kTmemCols = 512;

template <int D>
struct Geo {
    static_assert(D == 64 || D == 128, "head dimension 64 or 128");
    static constexpr int kChunks = D / 64;                    // 64-column TMA boxes per row
    static constexpr int kTileBytes = kBM * D * 2;            // one 128-row tile of Q, K or V
    static constexpr int kStepSlots = 2;                      // K_g and V_g go to step slot g & 1
    static constexpr int kSmemQ = 0;                          // [2] query tiles, by unit parity
    static constexpr int kSmemRing = kSmemQ + 2 * kTileBytes;
    static constexpr int kSmemStage = kSmemRing + kStepSlots * 2 * kTileBytes;
    static constexpr int kSmemStats = kSmemStage + 4 * kStageBytes;   // [2 unit parity][2 halves][128] (m, l)
    static constexpr int kSmemBars = kSmemStats + 2 * 2 * kBM * 8;
    // barrier indices
    static constexpr int kBarKFull = 0;               // [step slot] K_g loaded
    static constexpr int kBarVFull = 2;               // [step slot] V_g loaded
    static constexpr int kBarQFull = 4;               // [2] query buffer loaded
    static constexpr int kBarQEmpty = kBarQFull + 2;  // [2] query buffer's last S GEMM done
    static constexpr int kBarSFull = kBarQEmpty + 2;  // [S buffer] S_g done (and K_g's slot free)
    static constexpr int kBarPFull = kBarSFull + 2;   // [S buffer] P_g written by both halves (and O rescaled)
    static constexpr int kBarPVDone = kBarPFull + 2;  // [S buffer] PV_g done (P_g read, V_g's slot free)
    static constexpr int kBarOFull = kBarPVDone + 2;  // the unit's last PV GEMMs done
    static constexpr int kBarOEmpty = kBarOFull + 1;  // the epilogue has read O_a and O_b
    static constexpr int kBarStats = kBarOEmpty + 1;  // [unit parity] both halves' (m, l) written
    static constexpr int kBarStatsFree = kBarStats + 2;   // [unit parity] the epilogue has read them
    static constexpr int kBarDrain = kBarStatsFree + 2;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kSmemMisc = kSmemBars + kNumBars * 8;
    static constexpr int kSmemUsed = kSmemMisc + 16;
    static constexpr int kSmemAlloc = kSmemUsed + 1024;
    static_assert(kSmemAlloc <= 232448, "shared memory over the 227 KB limit");
};
}  // namespace sq

template <int D, bool kCausal>
__global__ void __launch_bounds__(sq::kThreads, 1)
attn_fwd_short_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
                const FwdParams p) {
    using G = sq::Geo<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bars = sbase + G::kSmemBars;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint32_t* tmem_holder = (uint32_t*)(smem + G::kSmemMisc);
    volatile uint32_t* abort_flag = (volatile uint32_t*)(smem + G::kSmemMisc + 4);
    float2* stats = (float2*)(smem + G::kSmemStats);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(bar(G::kBarKFull + i), 1);
            ptx::mbar_init(bar(G::kBarVFull + i), 1);
            ptx::mbar_init(bar(G::kBarQFull + i), 1);
            ptx::mbar_init(bar(G::kBarQEmpty + i), 1);
            ptx::mbar_init(bar(G::kBarSFull + i), 1);
            ptx::mbar_init(bar(G::kBarPFull + i), 2 * kBM);
            ptx::mbar_init(bar(G::kBarPVDone + i), 1);
            ptx::mbar_init(bar(G::kBarStats + i), 2 * kBM);
            ptx::mbar_init(bar(G::kBarStatsFree + i), kBM);
        }
        ptx::mbar_init(bar(G::kBarOFull), 1);
        ptx::mbar_init(bar(G::kBarOEmpty), kBM);
        ptx::mbar_init(bar(G::kBarDrain), 2);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == sq::kWarpMma) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_holder), sq::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const unsigned long long lim = p.wait_limit_ns;
    // launched as a programmatic dependent of the stream's previous kernel, whose output Q, K
    // and V may be and whose input O may be: only the prologue above overlaps its tail, and
    // every thread waits for its memory here before touching global memory
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the split-combine kernel may be scheduled as CTAs retire; it waits for this grid's memory
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == sq::kWarpTma) {
        if (lane == 0) {
            // -------------------------------------------------------------- TMA producer
            // Per unit: its query tile into buffer u & 1 (once the unit two back has had its
            // last S GEMM), then K_j, V_j for each key tile into step slot g & 1.
            const uint64_t pol_kv = ptx::policy_evict_last();
            const uint64_t pol_q = ptx::policy_evict_first();
            uint32_t g = 0;               // step index (monotonic over the CTA's units)
            int u = 0;
            bool ok = true;
            for (int k = blockIdx.x; k < p.n_items && ok; k += gridDim.x, ++u) {
                const Item it = decode_item<kCausal>(p, k);
                const int qb = u & 1;
                if (u >= 2 &&
                    !(ok = wait_bar(bar(G::kBarQEmpty + qb), ((u >> 1) - 1) & 1, kSiteQEmpty, abort_flag, lim)))
                    break;
                ptx::mbar_arrive_expect_tx(bar(G::kBarQFull + qb), G::kTileBytes);
                const int row = it.qb * kUnitRows;
                for (int c = 0; c < G::kChunks; ++c) {
                    const uint32_t dst = sbase + G::kSmemQ + qb * G::kTileBytes + c * kChunkBytes;
                    if (p.bshd)
                        ptx::tma_load_4d(dst, &qmap, bar(G::kBarQFull + qb), c * 64, it.h, row, it.b, pol_q);
                    else
                        ptx::tma_load_4d(dst, &qmap, bar(G::kBarQFull + qb), c * 64, row, it.h, it.b, pol_q);
                }
                for (int j = it.kv_begin; j < it.kv_end && ok; ++j, ++g) {
                    // K_g into step slot g & 1 once S_{g-2} has read it, V_g once PV_{g-2} has
                    const uint32_t ss = g & 1u, ph = ((g - 2u) >> 1) & 1u;
                    for (int kv = 0; kv < 2 && ok; ++kv) {
                        if (g >= 2u && !(ok = wait_bar(bar((kv ? G::kBarPVDone : G::kBarSFull) + (int)ss), ph,
                                                       kSiteRingEmpty, abort_flag, lim)))
                            break;
                        const uint32_t full = bar((kv ? G::kBarVFull : G::kBarKFull) + (int)ss);
                        ptx::mbar_arrive_expect_tx(full, G::kTileBytes);
                        const void* map = kv ? (const void*)&vmap : (const void*)&kmap;
                        const uint32_t base = sbase + G::kSmemRing + (2u * ss + (uint32_t)kv) * G::kTileBytes;
                        for (int c = 0; c < G::kChunks; ++c) {
                            const uint32_t dst = base + c * kChunkBytes;
                            if (p.bshd)
                                ptx::tma_load_4d(dst, map, full, c * 64, it.hk, j * kBN, it.b, pol_kv);
                            else
                                ptx::tma_load_4d(dst, map, full, c * 64, j * kBN, it.hk, it.b, pol_kv);
                        }
                    }
                }
            }
            // every load issued has landed before the CTA may exit: the last two steps' loads
            for (uint32_t q = (g > 2u ? g - 2u : 0u); q < g; ++q) {
                for (int kv = 0; kv < 2; ++kv) {
                    const uint64_t t0 = ptx::globaltimer_ns();
                    while (!ptx::mbar_try_wait(bar((kv ? G::kBarVFull : G::kBarKFull) + (int)(q & 1u)), (q >> 1) & 1u) &&
                           ptx::globaltimer_ns() - t0 < lim) {
                    }
                }
            }
        }
    } else if ((warp == sq::kWarpMma || warp == sq::kWarpMmaS) && lane == 0) {
        // ------------------------------------------------------------------ MMA issuers
        // Two threads on different sub-partitions: this one issues the S GEMMs, warp 13's
        // the PV GEMMs.  The CTA's steps (one per key tile of each of its units) run in
        // order g = 0, 1, ...: K_g and V_g are in step slot g & 1, S_g goes to S buffer g & 1,
        // and P_g overwrites it.  S_g may be issued once PV_{g-2} (the last
        // reader of that buffer) is done, so the next tile's logits are ready when the
        // softmax finishes P_{g-1}, also across a unit boundary.
        constexpr uint32_t idesc_s = idesc_bf16(kBM, kBN, false, false);
        constexpr uint32_t idesc_o = idesc_bf16(kBM, D, false, true);
        // Q_u / K_j: K-major, 128 B rows, 8-row swizzle atoms 1024 B apart; the k-th 16-element
        // step sits 32 B further inside the atom, the second 64-column half 16 KB further.
        // V_j: MN-major (d contiguous), the two 64-column halves 16 KB apart (leading offset),
        // 8-key groups 1024 B apart (stride offset); the k-th 16-key step is 2 KB further.
        // The address field counts 16-byte units, so moving the start address by b bytes adds
        // b >> 4 to the descriptor (no carry out of the field: every address stays below 256 KB).
        const uint64_t dq0 = sdesc(sbase + G::kSmemQ, 16, 1024);
        const uint64_t dring = sdesc(sbase + G::kSmemRing, 16, 1024);
        const uint64_t dvring = sdesc(sbase + G::kSmemRing, kChunkBytes, 1024);
        bool ok = true;
        uint32_t g = 0;
        int u = 0;
        if (warp == sq::kWarpMmaS) {
            for (int k = blockIdx.x; k < p.n_items && ok; k += gridDim.x, ++u) {
                const Item it = decode_item<kCausal>(p, k);
                const int nk = it.kv_end - it.kv_begin;
                const int qbuf = u & 1;
                if (!(ok = wait_bar(bar(G::kBarQFull + qbuf), (uint32_t)(u >> 1) & 1u, kSiteQFull, abort_flag, lim)))
                    break;
                for (int jj = 0; jj < nk; ++jj, ++g) {
                    const uint32_t sb = g & 1u;
                    if (!(ok = wait_bar(bar(G::kBarKFull + (int)sb), (g >> 1) & 1u, kSiteRingFull, abort_flag, lim)))
                        break;
                    // the PV GEMMs of step g - 2 have read their P from this buffer
                    if (g >= 2u &&
                        !(ok = wait_bar(bar(G::kBarPVDone + (int)sb), ((g - 2u) >> 1) & 1u, kSitePVDone, abort_flag, lim)))
                        break;
                    ptx::tc_fence_after();
                    // S = Q K^T: D/16 steps of 16 along d, fully unrolled with constant offsets
                    // from one base descriptor per operand (a rolled loop that recomputes
                    // descriptors costs ~200 cycles per MMA in issue)
                    const uint64_t a0 = dq0 + (uint64_t)((qbuf * G::kTileBytes) >> 4);
                    const uint64_t b0 = dring + (uint64_t)((2u * sb * G::kTileBytes) >> 4);
                    const uint32_t d = tmem + 128u * sb;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t off = (uint64_t)(((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4);
                        ptx::mma_ss(d, a0 + off, b0 + off, idesc_s, kk > 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(bar(G::kBarSFull + sb));
                    if (jj + 1 == nk) ptx::mma_commit(bar(G::kBarQEmpty + qbuf));
                }
            }
        } else {
            for (int k = blockIdx.x; k < p.n_items && ok; k += gridDim.x, ++u) {
                const Item it = decode_item<kCausal>(p, k);
                const int nk = it.kv_end - it.kv_begin;
                for (int jj = 0; jj < nk; ++jj, ++g) {
                    const uint32_t sb = g & 1u;
                    if (!(ok = wait_bar(bar(G::kBarVFull + (int)sb), (g >> 1) & 1u, kSiteRingFull, abort_flag, lim)))
                        break;
                    // the unit's first PV overwrites O_a, O_b: the previous unit's epilogue has read them
                    if (jj == 0 && u > 0 &&
                        !(ok = wait_bar(bar(G::kBarOEmpty), (uint32_t)(u - 1) & 1u, kSiteOEmpty, abort_flag, lim)))
                        break;
                    const uint64_t b0 = dvring + (uint64_t)(((2u * sb + 1u) * G::kTileBytes) >> 4);
                    // one barrier per S buffer: the softmax may finish the next step before
                    // this wait, and that arrival must not land on the barrier waited on here
                    if (!(ok = wait_bar(bar(G::kBarPFull + (int)sb), (g >> 1) & 1u, kSitePFull, abort_flag, lim)))
                        break;
                    ptx::tc_fence_after();
                    for (int h = 0; h < 2; ++h) {
                        // O_h += P_h V[64h .. 64h + 63]: 4 steps of 16 keys (P_h: 8 TMEM columns
                        // each, the first 32 columns of its half of the S buffer; V: 2 KB each)
                        const uint32_t dO = tmem + 256u + (uint32_t)(D * h), a = tmem + 128u * sb + (uint32_t)(sq::kHalfN * h);
#pragma unroll
                        for (int k4 = 0; k4 < sq::kHalfN / 16; ++k4) {
                            const int kk = h * (sq::kHalfN / 16) + k4;
                            ptx::mma_ts(dO, a + (uint32_t)k4 * 8u, b0 + (uint64_t)((kk * 2048) >> 4), idesc_o,
                                        (k4 > 0 || jj > 0) ? 1u : 0u);
                        }
                    }
                    ptx::mma_commit(bar(G::kBarPVDone + (int)sb));
                    // (test hook: CTA 0 withholds its first unit's O-ready signal)
                    if (jj + 1 == nk && !(p.test_hooks && u == 0 && blockIdx.x == 0))
                        ptx::mma_commit(bar(G::kBarOFull));
                }
            }
        }
        // drain: every MMA this thread issued has finished before TMEM is released
        ptx::mma_commit(bar(G::kBarDrain));
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(bar(G::kBarDrain), 0) && ptx::globaltimer_ns() - t0 < lim) {
        }
    } else if (warp < 8) {
        // ------------------------------------------------------------ softmax, key half h
        // Thread = one query row (its TMEM lane) and keys 64h .. 64h + 63 of every tile: an
        // online softmax of its own over those keys, into its own accumulator O_h, with its
        // own running max m_h and sum l_h (the two halves are merged by the epilogue).
        const int h = warp >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;        // row within the tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_off + 256u + (uint32_t)(D * h);
        const float c = p.scale_log2;
        uint32_t g = 0;
        int u = 0;
        bool ok = true;
        for (int k = blockIdx.x; k < p.n_items && ok; k += gridDim.x, ++u) {
            const Item it = decode_item<kCausal>(p, k);
            float m_ref = -INFINITY;      // running max of raw logits at the last rescale
            float l = 0.0f;               // running sum of weights relative to m_ref
            for (int j = it.kv_begin; j < it.kv_end; ++j, ++g) {
                const uint32_t tS = tmem + lane_off + 128u * (g & 1u) + (uint32_t)(sq::kHalfN * h);
                ok = wait_bar(bar(G::kBarSFull + (g & 1u)), (g >> 1) & 1u, kSiteSFull, abort_flag, lim);
                if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                ptx::tc_fence_after();
                uint32_t s[sq::kHalfN];
                ptx::tmem_ld64(tS, s);
                // keys of this half past `limit` are absent: beyond Skv, or (causal) past this
                // row's diagonal; they get -inf logits and so weight 0
                const int key0 = j * kBN + sq::kHalfN * h;
                if constexpr (kCausal) {
                    int limit = p.Skv - key0 - 1;
                    const int diag = it.qb * kUnitRows + row + p.causal_off - key0;
                    limit = diag < limit ? diag : limit;
                    if (__any_sync(0xFFFFFFFFu, limit < sq::kHalfN - 1)) {
#pragma unroll
                        for (int e = 0; e < sq::kHalfN; ++e)
                            if (e > limit) s[e] = __float_as_uint(-INFINITY);
                    }
                } else {
                    const int valid = p.Skv - key0;   // the same for every row of the tile
                    if (valid < sq::kHalfN) {
#pragma unroll
                        for (int e = 0; e < sq::kHalfN; ++e)
                            if (e >= valid) s[e] = __float_as_uint(-INFINITY);
                    }
                }
                // row max and min: 3-input trees over 4 independent chains each
                float mxa[4], mna[4];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) mxa[q4] = mna[q4] = __uint_as_float(s[q4]);
#pragma unroll
                for (int e = 4; e < sq::kHalfN - 4; e += 8) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const float a = __uint_as_float(s[e + q4]), b = __uint_as_float(s[e + 4 + q4]);
                        mxa[q4] = ptx::fmax3(mxa[q4], a, b);
                        mna[q4] = ptx::fmin3(mna[q4], a, b);
                    }
                }
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    mxa[q4] = fmaxf(mxa[q4], __uint_as_float(s[sq::kHalfN - 4 + q4]));
                    mna[q4] = fminf(mna[q4], __uint_as_float(s[sq::kHalfN - 4 + q4]));
                }
                const float mx = ptx::fmax3(mxa[0], mxa[1], fmaxf(mxa[2], mxa[3]));
                const float mn = ptx::fmin3(mna[0], mna[1], fminf(mna[2], mna[3]));
                const float m_new = fmaxf(m_ref, mx);
                bool rescale_o = false;
                float alpha = 1.0f;
                if (m_new > m_ref && (m_new - m_ref) * c > p.tau) {
                    if (m_ref == -INFINITY) {
                        alpha = 0.0f;      // nothing accumulated yet but 0*v terms
                    } else {
                        alpha = ptx::ex2_approx(fmaxf((m_ref - m_new) * c, -125.0f));
                        rescale_o = j > it.kv_begin;
                    }
                    l *= alpha;
                    m_ref = m_new;
                }
                const float m_use = (m_ref == -INFINITY) ? 0.0f : m_ref;
                // Every exponent of this row is >= -124 and no logit is -inf: the clamp that
                // keeps underflowing finite weights positive cannot fire, so skip it.
                const bool plain = mn > -INFINITY && (mn - m_use) * c >= kMinExponent;
                const float2 c2 = make_float2(c, c), nm2 = make_float2(-m_use, -m_use);
                float2 lsum[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                  make_float2(0.f, 0.f)};
                uint32_t pk[sq::kHalfN / 2];
                if (__all_sync(0xFFFFFFFFu, plain)) {
#pragma unroll
                    for (int e = 0; e < sq::kHalfN / 2; ++e) {
                        const float2 x = __fmul2_rn(
                            __fadd2_rn(make_float2(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1])), nm2), c2);
                        const float2 pp = make_float2(ptx::ex2_approx(x.x), ptx::ex2_approx(x.y));
                        lsum[e & 3] = __fadd2_rn(lsum[e & 3], pp);
                        pk[e] = ptx::pack_bf16x2(pp.x, pp.y);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < sq::kHalfN / 2; ++e) {
                        const float p0 = ptx::ex2_approx(weight_exponent(__uint_as_float(s[2 * e]), c, m_use));
                        const float p1 = ptx::ex2_approx(weight_exponent(__uint_as_float(s[2 * e + 1]), c, m_use));
                        lsum[e & 3] = __fadd2_rn(lsum[e & 3], make_float2(p0, p1));
                        pk[e] = ptx::pack_bf16x2(p0, p1);
                    }
                }
                // P_h over the first 32 columns of this half: the logits were read above, and
                // the other half's columns are not touched
                ptx::tmem_st32(tS, pk);
                const float2 ls = __fadd2_rn(__fadd2_rn(lsum[0], lsum[1]), __fadd2_rn(lsum[2], lsum[3]));
                l += ls.x + ls.y;
                if (__any_sync(0xFFFFFFFFu, rescale_o)) {
                    // O_h is stable once the previous step's PV into it is done (S_g was issued
                    // ahead of that PV, so S being ready does not imply it)
                    ok = wait_bar(bar(G::kBarPVDone + (int)((g - 1u) & 1u)), ((g - 1u) >> 1) & 1u, kSitePVDone,
                                  abort_flag, lim);
                    if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const float a = rescale_o ? alpha : 1.0f;
                    const float2 a2 = make_float2(a, a);
#pragma unroll 1
                    for (int ch = 0; ch < D / 32; ++ch) {
                        uint32_t o[32];
                        ptx::tmem_ld32(tO + ch * 32, o);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), a2);
                            o[2 * e] = __float_as_uint(v.x);
                            o[2 * e + 1] = __float_as_uint(v.y);
                        }
                        ptx::tmem_st32(tO + ch * 32, o);
                    }
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(G::kBarPFull + (int)(g & 1u)));
            }
            if (!ok) break;
            // this half's (m, l) for the epilogue, into the buffer of the unit two back once the
            // epilogue has read that unit's (units of one key tile can run that far ahead)
            if (u >= 2) {
                ok = wait_bar(bar(G::kBarStatsFree + (u & 1)), (uint32_t)((u >> 1) - 1) & 1u, kSiteStats, abort_flag,
                              lim);
                if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
            }
            stats[((u & 1) * 2 + h) * kBM + row] = make_float2(m_ref, l);
            ptx::mbar_arrive(bar(G::kBarStats + (u & 1)));
        }
    } else if (warp < sq::kWarpEpi + 4) {
        // ------------------------------------------------ merge of the halves and epilogue
        // O = (w_a O_a + w_b O_b) / (w_a l_a + w_b l_b) with w_h = 2^((m_h - m) c), m the
        // larger reference; a finite m_h keeps w_h >= 2^-125 (a finite logit never loses its
        // weight entirely) and m_h = -inf (no key of the half seen) gives w_h = 0.  The same
        // rule merges key splits in the combine kernel.
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tOa = tmem + lane_off + 256u, tOb = tOa + (uint32_t)D;
        const float c = p.scale_log2;
        const uint32_t region = sbase + G::kSmemStage + (uint32_t)((warp - sq::kWarpEpi) * kStageBytes);
        int u = 0;
        bool ok = true;
        for (int k = blockIdx.x; k < p.n_items && ok; k += gridDim.x, ++u) {
            const Item it = decode_item<kCausal>(p, k);
            ok = wait_bar(bar(G::kBarOFull), (uint32_t)u & 1u, kSiteOFull, abort_flag, lim) &&
                 wait_bar(bar(G::kBarStats + (u & 1)), (uint32_t)(u >> 1) & 1u, kSiteStats, abort_flag, lim);
            if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
            ptx::tc_fence_after();
            const float2 sa = stats[((u & 1) * 2 + 0) * kBM + row];
            const float2 sb = stats[((u & 1) * 2 + 1) * kBM + row];
            ptx::mbar_arrive(bar(G::kBarStatsFree + (u & 1)));
            const float m = fmaxf(sa.x, sb.x);
            const float wa = (sa.x == -INFINITY) ? 0.0f : ptx::ex2_approx(fmaxf((sa.x - m) * c, -125.0f));
            const float wb = (sb.x == -INFINITY) ? 0.0f : ptx::ex2_approx(fmaxf((sb.x - m) * c, -125.0f));
            const float l = fmaf(wa, sa.y, wb * sb.y);
            const int qrow = it.qb * kUnitRows + row;
            const bool valid_row = qrow < p.Sq;
            // 16 merged columns of O (still unnormalised) from the two accumulators
            auto merged16 = [&](int c16, uint32_t (&y)[16]) {
                uint32_t a[16], b[16];
                ptx::tmem_ld16_nowait(tOa + 16u * c16, a);
                ptx::tmem_ld16_nowait(tOb + 16u * c16, b);
                ptx::tmem_wait_ld16(a);
                ptx::tmem_wait_ld16(b);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    y[e] = __float_as_uint(fmaf(wa, __uint_as_float(a[e]), wb * __uint_as_float(b[e])));
            };
            if (it.split_slot < 0) {
                const float inv = 1.0f / l;
                // natural-log log-sum-exp of the scaled logits: (m*c + log2 l) * ln 2
                if (p.lse && valid_row)
                    p.lse[((long long)it.b * p.H + it.h) * p.Sq + qrow] = (m * c + log2f(l)) * kLn2;
                const int r0 = it.qb * kUnitRows + quarter * kStageRowsPerWarp;
#pragma unroll
                for (int hc = 0; hc < G::kChunks; ++hc) {
                    uint32_t w[32];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t y[16];
                        merged16(4 * hc + q, y);
                        scale_round_pairs<8>(y, inv, p.round_mode, w + 8 * q);
                    }
                    if (hc == G::kChunks - 1) {
                        // O_a and O_b are read: the next unit's PV GEMMs may overwrite them
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(bar(G::kBarOEmpty));
                    }
                    // the region's previous TMA store (if any) has finished reading it
                    if (lane == 0) ptx::bulk_wait_read0();
                    __syncwarp();
                    // row `lane` of the region; 16-byte piece pc is stored at pc ^ (lane & 7)
                    // (128-byte swizzle)
                    const uint32_t rowaddr = region + (uint32_t)lane * 128u;
#pragma unroll
                    for (int pc = 0; pc < 8; ++pc)
                        ptx::st_shared_v4(rowaddr + (((uint32_t)pc ^ (uint32_t)(lane & 7)) << 4), w[4 * pc],
                                          w[4 * pc + 1], w[4 * pc + 2], w[4 * pc + 3]);
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (p.bshd) ptx::tma_store_4d(&omap, region, hc * 64, it.h, r0, it.b);
                        else ptx::tma_store_4d(&omap, region, hc * 64, r0, it.h, it.b);
                        ptx::bulk_commit();
                    }
                }
            } else {
                // split partial: O/l in fp32 (the raw sum when l == 0) and LSE in log2 units
                const float inv = (l > 0.0f) ? 1.0f / l : 1.0f;
                const long long wrow = (long long)it.split_slot * kUnitRows + row;
#pragma unroll 1
                for (int c16 = 0; c16 < D / 16; ++c16) {
                    uint32_t y[16];
                    merged16(c16, y);
                    if (valid_row) {
                        float4* d4 = reinterpret_cast<float4*>(p.ws_o + wrow * D + 16 * c16);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            d4[v4] = make_float4(__uint_as_float(y[4 * v4]) * inv, __uint_as_float(y[4 * v4 + 1]) * inv,
                                                 __uint_as_float(y[4 * v4 + 2]) * inv, __uint_as_float(y[4 * v4 + 3]) * inv);
                    }
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(G::kBarOEmpty));
                if (valid_row) p.ws_lse[wrow] = m * c + log2f(l);
            }
        }
    }

    // ---------------------------------------------------------------------- teardown
    if (warp >= sq::kWarpEpi && warp < sq::kWarpEpi + 4 && lane == 0) ptx::bulk_wait0();   // output stores complete
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == sq::kWarpMma) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, sq::kTmemCols);
    }
}

// ------------------------------------------------------------------------------ combine
struct CombineParams {
    int H, Sq, nq, nsplit, n_full, split_units, round_mode;
    const float* ws_o;
    const float* ws_lse;
    __nv_bfloat16* o;
    long long o_sb, o_ss, o_sh;
    float* lse;            // optional [B][H][Sq] natural-log log-sum-exp, or null
};

// Merge of the split partials: one output row of a split unit per group of W warps (W = 1,
// 2, 4 or 8 by split count; 8 / W rows per 256-thread block).  Warp w of a row takes splits
// w, w + W, w + 2W, ..., four at a time, with all four partial rows and their LSEs loaded
// before the row's maximum LSE (read by the lanes in parallel) is reduced, so a row costs one
// memory round trip when it has at most 4W splits.  Weights are 2^(LSE_s - max), clamped at
// >= 2^-125 for a finite LSE_s; a -inf LSE weighs 0.  Each warp sums its splits in increasing
// order, and the row's warps are then summed in warp order through shared memory: a fixed
// order, so results are deterministic.  Each lane owns D/32 of the D columns.  Launched as a
// programmatic dependent of the attention kernel: it starts as that kernel's CTAs retire and
// waits for its memory before reading.  [MoonMath] "Data placement and the 16x16x16 choice"
// (tail KV split).
template <int D, int W>
__global__ void __launch_bounds__(256) attn_combine_kernel(const CombineParams p) {
    constexpr int kC = D / 32;                 // columns per lane: 4 or 2
    constexpr int kRowsPerBlock = 8 / W;
    constexpr int kLoads = 4;                  // splits a warp has in flight
    __shared__ float red[kRowsPerBlock][W > 1 ? W : 1][D + 1];   // per-warp sums (+ weight sum)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rsub = warp / W, w = warp % W;
    const long long gr = (long long)blockIdx.x * kRowsPerBlock + rsub;
    int t = 0, r = 0, b = 0, h = 0, qrow = 0;
    bool valid = gr < (long long)p.split_units * kUnitRows;
    if (valid) {
        t = (int)(gr / kUnitRows);
        r = (int)(gr % kUnitRows);
        const int unit = p.n_full + t;
        const int qb = unit % p.nq, bh = unit / p.nq;
        h = bh % p.H;
        b = bh / p.H;
        qrow = qb * kUnitRows + r;
        valid = qrow < p.Sq;
    }
    float acc[kC];
#pragma unroll
    for (int e = 0; e < kC; ++e) acc[e] = 0.f;
    float wsum = 0.f, mx = -INFINITY;
    bool any_nan = false;
    if (valid) {
        const long long base = (long long)t * p.nsplit * kUnitRows + r;
        const float* src = p.ws_o + base * D + lane * kC;
        auto load = [&](int s, float (&v)[kC], float& e) {
            const float* vq = src + (long long)s * kUnitRows * D;
            if constexpr (kC == 4) {
                const float4 x = *reinterpret_cast<const float4*>(vq);
                v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
            } else {
                const float2 x = *reinterpret_cast<const float2*>(vq);
                v[0] = x.x; v[1] = x.y;
            }
            e = p.ws_lse[base + (long long)s * kUnitRows];
        };
        // this warp's first splits, in flight while the row maximum is found
        float v[kLoads][kC], lse[kLoads];
#pragma unroll
        for (int i = 0; i < kLoads; ++i)
            if (w + i * W < p.nsplit) load(w + i * W, v[i], lse[i]);
        for (int s = lane; s < p.nsplit; s += 32) {
            const float e = p.ws_lse[base + (long long)s * kUnitRows];
            any_nan |= (e != e);
            mx = fmaxf(mx, e);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
        any_nan = __any_sync(0xFFFFFFFFu, any_nan);
        for (int s0 = w;; s0 += kLoads * W) {
#pragma unroll
            for (int i = 0; i < kLoads; ++i) {
                if (s0 + i * W < p.nsplit) {
                    const float wt = (lse[i] == -INFINITY) ? 0.0f : ptx::ex2_approx(fmaxf(lse[i] - mx, -125.0f));
                    wsum += wt;
#pragma unroll
                    for (int e = 0; e < kC; ++e) acc[e] += wt * v[i][e];
                }
            }
            if (s0 + kLoads * W >= p.nsplit) break;
#pragma unroll
            for (int i = 0; i < kLoads; ++i)
                if (s0 + (kLoads + i) * W < p.nsplit) load(s0 + (kLoads + i) * W, v[i], lse[i]);
        }
    }
    if constexpr (W > 1) {
        if (valid && w > 0) {
#pragma unroll
            for (int e = 0; e < kC; ++e) red[rsub][w][lane * kC + e] = acc[e];
            if (lane == 0) red[rsub][w][D] = wsum;
        }
        __syncthreads();
        if (valid && w == 0) {
#pragma unroll 1
            for (int ww = 1; ww < W; ++ww) {
#pragma unroll
                for (int e = 0; e < kC; ++e) acc[e] += red[rsub][ww][lane * kC + e];
                wsum += red[rsub][ww][D];
            }
        }
    }
    if (!valid || w != 0) return;
    const bool nan_row = any_nan || mx == -INFINITY;
    const float inv = 1.0f / wsum;
    // sum_s 2^LSE_s = 2^mx * wsum (base 2), reported in natural log
    if (p.lse && lane == 0)
        p.lse[((long long)b * p.H + h) * p.Sq + qrow] = any_nan ? NAN : (mx + log2f(wsum)) * kLn2;
    uint32_t bits[kC];
#pragma unroll
    for (int e = 0; e < kC; ++e) bits[e] = nan_row ? 0x7FC0u : round_bf16_bits(acc[e] * inv, p.round_mode);
    __nv_bfloat16* orow = p.o + (long long)b * p.o_sb + (long long)qrow * p.o_ss + (long long)h * p.o_sh;
    if constexpr (kC == 4)
        *reinterpret_cast<uint2*>(orow + lane * 4) = make_uint2(bits[0] | (bits[1] << 16), bits[2] | (bits[3] << 16));
    else
        *reinterpret_cast<uint32_t*>(orow + lane * 2) = bits[0] | (bits[1] << 16);
}

// ------------------------------------------------------------------------------ variable-length batches
// Preprocessing of a variable-length batch, one CTA, before the attention kernel (which is
// its programmatic dependent and waits for its memory):
//   * checks the offsets: cu_q and cu_k start at >= 0, never decrease, and end within the
//     packed tensors; otherwise it records ATTN_ERR_INVALID_ARG at the sequence-length site and
//     schedules no work, so no load or store is issued from a bad offset;
//   * per sequence with both queries and keys, tensor maps for its Q, K, V and O rows: copies
//     of the whole-tensor maps with the base moved to the sequence's first row and the row
//     count set to its length, so loads past its end read zeros and stores past its end are
//     dropped, as at the end of a dense tensor (tensormap.replace, then a release fence for
//     the tensor-map proxy; the attention kernel acquires each map before its first use);
//   * the work list: every (sequence, 256-row query block) pair, ordered by the key tiles it
//     runs, most first (a counting sort on that count, capped at kCostBuckets - 1; pairs of
//     equal count in any order, which moves work between CTAs but changes no result), and
//     the item count, H >> pack_shift per entry;
//   * key splits (max_splits >= 2), when the pairs' items number fewer than the attention
//     kernel's CTAs: with P pairs and Gp = CTAs / (items per pair) entry places (P < Gp), a
//     pair of cost c becomes n(c) = min(max_splits, Gp, ceil(c / M)) consecutive entries (b,
//     qb, part, n).  M is the smallest with sum n(c) <= Gp (one wave: every item a CTA of its
//     own), or, when the pairs' items fill at least half of the CTAs, the smallest with
//     sum n(c) <= 2 Gp (two waves, whose alternating order pairs a CTA's heavy first item
//     with a light second one) if that gives the busiest CTA less modelled work (key tiles
//     plus a fixed cost per item).  Split slots stay below twice the CTA count.  n depends
//     only on c (and the launch), so the result is a function of the inputs and the CTA
//     count;
//   * a sequence with queries but no keys: every query sees no key, so its O rows are NaN
//     (stored 0x7FC0) and its LSE rows -inf, written here.
constexpr int kCostBuckets = 4096;
constexpr int kMaxDistinct = 512;         // key splits: distinct pair costs considered
constexpr int kMaxSplitGrid = 1024;       // key splits: attention CTAs considered
constexpr int kItemOverheadTiles = 2;     // key splits: modelled fixed cost of an item, in key tiles

struct VarlenPrep {
    const int* cu_q;
    const int* cu_k;                       // unpaged: key offsets
    const int* seqlens_k;                  // paged: keys per sequence
    const int* block_table;                // paged: [B][max_pages]
    int paged, page_size, max_pages, num_pages;
    int pack_shift;                        // head packing: 2^shift heads per tile row group
    int max_splits;                        // key parts per pair at most (< 2: no splits)
    int grid;                              // the attention kernel's CTAs
    int B, H, causal;
    long long total_q, total_k;
    long long q_row_bytes, kv_row_bytes;   // bytes per token row: H*d*2, Hkv*d*2
    const char* q;
    const char* k;
    const char* v;
    char* o;
    float* lse;                            // optional [H][total_q]
    CUtensorMap* maps;                     // [B][4]: Q, K, V, O
    int4* blocks;                          // (sequence, query block, part, parts), heaviest first
    int* n_items;                          // [0] items; [1] items with key splits, else 0
};

__device__ __forceinline__ void copy_map(CUtensorMap* dst, const CUtensorMap* src) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(CUtensorMap) / 16); ++i) d4[i] = s4[i];
}

// the map at dst (a copy of a whole-tensor map) restricted to `rows` token rows from `base`
__device__ __forceinline__ void narrow_map(CUtensorMap* dst, const void* base, int rows) {
    asm volatile("tensormap.replace.tile.global_address.global.b1024.b64 [%0], %1;" ::"l"(dst),
                 "l"(reinterpret_cast<uint64_t>(base))
                 : "memory");
    asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 2, %1;" ::"l"(dst), "r"(rows) : "memory");
}

// key tiles the attention kernel runs for query block qb of a sequence (its bucket); a block
// holds 256 >> shift tokens (shift: the head packing's)
__device__ __forceinline__ int block_cost(int qb, int sq, int skv, int causal, int shift) {
    int tiles = (skv + kBN - 1) / kBN;
    if (causal) {
        const int last = ((qb + 1) * kUnitRows >> shift) - 1 + skv - sq;   // last visible key
        const int need = last < 0 ? 1 : last / kBN + 1;
        tiles = need < tiles ? need : tiles;
    }
    return tiles < kCostBuckets - 1 ? tiles : kCostBuckets - 1;
}

// key parts of a pair of cost c with at most M tiles a part (c >= 1, so every part has a tile:
// ceil(c / M) <= c)
__device__ __forceinline__ int split_parts(int c, int M, int max_splits) {
    const int n = (c + M - 1) / M;
    return n < max_splits ? n : max_splits;
}

// keys of sequence b (its own rows, or the used slots of its pages)
__device__ __forceinline__ int seq_keys(const VarlenPrep& a, int b) {
    return a.paged ? a.seqlens_k[b] : a.cu_k[b + 1] - a.cu_k[b];
}

__global__ void __launch_bounds__(1024) attn_varlen_prep_kernel(const __grid_constant__ CUtensorMap qmap,
                                                                const __grid_constant__ CUtensorMap kmap,
                                                                const __grid_constant__ CUtensorMap vmap,
                                                                const __grid_constant__ CUtensorMap omap,
                                                                const VarlenPrep a) {
    __shared__ int bad;
    __shared__ int bucket[kCostBuckets];   // counts, then (descending) start positions
    __shared__ int warp_sums[32];
    __shared__ int2 dist[kMaxDistinct];    // key splits: (cost, pairs) of each cost present
    __shared__ int2 sdist[kMaxDistinct];   // key splits: the same, heaviest first
    __shared__ int spre[2][kMaxDistinct];  // key splits: entries before each cost, per candidate
    __shared__ int n_dist, n_pairs, max_cost, cand[2], cand_load[2];
    __shared__ int part_tiles, part_cap;   // M of the key split (0: none), parts at most
    // the previous kernel in the stream may have written the offsets or still read this
    // workspace; the attention kernel may launch now and waits for this one's memory
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nthreads = blockDim.x;
    if (tid == 0)
        bad = (a.cu_q[0] < 0 || a.cu_q[a.B] > a.total_q ||
               (!a.paged && (a.cu_k[0] < 0 || a.cu_k[a.B] > a.total_k))) ? 1 : 0;
    for (int i = tid; i < kCostBuckets; i += nthreads) bucket[i] = 0;
    __syncthreads();
    for (int b = tid; b < a.B; b += nthreads) {
        if (a.cu_q[b + 1] < a.cu_q[b]) bad = 1;
        if (!a.paged) {
            if (a.cu_k[b + 1] < a.cu_k[b]) bad = 1;
        } else {
            const int skv = a.seqlens_k[b];
            if (skv < 0 || skv > a.max_pages * a.page_size) bad = 1;
        }
    }
    // the used page indices of each sequence: a warp per sequence, its lanes across the pages
    if (a.paged) {
        for (int b = wid; b < a.B; b += (nthreads >> 5)) {
            const int skv = a.seqlens_k[b];
            if (skv < 0 || skv > a.max_pages * a.page_size) continue;   // reported above
            const int npg = (skv + a.page_size - 1) / a.page_size;
            for (int pg = lane; pg < npg; pg += 32) {
                const int phys = a.block_table[(long long)b * a.max_pages + pg];
                if (phys < 0 || phys >= a.num_pages) bad = 1;
            }
        }
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) {
            a.n_items[0] = 0;
            a.n_items[1] = 0;
            if (atomicCAS(&g_status[0], 0u, (uint32_t)ATTN_ERR_INVALID_ARG) == 0u) atomicExch(&g_status[1], kSiteSeqlens);
        }
        return;
    }
    // per sequence: maps, NaN rows, and the cost histogram of its query blocks
    for (int base = 0; base < a.B; base += nthreads) {
        const int b = base + tid;
        int sq = 0, skv = 0;
        if (b < a.B) {
            sq = a.cu_q[b + 1] - a.cu_q[b];
            skv = seq_keys(a, b);
            if (sq > 0 && skv > 0) {
                CUtensorMap* m = a.maps + 4 * (long long)b;
                const long long q0 = a.cu_q[b];
                // K/V rows: the sequence's own, or (paged) the used slots of its last page
                long long k0 = 0;
                int krows = skv;
                if (a.paged) {
                    const int last = (skv - 1) / a.page_size;
                    k0 = (long long)a.block_table[(long long)b * a.max_pages + last] * a.page_size;
                    krows = skv - last * a.page_size;
                } else {
                    k0 = a.cu_k[b];
                }
                copy_map(m + 0, &qmap);
                copy_map(m + 1, &kmap);
                copy_map(m + 2, &vmap);
                copy_map(m + 3, &omap);
                narrow_map(m + 0, a.q + q0 * a.q_row_bytes, sq);
                narrow_map(m + 1, a.k + k0 * a.kv_row_bytes, krows);
                narrow_map(m + 2, a.v + k0 * a.kv_row_bytes, krows);
                narrow_map(m + 3, a.o + q0 * a.q_row_bytes, sq);
                const int tb = kUnitRows >> a.pack_shift;        // tokens per block
                const int nqb = (sq + tb - 1) / tb;
                for (int qb = 0; qb < nqb; ++qb)
                    atomicAdd(&bucket[block_cost(qb, sq, skv, a.causal, a.pack_shift)], 1);
            }
        }
        // queries with no keys: the warp writes each such sequence's NaN rows and -inf LSE
        unsigned nan_seqs = __ballot_sync(0xFFFFFFFFu, b < a.B && sq > 0 && skv == 0);
        while (nan_seqs) {
            const int src = __ffs(nan_seqs) - 1;
            nan_seqs &= nan_seqs - 1;
            const long long q0 = a.cu_q[base + (wid << 5) + src];
            const long long rows = __shfl_sync(0xFFFFFFFFu, sq, src);
            const uint4 nan8 = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
            uint4* dst = reinterpret_cast<uint4*>(a.o + q0 * a.q_row_bytes);
            for (long long e = lane; e < rows * a.q_row_bytes / 16; e += 32) dst[e] = nan8;
            if (a.lse)
                for (long long e = lane; e < rows * a.H; e += 32) a.lse[(e / rows) * a.total_q + q0 + e % rows] = -INFINITY;
        }
    }
    __syncthreads();
    // key splits, when the pairs' items number fewer than the CTAs (P < Gp).  Warp 0: the
    // smallest M (tiles per part) whose entries fit one wave, Gp places, by bisection with the
    // lanes summing over the costs present; every item then has a CTA of its own, and this
    // never loses to no split (its longest part is at most the largest cost).  When the items
    // fill at least half of the CTAs, warp 1 also finds the smallest M fitting two waves,
    // 2 Gp places, and warps 0 and 1 model the busiest CTA's work under each: with the costs
    // heaviest first (a rank sort; each cost is a bucket of its own), item k belongs to entry
    // k / per_block, which a search of the prefix of entries places in its cost and part; CTA c
    // runs items c and 2G - 1 - c (round_item's alternation); an item costs its key tiles plus
    // kItemOverheadTiles.  Two waves are taken only when that is less.  Each bucket's count
    // then becomes its entries.
    if (a.max_splits > 1) {
        if (tid == 0) {
            n_dist = 0;
            n_pairs = 0;
            max_cost = 0;
        }
        __syncthreads();
        for (int i = tid; i < kCostBuckets; i += nthreads) {
            const int n = bucket[i];
            if (n > 0) {
                const int pos = atomicAdd(&n_dist, 1);
                if (pos < kMaxDistinct) dist[pos] = make_int2(i, n);
                atomicAdd(&n_pairs, n);
                atomicMax(&max_cost, i);
            }
        }
        __syncthreads();
        const int per_block = a.H >> a.pack_shift;
        const int gp = a.grid / per_block;
        const int ms = a.max_splits < gp ? a.max_splits : gp;
        const int nd = n_dist, np = n_pairs, cmax = max_cost;
        int M = 0;
        if (np > 0 && gp > np && nd <= kMaxDistinct && a.grid <= kMaxSplitGrid) {
            const bool two = 2 * np * per_block >= a.grid;
            if (wid < (two ? 2 : 1)) {
                const int places = (wid + 1) * gp;
                int lo = 1, hi = cmax;         // cmax fits: every pair one entry, np < places
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    int e = 0;
                    for (int i = lane; i < nd; i += 32) e += dist[i].y * split_parts(dist[i].x, mid, ms);
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) e += __shfl_xor_sync(0xFFFFFFFFu, e, off);
                    if (e <= places) hi = mid;
                    else lo = mid + 1;
                }
                if (lane == 0) cand[wid] = lo;
            }
            if (two)
                for (int i = tid; i < nd; i += nthreads) {
                    const int c = dist[i].x;
                    int rank = 0;
                    for (int j = 0; j < nd; ++j) rank += dist[j].x > c ? 1 : 0;
                    sdist[rank] = dist[i];
                }
            __syncthreads();
            if (two) {
                if (wid < 2) {
                    const int m = cand[wid];
                    int* pre = spre[wid];
                    int carry = 0;
                    for (int i0 = 0; i0 < nd; i0 += 32) {
                        const int i = i0 + lane;
                        const int ent = i < nd ? sdist[i].y * split_parts(sdist[i].x, m, ms) : 0;
                        int incl = ent;
#pragma unroll
                        for (int off = 1; off < 32; off <<= 1) {
                            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
                            if (lane >= off) incl += y;
                        }
                        if (i < nd) pre[i] = carry + incl - ent;
                        carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
                    }
                    __syncwarp();
                    const int n_it = carry * per_block;   // items: at most 2 G
                    int worst = 0;
                    for (int c = lane; c < a.grid; c += 32) {
                        int load = 0;
                        for (int t = 0; t < 2; ++t) {
                            const int k = t == 0 ? c : 2 * a.grid - 1 - c;
                            if (k >= n_it) continue;
                            const int e = k / per_block;
                            int lo = 0, hi = nd - 1;  // the last cost whose entries start at or before e
                            while (lo < hi) {
                                const int mid = (lo + hi + 1) >> 1;
                                if (pre[mid] <= e) lo = mid;
                                else hi = mid - 1;
                            }
                            const int cst = sdist[lo].x, n = split_parts(cst, m, ms);
                            const int part = (e - pre[lo]) % n;
                            load += cst / n + (part < cst % n ? 1 : 0) + kItemOverheadTiles;
                        }
                        worst = max(worst, load);
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) worst = max(worst, __shfl_xor_sync(0xFFFFFFFFu, worst, off));
                    if (lane == 0) cand_load[wid] = worst;
                }
                __syncthreads();
            }
            M = (two && cand_load[1] < cand_load[0]) ? cand[1] : cand[0];
        }
        if (tid == 0) {
            part_tiles = M;
            part_cap = ms;
        }
        if (M > 0)
            for (int i = tid; i < kCostBuckets; i += nthreads) bucket[i] *= split_parts(i, M, ms);
        __syncthreads();
    } else if (tid == 0) {
        part_tiles = 0;
    }
    // start of each bucket in descending order: thread t owns buckets kCostBuckets - 4t - 1
    // down to kCostBuckets - 4t - 4; an exclusive scan of the threads' sums over t
    constexpr int kPer = kCostBuckets / 1024;
    int local = 0;
    if (tid < 1024)
        for (int i = 0; i < kPer; ++i) local += bucket[kCostBuckets - 1 - kPer * tid - i];
    int incl = local;
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
    int start = (wid > 0 ? warp_sums[wid - 1] : 0) + incl - local;
    if (tid == nthreads - 1) {
        a.n_items[0] = (start + local) * (a.H >> a.pack_shift);
        a.n_items[1] = part_tiles > 0 ? a.n_items[0] : 0;   // items the merge kernel visits
    }
    __syncthreads();
    if (tid < 1024)
        for (int i = 0; i < kPer; ++i) {
            const int key = kCostBuckets - 1 - kPer * tid - i;
            const int c = bucket[key];
            bucket[key] = start;
            start += c;
        }
    __syncthreads();
    // scatter every pair to its bucket's next position
    for (int b = tid; b < a.B; b += nthreads) {
        const int sq = a.cu_q[b + 1] - a.cu_q[b], skv = seq_keys(a, b);
        if (sq <= 0 || skv <= 0) continue;
        const int tb = kUnitRows >> a.pack_shift;
        const int nqb = (sq + tb - 1) / tb;
        for (int qb = 0; qb < nqb; ++qb) {
            const int cost = block_cost(qb, sq, skv, a.causal, a.pack_shift);
            const int n = part_tiles > 0 ? split_parts(cost, part_tiles, part_cap) : 1;
            const int pos = atomicAdd(&bucket[cost], n);
            for (int i = 0; i < n; ++i) a.blocks[pos + i] = make_int4(b, qb, i, n);
        }
    }
    asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
}

// Merge of a variable-length batch's key parts, a programmatic dependent of the attention
// kernel.  Block (x, y) takes tile rows 32 y .. 32 y + 31 of items k = x, x + G, ... (G blocks
// along x) whose entry is the first part of a split pair (others are skipped); warp w merges
// rows 32 y + w + 8 i (i = 0 .. 3, so that the few rows of a decoding step fall to different
// warps), lane l holding
// columns kC l .. kC l + kC - 1.  The parts' slots are k + s * per_block (s = 0 .. n - 1: the
// pair's entries are consecutive).  A row's part LSEs are read across the lanes at once, and
// its parts' partial rows four at a time.  Weights follow the dense combine: 2^(LSE_s - max),
// clamped at >= 2^-125 for a finite LSE_s, 0 for -inf; a NaN LSE or an all -inf row gives a
// NaN row (0x7FC0).  Parts are summed in order, so the result is deterministic.  Tile row r is
// token (256 qb + r) >> shift of the sequence, head h + (r & (2^shift - 1)).  [MoonMath] "Data
// placement and the 16x16x16 choice" (key splits of the tail), applied to the variable-length
// work list.
struct VarlenCombine {
    const int4* blocks;
    const int* n_items;                    // [1]: items when keys were split, else 0
    const int* cu_q;
    const float* ws_o;                     // [slot][256][D]
    const float* ws_lse;                   // [slot][256], log2 units
    __nv_bfloat16* o;                      // [total_q][H][D]
    float* lse;                            // optional [H][total_q], natural log
    long long total_q;
    int H, pack_shift, round_mode;
};

template <int D>
__global__ void __launch_bounds__(256) attn_varlen_combine_kernel(const VarlenCombine p) {
    constexpr int kC = D / 32;             // columns per lane: 4 or 2
    constexpr int kLoads = 4;              // parts' rows in flight
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int n_items = __ldg(p.n_items + 1);
    const int per_block = p.H >> p.pack_shift;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long pstride = (long long)per_block * kUnitRows;   // rows from one part to the next
    for (int k = blockIdx.x; k < n_items; k += gridDim.x) {
        const int4 e = __ldg(p.blocks + k / per_block);
        if (e.w < 2 || e.z != 0) continue;
        const int n = e.w;
        const int q0 = __ldg(p.cu_q + e.x);
        const int sq = __ldg(p.cu_q + e.x + 1) - q0;
        const int h0 = (k % per_block) << p.pack_shift;
        for (int i = 0; i < 4; ++i) {
            const int r = blockIdx.y * 32 + warp + 8 * i;
            const int tok = (e.y * kUnitRows + r) >> p.pack_shift;
            if (tok >= sq) break;              // tokens do not decrease with r
            const int h = h0 + (r & ((1 << p.pack_shift) - 1));
            const long long row0 = (long long)k * kUnitRows + r;      // part 0's row
            float mx = -INFINITY;
            bool any_nan = false;
            for (int s = lane; s < n; s += 32) {
                const float l = p.ws_lse[row0 + s * pstride];
                any_nan |= (l != l);
                mx = fmaxf(mx, l);
            }
    #pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
            any_nan = __any_sync(0xFFFFFFFFu, any_nan);
            float acc[kC];
    #pragma unroll
            for (int c = 0; c < kC; ++c) acc[c] = 0.f;
            float wsum = 0.f;
            for (int s0 = 0; s0 < n; s0 += 32) {
                // lane j holds the weight of part s0 + j
                float wt = 0.f;
                if (s0 + lane < n) {
                    const float l = p.ws_lse[row0 + (s0 + lane) * pstride];
                    wt = (l == -INFINITY) ? 0.0f : ptx::ex2_approx(fmaxf(l - mx, -125.0f));
                }
                const int m = n - s0 < 32 ? n - s0 : 32;
                for (int j0 = 0; j0 < m; j0 += kLoads) {
                    float v[kLoads][kC];
    #pragma unroll
                    for (int j = 0; j < kLoads; ++j) {
                        if (j0 + j < m) {
                            const float* src = p.ws_o + (row0 + (s0 + j0 + j) * pstride) * D + lane * kC;
                            if constexpr (kC == 4) {
                                const float4 x = *reinterpret_cast<const float4*>(src);
                                v[j][0] = x.x; v[j][1] = x.y; v[j][2] = x.z; v[j][3] = x.w;
                            } else {
                                const float2 x = *reinterpret_cast<const float2*>(src);
                                v[j][0] = x.x; v[j][1] = x.y;
                            }
                        }
                    }
    #pragma unroll
                    for (int j = 0; j < kLoads; ++j) {
                        if (j0 + j < m) {
                            const float w = __shfl_sync(0xFFFFFFFFu, wt, j0 + j);
                            wsum += w;
    #pragma unroll
                            for (int c = 0; c < kC; ++c) acc[c] += w * v[j][c];
                        }
                    }
                }
            }
            const bool nan_row = any_nan || mx == -INFINITY;
            const float inv = 1.0f / wsum;
            if (p.lse && lane == 0)
                p.lse[(long long)h * p.total_q + q0 + tok] = any_nan ? NAN : (mx + log2f(wsum)) * kLn2;
            uint32_t bits[kC];
    #pragma unroll
            for (int c = 0; c < kC; ++c) bits[c] = nan_row ? 0x7FC0u : round_bf16_bits(acc[c] * inv, p.round_mode);
            __nv_bfloat16* orow = p.o + ((long long)(q0 + tok) * p.H + h) * D;
            if constexpr (kC == 4)
                *reinterpret_cast<uint2*>(orow + lane * 4) = make_uint2(bits[0] | (bits[1] << 16), bits[2] | (bits[3] << 16));
            else
                *reinterpret_cast<uint32_t*>(orow + lane * 2) = bits[0] | (bits[1] << 16);
        }
    }
}

// ------------------------------------------------------------------------------ host side
struct DeviceInfo {
    bool init = false;
    int sms = 0, major = 0, minor = 0;
    bool attr_set = false;
    void* ws = nullptr;
    size_t ws_bytes = 0;
};
constexpr int kMaxDevices = 64;
std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

attn_args_t plain_args(const void* q, const void* k, const void* v, void* o, int64_t B, int64_t H, int64_t Sq,
                       int64_t Skv, int64_t d, int layout, int round_mode) {
    attn_args_t a;
    memset(&a, 0, sizeof a);
    a.q = q; a.k = k; a.v = v; a.o = o;
    a.B = B; a.H = H; a.Hkv = H; a.Sq = Sq; a.Skv = Skv; a.d = d;
    a.layout = layout; a.round_mode = round_mode;
    return a;
}

// Shape checks shared by the planner and the launchers (pointers are not looked at).
int validate_shape(const attn_args_t& a, const attn_options_t* opts) {
    if (a.B < 1 || a.H < 1 || a.Hkv < 1 || a.Sq < 1 || a.Skv < 1 || a.d < 1) return ATTN_ERR_INVALID_ARG;
    if (a.H % a.Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (a.layout != ATTN_LAYOUT_BSHD && a.layout != ATTN_LAYOUT_BHSD) return ATTN_ERR_INVALID_ARG;
    if (a.round_mode < ATTN_ROUND_RTNE || a.round_mode > ATTN_ROUND_RTZ) return ATTN_ERR_INVALID_ARG;
    if ((a.causal != 0 && a.causal != 1) || a.reserved != 0) return ATTN_ERR_INVALID_ARG;
    if (a.d != 128 && a.d != 64) return ATTN_ERR_UNSUPPORTED;
    if (a.causal && opts && opts->force_splits > 1) return ATTN_ERR_UNSUPPORTED;
    if (opts && opts->test_hooks != 0 && opts->test_hooks != ATTN_TEST_WITHHOLD_O_READY) return ATTN_ERR_INVALID_ARG;
    // TMA coordinates and the kernels' unit/row indices are int32
    const int64_t lim = (int64_t)1 << 30;
    if (a.Sq > lim || a.Skv > lim || a.B > lim || a.H > lim) return ATTN_ERR_UNSUPPORTED;
    if (a.B * a.H > lim || a.B * a.H * cdiv(a.Sq, kUnitRows) > lim) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

int validate(const attn_args_t& a, const attn_options_t* opts) {
    if (!a.q || !a.k || !a.v || !a.o) return ATTN_ERR_INVALID_ARG;
    const int st = validate_shape(a, opts);
    if (st != ATTN_OK) return st;
    if (((uintptr_t)a.q | (uintptr_t)a.k | (uintptr_t)a.v | (uintptr_t)a.o) & 15u) return ATTN_ERR_MISALIGNED;
    if ((uintptr_t)a.lse & 3u) return ATTN_ERR_MISALIGNED;
    const uintptr_t qbytes = (uintptr_t)(a.B * a.H * a.Sq * a.d * 2), kvbytes = (uintptr_t)(a.B * a.Hkv * a.Skv * a.d * 2);
    const uintptr_t ob = (uintptr_t)a.o, oe = ob + qbytes;
    const uintptr_t qb = (uintptr_t)a.q, qe = qb + qbytes;
    const uintptr_t kb = (uintptr_t)a.k, ke = kb + kvbytes;
    const uintptr_t vb = (uintptr_t)a.v, ve = vb + kvbytes;
    auto overlap = [](uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; };
    if (overlap(ob, oe, qb, qe) || overlap(ob, oe, kb, ke) || overlap(ob, oe, vb, ve)) return ATTN_ERR_ALIAS;
    if (a.lse) {
        const uintptr_t lb = (uintptr_t)a.lse, le = lb + (uintptr_t)(a.B * a.H * a.Sq * 4);
        if (overlap(lb, le, ob, oe) || overlap(lb, le, qb, qe) || overlap(lb, le, kb, ke) || overlap(lb, le, vb, ve))
            return ATTN_ERR_ALIAS;
    }
    return ATTN_OK;
}

void make_plan(const attn_args_t& a, int64_t sms, const attn_options_t* opts, attn_plan_t* pl) {
    const int64_t nq = cdiv(a.Sq, kUnitRows);
    const int64_t U = a.B * a.H * nq;
    const int64_t nkv = cdiv(a.Skv, kBN);
    int64_t G = sms;
    if (opts && opts->max_ctas > 0 && opts->max_ctas < G) G = opts->max_ctas;
    if (G < 1) G = 1;
    int64_t full = U, split_units = 0, ns = 1;
    if (a.causal) {
        // causal units differ in length and run heaviest first: no key split
    } else if (opts && opts->force_splits > 0) {
        ns = opts->force_splits < nkv ? opts->force_splits : nkv;
        if (ns > 1) { full = 0; split_units = U; }
        else ns = 1;
    } else {
        const int64_t T = U % G;
        if (T > 0) {
            int64_t cand = G / T;
            const int64_t by_tiles = nkv / kMinTilesPerSplit;
            if (by_tiles < cand) cand = by_tiles;
            if (cand >= 2) { ns = cand; full = U - T; split_units = T; }
        }
    }
    pl->units = U;
    pl->kv_tiles = nkv;
    pl->full_items = full;
    pl->split_units = split_units;
    pl->splits = split_units ? ns : 1;
    pl->items = full + split_units * pl->splits;
    pl->grid = pl->items < G ? pl->items : G;
    pl->workspace_bytes = split_units ? split_units * pl->splits * kUnitRows * (a.d * 4 + 4) : 0;
}

int device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return ATTN_ERR_NO_DEVICE; }
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> g(g_mutex);
    DeviceInfo& di = g_dev[dev];
    if (!di.init) {
        if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_NO_DEVICE;
        }
        di.init = true;
    }
    if (di.major != 10 || di.minor != 3) return ATTN_ERR_NO_DEVICE;
    if (!di.attr_set) {
        const int s128 = Geo<128>::kSmemAlloc, s64 = Geo<64>::kSmemAlloc;
        if (cudaFuncSetAttribute(attn_fwd_kernel<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, s128) !=
                cudaSuccess ||
            cudaFuncSetAttribute(attn_fwd_kernel<128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, s128) !=
                cudaSuccess ||
            cudaFuncSetAttribute(attn_fwd_kernel<64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, s64) !=
                cudaSuccess ||
            cudaFuncSetAttribute(attn_fwd_kernel<64, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, s64) !=
                cudaSuccess ||
            cudaFuncSetAttribute(attn_fwd_kernel<128, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 s128) != cudaSuccess ||
            cudaFuncSetAttribute(attn_fwd_kernel<128, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 s128) != cudaSuccess ||
            cudaFuncSetAttribute(attn_fwd_kernel<64, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, s64) !=
                cudaSuccess ||
            cudaFuncSetAttribute(attn_fwd_kernel<64, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, s64) !=
                cudaSuccess)
            return ATTN_ERR_CUDA;
        const int t128 = sq::Geo<128>::kSmemAlloc, t64 = sq::Geo<64>::kSmemAlloc;
        if (cudaFuncSetAttribute(attn_fwd_short_kernel<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 t128) != cudaSuccess ||
            cudaFuncSetAttribute(attn_fwd_short_kernel<128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 t128) != cudaSuccess ||
            cudaFuncSetAttribute(attn_fwd_short_kernel<64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, t64) !=
                cudaSuccess ||
            cudaFuncSetAttribute(attn_fwd_short_kernel<64, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, t64) !=
                cudaSuccess)
            return ATTN_ERR_CUDA;
        di.attr_set = true;
    }
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) !=
                cudaSuccess ||
            qr != cudaDriverEntryPointSuccess || !fn)
            return ATTN_ERR_CUDA;
        g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    *out = &di;
    return ATTN_OK;
}

// Tensor map over one bf16 tensor, dims ordered innermost-first so strides increase:
// BSHD -> (d, H, S, B), BHSD -> (d, S, H, B); box = 64 d x 128 rows, 128-byte swizzle.
bool encode_map(CUtensorMap* m, const void* ptr, int64_t B, int64_t H, int64_t S, int64_t d, bool bshd,
                uint32_t rows = kBM, uint32_t heads = 1) {
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
    dims[0] = (cuuint64_t)d;
    if (bshd) {
        dims[1] = H; dims[2] = S; dims[3] = B;
        strides[0] = d * 2; strides[1] = H * d * 2; strides[2] = S * H * d * 2;
        box[0] = 64; box[1] = heads; box[2] = rows; box[3] = 1;
    } else {
        dims[1] = S; dims[2] = H; dims[3] = B;
        strides[0] = d * 2; strides[1] = S * d * 2; strides[2] = H * S * d * 2;
        box[0] = 64; box[1] = rows; box[2] = 1; box[3] = 1;
    }
    const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int launch(const attn_args_t& a, const attn_plan_t& pl, const attn_options_t* opts, void* ws, cudaStream_t stream) {
    const int64_t B = a.B, H = a.H, Sq = a.Sq, Skv = a.Skv, d = a.d;
    const int round_mode = a.round_mode;
    void* o = a.o;
    const bool bshd = a.layout == ATTN_LAYOUT_BSHD;
    CUtensorMap qm, km, vm, om;
    if (!encode_map(&qm, a.q, B, H, Sq, d, bshd) || !encode_map(&km, a.k, B, a.Hkv, Skv, d, bshd) ||
        !encode_map(&vm, a.v, B, a.Hkv, Skv, d, bshd) || !encode_map(&om, o, B, H, Sq, d, bshd, kStageRowsPerWarp))
        return ATTN_ERR_CUDA;
    FwdParams p;
    memset(&p, 0, sizeof p);
    p.B = (int)B; p.H = (int)H; p.Sq = (int)Sq; p.Skv = (int)Skv;
    p.group = (int)(H / a.Hkv);
    p.causal = a.causal;
    p.causal_off = (int)(Skv - Sq);
    p.lse = a.lse;
    p.nq = (int)cdiv(Sq, kUnitRows);
    p.nkv = (int)pl.kv_tiles;
    p.n_items = (int)pl.items;
    p.n_full = (int)pl.full_items;
    p.nsplit = (int)pl.splits;
    p.bshd = bshd ? 1 : 0;
    p.round_mode = round_mode;
    p.scale_log2 = (float)((1.0 / std::sqrt((double)d)) * 1.4426950408889634);
    p.tau = 8.0f;
    p.o = reinterpret_cast<__nv_bfloat16*>(o);
    if (pl.split_units) {
        p.ws_o = reinterpret_cast<float*>(ws);
        p.ws_lse = p.ws_o + pl.split_units * pl.splits * kUnitRows * d;
    }
    if (bshd) { p.o_sb = Sq * H * d; p.o_ss = H * d; p.o_sh = d; }
    else { p.o_sb = H * Sq * d; p.o_ss = d; p.o_sh = Sq * d; }
    const uint32_t ms = (opts && opts->wait_limit_ms) ? opts->wait_limit_ms : 2000u;
    p.wait_limit_ns = (unsigned long long)ms * 1000000ull;
    p.test_hooks = opts ? (int)opts->test_hooks : 0;

    const attn_event_t* ev = opts ? opts->events : nullptr;
    if (ev && ev[0] && cudaEventRecord((cudaEvent_t)ev[0], stream) != cudaSuccess) return ATTN_ERR_CUDA;
    // the attention kernel is a programmatic dependent of the stream's previous kernel (it
    // waits for that kernel's memory after its prologue); the combine kernel is one of it
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t lc;
    memset(&lc, 0, sizeof lc);
    lc.gridDim = dim3((unsigned)pl.grid);
    lc.stream = stream;
    lc.attrs = pdl;
    lc.numAttrs = 1;
    cudaError_t le;
    if (Sq <= kBM) {
        // one query tile per (b, h): the short-query kernel (same items and workspace rows)
        lc.blockDim = dim3(sq::kThreads);
        if (d == 128) {
            lc.dynamicSmemBytes = sq::Geo<128>::kSmemAlloc;
            le = p.causal ? cudaLaunchKernelEx(&lc, attn_fwd_short_kernel<128, true>, qm, km, vm, om, p)
                          : cudaLaunchKernelEx(&lc, attn_fwd_short_kernel<128, false>, qm, km, vm, om, p);
        } else {
            lc.dynamicSmemBytes = sq::Geo<64>::kSmemAlloc;
            le = p.causal ? cudaLaunchKernelEx(&lc, attn_fwd_short_kernel<64, true>, qm, km, vm, om, p)
                          : cudaLaunchKernelEx(&lc, attn_fwd_short_kernel<64, false>, qm, km, vm, om, p);
        }
    } else {
        lc.blockDim = dim3(kThreads);
        if (d == 128) {
            lc.dynamicSmemBytes = Geo<128>::kSmemAlloc;
            le = p.causal ? cudaLaunchKernelEx(&lc, attn_fwd_kernel<128, true>, qm, km, vm, om, p)
                          : cudaLaunchKernelEx(&lc, attn_fwd_kernel<128, false>, qm, km, vm, om, p);
        } else {
            lc.dynamicSmemBytes = Geo<64>::kSmemAlloc;
            le = p.causal ? cudaLaunchKernelEx(&lc, attn_fwd_kernel<64, true>, qm, km, vm, om, p)
                          : cudaLaunchKernelEx(&lc, attn_fwd_kernel<64, false>, qm, km, vm, om, p);
        }
    }
    if (le != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    if (ev && ev[1] && cudaEventRecord((cudaEvent_t)ev[1], stream) != cudaSuccess) return ATTN_ERR_CUDA;
    if (pl.split_units) {
        CombineParams c;
        c.H = (int)H; c.Sq = (int)Sq; c.nq = p.nq; c.nsplit = p.nsplit; c.n_full = p.n_full;
        c.split_units = (int)pl.split_units; c.round_mode = round_mode;
        c.ws_o = p.ws_o; c.ws_lse = p.ws_lse; c.o = p.o;
        c.o_sb = p.o_sb; c.o_ss = p.o_ss; c.o_sh = p.o_sh;
        c.lse = a.lse;
        // warps per row by split count, so that a warp has at most four splits in flight
        const int W = pl.splits <= 4 ? 1 : pl.splits <= 8 ? 2 : pl.splits <= 16 ? 4 : 8;
        const long long rows = pl.split_units * kUnitRows;
        const int warps_per_block = 8;
        const unsigned blocks = (unsigned)cdiv(rows, warps_per_block / W);
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof cfg);
        cfg.gridDim = dim3(blocks);
        cfg.blockDim = dim3(warps_per_block * 32);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t ce;
        if (d == 128)
            ce = W == 1 ? cudaLaunchKernelEx(&cfg, attn_combine_kernel<128, 1>, c)
               : W == 2 ? cudaLaunchKernelEx(&cfg, attn_combine_kernel<128, 2>, c)
               : W == 4 ? cudaLaunchKernelEx(&cfg, attn_combine_kernel<128, 4>, c)
                        : cudaLaunchKernelEx(&cfg, attn_combine_kernel<128, 8>, c);
        else
            ce = W == 1 ? cudaLaunchKernelEx(&cfg, attn_combine_kernel<64, 1>, c)
               : W == 2 ? cudaLaunchKernelEx(&cfg, attn_combine_kernel<64, 2>, c)
               : W == 4 ? cudaLaunchKernelEx(&cfg, attn_combine_kernel<64, 4>, c)
                        : cudaLaunchKernelEx(&cfg, attn_combine_kernel<64, 8>, c);
        if (ce != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
    }
    if (ev && ev[2] && cudaEventRecord((cudaEvent_t)ev[2], stream) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

// ------------------------------------------------------------------------------ static scratch
// Scratch for attn_fwd_noalloc(): the split path's partial outputs live in this array compiled
// into the library instead of in memory the library allocates.  Every GPU that loads the
// library holds it until the process exits.  Host code must not pass the symbol itself to a
// kernel (on the host it only names a stand-in); noalloc_scratch() looks up the device address.
constexpr size_t kStaticScratchBytes = (size_t)24 << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];
void* g_static_scratch_ptr[kMaxDevices];

// Device address of the static scratch on the current device (looked up once per device).
int noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return ATTN_ERR_NO_DEVICE;
    }
    std::lock_guard<std::mutex> g(g_mutex);
    if (!g_static_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        g_static_scratch_ptr[dev] = ptr;
    }
    *out = g_static_scratch_ptr[dev];
    return ATTN_OK;
}

// Library-owned workspace of the current device, grown on demand (guarded by g_mutex).
int library_workspace(DeviceInfo* di, size_t bytes, void** ws) {
    std::lock_guard<std::mutex> g(g_mutex);
    if (di->ws_bytes < bytes) {
        if (di->ws) cudaFree(di->ws);   // synchronizes the device: old users are done
        di->ws = nullptr;
        di->ws_bytes = 0;
        if (cudaMalloc(&di->ws, bytes) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        di->ws_bytes = bytes;
    }
    *ws = di->ws;
    return ATTN_OK;
}

// The launch path shared by every entry point.  ws_mode: 0 = caller workspace (must be large
// enough), 1 = caller workspace or, if null, the library-owned one, 2 = the static scratch.
int run(const attn_args_t& a, const attn_options_t* opts, void* workspace, size_t workspace_bytes, int ws_mode,
        cudaStream_t stream) {
    int st = validate(a, opts);
    if (st != ATTN_OK) return st;
    DeviceInfo* di = nullptr;
    if ((st = device_info(&di)) != ATTN_OK) return st;
    attn_plan_t pl;
    make_plan(a, di->sms, opts, &pl);
    void* ws = nullptr;
    if (pl.workspace_bytes) {
        const size_t need = (size_t)pl.workspace_bytes;
        if (ws_mode == 2) {
            if (need > kStaticScratchBytes) return ATTN_ERR_WORKSPACE;
            // every scratch byte the combine reads is written by the attention kernel of the
            // same call, so stale contents from an earlier call need no clearing
            if ((st = noalloc_scratch(&ws)) != ATTN_OK) return st;
        } else if (workspace) {
            if (workspace_bytes < need) return ATTN_ERR_WORKSPACE;
            if ((uintptr_t)workspace & 15u) return ATTN_ERR_MISALIGNED;
            ws = workspace;
        } else if (ws_mode == 1) {
            if ((st = library_workspace(di, need, &ws)) != ATTN_OK) return st;
        } else {
            return ATTN_ERR_WORKSPACE;
        }
    }
    return launch(a, pl, opts, ws, stream);
}

// ---------------------------------------------------------------- variable-length batches
// The arguments of attn_fwd_varlen and attn_fwd_paged in one form.  kv_rows: token rows of
// the K/V tensors (total_k, or num_pages * page_size for a paged cache).
struct SeqBatch {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;
    const int32_t* cu_q;
    const int32_t* cu_k;
    const int32_t* seqlens_k;
    const int32_t* block_table;
    int64_t B, H, Hkv, total_q, kv_rows, max_seqlen_q, d;
    int64_t paged, page_size, max_pages, num_pages;
    int32_t round_mode, causal, pack_heads, max_splits;
};

// log2 of the heads packed into one tile's rows (0: no packing)
int pack_shift(const SeqBatch& a) {
    int sh = 0;
    if (a.pack_heads)
        while ((int64_t(1) << sh) < a.H / a.Hkv) ++sh;
    return sh;
}

SeqBatch from_varlen(const attn_varlen_args_t& a) {
    SeqBatch c;
    memset(&c, 0, sizeof c);
    c.q = a.q; c.k = a.k; c.v = a.v; c.o = a.o; c.lse = a.lse;
    c.cu_q = a.cu_seqlens_q; c.cu_k = a.cu_seqlens_k;
    c.B = a.B; c.H = a.H; c.Hkv = a.Hkv; c.total_q = a.total_q; c.kv_rows = a.total_k;
    c.max_seqlen_q = a.max_seqlen_q; c.d = a.d;
    c.round_mode = a.round_mode; c.causal = a.causal; c.pack_heads = a.pack_heads; c.max_splits = a.max_splits;
    return c;
}

SeqBatch from_paged(const attn_paged_args_t& a) {
    SeqBatch c;
    memset(&c, 0, sizeof c);
    c.q = a.q; c.k = a.k_cache; c.v = a.v_cache; c.o = a.o; c.lse = a.lse;
    c.cu_q = a.cu_seqlens_q; c.seqlens_k = a.seqlens_k; c.block_table = a.block_table;
    c.B = a.B; c.H = a.H; c.Hkv = a.Hkv; c.total_q = a.total_q;
    c.kv_rows = a.num_pages * a.page_size;
    c.max_seqlen_q = a.max_seqlen_q; c.d = a.d;
    c.paged = 1; c.page_size = a.page_size; c.max_pages = a.max_pages; c.num_pages = a.num_pages;
    c.round_mode = a.round_mode; c.causal = a.causal; c.pack_heads = a.pack_heads; c.max_splits = a.max_splits;
    return c;
}

int validate_seq_shape(const SeqBatch& a, const attn_options_t* opts) {
    if (a.B < 1 || a.H < 1 || a.Hkv < 1 || a.total_q < 0 || a.kv_rows < 0 || a.max_seqlen_q < 0 || a.d < 1)
        return ATTN_ERR_INVALID_ARG;
    if (a.H % a.Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (a.round_mode < ATTN_ROUND_RTNE || a.round_mode > ATTN_ROUND_RTZ) return ATTN_ERR_INVALID_ARG;
    if ((a.causal != 0 && a.causal != 1) || (a.pack_heads != 0 && a.pack_heads != 1) || a.max_splits < 0)
        return ATTN_ERR_INVALID_ARG;
    // packed heads: a power of two of at most 32 per K/V head, so that a warp's 32 rows hold
    // whole tokens
    if (a.pack_heads) {
        const int64_t g = a.H / a.Hkv;
        if (g > 32 || (g & (g - 1)) != 0) return ATTN_ERR_UNSUPPORTED;
    }
    if (a.paged && (a.num_pages < 1 || a.max_pages < 1 || a.page_size < kBN || a.page_size % kBN != 0))
        return ATTN_ERR_INVALID_ARG;
    if (a.d != 128 && a.d != 64) return ATTN_ERR_UNSUPPORTED;
    if (opts && opts->force_splits > 1) return ATTN_ERR_UNSUPPORTED;
    if (opts && opts->test_hooks != 0) return ATTN_ERR_INVALID_ARG;
    // offsets are int32; token rows, item indices and TMA coordinates stay below 2^30
    const int64_t lim = (int64_t)1 << 30;
    if (a.total_q > lim || a.kv_rows > lim || a.B > lim || a.H > lim) return ATTN_ERR_UNSUPPORTED;
    if (a.paged && (a.num_pages > lim || a.page_size > lim || a.max_pages > lim ||
                    a.max_pages * a.page_size > lim || a.B * a.max_pages > lim))
        return ATTN_ERR_UNSUPPORTED;
    if (a.H * (a.total_q / kUnitRows + a.B) > lim) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

// work-list entries a batch can need: a block has 256 >> shift tokens, so there are at most
// sum_b ceil(Sq_b / tokens) <= total_q / tokens + B pairs, and with key splits at most two
// items per CTA (sms: the device's SMs, which bound the CTA count)
int64_t seq_max_blocks(const SeqBatch& a, int64_t sms) {
    const int64_t pairs = a.total_q / (kUnitRows >> pack_shift(a)) + a.B;
    return a.max_splits > 1 && 2 * sms > pairs ? 2 * sms : pairs;
}

bool seq_split(const SeqBatch& a) { return a.max_splits > 1; }

// workspace: per-sequence tensor maps (128-byte aligned inside it), the item count, the work
// list, and with key splits (256-byte aligned) the parts' fp32 rows and LSEs, two slots per CTA
size_t seq_list_bytes(const SeqBatch& a, int64_t sms) {
    return 128 + (size_t)a.B * 4 * sizeof(CUtensorMap) + 16 + (size_t)seq_max_blocks(a, sms) * sizeof(int4);
}
size_t seq_ws_bytes(const SeqBatch& a, int64_t sms) {
    size_t n = seq_list_bytes(a, sms);
    if (seq_split(a)) n = ((n + 255) & ~(size_t)255) + (size_t)2 * sms * kUnitRows * (size_t)(a.d + 1) * 4;
    return n;
}

// the SM count the workspace of a batch is sized for (0 if a split batch finds no device)
int64_t seq_sms(const SeqBatch& a) {
    if (!seq_split(a)) return 0;
    DeviceInfo* di = nullptr;
    return device_info(&di) == ATTN_OK ? di->sms : 0;
}
size_t seq_ws_query(const SeqBatch& a) {
    if (validate_seq_shape(a, nullptr) != ATTN_OK) return 0;
    const int64_t sms = seq_sms(a);
    if (seq_split(a) && sms < 1) return 0;
    return seq_ws_bytes(a, sms);
}

int run_seq_batch(const SeqBatch& a, const attn_options_t* opts, void* workspace, size_t workspace_bytes,
                  cudaStream_t stream) {
    int st = validate_seq_shape(a, opts);
    if (st != ATTN_OK) return st;
    if (!a.q || !a.k || !a.v || !a.o || !a.cu_q) return ATTN_ERR_INVALID_ARG;
    if (a.paged ? (!a.seqlens_k || !a.block_table) : !a.cu_k) return ATTN_ERR_INVALID_ARG;
    if (((uintptr_t)a.q | (uintptr_t)a.k | (uintptr_t)a.v | (uintptr_t)a.o) & 15u) return ATTN_ERR_MISALIGNED;
    if (((uintptr_t)a.lse | (uintptr_t)a.cu_q | (uintptr_t)a.cu_k | (uintptr_t)a.seqlens_k |
         (uintptr_t)a.block_table) & 3u)
        return ATTN_ERR_MISALIGNED;
    const uintptr_t qbytes = (uintptr_t)(a.total_q * a.H * a.d * 2), kvbytes = (uintptr_t)(a.kv_rows * a.Hkv * a.d * 2);
    auto overlap = [](uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; };
    const uintptr_t ob = (uintptr_t)a.o, oe = ob + qbytes, qb = (uintptr_t)a.q, qe = qb + qbytes;
    const uintptr_t kb = (uintptr_t)a.k, ke = kb + kvbytes, vb = (uintptr_t)a.v, ve = vb + kvbytes;
    if (overlap(ob, oe, qb, qe) || overlap(ob, oe, kb, ke) || overlap(ob, oe, vb, ve)) return ATTN_ERR_ALIAS;
    if (a.lse) {
        const uintptr_t lb = (uintptr_t)a.lse, le = lb + (uintptr_t)(a.H * a.total_q * 4);
        if (overlap(lb, le, ob, oe) || overlap(lb, le, qb, qe) || overlap(lb, le, kb, ke) || overlap(lb, le, vb, ve))
            return ATTN_ERR_ALIAS;
    }
    DeviceInfo* di = nullptr;
    if ((st = device_info(&di)) != ATTN_OK) return st;
    const bool split = seq_split(a);
    const int64_t sms = split ? di->sms : 0;
    const size_t need = seq_ws_bytes(a, sms);
    void* ws = nullptr;
    if (workspace) {
        if (workspace_bytes < need) return ATTN_ERR_WORKSPACE;
        if ((uintptr_t)workspace & 15u) return ATTN_ERR_MISALIGNED;
        ws = workspace;
    } else if ((st = library_workspace(di, need, &ws)) != ATTN_OK) {
        return st;
    }
    const uintptr_t wsb = (uintptr_t)ws;
    if (overlap(wsb, wsb + need, ob, oe) || (a.lse && overlap(wsb, wsb + need, (uintptr_t)a.lse,
                                                              (uintptr_t)a.lse + (uintptr_t)(a.H * a.total_q * 4))))
        return ATTN_ERR_ALIAS;
    const int64_t d = a.d;
    // whole-tensor maps (token-major, one batch), which the preprocessing kernel narrows to
    // each sequence (a paged cache's maps also serve its full pages as they are); a tensor
    // with no rows gets a one-row map that no item ever uses
    const int64_t tq = a.total_q > 0 ? a.total_q : 1, tk = a.kv_rows > 0 ? a.kv_rows : 1;
    // with head packing a Q box is 2^shift heads x (128 >> shift) tokens and an O box 2^shift
    // heads x (32 >> shift) tokens: the same 128 and 32 rows, ordered token-major
    const int sh = pack_shift(a);
    CUtensorMap qm, km, vm, om;
    if (!encode_map(&qm, a.q, 1, a.H, tq, d, true, (uint32_t)(kBM >> sh), 1u << sh) ||
        !encode_map(&km, a.k, 1, a.Hkv, tk, d, true) || !encode_map(&vm, a.v, 1, a.Hkv, tk, d, true) ||
        !encode_map(&om, a.o, 1, a.H, tq, d, true, (uint32_t)(kStageRowsPerWarp >> sh), 1u << sh))
        return ATTN_ERR_CUDA;
    CUtensorMap* maps = reinterpret_cast<CUtensorMap*>((wsb + 127u) & ~(uintptr_t)127u);
    int* n_items = reinterpret_cast<int*>(maps + 4 * a.B);
    int4* blocks = reinterpret_cast<int4*>(reinterpret_cast<char*>(n_items) + 16);
    float* ws_o = nullptr;
    float* ws_lse = nullptr;
    if (split) {
        ws_o = reinterpret_cast<float*>((wsb + seq_list_bytes(a, sms) + 255u) & ~(uintptr_t)255u);
        ws_lse = ws_o + (size_t)2 * sms * kUnitRows * d;
    }
    VarlenPrep vp;
    memset(&vp, 0, sizeof vp);
    vp.cu_q = a.cu_q;
    vp.cu_k = a.cu_k;
    vp.seqlens_k = a.seqlens_k;
    vp.block_table = a.block_table;
    vp.paged = (int)a.paged;
    vp.page_size = (int)a.page_size;
    vp.max_pages = (int)a.max_pages;
    vp.num_pages = (int)a.num_pages;
    vp.pack_shift = sh;
    vp.max_splits = a.max_splits;
    vp.B = (int)a.B;
    vp.H = (int)a.H;
    vp.causal = a.causal;
    vp.total_q = a.total_q;
    vp.total_k = a.kv_rows;
    vp.q_row_bytes = a.H * d * 2;
    vp.kv_row_bytes = a.Hkv * d * 2;
    vp.q = reinterpret_cast<const char*>(a.q);
    vp.k = reinterpret_cast<const char*>(a.k);
    vp.v = reinterpret_cast<const char*>(a.v);
    vp.o = reinterpret_cast<char*>(a.o);
    vp.lse = a.lse;
    vp.maps = maps;
    vp.blocks = blocks;
    vp.n_items = n_items;

    FwdParams p;
    memset(&p, 0, sizeof p);
    p.B = (int)a.B;
    p.H = (int)a.H;
    p.group = (int)(a.H / a.Hkv);
    p.causal = a.causal;
    p.nsplit = 1;
    p.bshd = 1;
    p.round_mode = a.round_mode;
    p.scale_log2 = (float)((1.0 / std::sqrt((double)d)) * 1.4426950408889634);
    p.tau = 8.0f;
    p.o = reinterpret_cast<__nv_bfloat16*>(a.o);
    p.lse = a.lse;
    const uint32_t ms = (opts && opts->wait_limit_ms) ? opts->wait_limit_ms : 2000u;
    p.wait_limit_ns = (unsigned long long)ms * 1000000ull;
    p.vl_maps = maps;
    p.vl_blocks = blocks;
    p.vl_n_items = n_items;
    p.cu_q = a.cu_q;
    p.cu_k = a.cu_k;
    p.total_q = a.total_q;
    p.paged = (int)a.paged;
    p.seqlens_k = a.seqlens_k;
    p.block_table = a.block_table;
    p.page_size = (int)a.page_size;
    p.max_pages = (int)a.max_pages;
    p.pack_shift = sh;
    p.ws_o = ws_o;
    p.ws_lse = ws_lse;

    // CTAs: one per SM, at most max_ctas, and no more than the items can use (max_seqlen_q
    // bounds the pairs; key splits multiply them by up to max_splits)
    int64_t G = di->sms;
    if (opts && opts->max_ctas > 0 && opts->max_ctas < G) G = opts->max_ctas;
    if (a.max_seqlen_q > 0) {
        int64_t cap = a.B * (a.H >> sh) * cdiv(a.max_seqlen_q, kUnitRows >> sh);
        if (split) cap = cap > G ? G : cap * a.max_splits;
        if (cap < G) G = cap;
    }
    if (G < 1) G = 1;
    vp.grid = (int)G;

    // preprocessing -> attention kernel, each a programmatic dependent of the kernel before it
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t lc;
    memset(&lc, 0, sizeof lc);
    lc.gridDim = dim3(1);
    lc.blockDim = dim3(1024);
    lc.stream = stream;
    lc.attrs = pdl;
    lc.numAttrs = 1;
    if (cudaLaunchKernelEx(&lc, attn_varlen_prep_kernel, qm, km, vm, om, vp) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    const attn_event_t* ev = opts ? opts->events : nullptr;
    if (ev && ev[0] && cudaEventRecord((cudaEvent_t)ev[0], stream) != cudaSuccess) return ATTN_ERR_CUDA;
    lc.gridDim = dim3((unsigned)G);
    lc.blockDim = dim3(kThreads);
    cudaError_t le;
    if (d == 128) {
        lc.dynamicSmemBytes = Geo<128>::kSmemAlloc;
        le = a.causal ? cudaLaunchKernelEx(&lc, attn_fwd_kernel<128, true, true>, qm, km, vm, om, p)
                      : cudaLaunchKernelEx(&lc, attn_fwd_kernel<128, false, true>, qm, km, vm, om, p);
    } else {
        lc.dynamicSmemBytes = Geo<64>::kSmemAlloc;
        le = a.causal ? cudaLaunchKernelEx(&lc, attn_fwd_kernel<64, true, true>, qm, km, vm, om, p)
                      : cudaLaunchKernelEx(&lc, attn_fwd_kernel<64, false, true>, qm, km, vm, om, p);
    }
    if (le != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    if (ev && ev[1] && cudaEventRecord((cudaEvent_t)ev[1], stream) != cudaSuccess) return ATTN_ERR_CUDA;
    if (split) {
        // merge of the key parts (every block whose item is not a first part returns at once)
        VarlenCombine vc;
        vc.blocks = blocks;
        vc.n_items = n_items;
        vc.cu_q = a.cu_q;
        vc.ws_o = ws_o;
        vc.ws_lse = ws_lse;
        vc.o = reinterpret_cast<__nv_bfloat16*>(a.o);
        vc.lse = a.lse;
        vc.total_q = a.total_q;
        vc.H = (int)a.H;
        vc.pack_shift = sh;
        vc.round_mode = a.round_mode;
        lc.gridDim = dim3((unsigned)G, kUnitRows / 32);   // items < 2 G, two a block; 32 tile rows a block, 4 a warp
        lc.blockDim = dim3(256);
        lc.dynamicSmemBytes = 0;
        le = d == 128 ? cudaLaunchKernelEx(&lc, attn_varlen_combine_kernel<128>, vc)
                      : cudaLaunchKernelEx(&lc, attn_varlen_combine_kernel<64>, vc);
        if (le != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
    }
    if (ev && ev[2] && cudaEventRecord((cudaEvent_t)ev[2], stream) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

size_t workspace_for(const attn_args_t& a, const attn_options_t* opts) {
    if (validate_shape(a, opts) != ATTN_OK) return 0;
    DeviceInfo* di = nullptr;
    if (device_info(&di) != ATTN_OK) return 0;
    attn_plan_t pl;
    make_plan(a, di->sms, opts, &pl);
    return (size_t)pl.workspace_bytes;
}

}  // namespace

extern "C" {

int attn_plan_ex(const attn_args_t* args, int64_t num_sms, const attn_options_t* opts, attn_plan_t* plan) {
    if (!args || !plan || num_sms < 1) return ATTN_ERR_INVALID_ARG;
    const int st = validate_shape(*args, opts);
    if (st != ATTN_OK) return st;
    make_plan(*args, num_sms, opts, plan);
    return ATTN_OK;
}

int attn_plan(int64_t B, int64_t H, int64_t Sq, int64_t Skv, int64_t d, int64_t num_sms,
              const attn_options_t* opts, attn_plan_t* plan) {
    const attn_args_t a = plain_args(nullptr, nullptr, nullptr, nullptr, B, H, Sq, Skv, d, 0, 0);
    return attn_plan_ex(&a, num_sms, opts, plan);
}

size_t attn_fwd_ex_workspace_size(const attn_args_t* args, const attn_options_t* opts) {
    return args ? workspace_for(*args, opts) : 0;
}

size_t attn_fwd_workspace_size_opts(int64_t B, int64_t H, int64_t Sq, int64_t Skv, int64_t d,
                                    const attn_options_t* opts) {
    const attn_args_t a = plain_args(nullptr, nullptr, nullptr, nullptr, B, H, Sq, Skv, d, 0, 0);
    return workspace_for(a, opts);
}

size_t attn_fwd_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t Skv, int64_t d) {
    return attn_fwd_workspace_size_opts(B, H, Sq, Skv, d, nullptr);
}

size_t attn_fwd_varlen_workspace_size(const attn_varlen_args_t* args) {
    if (!args) return 0;
    const SeqBatch c = from_varlen(*args);
    return seq_ws_query(c);
}

int attn_fwd_varlen(const attn_varlen_args_t* args, const attn_options_t* opts, void* workspace,
                    size_t workspace_bytes, attn_stream_t stream) {
    if (!args) return ATTN_ERR_INVALID_ARG;
    return run_seq_batch(from_varlen(*args), opts, workspace, workspace_bytes, (cudaStream_t)stream);
}

size_t attn_fwd_paged_workspace_size(const attn_paged_args_t* args) {
    if (!args) return 0;
    const SeqBatch c = from_paged(*args);
    return seq_ws_query(c);
}

int attn_fwd_paged(const attn_paged_args_t* args, const attn_options_t* opts, void* workspace,
                   size_t workspace_bytes, attn_stream_t stream) {
    if (!args) return ATTN_ERR_INVALID_ARG;
    return run_seq_batch(from_paged(*args), opts, workspace, workspace_bytes, (cudaStream_t)stream);
}

int attn_fwd_ex(const attn_args_t* args, const attn_options_t* opts, void* workspace, size_t workspace_bytes,
                attn_stream_t stream) {
    if (!args) return ATTN_ERR_INVALID_ARG;
    return run(*args, opts, workspace, workspace_bytes, 1, (cudaStream_t)stream);
}

int attn_fwd_ws(const void* q, const void* k, const void* v, void* o, int64_t B, int64_t H, int64_t Sq,
                int64_t Skv, int64_t d, int layout, int round_mode, const attn_options_t* opts, void* workspace,
                size_t workspace_bytes, attn_stream_t stream) {
    const attn_args_t a = plain_args(q, k, v, o, B, H, Sq, Skv, d, layout, round_mode);
    return run(a, opts, workspace, workspace_bytes, 0, (cudaStream_t)stream);
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, int64_t B, int64_t H, int64_t Sq, int64_t Skv,
             int64_t d, int layout, int round_mode, attn_stream_t stream) {
    const attn_args_t a = plain_args(q, k, v, o, B, H, Sq, Skv, d, layout, round_mode);
    return run(a, nullptr, nullptr, 0, 1, (cudaStream_t)stream);
}

int attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, int64_t B, int64_t H, int64_t Sq,
                     int64_t Skv, int64_t d, int layout, int round_mode, attn_stream_t stream) {
    const attn_args_t a = plain_args(q, k, v, o, B, H, Sq, Skv, d, layout, round_mode);
    return run(a, nullptr, nullptr, 0, 2, (cudaStream_t)stream);
}

int attn_get_device_status(attn_stream_t stream, int32_t* site) {
    if (site) *site = 0;
    uint32_t h[2] = {0u, 0u};
    const uint32_t zero[2] = {0u, 0u};
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess ||
        cudaMemcpyFromSymbol(h, g_status, sizeof h) != cudaSuccess ||
        cudaMemcpyToSymbol(g_status, zero, sizeof zero) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    if (site) *site = (int32_t)h[1];
    return (int)h[0];
}

const char* attn_status_string(int status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "unsupported shape (d must be 64 or 128; sizes within int32 indexing)";
        case ATTN_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case ATTN_ERR_ALIAS: return "output overlaps an input";
        case ATTN_ERR_NO_DEVICE: return "no sm_103 CUDA device current";
        case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
        case ATTN_ERR_CUDA: return "CUDA runtime error";
        case ATTN_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel expired";
        default: return "unknown status";
    }
}

int attn_version(void) { return 300; }

}  // extern "C"
