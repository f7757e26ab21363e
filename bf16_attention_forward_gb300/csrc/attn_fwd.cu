// attn_fwd.cu -- bf16 attention forward for GB300 (sm_103a): kernels and the C ABI.
//
// O = softmax(Q K^T / sqrt(128)) V, non-causal, BSHD or BHSD, any Sq/Skv, output rounded
// RTNE/RTNA/RTZ.  Source page: "MoonMath AI open-sources a HIP attention kernel for AMD
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
//   * warp 8 streams Q and a K,V,K,V,... ring (4 x 32 KB stages) with TMA + mbarriers;
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
//     each split writes fp32 O/l and a base-2 log-sum-exp, and a combine kernel merges them.
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

constexpr int kD = 128;            // head dimension
constexpr int kBM = 128;           // query rows per tile (one TMEM lane per row)
constexpr int kBN = 128;           // keys per KV tile
constexpr int kQTiles = 2;         // query tiles per work unit
constexpr int kUnitRows = kBM * kQTiles;
constexpr int kStages = 4;         // K/V ring depth
constexpr int kTileBytes = kBM * kD * 2;       // 32 KB: 128 rows x 128 bf16
constexpr int kChunkBytes = kTileBytes / 2;    // 16 KB: 128 rows x 64 bf16 (one TMA box)
constexpr int kThreads = 384;      // WG0, WG1 softmax; warp 8 TMA; warp 9 MMA; 10-11 spare
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
constexpr int kMinTilesPerSplit = 4;
constexpr uint32_t kTmemCols = 512;   // S0 | S1 | O0 | O1, 128 fp32 columns each

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int kSmemQ = 0;
constexpr int kSmemRing = kSmemQ + kQTiles * kTileBytes;
constexpr int kSmemBars = kSmemRing + kStages * kTileBytes;
constexpr int kNumBars = 2 * kStages + 2 + 3 * kQTiles + 1;
constexpr int kSmemMisc = kSmemBars + kNumBars * 8;
constexpr int kSmemUsed = kSmemMisc + 16;
constexpr int kSmemAlloc = kSmemUsed + 1024;

// barrier indices
constexpr int kBarFull = 0;                 // [kStages] ring slot loaded
constexpr int kBarEmpty = kStages;          // [kStages] ring slot released by the MMAs
constexpr int kBarQFull = 2 * kStages;
constexpr int kBarQEmpty = kBarQFull + 1;
constexpr int kBarSFull = kBarQEmpty + 1;   // [2] S_i ready in TMEM
constexpr int kBarPFull = kBarSFull + 2;    // [2] P_i written (and O_i rescaled)
constexpr int kBarOFull = kBarPFull + 2;    // [2] last PV of the unit done
constexpr int kBarDrain = kBarOFull + 2;

// wait sites reported through the status word
enum : uint32_t {
    kSiteQEmpty = 1, kSiteRingEmpty, kSiteQFull, kSiteRingFull, kSitePFull, kSiteSFull,
    kSiteOFull, kSiteDrain, kSiteTeardown
};

__device__ uint32_t g_status[2];   // [0] status code, [1] wait site

struct FwdParams {
    int B, H, Sq, Skv;
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
    unsigned long long wait_limit_ns;
};

struct Item {
    int b, h, qb, kv_begin, kv_end, split_slot;
};

__device__ __forceinline__ Item decode_item(const FwdParams& p, int k) {
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
    it.qb = unit % p.nq;
    const int bh = unit / p.nq;
    it.h = bh % p.H;
    it.b = bh / p.H;
    return it;
}

// Bounded mbarrier wait.  On expiry it records the site in the status word, raises the
// CTA's abort flag and returns false; every other wait then gives up at once.
__device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity, uint32_t site,
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

// softmax weight exponent for logit s: x = s*c - m*c, kept >= -125 when s is finite so that
// a finite logit always has a positive bf16 weight; -inf stays -inf (weight exactly 0) and
// NaN stays NaN.  The fma with 2^-40 moves finite x by < 1e-9 relative.
__device__ __forceinline__ float weight_exponent(float s, float c, float neg_mc) {
    const float x = fmaf(s, c, neg_mc);
    return fmaf(x, 0x1p-40f, ptx::fmax_nan(x, -125.0f));
}

__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap vmap, const FwdParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bars = sbase + kSmemBars;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint32_t* tmem_holder = (uint32_t*)(smem + kSmemMisc);
    volatile uint32_t* abort_flag = (volatile uint32_t*)(smem + kSmemMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(bar(kBarFull + s), 1);
            ptx::mbar_init(bar(kBarEmpty + s), 1);
        }
        ptx::mbar_init(bar(kBarQFull), 1);
        ptx::mbar_init(bar(kBarQEmpty), 1);
        for (int i = 0; i < kQTiles; ++i) {
            ptx::mbar_init(bar(kBarSFull + i), 1);
            ptx::mbar_init(bar(kBarPFull + i), kBM);
            ptx::mbar_init(bar(kBarOFull + i), 1);
        }
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

    if (warp == kWarpTma) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_kv = ptx::policy_evict_last();
            const uint64_t pol_q = ptx::policy_evict_first();
            uint32_t pos = 0;             // ring position (monotonic)
            int last_pos[kStages];
            for (int s = 0; s < kStages; ++s) last_pos[s] = -1;
            int u = 0;
            bool ok = true;
            for (int k = blockIdx.x; k < p.n_items && ok; k += gridDim.x, ++u) {
                const Item it = decode_item(p, k);
                if (u > 0 && !(ok = wait_bar(bar(kBarQEmpty), (u - 1) & 1, kSiteQEmpty, abort_flag, lim)))
                    break;
                ptx::mbar_arrive_expect_tx(bar(kBarQFull), kQTiles * kTileBytes);
                for (int t = 0; t < kQTiles; ++t) {
                    const int row = it.qb * kUnitRows + t * kBM;
                    for (int c = 0; c < 2; ++c) {
                        const uint32_t dst = sbase + kSmemQ + (t * 2 + c) * kChunkBytes;
                        if (p.bshd)
                            ptx::tma_load_4d(dst, &qmap, bar(kBarQFull), c * 64, it.h, row, it.b, pol_q);
                        else
                            ptx::tma_load_4d(dst, &qmap, bar(kBarQFull), c * 64, row, it.h, it.b, pol_q);
                    }
                }
                for (int j = it.kv_begin; j < it.kv_end && ok; ++j) {
                    for (int kv = 0; kv < 2; ++kv, ++pos) {
                        const uint32_t slot = pos % kStages;
                        const uint32_t ph = (pos / kStages) & 1u;
                        if (!(ok = wait_bar(bar(kBarEmpty + slot), ph ^ 1u, kSiteRingEmpty, abort_flag, lim)))
                            break;
                        ptx::mbar_arrive_expect_tx(bar(kBarFull + slot), kTileBytes);
                        const void* map = kv ? (const void*)&vmap : (const void*)&kmap;
                        for (int c = 0; c < 2; ++c) {
                            const uint32_t dst = sbase + kSmemRing + slot * kTileBytes + c * kChunkBytes;
                            if (p.bshd)
                                ptx::tma_load_4d(dst, map, bar(kBarFull + slot), c * 64, it.h, j * kBN, it.b, pol_kv);
                            else
                                ptx::tma_load_4d(dst, map, bar(kBarFull + slot), c * 64, j * kBN, it.h, it.b, pol_kv);
                        }
                        last_pos[slot] = (int)pos;
                    }
                }
            }
            // every load issued has landed before the CTA may exit
            for (int s = 0; s < kStages; ++s)
                if (last_pos[s] >= 0) {
                    const uint32_t ph = ((uint32_t)last_pos[s] / kStages) & 1u;
                    const uint64_t t0 = ptx::globaltimer_ns();
                    while (!ptx::mbar_try_wait(bar(kBarFull + s), ph) &&
                           ptx::globaltimer_ns() - t0 < lim) {
                    }
                }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16(kBM, kBN, false, false);
            constexpr uint32_t idesc_o = idesc_bf16(kBM, kD, false, true);
            const uint32_t tS[2] = {tmem + 0u, tmem + 128u};
            const uint32_t tO[2] = {tmem + 256u, tmem + 384u};
            // Q_i / K_j: K-major, 128 B rows, 8-row swizzle atoms 1024 B apart; the k-th
            // 16-element step sits 32 B further inside the atom, the second 64-column half
            // 16 KB further.  V_j: MN-major (d contiguous), the two 64-column halves 16 KB
            // apart (leading offset), 8-key groups 1024 B apart (stride offset); the k-th
            // 16-key step is 2 KB further.
            auto qdesc = [&](int t, int kk) {
                return sdesc(sbase + kSmemQ + (t * 2 + (kk >> 2)) * kChunkBytes + (kk & 3) * 32, 16, 1024);
            };
            auto kdesc = [&](uint32_t slot, int kk) {
                return sdesc(sbase + kSmemRing + slot * kTileBytes + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024);
            };
            auto vdesc = [&](uint32_t slot, int kk) {
                return sdesc(sbase + kSmemRing + slot * kTileBytes + kk * 2048, kChunkBytes, 1024);
            };
            uint32_t pos = 0;
            uint32_t pcount[2] = {0u, 0u};
            int u = 0;
            bool ok = true;
            for (int k = blockIdx.x; k < p.n_items && ok; k += gridDim.x, ++u) {
                const Item it = decode_item(p, k);
                const int nk = it.kv_end - it.kv_begin;
                if (!(ok = wait_bar(bar(kBarQFull), u & 1, kSiteQFull, abort_flag, lim))) break;
                uint32_t kslot = pos % kStages;
                if (!(ok = wait_bar(bar(kBarFull + kslot), (pos / kStages) & 1u, kSiteRingFull, abort_flag, lim)))
                    break;
                ptx::tc_fence_after();
                for (int t = 0; t < kQTiles; ++t) {
                    for (int kk = 0; kk < kD / 16; ++kk)
                        ptx::mma_ss(tS[t], qdesc(t, kk), kdesc(kslot, kk), idesc_s, kk > 0);
                    ptx::mma_commit(bar(kBarSFull + t));
                }
                ptx::mma_commit(bar(kBarEmpty + kslot));
                if (nk == 1) ptx::mma_commit(bar(kBarQEmpty));
                ++pos;
                for (int jj = 0; jj < nk && ok; ++jj) {
                    const uint32_t vpos = pos;
                    const uint32_t vslot = vpos % kStages;
                    const bool more = jj + 1 < nk;
                    if (!(ok = wait_bar(bar(kBarFull + vslot), (vpos / kStages) & 1u, kSiteRingFull, abort_flag, lim)))
                        break;
                    const uint32_t kpos = vpos + 1;
                    kslot = kpos % kStages;
                    for (int t = 0; t < kQTiles; ++t) {
                        if (!(ok = wait_bar(bar(kBarPFull + t), pcount[t] & 1u, kSitePFull, abort_flag, lim)))
                            break;
                        ++pcount[t];
                        ptx::tc_fence_after();
                        for (int kk = 0; kk < kBN / 16; ++kk)
                            ptx::mma_ts(tO[t], tS[t] + (uint32_t)kk * 8u, vdesc(vslot, kk), idesc_o,
                                        (jj > 0 || kk > 0) ? 1u : 0u);
                        if (!more) ptx::mma_commit(bar(kBarOFull + t));
                        if (t == kQTiles - 1) ptx::mma_commit(bar(kBarEmpty + vslot));
                        if (more) {
                            if (t == 0) {
                                if (!(ok = wait_bar(bar(kBarFull + kslot), (kpos / kStages) & 1u, kSiteRingFull,
                                                    abort_flag, lim)))
                                    break;
                                ptx::tc_fence_after();
                            }
                            for (int kk = 0; kk < kD / 16; ++kk)
                                ptx::mma_ss(tS[t], qdesc(t, kk), kdesc(kslot, kk), idesc_s, kk > 0);
                            ptx::mma_commit(bar(kBarSFull + t));
                            if (t == kQTiles - 1) {
                                ptx::mma_commit(bar(kBarEmpty + kslot));
                                if (jj + 2 == nk) ptx::mma_commit(bar(kBarQEmpty));
                            }
                        }
                    }
                    pos += more ? 2 : 1;
                }
            }
            // drain: every MMA this thread issued has finished before TMEM is released
            ptx::mma_commit(bar(kBarDrain));
            const uint64_t t0 = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(bar(kBarDrain), 0) && ptx::globaltimer_ns() - t0 < lim) {
            }
        }
    } else if (warp < 2 * 4) {
        // ------------------------------------------------------------------ softmax + epilogue
        const int t = warp >> 2;                    // query tile owned by this warpgroup
        const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
        const int row = quarter * 32 + lane;        // row within the tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + (uint32_t)(t * 128);
        const uint32_t tO = tmem + lane_off + 256u + (uint32_t)(t * 128);
        const float c = p.scale_log2;
        uint32_t scount = 0;
        int u = 0;
        bool ok = true;
        for (int k = blockIdx.x; k < p.n_items && ok; k += gridDim.x, ++u) {
            const Item it = decode_item(p, k);
            float m_ref = -INFINITY;      // running max of raw logits at the last rescale
            float l = 0.0f;               // running sum of weights relative to m_ref
            for (int j = it.kv_begin; j < it.kv_end; ++j) {
                ok = wait_bar(bar(kBarSFull + t), scount & 1u, kSiteSFull, abort_flag, lim);
                if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                ++scount;
                ptx::tc_fence_after();
                uint32_t s[4][32];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) ptx::tmem_ld32(tS + ch * 32, s[ch]);
                const int valid = p.Skv - j * kBN;   // keys of this tile that exist
                if (valid < kBN) {
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch)
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (ch * 32 + e >= valid) s[ch][e] = __float_as_uint(-INFINITY);
                }
                // row max as 8 independent chains, then a tree
                float mp[8];
#pragma unroll
                for (int q8 = 0; q8 < 8; ++q8) mp[q8] = __uint_as_float(s[0][q8]);
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
#pragma unroll
                    for (int e = (ch == 0 ? 8 : 0); e < 32; ++e) mp[e & 7] = fmaxf(mp[e & 7], __uint_as_float(s[ch][e]));
                const float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                                       fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
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
                const float neg_mc = (m_ref == -INFINITY) ? 0.0f : -m_ref * c;
                float lp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // independent partial sums
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float p0 = ptx::ex2_approx(weight_exponent(__uint_as_float(s[ch][2 * e]), c, neg_mc));
                        const float p1 = ptx::ex2_approx(weight_exponent(__uint_as_float(s[ch][2 * e + 1]), c, neg_mc));
                        lp[(2 * e) & 7] += p0;
                        lp[(2 * e + 1) & 7] += p1;
                        pk[e] = ptx::pack_bf16x2(p0, p1);
                    }
                    ptx::tmem_st16(tS + ch * 16, pk);
                }
                l += ((lp[0] + lp[1]) + (lp[2] + lp[3])) + ((lp[4] + lp[5]) + (lp[6] + lp[7]));
                if (__any_sync(0xFFFFFFFFu, rescale_o)) {
                    const float a = rescale_o ? alpha : 1.0f;
#pragma unroll 1
                    for (int ch = 0; ch < 4; ++ch) {
                        uint32_t o[32];
                        ptx::tmem_ld32(tO + ch * 32, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
                        ptx::tmem_st32(tO + ch * 32, o);
                    }
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(kBarPFull + t));
            }
            if (!ok) break;
            // epilogue: O / l, rounding, store
            ok = wait_bar(bar(kBarOFull + t), u & 1, kSiteOFull, abort_flag, lim);
            if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
            ptx::tc_fence_after();
            const int qrow = it.qb * kUnitRows + t * kBM + row;
            const bool valid_row = qrow < p.Sq;
            if (it.split_slot < 0) {
                const float inv = 1.0f / l;
                __nv_bfloat16* orow = p.o + (long long)it.b * p.o_sb + (long long)qrow * p.o_ss +
                                      (long long)it.h * p.o_sh;
#pragma unroll 1
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t o[32];
                    ptx::tmem_ld32(tO + ch * 32, o);
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const uint32_t lo = round_bf16_bits(__uint_as_float(o[2 * e]) * inv, p.round_mode);
                        const uint32_t hi = round_bf16_bits(__uint_as_float(o[2 * e + 1]) * inv, p.round_mode);
                        w[e] = lo | (hi << 16);
                    }
                    if (valid_row) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            dst[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
                    }
                }
            } else {
                // split partial: O/l in fp32 (the raw sum when l == 0) and LSE in log2 units
                const float inv = (l > 0.0f) ? 1.0f / l : 1.0f;
                const long long wrow = (long long)it.split_slot * kUnitRows + t * kBM + row;
                float* dst = p.ws_o + wrow * kD;
#pragma unroll 1
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t o[32];
                    ptx::tmem_ld32(tO + ch * 32, o);
                    if (valid_row) {
                        float4* d4 = reinterpret_cast<float4*>(dst + ch * 32);
#pragma unroll
                        for (int v4 = 0; v4 < 8; ++v4)
                            d4[v4] = make_float4(__uint_as_float(o[4 * v4]) * inv, __uint_as_float(o[4 * v4 + 1]) * inv,
                                                 __uint_as_float(o[4 * v4 + 2]) * inv, __uint_as_float(o[4 * v4 + 3]) * inv);
                    }
                }
                if (valid_row) p.ws_lse[wrow] = m_ref * c + log2f(l);
            }
        }
    }

    // ---------------------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------------------ combine
struct CombineParams {
    int H, Sq, nq, nsplit, n_full, split_units, round_mode;
    const float* ws_o;
    const float* ws_lse;
    __nv_bfloat16* o;
    long long o_sb, o_ss, o_sh;
};

// One warp per output row of a split unit: merge the nsplit partials in fixed order s = 0..n-1
// with weights 2^(LSE_s - max LSE).  [MoonMath] "Data placement ..." (tail KV split).
__global__ void __launch_bounds__(256) attn_combine_kernel(const CombineParams p) {
    const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= (long long)p.split_units * kUnitRows) return;
    const int t = (int)(gw / kUnitRows);
    const int r = (int)(gw % kUnitRows);
    const int unit = p.n_full + t;
    const int qb = unit % p.nq, bh = unit / p.nq;
    const int h = bh % p.H, b = bh / p.H;
    const int qrow = qb * kUnitRows + r;
    if (qrow >= p.Sq) return;
    const long long base = (long long)t * p.nsplit * kUnitRows + r;
    float mx = -INFINITY;
    bool any_nan = false;
    for (int s = 0; s < p.nsplit; ++s) {
        const float e = p.ws_lse[base + (long long)s * kUnitRows];
        any_nan |= (e != e);
        mx = fmaxf(mx, e);
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float wsum = 0.f;
    for (int s = 0; s < p.nsplit; ++s) {
        const float e = p.ws_lse[base + (long long)s * kUnitRows];
        float w;
        if (e == -INFINITY) w = 0.0f;
        else w = ptx::ex2_approx(fmaxf(e - mx, -125.0f));
        wsum += w;
        const float4 v = *reinterpret_cast<const float4*>(p.ws_o + (base + (long long)s * kUnitRows) * kD + lane * 4);
        acc[0] += w * v.x;
        acc[1] += w * v.y;
        acc[2] += w * v.z;
        acc[3] += w * v.w;
    }
    const bool nan_row = any_nan || mx == -INFINITY;
    const float inv = 1.0f / wsum;
    uint32_t bits[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) bits[e] = nan_row ? 0x7FC0u : round_bf16_bits(acc[e] * inv, p.round_mode);
    __nv_bfloat16* orow = p.o + (long long)b * p.o_sb + (long long)qrow * p.o_ss + (long long)h * p.o_sh;
    *reinterpret_cast<uint2*>(orow + lane * 4) = make_uint2(bits[0] | (bits[1] << 16), bits[2] | (bits[3] << 16));
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

int validate(const void* q, const void* k, const void* v, const void* o, int64_t B, int64_t H,
             int64_t Sq, int64_t Skv, int64_t d, int layout, int round_mode) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || Sq < 1 || Skv < 1 || d < 1) return ATTN_ERR_INVALID_ARG;
    if (layout != ATTN_LAYOUT_BSHD && layout != ATTN_LAYOUT_BHSD) return ATTN_ERR_INVALID_ARG;
    if (round_mode < ATTN_ROUND_RTNE || round_mode > ATTN_ROUND_RTZ) return ATTN_ERR_INVALID_ARG;
    if (d != kD) return ATTN_ERR_UNSUPPORTED;
    // TMA coordinates and the kernels' unit/row indices are int32
    const int64_t lim = (int64_t)1 << 30;
    if (Sq > lim || Skv > lim || B > lim || H > lim) return ATTN_ERR_UNSUPPORTED;
    if (B * H > lim || B * H * cdiv(Sq, kUnitRows) > lim) return ATTN_ERR_UNSUPPORTED;
    if (((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)o) & 15u) return ATTN_ERR_MISALIGNED;
    const uintptr_t ob = (uintptr_t)o, oe = ob + (uintptr_t)(B * H * Sq * d * 2);
    const uintptr_t qb = (uintptr_t)q, qe = qb + (uintptr_t)(B * H * Sq * d * 2);
    const uintptr_t kb = (uintptr_t)k, ke = kb + (uintptr_t)(B * H * Skv * d * 2);
    const uintptr_t vb = (uintptr_t)v, ve = vb + (uintptr_t)(B * H * Skv * d * 2);
    auto overlap = [](uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; };
    if (overlap(ob, oe, qb, qe) || overlap(ob, oe, kb, ke) || overlap(ob, oe, vb, ve)) return ATTN_ERR_ALIAS;
    return ATTN_OK;
}

void make_plan(int64_t B, int64_t H, int64_t Sq, int64_t Skv, int64_t sms, const attn_options_t* opts,
               attn_plan_t* pl) {
    const int64_t nq = cdiv(Sq, kUnitRows);
    const int64_t U = B * H * nq;
    const int64_t nkv = cdiv(Skv, kBN);
    int64_t G = sms;
    if (opts && opts->max_ctas > 0 && opts->max_ctas < G) G = opts->max_ctas;
    if (G < 1) G = 1;
    int64_t full = U, split_units = 0, ns = 1;
    if (opts && opts->force_splits > 0) {
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
    pl->workspace_bytes = split_units ? split_units * pl->splits * kUnitRows * (kD * 4 + 4) : 0;
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
        if (cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc) !=
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
bool encode_map(CUtensorMap* m, const void* ptr, int64_t B, int64_t H, int64_t S, bool bshd) {
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
    dims[0] = kD;
    if (bshd) {
        dims[1] = H; dims[2] = S; dims[3] = B;
        strides[0] = kD * 2; strides[1] = H * kD * 2; strides[2] = S * H * kD * 2;
        box[0] = 64; box[1] = 1; box[2] = kBM; box[3] = 1;
    } else {
        dims[1] = S; dims[2] = H; dims[3] = B;
        strides[0] = kD * 2; strides[1] = S * kD * 2; strides[2] = H * S * kD * 2;
        box[0] = 64; box[1] = kBM; box[2] = 1; box[3] = 1;
    }
    const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int launch(const void* q, const void* k, const void* v, void* o, int64_t B, int64_t H, int64_t Sq, int64_t Skv,
           int layout, int round_mode, const attn_plan_t& pl, const attn_options_t* opts, void* ws,
           cudaStream_t stream) {
    const bool bshd = layout == ATTN_LAYOUT_BSHD;
    CUtensorMap qm, km, vm;
    if (!encode_map(&qm, q, B, H, Sq, bshd) || !encode_map(&km, k, B, H, Skv, bshd) ||
        !encode_map(&vm, v, B, H, Skv, bshd))
        return ATTN_ERR_CUDA;
    FwdParams p;
    memset(&p, 0, sizeof p);
    p.B = (int)B; p.H = (int)H; p.Sq = (int)Sq; p.Skv = (int)Skv;
    p.nq = (int)cdiv(Sq, kUnitRows);
    p.nkv = (int)pl.kv_tiles;
    p.n_items = (int)pl.items;
    p.n_full = (int)pl.full_items;
    p.nsplit = (int)pl.splits;
    p.bshd = bshd ? 1 : 0;
    p.round_mode = round_mode;
    p.scale_log2 = (float)((1.0 / std::sqrt((double)kD)) * 1.4426950408889634);
    p.tau = 8.0f;
    p.o = reinterpret_cast<__nv_bfloat16*>(o);
    if (pl.split_units) {
        p.ws_o = reinterpret_cast<float*>(ws);
        p.ws_lse = p.ws_o + pl.split_units * pl.splits * kUnitRows * kD;
    }
    if (bshd) { p.o_sb = Sq * H * kD; p.o_ss = H * kD; p.o_sh = kD; }
    else { p.o_sb = H * Sq * kD; p.o_ss = kD; p.o_sh = Sq * kD; }
    const uint32_t ms = (opts && opts->wait_limit_ms) ? opts->wait_limit_ms : 2000u;
    p.wait_limit_ns = (unsigned long long)ms * 1000000ull;

    attn_fwd_kernel<<<(unsigned)pl.grid, kThreads, kSmemAlloc, stream>>>(qm, km, vm, p);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    if (pl.split_units) {
        CombineParams c;
        c.H = (int)H; c.Sq = (int)Sq; c.nq = p.nq; c.nsplit = p.nsplit; c.n_full = p.n_full;
        c.split_units = (int)pl.split_units; c.round_mode = round_mode;
        c.ws_o = p.ws_o; c.ws_lse = p.ws_lse; c.o = p.o;
        c.o_sb = p.o_sb; c.o_ss = p.o_ss; c.o_sh = p.o_sh;
        const long long rows = pl.split_units * kUnitRows;
        const int warps_per_block = 8;
        const unsigned blocks = (unsigned)cdiv(rows, warps_per_block);
        attn_combine_kernel<<<blocks, warps_per_block * 32, 0, stream>>>(c);
        if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_plan(int64_t B, int64_t H, int64_t Sq, int64_t Skv, int64_t d, int64_t num_sms,
              const attn_options_t* opts, attn_plan_t* plan) {
    if (!plan || B < 1 || H < 1 || Sq < 1 || Skv < 1 || num_sms < 1) return ATTN_ERR_INVALID_ARG;
    if (d != kD) return ATTN_ERR_UNSUPPORTED;
    make_plan(B, H, Sq, Skv, num_sms, opts, plan);
    return ATTN_OK;
}

size_t attn_fwd_workspace_size_opts(int64_t B, int64_t H, int64_t Sq, int64_t Skv, int64_t d,
                                    const attn_options_t* opts) {
    if (B < 1 || H < 1 || Sq < 1 || Skv < 1 || d != kD) return 0;
    DeviceInfo* di = nullptr;
    if (device_info(&di) != ATTN_OK) return 0;
    attn_plan_t pl;
    make_plan(B, H, Sq, Skv, di->sms, opts, &pl);
    return (size_t)pl.workspace_bytes;
}

size_t attn_fwd_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t Skv, int64_t d) {
    return attn_fwd_workspace_size_opts(B, H, Sq, Skv, d, nullptr);
}

int attn_fwd_ws(const void* q, const void* k, const void* v, void* o, int64_t B, int64_t H, int64_t Sq,
                int64_t Skv, int64_t d, int layout, int round_mode, const attn_options_t* opts, void* workspace,
                size_t workspace_bytes, attn_stream_t stream) {
    int st = validate(q, k, v, o, B, H, Sq, Skv, d, layout, round_mode);
    if (st != ATTN_OK) return st;
    DeviceInfo* di = nullptr;
    if ((st = device_info(&di)) != ATTN_OK) return st;
    attn_plan_t pl;
    make_plan(B, H, Sq, Skv, di->sms, opts, &pl);
    if (pl.workspace_bytes) {
        if (!workspace || workspace_bytes < (size_t)pl.workspace_bytes) return ATTN_ERR_WORKSPACE;
        if ((uintptr_t)workspace & 15u) return ATTN_ERR_MISALIGNED;
    }
    return launch(q, k, v, o, B, H, Sq, Skv, layout, round_mode, pl, opts, workspace, (cudaStream_t)stream);
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, int64_t B, int64_t H, int64_t Sq, int64_t Skv,
             int64_t d, int layout, int round_mode, attn_stream_t stream) {
    int st = validate(q, k, v, o, B, H, Sq, Skv, d, layout, round_mode);
    if (st != ATTN_OK) return st;
    DeviceInfo* di = nullptr;
    if ((st = device_info(&di)) != ATTN_OK) return st;
    attn_plan_t pl;
    make_plan(B, H, Sq, Skv, di->sms, nullptr, &pl);
    void* ws = nullptr;
    if (pl.workspace_bytes) {
        std::lock_guard<std::mutex> g(g_mutex);
        if (di->ws_bytes < (size_t)pl.workspace_bytes) {
            if (di->ws) cudaFree(di->ws);   // synchronizes the device: old users are done
            di->ws = nullptr;
            di->ws_bytes = 0;
            if (cudaMalloc(&di->ws, (size_t)pl.workspace_bytes) != cudaSuccess) {
                cudaGetLastError();
                return ATTN_ERR_CUDA;
            }
            di->ws_bytes = (size_t)pl.workspace_bytes;
        }
        ws = di->ws;
    }
    return launch(q, k, v, o, B, H, Sq, Skv, layout, round_mode, pl, nullptr, ws, (cudaStream_t)stream);
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
        case ATTN_ERR_UNSUPPORTED: return "unsupported shape (d must be 128; sizes within int32 indexing)";
        case ATTN_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case ATTN_ERR_ALIAS: return "output overlaps an input";
        case ATTN_ERR_NO_DEVICE: return "no sm_103 CUDA device current";
        case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
        case ATTN_ERR_CUDA: return "CUDA runtime error";
        case ATTN_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel expired";
        default: return "unknown status";
    }
}

int attn_version(void) { return 100; }

}  // extern "C"
