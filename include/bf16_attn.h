/*
 * bf16_attn.h -- C ABI of the GB300 (sm_103a) bf16 attention forward library.
 *
 * Operation.  O = softmax(Q K^T / sqrt(d)) V, non-causal, head dimension d = 128 (64 is
 * accepted too), bf16 in and out, fp32 accumulation.  Extensions below: the causal mask,
 * grouped K/V heads and the row log-sum-exp (attn_fwd_ex), variable-length batches
 * (attn_fwd_varlen), a paged K/V cache (attn_fwd_paged) and the backward (attn_bwd).  Source: "MoonMath AI open-sources a HIP attention kernel for
 * AMD MI300X that beats AITER" (news.chathome.org), opening section: attention is the fused
 * softmax(QK^T/sqrt(d))V; the kernel takes BSHD or BHSD tensors without transposes, head
 * dimension fixed at 128, any query and key length including cross-attention; its
 * limitations paragraph: three output rounding modes (RTNE, RTNA, RTZ), NaN/Inf handled
 * bit-identically, deterministic results; section "Real use cases": a simple API that
 * launches on the caller's stream.  The long-KV split and its log-sum-exp combine follow the
 * section "Data placement and the 16x16x16 choice" (Flash-Decoding-style tail KV split).
 * Head dimension 64 is the second tile configuration of "HipKittens: Fast and Furious AMD
 * Kernels (MLSys 2026)", "Experiments and results" (attention forward at d = 64 and 128).
 *
 * Layouts.  All four tensors share one layout and are dense (contiguous):
 *   ATTN_LAYOUT_BSHD: element (b, s, h, x) at ((b*S + s)*H + h)*d + x
 *   ATTN_LAYOUT_BHSD: element (b, s, h, x) at ((b*H + h)*S + s)*d + x
 * with S = Sq for Q and O and S = Skv for K and V.  The scale is fixed at 1/sqrt(d).
 *
 * Numerics.  The output rounding mode applies to the final fp32 -> bf16 store only
 * (softmax weights are rounded to bf16, nearest-even, before the P.V product in every mode).
 * A row whose logits hold a NaN or +inf, or are all -inf, is NaN; every NaN is stored as
 * 0x7FC0; +-inf outputs keep their sign.  Results are bitwise reproducible for a given shape
 * on a given GPU model (the work split is a pure function of shape and SM count).
 *
 * Ownership.  The caller owns q, k, v, o and any workspace; the library never frees them.
 * All calls are asynchronous on `stream` and return before the GPU runs.  Each kernel is
 * launched as a programmatic dependent of the kernel before it on `stream`: it may start its
 * prologue while that kernel finishes, but waits for that kernel's memory before it reads or
 * writes global memory, so calls are ordered exactly as plain stream launches.  attn_fwd() keeps
 * one lazily grown workspace per device (guarded by a mutex): it may call cudaMalloc the
 * first time a shape needs the split path, so call it once before any CUDA-graph capture,
 * or use attn_fwd_ws() with caller memory.  attn_fwd_ex, attn_fwd_varlen and attn_fwd_paged
 * use the same library-owned workspace when given none (the last two always need one); calls
 * that share it and may run at the same time on the GPU (unordered streams) must be
 * serialized by the caller, or given workspaces of their own.
 *
 * Errors.  Argument problems are reported synchronously before anything is launched.  A
 * launch failure returns ATTN_ERR_CUDA.  Every wait inside the kernels is bounded: if one
 * expires the kernel records ATTN_ERR_DEVICE_TIMEOUT in a per-device status word and
 * returns (it never traps or spins forever); read it with attn_get_device_status().
 */
#ifndef BF16_ATTN_H_
#define BF16_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the same handle type, declared here without the CUDA headers). */
typedef struct CUstream_st* attn_stream_t;

typedef enum { ATTN_LAYOUT_BSHD = 0, ATTN_LAYOUT_BHSD = 1 } attn_layout_t;

/* Output rounding of the final fp32 value: IEEE roundTiesToEven, roundTiesToAway,
 * roundTowardZero. */
typedef enum { ATTN_ROUND_RTNE = 0, ATTN_ROUND_RTNA = 1, ATTN_ROUND_RTZ = 2 } attn_round_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,    /* null pointer, a size < 1, a bad enum value; also read
                                    back from the device for bad variable-length offsets,
                                    lengths or page indices                               */
    ATTN_ERR_UNSUPPORTED = 2,    /* d not 64 or 128, or a size beyond the kernels' int32 indexing */
    ATTN_ERR_MISALIGNED = 3,     /* a tensor or workspace base not 16-byte aligned         */
    ATTN_ERR_ALIAS = 4,          /* o overlaps q, k or v                                   */
    ATTN_ERR_NO_DEVICE = 5,      /* no CUDA device, or the current device is not sm_103    */
    ATTN_ERR_WORKSPACE = 6,      /* workspace null or smaller than attn_fwd_workspace_size */
    ATTN_ERR_CUDA = 7,           /* a CUDA runtime call failed                             */
    ATTN_ERR_DEVICE_TIMEOUT = 8  /* a bounded wait inside a kernel expired                 */
} attn_status_t;

/* A cudaEvent_t (the same handle type). */
typedef struct CUevent_st* attn_event_t;

/* Optional knobs (all zero / NULL = defaults). */
typedef struct {
    int32_t force_splits;   /* 0: planner decides. n >= 1: split every unit's keys n ways  */
    int32_t max_ctas;       /* 0: one persistent CTA per SM. n >= 1: at most n CTAs         */
    uint32_t wait_limit_ms; /* 0: 2000 ms. Bound on any single wait inside the kernels      */
    /* 0 for normal use.  ATTN_TEST_WITHHOLD_O_READY makes the first CTA skip the signal that
     * its first unit's output accumulator is complete, so that the epilogue's bounded wait
     * expires: the call then reports ATTN_ERR_DEVICE_TIMEOUT at site ATTN_SITE_O_READY
     * through attn_get_device_status(), with its output partly unwritten, and the device
     * stays usable.  It exists to test that path; any other value is ATTN_ERR_INVALID_ARG. */
    uint32_t test_hooks;
    /* Events recorded on `stream` (NULL entries skipped): [0] before the attention kernel,
     * [1] after it, [2] after the split-combine kernel (or right after [1] if none runs).
     * They let a caller time the two kernels separately on the launching stream. */
    attn_event_t events[3];
} attn_options_t;

/* attn_options_t.test_hooks / attn_bwd_args_t.test_hooks value, and the wait site the
 * expired wait reports (the forward's O-ready wait; the backward's dK/dV-ready wait). */
#define ATTN_TEST_WITHHOLD_O_READY 1
#define ATTN_SITE_O_READY 7
#define ATTN_BWD_SITE_DKV_READY 9
/* Site reported with ATTN_ERR_INVALID_ARG when attn_fwd_varlen's offsets, or attn_fwd_paged's
 * offsets, lengths or page indices, are inconsistent. */
#define ATTN_SITE_SEQLENS 13

/* The work split chosen for a shape (host only, launches nothing). */
typedef struct {
    int64_t units;          /* B*H*ceil(Sq/256): one unit = two 128-row query tiles         */
    int64_t kv_tiles;       /* ceil(Skv/128)                                                */
    int64_t full_items;     /* units run whole                                              */
    int64_t split_units;    /* units whose keys are split                                   */
    int64_t splits;         /* ways each split unit is divided                              */
    int64_t items;          /* full_items + split_units*splits                              */
    int64_t grid;           /* persistent CTAs launched                                     */
    int64_t workspace_bytes;/* scratch the split path needs (0 when nothing is split)       */
} attn_plan_t;

/*
 * Full argument set of the attention forward, for attn_fwd_ex().  Beyond attn_fwd it adds the
 * two features the MoonMath article's limitations paragraph lists as missing from its MI300X
 * kernel -- causal masking and grouped K/V heads (GQA; MQA when Hkv = 1) -- and the row
 * log-sum-exp, the intermediate that "AMD zverejnilo postup pre custom diffusion attention
 * kernel vo FlyDSL na ROCm" (section "Debug, profiling and integration") checks against a
 * baseline and that a backward pass needs.
 *   q            bf16, [B, Sq, H, d] (BSHD) or [B, H, Sq, d] (BHSD)
 *   k, v         bf16, same layout with Skv rows and Hkv heads; query head h reads K/V head
 *                h / (H / Hkv); Hkv must divide H
 *   o            bf16, like q; must not overlap q, k, v or lse
 *   lse          optional fp32 output, [B][H][Sq] (row (b, h, i) at (b*H + h)*Sq + i): natural
 *                log of sum_j exp(s_j) over the visible keys, s_j = q_i.k_j / sqrt(d); NaN for a
 *                row whose visible logits hold a NaN or +inf, -inf when every visible logit is
 *                -inf or no key is visible.  NULL: not written.  4-byte aligned.
 *   causal       0: every key visible.  1: key j visible to query i iff j <= i + (Skv - Sq)
 *                (aligned at the last query and key; plain causal when Sq = Skv).  Masked keys
 *                take no part in the row; a query with no visible key gets NaN outputs.  Known
 *                deviation: a masked key inside the 128-key tile that holds the row's diagonal
 *                still meets the P.V product with weight 0, so a +-inf or NaN in its V row turns
 *                that output column NaN (0 * inf).
 *   reserved     must be 0.
 */
typedef struct {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;
    int64_t B, H, Hkv, Sq, Skv, d;
    int32_t layout, round_mode, causal, reserved;
} attn_args_t;

/*
 * attn_fwd -- O = softmax(Q K^T / sqrt(d)) V on `stream`.
 *   q           device pointer, bf16, [B, Sq, H, d] (BSHD) or [B, H, Sq, d] (BHSD)
 *   k, v        device pointers, bf16, same layout with Skv rows
 *   o           device pointer, bf16, same shape as q; must not overlap q, k or v
 *   B, H        batch and heads (>= 1);  Sq, Skv  query and key lengths (>= 1);  d = 128 or 64
 *   layout      attn_layout_t;  round_mode  attn_round_t
 *   stream      cudaStream_t (NULL = legacy default stream)
 * Uses the library-owned workspace when the planner splits keys (see Ownership above).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, int64_t B, int64_t H,
             int64_t Sq, int64_t Skv, int64_t d, int layout, int round_mode,
             attn_stream_t stream);

/* Bytes of workspace attn_fwd_ws() needs for this shape with default options (0 if none). */
size_t attn_fwd_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t Skv, int64_t d);

/*
 * attn_fwd_ws -- attn_fwd with caller-owned workspace (device memory, 16-byte aligned,
 * at least attn_fwd_workspace_size() bytes for these options; may be NULL when that is 0)
 * and optional knobs (opts may be NULL).  Allocates nothing.
 */
int attn_fwd_ws(const void* q, const void* k, const void* v, void* o, int64_t B, int64_t H,
                int64_t Sq, int64_t Skv, int64_t d, int layout, int round_mode,
                const attn_options_t* opts, void* workspace, size_t workspace_bytes,
                attn_stream_t stream);

/* Workspace bytes for a shape under the given options (opts may be NULL). */
size_t attn_fwd_workspace_size_opts(int64_t B, int64_t H, int64_t Sq, int64_t Skv, int64_t d,
                                    const attn_options_t* opts);

/*
 * attn_plan -- the work split for a shape on a GPU with `num_sms` SMs (host only).  Returns
 * ATTN_OK and fills *plan, or an argument error.  The same function drives the launches.
 */
int attn_plan(int64_t B, int64_t H, int64_t Sq, int64_t Skv, int64_t d, int64_t num_sms,
              const attn_options_t* opts, attn_plan_t* plan);

/*
 * attn_fwd_ex -- the attention forward with every option (attn_args_t) on `stream`.
 * workspace: caller device memory of at least attn_fwd_ex_workspace_size() bytes, 16-byte
 * aligned; or NULL to use the library-owned workspace (which may be grown with cudaMalloc, as
 * in attn_fwd).  The causal planner never splits keys (no workspace); opts->force_splits > 1
 * with causal = 1 is ATTN_ERR_UNSUPPORTED.  Errors as for attn_fwd.
 */
int attn_fwd_ex(const attn_args_t* args, const attn_options_t* opts, void* workspace,
                size_t workspace_bytes, attn_stream_t stream);

/* Workspace bytes attn_fwd_ex needs for these arguments and options (0 if none or invalid). */
size_t attn_fwd_ex_workspace_size(const attn_args_t* args, const attn_options_t* opts);

/* attn_plan for the full argument set (host only; pointers in args are not read). */
int attn_plan_ex(const attn_args_t* args, int64_t num_sms, const attn_options_t* opts,
                 attn_plan_t* plan);

/*
 * attn_fwd_noalloc -- attn_fwd for callers that cannot allocate device memory.  (The paper
 * has no counterpart; this entry point exists for integration.)  Some callers must not see a
 * library call cudaMalloc: code recording a CUDA graph (an allocation there breaks the
 * capture), programs that hand all device memory to their own allocator or run under a fixed
 * memory budget, and host frameworks that forbid libraries from allocating on their behalf.
 * This call allocates nothing and frees nothing.  When the planner splits keys, the partial
 * results go to a scratch array of ATTN_NOALLOC_SCRATCH_BYTES (24 MiB) compiled into the
 * library; every GPU that loads the library holds that array until the process exits.
 *   Arguments, layouts, numerics and errors are those of attn_fwd, plus:
 *   - a shape whose split needs more scratch than the array holds returns ATTN_ERR_WORKSPACE
 *     (with the default planner that needs more than 190 SMs' worth of split work);
 *   - the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture;
 *   - all calls share the one array: each call writes every scratch byte it reads, so nothing
 *     carries over, but calls that can run at the same time on the GPU (unordered streams)
 *     race on it and must be serialized by the caller.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES ((size_t)24 << 20)
int attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, int64_t B, int64_t H,
                     int64_t Sq, int64_t Skv, int64_t d, int layout, int round_mode,
                     attn_stream_t stream);

/*
 * Variable-length batches -- the third feature the MoonMath article's limitations paragraph
 * lists as missing from its kernel.  B sequences of different lengths are packed along one
 * token axis (token-major, like BSHD without the batch axis); sequence b owns query rows
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key rows cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1
 * and attends only to its own keys: row i of sequence b is attention over that sequence's
 * keys, exactly as attn_fwd_ex on the sequence alone.
 *   q             bf16 [total_q][H][d];  k, v  bf16 [total_k][Hkv][d];  o  bf16 like q
 *   lse           optional fp32 [H][total_q] (row (h, i) at h*total_q + i), as in attn_fwd_ex
 *   cu_seqlens_q, cu_seqlens_k   device int32 [B + 1]: start >= 0, never decrease, end <=
 *                 total_q (total_k).  Checked on the device: a violation writes no output and
 *                 reports ATTN_ERR_INVALID_ARG at site ATTN_SITE_SEQLENS through
 *                 attn_get_device_status().  A sequence may be empty; one with queries but no
 *                 keys gets NaN outputs and -inf LSE (no key is visible).  Query rows outside
 *                 every sequence are not written.
 *   B             sequences (>= 1);  H, Hkv, d  as in attn_fwd_ex;  total_q, total_k >= 0
 *   max_seqlen_q  an upper bound on any sequence's query length, used only to size the grid
 *                 (0: unknown, one CTA per SM)
 *   causal        per sequence, aligned at its last query and key (attn_fwd_ex's rule)
 *   pack_heads    0 or 1.  1: the H / Hkv query heads that read one K/V head (a power of two,
 *                 at most 32; otherwise ATTN_ERR_UNSUPPORTED) share the rows of one 128-row
 *                 tile, 128 / (H / Hkv) tokens of each, so short query chunks (decoding, a
 *                 few speculative tokens) fill the tiles and each K/V tile is read once for
 *                 the group.  Every row is computed exactly as without packing: the results
 *                 are bit for bit the same.  Pays off when sequences have few queries
 *                 (for decoding a dense batch, pass cu_seqlens = 0, Sq, 2 Sq, ... here).
 *   max_splits    >= 0.  0 or 1: a query block's keys are never split.  n >= 2: when the
 *                 batch's (sequence, query block, head) items number fewer than the CTAs (a
 *                 few long sequences, decoding), the preprocessing kernel splits each block's
 *                 key tiles into up to n contiguous parts, more for costlier blocks, so that
 *                 the CTAs finish together: in one wave (every part a CTA of its own) or, when
 *                 the items already fill half the CTAs and a model of the work favours it, in
 *                 two (the MoonMath article's key split of the tail, on the variable-length
 *                 work list); a third kernel merges the parts.  The choice depends on the lengths and the CTA count
 *                 only, so results are deterministic for a given device and max_ctas; they
 *                 differ from the unsplit ones by rounding (same criteria against the exact
 *                 result).  Batches with at least as many items as CTAs run unsplit.
 * opts->force_splits must be 0 or 1.  workspace: caller device memory of at least
 * attn_fwd_varlen_workspace_size() bytes (per-sequence tensor maps and the work list; with
 * max_splits >= 2 also two fp32 partial tiles per SM of the current device), 16-byte aligned;
 * or NULL to use the library-owned workspace as attn_fwd_ex does.  The size query returns 0
 * for invalid arguments, and for max_splits >= 2 when no CUDA device is usable.  Kernels on
 * `stream`: a one-CTA preprocessing kernel, the attention kernel, and with max_splits >= 2
 * the merge of the parts.
 */
typedef struct {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;
    const int32_t* cu_seqlens_q;
    const int32_t* cu_seqlens_k;
    int64_t B, H, Hkv, total_q, total_k, max_seqlen_q, d;
    int32_t round_mode, causal, pack_heads, max_splits;
} attn_varlen_args_t;

size_t attn_fwd_varlen_workspace_size(const attn_varlen_args_t* args);
int attn_fwd_varlen(const attn_varlen_args_t* args, const attn_options_t* opts, void* workspace,
                    size_t workspace_bytes, attn_stream_t stream);

/*
 * Paged K/V -- "AMD zverejnilo postup pre custom diffusion attention kernel vo FlyDSL na ROCm",
 * section "Co AMD konkretne popisuje": attention kernels need flexible KV-cache layouts, a
 * paged cache among them.  Queries are packed as in attn_fwd_varlen; the keys and values of
 * sequence b are the first seqlens_k[b] token slots of its pages: key j sits in slot
 * j % page_size of physical page block_table[b * max_pages + j / page_size].  Row i of
 * sequence b is attention over those keys, exactly as attn_fwd_varlen on the gathered keys
 * (causal: aligned at the sequence's last query and key, so a chunk of new queries sees the
 * whole cache before it).
 *   q, o, lse     as in attn_fwd_varlen (packed [total_q][H][d]; lse [H][total_q])
 *   k_cache, v_cache  bf16 [num_pages][page_size][Hkv][d]
 *   cu_seqlens_q  device int32 [B + 1], as in attn_fwd_varlen
 *   seqlens_k     device int32 [B]: keys per sequence, 0 .. max_pages * page_size
 *   block_table   device int32 [B][max_pages]; entries past a sequence's last used page are
 *                 not read.  Pages may be shared between sequences.
 *   page_size     a multiple of 128 (a key tile never straddles pages)
 *   pack_heads    as in attn_fwd_varlen (the natural setting for decoding over a paged cache)
 *   max_splits    as in attn_fwd_varlen (decoding a few long sequences)
 * Checked on the device: bad query offsets, lengths or page indices (outside 0 ..
 * num_pages - 1) write no output and report ATTN_ERR_INVALID_ARG at ATTN_SITE_SEQLENS.  Slots
 * of a sequence's last page past its length are never read as keys (they read as zeros), so
 * stale values there cannot reach the output.  Workspace as attn_fwd_varlen.
 */
typedef struct {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    void* o;
    float* lse;
    const int32_t* cu_seqlens_q;
    const int32_t* seqlens_k;
    const int32_t* block_table;
    int64_t B, H, Hkv, total_q, num_pages, page_size, max_pages, max_seqlen_q, d;
    int32_t round_mode, causal, pack_heads, max_splits;
} attn_paged_args_t;

size_t attn_fwd_paged_workspace_size(const attn_paged_args_t* args);
int attn_fwd_paged(const attn_paged_args_t* args, const attn_options_t* opts, void* workspace,
                   size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_get_device_status -- synchronizes `stream`, then reads and clears the current
 * device's status word.  Returns ATTN_OK, ATTN_ERR_DEVICE_TIMEOUT (a bounded wait expired),
 * ATTN_ERR_INVALID_ARG (attn_fwd_varlen's offsets), or ATTN_ERR_CUDA.  If site != NULL it
 * receives the id of the wait or check that failed (0 if none).
 */
int attn_get_device_status(attn_stream_t stream, int32_t* site);

/* Static string for a status code. */
const char* attn_status_string(int status);

/* Library version, as major*10000 + minor*100 + patch. */
int attn_version(void);

/*
 * Attention backward (d = 128 or 64): the gradients of O = softmax(Q K^T / sqrt(d)) V with respect
 * to Q, K and V, with the causal mask and grouped K/V heads as in attn_fwd_ex.  Source:
 * "HipKittens: Fast and Furious AMD Kernels (MLSys 2026)", "Key observations" (observation 3)
 * and "Attention backward" -- the backward is the kernel after the forward.  With
 * c = 1/sqrt(d), P recomputed from the forward's row log-sum-exp, and the upstream gradient dO:
 *   dV = P^T dO,  dS = P * (dO V^T - D) with D_i = dO_i . O_i,  dQ = c dS K,  dK = c dS^T Q.
 *   q, k, v, o   the forward's inputs and output (bf16, one layout, as in attn_fwd_ex)
 *   dout         dO, bf16, like o
 *   lse          the forward's fp32 [B][H][Sq] natural-log log-sum-exp (attn_fwd_ex's lse)
 *   dq, dk, dv   outputs, bf16, like q, k, v (round to nearest even); must not overlap the
 *                inputs, each other or the workspace.  dk and dv are bitwise reproducible;
 *                with deterministic = 0 the last bits of dq can differ between runs (its
 *                fp32 accumulator takes one addition per key tile, in no fixed order)
 *   causal       0 or 1, as in the forward
 *   deterministic  0 or 1.  1: dq is bitwise reproducible too.  Each key tile's dQ terms go
 *                to an fp32 slice of their own in the workspace and a final pass adds a row's
 *                slices in key-tile order, so the workspace holds ceil(Skv/128) dQ-sized fp32
 *                slices instead of one accumulator, and the call moves that much more memory
 *   reserved     0
 *   wait_limit_ms  0: 2000 ms; otherwise the bound, in ms, on any single wait in the kernel
 *   test_hooks   0 for normal use; ATTN_TEST_WITHHOLD_O_READY makes the first CTA skip the
 *                signal that its first unit's dK/dV accumulators are complete, so that the
 *                writer's bounded wait expires and attn_bwd_get_device_status() reports
 *                ATTN_ERR_DEVICE_TIMEOUT at site ATTN_BWD_SITE_DKV_READY (the outputs are then
 *                partly unwritten; the device stays usable).  It exists to test that path.
 * Rows of K/V that no query sees, and queries that see no key (causal, Sq > Skv; their
 * forward output is NaN), get zero gradients.  Inputs are expected finite.
 */
typedef struct {
    const void* q;
    const void* k;
    const void* v;
    const void* o;
    const void* dout;
    const float* lse;
    void* dq;
    void* dk;
    void* dv;
    int64_t B, H, Hkv, Sq, Skv, d;
    int32_t layout, causal, wait_limit_ms, test_hooks;
    int32_t deterministic, reserved;
} attn_bwd_args_t;

/* Workspace bytes attn_bwd needs (0 if invalid): the fp32 dQ accumulator (deterministic: one
 * fp32 dQ slice per 128-key tile) and per-row statistics, plus fp32 dK/dV partials when the last, partial round of work units is split by
 * query range.  That split depends on the current device's SM count; attn_bwd given a
 * workspace sized without the partials runs unsplit (same results up to rounding). */
size_t attn_bwd_workspace_size(const attn_bwd_args_t* args);

/*
 * attn_bwd -- the backward on `stream`: zeroes the dQ accumulator, forms D and the base-2
 * LSE, runs the tcgen05 backward kernel and rounds dQ.  workspace: caller device memory of
 * at least attn_bwd_workspace_size() bytes, 16-byte aligned (required).  Errors as for
 * attn_fwd; device-side wait expiries are read with attn_bwd_get_device_status().
 */
int attn_bwd(const attn_bwd_args_t* args, void* workspace, size_t workspace_bytes,
             attn_stream_t stream);

/* Synchronize `stream`, then read and clear the backward kernel's device status word. */
int attn_bwd_get_device_status(attn_stream_t stream, int32_t* site);

/*
 * Variable-length backward: the gradients of attn_fwd_varlen (sequences packed along the token
 * axis, each attending to its own keys, causal per sequence, grouped heads).
 *   q, o, dout, dq   bf16 [total_q][H][d];  k, v, dk, dv  bf16 [total_k][Hkv][d]
 *   lse              fp32 [H][total_q], attn_fwd_varlen's
 *   cu_seqlens_q, cu_seqlens_k   device int32 [B + 1], as in attn_fwd_varlen.  Checked on the
 *                    device: a violation writes no gradient and reports ATTN_ERR_INVALID_ARG
 *                    at site ATTN_BWD_SITE_SEQLENS through attn_bwd_get_device_status().
 *   causal, wait_limit_ms  as in attn_bwd;  reserved, reserved2  0
 * Rows outside every sequence are not written.  Queries of a sequence without keys get zero
 * dq, keys of a sequence without queries zero dk and dv.  dk, dv are bitwise reproducible; dq's
 * last bits may vary between runs (fp32 reductions in no fixed order).  Four kernels run on
 * `stream`: a one-CTA planning kernel (offsets, per-sequence tensor maps, the work units),
 * the row statistics with the dq accumulator's zeroing, the tcgen05 backward kernel, and the
 * dq rounding.  workspace: caller device memory of attn_bwd_varlen_workspace_size() bytes,
 * 16-byte aligned.
 */
#define ATTN_BWD_SITE_SEQLENS 16
typedef struct {
    const void* q;
    const void* k;
    const void* v;
    const void* o;
    const void* dout;
    const float* lse;
    void* dq;
    void* dk;
    void* dv;
    const int32_t* cu_seqlens_q;
    const int32_t* cu_seqlens_k;
    int64_t B, H, Hkv, total_q, total_k, d;
    int32_t causal, wait_limit_ms, reserved, reserved2;
} attn_bwd_varlen_args_t;

size_t attn_bwd_varlen_workspace_size(const attn_bwd_varlen_args_t* args);
int attn_bwd_varlen(const attn_bwd_varlen_args_t* args, void* workspace, size_t workspace_bytes,
                    attn_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* BF16_ATTN_H_ */
