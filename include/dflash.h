/*
 * dflash.h -- paged draft-block attention for block speculative decoding
 * (DFlash / DSpark drafters), GB300 (sm_103a).
 *
 * One call computes, for every request of a batch, the attention of the K
 * draft-block query tokens of every query head over the request's paged
 * context keys plus the K block keys, and returns the bf16 output and the
 * fp32 base-2 log-sum-exp.  The operation is the one the TensorRT-LLM pages
 * describe:
 *   - non-causal unwindowed block (PR #20374 "Non-causal unwindowed DFlash
 *     draft block", description): every block query sees the whole context
 *     and the whole block;
 *   - non-causal windowed block (PR #21130 "Non-causal windowed DSpark draft
 *     block", description "Why" and change 2): query i at position L+i sees
 *     the context keys of the causal window (L+i-W, L+i] plus every block key;
 *     the block keys after i are folded in by a base-2 log-sum-exp merge,
 *     which is skipped exactly when no later key exists (K = 1, or the causal
 *     form);
 *   - the causal block (future_keys = 0): the causal (windowed) decode alone,
 *     or with a right window r (right_window = r): the causal window plus the
 *     next r block keys, which generalises both forms (r = K-1 is the
 *     non-causal block); a window W < K bounds the block keys as well.
 * The softmax statistics are returned as base-2 LSE (PR #21130 change 1) and
 * the caller sizes a workspace that includes the partial softmax statistics
 * (PR #21130 change 3); sequence lengths stay on the device so one captured
 * CUDA graph serves every step (PR #20374, description: a graph is captured
 * for a fixed batch; PR #16150, the commit that takes the drafter's context
 * from the target's paged pool: the lengths live on the device).
 *
 * Ownership: the caller owns every buffer it passes.  The library allocates
 * no device or host memory at run time and keeps no state beyond cached
 * device attributes and the per-kernel shared-memory opt-in, with one
 * exception: dflash_block_attn_static_ws uses a scratch array of
 * DFLASH_STATIC_SCRATCH_BYTES that the library itself holds on every device
 * that loads it, and caches that array's device address per context.  The
 * library is thread-safe and issues only stream-ordered work (no host
 * synchronisation) in dflash_block_attn.
 *
 * Errors are host-side return codes; nothing is launched when a code other
 * than DFLASH_OK is returned by validation.  Bad data found on the device (a
 * page id outside the pool, a context length outside [0, max_ctx_len]) never
 * traps: the kernels substitute zeros or clamp, record a flag in the
 * workspace status word and finish.
 */
#ifndef DFLASH_H_
#define DFLASH_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define DFLASH_OK                    0
#define DFLASH_ERR_INVALID          -1  /* bad sizes, null or misaligned pointer */
#define DFLASH_ERR_WORKSPACE        -2  /* workspace smaller than dflash_workspace_size */
#define DFLASH_ERR_DEVICE           -3  /* current device is not compute capability 10.3 */
#define DFLASH_ERR_LAUNCH           -4  /* a CUDA call or kernel launch failed */

/* Device status flags (OR-ed into the workspace status word by the kernels). */
#define DFLASH_STATUS_BAD_PAGE       1  /* a visible position's page id is outside [0, num_pages) */
#define DFLASH_STATUS_BAD_CTX_LEN    2  /* ctx_lens[b] < 0 or > max_ctx_len (clamped) */
#define DFLASH_STATUS_TIMEOUT        4  /* a pipeline wait ran out (never expected) */
#define DFLASH_STATUS_FP8_RANGE      8  /* fp8 context: a block row value outside the f16 range
                                           (v / v_scale on both paths; k on mma.sync) */

/* Element type of the page pools (dflash_params.kv_dtype). */
#define DFLASH_KV_BF16               0  /* bf16 pages: every entry point but the fp8 one */
#define DFLASH_KV_FP8_E4M3           1  /* E4M3 codes with per-tensor scales:
                                           dflash_block_attn_fp8_context only */

/* dflash_params.test_flags (tests only; 0 in use). */
#define DFLASH_TEST_WITHHOLD_LOADS   1  /* the split kernels' producers issue no K/V loads, so every
                                           pipeline wait runs out (after its 4 s bound): the call
                                           finishes with DFLASH_STATUS_TIMEOUT set and nothing in
                                           flight; its outputs are not meaningful.  Exercises the
                                           bounded-wait failure path without a fault or a hang. */

/* Kernel-path selection for dflash_params.force_path. */
#define DFLASH_PATH_AUTO             0
#define DFLASH_PATH_MMA              1  /* warp-level mma.sync tiles (any R <= 128) */
#define DFLASH_PATH_TCGEN05          2  /* tcgen05 / TMEM, one 128-row tile per kv head;
                                           batch <= 768 */

typedef struct dflash_params {
  int32_t batch;             /* B >= 1 requests */
  int32_t num_q_heads;       /* Hq; Hq % Hkv == 0 */
  int32_t num_kv_heads;      /* Hkv >= 1; G = Hq / Hkv query heads share one kv head */
  int32_t head_dim;          /* D: 64 or 128 */
  int32_t page_size;         /* P tokens per page: 16, 32 or 64 */
  int32_t max_pages_per_req; /* row stride of page_table */
  int32_t num_pages;         /* pages in the K pool (and in the V pool) */
  int32_t block_size;        /* K draft tokens per request, 1..16; G*K <= 128 */
  int32_t window;            /* W: 0 = unwindowed; W > 0 = causal window (L+i-W, L+i],
                                which also bounds the block keys when W < K */
  int32_t future_keys;       /* 1: non-causal block (every later block key);
                                0: causal block plus right_window later keys */
  float   scale;             /* softmax scale > 0, applied to q.k in fp32 */
  int32_t max_ctx_len;       /* host bound on every ctx_lens[b]; sizes the plan */
  int32_t force_path;        /* DFLASH_PATH_*; 0 picks: tcgen05 for R > 64 with B*Hkv > 8,
                                or D = 128 with R > 32 and B*Hkv > 32; else mma.sync
                                (tcgen05 also when an fp8 mma.sync plan would not
                                fit shared memory) */
  int32_t force_split_tiles; /* 1..256: key tiles per split unit (as many as leave the
                                unit's page ids room in shared memory), or per CTA
                                range on the tcgen05 path (tests); 0 = planner */
  int32_t right_window;      /* with future_keys = 0: row i also sees block keys
                                i+1 .. i+right_window (0 .. K-1); 0 when future_keys = 1 */
  int32_t kv_dtype;          /* DFLASH_KV_BF16 or DFLASH_KV_FP8_E4M3 (pool element type) */
  int32_t test_flags;        /* 0, or DFLASH_TEST_WITHHOLD_LOADS (tests of the failure path) */
  int32_t reserved[1];       /* must be zero */
} dflash_params;

/*
 * What the planner chose for a parameter set (for tests and benchmarks).
 * Flat split (flat = 1, the tcgen05 path): `units` persistent CTAs (at most
 * one per SM unless force_split_tiles is set) that share the key tiles of
 * all (request, kv head) pairs laid end to end, split_tiles each at
 * max_ctx_len (fewer, from the actual lengths, on the device), with
 * max_splits = 2 partial slots per CTA.  Unit grid (flat = 0, the mma.sync
 * path): a grid of B * Hkv * max_splits units of split_tiles tiles.
 */
typedef struct dflash_plan_info {
  int32_t path;              /* DFLASH_PATH_MMA or DFLASH_PATH_TCGEN05 */
  int32_t rows;              /* R = G*K packed query rows per kv head */
  int32_t rows_padded;       /* R rounded up to the kernel's row granule */
  int32_t tile_keys;         /* T: keys per pipeline stage */
  int32_t split_tiles;       /* C: key tiles per split unit / per CTA range */
  int32_t max_splits;        /* split units per (request, kv head) / slots per CTA */
  int64_t units;             /* CTAs of the split kernel */
  int32_t threads;           /* threads per CTA of the split kernel */
  int32_t smem_bytes;        /* dynamic shared memory per CTA of the split kernel */
  int32_t num_sms;           /* SM count the plan was sized for */
  int32_t flat;              /* 1: persistent flat split; 0: unit grid */
  int32_t ctas_per_sm;       /* split-kernel CTAs one SM holds at once */
  int32_t reserved[1];
} dflash_plan_info;

/*
 * Workspace bytes dflash_block_attn needs for *p on the current device: a
 * 256-byte header (status word) and the fp32 partial softmax state of every
 * split unit or CTA slot (normalised output [units, R, D], base-2 LSE
 * [units, R], and the base-2 log-sum of the rounded probabilities the output
 * was normalised by [units, R]).  Returns 0 when *p is invalid.  Deterministic for a given
 * device model.
 */
size_t dflash_workspace_size(const dflash_params* p);

/* Fills *info with the plan for *p.  Returns DFLASH_OK or DFLASH_ERR_INVALID. */
int dflash_plan(const dflash_params* p, dflash_plan_info* info);

/*
 * The attention call.  All pointers are device pointers on the current
 * device, 16-byte aligned; `stream` is a cudaStream_t (NULL = legacy default
 * stream).
 *   q          bf16 [B, K, Hq, D]              query rows, token-major
 *   k_pages    bf16 [num_pages, Hkv, P, D]     key pool (HND pages)
 *   v_pages    bf16 [num_pages, Hkv, P, D]     value pool (HND pages)
 *   page_table int32 [B, max_pages_per_req]    page id of each P-token slot;
 *              only slots holding a visible position are read
 *   ctx_lens   int32 [B]                       L_b: context tokens before the
 *              block; the block's K/V are already stored at positions
 *              L_b .. L_b+K-1 of the same pages.  Read on the device only.
 *   out        bf16 [B, K, Hq, D]              softmax(q.k * scale) v, RNE
 *   lse2       fp32 [B, K, Hq]                 log2 sum exp(scale q.k) over
 *              the visible keys (including the merged later block keys)
 *   workspace  device scratch of workspace_bytes >= dflash_workspace_size(p);
 *              contents need not be initialised; the status word in it is
 *              OR-ed, never cleared, by this call.
 * Returns DFLASH_OK, or an error code with nothing launched (validation) or
 * DFLASH_ERR_LAUNCH.  Capturable in a CUDA graph: the grid depends on *p
 * only, never on the values of ctx_lens or page_table.
 */
int dflash_block_attn(const dflash_params* p, const void* q, const void* k_pages,
                      const void* v_pages, const int32_t* page_table, const int32_t* ctx_lens,
                      void* out, float* lse2, void* workspace, size_t workspace_bytes,
                      void* stream);

/*
 * dflash_block_attn with per-kernel timing marks: `split_start` and
 * `split_done` (cudaEvent_t, or NULL) are recorded on `stream` immediately
 * before the split kernel and between the split kernel and the combine
 * kernel.  The computation is the same; with `split_done` given the combine
 * kernel starts after the event instead of overlapping the split kernel's
 * tail (no programmatic dependent launch).  Same return codes.
 */
int dflash_block_attn_timed(const dflash_params* p, const void* q, const void* k_pages,
                            const void* v_pages, const int32_t* page_table,
                            const int32_t* ctx_lens, void* out, float* lse2, void* workspace,
                            size_t workspace_bytes, void* stream, void* split_start,
                            void* split_done);

/*
 * Size of the scratch array compiled into the library for
 * dflash_block_attn_static_ws: 32 MiB on every GPU that loads the library,
 * held until the process exits.
 */
#define DFLASH_STATIC_SCRATCH_BYTES (32u << 20)

/*
 * dflash_block_attn without a caller workspace.  The pages have no
 * counterpart to this entry point; it exists for callers that cannot
 * allocate device memory where they call the attention: code running while a
 * stream is captured under a mode that forbids cudaMalloc, plugins whose host
 * framework owns all device memory and passes them no scratch buffer, and
 * latency-critical paths that must not enter an allocator.  The partial
 * softmax state lives in a file-scope device array of
 * DFLASH_STATIC_SCRATCH_BYTES instead; the call allocates nothing and runs
 * the same kernels as dflash_block_attn.  Inputs and outputs are as there.
 *   - Parameter sets whose dflash_workspace_size exceeds
 *     DFLASH_STATIC_SCRATCH_BYTES are refused with DFLASH_ERR_WORKSPACE and
 *     nothing is launched.
 *   - The first call in a device's context looks up the array's device
 *     address there (cudaGetSymbolAddress, which may also load the library's
 *     device code) and caches it for that context.  A context created anew
 *     (after cudaDeviceReset, say) gets a fresh lookup on its first call.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind.  The kernels need no part of it to start at zero, and the
 *     device status word inside it is not reported here.  Calls whose work
 *     overlaps on the GPU (other streams, other host threads) race on the
 *     array: order them on one stream.
 */
int dflash_block_attn_static_ws(const dflash_params* p, const void* q, const void* k_pages,
                                const void* v_pages, const int32_t* page_table,
                                const int32_t* ctx_lens, void* out, float* lse2, void* stream);

/*
 * Block placement: the pool slot of every block token's K/V.  Block token j
 * of request b sits at logical position L_b + j, i.e. page
 * page_table[b][(L_b + j) / P] at offset (L_b + j) % P (PR #20374: the
 * block's K/V are appended to the paged cache after the context; the fused
 * spec-tail kernels of the drafter report these positions as the draft block
 * placement).
 *   placement  int32 [B, K, 2], device: (page id, offset) per block token;
 *              page id -1 where the table entry is not a page of the pool.
 *   workspace  NULL, or a workspace whose status word receives
 *              DFLASH_STATUS_BAD_PAGE / DFLASH_STATUS_BAD_CTX_LEN.
 * ctx_lens outside [0, max_ctx_len] are clamped as in dflash_block_attn.
 * Stream-ordered, no allocation.  Returns DFLASH_OK, DFLASH_ERR_INVALID,
 * DFLASH_ERR_DEVICE or DFLASH_ERR_LAUNCH.
 */
int dflash_block_placement(const dflash_params* p, const int32_t* page_table,
                           const int32_t* ctx_lens, int32_t* placement, void* workspace,
                           void* stream);

/*
 * K/V append: writes the block's K and V rows, k_block / v_block bf16
 * [B, K, Hkv, D] (token-major, like q), into the pool rows of their
 * placement, k_pages[page][h][offset][:] and likewise V.  Rows whose page id
 * is not a page of the pool are skipped (and flagged when `workspace` is
 * given).  Every other pool row is untouched.  All pointers 16-byte aligned
 * (tables 4-byte); same return codes as dflash_block_placement.
 */
int dflash_append_block_kv(const dflash_params* p, const void* k_block, const void* v_block,
                           void* k_pages, void* v_pages, const int32_t* page_table,
                           const int32_t* ctx_lens, void* workspace, void* stream);

/*
 * The K/V append followed by the attention in one launch sequence: the split
 * kernel is launched as a programmatic dependent of the append kernel, so
 * its prologue (length prefix, page lookups, query load) overlaps the
 * append and its producers read the pages once the append has finished.
 * Arguments as dflash_append_block_kv and dflash_block_attn (workspace
 * required); the result equals dflash_append_block_kv then dflash_block_attn.
 */
int dflash_block_attn_append(const dflash_params* p, const void* q, const void* k_block,
                             const void* v_block, void* k_pages, void* v_pages,
                             const int32_t* page_table, const int32_t* ctx_lens, void* out,
                             float* lse2, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Dense-suffix form (PR #16150: the draft context read from the target's
 * paged pool, the dense block suffix fused into the same softmax): the
 * block's K/V rows come from k_block / v_block, bf16 [B, K, Hkv, D]
 * (token-major, 16-byte aligned), and the pages hold the context only --
 * page-table slots past ceil(L_b / P) are never read.  Otherwise identical
 * to dflash_block_attn (same parameters, workspace and return codes).
 */
int dflash_block_attn_dense_suffix(const dflash_params* p, const void* q, const void* k_block,
                                   const void* v_block, const void* k_pages, const void* v_pages,
                                   const int32_t* page_table, const int32_t* ctx_lens, void* out,
                                   float* lse2, void* workspace, size_t workspace_bytes,
                                   void* stream);

/*
 * Dense-suffix form over fp8 context pages (PR #16150: the drafter reads its
 * context from the target's paged pool, which may store it as fp8).
 * Requires p->kv_dtype = DFLASH_KV_FP8_E4M3.  k_pages / v_pages hold OCP
 * E4M3 codes, uint8 [num_pages, Hkv, P, D] (HND, 16-byte aligned), read as
 * k = k_scale * e4m3(code) and v = v_scale * e4m3(code) with one
 * dequantisation scale per pool (finite, > 0); they hold the context
 * positions < L_b only (slots past ceil(L_b / P) are never read).  The
 * block rows come from k_block / v_block, bf16 [B, K, Hkv, D], unscaled.
 * q, out, lse2, ctx_lens, page_table and the workspace as dflash_block_attn
 * (dflash_workspace_size(p) with the same *p).  The codes are widened
 * exactly on the chip; the scores and the output use the scales in fp32.
 * Both paths take it (the planner's choice as for bf16 pages; a forced
 * mma.sync plan whose code ring would not fit shared memory is refused).
 * The P.V product runs on f16 operands on both paths, and Q.K^T too on the
 * mma.sync path (q scaled per warp by a power of two, exactly; bf16 on the
 * tcgen05 path): a block row value v / v_scale (both paths) or k (mma.sync)
 * of magnitude 65520 or more flags DFLASH_STATUS_FP8_RANGE in the device
 * status (the output is then not meaningful).
 * Non-positive or non-finite scales are refused with DFLASH_ERR_INVALID.
 * Same return codes as dflash_block_attn.
 */
int dflash_block_attn_fp8_context(const dflash_params* p, const void* q, const void* k_block,
                                  const void* v_block, const void* k_pages, const void* v_pages,
                                  float k_scale, float v_scale, const int32_t* page_table,
                                  const int32_t* ctx_lens, void* out, float* lse2, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * dflash_block_attn_fp8_context with the timing marks of
 * dflash_block_attn_timed: `split_start` / `split_done` (cudaEvent_t or NULL)
 * recorded on `stream` immediately before the split kernel and between the
 * split and the combine kernel (which then starts after the event).  Same
 * computation and return codes.
 */
int dflash_block_attn_fp8_context_timed(const dflash_params* p, const void* q, const void* k_block,
                                        const void* v_block, const void* k_pages, const void* v_pages,
                                        float k_scale, float v_scale, const int32_t* page_table,
                                        const int32_t* ctx_lens, void* out, float* lse2,
                                        void* workspace, size_t workspace_bytes, void* stream,
                                        void* split_start, void* split_done);

/*
 * Context-parallel split of one call over ranks that each hold part of every
 * request's keys: the base-2 log-sum-exp merge of partial softmax states of
 * PR #21130 (change 1), applied across ranks, with one all-gather of the
 * parts' (out, lse2) between the two calls below.
 *
 * A part covers the logical key positions [key_begin[b], key_end[b]) of
 * request b's L_b + K positions (context positions 0 .. L_b-1, then the block
 * keys L_b .. L_b+K-1); each row sees the keys of its usual visible set that
 * lie in that range.  Parts whose ranges tile [0, L_b + K) for every request
 * merge into exactly the result of dflash_block_attn.  A rank's page table
 * need only name pages for the positions its part reads.
 *
 * dflash_partial_workspace_size: workspace bytes for dflash_block_attn_partial
 * with *p (0 when invalid; kv_dtype must be DFLASH_KV_BF16 and force_path
 * DFLASH_PATH_AUTO or DFLASH_PATH_MMA: parts run on the mma.sync kernel).
 */
size_t dflash_partial_workspace_size(const dflash_params* p);

/*
 * One part.  Arguments as dflash_block_attn, plus
 *   key_begin, key_end  int32 [B], device: the part's key range per request
 *              (any values; an empty or disjoint range gives empty rows)
 *   part_out   fp32 [B, K, Hq, D], device, 16-byte aligned: the output
 *              normalised over the part's keys (0 for a row that sees none)
 *   part_lse2  fp32 [B, K, Hq]: the base-2 LSE over the part's keys (-inf
 *              for a row that sees none)
 * in place of out / lse2.  Same return codes as dflash_block_attn.
 */
int dflash_block_attn_partial(const dflash_params* p, const void* q, const void* k_pages,
                              const void* v_pages, const int32_t* page_table, const int32_t* ctx_lens,
                              const int32_t* key_begin, const int32_t* key_end, float* part_out,
                              float* part_lse2, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Merge of n_parts parts (PR #21130 change 1: lse = log2 sum_s 2^lse_s,
 * out = sum_s 2^(lse_s - lse) out_s): part_out fp32 [n_parts, B, K, Hq, D]
 * (16-byte aligned) and part_lse2 fp32 [n_parts, B, K, Hq], as an all-gather
 * of the parts' outputs lays them out, into out bf16 [B, K, Hq, D] (nearest
 * even) and lse2 fp32 [B, K, Hq].  Uses batch, num_q_heads, block_size and
 * head_dim of *p.  No workspace; stream-ordered.  Returns DFLASH_OK,
 * DFLASH_ERR_INVALID, DFLASH_ERR_DEVICE or DFLASH_ERR_LAUNCH.
 */
int dflash_combine_partials(const dflash_params* p, int n_parts, const float* part_out,
                            const float* part_lse2, void* out, float* lse2, void* stream);

/* Static text for a return code. */
const char* dflash_status_string(int status);

/*
 * Reads the device status word of a workspace (DFLASH_STATUS_* flags) with a
 * stream-ordered copy and a synchronisation of `stream`.  Returns the flags,
 * or a negative DFLASH_ERR_* code.
 */
int dflash_read_device_status(const void* workspace, void* stream);

/* Clears the device status word of a workspace (stream-ordered memset). */
int dflash_clear_device_status(void* workspace, void* stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int dflash_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_H_ */
