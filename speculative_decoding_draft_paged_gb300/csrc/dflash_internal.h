// Internal declarations shared by the host API (api.cpp) and the kernels.
// Not installed; the public interface is include/dflash.h.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "dflash.h"

#ifdef __CUDACC__
#define DF_HD __host__ __device__ __forceinline__
#else
#define DF_HD inline
#endif

namespace dflash {

constexpr int kHeaderBytes = 256;      // workspace header: status word + padding
constexpr int kMaxRows = 128;          // packed query rows per kv head (G*K)
constexpr int kMaxBlock = 16;          // draft block size K
constexpr int kStages = 4;             // TMA pipeline depth of the split kernels
// mma.sync split kernel, fp8 context: code-widening warps beside the block
// of 1 + consumer warps (base_threads <= 288 or <= 416), as many as the
// kernel's registers leave room for at one CTA per SM (the consumer code
// takes 128 registers at D = 64, KPW <= 32 and up to 168 otherwise).
DF_HD constexpr int mma_widen_warps(int D, int kpw, int base_threads) {
  return base_threads > 288 ? 3 : ((D == 64 && kpw <= 32) ? 4 : 3);
}
constexpr int kMaxSplitTiles = 256;    // key tiles per split unit, at most
constexpr int kTcMaxBatch = 768;       // tcgen05 kernel: requests whose tile prefix fits shared memory
constexpr int kTcMinTiles = 4;         // tcgen05 kernel: fewest tiles one CTA's range takes

// Everything a kernel needs, by value (kernel parameter).
struct AttnArgs {
  const uint16_t* q;          // bf16 [B, K, Hq, D]
  const uint16_t* k_pages;    // bf16 [num_pages, Hkv, P, D]
  const uint16_t* v_pages;
  const int32_t* page_table;  // [B, max_pages]
  const int32_t* ctx_lens;    // [B]
  uint16_t* out;              // bf16 [B, K, Hq, D]
  float* lse2;                // [B, K, Hq]
  float* part_o;              // [units, R, D]  normalised partial output
  float* part_lse;            // [units, R]     partial base-2 LSE
  // [units, R]: m + log2 of the sum of the probabilities as rounded for the
  // P.V product, which the partial output was divided by.  The combine
  // weights the outputs by it (and the LSE by part_lse), so a row's output is
  // normalised by the same rounded sum whatever the split.
  float* part_lseo;
  uint32_t* status;           // workspace status word
  const uint16_t* k_block;    // dense-suffix form: bf16 [B, K, Hkv, D] block rows, else null
  const uint16_t* v_block;    //   (then the pages hold the context positions < L only)
  int B, Hq, Hkv, G, D, P, max_pages, num_pages, K, W, max_ctx_len;
  int rw;                     // later block keys each row sees (K-1: non-causal form)
  float scale_log2;           // scale * log2(e), applied to q.k in fp32
  int R;                      // G * K packed rows
  int R_pad;                  // rows rounded to the kernel granule
  int T;                      // keys per tile (pipeline stage)
  int C;                      // tiles per split unit
  int S;                      // split units per (request, kv head)
  // Flat split (tcgen05 kernel): the key tiles of all (request, kv head)
  // pairs laid end to end and cut into one contiguous range per CTA;
  // part_o/part_lse hold two slots per CTA.
  int ncta;                   // CTAs of the tcgen05 split kernel
  int qn_force;               // tiles per CTA range if > 0, else from the lengths
  int qn_min;                 // fewest cost units per CTA range (lengths-derived case)
  int seg_cost;               // cost units (tile times) of a segment's end, per pair
  // fp8 context (tcgen05 kernel, dense-suffix form): the pages hold E4M3
  // codes, dequantised by per-tensor scales.  scale_log2 then includes
  // k_scale; a block key's raw score is multiplied by kblk_mul = 1/k_scale,
  // a block value row by pblk_mul = 1/v_scale as it is written into the
  // value tile, and the output by out_mul = v_scale.  All three are 1
  // otherwise.
  int fp8;
  float kblk_mul, pblk_mul, out_mul;
  // Context-parallel part (mma.sync unit grid): only the keys at logical
  // positions [key_begin[b], key_end[b]) of each request's L + K positions,
  // or null for all of them.  keep_partials: every unit writes its partial
  // state (no direct output) and the combine writes the part's fp32 output
  // out_f32 ([B, K, Hq, D], normalised over the part's keys) and its LSE
  // to lse2, instead of bf16 out.
  const int32_t* key_begin;
  const int32_t* key_end;
  int keep_partials;
  float* out_f32;
  // Tests of the failure path: the producers issue no K/V loads, so every
  // pipeline wait runs out and the kernels wind down with nothing in flight.
  int withhold_loads;
};

// Per-(request, kv head) key-range geometry of the split kernel, which covers
// the causal part of every row: row i reads [lo_i, L+i+1); the union over the
// block's rows is [lo_min, L+K).  Tiles are T-aligned in logical position.
struct Geometry {
  int L;        // context length after clamping to [0, max_ctx_len]
  int lo_min;   // first position any row reads
  int hi_max;   // one past the last position any row reads (L+K)
  int t_begin;  // first tile index
  int n_tiles;  // tiles in [t_begin, ceil(hi_max/T))
  int n_splits; // ceil(n_tiles / C)
};

DF_HD Geometry make_geometry(int L_raw, int max_ctx_len, int K, int W, int T, int C) {
  Geometry g;
  int L = L_raw < 0 ? 0 : (L_raw > max_ctx_len ? max_ctx_len : L_raw);
  g.L = L;
  int lo = 0;
  if (W > 0) {
    lo = L - W + 1;
    if (lo < 0) lo = 0;
  }
  g.lo_min = lo;
  g.hi_max = L + K;
  g.t_begin = lo / T;
  const int t_end = (g.hi_max + T - 1) / T;
  g.n_tiles = t_end - g.t_begin;
  g.n_splits = (g.n_tiles + C - 1) / C;
  return g;
}

// A context-parallel part sees only the keys at logical positions [kb, ke):
// the union interval narrows to its intersection with them, and a part that
// meets it nowhere has no tiles.
DF_HD void narrow_geometry(Geometry& g, int kb, int ke, int T, int C) {
  const int lo = g.lo_min > kb ? g.lo_min : kb;
  const int hi = g.hi_max < ke ? g.hi_max : ke;
  g.lo_min = lo;
  g.hi_max = hi > lo ? hi : lo;
  g.t_begin = lo / T;
  g.n_tiles = hi > lo ? (hi + T - 1) / T - g.t_begin : 0;
  g.n_splits = (g.n_tiles + C - 1) / C;
}

// Upper bound of Geometry::n_tiles over every L in [0, max_ctx_len].
DF_HD int max_tiles(int max_ctx_len, int K, int W, int T) {
  if (W <= 0) return (max_ctx_len + K + T - 1) / T;
  const int span = (max_ctx_len < W - 1 ? max_ctx_len : W - 1) + K;
  return (span + T - 1) / T + 1;
}

// Host-side launch plan.
struct KernelPlan {
  int path;         // DFLASH_PATH_MMA / DFLASH_PATH_TCGEN05
  int R, R_pad, T;
  int C;            // mma: tiles per unit; tcgen05: tiles per CTA range at full lengths
  int S;            // mma: units per (request, kv head); tcgen05: partial slots per CTA (2)
  int64_t units;    // mma: split units; tcgen05: CTAs
  int threads, smem_bytes;
  int kpw;          // mma path: keys per warp per tile
  int seg_cost;     // tcgen05 path: cost units of a segment's end
  bool pdl;         // launch the split kernel as a programmatic dependent of the
                    // preceding kernel (its producers wait before the first K/V load)
  bool two_ctas;    // mma path: the two-CTAs-per-SM form (3-stage ring, 96 registers)
  int ctas_per_sm;  // split-kernel CTAs one SM holds at once
  int num_sms;
};

// Block placement / K/V append (append.cu).
struct AppendArgs {
  const uint16_t* k_block;    // bf16 [B, K, Hkv, D], or null: placement only
  const uint16_t* v_block;
  uint16_t* k_pages;          // bf16 [num_pages, Hkv, P, D]
  uint16_t* v_pages;
  const int32_t* page_table;  // [B, max_pages]
  const int32_t* ctx_lens;    // [B]
  int32_t* placement;         // [B, K, 2] (page, offset), or null
  uint32_t* status;           // workspace status word, or null
  int B, K, Hkv, D, P, max_pages, num_pages, max_ctx_len;
};

// mma.sync unit grid: the combine runs one block per output row (its
// partials spread over eight warps) when rows are few and partials many, one
// warp per row otherwise.
DF_HD bool combine_wide(int max_splits, long long rows) {
  return max_splits > 8 && max_splits <= 256 && rows <= 1024;
}

// Kernel launch with an optional programmatic-dependent-launch attribute.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Launchers (defined in the .cu files).  Return a cudaError_t value.
int launch_append(const AppendArgs& a, cudaStream_t stream);
int launch_split_mma(const AttnArgs& a, const KernelPlan& plan, const CUtensorMap& tm_k,
                     const CUtensorMap& tm_v, cudaStream_t stream);
int launch_split_tc(const AttnArgs& a, const KernelPlan& plan, const CUtensorMap& tm_k,
                    const CUtensorMap& tm_v, const CUtensorMap& tm_q, const CUtensorMap& tm_out,
                    const CUtensorMap& tm_part, cudaStream_t stream);
int launch_combine(const AttnArgs& a, cudaStream_t stream, bool pdl, bool flat);
// Merge of n_parts context-parallel parts: a.part_o / a.part_lse hold part s
// of row r at s * rows + r (rows = B*K*Hq); writes bf16 out and lse2.
int launch_combine_parts(const AttnArgs& a, int n_parts, cudaStream_t stream);

// Shared-memory bytes of each split kernel for a plan (used by the planner).
int split_mma_smem_bytes(int D, int R_pad, int kpw, bool fp8, int page_slots, bool two_ctas = false);
// Whether the mma.sync kernel has a two-CTAs-per-SM form for this shape.
bool split_mma_two_ctas_ok(int D, int R_pad, int kpw, bool fp8);
int split_tc_smem_bytes(int D);

}  // namespace dflash
