// Combine kernel: split-KV partials -> final output.
//
// One warp per output row (request b, block token i, query head hq): the
// base-2 log-sum-exp combine of the row's partials (lse = log2 sum_s
// 2^lse_s, O = sum_s 2^(lseo_s) O_s / sum_s 2^(lseo_s), lseo_s the log-sum of
// the rounded probabilities partial s was divided by), the flash-decoding
// merge of PR #16150 (split-KV rework), then out (bf16, nearest-even) and
// lse2 (fp32, base 2).  The later block keys of the non-causal form are already folded
// into the partial that holds them, so there is nothing else to merge here.
// Launched with programmatic dependent launch: everything that depends on
// the inputs only is done before griddepcontrol.wait.
//   mma.sync split kernel: the row's partials are the units s of its
//   (request, kv head) pair, when a request has more than one unit.
//   tcgen05 flat split: the pair's tiles [g0, g0 + nb) lie in the ranges of
//   CTAs c0..c1 (the same tile prefix and range map as the split kernel);
//   partial s is CTA c0 + s, slot 1 of c0 when the pair starts inside c0's
//   range (its last segment there), else slot 0 (the first segment of the
//   range).  A pair inside one range was written by the split kernel itself.

#include <cuda_runtime.h>

#include "device_common.cuh"

namespace dflash {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kThreads = kWarpsPerBlock * 32;

__device__ __forceinline__ float neg_inf_f() { return __int_as_float(0xff800000); }

// Weighted sum of a row's partials into this lane's D/32 columns.  The LSE
// combines the partial LSEs (exact probability sums); the outputs, each
// divided by the sum of its rounded probabilities, are weighted by those
// rounded sums (part_lseo), so the result is divided by the row's whole
// rounded sum as it would be without a split.  Few partials (the usual
// case): one partial per lane for the weights, then the partial rows GROUP
// at a time with their loads in flight together (8 for the unit grid; 4 for
// the flat split, whose six blocks per SM leave fewer registers).  Otherwise lanes take
// partials lane, lane+32, ... for the max and the sums, and the rows eight
// at a time.
template <int D, int GROUP, typename UnitOf>
__device__ __forceinline__ void combine_row(const AttnArgs& a, int r, int ns, UnitOf unit_of,
                                            int lane, float (&acc)[D / 32], float& M_out,
                                            float& den_out, float& deno_out) {
  constexpr int V = D / 32;
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  auto load_row = [&](int sp, float (&o)[V]) {
    const float* po = a.part_o + (unit_of(sp) * a.R + r) * D + lane * V;
    if constexpr (V == 2) {
      const float2 v = *reinterpret_cast<const float2*>(po);
      o[0] = v.x;
      o[1] = v.y;
    } else {
      const float4 v = *reinterpret_cast<const float4*>(po);
      o[0] = v.x;
      o[1] = v.y;
      o[2] = v.z;
      o[3] = v.w;
    }
  };
  auto warp_max = [](float x) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, m));
    return x;
  };
  auto warp_sum = [](float x) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
  };
  if (ns <= 32) {
    // The first GROUP partial rows are loaded beside the LSEs (their
    // addresses do not depend on the weights): one round of loads before
    // the first products instead of two.
    float ov[GROUP][V];
    auto load_group = [&](int s0) {
#pragma unroll
      for (int t = 0; t < GROUP; ++t) {
        if (s0 + t < ns) {
          load_row(s0 + t, ov[t]);
        } else {
#pragma unroll
          for (int e = 0; e < V; ++e) ov[t][e] = 0.f;
        }
      }
    };
    load_group(0);
    const size_t u = lane < ns ? unit_of(lane) * a.R + r : 0;
    const float ls = lane < ns ? a.part_lse[u] : neg_inf_f();
    const float lo = lane < ns ? a.part_lseo[u] : neg_inf_f();
    const float M = warp_max(ls);
    const float w = (ls == neg_inf_f()) ? 0.f : exp2f(ls - M);
    const float wo = (lo == neg_inf_f()) ? 0.f : exp2f(lo - M);
    M_out = M;
    den_out = warp_sum(w);
    deno_out = warp_sum(wo);
    if (M == neg_inf_f()) return;
    for (int s0 = 0; s0 < ns; s0 += GROUP) {
      if (s0 > 0) load_group(s0);
#pragma unroll
      for (int t = 0; t < GROUP; ++t) {
        const float wt = __shfl_sync(0xffffffffu, wo, (s0 + t) & 31);
        const float wv = s0 + t < ns ? wt : 0.f;
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = fmaf(wv, ov[t][e], acc[e]);
      }
    }
    return;
  }
  float M = neg_inf_f();
  for (int sp = lane; sp < ns; sp += 32) M = fmaxf(M, a.part_lse[unit_of(sp) * a.R + r]);
  M = warp_max(M);
  float den = 0.f, deno = 0.f;
  for (int sp = lane; sp < ns; sp += 32) {
    const size_t u = unit_of(sp) * a.R + r;
    const float ls = a.part_lse[u];
    const float lo = a.part_lseo[u];
    den += (ls == neg_inf_f()) ? 0.f : exp2f(ls - M);
    deno += (lo == neg_inf_f()) ? 0.f : exp2f(lo - M);
  }
  M_out = M;
  den_out = warp_sum(den);
  deno_out = warp_sum(deno);
  if (M == neg_inf_f()) return;
  for (int s0 = 0; s0 < ns; s0 += 8) {
    float ov[8][V];
    float wv[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int sp = s0 + t < ns ? s0 + t : ns - 1;
      load_row(sp, ov[t]);
      const float lo = a.part_lseo[unit_of(sp) * a.R + r];
      wv[t] = (s0 + t < ns && lo != neg_inf_f()) ? exp2f(lo - M) : 0.f;
    }
#pragma unroll
    for (int t = 0; t < 8; ++t)
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] = fmaf(wv[t], ov[t][e], acc[e]);
  }
}

template <int D>
__device__ __forceinline__ void write_row(const AttnArgs& a, long long row_id, int lane,
                                          const float (&acc)[D / 32], float M, float den, float deno) {
  constexpr int V = D / 32;
  const float inv = deno > 0.f ? 1.f / deno : 0.f;
  if (a.out_f32 != nullptr) {
    // A context-parallel part: its output in fp32, for the exchange.
    float* dst = a.out_f32 + static_cast<size_t>(row_id) * D + lane * V;
    if constexpr (V == 2)
      *reinterpret_cast<float2*>(dst) = make_float2(acc[0] * inv, acc[1] * inv);
    else
      *reinterpret_cast<float4*>(dst) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    if (lane == 0) a.lse2[row_id] = den > 0.f ? M + log2f(den) : neg_inf_f();
    return;
  }
  uint16_t* dst = a.out + static_cast<size_t>(row_id) * D + lane * V;
  if constexpr (V == 2) {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  } else {
    uint2 w;
    w.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    w.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = w;
  }
  if (lane == 0) a.lse2[row_id] = den > 0.f ? M + log2f(den) : neg_inf_f();
}

// Row id -> (b, i, hq) for the [B, K, Hq] row order.
__device__ __forceinline__ void row_coords(const AttnArgs& a, long long row_id, int& b, int& i,
                                           int& hq) {
  hq = static_cast<int>(row_id % a.Hq);
  const long long t = row_id / a.Hq;
  i = static_cast<int>(t % a.K);
  b = static_cast<int>(t / a.K);
}

template <int D>
__global__ void __launch_bounds__(kThreads) combine_kernel(const AttnArgs a) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long row_id = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + warp;
  const long long rows = static_cast<long long>(a.B) * a.K * a.Hq;
  const bool active = row_id < rows;
  int b = 0, i = 0, hq = 0;
  if (active) row_coords(a, row_id, b, i, hq);
  const int h = hq / a.G;
  const int r = i * a.G + (hq - h * a.G);
  Geometry geo = make_geometry(active ? __ldg(&a.ctx_lens[b]) : 0, a.max_ctx_len, a.K, a.W, a.T, a.C);
  if (active && a.key_begin != nullptr)
    narrow_geometry(geo, __ldg(&a.key_begin[b]), __ldg(&a.key_end[b]), a.T, a.C);
  const int ns = geo.n_splits;
  const size_t unit0 = (static_cast<size_t>(b) * a.Hkv + h) * a.S;

  pdl_wait_primary();
  if (!active) return;
  float acc[D / 32], M, den, deno;
  combine_row<D, 8>(a, r, ns, [&](int sp) -> size_t { return unit0 + sp; }, lane, acc, M, den, deno);
  write_row<D>(a, row_id, lane, acc, M, den, deno);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 6) combine_flat_kernel(const AttnArgs a) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long row_id = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + warp;
  const long long rows = static_cast<long long>(a.B) * a.K * a.Hq;
  if (row_id >= rows) return;
  int b, i, hq;
  row_coords(a, row_id, b, i, hq);
  const int h = hq / a.G;
  const int r = i * a.G + (hq - h * a.G);
  // The three entries of the split kernel's tile prefix this row needs (the
  // tiles of the requests before b, of b, of all requests), from the same
  // per-request tile counts as flat_tile_prefix, by a warp reduction.
  int before = 0, own = 0, all = 0;
  for (int bb = lane; bb < a.B; bb += 32) {
    const int nt = make_geometry(__ldg(&a.ctx_lens[bb]), a.max_ctx_len, a.K, a.W, kFlatTileKeys, 1).n_tiles;
    all += nt;
    before += bb < b ? nt : 0;
    own += bb == b ? nt : 0;
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    all += __shfl_xor_sync(0xffffffffu, all, m);
    before += __shfl_xor_sync(0xffffffffu, before, m);
    own += __shfl_xor_sync(0xffffffffu, own, m);
  }
  const FlatMap fmap = flat_map_total(a, all);
  const int nb = own;
  // Cost position of the pair's first tile (flat_pair_cost).
  const long long cp = static_cast<long long>(a.Hkv) * before + static_cast<long long>(h) * nb +
                       static_cast<long long>(fmap.w) * (static_cast<long long>(b) * a.Hkv + h);
  const int c0 = static_cast<int>(div_nonneg(cp, fmap.q));
  const int c1 = static_cast<int>(div_nonneg(cp + nb - 1, fmap.q));
  if (c0 == c1) return;  // the split kernel wrote this row
  // Slot 1 of c0 when c0's range starts before this pair, i.e. at or before
  // the previous pair's last tile: the cost positions between that tile and
  // this pair's first are the previous pair's end (fmap.w of them).
  const int slot0 = static_cast<long long>(c0) * fmap.q < cp - fmap.w ? 1 : 0;

  pdl_wait_primary();
  float acc[D / 32], M, den, deno;
  combine_row<D, 4>(
      a, r, c1 - c0 + 1,
      [&](int sp) -> size_t { return static_cast<size_t>(c0 + sp) * 2 + (sp == 0 ? slot0 : 0); },
      lane, acc, M, den, deno);
  write_row<D>(a, row_id, lane, acc, M, den, deno);
}

// The same merge for few rows with many partials (mma.sync unit grid, small
// batches): one block of eight warps per output row, warp w taking the
// partials w, w+8, w+16, ... with all of its row loads in flight together,
// then a shared-memory merge of the eight warps' states -- two dependent
// rounds of loads instead of one per four partials.  ns <= kWideMaxPartials.
constexpr int kWideMaxPartials = 256;

template <int D>
__global__ void __launch_bounds__(kThreads) combine_wide_kernel(const AttnArgs a) {
  constexpr int V = D / 32;
  __shared__ float s_m[kWarpsPerBlock], s_den[kWarpsPerBlock], s_deno[kWarpsPerBlock];
  __shared__ float s_acc[kWarpsPerBlock][D];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long row_id = blockIdx.x;
  int b, i, hq;
  row_coords(a, row_id, b, i, hq);
  const int h = hq / a.G;
  const int r = i * a.G + (hq - h * a.G);
  Geometry geo = make_geometry(__ldg(&a.ctx_lens[b]), a.max_ctx_len, a.K, a.W, a.T, a.C);
  if (a.key_begin != nullptr)
    narrow_geometry(geo, __ldg(&a.key_begin[b]), __ldg(&a.key_end[b]), a.T, a.C);
  const int ns = min(geo.n_splits, kWideMaxPartials);
  const size_t unit0 = (static_cast<size_t>(b) * a.Hkv + h) * a.S;

  pdl_wait_primary();
  // This warp's partials sp = warp + 8k, k < nk <= 32: lane k holds the LSEs.
  // Its first eight partial rows are loaded beside the LSEs (their addresses
  // do not depend on the weights).
  const int nk = ns > warp ? (ns - warp + 7) / 8 : 0;
  float ov[8][V];
  auto load_group = [&](int k0) {
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      if (k0 + t < nk) {
        const float* po = a.part_o + ((unit0 + warp + 8 * (k0 + t)) * a.R + r) * D + lane * V;
        if constexpr (V == 2) {
          const float2 v = *reinterpret_cast<const float2*>(po);
          ov[t][0] = v.x;
          ov[t][1] = v.y;
        } else {
          const float4 v = *reinterpret_cast<const float4*>(po);
          ov[t][0] = v.x;
          ov[t][1] = v.y;
          ov[t][2] = v.z;
          ov[t][3] = v.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < V; ++e) ov[t][e] = 0.f;
      }
    }
  };
  load_group(0);
  const size_t u = lane < nk ? (unit0 + warp + 8 * lane) * a.R + r : 0;
  const float ls = lane < nk ? a.part_lse[u] : neg_inf_f();
  const float lo = lane < nk ? a.part_lseo[u] : neg_inf_f();
  float M = ls;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
  const float w = (ls == neg_inf_f() || M == neg_inf_f()) ? 0.f : exp2f(ls - M);
  const float wo = (lo == neg_inf_f() || M == neg_inf_f()) ? 0.f : exp2f(lo - M);
  float den = w, deno = wo;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    den += __shfl_xor_sync(0xffffffffu, den, m);
    deno += __shfl_xor_sync(0xffffffffu, deno, m);
  }
  float acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  for (int k0 = 0; k0 < nk; k0 += 8) {
    if (k0 > 0) load_group(k0);
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const float wt = __shfl_sync(0xffffffffu, wo, (k0 + t) & 31);
      const float wv = k0 + t < nk ? wt : 0.f;
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] = fmaf(wv, ov[t][e], acc[e]);
    }
  }
  if (lane == 0) {
    s_m[warp] = M;
    s_den[warp] = den;
    s_deno[warp] = deno;
  }
#pragma unroll
  for (int e = 0; e < V; ++e) s_acc[warp][lane * V + e] = acc[e];
  __syncthreads();
  if (warp != 0) return;
  float Mb = neg_inf_f();
#pragma unroll
  for (int ww = 0; ww < kWarpsPerBlock; ++ww) Mb = fmaxf(Mb, s_m[ww]);
  float denb = 0.f, denob = 0.f, accb[V];
#pragma unroll
  for (int e = 0; e < V; ++e) accb[e] = 0.f;
  if (Mb != neg_inf_f()) {
#pragma unroll
    for (int ww = 0; ww < kWarpsPerBlock; ++ww) {
      const float f = s_m[ww] == neg_inf_f() ? 0.f : exp2f(s_m[ww] - Mb);
      denb += f * s_den[ww];
      denob += f * s_deno[ww];
#pragma unroll
      for (int e = 0; e < V; ++e) accb[e] = fmaf(f, s_acc[ww][lane * V + e], accb[e]);
    }
  }
  write_row<D>(a, row_id, lane, accb, Mb, denb, denob);
}

// Merge of exchanged context-parallel parts (the base-2 log-sum-exp combine
// of PR #21130 change 1, across the parts of one call): one warp per output
// row; part s of row r sits at s * rows + r.  The parts' outputs are weighted
// by their LSEs.
template <int D>
__global__ void __launch_bounds__(kThreads) combine_parts_kernel(const AttnArgs a, int n_parts) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long row_id = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + warp;
  const long long rows = static_cast<long long>(a.B) * a.K * a.Hq;
  if (row_id >= rows) return;
  float acc[D / 32], M, den, deno;
  combine_row<D, 8>(a, static_cast<int>(row_id), n_parts, [](int sp) -> size_t { return static_cast<size_t>(sp); },
                 lane, acc, M, den, deno);
  write_row<D>(a, row_id, lane, acc, M, den, deno);
}

template <int D>
int launch_t(const AttnArgs& a, cudaStream_t stream, bool pdl, bool flat) {
  const long long rows = static_cast<long long>(a.B) * a.K * a.Hq;
  const bool wide = !flat && combine_wide(a.S, rows);
  const unsigned grid = wide ? static_cast<unsigned>(rows)
                             : static_cast<unsigned>((rows + kWarpsPerBlock - 1) / kWarpsPerBlock);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (flat) return cudaLaunchKernelEx(&cfg, combine_flat_kernel<D>, a);
  if (wide) return cudaLaunchKernelEx(&cfg, combine_wide_kernel<D>, a);
  return cudaLaunchKernelEx(&cfg, combine_kernel<D>, a);
}

}  // namespace

int launch_combine(const AttnArgs& a, cudaStream_t stream, bool pdl, bool flat) {
  if (a.D == 64) return launch_t<64>(a, stream, pdl, flat);
  if (a.D == 128) return launch_t<128>(a, stream, pdl, flat);
  return cudaErrorInvalidValue;
}

int launch_combine_parts(const AttnArgs& a, int n_parts, cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.B) * a.K * a.Hq;
  const unsigned grid = static_cast<unsigned>((rows + kWarpsPerBlock - 1) / kWarpsPerBlock);
  if (a.D == 64) combine_parts_kernel<64><<<grid, kThreads, 0, stream>>>(a, n_parts);
  else if (a.D == 128) combine_parts_kernel<128><<<grid, kThreads, 0, stream>>>(a, n_parts);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace dflash
