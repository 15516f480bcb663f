// Combine kernel: split-KV partials -> final output.
//
// One warp per output row (request b, block token i, query head hq): the
// base-2 log-sum-exp combine of the row's split units (lse = log2 sum_s
// 2^lse_s, O = sum_s 2^(lse_s - lse) O_s), the flash-decoding merge of
// PR #16150 (split-KV rework), then out (bf16, nearest-even) and lse2 (fp32,
// base 2).  The later block keys of the non-causal form are already folded
// into the partial of the unit that holds them (its last tile), so there is
// nothing else to merge here.  Launched only when a request has more than
// one unit, with programmatic dependent launch: the row geometry is computed
// before griddepcontrol.wait.

#include <cuda_runtime.h>

#include "device_common.cuh"

namespace dflash {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ float neg_inf_f() { return __int_as_float(0xff800000); }

template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) combine_kernel(const AttnArgs a) {
  constexpr int V = D / 32;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long row_id = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + warp;
  const long long rows = static_cast<long long>(a.B) * a.K * a.Hq;
  const bool active = row_id < rows;

  int b = 0, i = 0, hq = 0;
  if (active) {
    hq = static_cast<int>(row_id % a.Hq);
    const long long t = row_id / a.Hq;
    i = static_cast<int>(t % a.K);
    b = static_cast<int>(t / a.K);
  }
  const int h = hq / a.G;
  const int r = i * a.G + (hq - h * a.G);
  const Geometry geo = make_geometry(active ? __ldg(&a.ctx_lens[b]) : 0, a.max_ctx_len, a.K, a.W,
                                     a.T, a.C);

  pdl_wait_primary();
  if (!active) return;

  // 1. Combine the split units.  Lanes take splits lane, lane+32, ...: their
  //    base-2 LSEs give the row max and the weights 2^(lse_s - M) in
  //    parallel; then every lane sums its D/32 output columns over the
  //    splits, eight partial rows in flight at a time.
  const size_t unit0 = (static_cast<size_t>(b) * a.Hkv + h) * a.S;
  const int ns = geo.n_splits;
  constexpr int kW = 8;  // weights kept in registers per lane: splits < 256
  float wreg[kW];
  float M = neg_inf_f();
#pragma unroll
  for (int k = 0; k < kW; ++k) {
    const int sp = lane + 32 * k;
    wreg[k] = sp < ns ? a.part_lse[(unit0 + sp) * a.R + r] : neg_inf_f();
    M = fmaxf(M, wreg[k]);
  }
  for (int sp = lane + 32 * kW; sp < ns; sp += 32) M = fmaxf(M, a.part_lse[(unit0 + sp) * a.R + r]);
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
  float den = 0.f;
#pragma unroll
  for (int k = 0; k < kW; ++k) {
    wreg[k] = (wreg[k] == neg_inf_f()) ? 0.f : exp2f(wreg[k] - M);
    den += wreg[k];
  }
  for (int sp = lane + 32 * kW; sp < ns; sp += 32) {
    const float ls = a.part_lse[(unit0 + sp) * a.R + r];
    den += (ls == neg_inf_f()) ? 0.f : exp2f(ls - M);
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) den += __shfl_xor_sync(0xffffffffu, den, m);

  float acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  if (M != neg_inf_f()) {
    for (int s0 = 0; s0 < ns; s0 += 8) {
      float ov[8][V];
      float wv[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int sp = s0 + t;
        const int spc = sp < ns ? sp : ns - 1;
        const float* po = a.part_o + ((unit0 + spc) * a.R + r) * D + lane * V;
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
        float w;
        if (sp < 32 * kW) {
          float wk = 0.f;
#pragma unroll
          for (int k = 0; k < kW; ++k)
            if ((sp >> 5) == k) wk = wreg[k];
          w = __shfl_sync(0xffffffffu, wk, sp & 31);
        } else {
          const float ls = a.part_lse[(unit0 + spc) * a.R + r];
          w = (ls == neg_inf_f()) ? 0.f : exp2f(ls - M);
        }
        wv[t] = sp < ns ? w : 0.f;
      }
#pragma unroll
      for (int t = 0; t < 8; ++t)
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = fmaf(wv[t], ov[t][e], acc[e]);
    }
  }

  const float m_run = M;
  const float l_run = den;

  // 2. Write.
  const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
  uint16_t* dst = a.out + static_cast<size_t>(row_id) * D + lane * V;
  if constexpr (V == 2) {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  } else {
    uint2 w;
    w.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    w.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = w;
  }
  if (lane == 0) a.lse2[row_id] = l_run > 0.f ? m_run + log2f(l_run) : neg_inf_f();
}

template <int D>
int launch_t(const AttnArgs& a, cudaStream_t stream, bool pdl) {
  const long long rows = static_cast<long long>(a.B) * a.K * a.Hq;
  const unsigned grid = static_cast<unsigned>((rows + kWarpsPerBlock - 1) / kWarpsPerBlock);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kWarpsPerBlock * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, combine_kernel<D>, a);
}

}  // namespace

int launch_combine(const AttnArgs& a, cudaStream_t stream, bool pdl) {
  if (a.D == 64) return launch_t<64>(a, stream, pdl);
  if (a.D == 128) return launch_t<128>(a, stream, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace dflash
