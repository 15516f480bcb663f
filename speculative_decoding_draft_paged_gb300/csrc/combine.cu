// Combine kernel: split-KV partials -> final output, with the merge of the
// later block keys fused in.
//
// One warp per output row (request b, block token i, query head hq).  Steps:
//  1. base-2 log-sum-exp combine of the split units' partial states
//     (lse = log2 sum_s 2^lse_s, O = sum_s 2^(lse_s - lse) O_s), the
//     flash-decoding merge of PR #16150 (split-KV rework);
//  2. non-causal form only: fold every block key j > i (position L+j, read
//     through the page table) into that state, one base-2 LSE update per key.
//     This is the merge of the block keys after the query that PR #21130
//     performs after the causal windowed decode (description "Why", change 1);
//     it is skipped exactly when no later key exists (K = 1, the last token,
//     or the causal form: PR #21130 change 2);
//  3. write out (bf16, round to nearest even) and lse2 (fp32, base 2).
// Launched with programmatic dependent launch: everything that does not read
// the partials (row geometry, the query row, the later block keys' scores) is
// done before griddepcontrol.wait.

#include <cuda_runtime.h>

#include "device_common.cuh"

namespace dflash {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ float neg_inf_f() { return __int_as_float(0xff800000); }

template <int D>
__device__ __forceinline__ void load_bf16_slice(const uint16_t* src, float (&dst)[D / 32]) {
  if constexpr (D / 32 == 2) {
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(src));
    dst[0] = bf16_bits_to_f32(w & 0xffffu);
    dst[1] = bf16_bits_to_f32(w >> 16);
  } else {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
    dst[0] = bf16_bits_to_f32(w.x & 0xffffu);
    dst[1] = bf16_bits_to_f32(w.x >> 16);
    dst[2] = bf16_bits_to_f32(w.y & 0xffffu);
    dst[3] = bf16_bits_to_f32(w.y >> 16);
  }
}

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

  // Scores and value rows of the later block keys (inputs only: this runs
  // while the split kernel finishes).  Lane t looks up the page of key
  // j = i+1+t; then every key and value row is requested before any is used.
  const bool fold = active && a.future_keys && (i + 1 < a.K);
  const int nf = fold ? a.K - 1 - i : 0;
  float sj[kMaxBlock - 1];
  float vv[kMaxBlock - 1][V];
  bool live[kMaxBlock - 1];
  if (fold) {
    int page = -1;
    int off_slot = 0;
    if (lane < nf) {
      const int pos = geo.L + i + 1 + lane;
      page = __ldg(&a.page_table[static_cast<size_t>(b) * a.max_pages + pos / a.P]);
      off_slot = pos % a.P;
      if (page < 0 || page >= a.num_pages) {
        flag_status(a.status, DFLASH_STATUS_BAD_PAGE);
        page = -1;
      }
    }
    float qv[V];
    load_bf16_slice<D>(a.q + static_cast<size_t>(row_id) * D + lane * V, qv);
    float kv[kMaxBlock - 1][V];
#pragma unroll
    for (int t = 0; t < kMaxBlock - 1; ++t) {
      const int pg = __shfl_sync(0xffffffffu, page, t);
      const int sl = __shfl_sync(0xffffffffu, off_slot, t);
      live[t] = t < nf && pg >= 0;
      if (live[t]) {
        const int64_t off =
            ((static_cast<int64_t>(pg) * a.Hkv + h) * a.P + sl) * static_cast<int64_t>(D) + lane * V;
        load_bf16_slice<D>(a.k_pages + off, kv[t]);
        load_bf16_slice<D>(a.v_pages + off, vv[t]);
      }
    }
#pragma unroll
    for (int t = 0; t < kMaxBlock - 1; ++t) {
      if (t >= nf) break;  // uniform over the warp
      float dot = 0.f;
      if (live[t]) {
#pragma unroll
        for (int e = 0; e < V; ++e) dot = fmaf(qv[e], kv[t][e], dot);
      }
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, m);
      sj[t] = dot * a.scale_log2;
    }
  }

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

  // 2. Fold the later block keys: running (m, l, acc) with O = acc / l.
  float m_run = M;
  float l_run = den;
  if (fold) {
#pragma unroll
    for (int t = 0; t < kMaxBlock - 1; ++t) {
      if (t >= nf) break;
      if (!live[t]) continue;
      const float m_new = fmaxf(m_run, sj[t]);
      const float c = (m_run == neg_inf_f()) ? 0.f : exp2f(m_run - m_new);
      const float p = exp2f(sj[t] - m_new);
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] = fmaf(p, vv[t][e], acc[e] * c);
      l_run = l_run * c + p;
      m_run = m_new;
    }
  }

  // 3. Write.
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
