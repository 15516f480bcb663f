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

  // Scores of the later block keys (inputs only: overlaps the split kernel).
  const bool fold = active && a.future_keys && (i + 1 < a.K);
  float sj[kMaxBlock];
  int64_t vrow[kMaxBlock];
  int n_fold = 0;
  if (fold) {
    float qv[V];
    load_bf16_slice<D>(a.q + static_cast<size_t>(row_id) * D + lane * V, qv);
    const int32_t* table_row = a.page_table + static_cast<size_t>(b) * a.max_pages;
    for (int j = i + 1; j < a.K; ++j) {
      const int pos = geo.L + j;
      const int page = __ldg(&table_row[pos / a.P]);
      if (page < 0 || page >= a.num_pages) {
        if (lane == 0) flag_status(a.status, DFLASH_STATUS_BAD_PAGE);
        continue;
      }
      const int64_t off =
          ((static_cast<int64_t>(page) * a.Hkv + h) * a.P + (pos % a.P)) * static_cast<int64_t>(D);
      float kv[V];
      load_bf16_slice<D>(a.k_pages + off + lane * V, kv);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < V; ++e) dot = fmaf(qv[e], kv[e], dot);
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, m);
      sj[n_fold] = dot * a.scale_log2;
      vrow[n_fold] = off;
      ++n_fold;
    }
  }

  pdl_wait_primary();
  if (!active) return;

  // 1. Combine the split units.
  const size_t unit0 = (static_cast<size_t>(b) * a.Hkv + h) * a.S;
  float M = neg_inf_f();
  for (int s = lane; s < geo.n_splits; s += 32)
    M = fmaxf(M, a.part_lse[(unit0 + s) * a.R + r]);
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));

  float acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  float den = 0.f;
  if (M != neg_inf_f()) {
    for (int s = 0; s < geo.n_splits; ++s) {
      const size_t u = unit0 + s;
      const float ls = a.part_lse[u * a.R + r];
      if (ls == neg_inf_f()) continue;
      const float w = exp2f(ls - M);
      den += w;
      const float* po = a.part_o + (u * a.R + r) * D + lane * V;
      if constexpr (V == 2) {
        const float2 v = *reinterpret_cast<const float2*>(po);
        acc[0] = fmaf(w, v.x, acc[0]);
        acc[1] = fmaf(w, v.y, acc[1]);
      } else {
        const float4 v = *reinterpret_cast<const float4*>(po);
        acc[0] = fmaf(w, v.x, acc[0]);
        acc[1] = fmaf(w, v.y, acc[1]);
        acc[2] = fmaf(w, v.z, acc[2]);
        acc[3] = fmaf(w, v.w, acc[3]);
      }
    }
  }

  // 2. Fold the later block keys: running (m, l, acc) with O = acc / l.
  float m_run = M;
  float l_run = den;
  for (int t = 0; t < n_fold; ++t) {
    const float m_new = fmaxf(m_run, sj[t]);
    const float c = (m_run == neg_inf_f()) ? 0.f : exp2f(m_run - m_new);
    const float p = exp2f(sj[t] - m_new);
    float vv[V];
    load_bf16_slice<D>(a.v_pages + vrow[t] + lane * V, vv);
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = fmaf(p, vv[e], acc[e] * c);
    l_run = l_run * c + p;
    m_run = m_new;
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
