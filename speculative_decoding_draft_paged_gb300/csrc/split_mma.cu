// Split-KV kernel, warp-level tensor-core form (mma.sync m16n8k16, bf16 in,
// fp32 accumulate), for packed row counts that do not fill a 128-row tcgen05
// tile.
//
// One CTA = one split unit (request b, kv head h, split s): a contiguous range
// of T-key tiles of the keys the draft block's rows see.  Row i sees the
// interval [lo_i, hi_i): lo_i = max(0, L+i-W+1) (0 unwindowed) and hi_i = L+K
// in the non-causal form -- the block keys after i are merged into the row's
// base-2 online softmax in the tile that holds them (TensorRT-LLM PR #21130,
// "Why" and change 1) -- or L+i+1 in the causal form, where with no later key
// the causal decode already gives the exact answer (change 2).  The G*K query rows that share
// kv head h are packed into one tile (row r = i*G + g), so every K/V byte of
// the unit is read from HBM once (PR #16150, split-KV rework: one tile of
// packed query rows per kv head).
//
// Roles: warp 0 lane 0 is the producer: it looks page ids up in the page table
// and issues one 128-byte-swizzled TMA box per (page, 64-column half) for K and
// V into a 4-stage ring (3 in the two-CTAs-per-SM form; full/empty
// mbarriers).  Pages outside the unit's visible range are fetched with page
// coordinate -1, which the TMA unit fills with zeros.  Consumer warps form
// an (R_pad/16) x (T/KPW) grid: warp (wr, wk) owns query rows [16 wr,
// 16 wr + 16) and keys [wk KPW, (wk+1) KPW) of every tile, keeps its own
// online-softmax state in registers (base 2), and the warps of a row group
// merge their states through shared memory at the end.
// Two row sums are kept: the exact one (for the LSE) and the sum of the
// probabilities as rounded for the P.V product (one more MMA per 16 keys,
// against an all-ones B fragment), which the output is divided by, so that
// the rounding of a dominant probability cancels instead of reaching the
// output.
// Output: the unit's normalised partial O and base-2 LSE in the workspace, or,
// with one unit per (request, kv head), the final bf16 output and LSE.
// fp8 context (dense-suffix form over E4M3 pages): each stage's codes land in
// a code ring beside the tile ring, and three or four extra warps widen them
// into the stage's tiles while the consumers run their MMAs on the tiles
// before (the consumers wait for the widened stage instead of the load).
// A stage's tiles are free when its codes land: the producer loaded them
// only after every consumer released the stage's previous tile.  The MMAs take f16
// operands then: every E4M3 value is an f16 value (one conversion per two
// codes), the warp's query rows are scaled by a power of two into f16 range,
// P is rounded to f16 with a 2^7 offset that keeps it above the f16
// subnormals, and the block rows are written as f16 (a value outside the f16
// range flags DFLASH_STATUS_FP8_RANGE).  The per-tensor scales fold into the
// score scale and the output, as in the tcgen05 kernel.  The TMA writes only
// the code ring, so the generic writes into the tiles need no proxy fence.

#include <cuda_runtime.h>

#include "device_common.cuh"

namespace dflash {
namespace {

template <int D>
struct MmaTile {
  static constexpr int T = (D == 64) ? 128 : 64;          // keys per stage
  static constexpr int kTileBytes = T * D * 2;             // one of K or V
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kCodeStageBytes = 2 * T * D;        // fp8 context: K and V codes
};

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }


// m16n8k16 MMA with f16 (fp8 context) or bf16 operands.
template <bool F16>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (F16)
    mma_f16_16816(d, a, b0, b1);
  else
    mma_bf16_16816(d, a, b0, b1);
}

template <bool F16>
__device__ __forceinline__ uint32_t pack_16x2(float lo, float hi) {
  if constexpr (F16)
    return pack_f16x2(lo, hi);
  else
    return pack_bf16x2(lo, hi);
}

// fp8 context: block rows [lo, hi) of one warp's key slice as f16 (times
// `mul`) into a stage tile whose row 0 is position p0; a value that rounds
// outside the f16 range flags DFLASH_STATUS_FP8_RANGE.
template <int D, int T>
__device__ __forceinline__ void write_suffix_rows_f16(uint8_t* tile, const uint16_t* src, const AttnArgs& a, int b,
                                                      int h, int L, int p0, int lo, int hi, int lane, float mul) {
  constexpr int CPR = D / 8;
  const int r_lo = max(L, lo);
  const int r_hi = min(L + a.K, hi);
  const int n = (r_hi - r_lo) * CPR;
  bool bad = false;
  for (int e = lane; e < n; e += 32) {
    const int pos = r_lo + e / CPR;
    const int c = e - (e / CPR) * CPR;
    const int rr = pos - p0;
    const uint4 x = __ldg(
        reinterpret_cast<const uint4*>(src + ((static_cast<size_t>(b) * a.K + (pos - L)) * a.Hkv + h) * D) + c);
    auto cv = [&](uint32_t w) {
      const float f0 = bf16_bits_to_f32(w & 0xffffu) * mul, f1 = bf16_bits_to_f32(w >> 16) * mul;
      bad |= fabsf(f0) >= 65520.f || fabsf(f1) >= 65520.f;
      return pack_f16x2(f0, f1);
    };
    *reinterpret_cast<uint4*>(tile + (c >> 3) * T * 128 + rr * 128 + (((c & 7) ^ (rr & 7)) << 4)) =
        make_uint4(cv(x.x), cv(x.y), cv(x.z), cv(x.w));
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(a.status, DFLASH_STATUS_FP8_RANGE);
}

// fp8 context: widening warp ww of nww converts the 8-row groups ww, ww+nww,
// ... of a stage's 2T code rows (K rows, then V rows) into the stage's f16
// tiles.  In a group, lane l takes row 2*(l/8) + (l%8)/4; at D = 64 its code
// word l%4, at D = 128 the words wa = l%4 + 4*((l%8)/4) and wa^4, so that
// every quarter-warp's 16-byte loads and stores fall in distinct bank groups.
// Row offsets of a group add r0*D (codes) and r0*128 (tiles) to per-lane
// offsets, as r0 is a multiple of 8 (both swizzles repeat every 8 rows).
template <int D, int T>
__device__ __forceinline__ void widen_stage_rows(const uint8_t* codes, uint8_t* k_tile, uint8_t* v_tile, int ww,
                                                 int nww, int lane) {
  const int r_in = 2 * (lane >> 3) + ((lane & 7) >> 2);
  if constexpr (D == 64) {
    const int w = lane & 3;
    const int cw = code_word<64>(r_in, w);
    const uint32_t t0 = swz_offset(r_in, 2 * w, T), t1 = swz_offset(r_in, 2 * w + 1, T);
#pragma unroll 4
    for (int g = ww; g < 2 * T / 8; g += nww) {
      const int r0 = 8 * g;
      const uint4 c = *reinterpret_cast<const uint4*>(codes + r0 * D + cw);
      uint8_t* t = r0 < T ? k_tile + r0 * 128 : v_tile + (r0 - T) * 128;
      *reinterpret_cast<uint4*>(t + t0) = widen8_f16(c.x, c.y);
      *reinterpret_cast<uint4*>(t + t1) = widen8_f16(c.z, c.w);
    }
  } else {
    const int wa = (lane & 3) + 4 * ((lane & 7) >> 2), wb = wa ^ 4;
    const int ca = code_word<128>(r_in, wa), cb = code_word<128>(r_in, wb);
    const uint32_t ta0 = swz_offset(r_in, 2 * wa, T), ta1 = swz_offset(r_in, 2 * wa + 1, T);
    const uint32_t tb0 = swz_offset(r_in, 2 * wb, T), tb1 = swz_offset(r_in, 2 * wb + 1, T);
#pragma unroll 2
    for (int g = ww; g < 2 * T / 8; g += nww) {
      const int r0 = 8 * g;
      const uint4 x = *reinterpret_cast<const uint4*>(codes + r0 * D + ca);
      const uint4 y = *reinterpret_cast<const uint4*>(codes + r0 * D + cb);
      uint8_t* t = r0 < T ? k_tile + r0 * 128 : v_tile + (r0 - T) * 128;
      *reinterpret_cast<uint4*>(t + ta0) = widen8_f16(x.x, x.y);
      *reinterpret_cast<uint4*>(t + ta1) = widen8_f16(x.z, x.w);
      *reinterpret_cast<uint4*>(t + tb0) = widen8_f16(y.x, y.y);
      *reinterpret_cast<uint4*>(t + tb1) = widen8_f16(y.z, y.w);
    }
  }
}

// Dense-suffix form: the block's K and V rows of one warp's key slice
// [lo, hi) into stage tiles whose row 0 is position p0 (f16, value rows
// divided by v_scale, with fp8 context).  Out of line: it runs on at most two
// tiles per unit and would otherwise crowd the tile loop.
template <int D, int T, bool FP8>
__device__ __noinline__ void write_slice_suffix(uint8_t* k_tile, uint8_t* v_tile, const AttnArgs& a,
                                                int b, int h, int L, int p0, int lo, int hi, int lane) {
  if constexpr (FP8) {
    write_suffix_rows_f16<D, T>(k_tile, a.k_block, a, b, h, L, p0, lo, hi, lane, 1.f);
    write_suffix_rows_f16<D, T>(v_tile, a.v_block, a, b, h, L, p0, lo, hi, lane, a.pblk_mul);
  } else {
    write_suffix_rows<D, T>(k_tile, a.k_block, a, b, h, L, p0, lo, hi, lane, 32);
    write_suffix_rows<D, T>(v_tile, a.v_block, a, b, h, L, p0, lo, hi, lane, 32);
  }
}

// MAXT: threads of the block without the widening warps (288 or 416).
// TWO: the form that two CTAs share an SM with (a 3-stage ring and at most
// 96 registers per thread), for plans of more than one wave: one CTA's
// prologue and key-slice merge then run while the other streams, and the
// SM holds twice the warps.
template <int D, int KPW, int MAXT, bool FP8, bool TWO>
__global__ void __launch_bounds__(MAXT + (FP8 ? 32 * mma_widen_warps(D, KPW, MAXT) : 0), TWO ? 2 : 1)
    split_mma_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v) {
  constexpr int T = MmaTile<D>::T;
  constexpr int NWK = T / KPW;              // key-slice warps per row group
  constexpr int NS = TWO ? 3 : kStages;
  constexpr int kTileBytes = MmaTile<D>::kTileBytes;
  constexpr int kStageBytes = MmaTile<D>::kStageBytes;
  constexpr int NT = KPW / 8;               // 8-key accumulator tiles per warp
  static_assert(KPW % 16 == 0 && T % KPW == 0, "bad key slice");
  constexpr int NWW = FP8 ? mma_widen_warps(D, KPW, MAXT) : 0;  // fp8 context: widening warps

  const int s = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;

  const int L_raw = __ldg(&a.ctx_lens[b]);
  Geometry geo = make_geometry(L_raw, a.max_ctx_len, a.K, a.W, T, a.C);
  // Context-parallel part: the keys [part_lo, part_hi) only.
  int part_lo = 0, part_hi = 0x7fffffff;
  if (a.key_begin != nullptr) {
    part_lo = __ldg(&a.key_begin[b]);
    part_hi = __ldg(&a.key_end[b]);
    narrow_geometry(geo, part_lo, part_hi, T, a.C);
  }
  if (threadIdx.x == 0 && s == 0 && h == 0 && (L_raw < 0 || L_raw > a.max_ctx_len))
    flag_status(a.status, DFLASH_STATUS_BAD_CTX_LEN);
  if (s >= geo.n_splits) return;  // empty split unit (uniform over the CTA)

  const int tile0 = geo.t_begin + s * a.C;
  int ntiles = geo.n_tiles - s * a.C;
  if (ntiles > a.C) ntiles = a.C;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  // fp8 context: a code ring of NS stages after the tile ring.
  constexpr int kCodeRing = FP8 ? NS * MmaTile<D>::kCodeStageBytes : 0;
  const uint32_t code_u32 = base_u32 + NS * kStageBytes;
  const uint32_t q_u32 = base_u32 + NS * kStageBytes + kCodeRing;
  uint8_t* q_smem = base + NS * kStageBytes + kCodeRing;
  const uint32_t bar_u32 = q_u32 + a.R_pad * D * 2;
  uint64_t* bars = reinterpret_cast<uint64_t*>(q_smem + a.R_pad * D * 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + (FP8 ? 3 : 2) * NS);
  volatile int* issued_count = abort_flag + 1;
  int* pg_smem = const_cast<int*>(abort_flag) + 4;  // the unit's page ids: C * T / P
  auto full_bar = [&](int st) { return bar_u32 + 8u * st; };
  auto empty_bar = [&](int st) { return bar_u32 + 8u * (NS + st); };
  // fp8 context: every widening warp has widened its share of stage st.
  auto widened_bar = [&](int st) { return bar_u32 + 8u * (2 * NS + st); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_consumer_warps = (a.R_pad / 16) * NWK;

  if (threadIdx.x == 0) {
    for (int st = 0; st < NS; ++st) {
      mbar_init(full_bar(st), 1);
      mbar_init(empty_bar(st), n_consumer_warps);
      if constexpr (FP8) mbar_init(widened_bar(st), NWW);
    }
    *abort_flag = 0;
    *issued_count = 0;
    fence_mbar_init();
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
  }

  // The first 128 CTAs pull the page table and the queries into L2 (each a
  // share), so that the units of later waves find their page ids and query
  // rows there rather than in DRAM.
  {
    const unsigned cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    if (cta < 128u) {
      const size_t tab_lines = (static_cast<size_t>(a.B) * a.max_pages * 4 + 127) / 128;
      const size_t q_lines = (static_cast<size_t>(a.B) * a.K * a.Hq * D * 2 + 127) / 128;
      const size_t per = (tab_lines + q_lines + 127) / 128;
      const size_t l0 = cta * per;
      const size_t l1 = l0 + per < tab_lines + q_lines ? l0 + per : tab_lines + q_lines;
      for (size_t l = l0 + threadIdx.x; l < l1; l += blockDim.x)
        prefetch_l2(l < tab_lines ? reinterpret_cast<const uint8_t*>(a.page_table) + l * 128
                                  : reinterpret_cast<const uint8_t*>(a.q) + (l - tab_lines) * 128);
    }
  }
  const int pages_per_tile = T / a.P;
  load_unit_pages(a, b, tile0 * pages_per_tile, ntiles * pages_per_tile, geo.lo_min / a.P,
                  (paged_end(a, geo) + a.P - 1) / a.P, pg_smem, threadIdx.x, blockDim.x);
  // Dense-suffix form: the unit that holds the block positions reads the
  // block rows from the dense tensors; pull them into L2 now.
  const bool dense = a.k_block != nullptr;
  if (dense && (tile0 + ntiles) * T > geo.L && tile0 * T < geo.L + a.K)
    prefetch_suffix_rows(a, b, h, threadIdx.x, blockDim.x);

  // Packed query tile: row r = i*G + g  <-  q[b, i, h*G + g, :]; rows >= R are zero.
  {
    constexpr int CPR = D / 8;  // 16-byte chunks per row
    const int chunks = a.R_pad * CPR;
    for (int idx = threadIdx.x; idx < chunks; idx += blockDim.x) {
      const int row = idx / CPR;
      const int c = idx - row * CPR;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (row < a.R) {
        const int i = row / a.G;
        const int g = row - i * a.G;
        const uint4* src = reinterpret_cast<const uint4*>(
            a.q + ((static_cast<size_t>(b) * a.K + i) * a.Hq + static_cast<size_t>(h) * a.G + g) * D);
        v = __ldg(src + c);
      }
      *reinterpret_cast<uint4*>(q_smem + swz_offset(row, c, a.R_pad)) = v;
    }
  }
  __syncthreads();
  // Every CTA of this grid is resident once the last one gets here: the
  // combine kernel may launch and start on its input-only work.
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // After a K/V append launched just before (programmatic dependent
      // launch), the pages are read only once that kernel has finished.
      pdl_wait_primary();
      // K/V rows are read once: evict them first.
      const uint64_t kv_policy = l2_policy_evict_first();
      const int n_issue = a.withhold_loads ? 0 : ntiles;  // tests of the failure path
      for (int it = 0; it < n_issue; ++it) {
        const int st = it % NS;
        if (it >= NS) {
          if (!mbar_wait(empty_bar(st), ((it / NS) - 1) & 1)) {
            flag_status(a.status, DFLASH_STATUS_TIMEOUT);
            *abort_flag = 1;
            break;
          }
        }
        if (*abort_flag) break;
        const uint32_t k_dst = base_u32 + st * kStageBytes;
        const uint32_t v_dst = k_dst + kTileBytes;
        if constexpr (FP8) {
          // One box of (D codes, P rows) per page, into the stage's codes.
          mbar_arrive_expect_tx(full_bar(st), 2 * T * D);
          const uint32_t kc = code_u32 + st * MmaTile<D>::kCodeStageBytes;
          for (int j = 0; j < pages_per_tile; ++j) {
            const int page = pg_smem[it * pages_per_tile + j];
            tma_load_4d_hint(kc + j * a.P * D, &tm_k, 0, 0, h, page, full_bar(st), kv_policy);
            tma_load_4d_hint(kc + T * D + j * a.P * D, &tm_v, 0, 0, h, page, full_bar(st), kv_policy);
          }
        } else {
          mbar_arrive_expect_tx(full_bar(st), kStageBytes);
          for (int j = 0; j < pages_per_tile; ++j) {
            const int page = pg_smem[it * pages_per_tile + j];
#pragma unroll
            for (int x = 0; x < D / 64; ++x) {
              const uint32_t off = x * T * 128 + j * a.P * 128;
              tma_load_4d_hint(k_dst + off, &tm_k, x * 64, 0, h, page, full_bar(st), kv_policy);
              tma_load_4d_hint(v_dst + off, &tm_v, x * 64, 0, h, page, full_bar(st), kv_policy);
            }
          }
        }
        *issued_count = it + 1;
      }
    }
  } else if (FP8 && warp > n_consumer_warps) {
    // ------------------------------------------------------------ widening
    const int ww = warp - 1 - n_consumer_warps;
    for (int it = 0; it < ntiles; ++it) {
      const int st = it % NS;
      if (*abort_flag) break;
      if (!mbar_wait_warp(full_bar(st), (it / NS) & 1)) {
        flag_status(a.status, DFLASH_STATUS_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      widen_stage_rows<D, T>(base + NS * kStageBytes + st * MmaTile<D>::kCodeStageBytes, base + st * kStageBytes,
                             base + st * kStageBytes + kTileBytes, ww, NWW, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(widened_bar(st));
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int cw = warp - 1;
    const int wr = cw / NWK;
    const int wk = cw - wr * NWK;
    const int kb = wk * KPW;  // first key of this warp's slice within a tile

    uint32_t qa[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      ldmatrix_x4(q_u32 + swz_offset(16 * wr + (lane & 15), kk * 2 + (lane >> 4), a.R_pad),
                  qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
    // fp8 context: the warp's query rows as f16, times the power of two qs
    // that puts their largest magnitude in [2^14, 2^15) (exact for every
    // value down to 2^-29 of it); the score scale takes 1/qs.
    float sl2 = 0.f;
    if constexpr (FP8) {
      float amax = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_f32(qa[kk][j] & 0xffffu)),
                                   fabsf(bf16_bits_to_f32(qa[kk][j] >> 16))));
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
      const int ex = (__float_as_int(amax) >> 23) & 0xff;
      const float qs = __int_as_float(min(max(268 - ex, 1), 254) << 23);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          qa[kk][j] = pack_f16x2(bf16_bits_to_f32(qa[kk][j] & 0xffffu) * qs, bf16_bits_to_f32(qa[kk][j] >> 16) * qs);
      sl2 = a.scale_log2 / qs;
    }

    // Visible interval [lo, hi) of the two rows this lane accumulates.
    const int L = geo.L;
    int lo_r[2], hi_r[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int r = 16 * wr + (lane >> 2) + 8 * e;
      if (r < a.R) {
        const int i = r / a.G;
        int lo = 0;
        if (a.W > 0) {
          lo = L + i - a.W + 1;
          if (lo < 0) lo = 0;
        }
        lo_r[e] = max(lo, part_lo);
        hi_r[e] = min(L + min(a.K, i + 1 + a.rw), part_hi);
      } else {
        lo_r[e] = 0x7fffffff;
        hi_r[e] = -0x7fffffff;
      }
    }
    int lo_rows_max = 0;  // largest row lower bound (row i = K-1)
    if (a.W > 0) {
      lo_rows_max = L + a.K - a.W;
      if (lo_rows_max < 0) lo_rows_max = 0;
    }
    lo_rows_max = max(lo_rows_max, part_lo);
    const int hi_rows_min = min(L + min(a.K, 1 + a.rw), part_hi);  // smallest row upper bound (row 0)

    float m_run[2] = {neg_inf(), neg_inf()};
    float l_run[2] = {0.f, 0.f};
    // Row sums of the probabilities as rounded for the P.V product, from one
    // extra MMA per 16 keys against an all-ones B fragment: lt[0..1] for row
    // lane/4, lt[2..3] for row lane/4 + 8 (every column holds the sum, and
    // every lane of a quad the whole sum over the warp's key slice).  The
    // output is divided by it, so the rounding of a dominant probability
    // cancels; the LSE keeps the exact sum l_run.
    float lt[4] = {0.f, 0.f, 0.f, 0.f};
    constexpr uint32_t kOnes = FP8 ? 0x3C003C00u : 0x3F803F80u;  // 1.0 in both halves
    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    bool aborted = false;
    for (int it = 0; it < ntiles; ++it) {
      const int st = it % NS;
      if (!mbar_wait_warp(FP8 ? widened_bar(st) : full_bar(st), (it / NS) & 1)) {
        flag_status(a.status, DFLASH_STATUS_TIMEOUT);
        *abort_flag = 1;
        aborted = true;
        break;
      }
      const uint32_t k_st = base_u32 + st * kStageBytes;
      const uint32_t v_st = k_st + kTileBytes;
      const int p0 = (tile0 + it) * T + kb;  // logical position of the slice's first key
      if (dense && p0 + KPW > L && p0 < L + a.K) {
        // The block rows of this warp's key slice, from the dense tensors
        // (warps of other row groups with the same slice write the same
        // bytes; each warp reads only after its own writes).
        uint8_t* k_tile = base + st * kStageBytes;
        write_slice_suffix<D, T, FP8>(k_tile, k_tile + kTileBytes, a, b, h, L, p0 - kb, p0, p0 + KPW, lane);
        __syncwarp();
      }

      // S = Q K^T over this warp's 16 rows x KPW keys.
      float sacc[NT][4];
#pragma unroll
      for (int n = 0; n < NT; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int np = 0; np < KPW / 16; ++np) {
          uint32_t b0, b1, b2, b3;
          const int key = kb + np * 16 + (lane & 7) + ((lane >> 4) << 3);
          ldmatrix_x4(k_st + swz_offset(key, kk * 2 + ((lane >> 3) & 1), T), b0, b1, b2, b3);
          mma_16816<FP8>(sacc[2 * np], qa[kk], b0, b1);
          mma_16816<FP8>(sacc[2 * np + 1], qa[kk], b2, b3);
        }
      }

      // Mask by select (boundary tiles only; uniform branch), then the row
      // max of the raw scores (the scale is positive).  With fp8 context the
      // scale includes k_scale, so a block key's score (f16 key, no scale)
      // is divided by k_scale first.
      const bool need_mask = (p0 < lo_rows_max) || (p0 + KPW > hi_rows_min) || (FP8 && p0 + KPW > L);
      if (need_mask) {
#pragma unroll
        for (int n = 0; n < NT; ++n) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int pos = p0 + n * 8 + 2 * (lane & 3) + (e & 1);
            const int ri = e >> 1;
            if (FP8 && pos >= L) sacc[n][e] *= a.kblk_mul;
            if (pos < lo_r[ri] || pos >= hi_r[ri]) sacc[n][e] = neg_inf();
          }
        }
      }
      // Online softmax, base 2.  The reference max of a row moves only when a
      // tile's max passes it by more than 8 (p stays <= 2^8); then O and l are
      // rescaled, which is exact.  The four lanes of a quad share their rows.
      float corr[2];
      bool any_resc = false;
#pragma unroll
      for (int ri = 0; ri < 2; ++ri) {
        float m4[4] = {neg_inf(), neg_inf(), neg_inf(), neg_inf()};
#pragma unroll
        for (int n = 0; n < NT; ++n)
          m4[n & 3] = fmaxf(m4[n & 3], fmaxf(sacc[n][2 * ri], sacc[n][2 * ri + 1]));
        float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        mx *= FP8 ? sl2 : a.scale_log2;
        // Selects, not a branch: the rows of a warp disagree on moving.
        const bool up = mx > m_run[ri] + 8.f;
        const float cr = (m_run[ri] == neg_inf()) ? 0.f : fast_exp2(m_run[ri] - mx);
        corr[ri] = up ? cr : 1.f;
        l_run[ri] *= corr[ri];
        m_run[ri] = up ? mx : m_run[ri];
        any_resc |= up;
        float neg_m = (m_run[ri] == neg_inf()) ? 0.f : -m_run[ri];
        if constexpr (FP8) neg_m += 7.f;  // f16 P: p * 2^7 <= 2^15
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const float p_a = fast_exp2(fmaf(sacc[n][2 * ri], FP8 ? sl2 : a.scale_log2, neg_m));
          const float p_b = fast_exp2(fmaf(sacc[n][2 * ri + 1], FP8 ? sl2 : a.scale_log2, neg_m));
          sacc[n][2 * ri] = p_a;
          sacc[n][2 * ri + 1] = p_b;
          s4[n & 3] += p_a + p_b;
        }
        l_run[ri] += (s4[0] + s4[1]) + (s4[2] + s4[3]);
      }
      if (__any_sync(0xffffffffu, any_resc)) {
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
          o[n][0] *= corr[0];
          o[n][1] *= corr[0];
          o[n][2] *= corr[1];
          o[n][3] *= corr[1];
        }
        lt[0] *= corr[0];
        lt[1] *= corr[0];
        lt[2] *= corr[1];
        lt[3] *= corr[1];
      }

      // O += P V.  Value rows outside the unit's visible range may hold
      // anything (page tails, recycled slots): zero them in registers so a
      // zero probability never meets a NaN.
      const bool sanitize = (p0 < geo.lo_min) || (p0 + KPW > geo.hi_max);
#pragma unroll
      for (int k2 = 0; k2 < KPW / 16; ++k2) {
        uint32_t pa[4];
        pa[0] = pack_16x2<FP8>(sacc[2 * k2][0], sacc[2 * k2][1]);
        pa[1] = pack_16x2<FP8>(sacc[2 * k2][2], sacc[2 * k2][3]);
        pa[2] = pack_16x2<FP8>(sacc[2 * k2 + 1][0], sacc[2 * k2 + 1][1]);
        pa[3] = pack_16x2<FP8>(sacc[2 * k2 + 1][2], sacc[2 * k2 + 1][3]);
        mma_16816<FP8>(lt, pa, kOnes, kOnes);
        uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;
        if (sanitize) {
          const int kp = p0 + k2 * 16 + 2 * (lane & 3);
          const bool v0 = kp >= geo.lo_min && kp < geo.hi_max;
          const bool v1 = kp + 1 >= geo.lo_min && kp + 1 < geo.hi_max;
          const bool v8 = kp + 8 >= geo.lo_min && kp + 8 < geo.hi_max;
          const bool v9 = kp + 9 >= geo.lo_min && kp + 9 < geo.hi_max;
          keep_lo = (v0 ? 0x0000ffffu : 0u) | (v1 ? 0xffff0000u : 0u);
          keep_hi = (v8 ? 0x0000ffffu : 0u) | (v9 ? 0xffff0000u : 0u);
        }
        const int vkey = kb + k2 * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int dn = 0; dn < D / 16; ++dn) {
          uint32_t v0, v1, v2, v3;
          ldmatrix_x4_trans(v_st + swz_offset(vkey, dn * 2 + (lane >> 4), T), v0, v1, v2, v3);
          v0 &= keep_lo;
          v2 &= keep_lo;
          v1 &= keep_hi;
          v3 &= keep_hi;
          mma_16816<FP8>(o[2 * dn], pa, v0, v1);
          mma_16816<FP8>(o[2 * dn + 1], pa, v2, v3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(st));
    }

    // Row sums: the four lanes of a quad hold disjoint keys of the same rows.
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
      l_run[ri] += __shfl_xor_sync(0xffffffffu, l_run[ri], 1);
      l_run[ri] += __shfl_xor_sync(0xffffffffu, l_run[ri], 2);
    }

    const size_t unit = (static_cast<size_t>(b) * a.Hkv + h) * a.S + s;
    float* part_o = a.part_o + unit * a.R * D;
    float* part_lse = a.part_lse + unit * a.R;
    float* part_lseo = a.part_lseo + unit * a.R;
    // One unit per (request, kv head): the final output, unless every unit
    // keeps its partial state (a context-parallel part).
    const bool direct = a.S == 1 && !a.keep_partials;
    (void)aborted;

    if constexpr (NWK == 1) {
#pragma unroll
      for (int ri = 0; ri < 2; ++ri) {
        const int r = 16 * wr + (lane >> 2) + 8 * ri;
        if (r < a.R) {
          const float l = l_run[ri];
          const float lr = lt[2 * ri];
          const float inv = lr > 0.f ? (FP8 ? a.out_mul : 1.f) / lr : 0.f;
#pragma unroll
          for (int n = 0; n < D / 8; ++n) {
            const float v0 = o[n][2 * ri] * inv, v1 = o[n][2 * ri + 1] * inv;
            if (direct)
              *reinterpret_cast<uint32_t*>(a.out + out_row_index(a, b, h, r) * D + n * 8 +
                                           2 * (lane & 3)) = pack_bf16x2(v0, v1);
            else
              *reinterpret_cast<float2*>(part_o + static_cast<size_t>(r) * D + n * 8 +
                                         2 * (lane & 3)) = make_float2(v0, v1);
          }
          if ((lane & 3) == 0) {
            const float lse = l > 0.f ? m_run[ri] + (FP8 ? log2f(l) - 7.f : log2f(l)) : neg_inf();
            if (direct) {
              a.lse2[out_row_index(a, b, h, r)] = lse;
            } else {
              part_lse[r] = lse;
              part_lseo[r] = lr > 0.f ? m_run[ri] + (FP8 ? log2f(lr) - 7.f : log2f(lr)) : neg_inf();
            }
          }
        }
      }
    } else {
      // Merge the NWK key-slice states of each row group through shared
      // memory (the stage ring is free: every issued tile was consumed).
      const int n_ct = n_consumer_warps * 32;
      named_barrier(1, n_ct);
      float* sc_o = reinterpret_cast<float*>(base);              // [cw][16][D]
      float* sc_m = sc_o + n_consumer_warps * 16 * D;            // [cw][16]
      float* sc_l = sc_m + n_consumer_warps * 16;                // [cw][16]
      float* sc_lt = sc_l + n_consumer_warps * 16;               // [cw][16]
#pragma unroll
      for (int ri = 0; ri < 2; ++ri) {
        const int rr = (lane >> 2) + 8 * ri;
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
          *reinterpret_cast<float2*>(sc_o + (cw * 16 + rr) * D + n * 8 + 2 * (lane & 3)) =
              make_float2(o[n][2 * ri], o[n][2 * ri + 1]);
        if ((lane & 3) == 0) {
          sc_m[cw * 16 + rr] = m_run[ri];
          sc_l[cw * 16 + rr] = l_run[ri];
          sc_lt[cw * 16 + rr] = lt[2 * ri];
        }
      }
      named_barrier(1, n_ct);
      const int ct = threadIdx.x - 32;
      // One item = 8 consecutive columns of one row: the row's merge weights
      // (one base-2 exponential per key-slice warp) are computed once per
      // item, and its values move as 16-byte pieces.
      for (int e = ct; e < a.R * (D / 8); e += n_ct) {
        const int r = e / (D / 8);
        const int d = (e - r * (D / 8)) * 8;
        const int g = r >> 4;
        const int rr = r & 15;
        float M = neg_inf();
#pragma unroll
        for (int w = 0; w < NWK; ++w) M = fmaxf(M, sc_m[(g * NWK + w) * 16 + rr]);
        float num[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float den = 0.f, dent = 0.f;
        if (M != neg_inf()) {
#pragma unroll
          for (int w = 0; w < NWK; ++w) {
            const int cwi = g * NWK + w;
            const float mw = sc_m[cwi * 16 + rr];
            const float wt = mw == neg_inf() ? 0.f : fast_exp2(mw - M);
            const float4 o0 = *reinterpret_cast<const float4*>(sc_o + (cwi * 16 + rr) * D + d);
            const float4 o1 = *reinterpret_cast<const float4*>(sc_o + (cwi * 16 + rr) * D + d + 4);
            num[0] = fmaf(wt, o0.x, num[0]);
            num[1] = fmaf(wt, o0.y, num[1]);
            num[2] = fmaf(wt, o0.z, num[2]);
            num[3] = fmaf(wt, o0.w, num[3]);
            num[4] = fmaf(wt, o1.x, num[4]);
            num[5] = fmaf(wt, o1.y, num[5]);
            num[6] = fmaf(wt, o1.z, num[6]);
            num[7] = fmaf(wt, o1.w, num[7]);
            den = fmaf(wt, sc_l[cwi * 16 + rr], den);
            dent = fmaf(wt, sc_lt[cwi * 16 + rr], dent);
          }
        }
        const float inv = dent > 0.f ? (FP8 ? a.out_mul : 1.f) / dent : 0.f;
        if (direct) {
          const size_t orow = out_row_index(a, b, h, r);
          *reinterpret_cast<uint4*>(a.out + orow * D + d) =
              make_uint4(pack_bf16x2(num[0] * inv, num[1] * inv), pack_bf16x2(num[2] * inv, num[3] * inv),
                         pack_bf16x2(num[4] * inv, num[5] * inv), pack_bf16x2(num[6] * inv, num[7] * inv));
          if (d == 0) a.lse2[orow] = den > 0.f ? M + (FP8 ? log2f(den) - 7.f : log2f(den)) : neg_inf();
        } else {
          float* dst = part_o + static_cast<size_t>(r) * D + d;
          *reinterpret_cast<float4*>(dst) = make_float4(num[0] * inv, num[1] * inv, num[2] * inv, num[3] * inv);
          *reinterpret_cast<float4*>(dst + 4) = make_float4(num[4] * inv, num[5] * inv, num[6] * inv, num[7] * inv);
          if (d == 0) {
            part_lse[r] = den > 0.f ? M + (FP8 ? log2f(den) - 7.f : log2f(den)) : neg_inf();
            part_lseo[r] = dent > 0.f ? M + (FP8 ? log2f(dent) - 7.f : log2f(dent)) : neg_inf();
          }
        }
      }
    }
  }


  // If a wait gave up, let every copy already issued land before the CTA's
  // shared memory is released.
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) {
    const int issued = *issued_count;
    for (int it = issued > NS ? issued - NS : 0; it < issued; ++it)
      (void)mbar_wait(full_bar(it % NS), (it / NS) & 1);
  }
}

int kpw_for(int D, int R_pad) {
  const int mt = R_pad / 16;
  if (D == 64) return mt == 1 ? 16 : (mt <= 3 ? 32 : (mt == 4 ? 64 : 128));
  return mt == 1 ? 16 : (mt == 2 ? 32 : 64);
}

template <int D, int KPW, int MAXT = 288, bool TWO = false>
int launch_t(const AttnArgs& a, const KernelPlan& plan, const CUtensorMap& tm_k,
             const CUtensorMap& tm_v, cudaStream_t stream) {
  // The two-CTA form exists for bf16 pages only.
  auto kern = TWO ? split_mma_kernel<D, KPW, MAXT, false, TWO>
                  : (a.fp8 ? split_mma_kernel<D, KPW, MAXT, true, false> : split_mma_kernel<D, KPW, MAXT, false, false>);
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         plan.smem_bytes);
  if (err != cudaSuccess) return err;
  dim3 grid(plan.S, a.Hkv, a.B);
  err = launch_kernel(kern, grid, dim3(plan.threads), plan.smem_bytes, stream, plan.pdl, a, tm_k, tm_v);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

int split_mma_smem_bytes(int D, int R_pad, int /*kpw*/, bool fp8, int page_slots, bool two_ctas) {
  const int ns = two_ctas ? 3 : kStages;
  const int stage = (D == 64) ? MmaTile<64>::kStageBytes : MmaTile<128>::kStageBytes;
  const int codes = fp8 ? ns * ((D == 64) ? MmaTile<64>::kCodeStageBytes : MmaTile<128>::kCodeStageBytes) : 0;
  return 1024 + ns * stage + codes + R_pad * D * 2 + 8 * (fp8 ? 3 : 2) * ns + 16 + 4 * page_slots;
}

// bf16 pages at D = 64 with two row groups of four 32-key warps (R_pad = 32:
// the 64/16- and 8/2-head shapes, 288 threads): that form holds 96 registers
// per thread with a few bytes of spill; the others would spill heavily.
bool split_mma_two_ctas_ok(int D, int R_pad, int kpw, bool fp8) {
  return D == 64 && R_pad == 32 && kpw == 32 && !fp8;
}

int split_mma_kpw(int D, int R_pad) { return kpw_for(D, R_pad); }

int split_mma_tile_keys(int D) { return D == 64 ? MmaTile<64>::T : MmaTile<128>::T; }

int launch_split_mma(const AttnArgs& a, const KernelPlan& plan, const CUtensorMap& tm_k,
                     const CUtensorMap& tm_v, cudaStream_t stream) {
  if (a.D == 64) {
    switch (plan.kpw) {
      case 16: return launch_t<64, 16>(a, plan, tm_k, tm_v, stream);
      case 32:
        // Three row groups of four key-slice warps need 416 threads; keep
        // the register budget of the 288-thread form otherwise.
        if (plan.two_ctas) return launch_t<64, 32, 288, true>(a, plan, tm_k, tm_v, stream);
        return 32 * (1 + plan.R_pad / 16 * (MmaTile<64>::T / 32)) > 288 ? launch_t<64, 32, 416>(a, plan, tm_k, tm_v, stream)
                                  : launch_t<64, 32, 288>(a, plan, tm_k, tm_v, stream);
      case 64: return launch_t<64, 64>(a, plan, tm_k, tm_v, stream);
      case 128: return launch_t<64, 128>(a, plan, tm_k, tm_v, stream);
    }
  } else if (a.D == 128) {
    switch (plan.kpw) {
      case 16: return launch_t<128, 16>(a, plan, tm_k, tm_v, stream);
      case 32: return launch_t<128, 32>(a, plan, tm_k, tm_v, stream);
      case 64: return launch_t<128, 64>(a, plan, tm_k, tm_v, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace dflash
