// Split-KV kernel, tcgen05 / TMEM form, for packed row counts above 64
// (R = G*K <= 128 rows in one M = 128 tile: the MiniMax-style 16/1-head and
// the attention-DP 64/4-head drafter ranks at block size 7).
//
// One CTA = one split unit (request b, kv head h, split s) over T = 64-key
// tiles of the keys the block's rows see (row i: [lo_i, L+K) non-causal, the
// later block keys merged in the tile that holds them, or [lo_i, L+i+1)
// causal; TensorRT-LLM PR #21130), like the mma.sync kernel; the packed
// query tile (row r = i*G + g, PR #16150: query rows of
// one kv head packed so the KV is read once) is the A operand of QK^T.
//
// Warp roles (352 threads):
//   warp 0, lane 0   K producer, warp 10 lane 0 V producer: page ids come from
//                    shared memory (looked up by the whole CTA up front); one
//                    128-byte-swizzled TMA box per (page, 64-column half) into
//                    separate K and V rings.  A K slot is released as soon as
//                    its QK^T has completed and a V slot after its PV, so the
//                    V loads run just ahead of their use and the K loads far
//                    ahead, with the same shared memory as one joint ring;
//   warp 1           allocates 512 TMEM columns; lane 0 issues the MMAs:
//                    S_j = Q K_j^T (M=128, N=64, K=D) into TMEM S buffer j%2,
//                    then O_{j%2} += P_j V_j (M=128, N=D, K=64);
//   warps 2..9       softmax, two groups of four warps: group g takes the
//                    tiles j = g, g+2, g+4, ... with its own running state
//                    and its own accumulator O_g in TMEM, so two independent
//                    chains share every SM sub-partition.  A thread owns one
//                    query row (= TMEM lane of its warp's quadrant): it reads
//                    its row of S_j, masks by select, keeps a base-2 reference
//                    max that moves only when a tile's max exceeds it by more
//                    than 8 (then O_g and the row sum are rescaled, exactly),
//                    and writes P_j = 2^(s - m) in bf16 to its group's shared
//                    P buffer, the A operand of the PV MMA.  At the end group 0
//                    merges both groups' (O, m, l), like two splits, and
//                    writes the unit's normalised partial -- or, with one unit
//                    per (request, kv head), the final bf16 output and LSE.
// Every mbarrier wait is bounded (DFLASH_STATUS_TIMEOUT, then drain).

#include <cuda_runtime.h>

#include "device_common.cuh"
#include "tcgen05.cuh"

namespace dflash {
namespace {

template <int D>
struct TcCfg {
  static constexpr int T = 64;               // keys per tile
  static constexpr int NSK = 4;              // K ring stages
  static constexpr int NSV = 4;              // V ring stages
  static constexpr int kQBytes = 128 * D * 2;
  static constexpr int kTileBytes = T * D * 2;  // one K or V tile
  static constexpr int kPBytes = 128 * T * 2;   // one group's P buffer
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + NSK * kTileBytes;
  static constexpr int kOffP = kOffV + NSV * kTileBytes;
  static constexpr int kOffBar = kOffP + 2 * kPBytes;
  // k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV], s_full[2],
  // s_free[2], p_full[2], pv_done[2], merge
  static constexpr int kNumBars = 2 * NSK + 2 * NSV + 9;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffXchg = kOffMisc + 64;            // group 1's (m, l) per row
  static constexpr int kOffPages = kOffXchg + 128 * 8;
  static constexpr int kSmem = kOffPages + 4 * kMaxUnitSlots + 1024;
  static constexpr int kTmemCols = 512;   // S0 [0,64) S1 [64,128) O0 [128,128+D) O1 [256,256+D)
  static constexpr int kColO0 = 128;
  static constexpr int kColO1 = 256;
  static constexpr int kThreads = 352;
};

__device__ __forceinline__ float ninf() { return __int_as_float(0xff800000); }

template <int D>
__global__ void __launch_bounds__(352, 1)
    split_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v) {
  using C = TcCfg<D>;
  constexpr int T = C::T;
  constexpr int NSK = C::NSK;
  constexpr int NSV = C::NSV;

  const int s = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int L_raw = __ldg(&a.ctx_lens[b]);
  const Geometry geo = make_geometry(L_raw, a.max_ctx_len, a.K, a.W, T, a.C);
  if (threadIdx.x == 0 && s == 0 && h == 0 && (L_raw < 0 || L_raw > a.max_ctx_len))
    flag_status(a.status, DFLASH_STATUS_BAD_CTX_LEN);
  if (s >= geo.n_splits) return;  // empty unit, uniform over the CTA
  const int tile0 = geo.t_begin + s * a.C;
  int n = geo.n_tiles - s * a.C;
  if (n > a.C) n = a.C;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_u32);
  const uint32_t sQ = base + C::kOffQ;
  const uint32_t sK = base + C::kOffK;
  const uint32_t sV = base + C::kOffV;
  const uint32_t sP = base + C::kOffP;
  const uint32_t bars = base + C::kOffBar;
  auto k_full = [&](int st) { return bars + 8u * st; };
  auto k_empty = [&](int st) { return bars + 8u * (NSK + st); };
  auto v_full = [&](int st) { return bars + 8u * (2 * NSK + st); };
  auto v_empty = [&](int st) { return bars + 8u * (2 * NSK + NSV + st); };
  constexpr int kB0 = 2 * NSK + 2 * NSV;
  auto s_full = [&](int g) { return bars + 8u * (kB0 + g); };
  auto s_free = [&](int g) { return bars + 8u * (kB0 + 2 + g); };
  auto p_full = [&](int g) { return bars + 8u * (kB0 + 4 + g); };
  auto pv_done = [&](int g) { return bars + 8u * (kB0 + 6 + g); };
  const uint32_t merge_bar = bars + 8u * (kB0 + 8);
  uint32_t* misc = reinterpret_cast<uint32_t*>(gbase + C::kOffMisc);
  volatile uint32_t* tmem_slot = misc;          // TMEM base address from tcgen05.alloc
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile int* issued_k = reinterpret_cast<volatile int*>(misc + 2);
  volatile int* issued_v = reinterpret_cast<volatile int*>(misc + 3);
  float2* xchg = reinterpret_cast<float2*>(gbase + C::kOffXchg);
  int* pg_smem = reinterpret_cast<int*>(gbase + C::kOffPages);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int st = 0; st < NSK; ++st) {
      mbar_init(k_full(st), 1);
      mbar_init(k_empty(st), 1);
    }
    for (int st = 0; st < NSV; ++st) {
      mbar_init(v_full(st), 1);
      mbar_init(v_empty(st), 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(s_full(g), 1);
      mbar_init(s_free(g), 4);
      mbar_init(p_full(g), 4);
      mbar_init(pv_done(g), 1);
    }
    mbar_init(merge_bar, 4);
    *abort_flag = 0;
    *issued_k = 0;
    *issued_v = 0;
    fence_mbar_init();
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(misc), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();  // barrier initialisation and the TMEM address are visible
  tc_fence_after();
  // Every CTA of this grid is resident once the last one gets here: the
  // combine kernel may launch and start on its input-only work.
  pdl_launch_dependents();

  const int pages_per_tile = T / a.P;
  uint32_t tmem = 0;
  if (warp == 0 || warp == 10) {
    // The producers start as soon as warp 0 has looked the unit's page ids
    // up; they do not wait for the query tile.
    if (warp == 0)
      load_unit_pages(a, b, tile0 * pages_per_tile, n * pages_per_tile, geo.lo_min / a.P,
                      (geo.hi_max + a.P - 1) / a.P, pg_smem, lane, 32);
    named_barrier(2, 64);
  } else {
    // Warps 1..9: packed query tile, K-major with the 128-byte swizzle the
    // MMA descriptor expects: rows r = i*G + g of kv head h; rows >= R zero.
    constexpr int CPR = D / 8;
    for (int idx = threadIdx.x - 32; idx < 128 * CPR; idx += 288) {
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
      *reinterpret_cast<uint4*>(gbase + C::kOffQ + swz_offset(row, c, 128)) = v;
    }
    fence_proxy_async_smem();
    named_barrier(1, 288);
    tmem = *tmem_slot;
  }

  if (warp == 0 || warp == 10) {
    // ------------------------------------------------------------ producers
    if (lane == 0) {
      const bool is_v = warp == 10;
      const int ns = is_v ? NSV : NSK;
      const uint32_t ring = is_v ? sV : sK;
      const CUtensorMap* map = is_v ? &tm_v : &tm_k;
      volatile int* issued = is_v ? issued_v : issued_k;
      for (int j = 0; j < n; ++j) {
        const int st = j % ns;
        const uint32_t empty = is_v ? v_empty(st) : k_empty(st);
        const uint32_t full = is_v ? v_full(st) : k_full(st);
        if (j >= ns && !mbar_wait(empty, ((j / ns) - 1) & 1)) {
          flag_status(a.status, DFLASH_STATUS_TIMEOUT);
          *abort_flag = 1;
        }
        if (*abort_flag) break;
        mbar_arrive_expect_tx(full, C::kTileBytes);
        const uint32_t dst = ring + st * C::kTileBytes;
        for (int pj = 0; pj < pages_per_tile; ++pj) {
          const int page = pg_smem[j * pages_per_tile + pj];
#pragma unroll
          for (int x = 0; x < D / 64; ++x)
            tma_load_4d(dst + x * T * 128 + pj * a.P * 128, map, x * 64, 0, h, page, full);
        }
        *issued = j + 1;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, T, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
      // Descriptors differ only in the start-address field (bits 0..13,
      // address >> 4): build each base once and add offsets >> 4.
      const uint64_t dq = smem_desc_sw128(sQ, 16, 1024);
      const uint64_t dk = smem_desc_sw128(sK, 16, 1024);
      const uint64_t dp = smem_desc_sw128(sP, 16, 1024);
      const uint64_t dv = smem_desc_sw128(sV, T * 128, 1024);
      int last_qk = -1, last_pv = -1;
      for (int j = 0; j <= n; ++j) {
        if (*abort_flag) break;
        if (j < n) {
          const int st = j % NSK;
          bool ok = mbar_wait(k_full(st), (j / NSK) & 1);
          if (ok && j >= 2) ok = mbar_wait(s_free(j & 1), ((j >> 1) - 1) & 1);
          if (!ok) {
            flag_status(a.status, DFLASH_STATUS_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem + (j & 1) * T;
          const uint32_t k_off = st * C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t x = kk >> 2;
            const uint32_t within = (kk & 3) * 32;
            umma_bf16(d_tmem, dq + ((x * (128 * 128) + within) >> 4),
                      dk + ((k_off + x * (T * 128) + within) >> 4), idesc_qk, kk > 0 ? 1u : 0u);
          }
          umma_commit(k_empty(st));
          umma_commit(s_full(j & 1));
          last_qk = j;
        }
        if (j >= 1) {
          const int jj = j - 1;
          const int st = jj % NSV;
          const int g = jj & 1;
          bool ok = mbar_wait(p_full(g), (jj >> 1) & 1);
          if (ok) ok = mbar_wait(v_full(st), (jj / NSV) & 1);
          if (!ok) {
            flag_status(a.status, DFLASH_STATUS_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          tc_fence_after();
          const uint32_t v_off = st * C::kTileBytes;
          const uint32_t o_col = g ? C::kColO1 : C::kColO0;
#pragma unroll
          for (int kk = 0; kk < T / 16; ++kk)
            umma_bf16(tmem + o_col, dp + ((g * C::kPBytes + kk * 32) >> 4),
                      dv + ((v_off + kk * 16 * 128) >> 4), idesc_pv, (jj >= 2 || kk > 0) ? 1u : 0u);
          umma_commit(v_empty(st));
          umma_commit(pv_done(g));
          last_pv = jj;
        }
      }
      // Let the last commits land before the CTA winds down.
      for (int jj = last_qk - NSK + 1; jj <= last_qk; ++jj)
        if (jj >= 0) (void)mbar_wait(k_empty(jj % NSK), (jj / NSK) & 1);
      for (int jj = last_pv - NSV + 1; jj <= last_pv; ++jj)
        if (jj >= 0) (void)mbar_wait(v_empty(jj % NSV), (jj / NSV) & 1);
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 2..9)
    const int sw = warp - 2;          // 0..7
    const int grp = sw >> 2;          // tiles j = grp, grp+2, ...
    const int quad = warp & 3;        // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;
    const int gthread = (sw & 3) * 32 + lane;  // 0..127 within the group
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t o_col = grp ? C::kColO1 : C::kColO0;
    const int L = geo.L;
    int lo_r = 0x7fffffff, hi_r = -0x7fffffff;
    if (row < a.R) {
      const int i = row / a.G;
      lo_r = 0;
      if (a.W > 0) {
        lo_r = L + i - a.W + 1;
        if (lo_r < 0) lo_r = 0;
      }
      hi_r = a.future_keys ? L + a.K : L + i + 1;
    }
    int lo_rows_max = 0;
    if (a.W > 0) {
      lo_rows_max = L + a.K - a.W;
      if (lo_rows_max < 0) lo_rows_max = 0;
    }
    const int hi_rows_min = a.future_keys ? L + a.K : L + 1;

    float m_ref = ninf();
    float l_run = 0.f;
    bool ok = true;
    for (int j = grp; j < n; j += 2) {
      if (!mbar_wait_warp(s_full(grp), (j >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld64_wait(lane_addr + grp * T, sr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free(grp));

      const int p0 = (tile0 + j) * T;
      const bool need_mask = (p0 < lo_rows_max) || (p0 + T > hi_rows_min);
      // Row max of the raw scores (the scale is positive), four independent
      // chains; masked keys become -inf by select.  Boundary tiles only.
      float mx[4] = {ninf(), ninf(), ninf(), ninf()};
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int pos = p0 + c;
          const float v = (pos >= lo_r && pos < hi_r) ? __uint_as_float(sr[c]) : ninf();
          sr[c] = __float_as_uint(v);
          mx[c & 3] = fmaxf(mx[c & 3], v);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) mx[c & 3] = fmaxf(mx[c & 3], __uint_as_float(sr[c]));
      }
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * a.scale_log2;
      // The reference max moves only when this tile's max passes it by more
      // than 8 (p stays <= 2^8); O_g and l are rescaled then, which is exact.
      const bool resc = mt > m_ref + 8.f;
      float corr = 1.f;
      if (resc) {
        corr = (m_ref == ninf()) ? 0.f : fast_exp2(m_ref - mt);
        l_run *= corr;
        m_ref = mt;
      }
      const float neg_m = (m_ref == ninf()) ? 0.f : -m_ref;
      float sm[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float pa = fast_exp2(fmaf(__uint_as_float(sr[2 * c]), a.scale_log2, neg_m));
        const float pb = fast_exp2(fmaf(__uint_as_float(sr[2 * c + 1]), a.scale_log2, neg_m));
        sm[c & 3] += pa + pb;
        pk[c] = pack_bf16x2(pa, pb);
      }
      l_run += (sm[0] + sm[1]) + (sm[2] + sm[3]);

      // This group's P buffer and O_g are free once its previous PV (tile
      // j-2) has completed.  The TMEM load/store of the rescale are
      // warp-collective: the whole warp runs them when any of its rows moved
      // its reference max (factor 1 for the other rows).
      const bool warp_resc = __any_sync(0xffffffffu, resc);
      if (j >= 2) {
        if (!mbar_wait_warp(pv_done(grp), ((j >> 1) - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        if (warp_resc) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32_wait(lane_addr + o_col + cc * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
            tmem_st32(lane_addr + o_col + cc * 32, o);
          }
          tmem_wait_st();
        }
      }
      // Value rows outside [lo_min, L+K) may hold anything: zero them in the
      // stage before the PV MMA reads it (boundary tiles only).
      if (p0 < geo.lo_min || p0 + T > geo.hi_max) {
        const int st = j % NSV;
        if (!mbar_wait_warp(v_full(st), (j / NSV) & 1)) { ok = false; break; }
        if (gthread < T) {
          const int pos = p0 + gthread;
          if (pos < geo.lo_min || pos >= geo.hi_max) {
            uint8_t* vrow = gbase + C::kOffV + st * C::kTileBytes + gthread * 128;
#pragma unroll
            for (int x2 = 0; x2 < D / 64; ++x2)
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(vrow + x2 * T * 128 + c * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      // P row -> this group's shared buffer, K-major, 128-byte swizzle.
      if (row < a.R) {
        uint8_t* prow = gbase + C::kOffP + grp * C::kPBytes + row * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(prow + ((c ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(grp));
    }

    // Group 1 hands its row state to group 0 once its last PV is done.
    const int last0 = (n - 1) & ~1;            // last even tile (n >= 1)
    const int last1 = (n >= 2) ? ((n - 2) | 1) : -1;
    if (grp == 1) {
      if (ok && last1 >= 0 && !mbar_wait_warp(pv_done(1), (last1 >> 1) & 1)) ok = false;
      xchg[row] = make_float2(m_ref, l_run);
      __syncwarp();
      if (lane == 0) mbar_arrive(merge_bar);
      if (!ok) {
        flag_status(a.status, DFLASH_STATUS_TIMEOUT);
        *abort_flag = 1;
      }
    } else {
      if (ok && !mbar_wait_warp(pv_done(0), (last0 >> 1) & 1)) ok = false;
      if (ok && last1 >= 0 && !mbar_wait_warp(pv_done(1), (last1 >> 1) & 1)) ok = false;
      if (ok && !mbar_wait_warp(merge_bar, 0)) ok = false;
      if (!ok) {
        flag_status(a.status, DFLASH_STATUS_TIMEOUT);
        *abort_flag = 1;
      } else {
        tc_fence_after();
        const float2 other = xchg[row];
        const float M = fmaxf(m_ref, other.x);
        const float w0 = (m_ref == ninf()) ? 0.f : fast_exp2(m_ref - M);
        const float w1 = (other.x == ninf() || other.y == 0.f) ? 0.f : fast_exp2(other.x - M);
        const float l = w0 * l_run + w1 * other.y;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const size_t unit = (static_cast<size_t>(b) * a.Hkv + h) * a.S + s;
        const bool direct = a.S == 1;  // one unit per (request, kv head): final output
        const size_t orow = row < a.R ? out_row_index(a, b, h, row) : 0;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o0[32], o1[32];
          tmem_ld32_wait(lane_addr + C::kColO0 + cc * 32, o0);
          tmem_ld32_wait(lane_addr + C::kColO1 + cc * 32, o1);
          if (row < a.R) {
            float v[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              // A group that saw no key never wrote its accumulator: select,
              // so its uninitialised columns cannot leak in.
              const float a0 = w0 > 0.f ? w0 * __uint_as_float(o0[e]) : 0.f;
              const float a1 = w1 > 0.f ? w1 * __uint_as_float(o1[e]) : 0.f;
              v[e] = (a0 + a1) * inv;
            }
            if (direct) {
              uint4* dst = reinterpret_cast<uint4*>(a.out + orow * D + cc * 32);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                dst[e] = make_uint4(pack_bf16x2(v[8 * e], v[8 * e + 1]),
                                    pack_bf16x2(v[8 * e + 2], v[8 * e + 3]),
                                    pack_bf16x2(v[8 * e + 4], v[8 * e + 5]),
                                    pack_bf16x2(v[8 * e + 6], v[8 * e + 7]));
            } else {
              float4* dst = reinterpret_cast<float4*>(a.part_o + (unit * a.R + row) * D + cc * 32);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
            }
          }
        }
        if (row < a.R) {
          const float lse = l > 0.f ? M + log2f(l) : ninf();
          if (direct)
            a.lse2[orow] = lse;
          else
            a.part_lse[unit * a.R + row] = lse;
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    const int ik = *issued_k, iv = *issued_v;
    for (int j = ik > NSK ? ik - NSK : 0; j < ik; ++j) (void)mbar_wait(k_full(j % NSK), (j / NSK) & 1);
    for (int j = iv > NSV ? iv - NSV : 0; j < iv; ++j) (void)mbar_wait(v_full(j % NSV), (j / NSV) & 1);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
int launch_t(const AttnArgs& a, const KernelPlan& plan, const CUtensorMap& tm_k,
             const CUtensorMap& tm_v, cudaStream_t stream) {
  auto kern = split_tc_kernel<D>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<D>::kSmem);
  if (err != cudaSuccess) return err;
  dim3 grid(plan.S, a.Hkv, a.B);
  kern<<<grid, TcCfg<D>::kThreads, TcCfg<D>::kSmem, stream>>>(a, tm_k, tm_v);
  return cudaGetLastError();
}

}  // namespace

bool split_tc_available() { return true; }
int split_tc_tile_keys(int) { return 64; }
int split_tc_threads() { return TcCfg<128>::kThreads; }
int split_tc_smem_bytes(int D) { return D == 64 ? TcCfg<64>::kSmem : TcCfg<128>::kSmem; }

int launch_split_tc(const AttnArgs& a, const KernelPlan& plan, const CUtensorMap& tm_k,
                    const CUtensorMap& tm_v, cudaStream_t stream) {
  if (a.D == 64) return launch_t<64>(a, plan, tm_k, tm_v, stream);
  if (a.D == 128) return launch_t<128>(a, plan, tm_k, tm_v, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dflash
