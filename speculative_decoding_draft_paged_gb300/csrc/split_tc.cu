// Split-KV kernel, tcgen05 / TMEM form, for packed row counts above 64
// (R = G*K <= 128 rows in one M = 128 tile: the MiniMax-style 16/1-head and
// the attention-DP 64/4-head drafter ranks at block size 7).
//
// Persistent flat split.  The key tiles of every (request, kv head) pair are
// laid end to end, pairs in b-major order, each pair's T = 64-key tiles
// covering the keys its block's rows see: row i sees [lo_i, L+K) in the
// non-causal form -- the block keys after i merged in the tile that holds
// them (TensorRT-LLM PR #21130, "Why" and change 1) -- or [lo_i, L+i+1) in
// the causal form (change 2).  One CTA per SM takes an equal contiguous range
// of that sequence, so every SM streams the same number of tiles whatever the
// lengths.  A range covers a few segments, one per pair: a pair that lies
// inside the range gets its final output written directly; the first and the
// last segment of a range may hold part of a pair only and write a partial
// state (normalised O, base-2 LSE) that the combine kernel merges.  The
// packed query tile of a pair (row r = i*G + g of one kv head, PR #16150: the
// query rows of one kv head packed so its KV is read once) is the A operand
// of QK^T.
//
// Warp roles (384 threads):
//   warp 10 / warp 0 K / V producer: the warp keeps the page ids of the next
//                    32 page-table slots in registers (one chunk ahead); lane
//                    0 issues one 128-byte-swizzled TMA box per (page,
//                    64-column half) into separate K and V rings.  A K slot is
//                    released when its QK^T has completed, a V slot after its
//                    PV;
//   warp 11 lane 0   query loader: the packed query tile of each segment's
//                    pair as TMA boxes of (64 columns, G heads, K tokens), once
//                    the previous segment's last QK^T is done; the next
//                    segment's tile is prefetched into L2 meanwhile;
//   warp 1           allocates 512 TMEM columns; lane 0 issues the MMAs:
//                    S_j = Q K_j^T (M=128, N=64, K=D) into TMEM S buffer j%2,
//                    then O_{j%2} += P_j V_j (M=128, N=D, K=64; P from TMEM);
//   warps 2..9       softmax, two groups of four warps: group g takes the
//                    range's tiles j = g, g+2, ... with its own running state
//                    and TMEM accumulator O_g.  A thread owns one query row
//                    (= TMEM lane of its warp's quadrant): it reads its row of
//                    S_j, masks by select, keeps a base-2 reference max that
//                    moves only when a tile's max exceeds it by more than 8
//                    (then O_g and the row sum are rescaled, exactly), and
//                    writes P_j = 2^(s - m) in bf16 (f16 with fp8 context)
//                    to its group's TMEM P columns, the A operand of the PV
//                    MMA and of a second MMA against an all-ones operand,
//                    which sums the rounded P_j per row into TMEM (L_g).  At
//                    the end of each segment both groups merge the two
//                    states, each for half of the output columns, and write
//                    them: the output divided by the rounded sum (so the
//                    rounding of a dominant probability cancels), the LSE
//                    from the exact one.
// fp8 context (dense-suffix form over E4M3 pages): each tile's codes land by
// TMA in the upper part of its ring stage and are widened there to the tile
// the MMAs read -- the K tiles to bf16 by warps 0 and 11 (even and odd
// tiles), each V tile to f16 by the softmax group that owns it (one
// conversion per two codes) -- and the per-tensor scales fold into the score
// scale and the output.  The PV product then runs on f16 operands: P is
// written as f16 with a 2^7 offset (at most 2^15 under the lazy rescale,
// clear of the f16 subnormals; the LSE takes it back), and the block's value
// rows as f16, divided by v_scale (a value past the f16 range flags
// DFLASH_STATUS_FP8_RANGE).
// Every mbarrier wait is bounded (DFLASH_STATUS_TIMEOUT, then drain).

#include <cuda_runtime.h>

#include "device_common.cuh"
#include "tcgen05.cuh"

namespace dflash {
namespace {

template <int D, bool DUAL = false>
struct TcCfg {
  static constexpr int T = 64;               // keys per tile
  static constexpr int NSK = 4;              // K ring stages
  static constexpr int NSV = DUAL ? 4 : 5;   // V ring stages (one issuer: V slots are held longer)
  // Tile j sits in stage j % NS of each ring.  With one MMA issuer per
  // softmax group (tiles j and j+1 in different groups), an even stage count
  // gives every stage to one group, so each stage's barriers are waited for
  // phase by phase by one thread.  With an odd count a group running ahead
  // could wait (by parity) for a stage's next phase before the other group's
  // current one has completed, pass early, and release the stage twice.
  // One issuer waits in tile order, which any count allows.
  static_assert(!DUAL || (NSK % 2 == 0 && NSV % 2 == 0), "ring stages per group");
  static constexpr int kQBytes = 128 * D * 2;
  static constexpr int kTileBytes = T * D * 2;  // one K or V tile
  static constexpr int kStageBytes = 128 * T * 2;   // one group's output staging buffer
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + NSK * kTileBytes;
  static constexpr int kOffStage = kOffV + NSV * kTileBytes;
  static constexpr int kOffBar = kOffStage + 2 * kStageBytes;
  // k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV], s_full[2],
  // s_free[2], p_full[2], pv_done[2], q_full, q_free, k_fix[NSK], v_read[2],
  // q_free1 (two-issuer path: group 1's release of the query tile)
  static constexpr int kNumBars = 3 * NSK + 2 * NSV + 13;
  // fp8 context: a stage's codes sit at byte kCodeOff of the stage, row r in
  // [kCodeOff + r*D, +D) (the bf16 tile's second half for D = 128), its
  // 16-byte words permuted by the TMA swizzle.
  static constexpr int kCodeOff = T * D;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffXchg = kOffMisc + 64;                 // both groups' (m, l) per row
  static constexpr int kOffPB = kOffXchg + 2 * 128 * 8;          // tile prefix per request
  static constexpr int kOffLc = kOffPB + 4 * (kTcMaxBatch + 1);  // clamped context lengths
  // Dense-suffix form: per softmax group, the block's value rows in flight.
  static constexpr int kOffVStage = (kOffLc + 4 * kTcMaxBatch + 15) / 16 * 16;
  static constexpr int kVStageBytes = kMaxBlock * D * 2;
  // An all-ones 16 x 16 B operand (K-major, no swizzle: four 8 x 16-byte
  // core matrices): P_j times it gives the row sums of the probabilities as
  // rounded for the P.V product, in TMEM beside O.
  static constexpr int kOffOnes = (kOffVStage + 2 * kVStageBytes + 127) / 128 * 128;
  static constexpr int kOnesBytes = 512;
  static constexpr int kSmem = kOffOnes + kOnesBytes + 1024;
  static_assert(kSmem <= 232448, "shared memory per CTA");
  // TMEM columns: S0 [0,64) S1 [64,128) O0 [128,128+D) O1 [256,256+D)
  // P0 [384,416) P1 [416,448) (bf16 pairs), rounded row sums L0 [448,464)
  // L1 [464,480) (16 equal columns each).
  static constexpr int kTmemCols = 512;
  static constexpr int kColO0 = 128;
  static constexpr int kColO1 = 256;
  static constexpr int kColP = 384;
  static constexpr int kColL = 448;
  static constexpr int kThreads = 384;
};

constexpr int kNoPage = -0x7fffffff - 1;  // page-table slot outside the keys a pair reads

__device__ __forceinline__ float ninf() { return __int_as_float(0xff800000); }

// One warp widens a K tile in place: lane l takes rows l and l + 32.  With
// D = 128 a row's bf16 bytes overwrite only its own codes (its second half
// is where they landed): word w's two bf16 chunks land where code words
// 2w-8 and 2w-7 were, so the words are widened in order, one at a time.
// With D = 64 a bf16 row covers the codes of two other rows, so both rows
// of every lane are read before any byte is written.  Rows at positions
// >= L are left alone (block rows, written next, or keys no row sees).
// Loops are kept rolled: this code runs beside the softmax on the same SM
// and competes with it for instruction-cache space.
template <int D, int T>
__device__ __forceinline__ void widen_k_tile(uint8_t* tile, int p0, int L, int lane) {
  if constexpr (D == 128) {
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
      const int r = lane + 32 * hh;
      if (p0 + r >= L) continue;
#pragma unroll 1
      for (int w = 0; w < D / 16; ++w) {
        const uint4 c = *reinterpret_cast<const uint4*>(tile + T * D + code_word<D>(r, w));
        *reinterpret_cast<uint4*>(tile + swz_offset(r, 2 * w, T)) = widen8(c.x, c.y);
        *reinterpret_cast<uint4*>(tile + swz_offset(r, 2 * w + 1, T)) = widen8(c.z, c.w);
      }
    }
  } else {
    uint4 raw[2][D / 16];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
      for (int w = 0; w < D / 16; ++w)
        raw[hh][w] = *reinterpret_cast<const uint4*>(tile + T * D + code_word<D>(lane + 32 * hh, w));
    __syncwarp();
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int r = lane + 32 * hh;
      if (p0 + r >= L) continue;
#pragma unroll
      for (int w = 0; w < D / 16; ++w) {
        *reinterpret_cast<uint4*>(tile + swz_offset(r, 2 * w, T)) = widen8(raw[hh][w].x, raw[hh][w].y);
        *reinterpret_cast<uint4*>(tile + swz_offset(r, 2 * w + 1, T)) = widen8(raw[hh][w].z, raw[hh][w].w);
      }
    }
  }
}

// The K fix of an fp8 tile, whole warp: once the codes have landed, widen
// them, write the dense suffix's block rows the tile holds, and arrive on
// k_fix.  False when the wait ran out.
template <int D, int T>
__device__ __noinline__ bool fp8_fix_k(const AttnArgs& a, uint8_t* tile, uint32_t full, uint32_t parity,
                                          uint32_t fix, int p0, int L, int b, int h, int lane) {
  if (!mbar_wait_warp(full, parity)) return false;
  widen_k_tile<D, T>(tile, p0, L, lane);
  if (p0 + T > L && p0 < L + a.K) write_suffix_rows<D, T>(tile, a.k_block, a, b, h, L, p0, p0, p0 + T, lane, 32);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) mbar_arrive(fix);
  return true;
}

// The dense suffix's block value rows of a tile, moved from the staging
// buffer (as write_staged_suffix) as f16 and multiplied by `mul` (1/v_scale:
// the PV product then carries v_scale for every key, applied to the output);
// a value that rounds past the f16 range flags DFLASH_STATUS_FP8_RANGE.
template <int D, int T, int MAXP>
__device__ __forceinline__ void write_staged_suffix_scaled(uint8_t* tile, const uint8_t* stage, const AttnArgs& a,
                                                           int L, int p0, int tid, int nthr, float mul) {
  asm volatile("cp.async.wait_all;" ::: "memory");
  constexpr int CPR = D / 8;
  const int n = a.K * CPR;
#pragma unroll 1
  for (int k = 0; k < MAXP; ++k) {
    const int e = tid + k * nthr;
    if (e >= n) break;
    const int j = e / CPR;
    const int c = e - j * CPR;
    const int rr = L + j - p0;
    if (rr < 0 || rr >= T) continue;
    const uint4 x = *reinterpret_cast<const uint4*>(stage + 16 * e);
    bool bad = false;
    auto sc = [&](uint32_t w) {
      const float f0 = bf16_bits_to_f32(w & 0xffffu) * mul, f1 = bf16_bits_to_f32(w >> 16) * mul;
      bad |= fabsf(f0) >= 65520.f || fabsf(f1) >= 65520.f;
      return pack_f16x2(f0, f1);
    };
    *reinterpret_cast<uint4*>(tile + (c >> 3) * T * 128 + rr * 128 + (((c & 7) ^ (rr & 7)) << 4)) =
        make_uint4(sc(x.x), sc(x.y), sc(x.z), sc(x.w));
    if (bad) flag_status(a.status, DFLASH_STATUS_FP8_RANGE);
  }
}

// D = 128: thread t of a softmax group's 128 widens V row t - 64 (t >= 64)
// to f16 when its position lies in [lo, L): a row's f16 bytes overwrite only
// its own codes, so no other thread need wait.
template <int T>
__device__ __forceinline__ void widen_v_row(uint8_t* tile, int t, int p0, int lo, int L) {
  constexpr int D = 128;
  const int r = t - 64;
  if (r < 0 || p0 + r < lo || p0 + r >= L) return;
#pragma unroll 1
  for (int w = 0; w < D / 16; ++w) {  // in order: see widen_k_tile
    const uint4 c = *reinterpret_cast<const uint4*>(tile + T * D + code_word<D>(r, w));
    *reinterpret_cast<uint4*>(tile + swz_offset(r, 2 * w, T)) = widen8_f16(c.x, c.y);
    *reinterpret_cast<uint4*>(tile + swz_offset(r, 2 * w + 1, T)) = widen8_f16(c.z, c.w);
  }
}

// D = 64: a bf16 row covers the codes of two other rows, so the group reads
// first and writes after joining.  Thread t of the group's 128 takes row
// t % 64, half t / 64 of its codes.
template <int D, int T>
__device__ __forceinline__ void read_v_codes(const uint8_t* tile, int t, uint4 (&raw)[D / 32]) {
#pragma unroll
  for (int w = 0; w < D / 32; ++w)
    raw[w] = *reinterpret_cast<const uint4*>(tile + T * D + code_word<D>(t & 63, (t >> 6) * (D / 32) + w));
}

// Writes those codes widened to f16, for rows at positions in [lo, L) (the
// context rows some key of the block sees); other rows are zeroed or
// written by the caller.
template <int D, int T>
__device__ __forceinline__ void write_v_widened(uint8_t* tile, int t, int p0, int lo, int L,
                                                const uint4 (&raw)[D / 32]) {
  const int r = t & 63;
  const int pos = p0 + r;
  if (pos < lo || pos >= L) return;
  const int c0 = (t >> 6) * (D / 16);
#pragma unroll 1
  for (int w = 0; w < D / 32; ++w) {
    *reinterpret_cast<uint4*>(tile + swz_offset(r, c0 + 2 * w, T)) = widen8_f16(raw[w].x, raw[w].y);
    *reinterpret_cast<uint4*>(tile + swz_offset(r, c0 + 2 * w + 1, T)) = widen8_f16(raw[w].z, raw[w].w);
  }
}

// One segment of a CTA's range: the part of pair (b, h) inside it.
struct Seg {
  int b, h;
  int g0;      // global index of the pair's first tile
  int nb;      // tiles of the pair
  int j0, j1;  // CTA-local tiles [j0, j1) of the segment
  int idx;     // segment number within the CTA
};

// Request whose pairs hold global tile gt: the last b with Hkv * PB[b] <= gt.
__device__ __forceinline__ int request_of_tile(const int* PB, int B, int Hkv, int gt) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (Hkv * PB[mid] <= gt) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ Seg seg_first(const int* PB, int B, int Hkv, int start, int end) {
  Seg s;
  s.b = request_of_tile(PB, B, Hkv, start);
  s.nb = PB[s.b + 1] - PB[s.b];
  s.h = (start - Hkv * PB[s.b]) / s.nb;
  s.g0 = Hkv * PB[s.b] + s.h * s.nb;
  s.j0 = 0;
  s.j1 = min(s.g0 + s.nb, end) - start;
  s.idx = 0;
  return s;
}

__device__ __forceinline__ void seg_next(Seg& s, const int* PB, int Hkv, int start, int end) {
  if (s.h + 1 < Hkv) {
    ++s.h;
  } else {
    ++s.b;
    s.h = 0;
  }
  s.nb = PB[s.b + 1] - PB[s.b];
  s.g0 = Hkv * PB[s.b] + s.h * s.nb;
  s.j0 = s.j1;
  s.j1 = min(s.g0 + s.nb, end) - start;
  ++s.idx;
}

// Raw page-table entry for one lane of page-id chunk k of a CTA's range: the
// chunk covers CTA-local tiles [k*tpc, (k+1)*tpc), tpc = 32 / ppt; lane l
// takes page l % ppt of tile k*tpc + l / ppt.  kNoPage where the tile is past
// the range or the slot lies outside the keys the pair reads.
__device__ __forceinline__ int chunk_page(const AttnArgs& a, const int* PB, const int* Lc, int start,
                                          int end, int k, int lane, int ppt) {
  const int tpc = 32 / ppt;
  const int lt = lane / ppt;
  const int gt = start + k * tpc + lt;
  if (gt >= end) return kNoPage;
  const int b = request_of_tile(PB, a.B, a.Hkv, gt);
  const int nb = PB[b + 1] - PB[b];
  const int within = gt - a.Hkv * PB[b];
  const int t = within - (within / nb) * nb;
  const Geometry geo = make_geometry(Lc[b], a.max_ctx_len, a.K, a.W, 64, 1);
  const int slot = (geo.t_begin + t) * ppt + (lane - lt * ppt);
  if (slot < geo.lo_min / a.P || slot >= (paged_end(a, geo) + a.P - 1) / a.P) return kNoPage;
  return __ldg(&a.page_table[static_cast<size_t>(b) * a.max_pages + slot]);
}

// End-of-segment output of one softmax group for output columns
// [col0, col0 + 64): w0 * O0 + w1 * O1 scaled by inv, as bf16 rows of the
// output (direct) or fp32 rows of the CTA's partial slot `unit`.  Each thread
// puts its row into the group's 16 KB staging buffer with the 128-byte
// swizzle, and one thread hands the box to the TMA engine, which writes it
// asynchronously: bf16 as one box (64 columns, G heads, K tokens) of the
// output, fp32 as two boxes (32 columns, R rows) of the partial slot.  The
// engine's read of a box is waited for only where the buffer is written
// again: at the next call (the previous segment's box) and, for fp32,
// between the two boxes, after the second half's accumulator columns have
// been fetched.  Kept out of line: it runs once per segment, and inlined it
// would crowd the tile loop's registers.
template <int D>
__device__ __noinline__ void store_segment_rows(const AttnArgs& a, const CUtensorMap* tm_out,
                                                const CUtensorMap* tm_part, uint8_t* stg,
                                                uint32_t stg_u32, uint32_t lane_addr, int col0, int grp,
                                                int row, bool leader, float w0, float w1, float inv,
                                                bool direct, int b, int h, int unit) {
  constexpr int kColO0 = 128, kColO1 = 256;
  const int bar_id = 4 + grp;
  uint8_t* srow = stg + row * 128;
  const int sw = row & 7;
  // The previous segment's box may still be reading this buffer.
  if (leader) bulk_wait_read_all();
  named_barrier(bar_id, 128);
#pragma unroll 1
  for (int cc = 0; cc < 2; ++cc) {
    uint32_t o0[32], o1[32];
    tmem_ld32x2_wait(lane_addr + kColO0 + col0 + cc * 32, lane_addr + kColO1 + col0 + cc * 32, o0, o1);
    if (!direct && cc == 1) {
      // The first fp32 box reads the buffer until here.
      if (leader) bulk_wait_read_all();
      named_barrier(bar_id, 128);
    }
    // A group that saw no key of this segment holds a stale or
    // uninitialised accumulator: select, so it cannot leak in.
    auto val = [&](int e) {
      const float a0 = w0 > 0.f ? w0 * __uint_as_float(o0[e]) : 0.f;
      const float a1 = w1 > 0.f ? w1 * __uint_as_float(o1[e]) : 0.f;
      return (a0 + a1) * inv;
    };
    if (direct) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(srow + (((cc * 4 + q) ^ sw) << 4)) =
            make_uint4(pack_bf16x2(val(8 * q), val(8 * q + 1)), pack_bf16x2(val(8 * q + 2), val(8 * q + 3)),
                       pack_bf16x2(val(8 * q + 4), val(8 * q + 5)), pack_bf16x2(val(8 * q + 6), val(8 * q + 7)));
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<float4*>(srow + ((q ^ sw) << 4)) =
            make_float4(val(4 * q), val(4 * q + 1), val(4 * q + 2), val(4 * q + 3));
    }
    if (!direct || cc == 1) {
      fence_proxy_async_smem();
      named_barrier(bar_id, 128);
      if (leader) {
        if (direct)
          tma_store_3d(tm_out, stg_u32, col0, h * a.G, b * a.K);
        else
          tma_store_3d(tm_part, stg_u32, col0 + cc * 32, 0, unit);
        bulk_commit();
      }
    }
  }
}

// The MMA issue of one softmax group on the two-issuer path (bf16 pages, no
// dense suffix): warp 1 issues for group 0 and warp 11 for group 1, each the
// QK^T of its tiles j = g, g+2, ... of the CTA's range and the PV of each
// tile after the group's next QK^T.  A group's next scores are then ready
// when its softmax of the current tile ends, whatever the other group is
// doing: one thread issuing for both serialises the two chains, since an
// MMA's issue lasts about as long as its execution (a single issuer measured
// 85.0 us against 64.6 us for two on the MiniMax shape at 65 tiles per CTA).
// Across a segment boundary the previous segment's PV goes first, so that
// segment's output does not wait for the next query tile.  The group
// releases each segment's query tile by one arrival on its own barrier
// (q_free for group 0, q_free1 for group 1), once its last QK^T there has
// completed (or at once when it has no tile there), and always after that
// query tile has landed: no release runs a phase ahead of the K producer,
// which reloads the query tile once both groups have released it.  Returns
// false when a wait ran out.
template <int D>
__device__ __noinline__ bool tc_issue_group(int g, int n, int start, int end, const int* PB, const AttnArgs& a,
                                            uint32_t tmem, uint32_t base, volatile int* abort_flag) {
  using C = TcCfg<D, true>;
  constexpr int T = C::T;
  constexpr int NSK = C::NSK;
  constexpr int NSV = C::NSV;
  const uint32_t bars = base + C::kOffBar;
  auto k_full = [&](int st) { return bars + 8u * st; };
  auto k_empty = [&](int st) { return bars + 8u * (NSK + st); };
  auto v_full = [&](int st) { return bars + 8u * (2 * NSK + st); };
  auto v_empty = [&](int st) { return bars + 8u * (2 * NSK + NSV + st); };
  constexpr int kB0 = 2 * NSK + 2 * NSV;
  const uint32_t s_full = bars + 8u * (kB0 + g);
  const uint32_t s_free = bars + 8u * (kB0 + 2 + g);
  const uint32_t p_full = bars + 8u * (kB0 + 4 + g);
  const uint32_t pv_done = bars + 8u * (kB0 + 6 + g);
  const uint32_t q_full = bars + 8u * (kB0 + 8);
  const uint32_t q_rel = bars + 8u * (g == 0 ? kB0 + 9 : kB0 + 12 + NSK);
  constexpr uint32_t idesc_qk = idesc_bf16_f32(128, T, false);
  constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
  constexpr uint32_t idesc_l = idesc_bf16_f32(128, 16, false);
  const uint64_t dq = smem_desc_sw128(base + C::kOffQ, 16, 1024);
  const uint64_t dk = smem_desc_sw128(base + C::kOffK, 16, 1024);
  const uint64_t dv = smem_desc_sw128(base + C::kOffV, T * 128, 1024);
  const uint64_t d_ones = smem_desc_noswz(base + C::kOffOnes, 128, 256);
  const uint32_t o_col = g ? C::kColO1 : C::kColO0;
  // This thread's latest commit (s_full or pv_done: barriers no other thread
  // moves, so its phase can be waited for at the end).
  uint32_t last_bar = 0, last_par = 0;
  int pv_seg = -1;                      // segment of the group's latest PV
  // O_g += P_j V_j (and L_g += P_j 1); the group's first PV in a segment
  // overwrites O_g: its P arrives only after every softmax thread has read
  // the previous segment's accumulators.
  auto pv = [&](int jj, int seg) -> bool {
    const int st = jj % NSV;
    if (!mbar_wait(p_full, (jj >> 1) & 1)) return false;
    if (!mbar_wait(v_full(st), (jj / NSV) & 1)) return false;
    tc_fence_after();
    const bool fresh = pv_seg != seg;
    pv_seg = seg;
    const uint32_t v_off = st * C::kTileBytes;
#pragma unroll
    for (int kk = 0; kk < T / 16; ++kk)
      umma_bf16_ts(tmem + o_col, tmem + C::kColP + g * (T / 2) + kk * 8, dv + ((v_off + kk * 16 * 128) >> 4),
                   idesc_pv, (!fresh || kk > 0) ? 1u : 0u);
#pragma unroll
    for (int kk = 0; kk < T / 16; ++kk)
      umma_bf16_ts(tmem + C::kColL + g * 16, tmem + C::kColP + g * (T / 2) + kk * 8, d_ones, idesc_l,
                   (!fresh || kk > 0) ? 1u : 0u);
    umma_commit(v_empty(st));
    umma_commit(pv_done);
    last_bar = pv_done;
    last_par = (jj >> 1) & 1;
    return true;
  };
  Seg sg = seg_first(PB, a.B, a.Hkv, start, end);
  int pend = -1, pend_seg = -1;  // the group's tile whose PV is still to go
  bool ok = true;
  for (;;) {
    if (pend >= 0 && pend_seg != sg.idx) {
      ok = pv(pend, pend_seg);
      pend = -1;
      if (!ok) break;
    }
    if (*abort_flag) break;
    if (!mbar_wait(q_full, sg.idx & 1)) {
      ok = false;
      break;
    }
    int last_here = -1;
    for (int j = sg.j0 + (((sg.j0 & 1) != g) ? 1 : 0); j < sg.j1; j += 2) {
      if (*abort_flag) break;
      const int st = j % NSK;
      if (!mbar_wait(k_full(st), (j / NSK) & 1) || (j >= 2 && !mbar_wait(s_free, ((j >> 1) - 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t k_off = st * C::kTileBytes;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t x = kk >> 2;
        const uint32_t within = (kk & 3) * 32;
        umma_bf16(tmem + g * T, dq + ((x * (128 * 128) + within) >> 4),
                  dk + ((k_off + x * (T * 128) + within) >> 4), idesc_qk, kk > 0 ? 1u : 0u);
      }
      umma_commit(k_empty(st));
      umma_commit(s_full);
      last_bar = s_full;
      last_par = (j >> 1) & 1;
      last_here = j;
      if (pend >= 0 && !pv(pend, pend_seg)) {
        ok = false;
        break;
      }
      pend = j;
      pend_seg = sg.idx;
    }
    if (!ok || *abort_flag || sg.j1 >= n) break;
    // Release the query tile once this group's QK^T products have read it.
    if (last_here >= 0 && !mbar_wait(s_full, (last_here >> 1) & 1)) {
      ok = false;
      break;
    }
    mbar_arrive(q_rel);
    seg_next(sg, PB, a.Hkv, start, end);
  }
  if (ok && pend >= 0 && !*abort_flag) ok = pv(pend, pend_seg);
  // This thread's MMAs have completed before the CTA winds down: its latest
  // commit (which covers all of them) has arrived.
  if (last_bar != 0) (void)mbar_wait(last_bar, last_par);
  return ok;
}

template <int D, bool FP8, bool DUAL>
__global__ void __launch_bounds__(384, 1)
    split_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_out,
                    const __grid_constant__ CUtensorMap tm_part) {
  using C = TcCfg<D, DUAL>;
  constexpr int T = C::T;
  constexpr int NSK = C::NSK;
  constexpr int NSV = C::NSV;

  extern __shared__ uint8_t smem_raw[];
  __shared__ int warp_sums[C::kThreads / 32];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_u32);
  int* PB = reinterpret_cast<int*>(gbase + C::kOffPB);
  int* Lc = reinterpret_cast<int*>(gbase + C::kOffLc);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // The page-table rows are needed right after the prefix: every CTA pulls
  // its share of the table into L2 while the lengths are being read.
  {
    const size_t lines = (static_cast<size_t>(a.B) * a.max_pages * 4 + 127) / 128;
    const size_t per = (lines + gridDim.x - 1) / gridDim.x;
    const size_t l0 = static_cast<size_t>(blockIdx.x) * per;
    const size_t l1 = l0 + per < lines ? l0 + per : lines;
    for (size_t l = l0 + threadIdx.x; l < l1; l += C::kThreads)
      touch_l2(reinterpret_cast<const uint8_t*>(a.page_table) + l * 128);
  }
  // Tile prefix over the requests, computed by every CTA.
  flat_tile_prefix<C::kThreads>(a, PB, Lc, warp_sums, blockIdx.x == 0);
  const FlatMap fmap = flat_map(a, PB);
  int start, end;
  flat_range(a, PB, fmap, blockIdx.x, start, end);
  if (end <= start) return;  // no tiles for this CTA (uniform)
  const int n = end - start;

  const uint32_t sQ = base + C::kOffQ;
  const uint32_t sK = base + C::kOffK;
  const uint32_t sV = base + C::kOffV;
  const uint32_t sStage = base + C::kOffStage;
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
  const uint32_t q_full = bars + 8u * (kB0 + 8);
  const uint32_t q_free = bars + 8u * (kB0 + 9);
  // Dense-suffix form: K tile st holds its block rows once k_fix(st) completes.
  auto k_fix = [&](int st) { return bars + 8u * (kB0 + 10 + st); };
  // fp8 context: every thread of softmax group g has read its codes of the
  // group's current V tile.
  auto v_read = [&](int g) { return bars + 8u * (kB0 + 10 + NSK + g); };
  // Two-issuer path: group 1's release of the query tile (group 0's is q_free).
  const uint32_t q_free1 = bars + 8u * (kB0 + 12 + NSK);
  const bool dense = a.k_block != nullptr;
  uint32_t* misc = reinterpret_cast<uint32_t*>(gbase + C::kOffMisc);
  volatile uint32_t* tmem_slot = misc;          // TMEM base address from tcgen05.alloc
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile int* issued_k = reinterpret_cast<volatile int*>(misc + 2);
  volatile int* issued_v = reinterpret_cast<volatile int*>(misc + 3);
  volatile int* issued_q = reinterpret_cast<volatile int*>(misc + 4);
  volatile int* stop_word = reinterpret_cast<volatile int*>(misc + 5);  // softmax warps only
  float2* xchg = reinterpret_cast<float2*>(gbase + C::kOffXchg);

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
    mbar_init(q_full, 1);
    mbar_init(q_free, 1);
    mbar_init(q_free1, 1);
    for (int st = 0; st < NSK; ++st) mbar_init(k_fix(st), 1);
    mbar_init(v_read(0), 4);
    mbar_init(v_read(1), 4);
    *abort_flag = 0;
    *issued_k = 0;
    *issued_v = 0;
    *issued_q = 0;
    *stop_word = 0;
    fence_mbar_init();
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_out);
    prefetch_tensormap(&tm_part);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(misc), C::kTmemCols);
    tmem_relinquish();
  }
  // Query rows R..127 stay zero (the TMA boxes cover rows 0..R-1 only), so
  // their scores are zero and never disturb a warp's rescale decision.
  {
    constexpr int CPR = D / 8;
    for (int idx = threadIdx.x; idx < (128 - a.R) * CPR; idx += C::kThreads) {
      const int row = a.R + idx / CPR;
      const int c = idx % CPR;
      *reinterpret_cast<uint4*>(gbase + C::kOffQ + swz_offset(row, c, 128)) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    // The all-ones operand of the row-sum MMA, in the P type (bf16, or f16
    // with fp8 context).
    constexpr uint32_t kOne2 = FP8 ? 0x3C003C00u : 0x3F803F80u;
    for (int idx = threadIdx.x; idx < C::kOnesBytes / 16; idx += C::kThreads)
      *reinterpret_cast<uint4*>(gbase + C::kOffOnes + 16 * idx) = make_uint4(kOne2, kOne2, kOne2, kOne2);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();  // barrier initialisation and the TMEM address are visible
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Every CTA of this grid is resident once the last one gets here: the
  // combine kernel may launch and start on its input-only work.
  pdl_launch_dependents();

  if (FP8 && warp == 0) {
    // ------------------------------------------------------------ fp8: even K tiles
    // Warp 0 widens the even K tiles as soon as their codes land (the odd
    // ones are warp 11's); warp 10 loads both rings.
    Seg sgc = seg_first(PB, a.B, a.Hkv, start, end);
    for (int jc = 0; jc < n; jc += 2) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      while (jc >= sgc.j1) seg_next(sgc, PB, a.Hkv, start, end);
      const Geometry geo = make_geometry(Lc[sgc.b], a.max_ctx_len, a.K, a.W, T, 1);
      const int p0 = (geo.t_begin - (sgc.g0 - start)) * T + jc * T;
      const int st = jc % NSK;
      if (!fp8_fix_k<D, T>(a, gbase + C::kOffK + st * C::kTileBytes, k_full(st), (jc / NSK) & 1, k_fix(st),
                           p0, geo.L, sgc.b, sgc.h, lane)) {
        if (lane == 0) flag_status(a.status, DFLASH_STATUS_TIMEOUT);
        *abort_flag = 1;
        break;
      }
    }
  } else if (warp == 0 || warp == 10) {
    // ------------------------------------------------------------ producers (whole warp)
    // Warp 0 reaches its first page-table shuffle about 2 us later than the
    // other warps (measured); the V tiles are needed a softmax later than the
    // K tiles, so warp 0 takes the V ring.  fp8 context: warp 10 takes both
    // rings (K then V per tile), one box of (D codes, P rows) per page each.
    const bool is_v = warp == 0;
    const int ppt = T / a.P;  // pages per tile: 1, 2 or 4
    const int tpc = 32 / ppt;  // tiles per page-id chunk
    auto checked = [&](int raw) {
      if (raw == kNoPage) return -1;  // zero fill
      if (raw < 0 || raw >= a.num_pages) {
        flag_status(a.status, DFLASH_STATUS_BAD_PAGE);
        return -1;
      }
      return raw;
    };
    int pg_cur = checked(chunk_page(a, PB, Lc, start, end, 0, lane, ppt));
    int pg_nxt = chunk_page(a, PB, Lc, start, end, 1, lane, ppt);
    // After a K/V append launched just before (programmatic dependent
    // launch), the pages are read only once that kernel has finished.
    pdl_wait_primary();
    int cur_k = 0;
    Seg sg = seg_first(PB, a.B, a.Hkv, start, end);
    // K/V rows are read once: evict them first, so that the partial states
    // (read back by the combine kernel), queries and page table stay in L2.
    const uint64_t kv_policy = l2_policy_evict_first();
    const int n_issue = a.withhold_loads ? 0 : n;  // tests of the failure path
    // Two-issuer path: the first V tile is needed a softmax after the first
    // K tile, so the V producer starts once that K tile has landed; the
    // opening burst of every CTA then carries its query and K tiles only
    // (measured 1-2 us faster on the 16/1-head and 64/4-head shapes).
    if (DUAL && is_v && n_issue > 0 && !mbar_wait_warp(k_full(0), 0)) {
      if (lane == 0) flag_status(a.status, DFLASH_STATUS_TIMEOUT);
      *abort_flag = 1;
    }
    for (int j = 0; j < n_issue; ++j) {
      while (j >= sg.j1) seg_next(sg, PB, a.Hkv, start, end);
      if (DUAL && !is_v && j == sg.j0) {
        // Two-issuer path: the K producer loads each segment's query tile,
        // once both groups have released the previous one.  Box (64
        // columns, G heads, K tokens) lands as rows r = i*G + g with the
        // 128-byte swizzle, one box per 64-column half.
        if (lane == 0) {
          if (sg.idx > 0 &&
              (!mbar_wait(q_free, (sg.idx - 1) & 1) || !mbar_wait(q_free1, (sg.idx - 1) & 1))) {
            flag_status(a.status, DFLASH_STATUS_TIMEOUT);
            *abort_flag = 1;
          } else {
            mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(a.R * D * 2));
#pragma unroll
            for (int x = 0; x < D / 64; ++x)
              tma_load_3d(sQ + x * 128 * 128, &tm_q, x * 64, sg.h * a.G, sg.b * a.K, q_full);
            *issued_q = sg.idx + 1;
          }
        }
        __syncwarp();
        if (*abort_flag != 0) break;
      }
      const int k = j / tpc;
      if (k != cur_k) {
        // The next chunk's table loads were issued a chunk ago.
        pg_cur = checked(pg_nxt);
        pg_nxt = chunk_page(a, PB, Lc, start, end, k + 1, lane, ppt);
        cur_k = k;
      }
      const int lane0 = (j - k * tpc) * ppt;
      int pages[4];
#pragma unroll
      for (int pj = 0; pj < 4; ++pj)
        pages[pj] = __shfl_sync(0xffffffffu, pg_cur, lane0 + (pj < ppt ? pj : 0));
#pragma unroll
      for (int rr = 0; rr < (FP8 ? 2 : 1); ++rr) {
        const bool v_ring = FP8 ? rr == 1 : is_v;
        const int ns = v_ring ? NSV : NSK;
        const int st = j % ns;
        const uint32_t empty = v_ring ? v_empty(st) : k_empty(st);
        const uint32_t full = v_ring ? v_full(st) : k_full(st);
        if (j >= ns && !mbar_wait_warp(empty, ((j / ns) - 1) & 1)) {
          if (lane == 0) flag_status(a.status, DFLASH_STATUS_TIMEOUT);
          *abort_flag = 1;
        }
        if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        if (lane == 0) {
          const uint32_t dst = (v_ring ? sV : sK) + st * C::kTileBytes;
          const CUtensorMap* map = v_ring ? &tm_v : &tm_k;
          if constexpr (FP8) {
            mbar_arrive_expect_tx(full, T * D);
#pragma unroll
            for (int pj = 0; pj < 4; ++pj) {
              if (pj >= ppt) break;
              tma_load_4d_hint(dst + C::kCodeOff + pj * a.P * D, map, 0, 0, sg.h, pages[pj], full, kv_policy);
            }
          } else {
            mbar_arrive_expect_tx(full, C::kTileBytes);
#pragma unroll
            for (int pj = 0; pj < 4; ++pj) {
              if (pj >= ppt) break;
#pragma unroll
              for (int x = 0; x < D / 64; ++x)
                tma_load_4d_hint(dst + x * T * 128 + pj * a.P * 128, map, x * 64, 0, sg.h, pages[pj], full,
                                 kv_policy);
            }
          }
          *(v_ring ? issued_v : issued_k) = j + 1;
        }
        __syncwarp();
      }
      if (*abort_flag != 0) break;
    }
  } else if (DUAL && (warp == 1 || warp == 11)) {
    // ------------------------------------------------------------ MMA issuers, one per group
    if (lane == 0 && !tc_issue_group<D>(warp == 1 ? 0 : 1, n, start, end, PB, a, tmem, base, abort_flag)) {
      flag_status(a.status, DFLASH_STATUS_TIMEOUT);
      *abort_flag = 1;
    }
  } else if (warp == 11) {
    // ------------------------------------------------------------ query loader
    // Lane 0 issues each segment's query boxes.  In the dense-suffix form the
    // whole warp also writes the block's K rows into the K tiles that hold
    // them, once they have landed, and arrives on k_fix (the MMA waits for it
    // on those tiles); the block rows are pulled into L2 a segment ahead.
    Seg sg = seg_first(PB, a.B, a.Hkv, start, end);
    uint32_t fixes = 0;  // per K slot: block-row fixes done (8 bits each)
    constexpr int kKPieces = (kMaxBlock * (D / 8) + 31) / 32;
    uint4 kreg[kKPieces];
    if (dense) prefetch_suffix_rows(a, sg.b, sg.h, lane, 32);
    for (;;) {
      int stop = 0;
      if (lane == 0) {
        if (sg.idx > 0 && !mbar_wait(q_free, (sg.idx - 1) & 1)) {
          flag_status(a.status, DFLASH_STATUS_TIMEOUT);
          *abort_flag = 1;
        }
        stop = *abort_flag;
        if (!stop) {
          // Box (64 columns, G heads, K tokens) lands as rows r = i*G + g with
          // the 128-byte swizzle, one box per 64-column half.
          mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(a.R * D * 2));
#pragma unroll
          for (int x = 0; x < D / 64; ++x)
            tma_load_3d(sQ + x * 128 * 128, &tm_q, x * 64, sg.h * a.G, sg.b * a.K, q_full);
          *issued_q = sg.idx + 1;
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) break;
      if constexpr (FP8) {
        // The odd K tiles of the segment (the even ones are warp 10's).
        const Geometry geo = make_geometry(Lc[sg.b], a.max_ctx_len, a.K, a.W, T, 1);
        const int pos_base = (geo.t_begin - (sg.g0 - start)) * T;
        for (int j = sg.j0 | 1; j < sg.j1; j += 2) {
          const int st = j % NSK;
          if (!fp8_fix_k<D, T>(a, gbase + C::kOffK + st * C::kTileBytes, k_full(st), (j / NSK) & 1, k_fix(st),
                               pos_base + j * T, geo.L, sg.b, sg.h, lane)) {
            if (lane == 0) flag_status(a.status, DFLASH_STATUS_TIMEOUT);
            *abort_flag = 1;
            stop = 1;
            break;
          }
        }
        if (stop) break;
      } else if (dense) {
        const Geometry geo = make_geometry(Lc[sg.b], a.max_ctx_len, a.K, a.W, T, 1);
        const int pos_base = (geo.t_begin - (sg.g0 - start)) * T;
        bool loaded = false;
        for (int j = sg.j0; j < sg.j1 && !stop; ++j) {
          const int p0 = pos_base + j * T;
          if (p0 + T <= geo.L || p0 >= geo.L + a.K) continue;
          if (!loaded) {  // the block's K rows, read while the tile is in flight
            load_suffix_pieces<D, kKPieces>(kreg, a.k_block, a, sg.b, sg.h, lane, 32);
            loaded = true;
          }
          const int st = j % NSK;
          if (!mbar_wait_warp(k_full(st), (j / NSK) & 1)) {
            if (lane == 0) flag_status(a.status, DFLASH_STATUS_TIMEOUT);
            *abort_flag = 1;
            stop = 1;
            break;
          }
          write_suffix_pieces<D, T, kKPieces>(gbase + C::kOffK + st * C::kTileBytes, kreg, a, geo.L, p0,
                                              lane, 32);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(k_fix(st));
          fixes += 1u << (8 * st);
        }
        if (stop) break;
      }
      if (sg.j1 >= n) break;
      seg_next(sg, PB, a.Hkv, start, end);
      if (lane == 0) {
#pragma unroll
        for (int x = 0; x < D / 64; ++x) tma_prefetch_3d(&tm_q, x * 64, sg.h * a.G, sg.b * a.K);
      }
      if (dense) prefetch_suffix_rows(a, sg.b, sg.h, lane, 32);
    }
    (void)fixes;
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, T, false);
      // fp8 context: P and the widened V tiles are f16.
      constexpr uint32_t idesc_pv = FP8 ? idesc_f16_f32(128, D, true) : idesc_bf16_f32(128, D, true);
      // Descriptors differ only in the start-address field (bits 0..13,
      // address >> 4): build each base once and add offsets >> 4.
      const uint64_t dq = smem_desc_sw128(sQ, 16, 1024);
      const uint64_t dk = smem_desc_sw128(sK, 16, 1024);
      const uint64_t dv = smem_desc_sw128(sV, T * 128, 1024);
      // The ones operand: B of N = 16 rows x K = 16, K-major without
      // swizzle, its four core matrices at 0, 128 (next K), 256 (next N).
      const uint64_t d_ones = smem_desc_noswz(base + C::kOffOnes, 128, 256);
      constexpr uint32_t idesc_l = FP8 ? idesc_f16_f32(128, 16, false) : idesc_bf16_f32(128, 16, false);
      Seg sg = seg_first(PB, a.B, a.Hkv, start, end);
      int q_seg = -1;            // segment whose query tile has been waited for
      int seg_prev = 0;          // segment of tile j-1
      int pv_seg[2] = {-1, -1};  // segment of each group's latest PV
      int last_qk = -1, last_pv = -1;
      uint32_t fixes = 0;  // per K slot: block-row fixes waited for (8 bits each)
      // S_j = Q K_j^T into TMEM S buffer j%2.
      auto issue_qk = [&](int j, int seg_j) -> bool {
        const int st = j % NSK;
        if (q_seg != seg_j) {
          if (!mbar_wait(q_full, seg_j & 1)) return false;
          q_seg = seg_j;
        }
        if (!mbar_wait(k_full(st), (j / NSK) & 1)) return false;
        if (FP8) {
          // Every tile is widened (warp 10 or 11) before its QK^T.
          if (!mbar_wait(k_fix(st), (j / NSK) & 1)) return false;
        } else if (dense) {
          // A tile holding block positions waits for its block rows.
          const Geometry geo = make_geometry(Lc[sg.b], a.max_ctx_len, a.K, a.W, T, 1);
          const int p0 = (geo.t_begin - (sg.g0 - start)) * T + j * T;
          if (p0 + T > geo.L && p0 < geo.L + a.K) {
            if (!mbar_wait(k_fix(st), (fixes >> (8 * st)) & 1)) return false;
            fixes += 1u << (8 * st);
          }
        }
        if (j >= 2 && !mbar_wait(s_free(j & 1), ((j >> 1) - 1) & 1)) return false;
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
        // The query tile may be replaced once the segment's last QK^T is done.
        if (j == sg.j1 - 1 && sg.j1 < n) umma_commit(q_free);
        last_qk = j;
        return true;
      };
      // O_g += P_j V_j, g = j%2, for tile jj of segment seg_prev.  The first
      // PV of a group in a segment overwrites O_g: its P arrives only after
      // every softmax thread has read the previous segment's accumulators.
      auto issue_pv = [&](int jj) -> bool {
        const int st = jj % NSV;
        const int g = jj & 1;
        const bool fresh = pv_seg[g] != seg_prev;
        if (!mbar_wait(p_full(g), (jj >> 1) & 1)) return false;
        if (!mbar_wait(v_full(st), (jj / NSV) & 1)) return false;
        tc_fence_after();
        pv_seg[g] = seg_prev;
        const uint32_t v_off = st * C::kTileBytes;
        const uint32_t o_col = g ? C::kColO1 : C::kColO0;
#pragma unroll
        for (int kk = 0; kk < T / 16; ++kk)
          umma_bf16_ts(tmem + o_col, tmem + C::kColP + g * (T / 2) + kk * 8,
                       dv + ((v_off + kk * 16 * 128) >> 4), idesc_pv, (!fresh || kk > 0) ? 1u : 0u);
        // L_g += P_j 1: the row sums of the rounded probabilities.
#pragma unroll
        for (int kk = 0; kk < T / 16; ++kk)
          umma_bf16_ts(tmem + C::kColL + g * 16, tmem + C::kColP + g * (T / 2) + kk * 8, d_ones, idesc_l,
                       (!fresh || kk > 0) ? 1u : 0u);
        umma_commit(v_empty(st));
        umma_commit(pv_done(g));
        last_pv = jj;
        return true;
      };
      for (int j = 0; j <= n; ++j) {
        if (*abort_flag) break;
        int seg_j = seg_prev;
        if (j < n) {
          while (j >= sg.j1) seg_next(sg, PB, a.Hkv, start, end);
          seg_j = sg.idx;
        }
        // QK^T runs one tile ahead of PV, except across a segment boundary:
        // there the previous segment's last PV goes first, so that segment's
        // output does not wait for the next query tile.
        const bool boundary = j < n && j > 0 && seg_j != seg_prev;
        bool ok = true;
        if (boundary) ok = issue_pv(j - 1);
        if (ok && j < n) ok = issue_qk(j, seg_j);
        if (ok && !boundary && j >= 1) ok = issue_pv(j - 1);
        if (!ok) {
          flag_status(a.status, DFLASH_STATUS_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        seg_prev = seg_j;
      }
      // Let the last commits land before the CTA winds down.
      for (int jj = last_qk - NSK + 1; jj <= last_qk; ++jj)
        if (jj >= 0) (void)mbar_wait(k_empty(jj % NSK), (jj / NSK) & 1);
      for (int jj = last_pv - NSV + 1; jj <= last_pv; ++jj)
        if (jj >= 0) (void)mbar_wait(v_empty(jj % NSV), (jj / NSV) & 1);
    }
  } else if (warp >= 2 && warp <= 9) {
    // ------------------------------------------------------------ softmax (warps 2..9)
    const int sw = warp - 2;          // 0..7
    const int grp = sw >> 2;          // tiles j = grp, grp+2, ...
    const int quad = warp & 3;        // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;
    const int gthread = (sw & 3) * 32 + lane;  // 0..127 within the group
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t o_col = grp ? C::kColO1 : C::kColO0;
    const int i_row = row < a.R ? row / a.G : 0;
    bool ok = true;
    Seg sg = seg_first(PB, a.B, a.Hkv, start, end);
    for (;;) {
      const Geometry geo = make_geometry(Lc[sg.b], a.max_ctx_len, a.K, a.W, T, 1);
      const int L = geo.L;
      int lo_r = 0x7fffffff, hi_r = -0x7fffffff;
      if (row < a.R) {
        lo_r = 0;
        if (a.W > 0) {
          lo_r = L + i_row - a.W + 1;
          if (lo_r < 0) lo_r = 0;
        }
        hi_r = L + min(a.K, i_row + 1 + a.rw);
      }
      int lo_rows_max = 0;
      if (a.W > 0) {
        lo_rows_max = L + a.K - a.W;
        if (lo_rows_max < 0) lo_rows_max = 0;
      }
      const int hi_rows_min = L + min(a.K, 1 + a.rw);
      const int pos_base = (geo.t_begin - (sg.g0 - start)) * T;  // position of CTA tile 0, this pair

      float m_ref = ninf();
      float l_run = 0.f;
      int last_j = -1;  // this group's latest tile in the segment
      const int jfirst = sg.j0 + (((sg.j0 & 1) != grp) ? 1 : 0);
      for (int j = jfirst; ok && j < sg.j1; j += 2) {
        // Dense-suffix form: a tile holding block positions takes its value
        // rows from the dense tensor; the loads are issued before the score
        // wait so they land meanwhile.
        constexpr int kVPieces = (kMaxBlock * (D / 8) + 127) / 128;
        const bool v_suffix = dense && pos_base + (j + 1) * T > L && pos_base + j * T < L + a.K;
        if (v_suffix)
          stage_suffix_async<D, kVPieces>(base + C::kOffVStage + grp * C::kVStageBytes, a.v_block, a,
                                          sg.b, sg.h, gthread, 128);
        if constexpr (FP8) {
          // Widen this tile's value codes in place before the score wait (the
          // codes land with the keys'; the PV product needs them only after
          // this group's P): rows at positions in [lo_min, L) widened, rows
          // outside [lo_min, L+K) zeroed, block rows written after the P
          // store.  D = 64: every thread reads its codes before any writes,
          // joining on v_read (a bounded wait).
          const int p0v = pos_base + j * T;
          const int st = j % NSV;
          uint8_t* vtile = gbase + C::kOffV + st * C::kTileBytes;
          const bool vok = mbar_wait_warp(v_full(st), (j / NSV) & 1);
          if constexpr (D == 128) {
            if (vok) widen_v_row<T>(vtile, gthread, p0v, geo.lo_min, L);
          } else {
            uint4 vraw[D / 32];
            if (vok) read_v_codes<D, T>(vtile, gthread, vraw);
            __syncwarp();
            if (lane == 0) mbar_arrive(v_read(grp));
            const bool rok = mbar_wait_warp(v_read(grp), (j >> 1) & 1);
            if (!vok || !rok) { ok = false; break; }
            write_v_widened<D, T>(vtile, gthread, p0v, geo.lo_min, L, vraw);
          }
          if (!vok) { ok = false; break; }
          if (gthread < T) {  // D = 128: not the threads that widen
            const int zr = gthread;
            const int pos = p0v + zr;
            if (pos < geo.lo_min || pos >= geo.hi_max) {
              uint8_t* vrow = vtile + zr * 128;
#pragma unroll
              for (int x2 = 0; x2 < D / 64; ++x2)
#pragma unroll
                for (int c = 0; c < 8; ++c)
                  *reinterpret_cast<uint4*>(vrow + x2 * T * 128 + c * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
          }
        }
        if (!mbar_wait_warp(s_full(grp), (j >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld64_wait(lane_addr + grp * T, sr);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free(grp));

        const int p0 = pos_base + j * T;
        // fp8 context: a tile holding block keys is a boundary tile too.
        const bool blk_cols = FP8 && p0 + T > L;
        const bool need_mask = (p0 < lo_rows_max) || (p0 + T > hi_rows_min) || blk_cols;
        // Row max of the raw scores (the scale is positive), four independent
        // chains; masked keys become -inf by select.  Boundary tiles only.
        // With fp8 context the scale includes k_scale, so a block key's score
        // (bf16 key, no scale) is divided by k_scale first.
        float mx[4] = {ninf(), ninf(), ninf(), ninf()};
        if (need_mask) {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int pos = p0 + c;
            float v = __uint_as_float(sr[c]);
            if (FP8 && pos >= L) v *= a.kblk_mul;
            v = (pos >= lo_r && pos < hi_r) ? v : ninf();
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
        // Selects, not a branch: rows of a warp disagree on moving.
        const bool resc = mt > m_ref + 8.f;
        const float cr = (m_ref == ninf()) ? 0.f : fast_exp2(m_ref - mt);
        const float corr = resc ? cr : 1.f;
        l_run *= corr;
        m_ref = resc ? mt : m_ref;
        float neg_m = (m_ref == ninf()) ? 0.f : -m_ref;
        if constexpr (FP8) neg_m += 7.f;  // f16 P: p * 2^7 <= 2^15
        float sm[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float pa = fast_exp2(fmaf(__uint_as_float(sr[2 * c]), a.scale_log2, neg_m));
          const float pb = fast_exp2(fmaf(__uint_as_float(sr[2 * c + 1]), a.scale_log2, neg_m));
          sm[c & 3] += pa + pb;
          pk[c] = FP8 ? pack_f16x2(pa, pb) : pack_bf16x2(pa, pb);
        }
        l_run += (sm[0] + sm[1]) + (sm[2] + sm[3]);

        // This group's P columns and O_g are free once its previous PV (tile
        // j-2, possibly of the previous segment) has completed.  O_g holds
        // this segment's sum only after the group's first tile in it.  The
        // rescale's TMEM load/store are warp-collective: the whole warp runs
        // them when any of its rows moved its reference max (factor 1 for
        // the other rows).
        const bool warp_resc = __any_sync(0xffffffffu, resc);
        if (j >= 2) {
          if (!mbar_wait_warp(pv_done(grp), ((j >> 1) - 1) & 1)) { ok = false; break; }
          tc_fence_after();
          if (warp_resc && last_j >= 0) {
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t o[32];
              tmem_ld32_wait(lane_addr + o_col + cc * 32, o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
              tmem_st32(lane_addr + o_col + cc * 32, o);
            }
            uint32_t lv[16];
            tmem_ld16_wait(lane_addr + C::kColL + grp * 16, lv);
#pragma unroll
            for (int e = 0; e < 16; ++e) lv[e] = __float_as_uint(__uint_as_float(lv[e]) * corr);
            tmem_st16(lane_addr + C::kColL + grp * 16, lv);
            tmem_wait_st();
          }
        }
        auto v_fix = [&]() -> bool {
          // Value rows outside [lo_min, L+K) may hold anything: zero them in the
          // stage before the PV MMA reads it (boundary tiles only).  In the
          // dense-suffix form the block's value rows are written here too.
          if constexpr (FP8) {
            // Widened and zeroed before the score wait: the block rows remain,
            // divided by v_scale.
            if (v_suffix)
              write_staged_suffix_scaled<D, T, kVPieces>(gbase + C::kOffV + (j % NSV) * C::kTileBytes,
                                                         gbase + C::kOffVStage + grp * C::kVStageBytes, a, L,
                                                         p0, gthread, 128, a.pblk_mul);
            return true;
          }
          if (p0 < geo.lo_min || p0 + T > geo.hi_max || v_suffix) {
            const int st = j % NSV;
            if (!mbar_wait_warp(v_full(st), (j / NSV) & 1)) return false;
            if (v_suffix)
              write_staged_suffix<D, T, kVPieces>(gbase + C::kOffV + st * C::kTileBytes,
                                                  gbase + C::kOffVStage + grp * C::kVStageBytes, a, L, p0,
                                                  gthread, 128);
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
          return true;
        };
        // P row -> this group's TMEM P columns (key pairs per column).  With
        // fp8 context the block's value rows are written after the P store
        // (fewer registers live across the cp.async wait).
        if (!FP8 && !v_fix()) { ok = false; break; }
        tmem_st32(lane_addr + C::kColP + grp * (T / 2), pk);
        tmem_wait_st();
        if (FP8 && !v_fix()) { ok = false; break; }
        fence_proxy_async_smem();  // the zeroed V rows, for the MMA
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(grp));
        last_j = j;
      }

      // ---- end of segment.  Each group publishes its row state once its last
      // PV of the segment is done; then both merge the two states, group g
      // for output columns [g*D/2, (g+1)*D/2).  Named barrier 3 joins the
      // eight softmax warps; the stop decision is read between two barriers
      // so that every softmax thread takes it alike.
      if (ok && last_j >= 0 && !mbar_wait_warp(pv_done(grp), (last_j >> 1) & 1)) ok = false;
      xchg[grp * 128 + row] = make_float2(m_ref, l_run);
      if (!ok) *stop_word = 1;
      tc_fence_before();
      named_barrier(3, 256);
      const bool stop = *stop_word != 0;
      const bool direct = sg.g0 >= start && sg.g0 + sg.nb <= end;
      const size_t orow = row < a.R ? out_row_index(a, sg.b, sg.h, row) : 0;
      // A cut pair's partial goes to slot 0 (the range's first segment) or
      // slot 1 (its last), for the combine kernel.
      const size_t unit = static_cast<size_t>(blockIdx.x) * 2 + (sg.idx == 0 ? 0 : 1);
      if (!stop) {
        tc_fence_after();
        const float2 s0 = xchg[row];
        const float2 s1 = xchg[128 + row];
        const float M = fmaxf(s0.x, s1.x);
        const float w0 = (s0.x == ninf() || s0.y == 0.f) ? 0.f : fast_exp2(s0.x - M);
        const float w1 = (s1.x == ninf() || s1.y == 0.f) ? 0.f : fast_exp2(s1.x - M);
        const float l = w0 * s0.y + w1 * s1.y;
        // The output is divided by the sum of the probabilities as rounded for
        // the P.V product (the MMA against the ones operand), so the rounding
        // of a dominant probability cancels; the LSE keeps the exact sum.  A
        // group with no key in the segment holds a stale sum: select.
        float lr = 0.f;
        {
          uint32_t r0[16], r1[16];
          tmem_ld16x2_wait(lane_addr + C::kColL, lane_addr + C::kColL + 16, r0, r1);
          lr = (w0 > 0.f ? w0 * __uint_as_float(r0[0]) : 0.f) + (w1 > 0.f ? w1 * __uint_as_float(r1[0]) : 0.f);
        }
        const float inv = lr > 0.f ? a.out_mul / lr : 0.f;
        // D = 128: group g writes columns [64g, 64g + 64); D = 64: group 0 all.
        if (grp * 64 < D)
          store_segment_rows<D>(a, &tm_out, &tm_part, gbase + C::kOffStage + grp * C::kStageBytes,
                                sStage + grp * C::kStageBytes, lane_addr, grp * 64, grp, row, gthread == 0, w0, w1,
                                inv, direct, sg.b, sg.h, static_cast<int>(unit));
        if (row < a.R && grp == 0) {
          const float lse = l > 0.f ? M + (FP8 ? log2f(l) - 7.f : log2f(l)) : ninf();
          if (direct) {
            a.lse2[orow] = lse;
          } else {
            a.part_lse[unit * a.R + row] = lse;
            a.part_lseo[unit * a.R + row] = lr > 0.f ? M + (FP8 ? log2f(lr) - 7.f : log2f(lr)) : ninf();
          }
        }
      }
      // Every softmax thread has read stop_word, the states and both
      // accumulators before any goes on (the next segment's first P, which
      // lets the MMA overwrite an accumulator, comes after this barrier).
      tc_fence_before();
      named_barrier(3, 256);
      if (stop) {
        if (lane == 0) flag_status(a.status, DFLASH_STATUS_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      if (sg.j1 >= n) break;
      seg_next(sg, PB, a.Hkv, start, end);
    }
    if (gthread == 0) bulk_wait_all();  // this group's output boxes are written
    asm volatile("cp.async.wait_all;" ::: "memory");  // no block-row copy left in flight
    tc_fence_before();
  }

  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    const int ik = *issued_k, iv = *issued_v, iq = *issued_q;
    for (int j = ik > NSK ? ik - NSK : 0; j < ik; ++j) (void)mbar_wait(k_full(j % NSK), (j / NSK) & 1);
    for (int j = iv > NSV ? iv - NSV : 0; j < iv; ++j) (void)mbar_wait(v_full(j % NSV), (j / NSV) & 1);
    if (iq > 0) (void)mbar_wait(q_full, (iq - 1) & 1);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool FP8>
int launch_t(const AttnArgs& a, const KernelPlan& plan, const CUtensorMap& tm_k,
             const CUtensorMap& tm_v, const CUtensorMap& tm_q, const CUtensorMap& tm_out,
             const CUtensorMap& tm_part, cudaStream_t stream) {
  // bf16 pages without a dense suffix: one MMA issuer per softmax group
  // (the other forms keep warp 11 for their query loads, K fixes or
  // widening, and one issuer).
  const bool dual = !FP8 && a.k_block == nullptr;
  auto kern = dual ? split_tc_kernel<D, FP8, !FP8> : split_tc_kernel<D, FP8, false>;
  const int smem = dual ? TcCfg<D, true>::kSmem : TcCfg<D, false>::kSmem;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  return launch_kernel(kern, dim3(static_cast<unsigned>(plan.units)), dim3(TcCfg<D>::kThreads), smem, stream,
                       plan.pdl, a, tm_k, tm_v, tm_q, tm_out, tm_part);
}

}  // namespace

bool split_tc_available() { return true; }
int split_tc_tile_keys(int) { return 64; }
int split_tc_threads() { return TcCfg<128>::kThreads; }
int split_tc_smem_bytes(int D) { return D == 64 ? TcCfg<64>::kSmem : TcCfg<128>::kSmem; }

int launch_split_tc(const AttnArgs& a, const KernelPlan& plan, const CUtensorMap& tm_k,
                    const CUtensorMap& tm_v, const CUtensorMap& tm_q, const CUtensorMap& tm_out,
                    const CUtensorMap& tm_part, cudaStream_t stream) {
  if (a.fp8) {
    if (a.k_block == nullptr) return cudaErrorInvalidValue;  // fp8 pages hold the context only
    if (a.D == 64) return launch_t<64, true>(a, plan, tm_k, tm_v, tm_q, tm_out, tm_part, stream);
    if (a.D == 128) return launch_t<128, true>(a, plan, tm_k, tm_v, tm_q, tm_out, tm_part, stream);
    return cudaErrorInvalidValue;
  }
  if (a.D == 64) return launch_t<64, false>(a, plan, tm_k, tm_v, tm_q, tm_out, tm_part, stream);
  if (a.D == 128) return launch_t<128, false>(a, plan, tm_k, tm_v, tm_q, tm_out, tm_part, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dflash
