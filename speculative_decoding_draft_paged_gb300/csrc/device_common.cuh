// Device helpers: mbarriers with bounded waits, TMA tile loads, warp-level
// MMA fragments, bf16 packing.  Hand-written PTX for sm_103a.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dflash_internal.h"

namespace dflash {

// A pipeline wait that has not completed after this long is treated as a
// failure: the kernel records DFLASH_STATUS_TIMEOUT and winds down.
constexpr unsigned long long kWaitTimeoutNs = 4000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false if it
// has not completed within kWaitTimeoutNs (never expected in a correct run).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitTimeoutNs) return false;
  }
  return true;
}

// Warp-uniform form of mbar_wait for code that continues with warp-collective
// instructions: lane 0 waits with the bound, every lane gets its verdict, and
// on success each lane observes the completed phase itself (acquire).  The
// caller guarantees the barrier cannot complete a further phase meanwhile.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  if (ok) (void)mbar_wait(bar, parity);
  return ok;
}

// 4-D tiled TMA load (box of the tensor map) into shared memory, completing
// transaction bytes on `bar`.  Coordinates: (x = dim, y = slot, z = head, w = page).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

// The same with an L2 cache policy (createpolicy), e.g. evict-first for data
// read exactly once.
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 int z, int w, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// TMA store of a shared-memory box to a 3-D tensor map (bulk async group of
// the issuing thread), and the waits on that thread's groups.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The shared-memory sources of every committed group have been read.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Every committed group has completed (its global writes are done).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Pull the 128-byte line holding `p` into L2.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

// The same by reading one word of the line (the value is not used; the
// thread does not wait for it).  For the page-table rows the producers read
// a few microseconds later this measured faster than prefetch_l2: the rows
// were then in L2 when read.
__device__ __forceinline__ void touch_l2(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(v) : "l"(p));
}

// Pull a box of a 3-D tensor map into L2 (no shared-memory destination).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Generic-proxy shared-memory writes -> visible to the async proxy (MMA, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier over `count` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D += A * B, m16n8k16, f16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Packs two fp32 values into an f16x2 word (round to nearest even).
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Packs two fp32 values into a bf16x2 word (round to nearest even); `lo` in
// the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Byte offset of 16-byte chunk `chunk` (0..D/8-1) of row `row` in a tile
// stored the way a 128-byte-swizzled TMA box lays it out: the row's 64-column
// half is a separate [rows x 128 B] block, and chunk c of row r within the
// block sits at r*128 + ((c ^ (r & 7)) * 16).
__device__ __forceinline__ uint32_t swz_offset(int row, int chunk, int rows_per_half) {
  const int half = chunk >> 3;
  const int c = chunk & 7;
  return static_cast<uint32_t>(half * rows_per_half * 128 + row * 128 + ((c ^ (row & 7)) << 4));
}

__device__ __forceinline__ void flag_status(uint32_t* status, uint32_t bits) {
  atomicOr(status, bits);
}

// Page ids of the unit's page-table slots [slot_first, slot_first + n_slots),
// looked up by threads tid, tid + nthreads, ... into shared memory before the
// pipeline starts, so the TMA producer never waits on a table read.  Slots
// outside [slot_lo, slot_hi) (not visible to any row) and out-of-range ids
// become -1, which the TMA unit turns into a zero-filled box.
__device__ __forceinline__ void load_unit_pages(const AttnArgs& a, int b, int slot_first,
                                                int n_slots, int slot_lo, int slot_hi,
                                                int* pg_smem, int tid, int nthreads) {
  const int32_t* table_row = a.page_table + static_cast<size_t>(b) * a.max_pages;
  for (int k = tid; k < n_slots; k += nthreads) {
    const int slot = slot_first + k;
    int page = -1;
    if (slot >= slot_lo && slot < slot_hi) {
      page = __ldg(&table_row[slot]);
      if (page < 0 || page >= a.num_pages) {
        flag_status(a.status, DFLASH_STATUS_BAD_PAGE);
        page = -1;
      }
    }
    pg_smem[k] = page;
  }
}

// Index of packed row r = i*G + g of kv head h of request b in the output
// layout [B, K, Hq] (times D for `out`).
__device__ __forceinline__ size_t out_row_index(const AttnArgs& a, int b, int h, int r) {
  const int i = r / a.G;
  const int g = r - i * a.G;
  return (static_cast<size_t>(b) * a.K + i) * a.Hq + static_cast<size_t>(h) * a.G + g;
}

// ---- flat split of the tcgen05 kernel (shared with the combine kernel, so
// both derive the same CTA ranges from the lengths).
constexpr int kFlatTileKeys = 64;

// PB[b] = sum over requests b' < b of their 64-key tile counts, b in [0, B];
// Lc[b] = context length clamped to [0, max_ctx_len].  Called by all NT
// threads of the block (NT a multiple of 32, at most 1024); warp_sums is
// shared scratch of NT/32 ints.  Ends with __syncthreads.
template <int NT>
__device__ __forceinline__ void flat_tile_prefix(const AttnArgs& a, int* PB, int* Lc, int* warp_sums,
                                                 bool flag_bad) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ipt = (a.B + NT - 1) / NT;
  const int b_lo = threadIdx.x * ipt;
  const int b_hi = min(b_lo + ipt, a.B);
  int sum = 0;
  for (int bb = b_lo; bb < b_hi; ++bb) {
    const int L_raw = __ldg(&a.ctx_lens[bb]);
    if (flag_bad && (L_raw < 0 || L_raw > a.max_ctx_len)) flag_status(a.status, DFLASH_STATUS_BAD_CTX_LEN);
    const Geometry g = make_geometry(L_raw, a.max_ctx_len, a.K, a.W, kFlatTileKeys, 1);
    Lc[bb] = g.L;
    sum += g.n_tiles;
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int ws = lane < NT / 32 ? warp_sums[lane] : 0;
    int wi = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < NT / 32) warp_sums[lane] = wi - ws;  // exclusive over warps
  }
  __syncthreads();
  int run = warp_sums[warp] + incl - sum;
  for (int bb = b_lo; bb < b_hi; ++bb) {
    PB[bb] = run;
    run += make_geometry(Lc[bb], a.max_ctx_len, a.K, a.W, kFlatTileKeys, 1).n_tiles;
  }
  if (b_lo < b_hi && b_hi == a.B) PB[a.B] = run;
  __syncthreads();
}

// CTA ranges of the flat split.  Pair p = b*Hkv + h has nb = PB[b+1] - PB[b]
// tiles; in "cost" units its tiles sit at C_p .. C_p + nb - 1 with
// C_p = Hkv*PB[b] + h*nb + w*p, followed by w units standing for the epilogue
// that ends the pair's segment.  CTA c takes the tiles whose cost position
// lies in [c*q, (c+1)*q), so a range that holds more pair ends holds fewer
// tiles.  w = 0 and q = a forced length when force_split_tiles is set.
struct FlatMap {
  int q;      // cost units per CTA range
  int w;      // cost units per pair end
  int total;  // tiles of all pairs
};

// a / b for 0 <= a and 0 < b, in 32 bits when both fit (the 64-bit division
// is a long instruction sequence).
__device__ __forceinline__ long long div_nonneg(long long a, long long b) {
  if (((a | b) >> 31) == 0) return static_cast<unsigned>(a) / static_cast<unsigned>(b);
  return a / b;
}

// The map from the tiles of all requests (tiles_all = PB[B]).
__device__ __forceinline__ FlatMap flat_map_total(const AttnArgs& a, int tiles_all) {
  FlatMap m;
  m.total = a.Hkv * tiles_all;
  if (a.qn_force > 0) {
    m.q = a.qn_force;
    m.w = 0;
    return m;
  }
  m.w = a.seg_cost;
  const long long cost = static_cast<long long>(m.total) + static_cast<long long>(m.w) * a.B * a.Hkv;
  long long q = div_nonneg(cost + a.ncta - 1, a.ncta);
  if (q < a.qn_min) q = a.qn_min;
  m.q = static_cast<int>(q);
  return m;
}

__device__ __forceinline__ FlatMap flat_map(const AttnArgs& a, const int* PB) { return flat_map_total(a, PB[a.B]); }

// Cost position of the first tile of pair (b, h).
__device__ __forceinline__ long long flat_pair_cost(const AttnArgs& a, const int* PB, const FlatMap& m,
                                                    int b, int h) {
  const int nb = PB[b + 1] - PB[b];
  return static_cast<long long>(a.Hkv) * PB[b] + static_cast<long long>(h) * nb +
         static_cast<long long>(m.w) * (static_cast<long long>(b) * a.Hkv + h);
}

// First tile whose cost position is >= x (m.total past the last one).
__device__ __forceinline__ int flat_tile_at(const AttnArgs& a, const int* PB, const FlatMap& m, long long x) {
  if (x <= 0) return 0;
  int lo = 0, hi = a.B - 1;  // last request whose first pair's cost is <= x
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (flat_pair_cost(a, PB, m, mid, 0) <= x) lo = mid; else hi = mid - 1;
  }
  const int nb = PB[lo + 1] - PB[lo];
  const long long rel = x - flat_pair_cost(a, PB, m, lo, 0);
  const long long per = static_cast<long long>(nb) + m.w;
  long long h = rel / per;
  if (h >= a.Hkv) return a.Hkv * PB[lo + 1];
  long long t = rel - h * per;
  if (t > nb) t = nb;
  return a.Hkv * PB[lo] + static_cast<int>(h) * nb + static_cast<int>(t);
}

// Tile range [start, end) of CTA c.
__device__ __forceinline__ void flat_range(const AttnArgs& a, const int* PB, const FlatMap& m, int c,
                                           int& start, int& end) {
  start = flat_tile_at(a, PB, m, static_cast<long long>(c) * m.q);
  end = flat_tile_at(a, PB, m, static_cast<long long>(c + 1) * m.q);
}

// ---- dense-suffix form: the block's K/V rows come from dense tensors and the
// pages hold the context only.

// One past the last position read from the pages.
__device__ __forceinline__ int paged_end(const AttnArgs& a, const Geometry& g) {
  return a.k_block != nullptr ? g.L : g.hi_max;
}

// Writes the block rows at positions [max(L, lo), min(L+K, hi)) of kv head h
// of request b from the dense tensor `src` ([B, K, Hkv, D] bf16) into a
// 128-byte-swizzled tile at `tile` whose row 0 is position p0 and which holds
// T rows per 64-column half (the layout the TMA boxes give).  Threads
// tid = 0..nthr-1 share the 16-byte pieces.
template <int D, int T>
__device__ __forceinline__ void write_suffix_rows(uint8_t* tile, const uint16_t* src, const AttnArgs& a,
                                                  int b, int h, int L, int p0, int lo, int hi, int tid,
                                                  int nthr, float mul = 1.f) {
  constexpr int CPR = D / 8;
  const int r_lo = max(L, lo);
  const int r_hi = min(L + a.K, hi);
  const int n = (r_hi - r_lo) * CPR;
  for (int e = tid; e < n; e += nthr) {
    const int pos = r_lo + e / CPR;
    const int c = e - (e / CPR) * CPR;
    const int rr = pos - p0;
    const uint4* row =
        reinterpret_cast<const uint4*>(src + ((static_cast<size_t>(b) * a.K + (pos - L)) * a.Hkv + h) * D);
    uint4 x = __ldg(row + c);
    if (mul != 1.f) {  // fp8 context: value rows divided by v_scale
      auto sc = [&](uint32_t w) {
        return pack_bf16x2(bf16_bits_to_f32(w & 0xffffu) * mul, bf16_bits_to_f32(w >> 16) * mul);
      };
      x = make_uint4(sc(x.x), sc(x.y), sc(x.z), sc(x.w));
    }
    *reinterpret_cast<uint4*>(tile + (c >> 3) * T * 128 + rr * 128 + (((c & 7) ^ (rr & 7)) << 4)) = x;
  }
}

// The same rows held in registers ahead of time: thread tid of nthr holds the
// 16-byte pieces e = tid + k*nthr (k < MAXP) of the K*D/8 pieces of the block
// (piece e = row e / (D/8), chunk e % (D/8)).  load_suffix_pieces reads them
// early; write_suffix_pieces stores those that fall in a tile starting at p0.
template <int D, int MAXP>
__device__ __forceinline__ void load_suffix_pieces(uint4 (&regs)[MAXP], const uint16_t* src,
                                                   const AttnArgs& a, int b, int h, int tid, int nthr) {
  constexpr int CPR = D / 8;
  const int n = a.K * CPR;
#pragma unroll
  for (int k = 0; k < MAXP; ++k) {
    const int e = tid + k * nthr;
    if (e < n) {
      const int j = e / CPR;
      const int c = e - j * CPR;
      regs[k] = __ldg(reinterpret_cast<const uint4*>(
                          src + ((static_cast<size_t>(b) * a.K + j) * a.Hkv + h) * D) + c);
    }
  }
}

template <int D, int T, int MAXP>
__device__ __forceinline__ void write_suffix_pieces(uint8_t* tile, const uint4 (&regs)[MAXP],
                                                    const AttnArgs& a, int L, int p0, int tid, int nthr) {
  constexpr int CPR = D / 8;
  const int n = a.K * CPR;
#pragma unroll
  for (int k = 0; k < MAXP; ++k) {
    const int e = tid + k * nthr;
    if (e < n) {
      const int j = e / CPR;
      const int c = e - j * CPR;
      const int rr = L + j - p0;
      if (rr >= 0 && rr < T)
        *reinterpret_cast<uint4*>(tile + (c >> 3) * T * 128 + rr * 128 + (((c & 7) ^ (rr & 7)) << 4)) =
            regs[k];
    }
  }
}

// The same pieces copied asynchronously (cp.async, 16 bytes each) into a
// linear staging buffer (piece e at byte 16e), then, after the copying
// thread's cp.async.wait_all, moved into a tile: each thread moves the pieces
// it copied itself, so no other synchronisation is needed.
template <int D, int MAXP>
__device__ __forceinline__ void stage_suffix_async(uint32_t stage, const uint16_t* src, const AttnArgs& a,
                                                   int b, int h, int tid, int nthr) {
  constexpr int CPR = D / 8;
  const int n = a.K * CPR;
#pragma unroll
  for (int k = 0; k < MAXP; ++k) {
    const int e = tid + k * nthr;
    if (e < n) {
      const int j = e / CPR;
      const int c = e - j * CPR;
      const uint16_t* g = src + ((static_cast<size_t>(b) * a.K + j) * a.Hkv + h) * D + c * 8;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(stage + 16u * e), "l"(g) : "memory");
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int D, int T, int MAXP>
__device__ __forceinline__ void write_staged_suffix(uint8_t* tile, const uint8_t* stage, const AttnArgs& a,
                                                    int L, int p0, int tid, int nthr) {
  asm volatile("cp.async.wait_all;" ::: "memory");
  constexpr int CPR = D / 8;
  const int n = a.K * CPR;
#pragma unroll
  for (int k = 0; k < MAXP; ++k) {
    const int e = tid + k * nthr;
    if (e < n) {
      const int j = e / CPR;
      const int c = e - j * CPR;
      const int rr = L + j - p0;
      if (rr >= 0 && rr < T)
        *reinterpret_cast<uint4*>(tile + (c >> 3) * T * 128 + rr * 128 + (((c & 7) ^ (rr & 7)) << 4)) =
            *reinterpret_cast<const uint4*>(stage + 16 * e);
    }
  }
}

// Pulls the block rows of kv head h of request b (K and V) into L2.
__device__ __forceinline__ void prefetch_suffix_rows(const AttnArgs& a, int b, int h, int tid, int nthr) {
  const int lines_per_row = (a.D * 2 + 127) / 128;
  const int n = 2 * a.K * lines_per_row;
  for (int e = tid; e < n; e += nthr) {
    const int kv = e / (a.K * lines_per_row);
    const int rem = e - kv * a.K * lines_per_row;
    const int j = rem / lines_per_row;
    const int l = rem - j * lines_per_row;
    const uint16_t* src = kv ? a.v_block : a.k_block;
    prefetch_l2(reinterpret_cast<const uint8_t*>(src + ((static_cast<size_t>(b) * a.K + j) * a.Hkv + h) * a.D) +
                l * 128);
  }
}

// Programmatic dependent launch controls.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---- fp8 (E4M3) context codes, widened to bf16 in shared memory.

// Four E4M3 codes (first code lowest) -> two f16x2 words, exactly (every
// E4M3 value is an f16 value); the 16-bit halves of the source go to the
// conversions as they are.
__device__ __forceinline__ uint2 e4m3x4_to_f16x4(uint32_t codes) {
  uint2 r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
      : "=r"(r.x), "=r"(r.y)
      : "r"(codes));
  return r;
}

// f16x2 holding E4M3 values -> bf16x2, exactly: f16 -> f32, then the upper
// half of each f32 (at most 4 significant bits, so the lower half is zero).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2_exact(uint32_t h2) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
  return __byte_perm(__float_as_uint(f.x), __float_as_uint(f.y), 0x7632);
}

// Byte offset of 16-byte word w of code row r in a stage's code area: the
// boxes land with the TMA swizzle of their row length (128-byte swizzle for
// D = 128: word w of row r at r*128 + (w ^ (r & 7))*16; 64-byte swizzle for
// D = 64: at r*64 + (w ^ ((r >> 1) & 3))*16), so that a warp reading one
// word per row hits every bank.
template <int D>
__device__ __forceinline__ int code_word(int r, int w) {
  if constexpr (D == 128) return r * 128 + ((w ^ (r & 7)) << 4);
  else return r * 64 + ((w ^ ((r >> 1) & 3)) << 4);
}

// Eight codes (two words) -> one 16-byte chunk of eight bf16 values.
__device__ __forceinline__ uint4 widen8(uint32_t w0, uint32_t w1) {
  const uint2 a = e4m3x4_to_f16x4(w0), b = e4m3x4_to_f16x4(w1);
  return make_uint4(f16x2_to_bf16x2_exact(a.x), f16x2_to_bf16x2_exact(a.y), f16x2_to_bf16x2_exact(b.x),
                    f16x2_to_bf16x2_exact(b.y));
}

// Eight codes (two words) -> one 16-byte chunk of eight f16 values.
__device__ __forceinline__ uint4 widen8_f16(uint32_t w0, uint32_t w1) {
  const uint2 a = e4m3x4_to_f16x4(w0), b = e4m3x4_to_f16x4(w1);
  return make_uint4(a.x, a.y, b.x, b.y);
}

}  // namespace dflash
