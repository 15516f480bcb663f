// C ABI of the paged draft-block attention library (include/dflash.h):
// argument validation, the split planner, workspace sizing, TMA descriptors
// and the launches: a split kernel (mma.sync or tcgen05) and, where a row may
// have several partials, the combine kernel.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "dflash.h"
#include "dflash_internal.h"

namespace dflash {

int split_mma_kpw(int D, int R_pad);
int split_mma_tile_keys(int D);
int split_tc_tile_keys(int D);
int split_tc_threads();
bool split_tc_available();

namespace {

constexpr int kDefaultSms = 152;       // GB300, used when no device can be queried
constexpr int kMaxDevices = 64;
constexpr int kSmemPerSm = 228 * 1024;
constexpr int kMaxSmemPerCta = 227 * 1024;  // dynamic shared memory one CTA may opt into

struct DeviceInfo {
  int sms = 0;
  int cc = 0;  // major * 10 + minor
  bool ok = false;
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];

DeviceInfo current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return DeviceInfo{};
  }
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (!g_dev[dev].ok) {
    int sms = 0, major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return DeviceInfo{};
    }
    g_dev[dev].sms = sms;
    g_dev[dev].cc = major * 10 + minor;
    g_dev[dev].ok = true;
  }
  return g_dev[dev];
}

int plan_sms() {
  const DeviceInfo d = current_device();
  return d.ok ? d.sms : kDefaultSms;
}

bool params_valid(const dflash_params* p) {
  if (p == nullptr) return false;
  for (int r : p->reserved)
    if (r != 0) return false;
  if (p->batch < 1 || p->num_kv_heads < 1 || p->num_q_heads < p->num_kv_heads) return false;
  if (p->num_q_heads % p->num_kv_heads != 0) return false;
  if (p->head_dim != 64 && p->head_dim != 128) return false;
  if (p->page_size != 16 && p->page_size != 32 && p->page_size != 64) return false;
  if (p->block_size < 1 || p->block_size > kMaxBlock) return false;
  const int64_t G = p->num_q_heads / p->num_kv_heads;
  if (G * p->block_size > kMaxRows) return false;
  if (p->window < 0) return false;
  if (p->future_keys != 0 && p->future_keys != 1) return false;
  if (p->right_window < 0 || p->right_window >= p->block_size) return false;
  if (p->future_keys == 1 && p->right_window != 0) return false;
  if (!std::isfinite(p->scale) || !(p->scale > 0.f)) return false;
  // Positions are 32-bit on the device: keep L + K + a tile well inside int32.
  if (p->max_ctx_len < 0 || p->max_ctx_len > (1 << 30)) return false;
  if (p->max_pages_per_req < 1 || p->num_pages < 1) return false;
  if (static_cast<int64_t>(p->max_ctx_len) + p->block_size >
      static_cast<int64_t>(p->max_pages_per_req) * p->page_size)
    return false;
  // One (page, head) slice of the pool is addressed with 32-bit TMA
  // coordinates and a stride below 2^40 bytes.
  if (static_cast<int64_t>(p->num_kv_heads) * p->page_size * p->head_dim * 2 >= (int64_t(1) << 40))
    return false;
  if (p->force_path < DFLASH_PATH_AUTO || p->force_path > DFLASH_PATH_TCGEN05) return false;
  if (p->force_split_tiles < 0 || p->force_split_tiles > kMaxSplitTiles) return false;
  if (p->kv_dtype != DFLASH_KV_BF16 && p->kv_dtype != DFLASH_KV_FP8_E4M3) return false;
  if (p->test_flags != 0 && p->test_flags != DFLASH_TEST_WITHHOLD_LOADS) return false;
  return true;
}

// The planner.  Every grid depends on the parameters only, never on the
// device-resident lengths, so a captured graph replays for any lengths up to
// max_ctx_len.  mma.sync kernel: grid (max_splits, Hkv, B); each request's
// visible key range is cut into units of C tiles, C chosen by a cost model
// (waves of units, the partial state each writes, the combine).  tcgen05
// kernel: one CTA per SM over the flat tile sequence of all pairs.
bool make_plan(const dflash_params* p, int num_sms, KernelPlan* out) {
  if (!params_valid(p)) return false;
  KernelPlan k{};
  const int G = p->num_q_heads / p->num_kv_heads;
  const int D = p->head_dim;
  k.R = G * p->block_size;
  k.num_sms = num_sms;
  // The tcgen05 kernel keeps the requests' tile prefix in shared memory and
  // numbers the tiles of all pairs in 32 bits.
  const int64_t tc_tiles = static_cast<int64_t>(p->batch) * p->num_kv_heads *
                           max_tiles(p->max_ctx_len, p->block_size, p->window, split_tc_tile_keys(D));
  const bool tc_ok = split_tc_available() && p->batch <= kTcMaxBatch && tc_tiles <= (int64_t(1) << 30);
  // Path choice (measured on GB300, split + combine per call): the tcgen05
  // kernel for R > 64 with more than 8 (request, kv head) pairs (16/1 heads,
  // K = 7, 16K context: 34 us against 36 on the mma.sync kernel at 16 pairs,
  // 40 against 48 at 32; 32 against 30 at 8 pairs, equal below), and for
  // D = 128 with R > 32 and more than 32 pairs (K = 3: equal at 32 pairs, 53
  // against 61 us at 64); the mma.sync kernel otherwise (its D = 64
  // long-context shapes run in about half the tcgen05 kernel's time).  Both
  // kernels read fp8 pages, by the same rule (16/1 heads, K = 7, fp8: 34 us
  // on mma.sync against 36 at 8 pairs, 26 against 30 at 1, 89 against 73 on
  // tcgen05 at 64); the mma.sync kernel then needs a code ring as well, which
  // must fit its shared memory (R = 128 at D = 128 does not).
  const int64_t pairs = static_cast<int64_t>(p->batch) * p->num_kv_heads;
  const bool fp8 = p->kv_dtype == DFLASH_KV_FP8_E4M3;
  const bool tc_pref = (k.R > 64 && pairs > 8) || (D == 128 && k.R > 32 && pairs > 32);
  const int R_pad_mma = (k.R + 15) / 16 * 16;
  // The mma.sync kernel keeps its unit's page ids in shared memory: at least
  // one tile's must fit.
  const int mma_ppt = split_mma_tile_keys(D) / p->page_size;  // pages per tile
  const bool mma_ok =
      split_mma_smem_bytes(D, R_pad_mma, split_mma_kpw(D, R_pad_mma), fp8, mma_ppt) <= kMaxSmemPerCta;
  int path = p->force_path;
  if (path == DFLASH_PATH_AUTO)
    path = ((tc_pref || !mma_ok) && tc_ok) ? DFLASH_PATH_TCGEN05 : DFLASH_PATH_MMA;
  if (path == DFLASH_PATH_MMA && !mma_ok) return false;
  if (path == DFLASH_PATH_TCGEN05 && !tc_ok) return false;
  k.path = path;
  if (path == DFLASH_PATH_MMA) {
    k.R_pad = (k.R + 15) / 16 * 16;
    k.T = split_mma_tile_keys(D);
    k.kpw = split_mma_kpw(D, k.R_pad);
    const int consumer_warps = (k.R_pad / 16) * (k.T / k.kpw);
    k.threads = 32 * (1 + consumer_warps);
    if (fp8) k.threads += 32 * mma_widen_warps(D, k.kpw, k.threads);
    k.smem_bytes = split_mma_smem_bytes(D, k.R_pad, k.kpw, fp8, 0);  // page ids added below
  } else {
    k.R_pad = 128;
    k.T = split_tc_tile_keys(D);
    k.kpw = 0;
    k.threads = split_tc_threads();
    k.smem_bytes = split_tc_smem_bytes(D);
  }
  const int mt = max_tiles(p->max_ctx_len, p->block_size, p->window, k.T);
  if (path == DFLASH_PATH_TCGEN05) {
    // Flat split: one CTA per SM, each taking an equal share of all pairs'
    // tiles (computed on the device from the actual lengths, at least
    // kTcMinTiles), or force_split_tiles tiles per CTA and enough CTAs for
    // every pair at max_ctx_len.  Two partial slots per CTA.
    if (p->force_split_tiles > 0) {
      k.C = p->force_split_tiles;
      k.seg_cost = 0;
      k.units = (tc_tiles + k.C - 1) / k.C;
    } else {
      // A segment's end (merge, output staging, query reload) costs about as
      // much time as this many key tiles (D = 128: 6 measured best of 4, 6, 9
      // on the 16/1-head and 64/4-head shapes).
      k.seg_cost = D == 128 ? 6 : 8;
      const int64_t cost = tc_tiles + static_cast<int64_t>(k.seg_cost) * p->batch * p->num_kv_heads;
      int64_t ctas = (cost + kTcMinTiles - 1) / kTcMinTiles;
      if (ctas > num_sms) ctas = num_sms;
      k.units = ctas;
      k.C = static_cast<int>((cost + ctas - 1) / ctas);
      if (k.C < kTcMinTiles) k.C = kTcMinTiles;
    }
    k.S = 2;
    k.ctas_per_sm = 1;
    if (k.units > 0x7fffffff) return false;
    *out = k;
    return true;
  }
  // Tiles per unit: at most kMaxSplitTiles, and as many as leave the unit's
  // page ids room in shared memory.  Cost in tile-times of one SM: the waves
  // of units, each C tiles plus a pipeline fill of about two tiles, plus the
  // partial state every unit writes and the combine reads back (2*R*D*4
  // bytes, 2R/T tiles' worth of K/V bytes), plus the combine's latency.
  // Sized for every request at max_ctx_len; shorter requests leave units
  // empty and the block scheduler fills the gaps.  Returns 0 when a forced
  // C is above the cap.
  const double npairs = static_cast<double>(pairs);
  auto ctas_per_sm_for = [&](int smem) {
    int c = kSmemPerSm / (smem + 1024);
    if (c > 2048 / k.threads) c = 2048 / k.threads;
    return c < 1 ? 1 : c;
  };
  auto choose_C = [&](int smem_base, int ctas_per_sm) {
    // Every CTA an SM holds keeps its page ids (and 1 KB the system reserves).
    const int budget = ctas_per_sm > 1 ? kSmemPerSm / ctas_per_sm - 1024 : kMaxSmemPerCta;
    int c_cap = (budget - smem_base) / (4 * mma_ppt);
    if (c_cap > kMaxSplitTiles) c_cap = kMaxSplitTiles;
    if (p->force_split_tiles > 0) return p->force_split_tiles <= c_cap ? p->force_split_tiles : 0;
    const double slots = static_cast<double>(num_sms) * ctas_per_sm;
    const double partial_tiles = 2.0 * k.R / k.T;
    double best = 1e300;
    int best_c = 1;
    const int c_hi = mt < c_cap ? mt : c_cap;
    for (int c = 1; c <= c_hi; ++c) {
      const int S = (mt + c - 1) / c;
      if (S > 65535) continue;
      const double units = npairs * S;
      const double waves = std::ceil(units / slots);
      // The combine walks a row's S partials eight at a time, each round
      // about one memory latency (~ one tile time); only when S > 1.  Its
      // block-per-row form takes two rounds whatever S.
      const long long rows = static_cast<long long>(p->batch) * p->block_size * p->num_q_heads;
      const double combine = S > 1 ? (combine_wide(S, rows) ? 2.0 : std::ceil(S / 8.0)) : 0.0;
      const double cost = waves * (c + 2.0) + units * partial_tiles / slots + combine;
      if (cost <= best * (1.0 + 1e-12)) {
        best = cost;
        best_c = c;
      }
    }
    return best_c;
  };
  k.ctas_per_sm = ctas_per_sm_for(k.smem_bytes);
  int C = choose_C(k.smem_bytes, k.ctas_per_sm);
  if (C <= 0) return false;
  // A plan of more than one wave takes the two-CTAs-per-SM form where the
  // kernel has one, with the unit length re-chosen for twice the slots: each
  // CTA's prologue and merge then overlap the other's streaming, and an SM
  // holds twice the warps and twice the loads in flight (the 64/16-head
  // batch of 256 requests: 10.88 -> 10.18 ms; 8/2 heads 32K at 16 requests
  // 64.3 -> 61.3 us).  Not where that would more than halve the unit length
  // (8/2 heads 128K at 32 requests, 147 -> 54 tiles: 349 -> 364 us), nor with
  // the one-CTA units kept (1.5 waves of pairs of CTAs: 349 -> 402 us).
  // Single-wave plans keep one CTA per SM, whose 4-stage ring and 140
  // registers run a short unit faster (8/2 heads 32K at 1 request: 19.5
  // against 21.5 us).
  if (split_mma_two_ctas_ok(D, k.R_pad, k.kpw, fp8) &&
      npairs * ((mt + C - 1) / C) > static_cast<double>(num_sms) * k.ctas_per_sm) {
    const int smem2 = split_mma_smem_bytes(D, k.R_pad, k.kpw, fp8, 0, true);
    const int cps2 = ctas_per_sm_for(smem2);
    const int C2 = choose_C(smem2, cps2);
    if (cps2 >= 2 && C2 > 0 && 2 * C2 >= C) {
      k.two_ctas = true;
      k.ctas_per_sm = cps2;
      C = C2;
    }
  }
  k.C = C;
  k.S = (mt + C - 1) / C;
  k.units = static_cast<int64_t>(p->batch) * p->num_kv_heads * k.S;
  k.smem_bytes = split_mma_smem_bytes(D, k.R_pad, k.kpw, fp8, C * mma_ppt, k.two_ctas);
  if (k.S > 65535 || p->num_kv_heads > 65535 || p->batch > 65535) return false;
  *out = k;
  return true;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace: header (status word) | partial LSEs | partial output weights
// (log-sums of the rounded probabilities) | partial outputs, each region
// 256-byte aligned.

size_t partial_rows_for(const KernelPlan& k) {
  return static_cast<size_t>(k.units) * (k.path == DFLASH_PATH_TCGEN05 ? k.S : 1) * k.R;
}

size_t workspace_bytes_for(const dflash_params* p, const KernelPlan& k) {
  const size_t rows = partial_rows_for(k);
  const size_t lse = align_up(rows * sizeof(float), 256);
  const size_t o = rows * p->head_dim * sizeof(float);
  return kHeaderBytes + 2 * lse + o;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
      cudaGetLastError();
  });
  return g_encode;
}

// 4-D view [num_pages][Hkv][P][D] of a page pool, box = (64 columns, P rows,
// one head, one page), 128-byte swizzle, zero fill outside the pool.
bool encode_pool(CUtensorMap* map, const void* pool, const dflash_params* p) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(p->head_dim),
                              static_cast<cuuint64_t>(p->page_size),
                              static_cast<cuuint64_t>(p->num_kv_heads),
                              static_cast<cuuint64_t>(p->num_pages)};
  const cuuint64_t row = static_cast<cuuint64_t>(p->head_dim) * 2;
  const cuuint64_t strides[3] = {row, row * p->page_size, row * p->page_size * p->num_kv_heads};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(p->page_size), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// fp8 context: 4-D view [num_pages][Hkv][P][D] of a pool of E4M3 codes, box
// = (D codes, P rows, one head, one page), rows packed at D bytes with the
// swizzle of that row length (128-byte for D = 128, 64-byte for D = 64),
// zero fill outside the pool.
bool encode_pool_fp8(CUtensorMap* map, const void* pool, const dflash_params* p) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(p->head_dim),
                              static_cast<cuuint64_t>(p->page_size),
                              static_cast<cuuint64_t>(p->num_kv_heads),
                              static_cast<cuuint64_t>(p->num_pages)};
  const cuuint64_t row = static_cast<cuuint64_t>(p->head_dim);
  const cuuint64_t strides[3] = {row, row * p->page_size, row * p->page_size * p->num_kv_heads};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(p->head_dim), static_cast<cuuint32_t>(p->page_size), 1,
                             1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(pool), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        p->head_dim == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D view [B*K][Hq][D] of the queries (or of the output), box = (64
// columns, G heads, K tokens): one box is the packed tile of one (request,
// kv head) pair, rows r = i*G + g, for one 64-column half; 128-byte swizzle.
bool encode_queries(CUtensorMap* map, const void* q, const dflash_params* p) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const int G = p->num_q_heads / p->num_kv_heads;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(p->head_dim),
                              static_cast<cuuint64_t>(p->num_q_heads),
                              static_cast<cuuint64_t>(p->batch) * p->block_size};
  const cuuint64_t row = static_cast<cuuint64_t>(p->head_dim) * 2;
  const cuuint64_t strides[2] = {row, row * p->num_q_heads};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(p->block_size)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D view [slots][R][D] of the fp32 partial outputs, box = (32 columns,
// R rows, one slot); 128-byte swizzle.
bool encode_partials(CUtensorMap* map, void* part_o, const dflash_params* p, int R, int64_t slots) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(p->head_dim), static_cast<cuuint64_t>(R),
                              static_cast<cuuint64_t>(slots)};
  const cuuint64_t row = static_cast<cuuint64_t>(p->head_dim) * 4;
  const cuuint64_t strides[2] = {row, row * R};
  const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(R), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, part_o, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// Device check shared by the entry points.
int check_device() {
  const DeviceInfo dev = current_device();
  if (!dev.ok) return DFLASH_ERR_LAUNCH;
  if (dev.cc != 103) return DFLASH_ERR_DEVICE;
  return DFLASH_OK;
}

bool append_pointers_ok(const void* k_block, const void* v_block, const void* k_pages,
                        const void* v_pages, const int32_t* page_table, const int32_t* ctx_lens,
                        const void* workspace) {
  if (!k_block || !v_block || !k_pages || !v_pages || !page_table || !ctx_lens) return false;
  return aligned(k_block, 16) && aligned(v_block, 16) && aligned(k_pages, 16) &&
         aligned(v_pages, 16) && aligned(page_table, 4) && aligned(ctx_lens, 4) &&
         (workspace == nullptr || aligned(workspace, 256));
}

AppendArgs append_args(const dflash_params* p, const void* k_block, const void* v_block,
                       void* k_pages, void* v_pages, const int32_t* page_table,
                       const int32_t* ctx_lens, void* workspace) {
  AppendArgs ap{};
  ap.k_block = static_cast<const uint16_t*>(k_block);
  ap.v_block = static_cast<const uint16_t*>(v_block);
  ap.k_pages = static_cast<uint16_t*>(k_pages);
  ap.v_pages = static_cast<uint16_t*>(v_pages);
  ap.page_table = page_table;
  ap.ctx_lens = ctx_lens;
  ap.placement = nullptr;
  ap.status = static_cast<uint32_t*>(workspace);
  ap.B = p->batch;
  ap.K = p->block_size;
  ap.Hkv = p->num_kv_heads;
  ap.D = p->head_dim;
  ap.P = p->page_size;
  ap.max_pages = p->max_pages_per_req;
  ap.num_pages = p->num_pages;
  ap.max_ctx_len = p->max_ctx_len;
  return ap;
}

// The attention call; with `append` given, the K/V append runs first and the
// split kernel is its programmatic dependent (its producers wait for it).
// With dense_k / dense_v given (dense-suffix form) the block rows come from
// them and the pages hold the context only; with fp8 given as well, the
// pages hold E4M3 codes dequantised by fp8->k_scale / fp8->v_scale.
struct Fp8Scales {
  float k_scale, v_scale;
};

// A context-parallel part: the key range per request and the fp32 output.
struct PartArgs {
  const int32_t* key_begin;
  const int32_t* key_end;
  float* out_f32;
};

// The parameters a context-parallel part runs with: the mma.sync unit grid,
// whose empty units and combine handle a pair that has no key in the part.
bool part_params(const dflash_params* p, dflash_params* pp) {
  if (!params_valid(p) || p->kv_dtype != DFLASH_KV_BF16) return false;
  if (p->force_path != DFLASH_PATH_AUTO && p->force_path != DFLASH_PATH_MMA) return false;
  *pp = *p;
  pp->force_path = DFLASH_PATH_MMA;
  return true;
}

int run_attention(const dflash_params* p_in, const void* q, const void* k_pages, const void* v_pages,
                  const int32_t* page_table, const int32_t* ctx_lens, void* out, float* lse2,
                  void* workspace, size_t workspace_bytes, void* stream, void* split_start,
                  void* split_done, const AppendArgs* append, const void* dense_k = nullptr,
                  const void* dense_v = nullptr, const Fp8Scales* fp8 = nullptr,
                  const PartArgs* part = nullptr) {
  dflash_params pp;
  const dflash_params* p = p_in;
  if (part != nullptr) {
    if (!part_params(p_in, &pp) || append != nullptr || dense_k != nullptr || fp8 != nullptr)
      return DFLASH_ERR_INVALID;
    if (!part->key_begin || !part->key_end || !part->out_f32 || !aligned(part->key_begin, 4) ||
        !aligned(part->key_end, 4) || !aligned(part->out_f32, 16))
      return DFLASH_ERR_INVALID;
    p = &pp;
    out = part->out_f32;  // checked for presence below; the bf16 output is not written
  }
  if (!params_valid(p)) return DFLASH_ERR_INVALID;
  if ((fp8 != nullptr) != (p->kv_dtype == DFLASH_KV_FP8_E4M3)) return DFLASH_ERR_INVALID;
  if (fp8 != nullptr) {
    if (dense_k == nullptr || append != nullptr) return DFLASH_ERR_INVALID;
    if (!std::isfinite(fp8->k_scale) || !(fp8->k_scale > 0.f) || !std::isfinite(fp8->v_scale) ||
        !(fp8->v_scale > 0.f))
      return DFLASH_ERR_INVALID;
  }
  if (!q || !k_pages || !v_pages || !page_table || !ctx_lens || !out || !lse2 || !workspace)
    return DFLASH_ERR_INVALID;
  if ((dense_k == nullptr) != (dense_v == nullptr) || !aligned(dense_k, 16) || !aligned(dense_v, 16))
    return DFLASH_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) ||
      !aligned(page_table, 4) || !aligned(ctx_lens, 4) || !aligned(lse2, 4) ||
      !aligned(workspace, 256))
    return DFLASH_ERR_INVALID;
  const DeviceInfo dev = current_device();
  if (!dev.ok) return DFLASH_ERR_LAUNCH;
  if (dev.cc != 103) return DFLASH_ERR_DEVICE;
  KernelPlan k;
  if (!make_plan(p, dev.sms, &k)) return DFLASH_ERR_INVALID;
  if (workspace_bytes < workspace_bytes_for(p, k)) return DFLASH_ERR_WORKSPACE;
  k.pdl = append != nullptr;

  const bool tc = k.path == DFLASH_PATH_TCGEN05;
  CUtensorMap tm_k, tm_v, tm_q, tm_out, tm_part;
  if (fp8 != nullptr) {
    if (!encode_pool_fp8(&tm_k, k_pages, p) || !encode_pool_fp8(&tm_v, v_pages, p)) return DFLASH_ERR_LAUNCH;
  } else if (!encode_pool(&tm_k, k_pages, p) || !encode_pool(&tm_v, v_pages, p)) {
    return DFLASH_ERR_LAUNCH;
  }

  AttnArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.k_pages = static_cast<const uint16_t*>(k_pages);
  a.v_pages = static_cast<const uint16_t*>(v_pages);
  a.page_table = page_table;
  a.ctx_lens = ctx_lens;
  a.out = static_cast<uint16_t*>(out);
  a.lse2 = lse2;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.k_block = static_cast<const uint16_t*>(dense_k);
  a.v_block = static_cast<const uint16_t*>(dense_v);
  const size_t off_lse = kHeaderBytes;
  const size_t lse_bytes = align_up(partial_rows_for(k) * sizeof(float), 256);
  a.part_lse = reinterpret_cast<float*>(ws + off_lse);
  a.part_lseo = reinterpret_cast<float*>(ws + off_lse + lse_bytes);
  a.part_o = reinterpret_cast<float*>(ws + off_lse + 2 * lse_bytes);
  if (tc && (!encode_queries(&tm_q, q, p) || !encode_queries(&tm_out, out, p) ||
             !encode_partials(&tm_part, a.part_o, p, k.R, k.units * k.S)))
    return DFLASH_ERR_LAUNCH;
  a.B = p->batch;
  a.Hq = p->num_q_heads;
  a.Hkv = p->num_kv_heads;
  a.G = p->num_q_heads / p->num_kv_heads;
  a.D = p->head_dim;
  a.P = p->page_size;
  a.max_pages = p->max_pages_per_req;
  a.num_pages = p->num_pages;
  a.K = p->block_size;
  a.W = p->window;
  a.rw = p->future_keys ? p->block_size - 1 : p->right_window;
  a.max_ctx_len = p->max_ctx_len;
  a.scale_log2 = p->scale * 1.4426950408889634f;
  a.R = k.R;
  a.R_pad = k.R_pad;
  a.T = k.T;
  a.C = k.C;
  a.S = k.S;
  a.ncta = tc ? static_cast<int>(k.units) : 0;
  a.qn_force = tc ? p->force_split_tiles : 0;
  a.qn_min = kTcMinTiles;
  a.seg_cost = tc ? k.seg_cost : 0;
  a.fp8 = fp8 != nullptr ? 1 : 0;
  a.withhold_loads = p->test_flags == DFLASH_TEST_WITHHOLD_LOADS ? 1 : 0;
  a.kblk_mul = 1.f;
  a.pblk_mul = 1.f;
  a.out_mul = 1.f;
  if (part != nullptr) {
    a.out = nullptr;
    a.key_begin = part->key_begin;
    a.key_end = part->key_end;
    a.keep_partials = 1;
    a.out_f32 = part->out_f32;
  }
  if (fp8 != nullptr) {
    a.scale_log2 *= fp8->k_scale;
    a.kblk_mul = 1.f / fp8->k_scale;
    a.pblk_mul = 1.f / fp8->v_scale;
    a.out_mul = fp8->v_scale;
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (split_start != nullptr &&
      cudaEventRecord(static_cast<cudaEvent_t>(split_start), s) != cudaSuccess)
    return DFLASH_ERR_LAUNCH;
  if (append != nullptr && launch_append(*append, s) != cudaSuccess) return DFLASH_ERR_LAUNCH;
  int err = tc ? launch_split_tc(a, k, tm_k, tm_v, tm_q, tm_out, tm_part, s)
               : launch_split_mma(a, k, tm_k, tm_v, s);
  if (err != cudaSuccess) return DFLASH_ERR_LAUNCH;
  if (split_done != nullptr &&
      cudaEventRecord(static_cast<cudaEvent_t>(split_done), s) != cudaSuccess)
    return DFLASH_ERR_LAUNCH;
  // With one unit per (request, kv head) the mma.sync kernel wrote the final
  // output itself; otherwise merge the partial states (the flat split of the
  // tcgen05 kernel always may cut a pair).
  if (tc || k.S > 1 || part != nullptr) {
    err = launch_combine(a, s, split_done == nullptr, tc);
    if (err != cudaSuccess) return DFLASH_ERR_LAUNCH;
  }
  return DFLASH_OK;
}

}  // namespace
}  // namespace dflash

using namespace dflash;

extern "C" {

size_t dflash_workspace_size(const dflash_params* p) {
  KernelPlan k;
  if (!make_plan(p, plan_sms(), &k)) return 0;
  return workspace_bytes_for(p, k);
}

int dflash_plan(const dflash_params* p, dflash_plan_info* info) {
  KernelPlan k;
  if (info == nullptr || !make_plan(p, plan_sms(), &k)) return DFLASH_ERR_INVALID;
  std::memset(info, 0, sizeof(*info));
  info->path = k.path;
  info->rows = k.R;
  info->rows_padded = k.R_pad;
  info->tile_keys = k.T;
  info->split_tiles = k.C;
  info->max_splits = k.S;
  info->units = k.units;
  info->threads = k.threads;
  info->smem_bytes = k.smem_bytes;
  info->num_sms = k.num_sms;
  info->flat = k.path == DFLASH_PATH_TCGEN05 ? 1 : 0;
  info->ctas_per_sm = k.ctas_per_sm;
  return DFLASH_OK;
}

int dflash_block_attn(const dflash_params* p, const void* q, const void* k_pages,
                      const void* v_pages, const int32_t* page_table, const int32_t* ctx_lens,
                      void* out, float* lse2, void* workspace, size_t workspace_bytes,
                      void* stream) {
  return dflash_block_attn_timed(p, q, k_pages, v_pages, page_table, ctx_lens, out, lse2,
                                 workspace, workspace_bytes, stream, nullptr, nullptr);
}

int dflash_block_attn_timed(const dflash_params* p, const void* q, const void* k_pages,
                            const void* v_pages, const int32_t* page_table,
                            const int32_t* ctx_lens, void* out, float* lse2, void* workspace,
                            size_t workspace_bytes, void* stream, void* split_start,
                            void* split_done) {
  return run_attention(p, q, k_pages, v_pages, page_table, ctx_lens, out, lse2, workspace,
                       workspace_bytes, stream, split_start, split_done, nullptr);
}

int dflash_block_attn_dense_suffix(const dflash_params* p, const void* q, const void* k_block,
                                   const void* v_block, const void* k_pages, const void* v_pages,
                                   const int32_t* page_table, const int32_t* ctx_lens, void* out,
                                   float* lse2, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  if (k_block == nullptr || v_block == nullptr) return DFLASH_ERR_INVALID;
  return run_attention(p, q, k_pages, v_pages, page_table, ctx_lens, out, lse2, workspace,
                       workspace_bytes, stream, nullptr, nullptr, nullptr, k_block, v_block);
}

int dflash_block_attn_fp8_context(const dflash_params* p, const void* q, const void* k_block,
                                  const void* v_block, const void* k_pages, const void* v_pages,
                                  float k_scale, float v_scale, const int32_t* page_table,
                                  const int32_t* ctx_lens, void* out, float* lse2, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  return dflash_block_attn_fp8_context_timed(p, q, k_block, v_block, k_pages, v_pages, k_scale, v_scale,
                                             page_table, ctx_lens, out, lse2, workspace, workspace_bytes,
                                             stream, nullptr, nullptr);
}

int dflash_block_attn_fp8_context_timed(const dflash_params* p, const void* q, const void* k_block,
                                        const void* v_block, const void* k_pages, const void* v_pages,
                                        float k_scale, float v_scale, const int32_t* page_table,
                                        const int32_t* ctx_lens, void* out, float* lse2,
                                        void* workspace, size_t workspace_bytes, void* stream,
                                        void* split_start, void* split_done) {
  if (k_block == nullptr || v_block == nullptr) return DFLASH_ERR_INVALID;
  const Fp8Scales sc{k_scale, v_scale};
  return run_attention(p, q, k_pages, v_pages, page_table, ctx_lens, out, lse2, workspace,
                       workspace_bytes, stream, split_start, split_done, nullptr, k_block, v_block, &sc);
}

int dflash_block_placement(const dflash_params* p, const int32_t* page_table,
                           const int32_t* ctx_lens, int32_t* placement, void* workspace,
                           void* stream) {
  if (!params_valid(p) || !page_table || !ctx_lens || !placement) return DFLASH_ERR_INVALID;
  if (!aligned(page_table, 4) || !aligned(ctx_lens, 4) || !aligned(placement, 4) ||
      (workspace != nullptr && !aligned(workspace, 256)))
    return DFLASH_ERR_INVALID;
  const int rc = check_device();
  if (rc != DFLASH_OK) return rc;
  AppendArgs ap = append_args(p, nullptr, nullptr, nullptr, nullptr, page_table, ctx_lens, workspace);
  ap.placement = placement;
  return launch_append(ap, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DFLASH_OK
                                                                             : DFLASH_ERR_LAUNCH;
}

int dflash_append_block_kv(const dflash_params* p, const void* k_block, const void* v_block,
                           void* k_pages, void* v_pages, const int32_t* page_table,
                           const int32_t* ctx_lens, void* workspace, void* stream) {
  // The append copies bf16 rows: fp8 pools are written by their owner.
  if (!params_valid(p) || p->kv_dtype != DFLASH_KV_BF16 ||
      !append_pointers_ok(k_block, v_block, k_pages, v_pages, page_table, ctx_lens, workspace))
    return DFLASH_ERR_INVALID;
  const int rc = check_device();
  if (rc != DFLASH_OK) return rc;
  const AppendArgs ap =
      append_args(p, k_block, v_block, k_pages, v_pages, page_table, ctx_lens, workspace);
  return launch_append(ap, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DFLASH_OK
                                                                             : DFLASH_ERR_LAUNCH;
}

int dflash_block_attn_append(const dflash_params* p, const void* q, const void* k_block,
                             const void* v_block, void* k_pages, void* v_pages,
                             const int32_t* page_table, const int32_t* ctx_lens, void* out,
                             float* lse2, void* workspace, size_t workspace_bytes, void* stream) {
  if (!params_valid(p) || workspace == nullptr ||
      !append_pointers_ok(k_block, v_block, k_pages, v_pages, page_table, ctx_lens, workspace))
    return DFLASH_ERR_INVALID;
  const AppendArgs ap =
      append_args(p, k_block, v_block, k_pages, v_pages, page_table, ctx_lens, workspace);
  return run_attention(p, q, k_pages, v_pages, page_table, ctx_lens, out, lse2, workspace,
                       workspace_bytes, stream, nullptr, nullptr, &ap);
}

size_t dflash_partial_workspace_size(const dflash_params* p) {
  dflash_params pp;
  if (!part_params(p, &pp)) return 0;
  return dflash_workspace_size(&pp);
}

int dflash_block_attn_partial(const dflash_params* p, const void* q, const void* k_pages,
                              const void* v_pages, const int32_t* page_table, const int32_t* ctx_lens,
                              const int32_t* key_begin, const int32_t* key_end, float* part_out,
                              float* part_lse2, void* workspace, size_t workspace_bytes, void* stream) {
  const PartArgs part{key_begin, key_end, part_out};
  return run_attention(p, q, k_pages, v_pages, page_table, ctx_lens, nullptr, part_lse2, workspace,
                       workspace_bytes, stream, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, &part);
}

int dflash_combine_partials(const dflash_params* p, int n_parts, const float* part_out,
                            const float* part_lse2, void* out, float* lse2, void* stream) {
  if (!params_valid(p) || n_parts < 1 || !part_out || !part_lse2 || !out || !lse2) return DFLASH_ERR_INVALID;
  if (!aligned(part_out, 16) || !aligned(part_lse2, 4) || !aligned(out, 16) || !aligned(lse2, 4))
    return DFLASH_ERR_INVALID;
  const int64_t rows = static_cast<int64_t>(p->batch) * p->block_size * p->num_q_heads;
  if (rows > 0x7fffffff) return DFLASH_ERR_INVALID;
  const int rc = check_device();
  if (rc != DFLASH_OK) return rc;
  AttnArgs a{};
  a.part_o = const_cast<float*>(part_out);
  a.part_lse = const_cast<float*>(part_lse2);
  a.part_lseo = const_cast<float*>(part_lse2);  // outputs weighted by the parts' LSEs
  a.out = static_cast<uint16_t*>(out);
  a.lse2 = lse2;
  a.B = p->batch;
  a.K = p->block_size;
  a.Hq = p->num_q_heads;
  a.D = p->head_dim;
  a.R = static_cast<int>(rows);
  return launch_combine_parts(a, n_parts, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DFLASH_OK
                                                                                          : DFLASH_ERR_LAUNCH;
}

const char* dflash_status_string(int status) {
  switch (status) {
    case DFLASH_OK: return "ok";
    case DFLASH_ERR_INVALID: return "invalid argument";
    case DFLASH_ERR_WORKSPACE: return "workspace too small";
    case DFLASH_ERR_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case DFLASH_ERR_LAUNCH: return "CUDA launch failed";
    default: return "unknown status";
  }
}

int dflash_read_device_status(const void* workspace, void* stream) {
  if (workspace == nullptr) return DFLASH_ERR_INVALID;
  uint32_t v = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return DFLASH_ERR_LAUNCH;
  return static_cast<int>(v & 0x7fffffffu);
}

int dflash_clear_device_status(void* workspace, void* stream) {
  if (workspace == nullptr) return DFLASH_ERR_INVALID;
  if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return DFLASH_ERR_LAUNCH;
  return DFLASH_OK;
}

int dflash_version(void) { return 100; }

}  // extern "C"
