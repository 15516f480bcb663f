// Oracle for paged draft-block attention: plain, slow, fp64, CPU.
//
// TEST INFRASTRUCTURE ONLY.  The product path never links, loads or calls
// this file; only the tests, the smoke check and the benchmark's CPU-baseline
// leg do.  It shares no code, header, table or constant with the CUDA library.
//
// What it computes is the plain definition of the attention a draft block
// takes in a DFlash / DSpark drafter (TensorRT-LLM PR #21130, "Non-causal
// windowed DSpark draft block": description, "Why" and change 2; PR #20374,
// "Non-causal unwindowed DFlash draft block": description).  For request b
// with L = ctx_lens[b] context tokens and a block of K draft tokens stored in
// the same pages at logical positions L .. L+K-1, query token i of the block
// (position L+i) of query head hq, which reads kv head hq / G (G = Hq / Hkv),
// sees
//   * the causal window (L+i-W, L+i] when a window W > 0 is given, else every
//     position up to L+i (context and block keys alike);
//   * the later block keys L+j, i < j <= i + r, where r = K-1 in the
//     non-causal form (future_keys = 1: every later block key) and r is the
//     given right window otherwise (0: the causal form) -- PR #21130 "Why":
//     the causal window plus the later keys of the block.
// Every key row is read through the page table: the row of logical position p
// is pages[page_table[b][p / P]][h][p % P][:] (HND page layout, PR #20374
// kernel sweep: "page 32, HND") -- or, in the dense-suffix form (PR #16150:
// the draft context in the target's paged pool, the block's noise rows a
// dense suffix inside the one softmax), the block's rows p = L+j come from dense tensors
// k_block[b][j][h][:], v_block[b][j][h][:] and only the context is paged.
// The context pages of that form may also be stored in fp8 (PR #16150: the
// drafter's context may be kept as fp8): the OCP 8-bit E4M3 format (sign,
// 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 is subnormal,
// S.1111.111 is NaN, no infinities) with one dequantisation scale per tensor,
// k = k_scale * e4m3(code), v = v_scale * e4m3(code); the block rows stay
// bf16 and take no scale.
// Then, in double precision,
//   s_p  = scale * sum_d q_d k_{p,d}
//   m    = max_p s_p,   Z = sum_p exp(s_p - m)
//   out  = sum_p exp(s_p - m) v_p / Z
//   lse2 = (m + ln Z) / ln 2         (the base-2 log-sum-exp, PR #21130 change 1)
// No blocking, splitting, merging or reordering beyond that definition.
//
// Context-parallel parts (the split of one request's keys across ranks that
// exchange their partial (O, lse2) once, then merge them): a part covers the
// logical key positions [key_begin[b], key_end[b]) of request b's L + K
// positions (context and block alike), and its result is the same
// definition over the visible positions that lie in that range -- out
// normalised over them, lse2 their base-2 log-sum-exp; a row that sees none
// of them gets out = 0 and lse2 = -inf.  Parts that tile [0, L+K) merge into
// the whole attention by the base-2 log-sum-exp combine of PR #21130
// (change 1): lse = log2 sum_s 2^lse_s, out = sum_s 2^(lse_s - lse) out_s.
//
// Inputs are bf16 bit patterns (uint16), widened exactly to double.

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

double bf16_to_double(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof(f));
  return static_cast<double>(f);
}

// Value of an E4M3 code: (1 + m/8) * 2^(e-7) for e > 0, (m/8) * 2^-6 for
// e = 0, NaN for e = 15, m = 7.
double e4m3_to_double(uint8_t code) {
  const int sign = code >> 7;
  const int e = (code >> 3) & 15;
  const int m = code & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = e == 0 ? std::ldexp(static_cast<double>(m), -9)
                            : std::ldexp(static_cast<double>(8 + m), e - 10);
  return sign ? -mag : mag;
}

struct Problem {
  int B, Hq, Hkv, D, P, max_pages, num_pages, K, W, future_keys, right_window;
  double scale;
  const uint16_t* q;
  const uint16_t* k_pages;
  const uint16_t* v_pages;
  const int32_t* page_table;
  const int32_t* ctx_lens;
  const uint16_t* k_block;  // [B, K, Hkv, D] dense block rows, or null (paged)
  const uint16_t* v_block;
  const uint8_t* k_pages8;  // fp8 context pages (then k_pages / v_pages are unused), or null
  const uint8_t* v_pages8;
  double k_scale, v_scale;
  const int32_t* key_begin;  // context-parallel part: keys [key_begin[b], key_end[b]), or null
  const int32_t* key_end;
};

// A key or value row: bf16 bits (scale 1), or fp8 codes with their scale.
struct RowRef {
  const uint16_t* bf16;
  const uint8_t* fp8;
  double scale;
  double at(int d) const { return scale * (fp8 ? e4m3_to_double(fp8[d]) : bf16_to_double(bf16[d])); }
};

// Address of the key/value row of logical position p of request b, head h;
// returns -1 when the page-table entry does not name a page of the pool.
int64_t row_offset(const Problem& pr, int b, int h, int64_t p) {
  const int64_t slot = p / pr.P;
  if (slot < 0 || slot >= pr.max_pages) return -1;
  const int32_t page = pr.page_table[static_cast<int64_t>(b) * pr.max_pages + slot];
  if (page < 0 || page >= pr.num_pages) return -1;
  return ((static_cast<int64_t>(page) * pr.Hkv + h) * pr.P + (p % pr.P)) * pr.D;
}

// One (request, query token, query head) row.  Returns 0 or a negative error.
int attend_row(const Problem& pr, int b, int i, int hq, double* out_row, double* lse_row) {
  const int G = pr.Hq / pr.Hkv;
  const int h = hq / G;
  const int64_t L = pr.ctx_lens[b];
  if (L < 0) return -2;

  // Visible logical positions, in increasing order: the causal window, then
  // the later block keys within the right window.
  std::vector<int64_t> pos;
  const int64_t lo = (pr.W > 0) ? std::max<int64_t>(0, L + i - pr.W + 1) : 0;
  for (int64_t p = lo; p <= L + i; ++p) pos.push_back(p);
  const int r = pr.future_keys ? pr.K - 1 : pr.right_window;
  const int j_last = std::min(pr.K - 1, i + r);
  for (int j = i + 1; j <= j_last; ++j) pos.push_back(L + j);
  if (pr.key_begin != nullptr) {
    std::vector<int64_t> kept;
    for (int64_t p : pos)
      if (p >= pr.key_begin[b] && p < pr.key_end[b]) kept.push_back(p);
    pos.swap(kept);
  }
  if (pos.empty()) {  // nothing visible: the empty sum
    for (int d = 0; d < pr.D; ++d) out_row[d] = 0.0;
    *lse_row = -INFINITY;
    return 0;
  }

  const uint16_t* qrow = pr.q + ((static_cast<int64_t>(b) * pr.K + i) * pr.Hq + hq) * pr.D;
  std::vector<double> qd(pr.D);
  for (int d = 0; d < pr.D; ++d) qd[d] = bf16_to_double(qrow[d]);

  // Key and value rows of each visible position.
  std::vector<RowRef> krow(pos.size()), vrow(pos.size());
  for (size_t t = 0; t < pos.size(); ++t) {
    if (pr.k_block != nullptr && pos[t] >= L) {
      const int64_t j = pos[t] - L;
      const int64_t o = ((static_cast<int64_t>(b) * pr.K + j) * pr.Hkv + h) * pr.D;
      krow[t] = RowRef{pr.k_block + o, nullptr, 1.0};
      vrow[t] = RowRef{pr.v_block + o, nullptr, 1.0};
    } else {
      const int64_t o = row_offset(pr, b, h, pos[t]);
      if (o < 0) return -3;
      if (pr.k_pages8 != nullptr) {
        krow[t] = RowRef{nullptr, pr.k_pages8 + o, pr.k_scale};
        vrow[t] = RowRef{nullptr, pr.v_pages8 + o, pr.v_scale};
      } else {
        krow[t] = RowRef{pr.k_pages + o, nullptr, 1.0};
        vrow[t] = RowRef{pr.v_pages + o, nullptr, 1.0};
      }
    }
  }

  std::vector<double> s(pos.size());
  for (size_t t = 0; t < pos.size(); ++t) {
    double acc = 0.0;
    for (int d = 0; d < pr.D; ++d) acc += qd[d] * krow[t].at(d);
    s[t] = pr.scale * acc;
  }

  double m = -INFINITY;
  for (double x : s) m = std::max(m, x);
  double Z = 0.0;
  for (double x : s) Z += std::exp(x - m);
  for (int d = 0; d < pr.D; ++d) out_row[d] = 0.0;
  for (size_t t = 0; t < pos.size(); ++t) {
    const double w = std::exp(s[t] - m);
    for (int d = 0; d < pr.D; ++d) out_row[d] += w * vrow[t].at(d);
  }
  for (int d = 0; d < pr.D; ++d) out_row[d] /= Z;
  *lse_row = (m + std::log(Z)) / std::log(2.0);
  return 0;
}

// Every (request, kv head) item of req_ids (all requests when null) on
// nthreads workers.
int run_items(const Problem& pr, const int32_t* req_ids, int n_req, double* out, double* lse2,
              int nthreads) {
  const int B = pr.B, Hq = pr.Hq, Hkv = pr.Hkv, K = pr.K, D = pr.D;
  if (req_ids == nullptr) n_req = B;
  const int G = Hq / Hkv;
  const int64_t n_items = static_cast<int64_t>(n_req) * Hkv;
  std::atomic<int64_t> next{0};
  std::atomic<int> status{0};

  auto worker = [&]() {
    for (;;) {
      const int64_t it = next.fetch_add(1);
      if (it >= n_items) return;
      const int n = static_cast<int>(it / Hkv);
      const int h = static_cast<int>(it % Hkv);
      const int b = req_ids ? req_ids[n] : n;
      if (b < 0 || b >= B) { status.store(-1); continue; }
      for (int i = 0; i < K; ++i)
        for (int g = 0; g < G; ++g) {
          const int hq = h * G + g;
          const int64_t row = (static_cast<int64_t>(n) * K + i) * Hq + hq;
          const int rc = attend_row(pr, b, i, hq, out + row * D, lse2 + row);
          if (rc != 0) status.store(rc);
        }
    }
  };

  if (nthreads <= 0) nthreads = static_cast<int>(std::thread::hardware_concurrency());
  if (nthreads <= 0) nthreads = 1;
  if (nthreads > n_items) nthreads = static_cast<int>(n_items > 0 ? n_items : 1);
  std::vector<std::thread> pool;
  for (int t = 1; t < nthreads; ++t) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
  return status.load();
}

}  // namespace

extern "C" {

// Computes out[n, i, hq, :] and lse2[n, i, hq] for the requests req_ids[0..n_req)
// (every request 0..B-1 when req_ids is NULL, n_req then ignored and taken as B).
// Threads: nthreads workers over (request, kv head) items; nthreads <= 0 means
// std::thread::hardware_concurrency().  Returns 0, or -1 for bad sizes, -2 for a
// negative context length, -3 for a visible position whose page-table entry is
// out of range.
int oracle_block_attn(int B, int Hq, int Hkv, int D, int P, int max_pages, int num_pages,
                      int K, int W, int future_keys, int right_window, double scale,
                      const uint16_t* q, const uint16_t* k_pages, const uint16_t* v_pages,
                      const int32_t* page_table, const int32_t* ctx_lens,
                      const uint16_t* k_block, const uint16_t* v_block,
                      const int32_t* req_ids, int n_req,
                      double* out, double* lse2, int nthreads) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || P <= 0 || K <= 0 ||
      W < 0 || max_pages <= 0 || num_pages <= 0 || right_window < 0)
    return -1;
  if ((k_block == nullptr) != (v_block == nullptr)) return -1;
  Problem pr{B, Hq, Hkv, D, P, max_pages, num_pages, K, W, future_keys ? 1 : 0, right_window, scale,
             q, k_pages, v_pages, page_table, ctx_lens, k_block, v_block, nullptr, nullptr, 1.0, 1.0,
             nullptr, nullptr};
  return run_items(pr, req_ids, n_req, out, lse2, nthreads);
}

// One context-parallel part: the attention over the visible keys whose
// logical positions lie in [key_begin[b], key_end[b]) (int32 [B]); out is
// normalised over them, lse2 is their base-2 log-sum-exp; a row that sees
// none gets 0 and -inf.  Otherwise as oracle_block_attn (paged block rows).
int oracle_block_attn_part(int B, int Hq, int Hkv, int D, int P, int max_pages, int num_pages,
                           int K, int W, int future_keys, int right_window, double scale,
                           const uint16_t* q, const uint16_t* k_pages, const uint16_t* v_pages,
                           const int32_t* page_table, const int32_t* ctx_lens,
                           const int32_t* key_begin, const int32_t* key_end,
                           const int32_t* req_ids, int n_req, double* out, double* lse2,
                           int nthreads) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || P <= 0 || K <= 0 ||
      W < 0 || max_pages <= 0 || num_pages <= 0 || right_window < 0)
    return -1;
  if (key_begin == nullptr || key_end == nullptr) return -1;
  Problem pr{B, Hq, Hkv, D, P, max_pages, num_pages, K, W, future_keys ? 1 : 0, right_window, scale,
             q, k_pages, v_pages, page_table, ctx_lens, nullptr, nullptr, nullptr, nullptr, 1.0, 1.0,
             key_begin, key_end};
  return run_items(pr, req_ids, n_req, out, lse2, nthreads);
}

// The merge of n_parts partial results of the same rows: part s holds
// out[s][row][0..D) and lse2[s][row] (rows = B*K*Hq).  Base-2 log-sum-exp
// combine (PR #21130, change 1): lse = log2 sum_s 2^lse_s and
// out = sum_s 2^(lse_s - lse) out_s; a row with every lse_s = -inf gets 0 and
// -inf.  Returns 0, or -1 for bad sizes.
int oracle_combine_parts(int n_parts, int64_t rows, int D, const double* part_out,
                         const double* part_lse2, double* out, double* lse2) {
  if (n_parts <= 0 || rows < 0 || D <= 0) return -1;
  for (int64_t r = 0; r < rows; ++r) {
    double m = -INFINITY;
    for (int s = 0; s < n_parts; ++s) m = std::max(m, part_lse2[s * rows + r]);
    for (int d = 0; d < D; ++d) out[r * D + d] = 0.0;
    if (m == -INFINITY) {
      lse2[r] = -INFINITY;
      continue;
    }
    double z = 0.0;
    for (int s = 0; s < n_parts; ++s) z += std::exp2(part_lse2[s * rows + r] - m);
    const double lse = m + std::log2(z);
    for (int s = 0; s < n_parts; ++s) {
      const double w = std::exp2(part_lse2[s * rows + r] - lse);
      for (int d = 0; d < D; ++d) out[r * D + d] += w * part_out[(s * rows + r) * D + d];
    }
    lse2[r] = lse;
  }
  return 0;
}

// The dense-suffix form over fp8 (E4M3) context pages: k_pages8 / v_pages8
// [num_pages, Hkv, P, D] hold codes, dequantised by k_scale / v_scale; the
// block rows k_block / v_block (bf16 [B, K, Hkv, D], required) are not
// scaled.  Same sizes, threads and return codes as oracle_block_attn.
int oracle_block_attn_fp8(int B, int Hq, int Hkv, int D, int P, int max_pages, int num_pages,
                          int K, int W, int future_keys, int right_window, double scale,
                          const uint16_t* q, const uint8_t* k_pages8, const uint8_t* v_pages8,
                          double k_scale, double v_scale, const int32_t* page_table,
                          const int32_t* ctx_lens, const uint16_t* k_block, const uint16_t* v_block,
                          const int32_t* req_ids, int n_req, double* out, double* lse2,
                          int nthreads) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || P <= 0 || K <= 0 ||
      W < 0 || max_pages <= 0 || num_pages <= 0 || right_window < 0)
    return -1;
  if (k_block == nullptr || v_block == nullptr || k_pages8 == nullptr || v_pages8 == nullptr)
    return -1;
  Problem pr{B, Hq, Hkv, D, P, max_pages, num_pages, K, W, future_keys ? 1 : 0, right_window, scale,
             q, nullptr, nullptr, page_table, ctx_lens, k_block, v_block, k_pages8, v_pages8,
             k_scale, v_scale, nullptr, nullptr};
  return run_items(pr, req_ids, n_req, out, lse2, nthreads);
}

// The value of one E4M3 code (for the tests' decoding pin).
double oracle_e4m3_to_double(int code) { return e4m3_to_double(static_cast<uint8_t>(code)); }

// Block placement: the pool slot of every block token's K/V.  Block token j
// of request b sits at logical position L_b + j (L_b = ctx_lens[b]), i.e. in
// page page_table[b][(L_b + j) / P] at offset (L_b + j) % P (PR #20374: the
// block's K/V are appended to the paged cache after the context; the fused
// spec-tail kernels report these positions as the draft block placement).
// placement[(b*K + j)*2 + 0] = page, [.. + 1] = offset.  Returns 0, -1 for bad
// sizes, -2 for a negative length, -3 for a slot whose entry is not a page.
int oracle_block_placement(int B, int K, int P, int max_pages, int num_pages,
                           const int32_t* page_table, const int32_t* ctx_lens, int32_t* placement) {
  if (B <= 0 || K <= 0 || P <= 0 || max_pages <= 0 || num_pages <= 0) return -1;
  for (int b = 0; b < B; ++b) {
    const int64_t L = ctx_lens[b];
    if (L < 0) return -2;
    for (int j = 0; j < K; ++j) {
      const int64_t p = L + j;
      const int64_t slot = p / P;
      if (slot >= max_pages) return -3;
      const int32_t page = page_table[static_cast<int64_t>(b) * max_pages + slot];
      if (page < 0 || page >= num_pages) return -3;
      placement[(static_cast<int64_t>(b) * K + j) * 2 + 0] = page;
      placement[(static_cast<int64_t>(b) * K + j) * 2 + 1] = static_cast<int32_t>(p % P);
    }
  }
  return 0;
}

// K/V append: copies the block's rows k_block[b][j][h][:], v_block[b][j][h][:]
// (bf16 bits, [B, K, Hkv, D]) into the pool rows of its placement,
// k_pages[page][h][offset][:] and likewise V.  Every other pool row is left as
// it was.  Same return codes as oracle_block_placement.
int oracle_append_block_kv(int B, int K, int Hkv, int D, int P, int max_pages, int num_pages,
                           const uint16_t* k_block, const uint16_t* v_block, uint16_t* k_pages,
                           uint16_t* v_pages, const int32_t* page_table, const int32_t* ctx_lens) {
  std::vector<int32_t> place(static_cast<size_t>(B) * K * 2);
  const int rc = oracle_block_placement(B, K, P, max_pages, num_pages, page_table, ctx_lens,
                                        place.data());
  if (rc != 0) return rc;
  for (int b = 0; b < B; ++b)
    for (int j = 0; j < K; ++j) {
      const int64_t page = place[(static_cast<int64_t>(b) * K + j) * 2 + 0];
      const int64_t off = place[(static_cast<int64_t>(b) * K + j) * 2 + 1];
      for (int h = 0; h < Hkv; ++h) {
        const int64_t src = ((static_cast<int64_t>(b) * K + j) * Hkv + h) * D;
        const int64_t dst = ((page * Hkv + h) * P + off) * D;
        for (int d = 0; d < D; ++d) {
          k_pages[dst + d] = k_block[src + d];
          v_pages[dst + d] = v_block[src + d];
        }
      }
    }
  return 0;
}

}  // extern "C"
