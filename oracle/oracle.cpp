// Test infrastructure -- NOT part of the product.
//
// A plain, slow, obviously-correct CPU oracle for paged-KV grouped-query
// attention (decode and prefix-prefill/extend).  Only the test suite, the
// smoke check and the benchmark's CPU-baseline leg may load this library; the
// product path never does.  It shares no code, header or table with the CUDA
// library: every step below is written out from the definition on the source
// pages, one query row and one head at a time, in double precision.
//
// Sources (web pages; cited by title and section):
//   [TDA] "vllm/attention/ops/triton_decode_attention.py" -- split-KV paged
//         decode: _fwd_grouped_kernel_stage1 (page-table addressing, GQA head
//         map, scale, tanh soft-cap, natural-log LSE), _fwd_kernel_stage2.
//   [PPF] "vllm/attention/ops/prefix_prefill.py" -- context_attention_fwd and
//         _fwd_kernel: context keys unmasked, new keys causal, sliding window
//         keep-rule, fp8 dequantisation (x.to(fp32) * scale).to(q.dtype).
//   [B12] "vllm/v1/attention/backends/b12x" B12xPagedAttentionImpl: kv-cache
//         views [pages, page_size, kv_heads, head_dim], sinks of shape
//         [num_heads] fp32, window_left = sliding_window - 1, seq_lens count
//         cached + new tokens.
//
// The oracle does no splitting, tiling or online softmax: split-KV with an LSE
// merge is an exact re-association of the same sum, so the plain definition
// is the reference for every split count.
//
// Parity status: every function here is pinned by tests/test_oracle_pins.py
// (library routines, closed forms, invariances); none is "parity unpinned".

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>
#include <algorithm>

namespace {

// ---- element decoding --------------------------------------------------------

// bfloat16: the upper 16 bits of an IEEE binary32 value.
double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// OCP FP8 E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
// bits; no infinities; S.1111.111 is NaN; exponent field 0 is subnormal with
// value 2^-6 * m/8.  [PPF] views the uint8 cache as float8_e4m3fn.
double e4m3_to_double(uint8_t code) {
  const int sign = (code >> 7) & 1;
  const int e = (code >> 3) & 0xF;
  const int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return std::numeric_limits<double>::quiet_NaN();
  if (e == 0) {
    mag = std::ldexp(static_cast<double>(m) / 8.0, -6);
  } else {
    mag = std::ldexp(1.0 + static_cast<double>(m) / 8.0, e - 7);
  }
  return sign ? -mag : mag;
}

// Round a binary32 value to bfloat16, round-to-nearest-even (the rounding a
// tensor .to(torch.bfloat16) performs), returned as double.
double round_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) {
    return std::numeric_limits<double>::quiet_NaN();
  }
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  u &= 0xFFFF0000u;
  float r;
  std::memcpy(&r, &u, sizeof r);
  return static_cast<double>(r);
}

// fp8 KV dequantisation as [PPF] _fwd_kernel writes it:
// k = (k_load.to(float32) * k_scale).to(q.dtype), with q in bfloat16.
// The product is a binary32 multiply, then one rounding to bfloat16.
double fp8_dequant(uint8_t code, float scale) {
  const double x = e4m3_to_double(code);
  const float prod = static_cast<float>(x) * scale;  // e4m3 -> fp32 is exact
  return round_to_bf16(prod);
}

// Encode a binary32 value as OCP E4M3 ("e4m3fn"), round to nearest with
// ties to even, saturating to +-448 (the largest finite code) and keeping NaN
// as S.1111.111.  Written from the format: exponent bias 7, 3 mantissa bits,
// subnormals 2^-6 * m/8, no infinities.
uint8_t e4m3_encode(float y) {
  const uint8_t sign = std::signbit(y) ? 0x80 : 0x00;
  if (std::isnan(y)) return sign | 0x7F;
  double a = std::fabs(static_cast<double>(y));
  if (a >= 448.0) return sign | 0x7E;                       // saturate (also +-inf)
  auto rne = [](double v) {                                  // round half to even
    const double f = std::floor(v);
    const double r = v - f;
    if (r > 0.5) return f + 1.0;
    if (r < 0.5) return f;
    return (std::fmod(f, 2.0) == 0.0) ? f : f + 1.0;
  };
  if (a < std::ldexp(1.0, -6)) {                             // subnormal range (and zero)
    const double m = rne(a / std::ldexp(1.0, -9));           // units of 2^-9; m == 8 is 2^-6
    return sign | static_cast<uint8_t>(m);
  }
  int e;
  const double fr = std::frexp(a, &e);                       // a = fr * 2^e, fr in [0.5, 1)
  int ex = e - 1;                                            // a = (1 + f) * 2^ex
  double m = rne((a / std::ldexp(1.0, ex) - 1.0) * 8.0);
  (void)fr;
  if (m >= 8.0) {
    m = 0.0;
    ex += 1;
  }
  const int code = ((ex + 7) << 3) | static_cast<int>(m);
  if (code > 0x7E) return sign | 0x7E;
  return sign | static_cast<uint8_t>(code);
}

}  // namespace

extern "C" {

uint8_t oracle_e4m3_encode(float y) { return e4m3_encode(y); }

// Append new tokens' K/V into the paged cache, as the b12x backend's
// do_kv_cache_update hands them to reshape_and_cache_flash: token t goes to
// page slot_mapping[t] / page_size, slot slot_mapping[t] % page_size (a
// negative slot is padding and is skipped).  bf16 caches store the values;
// e4m3 caches store e4m3(float(x) / scale) (binary32 division, then
// e4m3_encode).  Returns 0, or 1 for a slot outside the pool.
int oracle_append_kv(const uint16_t* k_new, const uint16_t* v_new, int64_t new_stride_tok, int64_t new_stride_head,
                     void* k_cache, void* v_cache, int64_t kv_stride_page, int64_t kv_stride_tok,
                     int64_t kv_stride_head, int num_pages, int page_size, const int64_t* slot_mapping,
                     int num_tokens, int num_kv_heads, int head_dim, int kv_fp8, float k_scale, float v_scale) {
  for (int t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    const int64_t page = slot / page_size;
    const int64_t off = slot % page_size;
    if (page >= num_pages) return 1;
    for (int h = 0; h < num_kv_heads; ++h) {
      for (int d = 0; d < head_dim; ++d) {
        const int64_t src = t * new_stride_tok + h * new_stride_head + d;
        const int64_t dst = page * kv_stride_page + off * kv_stride_tok + h * kv_stride_head + d;
        if (kv_fp8) {
          const float kx = static_cast<float>(bf16_bits_to_double(k_new[src]));
          const float vx = static_cast<float>(bf16_bits_to_double(v_new[src]));
          static_cast<uint8_t*>(k_cache)[dst] = e4m3_encode(kx / k_scale);
          static_cast<uint8_t*>(v_cache)[dst] = e4m3_encode(vx / v_scale);
        } else {
          static_cast<uint16_t*>(k_cache)[dst] = k_new[src];
          static_cast<uint16_t*>(v_cache)[dst] = v_new[src];
        }
      }
    }
  }
  return 0;
}

// Problem description shared with the Python test wrapper (plain C layout).
// Strides are in ELEMENTS of the respective arrays.
typedef struct {
  int mode;            // 0 = decode (one query row per request), 1 = extend
  int batch;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int page_size;
  int num_pages;       // pages in each of k_cache / v_cache
  const uint16_t* q;   // bf16 bits, row r head h at q[r*q_stride_row + h*q_stride_head + d]
  int64_t q_stride_row;
  int64_t q_stride_head;
  const void* k_cache; // bf16 bits (uint16) or e4m3 codes (uint8)
  const void* v_cache;
  int kv_fp8;          // 0 = bf16, 1 = fp8 e4m3 with per-tensor scales
  int64_t kv_stride_page;  // elements between pages
  int64_t kv_stride_tok;   // elements between slots of a page
  int64_t kv_stride_head;  // elements between kv heads of a slot
  const int32_t* block_table;  // [batch, bt_stride]
  int64_t bt_stride;
  const int32_t* seq_lens;     // [batch]; total KV length incl. new tokens
  const int32_t* query_start_loc;  // [batch+1]; extend only
  double scale;
  int window;          // <= 0: off; else keep key j iff pos_q - j < window
  double soft_cap;     // <= 0: off; else s = cap * tanh(s / cap)
  const float* sinks;  // [num_q_heads] or NULL
  float k_scale;
  float v_scale;
  // Per-request descales (the b12x backend's fp8 descale tensors, a scalar
  // expanded to [num_reqs] or given per request): [batch] each, or NULL for
  // the per-tensor k_scale / v_scale above.
  const float* k_scales;
  const float* v_scales;
  const int32_t* rows; // subset of query rows to evaluate, or NULL = all
  int num_rows;        // length of rows (ignored when rows == NULL)
  double* out;         // [n_rows_evaluated, num_q_heads, head_dim]
  double* lse;         // [n_rows_evaluated, num_q_heads]
  int num_threads;
} oracle_problem;

double oracle_bf16_to_double(uint16_t bits) { return bf16_bits_to_double(bits); }
double oracle_e4m3_to_double(uint8_t code) { return e4m3_to_double(code); }
double oracle_fp8_dequant(uint8_t code, float scale) { return fp8_dequant(code, scale); }

// Error codes: 0 ok; 1 bad argument; 2 a block-table entry outside the pool;
// 3 query_start_loc / seq_lens inconsistent.
int oracle_attention(const oracle_problem* P) {
  if (!P || P->batch < 0 || P->num_q_heads <= 0 || P->num_kv_heads <= 0 ||
      P->head_dim <= 0 || P->page_size <= 0 ||
      P->num_q_heads % P->num_kv_heads != 0) {
    return 1;
  }
  if (P->mode != 0 && P->mode != 1) return 1;
  if (P->mode == 1 && !P->query_start_loc) return 1;
  const int B = P->batch;
  const int Hq = P->num_q_heads;
  const int D = P->head_dim;
  const int ps = P->page_size;
  // [TDA] kv_group_num = q heads // kv heads; [PPF] num_queries_per_kv.
  const int G = Hq / P->num_kv_heads;

  const int total_rows = (P->mode == 0) ? B : (B > 0 ? P->query_start_loc[B] : 0);
  const int n_eval = P->rows ? P->num_rows : total_rows;

  // Per-row location: request b and query position pos_q.
  std::vector<int> row_b(n_eval), row_pos(n_eval), row_idx(n_eval);
  for (int k = 0; k < n_eval; ++k) {
    const int r = P->rows ? P->rows[k] : k;
    if (r < 0 || r >= total_rows) return 1;
    int b, pos;
    if (P->mode == 0) {
      // decode: one new token per request, at the last position of the
      // sequence ([TDA]: keys 0 .. seq_len-1 are all visible).
      b = r;
      pos = P->seq_lens[b] - 1;
    } else {
      // extend: [PPF] query_len = seq_len - ctx_len; query i of request b sits
      // at sequence position ctx_len + i.  Rows are packed by query_start_loc.
      b = -1;
      for (int bb = 0; bb < B; ++bb) {
        if (P->query_start_loc[bb] <= r && r < P->query_start_loc[bb + 1]) { b = bb; break; }
      }
      if (b < 0) return 3;
      const int qlen = P->query_start_loc[b + 1] - P->query_start_loc[b];
      const int ctx = P->seq_lens[b] - qlen;
      if (ctx < 0) return 3;
      pos = ctx + (r - P->query_start_loc[b]);
    }
    row_b[k] = b;
    row_pos[k] = pos;
    row_idx[k] = r;
  }

  // Validate every block-table entry any evaluated row can touch.
  for (int k = 0; k < n_eval; ++k) {
    const int b = row_b[k];
    for (int j = 0; j <= row_pos[k]; ++j) {
      const int32_t page = P->block_table[static_cast<int64_t>(b) * P->bt_stride + j / ps];
      if (page < 0 || page >= P->num_pages) return 2;
    }
  }

  auto load_kv = [&](const void* cache, int page, int slot, int kvh, int d, float sc) -> double {
    const int64_t off = static_cast<int64_t>(page) * P->kv_stride_page +
                        static_cast<int64_t>(slot) * P->kv_stride_tok +
                        static_cast<int64_t>(kvh) * P->kv_stride_head + d;
    if (P->kv_fp8) return fp8_dequant(static_cast<const uint8_t*>(cache)[off], sc);
    return bf16_bits_to_double(static_cast<const uint16_t*>(cache)[off]);
  };

  const double NEG_INF = -std::numeric_limits<double>::infinity();

  // One (row, head) evaluation, straight from the definition.
  auto eval_one = [&](int k, int h) {
    const int b = row_b[k];
    const int pos_q = row_pos[k];
    const int r = row_idx[k];
    const int kvh = h / G;  // GQA head map ([TDA] cur_head // kv_group_num)
    // fp8 descales of this request (per request when given, else per tensor)
    const float k_sc = P->k_scales ? P->k_scales[b] : P->k_scale;
    const float v_sc = P->v_scales ? P->v_scales[b] : P->v_scale;
    const uint16_t* qrow = P->q + static_cast<int64_t>(r) * P->q_stride_row +
                           static_cast<int64_t>(h) * P->q_stride_head;

    // 1. Key set J: causal (j <= pos_q) and, with a window, pos_q - j < W
    //    ([PPF] sliding-window condition; [B12] window_left = W - 1).
    std::vector<int> J;
    for (int j = 0; j <= pos_q; ++j) {
      if (P->window > 0 && !(pos_q - j < P->window)) continue;
      J.push_back(j);
    }

    // 2-4. Gather through the block table, score, soft-cap.
    std::vector<double> s(J.size());
    std::vector<double> V(J.size() * static_cast<size_t>(D));  // gathered value rows
    for (size_t t = 0; t < J.size(); ++t) {
      const int j = J[t];
      // [TDA] page = Req_to_tokens[b, j // PAGE_SIZE], slot = j % PAGE_SIZE.
      const int page = P->block_table[static_cast<int64_t>(b) * P->bt_stride + j / ps];
      const int slot = j % ps;
      double dot = 0.0;
      for (int d = 0; d < D; ++d) {
        const double kd = load_kv(P->k_cache, page, slot, kvh, d, k_sc);
        dot += bf16_bits_to_double(qrow[d]) * kd;
        V[t * D + d] = load_kv(P->v_cache, page, slot, kvh, d, v_sc);
      }
      double sj = P->scale * dot;  // [TDA] qk *= sm_scale
      if (P->soft_cap > 0.0) {
        sj = P->soft_cap * std::tanh(sj / P->soft_cap);  // [TDA] after scaling
      }
      s[t] = sj;
    }

    // 5. Normalise.  A sink is one extra logit of the softmax denominator with
    //    no value row (reading of [B12] attention_sink_bias, shape [Hq]).
    const bool has_sink = P->sinks != nullptr;
    const double sink = has_sink ? static_cast<double>(P->sinks[h]) : 0.0;
    double m = NEG_INF;
    for (double v : s) m = std::max(m, v);
    if (has_sink) m = std::max(m, sink);

    double* o = P->out + (static_cast<int64_t>(k) * Hq + h) * D;
    double* lse = P->lse + static_cast<int64_t>(k) * Hq + h;
    if (m == NEG_INF) {  // no key and no sink: empty softmax
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      *lse = NEG_INF;
      return;
    }
    double Z = 0.0;
    std::vector<double> acc(D, 0.0);
    for (size_t t = 0; t < J.size(); ++t) {
      const double w = std::exp(s[t] - m);
      Z += w;
      for (int d = 0; d < D; ++d) acc[d] += w * V[t * D + d];
    }
    if (has_sink) Z += std::exp(sink - m);
    for (int d = 0; d < D; ++d) o[d] = acc[d] / Z;
    *lse = m + std::log(Z);  // natural log, as [TDA] e_max + log(e_sum)
  };

  const int64_t n_items = static_cast<int64_t>(n_eval) * Hq;
  int nt = P->num_threads > 0 ? P->num_threads : 1;
  if (nt > n_items) nt = static_cast<int>(std::max<int64_t>(n_items, 1));
  if (nt <= 1) {
    for (int64_t it = 0; it < n_items; ++it) eval_one(static_cast<int>(it / Hq), static_cast<int>(it % Hq));
  } else {
    std::vector<std::thread> pool;
    for (int t = 0; t < nt; ++t) {
      pool.emplace_back([&, t]() {
        for (int64_t it = t; it < n_items; it += nt) {
          eval_one(static_cast<int>(it / Hq), static_cast<int>(it % Hq));
        }
      });
    }
    for (auto& th : pool) th.join();
  }
  return 0;
}

}  // extern "C"
