// Prefix-prefill / extend over the paged KV cache on the 5th-generation tensor
// cores (tcgen05, TMEM accumulators, TMA operand loads).
//
// Operation: "vllm/attention/ops/prefix_prefill.py", context_attention_fwd /
// _fwd_kernel: query i of request b sits at sequence position
// ctx_b + i (ctx_b = seq_len - query_len) and attends to every key j <= its
// position (the cached context unmasked, the new tokens causally), within the
// sliding window when one is set; all keys are read from the pages, as in the
// b12x backend ("vllm/v1/attention/backends/b12x", forward), where the new
// tokens are appended before attention runs.
//
// Design (GB300):
//   * Tile = 128 query rows x one kv head: the G q heads of each token are
//     packed into the MMA M dimension (row = token * G + head), so one K/V
//     tile feeds all heads that share it.
//   * Warp roles in a 256-thread CTA: warps 0 and 2 issue TMA (Q once, then
//     the K ring and the V ring: one box per page, page ids from the block
//     table), warp 1 allocates TMEM and issues the S = Q K^T MMAs, warp 7
//     issues the O += P V MMAs (one thread each: an MMA issue blocks while
//     the tensor pipe is busy, so one issuer would hold a ready PV behind the
//     next tile's QK), warps 3-6 run the softmax with one TMEM lane (= one
//     query row) per thread.  Two CTAs share an SM where TMEM and shared
//     memory allow.
//   * S = Q K^T (M=128, N=BN keys) lands in one of NSB TMEM buffers (as
//     many as fit beside O: 2 for head_dim 128), so the next tiles' QK
//     overlaps this tile's softmax (a buffer is reused once the PV that read
//     its P has completed); P (bf16) is written back
//     over S and consumed from TMEM by O += P V (V read MN-major from shared
//     memory); O stays in TMEM for the whole key loop.  The softmax releases
//     P in two 32-key halves on separate barriers, so PV starts on the first
//     half while the second half's exponentials run.
//   * head_dim 256 (one CTA per SM): the first half of Q's dims also lives
//     in TMEM, copied there by the softmax warps from its TMA staging area in
//     the last K ring stage, so half of QK's K steps read only K from shared
//     memory; the rings are three stages deep and three S buffers fit.
//   * Online softmax in the log2 domain with lazy rescaling: O and l are
//     rescaled only when the row maximum grows by more than 2^8, which is
//     exact because the final normalisation uses the same stale maximum.
//   * Key tiles wholly outside [first key of the window, last query] are not
//     visited; pages outside [window start, sequence end) are fetched as
//     out-of-bounds TMA boxes (zero fill), and value rows past the sequence end
//     inside the last page are zeroed, so stale or NaN slots never meet P = 0.
//   * A one-CTA scheduler kernel builds the (request, query tile) list from
//     the device metadata, heaviest first, each entry carrying the request's
//     query start, query count and length; CTA i takes item i / Hkv.
//   * e4m3 cache: a call first writes bf16(float(code) * scale) of every
//     attended page into a copy in the scratch workspace
//     (extend_kv_copy_kernel) and this kernel reads the copy; plans whose
//     copy would not fit dequantise each tile in shared memory instead (the
//     TMA producer warps convert it in place).  Either way the MMAs see the
//     same bf16 values.
#include <climits>
#include <cmath>
#include <cstdint>
#include <type_traits>

#include "extend.h"
#include "pa_internal.h"
#include "tcgen05.cuh"

namespace pa {
namespace {

constexpr int kThreads = 256;     // warps: 0 = Q/K TMA, 1 = QK MMA, 2 = V TMA, 3-6 = softmax, 7 = PV MMA
constexpr int kRows = 128;           // MMA M: query rows per tile
constexpr int kSchedThreads = 1024;
constexpr int kBuckets = 256;        // work classes for the longest-first order
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 2^8

struct ExtendParams {
  const int32_t* seq_lens;
  const int32_t* qsl;
  const int32_t* block_table;
  int64_t bt_stride;
  int batch, total_q, num_q_heads, num_kv_heads, group, page_size, num_pages;
  int tm;                 // tokens per tile (128 / group, rounded down)
  int max_kv;             // capacity: keys per request
  int block_n;            // keys per tile
  float scale_log2, cap_log2, scale_over_cap;
  int window;
  const float* sinks;
  float k_scale, v_scale;   // fp8 cache: per-tensor dequantisation scales
  const float* k_scales;    // fp8 cache: [B] per-request scales replacing them, or null
  const float* v_scales;
  uint16_t* out;
  int64_t out_stride_tok, out_stride_head;
  float* lse;
  int4* work;               // [work_cap][2]: WorkItem
  int* work_count;
  int work_cap;
  uint32_t* err;
};

// A work item: query tile mt of request b, with the request's first query
// row, query count and sequence length (read from the metadata once, by the
// scheduler), 32 bytes.
struct WorkItem {
  int b, mt, qs, qlen, L, pad0, pad1, pad2;
};
static_assert(sizeof(WorkItem) == 32, "two 16-byte loads per item");

__device__ __forceinline__ WorkItem load_item(const ExtendParams& p, int idx) {
  const int4 a = p.work[2 * idx];
  const int4 c = p.work[2 * idx + 1];
  return WorkItem{a.x, a.y, a.z, a.w, c.x, 0, 0, 0};
}

// Key tiles an item touches (its cost), from the rows it holds.
__device__ __forceinline__ bool item_range(const ExtendParams& p, const WorkItem& it, int& qs, int& qlen, int& ctx,
                                           int& t0, int& t_end, int& lo_min, int& kt0, int& n_tiles) {
  qs = it.qs;
  qlen = it.qlen;
  const int L = it.L;
  const int mt = it.mt;
  ctx = L - qlen;
  t0 = mt * p.tm;
  if (qlen <= 0 || ctx < 0 || L > p.max_kv || qs < 0 || qs + qlen > p.total_q || t0 >= qlen) return false;
  t_end = min(qlen, t0 + p.tm);
  const int pos_min = ctx + t0;
  const int pos_max = ctx + t_end - 1;
  lo_min = p.window > 0 ? max(0, pos_min - p.window + 1) : 0;
  kt0 = lo_min / p.block_n;
  n_tiles = pos_max / p.block_n - kt0 + 1;
  return true;
}

// Key tiles of query tile mt of a request (its cost): keys from the window
// start of its first row to its last row's position.
__device__ __forceinline__ int tile_cost(int ctx, int qlen, int mt, int tm, int window, int bn) {
  const int t0 = mt * tm;
  const int t_end = min(qlen, t0 + tm);
  const int pos_min = ctx + t0;
  const int pos_max = ctx + t_end - 1;
  const int lo = window > 0 ? max(0, pos_min - window + 1) : 0;
  return pos_max / bn - lo / bn + 1;
}

__global__ void __launch_bounds__(kSchedThreads) extend_schedule_kernel(const ExtendParams p) {
  // the attention kernel may start launching now; it waits for this grid's
  // results (griddepcontrol.wait) before it reads the work list
  pdl_launch_dependents();
  __shared__ int s_hist[kBuckets];
  __shared__ int s_off[kBuckets];
  __shared__ int s_total;
  const int tid = threadIdx.x;
  for (int i = tid; i < kBuckets; i += kSchedThreads) s_hist[i] = 0;
  if (tid == 0) s_total = 0;
  __syncthreads();
  // one warp per request, its lanes over the request's query tiles: the
  // attention kernel waits for this list, so it is built in few rounds
  const int warp = tid >> 5;
  const int lane = tid & 31;
  constexpr int kSchedWarps = kSchedThreads / 32;
  for (int b = warp; b < p.batch; b += kSchedWarps) {
    const int qs = p.qsl[b];
    const int qlen = p.qsl[b + 1] - qs;
    const int L = p.seq_lens[b];
    if (qlen == 0) continue;
    if (qlen < 0 || L < qlen || L > p.max_kv || qs < 0 || qs + qlen > p.total_q) {
      if (lane == 0) atomicOr(p.err, kErrCapacity);
      continue;
    }
    const int nmt = (qlen + p.tm - 1) / p.tm;
    for (int mt = lane; mt < nmt; mt += 32) {
      atomicAdd(&s_hist[min(tile_cost(L - qlen, qlen, mt, p.tm, p.window, p.block_n), kBuckets - 1)], 1);
    }
    if (lane == 0) atomicAdd(&s_total, nmt);
  }
  __syncthreads();
  // descending exclusive scan: heaviest class first (one warp, 8 classes per lane)
  if (tid < 32) {
    constexpr int per_lane = kBuckets / 32;
    int vals[per_lane];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < per_lane; ++i) {
      vals[i] = s_hist[kBuckets - 1 - (tid * per_lane + i)];
      sum += vals[i];
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (tid >= off) incl += v;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < per_lane; ++i) {
      s_off[kBuckets - 1 - (tid * per_lane + i)] = run;
      run += vals[i];
    }
  }
  __syncthreads();
  for (int b = warp; b < p.batch; b += kSchedWarps) {
    const int qs = p.qsl[b];
    const int qlen = p.qsl[b + 1] - qs;
    const int L = p.seq_lens[b];
    if (qlen <= 0 || L < qlen || L > p.max_kv || qs < 0 || qs + qlen > p.total_q) continue;
    const int nmt = (qlen + p.tm - 1) / p.tm;
    for (int mt = lane; mt < nmt; mt += 32) {
      const int pos = atomicAdd(&s_off[min(tile_cost(L - qlen, qlen, mt, p.tm, p.window, p.block_n), kBuckets - 1)], 1);
      if (pos < p.work_cap) {
        p.work[2 * pos] = make_int4(b, mt, qs, qlen);
        p.work[2 * pos + 1] = make_int4(L, 0, 0, 0);
      }
    }
  }
  if (tid == 0) {
    int total = s_total;
    if (total > p.work_cap) {
      atomicOr(p.err, kErrSchedOverflow);
      total = p.work_cap;
    }
    *p.work_count = total;
  }
}

// tanh(x) = 1 - 2 / (e^(2x) + 1), from the definition, with the hardware
// exp2 and a fast reciprocal: absolute error ~1e-7 (so ~5e-6 on a logit
// capped at 50), and few registers -- it is inlined once per score.
__device__ __forceinline__ float tanh_exp2(float x) {
  const float e = ex2(x * 2.8853900817779268f);  // e^(2x) = 2^(2x log2 e)
  return 1.f - __fdividef(2.f, e + 1.f);
}

// Exact softmax weights on a key tile: P = P_hi + P_lo (two bf16 halves, two
// PV MMAs, exact to ~2^-17) when some query row's largest weight from the
// tile exceeds 1 / kHotShare of its running denominator (a row that attends
// few keys, or whose weight sits on a few dominant keys).  One bf16 P is up to
// 2^-8 off per weight, which such rows do not average out; the denominator
// only grows, so every key of a tile given one bf16 P ends with a final
// weight below 1 / kHotShare.  Each softmax warp flags the tiles where one
// of its rows needs it; the PV issuer adds the P_lo pass when any did.
constexpr float kHotShare = 8.f;

template <int D, int BN, int NST, int CPS, bool FP8 = false>
struct ExtTraits {
  static constexpr int NCH = D / 64;                 // 128-byte column chunks per row
  static constexpr int Q_CHUNK = kRows * 128;        // 16 KB
  static constexpr int Q_BYTES = NCH * Q_CHUNK;
  static constexpr int KV_CHUNK = BN * 128;
  static constexpr int TILE = NCH * KV_CHUNK;        // K (or V) tile
  // head_dim 256 (bf16 tiles): the first half of Q's dims is held in TMEM,
  // so half of QK's K steps read only K from shared memory; that half lands
  // first in the last K stage of the ring and is copied to TMEM before the
  // stage is filled, the other half keeps its own area.  This leaves room
  // for three ring stages and three S buffers
  static constexpr bool QT = (D == 256) && !FP8;
  static constexpr int Q_TM_CH = QT ? NCH / 2 : 0;   // Q chunks held in TMEM
  static constexpr int SMEM_DATA = (NCH - Q_TM_CH) * Q_CHUNK + 2 * NST * TILE;  // Q, K ring, V ring
  // fp8 cache: the e4m3 tile lands in the second half of the bf16 stage
  // buffer, rows of RB8 bytes (row r under bf16 row r's upper chunks when
  // D >= 128), and is dequantised in place
  static constexpr int RB8 = D < 128 ? D : 128;      // bytes per fp8 box row
  static constexpr int NCC8 = D / RB8;               // fp8 boxes per page
  static constexpr int F8_OFF = TILE / 2;
  static constexpr uint32_t TMEM_COLS = 512 / CPS;   // CPS CTAs share an SM's 512 columns
  // S buffers: as many as the columns left beside O hold (2 for head_dim
  // 128, 3 for 64, 3 for 256 with one CTA per SM and half of Q in TMEM, 4
  // for its e4m3 form); QK runs up to NSB - 1
  // tiles ahead of the softmax
  static constexpr int Q_COLS = Q_TM_CH * 32;       // Q in TMEM: bf16 pairs, 32 columns per chunk
  static constexpr int NSB = (static_cast<int>(TMEM_COLS) - D - Q_COLS) / BN;
  static constexpr uint32_t TMEM_O = NSB * BN;       // S buffers, then O, then Q
  static constexpr uint32_t TMEM_Q = TMEM_O + D;
  static_assert(NSB >= 2 && NSB * BN + D + Q_COLS <= static_cast<int>(TMEM_COLS), "TMEM plan: S buffers, O, Q");
  static_assert(!QT || (NST >= 2 && Q_TM_CH * Q_CHUNK <= TILE), "Q staged in the last K stage");
  // S buffer of tile j and the phase parity of its barriers (unsigned: a
  // power-of-two count reduces to a mask and a shift)
  __device__ static __forceinline__ int sbuf(int j) {
    return static_cast<int>(static_cast<unsigned>(j) % static_cast<unsigned>(NSB));
  }
  __device__ static __forceinline__ uint32_t sphase(int j) {
    return (static_cast<unsigned>(j) / static_cast<unsigned>(NSB)) & 1u;
  }
  // mbarriers: q_full, six per ring stage, s_full/2 x p_half/o_done per S
  // buffer, q_moved (Q in TMEM)
  // then the TMEM address and 4 exact-P flag bytes per S buffer (one per
  // softmax warp)
  static constexpr int BAR_BYTES = ((1 + 6 * NST + 4 * NSB + (QT ? 1 : 0)) * 8 + 4 + 4 * NSB + 15) / 16 * 16;
  static constexpr int SMEM = 1024 + SMEM_DATA + BAR_BYTES;   // 1024: alignment slack for SW128
  static_assert(CPS * SMEM <= 232448, "shared memory for CPS CTAs per SM");
  static_assert(BN % 64 == 0, "P is stored 32 columns (64 keys) at a time");
};

// In-place dequantisation of one e4m3 K or V tile (BN rows) into the bf16
// layout the MMA reads (rows of 64-element chunks, 128-byte swizzle), by one
// warp: element = bf16(float(code) * scale), as the prefix-prefill page does.
template <int D, int BN, int NST, int CPS>
__device__ __forceinline__ void dequant_tile(uint8_t* tile, float scale, int lane) {
  using T = ExtTraits<D, BN, NST, CPS, true>;
  constexpr int UPR = T::RB8 / 16;         // 16-byte fp8 units per box row
  constexpr int U = T::NCC8 * UPR;         // units per key row
  const uint8_t* f8 = tile + T::F8_OFF;
  const uint64_t scale2 = dequant_scale2(scale);
  auto out_unit = [&](int r, int d16, const uint4& w) {
    // 16 codes = dims [16 d16, 16 d16 + 16) -> two 16-byte bf16 units
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      o[2 * k] = dequant_e4m3x2<0>(wv[k], scale2);
      o[2 * k + 1] = dequant_e4m3x2<1>(wv[k], scale2);
    }
    const int chunk = d16 >> 2;
    const int unit0 = (d16 & 3) * 2;
    uint8_t* rowp = tile + chunk * T::KV_CHUNK + r * 128;
    *reinterpret_cast<uint4*>(rowp + (((unit0) ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(rowp + (((unit0 + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
  };
  auto in_unit = [&](int r, int u) -> uint4 {
    const int box = u / UPR, uu = u % UPR;
    const int sw = T::RB8 == 128 ? (r & 7) : ((r >> 1) & 3);
    return *reinterpret_cast<const uint4*>(f8 + box * BN * T::RB8 + r * T::RB8 + ((uu ^ sw) << 4));
  };
  if constexpr (D >= 128) {
    // row r's e4m3 bytes lie under its own upper bf16 chunks: read the row, then write it
#pragma unroll
    for (int r = lane; r < BN; r += 32) {
      uint4 w[U];
#pragma unroll
      for (int u = 0; u < U; ++u) w[u] = in_unit(r, u);
#pragma unroll
      for (int u = 0; u < U; ++u) out_unit(r, u, w[u]);
    }
  } else {
    // 64-byte e4m3 rows straddle other rows' bf16 rows: read the whole tile first
    constexpr int RPT = BN / 32;
    uint4 w[RPT][U];
#pragma unroll
    for (int k = 0; k < RPT; ++k)
#pragma unroll
      for (int u = 0; u < U; ++u) w[k][u] = in_unit(lane + 32 * k, u);
    __syncwarp();
#pragma unroll
    for (int k = 0; k < RPT; ++k)
#pragma unroll
      for (int u = 0; u < U; ++u) out_unit(lane + 32 * k, u, w[k][u]);
  }
}

// Two CTAs per SM cap a thread at 128 registers (allocation counts 8 warps).
template <int D, int BN, int NST, int CPS, bool FP8>
__global__ void __launch_bounds__(kThreads, CPS)
extend_attn_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const ExtendParams p) {
  using T = ExtTraits<D, BN, NST, CPS, FP8>;
  const int idx = blockIdx.x / p.num_kv_heads;
  const int kvh = blockIdx.x - idx * p.num_kv_heads;
  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmq);
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  pdl_wait_primary();  // the scheduler's work list is complete and visible
  // the count and this CTA's entry in one round trip (idx < the list's
  // capacity: the entry is read only when idx < count)
  const int count = *p.work_count;
  const WorkItem item = load_item(p, idx);
  if (idx >= count) return;
  // another CTA's wait already expired: leave (CTA-uniform, before any TMEM
  // allocation).  Other error bits (a bad request or page id) leave the rest
  // of the call running.
  if (__syncthreads_or(threadIdx.x == 0 &&
                       (*reinterpret_cast<volatile uint32_t*>(p.err) & kErrWaitTimeout) != 0u))
    return;
  const int b = item.b;
  int qs, qlen, ctx, t0, t_end, lo_min, kt0, n;
  if (!item_range(p, item, qs, qlen, ctx, t0, t_end, lo_min, kt0, n)) return;
  const int L = ctx + qlen;
  const int G = p.group;
  const int ps = p.page_size;
  const int ps_log2 = __ffs(ps) - 1;   // page sizes are powers of two: no integer division in the loops

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* k_s = smem + (T::NCH - T::Q_TM_CH) * T::Q_CHUNK;
  uint8_t* v_s = k_s + NST * T::TILE;
  // Q chunk c (64 dims of the 128 rows): the chunks held in TMEM are staged
  // in the last K stage, the others have their own area
  auto q_chunk = [&](int c) -> uint8_t* {
    return c < T::Q_TM_CH ? k_s + (NST - 1) * T::TILE + c * T::Q_CHUNK
                          : smem + (c - T::Q_TM_CH) * T::Q_CHUNK;
  };
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::SMEM_DATA);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + NST;
  uint64_t* v_full = k_empty + NST;
  uint64_t* v_empty = v_full + NST;
  uint64_t* k_land = v_empty + NST;   // fp8: the e4m3 tile has landed (before dequantisation)
  uint64_t* v_land = k_land + NST;
  uint64_t* s_full = v_land + NST;
  uint64_t* p_half = s_full + T::NSB;      // [NSB][2]: a 32-key half of P stored (4 arrivals)
  uint64_t* o_done = p_half + 2 * T::NSB;
  uint64_t* q_moved = o_done + T::NSB;   // Q in TMEM: the softmax warps copied it (4 arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_moved + (T::QT ? 1 : 0));
  uint8_t* vflag = reinterpret_cast<uint8_t*>(tmem_slot + 1);   // [NSB][4]: softmax warp wants exact P

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // page coordinate of this lane's page of key tile j (TMA producers); pages
  // with no attended key are fetched out of bounds, where TMA writes zeros
  // (and so are ids outside the pool, which are flagged: the rest of the
  // call is unaffected)
  const int32_t* bt_row = p.block_table + static_cast<int64_t>(b) * p.bt_stride;
  auto page_coord = [&](int j) {
    const int pg = (((kt0 + j) * BN) >> ps_log2) + lane;
    const bool outside = (pg * ps >= L) || ((pg + 1) * ps <= lo_min);
    if (outside) return p.num_pages;
    const int id = bt_row[pg];
    if (static_cast<unsigned>(id) < static_cast<unsigned>(p.num_pages)) return id;
    atomicOr(p.err, kErrPageId);
    return p.num_pages;
  };
  // the producers read the first tile's page ids while the CTA sets up
  const int npg = BN >> ps_log2;
  const int coord0 = ((warp == 0 || warp == 2) && lane < npg) ? page_coord(0) : 0;

  if (warp == 1) tmem_alloc(tmem_slot, T::TMEM_COLS);
  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NST; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&k_land[i], 1);
      mbar_init(&v_land[i], 1);
    }
    for (int i = 0; i < T::NSB; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_half[2 * i], 4);
      mbar_init(&p_half[2 * i + 1], 4);
      mbar_init(&o_done[i], 1);
    }
    if (T::QT) mbar_init(q_moved, 4);
    fence_mbar_init();
    // Q right away (the other threads wait on q_full after the barrier below)
    mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(T::NCH * p.tm * G * 128));
#pragma unroll
    for (int c = 0; c < T::NCH; ++c) tma_load_3d(q_chunk(c), &tmq, c * 64, kvh * G, qs + t0, q_full);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0 || warp == 2) {
    // ---------------- TMA producers: warp 0 -> the K ring (Q was issued above), warp 2 -> the V ring ----------------
    const bool is_k = warp == 0;
    const CUtensorMap* map = is_k ? &tmk : &tmv;
    uint64_t* full = is_k ? k_full : v_full;
    uint64_t* empty = is_k ? k_empty : v_empty;
    uint8_t* ring = is_k ? k_s : v_s;
    bool ok = true;
    if constexpr (!FP8) {
      for (int j = 0; j < n && ok; ++j) {
        const int stage = j % NST;
        if (j >= NST) ok = __all_sync(0xffffffffu, wait_or_abort(&empty[stage], ((j / NST) - 1) & 1, p.err));
        if constexpr (T::QT) {
          // the last K stage holds Q's first chunks until the softmax warps
          // have copied them to TMEM
          if (is_k && j == NST - 1) {
            ok = ok && __all_sync(0xffffffffu, wait_or_abort(q_moved, 0, p.err));
            fence_proxy_async_smem();
          }
        }
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(T::TILE));
        __syncwarp();
        if (lane < npg) {
          const int coord = j == 0 ? coord0 : page_coord(j);
          uint8_t* dst = ring + stage * T::TILE + lane * ps * 128;
#pragma unroll
          for (int c = 0; c < T::NCH; ++c) tma_load_4d(dst + c * T::KV_CHUNK, map, c * 64, kvh, 0, coord, &full[stage]);
        }
      }
    } else {
      // e4m3 tiles land in the stage (NST ahead), then this warp dequantises
      // them in place and marks the stage full
      uint64_t* land = is_k ? k_land : v_land;
      const float* per_req = is_k ? p.k_scales : p.v_scales;
      const float scale = per_req != nullptr ? per_req[b] : (is_k ? p.k_scale : p.v_scale);
      auto fetch = [&](int j) {
        const int stage = j % NST;
        if (lane == 0) mbar_arrive_expect_tx(&land[stage], static_cast<uint32_t>(BN * D));
        __syncwarp();
        if (lane < npg) {
          const int coord = j == 0 ? coord0 : page_coord(j);
          uint8_t* dst = ring + stage * T::TILE + T::F8_OFF + lane * ps * T::RB8;
#pragma unroll
          for (int c = 0; c < T::NCC8; ++c)
            tma_load_4d(dst + c * BN * T::RB8, map, c * T::RB8, kvh, 0, coord, &land[stage]);
        }
      };
      for (int j = 0; j < n && j < NST; ++j) fetch(j);
      for (int j = 0; j < n && ok; ++j) {
        const int stage = j % NST;
        ok = __all_sync(0xffffffffu, wait_or_abort(&land[stage], (j / NST) & 1, p.err));
        if (!ok) break;
        dequant_tile<D, BN, NST, CPS>(ring + stage * T::TILE, scale, lane);
        fence_proxy_async_smem();   // generic writes -> tensor-core reads
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[stage]);
        const int jn = j + NST;
        if (jn < n) {
          ok = __all_sync(0xffffffffu, wait_or_abort(&empty[stage], ((jn / NST) - 1) & 1, p.err));
          if (!ok) break;
          fetch(jn);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- S = Q K^T issuer (one thread) ----------------
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(kRows, BN, false, false);
      const uint32_t q_u = smem_u32(q_chunk(T::Q_TM_CH));   // first Q chunk in its own area
      const uint32_t k_ring = smem_u32(k_s);
      bool ok = wait_or_abort(q_full, 0, p.err);
      if (T::QT) ok = ok && wait_or_abort(q_moved, 0, p.err);
      tc_fence_after();
      for (int j = 0; j < n && ok; ++j) {
        const int stage = j % NST;
        ok = poll_or_abort(&k_full[stage], (j / NST) & 1, p.err);
        // S buffer j % NSB holds P of tile j - NSB until the PV that reads it has completed
        if (ok && j >= T::NSB) ok = poll_or_abort(&o_done[T::sbuf(j)], T::sphase(j - T::NSB), p.err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tS = tbase + static_cast<uint32_t>(T::sbuf(j) * BN);
        const uint32_t k_u = k_ring + stage * T::TILE;
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint64_t bd = sdesc_sw128(k_u + (s >> 2) * T::KV_CHUNK + (s & 3) * 32, 16, 1024);
          if (s < T::Q_TM_CH * 4) {
            // A = Q from TMEM: k-step s is 16 dims, 8 columns
            umma_ts(tS, tbase + T::TMEM_Q + static_cast<uint32_t>(s * 8), bd, idesc_qk, s > 0 ? 1u : 0u);
          } else {
            const uint64_t ad = sdesc_sw128(q_u + ((s >> 2) - T::Q_TM_CH) * T::Q_CHUNK + (s & 3) * 32, 16, 1024);
            umma_ss(tS, ad, bd, idesc_qk, s > 0 ? 1u : 0u);
          }
        }
        umma_commit(&s_full[T::sbuf(j)]);
        umma_commit(&k_empty[stage]);
      }
    }
  } else if (warp == 7) {
    // ---------------- O += P V issuer (one thread) ----------------
    if (lane == 0) {
      constexpr uint32_t idesc_pv = idesc_bf16(kRows, D, false, true);
      const uint32_t v_ring = smem_u32(v_s);
      bool ok = true;
      for (int jj = 0; jj < n && ok; ++jj) {
        const int st = jj % NST;
        ok = poll_or_abort(&p_half[2 * T::sbuf(jj)], T::sphase(jj), p.err) &&
             poll_or_abort(&v_full[st], (jj / NST) & 1, p.err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tP = tbase + static_cast<uint32_t>(T::sbuf(jj) * BN);
        const uint32_t v_u = v_ring + st * T::TILE;
        // P columns: k-step s (16 keys): P_hi at 8s, P_lo at 32 + 8s; the
        // P_lo pass runs when a softmax warp flagged the tile (flags written
        // before the warps released the first half of P).  Steps 0 and 1
        // need only the first half.
        const uint32_t hot = *reinterpret_cast<volatile const uint32_t*>(vflag + 4 * T::sbuf(jj));
#pragma unroll
        for (int s = 0; s < BN / 16; ++s) {
          if (s == 2) {
            ok = poll_or_abort(&p_half[2 * T::sbuf(jj) + 1], T::sphase(jj), p.err);
            if (!ok) break;
            tc_fence_after();
          }
          const uint64_t bd = sdesc_sw128(v_u + s * 16 * 128, T::KV_CHUNK, 1024);
          umma_ts(tbase + T::TMEM_O, tP + s * 8, bd, idesc_pv, (jj > 0 || s > 0) ? 1u : 0u);
        }
        if (!ok) break;
        if (hot != 0u) {
          // P_lo pass over the rows (TMEM lanes) of the warps that flagged the tile
          uint32_t mask[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) mask[q] = ((hot >> (8 * q)) & 0xffu) ? 0u : 0xffffffffu;
#pragma unroll
          for (int s = 0; s < BN / 16; ++s) {
            const uint64_t bd = sdesc_sw128(v_u + s * 16 * 128, T::KV_CHUNK, 1024);
            umma_ts_masked(tbase + T::TMEM_O, tP + 32 + s * 8, bd, idesc_pv, 1u, mask);
          }
        }
        umma_commit(&o_done[T::sbuf(jj)]);
        umma_commit(&v_empty[st]);
      }
    }
  } else {
    // ---------------- softmax warpgroup: one query row per thread ----------------
    // warps 3-6 cover the four TMEM lane quarters (a warp may only access
    // lanes 32 * (warp % 4) .. + 31)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const int tok = t0 + r / G;
    const int hh = r - (r / G) * G;
    const bool row_ok = (r < p.tm * G) && (tok < qlen);
    const int pos = ctx + min(tok, t_end - 1);
    const int lo = p.window > 0 ? pos - p.window + 1 : INT_MIN / 2;
    const bool capped = p.cap_log2 > 0.f;
    const bool plain = !capped && p.scale_log2 > 0.f;
    const int l_pad = ((L + ps - 1) >> ps_log2) << ps_log2;   // end of the last page
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    if constexpr (T::QT) {
      // Q row r (= TMEM lane r) from its staging chunks into TMEM columns
      // TMEM_Q + 32c .. + 31 (dims 64c + 2w, 64c + 2w + 1 in column w); the
      // 16-byte units of a 128-byte row are XOR-swizzled by (row & 7)
      ok = __all_sync(0xffffffffu, wait_or_abort(q_full, 0, p.err));
      if (ok) {
#pragma unroll 1
        for (int c = 0; c < T::Q_TM_CH; ++c) {
          const uint8_t* row = q_chunk(c) + r * 128;
          uint32_t u[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint4 w = *reinterpret_cast<const uint4*>(row + ((k ^ (r & 7)) << 4));
            u[4 * k] = w.x;
            u[4 * k + 1] = w.y;
            u[4 * k + 2] = w.z;
            u[4 * k + 3] = w.w;
          }
          tmem_st32(tbase + lane_off + T::TMEM_Q + static_cast<uint32_t>(c * 32), u);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_moved);
      }
    }
    for (int j = 0; j < n && ok; ++j) {
      const int k0 = (kt0 + j) * BN;
      ok = __all_sync(0xffffffffu, wait_or_abort(&s_full[T::sbuf(j)], T::sphase(j), p.err));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tS = tbase + lane_off + static_cast<uint32_t>(T::sbuf(j) * BN);
      uint32_t sr[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
      tmem_wait_ld();
      const bool full = (k0 >= lo) && (k0 + BN - 1 <= pos);
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = -INFINITY;
      if (plain) {
        // raw scores: masked keys become -inf (it stays -inf through the
        // positive scale); the max is taken raw and the scale folds into the
        // exponent's FFMA
        if (!full) {
#pragma unroll
          for (int i = 0; i < BN; ++i)
            if (k0 + i > pos || k0 + i < lo) sr[i] = __float_as_uint(-INFINITY);
        }
#pragma unroll
        for (int i = 0; i < BN / 2; ++i)
          mx8[i & 7] = fmax3(mx8[i & 7], __uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1]));
      } else {
        // soft-cap (or a non-positive scale): transform every score first
#pragma unroll
        for (int i = 0; i < BN; ++i) {
          float v = __uint_as_float(sr[i]);
          v = capped ? p.cap_log2 * tanh_exp2(v * p.scale_over_cap) : v * p.scale_log2;
          if (!full && (k0 + i > pos || k0 + i < lo)) v = -INFINITY;
          sr[i] = __float_as_uint(v);
          mx8[i & 7] = fmaxf(mx8[i & 7], v);
        }
      }
      float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
      if (plain) mx *= p.scale_log2;
      const float m_new = fmaxf(m_run, mx);
      const bool need = m_new > m_run + kRescaleThreshold;
      const bool any_need = __any_sync(0xffffffffu, need);
      const float m_use = need ? m_new : m_run;
      const float m_base = (m_use == -INFINITY) ? 0.f : m_use;
      const float alpha = (m_use == m_run || m_use == -INFINITY) ? 1.f : ex2(m_run - m_use);
      // Does some row of this warp take more than 1/kHotShare of its running
      // denominator from one key of the tile?  Decided before the
      // exponentials on a lower bound of the new denominator (the old one
      // rescaled, plus the tile's largest weight pm, with mx in the
      // exponent's units; -inf gives 0): a superset of such rows.
      const float pm = ex2(mx - m_base);
      const bool hot = __any_sync(0xffffffffu, row_ok && pm * (kHotShare - 1.f) > l_run * alpha);
      // O is rescaled and value rows past the sequence end are zeroed before
      // any P is released: PV of this tile may start on its first half
      if (any_need && j > 0) {
        // O must hold PV of tile j-1 before it is rescaled (and no PV may run meanwhile)
        ok = __all_sync(0xffffffffu, wait_or_abort(&o_done[T::sbuf(j - 1)], T::sphase(j - 1), p.err));
        if (!ok) break;
        tc_fence_after();
        const uint32_t tO = tbase + lane_off + T::TMEM_O;
        // 16 columns at a time: the tile's 64 scores are live here
#pragma unroll 1
        for (int c = 0; c < D / 16; ++c) {
          uint32_t u[16];
          tmem_ld16(tO + c * 16, u);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            const float2 v = __fmul2_rn(make_float2(__uint_as_float(u[i]), __uint_as_float(u[i + 1])),
                                        make_float2(alpha, alpha));
            u[i] = __float_as_uint(v.x);
            u[i + 1] = __float_as_uint(v.y);
          }
          tmem_st16(tO + c * 16, u);
        }
        tmem_wait_st();
      }
      // value rows past the sequence end inside the last page of this tile
      const int pend = min(k0 + BN, l_pad);
      if (L < pend) {
        // V of this tile must have landed before its rows are overwritten
        ok = __all_sync(0xffffffffu, wait_or_abort(&v_full[j % NST], (j / NST) & 1, p.err));
        if (!ok) break;
        uint8_t* vs = v_s + (j % NST) * T::TILE;
        const int nrows = pend - L;
        const int units = nrows * T::NCH * 8;   // 16-byte units
        for (int u = r; u < units; u += kRows) {
          const int row = (L - k0) + u / (T::NCH * 8);
          const int c = (u / 8) % T::NCH;
          *reinterpret_cast<uint4*>(vs + c * T::KV_CHUNK + row * 128 + (u & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      if (lane == 0) vflag[4 * T::sbuf(j) + wq] = hot ? 1 : 0;   // read by the PV issuer after p_half
      // exponentials with packed fp32x2 FFMA / FADD (moving part of them to a
      // polynomial on the FMA pipe was measured slower: issue-bound, not
      // MUFU-bound).  P_hi of pair i overwrites score register i (the pairs
      // read before it) and lands in TMEM column i; a hot warp also stores
      // each 16-key block's 8 P_lo columns at 32 + 8 b as soon as they exist.
      // The PV issuer runs the P_lo pass with the rows of the other warps
      // masked, so their columns 32 .. 63 (old scores) are never read into O.
      // Each 32-key half of P is released on its own barrier as soon as it
      // is stored, so the first two PV MMAs overlap the second half's
      // exponentials.
      static_assert(BN == 64, "P is released in two 32-key halves of 16 columns");
      const float am = plain ? p.scale_log2 : 1.f;
      const float2 am2 = make_float2(am, am);
      const float2 nm2 = make_float2(-m_base, -m_base);
      float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      auto release = [&](int half) {
        tmem_st16(tS + 16 * half, *reinterpret_cast<const uint32_t(*)[16]>(&sr[16 * half]));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_half[2 * T::sbuf(j) + half]);
      };
      if (hot) {
#pragma unroll
        for (int blk = 0; blk < BN / 16; ++blk) {
          float2 ev[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int k = blk * 16 + 2 * i;
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), am2, nm2);
            ev[i] = make_float2(ex2(x.x), ex2(x.y));
            ls2[i & 1] = __fadd2_rn(ls2[i & 1], ev[i]);
          }
          uint32_t lo[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t hi = pack_bf16x2(ev[i].x, ev[i].y);
            sr[blk * 8 + i] = hi;   // registers 8 b .. 8 b + 7 were read by this block or an earlier one
            lo[i] = pack_bf16x2(ev[i].x - __uint_as_float(hi << 16), ev[i].y - __uint_as_float(hi & 0xffff0000u));
          }
          tmem_st8(tS + 32 + blk * 8, lo);
          if (blk == 1) release(0);
        }
      } else {
        // in place: pair i is written to register i after registers 2i, 2i + 1 were read
#pragma unroll
        for (int i = 0; i < BN / 2; ++i) {
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])), am2, nm2);
          const float2 ev = make_float2(ex2(x.x), ex2(x.y));
          ls2[i & 1] = __fadd2_rn(ls2[i & 1], ev);
          sr[i] = pack_bf16x2(ev.x, ev.y);
          if (i == 15) release(0);
        }
      }
      release(1);
      const float2 lt = __fadd2_rn(ls2[0], ls2[1]);
      const float ls = lt.x + lt.y;
      l_run = l_run * alpha + ls;
      m_run = m_use;
    }
    if (ok && n > 0)
      ok = __all_sync(0xffffffffu, wait_or_abort(&o_done[T::sbuf(n - 1)], T::sphase(n - 1), p.err));
    if (ok) {
      tc_fence_after();
      const int hq = kvh * G + hh;
      float M2 = m_run, f = 1.f, Z = l_run;
      if (p.sinks != nullptr) {
        const float sk = p.sinks[hq] * kLog2e;
        M2 = fmaxf(m_run, sk);
        f = (m_run == -INFINITY) ? 0.f : ex2(m_run - M2);
        Z = l_run * f + ex2(sk - M2);
      }
      const float inv = (Z > 0.f) ? f / Z : 0.f;
      const int64_t orow = static_cast<int64_t>(qs + min(tok, qlen - 1));
      uint16_t* op = p.out + orow * p.out_stride_tok + static_cast<int64_t>(hq) * p.out_stride_head;
      const bool row_a32 = (reinterpret_cast<uintptr_t>(op) & 31u) == 0;
      const uint32_t tO = tbase + lane_off + T::TMEM_O;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(tO + c * 32, u);
        tmem_wait_ld();
        if (row_ok) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(u[2 * e]) * inv, __uint_as_float(u[2 * e + 1]) * inv);
          uint16_t* dst = op + c * 32;
          if (row_a32) {
            // a whole 32-byte sector per lane: half the store instructions
            st_global_v8(dst, pk);
            st_global_v8(dst + 16, pk + 8);
          } else {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int v = 0; v < 4; ++v) d4[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      }
      if (row_ok && p.lse != nullptr) {
        p.lse[orow * p.num_q_heads + hq] = (Z > 0.f) ? (M2 + lg2(Z)) * kLn2 : -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, T::TMEM_COLS);
}

template <int D, int BN, int NST, int CPS, bool FP8>
cudaError_t launch_ext(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                       const ExtendParams& p, cudaStream_t stream) {
  using T = ExtTraits<D, BN, NST, CPS, FP8>;
  extend_schedule_kernel<<<1, kSchedThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto kern = extend_attn_kernel<D, BN, NST, CPS, FP8>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM);
  if (e != cudaSuccess) return e;
  const int64_t blocks = static_cast<int64_t>(p.work_cap) * p.num_kv_heads;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = T::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmq, tmk, tmv, p);
}


// e4m3 cache, dequantised once per call: every page a request attends to is
// written as bf16(float(code) * scale) into a dense copy, page i of request
// b at copy page b * maxp + i, with an identity block table beside it; the
// bf16 attention kernel then reads the copy.  Each K/V tile is otherwise
// dequantised by every query tile of its request.
struct KvCopyParams {
  const uint8_t* k;
  const uint8_t* v;
  int64_t stride_page, stride_tok, stride_head;   // bytes (e4m3)
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* seq_lens;
  const int32_t* qsl;
  int batch, num_pages, page_size, num_kv_heads, window, maxp, max_kv;
  float k_scale, v_scale;
  const float* k_scales;   // [B] per-request scales, or null
  const float* v_scales;
  uint16_t* kc;
  uint16_t* vc;
  int32_t* bt_copy;
  uint32_t* err;   // scratch header error word
};

template <int D>
__global__ void __launch_bounds__(256) extend_kv_copy_kernel(const KvCopyParams p) {
  const int i = blockIdx.x;   // page of the request
  const int b = blockIdx.y;
  const int64_t dst_page = static_cast<int64_t>(b) * p.maxp + i;
  if (threadIdx.x == 0) p.bt_copy[dst_page] = static_cast<int32_t>(dst_page);
  const int L = p.seq_lens[b];
  const int qlen = p.qsl[b + 1] - p.qsl[b];
  const int ctx = L - qlen;
  // malformed rows are reported by the scheduler; nothing to copy for them
  if (qlen <= 0 || ctx < 0 || L > p.max_kv) return;
  const int ps = p.page_size;
  const int first = p.window > 0 ? max(0, ctx - p.window + 1) : 0;   // first key any query attends
  if ((i + 1) * ps <= first || i * ps >= L) return;
  const int src = p.block_table[static_cast<int64_t>(b) * p.bt_stride + i];
  const uint64_t k_sc2 = dequant_scale2(p.k_scales != nullptr ? p.k_scales[b] : p.k_scale);
  const uint64_t v_sc2 = dequant_scale2(p.v_scales != nullptr ? p.v_scales[b] : p.v_scale);
  constexpr int UPH = D / 16;   // 16-code units per head row
  const int units = ps * p.num_kv_heads * UPH;
  const int64_t page_elems = static_cast<int64_t>(ps) * p.num_kv_heads * D;
  uint4* kd = reinterpret_cast<uint4*>(p.kc + dst_page * page_elems);
  uint4* vd = reinterpret_cast<uint4*>(p.vc + dst_page * page_elems);
  if (src < 0 || src >= p.num_pages) {
    // a page id outside the pool reads as zeros, as a TMA box outside it
    // does, and is flagged
    if (threadIdx.x == 0) atomicOr(p.err, kErrPageId);
    for (int u = threadIdx.x; u < 2 * units; u += blockDim.x) {
      kd[u] = make_uint4(0, 0, 0, 0);
      vd[u] = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  for (int u = threadIdx.x; u < units; u += blockDim.x) {
    const int tok = u / (p.num_kv_heads * UPH);
    const int rem = u - tok * (p.num_kv_heads * UPH);
    const int head = rem / UPH;
    const int d16 = rem - head * UPH;
    const int64_t off = static_cast<int64_t>(src) * p.stride_page + static_cast<int64_t>(tok) * p.stride_tok +
                        static_cast<int64_t>(head) * p.stride_head + d16 * 16;
    const uint4 kw = *reinterpret_cast<const uint4*>(p.k + off);
    const uint4 vw = *reinterpret_cast<const uint4*>(p.v + off);
    const uint32_t ka[4] = {kw.x, kw.y, kw.z, kw.w};
    const uint32_t va[4] = {vw.x, vw.y, vw.z, vw.w};
    uint32_t ko[8], vo[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      ko[2 * k] = dequant_e4m3x2<0>(ka[k], k_sc2);
      ko[2 * k + 1] = dequant_e4m3x2<1>(ka[k], k_sc2);
      vo[2 * k] = dequant_e4m3x2<0>(va[k], v_sc2);
      vo[2 * k + 1] = dequant_e4m3x2<1>(va[k], v_sc2);
    }
    kd[2 * u] = make_uint4(ko[0], ko[1], ko[2], ko[3]);
    kd[2 * u + 1] = make_uint4(ko[4], ko[5], ko[6], ko[7]);
    vd[2 * u] = make_uint4(vo[0], vo[1], vo[2], vo[3]);
    vd[2 * u + 1] = make_uint4(vo[4], vo[5], vo[6], vo[7]);
  }
}

constexpr int64_t kMaxKvCopyBytes = int64_t{2} << 30;   // bf16 K + V copy of an e4m3 cache

int64_t kv_copy_bytes(const pa_shape& s) {
  return static_cast<int64_t>(s.max_batch) * s.max_pages_per_seq * s.page_size * s.num_kv_heads * s.head_dim *
         2 /* bf16 */ * 2 /* K and V */;
}

// Per head_dim: keys per tile and pipeline stages (shared memory <= 227 KB).
struct ExtChoice {
  int block_n, stages, smem;
};

// Two CTAs per SM where TMEM and shared memory allow (64-key tiles, 256
// TMEM columns each): one CTA's prologue, epilogue and softmax overlap the
// other's MMAs.  head_dim 256 needs 256 O columns, so one CTA per SM.
ExtChoice ext_choice(int D) {
  if (D == 64) return {64, 4, ExtTraits<64, 64, 4, 2>::SMEM};
  if (D == 128) return {64, 2, ExtTraits<128, 64, 2, 2>::SMEM};
  return {64, 3, ExtTraits<256, 64, 3, 1>::SMEM};   // Q in TMEM, three stages
}

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Work items (query tiles) a plan has room for: every request's last tile
// may be partial.
int64_t work_capacity(const pa_shape& s) {
  const int tm = kRows / (s.num_q_heads / s.num_kv_heads);
  return (static_cast<int64_t>(s.max_total_q) + tm - 1) / tm + s.max_batch;
}

// Scratch an extend plan lays out: the header, the work list and, with an
// e4m3 copy, the identity block table and the bf16 K and V copies.
int64_t extend_scratch_bytes(const pa_shape& s, bool copy) {
  int64_t b = kScratchHeaderBytes + align_up(work_capacity(s) * 32, 256);
  if (copy)
    b += align_up(static_cast<int64_t>(s.max_batch) * s.max_pages_per_seq * 4, 256) +
         2 * align_up(kv_copy_bytes(s) / 2, 256);
  return b;
}

}  // namespace

pa_status plan_extend(const pa_shape& s, int num_sms, pa_plan_t* out) {
  (void)num_sms;
  const int G = s.num_q_heads / s.num_kv_heads;
  const int tm = kRows / G;
  const ExtChoice ch = ext_choice(s.head_dim);
  const int64_t work_cap = work_capacity(s);
  if (work_cap * s.num_kv_heads > INT32_MAX) return PA_ERR_UNSUPPORTED;
  out->tile_tokens = ch.block_n;
  out->split_tiles = tm;
  out->max_splits = 1;
  out->stages = ch.stages;
  out->warps = kThreads / 32;
  out->bt_cache = 0;
  out->smem_bytes = ch.smem;
  out->grid[0] = static_cast<int32_t>(work_cap * s.num_kv_heads);
  out->grid[1] = 1;
  out->grid[2] = 1;
  out->kv_copy = (s.kv_dtype == PA_KV_FP8_E4M3 && kv_copy_bytes(s) <= kMaxKvCopyBytes) ? 1 : 0;
  out->scratch_bytes = extend_scratch_bytes(s, out->kv_copy != 0);
  out->launches = out->kv_copy ? 3 : 2;  // (e4m3 copy,) scheduler, attention kernel
  return PA_OK;
}

}  // namespace pa

using namespace pa;

namespace {

constexpr float kLog2eHost = 1.4426950408889634f;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" pa_status pa_extend(const pa_plan_t* plan, const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                               const void* k_cache, const void* v_cache, int64_t kv_stride_page,
                               int64_t kv_stride_tok, int64_t kv_stride_head, int32_t num_pages,
                               const int32_t* block_table, int64_t bt_stride, const int32_t* seq_lens,
                               const int32_t* query_start_loc, int32_t batch, int32_t total_q, float scale,
                               const float* sinks, float k_scale, float v_scale, const float* k_scales,
                               const float* v_scales, void* out, int64_t out_stride_tok, int64_t out_stride_head,
                               float* lse, void* scratch, int64_t scratch_bytes, void* stream) {
  if (!plan) return PA_ERR_INVALID_ARG;
  const pa_shape& s = plan->shape;
  if (s.mode == PA_MODE_VERIFY) {
    // equal, small query counts per request: the split-KV kernels, one query
    // row per (token, head)
    if (batch < 0 || batch > s.max_batch || total_q != batch * s.q_len) return PA_ERR_INVALID_ARG;
    if (!query_start_loc && batch > 0) return PA_ERR_INVALID_ARG;
    return run_split_kv(plan, q, q_stride_tok, q_stride_head, k_cache, v_cache, kv_stride_page, kv_stride_tok,
                        kv_stride_head, num_pages, block_table, bt_stride, seq_lens, query_start_loc, batch, scale,
                        sinks, k_scale, v_scale, k_scales, v_scales, out, out_stride_tok, out_stride_head, lse,
                        scratch, scratch_bytes, stream);
  }
  if (s.mode != PA_MODE_EXTEND || validate_shape(s) != PA_OK) return PA_ERR_INVALID_ARG;
  const bool fp8 = s.kv_dtype == PA_KV_FP8_E4M3;
  if (!std::isfinite(k_scale) || !std::isfinite(v_scale)) return PA_ERR_INVALID_ARG;
  if (batch < 0 || batch > s.max_batch || total_q < 0 || total_q > s.max_total_q) return PA_ERR_INVALID_ARG;
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return PA_ERR_INVALID_ARG;
  if ((sinks != nullptr) != (s.has_sinks != 0)) return PA_ERR_INVALID_ARG;
  if (!scratch) return PA_ERR_INVALID_ARG;
  if (scratch_bytes < plan->scratch_bytes) return PA_ERR_SCRATCH_TOO_SMALL;
  // the work list (and an e4m3 copy) are laid out from the shape's
  // capacities: a plan edited by hand must still match them and leave room
  const int64_t cap_items = work_capacity(s);
  if (plan->grid[0] != cap_items * s.num_kv_heads) return PA_ERR_INVALID_ARG;
  if (scratch_bytes < extend_scratch_bytes(s, fp8 && plan->kv_copy != 0)) return PA_ERR_SCRATCH_TOO_SMALL;
  if ((reinterpret_cast<uintptr_t>(scratch) & 255u) != 0) return PA_ERR_UNSUPPORTED;
  if (batch == 0 || total_q == 0) return PA_OK;
  if (!q || !out || !block_table || !seq_lens || !query_start_loc || bt_stride < 0) return PA_ERR_INVALID_ARG;
  if (q_stride_tok <= 0 || q_stride_head <= 0 || out_stride_tok <= 0 || out_stride_head <= 0)
    return PA_ERR_INVALID_ARG;
  // q feeds a TMA tensor map and out is written in 16-byte vectors
  if (!aligned16(q) || !aligned16(out) || (q_stride_tok % 8) || (q_stride_head % 8) || (out_stride_tok % 8) ||
      (out_stride_head % 8))
    return PA_ERR_UNSUPPORTED;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return PA_ERR_UNSUPPORTED;
  pa_status st = check_kv(s, k_cache, v_cache, kv_stride_page, kv_stride_tok, kv_stride_head, num_pages);
  if (st != PA_OK) return st;

  const int G = s.num_q_heads / s.num_kv_heads;
  const int tm = kRows / G;
  const ExtChoice ch = ext_choice(s.head_dim);
  CUtensorMap tmq, tmk, tmv;
  if ((st = make_q_map(&tmq, q, s.head_dim, s.num_q_heads, total_q, q_stride_tok, q_stride_head, G, tm)) !=
      PA_OK)
    return st;
  uint8_t* sc = static_cast<uint8_t*>(scratch);
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  // e4m3 cache with a copy plan: dequantise the attended pages once into the
  // scratch workspace (after the work list), then attend over the bf16 copy
  const bool copy = fp8 && plan->kv_copy != 0 && batch <= 65535;
  const void* kbase = k_cache;
  const void* vbase = v_cache;
  const int32_t* bt = block_table;
  int64_t bts = bt_stride, st_page = kv_stride_page, st_tok = kv_stride_tok, st_head = kv_stride_head;
  int32_t pages = num_pages;
  if (copy) {
    const int64_t maxp = s.max_pages_per_seq;
    uint8_t* cbase = sc + kScratchHeaderBytes + align_up(cap_items * 32, 256);
    int32_t* bt_copy = reinterpret_cast<int32_t*>(cbase);
    uint8_t* kc = cbase + align_up(static_cast<int64_t>(s.max_batch) * maxp * 4, 256);
    uint8_t* vc = kc + align_up(kv_copy_bytes(s) / 2, 256);
    if (static_cast<int64_t>(batch) * maxp > INT32_MAX) return PA_ERR_UNSUPPORTED;
    KvCopyParams cp{};
    cp.k = static_cast<const uint8_t*>(k_cache);
    cp.v = static_cast<const uint8_t*>(v_cache);
    cp.stride_page = kv_stride_page;
    cp.stride_tok = kv_stride_tok;
    cp.stride_head = kv_stride_head;
    cp.block_table = block_table;
    cp.bt_stride = bt_stride;
    cp.seq_lens = seq_lens;
    cp.qsl = query_start_loc;
    cp.batch = batch;
    cp.num_pages = num_pages;
    cp.page_size = s.page_size;
    cp.num_kv_heads = s.num_kv_heads;
    cp.window = s.window;
    cp.maxp = static_cast<int>(maxp);
    cp.max_kv = s.max_pages_per_seq * s.page_size;
    cp.k_scale = k_scale;
    cp.v_scale = v_scale;
    cp.k_scales = k_scales;
    cp.v_scales = v_scales;
    cp.kc = reinterpret_cast<uint16_t*>(kc);
    cp.vc = reinterpret_cast<uint16_t*>(vc);
    cp.bt_copy = bt_copy;
    cp.err = reinterpret_cast<uint32_t*>(sc);
    const dim3 cgrid(static_cast<unsigned>(maxp), static_cast<unsigned>(batch));
    switch (s.head_dim) {
      case 64: extend_kv_copy_kernel<64><<<cgrid, 256, 0, strm>>>(cp); break;
      case 128: extend_kv_copy_kernel<128><<<cgrid, 256, 0, strm>>>(cp); break;
      default: extend_kv_copy_kernel<256><<<cgrid, 256, 0, strm>>>(cp); break;
    }
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    kbase = kc;
    vbase = vc;
    bt = bt_copy;
    bts = maxp;
    st_head = s.head_dim;
    st_tok = static_cast<int64_t>(s.num_kv_heads) * s.head_dim;
    st_page = st_tok * s.page_size;
    pages = static_cast<int32_t>(static_cast<int64_t>(batch) * maxp);
  }
  const bool fp8_tiles = fp8 && !copy;   // the attention kernel dequantises in shared memory
  if ((st = make_kv_map(&tmk, kbase, fp8_tiles, s.head_dim, s.num_kv_heads, s.page_size, pages, st_page, st_tok,
                        st_head, s.page_size)) != PA_OK)
    return st;
  if ((st = make_kv_map(&tmv, vbase, fp8_tiles, s.head_dim, s.num_kv_heads, s.page_size, pages, st_page, st_tok,
                        st_head, s.page_size)) != PA_OK)
    return st;

  ExtendParams p{};
  p.seq_lens = seq_lens;
  p.qsl = query_start_loc;
  p.block_table = bt;
  p.bt_stride = bts;
  p.batch = batch;
  p.total_q = total_q;
  p.num_q_heads = s.num_q_heads;
  p.num_kv_heads = s.num_kv_heads;
  p.group = G;
  p.page_size = s.page_size;
  p.num_pages = pages;
  p.tm = tm;
  p.max_kv = s.max_pages_per_seq * s.page_size;
  p.block_n = ch.block_n;
  p.scale_log2 = scale * kLog2eHost;
  p.cap_log2 = s.soft_cap > 0.f ? s.soft_cap * kLog2eHost : 0.f;
  p.scale_over_cap = s.soft_cap > 0.f ? scale / s.soft_cap : 0.f;
  p.window = s.window;
  p.sinks = sinks;
  p.k_scale = fp8_tiles ? k_scale : 1.f;
  p.v_scale = fp8_tiles ? v_scale : 1.f;
  p.k_scales = fp8_tiles ? k_scales : nullptr;
  p.v_scales = fp8_tiles ? v_scales : nullptr;
  p.out = static_cast<uint16_t*>(out);
  p.out_stride_tok = out_stride_tok;
  p.out_stride_head = out_stride_head;
  p.lse = lse;
  p.err = reinterpret_cast<uint32_t*>(sc);
  p.work_count = reinterpret_cast<int*>(sc + 16);
  p.work = reinterpret_cast<int4*>(sc + kScratchHeaderBytes);
  p.work_cap = static_cast<int>((plan->scratch_bytes - kScratchHeaderBytes) / 32);
  if (p.work_cap > cap_items) p.work_cap = static_cast<int>(cap_items);

  cudaError_t e;
  switch (s.head_dim * 2 + (fp8_tiles ? 1 : 0)) {
    case 128: e = launch_ext<64, 64, 4, 2, false>(tmq, tmk, tmv, p, strm); break;
    case 129: e = launch_ext<64, 64, 4, 2, true>(tmq, tmk, tmv, p, strm); break;
    case 256: e = launch_ext<128, 64, 2, 2, false>(tmq, tmk, tmv, p, strm); break;
    case 257: e = launch_ext<128, 64, 2, 2, true>(tmq, tmk, tmv, p, strm); break;
    case 512: e = launch_ext<256, 64, 3, 1, false>(tmq, tmk, tmv, p, strm); break;
    default: e = launch_ext<256, 64, 2, 1, true>(tmq, tmk, tmv, p, strm); break;
  }
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
