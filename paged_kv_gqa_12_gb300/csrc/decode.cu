// Split-KV paged decode for sm_103a.
//
// Operation: "vllm/attention/ops/triton_decode_attention.py",
// _fwd_grouped_kernel_stage1 (one partial softmax-attention result plus its
// log-sum-exp per KV split of each request and kv head) and _fwd_kernel_stage2
// (merge of the splits by LSE).  Sinks follow "vllm/v1/attention/backends/b12x"
// (attention_sink_bias, one fp32 logit per q head in the softmax denominator).
//
// Design (GB300): the KV stream is read once from HBM, so the kernel is built
// around bytes in flight, not arithmetic.
//   * One CTA = one (split, kv head, request) work item, 4 compute warps.
//     Warp w takes tiles w, w+4, w+8, ... of the split, each tile being
//     TS consecutive keys; every warp owns a private ring of NS stages that
//     its lane 0 refills with TMA tensor loads straight out of the pages
//     (page id from a block-table slice staged in shared memory).  No
//     producer warp, no cross-warp barrier in the main loop.
//   * The G q heads that share a kv head (times the query tokens per request:
//     1 for decode, 1 + speculative tokens for verify) form the N dimension
//     of warp-level bf16 MMAs: S^T = K Q^T (M = 16 keys, N = 8 rows) and
//     O^T += V^T P^T (M = 16 dims, N = 8 rows), so a K/V element fetched
//     once serves all rows, and the 8-wide N keeps 8 rows free of padding.
//     Verify rows mask keys after their own position (causal) and outside
//     their own window.
//     P^T is formed in registers with movmatrix.
//   * fp8-e4m3 K/V are dequantised in registers to bf16 exactly as the
//     prefix-prefill page does: bf16(float(code) * scale).
//   * Online softmax in the log2 domain (accumulators rescaled only on tiles
//     where a row maximum rose); per-thread partial row sums are reduced
//     once at the end; the 4 warps' states are merged in shared
//     memory.  A request with one split writes the final output directly;
//     otherwise each split writes its normalised partial and LSE, and the
//     split that finishes last for its (request, kv head) -- counted by an
//     atomic arrival counter in the scratch header -- merges them, so a call
//     is one launch.  Plans with more (request, kv head) pairs than the
//     header holds counters use the separate merge kernel instead.
#include <cfloat>
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"

namespace pa {
namespace {

constexpr int kWarps = 4;
constexpr float kLog2e = 1.4426950408889634f;
// A tile is computed with exact weights (P = P_hi + P_lo) when some row's
// largest weight from it exceeds 1 / kHotShare of the row's denominator.
constexpr float kHotShare = 8.f;
constexpr float kLn2 = 0.6931471805599453f;

// Attended keys of request b and their split partition.  Splits are
// tile-aligned; split boundaries are a free choice because the LSE merge is
// an exact re-association of the same softmax sum.
struct SplitRange {
  int lo, hi;            // attended keys [lo, hi)
  int tile0;             // first tile (tile t covers keys [t*TS, (t+1)*TS))
  int n_tiles;
  int tiles_per_split;
  int n_splits;
};

__device__ __forceinline__ SplitRange split_range(const DecodeParams& p, int L) {
  SplitRange r;
  r.hi = L;
  // the first query of the request sits at L - q_len; with a window it keeps
  // key j iff (L - q_len) - j < W, and later queries keep a subset of later keys
  r.lo = (p.window > 0) ? max(0, (L - p.q_len) - p.window + 1) : 0;
  const int ts = p.tile_tokens;
  if (r.hi <= r.lo) {
    r.tile0 = 0;
    r.n_tiles = 0;
    r.tiles_per_split = 1;
    r.n_splits = 0;
    return r;
  }
  r.tile0 = r.lo / ts;
  r.n_tiles = (r.hi + ts - 1) / ts - r.tile0;
  r.tiles_per_split = p.fixed_splits > 0 ? (r.n_tiles + p.fixed_splits - 1) / p.fixed_splits : p.split_tiles;
  r.n_splits = (r.n_tiles + r.tiles_per_split - 1) / r.tiles_per_split;
  // equal splits (a request of 4.5 split lengths gets five of 0.9, not four
  // full ones and a half): no split is longer than planned, and the CTAs a
  // request contributes to the last wave are all short
  r.tiles_per_split = (r.n_tiles + r.n_splits - 1) / r.n_splits;
  r.n_splits = (r.n_tiles + r.tiles_per_split - 1) / r.tiles_per_split;
  return r;
}

template <int D, bool FP8, int NH8, int TS, int NS>
struct Traits {
  static constexpr int E = FP8 ? 1 : 2;                        // bytes per element
  static constexpr int ROW = D * E;                            // bytes of one key row of one head
  static constexpr int RB = ROW < 128 ? ROW : 128;             // bytes per TMA box row
  static constexpr int NCC = ROW / RB;                         // column chunks per row
  static constexpr int TILE = TS * ROW;                        // K (or V) bytes per stage
  static constexpr int STAGE = 2 * TILE;
  static constexpr int WARP_BYTES = NS * STAGE;
  static constexpr int MT = TS / 16;                           // 16-key groups per tile
  static constexpr int KS = D / 16;                            // 16-wide steps over head_dim
  static constexpr int HW = NH8 * 8;                           // heads per warp (MMA N)
  static_assert(RB == 128 || RB == 64, "row bytes must use the 128B or 64B swizzle");
  static_assert(TS % 16 == 0, "tile must hold whole 16-key groups");

  // Byte offset of (row, byte-in-row) inside a K or V stage tile as TMA
  // writes it: column chunks of RB bytes, rows of RB bytes, 16-byte units
  // XOR-swizzled (128B swizzle: unit ^= row & 7; 64B swizzle: unit ^= (row>>1) & 3).
  __device__ static __forceinline__ uint32_t off(int row, int byte) {
    const int cc = byte / RB;
    const int x = byte % RB;
    const uint32_t sw = (RB == 128) ? (row & 7) : ((row >> 1) & 3);
    return static_cast<uint32_t>(cc * (TS * RB) + row * RB) + ((((x >> 4) ^ sw) << 4) | (x & 15));
  }
};

// LSE merge of one request's splits for the R rows (token, head) of one kv
// head group, by the CTA that finished last: thread t takes 4 consecutive
// dims of one row; the splits are folded eight at a time (their loads in
// flight together) into a running maximum, sum and weighted output.  The
// partials are read from L2: other SMs wrote them.
template <int D>
__device__ __forceinline__ void merge_splits(const DecodeParams& p, int n_splits, int R, int Gc, int hq0,
                                             int64_t qrow0) {
  constexpr int C = D / 4;   // float4 chunks per row
  constexpr int U = 8;
  for (int e = threadIdx.x; e < R * C; e += kWarps * 32) {
    const int h = e / C;
    const int d = (e - h * C) * 4;
    const int tq = h / Gc;
    const int hq = hq0 + (h - tq * Gc);
    const int64_t orow = qrow0 + tq;
    const int64_t row0 = (orow * p.num_q_heads + hq) * p.max_splits;
    const float* lp = p.lse_part + row0;
    const float* op = p.o_part + row0 * D + d;
    const bool has_sink = p.sinks != nullptr;
    float M = has_sink ? p.sinks[hq] * kLog2e : -INFINITY;
    float Z = has_sink ? 1.f : 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < n_splits; s0 += U) {
      float l[U];
      float4 o[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const bool ok = s0 + u < n_splits;
        l[u] = ok ? __ldcg(lp + s0 + u) * kLog2e : -INFINITY;
        o[u] = ok ? __ldcg(reinterpret_cast<const float4*>(op + static_cast<int64_t>(s0 + u) * D))
                  : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float mx = l[0];
#pragma unroll
      for (int u = 1; u < U; ++u) mx = fmaxf(mx, l[u]);
      if (mx > M) {   // rescale what was summed against the old maximum
        const float f = ex2(M - mx);
        Z *= f;
        acc.x *= f; acc.y *= f; acc.z *= f; acc.w *= f;
        M = mx;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (l[u] == -INFINITY) continue;   // padding, or a split with no key for this row
        const float w = ex2(l[u] - M);
        Z += w;
        acc.x += w * o[u].x; acc.y += w * o[u].y; acc.z += w * o[u].z; acc.w += w * o[u].w;
      }
    }
    const float inv = Z > 0.f ? 1.f / Z : 0.f;
    uint16_t* outp = p.out + orow * p.out_stride_tok + static_cast<int64_t>(hq) * p.out_stride_head + d;
    // (rows are 4-byte aligned: two bf16 pairs)
    reinterpret_cast<uint32_t*>(outp)[0] = pack_bf16x2(acc.x * inv, acc.y * inv);
    reinterpret_cast<uint32_t*>(outp)[1] = pack_bf16x2(acc.z * inv, acc.w * inv);
    if (d == 0 && p.lse != nullptr)
      p.lse[orow * p.num_q_heads + hq] = M == -INFINITY ? -INFINITY : (M + lg2(Z)) * kLn2;
  }
}

template <int D, bool FP8, int NH8, int TS, int NS, bool CAP>
__global__ void __launch_bounds__(kWarps * 32)
decode_split_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                    const DecodeParams p) {
  using T = Traits<D, FP8, NH8, TS, NS>;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y / p.head_groups;   // kv head; groups above 16 heads use several CTAs
  const int hg = blockIdx.y - kvh * p.head_groups;
  const int b = blockIdx.z;
  const int L = p.seq_lens[b];
  const SplitRange r = split_range(p, L);
  if (r.n_splits == 0) {
    // nothing to attend (an empty request): O = 0, and the LSE is the sink
    // logit, or -inf without sinks; the first split's CTA writes its rows
    if (split == 0) {
      const int G = p.group;
      const int head0 = hg * 16;
      const int Gc = p.head_groups > 1 ? min(16, G - head0) : G;
      const int R = p.q_len * Gc;
      const int64_t qrow0 = static_cast<int64_t>(b) * p.q_len;
      for (int i = threadIdx.x; i < R * D; i += blockDim.x) {
        const int rr = i / D, d = i - rr * D;
        const int tq = rr / Gc;
        const int hq = kvh * G + head0 + (rr - tq * Gc);
        p.out[(qrow0 + tq) * p.out_stride_tok + static_cast<int64_t>(hq) * p.out_stride_head + d] = 0;
        if (d == 0 && p.lse != nullptr)
          p.lse[(qrow0 + tq) * p.num_q_heads + hq] = p.sinks != nullptr ? p.sinks[hq] : -INFINITY;
      }
    }
    return;
  }
  if (split >= r.n_splits) return;
  if (r.n_splits > p.max_splits) {  // seq_lens beyond the planned capacity
    if (threadIdx.x == 0 && split == 0) atomicOr(p.err, kErrCapacity);
    return;
  }

  const int qrow0 = b * p.q_len;   // first query row of the request
  if (p.qsl != nullptr && (p.qsl[b] != qrow0 || p.qsl[b + 1] != qrow0 + p.q_len)) {
    if (threadIdx.x == 0 && split == 0) atomicOr(p.err, kErrCapacity);   // not equal-length packing
    return;
  }
  const int tile_begin = r.tile0 + split * r.tiles_per_split;
  const int tile_end = min(tile_begin + r.tiles_per_split, r.tile0 + r.n_tiles);
  const int tok_lo = max(r.lo, tile_begin * TS);
  const int tok_hi = min(r.hi, tile_end * TS);
  const int ps = p.page_size;
  const int ps_log2 = __ffs(ps) - 1;  // page sizes are powers of two: shifts, no integer division
  const int pg0 = (tile_begin * TS) >> ps_log2;
  const int pg1 = (tok_hi + ps - 1) >> ps_log2;   // <= ceil(L / ps): never past the request's pages
  const int G = p.group;
  const int head0 = hg * 16;          // first head (within the kv head's group) of this CTA
  const int Gc = p.head_groups > 1 ? min(16, G - head0) : G;   // heads this CTA covers
  const int R = p.q_len * Gc;         // query rows: (token, head) pairs
  // tiles where every row sees every key need no per-element mask
  const int pos_first = L - p.q_len;  // position of the first query
  const int lo_last = p.window > 0 ? (L - 1) - p.window + 1 : 0;
  const int full_lo = max(tok_lo, lo_last);
  const int full_hi = min(tok_hi, pos_first + 1);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWarps * T::WARP_BYTES);
  int32_t* bt_s = reinterpret_cast<int32_t*>(bars + kWarps * NS);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = lane >> 2;   // MMA group id
  const int c = lane & 3;    // thread in group

  // planner invariant, never expected to fail; a split that fails it reads
  // nothing but still reports to the merge, so the arrival count completes
  const bool bt_fits = pg1 - pg0 <= p.bt_cache;
  if (!bt_fits && tid == 0) atomicOr(p.err, kErrSchedOverflow);
  const int n_tiles = bt_fits ? tile_end - tile_begin : 0;
  const int32_t* bt_row = p.block_table + static_cast<int64_t>(b) * p.bt_stride;
  // A page id outside the pool becomes the out-of-range coordinate num_pages,
  // whose TMA box reads as zeros; it is an error when the page holds attended
  // keys (a page before the window start is fetched but wholly masked).
  for (int i = tid; i < (bt_fits ? pg1 - pg0 : 0); i += kWarps * 32) {
    int id = bt_row[pg0 + i];
    if (static_cast<unsigned>(id) >= static_cast<unsigned>(p.num_pages)) {
      if (((pg0 + i + 1) << ps_log2) > tok_lo) atomicOr(p.err, kErrPageId);
      id = p.num_pages;
    }
    bt_s[i] = id;
  }
  if (tid == 0) {
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
    for (int i = 0; i < kWarps * NS; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();

  uint8_t* wbase = smem + warp * T::WARP_BYTES;
  uint64_t* wbar = bars + warp * NS;

  // Lane 0: fetch local tile k of this split into `stage` (K and V, all
  // pages the tile touches, every column chunk).  Boxes wholly past the end
  // of the sequence are not fetched; their rows are masked.
  auto issue = [&](int k, int stage) {
    const int t0 = (tile_begin + k) * TS;
    const int br = ps < TS ? ps : TS;
    int nb = 0;
    for (int j = 0; j < TS / br; ++j) nb += (t0 + j * br < L) ? 1 : 0;
    uint8_t* kst = wbase + stage * T::STAGE;
    uint8_t* vst = kst + T::TILE;
    mbar_arrive_expect_tx(&wbar[stage], static_cast<uint32_t>(nb * br * T::ROW * 2));
    for (int j = 0; j < nb; ++j) {
      const int t = t0 + j * br;
      const int page = bt_s[(t >> ps_log2) - pg0];
      const int slot = t & (ps - 1);
#pragma unroll
      for (int cc = 0; cc < T::NCC; ++cc) {
        const int dst = cc * TS * T::RB + j * br * T::RB;
        tma_load_4d(kst + dst, &tmk, cc * (T::RB / T::E), kvh, slot, page, &wbar[stage]);
        tma_load_4d(vst + dst, &tmv, cc * (T::RB / T::E), kvh, slot, page, &wbar[stage]);
      }
    }
  };

  // Q^T fragments (MMA B operand: k = head_dim slot, n = query row).
  uint32_t qf[T::KS][NH8][2];
  {
#pragma unroll
    for (int j = 0; j < NH8; ++j) {
      const int rr = j * 8 + g;   // row = token * G + head
      const bool ok = rr < R;
      const int tq = ok ? rr / Gc : 0;
      const int hq = ok ? head0 + rr - tq * Gc : 0;
      const uint16_t* qh = p.q + static_cast<int64_t>(qrow0 + tq) * p.q_stride_tok +
                           static_cast<int64_t>(kvh * G + hq) * p.q_stride_head;
#pragma unroll
      for (int ks = 0; ks < T::KS; ++ks) {
        int d0, d1;
        if constexpr (FP8) {   // permuted head_dim: thread c owns dims [c*D/4, (c+1)*D/4)
          d0 = c * (D / 4) + ks * 4;
          d1 = d0 + 2;
        } else {
          d0 = ks * 16 + 2 * c;
          d1 = d0 + 8;
        }
        qf[ks][j][0] = ok ? *reinterpret_cast<const uint32_t*>(qh + d0) : 0u;
        qf[ks][j][1] = ok ? *reinterpret_cast<const uint32_t*>(qh + d1) : 0u;
      }
    }
  }

  float o[T::KS][NH8][4];
#pragma unroll
  for (int i = 0; i < T::KS; ++i)
#pragma unroll
    for (int j = 0; j < NH8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[i][j][e] = 0.f;
  float m_run[NH8][2], l_run[NH8][2];
  int rpos[NH8][2], rlo[NH8][2];   // this thread's two rows: last and first attended key
  bool rvalid[NH8][2];             // the row is a real (token, head), not MMA padding
#pragma unroll
  for (int j = 0; j < NH8; ++j) {
    m_run[j][0] = m_run[j][1] = -INFINITY;
    l_run[j][0] = l_run[j][1] = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int rr = j * 8 + 2 * c + h;
      rvalid[j][h] = rr < R;
      rpos[j][h] = pos_first + min(rr, R - 1) / Gc;
      rlo[j][h] = p.window > 0 ? rpos[j][h] - p.window + 1 : 0;
    }
  }

  if (lane == 0) {
    for (int s = 0; s < NS; ++s) {
      const int k = warp + s * kWarps;
      if (k < n_tiles) issue(k, s);
    }
  }
  __syncwarp();

  // e4m3 descales of this request (per request when given, else per tensor)
  const uint64_t k_sc2 = dequant_scale2(p.k_scales != nullptr ? p.k_scales[b] : p.k_scale);
  const uint64_t v_sc2 = dequant_scale2(p.v_scales != nullptr ? p.v_scales[b] : p.v_scale);
  bool l_small = true;   // some row's running denominator (summed over its lanes) is below kHotShare
  int it = 0;
  for (int k = warp; k < n_tiles; k += kWarps, ++it) {
    const int stage = it % NS;
    const uint32_t parity = static_cast<uint32_t>((it / NS) & 1);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&wbar[stage], parity, p.err));
    if (!ok) break;
    const uint8_t* kst = wbase + stage * T::STAGE;
    const uint8_t* vst = kst + T::TILE;
    const uint32_t kst_u = smem_u32(kst);
    const uint32_t vst_u = smem_u32(vst);
    const int t0 = (tile_begin + k) * TS;
    const bool partial = (t0 < full_lo) || (t0 + TS > full_hi);

    // ---- S^T = K Q^T ------------------------------------------------------
    float s[T::MT][NH8][4];
#pragma unroll
    for (int mt = 0; mt < T::MT; ++mt) {
#pragma unroll
      for (int j = 0; j < NH8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[mt][j][e] = 0.f;
      if constexpr (!FP8) {
        const int mi = lane >> 3, rr = lane & 7;
        const int tok = mt * 16 + rr + ((mi & 1) << 3);
#pragma unroll
        for (int ks = 0; ks < T::KS; ++ks) {
          uint32_t a[4];
          ldsm_x4(a, kst_u + T::off(tok, (ks * 16 + ((mi >> 1) << 3)) * 2));
#pragma unroll
          for (int j = 0; j < NH8; ++j) mma_bf16(s[mt][j], a, qf[ks][j][0], qf[ks][j][1]);
        }
      } else {
        constexpr int NV = D / 64;  // 16-byte units per thread per row
        uint4 r0[NV], r1[NV];
#pragma unroll
        for (int u = 0; u < NV; ++u) {
          r0[u] = *reinterpret_cast<const uint4*>(kst + T::off(mt * 16 + g, c * (D / 4) + 16 * u));
          r1[u] = *reinterpret_cast<const uint4*>(kst + T::off(mt * 16 + g + 8, c * (D / 4) + 16 * u));
        }
        const uint32_t* w0 = reinterpret_cast<const uint32_t*>(r0);
        const uint32_t* w1 = reinterpret_cast<const uint32_t*>(r1);
#pragma unroll
        for (int ks = 0; ks < T::KS; ++ks) {
          uint32_t a[4];
          a[0] = dequant_e4m3x2<0>(w0[ks], k_sc2);
          a[1] = dequant_e4m3x2<0>(w1[ks], k_sc2);
          a[2] = dequant_e4m3x2<1>(w0[ks], k_sc2);
          a[3] = dequant_e4m3x2<1>(w1[ks], k_sc2);
#pragma unroll
          for (int j = 0; j < NH8; ++j) mma_bf16(s[mt][j], a, qf[ks][j][0], qf[ks][j][1]);
        }
      }
    }

    // ---- scale, soft-cap, mask; online softmax (log2 domain) ----------------
    float mx[NH8][2];
#pragma unroll
    for (int j = 0; j < NH8; ++j) mx[j][0] = mx[j][1] = -INFINITY;
    // the soft-cap is compiled in only where a call uses it, and the mask
    // only into the version that masked tiles take
    auto scores = [&](auto masked_tag) {
      constexpr bool MASKED = decltype(masked_tag)::value;
#pragma unroll
      for (int mt = 0; mt < T::MT; ++mt)
#pragma unroll
        for (int j = 0; j < NH8; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float v = s[mt][j][e];
            if constexpr (CAP) {
              v = p.cap_log2 * tanhf(v * p.scale_over_cap);
            } else {
              v *= p.scale_log2;
            }
            if constexpr (MASKED) {
              const int tok = t0 + mt * 16 + g + ((e >> 1) << 3);
              if (tok < tok_lo || tok >= tok_hi || tok > rpos[j][e & 1] || tok < rlo[j][e & 1]) v = -INFINITY;
            }
            s[mt][j][e] = v;
            mx[j][e & 1] = fmaxf(mx[j][e & 1], v);
          }
    };
    if (partial) {
      scores(std::true_type{});
    } else {
      scores(std::false_type{});
    }
    float alpha[NH8][2], mu[NH8][2];
    bool grew = false;   // some row's running maximum rose (else every alpha is ex2(0) = 1)
#pragma unroll
    for (int j = 0; j < NH8; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float m = mx[j][h];
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
        mx[j][h] = m;   // the row's largest score in this tile
        const float m_new = fmaxf(m_run[j][h], m);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        grew |= m_new > m_run[j][h];
        alpha[j][h] = ex2(m_run[j][h] - m_use);
        m_run[j][h] = m_new;
        mu[j][h] = m_use;
      }
    // the accumulators need rescaling only after a maximum rose somewhere in
    // the warp; multiplying by exactly 1 is skipped
    const bool rescale = __any_sync(0xffffffffu, grew);
#pragma unroll
    for (int j = 0; j < NH8; ++j) {
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int mt = 0; mt < T::MT; ++mt) {
        s[mt][j][0] = ex2(s[mt][j][0] - mu[j][0]);
        s[mt][j][1] = ex2(s[mt][j][1] - mu[j][1]);
        s[mt][j][2] = ex2(s[mt][j][2] - mu[j][0]);
        s[mt][j][3] = ex2(s[mt][j][3] - mu[j][1]);
        ls0 += s[mt][j][0] + s[mt][j][2];
        ls1 += s[mt][j][1] + s[mt][j][3];
      }
      l_run[j][0] = l_run[j][0] * alpha[j][0] + ls0;
      l_run[j][1] = l_run[j][1] * alpha[j][1] + ls1;
      if (rescale) {
#pragma unroll
        for (int i = 0; i < T::KS; ++i) {
          o[i][j][0] *= alpha[j][0];
          o[i][j][1] *= alpha[j][1];
          o[i][j][2] *= alpha[j][0];
          o[i][j][3] *= alpha[j][1];
        }
      }
    }
    // Does some row take more than 1/kHotShare of its (warp's) running
    // denominator from one key of this tile?  The denominator only grows, so
    // such a share bounds the key's final weight.  Weights here are at most 1
    // (every row's maximum is exact), so a tile where no row's maximum rose
    // cannot be hot once every row's denominator is at least kHotShare: the
    // lane reduction of the denominators runs only on the other tiles.
    bool hot = false;
    if (rescale || l_small) {
      bool small = false;
#pragma unroll
      for (int j = 0; j < NH8; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float l = l_run[j][h];
          l += __shfl_xor_sync(0xffffffffu, l, 4);
          l += __shfl_xor_sync(0xffffffffu, l, 8);
          l += __shfl_xor_sync(0xffffffffu, l, 16);
          hot |= rvalid[j][h] && ex2(mx[j][h] - mu[j][h]) * kHotShare > l;
          small |= rvalid[j][h] && l < kHotShare;
        }
      hot = __any_sync(0xffffffffu, hot);
      l_small = __any_sync(0xffffffffu, small);
    }

    // ---- O^T += V^T P^T -----------------------------------------------------
    // P = P_hi + P_lo, both bf16 (two MMAs, weights exact to ~2^-17), on
    // tiles where some row masks a key (sequence start or end, window edge, a
    // verify row's own position; masked keys' V rows are zeroed there) or
    // where some row's largest weight from this tile exceeds 1/kHotShare of
    // its running denominator.  One bf16 P is up to 2^-8 off per weight, which
    // a row does not average out when a few keys carry its weight; on the
    // other tiles every key's final weight is below 1/kHotShare and one bf16
    // P, with no masks, is used.  Three compiled versions, chosen per tile.
    auto pv = [&](auto exact_tag, auto mask_tag) {
      constexpr bool EXACT = decltype(exact_tag)::value;
      constexpr bool MASK = decltype(mask_tag)::value;   // (masked tiles are always exact)
#pragma unroll
      for (int mt = 0; mt < T::MT; ++mt) {
        uint32_t pb[NH8][2], pl[NH8][2];
#pragma unroll
        for (int j = 0; j < NH8; ++j) {
          const uint32_t h0 = pack_bf16x2(s[mt][j][0], s[mt][j][1]);
          const uint32_t h1 = pack_bf16x2(s[mt][j][2], s[mt][j][3]);
          pb[j][0] = movmatrix_t(h0);
          pb[j][1] = movmatrix_t(h1);
          if constexpr (EXACT) {
            const uint32_t l0 = pack_bf16x2(s[mt][j][0] - __uint_as_float(h0 << 16),
                                            s[mt][j][1] - __uint_as_float(h0 & 0xffff0000u));
            const uint32_t l1 = pack_bf16x2(s[mt][j][2] - __uint_as_float(h1 << 16),
                                            s[mt][j][3] - __uint_as_float(h1 & 0xffff0000u));
            pl[j][0] = movmatrix_t(l0);
            pl[j][1] = movmatrix_t(l1);
          }
        }
        // Masked keys have P = 0, but their V rows may be stale or NaN: zero
        // them in the fragment so 0 * NaN never reaches the accumulator.
        uint32_t vm_lo = 0xffffffffu, vm_hi = 0xffffffffu;
        if constexpr (MASK) {
          const int tk = t0 + mt * 16 + 2 * c;
          auto valid = [&](int t) { return t >= tok_lo && t < tok_hi; };
          vm_lo = (valid(tk) ? 0x0000ffffu : 0u) | (valid(tk + 1) ? 0xffff0000u : 0u);
          vm_hi = (valid(tk + 8) ? 0x0000ffffu : 0u) | (valid(tk + 9) ? 0xffff0000u : 0u);
        }
        if constexpr (!FP8) {
          const int mi = lane >> 3, rr = lane & 7;
          const int tok = mt * 16 + rr + ((mi >> 1) << 3);
#pragma unroll
          for (int i = 0; i < T::KS; ++i) {
            uint32_t a[4];
            ldsm_x4_t(a, vst_u + T::off(tok, (i * 16 + ((mi & 1) << 3)) * 2));
            if constexpr (MASK) {
              a[0] &= vm_lo;
              a[1] &= vm_lo;
              a[2] &= vm_hi;
              a[3] &= vm_hi;
            }
#pragma unroll
            for (int j = 0; j < NH8; ++j) {
              mma_bf16(o[i][j], a, pb[j][0], pb[j][1]);
              if constexpr (EXACT) mma_bf16(o[i][j], a, pl[j][0], pl[j][1]);
            }
          }
        } else {
          // thread g owns output dims [g*D/8, (g+1)*D/8): m-tile i row g -> dim
          // g*D/8 + 2i, row g+8 -> g*D/8 + 2i + 1.
          constexpr int NW = D / 32;  // 32-bit words per thread per row
          uint32_t ra[NW], rb[NW], rc[NW], rd[NW];
          const int rowa = mt * 16 + 2 * c;
#pragma unroll
          for (int u = 0; u < NW; u += 2) {
            const int byte = g * (D / 8) + 4 * u;
            const uint2 xa = *reinterpret_cast<const uint2*>(vst + T::off(rowa, byte));
            const uint2 xb = *reinterpret_cast<const uint2*>(vst + T::off(rowa + 1, byte));
            const uint2 xc = *reinterpret_cast<const uint2*>(vst + T::off(rowa + 8, byte));
            const uint2 xd = *reinterpret_cast<const uint2*>(vst + T::off(rowa + 9, byte));
            ra[u] = xa.x; ra[u + 1] = xa.y;
            rb[u] = xb.x; rb[u + 1] = xb.y;
            rc[u] = xc.x; rc[u + 1] = xc.y;
            rd[u] = xd.x; rd[u + 1] = xd.y;
          }
#pragma unroll
          for (int i = 0; i < T::KS; ++i) {
            const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
            const uint32_t x = __byte_perm(ra[i >> 1], rb[i >> 1], sel);
            const uint32_t y = __byte_perm(rc[i >> 1], rd[i >> 1], sel);
            uint32_t a[4];
            a[0] = dequant_e4m3x2<0>(x, v_sc2);
            a[1] = dequant_e4m3x2<1>(x, v_sc2);
            a[2] = dequant_e4m3x2<0>(y, v_sc2);
            a[3] = dequant_e4m3x2<1>(y, v_sc2);
            if constexpr (MASK) {
              a[0] &= vm_lo;
              a[1] &= vm_lo;
              a[2] &= vm_hi;
              a[3] &= vm_hi;
            }
#pragma unroll
            for (int j = 0; j < NH8; ++j) {
              mma_bf16(o[i][j], a, pb[j][0], pb[j][1]);
              if constexpr (EXACT) mma_bf16(o[i][j], a, pl[j][0], pl[j][1]);
            }
          }
        }
      }
    };
    if (partial) {
      pv(std::true_type{}, std::true_type{});
    } else if (hot) {
      pv(std::true_type{}, std::false_type{});
    } else {
      pv(std::false_type{}, std::false_type{});
    }

    __syncwarp();
    const int kn = k + NS * kWarps;
    if (lane == 0 && kn < n_tiles) {
      fence_proxy_async_smem();
      issue(kn, stage);
    }
  }

  // the merge kernel may start launching; it waits for this grid's partials
  pdl_launch_dependents();

  // ---- merge the 4 warps' states in shared memory ----------------------------
  // Every TMA a warp issued was waited for inside its loop, so its stage
  // buffers are free; each warp writes its state into its own region.
  float* wo = reinterpret_cast<float*>(wbase);   // [HW][D]
  float* wm = wo + T::HW * D;                     // [HW]
  float* wl = wm + T::HW;                         // [HW]
#pragma unroll
  for (int j = 0; j < NH8; ++j)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float l = l_run[j][h];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      if (g == 0) {
        wm[j * 8 + 2 * c + h] = m_run[j][h];
        wl[j * 8 + 2 * c + h] = l;
      }
    }
#pragma unroll
  for (int i = 0; i < T::KS; ++i)
#pragma unroll
    for (int j = 0; j < NH8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = j * 8 + 2 * c + (e & 1);
        const int d = FP8 ? (g * (D / 8) + 2 * i + (e >> 1)) : (16 * i + g + ((e >> 1) << 3));
        wo[h * D + d] = o[i][j][e];
      }
  __syncthreads();

  const bool direct = (r.n_splits == 1);
  for (int e = tid; e < R * D; e += kWarps * 32) {
    const int h = e / D;   // row within this kv head's rows
    const int d = e - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float* ww = reinterpret_cast<const float*>(smem + w * T::WARP_BYTES) + T::HW * D;
      M = fmaxf(M, ww[h]);
    }
    if (M == -INFINITY) M = 0.f;
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float* wob = reinterpret_cast<const float*>(smem + w * T::WARP_BYTES);
      const float f = ex2(wob[T::HW * D + h] - M);
      num += wob[h * D + d] * f;
      den += wob[T::HW * D + T::HW + h] * f;
    }
    const int tq = h / Gc;
    const int hq = kvh * G + head0 + (h - tq * Gc);
    const int64_t orow = qrow0 + tq;
    if (direct) {
      float M2 = M, zs = 0.f;
      if (p.sinks != nullptr) {
        const float sk = p.sinks[hq] * kLog2e;
        M2 = fmaxf(M, sk);
        zs = ex2(sk - M2);
      }
      const float f = ex2(M - M2);
      const float Z = den * f + zs;
      const float ov = (Z > 0.f) ? num * f / Z : 0.f;
      p.out[orow * p.out_stride_tok + static_cast<int64_t>(hq) * p.out_stride_head + d] =
          __bfloat16_as_ushort(__float2bfloat16_rn(ov));
      if (d == 0 && p.lse != nullptr) p.lse[orow * p.num_q_heads + hq] = (M2 + lg2(Z)) * kLn2;
    } else {
      const int64_t row = (orow * p.num_q_heads + hq) * p.max_splits + split;
      p.o_part[row * D + d] = (den > 0.f) ? num / den : 0.f;
      if (d == 0) p.lse_part[row] = (M + lg2(den)) * kLn2;
    }
  }
  if (direct || p.merge_cnt == nullptr) return;

  // ---- the last split of this (request, kv head group) to finish merges ----
  // Release: every thread's partials, then (thread 0) a fence and the
  // arrival.  The CTA whose arrival completes the count acquires them all.
  // No CTA waits for another, and the last one resets the counter.
  __syncthreads();
  int* s_last = reinterpret_cast<int*>(smem);   // warp states are no longer read
  if (tid == 0) {
    uint32_t* cnt = p.merge_cnt + static_cast<int64_t>(b) * gridDim.y + blockIdx.y;
    __threadfence();
    const uint32_t prev = atomicAdd(cnt, 1u);
    const int last = prev + 1 == static_cast<uint32_t>(r.n_splits);
    if (last) {
      atomicExch(cnt, 0u);
      __threadfence();
    }
    *s_last = last;
  }
  __syncthreads();
  if (*s_last == 0) return;
  merge_splits<D>(p, r.n_splits, R, Gc, kvh * G + head0, qrow0);
}

// LSE merge: one warp per (query row, q head); lane owns D/32 consecutive dims.
template <int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeParams p) {
  pdl_wait_primary();  // split partials complete and visible
  const int wid = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= p.batch * p.q_len * p.num_q_heads) return;
  const int row = wid / p.num_q_heads;
  const int hq = wid - row * p.num_q_heads;
  const int b = row / p.q_len;
  const SplitRange r = split_range(p, p.seq_lens[b]);
  if (r.n_splits <= 1) return;  // written by the split kernel (no keys, or one split)
  if (r.n_splits > p.max_splits) {  // seq_lens beyond the planned capacity
    if (lane == 0) atomicOr(p.err, kErrCapacity);
    return;
  }
  constexpr int V = D / 32;
  const bool has_sink = p.sinks != nullptr;
  const float sk = has_sink ? p.sinks[hq] * kLog2e : -INFINITY;
  uint16_t* outp = p.out + static_cast<int64_t>(row) * p.out_stride_tok + static_cast<int64_t>(hq) * p.out_stride_head;
  float acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  float M = sk;
  const int64_t row0 = (static_cast<int64_t>(row) * p.num_q_heads + hq) * p.max_splits;
  for (int s = lane; s < r.n_splits; s += 32) M = fmaxf(M, p.lse_part[row0 + s] * kLog2e);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float Z = 0.f;
  if (M != -INFINITY) {
    Z = has_sink ? ex2(sk - M) : 0.f;
    for (int s = 0; s < r.n_splits; ++s) {
      const float w = ex2(p.lse_part[row0 + s] * kLog2e - M);
      Z += w;
      const float* op = p.o_part + (row0 + s) * D + lane * V;
#pragma unroll
      for (int v = 0; v < V; v += 2) {
        const float2 x = *reinterpret_cast<const float2*>(op + v);
        acc[v] += w * x.x;
        acc[v + 1] += w * x.y;
      }
    }
  }
  const float inv = (Z > 0.f) ? 1.f / Z : 0.f;
#pragma unroll
  for (int v = 0; v < V; v += 2) {
    *reinterpret_cast<uint32_t*>(outp + lane * V + v) = pack_bf16x2(acc[v] * inv, acc[v + 1] * inv);
  }
  if (lane == 0 && p.lse != nullptr) {
    p.lse[static_cast<int64_t>(row) * p.num_q_heads + hq] = (M == -INFINITY) ? -INFINITY : (M + lg2(Z)) * kLn2;
  }
}

template <int D, bool FP8, int NH8, int TS, int NS>
cudaError_t launch_variant(const CUtensorMap& tmk, const CUtensorMap& tmv, const DecodeParams& p, dim3 grid,
                           int smem, cudaStream_t stream) {
  auto kern = p.cap_log2 > 0.f ? decode_split_kernel<D, FP8, NH8, TS, NS, true>
                               : decode_split_kernel<D, FP8, NH8, TS, NS, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (grid.x > 0 && grid.y > 0 && grid.z > 0) {
    kern<<<grid, kWarps * 32, smem, stream>>>(tmk, tmv, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // with one split per request the split kernel writes the outputs itself
  // (and flags any request that would need more), and with arrival counters
  // the last split of each request merges: no merge launch
  const int warps = p.batch * p.q_len * p.num_q_heads;
  if (warps > 0 && p.max_splits > 1 && p.merge_cnt == nullptr) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((warps + 3) / 4);
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_merge_kernel<D>, p);
  }
  return e;
}

template <int D, bool FP8>
struct TileChoice;
// Keys per stage and stages per warp (measured on GB300): bf16 head_dim 128
// takes 2 stages of 8 KB so three CTAs share an SM (5.73 vs 5.57 TB/s with 3
// stages); e4m3 caches take small stages so four CTAs share an SM and hide
// the dequantisation (head_dim 64: 2.30 vs 1.83 TB/s with 64-key stages;
// head_dim 128: 3.34 vs 3.01 with 32-key stages).
template <> struct TileChoice<64, false> { static constexpr int TS = 16, NS = 4; };
template <> struct TileChoice<128, false> { static constexpr int TS = 16, NS = 2; };
template <> struct TileChoice<256, false> { static constexpr int TS = 16, NS = 3; };
template <> struct TileChoice<64, true> { static constexpr int TS = 32, NS = 3; };
template <> struct TileChoice<128, true> { static constexpr int TS = 16, NS = 3; };
template <> struct TileChoice<256, true> { static constexpr int TS = 16, NS = 3; };

template <int D, bool FP8>
int smem_for(int bt_cache) {
  using C = TileChoice<D, FP8>;
  using T = Traits<D, FP8, 1, C::TS, C::NS>;
  return 1024 + kWarps * T::WARP_BYTES + kWarps * C::NS * 8 + bt_cache * 4;
}

template <int D, bool FP8>
cudaError_t launch_d(const DecodeConfig& cfg, const CUtensorMap& tmk, const CUtensorMap& tmv,
                     const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  using C = TileChoice<D, FP8>;
  if (cfg.nh8 == 1) return launch_variant<D, FP8, 1, C::TS, C::NS>(tmk, tmv, p, grid, cfg.smem_bytes, stream);
  return launch_variant<D, FP8, 2, C::TS, C::NS>(tmk, tmv, p, grid, cfg.smem_bytes, stream);
}

}  // namespace

DecodeConfig decode_config(int head_dim, bool fp8, int rows, int bt_cache) {
  DecodeConfig c{};
  c.head_dim = head_dim;
  c.fp8 = fp8;
  c.nh8 = rows <= 8 ? 1 : 2;
  c.warps = kWarps;
#define PA_TILE_CASE(DD, F8)                                    \
  if (head_dim == DD && fp8 == F8) {                            \
    c.tile_tokens = TileChoice<DD, F8>::TS;                     \
    c.stages = TileChoice<DD, F8>::NS;                          \
    c.smem_bytes = smem_for<DD, F8>(bt_cache);                  \
  }
  PA_TILE_CASE(64, false)
  PA_TILE_CASE(128, false)
  PA_TILE_CASE(256, false)
  PA_TILE_CASE(64, true)
  PA_TILE_CASE(128, true)
  PA_TILE_CASE(256, true)
#undef PA_TILE_CASE
  return c;
}

cudaError_t launch_decode(const DecodeConfig& cfg, const CUtensorMap& tmk, const CUtensorMap& tmv,
                          const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  switch (cfg.head_dim) {
    case 64: return cfg.fp8 ? launch_d<64, true>(cfg, tmk, tmv, p, grid, stream)
                            : launch_d<64, false>(cfg, tmk, tmv, p, grid, stream);
    case 128: return cfg.fp8 ? launch_d<128, true>(cfg, tmk, tmv, p, grid, stream)
                             : launch_d<128, false>(cfg, tmk, tmv, p, grid, stream);
    case 256: return cfg.fp8 ? launch_d<256, true>(cfg, tmk, tmv, p, grid, stream)
                             : launch_d<256, false>(cfg, tmk, tmv, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
