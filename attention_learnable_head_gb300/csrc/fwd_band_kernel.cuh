// Forward kernel for sliding-window layers, sm_103a (tcgen05 + TMA).
//
// Same mathematics as attn_sink_fwd_kernel (the concat listing
// "带汇聚的注意力（GPT-OSS）" on the euno.news page and the P_ij / P_ih
// equations of its section "数学公式"; sliding-window layers are what that
// page's section "FlashAttention V3 中的注意力汇聚支持" says the sinks
// stabilise), arranged for a causal window of W keys.
//
// Work item = T = 128 / G consecutive query tokens of one sequence x the G
// query heads of one kv group.  Its 128 query rows (row = token * G + head,
// the order in which [tokens][heads][64] holds them, so one TMA box fetches
// them) all read the same kv head and see keys from the window
// [i_first + off - W + 1, i_first + off + T - 1]: N = T + W - 1 keys, rounded
// up to 16.  One product S = Q K^T (M = 128, N <= 176) covers every key any
// row of the item sees.  With G = 8 and W = 128 that is N = 144 columns of
// which each row uses 128, against 256 of which 128 are used for a 128-token
// tile of one head.  Because the whole window fits one S, the softmax is a
// single pass: row max (with the sink logit), P = exp2(S * scale log2 e - m)
// in fp16, O = P V and l = sum P in one product (K = N), plus the sink's term
// 2^(sink log2 e - m); out = O / l, lse = ln 2 (m + log2 l); no running max,
// no rescaling of O.
//
// Persistent: gridDim.x CTAs (two per SM) walk the items item = blockIdx.x +
// k gridDim.x, ordered kv group fastest, then token blocks, then sequences;
// each role decodes the next item (its cu_seqlens entries) while it works on
// the current one.  The TMA warp loads Q into two stages and K/V into one
// (each released by the product that reads it), and prefetches into L2 the
// K/V window of the next item and the Q tile of the one after.  The MMA warp
// issues S of the next item right behind PV of the current one.  The softmax
// warps write an item's output once the next item's P is in TMEM, so that
// this epilogue overlaps the tensor cores' PV and next S; out and its
// residual go through SMEM tiles that TMA stores asynchronously (an item
// whose tokens run past its sequence's end writes its valid rows directly).
//
// TMEM (256 columns): S in [0, N) as fp32; the softmax writes P (fp16 pairs)
// over the S columns it has read, half 0 (keys [0, N0)) into columns
// [0, N0/2), half 1 (keys [N0, N)) into [N0, N0 + (N - N0)/2), so every
// 16-key step of PV reads 8 consecutive columns; O in [176, 256): the product
// has N = 80, its columns 64..79 multiplying a constant block of ones, so
// column 64 is the row sum of the fp16 P (no sum in the softmax).  S of the
// next item is issued after PV of this one, which reads P first (tcgen05 MMAs
// of a CTA run in issue order).
//
// Warp roles (320 threads): warps 0-3 softmax of key half 0, warps 4-7 of key
// half 1 (thread = query row = TMEM lane), warp 8 TMA producer, warp 9 MMA
// issuer and TMEM owner.
#pragma once
#include "fwd_kernel.cuh"

namespace attn_sink {

constexpr int kBandThreads = 320;
constexpr int kBandTmaWarp = 8;
constexpr int kBandMmaWarp = 9;
constexpr uint32_t kBandTmemCols = 256;
constexpr uint32_t kBandColO = 176;    // O: 64 fp32 columns, then the row sum (16 columns)
constexpr int kBandOCols = 80;         // N of the O product: 64 columns of V and one of ones
constexpr int kBandMaxCols = 176;      // N: fits S below O and two CTAs' SMEM per SM
constexpr int kBandCtasPerSm = 2;
// Dynamic SMEM: Q (2 x 16 KB), K and V (N x 128 B each), the out and residual
// staging tiles (2 x 16 KB), the ones block of the row sum (16 x 128 B), plus
// 1 KB of alignment slack.
constexpr int kBandOnesBytes = 16 * 128;
__host__ __device__ constexpr int band_smem_bytes(int n_cols) {
  return 1024 + 2 * (int)kTileBytes + 2 * n_cols * 128 + 2 * (int)kTileBytes + kBandOnesBytes;
}
constexpr int kBandSmemMax = band_smem_bytes(kBandMaxCols);

struct FwdBandParams {
  CUtensorMap tm_q;   // [T_q][H_q][64] bf16, box 64 x G x T, 128B swizzle
  CUtensorMap tm_k;   // [T_k][H_kv][64] bf16, box 64 x 1 x N
  CUtensorMap tm_v;   // [T_k][H_kv][64] fp16 copy of v, box 64 x 1 x N
  CUtensorMap tm_out;     // out, box as tm_q (stores)
  CUtensorMap tm_out_lo;  // residual, box as tm_q (stores; unused without it)
  const int* cu_q;    // null for a dense batch
  const int* cu_k;
  const float* sink;  // [H_q] fp32, or
  const __nv_bfloat16* sink_bf16;   // [H_q] bf16 when non-null
  __nv_bfloat16* out;     // [T_q][H_q][64]
  __nv_bfloat16* out_lo;  // residual O/l - out, or null
  float* lse;             // [H_q][T_q]
  int* err;
  int seqlen_q, seqlen_k;
  int total_q;
  int heads_q, heads_kv;
  int group, log2_group;  // G (a power of two dividing 128) and log2 G
  int tokens;             // T = 128 / G query tokens per item
  int n_cols;             // N: keys of an item's window (multiple of 16, <= 176)
  int half0_cols;         // keys [0, N0) are softmax half 0's (multiple of 16)
  int window;             // W >= 1
  float scale_log2;
  int chunk, q_pos0;      // key-chunk mode, as in FwdParams
  int n_tb;               // token blocks of the longest sequence
  int n_items;            // sequences x n_tb x H_kv (< 2^30)
  // n / H_kv and n / n_tb for 0 <= n < 2^31 as (n * mul) >> shift (fast_div)
  unsigned long long div_hkv_mul, div_tb_mul;
  int div_hkv_shift, div_tb_shift;
#ifdef ATTN_SINK_TEST_HOOKS
  int skip_k_tile;        // test build: no CTA issues K of its item with this index (-1: none)
#endif
};

// Division by a divisor fixed for the launch: q = (n * mul) >> (32 + s) with
// s = ceil(log2 d) and mul = ceil(2^(32+s) / d).  The product's excess over
// n / d is below n / 2^(32+s) < 1 / (2 d) for n < 2^31, which never reaches
// the next integer, so q = floor(n / d) exactly (Granlund and Montgomery,
// "Division by invariant integers using multiplication", PLDI 1994).
__host__ __device__ inline void fast_div_init(int d, unsigned long long* mul, int* shift) {
  int s = 0;
  while ((1ll << s) < d) ++s;
  *mul = ((1ull << (32 + s)) + (unsigned long long)d - 1) / (unsigned long long)d;
  *shift = 32 + s;
}
__device__ __forceinline__ int fast_div(int n, unsigned long long mul, int shift) {
  return (int)(((unsigned long long)(unsigned)n * mul) >> shift);
}

// Query / key bounds of one sequence (cu_seqlens entries, or the dense batch's).
struct SeqBounds {
  int q0, q1, k0, k1;
};

__device__ __forceinline__ SeqBounds band_bounds(const FwdBandParams& p, int item) {
  SeqBounds b{0, 0, 0, 0};
  if (item >= p.n_items) return b;
  const int seq = fast_div(fast_div(item, p.div_hkv_mul, p.div_hkv_shift), p.div_tb_mul,
                           p.div_tb_shift);
  if (p.cu_q != nullptr) {
    b.q0 = __ldg(p.cu_q + seq);
    b.q1 = __ldg(p.cu_q + seq + 1);
    b.k0 = __ldg(p.cu_k + seq);
    b.k1 = __ldg(p.cu_k + seq + 1);
  } else {
    b.q0 = seq * p.seqlen_q;
    b.q1 = b.q0 + p.seqlen_q;
    b.k0 = seq * p.seqlen_k;
    b.k1 = b.k0 + p.seqlen_k;
  }
  return b;
}

struct BandItem {
  SeqSpan sp;
  int g;          // kv head
  int i_first;    // first query token of the item, within its sequence
  int kb;         // key (within the sequence) of the window's first column
  bool valid;     // the item holds tokens of its sequence
};

__device__ __forceinline__ BandItem band_decode(const FwdBandParams& p, int item,
                                                const SeqBounds& b) {
  BandItem it;
  const int gq = fast_div(item, p.div_hkv_mul, p.div_hkv_shift);
  it.g = item - gq * p.heads_kv;
  const int tb = gq - fast_div(gq, p.div_tb_mul, p.div_tb_shift) * p.n_tb;
  it.sp.q0 = b.q0;
  it.sp.nq = b.q1 - b.q0;
  it.sp.k0 = b.k0;
  it.sp.nk = b.k1 - b.k0;
  it.i_first = tb * p.tokens;
  it.valid = item < p.n_items && it.i_first < it.sp.nq;
  // query token i sits at key position i + off (bottom-right unless chunk mode)
  const int off = p.chunk ? p.q_pos0 : it.sp.nk - it.sp.nq;
  it.kb = it.i_first + off - p.window + 1;
  return it;
}

// A CTA's walk over its items, skipping those past their sequence's end.  The
// bounds of the next candidate item are loaded when the current one starts,
// so their latency is hidden behind its work.
struct BandWalk {
  int item;
  BandItem it;
  SeqBounds next;

  __device__ __forceinline__ void skip_invalid(const FwdBandParams& p) {
    while (item < p.n_items && !it.valid) {
      item += gridDim.x;
      it = band_decode(p, item, band_bounds(p, item));
    }
    next = band_bounds(p, item + gridDim.x);
  }
  __device__ __forceinline__ void start(const FwdBandParams& p) {
    item = blockIdx.x;
    it = band_decode(p, item, band_bounds(p, item));
    skip_invalid(p);
  }
  __device__ __forceinline__ bool more(const FwdBandParams& p) const { return item < p.n_items; }
  __device__ __forceinline__ void advance(const FwdBandParams& p) {
    item += gridDim.x;
    it = band_decode(p, item, next);
    skip_invalid(p);
  }
};

template <int NC>
__device__ __forceinline__ void band_ld(uint32_t taddr, uint32_t* a) {
  if constexpr (NC == 32) tmem_ld_x32(taddr, a);
  else tmem_ld_x16(taddr, a);
}

template <int NC>
__device__ __forceinline__ void band_st(uint32_t taddr, const uint32_t* a) {
  if constexpr (NC == 32) tmem_st_x32(taddr, a);
  else tmem_st_x16(taddr, a);
}

// Row max of one chunk of S (raw scores) over the row's visible keys [lo, hi]
// (counted from the chunk's first column).  Columns outside become -inf, each
// bound checked only when some row of the warp crosses it in this chunk, and
// a chunk that had any is written back to TMEM so that the exponentials need
// no mask.  Returns whether it wrote one back (warp-uniform).
template <int NC>
__device__ __forceinline__ float band_chunk_max(uint32_t taddr, int lo, int hi, bool& wrote) {
  uint32_t a[NC];
  band_ld<NC>(taddr, a);
  tmem_ld_wait();
  // per 16-column block: a window edge inside a chunk usually crosses one
  bool cut = false;
  #pragma unroll
  for (int b = 0; b < NC; b += 16) {
    if (__any_sync(0xffffffffu, lo > b)) {
      cut = true;
      #pragma unroll
      for (int e = b; e < b + 16; ++e)
        if (e < lo) a[e] = __float_as_uint(-INFINITY);
    }
    if (__any_sync(0xffffffffu, hi < b + 15)) {
      cut = true;
      #pragma unroll
      for (int e = b; e < b + 16; ++e)
        if (e > hi) a[e] = __float_as_uint(-INFINITY);
    }
  }
  if (cut) {
    band_st<NC>(taddr, a);
    wrote = true;
  }
  float q0 = __uint_as_float(a[0]), q1 = __uint_as_float(a[1]);
  #pragma unroll
  for (int e = 2; e + 3 < NC; e += 4) {
    q0 = fmax3(q0, __uint_as_float(a[e]), __uint_as_float(a[e + 1]));
    q1 = fmax3(q1, __uint_as_float(a[e + 2]), __uint_as_float(a[e + 3]));
  }
  q0 = fmax3(q0, __uint_as_float(a[NC - 2]), __uint_as_float(a[NC - 1]));
  return fmaxf(q0, q1);
}

// P = exp2(S * scale log2 e - m) of one chunk (masked columns hold -inf and
// give 0), written as fp16 pairs to TMEM at tp (NC / 2 columns).  The row sum
// of P is not formed here: the O product sums the fp16 P it multiplies.
template <int NC>
__device__ __forceinline__ void band_chunk_exp(uint32_t ts, uint32_t tp, uint64_t sl2x2,
                                               uint64_t negm2) {
  uint32_t a[NC];
  band_ld<NC>(ts, a);
  tmem_ld_wait();
  uint32_t pk[NC / 2];
  #pragma unroll
  for (int e = 0; e < NC; e += 2) {
    const uint64_t x =
        ffma2(f2(__uint_as_float(a[e]), __uint_as_float(a[e + 1])), sl2x2, negm2);
    pk[e >> 1] = pack_f16x2(ex2_approx(f2_lo(x)), ex2_approx(f2_hi(x)));
  }
  if constexpr (NC == 32) tmem_st_x16(tp, pk);
  else tmem_st_x8(tp, pk);
}

// Registers are split per SM sub-partition; two CTAs of 10 warps allow 102
// per thread: 96 is used.
__global__ void __maxnreg__(96)
attn_sink_fwd_band_kernel(const __grid_constant__ FwdBandParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t q_full[2], q_empty[2];
  __shared__ __align__(8) uint64_t k_full, k_empty, v_full, v_empty;
  __shared__ __align__(8) uint64_t s_full, p_full, pv_done, o_free, mma_drained;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;
  // The halves' row maxima ([half][row]).  One buffer is enough: S of the
  // next item, before whose pass 1 a half rewrites its entry, needs P of this
  // item from every thread, i.e. after its partner read it.
  __shared__ float s_mx[2][kBlockM];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int N = p.n_cols;
  const uint32_t kv_bytes = (uint32_t)N * 128u;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                        // 2 stages x 16 KB
  uint8_t* sK = sQ + 2 * kTileBytes;         // N x 128 B
  uint8_t* sV = sK + kv_bytes;               // N x 128 B
  uint8_t* sOut = sV + kv_bytes;             // 16 KB out tile, then 16 KB residual tile
  uint8_t* sOutLo = sOut + kTileBytes;
  uint8_t* sOnes = sOutLo + kTileBytes;      // 16 rows x 128 B, see below

  // The ones block: the second 64-wide block of the O product's B operand (V
  // is MN-major, 128-byte rows of 64 values), read for every 16-key step: 16
  // rows whose first value (output column 64, the row sum) is 1 and the rest 0,
  // 128B-swizzled like the V rows (16-byte chunk j of row r at chunk j ^ (r % 8)).
  for (int i = tid; i < kBandOnesBytes / 4; i += kBandThreads) {
    const int row = i >> 5, word = i & 31;             // 32 words a row
    const int first = ((0 ^ (row & 7)) << 2);          // word 0 of chunk 0, swizzled
    reinterpret_cast<uint32_t*>(sOnes)[i] = (word == first) ? 0x3C00u : 0u;   // fp16 1.0
  }
  fence_proxy_async_smem();                            // the MMA (async proxy) reads it
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    mbar_init(&k_full, 1);
    mbar_init(&k_empty, 1);
    mbar_init(&v_full, 1);
    mbar_init(&v_empty, 1);
    mbar_init(&s_full, 1);
    mbar_init(&p_full, 2 * kBlockM);
    mbar_init(&pv_done, 1);
    mbar_init(&o_free, 2 * kBlockM);
    mbar_init(&mma_drained, 1);
    fence_mbarrier_init();
  }
  if (warp == kBandMmaWarp) {
    tmem_alloc(&tmem_base_sh, kBandTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == kBandTmaWarp) {
    // ---------------------------------------------------------------- TMA producer
    // Item li (this CTA's li-th item): Q into stage li % 2 once S of item li - 2
    // has completed; K once S of item li - 1 has completed; V once PV of item
    // li - 1 has completed.
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_out);
      if (p.out_lo) tma_prefetch_desc(&p.tm_out_lo);
      const uint64_t keep = l2_policy_evict_last();    // K/V: re-read by neighbouring items
      const uint64_t once = l2_policy_evict_first();   // Q: read by this item only
      int last_q[2] = {-1, -1};
      int last_k = -1, last_v = -1;
      int li = 0;
      bool ok = true;
      BandWalk w, w1, w2;                    // this item, the next, the one after
      w.start(p);
      w1 = w;
      if (w1.more(p)) w1.advance(p);
      w2 = w1;
      if (w2.more(p)) w2.advance(p);
      for (; w.more(p); w.advance(p)) {
        const BandItem& it = w.it;
        // into L2 ahead of their loads: the next item's K/V window, and the Q
        // tile of the item after it
        if (w1.more(p)) {
          tma_prefetch_l2_3d(&p.tm_k, 0, w1.it.g, w1.it.sp.k0 + w1.it.kb);
          tma_prefetch_l2_3d(&p.tm_v, 0, w1.it.g, w1.it.sp.k0 + w1.it.kb);
        }
        if (w2.more(p))
          tma_prefetch_l2_3d(&p.tm_q, 0, w2.it.g * p.group, w2.it.sp.q0 + w2.it.i_first);
        const int qs = li & 1;
        if (li >= 2 && !mbar_wait(&q_empty[qs], ((li >> 1) & 1) ^ 1, &abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&q_full[qs], kTileBytes);
        tma_load_3d_hint(&p.tm_q, &q_full[qs], sQ + qs * kTileBytes, 0, it.g * p.group,
                         it.sp.q0 + it.i_first, once);
        last_q[qs] = li;
        if (li >= 1 && !mbar_wait(&k_empty, (li & 1) ^ 1, &abort_flag)) {
          ok = false;
          break;
        }
        if (TEST_HOOK_FWD_ISSUE_K(li)) {
          mbar_arrive_expect_tx(&k_full, kv_bytes);
          tma_load_3d_hint(&p.tm_k, &k_full, sK, 0, it.g, it.sp.k0 + it.kb, keep);
          last_k = li;
        }
        if (li >= 1 && !mbar_wait(&v_empty, (li & 1) ^ 1, &abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&v_full, kv_bytes);
        tma_load_3d_hint(&p.tm_v, &v_full, sV, 0, it.g, it.sp.k0 + it.kb, keep);
        last_v = li;
        ++li;
        if (w1.more(p)) w1.advance(p);
        if (w2.more(p)) w2.advance(p);
      }
      if (!ok) {
        abort_flag = 1;
        atomicCAS(p.err, 0, DEVERR_TIMEOUT_FWD + 4);
      }
      // Every copy lands before the CTA releases SMEM, also when another role
      // gave up: the last copy issued into each stage (the earlier ones had
      // completed before it was issued).
      for (int s = 0; s < 2; ++s)
        if (last_q[s] >= 0) mbar_wait(&q_full[s], (last_q[s] >> 1) & 1, nullptr);
      if (last_k >= 0) mbar_wait(&k_full, last_k & 1, nullptr);
      if (last_v >= 0) mbar_wait(&v_full, last_v & 1, nullptr);
    }
  } else if (warp == kBandMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    // Per item: S = Q K^T (M = 128, N, K = 64, bf16) into columns [0, N); once
    // the softmax has written P over them, O = P V (M = 128, N = 64, K = N,
    // A from TMEM, V fp16 from SMEM) into the O columns, after the previous
    // item's O has been read out.
    if (lane == 0) {
      const uint32_t idesc_s = make_idesc_bf16(kBlockM, N, false, false);
      const uint32_t idesc_o = make_idesc(kFmtF16, kBlockM, kBandOCols, false, true);
      const uint64_t dQ0 = make_sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dK = make_sdesc_sw128(smem_u32(sK), 16, 1024);
      // V, MN-major; its second 64-wide block (output columns 64..127, of which
      // the product reads 64..79) is the ones block, at the distance LBO from
      // each 16-key step's start
      const uint64_t dV = make_sdesc_sw128(smem_u32(sV), smem_u32(sOnes) - smem_u32(sV), 1024);
      constexpr uint32_t kQU = kTileBytes >> 4;
      const int ks0 = p.half0_cols >> 4;   // 16-key steps of half 0
      const int nks = N >> 4;
      int li = 0;
      bool ok = true;
      BandWalk w;
      w.start(p);
      bool have = w.more(p);
      while (have) {
        const int qs = li & 1;
        if (!mbar_wait(&q_full[qs], (li >> 1) & 1, &abort_flag) ||
            !mbar_wait(&k_full, li & 1, &abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        #pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k)
          mma_ss(tmem, dQ0 + qs * kQU + 2 * k, dK + 2 * k, idesc_s, k > 0);
        mma_commit(&s_full);
        mma_commit(&q_empty[qs]);
        mma_commit(&k_empty);
        // whether another item follows, found while the softmax works on this one
        w.advance(p);
        have = w.more(p);
        if (!mbar_wait(&p_full, li & 1, &abort_flag) || !mbar_wait(&v_full, li & 1, &abort_flag) ||
            (li > 0 && !mbar_wait(&o_free, (li - 1) & 1, &abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // P of half 0 in columns [0, N0/2), of half 1 from column N0 on
        uint32_t a_col = tmem;
        uint64_t b_desc = dV;
        mma_ts(tmem + kBandColO, a_col, b_desc, idesc_o, 0);
        for (int kk = 1; kk < nks; ++kk) {
          a_col += (kk == ks0) ? 8u + 8u * ks0 : 8u;
          // start 2048 bytes (16 rows) on, LBO 2048 bytes less: still the ones block
          b_desc += 128u;
          b_desc -= (uint64_t)128u << 16;
          mma_ts(tmem + kBandColO, a_col, b_desc, idesc_o, 1);
        }
        mma_commit(&pv_done);
        mma_commit(&v_empty);
        ++li;
      }
      if (!ok) {
        abort_flag = 1;
        atomicCAS(p.err, 0, DEVERR_TIMEOUT_FWD + 5);
      }
      // Drain: every MMA issued above has finished before TMEM is released.
      mma_commit(&mma_drained);
      mbar_wait(&mma_drained, 0, nullptr);
    }
  } else {
    // ---------------------------------------------------------------- softmax warps
    // Half c = warp / 4 owns keys [c0, c0 + nc) of every row; thread = row r =
    // token t * G + head hh.  The epilogue of item li - 1 (out = O / l, lse)
    // runs after P of item li is in TMEM: its O is read out first (which lets
    // PV of item li proceed), and the rest overlaps PV of item li and S of
    // item li + 1 on the tensor cores.  Every warp reaches every named barrier
    // (the pair barrier with its partner warp each item, the 256-thread
    // barriers of each epilogue), so a failed wait makes all of them leave
    // together.
    const int c = warp >> 2;
    const int r = tid & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int c0 = c ? p.half0_cols : 0;
    const int nc = c ? N - p.half0_cols : p.half0_cols;
    const uint32_t tS = tmem + lane_base + (uint32_t)c0;
    const uint32_t tO = tmem + lane_base + kBandColO + 32u * c;
    const int t = r >> p.log2_group;          // token of this row within the item
    const int hh = r & (p.group - 1);         // query head within the kv group
    const bool leader = (warp == 0 && lane == 0);   // issues the items' TMA stores
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2(sl2, sl2);
    const uint64_t store_policy = l2_policy_evict_first();
    int li = 0;
    bool ok = true;
    // the previous item: kv head, first token (in the packed tensor), tokens
    // left in its sequence from there, this row's max (log2 units)
    int pg = 0, ptok = 0, prem = 0;
    float pm = -INFINITY;
    float psink = 0.0f;   // the previous item's sink term of the row sum, 2^(sink - m)
    BandWalk w;
    w.start(p);
    while (true) {
      const bool have = w.more(p);
      int ng = 0, ntok = 0, nrem = 0;
      float m = -INFINITY, nsink = 0.0f;
      if (have) {
        const BandItem& it = w.it;
        const int h = it.g * p.group + hh;
        // chunk mode: no sink (its logit is -inf, i.e. absent from the normaliser)
        const float sink_h = p.chunk       ? -INFINITY
                            : p.sink_bf16 ? __bfloat162float(p.sink_bf16[h])
                                          : __ldg(p.sink + h);
        // the row's visible keys as window columns, relative to this half's first
        const int lo = max(t, -it.kb) - c0;
        const int hi = min(t + p.window - 1, it.sp.nk - 1 - it.kb) - c0;
        ng = it.g;
        ntok = it.sp.q0 + it.i_first;
        nrem = it.sp.nq - it.i_first;

        const bool got = ok && mbar_wait_warp(&s_full, li & 1, &abort_flag);
        float mx = -INFINITY;
        if (got) {
          tc_fence_after();
          bool wrote = false;
          int cc = 0;
          #pragma unroll 1
          for (; cc + 32 <= nc; cc += 32)
            mx = fmaxf(mx, band_chunk_max<32>(tS + cc, lo - cc, hi - cc, wrote));
          if (cc < nc) mx = fmaxf(mx, band_chunk_max<16>(tS + cc, lo - cc, hi - cc, wrote));
          if (wrote) tmem_st_wait();   // the masked chunks are back before pass 2 reads them
          s_mx[c][r] = mx;
        }
        ok = named_barrier_and(2 + (warp & 3), 64, got);
        if (ok) {
          const float sink_l2 = sink_h * kLog2e;          // -inf without a sink
          m = fmaxf(fmaxf(mx, s_mx[c ^ 1][r]) * sl2, sink_l2);
          const float m_use = (m == -INFINITY) ? 0.0f : m;
          const uint64_t negm2 = f2(-m_use, -m_use);

          // P of keys [cc, cc + 32) goes to columns [cc / 2, cc / 2 + 16) of the
          // half: S columns this thread has already read.
          int cc = 0;
          #pragma unroll 1
          for (; cc + 32 <= nc; cc += 32)
            band_chunk_exp<32>(tS + cc, tS + (cc >> 1), sl2x2, negm2);
          if (cc < nc) band_chunk_exp<16>(tS + cc, tS + (cc >> 1), sl2x2, negm2);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&p_full);
          if (sink_h > -INFINITY) nsink = ex2_approx(sink_l2 - m_use);
        } else {
          abort_flag = 1;
        }
      }
      if (li > 0) {
        // ---- epilogue of item li - 1: out = O / l (bf16, plus the residual), lse.
        // The staging tiles are free once the stores of item li - 2 have read them.
        if (leader) bulk_wait_group_read0();
        const bool fin = ok && mbar_wait_warp(&pv_done, (li - 1) & 1, &abort_flag);
        if (!named_barrier_and(1, 2 * kBlockM, fin)) {
          abort_flag = 1;
          atomicCAS(p.err, 0, DEVERR_TIMEOUT_FWD + 6);
          break;
        }
        tc_fence_after();
        // the row sum: the O product's column 64 (the fp16 P it multiplied,
        // summed in fp32) plus the sink's term
        uint32_t o[32];
        tmem_ld_x32(tO, o);
        const uint32_t lsum = tmem_ld_x1(tO - 32u * c + 64u);
        tmem_ld_wait();
        const float lt = __uint_as_float(lsum) + psink;
        tc_fence_before();
        mbar_arrive(&o_free);
        const float inv_l = (lt > 0.0f) ? 1.0f / lt : 0.0f;
        const bool whole = prem >= p.tokens;      // same for every row of the item
        const int h = pg * p.group + hh;
        const size_t row = (size_t)(ptok + t);
        const uint64_t inv_l2 = f2(inv_l, inv_l);
        #pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t hi2[4], lo2[4];
          #pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint64_t f = fmul2(f2(__uint_as_float(o[8 * u + 2 * e]),
                                        __uint_as_float(o[8 * u + 2 * e + 1])), inv_l2);
            hi2[e] = pack_bf16x2(f2_lo(f), f2_hi(f));
            const uint64_t res = fsub2(f, f2(bf16_lo(hi2[e]), bf16_hi(hi2[e])));
            lo2[e] = pack_bf16x2(f2_lo(res), f2_hi(res));
          }
          if (whole) {
            // row r of the item's [T][G][64] box, 128B-swizzled like the TMA tile
            const uint32_t off = sw128_offset((uint32_t)r, (uint32_t)(4 * c + u));
            st_shared_v4(smem_u32(sOut) + off, hi2[0], hi2[1], hi2[2], hi2[3]);
            if (p.out_lo) st_shared_v4(smem_u32(sOutLo) + off, lo2[0], lo2[1], lo2[2], lo2[3]);
          } else if (t < prem) {
            const size_t base = (row * p.heads_q + h) * kHeadDim + 32 * c;
            reinterpret_cast<uint4*>(p.out + base)[u] = make_uint4(hi2[0], hi2[1], hi2[2], hi2[3]);
            if (p.out_lo)
              reinterpret_cast<uint4*>(p.out_lo + base)[u] =
                  make_uint4(lo2[0], lo2[1], lo2[2], lo2[3]);
          }
        }
        if (c == 0 && t < prem)
          p.lse[(size_t)h * p.total_q + row] = (lt > 0.0f) ? (pm + __log2f(lt)) * kLn2 : -INFINITY;
        if (whole) {
          fence_proxy_async_smem();
          named_barrier_sync(6, 2 * kBlockM);
          if (leader) {
            tma_store_3d_hint(&p.tm_out, sOut, 0, pg * p.group, ptok, store_policy);
            if (p.out_lo) tma_store_3d_hint(&p.tm_out_lo, sOutLo, 0, pg * p.group, ptok, store_policy);
            bulk_commit_group();
          }
        }
      }
      if (!have) break;
      pg = ng;
      ptok = ntok;
      prem = nrem;
      pm = m;
      psink = nsink;
      ++li;
      w.advance(p);
    }
    // the last stores have read their SMEM tiles before the CTA ends
    if (leader) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kBandMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kBandTmemCols);
  }
}

}  // namespace attn_sink
