// Forward kernel: attention with a per-head sink, sm_103a (tcgen05 + TMA).
//
// One CTA per (query head h, sequence, 128-row query tile); two CTAs share an
// SM (320 threads x 96 registers, ~100 KB of SMEM and 256 TMEM columns each).
// Per key tile n:
//   S(n) = Q K_n^T (tcgen05, bf16 operands from SMEM, fp32 accumulators in TMEM),
//   online softmax whose running max and sum start from the sink logit
//   (m0 = sink[h] * log2 e, l0 = 1 in the exp2 domain),
//   P(n) (fp16) written to TMEM and consumed there by O += P(n) V_n (tcgen05, A
//   from TMEM; V read as fp16 from SMEM, converted into the workspace before
//   launch),
// then out = O / l (bf16, plus optionally the bf16 residual O/l - out) and
// lse = ln 2 * (m + log2 l), which includes the sink.  S = Q K^T multiplies the
// bf16 inputs exactly; P and V go to the tensor cores as fp16 (11-bit
// significand) so that O, and the backward's D = rowsum(dO o O), keep ~3 more
// bits than a bf16 P would give.
// The sink joins the softmax denominator only: it is the extra column of the
// concat listing "带汇聚的注意力（GPT-OSS）" on the euno.news page, and the
// P_ij / P_ih equations of its section "数学公式".
//
// Pipelining.  P has TMEM columns of its own, so S(n+1) is issued as soon as
// the softmax warps have read S(n) out of TMEM, before PV(n): the tensor cores
// compute the next scores while this tile's exponentials run, and the softmax
// warps find S(n+1) ready when they finish P(n).  Before writing P(n+1) they
// wait for PV(n) (which reads the P columns and updates O).  K and V come
// through separate rings (K: 3 stages, released by S; V: 2 stages, released by
// PV), because K(n+2) is needed before V(n+1).
//
// Each key tile's 128 columns are two halves of 64 (c = 0, 1), one softmax
// warpgroup each (thread = query row = TMEM lane).  The halves of a row
// exchange their maxima through SMEM once per tile and share one running max
// and one O; each keeps its part of the row sum (the sink's term in half 0).
// Rescaling of O is lazy: the running max only moves when a row's max grows by
// more than kRescaleThreshold (log2 units); P stays below 2^threshold, and
// out/lse are exact because l and O use the same max.
//
// Warp roles (320 threads):
//   warps 0-3   softmax of key half 0
//   warps 4-7   softmax of key half 1
//   warp 8      TMA producer: Q once, then K and V tiles through their rings
//   warp 9      MMA issuer (one lane) and TMEM owner
// TMEM columns (256 allocated): S 0-127 (fp32), P 128-191 (128 keys as fp16
// pairs), O 192-255 (fp32).
#pragma once
#include <cuda_bf16.h>
#include "sm103_ptx.cuh"

namespace attn_sink {

constexpr int kBlockM = 128;   // query rows per tile
constexpr int kBlockN = 128;   // keys per tile
constexpr int kHeadDim = 64;
constexpr uint32_t kTileBytes = kBlockM * kHeadDim * 2;   // 16 KB bf16 tile
constexpr uint32_t kPTileBytes = kBlockM * kBlockN * 2;   // 32 KB bf16 tile (bwd dS)

#ifdef ATTN_SINK_TEST_HOOKS
// test build: K tile n is issued unless the params say to withhold it, so that
// the waits for it run out (the bounded-wait path is exercised without a fault)
#define TEST_HOOK_FWD_ISSUE_K(n) ((n) != p.skip_k_tile)
#else
#define TEST_HOOK_FWD_ISSUE_K(n) true
#endif

// An unused entry of a tile-order table (schedule_kernel.cuh).
constexpr uint32_t kNoWork = 0xFFFFFFFFu;

constexpr int kFwdKStages = 3;      // K ring depth
constexpr int kFwdVStages = 2;      // V ring depth
constexpr int kFwdThreads = 320;    // 8 softmax warps, TMA warp, MMA warp
constexpr int kFwdTmaWarp = 8;
constexpr int kFwdMmaWarp = 9;
constexpr uint32_t kFwdTmemCols = 256;
constexpr uint32_t kFwdColS = 0;    // S: 128 fp32 columns
constexpr uint32_t kFwdColP = 128;  // P: 128 keys as fp16 pairs, 64 columns
constexpr uint32_t kFwdColO = 192;  // O: 64 fp32 columns
constexpr int kFwdSmemBytes = 1024 + (int)kTileBytes * (1 + kFwdKStages + kFwdVStages);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;

struct FwdParams {
  CUtensorMap tm_q;   // [T_q][H_q][64] bf16, box 64 x 1 x 128, 128B swizzle
  CUtensorMap tm_k;   // [T_k][H_kv][64]
  CUtensorMap tm_v;
  CUtensorMap tm_out;     // out, box 64 x 1 x 128 (stores of whole tiles)
  CUtensorMap tm_out_lo;  // its residual (unused without one)
  const int* cu_q;    // null for a dense batch
  const int* cu_k;
  const float* sink;  // [H_q] fp32, or
  const __nv_bfloat16* sink_bf16;   // [H_q] bf16 when non-null
  __nv_bfloat16* out; // [T_q][H_q][64]
  __nv_bfloat16* out_lo; // [T_q][H_q][64] residual O/l - out, or null
  float* lse;         // [H_q][T_q]
  int* err;           // device error word
  int seqlen_q, seqlen_k;
  int total_q;
  int heads_q, group;
  int causal, window;
  float scale_log2;   // softmax_scale * log2(e)
  int n_qtiles;       // 128-row query tiles of the longest sequence
  // Packed batches of several sequences: the tile of CTA row blockIdx.y, as
  // seq << 16 | query tile, heaviest first (null: blockIdx.y / z give them)
  const uint32_t* work;
  // Key-chunk mode: no sink term, and query row i of every sequence sits at key
  // position i + q_pos0 (the default is bottom-right: q_pos0 = N_k - N_q).
  int chunk;
  int q_pos0;
#ifdef ATTN_SINK_TEST_HOOKS
  int skip_k_tile;    // test build: the producer never issues this K tile (-1: none)
#endif
};

struct SeqSpan {
  int q0, nq, k0, nk;
};

__device__ __forceinline__ SeqSpan seq_span(const int* cu_q, const int* cu_k, int seq,
                                            int seqlen_q, int seqlen_k) {
  SeqSpan s;
  if (cu_q != nullptr) {
    s.q0 = __ldg(cu_q + seq);
    s.nq = __ldg(cu_q + seq + 1) - s.q0;
    s.k0 = __ldg(cu_k + seq);
    s.nk = __ldg(cu_k + seq + 1) - s.k0;
  } else {
    s.q0 = seq * seqlen_q;
    s.nq = seqlen_q;
    s.k0 = seq * seqlen_k;
    s.nk = seqlen_k;
  }
  return s;
}

// Key tiles [lo, lo + num) that query rows [r0, r1] (inclusive) can see.
struct KeyRange {
  int lo, num;
};

__device__ __forceinline__ KeyRange key_tiles(int r0, int r1, const SeqSpan& sp, int off,
                                              int causal, int window) {
  KeyRange kr{0, 0};
  if (r1 < r0) return kr;
  int kv_lo = 0, kv_hi = sp.nk;
  if (causal) {
    kv_hi = min(sp.nk, r1 + off + 1);
    if (window > 0) kv_lo = max(0, r0 + off - window + 1);
  }
  if (kv_hi <= kv_lo) return kr;
  kr.lo = kv_lo / kBlockN;
  kr.num = (kv_hi + kBlockN - 1) / kBlockN - kr.lo;
  return kr;
}

// Registers are split per SM sub-partition (16384 each); two CTAs of 10 warps
// place 5 warps on each, so a thread may use at most 102: 96 is used.
__global__ void __maxnreg__(96)
attn_sink_fwd_kernel(const __grid_constant__ FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t q_full, mma_drained;
  __shared__ __align__(8) uint64_t k_full[kFwdKStages], k_empty[kFwdKStages];
  __shared__ __align__(8) uint64_t v_full[kFwdVStages], v_empty[kFwdVStages];
  __shared__ __align__(8) uint64_t s_full, s_free, p_full, pv_done;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;
  __shared__ float s_mx[2][2][kBlockM];   // [tile parity][half][row]: the halves' row maxima
  __shared__ float s_red_l[2][kBlockM];   // [half][row], epilogue only

  // Heads vary fastest (the query heads of a GQA group share K/V tiles in L2),
  // then query tiles, longest work first, then sequences, so the CTAs resident
  // at one time read one sequence's keys; a packed batch of several sequences
  // takes its tiles from a table sorted by work across all sequences.
  const int h = blockIdx.x;
  int qtile, seq;
  if (p.work != nullptr) {
    const uint32_t wk = p.work[blockIdx.y];
    if (wk == kNoWork) return;                            // uniform per CTA
    seq = (int)(wk >> 16);
    qtile = (int)(wk & 0xFFFFu);
  } else {
    qtile = p.n_qtiles - 1 - (int)blockIdx.y;
    seq = blockIdx.z;
  }
  const SeqSpan sp = seq_span(p.cu_q, p.cu_k, seq, p.seqlen_q, p.seqlen_k);
  const int i0 = qtile * kBlockM;
  if (i0 >= sp.nq) return;                                // uniform per CTA
  const int g = h / p.group;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int tile_r1 = min(i0 + kBlockM, sp.nq) - 1;       // last row of the tile
  // key position of query row 0 (bottom-right alignment unless chunk mode sets it)
  const int off = p.chunk ? p.q_pos0 : sp.nk - sp.nq;
  const KeyRange kr = key_tiles(i0, tile_r1, sp, off, p.causal, p.window);
  const int lo = kr.lo, num = kr.num;
  // chunk mode: no sink (its logit is -inf, i.e. absent from the normaliser)
  const float sink_h = p.chunk       ? -INFINITY
                      : p.sink_bf16 ? __bfloat162float(p.sink_bf16[h])
                                    : __ldg(p.sink + h);

  if (num == 0) {
    // No row of this tile sees a key: out = 0, lse = sink (the sink alone).
    for (int t = tid; t < kBlockM; t += kFwdThreads) {
      if (i0 + t < sp.nq) {
        const size_t row = (size_t)(sp.q0 + i0 + t);
        uint4* o = reinterpret_cast<uint4*>(p.out + (row * p.heads_q + h) * kHeadDim);
        #pragma unroll
        for (int c = 0; c < 8; ++c) o[c] = make_uint4(0, 0, 0, 0);
        if (p.out_lo) {
          uint4* ol = reinterpret_cast<uint4*>(p.out_lo + (row * p.heads_q + h) * kHeadDim);
          #pragma unroll
          for (int c = 0; c < 8; ++c) ol[c] = make_uint4(0, 0, 0, 0);
        }
        p.lse[(size_t)h * p.total_q + row] = sink_h;
      }
    }
    return;
  }

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + kTileBytes;
  uint8_t* sV = sK + kFwdKStages * kTileBytes;

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&q_full, 1);
    mbar_init(&mma_drained, 1);
    for (int s = 0; s < kFwdKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kFwdVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(&s_full, 1);
    mbar_init(&s_free, 2 * kBlockM);
    mbar_init(&p_full, 2 * kBlockM);
    mbar_init(&pv_done, 1);
    fence_mbarrier_init();
  }
  if (warp == kFwdMmaWarp) {
    tmem_alloc(&tmem_base_sh, kFwdTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == kFwdTmaWarp) {
    // ---------------------------------------------------------------- TMA producer
    // Two rings filled in the order the MMA thread consumes them: K(n) is read
    // by S(n) only (3 stages, released when S(n) completes), V(n) by PV(n) only
    // (2 stages, released when PV(n) completes).  One thread polls both rings'
    // release barriers and issues whichever copy is free, so K runs up to three
    // tiles ahead regardless of when the V stages come back.
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      const uint64_t keep = l2_policy_evict_last();
      mbar_arrive_expect_tx(&q_full, kTileBytes);
      tma_load_3d(&p.tm_q, &q_full, sQ, 0, h, sp.q0 + i0);
      int nk = 0, nv = 0;                    // copies issued so far
      unsigned long long t_last = global_timer_ns();
      bool ok = true;
      while (nk < num || nv < num) {
        bool progress = false;
        // K(nk): its stage was last read by S(nk - 3)
        if (nk < num && TEST_HOOK_FWD_ISSUE_K(nk) && (nk < kFwdKStages ||
                         mbar_test_wait(smem_u32(&k_empty[nk % kFwdKStages]),
                                        ((nk / kFwdKStages) & 1) ^ 1))) {
          const int st = nk % kFwdKStages;
          mbar_arrive_expect_tx(&k_full[st], kTileBytes);
          tma_load_3d_hint(&p.tm_k, &k_full[st], sK + st * kTileBytes, 0, g,
                           sp.k0 + (lo + nk) * kBlockN, keep);
          ++nk;
          progress = true;
        }
        // V(nv): its stage was last read by PV(nv - 2); V never runs ahead of K
        if (nv < nk && (nv < kFwdVStages ||
                        mbar_test_wait(smem_u32(&v_empty[nv % kFwdVStages]),
                                       ((nv / kFwdVStages) & 1) ^ 1))) {
          const int st = nv % kFwdVStages;
          mbar_arrive_expect_tx(&v_full[st], kTileBytes);
          tma_load_3d_hint(&p.tm_v, &v_full[st], sV + st * kTileBytes, 0, g,
                           sp.k0 + (lo + nv) * kBlockN, keep);
          ++nv;
          progress = true;
        }
        if (progress) {
          t_last = global_timer_ns();
        } else if (abort_flag || global_timer_ns() - t_last > kWaitLimitNs) {
          ok = false;
          break;
        } else {
          __nanosleep(32);
        }
      }
      if (!ok) {
        abort_flag = 1;
        atomicCAS(p.err, 0, DEVERR_TIMEOUT_FWD + 1);
        // Let the copies already in flight land before the CTA releases SMEM.
        mbar_wait(&q_full, 0, nullptr);
        for (int it = max(0, nk - kFwdKStages); it < nk; ++it)
          mbar_wait(&k_full[it % kFwdKStages], (it / kFwdKStages) & 1, nullptr);
        for (int it = max(0, nv - kFwdVStages); it < nv; ++it)
          mbar_wait(&v_full[it % kFwdVStages], (it / kFwdVStages) & 1, nullptr);
      }
    }
  } else if (warp == kFwdMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    // Per key tile n: S(n) = Q K_n^T (M=N=128, bf16) into the S columns; the
    // softmax writes P(n) (fp16, 128 keys in 64 columns) into the P columns and
    // O += P(n) V_n (M=128, N=64, K=128, A from TMEM) accumulates in the O
    // columns.  S(n+1) is issued as soon as the softmax warps have read S(n)
    // (s_free), before PV(n): the tensor cores compute the next scores while
    // the current tile's exponentials run.
    if (lane == 0) {
      const uint32_t idesc_s = make_idesc_bf16(kBlockM, kBlockN, false, false);
      const uint32_t idesc_o = make_idesc(kFmtF16, kBlockM, kHeadDim, false, true);
      // Shared-memory descriptors, built once; an operand at byte offset o from a
      // base is the base's descriptor plus o / 16 (the start-address field).
      const uint64_t dQ = make_sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dK0 = make_sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV0 = make_sdesc_sw128(smem_u32(sV), 16384, 1024);   // MN-major
      constexpr uint32_t kTileU = kTileBytes >> 4;
      auto issue_s = [&](int n) -> bool {
        const int st = n % kFwdKStages;
        if (!mbar_wait(&k_full[st], (n / kFwdKStages) & 1, &abort_flag)) return false;
        tc_fence_after();
        #pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k)
          mma_ss(tmem + kFwdColS, dQ + 2 * k, dK0 + st * kTileU + 2 * k, idesc_s, k > 0);
        mma_commit(&s_full);
        mma_commit(&k_empty[st]);
        return true;
      };
      bool ok = mbar_wait(&q_full, 0, &abort_flag) && issue_s(0);
      for (int n = 0; ok && n < num; ++n) {
        // S(n+1) once S(n) has been read out of TMEM
        if (n + 1 < num) {
          if (!mbar_wait(&s_free, n & 1, &abort_flag) || !issue_s(n + 1)) { ok = false; break; }
        }
        // PV(n) once P(n) is in TMEM (and O rescaled) and V(n) has landed
        const int sv = n % kFwdVStages;
        if (!mbar_wait(&v_full[sv], (n / kFwdVStages) & 1, &abort_flag) ||
            !mbar_wait(&p_full, n & 1, &abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        #pragma unroll
        for (int k = 0; k < kBlockN / 16; ++k)
          mma_ts(tmem + kFwdColO, tmem + kFwdColP + 8 * k, dV0 + sv * kTileU + 128 * k, idesc_o,
                 (n > 0 || k > 0));
        mma_commit(&pv_done);
        mma_commit(&v_empty[sv]);
      }
      if (!ok) {
        abort_flag = 1;
        atomicCAS(p.err, 0, DEVERR_TIMEOUT_FWD + 2);
      }
      // Drain: every MMA issued above has finished before TMEM is released.
      mma_commit(&mma_drained);
      mbar_wait(&mma_drained, 0, nullptr);
    }
  } else {
    // ---------------------------------------------------------------- softmax warps
    // Key half c = warp / 4: S columns [64c, 64c+64).  Thread = row = TMEM lane.
    // The two halves of a row share one running max (exchanged through SMEM once
    // per tile) and one O; each half keeps its own part of the row sum.
    const int c = warp >> 2;
    const int r = tid & 127;
    const int i = i0 + r;                    // row within the sequence
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + kFwdColS + 64 * c + lane_base;
    const uint32_t tP = tmem + kFwdColP + 32 * c + lane_base;  // P of keys [64c, 64c+64)
    const uint32_t tO = tmem + kFwdColO + 32 * c + lane_base;  // O columns [32c, 32c+32)
    const bool sink_finite = sink_h > -INFINITY;
    // running max (log2 domain) starts at the sink logit; the sink's term of the
    // sum (1 at m = sink log2 e) is counted in half 0 only
    float m = sink_finite ? sink_h * kLog2e : -INFINITY;
    float l = (sink_finite && c == 0) ? 1.0f : 0.0f;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2(sl2, sl2);
    const int jmax = p.causal ? min(sp.nk - 1, i + off) : sp.nk - 1;   // inclusive
    const int jmin = (p.causal && p.window > 0) ? i + off - p.window + 1 : 0;
    bool ok = true;
    for (int it = 0; it < num; ++it) {
      // S(it) -> registers; S columns are then free for S(it + 1)
      uint32_t a[64];
      bool got = mbar_wait_warp(&s_full, it & 1, &abort_flag);
      float mx_half = -INFINITY;
      if (got) {
        tc_fence_after();
        tmem_ld_x32(tS, a);
        tmem_ld_x32(tS + 32, a + 32);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&s_free);
        const int j0 = (lo + it) * kBlockN + 64 * c;            // first key of this half
        const bool need_mask = (j0 + 64 > sp.nk) ||
                               (p.causal && (j0 + 63 > i0 + off ||
                                             (p.window > 0 && j0 <= tile_r1 + off - p.window)));
        if (need_mask) {
          #pragma unroll
          for (int e = 0; e < 64; ++e) {
            const int j = j0 + e;
            if (j > jmax || j < jmin) a[e] = __float_as_uint(-INFINITY);
          }
        }
        // row max over the 64 columns: four independent 3-input max chains
        float q0 = __uint_as_float(a[0]), q1 = __uint_as_float(a[1]);
        float q2 = __uint_as_float(a[2]), q3 = __uint_as_float(a[3]);
        #pragma unroll
        for (int e = 4; e < 64; e += 8) {
          q0 = fmax3(q0, __uint_as_float(a[e]), __uint_as_float(a[e + 1]));
          q1 = fmax3(q1, __uint_as_float(a[e + 2]), __uint_as_float(a[e + 3]));
          q2 = fmax3(q2, __uint_as_float(a[e + 4]), __uint_as_float(a[e + 5]));
          q3 = fmax3(q3, __uint_as_float(a[e + 6]), __uint_as_float(a[e + 7]));
        }
        mx_half = fmaxf(fmax3(q0, q1, q2), q3);
        s_mx[it & 1][c][r] = mx_half;
      }
      // The two warps that hold the halves of the same 32 rows (w and w + 4) meet
      // here once per tile, and leave together if either's wait failed.  The
      // exchange buffer alternates between tiles.
      if (!named_barrier_and(2 + (warp & 3), 64, got && ok)) {
        ok = false;
        abort_flag = 1;   // the other warp pairs stop at their next wait
        break;
      }
      const float mx = fmaxf(mx_half, s_mx[it & 1][c ^ 1][r]) * sl2;
      // Lazy rescale: the max only moves when it grows by more than the threshold.
      float alpha = 1.0f;
      if (mx > m + kRescaleThreshold || (m == -INFINITY && mx > -INFINITY)) {
        alpha = ex2_approx(m - mx);
        m = mx;
      }
      // P = exp2(S * scale * log2 e - m), fp16; row sum on pairs of columns
      const float m_use = (m == -INFINITY) ? 0.0f : m;
      const uint64_t negm2 = f2(-m_use, -m_use);
      uint64_t rs = f2(0.0f, 0.0f);
      uint32_t pk[16];
      #pragma unroll
      for (int e = 0; e < 32; e += 2) {
        const uint64_t x =
            ffma2(f2(__uint_as_float(a[e]), __uint_as_float(a[e + 1])), sl2x2, negm2);
        const float e0 = ex2_approx(f2_lo(x));
        const float e1 = ex2_approx(f2_hi(x));
        rs = fadd2(rs, f2(e0, e1));
        pk[e >> 1] = pack_f16x2(e0, e1);
      }
      // PV(it - 1) has read the P columns and updated O
      if (it > 0 && !mbar_wait_warp(&pv_done, (it - 1) & 1, &abort_flag)) ok = false;
      if (ok) {
        tc_fence_after();
        tmem_st_x16(tP, pk);
        #pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const uint64_t x =
              ffma2(f2(__uint_as_float(a[32 + e]), __uint_as_float(a[33 + e])), sl2x2, negm2);
          const float e0 = ex2_approx(f2_lo(x));
          const float e1 = ex2_approx(f2_hi(x));
          rs = fadd2(rs, f2(e0, e1));
          pk[e >> 1] = pack_f16x2(e0, e1);
        }
        tmem_st_x16(tP + 16, pk);
        l = l * alpha + (f2_lo(rs) + f2_hi(rs));
        // O columns [32c, 32c+32) of this row move with the max
        if (it > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
          #pragma unroll
          for (int q = 0; q < 32; q += 16) {
            uint32_t o[16];
            tmem_ld_x16(tO + q, o);
            tmem_ld_wait();
            #pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st_x16(tO + q, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full);
      } else {
        abort_flag = 1;
      }
    }
    // The last PV has landed in O.
    bool fin = ok && mbar_wait_warp(&pv_done, (num - 1) & 1, &abort_flag);
    s_red_l[c][r] = l;
    fin = named_barrier_and(1, 2 * kBlockM, fin);
    if (!fin) {
      abort_flag = 1;
      atomicCAS(p.err, 0, DEVERR_TIMEOUT_FWD + 3);
    } else {
      tc_fence_after();
      const float lt = s_red_l[0][r] + s_red_l[1][r];
      const float inv_l = (lt > 0.0f) ? 1.0f / lt : 0.0f;
      const bool valid = i < sp.nq;
      const size_t row = (size_t)(sp.q0 + i);
      // this half writes output columns [32c, 32c + 32); the load runs with the
      // whole warp (rows past the tail included), only the stores are guarded
      uint32_t o[32];
      tmem_ld_x32(tO, o);
      tmem_ld_wait();
      // A whole tile goes out through two 128B-swizzled SMEM tiles (the K ring,
      // idle now: every copy into it has been consumed) and TMA stores, which
      // run on while the CTA ends; a tile past its sequence's end stores its
      // valid rows directly.
      const bool whole = i0 + kBlockM <= sp.nq;             // same for every row
      if (whole || valid) {
        const size_t base = (row * p.heads_q + h) * kHeadDim + 32 * c;
        #pragma unroll
        for (int u = 0; u < 4; ++u) {
          float f[8];
          uint32_t hi[4], lo2[4];
          #pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(o[8 * u + e]) * inv_l;
          #pragma unroll
          for (int e = 0; e < 4; ++e) {
            hi[e] = pack_bf16x2(f[2 * e], f[2 * e + 1]);
            lo2[e] = pack_bf16x2(f[2 * e] - bf16_lo(hi[e]), f[2 * e + 1] - bf16_hi(hi[e]));
          }
          if (whole) {
            const uint32_t off = sw128_offset((uint32_t)r, (uint32_t)(4 * c + u));
            st_shared_v4(smem_u32(sK) + off, hi[0], hi[1], hi[2], hi[3]);
            if (p.out_lo)
              st_shared_v4(smem_u32(sK) + kTileBytes + off, lo2[0], lo2[1], lo2[2], lo2[3]);
          } else {
            reinterpret_cast<uint4*>(p.out + base)[u] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            if (p.out_lo)
              reinterpret_cast<uint4*>(p.out_lo + base)[u] =
                  make_uint4(lo2[0], lo2[1], lo2[2], lo2[3]);
          }
        }
        if (c == 0 && valid)
          p.lse[(size_t)h * p.total_q + row] = (lt > 0.0f) ? (m + __log2f(lt)) * kLn2 : -INFINITY;
      }
      if (whole) {
        fence_proxy_async_smem();
        named_barrier_sync(1, 2 * kBlockM);
        if (warp == 0 && lane == 0) {
          const uint64_t once = l2_policy_evict_first();
          tma_store_3d_hint(&p.tm_out, sK, 0, h, sp.q0 + i0, once);
          if (p.out_lo) tma_store_3d_hint(&p.tm_out_lo, sK + kTileBytes, 0, h, sp.q0 + i0, once);
          bulk_commit_group();
          bulk_wait_group_read0();   // the tiles are read before the CTA releases SMEM
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kFwdMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kFwdTmemCols);
  }
}

}  // namespace attn_sink
