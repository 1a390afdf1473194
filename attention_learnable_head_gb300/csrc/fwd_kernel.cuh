// Forward kernel: attention with a per-head sink, sm_103a (tcgen05 + TMA).
//
// One CTA per (query head h, sequence, 256-row query block).  The block is two
// 128-row tiles, A and B, that share every K/V tile and run in ping-pong: while
// one softmax warpgroup turns its S tile into P, the tensor cores run the other
// tile's MMAs.  Per tile and key tile:
//   S = Q K^T (tcgen05, fp32 accumulators in TMEM),
//   online softmax whose running max and sum start from the sink logit
//   (m0 = sink[h] * log2 e, l0 = 1 in the exp2 domain),
//   P (fp16) written to TMEM and consumed there by O += P V (tcgen05, A from
//   TMEM, V converted to fp16 in SMEM by a converter warp),
// then out = O / l (bf16, plus optionally the bf16 residual O/l - out) and
// lse = ln 2 * (m + log2 l), which includes the sink.  S = Q K^T multiplies the
// bf16 inputs exactly; P and V go to the tensor cores as fp16 (11-bit
// significand) so that O, and the backward's D = rowsum(dO o O), keep ~3 more
// bits than a bf16 P would give.
// The sink joins the softmax denominator only: it is the extra column of the
// concat listing "带汇聚的注意力（GPT-OSS）" on the euno.news page, and the
// P_ij / P_ih equations of its section "数学公式".
//
// Rescaling of O is lazy: the running max used for the exponentials only moves
// when a row's max grows by more than kRescaleThreshold (log2 units); P stays
// below 2^threshold, and out/lse are exact because l and O use the same max.
//
// Warp roles (576 threads):
//   warps 0-7   softmax + epilogue of tile A: warps 0-3 take S columns 0-63,
//               warps 4-7 columns 64-127 (thread t owns row t = TMEM lane t)
//   warps 8-15  the same for tile B
//   warp 16     TMA producer: Q_A, Q_B once, then K/V tiles through a ring
//   warp 17     MMA issuer (one lane) and TMEM owner
// TMEM columns: S_A 0, S_B 128 (128 fp32 each; P_x, 128 fp16 two per column, is
// written over the first 64 columns of S_x once S_x has been read), O_A 256,
// O_B 320 (64 fp32 each), Q_A 384, Q_B 416 (64 bf16 two per column: the A
// operand of S = Q K^T, so only K is read from shared memory).
// P_x overwrites S_x safely: PV_x(n) is issued before S_x(n+1) by the same
// thread, and tcgen05 MMAs from one thread execute in issue order.
// v is read as an fp16 copy (converted into the workspace before the launch).
#pragma once
#include <cuda_bf16.h>
#include "sm103_ptx.cuh"

namespace attn_sink {

constexpr int kBlockM = 128;   // query rows per tile
constexpr int kBlockN = 128;   // keys per tile
constexpr int kHeadDim = 64;
constexpr int kFwdTiles = 2;   // query tiles per CTA
constexpr int kFwdStages = 4;
constexpr int kFwdThreads = 576;    // 16 softmax warps, TMA warp, MMA warp
constexpr int kFwdTmaWarp = 16;
constexpr int kFwdMmaWarp = 17;
constexpr int kFwdRowsPerCta = kFwdTiles * kBlockM;
constexpr uint32_t kTileBytes = kBlockM * kHeadDim * 2;   // 16 KB bf16 tile
constexpr uint32_t kPTileBytes = kBlockM * kBlockN * 2;   // 32 KB bf16 tile (bwd dS)
constexpr int kFwdSmemBytes = 1024 + (int)kTileBytes * (kFwdTiles + 2 * kFwdStages);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;
constexpr uint32_t kColQ = 384;      // Q_x at kColQ + 32 x

struct FwdParams {
  CUtensorMap tm_q;   // [T_q][H_q][64] bf16, box 64 x 1 x 128, 128B swizzle
  CUtensorMap tm_k;   // [T_k][H_kv][64]
  CUtensorMap tm_v;
  const int* cu_q;    // null for a dense batch
  const int* cu_k;
  const float* sink;  // [H_q]
  __nv_bfloat16* out; // [T_q][H_q][64]
  __nv_bfloat16* out_lo; // [T_q][H_q][64] residual O/l - out, or null
  float* lse;         // [H_q][T_q]
  int* err;           // device error word
  int seqlen_q, seqlen_k;
  int total_q;
  int heads_q, group;
  int causal, window;
  float scale_log2;   // softmax_scale * log2(e)
  int n_qblocks;      // 256-row query blocks of the longest sequence
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

__device__ __forceinline__ KeyRange key_tiles(int r0, int r1, const SeqSpan& sp, int causal,
                                              int window) {
  KeyRange kr{0, 0};
  if (r1 < r0) return kr;
  const int off = sp.nk - sp.nq;
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

// Registers are split per SM sub-partition (16384 each); with 18 warps one of the
// four hosts 5 warps, so a thread may use at most 102: 96 is used.
__global__ void __maxnreg__(96)
attn_sink_fwd_kernel(const __grid_constant__ FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t q_full, mma_drained;
  __shared__ __align__(8) uint64_t k_full[kFwdStages], v_full[kFwdStages], kv_empty[kFwdStages];
  __shared__ __align__(8) uint64_t q_tmem;
  __shared__ __align__(8) uint64_t s_full[kFwdTiles], p_full[kFwdTiles], pv_done[kFwdTiles];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;
  __shared__ float s_red_max[kFwdTiles][2][2][kBlockM];   // [tile][iteration parity][half][row]
  __shared__ float s_red_l[kFwdTiles][2][kBlockM];        // [tile][half][row]

  const int h = blockIdx.x;
  const int seq = blockIdx.y;
  const int qblock = p.n_qblocks - 1 - (int)blockIdx.z;   // longest work first
  const SeqSpan sp = seq_span(p.cu_q, p.cu_k, seq, p.seqlen_q, p.seqlen_k);
  const int i0 = qblock * (kFwdTiles * kBlockM);
  if (i0 >= sp.nq) return;                                // uniform per CTA
  const int g = h / p.group;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const bool has_b = i0 + kBlockM < sp.nq;
  const KeyRange kr_a = key_tiles(i0, min(i0 + kBlockM, sp.nq) - 1, sp, p.causal, p.window);
  const KeyRange kr_b = has_b ? key_tiles(i0 + kBlockM, min(i0 + 2 * kBlockM, sp.nq) - 1, sp,
                                          p.causal, p.window)
                              : KeyRange{0, 0};
  // union of the two tiles' key ranges
  int lo, hi;
  if (kr_a.num > 0 && kr_b.num > 0) {
    lo = min(kr_a.lo, kr_b.lo);
    hi = max(kr_a.lo + kr_a.num, kr_b.lo + kr_b.num);
  } else if (kr_a.num > 0) {
    lo = kr_a.lo; hi = kr_a.lo + kr_a.num;
  } else {
    lo = kr_b.lo; hi = kr_b.lo + kr_b.num;
  }
  const int num = (kr_a.num > 0 || kr_b.num > 0) ? hi - lo : 0;
  const float sink_h = __ldg(p.sink + h);

  if (num == 0) {
    // No row of this block sees a key: out = 0, lse = sink (the sink alone).
    for (int t = tid; t < kFwdTiles * kBlockM; t += kFwdThreads) {
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
  uint8_t* sQ = smem;                                   // kFwdTiles tiles
  uint8_t* sK = sQ + kFwdTiles * kTileBytes;
  uint8_t* sV = sK + kFwdStages * kTileBytes;

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&q_full, 1);
    mbar_init(&mma_drained, 1);
    for (int s = 0; s < kFwdStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(&q_tmem, 2 * kFwdTiles * kBlockM);
    for (int x = 0; x < kFwdTiles; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 2 * kBlockM);
      mbar_init(&pv_done[x], 1);
    }
    fence_mbarrier_init();
  }
  if (warp == kFwdMmaWarp) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == kFwdTmaWarp) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      const uint64_t keep = l2_policy_evict_last();
      mbar_arrive_expect_tx(&q_full, (has_b ? 2 : 1) * kTileBytes);
      tma_load_3d(&p.tm_q, &q_full, sQ, 0, h, sp.q0 + i0);
      if (has_b) tma_load_3d(&p.tm_q, &q_full, sQ + kTileBytes, 0, h, sp.q0 + i0 + kBlockM);
      int issued = 0;
      for (int it = 0; it < num; ++it) {
        const int st = it % kFwdStages;
        if (it >= kFwdStages &&
            !mbar_wait(&kv_empty[st], ((it / kFwdStages) & 1) ^ 1, &abort_flag)) {
          abort_flag = 1;
          atomicCAS(p.err, 0, DEVERR_TIMEOUT_FWD + 1);
          break;
        }
        const int row = sp.k0 + (lo + it) * kBlockN;
        mbar_arrive_expect_tx(&k_full[st], kTileBytes);
        tma_load_3d_hint(&p.tm_k, &k_full[st], sK + st * kTileBytes, 0, g, row, keep);
        mbar_arrive_expect_tx(&v_full[st], kTileBytes);
        tma_load_3d_hint(&p.tm_v, &v_full[st], sV + st * kTileBytes, 0, g, row, keep);
        issued = it + 1;
      }
      if (abort_flag) {
        // Let the copies already in flight land before the CTA releases SMEM.
        mbar_wait(&q_full, 0, nullptr);
        for (int it = max(0, issued - kFwdStages); it < issued; ++it) {
          const int st = it % kFwdStages;
          mbar_wait(&k_full[st], (it / kFwdStages) & 1, nullptr);
          mbar_wait(&v_full[st], (it / kFwdStages) & 1, nullptr);
        }
      }
    }
  } else if (warp == kFwdMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = make_idesc_bf16(kBlockM, kBlockN, false, false);
      const uint32_t idesc_o = make_idesc(kFmtF16, kBlockM, kHeadDim, false, true);
      const KeyRange kr[kFwdTiles] = {kr_a, kr_b};
      // Q_A / Q_B are in TMEM once both softmax warpgroups have copied them there.
      bool ok = mbar_wait(&q_tmem, 0, &abort_flag);
      // Shared-memory descriptors, built once; an operand at byte offset o from a
      // base is the base's descriptor plus o / 16 (the start-address field).
      const uint64_t dK0 = make_sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV0 = make_sdesc_sw128(smem_u32(sV), 16384, 1024);   // MN-major
      constexpr uint32_t kTileU = kTileBytes >> 4;
      // S_x(n) = Q_x K_n^T into S_x; n is a union index.
      auto issue_s = [&](int x, int n) -> bool {
        const int st = n % kFwdStages;
        if (!mbar_wait(&k_full[st], (n / kFwdStages) & 1, &abort_flag)) return false;
        tc_fence_after();
        #pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k)
          mma_ts(tmem + x * 128, tmem + kColQ + 32 * x + 8 * k, dK0 + st * kTileU + 2 * k,
                 idesc_s, k > 0);
        mma_commit(&s_full[x]);
        return true;
      };
      auto in_range = [&](int x, int n) {
        const int a = lo + n;
        return kr[x].num > 0 && a >= kr[x].lo && a < kr[x].lo + kr[x].num;
      };
      // Stagger the tiles: S_B(first) is issued once tile A's first P is ready,
      // so B's softmax overlaps A's MMAs instead of competing with A's for MUFU.
      bool b_started = kr[1].num == 0;
      if (kr[0].num > 0) {
        ok = issue_s(0, kr[0].lo - lo);
      } else {
        ok = issue_s(1, kr[1].lo - lo);
        b_started = true;
      }
      for (int n = 0; ok && n < num; ++n) {
        const int st = n % kFwdStages;
        #pragma unroll
        for (int x = 0; x < kFwdTiles; ++x) {
          if (!ok || !in_range(x, n)) continue;
          const int local = lo + n - kr[x].lo;
          if (!mbar_wait(&p_full[x], local & 1, &abort_flag) ||
              !mbar_wait(&v_full[st], (n / kFwdStages) & 1, &abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tP = tmem + x * 128;       // P_x over the first half of S_x
          const uint32_t tO = tmem + 256 + x * 64;
          #pragma unroll
          for (int k = 0; k < kBlockN / 16; ++k)
            mma_ts(tO, tP + 8 * k, dV0 + st * kTileU + 128 * k, idesc_o, (local > 0 || k > 0));
          mma_commit(&pv_done[x]);
          if (!b_started) {
            ok = issue_s(1, kr[1].lo - lo);
            b_started = true;
          }
          if (ok && in_range(x, n + 1)) ok = issue_s(x, n + 1);
        }
        if (ok) mma_commit(&kv_empty[st]);
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
    // Tile x = warp / 8.  Half c = (warp / 4) & 1 owns S columns [64c, 64c + 64),
    // P columns [32c, 32c + 32) and O columns [32c, 32c + 32) of the tile's rows
    // (thread = row = TMEM lane).  The two halves of a tile exchange row maxima
    // and sums through shared memory behind the tile's named barrier; every exit
    // decision is taken at that barrier, so both halves always reach the same
    // barriers.
    const int x = warp >> 3;
    const int c = (warp >> 2) & 1;
    const int r = tid & 127;
    const int i = i0 + x * kBlockM + r;      // row within the sequence
    const KeyRange kx = x == 0 ? kr_a : kr_b;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + x * 128 + 64 * c + lane_base;
    const uint32_t tO = tmem + 256 + x * 64 + 32 * c + lane_base;
    const uint32_t tP = tmem + x * 128 + 32 * c + lane_base;   // P over S columns 0..63
    const uint32_t bar_id = 1 + x;
    const int off = sp.nk - sp.nq;
    const int tile_r0 = i0 + x * kBlockM;
    const int tile_r1 = min(tile_r0 + kBlockM, sp.nq) - 1;
    const bool sink_finite = sink_h > -INFINITY;
    float m = sink_finite ? sink_h * kLog2e : -INFINITY;   // running max, log2 domain
    // running sum of this half's columns; the sink's term (1) is counted in half 0
    float l = (sink_finite && c == 0) ? 1.0f : 0.0f;
    const float sl2 = p.scale_log2;
    const int jmax = p.causal ? min(sp.nk - 1, i + off) : sp.nk - 1;   // inclusive
    const int jmin = (p.causal && p.window > 0) ? i + off - p.window + 1 : 0;
    // Q_x row r into TMEM (the A operand of S = Q K^T), by half 0: the swizzled
    // SMEM row holds 8 chunks of 8 bf16, i.e. the 32 packed columns in order.
    bool ok = mbar_wait_warp(&q_full, 0, &abort_flag);
    if (ok && c == 0) {
      uint32_t qw[32];
      const uint32_t qrow = smem_u32(sQ + x * kTileBytes);
      #pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        uint4 w;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                     : "r"(qrow + sw128_offset(r, cc)));
        qw[4 * cc] = w.x; qw[4 * cc + 1] = w.y; qw[4 * cc + 2] = w.z; qw[4 * cc + 3] = w.w;
      }
      tmem_st_x32(tmem + kColQ + 32 * x + lane_base, qw);
      tmem_st_wait();
    }
    tc_fence_before();
    mbar_arrive(&q_tmem);
    for (int it = 0; it < kx.num; ++it) {
      const bool got_s = ok && mbar_wait_warp(&s_full[x], it & 1, &abort_flag);
      const int j0 = (kx.lo + it) * kBlockN + 64 * c;          // first key of this half
      uint32_t a[64];
      float pmax = -INFINITY;
      if (got_s) {
        tc_fence_after();
        tmem_ld_x32(tS, a);
        tmem_ld_x32(tS + 32, a + 32);
        tmem_ld_wait();
        const bool need_mask = (j0 + 64 > sp.nk) ||
                               (p.causal && (j0 + 63 > tile_r0 + off ||
                                             (p.window > 0 && j0 <= tile_r1 + off - p.window)));
        if (need_mask) {
          #pragma unroll
          for (int e = 0; e < 64; ++e) {
            const int j = j0 + e;
            if (j > jmax || j < jmin) a[e] = __float_as_uint(-INFINITY);
          }
        }
        #pragma unroll
        for (int e = 0; e < 64; e += 2)
          pmax = fmax3(pmax, __uint_as_float(a[e]), __uint_as_float(a[e + 1]));
      }
      s_red_max[x][it & 1][c][r] = pmax;
      // S columns of both halves are in registers before either half writes P
      // over S columns 0..63.
      tc_fence_before();
      if (!named_barrier_and(bar_id, 2 * kBlockM, got_s)) { ok = false; break; }
      tc_fence_after();
      const float mx = fmaxf(pmax, s_red_max[x][it & 1][c ^ 1][r]) * sl2;
      // Lazy rescale: move the max only when it grows by more than the threshold
      // (both halves take the same decision from the same values).
      float alpha = 1.0f;
      if (mx > m + kRescaleThreshold || (m == -INFINITY && mx > -INFINITY)) {
        alpha = ex2_approx(m - mx);
        m = mx;
      }
      // PV of the previous key tile has finished: O may be rescaled, P_x reused.
      // A failed wait is carried to the next barrier (never a one-sided exit).
      if (it > 0) {
        if (!mbar_wait_warp(&pv_done[x], (it - 1) & 1, &abort_flag)) {
          ok = false;
        } else {
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha != 1.0f)) {
            #pragma unroll
            for (int q0 = 0; q0 < 32; q0 += 16) {
              uint32_t o[16];
              tmem_ld_x16(tO + q0, o);
              tmem_ld_wait();
              #pragma unroll
              for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st_x16(tO + q0, o);
            }
          }
        }
      }
      // P = exp2(S * scale * log2 e - m), fp16, into this half's P columns.
      const float m_use = (m == -INFINITY) ? 0.0f : m;
      float rowsum = 0.0f;
      #pragma unroll
      for (int cc = 0; cc < 64; cc += 32) {
        uint32_t pk[16];
        #pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float e0 = ex2_approx(fmaf(__uint_as_float(a[cc + e]), sl2, -m_use));
          const float e1 = ex2_approx(fmaf(__uint_as_float(a[cc + e + 1]), sl2, -m_use));
          rowsum += e0 + e1;
          pk[e >> 1] = pack_f16x2(e0, e1);
        }
        tmem_st_x16(tP + (cc >> 1), pk);
      }
      l = l * alpha + rowsum;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[x]);
    }
    // the last PV has landed in O
    bool fin = ok;
    if (fin && kx.num > 0) fin = mbar_wait_warp(&pv_done[x], (kx.num - 1) & 1, &abort_flag);
    s_red_l[x][c][r] = l;
    fin = named_barrier_and(bar_id, 2 * kBlockM, fin);
    if (!fin) {
      abort_flag = 1;
      atomicCAS(p.err, 0, DEVERR_TIMEOUT_FWD + 3);
    } else {
      tc_fence_after();
      const float lt = l + s_red_l[x][c ^ 1][r];
      const float inv_l = (lt > 0.0f) ? 1.0f / lt : 0.0f;
      const bool valid = i < sp.nq;
      const size_t row = (size_t)(sp.q0 + i);
      uint32_t o[32];
      if (kx.num > 0) {
        tmem_ld_x32(tO, o);
        tmem_ld_wait();
      } else {
        #pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
      if (valid) {
        const size_t base = (row * p.heads_q + h) * kHeadDim + 32 * c;
        uint4* dst = reinterpret_cast<uint4*>(p.out + base);
        uint4* dlo = p.out_lo ? reinterpret_cast<uint4*>(p.out_lo + base) : nullptr;
        #pragma unroll
        for (int u = 0; u < 4; ++u) {
          float f[8];
          uint32_t hi[4], lo[4];
          #pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(o[8 * u + e]) * inv_l;
          #pragma unroll
          for (int e = 0; e < 4; ++e) {
            hi[e] = pack_bf16x2(f[2 * e], f[2 * e + 1]);
            lo[e] = pack_bf16x2(f[2 * e] - bf16_lo(hi[e]), f[2 * e + 1] - bf16_hi(hi[e]));
          }
          dst[u] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          if (dlo) dlo[u] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        if (c == 0)
          p.lse[(size_t)h * p.total_q + row] = (lt > 0.0f) ? (m + __log2f(lt)) * kLn2 : -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kFwdMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace attn_sink
