// Deterministic dQ of attention with a per-head sink, sm_103a (tcgen05 + TMA).
//
// The main backward adds each key tile's dQ contribution into one fp32
// accumulator in whatever order the hardware completes the reduce-adds, so dQ
// is not bitwise reproducible.  This kernel computes dQ query-stationary
// instead, with a fixed summation order over the keys:
//   S  = Q K^T,  P = exp2(S * scale * log2 e - lse * log2 e)   (lse includes the sink)
//   dP = dO V^T, dS = P o (dP - D)
//   dQ = scale * sum_j dS_j K_j          (key steps in increasing order)
// (the explicit backward of the concat-sink softmax; the sink adds no key row,
// so it enters dQ only through lse and D).  It costs two more products than
// the fused backward (S and dP are computed again): the price of
// reproducibility.
//
// One CTA per (query head h, sequence, 128-row query tile), longest first,
// two CTAs per SM, stepping over the visible keys 64 at a time.  Warps 0-7
// (thread = query row = TMEM lane; warps 4c..4c+3 take the key half c, columns
// [32c, 32c+32) of a step) read S, signal that it has been read
// (s_read), form P, then read dP and write dS (fp16) over the dP columns they
// have read; warp 8 issues TMA (Q, dO once; K/V through a ring); warp 9 issues
// the MMAs: S and dP of the next step (M=128, N=64, fp16 from SMEM; dP into
// the other of two buffers) as soon as this step's S has been read, and
// dQ += dS K (M=128, N=64, K=64: dS from TMEM, K read MN-major) once dS is
// written.  So the next step's S and dP are computed while this step's P and
// dS are formed, and the second CTA of the SM fills the remaining gaps.
// TMEM (256 columns): S 0-63, dP of even steps 64-127, dQ 128-191, dP of odd
// steps 192-255.
#pragma once
#include <cuda_bf16.h>
#include "fwd_kernel.cuh"

namespace attn_sink {

constexpr int kDqThreads = 320;
constexpr int kDqTmaWarp = 8;
constexpr int kDqMmaWarp = 9;
constexpr int kDqKeys = 64;                                   // keys per step
constexpr uint32_t kDqKvBytes = kDqKeys * kHeadDim * 2;       // 8 KB K or V tile
constexpr int kDqStages = 4;
// Q, dO, kDqStages x (K, V): ~99 KB, two CTAs per SM
constexpr int kDqSmemBytes = 1024 + 2 * (int)kTileBytes + kDqStages * 2 * (int)kDqKvBytes;
constexpr uint32_t kDqTmemCols = 256;
constexpr uint32_t kDqColS = 0, kDqColDP = 64, kDqColDQ = 128, kDqColDP1 = 192;
// dP (and, once formed, dS) of key step n
__host__ __device__ constexpr uint32_t dq_col_dp(int n) { return (n & 1) ? kDqColDP1 : kDqColDP; }

struct DqParams {
  CUtensorMap tm_q;    // [T_q][H_q][64] fp16 copy of q
  CUtensorMap tm_do;   // [T_q][H_q][64] fp16 copy of dout
  CUtensorMap tm_k;    // [T_k][H_kv][64] fp16 copy of k
  CUtensorMap tm_v;    // fp16 copy of v
  const int* cu_q;
  const int* cu_k;
  const float2* LD;    // [H_q][T_q]: (-lse * log2 e, D)
  void* dq;            // [T_q][H_q][64] bf16 (grad_fp32 = 0) or fp32
  int* err;
  int seqlen_q, seqlen_k;
  int total_q;
  int heads_q, group;
  int causal, window;
  float scale;         // softmax_scale
  float scale_log2;    // softmax_scale * log2(e)
  int n_qtiles;        // 128-row query tiles of the longest sequence
  int grad_fp32;
};

// P of 32 keys of one query row (thread = row), in place over S (fp32):
//   P = exp2(S * scale * log2 e - lse * log2 e)   (lse includes the sink)
// with kMask, keys outside [jmin, jmax] exactly 0.
template <bool kMask>
__device__ __forceinline__ void dq_p_chunk(uint32_t* sr, uint64_t sl2x2, uint64_t nlse2x2,
                                           int j_first, int jmin, int jmax) {
  #pragma unroll
  for (int e = 0; e < 32; e += 2) {
    const uint64_t x =
        ffma2(f2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sl2x2, nlse2x2);
    float p0 = ex2_approx(f2_lo(x));
    float p1 = ex2_approx(f2_hi(x));
    if (kMask) {
      const int j = j_first + e;
      if (j < jmin || j > jmax) p0 = 0.0f;
      if (j + 1 < jmin || j + 1 > jmax) p1 = 0.0f;
    }
    sr[e] = __float_as_uint(p0);
    sr[e + 1] = __float_as_uint(p1);
  }
}

// dS = P o (dP - D) of 32 keys of one query row, fp16-packed.
__device__ __forceinline__ void dq_ds_chunk(const uint32_t* pr, const uint32_t* dr, uint64_t d2,
                                            uint32_t* dk) {
  #pragma unroll
  for (int e = 0; e < 32; e += 2) {
    const uint64_t ds =
        fmul2(f2(__uint_as_float(pr[e]), __uint_as_float(pr[e + 1])),
              fsub2(f2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])), d2));
    dk[e >> 1] = pack_f16x2(f2_lo(ds), f2_hi(ds));
  }
}

__global__ void __launch_bounds__(kDqThreads, 2)
attn_sink_bwd_dq_kernel(const __grid_constant__ DqParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t q_full, s_full, s_read, dq_done;
  // Step n completes dp_full[n & 1] (its dP) and p_full[n & 1] (its dS): dP(n+1)
  // is issued before the compute warps wait for dP(n), and they may finish
  // step n+1 before the MMA thread waits for dS(n), so a single barrier could
  // run two phases ahead of its waiter
  __shared__ __align__(8) uint64_t dp_full[2], p_full[2];
  __shared__ __align__(8) uint64_t kv_full[kDqStages], kv_empty[kDqStages];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;

  const int h = blockIdx.x;
  const int seq = blockIdx.y;
  const int qt = p.n_qtiles - 1 - (int)blockIdx.z;        // longest work first
  const SeqSpan sp = seq_span(p.cu_q, p.cu_k, seq, p.seqlen_q, p.seqlen_k);
  const int i0 = qt * kBlockM;
  if (i0 >= sp.nq) return;                                // uniform per CTA
  const int g = h / p.group;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int off = sp.nk - sp.nq;                          // bottom-right alignment
  // the keys the tile's rows can see, in steps of 64
  const int tile_r1 = min(i0 + kBlockM, sp.nq) - 1;
  int kv_lo = 0, kv_hi = sp.nk;
  if (p.causal) {
    kv_hi = min(sp.nk, tile_r1 + off + 1);
    if (p.window > 0) kv_lo = max(0, i0 + off - p.window + 1);
  }
  const int lo64 = kv_lo / kDqKeys;
  const int num = kv_hi > kv_lo ? (kv_hi + kDqKeys - 1) / kDqKeys - lo64 : 0;

  if (num == 0) {
    // No row of this tile sees a key: dQ = 0.
    for (int t = tid; t < kBlockM * 8; t += kDqThreads) {
      const int rr = t >> 3, c8 = t & 7;
      if (i0 + rr < sp.nq) {
        const size_t base = ((size_t)(sp.q0 + i0 + rr) * p.heads_q + h) * kHeadDim + 8 * c8;
        if (p.grad_fp32) {
          float4* d4 = reinterpret_cast<float4*>(static_cast<float*>(p.dq) + base);
          d4[0] = make_float4(0.f, 0.f, 0.f, 0.f);
          d4[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
          *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dq) + base) =
              make_uint4(0, 0, 0, 0);
        }
      }
    }
    return;
  }

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sdO = sQ + kTileBytes;
  uint8_t* sK = sdO + kTileBytes;                         // kDqStages 64-key tiles
  uint8_t* sV = sK + kDqStages * kDqKvBytes;              // kDqStages 64-key tiles

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&q_full, 1);
    mbar_init(&s_full, 1);
    mbar_init(&s_read, 2 * kBlockM);
    mbar_init(&dp_full[0], 1);
    mbar_init(&dp_full[1], 1);
    mbar_init(&p_full[0], 2 * kBlockM);
    mbar_init(&p_full[1], 2 * kBlockM);
    mbar_init(&dq_done, 1);
    for (int s = 0; s < kDqStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    fence_mbarrier_init();
  }
  if (warp == kDqMmaWarp) {
    tmem_alloc(&tmem_base_sh, kDqTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == kDqTmaWarp) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_do);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      mbar_arrive_expect_tx(&q_full, 2 * kTileBytes);
      tma_load_3d(&p.tm_q, &q_full, sQ, 0, h, sp.q0 + i0);
      tma_load_3d(&p.tm_do, &q_full, sdO, 0, h, sp.q0 + i0);
      int issued = 0;
      for (int it = 0; it < num; ++it) {
        const int st = it % kDqStages;
        if (it >= kDqStages &&
            !mbar_wait(&kv_empty[st], ((it / kDqStages) & 1) ^ 1, &abort_flag)) {
          abort_flag = 1;
          atomicCAS(p.err, 0, DEVERR_TIMEOUT_BWD + 5);
          break;
        }
        const int row = sp.k0 + (lo64 + it) * kDqKeys;
        mbar_arrive_expect_tx(&kv_full[st], 2 * kDqKvBytes);
        tma_load_3d(&p.tm_k, &kv_full[st], sK + st * kDqKvBytes, 0, g, row);
        tma_load_3d(&p.tm_v, &kv_full[st], sV + st * kDqKvBytes, 0, g, row);
        issued = it + 1;
      }
      if (abort_flag) {
        // Let the copies already in flight land before the CTA releases SMEM.
        mbar_wait(&q_full, 0, nullptr);
        for (int it = max(0, issued - kDqStages); it < issued; ++it)
          mbar_wait(&kv_full[it % kDqStages], (it / kDqStages) & 1, nullptr);
      }
    }
  } else if (warp == kDqMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    // Per key step n, in issue order (tcgen05 MMAs of one thread run in that
    // order): S(n+1) and dP(n+1) once S(n) has been read (s_read; dP(n+1)'s
    // buffer last held dS(n-1), which dQ(n-1), issued before, has read), then
    // dQ(n) once dS(n) is in its dP buffer (p_full).
    if (lane == 0) {
      const uint32_t id_s = make_idesc(kFmtF16, kBlockM, kDqKeys, false, false);
      const uint32_t id_dq = make_idesc(kFmtF16, kBlockM, kHeadDim, false, true);
      const uint64_t dQ0 = make_sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dO0 = make_sdesc_sw128(smem_u32(sdO), 16, 1024);
      const uint64_t dK0 = make_sdesc_sw128(smem_u32(sK), 16, 1024);       // K-major
      const uint64_t dKmn = make_sdesc_sw128(smem_u32(sK), 16384, 1024);   // MN-major
      const uint64_t dV0 = make_sdesc_sw128(smem_u32(sV), 16, 1024);
      constexpr uint32_t kKvU = kDqKvBytes >> 4;
      auto issue_s = [&](int n) -> bool {
        const int st = n % kDqStages;
        if (!mbar_wait(&kv_full[st], (n / kDqStages) & 1, &abort_flag)) return false;
        tc_fence_after();
        #pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k)
          mma_ss(tmem + kDqColS, dQ0 + 2 * k, dK0 + st * kKvU + 2 * k, id_s, k > 0);
        mma_commit(&s_full);
        return true;
      };
      auto issue_dp = [&](int n) {
        const int st = n % kDqStages;
        #pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k)
          mma_ss(tmem + dq_col_dp(n), dO0 + 2 * k, dV0 + st * kKvU + 2 * k, id_s, k > 0);
        mma_commit(&dp_full[n & 1]);
      };
      bool ok = mbar_wait(&q_full, 0, &abort_flag) && issue_s(0);
      if (ok) issue_dp(0);
      for (int n = 0; ok && n < num; ++n) {
        const int st = n % kDqStages;
        // S(n+1) into the S columns the compute warps have read, dP(n+1) into
        // the other dP buffer (its stage landed before S(n+1) was issued)
        if (n + 1 < num) {
          if (!mbar_wait(&s_read, n & 1, &abort_flag) || !issue_s(n + 1)) { ok = false; break; }
          issue_dp(n + 1);
        }
        if (!mbar_wait(&p_full[n & 1], (n >> 1) & 1, &abort_flag)) { ok = false; break; }
        tc_fence_after();
        // dQ += dS K: k-step kk covers keys [16 kk, 16 kk + 16) of the step; the
        // key half c = kk / 2 wrote its dS over columns [32 c, 32 c + 16) of
        // the step's dP buffer.
        #pragma unroll
        for (int kk = 0; kk < kDqKeys / 16; ++kk)
          mma_ts(tmem + kDqColDQ, tmem + dq_col_dp(n) + 32 * (kk >> 1) + 8 * (kk & 1),
                 dKmn + st * kKvU + 128 * kk, id_dq, (n > 0 || kk > 0));
        mma_commit(&kv_empty[st]);          // K(n) and V(n) have been read
      }
      if (!ok) {
        abort_flag = 1;
        atomicCAS(p.err, 0, DEVERR_TIMEOUT_BWD + 6);
      }
      // every MMA has finished before the epilogue reads dQ and TMEM is released
      mma_commit(&dq_done);
      mbar_wait(&dq_done, 0, nullptr);
    }
  } else {
    // ---------------------------------------------------------------- compute warps
    const int c = warp >> 2;                      // key half
    const int r = tid & 127;                      // query row in tile = TMEM lane
    const int i = i0 + r;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = p.scale_log2;
    // this row's (lse log2 e, D); rows past the sequence read a valid row
    const float2 ld = __ldg(p.LD + (size_t)h * p.total_q + sp.q0 + min(i, sp.nq - 1));
    const uint64_t sl2x2 = f2(sl2, sl2), nlse2x2 = f2(ld.x, ld.x), d2 = f2(ld.y, ld.y);
    const int jmax = p.causal ? min(sp.nk - 1, i + off) : sp.nk - 1;   // inclusive
    const int jmin = (p.causal && p.window > 0) ? i + off - p.window + 1 : 0;
    bool ok = true;
    for (int it = 0; it < num; ++it) {
      if (!mbar_wait_warp(&s_full, it & 1, &abort_flag)) { ok = false; break; }
      tc_fence_after();
      const int j0 = (lo64 + it) * kDqKeys + 32 * c;           // first key of this half
      const bool need_mask = (j0 + 32 > sp.nk) ||
                             (p.causal && (j0 + 31 > i0 + off ||
                                           (p.window > 0 && j0 <= tile_r1 + off - p.window)));
      // S -> registers; its columns are then free for the next step's S
      uint32_t pr[32];
      tmem_ld_x32(tmem + lane_base + kDqColS + 32 * c, pr);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&s_read);
      // P in place (fp32), masked entries exactly 0
      if (need_mask)
        dq_p_chunk<true>(pr, sl2x2, nlse2x2, j0, jmin, jmax);
      else
        dq_p_chunk<false>(pr, sl2x2, nlse2x2, j0, jmin, jmax);
      if (!mbar_wait_warp(&dp_full[it & 1], (it >> 1) & 1, &abort_flag)) { ok = false; break; }
      tc_fence_after();
      {
        uint32_t dr[32], dk[16];
        tmem_ld_x32(tmem + lane_base + dq_col_dp(it) + 32 * c, dr);
        tmem_ld_wait();
        dq_ds_chunk(pr, dr, d2, dk);
        // dS (16 packed columns) over the dP columns this thread has read
        tmem_st_x16(tmem + lane_base + dq_col_dp(it) + 32 * c, dk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[it & 1]);
    }
    // fin is warp-uniform (every wait above is), so the whole warp reaches the
    // .sync.aligned TMEM load; only the stores depend on the row.
    bool fin = ok && mbar_wait_warp(&dq_done, 0, &abort_flag);
    if (!fin) {
      abort_flag = 1;
      atomicCAS(p.err, 0, DEVERR_TIMEOUT_BWD + 7);
    } else {
      // dQ columns [32 c, 32 c + 32) of this row, times the softmax scale
      tc_fence_after();
      uint32_t v[32];
      tmem_ld_x32(tmem + lane_base + kDqColDQ + 32 * c, v);
      tmem_ld_wait();
      if (i < sp.nq) {
        const size_t base = ((size_t)(sp.q0 + i) * p.heads_q + h) * kHeadDim + 32 * c;
        if (p.grad_fp32) {
          float4* d4 = reinterpret_cast<float4*>(static_cast<float*>(p.dq) + base);
          #pragma unroll
          for (int u = 0; u < 8; ++u)
            d4[u] = make_float4(__uint_as_float(v[4 * u]) * p.scale,
                                __uint_as_float(v[4 * u + 1]) * p.scale,
                                __uint_as_float(v[4 * u + 2]) * p.scale,
                                __uint_as_float(v[4 * u + 3]) * p.scale);
        } else {
          uint4* d4 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dq) + base);
          #pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint32_t w[4];
            #pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(v[8 * u + 2 * e]) * p.scale,
                                 __uint_as_float(v[8 * u + 2 * e + 1]) * p.scale);
            d4[u] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kDqMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kDqTmemCols);
  }
}

}  // namespace attn_sink
