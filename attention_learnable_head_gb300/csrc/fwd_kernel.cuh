// Forward kernel: attention with a per-head sink, sm_103a (tcgen05 + TMA).
//
// Computes, for one (query head h, sequence, 128-row query tile) per CTA,
//   S = Q K^T (tcgen05, fp32 in TMEM), an online softmax whose running max and
//   sum start from the sink logit (m0 = sink[h], l0 = 1 in the exp2 domain), and
//   O += P V (tcgen05), then out = O / l and lse = ln(l) + m (sink included).
// The sink enters the softmax denominator only: it is the extra column of the
// concat listing "带汇聚的注意力（GPT-OSS）" on the euno.news page, and the
// P_ij / P_ih equations of its section "数学公式".
//
// Warp roles (192 threads):
//   warps 0-3  softmax: thread t owns query row t (TMEM lane t); rescales O in
//              TMEM, writes P (bf16) to a swizzled SMEM tile, runs the epilogue.
//   warp 4     TMA producer: Q once, then K/V tiles through an NSTAGE ring.
//   warp 5     MMA issuer (one lane) and TMEM owner.
// TMEM columns: S double buffer at 0 and 128 (128 fp32 columns each), O at 256.
#pragma once
#include <cuda_bf16.h>
#include "sm103_ptx.cuh"

namespace attn_sink {

constexpr int kBlockM = 128;   // query rows per tile
constexpr int kBlockN = 128;   // keys per tile
constexpr int kHeadDim = 64;
constexpr int kFwdStages = 3;
constexpr int kFwdThreads = 192;
constexpr uint32_t kTileBytes = kBlockM * kHeadDim * 2;   // 16 KB bf16 tile
constexpr uint32_t kPTileBytes = kBlockM * kBlockN * 2;   // 32 KB bf16 P tile
constexpr int kFwdSmemBytes =
    1024 + (int)kTileBytes * (1 + 2 * kFwdStages) + 2 * (int)kPTileBytes;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct FwdParams {
  CUtensorMap tm_q;   // [T_q][H_q][64] bf16, box 64 x 1 x 128, 128B swizzle
  CUtensorMap tm_k;   // [T_k][H_kv][64]
  CUtensorMap tm_v;
  const int* cu_q;    // null for a dense batch
  const int* cu_k;
  const float* sink;  // [H_q]
  __nv_bfloat16* out; // [T_q][H_q][64]
  float* lse;         // [H_q][T_q]
  int* err;           // device error word
  int seqlen_q, seqlen_k;
  int total_q;
  int heads_q, group;
  int causal, window;
  float scale_log2;   // softmax_scale * log2(e)
  int n_qtiles;       // number of query tiles of the longest sequence
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

__global__ void __launch_bounds__(kFwdThreads, 1)
attn_sink_fwd_kernel(const __grid_constant__ FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t q_full, pv_done, mma_drained;
  __shared__ __align__(8) uint64_t k_full[kFwdStages], v_full[kFwdStages], kv_empty[kFwdStages];
  __shared__ __align__(8) uint64_t s_full[2], p_full[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;

  const int h = blockIdx.x;
  const int seq = blockIdx.y;
  const int qtile = p.n_qtiles - 1 - (int)blockIdx.z;   // longest work first
  const SeqSpan sp = seq_span(p.cu_q, p.cu_k, seq, p.seqlen_q, p.seqlen_k);
  const int i0 = qtile * kBlockM;
  if (i0 >= sp.nq) return;                              // uniform per CTA
  const int g = h / p.group;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int off = sp.nk - sp.nq;                         // bottom-right causal offset
  const int last_row = min(i0 + kBlockM, sp.nq) - 1;

  // Key range [kv_lo, kv_hi) any row of this tile can see.
  int kv_lo = 0, kv_hi = sp.nk;
  if (p.causal) {
    kv_hi = min(sp.nk, last_row + off + 1);
    if (p.window > 0) kv_lo = max(0, i0 + off - p.window + 1);
  }
  const int n_first = kv_lo / kBlockN;
  const int num = (kv_hi > kv_lo) ? ((kv_hi + kBlockN - 1) / kBlockN - n_first) : 0;
  const float sink_h = __ldg(p.sink + h);

  if (num == 0) {
    // No row of this tile sees a key: out = 0, lse = sink (the sink alone).
    if (tid < kBlockM && i0 + tid < sp.nq) {
      const size_t row = (size_t)(sp.q0 + i0 + tid);
      uint4* o = reinterpret_cast<uint4*>(p.out + (row * p.heads_q + h) * kHeadDim);
      #pragma unroll
      for (int c = 0; c < 8; ++c) o[c] = make_uint4(0, 0, 0, 0);
      p.lse[(size_t)h * p.total_q + row] = sink_h;
    }
    return;
  }

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + kTileBytes;
  uint8_t* sV = sK + kFwdStages * kTileBytes;
  uint8_t* sP = sV + kFwdStages * kTileBytes;

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&q_full, 1);
    mbar_init(&pv_done, 1);
    mbar_init(&mma_drained, 1);
    for (int s = 0; s < kFwdStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], kBlockM);
    }
    fence_mbarrier_init();
  }
  if (warp == 5) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t tm_o = tmem + 256;

  if (warp == 4) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      const uint64_t keep = l2_policy_evict_last();
      mbar_arrive_expect_tx(&q_full, kTileBytes);
      tma_load_3d(&p.tm_q, &q_full, sQ, 0, h, sp.q0 + i0);
      int issued = 0;
      for (int it = 0; it < num; ++it) {
        const int st = it % kFwdStages;
        if (it >= kFwdStages &&
            !mbar_wait(&kv_empty[st], ((it / kFwdStages) & 1) ^ 1, &abort_flag)) {
          abort_flag = 1;
          atomicCAS(p.err, 0, DEVERR_TIMEOUT_FWD + 1);
          break;
        }
        const int row = sp.k0 + (n_first + it) * kBlockN;
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
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = make_idesc_bf16(kBlockM, kBlockN, false, false);
      const uint32_t idesc_o = make_idesc_bf16(kBlockM, kHeadDim, false, true);
      const uint32_t aQ = smem_u32(sQ);
      bool ok = mbar_wait(&q_full, 0, &abort_flag) && mbar_wait(&k_full[0], 0, &abort_flag);
      if (ok) {
        tc_fence_after();
        const uint32_t aK = smem_u32(sK);
        #pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k)
          mma_bf16_ss(tmem, make_sdesc_sw128(aQ + 32 * k, 16, 1024),
                      make_sdesc_sw128(aK + 32 * k, 16, 1024), idesc_s, k > 0);
        mma_commit(&s_full[0]);
      }
      for (int it = 0; ok && it < num; ++it) {
        if (it + 1 < num) {
          const int st1 = (it + 1) % kFwdStages;
          if (!mbar_wait(&k_full[st1], ((it + 1) / kFwdStages) & 1, &abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t aK = smem_u32(sK + st1 * kTileBytes);
          const uint32_t dS = tmem + ((it + 1) & 1) * 128;
          #pragma unroll
          for (int k = 0; k < kHeadDim / 16; ++k)
            mma_bf16_ss(dS, make_sdesc_sw128(aQ + 32 * k, 16, 1024),
                        make_sdesc_sw128(aK + 32 * k, 16, 1024), idesc_s, k > 0);
          mma_commit(&s_full[(it + 1) & 1]);
        }
        const int b = it & 1;
        const int st = it % kFwdStages;
        if (!mbar_wait(&p_full[b], (it >> 1) & 1, &abort_flag) ||
            !mbar_wait(&v_full[st], (it / kFwdStages) & 1, &abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t aP = smem_u32(sP + b * kPTileBytes);
        const uint32_t aV = smem_u32(sV + st * kTileBytes);
        #pragma unroll
        for (int k = 0; k < kBlockN / 16; ++k)
          mma_bf16_ss(tm_o, make_sdesc_sw128(aP + (k >> 2) * kTileBytes + (k & 3) * 32, 16, 1024),
                      make_sdesc_sw128(aV + k * 2048, 16384, 1024), idesc_o, (it > 0 || k > 0));
        mma_commit(&kv_empty[st]);
        mma_commit(&pv_done);
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
    const int r = tid;                       // query row within the tile, TMEM lane
    const int i = i0 + r;                    // row within the sequence
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const bool sink_finite = sink_h > -INFINITY;
    float m = sink_finite ? sink_h * kLog2e : -INFINITY;   // running max, log2 domain
    float l = sink_finite ? 1.0f : 0.0f;                    // running sum, sink term = 1
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int it = 0; it < num; ++it) {
      const int b = it & 1;
      if (!mbar_wait_warp(&s_full[b], (it >> 1) & 1, &abort_flag)) { ok = false; break; }
      tc_fence_after();
      float s[kBlockN];
      #pragma unroll
      for (int c = 0; c < kBlockN; c += 32)
        tmem_ld_x32(tmem + lane_base + b * 128 + c, reinterpret_cast<uint32_t*>(s + c));
      tmem_ld_wait();

      const int j0 = (n_first + it) * kBlockN;
      const bool need_mask = (j0 + kBlockN > sp.nk) ||
                             (p.causal && (j0 + kBlockN - 1 > i0 + off ||
                                           (p.window > 0 && j0 <= last_row + off - p.window)));
      if (need_mask) {
        const int jmax = p.causal ? min(sp.nk - 1, i + off) : sp.nk - 1;   // inclusive
        const int jmin = (p.causal && p.window > 0) ? i + off - p.window + 1 : 0;
        #pragma unroll
        for (int c = 0; c < kBlockN; ++c) {
          const int j = j0 + c;
          if (j > jmax || j < jmin) s[c] = -INFINITY;
        }
      }
      float mx = -INFINITY;
      #pragma unroll
      for (int c = 0; c < kBlockN; ++c) mx = fmaxf(mx, s[c]);
      const float m_new = fmaxf(m, mx * sl2);
      const float alpha = (m_new == m) ? 1.0f : ex2_approx(m - m_new);
      const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;

      if (it > 0) {
        // P(it-1)V finished: O may be rescaled and the P buffer of it-2 is free.
        if (!mbar_wait_warp(&pv_done, (it - 1) & 1, &abort_flag)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
          #pragma unroll
          for (int c = 0; c < kHeadDim; c += 32) {
            uint32_t o[32];
            tmem_ld_x32(tm_o + lane_base + c, o);
            tmem_ld_wait();
            #pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st_x32(tm_o + lane_base + c, o);
          }
          tmem_st_wait();
        }
      }
      m = m_new;

      float rowsum = 0.0f;
      const uint32_t pbase = smem_u32(sP + b * kPTileBytes);
      #pragma unroll
      for (int c = 0; c < kBlockN; c += 8) {
        float e[8];
        #pragma unroll
        for (int u = 0; u < 8; ++u) {
          e[u] = ex2_approx(fmaf(s[c + u], sl2, -m_use));
          rowsum += e[u];
        }
        const uint32_t addr = pbase + (c >> 6) * kTileBytes + sw128_offset(r, (c & 63) >> 3);
        st_shared_v4(addr, pack_bf16x2(e[0], e[1]), pack_bf16x2(e[2], e[3]),
                     pack_bf16x2(e[4], e[5]), pack_bf16x2(e[6], e[7]));
      }
      l = l * alpha + rowsum;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[b]);
    }
    if (ok && !mbar_wait_warp(&pv_done, (num - 1) & 1, &abort_flag)) ok = false;
    if (!ok) {
      abort_flag = 1;
      atomicCAS(p.err, 0, DEVERR_TIMEOUT_FWD + 3);
    } else {
      tc_fence_after();
      const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
      const bool valid = i < sp.nq;
      const size_t row = (size_t)(sp.q0 + i);
      #pragma unroll
      for (int c = 0; c < kHeadDim; c += 32) {
        uint32_t o[32];
        tmem_ld_x32(tm_o + lane_base + c, o);
        tmem_ld_wait();
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + (row * p.heads_q + h) * kHeadDim + c);
          #pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float* f = reinterpret_cast<const float*>(o + 8 * u);
            dst[u] = make_uint4(pack_bf16x2(f[0] * inv_l, f[1] * inv_l),
                                pack_bf16x2(f[2] * inv_l, f[3] * inv_l),
                                pack_bf16x2(f[4] * inv_l, f[5] * inv_l),
                                pack_bf16x2(f[6] * inv_l, f[7] * inv_l));
          }
        }
      }
      if (valid)
        p.lse[(size_t)h * p.total_q + row] = (l > 0.0f) ? (m + __log2f(l)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace attn_sink
