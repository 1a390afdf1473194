// Backward kernels: attention with a per-head sink, sm_103a.
//
//   bwd_pre     D_i = sum_d dout_i[d] * out_i[d] (fp32; out = the stored bf16 out
//               plus, when given, its bf16 residual), per-block partials of
//               dsink[h] = -sum_i exp(sink[h] - lse_i) * D_i (the sink gradient of
//               section "反向传播" on the euno.news page: P_ih = exp(sink[h] - lse_i)
//               because lse includes the sink), fp16 copies of q and dout for the
//               tensor cores, and zeroes the fp32 dq accumulator.
//   kv_convert  fp16 copies of k and v.
//   bwd_main    key/value-stationary: one CTA per (kv head, GQA slice, sequence,
//               128 keys).  Loops over the query heads of its slice and the
//               query tiles that can see these keys; per step (128 queries, in
//               two halves of 64) five tcgen05 MMAs, all on fp16 operands (the
//               inputs convert exactly; P and dS keep 11 significand bits):
//                 S^T  = K Q^T        dP^T = V dO^T            (TMEM, fp32, per half)
//                 P^T  = exp(S^T * scale - lse)  dS^T = P^T o (dP^T - D)
//                 dV  += P^T dO       dK += dS^T Q             (per half, K = 64)
//                 dQ   = dS K         (A = dS^T read MN-major, once per step)
//               Two compute warpgroups own one query half each, so the tensor
//               cores run one half's products while the other half's exponentials
//               are computed; two threads issue the MMAs (S^T, dP^T, dV / dK, dQ)
//               so that one's waits do not idle the tensor pipe.  dK and dV stay
//               in TMEM for the whole loop; a
//               dedicated warpgroup moves each step's dQ from TMEM into a
//               swizzled shared-memory tile that a TMA reduce-add sums into
//               the fp32 accumulator.
//   dsink_reduce  fixed-order tree over the partials (bitwise reproducible).
//   dq_convert  fp32 accumulator -> bf16 dq.
#pragma once
#include <cuda_bf16.h>
#include "sm103_ptx.cuh"
#include "fwd_kernel.cuh"

namespace attn_sink {

constexpr int kBwdStages = 3;       // Q / dO ring depth
// warps 0-3 compute queries 0-63 of a step, 4-7 queries 64-127, 8 TMA, 9 MMA issuer A
// (S^T, dP^T, dV), 10-13 dQ, 14 MMA issuer B (dK, dQ)
constexpr int kBwdThreads = 480;
constexpr int kBwdProducerWarp = 8;
constexpr int kBwdMmaWarp = 9;
constexpr int kBwdDqWarp0 = 10;
constexpr int kBwdMma2Warp = 14;
constexpr int kPreRows = 128;      // rows per bwd_pre CTA
constexpr uint32_t kDqStageBytes = kBlockM * 32 * 4;   // 16 KB: half of a fp32 dQ tile
// K, V, kBwdStages x (Q, dO), 2 x dS^T, the dQ staging tile
constexpr int kBwdSmemBytes = 1024 + 2 * (int)kTileBytes + kBwdStages * 2 * (int)kTileBytes +
                              2 * (int)kPTileBytes + (int)kDqStageBytes;

// TMEM columns of bwd_main (S^T / dP^T: query half hh at +64 hh)
// Dynamic + static shared memory must stay within the 227 KB a CTA may use.
static_assert(kBwdSmemBytes + 4096 <= 232448, "backward shared memory over the per-CTA limit");

// P^T (fp16, two per column) of query half hh is written over the first 32
// columns of that half of S^T once read.  K and V (fp16, two per column) are
// copied into TMEM once, as the A operands of S^T = K Q^T and dP^T = V dO^T.
constexpr uint32_t kColST = 0, kColDPT = 128, kColDV = 256, kColDK = 320, kColDQ = 384,
                   kColK = 448, kColV = 480;

struct BwdParams {
  CUtensorMap tm_q;    // [T_q][H_q][64] fp16 copy of q
  CUtensorMap tm_do;   // [T_q][H_q][64] fp16 copy of dout
  CUtensorMap tm_k;    // [T_k][H_kv][64] fp16 copy of k
  CUtensorMap tm_v;    // fp16 copy of v
  CUtensorMap tm_dq;   // [T_q][H_q][64] fp32 dq accumulator, box 32 x 1 x 128, 128B swizzle
  const int* cu_q;
  const int* cu_k;
  const float2* LD;    // [H_q][T_q]: (-lse * log2 e, D) per query row
  float* dq_acc;       // [T_q][H_q][64], zeroed unless null fp32, pre-zeroed
  void* dk;            // [T_k][H_kv][64] bf16 or fp32 (split == 1)
  void* dv;
  float* dk_part;      // [split][T_k][H_kv][64] fp32 partials (split > 1)
  float* dv_part;
  int* err;
  int seqlen_q, seqlen_k;
  int total_q, total_k;
  int heads_q, heads_kv, group;
  int split;           // CTAs sharing one (kv head, key tile); each takes group/split q heads
  int causal, window;
  float scale;         // softmax_scale
  float scale_log2;    // softmax_scale * log2(e)
  int n_ktiles;        // key tiles of the longest sequence
  // Packed batches of several sequences: the key tile of CTA row blockIdx.y,
  // as seq << 16 | key tile, heaviest first (null: blockIdx.y / z give them)
  const uint32_t* work;
  int grad_fp32;
  int skip_dq;         // 1: no dQ here (the deterministic dQ kernel computes it)
#ifdef ATTN_SINK_TEST_HOOKS
  int skip_q_step;     // test build: the producer never loads this step's Q/dO (-1: none)
#endif
};

// ------------------------------------------------------------------ bwd_pre
struct PreParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* out;
  const __nv_bfloat16* out_lo;   // residual of out, or null
  const __nv_bfloat16* dout;
  const float* lse;
  const float* sink;
  const __nv_bfloat16* sink_bf16;   // bf16 sink when non-null
  float2* LD;          // [H_q][T_q]: (-lse * log2 e, D)
  float* partials;     // [H_q][n_blocks]
  float* dq_acc;       // [T_q][H_q][64]
  uint16_t* q16;       // [T_q][H_q][64] fp16 copy of q
  uint16_t* do16;      // [T_q][H_q][64] fp16 copy of dout
  int* err;
  int total_q, heads_q, n_blocks;
};

__global__ void __launch_bounds__(256) attn_sink_bwd_pre_kernel(const PreParams p) {
  const int h = blockIdx.y;
  const int blk = blockIdx.x;
  const int tid = threadIdx.x;
  const int sub = tid & 7;          // 16-byte slice of the 128-byte row
  const int rloc = tid >> 3;        // 0..31
  const float sink_h = p.sink_bf16 ? __bfloat162float(p.sink_bf16[h]) : p.sink[h];
  float acc = 0.0f;                 // dsink contribution of this thread's rows
  bool overflow = false;
  #pragma unroll 1
  for (int pass = 0; pass < kPreRows / 32; ++pass) {
    const int t = blk * kPreRows + pass * 32 + rloc;
    float d = 0.0f;
    if (t < p.total_q) {
      const size_t base = ((size_t)t * p.heads_q + h) * kHeadDim + sub * 8;
      const uint4 o = *reinterpret_cast<const uint4*>(p.out + base);
      const uint4 g = *reinterpret_cast<const uint4*>(p.dout + base);
      const uint4 qq = *reinterpret_cast<const uint4*>(p.q + base);
      uint4 ol = make_uint4(0, 0, 0, 0);
      if (p.out_lo) ol = *reinterpret_cast<const uint4*>(p.out_lo + base);
      const uint32_t ow[4] = {o.x, o.y, o.z, o.w}, gw[4] = {g.x, g.y, g.z, g.w};
      const uint32_t lw[4] = {ol.x, ol.y, ol.z, ol.w};
      #pragma unroll
      for (int u = 0; u < 4; ++u) {
        d = fmaf(bf16_lo(ow[u]) + bf16_lo(lw[u]), bf16_lo(gw[u]), d);
        d = fmaf(bf16_hi(ow[u]) + bf16_hi(lw[u]), bf16_hi(gw[u]), d);
      }
      *reinterpret_cast<uint4*>(p.q16 + base) =
          make_uint4(bf16x2_to_f16x2(qq.x, &overflow), bf16x2_to_f16x2(qq.y, &overflow),
                     bf16x2_to_f16x2(qq.z, &overflow), bf16x2_to_f16x2(qq.w, &overflow));
      *reinterpret_cast<uint4*>(p.do16 + base) =
          make_uint4(bf16x2_to_f16x2(g.x, &overflow), bf16x2_to_f16x2(g.y, &overflow),
                     bf16x2_to_f16x2(g.z, &overflow), bf16x2_to_f16x2(g.w, &overflow));
      if (p.dq_acc) {
        float4* z = reinterpret_cast<float4*>(p.dq_acc + base);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    d += __shfl_xor_sync(0xffffffffu, d, 1);
    d += __shfl_xor_sync(0xffffffffu, d, 2);
    d += __shfl_xor_sync(0xffffffffu, d, 4);
    if (sub == 0 && t < p.total_q) {
      const float lse = p.lse[(size_t)h * p.total_q + t];
      p.LD[(size_t)h * p.total_q + t] = make_float2(-lse * kLog2e, d);
      // P_ih = exp(sink - lse); zero when the sink is -inf.
      if (sink_h > -INFINITY && lse > -INFINITY)
        acc -= ex2_approx((sink_h - lse) * kLog2e) * d;
    }
  }
  if (overflow) atomicCAS(p.err, 0, DEVERR_FP16_RANGE);
  // fixed-order reduction: lanes (xor tree), then warps in index order
  #pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  __shared__ float wsum[8];
  if ((tid & 31) == 0) wsum[tid >> 5] = acc;
  __syncthreads();
  if (tid == 0) {
    float s = 0.0f;
    #pragma unroll
    for (int w = 0; w < 8; ++w) s += wsum[w];
    p.partials[(size_t)h * p.n_blocks + blk] = s;
  }
}

// ------------------------------------------------------------------ convert_f16
// fp16 copy of one bf16 tensor (n8 = elements / 8), for the forward's v.
__global__ void __launch_bounds__(256) attn_sink_convert_f16_kernel(const __nv_bfloat16* x,
                                                                    uint16_t* x16, size_t n8,
                                                                    int* err) {
  bool overflow = false;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const uint4 a = reinterpret_cast<const uint4*>(x)[i];
    reinterpret_cast<uint4*>(x16)[i] =
        make_uint4(bf16x2_to_f16x2(a.x, &overflow), bf16x2_to_f16x2(a.y, &overflow),
                   bf16x2_to_f16x2(a.z, &overflow), bf16x2_to_f16x2(a.w, &overflow));
  }
  if (overflow) atomicCAS(err, 0, DEVERR_FP16_RANGE);
}

// ------------------------------------------------------------------ kv_convert
// fp16 copies of k and v (n8 = elements / 8 of each).
__global__ void __launch_bounds__(256) attn_sink_kv_convert_kernel(
    const __nv_bfloat16* k, const __nv_bfloat16* v, uint16_t* k16, uint16_t* v16, size_t n8,
    int* err) {
  bool overflow = false;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const uint4 a = reinterpret_cast<const uint4*>(k)[i];
    const uint4 b = reinterpret_cast<const uint4*>(v)[i];
    reinterpret_cast<uint4*>(k16)[i] =
        make_uint4(bf16x2_to_f16x2(a.x, &overflow), bf16x2_to_f16x2(a.y, &overflow),
                   bf16x2_to_f16x2(a.z, &overflow), bf16x2_to_f16x2(a.w, &overflow));
    reinterpret_cast<uint4*>(v16)[i] =
        make_uint4(bf16x2_to_f16x2(b.x, &overflow), bf16x2_to_f16x2(b.y, &overflow),
                   bf16x2_to_f16x2(b.z, &overflow), bf16x2_to_f16x2(b.w, &overflow));
  }
  if (overflow) atomicCAS(err, 0, DEVERR_FP16_RANGE);
}

// ------------------------------------------------------------------ dsink_reduce
// dsink[h] (fp32, or bf16 with dsink_bf16) = the sum of the partials, or
// += it with accumulate.
__global__ void __launch_bounds__(256) attn_sink_dsink_reduce_kernel(const float* partials,
                                                                     int n_blocks, void* dsink,
                                                                     int dsink_bf16,
                                                                     int accumulate) {
  const int h = blockIdx.x;
  const int tid = threadIdx.x;
  float s = 0.0f;
  for (int j = tid; j < n_blocks; j += 256) s += partials[(size_t)h * n_blocks + j];
  #pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  __shared__ float wsum[8];
  if ((tid & 31) == 0) wsum[tid >> 5] = s;
  __syncthreads();
  if (tid == 0) {
    float t = 0.0f;
    #pragma unroll
    for (int w = 0; w < 8; ++w) t += wsum[w];
    if (dsink_bf16) {
      __nv_bfloat16* d = static_cast<__nv_bfloat16*>(dsink) + h;
      *d = __float2bfloat16_rn(accumulate ? __bfloat162float(*d) + t : t);
    } else {
      float* d = static_cast<float*>(dsink) + h;
      *d = accumulate ? *d + t : t;
    }
  }
}

// ------------------------------------------------------------------ dq_convert
__global__ void __launch_bounds__(256) attn_sink_dq_convert_kernel(const float* acc,
                                                                   __nv_bfloat16* dq,
                                                                   size_t n8) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    reinterpret_cast<uint4*>(dq)[i] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w),
                                                 pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
  }
}

// ------------------------------------------------------------------ dkdv_reduce
// dK = scale * sum_s dk_part[s], dV = sum_s dv_part[s], in a fixed order
// (s = 0, 1, ...), so the result is bitwise reproducible.
__global__ void __launch_bounds__(256) attn_sink_dkdv_reduce_kernel(
    const float* dk_part, const float* dv_part, int split, size_t n4, float scale, void* dk,
    void* dv, int grad_fp32) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    #pragma unroll
    for (int which = 0; which < 2; ++which) {
      const float4* src = reinterpret_cast<const float4*>(which == 0 ? dk_part : dv_part);
      float4 a = src[i];
      for (int s = 1; s < split; ++s) {
        const float4 b = src[(size_t)s * n4 + i];
        a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
      }
      const float mul = which == 0 ? scale : 1.0f;
      a.x *= mul; a.y *= mul; a.z *= mul; a.w *= mul;
      void* dst = which == 0 ? dk : dv;
      if (grad_fp32)
        reinterpret_cast<float4*>(dst)[i] = a;
      else
        reinterpret_cast<uint2*>(dst)[i] = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
    }
  }
}

// ------------------------------------------------------------------ bwd_main
// Store one 64-wide row of dK (which = 0) or dV (which = 1) for key `row`:
// the final output (times `mul`) when the GQA group is not split, else this
// CTA's fp32 partial (unscaled; the reduction applies the scale).
__device__ __forceinline__ void store_kv_grad_row(const BwdParams& p, int part, size_t row,
                                                  int g, int which, const float* v, float mul) {
  const size_t base = (row * p.heads_kv + g) * kHeadDim;
  if (p.split > 1) {
    float* dst = (which == 0 ? p.dk_part : p.dv_part) +
                 (size_t)part * p.total_k * p.heads_kv * kHeadDim + base;
    #pragma unroll
    for (int u = 0; u < kHeadDim / 4; ++u)
      reinterpret_cast<float4*>(dst)[u] =
          make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
  } else if (p.grad_fp32) {
    float* dst = reinterpret_cast<float*>(which == 0 ? p.dk : p.dv) + base;
    #pragma unroll
    for (int u = 0; u < kHeadDim / 4; ++u)
      reinterpret_cast<float4*>(dst)[u] = make_float4(v[4 * u] * mul, v[4 * u + 1] * mul,
                                                      v[4 * u + 2] * mul, v[4 * u + 3] * mul);
  } else {
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(which == 0 ? p.dk : p.dv) + base;
    #pragma unroll
    for (int u = 0; u < kHeadDim / 8; ++u)
      reinterpret_cast<uint4*>(dst)[u] = make_uint4(
          pack_bf16x2(v[8 * u] * mul, v[8 * u + 1] * mul), pack_bf16x2(v[8 * u + 2] * mul, v[8 * u + 3] * mul),
          pack_bf16x2(v[8 * u + 4] * mul, v[8 * u + 5] * mul), pack_bf16x2(v[8 * u + 6] * mul, v[8 * u + 7] * mul));
  }
}

// P^T of 64 queries of one key row (thread = key), fp16-packed:
//   P = exp2(S * scale * log2 e - lse * log2 e)   (lse includes the sink)
// nl_row holds -lse * log2 e of the 64 queries.  Pairs of queries go through
// the packed fp32 pair instructions; the exponentials stay per element.  With
// kMask, entries whose (query, key) pair is not visible, or whose row or key
// lies past the sequence, are exact zeros: per block of 16 queries, a block
// that no key of the warp sees is written as zeros without its exponentials,
// and only a block that some key sees in part is masked element by element.
// The thread's visible queries are [lo, hi] (within the sequence; lo > hi for
// none).
template <bool kMask>
__device__ __forceinline__ void bwd_p_chunk(const uint32_t* sr, const float* nl_row,
                                            uint64_t sl2x2, int i_first, int lo, int hi,
                                            uint32_t* pk) {
  #pragma unroll
  for (int b = 0; b < 64; b += 16) {
    const int b0 = i_first + b;               // first query of the block
    bool none = false, part = false;
    if (kMask) {
      none = __all_sync(0xffffffffu, b0 + 15 < lo || b0 > hi);
      part = __any_sync(0xffffffffu, b0 < lo || b0 + 15 > hi);
    }
    if (none) {
      #pragma unroll
      for (int e = b; e < b + 16; e += 2) pk[e >> 1] = 0u;
      continue;
    }
    #pragma unroll
    for (int e = b; e < b + 16; e += 4) {
      const float4 nl = *reinterpret_cast<const float4*>(nl_row + e);
      #pragma unroll
      for (int u = 0; u < 4; u += 2) {
        const uint64_t x = ffma2(f2(__uint_as_float(sr[e + u]), __uint_as_float(sr[e + u + 1])),
                                 sl2x2, u == 0 ? f2(nl.x, nl.y) : f2(nl.z, nl.w));
        float p0 = ex2_approx(f2_lo(x));
        float p1 = ex2_approx(f2_hi(x));
        if (part) {
          const int i = i_first + e + u;
          if (i < lo || i > hi) p0 = 0.0f;
          if (i + 1 < lo || i + 1 > hi) p1 = 0.0f;
        }
        pk[(e + u) >> 1] = pack_f16x2(p0, p1);
      }
    }
  }
}

// dS^T = P^T o (dP^T - D) of 32 queries of one key row, fp16-packed, from the
// fp16 P^T this thread stored for the dV product (pk, 16 words), dP^T (dr) and
// the queries' D (d_row).  Masked entries have P = 0, hence dS = 0.
__device__ __forceinline__ void bwd_ds_chunk(const uint32_t* dr, const uint32_t* pk,
                                             const float* d_row, uint32_t* dk) {
  #pragma unroll
  for (int e = 0; e < 32; e += 4) {
    const float4 dd = *reinterpret_cast<const float4*>(d_row + e);
    #pragma unroll
    for (int u = 0; u < 4; u += 2) {
      const uint64_t pp = f16x2_to_f2(pk[(e + u) >> 1]);
      const uint64_t ds = fmul2(
          pp, fsub2(f2(__uint_as_float(dr[e + u]), __uint_as_float(dr[e + u + 1])),
                    u == 0 ? f2(dd.x, dd.y) : f2(dd.z, dd.w)));
      dk[(e + u) >> 1] = pack_f16x2(f2_lo(ds), f2_hi(ds));
    }
  }
}

__global__ void __launch_bounds__(kBwdThreads, 1)
attn_sink_bwd_main_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t kv_full, kv_tmem, mma2_done, drained;
  __shared__ __align__(8) uint64_t q_full[kBwdStages], q_empty[kBwdStages];
  __shared__ __align__(8) uint64_t s_full, dp_full, p_ready, ds_ready, dq_free;
  __shared__ __align__(8) uint64_t ds_free[2], dpt_issued[2];
  __shared__ __align__(16) float s_nL[kBwdStages][kBlockM];   // -lse * log2 e of the step's rows
  __shared__ __align__(16) float s_D[kBwdStages][kBlockM];    // D of the step's rows
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;

  const int g = blockIdx.x / p.split;      // kv head
  const int part = blockIdx.x % p.split;   // which slice of the GQA group
  const int hpc = p.group / p.split;       // query heads handled by this CTA
  const int h_first = g * p.group + part * hpc;
  // Key tiles vary before sequences (low key tiles carry the most work: first),
  // so the CTAs resident at one time work on one sequence; a packed batch of
  // several sequences takes its tiles from a table sorted by work across all
  // sequences.
  int ktile, seq;
  if (p.work != nullptr) {
    const uint32_t wk = p.work[blockIdx.y];
    if (wk == kNoWork) return;                 // uniform per CTA
    seq = (int)(wk >> 16);
    ktile = (int)(wk & 0xFFFFu);
  } else {
    ktile = blockIdx.y;
    seq = blockIdx.z;
  }
  const SeqSpan sp = seq_span(p.cu_q, p.cu_k, seq, p.seqlen_q, p.seqlen_k);
  const int j0 = ktile * kBlockN;
  if (j0 >= sp.nk) return;                 // uniform per CTA
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int off = sp.nk - sp.nq;
  const int last_key = min(j0 + kBlockN, sp.nk) - 1;

  // Query rows that can see a key of this tile: i >= j - off, i < j - off + W.
  int q_lo = 0, q_hi = sp.nq;
  if (p.causal) {
    q_lo = max(0, j0 - off);
    if (p.window > 0) q_hi = min(sp.nq, last_key - off + p.window);
  }
  const int qt_first = q_lo / kBlockM;
  const int nqt = (q_hi > q_lo) ? ((q_hi + kBlockM - 1) / kBlockM - qt_first) : 0;
  const int num = nqt * hpc;               // steps: (query tile) x (query head), heads fastest

  if (num == 0) {
    // No query sees these keys: dK = dV = 0.
    if (tid < kBlockN && j0 + tid < sp.nk) {
      const size_t row = (size_t)(sp.k0 + j0 + tid);
      float zero[kHeadDim];
      #pragma unroll
      for (int c = 0; c < kHeadDim; ++c) zero[c] = 0.0f;
      store_kv_grad_row(p, part, row, g, 0, zero, 1.0f);
      store_kv_grad_row(p, part, row, g, 1, zero, 1.0f);
    }
    return;
  }

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + kTileBytes;
  uint8_t* sQ = sV + kTileBytes;                      // kBwdStages tiles
  uint8_t* sdO = sQ + kBwdStages * kTileBytes;        // kBwdStages tiles
  uint8_t* sdS = sdO + kBwdStages * kTileBytes;       // 2 x [128 keys][128 queries] fp16
  uint8_t* sdQ = sdS + 2 * kPTileBytes;                // [128 queries][32] fp32, swizzled

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&kv_full, 1);
    mbar_init(&kv_tmem, 2 * kBlockN);
    mbar_init(&mma2_done, 1);
    mbar_init(&drained, 2);               // one commit from each MMA issuer
    for (int s = 0; s < kBwdStages; ++s) {
      mbar_init(&q_full[s], 1 + 32);      // TMA arrival + 32 lanes' cp.async (lse / D)
      mbar_init(&q_empty[s], 2);          // read by both issuers' MMAs
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ds_free[b], 1);          // dS^T buffer b read by issuer B's MMAs
      mbar_init(&dpt_issued[b], 1);       // issuer A has issued the next dP^T
    }
    mbar_init(&s_full, 1);
    mbar_init(&dp_full, 1);
    mbar_init(&p_ready, 2 * kBlockN);     // both compute warpgroups
    mbar_init(&ds_ready, 2 * kBlockN);
    mbar_init(&dq_free, kBlockM);         // the dQ warps have read dQ out of TMEM
    fence_mbarrier_init();
  }
  if (warp == kBwdMmaWarp) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == kBwdProducerWarp) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_do);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      mbar_arrive_expect_tx(&kv_full, 2 * kTileBytes);
      tma_load_3d(&p.tm_k, &kv_full, sK, 0, g, sp.k0 + j0);
      tma_load_3d(&p.tm_v, &kv_full, sV, 0, g, sp.k0 + j0);
    }
    int issued = 0;
    for (int m = 0; m < num; ++m) {
      const int st = m % kBwdStages;
      if (m >= kBwdStages &&
          !mbar_wait_warp(&q_empty[st], ((m / kBwdStages) & 1) ^ 1, &abort_flag)) {
        if (lane == 0) {
          abort_flag = 1;
          atomicCAS(p.err, 0, DEVERR_TIMEOUT_BWD + 1);
        }
        break;
      }
      const int h = h_first + m % hpc;
      const int i0 = (qt_first + m / hpc) * kBlockM;
#ifdef ATTN_SINK_TEST_HOOKS
      if (m == p.skip_q_step) {
        // test build: withhold this step's tiles; every wait for them runs out
        const unsigned long long t0 = global_timer_ns();
        while (!abort_flag && global_timer_ns() - t0 <= kWaitLimitNs) __nanosleep(1000);
        if (lane == 0) {
          abort_flag = 1;
          atomicCAS(p.err, 0, DEVERR_TIMEOUT_BWD + 1);
        }
        break;
      }
#endif
      if (lane == 0) {
        mbar_arrive_expect_tx(&q_full[st], 2 * kTileBytes);
        tma_load_3d(&p.tm_q, &q_full[st], sQ + st * kTileBytes, 0, h, sp.q0 + i0);
        tma_load_3d(&p.tm_do, &q_full[st], sdO + st * kTileBytes, 0, h, sp.q0 + i0);
      }
      // (-lse log2 e, D) of the step's 128 query rows, copied asynchronously into
      // two planes (so that runs of rows load as one vector); rows past the
      // sequence read a valid row and are masked by the compute warps.
      #pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int t = lane + 32 * u;
        const size_t idx = (size_t)h * p.total_q + sp.q0 + min(i0 + t, sp.nq - 1);
        const float* src = reinterpret_cast<const float*>(p.LD + idx);
        cp_async_4(smem_u32(&s_nL[st][t]), src);
        cp_async_4(smem_u32(&s_D[st][t]), src + 1);
      }
      cp_async_mbar_arrive_noinc(&q_full[st]);
      issued = m + 1;
    }
    if (abort_flag && lane == 0) {
      mbar_wait(&kv_full, 0, nullptr);
      for (int m = max(0, issued - kBwdStages); m < issued; ++m)
        mbar_wait(&q_full[m % kBwdStages], (m / kBwdStages) & 1, nullptr);
    }
  } else if (warp == kBwdMmaWarp || warp == kBwdMma2Warp) {
    // ---------------------------------------------------------------- MMA issuers
    // Each step (one query head, 128 queries) splits the compute warps' work in
    // two phases, P^T then dS^T, so that the products waiting on P^T start
    // while dS^T is still being formed.  Two issuing threads, each owning its
    // accumulators so that its MMAs run in issue order:
    //   A (warp 9):  dV += P^T dO (after phase 1), S^T of the next step (into
    //                the columns phase 1 has read), dP^T of the next step (after
    //                phase 2 has read dP^T), all N = 128 / K = 128 queries
    //   B (warp 14): dK += dS^T Q, dQ = dS K (after phase 2), once A has issued
    //                the next dP^T, so that the compute warps' next operand is
    //                ahead of them in the tensor pipe
    // A stage of Q/dO is refilled once both issuers' commits on q_empty have
    // landed (A's after dV, B's after dK); B's commit on ds_free[b] releases
    // dS^T buffer b two steps later.
    if (lane == 0) {
      const bool issuer_a = warp == kBwdMmaWarp;
      const uint32_t id_s = make_idesc(kFmtF16, kBlockN, kBlockM, false, false);
      const uint32_t id_dvdk = make_idesc(kFmtF16, kBlockN, kHeadDim, false, true);
      const uint32_t id_dq = make_idesc(kFmtF16, kBlockM, kHeadDim, true, true);
      // Shared-memory descriptors, built once; an operand at byte offset o from
      // a base is that base's descriptor plus o / 16 (the start-address field).
      const uint64_t dK_mn = make_sdesc_sw128(smem_u32(sK), 16384, 1024);  // K, MN-major
      const uint64_t dQ_k = make_sdesc_sw128(smem_u32(sQ), 16, 1024);      // stage 0
      const uint64_t dQ_mn = make_sdesc_sw128(smem_u32(sQ), 16384, 1024);
      const uint64_t dO_k = make_sdesc_sw128(smem_u32(sdO), 16, 1024);
      const uint64_t dO_mn = make_sdesc_sw128(smem_u32(sdO), 16384, 1024);
      const uint64_t dS_k = make_sdesc_sw128(smem_u32(sdS), 16, 1024);     // buffer 0
      const uint64_t dS_mn = make_sdesc_sw128(smem_u32(sdS), 16384, 1024);
      constexpr uint32_t kTileU = kTileBytes >> 4, kPTileU = kPTileBytes >> 4;
      // S^T = K Q^T or dP^T = V dO^T of step m over its 128 queries (N = 128).
      auto issue_s = [&](int m) {
        const uint32_t qo = (m % kBwdStages) * kTileU;
        #pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k)
          mma_ts(tmem + kColST, tmem + kColK + 8 * k, dQ_k + qo + 2 * k, id_s, k > 0);
        mma_commit(&s_full);
      };
      auto issue_dp = [&](int m) {
        const uint32_t qo = (m % kBwdStages) * kTileU;
        #pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k)
          mma_ts(tmem + kColDPT, tmem + kColV + 8 * k, dO_k + qo + 2 * k, id_s, k > 0);
        mma_commit(&dp_full);
      };
      bool ok = true;
      if (issuer_a) {
        // kv_tmem: K and V are in TMEM (the compute warps copied them from SMEM)
        ok = mbar_wait(&kv_tmem, 0, &abort_flag) && mbar_wait(&q_full[0], 0, &abort_flag);
        if (ok) {
          tc_fence_after();
          issue_s(0);
          issue_dp(0);
        }
        for (int m = 0; ok && m < num; ++m) {
          const int st = m % kBwdStages;
          const bool more = m + 1 < num;
          // phase 1 done: P^T in TMEM (over the S^T columns it has read)
          if (!mbar_wait(&p_ready, m & 1, &abort_flag)) { ok = false; break; }
          tc_fence_after();
          // dV += P^T dO over the step's 128 queries; P^T of queries 64hh.. sits
          // in the first 32 columns of S^T half hh
          #pragma unroll
          for (int k = 0; k < kBlockM / 16; ++k)
            mma_ts(tmem + kColDV, tmem + kColST + 64 * (k >> 2) + 8 * (k & 3),
                   dO_mn + st * kTileU + 128 * k, id_dvdk, (m > 0 || k > 0));
          mma_commit(&q_empty[st]);
          if (more) {
            if (!mbar_wait(&q_full[(m + 1) % kBwdStages], ((m + 1) / kBwdStages) & 1,
                           &abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(m + 1);
          }
          // phase 2 done: dS^T in SMEM, dP^T read
          if (!mbar_wait(&ds_ready, m & 1, &abort_flag)) { ok = false; break; }
          tc_fence_after();
          if (more) issue_dp(m + 1);
          mbar_arrive(&dpt_issued[m & 1]);
        }
      } else {
        for (int m = 0; ok && m < num; ++m) {
          const int st = m % kBwdStages;
          const uint32_t so = (m & 1) * kPTileU;            // dS^T buffer of this step
          // A has seen phase 2 of this step and issued the next dP^T
          if (!mbar_wait(&dpt_issued[m & 1], (m >> 1) & 1, &abort_flag)) { ok = false; break; }
          tc_fence_after();
          // dK += dS^T Q over the step's 128 queries (dS^T tile hh holds queries 64hh..)
          #pragma unroll
          for (int k = 0; k < kBlockM / 16; ++k)
            mma_ss(tmem + kColDK, dS_k + so + (k >> 2) * kTileU + 2 * (k & 3),
                   dQ_mn + st * kTileU + 128 * k, id_dvdk, (m > 0 || k > 0));
          // dK is this step's last reader of its Q/dO stage (dQ reads dS^T and
          // K): release the stage now, not after dQ, so that its refill starts
          // earlier
          mma_commit(&q_empty[st]);
          if (!p.skip_dq) {
            // the dQ warps have read the previous dQ out of TMEM
            if (!mbar_wait(&dq_free, m & 1, &abort_flag)) { ok = false; break; }
            tc_fence_after();
            // dQ = dS K  (A: dS^T read MN-major, M = queries; B: K read MN-major)
            #pragma unroll
            for (int k = 0; k < kBlockN / 16; ++k)
              mma_ss(tmem + kColDQ, dS_mn + so + 128 * k, dK_mn + 128 * k, id_dq, k > 0);
            mma_commit(&mma2_done);
          }
          mma_commit(&ds_free[m & 1]);
        }
      }
      if (!ok) {
        abort_flag = 1;
        atomicCAS(p.err, 0, DEVERR_TIMEOUT_BWD + 2);
      }
      // both issuers commit once; `drained` completes when all their MMAs have
      mma_commit(&drained);
      mbar_wait(&drained, 0, nullptr);
    }
  } else if (warp < 8) {
    // ---------------------------------------------------------------- compute warps
    // warpgroup hh handles queries [64 hh, 64 hh + 64) of every step
    const int hh = warp >> 2;
    const int r = tid & 127;                        // key row in tile = TMEM lane
    const int j = j0 + r;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint64_t sl2x2 = f2(p.scale_log2, p.scale_log2);
    const int imin = p.causal ? j - off : 0;
    const int imax = (p.causal && p.window > 0) ? j - off + p.window - 1 : sp.nq - 1;
    const bool key_ok = j < sp.nk;
    // K (warpgroup 0) or V (warpgroup 1) row r into TMEM: the swizzled SMEM row
    // holds 8 chunks of 8 fp16, i.e. the 32 packed columns in order.
    bool ok = mbar_wait_warp(&kv_full, 0, &abort_flag);
    if (ok) {
      uint32_t w[32];
      const uint32_t row = smem_u32(hh == 0 ? sK : sV);
      #pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        uint4 q4;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(q4.x), "=r"(q4.y), "=r"(q4.z), "=r"(q4.w)
                     : "r"(row + sw128_offset(r, cc)));
        w[4 * cc] = q4.x; w[4 * cc + 1] = q4.y; w[4 * cc + 2] = q4.z; w[4 * cc + 3] = q4.w;
      }
      tmem_st_x32(tmem + lane_base + (hh == 0 ? kColK : kColV), w);
      tmem_st_wait();
    }
    tc_fence_before();
    mbar_arrive(&kv_tmem);
    const uint32_t tST = tmem + lane_base + kColST + 64 * hh;
    const uint32_t tDPT = tmem + lane_base + kColDPT + 64 * hh;
    for (int m = 0; ok && m < num; ++m) {
      const int st = m % kBwdStages;
      const int i0 = (qt_first + m / hpc) * kBlockM + 64 * hh;   // first query of this half
      // q_full: the producer's lse / D rows of this step are in SMEM.
      // s_full: S^T of this step (and every earlier MMA of issuer A) has completed.
      if (!mbar_wait_warp(&q_full[st], (m / kBwdStages) & 1, &abort_flag) ||
          !mbar_wait_warp(&s_full, m & 1, &abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool need_mask = (j0 + kBlockN > sp.nk) || (i0 + 64 > sp.nq) ||
                             (p.causal && (j0 + kBlockN - 1 > i0 + off ||
                                           (p.window > 0 && j0 <= i0 + 63 + off - p.window)));
      // Phase 1: P^T of this half's 64 queries, written (fp16) over the first 32
      // S^T columns of the half once S^T has been read.  The mask test is hoisted
      // out of the element loop (a branch per element keeps the compiler from
      // interleaving the elements' exponentials).
      uint32_t pk[32];
      {
        uint32_t sr[64];
        tmem_ld_x32(tST, sr);
        tmem_ld_x32(tST + 32, sr + 32);
        tmem_ld_wait();
        const float* nl_row = &s_nL[st][64 * hh];
        // this key's visible queries within the sequence
        const int vis_lo = key_ok ? imin : 1;
        const int vis_hi = key_ok ? min(imax, sp.nq - 1) : 0;
        if (need_mask)
          bwd_p_chunk<true>(sr, nl_row, sl2x2, i0, vis_lo, vis_hi, pk);
        else
          bwd_p_chunk<false>(sr, nl_row, sl2x2, i0, vis_lo, vis_hi, pk);
      }
      tmem_st_x16(tST, pk);
      tmem_st_x16(tST + 16, pk + 16);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_ready);
      // Phase 2: dS^T = P^T o (dP^T - D) into the step's SMEM buffer.
      // dp_full: dP^T of this step has completed.  ds_free: issuer B's MMAs of
      // step m - 2 (the last readers of this step's dS^T buffer) have completed;
      // buffer m & 1 is released once per two steps.
      if (!mbar_wait_warp(&dp_full, m & 1, &abort_flag) ||
          (m >= 2 && !mbar_wait_warp(&ds_free[m & 1], ((m >> 1) - 1) & 1, &abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sbase = smem_u32(sdS + (m & 1) * kPTileBytes) + hh * kTileBytes;
      #pragma unroll
      for (int c = 0; c < 64; c += 32) {
        uint32_t dr[32], dk[16];
        tmem_ld_x32(tDPT + c, dr);
        tmem_ld_wait();
        bwd_ds_chunk(dr, pk + (c >> 1), &s_D[st][64 * hh + c], dk);
        // dS^T row r, queries c..c+31 of this half: 4 chunks of 16 bytes
        #pragma unroll
        for (int u = 0; u < 4; ++u)
          st_shared_v4(sbase + sw128_offset(r, (c >> 3) + u), dk[4 * u], dk[4 * u + 1],
                       dk[4 * u + 2], dk[4 * u + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&ds_ready);
    }
    // `drained` completes once, after the MMA warp's last commit: every MMA into
    // dK / dV has landed.  (A parity wait on the per-step barriers could be two
    // phases behind here and pass early.)
    if (ok && !mbar_wait_warp(&drained, 0, &abort_flag)) ok = false;
    if (!ok) {
      abort_flag = 1;
      atomicCAS(p.err, 0, DEVERR_TIMEOUT_BWD + 3);
    } else {
      tc_fence_after();
      // Epilogue: warpgroup 0 stores dV, warpgroup 1 dK (times the softmax scale).
      const int which = hh == 0 ? 1 : 0;
      float v[kHeadDim];
      const uint32_t col = which == 0 ? kColDK : kColDV;
      tmem_ld_x32(tmem + lane_base + col, reinterpret_cast<uint32_t*>(v));
      tmem_ld_x32(tmem + lane_base + col + 32, reinterpret_cast<uint32_t*>(v + 32));
      tmem_ld_wait();
      if (key_ok)
        store_kv_grad_row(p, part, (size_t)(sp.k0 + j), g, which, v,
                          which == 0 ? p.scale : 1.0f);
    }
  } else if (warp >= kBwdDqWarp0 && warp < kBwdDqWarp0 + 4) {
    // ---------------------------------------------------------------- dQ warps
    // Each step's dQ tile (128 queries x 64, fp32, times the softmax scale) is
    // read out of TMEM and added to the fp32 accumulator in two halves of 32
    // columns, each staged in one 128-byte-swizzled SMEM tile and summed by a
    // TMA reduce-add.  Rows past the sequence end are exact zeros (their dS is
    // masked), so adding them into the next sequence's rows changes nothing.
    const int r = 32 * (warp & 3) + lane;            // query row in tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const bool leader = (warp == kBwdDqWarp0 && lane == 0);
    const uint32_t stage = smem_u32(sdQ);
    bool ok = true;
    // (with skip_dq there is no dQ here: the loop does not run)
    // The dQ TMEM columns are free for step 0.
    if (!p.skip_dq && num > 0) mbar_arrive(&dq_free);
    for (int m = 0; m < (p.skip_dq ? 0 : num); ++m) {
      const int h = h_first + m % hpc;
      const int i0 = (qt_first + m / hpc) * kBlockM;
      const bool waited = mbar_wait_warp(&mma2_done, m & 1, &abort_flag);
      // all four warps agree on the wait's outcome (and leave together)
      if (!named_barrier_and(1, 128, waited)) { ok = false; break; }
      tc_fence_after();
      uint32_t v[64];
      tmem_ld_x32(tmem + lane_base + kColDQ, v);
      tmem_ld_x32(tmem + lane_base + kColDQ + 32, v + 32);
      tmem_ld_wait();
      tc_fence_before();
      // dQ TMEM is free for the next step
      if (m + 1 < num) mbar_arrive(&dq_free);
      #pragma unroll
      for (int half = 0; half < 2; ++half) {
        // the previous reduce-add has read the staging tile
        if (leader) bulk_wait_group_read0();
        named_barrier_sync(1, 128);
        #pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t* w = v + 32 * half + 4 * c;
          st_shared_v4(stage + sw128_offset(r, c),
                       __float_as_uint(__uint_as_float(w[0]) * p.scale),
                       __float_as_uint(__uint_as_float(w[1]) * p.scale),
                       __float_as_uint(__uint_as_float(w[2]) * p.scale),
                       __float_as_uint(__uint_as_float(w[3]) * p.scale));
        }
        fence_proxy_async_smem();
        named_barrier_sync(1, 128);
        if (leader) {
          tma_reduce_add_3d(&p.tm_dq, sdQ, 32 * half, h, sp.q0 + i0);
          bulk_commit_group();
        }
      }
    }
    if (leader) bulk_wait_group0();
    if (!ok) {
      abort_flag = 1;
      if (lane == 0) atomicCAS(p.err, 0, DEVERR_TIMEOUT_BWD + 4);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kBwdMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace attn_sink
